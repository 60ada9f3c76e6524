"""Test-side packer for Q4_K super-blocks: parameters -> 144 bytes.

Written from the format description in the opposite direction to the oracle's unpacker
(the oracle reads bytes; this writes them), so that a round trip through both pins the
bit layout.  Format (GGUF Q4_K, the pages' "Q4_K_M"):
  bytes 0-1 d (fp16 LE), 2-3 dmin (fp16 LE), 4-15 scale bytes s[0..11], 16-143 qs[0..127].
  For j < 4:  low 6 bits of s[j] hold sc_j, low 6 bits of s[j+4] hold m_j.
  For j >= 4: the low nibble of s[j+4] holds the low 4 bits of sc_j, its high nibble the
              low 4 bits of m_j; the top 2 bits of s[j-4] hold sc_j >> 4 and the top
              2 bits of s[j] hold m_j >> 4.
  Weight i = 64c + r: r < 32 -> low nibble of qs[32c + r]; r >= 32 -> high nibble of
  qs[32c + r - 32].
"""
from __future__ import annotations

import numpy as np


def pack_scales(sc, mn) -> bytes:
    sc = [int(v) for v in sc]
    mn = [int(v) for v in mn]
    assert len(sc) == 8 and len(mn) == 8 and all(0 <= v < 64 for v in sc + mn)
    s = [0] * 12
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    return bytes(s)


def pack_quants(q) -> bytes:
    q = [int(v) for v in q]
    assert len(q) == 256 and all(0 <= v < 16 for v in q)
    qs = [0] * 128
    for c in range(4):
        for r in range(32):
            qs[32 * c + r] = q[64 * c + r] | (q[64 * c + 32 + r] << 4)
    return bytes(qs)


def pack_block(d_bits: int, dmin_bits: int, sc, mn, q) -> np.ndarray:
    raw = (int(d_bits).to_bytes(2, "little") + int(dmin_bits).to_bytes(2, "little")
           + pack_scales(sc, mn) + pack_quants(q))
    assert len(raw) == 144
    return np.frombuffer(raw, dtype=np.uint8).copy()
