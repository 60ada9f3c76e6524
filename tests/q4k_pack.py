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


def pack_q8_0(d_bits: int, q) -> np.ndarray:
    """Q8_0 block (GGUF): bytes 0-1 d (fp16 LE), then the 32 quants as int8."""
    q = [int(v) for v in q]
    assert len(q) == 32 and all(-128 <= v < 128 for v in q)
    raw = int(d_bits).to_bytes(2, "little") + bytes((v + 256) % 256 for v in q)
    return np.frombuffer(raw, dtype=np.uint8).copy()


def pack_q6_k(d_bits: int, sc, q) -> np.ndarray:
    """Q6_K super-block (GGUF) from 16 int8 scales and 256 6-bit quants.

    Written by walking the 256 weights and scattering each one's bits: weight i sits in
    half h = i // 128 at position r = i % 128; its quarter c = r // 32 picks the ql byte
    (first or second 32 of the half's 64) and its nibble (low for c < 2), and the 2-bit
    field (2c .. 2c+1) of qh byte 32h + i % 32.  Bytes: ql 0-127, qh 128-191, scales
    192-207, d 208-209."""
    q = [int(v) for v in q]
    sc = [int(v) for v in sc]
    assert len(q) == 256 and all(0 <= v < 64 for v in q)
    assert len(sc) == 16 and all(-128 <= v < 128 for v in sc)
    ql, qh = [0] * 128, [0] * 64
    for i, v in enumerate(q):
        h, r = divmod(i, 128)
        c, l = divmod(r, 32)
        ql_index = 64 * h + l + 32 * (c % 2)
        ql[ql_index] |= (v & 15) << (4 * (c // 2))
        qh[32 * h + l] |= (v >> 4) << (2 * c)
    raw = bytes(ql) + bytes(qh) + bytes((v + 256) % 256 for v in sc) + int(d_bits).to_bytes(2, "little")
    assert len(raw) == 210
    return np.frombuffer(raw, dtype=np.uint8).copy()
