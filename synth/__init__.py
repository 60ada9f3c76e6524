"""Seeded synthetic inputs for the Q4_K x M-row weight-streaming matmul.

This package feeds both the CPU oracle and the CUDA path.  It draws random bytes and
rounds random reals to fp16; it holds none of the method's arithmetic.  The generator
(a counter-based SplitMix64, see ``synth.c``) makes every block and every activation a
pure function of ``(seed, tensor_id, index)``, so a test can regenerate any rows of a
12.7 GB weight stack without holding it in host memory.

Workload shapes follow the decode step described on the page "Running 4 coding agents
on one RTX 3090: a custom CUDA engine for Qwen3.8-27B" (section "How parallel decoding
works": every active agent's next token plus two drafts, stacked into 12 rows, multiplied
against the whole weight set in one pass).  The 27B-shaped matrix list is in ``STACK``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_synth.so")

BLOCK_BYTES = 144      # one Q4_K super-block
BLOCK_WEIGHTS = 256    # weights per super-block
D_SCALE = 1e-3         # d, dmin = fp16(|N(0,1)| * 1e-3)


def build(force: bool = False) -> str:
    """Compile the generator with the host C compiler (OpenMP over blocks)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_key.restype = ctypes.c_uint64
        lib.synth_key.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_f16_from_double.restype = ctypes.c_uint16
        lib.synth_f16_from_double.argtypes = [ctypes.c_double]
        lib.synth_q4k_blocks.restype = None
        lib.synth_q4k_blocks.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                         ctypes.c_uint64, ctypes.c_int64, ctypes.c_double]
        lib.synth_x_f16.restype = None
        lib.synth_x_f16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                    ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                    ctypes.c_double]
        lib.synth_blocks.restype = None
        lib.synth_blocks.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                                     ctypes.c_uint64, ctypes.c_int64, ctypes.c_double]
        lib.synth_kv_records.restype = None
        lib.synth_kv_records.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
                                         ctypes.c_int64, ctypes.c_double]
        lib.synth_raw.restype = None
        lib.synth_raw.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                  ctypes.c_uint64]
        _lib = lib
    return _lib


def f16_bits(v: float) -> int:
    """fp16 bit pattern of a double, round-to-nearest-even (the generator's rounding)."""
    return int(_load().synth_f16_from_double(float(v)))


def raw(key: int, first: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_raw(out.ctypes.data, n, key, first)
    return out


def key(seed: int, tensor_id: int) -> int:
    return int(_load().synth_key(seed, tensor_id))


def q4k_blocks(nblocks: int, seed: int, tensor_id: int, first_block: int = 0,
               scale_mul: float = D_SCALE, out: np.ndarray | None = None) -> np.ndarray:
    """Blocks first_block .. first_block+nblocks-1 of a tensor, as uint8 [nblocks, 144]."""
    if out is None:
        out = np.empty((nblocks, BLOCK_BYTES), dtype=np.uint8)
    assert out.dtype == np.uint8 and out.flags.c_contiguous and out.size == nblocks * BLOCK_BYTES
    _load().synth_q4k_blocks(out.ctypes.data, nblocks, seed, tensor_id, first_block, scale_mul)
    return out


def q4k_matrix(n: int, k: int, seed: int, tensor_id: int, rows: np.ndarray | None = None,
               scale_mul: float = D_SCALE) -> np.ndarray:
    """Weight matrix W[n, k] as GGUF-ordered super-blocks, uint8 [n, k/256, 144].

    Row r of the matrix is blocks r*(k/256) .. (r+1)*(k/256)-1 of the tensor.  With
    ``rows`` given, only those rows are generated (in that order)."""
    assert k % BLOCK_WEIGHTS == 0
    kb = k // BLOCK_WEIGHTS
    if rows is None:
        out = np.empty((n, kb, BLOCK_BYTES), dtype=np.uint8)
        q4k_blocks(n * kb, seed, tensor_id, 0, scale_mul, out.reshape(n * kb, BLOCK_BYTES))
        return out
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((len(rows), kb, BLOCK_BYTES), dtype=np.uint8)
    for i, r in enumerate(rows):
        assert 0 <= r < n
        q4k_blocks(kb, seed, tensor_id, int(r) * kb, scale_mul, out[i].reshape(kb, BLOCK_BYTES))
    return out


# other block types of a mixed-quant model file: (block bytes, weights per block, d scale);
# the scales keep |w| below about 1, like the Q4_K workloads
Q6_K = (210, 256, 2e-4)
Q8_0 = (34, 32, 1e-2)


def fmt_matrix(fmt: tuple, n: int, k: int, seed: int, tensor_id: int,
               rows: np.ndarray | None = None) -> np.ndarray:
    """Weight matrix W[n, k] in block type fmt (Q6_K or Q8_0) as GGUF-ordered blocks,
    uint8 [n, k / weights per block, block bytes]; with ``rows``, only those rows."""
    nbytes, per, scale = fmt
    assert k % per == 0
    kb = k // per
    rows_ = range(n) if rows is None else np.asarray(rows, dtype=np.int64)
    if rows is None:
        out = np.empty((n, kb, nbytes), dtype=np.uint8)
        _load().synth_blocks(out.ctypes.data, n * kb, nbytes, seed, tensor_id, 0, scale)
        return out
    out = np.empty((len(rows_), kb, nbytes), dtype=np.uint8)
    for i, r in enumerate(rows_):
        assert 0 <= r < n
        _load().synth_blocks(out[i].ctypes.data, kb, nbytes, seed, tensor_id, int(r) * kb, scale)
    return out


def x_f16(m: int, k: int, seed: int, tensor_id: int, outlier_p: float = 0.0,
          outlier_mul: float = 20.0) -> np.ndarray:
    """Activations x[m, k] as fp16 (numpy float16), element index = row * k + col."""
    out = np.empty((m, k), dtype=np.uint16)
    _load().synth_x_f16(out.ctypes.data, m * k, seed, tensor_id, 0, outlier_p, outlier_mul)
    return out.view(np.float16)


# ----------------------------------------------------------------------------------------
# Workload shapes.  A matrix maps K inputs to N outputs; W is stored N rows of K/256 blocks.
# ----------------------------------------------------------------------------------------
@dataclass(frozen=True)
class Matrix:
    name: str
    n: int          # outputs
    k: int          # inputs
    tensor_id: int  # generator stream of the weights; activations use X_ID_OFFSET + tensor_id

    @property
    def weight_bytes(self) -> int:
        return self.n * self.k // BLOCK_WEIGHTS * BLOCK_BYTES


X_ID_OFFSET = 1000
LAYERS = 64
HIDDEN = 5120
LAYER_SHAPES = (("qkv", 8192, 5120), ("o", 5120, 6144), ("gate_up", 34816, 5120),
                ("down", 5120, 17408))
LM_HEAD = Matrix("lm_head", 151936, 5120, 256)


def layer_matrices(layer: int) -> list[Matrix]:
    return [Matrix(f"L{layer}.{nm}", n, k, layer * 4 + i)
            for i, (nm, n, k) in enumerate(LAYER_SHAPES)]


def stack(layers: int = LAYERS, lm_head: bool = True) -> list[Matrix]:
    """The 27B-shaped decode stack: per layer qkv, o, gate_up, down; then lm_head."""
    mats = [m for layer in range(layers) for m in layer_matrices(layer)]
    if lm_head:
        mats.append(LM_HEAD)
    return mats


SINGLE_PROJECTION = Matrix("proj4096", 4096, 4096, 0)
SWEEP_MATRICES = (layer_matrices(0)[2], layer_matrices(0)[3])   # gate_up, down
SWEEP_M = (1, 2, 4, 8, 12, 16, 32, 64)


# ----------------------------------------------------------------- decode attention inputs
# Attention shapes of the 27B-shaped stack: qkv 5120 -> 8192 = 48 query heads + 2 x 8 KV heads
# of 128, o 6144 -> 5120 (48 x 128 in).  KV pages of 64 tokens, one 17,408-byte record per
# (page, KV head); the pool layout is documented with the attention oracle.
ATTN_HEADS, ATTN_KV_HEADS, ATTN_DIM, ATTN_PAGE = 48, 8, 128, 64
KV_RECORD_BYTES = 17408
KV_SCALE = 1.0 / 64  # K, V = fp16(|N(0,1)| / 64) * int8: values of order one


def kv_pool(pages: int, kv_heads: int, seed: int, tensor_id: int, first_page: int = 0) -> np.ndarray:
    """Pages first_page .. first_page+pages-1 of a synthetic q8_0 KV pool, as uint8
    [pages * kv_heads * 17408] (record (page, head) at (page * kv_heads + head) * 17408)."""
    out = np.empty(pages * kv_heads * KV_RECORD_BYTES, dtype=np.uint8)
    _load().synth_kv_records(out.ctypes.data, pages * kv_heads, seed, tensor_id, first_page * kv_heads,
                             KV_SCALE)
    return out


@dataclass(frozen=True)
class AttnWorkload:
    """Agents with cache lengths, R stacked rows per agent (row j of agent a attends to the
    agent's first cache[a] + j + 1 tokens), and a shared pool whose pages are handed out in a
    seeded random order."""
    cache: tuple            # tokens already cached per agent
    rows_per_agent: int
    heads: int = ATTN_HEADS
    kv_heads: int = ATTN_KV_HEADS

    def lengths(self):
        return [c + self.rows_per_agent for c in self.cache]

    def pages_of(self):
        return [(n + ATTN_PAGE - 1) // ATTN_PAGE for n in self.lengths()]

    def build(self, seed: int = 0):
        """(page_table int32 [agents, max_pages], pool pages, row_agent, row_len)."""
        pages = self.pages_of()
        total = sum(pages)
        perm = np.random.default_rng(seed).permutation(total).astype(np.int32)
        max_pages = max(pages)
        table = np.zeros((len(pages), max_pages), dtype=np.int32)
        off = 0
        for a, n in enumerate(pages):
            table[a, :n] = perm[off:off + n]
            off += n
        row_agent = np.repeat(np.arange(len(pages), dtype=np.int32), self.rows_per_agent)
        row_len = np.array([c + j + 1 for c in self.cache for j in range(self.rows_per_agent)], dtype=np.int32)
        return table, total, row_agent, row_len


# The decode step of the pages: 4 agents with 23K-token contexts, 1 token + 2 drafts each.
ATTN_DECODE = AttnWorkload(cache=(23000, 23000, 23000, 23000), rows_per_agent=3)
# The wide speculative verify step: 8 streams x (1 token + 7 block drafts); 8 x 16,000 cached
# tokens fill most of the pages' shared 132K-token pool.
ATTN_VERIFY = AttnWorkload(cache=(16000,) * 8, rows_per_agent=8)


def attn_q(rows: int, heads: int, seed: int, tensor_id: int) -> np.ndarray:
    """Queries q[rows, heads, 128] fp16, N(0,1)."""
    return x_f16(rows, heads * ATTN_DIM, seed, tensor_id).reshape(rows, heads, ATTN_DIM)
