"""CPU oracle for the Q4_K x M-row matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The product path (``bit_weight_streaming_q4_gb300``) never does,
and shares no code with it.  The arithmetic lives in ``q4k_oracle.c`` (plain C, fp32
dequantisation, double accumulation, OpenMP over output channels); this module only
compiles it and marshals numpy arrays.

Pins (tests/test_oracle_pins.py) check it against closed forms, hand-packed blocks,
brute force in exact rational arithmetic, and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4k_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "attn_oracle.c")]
_LIB = os.path.join(_HERE, "_oracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler.  -ffp-contract=off keeps each
    operation rounded as written."""
    newest = max(os.path.getmtime(p) for p in _SRCS)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC",
                               "-shared", "-std=c11", *_SRCS, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_f16_to_double.restype = ctypes.c_double
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_scale_min.restype = None
        lib.oracle_scale_min.argtypes = [ctypes.c_void_p, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_int)]
        lib.oracle_quant.restype = ctypes.c_int
        lib.oracle_quant.argtypes = [ctypes.c_void_p, ctypes.c_int]
        lib.oracle_dequant_block.restype = None
        lib.oracle_dequant_block.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_qmm.restype = ctypes.c_int
        lib.oracle_qmm.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_qmm_fmt.restype = ctypes.c_int
        lib.oracle_qmm_fmt.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_int]
        lib.oracle_dequant_fmt.restype = ctypes.c_int
        lib.oracle_dequant_fmt.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_attn.restype = ctypes.c_int
        lib.oracle_attn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_kv.restype = ctypes.c_double
        lib.oracle_kv.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_q6k_quant.restype = ctypes.c_int
        lib.oracle_q6k_quant.argtypes = [ctypes.c_void_p, ctypes.c_int]
        _lib = lib
    return _lib


def f16_to_double(bits: int) -> float:
    return float(_load().oracle_f16_to_double(bits))


def scale_min(scales12: bytes | np.ndarray, j: int) -> tuple[int, int]:
    s = np.ascontiguousarray(np.frombuffer(bytes(scales12), dtype=np.uint8))
    assert s.size == 12
    sc, mn = ctypes.c_int(), ctypes.c_int()
    _load().oracle_scale_min(s.ctypes.data, j, ctypes.byref(sc), ctypes.byref(mn))
    return sc.value, mn.value


def quant(qs128: np.ndarray, i: int) -> int:
    q = np.ascontiguousarray(qs128, dtype=np.uint8)
    assert q.size == 128
    return int(_load().oracle_quant(q.ctypes.data, i))


def dequant_block(block: np.ndarray) -> np.ndarray:
    """One 144-byte super-block -> 256 fp32 weights."""
    b = np.ascontiguousarray(block, dtype=np.uint8).reshape(144)
    w = np.empty(256, dtype=np.float32)
    _load().oracle_dequant_block(b.ctypes.data, w.ctypes.data)
    return w


def dequant_matrix(blocks: np.ndarray) -> np.ndarray:
    """[N, K/256, 144] blocks -> fp32 W[N, K] (other formats: double, by block size)."""
    n, kb, nbytes = blocks.shape
    if nbytes != 144:
        per = FORMATS[nbytes][1]
        out = np.empty((n, kb * per), dtype=np.float64)
        for r in range(n):
            for b in range(kb):
                out[r, per * b:per * (b + 1)] = dequant_block_fmt(blocks[r, b])
        return out
    out = np.empty((n, kb * 256), dtype=np.float32)
    for r in range(n):
        for b in range(kb):
            out[r, 256 * b:256 * (b + 1)] = dequant_block(blocks[r, b])
    return out


# block bytes -> (format id of the C oracle, weights per block)
FORMATS = {144: (0, 256), 210: (1, 256), 34: (2, 32)}
FORMAT_NAMES = {144: "Q4_K", 210: "Q6_K", 34: "Q8_0"}


def qmm(blocks: np.ndarray, x: np.ndarray, nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """y[M, N] = x W^T in double and S[M, N] = sum_k |w x|.

    blocks: uint8 [N, blocks per row, block bytes] (GGUF order; 144 B Q4_K, 210 B Q6_K,
    34 B Q8_0 blocks); x: float16 [M, K]."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    assert blocks.ndim == 3 and blocks.shape[2] in FORMATS
    fmt, per = FORMATS[blocks.shape[2]]
    n, kb = blocks.shape[0], blocks.shape[1]
    k = kb * per
    x = np.ascontiguousarray(x, dtype=np.float16)
    assert x.ndim == 2 and x.shape[1] == k
    m = x.shape[0]
    y = np.empty((m, n), dtype=np.float64)
    s = np.empty((m, n), dtype=np.float64)
    rc = _load().oracle_qmm_fmt(fmt, blocks.ctypes.data, n, k, x.view(np.uint16).ctypes.data, m,
                                y.ctypes.data, s.ctypes.data, nthreads)
    if rc != 0:
        raise RuntimeError("oracle_qmm failed")
    return y, s


def dequant_block_fmt(block: np.ndarray) -> np.ndarray:
    """One block of any format (by its size) -> its weights in double."""
    b = np.ascontiguousarray(block, dtype=np.uint8).ravel()
    fmt, per = FORMATS[b.size]
    w = np.empty(per, dtype=np.float64)
    assert _load().oracle_dequant_fmt(fmt, b.ctypes.data, w.ctypes.data) == per
    return w


def q6k_quant(block: np.ndarray, i: int) -> int:
    """The 6-bit quant of weight i of a 210-byte Q6_K block."""
    b = np.ascontiguousarray(block, dtype=np.uint8).ravel()
    assert b.size == 210
    return int(_load().oracle_q6k_quant(b.ctypes.data, i))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def tolerance(s_abs: np.ndarray) -> np.ndarray:
    """Per-element bound for the GPU result: 2e-3 * sum_k |w x| + 1e-6."""
    return 2e-3 * s_abs + 1e-6


def argmax_rows(y: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Greedy verification of each row (page "Running 4 coding agents on one RTX 3090",
    section "How parallel decoding works": a drafted token is kept when it is the most likely
    next token, i.e. the largest logit of its row): idx[r] = the column holding the row's
    largest value, val[r] = that value.  The pages do not order equal maxima; the reading
    taken here is the lowest column (numpy's argmax returns the first one)."""
    y = np.asarray(y)
    assert y.ndim == 2 and y.shape[1] > 0
    idx = np.argmax(y, axis=1)
    return idx, y[np.arange(y.shape[0]), idx]


# --------------------------------------------------------------------- decode attention
ATTN_D, ATTN_PAGE_TOKENS, ATTN_RECORD_BYTES = 128, 64, 17408


def attn(pool: np.ndarray, page_table: np.ndarray, q: np.ndarray, row_agent, row_len, kv_heads: int,
         nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Stacked-row decode attention over a paged q8_0 KV pool (see attn_oracle.c for the
    definition and the pool layout): out[r, h] = softmax(q[r, h] . K^T / sqrt(128)) V over the
    first row_len[r] tokens of agent row_agent[r], K and V of KV head h // (H / kv_heads).
    Returns out and S = sum_t p_t |v_t| in double, both [rows, H, 128].

    pool: uint8, records of 17,408 bytes, (page P, head g) at (P * kv_heads + g) * 17408;
    page_table: int32 [agents, max_pages]; q: float16 [rows, H, 128]."""
    pool = np.ascontiguousarray(pool, dtype=np.uint8)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    assert pt.ndim == 2
    q = np.ascontiguousarray(q, dtype=np.float16)
    assert q.ndim == 3 and q.shape[2] == ATTN_D
    rows, heads = q.shape[0], q.shape[1]
    ra = np.ascontiguousarray(row_agent, dtype=np.int32)
    rl = np.ascontiguousarray(row_len, dtype=np.int32)
    assert ra.shape == (rows,) and rl.shape == (rows,)
    assert np.all(pt >= 0) and (pt.max(initial=0) + 1) * kv_heads * ATTN_RECORD_BYTES <= pool.size
    out = np.empty((rows, heads, ATTN_D))
    s = np.empty((rows, heads, ATTN_D))
    rc = _load().oracle_attn(pool.ctypes.data, pt.ctypes.data, pt.shape[1], q.view(np.uint16).ctypes.data,
                             ra.ctypes.data, rl.ctypes.data, rows, heads, kv_heads, out.ctypes.data,
                             s.ctypes.data, nthreads)
    if rc != 0:
        raise RuntimeError("oracle_attn failed")
    return out, s


def kv_value(record: np.ndarray, which: int, slot: int, d: int) -> float:
    """Element d of K (which 0) or V (which 1) of token `slot` of one 17,408-byte record."""
    r = np.ascontiguousarray(record, dtype=np.uint8).ravel()
    assert r.size == ATTN_RECORD_BYTES
    return float(_load().oracle_kv(r.ctypes.data, which, slot, d))
