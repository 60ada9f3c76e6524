"""Helpers for the GPU tests: device buffers through torch, runs through the C ABI,
and the element-wise tolerance check against the oracle."""
from __future__ import annotations

import numpy as np

TOL_REL = 2e-3
TOL_ABS = 1e-6


def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "GPU test run without a GPU"
    return torch


def to_device_blocks(blocks: np.ndarray):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(blocks).reshape(-1)).cuda()


def make(blocks: np.ndarray, m_max: int = 16, device_blocks: bool = True, **kw):
    """A handle for [N, blocks per row, block bytes] blocks (144: Q4_K, 210: Q6_K, 34: Q8_0;
    pass format= for the latter two)."""
    from bit_weight_streaming_q4_gb300 import Qmm
    n, kb, nbytes = blocks.shape
    per = 32 if nbytes == 34 else 256
    src = to_device_blocks(blocks) if device_blocks else np.ascontiguousarray(blocks)
    return Qmm(src, n, kb * per, m_max=m_max, **kw)


def run(q, x: np.ndarray, m: int | None = None) -> np.ndarray:
    torch = torch_cuda()
    m = x.shape[0] if m is None else m
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.float16)
    yd = torch.full((max(m, 1), q.n), float("nan"), dtype=torch.float32, device="cuda")
    q.run(xd, yd, m)
    torch.cuda.synchronize()
    return yd.cpu().numpy()[:m]


def assert_parity(y: np.ndarray, y_ref: np.ndarray, s_ref: np.ndarray, what: str = ""):
    """|y - y_ref| <= 2e-3 * sum_k |w x| + 1e-6 for every element."""
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y.astype(np.float64) - y_ref)
    bound = TOL_REL * s_ref + TOL_ABS
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        where = ""
        if bad.ndim == 2:
            # which activation rows (tokens) and output columns, to tell a row tile, a lane
            # group or a chunk of tokens apart
            toks = np.where(bad.any(axis=1))[0]
            cols = np.where(bad.any(axis=0))[0]
            where = (f"; tokens {toks.min()}..{toks.max()} ({toks.size}), output columns "
                     f"{cols.min()}..{cols.max()} ({cols.size}): {cols[:48].tolist()}")
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: got {y[i]!r}, want {y_ref[i]!r}, bound {bound[i]!r}{where}")
    return float((err / bound).max()) if err.size else 0.0
