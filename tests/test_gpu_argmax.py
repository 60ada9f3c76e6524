"""Greedy verification fused into the matmul (qmm_run_argmax), through the C ABI.

The kernel's argmax must be exactly the argmax of its own y (same arithmetic: the value's
bits equal, the lowest column among equal maxima), and a valid argmax of the oracle's exact
products within the tolerance: the chosen column's logit is within the two bounds of the
oracle's largest logit, and the returned value within the bound of the oracle's value."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL_ABS, TOL_REL, make, run, torch_cuda

pytestmark = pytest.mark.gpu


def run_argmax(q, x: np.ndarray, m: int | None = None):
    torch = torch_cuda()
    m = x.shape[0] if m is None else m
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.float16)
    idx = torch.full((max(m, 1),), -7, dtype=torch.int32, device="cuda")
    val = torch.full((max(m, 1),), float("nan"), dtype=torch.float32, device="cuda")
    q.run_argmax(xd, idx, val, m)
    torch.cuda.synchronize()
    return idx.cpu().numpy()[:m], val.cpu().numpy()[:m]


def check_against_own_run(q, x, idx, val):
    y = run(q, x)
    ref_idx = np.argmax(y, axis=1)
    assert np.array_equal(idx, ref_idx)
    assert np.array_equal(val.view(np.uint32), y[np.arange(len(idx)), ref_idx].view(np.uint32))


def check_against_oracle(blocks, x, idx, val):
    y_ref, s_ref = oracle.qmm(blocks, x)
    bound = TOL_REL * s_ref + TOL_ABS
    ref_idx, ref_val = oracle.argmax_rows(y_ref)
    rows = np.arange(len(idx))
    assert np.all(y_ref[rows, idx] + bound[rows, idx] >= ref_val - bound[rows, ref_idx])
    assert np.all(np.abs(val - y_ref[rows, idx]) <= bound[rows, idx])


CASES = [(20000, 1024, 1), (20000, 1024, 12), (3001, 2048, 5), (4096, 512, 16)]


@pytest.mark.parametrize("n,k,m", CASES, ids=[f"{n}x{k}-m{m}" for n, k, m in CASES])
def test_argmax_matches_own_run_and_oracle(n, k, m, backend):
    blocks = synth.q4k_matrix(n, k, seed=0, tensor_id=900 + m)
    x = synth.x_f16(m, k, seed=0, tensor_id=1900 + m)
    q = make(blocks, m_max=m, backend=backend)
    idx, val = run_argmax(q, x)
    check_against_own_run(q, x, idx, val)
    check_against_oracle(blocks, x, idx, val)


@pytest.mark.parametrize("m", [24, 40, 64, 100])
def test_argmax_wide_and_chunked(m, backend):
    """More rows than one launch takes (16 for mma.sync, 64 for tcgen05) run as chunks."""
    if backend == 1 and m > 24:
        pytest.skip("mma.sync covers the chunked case with 24 rows")
    n, k = 6000, 768
    blocks = synth.q4k_matrix(n, k, seed=1, tensor_id=950 + m)
    x = synth.x_f16(m, k, seed=1, tensor_id=1950 + m)
    q = make(blocks, m_max=m, backend=backend)
    idx, val = run_argmax(q, x)
    check_against_own_run(q, x, idx, val)
    check_against_oracle(blocks, x, idx, val)


def test_argmax_lm_head_rows_outliers(backend):
    """The lm_head shape (151936 x 5120) at M = 12 with outlier activations; the oracle
    checks the chosen columns and the true maxima on a sample of columns around them."""
    mat = synth.LM_HEAD
    m = 12
    blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
    x = synth.x_f16(m, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id, outlier_p=0.01)
    q = make(blocks, m_max=16, backend=backend)
    idx, val = run_argmax(q, x)
    check_against_own_run(q, x, idx, val)
    # the oracle on the chosen columns and on the kernel's runner-up candidates
    y = run(q, x)
    cols = np.unique(np.concatenate([idx, np.argsort(-y, axis=1)[:, :8].ravel()]))
    y_ref, s_ref = oracle.qmm(blocks[cols], x)
    bound = TOL_REL * s_ref + TOL_ABS
    pos = {c: i for i, c in enumerate(cols)}
    for r in range(m):
        i = pos[idx[r]]
        assert abs(val[r] - y_ref[r, i]) <= bound[r, i]
        assert np.all(y_ref[r, i] + bound[r, i] >= y_ref[r] - bound[r])


def test_argmax_ties_pick_the_lower_row(backend):
    """Two rows of one tile with identical blocks give bit-identical logits; when they are the
    largest, the lower row is returned."""
    n, k, m = 300, 512, 4
    blocks = synth.q4k_matrix(n, k, seed=2, tensor_id=960)
    x = synth.x_f16(m, k, seed=2, tensor_id=1960)
    y_ref, _ = oracle.qmm(blocks, x)
    r1 = int(np.argmax(y_ref[0]))
    r2 = r1 + 1 if (r1 + 1) % 128 != 0 and r1 + 1 < n else r1 - 1
    blocks[r2] = blocks[r1]
    q = make(blocks, m_max=m, backend=backend)
    idx, val = run_argmax(q, x)
    check_against_own_run(q, x, idx, val)
    y = run(q, x)
    assert y[0, r1] == y[0, r2]
    assert idx[0] == min(r1, r2)


def test_argmax_repeated_calls_reset_state(backend):
    """Consecutive calls on one handle with different activations each give their own
    argmax (the key buffer and counter are back to zero after every launch)."""
    n, k, m = 5000, 1024, 12
    blocks = synth.q4k_matrix(n, k, seed=3, tensor_id=970)
    q = make(blocks, m_max=m, backend=backend)
    for rep in range(4):
        x = synth.x_f16(m, k, seed=3 + rep, tensor_id=1970)
        idx, val = run_argmax(q, x)
        check_against_own_run(q, x, idx, val)
    assert q.error() == 0


def test_argmax_argument_errors(backend):
    from bit_weight_streaming_q4_gb300 import qmm as Q
    torch = torch_cuda()
    blocks = synth.q4k_matrix(256, 256, seed=4, tensor_id=980)
    q = make(blocks, m_max=4, backend=backend)
    lib = Q.load()
    x = torch.zeros((8, 256), dtype=torch.float16, device="cuda")
    idx = torch.zeros(8, dtype=torch.int32, device="cuda")
    val = torch.zeros(8, dtype=torch.float32, device="cuda")
    assert lib.qmm_run_argmax(q.handle, x.data_ptr(), 0, idx.data_ptr(), val.data_ptr(), None) == 0
    assert lib.qmm_run_argmax(q.handle, x.data_ptr(), 5, idx.data_ptr(), val.data_ptr(), None) == 2
    assert lib.qmm_run_argmax(q.handle, x.data_ptr(), -1, idx.data_ptr(), val.data_ptr(), None) == 1
    assert lib.qmm_run_argmax(q.handle, x.data_ptr(), 2, None, val.data_ptr(), None) == 1
    assert lib.qmm_run_argmax(q.handle, x.data_ptr(), 2, idx.data_ptr() + 2, val.data_ptr(), None) == 3
    assert lib.qmm_run_argmax(None, x.data_ptr(), 2, idx.data_ptr(), val.data_ptr(), None) == 7
