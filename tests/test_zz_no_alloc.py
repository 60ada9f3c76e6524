"""qmm_run_noalloc: the run for callers that cannot allocate device memory where they need
the matmul (a framework whose own memory pool owns the device, code that must not
synchronise the device, a plugin with a fixed memory budget).  It packs the raw Q4_K blocks
into the library's fixed scratch array and runs the mma.sync kernel with the same launch
shape as qmm_run on a handle of that kernel, so its result must agree with the oracle within
the tolerance and be bit-identical to qmm_run's, call after call (the scratch keeps the
previous call's contents, including tickets and packed weights of other shapes)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_parity, make, run, torch_cuda

pytestmark = pytest.mark.gpu


def _noalloc(blocks, x, n, k, m):
    from bit_weight_streaming_q4_gb300 import qmm as Q
    torch = torch_cuda()
    bd = torch.from_numpy(blocks.reshape(-1)).cuda()
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    yd = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    Q.run_noalloc(bd, n, k, xd, yd, m)
    torch.cuda.synchronize()
    return yd.cpu().numpy()


@pytest.mark.parametrize("n,k,m", [(4096, 4096, 12), (300, 1280, 5), (1000, 512, 19)])
def test_noalloc_matches_oracle_and_qmm_run_twice(n, k, m):
    blocks = synth.q4k_matrix(n, k, seed=8, tensor_id=n + k)
    x = synth.x_f16(m, k, seed=8, tensor_id=m)
    y_ref, s_ref = oracle.qmm(blocks, x)
    y_run = run(make(blocks, m_max=m, backend=1), x)
    for _ in range(2):
        y = _noalloc(blocks, x, n, k, m)
        assert_parity(y, y_ref, s_ref, "qmm_run_noalloc")
        assert np.array_equal(y.view(np.uint32), y_run.view(np.uint32))


def test_noalloc_larger_then_smaller_shape():
    """A large call (more tiles, tickets and workspace; 40 rows: three launches) followed by a
    smaller one: the second must not see anything the first left in the scratch."""
    shapes = [(9000, 2048, 40, 81), (700, 1536, 18, 82)]
    for n, k, m, tid in shapes:
        blocks = synth.q4k_matrix(n, k, seed=9, tensor_id=tid)
        x = synth.x_f16(m, k, seed=9, tensor_id=tid + 1000)
        y_ref, s_ref = oracle.qmm(blocks, x)
        y_run = run(make(blocks, m_max=m, backend=1), x)
        y = _noalloc(blocks, x, n, k, m)
        assert_parity(y, y_ref, s_ref, f"qmm_run_noalloc {n}x{k} m={m}")
        assert np.array_equal(y.view(np.uint32), y_run.view(np.uint32))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    from bit_weight_streaming_q4_gb300 import qmm as Q
    torch = torch_cuda()
    lib = Q.load()
    n, k = 34816, 5120   # 100 MB of Q4_K blocks: more than the fixed scratch holds
    bd = torch.zeros(n * k // 256 * 144, dtype=torch.uint8, device="cuda")
    xd = torch.zeros((4, k), dtype=torch.float16, device="cuda")
    yd = torch.zeros((4, n), dtype=torch.float32, device="cuda")
    st = Q.current_stream()
    assert lib.qmm_run_noalloc(bd.data_ptr(), n, k, xd.data_ptr(), 4, yd.data_ptr(), st) == 9
    assert lib.qmm_run_noalloc(None, n, k, xd.data_ptr(), 4, yd.data_ptr(), st) == 1
    assert lib.qmm_run_noalloc(bd.data_ptr(), 8, 300, xd.data_ptr(), 4, yd.data_ptr(), st) == 2
    assert b"scratch" in lib.qmm_status_str(9)
