"""qmm_run_noalloc: the run for callers that cannot allocate device memory where they need
the matmul (a framework whose own memory pool owns the device, code that must not
synchronise the device, a plugin with a fixed memory budget).  It packs the raw Q4_K blocks
into the library's fixed scratch array and must give what qmm_run gives on a handle, within
the parity tolerance, call after call (the scratch keeps the previous call's contents)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL_ABS, TOL_REL, make, run, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,k,m", [(4096, 4096, 12), (300, 1280, 5), (1000, 512, 19)])
def test_noalloc_matches_qmm_run_twice(n, k, m):
    from bit_weight_streaming_q4_gb300 import qmm as Q
    torch = torch_cuda()
    blocks = synth.q4k_matrix(n, k, seed=8, tensor_id=n + k)
    x = synth.x_f16(m, k, seed=8, tensor_id=m)
    _, s_ref = oracle.qmm(blocks, x)
    bound = TOL_REL * s_ref + TOL_ABS
    y_run = run(make(blocks, m_max=m, backend=1), x)
    bd = torch.from_numpy(blocks.reshape(-1)).cuda()
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    for _ in range(2):
        yd = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        Q.run_noalloc(bd, n, k, xd, yd, m)
        torch.cuda.synchronize()
        y = yd.cpu().numpy()
        assert np.all(np.isfinite(y))
        assert np.all(np.abs(y.astype(np.float64) - y_run) <= bound)


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
