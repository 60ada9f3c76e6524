"""The bounded-wait failure path, made to run on purpose without faulting or hanging the GPU.

Every wait between the kernels' own warps and CTAs gives up after a limit, sets the launch's
sticky error word and lets the kernel return (copies in flight land first, tensor memory is
released).  A handle created with wait_limit_us = 1 makes those waits run out: on a 94 MB
matrix (a launch of ~25 us) a CTA waits far longer than a microsecond for, e.g., the last row
tile of its piece to be finished.  The tests check that the
call returns, that the handle then reports QMM_ERR_DEVICE_TIMEOUT (status 6) and refuses
further runs, and that the GPU keeps answering: a fresh handle on the same device computes
the right product afterwards."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_parity, make, run, torch_cuda

pytestmark = pytest.mark.gpu

TIMEOUT = 6


def _inputs(n, k, m, tid):
    blocks = synth.q4k_matrix(n, k, seed=21, tensor_id=tid)
    x = synth.x_f16(m, k, seed=21, tensor_id=1000 + tid)
    return blocks, x


def test_short_wait_limit_is_reported_and_the_gpu_keeps_working(backend):
    from bit_weight_streaming_q4_gb300 import QmmError
    torch = torch_cuda()
    n, k, m = 32768, 5120, 12
    blocks, x = _inputs(n, k, m, 40)
    q = make(blocks, m_max=16, backend=backend, wait_limit_us=1)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    yd = torch.zeros((m, n), dtype=torch.float32, device="cuda")
    q.run(xd, yd, m)          # asynchronous: the launch itself is accepted
    torch.cuda.synchronize()  # ... and the kernel returns
    assert q.error() == TIMEOUT
    with pytest.raises(QmmError) as e:
        q.run(xd, yd, m)
    assert e.value.status == TIMEOUT
    q.close()
    # the context and the GPU are fine: a handle with the default limit gets the right answer
    y_ref, s_ref = oracle.qmm(blocks, x)
    fresh = make(blocks, m_max=16, backend=backend)
    assert_parity(run(fresh, x), y_ref, s_ref, "after a timed-out launch")
    assert fresh.error() == 0


def test_short_wait_limit_in_a_persistent_step(backend):
    """The same through a one-launch independent step of several matrices: the step's own
    error word reports the timeout, and the step refuses to launch again."""
    from bit_weight_streaming_q4_gb300 import QmmError, Step
    from bit_weight_streaming_q4_gb300.qmm import STEP_INDEPENDENT
    torch = torch_cuda()
    m = 8
    shapes = [(1280, 2048, 50), (16384, 5120, 51), (640, 4096, 52)]
    qs, xs, ys, data = [], [], [], []
    for n, k, tid in shapes:
        blocks, x = _inputs(n, k, m, tid)
        data.append((blocks, x))
        qs.append(make(blocks, m_max=m, backend=backend, wait_limit_us=1))
        xs.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16))
        ys.append(torch.zeros((m, n), dtype=torch.float32, device="cuda"))
    step = Step(qs, xs, ys, m, flags=STEP_INDEPENDENT)
    step.launch()
    torch.cuda.synchronize()
    with pytest.raises(QmmError) as e:
        step.launch()
    assert e.value.status == TIMEOUT
    step.close()
    for q in qs:
        q.close()
    # fresh handles on the same device compute every product correctly
    for (blocks, x) in data:
        y_ref, s_ref = oracle.qmm(blocks, x)
        assert_parity(run(make(blocks, m_max=m, backend=backend), x), y_ref, s_ref, "fresh handle")


def test_wait_limit_option_is_validated():
    from bit_weight_streaming_q4_gb300 import QmmError
    blocks, _ = _inputs(256, 256, 1, 60)
    with pytest.raises(QmmError) as e:
        make(blocks, m_max=4, wait_limit_us=-1)
    assert e.value.status == 1
