"""The rare path of the tcgen05 kernel's split-K sum, forced on every split row tile.

A row tile cut between CTAs pa..pb is normally finished by pa, which reaches it last and
finds the other pieces' partials published.  If some piece starts late (another kernel holds
SMs), pa parks its own partial and the last piece to arrive adds them all up in the same
piece order.  A handle created with QMM_SPLITK_PARK=1 takes that path on every split tile.
Its results must equal a normal handle's bit for bit (runs of 16, 64 and 128-row tiles, the
fused argmax, a one-launch step over several matrices) and agree with the oracle."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_parity, make, run, torch_cuda

pytestmark = pytest.mark.gpu


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def _pair(blocks, monkeypatch, **kw):
    normal = make(blocks, backend=2, **kw)
    with monkeypatch.context() as mp:
        mp.setenv("QMM_SPLITK_PARK", "1")
        parked = make(blocks, backend=2, **kw)
    return normal, parked


@pytest.mark.parametrize("m", [12, 64, 100])
def test_parked_sum_equals_direct_sum(monkeypatch, m):
    n, k = 8704, 5120  # 68 row tiles of 20 units over the CTAs: most tiles are cut
    blocks = synth.q4k_matrix(n, k, seed=4, tensor_id=80)
    x = synth.x_f16(m, k, seed=4, tensor_id=1080)
    normal, parked = _pair(blocks, monkeypatch, m_max=128)
    want = run(normal, x)
    for _ in range(3):
        assert np.array_equal(bits(run(parked, x)), bits(want))
    assert parked.error() == 0
    y_ref, s_ref = oracle.qmm(blocks, x)
    assert_parity(want, y_ref, s_ref, "parked")


def test_parked_argmax(monkeypatch):
    torch = torch_cuda()
    n, k, m = 6144, 4096, 12
    blocks = synth.q4k_matrix(n, k, seed=5, tensor_id=81)
    x = synth.x_f16(m, k, seed=5, tensor_id=1081)
    normal, parked = _pair(blocks, monkeypatch, m_max=16)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    out = []
    for q in (normal, parked):
        idx = torch.full((m,), -1, dtype=torch.int32, device="cuda")
        val = torch.full((m,), float("nan"), dtype=torch.float32, device="cuda")
        q.run_argmax(xd, idx, val, m)
        torch.cuda.synchronize()
        out.append((idx.cpu().numpy(), val.cpu().numpy()))
    assert np.array_equal(out[0][0], out[1][0])
    assert np.array_equal(bits(out[0][1]), bits(out[1][1]))


def test_parked_persistent_step(monkeypatch):
    from bit_weight_streaming_q4_gb300 import Step
    from bit_weight_streaming_q4_gb300.qmm import STEP_INDEPENDENT
    torch = torch_cuda()
    m = 24
    shapes = [(1280, 2048, 82), (5120, 6144, 83), (3000, 1536, 84), (640, 4096, 85)]
    results = []
    for park in (False, True):
        qs, xs, ys = [], [], []
        for n, k, tid in shapes:
            blocks = synth.q4k_matrix(n, k, seed=6, tensor_id=tid)
            x = synth.x_f16(m, k, seed=6, tensor_id=1000 + tid)
            with monkeypatch.context() as mp:
                if park:
                    mp.setenv("QMM_SPLITK_PARK", "1")
                qs.append(make(blocks, m_max=m, backend=2))
            xs.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16))
            ys.append(torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda"))
        step = Step(qs, xs, ys, m, flags=STEP_INDEPENDENT)
        step.launch()
        step.launch()
        torch.cuda.synchronize()
        results.append([y.cpu().numpy() for y in ys])
        step.close()
    for a, b in zip(*results):
        assert np.array_equal(bits(a), bits(b))
