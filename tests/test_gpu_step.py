"""The decode step (a CUDA graph of runs linked by programmatic dependent launch, or one
persistent kernel over all matrices) gives bit-identical results to the same runs issued one
by one, including matrices too small to give every CTA a piece."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_parity, make, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["graph", "persistent"])
def test_step_matches_individual_runs(backend, mode, monkeypatch):
    monkeypatch.setenv("QMM_STEP_MODE", mode)
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    mats = [synth.Matrix("a", 512, 1280, 1), synth.Matrix("b", 1280, 768, 2),
            synth.Matrix("c", 96, 2048, 3), synth.Matrix("d", 3000, 512, 4)]
    m = 12
    qs, xs, ys, refs = [], [], [], []
    for mat in mats:
        blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
        x = synth.x_f16(m, mat.k, seed=0, tensor_id=1000 + mat.tensor_id)
        refs.append(oracle.qmm(blocks, x))
        qs.append(make(blocks, m_max=m, backend=backend))
        xs.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16))
        ys.append(torch.zeros((m, mat.n), dtype=torch.float32, device="cuda"))
    single = []
    for q, x, y in zip(qs, xs, ys):
        q.run(x, y, m)
        torch.cuda.synchronize()
        single.append(y.cpu().numpy().copy())
        y.zero_()
    step = Step(qs, xs, ys, m)
    for _ in range(3):
        step.launch()
        torch.cuda.synchronize()
        for y, s, (y_ref, s_ref) in zip(ys, single, refs):
            got = y.cpu().numpy()
            assert np.array_equal(got.view(np.uint32), s.view(np.uint32))
            assert_parity(got, y_ref, s_ref, "step")
        for y in ys:
            y.zero_()
    step.close()
