"""The full synthetic 27B-shaped decode stack at its real size: 64 layers x {qkv 5120->8192,
o 6144->5120, gate_up 5120->34816, down 17408->5120} + lm_head 5120->151936 (257 Q4_K
matrices, 12.71 GB), every matrix with its own activations, run as the one-launch
independent step at M = 12 (4 streams x (1 token + 2 drafts)) and M = 64 (8 streams x
(1 + 7 drafts)).  Sampled output columns of every one of the 257 matrices are checked
against the oracle (all M rows of each sampled column), and a second launch must repeat the
first bit for bit."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL_ABS, TOL_REL, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m", [12, 64])
def test_full_stack_step(m):
    from bit_weight_streaming_q4_gb300 import Qmm, Step
    from bit_weight_streaming_q4_gb300.qmm import STEP_INDEPENDENT
    torch = torch_cuda()
    mats = synth.stack(synth.LAYERS)
    assert len(mats) == 257
    qs, xs, ys, xh = [], [], [], []
    for mat in mats:
        blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
        dev = torch.from_numpy(blocks.reshape(-1)).cuda()
        qs.append(Qmm(dev, mat.n, mat.k, m_max=m))
        del dev, blocks
        x = synth.x_f16(m, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
        xh.append(x)
        xs.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16))
        ys.append(torch.full((m, mat.n), float("nan"), dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    step = Step(qs, xs, ys, m, flags=STEP_INDEPENDENT)
    step.launch()
    torch.cuda.synchronize()
    first = [y.cpu().numpy() for y in ys]
    step.launch()
    torch.cuda.synchronize()
    rng = np.random.default_rng(m)
    worst, checked = 0.0, 0
    for i, mat in enumerate(mats):
        got = ys[i].cpu().numpy()
        assert np.array_equal(got.view(np.uint32), first[i].view(np.uint32)), mat.name
        # the matrix's first and last output channel (tile edges) and one at random
        cols = np.unique(np.array([0, mat.n - 1, rng.integers(1, mat.n - 1)]))
        blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id, rows=cols)
        y_ref, s_ref = oracle.qmm(blocks, xh[i])
        sub = got[:, cols]
        assert np.all(np.isfinite(sub)), mat.name
        ratio = np.abs(sub.astype(np.float64) - y_ref) / (TOL_REL * s_ref + TOL_ABS)
        assert ratio.max() <= 1.0, (mat.name, float(ratio.max()))
        worst = max(worst, float(ratio.max()))
        checked += ratio.size
    assert checked >= 257 * 2 * m
    step.close()
    for q in qs:
        q.close()
