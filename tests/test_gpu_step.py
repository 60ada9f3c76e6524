"""The decode step (one persistent kernel over all matrices for mma.sync handles, or a CUDA
graph of runs linked by programmatic dependent launch) gives bit-identical results to the same
runs issued one by one, in dependent and independent mode, including matrices too small to
give every CTA a piece; and a dependent step really waits for a run's output before the next
run reads it."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_parity, make, torch_cuda

pytestmark = pytest.mark.gpu

MODES = {"dependent": 0, "independent": 1, "graph": 2, "graph_independent": 3,
         "persistent_dependent": 4, "persistent_independent": 5}


def _setup(backend, m, mats):
    torch = torch_cuda()
    qs, xs, ys, refs = [], [], [], []
    for mat in mats:
        blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
        x = synth.x_f16(m, mat.k, seed=0, tensor_id=1000 + mat.tensor_id)
        refs.append(oracle.qmm(blocks, x))
        qs.append(make(blocks, m_max=m, backend=backend))
        xs.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16))
        ys.append(torch.zeros((m, mat.n), dtype=torch.float32, device="cuda"))
    return qs, xs, ys, refs


@pytest.mark.parametrize("mode", list(MODES))
def test_step_matches_individual_runs(backend, mode):
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    mats = [synth.Matrix("a", 512, 1280, 1), synth.Matrix("b", 1280, 768, 2),
            synth.Matrix("c", 96, 2048, 3), synth.Matrix("d", 3000, 512, 4),
            synth.Matrix("e", 4096, 4096, 5), synth.Matrix("f", 300, 256, 6)]
    m = 12
    qs, xs, ys, refs = _setup(backend, m, mats)
    single = []
    for q, x, y in zip(qs, xs, ys):
        q.run(x, y, m)
        torch.cuda.synchronize()
        single.append(y.cpu().numpy().copy())
        y.zero_()
    step = Step(qs, xs, ys, m, flags=MODES[mode])
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


@pytest.mark.parametrize("m", [1, 8, 16])
def test_persistent_step_many_small_matrices(m):
    """Forty matrices, most smaller than one unit per CTA, in one persistent launch."""
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    rng = np.random.default_rng(5)
    mats = [synth.Matrix(f"s{i}", int(rng.integers(1, 2000)), 256 * int(rng.integers(1, 12)), 100 + i)
            for i in range(40)]
    qs, xs, ys, refs = _setup(1, m, mats)
    step = Step(qs, xs, ys, m, flags=4)
    for _ in range(2):
        step.launch()
        torch.cuda.synchronize()
        for y, (y_ref, s_ref), mat in zip(ys, refs, mats):
            assert_parity(y.cpu().numpy(), y_ref, s_ref, mat.name)
    step.close()


def test_dependent_step_reads_previous_output():
    """Run 2's activations alias run 1's output buffer.  Run 1 writes exact zeros over a
    buffer prefilled with fp16 ones; a dependent step must give run 2 the zeros (so y2 = 0),
    the same as issuing the runs one by one."""
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    m, n1, k1 = 8, 2560, 4096
    k2, n2 = 2 * n1, 1024                     # x2 [m, 2 n1] fp16 is the bytes of y1 [m, n1] fp32
    b1 = synth.q4k_matrix(n1, k1, seed=1, tensor_id=50)
    b2 = synth.q4k_matrix(n2, k2, seed=1, tensor_id=51)
    q1, q2 = make(b1, m_max=m, backend=1), make(b2, m_max=m, backend=1)
    x1 = torch.zeros((m, k1), dtype=torch.float16, device="cuda")      # y1 = 0 exactly
    y1 = torch.empty((m, n1), dtype=torch.float32, device="cuda")
    x2 = y1.view(torch.float16)                                         # [m, 2 n1]
    y2 = torch.empty((m, n2), dtype=torch.float32, device="cuda")
    ones = np.full((m, 2 * n1), 1.0, dtype=np.float16).view(np.float32)
    steps = [Step([q1, q2], [x1, x2], [y1, y2], m, flags=f) for f in (0, 4)]
    for step in steps * 3:
        y1.copy_(torch.from_numpy(ones))
        y2.fill_(float("nan"))
        torch.cuda.synchronize()
        step.launch()
        torch.cuda.synchronize()
        assert np.all(y1.cpu().numpy() == 0.0)
        assert np.all(y2.cpu().numpy() == 0.0)
    for step in steps:
        step.close()


def test_persistent_step_rejects_repeated_handle():
    from bit_weight_streaming_q4_gb300 import QmmError, Step
    torch = torch_cuda()
    b = synth.q4k_matrix(256, 512, seed=0, tensor_id=7)
    q = make(b, m_max=4, backend=1)
    x = torch.zeros((4, 512), dtype=torch.float16, device="cuda")
    y = torch.zeros((4, 256), dtype=torch.float32, device="cuda")
    for flags in (1, 4):
        with pytest.raises(QmmError):
            Step([q, q], [x, x], [y, y], 4, flags=flags)
    Step([q, q], [x, x], [y, y], 4).close()   # the graph runs them one after the other
