"""Runs of two different handles in flight at once on two streams (the way a server overlaps
independent work).  No launch may wait for a CTA that cannot become resident: in the tcgen05
kernel's split-K reduction no CTA waits for another (a row tile's first piece adds the other
pieces' partials if they are all in, else the last piece to arrive does), and the mma.sync
kernel, whose reducer does wait for the other pieces,
is launched cooperatively (all its CTAs resident at once).  Twenty overlapped rounds must give
no device-side timeout, results bit-identical to the same runs issued alone, and parity with
the oracle."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_parity, make, run, torch_cuda

pytestmark = pytest.mark.gpu


def test_two_handles_on_two_streams(backend):
    torch = torch_cuda()
    m = 12
    shapes = [(34816 // 4, 5120, 70), (5120, 17408 // 2, 71)]  # gate_up- and down-like halves
    qs, xs, refs, alone = [], [], [], []
    for n, k, tid in shapes:
        blocks = synth.q4k_matrix(n, k, seed=3, tensor_id=tid)
        x = synth.x_f16(m, k, seed=3, tensor_id=1000 + tid)
        q = make(blocks, m_max=16, backend=backend)
        qs.append(q)
        xs.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16))
        refs.append(oracle.qmm(blocks, x))
        alone.append(run(q, x))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    rounds = 20
    outs = [[torch.full((m, q.n), float("nan"), dtype=torch.float32, device="cuda") for _ in range(rounds)]
            for q in qs]
    torch.cuda.synchronize()
    for r in range(rounds):
        for i in (0, 1):
            with torch.cuda.stream(streams[i]):
                qs[i].run(xs[i], outs[i][r], m, stream=streams[i].cuda_stream)
    torch.cuda.synchronize()
    for i, q in enumerate(qs):
        assert q.error() == 0
        y_ref, s_ref = refs[i]
        assert_parity(outs[i][0].cpu().numpy(), y_ref, s_ref, f"handle {i}")
        for r in range(rounds):
            got = outs[i][r].cpu().numpy()
            assert np.array_equal(got.view(np.uint32), alone[i].view(np.uint32)), (i, r)
