"""The decode step.  Dependent steps (a CUDA graph of runs linked by programmatic dependent
launch) give results bit-identical to the same runs issued one by one and really wait for a
run's output before the next run reads it.  Independent steps of mma.sync handles (one
persistent kernel, stream-K over all matrices) agree with the oracle within the tolerance, and
each row's bits do not depend on M; matrices too small to give every CTA a piece included."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_parity, make, torch_cuda

pytestmark = pytest.mark.gpu

MATS = [synth.Matrix("a", 512, 1280, 1), synth.Matrix("b", 1280, 768, 2),
        synth.Matrix("c", 96, 2048, 3), synth.Matrix("d", 3000, 512, 4),
        synth.Matrix("e", 4096, 4096, 5), synth.Matrix("f", 300, 256, 6)]


def _setup(backend, m, mats, m_max=None):
    torch = torch_cuda()
    qs, xs, ys, refs = [], [], [], []
    for mat in mats:
        blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
        x = synth.x_f16(m, mat.k, seed=0, tensor_id=1000 + mat.tensor_id)
        refs.append(oracle.qmm(blocks, x))
        qs.append(make(blocks, m_max=m_max or m, backend=backend))
        xs.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16))
        ys.append(torch.zeros((m, mat.n), dtype=torch.float32, device="cuda"))
    return qs, xs, ys, refs


@pytest.mark.parametrize("flags", [0, 2, 3, 4], ids=["dependent", "graph", "graph_independent", "persistent_dependent"])
def test_graph_step_matches_individual_runs(backend, flags):
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    m = 12
    qs, xs, ys, refs = _setup(backend, m, MATS)
    single = []
    for q, x, y in zip(qs, xs, ys):
        q.run(x, y, m)
        torch.cuda.synchronize()
        single.append(y.cpu().numpy().copy())
        y.zero_()
    step = Step(qs, xs, ys, m, flags=flags)
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


@pytest.mark.parametrize("m", [1, 5, 12, 16])
def test_independent_step_parity_and_repeatability(backend, m):
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    qs, xs, ys, refs = _setup(backend, m, MATS)
    step = Step(qs, xs, ys, m, flags=1)
    first = None
    for rep in range(3):
        for y in ys:
            y.fill_(float("nan"))
        step.launch()
        torch.cuda.synchronize()
        got = [y.cpu().numpy().copy() for y in ys]
        for g, (y_ref, s_ref), mat in zip(got, refs, MATS):
            assert_parity(g, y_ref, s_ref, mat.name)
        if first is None:
            first = got
        else:
            for a, b in zip(first, got):
                assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    step.close()


@pytest.mark.parametrize("backend_ms", [(1, (16, 9, 3)), (2, (64, 40, 17, 5)), (2, (128, 100, 65, 64, 17))],
                         ids=["mma_sync", "tcgen05", "tcgen05-wide"])
def test_independent_step_rows_do_not_depend_on_m(backend_ms):
    """The persistent step's rows are bit-identical whatever the number of rows of the step,
    including steps of more than 64 rows, whose activation sums come from a pre-pass over all
    the step's matrices."""
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    be, ms = backend_ms
    qs, xs, ys, refs = _setup(be, ms[0], MATS)
    outs = {}
    for m in ms:
        step = Step(qs, xs, ys, m, flags=1)
        for y in ys:
            y.fill_(float("nan"))
        step.launch()
        torch.cuda.synchronize()
        outs[m] = [y.cpu().numpy()[:m].copy() for y in ys]
        step.close()
    for (y_ref, s_ref), got, mat in zip(refs, outs[ms[0]], MATS):
        assert_parity(got, y_ref, s_ref, mat.name)
    for m in ms[1:]:
        for a, b in zip(outs[ms[0]], outs[m]):
            assert np.array_equal(a[:m].view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("be_m", [(1, 1), (1, 8), (1, 16), (2, 24), (2, 64), (2, 100)],
                         ids=["mma_sync-1", "mma_sync-8", "mma_sync-16", "tcgen05-24", "tcgen05-64", "tcgen05-100"])
def test_persistent_step_many_small_matrices(be_m):
    """Forty matrices, most smaller than one unit per CTA, in one persistent launch: pieces of
    one or two units, row tiles that only one of the tensor-core issuers touches."""
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    be, m = be_m
    rng = np.random.default_rng(5)
    mats = [synth.Matrix(f"s{i}", int(rng.integers(1, 2000)), 256 * int(rng.integers(1, 12)), 100 + i)
            for i in range(40)]
    qs, xs, ys, refs = _setup(be, m, mats)
    step = Step(qs, xs, ys, m, flags=1)
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
    step = Step([q1, q2], [x1, x2], [y1, y2], m)
    for _ in range(5):
        y1.copy_(torch.from_numpy(ones))
        y2.fill_(float("nan"))
        torch.cuda.synchronize()
        step.launch()
        torch.cuda.synchronize()
        assert np.all(y1.cpu().numpy() == 0.0)
        assert np.all(y2.cpu().numpy() == 0.0)
    step.close()


def test_persistent_step_rejects_repeated_handle():
    from bit_weight_streaming_q4_gb300 import QmmError, Step
    torch = torch_cuda()
    b = synth.q4k_matrix(256, 512, seed=0, tensor_id=7)
    q = make(b, m_max=4, backend=1)
    x = torch.zeros((4, 512), dtype=torch.float16, device="cuda")
    y = torch.zeros((4, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(QmmError):
        Step([q, q], [x, x], [y, y], 4, flags=1)
    Step([q, q], [x, x], [y, y], 4).close()   # the graph runs them one after the other


@pytest.mark.parametrize("m", [20, 32, 64])
def test_tcgen05_step_sustained_launches(m):
    """Forty back-to-back launches of a decode-sized persistent tcgen05 step (two layers of the
    27B shapes and the lm_head, 1.4 GB of weights): no wait runs out and every launch gives
    the first launch's bits.  The buffer handshakes only race under sustained load."""
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    mats = synth.stack(2)
    qs, xs, xs_host, ys = [], [], [], []
    for mat in mats:
        blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
        qs.append(make(blocks, m_max=m, backend=2))
        del blocks
        x = synth.x_f16(m, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
        xs_host.append(x)
        xs.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16))
        ys.append(torch.zeros((m, mat.n), dtype=torch.float32, device="cuda"))
    step = Step(qs, xs, ys, m, flags=1)
    step.launch()
    torch.cuda.synchronize()
    first = [y.cpu().numpy().copy() for y in ys]
    for rep in range(4):
        for _ in range(10):
            step.launch()
        torch.cuda.synchronize()
        for a, y, mat in zip(first, ys, mats):
            assert np.array_equal(a.view(np.uint32), y.cpu().numpy().view(np.uint32)), (rep, mat.name)
    assert all(q.error() == 0 for q in qs)
    step.close()
    # three sampled output rows of each matrix checked against the oracle
    for mat, a, x in zip(mats, first, xs_host):
        rows = np.array([0, mat.n // 2, mat.n - 1])
        blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id, rows=rows)
        y_ref, s_ref = oracle.qmm(blocks, x)
        assert_parity(a[:, rows], y_ref, s_ref, mat.name)


@pytest.mark.parametrize("m", [8, 64])
def test_tcgen05_dependent_step_reads_previous_output(m):
    """The persistent dependent step of the tensor-core backend really waits for run 1's
    output before run 2 loads it: run 2's activations alias run 1's output buffer, which run 1
    overwrites with exact zeros (over fp16 ones left there before every launch)."""
    from bit_weight_streaming_q4_gb300 import Step
    from bit_weight_streaming_q4_gb300.qmm import STEP_PERSISTENT
    torch = torch_cuda()
    n1, k1 = 2560, 4096
    k2, n2 = 2 * n1, 1024                     # x2 [m, 2 n1] fp16 is the bytes of y1 [m, n1] fp32
    b1 = synth.q4k_matrix(n1, k1, seed=1, tensor_id=52)
    b2 = synth.q4k_matrix(n2, k2, seed=1, tensor_id=53)
    q1, q2 = make(b1, m_max=m, backend=2), make(b2, m_max=m, backend=2)
    x1 = torch.zeros((m, k1), dtype=torch.float16, device="cuda")      # y1 = 0 exactly
    y1 = torch.empty((m, n1), dtype=torch.float32, device="cuda")
    x2 = y1.view(torch.float16)                                         # [m, 2 n1]
    y2 = torch.empty((m, n2), dtype=torch.float32, device="cuda")
    ones = np.full((m, 2 * n1), 1.0, dtype=np.float16).view(np.float32)
    step = Step([q1, q2], [x1, x2], [y1, y2], m, flags=STEP_PERSISTENT)
    for _ in range(5):
        y1.copy_(torch.from_numpy(ones))
        y2.fill_(float("nan"))
        torch.cuda.synchronize()
        step.launch()
        torch.cuda.synchronize()
        assert np.all(y1.cpu().numpy() == 0.0)
        assert np.all(y2.cpu().numpy() == 0.0)
    assert q1.error() == 0 and q2.error() == 0
    step.close()


def test_tcgen05_dependent_chain_with_repeated_handle():
    """A chain a -> b -> a -> b in one dependent step (a handle may appear more than once):
    each run reads the previous run's output buffer as its activations, so the step must
    match the same runs issued one by one, bit for bit, launch after launch."""
    from bit_weight_streaming_q4_gb300 import Step
    from bit_weight_streaming_q4_gb300.qmm import STEP_PERSISTENT
    torch = torch_cuda()
    m, n, k = 12, 2048, 4096
    ba = synth.q4k_matrix(n, k, seed=4, tensor_id=54)
    bb = synth.q4k_matrix(n, k, seed=4, tensor_id=55)
    qa, qb = make(ba, m_max=m, backend=2), make(bb, m_max=m, backend=2)
    # run i + 1's activations are the bytes of run i's output: y_i fp32 [m, n] is x fp16 [m, k]
    bufs = [torch.zeros((m, n), dtype=torch.float32, device="cuda") for _ in range(4)]
    x0 = torch.from_numpy(synth.x_f16(m, k, seed=4, tensor_id=1054).view(np.int16)).cuda().view(torch.float16)
    xs = [x0] + [bufs[i].view(torch.float16) for i in range(3)]
    qs = [qa, qb, qa, qb]
    # the same runs one by one (each after the previous one has finished)
    for q, x, y in zip(qs, xs, bufs):
        q.run(x, y, m)
        torch.cuda.synchronize()
    alone = [y.cpu().numpy().copy() for y in bufs]
    step = Step(qs, [x.data_ptr() for x in xs], bufs, m, flags=STEP_PERSISTENT)
    for _ in range(3):
        for y in bufs:
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        step.launch()
        torch.cuda.synchronize()
        for a, y in zip(alone, bufs):
            assert np.array_equal(a.view(np.uint32), y.cpu().numpy().view(np.uint32))
    assert qa.error() == 0 and qb.error() == 0
    step.close()


@pytest.mark.parametrize("m", [12, 64])
def test_tcgen05_dependent_step_sustained_launches(m):
    """Forty back-to-back launches of a dependent persistent step over two layers of the 27B
    shapes and the lm_head: the completion counters are back at zero for every launch (each
    launch gives the bits of the same runs issued one by one) and no wait runs out."""
    from bit_weight_streaming_q4_gb300 import Step
    from bit_weight_streaming_q4_gb300.qmm import STEP_PERSISTENT
    torch = torch_cuda()
    mats = synth.stack(2)
    qs, xs, ys = [], [], []
    for mat in mats:
        blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
        qs.append(make(blocks, m_max=m, backend=2))
        del blocks
        x = synth.x_f16(m, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
        xs.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16))
        ys.append(torch.zeros((m, mat.n), dtype=torch.float32, device="cuda"))
    alone = []
    for q, x, y in zip(qs, xs, ys):
        q.run(x, y, m)
        torch.cuda.synchronize()
        alone.append(y.cpu().numpy().copy())
    step = Step(qs, xs, ys, m, flags=STEP_PERSISTENT)
    for rep in range(4):
        for _ in range(10):
            step.launch()
        torch.cuda.synchronize()
        for a, y, mat in zip(alone, ys, mats):
            assert np.array_equal(a.view(np.uint32), y.cpu().numpy().view(np.uint32)), (rep, mat.name)
    assert all(q.error() == 0 for q in qs)
    step.close()


@pytest.mark.parametrize("m", [12, 64])
@pytest.mark.parametrize("layout", ["slab", "separate"])
@pytest.mark.parametrize("flags", [1, 0], ids=["independent", "dependent"])
def test_step_launch_host_matches_device_launch(backend, flags, layout, m):
    """qmm_step_launch_host: the activations from one host slab in step order, the outputs
    back to one host slab; bit-identical to the device launch with the caller's own copies,
    whether the device buffers form one slab (one copy each way) or are separate."""
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    if backend == 1 and m > 16:
        pytest.skip("mma.sync handles take at most 16 rows")
    blocks = [synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id) for mat in MATS]
    xh = [synth.x_f16(m, mat.k, seed=0, tensor_id=1000 + mat.tensor_id) for mat in MATS]
    qs = [make(b, m_max=m, backend=backend) for b in blocks]
    xsz = [m * mat.k for mat in MATS]
    ysz = [m * mat.n for mat in MATS]
    if layout == "slab":
        xd = torch.empty(sum(xsz), dtype=torch.float16, device="cuda")
        yd = torch.empty(sum(ysz), dtype=torch.float32, device="cuda")
        xs = [xd[a:a + n] for a, n in zip(np.cumsum([0] + xsz[:-1]), xsz)]
        ys = [yd[a:a + n] for a, n in zip(np.cumsum([0] + ysz[:-1]), ysz)]
    else:
        xs = [torch.empty(n, dtype=torch.float16, device="cuda") for n in xsz]
        ys = [torch.empty(n, dtype=torch.float32, device="cuda") for n in ysz]
    x_pin = torch.from_numpy(np.concatenate([x.reshape(-1) for x in xh]).view(np.int16)).view(torch.float16).pin_memory()
    y_pin = torch.full((sum(ysz),), float("nan"), dtype=torch.float32).pin_memory()
    step = Step(qs, xs, ys, m, flags=flags)
    # the device form: the caller's copies, then the launch
    for x, a in zip(xs, xh):
        x.copy_(torch.from_numpy(a.reshape(-1).view(np.int16)).view(torch.float16))
    step.launch()
    torch.cuda.synchronize()
    want = [y.cpu().numpy().copy() for y in ys]
    for y in ys:
        y.fill_(float("nan"))
    for x in xs:
        x.zero_()
    torch.cuda.synchronize()
    cin, out = torch.cuda.Stream(), torch.cuda.Stream()
    for split in (False, True, True, False):
        y_pin.fill_(float("nan"))
        step.launch_host(x_pin, y_pin, in_stream=cin.cuda_stream if split else None,
                         out_stream=out.cuda_stream if split else None)
        (out if split else torch.cuda.current_stream()).synchronize()
        got = y_pin.numpy()
        off = 0
        for w, n in zip(want, ysz):
            assert np.array_equal(got[off:off + n].view(np.uint32), w.view(np.uint32))
            off += n
    torch.cuda.synchronize()
    off = 0
    for b, x, mat, n in zip(blocks, xh, MATS, ysz):
        y_ref, s_ref = oracle.qmm(b, x)
        assert_parity(y_pin.numpy()[off:off + n].reshape(m, mat.n), y_ref, s_ref, mat.name)
        off += n
    step.close()


def test_two_host_steps_overlap_copies_and_stay_exact():
    """Two steps over two sets of device buffers, launched alternately on one stream with
    their copies in and out on two others: every call's host outputs equal the device
    launch's, bit for bit (a step's copy-in waits for its last kernel, and its next kernel
    for its last copy-out)."""
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    m = 12
    blocks = [synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id) for mat in MATS]
    qs = [make(b, m_max=m, backend=1) for b in blocks]
    xsz = [m * mat.k for mat in MATS]
    ysz = [m * mat.n for mat in MATS]
    xs2 = [[torch.empty(n, dtype=torch.float16, device="cuda") for n in xsz] for _ in range(2)]
    ys2 = [[torch.empty(n, dtype=torch.float32, device="cuda") for n in ysz] for _ in range(2)]
    steps = [Step(qs, xs2[b], ys2[b], m, flags=1) for b in range(2)]
    inputs = []
    for it in range(4):   # a different x slab per call, so that a stale copy would show
        xh = [synth.x_f16(m, mat.k, seed=it, tensor_id=1000 + mat.tensor_id) for mat in MATS]
        inputs.append(torch.from_numpy(np.concatenate([x.reshape(-1) for x in xh]).view(np.int16))
                      .view(torch.float16).pin_memory())
    # expected: each input through the device launch of step 0
    want = []
    for xp in inputs:
        off = 0
        for x, n in zip(xs2[0], xsz):
            x.copy_(xp[off:off + n])
            off += n
        steps[0].launch()
        torch.cuda.synchronize()
        want.append(np.concatenate([y.cpu().numpy() for y in ys2[0]]))
    outs = [torch.full((sum(ysz),), float("nan"), dtype=torch.float32).pin_memory() for _ in inputs]
    cin, out = torch.cuda.Stream(), torch.cuda.Stream()
    for it, (xp, yp) in enumerate(zip(inputs, outs)):
        steps[it % 2].launch_host(xp, yp, in_stream=cin.cuda_stream, out_stream=out.cuda_stream)
    out.synchronize()
    torch.cuda.synchronize()
    for w, yp in zip(want, outs):
        assert np.array_equal(yp.numpy().view(np.uint32), w.view(np.uint32))
    for st in steps:
        st.close()


def test_host_step_with_aliased_activations_reads_the_run_output():
    """A dependent step whose x_2 is the bytes of y_1, launched from host buffers: x_2's copied
    bytes (fp16 ones) are replaced by run 1's output (exact zeros) before run 2 reads them, as
    the host-buffer call documents, so y_2 = 0."""
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    m, n1, k1 = 8, 2560, 4096
    k2, n2 = 2 * n1, 1024
    b1 = synth.q4k_matrix(n1, k1, seed=1, tensor_id=50)
    b2 = synth.q4k_matrix(n2, k2, seed=1, tensor_id=51)
    q1, q2 = make(b1, m_max=m, backend=1), make(b2, m_max=m, backend=1)
    x1 = torch.empty((m, k1), dtype=torch.float16, device="cuda")
    y1 = torch.empty((m, n1), dtype=torch.float32, device="cuda")
    x2 = y1.view(torch.float16)
    y2 = torch.empty((m, n2), dtype=torch.float32, device="cuda")
    step = Step([q1, q2], [x1, x2], [y1, y2], m)
    x_host = torch.cat([torch.zeros(m * k1, dtype=torch.float16),
                        torch.ones(m * k2, dtype=torch.float16)]).pin_memory()
    y_host = torch.full((m * (n1 + n2),), float("nan"), dtype=torch.float32).pin_memory()
    for _ in range(3):
        step.launch_host(x_host, y_host)
        torch.cuda.synchronize()
        assert np.all(y_host.numpy() == 0.0)
        y_host.fill_(float("nan"))
    step.close()
