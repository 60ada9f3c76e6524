"""The other block formats (Q6_K, Q8_0) on the tcgen05 backend, element by element against
the oracle through the C ABI; hand-packed extreme blocks, unit vectors, M-independence of
rows, chunked runs, the persistent step and the fused argmax."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TOL_ABS, TOL_REL, assert_parity, make, run, torch_cuda
from q4k_pack import pack_q6_k, pack_q8_0

pytestmark = pytest.mark.gpu

Q4K, Q6K, Q80 = 0, 1, 2
FORMATS = {"Q6_K": (synth.Q6_K, Q6K), "Q8_0": (synth.Q8_0, Q80)}
CASES = [(4096, 4096, 1), (3001, 2048, 12), (1000, 768, 16), (2000, 1024, 40), (777, 1536, 64),
         (500, 512, 100)]


@pytest.fixture(params=sorted(FORMATS))
def fmt(request):
    return FORMATS[request.param]


@pytest.mark.parametrize("n,k,m", CASES, ids=[f"{n}x{k}-m{m}" for n, k, m in CASES])
def test_format_parity(fmt, n, k, m):
    f, code = fmt
    blocks = synth.fmt_matrix(f, n, k, seed=0, tensor_id=2000 + code * 100 + m)
    x = synth.x_f16(m, k, seed=0, tensor_id=3000 + m)
    y_ref, s_ref = oracle.qmm(blocks, x)
    q = make(blocks, m_max=m, format=code)
    assert q.info().backend == 2 and q.info().format == code
    assert q.info().weight_bytes == blocks.size
    assert_parity(run(q, x), y_ref, s_ref, f"fmt {code} {n}x{k} M={m}")


def test_format_outlier_activations(fmt):
    f, code = fmt
    n, k, m = 2048, 5120, 12
    blocks = synth.fmt_matrix(f, n, k, seed=1, tensor_id=2500 + code)
    x = synth.x_f16(m, k, seed=1, tensor_id=3500, outlier_p=0.01)
    y_ref, s_ref = oracle.qmm(blocks, x)
    assert_parity(run(make(blocks, m_max=m, format=code), x), y_ref, s_ref, "outliers")


def test_hand_packed_extremes():
    """Blocks at the ends of every field: Q8_0 quants -128 and 127 and d at the top of fp16
    weights' range used here; Q6_K quants 0 and 63, scales -128 and 127."""
    rng = np.random.default_rng(8)
    n, k = 256, 512
    q8 = np.zeros((n, k // 32, 34), dtype=np.uint8)
    for r in range(n):
        for b in range(k // 32):
            qs = rng.choice([-128, 127, -1, 0, 1], 32)
            q8[r, b] = pack_q8_0(int(rng.choice([0x2000, 0x1C00, 0x2400])), qs)
    q6 = np.zeros((n, k // 256, 210), dtype=np.uint8)
    for r in range(n):
        for b in range(k // 256):
            qs = rng.choice([0, 63, 31, 32, 33], 256)
            sc = rng.choice([-128, 127, 1, -1, 0], 16)
            q6[r, b] = pack_q6_k(int(rng.choice([0x1000, 0x0C00])), sc, qs)
    x = synth.x_f16(5, k, seed=2, tensor_id=3600)
    for blocks, code in ((q8, Q80), (q6, Q6K)):
        y_ref, s_ref = oracle.qmm(blocks, x)
        assert_parity(run(make(blocks, m_max=5, format=code), x), y_ref, s_ref, f"hand-packed {code}")


def test_unit_vectors_give_fp16_weights(fmt):
    """x = e_k returns column k of W rounded to fp16: exactly for Q8_0 (one rounding of d*q),
    within one fp16 ulp for Q6_K (d*sc split into two fp16 terms)."""
    f, code = fmt
    n, k = 300, 512
    blocks = synth.fmt_matrix(f, n, k, seed=3, tensor_id=2600 + code)
    w = oracle.dequant_matrix(blocks)
    q = make(blocks, m_max=8, format=code)
    cols = [0, 1, 31, 32, 255, 256, 300, 511]
    x = np.zeros((len(cols), k), dtype=np.float16)
    for i, c in enumerate(cols):
        x[i, c] = 1.0
    y = run(q, x)
    for i, c in enumerate(cols):
        want = w[:, c].astype(np.float16).astype(np.float64)
        if code == Q80:
            assert np.array_equal(y[i].astype(np.float64), want)
        else:
            ulp = np.spacing(np.abs(want).astype(np.float16)).astype(np.float64)
            assert np.all(np.abs(y[i] - w[:, c]) <= ulp)


def test_format_rows_do_not_depend_on_m(fmt):
    f, code = fmt
    n, k = 3000, 1024
    blocks = synth.fmt_matrix(f, n, k, seed=4, tensor_id=2700 + code)
    x = synth.x_f16(64, k, seed=4, tensor_id=3700)
    q = make(blocks, m_max=64, format=code)
    full = run(q, x)
    for m in (1, 5, 17, 33):
        assert np.array_equal(run(q, x[:m]).view(np.uint32), full[:m].view(np.uint32))


def test_format_persistent_step_and_mixed_step(fmt):
    """A persistent step over matrices of one format, and an independent step mixing it with
    Q4_K (one kernel cannot stream two formats, so that step runs as a graph of runs)."""
    from bit_weight_streaming_q4_gb300 import Step
    torch = torch_cuda()
    f, code = fmt
    m = 12
    shapes = [(1280, 1024), (512, 2048), (3000, 512), (96, 256)]
    qs, xs, ys, refs = [], [], [], []
    for i, (n, k) in enumerate(shapes):
        mixed_q4 = i == 1
        blocks = (synth.q4k_matrix(n, k, seed=5, tensor_id=2800 + i) if mixed_q4
                  else synth.fmt_matrix(f, n, k, seed=5, tensor_id=2800 + i))
        x = synth.x_f16(m, k, seed=5, tensor_id=3800 + i)
        refs.append(oracle.qmm(blocks, x))
        qs.append(make(blocks, m_max=16, backend=2, format=Q4K if mixed_q4 else code))
        xs.append(torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16))
        ys.append(torch.zeros((m, n), dtype=torch.float32, device="cuda"))
    for sel in ([0, 2, 3], [0, 1, 2, 3]):
        step = Step([qs[i] for i in sel], [xs[i] for i in sel], [ys[i] for i in sel], m, flags=1)
        for _ in range(2):
            for i in sel:
                ys[i].fill_(float("nan"))
            step.launch()
            torch.cuda.synchronize()
            for i in sel:
                assert_parity(ys[i].cpu().numpy(), *refs[i], f"step {sel} matrix {i}")
        step.close()


def test_format_argmax(fmt):
    torch = torch_cuda()
    f, code = fmt
    n, k, m = 20000, 1024, 12
    blocks = synth.fmt_matrix(f, n, k, seed=6, tensor_id=2900 + code)
    x = synth.x_f16(m, k, seed=6, tensor_id=3900)
    q = make(blocks, m_max=m, format=code)
    y = run(q, x)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    idx = torch.empty(m, dtype=torch.int32, device="cuda")
    val = torch.empty(m, dtype=torch.float32, device="cuda")
    q.run_argmax(xd, idx, val, m)
    torch.cuda.synchronize()
    ref = np.argmax(y, axis=1)
    assert np.array_equal(idx.cpu().numpy(), ref)
    y_ref, s_ref = oracle.qmm(blocks, x)
    bound = TOL_REL * s_ref + TOL_ABS
    rows = np.arange(m)
    j = np.argmax(y_ref, axis=1)
    assert np.all(y_ref[rows, ref] + bound[rows, ref] >= y_ref[rows, j] - bound[rows, j])
