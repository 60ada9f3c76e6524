"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Tolerance: |y - y_ref| <= 2e-3 * sum_k |w x| + 1e-6 (the oracle dequantises in fp32 and
accumulates in double; the GPU dequantises to fp16 and accumulates in fp32, and the pages
say outputs differ from other engines in the last bits because the order differs)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_parity, make, run, torch_cuda

pytestmark = pytest.mark.gpu


def test_single_projection_m1(backend):
    """4096 x 4096, M = 1, seed 0: every output checked."""
    mat = synth.SINGLE_PROJECTION
    blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
    x = synth.x_f16(1, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
    y_ref, s_ref = oracle.qmm(blocks, x)
    q = make(blocks, m_max=1, backend=backend)
    assert_parity(run(q, x), y_ref, s_ref, "proj4096 M=1")


@pytest.mark.parametrize("mat", synth.SWEEP_MATRICES, ids=lambda m: m.name)
def test_m_sweep_full_matrices(mat, backend):
    """gate_up [5120->34816] and down [17408->5120] at every M of the sweep; the oracle
    runs once on 64 rows (rows are independent, so the first M rows serve every M)."""
    blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
    x = synth.x_f16(64, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
    y_ref, s_ref = oracle.qmm(blocks, x)
    q = make(blocks, m_max=64, backend=backend)
    for m in synth.SWEEP_M:
        assert_parity(run(q, x[:m]), y_ref[:m], s_ref[:m], f"{mat.name} M={m}")


@pytest.mark.parametrize("n,k,m", [
    (1, 256, 1), (33, 256, 3), (40, 512, 5), (100, 768, 9), (257, 1024, 16), (31, 2560, 12),
    (5, 256, 17), (64, 4096, 8), (96, 256, 2), (500, 1280, 13), (1000, 512, 16), (77, 7680, 7),
    (300, 768, 65), (129, 512, 128), (700, 1024, 129), (33, 2304, 200),
])
def test_ragged_shapes(n, k, m, backend):
    """Several tiles, ragged row tails, tiles split between CTAs, M chunked past 16 (mma.sync)
    and past 128 (tcgen05), and the 64- and 128-row launch widths."""
    blocks = synth.q4k_matrix(n, k, seed=1, tensor_id=n * 7 + k)
    x = synth.x_f16(m, k, seed=1, tensor_id=n + k + m)
    y_ref, s_ref = oracle.qmm(blocks, x)
    q = make(blocks, m_max=max(m, 1), backend=backend)
    assert_parity(run(q, x), y_ref, s_ref, f"N={n} K={k} M={m}")


def test_outlier_activations(backend):
    """1% of activations x20 (the chunked-prefill workload's distribution)."""
    n, k, m = 512, 5120, 16
    blocks = synth.q4k_matrix(n, k, seed=0, tensor_id=2)
    x = synth.x_f16(m, k, seed=0, tensor_id=1002, outlier_p=0.01, outlier_mul=20.0)
    y_ref, s_ref = oracle.qmm(blocks, x)
    assert_parity(run(make(blocks, backend=backend), x), y_ref, s_ref, "outliers")


def _golden_matrix():
    from test_oracle_pins import GOLD
    by = {g["name"]: g["bytes"] for g in GOLD}
    order = ["ramp", "nibble_order", "scales", "closed_form", "subnormal", "zero_subblock",
             "zero_block"]
    rows = [np.stack([by[order[(r + j) % len(order)]] for j in range(4)]) for r in range(40)]
    return np.stack(rows)  # [40, 4, 144]: K = 1024


def test_hand_packed_blocks(backend):
    """Closed-form blocks (subnormal scales, zeroed pairs, top-bit crossings) in a matrix."""
    blocks = _golden_matrix()
    k = blocks.shape[1] * 256
    x = synth.x_f16(12, k, seed=4, tensor_id=4)
    y_ref, s_ref = oracle.qmm(blocks, x)
    assert_parity(run(make(blocks, backend=backend), x), y_ref, s_ref, "golden blocks")
    # a row made only of zero blocks gives exactly zero
    zb = np.repeat(blocks[:1, :1] * 0, 4, axis=1)
    zb = np.concatenate([zb, blocks[1:2]], axis=0)
    y = run(make(zb, backend=backend), x)
    assert np.all(y[:, 0] == 0)


def test_unit_vectors_pick_columns(backend):
    """x = e_k returns column k of W to within fp16 rounding of the dequantised weight."""
    n, k = 64, 512
    blocks = synth.q4k_matrix(n, k, seed=2, tensor_id=9)
    w = oracle.dequant_matrix(blocks)
    cols = [0, 1, 2, 3, 31, 32, 63, 64, 100, 255, 256, 300, 511]
    x = np.zeros((len(cols), k), dtype=np.float16)
    for i, c in enumerate(cols):
        x[i, c] = 1.0
    y = run(make(blocks, backend=backend), x)
    for i, c in enumerate(cols):
        ref = w[:, c].astype(np.float64)
        assert np.all(np.abs(y[i] - ref) <= 2e-3 * np.abs(ref) + 1e-6), c


def test_host_and_device_blocks_agree(backend):
    n, k, m = 70, 1024, 6
    blocks = synth.q4k_matrix(n, k, seed=3, tensor_id=3)
    x = synth.x_f16(m, k, seed=3, tensor_id=30)
    a = run(make(blocks, device_blocks=True, backend=backend), x)
    b = run(make(blocks, device_blocks=False, backend=backend), x)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_run_host_matches_device_run(backend):
    torch = torch_cuda()
    n, k, m = 300, 2048, 12
    blocks = synth.q4k_matrix(n, k, seed=5, tensor_id=5)
    x = synth.x_f16(m, k, seed=5, tensor_id=50)
    q = make(blocks, host_io=True, backend=backend)
    y_dev = run(q, x)
    xh = torch.from_numpy(x.view(np.int16).copy()).pin_memory()
    yh = torch.empty((m, n), dtype=torch.float32).pin_memory()
    q.run_host(xh, yh, m)
    torch.cuda.synchronize()
    assert np.array_equal(yh.numpy().view(np.uint32), y_dev.view(np.uint32))


def test_argument_errors_with_device(backend):
    from bit_weight_streaming_q4_gb300 import QmmError
    torch = torch_cuda()
    n, k = 64, 512
    blocks = synth.q4k_matrix(n, k, seed=6, tensor_id=6)
    q = make(blocks, m_max=4, backend=backend)
    x = torch.zeros((8, k), dtype=torch.float16, device="cuda")
    y = torch.zeros((8, n), dtype=torch.float32, device="cuda")
    q.run(x, y, 0)                                   # M = 0 is a no-op
    assert torch.all(y == 0)
    with pytest.raises(QmmError) as e:
        q.run(x, y, 5)                               # M > m_max
    assert e.value.status == 2
    xb = torch.zeros(8 * k + 8, dtype=torch.float16, device="cuda")
    with pytest.raises(QmmError) as e:
        q.run(xb[1:].data_ptr(), y, 1)               # misaligned x
    assert e.value.status == 3
    with pytest.raises(QmmError) as e:
        q.run(0, y, 1)
    assert e.value.status == 1
    assert q.error() == 0
    from bit_weight_streaming_q4_gb300 import qmm as Q
    lib = Q.load()
    raw = q.handle
    q.close()
    # use after destroy and destroy twice, with the stale handle value
    assert lib.qmm_run(raw, x.data_ptr(), 1, y.data_ptr(), None) == 7
    assert lib.qmm_destroy(raw) == 7
    assert lib.qmm_destroy(None) == 7


@pytest.mark.parametrize("mat", [synth.layer_matrices(0)[2], synth.layer_matrices(0)[3]], ids=lambda m: m.name)
def test_chunked_prefill_m524(mat, backend):
    """The chunked-prefill step: M = 524 rows (512-token prompt chunk + 12 decode rows) with 1%
    outlier activations x20, on gate_up and down at full size.  Sampled output columns (rows of
    W) against the oracle, every row; and each of a few rows bit-identical to the same row run
    alone (the run of 524 rows is cut into launches, which must not change any row's bits)."""
    torch = torch_cuda()
    m = 524
    blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
    x = synth.x_f16(m, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id,
                    outlier_p=0.01, outlier_mul=20.0)
    q = make(blocks, m_max=m, backend=backend)
    y = run(q, x)
    rng = np.random.default_rng(11)
    cols = np.sort(rng.choice(mat.n, size=24, replace=False))
    y_ref, s_ref = oracle.qmm(synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id, rows=cols), x)
    assert_parity(y[:, cols], y_ref, s_ref, f"{mat.name} M=524")
    for r in (0, 77, 511, 523):
        alone = run(q, x[r:r + 1])
        assert np.array_equal(alone[0].view(np.uint32), y[r].view(np.uint32)), r
