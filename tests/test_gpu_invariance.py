"""Batch invariance: a row's result is bit-identical alone or batched with other rows, at
any position in the batch (page "Running 4 coding agents on one RTX 3090", section on
keeping real agents fast: a prompt chunked in with other agents' rows gives bit-identical
results to running it alone).  Also run-to-run determinism."""
import numpy as np
import pytest

import synth
from gpu_util import make, run

pytestmark = pytest.mark.gpu


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


@pytest.mark.parametrize("mat", list(synth.SWEEP_MATRICES) + [synth.Matrix("small", 200, 1280, 77)],
                         ids=lambda m: m.name)
def test_sub_batches_bitwise(mat, backend):
    blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
    x = synth.x_f16(64, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
    q = make(blocks, m_max=64, backend=backend)
    full = bits(run(q, x))
    # every M of the sweep equals the prefix of the 64-row batch
    for m in synth.SWEEP_M:
        assert np.array_equal(bits(run(q, x[:m])), full[:m]), m
    # 12 = 4 + 8, 12 x 1, and 64 = 8 x 8 sub-batches
    for parts in ([4, 8], [1] * 12, [8] * 8, [3, 5, 7, 1, 16, 32]):
        r0 = 0
        for p in parts:
            assert np.array_equal(bits(run(q, x[r0:r0 + p])), full[r0:r0 + p]), (parts, r0)
            r0 += p
    # rows at other positions in the batch
    perm = np.random.default_rng(0).permutation(64)
    assert np.array_equal(bits(run(q, x[perm])), full[perm])
    # the same row surrounded by different neighbours
    x2 = synth.x_f16(16, mat.k, seed=9, tensor_id=9)
    x2[5] = x[0]
    assert np.array_equal(bits(run(q, x2))[5], full[0])


def test_repeat_determinism(backend):
    mat = synth.SWEEP_MATRICES[1]
    blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
    x = synth.x_f16(12, mat.k, seed=0, tensor_id=1003)
    q = make(blocks, m_max=12, backend=backend)
    ref = bits(run(q, x))
    for _ in range(100):
        assert np.array_equal(bits(run(q, x)), ref)


@pytest.mark.parametrize("mat", [synth.Matrix("wide_a", 1000, 2560, 78), synth.SWEEP_MATRICES[1]],
                         ids=lambda m: m.name)
def test_wide_launches_match_narrow_ones(mat):
    """tcgen05 handles of 200 rows: a 200-row run is one 128-row launch (whose activation sums
    come from the pre-pass, and whose dequantisation warps get more registers) and one of 72
    rows; every row equals, bit for bit, the same row run in 1-, 16-, 32- and 64-row batches
    (whose sums the dequantisation warps form themselves)."""
    blocks = synth.q4k_matrix(mat.n, mat.k, seed=0, tensor_id=mat.tensor_id)
    x = synth.x_f16(200, mat.k, seed=0, tensor_id=synth.X_ID_OFFSET + mat.tensor_id)
    q = make(blocks, m_max=200, backend=2)
    full = bits(run(q, x))
    for m in (1, 16, 32, 64, 65, 100, 127, 128, 129):
        assert np.array_equal(bits(run(q, x[:m])), full[:m]), m
    for parts in ([1] * 8, [16, 32, 64, 88], [129, 71], [7, 121, 72]):
        r0 = 0
        for p in parts:
            assert np.array_equal(bits(run(q, x[r0:r0 + p])), full[r0:r0 + p]), (parts, r0)
            r0 += p
