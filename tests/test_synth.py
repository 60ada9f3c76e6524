"""The seeded input generator: fp16 rounding, determinism, random access, distributions."""
import numpy as np

import oracle
import synth


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(20000) * 1e-3,                    # the d/dmin range, many subnormal
        rng.standard_normal(20000),
        rng.standard_normal(2000) * 30000,
        np.ldexp(rng.integers(0, 2048, 4000) + 0.5, -24),      # exact ties in the subnormal range
        np.ldexp(1024 + rng.integers(0, 1024, 4000) + 0.5, -10),  # exact ties around 1..2
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e-9, 2.0 ** -25, 3 * 2.0 ** -26,
                  2.0 ** -14, 2.0 ** -14 - 2.0 ** -25]),
    ])
    ours = np.array([synth.f16_bits(v) for v in vals], dtype=np.uint16)
    ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_blocks_deterministic_and_random_access():
    a = synth.q4k_blocks(100, seed=0, tensor_id=3)
    b = synth.q4k_blocks(100, seed=0, tensor_id=3)
    assert np.array_equal(a, b)
    c = synth.q4k_blocks(30, seed=0, tensor_id=3, first_block=40)
    assert np.array_equal(a[40:70], c)
    assert not np.array_equal(a, synth.q4k_blocks(100, seed=0, tensor_id=4))
    assert not np.array_equal(a, synth.q4k_blocks(100, seed=1, tensor_id=3))


def test_matrix_rows_subset():
    full = synth.q4k_matrix(10, 512, seed=0, tensor_id=9)
    rows = np.array([7, 2, 9])
    assert np.array_equal(synth.q4k_matrix(10, 512, seed=0, tensor_id=9, rows=rows), full[rows])


def test_x_prefix_property():
    """The first M rows of an activation tensor do not depend on how many rows were drawn."""
    x12 = synth.x_f16(12, 512, seed=0, tensor_id=1000)
    x3 = synth.x_f16(3, 512, seed=0, tensor_id=1000)
    assert np.array_equal(x12[:3].view(np.uint16), x3.view(np.uint16))


def test_distributions():
    blocks = synth.q4k_blocks(20000, seed=0, tensor_id=0)
    d = blocks[:, 0:2].copy().view(np.uint16).ravel()
    dmin = blocks[:, 2:4].copy().view(np.uint16).ravel()
    dv = np.array([oracle.f16_to_double(int(v)) for v in d[:5000]])
    mv = np.array([oracle.f16_to_double(int(v)) for v in dmin[:5000]])
    # |N(0,1)| has mean sqrt(2/pi) = 0.7979
    assert abs(dv.mean() / 1e-3 - 0.7979) < 0.03
    assert abs(mv.mean() / 1e-3 - 0.7979) < 0.03
    assert (dv >= 0).all() and (mv >= 0).all()
    # about 5% of |N|*1e-3 fall below fp16's smallest normal 2^-14 -> subnormal patterns
    frac_sub = np.mean(d < 0x0400)
    assert 0.03 < frac_sub < 0.07
    # scale/min bytes and quant bytes are uniform bytes
    for part in (blocks[:, 4:16], blocks[:, 16:]):
        counts = np.bincount(part.ravel(), minlength=256)
        expected = part.size / 256
        chi2 = ((counts - expected) ** 2 / expected).sum()
        assert chi2 < 400   # 255 degrees of freedom; 400 is far in the tail
    # 6-bit scales uniform on 0..63
    sc = [oracle.scale_min(blocks[i, 4:16].tobytes(), j)[0] for i in range(2000) for j in range(8)]
    counts = np.bincount(sc, minlength=64)
    assert counts.size == 64 and counts.min() > 150


def test_x_distribution_and_outliers():
    x = synth.x_f16(64, 5120, seed=0, tensor_id=1000).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    xo = synth.x_f16(64, 5120, seed=0, tensor_id=1000, outlier_p=0.01, outlier_mul=20.0)
    xo = xo.astype(np.float64)
    frac = np.mean(np.abs(xo - x) > 1e-9)
    assert 0.008 < frac < 0.012
    changed = np.abs(xo - x) > 1e-9
    ratio = xo[changed] / x[changed]
    assert np.all(np.abs(ratio - 20) < 0.02)


def test_stack_shapes():
    mats = synth.stack()
    assert len(mats) == 257
    total = sum(m.weight_bytes for m in mats)
    assert total == 12_705_914_880
    assert sum(m.weight_bytes for m in synth.stack(lm_head=False)) == 12_268_339_200
    assert synth.SINGLE_PROJECTION.weight_bytes == 9_437_184
    assert len({m.tensor_id for m in mats}) == 257
