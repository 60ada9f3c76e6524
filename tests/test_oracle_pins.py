"""Pins for the CPU oracle: checks against things the format and the mathematics fix,
independent of the oracle's own code.

- hand-packed blocks (tests/golden/q4k_handpacked.txt) with closed-form weights, computed
  here in exact rational arithmetic;
- a round trip through the test-side packer (written in the opposite direction);
- every fp16 bit pattern against numpy's float16 (a library routine);
- invariants: a zeroed (scale, min) pair zeroes its sub-block, d = dmin = 0 zeroes the
  block, x = e_k picks column k, row permutation, linearity;
- brute force on tiny shapes in exact rational arithmetic (fractions.Fraction).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from q4k_pack import pack_block, pack_scales

GOLDEN = __file__.rsplit("/", 1)[0] + "/golden/q4k_handpacked.txt"


def load_golden():
    blocks, cur = [], {}
    for line in open(GOLDEN):
        line = line.rstrip("\n")
        if not line or line.startswith("#"):
            if cur:
                blocks.append(cur)
                cur = {}
            continue
        key, val = line.split(": ", 1)
        cur[key] = val
    if cur:
        blocks.append(cur)
    out = []
    for b in blocks:
        dbits, dval = b["d"].split()
        mbits, mval = b["dmin"].split()
        out.append(dict(
            name=b["name"], d_bits=int(dbits, 16), d=Fraction(dval), dmin_bits=int(mbits, 16),
            dmin=Fraction(mval), sc=[int(v) for v in b["sc"].split()],
            m=[int(v) for v in b["m"].split()], q=[int(c, 16) for c in b["q"]],
            bytes=np.frombuffer(bytes.fromhex(b["bytes"]), dtype=np.uint8).copy()))
    return out


GOLD = load_golden()


def exact_weights(g):
    return [g["d"] * g["sc"][i // 32] * g["q"][i] - g["dmin"] * g["m"][i // 32] for i in range(256)]


def test_golden_file_is_complete():
    names = {g["name"] for g in GOLD}
    assert names == {"ramp", "nibble_order", "scales", "closed_form", "subnormal",
                     "zero_subblock", "zero_block"}
    for g in GOLD:
        assert g["bytes"].size == 144 and len(g["q"]) == 256


@pytest.mark.parametrize("g", GOLD, ids=lambda g: g["name"])
def test_packer_matches_hand_packed_bytes(g):
    assert np.array_equal(pack_block(g["d_bits"], g["dmin_bits"], g["sc"], g["m"], g["q"]),
                          g["bytes"])


@pytest.mark.parametrize("g", GOLD, ids=lambda g: g["name"])
def test_d_dmin_exact_values(g):
    assert Fraction(oracle.f16_to_double(g["d_bits"])) == g["d"]
    assert Fraction(oracle.f16_to_double(g["dmin_bits"])) == g["dmin"]


@pytest.mark.parametrize("g", GOLD, ids=lambda g: g["name"])
def test_scale_min_unpack(g):
    s = g["bytes"][4:16].tobytes()
    for j in range(8):
        assert oracle.scale_min(s, j) == (g["sc"][j], g["m"][j]), j


@pytest.mark.parametrize("g", GOLD, ids=lambda g: g["name"])
def test_nibble_order(g):
    qs = g["bytes"][16:]
    assert [oracle.quant(qs, i) for i in range(256)] == g["q"]


@pytest.mark.parametrize("g", GOLD, ids=lambda g: g["name"])
def test_dequant_closed_form(g):
    w = oracle.dequant_block(g["bytes"])
    exact = exact_weights(g)
    for i in range(256):
        # every golden block is exactly representable in fp32
        assert Fraction(float(w[i])) == exact[i], (g["name"], i, float(w[i]), exact[i])


def test_closed_form_values_by_hand():
    g = next(g for g in GOLD if g["name"] == "closed_form")
    w = oracle.dequant_block(g["bytes"])
    for j in range(8):
        assert np.all(w[32 * j:32 * j + 32] == np.float32(15 * (j + 1) / 16 - j / 4))
    g = next(g for g in GOLD if g["name"] == "scales")
    w = oracle.dequant_block(g["bytes"])
    assert [float(w[32 * j]) for j in range(8)] == [-2, 63, -63, 19, 14, -42, 38, -16]
    g = next(g for g in GOLD if g["name"] == "ramp")
    assert np.array_equal(oracle.dequant_block(g["bytes"]), np.arange(256) % 16)
    g = next(g for g in GOLD if g["name"] == "subnormal")
    assert np.all(oracle.dequant_block(g["bytes"]) == np.float32(-78 * 2.0 ** -24))


def test_zero_invariants():
    g = next(g for g in GOLD if g["name"] == "zero_subblock")
    w = oracle.dequant_block(g["bytes"])
    assert np.all(w[96:128] == 0) and np.all(w[:96] != 0)
    g = next(g for g in GOLD if g["name"] == "zero_block")
    assert np.all(oracle.dequant_block(g["bytes"]) == 0)


def test_fp16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    # signs of zero
    assert np.copysign(1.0, oracle.f16_to_double(0x8000)) == -1.0


def test_scale_round_trip_random():
    rng = np.random.default_rng(12345)
    for _ in range(4096):
        sc = rng.integers(0, 64, 8)
        mn = rng.integers(0, 64, 8)
        s = pack_scales(sc, mn)
        for j in range(8):
            assert oracle.scale_min(s, j) == (sc[j], mn[j])


def test_scale_bytes_bijection_single_bit_flips():
    """Every one of the 96 scale bits belongs to exactly one 6-bit value: flipping it
    changes exactly one (sc_j or m_j) by a power of two."""
    rng = np.random.default_rng(7)
    base = bytes(rng.integers(0, 256, 12, dtype=np.uint8))
    ref = [oracle.scale_min(base, j) for j in range(8)]
    owners = set()
    for bit in range(96):
        flipped = bytearray(base)
        flipped[bit // 8] ^= 1 << (bit % 8)
        new = [oracle.scale_min(bytes(flipped), j) for j in range(8)]
        diffs = [(j, f) for j in range(8) for f in range(2) if new[j][f] != ref[j][f]]
        assert len(diffs) == 1, bit
        j, f = diffs[0]
        delta = abs(new[j][f] - ref[j][f])
        assert delta & (delta - 1) == 0
        owners.add((j, f, delta))
    assert len(owners) == 96


def _brute_force(blocks, x):
    """y and S in exact rationals, one weight at a time from the listed parameters."""
    n, kb, _ = blocks.shape
    m = x.shape[0]
    xf = [[Fraction(float(v)) for v in row] for row in x.astype(np.float64)]
    y = [[Fraction(0)] * n for _ in range(m)]
    s = [[Fraction(0)] * n for _ in range(m)]
    for r in range(n):
        for b in range(kb):
            blk = blocks[r, b]
            d = Fraction(oracle.f16_to_double(int(blk[0]) | int(blk[1]) << 8))
            dmin = Fraction(oracle.f16_to_double(int(blk[2]) | int(blk[3]) << 8))
            s12 = blk[4:16].tobytes()
            for i in range(256):
                sc, mn = oracle.scale_min(s12, i // 32)
                q = oracle.quant(blk[16:], i)
                w = d * sc * q - dmin * mn
                for t in range(m):
                    p = w * xf[t][256 * b + i]
                    y[t][r] += p
                    s[t][r] += abs(p)
    return y, s


@pytest.mark.parametrize("n,k,m", [(1, 256, 1), (3, 256, 2), (4, 512, 3), (2, 512, 1)])
def test_brute_force_tiny(n, k, m):
    blocks = synth.q4k_matrix(n, k, seed=11, tensor_id=n * 100 + k + m, scale_mul=1e-3)
    x = synth.x_f16(m, k, seed=11, tensor_id=7 + m)
    y, s = oracle.qmm(blocks, x)
    ye, se = _brute_force(blocks, x)
    for t in range(m):
        for r in range(n):
            # fp32 weights are exact for these magnitudes except the a*q - c rounding; the
            # double sum rounds K times.  Both are far below 1e-6 of S.
            assert abs(Fraction(y[t, r]) - ye[t][r]) <= Fraction(1, 10**6) * se[t][r]
            assert abs(Fraction(s[t, r]) - se[t][r]) <= Fraction(1, 10**9) * se[t][r]


def test_unit_vector_picks_weight_column():
    n, k = 5, 512
    blocks = synth.q4k_matrix(n, k, seed=3, tensor_id=1)
    w = oracle.dequant_matrix(blocks)
    for col in (0, 1, 31, 32, 63, 64, 255, 256, 300, 511):
        x = np.zeros((1, k), dtype=np.float16)
        x[0, col] = 1.0
        y, s = oracle.qmm(blocks, x)
        assert np.array_equal(y[0], w[:, col].astype(np.float64))
        assert np.array_equal(s[0], np.abs(w[:, col]).astype(np.float64))


def test_row_permutation_and_linearity():
    n, k, m = 7, 768, 5
    blocks = synth.q4k_matrix(n, k, seed=5, tensor_id=2)
    x = synth.x_f16(m, k, seed=5, tensor_id=3)
    y, _ = oracle.qmm(blocks, x)
    perm = np.array([3, 0, 4, 1, 2])
    yp, _ = oracle.qmm(blocks, x[perm])
    assert np.array_equal(yp, y[perm])
    # x -> 2x is exact in fp16 and doubles every product and partial sum exactly
    y2, _ = oracle.qmm(blocks, (x.astype(np.float32) * 2).astype(np.float16))
    assert np.array_equal(y2, 2 * y)
    # y(x1) + y(x2) vs y(x1 + x2) for x values whose sums stay exact in fp16
    rng = np.random.default_rng(0)
    x1 = rng.integers(-8, 8, (m, k)).astype(np.float16)
    x2 = rng.integers(-8, 8, (m, k)).astype(np.float16)
    ya, sa = oracle.qmm(blocks, x1)
    yb, sb = oracle.qmm(blocks, x2)
    yc, _ = oracle.qmm(blocks, (x1.astype(np.float32) + x2).astype(np.float16))
    assert np.all(np.abs(yc - (ya + yb)) <= 1e-12 * (sa + sb))


def test_zero_pair_makes_output_independent_of_its_inputs():
    """With (sc_j, m_j) = (0, 0) in every block, y does not depend on x over sub-block j."""
    n, k = 4, 512
    blocks = synth.q4k_matrix(n, k, seed=9, tensor_id=4)
    for r in range(n):
        for b in range(k // 256):
            s = blocks[r, b, 4:16].tobytes()
            sc = [oracle.scale_min(s, j)[0] for j in range(8)]
            mn = [oracle.scale_min(s, j)[1] for j in range(8)]
            sc[5] = mn[5] = 0
            blocks[r, b, 4:16] = np.frombuffer(pack_scales(sc, mn), dtype=np.uint8)
    x = synth.x_f16(2, k, seed=9, tensor_id=5)
    y, _ = oracle.qmm(blocks, x)
    x2 = x.copy()
    for b in range(k // 256):
        x2[:, 256 * b + 160:256 * b + 192] = np.float16(1000.0)
    y2, _ = oracle.qmm(blocks, x2)
    assert np.array_equal(y, y2)


def test_empty_shapes():
    blocks = synth.q4k_matrix(3, 256, seed=1, tensor_id=1)
    y, s = oracle.qmm(blocks, np.zeros((0, 256), dtype=np.float16))
    assert y.shape == (0, 3)
    y, s = oracle.qmm(np.zeros((0, 1, 144), dtype=np.uint8), np.ones((2, 256), dtype=np.float16))
    assert y.shape == (2, 0)


# --------------------------------------------------------------------- greedy verification
def _brute_argmax(y):
    """Plain loop: the first column holding the row's largest value."""
    out = []
    for row in y:
        best = 0
        for j in range(1, len(row)):
            if row[j] > row[best]:
                best = j
        out.append(best)
    return out


def test_argmax_rows_brute_force_and_ties():
    rng = np.random.default_rng(4)
    # integer-valued rows with many repeated maxima, so ties are common
    y = rng.integers(-3, 4, (40, 17)).astype(np.float64)
    idx, val = oracle.argmax_rows(y)
    assert list(idx) == _brute_argmax(y)
    assert np.array_equal(val, y.max(axis=1))
    # a tie between columns 5 and 11 (both hold the maximum): the lower column
    t = np.zeros((1, 16))
    t[0, 5] = t[0, 11] = 2.0
    assert oracle.argmax_rows(t)[0][0] == 5
    # negative rows and one column
    assert oracle.argmax_rows(np.array([[-5.0, -1.0, -3.0]]))[0][0] == 1
    assert oracle.argmax_rows(np.array([[-7.0]]))[0][0] == 0


def test_argmax_of_identical_weight_rows_is_the_lower_row():
    """Two output rows with the same blocks have equal logits; with both ahead of every other
    row (closed form: all quants 15, every scale 63, min 0, so each weight is d*63*15, and
    x = 1), greedy verification must name the lower row."""
    n, k = 6, 256
    blocks = np.zeros((n, 1, 144), dtype=np.uint8)
    for r in range(n):
        d = 0x3C00 if r in (2, 4) else 0x3800  # 1.0 for rows 2 and 4, 0.5 elsewhere
        blocks[r, 0] = pack_block(d, 0, [63] * 8, [0] * 8, [15] * 256)
    x = np.ones((1, k), dtype=np.float16)
    y, _ = oracle.qmm(blocks, x)
    assert y[0, 2] == y[0, 4] == 256 * 63 * 15 and y[0, 0] == 256 * 63 * 15 / 2
    idx, val = oracle.argmax_rows(y)
    assert idx[0] == 2 and val[0] == 256 * 63 * 15


# --------------------------------------------------------------------- other block formats
def test_q8_0_closed_form_and_round_trip():
    from q4k_pack import pack_q8_0
    q = [-128, -1, 0, 1, 127] + [(7 * i) % 256 - 128 for i in range(27)]
    blk = pack_q8_0(0x3800, q)  # d = 0.5
    w = oracle.dequant_block_fmt(blk)
    assert list(w) == [0.5 * v for v in q]
    # x = e_k picks weight k of every row
    blocks = np.stack([pack_q8_0(0x3C00, q)[None], pack_q8_0(0x4000, q[::-1])[None]])
    for col in (0, 4, 31):
        x = np.zeros((1, 32), dtype=np.float16)
        x[0, col] = 1.0
        y, s = oracle.qmm(blocks, x)
        assert y[0, 0] == q[col] and y[0, 1] == 2.0 * q[::-1][col]


def test_q6_k_closed_form_and_round_trip():
    from q4k_pack import pack_q6_k
    rng = np.random.default_rng(12)
    q = rng.integers(0, 64, 256)
    sc = rng.integers(-128, 128, 16)
    blk = pack_q6_k(0x3400, sc, q)  # d = 0.25
    for i in range(256):
        assert oracle.q6k_quant(blk, i) == q[i]
    w = oracle.dequant_block_fmt(blk)
    assert np.array_equal(w, 0.25 * sc[np.arange(256) // 16] * (q - 32.0))
    # a scale of zero zeroes its sub-block of 16 weights; q = 32 is a zero weight
    sc2 = sc.copy()
    sc2[5] = 0
    q2 = q.copy()
    q2[200] = 32
    w2 = oracle.dequant_block_fmt(pack_q6_k(0x3400, sc2, q2))
    assert np.all(w2[80:96] == 0) and w2[200] == 0


@pytest.mark.parametrize("fmt,n,k,m", [("q8", 3, 64, 2), ("q8", 2, 256, 1), ("q6", 2, 256, 2), ("q6", 1, 512, 1)])
def test_brute_force_tiny_formats(fmt, n, k, m):
    """Exact rational sums for Q8_0 and Q6_K matrices against the oracle's double sums."""
    f = synth.Q8_0 if fmt == "q8" else synth.Q6_K
    blocks = synth.fmt_matrix(f, n, k, seed=13, tensor_id=n * 10 + m)
    x = synth.x_f16(m, k, seed=13, tensor_id=70 + m)
    y, s = oracle.qmm(blocks, x)
    per = f[1]
    for r in range(n):
        # weights from the bytes, written out here without the oracle
        wr = []
        for b in range(k // per):
            blk = blocks[r, b]
            if fmt == "q8":
                d = Fraction(float(np.frombuffer(blk[:2].tobytes(), dtype=np.float16)[0]))
                wr += [d * int(np.int8(v)) for v in blk[2:34].view(np.int8)]
            else:
                d = Fraction(float(np.frombuffer(blk[208:210].tobytes(), dtype=np.float16)[0]))
                scs = blk[192:208].view(np.int8)
                for i in range(256):
                    h, rr = divmod(i, 128)
                    c, l = divmod(rr, 32)
                    lo = (int(blk[64 * h + l + 32 * (c % 2)]) >> (4 * (c // 2))) & 15
                    hi = (int(blk[128 + 32 * h + l]) >> (2 * c)) & 3
                    wr.append(d * int(scs[i // 16]) * ((lo | hi << 4) - 32))
        for t in range(m):
            ye = sum(wk * Fraction(float(xv)) for wk, xv in zip(wr, x[t]))
            se = sum(abs(wk * Fraction(float(xv))) for wk, xv in zip(wr, x[t]))
            assert abs(Fraction(y[t, r]) - ye) <= Fraction(1, 10**9) * se + Fraction(1, 10**30)
            assert abs(Fraction(s[t, r]) - se) <= Fraction(1, 10**9) * se + Fraction(1, 10**30)
