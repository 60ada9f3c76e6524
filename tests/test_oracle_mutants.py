"""Planted mistakes in the oracle must fail its pins.

Each case copies the oracle's C source to a temporary directory, plants one plausible
mistake (a swapped nibble, a wrong bit index, a dropped or sign-flipped term, a wrong
exponent, a skipped element), compiles it, and runs the pin checks against the mutant.
The real oracle passes the same checks (see test_oracle_pins.py); every mutant must fail
at least one.  Nothing here touches a GPU.
"""
import ctypes
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import synth
from test_oracle_pins import GOLD, exact_weights

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "q4k_oracle.c")

MUTANTS = {
    "swap_nibbles": ("(qs[32 * c + r] & 15) : (qs[32 * c + r - 32] >> 4)",
                     "(qs[32 * c + r] >> 4) : (qs[32 * c + r - 32] & 15)"),
    "sc_high_bits_from_wrong_byte": ("*sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);",
                                     "*sc = (s[j + 4] & 15) | ((s[j] >> 6) << 4);"),
    "min_high_bits_from_wrong_byte": ("*mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);",
                                      "*mn = (s[j + 4] >> 4) | ((s[j - 4] >> 6) << 4);"),
    "min_mask_5_bits": ("*mn = s[j + 4] & 63;", "*mn = s[j + 4] & 31;"),
    "drop_min_term": ("w[i] = a * q - c;", "w[i] = a * q;"),
    "min_sign": ("w[i] = a * q - c;", "w[i] = a * q + c;"),
    "d_dmin_swapped": ("float d = (float)oracle_f16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));",
                       "float d = (float)oracle_f16_to_double((uint16_t)(blk[2] | (blk[3] << 8)));"),
    "subnormal_exponent": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "normal_exponent": ("v = ldexp((double)(1024 + f), e - 25);",
                        "v = ldexp((double)(1024 + f), e - 24);"),
    "skip_last_k": ("for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 0; k < K - 1; ++k) {"),
    "subblock_index": ("for (int i = 32 * j; i < 32 * j + 32; ++i) {",
                       "for (int i = 32 * (7 - j); i < 32 * (7 - j) + 32; ++i) {"),
    "abs_sum_signed": ("sabs += fabs(p);", "sabs += p;"),
    # Q8_0 and Q6_K
    "q8_unsigned_quants": ("w[i] = d * (double)(int8_t)blk[2 + i];", "w[i] = d * (double)blk[2 + i];"),
    "q8_d_offset": ("double d = oracle_f16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));\n    for (int i = 0; i < 32;",
                    "double d = oracle_f16_to_double((uint16_t)(blk[1] | (blk[0] << 8)));\n    for (int i = 0; i < 32;"),
    "q6_ql_half": ("int lo = (ql[64 * h + l + 32 * (c & 1)] >> (4 * (c >> 1))) & 15;",
                   "int lo = (ql[64 * h + l + 32 * (c >> 1)] >> (4 * (c & 1))) & 15;"),
    "q6_qh_shift": ("int hi = (qh[32 * h + l] >> (2 * c)) & 3;", "int hi = (qh[32 * h + l] >> c) & 3;"),
    "q6_offset": ("(double)(oracle_q6k_quant(blk, i) - 32);", "(double)(oracle_q6k_quant(blk, i) - 31);"),
    "q6_scale_index": ("w[i] = d * (double)sc[i / 16]", "w[i] = d * (double)sc[i / 32]"),
    "q6_unsigned_scales": ("const int8_t* sc = (const int8_t*)(blk + 192);",
                           "const uint8_t* sc = (const uint8_t*)(blk + 192);"),
    "fmt_skip_last_k": ("for (int64_t kk = 0; kk < K; ++kk) {", "for (int64_t kk = 1; kk < K; ++kk) {"),
}


def _compile(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mutated = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mutated)
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                           str(c), "-o", str(so), "-lm"])
    lib = ctypes.CDLL(str(so))
    lib.oracle_f16_to_double.restype = ctypes.c_double
    lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_dequant_block.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_qmm.restype = ctypes.c_int
    lib.oracle_qmm.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                               ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_qmm_fmt.restype = ctypes.c_int
    lib.oracle_qmm_fmt.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_int]
    lib.oracle_dequant_fmt.restype = ctypes.c_int
    lib.oracle_dequant_fmt.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    return lib


def _format_pins_hold(lib) -> bool:
    """Q8_0 and Q6_K: hand-packed blocks against their closed form, and x = -e_k picking
    column k of a matrix (y = -w[:, k], S = |w[:, k]|)."""
    from q4k_pack import pack_q6_k, pack_q8_0
    rng = np.random.default_rng(21)
    q8 = [int(v) for v in rng.integers(-128, 128, 32)]
    b8 = pack_q8_0(0x3800, q8)
    w8 = np.empty(32)
    lib.oracle_dequant_fmt(2, b8.ctypes.data, w8.ctypes.data)
    if list(w8) != [0.5 * v for v in q8]:
        return False
    q6 = rng.integers(0, 64, 256)
    sc6 = rng.integers(-128, 128, 16)
    b6 = pack_q6_k(0x3400, sc6, q6)
    w6 = np.empty(256)
    lib.oracle_dequant_fmt(1, b6.ctypes.data, w6.ctypes.data)
    if not np.array_equal(w6, 0.25 * sc6[np.arange(256) // 16] * (q6 - 32.0)):
        return False
    for fmt, f in ((2, synth.Q8_0), (1, synth.Q6_K)):
        blocks = np.ascontiguousarray(synth.fmt_matrix(f, 3, 512, seed=4, tensor_id=fmt))
        per = f[1]
        w = np.empty((3, 512))
        for r in range(3):
            for b in range(512 // per):
                out = np.empty(per)
                lib.oracle_dequant_fmt(fmt, np.ascontiguousarray(blocks[r, b]).ctypes.data, out.ctypes.data)
                w[r, per * b:per * (b + 1)] = out
        for col in (0, 31, 300, 511):
            x = np.zeros((1, 512), dtype=np.float16)
            x[0, col] = -1.0
            y, s = np.empty((1, 3)), np.empty((1, 3))
            lib.oracle_qmm_fmt(fmt, blocks.ctypes.data, 3, 512, x.view(np.uint16).ctypes.data, 1,
                               y.ctypes.data, s.ctypes.data, 1)
            if not (np.array_equal(y[0], -w[:, col]) and np.array_equal(s[0], np.abs(w[:, col]))):
                return False
    return True


def _pins_hold(lib) -> bool:
    # golden blocks against their closed form
    for g in GOLD:
        b = np.ascontiguousarray(g["bytes"])
        w = np.empty(256, dtype=np.float32)
        lib.oracle_dequant_block(b.ctypes.data, w.ctypes.data)
        if [Fraction(float(v)) for v in w] != exact_weights(g):
            return False
    # fp16 decode against numpy on every pattern
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([lib.oracle_f16_to_double(int(v)) for v in bits])
    if not np.all((got == ref) | (np.isnan(got) & np.isnan(ref))):
        return False
    # x = e_k picks column k; S = |column k|
    blocks = np.ascontiguousarray(synth.q4k_matrix(3, 512, seed=3, tensor_id=1))
    w = np.empty((3, 512), dtype=np.float32)
    for r in range(3):
        for kb in range(2):
            out = np.empty(256, dtype=np.float32)
            lib.oracle_dequant_block(np.ascontiguousarray(blocks[r, kb]).ctypes.data,
                                     out.ctypes.data)
            w[r, 256 * kb:256 * kb + 256] = out
    for col in (0, 255, 300, 511):
        x = np.zeros((1, 512), dtype=np.float16)
        x[0, col] = -1.0
        y = np.empty((1, 3))
        s = np.empty((1, 3))
        lib.oracle_qmm(blocks.ctypes.data, 3, 512, x.view(np.uint16).ctypes.data, 1,
                       y.ctypes.data, s.ctypes.data, 1)
        if not (np.array_equal(y[0], -w[:, col].astype(np.float64))
                and np.array_equal(s[0], np.abs(w[:, col]).astype(np.float64))):
            return False
    return True


def test_real_oracle_passes(tmp_path):
    lib = _compile(tmp_path, "identity", "int oracle_max_threads(void) {",
                   "int oracle_max_threads(void) {")
    assert _pins_hold(lib) and _format_pins_hold(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _compile(tmp_path, name, old, new)
    assert not (_pins_hold(lib) and _format_pins_hold(lib)), f"planted mistake {name} passed every pin"
