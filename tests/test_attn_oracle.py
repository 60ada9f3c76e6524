"""Pins for the decode-attention oracle (oracle/attn_oracle.c), checked against things the
definition fixes, not against the oracle's own code:

- a row that attends to one token returns that token's V exactly (softmax of one score is 1);
- all-zero K gives equal scores, so the output is the plain mean of the attended V rows,
  computed here in exact rational arithmetic from the pool bytes;
- brute force on small shapes: K and V decoded here from the documented record layout with
  numpy views, scores and softmax by scipy (a library routine), compared within 1e-12;
- moving the pages of the pool (and the page table with them) changes nothing, bit for bit;
- bytes of tokens past a row's length do not change that row;
- grouped-query attention: heads of one group read the same KV head.
Planted mistakes in a copy of the oracle must each fail one of these (test_mutants_fail).
"""
import ctypes
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

REC = oracle.ATTN_RECORD_BYTES
D = oracle.ATTN_D
PT = oracle.ATTN_PAGE_TOKENS


def decode_records(pool, kv_heads):
    """K [page, head, token, dim] and V [page, head, token, dim] in double, from the layout:
    K quants int8 in 128-byte token rows whose 16-byte pieces are permuted (piece p of token t
    stored at position p ^ (2 (t % 4) + (t / 4) % 2)), K scales fp16 [token][4], V quants int8 [dim][token], V
    scales fp16 [4][token]."""
    recs = pool.reshape(-1, kv_heads, REC)
    kq_stored = recs[:, :, :8192].view(np.int8).reshape(-1, kv_heads, PT, 8, 16)
    t = np.arange(PT)[:, None]
    pieces = np.arange(8)[None, :] ^ (2 * (t % 4) + (t // 4) % 2)   # [token][logical piece] -> stored
    kq = np.take_along_axis(kq_stored, pieces[None, None, :, :, None], axis=3).reshape(-1, kv_heads, PT, D)
    kq = kq.astype(np.float64)
    ks = recs[:, :, 8192:8704].copy().view(np.float16).reshape(-1, kv_heads, PT, 4).astype(np.float64)
    vq = recs[:, :, 8704:16896].view(np.int8).reshape(-1, kv_heads, D, PT).astype(np.float64)
    vs = recs[:, :, 16896:].copy().view(np.float16).reshape(-1, kv_heads, 4, PT).astype(np.float64)
    k = kq * np.repeat(ks, 32, axis=3)
    v = np.swapaxes(vq, 2, 3) * np.repeat(np.swapaxes(vs, 2, 3), 32, axis=3)
    return k, v


def reference(pool, table, q, row_agent, row_len, kv_heads):
    from scipy.special import softmax
    k, v = decode_records(pool, kv_heads)
    rows, heads, _ = q.shape
    group = heads // kv_heads
    out = np.zeros((rows, heads, D))
    for r in range(rows):
        n = row_len[r]
        pages = table[row_agent[r]]
        tok = np.arange(n)
        for h in range(heads):
            g = h // group
            kk = k[pages[tok // PT], g, tok % PT]
            vv = v[pages[tok // PT], g, tok % PT]
            p = softmax(kk @ q[r, h].astype(np.float64) / np.sqrt(D))
            out[r, h] = p @ vv
    return out


def small_case(seed=0, cache=(70, 5, 130), rows_per_agent=3, heads=12, kv_heads=2):
    w = synth.AttnWorkload(cache=cache, rows_per_agent=rows_per_agent, heads=heads, kv_heads=kv_heads)
    table, total, ra, rl = w.build(seed)
    pool = synth.kv_pool(total, kv_heads, seed, 40)
    q = synth.attn_q(len(ra), heads, seed, 41)
    return pool, table, q, ra, rl, kv_heads


def _single_token_holds(attn, pool, table, q, kvh):
    ra = np.array([0, 1], dtype=np.int32)
    rl = np.array([1, 1], dtype=np.int32)
    out, s = attn(pool, table, q[:2], ra, rl, kvh)
    _, v = decode_records(pool, kvh)
    group = q.shape[1] // kvh
    for r in range(2):
        for h in range(q.shape[1]):
            if not np.array_equal(out[r, h], v[table[ra[r], 0], h // group, 0]):
                return False
    return True


def _zero_k_holds(attn, pool, table, q, kvh):
    pool = pool.copy()
    recs = pool.reshape(-1, kvh, REC)
    recs[:, :, :8192] = 0
    ra = np.array([0], dtype=np.int32)
    rl = np.array([70], dtype=np.int32)
    out, _ = attn(pool, table, q[:1], ra, rl, kvh)
    group = q.shape[1] // kvh
    for h in (0, q.shape[1] - 1):
        g = h // group
        for d in (0, 31, 32, 127):
            total = Fraction(0)
            for t in range(70):
                rec = recs[table[0, t // PT], g]
                qv = int(rec[8704 + d * PT + t % PT].astype(np.int8))
                sc = Fraction(float(rec[16896 + 2 * ((d // 32) * PT + t % PT):][:2].copy().view(np.float16)[0]))
                total += sc * qv
            if abs(Fraction(out[0, h, d]) - total / 70) > Fraction(1, 10**12) * (1 + abs(total)):
                return False
    return True


def _brute_force_holds(attn, pool, table, q, ra, rl, kvh):
    out, s = attn(pool, table, q, ra, rl, kvh)
    ref = reference(pool, table, q, ra, rl, kvh)
    return bool(np.all(np.abs(out - ref) <= 1e-12 * (1 + np.abs(ref))))


def _paging_holds(attn, pool, table, q, ra, rl, kvh):
    out, _ = attn(pool, table, q, ra, rl, kvh)
    npages = pool.size // (kvh * REC)
    perm = np.random.default_rng(9).permutation(npages)
    moved = np.empty_like(pool).reshape(npages, kvh * REC)
    moved[perm] = pool.reshape(npages, kvh * REC)
    out2, _ = attn(moved.ravel(), perm[table].astype(np.int32), q, ra, rl, kvh)
    return np.array_equal(out, out2)


def _causal_holds(attn, pool, table, q, ra, rl, kvh):
    out, _ = attn(pool, table, q, ra, rl, kvh)
    pool2 = pool.copy()
    recs = pool2.reshape(-1, kvh, REC)
    # token 71 of agent 0 (row 0 attends to 71 tokens: 0..70): scramble its K and V quants
    p, slot = table[0, 71 // PT], 71 % PT
    recs[p, :, slot * D:(slot + 1) * D] ^= 0x55  # the token's whole (permuted) K row
    recs[p, :, 8704 + slot:8704 + 8192:PT] ^= 0x55
    out2, _ = attn(pool2, table, q, ra, rl, kvh)
    return np.array_equal(out[0], out2[0]) and not np.array_equal(out[1], out2[1])


def _gqa_holds(attn, pool, table, q, ra, rl, kvh):
    group = q.shape[1] // kvh
    q2 = q.copy()
    q2[:, 1] = q2[:, 0]          # heads 0 and 1 share KV head 0
    q2[:, group] = q2[:, 0]      # head `group` reads KV head 1
    out, _ = attn(pool, table, q2, ra, rl, kvh)
    return np.array_equal(out[:, 0], out[:, 1]) and not np.allclose(out[:, 0], out[:, group])


def all_pins_hold(attn) -> bool:
    pool, table, q, ra, rl, kvh = small_case()
    return (_single_token_holds(attn, pool, table, q, kvh) and _zero_k_holds(attn, pool, table, q, kvh)
            and _brute_force_holds(attn, pool, table, q, ra, rl, kvh)
            and _paging_holds(attn, pool, table, q, ra, rl, kvh)
            and _causal_holds(attn, pool, table, q, ra, rl, kvh)
            and _gqa_holds(attn, pool, table, q, ra, rl, kvh))


def test_single_token_returns_its_v():
    pool, table, q, ra, rl, kvh = small_case()
    assert _single_token_holds(oracle.attn, pool, table, q, kvh)


def test_zero_k_gives_the_mean_of_v():
    pool, table, q, ra, rl, kvh = small_case()
    assert _zero_k_holds(oracle.attn, pool, table, q, kvh)


@pytest.mark.parametrize("seed,heads,kvh", [(0, 12, 2), (1, 8, 8), (2, 6, 1)])
def test_brute_force_small(seed, heads, kvh):
    pool, table, q, ra, rl, kvh = small_case(seed, heads=heads, kv_heads=kvh)
    assert _brute_force_holds(oracle.attn, pool, table, q, ra, rl, kvh)


def test_page_placement_does_not_matter():
    pool, table, q, ra, rl, kvh = small_case()
    assert _paging_holds(oracle.attn, pool, table, q, ra, rl, kvh)


def test_tokens_past_a_row_do_not_matter():
    pool, table, q, ra, rl, kvh = small_case()
    assert _causal_holds(oracle.attn, pool, table, q, ra, rl, kvh)


def test_grouped_heads_share_kv():
    pool, table, q, ra, rl, kvh = small_case()
    assert _gqa_holds(oracle.attn, pool, table, q, ra, rl, kvh)


def test_abs_sum_bounds_output():
    pool, table, q, ra, rl, kvh = small_case()
    out, s = oracle.attn(pool, table, q, ra, rl, kvh)
    assert np.all(np.abs(out) <= s * (1 + 1e-12))


MUTANTS = {
    "no_score_scale": ("s[t] = dot / sqrt((double)ATTN_D);", "s[t] = dot;"),
    "v_not_transposed": ("(int8_t)base[d * ATTN_PT + slot]", "(int8_t)base[slot * ATTN_D + d]"),
    "scale_block_16": ("2 * (slot * 4 + d / 32)", "2 * (slot * 4 + (d / 16) % 4)"),
    "k_pieces_unpermuted": ("16 * ((d / 16) ^ (2 * (slot % 4) + (slot / 4) % 2)) + d % 16", "d"),
    "k_piece_key_plain": ("(2 * (slot % 4) + (slot / 4) % 2)", "(slot % 8)"),
    "v_scales_token_major": ("2 * ((d / 32) * ATTN_PT + slot)", "2 * (slot * 4 + d / 32)"),
    "one_token_short": ("for (int t = 0; t < len; ++t) {\n                const uint8_t* rec = pool + ((size_t)page_table[a * max_pages + t / ATTN_PT] * Hkv + g) * ATTN_REC;\n                const double p",
                        "for (int t = 0; t < len - 1; ++t) {\n                const uint8_t* rec = pool + ((size_t)page_table[a * max_pages + t / ATTN_PT] * Hkv + g) * ATTN_REC;\n                const double p"),
    "gqa_modulo": ("const int g = h / group,", "const int g = h % Hkv,"),
    "page_slot_shift": ("oracle_kv(rec, 0, t % ATTN_PT, d)", "oracle_kv(rec, 0, (t + 1) % ATTN_PT, d)"),
    "v_scale_from_k": ("sc = base + 8192 + 2 * ((d / 32) * ATTN_PT + slot);", "sc = rec + 8192 + 2 * ((d / 32) * ATTN_PT + slot);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_fail(tmp_path, name):
    here = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = open(os.path.join(here, "oracle", "attn_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    c = tmp_path / "attn.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / "attn.so"
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", str(c),
                           os.path.join(here, "oracle", "q4k_oracle.c"), "-o", str(so), "-lm"])
    lib = ctypes.CDLL(str(so))
    lib.oracle_attn.restype = ctypes.c_int
    lib.oracle_attn.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int] + [ctypes.c_void_p] * 3 + \
        [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2 + [ctypes.c_int]

    def attn(pool, table, q, ra, rl, kvh):
        pool = np.ascontiguousarray(pool, dtype=np.uint8)
        table = np.ascontiguousarray(table, dtype=np.int32)
        q = np.ascontiguousarray(q, dtype=np.float16)
        ra = np.ascontiguousarray(ra, dtype=np.int32)
        rl = np.ascontiguousarray(rl, dtype=np.int32)
        out = np.empty(q.shape)
        s = np.empty(q.shape)
        assert lib.oracle_attn(pool.ctypes.data, table.ctypes.data, table.shape[1], q.view(np.uint16).ctypes.data,
                               ra.ctypes.data, rl.ctypes.data, q.shape[0], q.shape[1], kvh, out.ctypes.data,
                               s.ctypes.data, 1) == 0
        return out, s

    assert not all_pins_hold(attn), f"planted mistake {name} passed every pin"


def test_real_oracle_passes_the_mutant_checks():
    assert all_pins_hold(oracle.attn)
