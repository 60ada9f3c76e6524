"""Stacked-row decode attention over a paged q8_0 KV pool (qmm_attn_decode) against the
oracle, through the C ABI.  Tolerance per element: |o - o_ref| <= 2e-3 * sum_t p_t |v_t| +
1e-6 (K and V are exact in fp16 as int8 quants with fp32 scaling of the scores; the
probabilities times the V scales go to the tensor core in fp16)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import torch_cuda

pytestmark = pytest.mark.gpu


def agent_rows_of(ra, agents):
    """[agents + 1] row offsets of agent-major rows."""
    return np.concatenate([[0], np.cumsum(np.bincount(np.asarray(ra), minlength=agents))]).astype(np.int32)


def run_attn(pool, table, q, ra, rl, kvh, agent_rows=None, max_agent_rows=0):
    from bit_weight_streaming_q4_gb300.qmm import attn_decode
    torch = torch_cuda()
    table = np.ascontiguousarray(table, dtype=np.int32)
    if agent_rows is None:
        agent_rows = agent_rows_of(ra, table.shape[0])
    pool_d = torch.from_numpy(pool).cuda()
    table_d = torch.from_numpy(table).cuda()
    ar_d = torch.from_numpy(np.ascontiguousarray(agent_rows, dtype=np.int32)).cuda()
    rl_d = torch.from_numpy(np.ascontiguousarray(rl, dtype=np.int32)).cuda()
    q_d = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).cuda().view(torch.float16)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    err = attn_decode(pool_d, table_d, ar_d, rl_d, q_d, out, kvh, max_agent_rows=max_agent_rows)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


def case(cache, rows_per_agent, heads, kvh, seed=0):
    w = synth.AttnWorkload(cache=cache, rows_per_agent=rows_per_agent, heads=heads, kv_heads=kvh)
    table, total, ra, rl = w.build(seed)
    pool = synth.kv_pool(total, kvh, seed, 50)
    q = synth.attn_q(len(ra), heads, seed, 51)
    return pool, table, q, ra, rl, kvh


def check(pool, table, q, ra, rl, kvh, what=""):
    got, err = run_attn(pool, table, q, ra, rl, kvh)
    assert err == 0
    ref, s = oracle.attn(pool, table, q, ra, rl, kvh)
    assert np.all(np.isfinite(got)), what
    bound = 2e-3 * s + 1e-6
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} out of tolerance, worst ratio {(np.abs(got - ref) / bound).max()}"
    return got


CASES = [((70, 5, 130), 3, 12, 2), ((1, 64, 65), 1, 8, 8), ((1000, 2000), 2, 48, 8), ((5000,), 5, 48, 8),
         ((300, 300, 300, 300), 3, 48, 8)]


@pytest.mark.parametrize("cache,rows,heads,kvh", CASES, ids=[f"{c}-r{r}-h{h}/{k}" for c, r, h, k in CASES])
def test_attention_matches_oracle(cache, rows, heads, kvh):
    check(*case(cache, rows, heads, kvh), what=str(cache))


def test_attention_long_context_decode_shape():
    """One agent of the pages' decode step: 23,000 cached tokens (360 pages, 23 work items
    per KV head), 1 token + 2 drafts, 48 query heads over 8 KV heads."""
    check(*case((23000,), 3, 48, 8, seed=1), what="23K")


def test_attention_page_placement_bitwise():
    """Moving the pool's pages (and the page table with them) gives the same bits."""
    pool, table, q, ra, rl, kvh = case((700, 130), 3, 48, 8, seed=2)
    a, _ = run_attn(pool, table, q, ra, rl, kvh)
    npages = pool.size // (kvh * synth.KV_RECORD_BYTES)
    perm = np.random.default_rng(3).permutation(npages)
    moved = np.empty_like(pool).reshape(npages, -1)
    moved[perm] = pool.reshape(npages, -1)
    b, _ = run_attn(moved.ravel(), perm[table].astype(np.int32), q, ra, rl, kvh)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_attention_rows_do_not_depend_on_the_batch():
    """A row's bits do not change when the other agents' rows, or later rows of its own
    agent, are left out of the batch (agents without rows are allowed)."""
    pool, table, q, ra, rl, kvh = case((700, 130, 2500), 3, 48, 8, seed=4)
    full, _ = run_attn(pool, table, q, ra, rl, kvh)
    # agent 1 alone, all three rows
    sel = np.where(ra == 1)[0]
    part, _ = run_attn(pool, table, q[sel], ra[sel], rl[sel], kvh)
    assert np.array_equal(part.view(np.uint32), full[sel].view(np.uint32))
    # agent 2's first row alone
    sel = np.where(ra == 2)[0][:1]
    part, _ = run_attn(pool, table, q[sel], ra[sel], rl[sel], kvh)
    assert np.array_equal(part.view(np.uint32), full[sel].view(np.uint32))


@pytest.mark.parametrize("rows,heads,kvh", [(6, 48, 8), (8, 48, 8), (11, 48, 8), (40, 8, 8)],
                         ids=["36q", "48q-verify", "66q", "40q-mha"])
def test_attention_wide_agents_in_query_tiles(rows, heads, kvh):
    """More than 24 queries per (agent, KV head) run as tiles of 24, each a pass over the
    agent's pages: 6, 8 (the wide-verify step's 1 + 7 drafts) and 11 rows at 6 queries per row
    and KV head, and 40 rows of plain multi-head attention."""
    check(*case((300, 1500), rows, heads, kvh, seed=6), what=f"{rows} rows")


def test_attention_query_tiles_match_narrow_batches():
    """A row computed in the second query tile of a wide agent has the bits it has when its
    agent's batch holds only that row's tile (tiles never mix)."""
    pool, table, q, ra, rl, kvh = case((900,), 8, 48, 8, seed=7)
    full, _ = run_attn(pool, table, q, ra, rl, kvh)
    # 8 rows x 6 heads per KV head = 48 queries: tile 0 holds queries 0..23 (rows 0-3), tile 1
    # holds 24..47 (rows 4-7, rows 6 and 7 at positions 12..23); alone, rows 6 and 7 make one
    # tile, at positions 0..11
    sel = np.arange(6, 8)
    sub = np.ascontiguousarray(q[sel])
    part, _ = run_attn(pool, table, sub, ra[sel], rl[sel], kvh)
    assert np.array_equal(part.view(np.uint32), full[sel].view(np.uint32))


def test_attention_agent_row_bound():
    """With a bound on any agent's rows the workspace and grid hold fewer query tiles; results
    are the same bits, and an agent above the bound is reported (4) with zero outputs while
    the others are computed."""
    pool, table, q, ra, rl, kvh = case((700, 130, 2500), 3, 48, 8, seed=8)
    full, _ = run_attn(pool, table, q, ra, rl, kvh)
    hinted, err = run_attn(pool, table, q, ra, rl, kvh, max_agent_rows=3)
    assert err == 0
    assert np.array_equal(hinted.view(np.uint32), full.view(np.uint32))
    pool, table, q, ra, rl, kvh = case((700, 130), 6, 48, 8, seed=9)
    keep = np.r_[np.where(ra == 0)[0], np.where(ra == 1)[0][:3]]  # 6 rows of agent 0, 3 of agent 1
    got, err = run_attn(pool, table, q[keep], ra[keep], rl[keep], kvh, max_agent_rows=4)
    assert err & 4
    assert np.all(got[:6] == 0)
    ref, s = oracle.attn(pool, table, q[keep[6:]], ra[keep[6:]], rl[keep[6:]], kvh)
    assert np.all(np.abs(got[6:] - ref) <= 2e-3 * s + 1e-6)


def test_attention_bad_page_is_reported():
    """A page-table entry outside the pool sets the error word (2); nothing is read there."""
    pool, table, q, ra, rl, kvh = case((200,), 2, 16, 8, seed=5)
    table = table.copy()
    table[0, 1] = 10**6
    _, err = run_attn(pool, table, q, ra, rl, kvh)
    assert err & 2


def _set_scales(pool, kvh, which, values):
    """Overwrite the K (which = 0) or V (which = 1) block scales of every record."""
    recs = pool.reshape(-1, synth.KV_RECORD_BYTES)
    off = 8192 if which == 0 else 16896
    recs[:, off:off + 512] = values.astype(np.float16).view(np.uint8).reshape(len(recs), 512)


def test_attention_peaked_softmax():
    """Queries scaled by 24 make the softmax nearly one-hot (score gaps of tens), the case where
    the running maximum moves most between pages."""
    pool, table, q, ra, rl, kvh = case((900, 3000), 3, 48, 8, seed=10)
    q = (q.astype(np.float32) * 24).astype(np.float16)
    check(pool, table, q, ra, rl, kvh, what="peaked")


def test_attention_v_scales_near_the_bound():
    """V block scales up to 250 (the documented bound is 255: probabilities carry 2^8) and K
    scales spread over four decades."""
    pool, table, q, ra, rl, kvh = case((700, 1500), 3, 48, 8, seed=11)
    n = pool.size // synth.KV_RECORD_BYTES
    rng = np.random.default_rng(11)
    _set_scales(pool, kvh, 1, rng.uniform(100.0, 250.0, size=(n, 256)))
    _set_scales(pool, kvh, 0, 10.0 ** rng.uniform(-4.0, 0.0, size=(n, 256)))
    check(pool, table, q, ra, rl, kvh, what="large V scales")


def test_attention_misaligned_output_is_refused():
    from bit_weight_streaming_q4_gb300.qmm import attn_decode
    torch = torch_cuda()
    pool, table, q, ra, rl, kvh = case((100,), 2, 16, 8, seed=12)
    buf = torch.zeros(q.size + 1, dtype=torch.float32, device="cuda")
    out = buf[1:].view(q.shape)  # 4 bytes past a 16-byte boundary
    with pytest.raises(RuntimeError):
        attn_decode(torch.from_numpy(pool).cuda(), torch.from_numpy(np.ascontiguousarray(table)).cuda(),
                    torch.from_numpy(agent_rows_of(ra, table.shape[0])).cuda(), torch.from_numpy(rl).cuda(),
                    torch.from_numpy(q.view(np.int16)).cuda().view(torch.float16), out, kvh)
