// Stacked-row decode attention over a paged q8_0 KV pool.
//
// The method (page "Running 4 coding agents on one RTX 3090: a custom CUDA engine for
// Qwen3.8-27B", section "How parallel decoding works"): a decode step stacks every agent's
// next token and its drafts into one batch of rows; the weights are shared by all rows, but
// attention is per agent, each agent's rows reading that agent's own KV cache, kept in one
// shared pool of q8_0 entries in pages.  For row r of agent a and query head h:
//
//   out[r][h] = softmax_t(q[r][h] . k_t / sqrt(128)) . v_t,   t < len[r],
//
// with k_t, v_t of KV head g = h / (heads / kv_heads).  The rows of one agent attend to the
// same tokens (each to a prefix of them), so every KV byte is read once per step for all of
// the agent's rows and all heads of the group.
//
// Pool record (page P, KV head g) of 17,408 bytes at (P * kv_heads + g) * 17408: K quants
// int8 in 128-byte token rows (16-byte piece p of token t's row stored at position
// p ^ (2 (t % 4) + (t / 4) % 2)), K scales fp16 [token 64][4], V quants int8
// [dim 128][token 64], V scales fp16 [4][token 64]; an element is scale * quant, with the
// scale of its 32-dim block (q8_0).  The layout makes every shared-memory read of the kernel
// below a conflict-free 8- or 16-byte load.
//
// Kernel 1, one CTA of 4 warps per work item (agent, KV head, run of up to 32 pages; the
// grid covers every agent x KV head x 32-page run of the page table, and a CTA whose run lies
// past its agent's longest row returns at once, so the plan needs no host work):
// the item's queries (the agent's rows x the group's heads, at most 32) are the A operand of
// mma.sync m16n8k16.  Pages stream into a 4-slot ring by bulk copies.  Per page, warp w
// computes the scores of tokens 16w .. 16w+15 against raw int8 K (exact in fp16), one 32-dim
// block at a time, and applies each block's scale to the block's partial sums in fp32.  The
// page's row maxima are combined through shared memory (an online softmax), the fp16
// probabilities go to shared memory, and warp w then accumulates P . V for dims 32w..32w+31
// (one scale block): A = P times the token's V scale (fp16), B = raw int8 V.  The item's
// (max, sum, unnormalised output) per query goes to the workspace.
// Kernel 2 combines the items of each (agent, KV head) in item order.
#include <cstring>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qmm.h"
#include "qmm_internal.h"
#include "qmm_ptx.cuh"

namespace qmm {
namespace attn {

constexpr int kD = 128, kPT = 64, kRec = 17408;
constexpr int kMaxQ = 24;   // queries per tile (an agent's rows x the group's heads, 24 at a time)
constexpr int kNT = kMaxQ / 8;  // n8 tiles of queries per tile
constexpr int kSlotCap = 1024;  // upper bound on the resident CTAs a launch is planned for
constexpr int kStages = 3;  // pages in flight per CTA (4 CTAs per SM keep 8 in flight)
constexpr int kThreads = 128;
constexpr int kPart = kD + 4;  // floats per query of an item's partial: o[128], m, l, 2 unused (16-byte rows)
constexpr float kNegBig = -1e30f;
constexpr int kPS = kPT + 4;  // halves per row of the probability tile (136 bytes: conflict-free 8-byte reads)

struct Item {
    int32_t agent, g;      // agent, KV head
    int32_t page0, npages; // logical pages page0 .. page0 + npages - 1 of the agent
    int32_t r0, nr;        // the agent's rows r0 .. r0 + nr - 1
};

struct Params {
    const uint8_t* pool;
    int64_t pool_pages;
    const int32_t* table;       // [agents][max_pages]
    int32_t max_pages;
    const __half* q;            // [rows][heads][128]
    const int32_t* row_len;     // [rows]
    const int32_t* agent_rows;  // [agents + 1]: agent a's rows are agent_rows[a] .. agent_rows[a+1] - 1
    int32_t heads, kv_heads, group;
    int32_t agents;
    int32_t runs, chunk;        // runs of pages per (agent, KV head), pages per run
    int32_t max_qt;             // query tiles of kMaxQ per (agent, KV head) the workspace holds
    float* ws;                  // [agent][kv head][run][query tile][kMaxQ][kPart]
    int* err;                   // sticky error word
    float* out;                 // [rows][heads][128]
    int64_t rows;
};

// Agent a's rows (r0, nr) and its number of runs of p.chunk pages, or -1 runs (and the error word)
// if its rows or lengths are outside what the kernels handle.
__device__ __forceinline__ int agent_runs(const Params& p, int a, int& r0, int& nr) {
    r0 = p.agent_rows[a];
    nr = p.agent_rows[a + 1] - r0;
    if (nr <= 0) return 0;
    if (r0 < 0 || r0 + nr > p.rows || nr * p.group > p.max_qt * kMaxQ) return -1;
    int maxlen = 0;
    for (int r = r0; r < r0 + nr; ++r) {
        const int len = p.row_len[r];
        if (len < 1 || len > p.max_pages * kPT) return -1;
        maxlen = len > maxlen ? len : maxlen;
    }
    const int pages = (maxlen + kPT - 1) / kPT;
    return (pages + p.chunk - 1) / p.chunk;
}

// Bytes 0, 1 (sel 0x4140) or 2, 3 (sel 0x4342) of four int8 already XORed with 0x80, as
// fp16x2, exact: the biased byte goes into the mantissa of 1024, and 1024 + 128 comes off.
__device__ __forceinline__ uint32_t i8pair_to_h2(uint32_t biased, uint32_t sel) {
    return as_u32(__hadd2(as_h2(prmt(biased, 0x64646464u, sel)), as_h2(0xE480E480u)));
}

// 2^x (the ex2 instruction, flush to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// d = A.B with a zero accumulator.
__device__ __forceinline__ void mma_m16n8k16_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

__global__ void __launch_bounds__(kThreads, 4) attn_partial(const Params p) {
    extern __shared__ __align__(128) uint8_t sm[];
    // the combine kernel may be scheduled as soon as every CTA of this grid has started; it
    // waits for the whole grid (and its writes) before reading the workspace
    griddep_launch_dependents();
    // ring slot i % kStages holds page i
    __half* P = reinterpret_cast<__half*>(sm + kStages * kRec);       // [kMaxQ][kPS] probabilities
    float* red_max = reinterpret_cast<float*>(P + kMaxQ * kPS);       // [kMaxQ][4 warps]
    float* red_sum = red_max + 4 * kMaxQ;                              // [kMaxQ][4 warps]
    uint64_t* bar = reinterpret_cast<uint64_t*>(red_sum + 4 * kMaxQ);  // [kStages]
    volatile int* flags = reinterpret_cast<volatile int*>(bar + kStages);  // [0] abort
    int* qlen_sm = const_cast<int*>(reinterpret_cast<volatile int*>(flags + 4));  // [kMaxQ] tokens per query

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    // this CTA's work item
    Item it;
    it.agent = blockIdx.x / (p.kv_heads * p.runs);
    it.g = (blockIdx.x / p.runs) % p.kv_heads;
    const int run = blockIdx.x % p.runs;
    int minlen = 0;  // the shortest row of the item: pages below it need no mask
    {
        const int runs = agent_runs(p, it.agent, it.r0, it.nr);
        if (runs < 0) {
            if (threadIdx.x == 0 && run == 0 && it.g == 0) atomicOr(p.err, 4);
            return;
        }
        if (run >= runs) return;
        int maxlen = 0;
        minlen = p.row_len[it.r0];
        for (int r = it.r0; r < it.r0 + it.nr; ++r) {
            maxlen = p.row_len[r] > maxlen ? p.row_len[r] : maxlen;
            minlen = p.row_len[r] < minlen ? p.row_len[r] : minlen;
        }
        const int pages = (maxlen + kPT - 1) / kPT;
        it.page0 = run * p.chunk;
        it.npages = pages - it.page0 < p.chunk ? pages - it.page0 : p.chunk;
    }
    // this CTA's query tile: the item's queries q0 .. q0 + nq - 1 (blockIdx.y = tile)
    const int q0 = static_cast<int>(blockIdx.y) * kMaxQ;
    const int nq = it.nr * p.group - q0 < kMaxQ ? it.nr * p.group - q0 : kMaxQ;
    if (nq <= 0) return;
    const int nnt = (nq + 7) >> 3;  // n8 tiles of queries (1 .. kNT)
    const float c2 = 1.4426950408889634f * 0.08838834764831845f;  // log2(e) / sqrt(128)

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&bar[i], 1);
        flags[0] = 0;
        fence_mbar_init();
    }
    if (tid < kMaxQ) qlen_sm[tid] = tid < nq ? p.row_len[it.r0 + (q0 + tid) / p.group] : 0;
    __syncthreads();

    // the record of logical page i of the item, or null (and the error word) if the page
    // table points outside the pool
    auto record = [&](int i) -> const uint8_t* {
        const int32_t pg = p.table[static_cast<int64_t>(it.agent) * p.max_pages + it.page0 + i];
        if (pg < 0 || pg >= p.pool_pages) return nullptr;
        return p.pool + (static_cast<int64_t>(pg) * p.kv_heads + it.g) * kRec;
    };
    int issued = 0;  // thread 0: copies issued (page i: slot i % kStages, phase i / kStages)
    auto issue = [&](int i) {
        const uint8_t* src = record(i);
        uint64_t* b = &bar[i % kStages];
        ++issued;
        if (!src) {
            flags[0] = 1;
            atomicOr(p.err, 2);
            mbar_arrive(b);  // completes the phase without data; the abort flag stops its use
            return;
        }
        // (a refill: every warp's generic reads of the slot, ordered by the CTA barrier before
        // this, precede the bulk write)
        if (i >= kStages) fence_proxy_async_smem();
        mbar_arrive_expect_tx(b, kRec);
        bulk_g2s(sm + (i % kStages) * kRec, src, kRec, b, l2_policy_evict_first());
    };
    if (tid == 0)
        for (int i = 0; i < kStages - 1 && i < it.npages; ++i) issue(i);

    // Both products run with tokens or dims as the MMA's M and the item's queries as N (n8
    // tiles nt: queries 8 nt .. 8 nt + 7 of the CTA's tile; its query qi is the item's query
    // qa = q0 + qi, head g * group + qa % group of row r0 + qa / group, and queries past nq
    // are zero).
    //
    // S^T = K . Q^T: warp w takes tokens 16w .. 16w + 15 of the page.  The dims of k-step
    // ks = 2 blk + k2 are assigned so that every thread's eight dims of a 32-dim block are
    // contiguous: k-slots (2t, 2t+1) are dims 32 blk + 8t + 4 k2 + {0, 1}, slots (2t+8, 2t+9)
    // dims 32 blk + 8t + 4 k2 + {2, 3}.  qb holds Q^T's B fragments for all k-steps.
    uint32_t qb[kNT][8][2];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
        const int qi = 8 * nt + g8;
        const __half* qrow = nullptr;
        if (qi < nq) {
            const int qa = q0 + qi;  // the item's query
            qrow = p.q + (static_cast<int64_t>(it.r0 + qa / p.group) * p.heads + it.g * p.group + qa % p.group) * kD;
        }
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
            const uint4 v = qrow ? *reinterpret_cast<const uint4*>(qrow + 32 * blk + 8 * t4) : make_uint4(0u, 0u, 0u, 0u);
            qb[nt][2 * blk][0] = v.x;
            qb[nt][2 * blk][1] = v.y;
            qb[nt][2 * blk + 1][0] = v.z;
            qb[nt][2 * blk + 1][1] = v.w;
        }
    }

    // Running state per accumulator column: the maximum score, the thread's share of the
    // sum of probabilities, and O^T (dims 32w + 16 mt + {g8, g8 + 8}).  Probabilities carry a
    // factor 2^8 (kept in the sum too) so that P times a V scale stays clear of the fp16
    // subnormal range.
    float m_run[kNT][2], l_part[kNT][2];
    float o[2][kNT][4];  // [m16 tile of dims][n8 tile of queries][accumulator]
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            m_run[nt][e] = kNegBig;
            l_part[nt][e] = 0.f;
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) o[mt][nt][c] = 0.f;
    }

    const int t0 = 16 * warp + g8;                           // the thread's tokens t0, t0 + 8
    const int kkey = 2 * (g8 & 3) + ((g8 >> 2) & 1);          // K piece key of both (t0 % 8 == g8)
    bool live = true;
    int consumed = 0;
    for (int i = 0; i < it.npages; ++i) {
        const bool ok = mbar_wait_bounded(&bar[i % kStages], (i / kStages) & 1, flags);
        const uint8_t* rec = sm + (i % kStages) * kRec;
        const int tbase = (it.page0 + i) * kPT;  // logical index of the page's first token

        // ---- scores s[nt][c]: c0 (token t0, query 8nt + 2t4), c1 (t0, +1), c2 (t0 + 8, ..), c3
        float s[kNT][4];
        {
            const uint2 sca = *reinterpret_cast<const uint2*>(rec + 8192 + t0 * 8);
            const uint2 scb = *reinterpret_cast<const uint2*>(rec + 8192 + (t0 + 8) * 8);
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                const uint8_t* kr = rec + t0 * kD + 16 * ((2 * blk + (t4 >> 1)) ^ kkey) + 8 * (t4 & 1);
                const uint2 ka = *reinterpret_cast<const uint2*>(kr);
                const uint2 kb = *reinterpret_cast<const uint2*>(kr + 8 * kD);
                const uint32_t xa = ka.x ^ 0x80808080u, ya = ka.y ^ 0x80808080u;
                const uint32_t xb = kb.x ^ 0x80808080u, yb = kb.y ^ 0x80808080u;
                // A fragments of k-steps 2 blk (from .x) and 2 blk + 1 (from .y)
                const uint32_t a00 = i8pair_to_h2(xa, 0x4140u), a01 = i8pair_to_h2(xb, 0x4140u);
                const uint32_t a02 = i8pair_to_h2(xa, 0x4342u), a03 = i8pair_to_h2(xb, 0x4342u);
                const uint32_t a10 = i8pair_to_h2(ya, 0x4140u), a11 = i8pair_to_h2(yb, 0x4140u);
                const uint32_t a12 = i8pair_to_h2(ya, 0x4342u), a13 = i8pair_to_h2(yb, 0x4342u);
                const uint32_t wa = (blk >> 1) ? sca.y : sca.x, wb = (blk >> 1) ? scb.y : scb.x;
                const float sa = __half2float((blk & 1) ? __high2half(as_h2(wa)) : __low2half(as_h2(wa)));
                const float sb = __half2float((blk & 1) ? __high2half(as_h2(wb)) : __low2half(as_h2(wb)));
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
                    if (nt < nnt) {
                        float tmp[4];
                        mma_m16n8k16_z(tmp, a00, a01, a02, a03, qb[nt][2 * blk][0], qb[nt][2 * blk][1]);
                        mma_m16n8k16(tmp, a10, a11, a12, a13, qb[nt][2 * blk + 1][0], qb[nt][2 * blk + 1][1]);
                        if (blk == 0) {
                            s[nt][0] = tmp[0] * sa;
                            s[nt][1] = tmp[1] * sa;
                            s[nt][2] = tmp[2] * sb;
                            s[nt][3] = tmp[3] * sb;
                        } else {
                            s[nt][0] = fmaf(tmp[0], sa, s[nt][0]);
                            s[nt][1] = fmaf(tmp[1], sa, s[nt][1]);
                            s[nt][2] = fmaf(tmp[2], sb, s[nt][2]);
                            s[nt][3] = fmaf(tmp[3], sb, s[nt][3]);
                        }
                    }
                }
            }
        }
        // ---- masks (only on pages reaching past the shortest row) and the warp's maxima
        if (tbase + kPT > minlen) {
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    if (nt < nnt) {
                        const int len = qlen_sm[8 * nt + 2 * t4 + e];
                        if (tbase + t0 >= len) s[nt][e] = kNegBig;
                        if (tbase + t0 + 8 >= len) s[nt][2 + e] = kNegBig;
                    }
                }
        }
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if (nt < nnt) {
                    float mx = fmaxf(s[nt][e], s[nt][2 + e]);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    if (g8 == 0) red_max[(8 * nt + 2 * t4 + e) * 4 + warp] = mx;
                }
            }
        // one decision for the whole CTA (every thread reaches this barrier); the scores of a
        // page whose wait failed are never used
        if (__syncthreads_or(!ok || flags[0])) {
            live = false;
            break;
        }
        consumed = i + 1;
        // every warp is past page i - 1: its slot takes page i + kStages - 1
        if (tid == 0 && i + kStages - 1 < it.npages) issue(i + kStages - 1);

        // ---- new maxima, rescaling, probabilities (x 2^8, fp16) to shared memory
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            if (nt < nnt) {
                float pr[4];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float4 rm = *reinterpret_cast<const float4*>(red_max + (8 * nt + 2 * t4 + e) * 4);
                    const float mn = fmaxf(fmaxf(m_run[nt][e], fmaxf(rm.x, rm.y)), fmaxf(rm.z, rm.w));
                    const float alpha = ex2((m_run[nt][e] - mn) * c2);
                    const float mc2 = mn == kNegBig ? __int_as_float(0x7f800000) : fmaf(mn, c2, -8.f);
                    pr[e] = ex2(fmaf(s[nt][e], c2, -mc2));
                    pr[2 + e] = ex2(fmaf(s[nt][2 + e], c2, -mc2));
                    l_part[nt][e] = fmaf(l_part[nt][e], alpha, pr[e] + pr[2 + e]);
                    m_run[nt][e] = mn;
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        o[mt][nt][e] *= alpha;
                        o[mt][nt][2 + e] *= alpha;
                    }
                }
                // P[query][token]: lanes g8 and g8 ^ 1 swap values so that each stores two
                // consecutive tokens of one query (even g8: query 2t4, odd: query 2t4 + 1)
                const bool odd = g8 & 1;
                const uint32_t mine_lo = as_u32(__floats2half2_rn(pr[0], pr[1]));  // (t0, q), (t0, q+1)
                const uint32_t mine_hi = as_u32(__floats2half2_rn(pr[2], pr[3]));  // (t0+8, q), (t0+8, q+1)
                // even sends its q+1 values, odd its q values: (token t0, token t0 + 8)
                const uint32_t send = odd ? prmt(mine_lo, mine_hi, 0x5410u) : prmt(mine_lo, mine_hi, 0x7632u);
                const uint32_t got = __shfl_xor_sync(0xffffffffu, send, 4);
                // even: (own q of t0, partner's q of t0 + 1), and the same for t0 + 8
                // odd:  (partner's q+1 of t0 - 1, own q+1 of t0), and the same for t0 + 7
                const uint32_t lo = odd ? prmt(got, mine_lo, 0x7610u) : prmt(mine_lo, got, 0x5410u);
                const uint32_t hi = odd ? prmt(got, mine_hi, 0x7632u) : prmt(mine_hi, got, 0x7610u);
                const int qrow = 8 * nt + 2 * t4 + (odd ? 1 : 0);
                const int tcol = odd ? t0 - 1 : t0;
                *reinterpret_cast<uint32_t*>(P + qrow * kPS + tcol) = lo;
                *reinterpret_cast<uint32_t*>(P + qrow * kPS + tcol + 8) = hi;
            }
        }
        __syncthreads();  // P complete

        // ---- O^T += V^T . (P x V scale)^T for dims 32w .. 32w + 31 (one V scale block).
        // Tokens of k-step ks are assigned so that every thread's sixteen tokens are
        // contiguous: k-slots (2t, 2t+1) are tokens 16t + 4 ks + {0, 1}, slots (2t+8, 2t+9)
        // tokens 16t + 4 ks + {2, 3}.
        {
            uint32_t wv[2][2][4];  // raw V: [m16 tile][row g8 / g8 + 8][word ks], biased
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 v = *reinterpret_cast<const uint4*>(rec + 8704 + (32 * warp + 16 * mt + 8 * h + g8) * kPT + 16 * t4);
                    wv[mt][h][0] = v.x ^ 0x80808080u;
                    wv[mt][h][1] = v.y ^ 0x80808080u;
                    wv[mt][h][2] = v.z ^ 0x80808080u;
                    wv[mt][h][3] = v.w ^ 0x80808080u;
                }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                // V scales of tokens 16 t4 + 4 ks .. + 3 (this warp's block)
                const uint2 dv = *reinterpret_cast<const uint2*>(rec + 16896 + (warp * kPT + 16 * t4 + 4 * ks) * 2);
                uint32_t pb[kNT][2];  // B fragments: (P x V scale) of query 8 nt + g8, the k-step's tokens
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
                    if (nt < nnt) {
                        const uint2 pw = *reinterpret_cast<const uint2*>(P + (8 * nt + g8) * kPS + 16 * t4 + 4 * ks);
                        pb[nt][0] = as_u32(__hmul2(as_h2(pw.x), as_h2(dv.x)));
                        pb[nt][1] = as_u32(__hmul2(as_h2(pw.y), as_h2(dv.y)));
                    }
                }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const uint32_t a0 = i8pair_to_h2(wv[mt][0][ks], 0x4140u), a2 = i8pair_to_h2(wv[mt][0][ks], 0x4342u);
                    const uint32_t a1 = i8pair_to_h2(wv[mt][1][ks], 0x4140u), a3 = i8pair_to_h2(wv[mt][1][ks], 0x4342u);
#pragma unroll
                    for (int nt = 0; nt < kNT; ++nt)
                        if (nt < nnt) mma_m16n8k16(o[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                }
            }
        }
    }
    if (!live) {
        if (tid == 0) {
            atomicOr(p.err, 1);
            // let every copy still in flight land before the CTA exits
            volatile int no_abort = 0;
            for (int j = consumed; j < issued; ++j) mbar_wait_bounded(&bar[j % kStages], (j / kStages) & 1, &no_abort);
        }
        return;
    }

    // ---- the item's partial: o, m and l per query
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            if (nt < nnt) {
                float l = l_part[nt][e];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                if (g8 == 0) red_sum[(8 * nt + 2 * t4 + e) * 4 + warp] = l;
            }
        }
    __syncthreads();
    // slot (agent, g, run, tile)
    float* part = p.ws + (static_cast<int64_t>(blockIdx.x) * p.max_qt + blockIdx.y) * kMaxQ * kPart;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int qi = 8 * nt + 2 * t4 + e;
            if (nt >= nnt || qi >= nq) continue;
            float* pq = part + qi * kPart;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int dim = 32 * warp + 16 * mt + g8;
                pq[dim] = o[mt][nt][e];
                pq[dim + 8] = o[mt][nt][2 + e];
            }
            if (warp == 0 && g8 == 0) {
                const float4 ls = *reinterpret_cast<const float4*>(red_sum + qi * 4);
                pq[kD] = m_run[nt][e];
                pq[kD + 1] = (ls.x + ls.y) + (ls.z + ls.w);
            }
        }
}

// One warp per (row, head): the partials of its (agent, KV head, query tile) merged in run
// order; lane l writes dims 4l .. 4l + 3.
__global__ void attn_combine(const Params p) {
    griddep_wait();  // the partial kernel has finished and its partials are visible
    const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= p.rows * p.heads) return;
    const int h = static_cast<int>(w % p.heads);
    const int64_t r = w / p.heads;
    float4* outp = reinterpret_cast<float4*>(p.out + w * kD);
    // the agent holding row r (agent_rows is non-decreasing)
    int lo = 0, hi = p.agents;
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (p.agent_rows[mid] <= r) lo = mid;
        else hi = mid;
    }
    const int a = lo;
    int r0, nr;
    const int n = agent_runs(p, a, r0, nr);
    if (n <= 0 || r < r0 || r >= r0 + nr) {  // a row of no agent, or an agent the kernels refused
        if (lane == 0 && h == 0) atomicOr(p.err, 4);
        outp[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    const int g = h / p.group;
    const int qa = static_cast<int>(r - r0) * p.group + h % p.group;  // the item's query
    const int qt = qa / kMaxQ, qi = qa % kMaxQ;                           // its tile, its slot there
    const int64_t first = (static_cast<int64_t>(a) * p.kv_heads + g) * p.runs;
    const float c2 = 1.4426950408889634f * 0.08838834764831845f;
    auto slot = [&](int c) { return p.ws + (((first + c) * p.max_qt + qt) * kMaxQ + qi) * kPart; };
    float m = kNegBig;
    for (int c = lane; c < n; c += 32) m = fmaxf(m, slot(c)[kD]);
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, k));
    // runs in groups of 32: lane j weighs run c0 + j (0 for a run without attended tokens),
    // then the warp adds the group's runs in order, with independent loads of their o rows
    float l = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < n; c0 += 32) {
        const int c = c0 + lane;
        float wt = 0.f, lw = 0.f;
        if (c < n) {
            const float* pq = slot(c);
            const float mc = pq[kD];
            if (mc != kNegBig) {
                wt = exp2f((mc - m) * c2);
                lw = pq[kD + 1] * wt;
            }
        }
        const int cn = n - c0 < 32 ? n - c0 : 32;
#pragma unroll 4
        for (int j = 0; j < cn; ++j) {
            const float wj = __shfl_sync(0xffffffffu, wt, j);
            l += __shfl_sync(0xffffffffu, lw, j);
            const float4 v = reinterpret_cast<const float4*>(slot(c0 + j))[lane];
            o.x = fmaf(v.x, wj, o.x);
            o.y = fmaf(v.y, wj, o.y);
            o.z = fmaf(v.z, wj, o.z);
            o.w = fmaf(v.w, wj, o.w);
        }
    }
    outp[lane] = make_float4(o.x / l, o.y / l, o.z / l, o.w / l);
}

constexpr int kSmem = kStages * kRec + kMaxQ * kPS * 2 + 2 * 4 * kMaxQ * 4 + kStages * 8 + 16 + kMaxQ * 4;

// Runs per (agent, KV head) and pages per run for a launch on `slots` resident CTAs: the
// runs of a full-width page table fill one wave.  The cut depends only on the dims and the
// device, never on the rows, so a row's result does not depend on the rest of the batch.
void plan_runs(const qmm_attn_dims* dims, int64_t slots, int32_t* runs, int32_t* chunk) {
    const int64_t items = static_cast<int64_t>(dims->agents) * dims->kv_heads;
    const int64_t cap = slots < kSlotCap ? slots : kSlotCap;
    int64_t r = cap / items;
    if (r < 1) r = 1;
    const int64_t c = (dims->max_pages + r - 1) / r;
    *chunk = static_cast<int32_t>(c);
    *runs = static_cast<int32_t>((dims->max_pages + c - 1) / c);
}

// Largest number of runs any device can be planned for (kSlotCap resident CTAs).
int64_t max_runs(const qmm_attn_dims* dims) {
    int32_t runs = 0, chunk = 0;
    plan_runs(dims, kSlotCap, &runs, &chunk);
    return runs;
}

// Query tiles of kMaxQ an agent of a call with `rows` rows can need: all of them, or at most
// dims->max_agent_rows rows in one agent when that bound is given.
int32_t max_tiles(const qmm_attn_dims* dims, int64_t rows) {
    const int64_t r = dims->max_agent_rows > 0 && dims->max_agent_rows < rows ? dims->max_agent_rows : rows;
    const int64_t q = r * (dims->heads / dims->kv_heads);
    return static_cast<int32_t>((q + kMaxQ - 1) / kMaxQ);
}

}  // namespace attn
}  // namespace qmm

extern "C" {

qmm_status qmm_attn_workspace_bytes(const qmm_attn_dims* dims, int64_t rows, int64_t* bytes) {
    if (!dims || !bytes) return QMM_ERR_INVALID_ARG;
    if (dims->heads < 1 || dims->kv_heads < 1 || dims->heads % dims->kv_heads != 0 || dims->agents < 1 ||
        dims->max_pages < 1 || dims->pool_pages < 1 || rows < 1 || rows > (int64_t{1} << 24) ||
        dims->max_agent_rows < 0 || dims->reserved != 0)
        return QMM_ERR_INVALID_ARG;
    *bytes = static_cast<int64_t>(dims->agents) * dims->kv_heads * qmm::attn::max_runs(dims) *
             qmm::attn::max_tiles(dims, rows) * qmm::attn::kMaxQ * qmm::attn::kPart * 4;
    return QMM_OK;
}

qmm_status qmm_attn_decode(const qmm_attn_dims* dims, const void* pool, const int32_t* page_table,
                           const int32_t* agent_rows, const int32_t* row_len, const void* q, int64_t rows, float* out,
                           void* workspace, int64_t workspace_bytes, int* err_word, void* stream) {
    if (!pool || !page_table || !agent_rows || !row_len || !q || !out || !workspace || !err_word || rows < 1)
        return QMM_ERR_INVALID_ARG;
    int64_t need = 0;
    qmm_status st = qmm_attn_workspace_bytes(dims, rows, &need);
    if (st != QMM_OK) return st;
    if ((reinterpret_cast<uintptr_t>(pool) & 15) || (reinterpret_cast<uintptr_t>(q) & 15) ||
        (reinterpret_cast<uintptr_t>(out) & 15) || (reinterpret_cast<uintptr_t>(workspace) & 15))
        return QMM_ERR_MISALIGNED;
    if (workspace_bytes < need) return QMM_ERR_SCRATCH_TOO_SMALL;
    // resident CTAs of the partial kernel on the current device (queried once per device)
    static int cached_device = -1;
    static int64_t slots = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_ERR_CUDA;
    if (dev != cached_device) {
        int sms = 0, per_sm = 0;
        if (cudaFuncSetAttribute(qmm::attn::attn_partial, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 qmm::attn::kSmem) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qmm::attn::attn_partial, qmm::attn::kThreads,
                                                          qmm::attn::kSmem) != cudaSuccess ||
            per_sm < 1)
            return QMM_ERR_CUDA;
        slots = static_cast<int64_t>(sms) * per_sm;
        cached_device = dev;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    qmm::attn::Params p = {};
    p.pool = static_cast<const uint8_t*>(pool);
    p.pool_pages = dims->pool_pages;
    p.table = page_table;
    p.max_pages = dims->max_pages;
    p.q = static_cast<const __half*>(q);
    p.row_len = row_len;
    p.agent_rows = agent_rows;
    p.heads = dims->heads;
    p.kv_heads = dims->kv_heads;
    p.group = dims->heads / dims->kv_heads;
    p.agents = dims->agents;
    qmm::attn::plan_runs(dims, slots, &p.runs, &p.chunk);
    p.max_qt = qmm::attn::max_tiles(dims, rows);
    p.ws = static_cast<float*>(workspace);
    p.err = err_word;
    p.out = out;
    p.rows = rows;
    // CTAs (agent, KV head, run) x query tile; the tiles past an agent's queries return at once
    const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(p.agents) * p.kv_heads * p.runs),
                    static_cast<unsigned>(p.max_qt));
    qmm::attn::attn_partial<<<grid, qmm::attn::kThreads, qmm::attn::kSmem, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return QMM_ERR_CUDA;
    // one warp per (row, head), launched as a programmatic dependent of the partial kernel
    const int64_t n = rows * dims->heads * 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((n + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, qmm::attn::attn_combine, p) != cudaSuccess) return QMM_ERR_CUDA;
    return QMM_OK;
}

}  // extern "C"
