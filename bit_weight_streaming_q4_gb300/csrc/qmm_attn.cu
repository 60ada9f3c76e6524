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
constexpr int kMaxQ = 32;   // queries per item: rows of the agent x heads of the group
constexpr int kChunk = 32;  // pages per work item (one wave of CTAs at the pages' decode step)
constexpr int kStages = 4;  // pages in flight per CTA
constexpr int kThreads = 128;
constexpr int kPart = kD + 2;  // floats per query of an item's partial: o[128], m, l
constexpr float kNegBig = -1e30f;
constexpr int kPS = kPT + 8;  // halves per row of the probability tile (16-byte padding: no bank conflicts)

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
    int32_t agents, max_chunks;
    float* ws;                  // [agent][kv head][run][kMaxQ][kPart]
    int* err;                   // sticky error word
    float* out;                 // [rows][heads][128]
    int64_t rows;
};

// Agent a's rows (r0, nr) and its number of 32-page runs, or -1 runs (and the error word)
// if its rows or lengths are outside what the kernels handle.
__device__ __forceinline__ int agent_runs(const Params& p, int a, int& r0, int& nr) {
    r0 = p.agent_rows[a];
    nr = p.agent_rows[a + 1] - r0;
    if (nr <= 0) return 0;
    if (r0 < 0 || r0 + nr > p.rows || nr * p.group > kMaxQ) return -1;
    int maxlen = 0;
    for (int r = r0; r < r0 + nr; ++r) {
        const int len = p.row_len[r];
        if (len < 1 || len > p.max_pages * kPT) return -1;
        maxlen = len > maxlen ? len : maxlen;
    }
    const int pages = (maxlen + kPT - 1) / kPT;
    return (pages + kChunk - 1) / kChunk;
}

// Bytes 0, 1 (sel 0x4140) or 2, 3 (sel 0x4342) of four int8 already XORed with 0x80, as
// fp16x2, exact: the biased byte goes into the mantissa of 1024, and 1024 + 128 comes off.
__device__ __forceinline__ uint32_t i8pair_to_h2(uint32_t biased, uint32_t sel) {
    return as_u32(__hadd2(as_h2(prmt(biased, 0x64646464u, sel)), as_h2(0xE480E480u)));
}

__global__ void __launch_bounds__(kThreads) attn_partial(const Params p) {
    extern __shared__ __align__(128) uint8_t sm[];
    // ring slot i % kStages holds page i
    __half* P = reinterpret_cast<__half*>(sm + kStages * kRec);       // [kMaxQ][kPS]
    float* red_max = reinterpret_cast<float*>(P + kMaxQ * kPS);       // [4][kMaxQ]
    float* red_sum = red_max + 4 * kMaxQ;                              // [4][kMaxQ]
    uint64_t* bar = reinterpret_cast<uint64_t*>(red_sum + 4 * kMaxQ);  // [kStages]
    volatile int* flags = reinterpret_cast<volatile int*>(bar + kStages);  // [0] abort

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    // this CTA's work item
    Item it;
    it.agent = blockIdx.x / (p.kv_heads * p.max_chunks);
    it.g = (blockIdx.x / p.max_chunks) % p.kv_heads;
    const int run = blockIdx.x % p.max_chunks;
    {
        const int runs = agent_runs(p, it.agent, it.r0, it.nr);
        if (runs < 0) {
            if (threadIdx.x == 0 && run == 0 && it.g == 0) atomicOr(p.err, 4);
            return;
        }
        if (run >= runs) return;
        int maxlen = 0;
        for (int r = it.r0; r < it.r0 + it.nr; ++r) maxlen = p.row_len[r] > maxlen ? p.row_len[r] : maxlen;
        const int pages = (maxlen + kPT - 1) / kPT;
        it.page0 = run * kChunk;
        it.npages = pages - it.page0 < kChunk ? pages - it.page0 : kChunk;
    }
    const int nq = it.nr * p.group;
    const int nmt = (nq + 15) >> 4;  // m16 tiles of queries (1 or 2)
    const float c2 = 1.4426950408889634f * 0.08838834764831845f;  // log2(e) / sqrt(128)

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&bar[i], 1);
        flags[0] = 0;
        fence_mbar_init();
    }
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
        mbar_arrive_expect_tx(b, kRec);
        bulk_g2s(sm + (i % kStages) * kRec, src, kRec, b, l2_policy_evict_first());
    };
    if (tid == 0)
        for (int i = 0; i < kStages - 1 && i < it.npages; ++i) issue(i);

    // Query fragments (A of QK^T).  The dims of k-step ks = 2 blk + k2 are assigned so that
    // each thread's eight dims of a 32-dim block are contiguous: slots (2t, 2t+1) are dims
    // 32 blk + 8t + 4 k2 + {0, 1} and slots (2t+8, 2t+9) dims 32 blk + 8t + 4 k2 + {2, 3};
    // K's B fragments use the same assignment.  Query qi = 16 mt + row is head
    // g * group + qi % group of row r0 + qi / group; queries past nq are zero.
    uint32_t qa[2][8][4];
    int qlen[2][2];  // tokens attended by this thread's two query rows of each m-tile
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int qi = 16 * mt + g8 + 8 * hh;
            qlen[mt][hh] = 0;
            const __half* qrow = nullptr;
            if (qi < nq) {
                const int r = it.r0 + qi / p.group;
                const int h = it.g * p.group + qi % p.group;
                qrow = p.q + (static_cast<int64_t>(r) * p.heads + h) * kD;
                qlen[mt][hh] = p.row_len[r];
            }
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint2 v = qrow ? *reinterpret_cast<const uint2*>(qrow + 32 * (ks >> 1) + 8 * t4 + 4 * (ks & 1))
                                     : make_uint2(0u, 0u);
                qa[mt][ks][hh] = v.x;      // a0 (row g8) / a1 (row g8 + 8)
                qa[mt][ks][2 + hh] = v.y;  // a2 / a3
            }
        }

    float m_run[2][2], l_run[2][2];
    float o[2][4][4];  // [m-tile][n8 tile of dims 32w + 8nt][accumulator]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            m_run[mt][hh] = kNegBig;
            l_run[mt][hh] = 0.f;
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
    }

    bool live = true;
    int consumed = 0;
    for (int i = 0; i < it.npages; ++i) {
        // slot (i + kStages - 1) % kStages held page i - 1, released at the end of the last iteration
        if (tid == 0 && i + kStages - 1 < it.npages) issue(i + kStages - 1);
        const bool ok = mbar_wait_bounded(&bar[i % kStages], (i / kStages) & 1, flags);
        // one decision for the whole CTA (every thread reaches this barrier)
        if (__syncthreads_or(!ok || flags[0])) {
            live = false;
            break;
        }
        consumed = i + 1;
        const uint8_t* rec = sm + (i % kStages) * kRec;
        const int tbase = (it.page0 + i) * kPT;  // logical index of the page's first token

        // ---- scores of tokens 16w .. 16w + 15: s[mt][nt][e], raw dot products
        float s[2][2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[mt][nt][e] = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int tokb = 16 * warp + 8 * nt + g8;      // this thread's B column (token)
            const int tokc = 16 * warp + 8 * nt + 2 * t4;  // its accumulator columns (tokens)
            // the four block scales of the two accumulator tokens
            const uint2 sc0v = *reinterpret_cast<const uint2*>(rec + 8192 + tokc * 8);
            const uint2 sc1v = *reinterpret_cast<const uint2*>(rec + 8192 + (tokc + 1) * 8);
            const uint32_t sc0w[2] = {sc0v.x, sc0v.y}, sc1w[2] = {sc1v.x, sc1v.y};
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                // eight contiguous dims 32 blk + 8 t4 .. + 7 of token tokb (16-byte piece p of
                // the row is stored at p ^ key, key = 2 (token % 4) + (token / 4) % 2: the 16
                // threads of a half-warp read 16 different 8-byte bank pairs)
                const int piece = (2 * blk + (t4 >> 1)) ^ (2 * (tokb & 3) + ((tokb >> 2) & 1));
                const uint2 kw = *reinterpret_cast<const uint2*>(rec + tokb * kD + 16 * piece + 8 * (t4 & 1));
                const float sc0 = __half2float((blk & 1) ? __high2half(as_h2(sc0w[blk >> 1])) : __low2half(as_h2(sc0w[blk >> 1])));
                const float sc1 = __half2float((blk & 1) ? __high2half(as_h2(sc1w[blk >> 1])) : __low2half(as_h2(sc1w[blk >> 1])));
                const uint32_t kx = kw.x ^ 0x80808080u, ky = kw.y ^ 0x80808080u;
                const uint32_t b00 = i8pair_to_h2(kx, 0x4140u), b01 = i8pair_to_h2(kx, 0x4342u);
                const uint32_t b10 = i8pair_to_h2(ky, 0x4140u), b11 = i8pair_to_h2(ky, 0x4342u);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    if (mt >= nmt) break;
                    float tmp[4] = {0.f, 0.f, 0.f, 0.f};
                    const int ks = 2 * blk;
                    mma_m16n8k16(tmp, qa[mt][ks][0], qa[mt][ks][1], qa[mt][ks][2], qa[mt][ks][3], b00, b01);
                    mma_m16n8k16(tmp, qa[mt][ks + 1][0], qa[mt][ks + 1][1], qa[mt][ks + 1][2], qa[mt][ks + 1][3], b10, b11);
                    s[mt][nt][0] += tmp[0] * sc0;
                    s[mt][nt][1] += tmp[1] * sc1;
                    s[mt][nt][2] += tmp[2] * sc0;
                    s[mt][nt][3] += tmp[3] * sc1;
                }
            }
        }
        // ---- masking and this warp's row maxima over its 16 tokens
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float mx = kNegBig;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e2 = 0; e2 < 2; ++e2) {
                        const int t = tbase + 16 * warp + 8 * nt + 2 * t4 + e2;
                        float& v = s[mt][nt][2 * hh + e2];
                        if (t >= qlen[mt][hh]) v = kNegBig;
                        mx = fmaxf(mx, v);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                if (t4 == 0) red_max[warp * kMaxQ + 16 * mt + g8 + 8 * hh] = mx;
            }
        __syncthreads();
        // ---- the page's maxima, new running maxima, probabilities (fp16) to shared memory
        float m_new[2][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int qi = 16 * mt + g8 + 8 * hh;
                float mx = m_run[mt][hh];
#pragma unroll
                for (int w = 0; w < 4; ++w) mx = fmaxf(mx, red_max[w * kMaxQ + qi]);
                m_new[mt][hh] = mx;
                float sum = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    float pr[2];
#pragma unroll
                    for (int e2 = 0; e2 < 2; ++e2) {
                        const float v = s[mt][nt][2 * hh + e2];
                        pr[e2] = v == kNegBig ? 0.f : exp2f((v - mx) * c2);
                        sum += pr[e2];
                    }
                    *reinterpret_cast<__half2*>(P + qi * kPS + 16 * warp + 8 * nt + 2 * t4) = __floats2half2_rn(pr[0], pr[1]);
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if (t4 == 0) red_sum[warp * kMaxQ + qi] = sum;
            }
        __syncthreads();
        // ---- running sums and rescaling of the output
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int qi = 16 * mt + g8 + 8 * hh;
                const float alpha = m_run[mt][hh] == m_new[mt][hh] ? 1.f : exp2f((m_run[mt][hh] - m_new[mt][hh]) * c2);
                float add = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) add += red_sum[w * kMaxQ + qi];
                l_run[mt][hh] = l_run[mt][hh] * alpha + add;
                m_run[mt][hh] = m_new[mt][hh];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    o[mt][nt][2 * hh] *= alpha;
                    o[mt][nt][2 * hh + 1] *= alpha;
                }
            }
        // ---- P . V for dims 32w .. 32w + 31 (one V scale block).  Tokens of k-step ks are
        // assigned so that each thread's sixteen tokens 16 t4 .. 16 t4 + 15 are contiguous:
        // slots (2t, 2t+1) are tokens 16t + 4 ks + {0, 1}, slots (2t+8, 2t+9) 16t + 4 ks + {2, 3}.
        {
            const uint4 dva = *reinterpret_cast<const uint4*>(rec + 16896 + (warp * kPT + 16 * t4) * 2);
            const uint4 dvb = *reinterpret_cast<const uint4*>(rec + 16896 + (warp * kPT + 16 * t4 + 8) * 2);
            const uint32_t dv[8] = {dva.x, dva.y, dva.z, dva.w, dvb.x, dvb.y, dvb.z, dvb.w};
            // A fragments: P times the tokens' V scales, [m-tile][row g8 / g8 + 8][token pair]
            uint32_t pa[2][2][8];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const __half* prow = P + (16 * mt + g8 + 8 * hh) * kPS + 16 * t4;
                    const uint4 x = *reinterpret_cast<const uint4*>(prow);
                    const uint4 y = *reinterpret_cast<const uint4*>(prow + 8);
                    const uint32_t pw[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) pa[mt][hh][j] = as_u32(__hmul2(as_h2(pw[j]), as_h2(dv[j])));
                }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int dim = 32 * warp + 8 * nt + g8;
                const uint4 vq = *reinterpret_cast<const uint4*>(rec + 8704 + dim * kPT + 16 * t4);
                const uint32_t vw[4] = {vq.x ^ 0x80808080u, vq.y ^ 0x80808080u, vq.z ^ 0x80808080u, vq.w ^ 0x80808080u};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t b0 = i8pair_to_h2(vw[ks], 0x4140u), b1 = i8pair_to_h2(vw[ks], 0x4342u);
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        if (mt >= nmt) break;
                        mma_m16n8k16(o[mt][nt], pa[mt][0][2 * ks], pa[mt][1][2 * ks], pa[mt][0][2 * ks + 1],
                                     pa[mt][1][2 * ks + 1], b0, b1);
                    }
                }
            }
        }
        __syncthreads();  // P and this page's buffer are free again
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

    // ---- the item's partial: o (this warp's dims), m and l per query
    float* part = p.ws + static_cast<int64_t>(blockIdx.x) * kMaxQ * kPart;  // slot (agent, g, run)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int qi = 16 * mt + g8 + 8 * hh;
            if (qi >= nq) continue;
            float* pq = part + qi * kPart;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int dim = 32 * warp + 8 * nt + 2 * t4;
                pq[dim] = o[mt][nt][2 * hh];
                pq[dim + 1] = o[mt][nt][2 * hh + 1];
            }
            if (warp == 0 && t4 == 0) {
                pq[kD] = m_run[mt][hh];
                pq[kD + 1] = l_run[mt][hh];
            }
        }
}

// One thread per output element: the items of (agent, KV head) combined in item order.
__global__ void attn_combine(const Params p) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= p.rows * p.heads * kD) return;
    const int d = static_cast<int>(idx % kD);
    const int h = static_cast<int>((idx / kD) % p.heads);
    const int64_t r = idx / (static_cast<int64_t>(kD) * p.heads);
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
        if (d == 0 && h == 0) atomicOr(p.err, 4);
        p.out[idx] = 0.f;
        return;
    }
    const int g = h / p.group;
    const int qi = static_cast<int>(r - r0) * p.group + h % p.group;
    const int64_t first = (static_cast<int64_t>(a) * p.kv_heads + g) * p.max_chunks;
    const float c2 = 1.4426950408889634f * 0.08838834764831845f;
    float m = kNegBig;
    for (int c = 0; c < n; ++c) m = fmaxf(m, p.ws[((first + c) * kMaxQ + qi) * kPart + kD]);
    float l = 0.f, o = 0.f;
    for (int c = 0; c < n; ++c) {
        const float* pq = p.ws + ((first + c) * kMaxQ + qi) * kPart;
        const float mc = pq[kD];
        if (mc == kNegBig) continue;  // no attended token in this item
        const float w = exp2f((mc - m) * c2);
        l += pq[kD + 1] * w;
        o += pq[d] * w;
    }
    p.out[idx] = o / l;
}

constexpr int kSmem = kStages * kRec + kMaxQ * kPS * 2 + 2 * 4 * kMaxQ * 4 + kStages * 8 + 16;

}  // namespace attn
}  // namespace qmm

extern "C" {

qmm_status qmm_attn_workspace_bytes(const qmm_attn_dims* dims, int64_t* bytes) {
    if (!dims || !bytes) return QMM_ERR_INVALID_ARG;
    if (dims->heads < 1 || dims->kv_heads < 1 || dims->heads % dims->kv_heads != 0 || dims->agents < 1 ||
        dims->max_pages < 1 || dims->pool_pages < 1)
        return QMM_ERR_INVALID_ARG;
    const int64_t runs = (dims->max_pages + qmm::attn::kChunk - 1) / qmm::attn::kChunk;
    *bytes = static_cast<int64_t>(dims->agents) * dims->kv_heads * runs * qmm::attn::kMaxQ * qmm::attn::kPart * 4;
    return QMM_OK;
}

qmm_status qmm_attn_decode(const qmm_attn_dims* dims, const void* pool, const int32_t* page_table,
                           const int32_t* agent_rows, const int32_t* row_len, const void* q, int64_t rows, float* out,
                           void* workspace, int64_t workspace_bytes, int* err_word, void* stream) {
    int64_t need = 0;
    qmm_status st = qmm_attn_workspace_bytes(dims, &need);
    if (st != QMM_OK) return st;
    if (!pool || !page_table || !agent_rows || !row_len || !q || !out || !workspace || !err_word || rows < 1)
        return QMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(pool) & 15) || (reinterpret_cast<uintptr_t>(q) & 15) ||
        (reinterpret_cast<uintptr_t>(workspace) & 15))
        return QMM_ERR_MISALIGNED;
    if (workspace_bytes < need) return QMM_ERR_SCRATCH_TOO_SMALL;
    static bool configured = false;
    if (!configured) {
        if (cudaFuncSetAttribute(qmm::attn::attn_partial, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 qmm::attn::kSmem) != cudaSuccess)
            return QMM_ERR_CUDA;
        configured = true;
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
    p.max_chunks = (dims->max_pages + qmm::attn::kChunk - 1) / qmm::attn::kChunk;
    p.ws = static_cast<float*>(workspace);
    p.err = err_word;
    p.out = out;
    p.rows = rows;
    const int64_t grid = static_cast<int64_t>(p.agents) * p.kv_heads * p.max_chunks;
    qmm::attn::attn_partial<<<static_cast<unsigned>(grid), qmm::attn::kThreads, qmm::attn::kSmem, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return QMM_ERR_CUDA;
    const int64_t n = rows * dims->heads * qmm::attn::kD;
    qmm::attn::attn_combine<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return QMM_ERR_CUDA;
    return QMM_OK;
}

}  // extern "C"
