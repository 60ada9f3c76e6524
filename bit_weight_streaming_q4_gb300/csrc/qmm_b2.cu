// Backend 2: Q4_K weight-streaming matmul on the 5th-generation tensor cores (tcgen05).
//
// The method (page "Running 4 coding agents on one RTX 3090: a custom CUDA engine for
// Qwen3.8-27B", section "How parallel decoding works"): every weight is read from memory
// once per step and multiplied against all M stacked token rows while it is on chip.
//
// One unit = 128 output rows x one super-block column (256 weights per row), 18432 bytes,
// stored contiguously by repack():
//   bytes [0, 16384):     quants, [sub-block s: 8][row: 128][16 B]; the 16 bytes are the
//                         four words of the row's 32 weights of sub-block s, word i covering
//                         weights 32s + 8i .. +7.  Inside a word the nibble of weight e
//                         (e = 0..7) sits at bit 0,16,4,20,8,24,12,28, so two masks and one
//                         shift give fp16x2 codes of consecutive weight pairs.
//   bytes [16384, 18432): the 16-byte block headers (d, dmin, scales) of the 128 rows.
//
// Warp roles of a persistent CTA (one per SM):
//   warps 0-7   dequantisation, two groups of four; group g takes the units j = g (mod 2)
//               of the CTA's piece, one output row per thread (warp w owns tensor-memory
//               lanes 32(w%4)..+31), and writes fp16 weights into the group's A buffer in
//               tensor memory;
//   warp 8      producer: 1-D bulk copies of the units into a shared-memory ring, 2-D TMA
//               loads (128-byte swizzle) of the activation tiles x[0..MP-1][kb*256..+256];
//   warp 9      per-sub-block activation sums and the tcgen05.mma issue: A = weights in
//               tensor memory (M = 128 rows), B = x in shared memory (N = MP tokens), fp32
//               accumulators in tensor memory, double-buffered per row tile;
//   warps 10-13 epilogue: accumulators -> y, or a split-K partial that the last CTA to
//               finish the row tile sums in CTA order.
// The piece of units of each CTA and every reduction order depend only on (N, K, grid),
// never on M, so each row's result is bit-identical across batchings.
//
// Dequantisation, exact to ~1 ulp of fp16 for every input: with code c = 1024 + q (or
// 1024 + 16q), P = sc*q is exact from one fp16 FMA; B = dmin*m splits error-free into
// B_h + B_l; the weight written is fp16(d*P - B_h), and the -B_l part goes to the tensor
// core as one extra K=16 step per unit: A = -B_l of the 8 sub-blocks, B = the activation
// sums of the 8 sub-blocks.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "qmm_internal.h"
#include "qmm_ptx.cuh"

namespace qmm {
namespace b2 {

constexpr int kQBytes = kRows * 128;
constexpr int kGroups = 2;                 // dequant warp groups
constexpr int kDqWarps = 4 * kGroups;
constexpr int kProducerWarp = kDqWarps;    // 8
constexpr int kMmaWarp = kDqWarps + 1;     // 9
constexpr int kEpiWarp0 = kDqWarps + 2;    // 10..13
constexpr int kThreads = (kEpiWarp0 + 4) * 32;  // 448
constexpr int kTmemCols = 512;
constexpr int kACols = 136;  // one unit: 128 columns of weights + 8 of the -B_l step
constexpr int kNA = kGroups; // one A buffer per group
constexpr int kWRing = 4;
static_assert(kWRing % kGroups == 0, "a weight slot must always feed the same group");
// named barriers
constexpr int kBarEpi = 1, kBarTmem = 2, kBarTeardown = 3;
constexpr int kTmemUsers = (kDqWarps + 1 + 4) * 32;  // dequant + MMA + epilogue warps
constexpr int kTeardownThreads = (1 + 4) * 32;       // MMA + epilogue warps

template <int MP>
struct Cfg {
    static constexpr int kXRing = MP <= 16 ? 4 : 2;
    static constexpr int kXBox = MP * 128;    // one 64-wide k box of x
    static constexpr int kXSlot = 4 * kXBox;  // x tile of one unit
    static constexpr int kXsBytes = MP * 32;  // the B tile of the -B_l step: [MP tokens][16 k]
    static constexpr int kAccCol = kNA * kACols;
    static_assert(kAccCol + 2 * MP <= kTmemCols, "tensor memory budget");
    static constexpr int kWOff = kXRing * kXSlot;
    static constexpr int kXsOff = kWOff + kWRing * kUnitBytes;
    static constexpr int kBarOff = kXsOff + kXRing * kXsBytes;
    static constexpr int kNumBars = 2 * kWRing + 2 * kXRing + 2 * kNA + 4;
    static constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024;  // + alignment slack
};

__device__ __forceinline__ int64_t dev_piece_of(int64_t u, int64_t units, int64_t grid) {
    return ((u + 1) * grid + units - 1) / units - 1;
}

__device__ __forceinline__ void fail(int* err, volatile int* flags) {
    if (!flags[0]) {
        flags[0] = 1;
        atomicOr(err, 1);
    }
}

// Scale constants of a pair of sub-blocks (fp16x2 lane .x / .y).
struct PairScale {
    uint32_t s1, n1;    // {sc}, {-1024 sc}:  c1 * s1 + n1 = sc*q   (c1 = 1024 + q)
    uint32_t s16, n16;  // {sc/16}, {-64 sc}: c16 * s16 + n16 = sc*q (c16 = 1024 + 16q)
    uint32_t nbh;       // {-B_h}
    uint32_t nbl;       // {-B_l}
};

__device__ __forceinline__ PairScale pair_scale(uint32_t SC, uint32_t MN, uint32_t byte0, uint32_t dm) {
    const uint32_t sel = byte0 | ((byte0 + 1) << 8);
    const __half2 k1024 = as_h2(0x64006400u);
    const __half2 sc = __hsub2(as_h2(and_or(prmt(SC, 0, sel), 0x00FF00FFu, 0x64006400u)), k1024);
    const __half2 mn = __hsub2(as_h2(and_or(prmt(MN, 0, sel), 0x00FF00FFu, 0x64006400u)), k1024);
    PairScale r;
    r.s1 = as_u32(sc);
    r.n1 = as_u32(__hmul2(sc, as_h2(0xE400E400u)));   // * -1024
    r.s16 = as_u32(__hmul2(sc, as_h2(0x2C002C00u)));  // * 1/16
    r.n16 = as_u32(__hmul2(sc, as_h2(0xD400D400u)));  // * -64
    const __half2 dmin = as_h2(dm);
    const __half2 bh = __hmul2(dmin, mn);
    r.nbh = as_u32(__hneg2(bh));
    r.nbl = as_u32(__hfma2(__hneg2(dmin), mn, bh));  // -(dmin*m - B_h), exact
    return r;
}

// One word (8 consecutive weights) -> 4 fp16x2 columns of fp16(d*sc*q - B_h).
__device__ __forceinline__ void dq_word(uint32_t w, __half2 s1, __half2 n1, __half2 s16, __half2 n16,
                                        __half2 d2, __half2 nbh, uint32_t* out) {
    const uint32_t w8 = w >> 8;
    const __half2 c01 = as_h2(and_or(w, 0x000F000Fu, 0x64006400u));
    const __half2 c23 = as_h2(and_or(w, 0x00F000F0u, 0x64006400u));
    const __half2 c45 = as_h2(and_or(w8, 0x000F000Fu, 0x64006400u));
    const __half2 c67 = as_h2(and_or(w8, 0x00F000F0u, 0x64006400u));
    out[0] = as_u32(__hfma2(__hfma2(c01, s1, n1), d2, nbh));
    out[1] = as_u32(__hfma2(__hfma2(c23, s16, n16), d2, nbh));
    out[2] = as_u32(__hfma2(__hfma2(c45, s1, n1), d2, nbh));
    out[3] = as_u32(__hfma2(__hfma2(c67, s16, n16), d2, nbh));
}

// Shared-memory descriptor of the -B_l step's B tile: K-major, no swizzle, core matrices of
// 8 tokens x 16 bytes; the two k halves 128 bytes apart, token groups 256 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_xs(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
           (static_cast<uint64_t>(256 >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
}

template <int MP>
__global__ void __launch_bounds__(kThreads, 1)
    tc_kernel(const __grid_constant__ CUtensorMap xmap, const B2Params p) {
    using C = Cfg<MP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* xring = smem;
    uint8_t* wring = smem + C::kWOff;
    uint8_t* xsum = smem + C::kXsOff;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* wfull = bars;
    uint64_t* wempty = wfull + kWRing;
    uint64_t* xfull = wempty + kWRing;
    uint64_t* xempty = xfull + C::kXRing;
    uint64_t* tfull = xempty + C::kXRing;
    uint64_t* tempty = tfull + kNA;
    uint64_t* accfull = tempty + kNA;
    uint64_t* accempty = accfull + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accempty + 2);
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort [1] last

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t c = blockIdx.x;
    const int64_t U = p.units;
    const int64_t u0 = c * U / p.grid;
    const int64_t u1 = (c + 1) * U / p.grid;
    const int nunits = static_cast<int>(u1 - u0);
    const int KB = p.kb;
    const int64_t t_first = u0 / KB;
    const int64_t t_last = (u1 - 1) / KB;

    if (tid == 0) {
        for (int i = 0; i < kWRing; ++i) {
            mbar_init(&wfull[i], 1);
            mbar_init(&wempty[i], 4);
        }
        for (int i = 0; i < C::kXRing; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&xempty[i], 1);
        }
        for (int i = 0; i < kNA; ++i) {
            mbar_init(&tfull[i], 4);
            mbar_init(&tempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accfull[i], 1);
            mbar_init(&accempty[i], 4);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    // the upper (always zero) k half of every -B_l step's B tile
    for (int i = tid; i < C::kXRing * MP * 4; i += kThreads) {
        const int slot = i / (MP * 4), r = (i / 4) % MP, e = i % 4;
        *reinterpret_cast<uint32_t*>(xsum + slot * C::kXsBytes + (r >> 3) * 256 + 128 + (r & 7) * 16 + e * 4) = 0u;
    }
    fence_proxy_async_smem();
    __syncthreads();
    griddep_launch_dependents();

    // ------------------------------------------------------------------ producer
    if (warp == kProducerWarp) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            const uint8_t* src = p.wq + u0 * kUnitBytes;
            const int pre = nunits < kWRing ? nunits : kWRing;
            for (int j = 0; j < pre; ++j) {
                mbar_arrive_expect_tx(&wfull[j], kUnitBytes);
                bulk_g2s(wring + j * kUnitBytes, src + static_cast<int64_t>(j) * kUnitBytes, kUnitBytes,
                         &wfull[j], pol);
            }
            int w_issued = pre, x_issued = 0;
            griddep_wait();  // activations may be written by the previous kernel
            prefetch_tmap(&xmap);
            for (int j = 0; j < nunits && !flags[0]; ++j) {
                const int xs = j % C::kXRing;
                if (j >= C::kXRing && !mbar_wait_bounded(&xempty[xs], ((j / C::kXRing) - 1) & 1, flags)) {
                    fail(p.err, flags);
                    break;
                }
                mbar_arrive_expect_tx(&xfull[xs], C::kXSlot);
                const int kb = static_cast<int>((u0 + j) % KB);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    tma_load_2d(xring + xs * C::kXSlot + i * C::kXBox, &xmap, kb * 256 + 64 * i, 0, &xfull[xs]);
                x_issued = j + 1;
                const int jj = j + kWRing;
                if (jj < nunits) {
                    const int s = jj % kWRing;
                    if (!mbar_wait_bounded(&wempty[s], ((jj / kWRing) - 1) & 1, flags)) {
                        fail(p.err, flags);
                        break;
                    }
                    mbar_arrive_expect_tx(&wfull[s], kUnitBytes);
                    bulk_g2s(wring + s * kUnitBytes, src + static_cast<int64_t>(jj) * kUnitBytes, kUnitBytes,
                             &wfull[s], pol);
                    w_issued = jj + 1;
                }
            }
            if (flags[0]) {
                // failure path: let every copy already issued land before the CTA can exit
                volatile int no_abort = 0;
                for (int j = w_issued > kWRing ? w_issued - kWRing : 0; j < w_issued; ++j)
                    mbar_wait_bounded(&wfull[j % kWRing], (j / kWRing) & 1, &no_abort);
                for (int j = x_issued > C::kXRing ? x_issued - C::kXRing : 0; j < x_issued; ++j)
                    mbar_wait_bounded(&xfull[j % C::kXRing], (j / C::kXRing) & 1, &no_abort);
            }
        }
        return;
    }

    // ------------------------------------------------------------------ activation sums + MMA
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
        named_bar_sync(kBarTmem, kTmemUsers);
        tc_fence_after();
        const uint32_t tbase = *tmem_slot;
        constexpr uint32_t kIdesc = idesc_f16_f32(kRows, MP);
        int seg = 0;
        for (int64_t tile = t_first; tile <= t_last; ++tile, ++seg) {
            const int64_t ja = (tile * KB > u0 ? tile * KB : u0) - u0;
            const int64_t jb = ((tile + 1) * KB < u1 ? (tile + 1) * KB : u1) - u0;
            const int b = seg & 1;
            if (seg >= 2 && !mbar_wait_bounded(&accempty[b], ((seg >> 1) - 1) & 1, flags)) fail(p.err, flags);
            tc_fence_after();
            const uint32_t d_tmem = tbase + C::kAccCol + b * MP;
            for (int64_t j = ja; j < jb; ++j) {
                const int xs = static_cast<int>(j % C::kXRing);
                const int a = static_cast<int>(j % kNA);
                bool ok = mbar_wait_bounded(&xfull[xs], (j / C::kXRing) & 1, flags);
                // X[t][s] = sum of the 32 activations of token t in sub-block s (fp16, clamped)
                if (ok) {
                    const uint8_t* xt = xring + xs * C::kXSlot;
                    uint8_t* xst = xsum + xs * C::kXsBytes;
#pragma unroll 1
                    for (int pi = lane; pi < MP * 8; pi += 32) {
                        const int t = pi % MP, s = pi / MP;
                        const uint8_t* rowp = xt + (s >> 1) * C::kXBox + t * 128;
                        __half2 acc2 = __float2half2_rn(0.f);
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            const int chunk = ((s & 1) * 4 + cc) ^ (t & 7);
                            const uint4 v = *reinterpret_cast<const uint4*>(rowp + chunk * 16);
                            acc2 = __hadd2(acc2, __hadd2(__hadd2(as_h2(v.x), as_h2(v.y)),
                                                         __hadd2(as_h2(v.z), as_h2(v.w))));
                        }
                        __half sum = __hadd(__low2half(acc2), __high2half(acc2));
                        sum = __hmin(__hmax(sum, __ushort_as_half(0xFBFFu)), __ushort_as_half(0x7BFFu));
                        *reinterpret_cast<__half*>(xst + (t >> 3) * 256 + (t & 7) * 16 + s * 2) = sum;
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) {
                    ok = ok && mbar_wait_bounded(&tfull[a], (j / kNA) & 1, flags);
                    if (!ok) fail(p.err, flags);
                    tc_fence_after();
                    if (ok) {
                        const uint32_t xaddr = smem_u32(xring + xs * C::kXSlot);
                        const uint32_t acol = tbase + a * kACols;
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk) {
                            const uint64_t bdesc = smem_desc_sw128(xaddr + (kk >> 2) * C::kXBox + (kk & 3) * 32);
                            tc_mma_f16_ts(d_tmem, acol + 8 * kk, bdesc, kIdesc, (j > ja || kk > 0) ? 1u : 0u);
                        }
                        tc_mma_f16_ts(d_tmem, acol + 128, smem_desc_xs(smem_u32(xsum + xs * C::kXsBytes)), kIdesc, 1u);
                    }
                    tc_commit(&tempty[a]);
                    tc_commit(&xempty[xs]);
                }
                __syncwarp();
            }
            if (lane == 0) tc_commit(&accfull[b]);
            __syncwarp();
        }
        named_bar_sync(kBarTeardown, kTeardownThreads);  // every accumulator has been read
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
        return;
    }

    // ------------------------------------------------------------------ epilogue
    if (warp >= kEpiWarp0) {
        const int q = warp & 3;  // tensor-memory lane quarter
        const int row = 32 * q + lane;
        const int etid = tid - kEpiWarp0 * 32;
        named_bar_sync(kBarTmem, kTmemUsers);
        tc_fence_after();
        const uint32_t tbase = *tmem_slot;
        griddep_wait();  // y and the workspace may still be in use by the previous kernel
        int seg = 0;
        for (int64_t tile = t_first; tile <= t_last; ++tile, ++seg) {
            const int64_t ja = (tile * KB > u0 ? tile * KB : u0) - u0;
            const int64_t jb = ((tile + 1) * KB < u1 ? (tile + 1) * KB : u1) - u0;
            const int b = seg & 1;
            if (!mbar_wait_bounded(&accfull[b], (seg >> 1) & 1, flags)) fail(p.err, flags);
            tc_fence_after();
            const bool whole = (ja + u0 == tile * KB) && (jb + u0 == (tile + 1) * KB);
            const int side = (tile == t_first) ? 0 : 1;
            float* part = p.ws + (c * 2 + side) * static_cast<int64_t>(kRows) * p.ws_cols;
            const int64_t n = tile * kRows + row;
#pragma unroll 1
            for (int c0 = 0; c0 < MP; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tbase + (static_cast<uint32_t>(32 * q) << 16) + C::kAccCol + b * MP + c0, v);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int m = c0 + i;
                    if (m < p.m) {
                        const float val = __uint_as_float(v[i]);
                        if (whole) {
                            if (n < p.n) p.y[static_cast<int64_t>(m) * p.n + n] = val;
                        } else {
                            part[m * kRows + row] = val;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&accempty[b]);
            if (!whole) {
                __threadfence();
                named_bar_sync(kBarEpi, 128);
                const int64_t pa = dev_piece_of(tile * KB, U, p.grid);
                const int64_t pb = dev_piece_of((tile + 1) * KB - 1, U, p.grid);
                if (etid == 0) {
                    const int old = atomicAdd(&p.tickets[tile], 1);
                    flags[1] = (old == static_cast<int>(pb - pa)) ? 1 : 0;
                }
                named_bar_sync(kBarEpi, 128);
                if (flags[1]) {
                    __threadfence();
                    // sum the CTA partials in CTA order; the loads of one part are independent
#pragma unroll 1
                    for (int m0 = 0; m0 < p.m; m0 += 16) {
                        float acc[16];
#pragma unroll 1
                        for (int64_t pc = pa; pc <= pb; ++pc) {
                            const int64_t pc_first_tile = (pc * U / p.grid) / KB;
                            const int sd = (tile == pc_first_tile) ? 0 : 1;
                            const float* src = p.ws + (pc * 2 + sd) * static_cast<int64_t>(kRows) * p.ws_cols + row;
                            float pv[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) pv[i] = (m0 + i < p.m) ? __ldcg(src + (m0 + i) * kRows) : 0.f;
#pragma unroll
                            for (int i = 0; i < 16; ++i) acc[i] = (pc == pa) ? pv[i] : acc[i] + pv[i];
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (m0 + i < p.m && n < p.n) p.y[static_cast<int64_t>(m0 + i) * p.n + n] = acc[i];
                    }
                    if (etid == 0) p.tickets[tile] = 0;  // ready for the next run
                }
                named_bar_sync(kBarEpi, 128);  // flags[1] is reused by the next tile
            }
        }
        named_bar_sync(kBarTeardown, kTeardownThreads);
        return;
    }

    // ------------------------------------------------------------------ dequant warps
    const int q = warp & 3;   // lane quarter: rows 32q .. 32q+31
    const int g = warp >> 2;  // group: units j = g (mod kGroups)
    const int row = 32 * q + lane;
    named_bar_sync(kBarTmem, kTmemUsers);
    tc_fence_after();
    const uint32_t tlane = *tmem_slot + (static_cast<uint32_t>(32 * q) << 16);

    for (int j = g; j < nunits; j += kGroups) {
        const int s = j % kWRing;
        const int a = j % kNA;
        if (!mbar_wait_bounded(&wfull[s], (j / kWRing) & 1, flags)) fail(p.err, flags);
        const uint8_t* u = wring + s * kUnitBytes;
        uint4 qv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) qv[i] = *reinterpret_cast<const uint4*>(u + (i * kRows + row) * 16);
        const uint4 hd = *reinterpret_cast<const uint4*>(u + kQBytes + row * 16);
        __syncwarp();
        if (lane == 0) mbar_arrive(&wempty[s]);

        // (scale, min) pairs of sub-blocks (0,1), (2,3) from the low 6 bits of s[0..7] and
        // (4,5), (6,7) from s[8..11] plus the top 2 bits of s[0..7]
        const uint32_t SClo = hd.y & 0x3F3F3F3Fu;
        const uint32_t MNlo = hd.z & 0x3F3F3F3Fu;
        const uint32_t SChi = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
        const uint32_t MNhi = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
        const uint32_t dm = prmt(hd.x, 0, 0x3232u);
        const __half2 d2 = as_h2(prmt(hd.x, 0, 0x1010u));
        PairScale ps[4];
        ps[0] = pair_scale(SClo, MNlo, 0, dm);
        ps[1] = pair_scale(SClo, MNlo, 2, dm);
        ps[2] = pair_scale(SChi, MNhi, 0, dm);
        ps[3] = pair_scale(SChi, MNhi, 2, dm);

        if (j >= kNA && !mbar_wait_bounded(&tempty[a], ((j / kNA) - 1) & 1, flags)) fail(p.err, flags);
        tc_fence_after();
        const uint32_t tcol = tlane + a * kACols;
#pragma unroll
        for (int sb = 0; sb < 8; ++sb) {
            const PairScale& z = ps[sb >> 1];
            const bool hiL = sb & 1;
            const __half2 s1 = hiL ? __high2half2(as_h2(z.s1)) : __low2half2(as_h2(z.s1));
            const __half2 n1 = hiL ? __high2half2(as_h2(z.n1)) : __low2half2(as_h2(z.n1));
            const __half2 s16 = hiL ? __high2half2(as_h2(z.s16)) : __low2half2(as_h2(z.s16));
            const __half2 n16 = hiL ? __high2half2(as_h2(z.n16)) : __low2half2(as_h2(z.n16));
            const __half2 nbh = hiL ? __high2half2(as_h2(z.nbh)) : __low2half2(as_h2(z.nbh));
            uint32_t out[16];
            dq_word(qv[sb].x, s1, n1, s16, n16, d2, nbh, out + 0);
            dq_word(qv[sb].y, s1, n1, s16, n16, d2, nbh, out + 4);
            dq_word(qv[sb].z, s1, n1, s16, n16, d2, nbh, out + 8);
            dq_word(qv[sb].w, s1, n1, s16, n16, d2, nbh, out + 12);
            tmem_st16(tcol + 16 * sb, out);
        }
        // the -B_l step: k slots 0..7 = sub-blocks 0..7, slots 8..15 zero
        const uint32_t bl[8] = {ps[0].nbl, ps[1].nbl, ps[2].nbl, ps[3].nbl, 0u, 0u, 0u, 0u};
        tmem_st8(tcol + 128, bl);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tfull[a]);
    }
}

// One thread per 16-byte piece of the packed layout.
__global__ void repack_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t n,
                              int32_t kb, int64_t units) {
    constexpr int kSegs = kUnitBytes / 16;  // 1152
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= units * kSegs) return;
    const int64_t u = idx / kSegs;
    const int seg = static_cast<int>(idx % kSegs);
    const int64_t tile = u / kb;
    const int b = static_cast<int>(u % kb);
    uint4 out = make_uint4(0, 0, 0, 0);
    if (seg < 1024) {
        const int sb = seg >> 7, row = seg & 127;  // sub-block sb of row
        const int64_t nrow = tile * kRows + row;
        if (nrow < n) {
            // sub-block sb = weights 32sb..32sb+31: chunk sb/2, low nibbles if sb even
            const uint8_t* bytes = src + (nrow * kb + b) * 144 + 16 + 32 * (sb >> 1);
            const bool high = sb & 1;
            const int pos[8] = {0, 16, 4, 20, 8, 24, 12, 28};
            uint32_t w4[4];
            for (int wi = 0; wi < 4; ++wi) {
                uint32_t w = 0;
                for (int e = 0; e < 8; ++e) {
                    const uint8_t byte = bytes[8 * wi + e];
                    const uint32_t nib = high ? (byte >> 4) : (byte & 15u);
                    w |= nib << pos[e];
                }
                w4[wi] = w;
            }
            out = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
    } else {
        const int row = seg - 1024;
        const int64_t nrow = tile * kRows + row;
        if (nrow < n) out = *reinterpret_cast<const uint4*>(src + (nrow * kb + b) * 144);
    }
    *reinterpret_cast<uint4*>(dst + u * kUnitBytes + static_cast<int64_t>(seg) * 16) = out;
}

cudaError_t repack(const uint8_t* src_dev, uint8_t* dst_dev, const Decomp& d, cudaStream_t s) {
    const int64_t total = d.units * (kUnitBytes / 16);
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    repack_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(src_dev, dst_dev, d.n, static_cast<int32_t>(d.kb),
                                                                   d.units);
    return cudaGetLastError();
}

template <int MP>
static cudaError_t set_attr() {
    return cudaFuncSetAttribute(tc_kernel<MP>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<MP>::kSmem);
}

cudaError_t configure() {
    cudaError_t e;
    if ((e = set_attr<16>()) != cudaSuccess) return e;
    if ((e = set_attr<32>()) != cudaSuccess) return e;
    return set_attr<64>();
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

int mp_for(int m) { return m <= 16 ? 16 : m <= 32 ? 32 : 64; }

template <int MP>
static cudaError_t launch_mp(const CUtensorMap& tmap, const B2Params& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<MP>::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_kernel<MP>, tmap, p);
}

cudaError_t launch(const void* x, int64_t k, const B2Params& p, cudaStream_t s, bool pdl) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int mp = mp_for(p.m);
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(p.m)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(k) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(mp)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    switch (mp) {
        case 16: return launch_mp<16>(tmap, p, s, pdl);
        case 32: return launch_mp<32>(tmap, p, s, pdl);
        default: return launch_mp<64>(tmap, p, s, pdl);
    }
}

}  // namespace b2
}  // namespace qmm
