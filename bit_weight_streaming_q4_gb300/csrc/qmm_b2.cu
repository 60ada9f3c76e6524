// Backend 2: Q4_K weight-streaming matmul on the 5th-generation tensor cores (tcgen05).
//
// The method (page "Running 4 coding agents on one RTX 3090: a custom CUDA engine for
// Qwen3.8-27B", section "How parallel decoding works"): every weight is read from memory
// once per step and multiplied against all M stacked token rows while it is on chip.  The
// tensor-core instruction costs the same for any N up to 64, so this backend serves runs of
// more than 16 rows (up to 64 per launch).
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
// Warp roles of a persistent CTA (one per SM, 16 warps):
//   warps 0-7   dequantisation, two groups of four; group g takes the units j = g (mod 2)
//               of the CTA's piece, one output row per thread (warp w owns tensor-memory
//               lanes 32(w%4)..+31), and writes fp16 weights into A buffer j mod kNA in
//               tensor memory (kNA = 3 where there is room, so that a group can dequantise
//               its next unit while the tensor core still reads the last two);
//   warp 8      weight producer: 1-D bulk copies of the units into a shared-memory ring,
//               across matrix boundaries;
//   warp 9      activations: 2-D TMA (128-byte swizzle) of x[0..MP-1][kb*256..+256] for each
//               unit (the dequantising group also forms the unit's per-sub-block activation
//               sums for the correction step);
//   warps 10, 15 tcgen05.mma issue (one thread each), warp 10 for the units of group 0 and
//               warp 15 for those of group 1: A = weights in tensor memory (M = 128 rows),
//               B = x in shared memory (N = MP tokens), fp32 accumulators in tensor memory,
//               one per issuing warp, double-buffered per row tile.  A single thread
//               cannot keep the tensor core busy: after a burst of MMAs its next
//               shared-memory access (the mbarrier wait for the next unit) stalls until the
//               burst has drained, so two issuers take turns;
//   warps 11-14 epilogue: the sum of the two accumulators -> y, a split-K partial, or the
//               reduction of a split row tile; warp 11 also publishes the CTA's partial and
//               resets the ticket of the tile it reduced.
// Decomposition as in the mma.sync backend: a launch concatenates its matrices' unit
// sequences, CTA c takes [c*U/P, (c+1)*U/P), and a row tile cut between CTAs pa..pb is
// reduced by pa in piece order.  Nothing in any output's arithmetic depends on M.
//
// Dequantisation, exact to ~1 ulp of fp16 for every input: with code c = 1024 + q (or
// 1024 + 16q), P = sc*q is exact from one fp16 FMA; B = dmin*m splits error-free into
// B_h + B_l; the weight written is fp16(d*P - B_h), and the -B_l part goes to the tensor
// core as one extra K=16 step per unit: A = -B_l of the 8 sub-blocks (a small tile in
// shared memory), B = the activation sums of the 8 sub-blocks.
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
constexpr int kXWarp = kDqWarps + 1;       // 9
constexpr int kMmaWarp0 = kDqWarps + 2;   // 10: MMAs of group 0's units
constexpr int kEpiWarp0 = kDqWarps + 3;   // 11..14
constexpr int kMmaWarp1 = kEpiWarp0 + 4;  // 15: MMAs of group 1's units
constexpr int kThreads = (kMmaWarp1 + 1) * 32;  // 512: 128 registers per thread
constexpr int kEpiThreads = 128;
constexpr int kTmemCols = 512;
constexpr int kACols = 128;  // one unit of fp16 weights: 128 rows x 256 k
// The handshakes on the A buffers (tfull: written; tempty: read by the MMAs) use a pair of
// mbarriers per unit j mod 6, so that each barrier only ever serves one dequant group, one
// issuer and one buffer (unit j -> buffer j mod kNA, kNA = 2 or 3), and no waiter can fall
// two phases behind (a parity wait cannot tell that from a phase already done).
constexpr int kTB = 6;
constexpr int kBlBytes = kRows * 32;  // A tile of the -B_l step: [128 rows][16 k] fp16
// named barriers
constexpr int kBarTmem = 1, kBarTeardown = 2;
constexpr int kTmemUsers = (kDqWarps + 2 + 4) * 32;  // dequant + MMA + epilogue warps

template <int MP>
struct Cfg {
    // ring depths, as deep as shared memory allows: weight slots and activation slots, each a
    // multiple of kGroups so that a slot (and its barriers) always serves the same group
    static constexpr int kWRing = MP == 16 ? 8 : MP == 32 ? 6 : 4;
    static constexpr int kXRing = MP == 16 ? 8 : MP == 32 ? 6 : 4;
    static constexpr int kXBox = MP * 128;    // one 64-wide k box of x
    static constexpr int kXSlot = 4 * kXBox;  // x tile of one unit
    static constexpr int kXsBytes = MP * 32;  // the B tile of the -B_l step: [MP tokens][16 k]
    // A buffers in tensor memory (unit j -> buffer j mod kNA): three where tensor memory has
    // room, so that a group can dequantise its next unit while the tensor core still reads
    // the last two; two at MP = 64, where the accumulators take the room.  Accumulators:
    // two buffers per issuer, so that the epilogue of a tile overlaps the next tile's MMAs.
    static constexpr int kNA = MP == 64 ? 2 : 3;
    static constexpr int kAccBufs = 2;
    static constexpr int kAccCol = kNA * kACols;  // accumulator (issuer e, buffer b) at + (e * kAccBufs + b) * MP
    static_assert(kAccCol + 2 * kAccBufs * MP <= kTmemCols, "tensor memory budget");
    static_assert(kTB % kNA == 0 && kTB % 2 == 0, "one barrier pair per unit mod kTB");
    static_assert(kWRing % kGroups == 0 && kXRing % kGroups == 0, "a slot must always feed the same group");
    static constexpr int kWOff = kXRing * kXSlot;
    static constexpr int kXsOff = kWOff + kWRing * kUnitBytes;
    static constexpr int kBlOff = kXsOff + kXRing * kXsBytes;
    static constexpr int kBarOff = kBlOff + kNA * kBlBytes;
    static constexpr int kNumBars = 2 * kWRing + 2 * kXRing + 2 * kTB + 4 + 2 + 2 + 1;
    // argmax launches: the epilogue warps' best keys, [warp 4][token MP]
    static constexpr int kAmaxOff = kBarOff + kNumBars * 8 + 16;
    static constexpr int kSmem = kAmaxOff + 4 * MP * 8 + 1024;  // + alignment slack
    static_assert(kSmem <= 232448, "shared memory budget");
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

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* flags) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, flags));
}

__device__ __forceinline__ bool wait_count(const int* p, int target, volatile int* flags) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (ld_acquire_gpu(p) >= target) return true;
        if (flags[0]) return false;
        if ((it & 63u) == 63u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
        __nanosleep(64);
    }
}

struct Cursor {
    int i;
    int64_t j, e;
};

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

// Shared-memory descriptor of the -B_l step's A and B tiles ([rows][16 k] fp16): K-major, no
// swizzle, core matrices of 8 rows x 16 bytes; the two k halves 128 bytes apart, 8-row groups
// 256 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_k16(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
           (static_cast<uint64_t>(256 >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
}

template <int MP>
__global__ void __launch_bounds__(kThreads, 1)
    tc_kernel(const __grid_constant__ MatDesc single, const LaunchParams p) {
    using C = Cfg<MP>;
    constexpr int kWRing = C::kWRing;
    constexpr int kXRing = C::kXRing;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* xring = smem;
    uint8_t* wring = smem + C::kWOff;
    uint8_t* xsum = smem + C::kXsOff;
    uint8_t* blt = smem + C::kBlOff;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* wfull = bars;
    uint64_t* wempty = wfull + kWRing;
    uint64_t* xfull = wempty + kWRing;
    uint64_t* xempty = xfull + kXRing;
    uint64_t* tfull = xempty + kXRing;
    uint64_t* tempty = tfull + kTB;
    uint64_t* accfull = tempty + kTB;   // [2]: both issuers' accumulators of buffer b are final
    uint64_t* accempty = accfull + 2;   // [2]: the epilogue has read buffer b
    uint64_t* evpart = accempty + 2;    // the four epilogue warps have written the partial
    uint64_t* evred = evpart + 1;       // ... have read the partials of the tile they reduced
    uint64_t* mmadone = evred + 1;      // [2]: every MMA of issuer e has finished
    uint64_t* evamax = mmadone + 2;     // argmax launches: the four epilogue warps' keys are in
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(evamax + 1);
    unsigned long long* amax_sm = reinterpret_cast<unsigned long long*>(smem + C::kAmaxOff);
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t c = blockIdx.x;
    const int count = p.count;
    const int64_t U = p.units;
    const int64_t P = gridDim.x;
    const int64_t g0 = c * U / P, g1 = (c + 1) * U / P;
    auto mat = [&](int i) -> const MatDesc& { return count == 1 ? single : p.mats[i]; };
    auto enter = [&](Cursor& k, int i) {
        for (; i < count; ++i) {
            const MatDesc& M = mat(i);
            if (M.base >= g1) break;
            const int64_t lo = g0 > M.base ? g0 - M.base : 0;
            const int64_t hi = g1 - M.base < M.units ? g1 - M.base : M.units;
            if (lo < hi) {
                k.i = i;
                k.j = lo;
                k.e = hi;
                return;
            }
        }
        k.i = count;
        k.j = k.e = 0;
    };
    auto first = [&](Cursor& k) { enter(k, count == 1 ? 0 : p.first_mat[c]); };
    auto next = [&](Cursor& k) {
        if (++k.j >= k.e) enter(k, k.i + 1);
    };

    if (tid == 0) {
        for (int i = 0; i < kWRing; ++i) {
            mbar_init(&wfull[i], 1);
            mbar_init(&wempty[i], 4);
        }
        for (int i = 0; i < kXRing; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&xempty[i], 1);
        }
        for (int i = 0; i < kTB; ++i) {
            mbar_init(&tfull[i], 4);
            mbar_init(&tempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accfull[i], 2);
            mbar_init(&accempty[i], 4);
            mbar_init(&mmadone[i], 1);
        }
        mbar_init(evpart, 4);
        mbar_init(evred, 4);
        mbar_init(evamax, 4);
        flags[0] = 0;
        fence_mbar_init();
    }
    // the upper (always zero) k half of every -B_l step's B tile
    for (int i = tid; i < kXRing * MP * 4; i += kThreads) {
        const int slot = i / (MP * 4), r = (i / 4) % MP, e = i % 4;
        *reinterpret_cast<uint32_t*>(xsum + slot * C::kXsBytes + (r >> 3) * 256 + 128 + (r & 7) * 16 + e * 4) = 0u;
    }
    // ... and of the A tiles of the -B_l step
    for (int i = tid; i < C::kNA * kRows * 4; i += kThreads) {
        const int slot = i / (kRows * 4), r = (i / 4) % kRows, e = i % 4;
        *reinterpret_cast<uint32_t*>(blt + slot * kBlBytes + (r >> 3) * 256 + 128 + (r & 7) * 16 + e * 4) = 0u;
    }
    fence_proxy_async_smem();
    __syncthreads();
    griddep_launch_dependents();

    // ------------------------------------------------------------------ weight producer
    if (warp == kProducerWarp) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            Cursor w;
            first(w);
            int64_t wseq = 0;
            bool ok = true;
            int cur = -1;
            const uint8_t* src = nullptr;
            while (w.i < count) {
                const int s = static_cast<int>(wseq % kWRing);
                if (wseq >= kWRing && !mbar_wait_bounded(&wempty[s], ((wseq / kWRing) - 1) & 1, flags)) {
                    ok = false;
                    break;
                }
                if (w.i != cur) {
                    cur = w.i;
                    src = mat(w.i).wq + w.j * kUnitBytes;
                }
                mbar_arrive_expect_tx(&wfull[s], kUnitBytes);
                bulk_g2s(wring + s * kUnitBytes, src, kUnitBytes, &wfull[s], pol);
                src += kUnitBytes;
                ++wseq;
                next(w);
            }
            if (!ok) fail(p.err, flags);
            if (flags[0]) {
                volatile int no_abort = 0;
                for (int64_t j = wseq > kWRing ? wseq - kWRing : 0; j < wseq; ++j)
                    mbar_wait_bounded(&wfull[j % kWRing], (j / kWRing) & 1, &no_abort);
            }
        }
        return;
    }

    // ------------------------------------------------------------------ activations
    // TMA of each unit's activation tile, up to kXRing units ahead of the tensor core (a slot
    // is reused once the MMAs that read it have finished).
    if (warp == kXWarp) {
        if (lane == 0) {
            Cursor xc;
            first(xc);
            int64_t issued = 0;
            int cur = -1, kbn = 1, kb = 0;
            const void* xmap = nullptr;
            bool ok = true;
            griddep_wait();  // activations may be written by the previous kernel
            while (xc.i < count) {
                const int xs = static_cast<int>(issued % kXRing);
                if (issued >= kXRing && !mbar_wait_bounded(&xempty[xs], ((issued / kXRing) - 1) & 1, flags)) {
                    ok = false;
                    break;
                }
                if (xc.i != cur) {
                    const MatDesc& M = mat(xc.i);
                    cur = xc.i;
                    xmap = &M.xmap;
                    kbn = M.kb;
                    kb = static_cast<int>(xc.j % kbn);
                }
                mbar_arrive_expect_tx(&xfull[xs], C::kXSlot);
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    tma_load_2d(xring + xs * C::kXSlot + b * C::kXBox, xmap, kb * 256 + 64 * b, 0, &xfull[xs]);
                kb = (kb + 1 == kbn) ? 0 : kb + 1;
                ++issued;
                next(xc);
            }
            if (!ok) fail(p.err, flags);
            if (flags[0]) {
                volatile int no_abort = 0;
                for (int64_t j = issued > kXRing ? issued - kXRing : 0; j < issued; ++j)
                    mbar_wait_bounded(&xfull[j % kXRing], (j / kXRing) & 1, &no_abort);
            }
        }
        return;
    }

    // ------------------------------------------------------------------ MMA issue
    // Issuer e takes the units j = e (mod 2) of the piece (those of dequant group e) and
    // accumulates them into its own accumulator of the tile's buffer; it walks every row tile
    // of the piece, also those holding none of its units, so that both issuers and the
    // epilogue agree on the buffer of each tile.
    if (warp == kMmaWarp0 || warp == kMmaWarp1) {
        const int e = warp == kMmaWarp0 ? 0 : 1;
        if (e == 0) {
            tmem_alloc(tmem_slot, kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        named_bar_sync(kBarTmem, kTmemUsers);
        tc_fence_after();
        const uint32_t tbase = *tmem_slot;
        constexpr uint32_t kIdesc = idesc_f16_f32(kRows, MP);
        int64_t seg = 0, j = 0;
        bool live = true;
        Cursor mk;
        first(mk);
        while (live && mk.i < count) {
            const int64_t KB = mat(mk.i).kb;
            const int64_t u0 = mk.j, u1 = mk.e;
            for (int64_t tile = u0 / KB; live && tile <= (u1 - 1) / KB; ++tile, ++seg) {
                const int64_t ja = tile * KB > u0 ? tile * KB : u0;
                const int64_t jb = (tile + 1) * KB < u1 ? (tile + 1) * KB : u1;
                const int b = static_cast<int>(seg % C::kAccBufs);
                if (seg >= C::kAccBufs && !warp_wait(&accempty[b], ((seg / C::kAccBufs) - 1) & 1, flags)) {
                    live = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tbase + C::kAccCol + (e * C::kAccBufs + b) * MP;
                bool fresh = true;
                for (int64_t u = ja; u < jb; ++u, ++j) {
                    if ((j & 1) != e) continue;
                    const int xs = static_cast<int>(j % kXRing);
                    const int a = static_cast<int>(j % C::kNA);
                    const int tb = static_cast<int>(j % kTB);
                    if (!warp_wait(&tfull[tb], (j / kTB) & 1, flags)) {
                        live = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t xaddr = smem_u32(xring + xs * C::kXSlot);
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk) {
                            const uint64_t bdesc = smem_desc_sw128(xaddr + (kk >> 2) * C::kXBox + (kk & 3) * 32);
                            tc_mma_f16_ts(d_tmem, tbase + a * kACols + 8 * kk, bdesc, kIdesc, (!fresh || kk > 0) ? 1u : 0u);
                        }
                        tc_mma_f16_ss(d_tmem, smem_desc_k16(smem_u32(blt + a * kBlBytes)),
                                      smem_desc_k16(smem_u32(xsum + xs * C::kXsBytes)), kIdesc, 1u);
                        tc_commit(&tempty[tb]);
                        tc_commit(&xempty[xs]);
                    }
                    __syncwarp();
                    fresh = false;
                }
                if (!live) break;
                if (lane == 0) tc_commit(&accfull[b]);
                __syncwarp();
            }
            enter(mk, mk.i + 1);
        }
        if (!live && lane == 0) fail(p.err, flags);
        // every MMA issued has finished before the tensor memory is released
        if (lane == 0) {
            tc_commit(&mmadone[e]);
            volatile int no_abort = 0;
            mbar_wait_bounded(&mmadone[e], 0, &no_abort);
        }
        __syncwarp();
        tc_fence_before();
        named_bar_sync(kBarTeardown, kTmemUsers);
        tc_fence_after();
        if (e == 0) tmem_dealloc(tbase, kTmemCols);
        return;
    }

    // ------------------------------------------------------------------ epilogue
    if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        const int q = warp & 3;  // tensor-memory lane quarter
        const int row = 32 * q + lane;
        const int etid = tid - kEpiWarp0 * 32;  // 0..127, one per row (in lane-quarter order)
        named_bar_sync(kBarTmem, kTmemUsers);
        tc_fence_after();
        const uint32_t tq = *tmem_slot + (static_cast<uint32_t>(32 * q) << 16) + C::kAccCol;
        griddep_wait();  // y, the partial slots and the tickets may still be in use by the previous kernel
        int64_t seg = 0, jl = 0;  // jl: local index of the tile's first unit in the piece
        bool live = true;
        // argmax launches: this warp's best key of token m in lane m % 32 (best0: m < 32, best1:
        // m >= 32), over the final values of the rows it owns
        const bool amax = p.amax_keys != nullptr;
        unsigned long long best0 = 0ull, best1 = 0ull;
        // All four warps arrive on `ev` (each at most once per launch); lane 0 of warp
        // kEpiWarp0 then waits for the other three.  False if that wait gave up.
        auto gather = [&](uint64_t* ev) -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(ev);
            return !(warp == kEpiWarp0 && lane == 0) || mbar_wait_bounded(ev, 0, flags);
        };
        Cursor mk;
        first(mk);
        while (live && mk.i < count) {
            const MatDesc& M = mat(mk.i);
            const int64_t KB = M.kb;
            const int64_t u0 = mk.j, u1 = mk.e;
            const int64_t base = M.base;
            for (int64_t tile = u0 / KB; live && tile <= (u1 - 1) / KB; ++tile, ++seg) {
                const int64_t ja = tile * KB > u0 ? tile * KB : u0;
                const int64_t jb = (tile + 1) * KB < u1 ? (tile + 1) * KB : u1;
                const int b = static_cast<int>(seg % C::kAccBufs);
                // which issuers hold units of this tile (issuer e takes local indices = e mod 2)
                const bool has0 = jb - ja >= 2 || (jl & 1) == 0;
                const bool has1 = jb - ja >= 2 || (jl & 1) == 1;
                jl += jb - ja;
                if (!warp_wait(&accfull[b], (seg / C::kAccBufs) & 1, flags)) {
                    live = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tacc0 = tq + b * MP, tacc1 = tq + (C::kAccBufs + b) * MP;
                // columns c0 .. c0 + 15 of the tile's result: issuer 0's sum + issuer 1's sum
                auto load_acc = [&](int c0, float (&acc)[16]) {
                    uint32_t v[16];
                    tmem_ld16((has0 ? tacc0 : tacc1) + c0, v);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] = __uint_as_float(v[i]);
                    if (has0 && has1) {
                        tmem_ld16(tacc1 + c0, v);
                        tc_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[i] += __uint_as_float(v[i]);
                    }
                };
                const bool whole = (ja == tile * KB) && (jb == (tile + 1) * KB);
                const int64_t pa = whole ? c : dev_piece_of(base + tile * KB, U, P);
                const int64_t n = tile * kRows + row;
                if (pa != c) {
                    // a partial for the tile's reducer: [float4 f][128 rows] in this CTA's slot
                    float4* part = reinterpret_cast<float4*>(p.ws + c * static_cast<int64_t>(kRows) * p.ws_cols);
#pragma unroll 1
                    for (int c0 = 0; c0 < MP; c0 += 16) {
                        float acc[16];
                        load_acc(c0, acc);
#pragma unroll
                        for (int f = 0; f < 4; ++f)
                            part[(c0 / 4 + f) * kEpiThreads + etid] =
                                make_float4(acc[4 * f], acc[4 * f + 1], acc[4 * f + 2], acc[4 * f + 3]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&accempty[b]);
                    // publish: one release increment of the tile's ticket after all four warps' writes
                    const bool ok = gather(evpart);
                    if (ok && warp == kEpiWarp0 && lane == 0) red_add_release_gpu(M.tickets + tile, 1);
                    live = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    continue;
                }
                int64_t pb = pa;
                if (!whole) {
                    pb = dev_piece_of(base + (tile + 1) * KB - 1, U, P);
                    bool got = true;
                    if (lane == 0) got = wait_count(M.tickets + tile, static_cast<int>(pb - pa), flags);
                    if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
                        live = false;
                        break;
                    }
                    __syncwarp();  // the other lanes' loads come after lane 0's acquire
                }
#pragma unroll 1
                for (int c0 = 0; c0 < MP; c0 += 16) {
                    float acc[16];
                    load_acc(c0, acc);
#pragma unroll 1
                    for (int64_t pc = pa + 1; pc <= pb; ++pc) {
                        const float4* src = reinterpret_cast<const float4*>(p.ws + pc * static_cast<int64_t>(kRows) * p.ws_cols);
                        float4 pv[4];
#pragma unroll
                        for (int f = 0; f < 4; ++f) pv[f] = __ldcg(src + (c0 / 4 + f) * kEpiThreads + etid);
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            acc[4 * f] += pv[f].x;
                            acc[4 * f + 1] += pv[f].y;
                            acc[4 * f + 2] += pv[f].z;
                            acc[4 * f + 3] += pv[f].w;
                        }
                    }
                    if (amax) {
                        // per token: the warp's largest value (one redux over order-mapped
                        // bits, 0 for rows past N; -0 counts as +0) and its lowest row
                        // (ballot), folded into the owning lane's best key
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int m = c0 + i;
                            if (m >= p.m) break;
                            const uint32_t u = __float_as_uint(acc[i] + 0.0f);  // -0 -> +0
                            const uint32_t o = n < M.n ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
                            const uint32_t mx = __reduce_max_sync(0xffffffffu, o);
                            const int first = __ffs(__ballot_sync(0xffffffffu, o == mx)) - 1;
                            if ((m & 31) == lane && mx != 0u) {
                                const uint32_t nf = static_cast<uint32_t>(n - lane + first);
                                const unsigned long long key =
                                    (static_cast<unsigned long long>(mx) << 32) | (0xFFFFFFFFu - nf);
                                if (m < 32) best0 = key > best0 ? key : best0;
                                else best1 = key > best1 ? key : best1;
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int m = c0 + i;
                            if (m < p.m && n < M.n) M.y[static_cast<int64_t>(m) * M.n + n] = acc[i];
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&accempty[b]);
                // the partials are read: the tile's ticket is ready for the next run
                if (!whole) {
                    const bool ok = gather(evred);
                    if (ok && warp == kEpiWarp0 && lane == 0) M.tickets[tile] = 0;
                    live = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                }
            }
            enter(mk, mk.i + 1);
        }
        if (amax && live) {
            // the CTA's best key per token (over the four warps) goes out as one atomic
            if (lane < MP) amax_sm[q * MP + lane] = best0;
            if (MP > 32 && lane + 32 < MP) amax_sm[q * MP + lane + 32] = best1;
            const bool ok = gather(evamax);
            if (warp == kEpiWarp0) {
                if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                    __syncwarp();  // the other lanes read after lane 0's wait
                    for (int m = lane; m < p.m; m += 32) {
                        unsigned long long k = amax_sm[m];
#pragma unroll
                        for (int w = 1; w < 4; ++w) k = amax_sm[w * MP + m] > k ? amax_sm[w * MP + m] : k;
                        atomicMax(p.amax_keys + m, k);
                    }
                    amax_finish_warp(p, static_cast<int>(gridDim.x), lane);
                } else {
                    live = false;
                }
            }
        }
        if (!live && lane == 0) fail(p.err, flags);
        named_bar_sync(kBarTeardown, kTmemUsers);
        return;
    }

    // ------------------------------------------------------------------ dequant warps
    {
        const int q = warp & 3;   // lane quarter: rows 32q .. 32q+31
        const int g = warp >> 2;  // group: units j = g (mod kGroups)
        const int row = 32 * q + lane;
        named_bar_sync(kBarTmem, kTmemUsers);
        tc_fence_after();
        const uint32_t tlane = *tmem_slot + (static_cast<uint32_t>(32 * q) << 16);
        const int64_t nunits = g1 - g0;
        for (int64_t j = g; j < nunits; j += kGroups) {
            const int s = static_cast<int>(j % kWRing);
            const int a = static_cast<int>(j % C::kNA);
            if (!warp_wait(&wfull[s], (j / kWRing) & 1, flags)) break;
            const uint8_t* u = wring + s * kUnitBytes;
            uint4 qv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) qv[i] = lds128(u + (i * kRows + row) * 16);
            const uint4 hd = lds128(u + kQBytes + row * 16);
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

            // the activation sums of this unit for the -B_l step: X[t][s] = sum of the 32
            // activations of token t in sub-block s (fp16, clamped); MP * 8 of them, shared
            // out over the group's 128 threads.  Formed before the wait for the A buffer: the
            // sums' slot was last read by the MMAs of unit j - kXRing, which finished before
            // the slot was refilled.
            const int xs = static_cast<int>(j % kXRing);
            if (!warp_wait(&xfull[xs], (j / kXRing) & 1, flags)) break;
            const uint8_t* xt = xring + xs * C::kXSlot;
            uint8_t* xst = xsum + xs * C::kXsBytes;
#pragma unroll
            for (int pi = row; pi < MP * 8; pi += kRows) {
                const int t = pi % MP, sb = pi / MP;
                const uint8_t* rowp = xt + (sb >> 1) * C::kXBox + t * 128;
                __half2 acc2 = __float2half2_rn(0.f);
#pragma unroll
                for (int cc4 = 0; cc4 < 4; ++cc4) {
                    const int chunk = ((sb & 1) * 4 + cc4) ^ (t & 7);
                    const uint4 v = lds128(rowp + chunk * 16);
                    acc2 = __hadd2(acc2, __hadd2(__hadd2(as_h2(v.x), as_h2(v.y)), __hadd2(as_h2(v.z), as_h2(v.w))));
                }
                __half sum = __hadd(__low2half(acc2), __high2half(acc2));
                sum = __hmin(__hmax(sum, __ushort_as_half(0xFBFFu)), __ushort_as_half(0x7BFFu));
                *reinterpret_cast<__half*>(xst + (t >> 3) * 256 + (t & 7) * 16 + sb * 2) = sum;
            }

            // the A buffer was last read by the MMAs of unit j - kNA
            if (j >= C::kNA && !warp_wait(&tempty[(j - C::kNA) % kTB], ((j - C::kNA) / kTB) & 1, flags)) break;
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
            // the -B_l step's A row: k slots 0..7 = sub-blocks 0..7 (slots 8..15 stay zero)
            *reinterpret_cast<uint4*>(blt + a * kBlBytes + (row >> 3) * 256 + (row & 7) * 16) =
                make_uint4(ps[0].nbl, ps[1].nbl, ps[2].nbl, ps[3].nbl);
            fence_proxy_async_smem();  // the sums and the -B_l row are read by the tensor core
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tfull[j % kTB]);
        }
        if (flags[0] && lane == 0) fail(p.err, flags);
        named_bar_sync(kBarTeardown, kTmemUsers);
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

int mp_for(int64_t m) { return m <= 16 ? 16 : m <= 32 ? 32 : 64; }

cudaError_t make_mat(MatDesc* out, const uint8_t* wq, const void* x, float* y, int* tickets, int64_t units,
                     int64_t n, int32_t kb, int32_t m) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int64_t k = static_cast<int64_t>(kb) * 256;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(m)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(k) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(mp_for(m))};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&out->xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    out->wq = wq;
    out->y = y;
    out->tickets = tickets;
    out->base = 0;
    out->units = units;
    out->n = n;
    out->kb = kb;
    out->pad = 0;
    return cudaSuccess;
}

template <int MP>
static cudaError_t launch_mp(const MatDesc& single, const LaunchParams& p, int grid, cudaStream_t s, bool pdl,
                             bool cooperative) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<MP>::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = cooperative ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, tc_kernel<MP>, single, p);
}

cudaError_t launch(const MatDesc& single, const LaunchParams& p, int grid, cudaStream_t s, bool pdl, bool cooperative) {
    switch (mp_for(p.m)) {
        case 16: return launch_mp<16>(single, p, grid, s, pdl, cooperative);
        case 32: return launch_mp<32>(single, p, grid, s, pdl, cooperative);
        default: return launch_mp<64>(single, p, grid, s, pdl, cooperative);
    }
}

}  // namespace b2
}  // namespace qmm
