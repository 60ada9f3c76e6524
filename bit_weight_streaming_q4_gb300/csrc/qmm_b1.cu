// Backend 1: Q4_K weight-streaming matmul on warp-level tensor cores (mma.sync m16n8k16),
// for up to 16 stacked rows per launch.
//
// The method (page "Running 4 coding agents on one RTX 3090: a custom CUDA engine for
// Qwen3.8-27B", section "How parallel decoding works"): the M stacked token rows of a
// decode step are multiplied against every weight while that weight is on chip, so the
// weights are read from memory once per step however many rows there are.  The weight
// operand comes straight from registers, so nothing but the packed 4-bit stream crosses
// shared memory.
//
// Arithmetic.  Per super-block and row, w_k = d * sc_j * q_k - dmin * m_j (j = sub-block of
// k), so y = sum over super-blocks of  d * sum_k (sc_j q_k) x_k  -  dmin * sum_j m_j X_j,
// with X_j the sum of the activations of sub-block j.  P_k = sc_j * q_k (an integer <= 945)
// is formed exactly in fp16 from one FMA on the code 1024 + q (or 1024 + 16 q); the tensor
// cores accumulate P x over the super-block in fp32 (exact products).  The min term is one
// more m16n8k16 step per super-block: A = m_j (exact small integers), B = X_j split into an
// fp16 high and low part (fp32 sum of the activations), so it is exact to ~2^-22.  The two
// partial sums are scaled by d and dmin and added to the fp32 accumulator.
//
// Unit = 256 output rows x one super-block column (36864 bytes), written once by repack():
//   bytes [0, 32768)     quants of eight 32-row slices, slice w read by consumer warp w:
//                        [w: 8][m16 tile r: 2][row half h: 2][i4: 2][lane: 32][16 B]; the 16
//                        bytes are the lane's words i = 4 i4 .. 4 i4 + 3; lane (g = lane/4,
//                        t = lane%4) word i of row 32w + 16r + 8h + g is bytes qs[32t + 4i' .. +3]
//                        with i' = (i + 2t) % 8.
//   bytes [32768, 36864) the 16-byte headers of the 256 rows: d and dmin as in the block, then
//                        the same 96 bits of 6-bit scales and mins re-laid as three words Y, Z,
//                        W whose byte t serves quad lane t (sub-blocks j0 = 2t, j1 = 2t+1):
//                        Y_t = sc_j0 << 2 | m_j0 >> 4, Z_t = sc_j1 << 2 | m_j1 >> 4,
//                        W_t = (m_j0 & 15) << 4 | (m_j1 & 15).  Two byte permutes and a few
//                        masks then give every lane its values without branching on t.
// Lane t of a quad reads qs[32t .. 32t+31] of its rows: the low nibbles are weights 64t..64t+31
// (sub-block 2t), the high nibbles weights 64t+32..64t+63 (sub-block 2t+1).  Its eight words
// are visited rotated by 2t, so that at any step the four lanes of a quad use four different
// 16-byte chunks of the swizzled activation tile (no shared-memory bank conflicts).
//
// MMA k-order.  For step s = 0..15 (i = s % 8, i' = (i + 2t) % 8, high = s >= 8) lane t fills
// the MMA k slots {2t, 2t+1, 2t+8, 2t+9} with weight offsets 64t + 32*high + 4i' + {0, 1, 2, 3}
// (repack swaps the middle bytes of each quant word to get this order), so that each pair of
// slots is a pair of adjacent activations.  The min-term step uses, with one n8 fragment,
// slots (2t, 2t+1) for the fp16 high parts of the sums of sub-blocks 2t and 2t+1 and
// (2t+8, 2t+9) for their low parts, so that its A fragment is the lane's pair
// (m_2t, m_2t+1) in every register; with two, (2t, 2t+1) for the high and low part of
// sub-block 2t and (2t+8, 2t+9) for those of 2t+1 (Cfg::kMinPairs).
//
// Warp roles (one persistent CTA per SM; 11 warps of up to 168 registers, or 20 of up to 96):
//   warps 0..W-1 consumers, two or four per SM sub-partition (W = 8 of 32 rows for launches
//               of up to 8 rows, 16 of 16 rows for 9-16): dequantise into MMA A fragments,
//               mma.sync, per-unit scaling, the row tile's result or split-K partial;
//   warp W      weight producer: 1-D bulk copies of whole units into a 4-slot ring, streaming
//               across matrix boundaries without waiting on anything but the ring;
//   warps W+1.. one fragment warp per 8 tokens: 2-D TMA (128-byte swizzle) of its 8 activation
//               rows of each unit, turned into MMA B fragments and sub-block sums (in a
//               persistent step a pre-pass forms each super-block column's fragments once,
//               and the first fragment warp only copies each unit's record);
//   last warp   helper: publishes the CTA's split-K partial with a device-scope release add
//               and resets the ticket of the tile the CTA reduced, so that no consumer waits
//               on a device-wide write.
// Decomposition: a launch concatenates the unit sequences of its matrices (one matrix for a
// run, every matrix of an independent decode step) and CTA c takes the units
// [c*U/P, (c+1)*U/P).  A row tile cut between CTAs pa..pb is reduced by pa, which holds the
// tile's first units and reaches them last, at the end of its piece: the others write their
// partials and move on; pa waits for the ticket to count them and adds them to its own in
// piece order.  Nothing in the order of any output's arithmetic depends on M, so rows are
// bit-identical across batchings.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "qmm_internal.h"
#include "qmm_ptx.cuh"

namespace qmm {
namespace b1 {

constexpr int kQBytes = kRows * 128;            // 32768
constexpr int kWRing = 4;                       // weight slots
constexpr int kXRing = 5;                       // activation slots per 8-token group
constexpr int kFRing = 4;                       // fragment slots
constexpr int kEv = 4;                          // consumer -> helper events in flight
constexpr int kXBox = 8 * 128;                  // one 64-wide k box of 8 tokens (SW128)
constexpr int kXSlot = 4 * kXBox;               // 8 tokens x 256 k

template <int NT>
struct Cfg {
    // Consumer warps: 8 of 32 rows (2 m16 row tiles) for one n8 fragment; 16 of 16 rows for
    // two, where the second fragment doubles the MMAs and four warps per sub-partition hide
    // their latency better (measured on GB300: +4.5 % at 12 rows, -3.6 % at 1 row).
    static constexpr int kWarps = NT == 1 ? 8 : 16;
    static constexpr int kRT = kRows / 16 / kWarps;            // m16 row tiles per consumer warp
    static constexpr int kConsumers = kWarps * 32;
    // Min-term operands: with one n8 fragment the A fragment is the lane's scale-min pair
    // (m_2t, m_2t+1) in every register, against B = the fp16 high parts of sub-blocks 2t, 2t+1,
    // then their low parts; with two, A holds m_2t twice, then m_2t+1 twice, against B =
    // (high, low) of sub-block 2t, then of 2t+1.  Same sums; each was measured the faster one
    // for its width on GB300 (by 4 % at 1-8 rows and 2-3 % at 9-16; the difference is in
    // the compiled schedule of 96-register consumer warps).
    static constexpr bool kMinPairs = NT == 1;
    static_assert(kConsumers <= kConsumerThreads && kWarps * kRT * 16 == kRows, "row split");
    static constexpr int kProducerWarp = kWarps;               // weight units
    static constexpr int kFragWarp0 = kProducerWarp + 1;      // NT fragment warps (one per 8 tokens)
    static constexpr int kHelperWarp = kFragWarp0 + NT;       // publishes partials, resets tickets
    static constexpr int kThreads = (kHelperWarp + 1) * 32;   // 7 or 8 warps: up to 255 registers
    static constexpr int kFragBytes = NT * 8 * 32 * 16;       // [nt][word i][lane][16 B]
    static constexpr int kFSlot = kFragBytes + NT * 32 * 8;   // + min-term fragments [nt][lane][8 B]
    static constexpr int kXOff = kWRing * kUnitBytes;         // 1024-aligned (36864 = 36 * 1024)
    static constexpr int kFOff = kXOff + NT * kXRing * kXSlot;
    static constexpr int kBarOff = kFOff + kFRing * kFSlot;
    static constexpr int kNumBars = 2 * kWRing + NT * kXRing + 2 * kFRing + 2 * kEv;
    // argmax launches: each consumer warp's best key per token, [consumer warp][token 16]
    static constexpr int kBestOff = kBarOff + kNumBars * 8 + 16;
    static constexpr int kSmem = kBestOff + kWarps * 16 * 8 + 1024;
    static_assert(kSmem <= 232448, "shared memory budget");
};

int smem_bytes(int nt) { return nt == 1 ? Cfg<1>::kSmem : Cfg<2>::kSmem; }

// Piece (CTA) holding unit u of the launch's unit sequence.
__device__ __forceinline__ int64_t dev_piece_of(int64_t u, int64_t units, int64_t grid) {
    return ((u + 1) * grid + units - 1) / units - 1;
}

// Record a failure once: the sticky word for the host, the shared abort flag for the CTA.
__device__ __forceinline__ void fail(int* err, volatile int* flags) {
    if (!flags[0]) {
        flags[0] = 1;
        atomicOr(err, 1);
    }
}

// Per row: constants of the lane's two sub-blocks j0 = 2t (fp16x2 lane .x) and j1 = 2t+1 (.y).
struct RowK {
    uint32_t s;    // {sc0, sc1/16}:  code * s + n = sc * q exactly
    uint32_t n;    // {-1024 sc0, -64 sc1}
    uint32_t m;    // {m0, m1}
    uint32_t dd;   // {d, dmin} as fp16
};

// Byte-permute selectors of quad lane t for row_consts: {Y_t, Y_t, Z_t, Z_t}, and then
// {W_t, Y_t, W_t, Z_t} from (W, the first result).
__device__ __forceinline__ uint32_t sel_sc(int t) { return t | (t << 4) | ((4 + t) << 8) | ((4 + t) << 12); }
__device__ __forceinline__ uint32_t sel_mn(int t) { return t | (4 << 4) | (t << 8) | (6 << 12); }

// The row's constants from its re-laid header (the unit layout above).  Every step is exact:
// the 6-bit values go into the mantissa of 1024 (at a power-of-two offset) and one fp16 FMA
// takes the offset and the scaling out.
__device__ __forceinline__ RowK row_consts(uint4 hd, uint32_t selsc, uint32_t selmn) {
    const uint32_t r1 = prmt(hd.y, hd.z, selsc);                  // {Y_t, Y_t, Z_t, Z_t}
    const uint32_t csc = and_or(r1, 0x00FC00FCu, 0x64006400u);    // {1024 + 4 sc0, 1024 + 4 sc1}
    const __half2 sc = __hfma2(as_h2(csc), as_h2(0x24003400u), as_h2(0xCC00DC00u));  // * {1/4, 1/64} - {256, 16}
    const uint32_t r2 = prmt(hd.w, r1, selmn);                   // {W_t, Y_t, W_t, Z_t}
    // {16 m0 at bits 4..9 | m1 low nibble at bits 16..19} | m1 high bits moved to 20..21
    const uint32_t cmn = and_or(r2, 0x000F03F0u, 0x64006400u) | ((r2 >> 4) & 0x00300000u);
    const __half2 mn = __hfma2(as_h2(cmn), as_h2(0x3C002C00u), as_h2(0xE400D400u));  // * {1/16, 1} - {64, 1024}
    RowK r;
    r.s = as_u32(sc);
    r.n = as_u32(__hmul2(sc, as_h2(0xE400E400u)));  // * -1024
    r.m = as_u32(mn);
    r.dd = hd.x;
    return r;
}

// Position in a CTA's piece: unit j of matrix i, whose part of the piece ends at unit e.
struct Cursor {
    int i;
    int64_t j, e;
};

// Bounded spin until *p >= target (acquire).  False on timeout or when the CTA aborts.
__device__ __forceinline__ bool wait_count(const int* p, int target, volatile int* flags, uint64_t lim) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (ld_acquire_gpu(p) >= target) return true;
        if (flags[0]) return false;
        if ((it & 7u) == 7u && globaltimer_ns() - t0 > lim) return false;
        __nanosleep(64);
    }
}

// mbarrier wait whose outcome the whole warp agrees on (all lanes call it).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* flags, uint64_t lim) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, flags, lim));
}

template <int NT>
__global__ void __launch_bounds__(Cfg<NT>::kThreads, 1)
    stream_kernel(const __grid_constant__ MatDesc single, const LaunchParams p) {
    using C = Cfg<NT>;
    constexpr int kWarps = C::kWarps, kRT = C::kRT, kProducerWarp = C::kProducerWarp;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* wring = smem;
    uint8_t* xring = smem + C::kXOff;
    uint8_t* fring = smem + C::kFOff;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* wfull = bars;
    uint64_t* wempty = wfull + kWRing;
    uint64_t* xfull = wempty + kWRing;      // [nt][kXRing]
    uint64_t* ffull = xfull + NT * kXRing;
    uint64_t* fempty = ffull + kFRing;
    uint64_t* evfull = fempty + kFRing;
    uint64_t* evempty = evfull + kEv;
    volatile int* flags = reinterpret_cast<volatile int*>(evempty + kEv);  // [0] abort

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t c = blockIdx.x;
    const int count = p.count;
    const int64_t U = p.units;                 // units of the launch, all matrices
    const int64_t P = gridDim.x;               // pieces
    const int64_t g0 = c * U / P, g1 = (c + 1) * U / P;  // this CTA's piece of the unit sequence
    // matrix i of the launch (a single run passes its matrix by value)
    auto mat = [&](int i) -> const MatDesc& { return count == 1 ? single : p.mats[i]; };
    // move k to the first matrix >= i that has units in the piece
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
            mbar_init(&wempty[i], kWarps);
        }
        for (int i = 0; i < NT * kXRing; ++i) mbar_init(&xfull[i], 1);
        for (int i = 0; i < kFRing; ++i) {
            // fragments formed by the NT fragment warps, or one bulk copy of a precomputed record
            mbar_init(&ffull[i], p.b1_frags ? 1 : NT);
            mbar_init(&fempty[i], kWarps);
        }
        for (int i = 0; i < kEv; ++i) {
            mbar_init(&evfull[i], kWarps);
            mbar_init(&evempty[i], 1);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    griddep_launch_dependents();

    // ------------------------------------------------------------------ weight producer
    if (warp == kProducerWarp) {
        if (lane == 0) {
            // Weights never depend on earlier kernels: stream them from the first instruction,
            // across matrix boundaries, limited only by the ring.
            const uint64_t pol = l2_policy_evict_first();
            Cursor w;
            first(w);
            int64_t wseq = 0;
            bool ok = true;
            int cur = -1;
            const uint8_t* src = nullptr;  // the current matrix's next unit
            while (w.i < count) {
                const int s = static_cast<int>(wseq % kWRing);
                if (wseq >= kWRing && !mbar_wait_bounded(&wempty[s], ((wseq / kWRing) - 1) & 1, flags, p.wait_ns)) {
                    ok = false;
                    break;
                }
                if (w.i != cur) {  // read the matrix's descriptor once
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
                // failure path: let every copy already issued land before the CTA can exit
                volatile int no_abort = 0;
                for (int64_t j = wseq > kWRing ? wseq - kWRing : 0; j < wseq; ++j)
                    mbar_wait_bounded(&wfull[j % kWRing], (j / kWRing) & 1, &no_abort);
            }
        }
        return;
    }

    // ------------------------------------------------------------------ activation fragments
    // Fragment warp nt loads the activations of tokens 8nt..8nt+7 for each unit (2-D TMA,
    // 128-byte swizzle, rows past M read as zero) and turns them into the consumers' MMA B
    // fragments (lane (g, t) of word step i: the 4+4 activations at k = 64t + 4i' and
    // 64t + 32 + 4i', i' = (i + 2t) % 8, in k order) and into the min-term fragments (fp32
    // sums of sub-blocks 2t and 2t+1, split into fp16 hi + lo).
    if (warp >= C::kFragWarp0 && warp < C::kHelperWarp && p.b1_frags) {
        // Precomputed fragments (persistent steps): a pre-pass formed each matrix's records,
        // one per super-block column, and each unit's record is one bulk copy into its slot.
        if (warp == C::kFragWarp0 && lane == 0) {
            Cursor fc;
            first(fc);
            int64_t j = 0;
            bool ok = true;
            int cur = -1, kbn = 1, kb = 0;
            const uint8_t* rec = nullptr;
            griddep_wait();  // the records are written by the pre-pass launched just before
            while (fc.i < count) {
                const int fs = static_cast<int>(j % kFRing);
                if (j >= kFRing && !mbar_wait_bounded(&fempty[fs], ((j / kFRing) - 1) & 1, flags, p.wait_ns)) {
                    ok = false;
                    break;
                }
                if (fc.i != cur) {
                    const MatDesc& M = mat(fc.i);
                    cur = fc.i;
                    rec = M.frag;
                    kbn = M.kb;
                    kb = static_cast<int>(fc.j % kbn);
                }
                uint8_t* fst = fring + fs * C::kFSlot;
                const uint8_t* src = rec + static_cast<int64_t>(kb) * C::kFSlot;
                mbar_arrive_expect_tx(&ffull[fs], C::kFSlot);
                bulk_g2s_nohint(fst, src, C::kFSlot, &ffull[fs]);
                kb = (kb + 1 == kbn) ? 0 : kb + 1;
                ++j;
                next(fc);
            }
            if (!ok) fail(p.err, flags);
            if (flags[0]) {
                // failure path: let every record copy already issued land before exiting
                volatile int no_abort = 0;
                for (int64_t jj = j > kFRing ? j - kFRing : 0; jj < j; ++jj)
                    mbar_wait_bounded(&ffull[jj % kFRing], (jj / kFRing) & 1, &no_abort);
            }
        }
        return;
    }
    if (warp >= C::kFragWarp0 && warp < C::kHelperWarp) {
        const int g = lane >> 2, t = lane & 3;
        const int nt = warp - C::kFragWarp0;
        uint8_t* myx = xring + nt * kXRing * kXSlot;
        uint64_t* myfull = xfull + nt * kXRing;
        Cursor xc;  // next unit whose activations are to be loaded (lane 0)
        first(xc);
        Cursor cc;  // next unit to turn into fragments
        first(cc);
        int64_t issued = 0;
        int cur = -1;   // matrix whose descriptor fields are cached (lane 0)
        const void* xmap = nullptr;
        int kbn = 1, kb = 0;
        // lane 0: TMA of the next unit's activation slice into its ring slot
        auto issue = [&]() {
            if (xc.i != cur) {  // read the matrix's descriptor once
                const MatDesc& M = mat(xc.i);
                cur = xc.i;
                xmap = &M.xmap;
                kbn = M.kb;
                kb = static_cast<int>(xc.j % kbn);
            }
            const int xs = static_cast<int>(issued % kXRing);
            if (issued >= kXRing) fence_proxy_async_smem();  // earlier generic reads of the slot
            mbar_arrive_expect_tx(&myfull[xs], kXSlot);
#pragma unroll
            for (int b = 0; b < 4; ++b) tma_load_2d(myx + xs * kXSlot + b * kXBox, xmap, kb * 256 + 64 * b, 8 * nt, &myfull[xs]);
            kb = (kb + 1 == kbn) ? 0 : kb + 1;
            ++issued;
            next(xc);
        };
        if (lane == 0) {
            griddep_wait();  // activations may be written by the previous kernel
            while (xc.i < count && issued < kXRing) issue();
        }
        __syncwarp();
        for (int64_t j = 0; cc.i < count; ++j, next(cc)) {
            const int xs = static_cast<int>(j % kXRing);
            const int fs = static_cast<int>(j % kFRing);
            bool ok = j < kFRing || warp_wait(&fempty[fs], ((j / kFRing) - 1) & 1, flags, p.wait_ns);
            ok = ok && warp_wait(&myfull[xs], (j / kXRing) & 1, flags, p.wait_ns);
            if (!ok) {
                if (lane == 0) fail(p.err, flags);
                break;
            }
            uint8_t* fst = fring + fs * C::kFSlot;
            const uint8_t* xrow = myx + xs * kXSlot + t * kXBox + g * 128;  // box t, token g of the group
            float sl[8], sh[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int ir = (i + 2 * t) & 7;
                const uint2 vl = lds64(xrow + (((ir >> 1) ^ g) * 16) + (ir & 1) * 8);
                const uint2 vh = lds64(xrow + (((4 + (ir >> 1)) ^ g) * 16) + (ir & 1) * 8);
                // slots (2t, 2t+1) and (2t+8, 2t+9) hold adjacent activation pairs
                *reinterpret_cast<uint4*>(fst + ((nt * 8 + i) * 32 + lane) * 16) = make_uint4(vl.x, vl.y, vh.x, vh.y);
                const float2 a0 = __half22float2(as_h2(vl.x)), a1 = __half22float2(as_h2(vl.y));
                const float2 b0 = __half22float2(as_h2(vh.x)), b1 = __half22float2(as_h2(vh.y));
                sl[i] = (a0.x + a0.y) + (a1.x + a1.y);
                sh[i] = (b0.x + b0.y) + (b1.x + b1.y);
            }
            const float x_lo = ((sl[0] + sl[1]) + (sl[2] + sl[3])) + ((sl[4] + sl[5]) + (sl[6] + sl[7]));
            const float x_hi = ((sh[0] + sh[1]) + (sh[2] + sh[3])) + ((sh[4] + sh[5]) + (sh[6] + sh[7]));
            // X = hi + lo, hi = fp16(X) saturated to the finite range, lo = fp16(X - hi)
            const float lim = 65504.f;
            const float cl = fminf(fmaxf(x_lo, -lim), lim), ch = fminf(fmaxf(x_hi, -lim), lim);
            const __half l_hi = __float2half_rn(cl), h_hi = __float2half_rn(ch);
            const __half l_lo = __float2half_rn(cl - __half2float(l_hi)), h_lo = __float2half_rn(ch - __half2float(h_hi));
            uint2 mt;
            if constexpr (C::kMinPairs) {
                mt.x = as_u32(__halves2half2(l_hi, h_hi));  // slots 2t, 2t+1: high parts
                mt.y = as_u32(__halves2half2(l_lo, h_lo));  // slots 2t+8, 2t+9: low parts
            } else {
                mt.x = as_u32(__halves2half2(l_hi, l_lo));  // slots 2t, 2t+1: sub-block 2t
                mt.y = as_u32(__halves2half2(h_hi, h_lo));  // slots 2t+8, 2t+9: sub-block 2t+1
            }
            *reinterpret_cast<uint2*>(fst + C::kFragBytes + (nt * 32 + lane) * 8) = mt;
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ffull[fs]);
                if (xc.i < count) issue();  // refill this slot (unit j + kXRing)
            }
            __syncwarp();
        }
        if (lane == 0 && flags[0]) {
            // failure path: let every activation copy already issued land before exiting
            volatile int no_abort = 0;
            for (int64_t j = issued > kXRing ? issued - kXRing : 0; j < issued; ++j)
                mbar_wait_bounded(&myfull[j % kXRing], (j / kXRing) & 1, &no_abort);
        }
        return;
    }

    // ------------------------------------------------------------------ helper
    // Publishes the CTA's split-K partial (release add on the tile's ticket) and, after the
    // CTA reduced a tile, resets that tile's ticket; the consumers hand over through the event
    // ring and never wait for a device-wide write.  A piece can share only its first tile
    // without owning it (a partial) and own only its last tile without finishing it (a
    // reduction), so each CTA has at most one of each per launch.
    if (warp == C::kHelperWarp) {
        if (lane == 0) {
            int64_t ev = 0;
            bool ok = true;
            auto take = [&]() -> bool { return mbar_wait_bounded(&evfull[ev % kEv], (ev / kEv) & 1, flags, p.wait_ns); };
            auto give = [&]() {
                mbar_arrive(&evempty[ev % kEv]);
                ++ev;
            };
            Cursor k;
            first(k);
            bool first_part = true;
            while (ok && k.i < count) {
                const MatDesc& M = mat(k.i);
                const int64_t KB = M.kb;
                const int64_t lo = k.j, hi = k.e;
                const int64_t tf = lo / KB, tl = (hi - 1) / KB;
                if (first_part && lo > tf * KB) {
                    // the first tile's first units belong to an earlier CTA: publish the partial
                    if (!(ok = take())) break;
                    red_add_release_gpu(M.tickets + tf, 1);
                    give();
                }
                if (tl * KB >= lo && hi < (tl + 1) * KB) {
                    // this CTA reduced its last tile: every consumer warp has read the ticket
                    if (!(ok = take())) break;
                    M.tickets[tl] = 0;  // ready for the next run
                    give();
                }
                first_part = false;
                enter(k, k.i + 1);
            }
            if (!ok) fail(p.err, flags);
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int g = lane >> 2;
    const int t = lane & 3;
    const uint32_t selsc = sel_sc(t), selmn = sel_mn(t);
    // argmax launches: the best key of each token over this warp's final rows (one lane
    // owns each entry)
    const bool amax = p.amax_keys != nullptr;
    unsigned long long* best = reinterpret_cast<unsigned long long*>(smem + C::kBestOff) + 16 * warp;
    if (lane < 16) best[lane] = 0ull;
    __syncwarp();
    griddep_wait();  // y, the partial slots and the tickets may still be in use by the previous kernel
    uint32_t gseq = 0;  // position in the CTA's unit sequence (ring slots and phases)
    int64_t ev = 0;    // events handed to the helper
    bool live = true;
    auto post = [&]() -> bool {  // hand an event to the helper (after this warp's writes)
        const int e = static_cast<int>(ev % kEv);
        __syncwarp();
        if (ev >= kEv && !warp_wait(&evempty[e], ((ev / kEv) - 1) & 1, flags, p.wait_ns)) {
            if (lane == 0) fail(p.err, flags);
            return false;
        }
        if (lane == 0) mbar_arrive(&evfull[e]);
        ++ev;
        return true;
    };
    Cursor mk;  // walks the matrices of the piece
    first(mk);
    while (live && mk.i < count) {
        const MatDesc& M = mat(mk.i);
        const int64_t u0 = mk.j, u1 = mk.e;  // this piece's units of matrix mk.i
        const int KB = M.kb;
        const int64_t base = M.base;
        for (int64_t tile = u0 / KB; live && tile <= (u1 - 1) / KB; ++tile) {
            const int64_t ja = tile * KB > u0 ? tile * KB : u0;
            const int64_t jb = (tile + 1) * KB < u1 ? (tile + 1) * KB : u1;

            float acc[kRT][NT][4];
#pragma unroll
            for (int r = 0; r < kRT; ++r)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[r][nt][e] = 0.f;

            const uint32_t nj = static_cast<uint32_t>(jb - ja);  // (a piece has < 2^31 units)
            for (uint32_t jj = 0; jj < nj; ++jj, ++gseq) {
                const int s = static_cast<int>(gseq % kWRing);
                const int fs = static_cast<int>(gseq % kFRing);
                if (!warp_wait(&wfull[s], (gseq / kWRing) & 1, flags, p.wait_ns)) {
                    if (lane == 0) fail(p.err, flags);
                    live = false;
                    break;
                }
                // this warp's words: [r][h][i4][lane][16 B], word i = 4 i4 + component (rows 64 warp + 16 r + 8 h + g)
                const uint8_t* myq = wring + s * kUnitBytes + warp * (kRT * 2048);
                RowK rk[kRT][2];
#pragma unroll
                for (int r = 0; r < kRT; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        rk[r][h] = row_consts(lds128(wring + s * kUnitBytes + kQBytes + (16 * kRT * warp + 16 * r + 8 * h + g) * 16), selsc, selmn);
                uint4 qv[kRT][2];  // words of the current half (i4) of the unit
#pragma unroll
                for (int r = 0; r < kRT; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        qv[r][h] = lds128(myq + (((r * 2 + h) * 2 + 0) * 32 + lane) * 16);

                if (!warp_wait(&ffull[fs], (gseq / kFRing) & 1, flags, p.wait_ns)) {
                    if (lane == 0) fail(p.err, flags);
                    live = false;
                    break;
                }
                const uint8_t* fst = fring + fs * C::kFSlot;

                float dp[kRT][NT][4];
#pragma unroll
                for (int r = 0; r < kRT; ++r)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) dp[r][nt][e] = 0.f;

#pragma unroll
                for (int i = 0; i < 8; ++i) {  // word i: step (i, low nibbles) then (i, high nibbles)
                    if (i == 4) {
                        // second half of the words; then the weight slot is no longer read
#pragma unroll
                        for (int r = 0; r < kRT; ++r)
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                qv[r][h] = lds128(myq + (((r * 2 + h) * 2 + 1) * 32 + lane) * 16);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&wempty[s]);
                    }
                    uint4 f[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) f[nt] = lds128(fst + ((nt * 8 + i) * 32 + lane) * 16);
#pragma unroll
                    for (int r = 0; r < kRT; ++r) {
                        uint32_t alo[4], ahi[4];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint4 qq = qv[r][h];
                            const uint32_t w = (i & 3) == 0 ? qq.x : (i & 3) == 1 ? qq.y : (i & 3) == 2 ? qq.z : qq.w;
                            const uint32_t w8 = w >> 8;
                            const __half2 s_lo = __low2half2(as_h2(rk[r][h].s)), n_lo = __low2half2(as_h2(rk[r][h].n));
                            const __half2 s_hi = __high2half2(as_h2(rk[r][h].s)), n_hi = __high2half2(as_h2(rk[r][h].n));
                            // P = sc*q, exact: code * s + n
                            alo[h] = as_u32(__hfma2(as_h2(and_or_pinned(w, 0x000F000Fu, 0x64006400u)), s_lo, n_lo));
                            alo[2 + h] = as_u32(__hfma2(as_h2(and_or_pinned(w8, 0x000F000Fu, 0x64006400u)), s_lo, n_lo));
                            ahi[h] = as_u32(__hfma2(as_h2(and_or_pinned(w, 0x00F000F0u, 0x64006400u)), s_hi, n_hi));
                            ahi[2 + h] = as_u32(__hfma2(as_h2(and_or_pinned(w8, 0x00F000F0u, 0x64006400u)), s_hi, n_hi));
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma_m16n8k16(dp[r][nt], alo[0], alo[1], alo[2], alo[3], f[nt].x, f[nt].y);
                            mma_m16n8k16(dp[r][nt], ahi[0], ahi[1], ahi[2], ahi[3], f[nt].z, f[nt].w);
                        }
                    }
                }

                // min term: sum_j m_j X_j with X split into fp16 hi + lo
                uint2 xb[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) xb[nt] = lds64(fst + C::kFragBytes + (nt * 32 + lane) * 8);
                __syncwarp();
                if (lane == 0) mbar_arrive(&fempty[fs]);
#pragma unroll
                for (int r = 0; r < kRT; ++r) {
                    // A (rows g and g+8): the pairs (m_2t, m_2t+1) as they are, or each m twice
                    uint32_t a0 = rk[r][0].m, a1 = rk[r][1].m, a2 = a0, a3 = a1;
                    if constexpr (!C::kMinPairs) {
                        a0 = as_u32(__low2half2(as_h2(rk[r][0].m)));
                        a2 = as_u32(__high2half2(as_h2(rk[r][0].m)));
                        a1 = as_u32(__low2half2(as_h2(rk[r][1].m)));
                        a3 = as_u32(__high2half2(as_h2(rk[r][1].m)));
                    }
                    const float2 dd0 = __half22float2(as_h2(rk[r][0].dd)), dd1 = __half22float2(as_h2(rk[r][1].dd));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        float dm[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_m16n8k16(dm, a0, a1, a2, a3, xb[nt].x, xb[nt].y);
                        acc[r][nt][0] = fmaf(dd0.x, dp[r][nt][0], acc[r][nt][0]);
                        acc[r][nt][1] = fmaf(dd0.x, dp[r][nt][1], acc[r][nt][1]);
                        acc[r][nt][2] = fmaf(dd1.x, dp[r][nt][2], acc[r][nt][2]);
                        acc[r][nt][3] = fmaf(dd1.x, dp[r][nt][3], acc[r][nt][3]);
                        acc[r][nt][0] = fmaf(-dd0.y, dm[0], acc[r][nt][0]);
                        acc[r][nt][1] = fmaf(-dd0.y, dm[1], acc[r][nt][1]);
                        acc[r][nt][2] = fmaf(-dd1.y, dm[2], acc[r][nt][2]);
                        acc[r][nt][3] = fmaf(-dd1.y, dm[3], acc[r][nt][3]);
                    }
                }
            }
            if (!live) break;

            // ---------------- the row tile: whole, reduced here, or a partial for its reducer
            // A tile cut between pieces pa..pb is reduced by pa, the CTA holding its first units
            // (it reaches them last, at the end of its piece): the others write their partials
            // and move on; pa waits for the ticket to count them and adds them in piece order.
            const bool whole = (ja == tile * KB) && (jb == (tile + 1) * KB);
            const int64_t pa = whole ? c : dev_piece_of(base + tile * KB, U, P);
            if (pa != c) {
                // (only the first tile of a piece can be shared without being owned)
                float4* part = reinterpret_cast<float4*>(p.ws + c * static_cast<int64_t>(kConsumerThreads) * p.ws_cols);
#pragma unroll
                for (int r = 0; r < kRT; ++r)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        part[(r * NT + nt) * C::kConsumers + tid] =
                            make_float4(acc[r][nt][0], acc[r][nt][1], acc[r][nt][2], acc[r][nt][3]);
                live = post();
                continue;
            }
            if (!whole) {
                // wait for the partials of pieces pa+1..pb, then add them in that order
                const int64_t pb = dev_piece_of(base + (tile + 1) * KB - 1, U, P);
                bool got = true;
                if (lane == 0) got = wait_count(M.tickets + tile, static_cast<int>(pb - pa), flags, p.wait_ns);
                if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
                    if (lane == 0) fail(p.err, flags);
                    live = false;
                    break;
                }
                __syncwarp();  // the other lanes' loads come after lane 0's acquire
                constexpr int kB = NT == 1 ? 8 : 4;  // partials whose loads are in flight together
#pragma unroll 1
                for (int64_t pc0 = pa + 1; pc0 <= pb; pc0 += kB) {
                    float4 v[kB][kRT * NT];
#pragma unroll
                    for (int q = 0; q < kB; ++q) {
                        const int64_t pq = pc0 + q <= pb ? pc0 + q : pb;  // (loaded, not added)
                        const float4* src = reinterpret_cast<const float4*>(
                            p.ws + pq * static_cast<int64_t>(kConsumerThreads) * p.ws_cols);
#pragma unroll
                        for (int f = 0; f < kRT * NT; ++f) v[q][f] = __ldcg(src + f * C::kConsumers + tid);
                    }
#pragma unroll
                    for (int q = 0; q < kB; ++q) {
                        if (pc0 + q <= pb) {
#pragma unroll
                            for (int r = 0; r < kRT; ++r)
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    acc[r][nt][0] += v[q][r * NT + nt].x;
                                    acc[r][nt][1] += v[q][r * NT + nt].y;
                                    acc[r][nt][2] += v[q][r * NT + nt].z;
                                    acc[r][nt][3] += v[q][r * NT + nt].w;
                                }
                        }
                    }
                }
            }
            if (amax) {
                // token m = 8 nt + 2 t + par: the best of this thread's 8 rows, then of the
                // 8 lanes sharing t (g = 0..7); lane t keeps the warp's best
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int par = 0; par < 2; ++par) {
                        unsigned long long key = 0ull;
#pragma unroll
                        for (int r = 0; r < kRT; ++r)
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int64_t n = tile * kRows + 16 * kRT * warp + 16 * r + g + 8 * h;
                                if (n < M.n) {
                                    const unsigned long long k = amax_key(acc[r][nt][2 * h + par], n);
                                    key = k > key ? k : key;
                                }
                            }
#pragma unroll
                        for (int sh = 4; sh < 32; sh <<= 1) {
                            const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, sh);
                            key = o > key ? o : key;
                        }
                        const int m = nt * 8 + 2 * t + par;
                        if (g == 0 && m < p.m && key > best[m]) best[m] = key;
                    }
            } else {
#pragma unroll
                for (int r = 0; r < kRT; ++r)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int row = 16 * kRT * warp + 16 * r + g + 8 * (e >> 1);
                            const int m = nt * 8 + 2 * t + (e & 1);
                            const int64_t n = tile * kRows + row;
                            if (m < p.m && n < M.n) M.y[static_cast<int64_t>(m) * M.n + n] = acc[r][nt][e];
                        }
            }
            if (!whole) live = post();  // the helper may now reset the tile's ticket
        }
        enter(mk, mk.i + 1);
    }
    if (amax && live) {
        __syncwarp();
        if (lane < p.m) atomicMax(p.amax_keys + lane, best[lane]);
        amax_finish_warp(p, kWarps * static_cast<int>(gridDim.x), lane);
    }
}

// One thread per 16-byte piece of the packed layout.
__global__ void repack_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t n, int32_t kb,
                              int64_t units) {
    constexpr int kSegs = kUnitBytes / 16;  // 2304
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= units * kSegs) return;
    const int64_t u = idx / kSegs;
    const int seg = static_cast<int>(idx % kSegs);
    const int64_t tile = u / kb;
    const int b = static_cast<int>(u % kb);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (seg < kQBytes / 16) {
        // 16 output bytes = words 4 i4 .. 4 i4 + 3 of one lane of one (w, r, h) row group
        const int w = seg >> 8, r = (seg >> 7) & 1, h = (seg >> 6) & 1, i4 = (seg >> 5) & 1, lane = seg & 31;
        const int g = lane >> 2, t = lane & 3;
        const int row = 32 * w + 16 * r + 8 * h + g;
        const int64_t nrow = tile * kRows + row;
        if (nrow < n) {
            const uint32_t* qs = reinterpret_cast<const uint32_t*>(src + (nrow * kb + b) * 144 + 16 + 32 * t);
            uint32_t wv[4];
            // bytes 1 and 2 of each word swapped: the low nibbles at bits 0 and 16 (and, after a
            // shift by 8, at bits 8 and 24) are then weights k, k+1 (k+2, k+3)
            for (int e = 0; e < 4; ++e) wv[e] = __byte_perm(qs[(4 * i4 + e + 2 * t) & 7], 0, 0x3120);
            v = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
    } else {
        // the row's header: d and dmin unchanged, the twelve scale bytes re-laid so that lane t
        // of a quad finds (sc, m) of its sub-blocks 2t, 2t+1 in byte t of words 1..3
        const int row = seg - kQBytes / 16;
        const int64_t nrow = tile * kRows + row;
        if (nrow < n) {
            const uint8_t* hb = src + (nrow * kb + b) * 144;
            uint32_t y = 0, z = 0, w = 0;
            for (int t = 0; t < 4; ++t) {
                int sc[2], mn[2];
                for (int e = 0; e < 2; ++e) {
                    const int j = 2 * t + e;  // GGUF 6-bit (scale, min) packing of sub-block j
                    if (j < 4) {
                        sc[e] = hb[4 + j] & 63;
                        mn[e] = hb[8 + j] & 63;
                    } else {
                        sc[e] = (hb[8 + j] & 0x0F) | ((hb[j] >> 6) << 4);
                        mn[e] = (hb[8 + j] >> 4) | ((hb[4 + j] >> 6) << 4);
                    }
                }
                y |= static_cast<uint32_t>((sc[0] << 2) | (mn[0] >> 4)) << (8 * t);
                z |= static_cast<uint32_t>((sc[1] << 2) | (mn[1] >> 4)) << (8 * t);
                w |= static_cast<uint32_t>(((mn[0] & 15) << 4) | (mn[1] & 15)) << (8 * t);
            }
            v = make_uint4(*reinterpret_cast<const uint32_t*>(hb), y, z, w);
        }
    }
    *reinterpret_cast<uint4*>(dst + u * kUnitBytes + static_cast<int64_t>(seg) * 16) = v;
}

cudaError_t repack(const uint8_t* src_dev, uint8_t* dst_dev, const Decomp& d, cudaStream_t s) {
    const int64_t total = d.units * (kUnitBytes / 16);
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    repack_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(src_dev, dst_dev, d.n, static_cast<int32_t>(d.kb),
                                                                   d.units);
    return cudaGetLastError();
}

cudaError_t configure() {
    cudaError_t e = cudaFuncSetAttribute(stream_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<1>::kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(stream_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<2>::kSmem);
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

template <int NT>
static cudaError_t launch_nt(const MatDesc& single, const LaunchParams& p, int grid, cudaStream_t s, bool pdl,
                             bool cooperative) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(Cfg<NT>::kThreads);
    cfg.dynamicSmemBytes = Cfg<NT>::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = cooperative ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, stream_kernel<NT>, single, p);
}

cudaError_t make_mat(MatDesc* out, const uint8_t* wq, const void* x, float* y, int* tickets, int64_t units,
                     int64_t n, int32_t kb, int32_t m) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int64_t k = static_cast<int64_t>(kb) * 256;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(m)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(k) * 2};
    const cuuint32_t box[2] = {64, 8};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&out->xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    out->xsrc = static_cast<const __half*>(x);
    out->xs = nullptr;
    out->frag = nullptr;
    memset(&out->ymap, 0, sizeof(out->ymap));
    out->ytma = 0;
    out->wq = wq;
    out->y = y;
    out->tickets = tickets;
    out->base = 0;
    out->units = units;
    out->n = n;
    out->kb = kb;
    out->pieces = 0;
    return cudaSuccess;
}

// One warp per 8 tokens, one block per (super-block column, matrix): the record of column kb
// of a matrix, exactly what the fragment warps form from the unit's activation tile (same
// loads, same fp32 additions in the same order), rows past m as zeros.
template <int NT>
__global__ void __launch_bounds__(32 * NT) frag_kernel(const __grid_constant__ MatDesc single, const LaunchParams p) {
    using C = Cfg<NT>;
    const MatDesc& M = p.count == 1 ? single : p.mats[blockIdx.y];
    const int kb = blockIdx.x;
    if (kb >= M.kb) return;
    const int nt = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int m = 8 * nt + g;
    const int64_t k = static_cast<int64_t>(M.kb) * 256;
    const __half* xr = M.xsrc + static_cast<int64_t>(m) * k + kb * 256 + 64 * t;
    uint8_t* fst = M.frag + static_cast<int64_t>(kb) * C::kFSlot;
    float sl[8], sh[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int ir = (i + 2 * t) & 7;
        uint2 vl = make_uint2(0u, 0u), vh = make_uint2(0u, 0u);
        if (m < p.m) {
            vl = *reinterpret_cast<const uint2*>(xr + 8 * (ir >> 1) + 4 * (ir & 1));
            vh = *reinterpret_cast<const uint2*>(xr + 32 + 8 * (ir >> 1) + 4 * (ir & 1));
        }
        *reinterpret_cast<uint4*>(fst + ((nt * 8 + i) * 32 + lane) * 16) = make_uint4(vl.x, vl.y, vh.x, vh.y);
        const float2 a0 = __half22float2(as_h2(vl.x)), a1 = __half22float2(as_h2(vl.y));
        const float2 b0 = __half22float2(as_h2(vh.x)), b1 = __half22float2(as_h2(vh.y));
        sl[i] = (a0.x + a0.y) + (a1.x + a1.y);
        sh[i] = (b0.x + b0.y) + (b1.x + b1.y);
    }
    const float x_lo = ((sl[0] + sl[1]) + (sl[2] + sl[3])) + ((sl[4] + sl[5]) + (sl[6] + sl[7]));
    const float x_hi = ((sh[0] + sh[1]) + (sh[2] + sh[3])) + ((sh[4] + sh[5]) + (sh[6] + sh[7]));
    const float lim = 65504.f;
    const float cl = fminf(fmaxf(x_lo, -lim), lim), ch = fminf(fmaxf(x_hi, -lim), lim);
    const __half l_hi = __float2half_rn(cl), h_hi = __float2half_rn(ch);
    const __half l_lo = __float2half_rn(cl - __half2float(l_hi)), h_lo = __float2half_rn(ch - __half2float(h_hi));
    uint2 mt;
    if constexpr (C::kMinPairs) {
        mt.x = as_u32(__halves2half2(l_hi, h_hi));
        mt.y = as_u32(__halves2half2(l_lo, h_lo));
    } else {
        mt.x = as_u32(__halves2half2(l_hi, l_lo));
        mt.y = as_u32(__halves2half2(h_hi, h_lo));
    }
    *reinterpret_cast<uint2*>(fst + C::kFragBytes + (nt * 32 + lane) * 8) = mt;
}

int64_t frag_record_bytes(int64_t m) { return m <= 8 ? Cfg<1>::kFSlot : Cfg<2>::kFSlot; }

cudaError_t prefrag(const MatDesc& single, const LaunchParams& p, int32_t max_kb, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(max_kb), static_cast<unsigned>(p.count));
    if (p.m <= 8)
        frag_kernel<1><<<grid, 32, 0, s>>>(single, p);
    else
        frag_kernel<2><<<grid, 64, 0, s>>>(single, p);
    return cudaGetLastError();
}

cudaError_t launch(const MatDesc& single, const LaunchParams& p, int grid, cudaStream_t s, bool pdl, bool cooperative) {
    return p.m <= 8 ? launch_nt<1>(single, p, grid, s, pdl, cooperative)
                    : launch_nt<2>(single, p, grid, s, pdl, cooperative);
}

}  // namespace b1
}  // namespace qmm
