// Backend 2: Q4_K weight-streaming matmul on the 5th-generation tensor cores (tcgen05).
//
// The method (page "Running 4 coding agents on one RTX 3090: a custom CUDA engine for
// Qwen3.8-27B", section "How parallel decoding works"): every weight is read from memory
// once per step and multiplied against all M stacked token rows while it is on chip.  The
// tensor-core instruction costs the same for any N up to 64, so this backend serves runs of
// more than 8 rows: up to 64 per launch for decode, and 128 per launch (twice the tensor-core
// time per unit, half the weight passes) for longer runs such as a chunked prefill.
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
//               burst has drained, so two issuers take turns.  At MP = 64 (Q4_K) a group
//               hands each unit over in two halves: the issuer starts the MMAs of
//               sub-blocks 0-3 while the group still dequantises sub-blocks 4-7;
//   warps 11-14 epilogue: the sum of the two accumulators -> y, a split-K partial, or the
//               reduction of a split row tile; warp 11 also publishes the CTA's partial and
//               resets the ticket of the tile it reduced.
// Decomposition: a launch concatenates its matrices' unit sequences and CTA c takes
// [c*U/P, (c+1)*U/P), so only CTA boundaries split a row tile.  A tile split between CTAs
// pa..pb is normally reduced by pa (it reaches the tile last, at the end of its piece):
// pa+1..pb write fp32 partials and publish them with one add on the tile's ticket; pa reads
// the ticket once and adds the partials to its own in piece order.  If they are not all in
// (a late CTA), pa parks its partial as well and the last CTA to arrive adds them up in the
// same order, so no CTA ever waits for another and launches need not be co-resident.
// Nothing in any output's arithmetic depends on M.
//
// Dequantisation, exact to ~1 ulp of fp16 for every input: with code c = 1024 + q (or
// 1024 + 16q), P = sc*q is exact from one fp16 FMA; B = dmin*m splits error-free into
// B_h + B_l; the weight written is fp16(d*P - B_h), and the -B_l part goes to the tensor
// core as one extra K=16 step per unit: A = -B_l of the 8 sub-blocks (a small tile in
// shared memory), B = the activation sums of the 8 sub-blocks.
#include <cstring>
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
constexpr int kBarTmem = 1, kBarTeardown = 2, kBarEpi = 3;
constexpr int kTmemUsers = (kDqWarps + 2 + 4) * 32;  // dequant + MMA + epilogue warps

// Ring depths (weight slots, activation slots) per block format and tile width, as deep as
// shared memory allows; each a multiple of kGroups so that a slot always serves one group.
constexpr int w_ring(int f, int mp) {
    return mp == 128 ? (f == QMM_FORMAT_Q4_K ? 4 : 2)
                     : f == QMM_FORMAT_Q4_K ? (mp == 16 ? 8 : mp == 32 ? 6 : 4) : f == QMM_FORMAT_Q6_K ? (mp == 64 ? 4 : 6) : 4;
}
// A dependent persistent step (dep) of Q4_K at up to 32 rows takes two x slots fewer, which
// makes room for the epilogue's staging tile: there every matrix's outputs must be complete
// before the next matrix's activations load, so the epilogue sits on the critical path
// (measured on GB300, 16-layer step at M = 12: 1.35 against 1.57 ms, while the independent
// step loses 4 % with the shallower ring and keeps it).
constexpr int x_ring(int f, int mp, bool dep = false) {
    return mp == 128 ? 2
                     : f == QMM_FORMAT_Q4_K ? (mp == 16 ? (dep ? 6 : 8) : mp == 32 ? (dep ? 4 : 6) : 4)
                                            : mp == 16 ? (f == QMM_FORMAT_Q6_K ? 6 : 8) : mp == 32 ? 4 : 2;
}

template <int MP, int F, bool D = false>
struct Cfg {
    static constexpr int kUnitBytes = unit_bytes(F);
    static constexpr bool kMin = F == QMM_FORMAT_Q4_K;  // the format has a min term (the -B_l step)
    // MP = 128: shared memory holds two x tiles only, so the MMA issuers wait for a unit's x
    // tile themselves and the dequantisation groups never touch x; the activation sums of the
    // -B_l step come from the pre-pass (presum_for) with the tile
    static constexpr bool kIssuerWaitsX = MP == 128;
    static constexpr bool kPre = kMin && kIssuerWaitsX;
    // registers per dequantisation thread after the warpgroup split (0: no split, 128 for all)
    static constexpr int kRegSplit = F == QMM_FORMAT_Q6_K ? 176 : (F == QMM_FORMAT_Q4_K && MP >= 64) ? 152 : 0;
    static constexpr int kWRing = w_ring(F, MP);
    static constexpr int kXRing = x_ring(F, MP, D);
    static constexpr int kXBox = MP * 128;    // one 64-wide k box of x
    static constexpr int kXSlot = 4 * kXBox;  // x tile of one unit
    static constexpr int kXsBytes = kMin ? MP * 32 : 0;  // the B tile of the -B_l step: [k half 2][MP tokens][8 fp16]
    // A buffers in tensor memory (unit j -> buffer j mod kNA): three where tensor memory has
    // room, so that a group can dequantise its next unit while the tensor core still reads
    // the last two; two from MP = 64 on, where the accumulators take the room.  Accumulators:
    // two buffers per issuer, so that the epilogue of a tile overlaps the next tile's MMAs,
    // except at MP = 128 (one: a tile's MMAs wait for the epilogue of the tile before).
    static constexpr int kNA = MP >= 64 ? 2 : 3;
    static constexpr int kAccBufs = MP == 128 ? 1 : 2;
    static constexpr int kAccCol = kNA * kACols;  // accumulator (issuer e, buffer b) at + (e * kAccBufs + b) * MP
    static_assert(kAccCol + 2 * kAccBufs * MP <= kTmemCols, "tensor memory budget");
    static_assert(kTB % kNA == 0 && kTB % 2 == 0, "one barrier pair per unit mod kTB");
    static_assert(kWRing % kGroups == 0 && kXRing % kGroups == 0, "a slot must always feed the same group");
    static constexpr int kWOff = kXRing * kXSlot;
    static constexpr int kXsOff = kWOff + kWRing * kUnitBytes;
    static constexpr int kBlOff = kXsOff + kXRing * kXsBytes;
    static constexpr int kBarOff = kBlOff + (kMin ? kNA * kBlBytes : 0);
    // Half-unit hand-off: the group signals sub-blocks 0-3 of a unit (tfull_lo) before it
    // writes 4-7, and the issuer runs their 8 MMAs meanwhile.  Measured on this GB300 with
    // identical outputs: +4-5 % at MP = 64, but -9 % at MP = 16, -3 % at MP = 32 and MP = 128,
    // where the issuer's extra wait right after a burst of MMAs costs more than it saves.
    static constexpr bool kSplit = F == QMM_FORMAT_Q4_K && MP == 64;
    static_assert(!kSplit || !kIssuerWaitsX, "the first half's MMAs rely on the group's wait for the x tile");
    // wfull, wempty, xfull, xempty, tfull, tempty, accfull[2], accempty[2], mmadone[2], tfull_lo
    static constexpr int kNumBars = 2 * kWRing + 2 * kXRing + 2 * kTB + 6 + (kSplit ? kTB : 0);
    // argmax launches: the epilogue warps' best keys, [warp 4][token MP]
    static constexpr int kAmaxOff = (kBarOff + kNumBars * 8 + 16 + 127) / 128 * 128;  // 128-byte aligned (bulk stores)
    // ... which y launches use instead, where shared memory has the room, as the epilogue's
    // staging tile, [token 16][row 128] fp32: the four warps write 16 tokens of their rows
    // there and one thread stores the tile to y with a bulk tensor store (one value per thread
    // and store instruction took ≈ 19 K clocks for a 128 x 128 tile while the weight stream
    // ran, measured on GB300)
    static constexpr int kStageBytes = 4 * 16 * 32 * 4;
    static constexpr int kAmaxBytes = 4 * MP * 8;
    static constexpr int kSmemPlain = kAmaxOff + kAmaxBytes + 1024;  // + alignment slack
    static constexpr int kSmemStaged = kAmaxOff + (kAmaxBytes > kStageBytes ? kAmaxBytes : kStageBytes) + 1024;
    // (not for Q6_K, whose epilogue warps run at 80 registers and would spill)
    static constexpr bool kStage = kSmemStaged <= 232448 && F != QMM_FORMAT_Q6_K;
    static constexpr int kSmem = kStage ? kSmemStaged : kSmemPlain;
    static_assert(kSmem <= 232448, "shared memory budget");
};

__device__ __forceinline__ int64_t dev_piece_of(int64_t u, int64_t units, int64_t grid) {
    return ((u + 1) * grid + units - 1) / units - 1;
}

// First unit of piece c of `units` cut into `grid` pieces.
__device__ __forceinline__ int64_t dev_piece_start(int64_t c, int64_t units, int64_t grid) {
    return c * units / grid;
}

__device__ __forceinline__ void fail(int* err, volatile int* flags) {
    if (!flags[0]) {
        flags[0] = 1;
        atomicOr(err, 1);
    }
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* flags, uint64_t lim) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, flags, lim));
}

// Bounded spin until *p >= target (acquire, device scope).  False on timeout or abort.
__device__ __forceinline__ bool wait_count(const int* p, int target, volatile int* flags, uint64_t lim) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (ld_acquire_gpu(p) >= target) return true;
        if (flags[0]) return false;
        if ((it & 7u) == 7u && globaltimer_ns() - t0 > lim) return false;
        __nanosleep(32);
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

// ---------------------------------------------------------------- Q8_0 and Q6_K units
// Q8_0 unit (34,816 B, by repack()): quants [block 8][row 128][32 B] (the 32 int8 of the
// row's block, in order), then the blocks' d [row 128][8 x fp16].  A byte b of quant q maps
// to the fp16 code 1024 + (q + 128) (byte ^ 0x80 OR-ed into the mantissa of 1024), so
// q = code - 1152 exactly and the weight is fp16(q * d), one rounding.
__device__ __forceinline__ void q80_word(uint32_t w, __half2 d2, uint32_t* out) {
    const uint32_t xw = w ^ 0x80808080u;
    const __half2 nb = as_h2(0xE480E480u);  // -1152
    out[0] = as_u32(__hmul2(__hadd2(as_h2(prmt(xw, 0x64646464u, 0x4140u)), nb), d2));
    out[1] = as_u32(__hmul2(__hadd2(as_h2(prmt(xw, 0x64646464u, 0x4342u)), nb), d2));
}

__device__ __forceinline__ void dq_unit_q80(const uint8_t* u, int row, uint32_t tcol) {
    const uint4 dv = lds128(u + kRows * 256 + row * 16);
    const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const uint4 qa = lds128(u + (b * kRows + row) * 32);
        const uint4 qb = lds128(u + (b * kRows + row) * 32 + 16);
        const __half2 d2 = (b & 1) ? __high2half2(as_h2(dw[b >> 1])) : __low2half2(as_h2(dw[b >> 1]));
        uint32_t out[16];
        q80_word(qa.x, d2, out + 0);
        q80_word(qa.y, d2, out + 2);
        q80_word(qa.z, d2, out + 4);
        q80_word(qa.w, d2, out + 6);
        q80_word(qb.x, d2, out + 8);
        q80_word(qb.y, d2, out + 10);
        q80_word(qb.z, d2, out + 12);
        q80_word(qb.w, d2, out + 14);
        tmem_st16(tcol + 16 * b, out);
    }
}

// Q6_K unit (26,880 B, by repack()): low nibbles [chunk 8][row 128][16 B] (chunk c = weights
// 32c .. 32c+31, words as in the Q4_K layout: nibble e of word i at bit 0,16,4,20,8,24,12,28),
// high bit pairs [chunk 8][row 128][8 B] (a 16-bit field per word: e0,e4,e2,e6 in the low
// byte, e1,e5,e3,e7 in the high byte, 2 bits each), scales [row 128][16 x int8], d [row 128]
// [fp16].  The field, spread to bits 4-11 and 20-27 of a word, supplies the high bits of
// codes 1024 + q (bits 4-5) and 1024 + 16q (bits 8-9) with one mask each, and those of the
// shifted codes after >> 2.  q - 32 is then exact in fp16, and the weight is
// fp16((q - 32) * (ds_h + ds_l)) with d * sc = ds_h + ds_l split exactly in fp32.
__device__ __forceinline__ void q6_word(uint32_t w, uint32_t h, __half2 dsh, __half2 dsl, uint32_t* out) {
    const uint32_t w8 = w >> 8, h2 = h >> 2;
    const uint32_t c01 = and_or(h, 0x00300030u, and_or(w, 0x000F000Fu, 0x64006400u));
    const uint32_t c23 = and_or(h, 0x03000300u, and_or(w, 0x00F000F0u, 0x64006400u));
    const uint32_t c45 = and_or(h2, 0x00300030u, and_or(w8, 0x000F000Fu, 0x64006400u));
    const uint32_t c67 = and_or(h2, 0x03000300u, and_or(w8, 0x00F000F0u, 0x64006400u));
    const __half2 n1056 = as_h2(0xE420E420u), s16 = as_h2(0x2C002C00u), n96 = as_h2(0xD600D600u);
    const __half2 p01 = __hadd2(as_h2(c01), n1056);          // q - 32
    const __half2 p23 = __hfma2(as_h2(c23), s16, n96);        // (1024 + 16q) / 16 - 96 = q - 32
    const __half2 p45 = __hadd2(as_h2(c45), n1056);
    const __half2 p67 = __hfma2(as_h2(c67), s16, n96);
    out[0] = as_u32(__hfma2(p01, dsh, __hmul2(p01, dsl)));
    out[1] = as_u32(__hfma2(p23, dsh, __hmul2(p23, dsl)));
    out[2] = as_u32(__hfma2(p45, dsh, __hmul2(p45, dsl)));
    out[3] = as_u32(__hfma2(p67, dsh, __hmul2(p67, dsl)));
}

__device__ __forceinline__ void dq_unit_q6k(const uint8_t* u, int row, uint32_t tcol) {
    constexpr int kQh = kRows * 128, kSc = kQh + kRows * 64, kD = kSc + kRows * 16;
    const uint4 scv = lds128(u + kSc + row * 16);
    const uint32_t scw[4] = {scv.x, scv.y, scv.z, scv.w};
    const float d = __half2float(*reinterpret_cast<const __half*>(u + kD + row * 2));
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 ql = lds128(u + (c * kRows + row) * 16);
        const uint2 qh = lds64(u + kQh + (c * kRows + row) * 8);
        __half2 dsh[2], dsl[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {  // sub-blocks 2c and 2c + 1 (16 weights each)
            const int sb = 2 * c + t;
            const float dsc = d * static_cast<float>(static_cast<int8_t>(scw[sb >> 2] >> (8 * (sb & 3))));
            const __half hh = __float2half_rn(dsc);
            dsh[t] = __half2half2(hh);
            dsl[t] = __half2half2(__float2half_rn(dsc - __half2float(hh)));
        }
        uint32_t out[16];
        q6_word(ql.x, prmt(qh.x, 0u, 0x4140u) << 4, dsh[0], dsl[0], out + 0);
        q6_word(ql.y, prmt(qh.x, 0u, 0x4342u) << 4, dsh[0], dsl[0], out + 4);
        q6_word(ql.z, prmt(qh.y, 0u, 0x4140u) << 4, dsh[1], dsl[1], out + 8);
        q6_word(ql.w, prmt(qh.y, 0u, 0x4342u) << 4, dsh[1], dsl[1], out + 12);
        tmem_st16(tcol + 16 * c, out);
    }
}

// Shared-memory descriptor of a -B_l step operand ([rows][16 k] fp16): K-major, no swizzle,
// core matrices of 8 rows x 16 bytes, the two k halves `kstride` bytes apart and 8-row groups
// `gstride` bytes apart.  The A tile is [group][k half][8 rows][16 B] (128, 256); the B tile
// of MP tokens is [k half][token][16 B] (MP * 16, 128): the eight sub-block sums of a token
// are one 16-byte row, written by the dequantisation warps.
__device__ __forceinline__ uint64_t smem_desc_k16(uint32_t saddr, uint32_t kstride, uint32_t gstride) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(kstride >> 4) << 16) |
           (static_cast<uint64_t>(gstride >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
}

template <int MP, int F, bool D>
__global__ void __launch_bounds__(kThreads, 1)
    tc_kernel(const __grid_constant__ MatDesc single, const LaunchParams p) {
    using C = Cfg<MP, F, D>;
    constexpr int kUnitBytes = C::kUnitBytes;
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
    uint64_t* mmadone = accempty + 2;   // [2]: every MMA of issuer e has finished
    // [kTB], kSplit only: sub-blocks 0-3 of the unit's A buffer are written (the other widths
    // keep the shared-memory layout without them)
    uint64_t* tfull_lo = mmadone + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull_lo + (C::kSplit ? kTB : 0));
    unsigned long long* amax_sm = reinterpret_cast<unsigned long long*>(smem + C::kAmaxOff);
    float* stage_sm = reinterpret_cast<float*>(smem + C::kAmaxOff);  // y launches only
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t c = blockIdx.x;
    const int count = p.count;
    const int64_t U = p.units;
    const int64_t P = gridDim.x;
    const int64_t g0 = dev_piece_start(c, U, P), g1 = dev_piece_start(c + 1, U, P);
    const uint64_t lim = p.wait_ns;
    const bool dep = p.done != nullptr;  // a dependent step: each matrix cut into its own pieces
    auto mat = [&](int i) -> const MatDesc& { return count == 1 ? single : p.mats[i]; };
    // where this CTA's piece of a matrix starts (in the units the split-K bookkeeping counts:
    // the matrix's own in a dependent step, the launch's concatenated sequence otherwise), and
    // how many units and pieces that sequence has
    auto piece_lo = [&](const MatDesc& M) -> int64_t {
        return dep ? (c < M.pieces ? c * M.units / M.pieces : M.units) : g0;
    };
    auto seq_units = [&](const MatDesc& M) -> int64_t { return dep ? M.units : U; };
    auto seq_pieces = [&](const MatDesc& M) -> int64_t { return dep ? M.pieces : P; };
    auto enter = [&](Cursor& k, int i) {
        for (; i < count; ++i) {
            const MatDesc& M = mat(i);
            int64_t lo, hi;
            if (dep) {
                lo = piece_lo(M);
                hi = c < M.pieces ? (c + 1) * M.units / M.pieces : M.units;
            } else {
                if (M.base >= g1) break;
                lo = g0 > M.base ? g0 - M.base : 0;
                hi = g1 - M.base < M.units ? g1 - M.base : M.units;
            }
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
    auto first = [&](Cursor& k) { enter(k, (count == 1 || dep) ? 0 : p.first_mat[c]); };
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
            if (C::kSplit) mbar_init(&tfull_lo[i], 4);
            mbar_init(&tempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accfull[i], 2);
            mbar_init(&accempty[i], 4);
            mbar_init(&mmadone[i], 1);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    if constexpr (C::kMin) {
        // the upper (always zero) k half of every -B_l step's B tile
        for (int i = tid; i < kXRing * MP * 4; i += kThreads) {
            const int slot = i / (MP * 4), r = (i / 4) % MP, e = i % 4;
            *reinterpret_cast<uint32_t*>(xsum + slot * C::kXsBytes + MP * 16 + r * 16 + e * 4) = 0u;
        }
        // ... and of the A tiles of the -B_l step
        for (int i = tid; i < C::kNA * kRows * 4; i += kThreads) {
            const int slot = i / (kRows * 4), r = (i / 4) % kRows, e = i % 4;
            *reinterpret_cast<uint32_t*>(blt + slot * kBlBytes + (r >> 3) * 256 + 128 + (r & 7) * 16 + e * 4) = 0u;
        }
    }
    fence_proxy_async_smem();
    __syncthreads();
    griddep_launch_dependents();
    // Registers moved to the dequantisation warpgroups (warps 0-7) from the other two
    // (producer, activations, issuers, epilogue), where measured faster: Q6_K 176 / 80 (+8 %),
    // Q4_K at MP >= 64 152 / 104 (+2-4 %; at MP <= 32 it lost 2 %, and 176 / 80 lost 7 %).
    // 2 x 128 x 176 + 2 x 128 x 80 = 2 x 128 x 152 + 2 x 128 x 104 = 65,536 = the launch's
    // 512 threads x 128 (checked on the host).  Every warp runs its instruction here, before
    // any role can return.
    static_assert(kDqWarps == 8 && kThreads == 512, "register split by warpgroup");
    if constexpr (C::kRegSplit == 176) {
        if (warp < kDqWarps) setmaxnreg_inc<176>();
        else setmaxnreg_dec<80>();
    } else if constexpr (C::kRegSplit == 152) {
        if (warp < kDqWarps) setmaxnreg_inc<152>();
        else setmaxnreg_dec<104>();
    }

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
                if (wseq >= kWRing && !mbar_wait_bounded(&wempty[s], ((wseq / kWRing) - 1) & 1, flags, lim)) {
                    ok = false;
                    break;
                }
                // the dequantisation warps' generic reads of the slot, before this bulk write
                if (wseq >= kWRing) fence_proxy_async_smem();
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
                    mbar_wait_bounded(&wfull[j % kWRing], (j / kWRing) & 1, &no_abort, kDrainLimitNs);
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
            const void* smap = nullptr;
            bool ok = true;
            griddep_wait();  // activations may be written by the previous kernel
            while (xc.i < count) {
                const int xs = static_cast<int>(issued % kXRing);
                if (issued >= kXRing && !mbar_wait_bounded(&xempty[xs], ((issued / kXRing) - 1) & 1, flags, lim)) {
                    ok = false;
                    break;
                }
                // the dequantisation warps' generic reads of the slot (the activation sums at
                // MP <= 64), before this bulk write
                if (issued >= kXRing) fence_proxy_async_smem();
                if (xc.i != cur) {
                    const MatDesc& M = mat(xc.i);
                    cur = xc.i;
                    xmap = &M.xmap;
                    smap = &M.smap;
                    kbn = M.kb;
                    kb = static_cast<int>(xc.j % kbn);
                    if (dep && xc.i > 0) {
                        // a dependent step: matrix i's activations may be matrix i - 1's output;
                        // load them only once every CTA has written its part of it, and order
                        // those (generic-proxy) writes before this thread's bulk tensor loads
                        if (!wait_count(p.done + (xc.i - 1), static_cast<int>(gridDim.x), flags, lim)) {
                            ok = false;
                            break;
                        }
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                    }
                }
                mbar_arrive_expect_tx(&xfull[xs], C::kXSlot + (C::kPre ? MP * 16 : 0));
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    tma_load_2d(xring + xs * C::kXSlot + b * C::kXBox, xmap, kb * 256 + 64 * b, 0, &xfull[xs]);
                // the unit's activation sums, tokens 0 .. MP-1 of column kb (zero past m)
                if constexpr (C::kPre) tma_load_3d(xsum + xs * C::kXsBytes, smap, 0, 0, kb, &xfull[xs]);
                kb = (kb + 1 == kbn) ? 0 : kb + 1;
                ++issued;
                next(xc);
            }
            if (!ok) fail(p.err, flags);
            if (flags[0]) {
                volatile int no_abort = 0;
                for (int64_t j = issued > kXRing ? issued - kXRing : 0; j < issued; ++j)
                    mbar_wait_bounded(&xfull[j % kXRing], (j / kXRing) & 1, &no_abort, kDrainLimitNs);
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
                if (seg >= C::kAccBufs && !warp_wait(&accempty[b], ((seg / C::kAccBufs) - 1) & 1, flags, lim)) {
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
                    const uint32_t xaddr = smem_u32(xring + xs * C::kXSlot);
                    // the start-address field is bits 0-13 (address / 16); shared-memory
                    // addresses stay below 256 KB, so the constant offsets never carry out of it
                    const uint64_t bdesc0 = smem_desc_sw128(xaddr);
                    const uint32_t abase = tbase + a * kACols;
                    if constexpr (C::kSplit) {
                        // sub-blocks 0-3 (k-steps 0-7) as soon as they are written; the x tile
                        // is in, since the group waited for it before forming the sums
                        if (!warp_wait(&tfull_lo[tb], (j / kTB) & 1, flags, lim)) {
                            live = false;
                            break;
                        }
                        tc_fence_after();
                        if (lane == 0) {
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(((kk >> 2) * C::kXBox + (kk & 3) * 32) >> 4);
                                tc_mma_f16_ts(d_tmem, abase + 8 * kk, bdesc, kIdesc, (!fresh || kk > 0) ? 1u : 0u);
                            }
                        }
                        __syncwarp();
                    }
                    if (!warp_wait(&tfull[tb], (j / kTB) & 1, flags, lim)) {
                        live = false;
                        break;
                    }
                    if (C::kIssuerWaitsX && !warp_wait(&xfull[xs], (j / kXRing) & 1, flags, lim)) {
                        live = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
#pragma unroll
                        for (int kk = C::kSplit ? 8 : 0; kk < 16; ++kk) {
                            const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(((kk >> 2) * C::kXBox + (kk & 3) * 32) >> 4);
                            tc_mma_f16_ts(d_tmem, abase + 8 * kk, bdesc, kIdesc, (!fresh || kk > 0) ? 1u : 0u);
                        }
                        if constexpr (C::kMin)
                            tc_mma_f16_ss(d_tmem, smem_desc_k16(smem_u32(blt + a * kBlBytes), 128, 256),
                                          smem_desc_k16(smem_u32(xsum + xs * C::kXsBytes), MP * 16, 128), kIdesc, 1u);
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
            mbar_wait_bounded(&mmadone[e], 0, &no_abort, kDrainLimitNs);
        }
        __syncwarp();
        tc_fence_before();
        named_bar_sync(kBarTeardown, kTmemUsers);
        tc_fence_after();
        if (e == 0) tmem_dealloc(tbase, kTmemCols);
        return;
    }

    // ------------------------------------------------------------------ epilogue
    // Every decision that ends or skips work is taken by the four warps together (a vote on
    // named barrier kBarEpi), so that they always meet at the same barriers.
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
        // argmax launches: this warp's best key of token m in lane m % 32 (best[m / 32]
        // m >= 32), over the final values of the rows it owns
        const bool amax = p.amax_keys != nullptr;
        unsigned long long best[(MP + 31) / 32];
#pragma unroll
        for (int i = 0; i < (MP + 31) / 32; ++i) best[i] = 0ull;
        // dependent steps: count this CTA done with matrices arrived .. upto - 1 (its outputs of
        // them are written, or it had none), one release add each after every warp's stores
        int arrived = 0;
        auto arrive_upto = [&](int upto) {
            if (!dep || arrived >= upto) return;
            named_bar_sync(kBarEpi, kEpiThreads);  // every warp's outputs are written
            if (warp == kEpiWarp0 && lane == 0) {
                // ... including the bulk tensor stores, which go through the async proxy
                bulk_wait_all();
                asm volatile("fence.proxy.async.global;" ::: "memory");
                for (int t = arrived; t < upto; ++t) red_add_release_gpu(p.done + t, 1);
            }
            arrived = upto;
        };
        Cursor mk;
        first(mk);
        while (live && mk.i < count) {
            arrive_upto(mk.i);
            const MatDesc& M = mat(mk.i);
            const int64_t KB = M.kb;
            const int64_t u0 = mk.j, u1 = mk.e;
            for (int64_t tile = u0 / KB; tile <= (u1 - 1) / KB; ++tile, ++seg) {
                const int64_t ja = tile * KB > u0 ? tile * KB : u0;
                const int64_t jb = (tile + 1) * KB < u1 ? (tile + 1) * KB : u1;
                const int b = static_cast<int>(seg % C::kAccBufs);
                // which issuers hold units of this tile (issuer e takes local indices = e mod 2)
                const bool has0 = jb - ja >= 2 || (jl & 1) == 0;
                const bool has1 = jb - ja >= 2 || (jl & 1) == 1;
                jl += jb - ja;
                const bool got = warp_wait(&accfull[b], (seg / C::kAccBufs) & 1, flags, lim);
                if (!bar_and(kBarEpi, kEpiThreads, got)) {
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
                // the accumulators of buffer b are read: the issuers may overwrite them
                auto release = [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&accempty[b]);
                };
                const int64_t n = tile * kRows + row;
                const int64_t tstart = M.base + tile * KB;  // the tile's first unit in the launch
                // final values of columns c0 .. c0 + 15: y, or the argmax fold
                auto emit = [&](int c0, const float (&acc)[16]) {
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
                            const int firstl = __ffs(__ballot_sync(0xffffffffu, o == mx)) - 1;
                            if ((m & 31) == lane && mx != 0u) {
                                const uint32_t nf = static_cast<uint32_t>(n - lane + firstl);
                                const unsigned long long key =
                                    (static_cast<unsigned long long>(mx) << 32) | (0xFFFFFFFFu - nf);
#pragma unroll
                                for (int bi = 0; bi < (MP + 31) / 32; ++bi)
                                    if (bi == (m >> 5)) best[bi] = key > best[bi] ? key : best[bi];
                            }
                        }
                    } else if (C::kStage && M.ytma) {
                        // the chunk goes through the staging tile [token 16][row 128] to one
                        // bulk tensor store (the tensor map clips rows past N and tokens past M)
#pragma unroll
                        for (int i = 0; i < 16; ++i) stage_sm[i * kRows + row] = acc[i];
                        fence_proxy_async_smem();  // the tile's generic writes, before the bulk read
                        named_bar_sync(kBarEpi, kEpiThreads);
                        if (warp == kEpiWarp0 && lane == 0) {
                            tma_store_2d(&M.ymap, stage_sm, static_cast<int32_t>(tile * kRows), c0);
                            bulk_commit_group();
                            bulk_wait_read_all();  // the tile may be written again
                        }
                        named_bar_sync(kBarEpi, kEpiThreads);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int m = c0 + i;
                            if (m < p.m && n < M.n) M.y[static_cast<int64_t>(m) * M.n + n] = acc[i];
                        }
                    }
                };
                const int64_t SU = seq_units(M), SP = seq_pieces(M);
                if (ja == tile * KB && jb == (tile + 1) * KB) {
                    // the whole tile is in this CTA's piece
#pragma unroll 1
                    for (int c0 = 0; c0 < MP; c0 += 16) {
                        float acc[16];
                        load_acc(c0, acc);
                        emit(c0, acc);
                    }
                    release();
                    continue;
                }
                // A tile split between pieces pa..pb: pa, the piece holding its first units,
                // reaches it last (at the end of its piece) and normally finds the partials of
                // pa+1..pb published on the tile's ticket; it then adds them to its own in piece
                // order.  Nobody waits for another CTA: a piece that finds the tile incomplete
                // parks its partial too, and whichever piece arrives last (the ticket's
                // acquire-release add returns pb - pa) sums the parked partials in the same
                // order.  Each CTA has two slots: its first tile (shared with earlier pieces)
                // and its last tile (reduced or parked).
                const int64_t pa = dev_piece_of(tstart, SU, SP);
                const int64_t pb = dev_piece_of(tstart + KB - 1, SU, SP);
                const int need = static_cast<int>(pb - pa);
                auto slot = [&](int64_t piece, int role) {
                    return reinterpret_cast<float4*>(p.ws + (2 * piece + role) * static_cast<int64_t>(kRows) * p.ws_cols);
                };
                // the partials of pa+1..pb added, in piece order, to acc (columns c0 .. c0 + 15)
                auto add_partials = [&](int c0, float (&acc)[16]) {
#pragma unroll 1
                    for (int64_t pc = pa + 1; pc <= pb; ++pc) {
                        const float4* src = slot(pc, 0);
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
                };
                bool direct = false;
                if (pa == c) {
                    // a short bounded poll (the other pieces normally published long ago; a
                    // piece that is not running yet must not be waited for); the vote is also
                    // the barrier that orders every warp's loads after the acquire
                    bool all = false;
                    if (warp == kEpiWarp0 && lane == 0 && !p.park_all) {
                        const uint64_t t0 = globaltimer_ns();
                        for (;;) {
                            if (ld_acquire_gpu(M.tickets + tile) == need) {
                                all = true;
                                break;
                            }
                            if (globaltimer_ns() - t0 > kParkAfterNs) break;
                            __nanosleep(64);
                        }
                    }
                    direct = bar_or(kBarEpi, kEpiThreads, all);
                }
                if (direct && (C::kRegSplit == 176 || MP == 64)) {
                    // no prefetch where the epilogue warps run at 80 registers (Q6_K), nor at
                    // MP = 64, where it measured 3 % slower on a 16-layer step (and 2-4 %
                    // faster at MP = 16 and 128)
#pragma unroll 1
                    for (int c0 = 0; c0 < MP; c0 += 16) {
                        float acc[16];
                        load_acc(c0, acc);
                        add_partials(c0, acc);
                        emit(c0, acc);
                    }
                } else if (direct) {
                    auto ld4 = [&](int c0, int64_t pc, float4 (&v)[4]) {
                        const float4* src = slot(pc, 0);
#pragma unroll
                        for (int f = 0; f < 4; ++f) v[f] = __ldcg(src + (c0 / 4 + f) * kEpiThreads + etid);
                    };
                    // piece pa+1's partial of the next chunk is loaded while this one is summed
                    // and written; the sum keeps the order acc + P(pa+1) + P(pa+2) + ...
                    float4 nxt[4];
                    ld4(0, pa + 1, nxt);
#pragma unroll 1
                    for (int c0 = 0; c0 < MP; c0 += 16) {
                        float acc[16];
                        load_acc(c0, acc);
                        float4 cur[4];
#pragma unroll
                        for (int f = 0; f < 4; ++f) cur[f] = nxt[f];
                        if (c0 + 16 < MP) ld4(c0 + 16, pa + 1, nxt);
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            acc[4 * f] += cur[f].x;
                            acc[4 * f + 1] += cur[f].y;
                            acc[4 * f + 2] += cur[f].z;
                            acc[4 * f + 3] += cur[f].w;
                        }
#pragma unroll 1
                        for (int64_t pc = pa + 2; pc <= pb; ++pc) {
                            float4 v[4];
                            ld4(c0, pc, v);
#pragma unroll
                            for (int f = 0; f < 4; ++f) {
                                acc[4 * f] += v[f].x;
                                acc[4 * f + 1] += v[f].y;
                                acc[4 * f + 2] += v[f].z;
                                acc[4 * f + 3] += v[f].w;
                            }
                        }
                        emit(c0, acc);
                    }
                }
                if (direct) {
                    release();
                    // every partial is read: the ticket is ready for the next launch
                    named_bar_sync(kBarEpi, kEpiThreads);
                    if (warp == kEpiWarp0 && lane == 0) M.tickets[tile] = 0;
                    continue;
                }
                float4* own = slot(c, pa == c ? 1 : 0);
#pragma unroll 1
                for (int c0 = 0; c0 < MP; c0 += 16) {
                    float acc[16];
                    load_acc(c0, acc);
#pragma unroll
                    for (int f = 0; f < 4; ++f)
                        own[(c0 / 4 + f) * kEpiThreads + etid] =
                            make_float4(acc[4 * f], acc[4 * f + 1], acc[4 * f + 2], acc[4 * f + 3]);
                }
                release();
                // every warp's partial is written (the barrier); one acquire-release add
                // publishes it and tells whether this CTA is the last to arrive
                named_bar_sync(kBarEpi, kEpiThreads);
                bool last = false;
                if (warp == kEpiWarp0 && lane == 0) last = atom_add_acq_rel_gpu(M.tickets + tile, 1) == need;
                if (!bar_or(kBarEpi, kEpiThreads, last)) continue;
                const float4* first_part = slot(pa, 1);
#pragma unroll 1
                for (int c0 = 0; c0 < MP; c0 += 16) {
                    float acc[16];
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        const float4 v = __ldcg(first_part + (c0 / 4 + f) * kEpiThreads + etid);
                        acc[4 * f] = v.x;
                        acc[4 * f + 1] = v.y;
                        acc[4 * f + 2] = v.z;
                        acc[4 * f + 3] = v.w;
                    }
                    add_partials(c0, acc);
                    emit(c0, acc);
                }
                named_bar_sync(kBarEpi, kEpiThreads);
                if (warp == kEpiWarp0 && lane == 0) M.tickets[tile] = 0;
            }
            enter(mk, mk.i + 1);
        }
        if (amax && live) {
            // the CTA's best key per token (over the four warps) goes out as one atomic
#pragma unroll
            for (int bi = 0; bi < (MP + 31) / 32; ++bi)
                if (32 * bi + lane < MP) amax_sm[q * MP + 32 * bi + lane] = best[bi];
            named_bar_sync(kBarEpi, kEpiThreads);
            if (warp == kEpiWarp0) {
                for (int m = lane; m < p.m; m += 32) {
                    unsigned long long k = amax_sm[m];
#pragma unroll
                    for (int w = 1; w < 4; ++w) k = amax_sm[w * MP + m] > k ? amax_sm[w * MP + m] : k;
                    atomicMax(p.amax_keys + m, k);
                }
                amax_finish_warp(p, static_cast<int>(gridDim.x), lane);
            }
        }
        if (dep && live) {
            arrive_upto(count);
            // the last CTA to finish zeroes the counters for the next launch (every CTA has
            // passed its last wait on them by then)
            if (warp == kEpiWarp0 && lane == 0 &&
                atom_add_acq_rel_gpu(p.done + count, 1) == static_cast<int>(gridDim.x) - 1)
                for (int t = 0; t <= count; ++t) p.done[t] = 0;
        }
        if (!live && lane == 0) fail(p.err, flags);
        if (warp == kEpiWarp0 && lane == 0) bulk_wait_all();  // y's bulk stores have completed
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
        const int64_t nunits = dep ? p.cta_units[c] : g1 - g0;
        int64_t j = g;
        for (; j < nunits; j += kGroups) {
            const int s = static_cast<int>(j % kWRing);
            const int a = static_cast<int>(j % C::kNA);
            if (!warp_wait(&wfull[s], (j / kWRing) & 1, flags, lim)) break;
            const uint8_t* u = wring + s * kUnitBytes;
            if constexpr (F == QMM_FORMAT_Q4_K) {
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
                // the slot was refilled.  At MP = 128 they come from the pre-pass with the x tile
                // (the same fp16 additions in the same order, so a row's bits do not depend on
                // MP), and the group does not wait for the tile at all.
                const int xs = static_cast<int>(j % kXRing);
                if (!C::kIssuerWaitsX && !warp_wait(&xfull[xs], (j / kXRing) & 1, flags, lim)) break;
                const uint8_t* xt = xring + xs * C::kXSlot;
                uint8_t* xst = xsum + xs * C::kXsBytes;
    #pragma unroll
                for (int pi = row; pi < (C::kPre ? 0 : MP * 8); pi += kRows) {
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
                    *reinterpret_cast<__half*>(xst + t * 16 + sb * 2) = sum;
                }

                // the A buffer was last read by the MMAs of unit j - kNA
                if (j >= C::kNA && !warp_wait(&tempty[(j - C::kNA) % kTB], ((j - C::kNA) / kTB) & 1, flags, lim)) break;
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
                    if (C::kSplit && sb == 3) {
                        tc_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tfull_lo[j % kTB]);
                    }
                }
                // the -B_l step's A row: k slots 0..7 = sub-blocks 0..7 (slots 8..15 stay zero)
                *reinterpret_cast<uint4*>(blt + a * kBlBytes + (row >> 3) * 256 + (row & 7) * 16) =
                    make_uint4(ps[0].nbl, ps[1].nbl, ps[2].nbl, ps[3].nbl);
            } else {
                // no sums to form: the wait on the activation tile keeps the MMAs of this unit
                // after its arrival, as the Q4_K path's sums do (at MP = 128 the issuers wait)
                const int xs = static_cast<int>(j % kXRing);
                if (!C::kIssuerWaitsX && !warp_wait(&xfull[xs], (j / kXRing) & 1, flags, lim)) break;
                if (j >= C::kNA && !warp_wait(&tempty[(j - C::kNA) % kTB], ((j - C::kNA) / kTB) & 1, flags, lim)) break;
                tc_fence_after();
                const uint32_t tcol = tlane + a * kACols;
                if constexpr (F == QMM_FORMAT_Q8_0)
                    dq_unit_q80(u, row, tcol);
                else
                    dq_unit_q6k(u, row, tcol);
                __syncwarp();
                if (lane == 0) mbar_arrive(&wempty[s]);
            }
            fence_proxy_async_smem();  // the sums and the -B_l row are read by the tensor core
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tfull[j % kTB]);
        }
        tc_wait_st();
        // a wait gave up (its own limit, or another warp's failure): report it
        if (j < nunits && lane == 0) fail(p.err, flags);
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

// Q8_0: one thread per 16-byte piece of a unit (34,816 B): pieces 0..2047 are the quant
// halves [block 8][row 128][2 x 16 B], pieces 2048..2175 the d's of a row's 8 blocks.
// Source row n holds K/32 blocks of 34 bytes; rows past N are zero.
__global__ void repack_q80_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t n,
                                  int32_t kb, int64_t units) {
    constexpr int kUnit = unit_bytes(QMM_FORMAT_Q8_0), kSegs = kUnit / 16;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= units * kSegs) return;
    const int64_t u = idx / kSegs;
    const int seg = static_cast<int>(idx % kSegs);
    const int64_t tile = u / kb;
    const int b = static_cast<int>(u % kb);  // super-block column: Q8_0 blocks 8b .. 8b + 7
    uint8_t out[16] = {};
    if (seg < 2048) {
        const int blk = seg >> 8, row = (seg >> 1) & 127, half = seg & 1;
        const int64_t nrow = tile * kRows + row;
        if (nrow < n) {
            const uint8_t* q = src + (nrow * kb * 8 + 8 * b + blk) * 34 + 2 + 16 * half;
            for (int i = 0; i < 16; ++i) out[i] = q[i];
        }
    } else {
        const int row = seg - 2048;
        const int64_t nrow = tile * kRows + row;
        if (nrow < n)
            for (int blk = 0; blk < 8; ++blk) {
                const uint8_t* q = src + (nrow * kb * 8 + 8 * b + blk) * 34;
                out[2 * blk] = q[0];
                out[2 * blk + 1] = q[1];
            }
    }
    uint4 v;
    memcpy(&v, out, 16);
    *reinterpret_cast<uint4*>(dst + u * kUnit + static_cast<int64_t>(seg) * 16) = v;
}

// Q6_K: one thread per 16-byte piece of a unit (26,880 B): pieces 0..1023 the low nibbles
// [chunk 8][row 128][16 B], 1024..1535 the high bit fields [chunk 8][row 128][8 B] (two rows
// per piece), 1536..1663 the scales [row 128][16 B], 1664..1679 the d's [row 128][2 B] (eight
// rows per piece).  Rows past N are zero.
__global__ void repack_q6k_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t n,
                                  int32_t kb, int64_t units) {
    constexpr int kUnit = unit_bytes(QMM_FORMAT_Q6_K), kSegs = kUnit / 16;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= units * kSegs) return;
    const int64_t u = idx / kSegs;
    const int seg = static_cast<int>(idx % kSegs);
    const int64_t tile = u / kb;
    const int b = static_cast<int>(u % kb);
    // the 6-bit quant of weight i of a source block (GGUF Q6_K order)
    auto quant = [](const uint8_t* blk, int i) -> int {
        const int h = i / 128, c = (i % 128) / 32, l = i % 32;
        const int lo = (blk[64 * h + l + 32 * (c & 1)] >> (4 * (c >> 1))) & 15;
        const int hi = (blk[128 + 32 * h + l] >> (2 * c)) & 3;
        return lo | (hi << 4);
    };
    auto block_of = [&](int row) -> const uint8_t* {
        const int64_t nrow = tile * kRows + row;
        return nrow < n ? src + (nrow * kb + b) * 210 : nullptr;
    };
    uint8_t out[16] = {};
    if (seg < 1024) {  // low nibbles of chunk c, row: 4 words, nibble e of word i at pos[e]
        const int c = seg >> 7, row = seg & 127;
        const uint8_t* blk = block_of(row);
        const int pos[8] = {0, 16, 4, 20, 8, 24, 12, 28};
        if (blk)
            for (int i = 0; i < 4; ++i) {
                uint32_t w = 0;
                for (int e = 0; e < 8; ++e) w |= static_cast<uint32_t>(quant(blk, 32 * c + 8 * i + e) & 15) << pos[e];
                memcpy(out + 4 * i, &w, 4);
            }
    } else if (seg < 1536) {  // high bit fields of chunk c, rows 2r and 2r + 1
        const int c = (seg - 1024) >> 6, r2 = ((seg - 1024) & 63) * 2;
        const int fpos[8] = {0, 8, 4, 12, 2, 10, 6, 14};
        for (int t = 0; t < 2; ++t) {
            const uint8_t* blk = block_of(r2 + t);
            if (!blk) continue;
            for (int i = 0; i < 4; ++i) {
                uint32_t f = 0;
                for (int e = 0; e < 8; ++e) f |= static_cast<uint32_t>(quant(blk, 32 * c + 8 * i + e) >> 4) << fpos[e];
                out[8 * t + 2 * i] = static_cast<uint8_t>(f);
                out[8 * t + 2 * i + 1] = static_cast<uint8_t>(f >> 8);
            }
        }
    } else if (seg < 1664) {  // scales of a row
        const uint8_t* blk = block_of(seg - 1536);
        if (blk)
            for (int i = 0; i < 16; ++i) out[i] = blk[192 + i];
    } else {  // d of rows 8p .. 8p + 7
        const int r0 = (seg - 1664) * 8;
        for (int t = 0; t < 8; ++t) {
            const uint8_t* blk = block_of(r0 + t);
            if (blk) {
                out[2 * t] = blk[208];
                out[2 * t + 1] = blk[209];
            }
        }
    }
    uint4 v;
    memcpy(&v, out, 16);
    *reinterpret_cast<uint4*>(dst + u * kUnit + static_cast<int64_t>(seg) * 16) = v;
}

cudaError_t repack(const uint8_t* src_dev, uint8_t* dst_dev, const Decomp& d, int format, cudaStream_t s) {
    const int64_t total = d.units * (unit_bytes(format) / 16);
    const int threads = 256;
    const unsigned blocks = static_cast<unsigned>((total + threads - 1) / threads);
    const int32_t kb = static_cast<int32_t>(d.kb);
    if (format == QMM_FORMAT_Q8_0)
        repack_q80_kernel<<<blocks, threads, 0, s>>>(src_dev, dst_dev, d.n, kb, d.units);
    else if (format == QMM_FORMAT_Q6_K)
        repack_q6k_kernel<<<blocks, threads, 0, s>>>(src_dev, dst_dev, d.n, kb, d.units);
    else
        repack_kernel<<<blocks, threads, 0, s>>>(src_dev, dst_dev, d.n, kb, d.units);
    return cudaGetLastError();
}

template <int MP, int F, bool D = false>
static cudaError_t set_attr() {
    cudaError_t e = cudaFuncSetAttribute(tc_kernel<MP, F, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<MP, F, D>::kSmem);
    if (e != cudaSuccess || Cfg<MP, F, D>::kRegSplit == 0) return e;
    // a register split (setmaxnreg) is sized for launches of exactly 128 registers per thread:
    // anything else and an increase could wait forever, so the library refuses to run
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, tc_kernel<MP, F, D>)) != cudaSuccess) return e;
    return fa.numRegs == 128 ? cudaSuccess : cudaErrorInvalidKernelImage;
}

template <int F>
static cudaError_t set_attr_all() {
    cudaError_t e;
    if ((e = set_attr<16, F>()) != cudaSuccess) return e;
    if ((e = set_attr<32, F>()) != cudaSuccess) return e;
    if ((e = set_attr<64, F>()) != cudaSuccess) return e;
    if constexpr (F == QMM_FORMAT_Q4_K) {
        if ((e = set_attr<16, F, true>()) != cudaSuccess) return e;
        if ((e = set_attr<32, F, true>()) != cudaSuccess) return e;
    }
    return set_attr<128, F>();
}

cudaError_t configure() {
    cudaError_t e;
    if ((e = set_attr_all<QMM_FORMAT_Q4_K>()) != cudaSuccess) return e;
    if ((e = set_attr_all<QMM_FORMAT_Q6_K>()) != cudaSuccess) return e;
    return set_attr_all<QMM_FORMAT_Q8_0>();
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

int mp_for(int64_t m) { return m <= 16 ? 16 : m <= 32 ? 32 : m <= 64 ? 64 : 128; }

cudaError_t make_mat(MatDesc* out, const uint8_t* wq, const void* x, float* y, int* tickets, int64_t units,
                     int64_t n, int32_t kb, int32_t m, __half* xs) {
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
    out->xsrc = static_cast<const __half*>(x);
    out->xs = xs;
    out->frag = nullptr;
    if (xs) {
        // the activation sums [kb][m][8 sub-blocks] fp16: box 8 x MP x 1, rows past m read as zero
        const cuuint64_t sdim[3] = {8, static_cast<cuuint64_t>(m), static_cast<cuuint64_t>(kb)};
        const cuuint64_t sstride[2] = {16, static_cast<cuuint64_t>(m) * 16};
        const cuuint32_t sbox[3] = {8, static_cast<cuuint32_t>(mp_for(m)), 1};
        const cuuint32_t sestr[3] = {1, 1, 1};
        if (enc(&out->smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, xs, sdim, sstride, sbox, sestr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        memset(&out->smap, 0, sizeof(out->smap));
    }
    // y [m, n] fp32 for the epilogue's bulk stores: 16 tokens x 128 rows per store (rows
    // past n and tokens past m are not written); the row stride must be a multiple of 16
    // bytes
    memset(&out->ymap, 0, sizeof(out->ymap));
    out->ytma = 0;
    if (y && (n & 3) == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0) {
        const cuuint64_t ydim[2] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(m)};
        const cuuint64_t ystride[1] = {static_cast<cuuint64_t>(n) * 4};
        const cuuint32_t ybox[2] = {static_cast<cuuint32_t>(kRows), 16};
        const cuuint32_t yestr[2] = {1, 1};
        if (enc(&out->ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, y, ydim, ystride, ybox, yestr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        out->ytma = 1;
    }
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

// One thread per (super-block column kb, token t) of a matrix (blockIdx.y): the eight sums of
// 32 activations of x[t][256 kb ..], with exactly the fp16 additions, in the same order, that
// the kernel's dequantisation warps make from the x tile at MP <= 64.
__global__ void __launch_bounds__(256) presum_kernel(const __grid_constant__ MatDesc single, const LaunchParams p) {
    const MatDesc& M = p.count == 1 ? single : p.mats[blockIdx.y];
    const int m = p.m;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<int64_t>(M.kb) * m) return;
    const int kb = static_cast<int>(idx / m), t = static_cast<int>(idx % m);
    const uint4* src = reinterpret_cast<const uint4*>(M.xsrc + (static_cast<int64_t>(t) * M.kb + kb) * 256);
    __half sums[8];
#pragma unroll
    for (int sb = 0; sb < 8; ++sb) {
        __half2 acc2 = __float2half2_rn(0.f);
#pragma unroll
        for (int cc4 = 0; cc4 < 4; ++cc4) {
            const uint4 v = src[sb * 4 + cc4];  // activations 32 sb + 8 cc4 .. + 7
            acc2 = __hadd2(acc2, __hadd2(__hadd2(as_h2(v.x), as_h2(v.y)), __hadd2(as_h2(v.z), as_h2(v.w))));
        }
        const __half sum = __hadd(__low2half(acc2), __high2half(acc2));
        sums[sb] = __hmin(__hmax(sum, __ushort_as_half(0xFBFFu)), __ushort_as_half(0x7BFFu));
    }
    *reinterpret_cast<uint4*>(M.xs + (static_cast<int64_t>(kb) * m + t) * 8) =
        make_uint4(as_u32(__halves2half2(sums[0], sums[1])), as_u32(__halves2half2(sums[2], sums[3])),
                   as_u32(__halves2half2(sums[4], sums[5])), as_u32(__halves2half2(sums[6], sums[7])));
}

cudaError_t presum(const MatDesc& single, const LaunchParams& p, int32_t max_kb, cudaStream_t s) {
    const int64_t n = static_cast<int64_t>(max_kb) * p.m;
    const dim3 grid(static_cast<unsigned>((n + 255) / 256), static_cast<unsigned>(p.count));
    presum_kernel<<<grid, 256, 0, s>>>(single, p);
    return cudaGetLastError();
}

template <int MP, int F, bool D = false>
static cudaError_t launch_mp(const MatDesc& single, const LaunchParams& p, int grid, cudaStream_t s, bool pdl,
                             bool cooperative) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<MP, F, D>::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = cooperative ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, tc_kernel<MP, F, D>, single, p);
}

template <int F>
static cudaError_t launch_f(const MatDesc& single, const LaunchParams& p, int grid, cudaStream_t s, bool pdl,
                            bool cooperative) {
    if constexpr (F == QMM_FORMAT_Q4_K) {
        if (p.done != nullptr && mp_for(p.m) <= 32)  // a dependent persistent step
            return mp_for(p.m) == 16 ? launch_mp<16, F, true>(single, p, grid, s, pdl, cooperative)
                                     : launch_mp<32, F, true>(single, p, grid, s, pdl, cooperative);
    }
    switch (mp_for(p.m)) {
        case 16: return launch_mp<16, F>(single, p, grid, s, pdl, cooperative);
        case 32: return launch_mp<32, F>(single, p, grid, s, pdl, cooperative);
        case 64: return launch_mp<64, F>(single, p, grid, s, pdl, cooperative);
        default: return launch_mp<128, F>(single, p, grid, s, pdl, cooperative);
    }
}

cudaError_t launch(const MatDesc& single, const LaunchParams& p, int grid, cudaStream_t s, bool pdl, bool cooperative,
                   int format) {
    switch (format) {
        case QMM_FORMAT_Q6_K: return launch_f<QMM_FORMAT_Q6_K>(single, p, grid, s, pdl, cooperative);
        case QMM_FORMAT_Q8_0: return launch_f<QMM_FORMAT_Q8_0>(single, p, grid, s, pdl, cooperative);
        default: return launch_f<QMM_FORMAT_Q4_K>(single, p, grid, s, pdl, cooperative);
    }
}

}  // namespace b2
}  // namespace qmm
