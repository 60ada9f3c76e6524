// Backend 1: Q4_K weight-streaming matmul on warp-level tensor cores (mma.sync m16n8k16).
//
// The method (page "Running 4 coding agents on one RTX 3090: a custom CUDA engine for
// Qwen3.8-27B", section "How parallel decoding works"): the M stacked token rows of a
// decode step are multiplied against every weight while that weight is on chip, so the
// weights are read from memory once per step however many rows there are.
//
// Layout of one unit (32 output rows x one super-block column of 256 weights, 4608 B),
// written once by repack():
//   bytes [0, 4096)    quants, in the order the consumer lanes read them:
//                      [m16 tile r: 2][load i: 4][lane: 32][16 B]
//                      load i = 2*h + bh gives lane (g = lane/4, t = lane%4) bytes
//                      qs[32t + 16bh .. +15] of row 16r + 8h + g.
//   bytes [4096, 4608) the 16-byte block headers (d, dmin, 12 scale bytes) of the 32 rows.
// Lane t of a quad therefore holds qs[32t .. 32t+31] of its two rows: the low nibbles are
// weights 64t + 0..31 (sub-block 2t) and the high nibbles weights 64t + 32..63 (sub-block
// 2t+1).  Each lane needs the (scale, min) pairs of just those two sub-blocks.
//
// MMA k-order.  For step s = 0..15 (i = s % 8, high = s >= 8) lane t supplies the four
// MMA k slots {2t, 2t+1, 2t+8, 2t+9} with weight offsets 64t + 32*high + 4i + {0, 2, 1, 3}
// inside the super-block; the activation fragment is loaded with the same permutation, so
// the MMA sums exactly the products w[n,k] x[m,k].  The order is fixed per handle.
//
// Work split.  CTA c owns the contiguous units [c*U/P, (c+1)*U/P) (U units, P CTAs).  One
// producer warp streams them into a shared-memory ring with 1-D bulk copies (TMA) and
// mbarriers; four consumer warps take the units of each row tile round-robin, dequantise
// in registers to fp16 fragments and accumulate in fp32 on the tensor cores.  At the end of
// a row tile the four warp partials are summed in warp order through shared memory; a tile
// split between CTAs is finished by the last CTA to arrive (atomic ticket), which sums the
// CTA partials in CTA order.  Nothing in this order depends on M or on the other rows, so
// every row's result is bit-identical however the rows are batched.
#include <cuda_fp16.h>

#include "qmm_internal.h"
#include "qmm_ptx.cuh"

namespace qmm {
namespace b1 {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kRing = 16;
constexpr int kQBytes = kRows * 128;
constexpr int kRedCols = 16;
constexpr int kRedFloats = kConsumerWarps * kRows * kRedCols;
constexpr int kConsumerThreads = kConsumerWarps * 32;
// Unit j - kRing of a row tile belongs to the same warp as unit j, so a warp that waits for
// unit j has already seen the previous fill of that slot complete: the parity it waits on
// is never a stale one.
static_assert(kRing % kConsumerWarps == 0, "ring depth must be a multiple of the consumer warps");

int smem_bytes() {
    return kRing * kUnitBytes + kRedFloats * 4 + 2 * kRing * 8 + 16;
}

__device__ __forceinline__ int64_t dev_piece_of(int64_t u, int64_t units, int64_t grid) {
    return ((u + 1) * grid + units - 1) / units - 1;
}

__device__ __forceinline__ void raise_error(int* err, volatile int* abort_flag, int code) {
    *abort_flag = 1;
    atomicOr(err, code);
}

// Per-row constants for the lane's two sub-blocks j0 = 2t (low nibbles, quant encoded as
// 1024 + q) and j1 = 2t + 1 (high nibbles, encoded as 1024 + 16q).  Lane .x of each fp16x2
// belongs to j0, lane .y to j1.
struct RowScales {
    uint32_t scx;   // {sc0, sc1 / 16}
    uint32_t nscx;  // {-1024 sc0, -64 sc1}: scx * code + nscx = sc * q exactly
    uint32_t d2;    // {d, d}
    uint32_t nbh;   // {-B_h0, -B_h1},  B_h = fp16(dmin * m)
    uint32_t nbl;   // {-B_l0, -B_l1},  B_l = dmin * m - B_h exactly (error-free product)
};

__device__ __forceinline__ RowScales row_scales(uint4 hd, int t) {
    const uint32_t s0 = hd.y, s1 = hd.z, s2 = hd.w;
    uint32_t SC, MN;
    if (t >= 2) {  // sub-blocks 4..7: low 4 bits from s[8..11], top 2 bits from s[0..7]
        SC = (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
        MN = ((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u);
    } else {       // sub-blocks 0..3: low 6 bits of s[0..3] and s[4..7]
        SC = s0 & 0x3F3F3F3Fu;
        MN = s1 & 0x3F3F3F3Fu;
    }
    const uint32_t b0 = 2u * (t & 1);
    // bytes b0, b0+1 -> 16-bit lanes {1024 + v0, 1024 + v1} -> {v0, v1} exactly
    const uint32_t sel = b0 | ((b0 + 1) << 8);
    const __half2 k1024 = as_h2(0x64006400u);
    const __half2 sc = __hsub2(as_h2(and_or(prmt(SC, 0, sel), 0x00FF00FFu, 0x64006400u)), k1024);
    const __half2 mn = __hsub2(as_h2(and_or(prmt(MN, 0, sel), 0x00FF00FFu, 0x64006400u)), k1024);
    RowScales r;
    r.scx = as_u32(__hmul2(sc, as_h2(0x2C003C00u)));    // * {1, 1/16}
    r.nscx = as_u32(__hmul2(sc, as_h2(0xD400E400u)));   // * {-1024, -64}
    const __half2 d = as_h2(prmt(hd.x, 0, 0x1010u));    // {d, d}
    const __half2 dm = as_h2(prmt(hd.x, 0, 0x3232u));   // {dmin, dmin}
    const __half2 bh = __hmul2(dm, mn);
    r.d2 = as_u32(d);
    r.nbh = as_u32(__hneg2(bh));
    r.nbl = as_u32(__hfma2(__hneg2(dm), mn, bh));       // -(dmin*m - B_h), exact
    return r;
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 2) stream_kernel(const B1Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;
    float* red = reinterpret_cast<float*>(smem + kRing * kUnitBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(red + kRedFloats);
    uint64_t* empty = full + kRing;
    volatile int* flags = reinterpret_cast<volatile int*>(empty + kRing);  // [0] abort [1] last

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t c = blockIdx.x;
    const int64_t U = p.units;
    const int64_t u0 = c * U / p.grid;
    const int64_t u1 = (c + 1) * U / p.grid;
    const int nunits = static_cast<int>(u1 - u0);

    if (tid == 0) {
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // Let the next kernel in the stream start its weight prefetch while this one runs.
    griddep_launch_dependents();

    if (warp == kConsumerWarps) {
        // ---------------- producer: weights do not depend on the previous kernel, so the
        // stream starts before griddepcontrol.wait.
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            const uint8_t* src = p.wq + u0 * kUnitBytes;
            int issued = 0;
            for (int j = 0; j < nunits; ++j) {
                const int slot = j % kRing;
                if (j >= kRing && !mbar_wait_bounded(&empty[slot], ((j / kRing) - 1) & 1, flags)) {
                    raise_error(p.err, flags, 1);
                    break;
                }
                mbar_arrive_expect_tx(&full[slot], kUnitBytes);
                bulk_g2s(ring + slot * kUnitBytes, src + static_cast<int64_t>(j) * kUnitBytes,
                         kUnitBytes, &full[slot], pol);
                issued = j + 1;
            }
            if (flags[0]) {
                // Failure path: do not leave bulk copies writing into a CTA that has exited.
                volatile int no_abort = 0;
                for (int j = issued > kRing ? issued - kRing : 0; j < issued; ++j)
                    mbar_wait_bounded(&full[j % kRing], (j / kRing) & 1, &no_abort);
            }
        }
        return;
    }

    // ---------------- consumers
    griddep_wait();  // x may be written by the previous kernel

    const int g = lane >> 2;
    const int t = lane & 3;
    const int KB = p.kb;
    const int64_t K = static_cast<int64_t>(KB) * 256;
    const int64_t t_first = u0 / KB;
    const int64_t t_last = (u1 - 1) / KB;

    // this lane's activation row pointer per 8-token group (nullptr for padding rows)
    const __half* xrow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int m = nt * 8 + g;
        xrow[nt] = (m < p.m) ? p.x + m * K + 64 * t : nullptr;
    }

    for (int64_t tile = t_first; tile <= t_last; ++tile) {
        const int64_t ja = (tile * KB > u0 ? tile * KB : u0) - u0;
        const int64_t jb = ((tile + 1) * KB < u1 ? (tile + 1) * KB : u1) - u0;

        float acc[2][NT][4];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[r][nt][e] = 0.f;

        for (int64_t j = ja + warp; j < jb; j += kConsumerWarps) {
            const int slot = static_cast<int>(j % kRing);
            const uint32_t ph = static_cast<uint32_t>((j / kRing) & 1);
            const int64_t kb = u0 + j - tile * KB;

            // activations for this super-block column: 64 halves per lane per token group
            uint4 xv[NT][8];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (xrow[nt]) {
                    const uint4* src = reinterpret_cast<const uint4*>(xrow[nt] + kb * 256);
#pragma unroll
                    for (int v = 0; v < 8; ++v) xv[nt][v] = src[v];
                } else {
#pragma unroll
                    for (int v = 0; v < 8; ++v) xv[nt][v] = make_uint4(0, 0, 0, 0);
                }
            }
            // warm L1 with this warp's next column
            if (j + kConsumerWarps < jb) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    if (xrow[nt])
                        asm volatile("prefetch.global.L1 [%0];" ::"l"(xrow[nt] + (kb + kConsumerWarps) * 256));
            }

            if (!mbar_wait_bounded(&full[slot], ph, flags)) {
                if (!flags[0]) raise_error(p.err, flags, 1);
                continue;  // keep the control flow (and barrier counts) of the other warps
            }
            const uint8_t* us = ring + slot * kUnitBytes;
            uint4 qv[2][4];
            uint4 hd[2][2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    qv[r][i] = *reinterpret_cast<const uint4*>(us + ((r * 4 + i) * 32 + lane) * 16);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    hd[r][h] = *reinterpret_cast<const uint4*>(us + kQBytes + (16 * r + 8 * h + g) * 16);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);

            RowScales rs[2][2];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int h = 0; h < 2; ++h) rs[r][h] = row_scales(hd[r][h], t);

#pragma unroll
            for (int s = 0; s < 16; ++s) {
                const int i = s & 7;
                const int hi = s >> 3;
                uint32_t b01[NT], b23[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint4 xq = xv[nt][hi * 4 + (i >> 1)];
                    const uint32_t x01 = (i & 1) ? xq.z : xq.x;  // halves 4i, 4i+1
                    const uint32_t x23 = (i & 1) ? xq.w : xq.y;  // halves 4i+2, 4i+3
                    b01[nt] = prmt(x01, x23, 0x5410u);           // {x[4i], x[4i+2]}
                    b23[nt] = prmt(x01, x23, 0x7632u);           // {x[4i+1], x[4i+3]}
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    uint32_t a[4];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 qq = qv[r][2 * h + (i >> 2)];
                        const uint32_t w = (i & 3) == 0 ? qq.x : (i & 3) == 1 ? qq.y : (i & 3) == 2 ? qq.z : qq.w;
                        // code = 1024 + q (low nibbles) or 1024 + 16q (high nibbles)
                        const uint32_t mask = hi ? 0x00F000F0u : 0x000F000Fu;
                        const __half2 c02 = as_h2(and_or(w, mask, 0x64006400u));
                        const __half2 c13 = as_h2(and_or(w >> 8, mask, 0x64006400u));
                        const RowScales& z = rs[r][h];
                        const __half2 scx = hi ? __high2half2(as_h2(z.scx)) : __low2half2(as_h2(z.scx));
                        const __half2 nsc = hi ? __high2half2(as_h2(z.nscx)) : __low2half2(as_h2(z.nscx));
                        const __half2 nbh = hi ? __high2half2(as_h2(z.nbh)) : __low2half2(as_h2(z.nbh));
                        const __half2 nbl = hi ? __high2half2(as_h2(z.nbl)) : __low2half2(as_h2(z.nbl));
                        const __half2 d2 = as_h2(z.d2);
                        // P = sc*q exactly; w = fp16(d*P - B_h) - B_l  (within ~1 ulp of w)
                        const __half2 p02 = __hfma2(c02, scx, nsc);
                        const __half2 p13 = __hfma2(c13, scx, nsc);
                        a[h] = as_u32(__hadd2(__hfma2(p02, d2, nbh), nbl));       // k slots 2t, 2t+1
                        a[2 + h] = as_u32(__hadd2(__hfma2(p13, d2, nbh), nbl));   // k slots 2t+8, 2t+9
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_m16n8k16(acc[r][nt], a[0], a[1], a[2], a[3], b01[nt], b23[nt]);
                }
            }
        }

        // ---------------- fixed-order reduction of the warp partials of this row tile
        float* rw = red + warp * kRows * kRedCols;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int col = nt * 8 + 2 * t;
                rw[(16 * r + g) * kRedCols + col] = acc[r][nt][0];
                rw[(16 * r + g) * kRedCols + col + 1] = acc[r][nt][1];
                rw[(16 * r + g + 8) * kRedCols + col] = acc[r][nt][2];
                rw[(16 * r + g + 8) * kRedCols + col + 1] = acc[r][nt][3];
            }
        }
        named_bar_sync(1, kConsumerThreads);

        const int nw = static_cast<int>(jb - ja < kConsumerWarps ? jb - ja : kConsumerWarps);
        const bool whole = (ja + u0 == tile * KB) && (jb + u0 == (tile + 1) * KB);
        const int nel = kRows * p.m;
        if (whole) {
            for (int e = tid; e < nel; e += kConsumerThreads) {
                const int row = e & (kRows - 1), m = e / kRows;
                float v = red[row * kRedCols + m];
                for (int w = 1; w < nw; ++w) v += red[(w * kRows + row) * kRedCols + m];
                const int64_t n = tile * kRows + row;
                if (n < p.n) p.y[m * p.n + n] = v;
            }
        } else {
            const int side = (tile == t_first) ? 0 : 1;
            float* part = p.ws + (c * 2 + side) * kRows * p.ws_cols;
            for (int e = tid; e < nel; e += kConsumerThreads) {
                const int row = e & (kRows - 1), m = e / kRows;
                float v = red[row * kRedCols + m];
                for (int w = 1; w < nw; ++w) v += red[(w * kRows + row) * kRedCols + m];
                part[m * kRows + row] = v;
            }
            __threadfence();
            named_bar_sync(1, kConsumerThreads);
            const int64_t pa = dev_piece_of(tile * KB, U, p.grid);
            const int64_t pb = dev_piece_of((tile + 1) * KB - 1, U, p.grid);
            if (tid == 0) {
                const int old = atomicAdd(&p.tickets[tile], 1);
                flags[1] = (old == static_cast<int>(pb - pa)) ? 1 : 0;
            }
            named_bar_sync(1, kConsumerThreads);
            if (flags[1]) {
                __threadfence();
                for (int e = tid; e < nel; e += kConsumerThreads) {
                    const int row = e & (kRows - 1), m = e / kRows;
                    float v = 0.f;
                    for (int64_t pc = pa; pc <= pb; ++pc) {
                        const int64_t pc_first_tile = (pc * U / p.grid) / KB;
                        const int sd = (tile == pc_first_tile) ? 0 : 1;
                        const float pv = __ldcg(p.ws + (pc * 2 + sd) * kRows * p.ws_cols + m * kRows + row);
                        v = (pc == pa) ? pv : v + pv;
                    }
                    const int64_t n = tile * kRows + row;
                    if (n < p.n) p.y[m * p.n + n] = v;
                }
                if (tid == 0) p.tickets[tile] = 0;  // ready for the next run
            }
        }
        named_bar_sync(1, kConsumerThreads);  // red and flags are reused by the next tile
    }
}

// One thread per 16-byte piece of the packed layout.
__global__ void repack_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                              int64_t n, int32_t kb, int64_t units) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    constexpr int kSegs = kUnitBytes / 16;  // 288
    if (idx >= units * kSegs) return;
    const int64_t u = idx / kSegs;
    const int seg = static_cast<int>(idx % kSegs);
    const int64_t tile = u / kb;
    const int b = static_cast<int>(u % kb);
    int row, off;
    if (seg < 256) {
        const int r = seg >> 7, i = (seg >> 5) & 3, L = seg & 31;
        const int g = L >> 2, t = L & 3, h = i >> 1, bh = i & 1;
        row = 16 * r + 8 * h + g;
        off = 16 + 32 * t + 16 * bh;
    } else {
        row = seg - 256;
        off = 0;
    }
    const int64_t nrow = tile * kRows + row;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (nrow < n) v = *reinterpret_cast<const uint4*>(src + (nrow * kb + b) * 144 + off);
    *reinterpret_cast<uint4*>(dst + u * kUnitBytes + seg * 16) = v;
}

cudaError_t repack(const uint8_t* src_dev, uint8_t* dst_dev, const Decomp& d, cudaStream_t s) {
    const int64_t total = d.units * (kUnitBytes / 16);
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    repack_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(src_dev, dst_dev, d.n,
                                                                   static_cast<int32_t>(d.kb), d.units);
    return cudaGetLastError();
}

cudaError_t configure() {
    cudaError_t e = cudaFuncSetAttribute(stream_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes());
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(stream_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes());
}

cudaError_t launch(const B1Params& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.m <= 8) return cudaLaunchKernelEx(&cfg, stream_kernel<1>, p);
    return cudaLaunchKernelEx(&cfg, stream_kernel<2>, p);
}

}  // namespace b1
}  // namespace qmm
