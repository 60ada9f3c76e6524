// Internal declarations shared by the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qmm.h"

namespace qmm {

// Work decomposition shared by the backends: the weight matrix is cut into units of
// (rows_per_unit output rows) x (one 256-wide super-block column).  Units are numbered
// row-tile-major, u = tile * KB + kb, and stored contiguously in that order, so a run of
// consecutive units is one contiguous byte range.  Each persistent CTA c takes the units
// [c*U/P, (c+1)*U/P): a fixed piece that depends only on (N, K, P), never on M.
struct Decomp {
    int64_t n = 0, k = 0, kb = 0;  // kb = K / 256
    int64_t tiles = 0;             // ceil(N / rows_per_unit)
    int64_t units = 0;             // tiles * kb
    int32_t rows = 0;              // rows per unit
    int32_t unit_bytes = 0;        // rows * 144
    int32_t grid = 0;              // P, persistent CTAs (<= units)
};

// Piece containing unit u (host mirror of the device formula).
inline int64_t piece_of(int64_t u, int64_t units, int64_t grid) {
    return ((u + 1) * grid + units - 1) / units - 1;
}

// One matrix of a backend-1 launch.  A launch works on the concatenation of its matrices' unit
// sequences (matrix i's units at base_i .. base_i + units_i - 1) and cuts it into one piece per
// CTA; a single run has one matrix and passes it by value, a decode step keeps an array of
// them in device memory (the tensor map needs 64-byte alignment).
struct alignas(128) MatDesc {
    CUtensorMap xmap;      // activations [m, k] fp16, 128-byte swizzle: box 64 x 8 (mma.sync) or 64 x MP (tcgen05)
    CUtensorMap smap;      // tcgen05 Q4_K launches of MP = 128: the activation sums [kb][m][8] fp16, box 8 x 128 x 1
    CUtensorMap ymap;      // tcgen05 y launches with N % 4 == 0: y [m, n] fp32, box 128 x 16 (bulk stores)
    const __half* xsrc;    // ... the activations they are formed from ([m, k], row stride k)
    __half* xs;            // ... and where the pre-pass writes them
    uint8_t* frag;         // mma.sync steps: the matrix's MMA B fragments, one record per super-block
                           // column, formed from xsrc by a pre-pass (null otherwise)
    const uint8_t* wq;     // repacked units
    float* y;              // [m, n] fp32
    int* tickets;          // [tiles]: partials published for the tile; zero between runs
    int64_t base;          // first unit of this matrix in the launch's sequence (0 in dependent steps)
    int64_t units;
    int64_t n;
    int32_t kb;
    int32_t pieces;        // dependent steps: pieces the matrix is cut into (its handle's grid)
    int32_t ytma;          // ymap is set: the epilogue may write y with bulk tensor stores
    int32_t pad[3];
};

struct LaunchParams {
    const MatDesc* mats;       // device array of `count` matrices (count > 1 only)
    const int32_t* first_mat;// [grid]: matrix holding each piece's first unit (count > 1 only)
    float* ws;               // split-K partials: per CTA one (mma.sync) or two (tcgen05) slots of
                             // 128 threads x ws_cols floats
    int* err;                // sticky error word (mapped host memory)
    int64_t units;           // units of all matrices of the launch
    int32_t count;           // matrices in this launch
    int32_t m;               // rows of this launch (1..16 mma.sync, 1..128 tcgen05)
    int32_t ws_cols;         // floats per consumer thread in a partial slot
    int32_t b1_frags;        // mma.sync: the matrices' fragments come from their frag records
    int32_t park_all;        // tcgen05, testing: every split tile's reducer parks its partial
                             // (the rare path of the split-K sum; same results)
    // Row-wise argmax instead of y (single-matrix launches only; null otherwise): the
    // launch folds (value, column) keys into amax_keys[m] (zero before and after a launch),
    // and the last of its writer warps, counted in amax_count (zero before and after),
    // decodes them into amax_idx[m] / amax_val[m].
    unsigned long long* amax_keys;
    int* amax_count;
    int32_t* amax_idx;
    float* amax_val;
    // Longest time a wait of the launch's protocol (ring slots, hand-offs, tickets) may take
    // before the launch gives up and reports QMM_ERR_DEVICE_TIMEOUT; the waits that let copies
    // in flight land before a CTA exits always use kDrainLimitNs.
    uint64_t wait_ns;
    // Dependent steps (tcgen05 backend; null otherwise): matrix i is cut into its own
    // mats[i].pieces pieces, exactly as a single run of its handle (CTA c takes piece c, CTAs
    // past the last piece none), the matrices are taken in order, and a CTA loads matrix i's
    // activations only once done[i - 1] counts every CTA of the launch, i.e. once every output
    // of matrix i - 1 is written.  done[count] counts the CTAs that have finished; the last of
    // them zeroes all count + 1 counters for the next launch.  cta_units[c] = CTA c's units
    // over all matrices.
    int* done;
    const int32_t* cta_units;
};

// Default wait limit of a launch, and the limit of the drains on a failure path.
constexpr uint64_t kDefaultWaitNs = 4000000000ull;  // 4 s
constexpr uint64_t kDrainLimitNs = 10000000000ull;  // 10 s
// How long the tcgen05 kernel's split-tile reducer polls for the other pieces' partials before
// it parks its own and leaves the sum to the last piece to arrive (a piece that has not
// started cannot be waited for).
constexpr uint64_t kParkAfterNs = 3000;  // 3 us

// Argmax keys: the value's bits mapped to an unsigned order (larger value, larger key; -0
// counts as +0) in the high half, the complement of the column in the low half, so that the
// largest key is the largest value at its lowest column.  Key 0 is below every value.
__device__ __forceinline__ unsigned long long amax_key(float v, int64_t n) {
    const uint32_t u = __float_as_uint(v + 0.0f);
    const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(o) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(n));
}

// Warp-collective, after the warp has folded its keys into p.amax_keys: the last of the
// launch's `writers` warps to arrive decodes every row's key into amax_idx / amax_val (column
// -1 if a row saw no column) and zeroes the keys and the counter for the next launch.
__device__ __forceinline__ void amax_finish_warp(const LaunchParams& p, int writers, int lane) {
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(p.amax_count, 1) == writers - 1;
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __threadfence();
    for (int m = lane; m < p.m; m += 32) {
        const unsigned long long k = atomicExch(p.amax_keys + m, 0ull);
        const uint32_t o = static_cast<uint32_t>(k >> 32);
        p.amax_idx[m] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k));
        p.amax_val[m] = __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
    }
    __syncwarp();
    if (lane == 0) atomicExch(p.amax_count, 0);
}

// Block formats: bytes per block and weights per block, by QMM_FORMAT_*.
__host__ __device__ constexpr int block_bytes(int format) { return format == QMM_FORMAT_Q6_K ? 210 : format == QMM_FORMAT_Q8_0 ? 34 : 144; }
__host__ __device__ constexpr int block_weights(int format) { return format == QMM_FORMAT_Q8_0 ? 32 : 256; }

// Backend 2: tcgen05 streaming kernel (weights dequantised into tensor memory, x by TMA).
namespace b2 {
constexpr int kRows = 128;
constexpr int kUnitBytes = kRows * 144;  // Q4_K
// bytes of one unit (128 rows x 256 weights) of a format
__host__ __device__ constexpr int unit_bytes(int format) { return kRows * block_bytes(format) * (256 / block_weights(format)); }
constexpr int kMaxM = 128;  // rows per launch
int mp_for(int64_t m);      // tokens per launch tile: 16, 32, 64 or 128
cudaError_t repack(const uint8_t* src_dev, uint8_t* dst_dev, const Decomp& d, int format, cudaStream_t s);
// Launches whose activation sums (the per-sub-block sums of x that the -B_l step needs) come
// from a pre-pass kernel instead of being formed by the dequantisation warps from each unit's
// x tile: Q4_K at more than 64 rows (MP = 128).  At that width shared memory holds only two
// x tiles, and a tile's L2 round trip would otherwise sit between one unit's MMAs and the
// dequantisation of the unit two places on.
inline bool presum_for(int64_t m, int format) { return format == QMM_FORMAT_Q4_K && m > 64; }
// Bytes of the activation sums of a launch of m rows of a matrix of kb super-block columns.
inline int64_t presum_bytes(int64_t m, int64_t kb) { return kb * m * 16; }
// Floats of the split-K partial slots of a launch of `grid` CTAs at tile width mp: two slots
// per CTA of 128 rows x mp columns (the partial of its piece's first row tile, and its last
// row tile's partial when it must leave that tile's reduction to a later CTA).
inline int64_t ws_floats(int64_t grid, int32_t mp) { return 2 * grid * kRows * mp; }
// Fill a matrix descriptor for a run of m rows (1..128) of x against the handle's weights;
// xs (presum_bytes(m, kb) bytes, 16-byte aligned) receives the activation sums of launches
// with presum_for(m, format), and is null otherwise.
cudaError_t make_mat(MatDesc* out, const uint8_t* wq, const void* x, float* y, int* tickets, int64_t units,
                     int64_t n, int32_t kb, int32_t m, __half* xs);
// Launch over `p.count` matrices of one format (`single` when count == 1) on `grid` CTAs;
// p.ws_cols = mp_for(p.m).  No CTA waits for another in the split-K reduction, so a launch
// needs to be cooperative only where it waits across CTAs for another reason (the dependent
// persistent step's completion counters).
cudaError_t launch(const MatDesc& single, const LaunchParams& p, int grid, cudaStream_t s, bool pdl, bool cooperative,
                   int format);
cudaError_t configure();
// The pre-pass of a launch with presum_for(p.m, format): the activation sums of every matrix
// of the launch (`single` when p.count == 1, p.mats otherwise; max_kb the largest kb), issued
// in stream order before the launch as a plain (not programmatic) launch.
cudaError_t presum(const MatDesc& single, const LaunchParams& p, int32_t max_kb, cudaStream_t s);
}  // namespace b2

// Backend 1: warp-level mma.sync streaming kernel.
namespace b1 {
constexpr int kRows = 256;
constexpr int kUnitBytes = kRows * 144;
constexpr int kMaxM = 16;  // rows per launch
constexpr int kConsumerThreads = 512;  // most consumer threads of a launch (16 warps at 9-16 rows)
// floats of a split-K partial per consumer thread for runs of up to m rows; a handle keeps
// one slot of kConsumerThreads x ws_floats per CTA
constexpr int32_t ws_floats(int64_t) { return 8; }  // 8 warps x 2 row tiles x 1 fragment, or 16 x 1 x 2
int smem_bytes(int nt);
cudaError_t repack(const uint8_t* src_dev, uint8_t* dst_dev, const Decomp& d, cudaStream_t s);
// Fill a matrix descriptor for a run of m rows (1..16) of x against the handle's weights.
cudaError_t make_mat(MatDesc* out, const uint8_t* wq, const void* x, float* y, int* tickets, int64_t units,
                     int64_t n, int32_t kb, int32_t m);
// Bytes of one fragment record (one super-block column of x: the MMA B fragments of the
// launch's rows and their sub-block sums) for launches of m rows.
int64_t frag_record_bytes(int64_t m);
// The pre-pass of a launch with p.b1_frags: writes every matrix's fragment records (MatDesc::frag,
// kb records each) from its activations, as a plain launch in stream order before the main one.
cudaError_t prefrag(const MatDesc& single, const LaunchParams& p, int32_t max_kb, cudaStream_t s);
// Launch over `p.count` matrices (`single` when count == 1) on `grid` persistent CTAs.
cudaError_t launch(const MatDesc& single, const LaunchParams& p, int grid, cudaStream_t s, bool pdl, bool cooperative);
cudaError_t configure();  // one-time function attributes
}  // namespace b1

}  // namespace qmm

struct qmm_handle_s {
    uint64_t magic;
    int device;
    int32_t backend;
    int32_t format = QMM_FORMAT_Q4_K;
    int64_t m_max;
    qmm::Decomp d;
    uint8_t* wq = nullptr;        // repacked weights
    int64_t wq_bytes = 0;
    float* ws = nullptr;          // split-K partials
    int32_t ws_cols = 0;
    int* tickets = nullptr;
    int32_t park = 0;             // QMM_SPLITK_PARK set at create: launches set park_all
    int* err_host = nullptr;      // mapped pinned word: host view
    int* err_dev = nullptr;       // device view of the same word
    void* x_stage = nullptr;      // host_io staging
    float* y_stage = nullptr;
    unsigned long long* amax_keys = nullptr;  // qmm_run_argmax: [128] keys, then the counter
    __half* xsum = nullptr;       // activation sums of one launch of up to 128 rows (tcgen05 Q4_K, m_max > 64)
    int* amax_count = nullptr;
    uint64_t wait_ns = qmm::kDefaultWaitNs;  // protocol wait limit of the handle's launches
};
