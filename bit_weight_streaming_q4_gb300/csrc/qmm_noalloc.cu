// qmm_run_noalloc: a run of the mma.sync streaming kernel that allocates nothing.
//
// Who needs it.  Some callers cannot call cudaMalloc at the point where they need a matmul:
// a host framework that owns all device memory through its own pool and forbids other
// allocations, code that must not synchronise the device (cudaMalloc and cudaFree can), or a
// plugin that runs inside someone else's process with a fixed memory budget.  qmm_create
// allocates the packed weights, the split-K workspace and the tile tickets; this entry point
// instead takes the raw Q4_K blocks, packs them into a fixed scratch area and runs from there.
//
// The scratch area is one file-scope __device__ array of kScratchBytes.  Every GPU that loads
// the library holds it until the process exits.  Each call packs the weights into it, clears
// the tile tickets and the error word, and runs; the array keeps the last call's contents.  All
// calls share it, so calls that overlap on the GPU (different streams, or different host
// threads) race and give wrong results: serialise them.
//
// A device-side wait that gives up cannot be reported through the return value (the call
// returns before the kernel runs, and reading the error word back would synchronise).  So a
// last small kernel of each call reads the call's error word and, if it is set, fills the
// call's y with NaN: a failed call never leaves plausible numbers behind.
#include <cuda_runtime.h>

#include <mutex>

#include "qmm.h"
#include "qmm_internal.h"

namespace {

// 48 MiB: packed weights of matrices up to ~40 MiB of Q4_K blocks plus the split-K workspace
// of a 16-row launch.
constexpr size_t kScratchBytes = size_t(48) << 20;
__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
bool g_configured[kMaxDevices] = {};  // kernel attributes set, per device

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// y[0 .. count) = NaN if the call's error word is set; nothing otherwise.
__global__ void poison_on_error(const int* __restrict__ err, float* __restrict__ y, int64_t count) {
    if (*reinterpret_cast<const volatile int*>(err) == 0) return;
    const float nan = __int_as_float(0x7FC00000);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        y[i] = nan;
}

}  // namespace

extern "C" qmm_status qmm_run_noalloc(const void* blocks, int64_t n, int64_t k, const void* x, int64_t m, float* y,
                                      void* stream) {
    if (!blocks || !x || !y) return QMM_ERR_INVALID_ARG;
    if (m < 0) return QMM_ERR_INVALID_ARG;
    if (n <= 0 || k <= 0 || k % 256 != 0) return QMM_ERR_UNSUPPORTED_SHAPE;
    if ((reinterpret_cast<uintptr_t>(blocks) | reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u)
        return QMM_ERR_MISALIGNED;

    // layout of the scratch area for this shape: packed weights, workspace, tickets, error word
    const int64_t kb = k / 256;
    const int64_t tiles = (n + qmm::b1::kRows - 1) / qmm::b1::kRows;
    const int64_t units = tiles * kb;
    const size_t packed = align256(static_cast<size_t>(units) * qmm::b1::kUnitBytes);
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return QMM_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return QMM_ERR_NO_DEVICE;
    const int64_t grid = units < sms ? units : sms;
    const int32_t cols = qmm::b1::ws_floats(m);
    const size_t ws = align256(static_cast<size_t>(grid) * qmm::b1::kConsumerThreads * cols * sizeof(float));
    const size_t tickets = align256(static_cast<size_t>(tiles) * sizeof(int));
    const size_t need = packed + ws + tickets + 256;
    if (need > kScratchBytes) return QMM_ERR_SCRATCH_TOO_SMALL;
    if (m == 0) return QMM_OK;

    // The host-side name g_scratch is only a stand-in: every call looks up the array's device
    // address on the current device (cheap, and never stale, e.g. after a device reset).  The
    // first call on each device also sets the kernel's attributes, so it must come before any
    // stream capture.
    unsigned char* base = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_setup_mu);
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return QMM_ERR_CUDA;
        if (!g_configured[dev]) {
            if (qmm::b1::configure() != cudaSuccess) return QMM_ERR_CUDA;
            g_configured[dev] = true;
        }
        base = static_cast<unsigned char*>(p);
    }
    uint8_t* wq = base;
    float* wsp = reinterpret_cast<float*>(base + packed);
    int* tk = reinterpret_cast<int*>(base + packed + ws);
    int* err = reinterpret_cast<int*>(base + packed + ws + tickets);

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    qmm::Decomp d;
    d.n = n;
    d.k = k;
    d.kb = kb;
    d.rows = qmm::b1::kRows;
    d.unit_bytes = qmm::b1::kUnitBytes;
    d.tiles = tiles;
    d.units = units;
    d.grid = static_cast<int32_t>(grid);
    if (qmm::b1::repack(static_cast<const uint8_t*>(blocks), wq, d, s) != cudaSuccess) return QMM_ERR_CUDA;
    // the tile tickets and the error word must start at zero; the previous call left them set
    if (cudaMemsetAsync(tk, 0, tickets + 256, s) != cudaSuccess) return QMM_ERR_CUDA;
    for (int64_t r0 = 0; r0 < m; r0 += qmm::b1::kMaxM) {
        const int64_t mc = (m - r0 < qmm::b1::kMaxM) ? m - r0 : qmm::b1::kMaxM;
        qmm::MatDesc mat;
        if (qmm::b1::make_mat(&mat, wq, static_cast<const __half*>(x) + r0 * k, y + r0 * n, tk, units, n,
                              static_cast<int32_t>(kb), static_cast<int32_t>(mc)) != cudaSuccess)
            return QMM_ERR_CUDA;
        qmm::LaunchParams p = {};
        p.ws = wsp;
        p.err = err;
        p.units = units;
        p.count = 1;
        p.m = static_cast<int32_t>(mc);
        p.ws_cols = cols;
        p.wait_ns = qmm::kDefaultWaitNs;
        // cooperative, as qmm_run's launches of this kernel: its split-K reducer waits for the
        // partials of CTAs after it
        if (qmm::b1::launch(mat, p, static_cast<int>(grid), s, false, true) != cudaSuccess) return QMM_ERR_CUDA;
    }
    const int64_t count = m * n;
    const int64_t nblk = (count + 255) / 256 < 1024 ? (count + 255) / 256 : 1024;
    poison_on_error<<<static_cast<unsigned>(nblk), 256, 0, s>>>(err, y, count);
    if (cudaGetLastError() != cudaSuccess) return QMM_ERR_CUDA;
    return QMM_OK;
}
