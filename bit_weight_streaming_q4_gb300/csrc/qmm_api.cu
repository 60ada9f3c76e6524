// C-ABI layer: argument checking, handle lifetime, device memory, launch, and the
// graph-recorded decode step.  See include/qmm.h for the contract.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <set>
#include <new>
#include <unordered_set>
#include <vector>

#include "qmm.h"
#include "qmm_internal.h"

namespace {

constexpr uint64_t kMagic = 0x514D4D5F48414E44ull;  // "QMM_HAND"

std::mutex g_mu;
std::unordered_set<const void*> g_handles;
std::unordered_set<const void*> g_steps;

bool live_handle(const qmm_handle h) {
    std::lock_guard<std::mutex> lk(g_mu);
    return h && g_handles.count(h) && h->magic == kMagic;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

qmm_status check_device(int* dev_out, int* sms_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_ERR_NO_DEVICE;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return QMM_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return QMM_ERR_NO_DEVICE;  // built for sm_103a only
    *dev_out = dev;
    *sms_out = sms;
    return QMM_OK;
}

void free_handle(qmm_handle h) {
    if (!h) return;
    cudaFree(h->wq);
    cudaFree(h->ws);
    cudaFree(h->tickets);
    if (h->err_host) cudaFreeHost(h->err_host);
    cudaFree(h->x_stage);
    cudaFree(h->y_stage);
    cudaFree(h->amax_keys);
    cudaFree(h->xsum);
    h->magic = 0;
    delete h;
}

int32_t per_launch(const qmm_handle h) {
    return h->backend == QMM_BACKEND_TCGEN05 ? qmm::b2::kMaxM : qmm::b1::kMaxM;
}

// Largest m_max for which QMM_BACKEND_AUTO picks the mma.sync backend (all it supports: one
// launch of up to 16 rows streams faster there than the tcgen05 kernel's, measured on GB300).
constexpr int64_t kAutoMmaSyncMaxM = 16;

// One run in launches of at most per_launch(h) rows.  With idx and val given, each launch
// writes its rows' argmax column and value there instead of y (y is not touched).
qmm_status launch_run(qmm_handle h, const void* x, int64_t m, float* y, cudaStream_t s, bool pdl,
                      int32_t* idx = nullptr, float* val = nullptr) {
    const int64_t K = h->d.k, N = h->d.n;
    const int64_t step = per_launch(h);
    for (int64_t r0 = 0; r0 < m; r0 += step) {
        const int64_t mc = (m - r0 < step) ? m - r0 : step;
        const __half* xc = reinterpret_cast<const __half*>(x) + r0 * K;
        float* yc = idx ? nullptr : y + r0 * N;
        const bool tc = h->backend == QMM_BACKEND_TCGEN05;
        const bool pre = tc && qmm::b2::presum_for(mc, h->format);
        qmm::MatDesc mat;
        cudaError_t e = tc ? qmm::b2::make_mat(&mat, h->wq, xc, yc, h->tickets, h->d.units, N,
                                               static_cast<int32_t>(h->d.kb), static_cast<int32_t>(mc),
                                               pre ? h->xsum : nullptr)
                           : qmm::b1::make_mat(&mat, h->wq, xc, yc, h->tickets, h->d.units, N,
                                               static_cast<int32_t>(h->d.kb), static_cast<int32_t>(mc));
        if (e == cudaSuccess) {
            qmm::LaunchParams p = {};
            p.mats = nullptr;
            p.first_mat = nullptr;
            p.ws = h->ws;
            p.err = h->err_dev;
            p.units = h->d.units;
            p.count = 1;
            p.wait_ns = h->wait_ns;
            p.park_all = h->park;
            p.m = static_cast<int32_t>(mc);
            p.ws_cols = tc ? qmm::b2::mp_for(mc) : h->ws_cols;
            if (idx) {
                p.amax_keys = h->amax_keys;
                p.amax_count = h->amax_count;
                p.amax_idx = idx + r0;
                p.amax_val = val + r0;
            }
            // the activation sums first, as a plain launch: that also keeps them from
            // overwriting the sums the handle's previous launch may still be reading
            if (pre) e = qmm::b2::presum(mat, p, static_cast<int32_t>(h->d.kb), s);
            // the mma.sync kernel's split-K reducer waits for the partials of the CTAs after it,
            // so its CTAs must be co-resident (a cooperative launch); in the tcgen05 kernel no
            // CTA waits for another, and without the attribute a run overlaps the one before
            // it (about 2 us per launch on GB300)
            if (e == cudaSuccess)
                e = tc ? qmm::b2::launch(mat, p, h->d.grid, s, pdl, false, h->format)
                       : qmm::b1::launch(mat, p, h->d.grid, s, pdl, true);
        }
        if (e != cudaSuccess) return QMM_ERR_CUDA;
    }
    return QMM_OK;
}

}  // namespace

extern "C" {

void qmm_default_options(qmm_options* opt) {
    if (!opt) return;
    opt->m_max = 16;
    opt->backend = QMM_BACKEND_AUTO;
    opt->ctas_per_sm = 0;
    opt->host_io = 0;
    opt->format = QMM_FORMAT_Q4_K;
    opt->wait_limit_us = 0;
}

const char* qmm_status_str(qmm_status s) {
    switch (s) {
        case QMM_OK: return "ok";
        case QMM_ERR_INVALID_ARG: return "invalid argument";
        case QMM_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case QMM_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case QMM_ERR_OOM: return "device allocation failed";
        case QMM_ERR_CUDA: return "CUDA error";
        case QMM_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case QMM_ERR_BAD_HANDLE: return "bad handle";
        case QMM_ERR_NO_DEVICE: return "no sm_103 device";
        case QMM_ERR_SCRATCH_TOO_SMALL: return "shape exceeds the fixed scratch of qmm_run_noalloc";
    }
    return "unknown status";
}

qmm_status qmm_create(qmm_handle* out, const void* blocks, int64_t n, int64_t k,
                      int32_t blocks_on_device, const qmm_options* opt_in, void* stream) {
    if (!out || !blocks) return QMM_ERR_INVALID_ARG;
    *out = nullptr;
    qmm_options opt;
    qmm_default_options(&opt);
    if (opt_in) opt = *opt_in;
    if (opt.m_max < 1 || opt.ctas_per_sm < 0 || opt.ctas_per_sm > 4 || opt.backend < 0 || opt.wait_limit_us < 0 ||
        opt.backend > QMM_BACKEND_TCGEN05 || opt.format < QMM_FORMAT_Q4_K || opt.format > QMM_FORMAT_Q8_0)
        return QMM_ERR_INVALID_ARG;
    // the mma.sync backend streams Q4_K only
    if (opt.format != QMM_FORMAT_Q4_K && opt.backend == QMM_BACKEND_MMA_SYNC) return QMM_ERR_INVALID_ARG;
    if (n <= 0 || k <= 0 || k % 256 != 0) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (blocks_on_device && !aligned16(blocks)) return QMM_ERR_MISALIGNED;

    int dev = 0, sms = 0;
    qmm_status st = check_device(&dev, &sms);
    if (st != QMM_OK) return st;
    static std::once_flag cfg_once;
    static cudaError_t cfg_err = cudaSuccess;
    std::call_once(cfg_once, [] {
        cfg_err = qmm::b1::configure();
        if (cfg_err == cudaSuccess) cfg_err = qmm::b2::configure();
    });
    if (cfg_err != cudaSuccess) return QMM_ERR_CUDA;

    qmm_handle h = new (std::nothrow) qmm_handle_s();
    if (!h) return QMM_ERR_OOM;
    h->magic = kMagic;
    h->device = dev;
    // Auto: the register-fed mma.sync stream for handles that never see more than 16 rows (one
    // launch, one or two n8 fragments per MMA), tcgen05 for wider handles.  Fixed per handle
    // (never per run), so that a row's result does not depend on how many rows it is batched
    // with.
    if (opt.backend == QMM_BACKEND_AUTO)
        h->backend = opt.m_max <= kAutoMmaSyncMaxM && opt.format == QMM_FORMAT_Q4_K ? QMM_BACKEND_MMA_SYNC
                                                                                    : QMM_BACKEND_TCGEN05;
    else
        h->backend = opt.backend;
    const bool tc = h->backend == QMM_BACKEND_TCGEN05;
    h->m_max = opt.m_max;
    h->wait_ns = opt.wait_limit_us ? static_cast<uint64_t>(opt.wait_limit_us) * 1000u : qmm::kDefaultWaitNs;
    {
        // testing: the rare path of the tcgen05 split-K sum on every split tile
        const char* park = std::getenv("QMM_SPLITK_PARK");
        h->park = park && park[0] == '1' ? 1 : 0;
    }
    qmm::Decomp& d = h->d;
    d.n = n;
    d.k = k;
    d.kb = k / 256;
    d.rows = tc ? qmm::b2::kRows : qmm::b1::kRows;
    h->format = opt.format;
    d.unit_bytes = tc ? qmm::b2::unit_bytes(opt.format) : qmm::b1::kUnitBytes;
    d.tiles = (n + d.rows - 1) / d.rows;
    d.units = d.tiles * d.kb;
    const int cps = opt.ctas_per_sm ? opt.ctas_per_sm : 1;
    d.grid = static_cast<int32_t>(d.units < static_cast<int64_t>(sms) * cps ? d.units
                                                                           : static_cast<int64_t>(sms) * cps);
    // split-K partial slot width: tcgen05, one column per row of x (up to 128); mma.sync, the
    // accumulator floats of a consumer thread (8 per 8-row group of x, up to 16)
    if (tc)
        h->ws_cols = qmm::b2::mp_for(opt.m_max < qmm::b2::kMaxM ? opt.m_max : qmm::b2::kMaxM);
    else
        h->ws_cols = qmm::b1::ws_floats(opt.m_max);
    h->wq_bytes = d.units * d.unit_bytes;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* staging = nullptr;
    auto fail = [&](qmm_status code) {
        cudaFree(staging);
        free_handle(h);
        return code;
    };
    if (cudaMalloc(&h->wq, h->wq_bytes) != cudaSuccess) return fail(QMM_ERR_OOM);
    // split-K partial slots, one per CTA: 128 rows x up to 128 columns (tcgen05), or the
    // accumulators of the consumer threads (mma.sync)
    const size_t ws_bytes =
        (tc ? static_cast<size_t>(qmm::b2::ws_floats(d.grid, h->ws_cols))
            : static_cast<size_t>(d.grid) * qmm::b1::kConsumerThreads * h->ws_cols) * sizeof(float);
    if (cudaMalloc(&h->ws, ws_bytes) != cudaSuccess) return fail(QMM_ERR_OOM);
    if (cudaMalloc(&h->tickets, d.tiles * sizeof(int)) != cudaSuccess) return fail(QMM_ERR_OOM);
    if (cudaMemsetAsync(h->tickets, 0, d.tiles * sizeof(int), s) != cudaSuccess) return fail(QMM_ERR_CUDA);
    // argmax keys (one per row of a launch, at most 128) and their launch counter
    constexpr int kKeys = qmm::b2::kMaxM > qmm::b1::kMaxM ? qmm::b2::kMaxM : qmm::b1::kMaxM;
    constexpr size_t kAmaxBytes = kKeys * sizeof(unsigned long long) + sizeof(unsigned long long);
    if (cudaMalloc(&h->amax_keys, kAmaxBytes) != cudaSuccess) return fail(QMM_ERR_OOM);
    h->amax_count = reinterpret_cast<int*>(h->amax_keys + kKeys);
    if (cudaMemsetAsync(h->amax_keys, 0, kAmaxBytes, s) != cudaSuccess) return fail(QMM_ERR_CUDA);
    // activation sums of launches of more than 64 rows (tcgen05 Q4_K)
    if (tc && qmm::b2::presum_for(opt.m_max, opt.format) &&
        cudaMalloc(&h->xsum, qmm::b2::presum_bytes(qmm::b2::kMaxM, d.kb)) != cudaSuccess)
        return fail(QMM_ERR_OOM);
    if (cudaHostAlloc(&h->err_host, sizeof(int), cudaHostAllocMapped) != cudaSuccess) return fail(QMM_ERR_OOM);
    *h->err_host = 0;
    if (cudaHostGetDevicePointer(&h->err_dev, h->err_host, 0) != cudaSuccess) return fail(QMM_ERR_CUDA);
    if (opt.host_io) {
        if (cudaMalloc(&h->x_stage, static_cast<size_t>(opt.m_max) * k * 2) != cudaSuccess) return fail(QMM_ERR_OOM);
        if (cudaMalloc(&h->y_stage, static_cast<size_t>(opt.m_max) * n * 4) != cudaSuccess) return fail(QMM_ERR_OOM);
    }

    const size_t src_bytes = static_cast<size_t>(n) * (k / qmm::block_weights(opt.format)) * qmm::block_bytes(opt.format);
    const uint8_t* src = static_cast<const uint8_t*>(blocks);
    if (!blocks_on_device) {
        if (cudaMalloc(&staging, src_bytes) != cudaSuccess) return fail(QMM_ERR_OOM);
        if (cudaMemcpyAsync(staging, blocks, src_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return fail(QMM_ERR_CUDA);
        src = staging;
    }
    const cudaError_t re = tc ? qmm::b2::repack(src, h->wq, d, opt.format, s) : qmm::b1::repack(src, h->wq, d, s);
    if (re != cudaSuccess) return fail(QMM_ERR_CUDA);
    if (cudaStreamSynchronize(s) != cudaSuccess) return fail(QMM_ERR_CUDA);
    cudaFree(staging);
    staging = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_handles.insert(h);
    }
    *out = h;
    return QMM_OK;
}

qmm_status qmm_run(qmm_handle h, const void* x, int64_t m, float* y, void* stream) {
    if (!live_handle(h)) return QMM_ERR_BAD_HANDLE;
    if (*reinterpret_cast<volatile int*>(h->err_host)) return QMM_ERR_DEVICE_TIMEOUT;
    if (m < 0) return QMM_ERR_INVALID_ARG;
    if (m == 0) return QMM_OK;
    if (m > h->m_max) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (!x || !y) return QMM_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return QMM_ERR_MISALIGNED;
    return launch_run(h, x, m, y, reinterpret_cast<cudaStream_t>(stream), true);
}

qmm_status qmm_run_argmax(qmm_handle h, const void* x, int64_t m, int32_t* idx, float* val, void* stream) {
    if (!live_handle(h)) return QMM_ERR_BAD_HANDLE;
    if (*reinterpret_cast<volatile int*>(h->err_host)) return QMM_ERR_DEVICE_TIMEOUT;
    if (m < 0) return QMM_ERR_INVALID_ARG;
    if (m == 0) return QMM_OK;
    if (m > h->m_max) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (!x || !idx || !val) return QMM_ERR_INVALID_ARG;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(idx) & 3) || (reinterpret_cast<uintptr_t>(val) & 3))
        return QMM_ERR_MISALIGNED;
    return launch_run(h, x, m, nullptr, reinterpret_cast<cudaStream_t>(stream), true, idx, val);
}

qmm_status qmm_run_host(qmm_handle h, const void* x_host, int64_t m, float* y_host, void* stream) {
    if (!live_handle(h)) return QMM_ERR_BAD_HANDLE;
    if (!h->x_stage) return QMM_ERR_INVALID_ARG;
    if (m < 0) return QMM_ERR_INVALID_ARG;
    if (m == 0) return QMM_OK;
    if (m > h->m_max) return QMM_ERR_UNSUPPORTED_SHAPE;
    if (!x_host || !y_host) return QMM_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(h->x_stage, x_host, static_cast<size_t>(m) * h->d.k * 2,
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QMM_ERR_CUDA;
    qmm_status st = qmm_run(h, h->x_stage, m, h->y_stage, stream);
    if (st != QMM_OK) return st;
    if (cudaMemcpyAsync(y_host, h->y_stage, static_cast<size_t>(m) * h->d.n * 4,
                        cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QMM_ERR_CUDA;
    return QMM_OK;
}

qmm_status qmm_get_error(qmm_handle h) {
    if (!live_handle(h)) return QMM_ERR_BAD_HANDLE;
    if (cudaDeviceSynchronize() != cudaSuccess) return QMM_ERR_CUDA;
    return *reinterpret_cast<volatile int*>(h->err_host) ? QMM_ERR_DEVICE_TIMEOUT : QMM_OK;
}

qmm_status qmm_get_info(qmm_handle h, qmm_info* info) {
    if (!live_handle(h)) return QMM_ERR_BAD_HANDLE;
    if (!info) return QMM_ERR_INVALID_ARG;
    info->n = h->d.n;
    info->k = h->d.k;
    info->m_max = h->m_max;
    info->backend = h->backend;
    info->grid = h->d.grid;
    info->units = h->d.units;
    info->rows_per_unit = h->d.rows;
    info->weight_bytes = h->d.n * (h->d.k / qmm::block_weights(h->format)) * qmm::block_bytes(h->format);
    info->packed_bytes = h->wq_bytes;
    info->workspace_bytes = (h->backend == QMM_BACKEND_TCGEN05
                                 ? qmm::b2::ws_floats(h->d.grid, h->ws_cols)
                                 : static_cast<int64_t>(h->d.grid) * qmm::b1::kConsumerThreads * h->ws_cols) * 4 +
                            h->d.tiles * 4;
    info->m_per_launch = per_launch(h);
    info->format = h->format;
    return QMM_OK;
}

qmm_status qmm_destroy(qmm_handle h) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!h || !g_handles.count(h)) return QMM_ERR_BAD_HANDLE;
        g_handles.erase(h);
    }
    cudaDeviceSynchronize();
    free_handle(h);
    return QMM_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------- decode step
// One host<->device copy of a step's host-buffer launch: `bytes` at device address `dev` and
// at byte offset `off` of the caller's host slab.
struct HostSeg {
    uint8_t* dev;
    size_t off;
    size_t bytes;
};

// Appends [dev, dev + bytes) at host offset off, merged into the previous copy when both
// ranges continue it.
static void add_seg(std::vector<HostSeg>& v, const void* dev, size_t off, size_t bytes) {
    uint8_t* d = static_cast<uint8_t*>(const_cast<void*>(dev));
    if (!v.empty() && v.back().dev + v.back().bytes == d && v.back().off + v.back().bytes == off)
        v.back().bytes += bytes;
    else
        v.push_back({d, off, bytes});
}

struct qmm_step_s {
    // qmm_step_launch_host: the copies in (x_i) and out (y_i), in matrix order, and the slabs' sizes
    std::vector<HostSeg> xin, yout;
    size_t x_bytes = 0, y_bytes = 0;
    // ... and, for copies on the caller's other streams: the last kernel's completion (which a
    // copy-out waits for, and the next copy-in, since it rewrites the x_i), the copy-in's (which
    // the kernel waits for) and the copy-out's (which the step's next kernel waits for, since it
    // rewrites the y_i)
    cudaEvent_t kernel_done = nullptr, in_done = nullptr, out_done = nullptr;
    bool out_pending = false;
    cudaGraph_t graph = nullptr;  // launch-per-run path (tcgen05 handles, or more than 16 rows)
    cudaGraphExec_t exec = nullptr;
    // persistent path: every matrix in one launch (cooperative for the mma.sync kernel)
    qmm::MatDesc* mats = nullptr;   // device
    int32_t* first_mat = nullptr; // device, [grid]: the matrix of each CTA's first unit
    float* ws = nullptr;          // split-K partial slots, one per CTA
    bool tcgen05 = false;         // the backend of every handle of a persistent step
    bool presum = false;          // ... whose activation sums come from a pre-pass
    int32_t max_kb = 0;
    __half* xsum = nullptr;       // device, the sums of every matrix
    int32_t format = QMM_FORMAT_Q4_K;  // ... and their block format
    uint8_t* frag = nullptr;      // device, mma.sync persistent steps: every matrix's fragment records
    int* done = nullptr;          // device, dependent persistent steps: [count + 1] completion counters
    int32_t* cta_units = nullptr; // device, dependent persistent steps: [grid] units of each CTA
    qmm::MatDesc single = {};     // the descriptor a one-matrix launch takes by value
    int* err_host = nullptr;
    int* err_dev = nullptr;
    qmm::LaunchParams params = {};
    int grid = 0;
};

static void free_step(qmm_step st) {
    if (!st) return;
    if (st->exec) cudaGraphExecDestroy(st->exec);
    if (st->graph) cudaGraphDestroy(st->graph);
    cudaFree(st->mats);
    cudaFree(st->first_mat);
    cudaFree(st->ws);
    cudaFree(st->xsum);
    cudaFree(st->done);
    cudaFree(st->cta_units);
    cudaFree(st->frag);
    if (st->err_host) cudaFreeHost(st->err_host);
    if (st->kernel_done) cudaEventDestroy(st->kernel_done);
    if (st->in_done) cudaEventDestroy(st->in_done);
    if (st->out_done) cudaEventDestroy(st->out_done);
    delete st;
}

extern "C" {

qmm_status qmm_step_create(qmm_step* out, int32_t count, const qmm_handle* handles,
                           const void* const* xs, float* const* ys, int64_t m, uint32_t flags, void* stream) {
    if (!out || count <= 0 || !handles || !xs || !ys || m < 1) return QMM_ERR_INVALID_ARG;
    if (flags & ~static_cast<uint32_t>(QMM_STEP_INDEPENDENT | QMM_STEP_GRAPH | QMM_STEP_PERSISTENT))
        return QMM_ERR_INVALID_ARG;
    *out = nullptr;
    for (int32_t i = 0; i < count; ++i) {
        if (!live_handle(handles[i])) return QMM_ERR_BAD_HANDLE;
        if (!xs[i] || !ys[i]) return QMM_ERR_INVALID_ARG;
        if (!aligned16(xs[i]) || !aligned16(ys[i])) return QMM_ERR_MISALIGNED;
        if (m > handles[i]->m_max) return QMM_ERR_UNSUPPORTED_SHAPE;
    }
    qmm_step st = new (std::nothrow) qmm_step_s();
    if (!st) return QMM_ERR_OOM;
    // One persistent kernel for the whole step, unless QMM_STEP_GRAPH asks for the graph, when
    // every handle has the same backend and block format and M fits one launch (16 rows
    // mma.sync, 128 tcgen05):
    //  - independent runs: the matrices' unit sequences are concatenated and cut into one
    //    piece per CTA (each handle at most once: its tickets serve one matrix of a launch);
    //  - dependent runs, when QMM_STEP_PERSISTENT asks for it (tcgen05 handles, M <= 64): the
    //    matrices are taken in order, each cut into its own pieces as a single run of its
    //    handle would be, and a CTA loads matrix i's activations only once every output of
    //    matrix i - 1 is written.
    // A CUDA graph of runs otherwise.
    const int32_t be = handles[0]->backend;
    const bool tc = be == QMM_BACKEND_TCGEN05;
    const bool indep = (flags & QMM_STEP_INDEPENDENT) != 0;
    bool persistent = m <= (tc ? qmm::b2::kMaxM : qmm::b1::kMaxM) && !(flags & QMM_STEP_GRAPH);
    // one persistent launch runs one kernel: one backend and one block format
    for (int32_t i = 0; i < count; ++i)
        persistent = persistent && handles[i]->backend == be && handles[i]->format == handles[0]->format;
    // a dependent step reads activations written during the launch, so they cannot come from a
    // pre-pass: the tensor-core kernel at up to 64 rows
    const bool dep = persistent && !indep;
    if (dep) persistent = (flags & QMM_STEP_PERSISTENT) && tc && !qmm::b2::presum_for(m, handles[0]->format);
    if (persistent && indep) {
        std::set<qmm_handle> seen(handles, handles + count);
        if (static_cast<int32_t>(seen.size()) != count) {
            delete st;
            return QMM_ERR_INVALID_ARG;
        }
    }
    qmm_status rc = QMM_OK;
    if (persistent) {
        std::vector<qmm::MatDesc> host(count);
        int64_t total = 0;
        // activation sums of every matrix (launches of more than 64 rows), one pre-pass per launch
        const bool pre = tc && qmm::b2::presum_for(m, handles[0]->format);
        int64_t sum_bytes = 0;
        int32_t max_kb = 0;
        for (int32_t i = 0; i < count; ++i) {
            sum_bytes += qmm::b2::presum_bytes(m, handles[i]->d.kb);
            max_kb = handles[i]->d.kb > max_kb ? static_cast<int32_t>(handles[i]->d.kb) : max_kb;
        }
        if (pre && cudaMalloc(&st->xsum, sum_bytes) != cudaSuccess) rc = QMM_ERR_OOM;
        // mma.sync: the MMA B fragments of every matrix's activations, formed once per launch by
        // a pre-pass (one record per super-block column) instead of once per unit in the kernel
        const int64_t frag_rec = tc ? 0 : qmm::b1::frag_record_bytes(m);
        int64_t frag_bytes = 0;
        for (int32_t i = 0; i < count && !tc; ++i) frag_bytes += handles[i]->d.kb * frag_rec;
        if (!tc && rc == QMM_OK && cudaMalloc(&st->frag, frag_bytes) != cudaSuccess) rc = QMM_ERR_OOM;
        int64_t frag_off = 0;
        int64_t sum_off = 0;
        for (int32_t i = 0; i < count && rc == QMM_OK; ++i) {
            const qmm_handle h = handles[i];
            __half* xsi = pre ? st->xsum + sum_off / 2 : nullptr;
            sum_off += qmm::b2::presum_bytes(m, h->d.kb);
            const cudaError_t me =
                tc ? qmm::b2::make_mat(&host[i], h->wq, xs[i], ys[i], h->tickets, h->d.units, h->d.n,
                                       static_cast<int32_t>(h->d.kb), static_cast<int32_t>(m), xsi)
                   : qmm::b1::make_mat(&host[i], h->wq, xs[i], ys[i], h->tickets, h->d.units, h->d.n,
                                       static_cast<int32_t>(h->d.kb), static_cast<int32_t>(m));
            if (me != cudaSuccess) rc = QMM_ERR_CUDA;
            if (!tc) {
                host[i].frag = st->frag + frag_off;
                frag_off += h->d.kb * frag_rec;
            }
            host[i].base = dep ? 0 : total;
            host[i].pieces = dep ? h->d.grid : 0;
            total += h->d.units;
        }
        int sms = 0;
        if (rc == QMM_OK && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, handles[0]->device) != cudaSuccess)
            rc = QMM_ERR_CUDA;
        int grid = static_cast<int>(total < sms ? total : sms);
        std::vector<int32_t> firsts(grid > 0 ? grid : 1);
        std::vector<int32_t> cta_units;
        if (dep) {
            // as many CTAs as the widest matrix has pieces; CTA c takes piece c of each matrix
            grid = 0;
            for (int32_t i = 0; i < count; ++i) grid = host[i].pieces > grid ? host[i].pieces : grid;
            cta_units.assign(grid, 0);
            for (int32_t i = 0; i < count; ++i)
                for (int c = 0; c < host[i].pieces; ++c)
                    cta_units[c] += static_cast<int32_t>((c + 1) * host[i].units / host[i].pieces -
                                                         c * host[i].units / host[i].pieces);
        } else {
            for (int c = 0, i = 0; c < grid; ++c) {
                const int64_t g0 = c * total / grid;
                while (host[i].base + host[i].units <= g0) ++i;
                firsts[c] = i;
            }
        }
        const int32_t ws_cols = tc ? qmm::b2::mp_for(m) : qmm::b1::ws_floats(m);
        const size_t ws_bytes =
            (tc ? static_cast<size_t>(qmm::b2::ws_floats(grid, ws_cols))
                : static_cast<size_t>(grid) * qmm::b1::kConsumerThreads * ws_cols) * sizeof(float);
        if (rc == QMM_OK && cudaMalloc(&st->mats, sizeof(qmm::MatDesc) * count) != cudaSuccess) rc = QMM_ERR_OOM;
        if (rc == QMM_OK && cudaMalloc(&st->first_mat, sizeof(int32_t) * firsts.size()) != cudaSuccess) rc = QMM_ERR_OOM;
        if (rc == QMM_OK && cudaMalloc(&st->ws, ws_bytes) != cudaSuccess) rc = QMM_ERR_OOM;
        if (rc == QMM_OK && dep &&
            (cudaMalloc(&st->done, sizeof(int) * (count + 1)) != cudaSuccess ||
             cudaMalloc(&st->cta_units, sizeof(int32_t) * cta_units.size()) != cudaSuccess))
            rc = QMM_ERR_OOM;
        if (rc == QMM_OK && dep &&
            (cudaMemset(st->done, 0, sizeof(int) * (count + 1)) != cudaSuccess ||
             cudaMemcpy(st->cta_units, cta_units.data(), sizeof(int32_t) * cta_units.size(), cudaMemcpyHostToDevice) !=
                 cudaSuccess))
            rc = QMM_ERR_CUDA;
        if (rc == QMM_OK && cudaHostAlloc(&st->err_host, sizeof(int), cudaHostAllocMapped) != cudaSuccess)
            rc = QMM_ERR_OOM;
        if (rc == QMM_OK) {
            *st->err_host = 0;
            if (cudaHostGetDevicePointer(&st->err_dev, st->err_host, 0) != cudaSuccess ||
                cudaMemcpy(st->mats, host.data(), sizeof(qmm::MatDesc) * count, cudaMemcpyHostToDevice) != cudaSuccess ||
                cudaMemcpy(st->first_mat, firsts.data(), sizeof(int32_t) * firsts.size(), cudaMemcpyHostToDevice) !=
                    cudaSuccess)
                rc = QMM_ERR_CUDA;
        }
        if (rc == QMM_OK) {
            st->tcgen05 = tc;
            st->presum = pre;
            st->max_kb = max_kb;
            st->format = handles[0]->format;
            st->grid = grid;
            st->params.mats = st->mats;
            st->params.first_mat = st->first_mat;
            st->params.ws = st->ws;
            st->params.err = st->err_dev;
            st->params.units = total;
            st->params.count = count;
            st->params.wait_ns = handles[0]->wait_ns;
            st->params.park_all = handles[0]->park;
            st->params.m = static_cast<int32_t>(m);
            st->params.ws_cols = ws_cols;
            st->params.done = st->done;
            st->params.cta_units = st->cta_units;
            st->params.b1_frags = tc ? 0 : 1;
            st->single = host[0];
        }
    } else {
        cudaStream_t cap = nullptr;
        if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess) rc = QMM_ERR_CUDA;
        if (rc == QMM_OK && cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
            rc = QMM_ERR_CUDA;
        for (int32_t i = 0; rc == QMM_OK && i < count; ++i)
            rc = launch_run(handles[i], xs[i], m, ys[i], cap, /*pdl=*/i > 0);
        if (cap) {
            cudaGraph_t g = nullptr;
            cudaError_t ec = cudaStreamEndCapture(cap, &g);
            if (rc == QMM_OK && ec != cudaSuccess) rc = QMM_ERR_CUDA;
            if (rc == QMM_OK && cudaGraphInstantiate(&st->exec, g, 0) != cudaSuccess) rc = QMM_ERR_CUDA;
            st->graph = g;
            cudaStreamDestroy(cap);
        }
    }
    if (rc != QMM_OK) {
        free_step(st);
        return rc;
    }
    (void)stream;
    if (cudaEventCreateWithFlags(&st->kernel_done, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&st->in_done, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&st->out_done, cudaEventDisableTiming) != cudaSuccess) {
        free_step(st);
        return QMM_ERR_CUDA;
    }
    for (int32_t i = 0; i < count; ++i) {
        const size_t xb = static_cast<size_t>(m) * handles[i]->d.k * 2;
        const size_t yb = static_cast<size_t>(m) * handles[i]->d.n * 4;
        add_seg(st->xin, xs[i], st->x_bytes, xb);
        add_seg(st->yout, ys[i], st->y_bytes, yb);
        st->x_bytes += xb;
        st->y_bytes += yb;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_steps.insert(st);
    }
    *out = st;
    return QMM_OK;
}

static qmm_status step_launch(qmm_step s, void* stream) {
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // a host-buffer launch may still be copying the y_i out on another stream
    if (s->out_pending && cudaStreamWaitEvent(cs, s->out_done, 0) != cudaSuccess) return QMM_ERR_CUDA;
    if (s->mats) {
        if (*reinterpret_cast<volatile int*>(s->err_host)) return QMM_ERR_DEVICE_TIMEOUT;
        // (a one-matrix step's kernel takes the descriptor by value)
        cudaError_t e = s->presum ? qmm::b2::presum(s->single, s->params, s->max_kb, cs)
                        : s->frag ? qmm::b1::prefrag(s->single, s->params, s->max_kb, cs)
                                  : cudaSuccess;
        if (e == cudaSuccess)
            e = s->tcgen05 ? qmm::b2::launch(s->single, s->params, s->grid, cs, true, true, s->format)
                           : qmm::b1::launch(s->single, s->params, s->grid, cs, true, true);
        return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
    }
    return cudaGraphLaunch(s->exec, cs) == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

qmm_status qmm_step_launch(qmm_step s, void* stream) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!s || !g_steps.count(s)) return QMM_ERR_BAD_HANDLE;
    }
    const qmm_status st = step_launch(s, stream);
    if (st != QMM_OK) return st;
    // a later host-buffer launch may copy its x_i in on another stream: after this kernel
    // (not while the stream is being captured into a graph, where the event would belong to
    // the capture; the caller then orders the graph's launches with the copies)
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(cs, &cap) != cudaSuccess) return QMM_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return QMM_OK;
    return cudaEventRecord(s->kernel_done, cs) == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

qmm_status qmm_step_launch_host(qmm_step s, const void* x_host, float* y_host, void* stream,
                                void* in_stream, void* out_stream) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!s || !g_steps.count(s)) return QMM_ERR_BAD_HANDLE;
    }
    if (!x_host || !y_host) return QMM_ERR_INVALID_ARG;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t is = reinterpret_cast<cudaStream_t>(in_stream);
    cudaStream_t os = reinterpret_cast<cudaStream_t>(out_stream);
    const bool split_in = in_stream != nullptr && is != cs;
    const bool split_out = out_stream != nullptr && os != cs;
    const uint8_t* xh = static_cast<const uint8_t*>(x_host);
    uint8_t* yh = reinterpret_cast<uint8_t*>(y_host);
    // copy-in: on in_stream once the step's last kernel has read the x_i, then the kernel waits
    if (split_in && cudaStreamWaitEvent(is, s->kernel_done, 0) != cudaSuccess) return QMM_ERR_CUDA;
    for (const HostSeg& g : s->xin)
        if (cudaMemcpyAsync(g.dev, xh + g.off, g.bytes, cudaMemcpyHostToDevice, split_in ? is : cs) != cudaSuccess)
            return QMM_ERR_CUDA;
    if (split_in && (cudaEventRecord(s->in_done, is) != cudaSuccess || cudaStreamWaitEvent(cs, s->in_done, 0) != cudaSuccess))
        return QMM_ERR_CUDA;
    const qmm_status st = step_launch(s, stream);
    if (st != QMM_OK) return st;
    if (cudaEventRecord(s->kernel_done, cs) != cudaSuccess) return QMM_ERR_CUDA;
    // copy-out: on out_stream after the kernel; the step's next kernel waits for it
    if (split_out && cudaStreamWaitEvent(os, s->kernel_done, 0) != cudaSuccess) return QMM_ERR_CUDA;
    for (const HostSeg& g : s->yout)
        if (cudaMemcpyAsync(yh + g.off, g.dev, g.bytes, cudaMemcpyDeviceToHost, split_out ? os : cs) != cudaSuccess)
            return QMM_ERR_CUDA;
    if (split_out && cudaEventRecord(s->out_done, os) != cudaSuccess) return QMM_ERR_CUDA;
    s->out_pending = split_out;
    return QMM_OK;
}

qmm_status qmm_step_destroy(qmm_step s) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!s || !g_steps.count(s)) return QMM_ERR_BAD_HANDLE;
        g_steps.erase(s);
    }
    cudaDeviceSynchronize();
    free_step(s);
    return QMM_OK;
}

}  // extern "C"
