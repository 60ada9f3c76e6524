/*
 * qmm -- Q4_K x M-row weight-streaming matmul for one GB300 (sm_103a).
 *
 * What it computes.  y[m, n] = sum_k w[n, k] * x[m, k] for M stacked activation rows
 * x[M, K] (fp16) against an N x K weight matrix stored as Q4_K super-blocks, with fp32
 * output y[M, N].  Each super-block covers 256 consecutive weights of one output row:
 *   bytes 0-1 d (fp16), 2-3 dmin (fp16), 4-15 six-bit (scale, min) pairs of its 8
 *   sub-blocks of 32 (GGUF Q4_K packing), 16-143 four-bit quants q,
 *   w = d * sc_j * q - dmin * m_j.
 * Source: page "Running 4 coding agents on one RTX 3090: a custom CUDA engine for
 * Qwen3.8-27B", section "How parallel decoding works" -- every active stream's next
 * token and its draft tokens are stacked into one row batch (4 agents x 3 = 12 rows),
 * the weights are streamed from memory once per step, and every weight is multiplied
 * against all rows while it is on chip.  The model file it runs is "Q4_K_M" (first
 * paragraph), i.e. GGUF Q4_K super-blocks.
 *
 * Guarantees.
 *  - Every weight byte is read from HBM once per qmm_run, whatever M is.
 *  - Batch invariance: for one handle, row m of y is bit-identical whether x holds that
 *    row alone or together with other rows, at any position (same page, section on
 *    keeping agents fast: a prompt chunked in with other agents' rows gives bit-identical
 *    results to running it alone).  The reduction order depends on (N, K) and the
 *    handle's launch shape only, never on M or on the other rows.
 *  - Accuracy: |y - y_exact| <= 2e-3 * sum_k |w x| + 1e-6 per element for weights whose
 *    dequantised values fit fp16 (|d * 63 * 15| < 65504).  Outputs are not byte-equal to
 *    other implementations (same page, section "Accuracy": arithmetic order differs).
 *
 * Conventions.  All functions return a qmm_status and never abort the process.  Device
 * pointers are plain CUDA device addresses (e.g. torch tensors' data_ptr()); `stream` is a
 * cudaStream_t passed as void* (NULL = legacy default stream).  Every call is ordered on
 * `stream`; qmm_run and qmm_step_launch perform no allocation and no host synchronisation.
 * One handle must not have two runs in flight at once (they share the handle's split-K
 * workspace); runs on one stream are serialised automatically.
 */
#ifndef QMM_H
#define QMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct qmm_handle_s* qmm_handle;

typedef enum {
    QMM_OK = 0,
    QMM_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad option value */
    QMM_ERR_UNSUPPORTED_SHAPE = 2,  /* K % 256 != 0, N or K <= 0, M > m_max */
    QMM_ERR_MISALIGNED = 3,         /* x, y or the weights not 16-byte aligned */
    QMM_ERR_OOM = 4,                /* a device allocation in qmm_create/qmm_step_create failed */
    QMM_ERR_CUDA = 5,               /* a CUDA runtime call or a launch failed */
    QMM_ERR_DEVICE_TIMEOUT = 6,     /* a kernel's bounded wait gave up (sticky, see qmm_get_error) */
    QMM_ERR_BAD_HANDLE = 7,         /* NULL, destroyed or never-created handle */
    QMM_ERR_NO_DEVICE = 8,          /* the current device is not an sm_103 GPU */
    QMM_ERR_SCRATCH_TOO_SMALL = 9   /* qmm_run_noalloc: the shape does not fit its fixed scratch */
} qmm_status;

enum {
    QMM_BACKEND_AUTO = 0,     /* chosen from m_max only (never from a run's M):
                                 m_max <= 16 -> MMA_SYNC (one launch of up to 16 rows, the
                                 faster stream there), else TCGEN05 */
    QMM_BACKEND_MMA_SYNC = 1, /* warp-level mma.sync m16n8k16, 16 rows per launch */
    QMM_BACKEND_TCGEN05 = 2   /* tcgen05.mma with TMEM accumulators, 128 rows per launch */
};

/*
 * Block formats of the weight matrix.  Q4_K is the format of the method; Q6_K and Q8_0 are
 * the other block types of a mixed-quant model file (page "Running 4 coding agents on one
 * RTX 3090", the note on mixed-quant builds) and int8 weights (page "Breaking the limits of
 * Qwen3.8-27B again", its int8 lm_head).  Byte layouts are the GGUF ones:
 *   Q4_K 144 B per 256 weights: d, dmin (fp16), 12 B of 6-bit scales/mins, 128 B of nibbles;
 *   Q6_K 210 B per 256 weights: ql[128], qh[64], 16 int8 scales, d (fp16);
 *        w = d * scale[i/16] * (q - 32) with q the 6-bit quant;
 *   Q8_0 34 B per 32 weights: d (fp16), 32 int8 quants; w = d * q.
 * Q6_K and Q8_0 run on the TCGEN05 backend only.
 */
enum {
    QMM_FORMAT_Q4_K = 0,
    QMM_FORMAT_Q6_K = 1,
    QMM_FORMAT_Q8_0 = 2
};

typedef struct {
    int32_t m_max;        /* largest M any run will pass; >= 1 */
    int32_t backend;      /* QMM_BACKEND_*; fixed for the handle's lifetime */
    int32_t ctas_per_sm;  /* 0 = default; persistent CTAs per SM (part of the reduction order) */
    int32_t host_io;      /* nonzero: also allocate staging buffers for qmm_run_host */
    int32_t format;       /* QMM_FORMAT_* of the blocks passed to qmm_create */
    int32_t wait_limit_us;/* 0 = default (4 s); otherwise the longest time, in microseconds, any
                             device-side wait of the handle's launches between the kernel's own
                             warps and CTAs may take before the launch gives up with
                             QMM_ERR_DEVICE_TIMEOUT.  Exists so that the timeout path can be
                             exercised; a limit far below a launch's duration fails every run. */
} qmm_options;

typedef struct {
    int64_t n, k, m_max;
    int32_t backend;          /* the backend actually used */
    int32_t grid;             /* persistent CTAs per run */
    int64_t units;            /* work units (row tile x super-block column) */
    int64_t rows_per_unit;
    int64_t weight_bytes;     /* bytes of the blocks (Q4_K N*K/256*144): streamed from HBM per run */
    int64_t packed_bytes;     /* bytes of the repacked on-device copy (N padded to a tile) */
    int64_t workspace_bytes;  /* split-K partials + tile tickets */
    int32_t m_per_launch;     /* rows one kernel launch handles; a run of M rows makes
                                 ceil(M / m_per_launch) launches */
    int32_t format;           /* QMM_FORMAT_* of the handle */
} qmm_info;

/* Fill `opt` with defaults: m_max 16, backend auto, ctas_per_sm 0, host_io 0, format Q4_K,
 * wait_limit_us 0. */
void qmm_default_options(qmm_options* opt);

/*
 * Create a handle for an N x K weight matrix in block format opt->format (K a multiple of
 * 256 for every format).
 *  blocks: N rows of blocks, row-major (GGUF order): K/256 Q4_K blocks of 144 bytes, K/256
 *          Q6_K blocks of 210 bytes or K/32 Q8_0 blocks of 34 bytes per row; on the device
 *          if blocks_on_device != 0 (16-byte aligned), else in host memory.  The handle
 *          copies and repacks them into its own device memory; the caller may free
 *          `blocks` once the call returns.  A Q6_K or Q8_0 handle with the MMA_SYNC backend
 *          is an INVALID_ARG.
 *  opt:    NULL for defaults.
 *  stream: the repack is ordered on it; qmm_create synchronises it before returning.
 * Testing: with QMM_SPLITK_PARK=1 in the environment at create, every run and step of the
 * handle takes the rare path of the tcgen05 kernel's split-K sum on each row tile cut
 * between CTAs (the tile's first CTA parks its partial and the last CTA to arrive adds them
 * up), which otherwise happens only when a CTA starts late.  Results are the same bit for
 * bit; launches are slower.  No effect on mma.sync handles.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, OOM, CUDA, NO_DEVICE.
 */
qmm_status qmm_create(qmm_handle* out, const void* blocks, int64_t n, int64_t k,
                      int32_t blocks_on_device, const qmm_options* opt, void* stream);

/*
 * y[M, N] (fp32, device, row-major, 16-byte aligned) = x[M, K] (fp16, device, row-major,
 * 16-byte aligned) times W^T.  M = 0 is a no-op returning QMM_OK.  1 <= M <= m_max.
 * Asynchronous: errors found on the device (a bounded wait timing out) are reported by a
 * later qmm_run or by qmm_get_error.
 * Calls on one handle must be ordered (same stream, or synchronised): they share its split-K
 * workspace.  Runs of different handles may overlap on the GPU (other streams, other
 * kernels): a run never waits for a CTA that might not be resident (mma.sync launches are
 * cooperative; in the tcgen05 kernel no CTA waits for another).
 * Errors: BAD_HANDLE, INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA, DEVICE_TIMEOUT.
 */
qmm_status qmm_run(qmm_handle h, const void* x, int64_t m, float* y, void* stream);

/*
 * Greedy verification head (page "Running 4 coding agents on one RTX 3090", sections "How
 * parallel decoding works" and the greedy acceptance of draft tokens): for every row r < M
 * of x, idx[r] = the column n of the largest y[r][n] and val[r] = that y[r][n], where y is
 * what qmm_run would compute (same arithmetic, same bits); among equal largest values the
 * lowest column wins.  y itself is never formed in memory: each launch folds the rows'
 * maxima into the handle's key buffer and its last finishing warp writes idx and val.
 *  x:    fp16 [M, K], device, row-major, 16-byte aligned.
 *  idx:  int32 [M], device, 4-byte aligned; val: fp32 [M], device, 4-byte aligned.
 * Calls on one handle must be ordered (same stream, or synchronised): they share its key
 * buffer.  Results are undefined if some y[r][n] is NaN.  After a DEVICE_TIMEOUT the handle
 * must be destroyed (its key buffer may hold a partial launch).
 * When to use it: measured on the lm_head shape (151936 x 5120) on one GB300, the fused call
 * is faster than qmm_run followed by a separate reduction of y at M = 1 and 12 (by about
 * 9 us) and takes about as long at M = 64, though it is slower than qmm_run alone; use it
 * whenever only each row's argmax is needed and y itself is not.
 * Errors: BAD_HANDLE, INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA, DEVICE_TIMEOUT.
 */
qmm_status qmm_run_argmax(qmm_handle h, const void* x, int64_t m, int32_t* idx, float* val,
                          void* stream);

/*
 * Stacked-row decode attention over a paged q8_0 KV pool (page "Running 4 coding agents on
 * one RTX 3090", section "How parallel decoding works": the step's rows are every agent's
 * next token and drafts, and each agent's rows attend to that agent's own cache in a shared
 * paged pool of q8_0 entries).  For row r of agent a and query head h, with
 * g = h / (heads / kv_heads):
 *     out[r][h] = softmax over t < row_len[r] of (q[r][h] . k_t / sqrt(128)), times v_t,
 * k_t and v_t being token t of agent a, KV head g.  Head dimension 128, pages of 64 tokens.
 * Every pointer is device memory; nothing is copied from the host, so the call can be
 * captured in a CUDA graph.
 *  pool:       16-byte aligned; record (page P, KV head g) of 17,408 bytes at
 *              (P * kv_heads + g) * 17408:
 *                bytes     0 ..  8191  K quants int8, dim d of token t at
 *                                      t * 128 + 16 * ((d / 16) ^ (2 (t % 4) + (t / 4) % 2)) + d % 16
 *                bytes  8192 ..  8703  K scales fp16 [token 64][dim block 4]
 *                bytes  8704 .. 16895  V quants int8 [dim 128][token 64]
 *                bytes 16896 .. 17407  V scales fp16 [dim block 4][token 64]
 *              element = scale of its 32-dim block * quant.
 *  page_table: int32 [agents][max_pages]: token t of agent a is in page page_table[a][t / 64],
 *              slot t % 64.  An entry outside [0, pool_pages) sets *err_word |= 2 and the
 *              run of pages holding it is skipped.
 *  agent_rows: int32 [agents + 1], non-decreasing: agent a's rows are agent_rows[a] ..
 *              agent_rows[a + 1] - 1 (an agent may have none).
 *  row_len:    int32 [rows]: 1 <= row_len[r] <= max_pages * 64.
 *  q:          fp16 [rows][heads][128], 16-byte aligned; out: fp32 [rows][heads][128], 16-byte
 *              aligned.
 *  An agent's queries per KV head (its rows x heads / kv_heads) are taken 24 at a time, each
 *  group of 32 a pass over the agent's pages.  A row length out of range sets
 *  *err_word |= 4, and the agent's rows' outputs are zero.
 *  workspace:  16-byte aligned, at least qmm_attn_workspace_bytes(dims, rows) bytes (fixed by
 *              dims and rows); used by this call until its kernels finish.
 *  err_word:   device-visible int, or-ed with 1 if a device-side wait ran out, 2 or 4 as
 *              above; the caller zeroes it and reads it after synchronising.
 * Errors: INVALID_ARG, MISALIGNED, SCRATCH_TOO_SMALL, CUDA.
 */
typedef struct {
    int32_t heads;       /* query heads, a multiple of kv_heads */
    int32_t kv_heads;
    int32_t agents;      /* rows of page_table */
    int32_t max_pages;   /* columns of page_table */
    int64_t pool_pages;  /* pages in the pool */
    int32_t max_agent_rows;  /* upper bound on any agent's rows in a call, or 0 (= the call's
                                rows): sizes the workspace and the grid; an agent above it
                                sets *err_word |= 4 */
    int32_t reserved;        /* zero */
} qmm_attn_dims;

/* Workspace bytes of qmm_attn_decode for these dims and at most `rows` rows (1 .. 2^24),
 * with at most min(rows, dims->max_agent_rows if > 0) rows in one agent: errors INVALID_ARG. */
qmm_status qmm_attn_workspace_bytes(const qmm_attn_dims* dims, int64_t rows, int64_t* bytes);

qmm_status qmm_attn_decode(const qmm_attn_dims* dims, const void* pool, const int32_t* page_table,
                           const int32_t* agent_rows, const int32_t* row_len, const void* q, int64_t rows,
                           float* out, void* workspace, int64_t workspace_bytes, int* err_word,
                           void* stream);

/*
 * Same as qmm_run with x and y in host memory (pinned memory gives asynchronous
 * copies): copies x to the handle's staging buffer, runs, copies y back, all on `stream`.
 * The caller must synchronise `stream` before reading y.  Needs opt.host_io at create.
 */
qmm_status qmm_run_host(qmm_handle h, const void* x_host, int64_t m, float* y_host,
                        void* stream);

/* Sticky device error word of the handle (synchronises the device to read it). */
qmm_status qmm_get_error(qmm_handle h);

/* Shape and sizing facts of a handle. */
qmm_status qmm_get_info(qmm_handle h, qmm_info* info);

/* Free the handle and its device memory (synchronises the device first).  Destroying a
 * handle twice, or using it afterwards, returns BAD_HANDLE. */
qmm_status qmm_destroy(qmm_handle h);

/* Static text for a status code. */
const char* qmm_status_str(qmm_status s);

/*
 * A decode step ("How parallel decoding works" on the RTX 3090 engine page: every weight
 * matrix of the step is streamed once, all stacked rows multiplied against it): `count` runs
 * (handle i: x_i -> y_i, all with the same M), set up once and replayed with one call.
 *  flags = 0:                    dependent runs: run i reads x_i only after run i-1 has
 *                                finished (as a layer waits for the one before), so x_i may be
 *                                run i-1's output.  Results are bit-identical to the same runs
 *                                issued one by one.  The runs are recorded into a CUDA graph,
 *                                consecutive kernels linked by programmatic dependent launch
 *                                (the weights of run i stream in while run i-1 ends).
 *  flags = QMM_STEP_PERSISTENT:  dependent runs as one persistent kernel ("How parallel
 *                                decoding works": one persistent kernel, no per-layer
 *                                launches), when every handle is a TCGEN05 handle of one block
 *                                format and M <= 64 (the graph otherwise): each matrix is cut
 *                                into the pieces a single run of its handle would use (so the
 *                                results are again bit-identical to single runs), the weights
 *                                stream in continuously across matrix boundaries, and a CTA
 *                                loads x_i only once every CTA has written its part of run
 *                                i-1's output (device-scope counters, bounded waits).  A handle
 *                                may appear more than once.  Measured on one GB300 with the
 *                                full 64-layer stack at M = 12 it is the fastest dependent
 *                                step (5.07-5.10 ms, against 5.30-5.32 for the graph of the
 *                                same handles and 5.37-5.40 for a graph of MMA_SYNC runs); at
 *                                M = 64 it is about even with the graph.  It is opt-in
 *                                because the launch is cooperative and holds every SM for the
 *                                whole step.
 *  flags = QMM_STEP_INDEPENDENT: the caller guarantees that no x_i is written by a run of
 *                                the step.  When every handle has the same backend and block
 *                                format and M fits one launch (M <= 16 for MMA_SYNC handles,
 *                                M <= 128 for TCGEN05 handles), one persistent kernel streams
 *                                all the matrices: their unit sequences are concatenated and
 *                                cut into one piece per CTA, so only CTA boundaries split a
 *                                row tile.  Each handle may then appear at most once.  The split-K order
 *                                differs from that of single runs, so results agree with them
 *                                within rounding (not bit for bit); a row's result still does
 *                                not depend on M.
 *  QMM_STEP_GRAPH:               use the CUDA graph even for an independent step (it takes
 *                                precedence over the other flags).
 *  qmm_step_create: builds the step (synchronous; `stream` is not used).
 *  qmm_step_launch: replays it on `stream` (asynchronous, no allocation).
 * The x_i/y_i pointers are baked in; the handles must outlive the step, and a step must not
 * run concurrently with another run of the same handles.
 * Errors: INVALID_ARG (also a repeated handle in a persistent step, unknown flags),
 * BAD_HANDLE, MISALIGNED, UNSUPPORTED_SHAPE (M > a handle's m_max), OOM, CUDA; a launch after
 * a device-side timeout of the persistent kernel returns DEVICE_TIMEOUT.
 */
enum {
    QMM_STEP_INDEPENDENT = 1u,
    QMM_STEP_GRAPH = 2u,
    QMM_STEP_PERSISTENT = 4u
};
typedef struct qmm_step_s* qmm_step;
qmm_status qmm_step_create(qmm_step* out, int32_t count, const qmm_handle* handles,
                           const void* const* xs, float* const* ys, int64_t m, uint32_t flags,
                           void* stream);
qmm_status qmm_step_launch(qmm_step s, void* stream);
qmm_status qmm_step_destroy(qmm_step s);

/*
 * A step with its activations and outputs in host memory (the end-to-end form of "How
 * parallel decoding works": one step's rows in, every matrix's products out).
 *  x_host: every matrix's activations, matrix after matrix in the step's order, each
 *          x_i [M, K_i] fp16 row-major (sum over i of M*K_i*2 bytes), read only.
 *  y_host: receives every output, y_i [M, N_i] fp32 row-major in the same order (sum of
 *          M*N_i*4 bytes).
 * Copies x_host into the step's device x_i, replays the step on `stream`, and copies the y_i
 * back to y_host.
 *  in_stream:  NULL (or `stream`): the copy-in is ordered on `stream` before the kernel.
 *              Otherwise it runs on in_stream once the step's last kernel has finished
 *              reading the x_i, and the kernel waits for it (the call orders both with
 *              events; a launch of the step captured into a CUDA graph is not tracked, so
 *              order that graph's launches with the copy-in yourself).
 *  out_stream: NULL (or `stream`): the copy-out is ordered on `stream` after the kernel, and
 *              y_host is complete once `stream` has been synchronised.  Otherwise it runs on
 *              out_stream after the kernel, y_host is complete once out_stream has been
 *              synchronised, and the step's next launch (host-buffer or not) waits for it
 *              before it rewrites the y_i.
 * So two steps over two sets of device buffers, called alternately on one `stream` with
 * their copies on two other streams, overlap one step's copies with the other's kernel.
 * Calls on one step must be ordered on `stream`.  Device ranges that continue one another
 * (buffers laid out as one slab in step order) move as one copy.  The host buffers should be
 * page-locked (cudaHostAlloc / cudaHostRegister), or the copies are not asynchronous.
 * Where an x_i is also written by a run of the step (a dependent step whose x_i aliases an
 * earlier y_j), it receives the copied bytes first and that run's output after, as in
 * qmm_step_launch.  Ownership: the caller keeps the host buffers and the streams; nothing is
 * allocated.
 * Errors: BAD_HANDLE, INVALID_ARG (a null buffer), CUDA, and those of qmm_step_launch.
 */
qmm_status qmm_step_launch_host(qmm_step s, const void* x_host, float* y_host, void* stream,
                                void* in_stream, void* out_stream);

/*
 * A run that allocates nothing (no counterpart on the pages: it exists for callers that
 * cannot call cudaMalloc where they need the matmul -- a framework whose memory pool owns the
 * device, code that must not synchronise the device, a plugin with a fixed memory budget).
 *  blocks: the N x K weight matrix as Q4_K super-blocks, row-major (GGUF order), on the
 *          device, 16-byte aligned; x [M, K] fp16 and y [M, N] fp32 on the device, 16-byte
 *          aligned.  Computes the same product as qmm_run with the mma.sync kernel.
 *  Scratch: every call packs the weights, the split-K workspace and the tile tickets into one
 *          fixed 48 MiB device array of the library (held by every GPU that loads it, until the
 *          process exits); the packed weights plus the workspace must fit, which allows Q4_K
 *          matrices up to about 40 MiB -- larger shapes return QMM_ERR_SCRATCH_TOO_SMALL.
 *          M may be any size (16 rows per launch).
 *  The first call on each device sets up the kernel (function attributes), so it must come
 *  before any stream capture.  Calls share the array and keep its last contents (each call
 *  clears what must start at zero): calls that overlap on the GPU race -- serialise them.
 *  A device-side wait that gives up (see QMM_ERR_DEVICE_TIMEOUT) cannot be returned by the
 *  call, which returns before its kernels run: instead such a call leaves its whole y NaN.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, NO_DEVICE, SCRATCH_TOO_SMALL, CUDA.
 */
qmm_status qmm_run_noalloc(const void* blocks, int64_t n, int64_t k, const void* x, int64_t m, float* y,
                           void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
