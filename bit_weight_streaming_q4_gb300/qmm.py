"""ctypes binding of libqmm (include/qmm.h): argument marshalling only.

Every step of the matmul runs in the library's CUDA kernels.  There is no fallback: if
libqmm.so is missing or the GPU is not an sm_103 device, creating a handle raises.
PyTorch is used only for device memory and streams (tensors' data_ptr(), the current
stream's handle).
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqmm.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "qmm.h")

QMM_OK = 0
STATUS = {0: "QMM_OK", 1: "QMM_ERR_INVALID_ARG", 2: "QMM_ERR_UNSUPPORTED_SHAPE",
          3: "QMM_ERR_MISALIGNED", 4: "QMM_ERR_OOM", 5: "QMM_ERR_CUDA",
          6: "QMM_ERR_DEVICE_TIMEOUT", 7: "QMM_ERR_BAD_HANDLE", 8: "QMM_ERR_NO_DEVICE",
          9: "QMM_ERR_SCRATCH_TOO_SMALL"}
BACKEND_AUTO, BACKEND_MMA_SYNC, BACKEND_TCGEN05 = 0, 1, 2
FORMAT_Q4_K, FORMAT_Q6_K, FORMAT_Q8_0 = 0, 1, 2


class QmmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class Options(ctypes.Structure):
    _fields_ = [("m_max", ctypes.c_int32), ("backend", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("host_io", ctypes.c_int32),
                ("format", ctypes.c_int32), ("wait_limit_us", ctypes.c_int32)]


class Info(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("k", ctypes.c_int64), ("m_max", ctypes.c_int64),
                ("backend", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("units", ctypes.c_int64), ("rows_per_unit", ctypes.c_int64),
                ("weight_bytes", ctypes.c_int64), ("packed_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("m_per_launch", ctypes.c_int32),
                ("format", ctypes.c_int32)]


class AttnDims(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32), ("agents", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("pool_pages", ctypes.c_int64), ("max_agent_rows", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_lib = None


def header_functions() -> list[str]:
    """Names of the functions declared in include/qmm.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:qmm_status|void|const char\*)\s+(qmm_\w+)\s*\(",
                                 text, flags=re.M)))


def load(path: str = LIB_PATH):
    """Load libqmm.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libqmm.so not built ({path}); run "
                           "`python -m bit_weight_streaming_q4_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "qmm_default_options": (None, [ctypes.POINTER(Options)]),
        "qmm_create": (ctypes.c_int, [ctypes.POINTER(vp), vp, i64, i64, i32,
                                      ctypes.POINTER(Options), vp]),
        "qmm_run": (ctypes.c_int, [vp, vp, i64, vp, vp]),
        "qmm_run_host": (ctypes.c_int, [vp, vp, i64, vp, vp]),
        "qmm_run_argmax": (ctypes.c_int, [vp, vp, i64, vp, vp, vp]),
        "qmm_get_error": (ctypes.c_int, [vp]),
        "qmm_get_info": (ctypes.c_int, [vp, ctypes.POINTER(Info)]),
        "qmm_destroy": (ctypes.c_int, [vp]),
        "qmm_status_str": (ctypes.c_char_p, [ctypes.c_int]),
        "qmm_step_create": (ctypes.c_int, [ctypes.POINTER(vp), i32, ctypes.POINTER(vp),
                                           ctypes.POINTER(vp), ctypes.POINTER(vp), i64, ctypes.c_uint32, vp]),
        "qmm_step_launch": (ctypes.c_int, [vp, vp]),
        "qmm_step_launch_host": (ctypes.c_int, [vp, vp, vp, vp, vp, vp]),
        "qmm_step_destroy": (ctypes.c_int, [vp]),
        "qmm_run_noalloc": (ctypes.c_int, [vp, i64, i64, vp, i64, vp, vp]),
        "qmm_attn_workspace_bytes": (ctypes.c_int, [ctypes.POINTER(AttnDims), i64, ctypes.POINTER(i64)]),
        "qmm_attn_decode": (ctypes.c_int, [ctypes.POINTER(AttnDims), vp, vp, vp, vp, vp, i64, vp, vp, i64,
                                           vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != QMM_OK:
        raise QmmError(status, what)


def _ptr(t) -> int:
    """Device or host address of a torch tensor, a numpy array, or an int."""
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(type(t))


def current_stream() -> int:
    import torch
    return torch.cuda.current_stream().cuda_stream


def default_options(m_max: int = 16, backend: int = BACKEND_AUTO, ctas_per_sm: int = 0,
                    host_io: bool = False, format: int = FORMAT_Q4_K, wait_limit_us: int = 0) -> Options:
    o = Options()
    load().qmm_default_options(ctypes.byref(o))
    o.m_max, o.backend, o.ctas_per_sm, o.host_io = m_max, backend, ctas_per_sm, int(host_io)
    o.format, o.wait_limit_us = format, wait_limit_us
    return o


class Qmm:
    """One N x K weight matrix resident on the GPU.

    blocks: GGUF-ordered blocks of `format` as uint8 ([N, K/256, 144] Q4_K, [N, K/256, 210]
    Q6_K, [N, K/32, 34] Q8_0), a torch CUDA tensor (device) or a numpy array / CPU tensor
    (host)."""

    def __init__(self, blocks, n: int, k: int, m_max: int = 16, backend: int = BACKEND_AUTO,
                 ctas_per_sm: int = 0, host_io: bool = False, stream: int | None = None,
                 format: int = FORMAT_Q4_K, wait_limit_us: int = 0):
        lib = load()
        on_dev = bool(getattr(blocks, "is_cuda", False))
        self._h = ctypes.c_void_p()
        opt = default_options(m_max, backend, ctas_per_sm, host_io, format, wait_limit_us)
        st = current_stream() if stream is None else stream
        _check(lib.qmm_create(ctypes.byref(self._h), _ptr(blocks), n, k, int(on_dev),
                              ctypes.byref(opt), st), "qmm_create")
        self.n, self.k, self.m_max = n, k, m_max

    @property
    def handle(self) -> int:
        return self._h.value

    def info(self) -> Info:
        i = Info()
        _check(load().qmm_get_info(self._h, ctypes.byref(i)), "qmm_get_info")
        return i

    def run(self, x, y, m: int | None = None, stream: int | None = None) -> None:
        """y[:m] = x[:m] @ W^T on the GPU (x fp16 [m, K], y fp32 [m, N], device)."""
        if m is None:
            m = x.shape[0]
        st = current_stream() if stream is None else stream
        _check(load().qmm_run(self._h, _ptr(x), m, _ptr(y), st), "qmm_run")

    def run_argmax(self, x, idx, val, m: int | None = None, stream: int | None = None) -> None:
        """idx[:m], val[:m] = the column and value of each row's largest entry of x[:m] @ W^T
        (lowest column on ties), without forming the product (idx int32, val fp32, device)."""
        if m is None:
            m = x.shape[0]
        st = current_stream() if stream is None else stream
        _check(load().qmm_run_argmax(self._h, _ptr(x), m, _ptr(idx), _ptr(val), st), "qmm_run_argmax")

    def run_host(self, x_host, y_host, m: int, stream: int | None = None) -> None:
        st = current_stream() if stream is None else stream
        _check(load().qmm_run_host(self._h, _ptr(x_host), m, _ptr(y_host), st), "qmm_run_host")

    def error(self) -> int:
        return load().qmm_get_error(self._h)

    def close(self) -> None:
        if self._h and self._h.value:
            _check(load().qmm_destroy(self._h), "qmm_destroy")
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def run_noalloc(blocks, n: int, k: int, x, y, m: int | None = None, stream: int | None = None) -> None:
    """y[:m] = x[:m] @ W^T from raw Q4_K blocks on the device, without any allocation: the
    library packs the weights into its fixed scratch array (see qmm_run_noalloc in qmm.h)."""
    if m is None:
        m = x.shape[0]
    st = current_stream() if stream is None else stream
    _check(load().qmm_run_noalloc(_ptr(blocks), n, k, _ptr(x), m, _ptr(y), st), "qmm_run_noalloc")


STEP_INDEPENDENT = 1   # no x of the step is written by one of its runs: runs may overlap
STEP_GRAPH = 2         # force the CUDA-graph implementation
STEP_PERSISTENT = 4    # dependent runs as one persistent kernel (tcgen05 handles, M <= 64)


class Step:
    """A list of runs set up once and replayed as one launch (see qmm_step_create): one
    persistent kernel for mma.sync handles, else a CUDA graph of runs."""

    def __init__(self, mats: list[Qmm], xs, ys, m: int, stream: int | None = None, flags: int = 0):
        lib = load()
        n = len(mats)
        H = (ctypes.c_void_p * n)(*[q.handle for q in mats])
        X = (ctypes.c_void_p * n)(*[_ptr(x) for x in xs])
        Y = (ctypes.c_void_p * n)(*[_ptr(y) for y in ys])
        self._s = ctypes.c_void_p()
        st = current_stream() if stream is None else stream
        _check(lib.qmm_step_create(ctypes.byref(self._s), n, H, X, Y, m, flags, st), "qmm_step_create")
        self._keep = (mats, xs, ys)

    def launch(self, stream: int | None = None) -> None:
        st = current_stream() if stream is None else stream
        _check(load().qmm_step_launch(self._s, st), "qmm_step_launch")

    def launch_host(self, x_host, y_host, stream: int | None = None, in_stream: int | None = None,
                    out_stream: int | None = None) -> None:
        """Copy every x_i in from x_host (one slab, step order), run, copy every y_i out to
        y_host (qmm_step_launch_host): y_host is complete once `out_stream` (if given, else
        `stream`) is synchronised."""
        st = current_stream() if stream is None else stream
        _check(load().qmm_step_launch_host(self._s, _ptr(x_host), _ptr(y_host), st, in_stream or 0,
                                           out_stream or 0), "qmm_step_launch_host")

    def close(self) -> None:
        if self._s and self._s.value:
            _check(load().qmm_step_destroy(self._s), "qmm_step_destroy")
            self._s = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


ATTN_RECORD_BYTES = 17408
ATTN_QUERY_TILE = 24  # queries per (agent, KV head) that one pass over the agent's pages serves


def attn_workspace_bytes(dims: AttnDims, rows: int) -> int:
    n = ctypes.c_int64()
    _check(load().qmm_attn_workspace_bytes(ctypes.byref(dims), int(rows), ctypes.byref(n)),
           "qmm_attn_workspace_bytes")
    return n.value


def attn_decode(pool, page_table, agent_rows, row_len, q, out, kv_heads: int, stream: int | None = None,
                workspace=None, err=None, max_agent_rows: int = 0):
    """Stacked-row decode attention over a paged q8_0 KV pool (qmm_attn_decode in qmm.h).

    pool: uint8 CUDA tensor of 17,408-byte records; page_table: int32 CUDA tensor [agents,
    max_pages]; agent_rows: int32 CUDA tensor [agents + 1]; row_len: int32 CUDA tensor [rows];
    q: fp16 CUDA tensor [rows, heads, 128]; out: fp32 CUDA tensor [rows, heads, 128].  The
    workspace and the error word are allocated unless given; returns the error word (a CUDA
    int32 tensor of one element, nonzero after the launch if the device reported a failure).
    max_agent_rows: an upper bound on any agent's rows (0: the call's rows), which sizes the
    workspace and the grid."""
    import torch
    lib = load()
    dims = AttnDims(int(q.shape[1]), int(kv_heads), int(page_table.shape[0]), int(page_table.shape[1]),
                    int(pool.numel() // (kv_heads * ATTN_RECORD_BYTES)), int(max_agent_rows))
    nbytes = attn_workspace_bytes(dims, int(q.shape[0]))
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=q.device)
    st = current_stream() if stream is None else stream
    _check(lib.qmm_attn_decode(ctypes.byref(dims), _ptr(pool), _ptr(page_table), _ptr(agent_rows), _ptr(row_len),
                               _ptr(q), int(q.shape[0]), _ptr(out), _ptr(workspace), workspace.numel(), _ptr(err), st),
           "qmm_attn_decode")
    return err
