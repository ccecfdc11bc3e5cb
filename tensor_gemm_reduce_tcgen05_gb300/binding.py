"""ctypes binding of the C ABI in ``include/gemm_rs.h`` and ``include/ag_gemm.h``.

Each function has the C function's name and only marshals arguments.  Device
pointers and streams are passed as Python ints (``tensor.data_ptr()``,
``torch.cuda.Stream.cuda_stream``).  Every step of the computation runs in the
CUDA library.  If the library is missing, :func:`lib` raises instead of
falling back to anything else.

:class:`GemmRS` and :class:`AgGemm` are convenience owners of a handle.  It keeps a torch-allocated
workspace and accepts torch tensors.  PyTorch is used there only for device
memory and the current stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# GEMM_RS_LIBRARY selects another build of this library (the tests load the
# checked build, libgemm_rs_checked.so, that way, in a process of their own).
LIB_PATH = os.environ.get("GEMM_RS_LIBRARY") or os.path.join(_HERE, "libgemm_rs.so")

GEMM_RS_BF16 = 0
GEMM_RS_FP32 = 1

GEMM_RS_OK = 0
GEMM_RS_ERR_ARG = -1
GEMM_RS_ERR_SHAPE = -2
GEMM_RS_ERR_ALIGN = -3
GEMM_RS_ERR_CUDA = -4
GEMM_RS_ERR_TIMEOUT = -5
GEMM_RS_ERR_UNSUPPORTED = -6
GEMM_RS_ERR_WORKSPACE = -7
GEMM_RS_ERR_BOUNDS = -8

GEMM_RS_DEBUG_STALL_PRODUCER = 1
GEMM_RS_DEBUG_SKIP_READY = 2

GEMM_RS_REDUCE_CHAIN = 0
GEMM_RS_REDUCE_LAST_ARRIVER = 1
GEMM_RS_REDUCE_TWO_LEVEL = 2
GEMM_RS_RANKS_DEFAULT = 0
GEMM_RS_RANKS_SEQUENTIAL = 1
GEMM_RS_RANKS_INTERLEAVED = 2

AG_GEMM_DEBUG_SKIP_COPIES = 1

_DTYPES = {"bf16": GEMM_RS_BF16, "fp32": GEMM_RS_FP32}

_lock = threading.Lock()
_lib = None


class GemmRSError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"gemm_rs error {code}: {message}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m tensor_gemm_reduce_tcgen05_gb300.build` (no fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        i64, i32, f32, sz, vp = (ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                                 ctypes.c_void_p)
        u64 = ctypes.c_uint64
        sig = {
            "gemm_rs_workspace_bytes": (sz, [i64, i64, i64, i32]),
            "gemm_rs_create": (i32, [ctypes.POINTER(vp), i64, i64, i64, i32, f32, f32, i32, i32,
                                     i32, vp, sz, vp]),
            "gemm_rs_run": (i32, [vp, vp, vp, vp, vp, vp]),
            "gemm_rs_run_streamed": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "gemm_rs_destroy": (i32, [vp]),
            "gemm_rs_last_error": (ctypes.c_char_p, []),
            "gemm_rs_status": (i32, [vp, vp]),
            "gemm_rs_reset": (i32, [vp, vp]),
            "gemm_rs_schedule": (i64, [i64, i64, i32, i32, i32, i32, i32, i32, vp, i64]),
            "gemm_rs_get_plan": (i32, [vp] + [ctypes.POINTER(i32)] * 8),
            "gemm_rs_set_reduce_mode": (i32, [vp, i32]),
            "gemm_rs_set_schedule": (i32, [vp, i32, i32, i32]),
            "gemm_rs_set_tile_n": (i32, [vp, i32]),
            "gemm_rs_set_tile": (i32, [vp, i32, i32]),
            "gemm_rs_set_timeout_cycles": (i32, [vp, u64]),
            "gemm_rs_set_debug": (i32, [vp, vp, i32]),
            "gemm_rs_reduce_partials": (i32, [vp, i32, vp, vp, i64, i64, i32, f32, f32, i32, vp]),
            "gemm_rs_version": (ctypes.c_char_p, []),
            "gemm_rs_run_noalloc": (i32, [i64, i64, i64, i32, f32, f32, i32, vp, vp, vp, vp, vp]),
            "gemm_rs_noalloc_scratch_bytes": (sz, []),
            "gemm_rs_noalloc_status": (i32, [vp]),
            "ag_gemm_workspace_bytes": (sz, [i64, i64, i64, i32]),
            "ag_gemm_create": (i32, [ctypes.POINTER(vp), i64, i64, i64, i32, f32, i32, vp, sz, vp]),
            "ag_gemm_run": (i32, [vp, vp, vp, vp, vp]),
            "ag_gemm_status": (i32, [vp, vp]),
            "ag_gemm_reset": (i32, [vp, vp]),
            "ag_gemm_destroy": (i32, [vp]),
            "ag_gemm_schedule": (i64, [i64, i64, i32, vp, i64]),
            "ag_gemm_get_plan": (i32, [vp] + [ctypes.POINTER(i32)] * 4),
            "ag_gemm_set_timeout_cycles": (i32, [vp, u64]),
            "ag_gemm_set_debug": (i32, [vp, vp, i32]),
            "ag_gemm_get_shape": (i32, [vp, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                        ctypes.POINTER(i64), ctypes.POINTER(i32),
                                        ctypes.POINTER(i32)]),
            "gemm_rs_get_shape": (i32, [vp, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                        ctypes.POINTER(i64), ctypes.POINTER(i32),
                                        ctypes.POINTER(i32)]),
            "ffn_tp_run": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def gemm_rs_last_error() -> str:
    return lib().gemm_rs_last_error().decode()


def _check(rc: int) -> int:
    if rc < 0:
        raise GemmRSError(rc, gemm_rs_last_error())
    return rc


def gemm_rs_version() -> str:
    return lib().gemm_rs_version().decode()


def gemm_rs_workspace_bytes(M: int, N: int, K: int, W: int) -> int:
    return int(lib().gemm_rs_workspace_bytes(M, N, K, W))


def gemm_rs_create(M, N, K, W, alpha, beta, ab_dtype, c_dtype, y_dtype, workspace,
                   workspace_bytes, stream=0) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(lib().gemm_rs_create(ctypes.byref(h), M, N, K, W, alpha, beta, ab_dtype, c_dtype,
                                y_dtype, workspace, workspace_bytes, stream))
    return h


def gemm_rs_run(h, A, B, C, Y, stream=0) -> None:
    _check(lib().gemm_rs_run(h, A, B, C, Y, stream))


def gemm_rs_run_streamed(h, A_host, B_host, C_host, Y_host, A, B, C, Y, stream, copy_stream) -> None:
    _check(lib().gemm_rs_run_streamed(h, A_host, B_host, C_host, Y_host, A, B, C, Y, stream,
                                      copy_stream))


def gemm_rs_destroy(h) -> None:
    _check(lib().gemm_rs_destroy(h))


def gemm_rs_status(h, stream=0) -> int:
    """Synchronises the stream.  Returns GEMM_RS_OK or GEMM_RS_ERR_TIMEOUT
    (other codes raise)."""
    rc = lib().gemm_rs_status(h, stream)
    if rc in (GEMM_RS_OK, GEMM_RS_ERR_TIMEOUT):
        return rc
    return _check(rc)


def gemm_rs_reset(h, stream=0) -> None:
    _check(lib().gemm_rs_reset(h, stream))


def gemm_rs_schedule(M: int, N: int, W: int, bm: int, bn: int, colgroup: int = 0,
                     rowgroup: int = 0, rank_order: int = 0) -> np.ndarray:
    nM, nN = -(-M // bm), -(-N // bn)
    out = np.zeros((W * nM * nN, 3), dtype=np.int32)
    n = _check(lib().gemm_rs_schedule(M, N, W, bm, bn, colgroup, rowgroup, rank_order,
                                      out.ctypes.data, out.shape[0]))
    return out[:n]


def gemm_rs_get_plan(h) -> dict:
    v = [ctypes.c_int() for _ in range(8)]
    _check(lib().gemm_rs_get_plan(h, *[ctypes.byref(x) for x in v]))
    return dict(zip(("bm", "bn", "stages", "grid", "colgroup", "rowgroup", "rank_order",
                     "reduce_mode"), (x.value for x in v)))


def gemm_rs_set_reduce_mode(h, mode: int) -> None:
    _check(lib().gemm_rs_set_reduce_mode(h, mode))


def gemm_rs_set_schedule(h, colgroup: int = 0, rowgroup: int = 0, rank_order: int = 0) -> None:
    _check(lib().gemm_rs_set_schedule(h, colgroup, rowgroup, rank_order))


def gemm_rs_set_tile_n(h, bn: int) -> None:
    _check(lib().gemm_rs_set_tile_n(h, bn))


def gemm_rs_set_tile(h, bm: int, bn: int) -> None:
    _check(lib().gemm_rs_set_tile(h, bm, bn))


def gemm_rs_set_timeout_cycles(h, cycles: int) -> None:
    _check(lib().gemm_rs_set_timeout_cycles(h, cycles))


def gemm_rs_set_debug(h, record=0, flags: int = 0) -> None:
    _check(lib().gemm_rs_set_debug(h, record, flags))


def gemm_rs_reduce_partials(partials, partial_dtype, C, Y, M, N, W, alpha, beta, y_dtype,
                            stream=0) -> None:
    _check(lib().gemm_rs_reduce_partials(partials, partial_dtype, C, Y, M, N, W, alpha, beta,
                                         y_dtype, stream))


def gemm_rs_run_noalloc(M, N, K, W, alpha, beta, y_dtype, A, B, C, Y, stream=0) -> None:
    """The handle-free entry point whose scratch is a static device array
    (see include/gemm_rs.h): it allocates nothing."""
    _check(lib().gemm_rs_run_noalloc(M, N, K, W, alpha, beta, y_dtype, A, B, C, Y, stream))


def gemm_rs_noalloc_scratch_bytes() -> int:
    """The size of gemm_rs_run_noalloc's static scratch, as compiled into the library."""
    return int(lib().gemm_rs_noalloc_scratch_bytes())


def gemm_rs_noalloc_status(stream=0) -> int:
    """Read and clear the status word of the static scratch (after waiting for
    `stream`): 0, or raises GemmRSError for a device timeout."""
    return _check(lib().gemm_rs_noalloc_status(stream))


def _cuda_device(device):
    """A CUDA torch.device with an index: None or "cuda" mean the current device,
    so that it compares equal to the device of the tensors placed there."""
    import torch
    d = torch.device("cuda") if device is None else torch.device(device)
    if d.type != "cuda":
        raise ValueError(f"the library runs on CUDA devices, not {d}")
    if d.index is None:
        d = torch.device("cuda", torch.cuda.current_device())
    return d


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


class GemmRS:
    """Owns one handle and its workspace (a torch uint8 CUDA tensor).

    Y = sum over r of (alpha * A[r] @ B[r] + beta * C), as W chunks of M/W rows.
    A is bf16 [W, M, K/W], B is bf16 [W, K/W, N], C is bf16 [M, N] (or None when
    beta == 0), and Y is [M, N] in y_dtype.
    """

    def __init__(self, M: int, N: int, K: int, W: int, alpha: float = 1.0, beta: float = 0.0,
                 y_dtype: str = "bf16", device=None, stream=None, tile_n: int | None = None,
                 tile_m: int | None = None):
        import torch
        lib()
        self.M, self.N, self.K, self.W = M, N, K, W
        self.alpha, self.beta, self.y_dtype = alpha, beta, y_dtype
        self.device = _cuda_device(device)
        nbytes = gemm_rs_workspace_bytes(M, N, K, W)
        if nbytes == 0:
            _check(GEMM_RS_ERR_SHAPE)
        with torch.cuda.device(self.device):
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            self.handle = gemm_rs_create(M, N, K, W, alpha, beta, GEMM_RS_BF16, GEMM_RS_BF16,
                                         _DTYPES[y_dtype], self.workspace.data_ptr(), nbytes,
                                         _stream_ptr(stream))
        if tile_m is not None:
            gemm_rs_set_tile(self.handle, tile_m, tile_n if tile_n is not None else 256)
        elif tile_n is not None:
            gemm_rs_set_tile_n(self.handle, tile_n)

    @property
    def plan(self) -> dict:
        return gemm_rs_get_plan(self.handle)

    def new_output(self):
        import torch
        dt = torch.bfloat16 if self.y_dtype == "bf16" else torch.float32
        return torch.empty((self.M, self.N), dtype=dt, device=self.device)

    def run(self, A, B, C=None, Y=None, stream=None):
        """Launch once (asynchronous).  Returns Y."""
        import torch
        for t, name in ((A, "A"), (B, "B")):
            if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != self.device:
                raise ValueError(f"{name} must be a contiguous bf16 tensor on {self.device}")
        if tuple(A.shape) != (self.W, self.M, self.K // self.W):
            raise ValueError(f"A must be [W, M, K/W] = {(self.W, self.M, self.K // self.W)}")
        if tuple(B.shape) != (self.W, self.K // self.W, self.N):
            raise ValueError(f"B must be [W, K/W, N] = {(self.W, self.K // self.W, self.N)}")
        if C is not None and (C.dtype != torch.bfloat16 or not C.is_contiguous()
                              or tuple(C.shape) != (self.M, self.N)):
            raise ValueError("C must be a contiguous bf16 [M, N] tensor")
        if Y is None:
            Y = self.new_output()
        gemm_rs_run(self.handle, A.data_ptr(), B.data_ptr(), 0 if C is None else C.data_ptr(),
                    Y.data_ptr(), _stream_ptr(stream))
        return Y

    def run_streamed(self, A_host, B_host, C_host, Y_host, A, B, C=None, Y=None, stream=None,
                     copy_stream=None):
        """gemm_rs_run_streamed: copy pinned host inputs into A, B (and C) on
        copy_stream, rank by rank, while the kernel on `stream` consumes the
        ranks that have landed; Y goes back into Y_host on `stream`.  Returns
        Y (device)."""
        import torch
        for t, name in ((A_host, "A_host"), (B_host, "B_host"), (Y_host, "Y_host")):
            if t.device.type != "cpu" or not t.is_pinned() or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous pinned host tensor")
        if C_host is not None and (not C_host.is_pinned() or not C_host.is_contiguous()):
            raise ValueError("C_host must be a contiguous pinned host tensor")
        if Y is None:
            Y = self.new_output()
        if copy_stream is None:
            raise ValueError("copy_stream is required (a stream other than `stream`)")
        gemm_rs_run_streamed(self.handle, A_host.data_ptr(), B_host.data_ptr(),
                             0 if C_host is None else C_host.data_ptr(), Y_host.data_ptr(),
                             A.data_ptr(), B.data_ptr(), 0 if C is None else C.data_ptr(),
                             Y.data_ptr(), _stream_ptr(stream), _stream_ptr(copy_stream))
        return Y

    def status(self, stream=None) -> int:
        return gemm_rs_status(self.handle, _stream_ptr(stream))

    def reset(self, stream=None) -> None:
        gemm_rs_reset(self.handle, _stream_ptr(stream))

    def flags_view(self):
        """The tile state words (a view into the workspace), for tests."""
        import torch
        nM, nN = -(-self.M // 128), -(-self.N // 64)
        return self.workspace[256:256 + 3 * 4 * nM * nN].view(torch.int32)

    def close(self) -> None:
        if getattr(self, "handle", None) is not None:
            gemm_rs_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# --------------------------------------------------------------------------- AG+GEMM
def ag_gemm_workspace_bytes(M: int, N: int, K: int, W: int) -> int:
    return lib().ag_gemm_workspace_bytes(M, N, K, W)


def ag_gemm_create(M, N, K, W, alpha, y_dtype, workspace, workspace_bytes, stream=0):
    h = ctypes.c_void_p()
    _check(lib().ag_gemm_create(ctypes.byref(h), M, N, K, W, alpha, y_dtype, workspace,
                                workspace_bytes, stream))
    return h


def ag_gemm_run(h, X, B1, H, stream=0) -> None:
    _check(lib().ag_gemm_run(h, X, B1, H, stream))


def ag_gemm_status(h, stream=0) -> int:
    rc = lib().ag_gemm_status(h, stream)
    if rc not in (GEMM_RS_OK, GEMM_RS_ERR_TIMEOUT):
        _check(rc)
    return rc


def ag_gemm_reset(h, stream=0) -> None:
    _check(lib().ag_gemm_reset(h, stream))


def ag_gemm_destroy(h) -> None:
    _check(lib().ag_gemm_destroy(h))


def ag_gemm_schedule(M: int, N: int, W: int) -> np.ndarray:
    nM, nN = M // 256, -(-N // 256)
    out = np.zeros((W * nM * nN, 3), dtype=np.int32)
    n = _check(lib().ag_gemm_schedule(M, N, W, out.ctypes.data, out.shape[0]))
    return out[:n]


def ag_gemm_get_plan(h) -> dict:
    v = [ctypes.c_int() for _ in range(4)]
    _check(lib().ag_gemm_get_plan(h, *[ctypes.byref(x) for x in v]))
    return dict(zip(("grid", "stages", "slice_rows", "slices"), (x.value for x in v)))


def ag_gemm_set_timeout_cycles(h, cycles: int) -> None:
    _check(lib().ag_gemm_set_timeout_cycles(h, cycles))


def ag_gemm_set_debug(h, record_ptr: int = 0, flags: int = 0) -> None:
    _check(lib().ag_gemm_set_debug(h, record_ptr, flags))


class AgGemm:
    """Owns one AG+GEMM handle and its workspace (a torch uint8 CUDA tensor).

    H[r] = alpha * X @ B1[r] for r = 0 .. W-1, where X ([M, K] bf16) is the
    all-gather of W row chunks and B1 ([W, K, N] bf16) holds the ranks' column
    shards.  H is [W, M, N] in y_dtype.
    """

    def __init__(self, M: int, N: int, K: int, W: int, alpha: float = 1.0, y_dtype: str = "bf16",
                 device=None, stream=None):
        import torch
        lib()
        self.M, self.N, self.K, self.W = M, N, K, W
        self.alpha, self.y_dtype = alpha, y_dtype
        self.device = _cuda_device(device)
        nbytes = ag_gemm_workspace_bytes(M, N, K, W)
        if nbytes == 0:
            lib().ag_gemm_create(ctypes.byref(ctypes.c_void_p()), M, N, K, W, alpha, 0, None, 0, None)
            _check(GEMM_RS_ERR_SHAPE)
        with torch.cuda.device(self.device):
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            self.handle = ag_gemm_create(M, N, K, W, alpha, _DTYPES[y_dtype],
                                         self.workspace.data_ptr(), nbytes, _stream_ptr(stream))

    @property
    def plan(self) -> dict:
        return ag_gemm_get_plan(self.handle)

    def new_output(self):
        import torch
        dt = torch.bfloat16 if self.y_dtype == "bf16" else torch.float32
        return torch.empty((self.W, self.M, self.N), dtype=dt, device=self.device)

    def run(self, X, B1, H=None, stream=None):
        """Launch once (asynchronous).  Returns H."""
        import torch
        for t, name in ((X, "X"), (B1, "B1")):
            if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != self.device:
                raise ValueError(f"{name} must be a contiguous bf16 tensor on {self.device}")
        if tuple(X.shape) != (self.M, self.K):
            raise ValueError(f"X must be [M, K] = {(self.M, self.K)}")
        if tuple(B1.shape) != (self.W, self.K, self.N):
            raise ValueError(f"B1 must be [W, K, N] = {(self.W, self.K, self.N)}")
        if H is None:
            H = self.new_output()
        ag_gemm_run(self.handle, X.data_ptr(), B1.data_ptr(), H.data_ptr(), _stream_ptr(stream))
        return H

    def status(self, stream=None) -> int:
        return ag_gemm_status(self.handle, _stream_ptr(stream))

    def reset(self, stream=None) -> None:
        ag_gemm_reset(self.handle, _stream_ptr(stream))

    def signals_view(self):
        """The W*W chunk signals (a view into the workspace), for tests."""
        import torch
        return self.workspace[256:256 + 4 * self.W * self.W].view(torch.int32)

    def close(self) -> None:
        if getattr(self, "handle", None) is not None:
            ag_gemm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ffn_tp_run(ag_handle, rs_handle, X, B1, H, B2, C, Y, stream=0) -> None:
    """AG+GEMM then GEMM+RS with A = H (device pointers as ints)."""
    _check(lib().ffn_tp_run(ag_handle, rs_handle, X, B1, H, B2, C, Y, stream))
