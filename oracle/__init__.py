"""CPU oracle for the fused GEMM + reduce-scatter path.

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package.  The product path
(the CUDA library and its Python binding) never does.  The oracle shares no
code with the product path.

The arithmetic lives in ``gemm_rs_oracle.c`` (GEMM+RS) and ``ag_gemm_oracle.c``
(AG+GEMM), plain C with fp64 accumulation.
This module compiles it on first use and marshals numpy arrays into it.  The
oracle's header comment states what is computed and which passages of the
pages each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "gemm_rs_oracle.c"), os.path.join(_HERE, "ag_gemm_oracle.c")]
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` and return its path."""
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(s) for s in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-std=c11", "-Wall", "-o", tmp] + _SRCS
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
        vp = ctypes.c_void_p
        lib.oracle_gemm_rs.restype = i32
        lib.oracle_gemm_rs.argtypes = [i32, i64, i64, i64, f32, f32, vp, vp, vp,
                                       i32, vp, i64, vp, vp, i32]
        lib.oracle_chunk_order.restype = i32
        lib.oracle_chunk_order.argtypes = [i32, vp]
        lib.oracle_tile_chunk.restype = i64
        lib.oracle_tile_chunk.argtypes = [i32, i64, i32, vp, i64]
        lib.oracle_gemm_rs_two_level.restype = i32
        lib.oracle_gemm_rs_two_level.argtypes = [i32, i64, i64, i64, f32, f32, vp, vp, vp,
                                                 i32, vp, i64, vp, vp, i32, i32]
        lib.oracle_ag_gemm.restype = i32
        lib.oracle_ag_gemm.argtypes = [i32, i64, i64, i64, f32, vp, vp, i32, vp, i64, vp, vp]
        lib.oracle_ag_chunk_order.restype = i32
        lib.oracle_ag_chunk_order.argtypes = [i32, vp]
        lib.oracle_row_chunk.restype = i32
        lib.oracle_row_chunk.argtypes = [i32, i64, vp, vp]
        lib.oracle_bf16_from_float.restype = None
        lib.oracle_bf16_from_float.argtypes = [vp, vp, i64]
        lib.oracle_float_from_bf16.restype = None
        lib.oracle_float_from_bf16.argtypes = [vp, vp, i64]
        _lib = lib
        return lib


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


def gemm_rs(A: np.ndarray, B: np.ndarray, C: np.ndarray | None, alpha: float, beta: float,
            y_dtype: str = "fp32", rows=None, threads: int | None = None,
            split: int = 0) -> np.ndarray:
    """Y (or the listed rows of Y) of the fused GEMM + reduce-scatter.

    A: uint16 [W, M, K/W] (bf16 bits); B: uint16 [W, K/W, N]; C: uint16 [M, N] or None.
    Returns float32 [rows, N] for y_dtype "fp32", uint16 bf16 bits for "bf16".
    split = 0: the W partials are folded in rank order; 0 < split < W: the two-level
    fold (ranks [0, split) and [split, W) each in rank order, then the two sums).
    """
    A, B = _u16(A), _u16(B)
    W, M, Kpr = A.shape
    W2, Kpr2, N = B.shape
    if W2 != W or Kpr2 != Kpr:
        raise ValueError("A and B shards disagree")
    if C is not None:
        C = _u16(C)
        if C.shape != (M, N):
            raise ValueError("C must be [M, N]")
    if rows is None:
        n_rows, rows_arr = M, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows = rows_arr.shape[0]
    y_bf16 = 1 if y_dtype == "bf16" else 0
    out = np.empty((n_rows, N), dtype=np.uint16 if y_bf16 else np.float32)
    lib = _load()
    rc = lib.oracle_gemm_rs_two_level(
        W, M, N, W * Kpr, ctypes.c_float(alpha), ctypes.c_float(beta),
        A.ctypes.data, B.ctypes.data, None if C is None else C.ctypes.data,
        y_bf16, None if rows_arr is None else rows_arr.ctypes.data, n_rows,
        None if y_bf16 else out.ctypes.data, out.ctypes.data if y_bf16 else None,
        int(threads or 0), int(split))
    if rc != 0:
        raise ValueError(f"oracle_gemm_rs rejected its arguments (rc={rc})")
    return out


def chunk_order(W: int) -> np.ndarray:
    """The rank-offset swizzle: an int32 [W, W] array whose row r lists the
    chunks rank r writes, step by step (remote chunks first, its own last)."""
    out = np.zeros((W, W), dtype=np.int32)
    if W < 1 or _load().oracle_chunk_order(W, out.ctypes.data) != 0:
        raise ValueError(f"oracle_chunk_order rejected W = {W}")
    return out


def tile_chunk(W: int, M: int, BM: int) -> np.ndarray:
    """The chunk each row tile of BM rows goes to (the chunk of its first row),
    as an int32 array of ceil(M/BM) entries."""
    nM = -(-M // BM) if BM > 0 else 0
    out = np.zeros(max(nM, 1), dtype=np.int32)
    n = _load().oracle_tile_chunk(W, M, BM, out.ctypes.data, out.shape[0])
    if n < 0:
        raise ValueError(f"oracle_tile_chunk rejected its arguments (rc={n})")
    return out[:n]


def row_chunk(W: int, M: int):
    """(chunk, row_in_chunk) of every output row."""
    c = np.zeros(M, dtype=np.int32)
    i = np.zeros(M, dtype=np.int64)
    if _load().oracle_row_chunk(W, M, c.ctypes.data, i.ctypes.data) != 0:
        raise ValueError("M must be a multiple of W")
    return c, i


def bf16_from_float(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_bf16_from_float(x.ctypes.data, out.ctypes.data, x.size)
    return out


def float_from_bf16(x: np.ndarray) -> np.ndarray:
    x = _u16(x)
    out = np.empty(x.shape, dtype=np.float32)
    _load().oracle_float_from_bf16(x.ctypes.data, out.ctypes.data, x.size)
    return out


def ag_gemm(X_bits: np.ndarray, B1_bits: np.ndarray, alpha: float, y_dtype: str,
            rows=None, threads=None) -> np.ndarray:
    """H[r] = alpha * X @ B1[r] for every rank r: X is [M][K] and B1 [W][K][N] as
    bf16 bit patterns (uint16).  Returns [W][M][N] (or [W][len(rows)][N]) as
    float32, or as uint16 bf16 bits when y_dtype == "bf16"."""
    X_bits = np.ascontiguousarray(X_bits, dtype=np.uint16)
    B1_bits = np.ascontiguousarray(B1_bits, dtype=np.uint16)
    M, K = X_bits.shape
    W, K2, N = B1_bits.shape
    if K2 != K:
        raise ValueError("X and B1 disagree on K")
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n_rows = M if rows_arr is None else rows_arr.shape[0]
    y_bf16 = 1 if y_dtype == "bf16" else 0
    out = np.zeros((W, n_rows, N), dtype=np.uint16 if y_bf16 else np.float32)
    rc = _load().oracle_ag_gemm(W, M, N, K, ctypes.c_float(alpha), X_bits.ctypes.data,
                                B1_bits.ctypes.data, y_bf16,
                                None if rows_arr is None else rows_arr.ctypes.data, n_rows,
                                None if y_bf16 else out.ctypes.data,
                                out.ctypes.data if y_bf16 else None)
    if rc != 0:
        raise ValueError(f"oracle_ag_gemm rejected its arguments (rc={rc})")
    return out


def ag_chunk_order(W: int) -> np.ndarray:
    """The AG+GEMM consumption order: an int32 [W, W] array whose row r lists
    the chunks of the gathered rows in the order rank r takes them (its own
    first)."""
    out = np.zeros((W, W), dtype=np.int32)
    if W < 1 or _load().oracle_ag_chunk_order(W, out.ctypes.data) != 0:
        raise ValueError(f"oracle_ag_chunk_order rejected W = {W}")
    return out
