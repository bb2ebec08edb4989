"""CPU oracle for the ConvRot INT8 layer (test infrastructure, not product).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this package.  It compiles `oracle.c` with the host C compiler into
`oracle/_build/liboracle.so` and exposes numpy-level wrappers.  The CUDA
library never imports it and it never imports the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (host compiler, portable C, no intrinsics)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            F = ctypes.c_float
            sig = {
                "oracle_hadamard": [I, P],
                "oracle_rotate_rows": [P, I64, I64, I, P],
                "oracle_quantize_rows_f64": [P, I64, I64, I64, I, P, P],
                "oracle_quantize_rows_bf16": [P, I64, I64, I64, I, P, P],
                "oracle_lora_merge": [P, I64, I64, I64, P, P, I, F, F, P],
                "oracle_quantize_weight": [P, I64, I64, I64, I, P, P, I, F, F, P, P],
                "oracle_gemm_s32": [P, P, I64, I64, I64, P],
                "oracle_dequant": [P, I64, I64, P, P, P, P],
                "oracle_linear_fwd": [P, I64, I64, P, P, I64, I, P, P, P, P],
                "oracle_prepare_bwd_weight": [P, P, I64, I64, I, P, P],
                "oracle_linear_bwd_x": [P, I64, I64, P, P, I64, I, P, P, P],
                "oracle_embedding_lookup": [P, I64, P, P, I64, I64, I, P, P],
                "oracle_dequant_weight_t": [P, P, I64, I64, I, P],
                "oracle_gemm_bf16": [P, P, I64, I64, I64, P],
                "oracle_linear_fwd_lora": [P, I64, I64, P, P, I64, I, P, P, P, I, F, F, P],
                "oracle_linear_bwd_x_r2": [P, I64, I64, P, P, I64, I, P, P, P],
                "oracle_num_threads": [],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = I
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
            lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def num_threads() -> int:
    return _load().oracle_num_threads()


def hadamard(b: int) -> np.ndarray:
    H = np.empty((b, b), dtype=np.float64)
    _check(_load().oracle_hadamard(b, _p(H)), "hadamard")
    return H


def rotate_rows(x: np.ndarray, b: int) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty_like(x)
    _check(_load().oracle_rotate_rows(_p(x), x.shape[0], x.shape[1], b, _p(out)), "rotate_rows")
    return out


def quantize_rows_f64(x: np.ndarray, b: int):
    x = _c(x, np.float64)
    rows, K = x.shape
    q = np.empty((rows, K), dtype=np.int8)
    s = np.empty(rows, dtype=np.float32)
    _check(_load().oracle_quantize_rows_f64(_p(x), rows, K, K, b, _p(q), _p(s)), "quantize_rows_f64")
    return q, s


def quantize_rows_bf16(x_bits: np.ndarray, b: int):
    x = _c(x_bits, np.uint16)
    rows, K = x.shape
    q = np.empty((rows, K), dtype=np.int8)
    s = np.empty(rows, dtype=np.float32)
    _check(_load().oracle_quantize_rows_bf16(_p(x), rows, K, K, b, _p(q), _p(s)), "quantize_rows_bf16")
    return q, s


def lora_merge(W_bits, A, B, alpha: float, scale: float) -> np.ndarray:
    W = _c(W_bits, np.uint16)
    A = _c(A, np.float32)
    B = _c(B, np.float32)
    N, K = W.shape
    out = np.empty_like(W)
    _check(_load().oracle_lora_merge(_p(W), N, K, K, _p(A), _p(B), A.shape[0], alpha, scale, _p(out)),
           "lora_merge")
    return out


def quantize_weight(W_bits, b: int, A=None, B=None, alpha: float = 1.0, scale: float = 1.0):
    W = _c(W_bits, np.uint16)
    N, K = W.shape
    A = _c(A, np.float32)
    B = _c(B, np.float32)
    rank = 0 if A is None else A.shape[0]
    q = np.empty((N, K), dtype=np.int8)
    s = np.empty(N, dtype=np.float32)
    _check(_load().oracle_quantize_weight(_p(W), N, K, K, b, _p(A), _p(B), rank, alpha, scale, _p(q), _p(s)),
           "quantize_weight")
    return q, s


def gemm_s32(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    A = _c(A, np.int8)
    B = _c(B, np.int8)
    M, K = A.shape
    N = B.shape[0]
    C = np.empty((M, N), dtype=np.int32)
    _check(_load().oracle_gemm_s32(_p(A), _p(B), M, N, K, _p(C)), "gemm_s32")
    return C


def dequant(acc, s_a, s_b, bias_bits=None) -> np.ndarray:
    acc = _c(acc, np.int32)
    M, N = acc.shape
    y = np.empty((M, N), dtype=np.uint16)
    _check(_load().oracle_dequant(_p(acc), M, N, _p(_c(s_a, np.float32)), _p(_c(s_b, np.float32)),
                                  _p(_c(bias_bits, np.uint16)), _p(y)), "dequant")
    return y


def linear_fwd(x_bits, Wq, s_w, b: int, bias_bits=None):
    """Returns (y bf16 bits [M,N], x codes [M,K], s_x [M])."""
    x = _c(x_bits, np.uint16)
    Wq = _c(Wq, np.int8)
    M, K = x.shape
    N = Wq.shape[0]
    y = np.empty((M, N), dtype=np.uint16)
    xq = np.empty((M, K), dtype=np.int8)
    sx = np.empty(M, dtype=np.float32)
    _check(_load().oracle_linear_fwd(_p(x), M, K, _p(Wq), _p(_c(s_w, np.float32)), N, b,
                                     _p(_c(bias_bits, np.uint16)), _p(y), _p(xq), _p(sx)), "linear_fwd")
    return y, xq, sx


def linear_fwd_lora(x_bits, Wq, s_w, b: int, A, B, alpha: float, scale: float, bias_bits=None) -> np.ndarray:
    """Forward with the LoRA branch as a bypass (not merged): bf16 bits [M, N]."""
    x = _c(x_bits, np.uint16)
    Wq = _c(Wq, np.int8)
    A = _c(A, np.float32)
    B = _c(B, np.float32)
    M, K = x.shape
    N = Wq.shape[0]
    rank = A.shape[0]
    y = np.empty((M, N), dtype=np.uint16)
    _check(_load().oracle_linear_fwd_lora(_p(x), M, K, _p(Wq), _p(_c(s_w, np.float32)), N, b,
                                          _p(_c(bias_bits, np.uint16)), _p(A), _p(B), rank, alpha, scale, _p(y)),
           "linear_fwd_lora")
    return y


def prepare_bwd_weight(Wq, s_w, b: int):
    Wq = _c(Wq, np.int8)
    N, K = Wq.shape
    WtQ = np.empty((K, N), dtype=np.int8)
    s_wt = np.empty(K, dtype=np.float32)
    _check(_load().oracle_prepare_bwd_weight(_p(Wq), _p(_c(s_w, np.float32)), N, K, b, _p(WtQ), _p(s_wt)),
           "prepare_bwd_weight")
    return WtQ, s_wt


def linear_bwd_x(dY_bits, WtQ, s_wt, b: int):
    """Returns (dX bf16 bits [M,K], dY codes [M,N], s_dy [M])."""
    dY = _c(dY_bits, np.uint16)
    WtQ = _c(WtQ, np.int8)
    M, N = dY.shape
    K = WtQ.shape[0]
    dX = np.empty((M, K), dtype=np.uint16)
    dyq = np.empty((M, N), dtype=np.int8)
    sdy = np.empty(M, dtype=np.float32)
    _check(_load().oracle_linear_bwd_x(_p(dY), M, N, _p(WtQ), _p(_c(s_wt, np.float32)), K, b, _p(dX),
                                       _p(dyq), _p(sdy)), "linear_bwd_x")
    return dX, dyq, sdy


def dequant_weight_t(Wq, s_w, b: int) -> np.ndarray:
    """W_eff^T = bf16((s_w (.) Wq) R)^T, bf16 bits [K, N] (the bf16-mode backward weight)."""
    Wq = _c(Wq, np.int8)
    N, K = Wq.shape
    out = np.empty((K, N), dtype=np.uint16)
    _check(_load().oracle_dequant_weight_t(_p(Wq), _p(_c(s_w, np.float32)), N, K, b, _p(out)), "dequant_weight_t")
    return out


def gemm_bf16(A_bits, B_bits) -> np.ndarray:
    """bf16(A . B^T) summed in fp64; A [M, K], B [N, K] bf16 bits."""
    A = _c(A_bits, np.uint16)
    B = _c(B_bits, np.uint16)
    M, K = A.shape
    N = B.shape[0]
    C = np.empty((M, N), dtype=np.uint16)
    _check(_load().oracle_gemm_bf16(_p(A), _p(B), M, N, K, _p(C)), "gemm_bf16")
    return C


def linear_bwd_x_bf16(dY_bits, Wq, s_w, b: int) -> np.ndarray:
    """bf16-mode grad_x: dX = bf16(dY . W_eff) with W_eff = bf16((s_w (.) Wq) R)."""
    return gemm_bf16(dY_bits, dequant_weight_t(Wq, s_w, b))


def linear_bwd_x_r2(dY_bits, Wq, s_w, b: int):
    """int8 backward, second reading: returns (dX bf16 bits [M,K], codes of dY*s_w [M,N], s_d [M])."""
    dY = _c(dY_bits, np.uint16)
    Wq = _c(Wq, np.int8)
    M, N = dY.shape
    K = Wq.shape[1]
    dX = np.empty((M, K), dtype=np.uint16)
    dq = np.empty((M, N), dtype=np.int8)
    sd = np.empty(M, dtype=np.float32)
    _check(_load().oracle_linear_bwd_x_r2(_p(dY), M, N, _p(Wq), _p(_c(s_w, np.float32)), K, b, _p(dX), _p(dq),
                                          _p(sd)), "linear_bwd_x_r2")
    return dX, dq, sd


def embedding_lookup(ids, Eq, s_e, b: int):
    """Returns (out bf16 bits [n, D], number of out-of-range ids)."""
    ids = _c(ids, np.int64)
    Eq = _c(Eq, np.int8)
    V, D = Eq.shape
    n = ids.shape[0]
    out = np.empty((n, D), dtype=np.uint16)
    bad = np.zeros(1, dtype=np.int64)
    _check(_load().oracle_embedding_lookup(_p(ids), n, _p(Eq), _p(_c(s_e, np.float32)), V, D, b, _p(out),
                                           _p(bad)), "embedding_lookup")
    return out, int(bad[0])


def bf16_to_f64(h: int) -> float:
    return _load().oracle_bf16_to_f64(h)


def f64_to_bf16(v: float) -> int:
    return _load().oracle_f64_to_bf16(v)
