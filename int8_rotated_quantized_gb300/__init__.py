"""Python binding of libconvrot (the ConvRot INT8 linear layer on sm_103a).

Thin marshalling only: every function below checks tensor dtypes/devices,
allocates outputs with PyTorch when the caller gives none, and calls the C
entry point of the same name on the current CUDA stream.  All arithmetic runs
in the library's CUDA kernels.  There is no fallback: if the shared library
has not been built (see `_build.build()`), importing works but every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

_lock = threading.Lock()
_libs = {}               # variant -> loaded CDLL
_variant = "release"     # "release" or "checked" (bounds-checked kernels)

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_INDEX, ERR_BOUNDS = range(7)


class ConvRotError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def library_path(variant: str = "release") -> str:
    return _build.CHECKED_LIB_PATH if variant == "checked" else _build.LIB_PATH


def select_library(variant: str) -> str:
    """Route every call of this module to the release library or to its checked
    variant (every kernel access checked against its tensor, CONVROT_ERR_BOUNDS on
    a violation).  Returns the previous choice."""
    global _variant
    if variant not in ("release", "checked"):
        raise ValueError(variant)
    with _lock:
        prev, _variant = _variant, variant
    return prev


def lib():
    """The loaded shared library (ctypes), with argument types declared."""
    with _lock:
        _lib = _libs.get(_variant)
        if _lib is None:
            path = library_path(_variant)
            if not os.path.exists(path):
                raise RuntimeError(f"libconvrot is not built ({path} missing); call "
                                   "int8_rotated_quantized_gb300._build.build() first")
            L = ctypes.CDLL(path)
            P, I64, I, F, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            sig = {
                "convrot_version": ([], I),
                "convrot_get_error": ([P], I),
                "convrot_quantize_weight": ([P, I64, I64, I64, I, P, P, I, F, F, P, P, P], I),
                "convrot_quantize_activation": ([P, I64, I64, I64, I, P, P, P], I),
                "convrot_gemm_dequant": ([P, P, I64, I64, P, P, I64, P, P, P], I),
                "convrot_act_workspace_bytes": ([I64, I64], S),
                "convrot_linear_fwd": ([P, I64, I64, P, P, I64, I, P, P, P, S, P], I),
                "convrot_bwd_weight_workspace_bytes": ([I64, I64], S),
                "convrot_prepare_bwd_weight": ([P, P, I64, I64, I, P, P, P, S, P], I),
                "convrot_linear_bwd_x": ([P, I64, I64, P, P, I64, I, P, P, S, P], I),
                "convrot_embedding_lookup": ([P, I64, P, P, I64, I64, I, P, P], I),
                "convrot_dequant_weight_t": ([P, P, I64, I64, I, P, P], I),
                "convrot_linear_workspace_bytes": ([I64, I64, I64], S),
                "convrot_linear_lora_workspace_bytes": ([I64, I64, I64], S),
                "convrot_linear_fwd_lora": ([P, I64, I64, P, P, I64, I, P, P, P, I, F, F, P, P, S, P], I),
                "convrot_widen_codes": ([P, I64, P, P], I),
                "convrot_gemm_dequant_w16": ([P, P, I64, I64, P, P, I64, P, P, P], I),
                "convrot_gemm_bf16": ([P, I64, I64, P, I64, P, P], I),
                "convrot_bwd_x_r2_workspace_bytes": ([I64, I64, I64], S),
                "convrot_linear_bwd_x_r2": ([P, I64, I64, P, P, I64, I, P, P, S, P], I),
                "convrot_bwd_x_bf16_workspace_bytes": ([I64, I64], S),
                "convrot_linear_bwd_x_bf16": ([P, I64, I64, P, P, I64, I, P, P, S, P], I),
                "convrot_gemm_s32_workspace_bytes": ([I64, I64], S),
                "convrot_gemm_s32": ([P, P, I64, I64, I64, P, P, S, P], I),
                "convrot_linear_fwd_noalloc": ([P, I64, I64, P, P, I64, I, P, P, P], I),
                "convrot_linear_fwd_noalloc_max_bytes": ([], S),
                "convrot_selftest_wait_timeout": ([ctypes.c_uint64, P], I),
                "convrot_selftest_bounds_flag": ([P], I),
                "convrot_probe_mma_s8_rate": ([I, P, S, ctypes.POINTER(ctypes.c_double), P], I),
                "convrot_selftest_gemm_fault": ([I, P, P, I64, I64, P, P, I64, P, ctypes.c_uint64, I64, I, P], I),
            }
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            L.convrot_status_string.argtypes = [I]
            L.convrot_status_string.restype = ctypes.c_char_p
            _libs[_variant] = _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().convrot_status_string(status).decode()
    except RuntimeError:
        return f"status {status}"


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, where: str):
    if rc != OK:
        raise ConvRotError(rc, where)


def _need(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _workspace(nbytes: int, device, workspace=None):
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


def convrot_version() -> int:
    return lib().convrot_version()


def convrot_get_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status."""
    return lib().convrot_get_error(_stream(stream))


def convrot_quantize_weight(W, block, lora_A=None, lora_B=None, alpha=1.0, scale=1.0, Wq=None, scale_w=None,
                            stream=None):
    """Rotate + quantize the rows of W (bf16 [N, K]); optional LoRA merge first.
    Returns (Wq int8 [N, K], scale_w fp32 [N])."""
    _need(W, torch.bfloat16, "W", 2)
    N, K = W.shape
    if (lora_A is None) != (lora_B is None):
        raise ValueError("lora_A and lora_B go together")
    rank = 0
    if lora_A is not None:
        _need(lora_A, torch.float32, "lora_A", 2)
        _need(lora_B, torch.float32, "lora_B", 2)
        rank = lora_A.shape[0]
        if lora_A.shape[1] != K or lora_B.shape != (N, rank):
            raise ValueError("LoRA shapes must be A [rank, K], B [N, rank]")
    if Wq is None:
        Wq = torch.empty((N, K), dtype=torch.int8, device=W.device)
    if scale_w is None:
        scale_w = torch.empty((N,), dtype=torch.float32, device=W.device)
    _check(lib().convrot_quantize_weight(_ptr(W), N, K, K, block, _ptr(lora_A), _ptr(lora_B), rank, alpha, scale,
                                         _ptr(Wq), _ptr(scale_w), _stream(stream)), "convrot_quantize_weight")
    return Wq, scale_w


def shard_rows(M: int, world: int, rank: int):
    """Token rows [start, start + count) of one data-parallel rank.  Every step of the
    layer is independent per token row (the rotation and the scale act within a row,
    the GEMM's rows are independent), so ranks run their shards with no exchange."""
    if world < 1 or not 0 <= rank < world or M < 0:
        raise ValueError("bad shard")
    base, extra = divmod(M, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def convrot_quantize_activation(x, block, xq=None, scale_x=None, stream=None):
    """Rotate + quantize the rows of x (bf16 [M, K]).  Returns (codes as fp16 [M, K], scale fp32 [M])."""
    _need(x, torch.bfloat16, "x", 2)
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.float16, device=x.device)
    if scale_x is None:
        scale_x = torch.empty((M,), dtype=torch.float32, device=x.device)
    _check(lib().convrot_quantize_activation(_ptr(x), M, K, K, block, _ptr(xq), _ptr(scale_x), _stream(stream)),
           "convrot_quantize_activation")
    return xq, scale_x


def convrot_gemm_dequant(xq, scale_x, Wq, scale_w, bias=None, y=None, stream=None):
    """y = bf16(float(xq . Wq^T) * scale_x[m] * scale_w[n] + bias[n])."""
    _need(xq, torch.float16, "xq", 2)
    _need(Wq, torch.int8, "Wq", 2)
    _need(scale_x, torch.float32, "scale_x", 1)
    _need(scale_w, torch.float32, "scale_w", 1)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = xq.shape
    N = Wq.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    _check(lib().convrot_gemm_dequant(_ptr(xq), _ptr(scale_x), M, K, _ptr(Wq), _ptr(scale_w), N, _ptr(bias), _ptr(y),
                                      _stream(stream)), "convrot_gemm_dequant")
    return y


def convrot_widen_codes(q, out=None, stream=None):
    """int8 codes -> fp16 values of the same integers (same shape)."""
    _need(q, torch.int8, "q", q.dim())
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float16, device=q.device)
    _check(lib().convrot_widen_codes(_ptr(q), q.numel(), _ptr(out), _stream(stream)), "convrot_widen_codes")
    return out


def convrot_gemm_dequant_w16(xq, scale_x, Wq16, scale_w, bias=None, y=None, stream=None):
    """convrot_gemm_dequant with fp16-held weight codes Wq16 [N, K] (from convrot_widen_codes)."""
    _need(xq, torch.float16, "xq", 2)
    _need(Wq16, torch.float16, "Wq16", 2)
    _need(scale_x, torch.float32, "scale_x", 1)
    _need(scale_w, torch.float32, "scale_w", 1)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = xq.shape
    N = Wq16.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    _check(lib().convrot_gemm_dequant_w16(_ptr(xq), _ptr(scale_x), M, K, _ptr(Wq16), _ptr(scale_w), N, _ptr(bias),
                                          _ptr(y), _stream(stream)), "convrot_gemm_dequant_w16")
    return y


def convrot_act_workspace_bytes(M: int, K: int) -> int:
    return lib().convrot_act_workspace_bytes(M, K)


def convrot_linear_workspace_bytes(M: int, K: int, N: int) -> int:
    return lib().convrot_linear_workspace_bytes(M, K, N)


def _linear_ws(M, K, N, device, workspace):
    """The caller's workspace (its whole size is passed on, so a large enough one
    takes the widened-weight path), or a new one of the fast size."""
    if workspace is None:
        nbytes = convrot_linear_workspace_bytes(M, K, N)
        return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device), nbytes
    nbytes = workspace.numel() * workspace.element_size()
    if nbytes < convrot_act_workspace_bytes(M, K):
        raise ValueError("workspace too small")
    return workspace, nbytes


def convrot_linear_fwd(x, Wq, scale_w, block, bias=None, y=None, workspace=None, stream=None):
    """Forward of the ConvRot INT8 linear layer: bf16 [M, K] -> bf16 [M, N]."""
    _need(x, torch.bfloat16, "x", 2)
    _need(Wq, torch.int8, "Wq", 2)
    _need(scale_w, torch.float32, "scale_w", 1)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = x.shape
    N = Wq.shape[0]
    if Wq.shape[1] != K or scale_w.shape[0] != N:
        raise ValueError("shape mismatch")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws, nbytes = _linear_ws(M, K, N, x.device, workspace)
    _check(lib().convrot_linear_fwd(_ptr(x), M, K, _ptr(Wq), _ptr(scale_w), N, block, _ptr(bias), _ptr(y), _ptr(ws),
                                    nbytes, _stream(stream)), "convrot_linear_fwd")
    return y


def convrot_linear_lora_workspace_bytes(M: int, K: int, N: int) -> int:
    return lib().convrot_linear_lora_workspace_bytes(M, K, N)


def convrot_linear_fwd_lora(x, Wq, scale_w, block, lora_A, lora_B, alpha, scale=1.0, bias=None, y=None,
                            workspace=None, stream=None):
    """Forward with an unmerged LoRA adapter as a bypass branch on the unrotated input."""
    _need(x, torch.bfloat16, "x", 2)
    _need(Wq, torch.int8, "Wq", 2)
    _need(scale_w, torch.float32, "scale_w", 1)
    _need(lora_A, torch.float32, "lora_A", 2)
    _need(lora_B, torch.float32, "lora_B", 2)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = x.shape
    N = Wq.shape[0]
    rank = lora_A.shape[0]
    if Wq.shape[1] != K or lora_A.shape[1] != K or lora_B.shape != (N, rank):
        raise ValueError("shape mismatch")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    nbytes = convrot_linear_lora_workspace_bytes(M, K, N)
    ws = _workspace(nbytes, x.device, workspace)
    _check(lib().convrot_linear_fwd_lora(_ptr(x), M, K, _ptr(Wq), _ptr(scale_w), N, block, _ptr(bias), _ptr(lora_A),
                                         _ptr(lora_B), rank, alpha, scale, _ptr(y), _ptr(ws), nbytes,
                                         _stream(stream)), "convrot_linear_fwd_lora")
    return y


def convrot_bwd_weight_workspace_bytes(N: int, K: int) -> int:
    return lib().convrot_bwd_weight_workspace_bytes(N, K)


def convrot_prepare_bwd_weight(Wq, scale_w, block, WtQ=None, scale_wt=None, workspace=None, stream=None):
    """One-off int8 backward weight: returns (WtQ int8 [K, N], scale_wt fp32 [K])."""
    _need(Wq, torch.int8, "Wq", 2)
    _need(scale_w, torch.float32, "scale_w", 1)
    N, K = Wq.shape
    if WtQ is None:
        WtQ = torch.empty((K, N), dtype=torch.int8, device=Wq.device)
    if scale_wt is None:
        scale_wt = torch.empty((K,), dtype=torch.float32, device=Wq.device)
    nbytes = convrot_bwd_weight_workspace_bytes(N, K)
    ws = _workspace(nbytes, Wq.device, workspace)
    _check(lib().convrot_prepare_bwd_weight(_ptr(Wq), _ptr(scale_w), N, K, block, _ptr(WtQ), _ptr(scale_wt), _ptr(ws),
                                            nbytes, _stream(stream)), "convrot_prepare_bwd_weight")
    return WtQ, scale_wt


def convrot_linear_bwd_x(dY, WtQ, scale_wt, block, dX=None, workspace=None, stream=None):
    """Input gradient of the frozen layer: dY bf16 [M, N] -> dX bf16 [M, K]."""
    _need(dY, torch.bfloat16, "dY", 2)
    _need(WtQ, torch.int8, "WtQ", 2)
    _need(scale_wt, torch.float32, "scale_wt", 1)
    M, N = dY.shape
    K = WtQ.shape[0]
    if WtQ.shape[1] != N:
        raise ValueError("shape mismatch")
    if dX is None:
        dX = torch.empty((M, K), dtype=torch.bfloat16, device=dY.device)
    ws, nbytes = _linear_ws(M, N, K, dY.device, workspace)
    _check(lib().convrot_linear_bwd_x(_ptr(dY), M, N, _ptr(WtQ), _ptr(scale_wt), K, block, _ptr(dX), _ptr(ws), nbytes,
                                      _stream(stream)), "convrot_linear_bwd_x")
    return dX


def convrot_dequant_weight_t(Wq, scale_w, block, out=None, stream=None):
    """bf16-mode backward weight: W_eff^T = bf16((scale_w (.) Wq) R)^T, bf16 [K, N]."""
    _need(Wq, torch.int8, "Wq", 2)
    _need(scale_w, torch.float32, "scale_w", 1)
    N, K = Wq.shape
    if out is None:
        out = torch.empty((K, N), dtype=torch.bfloat16, device=Wq.device)
    _check(lib().convrot_dequant_weight_t(_ptr(Wq), _ptr(scale_w), N, K, block, _ptr(out), _stream(stream)),
           "convrot_dequant_weight_t")
    return out


def convrot_gemm_bf16(A, B, out=None, stream=None):
    """C = bf16(A . B^T) on the tensor cores (fp32 accumulation): A bf16 [M, K], B bf16 [N, K]."""
    _need(A, torch.bfloat16, "A", 2)
    _need(B, torch.bfloat16, "B", 2)
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _check(lib().convrot_gemm_bf16(_ptr(A), M, K, _ptr(B), N, _ptr(out), _stream(stream)), "convrot_gemm_bf16")
    return out


def convrot_bwd_x_bf16_workspace_bytes(N: int, K: int) -> int:
    return lib().convrot_bwd_x_bf16_workspace_bytes(N, K)


def convrot_linear_bwd_x_bf16(dY, Wq, scale_w, block, dX=None, workspace=None, stream=None):
    """Input gradient in bf16 mode: dY bf16 [M, N], Wq int8 [N, K] -> dX = bf16(dY . W_eff) [M, K]."""
    _need(dY, torch.bfloat16, "dY", 2)
    _need(Wq, torch.int8, "Wq", 2)
    _need(scale_w, torch.float32, "scale_w", 1)
    M, N = dY.shape
    if Wq.shape[0] != N:
        raise ValueError("shape mismatch")
    K = Wq.shape[1]
    if dX is None:
        dX = torch.empty((M, K), dtype=torch.bfloat16, device=dY.device)
    nbytes = convrot_bwd_x_bf16_workspace_bytes(N, K)
    ws = _workspace(nbytes, dY.device, workspace)
    _check(lib().convrot_linear_bwd_x_bf16(_ptr(dY), M, N, _ptr(Wq), _ptr(scale_w), K, block, _ptr(dX), _ptr(ws),
                                           nbytes, _stream(stream)), "convrot_linear_bwd_x_bf16")
    return dX


def convrot_bwd_x_r2_workspace_bytes(M: int, N: int, K: int) -> int:
    return lib().convrot_bwd_x_r2_workspace_bytes(M, N, K)


def convrot_linear_bwd_x_r2(dY, Wq, scale_w, block, dX=None, workspace=None, stream=None):
    """Input gradient through the int8 GEMM, second reading: dY bf16 [M, N], Wq int8 [N, K] -> dX bf16 [M, K]."""
    _need(dY, torch.bfloat16, "dY", 2)
    _need(Wq, torch.int8, "Wq", 2)
    _need(scale_w, torch.float32, "scale_w", 1)
    M, N = dY.shape
    if Wq.shape[0] != N:
        raise ValueError("shape mismatch")
    K = Wq.shape[1]
    if dX is None:
        dX = torch.empty((M, K), dtype=torch.bfloat16, device=dY.device)
    nbytes = convrot_bwd_x_r2_workspace_bytes(M, N, K)
    ws = _workspace(nbytes, dY.device, workspace)
    _check(lib().convrot_linear_bwd_x_r2(_ptr(dY), M, N, _ptr(Wq), _ptr(scale_w), K, block, _ptr(dX), _ptr(ws),
                                         nbytes, _stream(stream)), "convrot_linear_bwd_x_r2")
    return dX


def convrot_embedding_lookup(ids, Eq, scale_e, block, out=None, stream=None):
    """Dequantize + inverse-rotate rows of an int8 table: ids int64 [n] -> bf16 [n, D]."""
    _need(ids, torch.int64, "ids", 1)
    _need(Eq, torch.int8, "Eq", 2)
    _need(scale_e, torch.float32, "scale_e", 1)
    V, D = Eq.shape
    n = ids.shape[0]
    if out is None:
        out = torch.empty((n, D), dtype=torch.bfloat16, device=Eq.device)
    _check(lib().convrot_embedding_lookup(_ptr(ids), n, _ptr(Eq), _ptr(scale_e), V, D, block, _ptr(out),
                                          _stream(stream)), "convrot_embedding_lookup")
    return out


def convrot_gemm_s32_workspace_bytes(M: int, K: int) -> int:
    return lib().convrot_gemm_s32_workspace_bytes(M, K)


def convrot_gemm_s32(A, B, C=None, workspace=None, stream=None):
    """Exact int32 C = A . B^T for int8 codes (the GEMM's accumulator, for checks)."""
    _need(A, torch.int8, "A", 2)
    _need(B, torch.int8, "B", 2)
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.int32, device=A.device)
    nbytes = convrot_gemm_s32_workspace_bytes(M, K)
    ws = _workspace(nbytes, A.device, workspace)
    _check(lib().convrot_gemm_s32(_ptr(A), _ptr(B), M, N, K, _ptr(C), _ptr(ws), nbytes, _stream(stream)),
           "convrot_gemm_s32")
    return C


def convrot_linear_fwd_noalloc_max_bytes() -> int:
    return lib().convrot_linear_fwd_noalloc_max_bytes()


def convrot_linear_fwd_noalloc(x, Wq, scale_w, block, bias=None, y=None, stream=None):
    """Forward without a caller workspace, for callers that cannot allocate on
    this path (the library keeps the activation codes in a fixed 64.25 MiB device
    array; calls that overlap on the GPU must be serialised by the caller).
    `y` must be given by such callers; it is allocated here only for
    convenience when omitted."""
    _need(x, torch.bfloat16, "x", 2)
    _need(Wq, torch.int8, "Wq", 2)
    _need(scale_w, torch.float32, "scale_w", 1)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = x.shape
    N = Wq.shape[0]
    if Wq.shape[1] != K or scale_w.shape[0] != N:
        raise ValueError("shape mismatch")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(lib().convrot_linear_fwd_noalloc(_ptr(x), M, K, _ptr(Wq), _ptr(scale_w), N, block, _ptr(bias), _ptr(y),
                                            _stream(stream)), "convrot_linear_fwd_noalloc")
    return y
