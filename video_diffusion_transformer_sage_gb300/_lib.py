"""ctypes binding of `libsage_gb300.so` (include/sage.h): argument marshalling only.

Every step of the attention path runs in the library's CUDA kernels; this module only turns
torch tensors into pointers, sizes and strides, allocates outputs and workspaces with
torch, and raises `SageError` on a non-OK status.  There is no fallback: if the library is
missing the import of any op raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsage_gb300.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "sage.h")

STATUS = {0: "SAGE_OK", 1: "SAGE_ERR_INVALID_ARG", 2: "SAGE_ERR_ALIGNMENT", 3: "SAGE_ERR_UNSUPPORTED",
          4: "SAGE_ERR_WORKSPACE", 5: "SAGE_ERR_CUDA", 6: "SAGE_ERR_DEVICE_TIMEOUT"}


class SageError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


class SageView(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("n_tokens", ctypes.c_int64), ("n_heads", ctypes.c_int64),
                ("head_dim", ctypes.c_int64), ("stride_token", ctypes.c_int64),
                ("stride_head", ctypes.c_int64)]


class SageQuantizedC(ctypes.Structure):
    _fields_ = [("q_codes", ctypes.c_void_p), ("q_scales", ctypes.c_void_p), ("k_codes", ctypes.c_void_p),
                ("k_scales", ctypes.c_void_p), ("k_mean", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("v_scales", ctypes.c_void_p), ("q_block", ctypes.c_int64), ("v_format", ctypes.c_int64),
                ("v_mean", ctypes.c_void_p)]

V_FORMATS = {"e4m3": 0, "int8": 1}


_lib = None


def header_functions() -> list:
    """Names of the functions include/sage.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**(sage_[a-z_0-9]+)\s*\(", text, re.M)))


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() (no CPU fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        VP = ctypes.POINTER(SageView)
        QP = ctypes.POINTER(SageQuantizedC)
        sig = {
            "sage_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "sage_quant_scratch_bytes": ([I, I, I], S),
            "sage_workspace_bytes": ([I, I, I], S),
            "sage_status_block_bytes": ([], S),
            "sage_smooth_quant_qk": ([VP, VP, QP, P, S, P], ctypes.c_int),
            "sage_quant_v": ([VP, QP, P, S, P], ctypes.c_int),
            "sage_quant_qkv": ([VP, VP, VP, QP, P, S, P], ctypes.c_int),
            "sage_smooth_quant_qk_noalloc": ([VP, VP, QP, P], ctypes.c_int),
            "sage_attn_fwd_quantized": ([I, I, I, QP, F, P, I, I, P, P], ctypes.c_int),
            "sage_attn_fwd": ([VP, VP, VP, F, P, I, I, P, S, P], ctypes.c_int),
            "sage_attn_dense_bf16": ([VP, VP, VP, F, P, I, I, P], ctypes.c_int),
            "sage_dense_workspace_bytes": ([I, I, I], S),
            "sage_attn_dense_bf16_tc": ([VP, VP, VP, F, P, I, I, P, S, P], ctypes.c_int),
            "sage_debug_qk_int32": ([I, I, I, QP, I, I, I, I, I, P, P, P], ctypes.c_int),
            "sage_check_device_status": ([P, P, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
            "sage_get_device_status": ([P, P, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
            "sage_debug_wait_timeout": ([P, I, P], ctypes.c_int),
            "sage_measure_mma_rate": ([I, I, I, P, P], ctypes.c_int),
            "sage_qk_rmsnorm_rope": ([VP, VP, P, P, P, P, F, P], ctypes.c_int),
            "sage_smooth_quant_qk_rmsnorm_rope": ([VP, VP, P, P, P, P, F, QP, P, S, P], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(code: int, what: str) -> None:
    if code != 0:
        raise SageError(code, what)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_view(t: torch.Tensor) -> SageView:
    """A bf16 CUDA [N, H, D] tensor (any token / head strides, unit channel stride)."""
    if t.dim() != 3 or t.dtype != torch.bfloat16 or not t.is_cuda or t.stride(2) != 1:
        raise ValueError("expected a bf16 CUDA [N, H, D] tensor with unit channel stride")
    n, h, d = t.shape
    return SageView(t.data_ptr(), n, h, d, t.stride(0), t.stride(1))


def pad128(n: int) -> int:
    return (n + 127) // 128 * 128


class Quantized:
    """Device buffers of the quantised operands (layouts of sage_quantized in include/sage.h)."""

    def __init__(self, n: int, h: int, d: int, device="cuda", q_block: int = 128, v_format: str = "e4m3",
                 smooth_v: bool = False):
        """q_block: rows per Q scale (128, the method's default, or a smaller power of two).
        v_format: "e4m3" (the method's FP8 V and P) or "int8" (the INT8 P.V variant; codes held
        as fp16).  smooth_v: quantise V minus its channel mean and add the mean back."""
        np_ = pad128(n)
        if q_block not in (1, 2, 4, 8, 16, 32, 64, 128):
            raise ValueError(f"q_block must be a power of two <= 128, got {q_block}")
        if v_format not in V_FORMATS:
            raise ValueError(f"v_format must be one of {sorted(V_FORMATS)}, got {v_format!r}")
        self.n, self.h, self.d, self.q_block, self.v_format = n, h, d, q_block, v_format
        self.q_codes = torch.empty((h, np_, d), dtype=torch.float16, device=device)
        self.k_codes = torch.empty((h, np_, d), dtype=torch.float16, device=device)
        self.v_codes = torch.empty((h, d, np_), dtype=torch.float16 if v_format == "int8" else torch.uint8,
                                   device=device)
        self.v_mean = torch.empty((h, d), dtype=torch.float32, device=device) if smooth_v else None
        self.q_scales = torch.empty((h, np_ // q_block), dtype=torch.float32, device=device)
        self.k_scales = torch.empty((h, np_ // 64), dtype=torch.float32, device=device)
        self.k_mean = torch.empty((h, d), dtype=torch.float32, device=device)
        self.v_scales = torch.empty((h, d), dtype=torch.float32, device=device)

    def c(self) -> SageQuantizedC:
        return SageQuantizedC(self.q_codes.data_ptr(), self.q_scales.data_ptr(), self.k_codes.data_ptr(),
                              self.k_scales.data_ptr(), self.k_mean.data_ptr(), self.v_codes.data_ptr(),
                              self.v_scales.data_ptr(), self.q_block, V_FORMATS[self.v_format],
                              None if self.v_mean is None else self.v_mean.data_ptr())


def quant_scratch(n: int, h: int, d: int, device="cuda") -> torch.Tensor:
    return torch.empty(int(lib().sage_quant_scratch_bytes(n, h, d)), dtype=torch.uint8, device=device)


def status_block(device="cuda") -> torch.Tensor:
    return torch.zeros(int(lib().sage_status_block_bytes()), dtype=torch.uint8, device=device)


def workspace(n: int, h: int, d: int, device="cuda") -> torch.Tensor:
    """Workspace for sage_attn_fwd; its leading status block starts zeroed."""
    ws = torch.empty(int(lib().sage_workspace_bytes(n, h, d)) + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + int(lib().sage_workspace_bytes(n, h, d))]
    ws[:256].zero_()
    return ws


def sage_smooth_quant_qk(q: torch.Tensor, k: torch.Tensor, qz: Optional[Quantized] = None,
                         scratch: Optional[torch.Tensor] = None, stream=None, q_block: int = 128,
                         v_format: str = "e4m3", smooth_v: bool = False) -> Quantized:
    """When qz is None a Quantized is made here; q_block, v_format and smooth_v set it up
    (the V options take effect in sage_quant_v and the attention)."""
    n, h, d = q.shape
    qz = qz or Quantized(n, h, d, q.device, q_block, v_format, smooth_v)
    scratch = scratch if scratch is not None else quant_scratch(n, h, d, q.device)
    vq, vk, c = make_view(q), make_view(k), qz.c()
    _check(lib().sage_smooth_quant_qk(ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(c), scratch.data_ptr(),
                                      scratch.numel(), _stream(stream)), "sage_smooth_quant_qk")
    return qz


def sage_smooth_quant_qk_noalloc(q: torch.Tensor, k: torch.Tensor, qz: Optional[Quantized] = None,
                                 stream=None) -> Quantized:
    """sage_smooth_quant_qk for callers that cannot allocate: the library's fixed device
    scratch array replaces the caller workspace (see include/sage.h for the size limit)."""
    n, h, d = q.shape
    qz = qz or Quantized(n, h, d, q.device)
    vq, vk, c = make_view(q), make_view(k), qz.c()
    _check(lib().sage_smooth_quant_qk_noalloc(ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(c), _stream(stream)),
           "sage_smooth_quant_qk_noalloc")
    return qz


def sage_quant_v(v: torch.Tensor, qz: Quantized, scratch: Optional[torch.Tensor] = None, stream=None) -> Quantized:
    n, h, d = v.shape
    scratch = scratch if scratch is not None else quant_scratch(n, h, d, v.device)
    vv, c = make_view(v), qz.c()
    _check(lib().sage_quant_v(ctypes.byref(vv), ctypes.byref(c), scratch.data_ptr(), scratch.numel(),
                              _stream(stream)), "sage_quant_v")
    return qz


def sage_quant_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, qz: Optional[Quantized] = None,
                   scratch: Optional[torch.Tensor] = None, stream=None, q_block: int = 128, v_format: str = "e4m3",
                   smooth_v: bool = False) -> Quantized:
    """sage_smooth_quant_qk then sage_quant_v in one call (5 launches on the default options).
    scratch: at least 2 * sage_quant_scratch_bytes bytes (made here when None)."""
    n, h, d = q.shape
    qz = qz or Quantized(n, h, d, q.device, q_block, v_format, smooth_v)
    if scratch is None:
        scratch = torch.empty(2 * int(lib().sage_quant_scratch_bytes(n, h, d)), dtype=torch.uint8, device=q.device)
    vq, vk, vv, c = make_view(q), make_view(k), make_view(v), qz.c()
    _check(lib().sage_quant_qkv(ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(vv), ctypes.byref(c),
                                scratch.data_ptr(), scratch.numel(), _stream(stream)), "sage_quant_qkv")
    return qz


def _out_args(out: Optional[torch.Tensor], n: int, h: int, d: int, device):
    if out is None:
        out = torch.empty((n, h, d), dtype=torch.bfloat16, device=device)
    if out.dtype != torch.bfloat16 or out.stride(2) != 1 or tuple(out.shape) != (n, h, d):
        raise ValueError("out must be bf16 [N, H, D] with unit channel stride")
    return out, out.stride(0), out.stride(1)


def sage_attn_fwd_quantized(qz: Quantized, sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                            status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    sm_scale = 1.0 / math.sqrt(qz.d) if sm_scale is None else sm_scale
    out, ost, osh = _out_args(out, qz.n, qz.h, qz.d, qz.q_codes.device)
    status = status if status is not None else status_block(qz.q_codes.device)
    c = qz.c()
    _check(lib().sage_attn_fwd_quantized(qz.n, qz.h, qz.d, ctypes.byref(c), sm_scale, out.data_ptr(), ost, osh,
                                         status.data_ptr(), _stream(stream)), "sage_attn_fwd_quantized")
    return out


def sage_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, sm_scale: Optional[float] = None,
                  out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    n, h, d = q.shape
    sm_scale = 1.0 / math.sqrt(d) if sm_scale is None else sm_scale
    out, ost, osh = _out_args(out, n, h, d, q.device)
    ws = ws if ws is not None else workspace(n, h, d, q.device)
    vq, vk, vv = make_view(q), make_view(k), make_view(v)
    _check(lib().sage_attn_fwd(ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(vv), sm_scale, out.data_ptr(), ost,
                               osh, ws.data_ptr(), ws.numel(), _stream(stream)), "sage_attn_fwd")
    return out


def sage_attn_dense_bf16(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, sm_scale: Optional[float] = None,
                         out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    n, h, d = q.shape
    sm_scale = 1.0 / math.sqrt(d) if sm_scale is None else sm_scale
    out, ost, osh = _out_args(out, n, h, d, q.device)
    vq, vk, vv = make_view(q), make_view(k), make_view(v)
    _check(lib().sage_attn_dense_bf16(ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(vv), sm_scale,
                                      out.data_ptr(), ost, osh, _stream(stream)), "sage_attn_dense_bf16")
    return out


def dense_workspace(n: int, h: int, d: int, device="cuda") -> torch.Tensor:
    """Workspace for sage_attn_dense_bf16_tc; its leading status block starts zeroed."""
    need = int(lib().sage_dense_workspace_bytes(n, h, d))
    ws = torch.empty(need + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + need]
    ws[:256].zero_()
    return ws


def sage_attn_dense_bf16_tc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, sm_scale: Optional[float] = None,
                            out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    n, h, d = q.shape
    sm_scale = 1.0 / math.sqrt(d) if sm_scale is None else sm_scale
    out, ost, osh = _out_args(out, n, h, d, q.device)
    ws = dense_workspace(n, h, d, q.device) if ws is None else ws
    vq, vk, vv = make_view(q), make_view(k), make_view(v)
    _check(lib().sage_attn_dense_bf16_tc(ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(vv), sm_scale,
                                         out.data_ptr(), ost, osh, ws.data_ptr(), ws.numel(), _stream(stream)),
           "sage_attn_dense_bf16_tc")
    return out


def sage_debug_qk_int32(qz: Quantized, head: int, i0: int, j0: int, row_tiles: int = 1, col_tiles: int = 1,
                        status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    out = torch.empty((128 * row_tiles, 128 * col_tiles), dtype=torch.int32, device=qz.q_codes.device)
    status = status if status is not None else status_block(qz.q_codes.device)
    c = qz.c()
    _check(lib().sage_debug_qk_int32(qz.n, qz.h, qz.d, ctypes.byref(c), head, i0, j0, row_tiles, col_tiles,
                                     out.data_ptr(), status.data_ptr(), _stream(stream)), "sage_debug_qk_int32")
    return out


def sage_debug_wait_timeout(status: torch.Tensor, limit_ns: int, stream=None) -> None:
    _check(lib().sage_debug_wait_timeout(status.data_ptr(), int(limit_ns), _stream(stream)), "sage_debug_wait_timeout")


# FLOPs per CTA and round of each sage_measure_mma_rate mode (2 M N K per MMA).
MMA_RATE_FLOPS = {0: 8 * 2 * 128 * 128 * 16, 1: 8 * 2 * 128 * 128 * 32, 2: 8 * 2 * 128 * 128 * 16 + 4 * 2 * 128 * 128 * 32,
                  3: 8 * 2 * 128 * 256 * 32, 4: 8 * 2 * 128 * 256 * 16, 5: 8 * 2 * 128 * 64 * 32,
                  6: 4 * 2 * 128 * 128 * 16 + 4 * 2 * 128 * 64 * 32}


def sage_measure_mma_rate(mode: int, iters: int, ctas: int, status: torch.Tensor, stream=None) -> None:
    _check(lib().sage_measure_mma_rate(int(mode), int(iters), int(ctas), status.data_ptr(), _stream(stream)),
           "sage_measure_mma_rate")


def sage_check_device_status(status: torch.Tensor, stream=None):
    """Synchronises `stream`; returns (status code, where) and clears a recorded timeout."""
    where = ctypes.c_int32(0)
    code = lib().sage_check_device_status(status.data_ptr(), _stream(stream), ctypes.byref(where))
    return int(code), int(where.value)


def sage_qk_rmsnorm_rope(q: torch.Tensor, k: torch.Tensor, gamma_q: torch.Tensor, gamma_k: torch.Tensor,
                         rope_cos: torch.Tensor, rope_sin: torch.Tensor, eps: float = 1e-6, stream=None) -> None:
    """In place on the bf16 [N, H, D] CUDA views q and k: RMSNorm over D (weights gamma_q /
    gamma_k, fp32 [D]) and the rotation of channel pairs by the fp32 [N, D/2] cos / sin table."""
    n, h, d = q.shape
    for t, shape in ((gamma_q, (d,)), (gamma_k, (d,)), (rope_cos, (n, d // 2)), (rope_sin, (n, d // 2))):
        if t.dtype != torch.float32 or not t.is_cuda or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"expected a contiguous fp32 CUDA tensor of shape {shape}")
    vq, vk = make_view(q), make_view(k)
    _check(lib().sage_qk_rmsnorm_rope(ctypes.byref(vq), ctypes.byref(vk), gamma_q.data_ptr(), gamma_k.data_ptr(),
                                      rope_cos.data_ptr(), rope_sin.data_ptr(), float(eps), _stream(stream)),
           "sage_qk_rmsnorm_rope")


def _check_transform_tables(n: int, d: int, gamma_q, gamma_k, rope_cos, rope_sin) -> None:
    for t, shape in ((gamma_q, (d,)), (gamma_k, (d,)), (rope_cos, (n, d // 2)), (rope_sin, (n, d // 2))):
        if t.dtype != torch.float32 or not t.is_cuda or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"expected a contiguous fp32 CUDA tensor of shape {shape}")


def sage_smooth_quant_qk_rmsnorm_rope(q: torch.Tensor, k: torch.Tensor, gamma_q: torch.Tensor, gamma_k: torch.Tensor,
                                      rope_cos: torch.Tensor, rope_sin: torch.Tensor, eps: float = 1e-6,
                                      qz: Optional[Quantized] = None, scratch: Optional[torch.Tensor] = None,
                                      stream=None, q_block: int = 128, v_format: str = "e4m3",
                                      smooth_v: bool = False) -> Quantized:
    """sage_qk_rmsnorm_rope then sage_smooth_quant_qk in one pass, without modifying q and k:
    the transform runs in the quantise kernels' prologue."""
    n, h, d = q.shape
    _check_transform_tables(n, d, gamma_q, gamma_k, rope_cos, rope_sin)
    qz = qz or Quantized(n, h, d, q.device, q_block, v_format, smooth_v)
    scratch = scratch if scratch is not None else quant_scratch(n, h, d, q.device)
    vq, vk, c = make_view(q), make_view(k), qz.c()
    _check(lib().sage_smooth_quant_qk_rmsnorm_rope(ctypes.byref(vq), ctypes.byref(vk), gamma_q.data_ptr(),
                                                   gamma_k.data_ptr(), rope_cos.data_ptr(), rope_sin.data_ptr(),
                                                   float(eps), ctypes.byref(c), scratch.data_ptr(), scratch.numel(),
                                                   _stream(stream)), "sage_smooth_quant_qk_rmsnorm_rope")
    return qz
