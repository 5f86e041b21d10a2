"""Host-side checks of the C ABI: the library loads, exports every function that
include/sage.h declares, sizes workspaces consistently, and rejects bad arguments before
launching anything (these calls never reach the GPU)."""
import ctypes

import pytest
import torch

import video_diffusion_transformer_sage_gb300 as sage
from video_diffusion_transformer_sage_gb300 import _lib

EXPECTED = {"sage_status_string", "sage_quant_scratch_bytes", "sage_workspace_bytes", "sage_status_block_bytes",
            "sage_smooth_quant_qk", "sage_quant_v", "sage_attn_fwd_quantized", "sage_attn_fwd",
            "sage_attn_dense_bf16", "sage_debug_qk_int32", "sage_check_device_status",
            "sage_smooth_quant_qk_noalloc", "sage_debug_wait_timeout", "sage_qk_rmsnorm_rope",
            "sage_smooth_quant_qk_rmsnorm_rope", "sage_measure_mma_rate", "sage_get_device_status",
            "sage_quant_qkv", "sage_dense_workspace_bytes", "sage_attn_dense_bf16_tc"}


@pytest.fixture(scope="module")
def L():
    from video_diffusion_transformer_sage_gb300 import build
    build.build()
    return sage.lib()


def test_header_declares_expected(L):
    assert set(sage.header_functions()) == EXPECTED


def test_library_exports_every_declared_symbol(L):
    for name in sage.header_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    for code in range(7):
        s = L.sage_status_string(code).decode()
        assert s.startswith(_lib.STATUS[code])


def test_workspace_sizes(L):
    n, h, d = 37810, 56, 128
    np_ = 37888
    ws = L.sage_workspace_bytes(n, h, d)
    need = 2 * h * np_ * d * 2 + h * d * np_ + h * (np_ // 128) * 4 + h * (np_ // 64) * 4 + 2 * h * d * 4
    need += 2 * (np_ // 128) * h * d * 4 + 256          # K and V column partials side by side
    assert need <= ws <= need + 16 * 256
    assert L.sage_quant_scratch_bytes(n, h, d) >= (np_ // 128) * h * d * 4
    assert L.sage_workspace_bytes(n, h, 96) == 0       # unsupported head_dim
    assert L.sage_workspace_bytes(0, h, d) == 0
    assert L.sage_status_block_bytes() >= 8


def _view(ptr=16, n=256, h=2, d=128, st=256, sh=128):
    return _lib.SageView(ptr, n, h, d, st, sh)


def _qz(ptr=4096):
    # seven distinct fake buffers, 16-byte aligned when ptr is
    return _lib.SageQuantizedC(*[ptr + 4096 * i for i in range(7)])


def test_argument_validation_never_launches(L):
    """Every bad argument is reported before any CUDA call: fake (non-null, aligned) device
    pointers are never dereferenced on these paths."""
    q, k, v = _view(), _view(), _view()
    qz = _qz()
    call = lambda *a: L.sage_smooth_quant_qk(*a)
    by = ctypes.byref
    # null view data; an empty input
    assert call(by(_view(ptr=0)), by(k), by(qz), 4096, 1 << 30, None) == 1
    assert call(by(_view(n=0)), by(_view(n=0)), by(qz), 4096, 1 << 30, None) == 1
    assert L.sage_attn_fwd(by(_view(n=0)), by(_view(n=0)), by(_view(n=0)), 0.1, 4096, 256, 128, 4096, 1 << 34,
                           None) == 1
    # unsupported head dim
    assert call(by(_view(d=96)), by(_view(d=96)), by(qz), 4096, 1 << 30, None) == 3
    # misaligned pointer / stride
    assert call(by(_view(ptr=18)), by(k), by(qz), 4096, 1 << 30, None) == 2
    assert call(by(_view(st=260)), by(k), by(qz), 4096, 1 << 30, None) == 2
    # mismatched shapes
    assert call(by(q), by(_view(n=255)), by(qz), 4096, 1 << 30, None) == 1
    # workspace too small / missing
    assert call(by(q), by(k), by(qz), 4096, 16, None) == 4
    assert call(by(q), by(k), by(qz), 0, 1 << 30, None) == 4
    # quantised buffers misaligned; one buffer for the Q and the K codes
    assert call(by(q), by(k), by(_qz(ptr=4100)), 4096, 1 << 30, None) == 2
    same = _qz()
    same.k_codes = same.q_codes
    assert call(by(q), by(k), by(same), 4096, 1 << 30, None) == 1
    assert L.sage_smooth_quant_qk_rmsnorm_rope(by(q), by(k), 4096, 4096, 4096, 4096, 1e-6, by(same), 4096, 1 << 30,
                                               None) == 1
    # fused path: bad out stride, bad scale, small workspace
    assert L.sage_attn_fwd(by(q), by(k), by(v), 0.1, 4096, 250, 128, 4096, 1 << 34, None) == 2
    assert L.sage_attn_fwd(by(q), by(k), by(v), -1.0, 4096, 256, 128, 4096, 1 << 34, None) == 1
    assert L.sage_attn_fwd(by(q), by(k), by(v), 0.1, 4096, 256, 128, 4096, 1024, None) == 4
    assert L.sage_attn_fwd(by(q), by(k), by(v), 0.1, 4096, 256, 128, 4100, 1 << 34, None) == 2
    assert L.sage_attn_fwd_quantized(256, 2, 128, by(qz), 0.1, 4096, 256, 128, 0, None) == 1
    assert L.sage_attn_dense_bf16(by(q), by(k), by(_view(h=3)), 0.1, 4096, 256, 128, None) == 1
    # tensor-core dense path: the dense path's checks, then its workspace (status block + V^T)
    dt = L.sage_attn_dense_bf16_tc
    need = L.sage_dense_workspace_bytes(256, 2, 128)
    assert need == 256 + 2 * 128 * 256 * 2
    assert L.sage_dense_workspace_bytes(256, 2, 96) == 0
    assert dt(by(q), by(k), by(_view(h=3)), 0.1, 4096, 256, 128, 4096, need, None) == 1
    assert dt(by(q), by(k), by(v), 0.1, 4096, 250, 128, 4096, need, None) == 2
    assert dt(by(q), by(k), by(v), -1.0, 4096, 256, 128, 4096, need, None) == 1
    assert dt(by(q), by(k), by(v), 0.1, 4096, 256, 128, 4096, need - 1, None) == 4
    assert dt(by(q), by(k), by(v), 0.1, 4096, 256, 128, 0, need, None) == 4
    assert dt(by(q), by(k), by(v), 0.1, 4096, 256, 128, 4352 + 16, need, None) == 2
    assert dt(by(_view(d=96)), by(_view(d=96)), by(_view(d=96)), 0.1, 4096, 256, 128, 4096, need, None) == 3
    # debug tiles outside N_pad
    assert L.sage_debug_qk_int32(256, 2, 128, by(qz), 0, 128, 0, 2, 1, 4096, 4096, None) == 1
    assert L.sage_debug_qk_int32(256, 2, 128, by(qz), 2, 0, 0, 1, 1, 4096, 4096, None) == 1
    # rows per Q scale: a power of two <= 128, or 0 for the default 128
    for bad in (3, 96, 256, -1):
        qb = _qz()
        qb.q_block = bad
        assert call(by(q), by(k), by(qb), 4096, 1 << 30, None) == 1, bad
        assert L.sage_attn_fwd_quantized(256, 2, 128, by(qb), 0.1, 4096, 256, 128, 4096, None) == 1, bad
    # V options: format 0 (E4M3) or 1 (INT8 held as fp16) only; a V mean pointer 16-byte aligned
    for bad in (2, -1):
        vb = _qz()
        vb.v_format = bad
        assert L.sage_quant_v(by(v), by(vb), 4096, 1 << 30, None) == 1, bad
        assert L.sage_attn_fwd_quantized(256, 2, 128, by(vb), 0.1, 4096, 256, 128, 4096, None) == 1, bad
    vb = _qz()
    vb.v_mean = 4100
    assert L.sage_quant_v(by(v), by(vb), 4096, 1 << 30, None) == 2
    assert L.sage_attn_fwd_quantized(256, 2, 128, by(vb), 0.1, 4096, 256, 128, 4096, None) == 2
    # in-place RMSNorm + RoPE: null tables, misaligned weights, bad eps, mismatched views
    rr = L.sage_qk_rmsnorm_rope
    assert rr(by(q), by(k), 4096, 4096, 0, 4096, 1e-6, None) == 1
    assert rr(by(q), by(k), 4100, 4096, 4096, 4096, 1e-6, None) == 2
    assert rr(by(q), by(k), 4096, 4096, 4096, 4096, -1.0, None) == 1
    assert rr(by(q), by(k), 4096, 4096, 4096, 4096, float("nan"), None) == 1
    assert rr(by(q), by(_view(h=3)), 4096, 4096, 4096, 4096, 1e-6, None) == 1
    # the same transform fused into the quantisation: its own checks and those of the quantisation
    fq = L.sage_smooth_quant_qk_rmsnorm_rope
    assert fq(by(q), by(k), 4096, 4096, 0, 4096, 1e-6, by(qz), 4096, 1 << 30, None) == 1
    assert fq(by(q), by(k), 4096, 4100, 4096, 4096, 1e-6, by(qz), 4096, 1 << 30, None) == 2
    assert fq(by(q), by(k), 4096, 4096, 4096, 4096, float("inf"), by(qz), 4096, 1 << 30, None) == 1
    assert fq(by(q), by(_view(n=255)), 4096, 4096, 4096, 4096, 1e-6, by(qz), 4096, 1 << 30, None) == 1
    assert fq(by(q), by(k), 4096, 4096, 4096, 4096, 1e-6, by(qz), 4096, 16, None) == 4
    assert fq(by(q), by(k), 4096, 4096, 4096, 4096, 1e-6, by(_qz(ptr=4100)), 4096, 1 << 30, None) == 2
    assert fq(by(_view(d=96)), by(_view(d=96)), 4096, 4096, 4096, 4096, 1e-6, by(qz), 4096, 1 << 30, None) == 3
    # Q, K and V quantised in one call: the checks of both stage calls, and twice their scratch
    qkv = L.sage_quant_qkv
    assert qkv(by(q), by(k), by(_view(n=255)), by(qz), 4096, 1 << 30, None) == 1
    assert qkv(by(q), by(k), by(_view(ptr=18)), by(qz), 4096, 1 << 30, None) == 2
    assert qkv(by(q), by(k), by(v), by(_qz(ptr=4100)), 4096, 1 << 30, None) == 2
    assert qkv(by(q), by(k), by(v), by(same), 4096, 1 << 30, None) == 1
    one = int(L.sage_quant_scratch_bytes(256, 2, 128))
    assert qkv(by(q), by(k), by(v), by(qz), 4096, one, None) == 4
    assert qkv(by(q), by(k), by(v), by(qz), 0, 1 << 30, None) == 4
    assert qkv(by(_view(d=96)), by(_view(d=96)), by(_view(d=96)), by(qz), 4096, 1 << 30, None) == 3
    assert L.sage_check_device_status(0, None, None) == 1
    assert L.sage_debug_wait_timeout(0, 1000, None) == 1
    assert L.sage_debug_wait_timeout(4096, 0, None) == 1


def test_binding_validates_options_before_allocating():
    """The Python binding rejects unknown options itself (no device memory is touched)."""
    with pytest.raises(ValueError):
        sage.Quantized(256, 2, 128, device="cpu", v_format="fp4")
    with pytest.raises(ValueError):
        sage.Quantized(256, 2, 128, device="cpu", q_block=96)
    qz = sage.Quantized(256, 2, 128, device="cpu", v_format="int8", smooth_v=True)
    assert qz.v_codes.dtype == torch.float16 and tuple(qz.v_codes.shape) == (2, 128, 256)
    assert qz.v_mean is not None and tuple(qz.v_mean.shape) == (2, 128)
    c = qz.c()
    assert c.v_format == 1 and c.v_mean == qz.v_mean.data_ptr() and c.q_block == 128
    c0 = sage.Quantized(256, 2, 128, device="cpu").c()
    assert c0.v_format == 0 and c0.v_mean is None
    assert ctypes.sizeof(_lib.SageQuantizedC) == 8 * 10          # the header's struct: 10 eight-byte fields
