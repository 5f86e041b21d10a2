"""sage_smooth_quant_qk_noalloc: the quantise entry point for callers that cannot allocate
device memory (plugin interfaces handed only inputs and outputs; code that must avoid the
device-wide synchronisation of cudaMalloc / cudaFree).  It uses the library's fixed device
scratch array instead of a caller workspace; its outputs must equal those of
sage_smooth_quant_qk bit for bit, call after call.

Collected last on purpose, and self-contained, so it passes alone in a fresh process and
after the rest of the suite."""
import ctypes

import pytest
import torch

from video_diffusion_transformer_sage_gb300 import _lib, build, synth

pytestmark = pytest.mark.gpu

FIELDS = ("q_codes", "q_scales", "k_codes", "k_scales", "k_mean")


def _device_inputs(name):
    inp = synth.make_inputs(name)
    storage = inp.storage.to("cuda")
    views = []
    for t in (inp.q, inp.k):
        off = t.storage_offset() - inp.storage.storage_offset()
        views.append(storage.as_strided(t.shape, t.stride(), storage.storage_offset() + off))
    return storage, views[0], views[1]


def _noalloc(q, k, qz):
    L = _lib.lib()
    vq, vk, c = _lib.make_view(q), _lib.make_view(k), qz.c()
    stream = torch.cuda.current_stream().cuda_stream
    return L.sage_smooth_quant_qk_noalloc(ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(c), stream)


@pytest.mark.parametrize("name", ["tails", "strided64"])
def test_noalloc_matches_allocating_entry_point(name):
    build.build()
    _, q, k = _device_inputs(name)
    n, h, d = q.shape
    ref = _lib.sage_smooth_quant_qk(q, k)           # caller-provided scratch
    for _ in range(2):                               # two calls in a row share the array
        got = _lib.Quantized(n, h, d)
        for f in FIELDS:
            getattr(got, f).fill_(-1)
        assert _noalloc(q, k, got) == 0
        torch.cuda.synchronize()
        for f in FIELDS:
            assert torch.equal(getattr(got, f), getattr(ref, f)), f


def test_noalloc_rejects_oversize_before_launch():
    build.build()
    L = _lib.lib()
    qz = _lib.SageQuantizedC(*[4096 * (i + 1) for i in range(7)])   # distinct fake buffers

    def call(n, h, d):
        v = _lib.SageView(16, n, h, d, 3 * h * d, d)
        return L.sage_smooth_quant_qk_noalloc(ctypes.byref(v), ctypes.byref(v), ctypes.byref(qz), None)

    # ceil(75620/128) * 56 * 128 = 4,236,288 floats > 4,194,304: refused, nothing launched
    assert call(75620, 56, 128) == 4                       # SAGE_ERR_WORKSPACE
    # beyond what sage_smooth_quant_qk accepts at all: its own status comes first
    assert call((1 << 22) + 1, 1, 64) == 3                 # SAGE_ERR_UNSUPPORTED, not WORKSPACE
    assert call(128, 1, 96) == 3                           # unsupported head dim
    misaligned = _lib.SageQuantizedC(*([4096 + 4] + [4096 * (i + 2) for i in range(6)]))
    v = _lib.SageView(16, 1024, 2, 128, 3 * 256, 128)
    assert L.sage_smooth_quant_qk_noalloc(ctypes.byref(v), ctypes.byref(v), ctypes.byref(misaligned), None) == 2
