"""GPU parity of the in-place RMSNorm + rotary embedding of Q and K (the qk_transform stage)
against the CPU oracle: every bf16 output bit-identical, V and everything outside the Q and K
views untouched."""
import math

import numpy as np
import pytest
import torch

import oracle
import parity
import video_diffusion_transformer_sage_gb300 as sage
from video_diffusion_transformer_sage_gb300 import synth

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _tables(n, d, n_text=514, grid=synth.VIDEO_GRID):
    gq, gk = synth.qk_norm_weights(d)
    cos, sin = synth.rope_table(synth.rope_positions(n, n_text=n_text, grid=grid), d)
    return gq, gk, cos, sin


def _run_both(inp, n_text=514, grid=synth.VIDEO_GRID):
    """(oracle result, GPU result) as whole input buffers (int16 bit patterns)."""
    n, h, d = inp.q.shape
    gq, gk, cos, sin = _tables(n, d, n_text, grid)
    dev = torch.device("cuda:0")
    storage = inp.storage.to(dev)

    def dview(t):
        off = t.storage_offset() - inp.storage.storage_offset()
        return storage.as_strided(t.shape, t.stride(), storage.storage_offset() + off)

    sage.sage_qk_rmsnorm_rope(dview(inp.q), dview(inp.k), gq.to(dev), gk.to(dev), cos.to(dev), sin.to(dev), EPS)
    torch.cuda.synchronize()
    oracle.rmsnorm_rope(inp.q, gq.numpy(), cos.numpy(), sin.numpy(), EPS)
    oracle.rmsnorm_rope(inp.k, gk.numpy(), cos.numpy(), sin.numpy(), EPS)
    return inp.storage.view(torch.int16).numpy(), storage.cpu().view(torch.int16).numpy()


@pytest.mark.parametrize("name", ["tiny", "strided64", "video"])
def test_rmsnorm_rope_bit_exact(name):
    inp = synth.make_inputs(name)
    before = inp.storage.clone().view(torch.int16).numpy()
    want, got = _run_both(inp)
    assert np.array_equal(got, want)
    if inp.storage.dim() == 2:                    # token-major QKV buffer: V slice untouched
        hd = inp.q.shape[1] * inp.q.shape[2]
        assert np.array_equal(got[:, 2 * hd:], before[:, 2 * hd:])
    assert (want != before).any()                 # the transform did change Q and K


@pytest.mark.parametrize("n,h,d", [(257, 3, 128), (129, 5, 64), (1, 1, 64)])
def test_rmsnorm_rope_ragged_row_counts(n, h, d):
    """Row counts that leave a partial CTA (and a single row)."""
    inp = synth.make_inputs(synth.custom(n, h, d, "qkv", seed=n + h, n_outlier=1))
    want, got = _run_both(inp, n_text=min(n, 20), grid=(4, 4, 8))
    assert np.array_equal(got, want)


def test_transform_then_attention_matches_oracle():
    """The stage composed with the quantised attention: transform Q and K in place, then
    sage_attn_fwd, against the oracle doing the same on the CPU."""
    inp = synth.make_inputs(synth.custom(600, 4, 128, "qkv", seed=3, n_outlier=2))
    n, h, d = inp.q.shape
    gq, gk, cos, sin = _tables(n, d, n_text=100, grid=(2, 10, 25))
    dev = torch.device("cuda:0")
    storage = inp.storage.to(dev)
    hd = h * d
    q, k, v = (storage[:, i * hd:(i + 1) * hd].view(n, h, d) for i in range(3))
    sage.sage_qk_rmsnorm_rope(q, k, gq.to(dev), gk.to(dev), cos.to(dev), sin.to(dev), EPS)
    sm = 1.0 / math.sqrt(d)
    out = sage.sage_attn_fwd(q, k, v, sm)
    torch.cuda.synchronize()
    oracle.rmsnorm_rope(inp.q, gq.numpy(), cos.numpy(), sin.numpy(), EPS)
    oracle.rmsnorm_rope(inp.k, gk.numpy(), cos.numpy(), sin.numpy(), EPS)
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    rows = list(range(n))
    got = out.float().cpu().numpy().astype(np.float64)
    parity.assert_close(got, qz, sm, rows)


def test_rmsnorm_rope_hnd_layout():
    """HND-contiguous Q and K (head stride N * D): heads are not contiguous within a token, so
    the row kernel runs instead of the token-slice (bulk copy) kernel; same bits as the oracle."""
    inp = synth.to_hnd(synth.make_inputs(synth.custom(700, 3, 128, "qkv", seed=5, n_outlier=1)))
    assert inp.q.stride(1) == 700 * 128
    want, got = _run_both(inp, n_text=50, grid=(5, 5, 26))
    assert np.array_equal(got, want)


def _fused_vs_oracle(inp, n_text, grid, q_block=128):
    """The fused call (transform in the quantise prologue) against the oracle's transform of
    copies of Q and K followed by its quantisation: codes, scales and K mean bit-identical, and
    the device Q, K, V left as they were."""
    n, h, d = inp.q.shape
    gq, gk, cos, sin = _tables(n, d, n_text, grid)
    dev = torch.device("cuda:0")
    storage = inp.storage.to(dev)

    def dview(t):
        off = t.storage_offset() - inp.storage.storage_offset()
        return storage.as_strided(t.shape, t.stride(), storage.storage_offset() + off)

    before = storage.clone()
    gz = sage.sage_smooth_quant_qk_rmsnorm_rope(dview(inp.q), dview(inp.k), gq.to(dev), gk.to(dev), cos.to(dev),
                                               sin.to(dev), EPS, q_block=q_block)
    torch.cuda.synchronize()
    assert torch.equal(storage.view(torch.int16), before.view(torch.int16))    # Q and K only read
    q, k = inp.q.clone(), inp.k.clone()
    oracle.rmsnorm_rope(q, gq.numpy(), cos.numpy(), sin.numpy(), EPS)
    oracle.rmsnorm_rope(k, gk.numpy(), cos.numpy(), sin.numpy(), EPS)
    oz = oracle.Quantized(q, k, inp.v, q_block=q_block)
    assert np.array_equal(gz.k_mean.cpu().numpy().view(np.uint32), oz.k_mean.view(np.uint32))
    assert np.array_equal(gz.q_scales.cpu().numpy().view(np.uint32), oz.q_scales.view(np.uint32))
    assert np.array_equal(gz.k_scales.cpu().numpy().view(np.uint32), oz.k_scales.view(np.uint32))
    assert np.array_equal(gz.q_codes.cpu().float().numpy(), oz.q_codes.astype(np.float32))
    assert np.array_equal(gz.k_codes.cpu().float().numpy(), oz.k_codes.astype(np.float32))
    return gz, oz


@pytest.mark.parametrize("name,q_block", [("tiny", 128), ("strided64", 128), ("video", 128), ("tails", 32)])
def test_fused_transform_quant_bit_exact(name, q_block):
    _fused_vs_oracle(synth.make_inputs(name), 514, synth.VIDEO_GRID, q_block)


@pytest.mark.parametrize("n,h,d", [(300, 3, 128), (129, 5, 64), (1, 1, 128)])
def test_fused_transform_quant_ragged(n, h, d):
    """Odd head counts (a warp's lanes past the last head run on zeros in the K-mean pass), a
    partial last block and a single token."""
    inp = synth.make_inputs(synth.custom(n, h, d, "qkv", seed=n + 2 * h, n_outlier=1))
    _fused_vs_oracle(inp, min(n, 20), (4, 4, 8))


def test_fused_transform_quant_hnd_and_attention():
    """HND-contiguous views, then the attention on the fused call's codes against the oracle."""
    inp = synth.to_hnd(synth.make_inputs(synth.custom(700, 3, 128, "qkv", seed=8, n_outlier=1)))
    gz, oz = _fused_vs_oracle(inp, 50, (5, 5, 26))
    dv = inp.v.to("cuda")
    sage.sage_quant_v(dv, gz)
    sm = 1.0 / math.sqrt(128)
    out = sage.sage_attn_fwd_quantized(gz, sm)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    parity.assert_close(got, oz, sm, list(range(700)))
