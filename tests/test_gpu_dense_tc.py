"""sage_attn_dense_bf16_tc: unquantised attention on the tensor cores (bf16 Q, K, V; fp32
scores and accumulators; P rounded to bf16), against the oracle's exact fp64 softmax attention.

Error model (per output element of row r, head h, channel c), from the arithmetic the header
states:
- P = bf16_rn(p) with l the sum of the unrounded p: |sum_t p_t d_t v_tc / l| <= 2^-9 max_t |v_tc|;
- the bf16 output: <= 2^-9 |out| <= 2^-9 max_t |v_tc|;
- S from fp32 accumulation of D exact bf16 products: |dS_t| <= D 2^-23 sum_i |q_ri k_ti|, so p_t
  is off by a factor exp2(+-c |dS_t|) with c = sm_scale log2 e, and out (a ratio of sums of
  p_t) by at most 2 ln2 c max_t |dS_t| max_t |v_tc|;
- ex2.approx, the fp32 sums and the rescales add relative errors near 2^-22, covered by the
  factor 1.01 below.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import video_diffusion_transformer_sage_gb300 as sage
from conftest import gpu_case
from video_diffusion_transformer_sage_gb300 import synth

pytestmark = pytest.mark.gpu


def _bound(inp, rows, sm):
    q, k, v = (t.float().numpy().astype(np.float64) for t in (inp.q, inp.k, inp.v))
    n, h, d = q.shape
    vmax = np.abs(v).max(axis=0)                                     # [H, D]
    # max_t sum_i |q_ri k_ti| per (row, head)
    qa, ka = np.abs(q[rows]), np.abs(k)
    qk = np.stack([(qa[:, hh] @ ka[:, hh].T).max(axis=1) for hh in range(h)], axis=1)   # [R, H]
    ds = d * 2.0 ** -23 * qk                                          # [R, H]
    c = sm * math.log2(math.e)
    s_term = 2.0 * math.log(2.0) * c * ds                             # [R, H]
    return 1.01 * (2.0 ** -8 + s_term[:, :, None]) * vmax[None] + 1e-7


@pytest.mark.parametrize("name,count", [("tiny", 64), ("tails", 64), ("strided64", 48), ("sweep8192", 24),
                                        ("tails_hndcopy", 32), ("video", 16)])
def test_dense_tc_within_bf16_bound_of_exact(name, count):
    case = gpu_case(name)
    inp = case["inp"]
    n, h, d = case["q"].shape
    sm = 1.0 / math.sqrt(d)
    out = sage.sage_attn_dense_bf16_tc(case["q"], case["k"], case["v"], sm)
    torch.cuda.synchronize()
    rows = synth.sample_rows(n, count, 11)
    ex = oracle.attn_exact(inp.q, inp.k, inp.v, sm, rows)
    got = out[rows].float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    lim = _bound(inp, rows, sm)
    excess = np.abs(got - ex) - lim
    assert excess.max() <= 0.0, (float(excess.max()), np.unravel_index(int(excess.argmax()), excess.shape))
    # and as a whole: bf16 rounding of P and of the output, a few 1e-3 at most
    assert float(np.linalg.norm(got - ex) / np.linalg.norm(ex)) <= 4e-3


def test_dense_tc_strided_output_and_status():
    """Into a token-major [N, H*D] output view (other columns untouched), with a caller workspace
    whose status block stays clear."""
    case = gpu_case("tails")
    n, h, d = case["q"].shape
    big = torch.full((n, 2 * h * d), -7.0, dtype=torch.bfloat16, device="cuda")
    view = big[:, h * d:].view(n, h, d)
    ws = sage.dense_workspace(n, h, d)
    sage.sage_attn_dense_bf16_tc(case["q"], case["k"], case["v"], out=view, ws=ws)
    ref = sage.sage_attn_dense_bf16_tc(case["q"], case["k"], case["v"])
    torch.cuda.synchronize()
    assert torch.equal(view, ref)
    assert bool((big[:, : h * d] == -7.0).all())
    assert sage.sage_check_device_status(ws[:256]) == (0, 0)


def test_dense_tc_close_to_fp32_dense_path():
    """The two dense paths differ by the bf16 rounding of P (and the output's last bit)."""
    case = gpu_case("strided64")
    tc = sage.sage_attn_dense_bf16_tc(case["q"], case["k"], case["v"]).float()
    f32 = sage.sage_attn_dense_bf16(case["q"], case["k"], case["v"]).float()
    torch.cuda.synchronize()
    assert float((tc - f32).norm() / f32.norm()) <= 4e-3


EDGE = [(1, 1, 128), (1, 2, 64), (100, 1, 128), (127, 1, 128), (129, 3, 64), (255, 2, 128), (257, 1, 64)]


@pytest.mark.parametrize("n,h,d", EDGE)
def test_dense_tc_edge_shapes(n, h, d):
    """Fewer tokens than one 128-row box (the tensor maps' boxes reach past N and read zeros),
    one key past a tile boundary, a second Q tile wholly in the padding, odd head counts."""
    inp = synth.make_inputs(synth.custom(n, h, d, "qkv", seed=7 * n + h + d, n_outlier=1))
    st = inp.storage.to("cuda")
    hd = h * d
    q, k, v = (st[:, i * hd:(i + 1) * hd].view(n, h, d) for i in range(3))
    sm = 1.0 / math.sqrt(d)
    ws = sage.dense_workspace(n, h, d)
    out = sage.sage_attn_dense_bf16_tc(q, k, v, sm, ws=ws)
    torch.cuda.synchronize()
    assert sage.sage_check_device_status(ws[:256]) == (0, 0)
    got = out.float().cpu().numpy().astype(np.float64)
    if n == 1:
        # softmax over one key: P = 1 exactly, so the output is that key's V
        assert torch.equal(out.cpu(), inp.v)
    rows = list(range(n))
    ex = oracle.attn_exact(inp.q, inp.k, inp.v, sm, rows)
    assert (np.abs(got - ex) - _bound(inp, rows, sm)).max() <= 0.0
