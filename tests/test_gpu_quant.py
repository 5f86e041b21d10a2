"""GPU parity of the smoothing / quantisation kernels against the CPU oracle: the K mean,
every INT8 Q/K code, every E4M3 V code and every scale must be bit-identical; so must the
INT8 V codes of the INT8 P.V variant, the V mean and the codes of smoothed V."""
import numpy as np
import pytest
import torch

import video_diffusion_transformer_sage_gb300 as sage
from conftest import gpu_case

pytestmark = pytest.mark.gpu

CASES = ["tiny", "tails", "strided64", "video"]


def _quantize(case):
    qz = sage.sage_smooth_quant_qk(case["q"], case["k"])
    sage.sage_quant_v(case["v"], qz)
    torch.cuda.synchronize()
    return qz


def _assert_same(gq, oq):
    n = oq.n
    assert np.array_equal(gq.k_mean.cpu().numpy().view(np.uint32), oq.k_mean.view(np.uint32))
    assert np.array_equal(gq.q_scales.cpu().numpy().view(np.uint32), oq.q_scales.view(np.uint32))
    assert np.array_equal(gq.k_scales.cpu().numpy().view(np.uint32), oq.k_scales.view(np.uint32))
    assert np.array_equal(gq.v_scales.cpu().numpy().view(np.uint32), oq.v_scales.view(np.uint32))
    qc = gq.q_codes.cpu().float().numpy()
    kc = gq.k_codes.cpu().float().numpy()
    assert np.array_equal(qc, oq.q_codes.astype(np.float32))
    assert np.array_equal(kc, oq.k_codes.astype(np.float32))
    assert np.array_equal(gq.v_codes.cpu().numpy(), oq.v_codes)
    # pad rows are zero
    assert not qc[:, n:].any() and not kc[:, n:].any() and not gq.v_codes[:, :, n:].any().item()


@pytest.mark.parametrize("name", CASES)
def test_quant_bit_exact(name):
    case = gpu_case(name)
    _assert_same(_quantize(case), case["qz"])


@pytest.mark.parametrize("name", CASES)
def test_quant_qkv_one_call_bit_exact(name):
    """sage_quant_qkv (K sums and V maxima in one launch, K mean and V scales in one) gives
    the oracle's codes, scales and mean bit for bit, as the two stage calls do."""
    case = gpu_case(name)
    qz = sage.sage_quant_qkv(case["q"], case["k"], case["v"])
    torch.cuda.synchronize()
    _assert_same(qz, case["qz"])


@pytest.mark.parametrize("opts", [dict(q_block=32), dict(v_format="int8"), dict(smooth_v=True),
                                  dict(q_block=1, v_format="int8", smooth_v=True)])
def test_quant_qkv_options_match_stage_calls(opts):
    """With options, sage_quant_qkv gives exactly what sage_smooth_quant_qk + sage_quant_v give,
    and its scratch contents do not matter."""
    case = gpu_case("tails")
    n, h, d = case["q"].shape
    a = sage.sage_smooth_quant_qk(case["q"], case["k"], **opts)
    sage.sage_quant_v(case["v"], a)
    scratch = torch.full((2 * sage.quant_scratch(n, h, d).numel(),), 0xAB, dtype=torch.uint8, device="cuda")
    b = sage.sage_quant_qkv(case["q"], case["k"], case["v"], scratch=scratch, **opts)
    torch.cuda.synchronize()
    for f in ("q_codes", "k_codes", "v_codes", "q_scales", "k_scales", "k_mean", "v_scales", "v_mean"):
        x, y = getattr(a, f), getattr(b, f)
        assert (x is None and y is None) or torch.equal(x, y), f


def test_hnd_layout_gives_identical_codes():
    """Strided-NHD and HND-contiguous inputs holding the same values quantise identically
    (the layout invariance the strided-NHD page reports as max_abs_difference 0)."""
    case = gpu_case("tails")
    hnd = gpu_case("tails_hndcopy")
    assert hnd["q"].stride(1) == case["q"].shape[0] * case["q"].shape[2]
    _assert_same(_quantize(hnd), case["qz"])


def test_quant_repeatable_and_scratch_reuse():
    case = gpu_case("tails")
    n, h, d = case["q"].shape
    scratch = sage.quant_scratch(n, h, d)
    scratch.fill_(0xAB)                      # scratch contents are ignored
    a = sage.sage_smooth_quant_qk(case["q"], case["k"], scratch=scratch)
    sage.sage_quant_v(case["v"], a, scratch=scratch)
    b = _quantize(case)
    torch.cuda.synchronize()
    for name in ("q_codes", "k_codes", "v_codes", "q_scales", "k_scales", "k_mean", "v_scales"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


@pytest.mark.parametrize("name,q_block", [("tails", 32), ("tails", 1), ("tails", 64), ("strided64", 32),
                                          ("strided64", 2), ("tiny", 16)])
def test_q_block_bit_exact(name, q_block):
    """Q scales per q_block rows (the per-warp granularity of the recorded kernel's warp_q, and
    finer): codes and scales bit-identical to the oracle's; K and V untouched."""
    case = gpu_case(name)
    import oracle
    codes, scales = oracle.quant_q(case["inp"].q, q_block)
    qz = sage.sage_smooth_quant_qk(case["q"], case["k"], q_block=q_block)
    torch.cuda.synchronize()
    assert qz.q_scales.shape == scales.shape
    assert np.array_equal(qz.q_scales.cpu().numpy().view(np.uint32), scales.view(np.uint32))
    assert np.array_equal(qz.q_codes.cpu().float().numpy(), codes.astype(np.float32))
    oq = case["qz"]
    assert np.array_equal(qz.k_codes.cpu().float().numpy(), oq.k_codes.astype(np.float32))
    assert np.array_equal(qz.k_scales.cpu().numpy().view(np.uint32), oq.k_scales.view(np.uint32))


V_OPTIONS = [("int8", False), ("int8", True), ("e4m3", True)]


def _quant_v_both(case, v_format, smooth):
    import oracle
    inp = case["inp"]
    n, h, d = inp.v.shape
    mean = oracle.channel_mean(inp.v) if smooth else None
    oc, osc = oracle.quant_v(inp.v, v_format, mean)
    gz = sage.Quantized(n, h, d, "cuda", v_format=v_format, smooth_v=smooth)
    sage.sage_quant_v(case["v"], gz)
    torch.cuda.synchronize()
    return gz, oc, osc, mean


def _assert_v_same(gz, oc, osc, mean, n):
    if mean is not None:
        assert np.array_equal(gz.v_mean.cpu().numpy().view(np.uint32), mean.view(np.uint32))
    assert np.array_equal(gz.v_scales.cpu().numpy().view(np.uint32), osc.view(np.uint32))
    if gz.v_format == "int8":
        got = gz.v_codes.cpu().float().numpy()
        assert np.array_equal(got, oc.astype(np.float32))      # the integer codes (+0 and -0 alike)
    else:
        got = gz.v_codes.cpu().numpy()
        assert np.array_equal(got, oc)
    assert not got[:, :, n:].any()


@pytest.mark.parametrize("name", ["tiny", "tails_voff", "strided64"])
@pytest.mark.parametrize("v_format,smooth", V_OPTIONS)
def test_v_options_bit_exact(name, v_format, smooth):
    case = gpu_case(name)
    _assert_v_same(*_quant_v_both(case, v_format, smooth), case["q"].shape[0])


def test_tiny_values_take_ieee_division():
    """A row, block or channel of values so small that its scale is subnormal (no finite
    reciprocal) still quantises exactly like the oracle's IEEE division.  The scaled rows
    also hold exact -0.0 (negative values that underflow bf16): IEEE -0 / s = -0, E4M3 0x80."""
    import oracle
    from video_diffusion_transformer_sage_gb300 import synth
    inp = synth.make_inputs(synth.custom(256, 2, 128, "qkv", seed=9, n_outlier=1))
    st = inp.storage.clone()
    hd = 2 * 128
    st[:130, :] = (st[:130, :].float() * 2.0 ** -124).to(torch.bfloat16)   # Q, K, V rows 0..129 tiny
    st[:, 2 * hd + 5] = (st[:, 2 * hd + 5].float() * 2.0 ** -124).to(torch.bfloat16)  # one V channel tiny
    q, k, v = (st[:, i * hd:(i + 1) * hd].view(256, 2, 128) for i in range(3))
    assert (v.view(torch.int16) == -32768).sum() >= 5                   # -0.0 present in V
    oz = oracle.Quantized(q, k, v, q_block=1)
    assert (oz.v_codes == 0x80).sum() > 100
    assert (oz.q_scales[:, :130] < 2.0 ** -126).sum() > 100 and (oz.q_scales[:, :130] > 0).all()
    assert 0 < oz.v_scales[0, 5] < 2.0 ** -126
    dst = st.cuda()
    dq, dk, dv = (dst[:, i * hd:(i + 1) * hd].view(256, 2, 128) for i in range(3))
    gz = sage.sage_smooth_quant_qk(dq, dk, q_block=1)
    sage.sage_quant_v(dv, gz)
    torch.cuda.synchronize()
    assert np.array_equal(gz.q_scales.cpu().numpy().view(np.uint32), oz.q_scales.view(np.uint32))
    assert np.array_equal(gz.q_codes.cpu().float().numpy(), oz.q_codes.astype(np.float32))
    assert np.array_equal(gz.v_scales.cpu().numpy().view(np.uint32), oz.v_scales.view(np.uint32))
    assert np.array_equal(gz.v_codes.cpu().numpy(), oz.v_codes)
    # the V options: the tiny channel's scale stays subnormal and takes the same IEEE route
    for fmt, smooth in V_OPTIONS:
        mean = oracle.channel_mean(v) if smooth else None
        oc, osc = oracle.quant_v(v, fmt, mean)
        assert 0 < osc[0, 5] < 2.0 ** -126, (fmt, smooth)
        gv = sage.Quantized(256, 2, 128, "cuda", v_format=fmt, smooth_v=smooth)
        sage.sage_quant_v(dv, gv)
        torch.cuda.synchronize()
        _assert_v_same(gv, oc, osc, mean, 256)
