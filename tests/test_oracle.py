"""Pins of the CPU oracle against facts fixed by the formats and the mathematics.

Each test names what it pins.  Nothing here runs on a GPU.
"""
import fractions
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from video_diffusion_transformer_sage_gb300 import synth


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def small_inputs(n=300, h=2, d=64, layout="qkv", seed=5, n_outlier=2, rms=False, bias_var=4.0):
    return synth.make_inputs(synth.custom(n, h, d, layout, seed, k_bias_var=bias_var,
                                          n_outlier=n_outlier, rms_norm=rms))


# ---------------------------------------------------------------- E4M3 (OCP FP8 format)

def test_e4m3_decode_closed_forms(oracle_lib):
    # largest finite, smallest subnormal, smallest normal, one, NaN, negative zero
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x3C) == 1.5
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    z = oracle.e4m3_decode(0x80)
    assert z == 0.0 and math.copysign(1.0, z) < 0
    assert oracle.e4m3_decode(0xFE) == -448.0


def test_e4m3_roundtrip_all_codes(oracle_lib):
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_e4m3_midpoints_ties_to_even(oracle_lib):
    vals = brute.e4m3_values()
    for i in range(len(vals) - 1):
        mid = 0.5 * (vals[i] + vals[i + 1])
        want = i if i % 2 == 0 else i + 1
        assert oracle.e4m3_encode(mid) == want, (i, mid)
        assert oracle.e4m3_encode(-mid) == (want | 0x80)


def test_e4m3_matches_torch_float8_cast(oracle_lib):
    """torch's float8_e4m3fn cast rounds to nearest-even within range (a library routine)."""
    g = torch.Generator().manual_seed(0)
    x = torch.cat([torch.randn(4000, generator=g, dtype=torch.float64) * s
                   for s in (1e-3, 1e-2, 0.1, 1.0, 10.0, 100.0)])
    vals = torch.tensor(brute.e4m3_values(), dtype=torch.float64)
    mids = 0.5 * (vals[:-1] + vals[1:])
    x = torch.cat([x, mids, -mids, vals, -vals]).clamp(-448.0, 448.0)
    ref = x.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(float(v)) for v in x.to(torch.float32).tolist()], np.uint8)
    # torch keeps the sign of zero; so does the oracle
    assert (ref == ours).all()


def test_e4m3_saturates(oracle_lib):
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(463.9) == 0x7E
    assert oracle.e4m3_encode(1e6) == 0x7E
    assert oracle.e4m3_encode(-500.0) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -11) == 0x00     # below half the smallest subnormal
    assert oracle.e4m3_encode(2.0 ** -10 * 1.0001) == 0x01


def test_e4m3_brute_agrees(oracle_lib):
    g = np.random.default_rng(1)
    x = np.concatenate([g.standard_normal(20000) * s for s in (1e-3, 0.1, 1, 30, 300)])
    ours = np.array([oracle.e4m3_encode(float(v)) for v in x], np.uint8)
    assert (ours == brute.e4m3_encode(x)).all()


# ---------------------------------------------------------------- K mean (smoothing)

def test_k_mean_constant_column_exact(oracle_lib):
    inp = small_inputs(n=1000, h=2, d=64, layout="nhd")
    k = inp.k.clone()
    k[:, 0, :] = 0.375
    k[:, 1, 5] = -3.0
    mu = oracle.k_mean(k)
    assert (mu[0] == np.float32(0.375)).all()
    assert mu[1, 5] == np.float32(-3.0)


def test_k_mean_vs_exact_rational(oracle_lib):
    """mu is within the fp32 chunk-summation error bound of the exact rational mean."""
    inp = small_inputs(n=4100, h=3, d=64, layout="qkv")
    mu = oracle.k_mean(inp.k)
    kf = inp.k.float().numpy().astype(np.float64)
    n = kf.shape[0]
    u = 2.0 ** -24
    for hh, c in [(0, 0), (1, 17), (2, 63), (0, 31)]:
        col = kf[:, hh, c]
        exact = sum((fractions.Fraction(float(x)) for x in col), fractions.Fraction(0)) / n
        bound = 127 * u * np.abs(col).sum() / n + 2 * u * abs(float(exact)) + 1e-30
        assert abs(float(mu[hh, c]) - float(exact)) <= bound


def test_smoothing_invariance_of_softmax():
    """softmax(q (k - mu)^T) == softmax(q k^T) row by row, so O_exact needs no mean correction."""
    g = np.random.default_rng(2)
    q, k, v = g.standard_normal((3, 50, 2, 32))
    mu = g.standard_normal((2, 32)) * 3
    a = brute.attn_exact(q, k, v, 0.2)
    b = brute.attn_exact(q, k - mu[None], v, 0.2)
    assert np.abs(a - b).max() < 1e-12


# ---------------------------------------------------------------- INT8 / E4M3 quantisation

@pytest.mark.parametrize("layout", ["nhd", "qkv", "hnd"])
def test_quant_matches_brute(oracle_lib, layout):
    inp = small_inputs(n=300, h=2, d=64, layout=layout)
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    qf = inp.q.float().numpy().transpose(1, 0, 2)
    kf = (inp.k.float().numpy() - qz.k_mean[None]).astype(np.float32).transpose(1, 0, 2)
    vf = inp.v.float().numpy().transpose(1, 0, 2)
    bq, bqs = brute.quant_int8_blocks(np.ascontiguousarray(qf), 128)
    bk, bks = brute.quant_int8_blocks(np.ascontiguousarray(kf), 64)
    bv, bvs = brute.quant_v(np.ascontiguousarray(vf))
    assert (bq == qz.q_codes).all() and (bqs == qz.q_scales).all()
    assert (bk == qz.k_codes).all() and (bks == qz.k_scales).all()
    assert (bv == qz.v_codes).all() and (bvs == qz.v_scales).all()


def test_int8_error_bound_and_range(oracle_lib):
    inp = synth.make_inputs("tails")
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    n = inp.q.shape[0]
    for codes, scales, block, x in (
            (qz.q_codes, qz.q_scales, 128, inp.q.float().numpy()),
            (qz.k_codes, qz.k_scales, 64, inp.k.float().numpy() - qz.k_mean[None])):
        xs = x.transpose(1, 0, 2)                                  # [H, N, D]
        s = np.repeat(scales, block, axis=1)[:, :n, None].astype(np.float64)
        deq = codes[:, :n].astype(np.float64) * s
        assert (np.abs(deq - xs) <= s * 0.5 * (1 + 2e-5) + 1e-30).all()
        assert np.abs(codes).max() <= 127
        # every nonzero block holds a code of magnitude 127 (its max element)
        nb = scales.shape[1]
        cb = np.abs(codes.astype(np.int32)).reshape(codes.shape[0], nb, block, -1).max(axis=(2, 3))
        assert ((cb == 127) | (scales == 0)).all()
        assert (codes[:, n:] == 0).all()


def test_v_quant_error_bound(oracle_lib):
    inp = small_inputs(n=500, h=2, d=64, layout="nhd")
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    v = inp.v.float().numpy().astype(np.float64)       # [N, H, D]
    dec = brute.e4m3_decode(qz.v_codes[:, :, :500])   # [H, D, N]
    deq = dec * qz.v_scales[:, :, None]
    vt = v.transpose(1, 2, 0)
    # half an E4M3 ulp at the value's magnitude: ulp = 2^(floor(log2|y|) - 3), >= 2^-9
    y = np.abs(vt / qz.v_scales[:, :, None])
    ulp = np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(y, 1e-30))) - 3))
    assert (np.abs(deq - vt) <= 0.5 * ulp * qz.v_scales[:, :, None] * (1 + 1e-6)).all()
    assert (np.abs(dec).max(axis=2) == 448.0).all()


def test_all_zero_block(oracle_lib):
    inp = small_inputs(n=256, h=1, d=64, layout="nhd")
    q = inp.q.clone()
    q[:128] = 0
    codes, scales = oracle.quant_q(q)
    assert scales[0, 0] == 0 and (codes[0, :128] == 0).all() and scales[0, 1] > 0


# ---------------------------------------------------------------- integer S and attention

def test_qk_int32_matches_integer_matmul(oracle_lib):
    inp = small_inputs(n=300, h=2, d=64)
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    S = oracle.qk_int32(qz, 1, 128, 64, 100, 200)
    ref = qz.q_codes[1, 128:228].astype(np.int64) @ qz.k_codes[1, 64:264].astype(np.int64).T
    assert (S == ref).all()
    # worst case magnitude fits: all +-127
    qz.q_codes[0, :128] = 127
    qz.k_codes[0, :128] = -127
    S = oracle.qk_int32(qz, 0, 0, 0, 4, 4)
    assert (S == -127 * 127 * 64).all()


def test_attn_exact_matches_brute(oracle_lib):
    inp = small_inputs(n=200, h=2, d=64, layout="qkv")
    rows = list(range(200))
    a = oracle.attn_exact(inp.q, inp.k, inp.v, 0.125, rows)
    b = brute.attn_exact(inp.q.float().numpy(), inp.k.float().numpy(), inp.v.float().numpy(), 0.125)
    assert np.abs(a - b).max() < 1e-12


def test_attn_exact_rows_sum_to_one(oracle_lib):
    inp = small_inputs(n=300, h=2, d=64, layout="nhd")
    v = torch.ones_like(inp.v)
    o = oracle.attn_exact(inp.q, inp.k, v, 0.125, [0, 7, 299])
    assert np.abs(o - 1.0).max() < 1e-12


def test_constant_keys_give_mean_of_v(oracle_lib):
    inp = small_inputs(n=300, h=2, d=64, layout="nhd")
    k = torch.empty_like(inp.k)
    k[:] = inp.k[3]
    o = oracle.attn_exact(inp.q, k, inp.v, 0.125, [0, 150])
    mean_v = inp.v.double().mean(dim=0).numpy()
    assert np.abs(o - mean_v[None]).max() < 1e-12
    # the quantised path: K~ = 0 -> all codes 0 -> uniform P8 -> O_sq = mean of dequantised V
    qz = oracle.Quantized(inp.q, k, inp.v)
    assert (qz.k_codes == 0).all()
    osq = oracle.attn_sq(qz, 0.125, [0, 150], tile=128)
    vdeq = brute.e4m3_decode(qz.v_codes[:, :, :300]) * qz.v_scales[:, :, None]
    assert np.abs(osq - vdeq.mean(axis=2)[None]).max() < 1e-12


def test_one_hot_query_selects_value(oracle_lib):
    n, h, d = 200, 1, 64
    inp = small_inputs(n=n, h=h, d=d, layout="nhd", n_outlier=0)
    q = torch.zeros_like(inp.q)
    q[:, 0, 0] = 8.0
    k = torch.zeros_like(inp.k)
    k[:, 0, 0] = torch.linspace(-1, 1, n).to(torch.bfloat16)
    k[77, 0, 0] = 4.0
    o = oracle.attn_exact(q, k, inp.v, 1.0, [5])
    assert np.abs(o[0, 0] - inp.v[77, 0].double().numpy()).max() < 1e-6


def test_attn_sq_matches_brute_global(oracle_lib):
    inp = small_inputs(n=300, h=2, d=64, layout="qkv")
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    rows = list(range(300))
    a = oracle.attn_sq(qz, 0.125, rows, tile=0)
    b = brute.attn_sq_global(qz.q_codes, qz.q_scales, qz.k_codes, qz.k_scales, qz.v_codes,
                             qz.v_scales, 300, 0.125)
    assert np.abs(a - b).max() < 1e-12


def test_attn_sq_single_tile_equals_global(oracle_lib):
    inp = small_inputs(n=128, h=2, d=64, layout="nhd")
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    rows = list(range(128))
    a = oracle.attn_sq(qz, 0.125, rows, tile=128, score_f32=False)
    b = oracle.attn_sq(qz, 0.125, rows, tile=0)
    assert (a == b).all()


# ---------------------------------------------------------------- fp32-scored schedule vs fp64
# The online schedule can form its base-2 scores in fp32 (the precision in which the kernel decides
# P's codes) or in fp64.  Both visit the same 128-key tiles against the same running max, so key by
# key they may differ only by rounding: the pins below bound that difference from the arithmetic
# and show that a P code differs only where the fp64 value lies within that bound of a rounding
# boundary of the code.

U32 = 2.0 ** -24          # fp32 unit roundoff


def _midpoints(v_format: str) -> np.ndarray:
    """Rounding boundaries of P's code: midpoints of adjacent E4M3 values, or the half-integers."""
    if v_format == "int8":
        return np.arange(0, 128) + 0.5
    vals = brute.e4m3_values()
    return 0.5 * (vals[:-1] + vals[1:])


def _score_bound(pp64: np.ndarray, lw: np.ndarray, v_format: str) -> np.ndarray:
    """Relative bound on |pp32 - pp64| / pp64 for one key.  With x = log2(pp) = S c + b the base-2
    score, b = log2(P scale) - m and m the running max (base 2): c = s_q (sm log2 e) s_k carries five
    fp32 roundings (the fp32 sm, log2 e, and three products), the fused multiply-add one, b two
    (the constant log2(P scale), the subtraction), m its own (up to 6: c's five, one product); 2^x
    is rounded once to fp32.  A deviation e in x scales pp by 2^e, i.e. by ln2 e to first order.
    The factor 2 covers the second-order terms and a running max that rises in one mode and stays
    (within rounding) in the other."""
    with np.errstate(divide="ignore"):
        x = np.log2(np.where(pp64 > 0, pp64, 1.0))
    b = np.log2(127.0 if v_format == "int8" else 448.0) - lw
    ex = U32 * (5 * np.abs(x - b) + np.abs(x) + 9 + 6 * np.abs(lw) + np.abs(b))
    return 2.0 * (math.log(2.0) * ex + U32)


def _v_values(qz, head: int) -> np.ndarray:
    """Dequantisation-free values of V's codes of one head: [D, N] (E4M3 numbers or INT8 integers)."""
    c = qz.v_codes[head, :, :qz.n]
    return c.astype(np.float64) if getattr(qz, "v_format", "e4m3") == "int8" else brute.e4m3_decode(c)


def _reconstruction_error(qz, head: int, out, pp, p8, lw) -> float:
    """The output rebuilt from the trace without any running rescale: O_c = sum_j P8_j w_j v_jc s_v[c] /
    sum_j pp_j w_j (+ the V mean), w_j = 2^(lw_j - lw_last).  Largest relative deviation."""
    w = np.exp2(lw - lw[:, -1:])
    vv = _v_values(qz, head)                                       # [D, N]
    num = (p8 * w) @ vv.T * qz.v_scales[head][None, :].astype(np.float64)
    rec = num / (pp * w).sum(axis=1, keepdims=True)
    if getattr(qz, "v_mean", None) is not None:
        rec = rec + qz.v_mean[head][None, :].astype(np.float64)
    return float(np.abs(rec - out).max() / max(np.abs(out).max(), 1e-300))


def _fp32_mode_agreement(qz, sm: float, rows, heads) -> dict:
    """Key by key agreement of the fp32-scored and fp64-scored schedules (128-key tiles)."""
    fmt = getattr(qz, "v_format", "e4m3")
    mids = _midpoints(fmt)
    keys = flips = at_risk = small = 0
    worst = recon = 0.0
    flips_outside = 0
    for head in heads:
        o32, pp32, p832, lw32 = oracle.attn_sq_trace(qz, sm, head, rows, tile=128, score_f32=True)
        o64, pp64, p864, lw64 = oracle.attn_sq_trace(qz, sm, head, rows, tile=128, score_f32=False)
        recon = max(recon, _reconstruction_error(qz, head, o32, pp32, p832, lw32),
                    _reconstruction_error(qz, head, o64, pp64, p864, lw64))
        big = pp64 >= 2.0 ** -120
        small += int((~big).sum())
        # below 2^-120 both values are far under the smallest code: both codes 0
        if (p832[~big] != 0).any() or (p864[~big] != 0).any() or (pp32[~big] > 2.0 ** -100).any():
            worst = math.inf
        bnd = _score_bound(pp64, lw64, fmt)
        rel = np.abs(pp32 - pp64) / np.where(big, pp64, 1.0)
        worst = max(worst, float((rel / bnd)[big].max()))
        i = np.clip(np.searchsorted(mids, pp64), 1, len(mids) - 1)
        dist = np.minimum(np.abs(pp64 - mids[i - 1]), np.abs(pp64 - mids[i]))
        risky = big & (dist <= bnd * pp64)
        flip = p832 != p864
        keys += int(big.sum())
        at_risk += int(risky.sum())
        flips += int(flip.sum())
        flips_outside += int((flip & ~risky).sum())
    return dict(keys=keys, tiny_keys=small, at_risk=at_risk, flips=flips, flips_outside=flips_outside,
                worst_over_bound=worst, reconstruction=recon)


def _agreement_holds(a: dict) -> bool:
    return (a["worst_over_bound"] <= 1.0 and a["flips_outside"] == 0 and a["reconstruction"] < 1e-12
            and a["flips"] <= max(8, 1e-4 * a["keys"]))


@pytest.mark.parametrize("name,nrows,v_format", [("tiny", None, "e4m3"), ("tails", 64, "e4m3"),
                                                  ("tails", 64, "int8"), ("strided64", 24, "e4m3")])
def test_fp32_scores_agree_with_fp64_key_by_key(oracle_lib, name, nrows, v_format):
    """For every (row, head, key): the fp32-scored 448 p is within the rounding bound of the
    fp64-scored one; a P code differs only where the fp64 value lies within that bound of a rounding
    boundary, and such keys are rare; and each mode's output is exactly what its trace of codes and
    running maxima gives without any running rescale."""
    inp = synth.make_inputs(name)
    qz = oracle.Quantized(inp.q, inp.k, inp.v, v_format=v_format)
    n, h, d = inp.q.shape
    rows = list(range(n)) if nrows is None else synth.sample_rows(n, nrows, 3)
    a = _fp32_mode_agreement(qz, 1 / math.sqrt(d), rows, range(h))
    print(name, v_format, a)
    assert _agreement_holds(a), a


def test_fp32_scores_agree_with_fp64_video_sample(oracle_lib):
    """The same key-by-key agreement on the full video shape (N=37810, H=56, D=128): 8 query rows
    (both ends, the segment borders 99/100/513/514 and the last tile's first two) against every
    key of every head."""
    inp = synth.make_inputs("video")
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    n, h, d = inp.q.shape
    rows = synth.sample_rows(n, 4, 7)
    a = _fp32_mode_agreement(qz, 1 / math.sqrt(d), rows, range(h))
    print("video", a)
    assert _agreement_holds(a), a


def _tiled_exact_case_error() -> float:
    """Scores that are integer multiples of ln 2 make every p an exact power of two, which
    E4M3 holds exactly, so tiled mode (with its rescales on each rise of the running max)
    must equal global mode and the closed form sum_j 2^k_j v_j / sum_j 2^k_j.  Returns the
    largest deviation from either."""
    n, d = 384, 64
    inp = small_inputs(n=n, h=1, d=d, layout="nhd")
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    g = np.random.default_rng(3)
    kexp = g.integers(-6, 1, size=n)                 # exponents in [-6, 0]
    kexp[: n // 3] -= 2                             # first tile lower: max rises later
    kexp[n - 5] = 1                                 # global max in the last tile
    qz.q_codes[:] = 0
    qz.q_codes[0, :n, 0] = 1
    qz.k_codes[:] = 0
    qz.k_codes[0, :n, 0] = kexp
    qz.q_scales[:] = 1.0
    qz.k_scales[:] = 1.0
    rows = [0, 5, 200]
    t = oracle.attn_sq(qz, math.log(2.0), rows, tile=128, score_f32=False)
    gl = oracle.attn_sq(qz, math.log(2.0), rows, tile=0)
    w = 2.0 ** (kexp - kexp.max())
    vdeq = brute.e4m3_decode(qz.v_codes[0, :, :n]) * qz.v_scales[0][:, None]   # [D, N]
    closed = (vdeq @ w) / w.sum()
    return max(np.abs(t - gl).max(), np.abs(t[:, 0] - closed[None]).max())


def test_attn_sq_tiled_rescale_exact_case(oracle_lib):
    assert _tiled_exact_case_error() < 1e-12


def test_attn_sq_method_gap_to_exact(oracle_lib):
    """Same-quantisation attention stays near exact attention; on N(0,1) values E4M3 V and
    P each cost about 2.5 % relative L2 (3 mantissa bits), which bounds the method's gap."""
    inp = synth.make_inputs("tiny")
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    rows = synth.sample_rows(1024, 64, 0)
    sm = 1 / math.sqrt(128)
    t = oracle.attn_sq(qz, sm, rows, tile=128)
    gl = oracle.attn_sq(qz, sm, rows, tile=0)
    e = oracle.attn_exact(inp.q, inp.k, inp.v, sm, rows)
    assert rel_l2(t, e) < 5e-2 and rel_l2(gl, e) < 5e-2
    assert rel_l2(t, gl) < 4e-2


def test_page_shapes_golden():
    """Tile counts of the pages' attention call, printed on the pages."""
    import json, os
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_shapes.json")))
    _, n, h, d = gold["q_shape"]["value"]
    segs = gold["segments"]["value"]
    assert segs[-1][1] == n == gold["packed_tokens"]["value"] == synth.WORKLOADS["video"].n_tokens
    assert sum(e - s for s, e, _ in segs) == n
    assert tuple(map(tuple, segs)) == synth.VIDEO_SEGMENTS
    cta_q = gold["scheduler"]["value"]["cta_q"]
    assert oracle.pad128(n) // cta_q * h == gold["scheduler"]["value"]["grid_ctas"]
    assert abs(synth.WORKLOADS["video"].flops - 40.989e12) / 40.989e12 < 1e-4


# ---------------------------------------------------------------- Q-scale granularity
# Q scales per q_block consecutive rows (q_block | 128): the method's 128 by default, 32 the
# per-warp granularity of the recorded kernel's warp_q, 1 per row.

@pytest.mark.parametrize("q_block", [1, 2, 8, 32, 64, 128])
def test_q_block_quant_matches_brute(oracle_lib, q_block):
    inp = small_inputs(n=300, h=2, d=64, layout="qkv")
    codes, scales = oracle.quant_q(inp.q, q_block)
    qf = np.ascontiguousarray(inp.q.float().numpy().transpose(1, 0, 2))
    bq, bqs = brute.quant_int8_blocks(qf, q_block)
    assert scales.shape == (2, 384 // q_block)
    assert (bq == codes).all() and (bqs == scales).all()
    assert (scales[:, 300 // q_block + (300 % q_block > 0):] == 0).all()   # blocks wholly in the padding


def test_q_block_128_is_the_default(oracle_lib):
    inp = small_inputs(n=300, h=2, d=64, layout="qkv")
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    c, s = oracle.quant_q(inp.q, 128)
    assert qz.q_block == 128 and (qz.q_codes == c).all() and (qz.q_scales == s).all()


def test_q_block_scales_nest(oracle_lib):
    """The max over a 128-row block is the max of its sub-blocks' maxima, and x -> fl32(x/127)
    is monotone, so the 128-row scale equals the largest scale of the finer blocks inside it."""
    inp = synth.make_inputs("tails")
    _, s128 = oracle.quant_q(inp.q, 128)
    for qb in (1, 4, 32, 64):
        _, s = oracle.quant_q(inp.q, qb)
        assert (s.reshape(s.shape[0], -1, 128 // qb).max(axis=2) == s128).all(), qb


def test_q_block_per_row_error_bound(oracle_lib):
    """Per-row scales: each row's largest |code| is 127 (unless the row is zero) and every
    element dequantises to within half its row's scale."""
    inp = synth.make_inputs("tails")
    codes, s = oracle.quant_q(inp.q, 1)
    n = inp.q.shape[0]
    x = inp.q.float().numpy().transpose(1, 0, 2).astype(np.float64)
    sc = s[:, :n, None].astype(np.float64)
    assert (np.abs(codes[:, :n].astype(np.float64) * sc - x) <= sc * 0.5 * (1 + 2e-5) + 1e-30).all()
    rowmax = np.abs(codes[:, :n].astype(np.int32)).max(axis=2)
    assert ((rowmax == 127) | (s[:, :n] == 0)).all()


@pytest.mark.parametrize("q_block", [1, 32])
def test_q_block_attention_matches_brute(oracle_lib, q_block):
    inp = small_inputs(n=300, h=2, d=64, layout="qkv")
    qz = oracle.Quantized(inp.q, inp.k, inp.v, q_block=q_block)
    rows = list(range(300))
    a = oracle.attn_sq(qz, 0.125, rows, tile=0)
    b = brute.attn_sq_global(qz.q_codes, qz.q_scales, qz.k_codes, qz.k_scales, qz.v_codes,
                             qz.v_scales, 300, 0.125, q_block=q_block)
    assert np.abs(a - b).max() < 1e-12
    t = oracle.attn_sq(qz, 0.125, rows[:128], tile=512, score_f32=False)   # one tile = global
    assert (t == a[:128]).all()


# ---------------------------------------------------------------- qk_transform: RMSNorm + RoPE

def _rr_inputs(n=96, h=3, d=128, seed=3):
    inp = small_inputs(n=n, h=h, d=d, layout="qkv", seed=seed)
    gq, _ = synth.qk_norm_weights(d)
    cos, sin = synth.rope_table(synth.rope_positions(n, n_text=20, grid=(2, 4, 10)), d)
    return inp, gq.numpy(), cos.numpy(), sin.numpy()


def _rr_closed_forms_hold() -> bool:
    """The two closed forms below, as one boolean (also used by the planted-mistake battery)."""
    for d in (64, 128):
        x = torch.full((5, 2, d), 2.0, dtype=torch.bfloat16)
        oracle.rmsnorm_rope(x, np.ones(d), np.ones((5, d // 2)), np.zeros((5, d // 2)), 0.0)
        if not (x.float() == 1.0).all():
            return False
    inp, g, _, _ = _rr_inputs()
    n, h, d = inp.q.shape
    a, b = inp.q.contiguous().clone(), inp.q.contiguous().clone()
    oracle.rmsnorm_rope(a, g, np.ones((n, d // 2)), np.zeros((n, d // 2)), 1e-6)
    oracle.rmsnorm_rope(b, g, np.zeros((n, d // 2)), np.ones((n, d // 2)), 1e-6)
    ab, bb = a.view(torch.int16).numpy(), b.view(torch.int16).numpy()
    return bool((bb[..., 1::2] == ab[..., 0::2]).all() and
                (bb[..., 0::2] == (ab[..., 1::2] ^ np.int16(-32768))).all())


def test_rmsnorm_rope_closed_forms(oracle_lib):
    """(1) x = 2 everywhere, eps = 0, gamma = 1, no turn: mean square 4, r = 1/2, every output
    exactly 1.  (2) A quarter turn (cos 0, sin 1): z_2i = -y_2i+1 and z_2i+1 = y_2i exactly,
    i.e. the unturned result with each pair swapped and its first element negated."""
    assert _rr_closed_forms_hold()


def test_rmsnorm_rope_gamma_power_of_two_scales_exactly(oracle_lib):
    inp, g, cos, sin = _rr_inputs()
    a, b = inp.k.contiguous().clone(), inp.k.contiguous().clone()
    oracle.rmsnorm_rope(a, g, cos, sin, 1e-6)
    oracle.rmsnorm_rope(b, 2.0 * g, cos, sin, 1e-6)
    assert torch.equal(b.float(), 2.0 * a.float())


@pytest.mark.parametrize("d", [64, 128])
def test_rmsnorm_rope_matches_brute(oracle_lib, d):
    inp, g, cos, sin = _rr_inputs(d=d)
    x = inp.q.contiguous().clone()
    want = brute.rmsnorm_rope(x.float().numpy(), g, cos, sin, 1e-6)
    got = oracle.rmsnorm_rope(x, g, cos, sin, 1e-6).float().numpy().astype(np.float64)
    # bf16 rounding (half an ulp, 2^-9 relative) plus the fp32 arithmetic before it
    assert (np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-6 * np.abs(want).max()).all()


def test_rmsnorm_rope_unit_rms(oracle_lib):
    """gamma = 1: the rotation keeps each pair's norm, so every (token, head) row leaves with
    mean square ms / (ms + eps) -- 1 to within the bf16 rounding of its elements."""
    inp, _, cos, sin = _rr_inputs()
    x = oracle.rmsnorm_rope(inp.v.contiguous().clone(), np.ones(128), cos, sin, 1e-6).float().numpy()
    ms = (x.astype(np.float64) ** 2).mean(axis=2)
    assert np.abs(ms - 1.0).max() < 2.0 ** -7


def test_rmsnorm_rope_in_place_on_strided_views(oracle_lib):
    """On the Q slice of a token-major QKV buffer: the K and V slices stay untouched, and Q
    becomes what the same op gives on a contiguous copy."""
    inp, g, cos, sin = _rr_inputs()
    before = inp.storage.clone()
    ref = oracle.rmsnorm_rope(inp.q.contiguous().clone(), g, cos, sin, 1e-6)
    oracle.rmsnorm_rope(inp.q, g, cos, sin, 1e-6)
    hd = inp.q.shape[1] * inp.q.shape[2]
    assert torch.equal(inp.storage[:, hd:].view(torch.int16), before[:, hd:].view(torch.int16))
    assert torch.equal(inp.q.contiguous().view(torch.int16), ref.view(torch.int16))


# ---------------------------------------------------------------- V options: INT8 P.V, V smoothing

def _grid_inputs(n=256, h=2, d=64, seed=11):
    """Q, K and V whose V values lie on a 2^-4 grid in (-2, 2): with n a power of two, the channel
    mean of V, of V + c (c in {2, 4, 8}) and every difference v - mean are exact in fp32."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(n, h, d, generator=g).to(torch.bfloat16)
    k = (torch.randn(n, h, d, generator=g) + 2.0 * torch.randn(1, h, d, generator=g)).to(torch.bfloat16)
    v = (torch.randint(-31, 32, (n, h, d), generator=g).float() / 16.0).to(torch.bfloat16)
    return q, k, v


def _shift_error(v_format: str) -> float:
    """|O(V + c) - O(V) - c| for smoothed V, c a per-channel constant: smoothing removes c before
    quantisation (same codes, same scales) and the attention adds the mean, c included, back."""
    q, k, v = _grid_inputs()
    c = torch.tensor([2.0, 4.0, 8.0])[torch.arange(v.shape[2]) % 3]
    v2 = (v.float() + c).to(torch.bfloat16)
    assert torch.equal(v2.float() - c, v.float())           # the shift is exact in bf16
    a = oracle.Quantized(q, k, v, v_format=v_format, smooth_v=True)
    b = oracle.Quantized(q, k, v2, v_format=v_format, smooth_v=True)
    assert (a.v_codes == b.v_codes).all() and (a.v_scales == b.v_scales).all()
    rows = list(range(0, 256, 5))
    oa = oracle.attn_sq(a, 0.125, rows, tile=128)
    ob = oracle.attn_sq(b, 0.125, rows, tile=128)
    return float(np.abs(ob - oa - c.double().numpy()[None, None, :]).max())


def _int8_two_level_error() -> float:
    """Closed form of the INT8 P.V variant: 64 keys score +s0 and 64 score -s0 for every query, so
    p is 1 or exp(-2 s0) and P's codes are 127 and rint(127 exp(-2 s0)) (= 47 for 2 s0 = 1); with V
    = +1 on the high keys and -1 on the low ones (codes +-127), every output is
    (127 - 47) / (127 (1 + exp(-1))) times the dequantised 1."""
    n, h, d = 128, 1, 64
    q = torch.zeros(n, h, d)
    q[:, 0, 0] = 1.0
    k = torch.zeros(n, h, d)
    k[:64, 0, 0] = 1.0
    k[64:, 0, 0] = -1.0
    v = torch.zeros(n, h, d)
    v[:64] = 1.0
    v[64:] = -1.0
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    qz = oracle.Quantized(q, k, v, v_format="int8")
    s_q, s_k, s_v = float(qz.q_scales[0, 0]), float(qz.k_scales[0, 0]), float(qz.v_scales[0, 0])
    assert (qz.k_codes[0, :64, 0] == 127).all() and (qz.v_codes[0, :, :64] == 127).all()
    sm = 0.5 / (127 * 127 * s_q * s_k)                      # s0 = 0.5 up to the fp32 scales
    s0 = 127 * 127 * s_q * s_k * sm
    low = math.exp(-2 * s0)
    code_low = float(np.rint(127 * low))
    assert code_low == 47.0
    want = (127 - code_low) * 127 * s_v / (127 * (1 + low))
    got = oracle.attn_sq(qz, sm, list(range(0, n, 9)), tile=0)
    err = float(np.abs(got - want).max())
    tiled = oracle.attn_sq(qz, sm, list(range(0, n, 9)), tile=128, score_f32=False)
    return max(err, float(np.abs(tiled - want).max()))


@pytest.mark.parametrize("smooth", [False, True])
def test_v_int8_quant_matches_brute(oracle_lib, smooth):
    inp = small_inputs(n=333, h=2, d=64, layout="nhd")
    mu = oracle.channel_mean(inp.v) if smooth else None
    codes, scales = oracle.quant_v(inp.v, "int8", mu)
    vf = np.ascontiguousarray(inp.v.float().numpy().transpose(1, 0, 2))
    bc, bs = brute.quant_v(vf, "int8", mu)
    assert (codes == bc).all() and (scales == bs).all()
    x = vf - (mu[:, None, :] if smooth else 0)
    deq = codes[:, :, :333].astype(np.float64) * scales[:, :, None]
    # half a step, plus the fp32 rounding of the quotient x / scale (|x / scale| <= 127)
    assert (np.abs(deq - x.transpose(0, 2, 1)) <= (0.5 + 2.0 ** -16) * scales[:, :, None]).all()
    assert (np.abs(codes[:, :, :333]).max(axis=2) == 127).all() and (codes[:, :, 333:] == 0).all()


def test_v_e4m3_smoothed_quant_matches_brute(oracle_lib):
    inp = small_inputs(n=333, h=2, d=64, layout="qkv")
    mu = oracle.channel_mean(inp.v)
    codes, scales = oracle.quant_v(inp.v, "e4m3", mu)
    bc, bs = brute.quant_v(np.ascontiguousarray(inp.v.float().numpy().transpose(1, 0, 2)), "e4m3", mu)
    assert (codes == bc).all() and (scales == bs).all()
    # the unsmoothed call of the same function is the method's default V quantisation
    c0, s0 = oracle.quant_v(inp.v, "e4m3", None)
    c1 = np.zeros_like(c0)
    s1 = np.zeros_like(s0)
    p, st, sh = inp.v.data_ptr(), inp.v.stride(0), inp.v.stride(1)
    oracle.lib().oracle_quant_v_fmt(p, 333, 2, 64, st, sh, None, 0, c1.ctypes.data, s1.ctypes.data)
    assert (c0 == c1).all() and (s0 == s1).all()


@pytest.mark.parametrize("v_format", ["e4m3", "int8"])
def test_v_smoothing_shift_invariance(oracle_lib, v_format):
    assert _shift_error(v_format) < 1e-12


@pytest.mark.parametrize("v_format", ["e4m3", "int8"])
def test_constant_v_smoothed_gives_the_constant(oracle_lib, v_format):
    """V constant per channel: V - mean = 0 exactly, so scales and codes are 0 and the output is
    the constant, whatever the scores."""
    inp = small_inputs(n=300, h=2, d=64, layout="nhd")
    v = inp.v[5:6].expand(300, 2, 64).contiguous()
    qz = oracle.Quantized(inp.q, inp.k, v, v_format=v_format, smooth_v=True)
    assert (qz.v_scales == 0).all() and (qz.v_codes == 0).all()
    o = oracle.attn_sq(qz, 0.125, [0, 150, 299], tile=128)
    assert (o == v[0].double().numpy()[None]).all()


@pytest.mark.parametrize("smooth", [False, True])
def test_int8_pv_attn_matches_brute_global(oracle_lib, smooth):
    inp = small_inputs(n=300, h=2, d=64, layout="qkv")
    qz = oracle.Quantized(inp.q, inp.k, inp.v, v_format="int8", smooth_v=smooth)
    rows = list(range(300))
    a = oracle.attn_sq(qz, 0.125, rows, tile=0)
    b = brute.attn_sq_global(qz.q_codes, qz.q_scales, qz.k_codes, qz.k_scales, qz.v_codes, qz.v_scales,
                             300, 0.125, v_format="int8", v_mean=qz.v_mean)
    assert np.abs(a - b).max() < 1e-12


def test_int8_pv_uniform_attention(oracle_lib):
    """Constant K: K~ = 0, every score 0, p = 1, every P code 127 and l = 127 N: the output is the
    mean of the dequantised INT8 V."""
    inp = small_inputs(n=300, h=2, d=64, layout="nhd")
    k = inp.k[3:4].expand(300, 2, 64).contiguous()
    qz = oracle.Quantized(inp.q, k, inp.v, v_format="int8")
    o = oracle.attn_sq(qz, 0.125, [0, 150, 299], tile=128)
    vdeq = qz.v_codes[:, :, :300].astype(np.float64) * qz.v_scales[:, :, None]
    assert np.abs(o - vdeq.mean(axis=2)[None]).max() < 1e-12


def test_int8_pv_two_level_closed_form(oracle_lib):
    assert _int8_two_level_error() < 1e-12


@pytest.mark.parametrize("v_format", ["e4m3", "int8"])
def test_tiled_schedule_close_to_global(oracle_lib, v_format):
    """The online schedule (P coded against the running max, fp32 scores) against the one-pass
    definition: the difference is P's coding noise only."""
    inp = small_inputs(n=600, h=2, d=64, layout="qkv")
    qz = oracle.Quantized(inp.q, inp.k, inp.v, v_format=v_format, smooth_v=True)
    rows = list(range(0, 600, 7))
    assert rel_l2(oracle.attn_sq(qz, 0.125, rows, tile=128), oracle.attn_sq(qz, 0.125, rows, tile=0)) < 2e-2


def test_v_smoothing_lowers_error_on_offset_v(oracle_lib):
    """A large per-channel offset in V costs E4M3 precision on the part that varies; taking the
    mean out first brings the quantised output closer to exact attention."""
    inp = small_inputs(n=400, h=2, d=64, layout="nhd")
    g = torch.Generator().manual_seed(3)
    v = (inp.v.float() + 20.0 * torch.randn(1, 2, 64, generator=g)).to(torch.bfloat16)
    rows = list(range(0, 400, 11))
    exact = oracle.attn_exact(inp.q, inp.k, v, 0.125, rows)
    plain = oracle.attn_sq(oracle.Quantized(inp.q, inp.k, v), 0.125, rows, tile=128)
    smooth = oracle.attn_sq(oracle.Quantized(inp.q, inp.k, v, smooth_v=True), 0.125, rows, tile=128)
    centred = exact - v.double().mean(dim=0).numpy()[None]
    e_plain = np.linalg.norm(plain - exact) / np.linalg.norm(centred)
    e_smooth = np.linalg.norm(smooth - exact) / np.linalg.norm(centred)
    assert e_smooth < 0.5 * e_plain, (e_smooth, e_plain)


# ---------------------------------------------------------------- planted mistakes

def _pins_pass(inp) -> bool:
    """A quick battery of the pins above; False as soon as one fails."""
    qz = oracle.Quantized(inp.q, inp.k, inp.v)
    n = inp.q.shape[0]
    kf = (inp.k.float().numpy() - brute_k_mean_exactish(inp.k)[None]).astype(np.float32)
    bk, bks = brute.quant_int8_blocks(np.ascontiguousarray(kf.transpose(1, 0, 2)), 64)
    if not ((bk == qz.k_codes).mean() > 0.999):
        return False
    bq, bqs = brute.quant_int8_blocks(np.ascontiguousarray(inp.q.float().numpy().transpose(1, 0, 2)), 128)
    if not ((bq == qz.q_codes).all() and (bqs == qz.q_scales).all()):
        return False
    bv, bvs = brute.quant_v(np.ascontiguousarray(inp.v.float().numpy().transpose(1, 0, 2)))
    if not ((bv == qz.v_codes).all() and (bvs == qz.v_scales).all()):
        return False
    rows = list(range(n))
    gl = oracle.attn_sq(qz, 0.125, rows, tile=0)
    g = brute.attn_sq_global(qz.q_codes, qz.q_scales, qz.k_codes, qz.k_scales, qz.v_codes,
                             qz.v_scales, n, 0.125)
    if not np.abs(gl - g).max() < 1e-12:
        return False
    if not _tiled_exact_case_error() < 1e-12:
        return False
    t32 = oracle.attn_sq(qz, 0.125, rows, tile=128, score_f32=True)
    if not rel_l2(t32, g) < 0.1:
        return False
    if not _agreement_holds(_fp32_mode_agreement(qz, 0.125, rows, range(qz.h))):
        return False
    q32 = oracle.Quantized(inp.q, inp.k, inp.v, q_block=32)
    bq32, bqs32 = brute.quant_int8_blocks(np.ascontiguousarray(inp.q.float().numpy().transpose(1, 0, 2)), 32)
    if not ((bq32 == q32.q_codes).all() and (bqs32 == q32.q_scales).all()):
        return False
    g32 = brute.attn_sq_global(q32.q_codes, q32.q_scales, q32.k_codes, q32.k_scales, q32.v_codes,
                               q32.v_scales, n, 0.125, q_block=32)
    if not np.abs(oracle.attn_sq(q32, 0.125, rows, tile=0) - g32).max() < 1e-12:
        return False
    if not _rr_closed_forms_hold():
        return False
    # the V options: INT8 P.V against the brute-force definition and its closed form, and the
    # shift invariance of smoothed V
    q8 = oracle.Quantized(inp.q, inp.k, inp.v, v_format="int8", smooth_v=True)
    bv8, bvs8 = brute.quant_v(np.ascontiguousarray(inp.v.float().numpy().transpose(1, 0, 2)), "int8", q8.v_mean)
    if not ((bv8 == q8.v_codes).all() and (bvs8 == q8.v_scales).all()):
        return False
    g8 = brute.attn_sq_global(q8.q_codes, q8.q_scales, q8.k_codes, q8.k_scales, q8.v_codes, q8.v_scales,
                              n, 0.125, v_format="int8", v_mean=q8.v_mean)
    if not np.abs(oracle.attn_sq(q8, 0.125, rows, tile=0) - g8).max() < 1e-12:
        return False
    if not (_int8_two_level_error() < 1e-12 and _shift_error("e4m3") < 1e-12):
        return False
    e = oracle.attn_exact(inp.q, inp.k, inp.v, 0.125, rows)
    b = brute.attn_exact(inp.q.float().numpy(), inp.k.float().numpy(), inp.v.float().numpy(), 0.125)
    return np.abs(e - b).max() < 1e-12


def brute_k_mean_exactish(k: torch.Tensor) -> np.ndarray:
    """fp64 mean rounded to fp32 (agrees with the oracle's mean to within an ulp or so)."""
    return k.double().mean(dim=0).float().numpy()


def test_pins_pass_unmutated(oracle_lib):
    inp = small_inputs(n=400, h=2, d=64, layout="qkv", bias_var=16.0)
    assert _pins_pass(inp)


@pytest.mark.parametrize("mutation", [m for m in oracle.MUTATIONS if m != "none"])
def test_planted_mistake_is_caught(oracle_lib, mutation):
    inp = small_inputs(n=400, h=2, d=64, layout="qkv", bias_var=16.0)
    try:
        oracle.set_mutation(mutation)
        caught = not _pins_pass(inp)
    finally:
        oracle.set_mutation("none")
    assert caught, mutation
