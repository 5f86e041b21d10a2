"""Independent numpy implementations for TINY inputs -- TEST INFRASTRUCTURE ONLY.

A second, differently structured implementation of the oracle's arithmetic, used to pin
`sage_oracle.c` on small cases: vectorised block quantisation, an E4M3 encoder that
searches the table of all finite E4M3 values for the nearest one (ties to the even
code), and global (one-pass) softmax attention via matrix products in fp64.
"""
from __future__ import annotations

import numpy as np


def e4m3_values() -> np.ndarray:
    """Value of codes 0..126 (the non-negative finite E4M3 numbers, increasing), from the
    OCP 8-bit floating point format: exponent bias 7, 3 mantissa bits, subnormals m*2^-9."""
    vals = []
    for code in range(127):
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


_VALS = e4m3_values()


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value (ties to the even code), saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.searchsorted(_VALS, a, side="left").clip(0, 126)   # first value >= a
    lo = (hi - 1).clip(0, 126)
    dlo, dhi = a - _VALS[lo], _VALS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def e4m3_decode(c: np.ndarray) -> np.ndarray:
    c = np.asarray(c, dtype=np.int64)
    v = _VALS[(c & 0x7F).clip(0, 126)]
    return np.where(c & 0x80, -v, v)


def quant_int8_blocks(x: np.ndarray, block: int):
    """x: fp32 [H, N, D].  Per (head, `block`-row block) symmetric INT8 with an fp32 scale
    amax/127 and IEEE fp32 division; returns codes [H, N_pad, D] and scales [H, N_pad/block]."""
    h, n, d = x.shape
    np_ = (n + 127) // 128 * 128
    xp = np.zeros((h, np_, d), np.float32)
    xp[:, :n] = x
    nb = np_ // block
    blocks = xp.reshape(h, nb, block, d)
    amax = np.abs(blocks).max(axis=(2, 3)).astype(np.float32)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale == 0, np.float32(1), scale)[:, :, None, None]
    y = (blocks / safe).astype(np.float32)
    codes = np.clip(np.rint(y), -127, 127).astype(np.int8)
    codes = np.where(scale[:, :, None, None] == 0, 0, codes).astype(np.int8)
    return codes.reshape(h, np_, d), scale


def quant_v(v: np.ndarray, v_format: str = "e4m3", mean=None):
    """v: fp32 [H, N, D] -> codes [H, D, N_pad] and scales [H, D]: E4M3 bytes with scale amax/448,
    or int8 codes with scale amax/127 (round half to even, clamped to +-127).  mean: None or the
    [H, D] fp32 mean subtracted (in fp32) before the maxima and the codes."""
    h, n, d = v.shape
    np_ = (n + 127) // 128 * 128
    x = v.astype(np.float32)
    if mean is not None:
        x = (x - np.asarray(mean, np.float32)[:, None, :]).astype(np.float32)
    amax = np.abs(x).max(axis=1).astype(np.float32)
    top = np.float32(127.0 if v_format == "int8" else 448.0)
    scale = (amax / top).astype(np.float32)
    safe = np.where(scale == 0, np.float32(1), scale)
    y = (x / safe[:, None, :]).astype(np.float32)
    if v_format == "int8":
        codes = np.where(scale[:, None, :] == 0, 0, np.clip(np.rint(y), -127, 127)).astype(np.int8)
        out = np.zeros((h, d, np_), np.int8)
    else:
        codes = np.where(scale[:, None, :] == 0, 0, e4m3_encode(y)).astype(np.uint8)
        out = np.zeros((h, d, np_), np.uint8)
    out[:, :, :n] = np.transpose(codes, (0, 2, 1))
    return out, scale


def attn_sq_global(qc, qs, kc, ks, vc, vs, n, sm_scale, q_block=128, v_format="e4m3", v_mean=None):
    """Global-max same-quantisation attention, all rows: [N, H, D] fp64.  qs holds one scale
    per (head, q_block consecutive rows).  v_format "int8": P = rint(127 p), V values are the
    integer codes; v_mean (or None) is added to the result."""
    h, np_, d = qc.shape
    out = np.zeros((n, h, d))
    qrow_scale = np.repeat(qs, q_block, axis=1)[:, :n]
    krow_scale = np.repeat(ks, 64, axis=1)[:, :n]
    top = 127.0 if v_format == "int8" else 448.0
    for hh in range(h):
        S = qc[hh, :n].astype(np.int64) @ kc[hh, :n].astype(np.int64).T
        s = S * qrow_scale[hh][:, None].astype(np.float64) * krow_scale[hh][None, :].astype(np.float64) * sm_scale
        p = np.exp(s - s.max(axis=1, keepdims=True))
        if v_format == "int8":
            p8 = np.rint(top * p)
            vdec = vc[hh, :, :n].astype(np.float64).T
        else:
            p8 = e4m3_decode(e4m3_encode(top * p))
            vdec = e4m3_decode(vc[hh, :, :n]).T           # [N, D]
        out[:, hh, :] = (p8 @ vdec) * vs[hh][None, :].astype(np.float64) / (top * p.sum(axis=1, keepdims=True))
        if v_mean is not None:
            out[:, hh, :] += np.asarray(v_mean, np.float64)[hh][None, :]
    return out


def attn_exact(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float) -> np.ndarray:
    """q, k, v: [N, H, D] -> softmax(sm_scale q k^T) v per head, fp64, [N, H, D]."""
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    n, h, d = q.shape
    out = np.zeros((n, h, d))
    for hh in range(h):
        s = sm_scale * (q[:, hh] @ k[:, hh].T)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        out[:, hh] = (p / p.sum(axis=1, keepdims=True)) @ v[:, hh]
    return out


def rmsnorm_rope(x: np.ndarray, gamma: np.ndarray, cos: np.ndarray, sin: np.ndarray, eps: float) -> np.ndarray:
    """fp64, [N, H, D]: RMSNorm over D with weight gamma, then each channel pair (2i, 2i+1)
    rotated by the angle whose cos / sin are cos[t, i], sin[t, i].  No rounding to bf16."""
    x = np.asarray(x, np.float64)
    r = 1.0 / np.sqrt((x * x).mean(axis=2, keepdims=True) + eps)
    y = x * r * np.asarray(gamma, np.float64)[None, None, :]
    c = np.asarray(cos, np.float64)[:, None, :]
    s = np.asarray(sin, np.float64)[:, None, :]
    z = np.empty_like(y)
    z[..., 0::2] = y[..., 0::2] * c - y[..., 1::2] * s
    z[..., 1::2] = y[..., 0::2] * s + y[..., 1::2] * c
    return z
