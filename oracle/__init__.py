"""CPU oracle for the quantised attention path -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke() check and bench.py's CPU-baseline / reference leg
may import this package.  It shares no code with the CUDA library: the arithmetic lives
in `sage_oracle.c` (plain C, fp64 loops) and, for tiny cases, in `brute.py` (numpy).

`build()` compiles `sage_oracle.c` with gcc into `oracle/_build/liboracle.so`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sage_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()

MUTATIONS = {"none": 0, "no_smooth": 1, "rescale_sign": 2, "scale_255": 3, "key_index": 4,
             "v_scale_channel": 5, "drop_last_key": 6, "e4m3_trunc": 7, "mean_n_pad": 8,
             "q_block_index": 9, "rope_sign": 10, "rms_sum": 11, "v_mean_sign": 12, "p_i8_255": 13,
             "v_i8_448": 14, "f32_half_scale": 15, "f32_kscale_tile": 16, "f32_l_codes": 17,
             "f32_exp_base": 18}

Q_BLOCKS = (1, 2, 4, 8, 16, 32, 64, 128)
V_FORMATS = {"e4m3": 0, "int8": 1}


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, OpenMP, no FMA contraction, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P, I = ctypes.c_void_p, ctypes.c_int64
            L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_decode.restype = ctypes.c_double
            L.oracle_e4m3_encode.argtypes = [ctypes.c_double]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_set_mutation.argtypes = [ctypes.c_int]
            L.oracle_k_mean.argtypes = [P, I, I, I, I, I, P]
            L.oracle_quant_q.argtypes = [P, I, I, I, I, I, P, P]
            L.oracle_quant_q_blk.argtypes = [P, I, I, I, I, I, I, P, P]
            L.oracle_quant_k.argtypes = [P, I, I, I, I, I, P, P, P]
            L.oracle_quant_v.argtypes = [P, I, I, I, I, I, P, P]
            L.oracle_quant_v_fmt.argtypes = [P, I, I, I, I, I, P, I, P, P]
            L.oracle_attn_sq_v.argtypes = [P, P, I, P, P, P, P, P, I, I, I, I, ctypes.c_double, P, I, I, I, P]
            L.oracle_attn_sq_trace.argtypes = [P, P, I, P, P, P, P, P, I, I, I, ctypes.c_double, I, P, I, I, I,
                                               P, P, P, P]
            L.oracle_qk_int32.argtypes = [P, P, I, I, I, I, I, I, I, I, P]
            L.oracle_attn_sq.argtypes = [P, P, P, P, P, P, I, I, I, ctypes.c_double, P, I, I, I, P]
            L.oracle_attn_sq_blk.argtypes = [P, P, I, P, P, P, P, I, I, I, ctypes.c_double, P, I, I, I, P]
            L.oracle_attn_exact.argtypes = [P, P, P, I, I, I, I, I, I, I, I, I, ctypes.c_double,
                                            P, I, P]
            L.oracle_rmsnorm_rope.argtypes = [P, I, I, I, I, I, P, P, P, ctypes.c_float]
            L.oracle_num_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def set_mutation(name: str) -> None:
    """Plants one deliberate mistake in the oracle (tests of the pins only)."""
    lib().oracle_set_mutation(MUTATIONS[name])


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def pad128(n: int) -> int:
    return (n + 127) // 128 * 128


def _view_args(x: torch.Tensor):
    """A bf16 [N, H, D] CPU view with unit channel stride -> (base pointer, st, sh, keepalive)."""
    assert x.dtype == torch.bfloat16 and x.device.type == "cpu" and x.dim() == 3
    assert x.stride(2) == 1
    return x.data_ptr(), x.stride(0), x.stride(1)


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_e4m3_encode(float(x)))


def e4m3_decode(c: int) -> float:
    return float(lib().oracle_e4m3_decode(int(c)))


def e4m3_table() -> np.ndarray:
    """Decoded value of every code 0..255 (NaN for the two NaN codes)."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def k_mean(k: torch.Tensor) -> np.ndarray:
    n, h, d = k.shape
    mu = np.zeros((h, d), np.float32)
    p, st, sh = _view_args(k)
    lib().oracle_k_mean(p, n, h, d, st, sh, _ptr(mu))
    return mu


def quant_q(q: torch.Tensor, q_block: int = 128):
    """INT8 Q codes [H, N_pad, D] and scales [H, N_pad / q_block] (q_block a power of two <= 128)."""
    assert q_block in Q_BLOCKS
    n, h, d = q.shape
    np_ = pad128(n)
    codes = np.zeros((h, np_, d), np.int8)
    scales = np.zeros((h, np_ // q_block), np.float32)
    p, st, sh = _view_args(q)
    lib().oracle_quant_q_blk(p, n, h, d, st, sh, q_block, _ptr(codes), _ptr(scales))
    return codes, scales


def quant_k(k: torch.Tensor, mu: np.ndarray):
    n, h, d = k.shape
    np_ = pad128(n)
    codes = np.zeros((h, np_, d), np.int8)
    scales = np.zeros((h, np_ // 64), np.float32)
    mu = np.ascontiguousarray(mu, dtype=np.float32)
    p, st, sh = _view_args(k)
    lib().oracle_quant_k(p, n, h, d, st, sh, _ptr(mu), _ptr(codes), _ptr(scales))
    return codes, scales


def channel_mean(x: torch.Tensor) -> np.ndarray:
    """Mean over the tokens of each (head, channel), in the order of the K mean: [H, D] fp32."""
    return k_mean(x)


def quant_v(v: torch.Tensor, v_format: str = "e4m3", mean=None):
    """V codes [H, D, N_pad] (uint8 E4M3 bytes, or int8 codes) and scales [H, D].
    mean: None, or the [H, D] fp32 mean taken out of V before quantisation."""
    n, h, d = v.shape
    np_ = pad128(n)
    fmt = V_FORMATS[v_format]
    codes = np.zeros((h, d, np_), np.int8 if fmt else np.uint8)
    scales = np.zeros((h, d), np.float32)
    p, st, sh = _view_args(v)
    if mean is None and not fmt:
        lib().oracle_quant_v(p, n, h, d, st, sh, _ptr(codes), _ptr(scales))
    else:
        mu = None if mean is None else np.ascontiguousarray(mean, dtype=np.float32)
        lib().oracle_quant_v_fmt(p, n, h, d, st, sh, None if mu is None else _ptr(mu), fmt, _ptr(codes),
                                 _ptr(scales))
    return codes, scales


class Quantized:
    """Steps 1-4 of the oracle for one set of inputs.  v_format "e4m3" (the method's FP8 V) or
    "int8" (the INT8 P.V variant); smooth_v: take the channel mean out of V first."""

    def __init__(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_block: int = 128,
                 v_format: str = "e4m3", smooth_v: bool = False):
        self.n, self.h, self.d = q.shape
        self.q_block = q_block
        self.v_format = v_format
        self.k_mean = k_mean(k)
        self.q_codes, self.q_scales = quant_q(q, q_block)
        self.k_codes, self.k_scales = quant_k(k, self.k_mean)
        self.v_mean = channel_mean(v) if smooth_v else None
        self.v_codes, self.v_scales = quant_v(v, v_format, self.v_mean)


def qk_int32(qz: Quantized, head: int, i0: int, j0: int, rows: int, cols: int) -> np.ndarray:
    out = np.zeros((rows, cols), np.int32)
    lib().oracle_qk_int32(_ptr(qz.q_codes), _ptr(qz.k_codes), qz.n, qz.h, qz.d, head, i0, j0,
                          rows, cols, _ptr(out))
    return out


def attn_sq(qz: Quantized, sm_scale: float, rows, tile: int = 128, score_f32=None) -> np.ndarray:
    """Same-quantisation attention O_sq for query `rows` (all heads): [len(rows), H, D] fp64.

    tile=0: the fp64 one-pass definition.  tile>0: the online schedule over `tile`-key tiles;
    by default (score_f32=None -> True for tile>0) the E4M3 rounding of P is decided on fp32
    scores formed as the kernel forms them; score_f32=False keeps those scores in fp64."""
    if score_f32 is None:
        score_f32 = tile > 0
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((len(rows), qz.h, qz.d), np.float64)
    v_mean = getattr(qz, "v_mean", None)
    mu = None if v_mean is None else np.ascontiguousarray(v_mean, dtype=np.float32)
    lib().oracle_attn_sq_v(_ptr(qz.q_codes), _ptr(qz.q_scales), int(getattr(qz, "q_block", 128)),
                           _ptr(qz.k_codes), _ptr(qz.k_scales), _ptr(qz.v_codes), _ptr(qz.v_scales),
                           None if mu is None else _ptr(mu), V_FORMATS[getattr(qz, "v_format", "e4m3")],
                           qz.n, qz.h, qz.d, float(sm_scale), _ptr(rows), len(rows), int(tile),
                           int(bool(score_f32)), _ptr(out))
    return out


def attn_sq_trace(qz: Quantized, sm_scale: float, head: int, rows, tile: int = 128, score_f32: bool = True):
    """attn_sq for query `rows` of one head, with each key's trace: returns (out [R, D], pp [R, N],
    p8 [R, N], lw [R, N]).  pp[r, j] is the 448 p (127 p for INT8 P) whose code P takes, p8 the value
    of that code, lw the running max key j's p is relative to, as a base-2 exponent: key j enters
    the final sums with weight 2^(lw[r, j] - lw[r, N-1])."""
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    r, n, d = len(rows), qz.n, qz.d
    out = np.zeros((r, d), np.float64)
    pp, p8, lw = (np.zeros((r, n), np.float64) for _ in range(3))
    v_mean = getattr(qz, "v_mean", None)
    mu = None if v_mean is None else np.ascontiguousarray(v_mean, dtype=np.float32)
    lib().oracle_attn_sq_trace(_ptr(qz.q_codes), _ptr(qz.q_scales), int(getattr(qz, "q_block", 128)),
                               _ptr(qz.k_codes), _ptr(qz.k_scales), _ptr(qz.v_codes), _ptr(qz.v_scales),
                               None if mu is None else _ptr(mu), V_FORMATS[getattr(qz, "v_format", "e4m3")],
                               n, d, float(sm_scale), int(head), _ptr(rows), r, int(tile), int(bool(score_f32)),
                               _ptr(out), _ptr(pp), _ptr(p8), _ptr(lw))
    return out, pp, p8, lw


def attn_exact(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, sm_scale: float, rows) -> np.ndarray:
    """Exact fp64 softmax attention O_exact for query `rows` (all heads): [len(rows), H, D]."""
    n, h, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((len(rows), h, d), np.float64)
    pq, qst, qsh = _view_args(q)
    pk, kst, ksh = _view_args(k)
    pv, vst, vsh = _view_args(v)
    lib().oracle_attn_exact(pq, pk, pv, n, h, d, qst, qsh, kst, ksh, vst, vsh, float(sm_scale),
                            _ptr(rows), len(rows), _ptr(out))
    return out


def rmsnorm_rope(x: torch.Tensor, gamma, cos, sin, eps: float) -> torch.Tensor:
    """In place on a bf16 CPU [N, H, D] view with unit channel stride: RMSNorm over D with
    weight gamma [D], then the rotation of channel pairs (2i, 2i+1) by the angles whose cos /
    sin are given as [N, D/2] fp32.  Returns x."""
    n, h, d = x.shape
    g = np.ascontiguousarray(np.asarray(gamma, dtype=np.float32))
    c = np.ascontiguousarray(np.asarray(cos, dtype=np.float32))
    s = np.ascontiguousarray(np.asarray(sin, dtype=np.float32))
    assert g.shape == (d,) and c.shape == (n, d // 2) and s.shape == (n, d // 2)
    p, st, sh = _view_args(x)
    lib().oracle_rmsnorm_rope(p, n, h, d, st, sh, _ptr(g), _ptr(c), _ptr(s), float(eps))
    return x
