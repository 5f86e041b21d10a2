"""GPU parity of the smoothing / quantisation kernels against the CPU oracle: the K mean,
every INT8 Q/K code, every E4M3 V code and every scale must be bit-identical."""
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
