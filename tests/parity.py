"""Output bars of the GPU attention against the oracle, shared by the GPU tests.

Three references, all computed by the oracle on the same quantised operands:
  ref32  the online schedule (128-key tiles, P coded against the running max, an exact rescale on
         every rise) with its base-2 scores formed in fp32 -- the precision in which the kernel
         takes P's rounding decisions
  ref64  the same schedule with its scores in fp64
  glob   the one-pass fp64 definition: P coded against each row's global max
Bars:
  - against ref32: relative L2 <= 5e-3 and max-abs <= 3e-2 (the same-quantisation bars);
  - against ref64: relative L2 <= 5e-3; max-abs <= 3e-2 + the oracle's own max-abs distance
    between ref32 and ref64.  The two schedules code P identically except where a key's 448 p
    lies within fp32 rounding of a code boundary (pinned key by key on the CPU), and one such
    flip on a dominant key moves an output element by up to one E4M3 step of its weight;
  - against glob: the schedule's own distance from the definition (ref64 against glob, which the
    CPU pins bound) plus the same bars, the max-abs one widened as above.  Coding P against a
    running max instead of the global max rounds each p at another scale; that difference
    belongs to the online method, and the GPU may add at most the same-quantisation error.
With `widen`, an element's max-abs allowance grows by 2^-8 of its magnitude (the bf16 rounding of
outputs far above 1, e.g. V with large channel offsets).
"""
import numpy as np

import oracle

SQ_REL, SQ_ABS = 5e-3, 3e-2


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _abs_excess(got, ref, allowance, widen):
    """Largest |got - ref| beyond the allowance (<= 0 when within it)."""
    lim = allowance + (2.0 ** -8 * np.abs(ref) if widen else 0.0)
    return float((np.abs(got - ref) - lim).max())


def check(got, oz, sm, rows, widen=False):
    """Returns (ok, numbers) for the GPU output `got` [R, H, D] of query `rows`."""
    ref32 = oracle.attn_sq(oz, sm, rows, tile=128, score_f32=True)
    ref64 = oracle.attn_sq(oz, sm, rows, tile=128, score_f32=False)
    glob = oracle.attn_sq(oz, sm, rows, tile=0)
    sched_rel = rel_l2(ref64, glob)
    sched_abs = float(np.abs(ref64 - glob).max())
    prec_abs = float(np.abs(ref32 - ref64).max())
    info = dict(rel32=rel_l2(got, ref32), abs32=float(np.abs(got - ref32).max()),
                rel64=rel_l2(got, ref64), abs64=float(np.abs(got - ref64).max()),
                rel_glob=rel_l2(got, glob), abs_glob=float(np.abs(got - glob).max()),
                sched_rel=sched_rel, sched_abs=sched_abs, prec_rel=rel_l2(ref32, ref64), prec_abs=prec_abs)
    ok = (info["rel32"] <= SQ_REL and _abs_excess(got, ref32, SQ_ABS, widen) <= 0
          and info["rel64"] <= SQ_REL and _abs_excess(got, ref64, SQ_ABS + prec_abs, widen) <= 0
          and info["rel_glob"] <= sched_rel + SQ_REL
          and _abs_excess(got, glob, sched_abs + prec_abs + SQ_ABS, widen) <= 0)
    return ok, info


def assert_close(got, oz, sm, rows, widen=False):
    ok, info = check(got, oz, sm, rows, widen)
    assert ok, info
    return info
