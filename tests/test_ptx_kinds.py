"""Which tcgen05.mma kinds the sm_103a target accepts -- a compile-only record (nvcc + ptxas, no GPU).

The method multiplies INT8 codes (QK^T, and P.V in the INT8 variant).  An INT8 tensor-core kind
(`kind::i8`) is rejected by ptxas for sm_103a, so the library holds the INT8 codes as fp16 values
(exact for |c| <= 2048) and multiplies them with `kind::f16` into fp32, where every partial sum of
the contraction is an exact integer.  `kind::f16` and `kind::f8f6f4` (the E4M3 P.V) assemble.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

NVCC = next((c for c in ("/usr/local/cuda/bin/nvcc", shutil.which("nvcc")) if c and os.path.exists(c)), None)

PROBE = r'''#include <cstdint>
__global__ void probe(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               " tcgen05.mma.cta_group::1.kind::KIND [%0], %1, %2, %3, p;\n}\n"
               :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(acc));
}
'''


def _compile(kind: str):
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, f"probe_{kind}.cu")
        with open(src, "w") as f:
            f.write(PROBE.replace("KIND", kind))
        r = subprocess.run([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-c", src, "-o",
                            os.path.join(tmp, "probe.o")], capture_output=True, text=True)
        return r.returncode, r.stdout + r.stderr


@pytest.mark.skipif(NVCC is None, reason="nvcc not found")
def test_kind_i8_rejected_for_sm_103a():
    rc, log = _compile("i8")
    print(log)
    assert rc != 0 and ".kind::i8" in log and "sm_103a" in log, log


@pytest.mark.skipif(NVCC is None, reason="nvcc not found")
@pytest.mark.parametrize("kind", ["f16", "f8f6f4"])
def test_kinds_used_by_the_library_assemble(kind):
    rc, log = _compile(kind)
    assert rc == 0, log
