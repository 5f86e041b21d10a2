import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


_CASES = {}


def gpu_case(name: str):
    """Seeded inputs of a named workload on the CPU and on cuda:0, plus the oracle's
    quantised operands (cached for the session)."""
    if name not in _CASES:
        import torch
        import oracle
        from video_diffusion_transformer_sage_gb300 import synth
        if name.endswith("_hndcopy"):
            base = gpu_case(name[: -len("_hndcopy")])
            inp = synth.to_hnd(base["inp"])
            qz = base["qz"]
        elif name.endswith("_voff"):
            inp = synth.with_v_offset(synth.make_inputs(name[: -len("_voff")]))
            qz = oracle.Quantized(inp.q, inp.k, inp.v)
        else:
            inp = synth.make_inputs(name)
            qz = oracle.Quantized(inp.q, inp.k, inp.v)
        dev = torch.device("cuda:0")
        storage = inp.storage.to(dev)
        # the same views of the device copy
        def dview(t):
            off = t.storage_offset() - inp.storage.storage_offset()
            return storage.as_strided(t.shape, t.stride(), storage.storage_offset() + off)
        _CASES[name] = dict(inp=inp, qz=qz, storage=storage, q=dview(inp.q), k=dview(inp.k), v=dview(inp.v))
    return _CASES[name]
