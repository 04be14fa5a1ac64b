import os
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a); run with -m gpu")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


@pytest.fixture(scope="session")
def decode_nvfp4():
    """The decode / prefill lm_head W[128256, 4096] (seed 1), quantized twice:
    on the GPU through the C ABI (``dev``: packed, scales, global as device
    tensors -- the buffers every product test of this workload multiplies
    with) and by the CPU oracle (``ref``: the bytes those must equal).
    ``test_gpu_workloads`` checks the two byte for byte."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import nvfp4_weight_only_rows_gb300 as nv
    import oracle
    import synth
    from tests._gpu import to_bf16_dev

    assert torch.cuda.is_available()
    W = synth.decode_weight()
    Wd = to_bf16_dev(W)
    dev = nv.nvfp4_quantize_rows(Wd)
    torch.cuda.synchronize()
    del Wd
    return SimpleNamespace(W=W, dev=dev, ref=oracle.quantize(W))
