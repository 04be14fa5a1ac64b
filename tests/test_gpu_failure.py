"""Failure detection on the GPU without faulting it: a pipeline wait that can
never complete gives up after its limit, the kernel reports NVFP4_ERR_TIMEOUT
in the workspace status word, and the CUDA context stays usable."""
import time

import numpy as np
import pytest
import torch

import nvfp4_weight_only_rows_gb300 as nv
import oracle
import synth
from tests._gpu import assert_logits_close, to_bf16_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def test_stuck_wait_reports_timeout_and_context_survives():
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    nv.nvfp4_selftest_bounded_wait(ws, limit_us=20000)  # 20 ms per wait
    status = nv.nvfp4_read_device_status(ws)
    elapsed = time.perf_counter() - t0
    assert status == nv.Status.ERR_TIMEOUT
    assert elapsed < 5.0
    # the context still works: a normal product right after
    W = synth.quant_weight(N=256, K=512, seed=77)
    x = synth.decode_x(3, K=512)
    p, s, g = oracle.quantize(W)
    out = nv.w4a16_lm_head(to_bf16_dev(x), torch.from_numpy(p).cuda(),
                           torch.from_numpy(s).cuda().view(torch.float8_e4m3fn),
                           torch.tensor([g], device="cuda"))
    assert_logits_close(out.double().cpu().numpy(), oracle.logits(x, p, s, g), "after timeout")


def test_selftest_argument_errors():
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_selftest_bounded_wait(ws, limit_us=0)
    assert e.value.status == nv.Status.ERR_SHAPE
    with pytest.raises(nv.NVFP4Error) as e:
        nv.nvfp4_selftest_bounded_wait(ws[:64], limit_us=10)
    assert e.value.status == nv.Status.ERR_WORKSPACE
