"""The allocation-free entry point w4a16_lm_head_noalloc, called through the C ABI.

It serves callers that cannot allocate device memory (a runtime with a device
budget fixed at start-up, or a plain C caller without a device allocator); it
runs the same kernels as w4a16_lm_head on a fixed static scratch array.  The
test compares two calls in a row with the workspace-taking entry point, and
checks that a shape too large for the fixed scratch is refused on the host.
This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from tests._gpu import assert_logits_close, to_bf16_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    import nvfp4_weight_only_rows_gb300 as nv

    assert torch.cuda.is_available()
    return nv, nv.load_library()


def _call_noalloc(lib, x, packed, scales, g, out, out_code):
    M, K = x.shape
    N = packed.shape[0]
    return lib.w4a16_lm_head_noalloc(
        ctypes.c_void_p(x.data_ptr()), M, K, ctypes.c_void_p(packed.data_ptr()),
        ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(g.data_ptr()), N,
        ctypes.c_void_p(out.data_ptr()), out_code,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("M,N,K,out_dtype", [(8, 3000, 4096, torch.float32),
                                             (64, 1000, 8192, torch.float32),
                                             (33, 777, 1024, torch.bfloat16)])
def test_noalloc_matches_workspace_entry_point(lib, M, N, K, out_dtype):
    nv, clib = lib
    W = synth.quant_weight(N=N, K=K, seed=M + N)
    p, s, g = oracle.quantize(W)
    packed = torch.from_numpy(p).cuda()
    scales = torch.from_numpy(s).cuda().view(torch.float8_e4m3fn)
    gd = torch.tensor([g], dtype=torch.float32, device="cuda")
    code = 0 if out_dtype == torch.float32 else 1
    ref_out = nv.w4a16_lm_head(to_bf16_dev(synth.decode_x(M, K=K)), packed, scales, gd,
                               out_dtype=out_dtype).double().cpu().numpy()
    for call in range(2):
        # a fresh input each call, so that the second call must overwrite the
        # scratch the first one left behind
        x_bits = synth.decode_x(M, K=K) if call == 0 else synth.sweep_x(M, K=K)
        x = to_bf16_dev(x_bits)
        want = nv.w4a16_lm_head(x, packed, scales, gd, out_dtype=out_dtype)
        got = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
        assert _call_noalloc(clib, x, packed, scales, gd, got, code) == 0
        torch.cuda.synchronize()
        assert_logits_close(got.double().cpu().numpy(), want.double().cpu().numpy(),
                            f"noalloc call {call}", out_dtype == torch.bfloat16)
        if call == 0:
            assert_logits_close(got.double().cpu().numpy(), ref_out, "first call")


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    nv, clib = lib
    M, K, N = 2048, 4096, 256   # rescaled activations alone would need 16 MiB
    x = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    packed = torch.empty(N, K // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(N, K // 16, dtype=torch.uint8, device="cuda")
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    rc = _call_noalloc(clib, x, packed, scales, g, out, 0)
    assert rc == nv.Status.ERR_SCRATCH_LIMIT
    assert b"fixed scratch" in clib.nvfp4_status_string(rc)
