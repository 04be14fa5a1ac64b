"""The allocation-free entry point w4a16_lm_head_noalloc, called through the C ABI.

It serves callers that cannot allocate device memory (a runtime with a device
budget fixed at start-up, or a plain C caller without a device allocator); it
runs the same kernels as w4a16_lm_head on a fixed static scratch array.  The
tests compare two calls in a row with the workspace-taking entry point and
with the CPU oracle (the logits tolerance), at shapes whose grid covers every
SM (so the split-K region of the scratch is used), read the scratch's status
word through w4a16_lm_head_noalloc_status, and check that a shape too large
for the fixed scratch is refused on the host.  This file is named to be
collected last.
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


def _status(lib):
    v = ctypes.c_int32(-1)
    rc = lib.w4a16_lm_head_noalloc_status(
        ctypes.byref(v), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    return v.value


def _two_calls(nv, clib, host_q, dev_q, M, K, out_dtype):
    """Two calls in a row, each on a fresh input (the second must overwrite
    what the first left in the scratch): against the workspace entry point
    and against the oracle."""
    N = dev_q[0].shape[0]
    code = 0 if out_dtype == torch.float32 else 1
    for call in range(2):
        x_bits = synth.decode_x(M, K=K) if call == 0 else synth.sweep_x(M, K=K)
        x = to_bf16_dev(x_bits)
        want = nv.w4a16_lm_head(x, *dev_q, out_dtype=out_dtype)
        got = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
        assert _call_noalloc(clib, x, *dev_q, got, code) == 0
        torch.cuda.synchronize()
        g = got.double().cpu().numpy()
        bf16 = out_dtype == torch.bfloat16
        assert_logits_close(g, want.double().cpu().numpy(), f"noalloc call {call}", bf16)
        assert_logits_close(g, oracle.logits(x_bits, *host_q), f"noalloc call {call} oracle", bf16)
        assert _status(clib) == nv.Status.OK


def _upload(host_q):
    p, s, g = host_q
    return (torch.from_numpy(p).cuda(), torch.from_numpy(s).cuda().view(torch.float8_e4m3fn),
            torch.tensor([g], dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("M,N,K,out_dtype", [(8, 3000, 4096, torch.float32),
                                             (64, 1000, 8192, torch.float32),
                                             (33, 777, 1024, torch.bfloat16),
                                             (5, 700, 2880, torch.float32),
                                             (64, 40000, 8192, torch.float32)])
def test_noalloc_matches_workspace_entry_point_and_oracle(lib, M, N, K, out_dtype):
    nv, clib = lib
    host_q = oracle.quantize(synth.quant_weight(N=N, K=K, seed=M + N))
    _two_calls(nv, clib, host_q, _upload(host_q), M, K, out_dtype)


def test_noalloc_decode_shape_every_sm(lib, decode_nvfp4):
    """W[128256, 4096] quantized on the GPU, M = 64: a grid on every SM with
    the stream-K tail's partials in the fixed scratch."""
    nv, clib = lib
    _two_calls(nv, clib, decode_nvfp4.ref, decode_nvfp4.dev, 64, 4096, torch.float32)


def test_noalloc_status_word(lib):
    """A NaN block scale raises NVFP4_ERR_NONFINITE in the scratch's status
    word; the next clean call resets it."""
    nv, clib = lib
    M, N, K = 4, 600, 512
    p, s, g = oracle.quantize(synth.quant_weight(N=N, K=K, seed=9))
    bad = s.copy()
    bad[17, 3] = 0x7F
    x = to_bf16_dev(synth.decode_x(M, K=K))
    out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    assert _call_noalloc(clib, x, *_upload((p, bad, g)), out, 0) == 0
    assert _status(clib) == nv.Status.ERR_NONFINITE
    assert _call_noalloc(clib, x, *_upload((p, s, g)), out, 0) == 0
    assert _status(clib) == nv.Status.OK


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
