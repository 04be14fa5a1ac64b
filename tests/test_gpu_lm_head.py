"""GPU parity of the W4A16 lm_head product against the CPU oracle.

The weights here are quantized by the CPU oracle and uploaded, so these
tests check the product alone (the full-size workloads, multiplied on the
GPU-quantized buffers, are in test_gpu_workloads.py); the bar is |err| <= 2e-3 * max|row of oracle
logits| + 1e-3 per element, and argmax agreement except where the oracle's
top two logits are closer than 1e-3.
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_only_rows_gb300 as nv
import oracle
import synth
from tests._gpu import assert_argmax_agrees, assert_logits_close, to_bf16_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def upload_quantized(W_bits):
    p, s, g = oracle.quantize(W_bits)
    pd = torch.from_numpy(p).cuda()
    sd = torch.from_numpy(s).cuda().view(torch.float8_e4m3fn)
    gd = torch.tensor([g], dtype=torch.float32, device="cuda")
    return (p, s, g), (pd, sd, gd)


def run(x_bits, dev_q, out_dtype=torch.float32):
    xd = to_bf16_dev(x_bits)
    out = nv.w4a16_lm_head(xd, *dev_q, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def test_tiny_workload():
    W, x = synth.tiny_weight(), synth.tiny_x()
    host_q, dev_q = upload_quantized(W)
    ref = oracle.logits(x, *host_q)
    for dt in (torch.float32, torch.bfloat16):
        got = run(x, dev_q, dt)
        assert_logits_close(got, ref, f"tiny {dt}", dt == torch.bfloat16)
        assert_argmax_agrees(got, ref, dt == torch.bfloat16)


@pytest.mark.parametrize("M,N,K", [(1, 300, 512), (5, 129, 256), (16, 128, 768),
                                   (17, 1000, 512), (64, 777, 1024), (100, 513, 256),
                                   (130, 260, 512), (200, 384, 1280), (1, 1, 256)])
def test_ragged_shapes(M, N, K):
    W = synth.quant_weight(N=N, K=K, seed=M + N)
    x = synth.decode_x(M, K=K)
    host_q, dev_q = upload_quantized(W)
    ref = oracle.logits(x, *host_q)
    got = run(x, dev_q)
    assert_logits_close(got, ref, f"M={M} N={N} K={K}")
    assert_argmax_agrees(got, ref)
    got16 = run(x, dev_q, torch.bfloat16)
    assert_logits_close(got16, ref, f"bf16 M={M} N={N} K={K}", True)


def test_activation_range_extremes():
    """Token rows of very different magnitude: the per-token rescale keeps them exact."""
    N, K, M = 256, 512, 6
    W = synth.quant_weight(N=N, K=K, seed=31)
    xf = synth.bf16_bits_to_f32(synth.decode_x(M, K=K)).copy()
    xf[0] *= 1e-30
    xf[1] *= 1e30
    xf[2] = 0.0
    xf[3, ::7] *= 1e-8
    xf[4] *= 3e4
    x = synth.f32_to_bf16_bits(xf)
    host_q, dev_q = upload_quantized(W)
    ref = oracle.logits(x, *host_q)
    assert_logits_close(run(x, dev_q), ref, "extremes")


def test_deterministic_and_empty():
    W = synth.quant_weight(N=500, K=512, seed=8)
    x = synth.decode_x(9, K=512)
    _, dev_q = upload_quantized(W)
    a = run(x, dev_q)
    b = run(x, dev_q)
    assert np.array_equal(a, b)
    xd = to_bf16_dev(x[:0])
    out = nv.w4a16_lm_head(xd, *dev_q)
    assert out.shape == (0, 500)


def test_errors_are_status_codes():
    W = synth.quant_weight(N=64, K=256, seed=1)
    _, (pd, sd, gd) = upload_quantized(W)
    x = to_bf16_dev(synth.decode_x(4, K=256))
    with pytest.raises(nv.NVFP4Error) as e:
        nv.w4a16_lm_head(x, pd, sd, gd, workspace=torch.empty(64, dtype=torch.uint8,
                                                               device="cuda"))
    assert e.value.status == nv.Status.ERR_WORKSPACE
    # K = 264 is not a multiple of 16: no NVFP4 weight has that width
    x2 = torch.zeros(4, 264, dtype=torch.bfloat16, device="cuda")
    p2 = torch.zeros(64, 132, dtype=torch.uint8, device="cuda")
    s2 = torch.zeros(64, 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.w4a16_lm_head(x2, p2, s2, gd, workspace=torch.empty(1 << 20, dtype=torch.uint8,
                                                               device="cuda"))
    assert e.value.status == nv.Status.ERR_SHAPE


def test_nan_block_scale_sets_device_status():
    """A NaN block scale (E4M3 0x7F / 0xFF, the unloaded-scale sentinel of
    `KNvfp4Static.process`) raises NVFP4_ERR_NONFINITE in the status word;
    the next call on clean scales resets it to OK."""
    N, K, M = 700, 1024, 4
    W = synth.quant_weight(N=N, K=K, seed=3)
    (p, s, g), (pd, sd, gd) = upload_quantized(W)
    x = to_bf16_dev(synth.decode_x(M, K=K))
    ws = torch.empty(nv.w4a16_lm_head_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    for row, col, byte in ((0, 0, 0x7F), (N - 1, K // 16 - 1, 0xFF), (345, 17, 0x7F)):
        bad = s.copy()
        bad[row, col] = byte
        sb = torch.from_numpy(bad).cuda().view(torch.float8_e4m3fn)
        out = nv.w4a16_lm_head(x, pd, sb, gd, workspace=ws)
        assert nv.nvfp4_read_device_status(ws) == nv.Status.ERR_NONFINITE, (row, col)
        assert torch.isnan(out[:, row]).all()
        nv.w4a16_lm_head(x, pd, sd, gd, workspace=ws)
        assert nv.nvfp4_read_device_status(ws) == nv.Status.OK
    # the largest finite scales (0x7E = 448, 0xFE = -448) are not NaN
    big = s.copy()
    big[5, ::2] = 0x7E
    big[5, 1::2] = 0xFE
    nv.w4a16_lm_head(x, pd, torch.from_numpy(big).cuda().view(torch.float8_e4m3fn), gd,
                     workspace=ws)
    assert nv.nvfp4_read_device_status(ws) == nv.Status.OK


@pytest.mark.parametrize("M,N,K", [(8, 216 * 128, 1024), (1, 153 * 128 + 5, 512),
                                   (40, 300 * 128, 768)])
def test_split_units_deterministic(M, N, K):
    """More weight tiles than SMs and not a multiple of them: the stream-K
    ranges cut units between CTAs, whose two fp32 partials are added by the
    CTA that finishes second.  Results match the oracle and repeat bit for bit."""
    W = synth.quant_weight(N=N, K=K, seed=N % 97)
    x = synth.decode_x(M, K=K)
    host_q, dev_q = upload_quantized(W)
    runs = [run(x, dev_q) for _ in range(3)]
    assert all(np.array_equal(runs[0], r) for r in runs[1:])
    cols = np.unique(np.linspace(0, N - 1, 4000).astype(np.int64))
    ref = oracle.logits(x, *host_q, cols=cols)
    assert_logits_close(runs[0][:, cols], ref, f"split M={M} N={N} K={K}")
