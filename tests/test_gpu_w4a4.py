"""GPU parity of the W4A4 NVFP4 path: the 128x4-interleaved scale copy and
the in-call activation quantization bit-exact against the CPU oracle, the
block-scaled FP4 logits within |err| <= 2e-3 * max|row| + 1e-3 of the
oracle's float64 product, and the fused argmax bit-exact against the argmax
of the plain fp32 logits."""
import numpy as np
import pytest
import torch

import nvfp4_weight_only_rows_gb300 as nv
import oracle
import synth
from tests._gpu import (assert_argmax_agrees, assert_logits_close, assert_topk_equal,
                        assert_topk_oracle_agrees, expected_topk, logits_tolerance, to_bf16_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def dev_weight(host_q):
    p, s, g = host_q
    pd = torch.from_numpy(p).cuda()
    sd = torch.from_numpy(s).cuda()
    sw = nv.nvfp4_swizzle_scales(sd)
    return pd, sw, torch.tensor([g], dtype=torch.float32, device="cuda")


def input_global(x_bits):
    amax = float(np.abs(synth.bf16_bits_to_f32(x_bits)).max())
    gx, igx = oracle.global_scale(amax)
    return gx, igx


def run(x, host_q, gx, dt=torch.float32):
    pd, sw, gd = dev_weight(host_q)
    out = nv.w4a4_lm_head(to_bf16_dev(x), pd, sw, gd,
                          torch.tensor([gx], dtype=torch.float32, device="cuda"), out_dtype=dt)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


@pytest.mark.parametrize("N,K", [(512, 256), (130, 320), (128256, 4096), (7, 64)])
def test_swizzle_bit_exact(N, K):
    W = synth.quant_weight(N=N, K=K, seed=N % 13) if N < 100000 else synth.decode_weight()
    _, s, _ = oracle.quantize(W)
    got = nv.nvfp4_swizzle_scales(torch.from_numpy(s).cuda()).cpu().numpy()
    assert np.array_equal(got, oracle.swizzle_scales(s))


def test_activation_quantization_bit_exact():
    """The workspace holds [256-byte status][x codes, M_pad x K/2][x scales,
    interleaved, round_up(M, 128) x K/16] after a call."""
    M, N, K = 37, 256, 1024
    x = synth.decode_x(M, K=K)
    host_q = oracle.quantize(synth.quant_weight(N=N, K=K, seed=3))
    gx, igx = input_global(x)
    pd, sw, gd = dev_weight(host_q)
    ws = torch.empty(nv.w4a4_lm_head_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    nv.w4a4_lm_head(to_bf16_dev(x), pd, sw, gd, torch.tensor([gx], device="cuda"), workspace=ws)
    torch.cuda.synchronize()
    xp, xs = oracle.quantize_rows(x, np.arange(M), gx, igx)
    m_pad = 48  # M rounded up to the token tile (16)
    got_p = ws[256:256 + M * K // 2].cpu().numpy().reshape(M, K // 2)
    assert np.array_equal(got_p, xp)
    off = 256 + m_pad * K // 2
    got_s = ws[off:off + 128 * K // 16].cpu().numpy()
    assert np.array_equal(got_s, oracle.swizzle_scales(xs))


def test_tiny_workload():
    W, x = synth.tiny_weight(), synth.tiny_x()
    host_q = oracle.quantize(W)
    gx, _ = input_global(x)
    ref = oracle.w4a4_logits(x, gx, *host_q)
    for dt in (torch.float32, torch.bfloat16):
        got = run(x, host_q, gx, dt)
        assert_logits_close(got, ref, f"tiny {dt}", dt == torch.bfloat16)
        assert_argmax_agrees(got, ref, dt == torch.bfloat16)


@pytest.mark.parametrize("M,N,K", [(1, 300, 512), (5, 129, 256), (16, 128, 768),
                                   (17, 1000, 512), (64, 777, 1024), (100, 513, 256),
                                   (130, 260, 512), (200, 384, 1280), (1, 1, 256),
                                   (8, 216 * 128, 1024), (40, 300 * 128, 768),
                                   (256, 1000, 768), (250, 1000, 272), (1024, 10240, 512)])
def test_product_shapes(M, N, K):
    """Logits of every shape class: token tiles of 16 to 128, ragged token and
    weight tiles, K % 32 != 0 (staged codes), and more 128 x 128 units than
    CTAs (every CTA walks several units)."""
    W = synth.quant_weight(N=N, K=K, seed=M + N)
    x = synth.decode_x(M, K=K)
    host_q = oracle.quantize(W)
    gx, _ = input_global(x)
    cols = np.unique(np.linspace(0, N - 1, min(N, 3000)).astype(np.int64))
    ref = oracle.w4a4_logits(x, gx, *host_q, cols=cols)
    got = run(x, host_q, gx)
    assert_logits_close(got[:, cols], ref, f"M={M} N={N} K={K}")


def test_invalid_input_global_is_a_status():
    M, N, K = 4, 128, 256
    x = synth.decode_x(M, K=K)
    pd, sw, gd = dev_weight(oracle.quantize(synth.quant_weight(N=N, K=K, seed=1)))
    ws = torch.empty(nv.w4a4_lm_head_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    nv.w4a4_lm_head(to_bf16_dev(x), pd, sw, gd, torch.tensor([0.0], device="cuda"), workspace=ws)
    assert nv.nvfp4_read_device_status(ws) == nv.Status.ERR_NONFINITE
    nv.w4a4_lm_head(to_bf16_dev(x), pd, sw, gd, torch.tensor([0.01], device="cuda"), workspace=ws)
    assert nv.nvfp4_read_device_status(ws) == nv.Status.OK


@pytest.fixture(scope="module")
def decode_case(decode_nvfp4):
    return decode_nvfp4.ref


@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_decode_workload(decode_case, M):
    x = synth.decode_x(M)
    gx, _ = input_global(x)
    got = run(x, decode_case, gx)
    ref = oracle.w4a4_logits(x, gx, *decode_case)
    assert_logits_close(got, ref, f"decode M={M}")
    assert_argmax_agrees(got, ref)


def test_prefill_workload_sampled(decode_case):
    x = synth.prefill_x()
    gx, _ = input_global(x)
    got = run(x, decode_case, gx, torch.bfloat16)
    rows = np.unique(np.concatenate([[0, 127, 128, 2047], np.random.default_rng(6).integers(0, 2048, 20)]))
    ref = oracle.w4a4_logits(x[rows], gx, *decode_case)
    assert_logits_close(got[rows], ref, "prefill", True)


def first_max(L):
    m = L.amax(dim=1, keepdim=True)
    ids = (L == m).to(torch.int32).argmax(dim=1).to(torch.int64)
    return ids, L.gather(1, ids[:, None])[:, 0]


@pytest.mark.parametrize("M,N,K", [(1, 300, 512), (64, 777, 1024), (200, 5000, 256),
                                   (8, 216 * 128, 1024)])
def test_argmax_matches_plain_logits(M, N, K):
    W = synth.quant_weight(N=N, K=K, seed=M * 3 + N)
    x = synth.decode_x(M, K=K)
    host_q = oracle.quantize(W)
    gx, _ = input_global(x)
    pd, sw, gd = dev_weight(host_q)
    gxd = torch.tensor([gx], dtype=torch.float32, device="cuda")
    xd = to_bf16_dev(x)
    ids, vals = nv.w4a4_lm_head_argmax(xd, pd, sw, gd, gxd)
    want_ids, want_vals = first_max(nv.w4a4_lm_head(xd, pd, sw, gd, gxd))
    torch.cuda.synchronize()
    assert torch.equal(ids, want_ids)
    assert torch.equal(vals, want_vals)
    sel = sorted({0, M - 1})
    ref = oracle.w4a4_logits(x[sel], gx, *host_q)
    onehot = np.full_like(ref, -np.inf)
    onehot[np.arange(len(sel)), ids.cpu().numpy()[sel]] = 0.0
    assert_argmax_agrees(onehot, ref)
    tol = logits_tolerance(ref)[:, 0]
    err = np.abs(vals.cpu().numpy()[sel] - ref[np.arange(len(sel)), ids.cpu().numpy()[sel]])
    assert np.all(err <= tol)


def test_argmax_prefill(decode_case):
    x = synth.prefill_x()
    gx, _ = input_global(x)
    pd, sw, gd = dev_weight(decode_case)
    gxd = torch.tensor([gx], dtype=torch.float32, device="cuda")
    xd = to_bf16_dev(x)
    ids, vals = nv.w4a4_lm_head_argmax(xd, pd, sw, gd, gxd)
    want_ids, want_vals = first_max(nv.w4a4_lm_head(xd, pd, sw, gd, gxd))
    torch.cuda.synchronize()
    assert torch.equal(ids, want_ids)
    assert torch.equal(vals, want_vals)


@pytest.mark.parametrize("M,N,K,k", [(1, 300, 512, 10), (64, 777, 1024, 50), (200, 5000, 256, 128),
                                     (8, 216 * 128, 1024, 50), (3, 7, 256, 7)])
def test_topk_matches_plain_logits(M, N, K, k):
    """The fused top-k of the W4A4 logits: bit for bit the k largest of the
    fp32 logits w4a4_lm_head writes, and oracle-agreeing on two tokens."""
    W = synth.quant_weight(N=N, K=K, seed=M * 11 + N)
    x = synth.decode_x(M, K=K)
    host_q = oracle.quantize(W)
    gx, _ = input_global(x)
    pd, sw, gd = dev_weight(host_q)
    gxd = torch.tensor([gx], dtype=torch.float32, device="cuda")
    xd = to_bf16_dev(x)
    ids, vals = nv.w4a4_lm_head_topk(xd, pd, sw, gd, gxd, k)
    want_ids, want_vals = expected_topk(nv.w4a4_lm_head(xd, pd, sw, gd, gxd), k)
    torch.cuda.synchronize()
    assert_topk_equal(ids, vals, want_ids, want_vals, f"M={M} N={N} k={k}")
    sel = sorted({0, M - 1})
    assert_topk_oracle_agrees(ids.cpu().numpy()[sel], vals.cpu().numpy()[sel],
                              oracle.w4a4_logits(x[sel], gx, *host_q))


def test_topk_decode_and_prefill(decode_case):
    pd, sw, gd = dev_weight(decode_case)
    for x in (synth.decode_x(64), synth.prefill_x()):
        gx, _ = input_global(x)
        gxd = torch.tensor([gx], dtype=torch.float32, device="cuda")
        xd = to_bf16_dev(x)
        ids, vals = nv.w4a4_lm_head_topk(xd, pd, sw, gd, gxd, 50)
        want_ids, want_vals = expected_topk(nv.w4a4_lm_head(xd, pd, sw, gd, gxd), 50)
        torch.cuda.synchronize()
        assert_topk_equal(ids, vals, want_ids, want_vals, f"M={x.shape[0]}")
