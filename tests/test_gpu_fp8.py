"""GPU parity of the fp8 lm_head copy: the per-row E4M3 quantizer (bit-exact
against the CPU oracle), the per-token activation quantization inside the
W8A8 product (bit-exact, read from the workspace), the W8A8 logits (within
|err| <= 2e-3 * max|row| + 1e-3 of the oracle's float64 product of the same
quantized operands) and the fused argmax (bit-exact against the argmax of
the plain fp32 logits, and agreeing with the oracle's)."""
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


def gpu_quant(W_bits):
    q, s = nv.fp8_quantize_rows(to_bf16_dev(W_bits))
    torch.cuda.synchronize()
    return q.view(torch.uint8).cpu().numpy(), s.cpu().numpy()


def upload(q, s):
    return (torch.from_numpy(q).cuda().view(torch.float8_e4m3fn), torch.from_numpy(s).cuda())


@pytest.mark.parametrize("N,K", [(512, 256), (129, 272), (7, 16), (300, 4096), (33, 8208),
                                 (5, 16384), (3, 65536)])
def test_quantizer_bit_exact(N, K):
    """Every code and every row scale, for row lengths that use 128 to 1024
    threads per row, ragged K included."""
    W = synth.quant_weight(N=N, K=K, seed=N + K)
    q, s = gpu_quant(W)
    rq, rs = oracle.fp8_quantize(W)
    assert np.array_equal(s.view(np.uint32), rs.view(np.uint32))
    bad = np.argwhere(q != rq)
    assert bad.size == 0, (bad[:5].tolist(), q[tuple(bad[0])], rq[tuple(bad[0])])


def test_quantizer_special_rows():
    """All-zero rows (scale 1e-12, codes 0 / 0x80 for -0), a row whose maximum
    is a single outlier, huge and tiny magnitudes, exact E4M3 ties."""
    K = 256
    Wf = synth.bf16_bits_to_f32(synth.quant_weight(N=8, K=K, seed=9)).copy()
    Wf[0] = 0.0
    Wf[1] = 0.0
    Wf[1, ::3] = -0.0
    Wf[2, 17] = 1e3
    Wf[3] *= 1e30
    Wf[4] *= 1e-30
    Wf[5, :16] = [448, -448, 1.0, 1.0625, 1.1875, 0, -0.0, 2 ** -9, 2 ** -10, 3 * 2 ** -10,
                  240, 232, -3.0, 2 ** -6, 7 * 2 ** -9, 100]
    Wf[5, 16:] = 0
    W = synth.f32_to_bf16_bits(Wf.astype(np.float32))
    q, s = gpu_quant(W)
    rq, rs = oracle.fp8_quantize(W)
    assert np.array_equal(s.view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q, rq)


def test_quantizer_nonfinite_status_and_refresh_in_place():
    W = synth.quant_weight(N=64, K=512, seed=2)
    Wd = to_bf16_dev(W)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    q, s = nv.fp8_quantize_rows(Wd, workspace=ws)
    assert nv.nvfp4_read_device_status(ws) == nv.Status.OK
    addr = (q.data_ptr(), s.data_ptr())
    W2 = synth.quant_weight(N=64, K=512, seed=3)
    Wd.copy_(to_bf16_dev(W2))
    nv.fp8_refresh(Wd, q, s, workspace=ws)
    torch.cuda.synchronize()
    rq, rs = oracle.fp8_quantize(W2)
    assert (q.data_ptr(), s.data_ptr()) == addr
    assert np.array_equal(q.view(torch.uint8).cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy(), rs)
    Wd[5, 7] = float("inf")
    nv.fp8_refresh(Wd, q, s, workspace=ws)
    assert nv.nvfp4_read_device_status(ws) == nv.Status.ERR_NONFINITE


def product_case(N, K, M, seed):
    W = synth.quant_weight(N=N, K=K, seed=seed)
    x = synth.decode_x(M, K=K)
    wq, ws = oracle.fp8_quantize(W)
    xq, xs = oracle.fp8_quantize(x)
    return x, (wq, ws), (xq, xs)


def test_tiny_workload():
    W, x = synth.tiny_weight(), synth.tiny_x()
    wq, ws = oracle.fp8_quantize(W)
    xq, xs = oracle.fp8_quantize(x)
    ref = oracle.fp8_logits(xq, xs, wq, ws)
    dev = upload(wq, ws)
    for dt in (torch.float32, torch.bfloat16):
        got = nv.w8a8_lm_head(to_bf16_dev(x), *dev, out_dtype=dt).double().cpu().numpy()
        assert_logits_close(got, ref, f"tiny {dt}", dt == torch.bfloat16)
        assert_argmax_agrees(got, ref, dt == torch.bfloat16)


@pytest.mark.parametrize("M,N,K", [(1, 300, 512), (5, 129, 256), (16, 128, 768),
                                   (17, 1000, 512), (64, 777, 1024), (100, 513, 256),
                                   (130, 260, 512), (200, 384, 1280), (1, 1, 256),
                                   (8, 216 * 128, 1024), (40, 300 * 128, 768), (3, 100, 16384),
                                   (256, 1000, 512), (300, 2000, 768), (600, 777, 272),
                                   (1024, 160 * 128, 256)])
def test_product_shapes(M, N, K):
    """Ragged tokens and rows, one and several token tiles, split-K tails,
    the longest K; from 256 tokens the 256-token tiles with 128-k stages
    (ragged token tile, K % 128 != 0, several units per CTA)."""
    x, (wq, ws), (xq, xs) = product_case(N, K, M, seed=M + N)
    ref_cols = np.unique(np.linspace(0, N - 1, min(N, 3000)).astype(np.int64))
    ref = oracle.fp8_logits(xq, xs, wq, ws, cols=ref_cols)
    got = nv.w8a8_lm_head(to_bf16_dev(x), *upload(wq, ws)).double().cpu().numpy()
    assert_logits_close(got[:, ref_cols], ref, f"M={M} N={N} K={K}")


def test_activation_quantization_bit_exact():
    """The workspace holds [256-byte status header][x as e4m3, M_pad x K]
    after a call: every activation code equals the oracle's."""
    M, N, K = 37, 256, 1024
    x, (wq, ws), (xq, xs) = product_case(N, K, M, seed=4)
    wsb = torch.empty(nv.w8a8_lm_head_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    nv.w8a8_lm_head(to_bf16_dev(x), *upload(wq, ws), workspace=wsb)
    torch.cuda.synchronize()
    got = wsb[256:256 + M * K].cpu().numpy().reshape(M, K)
    assert np.array_equal(got, xq)


def test_deterministic_and_errors():
    x, (wq, ws), _ = product_case(500, 512, 9, seed=8)
    xd, dev = to_bf16_dev(x), upload(wq, ws)
    a = nv.w8a8_lm_head(xd, *dev)
    b = nv.w8a8_lm_head(xd, *dev)
    assert torch.equal(a, b)
    assert nv.w8a8_lm_head(xd[:0], *dev).shape == (0, 500)
    with pytest.raises(nv.NVFP4Error) as e:
        nv.w8a8_lm_head(xd, *dev, workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.status == nv.Status.ERR_WORKSPACE


@pytest.fixture(scope="module")
def decode_case(decode_nvfp4):
    W = decode_nvfp4.W
    return W, oracle.fp8_quantize(W)


def test_decode_weight_quantizer_bit_exact(decode_case):
    W, (rq, rs) = decode_case
    q, s = gpu_quant(W)
    assert np.array_equal(s.view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q, rq)


@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_decode_workload(decode_case, M):
    """W[128256, 4096]: every logit of every token against the oracle."""
    _, (wq, ws) = decode_case
    x = synth.decode_x(M)
    xq, xs = oracle.fp8_quantize(x)
    got = nv.w8a8_lm_head(to_bf16_dev(x), *upload(wq, ws)).double().cpu().numpy()
    ref = oracle.fp8_logits(xq, xs, wq, ws)
    assert_logits_close(got, ref, f"decode M={M}")
    assert_argmax_agrees(got, ref)


def test_prefill_workload_sampled(decode_case):
    """x[2048, 4096], bf16 logits; 24 sampled tokens over all 128256 rows."""
    _, (wq, ws) = decode_case
    x = synth.prefill_x()
    got = nv.w8a8_lm_head(to_bf16_dev(x), *upload(wq, ws), out_dtype=torch.bfloat16)
    got = got.double().cpu().numpy()
    rows = np.unique(np.concatenate([[0, 127, 128, 2047], np.random.default_rng(5).integers(0, 2048, 20)]))
    xq, xs = oracle.fp8_quantize(x[rows])
    ref = oracle.fp8_logits(xq, xs, wq, ws)
    assert_logits_close(got[rows], ref, "prefill", True)


def first_max(L):
    m = L.amax(dim=1, keepdim=True)
    ids = (L == m).to(torch.int32).argmax(dim=1).to(torch.int64)
    return ids, L.gather(1, ids[:, None])[:, 0]


@pytest.mark.parametrize("M,N,K", [(1, 300, 512), (64, 777, 1024), (200, 5000, 256),
                                   (8, 216 * 128, 1024)])
def test_argmax_matches_plain_logits(M, N, K):
    x, (wq, ws), (xq, xs) = product_case(N, K, M, seed=M * 7 + N)
    xd, dev = to_bf16_dev(x), upload(wq, ws)
    ids, vals = nv.w8a8_lm_head_argmax(xd, *dev)
    want_ids, want_vals = first_max(nv.w8a8_lm_head(xd, *dev))
    torch.cuda.synchronize()
    assert torch.equal(ids, want_ids)
    assert torch.equal(vals, want_vals)
    sel = sorted({0, M - 1})
    ref = oracle.fp8_logits(xq[sel], xs[sel], wq, ws)
    onehot = np.full_like(ref, -np.inf)
    onehot[np.arange(len(sel)), ids.cpu().numpy()[sel]] = 0.0
    assert_argmax_agrees(onehot, ref)
    tol = logits_tolerance(ref)[:, 0]
    assert np.all(np.abs(vals.cpu().numpy()[sel] - ref[np.arange(len(sel)), ids.cpu().numpy()[sel]]) <= tol)


def test_argmax_decode_and_prefill(decode_case):
    _, (wq, ws) = decode_case
    dev = upload(wq, ws)
    for x in (synth.decode_x(64), synth.prefill_x()):
        xd = to_bf16_dev(x)
        ids, vals = nv.w8a8_lm_head_argmax(xd, *dev)
        want_ids, want_vals = first_max(nv.w8a8_lm_head(xd, *dev))
        torch.cuda.synchronize()
        assert torch.equal(ids, want_ids)
        assert torch.equal(vals, want_vals)


@pytest.mark.parametrize("M,N,K,k", [(1, 300, 512, 10), (64, 777, 1024, 50), (200, 5000, 256, 128),
                                     (8, 216 * 128, 1024, 50), (3, 7, 256, 7)])
def test_topk_matches_plain_logits(M, N, K, k):
    """The fused top-k of the W8A8 logits: bit for bit the k largest of the
    fp32 logits w8a8_lm_head writes, and oracle-agreeing on two tokens."""
    x, (wq, ws), (xq, xs) = product_case(N, K, M, seed=M * 5 + N)
    xd, dev = to_bf16_dev(x), upload(wq, ws)
    ids, vals = nv.w8a8_lm_head_topk(xd, *dev, k)
    want_ids, want_vals = expected_topk(nv.w8a8_lm_head(xd, *dev), k)
    torch.cuda.synchronize()
    assert_topk_equal(ids, vals, want_ids, want_vals, f"M={M} N={N} k={k}")
    sel = sorted({0, M - 1})
    assert_topk_oracle_agrees(ids.cpu().numpy()[sel], vals.cpu().numpy()[sel],
                              oracle.fp8_logits(xq[sel], xs[sel], wq, ws))


def test_topk_decode_and_prefill(decode_case):
    _, (wq, ws) = decode_case
    dev = upload(wq, ws)
    for x in (synth.decode_x(64), synth.prefill_x()):
        xd = to_bf16_dev(x)
        ids, vals = nv.w8a8_lm_head_topk(xd, *dev, 50)
        want_ids, want_vals = expected_topk(nv.w8a8_lm_head(xd, *dev), 50)
        torch.cuda.synchronize()
        assert_topk_equal(ids, vals, want_ids, want_vals, f"M={x.shape[0]}")
