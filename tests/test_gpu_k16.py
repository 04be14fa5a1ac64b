"""Every product over the whole K % 16 domain.

`KNvfp4Static.create_weights` on the page
"vllm/model_executor/layers/quantization/modelopt.py" asks only K % 16 == 0
of an NVFP4 weight, so every product must take any such K, not only the
multiples of 256 its fast path reads in place.  K in {16, 48, 272} has code
rows of an odd number of 8-byte words (K % 32 == 16), K in {896, 2880} has
scale rows that are not 16-byte multiples; K = 272 and 48 also end inside a
64-k scale atom of the W4A4 layout.  Each product is compared with the CPU
oracle (logits tolerance, argmax and top-k agreement) and, for the fused
argmax / top-k, bit for bit with the plain product's fp32 logits.
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_only_rows_gb300 as nv
import oracle
import synth
from tests._gpu import (assert_argmax_agrees, assert_logits_close, assert_topk_equal,
                        assert_topk_oracle_agrees, expected_topk, to_bf16_dev)

pytestmark = pytest.mark.gpu

KS = [16, 48, 272, 896, 2880]
SHAPES = [(5, 300), (130, 1000)]  # a decode-sized and a two-token-tile product


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def nvfp4_weight(N, K, seed):
    W = synth.quant_weight(N=N, K=K, seed=seed)
    host = oracle.quantize(W)
    p, s, g = host
    dev = (torch.from_numpy(p).cuda(), torch.from_numpy(s).cuda().view(torch.float8_e4m3fn),
           torch.tensor([g], dtype=torch.float32, device="cuda"))
    return W, host, dev


def argmax_rows(L):
    nan = torch.isnan(L)
    m = torch.where(nan, torch.full_like(L, -float("inf")), L).amax(dim=1, keepdim=True)
    return (L == m).to(torch.int32).argmax(dim=1).to(torch.int64)


@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("M,N", SHAPES)
def test_w4a16_products(M, N, K):
    _, host, dev = nvfp4_weight(N, K, seed=K + M)
    x = synth.decode_x(M, K=K)
    xd = to_bf16_dev(x)
    ref = oracle.logits(x, *host)
    L = nv.w4a16_lm_head(xd, *dev)
    got = L.double().cpu().numpy()
    assert_logits_close(got, ref, f"W4A16 M={M} N={N} K={K}")
    assert_argmax_agrees(got, ref)
    got16 = nv.w4a16_lm_head(xd, *dev, out_dtype=torch.bfloat16).double().cpu().numpy()
    assert_logits_close(got16, ref, f"W4A16 bf16 M={M} N={N} K={K}", True)
    ids, vals = nv.w4a16_lm_head_argmax(xd, *dev)
    assert torch.equal(ids, argmax_rows(L))
    assert torch.equal(vals, L.gather(1, ids[:, None])[:, 0])
    k = 20
    tids, tvals = nv.w4a16_lm_head_topk(xd, *dev, k)
    want_ids, want_vals = expected_topk(L, k)
    assert_topk_equal(tids, tvals, want_ids, want_vals, f"top-k K={K}")
    assert_topk_oracle_agrees(tids.cpu().numpy(), tvals.cpu().numpy(), ref)


@pytest.mark.parametrize("K", KS)
def test_w4a16_split_units(K):
    """More weight tiles than SMs: stream-K pieces over the ceil(K/256) stages."""
    M, N = 3, 153 * 128 + 5
    _, host, dev = nvfp4_weight(N, K, seed=K)
    x = synth.decode_x(M, K=K)
    got = nv.w4a16_lm_head(to_bf16_dev(x), *dev).double().cpu().numpy()
    assert_logits_close(got, oracle.logits(x, *host), f"W4A16 split K={K}")


@pytest.mark.parametrize("K", KS)
def test_w8a8_products(K):
    M, N = 9, 700
    W = synth.quant_weight(N=N, K=K, seed=K + 1)
    q, s = nv.fp8_quantize_rows(to_bf16_dev(W))
    rq, rs = oracle.fp8_quantize(W)
    assert np.array_equal(q.view(torch.uint8).cpu().numpy(), rq)
    x = synth.decode_x(M, K=K)
    xd = to_bf16_dev(x)
    xq, xs = oracle.fp8_quantize(x)
    ref = oracle.fp8_logits(xq, xs, rq, rs)
    L = nv.w8a8_lm_head(xd, q, s)
    got = L.double().cpu().numpy()
    assert_logits_close(got, ref, f"W8A8 K={K}")
    assert_argmax_agrees(got, ref)
    ids, vals = nv.w8a8_lm_head_argmax(xd, q, s)
    assert torch.equal(ids, argmax_rows(L))
    tids, tvals = nv.w8a8_lm_head_topk(xd, q, s, 16)
    want_ids, want_vals = expected_topk(L, 16)
    assert_topk_equal(tids, tvals, want_ids, want_vals, f"W8A8 top-k K={K}")


@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("M,N", SHAPES)
def test_w4a4_products(M, N, K):
    _, host, _ = nvfp4_weight(N, K, seed=K + 2)
    p, s, g = host
    sw = nv.nvfp4_swizzle_scales(torch.from_numpy(s).cuda())
    assert np.array_equal(sw.cpu().numpy(), oracle.swizzle_scales(s)), "interleave"
    x = synth.decode_x(M, K=K)
    xd = to_bf16_dev(x)
    gx, _ = oracle.global_scale(float(np.abs(synth.bf16_bits_to_f32(x)).max()))
    dev = (torch.from_numpy(p).cuda(), sw, torch.tensor([g], dtype=torch.float32, device="cuda"),
           torch.tensor([gx], dtype=torch.float32, device="cuda"))
    ref = oracle.w4a4_logits(x, gx, p, s, g)
    L = nv.w4a4_lm_head(xd, *dev)
    got = L.double().cpu().numpy()
    assert_logits_close(got, ref, f"W4A4 M={M} N={N} K={K}")
    assert_argmax_agrees(got, ref)
    ids, _ = nv.w4a4_lm_head_argmax(xd, *dev)
    assert torch.equal(ids, argmax_rows(L))
    tids, tvals = nv.w4a4_lm_head_topk(xd, *dev, 8)
    want_ids, want_vals = expected_topk(L, 8)
    assert_topk_equal(tids, tvals, want_ids, want_vals, f"W4A4 top-k K={K}")


@pytest.mark.parametrize("K", KS)
def test_grouped_product(K):
    E, N = 5, 200
    offs = np.array([0, 7, 7, 40, 41, 90], dtype=np.int32)
    qs = [oracle.quantize(synth.quant_weight(N=N, K=K, seed=K + e)) for e in range(E)]
    dev = (torch.from_numpy(np.stack([q[0] for q in qs])).cuda(),
           torch.from_numpy(np.stack([q[1] for q in qs])).cuda().view(torch.float8_e4m3fn),
           torch.tensor(np.array([q[2] for q in qs], dtype=np.float32)).cuda())
    x = synth.decode_x(int(offs[-1]), K=K)
    out = nv.w4a16_grouped_gemm(to_bf16_dev(x), torch.from_numpy(offs).cuda(), *dev)
    got = out.double().cpu().numpy()
    ref = oracle.grouped_logits(x, offs, [q[0] for q in qs], [q[1] for q in qs],
                                [q[2] for q in qs])
    assert_logits_close(got, ref, f"grouped K={K}")


def test_shapes_off_the_k16_grid_are_refused():
    W = synth.quant_weight(N=64, K=256, seed=1)
    _, _, dev = nvfp4_weight(64, 256, seed=1)
    for bad_k in (8, 264):
        x = torch.zeros(4, bad_k, dtype=torch.bfloat16, device="cuda")
        packed = torch.zeros(64, bad_k // 2, dtype=torch.uint8, device="cuda")
        scales = torch.zeros(64, bad_k // 16, dtype=torch.uint8, device="cuda")
        with pytest.raises(nv.NVFP4Error) as e:
            nv.w4a16_lm_head(x, packed, scales, dev[2],
                             workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
        assert e.value.status == nv.Status.ERR_SHAPE
    del W
