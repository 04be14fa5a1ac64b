"""GPU parity of the fused top-k (w4a16_lm_head_topk).

Two bars, as for the fused argmax:
* bit for bit against the fp32 logits the plain product writes for the same
  inputs: the k largest by value (a NaN above every number, -0 equal to +0
  and returned as +0), of equal values the smaller row first;
* against the CPU oracle's fp64 logits: every returned value is within the
  logits tolerance of the oracle's logit at that row, and no row left out
  has an oracle logit above the smallest returned one by more than twice the
  tolerance (what the tolerance allows two near-equal logits to swap).
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_only_rows_gb300 as nv
import oracle
import synth
from tests._gpu import (assert_topk_equal, assert_topk_oracle_agrees, expected_topk,
                        to_bf16_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def upload(p, s, g):
    return (torch.from_numpy(p).cuda(), torch.from_numpy(s).cuda().view(torch.float8_e4m3fn),
            torch.tensor([g], dtype=torch.float32, device="cuda"))


def assert_same_as_plain(xd, dev_q, k, what=""):
    L = nv.w4a16_lm_head(xd, *dev_q)
    ids, vals = nv.w4a16_lm_head_topk(xd, *dev_q, k)
    want_ids, want_vals = expected_topk(L, k)
    torch.cuda.synchronize()
    assert_topk_equal(ids, vals, want_ids, want_vals, what)
    return ids.cpu().numpy(), vals.cpu().numpy()


assert_oracle_agrees = assert_topk_oracle_agrees


def test_tiny_workload():
    W, x = synth.tiny_weight(), synth.tiny_x()
    host_q = oracle.quantize(W)
    ref = oracle.logits(x, *host_q)
    for k in (1, 4, 50, 128):
        ids, vals = assert_same_as_plain(to_bf16_dev(x), upload(*host_q), k, f"tiny k={k}")
        assert_oracle_agrees(ids, vals, ref)
        want_ids, _ = oracle.topk(ref, k)
        # the oracle's own top-k agrees wherever its neighbours are not near-tied
        assert ids[:, 0].tolist() == want_ids[:, 0].tolist()


@pytest.mark.parametrize("M,N,K,k", [(1, 300, 512, 10), (5, 129, 256, 128), (17, 1000, 512, 50),
                                     (64, 777, 1024, 33), (100, 513, 256, 64),
                                     (130, 260, 512, 7), (200, 384, 1280, 100), (1, 1, 256, 1),
                                     (3, 7, 256, 7), (300, 5000, 256, 50),
                                     (2, 262144, 256, 128), (2, 262144 + 33, 256, 50),
                                     (64, 40000, 256, 128), (256, 4097, 256, 128),
                                     (257, 3000, 256, 50), (300, 7, 256, 7), (270, 33, 512, 1)])
def test_ragged_shapes(M, N, K, k):
    """Ragged token and vocabulary tails, k up to N and up to the limit; the
    largest vocabulary the logits route takes (262144 rows) and one past it,
    the most tokens it takes (256) and one more; past 256 tokens, a
    vocabulary inside one 32-row group and one just past it."""
    W = synth.quant_weight(N=N, K=K, seed=M + N)
    x = synth.decode_x(M, K=K)
    host_q = oracle.quantize(W)
    ids, vals = assert_same_as_plain(to_bf16_dev(x), upload(*host_q), k, f"M={M} N={N} k={k}")
    sel = sorted({0, M // 2, M - 1})
    assert_oracle_agrees(ids[sel], vals[sel], oracle.logits(x[sel], *host_q))


@pytest.mark.parametrize("M,N,K,k", [(8, 216 * 128, 1024, 50), (1, 153 * 128 + 5, 512, 20),
                                     (40, 300 * 128, 768, 128), (260, 300 * 128 + 5, 512, 50),
                                     (513, 2000 * 8 + 3, 256, 128)])
def test_split_units_and_repeats(M, N, K, k):
    """Units cut between two CTAs by the stream-K tail; repeated calls agree.
    The cases past 256 tokens take the candidate route, with a vocabulary
    that is not a multiple of 8 rows, so that the candidate slots of one
    token start inside a 32-byte sector."""
    W = synth.quant_weight(N=N, K=K, seed=N % 89)
    x = synth.decode_x(M, K=K)
    host_q = oracle.quantize(W)
    dev_q = upload(*host_q)
    xd = to_bf16_dev(x)
    ids, vals = assert_same_as_plain(xd, dev_q, k, f"split M={M} N={N}")
    for _ in range(2):
        i2, v2 = nv.w4a16_lm_head_topk(xd, *dev_q, k)
        assert np.array_equal(i2.cpu().numpy(), ids)
        assert np.array_equal(v2.cpu().numpy().view(np.int32), vals.view(np.int32))


def test_first_column_is_the_argmax():
    N, K, M = 5000, 512, 37
    host_q = oracle.quantize(synth.quant_weight(N=N, K=K, seed=21))
    dev_q = upload(*host_q)
    xd = to_bf16_dev(synth.decode_x(M, K=K))
    ids, vals = nv.w4a16_lm_head_topk(xd, *dev_q, 16)
    a_ids, a_vals = nv.w4a16_lm_head_argmax(xd, *dev_q)
    torch.cuda.synchronize()
    assert torch.equal(ids[:, 0], a_ids)
    assert torch.equal(vals[:, 0], a_vals)


# Up to 256 tokens the call writes the fp32 logits and their 32-row maxima
# and one CTA per token selects from them (64 tokens and fewer on the
# decode-tile GEMM, more on the 128-token tile); more tokens keep
# thresholded candidates in the GEMM epilogue: the cases below run all three.
ROUTES = [1, 5, 70, 300]


@pytest.mark.parametrize("M", ROUTES)
def test_all_rows_tied(M):
    """Every vocabulary row equal: every logit of a token is the same number,
    so every one reaches the threshold (more candidates than the selection
    keeps in shared memory) and rows 0 .. k-1 must come out, in order."""
    N, K = 157 * 128 + 3, 256
    row = synth.quant_weight(N=1, K=K, seed=5)
    host_q = oracle.quantize(np.repeat(row, N, axis=0))
    x = synth.decode_x(M, K=K)
    for k in (1, 50, 128):
        ids, vals = assert_same_as_plain(to_bf16_dev(x), upload(*host_q), k, f"ties k={k}")
        assert np.all(ids == np.arange(k)[None, :])
        assert np.all(vals == vals[:, :1])


@pytest.mark.parametrize("M", ROUTES)
def test_tied_rows_within_shared_memory(M):
    """3000 equal rows: every logit is a candidate at the final threshold,
    more than the one-warp ranking takes and few enough for the radix
    selection over shared memory; rows 0 .. k-1 must come out, in order."""
    N, K = 3000, 256
    row = synth.quant_weight(N=1, K=K, seed=7)
    host_q = oracle.quantize(np.repeat(row, N, axis=0))
    x = synth.decode_x(M, K=K)
    for k in (1, 37, 128):
        ids, vals = assert_same_as_plain(to_bf16_dev(x), upload(*host_q), k, f"ties3000 k={k}")
        assert np.all(ids == np.arange(k)[None, :])


@pytest.mark.parametrize("M", ROUTES)
def test_rising_logits(M):
    """Logits that grow with the row: later tiles keep beating the
    thresholds that earlier ones set."""
    N, K = 30000, 256
    x = synth.decode_x(M, K=K)
    xf = synth.bf16_bits_to_f32(x)
    ramp = np.linspace(0.01, 1.0, N, dtype=np.float32)[:, None]
    W = synth.f32_to_bf16_bits((ramp * xf[0][None, :]).astype(np.float32))
    host_q = oracle.quantize(W)
    ids, vals = assert_same_as_plain(to_bf16_dev(x), upload(*host_q), 64, "rising")
    assert_oracle_agrees(ids[:1], vals[:1], oracle.logits(x[:1], *host_q))


@pytest.mark.parametrize("M", ROUTES)
def test_large_logits_clustered_by_row_residue(M):
    """50 large logit values, each repeated on every row with the same
    residue mod 256: equal values fill the largest group and super-group
    maxima of the selection from logits and the top histogram bins of the
    candidate route, and the k largest must still come out by value, then
    by row."""
    N, K = 2 * 4096 + 300, 256
    x = synth.decode_x(M, K=K)
    xf = synth.bf16_bits_to_f32(x)
    t = np.arange(N) % 256
    c = np.where(t < 50, 1.0 + t / 64.0, 0.01).astype(np.float32)[:, None]
    W = synth.f32_to_bf16_bits((c * xf[0][None, :]).astype(np.float32))
    host_q = oracle.quantize(W)
    for k in (1, 50, 128):
        ids, vals = assert_same_as_plain(to_bf16_dev(x), upload(*host_q), k, f"clustered k={k}")
        assert_oracle_agrees(ids[:1], vals[:1], oracle.logits(x[:1], *host_q))


@pytest.mark.parametrize("M", [3, 70, 300])
def test_negative_nan_and_zero_tokens(M):
    """All-negative logits, a NaN token (every logit NaN: rows 0 .. k-1, all
    values NaN) and an all-zero token (rows 0 .. k-1, values +0)."""
    N, K, k = 1000, 512, 20
    x = synth.decode_x(M, K=K)
    xf = synth.bf16_bits_to_f32(x).copy()
    rng = np.random.default_rng(3)
    Wf = -np.abs(rng.uniform(0.5, 1.5, (N, 1))) * xf[0][None, :]
    host_q = oracle.quantize(synth.f32_to_bf16_bits(Wf.astype(np.float32)))
    xf[1, 17] = np.nan
    xf[2] = 0.0
    xn = synth.f32_to_bf16_bits(xf)
    ids, vals = assert_same_as_plain(to_bf16_dev(xn), upload(*host_q), k, "neg/nan/zero")
    assert np.all(vals[0] < 0)
    assert ids[1].tolist() == list(range(k)) and np.all(np.isnan(vals[1]))
    assert ids[2].tolist() == list(range(k))
    assert np.all(vals[2] == 0) and not np.any(np.signbit(vals[2]))
    assert_oracle_agrees(ids[:1], vals[:1], oracle.logits(x[:1], *host_q))


def test_no_values_empty_and_status():
    N, K, M, k = 500, 512, 9, 5
    host_q = oracle.quantize(synth.quant_weight(N=N, K=K, seed=8))
    dev_q = upload(*host_q)
    xd = to_bf16_dev(synth.decode_x(M, K=K))
    ws = torch.empty(nv.w4a16_lm_head_topk_workspace_bytes(M, N, K, k), dtype=torch.uint8,
                     device="cuda")
    ids, vals = nv.w4a16_lm_head_topk(xd, *dev_q, k, with_values=False, workspace=ws)
    assert vals is None
    assert nv.nvfp4_read_device_status(ws) == nv.Status.OK
    ids2, _ = nv.w4a16_lm_head_topk(xd, *dev_q, k)
    assert torch.equal(ids, ids2)
    e_ids, e_vals = nv.w4a16_lm_head_topk(xd[:0], *dev_q, k)
    assert e_ids.shape == (0, k) and e_vals.shape == (0, k)
    for bad_k in (0, N + 1, nv.TOPK_MAX + 1):
        with pytest.raises(nv.NVFP4Error) as e:
            nv.w4a16_lm_head_topk(xd, *dev_q, bad_k)
        assert e.value.status == nv.Status.ERR_SHAPE


@pytest.mark.parametrize("M,k", [(1, 50), (8, 50), (32, 50), (64, 50), (64, 128), (16, 1)])
def test_decode_workload(decode_nvfp4, M, k):
    """W[128256, 4096] quantized on the GPU: every token bit for bit against
    the plain product and against the oracle over all 128256 rows."""
    x = synth.decode_x(M)
    ids, vals = assert_same_as_plain(to_bf16_dev(x), decode_nvfp4.dev, k, f"decode M={M}")
    assert_oracle_agrees(ids, vals, oracle.logits(x, *decode_nvfp4.ref))


def test_prefill_workload(decode_nvfp4):
    """x[2048, 4096] (16 token tiles), k = 50: all tokens against the plain
    product, 64 tokens (each tile's first and last two) against the oracle."""
    x = synth.prefill_x()
    ids, vals = assert_same_as_plain(to_bf16_dev(x), decode_nvfp4.dev, 50, "prefill")
    sel = np.array(sorted({t for t0 in range(0, 2048, 128) for t in (t0, t0 + 1, t0 + 126, t0 + 127)}))
    assert_oracle_agrees(ids[sel], vals[sel], oracle.logits(x[sel], *decode_nvfp4.ref))


def test_graph_replay():
    """Captured once (both kernels), replayed on new activations."""
    N, K, M, k = 3000, 1024, 16, 40
    host_q = oracle.quantize(synth.quant_weight(N=N, K=K, seed=12))
    dev_q = upload(*host_q)
    x1, x2 = synth.decode_x(M, K=K), synth.sweep_x(M, K=K)
    xd = to_bf16_dev(x1)
    ids = torch.empty((M, k), dtype=torch.int64, device="cuda")
    vals = torch.empty((M, k), dtype=torch.float32, device="cuda")
    ws = torch.empty(nv.w4a16_lm_head_topk_workspace_bytes(M, N, K, k), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        nv.w4a16_lm_head_topk(xd, *dev_q, k, token_ids=ids, values=vals, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nv.w4a16_lm_head_topk(xd, *dev_q, k, token_ids=ids, values=vals, workspace=ws)
    for xb in (x2, x1, x2):
        xd.copy_(to_bf16_dev(xb))
        g.replay()
        want_ids, want_vals = expected_topk(nv.w4a16_lm_head(xd, *dev_q), k)
        torch.cuda.synchronize()
        assert torch.equal(ids, want_ids)
        assert torch.equal(vals, want_vals)
