"""GPU parity of the fused greedy argmax (w4a16_lm_head_argmax).

Two bars:
* bit for bit against the fp32 logits the plain product writes for the same
  inputs: the token id is the smallest row holding the row maximum (a NaN
  counts as the maximum, first NaN wins; -0 equals +0), the value is that
  logit (+0 for a zero maximum);
* against the CPU oracle's fp64 logits: the chosen row agrees with the
  oracle's argmax unless the oracle's top two are closer than 1e-3, and the
  returned value is within the logits tolerance of the oracle's logit there.
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_only_rows_gb300 as nv
import oracle
import synth
from tests._gpu import assert_argmax_agrees, logits_tolerance, to_bf16_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def upload(p, s, g):
    return (torch.from_numpy(p).cuda(), torch.from_numpy(s).cuda().view(torch.float8_e4m3fn),
            torch.tensor([g], dtype=torch.float32, device="cuda"))


def expected_from_logits(L: torch.Tensor):
    """Row-wise (first index of the maximum, maximum) of fp32 logits on the
    device, a NaN counting as larger than every number."""
    nan = torch.isnan(L)
    has_nan = nan.any(dim=1)
    first_nan = nan.to(torch.int32).argmax(dim=1)
    m = torch.where(nan, torch.full_like(L, -float("inf")), L).amax(dim=1, keepdim=True)
    first_max = (L == m).to(torch.int32).argmax(dim=1)
    ids = torch.where(has_nan, first_nan, first_max).to(torch.int64)
    return ids, L.gather(1, ids[:, None])[:, 0]


def assert_same_as_plain(xd, dev_q, what=""):
    L = nv.w4a16_lm_head(xd, *dev_q)
    ids, vals = nv.w4a16_lm_head_argmax(xd, *dev_q)
    want_ids, want_vals = expected_from_logits(L)
    torch.cuda.synchronize()
    bad = (ids != want_ids).nonzero()
    assert bad.numel() == 0, (what, bad[:5].tolist(), ids[bad[:5, 0]].tolist(),
                              want_ids[bad[:5, 0]].tolist())
    both_nan = torch.isnan(vals) & torch.isnan(want_vals)
    both_zero = (vals == 0) & (want_vals == 0)  # a zero maximum is returned as +0
    same = (vals.view(torch.int32) == want_vals.view(torch.int32)) | both_nan | both_zero
    assert bool(same.all()), (what, vals[~same][:5].tolist(), want_vals[~same][:5].tolist())
    return ids.cpu().numpy(), vals.cpu().numpy()


def assert_oracle_agrees(ids, vals, ref):
    """ref: fp64 oracle logits of the same tokens over all N rows."""
    M = ref.shape[0]
    onehot = np.full_like(ref, -np.inf)
    onehot[np.arange(M), ids] = 0.0
    assert_argmax_agrees(onehot, ref)
    tol = logits_tolerance(ref)[:, 0]
    err = np.abs(vals.astype(np.float64) - ref[np.arange(M), ids])
    assert np.all(err <= tol), (err.max(), tol.min())


def test_tiny_workload():
    W, x = synth.tiny_weight(), synth.tiny_x()
    host_q = oracle.quantize(W)
    ids, vals = assert_same_as_plain(to_bf16_dev(x), upload(*host_q), "tiny")
    assert_oracle_agrees(ids, vals, oracle.logits(x, *host_q))


@pytest.mark.parametrize("M,N,K", [(1, 300, 512), (5, 129, 256), (16, 128, 768),
                                   (17, 1000, 512), (64, 777, 1024), (100, 513, 256),
                                   (130, 260, 512), (200, 384, 1280), (1, 1, 256),
                                   (300, 5000, 256)])
def test_ragged_shapes(M, N, K):
    """Ragged token and vocabulary tails, one and several token tiles."""
    W = synth.quant_weight(N=N, K=K, seed=M + N)
    x = synth.decode_x(M, K=K)
    host_q = oracle.quantize(W)
    ids, vals = assert_same_as_plain(to_bf16_dev(x), upload(*host_q), f"M={M} N={N} K={K}")
    assert_oracle_agrees(ids, vals, oracle.logits(x, *host_q))


@pytest.mark.parametrize("M,N,K", [(8, 216 * 128, 1024), (1, 153 * 128 + 5, 512),
                                   (40, 300 * 128, 768)])
def test_split_units(M, N, K):
    """Units cut between two CTAs by the stream-K tail; repeated calls agree."""
    W = synth.quant_weight(N=N, K=K, seed=N % 97)
    x = synth.decode_x(M, K=K)
    host_q = oracle.quantize(W)
    dev_q = upload(*host_q)
    xd = to_bf16_dev(x)
    ids, vals = assert_same_as_plain(xd, dev_q, f"split M={M} N={N}")
    for _ in range(2):
        i2, v2 = nv.w4a16_lm_head_argmax(xd, *dev_q)
        assert np.array_equal(i2.cpu().numpy(), ids)
        assert np.array_equal(v2.cpu().numpy().view(np.int32), vals.view(np.int32))
    sel = [0, M - 1]
    assert_oracle_agrees(ids[sel], vals[sel], oracle.logits(x[sel], *host_q))


def test_exact_ties_take_the_smallest_row():
    """Every vocabulary row equal: with one 256-k stage per unit no unit is
    split, all logits of a token are the same number and row 0 must win,
    across 157 weight tiles spread over all CTAs."""
    N, K, M = 157 * 128 + 3, 256, 9
    row = synth.quant_weight(N=1, K=K, seed=5)
    W = np.repeat(row, N, axis=0)
    x = synth.decode_x(M, K=K)
    host_q = oracle.quantize(W)
    dev_q = upload(*host_q)
    ids, vals = assert_same_as_plain(to_bf16_dev(x), dev_q, "ties")
    assert np.all(ids == 0)
    # the same with the tied maximum only at rows 4000 and 9000: 4000 wins
    Wb = synth.quant_weight(N=N, K=K, seed=6)
    xf = synth.bf16_bits_to_f32(x[:1])
    Wb[4000] = Wb[9000] = synth.f32_to_bf16_bits(xf * 8.0)[0]
    host_b = oracle.quantize(Wb)
    ids_b, _ = assert_same_as_plain(to_bf16_dev(x[:1]), upload(*host_b), "ties 2")
    assert ids_b[0] == 4000


def test_negative_maxima_and_nan_tokens():
    """A token whose logits are all negative, a token row holding a NaN
    (every logit of that token is NaN: row 0, value NaN) and an all-zero
    token row (all logits zero, of either sign: row 0, value +0)."""
    N, K, M = 1000, 512, 3
    x = synth.decode_x(M, K=K)
    xf = synth.bf16_bits_to_f32(x).copy()
    rng = np.random.default_rng(3)
    Wf = -np.abs(rng.uniform(0.5, 1.5, (N, 1))) * xf[0][None, :]
    W = synth.f32_to_bf16_bits(Wf.astype(np.float32))
    xf[1, 17] = np.nan
    xf[2] = 0.0  # every logit of token 2 is a zero (+0 or -0): row 0, value +0
    xn = synth.f32_to_bf16_bits(xf)
    host_q = oracle.quantize(W)
    ids, vals = assert_same_as_plain(to_bf16_dev(xn), upload(*host_q), "neg/nan")
    assert vals[0] < 0
    assert ids[1] == 0 and np.isnan(vals[1])
    assert ids[2] == 0 and vals[2] == 0 and not np.signbit(vals[2])
    assert_oracle_agrees(ids[:1], vals[:1], oracle.logits(x[:1], *host_q))


def test_no_values_empty_and_status():
    W = synth.quant_weight(N=500, K=512, seed=8)
    x = synth.decode_x(9, K=512)
    host_q = oracle.quantize(W)
    dev_q = upload(*host_q)
    xd = to_bf16_dev(x)
    ws = torch.empty(nv.w4a16_lm_head_argmax_workspace_bytes(9, 500, 512), dtype=torch.uint8,
                     device="cuda")
    ids, vals = nv.w4a16_lm_head_argmax(xd, *dev_q, with_values=False, workspace=ws)
    assert vals is None
    assert nv.nvfp4_read_device_status(ws) == nv.Status.OK
    ids2, _ = nv.w4a16_lm_head_argmax(xd, *dev_q)
    assert torch.equal(ids, ids2)
    e_ids, e_vals = nv.w4a16_lm_head_argmax(xd[:0], *dev_q)
    assert e_ids.shape == (0,) and e_vals.shape == (0,)


@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_decode_workload(decode_nvfp4, M):
    """W[128256, 4096] quantized on the GPU: every token bit for bit against
    the plain product and against the oracle over all 128256 rows."""
    x = synth.decode_x(M)
    ids, vals = assert_same_as_plain(to_bf16_dev(x), decode_nvfp4.dev, f"decode M={M}")
    assert_oracle_agrees(ids, vals, oracle.logits(x, *decode_nvfp4.ref))


def test_prefill_workload(decode_nvfp4):
    """x[2048, 4096] (16 token tiles): all tokens against the plain product,
    64 tokens (each tile's first and last two) against the oracle."""
    x = synth.prefill_x()
    ids, vals = assert_same_as_plain(to_bf16_dev(x), decode_nvfp4.dev, "prefill")
    sel = np.array(sorted({t for t0 in range(0, 2048, 128) for t in (t0, t0 + 1, t0 + 126, t0 + 127)}))
    assert_oracle_agrees(ids[sel], vals[sel], oracle.logits(x[sel], *decode_nvfp4.ref))


def test_graph_replay():
    """Captured once, replayed on new activations copied into the same buffer."""
    N, K, M = 3000, 1024, 16
    host_q = oracle.quantize(synth.quant_weight(N=N, K=K, seed=12))
    dev_q = upload(*host_q)
    x1, x2 = synth.decode_x(M, K=K), synth.sweep_x(M, K=K)
    xd = to_bf16_dev(x1)
    ids = torch.empty(M, dtype=torch.int64, device="cuda")
    vals = torch.empty(M, dtype=torch.float32, device="cuda")
    ws = torch.empty(nv.w4a16_lm_head_argmax_workspace_bytes(M, N, K), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        nv.w4a16_lm_head_argmax(xd, *dev_q, token_ids=ids, max_logits=vals, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nv.w4a16_lm_head_argmax(xd, *dev_q, token_ids=ids, max_logits=vals, workspace=ws)
    for xb in (x2, x1, x2):
        xd.copy_(to_bf16_dev(xb))
        g.replay()
        want_ids, want_vals = expected_from_logits(nv.w4a16_lm_head(xd, *dev_q))
        torch.cuda.synchronize()
        assert torch.equal(ids, want_ids)
        assert torch.equal(vals, want_vals)
