"""GPU parity of the grouped (MoE) NVFP4 W4A16 product: every output row
against the oracle's per-expert product (|err| <= 2e-3 * max|row| + 1e-3),
on ragged, empty and skewed groups, MoE-shaped w13 / w2 products, and a
CUDA graph replayed with new routing (the offsets are read on the device)."""
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


def experts(E, N, K, seed):
    qs = [oracle.quantize(synth.quant_weight(N=N, K=K, seed=seed + e)) for e in range(E)]
    host = ([q[0] for q in qs], [q[1] for q in qs], [q[2] for q in qs])
    dev = (torch.from_numpy(np.stack(host[0])).cuda(),
           torch.from_numpy(np.stack(host[1])).cuda().view(torch.float8_e4m3fn),
           torch.tensor(np.array(host[2], dtype=np.float32)).cuda())
    return host, dev


def routed_offsets(E, tokens, topk, seed):
    """A synthetic router: each token picks topk distinct experts (seeded);
    returns the expert-sorted row counts as offsets."""
    rng = np.random.default_rng(seed)
    counts = np.zeros(E, dtype=np.int64)
    for _ in range(tokens):
        counts[rng.choice(E, topk, replace=False)] += 1
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def run(x, offs, dev, dt=torch.float32):
    out = nv.w4a16_grouped_gemm(to_bf16_dev(x), torch.from_numpy(offs).cuda(), *dev, out_dtype=dt)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


@pytest.mark.parametrize("offs", [[0, 5, 5, 6, 37], [0, 37, 37, 37, 37], [0, 1, 2, 3, 4],
                                  [0, 0, 0, 0, 200], [0, 100, 130, 260, 300],
                                  [0, 129, 129, 385, 400]])
def test_ragged_and_empty_groups(offs):
    """Empty, single-row and ragged groups; the last two sets take 128-token
    tiles whose partly filled last tile per group gets MMAs only as wide as
    its tokens (16 to 112 of them)."""
    E, N, K = 4, 300, 512
    offs = np.array(offs, dtype=np.int32)
    host, dev = experts(E, N, K, seed=3)
    x = synth.decode_x(int(offs[-1]), K=K)
    ref = oracle.grouped_logits(x, offs, *host)
    got = run(x, offs, dev)
    assert_logits_close(got, ref, f"offs={offs.tolist()}")


@pytest.mark.parametrize("tokens,N,K", [(64, 1536, 2048), (64, 2048, 768), (512, 1536, 2048)])
def test_moe_shapes(tokens, N, K):
    """64 experts, top-8 routing: w13 (N = 2I = 1536, K = H = 2048) and w2
    (N = H = 2048, K = I = 768) for a decode batch, w13 for a larger batch."""
    E, topk = 64, 8
    offs = routed_offsets(E, tokens, topk, seed=tokens + N)
    host, dev = experts(E, N, K, seed=100)
    x = synth.decode_x(int(offs[-1]), K=K)
    got = run(x, offs, dev, torch.bfloat16 if tokens > 64 else torch.float32)
    rows = np.arange(int(offs[-1])) if tokens <= 64 else np.unique(
        np.concatenate([offs[:-1], offs[1:] - 1, np.random.default_rng(1).integers(0, offs[-1], 64)]))
    rows = rows[(rows >= 0) & (rows < offs[-1])]
    ref = oracle.grouped_logits(x, offs, *host)[rows]
    assert_logits_close(got[rows], ref, f"moe tokens={tokens} N={N} K={K}", tokens > 64)


def test_deterministic_and_graph_with_new_routing():
    E, N, K = 8, 512, 1024
    host, dev = experts(E, N, K, seed=7)
    M = 96
    x = synth.decode_x(M, K=K)
    xd = to_bf16_dev(x)
    offs_a = np.array([0, 10, 10, 40, 41, 60, 90, 95, 96], dtype=np.int32)
    offs_b = np.array([0, 0, 50, 50, 50, 51, 52, 96, 96], dtype=np.int32)
    od = torch.from_numpy(offs_a).cuda()
    out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    ws = torch.empty(nv.w4a16_grouped_workspace_bytes(M, N, K, E), dtype=torch.uint8, device="cuda")
    a1 = nv.w4a16_grouped_gemm(xd, od, *dev, out=out, workspace=ws).clone()
    a2 = nv.w4a16_grouped_gemm(xd, od, *dev, out=out, workspace=ws).clone()
    assert torch.equal(a1, a2)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        nv.w4a16_grouped_gemm(xd, od, *dev, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nv.w4a16_grouped_gemm(xd, od, *dev, out=out, workspace=ws)
    for offs in (offs_b, offs_a, offs_b):
        od.copy_(torch.from_numpy(offs))
        g.replay()
        torch.cuda.synchronize()
        assert_logits_close(out.double().cpu().numpy(), oracle.grouped_logits(x, offs, *host),
                            f"graph offs={offs.tolist()}")
