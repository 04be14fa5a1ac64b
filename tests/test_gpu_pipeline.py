"""The whole path on the GPU: quantize on the device, then the product, checked
against the oracle; and the CUDA-graph contract of refresh (captured
refresh + product replayed after the source weight changes)."""
import numpy as np
import pytest
import torch

import nvfp4_weight_only_rows_gb300 as nv
import oracle
import synth
from tests._gpu import assert_argmax_agrees, assert_logits_close, scales_bytes, to_bf16_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def test_device_quantize_then_product():
    N, K, M = 2000, 1536, 24
    W = synth.quant_weight(N=N, K=K, seed=40)
    x = synth.decode_x(M, K=K)
    packed, scales, g = nv.nvfp4_quantize_rows(to_bf16_dev(W))
    got = nv.w4a16_lm_head(to_bf16_dev(x), packed, scales, g).double().cpu().numpy()
    p, s, gg = oracle.quantize(W)
    ref = oracle.logits(x, p, s, gg)
    assert_logits_close(got, ref, "device quantize + product")
    assert_argmax_agrees(got, ref)


def test_cuda_graph_refresh_and_product():
    N, K, M = 1024, 1024, 8
    W1 = synth.quant_weight(N=N, K=K, seed=50)
    W2 = synth.quant_weight(N=N, K=K, seed=51)
    x = synth.decode_x(M, K=K)
    src = to_bf16_dev(W1)
    xd = to_bf16_dev(x)
    packed, scales, g = nv.nvfp4_quantize_rows(src)
    qws = torch.empty(nv.nvfp4_quantize_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    gws = torch.empty(nv.w4a16_lm_head_workspace_bytes(M, N, K), dtype=torch.uint8,
                      device="cuda")
    out = torch.empty(M, N, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up outside capture
        nv.nvfp4_refresh(src, packed, scales, g, workspace=qws)
        nv.w4a16_lm_head(xd, packed, scales, g, out=out, workspace=gws)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        nv.nvfp4_refresh(src, packed, scales, g, workspace=qws)
        nv.w4a16_lm_head(xd, packed, scales, g, out=out, workspace=gws)
    ptrs = (packed.data_ptr(), scales.data_ptr(), g.data_ptr(), out.data_ptr())
    for W in (W2, W1, W2):
        src.copy_(to_bf16_dev(W))
        graph.replay()
        torch.cuda.synchronize()
        p, sc, gg = oracle.quantize(W)
        assert np.array_equal(packed.cpu().numpy(), p)
        assert np.array_equal(scales_bytes(scales), sc)
        assert np.float32(g.item()) == gg
        ref = oracle.logits(x, p, sc, gg)
        assert_logits_close(out.double().cpu().numpy(), ref, "graph replay")
    assert (packed.data_ptr(), scales.data_ptr(), g.data_ptr(), out.data_ptr()) == ptrs
