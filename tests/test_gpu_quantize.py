"""GPU parity of the NVFP4 row quantizer against the CPU oracle (bit-exact).

Every case calls the CUDA kernels through the C ABI (the ctypes binding in
nvfp4_weight_only_rows_gb300) and compares packed codes, E4M3 scales and the
global scale byte for byte with oracle.quantize.  Every row of the
full-size workload weights is compared in test_gpu_workloads.py.
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_only_rows_gb300 as nv
import oracle
import synth
from tests import _fixtures
from tests._gpu import scales_bytes, to_bf16_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def gpu_quantize(W_bits):
    Wd = to_bf16_dev(W_bits)
    packed, scales, g = nv.nvfp4_quantize_rows(Wd)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), scales_bytes(scales), np.float32(g.item())


def assert_same(W_bits):
    p, s, g = gpu_quantize(W_bits)
    p_ref, s_ref, g_ref = oracle.quantize(W_bits)
    assert g == g_ref, (g, g_ref)
    assert np.array_equal(s, s_ref), np.argwhere(s != s_ref)[:5]
    assert np.array_equal(p, p_ref), np.argwhere(p != p_ref)[:5]


def test_hand_blocks():
    W, g, S, P = _fixtures.hand_blocks()
    p, s, gg = gpu_quantize(W)
    assert gg == g
    assert np.array_equal(s, S)
    assert np.array_equal(p, P)


def test_tiny_workload():
    assert_same(synth.tiny_weight())


@pytest.mark.parametrize("N,K", [(1, 16), (37, 48), (3, 272), (129, 256), (1000, 784),
                                 (257, 4096), (2, 8208)])
def test_ragged_shapes(N, K):
    assert_same(synth.quant_weight(N=N, K=K, seed=N + K))


def test_distributions_and_special_values():
    rng = np.random.default_rng(1)
    N, K = 64, 512
    W = synth.weight(N, K, seed=3, sigma=1.0)
    Wf = synth.bf16_bits_to_f32(W).copy()
    Wf[1] *= 1e-6                          # subnormal-range block scales
    Wf[2] = 0.0                             # all-zero row
    Wf[3, ::2] = -0.0                       # negative zeros
    Wf[4] = rng.choice([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], size=K) * \
        rng.choice([-1.0, 1.0], size=K)     # midpoints once scaled
    Wf[5, :16] = [6.0] + [5.0] * 15
    Wf[6] *= 1e3                            # heavy row
    W2 = synth.f32_to_bf16_bits(Wf)
    W2[3, ::2] = 0x8000
    assert_same(W2)
    # global scale clamped at 1e-12
    assert_same(np.zeros((8, 64), dtype=np.uint16))
    tiny = synth.f32_to_bf16_bits(np.full((4, 32), 1e-20, dtype=np.float32))
    assert_same(tiny)


def test_nonfinite_weight_sets_device_status():
    W = synth.quant_weight(N=16, K=64, seed=2)
    for bad in (0x7F80, 0xFF80, 0x7FC1):
        W2 = W.copy()
        W2[7, 33] = bad
        Wd = to_bf16_dev(W2)
        ws = torch.empty(nv.nvfp4_quantize_workspace_bytes(16, 64), dtype=torch.uint8,
                         device="cuda")
        packed, scales, g = nv.nvfp4_quantize_rows(Wd, workspace=ws)
        assert nv.nvfp4_read_device_status(ws) == nv.Status.ERR_NONFINITE
        assert torch.isnan(g).item()
    # a clean call on the same workspace resets the status word
    nv.nvfp4_quantize_rows(to_bf16_dev(W), workspace=ws)
    assert nv.nvfp4_read_device_status(ws) == nv.Status.OK


def test_refresh_in_place_keeps_addresses():
    N, K = 300, 1024
    W1 = synth.quant_weight(N=N, K=K, seed=4)
    W2 = synth.quant_weight(N=N, K=K, seed=5)
    src = to_bf16_dev(W1)
    packed, scales, g = nv.nvfp4_quantize_rows(src)
    ptrs = (packed.data_ptr(), scales.data_ptr(), g.data_ptr())
    src.copy_(to_bf16_dev(W2))
    nv.nvfp4_refresh(src, packed, scales, g)
    torch.cuda.synchronize()
    assert (packed.data_ptr(), scales.data_ptr(), g.data_ptr()) == ptrs
    p_ref, s_ref, g_ref = oracle.quantize(W2)
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    assert np.array_equal(scales_bytes(scales), s_ref)
    assert np.float32(g.item()) == g_ref
