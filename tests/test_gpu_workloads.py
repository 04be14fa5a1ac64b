"""GPU parity on the full-size seeded workloads, with nothing sampled where
the oracle can afford every value.

* The NVFP4 row quantizer (``_quantize_nvfp4`` on the page
  "vllm.model_executor.layers.quantization.online.lm_head") runs on the GPU
  through the C ABI on every workload's weight -- W[128256, 4096] (decode
  and prefill), W[151936, 5120] with Student-t row scales (seed 4, then the
  in-place refresh to seed 5), W[262144, 8192] (sweep) -- and every packed
  byte, every E4M3 scale byte and the global scale must equal the oracle's.
* The W4A16 product then multiplies those DEVICE-quantized buffers (not an
  upload of the oracle's bytes): decode M in {1, 8, 32, 64} and the sweep at
  M in {1, 4, 16, 64, 256} on every logit; prefill M = 2048 on the first and
  last 8 tokens of each of its 16 token tiles (256 tokens) over every
  vocabulary row; the sweep at M = 1024 on 64 tokens (every tile edge) over
  every row plus every token over 512 rows.  Bar: |err| <= 2e-3 * max|row| +
  1e-3 (plus half a bf16 ulp for bf16 logits), argmax agreeing unless the
  oracle's top two are within 1e-3.
"""
import numpy as np
import pytest
import torch

import nvfp4_weight_only_rows_gb300 as nv
import oracle
import synth
from tests._gpu import assert_argmax_agrees, assert_logits_close, scales_bytes, to_bf16_dev

pytestmark = pytest.mark.gpu


def assert_bytes_equal(dev, ref, what):
    packed, scales, g = dev
    p_ref, s_ref, g_ref = ref
    assert np.float32(g.item()) == g_ref, (what, "global", g.item(), g_ref)
    s = scales_bytes(scales)
    bad = np.argwhere(s != s_ref)
    assert bad.size == 0, (what, "scales", bad[:5].tolist())
    p = packed.cpu().numpy()
    bad = np.argwhere(p != p_ref)
    assert bad.size == 0, (what, "packed", bad[:5].tolist())


def product(x_bits, dev, out_dtype=torch.float32):
    out = nv.w4a16_lm_head(to_bf16_dev(x_bits), *dev, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out


def tile_edge_tokens(M, tile=128, each=8):
    """The first and last `each` token rows of every `tile`-row token tile."""
    rows = []
    for t0 in range(0, M, tile):
        t1 = min(M, t0 + tile)
        rows.extend(range(t0, min(t1, t0 + each)))
        rows.extend(range(max(t0, t1 - each), t1))
    return np.unique(np.array(rows, dtype=np.int64))


# ------------------------------------------------ decode / prefill weight
def test_decode_weight_quantized_bit_exact_every_row(decode_nvfp4):
    assert_bytes_equal(decode_nvfp4.dev, decode_nvfp4.ref, "W[128256,4096]")


@pytest.mark.parametrize("M", [1, 8, 32, 64])
def test_decode_on_device_quantized_weight(decode_nvfp4, M):
    """fp32 logits, every token x every one of the 128256 rows."""
    x = synth.decode_x(M)
    got = product(x, decode_nvfp4.dev).double().cpu().numpy()
    ref = oracle.logits(x, *decode_nvfp4.ref)
    assert_logits_close(got, ref, f"decode M={M}")
    assert_argmax_agrees(got, ref)


def test_prefill_tile_edges_on_device_quantized_weight(decode_nvfp4):
    """x[2048, 4096], bf16 logits: 256 tokens (the first and last 8 of each
    of the 16 token tiles) x every vocabulary row."""
    x = synth.prefill_x()
    got = product(x, decode_nvfp4.dev, torch.bfloat16)
    rows = tile_edge_tokens(2048)
    assert rows.size == 256
    sel = got[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    del got
    ref = oracle.logits(x[rows], *decode_nvfp4.ref)
    assert_logits_close(sel, ref, "prefill", True)
    assert_argmax_agrees(sel, ref, True)


# ------------------------------------------------ quantize / refresh weight
def test_quant_workload_and_refresh_bit_exact_every_row():
    """W[151936, 5120] (Student-t row scales): seed 4 quantized, then seed 5
    refreshed into the same buffers (addresses kept); both compared in full."""
    N, K = 151936, 5120
    W4 = synth.quant_weight(N=N, K=K, seed=4)
    src = to_bf16_dev(W4)
    dev = nv.nvfp4_quantize_rows(src)
    torch.cuda.synchronize()
    assert_bytes_equal(dev, oracle.quantize(W4), "W[151936,5120] seed 4")
    del W4
    ptrs = tuple(t.data_ptr() for t in dev)
    W5 = synth.quant_weight(N=N, K=K, seed=5)
    src.copy_(to_bf16_dev(W5))
    nv.nvfp4_refresh(src, *dev)
    torch.cuda.synchronize()
    assert tuple(t.data_ptr() for t in dev) == ptrs
    assert_bytes_equal(dev, oracle.quantize(W5), "W[151936,5120] seed 5 (refresh)")


# ------------------------------------------------ large-vocabulary sweep
@pytest.fixture(scope="module")
def sweep_nvfp4():
    W = synth.sweep_weight()
    Wd = to_bf16_dev(W)
    dev = nv.nvfp4_quantize_rows(Wd)
    torch.cuda.synchronize()
    del Wd
    ref = oracle.quantize(W)
    del W
    return dev, ref


def test_sweep_weight_quantized_bit_exact_every_row(sweep_nvfp4):
    dev, ref = sweep_nvfp4
    assert_bytes_equal(dev, ref, "W[262144,8192]")


@pytest.mark.parametrize("M", [1, 4, 16, 64, 256])
def test_sweep_on_device_quantized_weight(sweep_nvfp4, M):
    """fp32 logits, every token x every one of the 262144 rows."""
    dev, ref_q = sweep_nvfp4
    x = synth.sweep_x(1024)[:M]
    got = product(x, dev).double().cpu().numpy()
    ref = oracle.logits(x, *ref_q)
    assert_logits_close(got, ref, f"sweep M={M}")
    assert_argmax_agrees(got, ref)


def test_sweep_m1024_on_device_quantized_weight(sweep_nvfp4):
    """M = 1024: 64 tokens (the first and last 4 of each 128-token tile) x
    every row, and every token x 512 rows (first, last, seeded)."""
    dev, ref_q = sweep_nvfp4
    x = synth.sweep_x(1024)
    got = product(x, dev)
    rows = tile_edge_tokens(1024, each=4)
    sel = got[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    ref = oracle.logits(x[rows], *ref_q)
    assert_logits_close(sel, ref, "sweep M=1024 rows")
    assert_argmax_agrees(sel, ref)
    cols = np.unique(np.concatenate([[0, 262143],
                                     np.random.default_rng(6).integers(0, 262144, 510)]))
    got_c = got[:, torch.from_numpy(cols).cuda()].double().cpu().numpy()
    ref_c = oracle.logits(x, *ref_q, cols=cols)
    tol = 2e-3 * np.abs(ref_c).max(axis=1, keepdims=True) + 1e-3
    assert np.all(np.abs(got_c - ref_c) <= tol), "sweep M=1024 columns"
