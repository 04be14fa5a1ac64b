"""The C-ABI library builds, loads and exports every symbol its header declares,
and rejects bad arguments on the host before touching the GPU (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "nvfp4_lm_head.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    import nvfp4_weight_only_rows_gb300 as nv

    return nv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z0-9_]+)\s*\(", text)) - {"defined"})


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("nvfp4_quantize_rows", "nvfp4_refresh", "w4a16_lm_head",
              "nvfp4_quantize_workspace_bytes", "w4a16_lm_head_workspace_bytes",
              "nvfp4_status_string", "nvfp4_read_device_status", "nvfp4_abi_version",
              "w4a16_lm_head_argmax", "w4a16_lm_head_argmax_workspace_bytes",
              "fp8_quantize_rows", "fp8_refresh", "w8a8_lm_head", "w8a8_lm_head_argmax",
              "nvfp4_swizzle_scales", "w4a4_lm_head", "w4a4_lm_head_argmax",
              "w4a16_grouped_gemm", "w4a16_grouped_workspace_bytes", "w4a16_lm_head_topk",
              "w4a16_lm_head_topk_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    path = lib._name
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r" T (\S+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        getattr(lib, n)


def test_status_strings_and_version(lib):
    assert lib.nvfp4_abi_version() == 100
    for code in range(11):
        assert lib.nvfp4_status_string(code)
    assert lib.nvfp4_status_string(7) == b"weight holds Inf or NaN"


def test_workspace_sizes(lib):
    assert lib.nvfp4_quantize_workspace_bytes(10, 24) == 0      # K % 16 != 0
    assert lib.nvfp4_quantize_workspace_bytes(0, 32) == 0
    assert lib.nvfp4_quantize_workspace_bytes(10, 32) >= 256
    assert lib.w4a16_lm_head_workspace_bytes(4, 512, 300) == 0   # K % 16 != 0
    assert lib.w4a16_lm_head_workspace_bytes(4, 512, 272) > 0    # any K % 16 (staged rows)
    w = lib.w4a16_lm_head_workspace_bytes(64, 128256, 4096)
    assert w >= 64 * 4096 * 2 + 64 * 4 + 256


def test_host_argument_errors_before_any_cuda_call(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)  # never dereferenced: every case fails a host check first
    q = lib.nvfp4_quantize_rows
    assert q(fake, 4, 24, fake, fake, fake, fake, 1 << 20, None) == 1        # SHAPE
    assert q(fake, 0, 32, fake, fake, fake, fake, 1 << 20, None) == 1        # SHAPE
    assert q(None, 4, 32, fake, fake, fake, fake, 1 << 20, None) == 3        # NULL
    assert q(fake, 4, 32, fake, fake, fake, fake, 16, None) == 4             # WORKSPACE
    assert q(vp((1 << 20) + 8), 4, 32, fake, fake, fake, fake, 1 << 20, None) == 2  # ALIGN
    g = lib.w4a16_lm_head
    assert g(fake, 4, 300, fake, fake, fake, 8, fake, 0, fake, 1 << 30, None) == 1   # K % 16
    assert g(fake, -1, 256, fake, fake, fake, 8, fake, 0, fake, 1 << 30, None) == 1  # M < 0
    assert g(fake, 4, 256, fake, fake, fake, 8, fake, 7, fake, 1 << 30, None) == 5   # DTYPE
    assert g(fake, 0, 256, fake, fake, fake, 8, fake, 0, None, 0, None) == 0         # empty
    assert g(fake, 4, 256, fake, fake, fake, 0, fake, 0, None, 0, None) == 0         # empty
    assert g(None, 4, 256, fake, fake, fake, 8, fake, 0, fake, 1 << 30, None) == 3   # NULL
    assert g(fake, 4, 256, fake, fake, fake, 8, fake, 0, fake, 64, None) == 4        # WORKSPACE
    assert g(vp((1 << 20) + 2), 4, 256, fake, fake, fake, 8, fake, 0, fake, 1 << 30,
             None) == 2                                                              # ALIGN
    a = lib.w4a16_lm_head_argmax
    ids, vals = vp(1 << 20), vp(1 << 21)
    assert a(fake, 4, 256, fake, fake, fake, 0, ids, vals, fake, 1 << 30, None) == 1   # N == 0
    assert a(fake, 4, 300, fake, fake, fake, 8, ids, vals, fake, 1 << 30, None) == 1   # K % 16
    assert a(fake, 0, 256, fake, fake, fake, 8, ids, vals, None, 0, None) == 0         # empty
    assert a(fake, 4, 256, fake, fake, fake, 8, None, vals, fake, 1 << 30, None) == 3  # NULL ids
    assert a(fake, 4, 256, fake, fake, fake, 8, ids, vals, fake, 64, None) == 4        # WORKSPACE
    assert a(fake, 4, 256, fake, fake, fake, 8, vp((1 << 20) + 4), vals, fake, 1 << 30,
             None) == 2                                                              # ALIGN ids
    assert a(fake, 4, 256, fake, fake, fake, 8, ids, vp((1 << 21) + 2), fake, 1 << 30,
             None) == 2                                                              # ALIGN vals


def test_fp8_host_argument_errors(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    qz = lib.fp8_quantize_rows
    assert qz(fake, 4, 24, fake, fake, fake, 1 << 20, None) == 1          # K % 16
    assert qz(fake, 4, 65536 + 16, fake, fake, fake, 1 << 20, None) == 1  # K too large
    assert qz(fake, 0, 32, fake, fake, fake, 1 << 20, None) == 1          # N == 0
    assert qz(None, 4, 32, fake, fake, fake, 1 << 20, None) == 3          # NULL
    assert qz(fake, 4, 32, fake, fake, fake, 16, None) == 4               # WORKSPACE
    assert qz(fake, 4, 32, vp((1 << 20) + 4), fake, fake, 1 << 20, None) == 2  # ALIGN q
    g = lib.w8a8_lm_head
    assert g(fake, 4, 300, fake, fake, 8, fake, 0, fake, 1 << 30, None) == 1    # K % 16
    assert g(fake, 4, 16640, fake, fake, 8, fake, 0, fake, 1 << 30, None) == 1  # K > 16384
    assert g(fake, 4, 256, fake, fake, 8, fake, 9, fake, 1 << 30, None) == 5    # DTYPE
    assert g(fake, 0, 256, fake, fake, 8, fake, 0, None, 0, None) == 0          # empty
    assert g(fake, 4, 256, None, fake, 8, fake, 0, fake, 1 << 30, None) == 3    # NULL
    assert g(fake, 4, 256, fake, fake, 8, fake, 0, fake, 64, None) == 4         # WORKSPACE
    a = lib.w8a8_lm_head_argmax
    assert a(fake, 4, 256, fake, fake, 0, fake, fake, fake, 1 << 30, None) == 1  # N == 0
    assert a(fake, 4, 256, fake, fake, 8, None, fake, fake, 1 << 30, None) == 3  # NULL ids
    assert lib.fp8_quantize_workspace_bytes(4, 32) == 256
    assert lib.w8a8_lm_head_workspace_bytes(4, 8, 300) == 0
    assert lib.w8a8_lm_head_argmax_workspace_bytes(4, 0, 256) == 0


def test_w4a4_host_argument_errors(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    sw = lib.nvfp4_swizzle_scales
    assert sw(fake, 4, 40, fake, None) == 1                      # K % 16
    assert sw(None, 4, 64, fake, None) == 3                      # NULL
    assert sw(fake, 4, 64, vp((1 << 20) + 4), None) == 2         # ALIGN out
    assert lib.nvfp4_swizzled_scales_bytes(130, 128) == 256 * 8
    assert lib.nvfp4_swizzled_scales_bytes(130, 48) == 256 * 4   # 3 scale columns padded to 4
    g = lib.w4a4_lm_head
    assert g(fake, 4, 300, fake, fake, fake, fake, 8, fake, 0, fake, 1 << 30, None) == 1  # K
    assert g(fake, 4, 256, fake, fake, fake, fake, 8, fake, 3, fake, 1 << 30, None) == 5  # DTYPE
    assert g(fake, 0, 256, fake, fake, fake, fake, 8, fake, 0, None, 0, None) == 0       # empty
    assert g(fake, 4, 256, fake, fake, fake, None, 8, fake, 0, fake, 1 << 30, None) == 3  # NULL gx
    assert g(fake, 4, 256, fake, fake, fake, fake, 8, fake, 0, fake, 64, None) == 4     # WORKSPACE
    a = lib.w4a4_lm_head_argmax
    assert a(fake, 4, 256, fake, fake, fake, fake, 0, fake, fake, fake, 1 << 30, None) == 1  # N 0
    assert lib.w4a4_lm_head_argmax_workspace_bytes(4, 0, 256) == 0


def test_grouped_host_argument_errors(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    g = lib.w4a16_grouped_gemm
    assert g(fake, 8, 256, fake, 0, fake, fake, fake, 64, fake, 0, fake, 1 << 30, None) == 1    # E 0
    assert g(fake, 8, 256, fake, 257, fake, fake, fake, 64, fake, 0, fake, 1 << 30, None) == 1  # E
    assert g(fake, 8, 300, fake, 4, fake, fake, fake, 64, fake, 0, fake, 1 << 30, None) == 1    # K
    assert g(fake, 0, 256, fake, 4, fake, fake, fake, 64, fake, 0, None, 0, None) == 0          # empty
    assert g(fake, 8, 256, None, 4, fake, fake, fake, 64, fake, 0, fake, 1 << 30, None) == 3    # NULL
    assert g(fake, 8, 256, fake, 4, fake, fake, fake, 64, fake, 0, fake, 64, None) == 4         # WS
    assert g(fake, 8, 256, fake, 4, fake, fake, fake, 64, fake, 5, fake, 1 << 30, None) == 5    # DTYPE
    assert lib.w4a16_grouped_workspace_bytes(8, 64, 256, 4) > 8 * 256 * 2


def test_argmax_workspace_sizes(lib):
    assert lib.w4a16_lm_head_argmax_workspace_bytes(4, 0, 256) == 0
    for M in (1, 64, 200, 2048):
        plain = lib.w4a16_lm_head_workspace_bytes(M, 128256, 4096)
        am = lib.w4a16_lm_head_argmax_workspace_bytes(M, 128256, 4096)
        assert am >= plain + 128 * M


def test_topk_host_argument_errors_and_sizes(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    ids, vals = vp(1 << 20), vp(1 << 21)
    big = 1 << 44
    t = lib.w4a16_lm_head_topk
    assert t(fake, 4, 256, fake, fake, fake, 100, 0, ids, vals, fake, big, None) == 1     # k == 0
    assert t(fake, 4, 256, fake, fake, fake, 1000, 129, ids, vals, fake, big, None) == 1  # k > max
    assert t(fake, 4, 256, fake, fake, fake, 7, 8, ids, vals, fake, big, None) == 1       # k > N
    assert t(fake, 4, 300, fake, fake, fake, 100, 5, ids, vals, fake, big, None) == 1     # K % 16
    assert t(fake, 1 << 20, 256, fake, fake, fake, 1 << 17, 5, ids, vals, fake, big,
             None) == 1                                                                   # M*N > 2^36
    assert t(fake, 0, 256, fake, fake, fake, 100, 5, ids, vals, None, 0, None) == 0      # empty
    assert t(fake, 4, 256, fake, fake, fake, 100, 5, None, vals, fake, big, None) == 3   # NULL ids
    assert t(fake, 4, 256, fake, fake, fake, 100, 5, ids, vals, fake, 4096, None) == 4   # WORKSPACE
    assert t(fake, 4, 256, fake, fake, fake, 100, 5, vp((1 << 20) + 4), vals, fake, big,
             None) == 2                                                                   # ALIGN ids
    sz = lib.w4a16_lm_head_topk_workspace_bytes
    assert sz(4, 0, 256, 1) == 0 and sz(4, 100, 256, 0) == 0 and sz(4, 100, 256, 129) == 0
    for M in (1, 32, 64, 256, 257, 2048):
        am = lib.w4a16_lm_head_argmax_workspace_bytes(M, 128256, 4096)
        tk = sz(M, 128256, 4096, 50)
        if M <= 256:  # fp32 logits and the u32 maximum of every 32 rows
            plain = lib.w4a16_lm_head_workspace_bytes(M, 128256, 4096)
            assert tk >= plain + M * 128256 * 4 + M * (128256 // 32) * 4
        else:        # candidate slots, group words and histograms of the epilogue route
            assert tk >= am + M * 128256 * 4 + M * (128256 // 32) * 8 + M * 4112


def test_w8a8_w4a4_topk_host_errors_and_sizes(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    ids, vals = vp(1 << 20), vp(1 << 21)
    big = 1 << 44
    t8 = lib.w8a8_lm_head_topk
    assert t8(fake, 4, 256, fake, fake, 100, 0, ids, vals, fake, big, None) == 1      # k == 0
    assert t8(fake, 4, 256, fake, fake, 7, 8, ids, vals, fake, big, None) == 1        # k > N
    assert t8(fake, 4, 32768, fake, fake, 100, 5, ids, vals, fake, big, None) == 1    # K > max
    assert t8(fake, 0, 256, fake, fake, 100, 5, ids, vals, None, 0, None) == 0       # empty
    assert t8(fake, 4, 256, fake, fake, 100, 5, None, vals, fake, big, None) == 3    # NULL ids
    assert t8(fake, 4, 256, fake, fake, 100, 5, ids, vals, fake, 4096, None) == 4    # WORKSPACE
    t4 = lib.w4a4_lm_head_topk
    assert t4(fake, 4, 256, fake, fake, fake, fake, 100, 129, ids, vals, fake, big, None) == 1
    assert t4(fake, 0, 256, fake, fake, fake, fake, 100, 5, ids, vals, None, 0, None) == 0
    assert t4(fake, 4, 256, fake, fake, fake, fake, 100, 5, None, vals, fake, big, None) == 3
    assert t4(fake, 4, 256, fake, fake, fake, fake, 100, 5, ids, vals, fake, 4096, None) == 4
    for f, am in ((lib.w8a8_lm_head_topk_workspace_bytes, lib.w8a8_lm_head_argmax_workspace_bytes),
                  (lib.w4a4_lm_head_topk_workspace_bytes, lib.w4a4_lm_head_argmax_workspace_bytes)):
        assert f(4, 0, 256, 1) == 0 and f(4, 100, 256, 0) == 0
        assert f(64, 128256, 4096, 50) >= am(64, 128256, 4096) + 64 * 128256 * 4


def test_topk_histogram_bins_never_exceed_their_keys(lib):
    """Host check over every 32-bit order key: the threshold a raise can set
    (a bin's lower edge) is never above a key of that bin, bins never
    decrease with the key, and each edge lies in its own bin."""
    assert lib.nvfp4_selftest_topk_bins() == -1


def test_schedule_split_covers_every_stage_once(lib):
    """Host check of the persistent GEMM's work split: waves plus tail cover
    every stage once, tail ranges are contiguous and at least a unit long
    (skewed or not), no unit is cut twice, an unskewed tail splits evenly."""
    assert lib.nvfp4_selftest_schedule() == -1
