"""Online NVFP4 lm_head for GB300 (sm_103a): a thin ctypes binding.

Every step of the path runs in the CUDA kernels of ``libnvfp4_lm_head.so``
(see ``include/nvfp4_lm_head.h``); this module only checks tensor metadata,
allocates outputs and workspaces with PyTorch when the caller gives none,
and passes device pointers plus the current CUDA stream through the C ABI.
There is no CPU or PyTorch fallback: if the library is missing, every call
raises.

Entry points (same names as the C ABI):

* ``nvfp4_quantize_rows(W)`` -> ``(packed u8[N,K/2], scales e4m3[N,K/16], global f32[1])``
  -- ``_quantize_nvfp4`` of the page
  "vllm.model_executor.layers.quantization.online.lm_head".
* ``nvfp4_refresh(W, packed, scales, global_scale)`` -- in-place re-derivation
  (``refresh_quantized_lm_heads``); the buffers keep their addresses.
* ``w4a16_lm_head(x, packed, scales, global_scale)`` -> ``logits[M, N]`` -- the
  weight-only W4A16 product (``_LMHeadNvfp4Method.apply``).
* ``w4a16_lm_head_argmax(x, packed, scales, global_scale)`` ->
  ``(token_ids i64[M], max_logits f32[M])`` -- the same product reduced to each
  token's largest logit inside the kernel (greedy choice; logits never stored).
* ``w4a16_lm_head_topk(x, packed, scales, global_scale, k)`` ->
  ``(token_ids i64[M, k], values f32[M, k])`` -- each token's k largest logits,
  in descending order, selected without storing the logits.
* ``fp8_quantize_rows(W)`` -> ``(q e4m3[N,K], row_scale f32[N])`` and
  ``fp8_refresh`` -- the "fp8" copy of ``quantized_lm_head_copy`` (per-row
  scales); ``w8a8_lm_head(x, q, row_scale)`` / ``w8a8_lm_head_argmax`` /
  ``w8a8_lm_head_topk`` -- its
  product with per-token fp8 activations on the fp8 tensor cores.
* ``nvfp4_swizzle_scales(scales)`` and ``w4a4_lm_head(x, packed, scales_swizzled,
  global_scale, input_global_scale)`` / ``w4a4_lm_head_argmax`` / ``w4a4_lm_head_topk`` -- the
  W4A4 NVFP4
  product (``CompressedTensorsW4A4Fp4``): x quantized to NVFP4 in the call,
  block-scaled FP4 tensor cores, logits scaled by alpha = g_x * g_w.
* ``w4a16_grouped_gemm(x, group_offsets, packed, scales, global_scales)`` -- the
  NVFP4 W4A16 product of all experts of a MoE layer in one call, tokens grouped
  by expert (``ModelOptNvFp4FusedMoE`` weight layouts).
"""
from __future__ import annotations

import ctypes
import enum
import os

import torch

__all__ = [
    "NVFP4Error", "Status", "library_path", "load_library", "nvfp4_quantize_rows",
    "nvfp4_refresh", "w4a16_lm_head", "nvfp4_quantize_workspace_bytes",
    "w4a16_lm_head_workspace_bytes", "nvfp4_read_device_status", "w4a16_lm_head_noalloc",
    "w4a16_lm_head_noalloc_status",
    "nvfp4_selftest_bounded_wait", "nvfp4_selftest_topk_bins", "nvfp4_selftest_schedule",
    "OUT_F32", "OUT_BF16", "w4a16_lm_head_argmax",
    "w4a16_lm_head_argmax_workspace_bytes", "fp8_quantize_rows", "fp8_refresh",
    "fp8_quantize_workspace_bytes", "w8a8_lm_head", "w8a8_lm_head_argmax",
    "w8a8_lm_head_workspace_bytes", "w8a8_lm_head_argmax_workspace_bytes",
    "nvfp4_swizzle_scales", "nvfp4_swizzled_scales_bytes", "w4a4_lm_head",
    "w4a4_lm_head_argmax", "w4a4_lm_head_workspace_bytes", "w4a4_lm_head_argmax_workspace_bytes",
    "w4a16_grouped_gemm", "w4a16_grouped_workspace_bytes", "w4a16_lm_head_topk",
    "w4a16_lm_head_topk_workspace_bytes", "TOPK_MAX", "w8a8_lm_head_topk",
    "w8a8_lm_head_topk_workspace_bytes", "w4a4_lm_head_topk", "w4a4_lm_head_topk_workspace_bytes",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libnvfp4_lm_head.so")
_lib = None

OUT_F32 = 0
OUT_BF16 = 1
TOPK_MAX = 128  # NVFP4_TOPK_MAX: largest k of the fused top-k


class Status(enum.IntEnum):
    OK = 0
    ERR_SHAPE = 1
    ERR_ALIGN = 2
    ERR_NULL = 3
    ERR_WORKSPACE = 4
    ERR_DTYPE = 5
    ERR_CUDA = 6
    ERR_NONFINITE = 7
    ERR_TIMEOUT = 8
    ERR_UNSUPPORTED = 9
    ERR_SCRATCH_LIMIT = 10


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status)
        msg = load_library().nvfp4_status_string(int(status)).decode()
        super().__init__(f"{where}: {self.status.name} ({msg})")


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    st = ctypes.c_int
    lib.nvfp4_status_string.argtypes = [st]
    lib.nvfp4_status_string.restype = ctypes.c_char_p
    lib.nvfp4_abi_version.restype = ctypes.c_int
    lib.nvfp4_quantize_workspace_bytes.argtypes = [i64, i64]
    lib.nvfp4_quantize_workspace_bytes.restype = sz
    for name in ("nvfp4_quantize_rows", "nvfp4_refresh"):
        f = getattr(lib, name)
        f.argtypes = [vp, i64, i64, vp, vp, vp, vp, sz, vp]
        f.restype = st
    lib.nvfp4_read_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
    lib.nvfp4_read_device_status.restype = st
    lib.w4a16_lm_head_workspace_bytes.argtypes = [i64, i64, i64]
    lib.w4a16_lm_head_workspace_bytes.restype = sz
    lib.w4a16_lm_head.argtypes = [vp, i64, i64, vp, vp, vp, i64, vp, ctypes.c_int, vp, sz, vp]
    lib.w4a16_lm_head.restype = st
    lib.w4a16_lm_head_argmax_workspace_bytes.argtypes = [i64, i64, i64]
    lib.w4a16_lm_head_argmax_workspace_bytes.restype = sz
    lib.w4a16_lm_head_argmax.argtypes = [vp, i64, i64, vp, vp, vp, i64, vp, vp, vp, sz, vp]
    lib.w4a16_lm_head_argmax.restype = st
    lib.w4a16_lm_head_topk_workspace_bytes.argtypes = [i64, i64, i64, i64]
    lib.w4a16_lm_head_topk_workspace_bytes.restype = sz
    lib.w4a16_lm_head_topk.argtypes = [vp, i64, i64, vp, vp, vp, i64, i64, vp, vp, vp, sz, vp]
    lib.w4a16_lm_head_topk.restype = st
    lib.fp8_quantize_workspace_bytes.argtypes = [i64, i64]
    lib.fp8_quantize_workspace_bytes.restype = sz
    for name in ("fp8_quantize_rows", "fp8_refresh"):
        f = getattr(lib, name)
        f.argtypes = [vp, i64, i64, vp, vp, vp, sz, vp]
        f.restype = st
    for name in ("w8a8_lm_head_workspace_bytes", "w8a8_lm_head_argmax_workspace_bytes"):
        f = getattr(lib, name)
        f.argtypes = [i64, i64, i64]
        f.restype = sz
    lib.w8a8_lm_head.argtypes = [vp, i64, i64, vp, vp, i64, vp, ctypes.c_int, vp, sz, vp]
    lib.w8a8_lm_head.restype = st
    lib.w8a8_lm_head_argmax.argtypes = [vp, i64, i64, vp, vp, i64, vp, vp, vp, sz, vp]
    lib.w8a8_lm_head_argmax.restype = st
    lib.w8a8_lm_head_topk_workspace_bytes.argtypes = [i64, i64, i64, i64]
    lib.w8a8_lm_head_topk_workspace_bytes.restype = sz
    lib.w8a8_lm_head_topk.argtypes = [vp, i64, i64, vp, vp, i64, i64, vp, vp, vp, sz, vp]
    lib.w8a8_lm_head_topk.restype = st
    lib.nvfp4_swizzled_scales_bytes.argtypes = [i64, i64]
    lib.nvfp4_swizzled_scales_bytes.restype = sz
    lib.nvfp4_swizzle_scales.argtypes = [vp, i64, i64, vp, vp]
    lib.nvfp4_swizzle_scales.restype = st
    for name in ("w4a4_lm_head_workspace_bytes", "w4a4_lm_head_argmax_workspace_bytes"):
        f = getattr(lib, name)
        f.argtypes = [i64, i64, i64]
        f.restype = sz
    lib.w4a4_lm_head.argtypes = [vp, i64, i64, vp, vp, vp, vp, i64, vp, ctypes.c_int, vp, sz, vp]
    lib.w4a4_lm_head.restype = st
    lib.w4a4_lm_head_argmax.argtypes = [vp, i64, i64, vp, vp, vp, vp, i64, vp, vp, vp, sz, vp]
    lib.w4a4_lm_head_topk_workspace_bytes.argtypes = [i64, i64, i64, i64]
    lib.w4a4_lm_head_topk_workspace_bytes.restype = sz
    lib.w4a4_lm_head_topk.argtypes = [vp, i64, i64, vp, vp, vp, vp, i64, i64, vp, vp, vp, sz, vp]
    lib.w4a4_lm_head_topk.restype = st
    lib.w4a4_lm_head_argmax.restype = st
    lib.w4a16_grouped_workspace_bytes.argtypes = [i64, i64, i64, i64]
    lib.w4a16_grouped_workspace_bytes.restype = sz
    lib.w4a16_grouped_gemm.argtypes = [vp, i64, i64, vp, i64, vp, vp, vp, i64, vp, ctypes.c_int,
                                       vp, sz, vp]
    lib.w4a16_grouped_gemm.restype = st
    lib.w4a16_lm_head_noalloc.argtypes = [vp, i64, i64, vp, vp, vp, i64, vp, ctypes.c_int, vp]
    lib.w4a16_lm_head_noalloc.restype = st
    lib.w4a16_lm_head_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_int32), vp]
    lib.w4a16_lm_head_noalloc_status.restype = st
    lib.nvfp4_selftest_bounded_wait.argtypes = [vp, sz, i64, vp]
    lib.nvfp4_selftest_bounded_wait.restype = st
    lib.nvfp4_selftest_topk_bins.argtypes = []
    lib.nvfp4_selftest_topk_bins.restype = ctypes.c_int64
    lib.nvfp4_selftest_schedule.argtypes = []
    lib.nvfp4_selftest_schedule.restype = ctypes.c_int64
    _lib = lib
    return lib


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise NVFP4Error(rc, where)


def _need(t: torch.Tensor, dtype, name: str, shape=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _workspace(nbytes: int, device) -> torch.Tensor:
    # 256-byte alignment: torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def nvfp4_quantize_workspace_bytes(N: int, K: int) -> int:
    return int(load_library().nvfp4_quantize_workspace_bytes(N, K))


def w4a16_lm_head_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().w4a16_lm_head_workspace_bytes(M, N, K))


def nvfp4_quantize_rows(W: torch.Tensor, packed: torch.Tensor | None = None,
                        scales: torch.Tensor | None = None,
                        global_scale: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None):
    """Quantize W bf16[N, K] to (packed u8[N, K/2], scales e4m3[N, K/16], global f32[1])."""
    lib = load_library()
    _need(W, torch.bfloat16, "W")
    if W.dim() != 2:
        raise ValueError("W must be 2-D [N, K]")
    N, K = W.shape
    dev = W.device
    if packed is None:
        packed = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(N, K // 16, dtype=torch.float8_e4m3fn, device=dev)
    if global_scale is None:
        global_scale = torch.empty(1, dtype=torch.float32, device=dev)
    _quantize_into(lib.nvfp4_quantize_rows, "nvfp4_quantize_rows", W, packed, scales,
                   global_scale, workspace, stream)
    return packed, scales, global_scale


def nvfp4_refresh(W: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                  global_scale: torch.Tensor, workspace: torch.Tensor | None = None,
                  stream=None) -> None:
    """Re-derive the quantized copy of W into the existing buffers (addresses kept)."""
    lib = load_library()
    _need(W, torch.bfloat16, "W")
    _quantize_into(lib.nvfp4_refresh, "nvfp4_refresh", W, packed, scales, global_scale,
                   workspace, stream)


def _quantize_into(fn, where, W, packed, scales, global_scale, workspace, stream):
    N, K = W.shape
    _need(packed, torch.uint8, "packed", (N, K // 2))
    if scales.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise ValueError("scales must be float8_e4m3fn (or uint8 bit patterns)")
    _need(scales, scales.dtype, "scales", (N, K // 16))
    _need(global_scale, torch.float32, "global_scale")
    need = nvfp4_quantize_workspace_bytes(N, K)
    if workspace is None:
        workspace = _workspace(need, W.device)
    rc = fn(_ptr(W), N, K, _ptr(packed), _ptr(scales), _ptr(global_scale), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, where)


def w4a16_lm_head(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                  global_scale: torch.Tensor, out: torch.Tensor | None = None,
                  out_dtype: torch.dtype = torch.float32,
                  workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """logits[M, N] = x . dequant(W)^T for x bf16[M, K] and the packed NVFP4 weight."""
    lib = load_library()
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    N = packed.shape[0]
    _need(packed, torch.uint8, "packed", (N, K // 2))
    _need(scales, scales.dtype, "scales", (N, K // 16))
    _need(global_scale, torch.float32, "global_scale")
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=x.device)
    _need(out, out.dtype, "out", (M, N))
    code = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16}.get(out.dtype)
    if code is None:
        raise ValueError("out must be float32 or bfloat16")
    need = w4a16_lm_head_workspace_bytes(M, N, K)
    if workspace is None:
        workspace = _workspace(need, x.device)
    rc = lib.w4a16_lm_head(_ptr(x), M, K, _ptr(packed), _ptr(scales), _ptr(global_scale), N,
                           _ptr(out), code, _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "w4a16_lm_head")
    return out


def w4a16_lm_head_argmax_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().w4a16_lm_head_argmax_workspace_bytes(M, N, K))


def w4a16_lm_head_argmax(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                         global_scale: torch.Tensor, token_ids: torch.Tensor | None = None,
                         max_logits: torch.Tensor | None = None, with_values: bool = True,
                         workspace: torch.Tensor | None = None, stream=None):
    """Each token's largest logit and its vocabulary row (smallest row on ties),
    without writing the logits: returns (token_ids i64[M], max_logits f32[M] or None)."""
    lib = load_library()
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    N = packed.shape[0]
    _need(packed, torch.uint8, "packed", (N, K // 2))
    _need(scales, scales.dtype, "scales", (N, K // 16))
    _need(global_scale, torch.float32, "global_scale")
    if token_ids is None:
        token_ids = torch.empty(M, dtype=torch.int64, device=x.device)
    _need(token_ids, torch.int64, "token_ids", (M,))
    if max_logits is None and with_values:
        max_logits = torch.empty(M, dtype=torch.float32, device=x.device)
    if max_logits is not None:
        _need(max_logits, torch.float32, "max_logits", (M,))
    need = w4a16_lm_head_argmax_workspace_bytes(M, N, K)
    if workspace is None:
        workspace = _workspace(need, x.device)
    rc = lib.w4a16_lm_head_argmax(_ptr(x), M, K, _ptr(packed), _ptr(scales), _ptr(global_scale),
                                  N, _ptr(token_ids), _ptr(max_logits), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "w4a16_lm_head_argmax")
    return token_ids, max_logits


def w4a16_lm_head_topk_workspace_bytes(M: int, N: int, K: int, k: int) -> int:
    return int(load_library().w4a16_lm_head_topk_workspace_bytes(M, N, K, k))


def w4a16_lm_head_topk(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                       global_scale: torch.Tensor, k: int, token_ids: torch.Tensor | None = None,
                       values: torch.Tensor | None = None, with_values: bool = True,
                       workspace: torch.Tensor | None = None, stream=None):
    """Each token's k largest logits and their vocabulary rows, largest first
    (smaller row first on ties), without writing the logits: returns
    (token_ids i64[M, k], values f32[M, k] or None)."""
    lib = load_library()
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    N = packed.shape[0]
    _need(packed, torch.uint8, "packed", (N, K // 2))
    _need(scales, scales.dtype, "scales", (N, K // 16))
    _need(global_scale, torch.float32, "global_scale")
    if token_ids is None:
        token_ids = torch.empty((M, max(k, 0)), dtype=torch.int64, device=x.device)
    _need(token_ids, torch.int64, "token_ids", (M, max(k, 0)))
    if values is None and with_values:
        values = torch.empty((M, max(k, 0)), dtype=torch.float32, device=x.device)
    if values is not None:
        _need(values, torch.float32, "values", (M, max(k, 0)))
    if workspace is None:
        workspace = _workspace(w4a16_lm_head_topk_workspace_bytes(M, N, K, k), x.device)
    rc = lib.w4a16_lm_head_topk(_ptr(x), M, K, _ptr(packed), _ptr(scales), _ptr(global_scale),
                                N, k, _ptr(token_ids), _ptr(values), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "w4a16_lm_head_topk")
    return token_ids, values


def _topk_outputs(M: int, k: int, device, token_ids, values, with_values):
    kk = max(int(k), 0)
    if token_ids is None:
        token_ids = torch.empty((M, kk), dtype=torch.int64, device=device)
    _need(token_ids, torch.int64, "token_ids", (M, kk))
    if values is None and with_values:
        values = torch.empty((M, kk), dtype=torch.float32, device=device)
    if values is not None:
        _need(values, torch.float32, "values", (M, kk))
    return token_ids, values


def fp8_quantize_workspace_bytes(N: int, K: int) -> int:
    return int(load_library().fp8_quantize_workspace_bytes(N, K))


def w8a8_lm_head_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().w8a8_lm_head_workspace_bytes(M, N, K))


def w8a8_lm_head_argmax_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().w8a8_lm_head_argmax_workspace_bytes(M, N, K))


def fp8_quantize_rows(W: torch.Tensor, q: torch.Tensor | None = None,
                      row_scale: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None):
    """The fp8 copy of W bf16[N, K]: (q float8_e4m3fn[N, K], row_scale f32[N])."""
    _need(W, torch.bfloat16, "W")
    if W.dim() != 2:
        raise ValueError("W must be 2-D [N, K]")
    N, K = W.shape
    if q is None:
        q = torch.empty(N, K, dtype=torch.float8_e4m3fn, device=W.device)
    if row_scale is None:
        row_scale = torch.empty(N, dtype=torch.float32, device=W.device)
    fp8_refresh(W, q, row_scale, workspace, stream, _where="fp8_quantize_rows")
    return q, row_scale


def fp8_refresh(W: torch.Tensor, q: torch.Tensor, row_scale: torch.Tensor,
                workspace: torch.Tensor | None = None, stream=None, _where="fp8_refresh") -> None:
    """Re-derive the fp8 copy of W into the existing buffers (addresses kept)."""
    lib = load_library()
    _need(W, torch.bfloat16, "W")
    N, K = W.shape
    if q.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise ValueError("q must be float8_e4m3fn (or uint8 bit patterns)")
    _need(q, q.dtype, "q", (N, K))
    _need(row_scale, torch.float32, "row_scale", (N,))
    if workspace is None:
        workspace = _workspace(fp8_quantize_workspace_bytes(N, K), W.device)
    fn = lib.fp8_quantize_rows if _where == "fp8_quantize_rows" else lib.fp8_refresh
    rc = fn(_ptr(W), N, K, _ptr(q), _ptr(row_scale), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, _where)


def _w8a8_args(x, q, row_scale):
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    N = q.shape[0]
    _need(q, q.dtype, "q", (N, K))
    _need(row_scale, torch.float32, "row_scale", (N,))
    return M, K, N


def w8a8_lm_head(x: torch.Tensor, q: torch.Tensor, row_scale: torch.Tensor,
                 out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float32,
                 workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """logits[M, N] of the fp8 copy: x quantized per token to e4m3, fp8 tensor cores."""
    lib = load_library()
    M, K, N = _w8a8_args(x, q, row_scale)
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=x.device)
    _need(out, out.dtype, "out", (M, N))
    code = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16}.get(out.dtype)
    if code is None:
        raise ValueError("out must be float32 or bfloat16")
    if workspace is None:
        workspace = _workspace(w8a8_lm_head_workspace_bytes(M, N, K), x.device)
    rc = lib.w8a8_lm_head(_ptr(x), M, K, _ptr(q), _ptr(row_scale), N, _ptr(out), code,
                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                          _stream(stream))
    _check(rc, "w8a8_lm_head")
    return out


def w8a8_lm_head_argmax(x: torch.Tensor, q: torch.Tensor, row_scale: torch.Tensor,
                        token_ids: torch.Tensor | None = None,
                        max_logits: torch.Tensor | None = None, with_values: bool = True,
                        workspace: torch.Tensor | None = None, stream=None):
    """Greedy argmax of the fp8 copy's logits without storing them:
    (token_ids i64[M], max_logits f32[M] or None)."""
    lib = load_library()
    M, K, N = _w8a8_args(x, q, row_scale)
    if token_ids is None:
        token_ids = torch.empty(M, dtype=torch.int64, device=x.device)
    _need(token_ids, torch.int64, "token_ids", (M,))
    if max_logits is None and with_values:
        max_logits = torch.empty(M, dtype=torch.float32, device=x.device)
    if max_logits is not None:
        _need(max_logits, torch.float32, "max_logits", (M,))
    if workspace is None:
        workspace = _workspace(w8a8_lm_head_argmax_workspace_bytes(M, N, K), x.device)
    rc = lib.w8a8_lm_head_argmax(_ptr(x), M, K, _ptr(q), _ptr(row_scale), N, _ptr(token_ids),
                                 _ptr(max_logits), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "w8a8_lm_head_argmax")
    return token_ids, max_logits


def w8a8_lm_head_topk_workspace_bytes(M: int, N: int, K: int, k: int) -> int:
    return int(load_library().w8a8_lm_head_topk_workspace_bytes(M, N, K, k))


def w8a8_lm_head_topk(x: torch.Tensor, q: torch.Tensor, row_scale: torch.Tensor, k: int,
                      token_ids: torch.Tensor | None = None, values: torch.Tensor | None = None,
                      with_values: bool = True, workspace: torch.Tensor | None = None,
                      stream=None):
    """The k largest logits of the fp8 copy per token, largest first, without
    storing the logits: (token_ids i64[M, k], values f32[M, k] or None)."""
    lib = load_library()
    M, K, N = _w8a8_args(x, q, row_scale)
    token_ids, values = _topk_outputs(M, k, x.device, token_ids, values, with_values)
    if workspace is None:
        workspace = _workspace(w8a8_lm_head_topk_workspace_bytes(M, N, K, k), x.device)
    rc = lib.w8a8_lm_head_topk(_ptr(x), M, K, _ptr(q), _ptr(row_scale), N, k, _ptr(token_ids),
                               _ptr(values), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "w8a8_lm_head_topk")
    return token_ids, values


def nvfp4_swizzled_scales_bytes(N: int, K: int) -> int:
    return int(load_library().nvfp4_swizzled_scales_bytes(N, K))


def w4a4_lm_head_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().w4a4_lm_head_workspace_bytes(M, N, K))


def w4a4_lm_head_argmax_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load_library().w4a4_lm_head_argmax_workspace_bytes(M, N, K))


def nvfp4_swizzle_scales(scales: torch.Tensor, out: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """Row-major E4M3 block scales [N, K/16] -> the 128x4-interleaved copy (u8, flat)."""
    lib = load_library()
    N, C = scales.shape
    K = C * 16
    _need(scales, scales.dtype, "scales")
    nbytes = nvfp4_swizzled_scales_bytes(N, K)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=scales.device)
    if out.numel() * out.element_size() < nbytes:
        raise ValueError(f"out must hold {nbytes} bytes")
    _check(lib.nvfp4_swizzle_scales(_ptr(scales), N, K, _ptr(out), _stream(stream)),
           "nvfp4_swizzle_scales")
    return out


def _w4a4_args(x, packed, scales_swizzled, global_scale, input_global_scale):
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    N = packed.shape[0]
    _need(packed, torch.uint8, "packed", (N, K // 2))
    _need(scales_swizzled, torch.uint8, "scales_swizzled")
    if scales_swizzled.numel() < nvfp4_swizzled_scales_bytes(N, K):
        raise ValueError("scales_swizzled is smaller than nvfp4_swizzled_scales_bytes(N, K)")
    _need(global_scale, torch.float32, "global_scale")
    _need(input_global_scale, torch.float32, "input_global_scale")
    return M, K, N


def w4a4_lm_head(x: torch.Tensor, packed: torch.Tensor, scales_swizzled: torch.Tensor,
                 global_scale: torch.Tensor, input_global_scale: torch.Tensor,
                 out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float32,
                 workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """W4A4 NVFP4 logits[M, N]: x quantized to NVFP4 with input_global_scale."""
    lib = load_library()
    M, K, N = _w4a4_args(x, packed, scales_swizzled, global_scale, input_global_scale)
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=x.device)
    _need(out, out.dtype, "out", (M, N))
    code = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16}.get(out.dtype)
    if code is None:
        raise ValueError("out must be float32 or bfloat16")
    if workspace is None:
        workspace = _workspace(w4a4_lm_head_workspace_bytes(M, N, K), x.device)
    rc = lib.w4a4_lm_head(_ptr(x), M, K, _ptr(packed), _ptr(scales_swizzled), _ptr(global_scale),
                          _ptr(input_global_scale), N, _ptr(out), code, _ptr(workspace),
                          workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "w4a4_lm_head")
    return out


def w4a4_lm_head_argmax(x: torch.Tensor, packed: torch.Tensor, scales_swizzled: torch.Tensor,
                        global_scale: torch.Tensor, input_global_scale: torch.Tensor,
                        token_ids: torch.Tensor | None = None,
                        max_logits: torch.Tensor | None = None, with_values: bool = True,
                        workspace: torch.Tensor | None = None, stream=None):
    """Greedy argmax of the W4A4 logits without storing them."""
    lib = load_library()
    M, K, N = _w4a4_args(x, packed, scales_swizzled, global_scale, input_global_scale)
    if token_ids is None:
        token_ids = torch.empty(M, dtype=torch.int64, device=x.device)
    _need(token_ids, torch.int64, "token_ids", (M,))
    if max_logits is None and with_values:
        max_logits = torch.empty(M, dtype=torch.float32, device=x.device)
    if max_logits is not None:
        _need(max_logits, torch.float32, "max_logits", (M,))
    if workspace is None:
        workspace = _workspace(w4a4_lm_head_argmax_workspace_bytes(M, N, K), x.device)
    rc = lib.w4a4_lm_head_argmax(_ptr(x), M, K, _ptr(packed), _ptr(scales_swizzled),
                                 _ptr(global_scale), _ptr(input_global_scale), N, _ptr(token_ids),
                                 _ptr(max_logits), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "w4a4_lm_head_argmax")
    return token_ids, max_logits


def w4a4_lm_head_topk_workspace_bytes(M: int, N: int, K: int, k: int) -> int:
    return int(load_library().w4a4_lm_head_topk_workspace_bytes(M, N, K, k))


def w4a4_lm_head_topk(x: torch.Tensor, packed: torch.Tensor, scales_swizzled: torch.Tensor,
                      global_scale: torch.Tensor, input_global_scale: torch.Tensor, k: int,
                      token_ids: torch.Tensor | None = None, values: torch.Tensor | None = None,
                      with_values: bool = True, workspace: torch.Tensor | None = None,
                      stream=None):
    """The k largest W4A4 logits per token, largest first, without storing
    the logits: (token_ids i64[M, k], values f32[M, k] or None)."""
    lib = load_library()
    M, K, N = _w4a4_args(x, packed, scales_swizzled, global_scale, input_global_scale)
    token_ids, values = _topk_outputs(M, k, x.device, token_ids, values, with_values)
    if workspace is None:
        workspace = _workspace(w4a4_lm_head_topk_workspace_bytes(M, N, K, k), x.device)
    rc = lib.w4a4_lm_head_topk(_ptr(x), M, K, _ptr(packed), _ptr(scales_swizzled),
                               _ptr(global_scale), _ptr(input_global_scale), N, k,
                               _ptr(token_ids), _ptr(values), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "w4a4_lm_head_topk")
    return token_ids, values


def w4a16_grouped_workspace_bytes(M: int, N: int, K: int, n_groups: int) -> int:
    return int(load_library().w4a16_grouped_workspace_bytes(M, N, K, n_groups))


def w4a16_grouped_gemm(x: torch.Tensor, group_offsets: torch.Tensor, packed: torch.Tensor,
                       scales: torch.Tensor, global_scales: torch.Tensor,
                       out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float32,
                       workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[M, N] = each token row times its expert's NVFP4 weight: x bf16[M, K]
    grouped by expert (group_offsets int32[E + 1]), packed u8[E, N, K/2],
    scales e4m3[E, N, K/16], global_scales f32[E]."""
    lib = load_library()
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    E, N = packed.shape[0], packed.shape[1]
    _need(group_offsets, torch.int32, "group_offsets", (E + 1,))
    _need(packed, torch.uint8, "packed", (E, N, K // 2))
    _need(scales, scales.dtype, "scales", (E, N, K // 16))
    _need(global_scales, torch.float32, "global_scales", (E,))
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype, device=x.device)
    _need(out, out.dtype, "out", (M, N))
    code = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16}.get(out.dtype)
    if code is None:
        raise ValueError("out must be float32 or bfloat16")
    if workspace is None:
        workspace = _workspace(w4a16_grouped_workspace_bytes(M, N, K, E), x.device)
    rc = lib.w4a16_grouped_gemm(_ptr(x), M, K, _ptr(group_offsets), E, _ptr(packed), _ptr(scales),
                                _ptr(global_scales), N, _ptr(out), code, _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "w4a16_grouped_gemm")
    return out


def w4a16_lm_head_noalloc(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                          global_scale: torch.Tensor, out: torch.Tensor, stream=None) -> torch.Tensor:
    """w4a16_lm_head without a workspace: the library's fixed 8 MiB device scratch is
    used instead (for callers that cannot allocate; see the C header).  `out` must be
    given, so this call allocates nothing."""
    lib = load_library()
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    N = packed.shape[0]
    _need(packed, torch.uint8, "packed", (N, K // 2))
    _need(scales, scales.dtype, "scales", (N, K // 16))
    _need(global_scale, torch.float32, "global_scale")
    _need(out, out.dtype, "out", (M, N))
    code = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16}.get(out.dtype)
    if code is None:
        raise ValueError("out must be float32 or bfloat16")
    rc = lib.w4a16_lm_head_noalloc(_ptr(x), M, K, _ptr(packed), _ptr(scales), _ptr(global_scale),
                                   N, _ptr(out), code, _stream(stream))
    _check(rc, "w4a16_lm_head_noalloc")
    return out


def w4a16_lm_head_noalloc_status(stream=None) -> Status:
    """The device status word the last w4a16_lm_head_noalloc call left in the
    fixed scratch of the current context (synchronizes `stream`)."""
    v = ctypes.c_int32(0)
    _check(load_library().w4a16_lm_head_noalloc_status(ctypes.byref(v), _stream(stream)),
           "w4a16_lm_head_noalloc_status")
    return Status(v.value)


def nvfp4_selftest_topk_bins() -> int:
    """Host-only check of the fused top-k's histogram bins against every 32-bit
    order key: -1 when all pass, else the first failing key."""
    return int(load_library().nvfp4_selftest_topk_bins())


def nvfp4_selftest_schedule() -> int:
    """Host-only check of the persistent products' split of their units into
    whole-unit waves and a stream-K tail: -1 when all cases pass, else the
    index of the first failing case."""
    return int(load_library().nvfp4_selftest_schedule())


def nvfp4_selftest_bounded_wait(workspace: torch.Tensor, limit_us: int, stream=None) -> None:
    """Run the device self-test of the bounded pipeline waits (see the C header)."""
    rc = load_library().nvfp4_selftest_bounded_wait(
        _ptr(workspace), workspace.numel() * workspace.element_size(), limit_us, _stream(stream))
    _check(rc, "nvfp4_selftest_bounded_wait")


def nvfp4_read_device_status(workspace: torch.Tensor, stream=None) -> Status:
    """Status word a kernel left in `workspace` (synchronizes the stream)."""
    v = ctypes.c_int32(0)
    rc = load_library().nvfp4_read_device_status(_ptr(workspace), ctypes.byref(v),
                                                 _stream(stream))
    _check(rc, "nvfp4_read_device_status")
    return Status(v.value)
