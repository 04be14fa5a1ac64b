"""CPU oracle of the online NVFP4 lm_head path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it,
and it shares no code with the CUDA sources: the arithmetic lives in
``nvfp4_oracle.c`` (plain C, built with ``-ffp-contract=off``), and this file
only marshals numpy arrays into it.

What each function follows is stated in ``nvfp4_oracle.c``.  In short:

* ``quantize``     -- ``_quantize_nvfp4`` on the page
  *vllm.model_executor.layers.quantization.online.lm_head*: fp32 global
  scale amax/(6*448) clamped at 1e-12, per-16 E4M3 block scales, E2M1 codes
  with the sign in bit 3, two codes per byte, low nibble first.
* ``dequant_rows`` / ``logits`` -- the W4A16 product of
  ``CompressedTensorsW4A16Fp4`` (page *...compressed_tensors.schemes*):
  logits = x . (e2m1 * f32(scale) * global)^T, here in float64.
* ``fp8_quantize`` / ``fp8_logits`` -- the "fp8" copy of
  ``quantized_lm_head_copy`` (same lm_head page): per-row E4M3 weights with an
  fp32 scale amax/448, per-token E4M3 activations likewise, and the W8A8
  product xs * ws * (q_x . q_w) in float64.
* ``topk`` -- the k largest logits of each token (the sampler's top-k filter
  applied to the lm_head output; the pages define the logits, this selection
  is the plain definition: descending value, of equal values the smaller row).

Parity: every function is pinned in ``tests/test_oracle_*.py`` against what
the pages fix (the code table, the packing order, K % 16), closed forms,
brute-force nearest rounding, torch's own float8_e4m3fn cast and numpy's
matmul.  The one reading the pages cannot pin -- the multiply order inside
the unprinted per-16 block quantizer -- is stated as a reading, not pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, no FMA contraction, OpenMP if available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-std=gnu11", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(cmd[:6] + ["-fopenmp"] + cmd[6:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(cmd, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        f = ctypes.c_float
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = f
        lib.oracle_e4m3_encode.argtypes = [f]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e2m1_round.argtypes = [f]
        lib.oracle_e2m1_round.restype = f
        lib.oracle_e2m1_code.argtypes = [f]
        lib.oracle_e2m1_code.restype = ctypes.c_uint8
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_decode.restype = f
        lib.oracle_weight_amax.argtypes = [p, i64, p]
        lib.oracle_weight_amax.restype = ctypes.c_int
        lib.oracle_global_scale.argtypes = [f, p, p]
        lib.oracle_quantize_block.argtypes = [p, f, f, p, p]
        lib.oracle_quantize_rows.argtypes = [p, i64, i64, p, i64, f, f, p, p]
        lib.oracle_quantize.argtypes = [p, i64, i64, p, p, p]
        lib.oracle_quantize.restype = ctypes.c_int
        lib.oracle_dequant_rows.argtypes = [p, p, f, i64, p, i64, p]
        lib.oracle_logits_cols.argtypes = [p, i64, i64, p, p, f, p, i64, p]
        lib.oracle_e4m3_encode_array.argtypes = [p, i64, p]
        lib.oracle_w4a4_logits_cols.argtypes = [p, i64, i64, f, p, p, f, p, i64, p]
        lib.oracle_swizzle_scales.argtypes = [p, i64, i64, p]
        lib.oracle_fp8_quantize_rows.argtypes = [p, i64, i64, p, p]
        lib.oracle_fp8_quantize_rows.restype = ctypes.c_int
        lib.oracle_fp8_logits_cols.argtypes = [p, p, i64, i64, p, p, p, i64, p]
        lib.oracle_e2m1_round_array.argtypes = [p, i64, p]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"], "oracle needs contiguous arrays"
    return ctypes.c_void_p(a.ctypes.data)


class OracleError(ValueError):
    pass


# ------------------------------------------------------------------ scalars
def e4m3_decode(byte: int) -> float:
    return float(_load().oracle_e4m3_decode(byte))


def e4m3_encode(t: float) -> int:
    return int(_load().oracle_e4m3_encode(t))


def e2m1_round(q: float) -> float:
    return float(_load().oracle_e2m1_round(q))


def e2m1_code(v: float) -> int:
    return int(_load().oracle_e2m1_code(v))


def e2m1_decode(code: int) -> float:
    return float(_load().oracle_e2m1_decode(code))


def e4m3_encode_array(t: np.ndarray) -> np.ndarray:
    """Element-wise e4m3 encode (a loop over the scalar C routine)."""
    t = np.ascontiguousarray(t, dtype=np.float32).ravel()
    out = np.zeros(t.size, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(t), t.size, _ptr(out))
    return out


def e2m1_round_array(q: np.ndarray) -> np.ndarray:
    """Element-wise E2M1 grid rounding (a loop over the scalar C routine)."""
    q = np.ascontiguousarray(q, dtype=np.float32).ravel()
    out = np.zeros(q.size, dtype=np.float32)
    _load().oracle_e2m1_round_array(_ptr(q), q.size, _ptr(out))
    return out


# ------------------------------------------------------------- global scale
def weight_amax(W: np.ndarray) -> float:
    W = np.ascontiguousarray(W, dtype=np.uint16)
    out = np.zeros(1, dtype=np.float32)
    rc = _load().oracle_weight_amax(_ptr(W), W.size, _ptr(out))
    if rc != 0:
        raise OracleError("non-finite weight")
    return float(out[0])


def global_scale(amax: float) -> tuple[np.float32, np.float32]:
    g = np.zeros(1, dtype=np.float32)
    ig = np.zeros(1, dtype=np.float32)
    _load().oracle_global_scale(amax, _ptr(g), _ptr(ig))
    return g[0], ig[0]


# ------------------------------------------------------------ quantization
def quantize_block(x16: np.ndarray, g: float, ig: float) -> tuple[np.ndarray, int]:
    """One 16-value block: (grid values as float32[16], e4m3 scale byte)."""
    x = np.ascontiguousarray(x16, dtype=np.float32)
    assert x.shape == (16,)
    v = np.zeros(16, dtype=np.float32)
    s = np.zeros(1, dtype=np.uint8)
    _load().oracle_quantize_block(_ptr(x), g, ig, _ptr(v), _ptr(s))
    return v, int(s[0])


def quantize(W: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.float32]:
    """`_quantize_nvfp4`: (packed u8[N,K/2], scales u8(e4m3)[N,K/16], global f32)."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    N, K = W.shape
    packed = np.zeros((N, K // 2), dtype=np.uint8)
    scales = np.zeros((N, max(K // 16, 0)), dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    rc = _load().oracle_quantize(_ptr(W), N, K, _ptr(packed), _ptr(scales), _ptr(g))
    if rc == -1:
        raise OracleError("non-finite weight")
    if rc == -2:
        raise OracleError("shape rejected (K % 16 != 0 or empty)")
    return packed, scales, g[0]


def quantize_rows(W: np.ndarray, rows, g: float, ig: float) -> tuple[np.ndarray, np.ndarray]:
    """Quantize only the listed rows of W with a given global scale."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    N, K = W.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    packed = np.zeros((rows.size, K // 2), dtype=np.uint8)
    scales = np.zeros((rows.size, K // 16), dtype=np.uint8)
    _load().oracle_quantize_rows(_ptr(W), N, K, _ptr(rows), rows.size, g, ig, _ptr(packed),
                                 _ptr(scales))
    return packed, scales


def dequant_rows(packed: np.ndarray, scales: np.ndarray, g: float, rows=None) -> np.ndarray:
    """w = e2m1(code) * f32(scale) * global, float64 [len(rows), K]."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    N, K = packed.shape[0], packed.shape[1] * 2
    rows = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    out = np.zeros((rows.size, K), dtype=np.float64)
    _load().oracle_dequant_rows(_ptr(packed), _ptr(scales), g, K, _ptr(rows), rows.size,
                                _ptr(out))
    return out


def logits(x: np.ndarray, packed: np.ndarray, scales: np.ndarray, g: float,
           cols=None) -> np.ndarray:
    """float64 logits[M, len(cols)] = x . dequant(W[cols])^T (all rows if cols is None)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    M, K = x.shape
    N = packed.shape[0]
    assert packed.shape[1] * 2 == K
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, np.int64)
    out = np.zeros((M, cols.size), dtype=np.float64)
    _load().oracle_logits_cols(_ptr(x), M, K, _ptr(packed), _ptr(scales), g, _ptr(cols),
                               cols.size, _ptr(out))
    return out


def w4a4_logits(x: np.ndarray, gx: float, packed: np.ndarray, scales: np.ndarray, gw: float,
                cols=None) -> np.ndarray:
    """float64 logits[M, len(cols)] of the W4A4 product: x quantized to NVFP4 with
    the input global gx (dequant multiplier), times the dequantized weight rows."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    M, K = x.shape
    N = packed.shape[0]
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, np.int64)
    out = np.zeros((M, cols.size), dtype=np.float64)
    _load().oracle_w4a4_logits_cols(_ptr(x), M, K, float(gx), _ptr(packed), _ptr(scales),
                                    float(gw), _ptr(cols), cols.size, _ptr(out))
    return out


def grouped_logits(x: np.ndarray, offsets, packed: list, scales: list, globals_: list) -> np.ndarray:
    """The grouped (MoE) W4A16 product: rows offsets[e]..offsets[e+1] of x times
    expert e's dequantized weight, float64 [M, N] -- the plain product per group."""
    M = x.shape[0]
    N = packed[0].shape[0]
    out = np.zeros((M, N), dtype=np.float64)
    for e in range(len(packed)):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            out[a:b] = logits(x[a:b], packed[e], scales[e], globals_[e])
    return out


def swizzle_scales(scales: np.ndarray) -> np.ndarray:
    """`swizzle_blockscale` of an [N, C] scale matrix: flat bytes, rows padded to 128,
    columns to 4, in [N'/128][C'/4][32][4][4] order."""
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    N, C = scales.shape
    Np, Cp = (N + 127) // 128 * 128, (C + 3) // 4 * 4
    out = np.zeros(Np * Cp, dtype=np.uint8)
    _load().oracle_swizzle_scales(_ptr(scales), N, C, _ptr(out))
    return out


def fp8_quantize(W: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Per-row fp8 copy of bf16 rows (lm_head weights, or activation tokens):
    (q u8(e4m3)[N,K], scale f32[N]); dequant = e4m3(q) * scale[row]."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    N, K = W.shape
    q = np.zeros((N, K), dtype=np.uint8)
    s = np.zeros(N, dtype=np.float32)
    if _load().oracle_fp8_quantize_rows(_ptr(W), N, K, _ptr(q), _ptr(s)) != 0:
        raise OracleError("non-finite value")
    return q, s


def fp8_logits(xq: np.ndarray, xs: np.ndarray, wq: np.ndarray, ws: np.ndarray,
               cols=None) -> np.ndarray:
    """float64 logits[M, len(cols)] = xs * ws * (e4m3(xq) . e4m3(wq[cols])^T)."""
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    xs = np.ascontiguousarray(xs, dtype=np.float32)
    ws = np.ascontiguousarray(ws, dtype=np.float32)
    M, K = xq.shape
    N = wq.shape[0]
    assert wq.shape[1] == K
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, np.int64)
    out = np.zeros((M, cols.size), dtype=np.float64)
    _load().oracle_fp8_logits_cols(_ptr(xq), _ptr(xs), M, K, _ptr(wq), _ptr(ws), _ptr(cols),
                                   cols.size, _ptr(out))
    return out


def topk(L: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Rows and values of the k largest entries of each row of L ([M, N]
    float64, no NaN), largest first, of equal values the smaller index first:
    a stable sort of the negated values."""
    order = np.argsort(-L, axis=1, kind="stable")[:, :k]
    return order, np.take_along_axis(L, order, axis=1)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's loops use from now on (n <= 0: one per processor)."""
    _load().oracle_set_num_threads(int(n))
