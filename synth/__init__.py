"""Seeded synthetic inputs for the NVFP4 lm_head workloads.

This module holds no arithmetic of the quantization method: it draws random
numbers (counter-based SplitMix64, Box-Muller normals) and rounds them to
bf16, so that the CPU oracle and the GPU path see the same bytes.  Arrays are
returned as numpy ``uint16`` holding bf16 bit patterns.

Workload recipes (the pages give no data; these stand in for an lm_head of
the stated shape, with random weights):

* ``tiny``    W[512, 256] ~ N(0, 0.02), seed 0, four distinct rows (drawn from
  stream 1 of seed 0) scaled x50; x[4, 256] ~ N(0, 1), seed 100.
* ``decode``  W[128256, 4096] ~ N(0, 0.02), seed 1, each entry scaled x20 with
  probability 0.001 (uniform stream 2); x[M, 4096] RMS-normalised N(0, 1)
  rows, seed 101, M in {1, 8, 32, 64}.
* ``prefill`` same W as ``decode``; x[2048, 4096] RMS-normalised, seed 102.
* ``quant``   W[151936, 5120]: row n is N(0, 0.015) times |t_n|, t_n a
  Student-t (nu = 3) draw per row from stream 3; seed 4 (and seed 5 for the
  second weight that refresh alternates with).
* ``sweep``   W[262144, 8192] ~ N(0, 0.01), seed 6; x[M, 8192] RMS-normalised,
  seed 106, M in {1, 4, 16, 64, 256, 1024}.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into a shared library next to it (gcc, OpenMP if present)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11", _SRC, "-lm"]
    tmp = _LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run(base[:-1] + ["-fopenmp", "-o", tmp, "-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp], check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        u64 = ctypes.c_uint64
        d = ctypes.c_double
        lib.synth_uniform.argtypes = [p, i64, u64, u64]
        lib.synth_normal.argtypes = [p, i64, u64, u64]
        lib.synth_weight.argtypes = [p, i64, i64, u64, d, p, d, d]
        lib.synth_activations.argtypes = [p, i64, i64, u64, ctypes.c_int]
        lib.synth_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def uniform(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_uniform(_ptr(out), n, seed, stream)
    return out


def normal(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_normal(_ptr(out), n, seed, stream)
    return out


def weight(N: int, K: int, seed: int, sigma: float, row_mult: np.ndarray | None = None,
           p: float = 0.0, mult: float = 1.0, out: np.ndarray | None = None) -> np.ndarray:
    """W[N, K] bf16 bits = bf16(sigma * row_mult[n] * z * (u < p ? mult : 1))."""
    if out is None:
        out = np.empty((N, K), dtype=np.uint16)
    assert out.shape == (N, K) and out.dtype == np.uint16
    rm = None
    if row_mult is not None:
        rm = np.ascontiguousarray(row_mult, dtype=np.float64)
        assert rm.shape == (N,)
    _load().synth_weight(_ptr(out), N, K, seed, sigma,
                         _ptr(rm) if rm is not None else None, p, mult)
    return out


def activations(M: int, K: int, seed: int, rms_normalize: bool) -> np.ndarray:
    out = np.empty((M, K), dtype=np.uint16)
    _load().synth_activations(_ptr(out), M, K, seed, int(rms_normalize))
    return out


def distinct_rows(count: int, N: int, seed: int, stream: int) -> np.ndarray:
    """`count` distinct row indices in [0, N), drawn in order without replacement."""
    picked: list[int] = []
    draws = uniform(64 * count + 64, seed, stream)
    for u in draws:
        r = int(u * N)
        if r not in picked:
            picked.append(r)
            if len(picked) == count:
                return np.array(picked, dtype=np.int64)
    raise RuntimeError("not enough distinct draws")


def student_t3_row_scale(N: int, seed: int) -> np.ndarray:
    """|t_n| for a Student-t (nu = 3) draw per row: z0 / sqrt((z1^2+z2^2+z3^2)/3)."""
    z = normal(4 * N, seed, 3).reshape(N, 4)
    chi2 = (z[:, 1:] ** 2).sum(axis=1)
    return np.abs(z[:, 0] / np.sqrt(chi2 / 3.0))


# --------------------------------------------------------------------------- recipes
WORKLOADS = {
    "tiny": dict(N=512, K=256, Ms=(4,)),
    "decode": dict(N=128256, K=4096, Ms=(1, 8, 32, 64)),
    "prefill": dict(N=128256, K=4096, Ms=(2048,)),
    "quant": dict(N=151936, K=5120, Ms=()),
    "sweep": dict(N=262144, K=8192, Ms=(1, 4, 16, 64, 256, 1024)),
}


def tiny_weight(N: int = 512, K: int = 256) -> np.ndarray:
    rows = distinct_rows(4, N, seed=0, stream=1)
    rm = np.ones(N)
    rm[rows] = 50.0
    return weight(N, K, seed=0, sigma=0.02, row_mult=rm)


def tiny_outlier_rows(N: int = 512) -> np.ndarray:
    return distinct_rows(4, N, seed=0, stream=1)


def tiny_x(M: int = 4, K: int = 256) -> np.ndarray:
    return activations(M, K, seed=100, rms_normalize=False)


def decode_weight(N: int = 128256, K: int = 4096, seed: int = 1) -> np.ndarray:
    return weight(N, K, seed=seed, sigma=0.02, p=0.001, mult=20.0)


def decode_x(M: int, K: int = 4096) -> np.ndarray:
    return activations(M, K, seed=101, rms_normalize=True)


def prefill_x(M: int = 2048, K: int = 4096) -> np.ndarray:
    return activations(M, K, seed=102, rms_normalize=True)


def quant_weight(N: int = 151936, K: int = 5120, seed: int = 4) -> np.ndarray:
    return weight(N, K, seed=seed, sigma=0.015, row_mult=student_t3_row_scale(N, seed))


def sweep_weight(N: int = 262144, K: int = 8192) -> np.ndarray:
    return weight(N, K, seed=6, sigma=0.01)


def sweep_x(M: int, K: int = 8192) -> np.ndarray:
    return activations(M, K, seed=106, rms_normalize=True)


def num_threads() -> int:
    return int(_load().synth_num_threads())


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (plumbing for tests)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest even) and return the bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


os.environ.setdefault("OMP_WAIT_POLICY", "PASSIVE")
