"""Plumbing shared by the GPU tests: move bf16 bit-pattern arrays to and from
the device, and the logits tolerance of the W4A16 product."""
from __future__ import annotations

import numpy as np
import torch


def to_bf16_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def scales_bytes(scales: torch.Tensor) -> np.ndarray:
    return scales.view(torch.uint8).cpu().numpy()


def logits_tolerance(ref: np.ndarray) -> np.ndarray:
    """|err| <= 2e-3 * max|row of oracle logits| + 1e-3, per token row."""
    return 2e-3 * np.abs(ref).max(axis=1, keepdims=True) + 1e-3


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |v| (the most an RNE cast moves v)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 8)


def assert_logits_close(got: np.ndarray, ref: np.ndarray, what: str = "",
                        out_bf16: bool = False) -> None:
    """Logits tolerance; bf16 logits also get the half-ulp of their final RNE cast."""
    tol = logits_tolerance(ref)
    if out_bf16:
        tol = tol + bf16_half_ulp(ref)
    err = np.abs(got.astype(np.float64) - ref)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (
        f"{what}: {len(bad)} logits outside tolerance; first {bad[:5].tolist()} "
        f"got {[float(got[tuple(b)]) for b in bad[:5]]} want {[float(ref[tuple(b)]) for b in bad[:5]]}")


def assert_argmax_agrees(got: np.ndarray, ref: np.ndarray, out_bf16: bool = False) -> None:
    """argmax per row agrees unless the oracle's top two differ by < 1e-3.

    With bf16 logits two oracle values within one bf16 step of each other can
    round to the same value or swap, so the margin then also covers one bf16
    ulp of the oracle's maximum."""
    for m in range(ref.shape[0]):
        a, b = int(np.argmax(got[m])), int(np.argmax(ref[m]))
        if a != b:
            margin = 1e-3 + (2 * float(bf16_half_ulp(ref[m, b])) if out_bf16 else 0.0)
            assert ref[m, b] - ref[m, a] < margin, (m, a, b, ref[m, a], ref[m, b])
