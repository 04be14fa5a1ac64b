"""Plumbing shared by the GPU tests: move bf16 bit-pattern arrays to and from
the device, the logits tolerance of the products, and the expected top-k of
a logits matrix with its oracle-agreement check."""
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


def expected_topk(L: torch.Tensor, k: int):
    """(rows, values) of the k largest of each row of fp32 logits, on the
    device, by the 64-bit order key (value order with NaN on top, then the
    smaller row), -0 counted as +0."""
    L = torch.where(L == 0, torch.zeros_like(L), L)
    b = L.view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    ok = torch.where(b >= 2 ** 31, b ^ 0xFFFFFFFF, b | 0x80000000)
    n = torch.arange(L.shape[1], device=L.device, dtype=torch.int64)
    key = ((ok - 2 ** 31) << 32) | (~n & 0xFFFFFFFF)
    top = torch.topk(key, k, dim=1, sorted=True).values
    ids = ~top & 0xFFFFFFFF
    return ids, L.gather(1, ids)


def assert_topk_equal(ids: torch.Tensor, vals, want_ids: torch.Tensor, want_vals, what=""):
    """Rows identical; values identical bit for bit (or both NaN)."""
    bad = (ids != want_ids).any(dim=1).nonzero()[:, 0]
    assert bad.numel() == 0, (what, bad[:3].tolist(), ids[bad[:1]].tolist(),
                              want_ids[bad[:1]].tolist())
    if vals is not None:
        same = (vals.view(torch.int32) == want_vals.view(torch.int32)) | (
            torch.isnan(vals) & torch.isnan(want_vals))
        assert bool(same.all()), (what, vals[~same][:5].tolist(), want_vals[~same][:5].tolist())


def assert_topk_oracle_agrees(ids: np.ndarray, vals: np.ndarray, ref: np.ndarray) -> None:
    """ids, vals: [T, k] from the GPU; ref: the oracle's fp64 logits [T, N].
    Every returned value is within the logits tolerance of the oracle's logit
    at its row, and no row left out is above the smallest returned one by
    more than twice the tolerance."""
    tol = logits_tolerance(ref)[:, 0]
    k = ids.shape[1]
    for m in range(ref.shape[0]):
        sel = ids[m]
        assert len(set(sel.tolist())) == k, m
        err = np.abs(vals[m].astype(np.float64) - ref[m, sel])
        assert np.all(err <= tol[m]), (m, err.max(), tol[m])
        out = np.ones(ref.shape[1], dtype=bool)
        out[sel] = False
        if out.any():
            assert ref[m, out].max() <= ref[m, sel].min() + 2 * tol[m], m
