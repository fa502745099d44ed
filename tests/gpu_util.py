"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
from __future__ import annotations

import numpy as np
import torch

from oracle import gemm_tolerance


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str) -> None:
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if got.dtype == np.float32:
        got, want = got.view(np.uint32), want.view(np.uint32)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:5].tolist()}: " \
                          f"got {got[tuple(bad[0])]} want {want[tuple(bad[0])]}"


def assert_gemm_close(y_bits: np.ndarray, y_ref: np.ndarray, L: np.ndarray, what: str) -> float:
    """|y - y_ref| <= 2^-8 |y_ref| + 1e-4 L elementwise; returns max err/tol."""
    y = bf16_to_f64(y_bits)
    err = np.abs(y - y_ref)
    tol = gemm_tolerance(y_ref, L)
    ratio = err / np.maximum(tol, 1e-300)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, f"{what}: {len(bad)} of {err.size} outside tolerance; first {bad[:3].tolist()} " \
                          f"y={y[tuple(bad[0])]} ref={y_ref[tuple(bad[0])]} tol={tol[tuple(bad[0])]}"
    return float(ratio.max())


def sample_rows(M: int, n: int, seed: int = 0) -> np.ndarray:
    """Rows at both ends, around 128-row tile edges, and random ones."""
    rng = np.random.default_rng(seed)
    edges = [0, 1, M - 1, M - 2, 127, 128, 129, 255, 256, M // 2]
    rows = set(r for r in edges if 0 <= r < M)
    if M > len(rows):
        rows.update(rng.choice(M, size=min(n, M), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)
