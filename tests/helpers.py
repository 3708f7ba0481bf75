"""Helpers shared by the GPU parity tests: moving bf16 bit arrays to the device,
the GEMM tolerance, and running the library on oracle-made codes."""
import numpy as np
import torch

TILE = 128


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns (host) -> bfloat16 CUDA tensor, bit for bit."""
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def scales_to_dev(s: np.ndarray) -> torch.Tensor:
    """[chunks, n] float32 -> CUDA view with row stride rounded up to 4 (16-byte rows)."""
    chunks, n = s.shape
    ld = max((n + 3) // 4 * 4, 4)
    buf = torch.zeros((chunks, ld), dtype=torch.float32, device="cuda")
    buf[:, :n] = torch.from_numpy(np.ascontiguousarray(s, dtype=np.float32)).cuda()
    return buf[:, :n]


def from_dev_bf16(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def gemm_tolerance_ok(y: np.ndarray, y_ref: np.ndarray, rms_ref: float = None):
    """|y - y_ref| <= 1e-2 |y_ref| + 1e-3 rms(y_ref), rms over the compared output.

    Returns (ok, worst ratio of error to allowance).
    """
    if rms_ref is None:
        rms_ref = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    allow = 1e-2 * np.abs(y_ref) + 1e-3 * rms_ref
    err = np.abs(y - y_ref)
    if err.size == 0:
        return True, 0.0
    ratio = float(np.max(err / np.maximum(allow, 1e-300)))
    return bool(np.all(err <= allow)), ratio


def tile_rows(total: int, seed: int, extra: int = 32, tile: int = TILE) -> np.ndarray:
    """Row indices that cover every 128-row tile of an output: one random row in each tile
    (the last, ragged tile included), the first and the last row, and `extra` more random
    rows. Compared over all columns, they touch every output tile of the GEMM."""
    rng = np.random.default_rng(seed)
    picks = [0, total - 1]
    for t0 in range(0, total, tile):
        picks.append(int(rng.integers(t0, min(t0 + tile, total))))
    if extra:
        picks += list(rng.integers(0, total, size=extra))
    return np.unique(np.asarray(picks, dtype=np.int64))
