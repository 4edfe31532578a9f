"""Shared helpers for the GPU parity tests (no oracle arithmetic here)."""
import numpy as np
import pytest
import torch

# Tolerances against the fp64 oracle, on identical (bf16-rounded) inputs:
# bf16 inputs with fp32 accumulation: O max abs <= 2e-2, O mean abs <= 2e-3,
# lse max abs <= 1e-3; fp32 inputs: O max abs <= 1e-4 (lse held to the same).
BF16_O_MAX = 2e-2
BF16_O_MEAN = 2e-3
LSE_MAX = 1e-3
F32_O_MAX = 1e-4
F32_LSE_MAX = 1e-4
# FP8 (E4M3) inputs, against the oracle on the same dequantized inputs: O is held to a
# per-element bound derived from the rounding of P to E4M3 (tests/test_gpu_fp8.py,
# _p_rounding_bound), plus these two: O mean abs <= 1e-2; lse (fp32 S from exact E4M3
# products, unrounded P in l) <= 1e-3.
FP8_O_MEAN = 1e-2
FP8_LSE_MAX = 1e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from exact_tiled_attention_fattn_gb300 import build, fattn
    build.build()
    return fattn


def as_np(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().float().cpu().double().numpy()


def check(o_gpu, lse_gpu, o_ref, lse_ref, fp32=False, what=""):
    o = as_np(o_gpu) if isinstance(o_gpu, torch.Tensor) else o_gpu
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    if fp32:
        assert err.max() <= F32_O_MAX, f"{what}: O max err {err.max():.3e}"
    else:
        assert err.max() <= BF16_O_MAX, f"{what}: O max err {err.max():.3e}"
        assert err.mean() <= BF16_O_MEAN, f"{what}: O mean err {err.mean():.3e}"
    if lse_gpu is not None:
        lg = as_np(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lg), fin), f"{what}: lse finiteness differs"
        lerr = np.abs(lg[fin] - lse_ref[fin]) if fin.any() else np.zeros(1)
        assert lerr.max() <= (F32_LSE_MAX if fp32 else LSE_MAX), f"{what}: lse max err {lerr.max():.3e}"
    return float(err.max()), float(err.mean())


def tile_edge_rows(n_rows, tile=128):
    """The first and the last row of every `tile`-row query tile of a sequence of
    n_rows rows (the kernels give each tile, or pair of tiles, to one work item: a
    mis-mapped or dropped item shows at its tile's edges)."""
    rows = []
    for t0 in range(0, n_rows, tile):
        rows += [t0, min(t0 + tile, n_rows) - 1]
    return sorted(set(rows))


def tile_edge_samples(B, H, N, rng, extra=256):
    """(b, h, i) samples: both edge rows of every (b, h, 128-row tile), plus `extra` random rows."""
    edges = tile_edge_rows(N)
    s = [(b, h, i) for b in range(B) for h in range(H) for i in edges]
    s += [(int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N))) for _ in range(extra)]
    return np.array(s, dtype=np.int64)


def nan_outputs(shape_o, shape_lse, dtype=torch.bfloat16, device="cuda"):
    """Output buffers filled with NaN, so that a row no work item writes stays NaN
    and fails the finiteness check."""
    o = torch.full(shape_o, float("nan"), dtype=dtype, device=device)
    lse = torch.full(shape_lse, float("nan"), dtype=torch.float32, device=device)
    return o, lse
