"""FP8 (E4M3) prefill: the CUDA kernel through the C ABI against the fp64 oracle on
the dequantized inputs."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_fattn_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import FP8_LSE_MAX, FP8_O_MEAN, as_np, nan_outputs, need_gpu, tile_edge_samples

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    return need_gpu()


def _p_rounding_bound(x, rows):
    """Per-element error bound for O from the one rounding the definition does not have:
    P rounded to E4M3 before P V (the sums l use the unrounded P), on the oracle's weights
    w_j (true row max: p_j = e^{s_j - m}, l = sum_j p_j = 1 / max_j w_j).
    A weight in E4M3's normal range moves by at most 2^-4 of itself (half an ulp of 3
    mantissa bits); one in the subnormal range (p < 2^-6) by at most 2^-10 absolute, i.e.
    2^-10 / l after normalising (a stale running max only raises p and l together, which
    does not loosen either bound). Round-to-nearest errors of different weights are
    treated as independent, zero-mean, of variance at most (bound)^2 / 3, so
    sigma_ic^2 = (1/3) sum_j max(2^-4 w_j, 2^-10 w_max)^2 v_jc^2 over the visible keys;
    the bound is 6 sigma plus the bf16 output rounding (2^-9 |O|, doubled) plus 2^-10
    sum_j w_j |v_jc| for fp32 accumulation order. rows: int [n, 3] of (b, h, i)."""
    q = orc.e4m3_to_f64(x.q8) * x.q_descale
    k = orc.e4m3_to_f64(x.k8) * x.k_descale
    v = orc.e4m3_to_f64(x.v8) * x.v_descale
    g = q.shape[2] // k.shape[2]
    N = q.shape[1]
    sigma = np.zeros((len(rows), v.shape[-1]))
    l1 = np.zeros((len(rows), v.shape[-1]))
    for b, h in sorted({(int(b), int(h)) for b, h, _ in rows}):
        idx = np.nonzero((rows[:, 0] == b) & (rows[:, 1] == h))[0]
        r = rows[idx, 2]
        w = orc.attention_weights(q[b, :, h], k[b, :, h // g], x.scale, x.causal, rows=r)   # [n, N]
        vis = (np.arange(N)[None, :] <= r[:, None]) if x.causal else np.ones_like(w, dtype=bool)
        dw = np.where(vis, np.maximum(2.0 ** -4 * w, 2.0 ** -10 * w.max(axis=1, keepdims=True)), 0.0)
        vh = v[b, :, h // g]
        sigma[idx] = np.sqrt((dw ** 2) @ (vh ** 2) / 3.0)
        l1[idx] = w @ np.abs(vh)
    return sigma, l1


def _check_fp8(o, lse, o_ref, lse_ref, x, rows, what):
    """O within the per-element bound of _p_rounding_bound; mean |err| <= 1e-2; lse <= 1e-3."""
    og = as_np(o)
    err = np.abs(og - o_ref)
    lerr = np.abs(as_np(lse) - lse_ref)
    sigma, l1 = _p_rounding_bound(x, rows)
    bound = 6.0 * sigma + 2.0 ** -8 * np.abs(o_ref) + 2.0 ** -10 * l1 + 1e-4
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    print(what, f"O max {err.max():.3e} mean {err.mean():.3e} lse max {lerr.max():.3e}; "
                f"worst err/bound {float((err / bound)[worst]):.3f} (err {err[worst]:.3e}, bound {bound[worst]:.3e})")
    assert np.all(np.isfinite(og))
    assert np.all(err <= bound), f"{what}: O err {err[worst]:.3e} above its bound {bound[worst]:.3e} at {worst}"
    assert err.mean() <= FP8_O_MEAN, f"{what}: O mean err {err.mean():.3e}"
    assert lerr.max() <= FP8_LSE_MAX, f"{what}: lse max err {lerr.max():.3e}"


def _all_rows(B, H, N):
    return np.array([(b, h, i) for b in range(B) for h in range(H) for i in range(N)], dtype=np.int64)


def _flat(o, lse, rows):
    """O [n, d] and lse [n] of a dense [B, N, H, d] / [B, H, N] output at rows (b, h, i)."""
    og, lg = as_np(o), as_np(lse)
    return og[rows[:, 0], rows[:, 2], rows[:, 1]], lg[rows[:, 0], rows[:, 1], rows[:, 2]]


CASES = [(2, 300, 4, 2, True), (1, 513, 8, 1, True), (2, 256, 2, 2, False), (1, 1000, 4, 4, True),
         # shorter than one tile: V rows past N come from the next sequence (times P = 0) or as zeros
         (3, 37, 2, 1, True), (2, 1, 2, 2, False)]


@pytest.mark.parametrize("B,N,Hq,Hkv,causal", CASES)
def test_fp8_parity(fa, B, N, Hq, Hkv, causal):
    x = inputs.prefill_fp8(6000 + N, B, N, Hq, Hkv, 128, causal)
    o, lse = fa.fwd_fp8(x.q8.cuda(), x.k8.cuda(), x.v8.cuda(), x.q_descale, x.k_descale, x.v_descale,
                        causal=causal, scale=x.scale)
    assert fa.debug_read_status() == 0
    rows = _all_rows(B, Hq, N)
    o_ref, lse_ref = orc.attn_fwd_fp8(x.q8, x.k8, x.v8, x.q_descale, x.k_descale, x.v_descale, x.scale, causal,
                                      rows=rows)
    og, lg = _flat(o, lse, rows)
    _check_fp8(og, lg, o_ref, lse_ref, x, rows, f"fp8 {B, N, Hq, Hkv, causal}")


@pytest.mark.parametrize("scale", [-0.1, 0.25])
def test_fp8_parity_other_scales(fa, scale):
    """A negative and a large scale (folded with the q and k descales into the exponent
    scale), B=2 N=300 GQA 4:2 causal."""
    x = inputs.prefill_fp8(6500 + int(100 * scale), 2, 300, 4, 2, 128, True, scale=scale)
    o, lse = fa.fwd_fp8(x.q8.cuda(), x.k8.cuda(), x.v8.cuda(), x.q_descale, x.k_descale, x.v_descale,
                        causal=True, scale=x.scale)
    assert fa.debug_read_status() == 0
    rows = _all_rows(2, 4, 300)
    o_ref, lse_ref = orc.attn_fwd_fp8(x.q8, x.k8, x.v8, x.q_descale, x.k_descale, x.v_descale, x.scale, True,
                                      rows=rows)
    og, lg = _flat(o, lse, rows)
    _check_fp8(og, lg, o_ref, lse_ref, x, rows, f"fp8 scale {scale}")


def test_fp8_large_every_item(fa):
    """Causal MHA B=4, H=32, N=4096, d=128 in E4M3, on NaN-filled outputs: every row
    written, both edge rows of every (sequence, head, 128-row tile) and random rows
    against the oracle."""
    B, N, H = 4, 4096, 32
    x = inputs.prefill_fp8(6100, B, N, H, H, 128, True)
    o, lse = nan_outputs((B, N, H, 128), (B, H, N))
    fa.fwd_fp8(x.q8.cuda(), x.k8.cuda(), x.v8.cuda(), x.q_descale, x.k_descale, x.v_descale,
               causal=True, scale=x.scale, out=o, lse=lse)
    assert fa.debug_read_status() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all(), "rows left unwritten (NaN)"
    smp = tile_edge_samples(B, H, N, np.random.default_rng(11), extra=96)
    o_ref, lse_ref = orc.attn_fwd_fp8(x.q8, x.k8, x.v8, x.q_descale, x.k_descale, x.v_descale, x.scale, True,
                                      rows=smp)
    og, lg = _flat(o, lse, smp)
    _check_fp8(og, lg, o_ref, lse_ref, x, smp, "fp8 large")


def test_fp8_lazy_rescale_after_mass_jumps(fa):
    """E4M3 q = e_0, k[..., 0] = 6 per jump (tiles 3 and 7 of head 0, 1 and 5 of head 1;
    6 and 12 are exact in E4M3), scale 1: the running max rises by 8.7 > 8 in log2 units
    twice while the earlier tiles keep weight; V = (tile index + 1) / 8 + 0.02 N(0, 1), quantized."""
    N, H, d = 1024, 2, 128
    g = torch.Generator().manual_seed(43)
    tile = torch.arange(N) // 128
    q = torch.zeros(1, N, H, d)
    q[..., 0] = 1.0
    k = torch.zeros(1, N, H, d)
    for h, js in enumerate([(3, 7), (1, 5)]):
        k[0, :, h, 0] = 6.0 * sum((tile >= t).float() for t in js)
    v = (tile[None, :, None, None].float() + 1.0) / 8 + 0.02 * torch.randn(1, N, H, d, generator=g)
    q8, k8, v8 = (t.to(torch.float8_e4m3fn).view(torch.uint8) for t in (q, k, v))
    o, lse = fa.fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), 1.0, 1.0, 1.0, causal=True, scale=1.0)
    assert fa.debug_read_status() == 0
    rows = _all_rows(1, H, N)
    o_ref, lse_ref = orc.attn_fwd_fp8(q8, k8, v8, 1.0, 1.0, 1.0, 1.0, True, rows=rows)
    x = inputs.Fp8Inputs(q8, k8, v8, 1.0, 1.0, 1.0, True, 1.0)
    og, lg = _flat(o, lse, rows)
    _check_fp8(og, lg, o_ref, lse_ref, x, rows, "fp8 rescale jumps")
