"""FP8 (E4M3) prefill: the CUDA kernel through the C ABI against the fp64 oracle on
the dequantized inputs."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_fattn_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import FP8_LSE_MAX, FP8_O_MAX, FP8_O_MEAN, as_np, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    return need_gpu()


def _check_fp8(o, lse, o_ref, lse_ref, what):
    err = np.abs(as_np(o) - o_ref)
    lerr = np.abs(as_np(lse) - lse_ref)
    print(what, f"O max {err.max():.3e} mean {err.mean():.3e} lse max {lerr.max():.3e}")
    assert np.all(np.isfinite(as_np(o)))
    assert err.max() <= FP8_O_MAX, f"{what}: O max err {err.max():.3e}"
    assert err.mean() <= FP8_O_MEAN, f"{what}: O mean err {err.mean():.3e}"
    assert lerr.max() <= FP8_LSE_MAX, f"{what}: lse max err {lerr.max():.3e}"


CASES = [(2, 300, 4, 2, True), (1, 513, 8, 1, True), (2, 256, 2, 2, False), (1, 1000, 4, 4, True)]


@pytest.mark.parametrize("B,N,Hq,Hkv,causal", CASES)
def test_fp8_parity(fa, B, N, Hq, Hkv, causal):
    x = inputs.prefill_fp8(6000 + N, B, N, Hq, Hkv, 128, causal)
    o, lse = fa.fwd_fp8(x.q8.cuda(), x.k8.cuda(), x.v8.cuda(), x.q_descale, x.k_descale, x.v_descale,
                        causal=causal, scale=x.scale)
    assert fa.debug_read_status() == 0
    o_ref, lse_ref = orc.attn_fwd_fp8(x.q8, x.k8, x.v8, x.q_descale, x.k_descale, x.v_descale, x.scale, causal)
    _check_fp8(o, lse, o_ref, lse_ref, f"fp8 {B, N, Hq, Hkv, causal}")


def test_fp8_large_sampled(fa):
    """Causal MHA B=4, H=32, N=4096, d=128 in E4M3: sampled rows."""
    B, N, H = 4, 4096, 32
    x = inputs.prefill_fp8(6100, B, N, H, H, 128, True)
    o, lse = fa.fwd_fp8(x.q8.cuda(), x.k8.cuda(), x.v8.cuda(), x.q_descale, x.k_descale, x.v_descale,
                        causal=True, scale=x.scale)
    assert fa.debug_read_status() == 0
    rng = np.random.default_rng(11)
    smp = np.array([(int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N))) for _ in range(96)] +
                   [(0, 0, 0), (3, 31, N - 1)])
    o_ref, lse_ref = orc.attn_fwd_fp8(x.q8, x.k8, x.v8, x.q_descale, x.k_descale, x.v_descale, x.scale, True,
                                      rows=smp)
    bi, hi, ii = (torch.as_tensor(smp[:, c], device="cuda") for c in range(3))
    _check_fp8(o[bi, ii, hi], lse[bi, hi, ii], o_ref, lse_ref, "fp8 large")


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
    o_ref, lse_ref = orc.attn_fwd_fp8(q8, k8, v8, 1.0, 1.0, 1.0, 1.0, True)
    _check_fp8(o, lse, o_ref, lse_ref, "fp8 rescale jumps")
