"""Prefill with a general additive mask (the formula's M, added to each score
tile on chip): the CUDA kernel through the C ABI against the fp64 oracle."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_fattn_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import as_np, check, nan_outputs, need_gpu, tile_edge_samples

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    return need_gpu()


def _mask(seed, Bm, Hm, N, pad=8):
    """bf16 mask [Bm, Hm, N, L], L = N rounded up to 8 plus `pad`; entries 2 N(0, 1), about 5 %
    -inf, row 3 fully -inf; the padding past N is NaN (it must never be read)."""
    g = torch.Generator("cpu").manual_seed(seed)
    L = (N + 7) // 8 * 8 + pad
    m = 2.0 * torch.randn((Bm, Hm, N, L), generator=g)
    m[torch.rand((Bm, Hm, N, L), generator=g) < 0.05] = float("-inf")
    m[:, :, 3, :] = float("-inf")
    m[..., N:] = float("nan")
    return m.to(torch.bfloat16)


CASES = [
    # B, N, Hq, Hkv, d, causal, Bm, Hm
    (2, 300, 4, 2, 128, False, 1, 1),
    (2, 300, 4, 2, 128, True, 2, 4),
    (1, 513, 8, 1, 64, True, 1, 8),
    (2, 256, 2, 2, 64, False, 2, 1),
    (1, 1000, 2, 2, 128, True, 1, 1),
    # shorter than one tile; rows 32 entries long (32-byte loads of 16-key groups)
    (2, 24, 2, 2, 128, True, 2, 1),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal,Bm,Hm", CASES)
def test_masked_parity(fa, B, N, Hq, Hkv, d, causal, Bm, Hm):
    x = inputs.prefill_dense(5000 + N + d, B, N, Hq, Hkv, d, causal)
    m = _mask(5100 + N, Bm, Hm, N)
    o, lse = fa.fwd_masked(x.q.cuda(), x.k.cuda(), x.v.cuda(), m.cuda(), causal=causal, scale=x.scale)
    assert fa.debug_read_status() == 0
    o_ref, lse_ref = orc.attn_fwd_masked(x.q, x.k, x.v, x.scale, causal, m[..., :N].float().numpy())
    check(o, lse, o_ref, lse_ref, what=f"masked {B, N, Hq, Hkv, d, causal, Bm, Hm}")
    og = as_np(o)
    assert np.all(og[:, 3] == 0) and np.all(np.isneginf(as_np(lse)[:, :, 3]))   # the fully masked row


@pytest.mark.parametrize("scale,d", [(-0.2, 128), (0.3, 64)])
def test_masked_parity_other_scales(fa, scale, d):
    """The mask is added to the scaled scores, so a negative scale changes which keys
    dominate but not the max rule; B=2 N=300 GQA 4:2 causal, one mask per (b, h)."""
    x = inputs.prefill_dense(5500 + d, 2, 300, 4, 2, d, True, scale=scale)
    m = _mask(5600 + d, 2, 4, 300)
    o, lse = fa.fwd_masked(x.q.cuda(), x.k.cuda(), x.v.cuda(), m.cuda(), causal=True, scale=scale)
    assert fa.debug_read_status() == 0
    o_ref, lse_ref = orc.attn_fwd_masked(x.q, x.k, x.v, scale, True, m[..., :300].float().numpy())
    check(o, lse, o_ref, lse_ref, what=f"masked scale {scale} d {d}")


def test_lower_triangle_mask_equals_causal(fa):
    x = inputs.prefill_dense(5200, 1, 384, 4, 4, 128, True)
    N = 384
    tri = torch.where(torch.ones(N, N).tril() > 0, 0.0, float("-inf")).to(torch.bfloat16)[None, None]
    o1, l1 = fa.fwd_masked(x.q.cuda(), x.k.cuda(), x.v.cuda(), tri.cuda(), causal=False, scale=x.scale)
    o2, l2 = fa.fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True, scale=x.scale)
    o_ref, lse_ref = orc.attn_fwd(x.q, x.k, x.v, x.scale, True)
    check(o1, l1, o_ref, lse_ref, what="-inf above the diagonal")
    check(o2, l2, o_ref, lse_ref, what="causal")


def test_alibi_bias_large_every_item(fa):
    """B=4, H=32, N=4096, d=128, causal, one shared bias M[i, j] = -0.01 (i - j), on
    NaN-filled outputs: every row written, both edge rows of every (sequence, head,
    128-row tile) and random rows against the oracle."""
    B, N, H, d = 4, 4096, 32, 128
    x = inputs.prefill_dense(5300, B, N, H, H, d, True)
    i = torch.arange(N, dtype=torch.float32)
    m = (-0.01 * (i[:, None] - i[None, :])).to(torch.bfloat16)[None, None]
    o, lse = nan_outputs(x.q.shape, (B, H, N))
    fa.fwd_masked(x.q.cuda(), x.k.cuda(), x.v.cuda(), m.cuda(), causal=True, scale=x.scale, out=o, lse=lse)
    assert fa.debug_read_status() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all(), "rows left unwritten (NaN)"
    smp = tile_edge_samples(B, H, N, np.random.default_rng(9), extra=96)
    o_ref, lse_ref = orc.attn_fwd_masked(x.q, x.k, x.v, x.scale, True, m.float().numpy(), rows=smp)
    bi, hi, ii = (torch.as_tensor(smp[:, c], device="cuda") for c in range(3))
    check(o[bi, ii, hi], lse[bi, hi, ii], o_ref, lse_ref, what="ALiBi-style bias")


@pytest.mark.parametrize("d", [64, 128])
def test_lazy_rescale_from_mask_jumps(fa, d):
    """The mask raises whole key tiles (3 and 7) by 5.75 above the tiles before them
    (q, k random, so the scores stay within a few units): the running max jumps by more
    than 2^8 twice and O is rescaled while the earlier tiles still carry weight; V grows
    with the tile index."""
    N = 1024
    x = inputs.prefill_dense(5400 + d, 1, N, 2, 2, d, False)
    tile = torch.arange(N) // 128
    col = 5.75 * ((tile >= 3).float() + (tile >= 7).float())
    m = col[None, :].expand(N, N).to(torch.bfloat16)[None, None].contiguous()
    v = ((tile[None, :, None, None].float() + 1.0) / 8 + 0.1 * x.v.float()).to(torch.bfloat16)
    o, lse = fa.fwd_masked(x.q.cuda(), x.k.cuda(), v.cuda(), m.cuda(), causal=True, scale=x.scale)
    assert fa.debug_read_status() == 0
    o_ref, lse_ref = orc.attn_fwd_masked(x.q, x.k, v, x.scale, True, m.float().numpy())
    check(o, lse, o_ref, lse_ref, what=f"mask jumps d={d}")
