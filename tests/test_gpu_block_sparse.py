"""Block-sparse prefill ('Block-sparse FlashAttention': zero blocks of a fixed block
mask are skipped): the CUDA kernel through the C ABI against the fp64 oracle."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_fattn_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import as_np, check, nan_outputs, need_gpu, tile_edge_samples

pytestmark = pytest.mark.gpu
BLK = 128


@pytest.fixture(scope="module")
def fa():
    return need_gpu()


def _mask(rng, heads, nb, density, empty_row=None):
    m = (rng.random((heads, nb, nb)) < density).astype(np.uint8)
    if empty_row is not None:
        m[:, empty_row, :] = 0                 # these query blocks keep no key at all
    return m


def _run(fa, x, mask, causal):
    o, lse = fa.fwd_block_sparse(x.q.cuda(), x.k.cuda(), x.v.cuda(), torch.from_numpy(mask).cuda(),
                                 causal=causal, scale=x.scale)
    assert fa.debug_read_status() == 0
    return o, lse


CASES = [
    # B, N, Hq, Hkv, d, causal, per_head_mask, density
    (2, 300, 4, 2, 128, False, False, 0.5),
    (2, 300, 4, 2, 128, True, True, 0.6),
    (1, 513, 8, 1, 64, True, False, 0.5),
    (1, 1024, 4, 4, 128, False, True, 0.3),
    (1, 1000, 2, 1, 64, False, True, 0.7),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal,per_head,density", CASES)
def test_block_sparse_parity(fa, B, N, Hq, Hkv, d, causal, per_head, density):
    rng = np.random.default_rng(N + d + (7 if causal else 0))
    x = inputs.prefill_dense(3000 + N, B, N, Hq, Hkv, d, causal)
    nb = -(-N // BLK)
    mask = _mask(rng, Hq if per_head else 1, nb, density, empty_row=nb // 2)
    o, lse = _run(fa, x, mask, causal)
    o_ref, lse_ref = orc.attn_fwd_block_sparse(x.q, x.k, x.v, x.scale, causal, mask, BLK)
    check(o, lse, o_ref, lse_ref, what=f"block-sparse {B, N, Hq, Hkv, d, causal, per_head}")
    og = as_np(o)
    rows = slice((nb // 2) * BLK, min(N, (nb // 2 + 1) * BLK))
    assert np.all(og[:, rows] == 0) and np.all(np.isneginf(as_np(lse)[:, :, rows]))


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_equals_dense(fa, causal):
    x = inputs.prefill_dense(3100, 2, 640, 4, 2, 128, causal)
    nb = -(-640 // BLK)
    o1, l1 = _run(fa, x, np.ones((1, nb, nb), np.uint8), causal)
    o2, l2 = fa.fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=causal, scale=x.scale)
    o_ref, lse_ref = orc.attn_fwd(x.q, x.k, x.v, x.scale, causal)
    check(o1, l1, o_ref, lse_ref, what="all-ones sparse")
    check(o2, l2, o_ref, lse_ref, what="dense")
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_lower_triangular_blocks_with_causal_equal_causal(fa):
    x = inputs.prefill_dense(3200, 1, 777, 4, 4, 64, True)
    nb = -(-777 // BLK)
    mask = np.tril(np.ones((nb, nb), np.uint8))[None]
    o, lse = _run(fa, x, mask, True)
    o_ref, lse_ref = orc.attn_fwd(x.q, x.k, x.v, x.scale, True)
    check(o, lse, o_ref, lse_ref, what="tril blocks")


def test_local_global_pattern_large_every_item(fa):
    """B=1, H=32, N=4096, d=128: sliding window of 3 blocks plus the first block (~17% dense),
    on NaN-filled outputs: every row written, both edge rows of every (head, 128-row
    tile) and random rows against the oracle."""
    B, N, H, d = 1, 4096, 32, 128
    x = inputs.prefill_dense(3300, B, N, H, H, d, causal=True)
    nb = N // BLK
    m = np.zeros((1, nb, nb), np.uint8)
    for i in range(nb):
        m[0, i, max(0, i - 2): i + 1] = 1
        m[0, i, 0] = 1
    o, lse = nan_outputs(x.q.shape, (B, H, N))
    fa.fwd_block_sparse(x.q.cuda(), x.k.cuda(), x.v.cuda(), torch.from_numpy(m).cuda(), causal=True,
                        scale=x.scale, out=o, lse=lse)
    assert fa.debug_read_status() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all(), "rows left unwritten (NaN)"
    smp = tile_edge_samples(B, H, N, np.random.default_rng(5), extra=128)
    o_ref, lse_ref = orc.attn_fwd_block_sparse(x.q, x.k, x.v, x.scale, True, m, BLK, rows=smp)
    hi = torch.as_tensor(smp[:, 1], device="cuda")
    ii = torch.as_tensor(smp[:, 2], device="cuda")
    check(o[0, ii, hi], lse[0, hi, ii], o_ref, lse_ref, what="local+global")


def test_binding_rejects_mismatched_shapes(fa):
    dev, bf = "cuda", torch.bfloat16
    q = torch.zeros(1, 256, 4, 128, dtype=bf, device=dev)
    k_short = torch.zeros(1, 128, 2, 128, dtype=bf, device=dev)
    k = torch.zeros(1, 256, 2, 128, dtype=bf, device=dev)
    mask = torch.ones(1, 2, 2, dtype=torch.uint8, device=dev)
    with pytest.raises(ValueError):
        fa.fwd(q, k_short, k_short)
    with pytest.raises(ValueError):
        fa.fwd_block_sparse(q, k_short, k_short, mask)
    with pytest.raises(ValueError):
        fa.fwd_block_sparse(q, k, k, torch.ones(1, 3, 3, dtype=torch.uint8, device=dev))
    with pytest.raises(ValueError):
        fa.fwd(q, k, k, out=torch.empty(1, 256, 4, 64, dtype=bf, device=dev))
    with pytest.raises(TypeError):
        fa.fwd(q, k, k, lse=torch.empty(1, 4, 256, dtype=bf, device=dev))
