"""Paged (chunked) prefill ('Paged variants': the tiled computation with K/V read
through a block table): the CUDA kernel through the C ABI against the fp64 oracle."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_fattn_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import as_np, check, nan_outputs, need_gpu, tile_edge_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    return need_gpu()


def _run(fa, x, **kw):
    o, lse = fa.fwd_paged(x.q.cuda(), x.kcache.cuda(), x.vcache.cuda(), x.block_table.cuda(), x.seqlens_k.cuda(),
                          x.cu_seqlens_q.cuda(), max(x.lengths_q), causal=x.causal, scale=x.scale, **kw)
    return o, lse


CASES = [
    # seed, B, Hq, Hkv, d, page, lengths_k, lengths_q, causal, max_context
    (1, 3, 4, 2, 128, 16, (100, 700), None, True, 768),
    (2, 2, 8, 1, 64, 32, [300, 513], [300, 128], True, 640),
    (3, 4, 4, 4, 128, 64, [1000, 129, 5, 640], [256, 1, 5, 300], False, 1024),
    (4, 2, 2, 1, 128, 128, [384, 1023], 200, True, 1024),
    (5, 5, 4, 2, 64, 16, [1, 17, 255, 256, 257], [1, 17, 1, 256, 130], True, 512),
]


@pytest.mark.parametrize("seed,B,Hq,Hkv,d,P,lk,lq,causal,maxc", CASES)
def test_paged_prefill_parity(fa, seed, B, Hq, Hkv, d, P, lk, lq, causal, maxc):
    x = inputs.prefill_paged(600 + seed, B, Hq, Hkv, d, P, lk if isinstance(lk, list) else tuple(lk), lq, maxc,
                             causal=causal, spare_pages=3)
    o, lse = _run(fa, x)
    assert fa.debug_read_status() == 0
    o_ref, lse_ref = orc.attn_fwd_paged(x.q, x.kcache, x.vcache, x.block_table, x.seqlens_k, x.cu_seqlens_q,
                                        x.scale, causal)
    check(o, lse, o_ref, lse_ref, what=f"paged prefill case {seed}")


def test_full_prefill_from_cache_equals_varlen_bitwise(fa):
    """With every chunk the whole context (Lq = Lk), the paged kernel reads the same
    keys as the varlen kernel on the gathered K/V and must give identical bits."""
    x = inputs.prefill_paged(700, 3, 4, 2, 128, 32, [200, 777, 64], [200, 777, 64], 800, causal=True)
    o1, l1 = _run(fa, x)
    kk = torch.cat([torch.from_numpy(orc.gather_paged(x.kcache.float().numpy(), x.block_table.numpy(), b, n))
                    for b, n in enumerate(x.lengths_k)]).to(torch.bfloat16)
    vv = torch.cat([torch.from_numpy(orc.gather_paged(x.vcache.float().numpy(), x.block_table.numpy(), b, n))
                    for b, n in enumerate(x.lengths_k)]).to(torch.bfloat16)
    o2, l2 = fa.fwd(x.q.cuda(), kk.cuda(), vv.cuda(), causal=True, scale=x.scale, cu_seqlens=x.cu_seqlens_q.cuda(),
                    max_seqlen=max(x.lengths_q))
    assert fa.debug_read_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_chunked_prefill_large_every_item(fa):
    """B=4, Hq=32, Hkv=8, d=128, 16-token pages, contexts U[4096, 16384], a 2048-query
    chunk at the end of each context, on NaN-filled outputs: every row written, both
    edge rows of every (sequence, head, 128-row tile) and random rows against the oracle."""
    x = inputs.prefill_paged(710, 4, 32, 8, 128, 16, (4096, 16384), 2048, 16384, causal=True)
    Tq = x.q.shape[0]
    o, lse = nan_outputs(x.q.shape, (32, Tq))
    _run(fa, x, out=o, lse=lse)
    assert fa.debug_read_status() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all(), "rows left unwritten (NaN)"
    rng = np.random.default_rng(7)
    smp = [(b, h, i) for b in range(4) for h in range(32) for i in tile_edge_rows(x.lengths_q[b])]
    smp += [(b, int(rng.integers(32)), int(rng.integers(x.lengths_q[b]))) for b in range(4) for _ in range(24)]
    smp = np.array(smp)
    o_ref, lse_ref = orc.attn_fwd_paged(x.q, x.kcache, x.vcache, x.block_table, x.seqlens_k, x.cu_seqlens_q,
                                        x.scale, True, samples=smp)
    cu = x.cu_seqlens_q.tolist()
    rows = torch.as_tensor([cu[b] + i for b, _, i in smp], device="cuda")
    heads = torch.as_tensor(smp[:, 1], device="cuda")
    check(o[rows, heads], lse[heads, rows], o_ref, lse_ref, what="chunked prefill")


def test_bad_table_entry_and_seqlen_are_reported(fa):
    x = inputs.prefill_paged(720, 2, 2, 1, 64, 16, [100, 50], [40, 50], 128, causal=True)
    bt = x.block_table.clone()
    bt[0, 2] = x.kcache.shape[0] + 5                 # outside the pool
    fa.fwd_paged(x.q.cuda(), x.kcache.cuda(), x.vcache.cuda(), bt.cuda(), x.seqlens_k.cuda(),
                 x.cu_seqlens_q.cuda(), 50, causal=True, scale=x.scale)
    assert fa.debug_read_status() == fa.FATTN_ERR_DEVICE_CHECK
    sk = x.seqlens_k.clone()
    sk[1] = 20                                       # fewer context tokens than the chunk's queries
    o, _ = fa.fwd_paged(x.q.cuda(), x.kcache.cuda(), x.vcache.cuda(), x.block_table.cuda(), sk.cuda(),
                        x.cu_seqlens_q.cuda(), 50, causal=True, scale=x.scale)
    assert fa.debug_read_status() == fa.FATTN_ERR_DEVICE_CHECK
    # the valid sequence is still right
    o_ref, lse_ref = orc.attn_fwd_paged(x.q, x.kcache, x.vcache, x.block_table, x.seqlens_k, x.cu_seqlens_q,
                                        x.scale, True)
    check(as_np(o)[:40], None, o_ref[:40], None, what="valid chunk next to a bad one")
