"""Host-side checks of the seeded input generators (no GPU)."""
import torch

from exact_tiled_attention_fattn_gb300 import inputs


def test_varlen_lengths_and_cu_seqlens():
    x = inputs.prefill_varlen(3, (128, 2048), 16, 2, 2, 8, causal=True)
    assert x.lengths == [1402, 1130, 590, 319, 404, 422, 421, 1909, 1501, 245, 2033, 1583, 810, 335, 401, 289]
    cu = x.cu_seqlens.tolist()
    assert cu[0] == 0 and cu[-1] == 13794 == x.q.shape[0]
    assert all(b - a == n for a, b, n in zip(cu[:-1], cu[1:], x.lengths))
    assert x.cu_seqlens.dtype == torch.int32


def test_decode_pool_table_and_sentinels():
    x = inputs.decode_paged(4, 8, 4, 2, 8, 16, (1024, 65536), 65536, spare_pages=3)
    assert x.lengths == [15614, 5751, 8039, 15836, 44685, 10981, 3186, 44902]
    pages = [-(-n // 16) for n in x.lengths]
    used = []
    for b, p in enumerate(pages):
        used.extend(x.block_table[b, :p].tolist())
    assert len(used) == len(set(used)) == sum(pages)            # each page owned once
    pool = x.kcache.shape[0]
    assert pool == sum(pages) + 3
    spare = sorted(set(range(pool)) - set(used))
    assert len(spare) == 3
    for b, p in enumerate(pages):
        assert set(x.block_table[b, p:].tolist()) <= set(spare)
        tail = x.lengths[b] % 16
        last = int(x.block_table[b, p - 1])
        if tail:
            assert torch.all(x.kcache[last, tail:].float() == inputs.SENTINEL)
            assert torch.all(x.vcache[last, tail:].float() == inputs.SENTINEL)
        assert not torch.any(x.kcache[last, :tail if tail else 16].float() == inputs.SENTINEL)
    assert torch.all(x.kcache[spare].float() == inputs.SENTINEL)


def test_same_seed_same_bits():
    a = inputs.prefill_dense(1, 1, 64, 2, 1, 16, causal=True)
    b = inputs.prefill_dense(1, 1, 64, 2, 1, 16, causal=True)
    assert torch.equal(a.q, b.q) and torch.equal(a.k, b.k) and torch.equal(a.v, b.v)
    assert torch.equal(a.q, a.q32.to(torch.bfloat16))


def test_flop_convention():
    x = inputs.prefill_dense(1, 4, 64, 2, 2, 16, causal=True)
    assert x.flops() == 4 * 4 * 2 * 64 * 64 * 16 / 2


def test_paged_prefill_inputs():
    x = inputs.prefill_paged(5, 3, 4, 2, 8, 16, (20, 100), None, 128, spare_pages=2)
    assert len(x.lengths_k) == 3 and all(1 <= lq <= lk for lq, lk in zip(x.lengths_q, x.lengths_k))
    cu = x.cu_seqlens_q.tolist()
    assert cu[0] == 0 and cu[-1] == x.q.shape[0] == sum(x.lengths_q)
    assert x.seqlens_k.tolist() == x.lengths_k
    pages = [-(-n // 16) for n in x.lengths_k]
    used = [p for b, n in enumerate(pages) for p in x.block_table[b, :n].tolist()]
    assert len(set(used)) == len(used) == sum(pages) and x.kcache.shape[0] == sum(pages) + 2
    for b, n in enumerate(x.lengths_k):
        if n % 16:
            last = int(x.block_table[b, pages[b] - 1])
            assert torch.all(x.kcache[last, n % 16:].float() == inputs.SENTINEL)
    y = inputs.prefill_paged(5, 2, 4, 2, 8, 16, [64, 30], 32, 64, causal=True)
    assert y.lengths_q == [32, 30]
    assert y.flops() == 4 * 4 * 8 * (32 * 32 + 32 * 32 / 2 + 30 * 30 / 2)
