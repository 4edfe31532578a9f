"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module draws random numbers and lays them out; it holds none of the attention
arithmetic. Every workload is shaped like the ones on the FlashAttention pages
("FlashAttention" problem statement: Q, K, V are N x d per head; "Flash-Decoding"
and "Paged variants": one query row per sequence against a paged KV cache).

Draw convention (fixed so the oracle and the GPU path see identical bits):
``g = torch.Generator('cpu').manual_seed(seed)``; draws happen in the order
lengths -> page permutation -> Q -> K -> V, each float draw is
``torch.randn(shape, generator=g, dtype=torch.float32)``, integer draws are
``torch.randint(lo, hi + 1, ...)``, and the bf16 copy is ``.to(torch.bfloat16)``
(round to nearest even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = [
    "PrefillInputs",
    "DecodeInputs",
    "prefill_dense",
    "prefill_varlen",
    "decode_paged",
    "tiny_config",
    "causal_mha_config",
    "long_gqa_config",
    "varlen_config",
    "paged_decode_config",
    "SENTINEL",
]

# Value written into KV-cache slots that no sequence owns (tails of last pages,
# spare pages). Exact in bf16 (2^13); any read of it swamps a softmax row.
SENTINEL = 8192.0


@dataclass
class PrefillInputs:
    """Q/K/V for prefill.

    Dense layout: q [B, N, Hq, d], k/v [B, N, Hkv, d].
    Varlen layout: q [T, Hq, d], k/v [T, Hkv, d] with ``cu_seqlens`` int32 [B+1].
    ``q32/k32/v32`` are the fp32 draws; ``q/k/v`` the copies in ``dtype``.
    """

    q32: torch.Tensor
    k32: torch.Tensor
    v32: torch.Tensor
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    causal: bool
    scale: float
    cu_seqlens: torch.Tensor | None = None
    lengths: list[int] | None = None

    @property
    def varlen(self) -> bool:
        return self.cu_seqlens is not None

    @property
    def d(self) -> int:
        return self.q.shape[-1]

    @property
    def hq(self) -> int:
        return self.q.shape[-2]

    @property
    def hkv(self) -> int:
        return self.k.shape[-2]

    @property
    def batch(self) -> int:
        return len(self.lengths) if self.varlen else self.q.shape[0]

    @property
    def max_seqlen(self) -> int:
        return max(self.lengths) if self.varlen else self.q.shape[1]

    def seq_lengths(self) -> list[int]:
        if self.varlen:
            return list(self.lengths)
        return [self.q.shape[1]] * self.q.shape[0]

    def flops(self) -> float:
        """Causal-adjusted attention FLOPs: 4*Hq*N^2*d per sequence, halved when causal."""
        f = sum(4.0 * self.hq * n * n * self.d for n in self.seq_lengths())
        return f / 2 if self.causal else f


@dataclass
class DecodeInputs:
    """One query token per sequence against a paged KV cache.

    q [B, Hq, d]; kcache/vcache [num_pages, page_size, Hkv, d];
    block_table int32 [B, max_pages_per_seq]; seqlens int32 [B].
    Slots no sequence owns hold ``SENTINEL``. Unused block-table entries point
    at spare pages (all ``SENTINEL``) when ``spare_pages > 0``, else at page 0.
    """

    q32: torch.Tensor
    q: torch.Tensor
    kcache: torch.Tensor
    vcache: torch.Tensor
    block_table: torch.Tensor
    seqlens: torch.Tensor
    page_size: int
    scale: float
    spare_pages: int = 0
    lengths: list[int] = field(default_factory=list)

    @property
    def d(self) -> int:
        return self.q.shape[-1]

    @property
    def hq(self) -> int:
        return self.q.shape[1]

    @property
    def hkv(self) -> int:
        return self.kcache.shape[2]

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def max_pages_per_seq(self) -> int:
        return self.block_table.shape[1]

    def kv_bytes(self) -> int:
        """Bytes of K and V the sequences own (what a decode step must read)."""
        elem = self.kcache.element_size()
        return 2 * sum(self.lengths) * self.hkv * self.d * elem


def _randn(g: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32)


def prefill_dense(seed: int, B: int, N: int, Hq: int, Hkv: int, d: int, causal: bool,
                  dtype: torch.dtype = torch.bfloat16, scale: float | None = None) -> PrefillInputs:
    """Dense [B, N, H, d] Q/K/V, iid N(0, 1)."""
    g = torch.Generator("cpu").manual_seed(seed)
    q32 = _randn(g, (B, N, Hq, d))
    k32 = _randn(g, (B, N, Hkv, d))
    v32 = _randn(g, (B, N, Hkv, d))
    s = 1.0 / math.sqrt(d) if scale is None else scale
    return PrefillInputs(q32, k32, v32, q32.to(dtype), k32.to(dtype), v32.to(dtype), causal, s)


def prefill_varlen(seed: int, lengths_range: tuple[int, int] | None, n_seqs: int, Hq: int, Hkv: int,
                   d: int, causal: bool, dtype: torch.dtype = torch.bfloat16,
                   scale: float | None = None, lengths: list[int] | None = None) -> PrefillInputs:
    """Sequences packed back to back, [T, H, d] with int32 cu_seqlens [n_seqs + 1].

    Lengths are drawn uniform in ``lengths_range`` (inclusive) unless given.
    """
    g = torch.Generator("cpu").manual_seed(seed)
    if lengths is None:
        lo, hi = lengths_range
        lengths = torch.randint(lo, hi + 1, (n_seqs,), generator=g).tolist()
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    T = cu[-1]
    q32 = _randn(g, (T, Hq, d))
    k32 = _randn(g, (T, Hkv, d))
    v32 = _randn(g, (T, Hkv, d))
    s = 1.0 / math.sqrt(d) if scale is None else scale
    return PrefillInputs(q32, k32, v32, q32.to(dtype), k32.to(dtype), v32.to(dtype), causal, s,
                         cu_seqlens=torch.tensor(cu, dtype=torch.int32), lengths=[int(n) for n in lengths])


def _page_pool(g: torch.Generator, lengths: list[int], page_size: int, max_context: int, spare_pages: int):
    """Block table over a pool of exactly the pages ``lengths`` need plus ``spare_pages``,
    handed out through a random permutation (one draw from ``g``). Table entries past a
    sequence's pages point at spare pages (round robin) or at page 0 when there are none."""
    B = len(lengths)
    pages = [(n + page_size - 1) // page_size for n in lengths]
    used = sum(pages)
    pool = used + spare_pages
    perm = torch.randperm(pool, generator=g)
    max_pages = (max_context + page_size - 1) // page_size
    table = torch.empty((B, max_pages), dtype=torch.int32)
    spare = perm[used:]
    off = 0
    for b in range(B):
        table[b, : pages[b]] = perm[off: off + pages[b]].to(torch.int32)
        rest = max_pages - pages[b]
        if rest > 0:
            if spare_pages > 0:
                idx = torch.arange(rest) % spare_pages
                table[b, pages[b]:] = spare[idx].to(torch.int32)
            else:
                table[b, pages[b]:] = 0
        off += pages[b]
    return table, pages, pool, spare


def _fill_unowned(k32, v32, table, pages, lengths, spare, page_size: int):
    """Slots that belong to no sequence (spare pages, the tail of each last page) get SENTINEL."""
    if len(spare) > 0:
        k32[spare] = SENTINEL
        v32[spare] = SENTINEL
    for b, n in enumerate(lengths):
        tail = n % page_size
        if tail:
            last = int(table[b, pages[b] - 1])
            k32[last, tail:] = SENTINEL
            v32[last, tail:] = SENTINEL


def decode_paged(seed: int, B: int, Hq: int, Hkv: int, d: int, page_size: int,
                 context_range: tuple[int, int] | None, max_context: int,
                 spare_pages: int = 0, dtype: torch.dtype = torch.bfloat16,
                 scale: float | None = None, lengths: list[int] | None = None) -> DecodeInputs:
    """Paged decode inputs: contexts uniform in ``context_range`` (inclusive).

    The pool holds exactly the pages the sequences need plus ``spare_pages``;
    pages are handed out through a random permutation of the pool, so logical
    page p of sequence b lives at ``block_table[b, p]``.
    """
    g = torch.Generator("cpu").manual_seed(seed)
    if lengths is None:
        lo, hi = context_range
        lengths = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    lengths = [int(n) for n in lengths]
    assert len(lengths) == B and max(lengths) <= max_context
    table, pages, pool, spare = _page_pool(g, lengths, page_size, max_context, spare_pages)
    q32 = _randn(g, (B, Hq, d))
    k32 = _randn(g, (pool, page_size, Hkv, d))
    v32 = _randn(g, (pool, page_size, Hkv, d))
    _fill_unowned(k32, v32, table, pages, lengths, spare, page_size)
    s = 1.0 / math.sqrt(d) if scale is None else scale
    return DecodeInputs(q32, q32.to(dtype), k32.to(dtype), v32.to(dtype), table,
                        torch.tensor(lengths, dtype=torch.int32), page_size, s, spare_pages, lengths)


@dataclass
class PagedPrefillInputs:
    """Multi-token queries against a paged KV cache (chunked prefill).

    Sequence b owns context tokens [0, lengths_k[b]) in the cache; its
    lengths_q[b] <= lengths_k[b] queries are the last lengths_q[b] of them,
    packed back to back in q [Tq, Hq, d] with int32 cu_seqlens_q [B + 1].
    kcache/vcache [num_pages, page_size, Hkv, d]; block_table int32
    [B, max_pages_per_seq]; seqlens_k int32 [B]. Slots no sequence owns hold
    ``SENTINEL``.
    """

    q32: torch.Tensor
    q: torch.Tensor
    kcache: torch.Tensor
    vcache: torch.Tensor
    block_table: torch.Tensor
    seqlens_k: torch.Tensor
    cu_seqlens_q: torch.Tensor
    page_size: int
    causal: bool
    scale: float
    lengths_q: list[int] = field(default_factory=list)
    lengths_k: list[int] = field(default_factory=list)
    spare_pages: int = 0

    @property
    def d(self) -> int:
        return self.q.shape[-1]

    @property
    def hq(self) -> int:
        return self.q.shape[1]

    @property
    def hkv(self) -> int:
        return self.kcache.shape[2]

    @property
    def batch(self) -> int:
        return len(self.lengths_q)

    @property
    def max_pages_per_seq(self) -> int:
        return self.block_table.shape[1]

    def flops(self) -> float:
        """4*d FLOPs per (query, key) pair of each head: Lq*Lk pairs, or with the causal
        rule Lq*(Lk - Lq) + Lq^2/2 (the dense convention for the square part)."""
        pairs = 0.0
        for lq, lk in zip(self.lengths_q, self.lengths_k):
            pairs += lq * (lk - lq) + lq * lq / 2 if self.causal else lq * lk
        return 4.0 * self.hq * self.d * pairs


def prefill_paged(seed: int, B: int, Hq: int, Hkv: int, d: int, page_size: int,
                  lengths_k: list[int] | tuple[int, int], lengths_q: list[int] | int | None,
                  max_context: int, causal: bool = True, spare_pages: int = 0,
                  dtype: torch.dtype = torch.bfloat16, scale: float | None = None) -> PagedPrefillInputs:
    """Paged-prefill inputs. ``lengths_k``: a list, or a range (lo, hi) drawn uniform
    inclusive; ``lengths_q``: a list, an int (chunk of min(int, Lk) queries per
    sequence) or None (each drawn uniform in [1, Lk]). Draw order: context lengths,
    query lengths, page permutation, Q, K, V."""
    g = torch.Generator("cpu").manual_seed(seed)
    if isinstance(lengths_k, tuple):
        lo, hi = lengths_k
        lengths_k = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    lengths_k = [int(n) for n in lengths_k]
    if lengths_q is None:
        lengths_q = [int(torch.randint(1, n + 1, (1,), generator=g)) if n > 0 else 0 for n in lengths_k]
    elif isinstance(lengths_q, int):
        lengths_q = [min(lengths_q, n) for n in lengths_k]
    lengths_q = [int(n) for n in lengths_q]
    assert len(lengths_k) == len(lengths_q) == B and max(lengths_k) <= max_context
    assert all(0 <= lq <= lk for lq, lk in zip(lengths_q, lengths_k))
    table, pages, pool, spare = _page_pool(g, lengths_k, page_size, max_context, spare_pages)
    cu = [0]
    for n in lengths_q:
        cu.append(cu[-1] + n)
    q32 = _randn(g, (cu[-1], Hq, d))
    k32 = _randn(g, (pool, page_size, Hkv, d))
    v32 = _randn(g, (pool, page_size, Hkv, d))
    _fill_unowned(k32, v32, table, pages, lengths_k, spare, page_size)
    s = 1.0 / math.sqrt(d) if scale is None else scale
    return PagedPrefillInputs(q32, q32.to(dtype), k32.to(dtype), v32.to(dtype), table,
                              torch.tensor(lengths_k, dtype=torch.int32), torch.tensor(cu, dtype=torch.int32),
                              page_size, causal, s, lengths_q, lengths_k, spare_pages)


@dataclass
class Fp8Inputs:
    """Dense FP8 (E4M3) prefill inputs with per-tensor descale factors:
    x = descale * e4m3(x8). q8 [B, N, Hq, d], k8/v8 [B, N, Hkv, d] as uint8 codes."""

    q8: torch.Tensor
    k8: torch.Tensor
    v8: torch.Tensor
    q_descale: float
    k_descale: float
    v_descale: float
    causal: bool
    scale: float

    def flops(self) -> float:
        B, N, Hq, d = self.q8.shape
        f = 4.0 * B * Hq * N * N * d
        return f / 2 if self.causal else f


def prefill_fp8(seed: int, B: int, N: int, Hq: int, Hkv: int, d: int, causal: bool,
                scale: float | None = None) -> Fp8Inputs:
    """Q, K, V iid N(0, 1) (draw order Q, K, V), each quantized to E4M3 with the
    per-tensor descale amax / 448 (the largest finite E4M3 value)."""
    g = torch.Generator("cpu").manual_seed(seed)
    xs = [_randn(g, (B, N, Hq, d)), _randn(g, (B, N, Hkv, d)), _randn(g, (B, N, Hkv, d))]
    codes, descales = [], []
    for x in xs:
        ds = float(x.abs().max()) / 448.0
        codes.append((x / ds).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8))
        descales.append(ds)
    s = 1.0 / math.sqrt(d) if scale is None else scale
    return Fp8Inputs(codes[0], codes[1], codes[2], descales[0], descales[1], descales[2], causal, s)


# ---- the five workloads (shapes of the pages' problems; sizes fixed here) ----

def tiny_config(dtype: torch.dtype = torch.float32) -> PrefillInputs:
    """Single head, B=1, N=256, d=64, non-causal, seed 0 (fp32 draws + a copy in ``dtype``)."""
    return prefill_dense(0, 1, 256, 1, 1, 64, causal=False, dtype=dtype, scale=1.0 / 8.0)


def causal_mha_config() -> PrefillInputs:
    """Causal MHA prefill: B=4, Hq=Hkv=32, N=4096, d=128, bf16, seed 1."""
    return prefill_dense(1, 4, 4096, 32, 32, 128, causal=True, scale=1.0 / math.sqrt(128))


def long_gqa_config() -> PrefillInputs:
    """Long-context GQA causal prefill: B=1, Hq=32, Hkv=8, N=32768, d=128, bf16, seed 2."""
    return prefill_dense(2, 1, 32768, 32, 8, 128, causal=True, scale=1.0 / math.sqrt(128))


def varlen_config() -> PrefillInputs:
    """16 packed sequences, lengths U[128, 2048] (seed 3), Hq=Hkv=16, d=64, causal, bf16."""
    return prefill_varlen(3, (128, 2048), 16, 16, 16, 64, causal=True, scale=1.0 / 8.0)


def paged_decode_config(spare_pages: int = 0) -> DecodeInputs:
    """Batch 8, Hq=32, Hkv=8, d=128, contexts U[1024, 65536] (seed 4), 16-token pages."""
    return decode_paged(4, 8, 32, 8, 128, 16, (1024, 65536), 65536, spare_pages=spare_pages,
                        scale=1.0 / math.sqrt(128))
