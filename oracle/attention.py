"""CPU fp64 oracle for exact tiled attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The CUDA library never calls it and shares no code with it.

Sources (three web pages on one subject):
  [FA-LLM]  "FlashAttention", LLM-inference guide, chapter 10
            (shubhamtatvamasi.com/llm-inference/flash-attention):
            the attention formula; "The trick: tiles and an online softmax"
            (update rule and finalisation O'/l'); "Decode is a different problem"
            and "Flash-Decoding: split the KV cache to fill the GPU"
            (split-K partials merged with the same rule); the family table rows
            "Flash-Decoding" and "Paged variants"; the live-demo caption on the
            causal mask ("tiles above the diagonal are never touched").
  [FA-PAPER] "FlashAttention, explained" (vibeengines.com/paper/flash-attention):
            the worked example (row [2,1,3,0] in blocks [2,1],[3,0]);
            "The forward pass", steps 1-5 (normalised update form, saved
            statistics l and m).
  [CUDA-OPS] "Attention" CUDA operations guide (rightnowai.co): K/V heads shared
            by several Q heads (GQA/MQA); non-contiguous (paged) KV allocation.
  [FA-PAPER] "The backward pass recomputes instead of reading": P rebuilt from
            the saved statistics; dV += P^T dO, dP = dO V^T,
            dS = P o (dP - D) with D = rowsum(dO o O), dQ += dS K, dK += dS^T Q.
  [FA-PAPER] "Block-sparse FlashAttention": a fixed mask over blocks; every
            block that is zero in the mask is skipped, i.e. its scores are
            excluded from the softmax (an approximation of dense attention).

Everything is computed in float64 from inputs that the caller widens exactly
(bf16 and fp32 values are representable in fp64). The primary mode is the plain
definition O = softmax(Q K^T * scale + M) V; the blocked modes restate the
online-softmax rule and exist to pin the definition against the pages' worked
example.

Readings taken where the pages are silent:
  * statistics are exported as one natural-log logsumexp per row,
    lse = m + ln(l), over the scaled scores;
  * causal alignment is bottom-right: key j is allowed for query i when
    j <= i + (Nk - Nq) (identical to top-left for prefill, where Nq = Nk);
  * query head h reads KV head h // (Hq / Hkv);
  * a row with no allowed key has O = 0 and lse = -inf; a partial with
    lse = -inf carries no weight in a merge;
  * backward: the page writes the gradient steps for S = Q K^T; with the
    scale, S = scale * Q K^T, so dQ = scale * dS K and dK = scale * dS^T Q
    (chain rule); GQA: a KV head's dK, dV sum over the query heads sharing it;
  * decode splits: with P_b = ceil(L_b / page_size) pages and
    C = ceil(max_pages_per_seq / num_splits) pages per split, split s of
    sequence b covers tokens [s*C*page_size, min(L_b, (s+1)*C*page_size)),
    empty when s*C >= P_b.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "attention_definition",
    "attention_weights",
    "attn_fwd",
    "attn_fwd_rows",
    "attn_fwd_block_sparse",
    "block_sparse_allowed",
    "softmax_row_blocked",
    "attention_blocked",
    "attention_blocked_normalised",
    "gather_paged",
    "decode_paged",
    "attn_fwd_paged",
    "attn_bwd",
    "attn_bwd_rows",
    "attn_fwd_masked",
    "e4m3_to_f64",
    "attn_fwd_fp8",
    "decode_split_ranges",
    "decode_partials",
    "merge_partials",
]


def _f64(x) -> np.ndarray:
    """Widen a numpy array or a torch CPU tensor (any float dtype) to fp64 exactly."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()  # bf16 -> fp32 is exact
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# The plain definition ([FA-LLM] formula: O = softmax(QK^T/sqrt(d) + M) V)
# --------------------------------------------------------------------------

def _allowed(rows: np.ndarray, n_keys: int, n_queries: int, causal: bool) -> np.ndarray:
    """Boolean [len(rows), n_keys]: which keys each query row may attend to.

    Causal mask M = -inf above the diagonal ([FA-LLM] formula and live-demo
    caption), aligned bottom-right so the last query sees every key.
    """
    j = np.arange(n_keys)[None, :]
    if not causal:
        return np.ones((len(rows), n_keys), dtype=bool)
    return j <= (rows[:, None] + (n_keys - n_queries))


def attention_weights(q, k, scale: float, causal: bool = False, rows=None) -> np.ndarray:
    """Softmax weights P = softmax(scale * q k^T + M) for one head, fp64 [r, Nk].

    Safe softmax: subtract the row maximum before exponentiating ([FA-LLM]
    "The trick", finalisation paragraph). Fully masked rows get all-zero weights.
    """
    q = _f64(q)
    k = _f64(k)
    nq, nk = q.shape[0], k.shape[0]
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    s = scale * (q[rows] @ k.T)
    ok = _allowed(rows, nk, nq, causal)
    s = np.where(ok, s, -np.inf)
    m = s.max(axis=1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.where(ok, np.exp(s - m_safe[:, None]), 0.0)
    l = w.sum(axis=1)
    return np.where(l[:, None] > 0, w / np.where(l > 0, l, 1.0)[:, None], 0.0)


def attention_definition(q, k, v, scale: float, causal: bool = False, rows=None, allowed=None, bias=None):
    """Exact attention for one head by the definition, fp64.

    q [Nq, d], k [Nk, d], v [Nk, dv]. Returns (O [r, dv], lse [r]) for the
    requested query rows (all by default), lse = m + ln(l) of the scaled,
    masked scores (natural log). ``allowed`` (bool [Nq, Nk]) further restricts
    which keys each query sees (M = -inf where it is False); ``bias`` ([Nq, Nk])
    is the additive mask M of the formula, added to the scaled scores.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    nq, nk = q.shape[0], k.shape[0]
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    if nk == 0:                                        # no key at all: O = 0, lse = -inf
        return np.zeros((len(rows), v.shape[-1])), np.full(len(rows), -np.inf)
    s = scale * (q[rows] @ k.T)
    ok = _allowed(rows, nk, nq, causal)
    if allowed is not None:
        ok = ok & np.asarray(allowed, dtype=bool)[rows]
    if bias is not None:                               # softmax(scale Q K^T + M)
        s = s + _f64(bias)[rows]
        ok = ok & np.isfinite(s)                       # M = -inf removes the key
    s = np.where(ok, s, -np.inf)
    m = s.max(axis=1)                                  # running-max target m
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(ok, np.exp(s - m_safe[:, None]), 0.0)  # e^{s_j - m}
    l = w.sum(axis=1)                                  # l = sum_j e^{s_j - m}
    o = (w @ v) / np.where(finite, l, 1.0)[:, None]    # O = sum_j (e^{s_j-m}/l) v_j
    o = np.where(finite[:, None], o, 0.0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, l, 1.0)), -np.inf)
    return o, lse


def attn_fwd(q, k, v, scale: float, causal: bool, cu_seqlens=None):
    """Full prefill output by the definition.

    Dense: q [B, N, Hq, d], k/v [B, N, Hkv, d] -> O [B, N, Hq, d], lse [B, Hq, N].
    Varlen: q [T, Hq, d], k/v [T, Hkv, d], cu_seqlens [B+1] -> O [T, Hq, d],
    lse [Hq, T]; no attention across sequence boundaries.
    Query head h reads KV head h // (Hq/Hkv) ([CUDA-OPS] shared K/V heads).
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    if cu_seqlens is None:
        B, N, Hq, _ = q.shape
        Hkv = k.shape[2]
        g = Hq // Hkv
        o = np.zeros(q.shape[:3] + (v.shape[-1],))
        lse = np.zeros((B, Hq, N))
        for b in range(B):
            for h in range(Hq):
                o[b, :, h], lse[b, h] = attention_definition(q[b, :, h], k[b, :, h // g],
                                                             v[b, :, h // g], scale, causal)
        return o, lse
    cu = [int(x) for x in np.asarray(cu_seqlens)]
    T, Hq, _ = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    o = np.zeros((T, Hq, v.shape[-1]))
    lse = np.full((Hq, T), -np.inf)
    for b in range(len(cu) - 1):
        a, e = cu[b], cu[b + 1]
        if e == a:
            continue
        for h in range(Hq):
            o[a:e, h], lse[h, a:e] = attention_definition(q[a:e, h], k[a:e, h // g],
                                                          v[a:e, h // g], scale, causal)
    return o, lse


def attn_fwd_masked(q, k, v, scale: float, causal: bool, mask, rows=None):
    """Prefill with an additive mask, by the definition ([FA-LLM] formula
    O = softmax(Q K^T / sqrt(d) + M) V).

    Dense q [B, N, Hq, d], k/v [B, N, Hkv, d]; mask broadcastable to
    [B, Hq, N, N] (leading dimensions of size 1 are shared), added to the scaled
    scores; entries of -inf remove keys, and with ``causal`` the causal rule
    applies on top. A row left with no key has O = 0, lse = -inf.
    Returns O [B, N, Hq, d], lse [B, Hq, N]; with rows (int [n, 3] of
    (b, h, i)) only those: O [n, d], lse [n].
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    m = _f64(mask)
    B, N, Hq, _ = q.shape
    g = Hq // k.shape[2]
    mb = lambda b, h: m[b if m.shape[0] > 1 else 0, h if m.shape[1] > 1 else 0]
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        o = np.zeros((len(rows), v.shape[-1]))
        lse = np.zeros(len(rows))
        for b, h in sorted({(int(b), int(h)) for b, h, _ in rows}):
            idx = np.nonzero((rows[:, 0] == b) & (rows[:, 1] == h))[0]
            o[idx], lse[idx] = attention_definition(q[b, :, h], k[b, :, h // g], v[b, :, h // g], scale, causal,
                                                    rows=rows[idx, 2], bias=mb(b, h))
        return o, lse
    o = np.zeros(q.shape[:3] + (v.shape[-1],))
    lse = np.zeros((B, Hq, N))
    for b in range(B):
        for h in range(Hq):
            o[b, :, h], lse[b, h] = attention_definition(q[b, :, h], k[b, :, h // g], v[b, :, h // g], scale,
                                                         causal, bias=mb(b, h))
    return o, lse


def e4m3_to_f64(codes) -> np.ndarray:
    """Decode FP8 E4M3 bytes (the 'fn' variant: 1 sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits, subnormals at exponent 0, no infinities, S.1111.111
    = NaN) to float64, from the bit layout."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** (1 - 7), (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7))
    val = np.where((e == 0xF) & ((c & 0x7) == 0x7), np.nan, val)
    return sign * val


def attn_fwd_fp8(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float, scale: float, causal: bool,
                 rows=None):
    """FP8 prefill ([FA-LLM] family table, FlashAttention-3: FP8 inputs): the
    definition on the dequantized inputs Q = q_descale * dec(q8), K, V likewise.
    q8 [B, N, Hq, d], k8/v8 [B, N, Hkv, d] E4M3 bytes (uint8). Returns O, lse as
    attn_fwd, or at sampled rows (int [n, 3] of (b, h, i))."""
    q = e4m3_to_f64(q8) * q_descale
    k = e4m3_to_f64(k8) * k_descale
    v = e4m3_to_f64(v8) * v_descale
    if rows is None:
        return attn_fwd(q, k, v, scale, causal)
    return attn_fwd_rows(q, k, v, scale, causal, rows)


def attn_fwd_rows(q, k, v, scale: float, causal: bool, samples, cu_seqlens=None):
    """Definition evaluated only at sampled output rows (for sizes too big to do whole).

    samples: int array [n, 3] of (sequence b, query head h, row i within the
    sequence). Returns (O [n, d], lse [n]).
    """
    samples = np.asarray(samples, dtype=np.int64)
    if cu_seqlens is None:
        Hq, Hkv = q.shape[2], k.shape[2]
        starts = None
    else:
        Hq, Hkv = q.shape[1], k.shape[1]
        starts = [int(x) for x in np.asarray(cu_seqlens)]
    g = Hq // Hkv
    dv = v.shape[-1]
    o = np.zeros((len(samples), dv))
    lse = np.zeros(len(samples))
    # group rows by (b, h) so each head's K/V is widened once
    keys = sorted({(int(b), int(h)) for b, h, _ in samples})
    for b, h in keys:
        idx = np.nonzero((samples[:, 0] == b) & (samples[:, 1] == h))[0]
        rows = samples[idx, 2]
        if starts is None:
            qh, kh, vh = q[b, :, h], k[b, :, h // g], v[b, :, h // g]
        else:
            a, e = starts[b], starts[b + 1]
            qh, kh, vh = q[a:e, h], k[a:e, h // g], v[a:e, h // g]
        o[idx], lse[idx] = attention_definition(qh, kh, vh, scale, causal, rows=rows)
    return o, lse


def block_sparse_allowed(block_mask_2d, nq: int, nk: int, block: int) -> np.ndarray:
    """Expand a [ceil(nq/block), ceil(nk/block)] block mask to a key-visibility
    matrix [nq, nk]: key j is visible to query i iff block (i // block, j // block)
    is non-zero ("Block-sparse FlashAttention": zero blocks are skipped)."""
    bm = np.asarray(block_mask_2d) != 0
    i = np.arange(nq) // block
    j = np.arange(nk) // block
    return bm[i[:, None], j[None, :]]


def attn_fwd_block_sparse(q, k, v, scale: float, causal: bool, block_mask, block: int, rows=None):
    """Dense-layout prefill restricted by a block mask.

    q [B, N, Hq, d], k/v [B, N, Hkv, d]; block_mask [Hm, ceil(N/block),
    ceil(N/block)] with Hm = 1 (shared) or Hq (per query head). Visible keys are
    those the causal rule allows in a non-zero block; a row with none has O = 0,
    lse = -inf. Returns O [B, N, Hq, d], lse [B, Hq, N] (or, with ``rows`` as an
    int array [n, 3] of (b, h, i), O [n, d] and lse [n]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    bm = np.asarray(block_mask)
    B, N, Hq, _ = q.shape
    g = Hq // k.shape[2]
    if rows is None:
        o = np.zeros(q.shape[:3] + (v.shape[-1],))
        lse = np.zeros((B, Hq, N))
        for h in range(Hq):
            allow = block_sparse_allowed(bm[h % bm.shape[0]], N, N, block)
            for b in range(B):
                o[b, :, h], lse[b, h] = attention_definition(q[b, :, h], k[b, :, h // g], v[b, :, h // g],
                                                             scale, causal, allowed=allow)
        return o, lse
    rows = np.asarray(rows, dtype=np.int64)
    o = np.zeros((len(rows), v.shape[-1]))
    lse = np.zeros(len(rows))
    for b, h in sorted({(int(b), int(h)) for b, h, _ in rows}):   # each head's visibility formed once
        idx = np.nonzero((rows[:, 0] == b) & (rows[:, 1] == h))[0]
        allow = block_sparse_allowed(bm[h % bm.shape[0]], N, N, block)
        o[idx], lse[idx] = attention_definition(q[b, :, h], k[b, :, h // g], v[b, :, h // g], scale, causal,
                                                rows=rows[idx, 2], allowed=allow)
    return o, lse


# --------------------------------------------------------------------------
# The online-softmax rule, block by block ([FA-LLM] "The trick"; [FA-PAPER]
# worked example and "The forward pass" step 4). Used to pin the definition.
# --------------------------------------------------------------------------

def softmax_row_blocked(scores, block: int):
    """Softmax of one score row visited in blocks of ``block`` entries.

    Running state: m (max so far), l (sum of e^{s - m}); on each block
    m' = max(m, max_j s_j), l' = l e^{m - m'} + sum_j e^{s_j - m'}.
    The weights are e^{s_j - m_final} / l_final.
    Returns (m, l, weights, history) with history = [(m, l) after each block].
    """
    s = np.asarray(scores, dtype=np.float64)
    m, l = -np.inf, 0.0
    history = []
    for start in range(0, len(s), block):
        blk = s[start:start + block]
        m_new = max(m, float(blk.max()))
        l = l * math.exp(m - m_new) + float(np.exp(blk - m_new).sum())
        m = m_new
        history.append((m, l))
    weights = np.exp(s - m) / l
    return m, l, weights, history


def _blocked_head(q, k, v, scale, causal, block, normalised):
    """One head, keys visited in blocks; the per-row state (m, l, O) is rescaled per block."""
    nq, nk = q.shape[0], k.shape[0]
    dv = v.shape[1]
    m = np.full(nq, -np.inf)
    l = np.zeros(nq)
    o = np.zeros((nq, dv))
    rows = np.arange(nq)
    for start in range(0, nk, block):
        kj, vj = k[start:start + block], v[start:start + block]
        s = scale * (q @ kj.T)
        ok = _allowed(rows, nk, nq, causal)[:, start:start + block]
        s = np.where(ok, s, -np.inf)
        m_new = np.maximum(m, s.max(axis=1))
        m_use = np.where(np.isfinite(m_new), m_new, 0.0)
        alpha = np.where(np.isfinite(m), np.exp(m - m_use), 0.0)   # e^{m - m'}
        p = np.where(ok, np.exp(s - m_use[:, None]), 0.0)          # e^{s_j - m'}
        l_new = l * alpha + p.sum(axis=1)
        if normalised:
            # "The forward pass" step 4: O kept divided by l; rescale old O by
            # l_old * e^{m_old - m_new}, add P V, divide by the new l.
            num = (l * alpha)[:, None] * o + p @ vj
            o = np.where(l_new[:, None] > 0, num / np.where(l_new > 0, l_new, 1.0)[:, None], 0.0)
        else:
            # "The trick": O' = O e^{m - m'} + sum_j e^{s_j - m'} v_j, divided once at the end.
            o = o * alpha[:, None] + p @ vj
        m, l = m_new, l_new
    if not normalised:
        o = np.where(l[:, None] > 0, o / np.where(l > 0, l, 1.0)[:, None], 0.0)
    lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse


def attention_blocked(q, k, v, scale: float, causal: bool, block: int):
    """One head with the unnormalised update rule (divide by l once at the end)."""
    return _blocked_head(_f64(q), _f64(k), _f64(v), scale, causal, block, normalised=False)


def attention_blocked_normalised(q, k, v, scale: float, causal: bool, block: int):
    """One head with the normalised update form (O divided by the new l every block)."""
    return _blocked_head(_f64(q), _f64(k), _f64(v), scale, causal, block, normalised=True)


# --------------------------------------------------------------------------
# Paged decode and the split-K merge ([FA-LLM] "Decode is a different
# problem", "Flash-Decoding", "Paged variants"; [CUDA-OPS] paged KV)
# --------------------------------------------------------------------------

def gather_paged(cache, block_table, b: int, length: int):
    """Logical [length, Hkv, d] K or V of sequence b, read through the block table, fp64.

    Token t lives in page block_table[b, t // page_size], slot t % page_size.
    The gather happens in the cache's own dtype; only the gathered rows are widened.
    """
    table = np.asarray(block_table)
    page_size = cache.shape[1]
    n_pages = -(-length // page_size)
    pages = [int(p) for p in table[b, :n_pages]]
    rows = cache[pages]                       # [n_pages, page_size, Hkv, d]
    rows = rows.reshape((n_pages * page_size,) + tuple(cache.shape[2:]))
    return _f64(rows[:length])


def decode_paged(q, kcache, vcache, block_table, seqlens, scale: float):
    """One query token per sequence against its whole paged context.

    q [B, Hq, d] -> O [B, Hq, d], lse [B, Hq]. The single query is the last
    position, so bottom-right causal alignment lets it see all L_b keys.
    """
    q = _f64(q)
    lens = [int(x) for x in np.asarray(seqlens)]
    B, Hq, _ = q.shape
    Hkv = kcache.shape[2]
    g = Hq // Hkv
    o = np.zeros((B, Hq, vcache.shape[-1]))
    lse = np.zeros((B, Hq))
    for b in range(B):
        kb = gather_paged(kcache, block_table, b, lens[b])
        vb = gather_paged(vcache, block_table, b, lens[b])
        for h in range(Hq):
            ob, lb = attention_definition(q[b, h][None, :], kb[:, h // g], vb[:, h // g], scale, causal=True)
            o[b, h], lse[b, h] = ob[0], lb[0]
    return o, lse


def attn_fwd_paged(q, kcache, vcache, block_table, seqlens_k, cu_seqlens_q, scale: float, causal: bool,
                   samples=None):
    """Multi-token queries against a paged context (chunked prefill), by the definition.

    Sequence b's queries q[cu[b]:cu[b+1]] (Lq of them) are the last Lq positions
    of its Lk = seqlens_k[b] context tokens, read through the block table
    ([FA-LLM] "Paged variants"; [CUDA-OPS] non-contiguous KV). With causal, query
    i of the chunk sees keys j <= i + (Lk - Lq) (bottom-right alignment).
    q [Tq, Hq, d] -> O [Tq, Hq, d], lse [Hq, Tq]; or, with samples (int
    [n, 3] of (b, h, i)), O [n, d] and lse [n] at those rows only.
    """
    q = _f64(q)
    cu = [int(x) for x in np.asarray(cu_seqlens_q)]
    lens_k = [int(x) for x in np.asarray(seqlens_k)]
    Tq, Hq, _ = q.shape
    g = Hq // kcache.shape[2]
    dv = vcache.shape[-1]
    if samples is not None:
        samples = np.asarray(samples, dtype=np.int64)
        o = np.zeros((len(samples), dv))
        lse = np.zeros(len(samples))
        for b in sorted({int(x) for x in samples[:, 0]}):
            kb = gather_paged(kcache, block_table, b, lens_k[b])
            vb = gather_paged(vcache, block_table, b, lens_k[b])
            qb = q[cu[b]:cu[b + 1]]
            for n in np.nonzero(samples[:, 0] == b)[0]:
                h, i = int(samples[n, 1]), int(samples[n, 2])
                ob, lb = attention_definition(qb[:, h], kb[:, h // g], vb[:, h // g], scale, causal, rows=[i])
                o[n], lse[n] = ob[0], lb[0]
        return o, lse
    o = np.zeros((Tq, Hq, dv))
    lse = np.full((Hq, Tq), -np.inf)
    for b in range(len(cu) - 1):
        a, e = cu[b], cu[b + 1]
        if e == a:
            continue
        kb = gather_paged(kcache, block_table, b, lens_k[b])
        vb = gather_paged(vcache, block_table, b, lens_k[b])
        for h in range(Hq):
            o[a:e, h], lse[h, a:e] = attention_definition(q[a:e, h], kb[:, h // g], vb[:, h // g], scale, causal)
    return o, lse


def attn_bwd(q, k, v, do, scale: float, causal: bool):
    """Gradients of L = sum(O o dO) for dense q [B, N, Hq, d], k/v [B, N, Hkv, d], fp64.

    Per (b, h), with whole matrices as the one block ([FA-PAPER] "The backward
    pass recomputes instead of reading"): P = softmax(scale Q K^T + M),
    O = P V, D = rowsum(dO o O), dV = P^T dO, dP = dO V^T, dS = P o (dP - D),
    dQ = scale dS K, dK = scale dS^T Q. Returns (dq, dk, dv) in the input layouts.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    do = _f64(do)
    B, N, Hq, _ = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            kh, vh = k[b, :, h // g], v[b, :, h // g]
            p = attention_weights(q[b, :, h], kh, scale, causal)      # [N, N]
            o = p @ vh
            dOh = do[b, :, h]
            dmat = np.sum(dOh * o, axis=1)                           # D = rowsum(dO o O)
            dv[b, :, h // g] += p.T @ dOh                            # dV = P^T dO
            dp = dOh @ vh.T                                          # dP = dO V^T
            ds = p * (dp - dmat[:, None])                            # dS = P o (dP - D)
            dq[b, :, h] = scale * (ds @ kh)                          # dQ = scale dS K
            dk[b, :, h // g] += scale * (ds.T @ q[b, :, h])          # dK = scale dS^T Q
    return dq, dk, dv


def attn_bwd_rows(q, k, v, do, scale: float, causal: bool, dq_rows, dkv_rows):
    """Selected rows of the gradients of attn_bwd, for sizes too large to form whole.

    Same steps as attn_bwd ([FA-PAPER] "The backward pass recomputes instead of
    reading"), per (b, query head) with the whole head as one block: P, O = P V and
    D = rowsum(dO o O) are formed for the head, then only the requested rows of
    dQ = scale dS K (rows of dS) and the requested key rows of dV = P^T dO and
    dK = scale dS^T Q (columns of P and dS) are taken.
    dq_rows: int [n, 3] of (b, query head h, row i) -> dQ[b, i, h];
    dkv_rows: int [m, 3] of (b, KV head g, key row j) -> dK[b, j, g], dV[b, j, g],
    each summed over the query heads that share KV head g.
    Returns (dq [n, d], dk [m, d], dv [m, dv]).
    """
    dq_rows = np.asarray(dq_rows, dtype=np.int64).reshape(-1, 3)
    dkv_rows = np.asarray(dkv_rows, dtype=np.int64).reshape(-1, 3)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    dq = np.zeros((len(dq_rows), d))
    dk = np.zeros((len(dkv_rows), d))
    dv = np.zeros((len(dkv_rows), v.shape[-1]))
    heads = {(int(b), int(h)) for b, h, _ in dq_rows}
    heads |= {(int(b), int(hk) * g + r) for b, hk, _ in dkv_rows for r in range(g)}
    for b, h in sorted(heads):
        qh, kh, vh = _f64(q[b, :, h]), _f64(k[b, :, h // g]), _f64(v[b, :, h // g])
        dOh = _f64(do[b, :, h])
        p = attention_weights(qh, kh, scale, causal)                  # [N, N]
        dmat = np.sum(dOh * (p @ vh), axis=1)                          # D = rowsum(dO o O)
        iq = np.nonzero((dq_rows[:, 0] == b) & (dq_rows[:, 1] == h))[0]
        if len(iq):
            rows = dq_rows[iq, 2]
            dp = dOh[rows] @ vh.T                                      # dP rows = dO_i V^T
            ds = p[rows] * (dp - dmat[rows, None])                     # dS rows
            dq[iq] = scale * (ds @ kh)                                 # dQ_i = scale dS_i K
        ikv = np.nonzero((dkv_rows[:, 0] == b) & (dkv_rows[:, 1] == h // g))[0]
        if len(ikv):
            cols = dkv_rows[ikv, 2]
            pc = p[:, cols]                                            # P[:, j]
            dv[ikv] += pc.T @ dOh                                      # dV_j = P[:, j]^T dO
            dpc = dOh @ vh[cols].T                                     # dP[:, j] = dO V_j
            dsc = pc * (dpc - dmat[:, None])                           # dS[:, j]
            dk[ikv] += scale * (dsc.T @ qh)                            # dK_j = scale dS[:, j]^T Q
    return dq, dk, dv


def decode_split_ranges(seqlens, page_size: int, max_pages_per_seq: int, num_splits: int):
    """Token range [start, end) of every (sequence, split); int64 [B, num_splits, 2].

    Each split covers C = ceil(max_pages_per_seq / num_splits) whole pages of a
    sequence; an empty split has start == end.
    """
    lens = [int(x) for x in np.asarray(seqlens)]
    chunk = -(-max_pages_per_seq // num_splits) * page_size
    out = np.zeros((len(lens), num_splits, 2), dtype=np.int64)
    for b, n in enumerate(lens):
        for s in range(num_splits):
            a = min(n, s * chunk)
            e = min(n, (s + 1) * chunk)
            out[b, s] = (a, e)
    return out


def decode_partials(q, kcache, vcache, block_table, seqlens, scale: float,
                    num_splits: int, max_pages_per_seq: int | None = None):
    """Per-split partial results of paged decode, each over its own token range.

    Returns lse_part [B, Hq, S] and o_part [B, Hq, S, d] with o_part already
    divided by its own l (empty split: lse = -inf, O = 0).
    """
    q = _f64(q)
    table = np.asarray(block_table)
    lens = [int(x) for x in np.asarray(seqlens)]
    if max_pages_per_seq is None:
        max_pages_per_seq = table.shape[1]
    B, Hq, _ = q.shape
    Hkv = kcache.shape[2]
    g = Hq // Hkv
    dv = vcache.shape[-1]
    ranges = decode_split_ranges(lens, kcache.shape[1], max_pages_per_seq, num_splits)
    lse_p = np.full((B, Hq, num_splits), -np.inf)
    o_p = np.zeros((B, Hq, num_splits, dv))
    for b in range(B):
        kb = gather_paged(kcache, table, b, lens[b])
        vb = gather_paged(vcache, table, b, lens[b])
        for s in range(num_splits):
            a, e = ranges[b, s]
            if e <= a:
                continue
            for h in range(Hq):
                ob, lb = attention_definition(q[b, h][None, :], kb[a:e, h // g], vb[a:e, h // g],
                                              scale, causal=False)
                o_p[b, h, s], lse_p[b, h, s] = ob[0], lb[0]
    return lse_p, o_p


def merge_partials(lse_part, o_part):
    """Merge split partials with the online-softmax rule ([FA-LLM] Flash-Decoding).

    A partial exported as (lse_s, O_s) with O_s already normalised is the
    running state (m = lse_s, l = 1, O = O_s). Folding the partials in order:
    m' = max(m, lse_s); l' = l e^{m - m'} + e^{lse_s - m'};
    O' = O e^{m - m'} + e^{lse_s - m'} O_s; finally O = O'/l', lse = m' + ln l'.
    lse_part [..., S], o_part [..., S, d] -> (O [..., d], lse [...]).
    """
    lse_part = _f64(lse_part)
    o_part = _f64(o_part)
    lead = lse_part.shape[:-1]
    S = lse_part.shape[-1]
    dv = o_part.shape[-1]
    lp = lse_part.reshape(-1, S)
    op = o_part.reshape(-1, S, dv)
    o = np.zeros((lp.shape[0], dv))
    lse = np.full(lp.shape[0], -np.inf)
    for r in range(lp.shape[0]):
        m, l, acc = -np.inf, 0.0, np.zeros(dv)
        for s in range(S):
            ls = lp[r, s]
            if ls == -np.inf:          # an empty split carries no weight
                continue
            m_new = max(m, ls)
            a = math.exp(m - m_new) if m != -np.inf else 0.0
            w = math.exp(ls - m_new)
            l = l * a + w
            acc = acc * a + w * op[r, s]
            m = m_new
        if l > 0:
            o[r] = acc / l
            lse[r] = m + math.log(l)
    return o.reshape(lead + (dv,)), lse.reshape(lead)
