"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

Nothing here compares the oracle with a retyped copy of itself: the pins are the
worked example printed on "FlashAttention, explained", brute force with plain
Python loops, library routines (scipy softmax / logsumexp), closed forms and
invariants.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import attention as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- T1 ----
def test_worked_example_matches_printed_values():
    """'FlashAttention, explained', worked example: row [2,1,3,0] in blocks [2,1],[3,0]."""
    g = _golden("worked_example.txt")
    m, l, w, hist = orc.softmax_row_blocked(g["scores"], int(g["block"][0]))
    assert m == g["m"][0]
    assert abs(l - g["l"][0]) <= 5e-5
    assert np.max(np.abs(w - np.array(g["weights"]))) <= 5e-5
    # logsumexp consistent with the printed m and l (l printed to 4 decimals)
    assert abs((m + math.log(l)) - (g["m"][0] + math.log(g["l"][0]))) <= 5e-5 / 1.5


def test_worked_example_intermediate_state():
    """After block [2,1] the page's running state is m = 2 with every term e^{s-2}."""
    _, _, _, hist = orc.softmax_row_blocked([2, 1, 3, 0], 2)
    m1, l1 = hist[0]
    assert m1 == 2.0
    assert l1 == pytest.approx(1.0 + math.exp(-1.0), abs=1e-15)
    # second block: old sum corrected by the single factor e^{2-3}
    m2, l2 = hist[1]
    assert m2 == 3.0
    assert l2 == pytest.approx(l1 * math.exp(2 - 3) + math.exp(0) + math.exp(-3), abs=1e-15)


def test_planted_mistake_is_caught_by_worked_example():
    """Dropping the rescale factor (a plausible bug) breaks the printed l."""
    s = np.array([2.0, 1.0, 3.0, 0.0])
    m, l = -np.inf, 0.0
    for blk in (s[:2], s[2:]):
        m_new = max(m, blk.max())
        l = l + np.exp(blk - m_new).sum()      # missing l * e^{m - m'}
        m = m_new
    assert abs(l - 1.5530) > 5e-5


# ---------------------------------------------------------------- brute force ----
def _python_attention(q, k, v, scale, causal):
    """Textbook attention with plain Python loops (tiny inputs only)."""
    nq, nk, dv = len(q), len(k), len(v[0])
    out, lses = [], []
    for i in range(nq):
        scores = []
        for j in range(nk):
            if causal and j > i + (nk - nq):
                continue
            scores.append((j, scale * sum(q[i][c] * k[j][c] for c in range(len(q[i])))))
        mx = max(s for _, s in scores)
        ws = [(j, math.exp(s - mx)) for j, s in scores]
        tot = sum(w for _, w in ws)
        out.append([sum(w * v[j][c] for j, w in ws) / tot for c in range(dv)])
        lses.append(mx + math.log(tot))
    return np.array(out), np.array(lses)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk,d", [(1, 1, 3), (3, 5, 4), (5, 5, 2), (7, 4, 3)])
def test_definition_vs_python_loops(causal, nq, nk, d):
    if causal and nq > nk:
        pytest.skip("bottom-right causal with Nq > Nk leaves rows fully masked")
    rng = np.random.default_rng(nq * 100 + nk * 10 + d)
    q, k, v = _rand(rng, nq, d), _rand(rng, nk, d), _rand(rng, nk, d + 1)
    o, lse = orc.attention_definition(q, k, v, 0.7, causal)
    o_ref, lse_ref = _python_attention(q.tolist(), k.tolist(), v.tolist(), 0.7, causal)
    assert np.max(np.abs(o - o_ref)) <= 1e-13
    assert np.max(np.abs(lse - lse_ref)) <= 1e-13


# ---------------------------------------------------------------- T2 ----
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 13, 17, 31, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_blocked_equals_definition_for_every_block_size(n, causal):
    """'Tiles and an online softmax': the blocked result is the full softmax, any block size."""
    rng = np.random.default_rng(n + (1000 if causal else 0))
    d = 8
    q, k, v = _rand(rng, n, d), _rand(rng, n, d), _rand(rng, n, d)
    o_ref, lse_ref = orc.attention_definition(q, k, v, 0.5, causal)
    for bs in range(1, n + 1):
        for fn in (orc.attention_blocked, orc.attention_blocked_normalised):
            o, lse = fn(q, k, v, 0.5, causal, bs)
            assert np.max(np.abs(o - o_ref)) <= 1e-12, (fn.__name__, bs)
            assert np.max(np.abs(lse - lse_ref)) <= 1e-12, (fn.__name__, bs)


def test_blocked_row_equals_library_softmax():
    rng = np.random.default_rng(7)
    s = rng.standard_normal(37) * 4
    for bs in (1, 2, 5, 37):
        m, l, w, _ = orc.softmax_row_blocked(s, bs)
        assert np.max(np.abs(w - scipy.special.softmax(s))) <= 1e-15
        assert abs(m + math.log(l) - scipy.special.logsumexp(s)) <= 1e-13


# ---------------------------------------------------------------- T3 ----
@pytest.mark.parametrize("causal", [False, True])
def test_weights_sum_to_one_and_match_library(causal):
    rng = np.random.default_rng(3)
    q, k = _rand(rng, 33, 16), _rand(rng, 33, 16)
    w = orc.attention_weights(q, k, 0.25, causal)
    assert np.max(np.abs(w.sum(axis=1) - 1.0)) <= 1e-12
    s = 0.25 * (q @ k.T)
    if causal:
        s = np.where(np.tril(np.ones((33, 33), dtype=bool)), s, -np.inf)
    assert np.max(np.abs(w - scipy.special.softmax(s, axis=1))) <= 1e-15
    _, lse = orc.attention_definition(q, k, np.eye(33), 0.25, causal)
    assert np.max(np.abs(lse - scipy.special.logsumexp(s, axis=1))) <= 1e-13


# ---------------------------------------------------------------- T4 ----
def test_joint_kv_permutation_invariance():
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, 20, 8), _rand(rng, 50, 8), _rand(rng, 50, 8)
    perm = rng.permutation(50)
    o1, l1 = orc.attention_definition(q, k, v, 0.3, False)
    o2, l2 = orc.attention_definition(q, k[perm], v[perm], 0.3, False)
    assert np.max(np.abs(o1 - o2)) <= 1e-12
    assert np.max(np.abs(l1 - l2)) <= 1e-12


# ---------------------------------------------------------------- T5 ----
def test_causal_row0_is_v0_and_varlen_first_tokens():
    rng = np.random.default_rng(5)
    q, k, v = _rand(rng, 9, 4), _rand(rng, 9, 4), _rand(rng, 9, 4)
    o, lse = orc.attention_definition(q, k, v, 1.0, True)
    assert np.array_equal(o[0], v[0])
    assert lse[0] == pytest.approx(float(q[0] @ k[0]), abs=1e-15)
    # varlen: the first token of every packed sequence sees only itself
    lens = [3, 1, 5]
    cu = np.cumsum([0] + lens)
    T = cu[-1]
    qv, kv, vv = _rand(rng, T, 2, 4), _rand(rng, T, 2, 4), _rand(rng, T, 2, 4)
    ov, _ = orc.attn_fwd(qv, kv, vv, 0.5, True, cu_seqlens=cu)
    for a in cu[:-1]:
        assert np.array_equal(ov[a], vv[a])


# ---------------------------------------------------------------- T6 ----
def test_uniform_weights_closed_form():
    """K = 0 makes every score equal: O = mean(V) (causal: prefix means)."""
    rng = np.random.default_rng(6)
    q, v = _rand(rng, 12, 8), _rand(rng, 12, 5)
    k = np.zeros((12, 8))
    o, lse = orc.attention_definition(q, k, v, 1.0, False)
    assert np.max(np.abs(o - v.mean(axis=0))) <= 1e-14
    assert np.max(np.abs(lse - math.log(12))) <= 1e-14
    o, lse = orc.attention_definition(q, k, v, 1.0, True)
    prefix = np.cumsum(v, axis=0) / np.arange(1, 13)[:, None]
    assert np.max(np.abs(o - prefix)) <= 1e-14
    assert np.max(np.abs(lse - np.log(np.arange(1, 13)))) <= 1e-14


def test_dominant_score_and_no_overflow():
    """One score far above the rest picks its value row; huge scores stay finite."""
    d = 4
    q = np.array([[1.0, 0, 0, 0]])
    s = np.array([3.0, -1.0, 1000.0, 2.0])          # gap >= 200 at index 2
    k = np.zeros((4, d))
    k[:, 0] = s
    v = np.arange(16, dtype=float).reshape(4, 4)
    o, lse = orc.attention_definition(q, k, v, 1.0, False)
    assert np.array_equal(o[0], v[2])               # other weights underflow to 0
    assert lse[0] == 1000.0
    # e^{1000} overflows fp64 without the max subtraction
    for bs in (1, 2, 3):
        ob, lb = orc.attention_blocked(q, k, v, 1.0, False, bs)
        assert np.all(np.isfinite(ob)) and np.array_equal(ob[0], v[2]) and lb[0] == 1000.0


# ---------------------------------------------------------------- T7 ----
@pytest.mark.parametrize("seed", range(5))
def test_merge_of_split_partials_equals_unsplit(seed):
    """'Flash-Decoding': partials over chunks of K/V merged by the same rule."""
    rng = np.random.default_rng(100 + seed)
    nk, d = 61, 16
    q, k, v = _rand(rng, 3, d), _rand(rng, nk, d), _rand(rng, nk, d)
    o_ref, lse_ref = orc.attention_definition(q, k, v, 0.4, False)
    n_cuts = int(rng.integers(1, 8))
    cuts = sorted(set(rng.integers(1, nk, n_cuts).tolist()))
    bounds = [0] + cuts + [nk]
    lp, op = [], []
    for a, e in zip(bounds[:-1], bounds[1:]):
        o_s, l_s = orc.attention_definition(q, k[a:e], v[a:e], 0.4, False)
        lp.append(l_s)
        op.append(o_s)
    lp.append(np.full(3, -np.inf))                  # an empty split
    op.append(np.full((3, d), np.nan))              # never read
    lse_part = np.stack(lp, axis=-1)
    o_part = np.stack(op, axis=1)
    o, lse = orc.merge_partials(lse_part, o_part)
    assert np.max(np.abs(o - o_ref)) <= 1e-12
    assert np.max(np.abs(lse - lse_ref)) <= 1e-12


def test_empty_key_set_is_zero_and_minus_inf():
    """A row with no visible key (empty context) has O = 0 and lse = -inf; as a split it has no weight."""
    o, lse = orc.attention_definition(np.ones((2, 4)), np.zeros((0, 4)), np.zeros((0, 3)), 1.0)
    assert np.array_equal(o, np.zeros((2, 3))) and np.all(np.isneginf(lse))
    rng = np.random.default_rng(14)
    q, k, v = _rand(rng, 2, 4), _rand(rng, 6, 4), _rand(rng, 6, 3)
    o_ref, l_ref = orc.attention_definition(q, k, v, 1.0)
    lp = np.stack([lse, l_ref], axis=-1)
    op = np.stack([o, o_ref], axis=1)
    om, lm = orc.merge_partials(lp, op)
    assert np.max(np.abs(om - o_ref)) <= 1e-15 and np.max(np.abs(lm - l_ref)) <= 1e-15


def test_merge_all_empty_is_zero_and_minus_inf():
    o, lse = orc.merge_partials(np.full((2, 4), -np.inf), np.ones((2, 4, 3)))
    assert np.array_equal(o, np.zeros((2, 3)))
    assert np.all(lse == -np.inf)


# ---------------------------------------------------------------- GQA / varlen ----
def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(8)
    B, N, Hq, Hkv, d = 2, 9, 6, 2, 4
    q, k, v = _rand(rng, B, N, Hq, d), _rand(rng, B, N, Hkv, d), _rand(rng, B, N, Hkv, d)
    o, lse = orc.attn_fwd(q, k, v, 0.5, True)
    kr, vr = np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2)
    for h in range(Hq):
        assert np.array_equal(kr[:, :, h], k[:, :, h // 3])
    o2, lse2 = orc.attn_fwd(q, kr, vr, 0.5, True)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_varlen_has_no_cross_sequence_attention():
    rng = np.random.default_rng(9)
    lens = [4, 7, 1, 5]
    cu = np.cumsum([0] + lens)
    T, H, d = cu[-1], 2, 4
    q, k, v = _rand(rng, T, H, d), _rand(rng, T, H, d), _rand(rng, T, H, d)
    o, lse = orc.attn_fwd(q, k, v, 0.5, True, cu_seqlens=cu)
    for b, (a, e) in enumerate(zip(cu[:-1], cu[1:])):
        for h in range(H):
            o_ref, l_ref = _python_attention(q[a:e, h].tolist(), k[a:e, h].tolist(),
                                             v[a:e, h].tolist(), 0.5, True)
            assert np.max(np.abs(o[a:e, h] - o_ref)) <= 1e-13
            assert np.max(np.abs(lse[h, a:e] - l_ref)) <= 1e-13


def test_sampled_rows_match_full_output():
    rng = np.random.default_rng(10)
    q, k, v = _rand(rng, 2, 11, 4, 8), _rand(rng, 2, 11, 2, 8), _rand(rng, 2, 11, 2, 8)
    o, lse = orc.attn_fwd(q, k, v, 0.3, True)
    samples = np.array([[0, 0, 0], [1, 3, 10], [0, 2, 5], [1, 1, 7]])
    os_, ls_ = orc.attn_fwd_rows(q, k, v, 0.3, True, samples)
    for n, (b, h, i) in enumerate(samples):
        assert np.max(np.abs(os_[n] - o[b, i, h])) <= 1e-14 and abs(ls_[n] - lse[b, h, i]) <= 1e-14


# ---------------------------------------------------------------- paged decode ----
def _small_paged(rng, lens, page_size, Hkv, d, spare=3):
    pages = [-(-n // page_size) for n in lens]
    pool = sum(pages) + spare
    perm = rng.permutation(pool)
    max_pages = max(pages) + 2
    table = np.zeros((len(lens), max_pages), dtype=np.int32)
    kc = np.full((pool, page_size, Hkv, d), 1e4)
    vc = np.full((pool, page_size, Hkv, d), 1e4)
    k_log, v_log = [], []
    off = 0
    for b, n in enumerate(lens):
        table[b, : pages[b]] = perm[off: off + pages[b]]
        table[b, pages[b]:] = perm[-1]                       # a spare page
        kl, vl = _rand(rng, n, Hkv, d), _rand(rng, n, Hkv, d)
        for t in range(n):                                   # scatter token by token
            kc[table[b, t // page_size], t % page_size] = kl[t]
            vc[table[b, t // page_size], t % page_size] = vl[t]
        k_log.append(kl)
        v_log.append(vl)
        off += pages[b]
    return kc, vc, table, k_log, v_log


def test_paged_gather_is_bit_exact():
    rng = np.random.default_rng(11)
    lens = [1, 16, 17, 40]
    kc, vc, table, k_log, _ = _small_paged(rng, lens, 16, 2, 4)
    for b, n in enumerate(lens):
        assert np.array_equal(orc.gather_paged(kc, table, b, n), k_log[b])


def test_paged_decode_equals_contiguous_definition():
    rng = np.random.default_rng(12)
    lens = [5, 33, 64, 1]
    Hq, Hkv, d = 4, 2, 8
    kc, vc, table, k_log, v_log = _small_paged(rng, lens, 16, Hkv, d)
    q = _rand(rng, len(lens), Hq, d)
    o, lse = orc.decode_paged(q, kc, vc, table, lens, 0.35)
    for b, n in enumerate(lens):
        for h in range(Hq):
            o_ref, l_ref = _python_attention([q[b, h].tolist()], k_log[b][:, h // 2].tolist(),
                                             v_log[b][:, h // 2].tolist(), 0.35, False)
            assert np.max(np.abs(o[b, h] - o_ref[0])) <= 1e-13
            assert abs(lse[b, h] - l_ref[0]) <= 1e-13


def test_split_ranges_partition_each_sequence():
    lens = [1, 15, 16, 17, 100, 257, 0]
    for ps in (1, 16, 32):
        for max_pages in (-(-257 // ps), -(-257 // ps) + 5):
            for S in (1, 2, 3, 7, 16, 64, 400):
                r = orc.decode_split_ranges(lens, ps, max_pages, S)
                C = -(-max_pages // S)
                for b, n in enumerate(lens):
                    covered = []
                    for s in range(S):
                        a, e = r[b, s]
                        assert 0 <= a <= e <= n
                        assert e - a <= C * ps
                        if e > a:
                            assert a == s * C * ps           # whole pages, in order
                            covered.extend(range(a, e))
                    assert covered == list(range(n))


@pytest.mark.parametrize("S", [1, 2, 3, 5, 16])
def test_decode_partials_merge_to_decode(S):
    rng = np.random.default_rng(13)
    lens = [5, 33, 64, 1, 47]
    Hq, Hkv, d = 4, 1, 8
    kc, vc, table, _, _ = _small_paged(rng, lens, 16, Hkv, d)
    q = _rand(rng, len(lens), Hq, d)
    o_ref, lse_ref = orc.decode_paged(q, kc, vc, table, lens, 0.35)
    lp, op = orc.decode_partials(q, kc, vc, table, lens, 0.35, S)
    o, lse = orc.merge_partials(lp, op)
    assert np.max(np.abs(o - o_ref)) <= 1e-12
    assert np.max(np.abs(lse - lse_ref)) <= 1e-12


# ---------------------------------------------------------------- block-sparse ----
def test_block_sparse_vs_python_loops():
    """'Block-sparse FlashAttention': keys in zero blocks take no part in the softmax."""
    rng = np.random.default_rng(20)
    B, N, H, d, blk = 1, 11, 2, 4, 3
    q, k, v = _rand(rng, B, N, H, d), _rand(rng, B, N, H, d), _rand(rng, B, N, H, d)
    nb = -(-N // blk)
    bm = rng.integers(0, 2, size=(H, nb, nb)).astype(np.uint8)
    bm[:, :, 0] = 1                                   # every row keeps at least one block
    for causal in (False, True):
        o, lse = orc.attn_fwd_block_sparse(q, k, v, 0.5, causal, bm, blk)
        for h in range(H):
            for i in range(N):
                keys = [j for j in range(N) if bm[h, i // blk, j // blk] and (not causal or j <= i)]
                s = [0.5 * float(q[0, i, h] @ k[0, j, h]) for j in keys]
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                tot = sum(w)
                ref = sum(wi * v[0, j, h] for wi, j in zip(w, keys)) / tot
                assert np.max(np.abs(o[0, i, h] - ref)) <= 1e-13
                assert abs(lse[0, h, i] - (mx + math.log(tot))) <= 1e-13


def test_block_sparse_all_ones_is_dense_and_empty_rows():
    rng = np.random.default_rng(21)
    B, N, Hq, Hkv, d, blk = 2, 10, 4, 2, 8, 4
    q, k, v = _rand(rng, B, N, Hq, d), _rand(rng, B, N, Hkv, d), _rand(rng, B, N, Hkv, d)
    nb = -(-N // blk)
    for causal in (False, True):
        o1, l1 = orc.attn_fwd_block_sparse(q, k, v, 0.3, causal, np.ones((1, nb, nb), np.uint8), blk)
        o2, l2 = orc.attn_fwd(q, k, v, 0.3, causal)
        assert np.max(np.abs(o1 - o2)) <= 1e-14 and np.max(np.abs(l1 - l2)) <= 1e-14
    bm = np.ones((1, nb, nb), np.uint8)
    bm[0, 1, :] = 0                                   # query block 1 sees nothing
    o, lse = orc.attn_fwd_block_sparse(q, k, v, 0.3, False, bm, blk)
    assert np.all(o[:, blk:2 * blk] == 0) and np.all(np.isneginf(lse[:, :, blk:2 * blk]))
    smp = np.array([[1, 3, 9], [0, 0, 5], [1, 2, 0], [1, 3, 2], [0, 0, 5], [1, 3, 1]])
    os_, ls_ = orc.attn_fwd_block_sparse(q, k, v, 0.3, False, bm, blk, rows=smp)
    for n, (b, h, i) in enumerate(smp):
        assert np.array_equal(os_[n], o[b, i, h]) or np.max(np.abs(os_[n] - o[b, i, h])) <= 1e-14
        assert (np.isneginf(ls_[n]) and np.isneginf(lse[b, h, i])) or abs(ls_[n] - lse[b, h, i]) <= 1e-14


def test_paged_prefill_vs_python_loops():
    """Chunked prefill over a paged context: query i of a chunk of Lq sees keys
    j <= i + (Lk - Lq); the keys are gathered token by token through the table."""
    rng = np.random.default_rng(30)
    lens_k, lens_q = [5, 33, 17, 8], [5, 4, 1, 8]
    Hq, Hkv, d, P = 4, 2, 3, 8
    kc, vc, table, k_log, v_log = _small_paged(rng, lens_k, P, Hkv, d)
    cu = np.concatenate([[0], np.cumsum(lens_q)])
    q = _rand(rng, int(cu[-1]), Hq, d)
    for causal in (False, True):
        o, lse = orc.attn_fwd_paged(q, kc, vc, table, lens_k, cu, 0.4, causal)
        for b, (lq, lk) in enumerate(zip(lens_q, lens_k)):
            for h in range(Hq):
                for i in range(lq):
                    keys = [j for j in range(lk) if not causal or j <= i + lk - lq]
                    krow = [kc[table[b, j // P], j % P, h // 2] for j in keys]
                    vrow = [vc[table[b, j // P], j % P, h // 2] for j in keys]
                    s = [0.4 * sum(float(q[cu[b] + i, h, c]) * float(kr[c]) for c in range(d)) for kr in krow]
                    mx = max(s)
                    w = [math.exp(x - mx) for x in s]
                    tot = sum(w)
                    ref = [sum(wi * float(vr[c]) for wi, vr in zip(w, vrow)) / tot for c in range(d)]
                    assert np.max(np.abs(o[cu[b] + i, h] - np.array(ref))) <= 1e-13
                    assert abs(lse[h, cu[b] + i] - (mx + math.log(tot))) <= 1e-13


def test_paged_prefill_special_cases():
    rng = np.random.default_rng(31)
    lens_k = [9, 40, 16]
    Hq, Hkv, d, P = 2, 1, 4, 16
    kc, vc, table, k_log, v_log = _small_paged(rng, lens_k, P, Hkv, d)
    # a full prefill from the cache (Lq = Lk): the first query sees key 0 only -> O = V[0]
    cu = np.concatenate([[0], np.cumsum(lens_k)])
    q = _rand(rng, int(cu[-1]), Hq, d)
    o, lse = orc.attn_fwd_paged(q, kc, vc, table, lens_k, cu, 0.5, True)
    for b in range(len(lens_k)):
        for h in range(Hq):
            assert np.max(np.abs(o[cu[b], h] - v_log[b][0, 0])) <= 1e-15
    # chunks of one query are decode steps: the query sees its whole context
    cu1 = np.arange(len(lens_k) + 1)
    q1 = _rand(rng, len(lens_k), Hq, d)
    o1, lse1 = orc.attn_fwd_paged(q1, kc, vc, table, lens_k, cu1, 0.5, True)
    for b, n in enumerate(lens_k):
        for h in range(Hq):
            o_ref, l_ref = _python_attention([q1[b, h].tolist()], k_log[b][:, 0].tolist(),
                                             v_log[b][:, 0].tolist(), 0.5, False)
            assert np.max(np.abs(o1[b, h] - o_ref[0])) <= 1e-13 and abs(lse1[h, b] - l_ref[0]) <= 1e-13
    # relabelling the pool's pages (and the table with them) changes nothing
    perm = rng.permutation(kc.shape[0])
    inv = np.argsort(perm)
    o2, lse2 = orc.attn_fwd_paged(q, kc[perm], vc[perm], inv[table].astype(np.int32), lens_k, cu, 0.5, True)
    assert np.array_equal(o2, o) and np.array_equal(lse2, lse)
    # sampled rows agree with the full output
    smp = np.array([[0, 1, 8], [1, 0, 0], [1, 1, 39], [2, 0, 7]])
    os_, ls_ = orc.attn_fwd_paged(q, kc, vc, table, lens_k, cu, 0.5, True, samples=smp)
    for n, (b, h, i) in enumerate(smp):
        assert np.max(np.abs(os_[n] - o[cu[b] + i, h])) <= 1e-14 and abs(ls_[n] - lse[h, cu[b] + i]) <= 1e-14


def _loss(q, k, v, do, scale, causal):
    o, _ = orc.attn_fwd(q, k, v, scale, causal)
    return float(np.sum(o * do))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    """dQ, dK, dV are the gradients of L = sum(O o dO): central differences on every input."""
    rng = np.random.default_rng(40)
    B, N, Hq, Hkv, d, sc = 1, 5, 2, 1, 3, 0.7
    q, k, v = _rand(rng, B, N, Hq, d), _rand(rng, B, N, Hkv, d), _rand(rng, B, N, Hkv, d)
    do = _rand(rng, B, N, Hq, d)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, sc, causal)
    eps = 1e-6
    for x, gx in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(q, k, v, do, sc, causal)
            x[idx] = old - eps
            lm = _loss(q, k, v, do, sc, causal)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        assert np.max(np.abs(num - gx)) <= 1e-7


def test_backward_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(41)
    B, N, Hq, Hkv, d, sc = 2, 9, 4, 2, 6, 0.4
    q, k, v = _rand(rng, B, N, Hq, d), _rand(rng, B, N, Hkv, d), _rand(rng, B, N, Hkv, d)
    do = _rand(rng, B, N, Hq, d)
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
        kk = tk.repeat_interleave(Hq // Hkv, dim=2)
        vv = tv.repeat_interleave(Hq // Hkv, dim=2)
        s = sc * torch.einsum("bihc,bjhc->bhij", tq, kk)
        if causal:
            s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
        o = torch.einsum("bhij,bjhc->bihc", torch.softmax(s, dim=-1), vv)
        (o * torch.tensor(do)).sum().backward()
        dq, dk, dv = orc.attn_bwd(q, k, v, do, sc, causal)
        for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            assert np.max(np.abs(mine - ref.numpy())) <= 1e-12


def test_backward_closed_form_uniform_causal():
    """K = 0: row i of P is uniform over keys 0..i, so dV_j = sum_{i >= j} dO_i / (i + 1);
    and with every row's dO equal to c, O's gradient through V is all there is: dQ = dK = 0
    when V is constant along keys."""
    rng = np.random.default_rng(42)
    B, N, H, d = 1, 6, 1, 3
    q, v, do = _rand(rng, B, N, H, d), _rand(rng, B, N, H, d), _rand(rng, B, N, H, d)
    k = np.zeros((B, N, H, d))
    _, _, dv = orc.attn_bwd(q, k, v, do, 0.5, True)
    for j in range(N):
        ref = sum(do[0, i, 0] / (i + 1) for i in range(j, N))
        assert np.max(np.abs(dv[0, j, 0] - ref)) <= 1e-14
    vc = np.repeat(_rand(rng, 1, 1, 1, d), N, axis=1)
    kr = _rand(rng, B, N, H, d)
    dq, dk, _ = orc.attn_bwd(q, kr, vc, do, 0.5, False)
    assert np.max(np.abs(dq)) <= 1e-13 and np.max(np.abs(dk)) <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_backward_rows_equal_whole_gradients(causal):
    """attn_bwd_rows (the sampled form used at full size) equals the pinned attn_bwd at
    the requested rows, GQA included (dK, dV summed over the query heads of a group),
    with rows repeated and in any order; and one of its dK rows matches central
    differences of L = sum(O o dO) directly."""
    rng = np.random.default_rng(43)
    B, N, Hq, Hkv, d, sc = 2, 11, 4, 2, 5, 0.45
    q, k, v = _rand(rng, B, N, Hq, d), _rand(rng, B, N, Hkv, d), _rand(rng, B, N, Hkv, d)
    do = _rand(rng, B, N, Hq, d)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, sc, causal)
    rq = np.array([[0, 0, 0], [1, 3, 10], [0, 2, 5], [1, 3, 10], [1, 1, 7]])
    rkv = np.array([[0, 1, 0], [1, 0, 10], [1, 1, 4], [0, 0, 9], [0, 1, 0]])
    sq, sk, sv = orc.attn_bwd_rows(q, k, v, do, sc, causal, rq, rkv)
    for n, (b, h, i) in enumerate(rq):
        assert np.max(np.abs(sq[n] - dq[b, i, h])) <= 1e-13
    for n, (b, g, j) in enumerate(rkv):
        assert np.max(np.abs(sk[n] - dk[b, j, g])) <= 1e-13
        assert np.max(np.abs(sv[n] - dv[b, j, g])) <= 1e-13
    # central differences on dK[1, 4, 1]
    eps = 1e-6
    for c in range(d):
        old = k[1, 4, 1, c]
        k[1, 4, 1, c] = old + eps
        lp = _loss(q, k, v, do, sc, causal)
        k[1, 4, 1, c] = old - eps
        lm = _loss(q, k, v, do, sc, causal)
        k[1, 4, 1, c] = old
        assert abs((lp - lm) / (2 * eps) - sk[2, c]) <= 1e-7
    # no rows requested: empty results
    e = orc.attn_bwd_rows(q, k, v, do, sc, causal, np.zeros((0, 3)), np.zeros((0, 3)))
    assert e[0].shape == (0, d) and e[1].shape == (0, d) and e[2].shape == (0, d)


def test_additive_mask_vs_python_loops():
    """O = softmax(scale Q K^T + M) V with a general additive M (-inf entries remove keys)."""
    rng = np.random.default_rng(50)
    B, N, Hq, Hkv, d, sc = 2, 7, 2, 1, 3, 0.6
    q, k, v = _rand(rng, B, N, Hq, d), _rand(rng, B, N, Hkv, d), _rand(rng, B, N, Hkv, d)
    m = 2.0 * _rand(rng, 1, Hq, N, N)
    m[0, 1, 3, [0, 2, 5]] = -np.inf
    m[0, 0, 4, :] = -np.inf                                  # row 4 of head 0 sees nothing
    for causal in (False, True):
        o, lse = orc.attn_fwd_masked(q, k, v, sc, causal, m)
        for b in range(B):
            for h in range(Hq):
                for i in range(N):
                    keys = [j for j in range(N) if np.isfinite(m[0, h, i, j]) and (not causal or j <= i)]
                    if not keys:
                        assert np.all(o[b, i, h] == 0) and np.isneginf(lse[b, h, i])
                        continue
                    s = [sc * float(q[b, i, h] @ k[b, j, 0]) + m[0, h, i, j] for j in keys]
                    mx = max(s)
                    w = [math.exp(x - mx) for x in s]
                    tot = sum(w)
                    ref = sum(wi * v[b, j, 0] for wi, j in zip(w, keys)) / tot
                    assert np.max(np.abs(o[b, i, h] - ref)) <= 1e-13
                    assert abs(lse[b, h, i] - (mx + math.log(tot))) <= 1e-13


def test_additive_mask_special_cases():
    rng = np.random.default_rng(51)
    B, N, H, d, sc = 1, 9, 2, 4, 0.5
    q, k, v = _rand(rng, B, N, H, d), _rand(rng, B, N, H, d), _rand(rng, B, N, H, d)
    o0, l0 = orc.attn_fwd(q, k, v, sc, False)
    o1, l1 = orc.attn_fwd_masked(q, k, v, sc, False, np.zeros((1, 1, N, N)))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)          # M = 0 is no mask
    tri = np.where(np.tril(np.ones((N, N))) > 0, 0.0, -np.inf)[None, None]
    oc, lc = orc.attn_fwd(q, k, v, sc, True)
    o2, l2 = orc.attn_fwd_masked(q, k, v, sc, False, tri)
    assert np.max(np.abs(o2 - oc)) <= 1e-15 and np.max(np.abs(l2 - lc)) <= 1e-15  # -inf above the diagonal = causal
    c = rng.normal(size=(1, H, N, 1)) * 3                             # a per-row constant shifts lse only
    o3, l3 = orc.attn_fwd_masked(q, k, v, sc, False, np.broadcast_to(c, (1, H, N, N)))
    assert np.max(np.abs(o3 - o0)) <= 1e-13
    assert np.max(np.abs(l3 - (l0 + c[0, :, :, 0][None]))) <= 1e-13
    smp = np.array([[0, 1, 3], [0, 0, 8], [0, 1, 0], [0, 1, 3], [0, 0, 2]])
    os_, ls_ = orc.attn_fwd_masked(q, k, v, sc, False, tri, rows=smp)
    for n, (b, h, i) in enumerate(smp):
        assert np.max(np.abs(os_[n] - o2[b, i, h])) <= 1e-15 and abs(ls_[n] - l2[b, h, i]) <= 1e-15


def test_e4m3_decode_closed_forms():
    """E4M3 ('fn'): bias 7, 3 mantissa bits, subnormals, no infinities, 0x7f / 0xff NaN."""
    dec = orc.e4m3_to_f64
    assert dec([0x38])[0] == 1.0 and dec([0xB8])[0] == -1.0
    assert dec([0x7E])[0] == 448.0 and dec([0xFE])[0] == -448.0        # largest finite
    assert dec([0x08])[0] == 2.0 ** -6                                    # smallest normal
    assert dec([0x01])[0] == 2.0 ** -9 and dec([0x07])[0] == 7 * 2.0 ** -9  # subnormals
    assert dec([0x00])[0] == 0.0 and dec([0x80])[0] == 0.0
    assert np.isnan(dec([0x7F])[0]) and np.isnan(dec([0xFF])[0])
    assert dec([0x3C])[0] == 1.5 and dec([0x44])[0] == 3.0 and dec([0x78])[0] == 256.0
    v = dec(np.arange(256))
    fin = np.isfinite(v)
    assert fin.sum() == 254 and len(np.unique(v[fin])) == 253             # +0 and -0 coincide


def test_e4m3_decode_agrees_with_torch():
    torch = pytest.importorskip("torch")
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    mine = orc.e4m3_to_f64(codes.numpy())
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])


def test_fp8_attention_is_the_definition_on_dequantized_inputs():
    from exact_tiled_attention_fattn_gb300 import inputs
    x = inputs.prefill_fp8(60, 1, 40, 2, 1, 16, True)
    o, lse = orc.attn_fwd_fp8(x.q8, x.k8, x.v8, x.q_descale, x.k_descale, x.v_descale, x.scale, True)
    q = orc.e4m3_to_f64(x.q8.numpy()) * x.q_descale
    k = orc.e4m3_to_f64(x.k8.numpy()) * x.k_descale
    v = orc.e4m3_to_f64(x.v8.numpy()) * x.v_descale
    for h in range(2):
        for i in (0, 17, 39):
            o_ref, l_ref = _python_attention([q[0, i, h].tolist()], k[0, : i + 1, 0].tolist(), v[0, : i + 1, 0].tolist(),
                                             x.scale, False)
            assert np.max(np.abs(o[0, i, h] - o_ref[0])) <= 1e-12 and abs(lse[0, h, i] - l_ref[0]) <= 1e-12
    assert abs(np.max(np.abs(q)) - 448 * x.q_descale) <= 1e-9 * np.max(np.abs(q))  # amax scaled to 448
