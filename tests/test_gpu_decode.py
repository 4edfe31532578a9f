"""Paged split-KV decode and the partial merge: CUDA kernels through the C ABI
against the fp64 oracle."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_fattn_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import LSE_MAX, as_np, check, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    return need_gpu()


def _dev(x):
    d = torch.device("cuda")
    return (x.q.to(d), x.kcache.to(d), x.vcache.to(d), x.block_table.to(d), x.seqlens.to(d))


def _decode(fa, x, S, dev=None):
    q, kc, vc, bt, sl = dev if dev is not None else _dev(x)
    ws = torch.zeros(fa.decode_workspace_size(x.batch, x.hq, x.d, S), dtype=torch.uint8, device="cuda")
    o, lse = fa.decode_paged(q, kc, vc, bt, sl, S, scale=x.scale, workspace=ws)
    st = fa.debug_read_status()
    return o, lse, ws, st


@pytest.fixture(scope="module")
def cfg5():
    """Batch 8, Hq=32, Hkv=8, d=128, contexts U[1024, 65536] (seed 4), 16-token pages,
    plus spare pages full of sentinels that no table entry in range points at."""
    x = inputs.paged_decode_config(spare_pages=64)
    o_ref, lse_ref = orc.decode_paged(x.q, x.kcache, x.vcache, x.block_table, x.seqlens, x.scale)
    return x, o_ref, lse_ref


def test_paged_decode_config_full(fa, cfg5):
    x, o_ref, lse_ref = cfg5
    S = fa.choose_num_splits(x.batch, x.hkv, x.max_pages_per_seq)
    o, lse, _, st = _decode(fa, x, S)
    assert st == 0
    check(o, lse, o_ref, lse_ref, what=f"decode S={S}")


@pytest.mark.parametrize("S", [1, 2, 3, 7, 16, 64, 5000])
def test_num_splits_invariance(fa, cfg5, S):
    """Any split count (more splits than pages included) gives the same answer."""
    x, o_ref, lse_ref = cfg5
    o, lse, _, st = _decode(fa, x, S)
    assert st == 0
    check(o, lse, o_ref, lse_ref, what=f"decode S={S}")


@pytest.mark.parametrize("S", [3, 64])
def test_partials_match_oracle_split_by_split(fa, S):
    """Each split's partial (lse_s, O_s) covers exactly the oracle's token range."""
    x = inputs.decode_paged(21, 3, 8, 2, 128, 16, None, 4096, spare_pages=4, lengths=[1, 1000, 4096])
    o, lse, ws, st = _decode(fa, x, S)
    assert st == 0
    lp_ref, op_ref = orc.decode_partials(x.q, x.kcache, x.vcache, x.block_table, x.seqlens, x.scale, S)
    lp, op = fa.split_workspace(ws, x.batch, x.hq, x.d, S)
    lp, op = as_np(lp), as_np(op)
    empty = np.isneginf(lp_ref)
    assert np.array_equal(np.isneginf(lp), empty)       # the same splits are empty
    assert np.max(np.abs(lp[~empty] - lp_ref[~empty])) <= LSE_MAX
    assert np.max(np.abs(op[~empty] - op_ref[~empty])) <= 2e-2
    o_ref, lse_ref = orc.merge_partials(lp_ref, op_ref)
    check(o, lse, o_ref, lse_ref, what="merged partials")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 1), (24, 2), (16, 4)])
def test_gqa_mapping(fa, Hq, Hkv):
    """MHA (Hkv = Hq), MQA (Hkv = 1, two 16-head groups), uneven groups of 12."""
    x = inputs.decode_paged(30 + Hq, 2, Hq, Hkv, 128, 16, (1, 3000), 3072, spare_pages=2)
    o_ref, lse_ref = orc.decode_paged(x.q, x.kcache, x.vcache, x.block_table, x.seqlens, x.scale)
    o, lse, _, st = _decode(fa, x, 8)
    assert st == 0
    check(o, lse, o_ref, lse_ref, what=f"gqa {Hq}/{Hkv}")


@pytest.mark.parametrize("page_size,d", [(16, 64), (32, 128), (7, 128), (1, 64)])
def test_other_page_sizes_and_head_dims(fa, page_size, d):
    x = inputs.decode_paged(40 + page_size, 3, 8, 2, d, page_size, (1, 900), 1000, spare_pages=3)
    o_ref, lse_ref = orc.decode_paged(x.q, x.kcache, x.vcache, x.block_table, x.seqlens, x.scale)
    o, lse, _, st = _decode(fa, x, 5)
    assert st == 0
    check(o, lse, o_ref, lse_ref, what=f"page {page_size} d {d}")


@pytest.mark.parametrize("scale", [-0.12, 0.35])
def test_other_scales(fa, scale):
    """A negative and a large scale (any finite value is accepted), 3 sequences up to
    1000 tokens, GQA 8:2, d = 128, 16-token pages, 5 splits."""
    x = inputs.decode_paged(60, 3, 8, 2, 128, 16, (1, 900), 1000, spare_pages=3, scale=scale)
    o_ref, lse_ref = orc.decode_paged(x.q, x.kcache, x.vcache, x.block_table, x.seqlens, x.scale)
    o, lse, _, st = _decode(fa, x, 5)
    assert st == 0
    check(o, lse, o_ref, lse_ref, what=f"decode scale {scale}")


def test_zero_length_sequence(fa):
    x = inputs.decode_paged(50, 3, 4, 1, 64, 16, None, 256, spare_pages=1, lengths=[17, 1, 200])
    dev = list(_dev(x))
    dev[4] = torch.tensor([17, 0, 200], dtype=torch.int32, device="cuda")
    o, lse, _, st = _decode(fa, x, 4, dev=dev)
    assert st == 0
    og, lg = as_np(o), as_np(lse)
    assert np.all(og[1] == 0) and np.all(np.isneginf(lg[1]))
    o_ref, lse_ref = orc.decode_paged(x.q, x.kcache, x.vcache, x.block_table, [17, 0, 200], x.scale)
    check(og[[0, 2]], lg[[0, 2]], o_ref[[0, 2]], lse_ref[[0, 2]], what="zero-length")


def test_bad_block_table_entry_is_caught_on_device(fa):
    """An out-of-pool page index is skipped by the kernel's own bounds check and reported."""
    x = inputs.decode_paged(51, 2, 4, 1, 64, 16, None, 256, spare_pages=1, lengths=[100, 40])
    q, kc, vc, bt, sl = _dev(x)
    bt[1, 1] = x.kcache.shape[0] + 1000
    _, _, _, st = _decode(fa, x, 2, dev=(q, kc, vc, bt, sl))
    assert st == fa.FATTN_ERR_DEVICE_CHECK
    bt[1, 1] = -3
    _, _, _, st = _decode(fa, x, 2, dev=(q, kc, vc, bt, sl))
    assert st == fa.FATTN_ERR_DEVICE_CHECK
    assert fa.debug_read_status() == 0                    # reading clears the word


def test_seqlen_beyond_table_is_caught_on_device(fa):
    x = inputs.decode_paged(52, 2, 4, 1, 64, 16, None, 256, spare_pages=1, lengths=[100, 40])
    q, kc, vc, bt, sl = _dev(x)
    sl[0] = 256 + 16
    _, _, _, st = _decode(fa, x, 2, dev=(q, kc, vc, bt, sl))
    assert st == fa.FATTN_ERR_DEVICE_CHECK


# ------------------------------------------------------------ merge
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [64, 128, 36])
def test_merge_partials(fa, out_dtype, d):
    g = torch.Generator().manual_seed(d)
    B, H, S = 3, 5, 9
    lp = torch.randn(B, H, S, generator=g) * 4
    op = torch.randn(B, H, S, d, generator=g)
    lp[0, 1, 3] = -float("inf")
    lp[1, 2, :] = -float("inf")                          # a row with every split empty
    op[0, 1, 3] = float("nan")                           # an empty split's row is never read
    o, lse = fa.merge_partials(op.cuda(), lp.cuda(), out_dtype=out_dtype)
    o_ref, lse_ref = orc.merge_partials(lp, torch.nan_to_num(op))
    og, lg = as_np(o), as_np(lse)
    assert np.all(og[1, 2] == 0) and np.isneginf(lg[1, 2])
    tol = 1e-5 if out_dtype == torch.float32 else 8e-3
    assert np.max(np.abs(og - o_ref)) <= tol
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    assert np.max(np.abs(lg[fin] - lse_ref[fin])) <= 1e-5


def test_workspace_reused_across_calls(fa):
    """Each call leaves the workspace counters at zero, so one buffer serves many calls."""
    ws = torch.zeros(fa.decode_workspace_size(3, 8, 128, 64), dtype=torch.uint8, device="cuda")
    for seed, S in [(70, 64), (71, 5), (72, 64), (73, 1), (74, 17)]:
        x = inputs.decode_paged(seed, 3, 8, 2, 128, 16, (1, 3000), 3072, spare_pages=2)
        q, kc, vc, bt, sl = _dev(x)
        o, lse = fa.decode_paged(q, kc, vc, bt, sl, S, scale=x.scale, workspace=ws)
        assert fa.debug_read_status() == 0
        o_ref, lse_ref = orc.decode_paged(x.q, x.kcache, x.vcache, x.block_table, x.seqlens, x.scale)
        check(o, lse, o_ref, lse_ref, what=f"reuse seed {seed} S {S}")


def test_binding_rejects_non_bf16_decode_inputs(fa):
    """The decode kernels read bf16 only and the C ABI carries no dtype: the binding refuses
    fp32 q or caches in both decode entry points instead of reading them as bf16 pairs."""
    x = inputs.decode_paged(90, 2, 8, 2, 128, 16, None, 64, spare_pages=1, lengths=[10, 40])
    q, kc, vc, bt, sl = (t.cuda() for t in (x.q, x.kcache, x.vcache, x.block_table, x.seqlens))
    for args in ((q.float(), kc, vc), (q, kc.float(), vc), (q, kc, vc.float())):
        with pytest.raises(TypeError):
            fa.decode_paged(*args, bt, sl, 2, scale=x.scale)
        with pytest.raises(TypeError):
            fa.decode_paged_static(*args, bt, sl, 2, scale=x.scale)
