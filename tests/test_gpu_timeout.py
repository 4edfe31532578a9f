"""The bounded pipeline waits of the tensor-core kernels, made to run out on purpose.

Every mbarrier wait in the prefill and backward kernels gives up after a limit: it
records FATTN_ERR_TIMEOUT in the device status word, every role stops, the copies
and tensor-core products already issued are waited for, TMEM is freed and the kernel
returns. Here the test hook makes the softmax / element-wise warps wait on a barrier
that nothing arrives on (with a 1 ms limit), so that path runs; the process then
goes on with normal calls on the same context, which must be correct.
"""
import numpy as np
import pytest
import torch

from exact_tiled_attention_fattn_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import check, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    f = need_gpu()
    yield f
    f.debug_set_wait_limit(0, False)


def _stalled(fa, call):
    """Run `call` with the stall hook on; return the status word it left."""
    assert fa.debug_read_status() == 0
    fa.debug_set_wait_limit(1_000_000, True)     # 1 ms per wait
    try:
        call()
        torch.cuda.synchronize()
    finally:
        fa.debug_set_wait_limit(0, False)
    return fa.debug_read_status()


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_wait_runs_out_then_context_still_works(fa, d):
    x = inputs.prefill_dense(8000 + d, 2, 1000, 4, 2, d, causal=True)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    st = _stalled(fa, lambda: fa.fwd(q, k, v, causal=True, scale=x.scale, out=o))
    assert st == fa.FATTN_ERR_TIMEOUT
    assert torch.isnan(o.float()).all()          # the stalled launch wrote no output row
    o2, lse2 = fa.fwd(q, k, v, causal=True, scale=x.scale)
    assert fa.debug_read_status() == 0
    o_ref, lse_ref = orc.attn_fwd(x.q, x.k, x.v, x.scale, True)
    check(o2, lse2, o_ref, lse_ref, what=f"prefill after a timeout d={d}")


def test_block_sparse_and_paged_waits_run_out(fa):
    x = inputs.prefill_dense(8100, 1, 700, 2, 2, 128, causal=True)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    nb = -(-700 // 128)
    mask = torch.ones(1, nb, nb, dtype=torch.uint8, device="cuda")
    assert _stalled(fa, lambda: fa.fwd_block_sparse(q, k, v, mask, causal=True, scale=x.scale)) == \
        fa.FATTN_ERR_TIMEOUT
    xp = inputs.prefill_paged(8101, 2, 4, 2, 128, 16, [300, 513], [300, 128], 640, causal=True)
    args = [t.cuda() for t in (xp.q, xp.kcache, xp.vcache, xp.block_table, xp.seqlens_k, xp.cu_seqlens_q)]
    assert _stalled(fa, lambda: fa.fwd_paged(*args, max(xp.lengths_q), causal=True, scale=xp.scale)) == \
        fa.FATTN_ERR_TIMEOUT
    o, lse = fa.fwd_paged(*args, max(xp.lengths_q), causal=True, scale=xp.scale)
    assert fa.debug_read_status() == 0
    o_ref, lse_ref = orc.attn_fwd_paged(xp.q, xp.kcache, xp.vcache, xp.block_table, xp.seqlens_k, xp.cu_seqlens_q,
                                        xp.scale, True)
    check(o, lse, o_ref, lse_ref, what="paged prefill after a timeout")


def test_backward_waits_run_out_then_backward_still_works(fa):
    x = inputs.prefill_dense(8200, 1, 513, 4, 2, 128, causal=True)
    g = torch.Generator("cpu").manual_seed(8201)
    do = torch.randn(x.q.shape, generator=g).to(torch.bfloat16)
    q, k, v, dog = x.q.cuda(), x.k.cuda(), x.v.cuda(), do.cuda()
    o, lse = fa.fwd(q, k, v, causal=True, scale=x.scale)
    assert fa.debug_read_status() == 0
    assert _stalled(fa, lambda: fa.bwd(q, k, v, o, lse, dog, causal=True, scale=x.scale)) == fa.FATTN_ERR_TIMEOUT
    dq, dk, dv = fa.bwd(q, k, v, o, lse, dog, causal=True, scale=x.scale)
    assert fa.debug_read_status() == 0
    rq, rk, rv = orc.attn_bwd(x.q, x.k, x.v, do, x.scale, True)
    for name, a, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        err = np.abs(a.float().cpu().double().numpy() - r)
        assert err.max() <= 2e-2 * max(1.0, np.abs(r).max()), name
        assert err.mean() <= 4e-3 * max(np.abs(r).mean(), 1e-3), name
