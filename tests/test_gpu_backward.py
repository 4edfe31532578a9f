"""Attention backward ('The backward pass recomputes instead of reading'): the CUDA
kernels through the C ABI against the fp64 oracle's gradients."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_fattn_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import as_np, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    return need_gpu()


def _grad_err(g_gpu, g_ref):
    err = np.abs(as_np(g_gpu) - g_ref)
    return float(err.max()), float(err.mean()), float(np.abs(g_ref).max()), float(np.abs(g_ref).mean())


CASES = [
    # B, N, Hq, Hkv, d, causal
    (2, 300, 4, 2, 128, True),
    (1, 513, 8, 1, 64, True),
    (2, 256, 2, 2, 128, False),
    (1, 100, 1, 1, 64, False),
    (1, 1000, 4, 4, 128, True),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal", CASES)
def test_backward_parity(fa, B, N, Hq, Hkv, d, causal):
    x = inputs.prefill_dense(4000 + N + d, B, N, Hq, Hkv, d, causal)
    g = torch.Generator("cpu").manual_seed(4100 + N)
    do = torch.randn((B, N, Hq, d), generator=g).to(torch.bfloat16)
    q, k, v, dog = x.q.cuda(), x.k.cuda(), x.v.cuda(), do.cuda()
    o, lse = fa.fwd(q, k, v, causal=causal, scale=x.scale)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, dog, causal=causal, scale=x.scale)
    assert fa.debug_read_status() == 0
    rq, rk, rv = orc.attn_bwd(x.q, x.k, x.v, do, x.scale, causal)
    for name, a, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        mx, mean, rmax, rmean = _grad_err(a, r)
        print(name, f"max {mx:.3e} mean {mean:.3e} | ref max {rmax:.3f} mean {rmean:.3f}")
        assert np.all(np.isfinite(as_np(a)))
        assert mx <= 2e-2 * max(1.0, rmax), f"{name}: max err {mx:.3e} (ref max {rmax:.3f})"
        assert mean <= 4e-3 * max(rmean, 1e-3), f"{name}: mean err {mean:.3e} (ref mean {rmean:.3f})"


def test_backward_full_size_sampled_heads(fa):
    """The bench's workload (causal MHA B=4 H=32 N=4096 d=128) in the launch the bench times; the
    oracle's gradients for three whole (sequence, head) slices, every row."""
    x = inputs.causal_mha_config()
    B, N, H, d = x.q.shape
    g = torch.Generator("cpu").manual_seed(5)
    do = torch.randn((B, N, H, d), generator=g).to(torch.bfloat16)
    q, k, v, dog = x.q.cuda(), x.k.cuda(), x.v.cuda(), do.cuda()
    o, lse = fa.fwd(q, k, v, causal=True, scale=x.scale)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, dog, causal=True, scale=x.scale)
    assert fa.debug_read_status() == 0
    for b, h in ((0, 0), (2, 17), (3, 31)):
        sl = lambda t: t[b:b + 1, :, h:h + 1]
        rq, rk, rv = orc.attn_bwd(sl(x.q), sl(x.k), sl(x.v), sl(do), x.scale, True)
        for name, a, r in (("dq", sl(dq), rq), ("dk", sl(dk), rk), ("dv", sl(dv), rv)):
            mx, mean, rmax, rmean = _grad_err(a, r)
            assert mx <= 2e-2 * max(1.0, rmax), f"{name} ({b},{h}): max err {mx:.3e} (ref max {rmax:.3f})"
            assert mean <= 4e-3 * max(rmean, 1e-3), f"{name} ({b},{h}): mean err {mean:.3e}"
