"""Attention backward ('The backward pass recomputes instead of reading'): the CUDA
kernels through the C ABI against the fp64 oracle's gradients."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_fattn_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import as_np, need_gpu, tile_edge_samples

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
    # shorter than one tile: most of the per-row vectors are padding (-inf, 0)
    (2, 17, 2, 1, 128, True),
    (1, 1, 2, 2, 64, False),
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


@pytest.mark.parametrize("scale,d", [(-0.1, 128), (0.3, 64)])
def test_backward_parity_other_scales(fa, scale, d):
    """dQ = scale dS K, dK = scale dS^T Q with a negative and a large scale (B=2, N=300,
    GQA 4:2, causal)."""
    x = inputs.prefill_dense(4500 + d, 2, 300, 4, 2, d, True, scale=scale)
    g = torch.Generator("cpu").manual_seed(4600 + d)
    do = torch.randn((2, 300, 4, d), generator=g).to(torch.bfloat16)
    q, k, v, dog = x.q.cuda(), x.k.cuda(), x.v.cuda(), do.cuda()
    o, lse = fa.fwd(q, k, v, causal=True, scale=scale)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, dog, causal=True, scale=scale)
    assert fa.debug_read_status() == 0
    rq, rk, rv = orc.attn_bwd(x.q, x.k, x.v, do, scale, True)
    for name, a, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        mx, mean, rmax, rmean = _grad_err(a, r)
        print(name, f"max {mx:.3e} mean {mean:.3e} | ref max {rmax:.3f} mean {rmean:.3f}")
        assert np.all(np.isfinite(as_np(a)))
        assert mx <= 2e-2 * max(1.0, rmax), f"{name}: max err {mx:.3e} (ref max {rmax:.3f})"
        assert mean <= 4e-3 * max(rmean, 1e-3), f"{name}: mean err {mean:.3e} (ref mean {rmean:.3f})"


def test_backward_full_size_every_item(fa):
    """The bench's workload (causal MHA B=4 H=32 N=4096 d=128) in the launch the bench
    times, on NaN-filled gradient buffers: every entry must be written, and the
    oracle's gradients are compared at both edge rows of every (sequence, head,
    128-row query tile) for dQ (the dQ pass's items) and of every (sequence, KV head,
    128-key tile) for dK and dV (the dK/dV pass's items), plus random rows."""
    x = inputs.causal_mha_config()
    B, N, H, d = x.q.shape
    g = torch.Generator("cpu").manual_seed(5)
    do = torch.randn((B, N, H, d), generator=g).to(torch.bfloat16)
    q, k, v, dog = x.q.cuda(), x.k.cuda(), x.v.cuda(), do.cuda()
    o, lse = fa.fwd(q, k, v, causal=True, scale=x.scale)
    nan = lambda t: torch.full_like(t, float("nan"))
    dq, dk, dv = nan(q), nan(k), nan(v)
    fa.bwd(q, k, v, o, lse, dog, causal=True, scale=x.scale, dq=dq, dk=dk, dv=dv)
    assert fa.debug_read_status() == 0
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.isfinite(t.float()).all(), f"{name}: entries left unwritten (NaN)"
    rng = np.random.default_rng(6)
    sq = tile_edge_samples(B, H, N, rng, extra=128)
    skv = tile_edge_samples(B, x.hkv, N, rng, extra=128)
    rq, rk, rv = orc.attn_bwd_rows(x.q, x.k, x.v, do, x.scale, True, sq, skv)
    pick = lambda t, smp: t[tuple(torch.as_tensor(smp[:, c], device="cuda") for c in (0, 2, 1))]
    for name, a, r in (("dq", pick(dq, sq), rq), ("dk", pick(dk, skv), rk), ("dv", pick(dv, skv), rv)):
        mx, mean, rmax, rmean = _grad_err(a, r)
        print(name, f"max {mx:.3e} mean {mean:.3e} | ref max {rmax:.3f} mean {rmean:.3f}")
        assert mx <= 2e-2 * max(1.0, rmax), f"{name}: max err {mx:.3e} (ref max {rmax:.3f})"
        assert mean <= 4e-3 * max(rmean, 1e-3), f"{name}: mean err {mean:.3e} (ref mean {rmean:.3f})"
