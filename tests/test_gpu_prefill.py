"""Prefill parity: the CUDA kernels through the C ABI against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_fattn_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import as_np, check, nan_outputs, need_gpu, tile_edge_samples

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    return need_gpu()


def _run(fa, x, fp32=False):
    dev = torch.device("cuda")
    if fp32:
        q, k, v = x.q32.to(dev), x.k32.to(dev), x.v32.to(dev)
    else:
        q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    cu = x.cu_seqlens.to(dev) if x.varlen else None
    o, lse = fa.fwd(q, k, v, causal=x.causal, scale=x.scale, cu_seqlens=cu,
                    max_seqlen=x.max_seqlen if x.varlen else None)
    assert fa.debug_read_status() == 0
    return o, lse


def _ref(x, fp32=False):
    if fp32:
        return orc.attn_fwd(x.q32, x.k32, x.v32, x.scale, x.causal, x.cu_seqlens)
    return orc.attn_fwd(x.q, x.k, x.v, x.scale, x.causal, x.cu_seqlens)


# ------------------------------------------------------------ tiny single head
@pytest.mark.parametrize("fp32", [True, False])
def test_tiny_single_head(fa, fp32):
    """B=1, H=1, N=256, d=64, non-causal, seed 0: fp32 copy to 1e-4, bf16 copy to bf16 tolerances."""
    x = inputs.tiny_config()
    o, lse = _run(fa, x, fp32)
    o_ref, lse_ref = _ref(x, fp32)
    check(o, lse, o_ref, lse_ref, fp32=fp32, what="tiny")


# ------------------------------------------------------------ worked example
@pytest.mark.parametrize("fp32", [True, False])
def test_worked_example_through_gpu(fa, fp32):
    """'FlashAttention, explained' worked row: scores [2,1,3,0] -> weights [0.2369,0.0871,0.6439,0.0321]."""
    d, N = 64, 4
    s = torch.tensor([2.0, 1.0, 3.0, 0.0])
    q = torch.zeros(1, N, 1, d)
    q[..., 0] = 1.0
    k = torch.zeros(1, N, 1, d)
    k[0, :, 0, 0] = s
    v = torch.zeros(1, N, 1, d)
    for j in range(N):
        v[0, j, 0, j] = 1.0
    dt = torch.float32 if fp32 else torch.bfloat16
    o, lse = fa.fwd(q.to(dt).cuda(), k.to(dt).cuda(), v.to(dt).cuda(), causal=False, scale=1.0)
    w = np.array([0.2369, 0.0871, 0.6439, 0.0321])
    og = as_np(o)[0, :, 0, :4]
    tol = 5e-5 + 1e-6 if fp32 else 4e-3
    assert np.max(np.abs(og - w[None, :])) <= tol
    assert np.max(np.abs(as_np(lse)[0, 0] - (3 + math.log(1.5530)))) <= (1e-4 if fp32 else 1e-3)


# ------------------------------------------------------------ multi-tile shapes with ragged tails
CASES = [
    # B, N, Hq, Hkv, d, causal
    (1, 1, 1, 1, 64, True),
    (2, 127, 2, 1, 64, False),
    (1, 129, 2, 2, 128, True),
    (2, 300, 4, 2, 128, True),
    (2, 300, 4, 2, 128, False),
    (1, 513, 8, 1, 64, True),      # MQA
    (1, 384, 4, 4, 64, False),     # MHA, exact multiple of the tile
    (3, 200, 6, 2, 128, True),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal", CASES)
def test_dense_parity(fa, B, N, Hq, Hkv, d, causal):
    x = inputs.prefill_dense(1000 + N + d, B, N, Hq, Hkv, d, causal)
    o, lse = _run(fa, x)
    o_ref, lse_ref = _ref(x)
    check(o, lse, o_ref, lse_ref, what=f"dense {B,N,Hq,Hkv,d,causal}")


@pytest.mark.parametrize("scale", [-0.2, 0.02, 0.4])
@pytest.mark.parametrize("d,causal", [(64, True), (64, False), (128, True), (128, False)])
def test_dense_parity_other_scales(fa, scale, d, causal):
    """Any finite scale is accepted ('scale multiplies Q K^T'): a negative one (the row
    maximum of the scaled scores is then the minimum of Q K^T, and masked keys go to
    +inf before scaling), a small one (nearly uniform weights) and a large one (peaked
    weights), at both head dimensions (d = 64 runs the separate-P schedule), B=2 N=300
    (tiles plus a ragged tail), GQA 4:2."""
    x = inputs.prefill_dense(3000 + d + int(100 * scale), 2, 300, 4, 2, d, causal, scale=scale)
    o, lse = _run(fa, x)
    o_ref, lse_ref = _ref(x)
    check(o, lse, o_ref, lse_ref, what=f"dense scale {scale} d {d} causal {causal}")


@pytest.mark.parametrize("scale", [-0.15, 0.3])
def test_dense_parity_other_scales_fp32(fa, scale):
    x = inputs.prefill_dense(3500 + int(100 * scale), 2, 300, 4, 2, 64, True, dtype=torch.float32, scale=scale)
    o, lse = _run(fa, x, fp32=True)
    o_ref, lse_ref = _ref(x, fp32=True)
    check(o, lse, o_ref, lse_ref, fp32=True, what=f"fp32 scale {scale}")


@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal", CASES[:5])
def test_dense_parity_fp32(fa, B, N, Hq, Hkv, d, causal):
    x = inputs.prefill_dense(2000 + N + d, B, N, Hq, Hkv, d, causal)
    o, lse = _run(fa, x, fp32=True)
    o_ref, lse_ref = _ref(x, fp32=True)
    check(o, lse, o_ref, lse_ref, fp32=True, what=f"fp32 {B,N,Hq,Hkv,d,causal}")


@pytest.mark.parametrize("d,causal", [(64, True), (128, True), (128, False)])
def test_varlen_with_empty_and_ragged_sequences(fa, d, causal):
    x = inputs.prefill_varlen(77, None, 5, 4, 2, d, causal, lengths=[130, 0, 1, 257, 64])
    o, lse = _run(fa, x)
    o_ref, lse_ref = _ref(x)
    check(o, lse, o_ref, lse_ref, what=f"varlen d={d}")


def test_varlen_config_full(fa):
    """16 packed sequences, lengths U[128, 2048] (seed 3), H=16, d=64, causal: every row."""
    x = inputs.varlen_config()
    o, lse = _run(fa, x)
    o_ref, lse_ref = _ref(x)
    check(o, lse, o_ref, lse_ref, what="varlen config")


def test_varlen_fp32(fa):
    x = inputs.prefill_varlen(78, None, 3, 2, 1, 64, True, dtype=torch.float32, lengths=[70, 1, 140])
    o, lse = _run(fa, x, fp32=True)
    o_ref, lse_ref = _ref(x, fp32=True)
    check(o, lse, o_ref, lse_ref, fp32=True, what="varlen fp32")


# ------------------------------------------------------------ special cases and invariants
@pytest.mark.parametrize("fp32", [False, True])
def test_causal_first_row_is_v0_bit_exact(fa, fp32):
    x = inputs.prefill_dense(5, 2, 260, 4, 2, 128, causal=True)
    o, _ = _run(fa, x, fp32)
    v = x.v32 if fp32 else x.v
    og = o.cpu()
    for b in range(2):
        for h in range(4):
            assert torch.equal(og[b, 0, h], v[b, 0, h // 2]), (b, h)
    xv = inputs.prefill_varlen(6, None, 3, 2, 2, 64, True, lengths=[5, 300, 1])
    ov, _ = _run(fa, xv)
    ovc = ov.cpu()
    for a in xv.cu_seqlens[:-1].tolist():
        for h in range(2):
            assert torch.equal(ovc[a, h], xv.v[a, h]), (a, h)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_give_mean_of_v(fa, causal):
    """K = 0 makes every score equal: O = mean(V) (causal: prefix means), lse = ln(#keys)."""
    B, N, H, d = 1, 300, 2, 64
    x = inputs.prefill_dense(9, B, N, H, H, d, causal)
    k = torch.zeros_like(x.k)
    o, lse = fa.fwd(x.q.cuda(), k.cuda(), x.v.cuda(), causal=causal, scale=x.scale)
    v = as_np(x.v)
    if causal:
        ref = np.cumsum(v, axis=1) / np.arange(1, N + 1)[None, :, None, None]
        lref = np.log(np.arange(1, N + 1))[None, None, :].repeat(H, axis=1)
    else:
        ref = np.broadcast_to(v.mean(axis=1, keepdims=True), v.shape)
        lref = np.full((B, H, N), math.log(N))
    check(o, lse, ref, lref, what="uniform")


def test_dominant_score_picks_its_value_row(fa):
    """One key scoring far above the rest (gap >= 200 after scaling) -> O = V[that key]."""
    N, d = 200, 64
    q = torch.zeros(1, N, 1, d)
    q[..., 0] = 1.0
    k = torch.zeros(1, N, 1, d)
    k[0, :, 0, 0] = torch.linspace(-2, 2, N)
    k[0, 137, 0, 0] = 256.0
    v = torch.randn(1, N, 1, d, generator=torch.Generator().manual_seed(3))
    o, lse = fa.fwd(q.bfloat16().cuda(), k.bfloat16().cuda(), v.bfloat16().cuda(), causal=False, scale=1.0)
    og = o.cpu()
    for i in range(N):
        assert torch.equal(og[0, i, 0], v.bfloat16()[0, 137, 0])
    assert np.max(np.abs(as_np(lse) - 256.0)) <= 1e-3


def test_joint_kv_permutation_invariance(fa):
    x = inputs.prefill_dense(11, 1, 333, 2, 1, 128, causal=False)
    perm = torch.randperm(333, generator=torch.Generator().manual_seed(1))
    o1, l1 = fa.fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=False, scale=x.scale)
    o2, l2 = fa.fwd(x.q.cuda(), x.k[:, perm].contiguous().cuda(), x.v[:, perm].contiguous().cuda(),
                    causal=False, scale=x.scale)
    o_ref, lse_ref = _ref(x)
    check(o1, l1, o_ref, lse_ref, what="unpermuted")
    check(o2, l2, o_ref, lse_ref, what="permuted")


def test_empty_batch_launches_nothing(fa):
    q = torch.empty(0, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    o, lse = fa.fwd(q, q[:, :, :1], q[:, :, :1], causal=True)
    assert o.numel() == 0 and fa.debug_read_status() == 0


def test_output_guards_untouched(fa):
    """Only O and lse are written: canary words around both stay intact."""
    x = inputs.prefill_dense(12, 2, 200, 4, 2, 128, causal=True)
    pad = 64
    n = x.q.numel()
    buf = torch.full((pad + n + pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((pad + 2 * 4 * 200 + pad,), -7.0, dtype=torch.float32, device="cuda")
    o = buf[pad:pad + n].view(x.q.shape)
    lse = lbuf[pad:pad + 2 * 4 * 200].view(2, 4, 200)
    fa.fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True, scale=x.scale, out=o, lse=lse)
    assert torch.isnan(buf[:pad].float()).all() and torch.isnan(buf[pad + n:].float()).all()
    assert (lbuf[:pad] == -7).all() and (lbuf[pad + 1600:] == -7).all()
    o_ref, lse_ref = _ref(x)
    check(o, lse, o_ref, lse_ref, what="guarded")


# ------------------------------------------------------------ the full-size workloads
def _full_size_check(fa, x, what):
    """The launch the bench times, on NaN-filled outputs: every row must be written
    (finite), causal row 0 must be V[0] bit for bit, and the oracle is compared at
    both edge rows of every (sequence, head, 128-row tile) plus random rows, so every
    work item of the schedule (each a pair of tiles) is checked."""
    B, N, Hq = x.q.shape[0], x.q.shape[1], x.q.shape[2]
    o, lse = nan_outputs(x.q.shape, (B, Hq, N))
    fa.fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=x.causal, scale=x.scale, out=o, lse=lse)
    assert fa.debug_read_status() == 0
    assert torch.isfinite(o.float()).all(), f"{what}: rows left unwritten (NaN)"
    assert torch.isfinite(lse).all(), f"{what}: lse entries left unwritten (NaN)"
    G = x.hq // x.hkv
    v0 = x.v[:, 0].cuda()[:, torch.arange(Hq, device="cuda") // G]
    assert torch.equal(o[:, 0], v0)
    smp = tile_edge_samples(B, Hq, N, np.random.default_rng(N))
    o_ref, lse_ref = orc.attn_fwd_rows(x.q, x.k, x.v, x.scale, x.causal, smp)
    bi, hi, ii = (torch.as_tensor(smp[:, c], device="cuda") for c in range(3))
    check(o[bi, ii, hi], lse[bi, hi, ii], o_ref, lse_ref, what=what)


def test_causal_mha_config_every_item(fa):
    """B=4, Hq=Hkv=32, N=4096, d=128, causal, seed 1 (the benchmarked launch)."""
    _full_size_check(fa, inputs.causal_mha_config(), "causal MHA config")


def test_long_gqa_config_every_item(fa):
    """B=1, Hq=32, Hkv=8, N=32768, d=128, causal, seed 2."""
    _full_size_check(fa, inputs.long_gqa_config(), "long GQA config")


def test_varlen_config_nan_filled(fa):
    """The varlen workload (16 packed sequences, H=16, d=64) on NaN-filled outputs:
    every row written, every row equal to the oracle."""
    x = inputs.varlen_config()
    T, H = x.q.shape[0], x.q.shape[1]
    o, lse = nan_outputs(x.q.shape, (H, T))
    fa.fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True, scale=x.scale, cu_seqlens=x.cu_seqlens.cuda(),
           max_seqlen=x.max_seqlen, out=o, lse=lse)
    assert fa.debug_read_status() == 0
    o_ref, lse_ref = _ref(x)
    check(o, lse, o_ref, lse_ref, what="varlen config (NaN-filled outputs)")


def _jump_inputs(N, H, d, jumps, step, seed):
    """q = e_0 (scale 1), so a key's score is its k[..., 0]: every key of tile t of head h
    scores `step` times the number of head h's jump tiles <= t. V of a key = (its tile
    index + 1) / 8 plus 0.02 N(0, 1) noise (|O| <= 1, where the bf16 tolerances hold)."""
    g = torch.Generator().manual_seed(seed)
    q = torch.zeros(1, N, H, d)
    q[..., 0] = 1.0
    k = torch.zeros(1, N, H, d)
    tile = torch.arange(N) // 128
    for h, js in enumerate(jumps):
        k[0, :, h, 0] = step * sum((tile >= t).float() for t in js)
    v = (tile[None, :, None, None].float() + 1.0) / 8 + 0.02 * torch.randn(1, N, H, d, generator=g)
    return q, k, v


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_lazy_rescale_after_mass_jumps(fa, d, causal):
    """Whole key tiles (3 and 7 for head 0, 1 and 5 for head 1) score 5.75 above the tiles
    before them: the running max rises by 8.3 > 8 in log2 units twice, so O is rescaled
    while the earlier tiles still hold about 1 % of the weight, and V grows with the tile
    index. A rescale that missed or double-counted one P V product (one still in flight
    when O is scaled) moves O by about 0.8."""
    q, k, v = _jump_inputs(1024, 2, d, [(3, 7), (1, 5)], 5.75, 41)
    qb, kb, vb = q.bfloat16(), k.bfloat16(), v.bfloat16()
    o, lse = fa.fwd(qb.cuda(), kb.cuda(), vb.cuda(), causal=causal, scale=1.0)
    assert fa.debug_read_status() == 0
    o_ref, lse_ref = orc.attn_fwd(qb, kb, vb, 1.0, causal)
    check(o, lse, o_ref, lse_ref, what=f"rescale d={d} causal={causal}")


def test_binding_rejects_tensors_off_the_current_device(fa):
    """The library launches on the current device: tensors (or a stream) on another
    device are refused before any launch, as are tensors split across devices."""
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    q = torch.zeros(1, 128, 1, 64, dtype=torch.bfloat16, device="cuda:1")
    with pytest.raises(ValueError):
        fa.fwd(q, q, q)
    with pytest.raises(ValueError):
        fa.fwd(q.to("cuda:0"), q, q)
    with torch.cuda.device(1):
        o, _ = fa.fwd(q, q, q)
        assert o.device == q.device
