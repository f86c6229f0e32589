"""GPU parity of grouped / multi-query K/V heads (reading note 5.6) against the
float64 oracle, through fa_fwd_gqa and fa_bwd_gqa of the C ABI."""

import numpy as np
import pytest

import oracle
from attn_inputs import BASE_SEED
from gpu_util import TOL_GRAD_REL, TOL_LSE, TOL_O, inputs, scale_f32, to_device, to_host64

pytestmark = pytest.mark.gpu


def gqa_inputs(B, Hq, Hkv, N, d, seed):
    """q, do with Hq heads and k, v with Hkv heads, from independent seeded streams."""
    xq, fq = inputs(B, Hq, N, d, seed, tensors=("q", "do"))
    xk, fk = inputs(B, Hkv, N, d, seed + 1, tensors=("k", "v"))
    return {**xq, **xk}, {**fq, **fk}


def rel_err(got, ref):
    return np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-3)


def run(x, causal, scale):
    import exact_softmax_attention_fa_gb300 as fa
    q, k, v, do = (to_device(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    assert fa.fa_get_device_status() == 0
    return (q, k, v, do), (o, lse), (dq, dk, dv)


def check(B, Hq, Hkv, N, d, causal, seed):
    scale = scale_f32(d)
    x, f = gqa_inputs(B, Hq, Hkv, N, d, seed)
    _, (o, lse), grads = run(x, causal, scale)
    o_ref, lse_ref = oracle.attention_forward(f["q"], f["k"], f["v"], causal, scale)
    assert np.abs(to_host64(o) - o_ref).max() <= TOL_O
    assert np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max() <= TOL_LSE
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        assert tuple(g.shape) == r.shape, name
        e = rel_err(to_host64(g), r)
        assert e <= TOL_GRAD_REL, (name, B, Hq, Hkv, N, d, causal, e)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (4, 1), (3, 3)])
def test_grouped_heads_parity(d, causal, Hq, Hkv):
    check(2, Hq, Hkv, 300, d, causal, BASE_SEED + 400 + Hq * 10 + Hkv)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 65, 129])
def test_grouped_heads_ragged(causal, N):
    check(1, 6, 2, N, 128, causal, BASE_SEED + 450 + N)


def test_group_of_eight_several_tiles():
    # 8 query heads on one K/V head: every key tile sums 8 x 8 query tiles
    check(1, 8, 1, 1000, 128, True, BASE_SEED + 460)


def test_mha_through_gqa_entry_is_bitwise_fa_fwd():
    import exact_softmax_attention_fa_gb300 as fa
    import torch
    x, _ = inputs(2, 3, 333, 128, BASE_SEED + 470)
    q, k, v, do = (to_device(x[n]) for n in ("q", "k", "v", "do"))
    o1, l1 = torch.empty_like(q), torch.empty(2, 3, 333, device="cuda")
    o2, l2 = torch.empty_like(q), torch.empty(2, 3, 333, device="cuda")
    fa.fa_fwd(q, k, v, o1, l1, True, 0.1)
    fa.fa_fwd_gqa(q, k, v, o2, l2, True, 0.1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ws = torch.empty(fa.fa_bwd_workspace_size(2, 3, 333, 128), dtype=torch.uint8, device="cuda")
    g1 = [torch.empty_like(q) for _ in range(3)]
    g2 = [torch.empty_like(q) for _ in range(3)]
    fa.fa_bwd(q, k, v, o1, l1, do, *g1, True, 0.1, ws)
    fa.fa_bwd_gqa(q, k, v, o1, l1, do, *g2, True, 0.1, ws)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])  # dK, dV reproducible
    assert fa.fa_get_device_status() == 0


def test_grouped_dk_dv_bitwise_reproducible():
    import torch
    x, _ = gqa_inputs(2, 8, 2, 700, 64, BASE_SEED + 480)
    _, (o, lse), (dq1, dk1, dv1) = run(x, False, scale_f32(64))
    _, _, (dq2, dk2, dv2) = run(x, False, scale_f32(64))
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)


def test_grouped_heads_sum_of_replicated_heads():
    # the grouped dK equals the per-query-head dK of explicitly repeated K/V,
    # summed over each group (both computed by the library)
    import exact_softmax_attention_fa_gb300 as fa
    B, Hq, Hkv, N, d = 1, 4, 2, 256, 64
    x, f = gqa_inputs(B, Hq, Hkv, N, d, BASE_SEED + 490)
    (q, k, v, do), (o, lse), (dq, dk, dv) = run(x, False, scale_f32(d))
    kr, vr = k.repeat_interleave(Hq // Hkv, dim=1).contiguous(), v.repeat_interleave(Hq // Hkv, dim=1).contiguous()
    o_r, lse_r = fa.forward(q, kr, vr, causal=False, scale=scale_f32(d))
    assert (o_r.float() - o.float()).abs().max().item() == 0.0
    _, dk_r, dv_r = fa.backward(q, kr, vr, o_r, lse_r, do, causal=False, scale=scale_f32(d))
    dk_sum = dk_r.float().reshape(B, Hkv, Hq // Hkv, N, d).sum(2)
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], False, scale_f32(d))
    assert rel_err(dk_sum.cpu().numpy().astype(np.float64), ref[1]) <= TOL_GRAD_REL
    assert rel_err(to_host64(dk), ref[1]) <= TOL_GRAD_REL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_split_and_unsplit_groups_agree(causal, d):
    # a workspace of fa_bwd_workspace_size(B, Hq, N, d) bytes leaves no room for
    # partials, so each group stays in one work item; the grouped workspace
    # size lets the library split groups over several items
    import exact_softmax_attention_fa_gb300 as fa
    import torch
    B, Hq, Hkv, N = 2, 8, 2, 520
    scale = scale_f32(d)
    x, f = gqa_inputs(B, Hq, Hkv, N, d, BASE_SEED + 500 + d)
    q, k, v, do = (to_device(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    small = fa.fa_bwd_workspace_size(B, Hq, N, d)
    big = fa.fa_bwd_gqa_workspace_size(B, Hq, Hkv, N, d)
    assert big > small
    outs = []
    for size in (small, big):
        ws = torch.empty(size, dtype=torch.uint8, device="cuda")
        g = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        fa.fa_bwd_gqa(q, k, v, o, lse, do, *g, causal, scale, ws)
        assert fa.fa_get_device_status() == 0
        for name, t, r in zip(("dq", "dk", "dv"), g, ref):
            assert rel_err(to_host64(t), r) <= TOL_GRAD_REL, (name, size)
        outs.append(g)
    for a, b in zip(outs[0][1:], outs[1][1:]):
        assert rel_err(to_host64(a), to_host64(b)) <= 1e-2


@pytest.mark.parametrize("Hq,Hkv,N", [(16, 1, 1024), (2, 2, 4096)])
def test_work_queued_after_the_backward_sees_final_gradients(Hq, Hkv, N):
    """At d = 128 fa_bwd lets its dQ kernel start on SMs the dK/dV pass leaves
    idle; the call must still complete only when both have. With one K/V head
    for 16 query heads the dK/dV pass has a few long work items and the dQ
    kernel many short ones, so the dQ kernel ends first. dk, dv and dq are
    zeroed before every call, and a copy queued on the same stream right
    after the call must equal the final gradients, which match the oracle."""
    import torch
    import exact_softmax_attention_fa_gb300 as fa
    B, d, causal = 1, 128, False
    scale = scale_f32(d)
    x, f = gqa_inputs(B, Hq, Hkv, N, d, BASE_SEED + 470 + Hq)
    q, k, v, do = (to_device(x[n]) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    fa.fa_fwd_gqa(q, k, v, o, lse, causal, scale)
    ws = torch.empty(fa.fa_bwd_gqa_workspace_size(B, Hq, Hkv, N, d), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    copies = []
    for _ in range(4):
        for g in (dq, dk, dv):
            g.zero_()
        fa.fa_bwd_gqa(q, k, v, o, lse, do, dq, dk, dv, causal, scale, ws)
        copies.append(tuple(g.clone() for g in (dq, dk, dv)))
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == 0
    for c in copies:
        for got, final in zip(c, (dq, dk, dv)):
            assert bool((got.view(torch.int16) == final.view(torch.int16)).all())
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        e = rel_err(to_host64(g), r)
        assert e <= TOL_GRAD_REL, (name, Hq, Hkv, N, e)
