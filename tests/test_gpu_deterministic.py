"""GPU parity and bitwise reproducibility of the deterministic backward
(fa_bwd_deterministic, fa_bwd_gqa_deterministic): dQ summed on chip per query
tile in key order instead of with atomic adds."""

import numpy as np
import pytest

import oracle
from attn_inputs import BASE_SEED, WORKLOADS, seed_for
from gpu_util import TOL_GRAD_REL, inputs, scale_f32, to_device, to_host64

pytestmark = pytest.mark.gpu


def rel_err(got, ref):
    return np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-3)


def grouped_inputs(B, Hq, Hkv, N, d, seed):
    xq, fq = inputs(B, Hq, N, d, seed, tensors=("q", "do"))
    xk, fk = inputs(B, Hkv, N, d, seed + 1, tensors=("k", "v"))
    return {**xq, **xk}, {**fq, **fk}


def run(x, causal, scale, deterministic=True):
    import exact_softmax_attention_fa_gb300 as fa
    q, k, v, do = (to_device(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    grads = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, deterministic=deterministic)
    assert fa.fa_get_device_status() == 0
    return grads


def check(x, f, causal, d):
    scale = scale_f32(d)
    grads = run(x, causal, scale)
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        e = rel_err(to_host64(g), r)
        assert e <= TOL_GRAD_REL, (name, e)
    return grads


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 65, 128, 129, 300, 1000])
def test_deterministic_parity(d, causal, N):
    x, f = inputs(2, 3, N, d, BASE_SEED + 600 + N)
    check(x, f, causal, d)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (6, 1)])
def test_deterministic_grouped_parity(d, causal, Hq, Hkv):
    x, f = grouped_inputs(2, Hq, Hkv, 333, d, BASE_SEED + 650 + Hq)
    check(x, f, causal, d)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_bitwise_reproducible(d, causal):
    import torch
    x, _ = inputs(2, 4, 1500, d, BASE_SEED + 700)
    a = run(x, causal, scale_f32(d))
    b = run(x, causal, scale_f32(d))
    for t1, t2 in zip(a, b):
        assert torch.equal(t1, t2)


def _atomic_phases(x, B, H, N, d, causal, scale):
    """The exported atomic-dQ phases in order: preprocess, main (dK, dV and
    the fp32 dQ accumulation with reductions), postprocess (dq = bf16 of the
    accumulator). At d = 128 fa_bwd itself runs the per-query-tile dQ path, so
    these phases are reached only through their own entry points."""
    import exact_softmax_attention_fa_gb300 as fa
    import torch
    q, k, v, do = (to_device(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    fa.fa_bwd_preprocess(o, lse, do, ws)
    fa.fa_bwd_main(q, k, v, do, dk, dv, causal, scale, ws)
    fa.fa_bwd_postprocess(dq, ws)
    assert fa.fa_get_device_status() == 0
    return dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 1000])
def test_atomic_phases_parity(d, causal, N):
    # the atomic-dQ main kernel against the oracle, at the head dimension
    # where fa_bwd does not run it (d = 128) and at d = 64 where it does
    B, H = 2, 3
    x, f = inputs(B, H, N, d, BASE_SEED + 710 + N)
    scale = scale_f32(d)
    grads = _atomic_phases(x, B, H, N, d, causal, scale)
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        e = rel_err(to_host64(g), r)
        assert e <= TOL_GRAD_REL, (name, e)


@pytest.mark.parametrize("causal", [False, True])
def test_atomic_phases_sweep_point_sampled_heads(causal):
    # the pages' d = 128 microbenchmark point (B = 2, H = 16, N = 8192); the
    # oracle computes the sampled heads, whose dq, dk and dv are compared whole
    from gpu_util import sampled_pairs
    B, H, N, d = 2, 16, 8192, 128
    x, f = inputs(B, H, N, d, BASE_SEED + 715)
    scale = scale_f32(d)
    heads = sampled_pairs(B, H, BASE_SEED + 716, n_random=1)
    grads = _atomic_phases(x, B, H, N, d, causal, scale)
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale, heads=heads)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        host = to_host64(g)
        got = np.stack([host[b, h] for b, h in heads])
        want = np.stack([r[b, h] for b, h in heads])
        assert rel_err(got, want) <= TOL_GRAD_REL, name


def test_several_thousand_rows_sampled_heads():
    # the oracle computes only the sampled heads: compare those of every gradient
    x, f = inputs(1, 4, 4096, 128, BASE_SEED + 720)
    scale = scale_f32(128)
    heads = [(0, 0), (0, 3)]
    grads = run(x, True, scale)
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], True, scale, heads=heads)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        got = np.stack([to_host64(g)[b, h] for b, h in heads])
        want = np.stack([r[b, h] for b, h in heads])
        assert rel_err(got, want) <= TOL_GRAD_REL, name


def test_wide_head_d256_sampled_heads():
    # the d = 256 configuration (B = 1, H = 2, N = 16384), causal and not;
    # the oracle computes one head, compared whole in every gradient
    w = WORKLOADS["wide_head_d256"]
    for causal in (False, True):
        x, f = inputs(w["B"], w["H"], w["N"], w["d"], seed_for(w))
        scale = scale_f32(w["d"])
        heads = [(0, 1)]
        grads = run(x, causal, scale)
        ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale, heads=heads)
        for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
            got = np.stack([to_host64(g)[b, h] for b, h in heads])
            want = np.stack([r[b, h] for b, h in heads])
            assert rel_err(got, want) <= TOL_GRAD_REL, (causal, name)


@pytest.mark.parametrize("pre", ["fa_bwd_preprocess_stats", "fa_bwd_preprocess"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_phases_compose_to_the_deterministic_backward(d, pre):
    import exact_softmax_attention_fa_gb300 as fa
    import torch
    x, _ = inputs(1, 3, 700, d, BASE_SEED + 740)
    q, k, v, do = (to_device(x[n]) for n in ("q", "k", "v", "do"))
    scale = scale_f32(d)
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    ws = torch.empty(fa.fa_bwd_workspace_size(1, 3, 700, d), dtype=torch.uint8, device="cuda")
    a = [torch.empty_like(q) for _ in range(3)]
    b = [torch.empty_like(q) for _ in range(3)]
    fa.fa_bwd_deterministic(q, k, v, o, lse, do, *a, True, scale, ws)
    getattr(fa, pre)(o, lse, do, ws)  # the accumulator the full preprocess zeroes is not read
    fa.fa_bwd_dkdv(q, k, v, do, b[1], b[2], True, scale, ws)
    fa.fa_bwd_dq(q, k, v, do, b[0], True, scale, ws)
    assert fa.fa_get_device_status() == 0
    for t1, t2 in zip(a, b):
        assert torch.equal(t1, t2)


def test_default_backward_at_d128_is_the_deterministic_one():
    import exact_softmax_attention_fa_gb300 as fa
    import torch
    x, _ = inputs(2, 2, 555, 128, BASE_SEED + 750)
    q, k, v, do = (to_device(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=False, scale=0.1)
    a = fa.backward(q, k, v, o, lse, do, causal=False, scale=0.1)
    b = fa.backward(q, k, v, o, lse, do, causal=False, scale=0.1, deterministic=True)
    for t1, t2 in zip(a, b):
        assert torch.equal(t1, t2)
