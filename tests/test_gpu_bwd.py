"""GPU parity of the backward kernels against the float64 oracle (through the C ABI)."""

import numpy as np
import pytest

import oracle
from attn_inputs import BASE_SEED, WORKLOADS, seed_for, sweep_points
from gpu_util import TOL_GRAD_REL, inputs, to_device, to_host64, scale_f32, sampled_pairs, sampled_rows

pytestmark = pytest.mark.gpu


def run_fwd_bwd(x, causal, scale):
    import exact_softmax_attention_fa_gb300 as fa
    q, k, v, do = (to_device(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    assert fa.fa_get_device_status() == 0
    return (o, lse), (dq, dk, dv)


def rel_err(got, ref):
    """max|err| / max|ref|, with max|ref| floored at 1e-3: for N = 1 the exact dQ
    and dK vanish identically (P = 1 so dS = P o (dP - D) = 0) and only rounding
    noise remains."""
    return np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-3)


def check_full(B, H, N, d, causal, seed):
    scale = scale_f32(d)
    x, f = inputs(B, H, N, d, seed)
    _, grads = run_fwd_bwd(x, causal, scale)
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    errs = []
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        e = rel_err(to_host64(g), r)
        errs.append(e)
        assert e <= TOL_GRAD_REL, (name, B, H, N, d, causal, e)
    return errs


def test_small_causal_fwd_bwd():
    w = WORKLOADS["small_causal_fwdbwd"]
    check_full(w["B"], w["H"], w["N"], w["d"], w["causal"], seed_for(w))


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 63, 64, 65, 127, 128, 129, 200, 256, 383, 640])
def test_ragged_shapes(d, causal, N):
    check_full(1, 2, N, d, causal, BASE_SEED + 200 + N)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_several_tiles_with_tail(d, causal):
    check_full(2, 3, 1000, d, causal, BASE_SEED + 17)


def test_dk_dv_deterministic():
    x, _ = inputs(1, 3, 1100, 128, BASE_SEED + 19)
    _, g1 = run_fwd_bwd(x, True, scale_f32(128))
    _, g2 = run_fwd_bwd(x, True, scale_f32(128))
    import torch
    for a, b in zip(g1[1:], g2[1:]):
        assert bool((a.view(torch.int16) == b.view(torch.int16)).all())


def check_sampled(B, H, N, d, causal, seed, n_random=1, **kw):
    """dK, dV in full and dQ on sampled rows for sampled heads; identities on all heads."""
    scale = scale_f32(d)
    x, f = inputs(B, H, N, d, seed, **kw)
    _, (dq, dk, dv) = run_fwd_bwd(x, causal, scale)
    dq_h, dk_h, dv_h = to_host64(dq), to_host64(dk), to_host64(dv)
    assert np.isfinite(dq_h).all() and np.isfinite(dk_h).all() and np.isfinite(dv_h).all()
    for (b, h) in sampled_pairs(B, H, seed, n_random=n_random):
        rq, rk, rv = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale, heads=[(b, h)])
        rows = sampled_rows(N, seed + 31 * b + h)
        assert rel_err(dk_h[b, h], rk[b, h]) <= TOL_GRAD_REL
        assert rel_err(dv_h[b, h], rv[b, h]) <= TOL_GRAD_REL
        assert rel_err(dq_h[b, h, rows], rq[b, h, rows]) <= TOL_GRAD_REL
    # Identities that hold for every head: sum_j dK_j = 0, sum_j dV_j = sum_i dO_i.
    do_sum = f["do"].sum(axis=2)
    assert np.abs(dv_h.sum(axis=2) - do_sum).max() <= 2e-2 * np.abs(dv_h).sum(axis=2).max()
    assert np.abs(dk_h.sum(axis=2)).max() <= 2e-2 * np.abs(dk_h).sum(axis=2).max()


@pytest.mark.parametrize("name,p", [pt for pt in sweep_points() if pt[1]["N"] in (512, 8192)],
                         ids=lambda v: v if isinstance(v, str) else "")
def test_sweep_points_sampled(name, p):
    check_sampled(p["B"], p["H"], p["N"], p["d"], p["causal"], seed_for(p))


def test_long_causal_peaked_sampled():
    w = WORKLOADS["long_causal_peaked"]
    check_sampled(w["B"], w["H"], w["N"], w["d"], w["causal"], seed_for(w), n_random=0,
                  peaked_frac=w["peaked_frac"])


def test_wide_head_d256_sampled():
    w = WORKLOADS["wide_head_d256"]
    check_sampled(w["B"], w["H"], w["N"], w["d"], w["causal"], seed_for(w), n_random=0)
