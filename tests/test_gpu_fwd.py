"""GPU parity of the forward kernel against the float64 oracle (through the C ABI)."""

import numpy as np
import pytest

import oracle
from attn_inputs import BASE_SEED, WORKLOADS, seed_for, sweep_points
from gpu_util import TOL_O, TOL_LSE, inputs, to_device, to_host64, scale_f32, sampled_pairs, sampled_rows

pytestmark = pytest.mark.gpu


def run_fwd(cuda_lib, x, causal, scale):
    import exact_softmax_attention_fa_gb300 as fa
    q, k, v = (to_device(x[n]) for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    assert fa.fa_get_device_status() == 0
    return o, lse


def check_full(cuda_lib, B, H, N, d, causal, seed):
    scale = scale_f32(d)
    x, f = inputs(B, H, N, d, seed, tensors=("q", "k", "v"))
    o, lse = run_fwd(cuda_lib, x, causal, scale)
    o_ref, lse_ref = oracle.attention_forward(f["q"], f["k"], f["v"], causal, scale)
    err_o = np.abs(to_host64(o) - o_ref).max()
    err_l = np.abs(to_host64(lse) - lse_ref).max()
    assert err_o <= TOL_O, (B, H, N, d, causal, err_o)
    assert err_l <= TOL_LSE, (B, H, N, d, causal, err_l)
    return err_o, err_l


def test_tiny_forward(cuda_lib):
    w = WORKLOADS["tiny_fwd"]
    check_full(cuda_lib, w["B"], w["H"], w["N"], w["d"], w["causal"], seed_for(w))


def test_small_causal_forward(cuda_lib):
    w = WORKLOADS["small_causal_fwdbwd"]
    check_full(cuda_lib, w["B"], w["H"], w["N"], w["d"], w["causal"], seed_for(w))


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 7, 127, 128, 129, 200, 255, 256, 257, 383, 640])
def test_ragged_shapes(cuda_lib, d, causal, N):
    check_full(cuda_lib, 1, 2, N, d, causal, BASE_SEED + 100 + N)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_several_tiles_with_tail(cuda_lib, d, causal):
    check_full(cuda_lib, 2, 3, 1000, d, causal, BASE_SEED + 7)


def test_forward_is_deterministic(cuda_lib):
    x, _ = inputs(1, 4, 1500, 128, BASE_SEED + 9, tensors=("q", "k", "v"))
    o1, l1 = run_fwd(cuda_lib, x, True, scale_f32(128))
    o2, l2 = run_fwd(cuda_lib, x, True, scale_f32(128))
    import torch
    assert bool((o1.view(torch.int16) == o2.view(torch.int16)).all())
    assert bool((l1.view(torch.int32) == l2.view(torch.int32)).all())


def test_equal_logits_closed_form(cuda_lib):
    """Q = 0: O is the (causal-prefix) mean of V and L = log(count)."""
    import torch
    import exact_softmax_attention_fa_gb300 as fa
    B, H, N, d = 1, 2, 300, 64
    x, f = inputs(B, H, N, d, BASE_SEED + 11, tensors=("k", "v"))
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    for causal in (False, True):
        o, lse = fa.forward(q, to_device(x["k"]), to_device(x["v"]), causal=causal, scale=scale_f32(d))
        if causal:
            cnt = np.arange(1, N + 1)
            o_ref = np.cumsum(f["v"], axis=2) / cnt[:, None]
            l_ref = np.log(cnt)
        else:
            o_ref = np.broadcast_to(f["v"].mean(axis=2, keepdims=True), f["v"].shape)
            l_ref = np.full(N, np.log(N))
        assert np.abs(to_host64(o) - o_ref).max() <= TOL_O
        assert np.abs(to_host64(lse) - l_ref).max() <= TOL_LSE


def check_sampled(cuda_lib, B, H, N, d, causal, seed, **kw):
    scale = scale_f32(d)
    x, f = inputs(B, H, N, d, seed, tensors=("q", "k", "v"), **kw)
    o, lse = run_fwd(cuda_lib, x, causal, scale)
    o_h, l_h = to_host64(o), to_host64(lse)
    worst_o = worst_l = 0.0
    for (b, h) in sampled_pairs(B, H, seed):
        rows = sampled_rows(N, seed + b * H + h)
        o_ref, l_ref = oracle.attention_forward_rows(f["q"][b, h], f["k"][b, h], f["v"][b, h], rows, causal, scale)
        worst_o = max(worst_o, np.abs(o_h[b, h, rows] - o_ref).max())
        worst_l = max(worst_l, np.abs(l_h[b, h, rows] - l_ref).max())
    assert worst_o <= TOL_O, worst_o
    assert worst_l <= TOL_LSE, worst_l
    assert np.isfinite(o_h).all() and np.isfinite(l_h).all()


@pytest.mark.parametrize("name,p", [pt for pt in sweep_points() if pt[1]["N"] in (512, 4096, 16384)],
                         ids=lambda v: v if isinstance(v, str) else "")
def test_sweep_points_sampled(cuda_lib, name, p):
    check_sampled(cuda_lib, p["B"], p["H"], p["N"], p["d"], p["causal"], seed_for(p))


def test_long_causal_peaked_sampled(cuda_lib):
    w = WORKLOADS["long_causal_peaked"]
    check_sampled(cuda_lib, w["B"], w["H"], w["N"], w["d"], w["causal"], seed_for(w), peaked_frac=w["peaked_frac"])


def test_wide_head_d256_sampled(cuda_lib):
    w = WORKLOADS["wide_head_d256"]
    check_sampled(cuda_lib, w["B"], w["H"], w["N"], w["d"], w["causal"], seed_for(w))


def test_persistent_ctas_with_several_half_empty_items():
    # N = 300 gives 3 query tiles per head, so every head's last item has an
    # empty second tile slot; with 304 heads a CTA takes two such items in a
    # row (causal items come longest first). The idle slot must not run ahead.
    import exact_softmax_attention_fa_gb300 as fa
    from attn_inputs import BASE_SEED
    x, f = inputs(1, 304, 300, 64, BASE_SEED + 900, tensors=("q", "k", "v"))
    o, lse = fa.forward(to_device(x["q"]), to_device(x["k"]), to_device(x["v"]), causal=True, scale=scale_f32(64))
    assert fa.fa_get_device_status() == 0
    o_ref, lse_ref = oracle.attention_forward(f["q"], f["k"], f["v"], True, scale_f32(64))
    assert np.abs(to_host64(o) - o_ref).max() <= TOL_O
    assert np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max() <= TOL_LSE
