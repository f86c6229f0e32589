"""Failure detection without a GPU fault: a bounded device wait that nothing
satisfies gives up, records FA_ERR_TIMEOUT, and the context stays usable."""

import numpy as np
import pytest

import oracle
from gpu_util import TOL_GRAD_REL, TOL_O, inputs, to_device, to_host64, scale_f32

pytestmark = pytest.mark.gpu

FA_ERR_TIMEOUT = 6


def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib):
    import exact_softmax_attention_fa_gb300 as fa
    assert fa.fa_get_device_status() == 0
    fa.fa_debug_timeout_probe(2_000_000)  # 2 ms limit on a barrier no thread arrives at
    assert fa.fa_get_device_status() == FA_ERR_TIMEOUT
    assert fa.fa_get_device_status() == 0  # reading clears the word
    # the context is still usable: a normal forward runs and is correct
    x, f = inputs(1, 1, 256, 64, 77, tensors=("q", "k", "v"))
    o, _ = fa.forward(to_device(x["q"]), to_device(x["k"]), to_device(x["v"]), causal=True, scale=scale_f32(64))
    assert fa.fa_get_device_status() == 0
    o_ref, _ = oracle.attention_forward(f["q"], f["k"], f["v"], True, scale_f32(64))
    assert np.abs(to_host64(o) - o_ref).max() <= TOL_O


def test_status_detail_names_the_waiting_role(cuda_lib):
    """The whole status word: code, role (99 = the probe), block, thread; read and cleared."""
    import exact_softmax_attention_fa_gb300 as fa
    assert fa.fa_get_device_status_detail() == (0, 0, 0, 0)
    fa.fa_debug_timeout_probe(2_000_000)
    code, role, block, _thread = fa.fa_get_device_status_detail()
    assert (code, role, block) == (FA_ERR_TIMEOUT, 99, 0)
    assert fa.fa_get_device_status_detail() == (0, 0, 0, 0)


def test_probe_rejects_bad_limits(cuda_lib):
    import exact_softmax_attention_fa_gb300 as fa
    with pytest.raises(fa.FAError):
        fa.fa_debug_timeout_probe(0)


def test_wait_limit_setter_round_trip(cuda_lib):
    import exact_softmax_attention_fa_gb300 as fa
    fa.fa_set_wait_limit_ns(10_000_000_000)
    x, _ = inputs(1, 2, 300, 128, 78, tensors=("q", "k", "v"))
    fa.forward(to_device(x["q"]), to_device(x["k"]), to_device(x["v"]), causal=False, scale=scale_f32(128))
    assert fa.fa_get_device_status() == 0
    fa.fa_set_wait_limit_ns(0)  # back to the default


# ---------------------------------------------------------------------------
# The real kernels' own bounded waits: with fa_debug_skip_arrival, block 0 of
# a launch leaves out one arrival, so a wait on that barrier gives up after a
# 2 ms limit. The launch must record FA_ERR_TIMEOUT (block 0, a role of that
# kernel), leave the context usable, and the next normal launch must match the
# oracle. Which waiting role gives up first depends on which wait started
# first, so the test accepts any role of the kernel.
# ---------------------------------------------------------------------------
FWD_ROLES = {1, 2, 3}
BWD_ROLES = {11, 12, 13, 14}


def _run_phase(fa, kernel, t, causal, scale, ws):
    q, k, v, do, o, lse, dq, dk, dv = (t[n] for n in ("q", "k", "v", "do", "o", "lse", "dq", "dk", "dv"))
    if kernel == "fwd":
        fa.fa_fwd(q, k, v, o, lse, causal, scale)
    elif kernel == "dkdv":
        fa.fa_bwd_dkdv(q, k, v, do, dk, dv, causal, scale, ws)
    elif kernel == "dq":
        fa.fa_bwd_dq(q, k, v, do, dq, causal, scale, ws)
    elif kernel == "main":
        fa.fa_bwd_main(q, k, v, do, dk, dv, causal, scale, ws)
        fa.fa_bwd_postprocess(dq, ws)
    elif kernel == "bwd":  # the whole call: at d = 128 its dQ kernel overlaps the dK/dV pass
        fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal, scale, ws)


@pytest.mark.parametrize("kernel,role,d", [
    ("fwd", 1, 128), ("fwd", 2, 128), ("fwd", 3, 128), ("fwd", 3, 64),
    ("dkdv", 11, 128), ("dkdv", 12, 128), ("dkdv", 13, 128),
    ("dq", 11, 128), ("dq", 12, 128), ("dq", 13, 64),
    ("main", 11, 64), ("main", 12, 128), ("main", 13, 64), ("main", 14, 128), ("main", 14, 64),
    ("main", 11, 256), ("main", 12, 256), ("main", 13, 256), ("main", 14, 256),
    ("dkdv", 13, 256), ("dq", 11, 256), ("dq", 12, 256), ("dq", 13, 256),
    ("bwd", 11, 128), ("bwd", 12, 128), ("bwd", 13, 128),
])
def test_kernel_wait_gives_up_and_next_launch_is_correct(cuda_lib, kernel, role, d):
    import torch
    import exact_softmax_attention_fa_gb300 as fa
    B, H, N, causal = 1, 3, 700, True
    scale = scale_f32(d)
    x, f = inputs(B, H, N, d, 79 + role)
    t = {n: to_device(x[n]) for n in ("q", "k", "v", "do")}
    t["o"], t["lse"] = fa.forward(t["q"], t["k"], t["v"], causal=causal, scale=scale)
    for n in ("dq", "dk", "dv"):
        t[n] = torch.zeros_like(t["q"])
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa.fa_bwd_preprocess(t["o"], t["lse"], t["do"], ws)
    assert fa.fa_get_device_status_detail() == (0, 0, 0, 0)
    try:
        fa.fa_set_wait_limit_ns(2_000_000)
        fa.fa_debug_skip_arrival(role)
        _run_phase(fa, kernel, t, causal, scale, ws)
        code, where, block, _thread = fa.fa_get_device_status_detail()
    finally:
        fa.fa_debug_skip_arrival(0)
        fa.fa_set_wait_limit_ns(0)
    assert code == FA_ERR_TIMEOUT
    assert where in (FWD_ROLES if kernel == "fwd" else BWD_ROLES), where
    assert block == 0
    # the same launch again, normally: the context works and the result is right
    if kernel != "fwd":
        fa.fa_bwd_preprocess(t["o"], t["lse"], t["do"], ws)
    _run_phase(fa, kernel, t, causal, scale, ws)
    assert fa.fa_get_device_status_detail() == (0, 0, 0, 0)
    if kernel == "fwd":
        o_ref, lse_ref = oracle.attention_forward(f["q"], f["k"], f["v"], causal, scale)
        assert np.abs(to_host64(t["o"]) - o_ref).max() <= TOL_O
        return
    ref = dict(zip(("dq", "dk", "dv"), oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale)))
    names = {"dkdv": ("dk", "dv"), "dq": ("dq",), "main": ("dq", "dk", "dv"), "bwd": ("dq", "dk", "dv")}[kernel]
    for n in names:
        got = to_host64(t[n])
        assert np.abs(got - ref[n]).max() / np.abs(ref[n]).max() <= TOL_GRAD_REL, n


def test_skip_hook_rejects_unknown_roles(cuda_lib):
    import exact_softmax_attention_fa_gb300 as fa
    with pytest.raises(fa.FAError):
        fa.fa_debug_skip_arrival(4)
    fa.fa_debug_skip_arrival(0)
