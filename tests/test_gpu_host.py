"""GPU checks of fa_fwd_bwd_host: forward and backward of host (CPU) tensors
with the copies overlapped with the kernels. Its outputs are those of the
device-buffer path (fa_fwd, fa_bwd) on the same inputs, and within the parity
bar of the float64 oracle."""

import numpy as np
import pytest

import oracle
from attn_inputs import BASE_SEED
from gpu_util import TOL_GRAD_REL, TOL_LSE, TOL_O, inputs, scale_f32, to_device, to_host64

pytestmark = pytest.mark.gpu


def host_bf16(bits, pinned):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pinned else t.clone()


def run_host(x, causal, scale, pinned=True):
    import torch
    import exact_softmax_attention_fa_gb300 as fa
    B, H, N, d = x["q"].shape
    hq, hk, hv, hdo = (host_bf16(x[n], pinned) for n in ("q", "k", "v", "do"))
    outs = [torch.full((B, H, N, d), float("nan"), dtype=torch.bfloat16) for _ in range(4)]
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32)
    if pinned:
        outs = [t.pin_memory() for t in outs]
        lse = lse.pin_memory()
    o, dq, dk, dv = outs
    buf = torch.empty(fa.fa_fwd_bwd_host_device_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa.fa_fwd_bwd_host(hq, hk, hv, hdo, o, lse, dq, dk, dv, causal, scale, buf)
    assert fa.fa_get_device_status() == 0  # synchronises the stream: the host outputs are final
    return o, lse, dq, dk, dv


def run_device(x, causal, scale):
    import exact_softmax_attention_fa_gb300 as fa
    q, k, v, do = (to_device(x[n]) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    assert fa.fa_get_device_status() == 0
    return tuple(t.cpu() for t in (o, lse, dq, dk, dv))


CASES = [(1, 3, 1000, 128, False), (2, 3, 640, 128, True), (1, 5, 300, 64, False), (1, 2, 384, 64, True),
         (1, 2, 257, 256, False), (1, 1, 129, 128, True)]


@pytest.mark.parametrize("B,H,N,d,causal", CASES)
def test_host_entry_matches_device_path(B, H, N, d, causal):
    import torch
    x, f = inputs(B, H, N, d, BASE_SEED + 900 + N + d)
    scale = scale_f32(d)
    host = run_host(x, causal, scale)
    dev = run_device(x, causal, scale)
    # The forward runs per chunk of heads, each head's tiles on the same
    # kernel: O and L are bit-identical. dK, dV come from kernels without
    # atomics, and at d = 128 so does dQ; elsewhere dQ is summed with atomic
    # adds, whose order varies.
    for name, a, b in zip(("o", "lse", "dk", "dv"), (host[0], host[1], host[3], host[4]),
                          (dev[0], dev[1], dev[3], dev[4])):
        assert torch.equal(a, b), name
    if d == 128:
        assert torch.equal(host[2], dev[2])
    ref_o, ref_l = oracle.attention_forward(f["q"], f["k"], f["v"], causal, scale)
    assert np.abs(to_host64(host[0]) - ref_o).max() <= TOL_O
    assert np.abs(host[1].double().numpy() - ref_l).max() <= TOL_LSE
    ref = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    for name, g, r in zip(("dq", "dk", "dv"), host[2:], ref):
        e = np.abs(to_host64(g) - r).max() / max(np.abs(r).max(), 1e-3)
        assert e <= TOL_GRAD_REL, (name, e)


@pytest.mark.parametrize("causal", [False, True])
def test_host_entry_groups_at_full_tile_count_match_device_path(causal):
    """B*H = 8 heads of N = 8192 at d = 128: the heads flow through four
    groups (1, 3, 3 and 1 heads; the middle ones' forward in two launches),
    each group's dK/dV and dQ kernels run side by side on their own streams
    and workspace, and launches of different groups overlap. Every output
    equals the device path's bit for bit (no atomics at d = 128)."""
    import torch
    B, H, N, d = 1, 8, 8192, 128
    x, _ = inputs(B, H, N, d, BASE_SEED + 980 + int(causal))
    scale = scale_f32(d)
    host = run_host(x, causal, scale)
    dev = run_device(x, causal, scale)
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), host, dev):
        assert torch.equal(a, b), name


def test_host_entry_back_to_back_calls_never_stall():
    """40 back-to-back calls at B=1, H=16, N=16384, d=128 with a 250 ms limit
    on every device-side wait. The host-buffer step overlaps copies and
    kernels of different head groups, which shifts the relative speed of the
    warps inside a CTA; every pipeline wait must still complete (a waiter two
    barrier phases behind its producer would stall until the limit). The
    outputs of the last call equal the device path's."""
    import torch
    import exact_softmax_attention_fa_gb300 as fa
    B, H, N, d = 1, 16, 16384, 128
    x, _ = inputs(B, H, N, d, BASE_SEED + 1400)
    scale = scale_f32(d)
    hq, hk, hv, hdo = (host_bf16(x[n], True) for n in ("q", "k", "v", "do"))
    outs = [torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory() for _ in range(4)]
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    buf = torch.empty(fa.fa_fwd_bwd_host_device_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa.fa_set_wait_limit_ns(250_000_000)
    try:
        stalls = []
        for i in range(40):
            fa.fa_fwd_bwd_host(hq, hk, hv, hdo, outs[0], lse, outs[1], outs[2], outs[3], False, scale, buf)
            word = fa.fa_get_device_status_detail()
            if word[0] != 0:
                stalls.append((i, word))
    finally:
        fa.fa_set_wait_limit_ns(0)
    assert not stalls, stalls
    dev = run_device(x, False, scale)
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), (outs[0], lse, outs[1], outs[2], outs[3]), dev):
        assert torch.equal(a, b), name


def test_host_entry_pageable_buffers():
    """Pageable host tensors give the same outputs (the copies just do not overlap)."""
    import torch
    x, _ = inputs(1, 2, 500, 128, BASE_SEED + 990)
    scale = scale_f32(128)
    a = run_host(x, False, scale, pinned=True)
    b = run_host(x, False, scale, pinned=False)
    for name, s, t in zip(("o", "lse", "dq", "dk", "dv"), a, b):
        assert torch.equal(s, t), name


def test_host_entry_back_to_back_calls_reuse_the_buffer():
    """Two calls on one device buffer, queued without a synchronisation in
    between: the second call's uploads wait for the first call's work."""
    import torch
    import exact_softmax_attention_fa_gb300 as fa
    B, H, N, d = 1, 4, 768, 128
    xs = [inputs(B, H, N, d, BASE_SEED + 995 + i)[0] for i in range(2)]
    scale = scale_f32(d)
    buf = torch.empty(fa.fa_fwd_bwd_host_device_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    results = []
    for x in xs:
        ins = [host_bf16(x[n], True) for n in ("q", "k", "v", "do")]
        outs = [torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory() for _ in range(4)]
        lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        fa.fa_fwd_bwd_host(*ins, outs[0], lse, outs[1], outs[2], outs[3], False, scale, buf)
        results.append((outs[0], lse, outs[1], outs[2], outs[3]))
    assert fa.fa_get_device_status() == 0
    for x, got in zip(xs, results):
        want = run_device(x, False, scale)
        for name, s, t in zip(("o", "lse", "dq", "dk", "dv"), got, want):
            assert torch.equal(s, t), name


@pytest.mark.parametrize("B,H,N,d,causal", [(1, 3, 1000, 128, False), (2, 5, 640, 128, True), (1, 9, 300, 64, True),
                                            (1, 2, 257, 256, False), (1, 1, 65, 64, False)])
def test_forward_host_entry_matches_device_path(B, H, N, d, causal):
    """fa_fwd_host (8 head chunks; fewer when B*H < 8) equals fa_fwd bit for bit."""
    import torch
    import exact_softmax_attention_fa_gb300 as fa
    x, f = inputs(B, H, N, d, BASE_SEED + 1300 + N + d)
    scale = scale_f32(d)
    hq, hk, hv = (host_bf16(x[n], True) for n in ("q", "k", "v"))
    o = torch.full((B, H, N, d), float("nan"), dtype=torch.bfloat16).pin_memory()
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32).pin_memory()
    buf = torch.empty(fa.fa_fwd_host_device_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa.fa_fwd_host(hq, hk, hv, o, lse, causal, scale, buf)
    assert fa.fa_get_device_status() == 0
    q, k, v = (to_device(x[n]) for n in ("q", "k", "v"))
    od, ld = fa.forward(q, k, v, causal=causal, scale=scale)
    assert torch.equal(o, od.cpu())
    assert torch.equal(lse, ld.cpu())
    ref_o, ref_l = oracle.attention_forward(f["q"], f["k"], f["v"], causal, scale)
    assert np.abs(to_host64(o) - ref_o).max() <= TOL_O
    assert np.abs(lse.double().numpy() - ref_l).max() <= TOL_LSE
