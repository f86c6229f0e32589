"""Tensors with more than 2^31 elements: every global offset in the kernels
and host code must be 64-bit. B = 1, H = 512, N = 32768, d = 128 puts
2^31 elements (4 GiB of bf16) in each of Q, K, V, O, dO, dQ, dK, dV.

The inputs are eight seeded base heads (the standard generator), each head h
taking base h mod 8 rolled by h positions along the sequence, so every head
differs and a wrapped offset would read another head's values. The oracle
checks sampled rows of O, L and dQ on three heads, including the last one,
and dK, dV of the last head in full."""

import numpy as np
import pytest

import oracle
from attn_inputs import BASE_SEED, make_inputs, bf16_bits_to_f64
from gpu_util import TOL_GRAD_REL, TOL_LSE, TOL_O, scale_f32, to_host64

pytestmark = pytest.mark.gpu

B, H, N, D = 1, 512, 32768, 128
BASES = 8


def head_bits(base, h):
    return np.roll(base[0, h % BASES], h, axis=0)


def test_tensors_past_two_to_the_31_elements():
    import torch
    import exact_softmax_attention_fa_gb300 as fa
    assert H * N * D >= 2 ** 31
    base = make_inputs(1, BASES, N, D, BASE_SEED + 4000)
    dev = {}
    for name in ("q", "k", "v", "do"):
        host = np.empty((B, H, N, D), dtype=np.uint16)
        for h in range(H):
            host[0, h] = head_bits(base[name], h)
        dev[name] = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).to("cuda")
        del host
    scale = scale_f32(D)
    o, lse = fa.forward(dev["q"], dev["k"], dev["v"], causal=False, scale=scale)
    dq, dk, dv = fa.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], causal=False, scale=scale)
    assert fa.fa_get_device_status() == 0
    rng = np.random.default_rng(BASE_SEED + 4001)
    rows = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N), rng.choice(N, 128, replace=False)]))
    for h in (0, 301, H - 1):
        f = {n: bf16_bits_to_f64(head_bits(base[n], h)) for n in ("q", "k", "v", "do")}
        ro, rl, rdq, _, _ = oracle.attention_fwd_bwd_rows(f["q"], f["k"], f["v"], f["do"], rows, False, scale)
        got_o = to_host64(o[0, h, torch.from_numpy(rows).cuda()])
        assert np.abs(got_o - ro).max() <= TOL_O, h
        assert np.abs(lse[0, h].double().cpu().numpy()[rows] - rl).max() <= TOL_LSE, h
        got_dq = to_host64(dq[0, h, torch.from_numpy(rows).cuda()])
        assert np.abs(got_dq - rdq).max() / max(np.abs(rdq).max(), 1e-3) <= TOL_GRAD_REL, h
    # dK, dV of the last head in full: the row-block parts summed over all rows
    h = H - 1
    f = {n: bf16_bits_to_f64(head_bits(base[n], h)) for n in ("q", "k", "v", "do")}
    rk = np.zeros((N, D))
    rv = np.zeros((N, D))
    for r0 in range(0, N, 2048):
        _, _, _, dk_part, dv_part = oracle.attention_fwd_bwd_rows(f["q"], f["k"], f["v"], f["do"],
                                                                   np.arange(r0, r0 + 2048), False, scale)
        rk += dk_part
        rv += dv_part
    for got, ref in ((to_host64(dk[0, h]), rk), (to_host64(dv[0, h]), rv)):
        assert np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-3) <= TOL_GRAD_REL
