"""Seeded random shapes through the public forward / backward (and the
deterministic backward): batch, query and K/V head counts, sequence length
(ragged tails, single rows), head dimension, causal mask and scale drawn from
a fixed stream; every output against the float64 oracle.

The scale is drawn between half and once 1/sqrt(d); the fixed bars apply,
plus, for dQ and dK, a bound that comes from the method rather than the
kernels. D = rowsum(dO o O) is formed from the stored bf16 O (as the pages
define it), which differs from the exact O by its bf16 rounding (at most
2^-8 |O|) and the forward's own error, so D_i is off by at most
  delta_i = sum_k |dO_ik| |O_ik - O_ref,ik|   (+ 2^-20 sum_k |dO_ik O_ik| for
                                              D's fp32 sum).
Through dS_ij = P_ij (dP_ij - D_i) that error reaches
  dQ_ic: at most scale delta_i sum_j P_ij |K_jc|,
  dK_jc: at most scale sum_i P_ij delta_i |Q_ic|  (summed over a group),
and dV not at all. With many keys this is far below the 2e-2 bar; with a
handful of keys dS nearly cancels and the bound is a large part of the small
dQ and dK. Each element must lie within 2e-2 of the tensor's largest value
plus its own bound. (With larger scales the bf16 output alone can exceed the
O bar: half an ulp is 2^-8 at |O| in [2, 4), and P's bf16 rounding adds
about |O| 2^-9; a draw at twice 1/sqrt(d) measured 0.0108 on one element.)"""

import numpy as np
import pytest

import oracle
from attn_inputs import BASE_SEED
from gpu_util import TOL_GRAD_REL, TOL_LSE, TOL_O, inputs, to_device, to_host64

pytestmark = pytest.mark.gpu


def draw_cases(n):
    rng = np.random.default_rng(BASE_SEED + 5000)
    cases = []
    for i in range(n):
        d = int(rng.choice([64, 128, 256]))
        B = int(rng.integers(1, 4))
        Hkv = int(rng.integers(1, 4))
        g = int(rng.choice([1, 1, 2, 3, 4]))
        N = int(rng.choice([1, 2, int(rng.integers(3, 128)), 128, int(rng.integers(129, 700))]))
        causal = bool(rng.integers(0, 2))
        scale = float(np.float32(rng.uniform(0.5, 1.0) / np.sqrt(d)))
        det = bool(rng.integers(0, 2)) and d != 256
        cases.append((i, B, Hkv * g, Hkv, N, d, causal, scale, det))
    return cases


def rel_err(got, ref):
    return np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-3)


def d_error_bounds(f, o_gpu, o_ref, causal, scale):
    """Elementwise bounds on dQ and dK from the error of D = rowsum(dO o O)
    formed from the stored O (module docstring); float64 [B, Hq, N, d] and
    [B, Hkv, N, d]."""
    q, k, do = f["q"], f["k"], f["do"]
    g = q.shape[1] // k.shape[1]
    p = oracle.attention_probabilities(q, k, causal, scale)       # [B, Hq, N, N]
    delta = np.sum(np.abs(do) * np.abs(o_gpu - o_ref), axis=-1) + 2.0 ** -20 * np.sum(np.abs(do * o_ref), axis=-1)
    k_rep = np.repeat(np.abs(k), g, axis=1)                        # K/V head of each query head
    bq = scale * delta[..., None] * np.einsum("bhij,bhjc->bhic", p, k_rep)
    bk_q = scale * np.einsum("bhij,bhi,bhic->bhjc", p, delta, np.abs(q))
    bk = bk_q.reshape(q.shape[0], k.shape[1], g, *q.shape[2:]).sum(axis=2)
    return bq, bk


@pytest.mark.parametrize("case", draw_cases(30), ids=lambda c: "B{1}_Hq{2}_Hkv{3}_N{4}_d{5}_c{6:d}_det{8:d}".format(*c))
def test_random_shape(case):
    import exact_softmax_attention_fa_gb300 as fa
    i, B, Hq, Hkv, N, d, causal, scale, det = case
    xq, fq = inputs(B, Hq, N, d, BASE_SEED + 5100 + 2 * i, tensors=("q", "do"))
    xk, fk = inputs(B, Hkv, N, d, BASE_SEED + 5101 + 2 * i, tensors=("k", "v"))
    f = {**fq, **fk}
    q, do = to_device(xq["q"]), to_device(xq["do"])
    k, v = to_device(xk["k"]), to_device(xk["v"])
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, deterministic=det)
    assert fa.fa_get_device_status() == 0
    o_ref, l_ref = oracle.attention_forward(f["q"], f["k"], f["v"], causal, scale)
    assert np.abs(to_host64(o) - o_ref).max() <= TOL_O
    assert np.abs(lse.cpu().numpy().astype(np.float64) - l_ref).max() <= TOL_LSE
    refs = oracle.attention_backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    bq, bk = d_error_bounds(f, to_host64(o), o_ref, causal, scale)
    for name, g, r, b in zip(("dq", "dk", "dv"), (dq, dk, dv), refs, (bq, bk, 0.0)):
        err = np.abs(to_host64(g) - r)
        allowed = TOL_GRAD_REL * max(np.abs(r).max(), 1e-3) + b
        assert np.all(err <= allowed), (name, float(np.max(err - allowed)), rel_err(to_host64(g), r))
