"""Seeded random shapes through the public forward / backward (and the
deterministic backward): batch, query and K/V head counts, sequence length
(ragged tails, single rows), head dimension, causal mask and scale drawn from
a fixed stream; every output against the float64 oracle.

The scale is drawn between half and once 1/sqrt(d); the fixed bars apply,
with one allowance that comes from the method rather than the kernels:
gradients for sequences shorter than 16 keys. D = rowsum(dO o O) uses the
stored bf16 O (as the pages define it), and with a handful of keys
dS = P o (dP - D) sums to almost nothing, so D's rounding is a large part of
the small dQ and dK; the bound there is 0.1 of the tensor's largest value.
(With larger scales the bf16 output alone can exceed the O bar: half an ulp
is 2^-8 at |O| in [2, 4), and P's bf16 rounding adds about |O| 2^-9; a
draw at twice 1/sqrt(d) measured 0.0108 on one element.)"""

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
    tol = TOL_GRAD_REL if N >= 16 else 0.1
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        assert rel_err(to_host64(g), r) <= tol, name
