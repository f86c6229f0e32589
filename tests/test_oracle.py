"""Pins of the float64 oracle against facts the pages and the mathematics fix.

Each test checks one closed form, invariant or independent restatement, chosen
so that a plausible slip in the oracle (a dropped scale, a wrong sign, a
transposed operand, a missing or misplaced causal mask) fails at least one.
"""

import numpy as np
import pytest

import oracle
from oracle import attention as oa
from attn_inputs import make_inputs, bf16_bits_to_f64


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def qkv(B, H, N, d, seed):
    return rand((B, H, N, d), seed), rand((B, H, N, d), seed + 1), rand((B, H, N, d), seed + 2)


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    q, k, _ = qkv(2, 3, 37, 8, 1)
    p = oracle.attention_probabilities(q, k, causal, 0.3)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-13)
    assert (p >= 0).all()
    if causal:
        # entries right of the diagonal are exactly zero
        iu = np.triu_indices(37, 1)
        assert np.all(p[:, :, iu[0], iu[1]] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_value_column_passes_through(causal):
    q, k, v = qkv(1, 2, 29, 6, 2)
    v[..., 3] = 2.5
    o, _ = oracle.attention_forward(q, k, v, causal, 0.7)
    np.testing.assert_allclose(o[..., 3], 2.5, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_logits_give_prefix_mean(causal):
    B, H, N, d = 1, 2, 23, 5
    _, k, v = qkv(B, H, N, d, 3)
    q = np.zeros((B, H, N, d))
    o, lse = oracle.attention_forward(q, k, v, causal, 0.125)
    if causal:
        counts = np.arange(1, N + 1)
        expect = np.cumsum(v, axis=2) / counts[:, None]
        expect_lse = np.log(counts)
    else:
        expect = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
        expect_lse = np.full(N, np.log(N))
    np.testing.assert_allclose(o, expect, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.broadcast_to(expect_lse, lse.shape), rtol=0, atol=1e-13)


def test_causal_row_zero_returns_first_value():
    q, k, v = qkv(2, 2, 17, 4, 4)
    scale = 0.5
    o, lse = oracle.attention_forward(q, k, v, True, scale)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], scale * np.sum(q[:, :, 0] * k[:, :, 0], -1), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_single_key(causal):
    q, k, v = qkv(2, 3, 1, 7, 5)
    o, lse = oracle.attention_forward(q, k, v, causal, 0.9)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[..., 0], 0.9 * np.sum(q[..., 0, :] * k[..., 0, :], -1), atol=1e-13)


def test_two_keys_logistic_closed_form():
    q, k, v = qkv(1, 1, 2, 3, 6)
    scale = 0.8
    o, lse = oracle.attention_forward(q, k, v, False, scale)
    for i in range(2):
        s0 = scale * q[0, 0, i] @ k[0, 0, 0]
        s1 = scale * q[0, 0, i] @ k[0, 0, 1]
        w0 = 1.0 / (1.0 + np.exp(s1 - s0))
        w1 = 1.0 / (1.0 + np.exp(s0 - s1))
        np.testing.assert_allclose(o[0, 0, i], w0 * v[0, 0, 0] + w1 * v[0, 0, 1], atol=1e-14)
        np.testing.assert_allclose(lse[0, 0, i], np.log(np.exp(s0) + np.exp(s1)), atol=1e-13)


def test_joint_key_value_permutation_invariance():
    q, k, v = qkv(1, 2, 31, 8, 7)
    perm = np.random.default_rng(0).permutation(31)
    o1, l1 = oracle.attention_forward(q, k, v, False, 0.35)
    o2, l2 = oracle.attention_forward(q, k[:, :, perm], v[:, :, perm], False, 0.35)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_moves_lse_only(causal):
    q, k, v = qkv(1, 2, 19, 6, 8)
    u = rand((6,), 99)
    scale = 0.4
    o1, l1 = oracle.attention_forward(q, k, v, causal, scale)
    o2, l2 = oracle.attention_forward(q, k + u, v, causal, scale)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, scale * (q @ u), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sum_identities(causal):
    q, k, v = qkv(2, 2, 27, 5, 9)
    do = rand(q.shape, 10)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal, 0.6)
    # rows of dS sum to zero, so the key gradients sum to zero over keys
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    # P^T has columns summing to one, so sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)
    assert np.abs(dq).max() > 0


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("blocks", [(4, 4), (5, 3), (16, 7), (64, 64), (1, 9)])
def test_tiled_variants_agree(causal, blocks):
    B, H, N, d = 2, 2, 29, 6
    q, k, v = qkv(B, H, N, d, 11)
    do = rand(q.shape, 12)
    scale = 0.45
    o, lse = oracle.attention_forward(q, k, v, causal, scale)
    o_t, lse_t = oracle.tiled_forward(q, k, v, causal, scale, *blocks)
    np.testing.assert_allclose(o_t, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_t, lse, rtol=0, atol=1e-12)
    g = oracle.attention_backward(q, k, v, do, causal, scale)
    g_t = oracle.tiled_backward(q, k, v, o, lse, do, causal, scale, *blocks)
    for a, b in zip(g_t, g):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_row_sampled_forward_matches_full():
    q, k, v = qkv(1, 1, 300, 8, 13)
    rows = np.array([0, 1, 17, 255, 256, 299])
    for causal in (False, True):
        o, lse = oracle.attention_forward(q, k, v, causal, 0.3)
        o_r, l_r = oracle.attention_forward_rows(q[0, 0], k[0, 0], v[0, 0], rows, causal, 0.3)
        np.testing.assert_allclose(o_r, o[0, 0, rows], atol=1e-14)
        np.testing.assert_allclose(l_r, lse[0, 0, rows], atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_row_block_parts_sum_to_full(causal):
    q, k, v = qkv(1, 1, 70, 5, 24)
    do = rand(q.shape, 25)
    o, lse = oracle.attention_forward(q, k, v, causal, 0.3)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal, 0.3)
    dk_sum = np.zeros_like(dk[0, 0])
    dv_sum = np.zeros_like(dv[0, 0])
    for rows in (np.arange(0, 23), np.arange(23, 64), np.arange(64, 70)):
        o_r, l_r, dq_r, dk_p, dv_p = oracle.attention_fwd_bwd_rows(q[0, 0], k[0, 0], v[0, 0], do[0, 0], rows,
                                                                   causal, 0.3)
        np.testing.assert_allclose(o_r, o[0, 0, rows], atol=1e-14)
        np.testing.assert_allclose(l_r, lse[0, 0, rows], atol=1e-14)
        np.testing.assert_allclose(dq_r, dq[0, 0, rows], atol=1e-13)
        dk_sum += dk_p
        dv_sum += dv_p
    np.testing.assert_allclose(dk_sum, dk[0, 0], atol=1e-13)
    np.testing.assert_allclose(dv_sum, dv[0, 0], atol=1e-13)


def test_backward_head_subset():
    q, k, v = qkv(2, 2, 9, 3, 14)
    do = rand(q.shape, 15)
    full = oracle.attention_backward(q, k, v, do, True, 0.5)
    part = oracle.attention_backward(q, k, v, do, True, 0.5, heads=[(1, 0)])
    for a, b in zip(part, full):
        np.testing.assert_allclose(a[1, 0], b[1, 0], atol=1e-15)
        assert np.all(a[0] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_torch_float64_sdpa_and_autograd_agree(causal):
    torch = pytest.importorskip("torch")
    B, H, N, d = 2, 3, 33, 8
    q, k, v = qkv(B, H, N, d, 16)
    do = rand(q.shape, 17)
    scale = 0.21
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    to.backward(torch.tensor(do))
    o, lse = oracle.attention_forward(q, k, v, causal, scale)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=0, atol=1e-12)
    s = scale * torch.tensor(q) @ torch.tensor(k).transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal, scale)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_central_finite_differences(causal):
    B, H, N, d = 1, 1, 6, 3
    q, k, v = qkv(B, H, N, d, 18)
    do = rand(q.shape, 19)
    scale = 0.7
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal, scale)

    def loss(q_, k_, v_):
        o, _ = oracle.attention_forward(q_, k_, v_, causal, scale)
        return float(np.sum(o * do))

    h = 1e-6
    for idx, (x, g) in enumerate(((q, dq), (k, dk), (v, dv))):
        num = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            xp = x.copy()
            xm = x.copy()
            xp[pos] += h
            xm[pos] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[idx] = xp
            args_m[idx] = xm
            num[pos] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_lse_bounds_row_max():
    q, k, v = qkv(1, 2, 40, 8, 20)
    scale = 0.5
    _, lse = oracle.attention_forward(q, k, v, True, scale)
    s = scale * q @ np.swapaxes(k, -1, -2)
    s = np.where(np.triu(np.ones((40, 40), bool), 1), -np.inf, s)
    m = s.max(-1)
    assert np.all(lse >= m - 1e-12)
    assert np.all(lse <= m + np.log(np.arange(1, 41)) + 1e-12)


def test_bf16_inputs_promote_exactly():
    x = make_inputs(1, 1, 4, 8, 123, tensors=("q",))["q"]
    f = bf16_bits_to_f64(x)
    # every value has at most 8 significant bits
    mant, _ = np.frexp(f)
    assert np.all(mant * 256 == np.round(mant * 256))


# ---- planted mistakes: each must be caught by a pin above -------------------

def _forward_with(monkeypatch, fake_scores, causal):
    monkeypatch.setattr(oa, "_scores", fake_scores)
    q, k, v = qkv(1, 1, 5, 3, 21)
    return oracle.attention_forward(q, k, v, causal, 0.5), (q, k, v)


def test_planted_missing_scale_is_caught(monkeypatch):
    real = oa._scores

    def no_scale(q_rows, k, row_ids, causal, scale):
        return real(q_rows, k, row_ids, causal, 1.0)

    (o, lse), (q, k, v) = _forward_with(monkeypatch, no_scale, True)
    # causal row 0 pin: L_0 = scale * q_0 . k_0
    assert abs(lse[0, 0, 0] - 0.5 * q[0, 0, 0] @ k[0, 0, 0]) > 1e-6


def test_planted_mask_off_by_one_is_caught(monkeypatch):
    def shifted_mask(q_rows, k, row_ids, causal, scale):
        s = scale * (q_rows @ k.T)
        cols = np.arange(k.shape[0])
        return np.where(cols[None, :] >= row_ids[:, None], -np.inf, s) if causal else s

    with np.errstate(invalid="ignore"):
        (o, _), (q, k, v) = _forward_with(monkeypatch, shifted_mask, True)
    # causal row 0 pin: O_0 = V_0 (the shifted mask leaves row 0 empty -> NaN)
    assert not np.allclose(o[0, 0, 0], v[0, 0, 0])


def test_planted_wrong_softmax_gradient_sign_is_caught(monkeypatch):
    q, k, v = qkv(1, 1, 6, 3, 22)
    do = rand(q.shape, 23)
    real = oa.softmax_rows

    dq, dk, dv = oracle.attention_backward(q, k, v, do, False, 0.5)
    assert np.allclose(dk.sum(axis=2), 0.0, atol=1e-12)

    # a transposed-operand slip in dV breaks sum_j dV_j = sum_i dO_i
    monkeypatch.setattr(oa, "softmax_rows", lambda s: (real(s)[0].T.copy(), real(s)[1]))
    _, _, dv_bad = oracle.attention_backward(q, k, v, do, False, 0.5)
    assert not np.allclose(dv_bad.sum(axis=2), do.sum(axis=2), atol=1e-9)


# ---- grouped / multi-query K/V heads (reading note §5.6) ---------------------

def gqa_inputs(B, Hq, Hkv, N, d, seed):
    return (rand((B, Hq, N, d), seed), rand((B, Hkv, N, d), seed + 1), rand((B, Hkv, N, d), seed + 2),
            rand((B, Hq, N, d), seed + 3))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (6, 1), (3, 3)])
def test_grouped_heads_torch_sdpa_agrees(causal, Hq, Hkv):
    # torch's float64 CPU attention with enable_gqa (query head h reads K/V
    # head h // g) plus autograd, which sums dK, dV over each group
    torch = pytest.importorskip("torch")
    q, k, v, do = gqa_inputs(2, Hq, Hkv, 27, 8, 50)
    scale = 0.3
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale,
                                                          enable_gqa=True)
    to.backward(torch.tensor(do))
    o, _ = oracle.attention_forward(q, k, v, causal, scale)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=0, atol=1e-12)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal, scale)
    assert dk.shape == k.shape and dv.shape == v.shape
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads_equal_replicated_heads(causal):
    # K/V physically repeated along the head axis turn the grouped problem into
    # ordinary multi-head attention; its dK, dV summed over each group of
    # copies are the grouped gradients
    B, Hq, Hkv, N, d = 2, 6, 2, 21, 5
    g = Hq // Hkv
    q, k, v, do = gqa_inputs(B, Hq, Hkv, N, d, 60)
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    o, lse = oracle.attention_forward(q, k, v, causal, 0.4)
    o_r, lse_r = oracle.attention_forward(q, kr, vr, causal, 0.4)
    np.testing.assert_allclose(o, o_r, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse_r, rtol=0, atol=1e-14)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal, 0.4)
    dq_r, dk_r, dv_r = oracle.attention_backward(q, kr, vr, do, causal, 0.4)
    np.testing.assert_allclose(dq, dq_r, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, dk_r.reshape(B, Hkv, g, N, d).sum(2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dv_r.reshape(B, Hkv, g, N, d).sum(2), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads_tiled_variants_agree(causal):
    q, k, v, do = gqa_inputs(1, 4, 2, 45, 6, 70)
    o, lse = oracle.attention_forward(q, k, v, causal, 0.35)
    ot, lset = oracle.tiled_forward(q, k, v, causal, 0.35, 16, 12)
    np.testing.assert_allclose(ot, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lset, lse, rtol=0, atol=1e-12)
    grads = oracle.attention_backward(q, k, v, do, causal, 0.35)
    tgrads = oracle.tiled_backward(q, k, v, o, lse, do, causal, 0.35, 16, 12)
    for a, b in zip(tgrads, grads):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_grouped_heads_finite_differences():
    q, k, v, do = gqa_inputs(1, 2, 1, 5, 2, 80)
    scale = 0.8
    dq, dk, dv = oracle.attention_backward(q, k, v, do, True, scale)

    def loss(k_, v_):
        o, _ = oracle.attention_forward(q, k_, v_, True, scale)
        return float(np.sum(o * do))

    h = 1e-6
    for which, (x, g) in enumerate(((k, dk), (v, dv))):
        num = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[pos] += h
            xm[pos] -= h
            num[pos] = ((loss(xp, v) - loss(xm, v)) if which == 0 else (loss(k, xp) - loss(k, xm))) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_planted_wrong_group_mapping_is_caught(monkeypatch):
    # h mod H_kv instead of floor(h / g) gives a different, valid-looking
    # result that the replicated-heads identity rejects
    B, Hq, Hkv, N, d = 1, 4, 2, 9, 3
    q, k, v, _ = gqa_inputs(B, Hq, Hkv, N, d, 90)
    kr, vr = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    o_r, _ = oracle.attention_forward(q, kr, vr, False, 0.5)
    monkeypatch.setattr(oa, "_kv_head", lambda h, g: h % Hkv)
    o_bad, _ = oracle.attention_forward(q, k, v, False, 0.5)
    assert not np.allclose(o_bad, o_r, atol=1e-6)


# ---- query blocks shorter than the key sequence (decoding against a cache) ---

def test_single_causal_query_sees_every_key():
    # with the mask aligned to the last key, one query is the newest position
    q = rand((2, 3, 1, 8), 100)
    k, v = rand((2, 3, 37, 8), 101), rand((2, 3, 37, 8), 102)
    oc, lc = oracle.attention_forward(q, k, v, True, 0.4)
    on, ln = oracle.attention_forward(q, k, v, False, 0.4)
    np.testing.assert_allclose(oc, on, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lc, ln, rtol=0, atol=1e-15)


@pytest.mark.parametrize("nq", [1, 5, 16, 29])
def test_short_causal_block_is_tail_of_square_problem(nq):
    nk = 29
    q, k, v = qkv(1, 2, nk, 6, 110)
    o_full, l_full = oracle.attention_forward(q, k, v, True, 0.6)
    o, l = oracle.attention_forward(q[:, :, nk - nq:], k, v, True, 0.6)
    np.testing.assert_allclose(o, o_full[:, :, nk - nq:], rtol=0, atol=1e-14)
    np.testing.assert_allclose(l, l_full[:, :, nk - nq:], rtol=0, atol=1e-14)


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 1)])
def test_short_block_torch_sdpa_with_last_key_mask(Hq, Hkv):
    torch = pytest.importorskip("torch")
    nq, nk = 7, 40
    q = rand((2, Hq, nq, 8), 120)
    k, v = rand((2, Hkv, nk, 8), 121), rand((2, Hkv, nk, 8), 122)
    mask = torch.ones(nq, nk, dtype=torch.bool).tril(diagonal=nk - nq)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.3,
                                                          enable_gqa=Hq != Hkv)
    o, _ = oracle.attention_forward(q, k, v, True, 0.3)
    np.testing.assert_allclose(o, to.numpy(), rtol=0, atol=1e-12)
