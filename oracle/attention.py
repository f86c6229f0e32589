"""Float64 CPU oracle for exact softmax attention, forward and backward.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and the CPU-baseline
leg of bench.py may import this module. It shares no code with the CUDA path.

Sources (web pages on FlashAttention-2, cited by title and section):
  [note]    "FlashAttention 2: Faster Attention with Better Parallelism and Work
            Partitioning", reading note on papers.chlience.com
  [atlas]   "FlashAttention", llm-infra-atlas overview
  [summary] "FlashAttention-2: Faster Attention with Better Parallelism and Work
            Partitioning", paper-graph-ui summary

What is computed, per (batch, head), for Q, K, V in R^{N x d}:
  S = scale * Q K^T                     [note] §1, with the 1/sqrt(d) factor of
                                        [atlas] §1 passed in as `scale`
  S_ij = -inf for j > i when causal     [summary] Algorithm 1 walkthrough,
                                        "Causal masking optimization"
  P = softmax(S) row-wise, O = P V      [note] §1
  L_i = m_i + log(sum_j exp(S_ij - m_i)) with m_i = max_j S_ij
                                        [note] §5.2 (natural log)
  Backward by the chain rule:           [note] §5.3, [summary] "The Backward Pass"
    dV = P^T dO, dP = dO V^T,
    dS_i = P_i o (dP_i - <P_i, dP_i>)   (softmax Jacobian applied to dP_i)
    dQ = scale * dS K, dK = scale * dS^T Q   (the scale comes from S = scale*QK^T)
  Grouped / multi-query heads:          [note] §5.6, [summary] "Multi-query and
                                        grouped-query attention"
    K and V may have H_kv heads with H_q = g * H_kv; query head h reads K/V
    head floor(h / g), and dK, dV of a K/V head are the sums over its g query
    heads. g = 1 is ordinary multi-head attention.

attention_forward / attention_backward are the plain definitions: S and P are
materialised (in chunks of query rows, which changes nothing but memory use).
attention_fwd_bwd_rows restates both for a block of query rows of one head
(pinned by summing blocks back to the full result).
tiled_forward / tiled_backward are a second, separately written restatement of
the blocked algorithm (unscaled accumulator with running max and sum, then the
column-block-outer backward with D = rowsum(dO o O)); the tests use them to
cross-check the plain definitions, never the other way round.

Pins (tests/test_oracle.py): rows of P sum to 1; constant V columns pass
through; Q = 0 gives the (causal-prefix) mean of V with L = log(count); causal
row 0 returns V_0 with L_0 = scale q_0.k_0; N = 1 returns V; two keys give the
logistic closed form; non-causal results are invariant under a joint
permutation of K/V rows; shifting every key by u shifts L_i by scale q_i.u and
leaves O unchanged; sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i; the tiled
variants agree to 1e-12; torch's float64 CPU attention plus autograd agrees to
1e-12; central finite differences match the gradients. Grouped K/V heads:
torch's float64 attention with enable_gqa plus autograd agrees; K/V repeated
along the head axis give the same O, L, dQ and, summed over each group, dK and
dV; the tiled variants and finite differences agree. Shorter query blocks
(N_q < N_k, causal mask aligned to the last key): a single causal query equals
the unmasked one; the block equals the last N_q rows of the square causal
problem; torch's float64 attention with the explicit last-key-aligned mask
agrees. Every function here is pinned by at least one of these.
"""

from __future__ import annotations

import numpy as np

_ROW_CHUNK = 256


def _check(q, k, v=None):
    """Promote to float64 and return (q, k, v, g): q is [B, H_q, N_q, d], k and v
    are [B, H_kv, N_k, d] with H_q = g * H_kv ([note] §5.6)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    if q.ndim != 4 or k.ndim != 4 or k.shape[0] != q.shape[0] or k.shape[3] != q.shape[3]:
        raise ValueError("q must be [B, H_q, N_q, d] and k [B, H_kv, N_k, d]")
    if k.shape[1] < 1 or q.shape[1] % k.shape[1] != 0:
        raise ValueError("H_q must be a multiple of H_kv")
    if v is not None:
        v = np.asarray(v, dtype=np.float64)
        if v.shape != k.shape:
            raise ValueError("v must match k")
    return q, k, v, q.shape[1] // k.shape[1]


def _kv_head(h, g):
    """K/V head read by query head h when g query heads share one ([note] §5.6)."""
    return h // g


def _scores(q_rows, k, row_ids, causal, scale):
    """S for the given query rows of one head: scale * q k^T, future keys -> -inf.

    row_ids are the rows' positions on the key axis: query i of N_q sits at
    i + N_k - N_q, so a shorter query block is the last rows of the square
    causal problem (the mask aligned to the last key).
    """
    s = scale * (q_rows @ k.T)
    if causal:
        cols = np.arange(k.shape[0])
        s = np.where(cols[None, :] > row_ids[:, None], -np.inf, s)
    return s


def _key_pos(rows, nq, nk):
    """Positions on the key axis of query rows of an N_q-row block against N_k keys."""
    return rows + (nk - nq)


def softmax_rows(s):
    """Row-wise softmax of a score block and the row log-sum-exp ([note] §5.2)."""
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    total = np.sum(e, axis=1, keepdims=True)
    p = e / total
    lse = (m + np.log(total))[:, 0]
    return p, lse


def attention_probabilities(q, k, causal, scale):
    """The full P = softmax(S) as a [B, H, N, N] array (small inputs only)."""
    q, k, _, g = _check(q, k)
    B, H, N, _d = q.shape
    Nk = k.shape[2]
    out = np.zeros((B, H, N, Nk))
    rows = _key_pos(np.arange(N), N, Nk)
    for b in range(B):
        for h in range(H):
            out[b, h], _ = softmax_rows(_scores(q[b, h], k[b, _kv_head(h, g)], rows, causal, scale))
    return out


def attention_forward(q, k, v, causal, scale):
    """O = softmax(S) V and L = logsumexp(S) per row; returns (O [B,H,N_q,d], L [B,H,N_q]).

    K and V may hold N_k != N_q keys; under a causal mask query i then sees
    keys j <= i + N_k - N_q.
    """
    q, k, v, g = _check(q, k, v)
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            hk = _kv_head(h, g)
            for r0 in range(0, N, _ROW_CHUNK):
                rows = np.arange(r0, min(N, r0 + _ROW_CHUNK))
                p, l_rows = softmax_rows(_scores(q[b, h, rows], k[b, hk], _key_pos(rows, N, k.shape[2]), causal,
                                                 scale))
                o[b, h, rows] = p @ v[b, hk]
                lse[b, h, rows] = l_rows
    return o, lse


def attention_forward_rows(q_bh, k_bh, v_bh, rows, causal, scale):
    """O and L for selected query rows of ONE head (arrays [N, d]); rows are independent."""
    q_bh = np.asarray(q_bh, dtype=np.float64)
    k_bh = np.asarray(k_bh, dtype=np.float64)
    v_bh = np.asarray(v_bh, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    o = np.zeros((len(rows), q_bh.shape[1]))
    lse = np.zeros(len(rows))
    for c0 in range(0, len(rows), _ROW_CHUNK):
        rr = rows[c0:c0 + _ROW_CHUNK]
        p, l_rows = softmax_rows(_scores(q_bh[rr], k_bh, rr, causal, scale))
        o[c0:c0 + len(rr)] = p @ v_bh
        lse[c0:c0 + len(rr)] = l_rows
    return o, lse


def attention_backward(q, k, v, do, causal, scale, heads=None):
    """Gradients (dQ, dK, dV) of sum(O * dO) by the chain rule ([note] §5.3).

    P is rebuilt from S (not from a stored L), and the softmax backward uses
    <P_i, dP_i> directly rather than the rowsum(dO o O) shortcut. `heads`, if
    given, is a list of (b, h) query-head pairs to compute; other heads are
    left zero (and contribute nothing to dK, dV). With grouped K/V heads, dK
    and dV have K's shape and sum the contributions of each group's query
    heads ([note] §5.6).
    """
    q, k, v, g = _check(q, k, v)
    do = np.asarray(do, dtype=np.float64)
    B, H, N, d = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(k)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        hk = _kv_head(h, g)
        for r0 in range(0, N, _ROW_CHUNK):
            rows = np.arange(r0, min(N, r0 + _ROW_CHUNK))
            p, _ = softmax_rows(_scores(q[b, h, rows], k[b, hk], _key_pos(rows, N, k.shape[2]), causal, scale))
            do_rows = do[b, h, rows]
            dv[b, hk] += p.T @ do_rows
            dp = do_rows @ v[b, hk].T
            ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
            dq[b, h, rows] = scale * (ds @ k[b, hk])
            dk[b, hk] += scale * (ds.T @ q[b, h, rows])
    return dq, dk, dv


def attention_fwd_bwd_rows(q_bh, k_bh, v_bh, do_bh, rows, causal, scale):
    """Forward and backward restricted to a block of query rows of ONE head.

    Returns (O_rows, L_rows, dQ_rows, dK_part, dV_part): the outputs and dQ of
    those rows, and their additive contributions to dK and dV. Summing the
    parts over a partition of the rows gives attention_backward's dK and dV;
    this is how a bounded CPU sample of a large workload is timed.
    """
    q_bh, k_bh, v_bh, do_bh = (np.asarray(a, dtype=np.float64) for a in (q_bh, k_bh, v_bh, do_bh))
    rows = np.asarray(rows, dtype=np.int64)
    p, lse = softmax_rows(_scores(q_bh[rows], k_bh, rows, causal, scale))
    o = p @ v_bh
    do_rows = do_bh[rows]
    dv_part = p.T @ do_rows
    dp = do_rows @ v_bh.T
    ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
    dq = scale * (ds @ k_bh)
    dk_part = scale * (ds.T @ q_bh[rows])
    return o, lse, dq, dk_part, dv_part


def tiled_forward(q, k, v, causal, scale, block_rows, block_cols):
    """Blocked forward with an unscaled accumulator ([note] §5.1-5.2,
    [summary] "Algorithm 1 Walkthrough").

    For each query block Q_i: m = -inf, l = 0, acc = 0; for each key block j:
    S_ij = scale Q_i K_j^T (masked), m_new = max(m, rowmax S_ij),
    P~ = exp(S_ij - m_new), l = exp(m - m_new) l + rowsum P~,
    acc = diag(exp(m - m_new)) acc + P~ V_j; finally O_i = acc / l and
    L_i = m + log l. Blocks need not divide N. Causal key blocks entirely
    to the right of the query block are skipped.
    """
    q, k, v, g = _check(q, k, v)
    B, H, N, d = q.shape
    if k.shape[2] != N:
        raise ValueError("the blocked variants take N_q = N_k")
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            kh, vh = k[b, _kv_head(h, g)], v[b, _kv_head(h, g)]
            for i0 in range(0, N, block_rows):
                i1 = min(N, i0 + block_rows)
                qi = q[b, h, i0:i1]
                m = np.full(i1 - i0, -np.inf)
                l_run = np.zeros(i1 - i0)
                acc = np.zeros((i1 - i0, d))
                for j0 in range(0, N, block_cols):
                    if causal and j0 > i1 - 1:
                        break
                    j1 = min(N, j0 + block_cols)
                    s = scale * (qi @ kh[j0:j1].T)
                    if causal:
                        rr = np.arange(i0, i1)[:, None]
                        cc = np.arange(j0, j1)[None, :]
                        s = np.where(cc > rr, -np.inf, s)
                    m_new = np.maximum(m, np.max(s, axis=1))
                    p_tilde = np.exp(s - m_new[:, None])
                    corr = np.exp(m - m_new)
                    l_run = corr * l_run + np.sum(p_tilde, axis=1)
                    acc = corr[:, None] * acc + p_tilde @ vh[j0:j1]
                    m = m_new
                o[b, h, i0:i1] = acc / l_run[:, None]
                lse[b, h, i0:i1] = m + np.log(l_run)
    return o, lse


def tiled_backward(q, k, v, o, lse, do, causal, scale, block_rows, block_cols):
    """Blocked backward, key blocks outer ([note] §5.3, [summary] "The Backward Pass").

    D = rowsum(dO o O); for each key block j: dK_j = dV_j = 0; for each query
    block i: S_ij = scale Q_i K_j^T (masked), P_ij = exp(S_ij - L_i),
    dV_j += P_ij^T dO_i, dP_ij = dO_i V_j^T, dS_ij = P_ij o (dP_ij - D_i),
    dQ_i += scale dS_ij K_j, dK_j += scale dS_ij^T Q_i. With grouped K/V
    heads each query head adds its dK_j, dV_j into its K/V head's ([note] §5.6).
    """
    q, k, v, g = _check(q, k, v)
    o = np.asarray(o, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    B, H, N, d = q.shape
    if k.shape[2] != N:
        raise ValueError("the blocked variants take N_q = N_k")
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(k)
    D = np.sum(do * o, axis=-1)
    for b in range(B):
        for h in range(H):
            hk = _kv_head(h, g)
            for j0 in range(0, N, block_cols):
                j1 = min(N, j0 + block_cols)
                kj, vj = k[b, hk, j0:j1], v[b, hk, j0:j1]
                dkj = np.zeros((j1 - j0, d))
                dvj = np.zeros((j1 - j0, d))
                for i0 in range(0, N, block_rows):
                    i1 = min(N, i0 + block_rows)
                    if causal and j0 > i1 - 1:
                        continue
                    s = scale * (q[b, h, i0:i1] @ kj.T)
                    if causal:
                        rr = np.arange(i0, i1)[:, None]
                        cc = np.arange(j0, j1)[None, :]
                        s = np.where(cc > rr, -np.inf, s)
                    p = np.exp(s - lse[b, h, i0:i1, None])
                    dvj += p.T @ do[b, h, i0:i1]
                    dp = do[b, h, i0:i1] @ vj.T
                    ds = p * (dp - D[b, h, i0:i1, None])
                    dq[b, h, i0:i1] += scale * (ds @ kj)
                    dkj += scale * (ds.T @ q[b, h, i0:i1])
                dk[b, hk, j0:j1] += dkj
                dv[b, hk, j0:j1] += dvj
    return dq, dk, dv
