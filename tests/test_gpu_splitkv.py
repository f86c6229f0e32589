"""GPU parity of the split-key forward (fa_fwd_splitkv): key ranges merged by
their logsumexps, and query blocks shorter than the key sequence (decoding
against a cache, causal mask aligned to the last key)."""

import numpy as np
import pytest

import oracle
from attn_inputs import BASE_SEED
from gpu_util import TOL_LSE, TOL_O, inputs, scale_f32, to_device, to_host64

pytestmark = pytest.mark.gpu


def make(B, Hq, Hkv, Nq, Nk, d, seed):
    xq, fq = inputs(B, Hq, Nq, d, seed, tensors=("q",))
    xk, fk = inputs(B, Hkv, Nk, d, seed + 1, tensors=("k", "v"))
    return {**xq, **xk}, {**fq, **fk}


def run(x, causal, scale, splits, ws_splits=None):
    import exact_softmax_attention_fa_gb300 as fa
    import torch
    q, k, v = (to_device(x[n]) for n in ("q", "k", "v"))
    B, Hq, Nq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, Nq, device="cuda")
    n = splits if ws_splits is None else ws_splits
    size = fa.fa_fwd_splitkv_workspace_size(B, Hq, Nq, d, n) if n != 1 else 0
    ws = torch.empty(size, dtype=torch.uint8, device="cuda") if size else None
    fa.fa_fwd_splitkv(q, k, v, o, lse, causal, scale, num_splits=splits, workspace=ws)
    assert fa.fa_get_device_status() == 0
    return o, lse


def check(x, f, causal, d, splits, ws_splits=None):
    scale = scale_f32(d)
    o, lse = run(x, causal, scale, splits, ws_splits)
    o_ref, lse_ref = oracle.attention_forward(f["q"], f["k"], f["v"], causal, scale)
    assert np.abs(to_host64(o) - o_ref).max() <= TOL_O
    assert np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref).max() <= TOL_LSE


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_split_ranges_square(d, causal, splits):
    x, f = make(2, 2, 2, 1000, 1000, d, BASE_SEED + 800 + splits)
    check(x, f, causal, d, splits)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(1, 1000), (4, 4097), (17, 777), (128, 4096), (300, 2049), (1, 1)])
def test_short_query_blocks(d, causal, Nq, Nk):
    x, f = make(2, 4, 4, Nq, Nk, d, BASE_SEED + 820 + Nq)
    for splits in (1, 5):
        check(x, f, causal, d, splits)


@pytest.mark.parametrize("causal", [False, True])
def test_decode_grouped_heads_auto_splits(causal):
    # 8 query heads on 2 K/V heads, one new token against 8k cached keys; the
    # library picks the split count within the workspace given
    x, f = make(2, 8, 2, 1, 8192, 128, BASE_SEED + 850)
    check(x, f, causal, 128, 0, ws_splits=64)


def test_auto_without_workspace_is_unsplit():
    x, f = make(1, 2, 2, 3, 3000, 128, BASE_SEED + 860)
    check(x, f, True, 128, 0, ws_splits=1)


def test_more_splits_than_key_tiles():
    x, f = make(1, 2, 1, 50, 300, 64, BASE_SEED + 870)  # 3 key tiles
    check(x, f, False, 64, 16)


def test_unsplit_square_is_bitwise_fa_fwd():
    import exact_softmax_attention_fa_gb300 as fa
    import torch
    x, _ = make(2, 3, 3, 555, 555, 128, BASE_SEED + 880)
    q, k, v = (to_device(x[n]) for n in ("q", "k", "v"))
    o1, l1 = fa.forward(q, k, v, causal=True, scale=0.1)
    o2 = torch.empty_like(q)
    l2 = torch.empty_like(l1)
    fa.fa_fwd_splitkv(q, k, v, o2, l2, True, 0.1, num_splits=1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_long_keys_many_splits_peaked():
    # 1% peaked query rows (large logits) with the keys cut into 16 ranges
    xq, fq = inputs(1, 2, 256, 128, BASE_SEED + 890, tensors=("q",), peaked_frac=0.01)
    xk, fk = inputs(1, 2, 16384, 128, BASE_SEED + 891, tensors=("k", "v"))
    check({**xq, **xk}, {**fq, **fk}, True, 128, 16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (8, 1), (8, 2), (6, 2), (32, 1)])
@pytest.mark.parametrize("Nq", [1, 5, 31, 32, 33, 127])
def test_grouped_short_blocks_share_tiles(causal, Hq, Hkv, Nq):
    # short query blocks pack the group's query heads into one tile (power-of-
    # two groups); unsplit and split key ranges
    Nk = 1500
    x, f = make(2, Hq, Hkv, Nq, Nk, 128, BASE_SEED + 910 + Nq + Hq)
    for splits in (1, 4):
        check(x, f, causal, 128, splits)


@pytest.mark.parametrize("d", [64, 256])
def test_grouped_decode_other_head_dims(d):
    x, f = make(2, 8, 2, 3, 2100, d, BASE_SEED + 960 + d)
    check(x, f, True, d, 0, ws_splits=32)
