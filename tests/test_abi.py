"""CPU checks of the C ABI: the library loads, exports every function fa.h
declares, and rejects bad arguments before touching the GPU."""

import ctypes

import pytest

from exact_softmax_attention_fa_gb300 import _lib
from exact_softmax_attention_fa_gb300.build import build, LIB_PATH


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


OK, INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE = 0, 1, 2, 3, 4
P = 0x10000  # a 16-byte aligned fake device address.
# Every call below has at least one invalid argument, so the library returns
# before any CUDA call and the fake address is never used, even on a GPU machine.


def test_exports_every_header_function(lib):
    names = _lib.header_functions()
    assert {"fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_status_string"} <= set(names)
    raw = ctypes.CDLL(LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert set(_lib._SIGNATURES) == set(names)


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.fa_status_string(code).decode().startswith(name)
    assert lib.fa_version() >= 100


def test_status_detail_rejects_a_null_word(lib):
    """The argument check comes before any device access (no GPU needed)."""
    assert lib.fa_get_device_status_detail(None, None) == INVALID


def fwd(lib, q=P, k=P, v=P, o=P, lse=P, B=1, H=1, N=128, d=64, causal=0, scale=0.125):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, None)


def bwd(lib, ptr=P, lse=P, ws=P, ws_bytes=1 << 30, B=1, H=1, N=128, d=64, causal=0, scale=0.125):
    return lib.fa_bwd(ptr, ptr, ptr, ptr, lse, ptr, ptr, ptr, ptr, B, H, N, d, causal, scale, ws, ws_bytes, None)


@pytest.mark.parametrize("d", [0, 32, 96, 160, 512])
def test_unsupported_head_dim(lib, d):
    assert fwd(lib, d=d) == UNSUPPORTED
    assert bwd(lib, d=d) == UNSUPPORTED
    assert lib.fa_bwd_workspace_size(1, 1, 128, d) == 0


@pytest.mark.parametrize("kw", [dict(B=-1), dict(H=-2), dict(N=-1), dict(causal=2), dict(causal=-1),
                                dict(scale=0.0), dict(scale=-0.1), dict(scale=float("nan")),
                                dict(scale=float("inf")), dict(q=0), dict(o=0), dict(lse=0)])
def test_invalid_arguments(lib, kw):
    assert fwd(lib, **kw) == INVALID


def test_empty_problem_is_a_no_op(lib):
    for kw in (dict(N=0), dict(B=0), dict(H=0)):
        assert fwd(lib, q=0, k=0, v=0, o=0, lse=0, **kw) == OK
        assert bwd(lib, ptr=0, lse=0, ws=0, ws_bytes=0, **kw) == OK
        assert lib.fa_bwd_workspace_size(kw.get("B", 1), kw.get("H", 1), kw.get("N", 128), 64) == 0


def fwd_gqa(lib, ptr=P, lse=P, B=1, Hq=4, Hkv=2, N=128, d=64, causal=0, scale=0.125):
    return lib.fa_fwd_gqa(ptr, ptr, ptr, ptr, lse, B, Hq, Hkv, N, d, causal, scale, None)


def bwd_gqa(lib, ptr=P, lse=P, ws=P, ws_bytes=1 << 30, B=1, Hq=4, Hkv=2, N=128, d=64, causal=0, scale=0.125):
    return lib.fa_bwd_gqa(ptr, ptr, ptr, ptr, lse, ptr, ptr, ptr, ptr, B, Hq, Hkv, N, d, causal, scale, ws, ws_bytes,
                          None)


@pytest.mark.parametrize("Hq,Hkv", [(4, 0), (4, -1), (4, 3), (2, 4), (4, 8)])
def test_grouped_heads_must_divide(lib, Hq, Hkv):
    assert fwd_gqa(lib, Hq=Hq, Hkv=Hkv) == INVALID
    assert bwd_gqa(lib, Hq=Hq, Hkv=Hkv) == INVALID


def test_grouped_workspace_size(lib):
    for B, Hq, Hkv, N, d in ((2, 8, 2, 1000, 64), (1, 16, 1, 300, 128), (1, 4, 4, 100, 128), (1, 4, 2, 100, 256)):
        base = lib.fa_bwd_workspace_size(B, Hq, N, d)
        g = Hq // Hkv
        extra = 0 if (g == 1 or d == 256) else g * B * Hkv * N * d * 8  # fp32 dK + dV partial per chunk
        assert lib.fa_bwd_gqa_workspace_size(B, Hq, Hkv, N, d) == base + extra
    assert lib.fa_bwd_gqa_workspace_size(1, 4, 3, 128, 64) == 0
    assert lib.fa_bwd_gqa_workspace_size(1, 4, 0, 128, 64) == 0


def test_deterministic_backward_checks(lib):
    def det(d=64, Hq=4, Hkv=2, ws=P, ws_bytes=1 << 30, ptr=P):
        return lib.fa_bwd_gqa_deterministic(ptr, ptr, ptr, ptr, P, ptr, ptr, ptr, ptr, 1, Hq, Hkv, 128, d, 0, 0.125,
                                            ws, ws_bytes, None)
    assert det(d=256, ws=0) == WORKSPACE  # d = 256 is supported; the missing workspace is caught
    assert det(d=96) == UNSUPPORTED
    assert det(Hkv=3) == INVALID
    assert det(ptr=0) == INVALID
    assert det(ws=0) == WORKSPACE
    assert lib.fa_bwd_deterministic(P, P, P, P, P, P, P, P, P, 1, 1, 128, 256, 0, 0.125, 0, 0, None) == WORKSPACE
    assert lib.fa_bwd_deterministic(P, P, P, P, P, P, P, P, P, 1, 1, 128, 96, 0, 0.125, P, 1 << 30, None) == UNSUPPORTED


def test_split_key_forward_checks(lib):
    def fwd_split(Nq=64, Nk=256, causal=0, splits=1, ws=P, ws_bytes=1 << 30, Hq=2, Hkv=2, d=64, ptr=P):
        return lib.fa_fwd_splitkv(ptr, ptr, ptr, ptr, P, 1, Hq, Hkv, Nq, Nk, d, causal, 0.125, splits, ws, ws_bytes,
                                  None)
    assert fwd_split(Nq=300, Nk=200, causal=1) == INVALID  # a causal block longer than the keys
    assert fwd_split(Nk=0) == INVALID
    assert fwd_split(Nk=-1) == INVALID
    assert fwd_split(splits=-1) == INVALID
    assert fwd_split(splits=257) == INVALID
    assert fwd_split(Hkv=3) == INVALID
    assert fwd_split(d=96) == UNSUPPORTED
    assert fwd_split(splits=2, ws=0) == WORKSPACE
    assert fwd_split(splits=2, ws_bytes=16) == WORKSPACE
    assert fwd_split(splits=2, ws=P + 16) == MISALIGNED
    assert fwd_split(ptr=P + 8) == MISALIGNED
    assert fwd_split(Nq=0, ptr=0) == OK
    need = lib.fa_fwd_splitkv_workspace_size(1, 2, 64, 64, 3)
    assert need == 3 * 2 * 64 * 64 * 4 + ((3 * 2 * 64 * 4 + 255) // 256) * 256
    assert lib.fa_fwd_splitkv_workspace_size(1, 2, 64, 64, 1) == 0
    assert lib.fa_fwd_splitkv_workspace_size(1, 2, 64, 64, 300) == 0


def test_deterministic_phase_checks(lib):
    assert lib.fa_bwd_dkdv(P, P, P, P, P, P, 1, 1, 128, 96, 0, 0.125, P, 1 << 30, None) == UNSUPPORTED
    assert lib.fa_bwd_dq(P, P, P, P, P, 1, 1, 128, 96, 0, 0.125, P, 1 << 30, None) == UNSUPPORTED
    assert lib.fa_bwd_dkdv(P, P, P, P, 0, P, 1, 1, 128, 256, 0, 0.125, P, 1 << 30, None) == INVALID
    assert lib.fa_bwd_dq(P, P, P, P, P, 1, 1, 128, 256, 0, 0.125, 0, 0, None) == WORKSPACE
    assert lib.fa_bwd_dkdv(P, P, P, P, 0, P, 1, 1, 128, 64, 0, 0.125, P, 1 << 30, None) == INVALID
    assert lib.fa_bwd_dq(P, P, P, P, P, 1, 1, 128, 64, 0, 0.125, 0, 0, None) == WORKSPACE
    assert lib.fa_bwd_dq(P, P, P, P, P, 1, 1, 128, 64, 2, 0.125, P, 1 << 30, None) == INVALID
    assert lib.fa_bwd_dkdv(0, 0, 0, 0, 0, 0, 1, 1, 0, 64, 0, 0.125, 0, 0, None) == OK


def test_grouped_heads_other_checks(lib):
    assert fwd_gqa(lib, d=96) == UNSUPPORTED
    assert bwd_gqa(lib, scale=0.0) == INVALID
    assert fwd_gqa(lib, ptr=0) == INVALID
    assert bwd_gqa(lib, ws=0) == WORKSPACE
    assert fwd_gqa(lib, ptr=P + 8) == MISALIGNED
    # empty problems do nothing, null pointers allowed
    assert fwd_gqa(lib, ptr=0, lse=0, Hq=0, Hkv=0) == OK
    assert bwd_gqa(lib, ptr=0, lse=0, ws=0, ws_bytes=0, N=0) == OK


@pytest.mark.parametrize("which", ["q", "k", "v", "o"])
def test_misaligned_bf16(lib, which):
    assert fwd(lib, **{which: P + 8}) == MISALIGNED


def test_misaligned_lse(lib):
    assert fwd(lib, lse=P + 2) == MISALIGNED


def test_backward_workspace_checks(lib):
    need = lib.fa_bwd_workspace_size(1, 1, 128, 64)
    assert need > 0
    assert bwd(lib, ws=0) == WORKSPACE
    assert bwd(lib, ws_bytes=need - 1) == WORKSPACE
    assert bwd(lib, ws=P + 16, ws_bytes=need) == MISALIGNED
    assert bwd(lib, ptr=P + 8) == MISALIGNED


def test_workspace_size_formula(lib):
    # D and base-2 L (fp32 per padded row) + fp32 dQ accumulator, heads padded
    # to 128 rows, + 256 bytes of work-item counter
    for B, H, N, d in ((2, 4, 1024, 64), (1, 16, 1000, 128), (1, 2, 1, 256)):
        rows = B * H * ((N + 127) // 128 * 128)
        expect = 0
        for nbytes in (rows * 4, rows * 4, rows * d * 4, 256):
            expect = (expect + 255) // 256 * 256 + nbytes
        assert lib.fa_bwd_workspace_size(B, H, N, d) == expect


def test_python_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    import exact_softmax_attention_fa_gb300 as fa
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, q.clone(), torch.zeros(1, 1, 128), False, 0.125)
    with pytest.raises(TypeError):
        fa.fa_fwd(q.float(), q, q, q, torch.zeros(1, 1, 128), False, 0.125)


def test_noalloc_backward_validation(lib):
    """Argument errors and oversized problems are rejected before any CUDA call."""
    def call(B=1, H=1, N=128, d=64, causal=0, scale=0.125, ptr=P, lse=P):
        return lib.fa_bwd_noalloc(ptr, ptr, ptr, ptr, lse, ptr, ptr, ptr, ptr, B, H, N, d, causal, scale, None)
    assert call(d=96) == UNSUPPORTED
    assert call(scale=-1.0) == INVALID
    assert call(N=0, ptr=0, lse=0) == OK
    # 16 heads x 8192 rows at d=128 need ~68 MB of scratch, beyond the compiled 16 MiB
    assert lib.fa_bwd_workspace_size(1, 16, 8192, 128) > (16 << 20)
    assert call(B=1, H=16, N=8192, d=128) == WORKSPACE


def test_host_entry_checks(lib):
    """fa_fwd_bwd_host: size formula and argument errors (all before any CUDA call)."""
    def call(ptr=P, lse=P, buf=P, nbytes=1 << 34, B=1, H=2, N=128, d=64, causal=0, scale=0.125):
        return lib.fa_fwd_bwd_host(ptr, ptr, ptr, ptr, ptr, lse, ptr, ptr, ptr, B, H, N, d, causal, scale, buf,
                                   nbytes, None)
    a = lambda n: (n + 255) // 256 * 256

    def groups(BH):
        """Head counts of the plan the header states: an eighth of the heads,
        the rest (less another eighth) in two halves, then that eighth."""
        g0 = (BH + 7) // 8
        last = (BH + 7) // 8 if BH - g0 >= 2 else BH - g0
        mid = BH - g0 - last
        return [h for h in (g0, mid // 2, mid - mid // 2, last) if h > 0]

    assert groups(32) == [4, 12, 12, 4] and groups(3) == [1, 1, 1] and groups(2) == [1, 1] and groups(1) == [1]
    shapes = [(1, 2, 128, 64), (2, 3, 1000, 128), (1, 1, 1, 256), (2, 16, 8192, 128), (1, 5, 300, 64)]
    shapes += [(1, bh, 640, 128) for bh in range(1, 41)]  # every group split up to 40 heads
    for B, H, N, d in shapes:
        rows = B * H * N
        need = 8 * a(rows * d * 2) + a(rows * 4)
        need += sum(a(lib.fa_bwd_workspace_size(1, h, N, d)) for h in groups(B * H))
        assert lib.fa_fwd_bwd_host_device_bytes(B, H, N, d) == need
    need = lib.fa_fwd_bwd_host_device_bytes(1, 2, 128, 64)
    assert lib.fa_fwd_bwd_host_device_bytes(1, 2, 0, 64) == 0
    assert lib.fa_fwd_bwd_host_device_bytes(1, 2, 128, 96) == 0
    assert call(d=96) == UNSUPPORTED
    assert call(scale=0.0) == INVALID
    assert call(causal=3) == INVALID
    assert call(ptr=0) == INVALID
    assert call(lse=0) == INVALID
    assert call(buf=0) == WORKSPACE
    assert call(nbytes=need - 1) == WORKSPACE
    assert call(buf=P + 16, nbytes=need) == MISALIGNED
    assert call(N=0, ptr=0, lse=0, buf=0, nbytes=0) == OK


def test_forward_host_entry_checks(lib):
    """fa_fwd_host: size formula and argument errors (all before any CUDA call)."""
    def call(ptr=P, lse=P, buf=P, nbytes=1 << 34, B=1, H=2, N=128, d=64, causal=0, scale=0.125):
        return lib.fa_fwd_host(ptr, ptr, ptr, ptr, lse, B, H, N, d, causal, scale, buf, nbytes, None)
    a = lambda n: (n + 255) // 256 * 256
    for B, H, N, d in ((1, 2, 128, 64), (2, 3, 1000, 128), (1, 1, 1, 256)):
        rows = B * H * N
        assert lib.fa_fwd_host_device_bytes(B, H, N, d) == 4 * a(rows * d * 2) + a(rows * 4)
    need = lib.fa_fwd_host_device_bytes(1, 2, 128, 64)
    assert lib.fa_fwd_host_device_bytes(0, 2, 128, 64) == 0
    assert call(d=32) == UNSUPPORTED
    assert call(scale=float("nan")) == INVALID
    assert call(ptr=0) == INVALID
    assert call(lse=0) == INVALID
    assert call(buf=0) == WORKSPACE
    assert call(nbytes=need - 1) == WORKSPACE
    assert call(buf=P + 64, nbytes=need) == MISALIGNED
    assert call(H=0, ptr=0, lse=0, buf=0, nbytes=0) == OK


def test_preprocess_stats_checks(lib):
    """The stats-only preprocess validates like the full one (no GPU needed)."""
    assert lib.fa_bwd_preprocess_stats(P, P, P, 1, 1, 128, 96, P, 1 << 30, None) == UNSUPPORTED
    assert lib.fa_bwd_preprocess_stats(0, P, P, 1, 1, 128, 64, P, 1 << 30, None) == INVALID
    assert lib.fa_bwd_preprocess_stats(P, P, P, 1, 1, 128, 64, 0, 0, None) == WORKSPACE
    assert lib.fa_bwd_preprocess_stats(P + 8, P, P, 1, 1, 128, 64, P, 1 << 30, None) == MISALIGNED
    assert lib.fa_bwd_preprocess_stats(0, 0, 0, 1, 1, 0, 64, 0, 0, None) == OK


def test_debug_skip_hook_checks(lib):
    """Only the role codes of the status word are accepted; 0 turns the hook off."""
    for bad in (4, 10, 15, 99, 1 << 31):
        assert lib.fa_debug_skip_arrival(bad) == INVALID
    for good in (1, 2, 3, 11, 12, 13, 14):
        assert lib.fa_debug_skip_arrival(good) == OK
    assert lib.fa_debug_skip_arrival(0) == OK
