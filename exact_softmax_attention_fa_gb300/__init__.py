"""GB300 (sm_103a) exact softmax attention: Python binding of the C ABI.

The functions here only check and marshal arguments (torch tensors -> device
pointers, sizes, the current CUDA stream) and call libfa_gb300.so; every step
of the computation runs in the library's CUDA kernels. PyTorch supplies device
memory and streams.

    o, lse = forward(q, k, v, causal=True)            # q, k, v: bf16 [B, H, N, d] on CUDA
    dq, dk, dv = backward(q, k, v, o, lse, do, causal=True)
"""

from __future__ import annotations

import math

from ._lib import load, check, FAError, header_functions, STATUS_NAMES  # noqa: F401

__all__ = ["fa_fwd", "fa_bwd", "fa_fwd_gqa", "fa_bwd_gqa", "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_size", "fa_bwd_deterministic", "fa_bwd_gqa_deterministic", "fa_bwd_workspace_size", "fa_bwd_gqa_workspace_size", "fa_bwd_preprocess", "fa_bwd_preprocess_stats", "fa_bwd_main", "fa_bwd_postprocess", "fa_bwd_dkdv", "fa_bwd_dq", "fa_bwd_noalloc", "fa_fwd_bwd_host", "fa_fwd_bwd_host_device_bytes", "fa_fwd_host", "fa_fwd_host_device_bytes", "fa_get_device_status", "fa_get_device_status_detail", "fa_set_wait_limit_ns",
           "fa_debug_timeout_probe", "fa_debug_skip_arrival", "forward", "backward", "FAError", "flops"]

_SUPPORTED_D = (64, 128, 256)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dims(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    return tuple(int(x) for x in q.shape)


def _check_bf16(name, t, shape):
    import torch
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if tuple(t.shape) != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _check_lse(t, shape):
    import torch
    if t.dtype != torch.float32 or tuple(t.shape) != shape[:3] or not t.is_cuda or not t.is_contiguous():
        raise ValueError("lse must be a contiguous float32 CUDA tensor of shape [B, H, N]")


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def fa_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """fa_fwd of the C ABI on torch tensors (outputs o, lse written in place)."""
    shape = _dims(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _check_bf16(name, t, shape)
    _check_lse(lse, shape)
    B, H, N, d = shape
    lib = load()
    check("fa_fwd", lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               B, H, N, d, int(bool(causal)), float(scale), _stream_handle(stream)))


def _gqa_dims(q, k):
    """(B, Hq, Hkv, N, d) for q [B, Hq, N, d] and k [B, Hkv, N, d]."""
    B, Hq, N, d = _dims(q)
    if k.dim() != 4 or k.shape[0] != B or tuple(k.shape[2:]) != (N, d):
        raise ValueError("k must be [B, Hkv, N, d] with q's B, N, d")
    Hkv = int(k.shape[1])
    if Hkv < 1 or Hq % Hkv != 0:
        raise ValueError(f"the query heads ({Hq}) must be a multiple of the K/V heads ({Hkv})")
    return B, Hq, Hkv, N, d


def fa_fwd_gqa(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """fa_fwd_gqa of the C ABI: q, o [B, Hq, N, d]; k, v [B, Hkv, N, d]; lse [B, Hq, N]."""
    B, Hq, Hkv, N, d = _gqa_dims(q, k)
    for name, t, shape in (("q", q, (B, Hq, N, d)), ("k", k, (B, Hkv, N, d)), ("v", v, (B, Hkv, N, d)),
                           ("o", o, (B, Hq, N, d))):
        _check_bf16(name, t, shape)
    _check_lse(lse, (B, Hq, N, d))
    lib = load()
    check("fa_fwd_gqa", lib.fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                       B, Hq, Hkv, N, d, int(bool(causal)), float(scale), _stream_handle(stream)))


def fa_bwd_gqa(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float, workspace, stream=None) -> None:
    """fa_bwd_gqa of the C ABI: q, o, do, dq [B, Hq, N, d]; k, v, dk, dv [B, Hkv, N, d].

    `workspace` is a CUDA uint8 tensor of at least fa_bwd_workspace_size(B, Hq, N, d) bytes.
    """
    B, Hq, Hkv, N, d = _gqa_dims(q, k)
    qs, ks = (B, Hq, N, d), (B, Hkv, N, d)
    for name, t, shape in (("q", q, qs), ("k", k, ks), ("v", v, ks), ("o", o, qs), ("do", do, qs), ("dq", dq, qs),
                           ("dk", dk, ks), ("dv", dv, ks)):
        _check_bf16(name, t, shape)
    _check_lse(lse, qs)
    lib = load()
    check("fa_bwd_gqa", lib.fa_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                       do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                       B, Hq, Hkv, N, d, int(bool(causal)), float(scale), *_ws(workspace),
                                       _stream_handle(stream)))


def fa_fwd_splitkv_workspace_size(B: int, Hq: int, Nq: int, d: int, num_splits: int) -> int:
    return int(load().fa_fwd_splitkv_workspace_size(B, Hq, Nq, d, num_splits))


def fa_fwd_splitkv(q, k, v, o, lse, causal: bool, scale: float, num_splits: int = 0, workspace=None,
                   stream=None) -> None:
    """fa_fwd_splitkv of the C ABI: q, o [B, Hq, Nq, d]; k, v [B, Hkv, Nk, d]; lse [B, Hq, Nq].

    Causal masks align to the last key (query i sees keys j <= i + Nk - Nq).
    num_splits = 0 lets the library choose within `workspace` (a CUDA uint8
    tensor, or None for no split).
    """
    B, Hq, Nq, d = _dims(q)
    if k.dim() != 4 or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k must be [B, Hkv, Nk, d] with q's B and d")
    Hkv, Nk = int(k.shape[1]), int(k.shape[2])
    for name, t, shape in (("q", q, (B, Hq, Nq, d)), ("k", k, (B, Hkv, Nk, d)), ("v", v, (B, Hkv, Nk, d)),
                           ("o", o, (B, Hq, Nq, d))):
        _check_bf16(name, t, shape)
    _check_lse(lse, (B, Hq, Nq, d))
    check("fa_fwd_splitkv", load().fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                  lse.data_ptr(), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)),
                                                  float(scale), int(num_splits), *_ws(workspace),
                                                  _stream_handle(stream)))


def fa_bwd_deterministic(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float, workspace, stream=None) -> None:
    """fa_bwd_deterministic of the C ABI: fa_bwd with a bitwise-reproducible dq (d = 64, 128)."""
    shape = _dims(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_bf16(name, t, shape)
    _check_lse(lse, shape)
    B, H, N, d = shape
    check("fa_bwd_deterministic",
          load().fa_bwd_deterministic(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                      do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                                      int(bool(causal)), float(scale), *_ws(workspace), _stream_handle(stream)))


def fa_bwd_gqa_deterministic(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float, workspace,
                             stream=None) -> None:
    """fa_bwd_gqa_deterministic of the C ABI: fa_bwd_gqa with a bitwise-reproducible dq (d = 64, 128)."""
    B, Hq, Hkv, N, d = _gqa_dims(q, k)
    qs, ks = (B, Hq, N, d), (B, Hkv, N, d)
    for name, t, shape in (("q", q, qs), ("k", k, ks), ("v", v, ks), ("o", o, qs), ("do", do, qs), ("dq", dq, qs),
                           ("dk", dk, ks), ("dv", dv, ks)):
        _check_bf16(name, t, shape)
    _check_lse(lse, qs)
    check("fa_bwd_gqa_deterministic",
          load().fa_bwd_gqa_deterministic(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                          do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv,
                                          N, d, int(bool(causal)), float(scale), *_ws(workspace),
                                          _stream_handle(stream)))


def fa_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd_gqa_workspace_size(B: int, Hq: int, Hkv: int, N: int, d: int) -> int:
    return int(load().fa_bwd_gqa_workspace_size(B, Hq, Hkv, N, d))


def fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float, workspace, stream=None) -> None:
    """fa_bwd of the C ABI on torch tensors (dq, dk, dv written in place).

    `workspace` is a CUDA uint8 tensor of at least fa_bwd_workspace_size() bytes.
    """
    shape = _dims(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_bf16(name, t, shape)
    _check_lse(lse, shape)
    B, H, N, d = shape
    lib = load()
    check("fa_bwd", lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                               B, H, N, d, int(bool(causal)), float(scale), *_ws(workspace),
                               _stream_handle(stream)))


def _ws(workspace):
    if workspace is None:
        return 0, 0
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def fa_bwd_preprocess(o, lse, do, workspace, stream=None) -> None:
    """First phase of fa_bwd: D, base-2 L and a zeroed dQ accumulator in `workspace`."""
    shape = _dims(o)
    _check_bf16("o", o, shape)
    _check_bf16("do", do, shape)
    _check_lse(lse, shape)
    B, H, N, d = shape
    check("fa_bwd_preprocess", load().fa_bwd_preprocess(o.data_ptr(), lse.data_ptr(), do.data_ptr(), B, H, N, d,
                                                        *_ws(workspace), _stream_handle(stream)))


def fa_bwd_preprocess_stats(o, lse, do, workspace, stream=None) -> None:
    """First phase of fa_bwd_deterministic: D and base-2 L in `workspace` (no accumulator zeroing)."""
    shape = _dims(o)
    _check_bf16("o", o, shape)
    _check_bf16("do", do, shape)
    _check_lse(lse, shape)
    B, H, N, d = shape
    check("fa_bwd_preprocess_stats", load().fa_bwd_preprocess_stats(o.data_ptr(), lse.data_ptr(), do.data_ptr(), B,
                                                                    H, N, d, *_ws(workspace), _stream_handle(stream)))


def fa_bwd_main(q, k, v, do, dk, dv, causal: bool, scale: float, workspace, stream=None) -> None:
    """Second phase of fa_bwd: dk, dv, and dQ accumulated into `workspace`."""
    shape = _dims(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("do", do), ("dk", dk), ("dv", dv)):
        _check_bf16(name, t, shape)
    B, H, N, d = shape
    check("fa_bwd_main", load().fa_bwd_main(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), dk.data_ptr(),
                                            dv.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                            *_ws(workspace), _stream_handle(stream)))


def fa_bwd_dkdv(q, k, v, do, dk, dv, causal: bool, scale: float, workspace, stream=None) -> None:
    """Deterministic backward phase: dk, dv only (after fa_bwd_preprocess)."""
    shape = _dims(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("do", do), ("dk", dk), ("dv", dv)):
        _check_bf16(name, t, shape)
    B, H, N, d = shape
    check("fa_bwd_dkdv", load().fa_bwd_dkdv(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), dk.data_ptr(),
                                            dv.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                            *_ws(workspace), _stream_handle(stream)))


def fa_bwd_dq(q, k, v, do, dq, causal: bool, scale: float, workspace, stream=None) -> None:
    """Deterministic backward phase: dq summed per query tile on chip (after fa_bwd_preprocess)."""
    shape = _dims(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("do", do), ("dq", dq)):
        _check_bf16(name, t, shape)
    B, H, N, d = shape
    check("fa_bwd_dq", load().fa_bwd_dq(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), dq.data_ptr(),
                                        B, H, N, d, int(bool(causal)), float(scale), *_ws(workspace),
                                        _stream_handle(stream)))


def fa_bwd_postprocess(dq, workspace, stream=None) -> None:
    """Last phase of fa_bwd: dq = bf16(dQ accumulator)."""
    shape = _dims(dq)
    _check_bf16("dq", dq, shape)
    B, H, N, d = shape
    check("fa_bwd_postprocess", load().fa_bwd_postprocess(dq.data_ptr(), B, H, N, d, *_ws(workspace),
                                                          _stream_handle(stream)))


# Scratch size compiled into the library for fa_bwd_noalloc (include/fa.h).
FA_BWD_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, causal: bool, scale: float, stream=None) -> None:
    """fa_bwd without a caller workspace: the library's fixed scratch array is used.

    For callers that are given only input and output buffers and cannot
    allocate device memory. Sizes whose workspace exceeds
    FA_BWD_NOALLOC_SCRATCH_BYTES raise FAError(FA_ERR_WORKSPACE). Calls that
    overlap on the GPU share the array and race.
    """
    shape = _dims(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_bf16(name, t, shape)
    _check_lse(lse, shape)
    B, H, N, d = shape
    check("fa_bwd_noalloc", load().fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                  lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                                  dv.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                                  _stream_handle(stream)))


def fa_fwd_bwd_host_device_bytes(B: int, H: int, N: int, d: int) -> int:
    """Device buffer size fa_fwd_bwd_host needs (0 for invalid or empty problems)."""
    return int(load().fa_fwd_bwd_host_device_bytes(B, H, N, d))


def _check_host(name, t, shape, dtype):
    if t.dtype != dtype or tuple(t.shape) != shape or t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} CPU tensor of shape {shape}")


def fa_fwd_bwd_host(q, k, v, do, o, lse, dq, dk, dv, causal: bool, scale: float, device_buffer,
                    stream=None) -> None:
    """fa_fwd_bwd_host of the C ABI: forward and backward of CPU tensors.

    q, k, v, do (in) and o, dq, dk, dv (out) are contiguous bf16 CPU tensors
    [B, H, N, d], lse a float32 CPU tensor [B, H, N]; page-locked tensors
    (pin_memory) let the library overlap the copies with the kernels.
    device_buffer is a CUDA uint8 tensor of at least
    fa_fwd_bwd_host_device_bytes(B, H, N, d) bytes. Asynchronous on `stream`:
    the outputs are valid once the stream has synchronised.
    """
    import torch
    shape = _dims(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("do", do), ("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_host(name, t, shape, torch.bfloat16)
    _check_host("lse", lse, shape[:3], torch.float32)
    if not device_buffer.is_cuda or device_buffer.dtype != torch.uint8:
        raise ValueError("device_buffer must be a CUDA uint8 tensor")
    B, H, N, d = shape
    check("fa_fwd_bwd_host", load().fa_fwd_bwd_host(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), o.data_ptr(), lse.data_ptr(), dq.data_ptr(),
        dk.data_ptr(), dv.data_ptr(), B, H, N, d, int(bool(causal)), float(scale), device_buffer.data_ptr(),
        device_buffer.numel(), _stream_handle(stream)))


def fa_fwd_host_device_bytes(B: int, H: int, N: int, d: int) -> int:
    """Device buffer size fa_fwd_host needs (0 for invalid or empty problems)."""
    return int(load().fa_fwd_host_device_bytes(B, H, N, d))


def fa_fwd_host(q, k, v, o, lse, causal: bool, scale: float, device_buffer, stream=None) -> None:
    """fa_fwd_host of the C ABI: the forward of CPU tensors, pipelined over head chunks.

    q, k, v (in) and o (out) are contiguous bf16 CPU tensors [B, H, N, d], lse
    a float32 CPU tensor [B, H, N]; device_buffer a CUDA uint8 tensor of at
    least fa_fwd_host_device_bytes(B, H, N, d) bytes. Asynchronous on `stream`.
    """
    import torch
    shape = _dims(q)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _check_host(name, t, shape, torch.bfloat16)
    _check_host("lse", lse, shape[:3], torch.float32)
    if not device_buffer.is_cuda or device_buffer.dtype != torch.uint8:
        raise ValueError("device_buffer must be a CUDA uint8 tensor")
    B, H, N, d = shape
    check("fa_fwd_host", load().fa_fwd_host(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, int(bool(causal)),
        float(scale), device_buffer.data_ptr(), device_buffer.numel(), _stream_handle(stream)))


def fa_get_device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status (0 = FA_OK)."""
    return int(load().fa_get_device_status(_stream_handle(stream)))


def fa_get_device_status_detail(stream=None) -> tuple:
    """Synchronise the stream; return and clear the whole device status word:
    (code, role of the first wait that gave up, its block, its thread)."""
    import ctypes
    word = (ctypes.c_uint * 4)()
    st = int(load().fa_get_device_status_detail(ctypes.addressof(word), _stream_handle(stream)))
    if st == 7:  # FA_ERR_CUDA: the synchronisation failed, the word was not read
        check("fa_get_device_status_detail", st)
    return tuple(int(x) for x in word)


def fa_set_wait_limit_ns(limit_ns: int) -> None:
    load().fa_set_wait_limit_ns(int(limit_ns))


def fa_debug_timeout_probe(limit_ns: int, stream=None) -> None:
    check("fa_debug_timeout_probe", load().fa_debug_timeout_probe(int(limit_ns), _stream_handle(stream)))


def fa_debug_skip_arrival(role: int) -> None:
    """Test hook: block 0 of later launches leaves out the first arrival of
    `role` (a role code of fa_get_device_status_detail), so a bounded wait
    gives up; 0 turns it off."""
    check("fa_debug_skip_arrival", load().fa_debug_skip_arrival(int(role)))


def forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Allocate O (bf16) and L (fp32) with torch and run fa_fwd (fa_fwd_gqa when
    k, v have fewer heads than q)."""
    import torch
    B, H, N, d = _dims(q)
    if scale is None:
        scale = default_scale(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if k.dim() == 4 and k.shape[1] != H:
        fa_fwd_gqa(q, k, v, o, lse, causal, scale, stream)
    else:
        fa_fwd(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, workspace=None, stream=None,
             deterministic: bool = False):
    """Allocate dQ, dK, dV (and the workspace if not given) with torch and run fa_bwd
    (fa_bwd_gqa when k, v have fewer heads than q; the *_deterministic entry
    points when `deterministic`)."""
    import torch
    B, H, N, d = _dims(q)
    if scale is None:
        scale = default_scale(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    grouped = k.dim() == 4 and k.shape[1] != H
    if workspace is None:
        size = fa_bwd_gqa_workspace_size(B, H, int(k.shape[1]), N, d) if grouped else fa_bwd_workspace_size(B, H, N, d)
        workspace = torch.empty(max(1, size), dtype=torch.uint8, device=q.device)
    if grouped:
        fn = fa_bwd_gqa_deterministic if deterministic else fa_bwd_gqa
    else:
        fn = fa_bwd_deterministic if deterministic else fa_bwd
    fn(q, k, v, o, lse, do, dq, dk, dv, causal, scale, workspace, stream)
    return dq, dk, dv


def flops(B: int, H: int, N: int, d: int, causal: bool, mode: str = "fwd") -> float:
    """Algorithmic FLOPs of the pages' benchmark convention.

    forward = 4 * N^2 * d * H (* B), halved under a causal mask; backward = 2.5x
    forward (five matmuls instead of two); fwd+bwd = 3.5x forward. (Reading note
    on papers.chlience.com, "结果 1"; paper-graph-ui summary, "Evaluation
    Methodology".)
    """
    f = 4.0 * B * H * N * N * d
    if causal:
        f *= 0.5
    mult = {"fwd": 1.0, "bwd": 2.5, "fwd_bwd": 3.5}[mode]
    return f * mult
