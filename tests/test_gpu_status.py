"""Failure detection without a GPU fault: a bounded device wait that nothing
satisfies gives up, records FA_ERR_TIMEOUT, and the context stays usable."""

import numpy as np
import pytest

import oracle
from gpu_util import TOL_O, inputs, to_device, to_host64, scale_f32

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
