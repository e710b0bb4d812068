"""Device-side failure path on the GPU, made to happen without a fault.

Every wait of the split kernel is bounded: one that runs out records
MLA_ERR_DEVICE_TIMEOUT with the wait site, flags the peer CTA, and every role of
the cluster unwinds.  The test hook mla_test_forced_timeout runs the split kernel
with its load and copy warps idle, so that no TMA load or inter-CTA copy is ever in
flight, and gives the MMA warp's first wait for K data a 1 ms limit (every other
wait keeps its 1 s limit and leaves on the abort flag).  The call must report that
wait, come back well before a 1 s limit could have run out, and leave the context
usable: the next normal call passes parity.
"""
import time

import pytest
import torch

import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu

MLA_ERR_DEVICE_TIMEOUT = -8
MLA_WAIT_K_FULL = 4


@pytest.fixture(scope="module")
def mla():
    from mla_decode_gb300 import _build
    _build.build()
    import mla_decode_gb300 as m
    m._load()
    return m


@pytest.mark.parametrize("dtype,heads", [("bf16", 128), ("fp16", 16)])
def test_forced_wait_timeout_reported_and_context_usable(mla, dtype, heads):
    w = workloads.custom(4, heads, (300, 1000, 0, 4096), dtype, seed=21, name="forced_timeout")
    inputs = workloads.make_inputs(w, "cuda")
    meta, ns = mla.mla_get_metadata(inputs["cache_seqlens"], w.heads)
    call = mla.prepare_decode(inputs["q"], inputs["kv_cache"], inputs["block_table"],
                              inputs["cache_seqlens"], w.softmax_scale, meta, ns)
    torch.cuda.synchronize()
    assert mla.mla_get_device_error() == (0, 0)

    t0 = time.perf_counter()
    assert mla.mla_test_forced_timeout(call) == 0
    code, detail = mla.mla_get_device_error()
    elapsed = time.perf_counter() - t0
    assert code == MLA_ERR_DEVICE_TIMEOUT, mla.mla_status_string(code)
    assert detail == MLA_WAIT_K_FULL
    assert elapsed < 0.5, f"the 1 ms wait took {elapsed:.3f} s to be reported"
    # the word was cleared by the read
    assert mla.mla_get_device_error() == (0, 0)

    # the context is intact: the same problem, run normally, matches the oracle
    P.check_workload(w, inputs=inputs)
    assert mla.mla_get_device_error() == (0, 0)


def test_forced_timeout_rejects_bad_arguments_before_launch(mla):
    """The hook validates like mla_decode_fwd: a bad argument never reaches the GPU."""
    import ctypes
    p = mla.FwdParams()
    assert mla._load().mla_test_forced_timeout(ctypes.byref(p), None) == -1  # MLA_ERR_NULL
