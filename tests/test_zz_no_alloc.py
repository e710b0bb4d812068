"""mla_decode_fwd_static, the allocation-free entry point, against mla_decode_fwd.

Callers that cannot allocate device memory (a C host with no allocator of its
own, a runtime that reserved all memory up front) use this entry: its partials
go to one fixed scratch array per device that is reused and never cleared.  So
on consecutive calls it must give what the workspace entry point gives (the same
kernels run, so the same bits, and in any case within the parity tolerance),
whatever the previous call left in the array; and it must reject problems whose
partials do not fit, before touching the device.  The file name puts it last in
collection; it also passes when run alone in a fresh process.
"""
import ctypes
import os
import re

import pytest
import torch

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MLA_ERR_NULL = -1
MLA_ERR_SHAPE = -2
MLA_ERR_WORKSPACE = -6
OUT_MAX = 2e-2    # same bars as the parity tests (absolute)
LSE_MAX = 1e-3


@pytest.fixture(scope="module")
def mla():
    from mla_decode_gb300 import _build
    _build.build()
    import mla_decode_gb300 as m
    m._load()
    return m


def test_static_size_matches_header(mla):
    text = open(os.path.join(ROOT, "include", "mla_decode.h")).read()
    m = re.search(r"#define MLA_STATIC_WORKSPACE_BYTES \((\d+)u << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == mla.STATIC_WORKSPACE_BYTES


def test_rejects_oversized_problem_before_touching_device(mla):
    lib = mla._load()
    parts, h = 76, 128
    # 255 splits of 128 heads fit in 64 MiB, 256 do not
    assert mla.mla_workspace_size(255 - parts, h, parts) <= mla.STATIC_WORKSPACE_BYTES
    assert mla.mla_workspace_size(256 - parts, h, parts) > mla.STATIC_WORKSPACE_BYTES
    p = mla.FwdParams()
    p.b, p.seqlen_q, p.h, p.h_k, p.num_sm_parts = 256 - parts, 1, h, 1, parts
    assert lib.mla_decode_fwd_static(ctypes.byref(p), None) == MLA_ERR_WORKSPACE
    p.b = 0
    assert lib.mla_decode_fwd_static(ctypes.byref(p), None) == MLA_ERR_SHAPE
    assert lib.mla_decode_fwd_static(None, None) == MLA_ERR_NULL


def test_rejects_by_query_rows(mla):
    """With several query tokens the scratch holds seqlen_q * h rows per split: at two
    tokens of 128 heads, 127 splits fit in 64 MiB and 128 do not; more than 1024
    rows per sequence is a shape error."""
    lib = mla._load()
    rows = 2 * 128
    parts, _ = mla.mla_metadata_shape(1, rows, 152)
    assert mla.mla_workspace_size(127 - parts, rows, parts) <= mla.STATIC_WORKSPACE_BYTES
    assert mla.mla_workspace_size(128 - parts, rows, parts) > mla.STATIC_WORKSPACE_BYTES
    p = mla.FwdParams()
    p.b, p.seqlen_q, p.h, p.h_k, p.num_sm_parts = 128 - parts, 2, 128, 1, parts
    assert lib.mla_decode_fwd_static(ctypes.byref(p), None) == MLA_ERR_WORKSPACE
    p.b, p.seqlen_q = 1, 9  # 9 x 128 = 1152 rows
    assert lib.mla_decode_fwd_static(ctypes.byref(p), None) == MLA_ERR_SHAPE


def _compare_two_calls(mla, w, num_sm=None):
    inp = workloads.make_inputs(w, device="cuda")
    meta, num_splits = mla.mla_get_metadata(inp["cache_seqlens"], w.heads, num_sm)
    args = (inp["q"], inp["kv_cache"], inp["block_table"], inp["cache_seqlens"],
            w.softmax_scale, meta, num_splits)
    ref_out, ref_lse = mla.mla_decode_fwd(*args)
    code, detail = mla.mla_get_device_error()
    assert code == 0, f"reference call: device error {code}, detail {detail}"
    out = torch.empty_like(ref_out)
    lse = torch.empty_like(ref_lse)
    for call in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        mla.mla_decode_fwd_static(*args, out=out, lse=lse)
        code, detail = mla.mla_get_device_error()
        assert code == 0, f"call {call}: device error {code}, detail {detail}"
        ro, o = ref_out.float(), out.float()
        err = (o - ro).abs().max().item()
        assert err <= OUT_MAX, f"call {call}: out error {err}"
        fin = torch.isfinite(ref_lse)
        assert torch.equal(fin, torch.isfinite(lse)), f"call {call}: lse finiteness"
        if fin.any():
            assert (lse[fin] - ref_lse[fin]).abs().max().item() <= LSE_MAX, f"call {call}: lse"
        # the same kernels on the same inputs: the same bits
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"call {call}: out bits"
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), f"call {call}: lse bits"
    return meta.shape[0]


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["paged", "mqa", "tiny"])
def test_static_matches_workspace_entry(mla, name):
    _compare_two_calls(mla, workloads.get(name))


@pytest.mark.gpu
def test_static_many_splits_small_grid(mla):
    # few parts: long sequences split many ways, short and empty ones stay whole
    w = workloads.custom(batch=5, heads=128, seqlens=(4097, 1, 0, 2000, 640), seed=7)
    _compare_two_calls(mla, w, num_sm=6)


@pytest.mark.gpu
def test_static_largest_batch_that_fits(mla):
    h = 128
    parts = mla.mla_device_num_sm() // 2
    b = 255 - parts
    assert mla.mla_workspace_size(b, h, parts) <= mla.STATIC_WORKSPACE_BYTES
    gen = torch.Generator().manual_seed(3)
    lens = tuple(int(x) for x in torch.randint(0, 700, (b,), generator=gen))
    w = workloads.custom(batch=b, heads=h, seqlens=lens, seed=3)
    assert _compare_two_calls(mla, w) == parts


@pytest.mark.gpu
def test_static_fused_combine(mla):
    # the grid-synchronised combine in the static scratch: its barrier words sit in
    # the scratch's tail and keep the previous call's tag, which every call retags;
    # three calls in a row, each the same bits as the workspace entry's combine kernel
    w = workloads.custom(batch=5, heads=128, seqlens=(4097, 1, 0, 2000, 640), seed=8)
    inp = workloads.make_inputs(w, device="cuda")
    meta, num_splits = mla.mla_get_metadata(inp["cache_seqlens"], w.heads, 20)
    assert int(num_splits[-1]) > w.batch, "the case must split some sequence"
    args = (inp["q"], inp["kv_cache"], inp["block_table"], inp["cache_seqlens"],
            w.softmax_scale, meta, num_splits)
    ref_out, ref_lse = mla.mla_decode_fwd(*args)
    for call in range(3):
        out, lse = mla.mla_decode_fwd_static(*args, fused_combine=True)
        code, detail = mla.mla_get_device_error()
        assert code == 0, f"call {call}: device error {code}, detail {detail}"
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"call {call}: out bits"
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), f"call {call}: lse bits"
