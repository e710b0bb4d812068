"""GPU: the split kernel's own combine phase (fused_combine, a grid-wide barrier
between the split and combine phases, as in the persistent variant of the TileLang
kernels) against the separate combine kernel and the oracle: the same bits, on
batches whose sequences the scheduler splits, in every dtype; and its barrier
counters, which carry no initial value, under workspace garbage and CUDA graph
replays of one captured call."""
import pytest
import torch

import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mla_decode_gb300 import _build
    _build.build()
    import mla_decode_gb300 as mla
    mla._load()


def _uneven(dtype, seed):
    # lengths the scheduler splits unevenly (several sequences over several parts),
    # plus an empty sequence and a one-token one
    return workloads.custom(6, 128, (9000, 0, 3000, 1, 12000, 700), dtype, seed=seed,
                            name=f"fused_{dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "e4m3"])
@pytest.mark.parametrize("num_sm", [8, 20, 64, None])
def test_fused_combine_matches_combine_kernel_bitwise(dtype, num_sm):
    w = _uneven(dtype, 500 + num_sm if num_sm else 499)
    inputs = workloads.make_inputs(w, "cuda")
    out_f, lse_f, meta, ns = P.run_gpu(inputs, w.heads, w.softmax_scale, num_sm=num_sm,
                                       fused_combine=True)
    out_k, lse_k, *_ = P.run_gpu(inputs, w.heads, w.softmax_scale, num_sm=num_sm,
                                 fused_combine=False)
    assert int(ns[-1]) > w.batch, "the case must split some sequence"
    assert torch.equal(out_f.view(torch.int16), out_k.view(torch.int16))
    assert torch.equal(lse_f.view(torch.int32), lse_k.view(torch.int32))


def test_fused_combine_against_oracle_many_splits():
    # one long sequence over every part of the grid: the widest combine
    w = workloads.custom(1, 128, (40000,), "bf16", seed=77, name="fused_wide")
    stats, out, lse, meta, ns, _ = P.check_workload(w, fused_combine=True)
    assert int(ns[-1]) > 8


def test_fused_combine_varlen_full_size():
    # the serving-like batch (128 sequences of 1..16384 tokens, many split) with the
    # grid-synchronised combine: every sequence and head against the oracle
    w = workloads.get("varlen")
    stats, out, lse, meta, ns, _ = P.check_workload(w, fused_combine=True)
    assert int(ns[-1]) > w.batch


def test_fused_combine_paged_full_size():
    # the paged batch (64 x 4096 tokens, 76 SM pairs) in the mode the benchmark picks
    # for it: the schedule splits no sequence, so no combine runs; every sequence and
    # head against the oracle, and bit-identical to the combine-kernel mode
    w = workloads.get("paged")
    stats, out, lse, meta, ns, inputs = P.check_workload(w, fused_combine=True)
    assert int(ns[-1]) == w.batch
    out_k, lse_k, *_ = P.run_gpu(inputs, w.heads, w.softmax_scale, fused_combine=False)
    assert torch.equal(out.view(torch.int16), out_k.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_k.view(torch.int32))


@pytest.mark.parametrize("num_sm", [8, 20, 152])
def test_fused_combine_query_tokens_bitwise(num_sm):
    # three causal query tokens: the grid combines s * h rows per sequence (token-major,
    # two 128-row tiles), and rows that see none of a split's tokens drop that split
    w = workloads.custom(3, 64, (129, 2000, 3), "bf16", seed=411, name="fused_qtok", seqlen_q=3,
                         causal=True)
    x = workloads.make_inputs(w, "cuda")
    out_f, lse_f, meta, ns = P.run_gpu(x, w.heads, w.softmax_scale, num_sm=num_sm, is_causal=True,
                                       fused_combine=True)
    out_k, lse_k, *_ = P.run_gpu(x, w.heads, w.softmax_scale, num_sm=num_sm, is_causal=True)
    assert int(ns[-1]) > w.batch, "the case must split some sequence"
    assert torch.equal(out_f.view(torch.int16), out_k.view(torch.int16))
    assert torch.equal(lse_f.view(torch.int32), lse_k.view(torch.int32))


def test_fused_combine_rejects_a_grid_larger_than_the_device():
    # metadata shaped for 1024 SMs asks for 256 parts x 2 row tiles: more clusters than
    # the device holds at once, so the grid barrier could not pass; the call is refused
    # on the host before any launch, and the same call without fusing runs
    import mla_decode_gb300 as mla
    w = workloads.custom(3, 64, (129, 2000, 3), "bf16", seed=412, name="fused_big", seqlen_q=3,
                         causal=True)
    x = workloads.make_inputs(w, "cuda")
    meta, ns = mla.mla_get_metadata(x["cache_seqlens"], w.heads, 1024, seqlen_q=3)
    assert meta.shape[0] * 2 > mla.mla_device_num_sm() // 2
    args = (x["q"], x["kv_cache"], x["block_table"], x["cache_seqlens"], w.softmax_scale, meta, ns)
    with pytest.raises(mla.MlaError):
        mla.mla_decode_fwd(*args, is_causal=True, fused_combine=True)
    mla.mla_decode_fwd(*args, is_causal=True)
    torch.cuda.synchronize()
    code, detail = mla.mla_get_device_error()
    assert code == 0, f"device error {code} detail {detail}"


def test_fused_combine_mtp_full_size():
    # the two-token batch (64 x 4096 tokens, 256 rows) in the mode the benchmark picks
    # for it: 32 parts of whole sequences, nothing to combine; every sequence and row
    # against the oracle
    w = workloads.get("mtp")
    stats, out, lse, meta, ns, inputs = P.check_workload(w, fused_combine=True)
    assert int(ns[-1]) == w.batch


def test_fused_combine_garbage_workspace_and_graph_replays():
    import mla_decode_gb300 as mla
    w = _uneven("bf16", 321)
    x = workloads.make_inputs(w, "cuda")
    meta, ns = mla.mla_get_metadata(x["cache_seqlens"], w.heads, 20)
    assert int(ns[-1]) > w.batch
    need = mla.mla_workspace_size(w.batch, w.rows, meta.shape[0])
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # counters hold garbage
    call = mla.prepare_decode(x["q"], x["kv_cache"], x["block_table"], x["cache_seqlens"],
                              w.softmax_scale, meta, ns, workspace=ws, fused_combine=True)
    ref_o, ref_l, *_ = P.run_gpu(x, w.heads, w.softmax_scale, num_sm=20, fused_combine=False)
    call()
    torch.cuda.synchronize()
    assert torch.equal(call.out, ref_o) and torch.equal(call.lse, ref_l)
    # one captured call, replayed: the same tag each time, so the counters must come
    # back to zero after every run
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        call()
    for _ in range(4):
        call.out.zero_()
        call.lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(call.out, ref_o) and torch.equal(call.lse, ref_l)
    code, detail = mla.mla_get_device_error()
    assert code == 0, f"device error {code} detail {detail}"
