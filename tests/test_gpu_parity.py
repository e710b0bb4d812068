"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same
seeded inputs, element by element, plus scheduler bit-exactness and device-side
error reporting."""
import numpy as np
import pytest
import torch

import workloads
from oracle import scheduler as sch
from tests import _parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mla_decode_gb300 import _build
    _build.build()
    import mla_decode_gb300 as mla
    mla._load()


def test_tiny_config_full():
    w = workloads.get("tiny")
    stats, *_ = P.check_workload(w)
    assert stats["out_max_abs"] < P.OUT_MAX_ABS


SMALL = [
    dict(batch=3, heads=128, seqlens=(1, 64, 1000), dtype="bf16"),
    dict(batch=2, heads=16, seqlens=(65, 4097), dtype="fp16"),
    dict(batch=4, heads=100, seqlens=(0, 63, 129, 700), dtype="bf16", page_size=128),
    dict(batch=1, heads=1, seqlens=(300,), dtype="bf16"),
    dict(batch=5, heads=130, seqlens=(2, 5000, 191, 64, 1), dtype="fp16", page_size=256),
    dict(batch=2, heads=128, seqlens=(8192, 0), dtype="bf16", shuffle=False),
    dict(batch=3, heads=64, seqlens=(3000, 2999, 1), dtype="bf16", softmax_scale=1.0),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_cases(case):
    kw = dict(SMALL[case])
    w = workloads.custom(name=f"small{case}", seed=100 + case, **kw)
    P.check_workload(w)


@pytest.mark.parametrize("num_sm", [2, 6, 20, 64, None])
def test_split_invariance(num_sm):
    w = workloads.custom(4, 128, (3000, 50, 5000, 777), "bf16", seed=7, name="splits")
    inputs = workloads.make_inputs(w, "cuda")
    stats, out, lse, meta, ns, _ = P.check_workload(w, num_sm=num_sm, inputs=inputs)
    base_o, base_l, *_ = P.run_gpu(inputs, w.heads, w.softmax_scale, num_sm=2)  # one split each
    d = (out.float() - base_o.float()).abs().max().item()
    assert d <= P.OUT_MAX_ABS
    assert (lse - base_l).abs().max().item() <= P.LSE_MAX_ABS


def test_poisoned_tail_rows_are_never_read():
    w = workloads.custom(3, 128, (70, 130, 5), "bf16", seed=9, name="poison")
    P.check_workload(w, poison_tail=True)


@pytest.mark.parametrize("seed", range(12))
def test_metadata_bit_exact(seed):
    import mla_decode_gb300 as mla
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 400))
    lens = np.where(rng.random(b) < 0.1, 0, rng.integers(1, 40000, size=b)).astype(np.int32)
    num_sm = int(rng.integers(1, 400))
    h = int(rng.choice([1, 16, 128, 200]))
    meta, ns = mla.mla_get_metadata(torch.from_numpy(lens).cuda(), h, num_sm)
    parts, _ = mla.mla_metadata_shape(b, h, num_sm)
    ref_meta, ref_ns, _ = sch.schedule_auto([int(x) for x in lens], parts, mla.SCHED_FIXED_COST,
                                            mla.SCHED_SEGMENT_COST, mla.SCHED_SPLIT_COST)
    assert meta.cpu().tolist() == ref_meta
    assert ns.cpu().tolist() == ref_ns


@pytest.mark.parametrize("b,L,h,num_sm", [(128, 4096, 128, 152), (128, 8192, 128, 152),
                                          (64, 4096, 128, 152), (132, 8192, 128, 152),
                                          (128, 2048, 128, 152), (64, 4096, 256, 152),
                                          (96, 6000, 128, 152), (120, 4096, 16, 100)])
def test_metadata_bit_exact_equal_batches(b, L, h, num_sm):
    # batches of equal sequences, where the split cost decides between part counts
    # whose most expensive parts are close
    import mla_decode_gb300 as mla
    lens = np.full(b, L, dtype=np.int32)
    meta, ns = mla.mla_get_metadata(torch.from_numpy(lens).cuda(), h, num_sm)
    parts, _ = mla.mla_metadata_shape(b, h, num_sm)
    ref_meta, ref_ns, p = sch.schedule_auto([L] * b, parts, mla.SCHED_FIXED_COST,
                                            mla.SCHED_SEGMENT_COST, mla.SCHED_SPLIT_COST)
    assert meta.cpu().tolist() == ref_meta
    assert ns.cpu().tolist() == ref_ns
    if (b, L, h) == (128, 4096, 128):  # the case the split cost moves to whole sequences
        assert p == 64 and ref_ns[-1] == b
        assert sch.choose_parts([L] * b, parts, mla.SCHED_FIXED_COST, mla.SCHED_SEGMENT_COST, 0) == 76


def test_out_of_range_page_is_reported_and_gpu_stays_usable():
    import mla_decode_gb300 as mla
    w = workloads.custom(2, 16, (100, 100), "bf16", seed=3, name="bounds")
    inputs = workloads.make_inputs(w, "cuda")
    bad = dict(inputs)
    bt = inputs["block_table"].clone()
    bt[1, 1] = w.num_pages + 1000
    bad["block_table"] = bt
    meta, ns = mla.mla_get_metadata(bad["cache_seqlens"], w.heads)
    mla.mla_decode_fwd(bad["q"], bad["kv_cache"], bad["block_table"], bad["cache_seqlens"],
                       w.softmax_scale, meta, ns)
    code, detail = mla.mla_get_device_error()
    assert code == mla_status("MLA_ERR_DEVICE_BOUNDS") and detail == 1
    # the context is intact: a correct call afterwards passes parity
    P.check_workload(w, inputs=inputs)


def test_length_past_table_capacity_is_reported_and_gpu_stays_usable():
    """cache_seqlens beyond max_blocks * page_size: the kernel reports the sequence,
    reads only clamped, in-range pages, and the next correct call passes parity."""
    import mla_decode_gb300 as mla
    w = workloads.custom(2, 16, (100, 100), "bf16", seed=4, name="capacity")
    inputs = workloads.make_inputs(w, "cuda")
    bad = dict(inputs)
    bad["cache_seqlens"] = torch.tensor([100, 300], dtype=torch.int32, device="cuda")  # 300 > 2 * 64
    meta, ns = mla.mla_get_metadata(bad["cache_seqlens"], w.heads)
    mla.mla_decode_fwd(bad["q"], bad["kv_cache"], bad["block_table"], bad["cache_seqlens"],
                       w.softmax_scale, meta, ns)
    code, detail = mla.mla_get_device_error()
    assert code == mla_status("MLA_ERR_DEVICE_BOUNDS") and detail == 1
    P.check_workload(w, inputs=inputs)


def mla_status(name):
    return {"MLA_ERR_DEVICE_BOUNDS": -9, "MLA_ERR_DEVICE_TIMEOUT": -8}[name]


# --- the pages' workloads at full size: every sequence and every head ------------------

def test_paged_config_full_size():
    w = workloads.get("paged")
    P.check_workload(w)


def test_paged_8k_config_full_size():
    # batch 128 x 8192-token caches in bf16 (the far corner of the paged target
    # range): every sequence and head against the oracle
    P.check_workload(workloads.get("paged_8k"))


def test_split_config_full_size_split_vs_unsplit():
    """The split workload under three scheduler settings: the default partition, at
    least four splits per sequence (1024 SMs' worth of parts) and one split each
    (num_split = 1), all compared with the oracle, then with one another."""
    w = workloads.get("split")
    inputs = workloads.make_inputs(w, "cuda")
    results = []
    for label, num_sm in (("default", None), ("many", 1024), ("one", 2)):
        out, lse, meta, ns = P.run_gpu(inputs, w.heads, w.softmax_scale, num_sm)
        per_seq = (ns[1:] - ns[:-1]).cpu()
        if label == "many":
            assert int(per_seq.min()) >= 4   # at least four splits per sequence
        if label == "one":
            assert int(per_seq.max()) == 1   # num_split = 1
        results.append((label, out, lse))
    P.compare_chunked(w, inputs, results)
    one = results[-1]
    for label, out, lse in results[:-1]:
        assert (out.float() - one[1].float()).abs().max().item() <= P.OUT_MAX_ABS
        assert (lse - one[2]).abs().max().item() <= P.LSE_MAX_ABS


def test_varlen_config_full_size():
    w = workloads.get("varlen")
    P.check_workload(w)


def test_mqa_config_full_size():
    """h = 16 (one partial 128-row tile) with 1% of cache rows scaled x8."""
    w = workloads.get("mqa")
    P.check_workload(w)


def test_tilelang_example_shape_full_size():
    """example_mla_decode.py's default shape: b=132, h=128, 8192 tokens, one
    contiguous 8192-token page per sequence, fp16."""
    w = workloads.get("tl_example")
    P.check_workload(w)


@pytest.mark.parametrize("L", [workloads.BENCH_SEQLENS[0], workloads.BENCH_SEQLENS[-1]])
def test_benchmark_sweep_ends_full_size(L):
    """benchmark_mla.py's default b=128, h=128 at the shortest and longest cache
    (every sequence at 1024 tokens; 16 seeded sequences at 32768, whose oracle alone
    would take half a minute per full batch)."""
    w = workloads.get(f"tl_bench_{L}")
    P.check_workload(w, seqs=None if L <= 8192 else workloads.sample_seqs(w, 16))
