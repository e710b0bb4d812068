"""GPU parity of the FP8 (e4m3) KV cache against the fp64 oracle.

q and the cache are e4m3 bytes with one dequantisation scale each (the reading of
the TileLang guide's FP8-cache variant, section 变体内核); out is bf16.  Random
workloads are held to the bar derived from the e4m3 rounding of the softmax
weights (tests/_parity.py); inputs whose weights are exact powers of two are held
to half a bf16 ulp plus fp32 accumulation.
"""
import math

import numpy as np
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


SMALL = [
    dict(batch=5, heads=128, seqlens=(0, 1, 63, 130, 700)),
    dict(batch=3, heads=16, seqlens=(65, 4097, 2)),
    dict(batch=4, heads=100, seqlens=(17, 64, 129, 3000), page_size=128),
    dict(batch=2, heads=130, seqlens=(5000, 191), page_size=256),
    dict(batch=1, heads=1, seqlens=(300,)),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_fp8_small_cases(case):
    w = workloads.custom(name=f"fp8_small{case}", dtype="e4m3", seed=300 + case, **SMALL[case])
    stats, *_ = P.check_workload(w)
    assert stats["ref_max_abs"] > 0


def test_fp8_poisoned_tail_rows_are_never_read():
    # NaN bytes in the cache rows past each length (inside the last page)
    w = workloads.custom(3, 128, (70, 130, 5), "e4m3", seed=309, name="fp8_poison")
    P.check_workload(w, poison_tail=True)


@pytest.mark.parametrize("num_sm", [2, 20, None])
def test_fp8_split_invariance(num_sm):
    w = workloads.custom(4, 128, (3000, 50, 5000, 777), "e4m3", seed=310, name="fp8_splits")
    inputs = workloads.make_inputs(w, "cuda")
    stats, out, lse, meta, ns, _ = P.check_workload(w, num_sm=num_sm, inputs=inputs)
    if num_sm == 20:
        assert int(ns[-1]) > w.batch  # some sequence is split


def test_fp8_paged_config_full_size():
    """The paged shape with an FP8 cache (b = 64, h = 128, L = 4096), every row."""
    w = workloads.get("paged_fp8")
    P.check_workload(w)


def test_fp8_varlen_full_size():
    w = workloads.get("varlen", dtype="e4m3", seed=311)
    P.check_workload(w, seqs=workloads.sample_seqs(w, 32))


def test_fp8_hot_rows_few_heads():
    # 16 heads, long sequences, 1% of cache rows x8 before quantisation
    w = workloads.custom(16, 16, (32768,) * 16, "e4m3", seed=312, name="fp8_mqa",
                         hot_row_frac=0.01, hot_row_mult=8.0)
    P.check_workload(w)


def test_fp8_query_tokens_causal():
    w = workloads.custom(8, 128, (4096, 1, 2, 65, 700, 64, 3000, 129), "e4m3", seed=313,
                         name="fp8_mtp", seqlen_q=2, causal=True)
    P.check_workload(w)


def test_fp8_static_entry_matches():
    """The no-allocation entry on e4m3 inputs gives the same bits as mla_decode_fwd."""
    import mla_decode_gb300 as mla
    w = workloads.custom(4, 128, (3000, 50, 5000, 777), "e4m3", seed=314, name="fp8_static")
    x = workloads.make_inputs(w, "cuda")
    meta, ns = mla.mla_get_metadata(x["cache_seqlens"], w.heads)
    args = (x["q"], x["kv_cache"], x["block_table"], x["cache_seqlens"], w.softmax_scale, meta, ns)
    o1, l1 = mla.mla_decode_fwd(*args, **P.scales(x))
    o2, l2 = mla.mla_decode_fwd_static(*args, **P.scales(x))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert o1.dtype == torch.bfloat16


def _e4m3(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)


def _exact_case(lens, heads, seed, page_size=64, uniform=False):
    """Inputs whose softmax weights are exact powers of two: q has one nonzero column
    (540, in the RoPE part, so the value columns are untouched) equal to 1, the cache
    holds integers k_t in [-9, 0] in that column, q_scale = kv_scale = 1 and
    softmax_scale = ln 2, so the weights are 2^(k_t - m) for the reference max m
    (e4m3 holds 2^-9 .. 2^8 exactly).  uniform: q = 0, all weights equal."""
    rng = np.random.default_rng(seed)
    w = workloads.custom(len(lens), heads, lens, "e4m3", page_size=page_size,
                         softmax_scale=math.log(2.0), seed=seed, name="fp8_exact")
    x = workloads.make_inputs(w, "cpu")
    kv = x["kv_cache"].float()
    kv[:, :, 0, 540] = torch.from_numpy(rng.integers(-9, 1, size=kv.shape[:2]).astype(np.float32))
    q = torch.zeros(x["q"].shape)
    if not uniform:
        q[..., 540] = 1.0
    x["kv_cache"] = _e4m3(kv.numpy())
    x["q"] = _e4m3(q.numpy())
    x["q_scale"], x["kv_scale"] = 1.0, 1.0
    return w, {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}


@pytest.mark.parametrize("uniform", [False, True])
@pytest.mark.parametrize("num_sm", [20, None])
def test_fp8_exact_weights(uniform, num_sm):
    w, x = _exact_case((1, 63, 64, 200, 4096, 0, 1500), 128, seed=320, uniform=uniform)
    out, lse, meta, ns = P.run_gpu(x, w.heads, w.softmax_scale, num_sm=num_sm)
    ref_o, ref_l, ref_a = P.oracle_rows(w, x)
    full = np.isfinite(ref_l)
    d = P.check_exact_weights(out.reshape(w.batch, w.rows, -1)[torch.from_numpy(full).cuda()],
                              lse.reshape(w.batch, w.rows)[torch.from_numpy(full).cuda()],
                              ref_o[full], ref_l[full], ref_a[full], what="fp8 exact weights")
    assert d["out_max_abs"] >= 0
    # the empty sequence: zeros and -inf
    assert torch.all(out[5] == 0) and torch.all(torch.isneginf(lse[5]))


def test_fp8_scales_enter_linearly():
    """The scores take q_scale * kv_scale and out takes kv_scale: halving q_scale
    while doubling kv_scale leaves the scores (and lse) unchanged and doubles out
    exactly (a power-of-two factor is exact in every step)."""
    import mla_decode_gb300 as mla
    w = workloads.custom(3, 128, (700, 64, 1), "e4m3", seed=330, name="fp8_scales")
    x = workloads.make_inputs(w, "cuda")
    meta, ns = mla.mla_get_metadata(x["cache_seqlens"], w.heads)
    args = (x["q"], x["kv_cache"], x["block_table"], x["cache_seqlens"], w.softmax_scale, meta, ns)
    o1, l1 = mla.mla_decode_fwd(*args, q_scale=x["q_scale"], kv_scale=x["kv_scale"])
    o2, l2 = mla.mla_decode_fwd(*args, q_scale=x["q_scale"] / 2, kv_scale=x["kv_scale"] * 2)
    torch.cuda.synchronize()
    assert torch.equal(o2.float(), 2 * o1.float())
    assert torch.equal(l1, l2)
