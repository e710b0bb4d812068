"""GPU parity of the split layout: Q / Q_pe and KV / K_pe passed as separate
tensors, as the TileLang split kernel takes them ("用 TileLang 编写高性能 DeepSeek
MLA 内核…", section Split Kernel: the score is Q.KV^T + Q_pe.K_pe^T).

The oracle takes the concatenated rows (the same values), so the bar is the same
as for the fused layout.  The kernel fills its shared-memory tiles from either
layout in the same order, so a split-layout call must also give results
bit-identical to the fused call on the same values."""
import pytest
import torch

import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu

LAT = 512


@pytest.fixture(scope="module", autouse=True)
def built():
    from mla_decode_gb300 import _build
    _build.build()
    import mla_decode_gb300 as mla
    mla._load()


def split_views(inputs, mode):
    """(q, q_pe, kv, k_pe) for the split-layout call; None where the fused tensor is kept."""
    q, kv = inputs["q"], inputs["kv_cache"]
    if mode == "contiguous":
        return (q[..., :LAT].contiguous(), q[..., LAT:].contiguous(),
                kv[..., :LAT].contiguous(), kv[..., LAT:].contiguous())
    if mode == "views":  # the fused storage through split pointers (row stride 576)
        return q[..., :LAT], q[..., LAT:], kv[..., :LAT], kv[..., LAT:]
    if mode == "padded":  # wider rows and an offset inside them: strides 640 / 128
        qb = torch.full(q.shape[:3] + (640,), float("nan"), dtype=q.dtype, device=q.device)
        qb[..., 64:64 + LAT] = q[..., :LAT]
        pb = torch.full(q.shape[:3] + (128,), float("nan"), dtype=q.dtype, device=q.device)
        pb[..., 64:] = q[..., LAT:]
        kb = torch.full(kv.shape[:3] + (640,), float("nan"), dtype=kv.dtype, device=kv.device)
        kb[..., :LAT] = kv[..., :LAT]
        eb = torch.full(kv.shape[:3] + (128,), float("nan"), dtype=kv.dtype, device=kv.device)
        eb[..., 64:] = kv[..., LAT:]
        return qb[..., 64:64 + LAT], pb[..., 64:], kb[..., :LAT], eb[..., 64:]
    if mode == "k_only":
        return q, None, kv[..., :LAT].contiguous(), kv[..., LAT:].contiguous()
    if mode == "q_only":
        return q[..., :LAT].contiguous(), q[..., LAT:].contiguous(), kv, None
    raise ValueError(mode)


def run_split(inputs, w, mode, num_sm=None):
    import mla_decode_gb300 as mla
    q, q_pe, kv, k_pe = split_views(inputs, mode)
    meta, ns = mla.mla_get_metadata(inputs["cache_seqlens"], w.heads, num_sm)
    out, lse = mla.mla_decode_fwd(q, kv, inputs["block_table"], inputs["cache_seqlens"],
                                  w.softmax_scale, meta, ns, q_pe=q_pe, k_pe=k_pe)
    code, detail = mla.mla_get_device_error()
    assert code == 0, f"device error {code}, detail {detail}"
    return out, lse


CASES = [
    dict(batch=3, heads=128, seqlens=(1, 200, 1000), dtype="bf16"),
    dict(batch=2, heads=16, seqlens=(65, 4097), dtype="fp16", page_size=128),
    dict(batch=4, heads=130, seqlens=(0, 63, 129, 2500), dtype="bf16"),
]


@pytest.mark.parametrize("mode", ["contiguous", "views", "padded", "k_only", "q_only"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_split_layout_parity_and_identity(case, mode):
    w = workloads.custom(name=f"sep{case}", seed=300 + case, **CASES[case])
    inputs = workloads.make_inputs(w, "cuda")
    fused_o, fused_l, *_ = P.run_gpu(inputs, w.heads, w.softmax_scale)
    out, lse = run_split(inputs, w, mode)
    ref_o, ref_l, ref_a = P.oracle_rows(w, inputs)
    P.compare(out[:, 0], lse, ref_o, ref_l, ref_a, what=f"{w.name}/{mode}")
    assert torch.equal(out, fused_o), f"{mode}: out differs from the fused layout"
    assert torch.equal(lse, fused_l), f"{mode}: lse differs from the fused layout"


def test_split_layout_many_splits():
    w = workloads.custom(4, 128, (3000, 50, 5000, 777), "bf16", seed=11, name="sep_splits")
    inputs = workloads.make_inputs(w, "cuda")
    out, lse = run_split(inputs, w, "contiguous", num_sm=20)
    ref_o, ref_l, ref_a = P.oracle_rows(w, inputs)
    P.compare(out[:, 0], lse, ref_o, ref_l, ref_a, what="sep_splits")


def test_split_layout_paged_full_size():
    """The paged workload (b=64, h=128, L=4096) through separate tensors: identical
    to the fused call, and every sequence against the oracle."""
    w = workloads.get("paged")
    inputs = workloads.make_inputs(w, "cuda")
    fused_o, fused_l, *_ = P.run_gpu(inputs, w.heads, w.softmax_scale)
    out, lse = run_split(inputs, w, "contiguous")
    assert torch.equal(out, fused_o) and torch.equal(lse, fused_l)
    P.compare_chunked(w, inputs, [("split layout", out, lse)])
