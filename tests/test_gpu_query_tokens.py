"""GPU parity with several query tokens per sequence (seqlen_q > 1, causal or not),
FlashMLA's seqlen_q / is_causal fields ("DeepSeek开源周第一天：FlashMLA 深度分析",
section 内存访问优化): the s * h query rows of a sequence fold into one run of rows,
token-major, and under the causal mask query token qi sees the cached tokens
t < L - (s - 1 - qi).  Compared element by element with the oracle."""
import pytest

import workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mla_decode_gb300 import _build
    _build.build()
    import mla_decode_gb300 as mla
    mla._load()


CASES = [
    # L = 1 and 2 leave the first tokens' rows with nothing to see (out 0, lse -inf)
    dict(batch=4, heads=128, seqlens=(1, 2, 64, 1000), dtype="bf16", seqlen_q=2, causal=True),
    # 48 rows of three tokens in one 128-row tile: per-row limits differ inside a warp
    dict(batch=4, heads=16, seqlens=(2, 65, 129, 700), dtype="fp16", page_size=128, seqlen_q=3,
         causal=True),
    # four tokens over four 100-row tiles (the last one partial), no causal mask
    dict(batch=2, heads=100, seqlens=(63, 3000), dtype="bf16", seqlen_q=4, causal=False),
    # limits on both sides of a page boundary
    dict(batch=3, heads=128, seqlens=(64, 65, 128), dtype="bf16", seqlen_q=2, causal=True),
    # one query token through the causal path is the plain decode
    dict(batch=2, heads=128, seqlens=(300, 5), dtype="bf16", seqlen_q=1, causal=True),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_query_token_cases(case):
    w = workloads.custom(name=f"qtok{case}", seed=400 + case, **CASES[case])
    P.check_workload(w)


@pytest.mark.parametrize("num_sm", [2, 20, 1024, None])
def test_query_tokens_split_invariance(num_sm):
    """Splits of one block each (num_sm = 1024) leave causal rows whole splits that
    they cannot see; those partials must drop out of the combine."""
    w = workloads.custom(3, 64, (129, 2000, 3), "bf16", seed=410, name="qtok_splits",
                         seqlen_q=3, causal=True)
    P.check_workload(w, num_sm=num_sm)


def test_mtp_workload_full_size():
    """b=64, two causal query tokens, h=128, L=4096: 256 query rows per sequence."""
    w = workloads.get("mtp")
    P.check_workload(w)


def test_query_tokens_with_split_layout_and_static_entry():
    """Two causal query tokens with Q / Q_pe and KV / K_pe as separate tensors, through
    the workspace entry and the no-workspace entry: both bit-identical to the fused
    call, which matches the oracle."""
    import torch

    import mla_decode_gb300 as mla
    w = workloads.custom(3, 128, (2, 700, 1500), "bf16", seed=420, name="qtok_sep",
                         seqlen_q=2, causal=True)
    inputs = workloads.make_inputs(w, "cuda")
    stats, fused_o, fused_l, meta, ns, _ = P.check_workload(w, inputs=inputs)
    q, kv = inputs["q"], inputs["kv_cache"]
    sep = dict(q_pe=q[..., 512:].contiguous(), k_pe=kv[..., 512:].contiguous())
    args = (q[..., :512].contiguous(), kv[..., :512].contiguous(), inputs["block_table"],
            inputs["cache_seqlens"], w.softmax_scale, meta, ns)
    out, lse = mla.mla_decode_fwd(*args, is_causal=True, **sep)
    assert torch.equal(out, fused_o) and torch.equal(lse, fused_l)
    out_s, lse_s = mla.mla_decode_fwd_static(*args, is_causal=True, **sep)
    code, detail = mla.mla_get_device_error()
    assert code == 0, f"device error {code}, detail {detail}"
    assert torch.equal(out_s, fused_o) and torch.equal(lse_s, fused_l)
