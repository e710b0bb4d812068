"""The values the source pages print (tests/golden/page_values.txt, each cited there)
against the library's header constants, the binding, the workloads and the oracle."""
import math
import os
import re

import numpy as np

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "page_values.txt")


def page_values():
    vals = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            pairs = dict(r.split("=", 1) for r in rest if "=" in r)
            vals[key] = pairs if pairs else rest
    return vals


def header_macros():
    text = open(os.path.join(ROOT, "include", "mla_decode.h"), encoding="utf-8").read()
    return {m.group(1): m.group(2) for m in re.finditer(r"^#define\s+(MLA_\w+)\s+(\S+)", text,
                                                       flags=re.M)}


V = page_values()


def one(key):
    return V[key][0]


def test_fixture_is_complete():
    for key in ("head_dim_qk", "head_dim_latent", "head_dim_rope", "head_dim_v", "log2e",
                "kv_heads", "example_decode", "example_paged", "benchmark_mla",
                "benchmark_dtype", "benchmark_batches", "page_block", "flashmla_shape"):
        assert key in V, key


def test_head_dims_match_the_library():
    import mla_decode_gb300 as mla
    qk, lat, rope, v = (int(one(k)) for k in ("head_dim_qk", "head_dim_latent", "head_dim_rope",
                                              "head_dim_v"))
    assert qk == lat + rope
    h = header_macros()
    assert int(h["MLA_HEAD_DIM"]) == qk and int(h["MLA_HEAD_DIM_V"]) == v == lat
    assert (mla.HEAD_DIM, mla.HEAD_DIM_V, mla.ROPE_DIM) == (qk, v, rope)
    assert (workloads.D, workloads.DV) == (qk, v)
    fm = V["flashmla_shape"]
    assert (int(fm["q"]), int(fm["v"])) == (qk, v)
    assert int(one("kv_heads")) == 1


def test_printed_log2e():
    # printed to 8 decimals: the true value rounds to it
    assert abs(math.log2(math.e) - float(one("log2e"))) < 0.5e-8


def test_oracle_agrees_with_the_exp2_form_of_the_printed_constant():
    """The pages compute softmax as exp2 of the scores times scale*log2(e); the oracle
    uses exp of the scaled scores.  With the printed 8-decimal constant the two agree
    to the constant's precision (relative exponent error below 4e-9)."""
    import oracle
    w = workloads.custom(1, 4, (100,), "bf16", seed=21, shuffle=False, name="exp2")
    x = workloads.make_inputs(w, "cpu")
    qb = workloads.to_bits(x["q"][:, 0])
    kvb = workloads.to_bits(x["kv_cache"][:, :, 0])
    out, lse = oracle.decode(qb, kvb, x["block_table"].numpy(), x["cache_seqlens"].numpy(),
                             w.softmax_scale, w.dtype)
    q = x["q"][0, 0].double().numpy()                          # [h, 576]
    kv = x["kv_cache"][:, :, 0].double().numpy().reshape(-1, 576)[:100]
    c = float(one("log2e"))
    s2 = (q @ kv.T) * w.softmax_scale * c                       # base-2 scores
    m2 = s2.max(axis=1, keepdims=True)
    p = np.exp2(s2 - m2)
    ref_out = (p @ kv[:, :512]) / p.sum(axis=1, keepdims=True)
    ref_lse = (np.log2(p.sum(axis=1)) + m2[:, 0]) / c           # back to natural log
    assert np.abs(out[0] - ref_out).max() < 1e-7
    assert np.abs(lse[0] - ref_lse).max() < 1e-6


def test_workloads_cover_the_printed_shapes():
    cfg = workloads.configs()
    ex = V["example_decode"]
    w = cfg["tl_example"]
    assert (w.batch, w.heads, int(w.seqlens[0])) == (int(ex["batch"]), int(ex["heads"]),
                                                     int(ex["kv_ctx"]))
    assert int(ex["dim"]) + int(ex["pe_dim"]) == workloads.D and int(ex["kv_heads"]) == 1
    pg = V["example_paged"]
    w = cfg["split"]
    assert (w.batch, w.heads, int(w.seqlens[0])) == (int(pg["batch"]), int(pg["h_q"]),
                                                     int(pg["cache_seqlen"]))
    assert (int(pg["d"]), int(pg["dv"])) == (workloads.D, workloads.DV)
    bm = V["benchmark_mla"]
    lo, hi = int(bm["seqlen_min"]), int(bm["seqlen_max"])
    sweep = sorted(int(w.seqlens[0]) for n, w in cfg.items() if n.startswith("tl_bench_"))
    assert sweep[0] == lo and sweep[-1] == hi
    assert all(b == 2 * a for a, b in zip(sweep, sweep[1:]))
    for n, w in cfg.items():
        if n.startswith("tl_"):
            assert w.dtype == one("benchmark_dtype")
            assert w.heads == int(bm["h_q"])
            if n.startswith("tl_bench_"):
                assert w.batch == int(bm["batch"])
    batches = {w.batch for w in cfg.values() if w.heads == 128}
    assert {int(b) for b in V["benchmark_batches"]} <= batches


def test_page_block():
    blk = int(one("page_block"))
    assert int(header_macros()["MLA_BLOCK_N"]) == blk
    for n in ("paged", "split", "varlen", "mqa"):
        assert workloads.get(n).page_size == blk

