"""Helpers for the GPU parity tests: run the CUDA path through the C ABI, run the
oracle on host copies of the very same inputs, compare with the stated bar.

Tolerances (bf16/fp16 inputs, fp32 accumulation): out max-abs 2e-2 and
mean-abs 2e-3, lse max-abs 1e-3 (natural log).  An empty row (a sequence of
length 0, or a causal row that sees no token) must give out == 0 and lse == -inf
exactly.

How the out bar is read.  Each element's error is taken in units of the scale
of the terms it sums:  e = |gpu - ref| / max(1, w),  w = sum_t p_t |v_t| (the
oracle's weighted-absolute output, the forward-error bound of a weighted sum);
max(e) <= 2e-2 and mean(e) <= 2e-3 on every element.  Where w <= 1 (unit-scale
terms) this is the absolute error itself.  Two things the method fixes make the
error grow with w rather than stay absolute: P is rounded to the input dtype
before P.V (TileLang's split kernel casts acc_s to the input dtype), which moves
an output by up to about 2^-9 w in bf16, and `out` is returned in the input
dtype, whose own rounding at |out| = 8..16 is already 2^-5 in bf16.  Both bite
only on the workload whose cache has rows scaled x8 (|out| up to ~40).  So, in
addition, wherever the output format can hold the values to the bar (every
|ref| below 8 for bf16, 64 for fp16: all the N(0, 1) workloads), the plain
|gpu - ref| must meet max 2e-2 and mean 2e-3 too.  The log records the plain
error, the weighted one and the error beyond the output format's rounding.

e4m3 cache (bf16 out).  The weights are rounded to e4m3 before P.V (3 fraction
bits: a relative error |d_t| <= 2^-4 for weights in e4m3's normal range) and O
is divided by the sum of the unrounded weights (as TileLang's split kernel
sums acc_s before its cast), so the kernel's output is sum_t w_t (1 + d_t) v_t:
|gpu - ref| <= 2^-4 * w.  The bar adds the bf16 rounding of out (2^-9 |out|,
|out| <= w) and fp32 accumulation (1e-4 w): max(e) <= E4M3_OUT_MAX = 0.065.  For
the mean, with independent zero-mean rounding errors of rms at most
2^-4 / sqrt(3) (uniform absolute error within an ulp of 2^-3 of the binade),
E|gpu - ref| <= 2^-4 / sqrt(3) * w, so mean(e) <= E4M3_OUT_MEAN = 0.037.
The lse bar is the 16-bit one (the scores are exact products summed in fp32, and
the lse uses the unrounded weights).  Where every weight is a power of two that
e4m3 holds exactly, the rounding is exact and check_exact_weights holds the
output to half a bf16 ulp plus 1e-4 * max(1, w).

Whole workloads are compared in chunks of sequences, so that the host copy of
the pages a chunk reads stays within a fixed budget.
"""
import json
import os

import numpy as np
import torch

import oracle
import workloads

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3
E4M3_OUT_MAX = 0.065
E4M3_OUT_MEAN = 0.037
EXACT_REL = 1e-4

ORACLE_THREADS = max(1, min(32, os.cpu_count() or 1))
HOST_KV_BUDGET = 1 << 30  # bytes of cache pages copied to the host per chunk


def scales(inputs):
    """The e4m3 dequantisation scales of a workload's inputs (1, 1 for 16-bit ones)."""
    return dict(q_scale=inputs.get("q_scale", 1.0), kv_scale=inputs.get("kv_scale", 1.0))


def run_gpu(inputs, heads, scale, num_sm=None, is_causal=False, fused_combine=False):
    import mla_decode_gb300 as mla
    s_q = inputs["q"].shape[1]
    meta, num_splits = mla.mla_get_metadata(inputs["cache_seqlens"], heads, num_sm,
                                            seqlen_q=s_q)
    out, lse = mla.mla_decode_fwd(inputs["q"], inputs["kv_cache"], inputs["block_table"],
                                  inputs["cache_seqlens"], scale, meta, num_splits,
                                  is_causal=is_causal, fused_combine=fused_combine,
                                  **scales(inputs))
    code, detail = mla.mla_get_device_error()
    assert code == 0, f"device error {code} ({mla.mla_status_string(code)}), detail {detail}"
    return out, lse, meta, num_splits


def oracle_rows(w, inputs, seqs=None):
    """Oracle out [n_seq, rows, 512], lse [n_seq, rows] and the weighted-absolute scale
    [n_seq, rows, 512] for sequences `seqs` (all if None); rows = seqlen_q * h,
    token-major."""
    q = inputs["q"]
    kv = inputs["kv_cache"]
    bt = inputs["block_table"].cpu().numpy()
    sl = inputs["cache_seqlens"].cpu().numpy()
    if seqs is None:
        seqs = list(range(w.batch))
    seqs = list(seqs)

    def pages(idx):
        sel = kv.index_select(0, torch.as_tensor(idx, device=kv.device))
        return workloads.to_bits(sel[:, :, 0, :])

    kv_c, table_c, sl_c = oracle.compact_pages(pages, bt, sl, seqs, w.page_size)
    q_c = workloads.to_bits(q[torch.as_tensor(seqs, device=q.device)]).reshape(len(seqs), w.rows,
                                                                              -1)
    rows = np.stack(np.meshgrid(np.arange(len(seqs)), np.arange(w.rows), indexing="ij"),
                    -1).reshape(-1, 2)
    out, lse, absw = oracle.decode_rows(q_c, kv_c, table_c, sl_c, w.softmax_scale, w.dtype, rows,
                                        threads=ORACLE_THREADS, with_abs=True,
                                        seqlen_q=w.seqlen_q, is_causal=w.causal, **scales(inputs))
    return (out.reshape(len(seqs), w.rows, -1), lse.reshape(len(seqs), w.rows),
            absw.reshape(len(seqs), w.rows, -1))


def seq_chunks(w, seqs, budget=HOST_KV_BUDGET):
    """Consecutive groups of `seqs` whose pages take at most `budget` bytes on the host
    (a sequence larger than the budget forms a group of its own)."""
    page_bytes = w.page_size * workloads.D * w.elem_bytes
    chunk, used = [], 0
    for s in seqs:
        b = max(1, w.blocks_per_seq[s]) * page_bytes
        if chunk and used + b > budget:
            yield chunk
            chunk, used = [], 0
        chunk.append(s)
        used += b
    if chunk:
        yield chunk


def half_ulp(x, dtype):
    """Half the spacing of the 16-bit format `dtype` at |x| (0 at x = 0)."""
    x = np.abs(x)
    _, e = np.frexp(x)                    # x = m * 2^e, 0.5 <= m < 1
    bits = 8 if dtype == "bf16" else 11   # significand bits, the implicit one included
    h = np.ldexp(0.5, e - bits)
    if dtype == "fp16":
        h = np.maximum(h, 2.0 ** -25)     # subnormal spacing
    return np.where(x == 0, 0.0, h)


def representable_bar(dtype):
    """Largest |out| below which half an ulp of `dtype` stays within the max-abs bar."""
    return 8.0 if dtype == "bf16" else 64.0


class ErrorStats:
    """Running max and mean of the out error over every element compared (in units of
    max(1, w); plain; beyond the output format's rounding), and the lse error.
    dtype: the input dtype ("bf16", "fp16", "e4m3"); the output's is bf16 for e4m3."""

    def __init__(self, dtype):
        self.in_dtype = dtype
        self.dtype = "bf16" if dtype == "e4m3" else dtype
        self.w_max = 0.0        # |gpu - ref| / max(1, w)
        self.w_sum = 0.0
        self.raw_max = 0.0      # |gpu - ref|
        self.raw_sum = 0.0
        self.fmt_max = 0.0      # max(0, |gpu - ref| - ulp/2)
        self.count = 0
        self.lse_max = 0.0
        self.ref_max = 0.0
        self.rows = 0

    def add(self, out_gpu, lse_gpu, out_ref, lse_ref, abs_ref, what=""):
        og = out_gpu.float().cpu().numpy().astype(np.float64)
        lg = lse_gpu.float().cpu().numpy().astype(np.float64)
        empty = np.isneginf(lse_ref)
        assert np.all(np.isneginf(lg[empty])), f"{what}: empty rows must have lse -inf"
        assert np.all(og[empty] == 0), f"{what}: empty rows must be zero"
        assert np.all(np.isfinite(og)), f"{what}: non-finite output"
        raw = np.abs(og - out_ref)
        ew = raw / np.maximum(1.0, abs_ref)
        self.w_max = max(self.w_max, float(ew.max(initial=0.0)))
        self.w_sum += float(ew.sum())
        self.raw_max = max(self.raw_max, float(raw.max(initial=0.0)))
        self.raw_sum += float(raw.sum())
        fmt = raw - half_ulp(np.maximum(np.abs(og), np.abs(out_ref)), self.dtype)
        self.fmt_max = max(self.fmt_max, float(fmt.max(initial=0.0)))
        self.count += raw.size
        self.ref_max = max(self.ref_max, float(np.abs(out_ref).max(initial=0.0)))
        full = ~empty
        self.lse_max = max(self.lse_max, float(np.abs(lg[full] - lse_ref[full]).max(initial=0.0)))
        self.rows += lse_ref.size

    def mean(self, total):
        return total / self.count if self.count else 0.0

    def as_dict(self):
        return {"out_max_abs": self.raw_max, "out_mean_abs": self.mean(self.raw_sum),
                "out_max_weighted": self.w_max, "out_mean_weighted": self.mean(self.w_sum),
                "out_max_beyond_format": self.fmt_max, "lse_max_abs": self.lse_max,
                "ref_max_abs": self.ref_max, "rows": self.rows}

    def check(self, what=""):
        d = self.as_dict()
        msg = (f"{what}: out max {d['out_max_abs']:.3e} mean {d['out_mean_abs']:.3e} "
               f"(in units of max(1, w): max {d['out_max_weighted']:.3e} mean "
               f"{d['out_mean_weighted']:.3e}; beyond the {self.dtype} rounding: max "
               f"{d['out_max_beyond_format']:.3e}; |ref| up to {self.ref_max:.3g}); "
               f"lse {self.lse_max:.3e}; {self.rows} rows")
        assert self.lse_max <= LSE_MAX_ABS, msg
        if self.in_dtype == "e4m3":
            assert d["out_max_weighted"] <= E4M3_OUT_MAX, msg
            assert d["out_mean_weighted"] <= E4M3_OUT_MEAN, msg
            return d
        assert d["out_max_weighted"] <= OUT_MAX_ABS, msg
        assert d["out_mean_weighted"] <= OUT_MEAN_ABS, msg
        if self.ref_max < representable_bar(self.dtype):
            assert d["out_max_abs"] <= OUT_MAX_ABS, msg
            assert d["out_mean_abs"] <= OUT_MEAN_ABS, msg
        return d


def compare(out_gpu, lse_gpu, out_ref, lse_ref, abs_ref, what="", in_dtype=None):
    """out_gpu [n, rows, 512] (bf16 or fp16), lse_gpu [n, rows]; refs float64 numpy
    (abs_ref: the oracle's weighted-absolute scale of each output).  in_dtype: the
    inputs' dtype when it is not the output's (e4m3)."""
    st = ErrorStats(in_dtype or ("bf16" if out_gpu.dtype == torch.bfloat16 else "fp16"))
    st.add(out_gpu, lse_gpu, out_ref, lse_ref, abs_ref, what)
    return st.check(what)


def compare_chunked(w, inputs, outs, seqs=None, what=None):
    """Compare GPU results with the oracle over `seqs` (all by default), a chunk of
    sequences at a time.  outs: list of (label, out [b, s, h, 512], lse) to check
    against the same oracle values.  Returns {label: stats}."""
    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    stats = {label: ErrorStats(w.dtype) for label, _, _ in outs}
    for chunk in seq_chunks(w, seqs):
        ref_o, ref_l, ref_a = oracle_rows(w, inputs, chunk)
        for label, out, lse in outs:
            idx = torch.as_tensor(chunk, device=out.device)
            stats[label].add(out[idx].reshape(len(chunk), w.rows, -1),
                             lse[idx].reshape(len(chunk), w.rows), ref_o, ref_l, ref_a,
                             what=f"{what or w.name}/{label}")
    result = {}
    for label, st in stats.items():
        name = f"{what or w.name}/{label}" if len(stats) > 1 else (what or w.name)
        _log(w, name, st.as_dict())
        result[label] = st.check(name)
    return result


def _log(w, name, stats, num_sm=None):
    log = os.environ.get("MLA_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"workload": name, "batch": w.batch, "heads": w.heads,
                                "seqlen_q": w.seqlen_q, "causal": w.causal,
                                "num_sm": num_sm, **stats}) + "\n")


def check_workload(w, seqs=None, num_sm=None, poison_tail=False, inputs=None, fused_combine=False):
    if inputs is None:
        inputs = workloads.make_inputs(w, device="cuda", poison_tail=poison_tail)
    out, lse, meta, ns = run_gpu(inputs, w.heads, w.softmax_scale, num_sm, is_causal=w.causal,
                                 fused_combine=fused_combine)
    stats = compare_chunked(w, inputs, [("out", out, lse)], seqs)["out"]
    return stats, out, lse, meta, ns, inputs


def check_exact_weights(out_gpu, lse_gpu, out_ref, lse_ref, abs_ref, what=""):
    """e4m3 inputs whose softmax weights are all powers of two in e4m3's range, so
    that rounding them is exact: |gpu - ref| <= half a bf16 ulp of the larger of
    the two plus EXACT_REL * max(1, w) (fp32 accumulation), and the lse bar."""
    og = out_gpu.float().cpu().numpy().astype(np.float64)
    lg = lse_gpu.float().cpu().numpy().astype(np.float64)
    raw = np.abs(og - out_ref)
    bar = half_ulp(np.maximum(np.abs(og), np.abs(out_ref)), "bf16") + EXACT_REL * np.maximum(1.0, abs_ref)
    worst = float((raw - bar).max(initial=-1.0))
    lse_err = float(np.abs(lg - lse_ref).max(initial=0.0))
    assert worst <= 0, f"{what}: exceeds the exact-weight bar by {worst:.3e} (max |err| {raw.max():.3e})"
    assert lse_err <= LSE_MAX_ABS, f"{what}: lse {lse_err:.3e}"
    return {"out_max_abs": float(raw.max(initial=0.0)), "lse_max_abs": lse_err}
