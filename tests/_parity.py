"""Helpers for the GPU parity tests: run the CUDA path through the C ABI, run the
oracle on host copies of the very same inputs, compare with the stated bar.

Tolerances (bf16/fp16 inputs, fp32 accumulation): out max-abs 2e-2 and
mean-abs 2e-3; lse max-abs 1e-3 (natural log); an empty sequence must give
out == 0 and lse == -inf exactly.

The out bounds are applied to the error measured in units of the scale of the
terms each output element sums: |gpu - ref| / max(1, w), w = sum_t p_t |v_t|
(the oracle's weighted-absolute output, the forward-error bound of a weighted
sum).  For unit-scale data w < 1 and this is exactly the absolute bound (every
N(0,1) workload).  Where rows scaled x8 dominate, the terms reach |p v| ~ 24 and
rounding each weight to 16 bits, at a running max of the kernel's choosing,
moves an output by ~2^-9 * 24 even when the terms cancel to |out| < 1.
"""
import os

import numpy as np
import torch

import oracle
import workloads

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3

ORACLE_THREADS = max(1, min(32, os.cpu_count() or 1))


def run_gpu(inputs, heads, scale, num_sm=None, is_causal=False):
    import mla_decode_gb300 as mla
    s_q = inputs["q"].shape[1]
    meta, num_splits = mla.mla_get_metadata(inputs["cache_seqlens"], heads, num_sm,
                                            seqlen_q=s_q)
    out, lse = mla.mla_decode_fwd(inputs["q"], inputs["kv_cache"], inputs["block_table"],
                                  inputs["cache_seqlens"], scale, meta, num_splits,
                                  is_causal=is_causal)
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
                                        seqlen_q=w.seqlen_q, is_causal=w.causal)
    return (out.reshape(len(seqs), w.rows, -1), lse.reshape(len(seqs), w.rows),
            absw.reshape(len(seqs), w.rows, -1))


def compare(out_gpu, lse_gpu, out_ref, lse_ref, abs_ref, what=""):
    """out_gpu [n, h, 512] (any float dtype), lse_gpu [n, h]; refs float64 numpy
    (abs_ref: the oracle's weighted-absolute scale of each output)."""
    og = out_gpu.float().cpu().numpy().astype(np.float64)
    lg = lse_gpu.float().cpu().numpy().astype(np.float64)
    empty = np.isneginf(lse_ref)
    assert np.all(np.isneginf(lg[empty])), f"{what}: empty rows must have lse -inf"
    assert np.all(og[empty] == 0), f"{what}: empty rows must be zero"
    assert np.all(np.isfinite(og)), f"{what}: non-finite output"
    err = np.abs(og - out_ref) / np.maximum(1.0, abs_ref)
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    full = ~empty
    lerr = float(np.abs(lg[full] - lse_ref[full]).max(initial=0.0))
    msg = f"{what}: out max {mx:.3e} mean {mean:.3e} lse {lerr:.3e}"
    assert mx <= OUT_MAX_ABS, msg
    assert mean <= OUT_MEAN_ABS, msg
    assert lerr <= LSE_MAX_ABS, msg
    return {"out_max_abs": mx, "out_mean_abs": mean, "lse_max_abs": lerr}


def check_workload(w, seqs=None, num_sm=None, poison_tail=False, inputs=None):
    if inputs is None:
        inputs = workloads.make_inputs(w, device="cuda", poison_tail=poison_tail)
    out, lse, meta, ns = run_gpu(inputs, w.heads, w.softmax_scale, num_sm, is_causal=w.causal)
    ref_o, ref_l, ref_a = oracle_rows(w, inputs, seqs)
    idx = torch.as_tensor(list(range(w.batch)) if seqs is None else list(seqs), device=out.device)
    stats = compare(out[idx].reshape(len(idx), w.rows, -1), lse[idx].reshape(len(idx), w.rows),
                    ref_o, ref_l, ref_a, what=w.name)
    log = os.environ.get("MLA_PARITY_LOG")
    if log:
        import json
        with open(log, "a") as f:
            f.write(json.dumps({"workload": w.name, "batch": w.batch, "heads": w.heads,
                                "seqlen_q": w.seqlen_q, "causal": w.causal,
                                "num_sm": num_sm, "rows": int(idx.numel()) * w.rows,
                                **stats}) + "\n")
    return stats, out, lse, meta, ns, inputs
