"""Pins for the fp64 oracle: checks against what the pages and the mathematics fix.

None of these compares the oracle with itself.  Each pin comes from a
different statement of the same operation:
  * brute force: a naive softmax (no max subtraction, math.fsum) over the
    *logical* token sequence, before it is scattered into pages;
  * closed forms: len-1, identical scores, q = 0, two tokens, one dominant
    token, empty sequence;
  * invariants: page permutation, token permutation, head independence,
    softmax shift, and split + combine (the log-sum-exp merge of the TileLang
    MLA guide's combine kernel) equalling the unsplit result;
  * the 16-bit widening checked exhaustively against numpy / torch;
  * the weighted-absolute output (sum_t p_t |v_t|, the scale of the terms each
    output sums) against brute force, its closed forms and |out| <= absw;
  * several query tokens per sequence, causal and not, against brute force over
    each token's visible prefix of the logical cache.
Finally, mutants of the oracle source (a dropped RoPE term, v from the wrong
columns, a wrong page index, a missing max in lse, ...) must each fail a pin.
"""
import math
import os
import shutil
import tempfile

import numpy as np
import pytest
import torch

import oracle

D, DV = 576, 512


def bits(x, dtype):
    t = torch.as_tensor(np.asarray(x, dtype=np.float32))
    t = t.to(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16)


def vals(b, dtype):
    t = torch.from_numpy(np.asarray(b, dtype=np.uint16).view(np.int16))
    t = t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.to(torch.float64).numpy()


def paged(logical, page_size, rng, num_extra_pages=2):
    """Scatter logical caches [b][L_i, 576] into shuffled pages; return kv, table."""
    b = len(logical)
    nblk = [(x.shape[0] + page_size - 1) // page_size for x in logical]
    num_pages = sum(nblk) + num_extra_pages
    perm = rng.permutation(num_pages)
    kv = rng.integers(0, 2 ** 16, size=(num_pages, page_size, D)).astype(np.uint16)
    kv &= np.uint16(0x3FFF)  # finite garbage everywhere not overwritten
    table = np.full((b, max(1, max(nblk))), -1, dtype=np.int32)
    k = 0
    for i, x in enumerate(logical):
        for j in range(nblk[i]):
            page = int(perm[k]); k += 1
            table[i, j] = page
            rows = x[j * page_size:(j + 1) * page_size]
            kv[page, : rows.shape[0]] = rows
    return kv, table


def brute(qv, logical_v, scale):
    """Naive softmax over the logical sequence: exp without max subtraction."""
    s = [scale * math.fsum(qv * r) for r in logical_v]
    w = [math.exp(x) for x in s]
    z = math.fsum(w)
    out = np.array([math.fsum(w[t] * logical_v[t][d] for t in range(len(w))) / z
                    for d in range(DV)])
    return out, math.log(z)


def run_oracle(lib, q, kv, table, seqlens, scale, dtype):
    qq = np.asarray(q).reshape(q.shape[0], q.shape[1], D)
    b, h = qq.shape[:2]
    rows = np.stack(np.meshgrid(np.arange(b), np.arange(h), indexing="ij"), -1).reshape(-1, 2)
    out, lse = oracle.decode_rows(qq, kv, table, np.asarray(seqlens, np.int32), scale, dtype,
                                  rows, lib=lib)
    return out.reshape(b, h, DV), lse.reshape(b, h)


def run_oracle_abs(lib, q, kv, table, seqlens, scale, dtype):
    qq = np.asarray(q).reshape(q.shape[0], q.shape[1], D)
    b, h = qq.shape[:2]
    rows = np.stack(np.meshgrid(np.arange(b), np.arange(h), indexing="ij"), -1).reshape(-1, 2)
    out, lse, absw = oracle.decode_rows(qq, kv, table, np.asarray(seqlens, np.int32), scale, dtype,
                                        rows, lib=lib, with_abs=True)
    return out.reshape(b, h, DV), absw.reshape(b, h, DV)


# ----------------------------------------------------------------------------------------
# individual pins, written so that they can also be run against mutant builds

def pin_brute_force(lib):
    rng = np.random.default_rng(11)
    for dtype, page_size, lens in (("bf16", 16, (37, 80)), ("fp16", 64, (65, 3)),
                                   ("bf16", 256, (1, 300))):
        h = 3
        scale = 0.05
        logical = [bits(rng.standard_normal((L, D)), dtype) for L in lens]
        q = bits(rng.standard_normal((len(lens), h, D)), dtype)
        kv, table = paged(logical, page_size, rng)
        out, lse = run_oracle(lib, q, kv, table, lens, scale, dtype)
        for i in range(len(lens)):
            lv = vals(logical[i], dtype)
            for j in range(h):
                ref_o, ref_l = brute(vals(q[i, j], dtype), lv, scale)
                if not np.allclose(out[i, j], ref_o, rtol=1e-11, atol=1e-12):
                    return False
                if abs(lse[i, j] - ref_l) > 1e-11 * max(1.0, abs(ref_l)):
                    return False
    return True


def pin_len_one(lib):
    rng = np.random.default_rng(12)
    row = bits(rng.standard_normal((1, D)), "bf16")
    q = bits(rng.standard_normal((1, 2, D)), "bf16")
    kv, table = paged([row], 64, rng)
    out, lse = run_oracle(lib, q, kv, table, [1], 0.1, "bf16")
    v = vals(row[0], "bf16")
    for j in range(2):
        if not np.array_equal(out[0, j], v[:DV]):
            return False
        s0 = 0.1 * math.fsum(vals(q[0, j], "bf16") * v)
        if abs(lse[0, j] - s0) > 1e-12 * max(1, abs(s0)):
            return False
    return True


def pin_identical_scores(lib):
    """Zero latent query + equal RoPE keys: every score equal -> mean of v, lse = s + ln L."""
    rng = np.random.default_rng(13)
    L = 150
    x = rng.standard_normal((L, D))
    x[:, DV:] = rng.standard_normal(D - DV)  # same RoPE part for every token
    row = bits(x, "bf16")
    qf = rng.standard_normal((1, 1, D))
    qf[..., :DV] = 0.0
    q = bits(qf, "bf16")
    kv, table = paged([row], 64, rng)
    out, lse = run_oracle(lib, q, kv, table, [L], 0.07, "bf16")
    v = vals(row, "bf16")
    mean = v[:, :DV].mean(axis=0)
    s = 0.07 * math.fsum(vals(q[0, 0], "bf16") * v[0])
    return (np.allclose(out[0, 0], mean, rtol=1e-12, atol=1e-13)
            and abs(lse[0, 0] - (s + math.log(L))) < 1e-12)


def pin_zero_query(lib):
    rng = np.random.default_rng(14)
    L = 77
    row = bits(rng.standard_normal((L, D)), "fp16")
    q = np.zeros((1, 2, D), np.uint16)
    kv, table = paged([row], 16, rng)
    out, lse = run_oracle(lib, q, kv, table, [L], 0.3, "fp16")
    mean = vals(row, "fp16")[:, :DV].mean(axis=0)
    return (np.allclose(out[0], mean[None], rtol=1e-12, atol=1e-13)
            and np.allclose(lse[0], math.log(L), rtol=0, atol=1e-13))


def pin_two_tokens(lib):
    rng = np.random.default_rng(15)
    rows = bits(rng.standard_normal((2, D)), "bf16")
    q = bits(rng.standard_normal((1, 1, D)), "bf16")
    kv, table = paged([rows], 64, rng)
    scale = 0.11
    out, lse = run_oracle(lib, q, kv, table, [2], scale, "bf16")
    v = vals(rows, "bf16")
    qv = vals(q[0, 0], "bf16")
    s1, s2 = (scale * math.fsum(qv * v[k]) for k in range(2))
    a = 1.0 / (1.0 + math.exp(s2 - s1))  # sigmoid(s1 - s2)
    ref = a * v[0, :DV] + (1.0 - a) * v[1, :DV]
    ref_lse = max(s1, s2) + math.log1p(math.exp(-abs(s1 - s2)))
    return np.allclose(out[0, 0], ref, rtol=1e-12, atol=1e-13) and abs(lse[0, 0] - ref_lse) < 1e-12


def pin_dominant_token(lib):
    """One key aligned with q and scaled up: its weight is 1 to machine precision."""
    rng = np.random.default_rng(16)
    L = 130
    x = rng.standard_normal((L, D)) * 0.01
    qf = rng.standard_normal(D)
    x[57] = qf * 4.0
    rows = bits(x, "bf16")
    q = bits(qf[None, None], "bf16")
    kv, table = paged([rows], 64, rng)
    out, lse = run_oracle(lib, q, kv, table, [L], 1.0, "bf16")
    v = vals(rows, "bf16")
    s57 = math.fsum(vals(q[0, 0], "bf16") * v[57])
    return np.allclose(out[0, 0], v[57, :DV], rtol=0, atol=1e-12) and abs(lse[0, 0] - s57) < 1e-9


def pin_empty_sequence(lib):
    rng = np.random.default_rng(17)
    rows = bits(rng.standard_normal((10, D)), "bf16")
    q = bits(rng.standard_normal((2, 2, D)), "bf16")
    kv, table = paged([rows, rows], 64, rng)
    out, lse = run_oracle(lib, q, kv, table, [0, 10], 0.1, "bf16")
    return bool(np.all(out[0] == 0) and np.all(np.isneginf(lse[0])) and np.all(np.isfinite(lse[1])))


def pin_page_permutation(lib):
    rng = np.random.default_rng(18)
    logical = [bits(rng.standard_normal((L, D)), "bf16") for L in (200, 64)]
    q = bits(rng.standard_normal((2, 4, D)), "bf16")
    kv1, t1 = paged(logical, 64, np.random.default_rng(1))
    kv2, t2 = paged(logical, 64, np.random.default_rng(2))
    if np.array_equal(t1, t2):
        return False
    o1, l1 = run_oracle(lib, q, kv1, t1, [200, 64], 0.08, "bf16")
    o2, l2 = run_oracle(lib, q, kv2, t2, [200, 64], 0.08, "bf16")
    return np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_token_permutation(lib):
    rng = np.random.default_rng(19)
    L = 190
    rows = bits(rng.standard_normal((L, D)), "fp16")
    q = bits(rng.standard_normal((1, 3, D)), "fp16")
    perm = rng.permutation(L)
    kv1, t1 = paged([rows], 64, rng)
    kv2, t2 = paged([rows[perm]], 64, rng)
    o1, l1 = run_oracle(lib, q, kv1, t1, [L], 0.06, "fp16")
    o2, l2 = run_oracle(lib, q, kv2, t2, [L], 0.06, "fp16")
    return np.allclose(o1, o2, rtol=1e-12, atol=1e-14) and np.allclose(l1, l2, rtol=1e-13, atol=0)


def pin_head_independence(lib):
    rng = np.random.default_rng(20)
    rows = bits(rng.standard_normal((99, D)), "bf16")
    q = bits(rng.standard_normal((1, 5, D)), "bf16")
    kv, table = paged([rows], 64, rng)
    o_all, l_all = run_oracle(lib, q, kv, table, [99], 0.09, "bf16")
    for j in range(5):
        o1, l1 = run_oracle(lib, q[:, j:j + 1], kv, table, [99], 0.09, "bf16")
        if not (np.array_equal(o1[0, 0], o_all[0, j]) and l1[0, 0] == l_all[0, j]):
            return False
    return True


def pin_softmax_shift(lib):
    """A q component paired with a constant RoPE column adds the same constant to every
    score: out is unchanged and lse moves by exactly that constant."""
    rng = np.random.default_rng(21)
    L = 140
    x = rng.standard_normal((L, D))
    x[:, D - 1] = 2.0  # constant column outside the value part
    rows = bits(x, "bf16")
    qf = rng.standard_normal((1, 1, D))
    qa = qf.copy(); qa[..., D - 1] = 0.0
    qb = qf.copy(); qb[..., D - 1] = 3.0
    kv, table = paged([rows], 64, rng)
    scale = 0.125
    oa, la = run_oracle(lib, bits(qa, "bf16"), kv, table, [L], scale, "bf16")
    ob, lb = run_oracle(lib, bits(qb, "bf16"), kv, table, [L], scale, "bf16")
    shift = scale * 3.0 * 2.0
    return np.allclose(oa, ob, rtol=1e-12, atol=1e-14) and abs((lb - la)[0, 0] - shift) < 1e-12


def combine_natural(parts):
    """The combine kernel's merge (TileLang MLA guide, section Combine Kernel), in natural log."""
    lses = [l for _, l in parts]
    lmax = max(lses)
    if lmax == -math.inf:
        return np.zeros(DV), -math.inf
    tot = math.log(math.fsum(math.exp(l - lmax) for l in lses)) + lmax
    out = sum(math.exp(l - tot) * o for o, l in parts)
    return out, tot


def pin_split_combine(lib):
    """Evaluating two token ranges separately and merging them with the combine step gives
    the unsplit result (split-KV invariance of the definition)."""
    rng = np.random.default_rng(22)
    L = 333
    rows = bits(rng.standard_normal((L, D)), "bf16")
    q = bits(rng.standard_normal((1, 2, D)), "bf16")
    kv, table = paged([rows], 64, rng)
    full_o, full_l = run_oracle(lib, q, kv, table, [L], 0.1, "bf16")
    for cuts in ((128,), (64, 256), (1, 2, 300)):
        edges = (0,) + cuts + (L,)
        pieces = []
        for a, c in zip(edges[:-1], edges[1:]):
            kv_p, t_p = paged([rows[a:c]], 64, rng)
            pieces.append(run_oracle(lib, q, kv_p, t_p, [c - a], 0.1, "bf16"))
        for j in range(2):
            o, l = combine_natural([(p[0][0, j], p[1][0, j]) for p in pieces])
            if not (np.allclose(o, full_o[0, j], rtol=1e-12, atol=1e-13)
                    and abs(l - full_l[0, j]) < 1e-12):
                return False
    return True


def pin_batch_rows(lib):
    """q rows are indexed by (sequence, head): distinct shapes must not mix them up."""
    rng = np.random.default_rng(23)
    logical = [bits(rng.standard_normal((L, D)), "bf16") for L in (40, 70, 10)]
    q = bits(rng.standard_normal((3, 2, D)), "bf16")
    kv, table = paged(logical, 16, rng)
    out, lse = run_oracle(lib, q, kv, table, [40, 70, 10], 0.05, "bf16")
    for i in range(3):
        for j in range(2):
            ref_o, ref_l = brute(vals(q[i, j], "bf16"), vals(logical[i], "bf16"), 0.05)
            if not (np.allclose(out[i, j], ref_o, rtol=1e-11, atol=1e-12)
                    and abs(lse[i, j] - ref_l) < 1e-11):
                return False
    return True


def pin_abs_weights(lib):
    """sum_t p_t |v_t| per column: brute force (naive softmax, math.fsum), its closed
    forms (one token: |v|; identical scores: the mean of |v_t|) and |out| <= absw."""
    rng = np.random.default_rng(21)
    lens = (1, 50)
    scale = 0.07
    logical = [bits(rng.standard_normal((L, D)), "bf16") for L in lens]
    q = bits(rng.standard_normal((2, 2, D)), "bf16")
    kv, table = paged(logical, 16, rng)
    out, absw = run_oracle_abs(lib, q, kv, table, lens, scale, "bf16")
    if not np.array_equal(absw[0, 0], np.abs(vals(logical[0][0], "bf16"))[:DV]):
        return False
    if np.any(np.abs(out) > absw * (1 + 1e-12) + 1e-300):
        return False
    lv = vals(logical[1], "bf16")
    for j in range(2):
        qv = vals(q[1, j], "bf16")
        s_ = [scale * math.fsum(qv * r) for r in lv]
        w = [math.exp(x) for x in s_]
        z = math.fsum(w)
        ref = np.array([math.fsum(w[t] * abs(lv[t][d]) for t in range(len(w))) / z for d in range(DV)])
        if not np.allclose(absw[1, j], ref, rtol=1e-11, atol=1e-13):
            return False
    # identical scores: q = 0 gives every token the same weight
    q0 = np.zeros((2, 1, D), dtype=np.uint16)
    _, absw0 = run_oracle_abs(lib, q0, kv, table, lens, scale, "bf16")
    return np.allclose(absw0[1, 0], np.abs(lv).mean(axis=0)[:DV], rtol=1e-12, atol=1e-14)


def pin_query_tokens(lib):
    """seqlen_q query tokens per sequence, rows stored token-major (row = qi * h + head):
    against brute force over the logical cache.  Non-causal rows see all L tokens;
    causal token qi sees t < L - (seqlen_q - 1 - qi), nothing when that is <= 0
    (out = 0, lse = -inf)."""
    rng = np.random.default_rng(24)
    s_q, h, scale = 3, 2, 0.06
    lens = (1, 2, 5, 40)
    logical = [bits(rng.standard_normal((L, D)), "bf16") for L in lens]
    q = bits(rng.standard_normal((len(lens), s_q * h, D)), "bf16")
    kv, table = paged(logical, 16, rng)
    rows = np.stack(np.meshgrid(np.arange(len(lens)), np.arange(s_q * h), indexing="ij"),
                    -1).reshape(-1, 2)
    for causal in (False, True):
        out, lse = oracle.decode_rows(q, kv, table, np.asarray(lens, np.int32), scale, "bf16",
                                      rows, lib=lib, seqlen_q=s_q, is_causal=causal)
        out = out.reshape(len(lens), s_q * h, DV)
        lse = lse.reshape(len(lens), s_q * h)
        for i, L in enumerate(lens):
            lv = vals(logical[i], "bf16")
            for qi in range(s_q):
                n = max(0, L - (s_q - 1 - qi)) if causal else L
                for j in range(h):
                    r = qi * h + j
                    if n == 0:
                        if not (np.all(out[i, r] == 0) and lse[i, r] == -np.inf):
                            return False
                        continue
                    ref_o, ref_l = brute(vals(q[i, r], "bf16"), lv[:n], scale)
                    if not (np.allclose(out[i, r], ref_o, rtol=1e-11, atol=1e-12)
                            and abs(lse[i, r] - ref_l) < 1e-11 * max(1.0, abs(ref_l))):
                        return False
    return True


# ---- e4m3 cache with dequantisation scales

def bits8(x):
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def vals8(b):
    return torch.from_numpy(np.asarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def paged8(logical, page_size, rng, num_extra_pages=2):
    """paged() for e4m3 bytes: finite garbage everywhere not overwritten."""
    b = len(logical)
    nblk = [(x.shape[0] + page_size - 1) // page_size for x in logical]
    num_pages = sum(nblk) + num_extra_pages
    perm = rng.permutation(num_pages)
    kv = (rng.integers(0, 256, size=(num_pages, page_size, D)) & 0x77).astype(np.uint8)
    table = np.full((b, max(1, max(nblk))), -1, dtype=np.int32)
    k = 0
    for i, x in enumerate(logical):
        for j in range(nblk[i]):
            page = int(perm[k]); k += 1
            table[i, j] = page
            rows = x[j * page_size:(j + 1) * page_size]
            kv[page, : rows.shape[0]] = rows
    return kv, table


def pin_fp8_brute_force(lib):
    """e4m3 storage with scales against the naive softmax over the dequantised logical
    sequence (torch's e4m3 widening, an independent path)."""
    rng = np.random.default_rng(21)
    q_scale, kv_scale, scale = 0.37, 1.9, 0.05
    for page_size, lens in ((64, (37, 130)), (128, (1, 200))):
        h = 2
        logical = [bits8(rng.standard_normal((L, D)) * 3) for L in lens]
        q = bits8(rng.standard_normal((len(lens), h, D)) * 3)
        kv, table = paged8(logical, page_size, rng)
        rows = np.stack(np.meshgrid(np.arange(len(lens)), np.arange(h), indexing="ij"),
                        -1).reshape(-1, 2)
        out, lse = oracle.decode_rows(q, kv, table, np.asarray(lens, np.int32), scale, "e4m3",
                                      rows, lib=lib, q_scale=q_scale, kv_scale=kv_scale)
        out, lse = out.reshape(len(lens), h, DV), lse.reshape(len(lens), h)
        for i in range(len(lens)):
            lv = kv_scale * vals8(logical[i])
            for j in range(h):
                ref_o, ref_l = brute(q_scale * vals8(q[i, j]), lv, scale)
                if not np.allclose(out[i, j], ref_o, rtol=1e-11, atol=1e-12):
                    return False
                if abs(lse[i, j] - ref_l) > 1e-11 * max(1.0, abs(ref_l)):
                    return False
    return True


def pin_fp8_len_one(lib):
    """One cached token: out is exactly kv_scale times its value columns, lse its score."""
    rng = np.random.default_rng(22)
    row = bits8(rng.standard_normal((1, D)) * 4)
    q = bits8(rng.standard_normal((1, 1, D)) * 4)
    kv, table = paged8([row], 64, rng)
    out, lse = oracle.decode_rows(q, kv, table, np.asarray([1], np.int32), 0.1, "e4m3",
                                  np.array([[0, 0]], np.int32), lib=lib, q_scale=0.5,
                                  kv_scale=3.0)
    v = vals8(row[0])
    if not np.array_equal(out[0], 3.0 * v[:DV]):
        return False
    s0 = 0.1 * math.fsum(0.5 * vals8(q[0, 0]) * (3.0 * v))
    return abs(lse[0] - s0) <= 1e-12 * max(1, abs(s0))


PINS = [pin_brute_force, pin_len_one, pin_identical_scores, pin_zero_query, pin_two_tokens,
        pin_dominant_token, pin_empty_sequence, pin_page_permutation, pin_token_permutation,
        pin_head_independence, pin_softmax_shift, pin_split_combine, pin_batch_rows, pin_abs_weights,
        pin_query_tokens, pin_fp8_brute_force, pin_fp8_len_one]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    assert pin(oracle.load())


def test_widen_fp16_exhaustive():
    lib = oracle.load()
    allbits = np.arange(1 << 16, dtype=np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    got = np.array([lib.oracle_widen(int(x), 0) for x in allbits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_widen_bf16_exhaustive():
    lib = oracle.load()
    allbits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([lib.oracle_widen(int(x), 1) for x in allbits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_widen_e4m3_exhaustive():
    lib = oracle.load()
    allbits = np.arange(256, dtype=np.uint8)
    ref = vals8(allbits)
    got = np.array([lib.oracle_widen(int(x), 2) for x in allbits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_bad_table_is_an_error():
    rng = np.random.default_rng(3)
    rows = bits(rng.standard_normal((10, D)), "bf16")
    kv, table = paged([rows], 64, rng)
    table[0, 0] = kv.shape[0] + 5
    with pytest.raises(ValueError):
        run_oracle(oracle.load(), np.zeros((1, 1, D), np.uint16), kv, table, [10], 0.1, "bf16")


# ----------------------------------------------------------------------------------------
# mutants: each plausible slip in the oracle must be caught by some pin

MUTANTS = {
    "drop_rope_term": ("for (int c = 0; c < MLA_D; ++c)\n      dot +=",
                       "for (int c = 0; c < MLA_DV; ++c)\n      dot +="),
    "v_wrong_columns": ("out_row[d] += p * (kv_scale * elem(kv, v + d, dtype))",
                        "out_row[d] += p * (kv_scale * elem(kv, v + d + 64, dtype))"),
    "page_index_mod": ("int32_t page = table_row[t / page_size];\n    if (page < 0",
                       "int32_t page = table_row[t % page_size];\n    if (page < 0"),
    "row_in_page_div": ("(int64_t)page * page_size + t % page_size) * MLA_D;\n    double dot",
                        "(int64_t)page * page_size + t / page_size) * MLA_D;\n    double dot"),
    "lse_missing_max": ("*lse_out = m + log(z);", "*lse_out = log(z);"),
    "scale_dropped": ("scores[t] = softmax_scale * dot;", "scores[t] = dot;"),
    "max_sign_flip": ("z += exp(scores[t] - m);", "z += exp(m - scores[t]);"),
    "no_normalise": ("double p = exp(scores[t] - m) / z;", "double p = exp(scores[t] - m);"),
    "bf16_shift": ("(uint32_t)x << 16;", "(uint32_t)x << 15;"),
    "fp16_bias": ("e - 25);", "e - 24);"),
    "q_row_transposed": ("q + ((int64_t)bi * rows_per_seq + ri) * MLA_D",
                         "q + ((int64_t)ri * b + bi) * MLA_D"),
    "first_token_skipped": ("for (int t = 0; t < seqlen; ++t) z +=",
                            "for (int t = 1; t < seqlen; ++t) z +="),
    "abs_sign_kept": ("abs_row[d] += p * fabs(kv_scale * elem(kv, v + d, dtype));",
                      "abs_row[d] += p * (kv_scale * elem(kv, v + d, dtype));"),
    "causal_off_by_one": ("L - (seqlen_q - 1 - qi) : L", "L - (seqlen_q - qi) : L"),
    "causal_ignored": ("is_causal ? L - (seqlen_q - 1 - qi) : L", "L"),
    "query_token_reversed": ("int qi = ri / h;", "int qi = seqlen_q - 1 - ri / h;"),
    "query_rows_head_major": ("int qi = ri / h;", "int qi = ri % seqlen_q;"),
    "e4m3_bias": ("v = ldexp((double)(f | 8), e - 10);", "v = ldexp((double)(f | 8), e - 9);"),
    "e4m3_subnormal": ("v = ldexp((double)f, -9); /* subnormal", "v = ldexp((double)f, -10); /* subnormal"),
    "e4m3_nan_pattern": ("} else if (e == 15 && f == 7) {", "} else if (0) {"),
    "kv_scale_dropped_in_v": ("out_row[d] += p * (kv_scale * elem(kv, v + d, dtype));",
                              "out_row[d] += p * elem(kv, v + d, dtype);"),
    "q_scale_dropped": ("dot += q_scale * elem(q_row, c, dtype)", "dot += elem(q_row, c, dtype)"),
    "abs_unweighted": ("abs_row[d] += p * fabs(kv_scale * elem(kv, v + d, dtype));",
                       "abs_row[d] += fabs(kv_scale * elem(kv, v + d, dtype));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        path = os.path.join(tmp, "m.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        so = oracle.build(src=path, out=os.path.join(tmp, "m.so"))
        lib = oracle.load(so)
        caught = []
        for pin in PINS:
            try:
                ok = pin(lib)
            except Exception:
                ok = False
            if not ok:
                caught.append(pin.__name__)
        fp16 = (name == "fp16_bias")
        if fp16:  # only the exhaustive widening pin sees a bias slip on every value
            allbits = np.arange(0, 1 << 16, 97, dtype=np.uint16)
            ref = allbits.view(np.float16).astype(np.float64)
            got = np.array([lib.oracle_widen(int(x), 0) for x in allbits])
            if not (((got == ref) | (np.isnan(got) & np.isnan(ref))).all()):
                caught.append("widen_fp16")
        allbits8 = np.arange(256, dtype=np.uint8)  # the exhaustive e4m3 widening check
        got8 = np.array([lib.oracle_widen(int(x), 2) for x in allbits8])
        ref8 = vals8(allbits8)
        if not (((got8 == ref8) | (np.isnan(got8) & np.isnan(ref8))).all()):
            caught.append("widen_e4m3")
        assert caught, f"mutant {name} survived every pin"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
