"""CPU oracle for MLA decode (fp64), and the scheduler oracle.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
benchmark's CPU-baseline / reference leg import this package.  It shares no
code with the CUDA path and imports nothing from it.

`decode_rows` evaluates the plain definition in `mla_oracle.c` for chosen
(sequence, head) pairs; `decode` evaluates every pair.  Inputs are numpy
arrays holding the stored 16-bit patterns (fp16 or bf16), or the stored e4m3
bytes with one dequantisation scale each for q and the cache, and int32 tables.
"""
import ctypes
import os
import subprocess
import sysconfig
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import scheduler  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None

D = 576
DV = 512
DTYPES = {"fp16": 0, "bf16": 1, "e4m3": 2}


def build(src=_SRC, out=_LIB, extra_flags=()):
    """Compile the oracle with gcc (plain IEEE arithmetic: no fast-math, no FMA contraction)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def load(path=_LIB):
    """Load (building if needed) the oracle shared library."""
    global _lib
    with _lock:
        if path == _LIB and _lib is not None:
            return _lib
        if path == _LIB and (not os.path.exists(_LIB)
                             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
            build()
        lib = ctypes.CDLL(path)
        lib.oracle_mla_decode_rows.restype = ctypes.c_int
        lib.oracle_mla_decode_rows.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_double, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_mla_decode_rows_q.restype = ctypes.c_int
        lib.oracle_mla_decode_rows_q.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_double, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_mla_decode_rows_qs.restype = ctypes.c_int
        lib.oracle_mla_decode_rows_qs.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_double, ctypes.c_int, ctypes.c_double, ctypes.c_double,
            ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_widen.restype = ctypes.c_double
        lib.oracle_widen.argtypes = [ctypes.c_uint16, ctypes.c_int]
        if path == _LIB:
            _lib = lib
        return lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def decode_rows(q, kv, block_table, cache_seqlens, softmax_scale, dtype, rows,
                threads=1, lib=None, with_abs=False, seqlen_q=1, is_causal=False,
                q_scale=1.0, kv_scale=1.0):
    """Evaluate the definition for the (seq, row) pairs in `rows`.

    q            : uint16 [b, seqlen_q * h, 576]   (stored bits; row = qi * h + head),
                   or uint8 e4m3 bytes when dtype is "e4m3"
    kv           : uint16 [num_pages, page_size, 576] (uint8 for "e4m3")
    q_scale, kv_scale: dequantisation scales (e4m3 only; the values the definition
                   uses are q_scale * q and kv_scale * kv)
    block_table  : int32  [b, max_blocks]
    cache_seqlens: int32  [b]
    rows         : int array [n, 2] of (seq, row)
    seqlen_q, is_causal: query tokens per sequence; with is_causal, token qi sees
                   the cached tokens t < L - (seqlen_q - 1 - qi)
    Returns (out float64 [n, 512], lse float64 [n]), and with `with_abs` also
    absw float64 [n, 512] = sum_t p_t |v_t| per column: the scale of the terms
    each output sums, which bounds the error of any rounding of them.
    """
    lib = lib or load()
    fp8 = dtype == "e4m3"
    q = np.ascontiguousarray(q, dtype=np.uint8 if fp8 else np.uint16)
    kv = np.ascontiguousarray(kv, dtype=np.uint8 if fp8 else np.uint16)
    if not fp8:
        assert q_scale == 1.0 and kv_scale == 1.0, "scales apply to e4m3 inputs only"
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    b, nrows, d = q.shape
    assert d == D and kv.shape[2] == D and bt.shape[0] == b and sl.shape[0] == b
    assert seqlen_q >= 1 and nrows % seqlen_q == 0
    h = nrows // seqlen_q
    num_pages, page_size = kv.shape[0], kv.shape[1]
    n = rows.shape[0]
    out = np.zeros((n, DV), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    absw = np.zeros((n, DV), dtype=np.float64) if with_abs else None
    code = DTYPES[dtype]
    max_len = int(max(1, sl.max(initial=1)))

    def run(lo, hi):
        if hi <= lo:
            return 0
        rb = np.ascontiguousarray(rows[lo:hi, 0])
        rh = np.ascontiguousarray(rows[lo:hi, 1])
        o = out[lo:hi]
        ls = lse[lo:hi]
        ab = _ptr(absw[lo:hi]) if with_abs else None
        scratch = np.empty(max_len, dtype=np.float64)
        if fp8:
            return lib.oracle_mla_decode_rows_qs(
                b, int(seqlen_q), h, int(bool(is_causal)), _ptr(q), _ptr(kv), num_pages,
                page_size, _ptr(bt), bt.shape[1], _ptr(sl), float(softmax_scale), code,
                float(q_scale), float(kv_scale), hi - lo, _ptr(rb), _ptr(rh), _ptr(o), _ptr(ls),
                _ptr(scratch), ab)
        if seqlen_q == 1 and not is_causal:
            return lib.oracle_mla_decode_rows(
                b, h, _ptr(q), _ptr(kv), num_pages, page_size, _ptr(bt), bt.shape[1],
                _ptr(sl), float(softmax_scale), code, hi - lo, _ptr(rb), _ptr(rh),
                _ptr(o), _ptr(ls), _ptr(scratch), ab)
        return lib.oracle_mla_decode_rows_q(
            b, int(seqlen_q), h, int(bool(is_causal)), _ptr(q), _ptr(kv), num_pages, page_size,
            _ptr(bt), bt.shape[1], _ptr(sl), float(softmax_scale), code, hi - lo, _ptr(rb),
            _ptr(rh), _ptr(o), _ptr(ls), _ptr(scratch), ab)

    if threads <= 1 or n < 2:
        rc = run(0, n)
        if rc:
            raise ValueError("oracle: block table or row index out of range")
    else:
        bounds = np.linspace(0, n, threads + 1).astype(int)
        with ThreadPoolExecutor(threads) as ex:  # ctypes releases the GIL
            rcs = list(ex.map(lambda k: run(bounds[k], bounds[k + 1]), range(threads)))
        if any(rcs):
            raise ValueError("oracle: block table or row index out of range")
    return (out, lse, absw) if with_abs else (out, lse)


def decode(q, kv, block_table, cache_seqlens, softmax_scale, dtype, threads=1, seqlen_q=1,
           is_causal=False, q_scale=1.0, kv_scale=1.0):
    """Every (seq, row) pair; returns out [b, rows, 512] and lse [b, rows] (float64),
    rows = seqlen_q * h (token-major)."""
    b, h = q.shape[0], q.shape[1]
    rows = np.stack(np.meshgrid(np.arange(b), np.arange(h), indexing="ij"), -1).reshape(-1, 2)
    out, lse = decode_rows(q, kv, block_table, cache_seqlens, softmax_scale, dtype, rows,
                           threads=threads, seqlen_q=seqlen_q, is_causal=is_causal,
                           q_scale=q_scale, kv_scale=kv_scale)
    return out.reshape(b, h, DV), lse.reshape(b, h)


def widen(bits, dtype):
    """The oracle's own 16-bit -> double conversion (exported for its pin)."""
    lib = load()
    return lib.oracle_widen(int(bits), DTYPES[dtype])


def compact_pages(kv_pages_fn, block_table, cache_seqlens, seqs, page_size):
    """Gather only the pages that `seqs` use, and remap their table rows.

    kv_pages_fn(idx) must return the stored rows of physical pages `idx`
    (uint16 [len(idx), page_size, 576]).  Returns (kv, table, seqlens) for a
    cache that holds just those pages; the oracle then sees identical tokens.
    """
    bt = np.asarray(block_table, dtype=np.int64)
    sl = np.asarray(cache_seqlens, dtype=np.int64)
    seqs = np.asarray(seqs, dtype=np.int64)
    used = []
    for s in seqs:
        n = (int(sl[s]) + page_size - 1) // page_size
        used.extend(int(p) for p in bt[s, :n])
    uniq = np.array(sorted(set(used)), dtype=np.int64)
    remap = {int(p): k for k, p in enumerate(uniq)}
    table = np.zeros((len(seqs), bt.shape[1]), dtype=np.int32)
    for r, s in enumerate(seqs):
        n = (int(sl[s]) + page_size - 1) // page_size
        table[r, :n] = [remap[int(p)] for p in bt[s, :n]]
    kv = kv_pages_fn(uniq) if len(uniq) else np.zeros((0, page_size, D), np.uint16)  # (any dtype)
    return kv, table, sl[seqs].astype(np.int32)
