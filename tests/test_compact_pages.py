"""Pin for oracle.compact_pages, the helper that copies to the host only the cache
pages a chosen set of sequences reads and rewrites their block-table rows.

The GPU parity tests run the oracle on compacted caches, so the helper must change
nothing: for every selected sequence and every token t < L, the compacted cache
holds the very row the original table points at, and the oracle on the compacted
cache gives bit for bit what it gives on the whole cache.  Mutants of the helper
(a page dropped, an off-by-one remap, the wrong sequence's length) must fail.
"""
import inspect
import textwrap

import numpy as np
import pytest

import oracle

D = 576


def make_cache(rng, lens, page_size, extra_pages=3):
    nblk = [(L + page_size - 1) // page_size for L in lens]
    num_pages = sum(nblk) + extra_pages
    perm = rng.permutation(num_pages)
    kv = rng.integers(0, 1 << 16, size=(num_pages, page_size, D), dtype=np.uint16)
    kv &= np.uint16(0x3BFF)  # finite fp16 / bf16 patterns of moderate size
    table = np.full((len(lens), max(1, max(nblk))), -1, dtype=np.int32)
    k = 0
    for i, n in enumerate(nblk):
        table[i, :n] = perm[k:k + n]
        k += n
    q = rng.integers(0, 1 << 16, size=(len(lens), 4, D), dtype=np.uint16) & np.uint16(0x3BFF)
    return q, kv, table, np.asarray(lens, dtype=np.int32)


def pin_compact(compact, seed):
    """True when `compact` preserves every token of every selected sequence and the
    oracle's results on them, bit for bit."""
    rng = np.random.default_rng(seed)
    page_size = int(rng.choice([64, 128, 256]))
    b = int(rng.integers(2, 7))
    lens = [int(x) for x in rng.integers(0, 5 * page_size, size=b)]
    lens[0] = max(lens[0], 1)
    q, kv, table, sl = make_cache(rng, lens, page_size)
    seqs = [int(s) for s in rng.permutation(b)[: int(rng.integers(1, b + 1))]]
    kv_c, table_c, sl_c = compact(lambda idx: kv[np.asarray(idx, dtype=np.int64)], table, sl,
                                  seqs, page_size)
    if list(sl_c) != [int(sl[s]) for s in seqs]:
        return False
    for r, s in enumerate(seqs):
        for t in range(int(sl[s])):
            p, row = divmod(t, page_size)
            pc = int(table_c[r, p])
            if not (0 <= pc < kv_c.shape[0]):
                return False
            if not np.array_equal(kv_c[pc, row], kv[int(table[s, p]), row]):
                return False
    dtype = "fp16" if seed % 2 else "bf16"
    rows_full = np.array([(s, h) for s in seqs for h in range(q.shape[1])], dtype=np.int32)
    rows_c = np.array([(r, h) for r in range(len(seqs)) for h in range(q.shape[1])],
                      dtype=np.int32)
    full = oracle.decode_rows(q, kv, table, sl, 0.07, dtype, rows_full)
    comp = oracle.decode_rows(q[np.asarray(seqs)], kv_c, table_c, sl_c, 0.07, dtype, rows_c)
    return all(np.array_equal(a, c) for a, c in zip(full, comp))


@pytest.mark.parametrize("seed", range(10))
def test_compact_pages_changes_nothing(seed):
    assert pin_compact(oracle.compact_pages, seed)


MUTANTS = {
    "last_page_dropped": ("n = (int(sl[s]) + page_size - 1) // page_size\n        used",
                          "n = int(sl[s]) // page_size\n        used"),
    "remap_off_by_one": ("remap = {int(p): k for k, p in enumerate(uniq)}",
                         "remap = {int(p): (k + 1) % len(uniq) for k, p in enumerate(uniq)}"),
    "lengths_not_selected": ("return kv, table, sl[seqs].astype(np.int32)",
                             "return kv, table, sl[:len(seqs)].astype(np.int32)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_compact_pages_mutant_is_caught(name):
    src = textwrap.dedent(inspect.getsource(oracle.compact_pages))
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    ns = {"np": np, "D": oracle.D}
    exec(src.replace(old, new), ns)
    mutant = ns["compact_pages"]
    caught = False
    for seed in range(10):
        try:
            ok = pin_compact(mutant, seed)
        except Exception:
            ok = False
        if not ok:
            caught = True
            break
    assert caught, f"mutant {name} survived"
