"""Seeded synthetic MLA-decode workloads (shared by the tests, the smoke check and the bench).

This module only draws inputs: it holds none of the method's arithmetic.  Both
the CUDA path and the CPU oracle consume exactly the tensors built here (the
oracle gets host copies of the same stored 16-bit values).

Shapes follow the pages' decode workloads: one query token per sequence,
h query heads, one latent KV head, rows of 576 = 512 latent + 64 RoPE, a cache
paged in blocks of `page_size` tokens addressed through a block table.

Value recipe (all seeded):
  * q and every cached row ~ N(0, 1) drawn in fp32 with a torch.Generator on
    the target device, in fixed-size chunks, then rounded to the dtype;
  * optionally a fraction of physical cache rows is multiplied by a factor
    before rounding (all 576 columns), to stress the running-max logic;
  * the block table maps each sequence's logical blocks to a seeded random
    permutation of the physical pages (or the identity when not shuffled);
  * table entries past a sequence's last block are -1 (never read);
  * cache_seqlens are given or drawn from a numpy PCG64 stream (platform
    independent).
"""
from dataclasses import dataclass, replace

import numpy as np
import torch

D = 576
DV = 512
_CHUNK = 1 << 26  # elements drawn per generator call


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    seqlens: tuple          # per-sequence cache length
    dtype: str              # "bf16" | "fp16"
    page_size: int = 64
    softmax_scale: float = 192 ** -0.5
    seed: int = 0
    shuffle: bool = True
    hot_row_frac: float = 0.0
    hot_row_mult: float = 1.0
    notes: str = ""
    seqlen_q: int = 1       # query tokens per sequence (rows token-major)
    causal: bool = False    # token qi sees the cached tokens t < L - (seqlen_q - 1 - qi)

    @property
    def rows(self):
        """Query rows per sequence: seqlen_q * heads."""
        return self.seqlen_q * self.heads

    def visible(self, L, qi):
        """Cached tokens query token qi of a length-L sequence attends to."""
        return max(0, int(L) - (self.seqlen_q - 1 - qi)) if self.causal else int(L)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    @property
    def blocks_per_seq(self):
        return [(int(L) + self.page_size - 1) // self.page_size for L in self.seqlens]

    @property
    def max_blocks(self):
        return max(1, max(self.blocks_per_seq))

    @property
    def num_pages(self):
        return max(1, sum(self.blocks_per_seq))

    @property
    def total_tokens(self):
        return int(sum(int(L) for L in self.seqlens))

    def flops(self):
        """Algorithmic flops: 2*(576+512) per (query row, visible token), i.e.
        b*h*sum(L)*2*(576+512) for one query token per sequence."""
        pairs = sum(self.visible(L, qi) for L in self.seqlens for qi in range(self.seqlen_q))
        return float(self.heads) * pairs * 2 * (D + DV)

    def bytes(self):
        """Algorithmic bytes: KV rows (token granular) + Q + O."""
        esz = 2
        return float(self.total_tokens * D * esz + self.batch * self.rows * (D + DV) * esz)


def _varlen_lengths(batch, lo, hi, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(lo, hi + 1, size=batch)
    forced = [1, 2, 17, 63, 64, 65]  # one len-1 and a few short ones
    for k, v in enumerate(forced[: batch]):
        lens[k] = v
    return tuple(int(x) for x in lens)


# benchmark_mla.py's default cache lengths: 1024 to 32768
BENCH_SEQLENS = (1024, 2048, 4096, 8192, 16384, 32768)


def configs():
    """The decode workloads, by name (sizes as the pages' benchmarks use them)."""
    out = {
        "tiny": Workload("tiny", 2, 16, (256, 256), "fp16", page_size=256,
                         softmax_scale=576 ** -0.5, seed=0, shuffle=False,
                         notes="contiguous cache: page_size 256, block_table [[0],[1]]"),
        "paged": Workload("paged", 64, 128, (4096,) * 64, "bf16", page_size=64,
                          softmax_scale=192 ** -0.5, seed=1),
        "split": Workload("split", 128, 128, (8192,) * 128, "fp16", page_size=64,
                          softmax_scale=576 ** -0.5, seed=2),
        "varlen": Workload("varlen", 128, 128, _varlen_lengths(128, 1, 16384, 3), "bf16",
                           page_size=64, softmax_scale=192 ** -0.5, seed=3),
        "mqa": Workload("mqa", 256, 16, (32768,) * 256, "bf16", page_size=64,
                        softmax_scale=192 ** -0.5, seed=4, hot_row_frac=0.01,
                        hot_row_mult=8.0),
        # several query tokens per sequence (speculative / multi-token decoding): the
        # paged shape with two causal query tokens, 256 query rows per sequence
        "mtp": Workload("mtp", 64, 128, (4096,) * 64, "bf16", page_size=64,
                        softmax_scale=192 ** -0.5, seed=7, seqlen_q=2, causal=True),
        # the TileLang guide's own command lines (section 如何运行、验证与基准测试):
        # example_mla_decode.py defaults (contiguous cache, fp16 as in its comparison);
        # its example_mla_decode_paged.py line is the "split" workload above
        "tl_example": Workload("tl_example", 132, 128, (8192,) * 132, "fp16", page_size=8192,
                               softmax_scale=576 ** -0.5, seed=5, shuffle=False,
                               notes="contiguous cache: one 8192-token page per sequence"),
    }
    for k, L in enumerate(BENCH_SEQLENS):  # benchmark_mla.py default sweep, b=128 h=128
        name = f"tl_bench_{L}"
        out[name] = Workload(name, 128, 128, (L,) * 128, "fp16", page_size=64,
                             softmax_scale=576 ** -0.5, seed=10 + k)
    return out


def get(name, **overrides):
    w = configs()[name]
    return replace(w, **overrides) if overrides else w


def custom(batch, heads, seqlens, dtype="bf16", page_size=64, softmax_scale=192 ** -0.5,
           seed=0, shuffle=True, name="custom", **kw):
    if isinstance(seqlens, int):
        seqlens = (seqlens,) * batch
    return Workload(name, batch, heads, tuple(int(x) for x in seqlens), dtype, page_size,
                    softmax_scale, seed, shuffle, **kw)


def _randn_into(out, gen, scale_rows=None):
    """Fill `out` (any float dtype, contiguous) with N(0,1) drawn in fp32 chunks."""
    flat = out.view(-1)
    n = flat.numel()
    pos = 0
    while pos < n:
        m = min(_CHUNK, n - pos)
        x = torch.randn(m, generator=gen, device=out.device, dtype=torch.float32)
        flat[pos:pos + m] = x.to(out.dtype)
        pos += m


def make_inputs(w: Workload, device="cpu", poison_tail=False):
    """Build q, kv_cache, block_table, cache_seqlens for workload `w` on `device`.

    Layouts (contiguous):
      q            [b, seqlen_q, h, 576]
      kv_cache     [num_pages, page_size, 1, 576]
      block_table  int32 [b, max_blocks]
      cache_seqlens int32 [b]
    poison_tail fills cache rows past each sequence's length (inside its last
    page) with NaN, to prove they are never read into the result.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(w.seed))
    dt = w.torch_dtype
    b, h, P = w.batch, w.heads, w.page_size

    q = torch.empty((b, w.seqlen_q, h, D), dtype=dt, device=device)
    _randn_into(q, gen)

    kv = torch.empty((w.num_pages, P, 1, D), dtype=dt, device=device)
    if w.hot_row_frac > 0:
        # draw fp32 rows, scale the chosen ones, then round (chunked by pages)
        rows_per_chunk = max(1, _CHUNK // D)
        flat = kv.view(-1, D)
        nrows = flat.shape[0]
        pos = 0
        while pos < nrows:
            m = min(rows_per_chunk, nrows - pos)
            x = torch.randn((m, D), generator=gen, device=device, dtype=torch.float32)
            hot = torch.rand((m, 1), generator=gen, device=device) < w.hot_row_frac
            x = torch.where(hot, x * w.hot_row_mult, x)
            flat[pos:pos + m] = x.to(dt)
            pos += m
    else:
        _randn_into(kv, gen)

    # block table: seeded permutation of physical pages, or identity
    nb = w.blocks_per_seq
    cpu_gen = torch.Generator().manual_seed(int(w.seed) + 7919)
    if w.shuffle:
        perm = torch.randperm(w.num_pages, generator=cpu_gen).to(torch.int32)
    else:
        perm = torch.arange(w.num_pages, dtype=torch.int32)
    table = torch.full((b, w.max_blocks), -1, dtype=torch.int32)
    pos = 0
    for i in range(b):
        table[i, : nb[i]] = perm[pos: pos + nb[i]]
        pos += nb[i]
    seqlens = torch.tensor([int(L) for L in w.seqlens], dtype=torch.int32)

    if poison_tail:
        for i in range(b):
            L = int(w.seqlens[i])
            if L % P and nb[i] > 0:
                page = int(table[i, nb[i] - 1])
                kv[page, L % P:, :, :] = float("nan")

    return {
        "q": q,
        "kv_cache": kv,
        "block_table": table.to(device),
        "cache_seqlens": seqlens.to(device),
    }


def sample_seqs(w: Workload, n, seed=1234):
    """A seeded subset of sequence indices, always including the shortest and longest."""
    b = w.batch
    if n >= b:
        return list(range(b))
    lens = np.array([int(L) for L in w.seqlens])
    pick = {int(np.argmin(lens)), int(np.argmax(lens))}
    rng = np.random.Generator(np.random.PCG64(seed))
    for s in rng.permutation(b):
        if len(pick) >= n:
            break
        pick.add(int(s))
    return sorted(pick)


def to_bits(t):
    """Stored 16-bit patterns of a bf16/fp16 tensor as a numpy uint16 array (host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
