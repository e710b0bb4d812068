"""Seeded synthetic MLA-decode workloads (shared by the tests, the smoke check and the bench).

This module only draws inputs: it holds none of the method's arithmetic.  Both
the CUDA path and the CPU oracle consume exactly the tensors built here (the
oracle gets host copies of the same stored values: 16-bit patterns, or e4m3
bytes and their two scales).

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
  * e4m3 workloads (an FP8 cache with one dequantisation scale per tensor): q and
    the cache are drawn the same way in fp32, then quantised per tensor with
    scale = amax / 448 (448 is e4m3's largest finite value) as
    stored = e4m3(x / scale), rounded to nearest even; the draws are made twice
    from the same generator state (amax first, then the quantisation).
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
    dtype: str              # "bf16" | "fp16" | "e4m3"
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
        return {"bf16": torch.bfloat16, "fp16": torch.float16,
                "e4m3": torch.float8_e4m3fn}[self.dtype]

    @property
    def elem_bytes(self):
        """Bytes per stored q / cache element."""
        return 1 if self.dtype == "e4m3" else 2

    @property
    def out_dtype(self):
        """Format of the output: the input's, bf16 for an e4m3 cache."""
        return "bf16" if self.dtype == "e4m3" else self.dtype

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
        """Algorithmic bytes: KV rows (token granular) + Q + O (O is 16-bit)."""
        esz = self.elem_bytes
        return float(self.total_tokens * D * esz + self.batch * self.rows * (D * esz + DV * 2))


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
        # the far corner of the paged bf16 target range (batch 64-128 x 4-8K cache):
        # the paged shape at twice the batch and twice the cache
        "paged_8k": Workload("paged_8k", 128, 128, (8192,) * 128, "bf16", page_size=64,
                             softmax_scale=192 ** -0.5, seed=22),
        "varlen": Workload("varlen", 128, 128, _varlen_lengths(128, 1, 16384, 3), "bf16",
                           page_size=64, softmax_scale=192 ** -0.5, seed=3),
        "mqa": Workload("mqa", 256, 16, (32768,) * 256, "bf16", page_size=64,
                        softmax_scale=192 ** -0.5, seed=4, hot_row_frac=0.01,
                        hot_row_mult=8.0),
        # several query tokens per sequence (speculative / multi-token decoding): the
        # paged shape with two causal query tokens, 256 query rows per sequence
        "mtp": Workload("mtp", 64, 128, (4096,) * 64, "bf16", page_size=64,
                        softmax_scale=192 ** -0.5, seed=7, seqlen_q=2, causal=True),
        # the paged shape with an FP8 cache: q and the cache in e4m3 with one
        # dequantisation scale per tensor, bf16 out
        "paged_fp8": Workload("paged_fp8", 64, 128, (4096,) * 64, "e4m3", page_size=64,
                              softmax_scale=192 ** -0.5, seed=21),
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


E4M3_MAX = 448.0


def _fp32_rows(n_rows, gen, device, hot_frac=0.0, hot_mult=1.0):
    """The fp32 draws of `n_rows` rows of 576, chunk by chunk (the same sequence of
    generator calls as the 16-bit paths make)."""
    if hot_frac > 0:
        rows_per_chunk = max(1, _CHUNK // D)
        pos = 0
        while pos < n_rows:
            m = min(rows_per_chunk, n_rows - pos)
            x = torch.randn((m, D), generator=gen, device=device, dtype=torch.float32)
            hot = torch.rand((m, 1), generator=gen, device=device) < hot_frac
            yield torch.where(hot, x * hot_mult, x).view(-1)
            pos += m
    else:
        n = n_rows * D
        pos = 0
        while pos < n:
            m = min(_CHUNK, n - pos)
            yield torch.randn(m, generator=gen, device=device, dtype=torch.float32)
            pos += m


def _round_into(out, gen, **draw):
    """Fill the 16-bit tensor `out` (rows of 576) with the draws rounded to its dtype."""
    flat = out.view(-1)
    pos = 0
    for x in _fp32_rows(out.numel() // D, gen, out.device, **draw):
        flat[pos:pos + x.numel()] = x.to(out.dtype)
        pos += x.numel()


def _quantize_e4m3(out, gen, **draw):
    """Fill the e4m3 tensor `out` (rows of 576) with per-tensor quantised draws;
    returns the dequantisation scale (amax / 448, as an fp32 value)."""
    state = gen.get_state()
    n_rows = out.numel() // D
    amax = 0.0
    for x in _fp32_rows(n_rows, gen, out.device, **draw):
        amax = max(amax, float(x.abs().max()))
    scale = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
    gen.set_state(state)
    flat = out.view(-1)
    pos = 0
    for x in _fp32_rows(n_rows, gen, out.device, **draw):
        flat[pos:pos + x.numel()] = (x / scale).clamp_(-E4M3_MAX, E4M3_MAX).to(out.dtype)
        pos += x.numel()
    return scale


def make_inputs(w: Workload, device="cpu", poison_tail=False):
    """Build q, kv_cache, block_table, cache_seqlens for workload `w` on `device`.

    Layouts (contiguous):
      q            [b, seqlen_q, h, 576]
      kv_cache     [num_pages, page_size, 1, 576]
      block_table  int32 [b, max_blocks]
      cache_seqlens int32 [b]
    poison_tail fills cache rows past each sequence's length (inside its last
    page) with NaN, to prove they are never read into the result.
    e4m3 workloads add "q_scale" and "kv_scale" (floats).
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(w.seed))
    dt = w.torch_dtype
    b, h, P = w.batch, w.heads, w.page_size

    q = torch.empty((b, w.seqlen_q, h, D), dtype=dt, device=device)
    kv = torch.empty((w.num_pages, P, 1, D), dtype=dt, device=device)
    hot = dict(hot_frac=w.hot_row_frac, hot_mult=w.hot_row_mult)
    scales = {}
    if w.dtype == "e4m3":
        scales["q_scale"] = _quantize_e4m3(q, gen)
        scales["kv_scale"] = _quantize_e4m3(kv, gen, **hot)
    else:
        _round_into(q, gen)
        _round_into(kv, gen, **hot)

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
        **scales,
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
    """Stored bit patterns as a host numpy array: uint16 for bf16 / fp16, uint8 for
    e4m3."""
    if t.dtype == torch.float8_e4m3fn:
        return t.detach().contiguous().view(torch.uint8).cpu().numpy()
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
