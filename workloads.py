"""Seeded synthetic inputs for the paged decode path of looped transformers.

This module only *makes inputs*: request lengths, the physical page allocation
a scheduler would hand out, the layer structure of the model (which layers
loop), random bf16 Q/K/V values and the (seed, position) keys of new tokens.
None of the method's arithmetic lives here -- no slot addressing of the cached
tokens, no attention, no hashing, no inverse CDF -- so both the CUDA path and
the CPU oracle can take these arrays as plain inputs without sharing code.

The five workloads follow the shapes of the serving engine described in
"Faster fuzzy minds" (mini-sglang paged pool, recurrent depth as T*L banks)
and vllm-rlt PR #152 (Huginn 2 prelude + 4 recurrent + 2 coda layers, 32
loops, prompts up to 2000 tokens, 78% prefix-cache hit rate).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

WORKLOADS = ("tiny", "ouro", "huginn", "gqa", "longctx")


@dataclasses.dataclass
class NoiseSpec:
    """Keys of the latent-state noise draws: one row per token."""
    seeds: np.ndarray        # uint64 [rows]
    positions: np.ndarray    # int64  [rows]
    channels: int
    initializer_range: float

    @property
    def rows(self) -> int:
        return int(self.seeds.shape[0])


@dataclasses.dataclass
class PagedCase:
    """One decode batch over a paged KV pool with one bank per (layer, plane)."""
    name: str
    num_layers: int
    num_planes: int
    recurrent: np.ndarray    # uint8 [num_layers]: 1 if the layer is looped
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int           # physical pages per bank
    seq_lens: np.ndarray     # int32 [B], includes the token appended this step
    page_table: np.ndarray   # int32 [B][max_pages], -1 past a request's pages
    new_slots: np.ndarray    # int64 [B], slot the scheduler gave this step's token
    noise: NoiseSpec | None = None
    seed: int = 0

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.batch else 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def pages_of(self, b: int) -> int:
        return -(-int(self.seq_lens[b]) // self.page_size)

    def kv_tokens(self) -> int:
        """Cached tokens all requests read (logical: shared pages counted per request)."""
        return int(self.seq_lens.astype(np.int64).sum())

    def unique_pages(self) -> int:
        used = np.concatenate([self.page_table[b, : self.pages_of(b)] for b in range(self.batch)]) \
            if self.batch else np.zeros(0, np.int32)
        return int(np.unique(used).size)

    def unique_tokens(self) -> int:
        """Distinct physical token rows read (each shared page counted once)."""
        seen: dict[int, int] = {}
        for b in range(self.batch):
            n = self.pages_of(b)
            L = int(self.seq_lens[b])
            for i in range(n):
                used = min(self.page_size, L - i * self.page_size)
                p = int(self.page_table[b, i])
                seen[p] = max(seen.get(p, 0), used)
        return int(sum(seen.values()))


# --------------------------------------------------------------------------
# value generators
# --------------------------------------------------------------------------

def bf16_normal(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) samples rounded to bf16, returned as their uint16 bit patterns."""
    f = rng.standard_normal(size=shape, dtype=np.float32)
    return _round_bits(f)


def _round_bits(f: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even, in place on f's memory."""
    u = f.view(np.uint32)
    r = u >> 16
    r &= 1
    r += 0x7FFF
    u += r                                           # finite inputs: no carry out of bit 31
    u >>= 16
    return u.astype(np.uint16)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for building test cases)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def float_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest even), as bit patterns (for building test cases)."""
    return _round_bits(np.array(x, dtype=np.float32, copy=True, order="C"))


@dataclasses.dataclass
class HostTensors:
    """Host copies of one bank's pool plus this step's q / k_new / v_new (bf16 bits)."""
    k_pool: np.ndarray   # uint16 [num_pages][Hkv][ps][D]
    v_pool: np.ndarray
    q: np.ndarray        # uint16 [B][Hq][D]
    k_new: np.ndarray    # uint16 [B][Hkv][D]
    v_new: np.ndarray


def host_tensors(case: PagedCase, seed: int | None = None) -> HostTensors:
    """Random bf16 N(0,1) pool for ONE bank and this step's new q/k/v (numpy, seeded)."""
    rng = np.random.default_rng(case.seed + 1000 if seed is None else seed)
    pool_shape = (case.num_pages, case.num_kv_heads, case.page_size, case.head_dim)
    k_pool = bf16_normal(rng, pool_shape)
    v_pool = bf16_normal(rng, pool_shape)
    q = bf16_normal(rng, (case.batch, case.num_q_heads, case.head_dim))
    k_new = bf16_normal(rng, (case.batch, case.num_kv_heads, case.head_dim))
    v_new = bf16_normal(rng, (case.batch, case.num_kv_heads, case.head_dim))
    return HostTensors(k_pool, v_pool, q, k_new, v_new)


def device_pool(case: PagedCase, num_banks: int, device, seed: int | None = None):
    """Random bf16 N(0,1) K and V pools of ``num_banks`` banks, drawn on ``device``.

    For pools too large to draw on the host in seconds (tens to hundreds of GB).
    Uses torch's seeded generator; the values are plain inputs.
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(case.seed + 2000 if seed is None else seed)
    shape = (num_banks, case.num_pages, case.num_kv_heads, case.page_size, case.head_dim)
    k = torch.empty(shape, dtype=torch.bfloat16, device=device)
    v = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for t in (k, v):
        flat = t.view(num_banks, -1)
        for i in range(num_banks):          # bank by bank: no fp32 temporaries
            flat[i].normal_(generator=g)
    return k, v


# --------------------------------------------------------------------------
# page allocation (the scheduler's job, done once per workload)
# --------------------------------------------------------------------------

def _tables(seq_lens, page_size, num_pages, rng, shared_frac=0.0):
    """Allocate physical pages for every request.

    Private pages are drawn from a random permutation of the pool, so a
    request's pages are scattered.  With ``shared_frac`` > 0, one common prefix
    chain of floor(shared_frac * max_pages) pages is allocated first and
    request b maps its first floor(shared_frac * n_b) pages onto it, as a
    radix prefix cache would; the rest of its pages (always including the page
    holding its newest token) are private.
    """
    n = [-(-int(L) // page_size) for L in seq_lens]
    max_pages = max(n) if n else 0
    perm = rng.permutation(num_pages).astype(np.int32)
    cursor = 0
    chain = np.zeros(0, np.int32)
    if shared_frac > 0:
        c = int(math.floor(shared_frac * max_pages))
        chain = perm[:c]
        cursor = c
    table = np.full((len(seq_lens), max(max_pages, 1)), -1, np.int32)
    for b, nb in enumerate(n):
        s = int(math.floor(shared_frac * nb)) if shared_frac > 0 else 0
        table[b, :s] = chain[:s]
        table[b, s:nb] = perm[cursor: cursor + nb - s]
        cursor += nb - s
    assert cursor <= num_pages, "pool too small for the requested allocation"
    return table


def _new_slots(seq_lens, table, page_size):
    """Slot the scheduler hands this step's token: offset (L-1) % ps of its last page."""
    out = np.full(len(seq_lens), -1, np.int64)       # -1: empty request, no new token
    for b, L in enumerate(seq_lens):
        pos = int(L) - 1
        if pos < 0:
            continue
        out[b] = int(table[b, pos // page_size]) * page_size + pos % page_size
    return out


def _case(name, *, num_layers, num_planes, recurrent, B, Hq, Hkv, D, ps, seq_lens,
          pool_factor, rng, shared_frac=0.0, exact_pool=False, noise=None, seed=0):
    seq_lens = np.asarray(seq_lens, np.int32)
    live = sum(-(-int(L) // ps) for L in seq_lens)
    if shared_frac > 0:
        n = [-(-int(L) // ps) for L in seq_lens]
        c = int(math.floor(shared_frac * max(n)))
        live = c + sum(nb - int(math.floor(shared_frac * nb)) for nb in n)
    num_pages = live if exact_pool else int(math.ceil(pool_factor * live))
    table = _tables(seq_lens, ps, num_pages, rng, shared_frac)
    return PagedCase(name=name, num_layers=num_layers, num_planes=num_planes,
                     recurrent=np.asarray(recurrent, np.uint8), batch=B, num_q_heads=Hq,
                     num_kv_heads=Hkv, head_dim=D, page_size=ps, num_pages=num_pages,
                     seq_lens=seq_lens, page_table=table,
                     new_slots=_new_slots(seq_lens, table, ps), noise=noise, seed=seed)


def config(name: str, seed: int = 0) -> PagedCase:
    """The five synthetic workloads (shapes of the serving engine's decode step)."""
    rng = np.random.default_rng(seed)
    if name == "tiny":
        # 1 layer, 1 plane, B=4, L~U[17,300], ps=16, pool = exactly the live pages
        # in shuffled order, Hq=4, Hkv=2, D=64; noise 4 requests x 300 positions x 64
        # channels with seed = request index, initializer_range 0.02.
        L = rng.integers(17, 301, size=4)
        seeds = np.repeat(np.arange(4, dtype=np.uint64), 300)
        pos = np.tile(np.arange(300, dtype=np.int64), 4)
        return _case(name, num_layers=1, num_planes=1, recurrent=[0], B=4, Hq=4, Hkv=2,
                     D=64, ps=16, seq_lens=L, pool_factor=1.0, exact_pool=True, rng=rng,
                     noise=NoiseSpec(seeds, pos, 64, 0.02), seed=seed)
    if name == "ouro":
        # Ouro-shaped fixed-depth looped decode: 24 layers x 4 loop planes, all looped.
        L = rng.integers(512, 4097, size=64)
        return _case(name, num_layers=24, num_planes=4, recurrent=[1] * 24, B=64, Hq=16,
                     Hkv=16, D=128, ps=16, seq_lens=L, pool_factor=1.25, rng=rng, seed=seed)
    if name == "huginn":
        # Huginn-shaped: 2 prelude + 4 recurrent + 2 coda layers, 32 loops; B=16
        # sessions with prompts up to 2000 tokens (lengths ~ U[1024, 2000]); 78% of
        # pages on one shared prefix chain; new-token noise over 4096 channels.
        L = rng.integers(1024, 2001, size=16)
        seeds = rng.integers(0, 2**64, size=16, dtype=np.uint64)
        pos = (L - 1).astype(np.int64)
        return _case(name, num_layers=8, num_planes=32, recurrent=[0, 0, 1, 1, 1, 1, 0, 0],
                     B=16, Hq=32, Hkv=32, D=128, ps=16, seq_lens=L, pool_factor=1.25,
                     rng=rng, shared_frac=0.78, noise=NoiseSpec(seeds, pos, 4096, 0.02),
                     seed=seed)
    if name == "gqa":
        # Large-batch GQA: B=256, ln L ~ N(ln 2048, 1) clipped to [64, 16384].
        L = np.clip(np.rint(np.exp(rng.normal(math.log(2048.0), 1.0, size=256))), 64, 16384)
        return _case(name, num_layers=1, num_planes=1, recurrent=[0], B=256, Hq=32, Hkv=8,
                     D=128, ps=16, seq_lens=L.astype(np.int64), pool_factor=1.25, rng=rng,
                     seed=seed)
    if name == "longctx":
        # Long-context split-K stress: B=8, L~U[32768,131072], ps=64, 90% of each
        # request's pages on one shared chain; noise: 64 seeds x 64 positions x
        # 4096 channels = 2^24 draws, initializer_range 0.02.
        L = rng.integers(32768, 131073, size=8)
        seeds = np.repeat(rng.integers(0, 2**64, size=64, dtype=np.uint64), 64)
        pos = rng.integers(0, 131072, size=64 * 64).astype(np.int64)
        return _case(name, num_layers=1, num_planes=1, recurrent=[0], B=8, Hq=64, Hkv=8,
                     D=128, ps=64, seq_lens=L, pool_factor=1.0, rng=rng, shared_frac=0.9,
                     noise=NoiseSpec(seeds, pos, 4096, 0.02), seed=seed)
    raise ValueError(f"unknown workload {name!r}; expected one of {WORKLOADS}")


def custom(*, B, Hq, Hkv, D, ps, seq_lens, seed=0, pool_factor=1.25, shared_frac=0.0,
           name="custom") -> PagedCase:
    """A single-bank case with explicit lengths (edge cases, ragged tails, sweeps)."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, np.int64)
    return _case(name, num_layers=1, num_planes=1, recurrent=[0], B=B, Hq=Hq, Hkv=Hkv, D=D,
                 ps=ps, seq_lens=seq_lens, pool_factor=pool_factor, rng=rng,
                 shared_frac=shared_frac, seed=seed)


def noise_keys(rows: int, channels: int, seed: int = 0, initializer_range: float = 0.02,
               max_position: int = 1 << 20) -> NoiseSpec:
    """Random (seed, position) keys for ``rows`` tokens."""
    rng = np.random.default_rng(seed)
    seeds = rng.integers(0, 2**64, size=rows, dtype=np.uint64)
    pos = rng.integers(0, max_position, size=rows).astype(np.int64)
    return NoiseSpec(seeds, pos, channels, initializer_range)


def subcase(case: PagedCase, rows) -> PagedCase:
    """The requests ``rows`` of ``case`` alone, on a compact pool holding only their pages.

    Pages shared between the chosen requests stay shared.  Used to time or check
    the CPU oracle on a bounded sample of a large workload.
    """
    rows = np.asarray(rows, np.int64)
    pt = case.page_table[rows]
    sl = case.seq_lens[rows]
    used = np.unique(np.concatenate([pt[i, : -(-int(sl[i]) // case.page_size)] for i in range(len(rows))]))
    remap = {int(p): i for i, p in enumerate(used)}
    pt2 = np.full_like(pt, -1)
    for i in range(len(rows)):
        n = -(-int(sl[i]) // case.page_size)
        pt2[i, :n] = [remap[int(p)] for p in pt[i, :n]]
    return PagedCase(name=f"{case.name}[{len(rows)} rows]", num_layers=case.num_layers,
                     num_planes=case.num_planes, recurrent=case.recurrent, batch=len(rows),
                     num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads,
                     head_dim=case.head_dim, page_size=case.page_size, num_pages=int(used.size),
                     seq_lens=sl.copy(), page_table=pt2,
                     new_slots=_new_slots(sl, pt2, case.page_size), noise=None, seed=case.seed)
