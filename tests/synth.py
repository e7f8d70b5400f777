"""Seeded synthetic inputs for the tests and the benchmark.

This module only draws inputs: fact lengths, fact extents, bf16 pre-RoPE K/V
rows, unit-norm float32 embeddings, queries, block tables and canary-filled
pools.  It holds none of the method's arithmetic (no scoring, selection,
placement, rotation or paging); both the CUDA path and the oracle read the
same bytes it produces.

Workload shapes follow the serving setting of "InferScale: GPU-Native KV
Injection for Personalized LLM Serving" (Llama-3-8B / Mistral-7B /
Llama-3-70B KV geometries, k = 5..50 retrieved facts of a dozen to a hundred
tokens, 16- or 32-token pages).  The paper measures on LoCoMo with real models;
these stores stand in for that data with the same shapes and are not derived
from it.

Small stores are drawn on the host with numpy's PCG64 and copied to the
device; large ones are drawn on the device with torch's seeded generator.
Where a store's logical size exceeds the device, facts get extents (start
row, length) in a shared physical arena: within a store every fact has its
own start row, so a wrong fact id reads different bytes, and each request
moves exactly the bytes a real store would.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

CANARY_BITS = 0xA5A5  # bf16 pattern written into every pool element beforehand


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    kv_heads: int
    head_dim: int
    rope_theta: float
    block_size: int
    n_facts: int            # per store
    len_lo: int
    len_hi: int
    len_dist: str           # "fixed", "uniform" or "loguniform" (inclusive integers)
    embed_dim: int
    requests: int
    k: int
    start: int | None       # None: one random base in [0, start_hi) per request
    start_hi: int
    seed: int
    store: str              # "dense" (CSR) or "arena"
    arena_gb: float = 0.0
    pool_blocks: int = 0    # 0: just enough for every request's worst case
    ks: tuple = ()

    @property
    def token_bytes(self) -> int:
        """K and V bytes of one token over all layers."""
        return 2 * self.layers * self.kv_heads * self.head_dim * 2


WORKLOADS = {
    "tiny": Workload("tiny", 2, 2, 64, 1e4, 16, 200, 16, 16, "fixed", 384, 1, 5, 0, 0, 0,
                     "dense", pool_blocks=32),
    "llama3_8b_10k": Workload("llama3_8b_10k", 32, 8, 128, 5e5, 16, 10_000, 12, 48, "uniform",
                              1024, 1, 50, 64, 0, 1, "dense", pool_blocks=1024,
                              ks=(5, 10, 20, 50)),
    "concurrent_64x5k": Workload("concurrent_64x5k", 32, 8, 128, 5e5, 16, 5_000, 12, 48,
                                 "uniform", 1024, 64, 50, 64, 0, 2, "arena", arena_gb=40.0,
                                 pool_blocks=12_000, ks=(5, 10, 20, 50)),
    "mistral_long_50k": Workload("mistral_long_50k", 32, 8, 128, 1e6, 32, 50_000, 8, 128,
                                 "loguniform", 1024, 1, 50, None, 32_768, 3, "arena",
                                 arena_gb=48.0, pool_blocks=1_300),
    "llama3_70b_capacity": Workload("llama3_70b_capacity", 80, 8, 128, 5e5, 16, 2_000, 12, 48,
                                    "uniform", 1024, 256, 50, 64, 0, 4, "arena", arena_gb=48.0,
                                    pool_blocks=28_610),
}


def fact_lengths(rng: np.random.Generator, w: Workload, n: int) -> np.ndarray:
    if w.len_dist == "fixed":
        return np.full(n, w.len_lo, np.int32)
    if w.len_dist == "uniform":
        return rng.integers(w.len_lo, w.len_hi + 1, size=n).astype(np.int32)
    if w.len_dist == "loguniform":
        u = rng.uniform(math.log(w.len_lo), math.log(w.len_hi), size=n)
        return np.clip(np.rint(np.exp(u)), w.len_lo, w.len_hi).astype(np.int32)
    raise ValueError(w.len_dist)


def unit_rows(rng: np.random.Generator, n: int, e: int) -> np.ndarray:
    """Gaussian rows normalised in float64, stored as float32."""
    x = rng.standard_normal((n, e))
    x /= np.linalg.norm(x, axis=1, keepdims=True)
    return x.astype(np.float32)


def clustered_rows(rng: np.random.Generator, n: int, e: int, clusters: int,
                   spread: float = 0.5) -> np.ndarray:
    """Unit rows around `clusters` random unit centres (centre + spread *
    Gaussian / sqrt(e), renormalised in float64): embeddings of related facts
    lie near each other, as text embeddings of one user's memories do."""
    centres = rng.standard_normal((clusters, e))
    centres /= np.linalg.norm(centres, axis=1, keepdims=True)
    which = rng.integers(0, clusters, n)
    x = centres[which] + spread * rng.standard_normal((n, e)) / np.sqrt(e)
    x /= np.linalg.norm(x, axis=1, keepdims=True)
    return x.astype(np.float32)


def near_queries(rng: np.random.Generator, emb: np.ndarray, n: int, noise: float = 0.5) -> np.ndarray:
    """Unit queries near random stored rows (row + noise * Gaussian / sqrt(e))."""
    e = emb.shape[1]
    picks = rng.integers(0, emb.shape[0], n)
    q = emb[picks].astype(np.float64) + noise * rng.standard_normal((n, e)) / np.sqrt(e)
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    return q.astype(np.float32)


def clustered_rows_device(seed: int, n: int, e: int, clusters: int, spread: float = 0.5,
                          chunk: int = 1 << 16):
    """clustered_rows drawn on the device (torch, float32), for stores too
    large to draw on the host; chunked so that the draw needs little scratch."""
    torch = _torch()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    centres = torch.randn((clusters, e), generator=gen, device="cuda")
    centres /= centres.norm(dim=1, keepdim=True)
    out = torch.empty((n, e), dtype=torch.float32, device="cuda")
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        which = torch.randint(0, clusters, (b - a,), generator=gen, device="cuda")
        x = centres[which] + (spread / e ** 0.5) * torch.randn((b - a, e), generator=gen, device="cuda")
        out[a:b] = x / x.norm(dim=1, keepdim=True)
    return out


def latent_rows_device(seed: int, n: int, e: int, latent: int = 32, noise: float = 0.1,
                       chunk: int = 1 << 16):
    """Unit rows of low intrinsic dimension, drawn on the device: a random
    e x latent projection of latent-dimensional Gaussian points, plus noise
    * Gaussian / sqrt(e), renormalised.  Neighbourhoods vary continuously
    (no isolated clusters), as for text embeddings."""
    torch = _torch()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    proj = torch.randn((latent, e), generator=gen, device="cuda") / latent ** 0.5
    out = torch.empty((n, e), dtype=torch.float32, device="cuda")
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        z = torch.randn((b - a, latent), generator=gen, device="cuda")
        x = z @ proj + (noise / e ** 0.5) * torch.randn((b - a, e), generator=gen, device="cuda")
        out[a:b] = x / x.norm(dim=1, keepdim=True)
    return out


def near_queries_device(seed: int, emb, n: int, noise: float = 0.5):
    """near_queries on the device: unit queries near random stored rows."""
    torch = _torch()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    e = emb.shape[1]
    picks = torch.randint(0, emb.shape[0], (n,), generator=gen, device="cuda")
    q = emb[picks] + (noise / e ** 0.5) * torch.randn((n, e), generator=gen, device="cuda")
    return (q / q.norm(dim=1, keepdim=True)).contiguous()


def graph_seeds(rng: np.random.Generator, n_facts: int, R: int, n_seeds: int) -> np.ndarray:
    """Seed fact ids for R graph searches, drawn uniformly (with repeats)."""
    return rng.integers(0, n_facts, (R, n_seeds)).astype(np.int32)


def bf16_normal_bits(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) float32 rounded to bf16 (round to nearest even), as uint16 bits."""
    x = rng.standard_normal(shape).astype(np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def csr_starts(lens: np.ndarray) -> np.ndarray:
    out = np.zeros(lens.shape[0], np.int64)
    if lens.shape[0] > 1:
        out[1:] = np.cumsum(lens[:-1], dtype=np.int64)
    return out


def arena_starts(rng: np.random.Generator, n: int, arena_tokens: int, max_len: int) -> np.ndarray:
    """Distinct start rows for n facts inside an arena (injective per store)."""
    span = arena_tokens - max_len
    assert span >= n, "arena too small for distinct fact starts"
    return rng.choice(span, size=n, replace=False).astype(np.int64)


def shuffled_blocks(rng: np.random.Generator, num_blocks: int) -> np.ndarray:
    return rng.permutation(num_blocks).astype(np.int32)


def query_rows(rng: np.random.Generator, n: int, e: int) -> np.ndarray:
    return unit_rows(rng, n, e)


def planted_query(rng: np.random.Generator, emb: np.ndarray, picks, noise: float = 0.05):
    """A query close to the sum of a few stored embeddings, unit norm."""
    q = emb[list(picks)].astype(np.float64).sum(axis=0)
    q += noise * rng.standard_normal(q.shape[0])
    q /= np.linalg.norm(q)
    return q.astype(np.float32)


# ----------------------------------------------------------- device builder

HOST_LIMIT_BYTES = 256 << 20  # above this, tensors are drawn on the device


@dataclasses.dataclass
class StoreData:
    emb: object            # torch float32 [N][E] (device)
    fact_start: object     # torch int64 [N] (device)
    fact_len: object       # torch int32 [N] (device)
    emb_np: np.ndarray
    start_np: np.ndarray
    len_np: np.ndarray


@dataclasses.dataclass
class Built:
    w: Workload
    k: int
    kv: object             # torch bf16 [L][2][T][H][D]: dense store or shared arena
    kv_np: np.ndarray | None  # uint16 bits of kv when small enough to keep on the host
    stores: list
    queries: object        # torch float32 [R][E]
    queries_np: np.ndarray
    start_pos: np.ndarray  # int32 [R]
    pool: object           # torch bf16 [L][2][NB][B][H][D], canary-filled
    block_tables: np.ndarray  # int32 [R][max_blocks] (-1 past each table's length)
    table_lens: np.ndarray    # int32 [R]

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_blocks(self) -> int:
        return int(self.pool.shape[2])


def _torch():
    import torch
    return torch


def fill_canary(pool) -> None:
    torch = _torch()
    pool.view(torch.int16).fill_(CANARY_BITS - (1 << 16))


def build_workload(w: Workload, k: int | None = None, tokens_needed=None,
                   device: str = "cuda", pool_blocks: int | None = None,
                   with_pool: bool = True) -> Built:
    """Materialise a workload on the device.

    tokens_needed[r], when given, sizes request r's block table to its
    injected tokens (known from a prior selection); otherwise every table has
    room for k facts of the longest length.  with_pool=False leaves the pool
    and block tables for attach_pool().
    """
    torch = _torch()
    k = w.k if k is None else k
    rng = np.random.default_rng(w.seed)
    tgen = torch.Generator(device=device)
    tgen.manual_seed(w.seed)
    L, H, D, E, N, R = w.layers, w.kv_heads, w.head_dim, w.embed_dim, w.n_facts, w.requests

    lens = [fact_lengths(rng, w, N) for _ in range(R)]
    if w.store == "dense":
        # every fact of every store has its own rows, stores back to back
        starts, base = [], 0
        for r in range(R):
            starts.append(csr_starts(lens[r]) + base)
            base += int(lens[r].sum())
        T = max(base, 1)
    else:
        T = int(w.arena_gb * 1e9 // w.token_bytes)
        starts = [arena_starts(rng, N, T, w.len_hi) for _ in range(R)]
    shape = (L, 2, T, H, D)
    kv_np = None
    if T * w.token_bytes <= HOST_LIMIT_BYTES:
        kv_np = bf16_normal_bits(rng, shape)
        kv = torch.from_numpy(kv_np.view(np.int16)).to(device).view(torch.bfloat16)
    else:
        kv = torch.randn(shape, generator=tgen, device=device, dtype=torch.bfloat16)

    stores = []
    for r in range(R):
        if N * E * 4 <= HOST_LIMIT_BYTES // 4:
            emb_np = unit_rows(rng, N, E)
            emb = torch.from_numpy(emb_np).to(device)
        else:
            x = torch.randn((N, E), generator=tgen, device=device, dtype=torch.float64)
            emb = (x / x.norm(dim=1, keepdim=True)).float()
            del x
            emb_np = emb.cpu().numpy()
        stores.append(StoreData(emb, torch.from_numpy(starts[r]).to(device),
                                torch.from_numpy(lens[r]).to(device), emb_np, starts[r], lens[r]))

    queries_np = query_rows(rng, R, E)
    queries = torch.from_numpy(queries_np).to(device)
    if w.start is None:
        start_pos = rng.integers(0, w.start_hi, size=R).astype(np.int32)
    else:
        start_pos = np.full(R, w.start, np.int32)
    built = Built(w, k, kv, kv_np, stores, queries, queries_np, start_pos, None,
                  np.zeros((R, 1), np.int32), np.zeros(R, np.int32))
    built._rng = rng
    if with_pool:
        attach_pool(built, tokens_needed, pool_blocks, device)
    return built


def attach_pool(built: Built, tokens_needed=None, pool_blocks: int | None = None,
                device: str = "cuda", rng: np.random.Generator | None = None) -> None:
    """Allocate the canary-filled paged pool and draw block tables from a
    shuffled free list (distinct blocks across requests)."""
    torch = _torch()
    w, k, R = built.w, built.k, built.w.requests
    rng = rng or built._rng
    B = w.block_size
    if tokens_needed is None:
        need = [int(built.start_pos[r]) + k * w.len_hi for r in range(R)]
    else:
        need = [int(built.start_pos[r]) + int(tokens_needed[r]) for r in range(R)]
    table_lens = np.array([max(1, (n + B - 1) // B) for n in need], np.int32)
    max_blocks = int(table_lens.max())
    nb = pool_blocks or w.pool_blocks or int(table_lens.sum())
    assert int(table_lens.sum()) <= nb, "pool too small for the block tables"
    free = shuffled_blocks(rng, nb)
    block_tables = np.full((R, max_blocks), -1, np.int32)
    at = 0
    for r in range(R):
        block_tables[r, :table_lens[r]] = free[at:at + table_lens[r]]
        at += int(table_lens[r])
    built.pool = None
    pool = torch.empty((w.layers, 2, nb, B, w.kv_heads, w.head_dim), device=device,
                       dtype=torch.bfloat16)
    fill_canary(pool)
    built.pool = pool
    built.block_tables = block_tables
    built.table_lens = table_lens
