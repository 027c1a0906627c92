"""Seeded synthetic inputs for paged KV-cache attention.

This module is shared by the oracle tests, the GPU tests and the bench, and it
holds none of the attention method's arithmetic: it only draws random numbers
(numpy's seeded PCG64 normals, SplitMix64 keys), converts them to the storage dtypes with torch's CPU
casts (bf16 bits, e4m3 bytes), builds seeded block tables (permutations) and
request lengths, and places per-token rows into a pool at the block/slot that a
block table names (fixture construction, not the attention gather).

Workload shapes follow the pages: head_dim 256, 4 KV heads, 16 (or 24) query
heads, block_size 880 (HyperQwen PR #109, "Cost" paragraph of the review:
chunk 2048, 24/4 heads, D=256, block 880), 2,048-token prefill chunks, and a
2,600-block pool whose top blocks 2,577-2,599 cross the int32 overflow of
block_id x 901,120 (HyperQwen PR #109, item 2 of the description).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)


def splitmix64(seed: int, n: int) -> np.ndarray:
    """n outputs of SplitMix64 (Steele, Lea & Flood, OOPSLA 2014) from `seed`."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + np.arange(1, n + 1, dtype=np.uint64) * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def uniform01(seed: int, n: int) -> np.ndarray:
    """Uniform doubles in (0, 1] with 53 random bits (SplitMix64)."""
    return ((splitmix64(seed, n) >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def normal(seed: int, n: int) -> np.ndarray:
    """n standard normal float32 values from numpy's seeded PCG64 generator."""
    return np.random.Generator(np.random.PCG64(seed & 0xFFFFFFFFFFFFFFFF)).standard_normal(n, dtype=np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float array -> uint16 bf16 bit patterns (torch's CPU cast, round-to-nearest-even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """float array -> OCP e4m3 byte codes (torch's CPU cast to float8_e4m3fn)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def bf16_normal(seed: int, shape, scale: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return to_bf16_bits(normal(seed, n) * scale).reshape(shape)


def permutation(seed: int, n: int) -> np.ndarray:
    """A seeded permutation of 0..n-1 (argsort of SplitMix64 keys)."""
    return np.argsort(splitmix64(seed, n), kind="stable").astype(np.int64)


def int8_codes(seed: int, shape) -> np.ndarray:
    """Random int8 codes in [-127, 127] with a triangular (sum of two uniforms) distribution, the
    centred value mix of a symmetric per-token-head int8 cache, drawn without running a quantizer."""
    n = int(np.prod(shape))
    g = np.random.Generator(np.random.PCG64(seed & 0xFFFFFFFFFFFFFFFF))
    u = np.frombuffer(g.bytes(2 * n), dtype=np.uint8)
    a = (u[:n] >> 1).astype(np.int16)
    a += u[n:] >> 1
    a -= 127
    return a.astype(np.int8).reshape(shape)


def positive_scales(seed: int, shape, lo: float = 0.02, hi: float = 0.03) -> np.ndarray:
    """Per-token-head fp32 scales drawn uniformly in [lo, hi)."""
    n = int(np.prod(shape))
    return (lo + (hi - lo) * uniform01(seed, n)).astype(np.float32).reshape(shape)


def lognormal_lengths(seed: int, n: int, median: float, sigma: float, lo: int, hi: int) -> np.ndarray:
    z = normal(seed, n).astype(np.float64)
    return np.clip(np.rint(median * np.exp(sigma * z)), lo, hi).astype(np.int64)


def place_tokens(pool: np.ndarray, table_row: np.ndarray, tokens: np.ndarray, block_size: int) -> None:
    """Write per-token rows tokens[pos] into pool[table_row[pos // bs], pos % bs] (fixture setup)."""
    n = tokens.shape[0]
    pos = np.arange(n, dtype=np.int64)
    blk = np.asarray(table_row, dtype=np.int64)[pos // block_size]
    pool[blk, pos % block_size] = tokens


@dataclass
class Request:
    """One request of a paged-attention problem: its token rows and its block table row."""
    seq_len: int
    q_len: int
    blocks: np.ndarray                # int64 block ids, ceil(seq_len / block_size) of them
    k_tok: np.ndarray | None = None   # [seq_len][Hkv][D] storage dtype (bf16 bits, e4m3 bytes, int8)
    v_tok: np.ndarray | None = None
    ks_tok: np.ndarray | None = None  # [seq_len][Hkv] fp32 (int8 caches only)
    vs_tok: np.ndarray | None = None


@dataclass
class Problem:
    """A batch over one paged pool. Pools are materialised by the caller (host or device)."""
    name: str
    num_blocks: int
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    softmax_scale: float
    kv_dtype: str                     # "bf16" | "e4m3" | "int8"
    requests: list = field(default_factory=list)
    q: np.ndarray | None = None       # bf16 bits [total_q][Hq][D]
    kv_scale: tuple = (1.0, 1.0)      # per-tensor scales (e4m3 caches)

    @property
    def num_reqs(self) -> int:
        return len(self.requests)

    @property
    def query_start_loc(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum([r.q_len for r in self.requests])]).astype(np.int32)

    @property
    def seq_lens(self) -> np.ndarray:
        return np.array([r.seq_len for r in self.requests], dtype=np.int32)

    @property
    def total_q(self) -> int:
        return int(sum(r.q_len for r in self.requests))

    @property
    def max_blocks(self) -> int:
        return max(len(r.blocks) for r in self.requests)

    def block_table(self, fill: int = -1) -> np.ndarray:
        """int32 [num_reqs][max_blocks]; unused entries hold `fill` (never dereferenced)."""
        bt = np.full((self.num_reqs, self.max_blocks), fill, dtype=np.int32)
        for i, r in enumerate(self.requests):
            bt[i, : len(r.blocks)] = r.blocks
        return bt

    @property
    def elems_per_block(self) -> int:
        return self.block_size * self.num_kv_heads * self.head_dim

    def pool_numpy(self, which: str, fill=0) -> np.ndarray:
        """Host pool [num_blocks][bs][Hkv][D] holding every request's rows.

        np.zeros maps lazily, so a 2,600-block pool costs only the touched blocks."""
        dt = {"bf16": np.uint16, "e4m3": np.uint8, "int8": np.int8}[self.kv_dtype]
        shape = (self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim)
        pool = np.zeros(shape, dtype=dt) if fill == 0 else np.full(shape, fill, dtype=dt)
        for r in self.requests:
            place_tokens(pool, r.blocks, r.k_tok if which == "k" else r.v_tok, self.block_size)
        return pool

    def scale_pool_numpy(self, which: str) -> np.ndarray:
        """Host per-token-head scale pool [num_blocks][bs][Hkv] fp32 (int8 caches)."""
        pool = np.zeros((self.num_blocks, self.block_size, self.num_kv_heads), dtype=np.float32)
        for r in self.requests:
            place_tokens(pool, r.blocks, r.ks_tok if which == "k" else r.vs_tok, self.block_size)
        return pool


def _kv_rows(seed: int, n_tok: int, hkv: int, d: int, kv_dtype: str, scale: float = 1.0):
    shape = (n_tok, hkv, d)
    if kv_dtype == "bf16":
        return bf16_normal(seed, shape, scale)
    if kv_dtype == "e4m3":
        return to_e4m3_bytes(normal(seed, int(np.prod(shape))) * scale).reshape(shape)
    if kv_dtype == "int8":
        return int8_codes(seed, shape)
    raise ValueError(kv_dtype)


def make_problem(name: str, *, seed: int, seq_lens, q_lens, num_blocks: int, block_size: int,
                 num_q_heads: int = 16, num_kv_heads: int = 4, head_dim: int = 256,
                 kv_dtype: str = "bf16", placement: str = "permuted", block_lists=None,
                 kv_value_scale: float = 1.0, kv_scale=(1.0, 1.0), softmax_scale: float | None = None,
                 with_kv: bool = True) -> Problem:
    """Build a seeded paged problem.

    placement: "permuted" (a seeded permutation of the pool, blocks distinct across
    requests), "cyclic" (requests walk one permutation cyclically, so blocks repeat
    once the pool is exhausted - prefix-cache-like sharing) or "explicit" (block_lists).
    """
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(head_dim)
    p = Problem(name, num_blocks, block_size, num_q_heads, num_kv_heads, head_dim, softmax_scale,
                kv_dtype, kv_scale=tuple(kv_scale))
    need = [(int(L) + block_size - 1) // block_size for L in seq_lens]
    if placement == "explicit":
        lists = [np.asarray(b, dtype=np.int64) for b in block_lists]
    else:
        perm = permutation(seed ^ 0x5EED, num_blocks)
        lists, off = [], 0
        for nb in need:
            if placement == "permuted":
                if off + nb > num_blocks:
                    raise ValueError("pool too small for distinct placement")
                lists.append(perm[off: off + nb])
            else:
                lists.append(perm[(off + np.arange(nb)) % num_blocks])
            off += nb
    for i, (L, ql) in enumerate(zip(seq_lens, q_lens)):
        r = Request(int(L), int(ql), lists[i])
        if with_kv:
            r.k_tok = _kv_rows(seed * 1000 + 2 * i + 1, int(L), num_kv_heads, head_dim, kv_dtype, kv_value_scale)
            r.v_tok = _kv_rows(seed * 1000 + 2 * i + 2, int(L), num_kv_heads, head_dim, kv_dtype, kv_value_scale)
            if kv_dtype == "int8":
                r.ks_tok = positive_scales(seed * 1000 + 2 * i + 101, (int(L), num_kv_heads))
                r.vs_tok = positive_scales(seed * 1000 + 2 * i + 102, (int(L), num_kv_heads))
        p.requests.append(r)
    p.q = bf16_normal(seed * 7 + 3, (p.total_q, num_q_heads, head_dim))
    return p


def new_rows(p: Problem, which: str) -> np.ndarray:
    """The chunk's new K or V rows in query order: each request's last q_len token rows,
    concatenated as [total_q][Hkv][D] (the input of a cache write)."""
    parts = [(r.k_tok if which == "k" else r.v_tok)[r.seq_len - r.q_len: r.seq_len] for r in p.requests]
    return np.ascontiguousarray(np.concatenate(parts, axis=0))


def slot_owner_pool(p: Problem) -> np.ndarray:
    """int64 [num_blocks][bs][Hkv]: for every pool slot, 1 + the index (token row, head) of
    new_rows() stored there, 0 where no new row lands (fixture bookkeeping for cache-write tests)."""
    pool = np.zeros((p.num_blocks, p.block_size, p.num_kv_heads), dtype=np.int64)
    base = 0
    for r in p.requests:
        ids = np.zeros((r.seq_len, p.num_kv_heads), dtype=np.int64)
        rows = np.arange(r.q_len, dtype=np.int64)[:, None] * p.num_kv_heads + np.arange(p.num_kv_heads)
        ids[r.seq_len - r.q_len:] = 1 + base * p.num_kv_heads + rows
        tmp = np.zeros_like(pool)
        place_tokens(tmp, r.blocks, ids, p.block_size)
        pool = np.where(tmp != 0, tmp, pool)
        base += r.q_len
    return pool


# ---------------------------------------------------------------------------------------------
# The five workloads (sizes from the pages; values seeded and synthetic)
# ---------------------------------------------------------------------------------------------

def tiny_bf16(seed: int = 1) -> Problem:
    """1 request, context 512, last 128-query causal chunk; 16/4 heads, D 256; bs 16; 64-block
    pool; the block table is a seeded permutation."""
    return make_problem("tiny_bf16", seed=seed, seq_lens=[512], q_lens=[128], num_blocks=64,
                        block_size=16, softmax_scale=1.0 / 16.0)


BIGPOOL_BLOCKS = 2600
BIGPOOL_BS = 880
BIGPOOL_L = 20000
BIGPOOL_CHUNK = 2048


def bigpool(seed: int = 2, top: bool = True, kv_dtype: str = "bf16", with_kv: bool = True,
            q_len: int = BIGPOOL_CHUNK) -> Problem:
    """One 20,000-token request on blocks 2577-2599 (top) or 0-22 (bottom) of a 2,600-block
    bf16 pool with block_size 880; the last 2,048-token chunk is the query. Same seed gives
    identical bytes at both placements (HyperQwen PR #109, item 2)."""
    nb = (BIGPOOL_L + BIGPOOL_BS - 1) // BIGPOOL_BS
    first = BIGPOOL_BLOCKS - nb if top else 0
    return make_problem("bigpool_top" if top else "bigpool_bottom", seed=seed, seq_lens=[BIGPOOL_L],
                        q_lens=[q_len], num_blocks=BIGPOOL_BLOCKS, block_size=BIGPOOL_BS,
                        kv_dtype=kv_dtype, placement="explicit",
                        block_lists=[np.arange(first, first + nb)], softmax_scale=1.0 / 16.0,
                        with_kv=with_kv)


def chunk_schedule(context: int, chunk: int = 2048):
    """(seq_len, q_len) of each prefill chunk of a `context`-token prompt."""
    out, done = [], 0
    while done < context:
        q = min(chunk, context - done)
        done += q
        out.append((done, q))
    return out


def verify_batch(seed: int = 5, num_reqs: int = 32, T: int = 8, pool_tokens: int = 480_000,
                 distinct: bool = True, block_size: int = 880, lengths=None, with_kv: bool = True) -> Problem:
    """Speculative-verify batch: cached prefixes lognormal (median 16k, sigma 0.8, clipped to
    4,096..81,920), T query tokens each, int8 per-token-head KV, bs 880. `distinct=False` keeps
    the literal 480k-token pool (ceil(480,000 / 880) = 546 blocks) and lets tables wrap (shared
    blocks)."""
    if lengths is None:
        lengths = lognormal_lengths(seed, num_reqs, 16384.0, 0.8, 4096, 81920)
    seq = [int(L) + T for L in lengths]
    need = sum((s + block_size - 1) // block_size for s in seq)
    if distinct:
        nb, placement = need, "permuted"
    else:
        nb, placement = -(-pool_tokens // block_size), "cyclic"  # the blocks holding pool_tokens
    return make_problem("verify", seed=seed, seq_lens=seq, q_lens=[T] * len(seq), num_blocks=nb,
                        block_size=block_size, kv_dtype="int8", placement=placement,
                        softmax_scale=1.0 / 16.0, with_kv=with_kv)
