"""Device-side fixtures for the GPU tests: pools, tables and scratch built from workloads.Problem.

Fixture construction only (torch indexing on the device); every step of the attention path runs in
libpkv's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

import workloads as W

DEV = "cuda"
BF16_NAN = 0x7FC0


def u16_to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def bf16_to_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _storage_dtype(kv_dtype):
    return {"bf16": torch.bfloat16, "e4m3": torch.uint8, "int8": torch.int8}[kv_dtype]


def device_pool(p: W.Problem, which: str, poison: bool = True) -> torch.Tensor:
    """[nb][bs][hkv][D] pool on the device. Unused slots are poisoned (bf16 NaN, e4m3 NaN code) so
    that any read outside the request's blocks shows up in the output."""
    shape = (p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim)
    dt = _storage_dtype(p.kv_dtype)
    if p.kv_dtype == "bf16":
        pool = torch.full(shape, float("nan") if poison else 0.0, dtype=dt, device=DEV)
    elif p.kv_dtype == "e4m3":
        pool = torch.full(shape, 0x7F if poison else 0, dtype=dt, device=DEV)
    else:
        pool = torch.full(shape, 127 if poison else 0, dtype=dt, device=DEV)
    for r in p.requests:
        tok = r.k_tok if which == "k" else r.v_tok
        pos = torch.arange(r.seq_len, device=DEV)
        blocks = torch.from_numpy(np.asarray(r.blocks, dtype=np.int64)).to(DEV)
        if p.kv_dtype == "bf16":
            src = u16_to_bf16(tok).to(DEV)
        else:
            src = torch.from_numpy(np.ascontiguousarray(tok)).to(DEV).view(dt)
        pool[blocks[pos // p.block_size], pos % p.block_size] = src
    return pool


def device_scale_pool(p: W.Problem, which: str) -> torch.Tensor:
    pool = torch.full((p.num_blocks, p.block_size, p.num_kv_heads), float("nan"), dtype=torch.float32, device=DEV)
    for r in p.requests:
        sc = r.ks_tok if which == "k" else r.vs_tok
        pos = torch.arange(r.seq_len, device=DEV)
        blocks = torch.from_numpy(np.asarray(r.blocks, dtype=np.int64)).to(DEV)
        pool[blocks[pos // p.block_size], pos % p.block_size] = torch.from_numpy(sc).to(DEV)
    return pool


def device_meta(p: W.Problem):
    """block_table (int32, unused entries = -1), seq_lens, query_start_loc on the device."""
    bt = torch.from_numpy(p.block_table(fill=-1)).to(DEV)
    sl = torch.from_numpy(p.seq_lens).to(DEV)
    qsl = torch.from_numpy(p.query_start_loc).to(DEV)
    return bt, sl, qsl


def device_q(p: W.Problem) -> torch.Tensor:
    return u16_to_bf16(p.q).to(DEV)


def dev_err() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    d = np.abs(a - b)
    assert not np.isnan(d).any(), "NaN in comparison"
    return float(d.max()) if d.size else 0.0
