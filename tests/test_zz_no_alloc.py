"""The allocation-free verify entry point, for callers that cannot allocate device memory (a plugin
whose host process owns the device allocator, a path that must not allocate between steps): it
keeps the split partials in a fixed scratch array inside libpkv.so. Its output must match the
regular workspace path (partials + combine) through the same C ABI, on two calls in a row (the
second call reuses the array the first one filled).

Collected last (file name) so that a run stopping at the first failure has run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_int64_gb300 as m
    return m


def _p(t):
    return C.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_path_twice(pkv):
    """Two calls in a row, the second with fewer splits than the first, so the array still holds the
    first call's partials past the second's: the outputs equal the workspace path's bit for bit (the
    same kernels in the same order on the same inputs), which also shows that no stale partial is
    read."""
    from _devsetup import bf16_to_u16, device_meta, device_pool, device_q, device_scale_pool
    T, split = 8, 1024
    outs, splits = [], []
    for seed, prefixes in ((91, (5000, 900, 12000, 33)), (92, (3000, 900, 2000, 33))):
        p = W.make_problem("noalloc", seed=seed, seq_lens=[L + T for L in prefixes],
                           q_lens=[T] * 4, num_blocks=40, block_size=880, kv_dtype="int8",
                           softmax_scale=1.0 / 16.0)
        k, v = device_pool(p, "k"), device_pool(p, "v")
        ks, vs = device_scale_pool(p, "k"), device_scale_pool(p, "v")
        bt, sl, _ = device_meta(p)
        q = device_q(p)
        S = pkv.splits_needed(int(p.seq_lens.max()), split)
        splits.append(S)
        need = p.num_reqs * T * 16 * S * (256 + 1) * 4
        assert need <= pkv.lib.pkv_spec_verify_noalloc_capacity_bytes()
        # regular path with a caller workspace
        po = torch.empty((S, q.shape[0], 16, 256), dtype=torch.float32, device="cuda")
        pl = torch.empty((S, q.shape[0], 16), dtype=torch.float32, device="cuda")
        ref = torch.empty_like(q)
        pkv.spec_verify_attn_partial(q, k, v, ks, vs, bt, sl, T, p.softmax_scale, split, po, pl)
        pkv.spec_verify_combine(po, pl, sl, T, split, ref)
        # allocation-free path, straight through the C ABI
        out = torch.full_like(q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = pkv.lib.pkv_spec_verify_attn_noalloc(
            _p(q), _p(k), _p(v), _p(ks), _p(vs), k.shape[0], k.stride(0), k.stride(1), k.stride(2),
            ks.stride(0), ks.stride(1), _p(bt), bt.stride(0), bt.shape[1], _p(sl), p.num_reqs, T, 16, 4, 256,
            880, p.softmax_scale, split, S, _p(out), _p(err), stream)
        assert rc == 0, pkv.lib.pkv_last_error()
        torch.cuda.synchronize()
        assert err.item() == 0
        a, b = bf16_to_u16(out), bf16_to_u16(ref)
        assert np.isfinite(W.bf16_bits_to_f32(a)).all()
        assert np.array_equal(a, b)
        outs.append(a)
    assert splits[1] < splits[0]
    assert not np.array_equal(outs[0], outs[1])


def test_noalloc_rejects_oversized_partials(pkv):
    cap = pkv.lib.pkv_spec_verify_noalloc_capacity_bytes()
    # 64 requests x 8 tokens x 16 heads x 64 splits x 257 floats is far beyond the array
    z = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = pkv.lib.pkv_spec_verify_attn_noalloc(
        _p(z), _p(z), _p(z), _p(z), _p(z), 4, 901120, 1024, 256, 3520, 4, _p(z), 1, 1, _p(z), 64, 8, 16, 4, 256,
        880, 0.0625, 128, 64, _p(z), None, None)
    assert rc == pkv.PKV_ERR_INVALID_ARG
    msg = pkv.lib.pkv_last_error().decode()
    assert str(cap) in msg and "scratch" in msg
