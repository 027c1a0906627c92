"""GPU placement tests of the per-tensor fp8 e4m3 family in the pages' 2,600-block pool.

HyperQwen PR #109 (description, item 2): the same request at the top and at the bottom of a
2,600-block pool with block_size 880 must give identical bytes; past block id 2,383 the product
block_id x 901,120 no longer fits in 32 bits. At one byte per element an e4m3 pool reaches 2.34e9
bytes at its top block, so every fp8 call that forms a block offset is run with one request on
blocks 2,577-2,599 and again on blocks 0-22 with identical bytes, and must give bit-identical
results that also match the oracle:
  kv_fp8_dequant_dense      the dense bf16 scratch (bit-exact to the oracle as well);
  paged_prefill_attn_fp8    the last 2,048-token chunk of the 20,000-token request, both launches
                            (bit-identical to the dense-scratch path too);
  spec_verify_attn_partial_fp8 + combine   8 draft tokens after a 20,000-token prefix.
The cache write into an e4m3 pool at the same blocks is in test_gpu_write.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _parity import TOL_BF16, close, close_raw

pytestmark = pytest.mark.gpu

K_SCALE, V_SCALE = 0.5, 0.75
ROWS = sorted({0, 1, 127, 128, 2047} | set(range(1024, 1152)))  # a whole m-tile and tile edges


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_int64_gb300 as m
    return m


from _devsetup import bf16_to_u16, dev_err, device_meta, device_pool, device_q  # noqa: E402
from test_gpu_parity import oracle_rows  # noqa: E402


def _scales():
    return (torch.tensor([K_SCALE], dtype=torch.float32, device="cuda"),
            torch.tensor([V_SCALE], dtype=torch.float32, device="cuda"))


@pytest.fixture(scope="module")
def prefill_runs(pkv):
    """Dequantized scratch and prefill outputs of the 20,000-token e4m3 request at both placements."""
    res = {}
    for top in (True, False):
        p = W.bigpool(top=top, kv_dtype="e4m3")
        k, v = device_pool(p, "k"), device_pool(p, "v")
        bt, sl, qsl = device_meta(p)
        q = device_q(p)
        ks, vs = _scales()
        err = dev_err()
        L = int(p.seq_lens[0])
        kd = torch.full((1, L, 4, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
        vd = torch.full_like(kd, float("nan"))
        pkv.kv_fp8_dequant_dense(k, v, bt, sl, ks, vs, kd, vd, dev_err=err)
        ws = torch.empty(pkv.paged_prefill_workspace_bytes(), dtype=torch.uint8, device="cuda")
        outs = {}
        for name, w in (("fused", None), ("fused_persistent", ws)):
            out = torch.full_like(q, float("nan"))
            pkv.paged_prefill_attn_fp8(q, k, v, ks, vs, bt, sl, qsl, 2048, p.softmax_scale, out, dev_err=err,
                                       workspace=w)
            outs[name] = out
        ident = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
        for name, w in (("dense", None), ("dense_persistent", ws)):
            out = torch.full_like(q, float("nan"))
            pkv.paged_prefill_attn(q, kd, vd, ident, sl, qsl, 2048, p.softmax_scale, out, dev_err=err, workspace=w)
            outs[name] = out
        torch.cuda.synchronize()
        assert err.item() == 0, f"device status {err.item()}"
        res[top] = {"p": p, "kd": bf16_to_u16(kd), "vd": bf16_to_u16(vd)}
        res[top].update({n: bf16_to_u16(o) for n, o in outs.items()})
        del k, v, kd, vd, ws, outs
        torch.cuda.empty_cache()
    return res


def test_fp8_dequant_top_equals_bottom_and_oracle(prefill_runs):
    top, bot = prefill_runs[True], prefill_runs[False]
    assert top["p"].requests[0].blocks.min() == 2577 and bot["p"].requests[0].blocks.max() == 22
    assert np.array_equal(top["kd"], bot["kd"]) and np.array_equal(top["vd"], bot["vd"])
    p = top["p"]
    rk, rv = oracle.kv_fp8_dequant_dense(p.pool_numpy("k"), p.pool_numpy("v"), p.block_table(fill=0), p.seq_lens,
                                         int(p.seq_lens[0]), K_SCALE, V_SCALE)
    assert np.array_equal(top["kd"], rk) and np.array_equal(top["vd"], rv)


@pytest.mark.parametrize("name", ["fused", "fused_persistent", "dense", "dense_persistent"])
def test_fp8_prefill_top_equals_bottom(prefill_runs, name):
    top, bot = prefill_runs[True][name], prefill_runs[False][name]
    assert np.isfinite(W.bf16_bits_to_f32(top)).all()
    assert np.array_equal(top, bot)


def test_fp8_prefill_fused_equals_dense_and_oracle(prefill_runs):
    r = prefill_runs[True]
    # per-tile dequantization gives the scratch's values, so the same attention bit for bit, launch
    # for launch (the persistent launch cuts the same query tiles into the same key ranges)
    assert np.array_equal(r["fused"], r["dense"])
    assert np.array_equal(r["fused_persistent"], r["dense_persistent"])
    p = r["p"]
    L = int(p.seq_lens[0])
    kd = r["kd"].reshape(1, L, 4, 256)
    vd = r["vd"].reshape(1, L, 4, 256)
    ident = np.zeros((1, 1), np.int32)
    rows, ref = oracle_rows(lambda b, e: oracle.paged_prefill_attn(
        p.q, kd, vd, ident, p.seq_lens, p.query_start_loc, p.num_q_heads, p.softmax_scale, tok_begin=b, tok_end=e),
        ROWS)
    for name in ("fused", "fused_persistent"):
        close(r[name][rows], ref, TOL_BF16, name)


def test_fp8_verify_top_equals_bottom_and_oracle(pkv):
    T, L, split = 8, 20000, 2048
    nb = (L + T + 879) // 880
    res = {}
    for top in (True, False):
        first = 2600 - nb if top else 0
        p = W.make_problem("vf8big", seed=63, seq_lens=[L + T], q_lens=[T], num_blocks=2600, block_size=880,
                           kv_dtype="e4m3", placement="explicit", block_lists=[np.arange(first, first + nb)],
                           softmax_scale=1.0 / 16.0)
        k, v = device_pool(p, "k"), device_pool(p, "v")
        bt, sl, _ = device_meta(p)
        q = device_q(p)
        ks, vs = _scales()
        S = pkv.splits_needed(L + T, split)
        po = torch.full((S, T, 16, 256), float("nan"), dtype=torch.float32, device="cuda")
        pl = torch.full((S, T, 16), float("nan"), dtype=torch.float32, device="cuda")
        out = torch.full_like(q, float("nan"))
        err = dev_err()
        pkv.spec_verify_attn_partial_fp8(q, k, v, ks, vs, bt, sl, T, p.softmax_scale, split, po, pl, dev_err=err)
        pkv.spec_verify_combine(po, pl, sl, T, split, out)
        torch.cuda.synchronize()
        assert err.item() == 0
        res[top] = (p, po.cpu().numpy(), pl.cpu().numpy(), bf16_to_u16(out))
        del k, v
        torch.cuda.empty_cache()
    (p, po, pl, out), (_, po_b, pl_b, out_b) = res[True], res[False]
    assert np.array_equal(po.view(np.uint32), po_b.view(np.uint32))
    assert np.array_equal(pl.view(np.uint32), pl_b.view(np.uint32))
    assert np.array_equal(out, out_b)
    args = (p.q, p.pool_numpy("k"), p.pool_numpy("v"), K_SCALE, V_SCALE, p.block_table(fill=0), p.seq_lens)
    close(out, oracle.spec_verify_attn_fp8(*args, T, 16, p.softmax_scale), TOL_BF16)
    rpo, rpl = oracle.spec_verify_partial_fp8(*args, T, 16, p.softmax_scale, split, po.shape[0])
    close_raw(po, rpo, TOL_BF16, "partial O")
    close_raw(pl, rpl, 1e-3, "partial LSE")
