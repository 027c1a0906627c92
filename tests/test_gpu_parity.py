"""GPU parity: libpkv's kernels (through the C ABI) against the CPU oracle on the same seeded inputs.

Bars: bit-exact for the int8 codes / scales and the fp8 -> bf16 dense bytes, and for top-vs-bottom
pool placement; max-abs error <= 2e-3 (bf16 and fp8 paths, verify) and <= 5e-3 (int8-QK path)
against the oracle, after discounting only the rounding of the kernel's bf16 output (half a bf16
ulp of the value; see _parity.py). One bar per path, for every case: the five workloads of the pages
and the edge cases (ragged requests, first chunks whose rows see a handful of keys, other head
groups and block sizes).
"""
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _parity import TOL_BF16, TOL_INT8, close, close_raw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_int64_gb300 as m
    return m


from _devsetup import bf16_to_u16, dev_err, device_meta, device_pool, device_q, device_scale_pool  # noqa: E402


def _close(gpu_bf16_u16, ref, tol, what=""):
    return close(gpu_bf16_u16, ref, tol, what)


def oracle_rows(fn, rows, workers=None):
    """fn(begin, end) -> fp32 rows [begin, end) of an oracle output, evaluated over contiguous row
    ranges on a thread pool (the C oracle releases the GIL) and concatenated in order."""
    rows = sorted(set(int(r) for r in rows))
    ranges, b = [], None
    for r in rows:
        if b is None:
            b = e = r
        elif r == e + 1:
            e = r
        else:
            ranges.append((b, e + 1))
            b = e = r
    if b is not None:
        ranges.append((b, e + 1))
    pieces = []
    for b, e in ranges:  # ranges of at most 8 rows, so that the pool has work for every core
        pieces += [(x, min(x + 8, e)) for x in range(b, e, 8)]
    with ThreadPoolExecutor(workers or min(32, len(pieces))) as ex:
        outs = list(ex.map(lambda be: fn(*be), pieces))
    return rows, np.concatenate(outs, axis=0)


# ---------------------------------------------------------------------------------------------
# A1: int8 per-token-head quantization - bit exact
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("bs,seqs,begins", [(16, [300, 97, 1], [0, 13, 0]), (880, [2000, 881], [120, 0])])
def test_kv_int8_stats_quant_bit_exact(pkv, bs, seqs, begins):
    p = W.make_problem("q", seed=31, seq_lens=seqs, q_lens=[1] * len(seqs), num_blocks=64, block_size=bs)
    k = device_pool(p, "k")
    bt, sl, _ = device_meta(p)
    max_ctx = max(seqs) + 5
    pb = torch.tensor(begins, dtype=torch.int32, device="cuda")
    pe = torch.tensor(seqs, dtype=torch.int32, device="cuda")
    k8 = torch.zeros((p.num_reqs, max_ctx, 4, 256), dtype=torch.int8, device="cuda")
    ks = torch.zeros((p.num_reqs, max_ctx, 4), dtype=torch.float32, device="cuda")
    err = dev_err()
    pkv.kv_int8_stats_quant(k, bt, pb, pe, max(s - b for s, b in zip(seqs, begins)), k8, ks, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    rk8, rks = oracle.kv_int8_stats_quant(p.pool_numpy("k"), p.block_table(fill=0), begins, seqs, bs, max_ctx)
    assert np.array_equal(k8.cpu().numpy(), rk8)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), rks.view(np.uint32))


def test_kv_int8_stats_quant_tiny_rows_bit_exact(pkv):
    """Rows whose absmax is so small that 127 / absmax overflows to infinity (bf16 subnormals and
    normals below ~3.7e-37): every nonzero element's product is then infinite and the definition's
    clamp gives +-127; rows just above that bound, where the quotient stays finite; a normal row.
    (Zero elements in an overflowing row would multiply 0 by infinity, which the definition leaves
    undefined; these rows have none.)"""
    rng = np.random.default_rng(7)
    bs, H, D = 16, 4, 256
    rows = []
    sign = np.where(rng.random(D) < 0.5, -1.0, 1.0).astype(np.float32)
    rows.append(sign * rng.uniform(1e-38, 3e-37, D).astype(np.float32))            # normals, quotient overflows
    sub = rng.integers(1, 0x7f, D).astype(np.uint16) | np.where(sign < 0, 0x8000, 0).astype(np.uint16)
    rows.append(W.bf16_bits_to_f32(sub))                                              # bf16 subnormals
    mix = sign * np.float32(1e-40)
    mix[5] = np.float32(3e-37)
    rows.append(mix.astype(np.float32))                                               # one 3e-37, the rest subnormal
    rows.append(sign * rng.uniform(1e-37, 5e-37, D).astype(np.float32))              # absmax ~5e-37: finite quotient
    rows.append(rng.standard_normal(D).astype(np.float32))                            # ordinary
    n_tok = 2  # 2 tokens x 4 heads = 8 rows; the 5 special rows first, then ordinary ones
    while len(rows) < n_tok * H:
        rows.append(rng.standard_normal(D).astype(np.float32))
    vals = np.stack(rows)
    bits = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    pool = np.zeros((1, bs, H, D), dtype=np.uint16)
    pool[0, :n_tok] = bits.reshape(n_tok, H, D)
    k = torch.from_numpy(pool.view(np.int16)).view(torch.bfloat16).cuda()
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    pb = torch.zeros(1, dtype=torch.int32, device="cuda")
    pe = torch.full((1,), n_tok, dtype=torch.int32, device="cuda")
    k8 = torch.zeros((1, n_tok, H, D), dtype=torch.int8, device="cuda")
    ks = torch.zeros((1, n_tok, H), dtype=torch.float32, device="cuda")
    err = dev_err()
    pkv.kv_int8_stats_quant(k, bt, pb, pe, n_tok, k8, ks, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    rk8, rks = oracle.kv_int8_stats_quant(pool, np.zeros((1, 1), dtype=np.int32), [0], [n_tok], bs, n_tok)
    assert (np.abs(rk8[0, 0, :3]) == 127).all()  # the overflowing rows clamp
    assert np.array_equal(k8.cpu().numpy(), rk8)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), rks.view(np.uint32))


# ---------------------------------------------------------------------------------------------
# A4: fp8 -> dense bf16 - bit exact
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("bs,scale", [(16, 0.5), (880, 0.3)])
def test_kv_fp8_dequant_dense_bit_exact(pkv, bs, scale):
    p = W.make_problem("f", seed=41, seq_lens=[1500, 77], q_lens=[1, 1], num_blocks=120, block_size=bs,
                       kv_dtype="e4m3")
    k, v = device_pool(p, "k"), device_pool(p, "v")
    bt, sl, _ = device_meta(p)
    max_seq = 1600
    kd = torch.zeros((p.num_reqs, max_seq, 4, 256), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros_like(kd)
    ksc = torch.tensor([scale], dtype=torch.float32, device="cuda")
    vsc = torch.tensor([scale * 2], dtype=torch.float32, device="cuda")
    err = dev_err()
    pkv.kv_fp8_dequant_dense(k, v, bt, sl, ksc, vsc, kd, vd, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    rk, rv = oracle.kv_fp8_dequant_dense(p.pool_numpy("k"), p.pool_numpy("v"), p.block_table(fill=0), p.seq_lens,
                                         max_seq, scale, scale * 2)
    assert np.array_equal(bf16_to_u16(kd), rk)
    assert np.array_equal(bf16_to_u16(vd), rv)


# ---------------------------------------------------------------------------------------------
# A3: paged prefill attention
# ---------------------------------------------------------------------------------------------

def _run_prefill(pkv, p, mode=0, k_pool=None, v_pool=None, use_k16=False):
    k = device_pool(p, "k") if k_pool is None else k_pool
    v = device_pool(p, "v") if v_pool is None else v_pool
    bt, sl, qsl = device_meta(p)
    q = device_q(p)
    out = torch.full_like(q, float("nan"))
    err = dev_err()
    k8 = ks = None
    if mode == 1:
        max_ctx = int(p.seq_lens.max())
        k8 = torch.zeros((p.num_reqs, max_ctx, p.num_kv_heads, 256), dtype=torch.int8, device="cuda")
        ks = torch.zeros((p.num_reqs, max_ctx, p.num_kv_heads), dtype=torch.float32, device="cuda")
        pb = torch.zeros(p.num_reqs, dtype=torch.int32, device="cuda")
        k16 = torch.full((p.num_reqs, max_ctx, p.num_kv_heads, 256), float("nan"), dtype=torch.float16,
                         device="cuda") if use_k16 else None
        pkv.kv_int8_stats_quant(k, bt, pb, sl, max_ctx, k8, ks, dev_err=err, k16=k16)
        if use_k16:  # the fp16 copy holds exactly the int8 codes of the quantized positions; the
            # rest of the buffer is not written
            for r, L in enumerate(p.seq_lens.tolist()):
                assert torch.equal(k16[r, :L].float(), k8[r, :L].float())
                assert torch.isnan(k16[r, L:]).all()
    max_q = max(r.q_len for r in p.requests)
    pkv.paged_prefill_attn(q, None if mode == 1 else k, v, bt, sl, qsl, max_q, p.softmax_scale, out,
                           qk_mode=mode, k8=None if use_k16 else k8, k8_scale=ks, dev_err=err,
                           k16=k16 if mode == 1 and use_k16 else None)
    torch.cuda.synchronize()
    assert err.item() == 0, f"device status {err.item()}"
    return bf16_to_u16(out), (k8, ks)


def _oracle_prefill(p, mode=0, k8=None, ks=None, tok_begin=0, tok_end=None):
    kp, vp = p.pool_numpy("k"), p.pool_numpy("v")
    if mode == 1 and k8 is None:
        k8, ks = oracle.kv_int8_stats_quant(kp, p.block_table(fill=0), [0] * p.num_reqs, p.seq_lens, p.block_size,
                                            int(p.seq_lens.max()))
    return oracle.paged_prefill_attn(p.q, kp, vp, p.block_table(fill=0), p.seq_lens, p.query_start_loc,
                                     p.num_q_heads, p.softmax_scale, qk_mode=mode, k8=k8, k8_scale=ks,
                                     tok_begin=tok_begin, tok_end=tok_end)


def test_prefill_tiny_config_bf16(pkv):
    """1 request, context 512, last 128-query chunk, 16/4 heads, D 256, bs 16, permuted 64-block pool."""
    p = W.tiny_bf16()
    got, _ = _run_prefill(pkv, p)
    ref = _oracle_prefill(p)
    _close(got, ref, TOL_BF16)


@pytest.mark.parametrize("mode", [0, 1, 2])  # 2: int8 QK reading the fp16 copy of the codes
@pytest.mark.parametrize("case", ["ragged", "gqa6", "from_scratch", "bs880", "bs200"])
def test_prefill_ragged_cases(pkv, mode, case):
    if case == "ragged":     # several requests, q_len and seq_len off every tile boundary
        p = W.make_problem("r", seed=5, seq_lens=[700, 129, 300, 1], q_lens=[300, 129, 1, 1], num_blocks=80,
                           block_size=16)
    elif case == "gqa6":     # the pages' 24 query / 4 KV heads
        p = W.make_problem("g", seed=6, seq_lens=[517, 260], q_lens=[200, 133], num_blocks=64, block_size=16,
                           num_q_heads=24, num_kv_heads=4)
    elif case == "from_scratch":  # a first chunk: q_len == seq_len, queries from position 0
        p = W.make_problem("s", seed=7, seq_lens=[333], q_lens=[333], num_blocks=32, block_size=16)
    elif case == "bs880":    # block 880: key tiles follow the blocks (6 of 128 keys and one of 112)
        p = W.make_problem("b", seed=8, seq_lens=[2000, 1000], q_lens=[300, 1000], num_blocks=40, block_size=880)
    else:                    # block 200: tiles of 128 and 72 keys; the last tile of a request ragged too
        p = W.make_problem("c", seed=9, seq_lens=[1111, 333], q_lens=[400, 333], num_blocks=16, block_size=200)
    got, _ = _run_prefill(pkv, p, min(mode, 1), use_k16=mode == 2)
    ref = _oracle_prefill(p, min(mode, 1))
    _close(got, ref, TOL_INT8 if mode else TOL_BF16)


def test_prefill_block_size_dense_scratch(pkv):
    """block_size == max_seq with an identity table: the dense-scratch addressing of the fp8 path."""
    p = W.make_problem("d", seed=9, seq_lens=[3000, 2500], q_lens=[256, 700], num_blocks=2, block_size=4096,
                       placement="explicit", block_lists=[[0], [1]])
    got, _ = _run_prefill(pkv, p)
    _close(got, _oracle_prefill(p), TOL_BF16)


@pytest.fixture(scope="module")
def bigpool_gpu(pkv):
    """configs: 2,600-block bf16 pool (bs 880, 4.69 GB per K or V), 20,000-token request on blocks
    2577-2599 and on 0-22 with identical bytes; the last 2,048-token chunk."""
    out = {}
    for top in (True, False):
        p = W.bigpool(top=top)
        k, v = device_pool(p, "k"), device_pool(p, "v")
        for mode in (0, 1, 2):
            out[(top, mode)], _ = _run_prefill(pkv, p, min(mode, 1), k_pool=k, v_pool=v, use_k16=mode == 2)
        del k, v
        torch.cuda.empty_cache()
        out[("p", top)] = p
    return out


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_bigpool_top_equals_bottom_bit_exact(bigpool_gpu, mode):
    top, bot = bigpool_gpu[(True, mode)], bigpool_gpu[(False, mode)]
    assert np.isfinite(W.bf16_bits_to_f32(top)).all()
    assert np.array_equal(top, bot)


# rows of the big-pool chunk compared element by element: the chunk's first and last rows, both sides
# of m-tile boundaries, and one whole 128-row m-tile (rows 1,024-1,151: the middle of every tile row)
BIGPOOL_ROWS = sorted({0, 1, 127, 128, 2047} | set(range(1024, 1152)))


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_bigpool_rows_vs_oracle(bigpool_gpu, mode):
    p = bigpool_gpu[("p", True)]
    got = bigpool_gpu[(True, mode)]
    if mode == 2:  # the fp16 copy of the codes must give the very bytes of the converter path
        assert np.array_equal(got, bigpool_gpu[(True, 1)])
    kp, vp = p.pool_numpy("k"), p.pool_numpy("v")
    bt = p.block_table(fill=0)
    k8 = ks = None
    if mode:
        k8, ks = oracle.kv_int8_stats_quant(kp, bt, [0], p.seq_lens, p.block_size, int(p.seq_lens.max()))
    rows, ref = oracle_rows(lambda b, e: oracle.paged_prefill_attn(
        p.q, kp, vp, bt, p.seq_lens, p.query_start_loc, p.num_q_heads, p.softmax_scale, qk_mode=min(mode, 1), k8=k8,
        k8_scale=ks, tok_begin=b, tok_end=e), BIGPOOL_ROWS)
    _close(got[rows], ref, TOL_INT8 if mode else TOL_BF16)


@pytest.mark.parametrize("ctx", [24576, 47104])
def test_int8_prefill_chunked_context(pkv, ctx):
    """int8-QK prefill of a 24,576- and a 47,104-token context in 2,048-token chunks over a 2,600-block
    pool (bs 880, random table): every chunk quantizes its new K rows (A1) then attends (A3). The
    int8 codes and scales of the whole context are bit-exact; rows of the first, a middle and the
    last chunk (the last one's first m-tile whole) against the oracle."""
    bs = 880
    p = W.make_problem("i8", seed=33, seq_lens=[ctx], q_lens=[ctx], num_blocks=2600, block_size=bs)
    k, v = device_pool(p, "k"), device_pool(p, "v")
    bt, _, _ = device_meta(p)
    q_all = device_q(p)
    k8 = torch.zeros((1, ctx, 4, 256), dtype=torch.int8, device="cuda")
    ks = torch.zeros((1, ctx, 4), dtype=torch.float32, device="cuda")
    k16 = torch.zeros((1, ctx, 4, 256), dtype=torch.float16, device="cuda")
    err = dev_err()
    outs = {}
    sched = W.chunk_schedule(ctx)
    checked = (0, len(sched) // 2, len(sched) - 1)
    for ci, (L, ql) in enumerate(sched):
        sl = torch.tensor([L], dtype=torch.int32, device="cuda")
        pb = torch.tensor([L - ql], dtype=torch.int32, device="cuda")
        qsl = torch.tensor([0, ql], dtype=torch.int32, device="cuda")
        pkv.kv_int8_stats_quant(k, bt, pb, sl, ql, k8, ks, dev_err=err, k16=k16)
        q = q_all[L - ql:L].contiguous()
        out = torch.empty_like(q)
        pkv.paged_prefill_attn(q, None, v, bt, sl, qsl, ql, p.softmax_scale, out, qk_mode=1, k8_scale=ks,
                               dev_err=err, k16=k16)
        if ci in checked:
            outs[ci] = bf16_to_u16(out)
    torch.cuda.synchronize()
    assert err.item() == 0
    kp, vp = p.pool_numpy("k"), p.pool_numpy("v")
    rk8, rks = oracle.kv_int8_stats_quant(kp, p.block_table(fill=0), [0], [ctx], bs, ctx)
    assert np.array_equal(k8.cpu().numpy(), rk8)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), rks.view(np.uint32))
    for ci, got in outs.items():
        L, ql = sched[ci]
        sel = set(range(128)) | {777, ql - 1} if ci == checked[-1] else {0, 1, 777, ql - 1}
        rows, ref = oracle_rows(lambda b, e: oracle.paged_prefill_attn(
            p.q, kp, vp, p.block_table(fill=0), [L], [0, L], p.num_q_heads, p.softmax_scale, qk_mode=1, k8=rk8,
            k8_scale=rks, tok_begin=L - ql + b, tok_end=L - ql + e), sel)
        _close(got[rows], ref, TOL_INT8, f"chunk {ci}")


def test_fp8_prefill_through_dense_scratch(pkv):
    """fp8 e4m3 KV (values N(0,1) * 0.5 as e4m3 codes of N(0,1) with per-tensor scale 0.5), 32,768-token
    context; per 2,048-token chunk: dequantize [0, seq_len) to the dense bf16 scratch (identity table,
    block_size = max_seq), then bf16 attention on it. Checks the last chunk."""
    ctx = 32768
    p = W.make_problem("f8", seed=44, seq_lens=[ctx], q_lens=[2048], num_blocks=200, block_size=880,
                       kv_dtype="e4m3")
    k, v = device_pool(p, "k"), device_pool(p, "v")
    bt, sl, qsl = device_meta(p)
    scale = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    kd = torch.zeros((1, ctx, 4, 256), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros_like(kd)
    err = dev_err()
    pkv.kv_fp8_dequant_dense(k, v, bt, sl, scale, scale, kd, vd, dev_err=err)
    ident = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    q = device_q(p)
    out = torch.empty_like(q)
    pkv.paged_prefill_attn(q, kd, vd, ident, sl, qsl, 2048, p.softmax_scale, out, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    rk, rv = oracle.kv_fp8_dequant_dense(p.pool_numpy("k"), p.pool_numpy("v"), p.block_table(fill=0), [ctx], ctx,
                                         0.5, 0.5)
    assert np.array_equal(bf16_to_u16(kd), rk) and np.array_equal(bf16_to_u16(vd), rv)
    got = bf16_to_u16(out)
    worst = 0.0
    for t in (0, 1023, 2047):
        ref = oracle.paged_prefill_attn(p.q, rk.reshape(1, ctx, 4, 256), rv.reshape(1, ctx, 4, 256),
                                        np.zeros((1, 1), np.int32), [ctx], [0, 2048], 16, p.softmax_scale,
                                        tok_begin=t, tok_end=t + 1)
        worst = max(worst, _close(got[t:t + 1], ref, TOL_BF16))
    assert worst <= TOL_BF16


def _fp8_dense_then_prefill(pkv, p, k, v, scale):
    """The dequantize-once path: dense bf16 scratch (identity table, block_size = max_seq), then the
    bf16 prefill on it."""
    bt, sl, qsl = device_meta(p)
    max_seq = int(p.seq_lens.max())
    kd = torch.zeros((p.num_reqs, max_seq, p.num_kv_heads, 256), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros_like(kd)
    err = dev_err()
    pkv.kv_fp8_dequant_dense(k, v, bt, sl, scale, scale, kd, vd, dev_err=err)
    ident = torch.arange(p.num_reqs, dtype=torch.int32, device="cuda").reshape(p.num_reqs, 1)
    q = device_q(p)
    out = torch.empty_like(q)
    pkv.paged_prefill_attn(q, kd, vd, ident, sl, qsl, max(r.q_len for r in p.requests), p.softmax_scale, out,
                           dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return bf16_to_u16(out)


def _fp8_fused(pkv, p, k, v, scale, bt=None, expect_err=0):
    b, sl, qsl = device_meta(p)
    q = device_q(p)
    out = torch.full_like(q, float("nan"))
    err = dev_err()
    pkv.paged_prefill_attn_fp8(q, k, v, scale, scale, b if bt is None else bt, sl, qsl,
                               max(r.q_len for r in p.requests), p.softmax_scale, out, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == expect_err
    return bf16_to_u16(out)


@pytest.mark.parametrize("case", ["ctx32k_bs880", "ragged_bs16", "gqa6_bs80"])
def test_fp8_fused_prefill_equals_dense_path(pkv, case):
    """Per-tile dequantization inside the prefill against the dequantize-once dense scratch: both
    attend over the same bf16 values with the same kernel arithmetic, so the outputs are identical
    bit for bit; sampled rows are also checked against the oracle."""
    if case == "ctx32k_bs880":
        p = W.make_problem("f8f", seed=45, seq_lens=[32768], q_lens=[2048], num_blocks=200, block_size=880,
                           kv_dtype="e4m3")
    elif case == "ragged_bs16":
        p = W.make_problem("f8r", seed=46, seq_lens=[300, 1000, 129], q_lens=[300, 200, 1], num_blocks=120,
                           block_size=16, kv_dtype="e4m3")
    else:
        p = W.make_problem("f8g", seed=47, seq_lens=[704, 333], q_lens=[250, 333], num_blocks=40, block_size=80,
                           num_q_heads=24, num_kv_heads=4, kv_dtype="e4m3")
    k, v = device_pool(p, "k"), device_pool(p, "v")
    scale = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    dense = _fp8_dense_then_prefill(pkv, p, k, v, scale)
    fused = _fp8_fused(pkv, p, k, v, scale)
    assert np.array_equal(fused, dense)
    rk, rv = oracle.kv_fp8_dequant_dense(p.pool_numpy("k"), p.pool_numpy("v"), p.block_table(fill=0), p.seq_lens,
                                         int(p.seq_lens.max()), 0.5, 0.5)
    ident = np.arange(p.num_reqs, dtype=np.int32).reshape(p.num_reqs, 1)
    worst = 0.0
    for t in sorted({0, p.total_q // 2, p.total_q - 1}):
        ref = oracle.paged_prefill_attn(p.q, rk, rv, ident, p.seq_lens, p.query_start_loc, p.num_q_heads,
                                        p.softmax_scale, tok_begin=t, tok_end=t + 1)
        worst = max(worst, _close(fused[t:t + 1], ref, TOL_BF16))
    assert worst <= TOL_BF16


def test_fp8_fused_prefill_bad_block_reads_zero(pkv):
    p = W.make_problem("f8b", seed=48, seq_lens=[400], q_lens=[100], num_blocks=40, block_size=16, kv_dtype="e4m3")
    k, v = device_pool(p, "k"), device_pool(p, "v")
    scale = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    bt = p.block_table(fill=-1)
    bt[0, 3] = p.num_blocks + 7  # keys 48..63
    out = _fp8_fused(pkv, p, k, v, scale, bt=torch.from_numpy(bt).cuda(), expect_err=4)
    assert np.isfinite(W.bf16_bits_to_f32(out)).all()


# ---------------------------------------------------------------------------------------------
# A5 / A6: speculative verify
# ---------------------------------------------------------------------------------------------

def _run_verify(pkv, p, split, T=8, k_pool=None, v_pool=None):
    k = device_pool(p, "k") if k_pool is None else k_pool
    v = device_pool(p, "v") if v_pool is None else v_pool
    ksp, vsp = device_scale_pool(p, "k"), device_scale_pool(p, "v")
    bt, sl, _ = device_meta(p)
    q = device_q(p)
    S = pkv.splits_needed(int(p.seq_lens.max()), split)
    po = torch.full((S, q.shape[0], q.shape[1], 256), float("nan"), dtype=torch.float32, device="cuda")
    pl = torch.full((S, q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.full_like(q, float("nan"))
    err = dev_err()
    pkv.spec_verify_attn_partial(q, k, v, ksp, vsp, bt, sl, T, p.softmax_scale, split, po, pl, dev_err=err)
    pkv.spec_verify_combine(po, pl, sl, T, split, out)
    torch.cuda.synchronize()
    assert err.item() == 0, f"device status {err.item()}"
    return bf16_to_u16(out), po.cpu().numpy(), pl.cpu().numpy()


def _partials_close(po, pl, rpo, rpl, seq_lens, split, T, what=""):
    """Split partials against the oracle's: fp32 normalised outputs held to the bar raw (they carry
    no output rounding); natural-log LSEs within 1e-3, -inf exactly where the oracle has it."""
    for r, L in enumerate(seq_lens):
        ns = math.ceil(int(L) / split)
        rows = slice(r * T, (r + 1) * T)
        close_raw(po[:ns, rows], rpo[:ns, rows], TOL_BF16, what + " partial O")
        a, b = pl[:ns, rows], rpl[:ns, rows]
        assert np.array_equal(np.isneginf(a), np.isneginf(b))
        fin = np.isfinite(b)
        close_raw(a[fin], b[fin], 1e-3, what + " partial LSE")


def _verify_oracle_args(p):
    return (p.q, p.pool_numpy("k"), p.pool_numpy("v"), p.scale_pool_numpy("k"), p.scale_pool_numpy("v"),
            p.block_table(fill=0), p.seq_lens)


@pytest.mark.parametrize("split", [128, 512])
def test_verify_partials_and_combine(pkv, split):
    T = 8
    p = W.make_problem("v", seed=51, seq_lens=[L + T for L in (100, 1000, 4000, 129)], q_lens=[T] * 4,
                       num_blocks=80, block_size=80, kv_dtype="int8",
                       softmax_scale=1.0 / 16.0)
    got, po, pl = _run_verify(pkv, p, split, T)
    args = _verify_oracle_args(p)
    ref = oracle.spec_verify_attn(*args, T, p.num_q_heads, p.softmax_scale)
    _close(got, ref, TOL_BF16)
    S = po.shape[0]
    rpo, rpl = oracle.spec_verify_partial(*args, T, p.num_q_heads, p.softmax_scale, split, S)
    _partials_close(po, pl, rpo, rpl, p.seq_lens, split, T)


def test_verify_combine_more_than_32_splits(pkv):
    """A request cut into 40 splits (split 128): the combine's path for more splits than a warp has
    lanes (the LSEs reduced in strides of 32, then the partials merged one split at a time), next
    to a short request on the 32-or-fewer path."""
    T, split = 8, 128
    p = W.make_problem("vc", seed=61, seq_lens=[5000 + T, 300 + T], q_lens=[T] * 2, num_blocks=90,
                       block_size=64, kv_dtype="int8", softmax_scale=1.0 / 16.0)
    got, po, pl = _run_verify(pkv, p, split, T)
    assert po.shape[0] == 40
    args = _verify_oracle_args(p)
    ref = oracle.spec_verify_attn(*args, T, p.num_q_heads, p.softmax_scale)
    _close(got, ref, TOL_BF16)
    rpo, rpl = oracle.spec_verify_partial(*args, T, p.num_q_heads, p.softmax_scale, split, po.shape[0])
    _partials_close(po, pl, rpo, rpl, p.seq_lens, split, T)


@pytest.mark.parametrize("T,hq,hkv", [(1, 16, 4), (4, 24, 4), (5, 16, 4), (2, 32, 4), (8, 24, 4), (11, 16, 4)])
def test_verify_other_query_geometries(pkv, T, hq, hkv):
    """T * group other than 32 query columns: a T = 1 decode step; the pages' 24/4 heads with T = 4
    (24 columns, padded) and T = 8 (48 columns: the 48-column CTA shape); odd T; T = 11 with 4 heads
    (44 columns, 48-column shape, padded); 32/4 heads with T = 2. Padding columns must not leak into
    live ones, and only live rows are written."""
    p = W.make_problem("vq", seed=53 + T, seq_lens=[L + T for L in (700, 64, 2100)], q_lens=[T] * 3,
                       num_blocks=60, block_size=64, num_q_heads=hq, num_kv_heads=hkv, kv_dtype="int8",
                       softmax_scale=1.0 / 16.0)
    split = 256
    got, po, pl = _run_verify(pkv, p, split, T)
    args = _verify_oracle_args(p)
    ref = oracle.spec_verify_attn(*args, T, p.num_q_heads, p.softmax_scale)
    _close(got, ref, TOL_BF16)
    rpo, rpl = oracle.spec_verify_partial(*args, T, p.num_q_heads, p.softmax_scale, split, po.shape[0])
    _partials_close(po, pl, rpo, rpl, p.seq_lens, split, T)


@pytest.mark.parametrize("n_req", [7, 130])
def test_verify_launch_order_covers_every_split(pkv, n_req):
    """Batches of up to 128 requests run longest first (whole splits, then the requests' shorter
    last splits by length), larger ones in request order: every live (request, split) partial must
    match the oracle's wherever it falls in the order (the partials start as NaN). The lengths
    include exact multiples of the split (no shorter last split), equal last-split lengths, requests
    shorter than one split and the longest request last."""
    T, split = 8, 256
    if n_req == 7:
        lens = [512, 300, 300, 768, 40, 1000, 2048]
    else:
        rng = np.random.default_rng(59)
        lens = [int(x) for x in rng.integers(T, 420, size=n_req)]
        lens[3], lens[50], lens[129] = 256, 512, 700
    p = W.make_problem("vo", seed=59 + n_req, seq_lens=lens, q_lens=[T] * n_req,
                       num_blocks=sum((L + 63) // 64 for L in lens) + 4, block_size=64, kv_dtype="int8",
                       softmax_scale=1.0 / 16.0)
    got, po, pl = _run_verify(pkv, p, split, T)
    args = _verify_oracle_args(p)
    ref = oracle.spec_verify_attn(*args, T, p.num_q_heads, p.softmax_scale)
    _close(got, ref, TOL_BF16)
    rpo, rpl = oracle.spec_verify_partial(*args, T, p.num_q_heads, p.softmax_scale, split, po.shape[0])
    _partials_close(po, pl, rpo, rpl, p.seq_lens, split, T)


def test_verify_bigpool_top_equals_bottom(pkv):
    """int8 per-token-head cache, 2,600-block pool (bs 880), request of L = 20,000 + 8 tokens on the top
    blocks and on the bottom blocks with identical bytes: bit-identical outputs, and the oracle."""
    T = 8
    outs = {}
    for top in (True, False):
        nb = (20000 + T + 879) // 880
        first = 2600 - nb if top else 0
        p = W.make_problem("vb", seed=61, seq_lens=[20000 + T], q_lens=[T], num_blocks=2600, block_size=880,
                           kv_dtype="int8", placement="explicit", block_lists=[np.arange(first, first + nb)],
                           softmax_scale=1.0 / 16.0)
        outs[top], _, _ = _run_verify(pkv, p, 2048, T)
    assert np.array_equal(outs[True], outs[False])
    ref = oracle.spec_verify_attn(*_verify_oracle_args(p), T, p.num_q_heads, p.softmax_scale)
    _close(outs[True], ref, TOL_BF16)


def _verify_all_requests(p, T):
    """The oracle's verify output of every request, one request per worker thread."""
    args = _verify_oracle_args(p)
    with ThreadPoolExecutor(min(32, p.num_reqs)) as ex:
        parts = list(ex.map(lambda r: oracle.spec_verify_attn(*args, T, p.num_q_heads, p.softmax_scale, req_begin=r,
                                                              req_end=r + 1)[r * T:(r + 1) * T], range(p.num_reqs)))
    return np.concatenate(parts, axis=0)


@pytest.mark.parametrize("pool,split", [("distinct", 4096), ("literal", 2048), ("distinct", "planned")])
def test_verify_batch_config(pkv, pool, split):
    """32 requests, lognormal prefixes 4k-80k (median 16k), T = 8, int8 KV, bs 880; every request against
    the oracle. "distinct": a pool of just the blocks the batch needs; "literal": the pages'
    480k-token pool (546 blocks), which cannot hold the batch's ~670 blocks, so the tables walk one
    permutation cyclically and requests share blocks. "planned": the split the library's planner
    picks for the batch (the bench's launch; a large split, 6 or fewer per request)."""
    T = 8
    p = W.verify_batch(distinct=pool == "distinct")
    if split == "planned":
        split = pkv.spec_verify_pick_split(p.seq_lens, T, 16, 4, torch.cuda.get_device_properties(0).multi_processor_count)
        assert split % 512 == 0 and split >= 1024
    if pool == "literal":
        assert p.num_blocks == 546 and sum(len(r.blocks) for r in p.requests) > p.num_blocks
    got, _, _ = _run_verify(pkv, p, split, T)
    _close(got, _verify_all_requests(p, T), TOL_BF16)


# ---------------------------------------------------------------------------------------------
# boundary behaviour
# ---------------------------------------------------------------------------------------------

def test_empty_batch_is_a_no_op(pkv):
    q = torch.zeros((0, 16, 256), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((4, 16, 4, 256), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_prefill_attn(q, k, k, torch.zeros((1, 1), dtype=torch.int32, device="cuda"), z, torch.zeros(2, dtype=torch.int32, device="cuda"),
                           0, 0.0625, q)
    del bt


def test_unsupported_head_dim_is_rejected(pkv):
    q = torch.zeros((4, 16, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((4, 16, 4, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    one = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_prefill_attn(q, k, k, bt, one, torch.tensor([0, 1], dtype=torch.int32, device="cuda"), 1, 0.1, q)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED


def test_out_of_range_block_id_is_reported_not_read(pkv):
    p = W.make_problem("bad", seed=71, seq_lens=[200], q_lens=[50], num_blocks=16, block_size=16)
    k, v = device_pool(p, "k"), device_pool(p, "v")
    bt, sl, qsl = device_meta(p)
    bt[0, 3] = 16  # == num_blocks: one past the pool
    q = device_q(p)
    out = torch.empty_like(q)
    err = dev_err()
    pkv.paged_prefill_attn(q, k, v, bt, sl, qsl, 50, p.softmax_scale, out, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == pkv.PKV_ERR_DEVICE_BOUNDS
    assert np.isfinite(W.bf16_bits_to_f32(bf16_to_u16(out))).all()


# ---------------------------------------------------------------------------------------------
# verify over a per-tensor fp8 e4m3 cache
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("split,bs,hq", [(128, 16, 16), (2048, 880, 16), (256, 64, 24)])
def test_verify_fp8_partials_and_combine(pkv, split, bs, hq):
    """e4m3 cache with per-tensor scales; hq = 24 (8 tokens x 6 heads = 48 query columns) runs the
    48-column CTA shape."""
    T = 8
    p = W.make_problem("vf8", seed=81, seq_lens=[L + T for L in (100, 3000, 6000, 129)], q_lens=[T] * 4,
                       num_blocks=max(64, 4 * (6008 // bs + 2)), block_size=bs, kv_dtype="e4m3",
                       num_q_heads=hq, num_kv_heads=4, softmax_scale=1.0 / 16.0)
    k, v = device_pool(p, "k"), device_pool(p, "v")
    bt, sl, _ = device_meta(p)
    q = device_q(p)
    kd = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    vd = torch.tensor([0.75], dtype=torch.float32, device="cuda")
    S = pkv.splits_needed(int(p.seq_lens.max()), split)
    po = torch.full((S, q.shape[0], hq, 256), float("nan"), dtype=torch.float32, device="cuda")
    pl = torch.full((S, q.shape[0], hq), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    err = dev_err()
    pkv.spec_verify_attn_partial_fp8(q, k, v, kd, vd, bt, sl, T, p.softmax_scale, split, po, pl, dev_err=err)
    pkv.spec_verify_combine(po, pl, sl, T, split, out)
    torch.cuda.synchronize()
    assert err.item() == 0
    args = (p.q, p.pool_numpy("k"), p.pool_numpy("v"), 0.5, 0.75, p.block_table(fill=0), p.seq_lens)
    ref = oracle.spec_verify_attn_fp8(*args, T, hq, p.softmax_scale)
    _close(bf16_to_u16(out), ref, TOL_BF16)
    rpo, rpl = oracle.spec_verify_partial_fp8(*args, T, hq, p.softmax_scale, split, S)
    _partials_close(po.cpu().numpy(), pl.cpu().numpy(), rpo, rpl, p.seq_lens, split, T)
