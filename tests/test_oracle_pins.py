"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each pin is chosen so that a plausible mistake in the oracle (a dropped term, a wrong sign or
index, a transposed operand, a wrong rounding) fails at least one of them:
  - e4m3 decoding: the OCP E4M3 table (golden fixture) and torch's float8_e4m3fn cast, all 256 codes;
  - bf16 rounding: torch's float32 -> bfloat16 cast (ties included);
  - quantizer: a hand-worked example, the error bound |x - q*s| <= s/2, the absmax code +-127,
    odd symmetry, power-of-two scale equivariance, the zero row;
  - fp8 dense dequant: torch's decode and casts on the un-paged token rows;
  - paged attention: a dense non-paged brute force, closed forms (V = 1 -> 1; all K = 0 -> mean of
    visible V; position 0 -> V[0]; two keys -> logistic weights), causal and GQA invariances,
    the int8-QK mode equal to exact QK when quantization is lossless, top-vs-bottom placement in
    a 2,600-block pool, and a planted 32-bit block offset that the placement test must catch;
  - verify: the same values through the int8 verify path and the bf16 prefill path, and
    split-KV + combine equal to the unsplit result for several split sizes.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from conftest import read_golden_kv

# --------------------------------------------------------------------------------------------
# scalar formats
# --------------------------------------------------------------------------------------------


def test_e4m3_golden_table(golden_dir):
    with open(os.path.join(golden_dir, "e4m3_ocp_values.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 10
    for code, val in rows:
        got = oracle.e4m3_to_f32(int(code, 16))
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([oracle.e4m3_to_f32(int(c)) for c in codes], dtype=np.float32)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok].view(np.uint32), got[ok].view(np.uint32))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(20000).astype(np.float32)
    # exact ties: low 16 bits == 0x8000, both parities of the kept bit
    ties = ((rng.integers(0, 2**7, 2000).astype(np.uint32) << np.uint32(16)) | np.uint32(0x8000)
            | np.uint32(0x3F800000)).view(np.float32)
    x = np.concatenate([x, ties, np.array([0.0, -0.0, 1e-40, -3.4e38], dtype=np.float32)])
    ref = W.to_bf16_bits(x)
    got = np.array([oracle.f32_to_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(ref, got)


# --------------------------------------------------------------------------------------------
# quantizer
# --------------------------------------------------------------------------------------------


def test_quant_worked_example(golden_dir):
    g = read_golden_kv(os.path.join(golden_dir, "quant_worked_example.txt"))
    vals = np.zeros(256, dtype=np.float32)
    v = np.array([float(x) for x in g["values"]], dtype=np.float32)
    vals[: v.size] = v
    codes, scale = oracle.quant_row(W.to_bf16_bits(vals))
    assert list(codes[: v.size]) == [int(c) for c in g["codes"]]
    assert np.all(codes[v.size:] == 0)
    assert np.float32(scale).view(np.uint32) == int(g["scale_f32_hex"][0], 16)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_quant_properties(seed):
    x = W.bf16_normal(seed, (64, 256), scale=float(2.0 ** (seed - 2)))
    xf = W.bf16_bits_to_f32(x)
    for row, rowf in zip(x, xf):
        codes, s = oracle.quant_row(row)
        amax = np.abs(rowf).max()
        # scale and bound
        assert np.float32(s) == np.float32(amax) / np.float32(127.0)
        err = np.abs(rowf.astype(np.float64) - codes.astype(np.float64) * s)
        assert err.max() <= s * 0.5 * (1 + 1e-5) + 1e-30
        # the absmax element maps to +-127, codes within [-127, 127]
        i = int(np.argmax(np.abs(rowf)))
        assert abs(int(codes[i])) == 127 and np.sign(codes[i]) == np.sign(rowf[i])
        assert codes.min() >= -127
        # odd symmetry
        neg, s2 = oracle.quant_row(row ^ np.uint16(0x8000))
        assert s2 == s and np.array_equal(neg, -codes)
        # power-of-two equivariance: x * 4 has the same codes and 4x the scale
        up, s4 = oracle.quant_row(W.to_bf16_bits(rowf * 4.0))
        assert np.array_equal(up, codes) and s4 == np.float32(4.0) * np.float32(s)


def test_quant_zero_row():
    codes, s = oracle.quant_row(np.zeros(256, dtype=np.uint16))
    assert s == 0.0 and not codes.any()


def test_int8_stats_quant_gathers_each_token_row():
    p = W.make_problem("q", seed=11, seq_lens=[300, 97], q_lens=[1, 1], num_blocks=40, block_size=16)
    pool = p.pool_numpy("k")
    bt = p.block_table()
    pb, pe = np.array([0, 13], np.int32), np.array([300, 97], np.int32)
    k8, ks = oracle.kv_int8_stats_quant(pool, bt, pb, pe, 16, max_ctx=300)
    for r, req in enumerate(p.requests):
        for pos in range(pb[r], pe[r]):
            for h in range(p.num_kv_heads):
                c, s = oracle.quant_row(req.k_tok[pos, h])
                assert np.array_equal(k8[r, pos, h], c) and ks[r, pos, h] == np.float32(s)
        # positions outside [pos_begin, pos_end) are untouched
        assert not k8[r, : pb[r]].any() and not k8[r, pe[r]:].any()


# --------------------------------------------------------------------------------------------
# fp8 dense dequant
# --------------------------------------------------------------------------------------------


@pytest.mark.parametrize("scale", [0.5, 0.3])
def test_fp8_dense_dequant_matches_torch_decode(scale):
    p = W.make_problem("f", seed=21, seq_lens=[200, 64], q_lens=[1, 1], num_blocks=30, block_size=16,
                       kv_dtype="e4m3", kv_value_scale=1.0)
    kp, vp = p.pool_numpy("k"), p.pool_numpy("v")
    kd, vd = oracle.kv_fp8_dequant_dense(kp, vp, p.block_table(), p.seq_lens, 256, scale, scale * 2)
    for r, req in enumerate(p.requests):
        for which, dense, tok, sc in (("k", kd, req.k_tok, scale), ("v", vd, req.v_tok, scale * 2)):
            f = torch.from_numpy(tok).view(torch.float8_e4m3fn).to(torch.float32)
            ref = (f * torch.tensor(sc, dtype=torch.float32)).to(torch.bfloat16).view(torch.int16).numpy()
            assert np.array_equal(dense[r, : req.seq_len].view(np.int16), ref), which
            assert not dense[r, req.seq_len:].any()


# --------------------------------------------------------------------------------------------
# paged prefill attention
# --------------------------------------------------------------------------------------------


def _tiny(seed=3, seq_lens=(70, 45), q_lens=(20, 45), bs=16, hq=8, hkv=2, d=32, nb=32):
    return W.make_problem("t", seed=seed, seq_lens=list(seq_lens), q_lens=list(q_lens), num_blocks=nb,
                          block_size=bs, num_q_heads=hq, num_kv_heads=hkv, head_dim=d)


def _run_paged(p, kp=None, vp=None, **kw):
    kp = p.pool_numpy("k") if kp is None else kp
    vp = p.pool_numpy("v") if vp is None else vp
    return oracle.paged_prefill_attn(p.q, kp, vp, p.block_table(), p.seq_lens, p.query_start_loc,
                                     p.num_q_heads, p.softmax_scale, **kw)


def test_paged_equals_dense_brute_force():
    p = _tiny()
    out = _run_paged(p)
    qsl = p.query_start_loc
    for r, req in enumerate(p.requests):
        qpos = np.arange(req.seq_len - req.q_len, req.seq_len, dtype=np.int64)
        ref = oracle.dense_attn(p.q[qsl[r]: qsl[r + 1]], req.k_tok, req.v_tok, qpos, p.num_q_heads,
                                p.softmax_scale)
        np.testing.assert_allclose(out[qsl[r]: qsl[r + 1]], ref, atol=1e-6, rtol=0)


def test_values_all_one_give_one():
    p = _tiny()
    one = W.to_bf16_bits(np.ones(1, np.float32))[0]
    for r in p.requests:
        r.v_tok[:] = one
    out = _run_paged(p)
    assert np.array_equal(out, np.ones_like(out))


def test_zero_keys_give_mean_of_visible_values():
    p = _tiny()
    for r in p.requests:
        r.k_tok[:] = 0
    out = _run_paged(p)
    qsl, g = p.query_start_loc, p.num_q_heads // p.num_kv_heads
    for r, req in enumerate(p.requests):
        vf = W.bf16_bits_to_f32(req.v_tok).astype(np.float64)
        csum = np.cumsum(vf, axis=0)
        for i in range(req.q_len):
            pos = req.seq_len - req.q_len + i
            for h in range(p.num_q_heads):
                np.testing.assert_allclose(out[qsl[r] + i, h], csum[pos, h // g] / (pos + 1), atol=2e-6)


def test_position_zero_returns_first_value():
    p = _tiny(seq_lens=(33,), q_lens=(33,))
    out = _run_paged(p)
    g = p.num_q_heads // p.num_kv_heads
    v0 = W.bf16_bits_to_f32(p.requests[0].v_tok[0])
    for h in range(p.num_q_heads):
        assert np.array_equal(out[0, h], v0[h // g])


def test_two_keys_logistic_weights():
    d = 32
    p = _tiny(seq_lens=(2,), q_lens=(1,), hq=1, hkv=1, d=d)
    req = p.requests[0]
    q = np.zeros((1, 1, d), np.float32); q[0, 0, 0] = 1.5
    k = np.zeros((2, 1, d), np.float32); k[1, 0, 0] = 2.0
    p.q = W.to_bf16_bits(q); req.k_tok = W.to_bf16_bits(k)
    out = _run_paged(p)[0, 0]
    s1 = p.softmax_scale * 1.5 * 2.0
    w1 = 1.0 / (1.0 + math.exp(-s1))
    vf = W.bf16_bits_to_f32(req.v_tok[:, 0]).astype(np.float64)
    np.testing.assert_allclose(out, (1 - w1) * vf[0] + w1 * vf[1], atol=1e-6)


def test_causal_future_keys_do_not_matter():
    p = _tiny(seq_lens=(90,), q_lens=(40,))
    base = _run_paged(p)
    req = p.requests[0]
    cut = req.seq_len - req.q_len + 10           # queries 0..10 of the chunk see keys <= cut
    req.k_tok[cut + 1:] = W.bf16_normal(99, req.k_tok[cut + 1:].shape, 3.0)
    req.v_tok[cut + 1:] = W.bf16_normal(98, req.v_tok[cut + 1:].shape, 3.0)
    pert = _run_paged(p)
    assert np.array_equal(base[:11], pert[:11])
    assert not np.array_equal(base[11:], pert[11:])


def test_gqa_equals_replicated_kv_heads():
    p = _tiny(hq=8, hkv=2)
    out = _run_paged(p)
    g = p.num_q_heads // p.num_kv_heads
    rep = W.make_problem("rep", seed=3, seq_lens=[70, 45], q_lens=[20, 45], num_blocks=32, block_size=16,
                         num_q_heads=8, num_kv_heads=8, head_dim=32)
    for r_src, r_rep in zip(p.requests, rep.requests):
        r_rep.blocks = r_src.blocks
        r_rep.k_tok = np.repeat(r_src.k_tok, g, axis=1)
        r_rep.v_tok = np.repeat(r_src.v_tok, g, axis=1)
    rep.q = p.q
    assert np.array_equal(out, _run_paged(rep))


def test_int8_qk_equals_exact_qk_when_lossless():
    # entries are integers * 2^-6 with absmax 127 * 2^-6 in every row: scale 2^-6, codes exact
    p = _tiny(seq_lens=(60,), q_lens=(25,))
    req = p.requests[0]

    def lossless(seed, shape):
        z = np.clip(np.rint(W.normal(seed, int(np.prod(shape))) * 40), -126, 126).reshape(shape)
        z[..., 0] = 127
        return W.to_bf16_bits(z * 2.0 ** -6)

    p.q = lossless(5, p.q.shape)
    req.k_tok = lossless(6, req.k_tok.shape)
    kp = p.pool_numpy("k")
    k8, ks = oracle.kv_int8_stats_quant(kp, p.block_table(), [0], [req.seq_len], p.block_size, req.seq_len)
    assert np.all(ks == np.float32(2.0 ** -6))
    exact = _run_paged(p, kp=kp)
    i8 = _run_paged(p, kp=kp, qk_mode=1, k8=k8, k8_scale=ks)
    np.testing.assert_allclose(i8, exact, atol=1e-6, rtol=0)


def test_int8_qk_close_to_exact_qk():
    p = _tiny(seq_lens=(60,), q_lens=(25,))
    req = p.requests[0]
    kp = p.pool_numpy("k")
    k8, ks = oracle.kv_int8_stats_quant(kp, p.block_table(), [0], [req.seq_len], p.block_size, req.seq_len)
    exact = _run_paged(p, kp=kp)
    i8 = _run_paged(p, kp=kp, qk_mode=1, k8=k8, k8_scale=ks)
    err = np.abs(i8 - exact).max()
    assert 0 < err < 0.02


def test_int8_dot_equals_int64_brute_force():
    # the int8-QK score is scale * qs * ks * dot; recover dot from a one-key problem
    d = 256
    p = _tiny(seq_lens=(1,), q_lens=(1,), hq=1, hkv=1, d=d)
    req = p.requests[0]
    kp = p.pool_numpy("k")
    k8, ks = oracle.kv_int8_stats_quant(kp, p.block_table(), [0], [1], p.block_size, 1)
    q8, qs = oracle.quant_row(p.q[0, 0])
    dot64 = int(np.dot(q8.astype(np.int64), k8[0, 0, 0].astype(np.int64)))
    assert abs(dot64) <= 127 * 127 * d < 2 ** 24
    # with a single key the output is V[0] whatever the score; use two keys, K[1] = 0 (score 0)
    p2 = _tiny(seq_lens=(2,), q_lens=(1,), hq=1, hkv=1, d=d)
    r2 = p2.requests[0]
    r2.k_tok[0] = req.k_tok[0]; r2.k_tok[1] = 0; p2.q = p.q
    kp2 = p2.pool_numpy("k")
    k8b, ksb = oracle.kv_int8_stats_quant(kp2, p2.block_table(), [0], [2], p2.block_size, 2)
    out = oracle.paged_prefill_attn(p2.q, kp2, p2.pool_numpy("v"), p2.block_table(), p2.seq_lens,
                                    p2.query_start_loc, 1, p2.softmax_scale, qk_mode=1, k8=k8b,
                                    k8_scale=ksb)[0, 0].astype(np.float64)
    s0 = p2.softmax_scale * qs * float(ksb[0, 0, 0]) * dot64
    w0 = 1.0 / (1.0 + math.exp(-s0))
    vf = W.bf16_bits_to_f32(r2.v_tok[:, 0]).astype(np.float64)
    np.testing.assert_allclose(out, w0 * vf[0] + (1 - w0) * vf[1], atol=2e-6)


# --------------------------------------------------------------------------------------------
# big pool: placement invariance and the planted 32-bit offset
# --------------------------------------------------------------------------------------------


def test_bigpool_geometry_matches_pages(golden_dir):
    g = {k: int(v[0]) for k, v in read_golden_kv(os.path.join(golden_dir, "int32_overflow_threshold.txt")).items()}
    p = W.bigpool(top=True, with_kv=False)
    assert p.elems_per_block == g["block_stride_elems"] == g["block_size"] * g["num_kv_heads"] * g["head_dim"]
    assert p.num_blocks == g["pool_blocks"]
    blocks = p.requests[0].blocks
    assert (blocks[0], blocks[-1]) == (g["top_first_block"], g["top_last_block"])
    b = W.bigpool(top=False, with_kv=False).requests[0].blocks
    assert (b[0], b[-1]) == (g["bottom_first_block"], g["bottom_last_block"])
    # first block whose elements reach past 2^31 with a 32-bit product
    first = next(i for i in range(4000) if (i + 1) * g["block_stride_elems"] - 1 >= 2 ** 31)
    assert first == g["first_block_reaching_int32"]


@pytest.fixture(scope="module")
def bigpool_pair():
    top = W.bigpool(top=True, q_len=2048)
    bot = W.bigpool(top=False, q_len=2048)
    assert np.array_equal(top.requests[0].k_tok, bot.requests[0].k_tok)
    pools = {}
    for name, p in (("top", top), ("bot", bot)):
        pools[name] = (p, p.pool_numpy("k"), p.pool_numpy("v"))
    return pools


def _sample_tokens(p, kp, vp, toks, **kw):
    return np.stack([oracle.paged_prefill_attn(p.q, kp, vp, p.block_table(), p.seq_lens, p.query_start_loc,
                                               p.num_q_heads, p.softmax_scale, tok_begin=t, tok_end=t + 1,
                                               **kw)[0] for t in toks])


def test_bigpool_top_equals_bottom(bigpool_pair):
    toks = [0, 2047]
    outs = {n: _sample_tokens(*v, toks) for n, v in bigpool_pair.items()}
    assert np.isfinite(outs["top"]).all()
    assert np.array_equal(outs["top"], outs["bot"])


def test_planted_int32_offset_breaks_top_placement(bigpool_pair):
    toks = [2047]
    good = _sample_tokens(*bigpool_pair["bot"], toks)
    try:
        oracle.set_offset_mode_for_testing(1)
        bot = _sample_tokens(*bigpool_pair["bot"], toks)
        top = _sample_tokens(*bigpool_pair["top"], toks)
    finally:
        oracle.set_offset_mode_for_testing(0)
    assert np.array_equal(bot, good)          # low blocks never overflow
    assert not np.array_equal(top, good)      # the top placement is caught


# --------------------------------------------------------------------------------------------
# verify (A5 / A6)
# --------------------------------------------------------------------------------------------


def _small_verify(seed=7, lengths=(100, 37, 260), T=8, hq=8, hkv=2, d=32, bs=16):
    p = W.make_problem("v", seed=seed, seq_lens=[L + T for L in lengths], q_lens=[T] * len(lengths),
                       num_blocks=64, block_size=bs, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                       kv_dtype="int8", softmax_scale=0.2)
    return p


def _verify_args(p):
    return (p.q, p.pool_numpy("k"), p.pool_numpy("v"), p.scale_pool_numpy("k"), p.scale_pool_numpy("v"),
            p.block_table(), p.seq_lens)


def test_verify_equals_prefill_path_on_exact_values():
    # power-of-two scales make k8 * ks exact in bf16: the bf16 prefill oracle must agree
    p = _small_verify()
    T = 8
    for r in p.requests:
        r.ks_tok[:] = 2.0 ** -5
        r.vs_tok[:] = 2.0 ** -4
    ver = oracle.spec_verify_attn(*_verify_args(p), T, p.num_q_heads, p.softmax_scale)
    bf = W.make_problem("b", seed=1, seq_lens=list(p.seq_lens), q_lens=[T] * p.num_reqs, num_blocks=64,
                        block_size=p.block_size, num_q_heads=p.num_q_heads, num_kv_heads=p.num_kv_heads,
                        head_dim=p.head_dim, softmax_scale=p.softmax_scale)
    for rb, rv in zip(bf.requests, p.requests):
        rb.blocks = rv.blocks
        rb.k_tok = W.to_bf16_bits(rv.k_tok.astype(np.float32) * 2.0 ** -5)
        rb.v_tok = W.to_bf16_bits(rv.v_tok.astype(np.float32) * 2.0 ** -4)
    bf.q = p.q
    pre = _run_paged(bf)
    np.testing.assert_allclose(ver, pre, atol=1e-6, rtol=0)


@pytest.mark.parametrize("split", [16, 50, 64, 1000])
def test_verify_split_combine_equals_unsplit(split):
    p = _small_verify()
    T = 8
    args = _verify_args(p)
    full = oracle.spec_verify_attn(*args, T, p.num_q_heads, p.softmax_scale)
    max_splits = int(math.ceil(p.seq_lens.max() / split))
    po, pl = oracle.spec_verify_partial(*args, T, p.num_q_heads, p.softmax_scale, split, max_splits)
    comb = oracle.spec_verify_combine(po, pl, p.seq_lens, T, split)
    np.testing.assert_allclose(comb, full, atol=1e-6, rtol=1e-5)
    if split == 1000:   # one split: the combine returns the partial itself
        np.testing.assert_allclose(comb, po[0], atol=1e-7)


def test_verify_empty_split_has_neg_inf_lse():
    # split boundary right after the cached prefix: token t=0 sees no key of the last split
    T, L = 8, 64
    p = _small_verify(lengths=(L,), T=T)
    args = _verify_args(p)
    split = L + 2      # split 1 = keys [66, 72): visible to t >= 2 only
    po, pl = oracle.spec_verify_partial(*args, T, p.num_q_heads, p.softmax_scale, split, 2)
    assert np.all(np.isneginf(pl[1, 0:2])) and np.all(po[1, 0:2] == 0)
    assert np.all(np.isfinite(pl[1, 2:]))


def test_verify_zero_keys_mean_of_visible_dequantized_values():
    T = 4
    p = _small_verify(lengths=(30,), T=T)
    for r in p.requests:
        r.k_tok[:] = 0
    out = oracle.spec_verify_attn(*_verify_args(p), T, p.num_q_heads, p.softmax_scale)
    req, g = p.requests[0], p.num_q_heads // p.num_kv_heads
    vf = req.v_tok.astype(np.float64) * req.vs_tok[..., None].astype(np.float64)
    for t in range(T):
        n = 30 + t + 1
        for h in range(p.num_q_heads):
            np.testing.assert_allclose(out[t, h], vf[:n, h // g].mean(axis=0), atol=1e-6)


# --------------------------------------------------------------------------------------------
# verify over a per-tensor fp8 e4m3 cache
# --------------------------------------------------------------------------------------------


def _small_verify_fp8(seed=8, lengths=(100, 37, 260), T=8):
    return W.make_problem("vf", seed=seed, seq_lens=[L + T for L in lengths], q_lens=[T] * len(lengths),
                          num_blocks=64, block_size=16, num_q_heads=8, num_kv_heads=2, head_dim=32,
                          kv_dtype="e4m3", softmax_scale=0.2)


def test_verify_fp8_equals_prefill_path_on_bf16_copy():
    # every e4m3 value is exact in bf16, and so is its product with a power-of-two descale: the same
    # values through the bf16 prefill oracle must agree
    T = 8
    p = _small_verify_fp8()
    kd, vd = 0.5, 0.25
    ver = oracle.spec_verify_attn_fp8(p.q, p.pool_numpy("k"), p.pool_numpy("v"), kd, vd, p.block_table(),
                                      p.seq_lens, T, p.num_q_heads, p.softmax_scale)
    bf = W.make_problem("b", seed=1, seq_lens=list(p.seq_lens), q_lens=[T] * p.num_reqs, num_blocks=64,
                        block_size=16, num_q_heads=8, num_kv_heads=2, head_dim=32, softmax_scale=p.softmax_scale)
    for rb, rv in zip(bf.requests, p.requests):
        rb.blocks = rv.blocks
        f = lambda codes, sc: W.to_bf16_bits(
            torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy() * sc)
        rb.k_tok, rb.v_tok = f(rv.k_tok, kd), f(rv.v_tok, vd)
    bf.q = p.q
    np.testing.assert_allclose(ver, _run_paged(bf), atol=1e-6, rtol=0)


@pytest.mark.parametrize("split", [16, 64])
def test_verify_fp8_split_combine_equals_unsplit(split):
    T = 8
    p = _small_verify_fp8()
    args = (p.q, p.pool_numpy("k"), p.pool_numpy("v"), 0.5, 0.25, p.block_table(), p.seq_lens)
    full = oracle.spec_verify_attn_fp8(*args, T, p.num_q_heads, p.softmax_scale)
    S = int(math.ceil(p.seq_lens.max() / split))
    po, pl = oracle.spec_verify_partial_fp8(*args, T, p.num_q_heads, p.softmax_scale, split, S)
    np.testing.assert_allclose(oracle.spec_verify_combine(po, pl, p.seq_lens, T, split), full, atol=1e-6, rtol=1e-5)


# --------------------------------------------------------------------------------------------
# cache write (bf16 copy, int8 per token-head, e4m3 per tensor) and the e4m3 encoder
# --------------------------------------------------------------------------------------------


def test_e4m3_encode_round_trips_every_finite_code():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.f32_to_e4m3(oracle.e4m3_to_f32(c)) == c, hex(c)


def test_e4m3_encode_matches_torch_in_range():
    # torch's float32 -> float8_e4m3fn cast rounds to nearest even; below 464 it never overflows
    vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    mids = np.array([(vals[c] + vals[c + 1]) / 2 for c in range(0x7E)], dtype=np.float32)  # exact ties
    rng = np.random.default_rng(5)
    x = np.concatenate([mids, -mids, rng.standard_normal(4000).astype(np.float32) * np.float32(60),
                        rng.standard_normal(2000).astype(np.float32) * np.float32(3e-3),
                        np.array([463.9, -463.9, 0.0, -0.0, 1e-30], dtype=np.float32)])
    x = x[np.abs(x) < 464]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.f32_to_e4m3(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates_to_448():
    # the saturating ("satfinite") reading: every magnitude past 448, infinity included, becomes 448
    for v in (448.0, 449.0, 464.0, 480.0, 1e6, float("inf")):
        assert oracle.f32_to_e4m3(v) == 0x7E and oracle.f32_to_e4m3(-v) == 0xFE, v
    assert oracle.f32_to_e4m3(float("nan")) == 0x7F


def _write_problem(kv_dtype="bf16", q_lens=(70, 45, 33), seq_lens=(70, 80, 200), seed=31, bs=16, nb=40,
                   hkv=2, d=32):
    return W.make_problem("w", seed=seed, seq_lens=list(seq_lens), q_lens=list(q_lens), num_blocks=nb,
                          block_size=bs, num_q_heads=4, num_kv_heads=hkv, head_dim=d, kv_dtype=kv_dtype)


def _pool_shape(p):
    return (p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim)


def test_cache_write_whole_context_rebuilds_the_pool():
    # every position written (q_len == seq_len): the pool equals the fixture's own placement, and
    # slots no table points at keep their poison
    p = _write_problem(q_lens=(70, 80, 200))
    poison = 0x7FC1
    empty = np.full(_pool_shape(p), poison, dtype=np.uint16)
    kp, vp, _, _, rc = oracle.kv_cache_write(oracle.KV_BF16, W.new_rows(p, "k"), W.new_rows(p, "v"),
                                             p.block_table(), p.seq_lens, p.query_start_loc, empty, empty)
    assert rc == 0
    assert np.array_equal(kp, p.pool_numpy("k", fill=poison))
    assert np.array_equal(vp, p.pool_numpy("v", fill=poison))


def test_cache_write_chunks_compose():
    # a context written chunk by chunk (each chunk at positions seq_len - q_len ..) equals the
    # context written at once
    p_all = _write_problem(q_lens=(70, 80, 200))
    kp = np.zeros(_pool_shape(p_all), dtype=np.uint16)
    vp = kp.copy()
    bounds = [(0, 30), (30, 64), (64, 200)]
    for lo, hi in bounds:
        ends = [min(hi, L) for L in p_all.seq_lens]
        q_lens = [max(0, e - min(lo, e)) for e in ends]
        rows_k = np.concatenate([r.k_tok[e - q: e] for r, e, q in zip(p_all.requests, ends, q_lens)])
        rows_v = np.concatenate([r.v_tok[e - q: e] for r, e, q in zip(p_all.requests, ends, q_lens)])
        qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
        kp, vp, _, _, rc = oracle.kv_cache_write(oracle.KV_BF16, rows_k, rows_v, p_all.block_table(),
                                                 np.array(ends, np.int32), qsl, kp, vp)
        assert rc == 0
    assert np.array_equal(kp, p_all.pool_numpy("k"))
    assert np.array_equal(vp, p_all.pool_numpy("v"))


def test_cache_write_then_attend_equals_attention_on_the_fixture_pool():
    # a partial chunk written into a pool that holds only the older rows: attention over the written
    # pool is bit-identical to attention over the fixture's full pool
    p = _write_problem()
    owner = W.slot_owner_pool(p)
    kfull, vfull = p.pool_numpy("k"), p.pool_numpy("v")
    kold, vold = kfull.copy(), vfull.copy()
    kold[owner != 0] = 0x7FC0  # NaN where the chunk's rows go
    vold[owner != 0] = 0x7FC0
    kp, vp, _, _, rc = oracle.kv_cache_write(oracle.KV_BF16, W.new_rows(p, "k"), W.new_rows(p, "v"),
                                             p.block_table(), p.seq_lens, p.query_start_loc, kold, vold)
    assert rc == 0
    assert np.array_equal(_run_paged(p, kp, vp), _run_paged(p, kfull, vfull))


def test_cache_write_int8_rows_are_the_quantized_new_rows():
    p = _write_problem()
    owner = W.slot_owner_pool(p)
    kn, vn = W.new_rows(p, "k"), W.new_rows(p, "v")
    z8 = np.zeros(_pool_shape(p), dtype=np.int8)
    zs = np.full(_pool_shape(p)[:3], -1.0, dtype=np.float32)
    kp, vp, ksp, vsp, rc = oracle.kv_cache_write(oracle.KV_INT8, kn, vn, p.block_table(), p.seq_lens,
                                                 p.query_start_loc, z8, z8, zs, zs)
    assert rc == 0
    hkv = p.num_kv_heads
    for pool, sp, rows in ((kp, ksp, kn), (vp, vsp, vn)):
        assert np.array_equal(sp[owner == 0], zs[owner == 0])  # untouched slots keep their values
        assert not pool[owner == 0].any()
        for b, s, h in zip(*np.nonzero(owner)):
            t, hh = divmod(int(owner[b, s, h]) - 1, hkv)
            assert hh == h
            codes, scale = oracle.quant_row(rows[t, h])
            assert np.array_equal(pool[b, s, h], codes) and sp[b, s, h] == np.float32(scale)
            x = W.bf16_bits_to_f32(rows[t, h]).astype(np.float64)
            assert np.abs(x - pool[b, s, h].astype(np.float64) * scale).max() <= scale * 0.5 * (1 + 1e-5) + 1e-30


@pytest.mark.parametrize("scale", [0.5, 2.0])
def test_cache_write_fp8_recovers_representable_values(scale):
    # rows that are e4m3 values times a power-of-two scale are stored exactly: the code is the
    # original byte, and dense dequantization gives the row back bit for bit
    p = _write_problem(kv_dtype="e4m3", q_lens=(70, 80, 200))
    codes_k = np.concatenate([r.k_tok for r in p.requests])
    codes_v = np.concatenate([r.v_tok for r in p.requests])
    codes_k[(codes_k & 0x7F) == 0x7F] = 0x01  # no NaN inputs
    codes_v[(codes_v & 0x7F) == 0x7F] = 0x01
    codes_k[codes_k == 0x80] = 0  # -0 stores as -0 but compare the positive zero only
    codes_v[codes_v == 0x80] = 0
    dec = torch.from_numpy(np.stack([codes_k, codes_v])).view(torch.float8_e4m3fn).float() * scale
    rows = dec.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).float(), dec)  # exact bf16
    z = np.zeros(_pool_shape(p), dtype=np.uint8)
    kp, vp, _, _, rc = oracle.kv_cache_write(oracle.KV_FP8, rows[0], rows[1], p.block_table(), p.seq_lens,
                                             p.query_start_loc, z, z, k_scale=scale, v_scale=scale)
    assert rc == 0
    off = np.concatenate([[0], np.cumsum(p.seq_lens)])
    for i, r in enumerate(p.requests):
        place_k = np.zeros_like(z)
        W.place_tokens(place_k, r.blocks, codes_k[off[i]: off[i + 1]], p.block_size)
        used = np.zeros(_pool_shape(p)[:2], dtype=bool)
        used[np.asarray(r.blocks)[np.arange(r.seq_len) // p.block_size], np.arange(r.seq_len) % p.block_size] = True
        assert np.array_equal(kp[used], place_k[used])
    kd, vd = oracle.kv_fp8_dequant_dense(kp, vp, p.block_table(), p.seq_lens, 256, scale, scale)
    for i, r in enumerate(p.requests):
        assert np.array_equal(kd[i, : r.seq_len], rows[0][off[i]: off[i + 1]])
        assert np.array_equal(vd[i, : r.seq_len], rows[1][off[i]: off[i + 1]])


def test_cache_write_fp8_error_bound():
    # general values: |decode(code) * s - x| is at most half an e4m3 step (relative 2^-4 for normals,
    # 2^-10 absolute in the subnormal range), after the scale
    p = _write_problem(q_lens=(30, 20, 40))
    kn, vn = W.new_rows(p, "k"), W.new_rows(p, "v")
    s = 0.37
    z = np.zeros(_pool_shape(p), dtype=np.uint8)
    kp, _, _, _, rc = oracle.kv_cache_write(oracle.KV_FP8, kn, vn, p.block_table(), p.seq_lens,
                                            p.query_start_loc, z, z, k_scale=s, v_scale=s)
    assert rc == 0
    owner = W.slot_owner_pool(p)
    dec = torch.from_numpy(kp).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    for b, sl, h in zip(*np.nonzero(owner)):
        t, _ = divmod(int(owner[b, sl, h]) - 1, p.num_kv_heads)
        x = W.bf16_bits_to_f32(kn[t, h]).astype(np.float64) / np.float32(s)
        tol = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6)
        assert (np.abs(dec[b, sl, h] - x) <= tol).all()


def test_cache_write_bad_table_entry_is_reported_and_skipped():
    p = _write_problem()
    bt = p.block_table()
    bt[1, 2] = p.num_blocks + 5  # request 1, positions 32..47 (inside its new rows 35..79)
    z = np.zeros(_pool_shape(p), dtype=np.uint16)
    kp, _, _, _, rc = oracle.kv_cache_write(oracle.KV_BF16, W.new_rows(p, "k"), W.new_rows(p, "v"), bt,
                                            p.seq_lens, p.query_start_loc, z, z)
    assert rc == 4
    good = p.block_table()
    kref, _, _, _, _ = oracle.kv_cache_write(oracle.KV_BF16, W.new_rows(p, "k"), W.new_rows(p, "v"), good,
                                             p.seq_lens, p.query_start_loc, z, z)
    lost = good[1, 2]
    kref[lost] = 0  # only the rows of the bad entry are missing
    assert np.array_equal(kp, kref)


def test_planted_int32_offset_breaks_top_placement_write():
    # the last 2,048 rows of the 20,000-token request written into the 2,600-block pool: with the
    # planted 32-bit product the top placement's rows do not land in their blocks
    p = W.bigpool(top=True, q_len=2048)
    kn, vn = W.new_rows(p, "k"), W.new_rows(p, "v")
    shape = _pool_shape(p)
    blocks = np.asarray(p.requests[0].blocks)
    want = p.pool_numpy("k")[blocks]
    outs = {}
    for mode in (0, 1):
        try:
            oracle.set_offset_mode_for_testing(mode)
            z = np.zeros(shape, dtype=np.uint16)
            zv = np.zeros(shape, dtype=np.uint16)
            kp, _, _, _, rc = oracle.kv_cache_write(oracle.KV_BF16, kn, vn, p.block_table(), p.seq_lens,
                                                    p.query_start_loc, z, zv, inplace=True)
        finally:
            oracle.set_offset_mode_for_testing(0)
        got = kp[blocks]
        # compare only the chunk's slots: positions 17,952 .. 19,999
        pos = np.arange(p.seq_lens[0] - 2048, p.seq_lens[0])
        outs[mode] = np.array_equal(got[pos // p.block_size, pos % p.block_size],
                                    want[pos // p.block_size, pos % p.block_size])
    assert outs[0] and not outs[1]
