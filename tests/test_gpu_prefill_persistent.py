"""GPU parity of the persistent prefill launch: the same attention as the classic grid, with the
query tiles of the last partial wave cut into key ranges so that every SM has work.

Every case runs at several grid sizes (a workspace sized for P CTAs gives a grid of P): P = 1 (one
CTA walks every unit, nothing is cut), small P (many units per CTA, several cut), and the full SM
count. Bars: query tiles that the schedule does not cut are computed with the classic kernel's
arithmetic in the same order, so their rows equal the classic launch bit for bit; rows of cut tiles
are merged from fp32 partials; every row meets the parity bar against the oracle. The
workspace starts as NaN, so a read of a slot that no CTA wrote shows up.
"""
import numpy as np
import pytest
import torch

import oracle
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


from _devsetup import bf16_to_u16, dev_err, device_meta, device_pool, device_q  # noqa: E402
from _parity import TOL_BF16, TOL_INT8, close  # noqa: E402
from test_gpu_parity import _oracle_prefill  # noqa: E402


def split_count(R, P, k_max=4):
    """the number of key ranges each unit of the last partial wave is cut into: k in [1, 4]
    minimising ceil(R k / P) / k + 0.02 (k - 1)."""
    best, best_cost = 1, 2.0
    for k in range(1, k_max + 1):
        if R == 0:
            break
        cost = -(-R * k // P) / k + 0.02 * (k - 1)
        if cost < best_cost - 1e-6:
            best, best_cost = k, cost
    return best


def cut_rows(p, P):
    """Host model of the persistent schedule: a boolean per (token, q head), True where the row's
    query tile is cut into key ranges. Units with rows, in the order m-tile descending, request,
    head; the first P floor(U / P) are whole, the remaining R are cut when split_count(R, P) > 1."""
    n_mt = (max(r.q_len for r in p.requests) + 127) // 128
    units = []
    for mt in reversed(range(n_mt)):
        for r, req in enumerate(p.requests):
            if mt * 128 >= req.q_len or req.q_len > req.seq_len:
                continue
            rows = min(128, req.q_len - mt * 128)
            for qh in range(p.num_q_heads):
                units.append((int(p.query_start_loc[r]) + mt * 128, rows, qh))
    U = len(units)
    F = P * (U // P)
    cut = np.zeros((p.total_q, p.num_q_heads), dtype=bool)
    if split_count(U - F, P) > 1:
        for tok0, rows, qh in units[F:]:
            cut[tok0:tok0 + rows, qh] = True
    return cut


def _inputs(pkv, p, mode):
    k, v = device_pool(p, "k"), device_pool(p, "v")
    bt, sl, qsl = device_meta(p)
    q = device_q(p)
    kw = {}
    if mode:
        max_ctx = int(p.seq_lens.max())
        k8 = torch.zeros((p.num_reqs, max_ctx, p.num_kv_heads, 256), dtype=torch.int8, device="cuda")
        ks = torch.zeros((p.num_reqs, max_ctx, p.num_kv_heads), dtype=torch.float32, device="cuda")
        k16 = torch.zeros((p.num_reqs, max_ctx, p.num_kv_heads, 256), dtype=torch.float16, device="cuda")
        pb = torch.zeros(p.num_reqs, dtype=torch.int32, device="cuda")
        pkv.kv_int8_stats_quant(k, bt, pb, sl, max_ctx, k8, ks, k16=k16)
        kw = dict(qk_mode=1, k8_scale=ks, k8=k8 if mode == 1 else None, k16=k16 if mode == 2 else None)
        k = None
    return q, k, v, bt, sl, qsl, kw


def _prefill(pkv, p, inp, P):
    q, k, v, bt, sl, qsl, kw = inp
    out = torch.full_like(q, float("nan"))
    err = dev_err()
    ws = None
    if P:
        ws = torch.full((pkv.paged_prefill_workspace_bytes(P) // 4,), float("nan"), dtype=torch.float32,
                        device="cuda")
    pkv.paged_prefill_attn(q, k, v, bt, sl, qsl, max(r.q_len for r in p.requests), p.softmax_scale, out,
                           dev_err=err, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert err.item() == 0, f"device status {err.item()}"
    return bf16_to_u16(out)


CASES = {
    # several requests, q_len and seq_len off every tile boundary, one-tile units among long ones
    "ragged": dict(seq_lens=[700, 129, 300, 1], q_lens=[300, 129, 1, 1], num_blocks=80, block_size=16),
    # the pages' 24 query / 4 KV heads
    "gqa6": dict(seq_lens=[517, 260], q_lens=[200, 133], num_blocks=64, block_size=16, num_q_heads=24,
                 num_kv_heads=4),
    # block 880: key tiles follow the blocks (6 of 128 keys and one of 112 per block)
    "bs880": dict(seq_lens=[2000, 1000], q_lens=[300, 1000], num_blocks=40, block_size=880),
    # block 200: tiles of 128 and 72 keys
    "bs200": dict(seq_lens=[1111, 333], q_lens=[400, 333], num_blocks=16, block_size=200),
    # one decode-like row per head over 3,000 keys: fewer tiles than CTAs, units cut into many pieces
    "thin": dict(seq_lens=[3000], q_lens=[1], num_blocks=200, block_size=16, num_q_heads=4, num_kv_heads=4),
}


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("case", list(CASES))
def test_persistent_prefill_matches_classic_and_oracle(pkv, mode, case):
    p = W.make_problem(case, seed=60 + list(CASES).index(case), **CASES[case])
    inp = _inputs(pkv, p, mode)
    classic = _prefill(pkv, p, inp, 0)
    ref = _oracle_prefill(p, min(mode, 1))
    tol = TOL_INT8 if mode else TOL_BF16
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for P in (1, 3, 7, sms):
        got = _prefill(pkv, p, inp, P)
        cut = cut_rows(p, P)
        assert P > 1 or not cut.any()
        whole = ~cut
        assert np.array_equal(got.reshape(p.total_q, p.num_q_heads, 256)[whole],
                              classic.reshape(p.total_q, p.num_q_heads, 256)[whole]), f"P={P}"
        close(got, ref, tol, f"P={P}")


def test_persistent_fp8_fused_prefill(pkv):
    """The fused fp8 path on the persistent grid equals its classic launch on uncut query tiles and
    the dense-scratch oracle everywhere."""
    p = W.make_problem("f8p", seed=70, seq_lens=[1500, 300, 129], q_lens=[700, 300, 1], num_blocks=150,
                       block_size=16, kv_dtype="e4m3")
    k, v = device_pool(p, "k"), device_pool(p, "v")
    bt, sl, qsl = device_meta(p)
    q = device_q(p)
    scale = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    max_q = max(r.q_len for r in p.requests)

    def run(P):
        out = torch.full_like(q, float("nan"))
        err = dev_err()
        ws = None
        if P:
            ws = torch.full((pkv.paged_prefill_workspace_bytes(P) // 4,), float("nan"), dtype=torch.float32,
                            device="cuda")
        pkv.paged_prefill_attn_fp8(q, k, v, scale, scale, bt, sl, qsl, max_q, p.softmax_scale, out, dev_err=err,
                                   workspace=ws)
        torch.cuda.synchronize()
        assert err.item() == 0
        return bf16_to_u16(out)

    classic = run(0)
    rk, rv = oracle.kv_fp8_dequant_dense(p.pool_numpy("k"), p.pool_numpy("v"), p.block_table(fill=0), p.seq_lens,
                                         int(p.seq_lens.max()), 0.5, 0.5)
    ident = np.arange(p.num_reqs, dtype=np.int32).reshape(p.num_reqs, 1)
    ref = oracle.paged_prefill_attn(p.q, rk, rv, ident, p.seq_lens, p.query_start_loc, p.num_q_heads,
                                    p.softmax_scale)
    for P in (5, torch.cuda.get_device_properties(0).multi_processor_count):
        got = run(P)
        whole = ~cut_rows(p, P)
        assert np.array_equal(got.reshape(p.total_q, p.num_q_heads, 256)[whole],
                              classic.reshape(p.total_q, p.num_q_heads, 256)[whole])
        close(got, ref, TOL_BF16, f"P={P}")


def test_persistent_bigpool_sampled_rows(pkv):
    """The bench chunk (20,000-token request on the top blocks of a 2,600-block pool, last 2,048
    queries) on the full persistent grid: sampled rows against the oracle, in every qk mode."""
    p = W.bigpool(top=True)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cut = cut_rows(p, sms)
    for mode in (0, 2):
        inp = _inputs(pkv, p, mode)
        got = _prefill(pkv, p, inp, sms)
        classic = _prefill(pkv, p, inp, 0)
        whole = ~cut
        assert np.array_equal(got.reshape(p.total_q, p.num_q_heads, 256)[whole],
                              classic.reshape(p.total_q, p.num_q_heads, 256)[whole])
        # rows of cut and uncut tiles: the first and last rows of the chunk and of an m-tile boundary
        for t in (0, 127, 128, 1000, 2047):
            ref = _oracle_prefill(p, min(mode, 1), tok_begin=t, tok_end=t + 1)
            close(got[t:t + 1], ref, TOL_INT8 if mode else TOL_BF16, f"mode {mode}")
        assert cut.any() and whole.any()
        del inp
        torch.cuda.empty_cache()


def _run_both(pkv, p, bt, P_list):
    """classic then persistent launches (P CTAs each) on the same inputs: outputs and device status."""
    k, v = device_pool(p, "k"), device_pool(p, "v")
    _, sl, qsl = device_meta(p)
    q = device_q(p)
    max_q = max(max(r.q_len for r in p.requests), 1)
    res = []
    for P in [0] + list(P_list):
        out = torch.full_like(q, float("nan"))
        err = dev_err()
        ws = None
        if P:
            ws = torch.full((pkv.paged_prefill_workspace_bytes(P) // 4,), float("nan"), dtype=torch.float32,
                            device="cuda")
        pkv.paged_prefill_attn(q, k, v, bt, sl, qsl, max_q, p.softmax_scale, out, dev_err=err, workspace=ws)
        torch.cuda.synchronize()
        res.append((P, bf16_to_u16(out), err.item()))
    return res


def test_persistent_out_of_range_block_is_reported_and_zero_filled(pkv):
    """A table entry one past the pool: both launches report PKV_ERR_DEVICE_BOUNDS, read nothing
    through it (those keys count as zeros), and agree on every uncut query tile bit for bit."""
    p = W.make_problem("badp", seed=72, seq_lens=[700, 300], q_lens=[400, 300], num_blocks=80, block_size=16)
    bt, _, _ = device_meta(p)
    bt[0, 5] = p.num_blocks  # keys 80..95 of request 0
    res = _run_both(pkv, p, bt, (7, torch.cuda.get_device_properties(0).multi_processor_count))
    _, classic, err0 = res[0]
    assert err0 == pkv.PKV_ERR_DEVICE_BOUNDS
    assert np.isfinite(W.bf16_bits_to_f32(classic)).all()
    c = W.bf16_bits_to_f32(classic).astype(np.float64)
    for P, got, err in res[1:]:
        assert err == pkv.PKV_ERR_DEVICE_BOUNDS
        whole = ~cut_rows(p, P)
        g = got.reshape(p.total_q, p.num_q_heads, 256)
        assert np.array_equal(g[whole], classic.reshape(p.total_q, p.num_q_heads, 256)[whole])
        gf = W.bf16_bits_to_f32(got).astype(np.float64)
        assert np.isfinite(gf).all()
        assert (np.abs(gf - c) <= 2.0 ** -7 * np.abs(c) + 2e-3).all()


def test_persistent_skips_empty_and_inconsistent_requests(pkv):
    """A request with no queries and one whose q_len exceeds its seq_len (no causal chunk) have no
    query tiles: both launches leave the second's rows unwritten and compute the others alike."""
    p = W.make_problem("skip", seed=73, seq_lens=[300, 200, 30, 500], q_lens=[0, 150, 40, 130], num_blocks=80,
                       block_size=16)
    bt, _, _ = device_meta(p)
    res = _run_both(pkv, p, bt, (3, torch.cuda.get_device_properties(0).multi_processor_count))
    _, classic, err0 = res[0]
    c = W.bf16_bits_to_f32(classic).astype(np.float64)
    skipped = np.zeros(p.total_q, dtype=bool)
    skipped[150:190] = True  # request 2's rows
    assert np.isnan(c[skipped]).all() and np.isfinite(c[~skipped]).all()
    for P, got, err in res[1:]:
        assert err == err0
        gf = W.bf16_bits_to_f32(got).astype(np.float64)
        assert np.isnan(gf[skipped]).all() and np.isfinite(gf[~skipped]).all()
        whole = ~cut_rows(p, P)
        g = got.reshape(p.total_q, p.num_q_heads, 256)
        assert np.array_equal(g[whole & ~skipped[:, None]], classic.reshape(p.total_q, p.num_q_heads, 256)[
            whole & ~skipped[:, None]])
        assert (np.abs(gf[~skipped] - c[~skipped]) <= 2.0 ** -7 * np.abs(c[~skipped]) + 2e-3).all()
