"""GPU parity of pkv_kv_cache_write against the CPU oracle: the whole pool after the write is compared
byte for byte (every slot, written or not), for the bf16, int8-per-token-head and e4m3-per-tensor
caches, on ragged multi-request chunks, block sizes 16 and 880, rows with special values (all-zero,
NaN, magnitudes past the e4m3 range, negative zero, e4m3 subnormals), a bad table entry, and the
2,600-block pool with the request at the top (offsets past 2^31 elements)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _devsetup import DEV, bf16_to_u16, dev_err, u16_to_bf16
from _parity import TOL_BF16, close

pytestmark = pytest.mark.gpu

POISON = {oracle.KV_BF16: 0x7FC1, oracle.KV_INT8: 0x55, oracle.KV_FP8: 0x33}
NP_DT = {oracle.KV_BF16: np.uint16, oracle.KV_INT8: np.int8, oracle.KV_FP8: np.uint8}
TORCH_DT = {oracle.KV_BF16: torch.bfloat16, oracle.KV_INT8: torch.int8, oracle.KV_FP8: torch.uint8}


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_int64_gb300 as m
    assert torch.cuda.is_available()
    return m


def _special_rows(rows: np.ndarray) -> np.ndarray:
    """Plant the edge cases into a copy of the new rows (uint16 bf16 bits [total][hkv][D])."""
    x = rows.copy()
    n = x.shape[0]
    x[0, 0] = 0                                   # all-zero row: scale 0, codes 0
    if n > 1:
        x[1, 1 % x.shape[1], 17] = 0x7FC0        # a NaN element: int8 row scale NaN, e4m3 code NaN
    if n > 2:
        f = W.bf16_bits_to_f32(x[2]) * np.float32(1000.0)  # past 448 * scale: saturates in e4m3
        x[2] = W.to_bf16_bits(f)
    if n > 3:
        x[3, :, ::3] = 0x8000                     # negative zeros
    if n > 4:
        f = W.bf16_bits_to_f32(x[4]) * np.float32(1e-3)  # e4m3 subnormal range after the scale
        x[4] = W.to_bf16_bits(f)
    return x


def _to_dev_rows(rows_u16, stride_pad=0):
    """bf16 rows on the device; with stride_pad > 0 they are a view into wider token rows (as in a
    packed projection output), so the token stride is not hkv * D."""
    t = u16_to_bf16(rows_u16).to(DEV)
    if not stride_pad:
        return t
    total, hkv, d = t.shape
    wide = torch.full((total, hkv * d + stride_pad), float("nan"), dtype=torch.bfloat16, device=DEV)
    wide[:, :hkv * d] = t.reshape(total, hkv * d)
    return wide[:, :hkv * d].view(total, hkv, d)


def _run(pkv, p, dt, kn, vn, bt=None, scale=(0.5, 0.75), stride_pad=0, expect_err=0):
    shape = (p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim)
    poison = POISON[dt]
    host_k = np.full(shape, poison, dtype=NP_DT[dt])
    host_v = host_k.copy()
    sshape = shape[:3]
    host_s = np.full(sshape, -1.0, dtype=np.float32)
    bt_np = p.block_table(fill=-1) if bt is None else bt
    # device side
    if dt == oracle.KV_BF16:
        kc = torch.full(shape, int(np.uint16(poison).view(np.int16)), dtype=torch.int16, device=DEV).view(torch.bfloat16)
    else:
        kc = torch.full(shape, int(np.array(poison, NP_DT[dt])), dtype=TORCH_DT[dt], device=DEV)
    vc = kc.clone()
    ksc = torch.full(sshape, -1.0, dtype=torch.float32, device=DEV)
    vsc = ksc.clone()
    kscale = torch.tensor([scale[0]], dtype=torch.float32, device=DEV)
    vscale = torch.tensor([scale[1]], dtype=torch.float32, device=DEV)
    err = dev_err()
    bt_d = torch.from_numpy(bt_np).to(DEV)
    sl = torch.from_numpy(p.seq_lens).to(DEV)
    qsl = torch.from_numpy(p.query_start_loc).to(DEV)
    max_q = max(r.q_len for r in p.requests)
    pkv.kv_cache_write(_to_dev_rows(kn, stride_pad), _to_dev_rows(vn, stride_pad), bt_d, sl, qsl, max_q, kc, vc,
                       kv_dtype=dt, k_scale_cache=ksc if dt == oracle.KV_INT8 else None,
                       v_scale_cache=vsc if dt == oracle.KV_INT8 else None,
                       k_scale=kscale if dt == oracle.KV_FP8 else None, v_scale=vscale if dt == oracle.KV_FP8 else None,
                       dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == expect_err
    rk, rv, rks, rvs, rc = oracle.kv_cache_write(dt, kn, vn, bt_np, p.seq_lens, p.query_start_loc, host_k, host_v,
                                                 host_s, host_s, k_scale=scale[0], v_scale=scale[1])
    assert rc == expect_err
    return (kc, vc, ksc, vsc), (rk, rv, rks, rvs)


def _host(t, dt):
    if dt == oracle.KV_BF16:
        return bf16_to_u16(t)
    return t.cpu().numpy().view(NP_DT[dt])


def _assert_same(dev, ref, dt):
    kc, vc, ksc, vsc = dev
    rk, rv, rks, rvs = ref
    for got_t, want in ((kc, rk), (vc, rv)):
        got = _host(got_t, dt)
        if dt == oracle.KV_FP8:  # a NaN input gives a NaN code; its sign bit is not specified
            nan = want == 0x7F
            assert ((got[nan] & 0x7F) == 0x7F).all()
            assert np.array_equal(got[~nan], want[~nan])
        else:
            assert np.array_equal(got, want)
    if dt == oracle.KV_INT8:
        for got_t, want in ((ksc, rks), (vsc, rvs)):
            got = got_t.cpu().numpy()
            assert np.array_equal(np.isnan(got), np.isnan(want))
            ok = ~np.isnan(want)
            assert np.array_equal(got[ok].view(np.uint32), want[ok].view(np.uint32))


def _ragged(bs=16, nb=64, seed=41):
    # a from-scratch chunk (q_len == seq_len), a mid chunk, a request with no new rows, a 1-token chunk
    return W.make_problem("wr", seed=seed, seq_lens=[150, 333, 40, 77], q_lens=[150, 129, 0, 1], num_blocks=nb,
                          block_size=bs, num_q_heads=16, num_kv_heads=4, head_dim=256)


@pytest.mark.parametrize("dt", [oracle.KV_BF16, oracle.KV_INT8, oracle.KV_FP8])
@pytest.mark.parametrize("bs,nb", [(16, 64), (880, 4)])
def test_cache_write_ragged_bit_exact(pkv, dt, bs, nb):
    p = _ragged(bs=bs, nb=nb)
    kn, vn = _special_rows(W.new_rows(p, "k")), _special_rows(W.new_rows(p, "v"))
    dev, ref = _run(pkv, p, dt, kn, vn)
    _assert_same(dev, ref, dt)


@pytest.mark.parametrize("dt", [oracle.KV_INT8, oracle.KV_FP8])
def test_cache_write_strided_rows(pkv, dt):
    # new rows read out of wider token rows (token stride 1,024 + 64 elements)
    p = _ragged()
    kn, vn = W.new_rows(p, "k"), W.new_rows(p, "v")
    dev, ref = _run(pkv, p, dt, kn, vn, stride_pad=64)
    _assert_same(dev, ref, dt)


def test_cache_write_bad_entry_is_reported_and_skipped(pkv):
    p = _ragged()
    bt = p.block_table(fill=-1)
    bt[1, 15] = p.num_blocks + 3  # request 1, positions 240..255 (inside its new rows 204..332)
    kn, vn = W.new_rows(p, "k"), W.new_rows(p, "v")
    dev, ref = _run(pkv, p, oracle.KV_INT8, kn, vn, bt=bt, expect_err=4)
    _assert_same(dev, ref, oracle.KV_INT8)


def _write_bigpool(pkv, p, dt, kn, vn):
    """Write the chunk's rows into fresh poisoned 2,600-block device pools; returns the caches."""
    shape = (p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim)
    poison = POISON[dt]
    if dt == oracle.KV_BF16:
        kc = torch.full(shape, int(np.uint16(poison).view(np.int16)), dtype=torch.int16, device=DEV).view(torch.bfloat16)
    else:
        kc = torch.full(shape, poison, dtype=TORCH_DT[dt], device=DEV)
    vc = kc.clone()
    ksc = torch.full(shape[:3], -1.0, dtype=torch.float32, device=DEV)
    vsc = ksc.clone()
    kscale = torch.tensor([0.5], dtype=torch.float32, device=DEV)
    vscale = torch.tensor([0.75], dtype=torch.float32, device=DEV)
    err = dev_err()
    bt = torch.from_numpy(p.block_table(fill=-1)).to(DEV)
    sl = torch.from_numpy(p.seq_lens).to(DEV)
    qsl = torch.from_numpy(p.query_start_loc).to(DEV)
    pkv.kv_cache_write(_to_dev_rows(kn), _to_dev_rows(vn), bt, sl, qsl, 2048, kc, vc, kv_dtype=dt,
                       k_scale_cache=ksc if dt == oracle.KV_INT8 else None,
                       v_scale_cache=vsc if dt == oracle.KV_INT8 else None,
                       k_scale=kscale if dt == oracle.KV_FP8 else None, v_scale=vscale if dt == oracle.KV_FP8 else None,
                       dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return kc, vc, ksc, vsc


@pytest.mark.parametrize("dt", [oracle.KV_BF16, oracle.KV_INT8, oracle.KV_FP8])
def test_cache_write_bigpool_top_placement(pkv, dt):
    """The last 2,048 rows of the 20,000-token request into the 2,600-block pool, blocks 2,577-2,599:
    element offsets reach 2.34e9 > 2^31. The written blocks equal the oracle's write byte for byte
    (the oracle writes a pool holding just those blocks) and the same write at blocks 0-22 bit for
    bit; nothing outside the request's blocks changes."""
    p = W.bigpool(top=True, q_len=2048)
    kn, vn = W.new_rows(p, "k"), W.new_rows(p, "v")
    shape = (p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim)
    poison = POISON[dt]
    kc, vc, ksc, vsc = _write_bigpool(pkv, p, dt, kn, vn)
    blocks = np.asarray(p.requests[0].blocks)
    assert blocks.min() >= 2577
    # oracle on a pool holding just those blocks (same slots, block ids remapped to 0..22)
    small_bt = np.arange(len(blocks), dtype=np.int32)[None, :]
    hs = (len(blocks),) + shape[1:]
    hk = np.full(hs, poison, dtype=NP_DT[dt])
    hsc = np.full(hs[:3], -1.0, dtype=np.float32)
    rk, rv, rks, rvs, rc = oracle.kv_cache_write(dt, kn, vn, small_bt, p.seq_lens, p.query_start_loc, hk, hk.copy(),
                                                 hsc, hsc.copy(), k_scale=0.5, v_scale=0.75)
    assert rc == 0
    bidx = torch.from_numpy(blocks).to(DEV)
    top = (kc[bidx], vc[bidx], ksc[bidx], vsc[bidx])
    _assert_same(top, (rk, rv, rks, rvs), dt)
    # nothing outside the request's blocks was touched: every changed element lies in those blocks
    for c in (kc, vc):
        raw = c.view(torch.int16) if dt == oracle.KV_BF16 else c
        want = int(np.uint16(poison).view(np.int16)) if dt == oracle.KV_BF16 else poison
        assert int((raw != want).sum()) == int((raw[bidx] != want).sum())
    top = tuple(t.clone() for t in top)
    del kc, vc, ksc, vsc
    torch.cuda.empty_cache()
    # the same rows at the bottom of the pool: the written blocks are identical bit for bit
    pb = W.bigpool(top=False, q_len=2048)
    kc, vc, ksc, vsc = _write_bigpool(pkv, pb, dt, kn, vn)
    bb = torch.from_numpy(np.asarray(pb.requests[0].blocks)).to(DEV)
    for a, b in zip(top, (kc[bb], vc[bb], ksc[bb], vsc[bb])):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_written_int8_cache_feeds_verify(pkv):
    """An int8 cache written by the kernel, then read by the split-KV verify: equal to the oracle's
    verify on the oracle-written cache (the write and the read agree on addresses and scales)."""
    T = 8
    p = W.make_problem("wv", seed=43, seq_lens=[300 + T, 129 + T], q_lens=[300 + T, 129 + T], num_blocks=40,
                       block_size=16, num_q_heads=16, num_kv_heads=4, head_dim=256, softmax_scale=1.0 / 16.0)
    kn, vn = W.new_rows(p, "k"), W.new_rows(p, "v")
    dev, ref = _run(pkv, p, oracle.KV_INT8, kn, vn)
    _assert_same(dev, ref, oracle.KV_INT8)
    kc, vc, ksc, vsc = dev
    # verify queries: the last T tokens of each request
    q = W.bf16_normal(77, (2 * T, 16, 256))
    qd = u16_to_bf16(q).to(DEV)
    bt = torch.from_numpy(p.block_table(fill=-1)).to(DEV)
    sl = torch.from_numpy(p.seq_lens).to(DEV)
    split = 128
    S = pkv.splits_needed(int(p.seq_lens.max()), split)
    po = torch.empty((S, 2 * T, 16, 256), dtype=torch.float32, device=DEV)
    pl = torch.empty((S, 2 * T, 16), dtype=torch.float32, device=DEV)
    out = torch.empty_like(qd)
    err = dev_err()
    pkv.spec_verify_attn_partial(qd, kc, vc, ksc, vsc, bt, sl, T, p.softmax_scale, split, po, pl, dev_err=err)
    pkv.spec_verify_combine(po, pl, sl, T, split, out)
    torch.cuda.synchronize()
    assert err.item() == 0
    rk, rv, rks, rvs = ref
    want = oracle.spec_verify_attn(q, rk, rv, rks, rvs, p.block_table(fill=0), p.seq_lens, T, 16, p.softmax_scale)
    close(bf16_to_u16(out), want, TOL_BF16)
