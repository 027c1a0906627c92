"""CPU oracle for paged KV-cache attention - TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import this
package. It wraps the plain C oracle in pkv_oracle.c (built with gcc, -O2
-ffp-contract=off so the quantizers' fp32 operations are exactly the written ones)
through ctypes, with numpy arrays in and out. It shares no code with the CUDA
library and never imports it.

Every function is pinned by the `-m "not gpu"` tests in tests/test_oracle_pins.py;
none is "parity unpinned".
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source if missing or stale; returns its path."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                            "-shared", "-o", tmp, _SRC, "-lm"], check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        i32, i64, f32, vp = C.c_int32, C.c_int64, C.c_float, C.c_void_p
        L.orc_bf16_to_f32.argtypes = [C.c_uint16]
        L.orc_bf16_to_f32.restype = f32
        L.orc_f32_to_bf16_rne.argtypes = [f32]
        L.orc_f32_to_bf16_rne.restype = C.c_uint16
        L.orc_e4m3_to_f32.argtypes = [C.c_uint8]
        L.orc_e4m3_to_f32.restype = f32
        L.orc_f32_to_e4m3_sat.argtypes = [f32]
        L.orc_f32_to_e4m3_sat.restype = C.c_uint8
        L.orc_set_offset_mode_for_testing.argtypes = [C.c_int]
        L.orc_quant_row_i8.argtypes = [vp, C.c_int, vp, vp]
        L.orc_kv_int8_stats_quant.argtypes = [vp, i64, i64, i64, i64, vp, i64, vp, vp, i32, i32, i32,
                                              i32, vp, vp, i64]
        L.orc_kv_fp8_dequant_dense.argtypes = [vp, vp, i64, i64, i64, i64, vp, i64, vp, i32, i32, i32,
                                               i32, i32, f32, f32, vp, vp]
        L.orc_paged_prefill_attn.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, i64, vp, vp, i32, i32,
                                             i32, i32, i32, f32, i32, vp, vp, i64, i64, i64, vp]
        L.orc_dense_attn.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, f32, vp]
        L.orc_spec_verify_attn.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, i64,
                                           vp, i32, i32, i32, i32, i32, i32, f32, i32, i32, vp]
        L.orc_spec_verify_partial.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, i64,
                                              vp, i32, i32, i32, i32, i32, i32, f32, i32, i32, i32, i32,
                                              vp, vp]
        L.orc_spec_verify_combine.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
        L.orc_spec_verify_attn_fp8.argtypes = [vp, vp, vp, f32, f32, i64, i64, i64, i64, vp, i64, vp, i32, i32,
                                               i32, i32, i32, i32, f32, i32, i32, vp]
        L.orc_spec_verify_partial_fp8.argtypes = [vp, vp, vp, f32, f32, i64, i64, i64, i64, vp, i64, vp, i32,
                                                  i32, i32, i32, i32, i32, f32, i32, i32, i32, i32, vp, vp]
        L.orc_kv_cache_write.argtypes = [C.c_int, vp, vp, vp, i64, vp, vp, i32, i64, i64, i64, i64, i32, i32, i32,
                                         vp, vp, vp, vp, i64, i64, f32, f32]
        for name in ("orc_quant_row_i8", "orc_set_offset_mode_for_testing"):
            getattr(L, name).restype = None
        for name in ("orc_kv_int8_stats_quant", "orc_kv_fp8_dequant_dense", "orc_paged_prefill_attn",
                     "orc_dense_attn", "orc_spec_verify_attn", "orc_spec_verify_partial",
                     "orc_spec_verify_combine", "orc_spec_verify_attn_fp8", "orc_spec_verify_partial_fp8",
                     "orc_kv_cache_write"):
            getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what}: oracle status {rc}")


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ---- scalar formats -----------------------------------------------------------------------

def e4m3_to_f32(code: int) -> float:
    return lib().orc_e4m3_to_f32(int(code))


def f32_to_e4m3(x: float) -> int:
    """OCP E4M3 code of x: round to nearest even, +-448 for larger magnitudes, 0x7F for NaN."""
    return int(lib().orc_f32_to_e4m3_sat(float(x)))


def f32_to_bf16(x: float) -> int:
    return lib().orc_f32_to_bf16_rne(float(x))


def set_offset_mode_for_testing(mode: int) -> None:
    """0 = int64 block offsets (the method); 1 = 32-bit wraparound (planted mistake)."""
    lib().orc_set_offset_mode_for_testing(int(mode))


def quant_row(x_bf16: np.ndarray):
    x = _c(x_bf16, np.uint16)
    codes = np.zeros(x.size, dtype=np.int8)
    scale = np.zeros(1, dtype=np.float32)
    lib().orc_quant_row_i8(_p(x), x.size, _p(codes), _p(scale))
    return codes, float(scale[0])


# ---- cache write ----------------------------------------------------------------------------

KV_BF16, KV_INT8, KV_FP8 = 0, 1, 2


def kv_cache_write(kv_dtype, k_new, v_new, block_table, seq_lens, query_start_loc, k_pool, v_pool,
                   k_scale_pool=None, v_scale_pool=None, k_scale=1.0, v_scale=1.0, inplace=False):
    """Store the new rows k_new / v_new (uint16 bf16 bits [total][hkv][D]) into the pools (uint16
    [nb][bs][hkv][D] for bf16, int8 / uint8 for the int8 / fp8 caches; scale pools float32
    [nb][bs][hkv]), copies of them unless inplace (then they must be C-contiguous of that dtype);
    returns (k_pool, v_pool, k_scale_pool, v_scale_pool) after the write and the oracle status (0,
    or 4 when a table entry was outside the pool)."""
    dt = {KV_BF16: np.uint16, KV_INT8: np.int8, KV_FP8: np.uint8}[kv_dtype]

    def own(a, t):
        if inplace:
            assert a.dtype == t and a.flags.c_contiguous
            return a
        return np.array(a, dtype=t, copy=True)

    kp, vp_ = own(k_pool, dt), own(v_pool, dt)
    nb, bs, hkv, d = kp.shape
    ksp = vsp = None
    if kv_dtype == KV_INT8:
        ksp = own(k_scale_pool, np.float32)
        vsp = own(v_scale_pool, np.float32)
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    bt = _c(block_table, np.int32)
    sl, qsl = _c(seq_lens, np.int32), _c(query_start_loc, np.int32)
    rc = lib().orc_kv_cache_write(int(kv_dtype), _p(kn), _p(vn), _p(bt), bt.shape[1], _p(sl), _p(qsl), sl.size,
                                  nb, bs * hkv * d, hkv * d, d, bs, hkv, d, _p(kp), _p(vp_), _p(ksp), _p(vsp),
                                  bs * hkv, hkv, float(k_scale), float(v_scale))
    if rc not in (0, 4):
        _check(rc, "kv_cache_write")
    return kp, vp_, ksp, vsp, rc


# ---- A1 -----------------------------------------------------------------------------------

def kv_int8_stats_quant(k_pool, block_table, pos_begin, pos_end, block_size, max_ctx):
    """k_pool: uint16 [nb][bs][hkv][D]. Returns (k8 [R][max_ctx][hkv][D], ks [R][max_ctx][hkv])."""
    k_pool = _c(k_pool, np.uint16)
    nb, bs, hkv, d = k_pool.shape
    bt = _c(block_table, np.int32)
    pb, pe = _c(pos_begin, np.int32), _c(pos_end, np.int32)
    R = bt.shape[0]
    k8 = np.zeros((R, max_ctx, hkv, d), dtype=np.int8)
    ks = np.zeros((R, max_ctx, hkv), dtype=np.float32)
    rc = lib().orc_kv_int8_stats_quant(_p(k_pool), nb, bs * hkv * d, hkv * d, d, _p(bt), bt.shape[1],
                                       _p(pb), _p(pe), R, block_size, hkv, d, _p(k8), _p(ks), max_ctx)
    _check(rc, "kv_int8_stats_quant")
    return k8, ks


# ---- A4 -----------------------------------------------------------------------------------

def kv_fp8_dequant_dense(k_pool, v_pool, block_table, seq_lens, max_seq, k_scale, v_scale):
    """e4m3 pools uint8 [nb][bs][hkv][D] -> dense bf16 bits [R][max_seq][hkv][D] (K, V)."""
    k_pool, v_pool = _c(k_pool, np.uint8), _c(v_pool, np.uint8)
    nb, bs, hkv, d = k_pool.shape
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    R = bt.shape[0]
    kd = np.zeros((R, max_seq, hkv, d), dtype=np.uint16)
    vd = np.zeros((R, max_seq, hkv, d), dtype=np.uint16)
    rc = lib().orc_kv_fp8_dequant_dense(_p(k_pool), _p(v_pool), nb, bs * hkv * d, hkv * d, d, _p(bt),
                                        bt.shape[1], _p(sl), R, max_seq, bs, hkv, d, float(k_scale),
                                        float(v_scale), _p(kd), _p(vd))
    _check(rc, "kv_fp8_dequant_dense")
    return kd, vd


# ---- A3 -----------------------------------------------------------------------------------

def paged_prefill_attn(q, k_pool, v_pool, block_table, seq_lens, query_start_loc, num_q_heads,
                       softmax_scale, qk_mode=0, k8=None, k8_scale=None, tok_begin=0, tok_end=None,
                       block_size=None):
    """q: uint16 [total_q][Hq][D]; pools uint16 [nb][bs][hkv][D] (or any array whose first dims
    are (nb, bs) with `block_size` given). Returns fp32 [tok_end-tok_begin][Hq][D]."""
    q = _c(q, np.uint16)
    nb, bs, hkv, d = k_pool.shape
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    bt, sl, qsl = _c(block_table, np.int32), _c(seq_lens, np.int32), _c(query_start_loc, np.int32)
    R = bt.shape[0]
    total_q = q.shape[0]
    if tok_end is None:
        tok_end = total_q
    out = np.zeros((tok_end - tok_begin, num_q_heads, d), dtype=np.float32)
    max_ctx = 0 if k8 is None else k8.shape[1]
    k8c = None if k8 is None else _c(k8, np.int8)
    ksc = None if k8_scale is None else _c(k8_scale, np.float32)
    rc = lib().orc_paged_prefill_attn(_p(q), _p(k_pool), _p(v_pool), nb, bs * hkv * d, hkv * d, d,
                                      _p(bt), bt.shape[1], _p(sl), _p(qsl), R, num_q_heads, hkv, d, bs,
                                      float(softmax_scale), int(qk_mode), _p(k8c), _p(ksc), max_ctx,
                                      tok_begin, tok_end, _p(out))
    _check(rc, "paged_prefill_attn")
    return out


def dense_attn(q, k, v, qpos, num_q_heads, softmax_scale):
    """Non-paged brute force: q uint16 [nq][Hq][D], k/v uint16 [L][hkv][D], qpos int64 [nq]."""
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    qpos = _c(qpos, np.int64)
    hkv, d = k.shape[1], k.shape[2]
    out = np.zeros((q.shape[0], num_q_heads, d), dtype=np.float32)
    rc = lib().orc_dense_attn(_p(q), _p(k), _p(v), _p(qpos), q.shape[0], num_q_heads, hkv, d,
                              float(softmax_scale), _p(out))
    _check(rc, "dense_attn")
    return out


# ---- A5 / A6 ------------------------------------------------------------------------------

def _verify_common(q, k_pool, v_pool, ks_pool, vs_pool, block_table, seq_lens):
    q = _c(q, np.uint16)
    nb, bs, hkv, d = k_pool.shape
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    assert ks_pool.flags.c_contiguous and vs_pool.flags.c_contiguous
    bt, sl = _c(block_table, np.int32), _c(seq_lens, np.int32)
    return q, nb, bs, hkv, d, bt, sl


def spec_verify_attn(q, k_pool, v_pool, ks_pool, vs_pool, block_table, seq_lens, T, num_q_heads,
                     softmax_scale, req_begin=0, req_end=None):
    q, nb, bs, hkv, d, bt, sl = _verify_common(q, k_pool, v_pool, ks_pool, vs_pool, block_table, seq_lens)
    R = bt.shape[0]
    if req_end is None:
        req_end = R
    out = np.zeros((R * T, num_q_heads, d), dtype=np.float32)
    rc = lib().orc_spec_verify_attn(_p(q), _p(k_pool), _p(v_pool), _p(ks_pool), _p(vs_pool), nb,
                                    bs * hkv * d, hkv * d, d, bs * hkv, hkv, _p(bt), bt.shape[1], _p(sl),
                                    R, T, num_q_heads, hkv, d, bs, float(softmax_scale), req_begin,
                                    req_end, _p(out))
    _check(rc, "spec_verify_attn")
    return out


def spec_verify_partial(q, k_pool, v_pool, ks_pool, vs_pool, block_table, seq_lens, T, num_q_heads,
                        softmax_scale, split_tokens, max_splits, req_begin=0, req_end=None):
    q, nb, bs, hkv, d, bt, sl = _verify_common(q, k_pool, v_pool, ks_pool, vs_pool, block_table, seq_lens)
    R = bt.shape[0]
    if req_end is None:
        req_end = R
    part_o = np.zeros((max_splits, R * T, num_q_heads, d), dtype=np.float32)
    part_lse = np.full((max_splits, R * T, num_q_heads), -np.inf, dtype=np.float32)
    rc = lib().orc_spec_verify_partial(_p(q), _p(k_pool), _p(v_pool), _p(ks_pool), _p(vs_pool), nb,
                                       bs * hkv * d, hkv * d, d, bs * hkv, hkv, _p(bt), bt.shape[1],
                                       _p(sl), R, T, num_q_heads, hkv, d, bs, float(softmax_scale),
                                       split_tokens, max_splits, req_begin, req_end, _p(part_o),
                                       _p(part_lse))
    _check(rc, "spec_verify_partial")
    return part_o, part_lse


def spec_verify_combine(part_o, part_lse, seq_lens, T, split_tokens):
    part_o, part_lse = _c(part_o, np.float32), _c(part_lse, np.float32)
    max_splits, rows_t, hq, d = part_o.shape
    sl = _c(seq_lens, np.int32)
    R = sl.shape[0]
    out = np.zeros((rows_t, hq, d), dtype=np.float32)
    rc = lib().orc_spec_verify_combine(_p(part_o), _p(part_lse), _p(sl), R, T, hq, d, split_tokens,
                                       max_splits, _p(out))
    _check(rc, "spec_verify_combine")
    return out


# ---- fp8 verify (per-tensor e4m3 cache) ------------------------------------------------------

def spec_verify_attn_fp8(q, k_pool, v_pool, k_descale, v_descale, block_table, seq_lens, T, num_q_heads,
                         softmax_scale, req_begin=0, req_end=None):
    q = _c(q, np.uint16)
    k_pool, v_pool = _c(k_pool, np.uint8), _c(v_pool, np.uint8)
    nb, bs, hkv, d = k_pool.shape
    bt, sl = _c(block_table, np.int32), _c(seq_lens, np.int32)
    R = bt.shape[0]
    if req_end is None:
        req_end = R
    out = np.zeros((R * T, num_q_heads, d), dtype=np.float32)
    rc = lib().orc_spec_verify_attn_fp8(_p(q), _p(k_pool), _p(v_pool), float(k_descale), float(v_descale), nb,
                                        bs * hkv * d, hkv * d, d, _p(bt), bt.shape[1], _p(sl), R, T, num_q_heads,
                                        hkv, d, bs, float(softmax_scale), req_begin, req_end, _p(out))
    _check(rc, "spec_verify_attn_fp8")
    return out


def spec_verify_partial_fp8(q, k_pool, v_pool, k_descale, v_descale, block_table, seq_lens, T, num_q_heads,
                            softmax_scale, split_tokens, max_splits, req_begin=0, req_end=None):
    q = _c(q, np.uint16)
    k_pool, v_pool = _c(k_pool, np.uint8), _c(v_pool, np.uint8)
    nb, bs, hkv, d = k_pool.shape
    bt, sl = _c(block_table, np.int32), _c(seq_lens, np.int32)
    R = bt.shape[0]
    if req_end is None:
        req_end = R
    part_o = np.zeros((max_splits, R * T, num_q_heads, d), dtype=np.float32)
    part_lse = np.full((max_splits, R * T, num_q_heads), -np.inf, dtype=np.float32)
    rc = lib().orc_spec_verify_partial_fp8(_p(q), _p(k_pool), _p(v_pool), float(k_descale), float(v_descale), nb,
                                           bs * hkv * d, hkv * d, d, _p(bt), bt.shape[1], _p(sl), R, T,
                                           num_q_heads, hkv, d, bs, float(softmax_scale), split_tokens, max_splits,
                                           req_begin, req_end, _p(part_o), _p(part_lse))
    _check(rc, "spec_verify_partial_fp8")
    return part_o, part_lse
