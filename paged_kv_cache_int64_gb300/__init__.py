"""paged_kv_cache_int64_gb300 - attention over a paged KV cache with int64 block addressing, for
NVIDIA GB300 (sm_103a).

A thin Python binding over the C ABI of libpkv.so (include/pkv.h): every function here only
marshals torch tensors into pointers, strides and sizes and calls the library on the current
CUDA stream; all computation runs in the library's CUDA kernels. There is no CPU fallback: if the
library is missing or fails to load, importing this package raises.
"""
from __future__ import annotations

import ctypes as C
import math
import os

import torch

from . import _build

__all__ = [
    "PKV_OK", "PKV_ERR_INVALID_ARG", "PKV_ERR_UNSUPPORTED", "PKV_ERR_CUDA", "PKV_ERR_DEVICE_BOUNDS",
    "PKV_ERR_TIMEOUT", "PKV_QK_BF16", "PKV_QK_INT8", "PKV_KV_BF16", "PKV_KV_INT8", "PKV_KV_FP8", "PkvError", "lib",
    "library_path", "kv_cache_write", "kv_int8_stats_quant", "paged_prefill_attn_fp8", "kv_fp8_dequant_dense", "paged_prefill_attn", "paged_prefill_workspace_bytes", "spec_verify_workspace_bytes", "spec_verify_pick_split",
    "spec_verify_attn_partial", "spec_verify_attn_partial_fp8", "spec_verify_combine", "EXPORTED_SYMBOLS",
]

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA, PKV_ERR_DEVICE_BOUNDS, PKV_ERR_TIMEOUT = range(6)
PKV_QK_BF16, PKV_QK_INT8 = 0, 1
PKV_KV_BF16, PKV_KV_INT8, PKV_KV_FP8 = 0, 1, 2

EXPORTED_SYMBOLS = (
    "pkv_last_error", "pkv_abi_version", "pkv_kv_int8_stats_quant", "pkv_kv_fp8_dequant_dense",
    "pkv_paged_prefill_attn", "pkv_spec_verify_workspace_bytes", "pkv_spec_verify_attn_partial",
    "pkv_spec_verify_combine", "pkv_spec_verify_attn_partial_fp8", "pkv_spec_verify_noalloc_capacity_bytes",
    "pkv_spec_verify_attn_noalloc", "pkv_kv_cache_write", "pkv_paged_prefill_attn_fp8",
    "pkv_paged_prefill_workspace_bytes", "pkv_testing_set_wait_limit_ns", "pkv_spec_verify_pick_split",
)

library_path = _build.LIB


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pkv status {status}: {message}")
        self.status = status


def _load():
    if not os.path.exists(library_path):
        raise ImportError(f"{library_path} is missing: build it first with "
                          "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc); there is no CPU fallback")
    L = C.CDLL(library_path)
    i32, i64, f32, vp, sz = C.c_int32, C.c_int64, C.c_float, C.c_void_p, C.c_size_t
    L.pkv_last_error.restype = C.c_char_p
    L.pkv_abi_version.restype = i32
    L.pkv_testing_set_wait_limit_ns.argtypes = [C.c_uint64]
    L.pkv_testing_set_wait_limit_ns.restype = None
    L.pkv_kv_int8_stats_quant.argtypes = [vp, i64, i64, i64, i64, vp, i64, i32, vp, vp, i32, i32, i32, i32, i32,
                                          vp, vp, vp, i64, vp, vp]
    L.pkv_kv_fp8_dequant_dense.argtypes = [vp, vp, i64, i64, i64, i64, vp, i64, i32, vp, i32, i32, i32, i32, i32,
                                           vp, vp, vp, vp, vp, vp]
    L.pkv_paged_prefill_attn.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, i64, i32, vp, vp, i32, i32, i32, i32,
                                         i32, i32, i32, f32, i32, vp, vp, vp, i64, vp, vp, i64, vp, vp]
    L.pkv_paged_prefill_workspace_bytes.argtypes = [i32]
    L.pkv_paged_prefill_workspace_bytes.restype = sz
    L.pkv_spec_verify_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.pkv_spec_verify_workspace_bytes.restype = sz
    L.pkv_spec_verify_pick_split.argtypes = [vp, i32, i32, i32, i32, i32]
    L.pkv_spec_verify_pick_split.restype = i32
    L.pkv_spec_verify_attn_partial.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, i64, i32, vp,
                                               i32, i32, i32, i32, i32, i32, f32, i32, i32, vp, vp, vp, vp]
    L.pkv_spec_verify_combine.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
    L.pkv_spec_verify_attn_partial_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, vp, i64, i32, vp, i32,
                                                   i32, i32, i32, i32, i32, f32, i32, i32, vp, vp, vp, vp]
    L.pkv_spec_verify_noalloc_capacity_bytes.argtypes = []
    L.pkv_spec_verify_noalloc_capacity_bytes.restype = sz
    L.pkv_spec_verify_attn_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, i64, i32, vp,
                                               i32, i32, i32, i32, i32, i32, f32, i32, i32, vp, vp, vp]
    L.pkv_spec_verify_attn_noalloc.restype = i32
    L.pkv_kv_cache_write.argtypes = [vp, vp, i64, vp, i64, i32, vp, vp, i32, i32, i32, vp, vp, i64, i64, i64, i64,
                                     vp, vp, i64, i64, vp, vp, i32, i32, i32, vp, vp]
    L.pkv_paged_prefill_attn_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, vp, i64, i32, vp, vp, i32, i32,
                                             i32, i32, i32, i32, i32, f32, vp, vp, i64, vp, vp]
    for name in ("pkv_paged_prefill_attn_fp8", "pkv_kv_cache_write", "pkv_kv_int8_stats_quant", "pkv_kv_fp8_dequant_dense", "pkv_paged_prefill_attn",
                 "pkv_spec_verify_attn_partial", "pkv_spec_verify_combine", "pkv_spec_verify_attn_partial_fp8"):
        getattr(L, name).restype = i32
    return L


lib = _load()


def _check(status: int):
    if status != PKV_OK:
        raise PkvError(status, lib.pkv_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _cache_strides(cache: torch.Tensor):
    """[num_blocks][block_size][num_kv_heads][head_dim] view with a contiguous last dim."""
    assert cache.dim() == 4 and cache.stride(3) == 1, "cache must be [nb][bs][hkv][D] with contiguous D"
    nb, bs, hkv, d = cache.shape
    return nb, bs, hkv, d, cache.stride(0), cache.stride(1), cache.stride(2)


def _ws_bytes(ws):
    if ws is None:
        return 0
    assert ws.is_cuda and ws.is_contiguous(), "workspace must be a contiguous CUDA tensor"
    return ws.numel() * ws.element_size()


def _i32(t):
    assert t.dtype == torch.int32 and t.is_cuda, "expected a CUDA int32 tensor"
    return t


# ---------------------------------------------------------------------------------------------
# the five calls (names of the C ABI without the pkv_ prefix)
# ---------------------------------------------------------------------------------------------

def kv_cache_write(k_new, v_new, block_table, seq_lens, query_start_loc, max_q_len, k_cache, v_cache,
                   kv_dtype=PKV_KV_BF16, k_scale_cache=None, v_scale_cache=None, k_scale=None, v_scale=None,
                   dev_err=None, stream=None):
    """Store the chunk's new rows k_new / v_new (bf16 [total_q][hkv][D], token stride free) into the paged
    caches ([nb][bs][hkv][D]: bf16, int8 with fp32 scale caches [nb][bs][hkv], or uint8 e4m3 with device
    scalar scales k_scale / v_scale) at positions seq_lens[r] - q_len + i."""
    nb, bs, hkv, d, sb, st, sh = _cache_strides(k_cache)
    assert v_cache.stride() == k_cache.stride() and v_cache.shape == k_cache.shape
    want = {PKV_KV_BF16: torch.bfloat16, PKV_KV_INT8: torch.int8, PKV_KV_FP8: torch.uint8}[kv_dtype]
    assert k_cache.dtype == want and v_cache.dtype == want, f"cache dtype must be {want}"
    assert k_new.dtype == torch.bfloat16 and v_new.dtype == torch.bfloat16 and k_new.stride() == v_new.stride()
    assert k_new.dim() == 3 and k_new.stride(2) == 1 and k_new.stride(1) == d, "new rows: [total][hkv][D], heads contiguous"
    ssb = sst = 0
    if kv_dtype == PKV_KV_INT8:
        assert k_scale_cache.dtype == torch.float32 and k_scale_cache.stride() == v_scale_cache.stride()
        assert k_scale_cache.stride(2) == 1
        ssb, sst = k_scale_cache.stride(0), k_scale_cache.stride(1)
    _i32(block_table)
    R = block_table.shape[0]
    _check(lib.pkv_kv_cache_write(_ptr(k_new), _ptr(v_new), k_new.stride(0), _ptr(block_table), block_table.stride(0),
                                  block_table.shape[1], _ptr(_i32(seq_lens)), _ptr(_i32(query_start_loc)), R,
                                  int(max_q_len), int(kv_dtype), _ptr(k_cache), _ptr(v_cache), nb, sb, st, sh,
                                  _ptr(k_scale_cache), _ptr(v_scale_cache), ssb, sst, _ptr(k_scale), _ptr(v_scale), bs,
                                  hkv, d, _ptr(dev_err), _stream(stream)))


def kv_int8_stats_quant(k_cache, block_table, pos_begin, pos_end, max_tokens, k8, k8_scale, dev_err=None,
                        stream=None, k16=None):
    """Per-token-head int8 quantization of the paged bf16 K cache into k8 [R][max_ctx][hkv][D] int8 and
    k8_scale [R][max_ctx][hkv] fp32 for positions [pos_begin[r], pos_end[r]); k16 (optional, fp16, same
    shape as k8) also receives the codes as fp16 values."""
    nb, bs, hkv, d, sb, st, sh = _cache_strides(k_cache)
    assert k_cache.dtype == torch.bfloat16, "kv_int8_stats_quant reads a bf16 K cache"
    _i32(block_table)
    R = block_table.shape[0]
    assert k8.dtype == torch.int8 and k8.is_contiguous() and k8_scale.dtype == torch.float32
    _check(lib.pkv_kv_int8_stats_quant(_ptr(k_cache), nb, sb, st, sh, _ptr(block_table), block_table.stride(0),
                                       block_table.shape[1], _ptr(_i32(pos_begin)), _ptr(_i32(pos_end)), R,
                                       int(max_tokens), bs, hkv, d, _ptr(k8), _ptr(k8_scale), _ptr(k16), k8.shape[1],
                                       _ptr(dev_err), _stream(stream)))


def kv_fp8_dequant_dense(k_fp8, v_fp8, block_table, seq_lens, k_scale, v_scale, k_dense, v_dense, dev_err=None,
                         stream=None):
    """e4m3 paged K/V (uint8 [nb][bs][hkv][D]) -> dense bf16 [R][max_seq][hkv][D] for pos < seq_lens[r]."""
    nb, bs, hkv, d, sb, st, sh = _cache_strides(k_fp8)
    assert v_fp8.stride() == k_fp8.stride() and v_fp8.shape == k_fp8.shape
    assert k_fp8.dtype == torch.uint8 and v_fp8.dtype == torch.uint8, "e4m3 caches are uint8 tensors"
    _i32(block_table)
    R = block_table.shape[0]
    assert k_dense.is_contiguous() and v_dense.is_contiguous() and k_dense.dtype == torch.bfloat16
    _check(lib.pkv_kv_fp8_dequant_dense(_ptr(k_fp8), _ptr(v_fp8), nb, sb, st, sh, _ptr(block_table),
                                        block_table.stride(0), block_table.shape[1], _ptr(_i32(seq_lens)), R,
                                        k_dense.shape[1], bs, hkv, d, _ptr(k_scale), _ptr(v_scale), _ptr(k_dense),
                                        _ptr(v_dense), _ptr(dev_err), _stream(stream)))


def paged_prefill_attn(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, max_q_len, softmax_scale,
                       out, qk_mode=PKV_QK_BF16, k8=None, k8_scale=None, dev_err=None, stream=None, k16=None,
                       workspace=None):
    """Chunked causal prefill attention. q/out bf16 [total_q][Hq][D]; caches bf16 [nb][bs][hkv][D]
    (k_cache may be None in int8 mode, which reads k8 (or its fp16 copy k16) and k8_scale from
    kv_int8_stats_quant). workspace: None (one CTA per query tile) or a CUDA byte tensor of
    paged_prefill_workspace_bytes() bytes (persistent grid: full waves, last wave cut into key ranges)."""
    nb, bs, hkv, d, sb, st, sh = _cache_strides(v_cache)
    assert v_cache.dtype == torch.bfloat16 and (k_cache is None or k_cache.dtype == torch.bfloat16), \
        "paged_prefill_attn reads bf16 caches (e4m3 caches: paged_prefill_attn_fp8)"
    if k_cache is not None:
        assert k_cache.stride() == v_cache.stride() and k_cache.shape == v_cache.shape
    assert q.is_contiguous() and out.is_contiguous() and q.dtype == torch.bfloat16 and out.dtype == torch.bfloat16
    _i32(block_table)
    R = block_table.shape[0]
    max_ctx = 0 if k8 is None and k16 is None else (k8 if k8 is not None else k16).shape[1]
    _check(lib.pkv_paged_prefill_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), nb, sb, st, sh, _ptr(block_table),
                                      block_table.stride(0), block_table.shape[1], _ptr(_i32(seq_lens)),
                                      _ptr(_i32(query_start_loc)), R, q.shape[0], int(max_q_len), q.shape[1],
                                      hkv, d, bs, float(softmax_scale), int(qk_mode), _ptr(k8), _ptr(k8_scale),
                                      _ptr(k16), max_ctx, _ptr(out), _ptr(workspace), _ws_bytes(workspace),
                                      _ptr(dev_err), _stream(stream)))


def paged_prefill_attn_fp8(q, k_fp8, v_fp8, k_scale, v_scale, block_table, seq_lens, query_start_loc, max_q_len,
                           softmax_scale, out, dev_err=None, stream=None, workspace=None):
    """Chunked causal prefill attention read straight from per-tensor e4m3 paged K/V (uint8
    [nb][bs][hkv][D]) with device scalar scales; each tile is dequantized in shared memory."""
    nb, bs, hkv, d, sb, st, sh = _cache_strides(k_fp8)
    assert v_fp8.stride() == k_fp8.stride() and v_fp8.shape == k_fp8.shape
    assert k_fp8.dtype == torch.uint8 and v_fp8.dtype == torch.uint8
    assert q.is_contiguous() and out.is_contiguous() and q.dtype == torch.bfloat16 and out.dtype == torch.bfloat16
    _i32(block_table)
    R = block_table.shape[0]
    _check(lib.pkv_paged_prefill_attn_fp8(_ptr(q), _ptr(k_fp8), _ptr(v_fp8), _ptr(k_scale), _ptr(v_scale), nb, sb, st,
                                          sh, _ptr(block_table), block_table.stride(0), block_table.shape[1],
                                          _ptr(_i32(seq_lens)), _ptr(_i32(query_start_loc)), R, q.shape[0],
                                          int(max_q_len), q.shape[1], hkv, d, bs, float(softmax_scale), _ptr(out),
                                          _ptr(workspace), _ws_bytes(workspace), _ptr(dev_err), _stream(stream)))


def paged_prefill_workspace_bytes(num_ctas=None) -> int:
    """bytes of the persistent prefill workspace for num_ctas CTAs (default: the current device's SM
    count, the persistent grid's size)."""
    if num_ctas is None:
        num_ctas = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return int(lib.pkv_paged_prefill_workspace_bytes(int(num_ctas)))


def spec_verify_workspace_bytes(num_tokens, num_q_heads, head_dim, max_splits) -> int:
    return int(lib.pkv_spec_verify_workspace_bytes(num_tokens, num_q_heads, head_dim, max_splits))


def spec_verify_pick_split(seq_lens, T, num_q_heads, num_kv_heads, num_sms) -> int:
    """Host-side split_tokens choice for spec_verify_attn_partial from the batch's sequence lengths
    (host values); 0 on a bad argument."""
    import numpy as np
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    return int(lib.pkv_spec_verify_pick_split(sl.ctypes.data, int(sl.shape[0]), int(T), int(num_q_heads),
                                               int(num_kv_heads), int(num_sms)))


def spec_verify_attn_partial(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, T, softmax_scale,
                             split_tokens, part_o, part_lse, dev_err=None, stream=None):
    """Split-KV verify partials over an int8 cache ([nb][bs][hkv][D]) with fp32 per-token-head
    scales ([nb][bs][hkv]); part_o [S][R*T][Hq][D], part_lse [S][R*T][Hq] fp32."""
    nb, bs, hkv, d, sb, st, sh = _cache_strides(k_cache)
    assert k_cache.dtype == torch.int8 and v_cache.dtype == torch.int8, "int8 caches"
    assert v_cache.stride() == k_cache.stride() and k_scale.stride() == v_scale.stride()
    assert k_scale.dim() == 3 and k_scale.stride(2) == 1
    _i32(block_table)
    R = block_table.shape[0]
    max_splits = part_o.shape[0]
    _check(lib.pkv_spec_verify_attn_partial(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                            nb, sb, st, sh, k_scale.stride(0), k_scale.stride(1),
                                            _ptr(block_table), block_table.stride(0), block_table.shape[1],
                                            _ptr(_i32(seq_lens)), R, int(T), q.shape[1], hkv, d, bs,
                                            float(softmax_scale), int(split_tokens), max_splits, _ptr(part_o),
                                            _ptr(part_lse), _ptr(dev_err), _stream(stream)))


def spec_verify_attn_partial_fp8(q, k_fp8, v_fp8, k_descale, v_descale, block_table, seq_lens, T, softmax_scale,
                                 split_tokens, part_o, part_lse, dev_err=None, stream=None):
    """Split-KV verify partials over a per-tensor fp8 e4m3 cache (uint8 [nb][bs][hkv][D]); k_descale /
    v_descale: device fp32 scalars."""
    nb, bs, hkv, d, sb, st, sh = _cache_strides(k_fp8)
    assert v_fp8.stride() == k_fp8.stride()
    assert k_fp8.dtype == torch.uint8 and v_fp8.dtype == torch.uint8, "e4m3 caches are uint8 tensors"
    _i32(block_table)
    R = block_table.shape[0]
    _check(lib.pkv_spec_verify_attn_partial_fp8(_ptr(q), _ptr(k_fp8), _ptr(v_fp8), _ptr(k_descale),
                                                _ptr(v_descale), nb, sb, st, sh, _ptr(block_table),
                                                block_table.stride(0), block_table.shape[1], _ptr(_i32(seq_lens)), R,
                                                int(T), q.shape[1], hkv, d, bs, float(softmax_scale),
                                                int(split_tokens), part_o.shape[0], _ptr(part_o), _ptr(part_lse),
                                                _ptr(dev_err), _stream(stream)))


def spec_verify_combine(part_o, part_lse, seq_lens, T, split_tokens, out, stream=None):
    """Log-sum-exp merge of the partials into out bf16 [R*T][Hq][D]."""
    max_splits, rows_t, hq, d = part_o.shape
    R = seq_lens.shape[0]
    _check(lib.pkv_spec_verify_combine(_ptr(part_o), _ptr(part_lse), _ptr(_i32(seq_lens)), R, int(T), hq, d,
                                       int(split_tokens), max_splits, _ptr(out), _stream(stream)))


def splits_needed(max_seq_len: int, split_tokens: int) -> int:
    return max(1, math.ceil(max_seq_len / split_tokens))
