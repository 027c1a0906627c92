"""Host-side checks of the C ABI, no GPU needed: libpkv.so builds for sm_103a, loads, exports every
function include/pkv.h declares, and its argument validation rejects bad calls before anything is
launched (no CUDA call is reached on these paths)."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*PKV_API\s+(?:const\s+)?\w+\s*\*?\s*(pkv_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def libpath():
    import __graft_entry__
    return __graft_entry__._build_module().build()


@pytest.fixture(scope="module")
def pkv(libpath):
    import paged_kv_cache_int64_gb300 as m
    return m


def test_header_declares_the_five_calls():
    names = declared_functions()
    for base in ("kv_int8_stats_quant", "kv_fp8_dequant_dense", "paged_prefill_attn", "spec_verify_attn_partial",
                 "spec_verify_combine"):
        assert "pkv_" + base in names


def test_library_exports_every_declared_symbol(libpath, pkv):
    names = declared_functions()
    lib = C.CDLL(libpath)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported
    # the Python binding wraps exactly the declared calls
    assert set(pkv.EXPORTED_SYMBOLS) == set(names)
    # nothing but the ABI leaks out of the library (hidden visibility)
    assert not [s for s in exported if s.startswith("_ZN3pkv")]


def test_library_targets_sm103a(libpath):
    import __graft_entry__
    assert "arch=compute_103a,code=sm_103a" in " ".join(__graft_entry__._build_module().ARCH)


def test_abi_version(pkv):
    assert pkv.lib.pkv_abi_version() == 7


def test_workspace_bytes(pkv):
    n = pkv.spec_verify_workspace_bytes(256, 16, 256, 10)
    rows = 256 * 16 * 10
    assert n >= rows * 256 * 4 + rows * 4 and n % 256 == 0
    assert pkv.spec_verify_workspace_bytes(0, 16, 256, 10) == 0


def _prefill_args(**kw):
    a = dict(q=16, k=16, v=16, nb=4, sb=16384, st=1024, sh=256, bt=16, bts=1, mb=1, sl=16, qsl=16, R=1, total_q=1,
             max_q=1, hq=16, hkv=4, d=256, bs=16, scale=0.0625, mode=0, k8=None, k8s=None, k16=None, max_ctx=0,
             out=16, ws=None, ws_bytes=0, err=None, stream=None)
    a.update(kw)
    return [a[k] for k in ("q", "k", "v", "nb", "sb", "st", "sh", "bt", "bts", "mb", "sl", "qsl", "R", "total_q",
                           "max_q", "hq", "hkv", "d", "bs", "scale", "mode", "k8", "k8s", "k16", "max_ctx", "out",
                           "ws", "ws_bytes", "err", "stream")]


@pytest.mark.parametrize("kw,status", [
    (dict(d=128), 2),                 # head_dim != 256 -> unsupported
    (dict(q=None), 1),                # null pointer
    (dict(hq=15), 2),                 # q heads not a multiple of kv heads
    (dict(bs=20), 2),                 # block_size not a multiple of 8
    (dict(q=24), 1),                  # misaligned pointer
    (dict(mode=7), 1),                # unknown qk mode
    (dict(mode=1), 1),                # int8 mode without k8 / k8_scale
    (dict(sb=-5), 1),                 # negative stride
    (dict(ws=24, ws_bytes=1 << 20), 1),  # misaligned workspace
    (dict(ws=16, ws_bytes=1000), 1),  # workspace smaller than one CTA's slots
])
def test_prefill_rejects_bad_arguments(pkv, kw, status):
    rc = pkv.lib.pkv_paged_prefill_attn(*_prefill_args(**kw))
    assert rc == status
    assert pkv.lib.pkv_last_error().decode()


def test_verify_rejects_unsupported_geometry(pkv):
    f = pkv.lib.pkv_spec_verify_attn_partial
    # a group of 33 query heads per KV head exceeds the 32 query columns of a CTA
    rc = f(16, 16, 16, 16, 16, 4, 16384, 1024, 256, 64, 4, 16, 1, 1, 16, 1, 8, 132, 4, 256, 16, 0.1, 128, 2, 16, 16,
           None, None)
    assert rc == 2 and "32" in pkv.lib.pkv_last_error().decode()
    # split_tokens not a multiple of 128
    rc = f(16, 16, 16, 16, 16, 4, 16384, 1024, 256, 64, 4, 16, 1, 1, 16, 1, 8, 16, 4, 256, 16, 0.1, 100, 2, 16, 16,
           None, None)
    assert rc == 2


def test_quant_and_dequant_reject_bad_arguments(pkv):
    rc = pkv.lib.pkv_kv_int8_stats_quant(16, 4, 16384, 1024, 256, 16, 1, 1, 16, 16, 1, 4, 16, 4, 128, 16, 16, None,
                                         8, None, None)
    assert rc == 2
    rc = pkv.lib.pkv_kv_fp8_dequant_dense(16, 16, 4, 16384, 1024, 256, None, 1, 1, 16, 1, 16, 16, 4, 256, 16, 16,
                                          16, 16, None, None)
    assert rc == 1
    rc = pkv.lib.pkv_spec_verify_combine(16, 16, 16, 1, 8, 16, 512, 128, 2, 16, None)
    assert rc == 2


def test_empty_batches_launch_nothing(pkv):
    # num_reqs == 0 returns before any CUDA call (none is available here)
    assert pkv.lib.pkv_paged_prefill_attn(*_prefill_args(R=0, total_q=0, max_q=0)) == 0
    assert pkv.lib.pkv_spec_verify_combine(16, 16, 16, 0, 8, 16, 256, 128, 2, 16, None) == 0


def _write_args(**kw):
    a = dict(kn=16, vn=16, nst=1024, bt=16, bts=1, mb=1, sl=16, qsl=16, R=1, max_q=1, dt=0, kc=16, vc=16, nb=4,
             sb=16384, st=1024, sh=256, ksc=None, vsc=None, ssb=0, sst=0, ks=None, vs=None, bs=16, hkv=4, d=256,
             err=None, stream=None)
    a.update(kw)
    return [a[k] for k in ("kn", "vn", "nst", "bt", "bts", "mb", "sl", "qsl", "R", "max_q", "dt", "kc", "vc", "nb",
                           "sb", "st", "sh", "ksc", "vsc", "ssb", "sst", "ks", "vs", "bs", "hkv", "d", "err",
                           "stream")]


@pytest.mark.parametrize("kw,status", [
    (dict(d=128), 2),                 # head_dim != 256 -> unsupported
    (dict(dt=3), 1),                  # unknown cache dtype
    (dict(kn=None), 1),               # null pointer
    (dict(dt=1), 1),                  # int8 cache without scale caches
    (dict(dt=2), 1),                  # e4m3 cache without per-tensor scales
    (dict(nst=512), 1),               # token stride shorter than a token's rows
    (dict(kc=24), 1),                 # misaligned cache
    (dict(st=1020), 1),               # stride not a multiple of 8 elements
    (dict(dt=1, ksc=16, vsc=16, ssb=64, sst=2), 1),  # scale token stride < num_kv_heads
])
def test_cache_write_rejects_bad_arguments(pkv, kw, status):
    rc = pkv.lib.pkv_kv_cache_write(*_write_args(**kw))
    assert rc == status
    assert pkv.lib.pkv_last_error().decode()


def test_cache_write_empty_batch_launches_nothing(pkv):
    assert pkv.lib.pkv_kv_cache_write(*_write_args(R=0)) == 0
    assert pkv.lib.pkv_kv_cache_write(*_write_args(max_q=0, kn=None)) == 0


def test_fused_fp8_prefill_rejects_bad_arguments(pkv):
    f = pkv.lib.pkv_paged_prefill_attn_fp8
    base = [16, 16, 16, 16, 16, 4, 16384, 1024, 256, 16, 1, 1, 16, 16, 1, 1, 1, 16, 4, 256, 16, 0.0625, 16, None, 0,
            None, None]
    bad = list(base); bad[19] = 128   # head_dim != 256
    assert f(*bad) == 2
    bad = list(base); bad[1] = None   # null K pool
    assert f(*bad) == 1
    bad = list(base); bad[7] = 1000   # token stride not 16-byte aligned
    assert f(*bad) == 1
    bad = list(base); bad[17] = 15    # q heads not a multiple of kv heads
    assert f(*bad) == 2
    bad = list(base); bad[23] = 16; bad[24] = 4096  # workspace below one CTA's slots
    assert f(*bad) == 1
    empty = list(base); empty[14] = 0  # no requests: nothing launched
    assert f(*empty) == 0


def test_prefill_workspace_bytes(pkv):
    # four slots per CTA, each 128 x 256 fp32 partial outputs and 128 fp32 log-sum-exps
    assert pkv.paged_prefill_workspace_bytes(1) == 4 * (128 * 256 + 128) * 4
    assert pkv.paged_prefill_workspace_bytes(152) == 152 * 526336
    assert pkv.paged_prefill_workspace_bytes(0) == 0


def test_noalloc_rejects_sizes_whose_product_wraps(pkv):
    """The allocation-free verify checks its partials' size one factor at a time: factors whose
    product wraps a 64-bit size around to a small number are rejected before anything launches."""
    f = pkv.lib.pkv_spec_verify_attn_noalloc
    big = (1 << 31) - 1
    for num_reqs, T, hq, splits in ((big, big, big, big), (big, 1, 1, 1), (1, 1, 1, big), (65536, 65536, 65536, 65536)):
        rc = f(16, 16, 16, 16, 16, 4, 16384, 1024, 256, 64, 4, 16, 1, 1, 16, num_reqs, T, hq, 4, 256, 16, 0.0625,
               128, splits, 16, None, None)
        assert rc == pkv.PKV_ERR_INVALID_ARG
        assert "scratch" in pkv.lib.pkv_last_error().decode()


def test_verify_pick_split(pkv):
    """The split planner (host code, no device): a multiple of 512 in [1024, 16384]; a batch that
    cannot fill the SMs is cut fine (one 20k request over 152 SMs); a large batch whose splits fill
    the SMs many times over gets a large split; its choice agrees with a brute-force evaluation of
    the same longest-first list-schedule model written out here; bad arguments give 0."""
    import heapq
    import numpy as np
    import workloads as W
    L = W.verify_batch(distinct=True, with_kv=False).seq_lens
    for T, hq in ((8, 16), (8, 24), (1, 16)):
        sp = pkv.spec_verify_pick_split(L, T, hq, 4, 152)
        assert sp % 512 == 0 and 1024 <= sp <= 16384
    assert pkv.spec_verify_pick_split([20008], 8, 16, 4, 152) <= 2048
    assert pkv.spec_verify_pick_split([20008], 8, 16, 4, 0) == 0
    assert pkv.spec_verify_pick_split([20008], 8, 16, 3, 152) == 0
    assert pkv.spec_verify_pick_split([20008], 8, 160, 4, 152) == 0

    def model(split, lens, units=4, n_sm=152, cta=7.5, tile=2.08, empty=2.0):
        ms = max((int(x) + split - 1) // split for x in lens)
        full = [split] * (sum(int(x) // split for x in lens) * units)
        part = sorted([int(x) % split for x in lens if int(x) % split] * units, reverse=True)
        sms = [0.0] * n_sm
        for k in full + part:
            t = heapq.heappop(sms)
            heapq.heappush(sms, t + cta + tile * ((k + 127) // 128))
        live = len(full) + len(part)
        for _ in range(len(lens) * ms * units - live):
            t = heapq.heappop(sms)
            heapq.heappush(sms, t + empty)
        return max(sms)
    rng = np.random.default_rng(3)
    for lens in (L, rng.integers(1000, 60000, 20), rng.integers(8, 3000, 64)):
        got = pkv.spec_verify_pick_split(lens, 8, 16, 4, 152)
        times = {sp: model(sp, lens) for sp in range(1024, 16385, 512)}
        best = min(times.values())
        assert times[got] <= best * 1.02, (got, times[got], best)
