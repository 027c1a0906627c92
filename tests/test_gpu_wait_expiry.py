"""The give-up path of the attention kernels' bounded waits, exercised without a hung kernel.

Every wait inside the prefill and verify kernels is bounded (one second by default). When one
gives up, the CTA records PKV_ERR_TIMEOUT in the caller's dev_err, waits for the TMA copies and the
MMAs it still has in flight, frees its tensor memory and exits, so the GPU context stays usable.
These tests shorten the bound of one launch to a nanosecond (pkv_testing_set_wait_limit_ns), so
the CTAs give up at their first wait that is not already satisfied - the copies they issued are
still in flight then - and check that the launch reports the timeout, and that an ordinary launch
right after it on the same GPU runs clean and gives the same bytes as before.
"""
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


from _devsetup import bf16_to_u16, dev_err, device_meta, device_pool, device_q, device_scale_pool  # noqa: E402


def _expire_then_recover(pkv, launch):
    """launch(err) enqueues one call writing its status to err and returns its output tensor."""
    err = dev_err()
    ref = bf16_to_u16(launch(err))
    torch.cuda.synchronize()
    assert err.item() == 0
    err = dev_err()
    pkv.lib.pkv_testing_set_wait_limit_ns(1)
    launch(err)
    torch.cuda.synchronize()
    assert err.item() == pkv.PKV_ERR_TIMEOUT
    err = dev_err()
    again = bf16_to_u16(launch(err))  # the limit applied to one launch only
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(again, ref)


@pytest.mark.parametrize("mode", ["bf16", "bf16_persistent", "int8_k16", "fp8_fused"])
def test_prefill_gives_up_reports_timeout_and_recovers(pkv, mode):
    kv = "e4m3" if mode == "fp8_fused" else "bf16"
    p = W.make_problem("wx", seed=81, seq_lens=[1500, 300], q_lens=[700, 300], num_blocks=120, block_size=16,
                       kv_dtype=kv)
    k, v = device_pool(p, "k"), device_pool(p, "v")
    bt, sl, qsl = device_meta(p)
    q = device_q(p)
    max_q = max(r.q_len for r in p.requests)
    ws = torch.empty(pkv.paged_prefill_workspace_bytes(), dtype=torch.uint8, device="cuda")
    scale = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    kw = {}
    if mode == "int8_k16":
        L = int(p.seq_lens.max())
        k8 = torch.zeros((p.num_reqs, L, 4, 256), dtype=torch.int8, device="cuda")
        ks = torch.zeros((p.num_reqs, L, 4), dtype=torch.float32, device="cuda")
        k16 = torch.zeros((p.num_reqs, L, 4, 256), dtype=torch.float16, device="cuda")
        pkv.kv_int8_stats_quant(k, bt, torch.zeros(p.num_reqs, dtype=torch.int32, device="cuda"), sl, L, k8, ks,
                                k16=k16)
        kw = dict(qk_mode=pkv.PKV_QK_INT8, k8_scale=ks, k16=k16)

    def launch(err):
        out = torch.full_like(q, float("nan"))
        if mode == "fp8_fused":
            pkv.paged_prefill_attn_fp8(q, k, v, scale, scale, bt, sl, qsl, max_q, p.softmax_scale, out, dev_err=err)
        else:
            pkv.paged_prefill_attn(q, None if kw else k, v, bt, sl, qsl, max_q, p.softmax_scale, out, dev_err=err,
                                   workspace=ws if mode == "bf16_persistent" else None, **kw)
        return out

    _expire_then_recover(pkv, launch)


@pytest.mark.parametrize("cache", ["int8", "e4m3"])
def test_verify_gives_up_reports_timeout_and_recovers(pkv, cache):
    T, split = 8, 512
    p = W.make_problem("wxv", seed=82, seq_lens=[L + T for L in (3000, 900, 64)], q_lens=[T] * 3, num_blocks=80,
                       block_size=64, kv_dtype=cache, softmax_scale=1.0 / 16.0)
    k, v = device_pool(p, "k"), device_pool(p, "v")
    bt, sl, _ = device_meta(p)
    q = device_q(p)
    S = pkv.splits_needed(int(p.seq_lens.max()), split)
    po = torch.empty((S, q.shape[0], 16, 256), dtype=torch.float32, device="cuda")
    pl = torch.empty((S, q.shape[0], 16), dtype=torch.float32, device="cuda")
    if cache == "int8":
        ks, vs = device_scale_pool(p, "k"), device_scale_pool(p, "v")
    else:
        ks = torch.tensor([0.5], dtype=torch.float32, device="cuda")
        vs = torch.tensor([0.75], dtype=torch.float32, device="cuda")

    def launch(err):
        out = torch.full_like(q, float("nan"))
        if cache == "int8":
            pkv.spec_verify_attn_partial(q, k, v, ks, vs, bt, sl, T, p.softmax_scale, split, po, pl, dev_err=err)
        else:
            pkv.spec_verify_attn_partial_fp8(q, k, v, ks, vs, bt, sl, T, p.softmax_scale, split, po, pl, dev_err=err)
        pkv.spec_verify_combine(po, pl, sl, T, split, out)
        return out

    _expire_then_recover(pkv, launch)
