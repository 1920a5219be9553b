"""GPU checks of the runtime around the kernel: launch accounting, argument
errors on real tensors, and the bounded-wait failure path (no GPU fault: the
self-test kernel waits on an mbarrier nothing arrives on, gives up after a
bounded number of polls and reports ATTN_ERR_TIMEOUT; the context stays usable)."""
import math

import pytest

import attention_forward_11_gb300 as fa
from attention_forward_11_gb300 import inputs
from parity import check_full, to_device

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_and_cleared():
    assert fa.attn_check_device_status() == fa.ATTN_OK
    assert fa.attn_debug_wait_timeout(1000) == fa.ATTN_OK
    assert fa.attn_check_device_status() == fa.ATTN_ERR_TIMEOUT
    assert fa.attn_check_device_status() == fa.ATTN_OK
    # the context is still usable afterwards
    q, k, v = inputs.make_qkv(1, 256, 256, 2, 2, 128, seed=1)
    check_full(q, k, v, 1, 1 / math.sqrt(128), "after timeout self-test")


def test_last_device_status_reports_a_timeout_once():
    """The boundary's stream-less status call: it waits for the whole device,
    so it sees the self-test kernel's timeout without being given its stream."""
    import torch
    assert fa.attn_last_device_status() == fa.ATTN_OK
    side = torch.cuda.Stream()
    assert fa.attn_debug_wait_timeout(1000, side) == fa.ATTN_OK
    assert fa.attn_last_device_status() == fa.ATTN_ERR_TIMEOUT
    assert fa.attn_last_device_status() == fa.ATTN_OK
    assert fa.attn_check_device_status() == fa.ATTN_OK


def test_unit_rates_keep_an_earlier_timeout():
    """A timeout recorded before the diagnostic runs is reported by it, not wiped."""
    assert fa.attn_debug_wait_timeout(1000) == fa.ATTN_OK
    with pytest.raises(fa.AttnError) as e:
        fa.attn_debug_unit_rates()
    assert e.value.status == fa.ATTN_ERR_TIMEOUT
    assert fa.attn_last_device_status() == fa.ATTN_OK


def test_one_launch_per_call():
    import torch
    q, k, v = inputs.make_qkv(1, 256, 256, 2, 2, 128, seed=1)
    dq, dk, dv = to_device(q), to_device(k), to_device(v)
    before = fa.attn_kernel_launches()
    for _ in range(3):
        fa.attn_fwd(dq, dk, dv, causal=1)
    torch.cuda.synchronize()
    assert fa.attn_kernel_launches() - before == 3


def test_bad_tensors_raise_without_launch():
    import torch
    q = torch.zeros(1, 64, 2, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 64, 2, 128, dtype=torch.bfloat16, device="cuda")
    before = fa.attn_kernel_launches()
    with pytest.raises(fa.AttnError):
        fa.attn_fwd(q.float(), k, k)                     # wrong dtype
    with pytest.raises(fa.AttnError):
        fa.attn_fwd(q, k[:, :, :1].contiguous(), k)      # k/v shape mismatch
    with pytest.raises(fa.AttnError) as e:
        fa.attn_fwd(q[..., :32].contiguous(), k[..., :32].contiguous(), k[..., :32].contiguous())
    assert e.value.status == fa.ATTN_ERR_UNSUPPORTED
    with pytest.raises(fa.AttnError) as e:
        flat = torch.zeros(64 * 2 * 128 + 8, dtype=torch.bfloat16, device="cuda")
        mis = flat[1:1 + 64 * 2 * 128].view(1, 64, 2, 128)   # 2-byte offset: not 16-byte aligned
        fa.attn_fwd(mis, k, k)
    assert e.value.status == fa.ATTN_ERR_INVALID_ARG
    assert fa.attn_kernel_launches() == before


def test_unit_rates():
    """The measured rates the design rests on: a 128x128x16 MMA at 64 cycles from
    either operand source, N = 256 twice that, N = 64 slower than half (the
    tensor core is not fed faster at N = 64), and an exponential unit fast enough
    that one 128x128 tile's 16384 exponentials take fewer cycles than its
    sixteen 128x128x16 products (no exponential needs to move to the FMA pipe)."""
    r = fa.attn_debug_unit_rates()
    print("unit rates:", {k: round(v, 2) for k, v in r.items()})
    assert fa.attn_check_device_status() == fa.ATTN_OK
    assert r["sms"] >= 1
    for key in ("mma_ss_n128", "mma_ts_n128"):
        assert 56.0 <= r[key] <= 96.0, (key, r[key])
    assert 1.7 <= r["mma_ss_n256"] / r["mma_ss_n128"] <= 2.3
    assert r["mma_ss_n64"] > 0.5 * r["mma_ss_n128"]
    assert r["ex2_per_cycle_per_sm"] > 0.0
    assert 16384.0 / r["ex2_per_cycle_per_sm"] < 16.0 * r["mma_ss_n128"]
