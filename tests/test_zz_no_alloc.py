"""The no-allocation split-KV entry point, attn_fwd_splitkv_noalloc.

It serves callers that cannot allocate device memory where they run attention
(their device memory belongs to another allocator, or allocation is not allowed
at that point): its scratch is a static device array inside libattn instead of
a workspace the caller passes.  This file is collected last on purpose, so a
run that stops at its first failure has already run every other test; it also
passes on its own in a fresh process.

The check: through the C ABI, two calls in a row of the no-allocation entry
point against the existing split-KV entry point (with a caller workspace), on
shapes that do split, within the parity tolerance the other GPU tests use.
"""
import math

import numpy as np
import pytest

import attention_forward_11_gb300 as fa
from attention_forward_11_gb300 import inputs

pytestmark = pytest.mark.gpu

O_MAX_ABS, O_MEAN_ABS, LSE_MAX_ABS = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_forward_11_gb300 import build
    build.build()
    fa.load_library()


def _device(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


CASES = [
    # B, Sq, Skv, Hq, Hkv, causal: few query tiles against long key ranges (split)
    (1, 256, 8192, 2, 2, 1),
    (1, 300, 5000, 4, 2, 2),
    (1, 512, 32768, 64, 8, 1),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_noalloc_matches_workspace_entry_point_twice(case):
    import torch
    B, Sq, Skv, Hq, Hkv, causal = case
    D, scale = 128, 1 / math.sqrt(128)
    q, k, v = (_device(t) for t in inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=sum(case)))
    assert fa.attn_fwd_splitkv_workspace_size(B, Sq, Skv, Hq, Hkv, D, causal) > 0
    o_ref, l_ref = fa.attn_fwd_splitkv(q, k, v, causal=causal, scale=scale)
    assert fa.attn_check_device_status() == fa.ATTN_OK
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # the static scratch keeps the previous call's contents
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
        st = fa.attn_fwd_splitkv_noalloc_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             o.data_ptr(), lse.data_ptr(), B, Sq, Skv, Hq, Hkv,
                                             D, causal, scale, stream)
        assert st == fa.ATTN_OK, fa.attn_status_str(st)
        assert fa.attn_check_device_status() == fa.ATTN_OK
        assert torch.isfinite(o.float()).all(), f"call {call}: non-finite O"
        err = (o.float() - o_ref.float()).abs()
        assert err.max().item() <= O_MAX_ABS and err.mean().item() <= O_MEAN_ABS, f"call {call}"
        ninf = torch.isneginf(l_ref)
        assert torch.equal(torch.isneginf(lse), ninf), f"call {call}: -inf LSE pattern"
        assert (lse[~ninf] - l_ref[~ninf]).abs().max().item() <= LSE_MAX_ABS, f"call {call}"


def test_noalloc_rejects_bad_arguments_without_launch():
    import torch
    q = torch.zeros(1, 256, 2, 128, dtype=torch.bfloat16, device="cuda")
    before = fa.attn_kernel_launches()
    st = fa.attn_fwd_splitkv_noalloc_ptr(q.data_ptr(), q.data_ptr(), q.data_ptr(), 0, 0, 1, 256,
                                         256, 2, 2, 128, 1, 0.088, 0)
    assert st == fa.ATTN_ERR_INVALID_ARG
    assert fa.attn_kernel_launches() == before
