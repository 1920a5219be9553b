"""The no-allocation split-KV entry point, attn_fwd_splitkv_noalloc.

It serves callers that cannot allocate device memory where they run attention
(their device memory belongs to another allocator, or allocation is not allowed
at that point): its scratch is a static device array inside libattn instead of
a workspace the caller passes.  This file is collected last on purpose, so a
run that stops at its first failure has already run every other test; it also
passes on its own in a fresh process.

The checks, through the C ABI, two calls in a row each: the no-allocation entry
point runs the same plan and the same kernels as attn_fwd_splitkv with a caller
workspace, so its O and LSE must be bit-identical to that entry point's, and it
must launch the same kernels (two when the plan splits: the split forward and
the combine; one when it does not).  One shape is also compared with the fp64
oracle directly, and one takes the no-split fallback.
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
    # B, Sq, Skv, Hq, Hkv, D, causal: few query tiles against long key ranges (split) ...
    (1, 256, 8192, 2, 2, 128, 1),
    (1, 300, 5000, 4, 2, 128, 2),
    (1, 256, 6000, 4, 4, 64, 0),
    (1, 512, 32768, 64, 8, 128, 1),
    # ... and one with more units than the split plan takes: the plain schedule, no scratch
    (9, 2048, 2048, 16, 16, 64, 1),
]


def _noalloc(q, k, v, B, Sq, Skv, Hq, Hkv, D, causal, scale):
    import torch
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    before = fa.attn_kernel_launches()
    st = fa.attn_fwd_splitkv_noalloc_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), B, Sq, Skv, Hq, Hkv, D, causal, scale,
                                         stream)
    assert st == fa.ATTN_OK, fa.attn_status_str(st)
    launched = fa.attn_kernel_launches() - before
    assert fa.attn_check_device_status() == fa.ATTN_OK
    return o, lse, launched


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_noalloc_matches_workspace_entry_point_twice(case):
    import torch
    B, Sq, Skv, Hq, Hkv, D, causal = case
    scale = 1 / math.sqrt(D)
    q, k, v = (_device(t) for t in inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=sum(case)))
    ws = fa.attn_fwd_splitkv_workspace_size(B, Sq, Skv, Hq, Hkv, D, causal)
    before = fa.attn_kernel_launches()
    o_ref, l_ref = fa.attn_fwd_splitkv(q, k, v, causal=causal, scale=scale)
    expected_launches = fa.attn_kernel_launches() - before
    assert expected_launches == (2 if ws > 0 else 1)
    assert fa.attn_check_device_status() == fa.ATTN_OK
    for call in range(2):  # the static scratch keeps the previous call's contents
        o, lse, launched = _noalloc(q, k, v, B, Sq, Skv, Hq, Hkv, D, causal, scale)
        assert launched == expected_launches, f"call {call}: {launched} kernels launched"
        assert torch.equal(o, o_ref), f"call {call}: O differs from attn_fwd_splitkv"
        assert torch.equal(lse, l_ref), f"call {call}: LSE differs from attn_fwd_splitkv"


def test_noalloc_takes_the_plain_schedule_when_nothing_splits():
    import torch
    B, Sq, Skv, Hq, Hkv, D, causal = CASES[-1]
    assert fa.attn_fwd_splitkv_workspace_size(B, Sq, Skv, Hq, Hkv, D, causal) == 0
    q, k, v = (_device(t) for t in inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=5))
    o_ref, l_ref = fa.attn_fwd(q, k, v, causal=causal, scale=1 / math.sqrt(D))
    o, lse, launched = _noalloc(q, k, v, B, Sq, Skv, Hq, Hkv, D, causal, 1 / math.sqrt(D))
    assert launched == 1
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_noalloc_against_the_oracle():
    import oracle
    B, Sq, Skv, Hq, Hkv, D, causal = 1, 300, 5000, 4, 2, 128, 1
    scale = 1 / math.sqrt(D)
    qb, kb, vb = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=11, q_sigma=4.0)
    assert fa.attn_fwd_splitkv_workspace_size(B, Sq, Skv, Hq, Hkv, D, causal) > 0
    q, k, v = _device(qb), _device(kb), _device(vb)
    o_ref, l_ref = oracle.attn_full(qb, kb, vb, causal, scale)
    o_ref = oracle.round_bf16(o_ref)
    for call in range(2):
        o, lse, _ = _noalloc(q, k, v, B, Sq, Skv, Hq, Hkv, D, causal, scale)
        err = np.abs(o.float().double().cpu().numpy() - o_ref)
        assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, f"call {call}"
        l64 = lse.double().cpu().numpy()
        ninf = np.isneginf(l_ref)
        assert np.array_equal(np.isneginf(l64), ninf), f"call {call}: -inf LSE pattern"
        assert np.abs(l64[~ninf] - l_ref[~ninf]).max() <= LSE_MAX_ABS, f"call {call}"


def test_noalloc_rejects_bad_arguments_without_launch():
    import torch
    q = torch.zeros(1, 256, 2, 128, dtype=torch.bfloat16, device="cuda")
    before = fa.attn_kernel_launches()
    st = fa.attn_fwd_splitkv_noalloc_ptr(q.data_ptr(), q.data_ptr(), q.data_ptr(), 0, 0, 1, 256,
                                         256, 2, 2, 128, 1, 0.088, 0)
    assert st == fa.ATTN_ERR_INVALID_ARG
    assert fa.attn_kernel_launches() == before
