"""GPU parity for head size 64 (the kernel instantiated with one 64-column
swizzled half per row): every row of small shapes, sampled rows at full size,
the fp16 operand path and the split-KV path, against the fp64 oracle."""
import math

import pytest

import attention_forward_11_gb300 as fa
import oracle
from attention_forward_11_gb300 import inputs
from parity import check_full, check_rows, compare, to_device

pytestmark = pytest.mark.gpu
D = 64

CASES = [
    # B, Sq, Skv, Hq, Hkv, causal, q_sigma
    (1, 256, 256, 2, 2, 1, 1.0),
    (1, 256, 256, 2, 2, 0, 1.0),
    (2, 200, 333, 4, 2, 1, 1.0),
    (1, 300, 77, 2, 2, 1, 1.0),
    (1, 384, 640, 6, 2, 2, 1.0),
    (1, 1000, 1000, 2, 1, 0, 4.0),
    (1, 300, 77, 160, 160, 1, 1.0),   # more units than SMs, empty tiles
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_d64_every_row(case):
    B, Sq, Skv, Hq, Hkv, causal, qs = case
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=int(sum(case[:6])), q_sigma=qs)
    check_full(q, k, v, causal, 1 / math.sqrt(D), str(case))


@pytest.mark.parametrize("case", CASES[:4], ids=[str(c) for c in CASES[:4]])
def test_d64_f16_every_row(case):
    B, Sq, Skv, Hq, Hkv, causal, qs = case
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=int(sum(case[:6])) + 1, q_sigma=qs,
                              dtype="f16")
    check_full(q, k, v, causal, 1 / math.sqrt(D), str(case), dtype="f16")


def test_d64_full_size_sampled_rows():
    q, k, v = inputs.make_qkv(4, 4096, 4096, 16, 16, D, seed=64)
    rows = inputs.sample_rows(4, 16, 4096, n=512, seed=64)
    check_rows(q, k, v, 1, 1 / math.sqrt(D), rows, "mha causal d64")


# shapes the planner splits (few query tiles against many KV tiles)
@pytest.mark.parametrize("case", [(1, 256, 8192, 2, 2, 1), (1, 2048, 4096, 2, 2, 2)],
                         ids=["br", "tl"])
def test_d64_splitkv_every_row(case):
    B, Sq, Skv, Hq, Hkv, causal = case
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=sum(case))
    assert fa.attn_fwd_splitkv_workspace_size(B, Sq, Skv, Hq, Hkv, D, causal) > 0
    o, lse = fa.attn_fwd_splitkv(to_device(q), to_device(k), to_device(v), causal=causal,
                                 scale=1 / math.sqrt(D))
    assert fa.attn_check_device_status() == fa.ATTN_OK
    o_ref, l_ref = oracle.attn_full(q, k, v, causal, 1 / math.sqrt(D))
    compare(o.float().double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, l_ref, str(case))
