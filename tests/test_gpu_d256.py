"""GPU parity for head size 256 (its own kernel: one 128-row query tile per
CTA, S double-buffered in tensor memory, K and V streamed as 128-column
halves): every row of small shapes -- one, two and three KV tiles (each branch
of the load order), every mask mode, ragged lengths, GQA, rows that see no key,
sharp logits that raise the running maximum -- the fp16 path, the split-KV
entry points (which run this kernel unsplit), and sampled rows at full size,
against the fp64 oracle."""
import math

import pytest

import attention_forward_11_gb300 as fa
import oracle
from attention_forward_11_gb300 import inputs
from parity import check_full, check_rows, compare, to_device

pytestmark = pytest.mark.gpu
D = 256

CASES = [
    # B, Sq, Skv, Hq, Hkv, causal, q_sigma
    (1, 128, 128, 2, 2, 0, 1.0),      # one KV tile
    (1, 200, 256, 2, 2, 0, 1.0),      # two KV tiles
    (1, 256, 300, 2, 1, 0, 1.0),      # three KV tiles, ragged key tail
    (1, 256, 256, 2, 2, 1, 1.0),
    (2, 200, 333, 4, 2, 1, 1.0),
    (1, 300, 77, 2, 2, 1, 1.0),       # Sq > Skv: rows that see no key
    (1, 384, 640, 6, 2, 2, 1.0),      # top-left
    (1, 1000, 1000, 2, 1, 0, 4.0),    # sharp logits: the running max rises
    (1, 777, 1500, 3, 3, 1, 4.0),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_d256_every_row(case):
    B, Sq, Skv, Hq, Hkv, causal, qs = case
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=int(sum(case[:6])), q_sigma=qs)
    check_full(q, k, v, causal, 1 / math.sqrt(D), str(case))


@pytest.mark.parametrize("case", CASES[3:6], ids=[str(c) for c in CASES[3:6]])
def test_d256_f16_every_row(case):
    B, Sq, Skv, Hq, Hkv, causal, qs = case
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=int(sum(case[:6])) + 1, q_sigma=qs,
                              dtype="f16")
    check_full(q, k, v, causal, 1 / math.sqrt(D), str(case), dtype="f16")


def test_d256_single_query_row():
    for causal in (0, 1, 2):
        q, k, v = inputs.make_qkv(2, 1, 700, 4, 2, D, seed=256 + causal)
        check_full(q, k, v, causal, 1 / math.sqrt(D), f"Sq=1 causal={causal}")


def test_d256_full_size_sampled_rows():
    q, k, v = inputs.make_qkv(4, 4096, 4096, 16, 16, D, seed=256)
    rows = inputs.sample_rows(4, 16, 4096, n=256, seed=256)
    check_rows(q, k, v, 1, 1 / math.sqrt(D), rows, "mha causal d256")


def test_d256_splitkv_entry_points_run_unsplit():
    B, Sq, Skv, Hq, Hkv, causal = 1, 256, 3000, 2, 2, 1
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=257)
    assert fa.attn_fwd_splitkv_workspace_size(B, Sq, Skv, Hq, Hkv, D, causal) == 0
    o_ref, l_ref = oracle.attn_full(q, k, v, causal, 1 / math.sqrt(D))
    o, lse = fa.attn_fwd_splitkv(to_device(q), to_device(k), to_device(v), causal=causal,
                                 scale=1 / math.sqrt(D))
    assert fa.attn_check_device_status() == fa.ATTN_OK
    compare(o.float().double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, l_ref, "splitkv d256")
