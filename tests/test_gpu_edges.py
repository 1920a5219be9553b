"""GPU edge cases of the attention forward: single-row queries (decode-like)
through both entry points, a very long key range, many tiny batch entries and
a single head, each against the fp64 oracle (every row, or sampled rows where
the oracle would be slow)."""
import math

import numpy as np
import pytest

import attention_forward_11_gb300 as fa
import oracle
from attention_forward_11_gb300 import inputs
from parity import check_full, check_rows, compare, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_single_query_row(causal):
    """Sq = 1 against 3000 keys: with causal=1 the row sees every key, with
    causal=2 only key 0."""
    q, k, v = inputs.make_qkv(2, 1, 3000, 8, 2, 128, seed=71)
    check_full(q, k, v, causal, 1 / math.sqrt(128), f"Sq=1 causal={causal}")


def test_single_query_row_split_kv():
    q, k, v = inputs.make_qkv(1, 1, 65536, 8, 1, 128, seed=72)
    n = fa.attn_fwd_splitkv_workspace_size(1, 1, 65536, 8, 1, 128, 1)
    assert n > 0
    o, lse = fa.attn_fwd_splitkv(to_device(q), to_device(k), to_device(v), causal=1,
                                 scale=1 / math.sqrt(128))
    assert fa.attn_check_device_status() == fa.ATTN_OK
    o_ref, l_ref = oracle.attn_full(q, k, v, 1, 1 / math.sqrt(128))
    compare(o.float().double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, l_ref, "decode")


def test_half_million_keys():
    """One query tile pair against 524288 keys (4096 KV tiles in one unit)."""
    B, Sq, Skv, H = 1, 256, 524288, 1
    q, k, v = inputs.make_qkv(B, Sq, Skv, H, H, 128, seed=73)
    rows = np.array([(0, 0, i) for i in (0, 1, 77, 128, 200, 255)], dtype=np.int64)
    check_rows(q, k, v, 1, 1 / math.sqrt(128), rows, "524288 keys")


def test_many_tiny_batch_entries():
    q, k, v = inputs.make_qkv(96, 5, 9, 2, 1, 128, seed=74)
    for causal in (0, 1, 2):
        check_full(q, k, v, causal, 1 / math.sqrt(128), f"B=96 causal={causal}")


def test_one_head_long_causal():
    q, k, v = inputs.make_qkv(1, 3000, 3000, 1, 1, 128, seed=75)
    check_full(q, k, v, 1, 1 / math.sqrt(128), "one head")
