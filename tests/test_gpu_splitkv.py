"""GPU parity of the split-KV path (attn_fwd_splitkv): pieces of a query-tile
pair's KV range computed on different SMs and merged by the kernbench page's
(m, l, O) rule, against the fp64 oracle; plus its workspace contract."""
import math

import numpy as np
import pytest
import torch

import attention_forward_11_gb300 as fa
from attention_forward_11_gb300 import inputs
from parity import compare, run_gpu, to_device
import oracle

pytestmark = pytest.mark.gpu


def run_split(q, k, v, causal, scale):
    dq, dk, dv = to_device(q), to_device(k), to_device(v)
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    n = fa.attn_fwd_splitkv_workspace_size(B, Sq, Skv, Hq, Hkv, D, causal)
    o, lse = fa.attn_fwd_splitkv(dq, dk, dv, causal=causal, scale=scale)
    assert fa.attn_check_device_status() == fa.ATTN_OK
    return n, o.float().double().cpu().numpy(), lse.double().cpu().numpy()


SPLIT_CASES = [
    # B, Sq, Skv, Hq, Hkv, causal, q_sigma, split?   (few query tiles, long key ranges;
    # "split?" is the planner's choice: short key ranges keep the whole-unit schedule)
    (1, 256, 8192, 2, 2, 0, 1.0, True),
    (1, 256, 8192, 2, 2, 1, 1.0, True),
    (1, 256, 8192, 2, 2, 2, 1.0, False),   # top-left: each row sees <= 256 keys
    (1, 2048, 4096, 2, 2, 2, 1.0, True),   # top-left, long
    (1, 300, 5000, 4, 2, 1, 4.0, True),    # ragged, GQA head pairs, sharp softmax
    (1, 300, 77, 2, 2, 1, 1.0, False),     # rows that see no key
    (2, 200, 3333, 4, 2, 2, 1.0, False),   # top-left with Skv > Sq
    (1, 96, 20000, 8, 1, 1, 1.0, True),    # odd group (row pairs), chunked prefill
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=[str(c[:7]) for c in SPLIT_CASES])
def test_splitkv_every_row(case):
    B, Sq, Skv, Hq, Hkv, causal, qs, split = case
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, 128, seed=int(sum(case[:6])), q_sigma=qs)
    scale = 1 / math.sqrt(128)
    n, o, lse = run_split(q, k, v, causal, scale)
    o_ref, l_ref = oracle.attn_full(q, k, v, causal, scale)
    compare(o, lse, o_ref, l_ref, str(case))
    assert (n > 0) == split, f"planner split={n > 0}, expected {split}"


def test_splitkv_chunked_prefill_sampled_rows():
    """The chunked-prefill benchmark shape: 128 units of equal length on 152 SMs.
    The planner keeps the whole-unit schedule there (splitting measured slower:
    the shares lose the L2 sharing of each K/V tile among a head's units), so the
    entry point runs exactly what attn_fwd runs."""
    w = inputs.WORKLOADS["chunked_prefill_gqa_64x8_512x32768"]
    q, k, v = inputs.make_workload(w, seed=0)
    n, o, lse = run_split(q, k, v, w.causal, w.scale)
    assert n == 0
    rows = inputs.sample_rows(w.B, w.Hq, w.Sq, n=768, seed=3)
    o_ref, l_ref = oracle.attn_rows(q, k, v, rows, w.causal, w.scale)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    compare(o[b, i, h, :], lse[b, h, i], o_ref, l_ref, "chunked prefill split-KV")


@pytest.mark.parametrize("shape", [(1, 128, 32768, 64, 8), (1, 1, 65536, 8, 1)],
                         ids=["prefill_chunk_128", "decode_row"])
def test_splitkv_long_keys_split_sampled_rows(shape):
    """Few query tiles against long key ranges: the planner splits, at full size."""
    B, Sq, Skv, Hq, Hkv = shape
    scale = 1 / math.sqrt(128)
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, 128, seed=Sq + Hq)
    n, o, lse = run_split(q, k, v, 1, scale)
    assert n > 0, "expected the problem to be split"
    rows = inputs.sample_rows(B, Hq, Sq, n=min(512, B * Hq * Sq), seed=5)
    o_ref, l_ref = oracle.attn_rows(q, k, v, rows, 1, scale)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    compare(o[b, i, h, :], lse[b, h, i], o_ref, l_ref, f"split-KV {shape}")


def test_splitkv_matches_unsplit_closely():
    q, k, v = inputs.make_qkv(1, 512, 16384, 4, 4, 128, seed=7)
    _, o_s, l_s = run_split(q, k, v, 1, 0.088)
    o_p, l_p = run_gpu(q, k, v, 1, 0.088)
    assert np.max(np.abs(o_s - o_p)) <= 2 ** -7 + 1e-6   # at most about one bf16 ulp apart
    assert np.max(np.abs(l_s - l_p)) <= 1e-4


def test_splitkv_large_problem_needs_no_workspace():
    assert fa.attn_fwd_splitkv_workspace_size(4, 4096, 4096, 16, 16, 128, 1) == 0


def test_splitkv_rejects_short_workspace():
    q, k, v = (to_device(t) for t in inputs.make_qkv(1, 256, 8192, 2, 2, 128, seed=1))
    n = fa.attn_fwd_splitkv_workspace_size(1, 256, 8192, 2, 2, 128, 1)
    assert n > 0
    ws = torch.empty(n - 256, dtype=torch.uint8, device="cuda")
    before = fa.attn_kernel_launches()
    with pytest.raises(fa.AttnError) as e:
        fa.attn_fwd_splitkv(q, k, v, causal=1, workspace=ws)
    assert e.value.status == fa.ATTN_ERR_INVALID_ARG
    assert fa.attn_kernel_launches() == before
