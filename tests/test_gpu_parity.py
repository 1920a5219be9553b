"""GPU parity: libattn's CUDA path against the fp64 oracle, element by element,
on seeded inputs -- small shapes (every row, several tiles and ragged tails,
edge cases) and the five benchmark shapes at full size (sampled rows)."""
import math

import numpy as np
import pytest

import oracle
from attention_forward_11_gb300 import inputs
from parity import check_full, check_rows, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_forward_11_gb300 import build
    build.build()


@pytest.mark.parametrize("name", ["tiny_causal", "tiny_noncausal"])
def test_tiny_workloads_every_row(name):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.make_workload(w, seed=0)
    check_full(q, k, v, w.causal, w.scale, name)


SMALL = [
    # B, Sq, Skv, Hq, Hkv, causal, q_sigma
    (1, 1, 1, 1, 1, 0, 1.0),
    (1, 1, 1, 1, 1, 1, 1.0),
    (1, 17, 17, 2, 1, 1, 1.0),          # one ragged tile, GQA group 2 (head pairs)
    (2, 200, 333, 4, 2, 0, 1.0),        # ragged Sq and Skv
    (2, 200, 333, 4, 2, 1, 1.0),        # bottom-right causal, Skv > Sq
    (1, 129, 129, 1, 1, 1, 1.0),        # one row past a tile edge
    (1, 300, 77, 2, 2, 1, 1.0),         # Sq > Skv: leading rows see no key
    (1, 384, 640, 6, 2, 1, 1.0),        # odd GQA group (3): row-tile pairs
    (1, 520, 1000, 8, 2, 1, 1.0),       # group 4, ragged
    (1, 1000, 1000, 2, 1, 0, 4.0),      # sharp softmax, running-max rescale
    (2, 640, 640, 4, 4, 1, 4.0),        # sharp + causal
    (1, 96, 4096, 4, 1, 1, 1.0),        # chunked prefill: short query block, long key range
    # more units than SMs, each with an empty tile: CTAs run several units back to back
    (1, 300, 77, 160, 160, 1, 1.0),     # row pairs: one tile of every unit sees no key
    (1, 300, 77, 320, 160, 1, 1.0),     # head pairs: whole units without any key
    (1, 17, 33, 320, 320, 0, 1.0),      # row pairs: tile 1 of every unit is past Sq
    # top-left causal (causal = 2) with Sq != Skv
    (2, 200, 333, 4, 2, 2, 1.0),
    (1, 333, 200, 4, 4, 2, 1.0),
    (1, 640, 1500, 8, 2, 2, 4.0),
]


@pytest.mark.parametrize("case", SMALL, ids=[str(c) for c in SMALL])
def test_small_shapes_every_row(case):
    B, Sq, Skv, Hq, Hkv, causal, qs = case
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, 128, seed=hash(case) % 1000, q_sigma=qs)
    check_full(q, k, v, causal, 1 / math.sqrt(128), str(case))


@pytest.mark.parametrize("scale", [0.02, 0.25, 1.0])
def test_other_scales(scale):
    q, k, v = inputs.make_qkv(1, 256, 384, 2, 2, 128, seed=5)
    check_full(q, k, v, 1, scale, f"scale={scale}")


FULL = ["mha_causal_4x16x4096", "gqa_causal_2x32x8_8192", "long_sharp_1x16x16384",
        "chunked_prefill_gqa_64x8_512x32768"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(name):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.make_workload(w, seed=0)
    rows = inputs.sample_rows(w.B, w.Hq, w.Sq, n=768, seed=1)
    check_rows(q, k, v, w.causal, w.scale, rows, name)


# ----------------------------------------------------------------- invariants on the GPU


def test_constant_v_gives_v():
    q, k, _ = inputs.make_qkv(1, 300, 500, 4, 2, 128, seed=9)
    c = inputs.normal_bf16((1, 1, 2, 128), 1.0, 9, 7)
    v = np.ascontiguousarray(np.broadcast_to(c, (1, 500, 2, 128)))
    o, _ = run_gpu(q, k, v, 1, 0.088)
    cf = oracle.bf16_bits_to_f64(c)[0, 0]
    for h in range(4):
        err = np.abs(o[0, :, h, :] - cf[h // 2])
        assert err.max() <= np.abs(cf[h // 2]).max() * 2 ** -7  # one bf16 ulp


def test_causal_row0_is_v0_exactly():
    q, k, v = inputs.make_qkv(2, 256, 256, 2, 2, 128, seed=3)
    o, lse = run_gpu(q, k, v, 1, 0.088)
    vf = oracle.bf16_bits_to_f64(v)
    assert np.array_equal(o[:, 0], vf[:, 0])


def test_gqa_equals_repeated_heads_bitwise():
    q, k, v = inputs.make_qkv(1, 384, 512, 8, 2, 128, seed=4)
    k_rep = np.ascontiguousarray(np.repeat(k, 4, axis=2))
    v_rep = np.ascontiguousarray(np.repeat(v, 4, axis=2))
    o1, l1 = run_gpu(q, k, v, 1, 0.088)
    o2, l2 = run_gpu(q, k_rep, v_rep, 1, 0.088)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_bottom_right_equals_tail_of_square_bitwise():
    q_full, k, v = inputs.make_qkv(1, 700, 700, 2, 2, 128, seed=6)
    q_tail = np.ascontiguousarray(q_full[:, 700 - 200:])
    o_sq, l_sq = run_gpu(q_full, k, v, 1, 0.088)
    o_br, l_br = run_gpu(q_tail, k, v, 1, 0.088)
    assert np.array_equal(o_br, o_sq[:, 500:]) and np.array_equal(l_br, l_sq[:, :, 500:])


def test_deterministic():
    q, k, v = inputs.make_qkv(1, 1024, 1024, 4, 4, 128, seed=8)
    a = run_gpu(q, k, v, 1, 0.088)
    b = run_gpu(q, k, v, 1, 0.088)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_lse_null_skips_lse():
    q, k, v = inputs.make_qkv(1, 256, 256, 2, 2, 128, seed=2)
    o1, _ = run_gpu(q, k, v, 1, 0.088, want_lse=False)
    o2, _ = run_gpu(q, k, v, 1, 0.088)
    assert np.array_equal(o1, o2)
