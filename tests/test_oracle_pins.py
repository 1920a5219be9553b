"""Pins for the fp64 oracle: each test ties it to something other than itself.

The pages print no worked numeric example for the attention forward, so the
pins are closed forms, library routines, invariants of the definition and
brute force on tiny shapes.  Each is chosen so that a plausible slip in the
oracle (a dropped scale, a wrong sign, transposed operands, the wrong GQA head
mapping, a mis-aligned causal mask, a base-2 LSE, a missing max subtraction, a
missing division by the row sum) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import twin
from attention_forward_11_gb300 import inputs


def bits_from_f64(x):
    """Exact bf16 bit patterns of values that bf16 represents exactly."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    assert np.array_equal(f.astype(np.float64), x)
    b = inputs.f32_to_bf16_bits(f)
    assert np.array_equal(oracle.bf16_bits_to_f64(b), x), "value not exact in bf16"
    return b


def small_ints(rng, shape, lo=-3, hi=3):
    return bits_from_f64(rng.integers(lo, hi + 1, size=shape).astype(np.float64))


# --------------------------------------------------------------------------- rounding


def test_round_bf16_ties_to_even():
    ulp = 2.0 ** -7  # bf16 spacing in [1, 2)
    got = oracle.round_bf16([1 + ulp / 2, 1 + 1.5 * ulp, -(1 + ulp / 2), 1 + 0.75 * ulp,
                             3.0 * 2.0 ** -140, 0.6 * 2.0 ** -133, 0.0])
    assert got[0] == 1.0                 # tie -> even mantissa (0)
    assert got[1] == 1 + 2 * ulp         # tie -> even mantissa (2)
    assert got[2] == -1.0
    assert got[3] == 1 + ulp             # above the tie -> up
    assert got[4] == 0.0                 # below half the smallest subnormal step
    assert got[5] == 2.0 ** -133         # nearest subnormal grid point
    assert got[6] == 0.0


def test_round_bf16_matches_torch_and_bit_trick():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x32 = (rng.standard_normal(200_000) * np.exp(rng.uniform(-20, 20, 200_000))).astype(
        np.float32)
    # plant exact ties: fp32 values whose low 16 bits are 0x8000
    ties = (x32.view(np.uint32)[:1000] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    x32[:1000] = ties.view(np.float32)
    by_oracle = oracle.round_bf16(x32.astype(np.float64))
    by_torch = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    by_bits = oracle.bf16_bits_to_f64(inputs.f32_to_bf16_bits(x32))
    assert np.array_equal(by_oracle, by_torch)
    assert np.array_equal(by_bits, by_torch)


# --------------------------------------------------------------------------- definition


def test_hand_worked_two_keys():
    """q.k0 = 1, q.k1 = 0, scale = ln 3: weights 3/4 and 1/4 (worked by hand)."""
    D = 2
    q = bits_from_f64(np.array([1.0, 0.0]).reshape(1, 1, 1, D))
    k = bits_from_f64(np.array([[1.0, 0.0], [0.0, 5.0]]).reshape(1, 2, 1, D))
    v = bits_from_f64(np.array([[1.0, 2.0], [-1.0, 0.0]]).reshape(1, 2, 1, D))
    o, lse = oracle.attn_full(q, k, v, causal=False, scale=math.log(3.0))
    assert np.allclose(o[0, 0, 0], [0.75 * 1 + 0.25 * -1, 0.75 * 2 + 0.25 * 0], atol=1e-15)
    assert abs(lse[0, 0, 0] - math.log(4.0)) < 1e-15
    # causal, Sq = Skv = 2: row 0 sees key 0 only, row 1 sees both
    q2 = bits_from_f64(np.array([[1.0, 0.0], [1.0, 0.0]]).reshape(1, 2, 1, D))
    o2, lse2 = oracle.attn_full(q2, k, v, causal=True, scale=math.log(3.0))
    assert np.allclose(o2[0, 0, 0], [1.0, 2.0], atol=1e-15)
    assert abs(lse2[0, 0, 0] - math.log(3.0)) < 1e-15
    assert np.allclose(o2[0, 1, 0], [0.5, 1.5], atol=1e-15)


@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("Sq,Skv", [(64, 64), (16, 64), (1, 7), (40, 13)])
def test_zero_query_closed_form(causal, Sq, Skv):
    """Q = 0: every visible logit is 0, so lse = ln(#visible) and o = mean of the
    visible V rows (a cumulative mean under either causal mask); rows that see no
    key get o = 0 and lse = -inf."""
    rng = np.random.default_rng(1)
    B, Hq, Hkv, D = 2, 2, 1, 128
    q = np.zeros((B, Sq, Hq, D), dtype=np.uint16)  # +0.0 in bf16
    k = inputs.normal_bf16((B, Skv, Hkv, D), 1.0, 3, 1)
    v = inputs.normal_bf16((B, Skv, Hkv, D), 1.0, 3, 2)
    o, lse = oracle.attn_full(q, k, v, causal=causal, scale=0.37)
    vf = oracle.bf16_bits_to_f64(v)
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                n = {0: Skv, 1: min(Skv, i + Skv - Sq + 1), 2: min(Skv, i + 1)}[causal]
                if n <= 0:
                    assert np.isneginf(lse[b, h, i]) and np.all(o[b, i, h] == 0.0)
                    continue
                assert abs(lse[b, h, i] - math.log(n)) < 1e-13
                want = vf[b, :n, 0, :].mean(axis=0)
                assert np.max(np.abs(o[b, i, h] - want)) < 1e-13
    del rng


def test_constant_v_rows():
    """Weights sum to one: V rows all equal to c gives o = c on every row."""
    B, Sq, Skv, Hq, Hkv, D = 1, 33, 45, 4, 2, 128
    q, k, _ = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=5)
    c = inputs.normal_bf16((1, 1, Hkv, D), 1.0, 5, 9)
    v = np.ascontiguousarray(np.broadcast_to(c, (B, Skv, Hkv, D)))
    for causal in (False, True):
        o, _ = oracle.attn_full(q, k, v, causal=causal, scale=0.088)
        cf = oracle.bf16_bits_to_f64(c)[0, 0]
        for h in range(Hq):
            assert np.max(np.abs(o[0, :, h, :] - cf[h // 2])) < 1e-13


def test_causal_row0_is_v0():
    B, S, Hq, Hkv, D = 2, 50, 2, 2, 128
    q, k, v = inputs.make_qkv(B, S, S, Hq, Hkv, D, seed=11)
    o, lse = oracle.attn_full(q, k, v, causal=True, scale=1 / math.sqrt(D))
    vf = oracle.bf16_bits_to_f64(v)
    qf, kf = oracle.bf16_bits_to_f64(q), oracle.bf16_bits_to_f64(k)
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(o[b, 0, h], vf[b, 0, h])
            # one visible key: lse equals that single scaled logit
            s00 = float(qf[b, 0, h] @ kf[b, 0, h]) / math.sqrt(D)
            assert abs(lse[b, h, 0] - s00) < 1e-12


def test_one_hot_limit_pins_operand_roles():
    """k_j = 4 e_j, q_i = 4 e_pi(i): logits 16 on the matching key, 0 elsewhere,
    so o_i ~= v_pi(i).  A transposed QK^T or a V indexed by the query row fails."""
    D, S = 8, 8
    perm = np.array([3, 0, 7, 5, 1, 6, 2, 4])
    kf = 4.0 * np.eye(D)
    qf = 4.0 * np.eye(D)[perm]
    rng = np.random.default_rng(2)
    vf = rng.integers(-8, 9, size=(S, D)).astype(np.float64)
    q = bits_from_f64(qf.reshape(1, S, 1, D))
    k = bits_from_f64(kf.reshape(1, S, 1, D))
    v = bits_from_f64(vf.reshape(1, S, 1, D))
    o, lse = oracle.attn_full(q, k, v, causal=False, scale=1.0)
    w_other = 1.0 / (math.exp(16.0) + 7.0)
    for i in range(S):
        want = vf[perm[i]] * (1 - 7 * w_other) + w_other * (vf.sum(axis=0) - vf[perm[i]])
        assert np.max(np.abs(o[0, i, 0] - want)) < 1e-12
        assert abs(lse[0, 0, i] - (16.0 + math.log(1 + 7 * math.exp(-16.0)))) < 1e-12


def test_matches_scipy_softmax():
    """Special case reducing to library routines: scipy's softmax and logsumexp."""
    special = pytest.importorskip("scipy.special")
    B, Sq, Skv, Hq, Hkv, D = 1, 9, 13, 4, 2, 16
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=21)
    qf, kf, vf = (oracle.bf16_bits_to_f64(t) for t in (q, k, v))
    scale = 0.3
    for causal in (False, True):
        o, lse = oracle.attn_full(q, k, v, causal=causal, scale=scale)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            z = scale * np.einsum("id,jd->ij", qf[0, :, h], kf[0, :, g])
            if causal:
                z = np.where(np.tril(np.ones((Sq, Skv), bool), k=Skv - Sq), z, -np.inf)
            p = special.softmax(z, axis=1)
            assert np.max(np.abs(o[0, :, h] - p @ vf[0, :, g])) < 1e-13
            assert np.max(np.abs(lse[0, h] - special.logsumexp(z, axis=1))) < 1e-13


@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("shape", [
    (1, 1, 1, 1, 1), (1, 2, 2, 2, 1), (1, 3, 3, 2, 2), (2, 17, 17, 4, 2), (1, 64, 64, 4, 1),
    (1, 256, 256, 2, 2), (1, 17, 40, 4, 4), (1, 40, 17, 2, 1),
])
def test_brute_force_twin(shape, causal):
    B, Sq, Skv, Hq, Hkv = shape
    D = 128 if Sq * Skv < 10000 else 32
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=Sq * 7 + Skv)
    o1, l1 = oracle.attn_full(q, k, v, causal, 0.0884)
    o2, l2 = twin.attention(q, k, v, causal, 0.0884)
    assert np.array_equal(np.isneginf(l1), np.isneginf(l2))
    fin = np.isfinite(l1)
    assert np.max(np.abs(l1[fin] - l2[fin]), initial=0.0) < 1e-12
    assert np.max(np.abs(o1 - o2)) < 1e-12


def test_rows_entry_matches_full():
    B, Sq, Skv, Hq, Hkv, D = 2, 37, 37, 4, 2, 128
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=3)
    o, lse = oracle.attn_full(q, k, v, True, 0.1)
    rows = inputs.sample_rows(B, Hq, Sq, 40, seed=1)
    orr, lr = oracle.attn_rows(q, k, v, rows, True, 0.1)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(orr[n], o[b, i, h])
        assert lr[n] == lse[b, h, i]


# --------------------------------------------------------------------------- invariants


def test_gqa_head_repeat_equivalence():
    """The Pallas reference reshapes Q to (Hkv, Hq/Hkv): attention with shared
    K/V heads equals MHA with each K/V head repeated for its query group."""
    B, Sq, Skv, Hq, Hkv, D = 1, 20, 28, 8, 2, 128
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=8)
    grp = Hq // Hkv
    k_rep = np.ascontiguousarray(np.repeat(k, grp, axis=2))
    v_rep = np.ascontiguousarray(np.repeat(v, grp, axis=2))
    for causal in (False, True):
        o1, l1 = oracle.attn_full(q, k, v, causal, 0.09)
        o2, l2 = oracle.attn_full(q, k_rep, v_rep, causal, 0.09)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
        # the other plausible mapping (h % Hkv) gives a different answer
        k_tile = np.ascontiguousarray(np.tile(k, (1, 1, grp, 1)))
        v_tile = np.ascontiguousarray(np.tile(v, (1, 1, grp, 1)))
        o3, _ = oracle.attn_full(q, k_tile, v_tile, causal, 0.09)
        assert np.max(np.abs(o1 - o3)) > 1e-3


def test_bottom_right_equals_tail_of_square_causal():
    """Chunked prefill: Sq queries at the end of a Skv-long sequence see keys
    <= i + Skv - Sq; that is the last Sq rows of the square causal problem."""
    B, Skv, Sq, Hq, Hkv, D = 1, 70, 24, 4, 2, 128
    q_full, k, v = inputs.make_qkv(B, Skv, Skv, Hq, Hkv, D, seed=12)
    q_tail = np.ascontiguousarray(q_full[:, Skv - Sq:])
    o_sq, l_sq = oracle.attn_full(q_full, k, v, True, 0.09)
    o_br, l_br = oracle.attn_full(q_tail, k, v, True, 0.09)
    assert np.array_equal(o_br, o_sq[:, Skv - Sq:])
    assert np.array_equal(l_br, l_sq[:, :, Skv - Sq:])


def test_causal_is_truncated_noncausal():
    B, S, H, D = 1, 30, 2, 128
    q, k, v = inputs.make_qkv(B, S, S, H, H, D, seed=4)
    o, lse = oracle.attn_full(q, k, v, True, 0.09)
    for i in (0, 5, 29):
        kk = np.ascontiguousarray(k[:, :i + 1])
        vv = np.ascontiguousarray(v[:, :i + 1])
        qq = np.ascontiguousarray(q[:, i:i + 1])
        o1, l1 = oracle.attn_full(qq, kk, vv, False, 0.09)
        assert np.max(np.abs(o1[0, 0] - o[0, i])) < 1e-14
        assert np.max(np.abs(l1[0, :, 0] - lse[0, :, i])) < 1e-14


def test_key_permutation_invariance():
    B, Sq, Skv, H, D = 1, 11, 40, 2, 128
    q, k, v = inputs.make_qkv(B, Sq, Skv, H, H, D, seed=6)
    perm = np.random.default_rng(3).permutation(Skv)
    o1, l1 = oracle.attn_full(q, k, v, False, 0.09)
    o2, l2 = oracle.attn_full(q, np.ascontiguousarray(k[:, perm]),
                              np.ascontiguousarray(v[:, perm]), False, 0.09)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-12


def test_shift_invariance_large_logits():
    """Adding u to every key row shifts row i's logits by scale*q_i.u: o is
    unchanged and lse moves by that amount.  The shift makes the logits ~900,
    where exp overflows in fp64 unless the row maximum is subtracted."""
    rng = np.random.default_rng(9)
    B, Sq, Skv, H, D = 1, 6, 19, 1, 16
    qf = rng.integers(2, 4, size=(B, Sq, H, D)).astype(np.float64)
    kf = rng.integers(-2, 3, size=(B, Skv, H, D)).astype(np.float64)
    vf = rng.integers(-3, 4, size=(B, Skv, H, D)).astype(np.float64)
    u = np.full(D, 24.0)
    q, k, v = bits_from_f64(qf), bits_from_f64(kf), bits_from_f64(vf)
    k2 = bits_from_f64(kf + u)
    for causal in (False, True):
        o1, l1 = oracle.attn_full(q, k, v, causal, 1.0)
        o2, l2 = oracle.attn_full(q, k2, v, causal, 1.0)
        shift = qf[0, :, 0, :] @ u
        assert np.all(np.isfinite(o2)) and np.all(shift > 710)  # exp(710) overflows fp64
        assert np.max(np.abs(o1 - o2)) < 1e-12
        assert np.max(np.abs(l2[0, 0] - l1[0, 0] - shift)) < 1e-9


def test_scale_folds_into_q():
    B, Sq, Skv, H, D = 1, 8, 12, 2, 128
    rng = np.random.default_rng(10)
    qf = rng.integers(-3, 4, size=(B, Sq, H, D)).astype(np.float64)
    q = bits_from_f64(qf)
    q4 = bits_from_f64(4.0 * qf)
    _, k, v = inputs.make_qkv(B, Sq, Skv, H, H, D, seed=10)
    o1, l1 = oracle.attn_full(q4, k, v, True, 0.05)
    o2, l2 = oracle.attn_full(q, k, v, True, 0.2)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-12


def test_fully_masked_rows():
    """Causal with Sq > Skv: rows i < Sq - Skv see no key -> o = 0, lse = -inf."""
    B, Sq, Skv, H, D = 1, 10, 4, 1, 128
    q, k, v = inputs.make_qkv(B, Sq, Skv, H, H, D, seed=13)
    o, lse = oracle.attn_full(q, k, v, True, 0.09)
    assert np.all(o[0, :6] == 0.0) and np.all(np.isneginf(lse[0, 0, :6]))
    assert np.all(np.isfinite(lse[0, 0, 6:]))
    o2, l2 = twin.attention(q, k, v, True, 0.09)
    assert np.max(np.abs(o - o2)) < 1e-12


def test_merge_identity_random_chunks():
    """The kernbench page's merge of partial (m, l, o) triples, applied to any
    split of a row's keys in any tree order, reproduces the one-shot row."""
    B, Sq, Skv, Hq, Hkv, D = 1, 5, 300, 4, 2, 128
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=14, q_sigma=4.0)
    rng = np.random.default_rng(15)
    for causal in (False, True):
        o_ref, l_ref = oracle.attn_full(q, k, v, causal, 0.0884)
        for (b, h, i) in [(0, 0, 0), (0, 3, 4), (0, 1, 2)]:
            cuts = np.sort(rng.choice(np.arange(1, Skv), size=7, replace=False))
            edges = [0, *cuts.tolist(), Skv]
            parts = [oracle.partial_triple(q, k, v, causal, 0.0884, b, h, i, a, c)
                     for a, c in zip(edges[:-1], edges[1:])]
            # random tree: repeatedly merge two random neighbours
            while len(parts) > 1:
                j = int(rng.integers(0, len(parts) - 1))
                parts[j:j + 2] = [oracle.merge_triples(parts[j], parts[j + 1])]
            o, lse = oracle.finish_triple(parts[0])
            assert np.max(np.abs(o - o_ref[b, i, h])) < 1e-12
            assert abs(lse - l_ref[b, h, i]) < 1e-12


def test_merge_rule_closed_form():
    """Two single-key triples merge into the two-key softmax (sigmoid weights)."""
    t1 = (2.0, 1.0, np.array([1.0]))
    t2 = (0.5, 1.0, np.array([-3.0]))
    o, lse = oracle.finish_triple(oracle.merge_triples(t1, t2))
    w1 = 1.0 / (1.0 + math.exp(0.5 - 2.0))
    assert abs(o[0] - (w1 * 1.0 + (1 - w1) * -3.0)) < 1e-15
    assert abs(lse - math.log(math.exp(2.0) + math.exp(0.5))) < 1e-15
    empty = (-np.inf, 0.0, np.zeros(1))
    assert oracle.merge_triples(empty, t2)[0] == 0.5


def test_top_left_rules():
    """Top-left (causal=2) equals bottom-right when Sq == Skv; with Sq > Skv the
    rows i >= Skv - 1 see every key (non-causal), with Sq < Skv row i sees keys
    0..i only (the prefix problem)."""
    B, H, D = 1, 2, 128
    q, k, v = inputs.make_qkv(B, 30, 30, H, H, D, seed=31)
    assert np.array_equal(oracle.attn_full(q, k, v, 1, 0.09)[0], oracle.attn_full(q, k, v, 2, 0.09)[0])
    q, k, v = inputs.make_qkv(B, 40, 13, H, H, D, seed=32)
    o_tl, l_tl = oracle.attn_full(q, k, v, 2, 0.09)
    o_nc, l_nc = oracle.attn_full(q, k, v, 0, 0.09)
    assert np.array_equal(o_tl[:, 12:], o_nc[:, 12:]) and np.array_equal(l_tl[:, :, 12:], l_nc[:, :, 12:])
    q, k, v = inputs.make_qkv(B, 9, 50, H, H, D, seed=33)
    o_tl, l_tl = oracle.attn_full(q, k, v, 2, 0.09)
    kk, vv = np.ascontiguousarray(k[:, :9]), np.ascontiguousarray(v[:, :9])
    o_sq, l_sq = oracle.attn_full(q, kk, vv, 1, 0.09)
    assert np.array_equal(o_tl, o_sq) and np.array_equal(l_tl, l_sq)


# --------------------------------------------------------------------------- binary16 inputs


def test_f16_widening_every_finite_pattern():
    """Q = K = 0 and one key: o equals that key's V row exactly, so the oracle's
    own binary16 widening is checked against numpy's float16 for every finite
    bit pattern (both zeros, subnormals, normals up to 65504)."""
    bits = np.arange(65536, dtype=np.uint16)
    finite = np.isfinite(bits.view(np.float16))
    vrow = bits[finite]
    D = vrow.size
    q = np.zeros((1, 1, 1, D), dtype=np.uint16)
    k = np.zeros((1, 1, 1, D), dtype=np.uint16)
    v = np.ascontiguousarray(vrow.reshape(1, 1, 1, D))
    o, lse = oracle.attn_full(q, k, v, 0, 1.0, f16=True)
    want = vrow.view(np.float16).astype(np.float64)
    assert np.array_equal(o[0, 0, 0], want) and lse[0, 0, 0] == 0.0
    assert np.array_equal(oracle.f16_bits_to_f64(vrow), want)


def test_round_f16_matches_numpy():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(200_000) * np.exp(rng.uniform(-22, 12, 200_000))
    half = np.ldexp(1.0, -11)   # ties: 1 + (2k+1) 2^-11 in [1, 2)
    ties = 1.0 + (2 * rng.integers(0, 1024, 1000) + 1) * half
    x = np.concatenate([x, ties, -ties, [65504.0, 65519.9, 65520.0, 2.0 ** -25, 3 * 2.0 ** -26]])
    with np.errstate(over="ignore"):  # 65520 rounds up past the largest finite value
        want = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(oracle.round_f16(x), want)


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_f16_brute_force_twin(causal):
    B, Sq, Skv, Hq, Hkv, D = 1, 37, 50, 4, 2, 128
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=41, q_sigma=3.0, dtype="f16")
    o1, l1 = oracle.attn_full(q, k, v, causal, 0.0884, f16=True)
    o2, l2 = twin.attention(q, k, v, causal, 0.0884, f16=True)
    fin = np.isfinite(l1)
    assert np.array_equal(fin, np.isfinite(l2))
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1[fin] - l2[fin])) < 1e-12
    # the same bits read as bf16 give a different problem: the format flag matters
    o3, _ = oracle.attn_full(q, k, v, causal, 0.0884)
    assert not np.allclose(o1, o3)
