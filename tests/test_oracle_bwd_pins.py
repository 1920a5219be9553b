"""Pins for the oracle's backward (gradients of sum(dO * o)).

The pages print no numeric example of the backward pass, so each test ties the
oracle's gradients to something other than their own formulas: central finite
differences of the independent numpy forward twin, torch's float64 autograd of
the plain softmax attention, a hand-worked two-key case, closed forms at q = 0
and for constant value rows, and invariants of the softmax (shift invariance in
the keys, weights summing to one).  A dropped scale, a wrong sign of delta,
un-normalised weights, swapped operand roles or a wrong head grouping each
fails at least one of them (tests/test_oracle_mutants.py plants those slips).
"""
import math

import numpy as np
import pytest

import oracle
from oracle import twin
from attention_forward_11_gb300 import inputs


def _problem(B, Sq, Skv, Hq, Hkv, D, seed, f16=False):
    dt = "f16" if f16 else "bf16"
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=seed, dtype=dt)
    do = inputs.normal_bf16(q.shape, 1.0, seed, 3, dt)
    return q, k, v, do


def _widen(bits, f16=False):
    return oracle.f16_bits_to_f64(bits) if f16 else oracle.bf16_bits_to_f64(bits)


def _loss(qf, kf, vf, dof, causal, scale):
    o, _ = twin.attention_values(qf, kf, vf, causal, scale)
    return float((o * dof).sum())


def _finite_difference(qf, kf, vf, dof, causal, scale, h=1e-6):
    grads = []
    for which in range(3):
        args = [qf.copy(), kf.copy(), vf.copy()]
        x = args[which]
        g = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            x0 = x[idx]
            x[idx] = x0 + h
            up = _loss(*args, dof, causal, scale)
            x[idx] = x0 - h
            dn = _loss(*args, dof, causal, scale)
            x[idx] = x0
            g[idx] = (up - dn) / (2 * h)
        grads.append(g)
    return grads


@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("shape", [(1, 3, 5, 4, 2, 4), (1, 5, 3, 2, 1, 4), (2, 4, 4, 2, 2, 3)])
def test_bwd_finite_differences(shape, causal):
    """Every element of dq, dk, dv against central differences of the numpy
    twin's forward (h = 1e-6: truncation ~1e-12, rounding ~1e-9)."""
    q, k, v, do = _problem(*shape, seed=sum(shape) + causal)
    scale = 0.7
    got = oracle.attn_bwd(q, k, v, do, causal, scale)
    want = _finite_difference(_widen(q), _widen(k), _widen(v), _widen(do), causal, scale)
    for name, g, w in zip(("dq", "dk", "dv"), got, want):
        np.testing.assert_allclose(g, w, rtol=1e-6, atol=1e-6, err_msg=name)


def test_bwd_finite_differences_f16():
    q, k, v, do = _problem(1, 3, 4, 2, 1, 4, seed=7, f16=True)
    got = oracle.attn_bwd(q, k, v, do, 1, 0.5, f16=True)
    want = _finite_difference(*(_widen(t, True) for t in (q, k, v, do)), 1, 0.5)
    for name, g, w in zip(("dq", "dk", "dv"), got, want):
        np.testing.assert_allclose(g, w, rtol=1e-6, atol=1e-6, err_msg=name)


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_bwd_matches_torch_autograd(causal):
    """torch float64 autograd through softmax(scale Q K^T + mask) V, with K and V
    repeated over each head group (GQA), differentiates the definition itself."""
    torch = pytest.importorskip("torch")
    B, Sq, Skv, Hq, Hkv, D = 2, 9, 13, 4, 2, 8
    q, k, v, do = _problem(B, Sq, Skv, Hq, Hkv, D, seed=20 + causal)
    scale = 1 / math.sqrt(D)
    qt, kt, vt = (torch.tensor(_widen(t), dtype=torch.float64, requires_grad=True)
                  for t in (q, k, v))
    dot = torch.tensor(_widen(do), dtype=torch.float64)
    G = Hq // Hkv
    kk, vv = kt.repeat_interleave(G, dim=2), vt.repeat_interleave(G, dim=2)
    logits = torch.einsum("bihd,bjhd->bhij", qt, kk) * scale
    i = torch.arange(Sq)[:, None]
    j = torch.arange(Skv)[None, :]
    vis = {0: torch.ones(Sq, Skv, dtype=torch.bool), 1: j <= i + (Skv - Sq), 2: j <= i}[causal]
    logits = logits.masked_fill(~vis, float("-inf"))
    o = torch.einsum("bhij,bjhd->bihd", torch.softmax(logits, dim=-1), vv)
    (o * dot).sum().backward()
    got = oracle.attn_bwd(q, k, v, do, causal, scale)
    for name, g, t in zip(("dq", "dk", "dv"), got, (qt, kt, vt)):
        np.testing.assert_allclose(g, t.grad.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)


def test_bwd_hand_worked_two_keys():
    """One query q = 1 against keys (1, 0), values (2, 0), dO = 1, D = 1, scale ln 3:
    logits (ln 3, 0), weights (3/4, 1/4), dp = (2, 0), delta = 3/2,
    ds = (3/8, -3/8); dq = ln3 * 3/8, dk = ln3 * (3/8, -3/8), dv = (3/4, 1/4)."""
    def bits(vals):
        return inputs.f32_to_bf16_bits(np.array(vals, dtype=np.float32))
    q = bits([1.0]).reshape(1, 1, 1, 1)
    k = bits([1.0, 0.0]).reshape(1, 2, 1, 1)
    v = bits([2.0, 0.0]).reshape(1, 2, 1, 1)
    do = bits([1.0]).reshape(1, 1, 1, 1)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 0, math.log(3.0))
    l3 = math.log(3.0)
    assert dq.ravel() == pytest.approx([l3 * 3 / 8], abs=1e-15)
    assert dk.ravel() == pytest.approx([l3 * 3 / 8, -l3 * 3 / 8], abs=1e-15)
    assert dv.ravel() == pytest.approx([0.75, 0.25], abs=1e-15)


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_bwd_zero_query_closed_form(causal):
    """q = 0: every visible key of row i has weight 1/n_i, so
    dv_j = sum over the group's heads and the rows i that see j of dO_i / n_i,
    and dk = 0 (it is a sum of multiples of q)."""
    B, Sq, Skv, Hq, Hkv, D = 1, 6, 9, 4, 2, 4
    rng = np.random.default_rng(5)
    q = np.zeros((B, Sq, Hq, D), dtype=np.uint16)
    _, k, v, _ = _problem(B, Sq, Skv, Hq, Hkv, D, seed=6)
    dof = rng.integers(-4, 5, size=(B, Sq, Hq, D)).astype(np.float64)
    do = inputs.f32_to_bf16_bits(dof.astype(np.float32))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.3)
    assert np.all(dk == 0.0)
    want = np.zeros((B, Skv, Hkv, D))
    G = Hq // Hkv
    for h in range(Hq):
        for i in range(Sq):
            end = {0: Skv, 1: min(Skv, i + Skv - Sq + 1), 2: min(Skv, i + 1)}[causal]
            for j in range(max(end, 0)):
                want[0, j, h // G] += dof[0, i, h] / end
    np.testing.assert_allclose(dv, want, rtol=1e-13, atol=1e-13)


def test_bwd_constant_values_give_zero_dq_dk():
    """All value rows equal: o no longer depends on q or k, so dq = dk = 0."""
    B, Sq, Skv, Hq, Hkv, D = 1, 7, 11, 2, 1, 8
    q, k, _, do = _problem(B, Sq, Skv, Hq, Hkv, D, seed=8)
    row = inputs.normal_bf16((D,), 1.0, 8, 9)
    v = np.ascontiguousarray(np.broadcast_to(row, (B, Skv, Hkv, D)))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 1, 0.4)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    assert np.abs(dv).max() > 0.1


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_bwd_invariants(causal):
    """For any input: adding one vector to every key shifts each row's logits by
    a constant, so sum_j dk[b, j, g] = 0; the weights of a row sum to one, so
    sum_j dv[b, j, g] = sum of dO over the group's rows that see any key."""
    B, Sq, Skv, Hq, Hkv, D = 2, 10, 6, 4, 2, 8
    q, k, v, do = _problem(B, Sq, Skv, Hq, Hkv, D, seed=30 + causal)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.35)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    dof = _widen(do)
    G = Hq // Hkv
    want = np.zeros((B, Hkv, D))
    for i in range(Sq):
        end = {0: Skv, 1: min(Skv, i + Skv - Sq + 1), 2: min(Skv, i + 1)}[causal]
        if end > 0:
            for h in range(Hq):
                want[:, h // G] += dof[:, i, h]
    np.testing.assert_allclose(dv.sum(axis=1), want, rtol=1e-12, atol=1e-12)
    if causal == 1:  # Sq > Skv: rows 0..Sq-Skv-1 see no key and get no gradient
        assert np.all(dq[:, : Sq - Skv] == 0.0)


def test_bwd_gqa_equals_repeated_heads():
    """A GQA problem's dk/dv equal the per-head dk/dv of the same problem with K
    and V repeated for every query head, summed over each group."""
    B, Sq, Skv, Hq, Hkv, D = 1, 8, 8, 6, 2, 4
    q, k, v, do = _problem(B, Sq, Skv, Hq, Hkv, D, seed=40)
    G = Hq // Hkv
    krep = np.ascontiguousarray(np.repeat(k, G, axis=2))
    vrep = np.ascontiguousarray(np.repeat(v, G, axis=2))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 1, 0.5)
    dq_r, dk_r, dv_r = oracle.attn_bwd(q, krep, vrep, do, 1, 0.5)
    np.testing.assert_allclose(dq, dq_r, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dk, dk_r.reshape(B, Skv, Hkv, G, D).sum(axis=3), rtol=1e-12,
                               atol=1e-14)
    np.testing.assert_allclose(dv, dv_r.reshape(B, Skv, Hkv, G, D).sum(axis=3), rtol=1e-12,
                               atol=1e-14)


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_bwd_sampled_entry_points_match_full(causal):
    """The sampled-row dq and sampled-key dk/dv entry points (which recompute the
    row statistics their own way) equal the full gradient."""
    B, Sq, Skv, Hq, Hkv, D = 2, 12, 9, 4, 2, 8
    q, k, v, do = _problem(B, Sq, Skv, Hq, Hkv, D, seed=50 + causal)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.3)
    rows = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(Sq)]
    np.testing.assert_allclose(oracle.attn_bwd_dq_rows(q, k, v, do, rows, causal, 0.3),
                               dq.transpose(0, 2, 1, 3).reshape(-1, D)
                               [[(b * Hq + h) * Sq + i for b, h, i in rows]],
                               rtol=1e-12, atol=1e-13)
    keys = [(b, g, j) for b in range(B) for g in range(Hkv) for j in range(Skv)]
    gk, gv = oracle.attn_bwd_dkv_keys(q, k, v, do, keys, causal, 0.3)
    ref_k = np.array([dk[b, j, g] for b, g, j in keys])
    ref_v = np.array([dv[b, j, g] for b, g, j in keys])
    np.testing.assert_allclose(gk, ref_k, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(gv, ref_v, rtol=1e-11, atol=1e-13)


def test_bwd_fully_masked_rows_contribute_nothing():
    """causal = 1 with Sq > Skv: rows that see no key have dq = 0, and their dO
    changes neither dk nor dv."""
    B, Sq, Skv, Hq, Hkv, D = 1, 9, 4, 2, 2, 4
    q, k, v, do = _problem(B, Sq, Skv, Hq, Hkv, D, seed=60)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, 1, 0.5)
    do2 = do.copy()
    do2[:, : Sq - Skv] = inputs.normal_bf16((B, Sq - Skv, Hq, D), 1.0, 61, 0)
    dq2, dk2, dv2 = oracle.attn_bwd(q, k, v, do2, 1, 0.5)
    assert np.all(dq[:, : Sq - Skv] == 0.0)
    np.testing.assert_array_equal(dk, dk2)
    np.testing.assert_array_equal(dv, dv2)
    np.testing.assert_array_equal(dq, dq2)


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_bwd_supplied_delta_equal_to_exact(causal):
    """delta_i supplied as dO_i . o_i, with o the oracle forward's exact fp64 output,
    reproduces the exact gradient in every entry point (the identity
    sum_j p_ij dp_ij = dO_i . o_i); rows that see no key have o = 0."""
    B, Sq, Skv, Hq, Hkv, D = 2, 12, 9, 4, 2, 8
    q, k, v, do = _problem(B, Sq, Skv, Hq, Hkv, D, seed=70 + causal)
    o, _ = oracle.attn_full(q, k, v, causal, 0.3)
    delta = np.einsum("bihd,bihd->bhi", _widen(do), o)
    exact = oracle.attn_bwd(q, k, v, do, causal, 0.3)
    given = oracle.attn_bwd(q, k, v, do, causal, 0.3, delta=delta)
    for a, b in zip(exact, given):
        np.testing.assert_allclose(b, a, rtol=1e-10, atol=1e-13)
    rows = [(1, 3, 0), (0, 2, 5), (1, 0, Sq - 1)]
    np.testing.assert_allclose(oracle.attn_bwd_dq_rows(q, k, v, do, rows, causal, 0.3, delta=delta),
                               np.array([exact[0][b, i, h] for b, h, i in rows]), rtol=1e-10, atol=1e-13)
    keys = [(0, 1, 0), (1, 0, Skv - 1), (1, 1, 4)]
    gk, gv = oracle.attn_bwd_dkv_keys(q, k, v, do, keys, causal, 0.3, delta=delta)
    np.testing.assert_allclose(gk, np.array([exact[1][b, j, g] for b, g, j in keys]), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(gv, np.array([exact[2][b, j, g] for b, g, j in keys]), rtol=1e-10, atol=1e-13)


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_bwd_delta_shift(causal):
    """The gradients are affine in delta with the slopes of the softmax Jacobian:
    moving delta_i by e_i moves dq_i by -scale e_i sum_j p_ij k_j (the oracle's
    forward with v := k), moves dk_j by -scale sum_i p_ij e_i q_i (the exact
    backward's dv for dO_i := e_i q_i, exact in bf16 because every e_i is 0 or a
    power of two) and leaves dv unchanged.  Every entry point takes the same delta."""
    B, Sq, Skv, Hq, Hkv, D, scale = 1, 10, 7, 4, 2, 8, 0.3
    q, k, v, do = _problem(B, Sq, Skv, Hq, Hkv, D, seed=80 + causal)
    rng = np.random.default_rng(causal)
    e = rng.choice([-1.0, -0.5, 0.0, 0.25, 2.0], size=(B, Hq, Sq))
    o, _ = oracle.attn_full(q, k, v, causal, scale)
    delta = np.einsum("bihd,bihd->bhi", _widen(do), o)
    base = oracle.attn_bwd(q, k, v, do, causal, scale, delta=delta)
    moved = oracle.attn_bwd(q, k, v, do, causal, scale, delta=delta + e)
    pk, _ = oracle.attn_full(q, k, k, causal, scale)
    e_rows = e.transpose(0, 2, 1)[..., None]  # [B, Sq, Hq, 1]
    np.testing.assert_allclose(moved[0] - base[0], -scale * e_rows * pk, rtol=1e-9, atol=1e-12)
    eq = e_rows * _widen(q)
    do2 = inputs.f32_to_bf16_bits(eq.astype(np.float32))
    np.testing.assert_array_equal(_widen(do2), eq)
    _, _, dv2 = oracle.attn_bwd(q, k, v, do2, causal, scale)
    np.testing.assert_allclose(moved[1] - base[1], -scale * dv2, rtol=1e-9, atol=1e-12)
    np.testing.assert_array_equal(moved[2], base[2])
    rows = [(0, h, i) for h in range(Hq) for i in range(Sq)]
    np.testing.assert_allclose(oracle.attn_bwd_dq_rows(q, k, v, do, rows, causal, scale, delta=delta + e),
                               np.array([moved[0][b, i, h] for b, h, i in rows]), rtol=1e-10, atol=1e-13)
    keys = [(0, g, j) for g in range(Hkv) for j in range(Skv)]
    gk, _ = oracle.attn_bwd_dkv_keys(q, k, v, do, keys, causal, scale, delta=delta + e)
    np.testing.assert_allclose(gk, np.array([moved[1][b, j, g] for b, g, j in keys]), rtol=1e-10, atol=1e-13)


def test_bwd_delta_from_output_bits():
    """o= takes delta_i = sum_d dO . o from the 16-bit output, the same numbers as
    passing that sum explicitly; o and delta together are refused."""
    B, Sq, Skv, Hq, Hkv, D = 1, 6, 6, 2, 1, 8
    q, k, v, do = _problem(B, Sq, Skv, Hq, Hkv, D, seed=90)
    o, _ = oracle.attn_full(q, k, v, 1, 0.4)
    o_bits = inputs.f32_to_bf16_bits(oracle.round_bf16(o).astype(np.float32))
    d = np.einsum("bihd,bihd->bhi", _widen(do), _widen(o_bits))
    a = oracle.attn_bwd(q, k, v, do, 1, 0.4, o=o_bits)
    b = oracle.attn_bwd(q, k, v, do, 1, 0.4, delta=d)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    with pytest.raises(ValueError):
        oracle.attn_bwd(q, k, v, do, 1, 0.4, o=o_bits, delta=d)
