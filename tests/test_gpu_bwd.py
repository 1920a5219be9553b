"""GPU parity of the backward pass (attn_bwd, through the C ABI) against the fp64
oracle's gradients of sum(dO * O).

Reference.  attn_bwd forms delta_i = sum_d dO * O from the 16-bit O it is
given, as the Pallas page's backward takes delta from its stored `out`.  The
tests therefore compare with the oracle's gradient for that same delta
(`oracle.attn_bwd(..., o=...)`, pinned against the exact gradient by the
delta-identity and delta-shift pins).  The exact gradient differs from it by
the rounding of O itself: dq_i moves by -scale * ddelta_i * sum_j p_ij k_j,
with ddelta_i = sum_d dO * (O - o_exact), and dk by the matching sum over
rows.  That term is largest in rows that see two or three keys, where nothing
averages it down.  On the full headline shape it reaches 47 u rms of dq.
test_bwd_after_gpu_forward compares the forward-then-backward pipeline with
the exact gradient on shapes where it stays within the bound below.

Tolerance.  With u the unit roundoff of the element type (2^-8 for bf16,
2^-11 for binary16) and rms the root-mean-square of the oracle's gradient tensor
over the compared elements it does not make exactly zero:
    mean |g - g_oracle| <= 1 u rms      |g - g_oracle| <= 40 u rms + 2 u |g_oracle|
The kernels round P and dS to the element type before each product and the
outputs once at the end.  Each of those roundings moves one term of a
gradient sum by at most u of itself, so the error of an element is a sum of
many independent terms of size <= u |term|.  Its mean over a tensor stays
below u rms, and the largest of ~10^8 elements stays below 40 u rms, plus 2 u
of the element itself for the output's own rounding and a dominant term's
(elements far above the rms, as in a sparse dv, round on their own scale).
A wrong scale, sign, delta or mask moves elements by O(rms), hundreds of u.

Inputs.  Most cases hand attn_bwd the oracle's O (correctly rounded) and LSE,
so they test the backward kernels alone; the pipeline and full-size sampled
tests take O and LSE from attn_fwd.
"""
import math

import numpy as np
import pytest

import oracle
from attention_forward_11_gb300 import inputs
from parity import to_device

pytestmark = pytest.mark.gpu

U = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}
MEAN_U, MAX_U, REL_U = 1.0, 40.0, 2.0
FLOOR = 0.02  # fraction of one term's size below which a tensor's rms is not trusted


def problem(B, Sq, Skv, Hq, Hkv, D, seed, dtype="bf16"):
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=seed, dtype=dtype)
    do = inputs.normal_bf16(q.shape, 1.0, seed, 3, dtype)
    return q, k, v, do


def oracle_forward_bits(q, k, v, causal, scale, dtype="bf16"):
    """The forward's outputs as attn_bwd takes them, from the oracle: O correctly
    rounded to the element type (16-bit patterns) and the fp32 LSE."""
    o, lse = oracle.attn_full(q, k, v, causal, scale, f16=dtype == "f16")
    if dtype == "f16":
        o_bits = oracle.round_f16(o).astype(np.float16).view(np.uint16)
    else:
        o_bits = inputs.f32_to_bf16_bits(oracle.round_bf16(o).astype(np.float32))
    return np.ascontiguousarray(o_bits), lse.astype(np.float32)


def gpu_grads(q, k, v, do, causal, scale, dtype="bf16", raw=False, fwd="oracle", want_o=False):
    """dq, dk, dv from attn_bwd (fp64 numpy, or the device tensors with raw=True).
    fwd="oracle": O and LSE are the oracle's (O correctly rounded), which tests
    the backward kernels on exact inputs; fwd="gpu": they come from attn_fwd, the
    pipeline a training step runs.  want_o: also return the 16-bit O patterns
    attn_bwd was given (numpy uint16, q's layout)."""
    import torch
    import attention_forward_11_gb300 as fa
    tq, tk, tv, tdo = (to_device(x, dtype) for x in (q, k, v, do))
    if fwd == "gpu":
        o, lse = fa.attn_fwd(tq, tk, tv, causal=int(causal), scale=scale)
        o_bits = o.view(torch.int16).cpu().numpy().view(np.uint16) if want_o else None
    else:
        o_bits, lse_np = oracle_forward_bits(q, k, v, causal, scale, dtype)
        o, lse = to_device(o_bits, dtype), torch.from_numpy(lse_np).cuda()
    dq, dk, dv = fa.attn_bwd(tq, tk, tv, o, lse, tdo, causal=int(causal), scale=scale)
    assert fa.attn_check_device_status() == fa.ATTN_OK
    if raw:
        return dq, dk, dv
    out = tuple(t.float().double().cpu().numpy() for t in (dq, dk, dv))
    torch.cuda.synchronize()
    return (out, o_bits) if want_o else out


def term_sizes(q, k, v, do, scale, dtype="bf16"):
    """Natural size of one term of each gradient sum, from the inputs: a dS K
    term of dq is ~ scale |dP| |k| with |dP| ~ sqrt(D) |dO| |v| (likewise dk with
    |q|); a term of dv is ~ |dO|."""
    w = oracle.f16_bits_to_f64 if dtype == "f16" else oracle.bf16_bits_to_f64
    rq, rk, rv, rdo = (float(np.sqrt(np.mean(w(x) ** 2))) for x in (q, k, v, do))
    dp = math.sqrt(q.shape[-1]) * rdo * rv
    return scale * dp * rk, scale * dp * rq, rdo


def compare(got, ref, dtype, what, terms):
    """Errors are measured against each tensor's rms over its support (the
    elements the oracle does not make exactly zero: keys no row sees and rows
    that see no key are structural zeros, and a tensor that is mostly such zeros
    would otherwise have a diluted rms), floored at 2 % of the size of one term
    of its sums (`terms`).  Outside the support the result must be within the
    same bound of zero.  With dO = 0 every gradient must be exactly zero.
    Returns {name: (mean error, largest excess over 2 u |ref|)} in units of u rms."""
    u = U[dtype]
    stats = {}
    for name, g, r, term in zip(("dq", "dk", "dv"), got, ref, terms):
        assert np.all(np.isfinite(g)), f"{what} {name}: non-finite"
        if term == 0.0:
            assert np.all(g == 0.0), f"{what} {name}: expected zeros"
            continue
        sup = r != 0.0
        rms = float(np.sqrt(np.mean(r[sup] ** 2))) if sup.any() else 0.0
        norm = max(rms, FLOOR * term)
        err = np.abs(g - r)
        if sup.any():
            e = err[sup]
            assert e.mean() <= MEAN_U * u * norm, f"{what} {name}: mean err {e.mean() / norm:.3e} rms"
        excess = err - REL_U * u * np.abs(r)
        assert excess.max() <= MAX_U * u * norm, f"{what} {name}: max err {excess.max() / norm:.3e} rms"
        stats[name] = (float(err[sup].mean() / (u * norm)) if sup.any() else 0.0,
                       float(excess.max() / (u * norm)))
    return stats


def check(q, k, v, do, causal, scale, what, dtype="bf16", fwd="oracle", exact=False):
    """Every element against the oracle: the gradient for the delta of the O
    attn_bwd was given, or (exact=True) the exact gradient."""
    got, o_bits = gpu_grads(q, k, v, do, causal, scale, dtype=dtype, fwd=fwd, want_o=True)
    ref = oracle.attn_bwd(q, k, v, do, causal, scale, f16=dtype == "f16", o=None if exact else o_bits)
    return compare(got, ref, dtype, what, term_sizes(q, k, v, do, scale, dtype))


CASES = [
    # B, Sq, Skv, Hq, Hkv, D, causal
    (1, 256, 256, 2, 2, 128, 0),
    (1, 256, 256, 2, 2, 128, 1),
    (1, 300, 300, 4, 2, 128, 1),      # ragged tail, GQA group 2
    (2, 200, 333, 4, 1, 128, 1),      # Sq < Skv, bottom-right, group 4
    (1, 333, 200, 2, 1, 128, 1),      # Sq > Skv: rows that see no key
    (1, 200, 333, 2, 2, 128, 2),      # top-left, keys no row sees
    (1, 129, 517, 3, 3, 128, 0),
    (1, 1000, 1000, 2, 1, 128, 0),
    (1, 384, 384, 2, 2, 64, 1),       # head size 64
    (1, 250, 390, 4, 2, 64, 2),
    (1, 256, 256, 2, 2, 256, 0),      # head size 256: the dV, dK and dQ launches
    (1, 300, 300, 4, 2, 256, 1),
    (2, 200, 333, 4, 1, 256, 1),
    (1, 333, 200, 2, 1, 256, 1),
    (1, 200, 333, 2, 2, 256, 2),
    (1, 1000, 700, 2, 2, 256, 0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_Sq{}_Skv{}_H{}-{}_D{}_c{}".format(*c))
def test_bwd_matches_oracle(case):
    *shape, causal = case
    q, k, v, do = problem(*shape, seed=sum(case))
    scale = 1 / math.sqrt(shape[5])
    check(q, k, v, do, causal, scale, str(case))


@pytest.mark.parametrize("case", [(1, 256, 256, 2, 2, 128, 1), (2, 200, 333, 4, 1, 128, 1),
                                  (1, 1000, 1000, 2, 1, 128, 0), (1, 384, 384, 2, 2, 64, 1),
                                  (1, 384, 384, 2, 2, 256, 1)],
                         ids=lambda c: "B{}_Sq{}_Skv{}_H{}-{}_D{}_c{}".format(*c))
def test_bwd_after_gpu_forward(case):
    """O and LSE from attn_fwd, as a training step runs them, against the exact
    gradient (O's rounding included in the error) and against the gradient for
    the delta of that O."""
    *shape, causal = case
    q, k, v, do = problem(*shape, seed=sum(case) + 1)
    check(q, k, v, do, causal, 1 / math.sqrt(shape[5]), str(case), fwd="gpu", exact=True)
    check(q, k, v, do, causal, 1 / math.sqrt(shape[5]), str(case), fwd="gpu")


@pytest.mark.parametrize("case", [(1, 300, 300, 2, 1, 128, 1), (1, 200, 260, 2, 2, 64, 0),
                                  (1, 250, 300, 2, 1, 256, 1)])
def test_bwd_f16_matches_oracle(case):
    *shape, causal = case
    q, k, v, do = problem(*shape, seed=sum(case), dtype="f16")
    scale = 1 / math.sqrt(shape[5])
    check(q, k, v, do, causal, scale, str(case), dtype="f16")


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("causal", [0, 1, 2])
@pytest.mark.parametrize("Sq,Skv", [(1, 300), (300, 1), (1, 1), (7, 5)])
def test_bwd_degenerate_lengths(Sq, Skv, causal, D):
    q, k, v, do = problem(2, Sq, Skv, 4, 2, D, seed=Sq + 3 * Skv + causal + D)
    scale = 0.125
    check(q, k, v, do, causal, scale, f"Sq={Sq} Skv={Skv} causal={causal} D={D}")


@pytest.mark.parametrize("D", [128, 256])
def test_bwd_many_tiny_batch_entries(D):
    q, k, v, do = problem(64, 5, 9, 2, 1, D, seed=81)
    for causal in (0, 1, 2):
        check(q, k, v, do, causal, 0.1, f"B=64 causal={causal} D={D}")


@pytest.mark.parametrize("D", [128, 256])
def test_bwd_exact_zeros(D):
    """Keys that no row sees (top-left mask, Skv > Sq) get dk = dv = 0 exactly;
    rows that see no key (bottom-right mask, Sq > Skv) get dq = 0 exactly."""
    q, k, v, do = problem(1, 130, 400, 2, 1, D, seed=82)
    dq, dk, dv = gpu_grads(q, k, v, do, 2, 0.1)
    assert np.all(dk[:, 130:] == 0.0) and np.all(dv[:, 130:] == 0.0)
    assert np.abs(dk[:, :130]).max() > 0 and np.abs(dv[:, :130]).max() > 0
    q, k, v, do = problem(1, 400, 130, 2, 1, D, seed=83)
    dq, dk, dv = gpu_grads(q, k, v, do, 1, 0.1)
    assert np.all(dq[:, : 400 - 130] == 0.0)
    assert np.abs(dq[:, 400 - 130:]).max() > 0


@pytest.mark.parametrize("D", [128, 256])
def test_bwd_zero_output_gradient(D):
    q, k, v, do = problem(1, 300, 300, 2, 2, D, seed=84)
    do = np.zeros_like(do)
    for g in gpu_grads(q, k, v, do, 1, 0.1):
        assert np.all(g == 0.0)


@pytest.mark.parametrize("D", [128, 256])
def test_bwd_is_deterministic(D):
    """No atomics: two calls give bit-identical gradients."""
    import torch
    q, k, v, do = problem(2, 700, 700, 4, 2, D, seed=85)
    a = gpu_grads(q, k, v, do, 1, 0.1, raw=True)
    b = gpu_grads(q, k, v, do, 1, 0.1, raw=True)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def _sampled(shape, causal, seed, n_rows, kv_pairs, dtype="bf16"):
    B, Sq, Skv, Hq, Hkv, D = shape
    q, k, v, do = problem(*shape, seed=seed, dtype=dtype)
    scale = 1 / math.sqrt(D)
    (dq, dk, dv), o_bits = gpu_grads(q, k, v, do, causal, scale, dtype=dtype, fwd="gpu", want_o=True)
    rows = inputs.sample_rows(B, Hq, Sq, n_rows, seed)
    ref_dq = oracle.attn_bwd_dq_rows(q, k, v, do, rows, causal, scale, f16=dtype == "f16", o=o_bits)
    got_dq = np.array([dq[b, i, h] for b, h, i in rows])
    rng = np.random.default_rng(seed)
    keys = []
    for b, g in kv_pairs:
        js = {0, 1, 127, 128, Skv // 2, Skv - 129, Skv - 128, Skv - 1}
        js.update(rng.integers(0, Skv, 12).tolist())
        keys += [(b, g, j) for j in sorted(js) if 0 <= j < Skv]
    ref_dk, ref_dv = oracle.attn_bwd_dkv_keys(q, k, v, do, keys, causal, scale, f16=dtype == "f16",
                                              o=o_bits)
    got_dk = np.array([dk[b, j, g] for b, g, j in keys])
    got_dv = np.array([dv[b, j, g] for b, g, j in keys])
    compare((got_dq, got_dk, got_dv), (ref_dq, ref_dk, ref_dv), dtype, f"{shape} sampled",
            term_sizes(q, k, v, do, scale, dtype))


def test_bwd_headline_shape_sampled():
    """B=4, H=16, S=4096, D=128, causal (the forward's headline shape): sampled
    dq rows and dk/dv keys of two (batch, head) pairs against the oracle."""
    _sampled((4, 4096, 4096, 16, 16, 128), 1, seed=86, n_rows=48, kv_pairs=[(0, 0), (3, 15)])


def test_bwd_headline_shape_every_element():
    """The same shape with every element of dq, dk and dv against the oracle's
    full backward (about 0.7 TFLOP of fp64 work over the host's cores), the
    kernels given the oracle's O (correctly rounded) and LSE."""
    B, S, H, D = 4, 4096, 16, 128
    q, k, v, do = problem(B, S, S, H, H, D, seed=90)
    stats = check(q, k, v, do, 1, 1 / math.sqrt(D), "headline every element")
    print("headline every element, (mean, max excess) in u rms:",
          {k_: (round(a, 3), round(b, 2)) for k_, (a, b) in stats.items()})


def test_bwd_gqa_sampled():
    _sampled((1, 2048, 2048, 8, 2, 128), 1, seed=87, n_rows=32, kv_pairs=[(0, 1)])


@pytest.mark.parametrize("Sq,Skv,causal,D", [(128, 8192, 2, 128), (8192, 128, 1, 128), (200, 6000, 2, 128),
                                             (128, 4096, 2, 256), (4096, 128, 1, 256)],
                         ids=["keys_unseen", "rows_unseeing", "ragged_unseen", "keys_unseen_d256",
                              "rows_unseeing_d256"])
def test_bwd_queues_with_mostly_empty_items(Sq, Skv, causal, D):
    """More work items than SMs, nearly all of them empty: with a top-left mask
    and Skv >> Sq most KV tiles are seen by no row (the dK/dV queue), with a
    bottom-right mask and Sq >> Skv most query tiles see no key (the dQ queue).
    Empty items write exact zeros and must not upset the barrier phases of the
    items around them."""
    q, k, v, do = problem(1, Sq, Skv, 8, 8, D, seed=Sq + Skv + causal)
    check(q, k, v, do, causal, 1 / math.sqrt(D), f"Sq={Sq} Skv={Skv} causal={causal} D={D}")
    dq, dk, dv = gpu_grads(q, k, v, do, causal, 1 / math.sqrt(D))
    if causal == 2:
        assert np.all(dk[:, Sq:] == 0.0) and np.all(dv[:, Sq:] == 0.0)
    else:
        assert np.all(dq[:, : Sq - Skv] == 0.0)


def test_bwd_chunked_prefill_shape_sampled():
    """B=1, Hq=64, Hkv=8, Sq=512 against Skv=32768 keys, bottom-right mask: dq
    rows and the dk/dv keys of one key/value head (its 8 query heads)."""
    _sampled((1, 512, 32768, 64, 8, 128), 1, seed=88, n_rows=32, kv_pairs=[(0, 5)])


def test_bwd_long_noncausal_shape_sampled():
    """B=1, H=16, S=16384 without a mask, Q drawn with sigma 4 (sharp rows)."""
    B, Sq, Skv, Hq, Hkv, D = 1, 16384, 16384, 16, 16, 128
    q, k, v, do = problem(B, Sq, Skv, Hq, Hkv, D, seed=89)
    q = inputs.normal_bf16(q.shape, 4.0, 89, 0)
    scale = 1 / math.sqrt(D)
    (dq, dk, dv), o_bits = gpu_grads(q, k, v, do, 0, scale, fwd="gpu", want_o=True)
    rows = inputs.sample_rows(B, Hq, Sq, 16, 89)
    ref_dq = oracle.attn_bwd_dq_rows(q, k, v, do, rows, 0, scale, o=o_bits)
    got_dq = np.array([dq[b, i, h] for b, h, i in rows])
    keys = [(0, 9, j) for j in (0, 1, 127, 128, 8191, 16383)]
    ref_dk, ref_dv = oracle.attn_bwd_dkv_keys(q, k, v, do, keys, 0, scale, o=o_bits)
    got_dk = np.array([dk[b, j, g] for b, g, j in keys])
    got_dv = np.array([dv[b, j, g] for b, g, j in keys])
    compare((got_dq, got_dk, got_dv), (ref_dq, ref_dk, ref_dv), "bf16", "long non-causal sampled",
            term_sizes(q, k, v, do, scale))


def test_bwd_d256_shape_sampled():
    """B=4, H=16, S=4096, D=256, causal (the forward's head-size-256 benchmark
    shape): sampled dq rows and dk/dv keys of two (batch, head) pairs."""
    _sampled((4, 4096, 4096, 16, 16, 256), 1, seed=91, n_rows=32, kv_pairs=[(0, 3), (3, 12)])


def test_bwd_d256_shape_every_element():
    """B=4, H=16, S=4096, D=256, causal: every element of dq, dk and dv against
    the oracle's full backward (the kernels given the oracle's O and LSE)."""
    B, S, H, D = 4, 4096, 16, 256
    q, k, v, do = problem(B, S, S, H, H, D, seed=93)
    stats = check(q, k, v, do, 1, 1 / math.sqrt(D), "d256 full shape every element")
    print("d256 full shape every element, (mean, max excess) in u rms:",
          {k_: (round(a, 3), round(b, 2)) for k_, (a, b) in stats.items()})


def test_bwd_d256_every_element():
    """Head size 256 with every element of dq, dk and dv against the oracle:
    GQA group 2, 2048 rows and keys (16 tiles each way), causal."""
    B, S, Hq, Hkv, D = 1, 2048, 4, 2, 256
    q, k, v, do = problem(B, S, S, Hq, Hkv, D, seed=92)
    stats = check(q, k, v, do, 1, 1 / math.sqrt(D), "d256 every element")
    print("d256 every element, (mean, max excess) in u rms:",
          {k_: (round(a, 3), round(b, 2)) for k_, (a, b) in stats.items()})
