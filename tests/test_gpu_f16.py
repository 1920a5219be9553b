"""GPU parity of the binary16 path (attn_fwd_ex with ATTN_DTYPE_F16): the same
kernel with f16 operands, f16 P and f16 O, against the fp64 oracle reading
the same binary16 bits (O compared after round-to-nearest-even to binary16)."""
import math

import numpy as np
import pytest

from attention_forward_11_gb300 import inputs
from parity import check_full, check_rows, run_gpu

pytestmark = pytest.mark.gpu

CASES = [
    # B, Sq, Skv, Hq, Hkv, causal, q_sigma
    (1, 256, 256, 2, 2, 1, 1.0),
    (1, 256, 256, 2, 2, 0, 1.0),
    (2, 200, 333, 4, 2, 1, 1.0),
    (1, 300, 77, 2, 2, 1, 1.0),
    (1, 384, 640, 6, 2, 2, 1.0),
    (1, 1000, 1000, 2, 1, 0, 4.0),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_f16_every_row(case):
    B, Sq, Skv, Hq, Hkv, causal, qs = case
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, 128, seed=int(sum(case[:6])), q_sigma=qs,
                              dtype="f16")
    check_full(q, k, v, causal, 1 / math.sqrt(128), str(case), dtype="f16")


def test_f16_full_size_sampled_rows():
    w = inputs.WORKLOADS["mha_causal_4x16x4096"]
    q, k, v = inputs.make_qkv(w.B, w.Sq, w.Skv, w.Hq, w.Hkv, w.D, seed=5, dtype="f16")
    rows = inputs.sample_rows(w.B, w.Hq, w.Sq, n=512, seed=5)
    check_rows(q, k, v, w.causal, w.scale, rows, "mha causal f16", dtype="f16")


def test_f16_and_bf16_paths_differ_only_by_format():
    """Inputs exactly representable in both formats (small integers / 8): the two
    paths see the same real numbers and agree to the coarser output rounding."""
    rng = np.random.default_rng(3)
    vals = rng.integers(-16, 17, size=(1, 300, 2, 128)).astype(np.float32) / 8
    f16 = vals.astype(np.float16).view(np.uint16)
    bf = (vals.view(np.uint32) >> 16).astype(np.uint16)
    o_h, l_h = run_gpu(f16, f16, f16, 1, 0.05, dtype="f16")
    o_b, l_b = run_gpu(bf, bf, bf, 1, 0.05)
    assert np.max(np.abs(o_h - o_b)) <= 2e-2 and np.max(np.abs(l_h - l_b)) <= 1e-3
