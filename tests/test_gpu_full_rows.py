"""Acceptance at full size: every row of every (batch, head) of the four large
benchmark shapes, GPU against the fp64 oracle element by element, in the
launch configuration the benchmark times (`attn_fwd`, persistent grid).

The sampled-row tests elsewhere cover the same shapes in seconds; these cover
all of O and LSE: 4.1 TFLOP of fp64 oracle work in total, spread over the
host's cores by the oracle's OpenMP loop (7 to 45 s per shape, 90 s for the
four, on 16 Arm cores)."""
import time

import pytest

import oracle
from attention_forward_11_gb300 import inputs
from parity import check_full

pytestmark = pytest.mark.gpu

FULL = ["mha_causal_4x16x4096", "gqa_causal_2x32x8_8192", "long_sharp_1x16x16384",
        "chunked_prefill_gqa_64x8_512x32768"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_row(name):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.make_workload(w, seed=0)
    t0 = time.time()
    mx, mean, lmx = check_full(q, k, v, w.causal, w.scale, name)
    print(f"{name}: every row, O max-abs {mx:.3e} mean-abs {mean:.3e}, LSE max-abs {lmx:.3e}, "
          f"{time.time() - t0:.1f} s with {oracle.num_threads()} oracle threads")
