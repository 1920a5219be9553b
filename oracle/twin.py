"""Independent numpy fp64 restatement of attention, for tiny shapes only.

TEST INFRASTRUCTURE: it exists to cross-check the C oracle by brute force and
shares no code with it.  Written per head with a dense masked logit matrix
(one numpy matmul per head), a masked row maximum, exponentials, row sums and
a second matmul with V -- the Pallas page's ``attention_reference`` (fp32
einsum, ``logits.max``, ``exp``, divide by the row sum) in fp64 with the
caller's scale, a bottom-right (causal=1) or top-left (causal=2) mask and a
natural-log LSE.
"""
from __future__ import annotations

import numpy as np


def _widen(bits, f16=False):
    bits = np.asarray(bits, dtype=np.uint16)
    if f16:  # numpy's own binary16 type
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def attention(q_bits, k_bits, v_bits, causal: int, scale: float, f16: bool = False):
    """Returns (o [B,Sq,Hq,D] fp64, lse [B,Hq,Sq] fp64); f16: binary16 inputs."""
    return attention_values(_widen(q_bits, f16), _widen(k_bits, f16), _widen(v_bits, f16),
                            causal, scale)


def attention_values(q, k, v, causal: int, scale: float):
    """The same on fp64 arrays (any real values, e.g. perturbed inputs)."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    group = Hq // Hkv
    o = np.zeros((B, Sq, Hq, D))
    lse = np.zeros((B, Hq, Sq))
    qi = np.arange(Sq)[:, None]
    kj = np.arange(Skv)[None, :]
    if int(causal) == 1:      # bottom-right aligned
        visible = kj <= qi + (Skv - Sq)
    elif int(causal) == 2:    # top-left aligned
        visible = kj <= qi
    else:
        visible = np.ones((Sq, Skv), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            g = h // group
            logits = scale * (q[b, :, h, :] @ k[b, :, g, :].T)
            logits = np.where(visible, logits, -np.inf)
            for i in range(Sq):
                row = logits[i]
                if not np.any(visible[i]):
                    o[b, i, h, :] = 0.0
                    lse[b, h, i] = -np.inf
                    continue
                m = row[visible[i]].max()
                w = np.where(visible[i], np.exp(row - m), 0.0)
                l = w.sum()
                o[b, i, h, :] = (w @ v[b, :, g, :]) / l
                lse[b, h, i] = m + np.log(l)
    return o, lse
