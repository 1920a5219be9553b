"""Shared helpers for the GPU parity tests: run libattn through its C ABI on
seeded bf16 inputs and compare with the fp64 oracle, element by element.

Acceptance (the stated tolerance of this attention forward):
    O:   max |O_gpu - bf16(O_oracle)| <= 2e-2 and mean <= 2e-3
    LSE: max |LSE_gpu - LSE_oracle| <= 1e-3, and -inf exactly where the oracle has it
"""
import numpy as np

import oracle

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def to_device(bits, dtype="bf16"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16).cuda()


def run_gpu(q, k, v, causal, scale, want_lse=True, dtype="bf16"):
    """q/k/v: uint16 bit patterns (bf16, or binary16 with dtype="f16").
    Returns (o fp64 [B,Sq,Hq,D], lse fp64 [B,Hq,Sq] or None)."""
    import torch
    import attention_forward_11_gb300 as fa
    dq, dk, dv = to_device(q, dtype), to_device(k, dtype), to_device(v, dtype)
    o, lse = fa.attn_fwd(dq, dk, dv, causal=int(causal), scale=scale, want_lse=want_lse)
    st = fa.attn_check_device_status()
    assert st == fa.ATTN_OK, f"device status {st}"
    o64 = o.float().double().cpu().numpy()
    l64 = lse.double().cpu().numpy() if lse is not None else None
    del dq, dk, dv
    torch.cuda.synchronize()
    return o64, l64


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what="", dtype="bf16"):
    """Element-wise comparison; returns (max_abs, mean_abs, lse_max_abs)."""
    o_ref_b = oracle.round_f16(o_ref) if dtype == "f16" else oracle.round_bf16(o_ref)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    err = np.abs(o_gpu - o_ref_b)
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    assert mx <= O_MAX_ABS, f"{what}: O max abs err {mx:.3e}"
    assert mean <= O_MEAN_ABS, f"{what}: O mean abs err {mean:.3e}"
    lmx = 0.0
    if lse_gpu is not None:
        ninf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lse_gpu), ninf_ref), f"{what}: -inf LSE pattern differs"
        fin = ~ninf_ref
        lerr = np.abs(lse_gpu[fin] - lse_ref[fin])
        lmx = float(lerr.max(initial=0.0))
        assert lmx <= LSE_MAX_ABS, f"{what}: LSE max abs err {lmx:.3e}"
    return mx, mean, lmx


def check_full(q, k, v, causal, scale, what="", dtype="bf16"):
    o_gpu, l_gpu = run_gpu(q, k, v, causal, scale, dtype=dtype)
    o_ref, l_ref = oracle.attn_full(q, k, v, int(causal), scale, f16=dtype == "f16")
    return compare(o_gpu, l_gpu, o_ref, l_ref, what, dtype)


def check_rows(q, k, v, causal, scale, rows, what="", dtype="bf16"):
    """Full-size run; the oracle computes only the listed (b, h, i) rows."""
    o_gpu, l_gpu = run_gpu(q, k, v, causal, scale, dtype=dtype)
    o_ref, l_ref = oracle.attn_rows(q, k, v, rows, int(causal), scale, f16=dtype == "f16")
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    return compare(o_gpu[b, i, h, :], l_gpu[b, h, i], o_ref, l_ref, what, dtype)
