"""Out-of-bounds canaries (compute-sanitizer is closed on this machine): every
output and workspace buffer sits between two guard regions filled with a
sentinel pattern, and after each call the guards must be untouched and every
output element written.  Ragged lengths put rows past Sq and keys past Skv in
the last tiles, where a clipped TMA store or a masked epilogue store matters."""
import math

import numpy as np
import pytest

import attention_forward_11_gb300 as fa
from attention_forward_11_gb300 import inputs
from parity import to_device

pytestmark = pytest.mark.gpu

GUARD = 8192                 # bytes on each side (a multiple of 256: keeps the inner view aligned)
# sentinel words: two 16-bit halves 0x7E5A (bf16 4.2e37, binary16 NaN: never an
# attention output or gradient), or an fp32 NaN payload for 32-bit data
SENT_16 = 0x7E5A7E5A
SENT_32 = 0x7FC0DEAD


class Guarded:
    """A device tensor of `shape` and `dtype` inside [guard | data | guard],
    all laid out in 32-bit words filled with a sentinel."""

    def __init__(self, shape, dtype):
        import torch
        esize = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape))
        nbytes = n * esize
        assert nbytes % 4 == 0
        self.esize, self.n, self.nw, self.g = esize, n, nbytes // 4, GUARD // 4
        self.sent = SENT_32 if esize == 4 else SENT_16
        self.raw = torch.full((2 * self.g + self.nw,), self.sent, dtype=torch.int32, device="cuda")
        data = self.raw[self.g:self.g + self.nw]
        self.t = data.view(torch.uint8).view(dtype).view(*shape)

    def guards_intact(self):
        r = self.raw
        return bool((r[:self.g] == self.sent).all()) and bool((r[self.g + self.nw:] == self.sent).all())

    def fully_written(self):
        import torch
        data = self.raw[self.g:self.g + self.nw]
        if self.esize == 2:
            return not bool((data.view(torch.int16) == 0x7E5A).any())
        return not bool((data == self.sent).any())


def _check(*bufs, written=True):
    import torch
    torch.cuda.synchronize()
    assert fa.attn_check_device_status() == fa.ATTN_OK
    for name, b in bufs:
        assert b.guards_intact(), f"{name}: a guard was overwritten"
        if written:
            assert b.fully_written(), f"{name}: some element was not written"


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [0, 1, 2])
def test_forward_writes_exactly_its_outputs(D, dtype, causal):
    import torch
    B, Sq, Skv, Hq, Hkv = 2, 333, 201, 4, 2
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=D + causal, dtype=dtype)
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    o = Guarded((B, Sq, Hq, D), tdt)
    lse = Guarded((B, Hq, Sq), torch.float32)
    code = fa.ATTN_DTYPE_F16 if dtype == "f16" else fa.ATTN_DTYPE_BF16
    tq, tk, tv = (to_device(x, dtype) for x in (q, k, v))
    st = fa.attn_fwd_ex_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.t.data_ptr(), lse.t.data_ptr(),
                            B, Sq, Skv, Hq, Hkv, D, causal, 1 / math.sqrt(D), code,
                            torch.cuda.current_stream().cuda_stream)
    assert st == fa.ATTN_OK
    _check(("o", o), ("lse", lse))


@pytest.mark.parametrize("D", [64, 128])
def test_splitkv_writes_exactly_its_outputs_and_workspace(D):
    import torch
    B, Sq, Skv, Hq, Hkv, causal = 1, 300, 9000, 2, 2, 1
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=7)
    n = fa.attn_fwd_splitkv_workspace_size(B, Sq, Skv, Hq, Hkv, D, causal)
    assert n > 0
    ws = Guarded((n,), torch.uint8)
    o = Guarded((B, Sq, Hq, D), torch.bfloat16)
    lse = Guarded((B, Hq, Sq), torch.float32)
    tq, tk, tv = (to_device(x) for x in (q, k, v))
    st = fa.attn_fwd_splitkv_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.t.data_ptr(), lse.t.data_ptr(),
                                 B, Sq, Skv, Hq, Hkv, D, causal, 1 / math.sqrt(D), ws.t.data_ptr(), n,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == fa.ATTN_OK
    _check(("o", o), ("lse", lse))
    _check(("workspace", ws), written=False)


def test_noalloc_writes_exactly_its_outputs():
    import torch
    B, Sq, Skv, Hq, Hkv, D, causal = 1, 250, 7000, 2, 1, 128, 2
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=8)
    o = Guarded((B, Sq, Hq, D), torch.bfloat16)
    lse = Guarded((B, Hq, Sq), torch.float32)
    tq, tk, tv = (to_device(x) for x in (q, k, v))
    st = fa.attn_fwd_splitkv_noalloc_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.t.data_ptr(),
                                         lse.t.data_ptr(), B, Sq, Skv, Hq, Hkv, D, causal, 1 / math.sqrt(D),
                                         torch.cuda.current_stream().cuda_stream)
    assert st == fa.ATTN_OK
    _check(("o", o), ("lse", lse))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [0, 1, 2])
def test_backward_writes_exactly_its_outputs_and_workspace(D, causal):
    import torch
    B, Sq, Skv, Hq, Hkv = 2, 333, 201, 4, 2
    q, k, v = inputs.make_qkv(B, Sq, Skv, Hq, Hkv, D, seed=20 + D + causal)
    do = inputs.normal_bf16(q.shape, 1.0, 9, 3)
    tq, tk, tv, tdo = (to_device(x) for x in (q, k, v, do))
    o, lse = fa.attn_fwd(tq, tk, tv, causal=causal, scale=1 / math.sqrt(D))
    n = fa.attn_bwd_workspace_size(B, Sq, Skv, Hq, Hkv, D)
    ws = Guarded((n,), torch.uint8)
    dq = Guarded((B, Sq, Hq, D), torch.bfloat16)
    dk = Guarded((B, Skv, Hkv, D), torch.bfloat16)
    dv = Guarded((B, Skv, Hkv, D), torch.bfloat16)
    st = fa.attn_bwd_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                         tdo.data_ptr(), dq.t.data_ptr(), dk.t.data_ptr(), dv.t.data_ptr(), B, Sq, Skv, Hq, Hkv,
                         D, causal, 1 / math.sqrt(D), fa.ATTN_DTYPE_BF16, ws.t.data_ptr(), n,
                         torch.cuda.current_stream().cuda_stream)
    assert st == fa.ATTN_OK
    _check(("dq", dq), ("dk", dk), ("dv", dv))
    _check(("workspace", ws), written=False)
