"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, and its host-side validation rejects bad requests before any
CUDA call (no GPU is touched: every call here returns before launching)."""
import ctypes
import math
import os
import re

import pytest

import attention_forward_11_gb300 as fa
from attention_forward_11_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    assert declared_functions() == sorted(fa._binding.EXPORTED)


def _declaration(name):
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    m = re.search(r"(\w+)\s+" + name + r"\s*\(([^)]*)\)\s*;", text)
    assert m, f"{name} is not declared"
    params = [" ".join(p.split()) for p in m.group(2).split(",")]
    return m.group(1), params


def test_boundary_calls_have_their_specified_signatures():
    """The three calls of the boundary: the forward, the status string, and the
    device status of the calls made so far (no stream argument)."""
    ret, params = _declaration("attn_fwd")
    assert ret == "attn_status_t"
    assert params == ["const void* q", "const void* k", "const void* v", "void* o", "float* lse",
                      "int B", "int Sq", "int Skv", "int Hq", "int Hkv", "int D", "int causal",
                      "float scale", "cudaStream_t stream"]
    assert re.search(r"const char\*\s*attn_status_str\(attn_status_t status\);", open(HEADER).read())
    assert _declaration("attn_last_device_status") == ("attn_status_t", ["void"])
    text = open(HEADER).read()
    for name, value in (("ATTN_OK", 0), ("ATTN_ERR_INVALID_ARG", 1), ("ATTN_ERR_UNSUPPORTED", 2),
                        ("ATTN_ERR_CUDA", 3), ("ATTN_ERR_TIMEOUT", 4)):
        assert re.search(rf"\b{name}\s*=\s*{value}\b", text), name


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert fa.attn_status_str(0) == "ATTN_OK"
    assert fa.attn_status_str(1) == "ATTN_ERR_INVALID_ARG"
    assert fa.attn_status_str(2) == "ATTN_ERR_UNSUPPORTED"
    assert fa.attn_status_str(3) == "ATTN_ERR_CUDA"
    assert fa.attn_status_str(4) == "ATTN_ERR_TIMEOUT"
    assert fa.attn_status_str(99) == "ATTN_UNKNOWN_STATUS"


# fake, 16-byte aligned, non-overlapping addresses: validation never dereferences them
Q, K, V, O, L = 0x1000000, 0x2000000, 0x3000000, 0x4000000, 0x5000000
GOOD = dict(q=Q, k=K, v=V, o=O, lse=L, B=1, Sq=256, Skv=256, Hq=2, Hkv=2, D=128, causal=1,
            scale=0.088, stream=0)


def call(**over):
    a = {**GOOD, **over}
    return fa.attn_fwd_ptr(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Sq"], a["Skv"],
                           a["Hq"], a["Hkv"], a["D"], a["causal"], a["scale"], a["stream"])


@pytest.mark.parametrize("over", [
    dict(q=0), dict(k=0), dict(v=0), dict(o=0),
    dict(B=0), dict(Sq=0), dict(Skv=-1), dict(Hq=0), dict(Hkv=0), dict(D=0),
    dict(Hq=6, Hkv=4), dict(causal=3), dict(causal=-1),
    dict(scale=0.0), dict(scale=-1.0), dict(scale=math.nan), dict(scale=math.inf),
    dict(q=Q + 8), dict(k=K + 2), dict(v=V + 4), dict(o=O + 1), dict(lse=L + 2),
    dict(o=Q + 64), dict(o=K), dict(lse=O + 16), dict(lse=Q + 32), dict(lse=K + 64),
    dict(lse=V), dict(lse=V + 256 * 2 * 128 * 2 - 4),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_invalid_arguments_rejected(lib, over):
    assert call(**over) == fa.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("D", [32, 96, 192, 320])
def test_other_head_dims_unsupported(lib, D):
    assert call(D=D) == fa.ATTN_ERR_UNSUPPORTED


def test_wait_selftest_rejects_bad_limit(lib):
    assert fa._binding.attn_debug_wait_timeout(0, 0) == fa.ATTN_ERR_INVALID_ARG
    assert fa._binding.attn_debug_wait_timeout((1 << 20) + 1, 0) == fa.ATTN_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(fa._binding, "_lib", None)
    monkeypatch.setenv("LIBATTN_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(fa.AttnError):
        fa.load_library()
    monkeypatch.setattr(fa._binding, "_lib", None)


def test_library_does_not_link_the_oracle(lib):
    # the product library and the oracle share no code: no oracle symbol in libattn
    for name in ("oracle_attn_rows", "oracle_attn_fwd", "oracle_partial_triple"):
        assert not hasattr(lib, name)
    assert ctypes.CDLL(fa.library_path()) is not None


def call_split(**over):
    a = {**GOOD, "ws": 0x6000000, "ws_bytes": 1 << 20, **over}
    return fa.attn_fwd_splitkv_ptr(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Sq"],
                                   a["Skv"], a["Hq"], a["Hkv"], a["D"], a["causal"], a["scale"],
                                   a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over", [
    dict(q=0), dict(o=0), dict(B=0), dict(Hq=6, Hkv=4), dict(causal=3), dict(scale=0.0),
    dict(q=Q + 8), dict(o=Q), dict(ws=0x6000000 + 16),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_splitkv_invalid_arguments_rejected(lib, over):
    assert call_split(**over) == fa.ATTN_ERR_INVALID_ARG


def test_splitkv_other_head_dims_unsupported(lib):
    assert call_split(D=192) == fa.ATTN_ERR_UNSUPPORTED


def test_splitkv_workspace_size_argument_checks(lib):
    assert lib.attn_fwd_splitkv_workspace_size(1, 256, 256, 2, 2, 128, 1, None) == \
        fa.ATTN_ERR_INVALID_ARG
    with pytest.raises(fa.AttnError) as e:
        fa.attn_fwd_splitkv_workspace_size(1, 256, 256, 3, 2, 128, 1)
    assert e.value.status == fa.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", [-1, 2, 7])
def test_fwd_ex_rejects_unknown_dtype(lib, dtype):
    a = GOOD
    assert fa.attn_fwd_ex_ptr(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Sq"], a["Skv"],
                              a["Hq"], a["Hkv"], a["D"], a["causal"], a["scale"], dtype,
                              0) == fa.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", [0, 1])
def test_fwd_ex_validates_like_attn_fwd(lib, dtype):
    a = {**GOOD, "q": 0}
    assert fa.attn_fwd_ex_ptr(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Sq"], a["Skv"],
                              a["Hq"], a["Hkv"], a["D"], a["causal"], a["scale"], dtype,
                              0) == fa.ATTN_ERR_INVALID_ARG
    a = {**GOOD, "D": 192}
    assert fa.attn_fwd_ex_ptr(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Sq"], a["Skv"],
                              a["Hq"], a["Hkv"], a["D"], a["causal"], a["scale"], dtype,
                              0) == fa.ATTN_ERR_UNSUPPORTED


# ---- backward: argument checks (fake addresses, nothing launched)
BWD = dict(q=Q, k=K, v=V, o=O, lse=L, do=0x6000000, dq=0x7000000, dk=0x8000000, dv=0x9000000,
           B=1, Sq=256, Skv=256, Hq=2, Hkv=2, D=128, causal=1, scale=0.088, dtype=0,
           ws=0xA000000, ws_bytes=1 << 20, stream=0)


def call_bwd(**over):
    a = {**BWD, **over}
    return fa.attn_bwd_ptr(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"],
                           a["dv"], a["B"], a["Sq"], a["Skv"], a["Hq"], a["Hkv"], a["D"],
                           a["causal"], a["scale"], a["dtype"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over", [
    dict(q=0), dict(k=0), dict(v=0), dict(o=0), dict(lse=0), dict(do=0), dict(dq=0), dict(dk=0),
    dict(dv=0), dict(ws=0),
    dict(B=0), dict(Sq=0), dict(Skv=-1), dict(Hq=3, Hkv=2), dict(causal=3), dict(dtype=2),
    dict(scale=0.0), dict(scale=math.nan),
    dict(q=Q + 8), dict(do=0x6000000 + 4), dict(dq=0x7000000 + 2), dict(dk=0x8000000 + 8),
    dict(lse=L + 2), dict(ws=0xA000000 + 16), dict(ws_bytes=1024),
    dict(dq=Q), dict(dk=K + 256), dict(dv=0x6000000), dict(dk=0x9000000), dict(ws=0x7000000),
    dict(dq=L),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_bwd_invalid_arguments_rejected(lib, over):
    assert call_bwd(**over) == fa.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("over", [dict(ws_bytes=1024), dict(q=Q + 8), dict(dq=Q), dict(scale=0.0),
                                  dict(Hq=3, Hkv=2), dict(dk=K + 256)],
                         ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_bwd_head_size_256_validated_like_the_others(lib, over):
    """The head-size-256 backward (its own kernels) takes the same checks; a bad
    argument is rejected before anything is launched."""
    assert call_bwd(D=256, **over) == fa.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("D", [32, 96, 192])
def test_bwd_other_head_dims_unsupported(lib, D):
    assert call_bwd(D=D) == fa.ATTN_ERR_UNSUPPORTED


def test_bwd_workspace_size(lib):
    # two fp32 vectors of B * Hq * (Sq rounded up to 128) entries, each rounded up to 256
    # bytes, and 256 bytes for the kernels' work counters; the same at every head size
    assert fa.attn_bwd_workspace_size(1, 256, 256, 2, 2, 128) == 2 * 2 * 256 * 4 + 256
    assert fa.attn_bwd_workspace_size(1, 256, 256, 2, 2, 256) == 2 * 2 * 256 * 4 + 256
    assert fa.attn_bwd_workspace_size(3, 129, 7, 5, 1, 64) == 2 * 3 * 5 * 256 * 4 + 256
    assert fa.attn_bwd_workspace_size(1, 1, 1, 1, 1, 128) == 2 * 512 + 256
    assert lib.attn_bwd_workspace_size(1, 256, 256, 2, 2, 128, None) == fa.ATTN_ERR_INVALID_ARG
    with pytest.raises(fa.AttnError) as e:
        fa.attn_bwd_workspace_size(1, 256, 256, 3, 2, 128)
    assert e.value.status == fa.ATTN_ERR_INVALID_ARG
    with pytest.raises(fa.AttnError) as e:
        fa.attn_bwd_workspace_size(1, 256, 256, 2, 2, 192)
    assert e.value.status == fa.ATTN_ERR_UNSUPPORTED


def test_unit_rates_arguments_checked_before_any_launch(lib):
    import ctypes
    out = (ctypes.c_double * 8)()
    assert lib.attn_debug_unit_rates(None, 8, None) == fa.ATTN_ERR_INVALID_ARG
    assert lib.attn_debug_unit_rates(out, 7, None) == fa.ATTN_ERR_INVALID_ARG


# ---- the forward's unit table (host logic; no GPU)
def _kv_tiles(row0, Sq, Skv, causal):
    """KV tiles a 128-row query tile starting at row0 visits (key j visible from
    row i iff j <= i + diag; diag = Skv - Sq bottom-right, 0 top-left)."""
    if row0 >= Sq:
        return 0
    n_all = -(-Skv // 128)
    if not causal:
        return n_all
    diag = Skv - Sq if causal == 1 else 0
    last_key = min(row0 + 127, Sq - 1) + diag
    return 0 if last_key < 0 else min(n_all, last_key // 128 + 1)


def _unit_weights(B, Sq, Skv, Hq, Hkv, causal):
    """KV steps of every unit in the forward's causal numbering: row units
    outermost (longest first), then batch and head unit; a unit is two row
    tiles of one head, or one row tile of two heads when the group is even."""
    pairs = (Hq // Hkv) % 2 == 0
    n_head_units = Hq // 2 if pairs else Hq
    rows_per_unit = 128 if pairs else 256
    n_row_units = -(-Sq // rows_per_unit)
    w = []
    for ru in range(n_row_units):
        row_unit = n_row_units - 1 - ru
        for _ in range(B * n_head_units):
            if pairs:
                r0 = r1 = row_unit * 128
            else:
                r0, r1 = row_unit * 256, row_unit * 256 + 128
            w.append(max(_kv_tiles(r0, Sq, Skv, causal), _kv_tiles(r1, Sq, Skv, causal)))
    return w, B * n_head_units


@pytest.mark.parametrize("shape", [(4, 4096, 4096, 16, 16, 1), (2, 8192, 8192, 32, 8, 1), (1, 2048, 3000, 8, 8, 1),
                                   (3, 1000, 1000, 6, 3, 2), (1, 512, 32768, 64, 8, 1)])
def test_unit_table_is_a_balanced_permutation(shape):
    B, Sq, Skv, Hq, Hkv, causal = shape
    sms = 152
    table = fa.attn_debug_unit_schedule(B, Sq, Skv, Hq, Hkv, 128, causal, sms)
    weights, inner_count = _unit_weights(B, Sq, Skv, Hq, Hkv, causal)
    assert table is not None
    cta_begin, units = table
    n = len(weights)
    grid = min(n, sms)
    assert len(cta_begin) == grid + 1 and cta_begin[0] == 0 and cta_begin[-1] == n
    assert all(a <= b for a, b in zip(cta_begin, cta_begin[1:]))
    assert sorted(units) == list(range(n)), "every unit exactly once"
    # each unit went to the least-loaded CTA: the CTAs' totals (KV steps plus one
    # per unit) differ by at most the heaviest unit
    loads = [sum(weights[u] + 1 for u in units[cta_begin[c]:cta_begin[c + 1]]) for c in range(grid)]
    assert max(loads) - min(loads) <= max(weights) + 1
    # within a CTA the units come in the table's order: blocks of heads whose K
    # and V take at most 48 MB, in turn, longest first inside each block
    units_per_kv = max(1, inner_count // B // Hkv)
    per_block = min(inner_count, max(1, (48 << 20) // (4 * Skv * 128)) * units_per_kv)
    block_of = lambda u: (u % inner_count) // per_block
    for c in range(grid):
        mine = units[cta_begin[c]:cta_begin[c + 1]]
        assert [block_of(u) for u in mine] == sorted(block_of(u) for u in mine)
        for a, b in zip(mine, mine[1:]):
            if block_of(a) == block_of(b):
                assert weights[a] >= weights[b]


def test_unit_table_only_for_causal_head_size_128_up_to_its_size():
    assert fa.attn_debug_unit_schedule(1, 16384, 16384, 16, 16, 128, 0, 152) is None   # unmasked: head-major
    assert fa.attn_debug_unit_schedule(4, 4096, 4096, 16, 16, 64, 1, 152) is None     # head size 64: snake
    assert fa.attn_debug_unit_schedule(4, 4096, 4096, 16, 16, 256, 1, 152) is None    # own kernel
    assert fa.attn_debug_unit_schedule(16, 8192, 8192, 32, 32, 128, 1, 152) is None  # 8192 units > 2048


def test_unit_table_rejects_bad_arguments():
    lib = fa.load_library()
    n = ctypes.c_int(0)
    buf = (ctypes.c_int * 4096)()
    beg = (ctypes.c_int * 300)()
    for sms in (0, 257):
        assert lib.attn_debug_unit_schedule(4, 4096, 4096, 16, 16, 128, 1, sms, beg, buf, 4096,
                                            ctypes.byref(n)) == fa.ATTN_ERR_INVALID_ARG
    assert lib.attn_debug_unit_schedule(4, 4096, 4096, 16, 16, 128, 1, 152, None, buf, 4096,
                                        ctypes.byref(n)) == fa.ATTN_ERR_INVALID_ARG
    assert lib.attn_debug_unit_schedule(4, 4096, 4096, 16, 16, 128, 1, 152, beg, buf, 1000,
                                        ctypes.byref(n)) == fa.ATTN_ERR_INVALID_ARG   # 1024 units
    assert lib.attn_debug_unit_schedule(4, 4096, 4096, 15, 4, 128, 1, 152, beg, buf, 4096,
                                        ctypes.byref(n)) == fa.ATTN_ERR_INVALID_ARG   # Hq % Hkv
    assert lib.attn_debug_unit_schedule(4, 4096, 4096, 16, 16, 96, 1, 152, beg, buf, 4096,
                                        ctypes.byref(n)) == fa.ATTN_ERR_UNSUPPORTED
