"""CPU tests of the C ABI: the library loads, exports every declared entry
point, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import sequence_tensor_transformer_gb300 as st

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(st.LIB_PATH):
        from sequence_tensor_transformer_gb300 import build
        build.build()
    return st.load_library()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    raw = ctypes.CDLL(st.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert set(names) == set(st.EXPORTED_SYMBOLS)


def test_every_declared_function_is_documented():
    """Each entry point of include/sptp.h sits under a comment block (argument
    meaning, layout, ownership, errors): one directly above it, or the one
    above the group of declarations it belongs to."""
    src = open(os.path.join(ROOT, "include", "sptp.h")).read()
    decls = [(m.start(), m.group(1)) for m in re.finditer(
        r"^(?:const\s+)?(?:size_t|int|void|const char\s*\*)\s*\*?\s*(\w+)\s*\(", src, re.M)]
    assert len(decls) >= 20
    documented = set()
    for pos, name in decls:
        before = src[:pos].rstrip()
        if before.endswith("*/"):
            documented.add(pos)
        elif before.endswith(");"):
            # part of a group: the declaration just above must be documented
            prev = max(p for p, _ in decls if p < pos)
            assert prev in documented, name
            documented.add(pos)
        else:
            raise AssertionError(f"{name} has no comment block")


def test_status_strings(lib):
    assert st.sptp_status_string(0) == "ok"
    for name, c in st.STATUS.items():
        assert st.sptp_status_string(c) != "unknown status", name
    assert st.sptp_status_string(-12) == "unknown status"


def test_status_codes_match_the_header():
    """The binding's status and variant tables against the header's enums."""
    src = open(os.path.join(ROOT, "include", "sptp.h")).read()
    codes = {m.group(1).lower(): int(m.group(2)) for m in re.finditer(r"SPTP_(OK|ERR_\w+) = (-?\d+)", src)}
    assert {k.replace("err_", ""): v for k, v in codes.items()} == st.STATUS
    variants = {m.group(1).lower(): int(m.group(2)) for m in re.finditer(r"SPTP_VARIANT_(\w+) = (\d+)", src)}
    assert variants == st.VARIANTS
    # the page-given codes keep their numbers
    assert (codes["err_null"], codes["err_shape"], codes["err_dtype"], codes["err_workspace"], codes["err_cuda"],
            codes["err_timeout"], codes["err_unimplemented"]) == (-1, -2, -3, -4, -5, -6, -7)


FAKE = 1 << 20  # a 16-byte aligned non-null address that is never dereferenced


def fwd(lib, M=64, d=128, F=512, P=2, C=4, eps=1e-6, dt=0, ptrs=None, out=FAKE * 64, resid=None,
        ws=FAKE * 4096, ws_bytes=1 << 40):
    p = ptrs or [FAKE * (i + 1) for i in range(6)]
    return lib.sptp_ffn_forward(*p, M, d, F, P, C, eps, dt, out, resid, ws, ws_bytes, None)


def test_forward_rejects_bad_arguments_without_gpu(lib):
    SHAPE, NULL, DTYPE, WS, ALIAS = -2, -1, -3, -4, -8
    assert fwd(lib, ptrs=[None] + [FAKE] * 5) == NULL
    assert fwd(lib, out=None) == NULL
    assert fwd(lib, ws=None) == NULL
    assert fwd(lib, d=100) == SHAPE           # d % 8
    assert fwd(lib, F=500) == SHAPE           # F % P ... (F/P) % 8
    assert fwd(lib, F=24, P=2) == SHAPE       # F/P = 12 not a multiple of 8
    assert fwd(lib, P=9, F=9 * 64, C=9) == SHAPE
    assert fwd(lib, C=3) == SHAPE             # chunks % P
    assert fwd(lib, M=66, C=4) == SHAPE       # M % chunks
    assert fwd(lib, dt=7) == DTYPE
    assert fwd(lib, eps=float("nan")) == SHAPE
    assert fwd(lib, ws_bytes=10) == WS
    assert fwd(lib, ptrs=[FAKE + 8] + [FAKE * 2] * 5) == SHAPE   # misaligned
    # out overlapping an input
    assert fwd(lib, ptrs=[FAKE * 64] + [FAKE * (i + 2) * 1024 for i in range(5)], out=FAKE * 64) == ALIAS


def test_workspace_size_queries(lib):
    n = st.sptp_ffn_workspace_size(64, 128, 512, 2, 4, 1)
    assert n >= 4096 + 64 * 128 * 4 + 64 * 512 * 4
    assert st.sptp_ffn_workspace_size(64, 100, 512, 2, 4, 0) == 0
    m = st.dtp_ffn_stack_workspace_size(4096, 1024, 3072, 2, 4, 1, 0)
    act = 4096 * 1024 * 2
    assert m >= 4096 + 2 * act + 4096 * 3072 * 2 + 2 * 2 * act
    assert st.dtp_ffn_stack_workspace_size(4096, 1024, 3072, 2, 0, 1, 0) == 0


def test_dtp_rejects_bad_arguments_without_gpu(lib):
    p = [FAKE * (i + 1) * 4096 for i in range(5)]
    call = lambda **k: lib.dtp_ffn_stack_forward(
        *p, k.get("M", 64), k.get("d", 128), k.get("F", 512), k.get("P", 2), k.get("L", 2),
        k.get("delta", 1), 1, 1e-6, 0, FAKE * 64 * 4096, 1 << 40, None)
    assert call(delta=-1) == -2
    assert call(L=0) == -2
    assert call(P=8, F=8 * 64, L=40, delta=40) == -2   # too many pending sources
    assert call(P=8, F=8 * 64, L=10, delta=9) == -2    # 1 + 7 * 10 = 71 > 64 sources in one update
    assert lib.dtp_ffn_stack_forward(None, *p[1:], 64, 128, 512, 2, 2, 1, 1, 1e-6, 0, FAKE, 1 << 40, None) == -1


def test_step_entry_points_reject_bad_arguments(lib):
    assert lib.sptp_prologue(FAKE, FAKE * 2, FAKE * 3, 64, 100, 2, 1e-6, 0, None, FAKE * 4, None) == -2
    assert lib.sptp_prologue(FAKE, FAKE * 2, FAKE * 3, 64, 128, 2, 1e-6, 0, None, None, None) == -1
    assert lib.sptp_gateup_swiglu(FAKE, FAKE * 2, FAKE * 3, 64, 128, 500, 2, 0, FAKE * 4, FAKE * 5, 1 << 20,
                                  None) == -2
    assert lib.sptp_down_proj(FAKE, FAKE * 2, 64, 128, 512, 2, 0, FAKE * 3, FAKE * 4, 100, None) == -4
    assert lib.sptp_wait_selftest(FAKE, 100, 1000, 0, None) == -4


def test_fp8_entry_points_reject_bad_arguments(lib):
    SHAPE, NULL, WS, ALIAS = -2, -1, -4, -8
    q = lambda a=FAKE, R=64, K=128, qq=FAKE * 4096, sc=FAKE * 8192: lib.sptp_quantize_rows_e4m3(a, R, K, qq, sc, None)
    assert q(R=0) == 0                 # empty: a no-op before any CUDA call
    assert q(K=136) == SHAPE           # K % 16
    assert q(K=0) == SHAPE
    assert q(R=-1) == SHAPE
    assert q(a=None) == NULL
    assert q(a=FAKE + 8) == SHAPE      # misaligned
    assert q(qq=FAKE + 64) == ALIAS    # codes overlap the input
    assert q(sc=FAKE * 4096 + 64) == ALIAS

    def f8(M=64, d=128, F=512, P=2, C=4, ptrs=None, out=FAKE * 64 * 4096, ws=FAKE * 128 * 4096,
           ws_bytes=1 << 40):
        p = ptrs or [FAKE * (i + 1) * 4096 for i in range(9)]
        return lib.sptp_ffn_forward_fp8(*p, M, d, F, P, C, 1e-6, out, None, ws, ws_bytes, None)
    assert f8(d=136) == SHAPE          # d % 16 (TMA rows of E4M3 bytes)
    assert f8(F=2 * 24) == SHAPE       # F/P % 16
    assert f8(C=3) == SHAPE
    assert f8(ws_bytes=100) == WS
    assert f8(ptrs=[None] + [FAKE * 4096] * 8) == NULL
    assert f8(out=FAKE * 3 * 4096) == ALIAS   # out on top of gamma
    n = st.sptp_ffn_fp8_workspace_size(64, 128, 512, 2, 4)
    assert n >= 4096 + 64 * 128 * 3 + 64 * 4 + 64 * 512 * 3 + 2 * 64 * 4
    assert st.sptp_ffn_fp8_workspace_size(64, 136, 512, 2, 4) == 0
    assert lib.sptp_gateup_swiglu_e4m3(FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, 64, 128, 2 * 24, 2,
                                       FAKE * 7, FAKE * 8, 1 << 20, None) == SHAPE
    assert lib.sptp_down_proj_e4m3(FAKE, FAKE * 2, FAKE * 3, FAKE * 4, 64, 128, 512, 2, FAKE * 5, FAKE * 6, 100,
                                   None) == WS


def test_variants_are_checked_before_any_gpu_work(lib):
    """A variant that does not exist for an entry point or dtype is refused
    with SPTP_ERR_UNIMPLEMENTED before any CUDA call."""
    UNIMPL = st.STATUS["unimplemented"]
    p = [FAKE * (i + 1) for i in range(6)]
    ex = lambda dt, v: lib.sptp_ffn_forward_ex(*p, 64, 128, 512, 2, 4, 1e-6, dt, FAKE * 64, None, FAKE * 4096,
                                                1 << 40, None, v)
    V = st.VARIANTS
    for v in (V["chain"], V["fused"], V["layers"], 9, -1):
        assert ex(1, v) == UNIMPL, v            # fp32: PAIR only
    for v in (V["layers"], 9):
        assert ex(0, v) == UNIMPL, v            # bf16: no LAYERS form of the boundary
    q = [FAKE * (i + 1) * 4096 for i in range(5)]
    dtp = lambda dt, v: lib.dtp_ffn_stack_forward_ex(*q, 64, 128, 512, 2, 2, 1, 1, 1e-6, dt, FAKE * 64 * 4096,
                                                      1 << 40, None, v)
    for v in (V["pair"], V["chain"], 7):
        assert dtp(0, v) == UNIMPL, v
    assert dtp(1, V["fused"]) == UNIMPL
    attn = lambda dt, v: lib.sptp_attn_qkv_forward_ex(FAKE, FAKE * 2, FAKE * 3, FAKE * 4, 64, 128, 512, 2, 2, 1e-6,
                                                       dt, FAKE * 64, None, FAKE * 128, 1 << 40, None, v)
    for v in (V["chain"], V["layers"]):
        assert attn(0, v) == UNIMPL, v
    assert attn(1, V["fused"]) == UNIMPL
    # the plain entry points are the AUTO forms: shape errors as before
    assert lib.sptp_ffn_forward(*p, 64, 100, 512, 2, 4, 1e-6, 0, FAKE * 64, None, FAKE * 4096, 1 << 40,
                                None) == st.STATUS["shape"]
