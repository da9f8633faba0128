"""CPU tests of the Python binding's argument checks: every tensor's shape,
dtype and device is checked against the others before any pointer reaches
the C ABI (which takes pointers and sizes only, so a mis-shaped tensor would
be read past its end).  Tensors here live on the CPU, so a call whose
arguments pass every check stops at the device check, before the library
runs anything."""
import pytest
import torch

import sequence_tensor_transformer_gb300 as st

BF = torch.bfloat16


def z(*shape, dtype=BF):
    return torch.zeros(shape, dtype=dtype)


def boundary_args(M=16, d=64, F=128, P=2):
    return dict(x=z(M, d), partials=z(P, M, d), gamma=z(d), W1g=z(F, d), W1u=z(F, d), W2=z(d, F))


def call_ffn(a, P=2, **kw):
    return st.sptp_ffn_forward(a["x"], a["partials"], a["gamma"], a["W1g"], a["W1u"], a["W2"], P, 2, 1e-6, **kw)


def test_consistent_arguments_reach_the_device_check():
    with pytest.raises(ValueError, match="device tensors only"):
        call_ffn(boundary_args())


@pytest.mark.parametrize("name,bad", [("partials", z(2, 16, 32)), ("partials", z(3, 16, 64)), ("gamma", z(32)),
                                      ("W1u", z(64, 64)), ("W2", z(128, 64)), ("W2", z(64, 64))])
def test_boundary_rejects_mis_shaped_tensors(name, bad):
    a = boundary_args()
    a[name] = bad
    with pytest.raises(ValueError, match=name):
        call_ffn(a)


def test_boundary_rejects_mixed_dtypes_and_bad_outputs():
    with pytest.raises(TypeError, match="W1u"):  # every tensor takes x's dtype
        call_ffn(dict(boundary_args(), W1u=z(128, 64, dtype=torch.float32)))
    with pytest.raises(ValueError, match="out"):
        call_ffn(boundary_args(), out=z(2, 16, 32))
    with pytest.raises(ValueError, match="resid_out"):
        call_ffn(boundary_args(), resid_out=z(16, 32))
    with pytest.raises(ValueError, match="out is required"):
        a = boundary_args()
        st.sptp_ffn_forward_noalloc(a["x"], a["partials"], a["gamma"], a["W1g"], a["W1u"], a["W2"], 2, 2, 1e-6,
                                    None)


def test_dtp_stack_checks_every_module_tensor():
    P, M, d, F, L = 2, 16, 64, 128, 3
    good = dict(x_shards=z(P, M, d), gamma=z(L, d), W1g=z(L, F, d), W1u=z(L, F, d), W2=z(L, d, F))
    call = lambda a: st.dtp_ffn_stack_forward(a["x_shards"], a["gamma"], a["W1g"], a["W1u"], a["W2"], P, L, 1, 1,
                                              1e-6)
    with pytest.raises(ValueError, match="device tensors only"):
        call(good)
    for name, bad in (("gamma", z(L - 1, d)), ("W1u", z(L, F, d // 2)), ("W2", z(L, F, d)),
                      ("x_shards", z(P + 1, M, d))):
        with pytest.raises(ValueError, match=name):
            call(dict(good, **{name: bad}))


def test_step_entry_points_check_shapes():
    with pytest.raises(ValueError, match="gamma"):
        st.sptp_prologue(z(16, 64), z(2, 16, 64), z(63), 1e-6)
    with pytest.raises(ValueError, match="W1u"):
        st.sptp_gateup_swiglu(z(16, 64), z(128, 64), z(128, 32), 2)
    with pytest.raises(ValueError, match="s_out"):
        st.sptp_gateup_swiglu(z(16, 64), z(128, 64), z(128, 64), 2, s_out=z(2, 16, 128))
    with pytest.raises(ValueError, match="s:"):
        st.sptp_down_proj(z(2, 16, 32), z(64, 128), 2)          # s must be [P, M, F/P] = [2, 16, 64]
    with pytest.raises(ValueError, match="Wqkv"):
        st.sptp_attn_qkv_forward(z(16, 64), z(2, 16, 64), z(64), z(96, 32), 2, 2, 1e-6)
    with pytest.raises(TypeError, match="perm"):
        st.sptp_permute_ffn_neurons(z(2, 128, 64), z(2, 128, 64), z(2, 64, 128), z(2, 128, dtype=torch.int64))
    with pytest.raises(ValueError, match="W2"):
        st.sptp_permute_ffn_neurons(z(2, 128, 64), z(2, 128, 64), z(2, 128, 64),
                                    z(2, 128, dtype=torch.int32))


def test_fp8_entry_points_check_codes_and_scales():
    P, M, d, F = 2, 16, 64, 128
    u8, f32 = torch.uint8, torch.float32
    qw = (z(F, d, dtype=u8), z(F, dtype=f32), z(F, d, dtype=u8), z(F, dtype=f32), z(d, F, dtype=u8),
          z(d, P, dtype=f32))
    with pytest.raises(ValueError, match="device tensors only"):
        st.sptp_ffn_forward_fp8(z(M, d), z(P, M, d), z(d), qw, P, 2, 1e-6)
    bad = list(qw)
    bad[5] = z(d, dtype=f32)                                   # one W2 scale per row instead of per (row, shard)
    with pytest.raises(ValueError, match="sW2"):
        st.sptp_ffn_forward_fp8(z(M, d), z(P, M, d), z(d), tuple(bad), P, 2, 1e-6)
    bad = list(qw)
    bad[0] = z(F, d)                                           # bf16 instead of E4M3 codes
    with pytest.raises(TypeError, match="qW1g"):
        st.sptp_ffn_forward_fp8(z(M, d), z(P, M, d), z(d), tuple(bad), P, 2, 1e-6)
    with pytest.raises(ValueError, match="scale"):
        st.sptp_quantize_rows_e4m3(z(4, 64), scale=z(4, 1, dtype=f32))
    with pytest.raises(ValueError, match="ss"):
        st.sptp_down_proj_e4m3(z(P, M, F // P, dtype=u8), z(M, dtype=f32), z(d, F, dtype=u8), z(d, P, dtype=f32), P)
    with pytest.raises(ValueError, match="W1u"):
        st.quantize_ffn_weights_e4m3(z(F, d), z(F, d + 16), z(d, F), P)


class OnDevice:
    """Stands for a CUDA tensor on device `index` (shape and dtype of `t`):
    enough for the binding's checks, which run before any pointer is taken."""

    def __init__(self, t, index):
        self.shape, self.dtype = t.shape, t.dtype
        self.device = torch.device("cuda", index)


def test_tensors_off_the_current_device_are_rejected_before_any_launch(monkeypatch):
    """The library launches on the current device and takes its stream and
    scratch from it: tensors on another device are refused by the binding,
    before the library is called."""
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)

    def no_library():
        raise AssertionError("the library was called")
    monkeypatch.setattr(st, "lib", no_library)
    a = {k: OnDevice(v, 1) for k, v in boundary_args().items()}
    with pytest.raises(ValueError, match="current device is cuda:0"):
        call_ffn(a)
    with pytest.raises(ValueError, match="current device is cuda:0"):
        st.sptp_prologue(a["x"], a["partials"], a["gamma"], 1e-6)
    with pytest.raises(ValueError, match="current device is cuda:0"):
        st.sptp_ffn_forward_noalloc(a["x"], a["partials"], a["gamma"], a["W1g"], a["W1u"], a["W2"], 2, 2, 1e-6,
                                    OnDevice(z(2, 16, 64), 1))
    # tensors split over two devices
    b = dict(a, W2=OnDevice(z(64, 128), 0))
    with pytest.raises(ValueError, match="one device expected"):
        call_ffn(b)


def test_unknown_variant_names_are_rejected():
    with pytest.raises(ValueError, match="unknown variant"):
        st._variant("single")
    assert [st._variant(v) for v in ("auto", "pair", "chain", "fused", "layers")] == [0, 1, 2, 3, 4]
