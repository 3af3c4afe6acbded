"""The C-ABI library builds, loads and exports every symbol include/moe.h
declares; host-side validation rejects bad configs before touching the GPU.
No compute call is made here (this runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_mixture_experts_gb300 import build
    build.build()
    import sparse_mixture_experts_gb300 as moe
    return moe.load_library()


def _declared_symbols():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for required in ("moe_layer_create", "moe_forward", "moe_destroy", "moe_get_routing", "moe_get_status",
                     "moe_last_error", "moe_forward_host"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_abi_version(lib):
    header = open(os.path.join(ROOT, "include", "moe.h")).read()
    version = int(re.search(r"#define MOE_ABI_VERSION (\d+)", header).group(1))
    assert lib.moe_abi_version() == version == 7


def test_config_struct_layout_matches_header():
    import sparse_mixture_experts_gb300 as moe
    # 18 four-byte fields, no padding
    assert ctypes.sizeof(moe._Config) == 18 * 4
    assert ctypes.sizeof(moe._Weights) == 14 * ctypes.sizeof(ctypes.c_void_p)


@pytest.mark.parametrize("bad", [
    dict(top_k=9),                 # top_k > n_expert
    dict(top_k=0),
    dict(hidden=0),
    dict(hidden=60),               # not a multiple of 8
    dict(router_mode=7),
    dict(act=5),
    dict(w_dtype=7),               # no such dtype
    dict(w_dtype=3, act_dtype=0),  # Q4 needs bf16 activations
    dict(resident_experts=-1),
    dict(resident_experts=8),      # not below n_expert
    dict(resident_experts=4),      # below min(n_expert, 16 * top_k): a chunk could select 8
    dict(w_dtype=2, act_dtype=1, gate_up_interleaved=0),  # MXFP4 needs the interleaved gate_up
    dict(w_dtype=2, act_dtype=0, gate_up_interleaved=1),  # MXFP4 needs bf16 activations
    dict(act_dtype=1, w_dtype=0),  # mixed activation / weight dtype
    dict(max_tokens=-1),
])
def test_create_rejects_bad_configs_on_the_host(lib, bad):
    import sparse_mixture_experts_gb300 as moe
    kw = dict(hidden=64, n_expert=8, top_k=2, expert_ff=32, w_dtype=moe.DT_F32, act_dtype=moe.DT_F32,
              max_tokens=16)
    kw.update(bad)
    cfg = moe.MoEConfig(**kw)._c()
    w = moe._Weights()
    h = ctypes.c_void_p()
    rc = lib.moe_layer_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h))
    assert rc in (moe.ERR_INVALID_ARG, moe.ERR_UNSUPPORTED)
    assert h.value is None
    assert lib.moe_last_error()


def test_null_arguments_are_rejected(lib):
    import sparse_mixture_experts_gb300 as moe
    assert lib.moe_layer_create(None, None, None) == moe.ERR_INVALID_ARG
    assert lib.moe_forward(None, None, 1, None, None) == moe.ERR_INVALID_ARG
    lib.moe_destroy(None)  # no-op


def test_binding_does_not_import_the_oracle():
    import subprocess
    import sys
    code = ("import sys, sparse_mixture_experts_gb300 as m; "
            "bad=[k for k in sys.modules if k=='oracle' or k.startswith('oracle.')]; "
            "print(bad); sys.exit(1 if bad else 0)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_settings_reject_a_null_layer(lib):
    import sparse_mixture_experts_gb300 as moe
    assert lib.moe_set_wait_limit(None, 1000) == moe.ERR_INVALID_ARG
    assert lib.moe_set_fault_injection(None, 1) == moe.ERR_INVALID_ARG
    assert lib.moe_get_intermediate(None, 0, None, 0, None, None) == moe.ERR_INVALID_ARG
    assert lib.moe_get_residency(None, None, None) == moe.ERR_INVALID_ARG
    assert lib.moe_last_token_count(None) == 0 and lib.moe_last_launch_count(None) == 0


def _unbound_layer(monkeypatch, calls):
    """A MoELayer with its checks intact but no device layer behind it: the
    library is a stand-in that records the calls it gets."""
    import torch
    import sparse_mixture_experts_gb300 as moe

    class _Lib:
        def moe_forward(self, *args):
            calls.append(("moe_forward",) + args)
            return moe.OK

        def moe_forward_host(self, *args):
            calls.append(("moe_forward_host",) + args)
            return moe.OK

        def moe_last_token_count(self, h):
            return 4

    monkeypatch.setattr(moe, "_lib", _Lib())
    layer = object.__new__(moe.MoELayer)
    layer.config = moe.MoEConfig(hidden=64, n_expert=8, top_k=2, expert_ff=32, max_tokens=16)
    layer.device = torch.device("cuda", 0)
    layer.x_dtype, layer.out_dtype = torch.bfloat16, torch.float32
    layer._h = ctypes.c_void_p()
    return layer


def test_binding_checks_token_rows_before_the_call(monkeypatch):
    """The ABI takes bare pointers, so a tensor of the wrong shape, dtype,
    layout or device is refused by the binding before any call."""
    import torch
    calls = []
    layer = _unbound_layer(monkeypatch, calls)
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    out = torch.zeros((4, 64), dtype=torch.float32)
    bad_x = [torch.zeros((4, 63), dtype=torch.bfloat16),        # hidden
             torch.zeros((4, 64), dtype=torch.float32),         # dtype
             torch.zeros((64, 4), dtype=torch.bfloat16).t(),    # layout
             torch.zeros((4, 1, 64), dtype=torch.bfloat16),     # rank
             x]                                                 # a host tensor for the device entry point
    for t in bad_x:
        with pytest.raises(ValueError):
            layer.forward(t, stream=0)
    bad_out = [torch.zeros((3, 64), dtype=torch.float32),       # rows
               torch.zeros((4, 64), dtype=torch.bfloat16),      # dtype
               torch.zeros((64, 4), dtype=torch.float32).t()]   # layout
    for o in bad_out:
        with pytest.raises(ValueError):
            layer.forward_host(x, o, stream=0)
    with pytest.raises(ValueError):
        layer.forward_host(torch.zeros((4, 64), dtype=torch.float32), out, stream=0)
    assert not calls
    # well-formed host buffers reach the library with their pointers and count
    layer.forward_host(x, out, stream=0)
    layer.forward_host(x[:0], out[:0], stream=0)
    assert calls == [("moe_forward_host", layer._h, x.data_ptr(), 4, out.data_ptr(), 0),
                     ("moe_forward_host", layer._h, None, 0, None, 0)]


def test_binding_getters_take_the_last_forwards_rows(monkeypatch):
    """routing() and logits() size their buffers from the layer's last
    forward; a caller's different count is refused before any allocation."""
    calls = []
    layer = _unbound_layer(monkeypatch, calls)
    assert layer._last_tokens(None) == 4 and layer._last_tokens(4) == 4
    for n in (3, 5):
        with pytest.raises(ValueError):
            layer.routing(n)
        with pytest.raises(ValueError):
            layer.logits(n)
