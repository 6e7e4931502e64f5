"""Host-side checks of the C ABI: the library loads, exports every entry point
the header declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "linattn.h")


@pytest.fixture(scope="module")
def lib():
    import kernelized_linear_attention_gb300 as la
    if not os.path.exists(la.library_path()):
        from kernelized_linear_attention_gb300 import build
        build.build()
    return la.load_library()


def declared_entry_points():
    text = open(HEADER).read()
    return re.findall(r"LA_API\s+[\w\s\*]+?\b(la_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_entry_points())
    for need in ("la_feature_map", "la_forward_bidir", "la_forward_causal", "la_workspace_bytes",
                 "la_check_cu_seqlens", "la_status_string"):
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_entry_points()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/linattn.h but not exported"


def test_only_the_abi_is_exported(lib):
    import subprocess
    import kernelized_linear_attention_gb300 as la
    out = subprocess.run(["nm", "-D", "--defined-only", la.library_path()], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm unavailable")
    funcs = {l.split()[-1] for l in out.stdout.splitlines() if " T " in l}
    assert funcs == set(declared_entry_points())


def test_status_strings_and_version(lib):
    import kernelized_linear_attention_gb300 as la
    assert la.la_status_string(0) == "ok"
    assert "workspace" in la.la_status_string(3)
    assert la.la_version() >= 100


FWD = ["la_forward_bidir", "la_forward_causal"]


def _fwd(lib, name, **kw):
    a = dict(q=1 << 20, k=1 << 20, v=1 << 20, omega=1 << 20, map=2, dtype=1, cu=None, nseq=1, T=128, H=2,
             dk=64, dv=64, r=256, eps=1e-6, out=1 << 21, ws=1 << 22, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    fn = getattr(lib, name)
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                           ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                           ctypes.c_void_p]
    return fn(a["q"], a["k"], a["v"], a["omega"], a["map"], a["dtype"], a["cu"], a["nseq"], a["T"], a["H"],
              a["dk"], a["dv"], a["r"], a["eps"], a["out"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("name", FWD)
@pytest.mark.parametrize("bad,code", [
    (dict(map=7), 1), (dict(dtype=5), 1), (dict(nseq=0), 1), (dict(H=0), 1), (dict(T=-1), 1),
    (dict(dk=0), 1), (dict(map=1, r=256), 1),          # ELU+1 needs r == d_k
    (dict(map=0, r=32), 1),                             # identity needs r == d_k
    (dict(T=130, nseq=4), 1),                           # equal lengths need nseq | T
    (dict(omega=None), 1),                              # FAVOR+ needs omega
    (dict(eps=-1.0), 1), (dict(eps=float("nan")), 1), (dict(eps=float("inf")), 1),
    (dict(ws=None), 1), (dict(ws=(1 << 22) + 16), 1),   # workspace must be 256-byte aligned
    (dict(q=None), 1), (dict(out=None), 1),
    (dict(q=(1 << 20) + 1), 1),                         # misaligned for bf16
    (dict(dk=300, r=300, map=1), 2), (dict(r=1024), 2), (dict(dv=512), 2),
    (dict(map=3, r=100), 1),                            # DPFP needs r = 2 d_k nu
    (dict(map=3, dk=2, dv=2, r=16), 1),                 # and nu <= 2 d_k - 1
    (dict(map=4), 1),
])
def test_forward_rejects_bad_arguments_on_host(lib, name, bad, code):
    assert _fwd(lib, name, **bad) == code


def test_selected_path_and_workspace_queries_reject_bad_shapes(lib):
    import kernelized_linear_attention_gb300 as la
    assert la.la_selected_path(True, "elu1", 1, 64, 64, 128) == -1
    assert la.la_selected_path(True, "favor", 1, 64, 64, 256) in (0, 1)
    assert la.la_selected_path(True, "favor", 0, 64, 64, 256) == 0        # fp32 always on CUDA cores
    assert la.la_workspace_bytes(True, "elu1", 1, False, 3, 100, 2, 64, 64, 64) == 0   # 3 does not divide 100
    assert la.la_selected_path(True, "dpfp2", 1, 64, 64, 256) == 1      # causal DPFP-1/-2 on tensor cores
    assert la.la_selected_path(True, "dpfp1", 1, 64, 64, 128) == 1
    assert la.la_selected_path(False, "dpfp2", 1, 64, 64, 256) == 0     # bidirectional DPFP on CUDA cores
    assert la.la_selected_path(True, "dpfp3", 1, 64, 64, 384) == 0      # r above the kernels' 256
    assert la.la_selected_path(False, "dpfp1", 0, 64, 64, 128) == 0
    assert la.la_selected_path(True, "dpfp1", 1, 64, 64, 64) == -1      # r = 2 d_k nu


def test_feature_map_rejects_bad_arguments(lib):
    fn = lib.la_feature_map
    assert fn(1 << 20, None, 2, 1, 128, 2, 64, 256, 1 << 21, None) == 1     # FAVOR+ without omega
    assert fn(1 << 20, None, 1, 1, 128, 2, 64, 32, 1 << 21, None) == 1      # ELU+1 with r != d
    assert fn(None, None, 1, 1, 128, 2, 64, 64, 1 << 21, None) == 1
    assert fn(1 << 20, None, 1, 1, 0, 2, 64, 64, None, None) == 0           # T = 0: nothing to do
    assert fn(1 << 20, None, 3, 1, 128, 2, 64, 192, 1 << 21, None) == 1     # DPFP: r not 2 d nu
    assert fn(1 << 20, None, 3, 1, 0, 2, 64, 256, None, None) == 0          # DPFP-2, T = 0


def test_orthogonal_features_rejects_bad_arguments(lib):
    fn = lib.la_orthogonal_features
    assert fn(None, 1 << 20, 4, 2, 1 << 21, None) == 1
    assert fn(1 << 20, 1 << 20, 0, 2, 1 << 21, None) == 1
    assert fn(1 << 20, 1 << 20, 4, 256, 1 << 21, None) == 2


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    import kernelized_linear_attention_gb300 as la
    x = torch.zeros(4, 1, 8)
    with pytest.raises(ValueError):
        la.la_forward_causal(x, x, x, "elu1")


def _fwd_general(lib, **kw):
    a = dict(causal=1, norm=0, q=1 << 20, k=1 << 20, v=1 << 20, omega=1 << 20, map=2, dtype=1, cu=None, nseq=1,
             T=128, H=2, dk=64, dv=64, r=256, eps=1e-6, state_in=None, state_out=None, out=1 << 21, ws=1 << 22,
             ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.la_forward(a["causal"], a["norm"], a["q"], a["k"], a["v"], a["omega"], a["map"], a["dtype"], a["cu"],
                          a["nseq"], a["T"], a["H"], a["dk"], a["dv"], a["r"], a["eps"], a["state_in"],
                          a["state_out"], a["out"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("bad,code", [
    (dict(norm=3), 1), (dict(norm=-1), 1),
    (dict(norm=2, map=0, r=64), 1),                     # sum normalisation needs non-negative features
    (dict(state_in=(1 << 23) + 2), 1), (dict(state_out=(1 << 23) + 1), 1),   # fp32 state alignment
    (dict(map=1, r=256), 1), (dict(omega=None), 1), (dict(eps=-1.0), 1), (dict(ws=None), 1),
    (dict(dv=512), 2),
])
def test_general_forward_rejects_bad_arguments_on_host(lib, causal, bad, code):
    assert _fwd_general(lib, causal=causal, **bad) == code


def _decode(lib, **kw):
    a = dict(q=1 << 20, k=1 << 20, v=1 << 20, omega=1 << 20, map=2, dtype=1, norm=0, B=4, H=2, dk=64, dv=64,
             r=256, eps=1e-6, state=1 << 22, out=1 << 21, stream=None)
    a.update(kw)
    return lib.la_decode_step(a["q"], a["k"], a["v"], a["omega"], a["map"], a["dtype"], a["norm"], a["B"], a["H"],
                              a["dk"], a["dv"], a["r"], a["eps"], a["state"], a["out"], a["stream"])


@pytest.mark.parametrize("bad,code", [
    (dict(B=-1), 1), (dict(H=0), 1), (dict(map=7), 1), (dict(dtype=3), 1), (dict(norm=4), 1),
    (dict(norm=2, map=0, r=64), 1), (dict(omega=None), 1), (dict(map=1, r=128), 1),
    (dict(eps=-1.0), 1), (dict(eps=float("nan")), 1),
    (dict(state=None), 1), (dict(out=None), 1), (dict(q=None), 1),
    (dict(state=(1 << 22) + 2), 1), (dict(q=(1 << 20) + 1), 1),
    (dict(dk=300, r=300, map=1), 2), (dict(r=1024), 2),
    (dict(B=0), 0),                                     # nothing to do: returns before any launch
    (dict(B=0, state=None, out=None), 0),
])
def test_decode_step_rejects_bad_arguments_on_host(lib, bad, code):
    assert _decode(lib, **bad) == code


def test_binding_checks_state_shapes_and_devices():
    torch = pytest.importorskip("torch")
    import kernelized_linear_attention_gb300 as la
    x = torch.zeros(2, 1, 8)
    st = torch.zeros(2, 1, 8, 9)
    with pytest.raises(ValueError):
        la.la_decode_step(x, x, x, st, "elu1")
    with pytest.raises(ValueError):
        la.la_forward(x, x, x, "elu1", norm="sum", state_in=st)
    from kernelized_linear_attention_gb300._binding import _norm_id
    assert [_norm_id(n) for n in ("attention", "none", "sum")] == [0, 1, 2]
    with pytest.raises(KeyError):
        _norm_id("softmax")


def _bwd(lib, **kw):
    a = dict(causal=1, norm=0, q=1 << 20, k=1 << 20, v=1 << 20, omega=1 << 20, map=2, dtype=1, cu=None, nseq=1,
             T=128, H=2, dk=64, dv=64, r=256, eps=1e-6, dout=1 << 21, dq=1 << 22, dk_=1 << 23, dv_=1 << 24,
             ws=1 << 25, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.la_backward(a["causal"], a["norm"], a["q"], a["k"], a["v"], a["omega"], a["map"], a["dtype"], a["cu"],
                           a["nseq"], a["T"], a["H"], a["dk"], a["dv"], a["r"], a["eps"], a["dout"], a["dq"],
                           a["dk_"], a["dv_"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("bad,code", [
    (dict(norm=3), 1), (dict(norm=2, map=0, r=64), 1), (dict(map=7), 1), (dict(dtype=4), 1),
    (dict(omega=None), 1), (dict(map=1, r=128), 1), (dict(eps=-1.0), 1), (dict(ws=None), 1),
    (dict(ws=(1 << 25) + 8), 1), (dict(dout=None), 1), (dict(dq=None), 1), (dict(dv_=None), 1),
    (dict(dk_=(1 << 23) + 1), 1), (dict(T=130, nseq=4), 1),
    (dict(r=512, dv=256), 2),                           # state does not fit the CUDA-core kernels' shared memory
])
def test_backward_rejects_bad_arguments_on_host(lib, bad, code):
    assert _bwd(lib, **bad) == code


def test_backward_workspace_query_rejects_bad_shapes(lib):
    import kernelized_linear_attention_gb300 as la
    assert la.la_backward_workspace_bytes(True, "elu1", 1, False, 3, 100, 2, 64, 64, 64) == 0
    assert la.la_backward_workspace_bytes(True, "favor", 1, False, 1, 128, 2, 64, 256, 512) == 0
