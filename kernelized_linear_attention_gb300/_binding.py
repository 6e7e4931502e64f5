"""ctypes binding of liblinattn.so (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "lib", "liblinattn.so")

MAP_IDS = {"identity": 0, "elu1": 1, "favor": 2, "dpfp": 3}
DTYPE_IDS = {torch.float32: 0, torch.bfloat16: 1}
NORM_IDS = {"attention": 0, "none": 1, "sum": 2}

LA_OK = 0
_c_i64, _c_int, _c_float, _c_size, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

_lib = None


class LinAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({la_status_string(status)})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load liblinattn.so once.  Raises if it was not built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"` "
            "(kernelized linear attention has no CPU fallback)")
    lib = ctypes.CDLL(_LIB_PATH)
    fwd_args = [_vp, _vp, _vp, _vp, _c_int, _c_int, _vp, _c_int, _c_i64, _c_int, _c_int, _c_int, _c_int,
                _c_float, _vp, _vp, _c_size, _vp]
    sigs = {
        "la_feature_map": ([_vp, _vp, _c_int, _c_int, _c_i64, _c_int, _c_int, _c_int, _vp, _vp], _c_int),
        "la_forward_bidir": (fwd_args, _c_int),
        "la_forward_causal": (fwd_args, _c_int),
        "la_forward_phase": ([_c_int, _c_int, _c_int] + fwd_args[:14] + [_vp, _vp] + fwd_args[14:]
                             + [ctypes.POINTER(_c_int)], _c_int),
        "la_forward": ([_c_int, _c_int] + fwd_args[:14] + [_vp, _vp] + fwd_args[14:], _c_int),
        "la_backward": ([_c_int, _c_int] + fwd_args[:14] + [_vp, _vp, _vp, _vp] + fwd_args[15:], _c_int),
        "la_backward_workspace_bytes": ([_c_int, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_int, _c_int, _c_int,
                                         _c_int], _c_size),
        "la_decode_step": ([_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                            _c_float, _vp, _vp, _vp], _c_int),
        "la_forward_causal_noalloc": (fwd_args[:15] + [_vp], _c_int),
        "la_noalloc_error": ([ctypes.POINTER(_c_int), _vp], _c_int),
        "la_test_force_wait_timeout": ([_c_int], _c_int),
        "la_test_segment_plan": ([_c_i64, _c_i64, _c_int, _c_i64, ctypes.POINTER(_c_i64)], _c_i64),
        "la_workspace_bytes": ([_c_int, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_int, _c_int, _c_int, _c_int],
                               _c_size),
        "la_check_cu_seqlens": ([_vp, _c_int, _c_i64, _vp], _c_int),
        "la_workspace_error": ([_vp, ctypes.POINTER(_c_int), _vp], _c_int),
        "la_orthogonal_features": ([_vp, _vp, _c_int, _c_int, _vp, _vp], _c_int),
        "la_selected_path": ([_c_int, _c_int, _c_int, _c_int, _c_int, _c_int], _c_int),
        "la_status_string": ([_c_int], ctypes.c_char_p),
        "la_version": ([], _c_int),
    }
    for name, (argtypes, restype) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = argtypes
        fn.restype = restype
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != LA_OK:
        raise LinAttnError(fn, status)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype=None, cuda=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _map_id(m) -> int:
    """Map id from a name ("identity", "elu1", "favor", "dpfp<nu>") or an id."""
    if isinstance(m, str):
        return MAP_IDS["dpfp"] if m.startswith("dpfp") else MAP_IDS[m]
    return int(m)


def _norm_id(n) -> int:
    """Normalisation id from a name ("attention", "none", "sum") or an id."""
    return NORM_IDS[n] if isinstance(n, str) else int(n)


def _feature_dim(m, d_k: int, omega) -> int:
    """r of a map: Omega's rows (FAVOR+), 2 d_k nu (DPFP-nu, named "dpfp<nu>"), else d_k."""
    if _map_id(m) == MAP_IDS["favor"]:
        return omega.shape[0]
    if _map_id(m) == MAP_IDS["dpfp"]:
        if not (isinstance(m, str) and m[4:].isdigit()):
            raise ValueError('the DPFP map is named "dpfp<nu>", e.g. "dpfp2"')
        return 2 * d_k * int(m[4:])
    return d_k


def la_status_string(status: int) -> str:
    return load_library().la_status_string(int(status)).decode()


def la_version() -> int:
    return load_library().la_version()


def la_selected_path(causal: bool, map, dtype, d_k: int, d_v: int, r: int) -> int:
    dt = DTYPE_IDS[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return load_library().la_selected_path(int(causal), _map_id(map), dt, d_k, d_v, r)


def la_workspace_bytes(causal: bool, map, dtype, has_cu_seqlens: bool, nseq: int, T: int, H: int,
                       d_k: int, d_v: int, r: int) -> int:
    dt = DTYPE_IDS[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return load_library().la_workspace_bytes(int(causal), _map_id(map), dt, int(has_cu_seqlens), nseq, T, H,
                                             d_k, d_v, r)


def la_feature_map(x: torch.Tensor, map, omega: Optional[torch.Tensor] = None,
                   phi: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """phi(x) for x [T, H, d] (fp32 or bf16) -> fp32 [T, H, r]."""
    lib = load_library()
    _need(x, "x")
    m = _map_id(map)
    T, H, d = x.shape
    r = _feature_dim(map, d, omega)
    if omega is not None:
        _need(omega, "omega", torch.float32)
    if phi is None:
        phi = torch.empty((T, H, r), dtype=torch.float32, device=x.device)
    _need(phi, "phi", torch.float32)
    _check("la_feature_map", lib.la_feature_map(_ptr(x), _ptr(omega), m, DTYPE_IDS[x.dtype], T, H, d, r,
                                                _ptr(phi), _stream(stream)))
    return phi


def forward_ptrs(causal: bool, q, k, v, omega, map, dtype, cu_seqlens, nseq, T, H, d_k, d_v, r, eps,
                 out, workspace, workspace_bytes, stream) -> None:
    """Raw call with integer device pointers (for callers that manage memory)."""
    lib = load_library()
    fn = lib.la_forward_causal if causal else lib.la_forward_bidir
    dt = DTYPE_IDS[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    _check(fn.__name__, fn(q, k, v, omega, _map_id(map), dt, cu_seqlens, nseq, T, H, d_k, d_v, r, eps,
                           out, workspace, workspace_bytes, _stream(stream)))


def forward_general_ptrs(causal: bool, q, k, v, omega, map, dtype, cu_seqlens, nseq, T, H, d_k, d_v, r, eps,
                         out, workspace, workspace_bytes, stream, norm="attention", state_in=None,
                         state_out=None) -> None:
    """Raw la_forward call with integer device pointers (state_in / state_out too)."""
    dt = DTYPE_IDS[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    _check("la_forward", load_library().la_forward(int(causal), _norm_id(norm), q, k, v, omega, _map_id(map), dt,
                                                   cu_seqlens, nseq, T, H, d_k, d_v, r, eps, state_in, state_out,
                                                   out, workspace, workspace_bytes, _stream(stream)))


def la_forward_phase(causal: bool, phase: int, q, k, v, omega, map, dtype, cu_seqlens, nseq, T, H, d_k, d_v, r,
                     eps, out, workspace, workspace_bytes, stream=None, norm="attention", state_in=None,
                     state_out=None) -> int:
    """One phase (0 plan, 1 state, 2 scan, 3 output) with integer device
    pointers (state_in / state_out too); returns the number of kernels it
    enqueued."""
    lib = load_library()
    dt = DTYPE_IDS[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    n = _c_int(0)
    _check("la_forward_phase", lib.la_forward_phase(int(causal), int(phase), _norm_id(norm), q, k, v, omega,
                                                    _map_id(map), dt, cu_seqlens, nseq, T, H, d_k, d_v, r, eps,
                                                    state_in, state_out, out, workspace, workspace_bytes,
                                                    _stream(stream), ctypes.byref(n)))
    return n.value


def la_forward_causal_noalloc(q, k, v, map, omega=None, cu_seqlens=None, nseq=None, eps=1e-6, out=None,
                              stream=None) -> torch.Tensor:
    """Causal forward whose scratch is the library's fixed device array (no
    workspace, no device allocation inside the library); see
    include/linattn.h for the sharing rules."""
    _need(q, "q"); _need(k, "k"); _need(v, "v")
    T, H, d_k = q.shape
    d_v = v.shape[2]
    m = _map_id(map)
    r = _feature_dim(map, d_k, omega)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        nseq = cu_seqlens.numel() - 1
    elif nseq is None:
        nseq = 1
    if out is None:
        out = torch.empty((T, H, d_v), dtype=q.dtype, device=q.device)
    _need(out, "out", q.dtype)
    _check("la_forward_causal_noalloc", load_library().la_forward_causal_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(omega), m, DTYPE_IDS[q.dtype], _ptr(cu_seqlens), nseq, T, H, d_k, d_v, r,
        eps, _ptr(out), _stream(stream)))
    return out


def la_test_force_wait_timeout(enable: bool) -> None:
    """Test hook: while enabled, the causal tensor-core output kernel's bounded waits are made
    to run out (it records LA_DEVERR_WAIT_TIMEOUT and returns); see include/linattn.h."""
    st = load_library().la_test_force_wait_timeout(1 if enable else 0)
    if st != LA_OK:
        raise LinAttnError("la_test_force_wait_timeout", st)


def la_test_segment_plan(nchunks: int, pairs: int, nsm: int, force_chunks: int = 0):
    """Test hook (host only): (segment length in chunks, simulated makespan in chunk times)
    the tensor-core planner chooses, or evaluates for force_chunks; see include/linattn.h."""
    ms = _c_i64(0)
    lc = load_library().la_test_segment_plan(nchunks, pairs, nsm, force_chunks, ctypes.byref(ms))
    if lc < 0:
        raise ValueError("la_test_segment_plan: nchunks, pairs and nsm must be at least 1")
    return int(lc), int(ms.value)


def la_noalloc_error(stream=None) -> int:
    """Device error code the latest la_forward_causal_noalloc call on the current
    device recorded in the library's scratch array (0 = none; synchronises)."""
    code = _c_int(0)
    st = load_library().la_noalloc_error(ctypes.byref(code), _stream(stream))
    if st not in (LA_OK, 5):
        raise LinAttnError("la_noalloc_error", st)
    return code.value


def _forward(causal, q, k, v, map, omega, cu_seqlens, nseq, eps, out, workspace, stream, norm="attention",
             state_in=None, state_out=None):
    _need(q, "q"); _need(k, "k"); _need(v, "v")
    if q.dtype not in DTYPE_IDS or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share dtype float32 or bfloat16")
    T, H, d_k = q.shape
    d_v = v.shape[2]
    m = _map_id(map)
    r = _feature_dim(map, d_k, omega)
    if omega is not None:
        _need(omega, "omega", torch.float32)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        nseq = cu_seqlens.numel() - 1
    elif nseq is None:
        nseq = 1
    for name, st in (("state_in", state_in), ("state_out", state_out)):
        if st is not None:
            _need(st, name, torch.float32)
            if tuple(st.shape) != (nseq, H, r, d_v + 1):
                raise ValueError(f"{name} must have shape {(nseq, H, r, d_v + 1)}, got {tuple(st.shape)}")
    if out is None:
        out = torch.empty((T, H, d_v), dtype=q.dtype, device=q.device)
    _need(out, "out", q.dtype)
    need = la_workspace_bytes(causal, m, q.dtype, cu_seqlens is not None, nseq, T, H, d_k, d_v, r)
    if workspace is None:
        # a size of 0 means the call will be rejected: let the library say why
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    nid = _norm_id(norm)
    if nid == NORM_IDS["attention"] and state_in is None and state_out is None:
        forward_ptrs(causal, _ptr(q), _ptr(k), _ptr(v), _ptr(omega), m, q.dtype, _ptr(cu_seqlens), nseq, T, H,
                     d_k, d_v, r, eps, _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                     stream)
    else:
        _check("la_forward", load_library().la_forward(
            int(causal), nid, _ptr(q), _ptr(k), _ptr(v), _ptr(omega), m, DTYPE_IDS[q.dtype], _ptr(cu_seqlens),
            nseq, T, H, d_k, d_v, r, eps, _ptr(state_in), _ptr(state_out), _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, workspace


def la_forward_bidir(q, k, v, map, omega=None, cu_seqlens=None, nseq=None, eps=1e-6, out=None,
                     workspace=None, stream=None) -> torch.Tensor:
    """Bidirectional kernelized attention; returns out [T, H, d_v] (dtype of q)."""
    return _forward(False, q, k, v, map, omega, cu_seqlens, nseq, eps, out, workspace, stream)[0]


def la_forward_causal(q, k, v, map, omega=None, cu_seqlens=None, nseq=None, eps=1e-6, out=None,
                      workspace=None, stream=None) -> torch.Tensor:
    """Causal kernelized attention; returns out [T, H, d_v] (dtype of q)."""
    return _forward(True, q, k, v, map, omega, cu_seqlens, nseq, eps, out, workspace, stream)[0]


def la_forward(q, k, v, map, omega=None, causal=True, norm="attention", cu_seqlens=None, nseq=None, eps=1e-6,
               state_in=None, state_out=None, return_state=False, out=None, workspace=None, stream=None):
    """General forward: norm "attention" | "none" | "sum", optional carried
    state.  state_in / state_out: fp32 [nseq, H, r, d_v + 1] (row f: S[f, :]
    then z[f]).  With return_state=True a state_out is allocated when none is
    given and (out, state_out) is returned."""
    if return_state and state_out is None:
        T, H, d_k = q.shape
        nn = cu_seqlens.numel() - 1 if cu_seqlens is not None else (nseq or 1)
        r = _feature_dim(map, d_k, omega)
        state_out = torch.empty((nn, H, r, v.shape[2] + 1), dtype=torch.float32, device=q.device)
    o = _forward(bool(causal), q, k, v, map, omega, cu_seqlens, nseq, eps, out, workspace, stream, norm=norm,
                 state_in=state_in, state_out=state_out)[0]
    return (o, state_out) if return_state else o


def la_decode_step(q, k, v, state, map, omega=None, norm="attention", eps=1e-6, out=None, stream=None):
    """One token per sequence: q, k [B, H, d_k], v [B, H, d_v]; state fp32
    [B, H, r, d_v + 1] is updated in place; returns out [B, H, d_v]."""
    _need(q, "q"); _need(k, "k"); _need(v, "v"); _need(state, "state", torch.float32)
    if q.dtype not in DTYPE_IDS or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share dtype float32 or bfloat16")
    B, H, d_k = q.shape
    d_v = v.shape[2]
    r = _feature_dim(map, d_k, omega)
    if tuple(state.shape) != (B, H, r, d_v + 1):
        raise ValueError(f"state must have shape {(B, H, r, d_v + 1)}, got {tuple(state.shape)}")
    if omega is not None:
        _need(omega, "omega", torch.float32)
    if out is None:
        out = torch.empty((B, H, d_v), dtype=q.dtype, device=q.device)
    _need(out, "out", q.dtype)
    _check("la_decode_step", load_library().la_decode_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(omega), _map_id(map), DTYPE_IDS[q.dtype], _norm_id(norm), B, H, d_k, d_v,
        r, eps, _ptr(state), _ptr(out), _stream(stream)))
    return out


def la_backward_workspace_bytes(causal: bool, map, dtype, has_cu_seqlens: bool, nseq: int, T: int, H: int,
                                d_k: int, d_v: int, r: int) -> int:
    dt = DTYPE_IDS[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return load_library().la_backward_workspace_bytes(int(causal), _map_id(map), dt, int(has_cu_seqlens), nseq, T,
                                                      H, d_k, d_v, r)


def la_backward(q, k, v, dout, map, omega=None, causal=True, norm="attention", cu_seqlens=None, nseq=None,
                eps=1e-6, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of sum(dout * out) for the forward with the same
    arguments; allocates what is not given."""
    _need(q, "q"); _need(k, "k"); _need(v, "v"); _need(dout, "dout")
    if q.dtype not in DTYPE_IDS or any(t.dtype != q.dtype for t in (k, v, dout)):
        raise ValueError("q, k, v, dout must share dtype float32 or bfloat16")
    T, H, d_k = q.shape
    d_v = v.shape[2]
    m = _map_id(map)
    r = _feature_dim(map, d_k, omega)
    if omega is not None:
        _need(omega, "omega", torch.float32)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        nseq = cu_seqlens.numel() - 1
    elif nseq is None:
        nseq = 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _need(t, name, q.dtype)
    need = la_backward_workspace_bytes(causal, m, q.dtype, cu_seqlens is not None, nseq, T, H, d_k, d_v, r)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check("la_backward", load_library().la_backward(
        int(causal), _norm_id(norm), _ptr(q), _ptr(k), _ptr(v), _ptr(omega), m, DTYPE_IDS[q.dtype],
        _ptr(cu_seqlens), nseq, T, H, d_k, d_v, r, eps, _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return dq, dk, dv


def attention(q, k, v, map="favor", omega=None, causal=True, cu_seqlens=None, nseq=None, eps=1e-6,
              out=None, workspace=None, stream=None, return_workspace=False, norm="attention"):
    """Convenience wrapper: allocates out/workspace with torch, calls the library."""
    o, ws = _forward(bool(causal), q, k, v, map, omega, cu_seqlens, nseq, eps, out, workspace, stream, norm=norm)
    return (o, ws) if return_workspace else o


def la_check_cu_seqlens(cu_seqlens: torch.Tensor, T: int, stream=None) -> bool:
    """True when cu_seqlens obeys the packing rules (synchronises)."""
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    st = load_library().la_check_cu_seqlens(_ptr(cu_seqlens), cu_seqlens.numel() - 1, T, _stream(stream))
    if st not in (LA_OK, 1):
        raise LinAttnError("la_check_cu_seqlens", st)
    return st == LA_OK


def la_workspace_error(workspace: torch.Tensor, stream=None) -> int:
    """Device error code recorded in a workspace (0 = none; synchronises)."""
    code = _c_int(0)
    st = load_library().la_workspace_error(_ptr(workspace), ctypes.byref(code), _stream(stream))
    if st not in (LA_OK, 5):
        raise LinAttnError("la_workspace_error", st)
    return code.value


def la_orthogonal_features(gauss_blocks: torch.Tensor, gauss_lengths: torch.Tensor, r: int,
                           omega: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Orthogonal random-feature matrix [r, d] fp32 from fp64 Gaussian draws."""
    _need(gauss_blocks, "gauss_blocks", torch.float64)
    _need(gauss_lengths, "gauss_lengths", torch.float64)
    d = gauss_blocks.shape[-1]
    if omega is None:
        omega = torch.empty((r, d), dtype=torch.float32, device=gauss_blocks.device)
    _need(omega, "omega", torch.float32)
    _check("la_orthogonal_features", load_library().la_orthogonal_features(
        _ptr(gauss_blocks), _ptr(gauss_lengths), r, d, _ptr(omega), _stream(stream)))
    return omega
