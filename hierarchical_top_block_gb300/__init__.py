"""GB300 (sm_103a) log-linear block-sparse attention with pyramid-LSE block selection.

Python binding of the C ABI in ``include/pisa.h`` (library ``libpisa_gb300.so``).  The
functions carry the C names and only marshal arguments: every step of the computation
runs in the library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  If the library is missing, every call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes as ct
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpisa_gb300.so")

PISA_OK = 0
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "device wait timed out",
           5: "bad block index", 6: "workspace too small"}


class PisaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(status, status)} (status {status})")
        self.status = status


class pisa_params(ct.Structure):
    _fields_ = [("C", ct.c_int), ("g", ct.c_int), ("K", ct.c_int), ("causal", ct.c_int), ("scale", ct.c_float),
                ("scoring", ct.c_int)]


class pisa_shape(ct.Structure):
    _fields_ = [("B", ct.c_int), ("N", ct.c_int), ("H_q", ct.c_int), ("H_kv", ct.c_int), ("d", ct.c_int),
                ("N_cap", ct.c_int)]


_lib = None
_P = ct.c_void_p


def lib() -> ct.CDLL:
    """Load the library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with hierarchical_top_block_gb300.build.build()")
        L = ct.CDLL(LIB_PATH)
        L.pisa_pyramid_levels.restype = ct.c_int
        L.pisa_pyramid_levels.argtypes = [ct.c_longlong, ct.c_int, ct.c_int]
        L.pisa_pyramid_nodes.restype = ct.c_longlong
        L.pisa_pyramid_nodes.argtypes = [ct.c_longlong, ct.c_int, ct.c_int]
        L.pisa_select_workspace_bytes.restype = ct.c_size_t
        L.pisa_select_workspace_bytes.argtypes = [pisa_shape, pisa_params]
        L.pisa_attn_backward_workspace_bytes.restype = ct.c_size_t
        L.pisa_attn_backward_workspace_bytes.argtypes = [pisa_shape, pisa_params]
        L.pisa_attn_backward_min_workspace_bytes.restype = ct.c_size_t
        L.pisa_attn_backward_min_workspace_bytes.argtypes = [pisa_shape, pisa_params]
        L.pisa_sparse_attn_backward.restype = ct.c_int
        L.pisa_sparse_attn_backward.argtypes = [_P] * 10 + [_P, ct.c_size_t, pisa_shape, pisa_params, _P]
        L.pisa_prefill_host_workspace_bytes.restype = ct.c_size_t
        L.pisa_prefill_host_workspace_bytes.argtypes = [pisa_shape, pisa_params]
        L.pisa_prefill_host_chunks.restype = ct.c_int
        L.pisa_prefill_host_chunks.argtypes = [ct.c_longlong, ct.POINTER(ct.c_longlong), ct.c_int]
        L.pisa_build_pyramid.restype = ct.c_int
        L.pisa_build_pyramid.argtypes = [_P, _P, pisa_shape, pisa_params, _P]
        L.pisa_select_prefill.restype = ct.c_int
        L.pisa_select_prefill.argtypes = [_P, _P, _P, _P, _P, _P, _P, ct.c_size_t, pisa_shape, pisa_params, _P]
        L.pisa_select_prefill_noalloc.restype = ct.c_int
        L.pisa_select_prefill_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, pisa_shape, pisa_params, _P]
        L.pisa_select_bsa_workspace_bytes.restype = ct.c_size_t
        L.pisa_select_bsa_workspace_bytes.argtypes = [pisa_shape, pisa_params]
        L.pisa_select_bsa.restype = ct.c_int
        L.pisa_select_bsa.argtypes = [_P, _P, _P, _P, ct.c_size_t, pisa_shape, pisa_params, _P]
        L.pisa_sparse_attn_prefill.restype = ct.c_int
        L.pisa_sparse_attn_prefill.argtypes = [_P, _P, _P, _P, _P, _P, pisa_shape, pisa_params, _P]
        L.pisa_prefill_host.restype = ct.c_int
        L.pisa_prefill_host.argtypes = [_P, _P, _P, _P, _P, _P, _P, ct.c_size_t, pisa_shape, pisa_params, _P]
        L.pisa_decode_step.restype = ct.c_int
        L.pisa_decode_step.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, pisa_shape, pisa_params, _P]
        L.pisa_decode_workspace_bytes.restype = ct.c_size_t
        L.pisa_decode_workspace_bytes.argtypes = [pisa_shape, pisa_params]
        L.pisa_decode_step_ws.restype = ct.c_int
        L.pisa_decode_step_ws.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ct.c_size_t, pisa_shape,
                                          pisa_params, _P]
        L.pisa_status_string.restype = ct.c_char_p
        L.pisa_status_string.argtypes = [ct.c_int]
        L.pisa_get_last_device_error.restype = ct.c_int
        L.pisa_get_last_device_error.argtypes = [_P]
        L.pisa_version.restype = ct.c_char_p
        L.pisa_version.argtypes = []
        L.pisa_check_wait_timeout.restype = ct.c_int
        L.pisa_check_wait_timeout.argtypes = [ct.c_ulonglong, _P]
        L.pisa_phase_timing.restype = ct.c_int
        L.pisa_phase_timing.argtypes = [ct.c_int]
        L.pisa_phase_times.restype = ct.c_int
        L.pisa_phase_times.argtypes = [ct.POINTER(ct.c_double), ct.POINTER(ct.c_longlong), ct.c_int]
        L.pisa_phase_name.restype = ct.c_char_p
        L.pisa_phase_name.argtypes = [ct.c_int]
        _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != PISA_OK:
        raise PisaError(rc, what)


def _ptr(t):
    return None if t is None else ct.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return ct.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _bf16(t, name, dim=None):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or (dim is not None and t.dim() != dim):
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor" + (f" with {dim} dimensions" if dim else ""))


def _expect(t, name, shape, dtype, device):
    """The library reads and writes through raw pointers with the sizes the shape implies, so
    every tensor must have exactly that shape, dtype and device, and be contiguous (None is
    passed through as NULL where the C ABI allows it)."""
    if t is None:
        return
    if t.dtype != dtype or t.device != torch.device(device) or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device}; got "
                         f"{t.dtype} {tuple(t.shape)} on {t.device}{'' if t.is_contiguous() else ', not contiguous'}")


def _workspace(ws, need, device):
    """A caller's workspace if it is large enough, else a new one."""
    if ws is not None and (ws.dtype != torch.uint8 or ws.device != torch.device(device) or not ws.is_contiguous()):
        raise ValueError(f"workspace must be a contiguous uint8 tensor on {device}")
    if ws is None or ws.numel() < need:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return ws


# block scores: the LSE (PISA) or its first- / second-order truncations (PISA-1, PISA-2)
SCORING = {"lse": 0, "pisa1": 1, "pisa2": 2}


def make_params(K: int, causal: bool = True, scale: float = 0.0, C: int = 64, g: int = 2,
                scoring: int | str = 0) -> pisa_params:
    sc = SCORING[scoring] if isinstance(scoring, str) else int(scoring)
    return pisa_params(C, g, K, 1 if causal else 0, float(scale), sc)


def make_shape(B, N, H_q, H_kv, d, N_cap=0) -> pisa_shape:
    return pisa_shape(B, N, H_q, H_kv, d, N_cap)


# ---- geometry -------------------------------------------------------------------------
def pisa_pyramid_levels(N: int, C: int = 64, g: int = 2) -> int:
    return lib().pisa_pyramid_levels(N, C, g)


def pisa_pyramid_nodes(N: int, C: int = 64, g: int = 2) -> int:
    return int(lib().pisa_pyramid_nodes(N, C, g))


def pisa_select_workspace_bytes(shape: pisa_shape, params: pisa_params) -> int:
    return int(lib().pisa_select_workspace_bytes(shape, params))


def pisa_prefill_host_workspace_bytes(shape: pisa_shape, params: pisa_params) -> int:
    return int(lib().pisa_prefill_host_workspace_bytes(shape, params))


def pisa_prefill_host_chunks(N: int) -> list[int]:
    """Chunk bounds [0, ..., N] of the host-buffer prefill for N positions."""
    buf = (ct.c_longlong * 17)()
    n = lib().pisa_prefill_host_chunks(N, buf, 17)
    if n < 0:
        raise ValueError(f"pisa_prefill_host_chunks({N}) failed")
    return [int(buf[i]) for i in range(n + 1)]


def pisa_status_string(status: int) -> str:
    return lib().pisa_status_string(status).decode()


def pisa_version() -> str:
    return lib().pisa_version().decode()


def pisa_check_wait_timeout(limit_ns: int = 1_000_000, device=None) -> None:
    """Launch the kernel whose bounded waits run out after limit_ns (see include/pisa.h)."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    _check(lib().pisa_check_wait_timeout(int(limit_ns), ct.c_void_p(torch.cuda.current_stream(dev).cuda_stream)),
           "pisa_check_wait_timeout")


def pisa_phase_timing(enable: bool = True) -> None:
    """Start (clearing the totals) or stop per-phase event timing on the current device."""
    _check(lib().pisa_phase_timing(1 if enable else 0), "pisa_phase_timing")


def pisa_phase_name(phase: int):
    n = lib().pisa_phase_name(phase)
    return None if n is None else n.decode()


def pisa_phase_times() -> dict:
    """{phase name: (total ms, timed launches)} of the current device since timing started."""
    ms = (ct.c_double * 32)()
    cnt = (ct.c_longlong * 32)()
    n = lib().pisa_phase_times(ms, cnt, 32)
    if n < 0:
        raise PisaError(3, "pisa_phase_times")
    return {pisa_phase_name(i): (float(ms[i]), int(cnt[i])) for i in range(n)}


def pisa_get_last_device_error(device=None) -> int:
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    return lib().pisa_get_last_device_error(ct.c_void_p(torch.cuda.current_stream(dev).cuda_stream))


# ---- step 1 -----------------------------------------------------------------------------
def pisa_build_pyramid(K: torch.Tensor, N: int | None = None, P: torch.Tensor | None = None) -> torch.Tensor:
    """K [B, H_kv, N_cap, d] bf16 -> P [B, H_kv, nodes(N_cap), d]; levels built from the first N rows."""
    _bf16(K, "K", 4)
    B, H_kv, N_cap, d = K.shape
    N = N_cap if N is None else N
    nodes = pisa_pyramid_nodes(N_cap)
    if P is None:
        P = torch.empty(B, H_kv, nodes, d, dtype=torch.bfloat16, device=K.device)
    _expect(P, "P", (B, H_kv, nodes, d), torch.bfloat16, K.device)
    shape = make_shape(B, N, H_kv, H_kv, d, N_cap)
    _check(lib().pisa_build_pyramid(_ptr(K), _ptr(P), shape, make_params(1), _stream(K)), "pisa_build_pyramid")
    return P


# ---- step 2 -----------------------------------------------------------------------------
def _select_inputs(Q, K, P):
    """Q [B, N, H_q, d], K [B, H_kv, N, d] and P [B, H_kv, nodes(N), d], all bf16 on one device."""
    _bf16(Q, "Q", 4)
    _bf16(K, "K", 4)
    B, N, H_q, d = Q.shape
    H_kv = K.shape[1]
    _expect(K, "K", (B, H_kv, N, d), torch.bfloat16, Q.device)
    _expect(P, "P", (B, H_kv, pisa_pyramid_nodes(N), d), torch.bfloat16, Q.device)
    return B, N, H_q, d, H_kv


def pisa_select_prefill(Q, K, P, K_sel: int, causal: bool = True, scale: float = 0.0, want_scores: bool = False,
                        want_s2: bool = False, ws: torch.Tensor | None = None, idx: torch.Tensor | None = None,
                        scoring: int | str = 0, s2: torch.Tensor | None = None):
    """Returns idx [B, H_kv, N, K_sel] int32 (and leaf_score, s2 if asked).  An s2 tensor passed in
    receives the level-2 survivors without being returned."""
    B, N, H_q, d, H_kv = _select_inputs(Q, K, P)
    shape = make_shape(B, N, H_q, H_kv, d, N)
    params = make_params(K_sel, causal, scale, scoring=scoring)
    need = pisa_select_workspace_bytes(shape, params)
    if need == 0 and B * N > 0:
        raise PisaError(2, "pisa_select_prefill: unsupported shape or parameters")
    ws = _workspace(ws, need, Q.device)
    if idx is None:
        idx = torch.empty(B, H_kv, N, K_sel, dtype=torch.int32, device=Q.device)
    _expect(idx, "idx", (B, H_kv, N, K_sel), torch.int32, Q.device)
    score = torch.empty(B, H_kv, N, 2 * K_sel, dtype=torch.float32, device=Q.device) if want_scores else None
    if want_s2:
        s2 = torch.empty(B, H_kv, N, K_sel, dtype=torch.int32, device=Q.device)
    _expect(s2, "s2", (B, H_kv, N, K_sel), torch.int32, Q.device)
    _check(lib().pisa_select_prefill(_ptr(Q), _ptr(K), _ptr(P), _ptr(idx), _ptr(score), _ptr(s2), _ptr(ws),
                                     ws.numel(), shape, params, _stream(Q)), "pisa_select_prefill")
    out = [idx]
    if want_scores:
        out.append(score)
    if want_s2:
        out.append(s2)
    return out[0] if len(out) == 1 else tuple(out)


def pisa_select_prefill_noalloc(Q, K, P, K_sel: int, causal: bool = True, scale: float = 0.0, idx=None,
                                leaf_score=None, s2=None, scoring: int | str = 0):
    """pisa_select_prefill without a caller-supplied workspace: the library's fixed 32 MiB
    device scratch is used instead (for callers that cannot allocate device memory).
    Output tensors may be passed in so that the call itself allocates nothing."""
    B, N, H_q, d, H_kv = _select_inputs(Q, K, P)
    if idx is None:
        idx = torch.empty(B, H_kv, N, K_sel, dtype=torch.int32, device=Q.device)
    _expect(idx, "idx", (B, H_kv, N, K_sel), torch.int32, Q.device)
    _expect(leaf_score, "leaf_score", (B, H_kv, N, 2 * K_sel), torch.float32, Q.device)
    _expect(s2, "s2", (B, H_kv, N, K_sel), torch.int32, Q.device)
    _check(lib().pisa_select_prefill_noalloc(_ptr(Q), _ptr(K), _ptr(P), _ptr(idx), _ptr(leaf_score), _ptr(s2),
                                             make_shape(B, N, H_q, H_kv, d, N),
                                             make_params(K_sel, causal, scale, scoring=scoring),
                                             _stream(Q)), "pisa_select_prefill_noalloc")
    return idx


# ---- baseline: BSA flat selection --------------------------------------------------------
def pisa_select_bsa_workspace_bytes(shape: pisa_shape, params: pisa_params) -> int:
    return int(lib().pisa_select_bsa_workspace_bytes(shape, params))


def pisa_select_bsa(Q, P, K_sel: int, causal: bool = True, scale: float = 0.0, ws=None, idx=None):
    """BSA flat selection from the leaf summaries of P: returns idx [B, H_kv, N, K_sel] int32."""
    _bf16(Q, "Q", 4)
    _bf16(P, "P", 4)
    B, N, H_q, d = Q.shape
    H_kv = P.shape[1]
    _expect(P, "P", (B, H_kv, pisa_pyramid_nodes(N), d), torch.bfloat16, Q.device)
    shape = make_shape(B, N, H_q, H_kv, d, N)
    params = make_params(K_sel, causal, scale)
    need = pisa_select_bsa_workspace_bytes(shape, params)
    if need == 0 and B * N > 0:
        raise PisaError(2, "pisa_select_bsa: unsupported shape or parameters")
    ws = _workspace(ws, need, Q.device)
    if idx is None:
        idx = torch.empty(B, H_kv, N, K_sel, dtype=torch.int32, device=Q.device)
    _expect(idx, "idx", (B, H_kv, N, K_sel), torch.int32, Q.device)
    _check(lib().pisa_select_bsa(_ptr(Q), _ptr(P), _ptr(idx), _ptr(ws), ws.numel(), shape, params, _stream(Q)),
           "pisa_select_bsa")
    return idx


# ---- step 4 -----------------------------------------------------------------------------
def _attn_inputs(Q, K, V, idx):
    """Q [B, N, H_q, d], K and V [B, H_kv, N_cap, d] bf16, idx [B, H_kv, N, K] int32, one device."""
    _bf16(Q, "Q", 4)
    _bf16(K, "K", 4)
    B, N, H_q, d = Q.shape
    H_kv, N_cap = K.shape[1], K.shape[2]
    _expect(K, "K", (B, H_kv, N_cap, d), torch.bfloat16, Q.device)
    _expect(V, "V", (B, H_kv, N_cap, d), torch.bfloat16, Q.device)
    if idx.dim() != 4:
        raise ValueError("idx must be [B, H_kv, N, K]")
    _expect(idx, "idx", (B, H_kv, N, idx.shape[-1]), torch.int32, Q.device)
    return B, N, H_q, d, H_kv, N_cap


def pisa_sparse_attn_prefill(Q, K, V, idx, causal: bool = True, scale: float = 0.0, O=None, LSE=None,
                             want_lse: bool = True):
    """Returns O [B, N, H_q, d] bf16 and LSE [B, H_q, N] fp32 (None if not wanted)."""
    B, N, H_q, d, H_kv, N_cap = _attn_inputs(Q, K, V, idx)
    if O is None:
        O = torch.empty_like(Q)
    if want_lse and LSE is None:
        LSE = torch.empty(B, H_q, N, dtype=torch.float32, device=Q.device)
    _expect(O, "O", (B, N, H_q, d), torch.bfloat16, Q.device)
    if want_lse:
        _expect(LSE, "LSE", (B, H_q, N), torch.float32, Q.device)
    shape = make_shape(B, N, H_q, H_kv, d, N_cap)
    params = make_params(idx.shape[-1], causal, scale)
    _check(lib().pisa_sparse_attn_prefill(_ptr(Q), _ptr(K), _ptr(V), _ptr(idx), _ptr(O), _ptr(LSE if want_lse else None),
                                          shape, params, _stream(Q)), "pisa_sparse_attn_prefill")
    return O, (LSE if want_lse else None)


def pisa_attn_backward_workspace_bytes(shape: pisa_shape, params: pisa_params) -> int:
    return lib().pisa_attn_backward_workspace_bytes(shape, params)


def pisa_attn_backward_min_workspace_bytes(shape: pisa_shape, params: pisa_params) -> int:
    return lib().pisa_attn_backward_min_workspace_bytes(shape, params)


def pisa_sparse_attn_backward(Q, K, V, idx, O, LSE, dO, causal: bool = True, scale: float = 0.0, ws=None,
                              dQ=None, dK=None, dV=None):
    """Gradients of pisa_sparse_attn_prefill: returns dQ [B, N, H_q, d], dK, dV [B, H_kv, N_cap, d] (fp32).
    A caller's ws of at least pisa_attn_backward_min_workspace_bytes() is used as it is (below
    pisa_attn_backward_workspace_bytes() the dQ kernel forms S and dP again instead of reading dS);
    without one, the full size is allocated."""
    B, N, H_q, d, H_kv, N_cap = _attn_inputs(Q, K, V, idx)
    for t, n in ((O, "O"), (dO, "dO")):
        _expect(t, n, (B, N, H_q, d), torch.bfloat16, Q.device)
    if LSE is None:
        raise ValueError("LSE must be given")
    _expect(LSE, "LSE", (B, H_q, N), torch.float32, Q.device)
    shape = make_shape(B, N, H_q, H_kv, d, N_cap)
    params = make_params(idx.shape[-1], causal, scale)
    need = pisa_attn_backward_workspace_bytes(shape, params)
    if need == 0 and B * N > 0:
        raise PisaError(2, "pisa_sparse_attn_backward: unsupported shape or parameters")
    least = pisa_attn_backward_min_workspace_bytes(shape, params)
    ws = _workspace(ws, need if ws is None else least, Q.device)
    dQ = torch.empty(B, N, H_q, d, dtype=torch.float32, device=Q.device) if dQ is None else dQ
    dK = torch.empty(B, H_kv, N_cap, d, dtype=torch.float32, device=Q.device) if dK is None else dK
    dV = torch.empty(B, H_kv, N_cap, d, dtype=torch.float32, device=Q.device) if dV is None else dV
    _expect(dQ, "dQ", (B, N, H_q, d), torch.float32, Q.device)
    _expect(dK, "dK", (B, H_kv, N_cap, d), torch.float32, Q.device)
    _expect(dV, "dV", (B, H_kv, N_cap, d), torch.float32, Q.device)
    _check(lib().pisa_sparse_attn_backward(_ptr(Q), _ptr(K), _ptr(V), _ptr(idx), _ptr(O), _ptr(LSE), _ptr(dO),
                                           _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), ws.numel(), shape, params,
                                           _stream(Q)), "pisa_sparse_attn_backward")
    return dQ, dK, dV


def pisa_prefill_host(Q_host, K_host, V_host, K_sel: int, causal: bool = True, scale: float = 0.0, dev_ws=None,
                      O_host=None, LSE_host=None, idx_host=None, device=None, scoring: int | str = 0):
    """Whole prefill from host (ideally pinned) tensors; copies happen inside the call."""
    if Q_host.dim() != 4 or K_host.dim() != 4:
        raise ValueError("Q_host must be [B, N, H_q, d] and K_host [B, H_kv, N, d]")
    B, N, H_q, d = Q_host.shape
    H_kv = K_host.shape[1]
    cpu = torch.device("cpu")
    _expect(Q_host, "Q_host", (B, N, H_q, d), torch.bfloat16, cpu)
    _expect(K_host, "K_host", (B, H_kv, N, d), torch.bfloat16, cpu)
    _expect(V_host, "V_host", (B, H_kv, N, d), torch.bfloat16, cpu)
    if O_host is None:
        O_host = torch.empty_like(Q_host)
    _expect(O_host, "O_host", (B, N, H_q, d), torch.bfloat16, cpu)
    _expect(LSE_host, "LSE_host", (B, H_q, N), torch.float32, cpu)
    _expect(idx_host, "idx_host", (B, H_kv, N, K_sel), torch.int32, cpu)
    shape = make_shape(B, N, H_q, H_kv, d, N)
    params = make_params(K_sel, causal, scale, scoring=scoring)
    # the host buffers are all checked before anything touches the device
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    need = pisa_prefill_host_workspace_bytes(shape, params)
    dev_ws = _workspace(dev_ws, need, dev)
    stream = ct.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    _check(lib().pisa_prefill_host(_ptr(Q_host), _ptr(K_host), _ptr(V_host), _ptr(O_host), _ptr(LSE_host),
                                   _ptr(idx_host), _ptr(dev_ws), dev_ws.numel(), shape, params, stream),
           "pisa_prefill_host")
    return O_host


# ---- step 3 -----------------------------------------------------------------------------
def pisa_decode_workspace_bytes(shape, params) -> int:
    """Bytes of the decode step's logits scratch (0 for arguments the step refuses)."""
    return int(lib().pisa_decode_workspace_bytes(shape, params))


def pisa_decode_step_ws(q, k, v, Kc, Vc, Pc, seq_len, K_sel: int, ws=None, **kw):
    """pisa_decode_step with the logits scratch ws (allocated when None or too small)."""
    return pisa_decode_step(q, k, v, Kc, Vc, Pc, seq_len, K_sel, ws=ws, keep_logits=True, **kw)


def pisa_decode_step(q, k, v, Kc, Vc, Pc, seq_len, K_sel: int, scale: float = 0.0, o=None, lse=None, idx_out=None,
                     scoring: int | str = 0, ws=None, keep_logits: bool = True):
    """One decode step for every sequence; caches and seq_len are updated in place.  With
    keep_logits (pisa_decode_step_ws) the leaf scoring's logits are kept in ws (a uint8 device
    tensor, allocated when None or too small) and the attention reads them instead of the
    selected blocks' K rows; without it, pisa_decode_step.  The results are the same."""
    _bf16(q, "q", 3)
    _bf16(k, "k", 3)
    _bf16(Kc, "Kc", 4)
    B, H_q, d = q.shape
    H_kv = k.shape[1]
    N_cap = Kc.shape[2]
    dev = q.device
    for t, n in ((k, "k"), (v, "v")):
        _expect(t, n, (B, H_kv, d), torch.bfloat16, dev)
    for t, n in ((Kc, "Kc"), (Vc, "Vc")):
        _expect(t, n, (B, H_kv, N_cap, d), torch.bfloat16, dev)
    _expect(Pc, "Pc", (B, H_kv, pisa_pyramid_nodes(N_cap), d), torch.bfloat16, dev)
    _expect(seq_len, "seq_len", (B,), torch.int32, dev)
    if o is None:
        o = torch.empty_like(q)
    _expect(o, "o", (B, H_q, d), torch.bfloat16, dev)
    _expect(lse, "lse", (B, H_q), torch.float32, dev)
    _expect(idx_out, "idx_out", (B, H_kv, K_sel), torch.int32, dev)
    shape = make_shape(B, 0, H_q, H_kv, d, N_cap)
    params = make_params(K_sel, True, scale, scoring=scoring)
    if not keep_logits:
        _check(lib().pisa_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(Kc), _ptr(Vc), _ptr(Pc), _ptr(seq_len), _ptr(o),
                                      _ptr(lse), _ptr(idx_out), shape, params, _stream(q)),
               "pisa_decode_step")
        return o
    need = lib().pisa_decode_workspace_bytes(shape, params)
    ws = _workspace(ws, need, dev) if need > 0 else None  # 0: arguments the call refuses with its own status
    _check(lib().pisa_decode_step_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(Kc), _ptr(Vc), _ptr(Pc), _ptr(seq_len), _ptr(o),
                                     _ptr(lse), _ptr(idx_out), _ptr(ws), 0 if ws is None else ws.numel(), shape, params,
                                     _stream(q)),
           "pisa_decode_step_ws")
    return o
