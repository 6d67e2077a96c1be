"""Python access to the CPU oracle (``pisa_oracle.cpp``) through ctypes.

TEST INFRASTRUCTURE ONLY: imported by the test suite, by ``__graft_entry__.smoke()`` and
by the benchmark's CPU-baseline leg.  The GPU library never imports, links or runs it.

Arrays cross the boundary as numpy buffers: bf16 tensors as uint16 bit patterns,
indices as int32/int64, results as float64.
"""
from __future__ import annotations

import ctypes as ct
import math
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pisa_oracle.cpp")


LIB = os.path.join(HERE, "libpisa_oracle.so")


def compile_source(src: str, out: str) -> str:
    """Compile an oracle source file to a shared library (plain g++ -O2, no SIMD intrinsics)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", src, "-o", tmp], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    return compile_source(SRC, LIB)


_P = ct.c_void_p
_LL = ct.c_longlong
_I = ct.c_int
_D = ct.c_double


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ct.c_void_p)


class Oracle:
    def __init__(self, lib: str | None = None, nthreads: int = 0):
        self.lib = ct.CDLL(lib or build())
        self.nthreads = nthreads
        L = self.lib
        L.oracle_num_levels.restype = _I
        L.oracle_num_levels.argtypes = [_LL, _I, _I]
        L.oracle_level_sizes.restype = _I
        L.oracle_level_sizes.argtypes = [_LL, _I, _I, _P, _I]
        L.oracle_pyramid_nodes.restype = _LL
        L.oracle_pyramid_nodes.argtypes = [_LL, _I, _I]
        L.oracle_build_pyramid.restype = _I
        L.oracle_build_pyramid.argtypes = [_P, _P, _I, _I, _LL, _LL, _I, _I, _I, _I]
        L.oracle_select.restype = _I
        L.oracle_select.argtypes = [_P, _P, _P, _I, _LL, _I, _I, _I, _I, _I, _I, _I, _D, _I, _P, _P, _P, _P, _P, _P,
                                    _I, _I]
        L.oracle_selection_admissible.restype = _I
        L.oracle_selection_admissible.argtypes = [_P, _P, _P, _I, _LL, _I, _I, _I, _I, _I, _I, _I, _D, _I, _P, _P,
                                                  _D, _P, _I, _I]
        L.oracle_sparse_attention.restype = _I
        L.oracle_sparse_attention.argtypes = [_P, _P, _P, _P, _I, _LL, _I, _I, _I, _I, _I, _I, _D, _I, _P, _P, _P,
                                              _P, _I]
        L.oracle_sparse_attention_backward.restype = _I
        L.oracle_sparse_attention_backward.argtypes = [_P, _P, _P, _P, _P, _I, _LL, _I, _I, _I, _I, _I, _I, _D, _P,
                                                       _P, _P, _I]
        L.oracle_sparse_attention_backward_sampled.restype = _I
        L.oracle_sparse_attention_backward_sampled.argtypes = [_P, _P, _P, _P, _P, _I, _LL, _I, _I, _I, _I, _I, _I,
                                                               _D, _P, _I, _P, _I, _P, _P, _P, _I]
        L.oracle_decode_step.restype = _I
        L.oracle_decode_step.argtypes = [_P, _P, _P, _P, _P, _P, _P, _LL, _I, _I, _I, _I, _I, _I, _I, _D, _P, _P,
                                         _P, _I, _I]
        L.oracle_select_bsa.restype = _I
        L.oracle_select_bsa.argtypes = [_P, _P, _I, _LL, _I, _I, _I, _I, _I, _I, _I, _D, _I, _P, _P, _P, _P, _I]
        L.oracle_f64_to_bf16.restype = ct.c_uint16
        L.oracle_f64_to_bf16.argtypes = [_D]

    # ---- geometry -------------------------------------------------------------------
    def num_levels(self, n, C=64, g=2):
        return self.lib.oracle_num_levels(n, C, g)

    def level_sizes(self, n, C=64, g=2):
        buf = np.zeros(64, dtype=np.int64)
        L = self.lib.oracle_level_sizes(n, C, g, _ptr(buf), 64)
        return [int(x) for x in buf[:L]]

    def pyramid_nodes(self, n, C=64, g=2):
        return int(self.lib.oracle_pyramid_nodes(n, C, g))

    def f64_to_bf16(self, x: float) -> int:
        return int(self.lib.oracle_f64_to_bf16(float(x)))

    # ---- step 1 ---------------------------------------------------------------------
    def build_pyramid(self, K: np.ndarray, N: int | None = None, C=64, g=2) -> np.ndarray:
        """K: uint16 [B, H_kv, N_cap, d] -> P: uint16 [B, H_kv, nodes(N_cap), d]."""
        K = np.ascontiguousarray(K, dtype=np.uint16)
        B, H, N_cap, d = K.shape
        N = N_cap if N is None else N
        P = np.zeros((B, H, self.pyramid_nodes(N_cap, C, g), d), dtype=np.uint16)
        rc = self.lib.oracle_build_pyramid(_ptr(K), _ptr(P), B, H, N, N_cap, d, C, g, self.nthreads)
        assert rc == 0, rc
        return P

    # ---- step 2 ---------------------------------------------------------------------
    def select(self, Q, K, P, Ksel, rows, C=64, g=2, causal=True, scale=None, scoring=0):
        """Q uint16 [B,N,H_q,d]; K [B,H_kv,N,d]; P [B,H_kv,nodes,d]; rows int64 [R,3] (b,h_kv,t).
        scoring: 0 LSE, 1 PISA-1 (log m + mean), 2 PISA-2 (log m + mean + var/2)."""
        B, N, H_q, d = Q.shape
        H_kv = K.shape[1]
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        R = rows.shape[0]
        idx = np.zeros((R, Ksel), np.int32)
        s2 = np.zeros((R, Ksel), np.int32)
        cand = np.zeros((R, g * Ksel), np.int32)
        cs = np.zeros((R, g * Ksel), np.float64)
        gap = np.zeros(R, np.float64)
        rc = self.lib.oracle_select(_ptr(Q), _ptr(K), _ptr(P), B, N, H_q, H_kv, d, C, g, Ksel, int(causal), scale, R,
                                    _ptr(rows), _ptr(idx), _ptr(s2), _ptr(cand), _ptr(cs), _ptr(gap), self.nthreads,
                                    int(scoring))
        assert rc == 0, rc
        return dict(idx=idx, s2=s2, cand=cand, cand_score=cs, min_gap=gap)

    def select_bsa(self, Q, P, Ksel, rows, C=64, g=2, causal=True, scale=None, want_scores=False):
        """BSA flat selection (one level of mean summaries, head-summed dot products, top-K):
        Q uint16 [B,N,H_q,d]; P [B,H_kv,nodes,d] (level 1 = the leaf means); rows int64 [R,3].
        Returns idx [R,K], min_gap [R] and, if asked, score [R,M_1] (-inf where not ranked)."""
        B, N, H_q, d = Q.shape
        H_kv = P.shape[1]
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        R = rows.shape[0]
        M1 = (N + C - 1) // C
        idx = np.zeros((R, Ksel), np.int32)
        gap = np.zeros(R, np.float64)
        score = np.zeros((R, M1), np.float64) if want_scores else None
        rc = self.lib.oracle_select_bsa(_ptr(np.ascontiguousarray(Q, dtype=np.uint16)),
                                        _ptr(np.ascontiguousarray(P, dtype=np.uint16)), B, N, H_q, H_kv, d, C, g, Ksel,
                                        int(causal), scale, R, _ptr(rows), _ptr(idx), _ptr(score), _ptr(gap),
                                        self.nthreads)
        assert rc == 0, rc
        out = dict(idx=idx, min_gap=gap)
        if want_scores:
            out["score"] = score
        return out

    def admissible(self, Q, K, P, Ksel, rows, target_idx, tol=1e-3, C=64, g=2, causal=True, scale=None, scoring=0):
        B, N, H_q, d = Q.shape
        H_kv = K.shape[1]
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        tgt = np.ascontiguousarray(target_idx, dtype=np.int32).reshape(rows.shape[0], Ksel)
        ok = np.zeros(rows.shape[0], np.int32)
        self.lib.oracle_selection_admissible(_ptr(Q), _ptr(K), _ptr(P), B, N, H_q, H_kv, d, C, g, Ksel, int(causal),
                                             scale, rows.shape[0], _ptr(rows), _ptr(tgt), tol, _ptr(ok),
                                             self.nthreads, int(scoring))
        return ok

    # ---- step 4 ---------------------------------------------------------------------
    def sparse_attention(self, Q, K, V, idx, rows, C=64, causal=True, scale=None):
        """idx int32 [B,H_kv,N,Ksel]; rows int64 [R,2] (b,t) -> O [R,H_q,d], LSE [R,H_q], wsum [R,H_q]."""
        B, N, H_q, d = Q.shape
        H_kv = K.shape[1]
        Ksel = idx.shape[-1]
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 2)
        R = rows.shape[0]
        O = np.zeros((R, H_q, d), np.float64)
        LSE = np.zeros((R, H_q), np.float64)
        ws = np.zeros((R, H_q), np.float64)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        rc = self.lib.oracle_sparse_attention(_ptr(Q), _ptr(K), _ptr(V), _ptr(idx), B, N, H_q, H_kv, d, C, Ksel,
                                              int(causal), scale, R, _ptr(rows), _ptr(O), _ptr(LSE), _ptr(ws),
                                              self.nthreads)
        assert rc == 0, rc
        return O, LSE, ws

    def sparse_attention_backward(self, Q, K, V, idx, dO, C=64, causal=True, scale=None):
        """Gradients of the step-4 output: Q, dO uint16 [B,N,H_q,d]; K, V [B,H_kv,N,d];
        idx int32 [B,H_kv,N,Ksel] -> dQ [B,N,H_q,d], dK, dV [B,H_kv,N,d] (fp64)."""
        B, N, H_q, d = Q.shape
        H_kv = K.shape[1]
        Ksel = idx.shape[-1]
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        dQ = np.zeros((B, N, H_q, d), np.float64)
        dK = np.zeros((B, H_kv, N, d), np.float64)
        dV = np.zeros((B, H_kv, N, d), np.float64)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        dO = np.ascontiguousarray(dO, dtype=np.uint16)
        rc = self.lib.oracle_sparse_attention_backward(_ptr(Q), _ptr(K), _ptr(V), _ptr(idx), _ptr(dO), B, N, H_q,
                                                       H_kv, d, C, Ksel, int(causal), scale, _ptr(dQ), _ptr(dK),
                                                       _ptr(dV), self.nthreads)
        assert rc == 0, rc
        return dQ, dK, dV

    def sparse_attention_backward_sampled(self, Q, K, V, idx, dO, rows, blocks, C=64, causal=True, scale=None):
        """The backward at samples: rows = flat (b * N + t) query positions -> dQ [nrows, H_q, d];
        blocks = flat ((b * H_kv + h_kv) * M1 + j) key blocks -> dK, dV [nblocks, C, d] (fp64), equal
        to the corresponding values of sparse_attention_backward."""
        B, N, H_q, d = Q.shape
        H_kv = K.shape[1]
        Ksel = idx.shape[-1]
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        blocks = np.ascontiguousarray(blocks, dtype=np.int64)
        dQ = np.zeros((len(rows), H_q, d), np.float64)
        dK = np.zeros((len(blocks), C, d), np.float64)
        dV = np.zeros((len(blocks), C, d), np.float64)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        dO = np.ascontiguousarray(dO, dtype=np.uint16)
        rc = self.lib.oracle_sparse_attention_backward_sampled(
            _ptr(Q), _ptr(K), _ptr(V), _ptr(idx), _ptr(dO), B, N, H_q, H_kv, d, C, Ksel, int(causal), scale, _ptr(rows),
            len(rows), _ptr(blocks), len(blocks), _ptr(dQ), _ptr(dK), _ptr(dV), self.nthreads)
        assert rc == 0, rc
        return dQ, dK, dV

    # ---- step 3 ---------------------------------------------------------------------
    def decode_step(self, q, k, v, Kc, Vc, Pc, seq_len, Ksel, C=64, g=2, scale=None, scoring=0):
        """In place on Kc, Vc, Pc (uint16) and seq_len (int32).  Returns o, lse, idx."""
        B, H_q, d = q.shape
        H_kv = k.shape[1]
        N_cap = Kc.shape[2]
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        for a in (Kc, Vc, Pc, seq_len):
            assert a.flags["C_CONTIGUOUS"]
        o = np.zeros((B, H_q, d), np.float64)
        lse = np.zeros((B, H_q), np.float64)
        idx = np.zeros((B, H_kv, Ksel), np.int32)
        q = np.ascontiguousarray(q, dtype=np.uint16)
        k = np.ascontiguousarray(k, dtype=np.uint16)
        v = np.ascontiguousarray(v, dtype=np.uint16)
        rc = self.lib.oracle_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(Kc), _ptr(Vc), _ptr(Pc), _ptr(seq_len), N_cap,
                                         B, H_q, H_kv, d, C, g, Ksel, scale, _ptr(o), _ptr(lse), _ptr(idx),
                                         self.nthreads, int(scoring))
        assert rc == 0, rc
        return o, lse, idx
