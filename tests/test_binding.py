"""The Python binding's argument checks, on the host only.  The library reads and writes
through raw pointers with the sizes the shape implies, so every tensor handed to it must have
exactly the shape, dtype and device the C ABI states; a mismatch is refused with ValueError
before the library is called.  These tests run on CPU tensors against a stand-in library that
records the compute calls (the geometry and workspace queries go to the real library)."""
import types

import pytest
import torch

import hierarchical_top_block_gb300 as pisa
import workloads as W
from hierarchical_top_block_gb300.build import build

COMPUTE = ("pisa_build_pyramid", "pisa_select_prefill", "pisa_select_prefill_noalloc", "pisa_sparse_attn_prefill",
           "pisa_sparse_attn_backward", "pisa_prefill_host", "pisa_decode_step", "pisa_decode_step_ws", "pisa_select_bsa")


@pytest.fixture
def calls(monkeypatch):
    build()
    real = pisa.lib()
    made = []

    class StandIn:
        def __getattr__(self, name):
            if name in COMPUTE:
                return lambda *args: made.append(name) or 0
            return getattr(real, name)

    def bf16_any_device(t, name, dim=None):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or (dim is not None and t.dim() != dim):
            raise ValueError(name)

    monkeypatch.setattr(pisa, "_lib", StandIn())
    monkeypatch.setattr(pisa, "_bf16", bf16_any_device)
    monkeypatch.setattr(pisa, "_stream", lambda t: None)
    monkeypatch.setattr(pisa, "_workspace", lambda ws, need, dev: torch.empty(max(need, 256), dtype=torch.uint8))
    monkeypatch.setattr(torch.cuda, "current_stream", lambda dev=None: types.SimpleNamespace(cuda_stream=0))
    return made


def _ok(calls, fn):
    n = len(calls)
    fn()
    assert len(calls) == n + 1


def _refused(calls, fn):
    n = len(calls)
    with pytest.raises(ValueError):
        fn()
    assert len(calls) == n


def test_prefill_buffers(calls):
    w = W.WORKLOADS["prefill_32k"].with_(N=640)  # G_Q = 16, two KV heads
    Q, K, V = W.prefill_inputs(w, "cpu")
    P = torch.empty(w.B, w.H_kv, pisa.pisa_pyramid_nodes(w.N), w.d, dtype=torch.bfloat16)
    idx = torch.empty(w.B, w.H_kv, w.N, w.K, dtype=torch.int32)
    O, LSE = torch.empty_like(Q), torch.empty(w.B, w.H_q, w.N, dtype=torch.float32)
    _ok(calls, lambda: pisa.pisa_build_pyramid(K, P=P))
    _ok(calls, lambda: pisa.pisa_select_prefill(Q, K, P, w.K, idx=idx, want_scores=True, want_s2=True))
    _ok(calls, lambda: pisa.pisa_select_prefill_noalloc(Q, K, P, 8))
    _ok(calls, lambda: pisa.pisa_sparse_attn_prefill(Q, K, V, idx, O=O, LSE=LSE))
    _ok(calls, lambda: pisa.pisa_select_bsa(Q, P, w.K, idx=idx))
    _refused(calls, lambda: pisa.pisa_select_bsa(Q, P[:, :, :-1], w.K))
    _refused(calls, lambda: pisa.pisa_select_bsa(Q, P, w.K, idx=idx[..., :8].contiguous()))
    _refused(calls, lambda: pisa.pisa_build_pyramid(K, P=P[:, :, :-1]))
    _refused(calls, lambda: pisa.pisa_select_prefill(Q, K[:, :, :-64].contiguous(), P, w.K))
    _refused(calls, lambda: pisa.pisa_select_prefill(Q, K, P, w.K, idx=idx[..., :8].contiguous()))
    _refused(calls, lambda: pisa.pisa_select_prefill(Q, K, P, w.K, idx=idx.to(torch.int64)))
    _refused(calls, lambda: pisa.pisa_select_prefill_noalloc(Q, K, P, w.K, s2=idx[:, :1].contiguous()))
    _refused(calls, lambda: pisa.pisa_sparse_attn_prefill(Q, K, V[:, :, :-1].contiguous(), idx))
    _refused(calls, lambda: pisa.pisa_sparse_attn_prefill(Q, K, V, idx, O=O[:, :-1]))
    _refused(calls, lambda: pisa.pisa_sparse_attn_prefill(Q, K, V, idx, LSE=LSE.transpose(1, 2)))
    dO = torch.zeros_like(Q)
    dQ = torch.empty(Q.shape, dtype=torch.float32)
    dK = torch.empty(K.shape, dtype=torch.float32)
    _ok(calls, lambda: pisa.pisa_sparse_attn_backward(Q, K, V, idx, O, LSE, dO, dQ=dQ, dK=dK, dV=dK.clone()))
    _refused(calls, lambda: pisa.pisa_sparse_attn_backward(Q, K, V, idx, O, LSE, dO, dQ=dQ.to(torch.bfloat16)))
    _refused(calls, lambda: pisa.pisa_sparse_attn_backward(Q, K, V, idx, O, LSE[:, :, 1:], dO))


def test_decode_buffers(calls):
    w = W.WORKLOADS["decode_128k"].with_(B=3, H_q=8, H_kv=2, N=300)
    Kc = torch.zeros(w.B, w.H_kv, 512, w.d, dtype=torch.bfloat16)
    Pc = pisa.pisa_build_pyramid(Kc, N=300)
    seq = torch.full((w.B,), 300, dtype=torch.int32)
    q, k, v = W.decode_step_inputs(w, 0, "cpu")
    lse = torch.empty(w.B, w.H_q, dtype=torch.float32)
    idx = torch.empty(w.B, w.H_kv, w.K, dtype=torch.int32)
    _ok(calls, lambda: pisa.pisa_decode_step(q, k, v, Kc, Kc.clone(), Pc, seq, w.K, lse=lse, idx_out=idx))
    _refused(calls, lambda: pisa.pisa_decode_step(q, k, v, Kc, Kc.clone(), Pc, seq[:2], w.K))
    _refused(calls, lambda: pisa.pisa_decode_step(q, k, v, Kc, Kc[:, :, :256].contiguous(), Pc, seq, w.K))
    _refused(calls, lambda: pisa.pisa_decode_step(q, k, v, Kc, Kc.clone(), Pc, seq, w.K, idx_out=idx[..., :4]))
    _refused(calls, lambda: pisa.pisa_decode_step(q, k[:, :1].contiguous(), v, Kc, Kc.clone(), Pc, seq, w.K))
    # the same checks with the logits scratch off (pisa_decode_step) and through pisa_decode_step_ws
    _ok(calls, lambda: pisa.pisa_decode_step(q, k, v, Kc, Kc.clone(), Pc, seq, w.K, keep_logits=False))
    _ok(calls, lambda: pisa.pisa_decode_step_ws(q, k, v, Kc, Kc.clone(), Pc, seq, w.K, lse=lse))
    _refused(calls, lambda: pisa.pisa_decode_step_ws(q, k, v, Kc, Kc.clone(), Pc, seq[:2], w.K))


def test_host_prefill_buffers_checked_before_the_device_is_touched():
    """Runs with the real library: on a machine without a GPU, reaching the device would raise
    something other than ValueError."""
    w = W.WORKLOADS["tiny"]
    Q, K, V = W.prefill_inputs(w, "cpu")
    L = torch.empty(w.B, w.H_q, w.N, dtype=torch.float32)
    I = torch.empty(w.B, w.H_kv, w.N, w.K, dtype=torch.int32)
    for kwargs in ({"LSE_host": L[:, :, :-1]}, {"idx_host": I.to(torch.int64)}, {"O_host": torch.empty_like(Q)[:, 1:]},
                   {"idx_host": I[..., :2].contiguous()}):
        with pytest.raises(ValueError):
            pisa.pisa_prefill_host(Q, K, V, w.K, **kwargs)
    with pytest.raises(ValueError):
        pisa.pisa_prefill_host(Q, K[:, :, :-1].contiguous(), V, w.K)
    with pytest.raises(ValueError):
        pisa.pisa_prefill_host(Q.float(), K, V, w.K)


def _empty_calls(dev, host_prefill):
    """Every entry point on empty problems (N = 0, then B = 0), through the binding and the
    library; each returns outputs of the right (empty) shape and launches nothing."""
    for B, N in ((1, 0), (0, 256)):
        Q = torch.empty(B, N, 16, 128, dtype=torch.bfloat16, device=dev)
        K = torch.empty(B, 1, N, 128, dtype=torch.bfloat16, device=dev)
        V = torch.empty_like(K)
        P = pisa.pisa_build_pyramid(K)
        assert P.shape == (B, 1, pisa.pisa_pyramid_nodes(N), 128)
        idx, score = pisa.pisa_select_prefill(Q, K, P, 16, want_scores=True)
        assert idx.shape == (B, 1, N, 16) and score.shape == (B, 1, N, 32)
        O, LSE = pisa.pisa_sparse_attn_prefill(Q, K, V, idx)
        assert O.shape == Q.shape and LSE.shape == (B, 16, N)
        assert pisa.pisa_select_bsa(Q, P, 8).shape == (B, 1, N, 8)
        assert pisa.pisa_select_prefill(Q, K, P, 32).shape == (B, 1, N, 32)
        dQ, dK, dV = pisa.pisa_sparse_attn_backward(Q, K, V, idx, O, LSE, torch.empty_like(Q))
        assert dQ.shape == Q.shape and dK.shape == K.shape and dV.shape == V.shape
        if host_prefill:
            Oh = pisa.pisa_prefill_host(Q.cpu(), K.cpu(), V.cpu(), 16, device=0)
            assert Oh.shape == Q.shape and Oh.device.type == "cpu"
    Kc = torch.empty(0, 2, 256, 64, dtype=torch.bfloat16, device=dev)
    Pc = pisa.pisa_build_pyramid(Kc, N=0)
    q = torch.empty(0, 8, 64, dtype=torch.bfloat16, device=dev)
    kv = torch.empty(0, 2, 64, dtype=torch.bfloat16, device=dev)
    o = pisa.pisa_decode_step(q, kv, kv.clone(), Kc, Kc.clone(), Pc, torch.empty(0, dtype=torch.int32, device=dev), 16)
    assert o.shape == (0, 8, 64)


def test_empty_problems(monkeypatch):
    """The real library on CPU tensors: an empty problem returns before any device work, so the
    whole path from the binding through the C entry points runs without a GPU."""
    build()

    def bf16_any_device(t, name, dim=None):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or (dim is not None and t.dim() != dim):
            raise ValueError(name)

    monkeypatch.setattr(pisa, "_bf16", bf16_any_device)
    monkeypatch.setattr(pisa, "_stream", lambda t: None)
    monkeypatch.setattr(pisa, "_workspace", lambda ws, need, dev: torch.empty(max(need, 256), dtype=torch.uint8))
    monkeypatch.setattr(torch.cuda, "current_stream", lambda dev=None: types.SimpleNamespace(cuda_stream=0))
    _empty_calls("cpu", host_prefill=True)
