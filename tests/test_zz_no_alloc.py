"""The allocation-free selection entry point, called through the C ABI.

pisa_select_prefill_noalloc serves callers that cannot allocate device memory (a host
that owns the allocator, a pool they may not grow, a loop that must not call cudaMalloc):
it runs the same selection on the library's fixed device scratch array.  This file checks,
on two calls in a row with different shapes (so a stale scratch would show), that it gives
what pisa_select_prefill gives with a caller-supplied workspace, and that shapes too large
for the array are refused.  It is named so that pytest collects it last.
"""
import ctypes as ct

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pisa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hierarchical_top_block_gb300.build import build

    build()
    import hierarchical_top_block_gb300 as p

    return p


def _via_c_abi(pisa, Q, K, P, K_sel):
    """Calls the C entry point directly with preallocated outputs."""
    B, N, H_q, d = Q.shape
    H_kv = K.shape[1]
    idx = torch.full((B, H_kv, N, K_sel), -7, dtype=torch.int32, device=Q.device)
    score = torch.full((B, H_kv, N, 2 * K_sel), 1234.0, dtype=torch.float32, device=Q.device)
    s2 = torch.full((B, H_kv, N, K_sel), -7, dtype=torch.int32, device=Q.device)
    rc = pisa.lib().pisa_select_prefill_noalloc(
        ct.c_void_p(Q.data_ptr()), ct.c_void_p(K.data_ptr()), ct.c_void_p(P.data_ptr()), ct.c_void_p(idx.data_ptr()),
        ct.c_void_p(score.data_ptr()), ct.c_void_p(s2.data_ptr()), pisa.make_shape(B, N, H_q, H_kv, d, N),
        pisa.make_params(K_sel), ct.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, pisa.pisa_status_string(rc)
    return idx, score, s2


@pytest.mark.parametrize("calls", [("prefill_4k", "tiny")])
def test_noalloc_matches_workspace_entry_point_twice(pisa, calls):
    for name in calls:
        w = W.WORKLOADS[name]
        Q, K, V = W.prefill_inputs(w, "cuda")
        P = pisa.pisa_build_pyramid(K)
        idx_ref, score_ref, s2_ref = pisa.pisa_select_prefill(Q, K, P, w.K, want_scores=True, want_s2=True)
        idx, score, s2 = _via_c_abi(pisa, Q, K, P, w.K)
        torch.cuda.synchronize()
        assert pisa.pisa_get_last_device_error() == 0
        assert torch.equal(idx, idx_ref), name
        assert torch.equal(s2, s2_ref), name
        valid = torch.isfinite(score_ref) & (s2_ref.repeat_interleave(2, dim=-1) >= 0)
        diff = (score - score_ref).abs()[valid]
        assert diff.numel() == 0 or float(diff.max()) <= 1e-3, name


def test_noalloc_refuses_shapes_beyond_its_scratch(pisa):
    w = W.WORKLOADS["prefill_256k"]
    shape = pisa.make_shape(w.B, w.N, w.H_q, w.H_kv, w.d, w.N)
    assert pisa.pisa_select_workspace_bytes(shape, pisa.make_params(w.K)) > (32 << 20)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    rc = pisa.lib().pisa_select_prefill_noalloc(ct.c_void_p(dummy.data_ptr()), ct.c_void_p(dummy.data_ptr()),
                                                ct.c_void_p(dummy.data_ptr()), ct.c_void_p(dummy.data_ptr()), None,
                                                None, shape, pisa.make_params(w.K), None)
    assert rc == 6  # PISA_ERR_WORKSPACE, nothing launched
    assert pisa.pisa_get_last_device_error() == 0
