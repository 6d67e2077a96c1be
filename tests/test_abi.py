"""The C-ABI library builds, loads without a GPU and exports every entry point of
include/pisa.h; host-side geometry and argument checks (no compute launches)."""
import ctypes as ct
import os
import re

import pytest

import hierarchical_top_block_gb300 as pisa
from hierarchical_top_block_gb300.build import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pisa.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return pisa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pisa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("pisa_build_pyramid", "pisa_select_prefill", "pisa_sparse_attn_prefill", "pisa_decode_step",
                 "pisa_prefill_host", "pisa_pyramid_nodes", "pisa_select_workspace_bytes",
                 "pisa_get_last_device_error", "pisa_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} is declared in include/pisa.h but not exported"


def test_python_binding_has_the_same_names():
    for name in declared_functions():
        assert hasattr(pisa, name), f"binding lacks {name}"


def test_geometry_matches_the_oracle(lib, oracle_impl):
    for n in (0, 1, 63, 64, 65, 1000, 4096, 32768, 131073, 262144):
        assert pisa.pisa_pyramid_levels(n) == oracle_impl.num_levels(n)
        assert pisa.pisa_pyramid_nodes(n) == oracle_impl.pyramid_nodes(n)


def test_workspace_query(lib):
    ok = pisa.pisa_select_workspace_bytes(pisa.make_shape(1, 262144, 16, 1, 128), pisa.make_params(16))
    assert ok > 0 and ok % 256 == 0
    assert pisa.pisa_select_workspace_bytes(pisa.make_shape(1, 4096, 16, 1, 96), pisa.make_params(16)) == 0
    assert pisa.pisa_select_workspace_bytes(pisa.make_shape(1, 4096, 16, 1, 128), pisa.make_params(33)) == 0
    assert pisa.pisa_select_workspace_bytes(pisa.make_shape(1, 4096, 16, 1, 128), pisa.make_params(32)) > 0
    assert pisa.pisa_select_workspace_bytes(pisa.make_shape(1, 4096, 12, 4, 128), pisa.make_params(8)) == 0


def test_argument_errors_without_a_gpu(lib):
    shape = pisa.make_shape(1, 128, 4, 1, 64)
    # NULL pointers are rejected before anything touches the device
    assert lib.pisa_build_pyramid(None, None, shape, pisa.make_params(4), None) == 1
    assert lib.pisa_sparse_attn_prefill(None, None, None, None, None, None, shape, pisa.make_params(4), None) == 1
    # unsupported head dim / group size / block size
    assert lib.pisa_build_pyramid(None, None, pisa.make_shape(1, 128, 4, 1, 80), pisa.make_params(4), None) == 2
    assert lib.pisa_build_pyramid(None, None, shape, pisa.make_params(4, C=32), None) == 2
    # a scoring other than LSE / PISA-1 / PISA-2 is an argument error
    assert lib.pisa_build_pyramid(None, None, shape, pisa.make_params(4, scoring=3), None) == 1
    # empty problems are a no-op
    assert lib.pisa_build_pyramid(None, None, pisa.make_shape(0, 128, 4, 1, 64), pisa.make_params(4), None) == 0
    assert lib.pisa_status_string(2).decode() == "unsupported shape or parameter"
    assert b"sm_103a" in lib.pisa_version()


def test_prefill_host_chunk_plan(lib):
    """The host-buffer prefill's query chunks: they tile [0, N) in order, there are at most 11,
    they double from N/32 (at least 8192) up to N/4 and halve again at the end, and a short
    sequence runs as one chunk."""
    assert pisa.pisa_prefill_host_chunks(0) == [0]
    for n in (1, 63, 4096, 8192):
        assert pisa.pisa_prefill_host_chunks(n) == [0, n]
    for n in (8193, 20000, 35000, 65536, 245633, 262144, 262207, 1 << 20, (1 << 24) + 5, 10**10 + 7):
        b = pisa.pisa_prefill_host_chunks(n)
        sizes = [hi - lo for lo, hi in zip(b, b[1:])]
        assert b[0] == 0 and b[-1] == n and min(sizes) > 0 and len(sizes) <= 11, (n, sizes)
        lo = max(n // 32 // 64 * 64, 8192)
        cap = max(n // 4 // 64 * 64, lo)
        assert max(sizes) <= cap + 64, (n, sizes)
        # the rising ramp and the falling one mirror each other
        r = 0
        while r < len(sizes) and sizes[r] == lo << r and (lo << r) < cap:
            r += 1
        assert sizes[len(sizes) - r:] == sizes[:r][::-1], (n, sizes)
    # the 256K plan the benchmark's end-to-end leg runs
    sizes = [hi - lo for lo, hi in zip(pisa.pisa_prefill_host_chunks(262144), pisa.pisa_prefill_host_chunks(262144)[1:])]
    assert sizes == [8192, 16384, 32768, 49152, 49152, 49152, 32768, 16384, 8192]
    # errors: negative N, NULL bounds, too small a buffer
    buf = (ct.c_longlong * 17)()
    assert lib.pisa_prefill_host_chunks(-1, buf, 17) == -1
    assert lib.pisa_prefill_host_chunks(262144, None, 17) == -1
    assert lib.pisa_prefill_host_chunks(262144, buf, 9) == -1
    assert lib.pisa_prefill_host_chunks(262144, buf, 10) == 9


def test_entry_list_limit(lib):
    """The selection and the backward keep per-block lists of up to B * H_kv * N * K entries
    with 32-bit offsets: a shape at 2^31 entries is refused before anything touches the
    device (workspace queries give 0), one entry below it is accepted by the queries."""
    N = 1 << 23
    big = pisa.make_shape(1, N, 16, 16, 64, N)  # G_Q = 1, d = 64: B * N_cap * H_q = 2^27 passes the other checks
    at, below = pisa.make_params(16), pisa.make_params(15)
    assert pisa.pisa_select_workspace_bytes(big, at) == 0
    assert pisa.pisa_attn_backward_workspace_bytes(big, at) == 0
    assert pisa.pisa_prefill_host_workspace_bytes(big, at) == 0
    assert pisa.pisa_select_workspace_bytes(big, below) > 0
    assert pisa.pisa_attn_backward_workspace_bytes(big, below) > 0
    assert pisa.pisa_attn_backward_min_workspace_bytes(big, at) == 0
    assert pisa.pisa_attn_backward_min_workspace_bytes(big, below) > 0
    fake = ct.c_void_p(1 << 20)  # aligned, never dereferenced: the call returns before using it
    assert lib.pisa_select_prefill(fake, fake, fake, fake, None, None, fake, 1 << 40, big, at, None) == 2
    assert lib.pisa_select_prefill_noalloc(fake, fake, fake, fake, None, None, big, at, None) == 2
    assert lib.pisa_sparse_attn_backward(*([fake] * 11), 1 << 40, big, at, None) == 2
    assert lib.pisa_prefill_host(fake, fake, fake, fake, None, None, fake, 1 << 40, big, at, None) == 2


def test_parameter_rules(lib):
    """Each documented argument rule is enforced before anything touches the device (status 1
    invalid argument, 2 unsupported, 6 workspace too small); the pointers are aligned fakes
    that no refused call dereferences."""
    fake = ct.c_void_p(1 << 20)
    base = {"B": 1, "N": 4096, "H_q": 16, "H_kv": 1, "d": 128, "N_cap": 0}

    def shape(**kw):
        s = dict(base, **kw)
        return pisa.make_shape(s["B"], s["N"], s["H_q"], s["H_kv"], s["d"], s["N_cap"])

    def sel(sh, pr, ws=fake, Q=fake):
        return lib.pisa_select_prefill(Q, fake, fake, fake, None, None, ws, 1 << 40, sh, pr, None)

    p16 = pisa.make_params(16)
    cases = [
        (sel(shape(), pisa.make_params(0)), 2), (sel(shape(), pisa.make_params(33)), 2),
        (sel(shape(H_q=12, H_kv=8), p16), 1), (sel(shape(H_q=3, H_kv=1), p16), 2), (sel(shape(H_q=32, H_kv=1), p16), 2),
        (sel(shape(d=96), p16), 2), (sel(shape(B=-1), p16), 1), (sel(shape(H_q=0), p16), 1),
        (sel(shape(N_cap=100), p16), 1), (sel(shape(N_cap=8192), p16), 1),
        (sel(shape(N=1 << 25), p16), 2),
        (sel(shape(B=64, N=1 << 24, H_q=16, H_kv=16), pisa.make_params(1)), 2),
        (sel(shape(), pisa.make_params(16, scale=float("nan"))), 1),
        (sel(shape(), pisa.pisa_params(64, 2, 16, 2, 0.0, 0)), 1),      # causal must be 0 or 1
        (sel(shape(), pisa.make_params(16, scoring=3)), 1),
        (sel(shape(), pisa.make_params(16, g=4)), 2),
        (sel(shape(), p16, ws=ct.c_void_p((1 << 20) + 16)), 1),          # ws must be 256-byte aligned
        (sel(shape(), p16, Q=ct.c_void_p((1 << 20) + 2)), 1),            # tensors 16-byte aligned
        # the allocation-free selection reports the same statuses as the workspace one
        (lib.pisa_select_prefill_noalloc(fake, fake, fake, fake, None, None, shape(H_q=12, H_kv=8), p16, None), 1),
        (lib.pisa_select_prefill_noalloc(fake, fake, fake, fake, None, None, shape(),
                                         pisa.pisa_params(64, 2, 16, 2, 0.0, 0), None), 1),
        (lib.pisa_select_prefill_noalloc(fake, fake, fake, fake, None, None, shape(), pisa.make_params(33), None), 2),
        (lib.pisa_select_prefill_noalloc(None, None, None, None, None, None, shape(B=0), p16, None), 0),
        (lib.pisa_sparse_attn_prefill(fake, fake, fake, fake, fake, None, shape(N_cap=100), p16, None), 1),
        (lib.pisa_sparse_attn_prefill(fake, fake, fake, ct.c_void_p((1 << 20) + 4), fake, None, shape(), p16, None), 1),
        (lib.pisa_decode_step(*([fake] * 10), shape(N=0, N_cap=0), p16, None), 1),
        (lib.pisa_decode_step(*([fake] * 10), shape(N=0, N_cap=4096), pisa.make_params(16, causal=False), None), 2),
        # the decode step with the logits scratch: too small, misaligned, refused arguments
        (lib.pisa_decode_step_ws(*([fake] * 10), fake, 1024, shape(N=0, N_cap=4096), p16, None), 6),
        (lib.pisa_decode_step_ws(*([fake] * 10), ct.c_void_p((1 << 20) + 16), 1 << 40, shape(N=0, N_cap=4096), p16,
                                 None), 1),
        (lib.pisa_decode_step_ws(*([fake] * 10), fake, 1 << 40, shape(N=0, N_cap=0), p16, None), 1),
        (lib.pisa_decode_step_ws(*([fake] * 10), fake, 1 << 40, shape(N=0, N_cap=4096), pisa.make_params(33), None), 2),
        (lib.pisa_decode_step_ws(*([None] * 11), 0, shape(B=0, N=0, N_cap=4096), p16, None), 0),
        (lib.pisa_prefill_host(fake, fake, fake, fake, None, None, fake, 1 << 40, shape(N_cap=8192), p16, None), 1),
        (lib.pisa_prefill_host(fake, fake, fake, fake, None, None, ct.c_void_p((1 << 20) + 16), 1 << 40, shape(), p16,
                               None), 1),
        (lib.pisa_prefill_host(fake, fake, fake, fake, None, None, fake, 1024, shape(), p16, None), 6),
        (lib.pisa_prefill_host(None, fake, fake, fake, None, None, fake, 1 << 40, shape(), p16, None), 1),
        (lib.pisa_sparse_attn_backward(*([fake] * 11), 1024, shape(), p16, None), 6),
        (lib.pisa_select_bsa(fake, fake, fake, fake, 1024, shape(), p16, None), 6),
        (lib.pisa_select_bsa(fake, fake, fake, ct.c_void_p((1 << 20) + 16), 1 << 40, shape(), p16, None), 1),
        (lib.pisa_select_bsa(fake, fake, fake, fake, 1 << 40, shape(N_cap=8192), p16, None), 1),
        (lib.pisa_select_bsa(fake, fake, fake, fake, 1 << 40, shape(), pisa.make_params(33), None), 2),
        (lib.pisa_select_bsa(None, None, None, None, 0, shape(B=0), p16, None), 0),
        (lib.pisa_check_wait_timeout(999, None), 1), (lib.pisa_check_wait_timeout(10**10 + 1, None), 1),
        (lib.pisa_sparse_attn_backward(*([fake] * 10), ct.c_void_p((1 << 20) + 64), 1 << 40, shape(), p16, None), 1),
    ]
    assert [got for got, _ in cases] == [want for _, want in cases]


def test_decode_workspace_bytes(lib):
    """The decode step's logits scratch: B * H_kv * 2K candidate leaves * 8 key octets * 4 lanes
    per head (G_Q heads up to 8, all 32 lanes twice when G_Q > 8: the second MMA row tile) of
    fp32 pairs; 0 for the arguments the step refuses."""
    def need(B, H_q, H_kv, K, N_cap=4096, causal=True):
        return pisa.pisa_decode_workspace_bytes(pisa.make_shape(B, 0, H_q, H_kv, 128, N_cap),
                                                pisa.make_params(K, causal=causal))
    assert need(64, 32, 8, 16, N_cap=131072 + 300) == 64 * 8 * 32 * 8 * 16 * 8 == 16777216
    assert need(4, 64, 4, 32) == 4 * 4 * 64 * 8 * 2 * 32 * 8
    assert need(3, 24, 3, 5) == 3 * 3 * 10 * 8 * 32 * 8
    assert need(2, 4, 4, 16) == 2 * 4 * 32 * 8 * 4 * 8
    assert need(2, 16, 2, 33) == 0 and need(2, 16, 2, 16, N_cap=0) == 0 and need(2, 16, 2, 16, causal=False) == 0


def test_backward_workspace_with_and_without_ds():
    """With d = 128 and G_Q of 8 or 16 the full backward scratch adds dS of every (query,
    selected block) pair (bf16, G_Q x 64 per pair) and a 4-byte entry per pair to the least
    scratch; elsewhere the two sizes are equal."""
    B, N, K = 1, 4096, 16
    for H_q, H_kv, d, extra in ((16, 1, 128, True), (32, 4, 128, True), (16, 4, 128, False), (16, 1, 64, False)):
        shape, params = pisa.make_shape(B, N, H_q, H_kv, d, N), pisa.make_params(K)
        full = pisa.pisa_attn_backward_workspace_bytes(shape, params)
        least = pisa.pisa_attn_backward_min_workspace_bytes(shape, params)
        if extra:
            pairs = B * H_kv * N * K
            assert full - least >= pairs * (H_q // H_kv) * 64 * 2 + pairs * 4
            assert full - least <= pairs * (H_q // H_kv) * 64 * 2 + pairs * 4 + 512
        else:
            assert full == least > 0
