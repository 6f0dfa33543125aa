"""moe_permute_static: dispatch for callers that cannot provide scratch memory.

Some callers of this library cannot allocate device memory for it: a host
framework that hands its plug-ins no allocator or scratch hook, or a service
whose device memory budget is fixed at start-up. moe_permute_static keeps its
scratch in a fixed array inside the library instead of a caller workspace.
These tests call it through the C ABI and require the same results as
moe_permute (integer outputs, so bit for bit), on two calls in a row of
different shapes, since every call reuses the one array.

This file is collected last so that a failure here stops a run only after
every other test has run.
"""
import ctypes

import pytest
import torch

from token_dispatch_grouped_moe_gb300.inputs import make_inputs


@pytest.fixture(scope="module")
def lib():
    from token_dispatch_grouped_moe_gb300 import build, lib as L
    build.build()
    L.load()
    return L


@pytest.mark.gpu
def test_permute_static_matches_permute_on_two_calls(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    shapes = [(3000, 256, 64, 6), (517, 128, 8, 2)]   # (T, H, E, k), run in this order
    for T, H, E, k in shapes:
        inp = make_inputs(T, H, 64, E, seed=T, only=("x", "Wg"))
        x, Wg = inp["x"].cuda(), inp["Wg"].cuda()
        dims = lib.make_dims(T, H, 64, E, k)
        idx, _ = lib.route(dims, x, Wg)
        ws = lib.workspace(dims)
        ref = lib.permute(dims, idx, ws, x=x, want_x_perm=True)
        got = lib.permute_static(dims, idx, x=x, want_x_perm=True)
        torch.cuda.synchronize()
        assert lib.check(ws) == lib.MOE_OK
        for name, a, b in zip(("counts", "offsets", "src_row", "inv_pos", "x_perm"), ref, got):
            assert torch.equal(a, b), f"{name} differs for T={T} E={E} k={k}"
        assert int(got[1][E]) == T * k


def test_permute_static_rejects_oversize(lib):
    """A shape whose histogram does not fit in the fixed array is refused on the
    host, before any launch (so this needs no GPU)."""
    dims = lib.make_dims(1 << 20, 64, 64, 256, 8)   # 4096 chunks x 256 experts
    dummy = ctypes.c_void_p(256)
    st = lib.load().moe_permute_static(ctypes.byref(dims), dummy, dummy, dummy, dummy, dummy,
                                       None, None, None)
    assert st == 2   # MOE_ERR_UNSUPPORTED
