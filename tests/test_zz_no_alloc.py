"""moe_permute_static: dispatch for callers that cannot provide scratch memory.

Some callers of this library cannot allocate device memory for it: a host
framework that hands its plug-ins no allocator or scratch hook, or a service
whose device memory budget is fixed at start-up. moe_permute_static keeps its
scratch in a fixed array inside the library instead of a caller workspace.
These tests call it through the C ABI and require the same results as
moe_permute and as the oracle's dispatch (integer outputs, so bit for bit),
on calls in a row of different shapes, since every call reuses the one array:
the single cooperative launch, and the two-launch path (more chunks than can
be resident at once), where the histogram in the array is written by one
kernel and read back by the next.

This file is collected last so that a failure here stops a run only after
every other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

from token_dispatch_grouped_moe_gb300.inputs import make_inputs


@pytest.fixture(scope="module")
def lib():
    from token_dispatch_grouped_moe_gb300 import build, lib as L
    build.build()
    L.load()
    return L


def _routed(lib, T, H, E, k):
    inp = make_inputs(T, H, 64, E, seed=T, only=("x", "Wg"))
    x, Wg = inp["x"].cuda(), inp["Wg"].cuda()
    dims = lib.make_dims(T, H, 64, E, k)
    idx, _ = lib.route(dims, x, Wg)
    return dims, x, idx


@pytest.mark.gpu
def test_permute_static_matches_permute_on_two_calls(lib, oracle):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # (T, H, E, k), run in this order: one cooperative launch each, then the
    # two-launch path (512 chunks of 2048 assignments), then a small one again
    shapes = [(3000, 256, 64, 6), (517, 128, 8, 2), (131072, 64, 8, 8), (1000, 64, 16, 4)]
    for T, H, E, k in shapes:
        dims, x, idx = _routed(lib, T, H, E, k)
        ws = lib.workspace(dims)
        ref = lib.permute(dims, idx, ws, x=x, want_x_perm=True)
        got = lib.permute_static(dims, idx, x=x, want_x_perm=True)
        torch.cuda.synchronize()
        assert lib.check(ws) == lib.MOE_OK
        for name, a, b in zip(("counts", "offsets", "src_row", "inv_pos", "x_perm"), ref, got):
            assert torch.equal(a, b), f"{name} differs for T={T} E={E} k={k}"
        assert int(got[1][E]) == T * k
        # and the oracle's stable counting sort, directly
        want = oracle.permute(idx.cpu().numpy(), E)
        for name, a, b in zip(("counts", "offsets", "src_row", "inv_pos"), got, want):
            assert np.array_equal(a.cpu().numpy(), b), f"{name} differs from the oracle for T={T}"
        xp = x[torch.from_numpy(want[2].astype(np.int64) // k).cuda()]
        assert torch.equal(got[4], xp), f"x_perm is not x in dispatch order for T={T}"
        del ws, ref, got


@pytest.mark.gpu
def test_permute_static_skips_a_bad_id(lib):
    """An expert id outside [0, E) is skipped, as documented: offsets[E] ends one
    short of T*k, and every other output equals moe_permute's (which reports
    the id through its error word)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    T, H, E, k = 3000, 128, 64, 6
    dims, x, idx = _routed(lib, T, H, E, k)
    bad_f = 4321
    idx.view(-1)[bad_f] = E
    ws = lib.workspace(dims)
    ref = lib.permute(dims, idx, ws, x=x, want_x_perm=True)
    got = lib.permute_static(dims, idx, x=x, want_x_perm=True)
    torch.cuda.synchronize()
    assert lib.check(ws) == 1   # moe_permute: MOE_ERR_INVALID_ARG in the error word
    R = T * k
    assert int(got[1][E]) == R - 1
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    assert torch.equal(got[2][:R - 1], ref[2][:R - 1])
    keep = torch.ones(R, dtype=torch.bool, device=idx.device)
    keep[bad_f] = False
    assert torch.equal(got[3][keep], ref[3][keep])
    assert torch.equal(got[4][:R - 1], ref[4][:R - 1])
    assert bad_f not in set(got[2][:R - 1].tolist())


def test_permute_static_rejects_oversize(lib):
    """A shape whose histogram does not fit in the fixed array is refused on the
    host, before any launch (so this needs no GPU); so are the shapes that
    moe_permute refuses."""
    L = lib.load()
    dummy = ctypes.c_void_p(256)

    def call(dims):
        return L.moe_permute_static(ctypes.byref(dims), dummy, dummy, dummy, dummy, dummy, None, None,
                                    None)

    assert call(lib.make_dims(1 << 20, 64, 64, 256, 8)) == 2   # 4096 chunks x 256 experts: MOE_ERR_UNSUPPORTED
    assert call(lib.make_dims(64, 64, 100, 8, 2)) == 2         # F not a multiple of 64, as moe_permute
    assert call(lib.make_dims(64, 64, 64, 8, 9)) == 1          # k > E: MOE_ERR_INVALID_ARG
