"""The tensor-core router (GPU only), through the C ABI.

The expert ids must be the canonical fp32 order's bit for bit (the oracle's),
whatever path each token takes: proven by the error bound on the tensor-core
logits, or recomputed in the canonical order. Gate weights within 1e-5
relative. The bound's tensor-core part is checked against exact (fp64) dot
products, on ordinary and on wide-range inputs.
"""
import numpy as np
import pytest
import torch

from token_dispatch_grouped_moe_gb300.inputs import bf16_bits, make_inputs

pytestmark = pytest.mark.gpu

TOL_W = 1e-5


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_dispatch_grouped_moe_gb300 import build, lib as L
    build.build()
    L.load()
    return L


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _route(lib, x, Wg, k, bias=None, renormalize=True, force_exact=False, want_fast=False):
    T, H = x.shape
    E = Wg.shape[1]
    dims = lib.make_dims(T, H, 64, E, k)
    ws = lib.workspace(dims)
    bias_t = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).cuda()
    out = lib.route_tc_selftest(dims, x.cuda(), Wg.cuda(), ws, bias=bias_t, renormalize=renormalize,
                                force_exact=force_exact, want_fast=want_fast)
    torch.cuda.synchronize()
    assert lib.check(ws) == lib.MOE_OK
    return out


# (T, H, E, k): every padded width NP = 16, 32, 48, 64, ragged token tails
SHAPES = [(512, 256, 8, 2), (1000, 512, 16, 4), (777, 64, 24, 3), (3000, 2048, 32, 6),
          (600, 192, 40, 8), (1500, 1024, 48, 5), (700, 320, 56, 7), (2100, 2048, 64, 6),
          (513, 3584, 64, 8), (640, 4096, 8, 8),
          # from 8192 tokens the recomputation runs as (token, member pair) items and an
          # order pass; without renormalisation every expert is a member (32 pairs)
          (8200, 512, 64, 6), (8192, 256, 16, 4)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("variant", ["plain", "bias", "no_renorm"])
def test_route_tc_matches_oracle(lib, oracle, shape, variant):
    T, H, E, k = shape
    inp = make_inputs(T, H, 64, E, seed=T + E, only=("x", "Wg"))
    bias = None
    if variant == "bias":
        bias = (np.random.default_rng(E).standard_normal(E) * 0.5).astype(np.float32)
    renorm = variant != "no_renorm"
    idx, w, _, _, n_exact = _route(lib, inp["x"], inp["Wg"], k, bias=bias, renormalize=renorm)
    b = {n: bf16_bits(v) for n, v in inp.items()}
    logits, ridx, rw = oracle.route(b["x"], b["Wg"], k, bias)
    if not renorm:
        rw = oracle.gate_weights_full(logits, ridx)
    assert np.array_equal(idx.cpu().numpy(), ridx), "top-k ids differ from the canonical order"
    gw = w.cpu().numpy()
    assert np.allclose(gw, rw, rtol=TOL_W, atol=1e-7), f"gate weights differ: {np.max(np.abs(gw - rw))}"
    print(f"[T={T} H={H} E={E} k={k} {variant}] tokens recomputed in the canonical order: "
          f"{n_exact} of {T} ({100.0 * n_exact / T:.2f}%)")


@pytest.mark.parametrize("shape", [(2048, 4096, 8, 2), (2048, 2048, 64, 6), (1024, 3584, 64, 8),
                                   (20480, 512, 64, 6)])   # more tiles than SMs: two CTAs of 4 stages per SM
@pytest.mark.parametrize("inputs", ["randn", "wide_range"])
def test_route_tc_fast_logit_bound(lib, shape, inputs):
    """The tensor-core logits lie within the bound the screening assumes for
    them, c_fast ||x_t|| max_e ||w_e||, of the exact dot products (fp64 of the
    bf16 inputs); the margin is printed. wide_range: every element scaled by a
    random power of two in [2^-12, 2^12], so that each MMA step adds terms of
    very different magnitudes (the case its alignment and truncation bound)."""
    T, H, E, k = shape
    inp = make_inputs(T, H, 64, E, seed=H + E, only=("x", "Wg"))
    x, Wg = inp["x"], inp["Wg"]
    if inputs == "wide_range":
        rng = np.random.default_rng(5)
        x = (x.float() * torch.from_numpy(np.exp2(rng.integers(-12, 13, x.shape)).astype(np.float32))).to(torch.bfloat16)
        Wg = (Wg.float() * torch.from_numpy(np.exp2(rng.integers(-12, 13, Wg.shape)).astype(np.float32))).to(torch.bfloat16)
    idx, w, fast, bound, n_exact = _route(lib, x, Wg, k, want_fast=True)
    exact = _f64(bf16_bits(x)) @ _f64(bf16_bits(Wg))
    err = np.abs(fast.cpu().numpy().astype(np.float64) - exact)
    b = bound.cpu().numpy().astype(np.float64)[:, None]
    ratio = float(np.max(err / b))
    print(f"[{inputs} T={T} H={H} E={E}] max |fast - exact| / bound = {ratio:.3e}; "
          f"recomputed {n_exact} of {T}")
    assert np.all(err <= b), f"tensor-core logits outside the assumed bound (max ratio {ratio:.3f})"


ORDER_CASES = [
    (64, [(0, 2.0 ** 24), (8, 1.0), (9, -2.0 ** 24)], 1.0),
    (256, [(0, 2.0 ** 24), (8, 1.0), (128, -2.0 ** 24)], 1.0),
    (320, [(0, 2.0 ** 24), (256, 1.0), (8, -2.0 ** 24)], 0.0),
    (64, [(0, -2.0 ** 24), (1, 1.0), (2, 2.0 ** 24)], 1.0),
    (320, [(0, 2.0 ** 24), (128, -2.0 ** 24), (256, 1.0)], 0.0),
]


@pytest.mark.parametrize("E", [8, 16, 32, 64])
@pytest.mark.parametrize("case", range(len(ORDER_CASES)))
def test_route_tc_order_sensitive(lib, oracle, E, case):
    """Token 0 is a case whose fp32 logit depends on the summation order
    (2^24 + 1 rounds to 2^24): its tensor-core logit can be off by 1, far
    beyond its gap, so the bound must send it to the canonical recomputation,
    which gives expert 0 the canonical value. The other 511 tokens are random
    (through the same gate, whose column 0 holds the +-2^24 entries)."""
    H, placements, want = ORDER_CASES[case]
    T = 512
    rng = np.random.default_rng(case)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32))
    x[0].zero_()
    Wg = torch.full((H, E), 0.0)
    Wg[:, 2:] = -1.0 / H
    for h, v in placements:
        x[0, h] = 1.0
        Wg[h, 0] = v
    hb = placements[1][0] if placements[1][1] == 1.0 else placements[2][0]
    Wg[hb, 1] = 0.5
    x, Wg = x.to(torch.bfloat16), Wg.to(torch.bfloat16)
    idx, w, _, _, n_exact = _route(lib, x, Wg, 2)
    logits, ridx, rw = oracle.route(bf16_bits(x), bf16_bits(Wg), 2)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.allclose(w.cpu().numpy(), rw, rtol=TOL_W, atol=1e-7)
    assert float(logits[0, 0]) == want
    assert n_exact >= 1


@pytest.mark.parametrize("shape", [(1024, 2048, 64, 6), (2048, 4096, 8, 2), (600, 512, 24, 3),
                                   (8192, 512, 64, 6), (9000, 256, 16, 3)])
def test_route_tc_all_exact_equals_fma_router(lib, shape):
    """With every token sent through the canonical recomputation, the ids and
    weights equal the FMA router's (moe_route) bit for bit."""
    T, H, E, k = shape
    inp = make_inputs(T, H, 64, E, seed=11, only=("x", "Wg"))
    idx, w, _, _, n_exact = _route(lib, inp["x"], inp["Wg"], k, force_exact=True)
    assert n_exact == T
    dims = lib.make_dims(T, H, 64, E, k)
    ridx, rw = lib.route(dims, inp["x"].cuda(), inp["Wg"].cuda())
    torch.cuda.synchronize()
    assert torch.equal(idx, ridx)
    assert torch.equal(w, rw)


@pytest.mark.parametrize("shape", [(2048, 1024, 1408, 64, 6, 0), (1500, 512, 256, 8, 2, 0),
                                   (1024, 448, 320, 16, 4, 640)])
def test_layer_tensor_router_vs_fma_router(lib, shape):
    """The layer call with the tensor-core router and with the FMA router:
    the same ids, counts and dispatch bit for bit; gate weights within fp32
    rounding of each other; the outputs within two bf16 ulps, or 1e-5 rms
    where the weighted rows cancel to near zero."""
    T, H, F, E, k, Fs = shape
    inp = make_inputs(T, H, F, E, Fs=Fs, seed=19)
    g = {n: v.cuda() for n, v in inp.items()}
    dims = lib.make_dims(T, H, F, E, k, Fs)
    ws = lib.workspace(dims)
    res = {}
    try:
        for mode in (lib.ROUTER_OPT_TENSOR, lib.ROUTER_OPT_FMA):
            lib.set_router(mode)
            r = lib.routing_buffers(dims, "cuda")
            out = lib.layer_forward(dims, g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], ws, W1s=g.get("W1s"),
                                    W3s=g.get("W3s"), W2s=g.get("W2s"), routing=r)
            torch.cuda.synchronize()
            assert lib.check(ws) == lib.MOE_OK
            res[mode] = (r, out.clone())
    finally:
        lib.set_router(lib.ROUTER_OPT_AUTO)
    (ra, oa), (rb, ob) = res[lib.ROUTER_OPT_TENSOR], res[lib.ROUTER_OPT_FMA]
    for n in ("topk_idx", "counts", "offsets", "src_row", "inv_pos"):
        assert torch.equal(getattr(ra, n), getattr(rb, n)), n
    assert torch.allclose(ra.topk_w, rb.topk_w, rtol=2e-6, atol=1e-8)
    d = (oa.float() - ob.float()).abs()
    ulp = ob.float().abs() * 2.0 ** -7
    rms = float(ob.float().pow(2).mean().sqrt())
    assert bool((d <= 2 * ulp + 1e-5 * rms).all()), float((d - 2 * ulp).max() / rms)
