"""moe_layer_forward_host: the layer from and to host memory, the token
chunks' copies overlapping the kernels (GPU only).

Tokens are independent, so the chunked call must give the whole-batch
moe_layer_forward output bit for bit, whatever the chunk count; one small
case is also compared with the oracle directly.
"""
import numpy as np
import pytest
import torch

from token_dispatch_grouped_moe_gb300.inputs import bf16_bits, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from token_dispatch_grouped_moe_gb300 import build, lib as L
    build.build()
    L.load()
    return L


def _host_call(lib, dims, inp, g, ws, n_chunks):
    x_host = inp["x"].pin_memory()
    out_host = torch.full((dims.T, dims.H), float("nan"), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(g["x"])
    out_dev = torch.empty_like(g["x"])
    lib.layer_forward_host(dims, x_host, g["Wg"], g["W1"], g["W3"], g["W2"], ws, x_dev, out_dev, out_host,
                           W1s=g.get("W1s"), W3s=g.get("W3s"), W2s=g.get("W2s"), n_chunks=n_chunks)
    torch.cuda.synchronize()
    assert lib.check(ws) == lib.MOE_OK
    assert torch.equal(x_dev.cpu(), inp["x"])
    return out_host


# (T, H, F, E, k, F_shared): ragged chunk tails, a shared expert, more chunks
# asked for than 128-token chunks exist, and a shape whose whole batch takes
# CTA-pair GEMMs while its chunks do not
CASES = [(1000, 256, 192, 8, 2, 0), (700, 256, 128, 16, 4, 256), (300, 128, 128, 8, 2, 0),
         (8192, 512, 512, 8, 2, 0)]


@pytest.mark.parametrize("n_chunks", [0, 2, 3])
def test_host_call_keeps_the_batch_router(lib, n_chunks):
    """A batch that takes the tensor-core router (E >= 16 from 4096 tokens)
    in chunks of fewer tokens: each chunk still takes it, so the gate weights
    and the output are the whole batch's bit for bit."""
    T, H, F, E, k = 9000, 256, 128, 16, 2
    dims = lib.make_dims(T, H, F, E, k)
    assert lib.layer_plan(dims).router == lib.ROUTER_TENSOR
    inp = make_inputs(T, H, F, E, seed=9)
    g = {n: v.cuda() for n, v in inp.items()}
    ws = lib.workspace(dims)
    ref = lib.layer_forward(dims, g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], ws)
    torch.cuda.synchronize()
    out = _host_call(lib, dims, inp, g, ws, n_chunks)
    assert torch.equal(out.view(torch.int16), ref.cpu().view(torch.int16))


@pytest.mark.parametrize("shape", CASES)
@pytest.mark.parametrize("n_chunks", [0, 1, 2, 3, 8])
def test_host_call_matches_layer(lib, shape, n_chunks):
    T, H, F, E, k, Fs = shape
    inp = make_inputs(T, H, F, E, Fs=Fs, seed=5)
    g = {n: v.cuda() for n, v in inp.items()}
    dims = lib.make_dims(T, H, F, E, k, Fs)
    ws = lib.workspace(dims)
    ref = lib.layer_forward(dims, g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], ws, W1s=g.get("W1s"),
                            W3s=g.get("W3s"), W2s=g.get("W2s"))
    torch.cuda.synchronize()
    out = _host_call(lib, dims, inp, g, ws, n_chunks)
    assert torch.equal(out.view(torch.int16), ref.cpu().view(torch.int16))


def test_host_call_against_oracle(lib, oracle):
    T, H, F, E, k = 520, 256, 192, 8, 2
    inp = make_inputs(T, H, F, E, seed=7)
    g = {n: v.cuda() for n, v in inp.items()}
    dims = lib.make_dims(T, H, F, E, k)
    ws = lib.workspace(dims)
    out = _host_call(lib, dims, inp, g, ws, 3).float().numpy().astype(np.float64)
    b = {n: bf16_bits(v) for n, v in inp.items()}
    ref = oracle.layer_forward(b["x"], b["Wg"], b["W1"], b["W3"], b["W2"], k=k)["out"]
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert float(np.max(np.abs(out - ref))) <= 2e-2 * rms


def test_host_call_twice_and_stream_order(lib):
    """Two calls in a row on the caller's stream, the second reusing the
    staging buffers the first still reads: each result is the layer's."""
    T, H, F, E, k = 2048, 256, 128, 8, 2
    a = make_inputs(T, H, F, E, seed=11)
    bx = make_inputs(T, H, F, E, seed=12, only=("x",))["x"]
    g = {n: v.cuda() for n, v in a.items()}
    dims = lib.make_dims(T, H, F, E, k)
    ws = lib.workspace(dims)
    refs = []
    for x in (a["x"], bx):
        refs.append(lib.layer_forward(dims, x.cuda(), g["Wg"], g["W1"], g["W3"], g["W2"], ws).cpu())
    torch.cuda.synchronize()
    x_dev, out_dev = torch.empty_like(g["x"]), torch.empty_like(g["x"])
    outs = []
    for x in (a["x"], bx):
        o = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        lib.layer_forward_host(dims, x.pin_memory(), g["Wg"], g["W1"], g["W3"], g["W2"], ws, x_dev, out_dev, o,
                               n_chunks=2)
        outs.append(o)
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        assert torch.equal(o.view(torch.int16), r.view(torch.int16))
