"""Seeded generator and the stored Zipf bias (CPU only)."""
import os

import numpy as np
import torch

from token_dispatch_grouped_moe_gb300.configs import CONFIGS
from token_dispatch_grouped_moe_gb300.inputs import bf16_bits, bits_to_bf16, make_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_zipf_bias() -> np.ndarray:
    vals = [float.fromhex(l.strip()) for l in open(os.path.join(GOLDEN, "zipf_bias_mixtral.txt"))
            if l.strip() and not l.startswith("#")]
    return np.array(vals, np.float32)


def test_generator_is_seeded_and_shaped():
    a = make_inputs(16, 64, 32, 4, Fs=48, seed=3)
    b = make_inputs(16, 64, 32, 4, Fs=48, seed=3)
    c = make_inputs(16, 64, 32, 4, Fs=48, seed=4)
    shapes = dict(x=(16, 64), Wg=(64, 4), W1=(4, 64, 32), W3=(4, 64, 32), W2=(4, 32, 64),
                  W1s=(64, 48), W3s=(64, 48), W2s=(48, 64))
    for n, s in shapes.items():
        assert tuple(a[n].shape) == s and a[n].dtype == torch.bfloat16
        assert torch.equal(a[n], b[n])
        assert not torch.equal(a[n], c[n])
    # Each tensor has its own seed offset: x and W1 differ even at equal shapes.
    d = make_inputs(64, 64, 64, 1, seed=0)
    assert not torch.equal(d["x"], d["W1"][0] / 0.02)


def test_generator_sigmas():
    inp = make_inputs(512, 256, 256, 2, seed=0)
    assert abs(inp["x"].float().std().item() - 1.0) < 0.02
    for n in ("Wg", "W1", "W3", "W2"):
        assert abs(inp[n].float().std().item() - 0.02) < 0.001


def test_bits_roundtrip():
    t = make_inputs(4, 8, 8, 1, seed=1)["x"]
    assert torch.equal(bits_to_bf16(bf16_bits(t)), t)


def test_zipf_bias_shares(oracle):
    """The stored bias gives the hottest expert 38-45% of the assignments on
    the seeded Mixtral-shaped x, and a popularity that falls with the id."""
    cfg = CONFIGS["mixtral-zipf"]
    bias = load_zipf_bias()
    assert bias.shape == (cfg.E,)
    inp = make_inputs(cfg.T, cfg.H, 64, cfg.E, seed=cfg.seed, only=("x", "Wg"))
    _, idx, _ = oracle.route(bf16_bits(inp["x"]), bf16_bits(inp["Wg"]), cfg.k, bias)
    share = np.bincount(idx.reshape(-1), minlength=cfg.E) / idx.size
    assert 0.38 <= share[0] <= 0.45
    assert np.all(np.diff(share) < 0)
