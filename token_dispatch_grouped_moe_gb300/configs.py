"""The layer shapes this library is tested and measured on.

Shapes follow the model families the COMET page and the DisagMoE summary
evaluate on (Mixtral-8x7B, Qwen2-MoE, DeepSeek-MoE; "COMET's Performance";
DisagMoE section 4), with the token-length sweep of DisagMoE section 4
(4K-32K). Only shapes are taken: every value is synthetic and seeded.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int          # tokens
    H: int          # hidden size
    F: int          # expert FFN width
    E: int          # routed experts
    k: int          # experts per token
    Fs: int = 0     # shared (always-on) expert width, 0 = none
    zipf: bool = False   # gate bias skews routing to Zipf(1.2) popularity
    seed: int = 0

    @property
    def R(self) -> int:
        return self.T * self.k

    def flops(self) -> int:
        """Algorithmic FLOPs of one forward: gate + routed SwiGLU + shared."""
        return (2 * self.T * self.H * self.E + 6 * self.R * self.H * self.F
                + 6 * self.T * self.H * self.Fs)

    def with_T(self, T: int) -> "LayerConfig":
        return replace(self, T=T, name=f"{self.name.split('@')[0]}@T{T}")


CONFIGS = {
    "tiny": LayerConfig("tiny", T=256, H=512, F=1024, E=8, k=2),
    "mixtral": LayerConfig("mixtral", T=8192, H=4096, F=14336, E=8, k=2),
    "qwen2": LayerConfig("qwen2", T=4096, H=3584, F=2560, E=64, k=8, Fs=20480),
    "dsk-1k": LayerConfig("dsk-1k", T=1024, H=2048, F=1408, E=64, k=6),
    "dsk-4k": LayerConfig("dsk-4k", T=4096, H=2048, F=1408, E=64, k=6),
    "dsk-16k": LayerConfig("dsk-16k", T=16384, H=2048, F=1408, E=64, k=6),
    "dsk-32k": LayerConfig("dsk-32k", T=32768, H=2048, F=1408, E=64, k=6),
    "mixtral-zipf": LayerConfig("mixtral-zipf", T=8192, H=4096, F=14336, E=8, k=2, zipf=True),
    # Mixtral-shaped with T and F quartered: small enough (0.7 GB of weights)
    # for multi-pass profiler captures, still larger than L2.
    "mixtral-prof": LayerConfig("mixtral-prof", T=2048, H=4096, F=3584, E=8, k=2),
    # Qwen2-shaped routed experts (H, F, k, 512 rows per expert) with 16 experts
    # and no shared expert: 0.9 GB of weights, for multi-pass profiler captures.
    "qwen2-prof": LayerConfig("qwen2-prof", T=1024, H=3584, F=2560, E=16, k=8),
}
