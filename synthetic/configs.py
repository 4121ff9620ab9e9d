"""The five synthetic DiT workloads (shapes only; no arithmetic of the method).

Each workload is a stack of identical DiT blocks run over R requests of T
latent tokens each, with the block weights split into dp_size host shards.
Head width d = hidden / heads.  The tokens stand in for flattened latents:
a 1024x1024 image as a 64x64 latent with patch size 1 gives 4096 tokens, a
spatio-temporal video latent flattened gives 16384 tokens.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class WorkloadConfig:
    name: str
    blocks: int
    hidden: int
    heads: int
    mlp: int
    cond_dim: int
    requests: int
    tokens: int
    dp_size: int
    seed: int = 0

    @property
    def head_dim(self) -> int:
        return self.hidden // self.heads

    def describe(self) -> str:
        return (f"{self.name}: L={self.blocks} h={self.hidden} H={self.heads} d={self.head_dim} "
                f"m={self.mlp} C={self.cond_dim} R={self.requests} T={self.tokens} dp={self.dp_size}")


CONFIGS = {
    "tiny": WorkloadConfig("tiny", 4, 256, 4, 1024, 256, 1, 256, 4),
    "t2i": WorkloadConfig("t2i", 16, 1536, 24, 6144, 256, 1, 4096, 4),
    "deep": WorkloadConfig("deep", 28, 3072, 24, 12288, 256, 1, 8192, 8),
    "video": WorkloadConfig("video", 40, 5120, 40, 20480, 256, 1, 16384, 4),
    "large": WorkloadConfig("large", 24, 8192, 64, 32768, 256, 4, 4096, 4),
}


def get_config(name: str) -> WorkloadConfig:
    try:
        return CONFIGS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS)}") from None
