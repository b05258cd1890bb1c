"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no part of the method's arithmetic (no quantization, no dot
products, no scaling): only workload shapes and seeded normal draws.  It is
the one module both the tests/benchmark CUDA side and the oracle side use.

Workloads (decode projections of Llama-3.2-style decoders, the model family the
"Ember: packed Q8 decode" post measures):

* 1B: hidden 2048, 16 layers, Q 2048x2048, K/V 512x2048, O 2048x2048,
  gate/up 8192x2048 each, down 2048x8192, LM head 128256x2048.
* 3B: hidden 3072, 28 layers, Q/O 3072x3072, K/V 1024x3072, gate/up
  8192x3072 each, down 3072x8192, LM head 128256x3072.

Q/K/V are concatenated into one N = q + 2*kv projection and gate/up into one
N = 2*ffn projection, because each group reads one shared activation.

Distributions: weights fp32 N(0, 0.02), activations fp32 N(0, 1).

Generators: on the CPU, numpy's PCG64 (``numpy.random.default_rng(seed)``);
on a CUDA device, torch's Philox generator seeded with the same seed.  The two
streams differ; a test that compares the CUDA path with the oracle always
hands both sides the same tensor (generated once, copied to the other side).
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np

WEIGHT_STD = 0.02
ACT_STD = 1.0


@dataclass(frozen=True)
class Proj:
    name: str
    N: int
    K: int
    shares_input_with: str | None = None


@dataclass(frozen=True)
class StackShape:
    name: str
    hidden: int
    q_dim: int
    kv_dim: int
    ffn: int
    layers: int
    vocab: int

    def layer_projs(self):
        """The four GEMVs of one layer, with the shared groups concatenated."""
        h = self.hidden
        return [
            Proj("qkv", self.q_dim + 2 * self.kv_dim, h),
            Proj("o", h, self.q_dim),
            Proj("gate_up", 2 * self.ffn, h),
            Proj("down", h, self.ffn),
        ]

    def head(self) -> Proj:
        return Proj("lm_head", self.vocab, self.hidden)

    def weight_bytes(self) -> int:
        """Q8_0 bytes of the whole stack: 34 bytes per 32 weights."""
        tot = sum(p.N * p.K for p in self.layer_projs()) * self.layers
        tot += self.vocab * self.hidden
        return tot // 32 * 34


LLAMA_1B = StackShape("llama-3.2-1b", 2048, 2048, 512, 8192, 16, 128256)
LLAMA_3B = StackShape("llama-3.2-3b", 3072, 3072, 1024, 8192, 28, 128256)


def derive_seed(*parts) -> int:
    """Stable 63-bit seed from a tuple of labels (config, layer, projection)."""
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def normal_np(shape, std: float, seed: int) -> np.ndarray:
    """fp32 N(0, std^2) on the host, numpy PCG64."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def normal_torch(shape, std: float, seed: int, device):
    """fp32 N(0, std^2) as a torch tensor on ``device``.

    CPU tensors come from ``normal_np`` (PCG64); CUDA tensors from torch's
    CUDA generator seeded with ``seed``.
    """
    import torch

    dev = torch.device(device)
    if dev.type == "cpu":
        return torch.from_numpy(normal_np(shape, std, seed))
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def weights(N: int, K: int, seed: int, device="cpu"):
    return normal_torch((N, K), WEIGHT_STD, seed, device)


def activations(M: int, K: int, seed: int, device="cpu"):
    return normal_torch((M, K), ACT_STD, seed, device)
