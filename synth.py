"""Seeded synthetic inputs for VSA (Video Sparse Attention) workloads.

This module only draws numbers: it holds none of the attention method's
arithmetic, so both the CPU oracle and the CUDA path can take their inputs
from it without sharing any part of the computation.

Value recipe (a smooth spatio-temporal field plus noise, standing in for the
Q/K/V activations of a video DiT such as Wan2.1, which are not available):
for every tensor in {Q, K, V}, every batch row, head and channel, draw eight
frequency triples (a_j, b_j, c_j) ~ U[0, 0.8] and set

    x(t, h, w) = sum_j sin(a_j t + b_j h + c_j w) + N(0, 0.5^2) noise

at every token of the (T, H, W) latent grid, token n = (t*H + h)*W + w in
native raster order.  Values are produced in float32 and rounded to bfloat16
with round-to-nearest-even; every consumer gets the same bits.  The upstream
gradient dO is N(0, 1).  Gates (when used) are U[0, 1).

Seeds: numpy PCG64 seeded with base_seed XOR crc32("<config>/<tensor>").
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import numpy as np

BASE_SEED = 20250519  # fixed base seed for every workload


@dataclass(frozen=True)
class Workload:
    """One attention call: batch, heads, head dim, latent grid and Top-K."""

    name: str
    B: int
    heads: int
    d: int
    T: int
    H: int
    W: int
    topk: int

    @property
    def N(self) -> int:
        return self.T * self.H * self.W

    @property
    def Nc(self) -> int:
        return self.N // 64

    @property
    def BH(self) -> int:
        return self.B * self.heads

    @property
    def sparsity(self) -> float:
        return 1.0 - self.topk / self.Nc


# Attention-layer shapes used for parity and timing.  Grids are the latent
# (T, H, W) of each video; cubes are (4, 4, 4) = 64 tokens.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 64, 4, 8, 8, 2),
    "tiny_dense": Workload("tiny_dense", 1, 2, 64, 4, 8, 8, 4),
    "small": Workload("small", 1, 12, 128, 8, 16, 32, 16),
    "wan1.3b": Workload("wan1.3b", 1, 12, 128, 16, 32, 64, 154),
    "wan1.3b_k512": Workload("wan1.3b_k512", 1, 12, 128, 16, 32, 64, 512),
    "wan1.3b_k256": Workload("wan1.3b_k256", 1, 12, 128, 16, 32, 64, 256),
    "wan1.3b_k64": Workload("wan1.3b_k64", 1, 12, 128, 16, 32, 64, 64),
    "wan14b": Workload("wan14b", 1, 40, 128, 16, 32, 64, 154),
    "long": Workload("long", 1, 24, 128, 32, 48, 80, 192),
}


def seed_for(config: str, tensor: str, base: int = BASE_SEED) -> int:
    return (base ^ zlib.crc32(f"{config}/{tensor}".encode())) & 0xFFFFFFFF


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest bfloat16 (ties to even), returned as float32.

    Non-finite inputs are not expected here (the generator never makes them).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of bf16-exact float32 values, as uint16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def smooth_field(rng: np.random.Generator, B: int, heads: int, d: int,
                 T: int, H: int, W: int, nfreq: int = 8,
                 fmax: float = 0.8, noise_std: float = 0.5,
                 heads_subset=None) -> np.ndarray:
    """[B, len(heads), T*H*W, d] float32 (bf16-exact) smooth field plus noise.

    The frequencies are drawn for all heads first and the noise second, so
    that a head subset (``heads_subset``) yields exactly the rows of the full
    tensor for those heads.
    """
    freqs = rng.uniform(0.0, fmax, size=(B, heads, d, nfreq, 3))
    noise_state = rng.bit_generator.state
    hs = list(range(heads)) if heads_subset is None else list(heads_subset)
    N = T * H * W
    out = np.empty((B, len(hs), N, d), dtype=np.float32)
    t = np.arange(T, dtype=np.float64)
    h = np.arange(H, dtype=np.float64)
    w = np.arange(W, dtype=np.float64)
    for b in range(B):
        for oi, hd in enumerate(hs):
            f = freqs[b, hd]                                     # [d, j, 3]
            et = np.exp(1j * f[:, :, 0, None] * t)               # [d, j, T]
            eh = np.exp(1j * f[:, :, 1, None] * h)               # [d, j, H]
            ew = np.exp(1j * f[:, :, 2, None] * w)               # [d, j, W]
            eth = (et[:, :, :, None] * eh[:, :, None, :]).reshape(d, nfreq, T * H)
            # sum_j e^{i(a t + b h)} e^{i c w}, imaginary part -> [d, T*H, W]
            field = np.matmul(eth.transpose(0, 2, 1), ew).imag
            out[b, oi] = field.reshape(d, N).T
    # Noise: one stream per tensor, drawn head by head in a fixed order.
    nrng = np.random.Generator(np.random.PCG64())
    nrng.bit_generator.state = noise_state
    for b in range(B):
        for hd in range(heads):
            if hd in hs:
                out[b, hs.index(hd)] += nrng.normal(0.0, noise_std, size=(N, d)).astype(np.float32)
            else:
                nrng.normal(0.0, noise_std, size=(N, d))
    return round_to_bf16(out)


def make_qkv(wl: Workload, heads_subset=None, base: int = BASE_SEED):
    """Q, K, V as float32 bf16-exact arrays [B, heads, N, d] (native order)."""
    out = []
    for name in ("q", "k", "v"):
        rng = np.random.default_rng(seed_for(wl.name, name, base))
        out.append(smooth_field(rng, wl.B, wl.heads, wl.d, wl.T, wl.H, wl.W,
                                heads_subset=heads_subset))
    return tuple(out)


def make_dout(wl: Workload, heads_subset=None, base: int = BASE_SEED) -> np.ndarray:
    """Upstream gradient dO ~ N(0, 1), bf16-exact, [B, heads, N, d]."""
    rng = np.random.default_rng(seed_for(wl.name, "dout", base))
    full = rng.standard_normal(size=(wl.B, wl.heads, wl.N, wl.d), dtype=np.float32)
    if heads_subset is not None:
        full = full[:, list(heads_subset)]
    return round_to_bf16(full)


def make_gates(wl: Workload, heads_subset=None, base: int = BASE_SEED):
    """Coarse and fine gates U[0, 1), bf16-exact, [B, heads, N, d] each."""
    out = []
    for name in ("g_coarse", "g_fine"):
        rng = np.random.default_rng(seed_for(wl.name, name, base))
        g = rng.random(size=(wl.B, wl.heads, wl.N, wl.d), dtype=np.float32)
        if heads_subset is not None:
            g = g[:, list(heads_subset)]
        out.append(round_to_bf16(g))
    return tuple(out)


def make_random(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """Plain N(0, std^2) bf16-exact array, for unit cases."""
    rng = np.random.default_rng(seed)
    return round_to_bf16(rng.normal(0.0, std, size=shape).astype(np.float32))
