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

Seeds: every (batch row, head) of every tensor has its own numpy PCG64
stream, seeded with SeedSequence([base_seed XOR crc32("<config>/<tensor>"),
b, head]); the smooth field draws its frequencies first and its noise second.
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor
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
        """Cubes of (4, 4, 4) covering the grid (a side that is not a
        multiple of 4 ends in partial cubes)."""
        return ((self.T + 3) // 4) * ((self.H + 3) // 4) * ((self.W + 3) // 4)

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
    # Grids whose sides are not multiples of 4 (partial boundary cubes).
    "odd": Workload("odd", 1, 2, 64, 5, 6, 10, 3),
    "odd_small": Workload("odd_small", 1, 4, 128, 9, 14, 22, 12),
    # The Wan2.1 latent of an 832x480, 81-frame video after (1, 2, 2)
    # patchify: 21 x 30 x 52 = 32760 tokens, 6 x 8 x 13 = 624 cubes.
    "wan1.3b_latent": Workload("wan1.3b_latent", 1, 12, 128, 21, 30, 52, 187),
}


def seed_for(config: str, tensor: str, base: int = BASE_SEED) -> int:
    return (base ^ zlib.crc32(f"{config}/{tensor}".encode())) & 0xFFFFFFFF


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest bfloat16 (ties to even), returned as float32.

    Non-finite inputs are not expected here (the generator never makes them).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    # For finite x the sum stays below 2**32 (largest finite pattern 0xFF7FFFFF).
    u = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of bf16-exact float32 values, as uint16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _head_rng(seed: int, b: int, hd: int) -> np.random.Generator:
    """Independent PCG64 stream for one (batch row, head) of one tensor."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, b, hd])))


def _per_head(B: int, heads: int, heads_subset, N: int, d: int, fill) -> np.ndarray:
    """[B, len(hs), N, d] float32 with fill(b, head) -> [N, d] run on a thread
    pool (numpy releases the GIL in the bulk fills)."""
    hs = list(range(heads)) if heads_subset is None else list(heads_subset)
    out = np.empty((B, len(hs), N, d), dtype=np.float32)
    jobs = [(b, oi, hd) for b in range(B) for oi, hd in enumerate(hs)]

    def run(job):
        b, oi, hd = job
        out[b, oi] = fill(b, hd)

    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 1)) as ex:
        list(ex.map(run, jobs))
    return out


def smooth_field(seed: int, B: int, heads: int, d: int, T: int, H: int, W: int,
                 nfreq: int = 8, fmax: float = 0.8, noise_std: float = 0.5,
                 heads_subset=None) -> np.ndarray:
    """[B, len(heads), T*H*W, d] float32 (bf16-exact) smooth field plus noise.

    Each (batch row, head) draws its frequencies and then its noise from its
    own stream, so a head subset yields exactly those heads of the full tensor.
    """
    N = T * H * W
    t = np.arange(T, dtype=np.float64)
    h = np.arange(H, dtype=np.float64)
    w = np.arange(W, dtype=np.float64)

    def fill(b, hd):
        rng = _head_rng(seed, b, hd)
        f = rng.uniform(0.0, fmax, size=(d, nfreq, 3))
        # sin(A + C) = sin A cos C + cos A sin C with A = a t + b h and C = c w,
        # summed over j as one real product [T*H, 2j] x [2j, W] per channel.
        A = (f[:, :, 0, None, None] * t[:, None] + f[:, :, 1, None, None] * h[None, :]).reshape(d, nfreq, T * H)
        C = f[:, :, 2, None] * w                                  # [d, j, W]
        L = np.concatenate([np.sin(A), np.cos(A)], axis=1)        # [d, 2j, T*H]
        R = np.concatenate([np.cos(C), np.sin(C)], axis=1)        # [d, 2j, W]
        field = np.matmul(L.transpose(0, 2, 1), R).reshape(d, N).T
        noise = rng.standard_normal(size=(N, d), dtype=np.float32)
        return round_to_bf16(field.astype(np.float32) + np.float32(noise_std) * noise)

    return _per_head(B, heads, heads_subset, N, d, fill)


def make_qkv(wl: Workload, heads_subset=None, base: int = BASE_SEED):
    """Q, K, V as float32 bf16-exact arrays [B, heads, N, d] (native order)."""
    return tuple(smooth_field(seed_for(wl.name, name, base), wl.B, wl.heads, wl.d, wl.T, wl.H, wl.W,
                              heads_subset=heads_subset) for name in ("q", "k", "v"))


def make_dout(wl: Workload, heads_subset=None, base: int = BASE_SEED) -> np.ndarray:
    """Upstream gradient dO ~ N(0, 1), bf16-exact, [B, heads, N, d]."""
    seed = seed_for(wl.name, "dout", base)
    return _per_head(wl.B, wl.heads, heads_subset, wl.N, wl.d, lambda b, hd: round_to_bf16(
        _head_rng(seed, b, hd).standard_normal(size=(wl.N, wl.d), dtype=np.float32)))


def make_gates(wl: Workload, heads_subset=None, base: int = BASE_SEED):
    """Coarse and fine gates U[0, 1), bf16-exact, [B, heads, N, d] each."""
    out = []
    for name in ("g_coarse", "g_fine"):
        seed = seed_for(wl.name, name, base)
        out.append(_per_head(wl.B, wl.heads, heads_subset, wl.N, wl.d, lambda b, hd, seed=seed: round_to_bf16(
            _head_rng(seed, b, hd).random(size=(wl.N, wl.d), dtype=np.float32))))
    return tuple(out)


def make_random(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """Plain N(0, std^2) bf16-exact array, for unit cases."""
    rng = np.random.default_rng(seed)
    return round_to_bf16(rng.normal(0.0, std, size=shape).astype(np.float32))
