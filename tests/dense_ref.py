"""A second, independent statement of VSA for tiny inputs, used only to pin the
oracle: dense float64 torch tensors with an explicit token-level mask built
from the block index list, autograd for the backward pass.

Nothing here reorders tokens: cube ids are computed straight from the native
(t, h, w) coordinates, pooling is a one-hot matrix product and the fine stage is
a masked dense softmax.  It never touches the oracle's code, so agreement
between the two pins the oracle's permutation, pooling, coarse stage, fine
stage, combination and hand-derived backward.
"""
from __future__ import annotations

import numpy as np
import torch


def cube_ids(T: int, H: int, W: int, rank=None) -> np.ndarray:
    """Cube id of every native token n = (t*H + h)*W + w: cubes of (4, 4, 4)
    tokens in raster order over the ceil(T/4) x ceil(H/4) x ceil(W/4) cube
    grid (boundary cubes may be partial), relabelled by rank[] if given."""
    Hc, Wc = -(-H // 4), -(-W // 4)
    t, h, w = np.meshgrid(np.arange(T), np.arange(H), np.arange(W), indexing="ij")
    cid = (((t // 4) * Hc + h // 4) * Wc + w // 4).reshape(-1)
    return cid if rank is None else np.asarray(rank)[cid]


def dense_vsa(q, k, v, T, H, W, lut, scale, gc=None, gf=None, cnt=None, rank=None):
    """q, k, v: torch float64 [BH, N, d] native order; lut: int [BH, Nc, Kmax].

    Each cube's vector is the mean of the tokens that belong to it.
    Returns (out, O_f, O_c broadcast to tokens, coarse scores, lse), native order.
    """
    BH, N, d = q.shape
    cid = torch.as_tensor(cube_ids(T, H, W, rank), dtype=torch.long)
    Nc = (-(-T // 4)) * (-(-H // 4)) * (-(-W // 4))
    onehot = (cid[:, None] == torch.arange(Nc)[None, :]).to(torch.float64)  # [N, Nc]
    members = onehot.sum(0)[:, None]
    qc = onehot.T @ q / members
    kc = onehot.T @ k / members
    vc = onehot.T @ v / members
    sc = (qc @ kc.transpose(-1, -2)) * scale
    oc = torch.softmax(sc, dim=-1) @ vc                                  # [BH, Nc, d]
    lut = torch.as_tensor(np.asarray(lut), dtype=torch.long)
    allowed = torch.zeros(BH, Nc, Nc, dtype=torch.bool)
    for bh in range(BH):
        for a in range(Nc):
            n = lut.shape[-1] if cnt is None else int(cnt[bh][a])
            allowed[bh, a, lut[bh, a, :n]] = True
    mask = allowed[:, cid[:, None], cid[None, :]]                       # [BH, N, N]
    s = (q @ k.transpose(-1, -2)) * scale
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    of = torch.softmax(s, dim=-1) @ v
    ocb = oc[:, cid, :]
    a = torch.ones_like(q) if gc is None else gc
    b = torch.ones_like(q) if gf is None else gf
    out = a * ocb + b * of
    return out, of, ocb, sc, lse
