"""Pins for the CPU oracle, each against something other than the oracle itself:
brute force, closed forms, textbook special cases (dense SDPA), an independent
dense masked formulation with torch autograd, and finite differences.

Runs on the CPU only.
"""
import json
import os

import numpy as np
import pytest
import torch

import synth
from dense_ref import cube_ids, dense_vsa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

GRIDS = [(4, 8, 8), (8, 16, 32), (8, 12, 20), (4, 4, 4), (12, 4, 8)]


# ---------------------------------------------------------------------------
# 3D SFC reordering ("Pre-stage: 3D Space-Filling Curve (SFC) Token Reordering")

@pytest.mark.parametrize("grid", GRIDS)
def test_sfc_is_bijection_onto_contiguous_cubes(oracle_mod, grid):
    T, H, W = grid
    pos = oracle_mod.sfc_table(T, H, W)
    N = T * H * W
    assert sorted(pos.tolist()) == list(range(N))        # bijection
    # Every block of 64 consecutive reordered tokens is one 4x4x4 box.
    inv = np.empty(N, dtype=np.int64)
    inv[pos] = np.arange(N)
    t, h, w = inv // (H * W), (inv // W) % H, inv % W
    for c in range(N // 64):
        sl = slice(64 * c, 64 * c + 64)
        for axis in (t, h, w):
            vals = axis[sl]
            assert vals.max() - vals.min() == 3 and vals.min() % 4 == 0
        assert len(set(zip(t[sl], h[sl], w[sl]))) == 64


@pytest.mark.parametrize("grid", GRIDS)
def test_sfc_matches_reshape_transpose(oracle_mod, grid):
    """Cube-raster order equals the library reshape/transpose of the grid."""
    T, H, W = grid
    x = np.arange(T * H * W, dtype=np.float64).reshape(1, T * H * W, 1)
    y = oracle_mod.permute(x, T, H, W)
    ref = np.arange(T * H * W).reshape(T // 4, 4, H // 4, 4, W // 4, 4)
    ref = ref.transpose(0, 2, 4, 1, 3, 5).reshape(-1)
    np.testing.assert_array_equal(y.reshape(-1), ref)
    back = oracle_mod.permute(y, T, H, W, inverse=True)
    np.testing.assert_array_equal(back, x)


def test_sfc_golden_positions(oracle_mod):
    with open(os.path.join(GOLDEN, "sfc_positions.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        T, H, W = case["grid"]
        for (t, h, w), p in case["positions"]:
            assert oracle_mod._load().orc_sfc_position(t, h, w, T, H, W, None) == p


# ---------------------------------------------------------------------------
# Cube mean-pool ("Stage 1: Coarse Selection")

def test_pool_bruteforce_on_native_boxes(oracle_mod):
    T, H, W, d = 8, 12, 20, 5
    x = synth.make_random((2, T * H * W, d), seed=11)
    xc = oracle_mod.pool(oracle_mod.permute(x, T, H, W))
    xn = x.astype(np.float64).reshape(2, T, H, W, d)
    c = 0
    for ct in range(T // 4):
        for ch in range(H // 4):
            for cw in range(W // 4):
                box = xn[:, 4 * ct:4 * ct + 4, 4 * ch:4 * ch + 4, 4 * cw:4 * cw + 4]
                np.testing.assert_allclose(xc[:, c], box.reshape(2, 64, d).mean(1), rtol=0, atol=1e-13)
                c += 1


def test_pool_constant_cube(oracle_mod):
    T, H, W, d = 4, 8, 8, 3
    vals = np.array([1.5, -2.25, 7.0])
    xp = np.tile(vals, (T * H * W, 1))[None]
    assert np.array_equal(oracle_mod.pool(xp)[0], np.tile(vals, (4, 1)))
    assert np.array_equal(oracle_mod.pool(np.zeros((1, T * H * W, d))), np.zeros((1, 4, d)))


# ---------------------------------------------------------------------------
# Coarse stage and Top-K ("Stage 1", "Generating Sparsity Patterns")

def test_coarse_equals_sdpa_on_pooled(oracle_mod):
    rng = np.random.default_rng(3)
    qc, kc, vc = (rng.normal(size=(3, 20, 16)) for _ in range(3))
    scale = 0.3
    scores, oc, lse = oracle_mod.coarse(qc, kc, vc, scale)
    t = [torch.tensor(a) for a in (qc, kc, vc)]
    ref = torch.nn.functional.scaled_dot_product_attention(*t, scale=scale).numpy()
    np.testing.assert_allclose(oc, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(scores, scale * qc @ kc.transpose(0, 2, 1), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.tensor(scores), -1).numpy(), rtol=1e-13)


@pytest.mark.parametrize("grid", [(8, 8, 8), (6, 7, 5)])
def test_constant_cubes_tie_fine_to_coarse(oracle_mod, grid):
    """Every cube constant, all cubes selected: the fine stage's 64 (or, in a
    partial cube, fewer) copies of each key act as one key weighted by its
    token count, so O_f = sum_j n_j e^{s q.k_j} v_j / sum_j n_j e^{s q.k_j},
    LSE_f = log sum_j n_j e^{s q.k_j}, and O_c is the same sum without n_j.
    With full cubes O_f equals O_c: the pool, the coarse scale and the fine
    stage agree.  Closed form computed here from the cube values alone."""
    T, H, W = grid
    BH, d, scale = 2, 16, 0.3
    Tc, Hc, Wc = (T + 3) // 4, (H + 3) // 4, (W + 3) // 4
    Nc = Tc * Hc * Wc
    t, h, w = np.meshgrid(np.arange(T), np.arange(H), np.arange(W), indexing="ij")
    cube = ((t // 4 * Hc + h // 4) * Wc + w // 4).reshape(-1)       # raster cube of each native token
    ntok = np.bincount(cube, minlength=Nc).astype(np.float64)
    rng = np.random.default_rng(17)
    qv, kv, vv = (rng.normal(size=(BH, Nc, d)) for _ in range(3))
    q, k, v = (a[:, cube] for a in (qv, kv, vv))
    r = oracle_mod.forward(q, k, v, T, H, W, Nc, scale)
    e = np.exp(scale * np.einsum("bid,bjd->bij", qv, kv))
    oc = np.einsum("bij,bjd->bid", e, vv) / e.sum(-1, keepdims=True)
    en = e * ntok
    of = np.einsum("bij,bjd->bid", en, vv) / en.sum(-1, keepdims=True)
    lse = np.log(en.sum(-1))
    pos = oracle_mod.sfc_table(T, H, W)
    np.testing.assert_allclose(r["oc"], oc, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["of"][:, pos], of[:, cube], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(r["lse"][:, pos], lse[:, cube], rtol=1e-12)
    np.testing.assert_allclose(r["out"], (oc + of)[:, cube], rtol=1e-11, atol=1e-11)
    if T % 4 == 0 and H % 4 == 0 and W % 4 == 0:
        np.testing.assert_allclose(of, oc, rtol=1e-12, atol=1e-12)


def _bruteforce_topk(scores, K):
    Nc = scores.shape[-1]
    out = np.empty(scores.shape[:-1] + (K,), dtype=np.int64)
    for r in np.ndindex(scores.shape[:-1]):
        order = np.lexsort((np.arange(Nc), -scores[r]))   # score desc, id asc
        out[r] = order[:K]
    return out


@pytest.mark.parametrize("K", [1, 3, 16, 64])
def test_topk_bruteforce_random(oracle_mod, K):
    rng = np.random.default_rng(K)
    scores = rng.normal(size=(2, 64, 64))
    np.testing.assert_array_equal(oracle_mod.topk(scores, K), _bruteforce_topk(scores, K))


def test_topk_ties_go_to_lower_id(oracle_mod):
    rng = np.random.default_rng(7)
    scores = rng.integers(0, 4, size=(3, 40, 40)).astype(np.float64)   # many ties
    for K in (1, 5, 13, 40):
        np.testing.assert_array_equal(oracle_mod.topk(scores, K), _bruteforce_topk(scores, K))
    flat = np.zeros((1, 1, 10))
    np.testing.assert_array_equal(oracle_mod.topk(flat, 4)[0, 0], [0, 1, 2, 3])


def test_topk_golden(oracle_mod):
    with open(os.path.join(GOLDEN, "topk_cases.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        s = np.array(case["scores"], dtype=np.float64)[None, None]
        got = oracle_mod.topk(s, case["K"])[0, 0].tolist()
        assert got == case["expected"], case["note"]


# ---------------------------------------------------------------------------
# Fine stage ("Stage 2: Fine Computation", "Sparse Traversal")

def test_fine_all_cubes_is_dense_sdpa(oracle_mod):
    """K = all cubes: nothing is skipped, so the fine stage is plain SDPA."""
    BH, N, d = 2, 256, 64
    q, k, v = (synth.make_random((BH, N, d), seed=s) for s in (1, 2, 3))
    Nc = N // 64
    idx = np.tile(np.arange(Nc, dtype=np.int32), (BH, Nc, 1))[:, :, ::-1].copy()
    cnt = np.full((BH, Nc), Nc, dtype=np.int32)
    of, lse = oracle_mod.fine_fwd(q, k, v, idx, cnt, d ** -0.5)
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv).numpy()
    np.testing.assert_allclose(of, ref, rtol=1e-11, atol=1e-11)
    ref_lse = torch.logsumexp(tq @ tk.transpose(-1, -2) * d ** -0.5, -1).numpy()
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12)


def test_fine_single_cube_is_local_sdpa(oracle_mod):
    BH, N, d = 1, 512, 32
    q, k, v = (synth.make_random((BH, N, d), seed=s) for s in (4, 5, 6))
    Nc = N // 64
    own = np.arange(Nc, dtype=np.int32).reshape(1, Nc, 1)
    of, _ = oracle_mod.fine_fwd(q, k, v, own, np.ones((1, Nc), np.int32), 0.2)
    t = [torch.tensor(a, dtype=torch.float64).reshape(Nc, 64, d) for a in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(*t, scale=0.2).reshape(1, N, d).numpy()
    np.testing.assert_allclose(of, ref, rtol=1e-11, atol=1e-11)


def test_fine_zero_query_closed_form(oracle_mod):
    """Q = 0: every selected key has weight 1/(64 K); LSE = log(64 K)."""
    BH, N, d, K = 1, 512, 16, 3
    rng = np.random.default_rng(9)
    k, v = rng.normal(size=(2, BH, N, d))
    q = np.zeros((BH, N, d))
    idx = np.stack([rng.permutation(8)[:K] for _ in range(8)])[None].astype(np.int32)
    of, lse = oracle_mod.fine_fwd(q, k, v, idx, np.full((1, 8), K, np.int32), 0.5)
    for a in range(8):
        keys = np.concatenate([np.arange(64 * c, 64 * c + 64) for c in idx[0, a]])
        np.testing.assert_allclose(of[0, 64 * a:64 * a + 64], np.tile(v[0, keys].mean(0), (64, 1)), atol=1e-13)
    np.testing.assert_allclose(lse, np.log(64 * K), rtol=1e-14)


def test_fine_empty_and_ragged_counts(oracle_mod):
    BH, N, d = 1, 256, 8
    q, k, v = (synth.make_random((BH, N, d), seed=s) for s in (7, 8, 9))
    idx = np.array([[[2, 0, 1], [1, 3, 0], [0, 0, 0], [3, 2, 1]]], dtype=np.int32)
    cnt = np.array([[3, 1, 0, 2]], dtype=np.int32)
    of, lse = oracle_mod.fine_fwd(q, k, v, idx, cnt, 0.35)
    assert np.all(of[0, 128:192] == 0) and np.all(np.isneginf(lse[0, 128:192]))
    for a, n in enumerate(cnt[0]):
        if n == 0:
            continue
        keys = np.concatenate([np.arange(64 * c, 64 * c + 64) for c in idx[0, a, :n]])
        s = q[0, 64 * a:64 * a + 64].astype(np.float64) @ k[0, keys].T.astype(np.float64) * 0.35
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        np.testing.assert_allclose(of[0, 64 * a:64 * a + 64], p @ v[0, keys], atol=1e-12)


# ---------------------------------------------------------------------------
# Whole forward and backward against the independent dense formulation

def _tiny_inputs(wl, gates):
    q, k, v = synth.make_qkv(wl)
    sh = (wl.BH, wl.N, wl.d)
    q, k, v = (a.reshape(sh) for a in (q, k, v))
    gc = gf = None
    if gates:
        gc, gf = (a.reshape(sh) for a in synth.make_gates(wl))
    dout = synth.make_dout(wl).reshape(sh)
    return q, k, v, gc, gf, dout


def _t(a):
    return None if a is None else torch.tensor(a, dtype=torch.float64)


@pytest.mark.parametrize("name,gates", [("tiny", True), ("tiny", False), ("tiny_dense", True)])
def test_forward_matches_dense_masked(oracle_mod, name, gates):
    wl = synth.WORKLOADS[name]
    q, k, v, gc, gf, _ = _tiny_inputs(wl, gates)
    scale = wl.d ** -0.5
    r = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, scale, gc=gc, gf=gf)
    out, of, ocb, sc, lse = dense_vsa(_t(q), _t(k), _t(v), wl.T, wl.H, wl.W, r["idx"], scale,
                                      gc=_t(gc), gf=_t(gf))
    np.testing.assert_allclose(r["scores"], sc.numpy(), rtol=1e-12, atol=1e-10)
    # Selection: the dense formulation's own torch.topk gives the same sets.
    tk_idx = torch.topk(sc, wl.topk, dim=-1).indices.numpy()
    assert np.array_equal(np.sort(tk_idx, -1), np.sort(r["idx"], -1))
    np.testing.assert_allclose(r["out"], out.numpy(), rtol=1e-10, atol=1e-10)
    pos = oracle_mod.sfc_table(wl.T, wl.H, wl.W)
    np.testing.assert_allclose(r["of"][:, pos], of.numpy(), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(r["lse"][:, pos], lse.numpy(), rtol=1e-12)


@pytest.mark.parametrize("gates", [True, False])
def test_backward_matches_autograd(oracle_mod, gates):
    wl = synth.WORKLOADS["tiny"]
    q, k, v, gc, gf, dout = _tiny_inputs(wl, gates)
    scale = wl.d ** -0.5
    r = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, scale, gc=gc, gf=gf)
    g = oracle_mod.backward(q, k, v, dout, r["idx"], wl.T, wl.H, wl.W, scale, gc=gc, gf=gf)
    leaves = {n: torch.tensor(a, dtype=torch.float64, requires_grad=True)
              for n, a in (("q", q), ("k", k), ("v", v), ("gc", gc), ("gf", gf)) if a is not None}
    out, *_ = dense_vsa(leaves["q"], leaves["k"], leaves["v"], wl.T, wl.H, wl.W, r["idx"], scale,
                        gc=leaves.get("gc"), gf=leaves.get("gf"))
    (out * torch.tensor(dout, dtype=torch.float64)).sum().backward()
    for n, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("gc", "dgc"), ("gf", "dgf")):
        if n in leaves:
            np.testing.assert_allclose(g[key], leaves[n].grad.numpy(), rtol=1e-9, atol=1e-9,
                                       err_msg=key)


def test_backward_finite_differences(oracle_mod):
    """fp64 central differences of L = sum(out * dO) with the index list frozen."""
    wl = synth.WORKLOADS["tiny"]
    q, k, v, gc, gf, dout = (None if a is None else a.astype(np.float64)
                             for a in _tiny_inputs(wl, True))
    # Shrink Q and K so the softmax is not saturated and every term matters.
    q, k = q * 0.1, k * 0.1
    scale = wl.d ** -0.5
    r = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, scale, gc=gc, gf=gf)
    lut = r["idx"]
    g = oracle_mod.backward(q, k, v, dout, lut, wl.T, wl.H, wl.W, scale, gc=gc, gf=gf)
    inputs = dict(q=q, k=k, v=v, gc=gc, gf=gf)
    grads = dict(q=g["dq"], k=g["dk"], v=g["dv"], gc=g["dgc"], gf=g["dgf"])
    rng = np.random.default_rng(0)
    h = 1e-5

    def loss(ins):
        o = oracle_mod.forward(ins["q"], ins["k"], ins["v"], wl.T, wl.H, wl.W, wl.topk, scale,
                               gc=ins["gc"], gf=ins["gf"], lut=lut, want_scores=False)
        return float((o["out"] * dout).sum())

    for name in inputs:
        for _ in range(12):
            e = tuple(int(rng.integers(0, s)) for s in inputs[name].shape)
            ins = {n: a.copy() for n, a in inputs.items()}
            ins[name][e] += h
            lp = loss(ins)
            ins[name][e] -= 2 * h
            lm = loss(ins)
            fd = (lp - lm) / (2 * h)
            an = grads[name][e]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, e, fd, an)


def test_gate_special_cases(oracle_mod):
    """g_c = 0, g_f = 1 gives the fine output alone; g_c = 1, g_f = 0 the coarse one."""
    wl = synth.WORKLOADS["tiny"]
    q, k, v, *_ = _tiny_inputs(wl, False)
    zeros, ones = np.zeros_like(q), np.ones_like(q)
    pos = oracle_mod.sfc_table(wl.T, wl.H, wl.W)
    r = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=zeros, gf=ones)
    np.testing.assert_array_equal(r["out"], r["of"][:, pos])
    r2 = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=ones, gf=zeros)
    cid = cube_ids(wl.T, wl.H, wl.W)
    np.testing.assert_array_equal(r2["out"], r2["oc"][:, cid])


def test_dense_k_equals_sdpa_end_to_end(oracle_mod):
    """K = Nc with g_c = 0: VSA is exactly dense attention in native order."""
    wl = synth.WORKLOADS["tiny_dense"]
    q, k, v, *_ = _tiny_inputs(wl, False)
    r = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=np.zeros_like(q))
    t = [torch.tensor(a, dtype=torch.float64) for a in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(*t).numpy()
    np.testing.assert_allclose(r["out"], ref, rtol=1e-10, atol=1e-10)


def test_small_forward_one_head_matches_dense(oracle_mod):
    """A mid-size case (4096 tokens, 64 cubes, K=16) spanning many cubes."""
    wl = synth.WORKLOADS["small"]
    q, k, v = (a.reshape(1, wl.N, wl.d) for a in synth.make_qkv(wl, heads_subset=[3]))
    scale = wl.d ** -0.5
    r = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, scale)
    out, *_ = dense_vsa(_t(q), _t(k), _t(v), wl.T, wl.H, wl.W, r["idx"], scale)
    np.testing.assert_allclose(r["out"], out.numpy(), rtol=1e-10, atol=1e-10)


def test_head_subset_generator_matches_full(oracle_mod):
    """Heads are independent: the oracle on a generated head subset equals the
    same heads of a full run (the basis of sampled checks at full size)."""
    wl = synth.WORKLOADS["small"]
    full = synth.make_qkv(wl)
    sub = synth.make_qkv(wl, heads_subset=[0, 7])
    for f, s in zip(full, sub):
        np.testing.assert_array_equal(f[:, [0, 7]], s)


def test_sampled_backward_functions_match_full(oracle_mod):
    """The sampled dQ-row and dK/dV-key-cube functions (used at full size)
    reproduce the full fine backward, which autograd pins above."""
    wl = synth.WORKLOADS["small"]
    q, k, v = (a.reshape(1, wl.N, wl.d) for a in synth.make_qkv(wl, heads_subset=[2]))
    pos = oracle_mod.sfc_table(wl.T, wl.H, wl.W)
    qp, kp, vp = (oracle_mod.permute(a, wl.T, wl.H, wl.W) for a in (q, k, v))
    dof = synth.make_random((1, wl.N, wl.d), seed=5)
    r = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk)
    idx = r["idx"]
    cnt = np.full(idx.shape[:-1], wl.topk, np.int32)
    scale = wl.d ** -0.5
    dq, dk, dv = oracle_mod.fine_bwd(qp, kp, vp, dof, idx, cnt, scale)
    rows = np.array([0, 5, 64, 1000, wl.N - 1])
    np.testing.assert_allclose(oracle_mod.fine_bwd_query_rows(qp, kp, vp, dof, idx, cnt, scale, rows),
                               dq[0, rows], rtol=1e-10, atol=1e-12)
    for c in (0, 17, wl.Nc - 1):
        sk, sv = oracle_mod.fine_bwd_key_cube(qp, kp, vp, dof, idx, cnt, scale, 0, c)
        np.testing.assert_allclose(sk, dk[0, 64 * c:64 * c + 64], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(sv, dv[0, 64 * c:64 * c + 64], rtol=1e-10, atol=1e-12)
    assert pos.size == wl.N


@pytest.mark.parametrize("curve", ["raster", "hilbert"])
def test_sampled_forward_rows_match_full_and_dense(oracle_mod, curve):
    """The sampled fine-forward function (the checker of every full-size
    forward comparison) against the full fine forward and against the dense
    masked torch formulation, on a grid with partial cubes (padding slots
    masked through slot_ok) and ragged counts, empty rows included."""
    wl = synth.WORKLOADS["odd_small"]                      # 9 x 14 x 22: every side ends in a partial cube
    q, k, v = (a.reshape(1, wl.N, wl.d)[:, :, :32] for a in synth.make_qkv(wl, heads_subset=[1]))
    T, H, W = wl.T, wl.H, wl.W
    rank = None if curve == "raster" else oracle_mod.cube_rank(*oracle_mod.cube_grid(T, H, W), curve)
    qp, kp, vp = (oracle_mod.permute(a, T, H, W, curve=curve) for a in (q, k, v))
    slot_ok, _ = oracle_mod.cube_slots(T, H, W, curve)
    Nc = oracle_mod.num_cubes(T, H, W)
    rng = np.random.default_rng(17)
    kmax = 9
    idx = np.stack([rng.permutation(Nc)[:kmax] for _ in range(Nc)])[None].astype(np.int32)
    cnt = rng.integers(0, kmax + 1, size=(1, Nc)).astype(np.int32)
    cnt[0, 3] = 0                                          # an empty list
    scale = 32 ** -0.5
    of, lse = oracle_mod.fine_fwd(qp, kp, vp, idx, cnt, scale, slot_ok=slot_ok)
    rows = np.unique(np.r_[0, 63, 64 * 3 + 5, rng.choice(64 * Nc, 40, replace=False), 64 * Nc - 1])
    ro, rl = oracle_mod.fine_fwd_rows(qp, kp, vp, idx, cnt, scale, rows, slot_ok=slot_ok)
    np.testing.assert_allclose(ro, of[0, rows], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(rl), np.isneginf(lse[0, rows]))
    fin = ~np.isneginf(rl)
    np.testing.assert_allclose(rl[fin], lse[0, rows][fin], rtol=1e-12, atol=1e-12)
    assert np.all(ro[~fin] == 0)
    # dense masked formulation (native order, cube ids from the coordinates)
    _, dof_, _, _, dlse = dense_vsa(_t(q), _t(k), _t(v), T, H, W, idx, scale, cnt=cnt, rank=rank)
    pos = oracle_mod.sfc_table(T, H, W, curve)
    native_of = np.full(64 * Nc, -1, np.int64)
    native_of[pos] = np.arange(wl.N)
    real = rows[slot_ok[rows] == 1]
    sel = np.searchsorted(rows, real)
    nat = native_of[real]
    np.testing.assert_allclose(ro[sel][fin[sel]], dof_.numpy()[0, nat][fin[sel]], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(rl[sel][fin[sel]], dlse.numpy()[0, nat][fin[sel]], rtol=1e-12)
    assert fin.sum() > 10 and (~fin).sum() >= 1


# ---------------------------------------------------------------- index-list conversions
def test_mask_to_lut_matches_nonzero(oracle_mod):
    """Block matrix -> list: the ascending nonzero columns of each row (brute
    force with numpy), -1 after the count; overflow keeps the lowest ids."""
    rng = np.random.default_rng(21)
    for Nc, density, kmax in ((8, 0.3, 8), (40, 0.5, 40), (40, 0.5, 12), (70, 0.05, 9)):
        m = rng.random((3, Nc, Nc)) < density
        idx, cnt, ovf = oracle_mod.mask_to_lut(m, kmax)
        any_over = False
        for r in range(3 * Nc):
            cols = np.flatnonzero(m.reshape(-1, Nc)[r])
            any_over |= cols.size > kmax
            keep = cols[:kmax]
            assert cnt.reshape(-1)[r] == keep.size
            row = idx.reshape(-1, kmax)[r]
            assert np.array_equal(row[:keep.size], keep)
            assert np.all(row[keep.size:] == -1)
        assert ovf == any_over
    full, cnt, _ = oracle_mod.mask_to_lut(np.ones((1, 5, 5)), 5)
    assert np.array_equal(full[0], np.tile(np.arange(5), (5, 1))) and np.all(cnt == 5)
    empty, cnt, _ = oracle_mod.mask_to_lut(np.zeros((1, 5, 5)), 3)
    assert np.all(empty == -1) and np.all(cnt == 0)


def test_lut_add_neighbors_brute_force(oracle_mod):
    """List united with the radius-r neighbourhood, against explicit cube
    coordinates; an interior cube gains (2r+1)^3 cubes, a corner (r+1)^3."""
    rng = np.random.default_rng(22)
    T, H, W = 12, 16, 20
    Tc, Hc, Wc = T // 4, H // 4, W // 4
    Nc = Tc * Hc * Wc
    coords = np.array([(t, h, w) for t in range(Tc) for h in range(Hc) for w in range(Wc)])
    K = 6
    idx = np.stack([np.stack([rng.permutation(Nc)[:K] for _ in range(Nc)]) for _ in range(2)]).astype(np.int32)
    cnt = rng.integers(0, K + 1, size=(2, Nc)).astype(np.int32)
    for radius in (0, 1, 2):
        kout = K + (2 * radius + 1) ** 3
        out, ocnt, ovf = oracle_mod.lut_add_neighbors(idx, cnt, T, H, W, radius, kout)
        assert not ovf
        for h in range(2):
            for q in range(Nc):
                near = np.flatnonzero(np.abs(coords - coords[q]).max(axis=1) <= radius)
                want = np.union1d(near, idx[h, q, :cnt[h, q]])
                assert ocnt[h, q] == want.size
                assert np.array_equal(out[h, q, :want.size], want)
                assert np.all(out[h, q, want.size:] == -1)
    empty = np.full((1, Nc, 1), -1, np.int32)
    out, ocnt, _ = oracle_mod.lut_add_neighbors(empty, np.zeros((1, Nc), np.int32), T, H, W, 1, 27)
    interior = (1 * Hc + 1) * Wc + 1
    assert ocnt[0, interior] == 27 and ocnt[0, 0] == 8


# ---------------------------------------------------------------- Hilbert cube order
# The curve of Skilling's construction ("Programming the Hilbert curve", 2004)
# is pinned by the properties that define a Hilbert curve, not by retyping it:
# every cell visited once, unit steps between consecutive cells, and the
# recursive structure (each aligned run of 8^k indices fills one aligned
# 2^k cube), starting at the origin.
@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_hilbert_curve_is_continuous_and_nested(oracle_mod, b):
    pts = np.array([oracle_mod.hilbert_point(h, b) for h in range(8 ** b)], dtype=np.int64)
    assert len({tuple(p) for p in pts}) == 8 ** b and pts.max() == 2 ** b - 1
    assert np.all(np.abs(np.diff(pts, axis=0)).sum(1) == 1)
    assert tuple(pts[0]) == (0, 0, 0)
    for k in range(1, b):
        blk = pts.reshape(-1, 8 ** k, 3)
        lo, hi = blk.min(1), blk.max(1)
        assert np.all(hi - lo == 2 ** k - 1) and np.all(lo % 2 ** k == 0)


@pytest.mark.parametrize("grid", [(1, 1, 1), (1, 2, 2), (2, 4, 8), (3, 5, 7), (4, 4, 4)])
def test_cube_rank_follows_the_curve(oracle_mod, grid):
    Tc, Hc, Wc = grid
    rank = oracle_mod.cube_rank(Tc, Hc, Wc, "hilbert")
    Nc = Tc * Hc * Wc
    assert sorted(rank.tolist()) == list(range(Nc))
    assert np.array_equal(oracle_mod.cube_rank(Tc, Hc, Wc, "raster"), np.arange(Nc))
    # positions in curve order -> grid cells; brute force over the enclosing curve
    b = max(int(np.ceil(np.log2(max(grid)))), 0)
    inside = [p for p in (oracle_mod.hilbert_point(h, b) for h in range(8 ** b))
              if p[0] < Tc and p[1] < Hc and p[2] < Wc]
    order = np.argsort(rank)
    cells = [((r // (Hc * Wc)), (r // Wc) % Hc, r % Wc) for r in order]
    assert cells == inside
    if grid == (4, 4, 4):   # a full power-of-two grid: consecutive cubes are face neighbours
        c = np.array(cells)
        assert np.all(np.abs(np.diff(c, axis=0)).sum(1) == 1)


def test_forward_backward_invariant_to_cube_order(oracle_mod):
    """The cube order only relabels cubes: native-order outputs and gradients
    are the same for raster and Hilbert order (no score ties in this data),
    and the selected cubes are the same grid cells."""
    wl = synth.Workload("ord", 1, 2, 64, 8, 8, 16, 5)   # cube grid (2, 2, 4)
    q, k, v = synth.make_qkv(wl)
    gc, gf = synth.make_gates(wl)
    dout = synth.make_dout(wl)
    ra = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=gc, gf=gf)
    hi = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=gc, gf=gf, curve="hilbert")
    np.testing.assert_allclose(hi["out"], ra["out"], rtol=0, atol=1e-12)
    rank = oracle_mod.cube_rank(2, 2, 4, "hilbert")
    order = np.argsort(rank)                       # position -> raster cube
    sets_h = np.sort(order[hi["idx"]], axis=-1)[..., rank, :]   # per raster query cube
    np.testing.assert_array_equal(sets_h, np.sort(ra["idx"], axis=-1))
    ga = oracle_mod.backward(q, k, v, dout, ra["idx"], wl.T, wl.H, wl.W, gc=gc, gf=gf)
    gh = oracle_mod.backward(q, k, v, dout, hi["idx"], wl.T, wl.H, wl.W, gc=gc, gf=gf, curve="hilbert")
    for n in ("dq", "dk", "dv", "dgc", "dgf"):
        np.testing.assert_allclose(gh[n], ga[n], rtol=0, atol=1e-12)


def test_add_neighbors_is_order_independent(oracle_mod):
    """Neighbourhoods are grid cells: with Hilbert ids the lists map back to
    the raster-order result."""
    T, H, W = 12, 8, 20        # cube grid (3, 2, 5)
    Tc, Hc, Wc = 3, 2, 5
    Nc = Tc * Hc * Wc
    rank = oracle_mod.cube_rank(Tc, Hc, Wc, "hilbert")
    order = np.argsort(rank)
    rng = np.random.default_rng(3)
    idx_r = np.stack([rng.permutation(Nc)[:4] for _ in range(Nc)]).astype(np.int32)[None]
    out_r, cnt_r, _ = oracle_mod.lut_add_neighbors(idx_r, None, T, H, W, 1, Nc)
    idx_h = rank[idx_r][:, order]            # relabel entries and reorder rows by position
    out_h, cnt_h, _ = oracle_mod.lut_add_neighbors(idx_h, None, T, H, W, 1, Nc, curve="hilbert")
    np.testing.assert_array_equal(cnt_h[:, rank], cnt_r)
    for r in range(Nc):
        got = np.sort(order[out_h[0, rank[r], :cnt_h[0, rank[r]]]])
        np.testing.assert_array_equal(got, out_r[0, r, :cnt_r[0, r]])


# ---------------------------------------------------------------- grids not divisible by 4
# Reading: a side that is not a multiple of 4 ends in partial cubes; padding
# slots are zero in the reordered tensors, left out of the cube means, never
# attended to and never written back.  The dense formulation needs no padding
# at all (cube ids straight from the coordinates, means over cube members), so
# agreement pins the oracle's padded reordering, pooling and masking.
@pytest.mark.parametrize("curve", ["raster", "hilbert"])
@pytest.mark.parametrize("gates", [True, False])
def test_padded_grid_matches_dense(oracle_mod, curve, gates):
    wl = synth.WORKLOADS["odd"]
    q, k, v, gc, gf, dout = _tiny_inputs(wl, gates)
    scale = wl.d ** -0.5
    r = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, scale, gc=gc, gf=gf, curve=curve)
    rank = None if curve == "raster" else oracle_mod.cube_rank(*oracle_mod.cube_grid(wl.T, wl.H, wl.W), curve)
    out, of, ocb, sc, lse = dense_vsa(_t(q), _t(k), _t(v), wl.T, wl.H, wl.W, r["idx"], scale,
                                      gc=_t(gc), gf=_t(gf), rank=rank)
    np.testing.assert_allclose(r["scores"], sc.numpy(), rtol=1e-12, atol=1e-10)
    tk_idx = torch.topk(sc, wl.topk, dim=-1).indices.numpy()
    assert np.array_equal(np.sort(tk_idx, -1), np.sort(r["idx"], -1))
    np.testing.assert_allclose(r["out"], out.numpy(), rtol=1e-10, atol=1e-10)
    pos = oracle_mod.sfc_table(wl.T, wl.H, wl.W, curve)
    np.testing.assert_allclose(r["of"][:, pos], of.numpy(), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(r["lse"][:, pos], lse.numpy(), rtol=1e-12)
    # backward against autograd of the dense formulation
    g = oracle_mod.backward(q, k, v, dout, r["idx"], wl.T, wl.H, wl.W, scale, gc=gc, gf=gf, curve=curve)
    leaves = {n: torch.tensor(a, dtype=torch.float64, requires_grad=True)
              for n, a in (("q", q), ("k", k), ("v", v), ("gc", gc), ("gf", gf)) if a is not None}
    o2, *_ = dense_vsa(leaves["q"], leaves["k"], leaves["v"], wl.T, wl.H, wl.W, r["idx"], scale,
                       gc=leaves.get("gc"), gf=leaves.get("gf"), rank=rank)
    (o2 * torch.tensor(dout, dtype=torch.float64)).sum().backward()
    for n, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("gc", "dgc"), ("gf", "dgf")):
        if n in leaves:
            np.testing.assert_allclose(g[key], leaves[n].grad.numpy(), rtol=1e-9, atol=1e-9, err_msg=key)


# ---------------------------------------------------------------- adjacency-forced selection
# [AMD] "Comparison with Jenga": the block selection as the union of an
# importance mask (the Top-K) and an adjacency mask.  The expected lists are
# rebuilt here from torch.topk on the dense coarse scores and from the cube
# coordinates alone, and the whole forward and backward are checked against
# the dense masked formulation with those lists.
@pytest.mark.parametrize("curve,radius", [("raster", 1), ("hilbert", 1), ("raster", 0), ("hilbert", 2)])
def test_adjacency_selection_matches_dense(oracle_mod, curve, radius):
    wl = synth.WORKLOADS["odd"]                          # 5 x 6 x 10: partial cubes on every side
    q, k, v, gc, gf, dout = _tiny_inputs(wl, True)
    T, H, W = wl.T, wl.H, wl.W
    Tc, Hc, Wc = oracle_mod.cube_grid(T, H, W)
    Nc = Tc * Hc * Wc
    scale = wl.d ** -0.5
    rank = None if curve == "raster" else oracle_mod.cube_rank(Tc, Hc, Wc, curve)
    r = oracle_mod.forward(q, k, v, T, H, W, wl.topk, scale, gc=gc, gf=gf, curve=curve, radius=radius)
    kmax = oracle_mod.list_width(wl.topk, radius, Nc)
    assert r["idx"].shape == (wl.BH, Nc, kmax)
    # the expected selection, from the dense scores and the coordinates
    *_, sc, _ = dense_vsa(_t(q), _t(k), _t(v), T, H, W, np.zeros((wl.BH, Nc, 1), np.int64), scale, rank=rank)
    top = torch.topk(sc, wl.topk, dim=-1).indices.numpy()
    pos = np.arange(Nc) if rank is None else np.asarray(rank)          # raster id -> position
    coord = np.stack(np.unravel_index(np.arange(Nc), (Tc, Hc, Wc)), 1)  # raster id -> (t, h, w)
    exp_idx = np.full((wl.BH, Nc, kmax), -1, np.int32)
    exp_cnt = np.zeros((wl.BH, Nc), np.int32)
    for bh in range(wl.BH):
        for qpos in range(Nc):
            qr = int(np.flatnonzero(pos == qpos)[0])
            near = pos[np.flatnonzero(np.abs(coord - coord[qr]).max(1) <= radius)]
            sel = sorted(set(top[bh, qpos].tolist()) | set(near.tolist()))
            exp_cnt[bh, qpos] = len(sel)
            exp_idx[bh, qpos, :len(sel)] = sel
    np.testing.assert_array_equal(r["cnt"], exp_cnt)
    np.testing.assert_array_equal(r["idx"], exp_idx)
    assert exp_cnt.max() > wl.topk                       # the neighbourhood adds cubes
    out, of, _, _, lse = dense_vsa(_t(q), _t(k), _t(v), T, H, W, exp_idx, scale, gc=_t(gc), gf=_t(gf),
                                   cnt=exp_cnt, rank=rank)
    np.testing.assert_allclose(r["out"], out.numpy(), rtol=1e-10, atol=1e-10)
    p_ = oracle_mod.sfc_table(T, H, W, curve)
    np.testing.assert_allclose(r["lse"][:, p_], lse.numpy(), rtol=1e-12)
    g = oracle_mod.backward(q, k, v, dout, r["idx"], T, H, W, scale, gc=gc, gf=gf, curve=curve, cnt=r["cnt"])
    leaves = {n: torch.tensor(a, dtype=torch.float64, requires_grad=True)
              for n, a in (("q", q), ("k", k), ("v", v), ("gc", gc), ("gf", gf))}
    o2, *_ = dense_vsa(leaves["q"], leaves["k"], leaves["v"], T, H, W, exp_idx, scale, gc=leaves["gc"],
                       gf=leaves["gf"], cnt=exp_cnt, rank=rank)
    (o2 * torch.tensor(dout, dtype=torch.float64)).sum().backward()
    for n, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("gc", "dgc"), ("gf", "dgf")):
        np.testing.assert_allclose(g[key], leaves[n].grad.numpy(), rtol=1e-9, atol=1e-9, err_msg=key)


def test_padded_reordering_slots(oracle_mod):
    """Partial cubes: every token lands in its own cube's slot block, the
    padding slots are zero, the token counts are the partial box volumes, and
    the inverse drops the padding."""
    T, H, W = 5, 6, 10
    Tc, Hc, Wc = oracle_mod.cube_grid(T, H, W)
    assert (Tc, Hc, Wc) == (2, 2, 3)
    x = np.random.default_rng(5).standard_normal((2, T * H * W, 8))
    y = oracle_mod.permute(x, T, H, W)
    assert y.shape == (2, 64 * Tc * Hc * Wc, 8)
    slot_ok, ntok = oracle_mod.cube_slots(T, H, W)
    assert np.all(y[:, slot_ok == 0] == 0) and slot_ok.sum() == T * H * W
    box = lambda c, n: min(4, n - 4 * c)
    want = [box(ct, T) * box(ch, H) * box(cw, W) for ct in range(Tc) for ch in range(Hc) for cw in range(Wc)]
    assert ntok.tolist() == want
    pos = oracle_mod.sfc_table(T, H, W)
    np.testing.assert_array_equal(pos // 64, cube_ids(T, H, W))
    np.testing.assert_array_equal(oracle_mod.permute(y, T, H, W, inverse=True), x)
