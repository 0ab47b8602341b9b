"""GPU parity: every step of the CUDA path (through the C ABI) against the CPU
oracle on the same seeded inputs.  Integer work (reordering, Top-K on given
scores) must match bit for bit; floating-point outputs and gradients within
max-abs 2e-2 / mean-abs 2e-3 (tests/parity.py).  The Top-K selection is
checked against the oracle's float64 scores up to near-ties, and the fine
stage is then checked on the GPU-chosen lists."""
import zlib

import numpy as np
import pytest
import torch

import synth
from parity import LSE_MAX_ABS, LSE_MEAN_ABS, assert_close, check_topk_validity, exact_topk, lse_max_abs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vsa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from block_sparse_video_sfc_gb300 import build
    build.build()
    import block_sparse_video_sfc_gb300 as m
    return m


def dev(a, dtype=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dtype).contiguous()


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def status_ok(vsa):
    torch.cuda.synchronize()
    assert vsa.device_status() == 0


# ---------------------------------------------------------------- reorder + pool
@pytest.mark.parametrize("grid,d", [((4, 8, 8), 64), ((8, 12, 20), 128), ((12, 4, 8), 64), ((16, 32, 64), 128)])
def test_permute_pool(vsa, oracle_mod, grid, d):
    T, H, W = grid
    BH = 3
    x = synth.make_random((BH, T * H * W, d), seed=sum(grid) + d)
    y, pooled = vsa.permute(dev(x), T, H, W, pool=True)
    ref = oracle_mod.permute(x, T, H, W)
    assert np.array_equal(host(y), ref)                               # bit exact (data move)
    back = vsa.permute(y, T, H, W, inverse=True)
    assert np.array_equal(host(back), x.astype(np.float64))           # round trip
    np.testing.assert_allclose(host(pooled), oracle_mod.pool(ref), rtol=1e-5, atol=1e-6)
    status_ok(vsa)


# ---------------------------------------------------------------- coarse + Top-K
@pytest.mark.parametrize("name", ["tiny", "small", "wan1.3b", "long"])
def test_coarse_topk(vsa, oracle_mod, name):
    wl = synth.WORKLOADS[name]
    heads = list(range(wl.heads)) if wl.heads <= 12 else [0, wl.heads // 2, wl.heads - 1]
    q, k, v = synth.make_qkv(wl, heads_subset=heads)
    sh = (len(heads), wl.N, wl.d)
    q, k, v = (a.reshape(sh) for a in (q, k, v))
    pooled = [vsa.permute(dev(a), wl.T, wl.H, wl.W, pool=True)[1] for a in (q, k, v)]
    r = vsa.coarse_topk(*pooled, wl.topk, want_scores=True)
    status_ok(vsa)
    gidx = r["idx"].cpu().numpy()
    # 1) exact: the GPU Top-K of its own fp32 scores is the brute-force one
    gscores = r["scores"].cpu().numpy()
    np.testing.assert_array_equal(gidx, exact_topk(gscores, wl.topk))
    assert np.all(r["cnt"].cpu().numpy() == wl.topk)
    # 2) against the oracle's float64 scores: identical sets up to near-ties
    pq, pk, pv = (oracle_mod.pool(oracle_mod.permute(a, wl.T, wl.H, wl.W)) for a in (q, k, v))
    scores, oc, lse_c = oracle_mod.coarse(pq, pk, pv, wl.d ** -0.5)
    np.testing.assert_allclose(gscores, scores, rtol=1e-4, atol=1e-4)
    differing = check_topk_validity(gidx, scores, wl.topk)
    assert differing <= max(2, gidx.shape[0] * gidx.shape[1] // 100), differing
    np.testing.assert_allclose(host(r["oc"]), oc, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(host(r["lse_c"]), lse_c, rtol=1e-5, atol=1e-4)


def test_nan_scores_are_reported(vsa):
    """A NaN coarse score cannot be ranked: the Top-K latches an error that
    vsa_device_status reports as VSA_ERR_ARG (and clears); clean inputs then
    run clean."""
    g = torch.Generator().manual_seed(3)
    qc, kc, vc = (torch.randn(2, 64, 128, generator=g).cuda() for _ in range(3))
    vsa.coarse_topk(qc, kc, vc, 8)
    assert vsa.device_status() == 0
    qc[1, 17, 5] = float("nan")
    vsa.coarse_topk(qc, kc, vc, 8)
    assert vsa.device_status() == -1   # VSA_ERR_ARG
    assert vsa.device_status() == 0


# ---------------------------------------------------------------- fine forward
def _fine_case(oracle_mod, wl, heads=None):
    q, k, v = synth.make_qkv(wl, heads_subset=heads)
    nh = wl.heads if heads is None else len(heads)
    sh = (nh, wl.N, wl.d)
    qp, kp, vp = (oracle_mod.permute(a.reshape(sh), wl.T, wl.H, wl.W) for a in (q, k, v))
    return qp, kp, vp


@pytest.mark.parametrize("name", ["tiny", "tiny_dense", "small"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("workspace", [True, False])
def test_fine_fwd(vsa, oracle_mod, name, out_dtype, workspace):
    """vsa_fine_fwd with a workspace (fp16 copies, overlap pair plan) and
    without one (bf16 operands, V converted on chip)."""
    wl = synth.WORKLOADS[name]
    qp, kp, vp = _fine_case(oracle_mod, wl)
    rng = np.random.default_rng(1)
    idx = np.stack([np.stack([rng.permutation(wl.Nc)[:wl.topk] for _ in range(wl.Nc)])
                    for _ in range(wl.BH)]).astype(np.int32)
    cnt = np.full(idx.shape[:-1], wl.topk, np.int32)
    of, lse = vsa.fine_fwd(dev(qp), dev(kp), dev(vp), dev(idx, torch.int32), dev(cnt, torch.int32),
                           out_dtype=out_dtype, workspace=workspace)
    status_ok(vsa)
    rof, rlse = oracle_mod.fine_fwd(qp, kp, vp, idx, cnt, wl.d ** -0.5)
    assert_close(host(of), rof, bf16_out=out_dtype == torch.bfloat16, what="O_f")
    assert_close(host(lse), rlse, max_abs=LSE_MAX_ABS, mean_abs=LSE_MEAN_ABS, what="lse")


@pytest.mark.parametrize("workspace", [True, False])
def test_fine_fwd_ragged_and_edge_lists(vsa, oracle_mod, workspace):
    """Counts 0 / 1 / odd / K, K = 1 and an odd number of cubes (lone last pair)."""
    wl = synth.Workload("odd", 1, 3, 128, 4, 4, 20, 3)   # Nc = 5 cubes (odd)
    qp, kp, vp = _fine_case(oracle_mod, wl)
    idx = np.array([[[4, 0, 2], [1, 3, 0], [0, 1, 2], [2, 4, 3], [3, 2, 1]]] * 3, dtype=np.int32)
    cnt = np.array([[3, 0, 1, 2, 3], [0, 0, 0, 0, 1], [1, 1, 1, 1, 1]], dtype=np.int32)
    of, lse = vsa.fine_fwd(dev(qp), dev(kp), dev(vp), dev(idx, torch.int32), dev(cnt, torch.int32),
                           workspace=workspace)
    status_ok(vsa)
    rof, rlse = oracle_mod.fine_fwd(qp, kp, vp, idx, cnt, wl.d ** -0.5)
    assert_close(host(of), rof, what="O_f ragged")
    empty = np.isneginf(rlse)
    assert np.all(np.isneginf(host(lse)[empty])) and np.all(host(of)[empty] == 0)
    assert_close(host(lse)[~empty], rlse[~empty], max_abs=LSE_MAX_ABS, mean_abs=LSE_MEAN_ABS, what="lse")


@pytest.mark.parametrize("workspace", [True, False])
@pytest.mark.parametrize("d", [64, 128])
def test_fine_fwd_rising_scores_rescale_often(vsa, oracle_mod, workspace, d):
    """Scores that rise by ~3 log2 units per key cube, and lists whose first
    entry (the one a tile visits first) is their lowest-scored cube.  The
    kernel raises a row's running max only when it grows by more than 2^8, so
    here it does so every few steps, and each time rescales O after waiting
    for the PV product before it: a path that inputs whose largest scores sit
    in the first-visited cubes never take."""
    BH, Nc, K = 2, 48, 24
    N = 64 * Nc
    rng = np.random.default_rng(7 + d)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    scale = d ** -0.5
    beta = 3.0 / (scale * np.log2(np.e))          # q . k grows by 3 log2 units per cube
    cube = np.repeat(np.arange(Nc), 64)
    bf = lambda a: torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    q = bf(0.3 * rng.standard_normal((BH, N, d)) + u)
    k = bf(0.3 * rng.standard_normal((BH, N, d)) + (beta * cube)[None, :, None] * u)
    v = bf(rng.standard_normal((BH, N, d)))
    idx = np.empty((BH, Nc, K), np.int32)
    for b in range(BH):
        for c in range(Nc):
            pick = rng.permutation(Nc)[:K]
            lo = int(np.argmin(pick))
            idx[b, c] = np.concatenate([pick[lo:lo + 1], np.delete(pick, lo)])   # lowest cube first
    cnt = np.full((BH, Nc), K, np.int32)
    of, lse = vsa.fine_fwd(dev(q), dev(k), dev(v), dev(idx, torch.int32), dev(cnt, torch.int32),
                           workspace=workspace)
    status_ok(vsa)
    rof, rlse = oracle_mod.fine_fwd(q, k, v, idx, cnt, scale)
    assert rlse.max() > 50                                                      # the scores do rise
    assert_close(host(of), rof, what="O_f (rescaled rows)")
    assert_close(host(lse), rlse, max_abs=LSE_MAX_ABS, mean_abs=LSE_MEAN_ABS, what="lse (rescaled rows)")


def test_fine_fwd_dense_is_sdpa(vsa, oracle_mod):
    """K = all cubes: the fine kernel equals dense attention (torch SDPA, fp32)."""
    wl = synth.WORKLOADS["small"]
    qp, kp, vp = _fine_case(oracle_mod, wl, heads=[0, 1])
    idx = np.tile(np.arange(wl.Nc, dtype=np.int32), (2, wl.Nc, 1))
    cnt = np.full((2, wl.Nc), wl.Nc, np.int32)
    of, _ = vsa.fine_fwd(dev(qp), dev(kp), dev(vp), dev(idx, torch.int32), dev(cnt, torch.int32))
    ref = torch.nn.functional.scaled_dot_product_attention(*(torch.tensor(a) for a in (qp, kp, vp))).numpy()
    assert_close(host(of), ref, what="dense")


@pytest.mark.parametrize("workspace", [True, False])
def test_lut_errors_are_reported(vsa, oracle_mod, workspace):
    wl = synth.WORKLOADS["tiny"]
    qp, kp, vp = _fine_case(oracle_mod, wl)
    idx = np.zeros((wl.BH, wl.Nc, 2), np.int32)
    idx[..., 1] = 1
    idx[0, 1, 1] = 7            # out of range
    of, _ = vsa.fine_fwd(dev(qp), dev(kp), dev(vp), dev(idx, torch.int32), None, workspace=workspace)
    assert vsa.device_status() == -6
    idx[0, 1, 1] = 0            # repeated cube in a row
    vsa.fine_fwd(dev(qp), dev(kp), dev(vp), dev(idx, torch.int32), None, workspace=workspace)
    assert vsa.device_status() == -6
    idx[0, 1, 1] = 1
    vsa.fine_fwd(dev(qp), dev(kp), dev(vp), dev(idx, torch.int32), None, workspace=workspace)
    assert vsa.device_status() == 0


# ---------------------------------------------------------------- whole forward / backward
def _e2e(vsa, oracle_mod, wl, gates, out_dtype, grad_dtype, heads=None, cube_order=None, radius=-1):
    q, k, v = synth.make_qkv(wl, heads_subset=heads)
    gc = gf = None
    if gates:
        gc, gf = synth.make_gates(wl, heads_subset=heads)
    dout = synth.make_dout(wl, heads_subset=heads)
    D = lambda a: None if a is None else dev(a)
    out, st = vsa.forward(D(q), D(k), D(v), wl.T, wl.H, wl.W, wl.topk, g_coarse=D(gc), g_fine=D(gf),
                          out_dtype=out_dtype, cube_order=cube_order, radius=radius)
    bws = torch.empty(vsa.workspace_bytes(1, wl.B, wl.heads, wl.d, wl.T, wl.H, wl.W, wl.topk, radius),
                      dtype=torch.uint8, device="cuda")
    g = vsa.backward(st, D(dout), g_coarse=D(gc), g_fine=D(gf), grad_dtype=grad_dtype, ws=bws)
    status_ok(vsa)
    saved = st.saved()
    saved["key_pairs"] = vsa.backward_tile_pairs(st, bws)
    return q, k, v, gc, gf, dout, out, g, saved


def _gpu_lists(vsa, oracle_mod, wl, saved, scores_by_head, radius, curve="raster"):
    """The selection lists the GPU forward saved, checked: with radius < 0 they
    are a valid Top-K of the oracle's scores; with a radius, the GPU's own
    Top-K (the coarse kernel rerun on the saved pooled vectors) is a valid
    Top-K and the saved lists are exactly its union with the radius
    neighbourhood (the oracle's list transform, bit for bit).
    scores_by_head: {head: oracle scores [Nc, Nc]}.  Returns (idx, cnt) as
    [heads, Nc, kmax] and [heads, Nc]."""
    kmax = oracle_mod.list_width(wl.topk, radius, wl.Nc)
    idx = saved["idx"].view(wl.heads, wl.Nc, kmax).cpu().numpy()
    cnt = saved["cnt"].view(wl.heads, wl.Nc).cpu().numpy()
    if radius < 0:
        tk = idx
        assert np.all(cnt == wl.topk)
        # saved in ascending cube id: the sets the public (highest-first)
        # selection gives on the saved pooled vectors
        assert np.all(np.diff(idx, axis=-1) > 0)
        r = vsa.coarse_topk(saved["qc"], saved["kc"], saved["vc"], wl.topk, want_oc=False)
        np.testing.assert_array_equal(idx, np.sort(r["idx"].view(wl.heads, wl.Nc, wl.topk).cpu().numpy(), -1))
    else:
        r = vsa.coarse_topk(saved["qc"], saved["kc"], saved["vc"], wl.topk, want_oc=False)
        tk = r["idx"].view(wl.heads, wl.Nc, wl.topk).cpu().numpy()
        ridx, rcnt, ovf = oracle_mod.lut_add_neighbors(tk, None, wl.T, wl.H, wl.W, radius, kmax, curve=curve)
        assert not ovf
        np.testing.assert_array_equal(idx, ridx)
        np.testing.assert_array_equal(cnt, rcnt)
    for h, sc in scores_by_head.items():
        check_topk_validity(tk[h:h + 1], sc, wl.topk)
    return idx, cnt


def _key_cubes(idx1, kpairs0, keys_per_row, budget_flop=2.5e11):
    """Key cubes of one head whose dK / dV are compared element by element:
    the most-listed (longest inverse-list walk), a median one, the
    least-listed listed one, an unlisted one if any, and both cubes of the
    planned dK/dV tile holding the most-listed cube.  A cube is skipped when
    the oracle's cost for it (every listing query row recomputes its softmax
    over keys_per_row keys) exceeds budget_flop, except the first cube."""
    Nc = idx1.shape[-2]
    inv = np.bincount(idx1.reshape(-1)[idx1.reshape(-1) >= 0], minlength=Nc)
    listed = np.flatnonzero(inv > 0)
    order = listed[np.argsort(inv[listed], kind="stable")]
    top = int(order[-1])
    tile = [t for t in kpairs0 if top in (int(t[0]), int(t[1]))]
    assert len(tile) == 1, "the most-listed key cube sits in exactly one planned tile"
    picks = [top, int(order[len(order) // 2]), int(order[0])] + [int(c) for c in tile[0] if c >= 0]
    if (inv == 0).any():
        picks.append(int(np.flatnonzero(inv == 0)[0]))
    out, spent = [], 0.0
    for c in dict.fromkeys(picks):
        cost = 4.0 * inv[c] * 64 * keys_per_row * 128
        if out and spent + cost > budget_flop:
            continue
        out.append(c)
        spent += cost
    return out, tile[0]


@pytest.mark.parametrize("name,gates", [("tiny", True), ("tiny", False), ("tiny_dense", True), ("small", True)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_forward_backward(vsa, oracle_mod, name, gates, dtype):
    wl = synth.WORKLOADS[name]
    q, k, v, gc, gf, dout, out, g, saved = _e2e(vsa, oracle_mod, wl, gates, dtype, dtype)
    gidx = saved["idx"].cpu().numpy().reshape(wl.B, wl.heads, wl.Nc, wl.topk)
    ref0 = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=gc, gf=gf)
    check_topk_validity(gidx, ref0["scores"], wl.topk)
    # fine stage and everything after it on the GPU-chosen (validated) lists
    ref = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=gc, gf=gf, lut=gidx)
    bf = dtype == torch.bfloat16
    assert_close(host(out), ref["out"], bf16_out=bf, what="out")
    rg = oracle_mod.backward(q, k, v, dout, gidx, wl.T, wl.H, wl.W, gc=gc, gf=gf)
    for n in ("dq", "dk", "dv", "dgc", "dgf"):
        if rg[n] is not None:
            assert_close(host(g[n]), rg[n], bf16_out=bf, what=n)


@pytest.mark.parametrize("name,radius,curve", [("tiny", 0, "raster"), ("small", 1, "raster"),
                                               ("odd_small", 1, "hilbert"), ("small", 2, "hilbert")])
def test_adjacency_forward_backward(vsa, oracle_mod, name, radius, curve):
    """Top-K united with the radius-r cube neighbourhood ([AMD] "Comparison
    with Jenga": importance and adjacency masks), through vsa_forward and
    vsa_backward: lists checked by _gpu_lists, then the output and every
    gradient against the oracle run on the GPU's lists."""
    wl = synth.WORKLOADS[name]
    order = None if curve == "raster" else vsa.cube_order(wl.T, wl.H, wl.W, curve)
    q, k, v, gc, gf, dout, out, g, saved = _e2e(vsa, oracle_mod, wl, True, torch.float32, torch.float32,
                                                cube_order=order, radius=radius)
    ref0 = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=gc, gf=gf, curve=curve)
    scores = ref0["scores"].reshape(wl.heads, wl.Nc, wl.Nc)
    idx, cnt = _gpu_lists(vsa, oracle_mod, wl, saved, {h: scores[h] for h in range(wl.heads)}, radius, curve)
    assert cnt.max() > wl.topk
    lut, lcnt = idx.reshape((wl.B, wl.heads) + idx.shape[1:]), cnt.reshape(wl.B, wl.heads, wl.Nc)
    ref = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=gc, gf=gf, lut=lut, cnt=lcnt, curve=curve)
    assert_close(host(out), ref["out"], what="out")
    rg = oracle_mod.backward(q, k, v, dout, lut, wl.T, wl.H, wl.W, gc=gc, gf=gf, curve=curve, cnt=lcnt)
    for n in ("dq", "dk", "dv", "dgc", "dgf"):
        assert_close(host(g[n]), rg[n], what=n)


def test_fine_bwd_entry_point(vsa, oracle_mod):
    wl = synth.WORKLOADS["small"]
    heads = [1, 6]
    qp, kp, vp = _fine_case(oracle_mod, wl, heads=heads)
    rng = np.random.default_rng(4)
    idx = np.stack([np.stack([rng.permutation(wl.Nc)[:wl.topk] for _ in range(wl.Nc)])
                    for _ in heads]).astype(np.int32)
    cnt = np.full(idx.shape[:-1], wl.topk, np.int32)
    cnt[0, 3] = 0
    cnt[1, 7] = 5
    dof = synth.make_random(qp.shape, seed=8)
    of, lse = vsa.fine_fwd(dev(qp), dev(kp), dev(vp), dev(idx, torch.int32), dev(cnt, torch.int32))
    dq, dk, dv = vsa.fine_bwd(dev(qp), dev(kp), dev(vp), of, lse, dev(dof), dev(idx, torch.int32),
                              dev(cnt, torch.int32))
    status_ok(vsa)
    rq, rk, rv = oracle_mod.fine_bwd(qp, kp, vp, dof, idx, cnt, wl.d ** -0.5)
    assert_close(host(dq), rq, what="dq")
    assert_close(host(dk), rk, what="dk")
    assert_close(host(dv), rv, what="dv")


def test_full_size_head_sample(vsa, oracle_mod):
    """Wan-1.3B-shaped layer (32768 tokens, 512 cubes, K=154, 12 heads) in the
    launch configuration the benchmark times; the oracle recomputes head 0 in
    full for the forward, and sampled query rows / key cubes for the backward."""
    wl = synth.WORKLOADS["wan1.3b"]
    q, k, v, gc, gf, dout, out, g, saved = _e2e(vsa, oracle_mod, wl, True, torch.float32, torch.float32)
    h0 = lambda a: a[:, :1]
    gidx = saved["idx"].cpu().numpy().reshape(wl.B, wl.heads, wl.Nc, wl.topk)
    scale = wl.d ** -0.5
    ref = oracle_mod.forward(h0(q), h0(k), h0(v), wl.T, wl.H, wl.W, wl.topk, gc=h0(gc), gf=h0(gf))
    check_topk_validity(gidx[:, :1], ref["scores"], wl.topk)
    lut = gidx[:, :1]
    ref = oracle_mod.forward(h0(q), h0(k), h0(v), wl.T, wl.H, wl.W, wl.topk, gc=h0(gc), gf=h0(gf), lut=lut,
                             want_scores=False)
    assert_close(host(out)[:, :1], ref["out"], what="out head 0")
    # backward, head 0: sampled rows of the fine stage + exact coarse stage
    T_, H_, W_ = wl.T, wl.H, wl.W
    P = lambda a: oracle_mod.permute(a.reshape(1, wl.N, wl.d), T_, H_, W_)
    qp, kp, vp, gcp, gfp, dop = (P(h0(a)) for a in (q, k, v, gc, gf, dout))
    pos = oracle_mod.sfc_table(T_, H_, W_)
    dof, doc, _, _ = oracle_mod.combine_bwd(dop, gcp, gfp, ref["oc"].reshape(1, wl.Nc, wl.d),
                                            ref["of"].reshape(1, wl.N, wl.d))
    pq, pk, pv = (oracle_mod.pool(a) for a in (qp, kp, vp))
    dqc, dkc, dvc = oracle_mod.coarse_bwd(pq, pk, pv, doc, scale)
    idx1 = lut.reshape(1, wl.Nc, wl.topk)
    cnt1 = np.full((1, wl.Nc), wl.topk, np.int32)
    rows = np.random.default_rng(0).choice(wl.N, 48, replace=False)        # reordered positions
    dq_rows = oracle_mod.fine_bwd_query_rows(qp, kp, vp, dof, idx1, cnt1, scale, rows)
    dq_rows += dqc[0, rows // 64] / 64.0
    native = np.argsort(pos)[rows]                                          # native token of each row
    assert_close(host(g["dq"])[0, 0, native], dq_rows, what="dq rows")
    lse_rows = np.asarray(rows)
    _, rl = oracle_mod.fine_fwd_rows(qp, kp, vp, idx1, cnt1, scale, lse_rows)
    assert_close(host(saved["lse"])[0, lse_rows], rl, max_abs=lse_max_abs(64 * wl.topk), mean_abs=LSE_MEAN_ABS,
                 what="lse rows")
    kcubes, tile = _key_cubes(idx1, saved["key_pairs"][0].cpu().numpy(), 64 * wl.topk)
    assert tile[0] in kcubes and (tile[1] < 0 or tile[1] in kcubes)
    for c in kcubes:
        dk_c, dv_c = oracle_mod.fine_bwd_key_cube(qp, kp, vp, dof, idx1, cnt1, scale, 0, c)
        dk_c += dkc[0, c] / 64.0
        dv_c += dvc[0, c] / 64.0
        nat = np.argsort(pos)[64 * c:64 * c + 64]
        assert_close(host(g["dk"])[0, 0, nat], dk_c, what=f"dk cube {c}")
        assert_close(host(g["dv"])[0, 0, nat], dv_c, what=f"dv cube {c}")
    # properties at full size, all heads: sum_j dK_j = 0 per head and channel
    dk_sum = host(g["dk"]).sum(axis=2)
    assert np.abs(dk_sum).max() < 5e-2 * max(1.0, np.abs(host(g["dk"])).max())


# ---------------------------------------------------------------- full sizes, sampled
def _sampled_checks(vsa, oracle_mod, wl, dtype, n_cubes=4, n_rows=48, radius=-1):
    """Full-size run of `wl` (all heads, bench launch configuration); the
    oracle recomputes, for the first and last head: the coarse scores (Top-K
    validity of the GPU lists), whole query cubes of the output, the fine LSE
    and dQ on sampled rows and dg_c / dg_f on the sampled cubes; and, for head
    0, dK / dV of the key cubes _key_cubes picks (most-listed, median,
    least-listed, unlisted, both cubes of a planned dK/dV tile) within the
    oracle's time budget.  All heads: sum_j dK_j = 0 per channel."""
    q, k, v, gc, gf, dout, out, g, saved = _e2e(vsa, oracle_mod, wl, True, dtype, dtype, radius=radius)
    bf = dtype == torch.bfloat16
    kmax = oracle_mod.list_width(wl.topk, radius, wl.Nc)
    scale = wl.d ** -0.5
    pos = oracle_mod.sfc_table(wl.T, wl.H, wl.W)
    slot_ok, ntok = oracle_mod.cube_slots(wl.T, wl.H, wl.W)   # padding slots of partial cubes
    native_of = np.full(64 * wl.Nc, -1, np.int64)
    native_of[pos] = np.arange(wl.N)                     # reordered position -> native token
    real = np.flatnonzero(slot_ok)
    rng = np.random.default_rng(zlib.crc32(wl.name.encode()))
    at = lambda t, h, nat: host(t[0, h, torch.from_numpy(nat).to(t.device)])
    heads = sorted({0, wl.heads - 1})
    pooled, scores_h = {}, {}
    for h in heads:
        P = lambda a: oracle_mod.permute(a[0, h].reshape(1, wl.N, wl.d), wl.T, wl.H, wl.W)
        pooled[h] = [oracle_mod.pool(P(a), ntok) for a in (q, k, v)]
        scores_h[h] = oracle_mod.coarse(*pooled[h], scale)[0]
    gidx, gcnt = _gpu_lists(vsa, oracle_mod, wl, saved, scores_h, radius)
    for h in heads:
        P = lambda a: oracle_mod.permute(a[0, h].reshape(1, wl.N, wl.d), wl.T, wl.H, wl.W)
        qp, kp, vp, gcp, gfp, dop = (P(a) for a in (q, k, v, gc, gf, dout))
        pq, pk, pv = pooled[h]
        scores, oc, _ = oracle_mod.coarse(pq, pk, pv, scale)
        idx1 = gidx[h].reshape(1, wl.Nc, kmax)
        cnt1 = gcnt[h].reshape(1, wl.Nc)
        # whole query cubes of the output (the first, the last, two random)
        cubes = np.unique(np.r_[0, wl.Nc - 1, rng.choice(wl.Nc, n_cubes - 2, replace=False)])
        rows = (64 * cubes[:, None] + np.arange(64)).reshape(-1)
        rows = rows[slot_ok[rows] == 1]
        of_rows, _ = oracle_mod.fine_fwd_rows(qp, kp, vp, idx1, cnt1, scale, rows, slot_ok=slot_ok)
        sub = lambda a: a[:, rows]
        ocr = oc[0, rows // 64]                                          # O_c of each row's cube
        out_ref = (sub(gcp)[0] * ocr + sub(gfp)[0] * of_rows)[None]
        assert_close(at(out, h, native_of[rows]), out_ref[0], bf16_out=bf, what=f"out head {h}")
        assert_close(at(g["dgc"], h, native_of[rows]), sub(dop)[0] * ocr, bf16_out=bf, what=f"dgc head {h}")
        assert_close(at(g["dgf"], h, native_of[rows]), sub(dop)[0] * of_rows, bf16_out=bf, what=f"dgf head {h}")
        # dO_f and dO_c of every row (O_f enters only dg_f, not used from this call)
        dof, doc, _, _ = oracle_mod.combine_bwd(dop, gcp, gfp, oc, np.zeros_like(dop))
        dqc, dkc, dvc = oracle_mod.coarse_bwd(pq, pk, pv, doc, scale)
        qrows = np.unique(np.r_[real[0], real[-1], rng.choice(real, n_rows - 2, replace=False)])
        dq_ref = (oracle_mod.fine_bwd_query_rows(qp, kp, vp, dof, idx1, cnt1, scale, qrows, slot_ok=slot_ok)
                  + dqc[0, qrows // 64] / ntok[qrows // 64, None])
        assert_close(at(g["dq"], h, native_of[qrows]), dq_ref, bf16_out=bf, what=f"dq rows head {h}")
        _, rl = oracle_mod.fine_fwd_rows(qp, kp, vp, idx1, cnt1, scale, qrows, slot_ok=slot_ok)
        assert_close(host(saved["lse"][h])[qrows], rl, max_abs=lse_max_abs(64 * kmax), mean_abs=LSE_MEAN_ABS,
                     what=f"lse rows head {h}")
        if h == 0:
            kcubes, _ = _key_cubes(idx1, saved["key_pairs"][0].cpu().numpy(), 64 * kmax)
            for c in kcubes:
                dk_c, dv_c = oracle_mod.fine_bwd_key_cube(qp, kp, vp, dof, idx1, cnt1, scale, 0, c, slot_ok=slot_ok)
                ok = slot_ok[64 * c:64 * c + 64] == 1
                nat = native_of[64 * c:64 * c + 64][ok]
                assert_close(at(g["dk"], h, nat), (dk_c + dkc[0, c] / ntok[c])[ok], bf16_out=bf, what=f"dk cube {c}")
                assert_close(at(g["dv"], h, nat), (dv_c + dvc[0, c] / ntok[c])[ok], bf16_out=bf, what=f"dv cube {c}")
    dk_sum = g["dk"].float().sum(dim=2)
    dk_max = g["dk"].float().abs().amax()
    assert float(dk_sum.abs().amax()) < 5e-2 * max(1.0, float(dk_max))


@pytest.mark.parametrize("name,dtype", [("wan1.3b_k512", torch.float32), ("wan1.3b_k256", torch.float32),
                                        ("wan1.3b_k64", torch.float32), ("wan14b", torch.bfloat16),
                                        ("long", torch.float32)])
def test_full_size_sampled(vsa, oracle_mod, name, dtype):
    """The 32K-token sparsity sweep (K = 512, 256, 64 of 512 cubes), the
    40-head Wan-14B-shaped layer and the 122880-token long video, at full size."""
    _sampled_checks(vsa, oracle_mod, synth.WORKLOADS[name], dtype)


def test_full_size_adjacency(vsa, oracle_mod):
    """The Wan-1.3B-shaped layer with each Top-K list united with its radius-1
    cube neighbourhood (up to 154 + 27 cubes per row), fwd + bwd at full size."""
    _sampled_checks(vsa, oracle_mod, synth.WORKLOADS["wan1.3b"], torch.float32, radius=1)


@pytest.mark.parametrize("name", ["small", "wan1.3b"])
def test_tile_pairs_partition(vsa, oracle_mod, name):
    """The query-cube pairing of the fine kernels' tiles (a scheduling choice):
    every cube in exactly one tile, and the pairing never walks more list
    entries in total than pairing cubes 2t and 2t + 1 would."""
    wl = synth.WORKLOADS[name]
    heads = [0, wl.heads - 1]
    q, k, v = (dev(a) for a in synth.make_qkv(wl, heads_subset=heads))
    out, st = vsa.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, out_dtype=torch.float32)
    status_ok(vsa)
    sv = st.saved()
    pairs = sv["tile_pairs"].cpu().numpy()
    idx = sv["idx"].cpu().numpy()
    for h in range(len(heads)):
        cubes = pairs[h].reshape(-1)
        assert (cubes == -1).sum() == wl.Nc % 2
        assert np.array_equal(np.sort(cubes[cubes >= 0]), np.arange(wl.Nc))
        sets = [set(r) for r in idx[h]]
        plan = sum(len(sets[a] | (sets[b] if b >= 0 else set())) for a, b in pairs[h])
        adjacent = sum(len(sets[2 * t] | (sets[2 * t + 1] if 2 * t + 1 < wl.Nc else set()))
                       for t in range((wl.Nc + 1) // 2))
        assert plan <= adjacent, (plan, adjacent)


def test_bounded_wait_timeout_is_reported(vsa, oracle_mod):
    """A wait that never completes gives up after its poll limit, latches
    VSA_ERR_TIMEOUT and leaves the context usable (no GPU fault involved)."""
    assert vsa.device_status() == 0
    vsa.selftest_wait_timeout(1 << 12)
    assert vsa.device_status() == -5  # VSA_ERR_TIMEOUT
    assert vsa.device_status() == 0   # reading cleared it
    wl = synth.WORKLOADS["tiny"]
    q, k, v = synth.make_qkv(wl)
    out, st = vsa.forward(dev(q), dev(k), dev(v), wl.T, wl.H, wl.W, wl.topk, out_dtype=torch.float32)
    status_ok(vsa)
    gidx = st.saved()["idx"].cpu().numpy().reshape(wl.B, wl.heads, wl.Nc, wl.topk)
    ref = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, lut=gidx)
    assert_close(host(out), ref["out"], what="out after a timeout")


# ---------------------------------------------------------------- index-list conversions
@pytest.mark.parametrize("BH,Nc,density,kmax", [(2, 64, 0.3, 64), (12, 512, 0.3, 512), (3, 1920, 0.1, 256)])
def test_mask_to_lut(vsa, oracle_mod, BH, Nc, density, kmax):
    """Jenga-style block matrix -> index list + count, bit for bit."""
    rng = np.random.default_rng(Nc)
    m = rng.random((BH, Nc, Nc)) < density
    idx, cnt = vsa.mask_to_lut(torch.from_numpy(m).cuda(), kmax)
    torch.cuda.synchronize()
    ridx, rcnt, ovf = oracle_mod.mask_to_lut(m, kmax)
    assert vsa.device_status() == (-6 if ovf else 0)
    assert np.array_equal(cnt.cpu().numpy(), rcnt)
    assert np.array_equal(idx.cpu().numpy(), ridx)


def test_mask_to_lut_overflow_is_reported(vsa, oracle_mod):
    m = np.ones((1, 40, 40), bool)
    idx, cnt = vsa.mask_to_lut(torch.from_numpy(m).cuda(), 16)
    assert vsa.device_status() == -6  # VSA_ERR_LUT
    ridx, rcnt, ovf = oracle_mod.mask_to_lut(m, 16)
    assert ovf and np.array_equal(idx.cpu().numpy(), ridx) and np.array_equal(cnt.cpu().numpy(), rcnt)


@pytest.mark.parametrize("name,radius", [("small", 1), ("wan1.3b", 1), ("long", 1), ("small", 2)])
def test_lut_add_neighbors_and_fine_fwd(vsa, oracle_mod, name, radius):
    """Top-K lists united with the spatial neighbourhood (bit for bit against
    the oracle), then the fine forward on the widened, ragged lists."""
    wl = synth.WORKLOADS[name]
    heads = [0]
    rng = np.random.default_rng(radius)
    idx = np.stack([np.stack([rng.permutation(wl.Nc)[:wl.topk] for _ in range(wl.Nc)])
                    for _ in heads]).astype(np.int32)
    cnt = rng.integers(wl.topk // 2, wl.topk + 1, size=idx.shape[:-1]).astype(np.int32)
    kout = wl.topk + (2 * radius + 1) ** 3
    gi, gc = vsa.lut_add_neighbors(dev(idx, torch.int32), dev(cnt, torch.int32), wl.T, wl.H, wl.W, radius, kout)
    status_ok(vsa)
    ri, rc, ovf = oracle_mod.lut_add_neighbors(idx, cnt, wl.T, wl.H, wl.W, radius, kout)
    assert not ovf
    assert np.array_equal(gc.cpu().numpy(), rc) and np.array_equal(gi.cpu().numpy(), ri)
    if name == "small":
        qp, kp, vp = _fine_case(oracle_mod, wl, heads=heads)
        of, lse = vsa.fine_fwd(dev(qp), dev(kp), dev(vp), gi, gc)
        status_ok(vsa)
        rof, rlse = oracle_mod.fine_fwd(qp, kp, vp, ri, rc, wl.d ** -0.5)
        assert_close(host(of), rof, what="O_f on widened lists")
        assert_close(host(lse), rlse, what="lse on widened lists")


# ---------------------------------------------------------------- Hilbert cube order
@pytest.mark.parametrize("grid", [(4, 8, 8), (8, 16, 32), (16, 32, 64), (32, 48, 80), (12, 20, 28), (21, 30, 52)])
def test_cube_order_table(vsa, oracle_mod, grid):
    """vsa_cube_order (point -> curve index on the GPU) against the oracle's
    ranks (curve index -> point), both curves, bit for bit."""
    T, H, W = grid
    Tc, Hc, Wc = oracle_mod.cube_grid(T, H, W)
    Nc = Tc * Hc * Wc
    for curve in ("raster", "hilbert"):
        tab = vsa.cube_order(T, H, W, curve).cpu().numpy()
        rank = oracle_mod.cube_rank(Tc, Hc, Wc, curve)
        np.testing.assert_array_equal(tab[Nc:], rank)
        np.testing.assert_array_equal(tab[:Nc], np.argsort(rank))
    status_ok(vsa)


@pytest.mark.parametrize("grid,d", [((8, 12, 20), 128), ((12, 20, 28), 64), ((16, 32, 64), 128)])
def test_permute_hilbert(vsa, oracle_mod, grid, d):
    T, H, W = grid
    order = vsa.cube_order(T, H, W, "hilbert")
    x = synth.make_random((2, T * H * W, d), seed=7 + d)
    y, pooled = vsa.permute(dev(x), T, H, W, pool=True, cube_order=order)
    ref = oracle_mod.permute(x, T, H, W, curve="hilbert")
    assert np.array_equal(host(y), ref)
    back = vsa.permute(y, T, H, W, inverse=True, cube_order=order)
    assert np.array_equal(host(back), x.astype(np.float64))
    np.testing.assert_allclose(host(pooled), oracle_mod.pool(ref), rtol=1e-5, atol=1e-6)
    status_ok(vsa)


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_forward_backward_hilbert(vsa, oracle_mod, name):
    wl = synth.WORKLOADS[name]
    order = vsa.cube_order(wl.T, wl.H, wl.W, "hilbert")
    q, k, v, gc, gf, dout, out, g, saved = _e2e(vsa, oracle_mod, wl, True, torch.float32, torch.float32,
                                                cube_order=order)
    gidx = saved["idx"].cpu().numpy().reshape(wl.B, wl.heads, wl.Nc, wl.topk)
    ref0 = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=gc, gf=gf, curve="hilbert")
    check_topk_validity(gidx, ref0["scores"], wl.topk)
    ref = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=gc, gf=gf, lut=gidx, curve="hilbert")
    assert_close(host(out), ref["out"], what="out")
    rg = oracle_mod.backward(q, k, v, dout, gidx, wl.T, wl.H, wl.W, gc=gc, gf=gf, curve="hilbert")
    for n in ("dq", "dk", "dv", "dgc", "dgf"):
        assert_close(host(g[n]), rg[n], what=n)


def test_lut_add_neighbors_hilbert(vsa, oracle_mod):
    T, H, W = 16, 32, 64
    Nc = (T // 4) * (H // 4) * (W // 4)
    order = vsa.cube_order(T, H, W, "hilbert")
    rng = np.random.default_rng(11)
    idx = np.stack([np.stack([rng.permutation(Nc)[:40] for _ in range(Nc)]) for _ in range(2)]).astype(np.int32)
    cnt = np.full(idx.shape[:-1], 40, np.int32)
    got, gcnt = vsa.lut_add_neighbors(dev(idx, torch.int32), dev(cnt, torch.int32), T, H, W, 2, 200,
                                      cube_order=order)
    status_ok(vsa)
    ref, rcnt, ovf = oracle_mod.lut_add_neighbors(idx, cnt, T, H, W, 2, 200, curve="hilbert")
    assert not ovf
    np.testing.assert_array_equal(gcnt.cpu().numpy(), rcnt)
    np.testing.assert_array_equal(got.cpu().numpy(), ref)


# ---------------------------------------------------------------- grids not divisible by 4
@pytest.mark.parametrize("grid,d,curve", [((5, 6, 10), 64, "raster"), ((9, 14, 22), 128, "raster"),
                                          ((9, 14, 22), 128, "hilbert"), ((21, 30, 52), 128, "raster")])
def test_permute_pool_padded(vsa, oracle_mod, grid, d, curve):
    """Partial boundary cubes: padding slots are zero in cube order, dropped on
    the way back, and left out of the cube means (bit-exact data movement)."""
    T, H, W = grid
    order = None if curve == "raster" else vsa.cube_order(T, H, W, curve)
    x = synth.make_random((2, T * H * W, d), seed=T + H + W)
    y, pooled = vsa.permute(dev(x), T, H, W, pool=True, cube_order=order)
    ref = oracle_mod.permute(x, T, H, W, curve=curve)
    assert np.array_equal(host(y), ref)
    back = vsa.permute(y, T, H, W, inverse=True, cube_order=order)
    assert np.array_equal(host(back), x.astype(np.float64))
    _, ntok = oracle_mod.cube_slots(T, H, W, curve)
    np.testing.assert_allclose(host(pooled), oracle_mod.pool(ref, ntok), rtol=1e-5, atol=1e-6)
    status_ok(vsa)


@pytest.mark.parametrize("name,curve", [("odd", "raster"), ("odd", "hilbert"), ("odd_small", "raster"),
                                        ("odd_small", "hilbert")])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_forward_backward_padded(vsa, oracle_mod, name, curve, dtype):
    wl = synth.WORKLOADS[name]
    order = None if curve == "raster" else vsa.cube_order(wl.T, wl.H, wl.W, curve)
    q, k, v, gc, gf, dout, out, g, saved = _e2e(vsa, oracle_mod, wl, True, dtype, dtype, cube_order=order)
    gidx = saved["idx"].cpu().numpy().reshape(wl.B, wl.heads, wl.Nc, wl.topk)
    ref0 = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=gc, gf=gf, curve=curve)
    check_topk_validity(gidx, ref0["scores"], wl.topk)
    ref = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=gc, gf=gf, lut=gidx, curve=curve)
    bf = dtype == torch.bfloat16
    assert_close(host(out), ref["out"], bf16_out=bf, what="out")
    rg = oracle_mod.backward(q, k, v, dout, gidx, wl.T, wl.H, wl.W, gc=gc, gf=gf, curve=curve)
    for n in ("dq", "dk", "dv", "dgc", "dgf"):
        assert_close(host(g[n]), rg[n], bf16_out=bf, what=n)


def test_full_size_wan_latent(vsa, oracle_mod):
    """The Wan2.1 latent grid itself, 21 x 30 x 52 = 32760 tokens (624 cubes,
    partial along all three axes), 12 heads, K = 187, sampled as above."""
    _sampled_checks(vsa, oracle_mod, synth.WORKLOADS["wan1.3b_latent"], torch.float32)


@pytest.mark.parametrize("name,curve,dtype", [("odd", "hilbert", torch.bfloat16), ("odd_small", "raster", torch.float32),
                                              ("small", "hilbert", torch.float32), ("wan1.3b", "raster", torch.bfloat16)])
def test_every_output_element_is_written(vsa, name, curve, dtype):
    """out, dq, dk, dv, dg_c, dg_f are written in full by the library (the
    gradients by the fine backward epilogues, each native token once, padding
    slots never): buffers pre-filled with NaN come back finite and equal, bit
    for bit, to a run into zero-filled buffers."""
    wl = synth.WORKLOADS[name]
    order = None if curve == "raster" else vsa.cube_order(wl.T, wl.H, wl.W, curve)
    q, k, v = (dev(a) for a in synth.make_qkv(wl))
    gc, gf = (dev(a) for a in synth.make_gates(wl))
    dout = dev(synth.make_dout(wl))
    runs = []
    for fill in (float("nan"), 0.0):
        out = torch.full_like(q, fill, dtype=dtype)
        _, st = vsa.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, g_coarse=gc, g_fine=gf, out=out, cube_order=order)
        grads = {n: torch.full_like(q, fill, dtype=dtype) for n in ("dq", "dk", "dv", "dgc", "dgf")}
        vsa.backward(st, dout, g_coarse=gc, g_fine=gf, grads=grads)
        status_ok(vsa)
        runs.append([out] + [grads[n] for n in ("dq", "dk", "dv", "dgc", "dgf")])
    for a, b in zip(*runs):
        assert bool(torch.isfinite(a).all())
        assert torch.equal(a, b)


# ---------------------------------------------------------------- CUDA graphs
def test_forward_backward_capture_in_a_cuda_graph(vsa, oracle_mod):
    """The forward and backward enqueue only stream work (no host sync, no
    allocation), so a whole training step can be captured in a CUDA graph;
    replays give the eager results bit for bit."""
    wl = synth.WORKLOADS["small"]
    q, k, v = synth.make_qkv(wl)
    gc, gf = synth.make_gates(wl)
    dout = synth.make_dout(wl)
    ins = [dev(a) for a in (q, k, v, gc, gf, dout)]
    out = torch.empty_like(ins[0])
    grads = {n: torch.empty_like(ins[0]) for n in ("dq", "dk", "dv", "dgc", "dgf")}
    fws = torch.empty(vsa.workspace_bytes(0, wl.B, wl.heads, wl.d, wl.T, wl.H, wl.W, wl.topk), dtype=torch.uint8,
                      device="cuda")
    bws = torch.empty(vsa.workspace_bytes(1, wl.B, wl.heads, wl.d, wl.T, wl.H, wl.W, wl.topk), dtype=torch.uint8,
                      device="cuda")

    def step():
        _, st = vsa.forward(*ins[:3], wl.T, wl.H, wl.W, wl.topk, g_coarse=ins[3], g_fine=ins[4], out=out, ws=fws)
        vsa.backward(st, ins[5], g_coarse=ins[3], g_fine=ins[4], grads=grads, ws=bws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                     # eager, on the capture stream's device state
    torch.cuda.current_stream().wait_stream(side)
    status_ok(vsa)
    eager = [out.clone()] + [grads[n].clone() for n in ("dq", "dk", "dv", "dgc", "dgf")]
    for t in [out] + list(grads.values()):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    status_ok(vsa)
    replay = [out] + [grads[n] for n in ("dq", "dk", "dv", "dgc", "dgf")]
    for a, b in zip(eager, replay):
        assert torch.equal(a, b)


# ---------------------------------------------------------------- inference forward (permute folded into TMA)
@pytest.mark.parametrize("name,curve", [("tiny", "raster"), ("small", "raster"), ("small", "hilbert"),
                                        ("odd", "raster"), ("odd_small", "hilbert"), ("wan1.3b", "raster")])
def test_forward_inference(vsa, oracle_mod, name, curve):
    """vsa_forward_inference reads Q, K, V through 5-D TMA boxes in native
    layout and multiplies in bf16: the same index lists as vsa_forward, its
    output within the parity tolerance of vsa_forward's and of the oracle's."""
    wl = synth.WORKLOADS[name]
    order = None if curve == "raster" else vsa.cube_order(wl.T, wl.H, wl.W, curve)
    q, k, v = synth.make_qkv(wl)
    gc, gf = synth.make_gates(wl)
    ins = [dev(a) for a in (q, k, v, gc, gf)]
    out_f, st = vsa.forward(*ins[:3], wl.T, wl.H, wl.W, wl.topk, g_coarse=ins[3], g_fine=ins[4],
                            out_dtype=torch.float32, cube_order=order)
    out_i = vsa.forward_inference(*ins[:3], wl.T, wl.H, wl.W, wl.topk, g_coarse=ins[3], g_fine=ins[4],
                                  out_dtype=torch.float32, cube_order=order)
    status_ok(vsa)
    assert_close(host(out_i), host(out_f), what="out (inference vs forward)")
    if wl.N <= 4096:
        gidx = st.saved()["idx"].cpu().numpy().reshape(wl.B, wl.heads, wl.Nc, wl.topk)
        ref = oracle_mod.forward(q, k, v, wl.T, wl.H, wl.W, wl.topk, gc=gc, gf=gf, lut=gidx, curve=curve)
        assert_close(host(out_i), ref["out"], what="out (inference)")
