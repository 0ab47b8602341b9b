"""The C-ABI library loads, exports every entry point include/vsa.h declares,
and rejects bad arguments on the host before any CUDA call.  No GPU needed:
every call here returns from the argument checks."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_video_sfc_gb300 import build
    build.build()
    from block_sparse_video_sfc_gb300 import _lib
    return _lib


def _declared():
    src = open(os.path.join(ROOT, "include", "vsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vsa_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(so, n), n
    assert set(names) == set(lib.SIGNATURES)


def test_status_strings(lib):
    L = lib.load()
    for s in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert L.vsa_status_string(s)
    assert L.vsa_status_string(12345) == b"unknown status"


def test_workspace_bytes(lib):
    L = lib.load()
    g = lib.Grid.of(16, 32, 64)
    fwd = L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 12, 128, g, 154, -1)
    N, Nc = 32768, 512
    assert fwd >= 12 * N * 128 * (3 * 2 + 4)   # permuted Q/K/V + fp32 O_f at least
    bwd = L.vsa_workspace_bytes(lib.VSA_OP_BACKWARD, 1, 12, 128, g, 154, -1)
    # fp16 dO_f plus per-row and per-cube scratch; the fine gradients go straight to the outputs
    assert 12 * N * 128 * 2 < bwd < 12 * N * 128 * 3
    assert L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 12, 128, g, 0, -1) == 0        # K < 1
    assert L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 12, 128, g, Nc + 1, -1) == 0   # K > Nc
    assert L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 12, 96, g, 4, -1) == 0         # d
    # a side that is not a multiple of 4: partial cubes, sized like the covering grid
    assert (L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 12, 128, lib.Grid.of(6, 7, 5), 2, -1)
            == L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 12, 128, lib.Grid.of(8, 8, 8), 2, -1) > 0)
    assert L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 12, 128, lib.Grid.of(0, 8, 8), 1, -1) == 0
    assert L.vsa_workspace_bytes(7, 1, 12, 128, g, 4, -1) == 0
    # adjacency-forced selection: lists of topk + (2r + 1)^3 entries (at most Nc), radius in -1..7
    with_r1 = L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 12, 128, g, 154, 1)
    assert with_r1 > fwd and (with_r1 - fwd) >= 12 * Nc * (154 + 27) * 4 - 12 * Nc * 154 * 4
    assert L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 12, 128, g, 154, 8) == 0
    assert L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 12, 128, g, 154, -2) == 0
    # the backward's inverse lists (CSR) hold one id per listed (query, key) cube pair
    assert L.vsa_workspace_bytes(lib.VSA_OP_BACKWARD, 1, 12, 128, g, 154, 1) - bwd == 12 * Nc * 27 * 4
    # the public fine forward: fp16 Q, K, V plus the pair plan (pairs, window overlaps); the fine
    # backward: fp16 Q, K, V, dO_f, D, the inverse lists and two pair plans
    plan = 12 * Nc // 2 * 8 + 12 * Nc * 32 * 2
    ffwd = L.vsa_workspace_bytes(lib.VSA_OP_FINE_FWD, 1, 12, 128, g, 154, -1)
    assert 12 * N * 128 * 2 * 3 + plan <= ffwd < 12 * N * 128 * 2 * 3 + plan + 4096
    fbwd = L.vsa_workspace_bytes(lib.VSA_OP_FINE_BWD, 1, 12, 128, g, 154, -1)
    assert 12 * N * (128 * 2 * 4 + 4) + 12 * Nc * 154 * 4 + 2 * plan <= fbwd
    # the coarse rows must fit on chip: Nc = 2400 cubes is too many at d = 128, not at d = 64;
    # the fine calls have no such limit
    big = lib.Grid.of(4, 4 * 48, 4 * 50)
    assert L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 1, 128, big, 16, -1) == 0
    assert L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, 1, 64, big, 16, -1) > 0
    assert L.vsa_workspace_bytes(lib.VSA_OP_FINE_FWD, 1, 1, 128, big, 16, -1) > 0


def test_workspaces_hold_no_cube_by_cube_matrix(lib):
    """The long video (24 heads, 1920 cubes, Top-K 192): the workspaces grow
    with the tokens and the listed cubes, not with Nc x Nc (one fp32 [BH, Nc,
    Nc] matrix alone would be 354 MB)."""
    L = lib.load()
    g = lib.Grid.of(32, 48, 80)
    BH, N, Nc, K, d = 24, 122880, 1920, 192, 128
    fwd = L.vsa_workspace_bytes(lib.VSA_OP_FORWARD, 1, BH, d, g, K, -1)
    bwd = L.vsa_workspace_bytes(lib.VSA_OP_BACKWARD, 1, BH, d, g, K, -1)
    per_token_fwd = BH * N * (3 * d * 2 + d * 4 + 4)        # fp16 Q/K/V copies, fp32 O_f, the LSE
    plan = 4 + 32 * 2 + 8                                   # pair plan, its window overlaps, slot mask
    per_cube = BH * Nc * (4 * d * 4 + 4 + K * 4 + 4 + plan)  # pooled Q/K/V, O_c, LSE_c, lists, counts
    assert fwd < per_token_fwd + per_cube + (1 << 20)
    per_token_bwd = BH * N * (d * 2 + 4)                    # fp16 dO_f, D
    per_cube_bwd = BH * Nc * (4 * d * 4 + 4 + (K + 2) * 4 + 4 + plan)  # dO_c, dX_c, D_c, CSR
    assert bwd < per_token_bwd + per_cube_bwd + (1 << 20)   # 1 MB of slack against 354 MB per matrix


def test_host_side_argument_errors(lib):
    L = lib.load()
    fake = ctypes.c_void_p(0x1000)       # never dereferenced: every call fails its checks first
    fake2 = ctypes.c_void_p(0x2000)
    g = lib.Grid.of(4, 8, 8)
    # bad grid / cube / d
    assert L.vsa_permute(fake, fake2, None, 1, 64, lib.Grid.of(4, 0, 8), 0, None) == lib.VSA_ERR_ARG
    assert L.vsa_permute(fake, fake2, None, 1, 64, lib.Grid(4, 8, 8, 2, 4, 4), 0, None) == lib.VSA_ERR_UNSUPPORTED
    assert L.vsa_permute(fake, fake2, None, 1, 80, g, 0, None) == lib.VSA_ERR_UNSUPPORTED
    # null, aliasing, misaligned, pooled with inverse
    assert L.vsa_permute(None, fake2, None, 1, 64, g, 0, None) == lib.VSA_ERR_ARG
    assert L.vsa_permute(fake, fake, None, 1, 64, g, 0, None) == lib.VSA_ERR_ARG
    assert L.vsa_permute(ctypes.c_void_p(0x1002), fake2, None, 1, 64, g, 0, None) == lib.VSA_ERR_ARG
    assert L.vsa_permute(fake, fake2, fake, 1, 64, g, 1, None) == lib.VSA_ERR_ARG
    assert L.vsa_permute(fake, fake2, None, 1, 64, lib.Grid.of(4, 8, 8, 0x1002), 0, None) == lib.VSA_ERR_ARG
    assert L.vsa_cube_order(g, 5, fake2, None) == lib.VSA_ERR_ARG                # unknown curve
    # Top-K range
    for K in (0, 5):
        assert L.vsa_coarse_topk(fake, fake, fake, 1, 4, 64, K, 0.125, None, None, fake2, None, None,
                                 None) == lib.VSA_ERR_ARG
    # fine: N not a multiple of 64
    assert L.vsa_fine_fwd(fake, fake, fake, fake2, None, 2, 1, 100, 64, 0.125, fake2, 1, None,
                          None, 0, None) == lib.VSA_ERR_SHAPE
    assert L.vsa_fine_fwd(fake, fake, fake, fake2, None, 2, 1, 128, 64, 0.125, fake2, 7, None,
                          None, 0, None) == lib.VSA_ERR_ARG
    # fine forward given a workspace: too small, or misaligned
    assert L.vsa_fine_fwd(fake, fake, fake, fake2, None, 2, 1, 128, 64, 0.125, fake2, 1, None,
                          fake2, 16, None) == lib.VSA_ERR_WORKSPACE
    assert L.vsa_fine_fwd(fake, fake, fake, fake2, None, 2, 1, 128, 64, 0.125, fake2, 1, None,
                          ctypes.c_void_p(0x2008), 1 << 30, None) == lib.VSA_ERR_WORKSPACE
    # forward: workspace too small
    assert L.vsa_forward(fake, fake, fake, None, None, 1, 2, 64, g, 2, -1, 0.125, fake2, 0, fake2, 16,
                         None) == lib.VSA_ERR_WORKSPACE
    assert L.vsa_forward(fake, fake, fake, None, None, 1, 2, 64, g, 9, -1, 0.125, fake2, 0, fake2, 1 << 30,
                         None) == lib.VSA_ERR_ARG
    assert L.vsa_backward(fake, None, None, fake, 1, 2, 64, g, 2, -1, 0.125, fake2, fake2, fake2, None, None, 3,
                          fake2, 1 << 30, None) == lib.VSA_ERR_ARG
    # backward: workspace too small, null or misaligned outputs, Top-K out of range
    bf16 = lib.VSA_DTYPE_BF16
    assert L.vsa_backward(fake, None, None, fake, 1, 2, 64, g, 2, -1, 0.125, fake2, fake2, fake2, None, None, bf16,
                          fake2, 16, None) == lib.VSA_ERR_WORKSPACE
    assert L.vsa_backward(fake, None, None, fake, 1, 2, 64, g, 2, -1, 0.125, None, fake2, fake2, None, None, bf16,
                          fake2, 1 << 30, None) == lib.VSA_ERR_ARG
    assert L.vsa_backward(fake, None, None, fake, 1, 2, 64, g, 2, -1, 0.125, fake2, ctypes.c_void_p(0x2008), fake2,
                          None, None, bf16, fake2, 1 << 30, None) == lib.VSA_ERR_ARG
    for K in (0, 5):
        assert L.vsa_backward(fake, None, None, fake, 1, 2, 64, g, K, -1, 0.125, fake2, fake2, fake2, None, None, bf16,
                              fake2, 1 << 30, None) == lib.VSA_ERR_ARG
    for r in (-2, 8):   # radius out of range
        assert L.vsa_forward(fake, fake, fake, None, None, 1, 2, 64, g, 2, r, 0.125, fake2, 0, fake2, 1 << 30,
                             None) == lib.VSA_ERR_ARG
        assert L.vsa_backward(fake, None, None, fake, 1, 2, 64, g, 2, r, 0.125, fake2, fake2, fake2, None, None, bf16,
                              fake2, 1 << 30, None) == lib.VSA_ERR_ARG
