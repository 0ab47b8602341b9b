"""vsa_fine_bwd_noalloc: the fine backward for callers that cannot give the
library scratch memory -- code inside a runtime that hands out device memory
only through its own pool (or forbids allocation once running), and plain C
callers without an allocator.  It keeps its scratch in the library's fixed
device array.  Checked through the C ABI: its gradients equal the oracle's
(the tolerance of every parity test) and vsa_fine_bwd's, call after call (the
array keeps the previous call's contents), at d = 128 and d = 64 and at the
largest problem the array holds; one head more is refused before anything
runs.  This file is collected last so that a stop at the first failure has
run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from block_sparse_video_sfc_gb300 import build
    build.build()
    from block_sparse_video_sfc_gb300 import _lib
    return _lib


def _case(BH, N, d, K, seed):
    rng = np.random.default_rng(seed)
    Nc = N // 64
    q, k, v, dof = (synth.make_random((BH, N, d), seed=seed + i) for i in range(4))
    idx = np.stack([np.stack([rng.permutation(Nc)[:K] for _ in range(Nc)]) for _ in range(BH)]).astype(np.int32)
    cnt = np.full(idx.shape[:-1], K, np.int32)
    cnt[0, 1] = 0                                   # an empty list
    cnt[-1, Nc - 1] = 3                             # a short one
    D = lambda a, t=torch.bfloat16: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(t).contiguous()
    return D(q), D(k), D(v), D(dof), D(idx, torch.int32), D(cnt, torch.int32)


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _host(t):
    return t.float().cpu().numpy().astype(np.float64)


def _noalloc(lib, q, k, v, of, lse, dof, idx, cnt):
    BH, N, d = q.shape
    dq, dk, dv = (torch.full((BH, N, d), float("nan"), dtype=torch.float32, device="cuda") for _ in range(3))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.load().vsa_fine_bwd_noalloc(_p(q), _p(k), _p(v), _p(of), lib.VSA_DTYPE_F32, _p(lse), _p(dof), _p(idx),
                                         _p(cnt), idx.shape[-1], BH, N, d, d ** -0.5, _p(dq), _p(dk), _p(dv), stream)
    assert st == lib.VSA_OK, st
    return dq, dk, dv


def _check(lib, oracle_mod, BH, N, d, K, seed, oracle_heads):
    import block_sparse_video_sfc_gb300 as vsa
    q, k, v, dof, idx, cnt = _case(BH, N, d, K, seed)
    of, lse = vsa.fine_fwd(q, k, v, idx, cnt)
    ref = vsa.fine_bwd(q, k, v, of, lse, dof, idx, cnt)
    got = _noalloc(lib, q, k, v, of, lse, dof, idx, cnt)
    torch.cuda.synchronize()
    assert vsa.device_status() == 0
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert_close(_host(a), _host(b), what=f"{name} vs vsa_fine_bwd (BH={BH}, d={d}, seed {seed})")
    hs = list(oracle_heads)
    sub = lambda t: _host(t)[hs]
    oq, ok_, ov = oracle_mod.fine_bwd(sub(q), sub(k), sub(v), sub(dof), idx.cpu().numpy()[hs],
                                      cnt.cpu().numpy()[hs], d ** -0.5)
    for name, a, r in zip(("dq", "dk", "dv"), got, (oq, ok_, ov)):
        assert_close(sub(a), r, what=f"{name} vs oracle (heads {hs}, d={d}, seed {seed})")


def test_noalloc_matches_oracle_and_workspace_call_twice(lib, oracle_mod):
    """Two calls in a row on different data: the second finds the first one's
    contents in the shared array."""
    for seed in (11, 23):
        _check(lib, oracle_mod, 3, 4096, 128, 16, seed, oracle_heads=range(3))


def test_noalloc_head_dim_64(lib, oracle_mod):
    _check(lib, oracle_mod, 4, 2048, 64, 8, 31, oracle_heads=range(4))


def _limit_heads(lib, N, d, K):
    """The largest BH whose scratch fits the fixed array at (N, d, K)."""
    L = lib.load()
    need = lambda bh: L.vsa_workspace_bytes(lib.VSA_OP_FINE_BWD, 1, bh, d, lib.Grid.of(4, 4, N // 16), K, -1)
    bh = 1
    while need(bh + 1) <= lib.VSA_NOALLOC_SCRATCH_BYTES:
        bh += 1
    assert need(bh) <= lib.VSA_NOALLOC_SCRATCH_BYTES < need(bh + 1)
    return bh


def test_noalloc_at_the_largest_problem_it_holds(lib, oracle_mod):
    bh = _limit_heads(lib, 4096, 128, 16)
    assert bh >= 12                                 # 12 heads of 4096 tokens fit, as the header says
    _check(lib, oracle_mod, bh, 4096, 128, 16, 47, oracle_heads=(0, bh - 1))


def test_noalloc_refuses_one_head_more(lib):
    bh = _limit_heads(lib, 4096, 128, 16) + 1
    fake = ctypes.c_void_p(1 << 20)                 # never touched: the size check comes first
    st = lib.load().vsa_fine_bwd_noalloc(fake, fake, fake, fake, lib.VSA_DTYPE_F32, fake, fake, fake, None, 16, bh,
                                         4096, 128, 0.088, fake, fake, fake, None)
    assert st == lib.VSA_ERR_WORKSPACE
    st = lib.load().vsa_fine_bwd_noalloc(fake, fake, fake, fake, lib.VSA_DTYPE_F32, fake, fake, fake, None, 16, 40,
                                         32768, 128, 0.088, fake, fake, fake, None)
    assert st == lib.VSA_ERR_WORKSPACE
