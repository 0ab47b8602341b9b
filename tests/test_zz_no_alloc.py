"""vsa_fine_bwd_noalloc: the fine backward for callers that cannot give the
library scratch memory (code inside a runtime that hands out device memory
only through its own pool, or plain C callers without an allocator).  It must
give the same gradients as vsa_fine_bwd, call after call, with its scratch
held in the library's fixed device array, and must refuse problems larger
than that array.  Called through the C ABI."""
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


def _case(seed, heads):
    wl = synth.WORKLOADS["small"]
    rng = np.random.default_rng(seed)
    q, k, v = (synth.make_random((len(heads), wl.N, wl.d), seed=seed + i) for i in range(3))
    idx = np.stack([np.stack([rng.permutation(wl.Nc)[:wl.topk] for _ in range(wl.Nc)])
                    for _ in heads]).astype(np.int32)
    cnt = np.full(idx.shape[:-1], wl.topk, np.int32)
    cnt[0, 5] = 3
    dof = synth.make_random(q.shape, seed=seed + 9)
    D = lambda a, t=torch.bfloat16: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(t).contiguous()
    return wl, D(q), D(k), D(v), D(dof), D(idx, torch.int32), D(cnt, torch.int32)


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point_twice(lib):
    import block_sparse_video_sfc_gb300 as vsa
    L = lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, seed in enumerate((11, 23)):            # two calls in a row, different data
        wl, q, k, v, dof, idx, cnt = _case(seed, heads=[0, 1, 2])
        BH = q.shape[0]
        of, lse = vsa.fine_fwd(q, k, v, idx, cnt)
        ref = vsa.fine_bwd(q, k, v, of, lse, dof, idx, cnt)
        dq, dk, dv = (torch.full_like(ref[0], float("nan")) for _ in range(3))
        st = L.vsa_fine_bwd_noalloc(_p(q), _p(k), _p(v), _p(of), lib.VSA_DTYPE_F32, _p(lse), _p(dof), _p(idx),
                                    _p(cnt), idx.shape[-1], BH, wl.N, wl.d, wl.d ** -0.5, _p(dq), _p(dk), _p(dv),
                                    stream)
        assert st == lib.VSA_OK, st
        torch.cuda.synchronize()
        assert vsa.device_status() == 0
        for name, a, b in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
            assert_close(a.cpu().numpy(), b.cpu().numpy(), what=f"{name} call {call}")


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    L = lib.load()
    fake = ctypes.c_void_p(1 << 20)   # never touched: the size check comes first
    st = L.vsa_fine_bwd_noalloc(fake, fake, fake, fake, lib.VSA_DTYPE_F32, fake, fake, fake, None, 16, 40, 32768,
                                128, 0.088, fake, fake, fake, None)
    assert st == lib.VSA_ERR_WORKSPACE
