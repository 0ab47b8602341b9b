"""CPU oracle for VSA (Video Sparse Attention): a plain, slow float64 restatement
of the method, used only to check the CUDA library.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg import this package.  The arithmetic lives in
``vsa_oracle.c`` (plain loops, float64); this module only builds it with gcc
and marshals numpy arrays through ctypes.  It shares no code with the CUDA
library and never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vsa_oracle.c")
_LIB = os.path.join(_HERE, "libvsa_oracle.so")
_lock = threading.Lock()
_lib = None

CUBE = 64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            D = ctypes.c_double
            sig = {
                "orc_hilbert_point": ([ctypes.c_uint64, I, P], None),
                "orc_cube_rank": ([I, I, I, I, P], None),
                "orc_sfc_position": ([I, I, I, I, I, I, P], I64),
                "orc_sfc_table": ([I, I, I, P, P], None),
                "orc_permute": ([P, P, I64, I, I, I, I, P, I], None),
                "orc_num_cubes": ([I, I, I], I64),
                "orc_cube_slots": ([I, I, I, P, P, P], None),
                "orc_pool": ([P, P, I64, I64, I, P], None),
                "orc_coarse": ([P, P, P, I64, I, I, D, P, P, P], None),
                "orc_topk": ([P, I64, I, I, P], None),
                "orc_fine_fwd": ([P, P, P, P, P, I, I64, I64, I, D, P, P, P], None),
                "orc_fine_fwd_rows": ([P, P, P, P, P, I, I64, I64, I, D, P, P, I64, P, P], None),
                "orc_combine": ([P, P, P, P, I64, I64, I, P], None),
                "orc_forward": ([P, P, P, P, P, I64, I, I, I, I, P, I, I, I, D, P, P, P, P, P, P, P, P, P], None),
                "orc_fine_bwd": ([P, P, P, P, P, P, I, I64, I64, I, D, P, P, P, P], None),
                "orc_coarse_bwd": ([P, P, P, P, I64, I, I, D, P, P, P], None),
                "orc_backward": ([P, P, P, P, P, I64, I, I, I, I, P, I, D, P, P, P, P, P, P, P, P], None),
                "orc_fine_bwd_query_rows": ([P, P, P, P, P, P, I, I64, I, D, P, P, I64, P], None),
                "orc_fine_bwd_key_cube": ([P, P, P, P, P, P, I, I64, I, D, P, I64, I, P, P], None),
                "orc_combine_bwd": ([P, P, P, P, P, I64, I64, I, P, P, P, P], None),
                "orc_mask_to_lut": ([P, I64, I, I, P, P, P], None),
                "orc_lut_add_neighbors": ([P, P, I, I64, I, I, I, P, I, I, P, P, P], None),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def _f64(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float64)


def _i32(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.int32)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bh(x):
    """[B, heads, N, d] or [BH, N, d] -> (BH, N, d)."""
    if x.ndim == 4:
        return x.shape[0] * x.shape[1], x.shape[2], x.shape[3]
    return x.shape


def default_scale(d: int) -> float:
    return 1.0 / np.sqrt(d)


CURVES = {"raster": 0, "hilbert": 1}


def hilbert_point(hidx: int, b: int):
    """(t, h, w) of index hidx on the order-b 3-D Hilbert curve."""
    x = np.zeros(3, dtype=np.uint32)
    _load().orc_hilbert_point(hidx, b, _p(x))
    return tuple(int(v) for v in x)


def cube_rank(Tc: int, Hc: int, Wc: int, curve: str = "raster") -> np.ndarray:
    """rank[raster cube id] = the cube's position in the cube sequence."""
    rank = np.empty(Tc * Hc * Wc, dtype=np.int32)
    _load().orc_cube_rank(Tc, Hc, Wc, CURVES[curve], _p(rank))
    return rank


def cube_grid(T: int, H: int, W: int):
    """Cubes along t, h, w: a side that is not a multiple of 4 ends in partial cubes."""
    return (T + 3) // 4, (H + 3) // 4, (W + 3) // 4


def num_cubes(T: int, H: int, W: int) -> int:
    return int(_load().orc_num_cubes(T, H, W))


def _rank_of(T: int, H: int, W: int, curve: str):
    return None if curve == "raster" else cube_rank(*cube_grid(T, H, W), curve)


def cube_slots(T: int, H: int, W: int, curve: str = "raster"):
    """(slot_ok [Np] uint8: reordered slot holds a token, ntok [Nc] int32: tokens per cube)."""
    Nc = num_cubes(T, H, W)
    slot_ok = np.empty(64 * Nc, dtype=np.uint8)
    ntok = np.empty(Nc, dtype=np.int32)
    _load().orc_cube_slots(T, H, W, _p(_rank_of(T, H, W, curve)), _p(slot_ok), _p(ntok))
    return slot_ok, ntok


def sfc_table(T: int, H: int, W: int, curve: str = "raster") -> np.ndarray:
    """pos[n]: reordered position of native token n = (t*H + h)*W + w."""
    pos = np.empty(T * H * W, dtype=np.int64)
    _load().orc_sfc_table(T, H, W, _p(_rank_of(T, H, W, curve)), _p(pos))
    return pos


def permute(x, T: int, H: int, W: int, inverse: bool = False, curve: str = "raster") -> np.ndarray:
    """Native [.., N, d] -> reordered [.., Np, d] (padding slots zero), or back."""
    x = _f64(x)
    BH, N, d = _bh(x)
    n_out = T * H * W if inverse else 64 * num_cubes(T, H, W)
    y = np.empty(x.shape[:-2] + (n_out, d), dtype=np.float64)
    rank = _rank_of(T, H, W, curve)
    _load().orc_permute(_p(x), _p(y), BH, d, T, H, W, _p(rank), int(bool(inverse)))
    return y


def pool(xp, ntok=None) -> np.ndarray:
    """Cube means; ntok (tokens per cube, default 64) divides each sum."""
    xp = _f64(xp)
    BH, N, d = _bh(xp)
    out = np.empty(xp.shape[:-2] + (N // CUBE, d), dtype=np.float64)
    _load().orc_pool(_p(xp), _p(out), BH, N, d, _p(_i32(ntok)))
    return out


def coarse(qc, kc, vc, scale: float):
    """-> (scores [.., Nc, Nc], O_c [.., Nc, d], lse_c [.., Nc])."""
    qc, kc, vc = _f64(qc), _f64(kc), _f64(vc)
    BH, Nc, d = _bh(qc)
    scores = np.empty(qc.shape[:-1] + (Nc,), dtype=np.float64)
    oc = np.empty_like(qc)
    lse = np.empty(qc.shape[:-1], dtype=np.float64)
    _load().orc_coarse(_p(qc), _p(kc), _p(vc), BH, Nc, d, float(scale),
                       _p(scores), _p(oc), _p(lse))
    return scores, oc, lse


def topk(scores, K: int) -> np.ndarray:
    """Index list [.., Nc, K], highest score first, ties to the lower id."""
    scores = _f64(scores)
    Nc = scores.shape[-1]
    rows = int(np.prod(scores.shape[:-1]))
    if not 1 <= K <= Nc:
        raise ValueError(f"K={K} outside [1, {Nc}]")
    idx = np.empty(scores.shape[:-1] + (K,), dtype=np.int32)
    _load().orc_topk(_p(scores), rows, Nc, K, _p(idx))
    return idx


def _u8(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.uint8)


def fine_fwd(qp, kp, vp, idx, cnt, scale: float, slot_ok=None):
    """-> (O_f [.., N, d], lse [.., N]) over the listed cubes only."""
    qp, kp, vp = _f64(qp), _f64(kp), _f64(vp)
    idx, cnt = _i32(idx), _i32(cnt)
    BH, N, d = _bh(qp)
    of = np.empty_like(qp)
    lse = np.empty(qp.shape[:-1], dtype=np.float64)
    _load().orc_fine_fwd(_p(qp), _p(kp), _p(vp), _p(idx), _p(cnt), idx.shape[-1], BH, N, d,
                         float(scale), _p(_u8(slot_ok)), _p(of), _p(lse))
    return of, lse


def fine_fwd_rows(qp, kp, vp, idx, cnt, scale: float, rows, slot_ok=None):
    """Fine output for the listed flat rows r = bh*N + i only."""
    qp, kp, vp = _f64(qp), _f64(kp), _f64(vp)
    idx, cnt = _i32(idx), _i32(cnt)
    BH, N, d = _bh(qp)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    of = np.empty((rows.size, d), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    _load().orc_fine_fwd_rows(_p(qp), _p(kp), _p(vp), _p(idx), _p(cnt), idx.shape[-1],
                              BH, N, d, float(scale), _p(_u8(slot_ok)), _p(rows), rows.size, _p(of), _p(lse))
    return of, lse


def combine(gc, gf, oc, of) -> np.ndarray:
    """Reordered-order output g_c*O_c[cube] + g_f*O_f (None gate = ones)."""
    oc, of = _f64(oc), _f64(of)
    gc, gf = _f64(gc), _f64(gf)
    BH, N, d = _bh(of)
    out = np.empty_like(of)
    _load().orc_combine(_p(gc), _p(gf), _p(oc), _p(of), BH, N, d, _p(out))
    return out


def list_width(K: int, radius: int, Nc: int) -> int:
    """Width of the selection lists: K for a pure Top-K (radius < 0); with the
    radius-r neighbourhood added, room for K + (2r + 1)^3 cubes (at most Nc)."""
    return K if radius < 0 else min(Nc, K + (2 * radius + 1) ** 3)


def forward(q, k, v, T: int, H: int, W: int, K: int, scale=None,
            gc=None, gf=None, lut=None, want_scores: bool = True, curve: str = "raster",
            radius: int = -1, cnt=None):
    """Whole forward pass (native order in/out).

    The selection: lut [.., Nc, kmax] with counts cnt (None: every row full)
    if given; otherwise the Top-K of the coarse scores, united with the
    radius-r cube neighbourhood when radius >= 0 (ascending lists).
    Returns a dict with out, idx, cnt, of, lse, oc and scores.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    gc, gf = _f64(gc), _f64(gf)
    BH, N, d = _bh(q)
    assert N == T * H * W
    Nc = num_cubes(T, H, W)
    if scale is None:
        scale = default_scale(d)
    lead = q.shape[:-2]
    out = np.empty_like(q)
    kmax = np.asarray(lut).shape[-1] if lut is not None else list_width(K, radius, Nc)
    idx = np.empty(lead + (Nc, kmax), dtype=np.int32)
    cnt_out = np.empty(lead + (Nc,), dtype=np.int32)
    of = np.empty(lead + (64 * Nc, d), dtype=np.float64)
    lse = np.empty(lead + (64 * Nc,), dtype=np.float64)
    oc = np.empty(lead + (Nc, d), dtype=np.float64)
    scores = np.empty(lead + (Nc, Nc), dtype=np.float64) if want_scores else None
    lut = _i32(lut)
    cnt = None if cnt is None or lut is None else _i32(cnt)
    rank = _rank_of(T, H, W, curve)
    _load().orc_forward(_p(q), _p(k), _p(v), _p(gc), _p(gf), BH, d, T, H, W, _p(rank), K, radius, kmax,
                        float(scale), _p(lut), _p(cnt), _p(out), _p(idx), _p(cnt_out), _p(of), _p(lse),
                        _p(oc), _p(scores))
    return dict(out=out, idx=idx, cnt=cnt_out, of=of, lse=lse, oc=oc, scores=scores)


def fine_bwd(qp, kp, vp, dof, idx, cnt, scale: float, slot_ok=None):
    qp, kp, vp, dof = _f64(qp), _f64(kp), _f64(vp), _f64(dof)
    idx, cnt = _i32(idx), _i32(cnt)
    BH, N, d = _bh(qp)
    dq, dk, dv = np.empty_like(qp), np.empty_like(qp), np.empty_like(qp)
    _load().orc_fine_bwd(_p(qp), _p(kp), _p(vp), _p(dof), _p(idx), _p(cnt), idx.shape[-1],
                         BH, N, d, float(scale), _p(_u8(slot_ok)), _p(dq), _p(dk), _p(dv))
    return dq, dk, dv


def fine_bwd_query_rows(qp, kp, vp, dof, idx, cnt, scale: float, rows, slot_ok=None):
    """dQ of the fine stage for the listed flat rows r = bh*N + i."""
    qp, kp, vp, dof = _f64(qp), _f64(kp), _f64(vp), _f64(dof)
    idx, cnt = _i32(idx), _i32(cnt)
    BH, N, d = _bh(qp)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, d), dtype=np.float64)
    _load().orc_fine_bwd_query_rows(_p(qp), _p(kp), _p(vp), _p(dof), _p(idx), _p(cnt), idx.shape[-1],
                                    N, d, float(scale), _p(_u8(slot_ok)), _p(rows), rows.size, _p(out))
    return out


def fine_bwd_key_cube(qp, kp, vp, dof, idx, cnt, scale: float, bh: int, kcube: int, slot_ok=None):
    """(dK, dV) of the 64 tokens of key cube `kcube` in head `bh`, fine stage."""
    qp, kp, vp, dof = _f64(qp), _f64(kp), _f64(vp), _f64(dof)
    idx, cnt = _i32(idx), _i32(cnt)
    BH, N, d = _bh(qp)
    dk = np.empty((64, d), dtype=np.float64)
    dv = np.empty((64, d), dtype=np.float64)
    _load().orc_fine_bwd_key_cube(_p(qp), _p(kp), _p(vp), _p(dof), _p(idx), _p(cnt), idx.shape[-1],
                                  N, d, float(scale), _p(_u8(slot_ok)), bh, kcube, _p(dk), _p(dv))
    return dk, dv


def combine_bwd(dout_p, gc_p, gf_p, oc, of):
    """Backward of the gated combination (reordered order) -> dof, doc, dgc, dgf."""
    dout_p, oc, of = _f64(dout_p), _f64(oc), _f64(of)
    gc_p, gf_p = _f64(gc_p), _f64(gf_p)
    BH, N, d = _bh(of)
    dof, dgc, dgf = np.empty_like(of), np.empty_like(of), np.empty_like(of)
    doc = np.empty_like(oc)
    _load().orc_combine_bwd(_p(dout_p), _p(gc_p), _p(gf_p), _p(oc), _p(of), BH, N, d,
                            _p(dof), _p(doc), _p(dgc), _p(dgf))
    return dof, doc, dgc, dgf


def coarse_bwd(qc, kc, vc, doc, scale: float):
    qc, kc, vc, doc = _f64(qc), _f64(kc), _f64(vc), _f64(doc)
    BH, Nc, d = _bh(qc)
    dq, dk, dv = np.empty_like(qc), np.empty_like(qc), np.empty_like(qc)
    _load().orc_coarse_bwd(_p(qc), _p(kc), _p(vc), _p(doc), BH, Nc, d, float(scale),
                           _p(dq), _p(dk), _p(dv))
    return dq, dk, dv


def backward(q, k, v, dout, idx, T: int, H: int, W: int, scale=None,
             gc=None, gf=None, curve: str = "raster", cnt=None):
    """Whole backward pass for the lists idx [.., Nc, kmax] (counts cnt; None:
    every row full); returns dict dq, dk, dv, dgc, dgf (native order)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    gc, gf = _f64(gc), _f64(gf)
    idx = _i32(idx)
    cnt = None if cnt is None else _i32(cnt)
    BH, N, d = _bh(q)
    K = idx.shape[-1]
    if scale is None:
        scale = default_scale(d)
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    dgc = np.empty_like(q) if gc is not None else None
    dgf = np.empty_like(q) if gf is not None else None
    rank = _rank_of(T, H, W, curve)
    _load().orc_backward(_p(q), _p(k), _p(v), _p(gc), _p(gf), BH, d, T, H, W, _p(rank), K,
                         float(scale), _p(idx), _p(cnt), _p(dout), _p(dq), _p(dk), _p(dv),
                         _p(dgc), _p(dgf))
    return dict(dq=dq, dk=dk, dv=dv, dgc=dgc, dgf=dgf)


def mask_to_lut(mask, max_kv_blocks: int):
    """Block relation matrix [.., Nc, Nc] (nonzero = keep) -> (idx, cnt, overflow)."""
    m = np.ascontiguousarray(np.asarray(mask) != 0, dtype=np.uint8)
    Nc = m.shape[-1]
    rows = m.size // Nc
    idx = np.empty(m.shape[:-1] + (max_kv_blocks,), dtype=np.int32)
    cnt = np.empty(m.shape[:-1], dtype=np.int32)
    ovf = ctypes.c_int(0)
    _load().orc_mask_to_lut(m.ctypes.data_as(ctypes.c_void_p), rows, Nc, max_kv_blocks, _p(idx), _p(cnt),
                            ctypes.byref(ovf))
    return idx, cnt, bool(ovf.value)


def lut_add_neighbors(idx, cnt, T: int, H: int, W: int, radius: int, max_kv_blocks: int,
                      curve: str = "raster"):
    """Lists united with the radius-r cube neighbourhood -> (idx, cnt, overflow)."""
    idx = _i32(idx)
    cnt = None if cnt is None else _i32(cnt)
    Tc, Hc, Wc = cube_grid(T, H, W)
    Nc, kin = idx.shape[-2], idx.shape[-1]
    BH = idx.size // (Nc * kin)
    out = np.empty(idx.shape[:-1] + (max_kv_blocks,), dtype=np.int32)
    ocnt = np.empty(idx.shape[:-1], dtype=np.int32)
    ovf = ctypes.c_int(0)
    rank = _rank_of(T, H, W, curve)
    _load().orc_lut_add_neighbors(_p(idx), _p(cnt), kin, BH, Tc, Hc, Wc, _p(rank), radius, max_kv_blocks, _p(out),
                                  _p(ocnt),
                                  ctypes.byref(ovf))
    return out, ocnt, bool(ovf.value)
