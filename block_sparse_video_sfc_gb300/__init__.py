"""GB300 (sm_103a) implementation of VSA, the trainable coarse-to-fine
block-sparse attention for video diffusion transformers.

All compute runs in libvsa.so (hand-written CUDA: SFC reorder + cube pool,
coarse attention + Top-K, tcgen05 fine attention forward and backward).  This
module only allocates torch device tensors and passes pointers and the current
stream through the C ABI of include/vsa.h.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib
from ._lib import Grid, VSAError, VSA_DTYPE_BF16, VSA_DTYPE_F32

__all__ = ["num_cubes", "cube_order", "permute", "coarse_topk", "fine_fwd", "fine_bwd", "forward", "forward_inference", "backward",
           "backward_tile_pairs",
           "workspace_bytes", "device_status", "timing_enable", "timing_read", "VSAError",
           "ForwardState", "Grid"]

_DT = {torch.bfloat16: VSA_DTYPE_BF16, torch.float32: VSA_DTYPE_F32}


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libvsa takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libvsa takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _bhnd(x: torch.Tensor):
    if x.dim() == 4:
        return x.shape[0] * x.shape[1], x.shape[2], x.shape[3]
    if x.dim() == 3:
        return tuple(x.shape)
    raise ValueError("expected [B, heads, N, d] or [BH, N, d]")


def num_cubes(T: int, H: int, W: int) -> int:
    """Cubes of (4, 4, 4) covering a (T, H, W) grid (partial ones included)."""
    return ((T + 3) // 4) * ((H + 3) // 4) * ((W + 3) // 4)


def cube_order(T: int, H: int, W: int, curve: str = "hilbert", device="cuda") -> torch.Tensor:
    """vsa_cube_order: int32 [2 * Nc] table (position -> raster cube id, then
    raster cube id -> position) for curve "raster" or "hilbert"."""
    Nc = num_cubes(T, H, W)
    order = torch.empty(2 * Nc, dtype=torch.int32, device=device)
    code = {"raster": _lib.VSA_CURVE_RASTER, "hilbert": _lib.VSA_CURVE_HILBERT}[curve]
    _lib.check("vsa_cube_order", _lib.load().vsa_cube_order(Grid.of(T, H, W), code, _ptr(order), _stream()))
    return order


def permute(x: torch.Tensor, T: int, H: int, W: int, inverse: bool = False, pool: bool = False,
            cube_order=None):
    """vsa_permute: native [.., T*H*W, d] <-> cube order [.., 64*Nc, d] (a grid
    side that is not a multiple of 4 ends in partial cubes whose padding slots
    are zero); with pool=True also the cube means [.., Nc, d]."""
    BH, N, d = _bhnd(x)
    Nc = num_cubes(T, H, W)
    y = torch.empty(x.shape[:-2] + ((T * H * W) if inverse else 64 * Nc, d), dtype=x.dtype, device=x.device)
    pooled = None
    if pool:
        pooled = torch.empty(x.shape[:-2] + (Nc, d), dtype=torch.float32, device=x.device)
    _lib.check("vsa_permute", _lib.load().vsa_permute(_ptr(x), _ptr(y), _ptr(pooled), BH, d,
                                                       Grid.of(T, H, W, _ptr(cube_order)), int(inverse),
                                                       _stream()))
    return (y, pooled) if pool else y


def coarse_topk(qc, kc, vc, topk: int, scale: Optional[float] = None, want_oc: bool = True,
                want_scores: bool = False):
    """vsa_coarse_topk -> dict(idx, cnt, oc, lse_c, scores)."""
    BH, Nc, d = _bhnd(qc)
    scale = d ** -0.5 if scale is None else scale
    lead = qc.shape[:-2]
    dev = qc.device
    idx = torch.empty(lead + (Nc, topk), dtype=torch.int32, device=dev)
    cnt = torch.empty(lead + (Nc,), dtype=torch.int32, device=dev)
    oc = torch.empty_like(qc) if want_oc else None
    lse_c = torch.empty(lead + (Nc,), dtype=torch.float32, device=dev)
    scores = torch.empty(lead + (Nc, Nc), dtype=torch.float32, device=dev) if want_scores else None
    _lib.check("vsa_coarse_topk", _lib.load().vsa_coarse_topk(
        _ptr(qc), _ptr(kc), _ptr(vc if want_oc else None), BH, Nc, d, topk, float(scale), _ptr(oc),
        _ptr(lse_c), _ptr(idx), _ptr(cnt), _ptr(scores), _stream()))
    return dict(idx=idx, cnt=cnt, oc=oc, lse_c=lse_c, scores=scores)


def mask_to_lut(mask, max_kv_blocks: int):
    """vsa_mask_to_lut: uint8/bool block matrix [.., Nc, Nc] -> (idx [.., Nc, max_kv_blocks], cnt [.., Nc])."""
    mask = mask.to(torch.uint8).contiguous()
    Nc = mask.shape[-1]
    BH = mask.numel() // (Nc * Nc)
    lead = mask.shape[:-2]
    idx = torch.empty(lead + (Nc, max_kv_blocks), dtype=torch.int32, device=mask.device)
    cnt = torch.empty(lead + (Nc,), dtype=torch.int32, device=mask.device)
    _lib.check("vsa_mask_to_lut", _lib.load().vsa_mask_to_lut(
        _ptr(mask), BH, Nc, max_kv_blocks, _ptr(idx), _ptr(cnt), _stream()))
    return idx, cnt


def lut_add_neighbors(idx, cnt, T: int, H: int, W: int, radius: int, max_kv_blocks: int, cube_order=None):
    """vsa_lut_add_neighbors: list united with the radius-r cube neighbourhood -> (idx, cnt)."""
    Nc, kin = idx.shape[-2], idx.shape[-1]
    BH = idx.numel() // (Nc * kin)
    lead = idx.shape[:-2]
    out = torch.empty(lead + (Nc, max_kv_blocks), dtype=torch.int32, device=idx.device)
    ocnt = torch.empty(lead + (Nc,), dtype=torch.int32, device=idx.device)
    _lib.check("vsa_lut_add_neighbors", _lib.load().vsa_lut_add_neighbors(
        _ptr(idx), _ptr(cnt), kin, BH, Grid.of(T, H, W, _ptr(cube_order)), radius, max_kv_blocks, _ptr(out),
        _ptr(ocnt),
        _stream()))
    return out, ocnt


def fine_fwd(qp, kp, vp, idx, cnt, scale: Optional[float] = None, out_dtype=torch.float32, workspace: bool = True):
    """vsa_fine_fwd on cube-ordered bf16 tensors -> (O_f, lse).  workspace:
    give the call its workspace (fp16 copies and the overlap pair plan);
    False runs the allocation-free form."""
    BH, N, d = _bhnd(qp)
    scale = d ** -0.5 if scale is None else scale
    of = torch.empty(qp.shape, dtype=out_dtype, device=qp.device)
    lse = torch.empty(qp.shape[:-1], dtype=torch.float32, device=qp.device)
    kmax = idx.shape[-1] if idx is not None else 0
    nbytes = 0
    if workspace and N % 64 == 0:
        nbytes = workspace_bytes(_lib.VSA_OP_FINE_FWD, 1, BH, d, 4, 4, N // 16, max(kmax, 1))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=qp.device) if nbytes else None
    _lib.check("vsa_fine_fwd", _lib.load().vsa_fine_fwd(
        _ptr(qp), _ptr(kp), _ptr(vp), _ptr(idx), _ptr(cnt), kmax, BH, N, d, float(scale),
        _ptr(of), _DT[out_dtype], _ptr(lse), _ptr(ws), nbytes, _stream()))
    return of, lse


def workspace_bytes(op: int, B: int, heads: int, d: int, T: int, H: int, W: int, topk: int, radius: int = -1) -> int:
    return int(_lib.load().vsa_workspace_bytes(op, B, heads, d, Grid.of(T, H, W), topk, radius))


def fine_bwd(qp, kp, vp, of, lse, dof, idx, cnt, scale: Optional[float] = None):
    """vsa_fine_bwd -> (dq, dk, dv) fp32, cube order."""
    BH, N, d = _bhnd(qp)
    scale = d ** -0.5 if scale is None else scale
    kmax = idx.shape[-1]
    nbytes = workspace_bytes(_lib.VSA_OP_FINE_BWD, 1, BH, d, 4, 4, N // 16, kmax) if N % 64 == 0 else 0
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=qp.device)
    dq = torch.empty(qp.shape, dtype=torch.float32, device=qp.device)
    dk = torch.empty_like(dq)
    dv = torch.empty_like(dq)
    _lib.check("vsa_fine_bwd", _lib.load().vsa_fine_bwd(
        _ptr(qp), _ptr(kp), _ptr(vp), _ptr(of), _DT[of.dtype], _ptr(lse), _ptr(dof), _ptr(idx), _ptr(cnt),
        kmax, BH, N, d, float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), nbytes, _stream()))
    return dq, dk, dv


@dataclass
class ForwardState:
    """The saved state of one forward call (lives in `ws`)."""

    ws: torch.Tensor
    B: int
    heads: int
    d: int
    T: int
    H: int
    W: int
    topk: int
    scale: float
    cube_order: Optional[torch.Tensor] = None
    radius: int = -1

    def saved(self) -> dict:
        """Views of the saved intermediates as torch tensors."""
        s = _lib.Saved()
        _lib.check("vsa_forward_saved", _lib.load().vsa_forward_saved(
            _ptr(self.ws), self.B, self.heads, self.d, Grid.of(self.T, self.H, self.W), self.topk, self.radius,
            ctypes.byref(s)))
        BH, d, K = self.B * self.heads, self.d, s.max_kv_blocks
        Nc = num_cubes(self.T, self.H, self.W)
        N = 64 * Nc  # reordered length (padding slots included)
        base = self.ws.data_ptr()

        def view(ptr, shape, dtype):
            esize = torch.empty((), dtype=dtype).element_size()
            off = ptr - base
            n = 1
            for x in shape:
                n *= x
            return self.ws[off:off + n * esize].view(dtype).view(shape)

        return dict(
            qp=view(s.qp, (BH, N, d), torch.float16), kp=view(s.kp, (BH, N, d), torch.float16),
            vp=view(s.vp, (BH, N, d), torch.float16), qc=view(s.qc, (BH, Nc, d), torch.float32),
            kc=view(s.kc, (BH, Nc, d), torch.float32), vc=view(s.vc, (BH, Nc, d), torch.float32),
            oc=view(s.o_coarse, (BH, Nc, d), torch.float32),
            lse_c=view(s.lse_coarse, (BH, Nc), torch.float32),
            idx=view(s.kv_block_idx, (BH, Nc, K), torch.int32),
            cnt=view(s.valid_block_num, (BH, Nc), torch.int32),
            of=view(s.o_fine, (BH, N, d), torch.float32), lse=view(s.lse, (BH, N), torch.float32),
            tile_pairs=view(s.tile_pairs, (BH, (Nc + 1) // 2, 2), torch.int32))


def forward(q, k, v, T: int, H: int, W: int, topk: int, g_coarse=None, g_fine=None,
            scale: Optional[float] = None, out_dtype=torch.bfloat16, out=None, ws=None, cube_order=None,
            radius: int = -1):
    """vsa_forward on native-order [B, heads, N, d] bf16 -> (out, ForwardState).
    radius >= 0 unites each Top-K list with the radius-r cube neighbourhood."""
    B, heads, N, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    nbytes = workspace_bytes(_lib.VSA_OP_FORWARD, B, heads, d, T, H, W, topk, radius)
    if nbytes == 0:
        raise VSAError("vsa_workspace_bytes", _lib.VSA_ERR_ARG)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    _lib.check("vsa_forward", _lib.load().vsa_forward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g_coarse), _ptr(g_fine), B, heads, d, Grid.of(T, H, W, _ptr(cube_order)), topk,
        radius, float(scale), _ptr(out), _DT[out.dtype], _ptr(ws), nbytes, _stream()))
    return out, ForwardState(ws, B, heads, d, T, H, W, topk, scale, cube_order, radius)


def forward_inference(q, k, v, T: int, H: int, W: int, topk: int, g_coarse=None, g_fine=None,
                      scale: Optional[float] = None, out_dtype=torch.bfloat16, out=None, ws=None, cube_order=None,
                      radius: int = -1):
    """vsa_forward_inference: the forward output without saved state; the fine
    stage reads Q, K, V in their native layout (no reordered copies)."""
    B, heads, N, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    nbytes = workspace_bytes(_lib.VSA_OP_FORWARD_INFERENCE, B, heads, d, T, H, W, topk, radius)
    if nbytes == 0:
        raise VSAError("vsa_workspace_bytes", _lib.VSA_ERR_ARG)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    _lib.check("vsa_forward_inference", _lib.load().vsa_forward_inference(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g_coarse), _ptr(g_fine), B, heads, d, Grid.of(T, H, W, _ptr(cube_order)),
        topk, radius, float(scale), _ptr(out), _DT[out.dtype], _ptr(ws), nbytes, _stream()))
    return out


def backward(state: ForwardState, dout, g_coarse=None, g_fine=None, grad_dtype=torch.float32,
             grads=None, ws=None):
    """vsa_backward -> dict(dq, dk, dv, dgc, dgf) in native order."""
    B, heads, d = state.B, state.heads, state.d
    nbytes = workspace_bytes(_lib.VSA_OP_BACKWARD, B, heads, d, state.T, state.H, state.W, state.topk, state.radius)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dout.device)
    if grads is None:
        mk = lambda: torch.empty(dout.shape, dtype=grad_dtype, device=dout.device)
        grads = dict(dq=mk(), dk=mk(), dv=mk(), dgc=mk() if g_coarse is not None else None,
                     dgf=mk() if g_fine is not None else None)
    dt = grads["dq"].dtype
    _lib.check("vsa_backward", _lib.load().vsa_backward(
        _ptr(state.ws), _ptr(g_coarse), _ptr(g_fine), _ptr(dout), B, heads, d,
        Grid.of(state.T, state.H, state.W, _ptr(state.cube_order)), state.topk, state.radius, float(state.scale),
        _ptr(grads["dq"]),
        _ptr(grads["dk"]), _ptr(grads["dv"]), _ptr(grads.get("dgc")), _ptr(grads.get("dgf")), _DT[dt],
        _ptr(ws), nbytes, _stream()))
    return grads


def backward_tile_pairs(state: ForwardState, ws: torch.Tensor) -> torch.Tensor:
    """vsa_backward_tile_pairs: view of the key-cube pairs [BH, (Nc + 1) // 2, 2]
    that the dK/dV kernel's tiles used in the backward call made with `ws`."""
    ptr = ctypes.c_void_p()
    _lib.check("vsa_backward_tile_pairs", _lib.load().vsa_backward_tile_pairs(
        _ptr(ws), state.B, state.heads, state.d, Grid.of(state.T, state.H, state.W), state.topk, state.radius,
        ctypes.byref(ptr)))
    Nc = num_cubes(state.T, state.H, state.W)
    n = state.B * state.heads * ((Nc + 1) // 2) * 2
    off = ptr.value - ws.data_ptr()
    return ws[off:off + 4 * n].view(torch.int32).view(state.B * state.heads, (Nc + 1) // 2, 2)


def timing_enable(on: bool = True) -> None:
    """Bracket each main-kernel launch with CUDA events (vsa_timing_enable)."""
    _lib.check("vsa_timing_enable", _lib.load().vsa_timing_enable(int(on)))


def timing_read() -> dict:
    """{kernel: (total_ms, launches)} since the last read (vsa_timing_read)."""
    out = {}
    for i, name in enumerate(_lib.KERNELS):
        ms, n = ctypes.c_double(), ctypes.c_int()
        _lib.check("vsa_timing_read", _lib.load().vsa_timing_read(i, ctypes.byref(ms), ctypes.byref(n)))
        out[name] = (ms.value, n.value)
    return out


def selftest_wait_timeout(polls: int = 1 << 16) -> None:
    """Runs the bounded-wait failure path once (vsa_selftest_wait_timeout);
    device_status() then reports VSA_ERR_TIMEOUT."""
    _lib.check("vsa_selftest_wait_timeout", _lib.load().vsa_selftest_wait_timeout(polls, _stream()))


def device_status() -> int:
    """Waits for the current stream; returns and clears the device error word."""
    return int(_lib.load().vsa_device_status(_stream()))
