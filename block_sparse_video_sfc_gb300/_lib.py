"""ctypes view of libvsa.so (declared in include/vsa.h).

Loading fails loudly when the library has not been built: there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libvsa.so")

VSA_OK = 0
VSA_ERR_ARG = -1
VSA_ERR_SHAPE = -2
VSA_ERR_UNSUPPORTED = -3
VSA_ERR_CUDA = -4
VSA_ERR_TIMEOUT = -5
VSA_ERR_LUT = -6
VSA_ERR_WORKSPACE = -7
VSA_ERR_RANGE = -8

VSA_DTYPE_BF16 = 0
VSA_DTYPE_F32 = 1

VSA_OP_FORWARD = 0
VSA_OP_BACKWARD = 1
VSA_OP_FINE_BWD = 2
VSA_OP_FORWARD_INFERENCE = 3
VSA_OP_FINE_FWD = 4
VSA_CURVE_RASTER = 0
VSA_CURVE_HILBERT = 1
VSA_NOALLOC_SCRATCH_BYTES = 64 << 20   # the fixed scratch array of vsa_fine_bwd_noalloc

# Every function the header declares, with its ctypes signature.
P = ctypes.c_void_p
I = ctypes.c_int
F = ctypes.c_float
SZ = ctypes.c_size_t


class Grid(ctypes.Structure):
    """vsa_grid_t: latent grid (T, H, W), cube shape (must be 4, 4, 4) and the
    device address of a cube order table (0: cube-raster order)."""

    _fields_ = [("T", I), ("H", I), ("W", I), ("ct", I), ("ch", I), ("cw", I), ("cube_order", P)]

    @classmethod
    def of(cls, T, H, W, cube_order=None):
        return cls(T, H, W, 4, 4, 4, cube_order)


class Saved(ctypes.Structure):
    """vsa_saved_t: device pointers into a forward workspace, and the list width."""

    _fields_ = [(n, P) for n in ("qp", "kp", "vp", "qc", "kc", "vc", "o_coarse", "lse_coarse",
                                 "kv_block_idx", "valid_block_num", "o_fine", "lse", "tile_pairs")] + \
        [("max_kv_blocks", I)]


SIGNATURES = {
    "vsa_permute": ([P, P, P, I, I, Grid, I, P], I),
    "vsa_cube_order": ([Grid, I, P, P], I),
    "vsa_coarse_topk": ([P, P, P, I, I, I, I, F, P, P, P, P, P, P], I),
    "vsa_fine_fwd": ([P, P, P, P, P, I, I, I, I, F, P, I, P, P, SZ, P], I),
    "vsa_fine_bwd": ([P, P, P, P, I, P, P, P, P, I, I, I, I, F, P, P, P, P, SZ, P], I),
    "vsa_fine_bwd_noalloc": ([P, P, P, P, I, P, P, P, P, I, I, I, I, F, P, P, P, P], I),
    "vsa_forward": ([P, P, P, P, P, I, I, I, Grid, I, I, F, P, I, P, SZ, P], I),
    "vsa_forward_inference": ([P, P, P, P, P, I, I, I, Grid, I, I, F, P, I, P, SZ, P], I),
    "vsa_backward": ([P, P, P, P, I, I, I, Grid, I, I, F, P, P, P, P, P, I, P, SZ, P], I),
    "vsa_workspace_bytes": ([I, I, I, I, Grid, I, I], SZ),
    "vsa_forward_saved": ([P, I, I, I, Grid, I, I, ctypes.POINTER(Saved)], I),
    "vsa_backward_tile_pairs": ([P, I, I, I, Grid, I, I, ctypes.POINTER(P)], I),
    "vsa_device_status": ([P], I),
    "vsa_selftest_wait_timeout": ([ctypes.c_uint32, P], I),
    "vsa_mask_to_lut": ([P, I, I, I, P, P, P], I),
    "vsa_lut_add_neighbors": ([P, P, I, I, Grid, I, I, P, P, P], I),
    "vsa_status_string": ([I], ctypes.c_char_p),
    "vsa_timing_enable": ([I], I),
    "vsa_timing_read": ([I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I)], I),
}

KERNELS = ["permute", "coarse_topk", "fine_fwd", "combine", "bwd_prep", "coarse_bwd", "fine_bwd_kv", "fine_bwd_dq"]

_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(or python block_sparse_video_sfc_gb300/build.py); the library has no fallback.")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


class VSAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = load().vsa_status_string(status).decode()
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


def check(fn: str, status: int) -> None:
    if status != VSA_OK:
        raise VSAError(fn, status)
