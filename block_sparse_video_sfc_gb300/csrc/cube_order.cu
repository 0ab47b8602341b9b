// cube_order.cu -- the order of the cubes along the 3D space-filling curve.
//
// "VSA: Accelerating Video Diffusion Inference with Sparse Attention on AMD
// GPUs", "Two-Stage Architecture" (pre-stage: tokens are reordered along a 3D
// space-filling curve so that each block of the 1D sequence is one compact
// spatio-temporal region; the curve is Jenga's and the page does not print
// it).  Two orders of the (T/4, H/4, W/4) cube grid are offered:
//   VSA_CURVE_RASTER   cube (ct, ch, cw) at position (ct*Hc + ch)*Wc + cw;
//   VSA_CURVE_HILBERT  cubes in the order the 3-D Hilbert curve of the
//                      smallest enclosing 2^b grid meets them (cells outside
//                      the grid skipped).  The curve is J. Skilling's
//                      ("Programming the Hilbert curve", AIP Conf. Proc. 707,
//                      2004), here taken from point to index.
// Tokens inside a cube keep (t%4, h%4, w%4) raster order either way.
//
// The table holds 2*Nc int32: order[p] = raster id of the cube at position p,
// order[Nc + r] = position of raster cube r.
#include "common.cuh"

namespace vsa {
namespace {

constexpr int kOrderThreads = 1024;

// Index of cell (t, h, w) on the order-b 3-D Hilbert curve.  From the top
// level down, an axis whose bit is set reflects the lower bits of axis t,
// and an axis whose bit is clear swaps its lower bits with those of axis t;
// the three axes are then Gray-encoded (each takes the running parity of the
// axes before it, and all take the levels at which the last axis is odd) and
// the index is read off three bits per level, t first.
__host__ __device__ uint32_t hilbert_index(uint32_t t, uint32_t h, uint32_t w, int b) {
  if (b == 0) return 0;
  uint32_t x[3] = {t, h, w};
  for (uint32_t bit = 1u << (b - 1); bit > 1; bit >>= 1) {
    const uint32_t low = bit - 1;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      if (x[a] & bit) {
        x[0] ^= low;
      } else {
        const uint32_t sw = (x[0] ^ x[a]) & low;
        x[0] ^= sw;
        x[a] ^= sw;
      }
    }
  }
  x[1] ^= x[0];
  x[2] ^= x[1];
  uint32_t flip = 0;
  for (uint32_t bit = 1u << (b - 1); bit > 1; bit >>= 1)
    if (x[2] & bit) flip ^= bit - 1;
  uint32_t hidx = 0;
  for (int level = b - 1; level >= 0; --level)
#pragma unroll
    for (int a = 0; a < 3; ++a) hidx = (hidx << 1) | (((x[a] ^ flip) >> level) & 1u);
  return hidx;
}

// One CTA: the curve key of every cube into shared memory, then each cube's
// position = the number of cubes with a smaller key (the keys are distinct).
__global__ void __launch_bounds__(kOrderThreads) cube_order_kernel(int Tc, int Hc, int Wc, int b, int curve,
                                                                   int32_t* __restrict__ order) {
  extern __shared__ uint32_t key[];
  const int Nc = Tc * Hc * Wc;
  for (int r = threadIdx.x; r < Nc; r += blockDim.x) {
    const int ct = r / (Hc * Wc), ch = (r / Wc) % Hc, cw = r % Wc;
    key[r] = curve == VSA_CURVE_HILBERT ? hilbert_index(ct, ch, cw, b) : static_cast<uint32_t>(r);
  }
  __syncthreads();
  for (int r = threadIdx.x; r < Nc; r += blockDim.x) {
    const uint32_t mine = key[r];
    int pos = 0;
    for (int q = 0; q < Nc; ++q) pos += key[q] < mine;
    order[pos] = r;
    order[Nc + r] = pos;
  }
}

// kmask[c]: bit o set when slot o of the cube at position c holds a grid
// token (all 64 bits unless the cube sticks out of a grid whose side is not a
// multiple of 4).
__global__ void slot_mask_kernel(int Nc, CubeGrid g, const int32_t* __restrict__ order, uint64_t* __restrict__ kmask) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= Nc) return;
  const int rc = raster_cube(order, c);
  uint64_t m = 0;
  for (int o = 0; o < kCube; ++o)
    if (native_token(rc, o, g) >= 0) m |= 1ull << o;
  kmask[c] = m;
}

}  // namespace

int launch_slot_masks(int T, int H, int W, const int32_t* order, uint64_t* kmask, cudaStream_t s) {
  const CubeGrid g = cube_grid(T, H, W);
  const int Nc = ((T + 3) / 4) * g.Hc * g.Wc;
  slot_mask_kernel<<<(Nc + 255) / 256, 256, 0, s>>>(Nc, g, order, kmask);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

int launch_cube_order(int Tc, int Hc, int Wc, int curve, int32_t* order, cudaStream_t s) {
  int b = 0;
  while ((1 << b) < Tc || (1 << b) < Hc || (1 << b) < Wc) ++b;
  if (b > 10) return VSA_ERR_UNSUPPORTED;  // 30-bit curve index
  const int Nc = Tc * Hc * Wc;
  const size_t smem = sizeof(uint32_t) * Nc;
  if (smem > 200 * 1024) return VSA_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(cube_order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return VSA_ERR_CUDA;
  cube_order_kernel<<<1, kOrderThreads, smem, s>>>(Tc, Hc, Wc, b, curve, order);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace vsa
