// lut_ops.cu -- building and widening the per-query-cube index lists.
//
// "VSA: Accelerating Video Diffusion Inference with Sparse Attention on AMD
// GPUs", "Sparse Encoding in CK Tile": VSA keeps, per query block, the list
// of selected K/V blocks and a valid count; Jenga keeps the full M x M block
// relation matrix B and skips the cells with B[i][j] = 0.  "Comparison with
// Jenga", "Algorithmic Design": Jenga's selection is the union of three
// masks, one of them the spatial adjacency of the block.
//
//   vsa_mask_to_lut        B (one byte per cell) -> ascending list + count
//   vsa_lut_add_neighbors  list -> list united with every cube within a
//                          Chebyshev radius on the (T/4, H/4, W/4) cube grid
//                          (ids are positions in the cube sequence; a cube
//                          order table maps them to and from grid cells)
//
// Both write each row's cubes in ascending id, the count, and -1 in the
// unused slots.  A row with more cubes than the output holds keeps its first
// `max_kv_blocks` (lowest ids) and latches the list error (VSA_ERR_LUT).
#include "common.cuh"

namespace vsa {
namespace {

constexpr int kRowThreads = 128;

// One warp turns the row bitmap into the ascending list; returns nothing,
// writes idx[0..kmax) and *cnt.
__device__ void write_list_from_bits(const uint32_t* bits, int nwords, int kmax, int32_t* idx, int32_t* cnt,
                                     int* err) {
  const int lane = threadIdx.x & 31;
  int pos = 0;
  for (int w0 = 0; w0 < nwords; w0 += 32) {
    const int w = w0 + lane;
    uint32_t u = w < nwords ? bits[w] : 0u;
    const int n = __popc(u);
    int incl = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int o = pos + incl - n;
    while (u) {
      const int bit = __ffs(u) - 1;
      u &= u - 1;
      if (o < kmax) idx[o] = w * 32 + bit;
      ++o;
    }
    pos += __shfl_sync(0xffffffffu, incl, 31);
  }
  for (int e = pos + lane; e < kmax; e += 32) idx[e] = -1;
  if (lane == 0) {
    if (pos > kmax) flag_error(err, kErrLut);
    *cnt = pos < kmax ? pos : kmax;
  }
}

__global__ void __launch_bounds__(kRowThreads) mask_to_lut_kernel(const uint8_t* __restrict__ mask, int Nc, int kmax,
                                                                  int32_t* __restrict__ idx, int32_t* __restrict__ cnt,
                                                                  int* err) {
  extern __shared__ uint32_t bits[];
  const int64_t row = blockIdx.x;  // bh * Nc + query cube
  const int nwords = (Nc + 31) >> 5;
  const uint8_t* m = mask + row * Nc;
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) {
    uint32_t v = 0;
    const int c0 = w * 32;
    for (int b = 0; b < 32 && c0 + b < Nc; ++b) v |= (m[c0 + b] != 0 ? 1u : 0u) << b;
    bits[w] = v;
  }
  __syncthreads();
  if (threadIdx.x < 32) write_list_from_bits(bits, nwords, kmax, idx + row * kmax, cnt + row, err);
}

__global__ void __launch_bounds__(kRowThreads) add_neighbors_kernel(const int32_t* __restrict__ idx_in,
                                                                    const int32_t* __restrict__ cnt_in, int kmax_in,
                                                                    int Tc, int Hc, int Wc,
                                                                    const int32_t* __restrict__ order, int radius,
                                                                    int kmax_out,
                                                                    int32_t* __restrict__ idx_out,
                                                                    int32_t* __restrict__ cnt_out, int* err) {
  extern __shared__ uint32_t bits[];
  const int Nc = Tc * Hc * Wc, nwords = (Nc + 31) >> 5;
  const int64_t row = blockIdx.x;
  const int q = static_cast<int>(row % Nc);
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) bits[w] = 0u;
  __syncthreads();
  int n = cnt_in ? cnt_in[row] : kmax_in;
  if (n < 0 || n > kmax_in) {
    if (threadIdx.x == 0) flag_error(err, kErrLut);
    n = min(max(n, 0), kmax_in);
  }
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int c = idx_in[row * kmax_in + e];
    if (c < 0 || c >= Nc) {
      flag_error(err, kErrLut);
      continue;
    }
    atomicOr(&bits[c >> 5], 1u << (c & 31));
  }
  // The neighbourhood: every cube whose grid coordinates differ from the
  // query cube's by at most `radius` in each of t, h, w (the cube itself too).
  const int qr = raster_cube(order, q);
  const int qt = qr / (Hc * Wc), qh = (qr / Wc) % Hc, qw = qr % Wc;
  const int side = 2 * radius + 1, count = side * side * side;
  for (int e = threadIdx.x; e < count; e += blockDim.x) {
    const int t = qt + e / (side * side) - radius, h = qh + (e / side) % side - radius, w = qw + e % side - radius;
    if (t < 0 || t >= Tc || h < 0 || h >= Hc || w < 0 || w >= Wc) continue;
    const int r = (t * Hc + h) * Wc + w;
    const int c = order ? __ldg(order + Nc + r) : r;  // raster id -> position
    atomicOr(&bits[c >> 5], 1u << (c & 31));
  }
  __syncthreads();
  if (threadIdx.x < 32) write_list_from_bits(bits, nwords, kmax_out, idx_out + row * kmax_out, cnt_out + row, err);
}

}  // namespace

int launch_mask_to_lut(const uint8_t* mask, int BH, int Nc, int kmax, int32_t* idx, int32_t* cnt, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(BH) * Nc;
  if (rows == 0) return VSA_OK;
  const size_t smem = sizeof(uint32_t) * ((Nc + 31) / 32);
  mask_to_lut_kernel<<<static_cast<unsigned>(rows), kRowThreads, smem, s>>>(mask, Nc, kmax, idx, cnt,
                                                                            device_error_word());
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

int launch_add_neighbors(const int32_t* idx_in, const int32_t* cnt_in, int kmax_in, int BH, int Tc, int Hc, int Wc,
                         const int32_t* order, int radius, int kmax_out, int32_t* idx_out, int32_t* cnt_out,
                         cudaStream_t s) {
  const int Nc = Tc * Hc * Wc;
  const int64_t rows = static_cast<int64_t>(BH) * Nc;
  if (rows == 0) return VSA_OK;
  const size_t smem = sizeof(uint32_t) * ((Nc + 31) / 32);
  add_neighbors_kernel<<<static_cast<unsigned>(rows), kRowThreads, smem, s>>>(
      idx_in, cnt_in, kmax_in, Tc, Hc, Wc, order, radius, kmax_out, idx_out, cnt_out, device_error_word());
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace vsa
