// permute_pool.cu -- 3D space-filling-curve token reordering with the cube
// mean-pool fused ("VSA: Accelerating Video Diffusion Inference with Sparse
// Attention on AMD GPUs", "Two-Stage Architecture": pre-stage SFC reordering
// and the Stage 1 cube mean-pool).
//
// One CTA moves one cube (64 tokens x d) of one tensor: 16-byte vector loads
// and stores; a cube's native tokens are 16 runs of 4 contiguous tokens, its
// cube-order destination is one contiguous 64*d*2-byte block.  The pooled
// mean is summed in fp32 while the data passes through registers.
// HBM-bound: per tensor, N*d*2 bytes read + N*d*2 written (+ Nc*d*4 pooled).
// A grid side that is not a multiple of 4 ends in partial cubes: their slots
// outside the grid are written as zeros (cube order) or skipped (native
// order), and the pooled mean divides by the cube's token count.
#include "common.cuh"

namespace vsa {

struct PermuteArgs {
  const __nv_bfloat16* src[3];
  void* dst[3];
  float* pooled[3];
};

// F16OUT: the destination holds the same values as fp16 (exact for inputs of
// magnitude <= 65504; larger ones saturate and latch kErrRange).
template <int D, bool F16OUT>
__global__ void __launch_bounds__(256) permute_pool_kernel(PermuteArgs a, int Nc, CubeGrid g, int64_t Nn,
                                                           const int32_t* __restrict__ order, int inverse, int* err) {
  constexpr int kChunks = D / 8;           // 16-byte chunks per token
  constexpr int kTokPerPass = 256 / kChunks;
  constexpr int kPasses = kCube / kTokPerPass;
  __shared__ float red[kTokPerPass][D];
  const int tensor = blockIdx.y;
  const int64_t cube_glob = blockIdx.x;    // bh * Nc + cube
  const int64_t bh = cube_glob / Nc;
  const int cube = static_cast<int>(cube_glob % Nc);
  const int rcube = raster_cube(order, cube);
  const int64_t Np = static_cast<int64_t>(Nc) * kCube;  // reordered tokens per (batch, head)
  const __nv_bfloat16* src = a.src[tensor] + bh * (inverse ? Np : Nn) * D;
  // A null destination pools only (the inference forward reads the native
  // layout directly and needs no reordered copy).
  uint16_t* dst = a.dst[tensor] ? static_cast<uint16_t*>(a.dst[tensor]) + bh * (inverse ? Nn : Np) * D : nullptr;
  float* pooled = a.pooled[tensor];
  const int j = threadIdx.x % kChunks;     // channel chunk, fixed per thread
  const int o0 = threadIdx.x / kChunks;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  // All of this thread's loads are issued before any store, so that each
  // thread keeps kPasses 16-byte reads in flight.
  uint4 vin[kPasses];
  int64_t nat_of[kPasses];
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int o = o0 + p * kTokPerPass;
    const int64_t nat = native_token(rcube, o, g);
    const int64_t cub = static_cast<int64_t>(cube) * kCube + o;
    nat_of[p] = nat;
    const int64_t s_tok = inverse ? cub : nat;
    vin[p] = nat < 0 ? make_uint4(0, 0, 0, 0) : __ldg(reinterpret_cast<const uint4*>(src + s_tok * D + j * 8));
  }
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int o = o0 + p * kTokPerPass;
    const int64_t nat = nat_of[p];
    const int64_t cub = static_cast<int64_t>(cube) * kCube + o;
    if (nat < 0 && inverse) continue;  // padding slot: nothing to write back
    const int64_t d_tok = inverse ? nat : cub;
    const uint4 v = vin[p];
    if (!dst) {
      // pool only
    } else if (F16OUT) {
      const float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                          bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
      bool big = false;
#pragma unroll
      for (int e = 0; e < 8; ++e) big |= !(fabsf(f[e]) <= kF16Max);
      if (big) flag_error(err, kErrRange);
      uint4 h = make_uint4(pack_f16(f[0], f[1]), pack_f16(f[2], f[3]), pack_f16(f[4], f[5]), pack_f16(f[6], f[7]));
      *reinterpret_cast<uint4*>(dst + d_tok * D + j * 8) = h;
    } else {
      *reinterpret_cast<uint4*>(dst + d_tok * D + j * 8) = v;
    }
    if (pooled) {
      acc[0] += bf16_lo(v.x); acc[1] += bf16_hi(v.x);
      acc[2] += bf16_lo(v.y); acc[3] += bf16_hi(v.y);
      acc[4] += bf16_lo(v.z); acc[5] += bf16_hi(v.z);
      acc[6] += bf16_lo(v.w); acc[7] += bf16_hi(v.w);
    }
  }
  if (pooled) {
#pragma unroll
    for (int e = 0; e < 8; ++e) red[o0][j * 8 + e] = acc[e];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += 256) {
      float s = 0.f;
#pragma unroll 8
      for (int r = 0; r < kTokPerPass; ++r) s += red[r][c];
      pooled[cube_glob * D + c] = s / static_cast<float>(cube_tokens(rcube, g));
    }
  }
}

int launch_permute(const void* const* src, void* const* dst, float* const* pooled, int ntensors, int BH, int d,
                   int T, int H, int W, const int32_t* order, int inverse, int f16_out, cudaStream_t s) {
  PermuteArgs a{};
  for (int i = 0; i < ntensors; ++i) {
    a.src[i] = static_cast<const __nv_bfloat16*>(src[i]);
    a.dst[i] = dst[i];
    a.pooled[i] = pooled ? pooled[i] : nullptr;
  }
  const CubeGrid g = cube_grid(T, H, W);
  const int Nc = ((T + 3) / 4) * g.Hc * g.Wc;
  const int64_t Nn = static_cast<int64_t>(T) * H * W;
  dim3 grid(static_cast<unsigned>(static_cast<int64_t>(BH) * Nc), ntensors);
  int* err = device_error_word();
  timing_mark(VSA_K_PERMUTE, true, s);
  if (d == 128) {
    if (f16_out)
      permute_pool_kernel<128, true><<<grid, 256, 0, s>>>(a, Nc, g, Nn, order, inverse, err);
    else
      permute_pool_kernel<128, false><<<grid, 256, 0, s>>>(a, Nc, g, Nn, order, inverse, err);
  } else {
    if (f16_out)
      permute_pool_kernel<64, true><<<grid, 256, 0, s>>>(a, Nc, g, Nn, order, inverse, err);
    else
      permute_pool_kernel<64, false><<<grid, 256, 0, s>>>(a, Nc, g, Nn, order, inverse, err);
  }
  timing_mark(VSA_K_PERMUTE, false, s);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace vsa
