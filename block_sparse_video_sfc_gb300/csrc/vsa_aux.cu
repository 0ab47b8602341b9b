// vsa_aux.cu -- the HBM-bound and small steps around the fine kernels:
//   combine   out = g_c * O_c + g_f * O_f, written in native token order
//             ("VSA: Accelerating Video Diffusion Inference with Sparse
//             Attention on AMD GPUs", "Stage 2: Fine Computation": the output
//             combines the coarse and fine outputs through learnable gates).
//   bwd_prep  backward of the combine: dO to cube order, dO_f = g_f * dO
//             (fp16 for the fine backward), D = dO_f . O_f, dO_c = sum over the
//             cube of g_c * dO, D_c = dO_c . O_c (the coarse backward's row
//             statistic: sum_j P_j dP_j = dO_c . sum_j P_j V_j), and the gate
//             gradients.
// (The mean-pool backward and the inverse reordering of dQ, dK, dV run in
// the epilogues of the fine backward kernels.)
// The backward pass follows "VSA: Faster Video Diffusion with Trainable Sparse
// Attention" (Abstract: trained end to end); derivatives are the textbook ones.
// The per-cube kernels use one CTA per cube of one tensor, 16-byte accesses.
#include "common.cuh"

namespace vsa {
namespace {

// ---------------------------------------------------------------- combine
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ oc, const float* __restrict__ of,
                                                      const __nv_bfloat16* __restrict__ gc,
                                                      const __nv_bfloat16* __restrict__ gf, void* __restrict__ out,
                                                      int out_dtype, int Nc, CubeGrid g, int64_t Nn,
                                                      const int32_t* __restrict__ order) {
  constexpr int kChunks = D / 8, kTok = 256 / kChunks, kPasses = kCube / kTok;
  const int64_t cg = blockIdx.x;
  const int64_t bh = cg / Nc;
  const int cube = static_cast<int>(cg % Nc);
  const int rcube = raster_cube(order, cube);
  const int j = threadIdx.x % kChunks, o0 = threadIdx.x / kChunks;
  float c[8];
  load8_f32(oc, cg * D + j * 8, c);
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int o = o0 + p * kTok;
    const int64_t tok = native_token(rcube, o, g);
    if (tok < 0) continue;  // padding slot
    const int64_t nat = bh * Nn + tok;
    const int64_t cub = (bh * Nc + cube) * kCube + o;
    float f[8], a[8], b[8], r[8];
    load8_f32(of, cub * D + j * 8, f);
    if (gc) load8_bf16(gc, nat * D + j * 8, a);
    if (gf) load8_bf16(gf, nat * D + j * 8, b);
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = (gc ? a[e] : 1.f) * c[e] + (gf ? b[e] : 1.f) * f[e];
    store8(out, nat * D + j * 8, r, out_dtype);
  }
}

// ---------------------------------------------------------------- bwd_prep
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ dout,
                                                       const __nv_bfloat16* __restrict__ gc,
                                                       const __nv_bfloat16* __restrict__ gf,
                                                       const float* __restrict__ oc, const float* __restrict__ of,
                                                       __half* __restrict__ dof, float* __restrict__ delta,
                                                       float* __restrict__ doc, float* __restrict__ delta_c,
                                                       void* __restrict__ dgc,
                                                       void* __restrict__ dgf, int grad_dtype, int Nc, CubeGrid grid,
                                                       int64_t Nn, const int32_t* __restrict__ order, int* err) {
  constexpr int kChunks = D / 8, kTok = 256 / kChunks, kPasses = kCube / kTok;
  __shared__ float red[kTok][D];
  __shared__ float dcw[D / 32];
  const int64_t cg = blockIdx.x;
  const int64_t bh = cg / Nc;
  const int cube = static_cast<int>(cg % Nc);
  const int rcube = raster_cube(order, cube);
  const int j = threadIdx.x % kChunks, o0 = threadIdx.x / kChunks;
  float c[8], acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  load8_f32(oc, cg * D + j * 8, c);
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int o = o0 + p * kTok;
    const int64_t tok = native_token(rcube, o, grid);
    const bool real = tok >= 0;  // padding slots get dO = 0: zero dO_f and D
    const int64_t nat = bh * Nn + (real ? tok : 0);
    const int64_t cub = (bh * Nc + cube) * kCube + o;
    float g[8], a[8], b[8], f[8], t[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) g[e] = a[e] = b[e] = 0.f;
    if (real) load8_bf16(dout, nat * D + j * 8, g);
    load8_f32(of, cub * D + j * 8, f);
    if (gc && real) load8_bf16(gc, nat * D + j * 8, a);
    if (gf && real) load8_bf16(gf, nat * D + j * 8, b);
    uint4 packed;
    uint32_t* pk = reinterpret_cast<uint32_t*>(&packed);
    float dsum = 0.f;
    bool big = false;
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float x0 = (gf ? b[e] : 1.f) * g[e], x1 = (gf ? b[e + 1] : 1.f) * g[e + 1];
      big |= !(fabsf(x0) <= kF16Max) || !(fabsf(x1) <= kF16Max);
      pk[e >> 1] = pack_f16(x0, x1);
      // D uses the fp16 values the fine backward multiplies with.
      dsum = fmaf(f16_lo(pk[e >> 1]), f[e], dsum);
      dsum = fmaf(f16_hi(pk[e >> 1]), f[e + 1], dsum);
    }
    if (big) flag_error(err, kErrRange);
    *reinterpret_cast<uint4*>(dof + cub * D + j * 8) = packed;
#pragma unroll
    for (int off = kChunks / 2; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
    if (j == 0) delta[cub] = dsum;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = fmaf(gc ? a[e] : 1.f, g[e], acc[e]);
    if (gc && dgc && real) {
#pragma unroll
      for (int e = 0; e < 8; ++e) t[e] = g[e] * c[e];
      store8(dgc, nat * D + j * 8, t, grad_dtype);
    }
    if (gf && dgf && real) {
#pragma unroll
      for (int e = 0; e < 8; ++e) t[e] = g[e] * f[e];
      store8(dgf, nat * D + j * 8, t, grad_dtype);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[o0][j * 8 + e] = acc[e];
  __syncthreads();
  float dprod = 0.f;
  for (int ch = threadIdx.x; ch < D; ch += 256) {
    float s = 0.f;
    for (int r = 0; r < kTok; ++r) s += red[r][ch];
    doc[cg * D + ch] = s;
    dprod = s * oc[cg * D + ch];
  }
  if (delta_c) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dprod += __shfl_xor_sync(0xffffffffu, dprod, off);
    if (threadIdx.x < D && (threadIdx.x & 31) == 0) dcw[threadIdx.x >> 5] = dprod;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < D / 32; ++w) t += dcw[w];
      delta_c[cg] = t;
    }
  }
}

}  // namespace

int launch_combine(const float* oc, const float* of, const void* gc, const void* gf, void* out, int out_dtype, int BH,
                   int d, int T, int H, int W, const int32_t* order, cudaStream_t s) {
  const CubeGrid cg = cube_grid(T, H, W);
  const int Nc = ((T + 3) / 4) * cg.Hc * cg.Wc;
  const int64_t Nn = static_cast<int64_t>(T) * H * W;
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(BH) * Nc);
  auto g = static_cast<const __nv_bfloat16*>(gc);
  auto f = static_cast<const __nv_bfloat16*>(gf);
  timing_mark(VSA_K_COMBINE, true, s);
  if (d == 128)
    combine_kernel<128><<<grid, 256, 0, s>>>(oc, of, g, f, out, out_dtype, Nc, cg, Nn, order);
  else
    combine_kernel<64><<<grid, 256, 0, s>>>(oc, of, g, f, out, out_dtype, Nc, cg, Nn, order);
  timing_mark(VSA_K_COMBINE, false, s);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

int launch_bwd_prep(const void* dout, const void* gc, const void* gf, const float* oc, const float* of,
                    __half* dof, float* delta, float* doc, float* delta_c, void* dgc, void* dgf, int grad_dtype,
                    int BH, int d, int T, int H, int W, const int32_t* order, cudaStream_t s) {
  const CubeGrid cg = cube_grid(T, H, W);
  const int Nc = ((T + 3) / 4) * cg.Hc * cg.Wc;
  const int64_t Nn = static_cast<int64_t>(T) * H * W;
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(BH) * Nc);
  auto dO = static_cast<const __nv_bfloat16*>(dout);
  auto g = static_cast<const __nv_bfloat16*>(gc);
  auto f = static_cast<const __nv_bfloat16*>(gf);
  timing_mark(VSA_K_BWD_PREP, true, s);
  if (d == 128)
    bwd_prep_kernel<128><<<grid, 256, 0, s>>>(dO, g, f, oc, of, dof, delta, doc, delta_c, dgc, dgf, grad_dtype, Nc,
                                              cg, Nn, order, device_error_word());
  else
    bwd_prep_kernel<64><<<grid, 256, 0, s>>>(dO, g, f, oc, of, dof, delta, doc, delta_c, dgc, dgf, grad_dtype, Nc,
                                             cg, Nn, order, device_error_word());
  timing_mark(VSA_K_BWD_PREP, false, s);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace vsa
