// vsa_aux.cu -- the HBM-bound and small steps around the fine kernels:
//   combine   out = g_c * O_c + g_f * O_f, written in native token order
//             ("VSA: Accelerating Video Diffusion Inference with Sparse
//             Attention on AMD GPUs", "Stage 2: Fine Computation": the output
//             combines the coarse and fine outputs through learnable gates).
//   bwd_prep  backward of the combine: dO to cube order, dO_f = g_f * dO
//             (fp16 for the fine backward), D = dO_f . O_f, dO_c = sum over the
//             cube of g_c * dO, and the gate gradients.
//   coarse backward  softmax Jacobian of the coarse stage (fp32 SIMT).
//   finalize  mean-pool backward (+ dXc / 64 to every token of a cube) and
//             the inverse reordering of dQ, dK, dV.
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
                                                      int out_dtype, int Nc, int H, int W, int N) {
  constexpr int kChunks = D / 8, kTok = 256 / kChunks, kPasses = kCube / kTok;
  const int64_t cg = blockIdx.x;
  const int64_t bh = cg / Nc;
  const int cube = static_cast<int>(cg % Nc);
  const int j = threadIdx.x % kChunks, o0 = threadIdx.x / kChunks;
  float c[8];
  load8_f32(oc, cg * D + j * 8, c);
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int o = o0 + p * kTok;
    const int64_t nat = bh * N + native_token(cube, o, H, W);
    const int64_t cub = bh * N + static_cast<int64_t>(cube) * kCube + o;
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
                                                       float* __restrict__ doc, void* __restrict__ dgc,
                                                       void* __restrict__ dgf, int grad_dtype, int Nc, int H, int W,
                                                       int N, int* err) {
  constexpr int kChunks = D / 8, kTok = 256 / kChunks, kPasses = kCube / kTok;
  __shared__ float red[kTok][D];
  const int64_t cg = blockIdx.x;
  const int64_t bh = cg / Nc;
  const int cube = static_cast<int>(cg % Nc);
  const int j = threadIdx.x % kChunks, o0 = threadIdx.x / kChunks;
  float c[8], acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  load8_f32(oc, cg * D + j * 8, c);
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int o = o0 + p * kTok;
    const int64_t nat = bh * N + native_token(cube, o, H, W);
    const int64_t cub = bh * N + static_cast<int64_t>(cube) * kCube + o;
    float g[8], a[8], b[8], f[8], t[8];
    load8_bf16(dout, nat * D + j * 8, g);
    load8_f32(of, cub * D + j * 8, f);
    if (gc) load8_bf16(gc, nat * D + j * 8, a);
    if (gf) load8_bf16(gf, nat * D + j * 8, b);
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
    if (gc && dgc) {
#pragma unroll
      for (int e = 0; e < 8; ++e) t[e] = g[e] * c[e];
      store8(dgc, nat * D + j * 8, t, grad_dtype);
    }
    if (gf && dgf) {
#pragma unroll
      for (int e = 0; e < 8; ++e) t[e] = g[e] * f[e];
      store8(dgf, nat * D + j * 8, t, grad_dtype);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[o0][j * 8 + e] = acc[e];
  __syncthreads();
  for (int ch = threadIdx.x; ch < D; ch += 256) {
    float s = 0.f;
    for (int r = 0; r < kTok; ++r) s += red[r][ch];
    doc[cg * D + ch] = s;
  }
}

// ---------------------------------------------------------------- coarse backward
// Per query cube a (R rows per CTA):  S = scale Qc Kc^T, P = exp(S - lse_c),
// dP = dOc Vc^T, dS = P (dP - sum_b P dP); dQc = scale dS Kc (row-local).
// P and dS rows go to global for the column products dKc, dVc.
constexpr int kCT = 256, kCChunk = 32;

template <int D>
__global__ void __launch_bounds__(kCT) coarse_bwd_rows(const float* __restrict__ qc, const float* __restrict__ kc,
                                                       const float* __restrict__ vc, const float* __restrict__ doc,
                                                       const float* __restrict__ lse_c, int Nc, int R, float scale,
                                                       float* __restrict__ Pg, float* __restrict__ dSg,
                                                       float* __restrict__ dqc) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr int KVS = D + 4;
  float* sQ = reinterpret_cast<float*>(smem);        // [R][D]
  float* sG = sQ + R * D;                            // [R][D] dOc rows
  float* sS = sG + R * D;                            // [R][Nc]
  float* sP = sS + R * Nc;                           // [R][Nc]
  float* sKV = sP + R * Nc;                          // [32][KVS]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t bh = blockIdx.y;
  const int row0 = blockIdx.x * R;
  for (int e = tid; e < R * D; e += kCT) {
    int r = e / D, ch = e % D;
    bool v = row0 + r < Nc;
    sQ[e] = v ? qc[(bh * Nc + row0 + r) * D + ch] : 0.f;
    sG[e] = v ? doc[(bh * Nc + row0 + r) * D + ch] : 0.f;
  }
  for (int pass = 0; pass < 2; ++pass) {
    const float* src = (pass == 0 ? kc : vc) + bh * static_cast<int64_t>(Nc) * D;
    const float* lhs = pass == 0 ? sQ : sG;
    float* dst = pass == 0 ? sS : sP;
    for (int kb = 0; kb < Nc; kb += kCChunk) {
      __syncthreads();
      for (int e = tid; e < kCChunk * D / 4; e += kCT) {
        int r = e / (D / 4), c4 = e % (D / 4);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (kb + r < Nc) v = reinterpret_cast<const float4*>(src + static_cast<int64_t>(kb + r) * D)[c4];
        *reinterpret_cast<float4*>(sKV + r * KVS + 4 * c4) = v;
      }
      __syncthreads();
      for (int pi = tid; pi < R * kCChunk; pi += kCT) {
        int r = pi / kCChunk, jj = pi % kCChunk;
        const float4* a4 = reinterpret_cast<const float4*>(lhs + r * D);
        const float4* b4 = reinterpret_cast<const float4*>(sKV + jj * KVS);
        float acc = 0.f;
#pragma unroll 8
        for (int c = 0; c < D / 4; ++c) {
          float4 a = a4[c], b = b4[c];
          acc = fmaf(a.x, b.x, acc);
          acc = fmaf(a.y, b.y, acc);
          acc = fmaf(a.z, b.z, acc);
          acc = fmaf(a.w, b.w, acc);
        }
        if (kb + jj < Nc) dst[r * Nc + kb + jj] = pass == 0 ? acc * scale : acc;
      }
    }
  }
  __syncthreads();
  for (int r = warp; r < R; r += kCT / 32) {
    const int row = row0 + r;
    if (row >= Nc) continue;
    const int64_t g = bh * Nc + row;
    const float l = lse_c[g];
    float* s = sS + r * Nc;
    float* dp = sP + r * Nc;
    float dsum = 0.f;
    for (int b = lane; b < Nc; b += 32) {
      float pv = __expf(s[b] - l);
      s[b] = pv;
      dsum = fmaf(pv, dp[b], dsum);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
    for (int b = lane; b < Nc; b += 32) {
      float ds = s[b] * (dp[b] - dsum);
      dp[b] = ds;
      Pg[g * Nc + b] = s[b];
      dSg[g * Nc + b] = ds;
    }
  }
  // dQc = scale * dS Kc
  constexpr int kGroups = D / 4;
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* Kb = kc + bh * static_cast<int64_t>(Nc) * D;
  for (int kb = 0; kb < Nc; kb += kCChunk) {
    __syncthreads();
    for (int e = tid; e < kCChunk * D / 4; e += kCT) {
      int r = e / (D / 4), c4 = e % (D / 4);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kb + r < Nc) v = reinterpret_cast<const float4*>(Kb + static_cast<int64_t>(kb + r) * D)[c4];
      *reinterpret_cast<float4*>(sKV + r * KVS + 4 * c4) = v;
    }
    __syncthreads();
    const int jmax = min(kCChunk, Nc - kb);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int pi = tid + i * kCT;
      if (pi >= R * kGroups) break;
      int r = pi / kGroups, c4 = pi % kGroups;
      const float* dsr = sP + r * Nc + kb;
      float4 a = acc[i];
      for (int jj = 0; jj < jmax; ++jj) {
        float w = dsr[jj];
        float4 v = *reinterpret_cast<const float4*>(sKV + jj * KVS + 4 * c4);
        a.x = fmaf(w, v.x, a.x);
        a.y = fmaf(w, v.y, a.y);
        a.z = fmaf(w, v.z, a.z);
        a.w = fmaf(w, v.w, a.w);
      }
      acc[i] = a;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int pi = tid + i * kCT;
    if (pi >= R * kGroups) break;
    int r = pi / kGroups, c4 = pi % kGroups;
    if (row0 + r < Nc) {
      float4 a = acc[i];
      a.x *= scale; a.y *= scale; a.z *= scale; a.w *= scale;
      reinterpret_cast<float4*>(dqc + (bh * Nc + row0 + r) * D)[c4] = a;
    }
  }
}

// C[bh][b][c] = alpha * sum_a X[bh][a][b] * Y[bh][a][c]  (X: [Nc, Nc], Y: [Nc, D]).
// CTA: 32 output rows b x D columns; threads: 32 x 8, each 4 rows x D/8 cols.
template <int D>
__global__ void __launch_bounds__(256) coarse_atb(const float* __restrict__ X, const float* __restrict__ Y, int Nc,
                                                  float alpha, float* __restrict__ C) {
  __shared__ float sX[32][33];
  __shared__ float sY[32][D + 4];
  const int64_t bh = blockIdx.y;
  const int b0 = blockIdx.x * 32;
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;  // tx: column group, ty: row group
  constexpr int CPT = D / 32;                               // columns per thread
  float acc[4][CPT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int k = 0; k < CPT; ++k) acc[i][k] = 0.f;
  const float* Xb = X + bh * static_cast<int64_t>(Nc) * Nc;
  const float* Yb = Y + bh * static_cast<int64_t>(Nc) * D;
  for (int a0 = 0; a0 < Nc; a0 += 32) {
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * 32; e += 256) {
      int ar = e / 32, bc = e % 32;
      sX[ar][bc] = (a0 + ar < Nc && b0 + bc < Nc) ? Xb[static_cast<int64_t>(a0 + ar) * Nc + b0 + bc] : 0.f;
    }
    for (int e = threadIdx.x; e < 32 * D; e += 256) {
      int ar = e / D, ch = e % D;
      sY[ar][ch] = (a0 + ar < Nc) ? Yb[static_cast<int64_t>(a0 + ar) * D + ch] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int ar = 0; ar < 32; ++ar) {
      float xv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = sX[ar][ty * 4 + i];
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        float yv = sY[ar][tx + 32 * k];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][k] = fmaf(xv[i], yv, acc[i][k]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int b = b0 + ty * 4 + i;
    if (b >= Nc) continue;
#pragma unroll
    for (int k = 0; k < CPT; ++k) C[(bh * Nc + b) * D + tx + 32 * k] = alpha * acc[i][k];
  }
}

// ---------------------------------------------------------------- finalize
struct FinalizeArgs {
  const float* fine[3];
  const float* pooled[3];
  void* out[3];
};

template <int D>
__global__ void __launch_bounds__(256) finalize_kernel(FinalizeArgs a, int grad_dtype, int Nc, int H, int W, int N) {
  constexpr int kChunks = D / 8, kTok = 256 / kChunks, kPasses = kCube / kTok;
  const int t = blockIdx.y;
  const int64_t cg = blockIdx.x;
  const int64_t bh = cg / Nc;
  const int cube = static_cast<int>(cg % Nc);
  const int j = threadIdx.x % kChunks, o0 = threadIdx.x / kChunks;
  float c[8];
  load8_f32(a.pooled[t], cg * D + j * 8, c);
#pragma unroll
  for (int e = 0; e < 8; ++e) c[e] *= (1.0f / kCube);
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int o = o0 + p * kTok;
    const int64_t nat = bh * N + native_token(cube, o, H, W);
    const int64_t cub = bh * N + static_cast<int64_t>(cube) * kCube + o;
    float f[8];
    load8_f32(a.fine[t], cub * D + j * 8, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] += c[e];
    store8(a.out[t], nat * D + j * 8, f, grad_dtype);
  }
}

}  // namespace

int launch_combine(const float* oc, const float* of, const void* gc, const void* gf, void* out, int out_dtype, int BH,
                   int d, int T, int H, int W, cudaStream_t s) {
  const int N = T * H * W, Nc = N / kCube;
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(BH) * Nc);
  auto g = static_cast<const __nv_bfloat16*>(gc);
  auto f = static_cast<const __nv_bfloat16*>(gf);
  timing_mark(VSA_K_COMBINE, true, s);
  if (d == 128)
    combine_kernel<128><<<grid, 256, 0, s>>>(oc, of, g, f, out, out_dtype, Nc, H, W, N);
  else
    combine_kernel<64><<<grid, 256, 0, s>>>(oc, of, g, f, out, out_dtype, Nc, H, W, N);
  timing_mark(VSA_K_COMBINE, false, s);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

int launch_bwd_prep(const void* dout, const void* gc, const void* gf, const float* oc, const float* of,
                    __half* dof, float* delta, float* doc, void* dgc, void* dgf, int grad_dtype, int BH, int d,
                    int T, int H, int W, cudaStream_t s) {
  const int N = T * H * W, Nc = N / kCube;
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(BH) * Nc);
  auto dO = static_cast<const __nv_bfloat16*>(dout);
  auto g = static_cast<const __nv_bfloat16*>(gc);
  auto f = static_cast<const __nv_bfloat16*>(gf);
  timing_mark(VSA_K_BWD_PREP, true, s);
  if (d == 128)
    bwd_prep_kernel<128><<<grid, 256, 0, s>>>(dO, g, f, oc, of, dof, delta, doc, dgc, dgf, grad_dtype, Nc, H, W, N,
                                              device_error_word());
  else
    bwd_prep_kernel<64><<<grid, 256, 0, s>>>(dO, g, f, oc, of, dof, delta, doc, dgc, dgf, grad_dtype, Nc, H, W, N,
                                             device_error_word());
  timing_mark(VSA_K_BWD_PREP, false, s);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

size_t coarse_bwd_smem(int R, int Nc, int d) {
  return sizeof(float) * (2 * R * d + 2 * R * Nc + kCChunk * (d + 4));
}

int launch_coarse_bwd(const float* qc, const float* kc, const float* vc, const float* doc, const float* lse_c, int BH,
                      int Nc, int d, float scale, float* P, float* dS, float* dqc, float* dkc, float* dvc,
                      cudaStream_t s) {
  int R = 16;
  while (R > 1 && (coarse_bwd_smem(R, Nc, d) > 200 * 1024 || R * d / 4 > 4 * kCT)) R >>= 1;
  const size_t smem = coarse_bwd_smem(R, Nc, d);
  if (smem > 200 * 1024) return VSA_ERR_UNSUPPORTED;
  dim3 grid((Nc + R - 1) / R, BH);
  dim3 g2((Nc + 31) / 32, BH);
  timing_mark(VSA_K_COARSE_BWD, true, s);
  if (d == 128) {
    if (cudaFuncSetAttribute(coarse_bwd_rows<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return VSA_ERR_CUDA;
    coarse_bwd_rows<128><<<grid, kCT, smem, s>>>(qc, kc, vc, doc, lse_c, Nc, R, scale, P, dS, dqc);
    coarse_atb<128><<<g2, 256, 0, s>>>(dS, qc, Nc, scale, dkc);
    coarse_atb<128><<<g2, 256, 0, s>>>(P, doc, Nc, 1.0f, dvc);
  } else {
    if (cudaFuncSetAttribute(coarse_bwd_rows<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return VSA_ERR_CUDA;
    coarse_bwd_rows<64><<<grid, kCT, smem, s>>>(qc, kc, vc, doc, lse_c, Nc, R, scale, P, dS, dqc);
    coarse_atb<64><<<g2, 256, 0, s>>>(dS, qc, Nc, scale, dkc);
    coarse_atb<64><<<g2, 256, 0, s>>>(P, doc, Nc, 1.0f, dvc);
  }
  timing_mark(VSA_K_COARSE_BWD, false, s);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

int launch_finalize(const float* dqp, const float* dkp, const float* dvp, const float* dqc, const float* dkc,
                    const float* dvc, void* dq, void* dk, void* dv, int grad_dtype, int BH, int d, int T, int H,
                    int W, cudaStream_t s) {
  const int N = T * H * W, Nc = N / kCube;
  FinalizeArgs a{{dqp, dkp, dvp}, {dqc, dkc, dvc}, {dq, dk, dv}};
  dim3 grid(static_cast<unsigned>(static_cast<int64_t>(BH) * Nc), 3);
  timing_mark(VSA_K_FINALIZE, true, s);
  if (d == 128)
    finalize_kernel<128><<<grid, 256, 0, s>>>(a, grad_dtype, Nc, H, W, N);
  else
    finalize_kernel<64><<<grid, 256, 0, s>>>(a, grad_dtype, Nc, H, W, N);
  timing_mark(VSA_K_FINALIZE, false, s);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace vsa
