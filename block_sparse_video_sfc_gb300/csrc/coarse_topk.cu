// coarse_topk.cu -- coarse cube-to-cube attention and per-query-cube Top-K.
// "VSA: Accelerating Video Diffusion Inference with Sparse Attention on AMD
// GPUs", "Stage 1: Coarse Selection" and "Generating Sparsity Patterns"
// (scores of pooled Q against pooled K; Top-K over the last dimension), and
// the coarse output of "Stage 2: Fine Computation".
//
// One CTA (8 warps) owns R query cubes of one head.  Their fp32 score rows
// (R x Nc) stay in shared memory; pooled K and V stream through in chunks of
// 32 cubes.  Each warp then selects its rows' Top-K: a 4-pass radix select
// finds the K-th largest score, a ballot-ordered compaction keeps every score
// above it plus the lowest-id ties, and a bitonic sort orders the picks by
// (score descending, id ascending).  The softmax and O_c = P Vc follow.
// All arithmetic is fp32 on the SIMT units (<= 4*Nc^2*d FLOP per head).
#include "common.cuh"

namespace vsa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 32;

__device__ __forceinline__ uint32_t orderable(float f) {
  uint32_t b = __float_as_uint(f);
  if (f == 0.0f) b = 0;  // +0 and -0 compare equal
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct CoarseSmem {
  int R, Kpad, D, Nc;
  __host__ __device__ size_t q_off() const { return 0; }
  __host__ __device__ size_t s_off() const { return q_off() + sizeof(float) * R * D; }
  __host__ __device__ size_t kv_off() const { return s_off() + sizeof(float) * R * Nc; }
  __host__ __device__ size_t hist_off() const { return kv_off() + sizeof(float) * kChunk * (D + 4); }
  __host__ __device__ size_t sort_off() const { return hist_off() + sizeof(uint32_t) * kWarps * 256; }
  __host__ __device__ size_t total() const { return sort_off() + sizeof(uint64_t) * kWarps * Kpad; }
};

// Selects the K largest entries of row s[0..Nc) into out[0..K), highest score
// first, ties to the lower index.  Executed by one full warp.
__device__ void warp_topk(const float* s, int Nc, int K, int Kpad, uint32_t* hist, uint64_t* buf, int32_t* out) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t prefix = 0, pmask = 0;
  int k = K;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = lane; b < 256; b += 32) hist[b] = 0;
    __syncwarp();
    for (int j = lane; j < Nc; j += 32) {
      uint32_t u = orderable(s[j]);
      if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
    }
    __syncwarp();
    // lane L owns bins 255-8L .. 248-8L (descending order)
    uint32_t c[8], local = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[i] = hist[255 - 8 * lane - i];
      local += c[i];
    }
    uint32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    uint32_t excl = incl - local;
    bool here = excl < static_cast<uint32_t>(k) && static_cast<uint32_t>(k) <= incl;
    uint32_t who = __ballot_sync(0xffffffffu, here);
    int src = __ffs(who) - 1;
    uint32_t bin = 0, above = 0;
    if (lane == src) {
      uint32_t run = excl;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (run + c[i] >= static_cast<uint32_t>(k)) {
          bin = 255 - 8 * lane - i;
          above = run;
          break;
        }
        run += c[i];
      }
    }
    bin = __shfl_sync(0xffffffffu, bin, src);
    above = __shfl_sync(0xffffffffu, above, src);
    k -= static_cast<int>(above);
    prefix |= bin << shift;
    pmask |= 255u << shift;
    __syncwarp();
  }
  const uint32_t thr = prefix;  // the K-th largest key; k ties at thr are taken
  int nsel = 0, eq_seen = 0;
  for (int base = 0; base < Nc; base += 32) {
    int j = base + lane;
    bool valid = j < Nc;
    uint32_t u = valid ? orderable(s[j]) : 0u;
    bool gt = valid && u > thr;
    bool eq = valid && u == thr;
    uint32_t eqm = __ballot_sync(0xffffffffu, eq);
    int eqrank = __popc(eqm & lt_mask);
    bool take = gt || (eq && eq_seen + eqrank < k);
    uint32_t tm = __ballot_sync(0xffffffffu, take);
    if (take) buf[nsel + __popc(tm & lt_mask)] = (static_cast<uint64_t>(u) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(j));
    nsel += __popc(tm);
    eq_seen += __popc(eqm);
  }
  for (int i = nsel + lane; i < Kpad; i += 32) buf[i] = 0;
  __syncwarp();
  for (int size = 2; size <= Kpad; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = lane; i < Kpad; i += 32) {
        int p = i ^ stride;
        if (p > i) {
          uint64_t a = buf[i], b = buf[p];
          bool desc = (i & size) == 0;
          if (desc ? (a < b) : (a > b)) {
            buf[i] = b;
            buf[p] = a;
          }
        }
      }
      __syncwarp();
    }
  }
  for (int i = lane; i < K; i += 32) out[i] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(buf[i] & 0xFFFFFFFFu));
  __syncwarp();
}

template <int D>
__global__ void __launch_bounds__(kThreads) coarse_topk_kernel(const float* __restrict__ qc, const float* __restrict__ kc,
                                                               const float* __restrict__ vc, int Nc, int K, int R,
                                                               int Kpad, float scale, float* __restrict__ oc,
                                                               float* __restrict__ lse_c, int32_t* __restrict__ idx,
                                                               int32_t* __restrict__ cnt, float* __restrict__ scores) {
  extern __shared__ __align__(16) uint8_t smem[];
  CoarseSmem L{R, Kpad, D, Nc};
  float* sQ = reinterpret_cast<float*>(smem + L.q_off());
  float* sS = reinterpret_cast<float*>(smem + L.s_off());
  float* sKV = reinterpret_cast<float*>(smem + L.kv_off());
  uint32_t* sHist = reinterpret_cast<uint32_t*>(smem + L.hist_off());
  uint64_t* sSort = reinterpret_cast<uint64_t*>(smem + L.sort_off());
  constexpr int KVS = D + 4;  // padded row stride of the K/V chunk
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t bh = blockIdx.y;
  const int row0 = blockIdx.x * R;
  const float* Kb = kc + bh * static_cast<int64_t>(Nc) * D;
  const float* Vb = vc ? vc + bh * static_cast<int64_t>(Nc) * D : nullptr;

  for (int e = tid; e < R * D / 4; e += kThreads) {
    int r = e / (D / 4), c4 = e % (D / 4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + r < Nc) v = reinterpret_cast<const float4*>(qc + (bh * Nc + row0 + r) * D)[c4];
    reinterpret_cast<float4*>(sQ + r * D)[c4] = v;
  }
  // ---- scores: sS[r][j] = scale * Qc[r] . Kc[j]
  for (int kb = 0; kb < Nc; kb += kChunk) {
    __syncthreads();
    for (int e = tid; e < kChunk * D / 4; e += kThreads) {
      int r = e / (D / 4), c4 = e % (D / 4);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kb + r < Nc) v = reinterpret_cast<const float4*>(Kb + static_cast<int64_t>(kb + r) * D)[c4];
      *reinterpret_cast<float4*>(sKV + r * KVS + 4 * c4) = v;
    }
    __syncthreads();
    for (int p = tid; p < R * kChunk; p += kThreads) {
      int r = p / kChunk, j = p % kChunk;
      const float4* q4 = reinterpret_cast<const float4*>(sQ + r * D);
      const float4* k4 = reinterpret_cast<const float4*>(sKV + j * KVS);
      float acc = 0.f;
#pragma unroll 8
      for (int c = 0; c < D / 4; ++c) {
        float4 a = q4[c], b = k4[c];
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
        acc = fmaf(a.z, b.z, acc);
        acc = fmaf(a.w, b.w, acc);
      }
      if (kb + j < Nc) sS[r * Nc + kb + j] = acc * scale;
    }
  }
  __syncthreads();
  // ---- per row: optional score dump, Top-K, softmax statistics, P in place
  for (int r = warp; r < R; r += kWarps) {
    const int row = row0 + r;
    if (row >= Nc) continue;
    float* s = sS + r * Nc;
    const int64_t grow = bh * Nc + row;
    if (scores)
      for (int j = lane; j < Nc; j += 32) scores[grow * Nc + j] = s[j];
    warp_topk(s, Nc, K, Kpad, sHist + warp * 256, sSort + static_cast<size_t>(warp) * Kpad, idx + grow * K);
    if (cnt && lane == 0) cnt[grow] = K;
    float m = -INFINITY;
    for (int j = lane; j < Nc; j += 32) m = fmaxf(m, s[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float l = 0.f;
    for (int j = lane; j < Nc; j += 32) {
      float p = __expf(s[j] - m);
      s[j] = p;
      l += p;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lse_c && lane == 0) lse_c[grow] = m + __logf(l);
    const float inv = 1.0f / l;
    for (int j = lane; j < Nc; j += 32) s[j] *= inv;
  }
  if (!oc) return;
  // ---- O_c = P Vc
  constexpr int kGroups = D / 4;
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int kb = 0; kb < Nc; kb += kChunk) {
    __syncthreads();
    for (int e = tid; e < kChunk * D / 4; e += kThreads) {
      int r = e / (D / 4), c4 = e % (D / 4);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kb + r < Nc) v = reinterpret_cast<const float4*>(Vb + static_cast<int64_t>(kb + r) * D)[c4];
      *reinterpret_cast<float4*>(sKV + r * KVS + 4 * c4) = v;
    }
    __syncthreads();
    const int jmax = min(kChunk, Nc - kb);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int p = tid + i * kThreads;
      if (p >= R * kGroups) break;
      int r = p / kGroups, c4 = p % kGroups;
      const float* prow = sS + r * Nc + kb;
      float4 a = acc[i];
      for (int j = 0; j < jmax; ++j) {
        float w = prow[j];
        float4 v = *reinterpret_cast<const float4*>(sKV + j * KVS + 4 * c4);
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
    int p = tid + i * kThreads;
    if (p >= R * kGroups) break;
    int r = p / kGroups, c4 = p % kGroups;
    if (row0 + r < Nc) reinterpret_cast<float4*>(oc + (bh * Nc + row0 + r) * D)[c4] = acc[i];
  }
}

}  // namespace

int launch_coarse_topk(const float* qc, const float* kc, const float* vc, int BH, int Nc, int d, int topk, float scale,
                       float* oc, float* lse_c, int32_t* idx, int32_t* cnt, float* scores, cudaStream_t s) {
  int Kpad = 32;
  while (Kpad < topk) Kpad <<= 1;
  constexpr size_t kMaxSmem = 200 * 1024;
  int R = 16;
  // R * D / 4 float4 groups must fit 4 per thread in the O_c phase.
  while (R > 1 && (CoarseSmem{R, Kpad, d, Nc}.total() > kMaxSmem || R * d / 4 > 4 * kThreads)) R >>= 1;
  size_t smem = CoarseSmem{R, Kpad, d, Nc}.total();
  if (smem > kMaxSmem) return VSA_ERR_UNSUPPORTED;
  dim3 grid((Nc + R - 1) / R, BH);
  timing_mark(VSA_K_COARSE, true, s);
  if (d == 128) {
    auto k = coarse_topk_kernel<128>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
      return VSA_ERR_CUDA;
    k<<<grid, kThreads, smem, s>>>(qc, kc, vc, Nc, topk, R, Kpad, scale, oc, lse_c, idx, cnt, scores);
  } else {
    auto k = coarse_topk_kernel<64>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
      return VSA_ERR_CUDA;
    k<<<grid, kThreads, smem, s>>>(qc, kc, vc, Nc, topk, R, Kpad, scale, oc, lse_c, idx, cnt, scores);
  }
  timing_mark(VSA_K_COARSE, false, s);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace vsa
