// coarse.cu -- the coarse stage: cube-to-cube attention, the per-query-cube
// Top-K, and its backward.
//
// "VSA: Accelerating Video Diffusion Inference with Sparse Attention on AMD
// GPUs", "Stage 1: Coarse Selection" and "Generating Sparsity Patterns"
// (scores of pooled Q against pooled K; torch.topk over the last dimension,
// highest first), and the coarse output of "Stage 2: Fine Computation".
//
// Every product here is a small fp32 matrix product per (batch, head): the
// score matrix S = scale Qc Kc^T (Nc x Nc), O_c = softmax(S) Vc, and in the
// backward dP = dOc Vc^T, dQc = scale dS Kc, dKc = scale dS^T Qc, dVc = P^T dOc.
// They all run through one register-tiled SIMT kernel (coarse_gemm); the
// row-wise steps (Top-K and log-sum-exp of each score row; P and dS of each
// row in the backward) are one warp per row.  The score rows live in a
// caller-provided [BH, Nc, Nc] buffer (12.6 MB for 12 heads of 512 cubes,
// L2-resident between the launches).  All arithmetic is fp32.
#include "common.cuh"

namespace vsa {
namespace {

// ---------------------------------------------------------------- GEMM
// C[bh] (M x N) = alpha * op(A[bh]) * op(B[bh]), row-major operands:
//   kNT: A [M x K], B [N x K]     (C = A B^T)
//   kNN: A [M x K], B [K x N]     (C = A B)
//   kTN: A [K x M], B [K x N]     (C = A^T B)
// With row_lse set (kNN only), every A element is replaced by
// exp(A - row_lse[row]) on load: the softmax of a score row, applied on the fly.
enum { kNT = 0, kNN = 1, kTN = 2 };

struct GemmJob {
  const float* A;
  const float* B;
  float* C;
  const float* row_lse;
  float alpha;
  int op, M, N, K;
  int64_t bsA, bsB, bsC, bsL;  // per-(batch, head) strides in elements
};
constexpr int kMaxJobs = 3;
struct GemmBatch {
  GemmJob job[kMaxJobs];
};

// CTA tile 64 x 64, k-step 16, 256 threads.  Warp w covers rows 16*(w/2)..+15
// and columns 32*(w%2)..+31; lane l computes the 4 x 4 block at rows
// 4*(l/8), columns 4*(l%8) of that.  Per k both operands come from shared
// memory as one float4 each (one wavefront per warp for A and one for B), so
// the 16 FMAs per k keep the FMA pipe, not shared memory, the limit.
constexpr int kBM = 64, kBN = 64, kBK = 16, kGThreads = 256, kSPad = 4;

struct TileRegs {
  float a[4], b[4];
};

// Four consecutive floats from p (all in range: ok), else those of the first
// n (n <= 4, possibly 0) and zeros.
__device__ __forceinline__ void load4(const float* p, int n, float* v) {
  if (n >= 4 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = x.x;
    v[1] = x.y;
    v[2] = x.z;
    v[3] = x.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = i < n ? __ldg(p + i) : 0.f;
  }
}

// Loads this thread's 4 elements of the A tile (rows m0.., k0..) and of the B
// tile into registers; out-of-range elements read 0.
__device__ __forceinline__ void gemm_load(const GemmJob& j, const float* A, const float* B, const float* lse,
                                          int m0, int n0, int k0, TileRegs& r) {
  const int t = threadIdx.x;
  if (j.op == kTN) {  // A is [K x M]: thread -> (k, 4 consecutive m)
    const int k = k0 + (t >> 4), m = m0 + (t & 15) * 4;
    load4(A + static_cast<int64_t>(k) * j.M + m, k < j.K ? min(4, j.M - m) : 0, r.a);
  } else {  // A is [M x K]: thread -> (m, 4 consecutive k)
    const int m = m0 + (t >> 2), k = k0 + (t & 3) * 4;
    const int n = m < j.M ? min(4, j.K - k) : 0;
    load4(A + static_cast<int64_t>(m) * j.K + k, n, r.a);
    if (lse) {
      const float l = m < j.M ? lse[m] : 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) r.a[i] = i < n ? __expf(r.a[i] - l) : 0.f;
    }
  }
  if (j.op == kNT) {  // B is [N x K]: thread -> (n, 4 consecutive k)
    const int n = n0 + (t >> 2), k = k0 + (t & 3) * 4;
    load4(B + static_cast<int64_t>(n) * j.K + k, n < j.N ? min(4, j.K - k) : 0, r.b);
  } else {  // B is [K x N]: thread -> (k, 4 consecutive n)
    const int k = k0 + (t >> 4), n = n0 + (t & 15) * 4;
    load4(B + static_cast<int64_t>(k) * j.N + n, k < j.K ? min(4, j.N - n) : 0, r.b);
  }
}

__device__ __forceinline__ void gemm_store(int op, const TileRegs& r, float (*sA)[kBM + kSPad],
                                           float (*sB)[kBN + kSPad]) {
  const int t = threadIdx.x;
  if (op == kTN) {
    *reinterpret_cast<float4*>(&sA[t >> 4][(t & 15) * 4]) = make_float4(r.a[0], r.a[1], r.a[2], r.a[3]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) sA[(t & 3) * 4 + i][t >> 2] = r.a[i];
  }
  if (op == kNT) {
#pragma unroll
    for (int i = 0; i < 4; ++i) sB[(t & 3) * 4 + i][t >> 2] = r.b[i];
  } else {
    *reinterpret_cast<float4*>(&sB[t >> 4][(t & 15) * 4]) = make_float4(r.b[0], r.b[1], r.b[2], r.b[3]);
  }
}

// grid: (ceil(N/64), ceil(M/64), BH * njobs); blockIdx.z = job * BH + bh.
__global__ void __launch_bounds__(kGThreads) coarse_gemm(GemmBatch batch, int BH) {
  __shared__ __align__(16) float sA[2][kBK][kBM + kSPad];
  __shared__ __align__(16) float sB[2][kBK][kBN + kSPad];
  const GemmJob& j = batch.job[blockIdx.z / BH];
  const int64_t bh = blockIdx.z % BH;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  if (m0 >= j.M || n0 >= j.N) return;
  const float* A = j.A + bh * j.bsA;
  const float* B = j.B + bh * j.bsB;
  const float* lse = j.row_lse ? j.row_lse + bh * j.bsL : nullptr;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rm = (warp >> 1) * 16 + (lane >> 3) * 4, cn = (warp & 1) * 32 + (lane & 7) * 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;

  const int nk = (j.K + kBK - 1) / kBK;
  TileRegs r;
  gemm_load(j, A, B, lse, m0, n0, 0, r);
  gemm_store(j.op, r, sA[0], sB[0]);
  __syncthreads();
  for (int kt = 0; kt < nk; ++kt) {
    const int cur = kt & 1;
    if (kt + 1 < nk) gemm_load(j, A, B, lse, m0, n0, (kt + 1) * kBK, r);
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      const float4 a = *reinterpret_cast<const float4*>(&sA[cur][k][rm]);
      const float4 b = *reinterpret_cast<const float4*>(&sB[cur][k][cn]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][c] = fmaf(av[i], bv[c], acc[i][c]);
    }
    // The other buffer was last read in iteration kt-1, before its barrier.
    if (kt + 1 < nk) gemm_store(j.op, r, sA[cur ^ 1], sB[cur ^ 1]);
    __syncthreads();
  }
  float* C = j.C + bh * j.bsC;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + rm + i;
    if (m >= j.M) continue;
    const int n = n0 + cn;
    float* crow = C + static_cast<int64_t>(m) * j.N;
    if (n + 3 < j.N && (reinterpret_cast<uintptr_t>(crow + n) & 15) == 0) {
      *reinterpret_cast<float4*>(crow + n) =
          make_float4(j.alpha * acc[i][0], j.alpha * acc[i][1], j.alpha * acc[i][2], j.alpha * acc[i][3]);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (n + c < j.N) crow[n + c] = j.alpha * acc[i][c];
    }
  }
}

int launch_gemm(const GemmBatch& b, int njobs, int BH, int M, int N, cudaStream_t s) {
  if (njobs < 1 || njobs > kMaxJobs || static_cast<int64_t>(BH) * njobs > 65535) return VSA_ERR_UNSUPPORTED;
  dim3 grid((N + kBN - 1) / kBN, (M + kBM - 1) / kBM, BH * njobs);
  coarse_gemm<<<grid, kGThreads, 0, s>>>(b, BH);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

// ---------------------------------------------------------------- Top-K rows
constexpr int kRowWarps = 8;

// Float -> unsigned key with the same order (+0 and -0 equal).
__device__ __forceinline__ uint32_t orderable(float f) {
  uint32_t b = __float_as_uint(f);
  if (f == 0.0f) b = 0;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// One warp per score row.  Selection: the K-th largest key is found bit by bit
// (the largest t with #{key >= t} >= K), then every key above it and, in
// ascending id, as many keys equal to it as K still needs are kept.  Order:
// each pick's rank is the number of picks that beat it (higher score, or the
// same score and a lower id), so the row comes out highest first.
// A NaN score has no place in the order: it latches kErrNan (the row is still
// completed, NaN ranking above every number).
__global__ void __launch_bounds__(kRowWarps * 32) topk_rows_kernel(const float* __restrict__ S, int64_t rows, int Nc,
                                                                   int K, int32_t* __restrict__ idx,
                                                                   int32_t* __restrict__ cnt,
                                                                   float* __restrict__ lse, int* err) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + warp;
  if (row >= rows) return;
  const size_t per_warp = (static_cast<size_t>(Nc) * 4 + static_cast<size_t>(K) * 8 + 15) & ~size_t(15);
  uint64_t* picks = reinterpret_cast<uint64_t*>(smem + per_warp * warp);
  uint32_t* keys = reinterpret_cast<uint32_t*>(picks + K);
  const float* s = S + row * Nc;

  float m = -INFINITY;
  bool nan = false;
  for (int j = lane; j < Nc; j += 32) {
    const float v = s[j];
    keys[j] = orderable(v);
    m = fmaxf(m, v);
    nan |= v != v;
  }
  if (__any_sync(0xffffffffu, nan) && lane == 0) flag_error(err, kErrNan);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float l = 0.f;
  for (int j = lane; j < Nc; j += 32) l += __expf(s[j] - m);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  if (lse && lane == 0) lse[row] = m + __logf(l);
  __syncwarp();

  uint32_t thr = 0;
  for (int b = 31; b >= 0; --b) {
    const uint32_t cand = thr | (1u << b);
    unsigned c = 0;
    for (int j = lane; j < Nc; j += 32) c += keys[j] >= cand;
    if (__reduce_add_sync(0xffffffffu, c) >= static_cast<unsigned>(K)) thr = cand;
  }
  unsigned above = 0;
  for (int j = lane; j < Nc; j += 32) above += keys[j] > thr;
  const int need_eq = K - static_cast<int>(__reduce_add_sync(0xffffffffu, above));
  const uint32_t lt = (1u << lane) - 1u;
  int nsel = 0, eq_seen = 0;
  for (int base = 0; base < Nc; base += 32) {
    const int j = base + lane;
    const uint32_t u = j < Nc ? keys[j] : 0u;
    const bool eq = j < Nc && u == thr;
    const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
    const bool take = (j < Nc && u > thr) || (eq && eq_seen + __popc(eqm & lt) < need_eq);
    const uint32_t tm = __ballot_sync(0xffffffffu, take);
    if (take) picks[nsel + __popc(tm & lt)] = (static_cast<uint64_t>(u) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(j));
    nsel += __popc(tm);
    eq_seen += __popc(eqm);
  }
  __syncwarp();
  // nsel == K: the keys above thr number < K and those >= thr number >= K.
  int32_t* out = idx + row * K;
  constexpr int kPer = 8;
  for (int i0 = 0; i0 < K; i0 += 32 * kPer) {
    uint64_t mine[kPer];
    int rank[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int i = i0 + q * 32 + lane;
      mine[q] = i < K ? picks[i] : ~0ull;  // the sentinel is beaten by nothing
      rank[q] = 0;
    }
    for (int jx = 0; jx < K; ++jx) {
      const uint64_t v = picks[jx];
#pragma unroll
      for (int q = 0; q < kPer; ++q) rank[q] += v > mine[q];
    }
#pragma unroll
    for (int q = 0; q < kPer; ++q)
      if (i0 + q * 32 + lane < K)
        out[rank[q]] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(mine[q] & 0xFFFFFFFFu));
  }
  if (cnt && lane == 0) cnt[row] = K;
}

// ---------------------------------------------------------------- backward rows
// Row a of the backward: P = exp(S - lse_c), dS = P (dP - sum_b P dP).  S and
// dP come in the two buffers; P and dS are written over them.
__global__ void __launch_bounds__(kRowWarps * 32) bwd_rows_kernel(float* __restrict__ SP, float* __restrict__ dPdS,
                                                                  const float* __restrict__ lse, int64_t rows,
                                                                  int Nc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + warp;
  if (row >= rows) return;
  float* s = SP + row * Nc;
  float* dp = dPdS + row * Nc;
  const float l = lse[row];
  float dsum = 0.f;
  for (int b = lane; b < Nc; b += 32) dsum = fmaf(__expf(s[b] - l), dp[b], dsum);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
  for (int b = lane; b < Nc; b += 32) {
    const float p = __expf(s[b] - l);
    s[b] = p;
    dp[b] = p * (dp[b] - dsum);
  }
}

GemmJob job(int op, const float* A, const float* B, float* C, float alpha, int M, int N, int K, int64_t bsA,
            int64_t bsB, int64_t bsC, const float* row_lse = nullptr, int64_t bsL = 0) {
  GemmJob j{};
  j.A = A;
  j.B = B;
  j.C = C;
  j.row_lse = row_lse;
  j.alpha = alpha;
  j.op = op;
  j.M = M;
  j.N = N;
  j.K = K;
  j.bsA = bsA;
  j.bsB = bsB;
  j.bsC = bsC;
  j.bsL = bsL;
  return j;
}

}  // namespace

size_t topk_rows_smem(int Nc, int K) {
  return kRowWarps * ((static_cast<size_t>(Nc) * 4 + static_cast<size_t>(K) * 8 + 15) & ~size_t(15));
}

// O_c = softmax(scores) Vc (the row softmax applied as the scores load).
int launch_coarse_oc(const float* scores, const float* lse_c, const float* vc, int BH, int Nc, int d, float* oc,
                     cudaStream_t s) {
  const int64_t nd = static_cast<int64_t>(Nc) * d, nn = static_cast<int64_t>(Nc) * Nc;
  GemmBatch b{};
  b.job[0] = job(kNN, scores, vc, oc, 1.0f, Nc, d, Nc, nn, nd, nd, lse_c, Nc);
  return launch_gemm(b, 1, BH, Nc, d, s);
}

int launch_coarse_topk(const float* qc, const float* kc, const float* vc, int BH, int Nc, int d, int topk, float scale,
                       float* oc, float* lse_c, int32_t* idx, int32_t* cnt, float* scores, cudaStream_t s) {
  const size_t smem = topk_rows_smem(Nc, topk);
  if (smem > 200 * 1024) return VSA_ERR_UNSUPPORTED;
  if (!scores || (oc && (!lse_c || !vc))) return VSA_ERR_ARG;
  const int64_t nd = static_cast<int64_t>(Nc) * d, nn = static_cast<int64_t>(Nc) * Nc, rows = int64_t(BH) * Nc;
  timing_mark(VSA_K_COARSE, true, s);
  GemmBatch b{};
  b.job[0] = job(kNT, qc, kc, scores, scale, Nc, Nc, d, nd, nd, nn);
  int st = launch_gemm(b, 1, BH, Nc, Nc, s);
  if (st != VSA_OK) return st;
  if (cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return VSA_ERR_CUDA;
  topk_rows_kernel<<<static_cast<unsigned>((rows + kRowWarps - 1) / kRowWarps), kRowWarps * 32, smem, s>>>(
      scores, rows, Nc, topk, idx, cnt, lse_c, device_error_word());
  if (cudaGetLastError() != cudaSuccess) return VSA_ERR_CUDA;
  if (oc && (st = launch_coarse_oc(scores, lse_c, vc, BH, Nc, d, oc, s)) != VSA_OK) return st;
  timing_mark(VSA_K_COARSE, false, s);
  return VSA_OK;
}

int launch_coarse_bwd(const float* qc, const float* kc, const float* vc, const float* doc, const float* lse_c, int BH,
                      int Nc, int d, float scale, float* P, float* dS, float* dqc, float* dkc, float* dvc,
                      cudaStream_t s) {
  const int64_t nd = static_cast<int64_t>(Nc) * d, nn = static_cast<int64_t>(Nc) * Nc, rows = int64_t(BH) * Nc;
  timing_mark(VSA_K_COARSE_BWD, true, s);
  GemmBatch b{};
  b.job[0] = job(kNT, qc, kc, P, scale, Nc, Nc, d, nd, nd, nn);   // S
  b.job[1] = job(kNT, doc, vc, dS, 1.0f, Nc, Nc, d, nd, nd, nn);  // dP
  int st = launch_gemm(b, 2, BH, Nc, Nc, s);
  if (st != VSA_OK) return st;
  bwd_rows_kernel<<<static_cast<unsigned>((rows + kRowWarps - 1) / kRowWarps), kRowWarps * 32, 0, s>>>(P, dS, lse_c,
                                                                                                    rows, Nc);
  if (cudaGetLastError() != cudaSuccess) return VSA_ERR_CUDA;
  b.job[0] = job(kNN, dS, kc, dqc, scale, Nc, d, Nc, nn, nd, nd);  // dQc = scale dS Kc
  b.job[1] = job(kTN, dS, qc, dkc, scale, Nc, d, Nc, nn, nd, nd);  // dKc = scale dS^T Qc
  b.job[2] = job(kTN, P, doc, dvc, 1.0f, Nc, d, Nc, nn, nd, nd);   // dVc = P^T dOc
  if ((st = launch_gemm(b, 3, BH, Nc, d, s)) != VSA_OK) return st;
  timing_mark(VSA_K_COARSE_BWD, false, s);
  return VSA_OK;
}

}  // namespace vsa
