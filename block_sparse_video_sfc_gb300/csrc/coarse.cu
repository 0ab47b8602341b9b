// coarse.cu -- the coarse stage: cube-to-cube attention, the per-query-cube
// Top-K, and its backward.
//
// "VSA: Accelerating Video Diffusion Inference with Sparse Attention on AMD
// GPUs", "Stage 1: Coarse Selection" and "Generating Sparsity Patterns"
// (scores of pooled Q against pooled K; torch.topk over the last dimension,
// highest first), and the coarse output of "Stage 2: Fine Computation".
//
// Every product here is a small fp32 product per (batch, head): the score
// rows S = scale Qc Kc^T, O_c = softmax(S) Vc, and in the backward
// dP = dOc Vc^T, dS = P (dP - D) with D = rowsum(P dP) = dOc . O_c (the
// latter computed by the combine backward), dQc = scale dS Kc,
// dKc = scale dS^T Qc, dVc = P^T dOc.  No Nc x Nc matrix is ever stored:
//   coarse_fwd_kernel  a CTA keeps the score rows of 16 query cubes in shared
//                      memory (Kc streamed through in tiles of 128 cubes),
//                      takes each row's log-sum-exp and Top-K there (one warp
//                      per row, radix selection), turns the rows into P and
//                      streams Vc through for O_c;
//   coarse_bwd_kernel  one launch, two kinds of CTA over 16 cubes each: a
//                      key CTA streams every query cube through in tiles of
//                      64 (S^T, dP^T, then dKc and dVc accumulated in
//                      registers), a query CTA every key cube (S, dP, then
//                      dQc).  Both recompute the scores instead of reading
//                      them.
// The products are register-tiled SIMT fp32: a lane owns a 4 x 4 or 4 x 2
// block of the output; the operand layouts in shared memory (row strides of
// 4 or 8 mod 32 floats) make every operand load one wavefront per warp.
// Tiles arrive by cp.async (16 bytes, zero fill past the last cube).
#include <algorithm>

#include "common.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 256, kWarps = kThreads / 32;
constexpr int kRows = 16;      // cubes per CTA
constexpr int kFwdTile = 128;  // key cubes per streamed tile, forward
constexpr int kBwdTile = 64;   // cubes per streamed tile, backward
constexpr int kHist = 256;     // radix histogram bins per warp

// Row stride of the score / probability rows: 8 (mod 32) floats, so that the
// stores of a 4 x 8 lane grid and the float4 loads of 4 rows hit distinct
// banks; the key dimension is padded to whole tiles (zeros past Nc).
__host__ __device__ __forceinline__ int score_ld(int Nc) { return (Nc + kFwdTile - 1) / kFwdTile * kFwdTile + 8; }
constexpr int kProbLd = kBwdTile + 8;

// Float -> unsigned key with the same order (+0 and -0 equal), and back.
__device__ __forceinline__ uint32_t orderable(float f) {
  uint32_t b = __float_as_uint(f);
  if (f == 0.0f) b = 0;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_orderable(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// ---------------------------------------------------------------- tiles
__device__ __forceinline__ void cp_async16(float* dst, const float* src, int src_bytes) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Rows row0 .. row0 + n - 1 of a [rows, D] fp32 matrix into dst [n][D + 4],
// asynchronously; rows at or past `rows` read zero.
template <int D>
__device__ __forceinline__ void load_rows_async(float* dst, const float* src, int row0, int n, int rows) {
  constexpr int kVec = D / 4;
  for (int i = threadIdx.x; i < n * kVec; i += kThreads) {
    const int r = i / kVec, c = (i % kVec) * 4;
    const bool in = row0 + r < rows;
    cp_async16(dst + r * (D + 4) + c, src + static_cast<int64_t>(in ? row0 + r : 0) * D + c, in ? 16 : 0);
  }
}

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }
template <int kk>
__device__ __forceinline__ float comp(const float4& v) {
  return kk == 0 ? v.x : kk == 1 ? v.y : kk == 2 ? v.z : v.w;
}

// acc[i][j] += sum_{k < kdim} A[4 i lda + k] B[8 j ldb + k]  (kdim % 4 == 0).
// A points at the lane's first row (row group lane / 8 of four consecutive
// rows), B at its first column row (lane % 8 of eight consecutive rows).
template <int NT>
__device__ __forceinline__ void mma_nt(float (&acc)[4][NT], const float* A, int lda, const float* B, int ldb,
                                       int kdim) {
#pragma unroll 2
  for (int k = 0; k < kdim; k += 4) {
    float4 a[4], b[NT];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = lds4(A + 4 * i * lda + k);
#pragma unroll
    for (int j = 0; j < NT; ++j) b[j] = lds4(B + 8 * j * ldb + k);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        acc[i][j] = fmaf(a[i].x, b[j].x, acc[i][j]);
        acc[i][j] = fmaf(a[i].y, b[j].y, acc[i][j]);
        acc[i][j] = fmaf(a[i].z, b[j].z, acc[i][j]);
        acc[i][j] = fmaf(a[i].w, b[j].w, acc[i][j]);
      }
  }
}

template <int NT>
__device__ __forceinline__ void load_row(float (&b)[NT], const float* p) {
  if constexpr (NT == 4) {
    const float4 v = lds4(p);
    b[0] = v.x, b[1] = v.y, b[2] = v.z, b[3] = v.w;
  } else if constexpr (NT == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    b[0] = v.x, b[1] = v.y;
  } else {
    b[0] = *p;
  }
}

template <int kk, int NT>
__device__ __forceinline__ void nn_step(float (&acc)[4][NT], const float4 (&a)[4], const float* B) {
  float b[NT];
  load_row<NT>(b, B);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[i][j] = fmaf(comp<kk>(a[i]), b[j], acc[i][j]);
}

// acc[i][j] += sum_{k < kdim} A[4 i lda + k] B[k ldb + j]  (kdim % 4 == 0):
// A as in mma_nt, B at the lane's NT consecutive columns of row 0.
template <int NT>
__device__ __forceinline__ void mma_nn(float (&acc)[4][NT], const float* A, int lda, const float* B, int ldb,
                                       int kdim) {
#pragma unroll 2
  for (int k = 0; k < kdim; k += 4) {
    float4 a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = lds4(A + 4 * i * lda + k);
    nn_step<0, NT>(acc, a, B + (k + 0) * ldb);
    nn_step<1, NT>(acc, a, B + (k + 1) * ldb);
    nn_step<2, NT>(acc, a, B + (k + 2) * ldb);
    nn_step<3, NT>(acc, a, B + (k + 3) * ldb);
  }
}

// ---------------------------------------------------------------- Top-K
// One warp: the K-th largest of keys[0 .. Nc) (orderable keys), by radix
// selection on 8-bit digits from the top: each pass counts the keys that
// share the digits found so far by their next digit (a 256-bin histogram in
// shared memory) and keeps the digit in which the K-th largest falls.  thr
// is that key; need (>= 1) is how many keys equal to thr the Top-K holds.
__device__ void radix_select(const uint32_t* keys, int Nc, int K, uint32_t* hist, uint32_t& thr, int& need) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0, mask = 0;
  int want = K;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    reinterpret_cast<uint4*>(hist)[lane] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(hist)[lane + 32] = make_uint4(0, 0, 0, 0);
    __syncwarp();
    for (int j = lane; j < Nc; j += 32) {
      const uint32_t u = keys[j];
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
    }
    __syncwarp();
    // Lane l owns bins 255 - 8 l - e (e = 0 .. 7), counted from the top.
    const uint4 lo = reinterpret_cast<const uint4*>(hist)[62 - 2 * lane];
    const uint4 hi = reinterpret_cast<const uint4*>(hist)[63 - 2 * lane];
    const int c[8] = {static_cast<int>(hi.w), static_cast<int>(hi.z), static_cast<int>(hi.y), static_cast<int>(hi.x),
                      static_cast<int>(lo.w), static_cast<int>(lo.z), static_cast<int>(lo.y), static_cast<int>(lo.x)};
    int tot = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) tot += c[e];
    int incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    const int excl = incl - tot;
    const uint32_t hit = __ballot_sync(0xffffffffu, excl < want && want <= incl);
    const int src = __ffs(hit) - 1;
    int digit = 0, above = 0;
    if (lane == src) {
      int cum = excl;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (cum + c[e] >= want) {
          digit = 255 - 8 * lane - e;
          above = cum;
          break;
        }
        cum += c[e];
      }
    }
    digit = __shfl_sync(0xffffffffu, digit, src);
    above = __shfl_sync(0xffffffffu, above, src);
    want -= above;
    prefix |= static_cast<uint32_t>(digit) << shift;
    mask |= 255u << shift;
    __syncwarp();
  }
  thr = prefix;
  need = want;
}

// Calls f(position, j) for the Top-K entries in ascending j: every key above
// thr and the first `need` keys equal to it.
template <typename F>
__device__ __forceinline__ void for_each_pick(const uint32_t* keys, int Nc, uint32_t thr, int need, F f) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  int nsel = 0, eq_seen = 0;
  for (int base = 0; base < Nc; base += 32) {
    const int j = base + lane;
    const uint32_t u = j < Nc ? keys[j] : 0u;
    const bool eq = j < Nc && u == thr;
    const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
    const bool take = (j < Nc && u > thr) || (eq && eq_seen + __popc(eqm & lt) < need);
    const uint32_t tm = __ballot_sync(0xffffffffu, take);
    if (take) f(nsel + __popc(tm & lt), j);
    nsel += __popc(tm);
    eq_seen += __popc(eqm);
  }
}

// Highest first, ties to the lower id: each pick's rank is the number of
// picks that beat it.  picks: K entries of scratch (key << 32 | ~id).
__device__ void sorted_picks(const uint32_t* keys, int Nc, int K, uint32_t thr, int need, uint64_t* picks,
                             int32_t* out) {
  const int lane = threadIdx.x & 31;
  for_each_pick(keys, Nc, thr, need, [&](int pos, int j) {
    picks[pos] = (static_cast<uint64_t>(keys[j]) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(j));
  });
  __syncwarp();
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
  __syncwarp();
}

// ---------------------------------------------------------------- forward
// Shared memory (bytes): score rows [16][score_ld], the Q block [16][D + 4],
// and a region used in turn by the streamed Kc / Vc tile [128][D + 4], the
// selecting warps' histograms and (sorted lists) their Top-K scratch, and
// the split partials of O_c.
template <int D>
size_t fwd_smem(int Nc, int K, int sort_warps) {
  const size_t tile = sizeof(float) * kFwdTile * (D + 4);
  const size_t sel = sizeof(uint32_t) * kWarps * kHist + sizeof(uint64_t) * static_cast<size_t>(sort_warps) * K;
  return sizeof(float) * (static_cast<size_t>(kRows) * score_ld(Nc) + kRows * (D + 4)) + std::max(tile, sel);
}

// grid (ceil(Nc / 16), BH).  sort_warps == 0: each list in ascending cube
// id; else highest first, with that many warps selecting (the Top-K scratch
// of each must fit).  scores: null, or [BH, Nc, Nc] to receive the score
// rows as well; oc null skips O_c (then vc may be null).
template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    coarse_fwd_kernel(const float* __restrict__ qc, const float* __restrict__ kc, const float* __restrict__ vc, int Nc,
                      int K, float scale, int sort_warps, float* __restrict__ oc, float* __restrict__ lse_c,
                      int32_t* __restrict__ idx, int32_t* __restrict__ cnt, float* __restrict__ scores, int* err) {
  extern __shared__ __align__(16) float smem[];
  constexpr int ldt = D + 4;
  const int lds = score_ld(Nc);
  float* srow = smem;
  float* qa = srow + kRows * lds;
  float* region = qa + kRows * ldt;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, rg = lane >> 3, cg = lane & 7;
  const int64_t bh = blockIdx.y;
  const int q0 = blockIdx.x * kRows, nr = min(kRows, Nc - q0);
  const float* Kc = kc + bh * Nc * D;
  load_rows_async<D>(qa, qc + bh * Nc * D, q0, kRows, Nc);
  // Score rows: warp w computes keys 16 w .. 16 w + 15 of each tile.
  for (int t0 = 0; t0 < Nc; t0 += kFwdTile) {
    __syncthreads();  // the previous tile is used up
    load_rows_async<D>(region, Kc, t0, kFwdTile, Nc);
    cp_async_wait_all();
    __syncthreads();
    float acc[4][2] = {};
    mma_nt<2>(acc, qa + rg * ldt, ldt, region + (16 * warp + cg) * ldt, ldt, D);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int key = t0 + 16 * warp + cg + 8 * j;
        srow[(rg + 4 * i) * lds + key] = key < Nc ? scale * acc[i][j] : 0.f;
      }
  }
  __syncthreads();
  // Per row (one warp each): log-sum-exp, Top-K, then P in place.
  const int sel_warps = sort_warps ? sort_warps : kWarps;
  if (warp < sel_warps) {
    uint32_t* hist = reinterpret_cast<uint32_t*>(region) + warp * kHist;
    uint64_t* picks = reinterpret_cast<uint64_t*>(region + kWarps * kHist) + static_cast<size_t>(warp) * K;
    for (int r = warp; r < nr; r += sel_warps) {
      float* s = srow + r * lds;
      const int64_t row = bh * Nc + q0 + r;
      if (scores)
        for (int j = lane; j < Nc; j += 32) scores[row * Nc + j] = s[j];
      float m = -INFINITY;
      bool nan = false;
      for (int j = lane; j < Nc; j += 32) {
        m = fmaxf(m, s[j]);
        nan |= s[j] != s[j];
      }
      // A NaN score has no place in the order: it latches kErrNan (the row is
      // still completed, NaN ranking above every number).
      if (__any_sync(0xffffffffu, nan) && lane == 0) flag_error(err, kErrNan);
      m = warp_max(m);
      float l = 0.f;
      for (int j = lane; j < Nc; j += 32) l += __expf(s[j] - m);
      const float lse = m + __logf(warp_sum(l));
      if (lane == 0 && lse_c) lse_c[row] = lse;
      uint32_t* keys = reinterpret_cast<uint32_t*>(s);
      for (int j = lane; j < Nc; j += 32) keys[j] = orderable(s[j]);
      __syncwarp();
      uint32_t thr;
      int need;
      radix_select(keys, Nc, K, hist, thr, need);
      int32_t* out = idx + row * K;
      if (sort_warps)
        sorted_picks(keys, Nc, K, thr, need, picks, out);
      else
        for_each_pick(keys, Nc, thr, need, [&](int pos, int j) { out[pos] = j; });
      if (cnt && lane == 0) cnt[row] = K;
      if (oc)
        for (int j = lane; j < Nc; j += 32) s[j] = __expf(from_orderable(keys[j]) - lse);
      __syncwarp();
    }
  }
  if (!oc) return;
  // O_c = P Vc: warp w owns columns 32 (w % (D / 32)) .. + 31 and a share of
  // the keys of each tile; the shares are summed at the end.
  constexpr int kColWarps = D / 32, kSplits = kWarps / kColWarps, kPer = kFwdTile / kSplits;
  const int col0 = 32 * (warp % kColWarps), h = warp / kColWarps;
  const float* V = vc + bh * Nc * D;
  float acc[4][4] = {};
  for (int t0 = 0; t0 < Nc; t0 += kFwdTile) {
    __syncthreads();  // histograms / the previous tile are used up
    load_rows_async<D>(region, V, t0, kFwdTile, Nc);
    cp_async_wait_all();
    __syncthreads();
    mma_nn<4>(acc, srow + rg * lds + t0 + h * kPer, lds, region + h * kPer * ldt + col0 + 4 * cg, ldt, kPer);
  }
  __syncthreads();
  float* part = region;  // [kSplits - 1][16][D + 4]
  if (h > 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(part + ((h - 1) * kRows + rg + 4 * i) * ldt + col0 + 4 * cg) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
  __syncthreads();
  if (h == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4 o = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      for (int p = 0; p < kSplits - 1; ++p) {
        const float4 v = lds4(part + (p * kRows + rg + 4 * i) * ldt + col0 + 4 * cg);
        o.x += v.x, o.y += v.y, o.z += v.z, o.w += v.w;
      }
      const int r = rg + 4 * i;
      if (r < nr) *reinterpret_cast<float4*>(oc + (bh * Nc + q0 + r) * D + col0 + 4 * cg) = o;
    }
  }
}

// ---------------------------------------------------------------- backward
// Shared memory (bytes): the CTA's two blocks [16][D + 4], two streamed
// tiles [64][D + 4], the P and dS tiles [16][72], and the streamed query
// cubes' log-sum-exp and D.
template <int D>
constexpr size_t bwd_smem() {
  return sizeof(float) * (2 * kRows * (D + 4) + 2 * kBwdTile * (D + 4) + 2 * kRows * kProbLd + 2 * kBwdTile);
}

// Key CTA: dKc and dVc of key cubes r0 .. r0 + 15.  Warps 0-3 compute S^T
// (then P^T) and accumulate dKc; warps 4-7 compute dP^T (then dS^T) and
// accumulate dVc.
template <int D>
__device__ __forceinline__ void bwd_keys(const float* Q, const float* Kc, const float* V, const float* G,
                                         const float* lse, const float* delta, int Nc, float scale, int r0,
                                         float* dk, float* dv, float* smem) {
  constexpr int ldt = D + 4, kNk = D / 32;
  float* a1 = smem;
  float* a2 = a1 + kRows * ldt;
  float* t1 = a2 + kRows * ldt;
  float* t2 = t1 + kBwdTile * ldt;
  float* pt = t2 + kBwdTile * ldt;
  float* dt = pt + kRows * kProbLd;
  float* sl = dt + kRows * kProbLd;
  float* sd = sl + kBwdTile;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, rg = lane >> 3, cg = lane & 7;
  const int half = warp >> 2, w4 = warp & 3;
  load_rows_async<D>(a1, Kc, r0, kRows, Nc);
  load_rows_async<D>(a2, V, r0, kRows, Nc);
  const int col0 = w4 * (D / 4) + kNk * cg;
  float acc[4][kNk] = {};
  for (int t0 = 0; t0 < Nc; t0 += kBwdTile) {
    __syncthreads();  // the previous tiles are used up
    load_rows_async<D>(t1, Q, t0, kBwdTile, Nc);
    load_rows_async<D>(t2, G, t0, kBwdTile, Nc);
    if (tid < kBwdTile) {
      const bool in = t0 + tid < Nc;
      sl[tid] = in ? lse[t0 + tid] : INFINITY;  // past the last query cube: P = 0
      sd[tid] = in ? delta[t0 + tid] : 0.f;
    }
    cp_async_wait_all();
    __syncthreads();
    float x[4][2] = {};
    mma_nt<2>(x, (half ? a2 : a1) + rg * ldt, ldt, (half ? t2 : t1) + (16 * w4 + cg) * ldt, ldt, D);
    if (half == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int q = 16 * w4 + cg + 8 * j;
          pt[(rg + 4 * i) * kProbLd + q] = __expf(scale * x[i][j] - sl[q]);
        }
    }
    __syncthreads();
    if (half == 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int q = 16 * w4 + cg + 8 * j, e = (rg + 4 * i) * kProbLd + q;
          dt[e] = pt[e] * (x[i][j] - sd[q]);
        }
    }
    __syncthreads();
    // dKc += dS^T Q (warps 0-3), dVc += P^T dOc (warps 4-7).
    mma_nn<kNk>(acc, (half ? pt : dt) + rg * kProbLd, kProbLd, (half ? t2 : t1) + col0, ldt, kBwdTile);
  }
  float* dst = half ? dv : dk;
  const float f = half ? 1.f : scale;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + rg + 4 * i;
    if (r < Nc)
#pragma unroll
      for (int j = 0; j < kNk; ++j) dst[static_cast<int64_t>(r) * D + col0 + j] = f * acc[i][j];
  }
}

// Query CTA: dQc of query cubes r0 .. r0 + 15.  Warps 0-3 compute S (then
// P), warps 4-7 dP (then dS); all eight accumulate dQc.
template <int D>
__device__ __forceinline__ void bwd_queries(const float* Q, const float* Kc, const float* V, const float* G,
                                            const float* lse, const float* delta, int Nc, float scale, int r0,
                                            float* dq, float* smem) {
  constexpr int ldt = D + 4, kNq = D / 64;
  float* a1 = smem;
  float* a2 = a1 + kRows * ldt;
  float* t1 = a2 + kRows * ldt;
  float* t2 = t1 + kBwdTile * ldt;
  float* pt = t2 + kBwdTile * ldt;
  float* dt = pt + kRows * kProbLd;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, rg = lane >> 3, cg = lane & 7;
  const int half = warp >> 2, w4 = warp & 3;
  load_rows_async<D>(a1, Q, r0, kRows, Nc);
  load_rows_async<D>(a2, G, r0, kRows, Nc);
  float own_l[4], own_d[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + rg + 4 * i;
    own_l[i] = r < Nc ? lse[r] : 0.f;
    own_d[i] = r < Nc ? delta[r] : 0.f;
  }
  const int col0 = warp * (D / 8) + kNq * cg;
  float acc[4][kNq] = {};
  for (int t0 = 0; t0 < Nc; t0 += kBwdTile) {
    __syncthreads();
    load_rows_async<D>(t1, Kc, t0, kBwdTile, Nc);
    load_rows_async<D>(t2, V, t0, kBwdTile, Nc);
    cp_async_wait_all();
    __syncthreads();
    float x[4][2] = {};
    mma_nt<2>(x, (half ? a2 : a1) + rg * ldt, ldt, (half ? t2 : t1) + (16 * w4 + cg) * ldt, ldt, D);
    if (half == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int kk = 16 * w4 + cg + 8 * j;
          pt[(rg + 4 * i) * kProbLd + kk] = t0 + kk < Nc ? __expf(scale * x[i][j] - own_l[i]) : 0.f;
        }
    }
    __syncthreads();
    if (half == 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int e = (rg + 4 * i) * kProbLd + 16 * w4 + cg + 8 * j;
          dt[e] = pt[e] * (x[i][j] - own_d[i]);
        }
    }
    __syncthreads();
    mma_nn<kNq>(acc, dt + rg * kProbLd, kProbLd, t1 + col0, ldt, kBwdTile);  // dQc += dS Kc
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + rg + 4 * i;
    if (r < Nc)
#pragma unroll
      for (int j = 0; j < kNq; ++j) dq[static_cast<int64_t>(r) * D + col0 + j] = scale * acc[i][j];
  }
}

// grid (2 ceil(Nc / 16), BH): the key CTAs first, then the query CTAs.
template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    coarse_bwd_kernel(const float* __restrict__ qc, const float* __restrict__ kc, const float* __restrict__ vc,
                      const float* __restrict__ doc, const float* __restrict__ lse_c,
                      const float* __restrict__ delta_c, int Nc, float scale, float* __restrict__ dqc,
                      float* __restrict__ dkc, float* __restrict__ dvc) {
  extern __shared__ __align__(16) float smem[];
  const int64_t bh = blockIdx.y, off = bh * Nc * D;
  const int nb = (Nc + kRows - 1) / kRows;
  if (static_cast<int>(blockIdx.x) < nb)
    bwd_keys<D>(qc + off, kc + off, vc + off, doc + off, lse_c + bh * Nc, delta_c + bh * Nc, Nc, scale,
                blockIdx.x * kRows, dkc + off, dvc + off, smem);
  else
    bwd_queries<D>(qc + off, kc + off, vc + off, doc + off, lse_c + bh * Nc, delta_c + bh * Nc, Nc, scale,
                   (blockIdx.x - nb) * kRows, dqc + off, smem);
}

constexpr size_t kSmemLimit = 226 * 1024;  // of the 227 KB per block; the static shared memory is a few words

template <int D>
int fwd_launch(const float* qc, const float* kc, const float* vc, int BH, int Nc, int topk, float scale, bool sorted,
               float* oc, float* lse_c, int32_t* idx, int32_t* cnt, float* scores, cudaStream_t s) {
  int sort_warps = 0;
  if (sorted) {  // as many selecting warps as have room for their scratch
    sort_warps = kWarps;
    while (sort_warps > 1 && fwd_smem<D>(Nc, topk, sort_warps) > kSmemLimit) sort_warps >>= 1;
  }
  const size_t smem = fwd_smem<D>(Nc, topk, sort_warps);
  if (smem > kSmemLimit) return VSA_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(coarse_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return VSA_ERR_CUDA;
  dim3 grid((Nc + kRows - 1) / kRows, BH);
  coarse_fwd_kernel<D><<<grid, kThreads, smem, s>>>(qc, kc, vc, Nc, topk, scale, sort_warps, oc, lse_c, idx, cnt,
                                                    scores, device_error_word());
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

template <int D>
int bwd_launch(const float* qc, const float* kc, const float* vc, const float* doc, const float* lse_c,
               const float* delta_c, int BH, int Nc, float scale, float* dqc, float* dkc, float* dvc,
               cudaStream_t s) {
  constexpr size_t smem = bwd_smem<D>();
  if (cudaFuncSetAttribute(coarse_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return VSA_ERR_CUDA;
  dim3 grid(2 * ((Nc + kRows - 1) / kRows), BH);
  coarse_bwd_kernel<D><<<grid, kThreads, smem, s>>>(qc, kc, vc, doc, lse_c, delta_c, Nc, scale, dqc, dkc, dvc);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace

bool coarse_fits(int Nc, int d, int topk, int sorted) {
  const int w = sorted ? 1 : 0;
  return (d == 128 ? fwd_smem<128>(Nc, topk, w) : fwd_smem<64>(Nc, topk, w)) <= kSmemLimit;
}

int launch_coarse_topk(const float* qc, const float* kc, const float* vc, int BH, int Nc, int d, int topk, float scale,
                       int sorted, float* oc, float* lse_c, int32_t* idx, int32_t* cnt, float* scores,
                       cudaStream_t s) {
  if (oc && (!lse_c || !vc)) return VSA_ERR_ARG;
  if (BH > 65535) return VSA_ERR_UNSUPPORTED;
  timing_mark(VSA_K_COARSE, true, s);
  const int st = d == 128 ? fwd_launch<128>(qc, kc, vc, BH, Nc, topk, scale, sorted != 0, oc, lse_c, idx, cnt, scores, s)
                          : fwd_launch<64>(qc, kc, vc, BH, Nc, topk, scale, sorted != 0, oc, lse_c, idx, cnt, scores, s);
  timing_mark(VSA_K_COARSE, false, s);
  return st;
}

int launch_coarse_bwd(const float* qc, const float* kc, const float* vc, const float* doc, const float* lse_c,
                      const float* delta_c, int BH, int Nc, int d, float scale, float* dqc, float* dkc, float* dvc,
                      cudaStream_t s) {
  if (BH > 65535) return VSA_ERR_UNSUPPORTED;
  timing_mark(VSA_K_COARSE_BWD, true, s);
  const int st = d == 128 ? bwd_launch<128>(qc, kc, vc, doc, lse_c, delta_c, BH, Nc, scale, dqc, dkc, dvc, s)
                          : bwd_launch<64>(qc, kc, vc, doc, lse_c, delta_c, BH, Nc, scale, dqc, dkc, dvc, s);
  timing_mark(VSA_K_COARSE_BWD, false, s);
  return st;
}

}  // namespace vsa
