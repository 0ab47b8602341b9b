// fine_fwd.cu -- fine block-sparse attention, forward, on tcgen05 tensor cores.
// "VSA: Accelerating Video Diffusion Inference with Sparse Attention on AMD
// GPUs", "Stage 2: Fine Computation" (token-level attention over the selected
// cubes only), "Kernel Architecture" (QK GEMM with running max M and sum L,
// softmax, PV GEMM accumulated across tiles) and "Sparse Traversal" (walk the
// index list instead of every key block).
//
// GB300 mapping.  The tensor core's full rate needs M = 128 rows and N >= 128
// columns per MMA, while the index list is per 64-token query cube.  One CTA
// therefore owns a PAIR of consecutive query cubes (128 query rows) and walks
// the UNION of their two lists, two key cubes (128 keys) per step; each half
// of the tile masks the cubes its own list does not hold.  Per step:
//   S  = Q K^T         tcgen05.mma, A = Q (smem), B = K (smem), D = TMEM
//   P  = exp2(S - m)   softmax warps, one thread per row, P -> TMEM (fp16)
//   O += P V           tcgen05.mma, A = P (TMEM), B = V (smem, fp16), D = TMEM
// K/V tiles arrive by TMA (128-byte swizzle), one K and one V stage; K(j+1)
// streams in while softmax(j) and PV(j) run.  Each CTA uses 256 TMEM columns
// (S, with P written over it, and O) and ~100 KB of shared memory, so two
// CTAs share an SM and hide each other's latencies.  The running max is only
// raised (and O rescaled) when a row's max grows by more than 2^8, so P <= 256
// and the fp32 accumulators stay exact enough.
// Roles: warp 0 TMA producer, warp 1 MMA issuer, warps 2-5 softmax/epilogue.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100.cuh"

namespace vsa {
namespace {

constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kTmemCols = 256;        // two CTAs share an SM's 512 columns
constexpr uint32_t kColS = 0, kColP = 0, kColO = 128;  // P (fp16) overwrites S

struct FwdParams {
  CUtensorMap tq, tk, tv;  // [BH*N, d] bf16, box {64, 64}, 128B swizzle
  const int32_t* idx;
  const int32_t* cnt;
  int kmax, N, Nc, npairs;
  float scale_log2;  // scale * log2(e)
  void* of;
  int of_dtype;
  float* lse;
  int* err;
};

template <int D>
struct FwdLayout {
  static constexpr int kTile = 128 * D * 2;  // 128 rows x D bf16
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kTile;
  static constexpr int kEnd = kV + kTile;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// F16IN: Q, K, V arrive as fp16; otherwise as bf16, and the softmax warps
// convert each V tile to fp16 in shared memory (exact within +-65504) so that
// P V always runs on fp16 operands (P rounded to 2^-12, not bf16's 2^-9).
// Accumulation is fp32 either way.
template <int D, bool F16IN>
__global__ void __launch_bounds__(kThreads, 2) fine_fwd_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using L = FwdLayout<D>;
  uint32_t* ulist = reinterpret_cast<uint32_t*>(sm + L::kEnd);  // union entries: id | inA<<30 | inB<<31
  const int nwords = (p.Nc + 31) >> 5;
  uint32_t* bitA = ulist + 2 * p.kmax + 2;
  uint32_t* bitB = bitA + nwords;

  // Each barrier completes once per step (bar_q once): K(j) / V(j) loaded,
  // S(j) done, P(j) written (128 softmax threads), PV(j) done.
  __shared__ uint64_t bar_q, bar_k, bar_v, bar_s, bar_p, bar_pv;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int n_union, n_cnt[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int qa = 2 * pair, qb = 2 * pair + 1;
  const bool has_b = qb < p.Nc;

  // ---------------- prologue: barriers, TMEM, union of the two index lists
  if (tid == 0) {
    mbar_init(&bar_q, 1);
    mbar_init(&bar_k, 1);
    mbar_init(&bar_v, 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_p, 128);
    mbar_init(&bar_pv, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  for (int w = tid; w < 2 * nwords; w += kThreads) bitA[w] = 0;  // bitA and bitB are contiguous
  __syncthreads();
  {
    const int64_t rowa = bh * p.Nc + qa;
    int ca = p.cnt ? p.cnt[rowa] : p.kmax;
    int cb = has_b ? (p.cnt ? p.cnt[rowa + 1] : p.kmax) : 0;
    if (ca < 0 || ca > p.kmax || cb < 0 || cb > p.kmax) {
      if (tid == 0) flag_error(p.err, kErrLut);
      ca = min(max(ca, 0), p.kmax);
      cb = min(max(cb, 0), p.kmax);
    }
    if (tid == 0) {
      n_cnt[0] = ca;
      n_cnt[1] = cb;
    }
    const int32_t* la = p.idx + rowa * p.kmax;
    const int32_t* lb = la + p.kmax;
    for (int e = tid; e < ca + cb; e += kThreads) {
      const bool isA = e < ca;
      const int c = isA ? la[e] : lb[e - ca];
      if (c < 0 || c >= p.Nc) {
        flag_error(p.err, kErrLut);
        continue;
      }
      uint32_t* bits = isA ? bitA : bitB;
      uint32_t old = atomicOr(&bits[c >> 5], 1u << (c & 31));
      if (old & (1u << (c & 31))) flag_error(p.err, kErrLut);  // repeated cube in a row
    }
  }
  __syncthreads();
  if (warp == 0) {
    // Visit order: the first (highest-scored) entry of each list, then the
    // rest of the union by increasing cube id.
    const int ca = n_cnt[0], cb = n_cnt[1];
    const int32_t* la = p.idx + (bh * p.Nc + qa) * p.kmax;
    int first[2] = {-1, -1};
    int nf = 0;
    if (ca > 0) {
      int c = la[0];
      if (c >= 0 && c < p.Nc) first[nf++] = c;
    }
    if (cb > 0) {
      int c = la[p.kmax];
      if (c >= 0 && c < p.Nc && (nf == 0 || c != first[0])) first[nf++] = c;
    }
    if (lane < nf) {
      int c = first[lane];
      uint32_t ina = (bitA[c >> 5] >> (c & 31)) & 1u, inb = (bitB[c >> 5] >> (c & 31)) & 1u;
      ulist[lane] = static_cast<uint32_t>(c) | (ina << 30) | (inb << 31);
    }
    int pos = nf;
    for (int w0 = 0; w0 < nwords; w0 += 32) {
      int w = w0 + lane;
      uint32_t a = w < nwords ? bitA[w] : 0u, b = w < nwords ? bitB[w] : 0u;
      uint32_t u = a | b;
      for (int f = 0; f < nf; ++f)
        if ((first[f] >> 5) == w) u &= ~(1u << (first[f] & 31));
      int n = __popc(u), incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      int o = pos + incl - n;
      while (u) {
        int bit = __ffs(u) - 1;
        u &= u - 1;
        uint32_t c = static_cast<uint32_t>(w * 32 + bit);
        ulist[o++] = c | (((a >> bit) & 1u) << 30) | (((b >> bit) & 1u) << 31);
      }
      pos += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) n_union = pos;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int U = n_union;
  const int steps = (U + 1) >> 1;
  const int64_t row_base = bh * p.N;  // first row of this head in the 2D tensor maps

  if (warp == 0) {
    // ---------------- TMA producer: one K stage and one V stage.  K(j) may be
    // loaded once S(j-1) is done with K(j-1); V(j) once PV(j-1) is done.
    if (lane == 0 && steps > 0) {
      tma_prefetch_desc(&p.tq);
      tma_prefetch_desc(&p.tk);
      tma_prefetch_desc(&p.tv);
      mbar_expect_tx(&bar_q, L::kTile);
      for (int b = 0; b < D / 64; ++b)
        for (int h = 0; h < 2; ++h)
          tma_load_2d(sm + L::kQ + b * 16384 + h * 8192, &p.tq, &bar_q, 64 * b,
                      static_cast<int>(row_base + 128 * pair + 64 * h));
      for (int j = 0; j < steps; ++j) {
        const int c0 = ulist[2 * j] & 0x3FFFFFFF;
        const int c1 = (2 * j + 1 < U) ? (ulist[2 * j + 1] & 0x3FFFFFFF) : c0;
        if (j > 0 && !mbar_wait(&bar_s, (j - 1) & 1)) {
          flag_error(p.err, kErrTimeout);
          break;
        }
        mbar_expect_tx(&bar_k, L::kTile);
        for (int b = 0; b < D / 64; ++b) {
          tma_load_2d(sm + L::kK + b * 16384, &p.tk, &bar_k, 64 * b, static_cast<int>(row_base + 64 * c0));
          tma_load_2d(sm + L::kK + b * 16384 + 8192, &p.tk, &bar_k, 64 * b, static_cast<int>(row_base + 64 * c1));
        }
        if (j > 0 && !mbar_wait(&bar_pv, (j - 1) & 1)) {
          flag_error(p.err, kErrTimeout);
          break;
        }
        mbar_expect_tx(&bar_v, L::kTile);
        for (int b = 0; b < D / 64; ++b) {
          tma_load_2d(sm + L::kV + b * 16384, &p.tv, &bar_v, 64 * b, static_cast<int>(row_base + 64 * c0));
          tma_load_2d(sm + L::kV + b * 16384 + 8192, &p.tv, &bar_v, 64 * b, static_cast<int>(row_base + 64 * c1));
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer.  S and P share TMEM columns [0, 128): S(j)
    // is issued only after PV(j-1) has read P(j-1).
    if (lane == 0 && steps > 0) {
      constexpr uint32_t idesc_s = idesc_f32acc(128, 128, 0, 0, F16IN);
      constexpr uint32_t idesc_pv = idesc_f32acc(128, D, 0, 1, 1);
      bool ok = mbar_wait(&bar_q, 0);
      for (int j = 0; j < steps && ok; ++j) {
        ok = ok && mbar_wait(&bar_k, j & 1);
        if (j > 0) ok = ok && mbar_wait(&bar_pv, (j - 1) & 1);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int b = kk >> 2, w = kk & 3;
          uint64_t ad = sdesc_sw128(smem_u32(sm + L::kQ + b * 16384 + w * 32), 16, 1024);
          uint64_t bd = sdesc_sw128(smem_u32(sm + L::kK + b * 16384 + w * 32), 16, 1024);
          mma_ss(tmem + kColS, ad, bd, idesc_s, kk > 0);
        }
        mma_commit(&bar_s);
        ok = ok && mbar_wait(&bar_p, j & 1);
        ok = ok && mbar_wait(&bar_v, j & 1);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint64_t bd = sdesc_sw128(smem_u32(sm + L::kV + kk * 2048), 16384, 1024);
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem + kColO),
              "r"(tmem + kColP + kk * 8), "l"(bd), "r"(idesc_pv), "r"(static_cast<uint32_t>(j > 0 || kk > 0)));
        }
        mma_commit(&bar_pv);
      }
      if (!ok) flag_error(p.err, kErrTimeout);
    }
  } else {
    // ---------------- softmax + epilogue: one thread per query row.  The two
    // 64-column halves of S are the step's two key cubes.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // TMEM lane == tile row
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t my_bit = row < 64 ? 30u : 31u;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < steps; ++j) {
      // S(j) done implies PV(j-1) done: O may be rescaled without another wait.
      if (!mbar_wait(&bar_s, j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t e0 = ulist[2 * j];
      const uint32_t e1 = (2 * j + 1 < U) ? ulist[2 * j + 1] : 0u;
      const bool vh[2] = {((e0 >> my_bit) & 1u) != 0, ((e1 >> my_bit) & 1u) != 0};
      // pass 1: row max over the valid halves (warp-uniform loads)
      float mx = -INFINITY;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!__any_sync(0xffffffffu, vh[h])) continue;
        float sv[64];
#pragma unroll
        for (int c = 0; c < 64; c += 16) tmem_ld16(lane_addr + kColS + 64 * h + c, sv + c);
        tmem_wait_ld();
        if (vh[h]) {
#pragma unroll
          for (int c = 0; c < 64; ++c) mx = fmaxf(mx, sv[c]);
        }
      }
      mx *= p.scale_log2;
      // Raise the running max only when it grows by more than the threshold.
      const bool raise = mx > m + kRescaleThreshold;
      const float m_new = raise ? mx : m;
      const bool need_rescale = raise && (l > 0.f);
      if (__any_sync(0xffffffffu, need_rescale)) {
        const float alpha = need_rescale ? fast_exp2(m - m_new) : 1.0f;
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          float ov[16];
          tmem_ld16(lane_addr + kColO + c, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) ov[i] *= alpha;
          tmem_st16(lane_addr + kColO + c, ov);
        }
        tmem_wait_st();
        l *= alpha;
      }
      m = m_new;
      // pass 2: P = exp2(S*scale - m) per half, packed fp16 into TMEM columns
      // [32h, 32h + 32) (over S columns this thread has already read).
      float rs = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float pk[32];
        const bool any = __any_sync(0xffffffffu, vh[h]);
        if (any) {
          float sv[64];
#pragma unroll
          for (int c = 0; c < 64; c += 16) tmem_ld16(lane_addr + kColS + 64 * h + c, sv + c);
          tmem_wait_ld();
          const bool use = vh[h] && m != -INFINITY;
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float a = use ? fast_exp2(fmaf(sv[c], p.scale_log2, -m)) : 0.f;
            const float b = use ? fast_exp2(fmaf(sv[c + 1], p.scale_log2, -m)) : 0.f;
            const uint32_t pp = pack_f16(a, b);
            // The row sum uses the same rounded weights the PV MMA sees, so
            // O / l stays an exact convex combination of V rows.
            rs += f16_lo(pp) + f16_hi(pp);
            pk[c >> 1] = __uint_as_float(pp);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = 0.f;
        }
#pragma unroll
        for (int c = 0; c < 32; c += 16) tmem_st16(lane_addr + kColP + 32 * h + c, pk + c);
      }
      l += rs;
      if (!F16IN) {
        // bf16 V tile -> fp16 in place, before the PV MMA may read it.
        if (!mbar_wait(&bar_v, j & 1)) {
          ok = false;
          break;
        }
        uint4* vt = reinterpret_cast<uint4*>(sm + L::kV);
        const int t128 = threadIdx.x - 64;
        for (int e = t128; e < L::kTile / 16; e += 128) {
          uint4 u = vt[e];
          vt[e] = make_uint4(pack_f16(bf16_lo(u.x), bf16_hi(u.x)), pack_f16(bf16_lo(u.y), bf16_hi(u.y)),
                             pack_f16(bf16_lo(u.z), bf16_hi(u.z)), pack_f16(bf16_lo(u.w), bf16_hi(u.w)));
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_p);
    }
    if (ok && steps > 0 && !mbar_wait(&bar_pv, (steps - 1) & 1)) ok = false;
    if (!ok) flag_error(p.err, kErrTimeout);
    tc_fence_after();
    // ---------------- epilogue: O / l, LSE
    const bool row_valid = row < 64 || has_b;
    const int64_t grow = row_base + 128 * pair + row;
    const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
    for (int c = 0; c < D; c += 16) {
      float ov[16];
      if (steps > 0) {
        tmem_ld16(lane_addr + kColO + c, ov);
        tmem_wait_ld();
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) ov[i] = (steps > 0 && ok) ? ov[i] * inv : 0.f;
      if (row_valid) {
        store8(p.of, grow * D + c, ov, p.of_dtype);
        store8(p.of, grow * D + c + 8, ov + 8, p.of_dtype);
      }
    }
    if (row_valid && p.lse) p.lse[grow] = (l > 0.f) ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

}  // namespace

// 2D bf16 / fp16 tensor map over [rows, d] with a {64, 64} box and 128-byte swizzle.
int make_tile_map(void* map_out, const void* base, int64_t rows, int d, int f16) {
  CUtensorMap* map = static_cast<CUtensorMap*>(map_out);
  auto enc = get_encoder();
  if (!enc) return VSA_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VSA_OK : VSA_ERR_CUDA;
}

int launch_fine_fwd(const void* qp, const void* kp, const void* vp, const int32_t* idx, const int32_t* cnt, int kmax,
                    int BH, int N, int d, float scale, void* of, int of_dtype, float* lse, int f16_in,
                    cudaStream_t s) {
  FwdParams p{};
  const int64_t rows = static_cast<int64_t>(BH) * N;
  int st;
  if ((st = make_tile_map(&p.tq, qp, rows, d, f16_in)) != VSA_OK) return st;
  if ((st = make_tile_map(&p.tk, kp, rows, d, f16_in)) != VSA_OK) return st;
  if ((st = make_tile_map(&p.tv, vp, rows, d, f16_in)) != VSA_OK) return st;
  p.idx = idx;
  p.cnt = cnt;
  p.kmax = kmax;
  p.N = N;
  p.Nc = N / kCube;
  p.npairs = (p.Nc + 1) / 2;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.of = of;
  p.of_dtype = of_dtype;
  p.lse = lse;
  p.err = device_error_word();
  const int nwords = (p.Nc + 31) / 32;
  const size_t extra = sizeof(uint32_t) * (2 * kmax + 2 + 2 * nwords);
  dim3 grid(p.npairs, BH);
  auto go = [&](auto kernel, size_t tiles) -> int {
    const size_t smem = tiles + 1024 + extra;
    if (smem > 227 * 1024) return VSA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return VSA_ERR_CUDA;
    timing_mark(VSA_K_FINE_FWD, true, s);
    kernel<<<grid, kThreads, smem, s>>>(p);
    timing_mark(VSA_K_FINE_FWD, false, s);
    return VSA_OK;
  };
  if (d == 128)
    st = f16_in ? go(fine_fwd_kernel<128, true>, FwdLayout<128>::kEnd) : go(fine_fwd_kernel<128, false>, FwdLayout<128>::kEnd);
  else
    st = f16_in ? go(fine_fwd_kernel<64, true>, FwdLayout<64>::kEnd) : go(fine_fwd_kernel<64, false>, FwdLayout<64>::kEnd);
  if (st != VSA_OK) return st;
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace vsa
