// fine_bwd.cu -- gradient of the fine block-sparse attention on tcgen05.
// "VSA: Faster Video Diffusion with Trainable Sparse Attention" (Abstract: VSA
// trains end to end as one differentiable kernel); the forward is the fine
// stage of "VSA: Accelerating Video Diffusion Inference with Sparse Attention
// on AMD GPUs" ("Stage 2: Fine Computation").  The index list is constant.
//
// Per query row i and listed key j (S = scale * Q K^T, P = softmax(S) with the
// forward's LSE, D_i = dO_i . O_i):
//   dV_j += P_ij dO_i,  dP_ij = dO_i . V_j,  dS_ij = P_ij (dP_ij - D_i),
//   dQ_i += scale dS_ij K_j,  dK_j += scale dS_ij Q_i.
//
// GB300 mapping: two kernels, neither of which reduces partial sums through
// global memory (an fp32 reduce-add into L2 runs at only ~3-4 TB/s on GB300,
// which would bound a fused key-stationary kernel's dQ traffic).
//
// fine_bwd_kv_kernel (key-stationary): one CTA owns a PAIR of key cubes (128
// keys; K, V in shared memory; dK, dV accumulated in TMEM) and walks the union
// of the two cubes' inverse lists (the query cubes whose index list holds
// either key cube), one query cube (64 rows) per step, masking the half of
// the tile whose key cube the query cube does not list.  Keys sit on the MMA
// M dimension:
//   S^T = K Q^T, dP^T = V dO^T        (A, B in shared memory)
//   dV += P^T dO, dK += dS^T Q        (A = P^T / dS^T in TMEM)
// One S^T / dP^T buffer, released as soon as the compute warps have read it
// into registers, and two P^T / dS^T buffers: S^T(j + 1) waits only for that
// read, never for an MMA to complete (the MMA issuer is the busy resource: an
// issue returns about when the tensor core takes the instruction, so each
// wait for a completion leaves it idle), and dV / dK(j) run after S^T(j + 1).
// Q and dO go through a 4-stage ring.
//
// fine_bwd_dq_kernel (query-stationary): one CTA owns a pair of query cubes
// (128 rows; Q, dO in shared memory; dQ accumulated in TMEM) and walks the
// union of their index lists two key cubes per step, like the forward:
//   S = Q K^T, dP = dO V^T            (A, B in shared memory)
//   dQ += dS K                        (A = dS in TMEM)
// S and dP are released as soon as the compute warps have read them, so
// S(j+1) and dP(j+1) run while dS(j) is computed; dS is double-buffered.  K
// is read by S(j) and again by dQ(j), a step later, so it has a 3-stage ring;
// V only by dP(j), so one stage suffices: V(j+1) lands while S(j+1) runs.
//
// Operands are fp16 (exact for the bf16 inputs within +-65504), accumulation
// fp32.  The inverse lists (the query cubes whose list holds a key cube) are
// built from the index lists in CSR form, by counting sort (workspace).
//
// Epilogues: each kernel writes its rows once.  For the whole VSA backward
// they also finish the gradient: a row of cube c gets c's coarse-stage
// gradient divided by c's token count (the backward of the mean pool) and
// goes to its native token in the caller's dtype (the inverse reorder), so no
// fp32 copy in cube order is written and read back.
#include <cuda.h>

#include "common.cuh"
#include "sm100.cuh"

namespace vsa {

int make_tile_map(void* map, const void* base, int64_t rows, int d, int f16);

namespace {

// Warp 0: TMA producer; warps 1 and 10: MMA issuers; warps 2-9: two compute
// warpgroups.
constexpr int kThreads = 352;
constexpr int kCompute = 256;

struct BwdParams {
  CUtensorMap tq, tk, tv, tdo;  // fp16 [BH*N, d], box {64, 64}, 128B swizzle
  const uint16_t* dof;          // the same dO_f rows (fp16), read directly into TMEM by the dQ kernel
  const float* lse;             // natural-log LSE per row [BH*N]
  const float* delta;           // D per row [BH*N]
  InverseLists inv;             // CSR inverse lists
  const int32_t* idx;           // forward index list [BH][Nc][kmax]
  const int32_t* cnt;           // [BH][Nc] or null (= kmax)
  float* dq;                    // fp32 rows in cube order (fused == 0)
  float* dk;
  float* dv;
  FusedGrads fused;             // fused pool backward + inverse reorder (fused.dq != null)
  int64_t Nn;                   // tokens of one head's grid (fused)
  const int32_t* qpairs;        // [BH][npairs][2] query-cube tiles of the dQ kernel, or null (2t, 2t + 1)
  const int32_t* kpairs;        // [BH][npairs][2] key-cube tiles of the dK/dV kernel, or null
  int N, Nc, nwords, kmax, npairs;
  float scale, scale_log2;
  int* err;
};

// Destination of one gradient row (cube `cube`, slot `slot` of head bh).
// Unfused: the fp32 row in cube order.  Fused: its native token (row -1 for a
// padding slot), and the cube's coarse gradient row with 1 / token count.
struct GradRow {
  void* out;
  int64_t row;
  const float* coarse;
  float inv_tokens;
};
// coarse_row: the cube's coarse gradient row (global or shared memory).
__device__ __forceinline__ GradRow grad_row(const BwdParams& p, void* fused_out, float* cube_out,
                                            const float* coarse_row, int64_t bh, int cube, int slot) {
  if (!fused_out) return GradRow{cube_out, bh * p.N + 64 * static_cast<int64_t>(cube) + slot, nullptr, 0.f};
  const int rc = raster_cube(p.fused.order, cube);
  const int64_t tok = native_token(rc, slot, p.fused.grid);
  return GradRow{fused_out, tok < 0 ? -1 : bh * p.Nn + tok, coarse_row,
                 1.0f / static_cast<float>(cube_tokens(rc, p.fused.grid))};
}
// Columns [c, c + 32) of a gradient row (v is consumed).
template <int D>
__device__ __forceinline__ void store_grad32(const BwdParams& p, const GradRow& g, float* v, int c) {
  if (g.row < 0) return;
  if (!g.coarse) {
#pragma unroll
    for (int i = 0; i < 32; i += 8) store8(g.out, g.row * D + c + i, v + i, VSA_DTYPE_F32);
    return;
  }
#pragma unroll
  for (int i = 0; i < 32; i += 8) {
    float cv[8];
    load8_f32(g.coarse, c + i, cv);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[i + e] += cv[e] * g.inv_tokens;
    store8(g.out, g.row * D + c + i, v + i, p.fused.grad_dtype);
  }
}

// The two cubes of tile `t`: from a pair plan (second -1: none), else 2t and
// 2t + 1.  A plan entry out of range latches kErrLut and leaves one cube.
__device__ __forceinline__ void tile_cubes(const int32_t* plan, int64_t bh, int t, int npairs, int Nc, int* err,
                                           int& a, int& b) {
  a = 2 * t;
  b = 2 * t + 1 < Nc ? 2 * t + 1 : -1;
  if (plan) {
    a = plan[(bh * npairs + t) * 2];
    b = plan[(bh * npairs + t) * 2 + 1];
    if (a < 0 || a >= Nc || b < -1 || b >= Nc) {
      if (threadIdx.x == 0) flag_error(err, kErrLut);
      a = min(max(a, 0), Nc - 1);
      b = -1;
    }
  }
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (one instruction for two lanes of arithmetic).  The
// compute warps' budget per step is set by the special-function pipe (ex2 and
// the f32 -> f16x2 conversion both take 4 clk per warp instruction per SM
// sub-partition on GB300), so the surrounding arithmetic runs as f32x2 and the
// fp16 packs saturate in the conversion itself instead of through min / max.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t f2u(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// exp2 of both lanes.
__device__ __forceinline__ uint64_t exp2x2(uint64_t x) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
  return f2(fast_exp2(a), fast_exp2(b));
}
// Both lanes to an fp16 pair (low lane in the low half), round to nearest,
// saturating at +-65504 (beyond-range values are clamped, never infinite).
__device__ __forceinline__ uint32_t f16x2_sat(uint64_t x) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
  uint32_t h;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(b), "f"(a));
  return h;
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc));
}

// Union of two cube bitmaps as an ascending list: entry = id | inA<<30 | inB<<31.
// Executed by one full warp; returns the length (to every lane).
__device__ int warp_union_list(const uint32_t* bitA, const uint32_t* bitB, int nwords, uint32_t* ulist) {
  const int lane = threadIdx.x & 31;
  int pos = 0;
  for (int w0 = 0; w0 < nwords; w0 += 32) {
    const int w = w0 + lane;
    const uint32_t a = w < nwords ? bitA[w] : 0u, b = w < nwords ? bitB[w] : 0u;
    uint32_t u = a | b;
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
      ulist[o++] = static_cast<uint32_t>(w * 32 + bit) | (((a >> bit) & 1u) << 30) | (((b >> bit) & 1u) << 31);
    }
    pos += __shfl_sync(0xffffffffu, incl, 31);
  }
  return pos;
}

// Loads the two 64-row cubes c0, c1 of a [BH*N, D] tensor into a 128-row
// 128B-swizzled tile ([D/64][128 rows][128 B]).
template <int D>
__device__ __forceinline__ void load_cube_pair(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int64_t row_base,
                                               int c0, int c1) {
#pragma unroll
  for (int b = 0; b < D / 64; ++b) {
    tma_load_2d(dst + b * 16384, map, bar, 64 * b, static_cast<int>(row_base + 64 * c0));
    tma_load_2d(dst + b * 16384 + 8192, map, bar, 64 * b, static_cast<int>(row_base + 64 * c1));
  }
}


// =============================================================== dK, dV
// One CTA per pair of key cubes (128 key rows, K and V resident in shared
// memory); it walks the union of the two cubes' inverse lists ONE query cube
// (64 queries) per step:
//   S^T = K Q^T, dP^T = V dO^T       (M = 128 keys, N = 64 queries, SS)
//   P^T = exp2(S^T scale - LSE), dS^T = P^T (dP^T - D)   compute warps
//   dV += P^T dO, dK += dS^T Q       (A from TMEM, N = d)
// With 64-query steps the Q / dO stages are 16 KB each, so the rings are
// four deep (the loads of a step start four steps ahead).  S^T / dP^T are
// released as soon as the compute warps have read them into registers, and
// P^T / dS^T go to one of two separate buffers, so S^T(j+1) and dV(j-1),
// dK(j-1) run while the compute warps work on step j and the tensor pipe
// never drains between steps.  N = 64 SS products run at about two thirds
// of the full rate (shared-memory operand bandwidth); the overlap buys more.
constexpr int kKvStages = 4;
template <int D>
struct KvLayout {
  static constexpr int kTileK = 128 * D * 2;  // K or V: 128 key rows
  static constexpr int kTileQ = 64 * D * 2;   // Q or dO of one query cube
  static constexpr int kK = 0, kV = kTileK, kRing = 2 * kTileK;
  static constexpr int kStage = 2 * kTileQ;   // Q, then dO
  static constexpr int kStats = kRing + kKvStages * kStage;  // [stage][LSE 64 | D 64] fp32
  static constexpr int kEnd = kStats + kKvStages * 512;
};
// TMEM: two step buffers, b = j % 2 at 128 b: S^T(j) in its columns [0, 64)
// and dP^T(j) in [64, 128) (fp32).  Compute warpgroup g reads query columns
// [32 g, 32 g + 32) of S^T and of dP^T and overwrites the first 16 of each
// range with its P^T and dS^T (fp16 pairs): every thread rewrites only
// columns of its own lane that it has itself read, so the two warpgroups
// never touch each other's values.  The dV / dK MMA takes queries
// 16 kk .. 16 kk + 15 from column 32 (kk / 2) + 8 (kk % 2).  dV at 256, dK
// at 384.
constexpr uint32_t kKvBuf = 128, kKvDPOff = 64, kKvDV = 256, kKvDK = 384;
template <int D>
constexpr int kKvCoarseBytes = 4 * D * static_cast<int>(sizeof(float));  // crow (fused epilogue)

template <int D>
__global__ void __launch_bounds__(kThreads, 1) fine_bwd_kv_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using L = KvLayout<D>;
  // The coarse dV and dK rows of the two key cubes, [cube][dV, dK][D], read
  // by the fused epilogue (staged here so that it waits on no global load).
  float* crow = reinterpret_cast<float*>(sm + L::kEnd);
  uint32_t* ulist = reinterpret_cast<uint32_t*>(sm + L::kEnd + kKvCoarseBytes<D>);
  uint32_t* bitA = ulist + 2 * p.Nc + 2;
  uint32_t* bitB = bitA + p.nwords;

  // full[s]: Q, dO, LSE and D of the step in stage s landed; stage_free[s]:
  // dK of that step (the last reader of the stage) completed.  For step
  // buffer b = j % 2, whose S^T half and dP^T half are pipelined apart:
  // st_done[b] / dpt_done[b]: S^T(j) / dP^T(j) done; p_ready[b] / ds_ready[b]:
  // P^T(j) / dS^T(j) written over them (all compute threads); st_free[b] /
  // dpt_free[b]: dV(j) / dK(j), which read them, completed, so S^T(j + 2) /
  // dP^T(j + 2) may overwrite that half.  Every parity wait targets a
  // barrier in the awaited phase or the one after it.
  __shared__ uint64_t bar_kv, full[kKvStages], stage_free[kKvStages], st_done[2], dpt_done[2], p_ready[2],
      ds_ready[2], st_free[2], dpt_free[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int n_union;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = blockIdx.x;
  const int64_t bh = blockIdx.y;
  int k1, k2;
  tile_cubes(p.kpairs, bh, pair, p.npairs, p.Nc, p.err, k1, k2);
  const bool has_k2 = k2 >= 0;
  const int64_t row_base = bh * p.N;

  if (tid == 0) {
    mbar_init(&bar_kv, 1);
    for (int i = 0; i < kKvStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&stage_free[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&st_done[i], 1);
      mbar_init(&dpt_done[i], 1);
      mbar_init(&p_ready[i], kCompute);
      mbar_init(&ds_ready[i], kCompute);
      mbar_init(&st_free[i], 1);
      mbar_init(&dpt_free[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  if (p.fused.dk) {
    for (int e = tid; e < 4 * D; e += kThreads) {
      const int kc = e < 2 * D || !has_k2 ? k1 : k2;
      const float* src = (((e / D) & 1) ? p.fused.dkc : p.fused.dvc) + (bh * p.Nc + kc) * D + (e % D);
      crow[e] = *src;
    }
  }
  for (int w = tid; w < 2 * p.nwords; w += kThreads) bitA[w] = 0u;  // bitA and bitB are contiguous
  __syncthreads();
  {
    // The two key cubes' inverse lists as bitmaps of query cubes.
    const int32_t* off = p.inv.off + bh * (p.Nc + 1);
    const int32_t* ids = p.inv.ids + bh * p.inv.stride;
    const int a0 = off[k1], na = off[k1 + 1] - a0;
    const int b0 = has_k2 ? off[k2] : 0, nb = has_k2 ? off[k2 + 1] - b0 : 0;
    for (int e = tid; e < na + nb; e += kThreads) {
      const bool isA = e < na;
      const int q = ids[isA ? a0 + e : b0 + e - na];
      const uint32_t old = atomicOr(&(isA ? bitA : bitB)[q >> 5], 1u << (q & 31));
      if (old & (1u << (q & 31))) flag_error(p.err, kErrLut);  // a list holding this key cube twice
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int n = warp_union_list(bitA, bitB, p.nwords, ulist);
    if (lane == 0) n_union = n;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int steps = n_union;  // one query cube per step

  if (warp == 0) {
    // ---------------- TMA producer: K, V once; then per step the query cube's
    // Q and dO tiles and its 64 LSE and D values into stage j % 4.
    if (lane == 0 && steps > 0) {
      mbar_expect_tx(&bar_kv, 2 * L::kTileK);
      const int c1 = has_k2 ? k2 : k1;
      load_cube_pair<D>(sm + L::kK, &p.tk, &bar_kv, row_base, k1, c1);
      load_cube_pair<D>(sm + L::kV, &p.tv, &bar_kv, row_base, k1, c1);
      for (int j = 0; j < steps; ++j) {
        const int st = j & (kKvStages - 1);
        // A suspended wait: the ring has slack, and a polling producer would
        // take issue slots from the two compute warps on its sub-partition.
        if (j >= kKvStages && !mbar_wait(&stage_free[st], ((j / kKvStages) - 1) & 1)) {
          flag_error(p.err, kErrTimeout);
          break;
        }
        const int q = static_cast<int>(ulist[j] & 0x3FFFFFFF);
        const int64_t qrow = row_base + 64 * static_cast<int64_t>(q);
        uint8_t* stage = sm + L::kRing + st * L::kStage;
        float* stats = reinterpret_cast<float*>(sm + L::kStats + st * 512);
        mbar_expect_tx(&full[st], L::kStage + 512);
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          tma_load_2d(stage + b * 8192, &p.tq, &full[st], 64 * b, static_cast<int>(qrow));
          tma_load_2d(stage + L::kTileQ + b * 8192, &p.tdo, &full[st], 64 * b, static_cast<int>(qrow));
        }
        bulk_load(stats, p.lse + qrow, 256, &full[st]);
        bulk_load(stats + 64, p.delta + qrow, 256, &full[st]);
      }
    }
  } else if (warp == 1 || warp == 10) {
    // ---------------- MMA issuers, each in its own fixed order: warp 1
    // S^T(j) into step buffer j % 2 once dV(j - 2) has read that half, then
    // dP^T(j) once dK(j - 2) has; warp 10 dV(j) once P^T(j) is written, then
    // dK(j) once dS^T(j) is.  The compute warps start on S^T(j) while dP^T(j)
    // runs, and dV(j) runs while they finish dS^T(j).  (An MMA issue
    // holds its thread about as long as the group runs, and a barrier poll
    // costs ~100+ cycles under the tensor core's shared-memory traffic: one
    // thread issuing both kinds leaves the pipe idle between groups.)  The
    // two threads' groups touch disjoint TMEM columns; each thread's commits
    // track its own MMAs.
    if (lane == 0 && steps > 0) {
      constexpr uint32_t idesc_s = idesc_f32acc(128, 64, 0, 0, 1);
      constexpr uint32_t idesc_g = idesc_f32acc(128, D, 0, 1, 1);
      constexpr uint32_t kStageU = L::kStage >> 4, kTileQU = L::kTileQ >> 4;
      bool ok = true;
      if (warp == 1) {
        // Descriptors precomputed: K / V per K-step, the Q / dO stage base
        // (the start-address field is linear in the byte address).
        uint64_t kdesc[D / 16], vdesc[D / 16];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int off = (kk >> 2) * 16384 + (kk & 3) * 32;
          kdesc[kk] = sdesc_sw128(smem_u32(sm + L::kK + off), 16, 1024);
          vdesc[kk] = sdesc_sw128(smem_u32(sm + L::kV + off), 16, 1024);
        }
        const uint64_t qkm0 = sdesc_sw128(smem_u32(sm + L::kRing), 16, 1024);  // Q / dO, K-major
        ok = mbar_spin(&bar_kv, 0);
        for (int j = 0; ok && j < steps; ++j) {
          const int st = j & (kKvStages - 1), b = j & 1;
          const uint32_t ph = ((j >> 1) - 1) & 1;
          if ((j >= 2 && !mbar_spin(&st_free[b], ph)) || !mbar_spin(&full[st], (j / kKvStages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t qd = qkm0 + st * kStageU;
          const uint32_t sb = tmem + kKvBuf * b;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(sb, kdesc[kk], qd + (((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), idesc_s, kk > 0);
          mma_commit(&st_done[b]);
          if (j >= 2 && !mbar_spin(&dpt_free[b], ph)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(sb + kKvDPOff, vdesc[kk], qd + kTileQU + (((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), idesc_s,
                   kk > 0);
          mma_commit(&dpt_done[b]);
        }
      } else {
        const uint64_t qmn0 = sdesc_sw128(smem_u32(sm + L::kRing), 8192, 1024);  // Q / dO, MN-major
        for (int j = 0; ok && j < steps; ++j) {
          const int st = j & (kKvStages - 1), b = j & 1;
          const uint32_t ph = (j >> 1) & 1;
          const uint64_t qd = qmn0 + st * kStageU;
          const uint32_t pb = tmem + kKvBuf * b;
          // A = P^T / dS^T (K = 64 queries in 4 steps of 16), B = dO / Q
          // (MN-major).
          if (!mbar_spin(&p_ready[b], ph)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + kKvDV, pb + 32 * (kk >> 1) + 8 * (kk & 1), qd + kTileQU + ((kk * 2048) >> 4), idesc_g,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&st_free[b]);
          if (!mbar_spin(&ds_ready[b], ph)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + kKvDK, pb + kKvDPOff + 32 * (kk >> 1) + 8 * (kk & 1), qd + ((kk * 2048) >> 4), idesc_g,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&stage_free[st]);
          mma_commit(&dpt_free[b]);
        }
      }
      if (!ok) flag_error(p.err, kErrTimeout);
    }
  } else {
    // ---------------- compute warps: thread = key row r (TMEM lane);
    // warpgroup g takes query columns [32 g, 32 g + 32) of each step.
    const int quarter = warp & 3;
    const int g = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t key_bit = r < 64 ? 30u : 31u;  // warp-uniform
    bool ok = true;
    for (int j = 0; j < steps; ++j) {
      const int st = j & (kKvStages - 1), b = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      // The stage's LSE / D are read from shared memory: wait for its fill
      // too (it has landed once S^T(j) is done, but this makes it visible).
      // The compute warps' waits suspend: a polling warp takes issue slots
      // and memory-pipe bandwidth from the warps beside it, the MMA issuers
      // among them (measured: the backward 1% faster than with polling).
      if (!mbar_wait(&st_done[b], ph) || !mbar_wait(&full[st], (j / kKvStages) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool valid = ((ulist[j] >> key_bit) & 1u) != 0;
      const float* lse = reinterpret_cast<const float*>(sm + L::kStats + st * 512) + 32 * g;
      const float* dlt = lse + 64;
      const uint32_t sb = lane_addr + kKvBuf * b + 32 * g;  // this warpgroup's S^T columns
      // P^T = exp2(log2e (S^T scale - LSE)) = exp2((LSE - scale S^T) (-log2e)),
      // two query columns per packed operation; written over the first 16 of
      // the S^T columns this thread read (its own lane; its loads completed).
      uint64_t pr[16];
      uint32_t pk[16];
      if (valid) {
        uint32_t sv[32];
        tmem_ld32_wait(sb, sv);
        const uint64_t nsc = f2(-p.scale, -p.scale), nl2e = f2(-1.4426950408889634f, -1.4426950408889634f);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(lse + c);
          pr[c >> 1] = exp2x2(mul2(fma2(f2u(sv[c], sv[c + 1]), nsc, f2(l4.x, l4.y)), nl2e));
          pr[(c >> 1) + 1] = exp2x2(mul2(fma2(f2u(sv[c + 2], sv[c + 3]), nsc, f2(l4.z, l4.w)), nl2e));
          pk[c >> 1] = f16x2_sat(pr[c >> 1]);
          pk[(c >> 1) + 1] = f16x2_sat(pr[(c >> 1) + 1]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          pk[i] = 0u;
          pr[i] = 0ull;
        }
      }
      tmem_st8(sb, pk);
      tmem_st8(sb + 8, pk + 8);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_ready[b]);
      // dS^T = P^T (dP^T - D), over the first 16 of this thread's dP^T columns.
      if (!mbar_wait(&dpt_done[b], ph)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t dk[16];
      if (valid) {
        uint32_t dv[32];
        tmem_ld32_wait(sb + kKvDPOff, dv);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(dlt + c);
          dk[c >> 1] = f16x2_sat(mul2(pr[c >> 1], sub2(f2u(dv[c], dv[c + 1]), f2(d4.x, d4.y))));
          dk[(c >> 1) + 1] = f16x2_sat(mul2(pr[(c >> 1) + 1], sub2(f2u(dv[c + 2], dv[c + 3]), f2(d4.z, d4.w))));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) dk[i] = 0u;
      }
      tmem_st8(sb + kKvDPOff, dk);
      tmem_st8(sb + kKvDPOff + 8, dk + 8);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&ds_ready[b]);
    }
    if (ok && steps > 0 && !mbar_spin(&dpt_free[(steps - 1) & 1], ((steps - 1) >> 1) & 1)) ok = false;
    if (!ok) flag_error(p.err, kErrTimeout);
    tc_fence_after();
    // ---------------- dK, dV rows of this key pair (warpgroup 0: dV, 1: dK)
    const bool key_valid = r < 64 || has_k2;
    const int kc = r < 64 || !has_k2 ? k1 : k2;
    const GradRow dst = grad_row(p, g == 0 ? p.fused.dv : p.fused.dk, g == 0 ? p.dv : p.dk,
                                 crow + (2 * (r < 64 ? 0 : 1) + g) * D, bh, kc, r & 63);
    const float mul = g == 0 ? 1.0f : p.scale;
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      uint32_t a[32];
      if (steps > 0 && ok) {
        tmem_ld32_wait(lane_addr + (g == 0 ? kKvDV : kKvDK) + c, a);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] = 0u;
      }
      float o[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(a[i]) * mul;
      if (key_valid) store_grad32<D>(p, dst, o, c);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

// =============================================================== dQ
template <int D>
struct DqLayout {
  static constexpr int kTile = 128 * D * 2;
  // K: 3 stages (read by S(j) and, much later, by dQ(j)); V: 2 stages (read
  // by dP(j) only, so V(j + 1) lands while step j runs).  dO is not here: it
  // is the A operand of dP from TMEM.
  static constexpr int kQ = 0, kK = kTile, kV = 4 * kTile;
  static constexpr int kEnd = 6 * kTile;
};
constexpr int kDqKStages = 3, kDqVStages = 2;
// TMEM: S 0 and dP 128 (128 fp32 columns each, released once the compute
// warps have read them); dS 256 (64 columns of fp16 pairs); dO 320 (D / 2
// columns of fp16 pairs, written once); dQ 384.
constexpr uint32_t kDqS = 0, kDqDP = 128, kDqDS = 256, kDqDO = 320, kDqDQ = 384;

template <int D>
__global__ void __launch_bounds__(kThreads, 1) fine_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using L = DqLayout<D>;
  uint32_t* ulist = reinterpret_cast<uint32_t*>(sm + L::kEnd);
  const int nwords = p.nwords;
  uint32_t* bitA = ulist + 2 * p.kmax + 2;
  uint32_t* bitB = bitA + nwords;

  // bar_q: the Q tile landed.  bar_dot: the compute warps have written dO
  // into TMEM (all compute threads).  bar_k[s]: K stage s filled;
  // bar_kvfree[s]: dQ of the step using stage s done (K read).  bar_v[s]: V
  // stage s filled; bar_vfree[s]: dP of the step using it done (V read).
  // s_done: S(j) and dP(j) done; s_free: the compute warps have read them
  // (all compute threads); bar_ds: dS(j) written; ds_free: dQ(j), which read
  // it, done.  Every parity wait targets a barrier in the awaited phase or
  // the one after it.
  __shared__ uint64_t bar_q, bar_dot, bar_k[kDqKStages], bar_kvfree[kDqKStages], bar_v[kDqVStages],
      bar_vfree[kDqVStages], s_done, s_free, bar_ds, ds_free;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int n_union, n_cnt[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = blockIdx.x;
  const int64_t bh = blockIdx.y;
  int qa, qb;
  tile_cubes(p.qpairs, bh, pair, p.npairs, p.Nc, p.err, qa, qb);
  const bool has_b = qb >= 0;
  const int64_t row_base = bh * p.N;

  if (tid == 0) {
    mbar_init(&bar_q, 1);
    mbar_init(&bar_dot, kCompute);
    for (int i = 0; i < kDqKStages; ++i) {
      mbar_init(&bar_k[i], 1);
      mbar_init(&bar_kvfree[i], 1);
    }
    for (int i = 0; i < kDqVStages; ++i) {
      mbar_init(&bar_v[i], 1);
      mbar_init(&bar_vfree[i], 1);
    }
    mbar_init(&bar_ds, kCompute);
    mbar_init(&ds_free, 1);
    mbar_init(&s_done, 1);
    mbar_init(&s_free, kCompute);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  for (int w = tid; w < 2 * nwords; w += kThreads) bitA[w] = 0;  // bitA and bitB are contiguous
  __syncthreads();
  {
    const int64_t rowa = bh * p.Nc + qa, rowb = bh * p.Nc + (has_b ? qb : qa);
    int ca = p.cnt ? p.cnt[rowa] : p.kmax;
    int cb = has_b ? (p.cnt ? p.cnt[rowb] : p.kmax) : 0;
    ca = min(max(ca, 0), p.kmax);
    cb = min(max(cb, 0), p.kmax);
    if (tid == 0) {
      n_cnt[0] = ca;
      n_cnt[1] = cb;
    }
    const int32_t* la = p.idx + rowa * p.kmax;
    const int32_t* lb = p.idx + rowb * p.kmax;
    for (int e = tid; e < ca + cb; e += kThreads) {
      const bool isA = e < ca;
      const int c = isA ? la[e] : lb[e - ca];
      if (c < 0 || c >= p.Nc) continue;  // reported by the inverse-list build
      atomicOr(&(isA ? bitA : bitB)[c >> 5], 1u << (c & 31));
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int n = warp_union_list(bitA, bitB, nwords, ulist);
    if (lane == 0) n_union = n;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int U = n_union;
  const int steps = (U + 1) >> 1;
  auto kcube = [&](int j, int g) -> int {
    const int e = (g == 1 && 2 * j + 1 < U) ? 2 * j + 1 : 2 * j;
    return static_cast<int>(ulist[e] & 0x3FFFFFFF);
  };

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0 && steps > 0) {
      mbar_expect_tx(&bar_q, L::kTile);
      load_cube_pair<D>(sm + L::kQ, &p.tq, &bar_q, row_base, qa, has_b ? qb : qa);
      // K(j) goes into stage j % 3 once dQ(j - 3) is done; V(j) into stage
      // j % 2 once dP(j - 2) is.  V(j) is needed first (dP(j) follows S(j)),
      // so it goes out before K(j + 1), and the waits spin: a suspended wait
      // wakes hundreds of cycles late.
      auto load_k = [&](int j) -> bool {
        const int s = j % kDqKStages;
        if (j >= kDqKStages && !mbar_spin(&bar_kvfree[s], ((j / kDqKStages) - 1) & 1)) return false;
        mbar_expect_tx(&bar_k[s], L::kTile);
        load_cube_pair<D>(sm + L::kK + s * L::kTile, &p.tk, &bar_k[s], row_base, kcube(j, 0), kcube(j, 1));
        return true;
      };
      bool ok = load_k(0);
      for (int j = 0; ok && j < steps; ++j) {
        const int vs = j % kDqVStages;
        if (j >= kDqVStages && !mbar_spin(&bar_vfree[vs], ((j / kDqVStages) - 1) & 1)) ok = false;
        if (!ok) break;
        mbar_expect_tx(&bar_v[vs], L::kTile);
        load_cube_pair<D>(sm + L::kV + vs * L::kTile, &p.tv, &bar_v[vs], row_base, kcube(j, 0), kcube(j, 1));
        if (j + 1 < steps) ok = load_k(j + 1);
      }
      if (!ok) flag_error(p.err, kErrTimeout);
    }
  } else if (warp == 1 || warp == 10) {
    // ---------------- MMA issuers.  An MMA issue holds the issuing thread
    // about as long as the tensor core takes to run it, and each barrier poll
    // costs ~100+ cycles while the tensor core streams shared memory, so one
    // thread issuing everything leaves the pipe idle between groups.  Two
    // threads issue instead, each in its own fixed order: warp 1 S(j) then
    // dP(j) (S(j) once the compute warps have read S / dP(j - 1)), warp 10
    // dQ(j) once dS(j) is written.  Their groups touch disjoint TMEM columns;
    // each thread's commits track its own MMAs.
    if (lane == 0 && steps > 0) {
      constexpr uint32_t idesc_s = idesc_f32acc(128, 128, 0, 0, 1);
      constexpr uint32_t idesc_q = idesc_f32acc(128, D, 0, 1, 1);
      constexpr uint32_t kTileU = L::kTile >> 4;
      bool ok = true;
      if (warp == 1) {
        uint64_t qdesc[D / 16];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          qdesc[kk] = sdesc_sw128(smem_u32(sm + L::kQ + (kk >> 2) * 16384 + (kk & 3) * 32), 16, 1024);
        const uint64_t kkm0 = sdesc_sw128(smem_u32(sm + L::kK), 16, 1024);  // K stages, K-major
        const uint64_t vkm0 = sdesc_sw128(smem_u32(sm + L::kV), 16, 1024);  // V stages, K-major
        ok = mbar_spin(&bar_q, 0) && mbar_spin(&bar_dot, 0);
        uint32_t ks = 0, kph = 0, vs = 0, vph = 0;  // ring stages of step j and their fill parities
        for (int j = 0; ok && j < steps; ++j) {
          if ((j > 0 && !mbar_spin(&s_free, (j - 1) & 1)) || !mbar_spin(&bar_k[ks], kph)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd = kkm0 + ks * kTileU;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + kDqS, qdesc[kk], kd + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4), idesc_s, kk > 0);
          // dP(j) = dO V^T (A = dO from TMEM); then S and dP are done together.
          if (!mbar_spin(&bar_v[vs], vph)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t vd = vkm0 + vs * kTileU;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ts(tmem + kDqDP, tmem + kDqDO + kk * 8, vd + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4), idesc_s,
                   kk > 0);
          mma_commit(&s_done);
          mma_commit(&bar_vfree[vs]);
          if (++ks == static_cast<uint32_t>(kDqKStages)) {
            ks = 0;
            kph ^= 1u;
          }
          if (++vs == static_cast<uint32_t>(kDqVStages)) {
            vs = 0;
            vph ^= 1u;
          }
        }
      } else {
        const uint64_t kmn0 = sdesc_sw128(smem_u32(sm + L::kK), 16384, 1024);  // K stages, MN-major
        uint32_t kg = 0;  // K stage of dQ(j)
        for (int j = 0; ok && j < steps; ++j) {
          if (!mbar_spin(&bar_ds, j & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd = kmn0 + kg * kTileU;
          // A = dS (K = 128 keys in 8 steps of 16), B = the K stage (MN-major).
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + kDqDQ, tmem + kDqDS + kk * 8, kd + ((kk * 2048) >> 4), idesc_q, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar_kvfree[kg]);
          mma_commit(&ds_free);
          if (++kg == static_cast<uint32_t>(kDqKStages)) kg = 0;
        }
      }
      if (!ok) flag_error(p.err, kErrTimeout);
    }
  } else {
    // ---------------- compute warps: warpgroup g takes key cube g of each
    // step (TMEM columns 64g..64g+63); thread = query row (TMEM lane).
    const int quarter = warp & 3;
    const int g = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t my_bit = row < 64 ? 30u : 31u;
    const bool row_valid = row < 64 || has_b;
    const int64_t grow = row_base + 64 * static_cast<int64_t>(row < 64 ? qa : (has_b ? qb : qa)) + (row & 63);
    const float lse2 = row_valid ? p.lse[grow] * 1.4426950408889634f : 0.f;
    const float dlt = row_valid ? p.delta[grow] : 0.f;
    const uint64_t sl2 = f2(p.scale_log2, p.scale_log2), nlse2 = f2(-lse2, -lse2), dlt2 = f2(dlt, dlt);
    bool ok = true;
    {
      // dO rows into TMEM (lane = row, column c = elements 2c and 2c + 1):
      // warpgroup g writes elements [g D/2, (g + 1) D/2) of its rows.
      const uint4* src = reinterpret_cast<const uint4*>(p.dof + grow * D + g * (D / 2));
#pragma unroll
      for (int c = 0; c < D / 4; c += 8) {
        uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
        if (row_valid && steps > 0) {
          a = src[c / 4];
          b = src[c / 4 + 1];
        }
        const uint32_t r[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        tmem_st8(lane_addr + kDqDO + g * (D / 4) + c, r);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_dot);
    }
    for (int j = 0; j < steps; ++j) {
      const bool has1 = 2 * j + 1 < U;
      const uint32_t e = (g == 0) ? ulist[2 * j] : (has1 ? ulist[2 * j + 1] : 0u);
      const bool valid = (g == 0 || has1) && ((e >> my_bit) & 1u) != 0;  // warp-uniform
      // Suspended waits here too, for the same reason as in the dK/dV kernel.
      if (!mbar_wait(&s_done, j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S and dP of this warpgroup's key cube into registers, then release them.
      uint32_t sv[64], dv[64];
      if (valid) tmem_ld64x2_wait(lane_addr + kDqS + 64 * g, sv, lane_addr + kDqDP + 64 * g, dv);
      tc_fence_before();
      mbar_arrive(&s_free);
      // P = exp2(S * scale - LSE), dS = P (dP - D), packed fp16.
      uint32_t ds[32];
      if (valid) {
        // P = exp2(S scale log2e - LSE log2e), dS = P (dP - D), packed pairs.
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const uint64_t pr = exp2x2(fma2(f2u(sv[i], sv[i + 1]), sl2, nlse2));
          ds[i >> 1] = f16x2_sat(mul2(pr, sub2(f2u(dv[i], dv[i + 1]), dlt2)));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) ds[i] = 0u;
      }
      // Into the dS buffer once dQ(j - 1) has read it (dQ(j - 1) runs right
      // after dP(j), so this rarely waits).
      if (j >= 1) {
        if (!mbar_wait(&ds_free, (j - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
#pragma unroll
      for (int c = 0; c < 32; c += 8) tmem_st8(lane_addr + kDqDS + 32 * g + c, ds + c);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_ds);
    }
    if (ok && steps > 0 && !mbar_spin(&ds_free, (steps - 1) & 1)) ok = false;
    if (!ok) flag_error(p.err, kErrTimeout);
    tc_fence_after();
    // ---------------- dQ rows (warpgroup g writes columns [g*D/2, (g+1)*D/2))
    const int qc = row < 64 || !has_b ? qa : qb;
    const GradRow dst = grad_row(p, p.fused.dq, p.dq, p.fused.dqc + (bh * p.Nc + qc) * D, bh, qc, row & 63);
#pragma unroll
    for (int c0 = 0; c0 < D / 2; c0 += 32) {
      const int c = g * (D / 2) + c0;
      uint32_t a[32];
      if (steps > 0 && ok) {
        tmem_ld32_wait(lane_addr + kDqDQ + c, a);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] = 0u;
      }
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(a[i]) * p.scale;
      if (row_valid) store_grad32<D>(p, dst, v, c);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

// Inverse lists by counting sort: counts[bh][c] = number of query cubes
// listing key cube c (entries outside [0, Nc) and counts outside [0, kmax]
// latch kErrLut and are skipped).
__global__ void inv_count_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt, int kmax, int Nc,
                                 int64_t rows, int* __restrict__ counts, int* err) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= rows * kmax) return;
  const int64_t row = e / kmax;  // bh * Nc + query cube
  const int slot = static_cast<int>(e % kmax);
  int n = cnt ? cnt[row] : kmax;
  if (n < 0 || n > kmax) {
    if (slot == 0) flag_error(err, kErrLut);
    n = min(max(n, 0), kmax);
  }
  if (slot >= n) return;
  const int c = idx[e];
  if (c < 0 || c >= Nc) {
    flag_error(err, kErrLut);
    return;
  }
  atomicAdd(counts + (row / Nc) * Nc + c, 1);
}

// One CTA per head: off[0 .. Nc] = exclusive prefix sums of the counts, and
// the counts replaced by the same offsets (the fill kernel's cursors).
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads) inv_scan_kernel(int* __restrict__ counts, int Nc,
                                                                int32_t* __restrict__ off) {
  __shared__ int warp_sum[32];
  const int64_t bh = blockIdx.x;
  int* cnt = counts + bh * Nc;
  int32_t* o = off + bh * (Nc + 1);
  const int per = (Nc + kScanThreads - 1) / kScanThreads;
  const int c0 = threadIdx.x * per, c1 = min(Nc, c0 + per);
  int mine = 0;
  for (int c = c0; c < c1; ++c) mine += cnt[c];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = mine;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += t;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = warp_sum[lane];
    int wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += t;
    }
    warp_sum[lane] = wi - w;  // exclusive sum of the warps before
  }
  __syncthreads();
  int run = warp_sum[warp] + incl - mine;
  for (int c = c0; c < c1; ++c) {
    const int v = cnt[c];
    o[c] = run;
    cnt[c] = run;
    run += v;
  }
  if (threadIdx.x == kScanThreads - 1) o[Nc] = run;
}

// ids[bh * stride + slot] = query cube, one slot per (query, key) entry.
__global__ void inv_fill_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt, int kmax, int Nc,
                                int64_t rows, int* __restrict__ cursor, int32_t* __restrict__ ids, int64_t stride) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= rows * kmax) return;
  const int64_t row = e / kmax;
  const int slot = static_cast<int>(e % kmax);
  const int n = min(max(cnt ? cnt[row] : kmax, 0), kmax);
  if (slot >= n) return;
  const int c = idx[e];
  if (c < 0 || c >= Nc) return;
  const int64_t bh = row / Nc;
  const int pos = atomicAdd(cursor + bh * Nc + c, 1);
  ids[bh * stride + pos] = static_cast<int32_t>(row % Nc);
}

// D_i = dO_i . O_i (fp32, dO as the fp16 operand the MMAs use), one warp per row.
__global__ void delta_kernel(const void* __restrict__ of, int of_dtype, const __half* __restrict__ dof,
                             int64_t rows, int d, float* __restrict__ delta) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float s = 0.f;
  for (int c = lane * 8; c < d; c += 256) {
    float a[8], b[8];
    load8(of, row * d + c, of_dtype, a);
    uint4 u = *reinterpret_cast<const uint4*>(dof + row * d + c);
    b[0] = f16_lo(u.x); b[1] = f16_hi(u.x); b[2] = f16_lo(u.y); b[3] = f16_hi(u.y);
    b[4] = f16_lo(u.z); b[5] = f16_hi(u.z); b[6] = f16_lo(u.w); b[7] = f16_hi(u.w);
#pragma unroll
    for (int i = 0; i < 8; ++i) s = fmaf(a[i], b[i], s);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) delta[row] = s;
}

// bf16 -> fp16 copies (exact within the fp16 range; larger values saturate
// and latch kErrRange): tensor blockIdx.y, n8 = its 8-element groups.
struct F16Copies {
  const uint4* src[4];
  uint4* dst[4];
};
__global__ void to_f16_kernel(F16Copies c, int64_t n8, int* err) {
  const uint4* __restrict__ src = c.src[blockIdx.y];
  uint4* __restrict__ dst = c.dst[blockIdx.y];
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    uint4 v = src[i];
    const float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                        bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    bool big = false;
#pragma unroll
    for (int e = 0; e < 8; ++e) big |= !(fabsf(f[e]) <= kF16Max);
    if (big) flag_error(err, kErrRange);
    dst[i] = make_uint4(pack_f16(f[0], f[1]), pack_f16(f[2], f[3]), pack_f16(f[4], f[5]), pack_f16(f[6], f[7]));
  }
}

}  // namespace

size_t inverse_lists_bytes(int BH, int Nc, int kmax) {
  auto a = [](size_t x) { return (x + 255) & ~size_t(255); };
  return a(sizeof(int32_t) * static_cast<size_t>(BH) * (Nc + 1)) + a(sizeof(int) * static_cast<size_t>(BH) * Nc) +
         a(sizeof(int32_t) * static_cast<size_t>(BH) * Nc * kmax);
}

int launch_inverse_lists(const int32_t* idx, const int32_t* cnt, int kmax, int BH, int Nc, void* ws,
                         InverseLists* out, cudaStream_t s) {
  auto a = [](size_t x) { return (x + 255) & ~size_t(255); };
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* off = reinterpret_cast<int32_t*>(w);
  w += a(sizeof(int32_t) * static_cast<size_t>(BH) * (Nc + 1));
  int* counts = reinterpret_cast<int*>(w);
  w += a(sizeof(int) * static_cast<size_t>(BH) * Nc);
  int32_t* ids = reinterpret_cast<int32_t*>(w);
  *out = InverseLists{off, ids, static_cast<int64_t>(Nc) * kmax};
  if (cudaMemsetAsync(counts, 0, sizeof(int) * static_cast<size_t>(BH) * Nc, s) != cudaSuccess) return VSA_ERR_CUDA;
  const int64_t rows = static_cast<int64_t>(BH) * Nc, entries = rows * kmax;
  int* err = device_error_word();
  const unsigned blocks = static_cast<unsigned>((entries + 255) / 256);
  if (entries > 0) inv_count_kernel<<<blocks, 256, 0, s>>>(idx, cnt, kmax, Nc, rows, counts, err);
  inv_scan_kernel<<<BH, kScanThreads, 0, s>>>(counts, Nc, off);
  if (entries > 0) inv_fill_kernel<<<blocks, 256, 0, s>>>(idx, cnt, kmax, Nc, rows, counts, ids, out->stride);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

int launch_to_f16(const void* const* src, void* const* dst, int n, int64_t elems, cudaStream_t s) {
  if (n < 1 || n > 4 || elems % 8) return VSA_ERR_ARG;
  F16Copies c{};
  for (int i = 0; i < n; ++i) {
    c.src[i] = static_cast<const uint4*>(src[i]);
    c.dst[i] = static_cast<uint4*>(dst[i]);
  }
  const int64_t n8 = elems / 8, nblk = (n8 + 255) / 256;
  // Enough CTAs to cover the SMs several times over; each strides the rest.
  const unsigned gx = static_cast<unsigned>(nblk < 4096 ? (nblk > 0 ? nblk : 1) : 4096);
  to_f16_kernel<<<dim3(gx, n), 256, 0, s>>>(c, n8, device_error_word());
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

size_t fine_bwd_ws_bytes(int BH, int N, int kmax) {
  const int64_t Nc = N / kCube;
  size_t inv = inverse_lists_bytes(BH, static_cast<int>(Nc), kmax);
  size_t delta = sizeof(float) * static_cast<size_t>(BH) * N;
  size_t copy = sizeof(__half) * static_cast<size_t>(BH) * N * 128;  // room for d <= 128
  size_t plan = pair_plan_ws_bytes(BH, static_cast<int>(Nc));
  return ((inv + 255) & ~size_t(255)) + ((delta + 255) & ~size_t(255)) + 4 * ((copy + 255) & ~size_t(255)) +
         2 * ((plan + 255) & ~size_t(255));
}

int launch_delta(const void* of, int of_dtype, const void* dof, int64_t rows, int d, float* delta, cudaStream_t s) {
  const int warps = 8;
  delta_kernel<<<static_cast<unsigned>((rows + warps - 1) / warps), warps * 32, 0, s>>>(
      of, of_dtype, static_cast<const __half*>(dof), rows, d, delta);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

// Fine backward with the row statistics D given.  qp, kp, vp, dof are fp16
// (cube order); fused: where the gradient rows go (null: fp32 dq, dk, dv in
// cube order); inv_ws: scratch for the inverse lists (inverse_lists_bytes); qpairs: the
// query-cube tiles of the dQ kernel (null: cubes 2t, 2t + 1); kpairs_ws:
// scratch for the key-cube pair plan (null: cubes 2t, 2t + 1).  The inverse
// lists, the key plan and the dK/dV kernel go on s_kv (the kernel after
// kv_after, when given), the dQ kernel on s (the two kernels are independent;
// s_kv may be s).
int launch_fine_bwd_core(const void* qp, const void* kp, const void* vp, const void* dof, const float* lse,
                         const float* delta, const int32_t* idx, const int32_t* cnt, int kmax, int BH, int N, int d,
                         float scale, float* dq, float* dk, float* dv, const FusedGrads* fused, void* inv_ws,
                         const int32_t* qpairs, int32_t* kpairs_ws, cudaStream_t s, cudaStream_t s_kv,
                         cudaEvent_t kv_after) {
  BwdParams p{};
  const int64_t rows = static_cast<int64_t>(BH) * N;
  int st;
  if ((st = make_tile_map(&p.tq, qp, rows, d, 1)) != VSA_OK) return st;
  if ((st = make_tile_map(&p.tk, kp, rows, d, 1)) != VSA_OK) return st;
  if ((st = make_tile_map(&p.tv, vp, rows, d, 1)) != VSA_OK) return st;
  if ((st = make_tile_map(&p.tdo, dof, rows, d, 1)) != VSA_OK) return st;
  p.dof = static_cast<const uint16_t*>(dof);
  const int Nc = N / kCube, nwords = (Nc + 31) / 32;
  p.lse = lse;
  p.delta = delta;
  p.idx = idx;
  p.cnt = cnt;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  if (fused) {
    p.fused = *fused;
    p.Nn = static_cast<int64_t>(fused->grid.T) * fused->grid.H * fused->grid.W;
  }
  p.N = N;
  p.Nc = Nc;
  p.nwords = nwords;
  p.kmax = kmax;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = device_error_word();
  p.npairs = (Nc + 1) / 2;
  p.qpairs = qpairs;
  p.kpairs = kpairs_ws;
  if ((st = launch_inverse_lists(idx, cnt, kmax, BH, Nc, inv_ws, &p.inv, s_kv)) != VSA_OK) return st;
  if (kpairs_ws) {
    st = launch_pair_plan_inverse(p.inv, BH, Nc, kpairs_ws, s_kv);
    if (st == VSA_ERR_UNSUPPORTED)
      p.kpairs = nullptr;  // too many cubes for the planner's shared memory: cubes 2t, 2t + 1
    else if (st != VSA_OK)
      return st;
  }
  if (kv_after && cudaStreamWaitEvent(s_kv, kv_after, 0) != cudaSuccess) return VSA_ERR_CUDA;
  const size_t kv_extra = sizeof(uint32_t) * (2 * Nc + 2 + 2 * nwords) + 4 * sizeof(float) * d;
  const size_t dq_extra = sizeof(uint32_t) * (2 * kmax + 2 + 2 * nwords);
  dim3 grid((Nc + 1) / 2, BH);
  auto go = [&](auto kernel, size_t bytes, cudaStream_t st_) -> int {
    const size_t smem = bytes + 1024;
    if (smem > 226 * 1024) return VSA_ERR_UNSUPPORTED;  // 1 KB of the 227 KB is left for static shared memory
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return VSA_ERR_CUDA;
    kernel<<<grid, kThreads, smem, st_>>>(p);
    return VSA_OK;
  };
  timing_mark(VSA_K_FINE_BWD, true, s_kv);
  st = d == 128 ? go(fine_bwd_kv_kernel<128>, KvLayout<128>::kEnd + kv_extra, s_kv)
                : go(fine_bwd_kv_kernel<64>, KvLayout<64>::kEnd + kv_extra, s_kv);
  timing_mark(VSA_K_FINE_BWD, false, s_kv);
  if (st != VSA_OK) return st;
  timing_mark(VSA_K_FINE_BWD_DQ, true, s);
  st = d == 128 ? go(fine_bwd_dq_kernel<128>, DqLayout<128>::kEnd + dq_extra, s)
                : go(fine_bwd_dq_kernel<64>, DqLayout<64>::kEnd + dq_extra, s);
  timing_mark(VSA_K_FINE_BWD_DQ, false, s);
  if (st != VSA_OK) return st;
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

// Public fine backward: bf16 inputs are copied to fp16 in the workspace
// first; the query cubes of the dQ kernel and the key cubes of the dK/dV
// kernel are paired by list overlap, as in vsa_backward.
int launch_fine_bwd(const void* qp, const void* kp, const void* vp, const void* of, int of_dtype, const float* lse,
                    const void* dof, const int32_t* idx, const int32_t* cnt, int kmax, int BH, int N, int d,
                    float scale, float* dq, float* dk, float* dv, void* ws, size_t ws_bytes, cudaStream_t s,
                    cudaStream_t s_kv, cudaEvent_t ready) {
  if (!ws || ws_bytes < fine_bwd_ws_bytes(BH, N, kmax)) return VSA_ERR_WORKSPACE;
  const int64_t Nc = N / kCube, rows = static_cast<int64_t>(BH) * N;
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  uint8_t* w = static_cast<uint8_t*>(ws);
  void* inv_ws = w;
  w += inverse_lists_bytes(BH, static_cast<int>(Nc), kmax);
  float* delta = reinterpret_cast<float*>(w);
  w += a256(sizeof(float) * rows);
  const size_t copy = a256(sizeof(__half) * static_cast<size_t>(rows) * 128);
  const void* srcs[4] = {qp, kp, vp, dof};
  void* h[4];
  for (int i = 0; i < 4; ++i, w += copy) h[i] = w;
  const size_t plan = a256(pair_plan_ws_bytes(BH, static_cast<int>(Nc)));
  int32_t* kpairs = reinterpret_cast<int32_t*>(w);
  int32_t* qpairs = reinterpret_cast<int32_t*>(w + plan);
  int st = launch_to_f16(srcs, h, 4, rows * d, s);
  if (st != VSA_OK) return st;
  if ((st = launch_delta(of, of_dtype, h[3], rows, d, delta, s)) != VSA_OK) return st;
  st = launch_pair_plan(idx, cnt, kmax, BH, static_cast<int>(Nc), qpairs, s);
  if (st == VSA_ERR_UNSUPPORTED)
    qpairs = nullptr;  // too many cubes for the planner's shared memory: cubes 2t, 2t + 1
  else if (st != VSA_OK)
    return st;
  if (ready && cudaEventRecord(ready, s) != cudaSuccess) return VSA_ERR_CUDA;
  return launch_fine_bwd_core(h[0], h[1], h[2], h[3], lse, delta, idx, cnt, kmax, BH, N, d, scale, dq, dk, dv, nullptr,
                              inv_ws, qpairs, kpairs, s, s_kv, ready);
}

}  // namespace vsa
