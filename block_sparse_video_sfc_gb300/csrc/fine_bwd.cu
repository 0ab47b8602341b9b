// fine_bwd.cu -- gradient of the fine block-sparse attention on tcgen05.
// "VSA: Faster Video Diffusion with Trainable Sparse Attention" (Abstract: VSA
// trains end to end as one differentiable kernel); the forward is the fine
// stage of "VSA: Accelerating Video Diffusion Inference with Sparse Attention
// on AMD GPUs" ("Stage 2: Fine Computation").  The index list is constant.
//
// Per query row i and listed key j (S = scale * Q K^T, P = softmax(S)):
//   dV_j += P_ij dO_i,  dP_ij = dO_i . V_j,  dS_ij = P_ij (dP_ij - D_i),
//   D_i = dO_i . O_i,  dQ_i += scale dS_ij K_j,  dK_j += scale dS_ij Q_i.
//
// GB300 mapping (key-stationary).  One CTA owns a PAIR of consecutive key
// cubes (128 keys; their K and V stay in shared memory, dK and dV accumulate
// in TMEM) and walks the union of the two cubes' inverse lists -- the query
// cubes whose index list holds either key cube -- two query cubes (128 rows)
// per step.  Quadrants (key cube, query cube) that are not in the list are
// masked.  With keys on the MMA M dimension every product is an M = 128 MMA:
//   S^T  = K Q^T      (SS)          dP^T = V dO^T     (SS)
//   dV  += P^T dO     (A = P^T in TMEM)
//   dK  += dS^T Q     (A = dS^T in TMEM)
//   dQ^T = K^T dS^T   (SS; dS^T also staged in shared memory)
// and dQ^T is added to a global fp32 dQ with warp-coalesced reductions.
// The inverse lists come from a bit matrix inv[bh][key cube][query cube]
// built from the index list (workspace).
#include <cuda.h>

#include "common.cuh"
#include "sm100.cuh"

namespace vsa {

namespace {

constexpr int kThreads = 192;
constexpr uint32_t kColS = 0, kColP = 0, kColDS = 64, kColDP = 128, kColDQ = 128, kColDV = 256, kColDK = 384;

struct BwdParams {
  CUtensorMap tq, tk, tv, tdo;
  const float* lse;    // natural-log LSE per row [BH*N]
  const float* delta;  // D per row [BH*N]
  const uint32_t* inv; // [BH][Nc][nwords]
  float* dq;           // fp32 accumulator [BH*N, d] (zeroed by the launcher)
  float* dk;
  float* dv;
  int N, Nc, nwords;
  float scale, scale_log2;
  int* err;
};

template <int D>
struct BwdLayout {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;
  static constexpr int kDO = kQ + kTile;
  static constexpr int kDS = kDO + kTile;               // [2 query atoms][128 key rows][128 B]
  static constexpr int kZero = kDS + 32768;             // zero atom (D = 64 only)
  static constexpr int kEnd = kZero + (D == 64 ? 16384 : 0);
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) fine_bwd_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using L = BwdLayout<D>;
  float* s_lse = reinterpret_cast<float*>(sm + L::kEnd);  // [2][128]
  float* s_del = s_lse + 256;                              // [2][128]
  uint32_t* ulist = reinterpret_cast<uint32_t*>(s_del + 256);
  uint32_t* bitA = ulist + 2 * p.Nc + 2;
  uint32_t* bitB = bitA + p.nwords;

  // Per-step barriers (each completes once per step): Q(j) / dO(j) loaded;
  // S^T, dP^T done (mma1); P^T, dS^T written (ds, 128 threads); dV done (dO
  // free); dK done (Q free); dQ^T done (mma2); dQ^T read out (dqr, 128).
  __shared__ uint64_t bar_kv, bar_qld, bar_dold, bar_mma1, bar_ds, bar_dofree, bar_qfree, bar_mma2, bar_dqr;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int n_union;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int k1 = 2 * pair, k2 = 2 * pair + 1;
  const bool has_k2 = k2 < p.Nc;
  const int64_t row_base = bh * p.N;

  if (tid == 0) {
    mbar_init(&bar_kv, 1);
    mbar_init(&bar_qld, 1);
    mbar_init(&bar_dold, 1);
    mbar_init(&bar_dofree, 1);
    mbar_init(&bar_qfree, 1);
    mbar_init(&bar_mma1, 1);
    mbar_init(&bar_ds, 128);
    mbar_init(&bar_mma2, 1);
    mbar_init(&bar_dqr, 128);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  {
    const uint32_t* ra = p.inv + (bh * p.Nc + k1) * p.nwords;
    for (int w = tid; w < p.nwords; w += kThreads) {
      bitA[w] = ra[w];
      bitB[w] = has_k2 ? ra[p.nwords + w] : 0u;
    }
    if (D == 64)
      for (int e = tid; e < 16384 / 16; e += kThreads)
        reinterpret_cast<uint4*>(sm + L::kZero)[e] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (warp == 0) {
    int pos = 0;
    for (int w0 = 0; w0 < p.nwords; w0 += 32) {
      int w = w0 + lane;
      uint32_t a = w < p.nwords ? bitA[w] : 0u, b = w < p.nwords ? bitB[w] : 0u;
      uint32_t u = a | b;
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
        ulist[o++] = static_cast<uint32_t>(w * 32 + bit) | (((a >> bit) & 1u) << 30) | (((b >> bit) & 1u) << 31);
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

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0 && steps > 0) {
      const int c1 = has_k2 ? k2 : k1;
      mbar_expect_tx(&bar_kv, 2 * L::kTile);
      for (int b = 0; b < D / 64; ++b) {
        tma_load_2d(sm + L::kK + b * 16384, &p.tk, &bar_kv, 64 * b, static_cast<int>(row_base + 64 * k1));
        tma_load_2d(sm + L::kK + b * 16384 + 8192, &p.tk, &bar_kv, 64 * b, static_cast<int>(row_base + 64 * c1));
        tma_load_2d(sm + L::kV + b * 16384, &p.tv, &bar_kv, 64 * b, static_cast<int>(row_base + 64 * k1));
        tma_load_2d(sm + L::kV + b * 16384 + 8192, &p.tv, &bar_kv, 64 * b, static_cast<int>(row_base + 64 * c1));
      }
      for (int j = 0; j < steps; ++j) {
        const int q0 = ulist[2 * j] & 0x3FFFFFFF;
        const int q1 = (2 * j + 1 < U) ? (ulist[2 * j + 1] & 0x3FFFFFFF) : q0;
        // dO(j) replaces dO(j-1) once dV(j-1) is done; Q(j) once dK(j-1) is.
        if (j > 0 && !mbar_wait(&bar_dofree, (j - 1) & 1)) {
          flag_error(p.err, kErrTimeout);
          break;
        }
        mbar_expect_tx(&bar_dold, L::kTile);
        for (int b = 0; b < D / 64; ++b) {
          tma_load_2d(sm + L::kDO + b * 16384, &p.tdo, &bar_dold, 64 * b, static_cast<int>(row_base + 64 * q0));
          tma_load_2d(sm + L::kDO + b * 16384 + 8192, &p.tdo, &bar_dold, 64 * b, static_cast<int>(row_base + 64 * q1));
        }
        if (j > 0 && !mbar_wait(&bar_qfree, (j - 1) & 1)) {
          flag_error(p.err, kErrTimeout);
          break;
        }
        mbar_expect_tx(&bar_qld, L::kTile);
        for (int b = 0; b < D / 64; ++b) {
          tma_load_2d(sm + L::kQ + b * 16384, &p.tq, &bar_qld, 64 * b, static_cast<int>(row_base + 64 * q0));
          tma_load_2d(sm + L::kQ + b * 16384 + 8192, &p.tq, &bar_qld, 64 * b, static_cast<int>(row_base + 64 * q1));
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0 && steps > 0) {
      constexpr uint32_t id_ss = idesc_f32acc(128, 128, 0, 0, 1);
      constexpr uint32_t id_ts = idesc_f32acc(128, D, 0, 1, 1);
      constexpr uint32_t id_dq = idesc_f32acc(128, 128, 1, 1, 1);
      constexpr uint32_t lbo_kt = D == 128 ? 16384u : static_cast<uint32_t>(L::kZero - L::kK);
      bool ok = mbar_wait(&bar_kv, 0);
      for (int j = 0; j < steps && ok; ++j) {
        if (j > 0) ok = ok && mbar_wait(&bar_qfree, (j - 1) & 1);  // P/dS of step j-1 consumed
        ok = ok && mbar_wait(&bar_qld, j & 1);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int b = kk >> 2, w = kk & 3;
          mma_ss(tmem + kColS, sdesc_sw128(smem_u32(sm + L::kK + b * 16384 + w * 32), 16, 1024),
                      sdesc_sw128(smem_u32(sm + L::kQ + b * 16384 + w * 32), 16, 1024), id_ss, kk > 0);
        }
        if (j > 0) ok = ok && mbar_wait(&bar_dqr, (j - 1) & 1);  // dQ^T of step j-1 read out
        ok = ok && mbar_wait(&bar_dold, j & 1);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int b = kk >> 2, w = kk & 3;
          mma_ss(tmem + kColDP, sdesc_sw128(smem_u32(sm + L::kV + b * 16384 + w * 32), 16, 1024),
                      sdesc_sw128(smem_u32(sm + L::kDO + b * 16384 + w * 32), 16, 1024), id_ss, kk > 0);
        }
        mma_commit(&bar_mma1);
        ok = ok && mbar_wait(&bar_ds, j & 1);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + kColDV, tmem + kColP + kk * 8, sdesc_sw128(smem_u32(sm + L::kDO + kk * 2048), 16384, 1024),
                 id_ts, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar_dofree);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + kColDK, tmem + kColDS + kk * 8, sdesc_sw128(smem_u32(sm + L::kQ + kk * 2048), 16384, 1024),
                 id_ts, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar_qfree);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + kColDQ, sdesc_sw128(smem_u32(sm + L::kK + kk * 2048), lbo_kt, 1024),
                      sdesc_sw128(smem_u32(sm + L::kDS + kk * 2048), 16384, 1024), id_dq, kk > 0);
        mma_commit(&bar_mma2);
      }
      if (!ok) flag_error(p.err, kErrTimeout);
    }
  } else {
    // ---------------- compute warps: thread = TMEM lane (key row, then d row)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int ct = tid - 64;  // 0..127, index for cooperative loads
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t key_bit = r < 64 ? 30u : 31u;
    bool ok = true;
    for (int j = 0; j < steps; ++j) {
      const uint32_t e0 = ulist[2 * j];
      const bool has1 = 2 * j + 1 < U;
      const uint32_t e1 = has1 ? ulist[2 * j + 1] : 0u;
      {
        const int g = ct >> 6;
        const int qc = static_cast<int>((g ? (has1 ? e1 : e0) : e0) & 0x3FFFFFFF);
        const int64_t qrow = row_base + 64 * qc + (ct & 63);
        s_lse[(j & 1) * 128 + ct] = p.lse[qrow] * 1.4426950408889634f;
        s_del[(j & 1) * 128 + ct] = p.delta[qrow];
      }
      named_bar_sync(1, 128);
      if (!mbar_wait(&bar_mma1, j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool v0 = (e0 >> key_bit) & 1u, v1 = has1 && ((e1 >> key_bit) & 1u);
      const float* lse2 = s_lse + (j & 1) * 128;
      const float* del = s_del + (j & 1) * 128;
      uint32_t dsp[64];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const bool valid = h ? v1 : v0;
        float sv[64], dv[64];
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          tmem_ld16(lane_addr + kColS + 64 * h + c, sv + c);
          tmem_ld16(lane_addr + kColDP + 64 * h + c, dv + c);
        }
        tmem_wait_ld();
        float pp[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const int q = 64 * h + c;
          float pa = valid ? fast_exp2(sv[c] * p.scale_log2 - lse2[q]) : 0.f;
          float pb = valid ? fast_exp2(sv[c + 1] * p.scale_log2 - lse2[q + 1]) : 0.f;
          float da = pa * (dv[c] - del[q]);
          float db = pb * (dv[c + 1] - del[q + 1]);
          pp[c >> 1] = __uint_as_float(pack_f16(pa, pb));
          dsp[32 * h + (c >> 1)] = pack_f16(da, db);
        }
#pragma unroll
        for (int c = 0; c < 32; c += 16) tmem_st16(lane_addr + kColP + 32 * h + c, pp + c);
        // dS^T row r, queries 64h..64h+63 -> shared tile (query atom h, key row r)
        uint8_t* dst = sm + L::kDS + h * 16384;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint4 v = make_uint4(dsp[32 * h + 4 * ch], dsp[32 * h + 4 * ch + 1], dsp[32 * h + 4 * ch + 2],
                               dsp[32 * h + 4 * ch + 3]);
          *reinterpret_cast<uint4*>(dst + sw128_offset(r, ch * 8)) = v;
        }
      }
      float* dsf = reinterpret_cast<float*>(dsp);
#pragma unroll
      for (int c = 0; c < 64; c += 16) tmem_st16(lane_addr + kColDS + c, dsf + c);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_ds);
      // dQ^T: lane = d row, columns = the step's 128 query rows.
      if (!mbar_wait(&bar_mma2, j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int64_t qbase0 = row_base + 64 * static_cast<int64_t>(e0 & 0x3FFFFFFF);
      const int64_t qbase1 = row_base + 64 * static_cast<int64_t>(e1 & 0x3FFFFFFF);
      // Read the whole dQ^T row out of TMEM first so the next step's dP^T
      // may overwrite it while the reductions drain.
      float qv[128];
#pragma unroll
      for (int c = 0; c < 128; c += 16) tmem_ld16(lane_addr + kColDQ + c, qv + c);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar_dqr);
      if (r < D) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < 64 || has1) atomicAdd(p.dq + ((c < 64 ? qbase0 : qbase1) + (c & 63)) * D + r, qv[c] * p.scale);
      }
    }
    if (!ok) flag_error(p.err, kErrTimeout);
    // ---------------- dK, dV rows of this key pair
    const int kc = r < 64 ? k1 : k2;
    const bool key_valid = r < 64 || has_k2;
    const int64_t krow = row_base + 64 * static_cast<int64_t>(kc) + (r & 63);
#pragma unroll
    for (int c = 0; c < D; c += 16) {
      float a[16], b[16];
      if (steps > 0 && ok) {
        tmem_ld16(lane_addr + kColDV + c, a);
        tmem_ld16(lane_addr + kColDK + c, b);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) a[i] = b[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) b[i] *= p.scale;
      if (key_valid) {
        store8(p.dv, krow * D + c, a, VSA_DTYPE_F32);
        store8(p.dv, krow * D + c + 8, a + 8, VSA_DTYPE_F32);
        store8(p.dk, krow * D + c, b, VSA_DTYPE_F32);
        store8(p.dk, krow * D + c + 8, b + 8, VSA_DTYPE_F32);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

// inv[bh][key cube][query cube / 32] |= bit for every listed (query, key).
__global__ void build_inverse_bits(const int32_t* __restrict__ idx, const int32_t* __restrict__ cnt, int kmax,
                                   int Nc, int nwords, int64_t rows, uint32_t* __restrict__ inv, int* err) {
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
  const int64_t bh = row / Nc;
  const int q = static_cast<int>(row % Nc);
  atomicOr(inv + (bh * Nc + c) * nwords + (q >> 5), 1u << (q & 31));
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

// bf16 -> fp16 copy (exact within the fp16 range; larger values saturate and
// latch kErrRange).  n8 = number of 8-element groups.
__global__ void to_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n8, int* err) {
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

size_t fine_bwd_ws_bytes(int BH, int N, int kmax) {
  (void)kmax;
  const int64_t Nc = N / kCube, nwords = (Nc + 31) / 32;
  size_t inv = sizeof(uint32_t) * static_cast<size_t>(BH) * Nc * nwords;
  size_t delta = sizeof(float) * static_cast<size_t>(BH) * N;
  size_t copy = sizeof(__half) * static_cast<size_t>(BH) * N * 128;  // room for d <= 128
  return ((inv + 255) & ~size_t(255)) + ((delta + 255) & ~size_t(255)) + 4 * ((copy + 255) & ~size_t(255));
}

int launch_delta(const void* of, int of_dtype, const void* dof, int64_t rows, int d, float* delta, cudaStream_t s) {
  const int warps = 8;
  delta_kernel<<<static_cast<unsigned>((rows + warps - 1) / warps), warps * 32, 0, s>>>(
      of, of_dtype, static_cast<const __half*>(dof), rows, d, delta);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

// Fine backward with the row statistics D given.  qp, kp, vp, dof are fp16
// (cube order); inv_ws: scratch for the inverse-list bit matrix.
int launch_fine_bwd_core(const void* qp, const void* kp, const void* vp, const void* dof, const float* lse,
                         const float* delta, const int32_t* idx, const int32_t* cnt, int kmax, int BH, int N, int d,
                         float scale, float* dq, float* dk, float* dv, uint32_t* inv_ws, cudaStream_t s) {
  BwdParams p{};
  const int64_t rows = static_cast<int64_t>(BH) * N;
  int st;
  if ((st = make_tile_map(&p.tq, qp, rows, d, 1)) != VSA_OK) return st;
  if ((st = make_tile_map(&p.tk, kp, rows, d, 1)) != VSA_OK) return st;
  if ((st = make_tile_map(&p.tv, vp, rows, d, 1)) != VSA_OK) return st;
  if ((st = make_tile_map(&p.tdo, dof, rows, d, 1)) != VSA_OK) return st;
  const int Nc = N / kCube, nwords = (Nc + 31) / 32;
  p.lse = lse;
  p.delta = delta;
  p.inv = inv_ws;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.N = N;
  p.Nc = Nc;
  p.nwords = nwords;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = device_error_word();
  const size_t inv_bytes = sizeof(uint32_t) * static_cast<size_t>(BH) * Nc * nwords;
  if (cudaMemsetAsync(inv_ws, 0, inv_bytes, s) != cudaSuccess) return VSA_ERR_CUDA;
  if (cudaMemsetAsync(dq, 0, sizeof(float) * rows * d, s) != cudaSuccess) return VSA_ERR_CUDA;
  const int64_t entries = static_cast<int64_t>(BH) * Nc * kmax;
  if (entries > 0)
    build_inverse_bits<<<static_cast<unsigned>((entries + 255) / 256), 256, 0, s>>>(
        idx, cnt, kmax, Nc, nwords, static_cast<int64_t>(BH) * Nc, inv_ws, p.err);
  const size_t extra = sizeof(float) * 512 + sizeof(uint32_t) * (2 * Nc + 2 + 2 * nwords);
  dim3 grid((Nc + 1) / 2, BH);
  if (d == 128) {
    size_t smem = BwdLayout<128>::kEnd + 1024 + extra;
    if (smem > 227 * 1024) return VSA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(fine_bwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return VSA_ERR_CUDA;
    timing_mark(VSA_K_FINE_BWD, true, s);
    fine_bwd_kernel<128><<<grid, kThreads, smem, s>>>(p);
    timing_mark(VSA_K_FINE_BWD, false, s);
  } else {
    size_t smem = BwdLayout<64>::kEnd + 1024 + extra;
    if (smem > 227 * 1024) return VSA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(fine_bwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return VSA_ERR_CUDA;
    timing_mark(VSA_K_FINE_BWD, true, s);
    fine_bwd_kernel<64><<<grid, kThreads, smem, s>>>(p);
    timing_mark(VSA_K_FINE_BWD, false, s);
  }
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

// Public fine backward: bf16 inputs are copied to fp16 in the workspace first.
int launch_fine_bwd(const void* qp, const void* kp, const void* vp, const void* of, int of_dtype, const float* lse,
                    const void* dof, const int32_t* idx, const int32_t* cnt, int kmax, int BH, int N, int d,
                    float scale, float* dq, float* dk, float* dv, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!ws || ws_bytes < fine_bwd_ws_bytes(BH, N, kmax)) return VSA_ERR_WORKSPACE;
  const int64_t Nc = N / kCube, nwords = (Nc + 31) / 32, rows = static_cast<int64_t>(BH) * N;
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint32_t* inv_ws = reinterpret_cast<uint32_t*>(w);
  w += a256(sizeof(uint32_t) * static_cast<size_t>(BH) * Nc * nwords);
  float* delta = reinterpret_cast<float*>(w);
  w += a256(sizeof(float) * rows);
  const size_t copy = a256(sizeof(__half) * static_cast<size_t>(rows) * 128);
  const void* srcs[4] = {qp, kp, vp, dof};
  void* h[4];
  int* err = device_error_word();
  for (int i = 0; i < 4; ++i, w += copy) {
    h[i] = w;
    const int64_t n8 = rows * d / 8;
    const int64_t nblk = (n8 + 255) / 256;
    to_f16_kernel<<<static_cast<unsigned>(nblk < 65535 ? nblk : 65535), 256, 0, s>>>(
        static_cast<const uint4*>(srcs[i]), static_cast<uint4*>(h[i]), n8, err);
  }
  int st = launch_delta(of, of_dtype, h[3], rows, d, delta, s);
  if (st != VSA_OK) return st;
  return launch_fine_bwd_core(h[0], h[1], h[2], h[3], lse, delta, idx, cnt, kmax, BH, N, d, scale, dq, dk, dv, inv_ws,
                              s);
}

}  // namespace vsa
