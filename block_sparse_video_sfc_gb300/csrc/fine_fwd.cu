// fine_fwd.cu -- fine block-sparse attention, forward, on tcgen05 tensor cores.
// "VSA: Accelerating Video Diffusion Inference with Sparse Attention on AMD
// GPUs", "Stage 2: Fine Computation" (token-level attention over the selected
// cubes only), "Kernel Architecture" (QK GEMM with running max M and sum L,
// softmax, PV GEMM accumulated across tiles) and "Sparse Traversal" (walk the
// index list instead of every key block).
//
// GB300 mapping.  The tensor core's full rate needs M = 128 rows and N >= 128
// columns per MMA, while the index list is per 64-token query cube.  One CTA
// therefore owns a PAIR of query cubes (128 query rows; the pairs come from
// the overlap plan of pair_plan.cu, or are cubes 2t, 2t + 1) and walks the
// UNION of their two lists, two key cubes (128 keys) per step; each half of
// the tile masks the cubes its own list does not hold.  Per step j:
//   S(j) = Q K(j)^T     tcgen05.mma, A = Q (TMEM), B = K (smem), D = TMEM
//   P(j) = exp2(S - m)  softmax warps, one thread per row, P -> TMEM (fp16)
//   O   += P(j) V(j)    tcgen05.mma, A = P (TMEM), B = V (smem, fp16)
// Padding slots of partial cubes (a grid side not a multiple of 4) are masked
// out of the keys through a per-cube slot mask.
// One CTA per SM.  K and V stream through rings of up to three 32 KB shared-
// memory stages each.  Q sits in TMEM and is the A operand of S = Q K^T, so
// the tensor core reads only K and V from shared memory: every byte of it
// also has to be written there by the TMA, and the two share the shared-
// memory bandwidth (a step moves 128 KB through it, ~1000 cycles at
// 128 B/clk, about the step's 1024 cycles of tensor work).  TMEM columns:
// two S buffers (2 x 128), O (D) and Q (D / 2).  S(j) goes into buffer j % 2
// and P(j) (fp16 pairs, 64 columns) is written over the first half of S(j)
// once both softmax warps of a lane quarter hold their half of S(j) in
// registers; S(j + 2) may take the buffer once PV(j) has read P(j).  So
// S(j + 1) runs while the softmax warps work on step j, and waits for
// neither their loads nor a separate P buffer.
// The running max is only raised (and O rescaled) when a row's max grows by
// more than 2^8, so P <= 256.
// A warp's 32 rows all belong to one query cube, so a key cube outside that
// cube's list is skipped by the whole warp (no loads, no exponentials).
// Roles: warp 0 loads K and warp 10 loads V (TMA), warp 1 issues the MMAs
// (S only, with warp 11 issuing PV, in the kernels that read reordered
// tiles), warps 2-9 compute the softmax and the epilogue (two warps per TMEM
// lane quarter, one per key cube of the step).
#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100.cuh"

namespace vsa {
namespace {

constexpr int kSoftmaxThreads = 256;  // 8 softmax warps (2-9)
// + warp 0 (K loads), warp 1 (MMA issue), warp 10 (V loads), and for the
// kernels that read reordered tiles warp 11 (PV issue, see the issuers).
template <bool NATIVE>
__host__ __device__ constexpr int fwd_threads() {
  return (NATIVE ? 96 : 128) + kSoftmaxThreads;
}
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kTmemCols = 512;        // the whole SM: one CTA per SM
constexpr uint32_t kColS = 0;              // S(j) in 128 (j % 2): 128 fp32 columns; P(j) over its first 64
constexpr uint32_t kColO = 256;            // O: D columns
constexpr uint32_t kColQ = 384;            // Q as the A operand: D / 2 columns of fp16 pairs
constexpr int kMaxStages = 3;              // K and V ring depth

struct FwdParams {
  CUtensorMap tk, tv;  // [BH*N, d] fp16 / bf16, box {64, 64}, 128B swizzle
  const uint16_t* q;   // [BH*N, d] fp16 / bf16, row-major
  const int32_t* idx;
  const int32_t* cnt;
  const int32_t* pairs;  // [BH][npairs][2] tile -> query cubes (second -1: none), or null
  const uint64_t* kmask;  // [Nc]: bit o set when slot o of the cube holds a token; null: every slot does
  // Native layout (the NATIVE kernels): Q, K, V are the [BH, T, H, W, d]
  // tensors; tk / tv are 5-D maps whose {64, 4, 4, 4, 1} box is one (4, 4, 4)
  // cube (zeros outside the grid), and Q rows are addressed through the grid.
  CubeGrid cgrid;
  const int32_t* order;  // cube position -> raster cube (null: raster order)
  int64_t Nn;            // T * H * W
  int kmax, N, Nc, npairs;
  int nk, nv;        // K and V ring depths (1..kMaxStages)
  float scale_log2;  // scale * log2(e)
  void* of;
  int of_dtype;
  float* lse;
  int* err;
};

template <int D>
struct FwdLayout {
  static constexpr int kTile = 128 * D * 2;  // 128 rows x D 16-bit
  static constexpr int kRing = 0;  // nk K stages, then nv V stages
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of 64 values as a shallow tree of three-input maxima.
__device__ __forceinline__ float max64(const uint32_t* v) {
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float* x = reinterpret_cast<const float*>(v + 8 * k);
    float t = fmax3(x[0], x[1], x[2]);
    t = fmax3(t, x[3], x[4]);
    t = fmax3(t, x[5], x[6]);
    a[k] = fmaxf(t, x[7]);
  }
  return fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

// 64 weights P = exp2(S * sl2 - m) of one key cube: packed fp16 (F16) or
// bf16 pairs into pk[32], and their rounded values (what the PV product
// multiplies with) added to the two row-sum partials.  S * sl2 - m runs as a
// packed fp32 pair.
template <bool F16>
__device__ __forceinline__ void softmax64(const uint32_t* sv, uint64_t sl2x2, uint64_t negmx2, uint32_t* pk, float& acc0,
                                          float& acc1) {
#pragma unroll
  for (int c = 0; c < 64; c += 2) {
    uint64_t x, t;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(sv[c]), "r"(sv[c + 1]));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(t) : "l"(x), "l"(sl2x2), "l"(negmx2));
    float t0, t1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(t0), "=f"(t1) : "l"(t));
    const float a = fast_exp2(t0), b = fast_exp2(t1);
    uint32_t h;
    if (F16) {
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(b), "f"(a));  // a -> low half
      asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
          "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
          : "+f"(acc0), "+f"(acc1)
          : "r"(h));
    } else {
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(b), "f"(a));
      acc0 += __uint_as_float(h << 16);  // a bf16 is the top half of its fp32
      acc1 += __uint_as_float(h & 0xFFFF0000u);
    }
    pk[c >> 1] = h;
  }
}

__device__ __forceinline__ uint64_t splat2(float v) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
  return r;
}

// F16IN: Q, K, V arrive as fp16; otherwise as bf16, and the softmax warps
// convert each V tile to fp16 in shared memory (exact within +-65504) so that
// P V always runs on fp16 operands (P rounded to 2^-12, not bf16's 2^-9: with
// bf16 weights the output is too coarse for the D = dO . O_f of a following
// backward).  Accumulation is fp32 either way.
// NATIVE (bf16 only): Q, K, V in their native layout, K / V through 5-D boxes,
// and P V in bf16 (P rounded to 2^-9): no V conversion on the softmax warps'
// critical path.  The inference forward has no backward to feed, and its
// output stays well within the forward tolerance.
template <int D, bool F16IN, bool NATIVE>
__global__ void __launch_bounds__(fwd_threads<NATIVE>(), 1) fine_fwd_kernel(const __grid_constant__ FwdParams p) {
  constexpr int kThreads = fwd_threads<NATIVE>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using L = FwdLayout<D>;
  const int nk = p.nk, nv = p.nv;
  uint8_t* kring = sm + L::kRing;
  uint8_t* vring = kring + nk * L::kTile;
  uint32_t* ulist = reinterpret_cast<uint32_t*>(vring + nv * L::kTile);  // id | inA<<30 | inB<<31
  const int nwords = (p.Nc + 31) >> 5;
  uint32_t* bitA = ulist + 2 * p.kmax + 2;
  uint32_t* bitB = bitA + nwords;

  // kfull/vfull: a stage's TMA landed.  kfree/vfree: the MMA that read the
  // stage completed.  With b = j % 2: bar_s[b]: S(j) done.  bar_p[b]: P(j)
  // written over S(j) (all softmax threads).  pv_done[b]: PV(j) completed (O
  // includes it, and buffer b may take S(j + 2)).  A parity wait is only
  // correct while the barrier is in the awaited phase or the one after it;
  // each wait below keeps to that (S(j) is issued only after PV(j - 2) has
  // completed, so a warp that sees S(j) knows PV(0..j-2) are done).
  __shared__ uint64_t bar_qt, kfull[kMaxStages], kfree[kMaxStages], vfull[kMaxStages], vfree[kMaxStages];
  __shared__ uint64_t bar_s[2], bar_p[2], pv_done[2];
  __shared__ uint64_t pair_bar[4];  // per lane quarter: its two softmax warps (64 threads)
  __shared__ uint32_t tmem_base_sh;
  __shared__ int n_union, n_first, n_cnt[2];
  __shared__ float xmax[2][2][128];  // row max / sum exchange between the two warps of a pair

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = blockIdx.x;
  const int64_t bh = blockIdx.y;
  // The tile's two query cubes: the pair plan's, else cubes 2t and 2t + 1.
  int qa = 2 * pair, qb = 2 * pair + 1 < p.Nc ? 2 * pair + 1 : -1;
  if (p.pairs) {
    qa = p.pairs[(bh * p.npairs + pair) * 2];
    qb = p.pairs[(bh * p.npairs + pair) * 2 + 1];
    if (qa < 0 || qa >= p.Nc || qb < -1 || qb >= p.Nc) {  // not a plan this library wrote
      if (threadIdx.x == 0) flag_error(p.err, kErrLut);
      qa = min(max(qa, 0), p.Nc - 1);
      qb = -1;
    }
  }
  const bool has_b = qb >= 0;

  // ---------------- prologue: barriers, TMEM, union of the two index lists
  if (tid == 0) {
    mbar_init(&bar_qt, kSoftmaxThreads);
    for (int i = 0; i < 4; ++i) mbar_init(&pair_bar[i], 64);
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kfree[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&vfree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s[i], 1);
      mbar_init(&bar_p[i], kSoftmaxThreads);
      mbar_init(&pv_done[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  for (int w = tid; w < 2 * nwords; w += kThreads) bitA[w] = 0;  // bitA and bitB are contiguous
  __syncthreads();
  {
    const int64_t rowa = bh * p.Nc + qa, rowb = bh * p.Nc + (has_b ? qb : qa);
    int ca = p.cnt ? p.cnt[rowa] : p.kmax;
    int cb = has_b ? (p.cnt ? p.cnt[rowb] : p.kmax) : 0;
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
    const int32_t* lb = p.idx + rowb * p.kmax;
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
    // rest of the union by increasing cube id (walked from a rotated start).
    const int ca = n_cnt[0], cb = n_cnt[1];
    const int32_t* la = p.idx + (bh * p.Nc + qa) * p.kmax;
    const int32_t* lb = p.idx + (bh * p.Nc + (has_b ? qb : qa)) * p.kmax;
    int first[2] = {-1, -1};
    int nf = 0;
    if (ca > 0) {
      int c = la[0];
      if (c >= 0 && c < p.Nc) first[nf++] = c;
    }
    if (cb > 0) {
      int c = lb[0];
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
    if (lane == 0) {
      n_union = pos;
      n_first = nf;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int U = n_union;
  // The part of the union after the first entries is walked from a rotated
  // start, so that the CTAs running at the same time read different key
  // cubes instead of all sweeping the head's cubes in the same order.
  const int nf = n_first, ntail = U - nf;
  const int rot = ntail > 0 ? static_cast<int>((static_cast<uint32_t>(pair) * 2654435761u >> 7) % ntail) : 0;
  auto uent = [&](int e) -> uint32_t {
    if (e < nf) return ulist[e];
    int t = e - nf + rot;
    if (t >= ntail) t -= ntail;
    return ulist[nf + t];
  };
  const int steps = (U + 1) >> 1;
  const int64_t row_base = bh * p.N;  // first row of this head in the 2D tensor maps

  if (warp == 0 || warp == 10) {
    // ---------------- TMA producers: warp 0 loads K(j) into stage j % nk once
    // S(j - nk) has completed, warp 10 V(j) into stage j % nv once PV(j - nv)
    // has.  One thread loading both spent ~650 cycles per tile on its waits,
    // bookkeeping and four TMA instructions, ~1300 per step, and so ran
    // barely a step ahead of the MMAs; split, each runs its ring ahead.
    // The waits suspend: the producers are ahead, and a polling thread
    // would take issue slots from the softmax warps on its sub-partition.
    if (lane == 0 && steps > 0) {
      tma_prefetch_desc(&p.tk);
      tma_prefetch_desc(&p.tv);
      auto load = [&](int j, const CUtensorMap* map, uint8_t* ring, int depth, uint64_t* full,
                      uint64_t* free_) -> bool {
        const int st = j % depth, use = j / depth;
        if (use > 0 && !mbar_wait(&free_[st], (use - 1) & 1)) return false;
        const int c0 = uent(2 * j) & 0x3FFFFFFF;
        const int c1 = (2 * j + 1 < U) ? (uent(2 * j + 1) & 0x3FFFFFFF) : c0;
        uint8_t* dst = ring + st * L::kTile;
        mbar_expect_tx(&full[st], L::kTile);
        if (NATIVE) {
          // One 5-D box per cube and 64 channels: rows come out in (t%4, h%4,
          // w%4) order, which is the cube order inside a cube.
          const int r0 = raster_cube(p.order, c0), r1 = raster_cube(p.order, c1);
          const int Wc = p.cgrid.Wc, HWc = p.cgrid.Hc * p.cgrid.Wc;
          for (int b = 0; b < D / 64; ++b) {
            tma_load_5d(dst + b * 16384, map, &full[st], 64 * b, 4 * (r0 % Wc), 4 * ((r0 / Wc) % p.cgrid.Hc),
                        4 * (r0 / HWc), static_cast<int>(bh));
            tma_load_5d(dst + b * 16384 + 8192, map, &full[st], 64 * b, 4 * (r1 % Wc), 4 * ((r1 / Wc) % p.cgrid.Hc),
                        4 * (r1 / HWc), static_cast<int>(bh));
          }
        } else {
          for (int b = 0; b < D / 64; ++b) {
            tma_load_2d(dst + b * 16384, map, &full[st], 64 * b, static_cast<int>(row_base + 64 * c0));
            tma_load_2d(dst + b * 16384 + 8192, map, &full[st], 64 * b, static_cast<int>(row_base + 64 * c1));
          }
        }
        return true;
      };
      bool ok = true;
      for (int j = 0; ok && j < steps; ++j)
        ok = warp == 0 ? load(j, &p.tk, kring, nk, kfull, kfree) : load(j, &p.tv, vring, nv, vfull, vfree);
      if (!ok) flag_error(p.err, kErrTimeout);
    }
  } else if (NATIVE && warp == 1) {
    // ---------------- MMA issuer: S(j+1) runs while the softmax warps work on
    // S(j); PV(j) follows once P(j) is written.
    // S = Q K^T takes Q from TMEM, so that the tensor core reads only K (not
    // Q as well) from shared memory while the TMA writes the next tiles.
    if (lane == 0 && steps > 0) {
      constexpr uint32_t idesc_s = idesc_f32acc(128, 128, 0, 0, F16IN);
      constexpr uint32_t idesc_pv = idesc_f32acc(128, D, 0, 1, NATIVE ? 0 : 1);
      bool ok = mbar_wait(&bar_qt, 0);
      // The issuer shares its SM sub-partition with two busy softmax warps, so
      // it is kept lean: ring slots and parities are stepped, not divided,
      // and the operand descriptors are advanced from per-ring bases (the
      // start-address field is linear in the byte address).
      const uint64_t kdesc0 = sdesc_sw128(smem_u32(kring), 16, 1024);
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(vring), 16384, 1024);
      constexpr uint32_t kTileUnits = L::kTile >> 4;
      int ns = 0, npv = 0;                 // next S and next PV to issue
      uint32_t ks = 0, kph = 0;            // K stage of S(ns) and its fill parity
      uint32_t vs = 0, vph = 0;            // V stage of PV(npv) and its fill parity
      uint32_t idle = 0;
      // A suspended wait (try_wait) wakes up hundreds of cycles after the
      // phase completes, so the issuer polls with test_wait and issues
      // whichever of S(ns) and PV(npv) is ready first.
      while (ok && npv < steps) {
        bool progressed = false;
        // S(ns) once PV(ns - 2) has read P(ns - 2) out of its buffer.
        if (ns < steps && (ns < 2 || mbar_test(&pv_done[ns & 1], ((ns >> 1) - 1) & 1)) &&
            mbar_test(&kfull[ks], kph)) {
          tc_fence_after();
          const uint64_t kd = kdesc0 + ks * kTileUnits;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t bd = kd + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem + kColS + 128 * (ns & 1)),
                "r"(tmem + kColQ + kk * 8), "l"(bd), "r"(idesc_s), "r"(static_cast<uint32_t>(kk > 0)));
          }
          mma_commit(&bar_s[ns & 1]);
          mma_commit(&kfree[ks]);
          ++ns;
          if (++ks == static_cast<uint32_t>(nk)) {
            ks = 0;
            kph ^= 1u;
          }
          progressed = true;
        }
        if (npv < ns && mbar_test(&bar_p[npv & 1], (npv >> 1) & 1) && mbar_test(&vfull[vs], vph)) {
          tc_fence_after();
          const uint32_t pcol = tmem + kColS + 128 * (npv & 1);
          const uint64_t vd = vdesc0 + vs * kTileUnits;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem + kColO),
                "r"(pcol + kk * 8), "l"(vd + ((kk * 2048) >> 4)), "r"(idesc_pv),
                "r"(static_cast<uint32_t>(npv > 0 || kk > 0)));
          }
          mma_commit(&vfree[vs]);
          mma_commit(&pv_done[npv & 1]);
          ++npv;
          if (++vs == static_cast<uint32_t>(nv)) {
            vs = 0;
            vph ^= 1u;
          }
          progressed = true;
        }
        idle = progressed ? 0u : idle + 1u;
        if (idle > (1u << 26)) ok = false;
      }
      if (!ok) flag_error(p.err, kErrTimeout);
    }
  } else if (!NATIVE && (warp == 1 || warp == 11)) {
    // ---------------- MMA issuers, one per kind of group: warp 1 issues S(j)
    // once PV(j - 2) is done (its buffer is free) and K(j) has landed; warp 11
    // issues PV(j) once P(j) is written and V(j) has landed.  Issuing a group
    // holds its thread for about the group's run time, so with one thread the
    // next group waited behind it and behind the barrier tests that follow.
    // Measured on the reordered kernels: 2.496 -> 2.374 ms at 32K tokens,
    // K = 154.  (On the native-layout kernel, whose 5-D TMA boxes arrive
    // later, two threads measured slower: 2.57 -> 2.94 ms; it keeps the
    // single polling issuer above.)  Each thread's commits track its own
    // MMAs: S(j) waits for PV(j - 2) through pv_done, so a softmax warp that
    // sees S(j) still knows that PV(j - 2) is done.
    if (lane == 0 && steps > 0) {
      constexpr uint32_t idesc_s = idesc_f32acc(128, 128, 0, 0, F16IN);
      constexpr uint32_t idesc_pv = idesc_f32acc(128, D, 0, 1, NATIVE ? 0 : 1);
      constexpr uint32_t kTileUnits = L::kTile >> 4;
      bool ok = true;
      if (warp == 1) {
        ok = mbar_wait(&bar_qt, 0);
        const uint64_t kdesc0 = sdesc_sw128(smem_u32(kring), 16, 1024);
        uint32_t ks = 0, kph = 0;  // K stage of S(j) and its fill parity
        for (int j = 0; ok && j < steps; ++j) {
          ok = mbar_spin(&kfull[ks], kph) && (j < 2 || mbar_spin(&pv_done[j & 1], ((j >> 1) - 1) & 1));
          if (!ok) break;
          tc_fence_after();
          const uint64_t kd = kdesc0 + ks * kTileUnits;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t bd = kd + (((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem + kColS + 128 * (j & 1)),
                "r"(tmem + kColQ + kk * 8), "l"(bd), "r"(idesc_s), "r"(static_cast<uint32_t>(kk > 0)));
          }
          mma_commit(&bar_s[j & 1]);
          mma_commit(&kfree[ks]);
          if (++ks == static_cast<uint32_t>(nk)) {
            ks = 0;
            kph ^= 1u;
          }
        }
      } else {
        const uint64_t vdesc0 = sdesc_sw128(smem_u32(vring), 16384, 1024);
        uint32_t vs = 0, vph = 0;  // V stage of PV(j) and its fill parity
        for (int j = 0; ok && j < steps; ++j) {
          ok = mbar_spin(&vfull[vs], vph) && mbar_spin(&bar_p[j & 1], (j >> 1) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t pcol = tmem + kColS + 128 * (j & 1);
          const uint64_t vd = vdesc0 + vs * kTileUnits;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem + kColO),
                "r"(pcol + kk * 8), "l"(vd + ((kk * 2048) >> 4)), "r"(idesc_pv),
                "r"(static_cast<uint32_t>(j > 0 || kk > 0)));
          }
          mma_commit(&vfree[vs]);
          mma_commit(&pv_done[j & 1]);
          if (++vs == static_cast<uint32_t>(nv)) {
            vs = 0;
            vph ^= 1u;
          }
        }
      }
      if (!ok) flag_error(p.err, kErrTimeout);
    }
  } else {
    // ---------------- softmax + epilogue.  Two warps share each 32-row lane
    // quarter: warp (q, h) handles key cube h (columns [64h, 64h + 64)) of
    // the step for rows 32q..32q+31, so each SM sub-partition runs two
    // softmax warps.  The pair agrees on the row max through shared memory;
    // each keeps a partial row sum over its own key cubes.
    const int sw = warp - 2;               // 0..7
    const int quarter = warp & 3;          // TMEM lane quarter this warp may access
    const int half = sw >> 2;              // key cube of the step (S columns)
    const int row = quarter * 32 + lane;   // TMEM lane == tile row
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t my_bit = row < 64 ? 30u : 31u;  // warp-uniform
    uint64_t* pair_mb = &pair_bar[quarter];       // 64-thread barrier of the two warps
    uint32_t pair_uses = 0;
    float m = -INFINITY, l = 0.f;                  // m is identical in both warps
    bool ok = true;
    {
      // Q rows into TMEM (lane = row, column c = elements 2c and 2c + 1):
      // warp (q, h) writes elements [h D/2, (h + 1) D/2) of its 32 rows.
      bool qrow = row < 64 || has_b;
      int64_t qsrc = row_base + 64 * static_cast<int64_t>(row < 64 ? qa : (has_b ? qb : qa)) + (row & 63);
      if (NATIVE) {
        const int64_t tok = native_token(raster_cube(p.order, row < 64 ? qa : (has_b ? qb : qa)), row & 63, p.cgrid);
        qrow = qrow && tok >= 0;  // a padding slot of a partial cube: zero row
        qsrc = bh * p.Nn + (tok >= 0 ? tok : 0);
      }
      const uint4* src = reinterpret_cast<const uint4*>(p.q + qsrc * D + half * (D / 2));
#pragma unroll
      for (int c = 0; c < D / 4; c += 8) {
        uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
        if (qrow && steps > 0) {
          a = src[c / 4];
          b = src[c / 4 + 1];
        }
        const uint32_t r[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        tmem_st8(lane_addr + kColQ + half * (D / 4) + c, r);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_qt);
    }
    for (int j = 0; j < steps; ++j) {
      // A suspended wait: the pair usually finds S(j) done, and a spinning
      // warp would take issue slots from the MMA issuer on its sub-partition.
      if (!mbar_wait(&bar_s[j & 1], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sb = lane_addr + kColS + 128 * (j & 1);
      const uint32_t e = (2 * j + half < U) ? uent(2 * j + half) : 0u;
      const bool valid = ((e >> my_bit) & 1u) != 0;  // warp-uniform
      uint32_t sr[64];
      float mx = -INFINITY;
      if (valid) {
        tmem_ld64_wait(sb + 64 * half, sr);
        if (p.kmask) {
          // A partial cube (a grid side not a multiple of 4): its padding
          // slots are no keys.  Column c of this half is slot c of the cube.
          const uint64_t km = __ldg(p.kmask + (e & 0x3FFFFFFF));
          if (km != ~0ull) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (!((km >> c) & 1ull)) sr[c] = 0xFF800000u;  // -inf
          }
        }
        mx = max64(sr) * p.scale_log2;
      }
      // Exchange the half maxima (double-buffered by step parity).  The
      // exchange also tells each warp that its partner holds its half of
      // S(j), so P(j) may then be written over the first half.
      tc_fence_before();
      xmax[j & 1][half][row] = mx;
      mbar_arrive(pair_mb);
      if (!mbar_spin(pair_mb, pair_uses++ & 1)) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, xmax[j & 1][half ^ 1][row]);

      // Raise the running max only when it grows by more than the threshold.
      const bool raise = mx > m + kRescaleThreshold;
      const float m_new = raise ? mx : m;
      const bool need_rescale = raise && (m != -INFINITY);
      if (__any_sync(0xffffffffu, need_rescale)) {
        // O holds PV(0..j-1); the last of them may still be running.  Each
        // warp of the pair rescales its half of O's columns.
        if (!mbar_spin(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float alpha = need_rescale ? fast_exp2(m - m_new) : 1.0f;
#pragma unroll
        for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32) {
          uint32_t ov[32];
          tmem_ld32_wait(lane_addr + kColO + c, ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
#pragma unroll
          for (int i = 0; i < 32; i += 8) tmem_st8(lane_addr + kColO + c + i, ov + i);
        }
        tmem_wait_st();
        l *= alpha;
      }
      m = m_new;
      // P = exp2(S * scale - m), fp16 pairs into columns [32h, 32h + 32) of
      // S(j)'s buffer.
      // The row sum adds the same rounded weights the PV MMA sees, so O / l
      // stays an exact convex combination of V rows (summing the unrounded
      // weights instead made the output ~4x and dK ~6x less accurate).
      uint32_t pk[32];
      if (valid) {
        float acc0 = 0.f, acc1 = 0.f;
        softmax64<!NATIVE>(sr, splat2(p.scale_log2), splat2(-m), pk, acc0, acc1);
        l += acc0 + acc1;
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = 0u;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 32; c += 8) tmem_st8(sb + 32 * half + c, pk + c);
      if (!F16IN && !NATIVE) {
        // bf16 V tile -> fp16 in place, before the PV MMA may read it.
        const int st = j % nv;
        if (!mbar_wait(&vfull[st], (j / nv) & 1)) {
          ok = false;
          break;
        }
        uint4* vt = reinterpret_cast<uint4*>(vring + st * L::kTile);
        for (int e2 = threadIdx.x - 64; e2 < L::kTile / 16; e2 += kSoftmaxThreads) {
          uint4 u = vt[e2];
          vt[e2] = make_uint4(pack_f16(bf16_lo(u.x), bf16_hi(u.x)), pack_f16(bf16_lo(u.y), bf16_hi(u.y)),
                              pack_f16(bf16_lo(u.z), bf16_hi(u.z)), pack_f16(bf16_lo(u.w), bf16_hi(u.w)));
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_p[j & 1]);
    }
    if (ok && steps > 0 && !mbar_wait(&pv_done[(steps - 1) & 1], ((steps - 1) >> 1) & 1)) ok = false;
    if (!ok) flag_error(p.err, kErrTimeout);
    tc_fence_after();
    // ---------------- epilogue: O / l (each warp of the pair writes half of
    // the columns), LSE.
    // The row sums go through the exchange buffer of the parity no warp of
    // the pair reads any more.
    xmax[steps & 1][half][row] = l;
    mbar_arrive(pair_mb);
    if (!mbar_wait(pair_mb, pair_uses & 1)) {
      ok = false;
      flag_error(p.err, kErrTimeout);
    }
    const float lt = l + xmax[steps & 1][half ^ 1][row];
    const bool row_valid = row < 64 || has_b;
    const int64_t grow = row_base + 64 * static_cast<int64_t>(row < 64 ? qa : (has_b ? qb : qa)) + (row & 63);
    const float inv = lt > 0.f ? 1.0f / lt : 0.f;
#pragma unroll
    for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32) {
      uint32_t ov[32];
      if (steps > 0) tmem_ld32_wait(lane_addr + kColO + c, ov);
      float o[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = (steps > 0 && ok) ? __uint_as_float(ov[i]) * inv : 0.f;
      if (row_valid) {
#pragma unroll
        for (int i = 0; i < 32; i += 8) store8(p.of, grow * D + c + i, o + i, p.of_dtype);
      }
    }
    if (half == 0 && row_valid && p.lse)
      p.lse[grow] = (lt > 0.f) ? (m + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
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

// 5-D bf16 tensor map over the native [BH, T, H, W, d] layout with a
// {64, 4, 4, 4, 1} box: one (4, 4, 4) cube of 64 channels, 128-byte swizzle,
// zeros where the box leaves the grid.
int make_cube_map(void* map_out, const void* base, int BH, int T, int H, int W, int d) {
  CUtensorMap* map = static_cast<CUtensorMap*>(map_out);
  auto enc = get_encoder();
  if (!enc) return VSA_ERR_CUDA;
  const cuuint64_t row = static_cast<cuuint64_t>(d) * 2;
  cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[4] = {row, row * W, row * W * H, row * W * H * T};
  cuuint32_t box[5] = {64, 4, 4, 4, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VSA_OK : VSA_ERR_CUDA;
}

namespace {

// Fills the common fields, sizes the K / V rings and launches.
int run_fine_fwd(FwdParams& p, const int32_t* idx, const int32_t* cnt, int kmax, int BH, int N, int d, float scale,
                 void* of, int of_dtype, float* lse, int f16_in, bool native, const int32_t* pairs,
                 const uint64_t* kmask, cudaStream_t s) {
  p.pairs = pairs;
  p.kmask = kmask;
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
  auto go = [&](auto kernel, size_t tile, int threads) -> int {
    // Q plus as many K/V stages as fit (at most three each, at least one).
    // The 227 KB per-block limit covers the kernel's static shared memory
    // (barriers, row-max exchange) as well.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return VSA_ERR_CUDA;
    const size_t kSmemMax = 227 * 1024 - fa.sharedSizeBytes;
    const size_t fixed = 1024 + extra;
    const long slots = fixed + 2 * tile <= kSmemMax ? static_cast<long>((kSmemMax - fixed) / tile) : 0;
    if (slots < 2) return VSA_ERR_UNSUPPORTED;
    p.nk = static_cast<int>(std::min<long>((slots + 1) / 2, kMaxStages));
    p.nv = static_cast<int>(std::min<long>(slots / 2, kMaxStages));
    // At least 120 KB, so that two CTAs (2 x 512 TMEM columns) never share an SM.
    const size_t smem = std::max<size_t>(fixed + static_cast<size_t>(p.nk + p.nv) * tile, 120 * 1024);
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return VSA_ERR_CUDA;
    timing_mark(VSA_K_FINE_FWD, true, s);
    kernel<<<grid, threads, smem, s>>>(p);
    timing_mark(VSA_K_FINE_FWD, false, s);
    return VSA_OK;
  };
  int st;
  if (d == 128)
    st = native   ? go(fine_fwd_kernel<128, false, true>, FwdLayout<128>::kTile, fwd_threads<true>())
         : f16_in ? go(fine_fwd_kernel<128, true, false>, FwdLayout<128>::kTile, fwd_threads<false>())
                  : go(fine_fwd_kernel<128, false, false>, FwdLayout<128>::kTile, fwd_threads<false>());
  else
    st = native   ? go(fine_fwd_kernel<64, false, true>, FwdLayout<64>::kTile, fwd_threads<true>())
         : f16_in ? go(fine_fwd_kernel<64, true, false>, FwdLayout<64>::kTile, fwd_threads<false>())
                  : go(fine_fwd_kernel<64, false, false>, FwdLayout<64>::kTile, fwd_threads<false>());
  if (st != VSA_OK) return st;
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace

int launch_fine_fwd(const void* qp, const void* kp, const void* vp, const int32_t* idx, const int32_t* cnt, int kmax,
                    int BH, int N, int d, float scale, void* of, int of_dtype, float* lse, int f16_in,
                    const int32_t* pairs, const uint64_t* kmask, cudaStream_t s) {
  FwdParams p{};
  const int64_t rows = static_cast<int64_t>(BH) * N;
  int st;
  if ((st = make_tile_map(&p.tk, kp, rows, d, f16_in)) != VSA_OK) return st;
  if ((st = make_tile_map(&p.tv, vp, rows, d, f16_in)) != VSA_OK) return st;
  p.q = static_cast<const uint16_t*>(qp);
  return run_fine_fwd(p, idx, cnt, kmax, BH, N, d, scale, of, of_dtype, lse, f16_in, false, pairs, kmask, s);
}

size_t fine_fwd_ws_bytes(int BH, int N, int d) {
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  return 3 * a256(sizeof(uint16_t) * static_cast<size_t>(BH) * N * d) + a256(pair_plan_ws_bytes(BH, N / kCube));
}

int launch_fine_fwd_native(const void* q, const void* k, const void* v, int T, int H, int W, const int32_t* order,
                           const int32_t* idx, const int32_t* cnt, int kmax, int BH, int d, float scale, void* of,
                           int of_dtype, float* lse, const int32_t* pairs, const uint64_t* kmask, cudaStream_t s) {
  FwdParams p{};
  int st;
  if ((st = make_cube_map(&p.tk, k, BH, T, H, W, d)) != VSA_OK) return st;
  if ((st = make_cube_map(&p.tv, v, BH, T, H, W, d)) != VSA_OK) return st;
  p.q = static_cast<const uint16_t*>(q);
  p.cgrid = cube_grid(T, H, W);
  p.order = order;
  p.Nn = static_cast<int64_t>(T) * H * W;
  const int Nc = ((T + 3) / 4) * p.cgrid.Hc * p.cgrid.Wc;
  return run_fine_fwd(p, idx, cnt, kmax, BH, Nc * kCube, d, scale, of, of_dtype, lse, 0, true, pairs, kmask, s);
}

}  // namespace vsa
