// pair_plan.cu -- which two 64-token cubes share a 128-row tile of the fine
// kernels.
//
// The fine kernels run 128-row tensor-core tiles over pairs of cubes and walk
// the UNION of the pair's two cube lists ("Sparse Traversal" of "VSA:
// Accelerating Video Diffusion Inference with Sparse Attention on AMD GPUs"
// walks one list per tile; the pairing is this implementation's, see
// fine_fwd.cu).  The work of a tile is proportional to the size of that
// union, so pairing cubes whose lists overlap most saves work; it changes
// the schedule only, never a result.  Query cubes are paired by their Top-K
// lists (forward and dQ), key cubes by their inverse lists (dK, dV).
//
// Heuristic (deterministic): within a window of +-kWindow cubes in curve
// order, every unpaired cube picks the unpaired cube it shares the most list
// entries with (ties: nearer, then lower id); mutual picks become pairs.
// After kRounds rounds the cubes left over are paired in curve order.  On
// the synthetic 32K-token layer (K = 154 cubes per list) this cuts the mean
// union per pair from 1.63 K to about 1.51 K cubes, i.e. from 251 to 233
// (a global greedy matching reaches 1.48 K).
//
// The overlaps come straight from the lists: a CTA takes kBlock consecutive
// cubes, turns their lists and those of the kWindow cubes after them into
// bitmaps in shared memory and counts the common bits, so no Nc x Nc matrix
// is ever stored.  The lists are either the forward index lists (row c:
// kv_block_idx[c][0 .. valid_block_num[c])) or the inverse lists of the
// backward in CSR form (row c: the query cubes listing key cube c).
#include "common.cuh"

namespace vsa {
namespace {

constexpr int kWindow = 32;
constexpr int kRounds = 8;
constexpr int kPlanThreads = 512;
constexpr int kBlock = 64;               // cubes whose overlaps one CTA counts
constexpr int kOverlapThreads = 256;

// Row c of the forward index lists of head bh.
struct ListRows {
  const int32_t* idx;
  const int32_t* cnt;  // null: every row holds kmax entries
  int kmax, Nc;
  __device__ __forceinline__ int get(int64_t bh, int c, const int32_t** p) const {
    const int64_t row = bh * Nc + c;
    *p = idx + row * kmax;
    const int n = cnt ? __ldg(cnt + row) : kmax;
    return min(max(n, 0), kmax);
  }
};
// Row c of the inverse lists (CSR) of head bh.
struct CsrRows {
  InverseLists inv;
  int Nc;
  __device__ __forceinline__ int get(int64_t bh, int c, const int32_t** p) const {
    const int32_t* off = inv.off + bh * (Nc + 1);
    *p = inv.ids + bh * inv.stride + __ldg(off + c);
    return __ldg(off + c + 1) - __ldg(off + c);
  }
};

// Exclusive prefix sum of one int per thread over the block; returns the
// thread's offset, and the total in *total.
__device__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? scratch[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += t;
    }
    if (lane < nwarps) scratch[lane] = wi - w;
    if (lane == 31) scratch[32] = wi;
  }
  __syncthreads();
  const int res = scratch[warp] + incl - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

// ov[bh][c][d - 1] = |list c & list c + d| for d = 1..kWindow (0 past the
// last cube).  CTA (block, bh): cubes c0 .. c0 + kBlock - 1 and the kWindow
// after them become bitmaps in shared memory (row stride nwords + 1 words,
// odd, so that the threads of a warp, which read different rows at the same
// word, hit different banks); then one thread per (cube, offset) counts.
template <class Rows>
__global__ void __launch_bounds__(kOverlapThreads) pair_overlap_kernel(Rows rows, int Nc, uint16_t* __restrict__ ov) {
  extern __shared__ uint32_t wbits[];
  const int64_t bh = blockIdx.y;
  const int c0 = blockIdx.x * kBlock;
  const int nwords = (Nc + 31) >> 5, stride = nwords + 1;
  const int ncubes = min(kBlock + kWindow, Nc - c0);
  for (int i = threadIdx.x; i < ncubes * stride; i += blockDim.x) wbits[i] = 0u;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < ncubes; i += kOverlapThreads / 32) {
    const int32_t* list;
    const int n = rows.get(bh, c0 + i, &list);
    for (int e = lane; e < n; e += 32) {
      const int c = __ldg(list + e);
      if (c >= 0 && c < Nc) atomicOr(&wbits[i * stride + (c >> 5)], 1u << (c & 31));  // others: reported elsewhere
    }
  }
  __syncthreads();
  for (int it = threadIdx.x; it < kBlock * kWindow; it += blockDim.x) {
    const int i = it / kWindow, d = it % kWindow + 1;
    const int c = c0 + i;
    if (c >= Nc) continue;
    int n = 0;
    if (c + d < Nc) {
      const uint32_t* a = wbits + i * stride;
      const uint32_t* b = wbits + (i + d) * stride;
      for (int w = 0; w < nwords; ++w) n += __popc(a[w] & b[w]);
    }
    ov[(bh * Nc + c) * kWindow + d - 1] = static_cast<uint16_t>(n);
  }
}

// One CTA per (batch, head).  Shared memory: the head's overlaps
// [Nc][kWindow] (uint16), partner[Nc], pick[Nc], rank list[Nc] (int16).
__global__ void __launch_bounds__(kPlanThreads) plan_pairs_kernel(const uint16_t* __restrict__ ov_g, int Nc,
                                                                  int32_t* __restrict__ pairs) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* ov = reinterpret_cast<uint16_t*>(smem);  // ov[c * kWindow + d - 1] = |list c & list c+d|
  int16_t* partner = reinterpret_cast<int16_t*>(ov + static_cast<size_t>(Nc) * kWindow);
  int16_t* pick = partner + Nc;
  int16_t* order = pick + Nc;
  __shared__ int scan_scratch[33];
  const int64_t bh = blockIdx.x;
  const int tid = threadIdx.x;
  {
    const uint4* src = reinterpret_cast<const uint4*>(ov_g + bh * Nc * kWindow);  // kWindow * 2 B = 4 x 16 B per cube
    uint4* dst = reinterpret_cast<uint4*>(ov);
    for (int i = tid; i < Nc * kWindow / 8; i += blockDim.x) dst[i] = src[i];
  }
  for (int c = tid; c < Nc; c += blockDim.x) partner[c] = -1;
  __syncthreads();

  auto overlap = [&](int c, int b) -> int {
    return c < b ? ov[c * kWindow + (b - c - 1)] : ov[b * kWindow + (c - b - 1)];
  };
  for (int round = 0; round < kRounds; ++round) {
    for (int c = tid; c < Nc; c += blockDim.x) {
      int best = -1, best_ov = -1, best_dist = 0;
      if (partner[c] < 0) {
        const int lo = max(0, c - kWindow), hi = min(Nc - 1, c + kWindow);
        for (int b = lo; b <= hi; ++b) {
          if (b == c || partner[b] >= 0) continue;
          const int o = overlap(c, b), dist = abs(b - c);
          if (o > best_ov || (o == best_ov && dist < best_dist)) {  // scanning b upward keeps the lower id on a full tie
            best = b;
            best_ov = o;
            best_dist = dist;
          }
        }
      }
      pick[c] = static_cast<int16_t>(best);
    }
    __syncthreads();
    for (int c = tid; c < Nc; c += blockDim.x) {
      const int b = pick[c];
      if (partner[c] < 0 && b >= 0 && pick[b] == c) partner[c] = static_cast<int16_t>(b);
    }
    __syncthreads();
  }

  // Cubes still unpaired: pair them in curve order (a lone cube when the count is odd).
  const int per = (Nc + blockDim.x - 1) / blockDim.x;
  const int c0 = tid * per, c1 = min(Nc, c0 + per);
  int mine = 0;
  for (int c = c0; c < c1; ++c) mine += partner[c] < 0;
  int nleft = 0;
  int r = block_exclusive_scan(mine, scan_scratch, &nleft);
  for (int c = c0; c < c1; ++c)
    if (partner[c] < 0) order[r++] = static_cast<int16_t>(c);
  __syncthreads();
  for (int i = tid; 2 * i + 1 < nleft; i += blockDim.x) {
    partner[order[2 * i]] = order[2 * i + 1];
    partner[order[2 * i + 1]] = order[2 * i];
  }
  __syncthreads();

  // One tile per pair, listed by the pair's lower cube (curve order).
  const int lone = (nleft & 1) ? order[nleft - 1] : -1;
  mine = 0;
  for (int c = c0; c < c1; ++c) mine += (partner[c] > c) || (c == lone);
  int total = 0;
  r = block_exclusive_scan(mine, scan_scratch, &total);
  const int npairs = (Nc + 1) / 2;
  int32_t* out = pairs + bh * npairs * 2;
  for (int c = c0; c < c1; ++c) {
    if (partner[c] > c || c == lone) {
      out[2 * r] = c;
      out[2 * r + 1] = c == lone ? -1 : partner[c];
      ++r;
    }
  }
}

}  // namespace

size_t pair_plan_smem(int Nc) { return static_cast<size_t>(Nc) * (kWindow * 2 + 3 * 2); }
static size_t a256(size_t x) { return (x + 255) & ~size_t(255); }
size_t pair_plan_ws_bytes(int BH, int Nc) {
  return a256(sizeof(int32_t) * static_cast<size_t>(BH) * ((Nc + 1) / 2) * 2) +
         a256(sizeof(uint16_t) * static_cast<size_t>(BH) * Nc * kWindow);
}

namespace {

template <class Rows>
int plan(const Rows& rows, int BH, int Nc, int32_t* pairs_ws, cudaStream_t s) {
  if (Nc > 32767) return VSA_ERR_UNSUPPORTED;
  const size_t smem = pair_plan_smem(Nc);
  if (smem > 200 * 1024) return VSA_ERR_UNSUPPORTED;
  const size_t osmem = sizeof(uint32_t) * static_cast<size_t>(kBlock + kWindow) * ((Nc + 31) / 32 + 1);
  if (osmem > 200 * 1024) return VSA_ERR_UNSUPPORTED;
  uint16_t* ov = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(pairs_ws) +
                                             a256(sizeof(int32_t) * static_cast<size_t>(BH) * ((Nc + 1) / 2) * 2));
  if (cudaFuncSetAttribute(pair_overlap_kernel<Rows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(osmem)) != cudaSuccess)
    return VSA_ERR_CUDA;
  dim3 g1((Nc + kBlock - 1) / kBlock, BH);
  pair_overlap_kernel<Rows><<<g1, kOverlapThreads, osmem, s>>>(rows, Nc, ov);
  if (cudaFuncSetAttribute(plan_pairs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return VSA_ERR_CUDA;
  plan_pairs_kernel<<<BH, kPlanThreads, smem, s>>>(ov, Nc, pairs_ws);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // namespace

// pairs_ws: pair_plan_ws_bytes(BH, Nc) bytes; the pairs come first, the
// overlap scratch after them.
int launch_pair_plan(const int32_t* idx, const int32_t* cnt, int kmax, int BH, int Nc, int32_t* pairs_ws,
                     cudaStream_t s) {
  return plan(ListRows{idx, cnt, kmax, Nc}, BH, Nc, pairs_ws, s);
}
int launch_pair_plan_inverse(const InverseLists& inv, int BH, int Nc, int32_t* pairs_ws, cudaStream_t s) {
  return plan(CsrRows{inv, Nc}, BH, Nc, pairs_ws, s);
}

}  // namespace vsa
