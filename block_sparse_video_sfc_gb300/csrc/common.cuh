// common.cuh -- shared definitions of the VSA CUDA library (host and device).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/vsa.h"

namespace vsa {

constexpr int kCube = 64;  // (4, 4, 4) tokens per cube

// Bits of the device-side error word (see vsa_device_status).
enum : int { kErrLut = 1, kErrTimeout = 2, kErrRange = 4, kErrNan = 8 };

__device__ __forceinline__ void flag_error(int* err, int bit) {
  if (err) atomicOr(err, bit);
}

// A (T, H, W) token grid covered by cubes of (4, 4, 4): Hc = ceil(H / 4)
// and Wc = ceil(W / 4) cubes along h and w.  When a side is not a multiple
// of 4 the boundary cubes stick out of the grid; their slots outside it are
// padding.
struct CubeGrid {
  int T, H, W, Hc, Wc;
};
inline CubeGrid cube_grid(int T, int H, int W) { return CubeGrid{T, H, W, (H + 3) / 4, (W + 3) / 4}; }

// Native token n = (t*H + h)*W + w at offset o (0..63) of raster cube rc =
// (ct*Hc + ch)*Wc + cw, with t = 4ct + o/16, h = 4ch + (o/4)%4, w = 4cw + o%4;
// -1 when that slot is padding.
__host__ __device__ __forceinline__ int64_t native_token(int rc, int o, const CubeGrid& g) {
  const int cw = rc % g.Wc, ch = (rc / g.Wc) % g.Hc, ct = rc / (g.Wc * g.Hc);
  const int t = 4 * ct + (o >> 4), h = 4 * ch + ((o >> 2) & 3), w = 4 * cw + (o & 3);
  if (t >= g.T || h >= g.H || w >= g.W) return -1;
  return (static_cast<int64_t>(t) * g.H + h) * g.W + w;
}

// Number of grid tokens in raster cube rc (64 unless the cube is partial).
__host__ __device__ __forceinline__ int cube_tokens(int rc, const CubeGrid& g) {
  const int cw = rc % g.Wc, ch = (rc / g.Wc) % g.Hc, ct = rc / (g.Wc * g.Hc);
  return min(4, g.T - 4 * ct) * min(4, g.H - 4 * ch) * min(4, g.W - 4 * cw);
}

// Raster id of the cube at position `pos` of the cube sequence: the first
// half of a vsa_cube_order table, or pos itself when there is none.
__device__ __forceinline__ int raster_cube(const int32_t* order, int pos) { return order ? __ldg(order + pos) : pos; }

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
// fp16 pair, round to nearest; values beyond the fp16 range saturate to
// +-65504 instead of becoming infinite.
constexpr float kF16Max = 65504.0f;
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 p = __floats2half2_rn(fminf(fmaxf(lo, -kF16Max), kF16Max), fminf(fmaxf(hi, -kF16Max), kF16Max));
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ float f16_lo(uint32_t v) { return __low2float(*reinterpret_cast<const __half2*>(&v)); }
__device__ __forceinline__ float f16_hi(uint32_t v) { return __high2float(*reinterpret_cast<const __half2*>(&v)); }

// Store 8 consecutive floats as bf16 (16 bytes) or f32 (32 bytes).
__device__ __forceinline__ void store8(void* base, int64_t elem, const float* v, int dtype) {
  if (dtype == VSA_DTYPE_BF16) {
    uint4 u;
    u.x = pack_bf16(v[0], v[1]);
    u.y = pack_bf16(v[2], v[3]);
    u.z = pack_bf16(v[4], v[5]);
    u.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + elem) = u;
  } else {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + elem);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    p[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}
__device__ __forceinline__ void load8_bf16(const void* base, int64_t elem, float* v) {
  uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + elem);
  v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x);
  v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
  v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z);
  v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void load8_f32(const float* base, int64_t elem, float* v) {
  float4 a = *reinterpret_cast<const float4*>(base + elem);
  float4 b = *reinterpret_cast<const float4*>(base + elem + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const void* base, int64_t elem, int dtype, float* v) {
  if (dtype == VSA_DTYPE_BF16) load8_bf16(base, elem, v);
  else load8_f32(static_cast<const float*>(base), elem, v);
}

// ---------------------------------------------------------------- host side
int* device_error_word();          // per-device error word (vsa_api.cu)
// Kernel timing hooks (vsa_timing_enable): no-ops unless enabled.
void timing_mark(int kernel, bool begin, cudaStream_t s);
int num_sms();                     // SM count of the current device

int launch_permute(const void* const* src, void* const* dst, float* const* pooled, int ntensors, int BH,
                   int d, int T, int H, int W, const int32_t* order, int inverse, int f16_out, cudaStream_t s);
int launch_cube_order(int Tc, int Hc, int Wc, int curve, int32_t* order, cudaStream_t s);
int make_tile_map(void* map, const void* base, int64_t rows, int d, int f16);
// Coarse scores, each row's log-sum-exp and Top-K, and O_c (oc non-null),
// score rows kept on chip; scores non-null receives them as well.  sorted:
// lists highest first (ties to the lower id), else in ascending cube id.  A
// NaN score latches kErrNan.
int launch_coarse_topk(const float* qc, const float* kc, const float* vc, int BH, int Nc, int d, int topk,
                       float scale, int sorted, float* oc, float* lse_c, int32_t* idx, int32_t* cnt, float* scores,
                       cudaStream_t s);
// Whether the coarse forward's score rows and scratch fit shared memory.
bool coarse_fits(int Nc, int d, int topk, int sorted);
int launch_fine_fwd(const void* qp, const void* kp, const void* vp, const int32_t* idx, const int32_t* cnt,
                    int kmax, int BH, int N, int d, float scale, void* of, int of_dtype, float* lse, int f16_in,
                    const int32_t* pairs, const uint64_t* kmask, cudaStream_t s);
// The fine forward reading Q, K, V straight from the native [BH, T, H, W, d]
// bf16 layout (5-D TMA boxes, one per cube); O_f and lse come out in cube order.
int launch_fine_fwd_native(const void* q, const void* k, const void* v, int T, int H, int W, const int32_t* order,
                           const int32_t* idx, const int32_t* cnt, int kmax, int BH, int d, float scale, void* of,
                           int of_dtype, float* lse, const int32_t* pairs, const uint64_t* kmask, cudaStream_t s);
// kmask[c] (c = cube position): bit o set when slot o holds a grid token.
int launch_slot_masks(int T, int H, int W, const int32_t* order, uint64_t* kmask, cudaStream_t s);
size_t pair_plan_smem(int Nc);
size_t pair_plan_ws_bytes(int BH, int Nc);  // pairs + overlap scratch of launch_pair_plan
// Inverse lists in CSR form: for head bh, the query cubes whose index list
// holds key cube c are ids[bh * stride + off[bh][c] .. off[bh][c + 1]) (in no
// particular order); off is [BH][Nc + 1].
struct InverseLists {
  const int32_t* off;
  const int32_t* ids;
  int64_t stride;
};
size_t inverse_lists_bytes(int BH, int Nc, int kmax);  // off, cursors and ids of build_inverse_lists
// Builds the CSR inverse lists of [BH, Nc, kmax] index lists (counts cnt, or
// null for full rows) in ws (inverse_lists_bytes); entries outside [0, Nc)
// and counts outside [0, kmax] latch kErrLut.
int launch_inverse_lists(const int32_t* idx, const int32_t* cnt, int kmax, int BH, int Nc, void* ws,
                         InverseLists* out, cudaStream_t s);
// Pairs query cubes by their index lists / key cubes by their inverse lists.
int launch_pair_plan(const int32_t* idx, const int32_t* cnt, int kmax, int BH, int Nc, int32_t* pairs,
                     cudaStream_t s);
int launch_pair_plan_inverse(const InverseLists& inv, int BH, int Nc, int32_t* pairs, cudaStream_t s);
int launch_mask_to_lut(const uint8_t* mask, int BH, int Nc, int kmax, int32_t* idx, int32_t* cnt, cudaStream_t s);
int launch_add_neighbors(const int32_t* idx_in, const int32_t* cnt_in, int kmax_in, int BH, int Tc, int Hc, int Wc,
                         const int32_t* order, int radius, int kmax_out, int32_t* idx_out, int32_t* cnt_out,
                         cudaStream_t s);
size_t fine_bwd_ws_bytes(int BH, int N, int kmax);
// Where the fine backward kernels put their gradient rows.  With no
// FusedGrads, fp32 rows in cube order into dq / dk / dv [BH*N, d].  With one,
// the backward of the mean pool and the inverse reorder run in the kernels'
// epilogues: row (cube c, slot o) plus c's coarse gradient divided by c's
// token count goes to its native token of the grad_dtype outputs
// [BH, T*H*W, d]; padding slots are dropped.
struct FusedGrads {
  void* dq;
  void* dk;
  void* dv;
  const float* dqc;  // coarse gradients [BH, Nc, d], cube order
  const float* dkc;
  const float* dvc;
  int grad_dtype;
  CubeGrid grid;
  const int32_t* order;  // cube order table, or null (raster)
};
// bf16 -> fp16 copies of n (1..4) tensors of elems elements each (elems % 8
// == 0, 16-byte aligned), one launch; out-of-range values latch kErrRange.
int launch_to_f16(const void* const* src, void* const* dst, int n, int64_t elems, cudaStream_t s);
// Workspace of the public fine forward: fp16 copies of Q, K, V and the
// query-cube pair plan.
size_t fine_fwd_ws_bytes(int BH, int N, int d);
// The public fine backward.  s_kv: the stream of the dK/dV chain (may be s);
// ready: an event recorded on s once the fp16 copies exist, which the dK/dV
// kernel waits for (null when s_kv is s).
int launch_fine_bwd(const void* qp, const void* kp, const void* vp, const void* of, int of_dtype,
                    const float* lse, const void* dof, const int32_t* idx, const int32_t* cnt, int kmax, int BH,
                    int N, int d, float scale, float* dq, float* dk, float* dv, void* ws, size_t ws_bytes,
                    cudaStream_t s, cudaStream_t s_kv, cudaEvent_t ready);
// kv_after: an event the dK/dV kernel waits for on s_kv (its inverse lists
// and plan do not), or null.
int launch_fine_bwd_core(const void* qp, const void* kp, const void* vp, const void* dof, const float* lse,
                         const float* delta, const int32_t* idx, const int32_t* cnt, int kmax, int BH, int N, int d,
                         float scale, float* dq, float* dk, float* dv, const FusedGrads* fused, void* inv_ws,
                         const int32_t* qpairs, int32_t* kpairs_ws, cudaStream_t s, cudaStream_t s_kv,
                         cudaEvent_t kv_after);
int launch_combine(const float* oc, const float* of, const void* gc, const void* gf, void* out, int out_dtype,
                   int BH, int d, int T, int H, int W, const int32_t* order, cudaStream_t s);
// delta_c (may be null) receives D_c = dO_c . O_c of each cube.
int launch_bwd_prep(const void* dout, const void* gc, const void* gf, const float* oc, const float* of,
                    __half* dof, float* delta, float* doc, float* delta_c, void* dgc, void* dgf, int grad_dtype,
                    int BH, int d, int T, int H, int W, const int32_t* order, cudaStream_t s);
// Coarse backward from the row statistic delta_c [BH, Nc] (D = dO_c . O_c,
// written by launch_bwd_prep).
int launch_coarse_bwd(const float* qc, const float* kc, const float* vc, const float* doc, const float* lse_c,
                      const float* delta_c, int BH, int Nc, int d, float scale, float* dqc, float* dkc, float* dvc,
                      cudaStream_t s);

}  // namespace vsa
