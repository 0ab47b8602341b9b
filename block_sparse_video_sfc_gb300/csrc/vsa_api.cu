// vsa_api.cu -- the C ABI declared in include/vsa.h: argument checks, the
// workspace layouts, and the order in which the kernels run.  Nothing here
// allocates memory; every buffer belongs to the caller.
#include <mutex>
#include <vector>

#include "common.cuh"
#include "sm100.cuh"

namespace vsa {
namespace {

__device__ int g_error_word;  // latched kernel-side errors (kErrLut | kErrTimeout)

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
std::mutex g_mu;

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// N is the reordered length 64 * Nc (>= T * H * W when a side of the grid is
// not a multiple of 4 and the boundary cubes carry padding slots).
struct Dims {
  int64_t BH, N, Nc;
  int d, T, H, W;
  bool padded;
};

int check_grid(const vsa_grid_t& g, int d, Dims* out, int64_t BH) {
  if (g.ct != 4 || g.ch != 4 || g.cw != 4) return VSA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return VSA_ERR_UNSUPPORTED;
  if (g.T <= 0 || g.H <= 0 || g.W <= 0 || BH <= 0) return VSA_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(g.cube_order) & 3u) return VSA_ERR_ARG;
  const int64_t Nc = static_cast<int64_t>((g.T + 3) / 4) * ((g.H + 3) / 4) * ((g.W + 3) / 4);
  const int64_t N = Nc * kCube;
  if (N * BH >= (int64_t(1) << 31)) return VSA_ERR_UNSUPPORTED;  // TMA row coordinates are int32
  *out = Dims{BH, N, Nc, d, g.T, g.H, g.W, (g.T % 4) || (g.H % 4) || (g.W % 4)};
  return VSA_OK;
}

template <typename T>
T* at(const void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(const_cast<void*>(base)) + off);
}

// Width of the selection lists: the Top-K alone (radius < 0), or with room
// for the radius-r cube neighbourhood added ((2r + 1)^3 cubes at most).
int list_width(int topk, int radius, int64_t Nc) {
  if (radius < 0) return topk;
  const int64_t n = static_cast<int64_t>(topk) + (2 * radius + 1) * (2 * radius + 1) * (2 * radius + 1);
  return static_cast<int>(n < Nc ? n : Nc);
}
// coarse: the coarse stage runs too (its score rows must fit on chip).
int check_selection(const Dims& D, int topk, int radius, bool coarse = true) {
  if (topk < 1 || topk > D.Nc) return VSA_ERR_ARG;
  if (radius < -1 || radius > 7) return VSA_ERR_ARG;
  if (coarse && !coarse_fits(static_cast<int>(D.Nc), D.d, topk, 0)) return VSA_ERR_UNSUPPORTED;
  return VSA_OK;
}

// Forward workspace: the saved state of one vsa_forward call.
struct FwdWs {
  size_t qp, kp, vp, qc, kc, vc, oc, lsec, idx, cnt, of, lse, pairs, kmask, idx_tk, total;
  int kmax;  // width of the saved lists
};
// copies = false: the inference forward, which reads Q, K, V in place.
FwdWs fwd_layout(const Dims& D, int topk, int radius, bool copies = true) {
  FwdWs w{};
  const int K = list_width(topk, radius, D.Nc);
  w.kmax = K;
  size_t o = 0;
  const size_t big_bf16 = copies ? sizeof(__half) * D.BH * D.N * D.d : 0;  // fp16 copies of Q, K, V
  const size_t pooled = sizeof(float) * D.BH * D.Nc * D.d;
  w.qp = o; o += align256(big_bf16);
  w.kp = o; o += align256(big_bf16);
  w.vp = o; o += align256(big_bf16);
  w.qc = o; o += align256(pooled);
  w.kc = o; o += align256(pooled);
  w.vc = o; o += align256(pooled);
  w.oc = o; o += align256(pooled);
  w.lsec = o; o += align256(sizeof(float) * D.BH * D.Nc);
  w.idx = o; o += align256(sizeof(int32_t) * D.BH * D.Nc * K);
  w.cnt = o; o += align256(sizeof(int32_t) * D.BH * D.Nc);
  w.of = o; o += align256(sizeof(float) * D.BH * D.N * D.d);
  w.lse = o; o += align256(sizeof(float) * D.BH * D.N);
  w.pairs = o; o += align256(pair_plan_ws_bytes(static_cast<int>(D.BH), static_cast<int>(D.Nc)));
  w.kmask = o; o += align256(sizeof(uint64_t) * D.Nc);
  w.idx_tk = o; o += radius >= 0 ? align256(sizeof(int32_t) * D.BH * D.Nc * topk) : 0;  // the Top-K before the union
  w.total = o;
  return w;
}

// The coarse stage of vsa_forward / vsa_forward_inference: O_c, the coarse
// log-sum-exp and the selection -- Top-K lists into the saved lists, or, with
// a radius, into scratch and then united with each query cube's neighbourhood
// (ascending lists with counts).
int select_lists(const float* qc, const float* kc, const float* vc, const Dims& D, const vsa_grid_t& g, int topk,
                 int radius, float scale, const FwdWs& w, void* ws, cudaStream_t s) {
  const int BH = static_cast<int>(D.BH), Nc = static_cast<int>(D.Nc);
  int32_t* idx = at<int32_t>(ws, w.idx);
  int32_t* cnt = at<int32_t>(ws, w.cnt);
  int st = launch_coarse_topk(qc, kc, vc, BH, Nc, D.d, topk, scale, 0, at<float>(ws, w.oc), at<float>(ws, w.lsec),
                              radius >= 0 ? at<int32_t>(ws, w.idx_tk) : idx, radius >= 0 ? nullptr : cnt, nullptr, s);
  if (st != VSA_OK || radius < 0) return st;
  return launch_add_neighbors(at<int32_t>(ws, w.idx_tk), nullptr, topk, BH, (g.T + 3) / 4, (g.H + 3) / 4,
                              (g.W + 3) / 4, g.cube_order, radius, w.kmax, idx, cnt, s);
}

// Backward workspace (scratch of one vsa_backward call).
struct BwdWs {
  size_t dof, delta, doc, deltac, dqc, dkc, dvc, inv, kpairs, total;
};
// kmax: the width of the forward's saved lists.
BwdWs bwd_layout(const Dims& D, int kmax) {
  BwdWs w{};
  size_t o = 0;
  const size_t pooled = sizeof(float) * D.BH * D.Nc * D.d;
  w.dof = o; o += align256(sizeof(__half) * D.BH * D.N * D.d);
  w.delta = o; o += align256(sizeof(float) * D.BH * D.N);
  w.doc = o; o += align256(pooled);
  w.deltac = o; o += align256(sizeof(float) * D.BH * D.Nc);
  w.dqc = o; o += align256(pooled);
  w.dkc = o; o += align256(pooled);
  w.dvc = o; o += align256(pooled);
  w.inv = o; o += align256(inverse_lists_bytes(static_cast<int>(D.BH), static_cast<int>(D.Nc), kmax));
  w.kpairs = o; o += align256(pair_plan_ws_bytes(static_cast<int>(D.BH), static_cast<int>(D.Nc)));
  w.total = o;
  return w;
}

struct TimedLaunch {
  cudaEvent_t start, stop;
};
bool g_timing = false;
std::vector<TimedLaunch> g_timed[VSA_K_COUNT];
std::vector<cudaEvent_t> g_event_pool;
cudaEvent_t pooled_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// One thread waits on a barrier that nothing completes, with the bounded
// wait of the fine kernels, then records the timeout like they do.
__global__ void wait_timeout_kernel(uint32_t polls, int* err) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait(&bar, 0, polls)) flag_error(err, kErrTimeout);
}

}  // namespace

void timing_mark(int kernel, bool begin, cudaStream_t s) {
  if (!g_timing || kernel < 0 || kernel >= VSA_K_COUNT) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (begin) {
    cudaEvent_t e = pooled_event();
    if (!e) return;
    cudaEventRecord(e, s);
    g_timed[kernel].push_back(TimedLaunch{e, nullptr});
  } else if (!g_timed[kernel].empty() && !g_timed[kernel].back().stop) {
    cudaEvent_t e = pooled_event();
    if (!e) return;
    cudaEventRecord(e, s);
    g_timed[kernel].back().stop = e;
  }
}

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

// Per device, a stream of the highest priority for the dK/dV chain of
// vsa_backward and the events of its fork from, wait on and join to the
// caller's stream (created on first use).  At that priority the block
// scheduler runs dK/dV first and the dQ kernel, queued on the caller's
// stream, fills the SMs that the dK/dV kernel's last wave leaves idle.
struct AuxStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, mid = nullptr;
  std::mutex mu;  // one fork / join at a time per device (the events are shared)
};
AuxStream g_aux[kMaxDevices];

AuxStream* aux_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  AuxStream& a = g_aux[dev];
  std::lock_guard<std::mutex> lk(g_mu);
  if (!a.s) {
    int least = 0, greatest = 0;
    cudaStream_t st = nullptr;
    cudaEvent_t e1 = nullptr, e2 = nullptr, e3 = nullptr;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&st, cudaStreamNonBlocking, greatest) != cudaSuccess ||
        cudaEventCreateWithFlags(&e1, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&e2, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&e3, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();  // not fatal: the backward then runs on the caller's stream alone
      if (st) cudaStreamDestroy(st);
      if (e1) cudaEventDestroy(e1);
      if (e2) cudaEventDestroy(e2);
      if (e3) cudaEventDestroy(e3);
      return nullptr;
    }
    a.fork = e1;
    a.join = e2;
    a.mid = e3;
    a.s = st;
  }
  return &a;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_num_sms[dev]) cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
  return g_num_sms[dev] > 0 ? g_num_sms[dev] : 148;
}

}  // namespace vsa

using namespace vsa;

extern "C" {

const char* vsa_status_string(int status) {
  switch (status) {
    case VSA_OK: return "ok";
    case VSA_ERR_ARG: return "invalid argument (null pointer, misaligned pointer, bad enum or size)";
    case VSA_ERR_SHAPE: return "shape error (grid not divisible by the (4,4,4) cube or sizes inconsistent)";
    case VSA_ERR_UNSUPPORTED: return "unsupported configuration (d must be 64 or 128, cube (4,4,4))";
    case VSA_ERR_CUDA: return "a CUDA runtime call failed";
    case VSA_ERR_TIMEOUT: return "a kernel's bounded wait expired";
    case VSA_ERR_LUT: return "block index list entry or count out of range, or a repeated cube";
    case VSA_ERR_WORKSPACE: return "workspace missing or too small";
    case VSA_ERR_RANGE: return "a value exceeded the fp16 operand range (|x| > 65504) and was saturated";
    default: return "unknown status";
  }
}

int vsa_timing_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timing = on != 0;
  return VSA_OK;
}

int vsa_timing_read(int kernel, double* total_ms, int* launches) {
  if (kernel < 0 || kernel >= VSA_K_COUNT || !total_ms || !launches) return VSA_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  double sum = 0.0;
  int n = 0, st = VSA_OK;
  for (auto& t : g_timed[kernel]) {
    if (t.stop) {
      float ms = 0.f;
      if (cudaEventSynchronize(t.stop) != cudaSuccess || cudaEventElapsedTime(&ms, t.start, t.stop) != cudaSuccess)
        st = VSA_ERR_CUDA;
      sum += ms;
      ++n;
      g_event_pool.push_back(t.stop);
    }
    g_event_pool.push_back(t.start);
  }
  g_timed[kernel].clear();
  *total_ms = sum;
  *launches = n;
  return st;
}

int vsa_mask_to_lut(const uint8_t* mask, int BH, int Nc, int max_kv_blocks, int32_t* kv_block_idx,
                    int32_t* valid_block_num, void* stream) {
  if (!mask || !kv_block_idx || !valid_block_num) return VSA_ERR_ARG;
  if (BH <= 0 || Nc <= 0 || max_kv_blocks < 1) return VSA_ERR_ARG;
  if (static_cast<int64_t>(BH) * Nc >= (int64_t(1) << 31) || Nc > (1 << 16)) return VSA_ERR_UNSUPPORTED;
  return launch_mask_to_lut(mask, BH, Nc, max_kv_blocks, kv_block_idx, valid_block_num, as_stream(stream));
}

int vsa_lut_add_neighbors(const int32_t* kv_block_idx_in, const int32_t* valid_block_num_in, int max_kv_blocks_in,
                          int BH, vsa_grid_t g, int radius, int max_kv_blocks_out, int32_t* kv_block_idx_out,
                          int32_t* valid_block_num_out, void* stream) {
  Dims D;
  if (BH <= 0) return VSA_ERR_ARG;
  int st = check_grid(g, 128, &D, BH);
  if (st != VSA_OK) return st;
  if (!kv_block_idx_in || !kv_block_idx_out || !valid_block_num_out) return VSA_ERR_ARG;
  if (max_kv_blocks_in < 1 || max_kv_blocks_out < 1 || radius < 0 || radius > 7) return VSA_ERR_ARG;
  if (D.Nc > (1 << 16)) return VSA_ERR_UNSUPPORTED;
  return launch_add_neighbors(kv_block_idx_in, valid_block_num_in, max_kv_blocks_in, BH, (g.T + 3) / 4,
                              (g.H + 3) / 4, (g.W + 3) / 4,
                              g.cube_order, radius, max_kv_blocks_out, kv_block_idx_out, valid_block_num_out, as_stream(stream));
}

int vsa_cube_order(vsa_grid_t g, int curve, int32_t* order, void* stream) {
  g.cube_order = nullptr;
  Dims D;
  int st = check_grid(g, 128, &D, 1);
  if (st != VSA_OK) return st;
  if (!order || (reinterpret_cast<uintptr_t>(order) & 3u)) return VSA_ERR_ARG;
  if (curve != VSA_CURVE_RASTER && curve != VSA_CURVE_HILBERT) return VSA_ERR_ARG;
  return launch_cube_order((g.T + 3) / 4, (g.H + 3) / 4, (g.W + 3) / 4, curve, order, as_stream(stream));
}

int vsa_selftest_wait_timeout(uint32_t polls, void* stream) {
  if (polls < 1 || polls > (1u << 24)) return VSA_ERR_ARG;
  int* err = device_error_word();
  if (!err) return VSA_ERR_CUDA;
  wait_timeout_kernel<<<1, 1, 0, as_stream(stream)>>>(polls, err);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

int vsa_device_status(void* stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return VSA_ERR_CUDA;
  int* p = device_error_word();
  if (!p) return VSA_ERR_CUDA;
  int v = 0, zero = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return VSA_ERR_CUDA;
  if (v && cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return VSA_ERR_CUDA;
  if (v & kErrTimeout) return VSA_ERR_TIMEOUT;
  if (v & kErrLut) return VSA_ERR_LUT;
  if (v & kErrRange) return VSA_ERR_RANGE;
  if (v & kErrNan) return VSA_ERR_ARG;
  return VSA_OK;
}

int vsa_permute(const void* x, void* y, float* pooled, int BH, int d, vsa_grid_t g, int inverse, void* stream) {
  Dims D;
  int st = check_grid(g, d, &D, BH);
  if (st != VSA_OK) return st;
  if (!x || !y || x == y || !aligned16(x) || !aligned16(y) || (pooled && !aligned16(pooled))) return VSA_ERR_ARG;
  if (inverse != 0 && inverse != 1) return VSA_ERR_ARG;
  if (inverse && pooled) return VSA_ERR_ARG;
  const void* src[1] = {x};
  void* dst[1] = {y};
  float* pl[1] = {pooled};
  return launch_permute(src, dst, pl, 1, BH, d, g.T, g.H, g.W, g.cube_order, inverse, 0, as_stream(stream));
}

int vsa_coarse_topk(const float* qc, const float* kc, const float* vc, int BH, int Nc, int d, int topk, float scale,
                    float* o_coarse, float* lse_coarse, int32_t* kv_block_idx, int32_t* valid_block_num,
                    float* scores, void* stream) {
  if (d != 64 && d != 128) return VSA_ERR_UNSUPPORTED;
  if (BH <= 0 || Nc <= 0) return VSA_ERR_ARG;
  if (topk < 1 || topk > Nc) return VSA_ERR_ARG;
  if (!qc || !kc || !kv_block_idx || (o_coarse && (!vc || !lse_coarse))) return VSA_ERR_ARG;
  if (!aligned16(qc) || !aligned16(kc) || (vc && !aligned16(vc)) || (o_coarse && !aligned16(o_coarse)))
    return VSA_ERR_ARG;
  if (!coarse_fits(Nc, d, topk, 1)) return VSA_ERR_UNSUPPORTED;
  return launch_coarse_topk(qc, kc, vc, BH, Nc, d, topk, scale, 1, o_coarse, lse_coarse, kv_block_idx,
                            valid_block_num, scores, as_stream(stream));
}

static int check_fine(const void* qp, const void* kp, const void* vp, const int32_t* idx, int kmax, int BH, int N,
                      int d) {
  if (d != 64 && d != 128) return VSA_ERR_UNSUPPORTED;
  if (BH <= 0 || N <= 0 || kmax < 0) return VSA_ERR_ARG;
  if (N % kCube) return VSA_ERR_SHAPE;
  if (static_cast<int64_t>(BH) * N >= (int64_t(1) << 31)) return VSA_ERR_UNSUPPORTED;
  if (!qp || !kp || !vp || (kmax > 0 && !idx)) return VSA_ERR_ARG;
  if (!aligned16(qp) || !aligned16(kp) || !aligned16(vp)) return VSA_ERR_ARG;
  return VSA_OK;
}

int vsa_fine_fwd(const void* qp, const void* kp, const void* vp, const int32_t* kv_block_idx,
                 const int32_t* valid_block_num, int max_kv_blocks, int BH, int N, int d, float scale, void* o_fine,
                 int o_dtype, float* lse, void* ws, size_t ws_bytes, void* stream) {
  int st = check_fine(qp, kp, vp, kv_block_idx, max_kv_blocks, BH, N, d);
  if (st != VSA_OK) return st;
  if (!o_fine || !aligned16(o_fine)) return VSA_ERR_ARG;
  if (o_dtype != VSA_DTYPE_BF16 && o_dtype != VSA_DTYPE_F32) return VSA_ERR_ARG;
  cudaStream_t s = as_stream(stream);
  if (!ws)  // bf16 operands as given, V converted on chip, cubes 2t and 2t + 1 paired
    return launch_fine_fwd(qp, kp, vp, kv_block_idx, valid_block_num, max_kv_blocks, BH, N, d, scale, o_fine,
                           o_dtype, lse, 0, nullptr, nullptr, s);
  if (ws_bytes < fine_fwd_ws_bytes(BH, N, d) || !aligned16(ws)) return VSA_ERR_WORKSPACE;
  // fp16 copies of Q, K, V (one pass), the query cubes paired by list
  // overlap, then the kernel vsa_forward runs.
  const size_t copy = align256(sizeof(uint16_t) * static_cast<size_t>(BH) * N * d);
  void* h[3] = {at<void>(ws, 0), at<void>(ws, copy), at<void>(ws, 2 * copy)};
  const void* src[3] = {qp, kp, vp};
  int32_t* pairs = at<int32_t>(ws, 3 * copy);
  if ((st = launch_to_f16(src, h, 3, static_cast<int64_t>(BH) * N * d, s)) != VSA_OK) return st;
  st = launch_pair_plan(kv_block_idx, valid_block_num, max_kv_blocks, BH, N / kCube, pairs, s);
  if (st == VSA_ERR_UNSUPPORTED)
    pairs = nullptr;  // too many cubes for the planner's shared memory: cubes 2t, 2t + 1
  else if (st != VSA_OK)
    return st;
  return launch_fine_fwd(h[0], h[1], h[2], kv_block_idx, valid_block_num, max_kv_blocks, BH, N, d, scale, o_fine,
                         o_dtype, lse, 1, pairs, nullptr, s);
}

int vsa_fine_bwd(const void* qp, const void* kp, const void* vp, const void* o_fine, int o_dtype, const float* lse,
                 const void* do_fine, const int32_t* kv_block_idx, const int32_t* valid_block_num, int max_kv_blocks,
                 int BH, int N, int d, float scale, float* dq, float* dk, float* dv, void* ws, size_t ws_bytes,
                 void* stream) {
  int st = check_fine(qp, kp, vp, kv_block_idx, max_kv_blocks, BH, N, d);
  if (st != VSA_OK) return st;
  if (!o_fine || !lse || !do_fine || !dq || !dk || !dv) return VSA_ERR_ARG;
  if (!aligned16(o_fine) || !aligned16(lse) || !aligned16(do_fine) || !aligned16(dq) || !aligned16(dk) ||
      !aligned16(dv))
    return VSA_ERR_ARG;
  if (o_dtype != VSA_DTYPE_BF16 && o_dtype != VSA_DTYPE_F32) return VSA_ERR_ARG;
  if (!ws || ws_bytes < fine_bwd_ws_bytes(BH, N, max_kv_blocks)) return VSA_ERR_WORKSPACE;
  // As in vsa_backward: the dK/dV chain on the auxiliary stream, the dQ
  // kernel on the caller's.
  cudaStream_t s = as_stream(stream), s_kv = s;
  AuxStream* aux = aux_stream();
  std::unique_lock<std::mutex> fork_lock;
  if (aux) {
    fork_lock = std::unique_lock<std::mutex>(aux->mu);
    if (cudaEventRecord(aux->fork, s) != cudaSuccess || cudaStreamWaitEvent(aux->s, aux->fork, 0) != cudaSuccess)
      return VSA_ERR_CUDA;
    s_kv = aux->s;
  }
  st = launch_fine_bwd(qp, kp, vp, o_fine, o_dtype, lse, do_fine, kv_block_idx, valid_block_num, max_kv_blocks, BH,
                       N, d, scale, dq, dk, dv, ws, ws_bytes, s, s_kv, aux ? aux->mid : nullptr);
  if (aux && (cudaEventRecord(aux->join, s_kv) != cudaSuccess || cudaStreamWaitEvent(s, aux->join, 0) != cudaSuccess))
    return VSA_ERR_CUDA;
  return st;
}

size_t vsa_workspace_bytes(int op, int B, int heads, int d, vsa_grid_t g, int topk, int radius) {
  Dims D;
  if (B <= 0 || heads <= 0) return 0;
  if (check_grid(g, d, &D, static_cast<int64_t>(B) * heads) != VSA_OK) return 0;
  const bool fine = op == VSA_OP_FINE_BWD || op == VSA_OP_FINE_FWD;
  if (check_selection(D, topk, fine ? -1 : radius, !fine) != VSA_OK) return 0;
  switch (op) {
    case VSA_OP_FORWARD: return fwd_layout(D, topk, radius).total;
    case VSA_OP_BACKWARD: return bwd_layout(D, list_width(topk, radius, D.Nc)).total;
    case VSA_OP_FINE_BWD: return fine_bwd_ws_bytes(static_cast<int>(D.BH), static_cast<int>(D.N), topk);
    case VSA_OP_FINE_FWD: return fine_fwd_ws_bytes(static_cast<int>(D.BH), static_cast<int>(D.N), d);
    case VSA_OP_FORWARD_INFERENCE: return fwd_layout(D, topk, radius, false).total;
    default: return 0;
  }
}

int vsa_forward_saved(const void* fwd_ws, int B, int heads, int d, vsa_grid_t g, int topk, int radius,
                      vsa_saved_t* out) {
  Dims D;
  if (!fwd_ws || !out || B <= 0 || heads <= 0) return VSA_ERR_ARG;
  int st = check_grid(g, d, &D, static_cast<int64_t>(B) * heads);
  if (st != VSA_OK) return st;
  if ((st = check_selection(D, topk, radius)) != VSA_OK) return st;
  FwdWs w = fwd_layout(D, topk, radius);
  out->qp = at<void>(fwd_ws, w.qp);
  out->kp = at<void>(fwd_ws, w.kp);
  out->vp = at<void>(fwd_ws, w.vp);
  out->qc = at<float>(fwd_ws, w.qc);
  out->kc = at<float>(fwd_ws, w.kc);
  out->vc = at<float>(fwd_ws, w.vc);
  out->o_coarse = at<float>(fwd_ws, w.oc);
  out->lse_coarse = at<float>(fwd_ws, w.lsec);
  out->kv_block_idx = at<int32_t>(fwd_ws, w.idx);
  out->valid_block_num = at<int32_t>(fwd_ws, w.cnt);
  out->o_fine = at<float>(fwd_ws, w.of);
  out->lse = at<float>(fwd_ws, w.lse);
  out->tile_pairs = at<int32_t>(fwd_ws, w.pairs);
  out->max_kv_blocks = w.kmax;
  return VSA_OK;
}

int vsa_backward_tile_pairs(const void* bwd_ws, int B, int heads, int d, vsa_grid_t g, int topk, int radius,
                            int32_t** key_pairs) {
  Dims D;
  if (!bwd_ws || !key_pairs || B <= 0 || heads <= 0) return VSA_ERR_ARG;
  int st = check_grid(g, d, &D, static_cast<int64_t>(B) * heads);
  if (st != VSA_OK) return st;
  if ((st = check_selection(D, topk, radius)) != VSA_OK) return st;
  *key_pairs = at<int32_t>(bwd_ws, bwd_layout(D, list_width(topk, radius, D.Nc)).kpairs);
  return VSA_OK;
}

int vsa_forward(const void* q, const void* k, const void* v, const void* g_coarse, const void* g_fine, int B,
                int heads, int d, vsa_grid_t g, int topk, int radius, float scale, void* out, int out_dtype, void* ws,
                size_t ws_bytes, void* stream) {
  Dims D;
  if (B <= 0 || heads <= 0) return VSA_ERR_ARG;
  int st = check_grid(g, d, &D, static_cast<int64_t>(B) * heads);
  if (st != VSA_OK) return st;
  if ((st = check_selection(D, topk, radius)) != VSA_OK) return st;
  if (!q || !k || !v || !out) return VSA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (g_coarse && !aligned16(g_coarse)) ||
      (g_fine && !aligned16(g_fine)))
    return VSA_ERR_ARG;
  if (out_dtype != VSA_DTYPE_BF16 && out_dtype != VSA_DTYPE_F32) return VSA_ERR_ARG;
  FwdWs w = fwd_layout(D, topk, radius);
  if (!ws || ws_bytes < w.total || !aligned16(ws)) return VSA_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  const int BH = static_cast<int>(D.BH), Nc = static_cast<int>(D.Nc), N = static_cast<int>(D.N);
  const int kmax = w.kmax;
  const void* src[3] = {q, k, v};
  void* dst[3] = {at<void>(ws, w.qp), at<void>(ws, w.kp), at<void>(ws, w.vp)};
  float* pooled[3] = {at<float>(ws, w.qc), at<float>(ws, w.kc), at<float>(ws, w.vc)};
  if ((st = launch_permute(src, dst, pooled, 3, BH, d, g.T, g.H, g.W, g.cube_order, 0, 1, s)) != VSA_OK) return st;
  if ((st = select_lists(pooled[0], pooled[1], pooled[2], D, g, topk, radius, scale, w, ws, s)) != VSA_OK) return st;
  // Pair query cubes whose lists overlap most into the fine kernels' tiles.
  if ((st = launch_pair_plan(at<int32_t>(ws, w.idx), at<int32_t>(ws, w.cnt), kmax, BH, Nc, at<int32_t>(ws, w.pairs),
                              s)) != VSA_OK)
    return st;
  // Padding slots of partial cubes are masked out of the keys.
  uint64_t* kmask = D.padded ? at<uint64_t>(ws, w.kmask) : nullptr;
  if (kmask && (st = launch_slot_masks(g.T, g.H, g.W, g.cube_order, kmask, s)) != VSA_OK) return st;
  if ((st = launch_fine_fwd(dst[0], dst[1], dst[2], at<int32_t>(ws, w.idx), at<int32_t>(ws, w.cnt), kmax, BH, N, d,
                            scale, at<float>(ws, w.of), VSA_DTYPE_F32, at<float>(ws, w.lse), 1,
                            at<int32_t>(ws, w.pairs), kmask, s)) != VSA_OK)
    return st;
  return launch_combine(at<float>(ws, w.oc), at<float>(ws, w.of), g_coarse, g_fine, out, out_dtype, BH, d, g.T, g.H,
                        g.W, g.cube_order, s);
}

int vsa_forward_inference(const void* q, const void* k, const void* v, const void* g_coarse, const void* g_fine,
                          int B, int heads, int d, vsa_grid_t g, int topk, int radius, float scale, void* out,
                          int out_dtype, void* ws, size_t ws_bytes, void* stream) {
  Dims D;
  if (B <= 0 || heads <= 0) return VSA_ERR_ARG;
  int st = check_grid(g, d, &D, static_cast<int64_t>(B) * heads);
  if (st != VSA_OK) return st;
  if ((st = check_selection(D, topk, radius)) != VSA_OK) return st;
  if (!q || !k || !v || !out) return VSA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (g_coarse && !aligned16(g_coarse)) ||
      (g_fine && !aligned16(g_fine)))
    return VSA_ERR_ARG;
  if (out_dtype != VSA_DTYPE_BF16 && out_dtype != VSA_DTYPE_F32) return VSA_ERR_ARG;
  FwdWs w = fwd_layout(D, topk, radius, false);
  if (!ws || ws_bytes < w.total || !aligned16(ws)) return VSA_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  const int BH = static_cast<int>(D.BH), Nc = static_cast<int>(D.Nc);
  const int kmax = w.kmax;
  // Cube means only: the fine kernel reads Q, K, V in their native layout.
  const void* src[3] = {q, k, v};
  void* none[3] = {nullptr, nullptr, nullptr};
  float* pooled[3] = {at<float>(ws, w.qc), at<float>(ws, w.kc), at<float>(ws, w.vc)};
  if ((st = launch_permute(src, none, pooled, 3, BH, d, g.T, g.H, g.W, g.cube_order, 0, 0, s)) != VSA_OK) return st;
  if ((st = select_lists(pooled[0], pooled[1], pooled[2], D, g, topk, radius, scale, w, ws, s)) != VSA_OK) return st;
  if ((st = launch_pair_plan(at<int32_t>(ws, w.idx), at<int32_t>(ws, w.cnt), kmax, BH, Nc, at<int32_t>(ws, w.pairs),
                              s)) != VSA_OK)
    return st;
  uint64_t* kmask = D.padded ? at<uint64_t>(ws, w.kmask) : nullptr;
  if (kmask && (st = launch_slot_masks(g.T, g.H, g.W, g.cube_order, kmask, s)) != VSA_OK) return st;
  if ((st = launch_fine_fwd_native(q, k, v, g.T, g.H, g.W, g.cube_order, at<int32_t>(ws, w.idx),
                                   at<int32_t>(ws, w.cnt), kmax, BH, d, scale, at<float>(ws, w.of), VSA_DTYPE_F32,
                                   at<float>(ws, w.lse), at<int32_t>(ws, w.pairs), kmask, s)) != VSA_OK)
    return st;
  return launch_combine(at<float>(ws, w.oc), at<float>(ws, w.of), g_coarse, g_fine, out, out_dtype, BH, d, g.T, g.H,
                        g.W, g.cube_order, s);
}

int vsa_backward(const void* fwd_ws, const void* g_coarse, const void* g_fine, const void* dout, int B, int heads,
                 int d, vsa_grid_t g, int topk, int radius, float scale, void* dq, void* dk, void* dv, void* dg_coarse,
                 void* dg_fine, int grad_dtype, void* ws, size_t ws_bytes, void* stream) {
  Dims D;
  if (B <= 0 || heads <= 0) return VSA_ERR_ARG;
  int st = check_grid(g, d, &D, static_cast<int64_t>(B) * heads);
  if (st != VSA_OK) return st;
  if ((st = check_selection(D, topk, radius)) != VSA_OK) return st;
  if (!fwd_ws || !dout || !dq || !dk || !dv) return VSA_ERR_ARG;
  if (!aligned16(fwd_ws) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (g_coarse && !aligned16(g_coarse)) || (g_fine && !aligned16(g_fine)) || (dg_coarse && !aligned16(dg_coarse)) ||
      (dg_fine && !aligned16(dg_fine)))
    return VSA_ERR_ARG;
  if (grad_dtype != VSA_DTYPE_BF16 && grad_dtype != VSA_DTYPE_F32) return VSA_ERR_ARG;
  BwdWs w = bwd_layout(D, list_width(topk, radius, D.Nc));
  if (!ws || ws_bytes < w.total || !aligned16(ws)) return VSA_ERR_WORKSPACE;
  FwdWs f = fwd_layout(D, topk, radius);
  cudaStream_t s = as_stream(stream);
  const int BH = static_cast<int>(D.BH), Nc = static_cast<int>(D.Nc), N = static_cast<int>(D.N);
  // Fork at the start: the dK/dV chain on the auxiliary stream (highest
  // priority), whose inverse lists and key plan need only the forward's index
  // lists and so run beside the combine backward; the dK/dV kernel itself
  // waits for the coarse backward (its epilogue adds dK_c, dV_c).  The combine
  // backward, the coarse backward and the dQ kernel run on the caller's
  // stream, which joins the chain at the end.  Without an auxiliary stream
  // everything runs on s.
  AuxStream* aux = aux_stream();
  std::unique_lock<std::mutex> fork_lock;
  cudaStream_t s_kv = s;
  if (aux) {
    fork_lock = std::unique_lock<std::mutex>(aux->mu);
    if (cudaEventRecord(aux->fork, s) != cudaSuccess || cudaStreamWaitEvent(aux->s, aux->fork, 0) != cudaSuccess)
      return VSA_ERR_CUDA;
    s_kv = aux->s;
  }
  if ((st = launch_bwd_prep(dout, g_coarse, g_fine, at<float>(fwd_ws, f.oc), at<float>(fwd_ws, f.of),
                            at<__half>(ws, w.dof), at<float>(ws, w.delta), at<float>(ws, w.doc),
                            at<float>(ws, w.deltac), g_coarse ? dg_coarse : nullptr, g_fine ? dg_fine : nullptr,
                            grad_dtype, BH, d, g.T, g.H, g.W, g.cube_order, s)) != VSA_OK)
    return st;
  if ((st = launch_coarse_bwd(at<float>(fwd_ws, f.qc), at<float>(fwd_ws, f.kc), at<float>(fwd_ws, f.vc),
                              at<float>(ws, w.doc), at<float>(fwd_ws, f.lsec), at<float>(ws, w.deltac), BH, Nc, d,
                              scale, at<float>(ws, w.dqc), at<float>(ws, w.dkc), at<float>(ws, w.dvc), s)) != VSA_OK)
    return st;
  if (aux && cudaEventRecord(aux->mid, s) != cudaSuccess) return VSA_ERR_CUDA;
  FusedGrads fg{dq,
                dk,
                dv,
                at<float>(ws, w.dqc),
                at<float>(ws, w.dkc),
                at<float>(ws, w.dvc),
                grad_dtype,
                cube_grid(g.T, g.H, g.W),
                g.cube_order};
  if ((st = launch_fine_bwd_core(at<void>(fwd_ws, f.qp), at<void>(fwd_ws, f.kp), at<void>(fwd_ws, f.vp),
                                 at<void>(ws, w.dof), at<float>(fwd_ws, f.lse), at<float>(ws, w.delta),
                                 at<int32_t>(fwd_ws, f.idx), at<int32_t>(fwd_ws, f.cnt), f.kmax, BH, N, d, scale,
                                 nullptr, nullptr, nullptr, &fg, at<void>(ws, w.inv), at<int32_t>(fwd_ws, f.pairs),
                                 at<int32_t>(ws, w.kpairs), s, s_kv, aux ? aux->mid : nullptr)) != VSA_OK)
    return st;
  if (aux && (cudaEventRecord(aux->join, s_kv) != cudaSuccess || cudaStreamWaitEvent(s, aux->join, 0) != cudaSuccess))
    return VSA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

}  // extern "C"
