// vsa_noalloc.cu -- vsa_fine_bwd_noalloc: the fine-stage backward for callers
// that cannot hand the library any scratch memory.
//
// Some callers own no device allocator of their own: code embedded in a
// runtime or framework that hands out device memory only through its own pool
// (or forbids new allocations once it is running), and plain C callers that
// have the input and output buffers but nothing to pass as a workspace.  For
// them this entry point keeps its scratch (the inverse-list bit matrix, the
// per-row D and the fp16 copies of Q, K, V, dO) in one file-scope device
// array of fixed size.  The array belongs to this file's device module: a
// device holds it from the first call on that device (CUDA loads modules
// lazily by default; with CUDA_MODULE_LOADING=EAGER from library load) until
// the process exits.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the device address is looked up once per
// device with cudaGetSymbolAddress, on the first call made with that device
// current, and cached.  A cudaDeviceReset destroys the array with the
// context, which leaves the cached address stale.
#include <mutex>

#include "common.cuh"

namespace vsa {
namespace {

constexpr size_t kScratchBytes = VSA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set up on the
// first call per device); nullptr on failure.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace vsa

using namespace vsa;

extern "C" int vsa_fine_bwd_noalloc(const void* qp, const void* kp, const void* vp, const void* o_fine, int o_dtype,
                                    const float* lse, const void* do_fine, const int32_t* kv_block_idx,
                                    const int32_t* valid_block_num, int max_kv_blocks, int BH, int N, int d,
                                    float scale, float* dq, float* dk, float* dv, void* stream) {
  if (d != 64 && d != 128) return VSA_ERR_UNSUPPORTED;
  if (BH <= 0 || N <= 0 || max_kv_blocks < 0) return VSA_ERR_ARG;
  if (N % kCube) return VSA_ERR_SHAPE;
  const size_t need = fine_bwd_ws_bytes(BH, N, max_kv_blocks);
  if (need > kScratchBytes) return VSA_ERR_WORKSPACE;  // beyond the fixed scratch: use vsa_fine_bwd
  void* scratch = scratch_address();
  if (!scratch) return VSA_ERR_CUDA;
  // Every buffer of the shared scratch that must start at zero (the inverse
  // bit matrix) is cleared on the stream by the launcher before use.
  return vsa_fine_bwd(qp, kp, vp, o_fine, o_dtype, lse, do_fine, kv_block_idx, valid_block_num, max_kv_blocks, BH,
                      N, d, scale, dq, dk, dv, scratch, kScratchBytes, stream);
}
