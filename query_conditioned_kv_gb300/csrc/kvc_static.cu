// kvc_static.cu — kvc_score for callers that cannot allocate device memory.
//
// Some hosts cannot hand this library a workspace: a serving runtime that
// carves all of HBM into its own KV pool at start-up and forbids device
// allocations afterwards (a cudaMalloc on its serving path would fail or
// fragment the pool), or a plugin running inside such a runtime that is
// given input and output tensors but no allocator.  kvc_score_static serves
// them: it is kvc_score with its scratch taken from a fixed array compiled
// into this library (g_score_scratch below) instead of a caller buffer.
//
// The array is a file-scope __device__ object, so every GPU that loads the
// library holds it until the process exits.  In host code its name is only a
// host-side stand-in for the symbol, never a device address: the device
// address is looked up with cudaGetSymbolAddress, once per device, with
// that device current, on the first call made on that device.
#include <mutex>

#include "kvc_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = KVC_SCORE_STATIC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_score_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];  // device address of g_score_scratch, per device
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.
kvc_status scratch_on_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_score_scratch) != cudaSuccess || !p) return KVC_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KVC_OK;
}

}  // namespace

extern "C" kvc_status kvc_score_static(const kvc_bf16 *q, const kvc_bf16 *meank, float *scores,
                                       int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t W,
                                       const int64_t *blk_off, int32_t n_sess, int64_t nb_total,
                                       int32_t nb_max, int32_t *dev_status,
                                       cudaStream_t stream) {
  if (!q || !meank || !scores || !blk_off) return KVC_ERR_INVALID_ARG;
  // The sizes must be valid and their scratch must fit the fixed array; this
  // is checked before the array is touched or anything is launched.
  const size_t need = kvc_score_workspace_size(L, H, Hq, W, n_sess, nb_max, nb_total);
  if (need == 0) return KVC_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return KVC_ERR_WORKSPACE;
  void *scratch = nullptr;
  kvc_status st = scratch_on_current_device(&scratch);
  if (st != KVC_OK) return st;
  return kvc_score(q, meank, scores, L, H, Hq, D, W, blk_off, n_sess, nb_total, nb_max, scratch,
                   kStaticScratchBytes, dev_status, stream);
}
