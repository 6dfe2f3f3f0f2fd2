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
// address is looked up with cudaGetSymbolAddress, with the device current,
// on the first call made on that device (the set-up), and kept for later
// calls.  The kept address belongs to the CUDA context that was current at
// the set-up: a call made under another context of that device (a context
// the caller made current itself) repeats the set-up for it.
#include <cuda.h>

#include <mutex>

#include "kvc_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = KVC_SCORE_STATIC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_score_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  CUcontext ctx;  // context current at the set-up
  void *addr;     // device address of g_score_scratch in that context
};
ScratchAddr g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

using CtxGetCurrent = CUresult (*)(CUcontext *);

// The driver's cuCtxGetCurrent, through the runtime's entry-point query (the
// library links only the runtime); NULL if it cannot be found.
CtxGetCurrent ctx_get_current() {
  static CtxGetCurrent fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (CtxGetCurrent) nullptr;
    return reinterpret_cast<CtxGetCurrent>(p);
  }();
  return fn;
}

// Device address of the scratch array in the current device's current
// context.
kvc_status scratch_on_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_ERR_CUDA;
  CtxGetCurrent get = ctx_get_current();
  CUcontext ctx = nullptr;
  // NULL before the runtime's first use of the device: the set-up below
  // makes its context current
  if (!get || get(&ctx) != CUDA_SUCCESS) return KVC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr &e = g_scratch[dev];
  if (!ctx || !e.addr || e.ctx != ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_score_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return KVC_ERR_CUDA;
    }
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return KVC_ERR_CUDA;
    e.ctx = ctx;
    e.addr = p;
  }
  *out = e.addr;
  return KVC_OK;
}

}  // namespace

extern "C" size_t kvc_score_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" kvc_status kvc_score_static(const kvc_bf16 *q, const kvc_bf16 *meank, float *scores,
                                       int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t W,
                                       const int64_t *blk_off, int32_t n_sess, int64_t nb_total,
                                       int32_t nb_max, int32_t *dev_status,
                                       cudaStream_t stream) {
  // kvc_score's own argument, shape and alignment checks come first, so a
  // call that kvc_score would refuse gets the same status here
  const kvc_status args = kvc::score_args_status(q, meank, scores, blk_off, L, H, Hq, D, W,
                                                 n_sess, nb_total, nb_max);
  if (args != KVC_OK) return args;
  // then the scratch these sizes need must fit the fixed array; both checks
  // run before the array is touched or anything is launched
  const size_t need = kvc_score_workspace_size(L, H, Hq, W, n_sess, nb_max, nb_total);
  if (need == 0) return KVC_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return KVC_ERR_WORKSPACE;
  void *scratch = nullptr;
  const kvc_status st = scratch_on_current_device(&scratch);
  if (st != KVC_OK) return st;
  return kvc_score(q, meank, scores, L, H, Hq, D, W, blk_off, n_sess, nb_total, nb_max, scratch,
                   kStaticScratchBytes, dev_status, stream);
}
