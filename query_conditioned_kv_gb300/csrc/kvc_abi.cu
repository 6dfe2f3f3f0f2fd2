// kvc_abi.cu — the extern "C" boundary of libkvc: host-side validation of
// every call (before any launch), then the launch of the kernels in this
// directory on the caller's stream.  No allocation, no state.
#include <math.h>

#include "kvc_internal.cuh"
#include "tc_ptx.cuh"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool head_dim_ok(int D) { return D == 64 || D == 128; }

kvc_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA; }

// A launch refused because the named kernel does not cover the sizes.
kvc_status from_cuda_kernel(cudaError_t e) {
  if (e == cudaErrorNotSupported) {
    (void)cudaGetLastError();
    return KVC_ERR_SHAPE;
  }
  return from_cuda(e);
}

bool score_kernel_ok(kvc_kernel k) {
  return k == KVC_KERNEL_AUTO || (k >= KVC_KERNEL_SCORE_FUSED && k <= KVC_KERNEL_SCORE_GROUP);
}

__global__ void k_init_sentinel(uint16_t *kpool, uint16_t *vpool, int L, int H,
                                int D, int64_t n_slots, int32_t sentinel) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t per_layer = (int64_t)H * D;
  if (t >= (int64_t)L * per_layer) return;
  int64_t l = t / per_layer, e = t - l * per_layer;
  int64_t idx = (l * n_slots + sentinel) * per_layer + e;
  kpool[idx] = (uint16_t)KVC_SENTINEL_K_BITS;
  if (vpool) vpool[idx] = 0;
}

// One thread waits, through the kernels' bounded wait, on an mbarrier that no
// thread arrives on; the wait gives up after a second and the kernel records
// KVC_ERR_TIMEOUT.
__global__ void k_selftest_wait(int32_t *status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int failed;
  if (threadIdx.x == 0) {
    kvc::tc::mbar_init(kvc::tc::smem_u32(&bar), 1);
    failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0 &&
      !kvc::tc::mbar_wait_bounded(kvc::tc::smem_u32(&bar), 0, (volatile int *)&failed))
    kvc::record_error(status, KVC_ERR_TIMEOUT);
}

}  // namespace

namespace kvc {

kvc_status score_args_status(const void *q, const void *meank, const void *scores,
                             const int64_t *blk_off, int L, int H, int Hq, int D, int W,
                             int n_sess, int64_t nb_total, int nb_max) {
  if (!q || !meank || !scores || !blk_off) return KVC_ERR_INVALID_ARG;
  if (L < 1 || H < 1 || Hq < 1 || W < 1 || n_sess < 1 || nb_total < 1 || nb_max < 1 ||
      nb_max > nb_total)
    return KVC_ERR_INVALID_ARG;
  if (!head_dim_ok(D) || Hq % H || (int64_t)(Hq / H) * W > KVC_SCORE_MAX_ROWS ||
      (int64_t)L * H * n_sess > 65535)
    return KVC_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(meank) || !aligned16(scores)) return KVC_ERR_ALIGN;
  return KVC_OK;
}

}  // namespace kvc

extern "C" {

const char *kvc_status_string(kvc_status s) {
  switch (s) {
    case KVC_OK: return "ok";
    case KVC_ERR_INVALID_ARG: return "invalid argument (NULL pointer or size out of range)";
    case KVC_ERR_SHAPE: return "unsupported shape";
    case KVC_ERR_BUDGET: return "invalid budget (budget < 1 or sink + recent > budget)";
    case KVC_ERR_ALIGN: return "pointer not 16-byte aligned";
    case KVC_ERR_WORKSPACE: return "workspace too small";
    case KVC_ERR_CUDA: return "CUDA launch or copy failed";
    case KVC_ERR_BOUNDS: return "device: index or offset out of range";
    case KVC_ERR_NAN: return "device: NaN score";
    case KVC_ERR_TIMEOUT: return "device: bounded wait timed out";
    case KVC_ERR_CAPACITY:
      return "capacity exceeded (device: the freed-slot list; host: more blocks needed at once "
             "than repository slots)";
    case KVC_ERR_IO: return "host: reading or writing the repository's backing file failed";
    case KVC_ERR_NOMEM: return "host: out of memory for the repository's tables";
  }
  return "unknown status";
}

const char *kvc_version(void) { return "0.1.0"; }

kvc_status kvc_selftest_bounded_wait(int32_t *dev_status, cudaStream_t stream) {
  if (!dev_status) return KVC_ERR_INVALID_ARG;
  k_selftest_wait<<<1, 32, 0, stream>>>(dev_status);
  return from_cuda(cudaGetLastError());
}

kvc_status kvc_device_status(const int32_t *dev_status, int32_t *host_out) {
  if (!dev_status || !host_out) return KVC_ERR_INVALID_ARG;
  return from_cuda(cudaMemcpy(host_out, dev_status, sizeof(int32_t),
                              cudaMemcpyDeviceToHost));
}

kvc_status kvc_build_meank(const kvc_bf16 *kraw, kvc_bf16 *meank, int32_t L,
                           int32_t H, int32_t D, int64_t n_tok,
                           int32_t *dev_status, cudaStream_t stream) {
  (void)dev_status;
  if (!kraw || !meank || L < 1 || H < 1 || n_tok < 1) return KVC_ERR_INVALID_ARG;
  if (!head_dim_ok(D) || n_tok % KVC_BLOCK_TOKENS) return KVC_ERR_SHAPE;
  if (!aligned16(kraw) || !aligned16(meank)) return KVC_ERR_ALIGN;
  return from_cuda(kvc::launch_build_meank(kraw, meank, (int64_t)L * H, n_tok, D, stream));
}

size_t kvc_score_workspace_size(int32_t L, int32_t H, int32_t Hq, int32_t W,
                                int32_t n_sess, int32_t nb_max, int64_t nb_total) {
  if (L < 1 || H < 1 || Hq < H || Hq % H || W < 1 || n_sess < 1 || nb_max < 1 ||
      nb_total < nb_max || (int64_t)L * H * n_sess > 65535 ||
      (int64_t)(Hq / H) * W > KVC_SCORE_MAX_ROWS)
    return 0;
  return kvc::score_meank_ws_bytes(L, H, Hq, W, n_sess, nb_max, nb_total);
}

kvc_status kvc_score_ex(const kvc_bf16 *q, const kvc_bf16 *meank, float *scores,
                        int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t W,
                        const int64_t *blk_off, int32_t n_sess, int64_t nb_total,
                        int32_t nb_max, void *ws, size_t ws_bytes,
                        int32_t *dev_status, kvc_kernel kernel, cudaStream_t stream) {
  if (!ws || !score_kernel_ok(kernel)) return KVC_ERR_INVALID_ARG;
  const kvc_status args = kvc::score_args_status(q, meank, scores, blk_off, L, H, Hq, D, W,
                                                 n_sess, nb_total, nb_max);
  if (args != KVC_OK) return args;
  if (!aligned16(ws)) return KVC_ERR_ALIGN;
  if (ws_bytes < kvc_score_workspace_size(L, H, Hq, W, n_sess, nb_max, nb_total))
    return KVC_ERR_WORKSPACE;
  return from_cuda_kernel(kvc::launch_score_meank(q, meank, scores, L, H, Hq, D, W, blk_off,
                                                  n_sess, nb_total, nb_max, ws, dev_status,
                                                  (int)kernel, stream));
}

kvc_status kvc_score(const kvc_bf16 *q, const kvc_bf16 *meank, float *scores,
                     int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t W,
                     const int64_t *blk_off, int32_t n_sess, int64_t nb_total,
                     int32_t nb_max, void *ws, size_t ws_bytes,
                     int32_t *dev_status, cudaStream_t stream) {
  return kvc_score_ex(q, meank, scores, L, H, Hq, D, W, blk_off, n_sess, nb_total, nb_max, ws,
                      ws_bytes, dev_status, KVC_KERNEL_AUTO, stream);
}

int32_t kvc_score_launches(int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t W,
                           int32_t n_sess, int32_t nb_max) {
  if (L < 1 || H < 1 || Hq < H || Hq % H || W < 1 || n_sess < 1 || nb_max < 1 || !head_dim_ok(D))
    return 0;
  return kvc::score_meank_launches(H, Hq, D, W, n_sess, nb_max);
}

kvc_status kvc_qmem_update(float *M, const kvc_bf16 *q_turn, int32_t n_sess,
                           int32_t L, int32_t Hq, int32_t D, int32_t T,
                           float decay, float gain, int32_t renorm,
                           cudaStream_t stream) {
  if (!M || !q_turn || n_sess < 1 || L < 1 || Hq < 1 || T < 1) return KVC_ERR_INVALID_ARG;
  if (!head_dim_ok(D)) return KVC_ERR_SHAPE;
  if (!aligned16(M) || !aligned16(q_turn)) return KVC_ERR_ALIGN;
  return from_cuda(kvc::launch_qmem_update(M, q_turn, (int64_t)n_sess * L * Hq, D, T, decay,
                                           gain, renorm, stream));
}

size_t kvc_score_qmem_workspace_size(int32_t n_sess, int32_t L, int32_t Hq,
                                     int32_t N) {
  if (n_sess < 1 || L < 1 || Hq < 1 || N < 1) return 0;
  return kvc::score_qmem_ws_bytes(n_sess, L, Hq, N);
}

kvc_status kvc_score_qmem_ex(const float *M, const kvc_bf16 *kpool,
                             const int32_t *slot_map, int32_t sentinel,
                             float *rule, int32_t n_sess, int32_t L, int32_t H,
                             int32_t Hq, int32_t D, int32_t N, int64_t n_slots,
                             void *ws, size_t ws_bytes, int32_t *dev_status,
                             kvc_kernel kernel, cudaStream_t stream) {
  if (!M || !kpool || !slot_map || !rule || !ws) return KVC_ERR_INVALID_ARG;
  if (kernel != KVC_KERNEL_AUTO && kernel != KVC_KERNEL_QMEM_TC && kernel != KVC_KERNEL_QMEM_CC &&
      kernel != KVC_KERNEL_QMEM_TC_SPILL)
    return KVC_ERR_INVALID_ARG;
  if (n_sess < 1 || L < 1 || H < 1 || Hq < 1 || N < 1 || n_slots < 1 || n_slots > INT32_MAX)
    return KVC_ERR_INVALID_ARG;
  if (!head_dim_ok(D) || Hq % H || H > 32 || 32 % H || Hq / H > 8 || n_sess > 65535 ||
      (N + 255) / 256 > 65535 || L > 65535)
    return KVC_ERR_SHAPE;
  if (!aligned16(M) || !aligned16(kpool) || !aligned16(ws)) return KVC_ERR_ALIGN;
  if (ws_bytes < kvc_score_qmem_workspace_size(n_sess, L, Hq, N)) return KVC_ERR_WORKSPACE;
  return from_cuda_kernel(kvc::launch_score_qmem(M, kpool, slot_map, sentinel, rule, n_sess, L,
                                                 H, Hq, D, N, n_slots, ws, dev_status,
                                                 (int)kernel, stream));
}

kvc_status kvc_score_qmem(const float *M, const kvc_bf16 *kpool,
                          const int32_t *slot_map, int32_t sentinel,
                          float *rule, int32_t n_sess, int32_t L, int32_t H,
                          int32_t Hq, int32_t D, int32_t N, int64_t n_slots,
                          void *ws, size_t ws_bytes, int32_t *dev_status,
                          cudaStream_t stream) {
  return kvc_score_qmem_ex(M, kpool, slot_map, sentinel, rule, n_sess, L, H, Hq, D, N, n_slots,
                           ws, ws_bytes, dev_status, KVC_KERNEL_AUTO, stream);
}

kvc_status kvc_select(const float *scores, const int64_t *seg_off,
                      int32_t n_seg, int32_t max_seg_len, int32_t budget,
                      int32_t n_sink, int32_t n_recent, int32_t *kept,
                      int32_t *kept_count, uint32_t *keepmask,
                      int32_t *dev_status, cudaStream_t stream) {
  if (!scores || !seg_off || !kept || !kept_count || n_seg < 1 || max_seg_len < 1)
    return KVC_ERR_INVALID_ARG;
  if (budget < 1 || n_sink < 0 || n_recent < 0 || (int64_t)n_sink + n_recent > budget)
    return KVC_ERR_BUDGET;
  if (max_seg_len > KVC_SELECT_MAX_SEG) return KVC_ERR_SHAPE;
  return from_cuda(kvc::launch_select(scores, seg_off, n_seg, max_seg_len, budget, n_sink,
                                      n_recent, kept, kept_count, keepmask, dev_status, stream));
}

kvc_status kvc_rope_table(float *tab, int32_t n_pos, int32_t pos0, int32_t D,
                          double theta, cudaStream_t stream) {
  if (!tab || n_pos < 1 || pos0 < 0 || !(theta > 1.0) || !isfinite(theta))
    return KVC_ERR_INVALID_ARG;
  if ((int64_t)pos0 + n_pos > INT32_MAX) return KVC_ERR_INVALID_ARG;
  if (!head_dim_ok(D)) return KVC_ERR_SHAPE;
  if (!aligned16(tab)) return KVC_ERR_ALIGN;
  return from_cuda(kvc::launch_rope_table(tab, n_pos, pos0, D, theta, stream));
}

kvc_status kvc_pack_rerope(const kvc_bf16 *kraw, const kvc_bf16 *vraw,
                           const int32_t *kept, const int32_t *kept_count,
                           int32_t L, int32_t H, int32_t D,
                           const int64_t *tok_off, int32_t n_sess,
                           int64_t n_tok, int32_t budget,
                           const float *rope_tab, kvc_bf16 *kview,
                           kvc_bf16 *vview, int32_t *dev_status,
                           cudaStream_t stream) {
  if (!kraw || !vraw || !kept || !kept_count || !tok_off || !rope_tab || !kview || !vview)
    return KVC_ERR_INVALID_ARG;
  if (L < 1 || H < 1 || n_sess < 1 || n_tok < 1) return KVC_ERR_INVALID_ARG;
  if (budget < 1 || budget > 65535) return KVC_ERR_BUDGET;
  if (!head_dim_ok(D) || n_tok % KVC_BLOCK_TOKENS) return KVC_ERR_SHAPE;
  if (!aligned16(kraw) || !aligned16(vraw) || !aligned16(rope_tab) || !aligned16(kview) ||
      !aligned16(vview))
    return KVC_ERR_ALIGN;
  if ((int64_t)L * n_sess > 65535) return KVC_ERR_SHAPE;
  return from_cuda(kvc::launch_pack_rerope(kraw, vraw, kept, kept_count, L, H, D, tok_off,
                                           n_sess, n_tok, budget, rope_tab, kview, vview,
                                           dev_status, stream));
}

namespace {

// Shared checks and launch of kvc_pack_tiered / kvc_pack_tiered_slots.
kvc_status pack_tiered_common(const kvc_bf16 *kraw_host, const kvc_bf16 *vraw_host,
                              const int32_t *host_slot, int64_t slot_elems, int32_t n_slots,
                              const int32_t *kept_prev, const int32_t *kept_count_prev,
                              const kvc_bf16 *kcache_prev, const kvc_bf16 *vview_prev,
                              const int32_t *kept, const int32_t *kept_count, int32_t L,
                              int32_t H, int32_t D, const int64_t *tok_off, int32_t n_sess,
                              int64_t n_tok, int32_t budget, const float *rope_tab,
                              kvc_bf16 *kcache, kvc_bf16 *kview, kvc_bf16 *vview,
                              int32_t *n_hits, int32_t *dev_status, cudaStream_t stream) {
  if (!kraw_host || !vraw_host || !kept || !kept_count || !tok_off || !rope_tab || !kcache ||
      !kview || !vview)
    return KVC_ERR_INVALID_ARG;
  if (kept_prev && (!kept_count_prev || !kcache_prev || !vview_prev)) return KVC_ERR_INVALID_ARG;
  if (L < 1 || H < 1 || n_sess < 1 || n_tok < 1) return KVC_ERR_INVALID_ARG;
  if (budget < 1 || budget > 65535) return KVC_ERR_BUDGET;
  if (!head_dim_ok(D) || n_tok % KVC_BLOCK_TOKENS || (int64_t)L * n_sess > 65535)
    return KVC_ERR_SHAPE;
  if (host_slot && (n_slots < 1 || slot_elems < (int64_t)KVC_BLOCK_TOKENS * D))
    return KVC_ERR_INVALID_ARG;
  if (!aligned16(kraw_host) || !aligned16(vraw_host) || !aligned16(rope_tab) ||
      !aligned16(kcache) || !aligned16(kview) || !aligned16(vview) ||
      (kcache_prev && !aligned16(kcache_prev)) || (vview_prev && !aligned16(vview_prev)) ||
      (host_slot && (slot_elems * 2) % 16))
    return KVC_ERR_ALIGN;
  // the host history must be page-locked and mapped: use its device-side address
  void *kdev = nullptr, *vdev = nullptr;
  if (cudaHostGetDevicePointer(&kdev, const_cast<kvc_bf16 *>(kraw_host), 0) != cudaSuccess ||
      cudaHostGetDevicePointer(&vdev, const_cast<kvc_bf16 *>(vraw_host), 0) != cudaSuccess) {
    cudaGetLastError();  // clear the query's error
    return KVC_ERR_INVALID_ARG;
  }
  return from_cuda(kvc::launch_pack_tiered(
      static_cast<const kvc_bf16 *>(kdev), static_cast<const kvc_bf16 *>(vdev), host_slot,
      slot_elems, n_slots, kept_prev, kept_count_prev, kcache_prev, vview_prev, kept,
      kept_count, L, H, D, tok_off, n_sess, n_tok, budget, rope_tab, kcache, kview, vview,
      n_hits, dev_status, stream));
}

}  // namespace

kvc_status kvc_pack_tiered(const kvc_bf16 *kraw_host, const kvc_bf16 *vraw_host,
                           const int32_t *kept_prev, const int32_t *kept_count_prev,
                           const kvc_bf16 *kcache_prev, const kvc_bf16 *vview_prev,
                           const int32_t *kept, const int32_t *kept_count, int32_t L,
                           int32_t H, int32_t D, const int64_t *tok_off, int32_t n_sess,
                           int64_t n_tok, int32_t budget, const float *rope_tab,
                           kvc_bf16 *kcache, kvc_bf16 *kview, kvc_bf16 *vview, int32_t *n_hits,
                           int32_t *dev_status, cudaStream_t stream) {
  return pack_tiered_common(kraw_host, vraw_host, nullptr, 0, 0, kept_prev, kept_count_prev,
                            kcache_prev, vview_prev, kept, kept_count, L, H, D, tok_off, n_sess,
                            n_tok, budget, rope_tab, kcache, kview, vview, n_hits, dev_status,
                            stream);
}

kvc_status kvc_pack_tiered_slots(const kvc_bf16 *kslots_host, const kvc_bf16 *vslots_host,
                                 int64_t slot_elems, int32_t n_slots, const int32_t *host_slot,
                                 const int32_t *kept_prev, const int32_t *kept_count_prev,
                                 const kvc_bf16 *kcache_prev, const kvc_bf16 *vview_prev,
                                 const int32_t *kept, const int32_t *kept_count, int32_t L,
                                 int32_t H, int32_t D, const int64_t *tok_off, int32_t n_sess,
                                 int64_t n_tok, int32_t budget, const float *rope_tab,
                                 kvc_bf16 *kcache, kvc_bf16 *kview, kvc_bf16 *vview,
                                 int32_t *n_hits, int32_t *dev_status, cudaStream_t stream) {
  if (!host_slot) return KVC_ERR_INVALID_ARG;
  return pack_tiered_common(kslots_host, vslots_host, host_slot, slot_elems, n_slots, kept_prev,
                            kept_count_prev, kcache_prev, vview_prev, kept, kept_count, L, H, D,
                            tok_off, n_sess, n_tok, budget, rope_tab, kcache, kview, vview,
                            n_hits, dev_status, stream);
}

kvc_status kvc_init_sentinel(kvc_bf16 *kpool, kvc_bf16 *vpool, int32_t L,
                             int32_t H, int32_t D, int64_t n_slots,
                             int32_t sentinel, cudaStream_t stream) {
  if (!kpool || L < 1 || H < 1 || n_slots < 1 || sentinel < 0 || sentinel >= n_slots)
    return KVC_ERR_INVALID_ARG;
  if (!head_dim_ok(D)) return KVC_ERR_SHAPE;
  int64_t n = (int64_t)L * H * D;
  k_init_sentinel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(kpool, vpool, L, H, D,
                                                                    n_slots, sentinel);
  return from_cuda(cudaGetLastError());
}

size_t kvc_redirect_free_workspace_size(int32_t n_sess, int32_t N,
                                        int64_t n_slots) {
  if (n_sess < 1 || N < 1 || n_slots < 1) return 0;
  return kvc::redirect_free_ws_bytes(n_sess, N, n_slots);
}

kvc_status kvc_redirect_free(int32_t *slot_map, const uint32_t *keepmask,
                             int32_t n_sess, int32_t N, int32_t *refcnt,
                             int64_t n_slots, int32_t prefix_len,
                             int32_t sentinel, int32_t *freed,
                             int32_t freed_cap, int32_t *n_freed, void *ws,
                             size_t ws_bytes, int32_t *dev_status,
                             cudaStream_t stream) {
  if (!slot_map || !keepmask || !refcnt || !n_freed || !ws || (!freed && freed_cap > 0))
    return KVC_ERR_INVALID_ARG;
  if (n_sess < 1 || N < 1 || n_slots < 1 || n_slots > INT32_MAX || freed_cap < 0 ||
      prefix_len < 0 || (int64_t)n_sess * N > INT32_MAX)
    return KVC_ERR_INVALID_ARG;
  if (!aligned16(ws)) return KVC_ERR_ALIGN;
  if (ws_bytes < kvc_redirect_free_workspace_size(n_sess, N, n_slots)) return KVC_ERR_WORKSPACE;
  return from_cuda(kvc::launch_redirect_free(slot_map, keepmask, n_sess, N, refcnt, n_slots,
                                             prefix_len, sentinel, freed, freed_cap, n_freed,
                                             ws, dev_status, stream));
}

size_t kvc_recover_score_workspace_size(int32_t n_req, int32_t max_blocks, int32_t L, int32_t H,
                                        int32_t Hq, int32_t D, int32_t block_size) {
  if (n_req < 1 || max_blocks < 1 || L < 1 || H < 1 || Hq < H || Hq % H || block_size < 1)
    return 0;
  return kvc::recover_ws_bytes(n_req, max_blocks, block_size, L, H, Hq, D);
}

kvc_status kvc_recover_score_ex(const kvc_bf16 *q, const float *lse, const kvc_bf16 *kpool,
                                int64_t n_slots, const int32_t *block_table, int32_t max_blocks,
                                const int32_t *seqused_k, const int32_t *count, int32_t n_req,
                                int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t block_size,
                                float *state, void *ws, size_t ws_bytes, int32_t *dev_status,
                                kvc_kernel kernel, cudaStream_t stream) {
  if (!q || !lse || !kpool || !block_table || !seqused_k || !count || !state)
    return KVC_ERR_INVALID_ARG;
  if (kernel != KVC_KERNEL_AUTO && kernel != KVC_KERNEL_RECOVER_TC &&
      kernel != KVC_KERNEL_RECOVER_CC)
    return KVC_ERR_INVALID_ARG;
  if (n_req < 1 || L < 1 || H < 1 || Hq < 1 || block_size < 1 || max_blocks < 1 ||
      n_slots < block_size)
    return KVC_ERR_INVALID_ARG;
  if (!head_dim_ok(D) || Hq % H || Hq > 256 || block_size > 64 || H > 256 ||
      (int64_t)block_size * H > 4096 || (int64_t)max_blocks * block_size > INT32_MAX ||
      (int64_t)n_req * max_blocks > INT32_MAX || (int64_t)n_req * L * Hq > INT32_MAX)
    return KVC_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(kpool) || !aligned16(lse) || !aligned16(state) ||
      (ws && !aligned16(ws)))
    return KVC_ERR_ALIGN;
  return from_cuda_kernel(kvc::launch_recover_score(
      q, lse, kpool, n_slots, block_table, max_blocks, seqused_k, count, n_req, L, H, Hq, D,
      block_size, state, ws, ws ? ws_bytes : 0, dev_status, (int)kernel, stream));
}

kvc_status kvc_recover_score(const kvc_bf16 *q, const float *lse, const kvc_bf16 *kpool,
                             int64_t n_slots, const int32_t *block_table, int32_t max_blocks,
                             const int32_t *seqused_k, const int32_t *count, int32_t n_req,
                             int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t block_size,
                             float *state, void *ws, size_t ws_bytes, int32_t *dev_status,
                             cudaStream_t stream) {
  return kvc_recover_score_ex(q, lse, kpool, n_slots, block_table, max_blocks, seqused_k, count,
                              n_req, L, H, Hq, D, block_size, state, ws, ws_bytes, dev_status,
                              KVC_KERNEL_AUTO, stream);
}

kvc_status kvc_lrfu_update(const float *scores, const int64_t *seg_off, int32_t n_seg,
                           int32_t max_seg_len, float top_p, float lambda, float *keep_score,
                           uint32_t *hitmask, int32_t *dev_status, cudaStream_t stream) {
  if (!scores || !seg_off || !keep_score || n_seg < 1 || max_seg_len < 1)
    return KVC_ERR_INVALID_ARG;
  if (!(top_p >= 0.f && top_p <= 1.f) || !(lambda >= 0.f && lambda <= 1.f))
    return KVC_ERR_INVALID_ARG;
  if (max_seg_len > KVC_LRFU_MAX_SEG) return KVC_ERR_SHAPE;
  return from_cuda(kvc::launch_lrfu(scores, seg_off, n_seg, max_seg_len, top_p, lambda,
                                    keep_score, hitmask, dev_status, stream));
}

kvc_status kvc_token_confidence(const float *logits, int32_t n_tok, int32_t V, int32_t top_k,
                                float *conf, int32_t *dev_status, cudaStream_t stream) {
  if (!logits || !conf || n_tok < 1 || V < 1 || top_k < 1 || top_k > V)
    return KVC_ERR_INVALID_ARG;
  if (n_tok > INT32_MAX / 2) return KVC_ERR_SHAPE;
  return from_cuda(kvc::launch_token_confidence(logits, n_tok, V, top_k, conf, dev_status,
                                                stream));
}

kvc_status kvc_conf_trend_budget(const float *conf, const int64_t *trace_off, int32_t n_trace,
                                 int32_t max_trace_len, int32_t window, int32_t stride,
                                 float bottom_pct, int32_t budget_step, int32_t max_budget,
                                 double *slope, int32_t *budget, int32_t *n_kept,
                                 int32_t *dev_status, cudaStream_t stream) {
  if (!conf || !trace_off || !slope || !budget || !n_kept || n_trace < 1 || max_trace_len < 1 ||
      window < 1 || stride < 1 || budget_step < 0 || max_budget < 1)
    return KVC_ERR_INVALID_ARG;
  if (!(bottom_pct >= 0.f && bottom_pct <= 100.f)) return KVC_ERR_INVALID_ARG;
  if (max_trace_len >= window &&
      (max_trace_len - window) / stride + 1 > kvc::conf_trend_max_windows())
    return KVC_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(slope) & 7u) return KVC_ERR_ALIGN;
  return from_cuda(kvc::launch_conf_trend(conf, trace_off, n_trace, max_trace_len, window,
                                          stride, bottom_pct, budget_step, max_budget, slope,
                                          budget, n_kept, dev_status, stream));
}

int32_t kvc_recover_tensor_core(int32_t H, int32_t Hq, int32_t D, int32_t block_size) {
  return kvc::recover_tc_supported(H, Hq, D, block_size) ? 1 : 0;
}

kvc_status kvc_tail_plan(const uint32_t *keepmask, int32_t mask_words,
                         const int32_t *seqused_k, const int32_t *block_table,
                         int32_t max_blocks, int32_t n_req, int32_t block_size, int64_t n_slots,
                         int32_t *src_slot, int32_t *dst_slot, int32_t *n_pairs,
                         int32_t *n_tail_blocks, int32_t *freed_blocks, int32_t *n_freed,
                         int32_t *new_table, uint32_t *tail_mask, int32_t *dev_status,
                         cudaStream_t stream) {
  if (!keepmask || !seqused_k || !block_table || !src_slot || !dst_slot || !n_pairs ||
      !n_tail_blocks || !freed_blocks || !n_freed || !new_table || !tail_mask)
    return KVC_ERR_INVALID_ARG;
  if (n_req < 1 || mask_words < 1 || max_blocks < 1 || block_size < 1 || n_slots < 1 ||
      n_slots > INT32_MAX)
    return KVC_ERR_INVALID_ARG;
  if ((int64_t)max_blocks * block_size > KVC_TAIL_MAX_TOKENS) return KVC_ERR_SHAPE;
  return from_cuda(kvc::launch_tail_plan(keepmask, mask_words, seqused_k, block_table,
                                         max_blocks, n_req, block_size, n_slots, src_slot,
                                         dst_slot, n_pairs, n_tail_blocks, freed_blocks, n_freed,
                                         new_table, tail_mask, dev_status, stream));
}

kvc_status kvc_tail_compact(kvc_bf16 *kpool, kvc_bf16 *vpool, int64_t n_slots, int32_t L,
                            int32_t H, int32_t D, const int32_t *src_slot,
                            const int32_t *dst_slot, const int32_t *n_pairs, int32_t pair_cap,
                            int32_t n_req, int32_t *dev_status, cudaStream_t stream) {
  if (!kpool || !vpool || !src_slot || !dst_slot || !n_pairs) return KVC_ERR_INVALID_ARG;
  if (n_slots < 1 || L < 1 || H < 1 || pair_cap < 1 || n_req < 1) return KVC_ERR_INVALID_ARG;
  if (!head_dim_ok(D) || n_req > 65535) return KVC_ERR_SHAPE;
  if (!aligned16(kpool) || !aligned16(vpool)) return KVC_ERR_ALIGN;
  return from_cuda(kvc::launch_tail_compact(kpool, vpool, n_slots, L, H, D, src_slot, dst_slot,
                                            n_pairs, pair_cap, n_req, dev_status, stream));
}

}  // extern "C"
