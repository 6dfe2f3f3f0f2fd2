// kvc_internal.cuh — shared device helpers and the internal launch API of
// libkvc (sm_103a).  Nothing here is part of the public C ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

constexpr int kBlock = KVC_BLOCK_TOKENS;

// First device-side error wins; a NULL status word disables the record.
__device__ __forceinline__ void record_error(int32_t *status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) {
  return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t w) {
  return __uint_as_float(w & 0xFFFF0000u);
}
// Two fp32 → packed bf16x2 (round to nearest even); `a` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Streaming 16-byte global accesses (data touched once per event).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream(void *p, uint4 v) {
  __stcs(reinterpret_cast<uint4 *>(p), v);
}

// SM count of the current device (cached per device; 1 if the query fails).
inline int device_sm_count() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  int *n = (dev >= 0 && dev < 64) ? &cache[dev] : nullptr;
  if (n && *n) return *n;
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
    v = 1;
  if (n) *n = v;
  return v;
}

// kvc_score's host-side argument, shape and alignment checks (everything
// but the workspace), shared by the entry points that score (kvc_abi.cu).
kvc_status score_args_status(const void *q, const void *meank, const void *scores,
                             const int64_t *blk_off, int L, int H, int Hq, int D, int W,
                             int n_sess, int64_t nb_total, int nb_max);

// ------------------------------------------------------------ launches
// Each returns cudaGetLastError() of its launch(es).

cudaError_t launch_build_meank(const uint16_t *kraw, uint16_t *meank,
                               int64_t rows, int64_t n_tok, int D,
                               cudaStream_t s);

// `path`: a kvc_kernel value (KVC_KERNEL_AUTO or one KVC_KERNEL_SCORE_*);
// cudaErrorNotSupported when the named kernel cannot run these sizes.
cudaError_t launch_score_meank(const uint16_t *q, const uint16_t *meank,
                               float *scores, int L, int H, int Hq, int D,
                               int W, const int64_t *blk_off, int n_sess,
                               int64_t nb_total, int nb_max, void *ws,
                               int32_t *status, int path, cudaStream_t s);
size_t score_meank_ws_bytes(int L, int H, int Hq, int W, int n_sess,
                            int nb_max, int64_t nb_total);

// tcgen05 scorer (score_tc.cu); cudaErrorNotSupported if the shape is not
// covered (the caller then uses the CUDA-core scorer).
bool score_tc_supported(int R, int W, int D);
int score_tc_launches(int R, int W, int D, int n_sess, int nb_max);  // 1 persistent, 2 split
int score_meank_launches(int H, int Hq, int D, int W, int n_sess, int nb_max);
size_t score_tc_ws_bytes(int L, int H, int Hq, int W, int n_sess, int nb_max, int64_t nb_total);
cudaError_t launch_score_tc(const uint16_t *q, const uint16_t *meank, float *scores, int L,
                            int H, int Hq, int D, int W, const int64_t *blk_off, int n_sess,
                            int64_t nb_total, int nb_max, void *ws, int32_t *status,
                            int path, cudaStream_t s);

// single-read tcgen05 scorer for 4 query heads per KV head, W = 32, D = 128
// (score_fused.cu); cudaErrorNotSupported outside that shape.
bool score_fused_supported(int G, int D, int W, int nb_max);
cudaError_t launch_score_fused(const uint16_t *q, const uint16_t *meank, float *scores, int L,
                               int H, int Hq, int D, int W, const int64_t *blk_off, int n_sess,
                               int64_t nb_total, int nb_max, int32_t *status, cudaStream_t s);

// grouped two-pass tcgen05 scorer for 129–192 query rows per KV head, D = 128
// (score_group.cu); cudaErrorNotSupported outside that shape.
bool score_group_supported(int G, int D, int W, int nb_max);
size_t score_group_ws_bytes();
cudaError_t launch_score_group(const uint16_t *q, const uint16_t *meank, float *scores, int L,
                               int H, int Hq, int D, int W, const int64_t *blk_off, int n_sess,
                               int64_t nb_total, int nb_max, void *ws, int32_t *status,
                               cudaStream_t s);

cudaError_t launch_qmem_update(float *M, const uint16_t *q, int64_t rows,
                               int D, int T, float decay, float gain,
                               int renorm, cudaStream_t s);

// `path`: KVC_KERNEL_AUTO, KVC_KERNEL_QMEM_TC, KVC_KERNEL_QMEM_TC_SPILL or
// KVC_KERNEL_QMEM_CC.
cudaError_t launch_score_qmem(const float *M, const uint16_t *kpool,
                              const int32_t *slot_map, int32_t sentinel,
                              float *rule, int n_sess, int L, int H, int Hq,
                              int D, int N, int64_t n_slots, void *ws,
                              int32_t *status, int path, cudaStream_t s);
size_t score_qmem_ws_bytes(int n_sess, int L, int Hq, int N);
// tensor-core logits of the rule score (qmem_tc.cu)
bool qmem_tc_supported(int H, int Hq, int D, int64_t L, int64_t n_slots);
size_t qmem_tc_mb_bytes(int n_sess, int L, int Hq);
// fused: the rule phase runs inside the logits kernel from L2 (writes
// rule_l, [n_sess][L][N]); otherwise the logits and tile partials are
// spilled for k_qmem_lse / k_qmem_rule.  cudaErrorNotSupported for a fused
// launch with groups of 8 query heads or one that cannot make every CTA
// resident.
cudaError_t launch_qmem_logits_tc(const float *M, const uint16_t *kpool, const int32_t *slot_map,
                                  int32_t sentinel, float *logits, float2 *part, float *lse,
                                  int *counter, float *rule_l, uint16_t *mb, int n_sess, int L,
                                  int H, int Hq, int D, int N, int64_t n_slots, int n_tiles,
                                  bool fused, int32_t *status, cudaStream_t s);

cudaError_t launch_select(const float *scores, const int64_t *seg_off,
                          int n_seg, int max_seg_len, int budget, int n_sink,
                          int n_recent, int32_t *kept, int32_t *kept_count,
                          uint32_t *keepmask, int32_t *status,
                          cudaStream_t s);

cudaError_t launch_rope_table(float *tab, int n_pos, int pos0, int D,
                              double theta, cudaStream_t s);

cudaError_t launch_pack_rerope(const uint16_t *kraw, const uint16_t *vraw,
                               const int32_t *kept, const int32_t *kept_count,
                               int L, int H, int D, const int64_t *tok_off,
                               int n_sess, int64_t n_tok, int budget,
                               const float *rope_tab, uint16_t *kview,
                               uint16_t *vview, int32_t *status,
                               cudaStream_t s);

// host_slot: NULL (the history is [L][H][n_tok][D] in host memory) or the
// slot of each block in host slot arenas (slot_elems apart, n_slots slots).
cudaError_t launch_pack_tiered(const uint16_t *kraw_host, const uint16_t *vraw_host,
                               const int32_t *host_slot, int64_t slot_elems, int32_t n_slots,
                               const int32_t *kept_prev, const int32_t *kept_count_prev,
                               const uint16_t *kcache_prev, const uint16_t *vview_prev,
                               const int32_t *kept, const int32_t *kept_count, int L, int H,
                               int D, const int64_t *tok_off, int n_sess, int64_t n_tok,
                               int budget, const float *rope_tab, uint16_t *kcache,
                               uint16_t *kview, uint16_t *vview, int32_t *n_hits,
                               int32_t *status, cudaStream_t s);

cudaError_t launch_init_sentinel(uint16_t *kpool, uint16_t *vpool, int L,
                                 int H, int D, int64_t n_slots,
                                 int32_t sentinel, cudaStream_t s);

cudaError_t launch_redirect_free(int32_t *slot_map, const uint32_t *keepmask,
                                 int n_sess, int N, int32_t *refcnt,
                                 int64_t n_slots, int prefix_len,
                                 int32_t sentinel, int32_t *freed,
                                 int freed_cap, int32_t *n_freed, void *ws,
                                 int32_t *status, cudaStream_t s);
size_t redirect_free_ws_bytes(int n_sess, int N, int64_t n_slots);

// ActKV LRFU keep score (lrfu.cu)
cudaError_t launch_lrfu(const float *scores, const int64_t *seg_off, int n_seg, int max_seg_len,
                        float p, float lambda, float *ks, uint32_t *hitmask, int32_t *status,
                        cudaStream_t s);

// ActKV confidence monitor (confidence.cu)
cudaError_t launch_token_confidence(const float *logits, int n_tok, int V, int k, float *conf,
                                    int32_t *status, cudaStream_t s);
cudaError_t launch_conf_trend(const float *conf, const int64_t *trace_off, int n_trace,
                              int max_len, int w, int stride, float b, int step, int max_budget,
                              double *slope, int32_t *budget, int32_t *n_kept, int32_t *status,
                              cudaStream_t s);
int conf_trend_max_windows();

// ActKV paged primitives (recover.cu)
bool recover_tc_supported(int H, int Hq, int D, int BS);
size_t recover_ws_bytes(int n_req, int max_blocks, int BS, int L, int H, int Hq, int D);
// `path`: KVC_KERNEL_AUTO, KVC_KERNEL_RECOVER_TC or KVC_KERNEL_RECOVER_CC.
cudaError_t launch_recover_score(const uint16_t *q, const float *lse, const uint16_t *kpool,
                                 int64_t n_slots, const int32_t *block_table, int max_blocks,
                                 const int32_t *seqused, const int32_t *count, int n_req, int L,
                                 int H, int Hq, int D, int BS, float *state, void *ws,
                                 size_t ws_bytes, int32_t *status, int path, cudaStream_t s);
cudaError_t launch_tail_plan(const uint32_t *keepmask, int mask_words, const int32_t *seqused,
                             const int32_t *block_table, int max_blocks, int n_req, int BS,
                             int64_t n_slots, int32_t *src, int32_t *dst, int32_t *n_pairs,
                             int32_t *n_tail, int32_t *freed, int32_t *n_freed,
                             int32_t *new_table, uint32_t *tail_mask, int32_t *status,
                             cudaStream_t s);
cudaError_t launch_tail_compact(uint16_t *kpool, uint16_t *vpool, int64_t n_slots, int L, int H,
                                int D, const int32_t *src, const int32_t *dst,
                                const int32_t *n_pairs, int cap, int n_req, int32_t *status,
                                cudaStream_t s);

}  // namespace kvc
