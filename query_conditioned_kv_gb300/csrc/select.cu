// select.cu — budgeted top-k with a forced set, chronological output and
// keep mask; one CTA per segment.
//
// IntentKV §4 "Top-k selection": K* = F ∪ argtop_{C*} s, the C* highest
// scores among the non-forced items plus the forced set; KVMem "Query-
// conditioned retrieval": sink and recent blocks are always kept and the
// survivors are restored in chronological order; ActKV §3.3: the eviction
// output is a Boolean keep mask.  Ties rank by index (lower first).
//
// Per segment of n items (n > budget):
//   1. the scores are mapped to order-preserving uint32 keys (−0.0 folded
//      onto +0.0, NaN below −inf) and staged in shared memory;
//   2. a 4-pass, 8-bit MSB radix select over the non-forced keys finds the
//      k-th largest key T and how many items equal to T are still needed;
//   3. one ordered sweep (tiles of blockDim items, two block-wide scans
//      per tile) keeps forced ∪ {key > T} ∪ {the first `need`
//      items with key == T}, writes their indices ascending and the mask
//      words (one warp ballot per 32 items).
// No global scratch; the output is exact and deterministic.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kSelThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float s, bool &nan) {
  if (s != s) {
    nan = true;
    return 0u;
  }
  if (s == 0.f) s = 0.f;  // −0.0 ranks with +0.0
  uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block scan of v (all threads); *total gets the block sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *total,
                                                    uint32_t *warp_tot) {
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int n_warps = blockDim.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < n_warps ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  uint32_t excl = x - v + (warp > 0 ? warp_tot[warp - 1] : 0u);
  *total = warp_tot[n_warps - 1];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(kSelThreads)
k_select(const float *__restrict__ scores, const int64_t *__restrict__ seg_off,
         int max_seg_len, int budget, int n_sink, int n_recent,
         int32_t *__restrict__ kept, int32_t *__restrict__ kept_count,
         uint32_t *__restrict__ keepmask, int words, int32_t *status) {
  extern __shared__ uint32_t keys[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t s_digit, s_need;
  __shared__ int s_nan;

  const int seg = blockIdx.x;
  const int tid = threadIdx.x;
  int32_t *kept_row = kept + (int64_t)seg * budget;
  uint32_t *mask_row = keepmask ? keepmask + (int64_t)seg * words : nullptr;

  int64_t off = seg_off[seg], end = seg_off[seg + 1];
  bool bad = end < off || end - off > max_seg_len || off < 0;
  int n = bad ? 0 : (int)(end - off);
  if (bad && tid == 0) record_error(status, KVC_ERR_BOUNDS);

  if (n <= budget) {  // keep everything (or nothing, on a bad segment)
    for (int i = tid; i < budget; i += blockDim.x) kept_row[i] = i < n ? i : -1;
    if (mask_row)
      for (int w = tid; w < words; w += blockDim.x) {
        int lo = w * 32;
        uint32_t m = lo >= n ? 0u : (n - lo >= 32 ? 0xFFFFFFFFu : ((1u << (n - lo)) - 1u));
        mask_row[w] = m;
      }
    if (tid == 0) kept_count[seg] = n;
    return;
  }

  // n > budget ≥ n_sink + n_recent: the sink and recent ranges are disjoint.
  const int rec0 = n - n_recent;
  const int k = budget - n_sink - n_recent;
  if (tid == 0) s_nan = 0;
  __syncthreads();
  bool nan = false;
  for (int i = tid; i < n; i += blockDim.x) keys[i] = order_key(scores[off + i], nan);
  if (nan) s_nan = 1;

  // Radix select: the k-th largest non-forced key.
  uint32_t prefix = 0, hi_mask = 0, need = (uint32_t)k;
  if (k > 0) {
    for (int pass = 0; pass < 4; pass++) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      // warp-aggregated: lanes with the same digit add once (scores of one
      // segment share their leading bits, so plain atomics would serialise)
      for (int base = 0; base < n; base += blockDim.x) {
        const int i = base + tid;
        bool cand = false;
        uint32_t digit = 0;
        if (i < n && i >= n_sink && i < rec0) {
          uint32_t key = keys[i];
          cand = (key & hi_mask) == prefix;
          digit = (key >> shift) & 255u;
        }
        const uint32_t active = __ballot_sync(0xFFFFFFFFu, cand);
        if (cand) {
          const uint32_t peers = __match_any_sync(active, digit);
          if ((int)(__ffs(peers) - 1) == (tid & 31)) atomicAdd(&hist[digit], __popc(peers));
        }
      }
      __syncthreads();
      if (tid < 32) {
        // lane owns bins 255-8·lane … 248-8·lane (descending)
        uint32_t loc = 0;
#pragma unroll
        for (int e = 0; e < 8; e++) loc += hist[255 - 8 * tid - e];
        uint32_t inc = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          uint32_t y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
          if (tid >= o) inc += y;
        }
        uint32_t run = inc - loc;  // count of keys in higher bins
#pragma unroll
        for (int e = 0; e < 8; e++) {
          int bin = 255 - 8 * tid - e;
          uint32_t hcount = hist[bin];
          if (run < need && run + hcount >= need) {
            s_digit = (uint32_t)bin;
            s_need = need - run;
          }
          run += hcount;
        }
      }
      __syncthreads();
      prefix |= s_digit << shift;
      hi_mask |= 0xFFu << shift;
      need = s_need;
      __syncthreads();
    }
  }
  const uint32_t T = prefix;  // threshold key (valid when k > 0)

  // Ordered sweep: forced ∪ {key > T} ∪ first `need` of {key == T}.
  uint32_t eq_before = 0, out_pos = 0;
  const int lane = tid & 31, warp = tid >> 5;
  for (int base = 0; base < n; base += blockDim.x) {
    int i = base + tid;
    bool valid = i < n;
    bool forced = valid && (i < n_sink || i >= rec0);
    uint32_t key = valid ? keys[i] : 0u;
    bool is_eq = valid && !forced && k > 0 && key == T;
    bool above = valid && !forced && k > 0 && key > T;
    uint32_t tot;
    uint32_t rank_eq = eq_before + block_excl_scan(is_eq ? 1u : 0u, &tot, warp_tot);
    bool keep = forced || above || (is_eq && rank_eq < need);
    uint32_t tot2;
    uint32_t pos = out_pos + block_excl_scan(keep ? 1u : 0u, &tot2, warp_tot);
    if (keep && pos < (uint32_t)budget) kept_row[pos] = i;
    uint32_t ballot = __ballot_sync(0xFFFFFFFFu, keep);
    if (mask_row && lane == 0) {
      int w = (base >> 5) + warp;
      if (w < words) mask_row[w] = ballot;
    }
    eq_before += tot;
    out_pos += tot2;
  }
  // mask words past the last tile
  if (mask_row) {
    int first = (n + blockDim.x - 1) / blockDim.x * (blockDim.x / 32);
    for (int w = first + tid; w < words; w += blockDim.x) mask_row[w] = 0u;
  }
  for (int i = (int)out_pos + tid; i < budget; i += blockDim.x) kept_row[i] = -1;
  if (tid == 0) {
    kept_count[seg] = (int32_t)out_pos;
    if (s_nan) record_error(status, KVC_ERR_NAN);
  }
}

}  // namespace

cudaError_t launch_select(const float *scores, const int64_t *seg_off,
                          int n_seg, int max_seg_len, int budget, int n_sink,
                          int n_recent, int32_t *kept, int32_t *kept_count,
                          uint32_t *keepmask, int32_t *status,
                          cudaStream_t s) {
  int words = (max_seg_len + 31) / 32;
  size_t smem = (size_t)max_seg_len * sizeof(uint32_t);
  int threads = max_seg_len >= 4 * kSelThreads ? kSelThreads
                : max_seg_len >= 1024          ? 512
                                               : 256;
  cudaError_t e = cudaFuncSetAttribute(
      k_select, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_select<<<n_seg, threads, smem, s>>>(scores, seg_off, max_seg_len, budget,
                                        n_sink, n_recent, kept, kept_count,
                                        keepmask, words, status);
  return cudaGetLastError();
}

}  // namespace kvc
