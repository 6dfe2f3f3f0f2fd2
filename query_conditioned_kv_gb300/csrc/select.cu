// select.cu — budgeted top-k with a forced set, chronological output and
// keep mask; one CTA per segment.
//
// IntentKV §4 "Top-k selection": K* = F ∪ argtop_{C*} s, the C* highest
// scores among the non-forced items plus the forced set; KVMem "Query-
// conditioned retrieval": sink and recent blocks are always kept and the
// survivors are restored in chronological order; ActKV §3.3: the eviction
// output is a Boolean keep mask.  Ties rank by index (lower first).
//
// Per segment of n items (n > budget), thread t owning the contiguous
// items [t·ipt, (t+1)·ipt), ipt = ⌈n / threads⌉:
//   1. the scores are mapped to order-preserving uint32 keys (−0.0 folded
//      onto +0.0, NaN below −inf) and staged in shared memory;
//   2. the k-th largest non-forced key T is the largest T with
//      #(key ≥ T) ≥ k: it is found eight bits at a time (MSB radix levels),
//      from the highest bit where the candidates differ.  A level counts the
//      next digit of the keys that still match the decided bits into shared
//      histograms (after the first level few keys match) and takes the
//      largest digit whose count from the top reaches the number still
//      needed.  The count left at the end is the number of items equal to T
//      still needed, k − #(key > T);
//   3. an ordered sweep in two block scans (equal-to-T counts, then keep
//      counts, from per-thread bit masks) keeps forced ∪ {key > T} ∪ {the
//      first `need` items with key == T} and writes their indices
//      ascending; the keep mask is built in shared memory and written out
//      word by word.
// No global scratch; the output is exact and deterministic.
//
// Segments longer than shared memory can stage (KVC_SELECT_STAGED_SEG items)
// take k_select_stream: the same three steps with every pass reading the
// scores from global memory (the segment stays in L2 between passes), and the
// ordered sweep run in rounds of 64 items per thread with the scans' totals
// carried from round to round.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kSelThreads = 1024;
// Items per thread the launch aims for (at most 64: the sweep's bit masks).
// Fewer threads per segment mean cheaper barriers in the threshold search.
constexpr int kSelIPT = 8;
// Histogram copies of the radix levels (warp w counts into copy w mod 8), so
// conflicting atomics come from at most a few warps.
constexpr int kSelHist = 8;

// Keys are stored with one pad word per 32: a thread's contiguous chunk and
// the strided sweeps both read distinct banks.
__device__ __forceinline__ int kp(int i) { return i + (i >> 5); }

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

// Warp 0: from the radix level's histograms (kSelHist copies of 256 bins),
// the largest digit d whose count from the top reaches `need`; writes the
// extended prefix and the count still needed among the keys equal to it.
__device__ __forceinline__ void pick_digit(const uint32_t *hist, int lane, uint32_t prefix,
                                           uint32_t need, int lo, uint32_t *s_prefix,
                                           uint32_t *s_need) {
  // lane l: bins 8l … 8l+7 summed over the histogram copies
  uint32_t loc[8], lsum = 0;
#pragma unroll
  for (int b = 0; b < 8; b++) {
    uint32_t v = 0;
    for (int c = 0; c < kSelHist; c++) v += hist[c * 256 + 8 * lane + b];
    loc[b] = v;
    lsum += v;
  }
  uint32_t sfx = lsum;  // Σ of the bins ≥ 8·lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, sfx, o);
    if (lane + o < 32) sfx += y;
  }
  const uint32_t above = sfx - lsum;  // Σ of the bins ≥ 8·(lane + 1)
  if (above < need && sfx >= need) {  // exactly one lane
    uint32_t acc = above;
    int d = 8 * lane;
#pragma unroll
    for (int b = 7; b >= 0; b--)
      if (acc + loc[b] >= need) {
        d = 8 * lane + b;
        break;
      } else {
        acc += loc[b];
      }
    *s_prefix = prefix | ((uint32_t)d << lo);
    *s_need = need - acc;
  }
}

__global__ void __launch_bounds__(kSelThreads)
k_select(const float *__restrict__ scores, const int64_t *__restrict__ seg_off,
         int max_seg_len, int budget, int n_sink, int n_recent,
         int32_t *__restrict__ kept, int32_t *__restrict__ kept_count,
         uint32_t *__restrict__ keepmask, int words, int32_t *status) {
  extern __shared__ uint32_t dyn[];
  uint32_t *keys = dyn;                               // [kp(max_seg_len)]
  uint32_t *mask_s = dyn + kp(max_seg_len) + 1;       // [words]
  uint32_t *hist = mask_s + words;                    // [kSelHist][256]
  __shared__ uint32_t s_red[3][32];
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t s_kmax, s_kmin, s_prefix, s_need;
  __shared__ int s_nan;

  const int seg = blockIdx.x;
  const int tid = threadIdx.x, nt = blockDim.x;
  int32_t *kept_row = kept + (int64_t)seg * budget;
  uint32_t *mask_row = keepmask ? keepmask + (int64_t)seg * words : nullptr;

  int64_t off = seg_off[seg], end = seg_off[seg + 1];
  bool bad = end < off || end - off > max_seg_len || off < 0;
  int n = bad ? 0 : (int)(end - off);
  if (bad && tid == 0) record_error(status, KVC_ERR_BOUNDS);

  if (n <= budget) {  // keep everything (or nothing, on a bad segment)
    for (int i = tid; i < budget; i += nt) kept_row[i] = i < n ? i : -1;
    if (mask_row)
      for (int w = tid; w < words; w += nt) {
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
  for (int i = tid; i < n; i += nt) keys[kp(i)] = order_key(scores[off + i], nan);
  if (nan) s_nan = 1;
  for (int w = tid; w < words; w += nt) mask_s[w] = 0u;

  // T = the k-th largest non-forced key: the largest T with #(key ≥ T) ≥ k,
  // found eight bits at a time from the most significant bit where the
  // candidates differ (the bits above it are common to all of them).
  uint32_t prefix = 0, need = (uint32_t)k;
  const int lane = tid & 31, warp = tid >> 5, n_warps = nt >> 5;
  if (k > 0) {
    uint32_t lmax = 0u, lmin = 0xFFFFFFFFu;
    for (int i = n_sink + tid; i < rec0; i += nt) {
      const uint32_t key = keys[kp(i)];
      lmax = max(lmax, key);
      lmin = min(lmin, key);
    }
    lmax = __reduce_max_sync(0xFFFFFFFFu, lmax);
    lmin = __reduce_min_sync(0xFFFFFFFFu, lmin);
    if (lane == 0) {
      s_red[0][warp] = lmax;
      s_red[1][warp] = lmin;
    }
    __syncthreads();
    if (warp == 0) {
      const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, lane < n_warps ? s_red[0][lane] : 0u);
      const uint32_t mn =
          __reduce_min_sync(0xFFFFFFFFu, lane < n_warps ? s_red[1][lane] : 0xFFFFFFFFu);
      if (lane == 0) {
        s_kmax = mx;
        s_kmin = mn;
      }
    }
    __syncthreads();
    const uint32_t kmax = s_kmax, kmin = s_kmin;
    int hi = kmax == kmin ? -1 : 31 - __clz(kmax ^ kmin);  // highest undecided bit
    prefix = hi < 0 ? kmax : hi == 31 ? 0u : (kmax >> (hi + 1)) << (hi + 1);
    // Eight bits per level: a histogram of the next digit over the keys that
    // still match the decided bits (after the first level, few do), then the
    // largest digit whose count from the top reaches `need`.
    while (hi >= 0) {
      const int lo = hi >= 7 ? hi - 7 : 0;
      const uint32_t dmask = (2u << (hi - lo)) - 1u;
      const uint32_t pmask = hi == 31 ? 0u : ~((2u << hi) - 1u);
      uint32_t *h = hist + (warp % kSelHist) * 256;
      for (int j = tid; j < kSelHist * 256; j += nt) hist[j] = 0u;
      __syncthreads();
      for (int i = n_sink + tid; i < rec0; i += nt) {
        const uint32_t key = keys[kp(i)];
        if ((key & pmask) == prefix) atomicAdd(&h[(key >> lo) & dmask], 1u);
      }
      __syncthreads();
      if (warp == 0) pick_digit(hist, lane, prefix, need, lo, &s_prefix, &s_need);
      __syncthreads();
      prefix = s_prefix;
      need = s_need;
      hi = lo - 1;
    }
  }
  const uint32_t T = prefix;  // threshold key (valid when k > 0)

  // Ordered sweep over this thread's contiguous items (ipt ≤ 64, bit e of a
  // mask = item i0 + e): forced ∪ {key > T} ∪ the first `need` of
  // {key == T} in index order.  Ranks come from popcounts of the masks, so
  // the items can be read in any order.
  const int ipt = (n + nt - 1) / nt;
  const int i0 = min(n, tid * ipt), cnt = min(n, i0 + ipt) - i0;
  uint64_t eqm = 0, km = 0;
  for (int e = 0; e < cnt; e++) {
    const int i = i0 + e;
    bool keep = i < n_sink || i >= rec0, eq = false;
    if (!keep && k > 0) {
      const uint32_t key = keys[kp(i)];
      keep = key > T;
      eq = key == T;
    }
    km |= (uint64_t)keep << e;
    eqm |= (uint64_t)eq << e;
  }
  uint32_t tot_eq;
  const uint32_t eq_before = block_excl_scan((uint32_t)__popcll(eqm), &tot_eq, warp_tot);
  // equal items in rank order: keep while the running rank is below `need`
  if (eq_before < need) {
    const uint32_t take = min((uint32_t)__popcll(eqm), need - eq_before);
    uint64_t m = eqm;
    for (uint32_t t = 0; t < take; t++) {
      km |= m & (~m + 1);  // lowest remaining equal item
      m &= m - 1;
    }
  }
  uint32_t tot_keep;
  const uint32_t pos0 = block_excl_scan((uint32_t)__popcll(km), &tot_keep, warp_tot);
  {
    uint64_t m = km;
    uint32_t pos = pos0;
    while (m) {
      const int e = __ffsll((long long)m) - 1;
      m &= m - 1;
      if (pos < (uint32_t)budget) kept_row[pos] = i0 + e;
      pos++;
    }
    // this chunk's keep bits into the mask words it overlaps
    if (cnt > 0)
      for (int w = i0 >> 5; w <= (i0 + cnt - 1) >> 5; w++) {
        const int lo = w * 32 - i0;  // bit of item w·32 in km (may be < 0)
        const uint64_t part = lo >= 0 ? (km >> lo) : (km << -lo);
        const uint32_t bits = (uint32_t)part;
        if (bits) atomicOr(&mask_s[w], bits);
      }
  }
  __syncthreads();
  if (mask_row)
    for (int w = tid; w < words; w += nt) mask_row[w] = mask_s[w];
  for (int i = (int)tot_keep + tid; i < budget; i += nt) kept_row[i] = -1;
  if (tid == 0) {
    kept_count[seg] = (int32_t)tot_keep;
    if (s_nan) record_error(status, KVC_ERR_NAN);
  }
}

// Items per thread in one round of the streaming sweep (the bit masks).
constexpr int kStreamIPT = 64;

__global__ void __launch_bounds__(kSelThreads)
k_select_stream(const float *__restrict__ scores, const int64_t *__restrict__ seg_off,
                int64_t max_seg_len, int budget, int n_sink, int n_recent,
                int32_t *__restrict__ kept, int32_t *__restrict__ kept_count,
                uint32_t *__restrict__ keepmask, int64_t words, int32_t *status) {
  __shared__ uint32_t hist[kSelHist * 256];
  __shared__ uint32_t s_red[2][32];
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t s_kmax, s_kmin, s_prefix, s_need;
  __shared__ int s_nan;

  const int seg = blockIdx.x;
  const int tid = threadIdx.x, nt = blockDim.x;
  int32_t *kept_row = kept + (int64_t)seg * budget;
  uint32_t *mask_row = keepmask ? keepmask + (int64_t)seg * words : nullptr;

  const int64_t off = seg_off[seg], end = seg_off[seg + 1];
  const bool bad = end < off || end - off > max_seg_len || off < 0;
  const int n = bad ? 0 : (int)(end - off);
  if (bad && tid == 0) record_error(status, KVC_ERR_BOUNDS);
  const float *sc = scores + (bad ? 0 : off);

  if (n <= budget) {  // keep everything (or nothing, on a bad segment)
    for (int i = tid; i < budget; i += nt) kept_row[i] = i < n ? i : -1;
    if (mask_row)
      for (int64_t w = tid; w < words; w += nt) {
        const int64_t lo = w * 32;
        mask_row[w] = lo >= n ? 0u : (n - lo >= 32 ? 0xFFFFFFFFu : ((1u << (n - lo)) - 1u));
      }
    if (tid == 0) kept_count[seg] = n;
    return;
  }
  const int rec0 = n - n_recent;
  const int k = budget - n_sink - n_recent;
  const int lane = tid & 31, warp = tid >> 5, n_warps = nt >> 5;
  if (tid == 0) s_nan = 0;
  __syncthreads();

  // pass 1: NaN check over every item, key range of the non-forced ones
  bool nan = false;
  uint32_t lmax = 0u, lmin = 0xFFFFFFFFu;
  for (int i = tid; i < n; i += nt) {
    const uint32_t key = order_key(sc[i], nan);
    if (i >= n_sink && i < rec0) {
      lmax = max(lmax, key);
      lmin = min(lmin, key);
    }
  }
  if (nan) s_nan = 1;
  uint32_t prefix = 0, need = (uint32_t)k;
  if (k > 0) {
    lmax = __reduce_max_sync(0xFFFFFFFFu, lmax);
    lmin = __reduce_min_sync(0xFFFFFFFFu, lmin);
    if (lane == 0) {
      s_red[0][warp] = lmax;
      s_red[1][warp] = lmin;
    }
    __syncthreads();
    if (warp == 0) {
      const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, lane < n_warps ? s_red[0][lane] : 0u);
      const uint32_t mn =
          __reduce_min_sync(0xFFFFFFFFu, lane < n_warps ? s_red[1][lane] : 0xFFFFFFFFu);
      if (lane == 0) {
        s_kmax = mx;
        s_kmin = mn;
      }
    }
    __syncthreads();
    const uint32_t kmax = s_kmax, kmin = s_kmin;
    int hi = kmax == kmin ? -1 : 31 - __clz(kmax ^ kmin);
    prefix = hi < 0 ? kmax : hi == 31 ? 0u : (kmax >> (hi + 1)) << (hi + 1);
    // radix levels, each a pass over the scores
    while (hi >= 0) {
      const int lo = hi >= 7 ? hi - 7 : 0;
      const uint32_t dmask = (2u << (hi - lo)) - 1u;
      const uint32_t pmask = hi == 31 ? 0u : ~((2u << hi) - 1u);
      uint32_t *h = hist + (warp % kSelHist) * 256;
      for (int j = tid; j < kSelHist * 256; j += nt) hist[j] = 0u;
      __syncthreads();
      for (int i = n_sink + tid; i < rec0; i += nt) {
        bool dummy = false;
        const uint32_t key = order_key(sc[i], dummy);
        if ((key & pmask) == prefix) atomicAdd(&h[(key >> lo) & dmask], 1u);
      }
      __syncthreads();
      if (warp == 0) pick_digit(hist, lane, prefix, need, lo, &s_prefix, &s_need);
      __syncthreads();
      prefix = s_prefix;
      need = s_need;
      hi = lo - 1;
    }
  }
  const uint32_t T = prefix;

  // words past the segment's last item are zero (written once, before the
  // sweep, and never touched by it)
  const int64_t used_words = ((int64_t)n + 31) / 32;
  if (mask_row)
    for (int64_t w = used_words + tid; w < words; w += nt) mask_row[w] = 0u;

  // ordered sweep in rounds of nt·64 items; thread t owns the 64 items from
  // base + 64t, i.e. mask words 2·(base/64 + t) and 2·(base/64 + t) + 1
  uint32_t eq_carry = 0, keep_carry = 0;
  for (int base = 0; base < n; base += nt * kStreamIPT) {
    const int i0 = base + tid * kStreamIPT;
    const int cnt = i0 >= n ? 0 : min(kStreamIPT, n - i0);
    uint64_t eqm = 0, km = 0;
    for (int e = 0; e < cnt; e++) {
      const int i = i0 + e;
      bool keep = i < n_sink || i >= rec0, eq = false;
      if (!keep && k > 0) {
        bool dummy = false;
        const uint32_t key = order_key(sc[i], dummy);
        keep = key > T;
        eq = key == T;
      }
      km |= (uint64_t)keep << e;
      eqm |= (uint64_t)eq << e;
    }
    uint32_t tot_eq;
    const uint32_t eq_before = eq_carry + block_excl_scan((uint32_t)__popcll(eqm), &tot_eq,
                                                         warp_tot);
    if (eq_before < need) {
      const uint32_t take = min((uint32_t)__popcll(eqm), need - eq_before);
      uint64_t m = eqm;
      for (uint32_t t = 0; t < take; t++) {
        km |= m & (~m + 1);
        m &= m - 1;
      }
    }
    uint32_t tot_keep;
    uint32_t pos = keep_carry + block_excl_scan((uint32_t)__popcll(km), &tot_keep, warp_tot);
    for (uint64_t m = km; m; m &= m - 1) {
      if (pos < (uint32_t)budget) kept_row[pos] = i0 + __ffsll((long long)m) - 1;
      pos++;
    }
    if (mask_row && cnt > 0) {
      const int64_t w0 = i0 / 32;
      mask_row[w0] = (uint32_t)km;
      if (w0 + 1 < used_words) mask_row[w0 + 1] = (uint32_t)(km >> 32);
    }
    eq_carry += tot_eq;
    keep_carry += tot_keep;
  }
  for (int i = (int)keep_carry + tid; i < budget; i += nt) kept_row[i] = -1;
  if (tid == 0) {
    kept_count[seg] = (int32_t)keep_carry;
    if (s_nan) record_error(status, KVC_ERR_NAN);
  }
}

}  // namespace

cudaError_t launch_select(const float *scores, const int64_t *seg_off,
                          int n_seg, int max_seg_len, int budget, int n_sink,
                          int n_recent, int32_t *kept, int32_t *kept_count,
                          uint32_t *keepmask, int32_t *status,
                          cudaStream_t s) {
  if (max_seg_len > KVC_SELECT_STAGED_SEG) {
    k_select_stream<<<n_seg, kSelThreads, 0, s>>>(scores, seg_off, max_seg_len, budget, n_sink,
                                                  n_recent, kept, kept_count, keepmask,
                                                  ((int64_t)max_seg_len + 31) / 32, status);
    return cudaGetLastError();
  }
  int words = (max_seg_len + 31) / 32;
  size_t smem = ((size_t)max_seg_len + max_seg_len / 32 + 1 + words + kSelHist * 256) *
                sizeof(uint32_t);
  // Segments are independent and latency-bound: CTAs small enough that
  // several fit on an SM (registers and shared memory) put a few hundred
  // segments in one wave; long segments get more threads per CTA.
  // With many segments the GPU is full anyway: fewer threads per segment (up
  // to 64 items each, the sweep's bit masks) put more segments in flight,
  // while a few hundred segments want the shorter per-step passes.
  int ipt = kSelIPT;
  const int64_t waves_threads = (int64_t)device_sm_count() * 2048 * 4;
  while (ipt < 64 && (int64_t)n_seg * ((max_seg_len + ipt - 1) / ipt) > waves_threads) ipt *= 2;
  int threads = 128;
  while (threads < kSelThreads && (max_seg_len + threads - 1) / threads > ipt) threads *= 2;
  // 256 threads wherever they stay within 64 items each: shared memory,
  // sized for the longest segment, already caps the CTAs per SM, so larger
  // CTAs give the same segments more warps (measured: ragged 36,864 segments
  // of ≤ 8192, 1.20 → 1.04 ms; 8B 288 of 4096, 0.038 → 0.036 ms; 512 and 1024
  // threads were slower)
  if (max_seg_len >= 2048 && (max_seg_len + 255) / 256 <= 64) threads = 256;
  cudaError_t e = cudaFuncSetAttribute(
      k_select, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_select, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  k_select<<<n_seg, threads, smem, s>>>(scores, seg_off, max_seg_len, budget,
                                        n_sink, n_recent, kept, kept_count,
                                        keepmask, words, status);
  return cudaGetLastError();
}

}  // namespace kvc
