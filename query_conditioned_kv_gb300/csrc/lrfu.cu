// lrfu.cu — ActKV's attention-aware LRFU keep score (§5.2, Algorithm 1).
//
// After an action region every KV entry's keep score decays by λ and gains
// the entry's action-region attention score s when the entry is a hit, a
// hit being membership of the region's top-p set:
//   KS ← λ·KS + hit·s,
//   hit ⇔ the entry is in the shortest prefix of the entries ordered by
//         score (descending, lower index first) whose mass reaches p·Σ s.
// Scores that are not positive finite numbers have no mass and never hit.
//
// One CTA per segment (a request's entries).  The score bits of a positive
// finite float order like the float, so the top-p boundary is a key
// threshold: T = the largest key with mass(key ≥ T) ≥ p·total, found two
// bits per pass from the top (16 passes, three candidate masses each).
// Masses are (hi, lo) fp32 pairs with every rounding error kept (about 48
// significant bits; GB300's fp64 rate is too low for per-item fp64 sums),
// summed over the CTA in one fixed order, so the total and every candidate
// mass are computed alike.
// Entries with key > T are hits; of those equal to T, the first
// ⌈(p·total − mass(key > T)) / τ⌉ by index are (a block scan of per-thread
// tie counts gives each tie its rank).  Then the keep score is updated in
// place and the hit mask written.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kLrfuThreads = 512;

__device__ __forceinline__ uint32_t mass_key(float s, bool &bad) {
  if (s != s || isinf(s)) {
    bad = bad || s != s;
    return 0u;
  }
  return s > 0.f ? __float_as_uint(s) : 0u;
}

// hi + lo += x with the rounding error of every addition kept (Knuth's
// TwoSum): a partial mass carries ~48 significant bits in fp32 arithmetic,
// which GB300 runs far faster than fp64.
__device__ __forceinline__ void two_sum_acc(float &hi, float &lo, float x) {
  const float s = hi + x;
  const float bp = s - hi;
  const float e = (hi - (s - bp)) + (x - bp);
  hi = s;
  lo += e;
}

// (hi, lo) += (h2, l2), renormalised so that |lo| stays below an ulp of hi.
__device__ __forceinline__ void pair_add(float &hi, float &lo, float h2, float l2) {
  two_sum_acc(hi, lo, h2);
  lo += l2;
  const float s = hi + lo;
  lo = lo - (s - hi);
  hi = s;
}

// Sum over the CTA of N (hi, lo) pairs per thread, in one fixed order: a
// shuffle tree inside each warp, then one warp over the warp sums; every
// thread gets the N totals as fp64.
template <int N>
__device__ __forceinline__ void block_sum(float (&hi)[N], float (&lo)[N], double (&out)[N],
                                          float2 *red, double *res) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = kLrfuThreads / 32;
#pragma unroll
  for (int k = 0; k < N; k++) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float h2 = __shfl_xor_sync(0xFFFFFFFFu, hi[k], o);
      const float l2 = __shfl_xor_sync(0xFFFFFFFFu, lo[k], o);
      pair_add(hi[k], lo[k], h2, l2);
    }
    if (lane == 0) red[k * NW + warp] = make_float2(hi[k], lo[k]);
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < N; k++) {
      const float2 v = lane < NW ? red[k * NW + lane] : make_float2(0.f, 0.f);
      float h = v.x, l = v.y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xFFFFFFFFu, h, o);
        const float l2 = __shfl_xor_sync(0xFFFFFFFFu, l, o);
        pair_add(h, l, h2, l2);
      }
      if (lane == 0) res[k] = (double)h + (double)l;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < N; k++) out[k] = res[k];
  __syncthreads();
}

__device__ __forceinline__ int block_excl_scan_int(int v, int *red, int &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  int before = 0;
  total = 0;
  for (int w = 0; w < kLrfuThreads / 32; w++) {
    if (w < warp) before += red[w];
    total += red[w];
  }
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kLrfuThreads)
k_lrfu(const float *__restrict__ scores, const int64_t *__restrict__ seg_off, int max_seg_len,
       float p, float lambda, float *__restrict__ ks, uint32_t *__restrict__ hitmask, int words,
       int32_t *status) {
  extern __shared__ uint32_t keys[];  // [max_seg_len]
  __shared__ float2 red_f[3 * (kLrfuThreads / 32)];
  __shared__ double red_d[3];
  __shared__ int red_i[kLrfuThreads / 32];
  const int seg = blockIdx.x, tid = threadIdx.x;
  const int64_t off = seg_off[seg], end = seg_off[seg + 1];
  const bool badseg = end < off || end - off > max_seg_len || off < 0;
  const int n = badseg ? 0 : (int)(end - off);
  if (badseg && tid == 0) record_error(status, KVC_ERR_BOUNDS);
  // this thread's contiguous items [i0, i1)
  const int ipt = (n + kLrfuThreads - 1) / kLrfuThreads;
  const int i0 = min(n, tid * ipt), i1 = min(n, i0 + ipt);
  bool nan = false;
  for (int i = i0; i < i1; i++) keys[i] = mass_key(scores[off + i], nan);
  if (nan) record_error(status, KVC_ERR_NAN);
  __syncthreads();
  // masses of the items with key ≥ t[k], in one fixed order
  auto mass_ge = [&](const uint32_t (&t)[3], double (&m)[3]) {
    float hi[3] = {0.f, 0.f, 0.f}, lo[3] = {0.f, 0.f, 0.f};
    for (int i = i0; i < i1; i++) {
      const uint32_t k = keys[i];
      const float x = __uint_as_float(k);
#pragma unroll
      for (int c = 0; c < 3; c++)
        if (k && k >= t[c]) two_sum_acc(hi[c], lo[c], x);
    }
    block_sum<3>(hi, lo, m, red_f, red_d);
  };
  double m3[3];
  {
    const uint32_t t[3] = {1u, 1u, 1u};
    mass_ge(t, m3);
  }
  const double total = m3[0];
  const double target = (double)p * total;
  uint32_t T = 0xFFFFFFFFu;  // no hits unless some mass is asked for
  double above = 0.0;
  int need = 0;
  const bool any = total > 0.0 && target > 0.0;  // p = 0: the empty prefix suffices
  if (any) {
    // two bits per pass: the largest of the three candidates that still
    // holds p of the mass extends the threshold
    uint32_t prefix = 0u;
    for (int b = 30; b >= 0; b -= 2) {
      const uint32_t t[3] = {prefix | (1u << b), prefix | (2u << b), prefix | (3u << b)};
      mass_ge(t, m3);
      if (m3[2] >= target) prefix = t[2];
      else if (m3[1] >= target) prefix = t[1];
      else if (m3[0] >= target) prefix = t[0];
    }
    T = prefix;
    const uint32_t t[3] = {T + 1u, T + 1u, T + 1u};
    mass_ge(t, m3);
    above = m3[0];
    const double tau = (double)__uint_as_float(T);
    const double c = ceil((target - above) / tau);
    need = c < 1.0 ? 1 : (c > (double)n ? n : (int)c);
  }
  // rank of each tie by index
  int my_ties = 0;
  for (int i = i0; i < i1; i++) my_ties += keys[i] == T;
  int n_ties;
  int rank = block_excl_scan_int(my_ties, red_i, n_ties);
  uint32_t *mrow = hitmask ? hitmask + (int64_t)seg * words : nullptr;
  if (mrow)
    for (int w = tid; w < words; w += kLrfuThreads) mrow[w] = 0u;
  __syncthreads();
  for (int i = i0; i < i1; i++) {
    const uint32_t k = keys[i];
    bool hit = false;
    if (any && k) {
      if (k > T) hit = true;
      else if (k == T) hit = rank++ < need;
    }
    const float s = hit ? __uint_as_float(k) : 0.f;
    float *kp = ks + off + i;
    *kp = fmaf(lambda, *kp, s);
    if (hit && mrow) atomicOr(mrow + i / 32, 1u << (i % 32));
  }
}

}  // namespace

cudaError_t launch_lrfu(const float *scores, const int64_t *seg_off, int n_seg, int max_seg_len,
                        float p, float lambda, float *ks, uint32_t *hitmask, int32_t *status,
                        cudaStream_t s) {
  const size_t smem = (size_t)max_seg_len * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_lrfu, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int words = (max_seg_len + 31) / 32;
  k_lrfu<<<n_seg, kLrfuThreads, smem, s>>>(scores, seg_off, max_seg_len, p, lambda, ks, hitmask,
                                           words, status);
  return cudaGetLastError();
}

}  // namespace kvc
