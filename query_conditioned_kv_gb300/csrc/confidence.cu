// confidence.cu — ActKV's confidence monitor and adaptive budget (§6.1,
// §6.2 Algorithm 2) on the GPU.
//
// Token confidence of one predicted distribution (a row of logits):
//   C = −(1/k) Σ_{j ≤ k} log P(j) = LSE − (1/k) Σ_{j ≤ k} logit(j).
// One CTA per row.  Pass 1 forms the row's LSE (per-thread online max/sum,
// merged in a fixed order) and the histogram of the top byte of each
// logit's order-preserving key; three more passes narrow the byte of the
// k-th largest key, so its exact value τ and the count of larger logits are
// known; a last pass sums the logits above τ, and the k − count ties add
// k − count copies of τ.  The row is re-read from L2 by every pass, with
// 16-byte loads, four in flight per thread.
//
// Trace trend and budget: per trace (one request's confidence sequence),
// min pooling over windows of w tokens at stride s, the windows at or below
// the b-th percentile (linear interpolation of the order statistics, after
// a bitonic sort in shared memory), the least-squares slope of those
// windows against their index (fp64 sums in a fixed order), and the budget
// rule: raised by `step` (capped) when the slope is negative, never lowered.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kConfThreads = 1024;
constexpr int kTrendThreads = 1024;
constexpr int kTrendMaxWindows = 8192;

__device__ __forceinline__ uint32_t okey(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ofloat(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Calls f(x) for every logit of the row: 16-byte loads, four in flight per
// thread, when the row is 16-byte aligned (V % 4 == 0), else scalar loads.
template <typename F>
__device__ __forceinline__ void for_each_logit(const float *row, int V, bool vec, F f) {
  const int tid = threadIdx.x;
  if (vec) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    const int n4 = V / 4;
    int i = tid;
    for (; i + 3 * kConfThreads < n4; i += 4 * kConfThreads) {
      float4 a[4];
#pragma unroll
      for (int u = 0; u < 4; u++) a[u] = __ldg(r4 + i + u * kConfThreads);
#pragma unroll
      for (int u = 0; u < 4; u++) {
        f(a[u].x);
        f(a[u].y);
        f(a[u].z);
        f(a[u].w);
      }
    }
    for (; i < n4; i += kConfThreads) {
      const float4 a = __ldg(r4 + i);
      f(a.x);
      f(a.y);
      f(a.z);
      f(a.w);
    }
  } else {
    for (int v = tid; v < V; v += kConfThreads) f(__ldg(row + v));
  }
}

__global__ void __launch_bounds__(kConfThreads)
k_token_confidence(const float *__restrict__ logits, int V, int k, float *__restrict__ conf,
                   int32_t *status) {
  __shared__ uint32_t hist[256];
  __shared__ float red_m[kConfThreads / 32], red_s[kConfThreads / 32];
  __shared__ uint32_t s_prefix, s_need;
  __shared__ float s_sum[kConfThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float *row = logits + (int64_t)blockIdx.x * V;
  constexpr float kL2e = 1.4426950408889634f;

  // pass 1: online (max, Σ 2^((x − max)·log2 e)) and the top-byte histogram
  for (int i = tid; i < 256; i += kConfThreads) hist[i] = 0u;
  __syncthreads();
  const bool vec = (V % 4) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
  float m = -INFINITY, s = 0.f;
  bool nan = false;
  for_each_logit(row, V, vec, [&](float x) {
    if (x != x) nan = true;
    if (x > m) {
      s = (m == -INFINITY ? 0.f : s * exp2f((m - x) * kL2e)) + 1.f;
      m = x;
    } else {
      s += exp2f((x - m) * kL2e);
    }
    atomicAdd(&hist[okey(x) >> 24], 1u);
  });
  if (nan) record_error(status, KVC_ERR_NAN);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    const float mn = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * exp2f((m - mn) * kL2e)) +
        (m2 == -INFINITY ? 0.f : s2 * exp2f((m2 - mn) * kL2e));
    m = mn;
  }
  if (lane == 0) {
    red_m[warp] = m;
    red_s[warp] = s;
  }
  __syncthreads();
  float M = -INFINITY;
  for (int w = 0; w < kConfThreads / 32; w++) M = fmaxf(M, red_m[w]);
  float S = 0.f;
  for (int w = 0; w < kConfThreads / 32; w++)
    if (red_m[w] != -INFINITY) S += red_s[w] * exp2f((red_m[w] - M) * kL2e);
  const float lse = M + logf(S);

  // the k-th largest key, one byte per pass (the histogram of pass 1 first)
  uint32_t prefix = 0u, need = (uint32_t)k;
  for (int d = 3; d >= 0; d--) {
    if (d < 3) {
      __syncthreads();
      for (int i = tid; i < 256; i += kConfThreads) hist[i] = 0u;
      __syncthreads();
      const int sh = 8 * (d + 1);
      const uint32_t want = prefix >> sh;
      const int dsh = 8 * d;
      for_each_logit(row, V, vec, [&](float x) {
        const uint32_t key = okey(x);
        if ((key >> sh) == want) atomicAdd(&hist[(key >> dsh) & 255u], 1u);
      });
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t acc = 0u;
      int bkt = 255;
      for (; bkt > 0; bkt--) {
        if (acc + hist[bkt] >= need) break;
        acc += hist[bkt];
      }
      s_prefix = prefix | ((uint32_t)bkt << (8 * d));
      s_need = need - acc;
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
  }
  // τ = the k-th largest logit; (k − need) logits lie strictly above it
  const float tau = ofloat(prefix);
  float part = 0.f;
  for_each_logit(row, V, vec, [&](float x) {
    if (okey(x) > prefix) part += x;
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
  if (lane == 0) s_sum[warp] = part;
  __syncthreads();
  if (tid == 0) {
    float top = 0.f;
    for (int w = 0; w < kConfThreads / 32; w++) top += s_sum[w];
    top += (float)need * tau;
    conf[blockIdx.x] = lse - top / (float)k;
  }
}

// ------------------------------------------------------------- trend

__device__ __forceinline__ double block_sum_d(double v, double *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < kTrendThreads / 32; w++) t += red[w];
  __syncthreads();
  return t;
}

__global__ void __launch_bounds__(kTrendThreads)
k_conf_trend(const float *__restrict__ conf, const int64_t *__restrict__ trace_off,
             int max_len, int n_max, int w, int s, float b, int step, int max_budget,
             double *__restrict__ slope, int32_t *__restrict__ budget,
             int32_t *__restrict__ n_kept, int32_t *status) {
  extern __shared__ float tsm[];  // rp [n_max], then srt [pow2 ≥ n_max]
  __shared__ double red[kTrendThreads / 32];
  const int t = blockIdx.x, tid = threadIdx.x;
  const int64_t off = trace_off[t], end = trace_off[t + 1];
  const bool bad = end < off || end - off > max_len || off < 0;
  const int L = bad ? 0 : (int)(end - off);
  if (bad && tid == 0) record_error(status, KVC_ERR_BOUNDS);
  const int n = L < w ? 0 : (L - w) / s + 1;
  float *rp = tsm, *srt = tsm + n_max;
  if (n == 0) {
    if (tid == 0) {
      slope[t] = 0.0;
      n_kept[t] = 0;
    }
    return;
  }
  const float *c = conf + off;
  for (int m = tid; m < n; m += kTrendThreads) {
    float mn = INFINITY;
    for (int i = m * s; i < m * s + w; i++) mn = fminf(mn, c[i]);
    rp[m] = mn;
  }
  // bitonic sort of a copy (ascending), padded with +∞
  int np2 = 1;
  while (np2 < n) np2 <<= 1;
  for (int i = tid; i < np2; i += kTrendThreads) srt[i] = i < n ? rp[i] : INFINITY;
  __syncthreads();
  for (int size = 2; size <= np2; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < np2; i += kTrendThreads) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const float a = srt[i], bb = srt[j];
          if ((a > bb) == up) {
            srt[i] = bb;
            srt[j] = a;
          }
        }
      }
      __syncthreads();
    }
  const double pos = (double)b / 100.0 * (double)(n - 1);
  const int lo = (int)floor(pos);
  const int hi = lo + 1 < n ? lo + 1 : lo;
  const double q = (double)srt[lo] + (pos - (double)lo) * ((double)srt[hi] - (double)srt[lo]);
  double sx = 0.0, sy = 0.0, sxx = 0.0, sxy = 0.0, cnt = 0.0;
  for (int m = tid; m < n; m += kTrendThreads) {
    const double y = (double)rp[m];
    if (y <= q) {
      sx += m;
      sy += y;
      sxx += (double)m * m;
      sxy += (double)m * y;
      cnt += 1.0;
    }
  }
  sx = block_sum_d(sx, red);
  sy = block_sum_d(sy, red);
  sxx = block_sum_d(sxx, red);
  sxy = block_sum_d(sxy, red);
  cnt = block_sum_d(cnt, red);
  if (tid == 0) {
    const double den = cnt * sxx - sx * sx;
    const double a = (cnt >= 2.0 && den > 0.0) ? (cnt * sxy - sx * sy) / den : 0.0;
    slope[t] = a;
    n_kept[t] = (int32_t)cnt;
    if (a < 0.0) {
      const int nb = budget[t] + step;
      budget[t] = nb < max_budget ? nb : (budget[t] > max_budget ? budget[t] : max_budget);
    }
  }
}

}  // namespace

cudaError_t launch_token_confidence(const float *logits, int n_tok, int V, int k, float *conf,
                                    int32_t *status, cudaStream_t s) {
  k_token_confidence<<<n_tok, kConfThreads, 0, s>>>(logits, V, k, conf, status);
  return cudaGetLastError();
}

cudaError_t launch_conf_trend(const float *conf, const int64_t *trace_off, int n_trace,
                              int max_len, int w, int stride, float b, int step, int max_budget,
                              double *slope, int32_t *budget, int32_t *n_kept, int32_t *status,
                              cudaStream_t s) {
  const int n_max = max_len < w ? 1 : (max_len - w) / stride + 1;
  int np2 = 1;
  while (np2 < n_max) np2 <<= 1;
  const size_t smem = (size_t)(n_max + np2) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_conf_trend,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_conf_trend<<<n_trace, kTrendThreads, smem, s>>>(conf, trace_off, max_len, n_max, w, stride,
                                                    b, step, max_budget, slope, budget, n_kept,
                                                    status);
  return cudaGetLastError();
}

int conf_trend_max_windows() { return kTrendMaxWindows; }

}  // namespace kvc
