// meank.cu — Mean-K index build (KVMem, "Query-conditioned retrieval": one
// RoPE-stripped mean key per layer, KV head and 32-token block).
//
// The mean is defined as the exact sum of the block's 32 bf16 values, divided
// by 32 and rounded once to bf16 (round to nearest even).  fp64 would give
// that directly, but GB300's fp64 rate is a small fraction of its fp32 rate:
// an fp64 sum of every element keeps the build far from the HBM bound.  So
// the sum is kept error-free in fp32 instead:
//
//   * one thread owns 8 consecutive head-dim columns of one block row and
//     walks the block's 32 tokens with 16-byte loads (the D/8 threads of a
//     block row read each 2·D-byte token row as one coalesced segment);
//   * per column it keeps s (the fp32 running sum) and c (the fp32 sum of
//     the exact rounding errors of each s + x, from Knuth's TwoSum); over
//     its 8 columns it keeps max|x| and min|x|;
//   * every bf16 input, partial sum and error is a multiple of u, the finest
//     ulp among the column's non-zero inputs, and |c| < 2^-19·A for any
//     A ≥ Σ|x| (A = 32·max|x| here).  When min|x| > 2^-34·A, c therefore
//     stays below 2^24·u and every update of c is exact: s + c is the exact
//     sum;
//   * the exact sum is split once more by TwoSum into t = RN_fp32(sum) and
//     e = sum − t.  Rounding t to bf16 gives the correctly rounded result
//     except when t lies exactly on a bf16 midpoint while e ≠ 0, and then
//     the sign of e decides the direction;
//   * dividing by 32 is an exact exponent shift, given the magnitude guards.
//
// A column outside those guards (a zero or subnormal next to non-zero
// values, magnitudes spanning more than 34 binades, values near the fp32
// range limits, NaN or Inf) sends the thread's 8 columns through a plain
// fp64 sum in token order instead.  That sum is exact for the spans that
// reach it in practice, and its rounding matches the exact mean whenever
// the fp64 sum is exact.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kCols = 8;  // head-dim columns per thread (one 16-byte chunk)

// Knuth's TwoSum: a + b == s + e exactly, for any finite fp32 a and b.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  const float ap = __fsub_rn(s, bp);
  e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

// bf16 (round to nearest even) of the exact value t + e, where t is the fp32
// nearest to it.  Rounding t alone is correct unless t sits exactly halfway
// between two bf16 values while the exact value does not: then e's sign
// picks the neighbour.
__device__ __forceinline__ uint32_t bf16_rne_of_pair(float t, float e) {
  const uint32_t b = __float_as_uint(t);
  if ((b & 0xFFFFu) == 0x8000u && e != 0.f) {
    const bool grows = (e > 0.f) == ((b >> 31) == 0u);  // same sign as t
    return (b >> 16) + (grows ? 1u : 0u);
  }
  return (b + 0x7FFFu + ((b >> 16) & 1u)) >> 16;
}

// Fast-path guard (see the file comment) for the thread's 8 columns, from
// the largest and smallest |x| it read: all zeros, or A = 32·max|x| (an upper
// bound on every column's Σ|x|) inside [2^-60, 2^100) with min|x| > 2^-34·A,
// which also keeps t/32 and e/32 normal so the ÷32 below is exact.
__device__ __forceinline__ bool chunk_exact(float abs_max, float abs_min) {
  if (abs_max == 0.f) return true;
  const float A = abs_max * (float)kBlock;
  return A >= 0x1p-60f && A < 0x1p100f && abs_min > A * 0x1p-34f;
}

__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi) {
  return (lo & 0xFFFFu) | (hi << 16);
}

constexpr int kBatch = 8;  // token rows loaded ahead of their arithmetic

__global__ void __launch_bounds__(256, 4)
k_build_meank(const uint16_t *__restrict__ kraw, uint16_t *__restrict__ meank,
              int64_t n_out_chunks, int chunks_per_row) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n_out_chunks) return;
  const int64_t row_blk = t / chunks_per_row;  // (row, block)
  const int c8 = (int)(t - row_blk * chunks_per_row);
  const int D = chunks_per_row * kCols;
  const uint16_t *src = kraw + row_blk * (int64_t)kBlock * D + c8 * kCols;

  float s[kCols], c[kCols];
#pragma unroll
  for (int e = 0; e < kCols; e++) {
    s[e] = 0.f;
    c[e] = 0.f;
  }
  // two partial extremes each, to shorten the dependency chains
  float amax[2] = {0.f, 0.f}, amin[2] = {INFINITY, INFINITY};
#pragma unroll 1
  for (int t0 = 0; t0 < kBlock; t0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; i++) v[i] = ld_stream(src + (int64_t)(t0 + i) * D);
#pragma unroll
    for (int i = 0; i < kBatch; i++) {
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int e = 0; e < kCols; e++) {
        const float x = (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
        float sn, err;
        two_sum(s[e], x, sn, err);
        s[e] = sn;
        c[e] = __fadd_rn(c[e], err);
        amax[e & 1] = fmaxf(amax[e & 1], fabsf(x));
        amin[e & 1] = fminf(amin[e & 1], fabsf(x));
      }
    }
  }
  const bool exact = chunk_exact(fmaxf(amax[0], amax[1]), fminf(amin[0], amin[1]));

  uint32_t o[kCols];
  if (exact) {
#pragma unroll
    for (int e = 0; e < kCols; e++) {
      float tt, ee;
      two_sum(s[e], c[e], tt, ee);
      // ÷32: an exact exponent shift inside the guarded range
      o[e] = bf16_rne_of_pair(tt * (1.f / kBlock), ee * (1.f / kBlock));
    }
  } else {
    // outside the guards: fp64 sum in token order (rare; re-reads the block)
    double acc[kCols];
#pragma unroll
    for (int e = 0; e < kCols; e++) acc[e] = 0.0;
    for (int tok = 0; tok < kBlock; tok++) {
      const uint4 v = *reinterpret_cast<const uint4 *>(src + (int64_t)tok * D);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < kCols; e++)
        acc[e] += (double)((e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]));
    }
#pragma unroll
    for (int e = 0; e < kCols; e++) {
      __nv_bfloat16 r = __double2bfloat16(acc[e] * (1.0 / kBlock));
      // one NaN encoding (quiet, positive) whatever the inputs' payloads
      o[e] = isnan(acc[e]) ? 0x7FC0u : *reinterpret_cast<uint16_t *>(&r);
    }
  }
  *reinterpret_cast<uint4 *>(meank + row_blk * D + c8 * kCols) =
      make_uint4(pack2(o[0], o[1]), pack2(o[2], o[3]), pack2(o[4], o[5]), pack2(o[6], o[7]));
}

}  // namespace

cudaError_t launch_build_meank(const uint16_t *kraw, uint16_t *meank,
                               int64_t rows, int64_t n_tok, int D,
                               cudaStream_t s) {
  const int64_t nb = n_tok / kBlock;
  const int cpr = D / kCols;
  const int64_t n = rows * nb * cpr;
  const int64_t grid = (n + 255) / 256;
  k_build_meank<<<(unsigned)grid, 256, 0, s>>>(kraw, meank, n, cpr);
  return cudaGetLastError();
}

}  // namespace kvc
