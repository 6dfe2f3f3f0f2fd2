// qmem.cu — QueryMemory update and the rule score over a paged K pool.
//
// IntentKV §4 "Memory recurrence" / §7 item 1: M ← e^{−λ}·M + Enc(q_t), then
// renormalised to unit norm along the head dimension.
// IntentKV §4 "Rule score": rule_j = Σ_{l,hq} softmax_j(M[l,hq]·K[l,h,j]/√D),
// with §4 check 1's GQA expansion (query head hq reads KV head hq / G) and
// K addressed through the paged slot map (ActKV §2).
//
// The rule score is a softmax per (session, layer, query head) over all
// history positions, summed over (layer, query head) per position.  Every
// (l, hq) has its own normaliser, so the per-position sum can only be formed
// once all normalisers are known.  The pool is read once:
//   k_qmem_logits  grid (session, position tile, layer), session fastest so
//                  that the sessions' reads of the shared prefix rows meet in
//                  L2.  A lane takes one KV head of one position, reads its
//                  D-element K slice and forms its GQA group's logits against
//                  M staged in shared memory; the tile's logits go to ws
//                  (coalesced along positions) with a per-tile
//                  (max, Σ2^(z−max)) per (l, hq);
//   k_qmem_lse     combines the tiles into one LSE per (session, l, hq);
//   k_qmem_rule    re-reads the logits (1/16 of the K bytes) and sums
//                  2^(z − LSE) over (l, hq) per position.
// Dead positions (slot = sentinel) carry z = −inf and rule = −1.
// For 8 KV heads and groups of 2, 4 or 8 query heads the logits come from
// the tensor-core kernel of qmem_tc.cu instead; by default that kernel also
// forms each layer's share of the rule score while the logits are still in
// L2 (k_qmem_rule_sum then adds the layers), so the logits never go to DRAM.
// The CUDA-core kernel below covers every other shape.

#include <string.h>

#include <type_traits>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTJ = 256;        // positions per logits tile
constexpr int kLogitThreads = 256;

// ----------------------------------------------------------- update

// One warp per (session, layer, query head) row; lane takes PER = D/32
// consecutive elements (one 8- or 4-byte word per token), eight tokens of
// loads in flight.  The token sum runs in token order per element.
template <int PER>
__global__ void __launch_bounds__(256)
k_qmem_update(float *__restrict__ M, const uint16_t *__restrict__ q,
              int64_t rows, int T, float decay, float gain, int renorm) {
  using Word = typename std::conditional<PER == 4, uint2, uint32_t>::type;
  constexpr int D = 32 * PER;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; e++) acc[e] = 0.f;
  const Word *src = reinterpret_cast<const Word *>(q + row * (int64_t)T * D) + lane;
  auto add = [&](const Word &w) {
    uint32_t u[PER / 2];
    memcpy(u, &w, sizeof(w));
#pragma unroll
    for (int e = 0; e < PER; e++) acc[e] += (e & 1) ? bf16_hi(u[e >> 1]) : bf16_lo(u[e >> 1]);
  };
  int t = 0;
  for (; t + 8 <= T; t += 8) {
    Word w[8];
#pragma unroll
    for (int k = 0; k < 8; k++) w[k] = __ldcs(src + (int64_t)(t + k) * (D / PER));
#pragma unroll
    for (int k = 0; k < 8; k++) add(w[k]);
  }
  for (; t < T; t++) add(__ldcs(src + (int64_t)t * (D / PER)));
  float *m = M + row * D + lane * PER;
  float v[PER], n2 = 0.f;
#pragma unroll
  for (int e = 0; e < PER; e++) {
    v[e] = fmaf(decay, m[e], gain * (acc[e] / (float)T));
    n2 = fmaf(v[e], v[e], n2);
  }
  if (renorm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xFFFFFFFFu, n2, o);
    const float n = sqrtf(n2);
    if (n > 0.f)
#pragma unroll
      for (int e = 0; e < PER; e++) v[e] = v[e] / n;
  }
#pragma unroll
  for (int e = 0; e < PER; e++) m[e] = v[e];
}

// ------------------------------------------------------------ score

struct QArgs {
  const float *M;
  const uint16_t *kpool;
  const int32_t *slot_map;
  float *rule;
  float *logits;  // [n_sess][L][Hq][N]
  float2 *part;   // [n_sess][L][Hq][n_tiles]
  float *lse;     // [n_sess][L][Hq]
  int32_t *status;
  int n_sess, L, H, Hq, D, G, N, n_tiles, sentinel;
  int64_t n_slots;
  float zscale;
};

// Logits of one (session, position tile, layer).
//
// A warp is split into S = 32/NC slices of NC = D/8 lanes; lane c of a slice
// owns head-dim elements [8c, 8c+8).  A slice works through items of kPB
// positions of one KV head h: per position its NC lanes read the head's K
// slice as one contiguous 2·D-byte segment (16 bytes per lane), and each
// lane keeps its 8 elements of M for the GP query heads of h's GQA group in
// registers.  A batch of kB = 16/GP positions gives each lane 16 partial
// dot products; a recursive-halving reduce-scatter over the slice's lanes
// (log2 NC shuffle stages) sums them, leaving the finished logits spread
// over the lanes.  K streams kPF batches ahead of the arithmetic.  The
// tile's logits are transposed through shared memory ([hq][position],
// padded) and written coalesced along positions, with a per-tile
// (max, Σ2^(z−max)) per query head reduced by whole warps.
constexpr int kPB = 32;  // positions per item
constexpr int kPF = 2;   // batches of K in flight ahead of the one in use

template <int D, int GP>
__global__ void __launch_bounds__(kLogitThreads, 2)
k_qmem_logits(QArgs a) {
  extern __shared__ float sm[];
  constexpr int NC = D / 8;                // lanes per slice
  constexpr int S = 32 / NC;               // slices per warp
  constexpr int kB = 16 / GP;              // positions per batch
  constexpr int NV = kB * GP;              // partial sums per lane per batch
  constexpr int ZS = kTJ + 1;              // row stride of Z
  constexpr int n_warps = kLogitThreads / 32;
  static_assert(NV % NC == 0, "reduce-scatter leaves whole values per lane");
  constexpr int NOUT = NV / NC;            // finished logits per lane per batch
  float *Z = sm;                           // [Hq][ZS]
  const int r = blockIdx.x, tile = blockIdx.y, l = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = lane % NC, slice = warp * S + lane / NC;
  const int j0 = tile * kTJ;
  const int32_t *smap = a.slot_map + (int64_t)r * a.N;
  const float *Mrl = a.M + ((int64_t)r * a.L + l) * a.Hq * D;
  const uint16_t *kl = a.kpool + (int64_t)l * a.n_slots * a.H * D;

  const int n_items = a.H * (kTJ / kPB);
  for (int item = slice; item < n_items; item += n_warps * S) {
    const int h = item % a.H, jb = (item / a.H) * kPB;
    // this lane's 8 elements of M for the group's query heads (zero past G)
    float m[GP][8];
#pragma unroll
    for (int g = 0; g < GP; g++) {
      if (g < a.G) {
        const float4 *src = reinterpret_cast<const float4 *>(Mrl + (h * a.G + g) * D + c * 8);
        const float4 lo = __ldg(src), hi = __ldg(src + 1);
        m[g][0] = lo.x; m[g][1] = lo.y; m[g][2] = lo.z; m[g][3] = lo.w;
        m[g][4] = hi.x; m[g][5] = hi.y; m[g][6] = hi.z; m[g][7] = hi.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; e++) m[g][e] = 0.f;
      }
    }
    // slot and liveness of each position (every lane of the slice reads the
    // same slot-map word: one broadcast load)
    const int32_t *sitem = smap + j0 + jb;
    const bool whole = j0 + jb + kPB <= a.N;   // no position past the end
    const uint16_t *kh = kl + (int64_t)h * D + c * 8;
    const uint32_t row = (uint32_t)(a.H * D);
    auto slot_of = [&](int jj, bool &live) -> uint32_t {
      int32_t u = (whole || j0 + jb + jj < a.N) ? sitem[jj] : a.sentinel;
      live = u != a.sentinel;
      if (live && (u < 0 || u >= a.n_slots)) {
        if (c == 0) record_error(a.status, KVC_ERR_BOUNDS);
        live = false;
      }
      return live ? (uint32_t)u : 0u;
    };
    uint4 kbuf[kPF + 1][kB];
    uint32_t lbuf[kPF + 1];  // bit i: position i of the batch is live
    auto fetch = [&](int batch, int buf) {
      lbuf[buf] = 0u;
#pragma unroll
      for (int i = 0; i < kB; i++) {
        bool live;
        const uint32_t u = slot_of(batch * kB + i, live);
        lbuf[buf] |= (uint32_t)live << i;
        kbuf[buf][i] = live ? __ldg(reinterpret_cast<const uint4 *>(
                                  kh + (uint64_t)u * row))
                            : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    constexpr int NBATCH = kPB / kB;
#pragma unroll
    for (int bt = 0; bt < kPF; bt++) fetch(bt, bt);
#pragma unroll
    for (int bt = 0; bt < NBATCH; bt++) {
      if (bt + kPF < NBATCH) fetch(bt + kPF, (bt + kPF) % (kPF + 1));
      const int buf = bt % (kPF + 1);
      float v[NV];  // [position i][g]
#pragma unroll
      for (int i = 0; i < kB; i++) {
        const uint4 w4 = kbuf[buf][i];
        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; e++) x[e] = (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
#pragma unroll
        for (int g = 0; g < GP; g++) {
          float t = 0.f;
#pragma unroll
          for (int e = 0; e < 8; e++) t = fmaf(m[g][e], x[e], t);
          v[i * GP + g] = t;
        }
      }
      // reduce-scatter over the NC lanes of the slice: at the stage with
      // offset o the lane keeps the half of its values selected by bit o of
      // its index and adds the partner's copy of that half
#pragma unroll
      for (int o = NC / 2, n = NV; o >= 1; o >>= 1, n >>= 1) {
        const bool up = (c & o) != 0;
#pragma unroll
        for (int k = 0; k < n / 2; k++) {
          const float keep = up ? v[k + n / 2] : v[k];
          const float send = up ? v[k] : v[k + n / 2];
          v[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
        }
      }
      // lane c now holds values c·NOUT … c·NOUT + NOUT − 1 of [i][g]
#pragma unroll
      for (int k = 0; k < NOUT; k++) {
        const int idx = c * NOUT + k, i = idx / GP, g = idx % GP;
        if (g < a.G) {
          const int jj = jb + bt * kB + i;
          Z[(h * a.G + g) * ZS + jj] = ((lbuf[buf] >> i) & 1u) ? v[k] * a.zscale : -INFINITY;
        }
      }
    }
  }
  __syncthreads();

  // logits out, coalesced along positions
  const int64_t lrow = ((int64_t)r * a.L + l) * a.Hq;
  const int valid = min(kTJ, a.N - j0);
  for (int i = threadIdx.x; i < a.Hq * kTJ; i += kLogitThreads) {
    const int hq = i / kTJ, jj = i - hq * kTJ;
    if (jj < valid) a.logits[(lrow + hq) * a.N + j0 + jj] = Z[hq * ZS + jj];
  }
  // per-tile (max, Σ 2^(z − max)) per query head, one warp per head
  for (int hq = warp; hq < a.Hq; hq += n_warps) {
    const float *zr = Z + hq * ZS;
    float mx = -INFINITY;
    for (int jj = lane; jj < valid; jj += 32) mx = fmaxf(mx, zr[jj]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    float sum = 0.f;
    if (mx > -INFINITY)
      for (int jj = lane; jj < valid; jj += 32) sum += exp2f(zr[jj] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane == 0) a.part[(lrow + hq) * a.n_tiles + tile] = make_float2(mx, sum);
  }
}

__global__ void __launch_bounds__(256)
k_qmem_lse(QArgs a) {
  int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (r, l, hq)
  if (row >= (int64_t)a.n_sess * a.L * a.Hq) return;
  const float2 *p = a.part + row * a.n_tiles;
  float m = -INFINITY;
  for (int t = 0; t < a.n_tiles; t++) m = fmaxf(m, p[t].x);
  float s = 0.f;
  if (m > -INFINITY)
    for (int t = 0; t < a.n_tiles; t++)
      if (p[t].y > 0.f) s += p[t].y * exp2f(p[t].x - m);
  a.lse[row] = m > -INFINITY ? m + log2f(s) : -INFINITY;
}

// rule_j = Σ_{l,hq} 2^(z − LSE): one thread per position, reading the
// session's L·Hq logit rows (coalesced across the warp's positions) with
// eight independent loads and partial sums in flight.
__global__ void __launch_bounds__(256)
k_qmem_rule(QArgs a) {
  extern __shared__ float lse_s[];  // [L·Hq] of this session
  constexpr int U = 8;
  const int r = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int LH = a.L * a.Hq;
  for (int i = threadIdx.x; i < LH; i += blockDim.x) lse_s[i] = a.lse[(int64_t)r * LH + i];
  __syncthreads();
  if (j >= a.N) return;
  int32_t u = a.slot_map[(int64_t)r * a.N + j];
  bool live = u != a.sentinel && u >= 0 && u < a.n_slots;
  float out = -1.f;
  if (live) {
    const float *z = a.logits + (int64_t)r * LH * a.N + j;
    float acc[U];
#pragma unroll
    for (int k = 0; k < U; k++) acc[k] = 0.f;
    int i = 0;
    for (; i + U <= LH; i += U) {
      float zz[U];
#pragma unroll
      for (int k = 0; k < U; k++) zz[k] = __ldcs(z + (int64_t)(i + k) * a.N);
#pragma unroll
      for (int k = 0; k < U; k++) acc[k] += exp2f(zz[k] - lse_s[i + k]);
    }
    for (; i < LH; i++) acc[0] += exp2f(__ldcs(z + (int64_t)i * a.N) - lse_s[i]);
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < U; k++) t += acc[k];
    out = t;
  }
  a.rule[(int64_t)r * a.N + j] = out;
}

// rule[r][j] = Σ_l rule_l[r][l][j] (each layer's Σ_hq 2^(z − LSE), formed
// by the fused tensor-core kernel), −1 for a dead position.
__global__ void __launch_bounds__(256)
k_qmem_rule_sum(const float *__restrict__ rule_l, const int32_t *__restrict__ slot_map,
                float *__restrict__ rule, int L, int N, int32_t sentinel, int64_t n_slots) {
  const int r = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= N) return;
  const int32_t u = slot_map[(int64_t)r * N + j];
  const bool live = u != sentinel && u >= 0 && u < n_slots;
  float out = -1.f;
  if (live) {
    const float *src = rule_l + (int64_t)r * L * N + j;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int l = 0;
    for (; l + 4 <= L; l += 4) {
      float v[4];
#pragma unroll
      for (int k = 0; k < 4; k++) v[k] = __ldcs(src + (int64_t)(l + k) * N);
#pragma unroll
      for (int k = 0; k < 4; k++) acc[k] += v[k];
    }
    for (; l < L; l++) acc[0] += __ldcs(src + (int64_t)l * N);
    out = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  }
  rule[(int64_t)r * N + j] = out;
}

// LSE per (session, layer, query head) from the tile partials, then the
// rule sum over (layer, query head) per position.
cudaError_t launch_qmem_reduce(const QArgs &a, cudaStream_t s) {
  const int64_t rows = (int64_t)a.n_sess * a.L * a.Hq;
  k_qmem_lse<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g3((a.N + 255) / 256, a.n_sess);
  size_t smem3 = (size_t)a.L * a.Hq * sizeof(float);
  if (smem3 > 48 * 1024) {
    e = cudaFuncSetAttribute(k_qmem_rule, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem3);
    if (e != cudaSuccess) return e;
  }
  k_qmem_rule<<<g3, 256, smem3, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qmem_update(float *M, const uint16_t *q, int64_t rows,
                               int D, int T, float decay, float gain,
                               int renorm, cudaStream_t s) {
  const int64_t threads = rows * 32;
  const unsigned grid = (unsigned)((threads + 255) / 256);
  if (D == 128)
    k_qmem_update<4><<<grid, 256, 0, s>>>(M, q, rows, T, decay, gain, renorm);
  else if (D == 64)
    k_qmem_update<2><<<grid, 256, 0, s>>>(M, q, rows, T, decay, gain, renorm);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// Scratch: logits [n_sess][L][Hq][N] fp32, tile partials, LSEs, the
// two-term bf16 copy of M that the tensor-core logits read, and for the
// fused finish one counter per (session, layer) and rule_l [n_sess][L][N].
size_t score_qmem_ws_bytes(int n_sess, int L, int Hq, int N) {
  int64_t rows = (int64_t)n_sess * L * Hq;
  int n_tiles = (N + kTJ - 1) / kTJ;
  size_t logits = (size_t)rows * N * sizeof(float);
  size_t part = (size_t)rows * n_tiles * sizeof(float2);
  size_t lse = (size_t)rows * sizeof(float);
  size_t counters = (size_t)n_sess * L * sizeof(int);
  size_t rule_l = (size_t)n_sess * L * N * sizeof(float);
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  return al(logits) + al(part) + al(lse) + al(qmem_tc_mb_bytes(n_sess, L, Hq)) + al(counters) +
         al(rule_l);
}

cudaError_t launch_score_qmem(const float *M, const uint16_t *kpool,
                              const int32_t *slot_map, int32_t sentinel,
                              float *rule, int n_sess, int L, int H, int Hq,
                              int D, int N, int64_t n_slots, void *ws,
                              int32_t *status, int path, cudaStream_t s) {
  QArgs a;
  int64_t rows = (int64_t)n_sess * L * Hq;
  a.n_tiles = (N + kTJ - 1) / kTJ;
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  char *w = static_cast<char *>(ws);
  a.logits = reinterpret_cast<float *>(w);
  w += al((size_t)rows * N * sizeof(float));
  a.part = reinterpret_cast<float2 *>(w);
  w += al((size_t)rows * a.n_tiles * sizeof(float2));
  a.lse = reinterpret_cast<float *>(w);
  w += al((size_t)rows * sizeof(float));
  uint16_t *mb = reinterpret_cast<uint16_t *>(w);
  w += al(qmem_tc_mb_bytes(n_sess, L, Hq));
  int *counter = reinterpret_cast<int *>(w);
  w += al((size_t)n_sess * L * sizeof(int));
  float *rule_l = reinterpret_cast<float *>(w);
  a.M = M;
  a.kpool = kpool;
  a.slot_map = slot_map;
  a.rule = rule;
  a.status = status;
  a.n_sess = n_sess;
  a.L = L;
  a.H = H;
  a.Hq = Hq;
  a.D = D;
  a.G = Hq / H;
  a.N = N;
  a.sentinel = sentinel;
  a.n_slots = n_slots;
  a.zscale = kLog2e / sqrtf((float)D);
  cudaError_t e;
  const bool tc = qmem_tc_supported(H, Hq, D, L, n_slots);
  if ((path == KVC_KERNEL_QMEM_TC || path == KVC_KERNEL_QMEM_TC_SPILL) && !tc)
    return cudaErrorNotSupported;
  if (tc && (path == KVC_KERNEL_AUTO || path == KVC_KERNEL_QMEM_TC)) {
    e = launch_qmem_logits_tc(M, kpool, slot_map, sentinel, a.logits, a.part, a.lse, counter,
                              rule_l, mb, n_sess, L, H, Hq, D, N, n_slots, a.n_tiles, true,
                              status, s);
    if (e == cudaSuccess) {
      k_qmem_rule_sum<<<dim3((N + 255) / 256, n_sess), 256, 0, s>>>(rule_l, slot_map, rule, L, N,
                                                                     sentinel, n_slots);
      return cudaGetLastError();
    }
    if (e != cudaErrorNotSupported || path == KVC_KERNEL_QMEM_TC) return e;
  }
  if (tc && path != KVC_KERNEL_QMEM_CC) {
    e = launch_qmem_logits_tc(M, kpool, slot_map, sentinel, a.logits, a.part, a.lse, counter,
                              rule_l, mb, n_sess, L, H, Hq, D, N, n_slots, a.n_tiles, false,
                              status, s);
    if (e != cudaSuccess) return e;
    return launch_qmem_reduce(a, s);
  }
  const int GP = a.G <= 4 ? 4 : 8;
  const size_t smem = (size_t)Hq * (kTJ + 1) * sizeof(float);
  dim3 g1(n_sess, a.n_tiles, L);
#define KVC_LOGITS_CASE(DV, GV)                                              \
  if (D == DV && GP == GV) {                                                 \
    e = cudaFuncSetAttribute(k_qmem_logits<DV, GV>,                          \
                             cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                             (int)smem);                                     \
    if (e != cudaSuccess) return e;                                          \
    k_qmem_logits<DV, GV><<<g1, kLogitThreads, smem, s>>>(a);                \
  } else
  KVC_LOGITS_CASE(128, 4)
  KVC_LOGITS_CASE(128, 8)
  KVC_LOGITS_CASE(64, 4)
  KVC_LOGITS_CASE(64, 8)
  return cudaErrorInvalidValue;
#undef KVC_LOGITS_CASE
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_qmem_reduce(a, s);
}

}  // namespace kvc
