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
//                  L2.  A warp takes one position at a time, reads the
//                  slot's H·D K row (one 16-byte-vector sweep per lane) and
//                  forms the Hq logits against M staged in shared memory;
//                  the tile's logits go to ws (coalesced along positions)
//                  with a per-tile (max, Σ2^(z−max)) per (l, hq);
//   k_qmem_lse     combines the tiles into one LSE per (session, l, hq);
//   k_qmem_rule    re-reads the logits (1/16 of the K bytes) and sums
//                  2^(z − LSE) over (l, hq) per position.
// Dead positions (slot = sentinel) carry z = −inf and rule = −1.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTJ = 128;        // positions per logits tile
constexpr int kLogitThreads = 256;

// ----------------------------------------------------------- update

__global__ void __launch_bounds__(256)
k_qmem_update(float *__restrict__ M, const uint16_t *__restrict__ q,
              int64_t rows, int D, int T, float decay, float gain,
              int renorm) {
  int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int per = D / 32;  // 2 or 4 elements per lane
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint16_t *src = q + row * (int64_t)T * D + lane * per;
  for (int t = 0; t < T; t++)
    for (int e = 0; e < per; e++)
      acc[e] += __uint_as_float((uint32_t)src[(int64_t)t * D + e] << 16);
  float *m = M + row * D + lane * per;
  float v[4], n2 = 0.f;
  for (int e = 0; e < per; e++) {
    v[e] = fmaf(decay, m[e], gain * (acc[e] / (float)T));
    n2 = fmaf(v[e], v[e], n2);
  }
  if (renorm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xFFFFFFFFu, n2, o);
    float n = sqrtf(n2);
    if (n > 0.f)
      for (int e = 0; e < per; e++) v[e] = v[e] / n;
  }
  for (int e = 0; e < per; e++) m[e] = v[e];
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

// E = H·D/32 contiguous K elements per lane (a multiple of 8); the lanes of
// one KV head are 32/H consecutive lanes.
template <int E>
__global__ void __launch_bounds__(kLogitThreads)
k_qmem_logits(QArgs a) {
  extern __shared__ float sm[];
  float *Ms = sm;                            // [Hq][D]
  float *Z = Ms + (size_t)a.Hq * a.D;        // [Hq][kTJ + 1]
  const int r = blockIdx.x, tile = blockIdx.y, l = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_warps = kLogitThreads / 32;
  const int lanes_per_head = 32 / a.H;
  const int h = lane / lanes_per_head;
  const int d0 = (lane % lanes_per_head) * E;

  const float *Msrc = a.M + ((int64_t)r * a.L + l) * a.Hq * a.D;
  for (int i = threadIdx.x; i < a.Hq * a.D; i += blockDim.x) Ms[i] = Msrc[i];
  __syncthreads();

  const int j0 = tile * kTJ;
  const int32_t *smap = a.slot_map + (int64_t)r * a.N;
  for (int jj = warp; jj < kTJ; jj += n_warps) {
    const int j = j0 + jj;
    int32_t u = j < a.N ? smap[j] : a.sentinel;
    bool live = u != a.sentinel;
    if (live && (u < 0 || u >= a.n_slots)) {
      if (lane == 0) record_error(a.status, KVC_ERR_BOUNDS);
      live = false;
    }
    float kv[E];
    if (live) {
      const uint16_t *krow = a.kpool + (((int64_t)l * a.n_slots + u) * a.H) * a.D +
                             (int64_t)lane * E;
#pragma unroll
      for (int v = 0; v < E / 8; v++) {
        uint4 w = __ldg(reinterpret_cast<const uint4 *>(krow) + v);
        kv[8 * v + 0] = bf16_lo(w.x);
        kv[8 * v + 1] = bf16_hi(w.x);
        kv[8 * v + 2] = bf16_lo(w.y);
        kv[8 * v + 3] = bf16_hi(w.y);
        kv[8 * v + 4] = bf16_lo(w.z);
        kv[8 * v + 5] = bf16_hi(w.z);
        kv[8 * v + 6] = bf16_lo(w.w);
        kv[8 * v + 7] = bf16_hi(w.w);
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; e++) kv[e] = 0.f;
    }
    for (int g = 0; g < a.G; g++) {
      const int hq = h * a.G + g;
      const float *mrow = Ms + hq * a.D + d0;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; e++) dot = fmaf(mrow[e], kv[e], dot);
      for (int o = lanes_per_head >> 1; o > 0; o >>= 1)
        dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
      if ((lane % lanes_per_head) == 0)
        Z[hq * (kTJ + 1) + jj] = live ? dot * a.zscale : -INFINITY;
    }
  }
  __syncthreads();
  // logits out, coalesced along positions
  const int64_t lrow = ((int64_t)r * a.L + l) * a.Hq;
  for (int i = threadIdx.x; i < a.Hq * kTJ; i += blockDim.x) {
    int hq = i / kTJ, jj = i - hq * kTJ;
    int j = j0 + jj;
    if (j < a.N) a.logits[(lrow + hq) * a.N + j] = Z[hq * (kTJ + 1) + jj];
  }
  // per-tile (max, Σ 2^(z − max)) per query head
  for (int hq = threadIdx.x; hq < a.Hq; hq += blockDim.x) {
    const float *zr = Z + hq * (kTJ + 1);
    int valid = min(kTJ, a.N - j0);
    float m = -INFINITY;
    for (int jj = 0; jj < valid; jj++) m = fmaxf(m, zr[jj]);
    float s = 0.f;
    if (m > -INFINITY)
      for (int jj = 0; jj < valid; jj++) s += exp2f(zr[jj] - m);
    a.part[(lrow + hq) * a.n_tiles + tile] = make_float2(m, s);
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

__global__ void __launch_bounds__(256)
k_qmem_rule(QArgs a) {
  extern __shared__ float lse_s[];  // [L·Hq] of this session
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
    float acc = 0.f;
    for (int i = 0; i < LH; i++) acc += exp2f(__ldcs(z + (int64_t)i * a.N) - lse_s[i]);
    out = acc;
  }
  a.rule[(int64_t)r * a.N + j] = out;
}

}  // namespace

cudaError_t launch_qmem_update(float *M, const uint16_t *q, int64_t rows,
                               int D, int T, float decay, float gain,
                               int renorm, cudaStream_t s) {
  int64_t threads = rows * 32;
  k_qmem_update<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(
      M, q, rows, D, T, decay, gain, renorm);
  return cudaGetLastError();
}

size_t score_qmem_ws_bytes(int n_sess, int L, int Hq, int N) {
  int64_t rows = (int64_t)n_sess * L * Hq;
  int n_tiles = (N + kTJ - 1) / kTJ;
  size_t logits = (size_t)rows * N * sizeof(float);
  size_t part = (size_t)rows * n_tiles * sizeof(float2);
  size_t lse = (size_t)rows * sizeof(float);
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  return al(logits) + al(part) + al(lse);
}

cudaError_t launch_score_qmem(const float *M, const uint16_t *kpool,
                              const int32_t *slot_map, int32_t sentinel,
                              float *rule, int n_sess, int L, int H, int Hq,
                              int D, int N, int64_t n_slots, void *ws,
                              int32_t *status, cudaStream_t s) {
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
  const int E = H * D / 32;
  size_t smem = ((size_t)Hq * D + (size_t)Hq * (kTJ + 1)) * sizeof(float);
  dim3 g1(n_sess, a.n_tiles, L);
  cudaError_t e;
#define KVC_LOGITS_CASE(EV)                                                  \
  case EV:                                                                   \
    e = cudaFuncSetAttribute(k_qmem_logits<EV>,                              \
                             cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                             (int)smem);                                     \
    if (e != cudaSuccess) return e;                                          \
    k_qmem_logits<EV><<<g1, kLogitThreads, smem, s>>>(a);                    \
    break;
  switch (E) {
    KVC_LOGITS_CASE(8)
    KVC_LOGITS_CASE(16)
    KVC_LOGITS_CASE(32)
    KVC_LOGITS_CASE(64)
    default: return cudaErrorInvalidValue;
  }
#undef KVC_LOGITS_CASE
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_qmem_lse<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g3((N + 255) / 256, n_sess);
  size_t smem3 = (size_t)L * Hq * sizeof(float);
  if (smem3 > 48 * 1024) {
    e = cudaFuncSetAttribute(k_qmem_rule, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem3);
    if (e != cudaSuccess) return e;
  }
  k_qmem_rule<<<g3, 256, smem3, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvc
