// score_meank.cu — Mean-K block scoring on the CUDA cores.
//
// KVMem, "Query-conditioned retrieval": history blocks are scored in the
// model's own attention space against RoPE-stripped Mean-K and turned into
// attention mass by a softmax over blocks; ActKV §7.1 (Algorithm 3) fixes
// the per-KV-head aggregation: max over the query heads of the GQA group,
// mean over the query tokens.  For one unit (layer l, KV head h, session r)
// with rows ρ = g·W + w (R = G·W query rows):
//   z[ρ,b]   = q[ρ]·meank[b] / sqrt(D)
//   LSE[ρ]   = log Σ_b exp z[ρ,b]
//   score[b] = (1/W) Σ_w max_g exp(z[g·W+w, b] − LSE[g·W+w])
// Everything is carried in base 2 (z₂ = z·log2 e, 2^(z₂ − LSE₂)), which is
// the same quantity.
//
// Two passes, because the probability of a block needs the row's LSE over
// all blocks first:
//   pass 1  grid (split, unit): each CTA streams its share of the unit's
//           Mean-K in 64-block chunks, computes the R×64 logit tile and
//           keeps a running (max, Σ2^(z−max)) per row → ws partials.
//   pass 2  grid (chunk, unit): combines the unit's partials into LSE,
//           recomputes the chunk's logits and reduces max over g, mean over
//           w into the block scores.
// The logit tile is an R×64×D fp32 product from shared memory (q and Mean-K
// staged transposed so that both operand reads are bank-conflict free).

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kCH = 64;        // blocks per chunk (logit-tile width)
constexpr int kThreads = 256;  // 32 row groups × 8 block groups
constexpr int kMaxSplit = 8;
constexpr float kLog2e = 1.4426950408889634f;

struct ScoreArgs {
  const uint16_t *q;
  const uint16_t *meank;
  float *scores;
  const int64_t *blk_off;
  float2 *part;  // [unit][split][R] (max₂, Σ2^(z₂−max₂))
  int32_t *status;
  int L, H, Hq, D, W, G, R, n_sess, nb_max, n_split;
  int64_t nb_total;
  float zscale;  // log2(e)/sqrt(D)
};


struct SmemLayout {
  // qT[D][RP] | mkT[D][kCH+1] | S[RP][kCH+1]
  int RP;
  __host__ __device__ size_t qT_floats(int D) const { return (size_t)D * RP; }
  __host__ __device__ size_t mk_floats(int D) const { return (size_t)D * (kCH + 1); }
  __host__ __device__ size_t s_floats() const { return (size_t)RP * (kCH + 1); }
  __host__ __device__ size_t bytes(int D) const {
    return 4 * (qT_floats(D) + mk_floats(D) + s_floats());
  }
};

// Unit u → (l, h, r), r fastest.
__device__ __forceinline__ void unit_coords(const ScoreArgs &a, int u, int &l,
                                            int &h, int &r) {
  r = u % a.n_sess;
  int lh = u / a.n_sess;
  h = lh % a.H;
  l = lh / a.H;
}

// Validates the session's block range; returns false (and records) if bad.
__device__ __forceinline__ bool session_range(const ScoreArgs &a, int r,
                                              int64_t &b0, int &nb) {
  b0 = a.blk_off[r];
  int64_t b1 = a.blk_off[r + 1];
  if (b0 < 0 || b1 <= b0 || b1 > a.nb_total || b1 - b0 > a.nb_max) {
    record_error(a.status, KVC_ERR_BOUNDS);
    return false;
  }
  nb = (int)(b1 - b0);
  return true;
}

// Stage the unit's R query rows transposed (fp32, zero rows past R).
__device__ void stage_q(const ScoreArgs &a, float *qT, int RP, int l, int h,
                        int r) {
  const uint16_t *src =
      a.q + ((((int64_t)l * a.n_sess + r) * a.Hq + (int64_t)h * a.G) * a.W) * a.D;
  int n = RP * a.D;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    int row = i / a.D, d = i - row * a.D;
    float v = 0.f;
    if (row < a.R) v = __uint_as_float((uint32_t)src[(int64_t)row * a.D + d] << 16);
    qT[d * RP + row] = v;
  }
}

// Stage Mean-K blocks [c0, c0+kCH) of the unit transposed (zeros past nb).
__device__ void stage_mk(const ScoreArgs &a, float *mkT, const uint16_t *mk_unit,
                         int c0, int nb) {
  int n = kCH * a.D;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    int b = i / a.D, d = i - b * a.D;
    float v = 0.f;
    if (c0 + b < nb) v = __uint_as_float((uint32_t)mk_unit[(int64_t)(c0 + b) * a.D + d] << 16);
    mkT[d * (kCH + 1) + b] = v;
  }
}

// S[row][b] = z₂ of the R×kCH tile (thread: RPG rows × 8 blocks).
template <int RPG>
__device__ void logit_tile(const ScoreArgs &a, const float *qT,
                           const float *mkT, float *S, int RP) {
  int bg = threadIdx.x & 7, rg = threadIdx.x >> 3;
  float acc[RPG][8];
#pragma unroll
  for (int i = 0; i < RPG; i++)
#pragma unroll
    for (int k = 0; k < 8; k++) acc[i][k] = 0.f;
  for (int d = 0; d < a.D; d++) {
    float qv[RPG], mv[8];
#pragma unroll
    for (int i = 0; i < RPG; i++) qv[i] = qT[d * RP + rg * RPG + i];
#pragma unroll
    for (int k = 0; k < 8; k++) mv[k] = mkT[d * (kCH + 1) + bg + 8 * k];
#pragma unroll
    for (int i = 0; i < RPG; i++)
#pragma unroll
      for (int k = 0; k < 8; k++) acc[i][k] = fmaf(qv[i], mv[k], acc[i][k]);
  }
#pragma unroll
  for (int i = 0; i < RPG; i++)
#pragma unroll
    for (int k = 0; k < 8; k++)
      S[(rg * RPG + i) * (kCH + 1) + bg + 8 * k] = acc[i][k] * a.zscale;
}

template <int RPG>
__global__ void __launch_bounds__(kThreads)
k_score_pass1(ScoreArgs a) {
  extern __shared__ float smem[];
  const int RP = 32 * RPG;
  SmemLayout lay{RP};
  float *qT = smem;
  float *mkT = qT + lay.qT_floats(a.D);
  float *S = mkT + lay.mk_floats(a.D);
  int u = blockIdx.y, split = blockIdx.x;
  int l, h, r;
  unit_coords(a, u, l, h, r);
  int64_t b0;
  int nb;
  if (!session_range(a, r, b0, nb)) return;
  int n_chunks = (nb + kCH - 1) / kCH;
  int per = (n_chunks + a.n_split - 1) / a.n_split;
  int c_begin = split * per, c_end = min(n_chunks, c_begin + per);
  const uint16_t *mk_unit = a.meank + (((int64_t)l * a.H + h) * a.nb_total + b0) * a.D;
  stage_q(a, qT, RP, l, h, r);
  float run_m = -INFINITY, run_s = 0.f;  // thread row = threadIdx.x (< R)
  for (int c = c_begin; c < c_end; c++) {
    __syncthreads();
    stage_mk(a, mkT, mk_unit, c * kCH, nb);
    __syncthreads();
    logit_tile<RPG>(a, qT, mkT, S, RP);
    __syncthreads();
    if (threadIdx.x < a.R) {
      int valid = min(kCH, nb - c * kCH);
      const float *row = S + threadIdx.x * (kCH + 1);
      float m = run_m;
      for (int b = 0; b < valid; b++) m = fmaxf(m, row[b]);
      float s = run_s * exp2f(run_m - m);
      for (int b = 0; b < valid; b++) s += exp2f(row[b] - m);
      run_m = m;
      run_s = s;
    }
  }
  if (threadIdx.x < a.R)
    a.part[((int64_t)u * a.n_split + split) * a.R + threadIdx.x] =
        make_float2(run_m, run_s);
}

template <int RPG>
__global__ void __launch_bounds__(kThreads)
k_score_pass2(ScoreArgs a) {
  extern __shared__ float smem[];
  const int RP = 32 * RPG;
  SmemLayout lay{RP};
  float *qT = smem;
  float *mkT = qT + lay.qT_floats(a.D);
  float *S = mkT + lay.mk_floats(a.D);
  __shared__ float lse[32 * 8];
  float *red = mkT;  // Mean-K tile is dead once the logits are in S
  int u = blockIdx.y, c = blockIdx.x;
  int l, h, r;
  unit_coords(a, u, l, h, r);
  int64_t b0;
  int nb;
  if (!session_range(a, r, b0, nb)) return;
  if (c * kCH >= nb) return;
  const uint16_t *mk_unit = a.meank + (((int64_t)l * a.H + h) * a.nb_total + b0) * a.D;
  if (threadIdx.x < a.R) {
    const float2 *p = a.part + (int64_t)u * a.n_split * a.R + threadIdx.x;
    float m = -INFINITY;
    for (int s = 0; s < a.n_split; s++) m = fmaxf(m, p[(int64_t)s * a.R].x);
    float sum = 0.f;
    for (int s = 0; s < a.n_split; s++) {
      float2 v = p[(int64_t)s * a.R];
      if (v.y > 0.f) sum += v.y * exp2f(v.x - m);
    }
    lse[threadIdx.x] = m + log2f(sum);
  }
  stage_q(a, qT, RP, l, h, r);
  stage_mk(a, mkT, mk_unit, c * kCH, nb);
  __syncthreads();
  logit_tile<RPG>(a, qT, mkT, S, RP);
  __syncthreads();
  // thread → (block b, quarter of the window)
  int b = threadIdx.x % kCH, part = threadIdx.x / kCH;
  int wq = (a.W + 3) / 4;
  float acc = 0.f;
  for (int w = part * wq; w < min(a.W, (part + 1) * wq); w++) {
    float t = -INFINITY;
    for (int g = 0; g < a.G; g++) {
      int row = g * a.W + w;
      t = fmaxf(t, S[row * (kCH + 1) + b] - lse[row]);
    }
    acc += exp2f(t);
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  if (part == 0 && c * kCH + b < nb) {
    float s = red[b] + red[b + kCH] + red[b + 2 * kCH] + red[b + 3 * kCH];
    a.scores[((int64_t)l * a.H + h) * a.nb_total + b0 + c * kCH + b] =
        s / (float)a.W;
  }
}

int rows_per_group(int R) {
  int rpg = 1;
  while (32 * rpg < R) rpg *= 2;
  return rpg;
}

int pick_split(int n_units, int nb_max) {
  int n_chunks = (nb_max + kCH - 1) / kCH;
  int s = (2 * 152 + n_units - 1) / n_units;
  s = s < 1 ? 1 : (s > kMaxSplit ? kMaxSplit : s);
  return s > n_chunks ? n_chunks : s;
}

template <int RPG>
cudaError_t launch_rpg(const ScoreArgs &a, int n_units, cudaStream_t s) {
  SmemLayout lay{32 * RPG};
  size_t smem = lay.bytes(a.D);
  cudaError_t e;
  e = cudaFuncSetAttribute(k_score_pass1<RPG>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_score_pass2<RPG>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 g1(a.n_split, n_units);
  k_score_pass1<RPG><<<g1, kThreads, smem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2((a.nb_max + kCH - 1) / kCH, n_units);
  k_score_pass2<RPG><<<g2, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t score_meank_ws_bytes(int L, int H, int Hq, int W, int n_sess,
                            int nb_max, int64_t nb_total) {
  int n_units = L * H * n_sess;
  int R = (Hq / H) * W;
  int split = pick_split(n_units, nb_max);
  size_t cc = (size_t)n_units * split * R * sizeof(float2);
  size_t tc = score_tc_ws_bytes(L, H, Hq, W, n_sess, nb_max, nb_total);
  return cc > tc ? cc : tc;
}

// Which scorer runs: by default (KVC_KERNEL_AUTO) the tensor-core one
// whenever it covers the shape, else the CUDA-core one; `path` may name one
// kernel (both kinds compute the same scores within the stated bound).
int score_meank_launches(int H, int Hq, int D, int W, int n_sess, int nb_max) {
  int R = (Hq / H) * W;
  if (score_tc_supported(R, W, D)) {
    int n = score_tc_launches(R, W, D, n_sess, nb_max);
    if (n > 0) return n;
  }
  return 2;
}

cudaError_t launch_score_meank(const uint16_t *q, const uint16_t *meank,
                               float *scores, int L, int H, int Hq, int D,
                               int W, const int64_t *blk_off, int n_sess,
                               int64_t nb_total, int nb_max, void *ws,
                               int32_t *status, int path, cudaStream_t s) {
  if (path != KVC_KERNEL_SCORE_CC) {
    const bool tc = score_tc_supported((Hq / H) * W, W, D);
    if (!tc && path != KVC_KERNEL_AUTO) return cudaErrorNotSupported;
    if (tc) {
      cudaError_t e = launch_score_tc(q, meank, scores, L, H, Hq, D, W, blk_off, n_sess,
                                      nb_total, nb_max, ws, status, path, s);
      if (path != KVC_KERNEL_AUTO || e != cudaErrorNotSupported) return e;
    }
  }
  ScoreArgs a;
  a.q = q;
  a.meank = meank;
  a.scores = scores;
  a.blk_off = blk_off;
  a.part = reinterpret_cast<float2 *>(ws);
  a.status = status;
  a.L = L;
  a.H = H;
  a.Hq = Hq;
  a.D = D;
  a.W = W;
  a.G = Hq / H;
  a.R = a.G * W;
  a.n_sess = n_sess;
  a.nb_max = nb_max;
  a.nb_total = nb_total;
  a.zscale = kLog2e / sqrtf((float)D);
  int n_units = L * H * n_sess;
  a.n_split = pick_split(n_units, nb_max);
  switch (rows_per_group(a.R)) {
    case 1: return launch_rpg<1>(a, n_units, s);
    case 2: return launch_rpg<2>(a, n_units, s);
    case 4: return launch_rpg<4>(a, n_units, s);
    default: return launch_rpg<8>(a, n_units, s);
  }
}

}  // namespace kvc
