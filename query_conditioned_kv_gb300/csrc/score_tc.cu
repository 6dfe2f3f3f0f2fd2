// score_tc.cu — Mean-K block scoring on the 5th-generation tensor cores.
//
// Same quantity as the CUDA-core scorer (KVMem "Query-conditioned
// retrieval"; ActKV §7.1 aggregation): for one unit (layer l, KV head h,
// session r) with query rows ρ = g·W + w,
//   z[ρ,b] = q[ρ]·meank[b]/sqrt(D),  LSE[ρ] = log Σ_b e^z,
//   score[b] = (1/W) Σ_w max_g exp(z[g·W+w,b] − LSE[g·W+w]).
//
// Work item = (unit, chunk of CH = S·128 consecutive blocks).  A CTA brings
// the chunk's Mean-K (CH × D bf16) and the unit's query rows into shared
// memory with TMA (128-byte swizzle = the UMMA K-major layout); they stay
// there for both passes, so Mean-K is read from HBM once.  Both logit
// products are tcgen05.mma (bf16 × bf16 → fp32 in TMEM) issued by one thread:
//   pass 1  D[ρ][b] (M = 128 query rows, N = 128 blocks): each epilogue
//           thread owns one query row (one TMEM lane) and keeps an online
//           (max, Σ2^(z−max)) over the chunk;
//   LSE     the chunk partials of a unit are combined through L2: every
//           item publishes its partials and bumps the unit's counter, then
//           waits (bounded) until all of the unit's chunks have published;
//   pass 2  D[b][ρ] (operands swapped: M = 128 blocks, N = R query rows):
//           each thread owns one block and forms max over g and the mean
//           over w of 2^(z−LSE) from its own TMEM lane — W exponentials per
//           block, no cross-lane traffic.
//
// Persistent kernel: two CTAs per SM (≤ 256 TMEM columns, ≈ 100 KB shared
// memory each), items claimed in order from an atomic counter.  A claimed
// item is always held by a running CTA and pass 1 waits on nothing, so the
// only CTAs that can wait are those of the last, partially claimed unit; as
// long as a unit has no more chunks than CTAs fit on the GPU, every wait
// ends.  Longer units use the two-launch split mode (pass 1 → partials in
// global memory → pass 2, Mean-K read twice).
//
// Warp roles: warps 0–3 read TMEM (warp i owns lanes 32i…32i+31), warp 4
// issues TMA and MMA.  Every wait is bounded; on a timeout the CTA records
// KVC_ERR_TIMEOUT, stops claiming work, waits (bounded) for its own copies
// and MMAs and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "kvc_internal.cuh"
#include "tc_ptx.cuh"

namespace kvc {
namespace {

using namespace tc;

constexpr int kEpiThreads = 128;
constexpr int kThreadsTC = kEpiThreads + 32;
constexpr uint32_t kTmemCols = 256;  // two CTAs share an SM's 512 columns
constexpr float kLog2eTC = 1.4426950408889634f;
constexpr uint32_t kWaitLimit = 1u << 24;  // ≈ 1–2 s with the back-off below
constexpr int kMaxSessPersist = 2048;      // per-session chunk prefix in smem

enum Mode { kPass1 = 1, kPass2 = 2 };

struct TcArgs {
  float *scores;
  const int64_t *blk_off;
  float2 *part;    // persistent: [item][RT·128]; split: [unit][chunk][RT·128]
  int *counter;    // persistent: next item
  int *unit_done;  // persistent: [n_units] chunks published
  int32_t *status;
  int L, H, Hq, W, G, R, D, n_sess, n_chunk;
  int64_t nb_total;
  float zscale;
  uint32_t idesc1, idesc2;
  int n2;   // pass-2 N (R rounded up to 16)
  int n2c;  // pass-2 TMEM column stride per sub-tile (n2 rounded up to 32)
};

// ------------------------------------------------------------ PTX helpers

// Bounded wait for the completion of the phase with parity `parity`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; i++) {
    if (mbar_try(bar, parity)) return true;
    if (i > 64) __nanosleep(64);
  }
  return false;
}

__device__ __forceinline__ void named_sync_epi() {
  asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// (max, sum) ⊕ (max, sum) in base 2.
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  float mn = fmaxf(m, m2);
  s = s * exp2f(m - mn) + s2 * exp2f(m2 - mn);
  m = mn;
}

// LSE (base 2) of one query row from its per-chunk partials p[c·stride],
// c < n; loads are issued 16 at a time so their L2 latencies overlap.
__device__ __forceinline__ float combine_partials(const float2 *p, int n, int stride) {
  float m = -INFINITY, s = 0.f;
  for (int c0 = 0; c0 < n; c0 += 16) {
    float2 v[16];
#pragma unroll
    for (int k = 0; k < 16; k++)
      v[k] = c0 + k < n ? __ldcg(p + (int64_t)(c0 + k) * stride) : make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int k = 0; k < 16; k++) lse_merge(m, s, v[k].x, v[k].y);
  }
  return (m == -INFINITY) ? INFINITY : m + log2f(s);
}

// ------------------------------------------------------------ the stages

// Shared memory of a CTA: [mk: S·KB boxes of 128 rows × 128 B][q: KB boxes
// of RT·128 rows × 128 B][barriers][tmem holder, flags][lse][prefix]
template <int RT, int S>
struct Smem {
  uint8_t *mk, *q;
  uint64_t *bars;  // 0 tma, 1 mma1, 2 mma2, 3 tmem_free
  uint32_t *tmem_holder;
  volatile int *flags;  // [0] failed, [1] claimed item
  float *lse;
  int *prefix;
  __device__ Smem(uint8_t *raw, int KB) {
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    mk = base;
    q = mk + S * KB * 16384;
    bars = reinterpret_cast<uint64_t *>(q + KB * RT * 16384);
    tmem_holder = reinterpret_cast<uint32_t *>(bars + 4);
    flags = reinterpret_cast<volatile int *>(tmem_holder + 1);
    lse = reinterpret_cast<float *>(tmem_holder + 8);
    prefix = reinterpret_cast<int *>(lse + 256);
  }
  static size_t bytes(int D, int n_prefix) {
    int KB = D / 64;
    return 1024 + (size_t)S * KB * 16384 + (size_t)KB * RT * 16384 + 4 * 8 + 8 * 4 + 256 * 4 +
           (size_t)n_prefix * 4;
  }
};

template <int RT, int S>
__device__ __forceinline__ void issue_loads(const CUtensorMap *tm_q, const CUtensorMap *tm_mk,
                                            const Smem<RT, S> &sm, int KB, int q_row0,
                                            int mk_row0, uint32_t bar) {
  mbar_expect_tx(bar, (uint32_t)(KB * RT * 16384 + S * KB * 16384));
  for (int kb = 0; kb < KB; kb++)
    tma_load_2d(smem_u32(sm.q + kb * RT * 16384), tm_q, kb * 64, q_row0, bar);
  for (int s = 0; s < S; s++)
    for (int kb = 0; kb < KB; kb++)
      tma_load_2d(smem_u32(sm.mk + (s * KB + kb) * 16384), tm_mk, kb * 64, mk_row0 + s * 128, bar);
}

// pass 1: D[ρ][b] = Q · Mean-Kᵀ into TMEM columns (rt·S + s)·128
template <int RT, int S>
__device__ __forceinline__ void issue_pass1(uint32_t tmem, const Smem<RT, S> &sm, int KB,
                                            uint32_t idesc) {
  for (int s = 0; s < S; s++)
    for (int rt = 0; rt < RT; rt++)
      for (int kk = 0; kk < 4 * KB; kk++) {
        const uint32_t koff = (uint32_t)(kk & 3) * 32u;
        uint64_t a = smem_desc(smem_u32(sm.q + (kk >> 2) * RT * 16384 + rt * 16384) + koff);
        uint64_t b = smem_desc(smem_u32(sm.mk + (s * KB + (kk >> 2)) * 16384) + koff);
        mma_bf16(tmem + (uint32_t)((rt * S + s) * 128), a, b, idesc, kk > 0);
      }
}

// pass 2: D[b][ρ] = Mean-K · Qᵀ into TMEM columns s·n2c
template <int RT, int S>
__device__ __forceinline__ void issue_pass2(uint32_t tmem, const Smem<RT, S> &sm, int KB,
                                            uint32_t idesc, int n2c) {
  for (int s = 0; s < S; s++)
    for (int kk = 0; kk < 4 * KB; kk++) {
      const uint32_t koff = (uint32_t)(kk & 3) * 32u;
      uint64_t a = smem_desc(smem_u32(sm.mk + (s * KB + (kk >> 2)) * 16384) + koff);
      uint64_t b = smem_desc(smem_u32(sm.q + (kk >> 2) * RT * 16384) + koff);
      mma_bf16(tmem + (uint32_t)(s * n2c), a, b, idesc, kk > 0);
    }
}

// Pass-1 epilogue: online (max, Σ2^(z−max)) of this thread's query row(s)
// over the item's `valid` blocks (base 2, z₂ = raw · zs).
template <int RT, int S>
__device__ __forceinline__ void epi_pass1(uint32_t tmem, uint32_t lane_base, int valid, float zs,
                                          float (&pm)[RT], float (&ps)[RT]) {
#pragma unroll
  for (int rt = 0; rt < RT; rt++) {
    pm[rt] = -INFINITY;
    ps[rt] = 0.f;
  }
  for (int s = 0; s < S; s++)
#pragma unroll
    for (int rt = 0; rt < RT; rt++)
      for (int c = 0; c < 4; c++) {
        const int col0 = s * 128 + 32 * c;
        const int nv = min(32, valid - col0);
        if (nv <= 0) continue;  // warp-uniform
        float v[32];
        tmem_ld32(tmem + lane_base + (uint32_t)((rt * S + s) * 128 + 32 * c), v);
        if (nv < 32) {
#pragma unroll
          for (int j = 0; j < 32; j++)
            if (j >= nv) v[j] = -INFINITY;
        }
        // max of the raw products (zs > 0), then 2^(v·zs − max) by FFMA
        float m01 = fmaxf(v[0], v[1]), m23 = fmaxf(v[2], v[3]);
#pragma unroll
        for (int j = 4; j < 32; j += 4) {
          m01 = fmaxf(m01, fmaxf(v[j], v[j + 1]));
          m23 = fmaxf(m23, fmaxf(v[j + 2], v[j + 3]));
        }
        const float mn = fmaxf(pm[rt], fmaxf(m01, m23) * zs);
        float a0 = (pm[rt] == -INFINITY) ? 0.f : ps[rt] * exp2f(pm[rt] - mn);
        float a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          a0 += exp2f(fmaf(v[j], zs, -mn));
          a1 += exp2f(fmaf(v[j + 1], zs, -mn));
          a2 += exp2f(fmaf(v[j + 2], zs, -mn));
          a3 += exp2f(fmaf(v[j + 3], zs, -mn));
        }
        pm[rt] = mn;
        ps[rt] = (a0 + a1) + (a2 + a3);
      }
}

// Pass-2 epilogue: thread = block; writes the item's block scores.
template <int S, int W>
__device__ __forceinline__ void epi_pass2(uint32_t tmem, uint32_t lane_base, int warp, int lane,
                                          int valid, int n2c, int R, float zs, float invW,
                                          const float *lse, float *out) {
  for (int s = 0; s < S; s++) {
    if (s * 128 >= valid) break;  // uniform
    float mw[W];
#pragma unroll
    for (int w = 0; w < W; w++) mw[w] = -INFINITY;
    for (int c = 0; c < n2c / 32; c++) {
      float v[32];
      tmem_ld32(tmem + lane_base + (uint32_t)(s * n2c + 32 * c), v);
#pragma unroll
      for (int j = 0; j < 32; j++) {
        const int rho = 32 * c + j;
        if (rho < R) mw[j % W] = fmaxf(mw[j % W], fmaf(v[j], zs, -lse[rho]));
      }
    }
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < W; w++) acc += exp2f(mw[w]);
    const int bl = s * 128 + warp * 32 + lane;
    if (bl < valid) out[bl] = acc * invW;
  }
}

__device__ __forceinline__ void alloc_tmem(uint32_t *holder) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(holder)),
               "r"(kTmemCols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}

__device__ __forceinline__ void free_tmem(uint32_t tmem) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
               "r"(kTmemCols));
}

// ------------------------------------------------------ persistent kernel

template <int RT, int S, int W>
__global__ void __launch_bounds__(kThreadsTC, 1)
k_score_tc(const __grid_constant__ CUtensorMap tm_mk, const __grid_constant__ CUtensorMap tm_q,
           TcArgs a) {
  static_assert(W == 8 || W == 16 || W == 32, "W divides 32");
  extern __shared__ uint8_t smem_raw[];
  const int KB = a.D / 64;
  Smem<RT, S> sm(smem_raw, KB);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CH = S * 128;
  const uint32_t bar0 = smem_u32(sm.bars);
  const uint32_t BAR_TMA = bar0, BAR_MMA1 = bar0 + 8, BAR_MMA2 = bar0 + 16, BAR_FREE = bar0 + 24;

  // per-session chunk counts → prefix (items of one (layer, KV head))
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < a.n_sess; base += 32) {
      int r = base + lane, cnt = 0;
      if (r < a.n_sess) {
        int64_t b0 = a.blk_off[r], b1 = a.blk_off[r + 1];
        if (b0 >= 0 && b1 > b0 && b1 <= a.nb_total && b1 - b0 <= (int64_t)a.n_chunk * CH)
          cnt = (int)((b1 - b0 + CH - 1) / CH);
        else if (blockIdx.x == 0)
          record_error(a.status, KVC_ERR_BOUNDS);
      }
      int x = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      if (r < a.n_sess) sm.prefix[r] = carry + x - cnt;
      carry += __shfl_sync(0xFFFFFFFFu, x, 31);
    }
    if (lane == 0) sm.prefix[a.n_sess] = carry;
  }
  if (threadIdx.x == 0) {
    sm.flags[0] = 0;
    mbar_init(BAR_TMA, 1);
    mbar_init(BAR_MMA1, 1);
    mbar_init(BAR_MMA2, 1);
    mbar_init(BAR_FREE, 4);  // one arrive per epilogue warp
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) alloc_tmem(sm.tmem_holder);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_holder;
  const int per_lh = sm.prefix[a.n_sess];
  const int total = a.L * a.H * per_lh;
  const float zs = a.zscale, invW = 1.f / (float)a.W;
  bool committed = false;

  for (uint32_t iter = 0;; iter++) {
    if (threadIdx.x == kEpiThreads) sm.flags[1] = atomicAdd(a.counter, 1);
    __syncthreads();
    const int item = sm.flags[1];
    if (item >= total || sm.flags[0] != 0) break;  // CTA-uniform
    const uint32_t ph = iter & 1u;
    // item → (layer, head, session, chunk)
    const int lh = item / per_lh, rem = item - lh * per_lh;
    int lo = 0, hi = a.n_sess - 1;  // last r with prefix[r] <= rem
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (sm.prefix[mid] <= rem)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int r = lo, chunk = rem - sm.prefix[r];
    const int n_chunks = sm.prefix[r + 1] - sm.prefix[r];
    const int h = lh % a.H, l = lh / a.H;
    const int unit = lh * a.n_sess + r;
    const int64_t b0 = a.blk_off[r];
    const int nb = (int)(a.blk_off[r + 1] - b0);
    const int valid = min(CH, nb - chunk * CH);
    const int mk_row0 = (int)(((int64_t)l * a.H + h) * a.nb_total + b0 + (int64_t)chunk * CH);
    const int q_row0 = (int)((((int64_t)l * a.n_sess + r) * a.Hq + (int64_t)h * a.G) * a.W);

    if (warp == 4) {
      if (lane == 0) {
        issue_loads<RT, S>(&tm_q, &tm_mk, sm, KB, q_row0, mk_row0, BAR_TMA);
        bool ok = mbar_wait(BAR_TMA, ph);
        if (ok) {
          tc_fence_after();
          issue_pass1<RT, S>(tmem, sm, KB, a.idesc1);
          mma_commit(BAR_MMA1);
          committed = true;
          ok = mbar_wait(BAR_FREE, ph);  // pass-1 TMEM reads done
        }
        if (ok) {
          tc_fence_after();
          issue_pass2<RT, S>(tmem, sm, KB, a.idesc2, a.n2c);
          mma_commit(BAR_MMA2);
        } else {
          sm.flags[0] = 1;
          record_error(a.status, KVC_ERR_TIMEOUT);
        }
      }
      __syncwarp();
    } else {
      const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
      float pm[RT], ps[RT];
      bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(BAR_MMA1, ph));
      if (ok) {
        tc_fence_after();
        epi_pass1<RT, S>(tmem, lane_base, valid, zs, pm, ps);
      } else {
#pragma unroll
        for (int rt = 0; rt < RT; rt++) {
          pm[rt] = -INFINITY;
          ps[rt] = 0.f;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_FREE);
      // publish this chunk's partials, then wait for the unit's other chunks
      float2 *mine = a.part + (int64_t)item * (RT * 128);
#pragma unroll
      for (int rt = 0; rt < RT; rt++) mine[rt * 128 + threadIdx.x] = make_float2(pm[rt], ps[rt]);
      __threadfence();
      named_sync_epi();
      if (threadIdx.x == 0) {
        atomicAdd(&a.unit_done[unit], 1);
        uint32_t i = 0;
        while (ld_acquire(&a.unit_done[unit]) < n_chunks && ++i < kWaitLimit)
          if (i > 32) __nanosleep(128);
        if (i >= kWaitLimit) {
          sm.flags[0] = 1;
          record_error(a.status, KVC_ERR_TIMEOUT);
        }
      }
      named_sync_epi();
      __threadfence();
      if (!ok) {
        sm.flags[0] = 1;
        if (lane == 0) record_error(a.status, KVC_ERR_TIMEOUT);
      }
      // LSE of every query row (thread t: rows t and t + 128)
      const float2 *unit_part = a.part + (int64_t)(item - chunk) * (RT * 128);
      for (int rr = threadIdx.x; rr < RT * 128; rr += kEpiThreads)
        sm.lse[rr] = combine_partials(unit_part + rr, n_chunks, RT * 128);
      named_sync_epi();
      bool ok2 = __all_sync(0xFFFFFFFFu, ok && mbar_wait(BAR_MMA2, ph));
      if (ok2) {
        tc_fence_after();
        float *out = a.scores + ((int64_t)l * a.H + h) * a.nb_total + b0 + (int64_t)chunk * CH;
        epi_pass2<S, W>(tmem, lane_base, warp, lane, valid, a.n2c, a.R, zs, invW, sm.lse, out);
      } else {
        sm.flags[0] = 1;
      }
      tc_fence_before();
    }
    __syncthreads();  // item done: TMEM and shared memory are free again
    tc_fence_after();
  }

  // teardown
  if (warp == 4 && lane == 0 && committed && sm.flags[0] != 0) {
    // a wait gave up: let this CTA's own copies and MMAs drain (bounded)
    mbar_wait(BAR_TMA, 0);
    mbar_wait(BAR_TMA, 1);
    mbar_wait(BAR_MMA1, 0);
    mbar_wait(BAR_MMA2, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    free_tmem(tmem);
  }
}

// --------------------------------------------------- split-mode kernels

// One item per CTA (grid: chunk × unit).  kPass1 publishes the chunk's
// partials to global memory; kPass2 (a second launch) combines them, reloads
// the chunk and writes its scores.
template <int MODE, int RT, int S, int W>
__global__ void __launch_bounds__(kThreadsTC, 1)
k_score_split(const __grid_constant__ CUtensorMap tm_mk, const __grid_constant__ CUtensorMap tm_q,
              TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int KB = a.D / 64;
  Smem<RT, S> sm(smem_raw, KB);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CH = S * 128;
  const int chunk = blockIdx.x, unit = blockIdx.y;
  const int r = unit % a.n_sess, lh = unit / a.n_sess;
  const int h = lh % a.H, l = lh / a.H;
  const int64_t b0 = a.blk_off[r], b1 = a.blk_off[r + 1];
  if (!(b0 >= 0 && b1 > b0 && b1 <= a.nb_total)) {
    if (chunk == 0 && threadIdx.x == 0) record_error(a.status, KVC_ERR_BOUNDS);
    return;
  }
  const int nb = (int)(b1 - b0);
  const int valid = min(CH, nb - chunk * CH);
  if (valid <= 0) return;  // CTA-uniform, before any barrier
  const int n_chunks = (nb + CH - 1) / CH;
  const int mk_row0 = (int)(((int64_t)l * a.H + h) * a.nb_total + b0 + (int64_t)chunk * CH);
  const int q_row0 = (int)((((int64_t)l * a.n_sess + r) * a.Hq + (int64_t)h * a.G) * a.W);
  const uint32_t bar0 = smem_u32(sm.bars);
  const uint32_t BAR_TMA = bar0, BAR_MMA = bar0 + 8;
  if (threadIdx.x == 0) {
    sm.flags[0] = 0;
    mbar_init(BAR_TMA, 1);
    mbar_init(BAR_MMA, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) alloc_tmem(sm.tmem_holder);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_holder;
  const float zs = a.zscale;
  bool committed = false;

  if (warp == 4) {
    if (lane == 0) {
      issue_loads<RT, S>(&tm_q, &tm_mk, sm, KB, q_row0, mk_row0, BAR_TMA);
      if (mbar_wait(BAR_TMA, 0)) {
        tc_fence_after();
        if (MODE == kPass1)
          issue_pass1<RT, S>(tmem, sm, KB, a.idesc1);
        else
          issue_pass2<RT, S>(tmem, sm, KB, a.idesc2, a.n2c);
        mma_commit(BAR_MMA);
        committed = true;
      } else {
        sm.flags[0] = 1;
        record_error(a.status, KVC_ERR_TIMEOUT);
      }
    }
    __syncwarp();
  } else {
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    if (MODE == kPass2) {
      const float2 *unit_part = a.part + (int64_t)unit * a.n_chunk * (RT * 128);
      for (int rr = threadIdx.x; rr < RT * 128; rr += kEpiThreads)
        sm.lse[rr] = combine_partials(unit_part + rr, n_chunks, RT * 128);
      named_sync_epi();
    }
    bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(BAR_MMA, 0));
    if (ok) {
      tc_fence_after();
      if (MODE == kPass1) {
        float pm[RT], ps[RT];
        epi_pass1<RT, S>(tmem, lane_base, valid, zs, pm, ps);
        float2 *dst = a.part + ((int64_t)unit * a.n_chunk + chunk) * (RT * 128);
#pragma unroll
        for (int rt = 0; rt < RT; rt++) dst[rt * 128 + threadIdx.x] = make_float2(pm[rt], ps[rt]);
      } else {
        float *out = a.scores + ((int64_t)l * a.H + h) * a.nb_total + b0 + (int64_t)chunk * CH;
        epi_pass2<S, W>(tmem, lane_base, warp, lane, valid, a.n2c, a.R, zs, 1.f / (float)a.W,
                        sm.lse, out);
      }
    } else {
      sm.flags[0] = 1;
      if (lane == 0) record_error(a.status, KVC_ERR_TIMEOUT);
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 4 && lane == 0 && committed && sm.flags[0] != 0) mbar_wait(BAR_MMA, 0);
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    free_tmem(tmem);
  }
}

// ------------------------------------------------ pipelined cluster kernel
//
// k_score_ring: a cluster of C CTAs (C ≤ 4) owns one unit at a time and
// walks the units round-robin; CTA `rank` of the cluster takes the unit's
// 128-block tiles rank, rank + C, …  Roles inside a CTA:
//   warp 0      TMA producer: the unit's query rows (double-buffered), then
//               its tiles twice (pass 1, pass 2) through an NS-stage ring;
//   warp 1      MMA issuer: per tile, pass-1 or pass-2 tcgen05.mma into one
//               of NBUF TMEM accumulators;
//   warps 2…     epilogue warpgroups (three, or two for > 128 query rows)
//               taking tiles round-robin: pass-1 online row LSE, then
//               (after the exchange) pass-2 scores.
// Between a unit's two passes the CTAs exchange their row partials through
// distributed shared memory: every CTA stores its partials into each peer's
// receive slot and arrives on the peer's mbarrier (release at cluster
// scope); no full-cluster barrier stalls the producer or the MMA warp, which
// keep prefetching the pass-2 tiles.  The second read of a tile usually hits
// L2 (a CTA's share of a unit is ≤ 1/C of its Mean-K).

constexpr int kRingMaxC = 4;
// Epilogue warpgroups: three for ≤ 128 query rows (4 TMEM accumulators of
// 128 columns), two for up to 256 rows (2 accumulators of 256 columns); two
// more warps produce and issue.  Three groups keep ≤ 4 warps per SM
// sub-partition, so each thread can hold 128 registers without spilling.
template <int RT> constexpr int ring_groups() { return RT == 1 ? 3 : 2; }
template <int RT> constexpr int ring_threads() { return 64 + 128 * ring_groups<RT>(); }

template <int RT>
struct RingSmem {
  // Ring depth: the loaded latency of a 32 KB tile is ≈ 3 µs, so the ring
  // holds as many tiles as shared memory allows next to two query buffers.
  // The second query buffer lets the producer move on to the next unit's
  // rows and tiles while this unit's last MMAs and epilogues finish, so the
  // ring does not drain at unit boundaries.
  static constexpr int NS = RT == 1 ? 4 : 2;    // Mean-K ring stages
  static constexpr int QB = 2;                  // query-row buffers
  static constexpr int ROWS = 128 * RT;         // query rows (padded)
  static constexpr int NBUF = RT == 1 ? 4 : 2;  // TMEM accumulators
  static constexpr int NEG = ring_groups<RT>();  // epilogue warpgroups
  static constexpr int BUFCOLS = 128 * RT;      // columns per accumulator
  uint8_t *ring, *q;
  uint64_t *full, *empty, *tfull, *tempty, *qfull, *qempty, *recv;
  uint32_t *tmem_holder;
  volatile int *failed;
  float2 *egpart;  // [NEG groups][ROWS]
  float2 *rbuf;    // [2 parities][kRingMaxC ranks][ROWS]
  float *lse;      // [ROWS]
  __device__ RingSmem(uint8_t *raw, int KB) {
    uint8_t *p = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    ring = p;
    p += NS * KB * 16384;
    q = p;
    p += QB * KB * RT * 16384;
    uint64_t *b = reinterpret_cast<uint64_t *>(p);
    full = b;
    empty = full + NS;
    tfull = empty + NS;
    tempty = tfull + NBUF;
    qfull = tempty + NBUF;
    qempty = qfull + 2;
    recv = qempty + 2;
    tmem_holder = reinterpret_cast<uint32_t *>(recv + 2);
    failed = reinterpret_cast<volatile int *>(tmem_holder + 1);
    egpart = reinterpret_cast<float2 *>(tmem_holder + 4);  // 16-byte aligned
    rbuf = egpart + NEG * ROWS;
    lse = reinterpret_cast<float *>(rbuf + 2 * kRingMaxC * ROWS);
  }
  static size_t bytes(int D) {
    int KB = D / 64;
    return 1024 + (size_t)NS * KB * 16384 + (size_t)QB * KB * RT * 16384 +
           (2 * NS + 2 * NBUF + 6) * 8 + 16 + (NEG * ROWS + 2 * kRingMaxC * ROWS) * 8 + ROWS * 4;
  }
};

struct UnitInfo {
  int l, h, r, nb, n_tiles, my_tiles, mk_row0, q_row0;
  int64_t b0;
};

__device__ __forceinline__ UnitInfo unit_info(const TcArgs &a, int unit, int C, int rank) {
  UnitInfo u;
  u.r = unit % a.n_sess;
  const int lh = unit / a.n_sess;
  u.h = lh % a.H;
  u.l = lh / a.H;
  const int64_t b0 = a.blk_off[u.r], b1 = a.blk_off[u.r + 1];
  const bool ok = b0 >= 0 && b1 > b0 && b1 <= a.nb_total && b1 - b0 <= (int64_t)a.n_chunk * 128;
  u.b0 = ok ? b0 : 0;
  u.nb = ok ? (int)(b1 - b0) : 0;
  u.n_tiles = (u.nb + 127) / 128;
  u.my_tiles = u.n_tiles > rank ? (u.n_tiles - rank + C - 1) / C : 0;
  u.mk_row0 = (int)(((int64_t)u.l * a.H + u.h) * a.nb_total + u.b0);
  u.q_row0 = (int)((((int64_t)u.l * a.n_sess + u.r) * a.Hq + (int64_t)u.h * a.G) * a.W);
  return u;
}

// Pass-2 order of a CTA's tiles (local indices).  When the CTA has at least
// NS tiles, the last NS tiles of pass 1 are still in the ring, in the slots
// that pass 2's first NS steps map to (FIFO slot order, NS apart): pass 2
// takes those first, without loading them again, then the rest in order.
template <int NS>
__device__ __forceinline__ int pass2_tile(int j, int my_tiles) {
  if (my_tiles < NS) return j;
  return j < NS ? my_tiles - NS + j : j - NS;
}

// Pass-1 epilogue of one 128-block tile: (max, Σ2^(z−max)) of this lane's
// query row(s), in 32-column chunks whose TMEM loads are double-buffered.
template <int RT>
__device__ __forceinline__ void ring_pass1(uint32_t taddr, int valid, float zs, float (&pm)[RT],
                                           float (&ps)[RT]) {
  constexpr int NCH = 4 * RT;  // (row tile, 32-column chunk)
  const int nvc = (valid + 31) / 32;  // chunks with at least one valid column
  uint32_t r[2][32];
#pragma unroll
  for (int rt = 0; rt < RT; rt++) {
    pm[rt] = -INFINITY;
    ps[rt] = 0.f;
  }
  tmem_issue32(taddr, r[0]);
  tmem_wait32(r[0]);
#pragma unroll
  for (int ch = 0; ch < NCH; ch++) {
    const int rt = ch / 4, c = ch % 4;
    const bool have_next = ch + 1 < NCH && ((ch + 1) % 4) < nvc;
    if (have_next)  // warp-uniform
      tmem_issue32(taddr + (uint32_t)(((ch + 1) / 4) * 128 + 32 * ((ch + 1) % 4)), r[(ch + 1) & 1]);
    if (c < nvc) {
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[ch & 1][j]);
      const int nv = valid - 32 * c;
      if (nv < 32) {
#pragma unroll
        for (int j = 0; j < 32; j++)
          if (j >= nv) v[j] = -INFINITY;
      }
      float m0 = fmaxf(v[0], v[1]), m1 = fmaxf(v[2], v[3]);
#pragma unroll
      for (int j = 4; j < 32; j += 4) {
        m0 = fmaxf(m0, fmaxf(v[j], v[j + 1]));
        m1 = fmaxf(m1, fmaxf(v[j + 2], v[j + 3]));
      }
      const float mn = fmaxf(pm[rt], fmaxf(m0, m1) * zs);
      float acc[8];
      acc[0] = (pm[rt] == -INFINITY) ? 0.f : ps[rt] * ex2(pm[rt] - mn);
#pragma unroll
      for (int k = 1; k < 8; k++) acc[k] = 0.f;
#pragma unroll
      for (int j = 0; j < 32; j++) acc[j & 7] += ex2(fmaf(v[j], zs, -mn));
      pm[rt] = mn;
      ps[rt] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    }
    if (have_next) tmem_wait32(r[(ch + 1) & 1]);
  }
}

// Pass-2 epilogue of one tile: this lane is block `row`; max over g of
// z·zs − LSE (LSE read four at a time), then the mean over w of 2^max.
template <int W>
__device__ __forceinline__ void ring_pass2(uint32_t taddr, int row, int valid, int n2c, int R,
                                           float zs, float invW, const float *lse, float *out) {
  float mw[W];
#pragma unroll
  for (int w = 0; w < W; w++) mw[w] = -INFINITY;
#pragma unroll 1
  for (int c = 0; c < n2c / 32; c++) {
    uint32_t r[32];
    tmem_issue32(taddr + (uint32_t)(32 * c), r);
    tmem_wait32(r);
    if (32 * c + 32 <= R) {
      const float4 *l4 = reinterpret_cast<const float4 *>(lse + 32 * c);
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 L = l4[j / 4];
        mw[(j + 0) % W] = fmaxf(mw[(j + 0) % W], fmaf(__uint_as_float(r[j + 0]), zs, -L.x));
        mw[(j + 1) % W] = fmaxf(mw[(j + 1) % W], fmaf(__uint_as_float(r[j + 1]), zs, -L.y));
        mw[(j + 2) % W] = fmaxf(mw[(j + 2) % W], fmaf(__uint_as_float(r[j + 2]), zs, -L.z));
        mw[(j + 3) % W] = fmaxf(mw[(j + 3) % W], fmaf(__uint_as_float(r[j + 3]), zs, -L.w));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; j++)
        if (32 * c + j < R)
          mw[j % W] = fmaxf(mw[j % W], fmaf(__uint_as_float(r[j]), zs, -lse[32 * c + j]));
    }
  }
  float acc = 0.f;
#pragma unroll
  for (int w = 0; w < W; w++) acc += ex2(mw[w]);
  if (row < valid) out[row] = acc * invW;
}

template <int RT, int W>
__global__ void __launch_bounds__(ring_threads<RT>(), 1)
k_score_ring(const __grid_constant__ CUtensorMap tm_mk, const __grid_constant__ CUtensorMap tm_q,
             TcArgs a) {
  static_assert(W == 8 || W == 16 || W == 32, "W divides 32");
  using SM = RingSmem<RT>;
  constexpr int NS = SM::NS, NBUF = SM::NBUF, BUFCOLS = SM::BUFCOLS;
  extern __shared__ uint8_t smem_raw[];
  const int KB = a.D / 64;
  SM sm(smem_raw, KB);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = (int)cluster_nrank(), rank = (int)cluster_rank();
  const int cluster_id = blockIdx.x / C, n_clusters = gridDim.x / C;
  const int n_units = a.L * a.H * a.n_sess;
  const uint32_t stage_bytes = (uint32_t)KB * 16384u, q_bytes = (uint32_t)(KB * RT) * 16384u;

  if (threadIdx.x == 0) {
    *sm.failed = 0;
    for (int i = 0; i < NS; i++) {
      mbar_init(smem_u32(sm.full + i), 1);
      mbar_init(smem_u32(sm.empty + i), 1);
    }
    for (int i = 0; i < NBUF; i++) {
      mbar_init(smem_u32(sm.tfull + i), 1);
      mbar_init(smem_u32(sm.tempty + i), 4);  // the 4 warps of one epilogue group
    }
    for (int i = 0; i < 2; i++) {
      mbar_init(smem_u32(sm.qfull + i), 1);
      mbar_init(smem_u32(sm.qempty + i), 1);
      mbar_init(smem_u32(sm.recv + i), C > 1 ? C - 1 : 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) alloc_tmem_cols(sm.tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (C > 1) cluster_sync_all();  // peers' barriers exist before any remote arrive
  const uint32_t tmem = *sm.tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t s = 0, qi = 0;
      for (int unit = cluster_id; unit < n_units && !*sm.failed; unit += n_clusters) {
        const UnitInfo u = unit_info(a, unit, C, rank);
        if (u.nb == 0 && rank == 0) record_error(a.status, KVC_ERR_BOUNDS);
        if (u.my_tiles == 0) continue;
        // The unit's query rows.  With one buffer they wait for the previous
        // unit's last MMA, so the unit's first tiles are issued before them
        // (at most NS steps: every slot wait up to that point depends only
        // on earlier units' MMAs, never on this unit's).
        const int qb = qi % SM::QB;
        const int q_at = SM::QB == 1 ? min(NS, u.my_tiles) : 0;
        auto load_q = [&]() -> bool {
          if (!wait_or_abort(smem_u32(sm.qempty + qb), ((qi / SM::QB) & 1) ^ 1, sm.failed))
            return false;
          mbar_expect_tx(smem_u32(sm.qfull + qb), q_bytes);
          for (int kb = 0; kb < KB; kb++)
            tma_load_2d(smem_u32(sm.q + qb * q_bytes + kb * RT * 16384), &tm_q, kb * 64, u.q_row0,
                        smem_u32(sm.qfull + qb));
          return true;
        };
        bool ok = true;
        for (int pass = 0; pass < 2 && ok; pass++)
          for (int j = 0; j < u.my_tiles; j++, s++) {
            if (pass * u.my_tiles + j == q_at && !(ok = load_q())) break;
            const int slot = s % NS;
            if (!wait_or_abort(smem_u32(sm.empty + slot), ((s / NS) & 1) ^ 1, sm.failed)) {
              ok = false;
              break;
            }
            if (pass == 1 && u.my_tiles >= NS && j < NS) {
              // the tile is still in this slot from pass 1: re-arm, no copy
              mbar_arrive(smem_u32(sm.full + slot));
              continue;
            }
            const int tile = rank + (pass == 0 ? j : pass2_tile<NS>(j, u.my_tiles)) * C;
            mbar_expect_tx(smem_u32(sm.full + slot), stage_bytes);
            for (int kb = 0; kb < KB; kb++)
              tma_load_2d(smem_u32(sm.ring + slot * stage_bytes + kb * 16384), &tm_mk, kb * 64,
                          u.mk_row0 + tile * 128, smem_u32(sm.full + slot));
          }
        qi++;
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t s = 0, t = 0, qi = 0;
      bool ok = true;
      for (int unit = cluster_id; unit < n_units && ok; unit += n_clusters) {
        const UnitInfo u = unit_info(a, unit, C, rank);
        if (u.my_tiles == 0) continue;
        const int qb = qi % SM::QB;
        if (!(ok = wait_or_abort(smem_u32(sm.qfull + qb), (qi / SM::QB) & 1, sm.failed))) break;
        const uint8_t *qbase = sm.q + qb * q_bytes;
        for (int pass = 0; pass < 2 && ok; pass++)
          for (int j = 0; j < u.my_tiles; j++, s++, t++) {
            const int slot = s % NS, buf = t % NBUF;
            if (!(ok = wait_or_abort(smem_u32(sm.full + slot), (s / NS) & 1, sm.failed))) break;
            if (!(ok = wait_or_abort(smem_u32(sm.tempty + buf), ((t / NBUF) & 1) ^ 1,
                                     sm.failed)))
              break;
            tc_fence_after();
            const uint8_t *mk = sm.ring + slot * stage_bytes;
            const uint32_t d = tmem + (uint32_t)(buf * BUFCOLS);
            for (int kk = 0; kk < 4 * KB; kk++) {
              const uint32_t koff = (uint32_t)(kk & 3) * 32u;
              const uint64_t mdesc = smem_desc(smem_u32(mk + (kk >> 2) * 16384) + koff);
              if (pass == 0) {
                for (int rt = 0; rt < RT; rt++) {
                  const uint64_t qdesc =
                      smem_desc(smem_u32(qbase + (kk >> 2) * RT * 16384 + rt * 16384) + koff);
                  mma_bf16(d + (uint32_t)(rt * 128), qdesc, mdesc, a.idesc1, kk > 0);
                }
              } else {
                const uint64_t qdesc = smem_desc(smem_u32(qbase + (kk >> 2) * RT * 16384) + koff);
                mma_bf16(d, mdesc, qdesc, a.idesc2, kk > 0);
              }
            }
            mma_commit(smem_u32(sm.empty + slot));
            mma_commit(smem_u32(sm.tfull + buf));
          }
        if (ok) mma_commit(smem_u32(sm.qempty + qb));  // after the unit's last MMA
        qi++;
      }
      if (!ok) *sm.failed = 1;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- epilogue
    constexpr int NEG = SM::NEG;                // epilogue groups
    const int eg = (warp - 2) >> 2;             // this thread's group
    const int row = 32 * (warp & 3) + lane;     // this thread's TMEM lane
    const int et = (warp - 2) * 32 + lane;      // 0 … 128·NEG − 1
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float zs = a.zscale, invW = 1.f / (float)a.W;
    uint32_t t = 0, ui = 0;
    bool ok = true;
    for (int unit = cluster_id; unit < n_units; unit += n_clusters, ui++) {
      const UnitInfo u = unit_info(a, unit, C, rank);
      if (C == 1 && u.my_tiles == 0) continue;
      // pass 1: this group's tiles
      float pm[RT], ps[RT];
#pragma unroll
      for (int rt = 0; rt < RT; rt++) {
        pm[rt] = -INFINITY;
        ps[rt] = 0.f;
      }
      for (int j = 0; j < u.my_tiles; j++, t++) {
        // the group of a tile follows its index within the unit, so a unit's
        // partial sums merge in the same order whatever ran on this CTA
        // before it (scores do not depend on how units are split between
        // launches)
        if (j % NEG != eg) continue;
        const int buf = t % NBUF;
        ok = __all_sync(0xFFFFFFFFu,
                        ok && wait_or_abort(smem_u32(sm.tfull + buf), (t / NBUF) & 1, sm.failed));
        if (ok) {
          tc_fence_after();
          const int valid = min(128, u.nb - (rank + j * C) * 128);
          float qm[RT], qs[RT];
          ring_pass1<RT>(tmem + lane_base + (uint32_t)(buf * BUFCOLS), valid, zs, qm, qs);
#pragma unroll
          for (int rt = 0; rt < RT; rt++) lse_merge(pm[rt], ps[rt], qm[rt], qs[rt]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(sm.tempty + buf));
      }
      // exchange: group partials → CTA partial → every CTA of the cluster
      const int par = ui & 1;
#pragma unroll
      for (int rt = 0; rt < RT; rt++) sm.egpart[eg * SM::ROWS + rt * 128 + row] = make_float2(pm[rt], ps[rt]);
      named_sync(2, 128 * NEG);
      if (eg == 0) {
        for (int rt = 0; rt < RT; rt++) {
          float m = pm[rt], s2 = ps[rt];
          for (int g2 = 1; g2 < NEG; g2++) {
            const float2 o = sm.egpart[g2 * SM::ROWS + rt * 128 + row];
            lse_merge(m, s2, o.x, o.y);
          }
          const float2 v = make_float2(m, s2);
          float2 *mine = sm.rbuf + (par * kRingMaxC + rank) * SM::ROWS + rt * 128 + row;
          *mine = v;
          for (int p = 0; p < C; p++)
            if (p != rank) st_cluster_f2(mapa_u32(smem_u32(mine), (uint32_t)p), v);
        }
        if (C > 1) {
          fence_acqrel_cluster();
          named_sync(3, 128);
          if (et == 0)
            for (int p = 0; p < C; p++)
              if (p != rank) mbar_arrive_remote(mapa_u32(smem_u32(sm.recv + par), (uint32_t)p));
        }
      }
      if (C > 1)
        ok = __all_sync(0xFFFFFFFFu,
                        ok && wait_or_abort(smem_u32(sm.recv + par), (ui >> 1) & 1, sm.failed, true));
      named_sync(2, 128 * NEG);
      if (et < RT * 128) {
        float m = -INFINITY, s2 = 0.f;
        for (int c = 0; c < C; c++) {
          const float2 v = sm.rbuf[(par * kRingMaxC + c) * SM::ROWS + et];
          lse_merge(m, s2, v.x, v.y);
        }
        sm.lse[et] = (m == -INFINITY) ? INFINITY : m + log2f(s2);
      }
      named_sync(2, 128 * NEG);
      // pass 2: this group's tiles
      for (int j = 0; j < u.my_tiles; j++, t++) {
        if ((int)(t % NEG) != eg) continue;
        const int buf = t % NBUF;
        ok = __all_sync(0xFFFFFFFFu,
                        ok && wait_or_abort(smem_u32(sm.tfull + buf), (t / NBUF) & 1, sm.failed));
        if (ok) {
          tc_fence_after();
          const int tile = rank + pass2_tile<NS>(j, u.my_tiles) * C;
          const int valid = min(128, u.nb - tile * 128);
          float *out = a.scores + ((int64_t)u.l * a.H + u.h) * a.nb_total + u.b0 + tile * 128;
          ring_pass2<W>(tmem + lane_base + (uint32_t)(buf * BUFCOLS), row, valid, a.n2c, a.R, zs,
                        invW, sm.lse, out);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(sm.tempty + buf));
      }
      if (!ok) {
        *sm.failed = 1;
        if (et == 0) record_error(a.status, KVC_ERR_TIMEOUT);
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*sm.failed && threadIdx.x == 0) {
    record_error(a.status, KVC_ERR_TIMEOUT);
    // let this CTA's own copies and MMAs drain (bounded; stale phases return at once)
    for (int i = 0; i < NS; i++) {
      mbar_wait(smem_u32(sm.full + i), 0);
      mbar_wait(smem_u32(sm.full + i), 1);
    }
    for (int i = 0; i < NBUF; i++) {
      mbar_wait(smem_u32(sm.tfull + i), 0);
      mbar_wait(smem_u32(sm.tfull + i), 1);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    free_tmem_cols(tmem, 512);
  }
  if (C > 1) cluster_sync_all();  // no peer still writes into this CTA's memory
}

// --------------------------------------------------------------- host

struct Plan {
  int RT, S, CH, C, n2, n2c;
  bool ok;
};

Plan plan(int R, int W, int D, int nb_max) {
  Plan p{};
  p.ok = (D == 64 || D == 128) && (W == 8 || W == 16 || W == 32) && R >= 1 && R <= 256;
  p.RT = R <= 128 ? 1 : 2;
  p.S = p.RT == 1 ? 2 : 1;  // TMEM: RT·S·128 ≤ 256 and S·n2c ≤ 256
  p.CH = p.S * 128;
  p.C = (nb_max + p.CH - 1) / p.CH;
  p.n2 = (R + 15) / 16 * 16;
  p.n2c = (p.n2 + 31) / 32 * 32;
  return p;
}

size_t smem_bytes(int RT, int D, int n_sess) {
  size_t b = RT == 1 ? Smem<1, 2>::bytes(D, n_sess + 1) : Smem<2, 1>::bytes(D, n_sess + 1);
  // at most two CTAs per SM, so their 2 × 256 TMEM columns always fit
  return b < 80 * 1024 ? 80 * 1024 : b;
}

// CTAs of the persistent kernel: two per SM (its shared memory allows two
// and its TMEM allocation is sized for two).  Launching more CTAs than can
// be resident at once is safe for this kernel — a CTA that is not running
// holds no item — so the count does not rely on the occupancy calculator
// (which may report one).  0 if the kernel cannot run on this device.
template <int RT, int S, int W>
int persistent_capacity(size_t smem) {
  auto kern = k_score_tc<RT, S, W>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreadsTC, smem) !=
          cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return per_sm > 0 ? 2 * sms : 0;
}

// Which tensor-core kernel runs: kvc_score (KVC_KERNEL_AUTO) takes the
// single-read kernel where the shape allows it, else the pipelined cluster
// kernel, else the persistent one, else split mode; kvc_score_ex names one
// of them (cudaErrorNotSupported when it cannot run these sizes).
bool path_allows(int path, int kernel) { return path == KVC_KERNEL_AUTO || path == kernel; }

int ring_cluster(int nb_max) {
  int c = (nb_max + 2047) / 2048;
  return c < 1 ? 1 : (c > kRingMaxC ? kRingMaxC : c);
}

size_t ring_smem(int RT, int D) {
  size_t b = RT == 1 ? RingSmem<1>::bytes(D) : RingSmem<2>::bytes(D);
  return b < 120 * 1024 ? 120 * 1024 : b;  // one CTA per SM: 512 TMEM columns are free
}

// Clusters of the pipelined kernel that can be resident at once (0: none).
template <int RT, int W>
int ring_clusters(int C, int D) {
  auto kern = k_score_ring<RT, W>;
  const size_t smem = ring_smem(RT, D);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(ring_threads<RT>());
  cfg.dynamicSmemBytes = smem;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

template <int RT, int W>
cudaError_t launch_ring(const CUtensorMap &mk, const CUtensorMap &qm, TcArgs a, int n_units,
                        int C, int n_clusters, cudaStream_t s) {
  auto kern = k_score_ring<RT, W>;
  const size_t smem = ring_smem(RT, a.D);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((n_clusters < n_units ? n_clusters : n_units) * C);
  cfg.blockDim = dim3(ring_threads<RT>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mk, qm, a);
}

template <int RT, int S, int W>
cudaError_t launch_plan(const CUtensorMap &mk, const CUtensorMap &qm, TcArgs a, int n_units,
                        const Plan &p, void *ws, int path, cudaStream_t s) {
  if (path_allows(path, KVC_KERNEL_SCORE_RING)) {
    const int C = ring_cluster(p.C * p.CH);
    const int nc = ring_clusters<RT, W>(C, a.D);
    if (nc > 0) {
      TcArgs b = a;
      b.n_chunk = (p.C * p.CH + 127) / 128;  // session length limit in 128-block tiles
      return launch_ring<RT, W>(mk, qm, b, n_units, C, nc, s);
    }
    if (path == KVC_KERNEL_SCORE_RING) return cudaErrorNotSupported;
  }
  const size_t smem = smem_bytes(RT, a.D, a.n_sess);
  const int cap = (a.n_sess <= kMaxSessPersist && path_allows(path, KVC_KERNEL_SCORE_PERSIST))
                      ? persistent_capacity<RT, S, W>(smem)
                      : 0;
  cudaError_t e;
  if (path == KVC_KERNEL_SCORE_PERSIST && !(cap > 0 && cap >= p.C)) return cudaErrorNotSupported;
  if (cap > 0 && cap >= p.C) {
    // ws: [counter, pad to 256 B][unit_done[n_units], pad][partials]
    char *w = static_cast<char *>(ws);
    size_t done_bytes = ((size_t)n_units * 4 + 255) / 256 * 256;
    a.counter = reinterpret_cast<int *>(w);
    a.unit_done = reinterpret_cast<int *>(w + 256);
    a.part = reinterpret_cast<float2 *>(w + 256 + done_bytes);
    e = cudaMemsetAsync(w, 0, 256 + done_bytes, s);
    if (e != cudaSuccess) return e;
    k_score_tc<RT, S, W><<<cap, kThreadsTC, smem, s>>>(mk, qm, a);
    return cudaGetLastError();
  }
  a.part = reinterpret_cast<float2 *>(ws);
  auto k1 = k_score_split<kPass1, RT, S, W>;
  auto k2 = k_score_split<kPass2, RT, S, W>;
  for (auto k : {k1, k2}) {
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
  }
  dim3 grid(p.C, n_units);
  k1<<<grid, kThreadsTC, smem, s>>>(mk, qm, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k2<<<grid, kThreadsTC, smem, s>>>(mk, qm, a);
  return cudaGetLastError();
}

template <int RT, int S>
int launches_rt(const Plan &p, int W, int D, int n_sess) {
  const int C = ring_cluster(p.C * p.CH);
  const int nc = W == 8    ? ring_clusters<RT, 8>(C, D)
                 : W == 16 ? ring_clusters<RT, 16>(C, D)
                           : ring_clusters<RT, 32>(C, D);
  if (nc > 0) return 1;
  size_t smem = smem_bytes(RT, D, n_sess);
  int cap = n_sess > kMaxSessPersist ? 0
            : W == 8              ? persistent_capacity<RT, S, 8>(smem)
            : W == 16             ? persistent_capacity<RT, S, 16>(smem)
                                  : persistent_capacity<RT, S, 32>(smem);
  return (cap > 0 && cap >= p.C) ? 1 : 2;
}

}  // namespace

bool score_tc_supported(int R, int W, int D) { return plan(R, W, D, 1).ok; }

int score_tc_launches(int R, int W, int D, int n_sess, int nb_max) {
  Plan p = plan(R, W, D, nb_max);
  if (!p.ok) return 0;
  if (R % W == 0 && score_fused_supported(R / W, D, W, nb_max)) return 1;
  if (R % W == 0 && score_group_supported(R / W, D, W, nb_max)) return 1;
  return p.RT == 1 ? launches_rt<1, 2>(p, W, D, n_sess) : launches_rt<2, 1>(p, W, D, n_sess);
}

size_t score_tc_ws_bytes(int L, int H, int Hq, int W, int n_sess, int nb_max, int64_t nb_total) {
  int R = (Hq / H) * W;
  Plan p = plan(R, W, 128, nb_max);
  if (!p.ok) return 0;
  const int64_t n_units = (int64_t)L * H * n_sess;
  const size_t row_bytes = (size_t)p.RT * 128 * sizeof(float2);
  // persistent: one partial row set per item (≤ L·H·(nb_total/CH + n_sess) items)
  int64_t items = (int64_t)L * H * ((nb_total + p.CH - 1) / p.CH + n_sess);
  size_t persist = 256 + ((size_t)n_units * 4 + 255) / 256 * 256 + (size_t)items * row_bytes;
  size_t split = (size_t)n_units * p.C * row_bytes;
  size_t ws = persist > split ? persist : split;
  const size_t group = score_group_ws_bytes();
  return ws > group ? ws : group;
}

cudaError_t launch_score_tc(const uint16_t *q, const uint16_t *meank, float *scores, int L,
                            int H, int Hq, int D, int W, const int64_t *blk_off, int n_sess,
                            int64_t nb_total, int nb_max, void *ws, int32_t *status,
                            int path, cudaStream_t s) {
  const int G = Hq / H, R = G * W;
  Plan p = plan(R, W, D, nb_max);
  if (!p.ok) return cudaErrorNotSupported;
  if (path_allows(path, KVC_KERNEL_SCORE_FUSED)) {
    cudaError_t e = launch_score_fused(q, meank, scores, L, H, Hq, D, W, blk_off, n_sess,
                                       nb_total, nb_max, status, s);
    // named, or a shape the single-read kernel covers: its result stands
    if (path == KVC_KERNEL_SCORE_FUSED || e != cudaErrorNotSupported) return e;
  }
  if (path_allows(path, KVC_KERNEL_SCORE_GROUP)) {
    cudaError_t e = launch_score_group(q, meank, scores, L, H, Hq, D, W, blk_off, n_sess,
                                       nb_total, nb_max, ws, status, s);
    if (path == KVC_KERNEL_SCORE_GROUP || e != cudaErrorNotSupported) return e;
  }
  CUtensorMap mk_map, q_map;
  uint64_t mk_rows = (uint64_t)L * H * nb_total;
  uint64_t q_rows = (uint64_t)L * n_sess * Hq * W;
  if (!make_map(&mk_map, meank, mk_rows, D, 128) ||
      !make_map(&q_map, q, q_rows, D, (uint32_t)(p.RT * 128)))
    return cudaErrorNotSupported;
  TcArgs a{};
  a.scores = scores;
  a.blk_off = blk_off;
  a.status = status;
  a.L = L;
  a.H = H;
  a.Hq = Hq;
  a.W = W;
  a.G = G;
  a.R = R;
  a.D = D;
  a.n_sess = n_sess;
  a.n_chunk = p.C;
  a.nb_total = nb_total;
  a.zscale = kLog2eTC / sqrtf((float)D);
  a.idesc1 = make_idesc(128, 128);
  a.idesc2 = make_idesc(128, p.n2);
  a.n2 = p.n2;
  a.n2c = p.n2c;
  const int n_units = L * H * n_sess;
#define KVC_TC_W(RTv, Sv)                                                           \
  switch (W) {                                                                      \
    case 8: return launch_plan<RTv, Sv, 8>(mk_map, q_map, a, n_units, p, ws, path, s);   \
    case 16: return launch_plan<RTv, Sv, 16>(mk_map, q_map, a, n_units, p, ws, path, s); \
    default: return launch_plan<RTv, Sv, 32>(mk_map, q_map, a, n_units, p, ws, path, s); \
  }
  if (p.RT == 1) {
    KVC_TC_W(1, 2)
  } else {
    KVC_TC_W(2, 1)
  }
#undef KVC_TC_W
}

}  // namespace kvc
