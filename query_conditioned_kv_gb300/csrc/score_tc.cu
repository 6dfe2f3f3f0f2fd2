// score_tc.cu — Mean-K block scoring on the 5th-generation tensor cores.
//
// Same quantity as the CUDA-core scorer (KVMem "Query-conditioned
// retrieval"; ActKV §7.1 aggregation): for one unit (layer l, KV head h,
// session r) with query rows ρ = g·W + w,
//   z[ρ,b] = q[ρ]·meank[b]/sqrt(D),  LSE[ρ] = log Σ_b e^z,
//   score[b] = (1/W) Σ_w max_g exp(z[g·W+w,b] − LSE[g·W+w]).
//
// A CTA owns CH = S·128 consecutive blocks of one unit.  Its Mean-K tile
// (CH × D bf16) and the unit's query rows are brought into shared memory by
// TMA (128-byte swizzle, the UMMA K-major layout) and stay there for both
// passes, so Mean-K is read from HBM once.  Both logit products run as
// tcgen05.mma (bf16 × bf16 → fp32 in TMEM), issued by one thread:
//   pass 1  D[ρ][b] (M = 128 query rows, N = 128 blocks per MMA): each
//           epilogue thread owns one query row (one TMEM lane) and keeps an
//           online (max, Σ2^(z−max)) over its CH columns;
//   LSE     the per-CTA partials are combined across the unit's CTAs —
//           through distributed shared memory inside a thread-block cluster
//           (cluster mode), or through global scratch between two launches
//           (split mode, histories longer than 8 CTAs' worth);
//   pass 2  D[b][ρ] (operands swapped: M = 128 blocks, N = R query rows):
//           each thread owns one block and forms max over g and the mean
//           over w of 2^(z−LSE) from its own TMEM lane — W exponentials
//           per block, no cross-lane traffic.
// Two CTAs share each SM (≤ 256 TMEM columns and ≈ 100 KB of shared memory
// each), so one CTA's TMA load overlaps the other's epilogue.
// Warp roles: warps 0–3 read TMEM (warp i owns lanes 32i…32i+31), warp 4
// issues TMA and MMA.  Every wait is bounded; on a timeout the CTA records
// KVC_ERR_TIMEOUT, skips the remaining math, still meets every cluster
// barrier, waits (bounded) for its own copies/MMAs and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kEpiThreads = 128;
constexpr int kThreadsTC = kEpiThreads + 32;
constexpr uint32_t kTmemCols = 256;  // two CTAs share an SM's 512 columns
constexpr float kLog2eTC = 1.4426950408889634f;
constexpr uint32_t kWaitLimit = 1u << 24;  // ≈ 1–2 s with the back-off below

enum Mode { kCluster = 0, kPass1 = 1, kPass2 = 2 };
constexpr int kMaxCluster = 16;  // non-portable above 8

struct TcArgs {
  float *scores;
  const int64_t *blk_off;
  float2 *part;  // split mode: [unit][chunk][RT·128]
  int32_t *status;
  int L, H, Hq, W, G, R, D, n_sess, n_chunk;
  int64_t nb_total;
  float zscale;
  uint32_t idesc1, idesc2;
  int n2;   // pass-2 N (R rounded up to 16)
  int n2c;  // pass-2 TMEM column stride per sub-tile (n2 rounded up to 32)
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on phase `parity`; false after the limit.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; i++) {
    if (mbar_try(bar, parity)) return true;
    if (i > 64) __nanosleep(64);
  }
  return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major, 128-byte-swizzled operand: 8-row atoms of 128 B, atoms 1024 B
// apart (SBO); the leading offset is unused for this layout.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
               : "=f"(v.x), "=f"(v.y)
               : "r"(remote)
               : "memory");
  return v;
}

__device__ __forceinline__ void named_sync_epi() {
  asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
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

// ------------------------------------------------------------ the kernel

// Shared memory: [mk: S·KB boxes of 128 rows × 128 B][q: KB boxes of
// RT·128 rows × 128 B][barriers][tmem holder][part float2 RT·128][lse 256]
template <int MODE, int RT, int S, int W>
__global__ void __launch_bounds__(kThreadsTC, 1)
k_score_tc(const __grid_constant__ CUtensorMap tm_mk, const __grid_constant__ CUtensorMap tm_q,
           TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int KB = a.D / 64;                   // 64-element k-blocks
  const uint32_t mk_box = 128 * 128;         // bytes per Mean-K box
  const uint32_t q_box = RT * 128 * 128;     // bytes per query box
  uint8_t *mk_s = smem;
  uint8_t *q_s = mk_s + S * KB * mk_box;
  uint64_t *bars = reinterpret_cast<uint64_t *>(q_s + KB * q_box);
  // bars: 0 tma_q | 1..S tma_mk | S+1..2S mma1 | 2S+1..3S mma2 | 3S+1 tmem_free
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 3 * S + 2);
  static_assert(W == 8 || W == 16 || W == 32, "W divides 32");
  volatile int *flags = reinterpret_cast<volatile int *>(tmem_holder + 1);  // [0] failed
  float2 *part = reinterpret_cast<float2 *>(
      (reinterpret_cast<uintptr_t>(tmem_holder + 5) + 15) & ~uintptr_t(15));
  float *lse_s = reinterpret_cast<float *>(part + RT * 128);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int unit, chunk;
  if (MODE == kCluster) {
    chunk = (int)cluster_rank();
    unit = blockIdx.x / a.n_chunk;
  } else {
    chunk = blockIdx.x;
    unit = blockIdx.y;
  }
  const int r = unit % a.n_sess;
  const int lh = unit / a.n_sess;
  const int h = lh % a.H, l = lh / a.H;
  const int64_t b0 = a.blk_off[r], b1 = a.blk_off[r + 1];
  bool sess_ok = b0 >= 0 && b1 > b0 && b1 <= a.nb_total;
  const int nb = sess_ok ? (int)(b1 - b0) : 0;
  const int CH = S * 128;
  const int blk_base = chunk * CH;
  const int valid = max(0, min(CH, nb - blk_base));
  // Split-mode CTAs past the unit's end have nothing to do.
  if (MODE != kCluster && valid == 0) {
    if (!sess_ok && chunk == 0 && threadIdx.x == 0) record_error(a.status, KVC_ERR_BOUNDS);
    return;
  }
  if (!sess_ok && chunk == 0 && threadIdx.x == 0) record_error(a.status, KVC_ERR_BOUNDS);

  const int mk_row0 = (int)(((int64_t)l * a.H + h) * a.nb_total + b0 + blk_base);
  const int q_row0 = (int)((((int64_t)l * a.n_sess + r) * a.Hq + (int64_t)h * a.G) * a.W);
  const uint32_t bar0 = smem_u32(bars);
  auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };

  if (threadIdx.x == 0) {
    flags[0] = 0;
    for (int i = 0; i < 3 * S + 1; i++) mbar_init(BAR(i), 1);
    mbar_init(BAR(3 * S + 1), 4);  // tmem_free: one arrive per epilogue warp
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // ------------------------------------------------------------ producer
  if (warp == 4) {
    if (lane == 0 && valid > 0) {
      bool ok = true;
      // loads
      mbar_expect_tx(BAR(0), KB * q_box);
      for (int kb = 0; kb < KB; kb++)
        tma_load_2d(smem_u32(q_s + kb * q_box), &tm_q, kb * 64, q_row0, BAR(0));
      for (int s = 0; s < S; s++) {
        mbar_expect_tx(BAR(1 + s), KB * mk_box);
        for (int kb = 0; kb < KB; kb++)
          tma_load_2d(smem_u32(mk_s + (s * KB + kb) * mk_box), &tm_mk, kb * 64,
                      mk_row0 + s * 128, BAR(1 + s));
      }
      ok = mbar_wait(BAR(0), 0);
      if (MODE != kPass2) {
        // pass 1: D[ρ][b] = Q · Mean-Kᵀ, TMEM columns (rt·S + s)·128
        for (int s = 0; s < S && ok; s++) {
          ok = mbar_wait(BAR(1 + s), 0);
          if (!ok) break;
          tc_fence_after();
          for (int rt = 0; rt < RT; rt++)
            for (int kk = 0; kk < 4 * KB; kk++) {
              uint32_t koff = (uint32_t)(kk & 3) * 32u;
              uint64_t adesc = smem_desc(smem_u32(q_s + (kk >> 2) * q_box + rt * 128 * 128) + koff);
              uint64_t bdesc = smem_desc(smem_u32(mk_s + (s * KB + (kk >> 2)) * mk_box) + koff);
              mma_bf16(tmem + (uint32_t)((rt * S + s) * 128), adesc, bdesc, a.idesc1, kk > 0);
            }
          mma_commit(BAR(1 + S + s));
        }
        if (MODE == kCluster && ok) {
          ok = mbar_wait(BAR(3 * S + 1), 0);  // pass-1 TMEM reads finished
          tc_fence_after();
        }
      } else {
        for (int s = 0; s < S && ok; s++) ok = mbar_wait(BAR(1 + s), 0);
        tc_fence_after();
      }
      if (MODE != kPass1 && ok) {
        // pass 2: D[b][ρ] = Mean-K · Qᵀ, TMEM columns s·n2c
        for (int s = 0; s < S; s++) {
          for (int kk = 0; kk < 4 * KB; kk++) {
            uint32_t koff = (uint32_t)(kk & 3) * 32u;
            uint64_t adesc = smem_desc(smem_u32(mk_s + (s * KB + (kk >> 2)) * mk_box) + koff);
            uint64_t bdesc = smem_desc(smem_u32(q_s + (kk >> 2) * q_box) + koff);
            mma_bf16(tmem + (uint32_t)(s * a.n2c), adesc, bdesc, a.idesc2, kk > 0);
          }
          mma_commit(BAR(1 + 2 * S + s));
        }
      }
      if (!ok) {
        flags[0] = 1;
        record_error(a.status, KVC_ERR_TIMEOUT);
      }
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ epilogue
  const float zs = a.zscale;
  float pm[RT], ps[RT];
#pragma unroll
  for (int rt = 0; rt < RT; rt++) {
    pm[rt] = -INFINITY;
    ps[rt] = 0.f;
  }
  if (warp < 4) {
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    if (MODE != kPass2 && valid > 0) {
      for (int s = 0; s < S; s++) {
        bool ok = __all_sync(0xFFFFFFFFu, flags[0] == 0 && mbar_wait(BAR(1 + S + s), 0));
        if (!ok) {  // warp-uniform
          if (lane == 0) record_error(a.status, KVC_ERR_TIMEOUT);
          flags[0] = 1;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int rt = 0; rt < RT; rt++) {
          for (int c = 0; c < 4; c++) {
            float v[32];
            tmem_ld32(tmem + lane_base + (uint32_t)((rt * S + s) * 128 + 32 * c), v);
            const int col0 = s * 128 + 32 * c;  // block offset within the CTA
            const int nv = min(32, valid - col0);
            if (nv <= 0) continue;
            if (nv < 32) {
#pragma unroll
              for (int j = 0; j < 32; j++)
                if (j >= nv) v[j] = -INFINITY;
            }
            // max of the raw products (zs > 0), then 2^(v·zs − max·zs) by FFMA
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
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(BAR(3 * S + 1));
#pragma unroll
    for (int rt = 0; rt < RT; rt++) part[rt * 128 + threadIdx.x] = make_float2(pm[rt], ps[rt]);
    if (MODE == kPass1) {
      float2 *dst = a.part + ((int64_t)unit * a.n_chunk + chunk) * (RT * 128);
#pragma unroll
      for (int rt = 0; rt < RT; rt++) dst[rt * 128 + threadIdx.x] = make_float2(pm[rt], ps[rt]);
    }
  }
  if (MODE == kCluster) cluster_sync_all();  // partials visible cluster-wide

  if (warp < 4 && MODE != kPass1) {
    // LSE of every query row (thread t combines rows t and t+128)
    const int n_ct = (nb + CH - 1) / CH;
    for (int rr = threadIdx.x; rr < RT * 128; rr += kEpiThreads) {
      float m = -INFINITY, s = 0.f;
      if (MODE == kCluster) {
        float2 pv[16];
#pragma unroll
        for (int c = 0; c < 16; c++)
          pv[c] = c < n_ct ? ld_dsmem_f2(smem_u32(part + rr), (uint32_t)c)
                           : make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int c = 0; c < 16; c++) lse_merge(m, s, pv[c].x, pv[c].y);
      } else {
        const float2 *src = a.part + (int64_t)unit * a.n_chunk * (RT * 128) + rr;
        for (int c = 0; c < n_ct; c++) {
          float2 p = src[(int64_t)c * (RT * 128)];
          lse_merge(m, s, p.x, p.y);
        }
      }
      lse_s[rr] = (m == -INFINITY) ? INFINITY : m + log2f(s);
    }
    named_sync_epi();
    // pass 2 epilogue: thread = block
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    if (valid > 0) {
      const int n_chunks2 = a.n2c / 32;
      for (int s = 0; s < S; s++) {
        bool ok = __all_sync(0xFFFFFFFFu, flags[0] == 0 && mbar_wait(BAR(1 + 2 * S + s), 0));
        if (!ok) {  // warp-uniform
          if (lane == 0) record_error(a.status, KVC_ERR_TIMEOUT);
          flags[0] = 1;
          break;
        }
        tc_fence_after();
        float mw[W];
#pragma unroll
        for (int w = 0; w < W; w++) mw[w] = -INFINITY;
        for (int c = 0; c < n_chunks2; c++) {
          float v[32];
          tmem_ld32(tmem + lane_base + (uint32_t)(s * a.n2c + 32 * c), v);
#pragma unroll
          for (int j = 0; j < 32; j++) {
            const int rho = 32 * c + j;
            if (rho < a.R) mw[j % W] = fmaxf(mw[j % W], v[j] * zs - lse_s[rho]);
          }
        }
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < W; w++) acc += exp2f(mw[w]);
        const int bl = s * 128 + warp * 32 + lane;
        if (bl < valid)
          a.scores[((int64_t)l * a.H + h) * a.nb_total + b0 + blk_base + bl] = acc / (float)a.W;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 4 && lane == 0 && valid > 0 && flags[0] != 0) {
    // a wait gave up: let this CTA's own copies and MMAs drain (bounded)
    for (int i = 0; i < 3 * S + 1; i++) mbar_wait(BAR(i), 0);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols));
  }
  if (MODE == kCluster) cluster_sync_all();  // peers are done reading `part`
}

// --------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_map(CUtensorMap *m, const void *base, uint64_t rows, int D, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

uint32_t make_idesc(int M, int N) {
  return (1u << 4)      // D: fp32
         | (1u << 7)    // A: bf16
         | (1u << 10)   // B: bf16 (both K-major: bits 15, 16 = 0)
         | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct Plan {
  int RT, S, C, n2, n2c;
  bool ok;
};

Plan plan(int R, int W, int D, int nb_max) {
  Plan p{};
  p.ok = (D == 64 || D == 128) && (W == 8 || W == 16 || W == 32) && R >= 1 && R <= 256;
  p.RT = R <= 128 ? 1 : 2;
  p.S = p.RT == 1 ? 2 : 1;  // TMEM: RT·S·128 ≤ 256 and S·n2c ≤ 256
  p.C = (nb_max + p.S * 128 - 1) / (p.S * 128);
  p.n2 = (R + 15) / 16 * 16;
  p.n2c = (p.n2 + 31) / 32 * 32;
  return p;
}

size_t smem_bytes(int RT, int S, int D) {
  int KB = D / 64;
  size_t b = 1024 /*align slack*/ + (size_t)S * KB * 16384 + (size_t)KB * RT * 16384 +
             (3 * S + 2) * 8 + 4 + 16 + 16 + RT * 128 * 8 + 256 * 4;
  // at most two CTAs per SM, so their 2 × 256 TMEM columns always fit
  return b < 80 * 1024 ? 80 * 1024 : b;
}

template <int MODE, int RT, int S, int W>
cudaError_t launch_mode(const CUtensorMap &mk, const CUtensorMap &qm, const TcArgs &a,
                        int n_units, int C, cudaStream_t s) {
  auto kern = k_score_tc<MODE, RT, S, W>;
  size_t smem = smem_bytes(RT, S, a.D);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  if (MODE == kCluster && C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kThreadsTC);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  if (MODE == kCluster) {
    cfg.gridDim = dim3(n_units * C);
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  } else {
    cfg.gridDim = dim3(C, n_units);
    cfg.numAttrs = 0;
  }
  return cudaLaunchKernelEx(&cfg, kern, mk, qm, a);
}

// Whether clusters of C CTAs of this kernel can be resident at all.
template <int RT, int S, int W>
bool cluster_fits(int C, int D) {
  auto kern = k_score_tc<kCluster, RT, S, W>;
  size_t smem = smem_bytes(RT, S, D);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return false;
  if (C > 8 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return false;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(kThreadsTC);
  cfg.dynamicSmemBytes = smem;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return n > 0;
}

template <int RT, int S, int W>
cudaError_t launch_plan(const CUtensorMap &mk, const CUtensorMap &qm, const TcArgs &a,
                        int n_units, int C, cudaStream_t s) {
  if (C <= kMaxCluster && cluster_fits<RT, S, W>(C, a.D))
    return launch_mode<kCluster, RT, S, W>(mk, qm, a, n_units, C, s);
  cudaError_t e = launch_mode<kPass1, RT, S, W>(mk, qm, a, n_units, C, s);
  if (e != cudaSuccess) return e;
  return launch_mode<kPass2, RT, S, W>(mk, qm, a, n_units, C, s);
}

template <int RT, int S>
int launches_rt(int C, int W, int D) {
  bool fits = W == 8    ? cluster_fits<RT, S, 8>(C, D)
              : W == 16 ? cluster_fits<RT, S, 16>(C, D)
                        : cluster_fits<RT, S, 32>(C, D);
  return (C <= kMaxCluster && fits) ? 1 : 2;
}

}  // namespace

bool score_tc_supported(int R, int W, int D) { return plan(R, W, D, 1).ok; }

int score_tc_launches(int R, int W, int D, int nb_max) {
  Plan p = plan(R, W, D, nb_max);
  if (!p.ok) return 0;
  return p.RT == 1 ? launches_rt<1, 2>(p.C, W, D) : launches_rt<2, 1>(p.C, W, D);
}

size_t score_tc_ws_bytes(int L, int H, int Hq, int W, int n_sess, int nb_max) {
  int R = (Hq / H) * W;
  Plan p = plan(R, W, 128, nb_max);
  if (!p.ok) return 0;  // split-mode partials (also reserved when clusters would do)
  return (size_t)L * H * n_sess * p.C * p.RT * 128 * sizeof(float2);
}

cudaError_t launch_score_tc(const uint16_t *q, const uint16_t *meank, float *scores, int L,
                            int H, int Hq, int D, int W, const int64_t *blk_off, int n_sess,
                            int64_t nb_total, int nb_max, void *ws, int32_t *status,
                            cudaStream_t s) {
  const int G = Hq / H, R = G * W;
  Plan p = plan(R, W, D, nb_max);
  if (!p.ok) return cudaErrorNotSupported;
  CUtensorMap mk_map, q_map;
  uint64_t mk_rows = (uint64_t)L * H * nb_total;
  uint64_t q_rows = (uint64_t)n_sess * L * Hq * W;
  if (!make_map(&mk_map, meank, mk_rows, D, 128) ||
      !make_map(&q_map, q, q_rows, D, (uint32_t)(p.RT * 128)))
    return cudaErrorNotSupported;
  TcArgs a;
  a.scores = scores;
  a.blk_off = blk_off;
  a.part = reinterpret_cast<float2 *>(ws);
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
#define KVC_TC_W(RTv, Sv)                                                         \
  switch (W) {                                                                    \
    case 8: return launch_plan<RTv, Sv, 8>(mk_map, q_map, a, n_units, p.C, s);   \
    case 16: return launch_plan<RTv, Sv, 16>(mk_map, q_map, a, n_units, p.C, s); \
    default: return launch_plan<RTv, Sv, 32>(mk_map, q_map, a, n_units, p.C, s); \
  }
  if (p.RT == 1) {
    KVC_TC_W(1, 2)
  } else {
    KVC_TC_W(2, 1)
  }
#undef KVC_TC_W
}

}  // namespace kvc
