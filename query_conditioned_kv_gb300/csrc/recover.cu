// recover.cu — ActKV's paged primitives on sm_103a.
//
// ActKV: Efficient LLM Agents through Action-Guided KV Cache Management,
// §7.1 (Algorithm 3, recovery-based attention calculation) and §7.2
// (Algorithm 4, conflict-free slot planning and one-shot in-place
// compaction), on the paged layout of §2: K and V pools of one row of H·D
// elements per (layer, physical slot), a block table per request.
//
// Recovery score (one decode step of an action token): for every visible
// key position p of request r, with slot = bt[p/BS]·BS + p%BS,
//   x[p] = Σ_l Σ_h max_{g<G} exp(q[l,hG+g]·K[l,slot,h]/√D − LSE[l,hG+g])
// and the per-position state keeps the running mean over the action tokens
// (count = 1 restarts it).  The contraction is a real GEMM once the page is
// the M dimension: one physical page of BS = 16 slots × H = 8 KV heads is a
// 128-row K-major tile (32 KB at D = 128, contiguous in the pool) that TMA
// brings into shared memory by its block-table coordinate, and
//   D[s·H + h][hq] = K[slot s, head h] · q[hq]          (M 128, N Hq, K D)
// runs on tcgen05 into TMEM.  Only the G columns of the row's own group are
// used (the other 7/8 of the products are free on the tensor pipe); the
// epilogue takes the max over the group in the log2 domain first, so one
// ex2 per (slot, head, layer) remains.  Shapes outside that tile (other
// page sizes, head counts or group sizes) run on a CUDA-core kernel with
// the same arithmetic order.
//
// Tail plan + compaction: per request, m retained tokens go to the last
// X = ⌈m/BS⌉ logical blocks; the k-th retained position before that region
// is copied to the k-th non-retained slot inside it, so sources and
// destinations are disjoint and every copy can run at once.
#include <math.h>

#include <algorithm>

#include "kvc_internal.cuh"
#include "tc_ptx.cuh"

namespace kvc {
namespace {

using namespace tc;

constexpr float kLog2eR = 1.4426950408889634f;

// ---------------------------------------------------------- recovery

struct RecArgs {
  const uint16_t *q;            // [n_req][L][Hq][D]
  const uint16_t *kpool;        // [L][n_slots][H][D]
  const float *lse;             // [n_req][L][Hq], natural log
  const int32_t *block_table;   // [n_req][max_blocks]
  const int32_t *seqused;       // [n_req]
  const int32_t *count;         // [n_req]
  float *state;                 // [n_req][max_blocks·BS]
  int32_t *status;
  int n_req, L, H, Hq, G, D, BS, max_blocks;
  int P;         // pages per work item
  int n_chunks;  // page chunks per request = ⌈max_blocks / P⌉
  int n_lg;      // layer groups per chunk (> 1: partial sums, then a finalize)
  float *partial;  // [n_lg][n_req][max_blocks·BS] when n_lg > 1
  int64_t n_slots;
  float zscale;  // log2(e)/√D
  uint32_t idesc;
};

struct Item {
  int r, j0, seq, cnt, lg, l0, l1;
  uint32_t mask;  // bit jj: page j0 + jj is visible and maps to a valid block
  bool active;    // request generating an action token, sizes valid
};

// Every role of a CTA derives the same item description from the same
// (read-only) inputs, so producer, MMA issuer and epilogue agree on which
// tiles exist.  Only the caller passing `record` reports bad inputs.
__device__ __forceinline__ Item item_info(const RecArgs &a, int item, bool record) {
  Item it;
  it.lg = item % a.n_lg;
  const int rest = item / a.n_lg;
  it.r = rest / a.n_chunks;
  it.j0 = (rest - it.r * a.n_chunks) * a.P;
  it.l0 = it.lg * a.L / a.n_lg;
  it.l1 = (it.lg + 1) * a.L / a.n_lg;
  it.seq = a.seqused[it.r];
  it.cnt = a.count[it.r];
  it.mask = 0u;
  it.active = it.cnt >= 1;
  if (!it.active) return it;
  if (it.seq < 0 || (int64_t)it.seq > (int64_t)a.max_blocks * a.BS) {
    if (record) record_error(a.status, KVC_ERR_BOUNDS);
    it.active = false;
    return it;
  }
  const int64_t n_blocks = a.n_slots / a.BS;
  for (int jj = 0; jj < a.P; jj++) {
    const int j = it.j0 + jj;
    if (j >= a.max_blocks || (int64_t)j * a.BS >= it.seq) break;
    const int32_t b = a.block_table[(int64_t)it.r * a.max_blocks + j];
    if (b < 0 || b >= n_blocks) {
      if (record) record_error(a.status, KVC_ERR_BOUNDS);
      continue;
    }
    it.mask |= 1u << jj;
  }
  return it;
}

// Running mean over action tokens; count 1 starts a new action region.
__device__ __forceinline__ void update_state(float *st, float x, int cnt) {
  *st = cnt == 1 ? x : *st + (x - *st) / (float)cnt;
}

// ------------------------------------------------- tensor-core kernel

constexpr int kRecThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2–5 epilogue
constexpr int kRecQB = 4;         // query-row buffers
constexpr int kRecNacc = 4;       // TMEM accumulators
constexpr int kRecPmax = 8;       // pages per item, at most
constexpr int kRecH = 8, kRecBS = 16;  // the tile: 16 slots × 8 KV heads = 128 rows

struct RecSmem {
  uint8_t *ring, *q;
  uint64_t *full, *empty, *qfull, *qempty, *tfull, *tempty;
  uint32_t *tmem_holder;
  volatile int *failed;
  __device__ RecSmem(uint8_t *raw, int NS, int KB, int ncol) {
    uint8_t *p = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    ring = p;
    p += (size_t)NS * KB * 16384;
    q = p;
    p += (size_t)kRecQB * KB * ncol * 128;
    uint64_t *b = reinterpret_cast<uint64_t *>(p);
    full = b;
    empty = full + NS;
    qfull = empty + NS;
    qempty = qfull + kRecQB;
    tfull = qempty + kRecQB;
    tempty = tfull + kRecNacc;
    tmem_holder = reinterpret_cast<uint32_t *>(tempty + kRecNacc);
    failed = reinterpret_cast<volatile int *>(tmem_holder + 1);
  }
  static size_t bytes(int NS, int KB, int ncol) {
    return 1024 + (size_t)NS * KB * 16384 + (size_t)kRecQB * KB * ncol * 128 +
           (size_t)(2 * NS + 2 * kRecQB + 2 * kRecNacc) * 8 + 16;
  }
};

template <int G>
__global__ void __launch_bounds__(kRecThreads, 1)
k_recover_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
             RecArgs a, int NS, uint32_t tmem_cols) {
  constexpr int H = kRecH, BS = kRecBS, NCOL = H * G;
  extern __shared__ uint8_t smem_raw[];
  const int KB = a.D / 64;
  RecSmem sm(smem_raw, NS, KB, NCOL);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = a.n_req * a.n_chunks * a.n_lg;
  const uint32_t tile_bytes = (uint32_t)KB * 16384u;
  const uint32_t q_bytes = (uint32_t)(KB * NCOL * 128);

  if (threadIdx.x == 0) {
    *sm.failed = 0;
    for (int i = 0; i < NS; i++) {
      mbar_init(smem_u32(sm.full + i), 1);
      mbar_init(smem_u32(sm.empty + i), 1);
    }
    for (int i = 0; i < kRecQB; i++) {
      mbar_init(smem_u32(sm.qfull + i), 1);
      mbar_init(smem_u32(sm.qempty + i), 1);
    }
    for (int i = 0; i < kRecNacc; i++) {
      mbar_init(smem_u32(sm.tfull + i), 1);
      mbar_init(smem_u32(sm.tempty + i), 4);  // one arrival per epilogue warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) alloc_tmem_cols(sm.tmem_holder, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_holder;

  if (warp == 0) {
    // --------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t s = 0, qi = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const Item it = item_info(a, item, true);
        if (!it.active || !it.mask) continue;
        const int32_t *bt = a.block_table + (int64_t)it.r * a.max_blocks + it.j0;
        for (int l = it.l0; l < it.l1 && ok; l++) {
          const int qb = qi % kRecQB;
          if (!(ok = mbar_wait_bounded(smem_u32(sm.qempty + qb), ((qi / kRecQB) & 1) ^ 1,
                                       sm.failed)))
            break;
          mbar_expect_tx(smem_u32(sm.qfull + qb), q_bytes);
          const int qrow = (it.r * a.L + l) * NCOL;
          for (int kb = 0; kb < KB; kb++)
            tma_load_2d(smem_u32(sm.q + qb * q_bytes + kb * NCOL * 128), &tm_q, kb * 64, qrow,
                        smem_u32(sm.qfull + qb));
          qi++;
          for (int jj = 0; jj < a.P; jj++) {
            if (!((it.mask >> jj) & 1u)) continue;
            const int st = s % NS;
            if (!(ok = mbar_wait_bounded(smem_u32(sm.empty + st), ((s / NS) & 1) ^ 1,
                                         sm.failed)))
              break;
            const int row0 = (int)(((int64_t)l * a.n_slots + (int64_t)bt[jj] * BS) * H);
            mbar_expect_tx(smem_u32(sm.full + st), tile_bytes);
            for (int kb = 0; kb < KB; kb++)
              tma_load_2d(smem_u32(sm.ring + st * tile_bytes + kb * 16384), &tm_k, kb * 64, row0,
                          smem_u32(sm.full + st));
            s++;
          }
        }
      }
      if (!ok) *sm.failed = 1;
    }
    __syncwarp();
  } else if (warp == 1) {
    // --------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t s = 0, t = 0, qi = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const Item it = item_info(a, item, false);
        if (!it.active || !it.mask) continue;
        for (int l = it.l0; l < it.l1 && ok; l++) {
          const int qb = qi % kRecQB;
          if (!(ok = mbar_wait_bounded(smem_u32(sm.qfull + qb), (qi / kRecQB) & 1, sm.failed)))
            break;
          const uint8_t *qbase = sm.q + qb * q_bytes;
          for (int jj = 0; jj < a.P && ok; jj++) {
            if (!((it.mask >> jj) & 1u)) continue;
            const int st = s % NS, buf = t % kRecNacc;
            if (!(ok = mbar_wait_bounded(smem_u32(sm.full + st), (s / NS) & 1, sm.failed))) break;
            if (!(ok = mbar_wait_bounded(smem_u32(sm.tempty + buf), ((t / kRecNacc) & 1) ^ 1,
                                         sm.failed)))
              break;
            tc_fence_after();
            const uint8_t *kt = sm.ring + st * tile_bytes;
            const uint32_t d = tmem + (uint32_t)(buf * NCOL);
            for (int kk = 0; kk < 4 * KB; kk++) {
              const uint32_t koff = (uint32_t)(kk & 3) * 32u;
              const uint64_t adesc = smem_desc(smem_u32(kt + (kk >> 2) * 16384) + koff);
              const uint64_t bdesc = smem_desc(smem_u32(qbase + (kk >> 2) * NCOL * 128) + koff);
              mma_bf16(d, adesc, bdesc, a.idesc, kk > 0);
            }
            mma_commit(smem_u32(sm.empty + st));
            mma_commit(smem_u32(sm.tfull + buf));
            s++;
            t++;
          }
          if (ok) mma_commit(smem_u32(sm.qempty + qb));  // after the last MMA reading it
          qi++;
        }
      }
      if (!ok) *sm.failed = 1;
    }
    __syncwarp();
  } else {
    // --------------------------------------------------- epilogue
    // TMEM lane = tile row = s·H + h; a warp may read only its own quarter
    // of the lanes (warp id mod 4).
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;
    const int s_ = row / H, h = row % H;
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    const float zs = a.zscale;
    const int cap = a.max_blocks * BS;
    uint32_t t = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const Item it = item_info(a, item, false);
      if (!it.active) continue;
      float xacc[kRecPmax];
#pragma unroll
      for (int jj = 0; jj < kRecPmax; jj++) xacc[jj] = 0.f;
      if (it.mask) {
        const float *lse_r = a.lse + (int64_t)it.r * a.L * NCOL + h * G;
        for (int l = it.l0; l < it.l1 && ok; l++) {
          float l2[G];
#pragma unroll
          for (int g = 0; g < G; g++) l2[g] = __ldg(lse_r + l * NCOL + g) * kLog2eR;
#pragma unroll
          for (int jj = 0; jj < kRecPmax; jj++) {
            if (jj >= a.P || !((it.mask >> jj) & 1u)) continue;  // warp-uniform
            const int buf = t % kRecNacc;
            ok = __all_sync(0xFFFFFFFFu, ok && mbar_wait_bounded(smem_u32(sm.tfull + buf),
                                                                 (t / kRecNacc) & 1, sm.failed));
            if (ok) {
              tc_fence_after();
              float v[NCOL];
              const uint32_t taddr = tmem + lane_base + (uint32_t)(buf * NCOL);
              if constexpr (NCOL == 16) tmem_ld16(taddr, v);
              else if constexpr (NCOL == 32) tmem_ld32(taddr, v);
              else tmem_ld64(taddr, v);
              // max over the group, in the log2 domain, then one ex2
              float mx = -INFINITY;
#pragma unroll
              for (int g = 0; g < G; g++) {
                float z = v[g];
#pragma unroll
                for (int hh = 1; hh < H; hh++) z = (h == hh) ? v[hh * G + g] : z;
                mx = fmaxf(mx, fmaf(z, zs, -l2[g]));
              }
              xacc[jj] += ex2(mx);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(sm.tempty + buf));
            t++;
          }
        }
      }
      if (!ok) break;
      // Σ over the 8 heads of each slot (lanes 8k … 8k+7), then the state
#pragma unroll
      for (int jj = 0; jj < kRecPmax; jj++) {
        if (jj >= a.P || it.j0 + jj >= a.max_blocks) break;  // warp-uniform
        float x = xacc[jj];
        x += __shfl_xor_sync(0xFFFFFFFFu, x, 1);
        x += __shfl_xor_sync(0xFFFFFFFFu, x, 2);
        x += __shfl_xor_sync(0xFFFFFFFFu, x, 4);
        const int p = (it.j0 + jj) * BS + s_;
        if (h == 0) {
          const float xf = (((it.mask >> jj) & 1u) && p < it.seq) ? x : 0.f;
          if (a.n_lg == 1)
            update_state(a.state + (int64_t)it.r * cap + p, xf, it.cnt);
          else
            a.partial[((int64_t)it.lg * a.n_req + it.r) * cap + p] = xf;
        }
      }
    }
    if (!ok) {
      *sm.failed = 1;
      if (lane == 0) record_error(a.status, KVC_ERR_TIMEOUT);
    }
  }

  // ------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*sm.failed && threadIdx.x == 0) {
    record_error(a.status, KVC_ERR_TIMEOUT);
    // let this CTA's own copies and MMAs finish before its memory is released
    for (int i = 0; i < NS; i++) {
      mbar_drain(smem_u32(sm.full + i), 0);
      mbar_drain(smem_u32(sm.full + i), 1);
    }
    for (int i = 0; i < kRecQB; i++) {
      mbar_drain(smem_u32(sm.qfull + i), 0);
      mbar_drain(smem_u32(sm.qfull + i), 1);
    }
    for (int i = 0; i < kRecNacc; i++) {
      mbar_drain(smem_u32(sm.tfull + i), 0);
      mbar_drain(smem_u32(sm.tfull + i), 1);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    free_tmem_cols(tmem, tmem_cols);
  }
}

// The layer groups' partial sums, added in group order, then the state.
__global__ void __launch_bounds__(256)
k_recover_finalize(RecArgs a) {
  const int cap = a.max_blocks * a.BS;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)a.n_req * cap) return;
  const int r = (int)(i / cap), p = (int)(i - (int64_t)r * cap);
  const int cnt = a.count[r], seq = a.seqused[r];
  if (cnt < 1 || seq < 0 || seq > cap) return;  // skipped (a bad length was recorded)
  float x = 0.f;
  if (p < seq)
    for (int g = 0; g < a.n_lg; g++) x += a.partial[((int64_t)g * a.n_req + r) * cap + p];
  update_state(a.state + i, x, cnt);
}

// ------------------------------------------------- CUDA-core kernel

// One CTA per (request, page); warps take (slot, head) pairs, lanes split
// the head dimension.  The per-(slot, head) sums over layers live in shared
// memory (each pair has one owning warp), then the heads are summed in order.
constexpr int kRecCcThreads = 256;

__global__ void __launch_bounds__(kRecCcThreads)
k_recover_cc(RecArgs a) {
  extern __shared__ float smf[];
  const int nq = a.Hq * a.D;
  uint16_t *qs = reinterpret_cast<uint16_t *>(smf);                // [Hq][D]
  float *l2 = smf + (nq + 1) / 2;                                   // [Hq]
  float *xs = l2 + a.Hq;                                            // [BS·H]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_warps = kRecCcThreads / 32;
  const Item it = item_info(a, blockIdx.x, true);
  if (!it.active) return;
  const int j = it.j0;  // one page per item
  if (j >= a.max_blocks) return;
  const bool loaded = it.mask & 1u;
  const int npair = a.BS * a.H;
  for (int e = threadIdx.x; e < npair; e += kRecCcThreads) xs[e] = 0.f;
  const int per = a.D / 32;
  if (loaded) {
    const int64_t slot0 = (int64_t)a.block_table[(int64_t)it.r * a.max_blocks + j] * a.BS;
    for (int l = 0; l < a.L; l++) {
      __syncthreads();
      const uint16_t *qrl = a.q + ((int64_t)it.r * a.L + l) * nq;
      for (int i = threadIdx.x; i < nq; i += kRecCcThreads) qs[i] = qrl[i];
      for (int i = threadIdx.x; i < a.Hq; i += kRecCcThreads)
        l2[i] = a.lse[((int64_t)it.r * a.L + l) * a.Hq + i] * kLog2eR;
      __syncthreads();
      for (int e = warp; e < npair; e += n_warps) {
        const int s = e / a.H, h = e % a.H;
        if (j * a.BS + s >= it.seq) continue;  // past the sequence: not visible
        const uint16_t *kr = a.kpool + ((l * a.n_slots + slot0 + s) * a.H + h) * (int64_t)a.D;
        float kv[4];
#pragma unroll
        for (int i = 0; i < 4; i++)
          kv[i] = i < per ? __uint_as_float((uint32_t)kr[lane + 32 * i] << 16) : 0.f;
        float mx = -INFINITY;
        for (int g = 0; g < a.G; g++) {
          const uint16_t *qq = qs + (h * a.G + g) * a.D;
          float dot = 0.f;
#pragma unroll
          for (int i = 0; i < 4; i++)
            if (i < per) dot = fmaf(__uint_as_float((uint32_t)qq[lane + 32 * i] << 16), kv[i], dot);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
          mx = fmaxf(mx, fmaf(dot, a.zscale, -l2[h * a.G + g]));
        }
        if (lane == 0) xs[e] += ex2(mx);
      }
    }
  }
  __syncthreads();
  const int cap = a.max_blocks * a.BS;
  for (int s = threadIdx.x; s < a.BS; s += kRecCcThreads) {
    const int p = j * a.BS + s;
    float x = 0.f;
    if (loaded && p < it.seq)
      for (int h = 0; h < a.H; h++) x += xs[s * a.H + h];
    update_state(a.state + (int64_t)it.r * cap + p, x, it.cnt);
  }
}

// ------------------------------------------------------ tail planning

constexpr int kPlanThreads = 256;

struct PlanArgs {
  const uint32_t *keepmask;
  const int32_t *seqused, *block_table;
  int32_t *src, *dst, *n_pairs, *n_tail, *freed, *n_freed, *new_table;
  uint32_t *tail_mask;
  int32_t *status;
  int n_req, BS, max_blocks, mask_words, cap, tm_words;
  int64_t n_blocks;  // physical blocks in the pool (for the bounds check)
};

// Inclusive scan of one int per thread over the CTA (returns the total).
__device__ __forceinline__ int block_scan_incl(int v, int *sbuf, int &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) sbuf[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kPlanThreads / 32 ? sbuf[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kPlanThreads / 32) sbuf[lane] = w;
  }
  __syncthreads();
  const int before = warp > 0 ? sbuf[warp - 1] : 0;
  total = sbuf[kPlanThreads / 32 - 1];
  __syncthreads();
  return v + before;
}

// One CTA per request.  Positions are visited as 32-bit words of the keep
// mask; each thread owns a contiguous run of words, so the ranks of its
// sources and destinations follow from one block scan of its counts.
__global__ void __launch_bounds__(kPlanThreads)
k_tail_plan(PlanArgs a) {
  extern __shared__ uint32_t tm_s[];  // [tm_words] region mask being built
  __shared__ int sbuf[kPlanThreads / 32];
  const int r = blockIdx.x;
  const int n = a.seqused[r];
  const int32_t *bt = a.block_table + (int64_t)r * a.max_blocks;
  int32_t *src = a.src + (int64_t)r * a.cap, *dst = a.dst + (int64_t)r * a.cap;
  for (int i = threadIdx.x; i < a.tm_words; i += kPlanThreads) tm_s[i] = 0u;
  const bool bad = n < 0 || (int64_t)n > (int64_t)a.max_blocks * a.BS ||
                   (int64_t)(n + 31) / 32 > a.mask_words;
  const int nn = bad ? 0 : n;
  if (bad && threadIdx.x == 0) record_error(a.status, KVC_ERR_BOUNDS);
  const int Y = (nn + a.BS - 1) / a.BS;
  const int end = Y * a.BS;
  const int n_words = (end + 31) / 32;
  const int per = (n_words + kPlanThreads - 1) / kPlanThreads;
  const int w0 = min(n_words, threadIdx.x * per), w1 = min(n_words, w0 + per);
  const uint32_t *km = a.keepmask + (int64_t)r * a.mask_words;
  auto kept_bits = [&](int w) -> uint32_t {  // retained tokens among positions 32w…32w+31
    if (32 * w >= nn) return 0u;
    const uint32_t v = km[w];
    const int valid = nn - 32 * w;
    return valid >= 32 ? v : (v & ((1u << valid) - 1u));
  };
  auto range_bits = [](int w, int lo, int hi) -> uint32_t {  // positions in [lo, hi)
    const int b = 32 * w;
    const int a0 = max(lo - b, 0), a1 = min(hi - b, 32);
    if (a1 <= a0) return 0u;
    const uint32_t up = a1 == 32 ? 0xFFFFFFFFu : ((1u << a1) - 1u);
    return up & ~((1u << a0) - 1u);
  };
  // m = number of retained tokens
  int my_m = 0;
  for (int w = w0; w < w1; w++) my_m += __popc(kept_bits(w));
  int m;
  block_scan_incl(my_m, sbuf, m);
  const int X = (m + a.BS - 1) / a.BS;
  const int start = (Y - X) * a.BS;
  // sources: retained before the region; holes: non-retained inside it
  int my_src = 0, my_hole = 0;
  for (int w = w0; w < w1; w++) {
    const uint32_t k = kept_bits(w);
    my_src += __popc(k & range_bits(w, 0, start));
    my_hole += __popc(~k & range_bits(w, start, end));
  }
  int ns, nh;
  int src_rank = block_scan_incl(my_src, sbuf, ns) - my_src;
  int hole_rank = block_scan_incl(my_hole, sbuf, nh) - my_hole;
  auto phys = [&](int p) -> int32_t {
    const int32_t b = bt[p / a.BS];
    if (b < 0 || b >= a.n_blocks) {
      record_error(a.status, KVC_ERR_BOUNDS);
      return -1;
    }
    return b * a.BS + p % a.BS;
  };
  for (int w = w0; w < w1; w++) {
    const uint32_t k = kept_bits(w);
    uint32_t sb = k & range_bits(w, 0, start);
    while (sb) {
      const int p = 32 * w + __ffs(sb) - 1;
      sb &= sb - 1;
      src[src_rank++] = phys(p);
    }
    uint32_t kr = k & range_bits(w, start, end);
    while (kr) {  // retained inside the region: stays where it is
      const int p = 32 * w + __ffs(kr) - 1;
      kr &= kr - 1;
      atomicOr(&tm_s[(p - start) / 32], 1u << ((p - start) % 32));
    }
    uint32_t hb = ~k & range_bits(w, start, end);
    while (hb && hole_rank < ns) {
      const int p = 32 * w + __ffs(hb) - 1;
      hb &= hb - 1;
      dst[hole_rank++] = phys(p);
      atomicOr(&tm_s[(p - start) / 32], 1u << ((p - start) % 32));
    }
  }
  // unused list entries, block lists and counts
  for (int i = ns + threadIdx.x; i < a.cap; i += kPlanThreads) {
    src[i] = -1;
    dst[i] = -1;
  }
  int32_t *fr = a.freed + (int64_t)r * a.max_blocks, *nt = a.new_table + (int64_t)r * a.max_blocks;
  for (int b = threadIdx.x; b < a.max_blocks; b += kPlanThreads) {
    fr[b] = b < Y - X ? bt[b] : -1;
    nt[b] = b < X ? bt[Y - X + b] : -1;
  }
  if (threadIdx.x == 0) {
    a.n_pairs[r] = ns;
    a.n_tail[r] = X;
    a.n_freed[r] = Y - X;
  }
  __syncthreads();
  uint32_t *tm = a.tail_mask + (int64_t)r * a.tm_words;
  for (int i = threadIdx.x; i < a.tm_words; i += kPlanThreads) tm[i] = tm_s[i];
}

// ---------------------------------------------------- compaction copy

constexpr int kCopyThreads = 256;
constexpr int kCopyRows = 4;  // rows in flight per warp

// Every (pair, layer, pool) row is one warp-wide copy of H·D·2 bytes in
// 16-byte pieces; a warp keeps kCopyRows rows in flight.  Sources and
// destinations of a plan are disjoint, so the order of the copies is free.
__global__ void __launch_bounds__(kCopyThreads)
k_tail_compact(uint16_t *kpool, uint16_t *vpool, int64_t n_slots, int L, int row_chunks,
               const int32_t *src, const int32_t *dst, const int32_t *n_pairs, int cap,
               int32_t *status) {
  const int r = blockIdx.y;
  const int np = min(max(n_pairs[r], 0), cap);
  const int64_t n_rows = (int64_t)np * L * 2;
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5);
  const int64_t n_w = (int64_t)gridDim.x * (kCopyThreads / 32);
  const int32_t *sr = src + (int64_t)r * cap, *dr = dst + (int64_t)r * cap;
  const int64_t row_elems = (int64_t)row_chunks * 8;
  for (int64_t base = wid * kCopyRows; base < n_rows; base += n_w * kCopyRows) {
    uint4 buf[kCopyRows][4];
    uint16_t *to[kCopyRows];
#pragma unroll
    for (int k = 0; k < kCopyRows; k++) {
      to[k] = nullptr;
      const int64_t i = base + k;
      if (i >= n_rows) continue;
      const int pair = (int)(i / (2 * L)), l = (int)((i / 2) % L);
      uint16_t *pool = (i & 1) ? vpool : kpool;
      const int32_t us = sr[pair], ud = dr[pair];
      if (us < 0 || us >= n_slots || ud < 0 || ud >= n_slots) {
        if (lane == 0) record_error(status, KVC_ERR_BOUNDS);
        continue;
      }
      const uint16_t *from = pool + ((int64_t)l * n_slots + us) * row_elems;
      to[k] = pool + ((int64_t)l * n_slots + ud) * row_elems;
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const int ch = lane + 32 * c;
        buf[k][c] = ch < row_chunks ? ld_stream(from + ch * 8) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int k = 0; k < kCopyRows; k++) {
      if (!to[k]) continue;
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const int ch = lane + 32 * c;
        if (ch < row_chunks) st_stream(to[k] + ch * 8, buf[k][c]);
      }
    }
    // rows wider than 128 chunks (H·D > 1024) take the remaining pieces here
    for (int k = 0; k < kCopyRows; k++) {
      if (!to[k]) continue;
      const int64_t i = base + k;
      const int pair = (int)(i / (2 * L)), l = (int)((i / 2) % L);
      const uint16_t *pool = (i & 1) ? vpool : kpool;
      const uint16_t *from = pool + ((int64_t)l * n_slots + sr[pair]) * row_elems;
      for (int ch = lane + 128; ch < row_chunks; ch += 32)
        st_stream(to[k] + ch * 8, ld_stream(from + ch * 8));
    }
  }
}

}  // namespace

bool recover_tc_supported(int H, int Hq, int D, int BS) {
  const int G = H > 0 ? Hq / H : 0;
  return H == kRecH && BS == kRecBS && Hq % H == 0 && (G == 2 || G == 4 || G == 8) &&
         (D == 64 || D == 128);
}

// Work items per CTA that keep the persistent grid balanced.
constexpr int kRecItemsPerCta = 16;

// Layer groups of a launch (with a workspace): items keep kRecPmax pages,
// so the query rows of a layer are loaded once per kRecPmax page tiles, and
// the layers are split until there are kRecItemsPerCta items per SM (at most
// one layer per item).  1 when the requests' pages already give that many.
int recover_layer_groups(int n_req, int max_blocks, int BS, int L, int H, int Hq, int D) {
  if (!recover_tc_supported(H, Hq, D, BS)) return 1;
  const int64_t items = (int64_t)n_req * ((max_blocks + kRecPmax - 1) / kRecPmax);
  const int64_t want = (int64_t)kRecItemsPerCta * device_sm_count();
  if (items >= want) return 1;
  const int64_t n = (want + items - 1) / items;
  return n > L ? L : (int)n;
}

size_t recover_ws_bytes(int n_req, int max_blocks, int BS, int L, int H, int Hq, int D) {
  const int n_lg = recover_layer_groups(n_req, max_blocks, BS, L, H, Hq, D);
  return n_lg > 1 ? (size_t)n_lg * n_req * max_blocks * BS * sizeof(float) : 0;
}

cudaError_t launch_recover_score(const uint16_t *q, const float *lse, const uint16_t *kpool,
                                 int64_t n_slots, const int32_t *block_table, int max_blocks,
                                 const int32_t *seqused, const int32_t *count, int n_req, int L,
                                 int H, int Hq, int D, int BS, float *state, void *ws,
                                 size_t ws_bytes, int32_t *status, int path, cudaStream_t s) {
  RecArgs a{};
  a.q = q;
  a.kpool = kpool;
  a.lse = lse;
  a.block_table = block_table;
  a.seqused = seqused;
  a.count = count;
  a.state = state;
  a.status = status;
  a.n_req = n_req;
  a.L = L;
  a.H = H;
  a.Hq = Hq;
  a.G = Hq / H;
  a.D = D;
  a.BS = BS;
  a.max_blocks = max_blocks;
  a.n_slots = n_slots;
  a.zscale = kLog2eR / sqrtf((float)D);
  const int n_sm = device_sm_count();
  const bool tc_ok = recover_tc_supported(H, Hq, D, BS) && (int64_t)L * n_slots * H < INT32_MAX;
  if (path == KVC_KERNEL_RECOVER_TC && !tc_ok) return cudaErrorNotSupported;
  const bool tc_path = tc_ok && path != KVC_KERNEL_RECOVER_CC;
  a.n_lg = 1;
  a.partial = nullptr;
  if (!tc_path) {
    a.P = 1;
    a.n_chunks = max_blocks;
    const size_t smem = (size_t)((Hq * D + 1) / 2 + Hq + BS * H) * sizeof(float);
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(k_recover_cc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
      if (e != cudaSuccess) return e;
    }
    k_recover_cc<<<(unsigned)((int64_t)n_req * max_blocks), kRecCcThreads, smem, s>>>(a);
    return cudaGetLastError();
  }
  // Too few pages to fill the GPU: with the caller's workspace, keep
  // kRecPmax pages per item and split the layers into groups (partial sums,
  // then a finalize); without it, fewer pages per item (one kernel).
  const int n_lg = recover_layer_groups(n_req, max_blocks, BS, L, H, Hq, D);
  int P = kRecPmax;
  if (n_lg > 1 && ws && ws_bytes >= recover_ws_bytes(n_req, max_blocks, BS, L, H, Hq, D)) {
    a.n_lg = n_lg;
    a.partial = static_cast<float *>(ws);
  } else {
    const int64_t pages = (int64_t)n_req * max_blocks;
    while (P > 1 && pages / P < (int64_t)kRecItemsPerCta * n_sm) P >>= 1;
  }
  a.P = P;
  a.n_chunks = (max_blocks + P - 1) / P;
  const int64_t n_items = (int64_t)n_req * a.n_chunks * a.n_lg;
  const int KB = D / 64, ncol = Hq;
  a.idesc = make_idesc(128, ncol);
  CUtensorMap tm_k, tm_q;
  if (!make_map(&tm_k, kpool, (uint64_t)L * n_slots * H, D, 128) ||
      !make_map(&tm_q, q, (uint64_t)n_req * L * Hq, D, (uint32_t)ncol))
    return cudaErrorInvalidValue;
  const size_t budget = 220 * 1024;
  int NS = 6;
  while (NS > 2 && RecSmem::bytes(NS, KB, ncol) > budget) NS--;
  const size_t smem = RecSmem::bytes(NS, KB, ncol);
  uint32_t cols = 32;
  while (cols < (uint32_t)(kRecNacc * ncol)) cols <<= 1;
  const unsigned grid = (unsigned)std::min<int64_t>(n_items, n_sm);
  cudaError_t e;
#define KVC_RECOVER_CASE(GV)                                                                   \
  if (a.G == GV) {                                                                             \
    e = cudaFuncSetAttribute(k_recover_tc<GV>, cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                             (int)smem);                                                       \
    if (e != cudaSuccess) return e;                                                            \
    k_recover_tc<GV><<<grid, kRecThreads, smem, s>>>(tm_k, tm_q, a, NS, cols);                 \
    e = cudaGetLastError();                                                                    \
    if (e != cudaSuccess || a.n_lg == 1) return e;                                             \
    const int64_t n_pos = (int64_t)n_req * max_blocks * BS;                                    \
    k_recover_finalize<<<(unsigned)((n_pos + 255) / 256), 256, 0, s>>>(a);                     \
    return cudaGetLastError();                                                                 \
  }
  KVC_RECOVER_CASE(2)
  KVC_RECOVER_CASE(4)
  KVC_RECOVER_CASE(8)
#undef KVC_RECOVER_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_tail_plan(const uint32_t *keepmask, int mask_words, const int32_t *seqused,
                             const int32_t *block_table, int max_blocks, int n_req, int BS,
                             int64_t n_slots, int32_t *src, int32_t *dst, int32_t *n_pairs,
                             int32_t *n_tail, int32_t *freed, int32_t *n_freed,
                             int32_t *new_table, uint32_t *tail_mask, int32_t *status,
                             cudaStream_t s) {
  PlanArgs a{};
  a.keepmask = keepmask;
  a.seqused = seqused;
  a.block_table = block_table;
  a.src = src;
  a.dst = dst;
  a.n_pairs = n_pairs;
  a.n_tail = n_tail;
  a.freed = freed;
  a.n_freed = n_freed;
  a.new_table = new_table;
  a.tail_mask = tail_mask;
  a.status = status;
  a.n_req = n_req;
  a.BS = BS;
  a.max_blocks = max_blocks;
  a.mask_words = mask_words;
  a.cap = max_blocks * BS;
  a.tm_words = (a.cap + 31) / 32;
  a.n_blocks = n_slots / BS;
  const size_t smem = (size_t)a.tm_words * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_tail_plan, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_tail_plan<<<n_req, kPlanThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_tail_compact(uint16_t *kpool, uint16_t *vpool, int64_t n_slots, int L, int H,
                                int D, const int32_t *src, const int32_t *dst,
                                const int32_t *n_pairs, int cap, int n_req, int32_t *status,
                                cudaStream_t s) {
  const int row_chunks = H * D / 8;  // 16-byte pieces per row
  const int per_req = std::max(1, 8 * device_sm_count() / n_req);
  dim3 grid((unsigned)per_req, (unsigned)n_req);
  k_tail_compact<<<grid, kCopyThreads, 0, s>>>(kpool, vpool, n_slots, L, row_chunks, src, dst,
                                               n_pairs, cap, status);
  return cudaGetLastError();
}

}  // namespace kvc
