// qmem_tc.cu — the QueryMemory logits of the rule score on the tensor cores.
//
// IntentKV §4 "Rule score": z[l,hq,j] = M[l,hq]·K[l, hq/G, S[j]]/√D for every
// history position j of a session, K read through the paged slot map (ActKV
// §2).  Sixteen consecutive positions × the 8 KV heads are 128 rows of the
// K pool, [slot][head][D] row-major; they form the A operand of one
// tcgen05.mma (M 128, K D) against the session's memory rows of one layer:
//   D[s·8 + h][c] = K[S[j0+s], h] · Mb[c],   c < 2·Hq
// where Mb = [bf16(M); bf16(M − bf16(M))] splits fp32 M into two bf16 terms
// (z = D[·][hq] + D[·][Hq+hq] keeps M to ~16 significant bits).  Each row
// uses only the G columns of its own group, the rest of the products are
// free on the tensor pipe.
//
// The A tile comes in by TMA: when the 16 positions' live slots are
// consecutive (the paged layout: one page per 16 positions) as one 128-row
// box per 64 columns; otherwise as one 8-row box per live position (a row
// gather through the slot map).  Both fill the same 128-byte-swizzled
// layout.  Dead positions (slot = sentinel) get z = −inf.
//
// Two ways to finish the rule score from the logits:
//  * spilled: the kernel writes what the CUDA-core logits kernel writes, the
//    fp32 logits (base 2) and, per 256-position tile, (max, Σ2^(z−max)) per
//    query head; k_qmem_lse and k_qmem_rule reduce them afterwards, so the
//    logits go to DRAM and come back (one fp32 per position and query head).
//  * fused (FUSED = true, groups of 2 or 4): items walk blocks of eight
//    sessions tile by tile (the block's sessions fastest), so the sessions
//    that share a prefix read each prefix tile back to back (from L2 after
//    the first) and all tiles of one (session, layer) row are done within
//    a few waves of the grid.  Three more roles join the kernel.  A publisher warp
//    counts each item the epilogue finished into its row's counter; the
//    publisher holding the row's last tile then merges the tile partials
//    into the row's LSEs and publishes them.  A share team of four warps takes this CTA's items in
//    order: once an item's row is published it forms Σ_hq 2^(z − LSE) per
//    position from the logits still in L2, writes that layer's share of the
//    rule score, and drops the logit lines from L2 without a write-back.
//    k_qmem_rule_sum adds the layers; the logits never reach DRAM.
//    Publishers wait only for epilogues, which wait for no other CTA, and
//    nothing waits for a share team, so every wait ends once every CTA is
//    resident (the launch is cooperative).

#include <algorithm>

#include "kvc_internal.cuh"
#include "tc_ptx.cuh"

namespace kvc {
namespace {

using namespace tc;

constexpr int kTJ = 256;         // positions per item (one LSE-partial tile)
constexpr int kPos = 16;         // positions per MMA tile
constexpr int kH = 8;            // KV heads: kPos · kH = 128 rows
constexpr int kThreads = 192;    // warp 0 TMA, warp 1 MMA, warps 2–5 epilogue
constexpr int kThreadsFused = 352;  // + warp 6, the publisher, and warps 7–10, the share team
constexpr int kSessBlock = 8;    // fused: sessions that walk their tiles together
constexpr int kMB = 2;           // memory-row buffers
constexpr int kNacc = 4;         // TMEM accumulators

struct QtcArgs {
  const int32_t *slot_map;  // [n_sess][N]
  float *logits;            // [n_sess][L][Hq][N], base-2 logits
  float2 *part;             // spilled: [n_sess][L][Hq][n_tiles]; fused: [n_sess][L][n_tiles][Hq]
  int *counter;             // fused: [n_sess][L] items done (+1 once the LSEs are out)
  float *lse;               // fused: [n_sess][L][Hq], base 2
  float *rule_l;            // fused: [n_sess][L][N], Σ_hq 2^(z − LSE)
  int32_t *status;
  int n_sess, L, Hq, G, D, N, n_tiles, sentinel;
  int64_t n_slots;
  float zscale;             // log2(e)/√D
  uint32_t idesc;
};

struct QtcSmem {
  uint8_t *ring, *mb;
  uint64_t *full, *empty, *mfull, *mempty, *tfull, *tempty;
  float2 *red;  // [4 warps][8 heads][G]
  float *lse_w;  // fused: [4 share warps][Hq] LSEs of the row being shared
  uint32_t *tmem_holder;
  volatile int *failed;
  int *items_done;  // fused: items whose logits and partials the epilogue wrote
  __device__ QtcSmem(uint8_t *raw, int NS, int KB, int Hq) {
    uint8_t *p = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    ring = p;
    p += (size_t)NS * KB * 16384;
    mb = p;
    p += (size_t)kMB * KB * 2 * Hq * 128;
    uint64_t *b = reinterpret_cast<uint64_t *>(p);
    full = b;
    empty = full + NS;
    mfull = empty + NS;
    mempty = mfull + kMB;
    tfull = mempty + kMB;
    tempty = tfull + kNacc;
    red = reinterpret_cast<float2 *>(tempty + kNacc);
    lse_w = reinterpret_cast<float *>(red + 4 * Hq);
    tmem_holder = reinterpret_cast<uint32_t *>(lse_w + 4 * Hq);
    failed = reinterpret_cast<volatile int *>(tmem_holder + 1);
    items_done = const_cast<int *>(failed + 1);
  }
  static size_t bytes(int NS, int KB, int Hq) {
    return 1024 + (size_t)NS * KB * 16384 + (size_t)kMB * KB * 2 * Hq * 128 +
           (size_t)(2 * NS + 2 * kMB + 2 * kNacc) * 8 + (size_t)4 * Hq * 8 +
           (size_t)4 * Hq * 4 + 16;
  }
};

// (max, sum) ⊕ (max, sum), base 2.
__device__ __forceinline__ void merge(float &m, float &s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  const float mn = fmaxf(m, m2);
  s = s * ex2(m - mn) + s2 * ex2(m2 - mn);
  m = mn;
}

template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[NC]) {
  if constexpr (NC == 16) tmem_ld16(taddr, v);
  else if constexpr (NC == 32) tmem_ld32(taddr, v);
  else tmem_ld64(taddr, v);
}

// Two TMEM loads of NC columns (a tile's hi and lo products) in flight at
// once, with one wait.
template <int NC>
__device__ __forceinline__ void tmem_ld_two(uint32_t ta, uint32_t tb, float (&va)[NC],
                                            float (&vb)[NC]) {
  if constexpr (NC == 16 || NC == 32) {
    uint32_t ra[NC], rb[NC];
    if constexpr (NC == 32) {
      tmem_issue32(ta, ra);
      tmem_issue32(tb, rb);
    } else {
      tmem_issue<16>(ta, ra);
      tmem_issue<16>(tb, rb);
    }
    tmem_wait<NC>(ra);
    // rb's loads completed at the same wait; the empty statement keeps its
    // uses below it
#pragma unroll
    for (int i = 0; i < NC; i += 4)
      asm volatile("" : "+r"(rb[i]), "+r"(rb[i + 1]), "+r"(rb[i + 2]), "+r"(rb[i + 3])::"memory");
#pragma unroll
    for (int i = 0; i < NC; i++) {
      va[i] = __uint_as_float(ra[i]);
      vb[i] = __uint_as_float(rb[i]);
    }
  } else {
    tmem_ld_cols<NC>(ta, va);
    tmem_ld_cols<NC>(tb, vb);
  }
}

// The G columns of head h's group among NC = 8·G consecutive ones.
template <int G>
__device__ __forceinline__ void group_cols(const float (&v)[8 * G], int h, float (&z)[G]) {
#pragma unroll
  for (int g = 0; g < G; g++) {
    float x = v[g];
#pragma unroll
    for (int hh = 1; hh < kH; hh++) x = (h == hh) ? v[hh * G + g] : x;
    z[g] = x;
  }
}

template <int G, bool FUSED>
__global__ void __launch_bounds__(FUSED ? kThreadsFused : kThreads, 1)
k_qmem_logits_tc(const __grid_constant__ CUtensorMap tm_k128,
                 const __grid_constant__ CUtensorMap tm_k8,
                 const __grid_constant__ CUtensorMap tm_m, QtcArgs a, int NS,
                 uint32_t tmem_cols) {
  constexpr int HQ = kH * G, NC2 = 2 * HQ;
  extern __shared__ uint8_t smem_raw[];
  const int KB = a.D / 64;
  QtcSmem sm(smem_raw, NS, KB, HQ);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n_items = (int64_t)a.n_sess * a.n_tiles * a.L;
  const uint32_t tile_bytes = (uint32_t)KB * 16384u;
  const uint32_t m_bytes = (uint32_t)(KB * NC2 * 128);

  if (threadIdx.x == 0) {
    *sm.failed = 0;
    for (int i = 0; i < NS; i++) {
      mbar_init(smem_u32(sm.full + i), 1);
      mbar_init(smem_u32(sm.empty + i), 1);
    }
    for (int i = 0; i < kMB; i++) {
      mbar_init(smem_u32(sm.mfull + i), 1);
      mbar_init(smem_u32(sm.mempty + i), 1);
    }
    for (int i = 0; i < kNacc; i++) {
      mbar_init(smem_u32(sm.tfull + i), 1);
      mbar_init(smem_u32(sm.tempty + i), 4);
    }
    *sm.items_done = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) alloc_tmem_cols(sm.tmem_holder, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_holder;

  // spilled: item → (session fastest, tile, layer), so the sessions that
  // share a prefix read its rows at about the same time, from L2 after the
  // first.  fused: item → (tile fastest, session, layer), so a row's tiles
  // are done together; the next session's prefix tiles follow one row (less
  // than a wave) later.
  auto decode = [&](int64_t item, int &r, int &tile, int &l) {
    if constexpr (FUSED) {
      // blocks of kSessBlock sessions (the last one may be smaller), walked
      // tile by tile with the block's sessions fastest
      const int64_t per_layer = (int64_t)a.n_sess * a.n_tiles;
      l = (int)(item / per_layer);
      const int64_t rem = item % per_layer;
      const int full = a.n_sess / kSessBlock;
      const int64_t in_full = (int64_t)full * kSessBlock * a.n_tiles;
      if (rem < in_full) {
        const int sb = (int)(rem / ((int64_t)kSessBlock * a.n_tiles));
        const int q = (int)(rem % ((int64_t)kSessBlock * a.n_tiles));
        tile = q / kSessBlock;
        r = sb * kSessBlock + q % kSessBlock;
      } else {
        const int rb = a.n_sess - full * kSessBlock;
        const int q = (int)(rem - in_full);
        tile = q / rb;
        r = full * kSessBlock + q % rb;
      }
    } else {
      r = (int)(item % a.n_sess);
      const int64_t rest = item / a.n_sess;
      tile = (int)(rest % a.n_tiles);
      l = (int)(rest / a.n_tiles);
    }
  };

  if (warp == 0) {
    // ------------------------------------------- TMA producer (whole warp)
    uint32_t s = 0, mi = 0;
    bool ok = true;
    for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      int r, tile, l;
      decode(item, r, tile, l);
      const int j0 = tile * kTJ;
      // memory rows of (r, l)
      const int mb_i = mi % kMB;
      if (lane == 0)
        ok = mbar_wait_bounded(smem_u32(sm.mempty + mb_i), ((mi / kMB) & 1) ^ 1, sm.failed);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        mbar_expect_tx(smem_u32(sm.mfull + mb_i), m_bytes);
        for (int kb = 0; kb < KB; kb++)
          tma_load_2d(smem_u32(sm.mb + mb_i * m_bytes + kb * NC2 * 128), &tm_m, kb * 64,
                      (r * a.L + l) * NC2, smem_u32(sm.mfull + mb_i));
      }
      mi++;
      // slots of the item's 256 positions: lane i holds positions 8i … 8i+7
      const int32_t *smap = a.slot_map + (int64_t)r * a.N;
      int32_t sv[8];
      uint32_t lv = 0u;
#pragma unroll
      for (int e = 0; e < 8; e++) {
        const int p = j0 + 8 * lane + e;
        sv[e] = p < a.N ? __ldg(smap + p) : a.sentinel;
      }
#pragma unroll
      for (int e = 0; e < 8; e++) {
        const bool live = sv[e] != a.sentinel;
        const bool in = sv[e] >= 0 && sv[e] < a.n_slots;
        if (live && !in) record_error(a.status, KVC_ERR_BOUNDS);
        lv |= (uint32_t)(live && in) << e;
      }
      // per lane: the slot its first live position implies for the block's
      // position 0, and whether every live slot follows from it
      const int half = 8 * (lane & 1);
      int64_t base = INT64_MIN;
      bool cons = true;
      if (lv) {
        const int f = __ffs(lv) - 1;
        int32_t sf = sv[0];
#pragma unroll
        for (int e = 1; e < 8; e++) sf = (e == f) ? sv[e] : sf;
        base = (int64_t)sf - (half + f);
#pragma unroll
        for (int e = 0; e < 8; e++)
          if ((lv >> e) & 1u) cons = cons && (int64_t)sv[e] == base + half + e;
      }
      const uint32_t o_lv = __shfl_xor_sync(0xFFFFFFFFu, lv, 1);
      const int64_t o_base = __shfl_xor_sync(0xFFFFFFFFu, base, 1);
      const bool o_cons = __shfl_xor_sync(0xFFFFFFFFu, cons, 1);
      const uint32_t blive = (lane & 1) ? (o_lv | (lv << 8)) : (lv | (o_lv << 8));
      const int64_t bbase = (lane & 1) ? (o_lv ? o_base : base) : (lv ? base : o_base);
      const bool regular = cons && o_cons && (!lv || !o_lv || base == o_base) && bbase >= 0 &&
                           bbase + kPos <= a.n_slots;
      for (int b = 0; b < kTJ / kPos; b++) {
        const uint32_t bl = __shfl_sync(0xFFFFFFFFu, blive, 2 * b);
        const bool reg = __shfl_sync(0xFFFFFFFFu, regular, 2 * b);
        const int64_t b0 = __shfl_sync(0xFFFFFFFFu, bbase, 2 * b);
        const int st = s % NS;
        if (lane == 0)
          ok = mbar_wait_bounded(smem_u32(sm.empty + st), ((s / NS) & 1) ^ 1, sm.failed);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        const uint32_t fb = smem_u32(sm.full + st);
        uint8_t *dst = sm.ring + st * tile_bytes;
        if (bl == 0u) {
          if (lane == 0) mbar_arrive(fb);  // nothing live: an empty tile
        } else if (reg) {
          if (lane == 0) {
            mbar_expect_tx(fb, tile_bytes);
            const int row = (int)(((int64_t)l * a.n_slots + b0) * kH);
            for (int kb = 0; kb < KB; kb++)
              tma_load_2d(smem_u32(dst + kb * 16384), &tm_k128, kb * 64, row, fb);
          }
        } else {
          if (lane == 0) mbar_expect_tx(fb, (uint32_t)(__popc(bl) * KB * 1024));
          __syncwarp();
          if ((lane >> 1) == b) {  // the two lanes holding this block's slots
#pragma unroll
            for (int e = 0; e < 8; e++)
              if ((lv >> e) & 1u) {
                const int row = (int)(((int64_t)l * a.n_slots + sv[e]) * kH);
                for (int kb = 0; kb < KB; kb++)
                  tma_load_2d(smem_u32(dst + kb * 16384 + (half + e) * 1024), &tm_k8, kb * 64,
                              row, fb);
              }
          }
        }
        __syncwarp();
        s++;
      }
    }
    if (!ok && lane == 0) *sm.failed = 1;
  } else if (warp == 1) {
    // --------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t s = 0, t = 0, mi = 0;
      bool ok = true;
      for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int mb_i = mi % kMB;
        if (!(ok = mbar_wait_bounded(smem_u32(sm.mfull + mb_i), (mi / kMB) & 1, sm.failed)))
          break;
        const uint8_t *mbase = sm.mb + mb_i * m_bytes;
        for (int b = 0; b < kTJ / kPos && ok; b++) {
          const int st = s % NS, buf = t % kNacc;
          if (!(ok = mbar_wait_bounded(smem_u32(sm.full + st), (s / NS) & 1, sm.failed))) break;
          if (!(ok = mbar_wait_bounded(smem_u32(sm.tempty + buf), ((t / kNacc) & 1) ^ 1,
                                       sm.failed)))
            break;
          tc_fence_after();
          const uint8_t *kt = sm.ring + st * tile_bytes;
          const uint32_t d = tmem + (uint32_t)(buf * NC2);
          for (int kk = 0; kk < 4 * KB; kk++) {
            const uint32_t koff = (uint32_t)(kk & 3) * 32u;
            const uint64_t adesc = smem_desc(smem_u32(kt + (kk >> 2) * 16384) + koff);
            const uint64_t bdesc = smem_desc(smem_u32(mbase + (kk >> 2) * NC2 * 128) + koff);
            mma_bf16(d, adesc, bdesc, a.idesc, kk > 0);
          }
          mma_commit(smem_u32(sm.empty + st));
          mma_commit(smem_u32(sm.tfull + buf));
          s++;
          t++;
        }
        if (ok) mma_commit(smem_u32(sm.mempty + mb_i));
        mi++;
      }
      if (!ok) *sm.failed = 1;
    }
    __syncwarp();
  } else if (warp < 6) {
    // --------------------------------------------------- epilogue
    // The four warps pass the same named barriers in the same order whatever
    // happens: a failed wait skips work, never a barrier, and the warps agree
    // on failure (named_sync_and) before leaving the item loop together.
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;
    const int sp = row / kH, h = row % kH;  // position in the tile, KV head
    const int et = (warp - 2) * 32 + lane;  // 0 … 127
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    uint64_t keep = 0;
    if constexpr (FUSED) keep = l2_evict_last();
    uint32_t t = 0;
    bool ok = true;
    int n_done = 0;
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
      int r, tile, l;
      decode(item, r, tile, l);
      const int j0 = tile * kTJ;
      const int32_t *smap = a.slot_map + (int64_t)r * a.N;
      float *lrow = a.logits + (((int64_t)r * a.L + l) * HQ + h * G) * a.N;
      float m[G], sum[G];
#pragma unroll
      for (int g = 0; g < G; g++) {
        m[g] = -INFINITY;
        sum[g] = 0.f;
      }
      // liveness of this thread's position in each of the item's 16 tiles,
      // loaded together so that one load latency is paid per item, not per tile
      uint32_t live_mask = 0u;
#pragma unroll
      for (int b = 0; b < kTJ / kPos; b++) {
        const int j = j0 + b * kPos + sp;
        const int32_t u = j < a.N ? __ldg(smap + j) : a.sentinel;
        live_mask |= (uint32_t)(u != a.sentinel && u >= 0 && u < a.n_slots) << b;
      }
      for (int b = 0; b < kTJ / kPos; b++) {
        const int j = j0 + b * kPos + sp;
        const bool live = (live_mask >> b) & 1u;
        const int buf = t % kNacc;
        const bool got =
            ok && mbar_wait_bounded(smem_u32(sm.tfull + buf), (t / kNacc) & 1, sm.failed);
        ok = __all_sync(0xFFFFFFFFu, got);
        float zh[G], zl[G];
        if (ok) {
          tc_fence_after();
          const uint32_t taddr = tmem + lane_base + (uint32_t)(buf * NC2);
          float vh[HQ], vl[HQ];
          tmem_ld_two<HQ>(taddr, taddr + HQ, vh, vl);
          group_cols<G>(vh, h, zh);
          group_cols<G>(vl, h, zl);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(sm.tempty + buf));
        t++;
        if (!ok) continue;
#pragma unroll
        for (int g = 0; g < G; g++) {
          const float z = (zh[g] + zl[g]) * a.zscale;
          if (j < a.N) {
            float *dst = lrow + (int64_t)g * a.N + j;
            const float zv = live ? z : -INFINITY;
            if constexpr (FUSED) st_hint_f32(dst, zv, keep);
            else *dst = zv;
          }
          if (live) {
            if (z > m[g]) {
              sum[g] = sum[g] * ex2(m[g] - z) + 1.f;
              m[g] = z;
            } else {
              sum[g] += ex2(z - m[g]);
            }
          }
        }
      }
      // (max, sum) per query head over the item's 256 positions
#pragma unroll
      for (int g = 0; g < G; g++) {
#pragma unroll
        for (int o = 8; o < 32; o <<= 1) {
          const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m[g], o);
          const float s2 = __shfl_xor_sync(0xFFFFFFFFu, sum[g], o);
          merge(m[g], sum[g], m2, s2);
        }
      }
      if (lane < kH)
#pragma unroll
        for (int g = 0; g < G; g++) sm.red[(quarter * kH + h) * G + g] = make_float2(m[g], sum[g]);
      ok = named_sync_and(1, 128, ok);
      if (ok && et < HQ) {
        float mm = -INFINITY, ss = 0.f;
        for (int q4 = 0; q4 < 4; q4++) {
          const float2 v = sm.red[q4 * HQ + et];
          merge(mm, ss, v.x, v.y);
        }
        const int64_t rl = (int64_t)r * a.L + l;
        a.part[FUSED ? (rl * a.n_tiles + tile) * HQ + et : (rl * HQ + et) * a.n_tiles + tile] =
            make_float2(mm, ss);
      }
      named_sync(1, 128);
      if (!ok) break;
      if constexpr (FUSED) {
        // hand the item to the publisher: every epilogue write of it comes
        // before this release (the barrier above orders the other threads')
        n_done++;
        if (et == 0) st_release_cta(sm.items_done, n_done);
      }
    }
    if (!ok) {
      *sm.failed = 1;
      if (lane == 0) record_error(a.status, KVC_ERR_TIMEOUT);
    }
  } else if (warp == 6) {
    // --------------------------------------------- publisher (fused only)
    // Counts each item the epilogue finished into its (session, layer) row;
    // the CTA holding the row's last tile waits for the row's count, merges
    // the row's tile partials into its LSEs and publishes them (the counter
    // then reads n_tiles + 1).  Waits only for epilogues, which wait for no
    // other CTA.
    if constexpr (FUSED) {
      bool ok = true;
      int k = 0;
      for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x, k++) {
        if (lane == 0) {
          const uint64_t t0 = global_ns();
          while (ld_acquire_cta(sm.items_done) < k + 1) {
            if (*sm.failed || global_ns() - t0 > 1000000000ull) {
              ok = false;
              break;
            }
            __nanosleep(256);
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        int r, tile, l;
        decode(item, r, tile, l);
        const int64_t rl = (int64_t)r * a.L + l;
        // release the epilogue's writes of the item (acquired above at CTA
        // scope) to the row
        if (lane == 0) atom_add_acq_rel_gpu(a.counter + rl, 1);
        if (tile == a.n_tiles - 1) {
          // The row's merger: the CTA holding its last tile, which is this
          // CTA's last item of the row, so the wait below never waits on
          // this publisher.  (The last finisher, the natural choice, is
          // mostly one slow CTA, which then falls further behind.)
          if (lane == 0) {
            const uint64_t t0 = global_ns();
            while (ld_acquire_gpu(a.counter + rl) < a.n_tiles) {
              if (*sm.failed || global_ns() - t0 > 1000000000ull) {
                ok = false;
                break;
              }
              __nanosleep(128);
            }
          }
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          __syncwarp();  // lane 0's acquire orders the other lanes' loads too
          if (!ok) break;
          // the row's tile partials, [tile][Hq]: lanes take consecutive query
          // heads (one 256-byte read per instruction for 32 heads), 32 tiles
          // in flight, merged in tile order
          for (int hq = lane; hq < HQ; hq += 32) {
            const float2 *src = a.part + rl * a.n_tiles * HQ + hq;
            float mm = -INFINITY, ss = 0.f;
            for (int t0 = 0; t0 < a.n_tiles; t0 += 32) {
              float2 v[32];
#pragma unroll
              for (int kk = 0; kk < 32; kk++)
                v[kk] = t0 + kk < a.n_tiles ? __ldcg(src + (int64_t)(t0 + kk) * HQ)
                                            : make_float2(-INFINITY, 0.f);
#pragma unroll
              for (int kk = 0; kk < 32; kk++) merge(mm, ss, v[kk].x, v[kk].y);
            }
            a.lse[rl * HQ + hq] = mm == -INFINITY ? -INFINITY : mm + log2f(ss);
          }
          __syncwarp();
          if (lane == 0) atom_add_acq_rel_gpu(a.counter + rl, 1);
        }
      }
      if (!ok) {
        *sm.failed = 1;
        if (lane == 0) record_error(a.status, KVC_ERR_TIMEOUT);
      }
    }
  } else {
    // ---------------------------------------------- share team (fused only)
    // Each warp takes 64 of an item's 256 positions, for this CTA's items in
    // order: once the item's row has published its LSEs, it forms
    // Σ_hq 2^(z − LSE) per position from the logits still in L2, writes that
    // layer's share, and drops its whole 128-byte logit lines from L2.  No
    // other role waits for it.
    if constexpr (FUSED) {
      const int w = warp - 7;
      float *lw = sm.lse_w + w * HQ;
      bool ok = true;
      for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        int r, tile, l;
        decode(item, r, tile, l);
        const int64_t rl = (int64_t)r * a.L + l;
        if (lane == 0) {
          const uint64_t t0 = global_ns();
          while (ld_acquire_gpu(a.counter + rl) < a.n_tiles + 1) {
            if (*sm.failed || global_ns() - t0 > 1000000000ull) {
              ok = false;
              break;
            }
            __nanosleep(256);
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        __syncwarp();  // lane 0's acquire orders the other lanes' loads too
        if (!ok) break;
        for (int hq = lane; hq < HQ; hq += 32) lw[hq] = __ldcg(a.lse + rl * HQ + hq);
        __syncwarp();
        const int j0 = tile * kTJ;
        const int valid = min(kTJ, a.N - j0);
        const float *zb = a.logits + rl * HQ * a.N + j0;
#pragma unroll 1
        for (int hf = 0; hf < 2; hf++) {
          const int pp = 64 * w + 32 * hf + lane;
          float acc = 0.f;
#pragma unroll 1
          for (int h0 = 0; h0 < HQ; h0 += 16) {
            float z[16];
#pragma unroll
            for (int kk = 0; kk < 16; kk++)
              z[kk] = pp < valid ? __ldcg(zb + (int64_t)(h0 + kk) * a.N + pp) : -INFINITY;
#pragma unroll
            for (int kk = 0; kk < 16; kk++) {
              const float L2v = lw[h0 + kk];
              if (L2v != -INFINITY) acc += ex2(z[kk] - L2v);
            }
          }
          if (pp < valid) a.rule_l[rl * a.N + j0 + pp] = acc;
        }
        // every value this warp read has been used: drop its lines
        __syncwarp();
        for (int idx = lane; idx < 2 * HQ; idx += 32) {
          const int c0 = 64 * w + 32 * (idx / HQ), hq = idx % HQ;
          if (c0 + 32 > valid) continue;
          const float *line = zb + (int64_t)hq * a.N + c0;
          if ((reinterpret_cast<uintptr_t>(line) & 127u) == 0u) l2_discard_line(line);
        }
      }
      if (!ok) {
        *sm.failed = 1;
        if (lane == 0) record_error(a.status, KVC_ERR_TIMEOUT);
      }
    }
  }

  // ------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*sm.failed && threadIdx.x == 0) {
    record_error(a.status, KVC_ERR_TIMEOUT);
    for (int i = 0; i < NS; i++) {
      mbar_drain(smem_u32(sm.full + i), 0);
      mbar_drain(smem_u32(sm.full + i), 1);
    }
    for (int i = 0; i < kMB; i++) {
      mbar_drain(smem_u32(sm.mfull + i), 0);
      mbar_drain(smem_u32(sm.mfull + i), 1);
    }
    for (int i = 0; i < kNacc; i++) {
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

// Mb[(r·L + l)·2Hq + hq] = bf16(M), Mb[… + Hq + hq] = bf16(M − bf16(M)).
__global__ void __launch_bounds__(256)
k_qmem_split(const float *__restrict__ M, uint16_t *__restrict__ mb, int64_t rows_rl, int Hq,
             int D) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t n = rows_rl * Hq * D;
  if (i >= n) return;
  const int64_t rl = i / ((int64_t)Hq * D), rem = i - rl * Hq * D;
  const float x = M[i];
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
  mb[rl * 2 * Hq * D + rem] = *reinterpret_cast<const uint16_t *>(&hi);
  mb[rl * 2 * Hq * D + (int64_t)Hq * D + rem] = *reinterpret_cast<const uint16_t *>(&lo);
}

bool make_map_box8(CUtensorMap *m, const void *base, uint64_t rows, int D) {
  return make_map(m, base, rows, D, 8);
}

}  // namespace

bool qmem_tc_supported(int H, int Hq, int D, int64_t L, int64_t n_slots) {
  const int G = H > 0 ? Hq / H : 0;
  return H == kH && Hq % H == 0 && (G == 2 || G == 4 || G == 8) && (D == 64 || D == 128) &&
         L * n_slots * kH < INT32_MAX;
}

size_t qmem_tc_mb_bytes(int n_sess, int L, int Hq) {
  return (size_t)n_sess * L * 2 * Hq * 128 * sizeof(uint16_t);
}

cudaError_t launch_qmem_logits_tc(const float *M, const uint16_t *kpool, const int32_t *slot_map,
                                  int32_t sentinel, float *logits, float2 *part, float *lse,
                                  int *counter, float *rule_l, uint16_t *mb, int n_sess, int L,
                                  int H, int Hq, int D, int N, int64_t n_slots, int n_tiles,
                                  bool fused, int32_t *status, cudaStream_t s) {
  const int64_t rows_rl = (int64_t)n_sess * L;
  const int64_t n = rows_rl * Hq * D;
  QtcArgs a{};
  a.slot_map = slot_map;
  a.logits = logits;
  a.part = part;
  a.counter = counter;
  a.lse = lse;
  a.rule_l = rule_l;
  a.status = status;
  a.n_sess = n_sess;
  a.L = L;
  a.Hq = Hq;
  a.G = Hq / H;
  a.D = D;
  a.N = N;
  a.n_tiles = n_tiles;
  a.sentinel = sentinel;
  a.n_slots = n_slots;
  a.zscale = 1.4426950408889634f / sqrtf((float)D);
  a.idesc = make_idesc(128, 2 * Hq);
  CUtensorMap tm_k128, tm_k8, tm_m;
  const uint64_t krows = (uint64_t)L * n_slots * kH;
  if (!make_map(&tm_k128, kpool, krows, D, 128) || !make_map_box8(&tm_k8, kpool, krows, D) ||
      !make_map(&tm_m, mb, (uint64_t)rows_rl * 2 * Hq, D, (uint32_t)(2 * Hq)))
    return cudaErrorInvalidValue;
  const int KB = D / 64;
  int NS = 6;
  while (NS > 2 && QtcSmem::bytes(NS, KB, Hq) > 220 * 1024) NS--;
  const size_t smem = QtcSmem::bytes(NS, KB, Hq);
  uint32_t cols = 32;
  while (cols < (uint32_t)(kNacc * 2 * Hq)) cols <<= 1;
  const int64_t n_items = (int64_t)n_sess * n_tiles * L;
  int64_t grid = std::min<int64_t>(n_items, device_sm_count());
  cudaError_t e = cudaSuccess;
  // kernel of group size GV and the chosen finish
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t e2 =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e2 != cudaSuccess) return e2;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(fused ? kThreadsFused : kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    if (fused) {
      // a CTA's share team waits for rows that other CTAs finish: all of
      // them must be resident
      int per_sm = 0;
      e2 = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreadsFused, smem);
      if (e2 != cudaSuccess) return e2;
      if (per_sm < 1) return cudaErrorNotSupported;
      grid = std::min<int64_t>(grid, (int64_t)per_sm * device_sm_count());
      e2 = cudaMemsetAsync(counter, 0, (size_t)rows_rl * sizeof(int), s);
      if (e2 != cudaSuccess) return e2;
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
    }
    cfg.gridDim = dim3((unsigned)grid);
    k_qmem_split<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(M, mb, rows_rl, Hq, D);
    e2 = cudaGetLastError();
    if (e2 != cudaSuccess) return e2;
    return cudaLaunchKernelEx(&cfg, kern, tm_k128, tm_k8, tm_m, a, NS, cols);
  };
  switch (a.G) {
    case 2: e = fused ? launch(k_qmem_logits_tc<2, true>) : launch(k_qmem_logits_tc<2, false>); break;
    case 4: e = fused ? launch(k_qmem_logits_tc<4, true>) : launch(k_qmem_logits_tc<4, false>); break;
    // G = 8: the epilogue's registers leave no room for the fused finish's
    // extra warps (352 threads at 254 registers exceed the register file)
    case 8: e = fused ? cudaErrorNotSupported : launch(k_qmem_logits_tc<8, false>); break;
    default: return cudaErrorInvalidValue;
  }
  return e;
}

}  // namespace kvc
