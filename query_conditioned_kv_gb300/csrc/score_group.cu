// score_group.cu — tensor-core Mean-K scorer for wide query sets: more than
// 128 and at most 192 query rows per KV head (G·W, e.g. 6 query heads × a
// 32-query window), D = 128.
//
// The quantity is the one every scorer of this library computes (KVMem
// "Query-conditioned retrieval"; ActKV §7.1 aggregation): for a unit (layer
// l, KV head h, session r) and query row ρ = g·W + w,
//   z[ρ,b] = q[ρ]·meank[b]/sqrt(D),   LSE[ρ] = log Σ_b e^z,
//   score[b] = (1/W) Σ_w max_g exp(z[g·W+w,b] − LSE[g·W+w]).
//
// At these widths a unit's logits (rows × blocks) are far larger than the
// tensor memory of the SMs that share the unit, so every tile is multiplied
// twice: once for the row LSEs, once for the scores.  The design keeps both
// products on the fast MMA shapes and the second read of each Mean-K tile in
// L2:
//   * tiles of 256 blocks.  Pass 1 multiplies the query rows (M, two row
//     tiles of 128: rows 0–127 and 128–255, the rows past R ignored) by the
//     tile (N = 256), each row tile a job of its own in a 256-column TMEM
//     buffer.  Pass 2 multiplies the tile's two 128-block halves (M) by the
//     R query rows (N = R), one job per half.  (An M = 128 × N = 256
//     instruction runs at about 1.7 times the rate of N = 128, and M = 64
//     costs as much as M = 128, so padding rows to 256 is the cheaper way.)
//   * groups of g CTAs (one CTA per SM, the grid launched cooperatively so
//     that every CTA is resident) share a unit: CTA rank takes the unit's
//     tiles rank', rank' + g, … (rank' rotating from unit to unit so that the
//     extra tiles spread).  The g CTAs exchange their row partials (max,
//     Σ2^(z−max)) through L2: each publishes its partials and bumps the
//     group's counter; each waits (bounded) for the counter and merges the g
//     partials in rank order, so the result does not depend on timing.
//     With g chosen so that a CTA holds about seven tiles of a unit, only
//     #SMs/g units are in flight (8 × 8 MB for the 27B-class workload) and
//     the second read of a tile hits L2; the loads carry evict-last and
//     evict-first hints.
//   * a CTA runs pass 1 of its next unit's first tiles while its group
//     exchanges, so the tensor pipe keeps working through the exchange:
//         P1(u0) | P1a(u1) P2(u0) P1b(u1) | P1a(u2) P2(u1) P1b(u2) | … | P2(u_last)
//   * roles: warp 0 issues TMA, warp 1 issues tcgen05.mma into TMEM buffer
//     j mod 2 for job j (a row tile or a block half), warps 4–11 (two
//     warpgroups) read every job back, each warp one lane quarter and one
//     half of the job's columns; setmaxnreg moves registers from the control
//     warpgroup to them, so that TMEM loads can run ahead of the arithmetic.
// Every wait is bounded (1 s of %globaltimer) and records KVC_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <math.h>

#include <atomic>

#include "kvc_internal.cuh"
#include "tc_ptx.cuh"

namespace kvc {
namespace {

using namespace tc;

constexpr int kGD = 128;                // head dim
constexpr int kGTB = 256;               // Mean-K blocks per tile (pass-1 N)
constexpr uint32_t kGSlot = 32768;      // ring slot: one K-half of a tile, or a half-tile
constexpr int kGMaxR = 192;             // widest query-row set
constexpr int kGLook = 3;               // next-unit tiles run ahead of an exchange
constexpr int kGThreads = 384;          // warpgroup 0: TMA, MMA (+2 idle warps); 1-2: epilogue
constexpr int kGCtlRegs = 80;           // registers of warpgroup 0 after setmaxnreg.dec
constexpr int kGEpiRegs = 208;          // registers of warpgroups 1-2 after setmaxnreg.inc
constexpr uint32_t kGBufCols = 256;     // TMEM columns per job buffer
constexpr size_t kGSmemMax = 232448;    // the opt-in per-CTA maximum
constexpr int kGTarget = 7;             // tiles of a unit a CTA aims to hold

struct GroupArgs {
  float *scores;
  const int64_t *blk_off;
  int32_t *status;
  int *counter;   // [n_groups]: partials published so far (g per unit)
  float2 *part;   // [n_groups][2][g][256] row partials (max, Σ2^(z−max)), base 2
  int L, H, n_sess, R, n2, g, n_groups, max_tiles, ns;
  int64_t nb_total;
  float zscale;   // log2(e)/sqrt(D)
  uint32_t idesc1, idesc2;
  uint32_t q_half;  // bytes of one K-half of a q buffer (R·128)
};

struct GroupSmem {
  uint8_t *q, *ring;
  uint64_t *full, *empty, *tfull, *tempty, *qfull, *qempty;
  uint32_t *tmem_holder;
  volatile int *failed;
  float *lse;   // [kGMaxR] row LSEs (base 2) of the unit in pass 2
  float *comb;  // [2][128] pass-2 partial sums handed from the upper to the lower half
  __device__ GroupSmem(uint8_t *raw, uint32_t q_half, int ns) {
    uint8_t *p = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    q = p;  // two buffers of 2·q_half; pass 1's second row tile reads past a
            // buffer's end into the next region (rows ≥ R, ignored)
    p += 4 * (size_t)q_half;
    ring = p;
    p += (size_t)ns * kGSlot;
    uint64_t *b = reinterpret_cast<uint64_t *>(p);
    full = b;
    empty = full + ns;
    tfull = empty + ns;
    tempty = tfull + 2;
    qfull = tempty + 2;
    qempty = qfull + 2;
    tmem_holder = reinterpret_cast<uint32_t *>(qempty + 2);
    failed = reinterpret_cast<volatile int *>(tmem_holder + 1);
    lse = reinterpret_cast<float *>(tmem_holder + 4);
    comb = lse + kGMaxR;
  }
  static size_t bytes(uint32_t q_half, int ns) {
    return 1024 + 4 * (size_t)q_half + (size_t)ns * kGSlot + (2 * (size_t)ns + 8) * 8 + 16 +
           kGMaxR * 4 + 256 * 4;
  }
};

// A unit of this group and this CTA's share of it.
struct GUnit {
  int l, h, r, nb, n_tiles, my, look, mk_row0, q_row0;
  int rank_eff;  // which residue mod g this CTA takes in this unit
  int64_t b0;
};

__device__ __forceinline__ GUnit gunit(const GroupArgs &a, int i, int grp, int rank) {
  GUnit u;
  const int unit = grp + i * a.n_groups;
  u.r = unit % a.n_sess;
  const int lh = unit / a.n_sess;
  u.h = lh % a.H;
  u.l = lh / a.H;
  const int64_t b0 = a.blk_off[u.r], b1 = a.blk_off[u.r + 1];
  const bool ok =
      b0 >= 0 && b1 > b0 && b1 <= a.nb_total && b1 - b0 <= (int64_t)a.max_tiles * kGTB;
  u.b0 = ok ? b0 : 0;
  u.nb = ok ? (int)(b1 - b0) : 0;
  u.n_tiles = (u.nb + kGTB - 1) / kGTB;
  u.rank_eff = (rank + i) % a.g;
  u.my = u.n_tiles > u.rank_eff ? (u.n_tiles - u.rank_eff + a.g - 1) / a.g : 0;
  u.look = i == 0 ? 0 : (u.my < kGLook ? u.my : kGLook);
  u.mk_row0 = (int)(((int64_t)u.l * a.H + u.h) * a.nb_total + u.b0);
  u.q_row0 = (int)((((int64_t)u.l * a.n_sess + u.r) * a.H + u.h) * a.R);
  return u;
}

__device__ __forceinline__ int group_units(const GroupArgs &a, int grp) {
  const int n_units = a.L * a.H * a.n_sess;
  return grp < n_units ? (n_units - grp + a.n_groups - 1) / a.n_groups : 0;
}

__device__ __forceinline__ void lse_merge_g(float &m, float &s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  const float mn = fmaxf(m, m2);
  s = s * exp2f(m - mn) + s2 * exp2f(m2 - mn);
  m = mn;
}

// Pass 1 of this warp's 128 columns (blocks) of one row tile for this
// lane's query row: online (max, Σ2^(z·zs − max)) over the `valid` columns,
// 64 at a time (two TMEM loads per job).  Column j adds into accumulator
// j mod 8 (four packed pairs).
__device__ __forceinline__ void group_pass1(uint32_t taddr, int valid, float zs, float &pm,
                                            float &ps) {
  pm = -INFINITY;
  ps = 0.f;
  const int nch = valid <= 0 ? 0 : (valid >= 128 ? 2 : (valid + 63) / 64);
  const uint64_t zs2 = pk2(zs, zs);
#pragma unroll 1
  for (int c = 0; c < nch; c++) {
    float v[64];
    tmem_ld64(taddr + (uint32_t)(64 * c), v);
    const int nv = valid - 64 * c;
    if (nv < 64) {
#pragma unroll
      for (int j = 0; j < 64; j++)
        if (j >= nv) v[j] = -INFINITY;
    }
    float m0 = max3(v[0], v[1], v[2]), m1 = max3(v[3], v[4], v[5]);
    float m2 = max3(v[6], v[7], v[8]), m3 = max3(v[9], v[10], v[11]);
#pragma unroll
    for (int j = 12; j < 60; j += 8) {
      m0 = max3(m0, v[j], v[j + 1]);
      m1 = max3(m1, v[j + 2], v[j + 3]);
      m2 = max3(m2, v[j + 4], v[j + 5]);
      m3 = max3(m3, v[j + 6], v[j + 7]);
    }
    m0 = max3(m0, v[60], v[61]);
    m1 = max3(m1, v[62], v[63]);
    const float mn = fmaxf(pm, fmaxf(max3(m0, m1, m2), m3) * zs);
    const uint64_t nmn2 = pk2(-mn, -mn);
    uint64_t acc[4];
    acc[0] = pk2((pm == -INFINITY) ? 0.f : ps * ex2(pm - mn), 0.f);
#pragma unroll
    for (int k = 1; k < 4; k++) acc[k] = pk2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 64; j += 2) {
      float x0, x1;
      upk2(fma2(pk2(v[j], v[j + 1]), zs2, nmn2), x0, x1);
      acc[(j & 7) >> 1] = add2(acc[(j & 7) >> 1], pk2(ex2(x0), ex2(x1)));
    }
    float a8[8];
#pragma unroll
    for (int k = 0; k < 4; k++) upk2(acc[k], a8[2 * k], a8[2 * k + 1]);
    pm = mn;
    ps = ((a8[0] + a8[1]) + (a8[2] + a8[3])) + ((a8[4] + a8[5]) + (a8[6] + a8[7]));
  }
}

// Pass 2 of this warp's half of the window positions for this lane's block:
// for w in [half·W/2, (half+1)·W/2), the max over the G heads of
// z·zs − LSE (columns g·W + w, each head's W/2 columns one TMEM load, the
// next head's load in flight), then Σ_w 2^max over this half.
template <int W>
__device__ __forceinline__ float group_pass2(uint32_t taddr, int G, int half, float zs,
                                             const float *lse) {
  constexpr int HW = W / 2;
  float mw[HW];
#pragma unroll
  for (int w = 0; w < HW; w++) mw[w] = -INFINITY;
  const uint64_t zs2 = pk2(zs, zs);
  // head g's columns: x = z·zs − LSE, max into mw
  auto fold = [&](const uint32_t(&rr)[HW], int g) {
    const float4 *l4 = reinterpret_cast<const float4 *>(lse + g * W + half * HW);
#pragma unroll
    for (int j = 0; j < HW; j += 4) {
      const float4 Lv = l4[j / 4];
      float x0, x1, x2, x3;
      upk2(fma2(pk2(__uint_as_float(rr[j]), __uint_as_float(rr[j + 1])), zs2, pk2(-Lv.x, -Lv.y)),
           x0, x1);
      upk2(fma2(pk2(__uint_as_float(rr[j + 2]), __uint_as_float(rr[j + 3])), zs2,
                pk2(-Lv.z, -Lv.w)),
           x2, x3);
      mw[j] = fmaxf(mw[j], x0);
      mw[j + 1] = fmaxf(mw[j + 1], x1);
      mw[j + 2] = fmaxf(mw[j + 2], x2);
      mw[j + 3] = fmaxf(mw[j + 3], x3);
    }
  };
  uint32_t ra[HW], rb[HW];
  const uint32_t col0 = (uint32_t)(half * HW);
  tmem_issue<HW>(taddr + col0, ra);
  tmem_wait<HW>(ra);
#pragma unroll 1
  for (int g = 0; g < G; g += 2) {  // head g in ra, head g + 1 in rb
    if (g + 1 < G) tmem_issue<HW>(taddr + col0 + (uint32_t)((g + 1) * W), rb);
    fold(ra, g);
    if (g + 1 < G) {
      tmem_wait<HW>(rb);
      if (g + 2 < G) tmem_issue<HW>(taddr + col0 + (uint32_t)((g + 2) * W), ra);
      fold(rb, g + 1);
      if (g + 2 < G) tmem_wait<HW>(ra);
    }
  }
  float acc = 0.f;
#pragma unroll
  for (int w = 0; w < HW; w++) acc += ex2(mw[w]);
  return acc;
}

template <int W>
__global__ void __launch_bounds__(kGThreads, 1)
k_score_group(const __grid_constant__ CUtensorMap tm_mk256,
              const __grid_constant__ CUtensorMap tm_mk128,
              const __grid_constant__ CUtensorMap tm_q, GroupArgs a) {
  extern __shared__ uint8_t smem_raw[];
  GroupSmem sm(smem_raw, a.q_half, a.ns);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = blockIdx.x / a.g, rank = blockIdx.x % a.g;
  const int n_mine = group_units(a, grp);
  const int ns = a.ns;
  const uint32_t q_buf = 2 * a.q_half;

  if (threadIdx.x == 0) {
    *sm.failed = 0;
    for (int i = 0; i < ns; i++) {
      mbar_init(smem_u32(sm.full + i), 1);
      mbar_init(smem_u32(sm.empty + i), 1);
    }
    for (int i = 0; i < 2; i++) {
      mbar_init(smem_u32(sm.tfull + i), 1);
      mbar_init(smem_u32(sm.tempty + i), 8);  // every epilogue warp reads every job
      mbar_init(smem_u32(sm.qfull + i), 1);
      mbar_init(smem_u32(sm.qempty + i), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) alloc_tmem_cols(sm.tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_holder;
  // Registers move from the control warpgroup (TMA, MMA, two idle warps) to
  // the two epilogue warpgroups: 128·kGCtlRegs + 256·kGEpiRegs stays within
  // the 384·168 the block is launched with.  Each branch starts with its
  // setmaxnreg, so the budget covers all the code of that role.

  // The step order every role walks, for this CTA's units u_0 … u_{n−1}:
  //   P1(u0) | P1a(u1) P2(u0) P1b(u1) | … | P2(u_{n−1})
  // with P1a = the first `look` tiles of a unit and P1b = the rest.
  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kGCtlRegs));
  if (warp == 0) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t keep = l2_evict_last(), drop = l2_evict_first();
      uint32_t s = 0, qi = 0;
      bool ok = true;
      auto take_slot = [&](uint32_t bytes) -> int {
        const int slot = (int)(s % (uint32_t)ns);
        if (!wait_or_abort(smem_u32(sm.empty + slot), ((s / ns) & 1) ^ 1, sm.failed)) return -1;
        mbar_expect_tx(smem_u32(sm.full + slot), bytes);
        s++;
        return slot;
      };
      auto p1_tiles = [&](const GUnit &u, int j0, int j1) {
        for (int j = j0; j < j1 && ok; j++) {
          const int row = u.mk_row0 + (u.rank_eff + j * a.g) * kGTB;
          for (int kb = 0; kb < 2 && ok; kb++) {
            const int slot = take_slot(kGSlot);
            if (slot < 0) {
              ok = false;
              break;
            }
            tma_load_2d_hint(smem_u32(sm.ring + slot * kGSlot), &tm_mk256, kb * 64, row,
                             smem_u32(sm.full + slot), keep);
          }
        }
      };
      auto p2_tiles = [&](const GUnit &u) {
        for (int j = 0; j < u.my && ok; j++)
          for (int hf = 0; hf < 2 && ok; hf++) {
            const int row = u.mk_row0 + (u.rank_eff + j * a.g) * kGTB + hf * 128;
            const int slot = take_slot(kGSlot);
            if (slot < 0) {
              ok = false;
              break;
            }
            for (int kb = 0; kb < 2; kb++)
              tma_load_2d_hint(smem_u32(sm.ring + slot * kGSlot + kb * (kGSlot / 2)), &tm_mk128,
                               kb * 64, row, smem_u32(sm.full + slot), drop);
          }
      };
      GUnit prev{};
      for (int i = 0; i < n_mine && ok; i++) {
        const GUnit u = gunit(a, i, grp, rank);
        if (u.nb == 0 && rank == 0) record_error(a.status, KVC_ERR_BOUNDS);
        if (u.my > 0) {  // the unit's query rows
          const int qb = qi & 1;
          if (!(ok = wait_or_abort(smem_u32(sm.qempty + qb), ((qi >> 1) & 1) ^ 1, sm.failed)))
            break;
          mbar_expect_tx(smem_u32(sm.qfull + qb), q_buf);
          for (int kb = 0; kb < 2; kb++)
            tma_load_2d(smem_u32(sm.q + qb * q_buf + kb * a.q_half), &tm_q, kb * 64, u.q_row0,
                        smem_u32(sm.qfull + qb));
          qi++;
        }
        p1_tiles(u, 0, u.look);
        if (i > 0) p2_tiles(prev);
        p1_tiles(u, u.look, u.my);
        prev = u;
      }
      if (ok && n_mine > 0) p2_tiles(prev);
      if (!ok) *sm.failed = 1;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t s = 0, job = 0, qi = 0;
      bool ok = true;
      auto wait_slot = [&]() -> int {
        const int slot = (int)(s % (uint32_t)ns);
        if (!wait_or_abort(smem_u32(sm.full + slot), (s / ns) & 1, sm.failed)) return -1;
        s++;
        return slot;
      };
      auto wait_buf = [&]() -> int {
        const int buf = (int)(job & 1);
        if (!wait_or_abort(smem_u32(sm.tempty + buf), ((job >> 1) & 1) ^ 1, sm.failed))
          return -1;
        tc_fence_after();
        return buf;
      };
      auto p1_tiles = [&](int qb, int n) {
        for (int j = 0; j < n && ok; j++) {
          const int s0 = wait_slot(), s1 = s0 < 0 ? -1 : wait_slot();
          if (s1 < 0) {
            ok = false;
            break;
          }
          for (int rt = 0; rt < 2; rt++) {
            const int buf = wait_buf();
            if (buf < 0) {
              ok = false;
              break;
            }
            const uint32_t qa = smem_u32(sm.q + qb * q_buf) + (uint32_t)rt * 16384u;
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {
              const uint32_t k32 = (uint32_t)(kk & 3) * 32u;
              const uint32_t mb = smem_u32(sm.ring + (kk >> 2 ? s1 : s0) * kGSlot);
              mma_bf16(tmem + (uint32_t)buf * kGBufCols, smem_desc(qa + (kk >> 2) * a.q_half + k32),
                       smem_desc(mb + k32), a.idesc1, kk > 0);
            }
            mma_commit(smem_u32(sm.tfull + buf));
            job++;
          }
          if (!ok) break;
          mma_commit(smem_u32(sm.empty + s0));
          mma_commit(smem_u32(sm.empty + s1));
        }
      };
      auto p2_tiles = [&](int qb, int n) {
        for (int j = 0; j < 2 * n && ok; j++) {  // two halves per tile
          const int slot = wait_slot();
          const int buf = slot < 0 ? -1 : wait_buf();
          if (buf < 0) {
            ok = false;
            break;
          }
          const uint32_t ma = smem_u32(sm.ring + slot * kGSlot);
          const uint32_t qbb = smem_u32(sm.q + qb * q_buf);
#pragma unroll
          for (int kk = 0; kk < 8; kk++) {
            const uint32_t k32 = (uint32_t)(kk & 3) * 32u;
            mma_bf16(tmem + (uint32_t)buf * kGBufCols,
                     smem_desc(ma + (kk >> 2) * (kGSlot / 2) + k32),
                     smem_desc(qbb + (kk >> 2) * a.q_half + k32), a.idesc2, kk > 0);
          }
          mma_commit(smem_u32(sm.tfull + buf));
          mma_commit(smem_u32(sm.empty + slot));
          job++;
        }
        if (ok && n > 0) mma_commit(smem_u32(sm.qempty + qb));  // the unit's last MMA
      };
      int prev_qb = -1, prev_my = 0;
      for (int i = 0; i < n_mine && ok; i++) {
        const GUnit u = gunit(a, i, grp, rank);
        int qb = -1;
        if (u.my > 0) {
          qb = qi & 1;
          if (!(ok = wait_or_abort(smem_u32(sm.qfull + qb), (qi >> 1) & 1, sm.failed))) break;
          qi++;
        }
        p1_tiles(qb, u.look);
        if (i > 0) p2_tiles(prev_qb, prev_my);
        p1_tiles(qb, u.my - u.look);
        prev_qb = qb;
        prev_my = u.my;
      }
      if (ok && n_mine > 0) p2_tiles(prev_qb, prev_my);
      if (!ok) *sm.failed = 1;
    }
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kGEpiRegs));
    // ------------------------------------------------------- epilogue
    // All eight warps take every job; warp (half, quarter) reads TMEM lanes
    // 32·quarter … + 31 and one half of the job's columns: in pass 1 the
    // blocks [128·half, 128·half + 128) of the tile, in pass 2 the window
    // positions [half·W/2, (half + 1)·W/2) of every head.
    const int half = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int trow = 32 * quarter + lane;     // this thread's TMEM lane
    const int et = (warp - 4) * 32 + lane;    // 0 … 255
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    const float zs = a.zscale, invW = 1.f / (float)W;
    const int G = a.R / W;
    uint32_t job = 0, p2n = 0;
    bool ok = true;
    // this thread's partials of the unit in pass 1: its row of each row tile
    // (rows trow and 128 + trow), over this half's columns
    float pm0 = -INFINITY, ps0 = 0.f, pm1 = -INFINITY, ps1 = 0.f;
    auto take = [&]() -> uint32_t {  // wait for the next job; its TMEM buffer
      const uint32_t buf = job & 1;
      ok = __all_sync(0xFFFFFFFFu, ok && wait_or_abort(smem_u32(sm.tfull + buf),
                                                        (job >> 1) & 1, sm.failed));
      if (ok) tc_fence_after();
      return tmem + lane_base + buf * kGBufCols;
    };
    auto give = [&]() {  // release the job's buffer to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(sm.tempty + (job & 1)));
      job++;
    };
    auto p1_tiles = [&](const GUnit &u, int j0, int j1) {
      for (int j = j0; j < j1; j++) {
        const int valid = min(kGTB, u.nb - (u.rank_eff + j * a.g) * kGTB) - 128 * half;
        for (int rt = 0; rt < 2; rt++) {
          const uint32_t tb = take();
          if (ok && rt * 128 + 32 * quarter < a.R) {  // some lane of the warp is a row
            float qm, qs;
            group_pass1(tb + (uint32_t)(128 * half), valid, zs, qm, qs);
            if (rt == 0)
              lse_merge_g(pm0, ps0, qm, qs);
            else if (128 + trow < a.R)
              lse_merge_g(pm1, ps1, qm, qs);
          }
          give();
        }
      }
    };
    auto p2_tiles = [&](const GUnit &u) {
      for (int j = 0; j < u.my; j++) {
        const int tile = u.rank_eff + j * a.g;
        for (int hf = 0; hf < 2; hf++) {
          const uint32_t tb = take();
          float part = 0.f;
          if (ok) part = group_pass2<W>(tb, G, half, zs, sm.lse);
          give();
          // the upper half's sum to the lower half's thread of the same lane
          float *cb = sm.comb + (p2n & 1) * 128;
          if (half == 1) cb[trow] = part;
          named_sync(3 + quarter, 64);
          if (half == 0) {
            const int blk = tile * kGTB + hf * 128 + trow;  // this lane's block in the unit
            if (ok && blk < u.nb)
              a.scores[((int64_t)u.l * a.H + u.h) * a.nb_total + u.b0 + blk] =
                  (part + cb[trow]) * invW;
          }
          p2n++;
        }
      }
    };
    // publish this CTA's row partials of the i-th unit and count them: the
    // upper column half hands its partials to the lower half through shared
    // memory (the LSE and combine buffers, both idle between a unit's pass 2
    // and the next exchange), which merges them (lower half first) and
    // writes one partial per row
    auto publish = [&](int i) {
      float2 *tmp = reinterpret_cast<float2 *>(sm.lse);  // [kGMaxR] (lse + comb)
      if (half == 1) {
        tmp[trow] = make_float2(pm0, ps0);
        if (128 + trow < a.R) tmp[128 + trow] = make_float2(pm1, ps1);
      }
      named_sync(2, 256);
      if (half == 0) {
        float2 *dst = a.part + (((int64_t)grp * 2 + (i & 1)) * a.g + rank) * 256;
        float2 o = tmp[trow];
        lse_merge_g(pm0, ps0, o.x, o.y);
        dst[trow] = make_float2(pm0, ps0);
        if (128 + trow < a.R) {
          o = tmp[128 + trow];
          lse_merge_g(pm1, ps1, o.x, o.y);
          dst[128 + trow] = make_float2(pm1, ps1);
        }
      }
      pm0 = pm1 = -INFINITY;
      ps0 = ps1 = 0.f;
      named_sync(2, 256);
      if (et == 0) {
        __threadfence();
        atomicAdd(a.counter + grp, 1);
      }
    };
    // wait until the group has published the i-th unit, then form its LSEs
    // (partials merged in rank order)
    auto exchange = [&](int i) {
      if (et == 0 && ok && !*sm.failed) {
        const int want = a.g * (i + 1);
        const uint64_t t0 = global_ns();
        while (ld_acquire_gpu(a.counter + grp) < want) {
          if (*sm.failed || global_ns() - t0 > 1000000000ull) {
            *sm.failed = 1;
            break;
          }
          __nanosleep(64);
        }
      }
      named_sync(2, 256);
      if (*sm.failed) ok = false;
      if (et < a.R) {
        // g partials, loaded 20 at a time so that their L2 latencies overlap
        const float2 *src = a.part + ((int64_t)grp * 2 + (i & 1)) * a.g * 256 + et;
        float m = -INFINITY, s2 = 0.f;
        for (int c0 = 0; c0 < a.g; c0 += 20) {
          float2 v[20];
#pragma unroll
          for (int k = 0; k < 20; k++)
            v[k] = c0 + k < a.g ? __ldcg(src + (int64_t)(c0 + k) * 256)
                                : make_float2(-INFINITY, 0.f);
#pragma unroll
          for (int k = 0; k < 20; k++) lse_merge_g(m, s2, v[k].x, v[k].y);
        }
        sm.lse[et] = (m == -INFINITY) ? INFINITY : m + log2f(s2);
      }
      named_sync(2, 256);
    };
    // Every CTA waits for every exchange, even of a unit it holds no tile
    // of: a CTA then never publishes unit i + 2 (the same partial buffer as
    // unit i) before all its peers have read unit i's partials.
    GUnit prev{};
    for (int i = 0; i < n_mine; i++) {
      const GUnit u = gunit(a, i, grp, rank);
      p1_tiles(u, 0, u.look);
      if (i > 0) {
        exchange(i - 1);
        p2_tiles(prev);
      }
      p1_tiles(u, u.look, u.my);
      publish(i);
      prev = u;
    }
    if (n_mine > 0) {
      exchange(n_mine - 1);
      p2_tiles(prev);
    }
    if (!ok) {
      *sm.failed = 1;
      if (et == 0) record_error(a.status, KVC_ERR_TIMEOUT);
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*sm.failed && threadIdx.x == 0) {
    record_error(a.status, KVC_ERR_TIMEOUT);
    // let this CTA's own copies and MMAs drain (bounded; stale phases return at once)
    for (int i = 0; i < ns; i++) {
      mbar_drain(smem_u32(sm.full + i), 0);
      mbar_drain(smem_u32(sm.full + i), 1);
    }
    for (int i = 0; i < 2; i++) {
      mbar_drain(smem_u32(sm.tfull + i), 0);
      mbar_drain(smem_u32(sm.tfull + i), 1);
      mbar_drain(smem_u32(sm.qfull + i), 0);
      mbar_drain(smem_u32(sm.qfull + i), 1);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    free_tmem_cols(tmem, 512);
  }
}

// --------------------------------------------------------------- host

// Ring slots that fit next to two query buffers of `R` rows.
int group_slots(int R) {
  const uint32_t q_half = (uint32_t)R * 128u;
  int ns = 0;
  while (GroupSmem::bytes(q_half, ns + 1) <= kGSmemMax) ns++;
  return ns;
}

// CTAs of k_score_group<W> with `smem` bytes that can be resident at once
// (one per SM, or 0 if it cannot run), cached per device and (W, R class);
// −1 marks an entry not yet queried (two host threads that race on one entry
// run the same query and store the same value).
template <int W>
int group_resident_ctas(size_t smem, int R) {
  using Row = std::atomic<int>[kGMaxR / 8 + 1];
  static Row *const cached = [] {
    Row *rows = new Row[64];
    for (int d = 0; d < 64; d++)
      for (int c = 0; c <= kGMaxR / 8; c++) rows[d][c].store(-1, std::memory_order_relaxed);
    return rows;
  }();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || R < 8 || R > kGMaxR) return 0;
  const int have = cached[dev][R / 8].load(std::memory_order_acquire);
  if (have >= 0) return have;
  auto kern = k_score_group<W>;
  int n = 0, per_sm = 0;
  cudaFuncAttributes fa{};
  // the register split (setmaxnreg) needs the block launched with at least
  // (128·kGCtlRegs + 256·kGEpiRegs) / 384 registers a thread
  const bool regs_ok =
      cudaFuncGetAttributes(&fa, kern) == cudaSuccess &&
      (int64_t)fa.numRegs * kGThreads >= 128 * (int64_t)kGCtlRegs + 256 * (int64_t)kGEpiRegs;
  if (regs_ok &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
          cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGThreads, smem) ==
          cudaSuccess &&
      per_sm >= 1)
    n = device_sm_count();
  (void)cudaGetLastError();
  cached[dev][R / 8].store(n, std::memory_order_release);
  return n;
}

// Group size: the divisor g of the SM count closest (in ratio) to the number
// of CTAs that gives each about kGTarget tiles of a mean-length unit.
int group_size(int n_sm, int64_t nb_total, int n_sess) {
  const double mean_tiles =
      (double)((nb_total + n_sess - 1) / (n_sess > 0 ? n_sess : 1)) / (double)kGTB;
  const double want = mean_tiles / kGTarget < 1.0 ? 1.0 : mean_tiles / kGTarget;
  int best = 1;
  double best_err = 1e30;
  for (int g = 1; g <= n_sm; g++) {
    if (n_sm % g) continue;
    const double err = fabs(log((double)g / want));
    if (err < best_err) {
      best_err = err;
      best = g;
    }
  }
  return best;
}

// q rows [units][R][D] seen as 2-D (D, rows), boxes of 64 columns × R rows.
bool make_q_group_map(CUtensorMap *m, const void *q, uint64_t rows, int R) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kGD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kGD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)R};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool score_group_supported(int G, int D, int W, int nb_max) {
  const int R = G * W;
  if (D != kGD || R <= 128 || R > kGMaxR || nb_max < 1 || (W != 8 && W != 16 && W != 32) ||
      R % 8)
    return false;
  const int ns = group_slots(R);
  if (ns < 4) return false;
  const size_t smem = GroupSmem::bytes((uint32_t)R * 128u, ns);
  return (W == 8    ? group_resident_ctas<8>(smem, R)
          : W == 16 ? group_resident_ctas<16>(smem, R)
                    : group_resident_ctas<32>(smem, R)) > 0;
}

size_t score_group_ws_bytes() {
  const int n_sm = device_sm_count();
  // counters (one per group, at most n_sm) + partials [n_sm][2][256] float2
  return 256 + ((size_t)n_sm * 4 + 255) / 256 * 256 + (size_t)n_sm * 2 * 256 * sizeof(float2);
}

cudaError_t launch_score_group(const uint16_t *q, const uint16_t *meank, float *scores, int L,
                               int H, int Hq, int D, int W, const int64_t *blk_off, int n_sess,
                               int64_t nb_total, int nb_max, void *ws, int32_t *status,
                               cudaStream_t s) {
  if (H <= 0 || Hq % H || !score_group_supported(Hq / H, D, W, nb_max))
    return cudaErrorNotSupported;
  const int R = (Hq / H) * W;
  const int n_sm = device_sm_count();
  const int n_units = L * H * n_sess;
  int g = group_size(n_sm, nb_total, n_sess);
  int n_groups = n_sm / g;
  if (n_groups > n_units) n_groups = n_units;
  const int ns = group_slots(R);
  const uint32_t q_half = (uint32_t)R * 128u;
  const size_t smem = GroupSmem::bytes(q_half, ns);
  CUtensorMap mk256, mk128, qmap;
  const uint64_t mk_rows = (uint64_t)L * H * nb_total;
  if (!make_map(&mk256, meank, mk_rows, D, 256) || !make_map(&mk128, meank, mk_rows, D, 128) ||
      !make_q_group_map(&qmap, q, (uint64_t)L * n_sess * Hq * W, R))
    return cudaErrorNotSupported;
  char *w = static_cast<char *>(ws);
  const size_t cnt_bytes = ((size_t)n_sm * 4 + 255) / 256 * 256;
  GroupArgs a{};
  a.scores = scores;
  a.blk_off = blk_off;
  a.status = status;
  a.counter = reinterpret_cast<int *>(w + 256);
  a.part = reinterpret_cast<float2 *>(w + 256 + cnt_bytes);
  a.L = L;
  a.H = H;
  a.n_sess = n_sess;
  a.R = R;
  a.n2 = (R + 15) / 16 * 16;
  a.g = g;
  a.n_groups = n_groups;
  a.max_tiles = (nb_max + kGTB - 1) / kGTB;
  a.ns = ns;
  a.nb_total = nb_total;
  a.zscale = 1.4426950408889634f / sqrtf((float)D);
  a.idesc1 = make_idesc(128, 256);
  a.idesc2 = make_idesc(128, a.n2);
  a.q_half = q_half;
  cudaError_t e = cudaMemsetAsync(a.counter, 0, cnt_bytes, s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(n_groups * g);
  cfg.blockDim = dim3(kGThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // every CTA of a group waits for its peers: the launch must make them all
  // resident at once
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (W) {
    case 8: return cudaLaunchKernelEx(&cfg, k_score_group<8>, mk256, mk128, qmap, a);
    case 16: return cudaLaunchKernelEx(&cfg, k_score_group<16>, mk256, mk128, qmap, a);
    default: return cudaLaunchKernelEx(&cfg, k_score_group<32>, mk256, mk128, qmap, a);
  }
}

}  // namespace kvc
