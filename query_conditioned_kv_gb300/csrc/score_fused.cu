// score_fused.cu — single-read tensor-core Mean-K scorer for query sets of
// 4 query heads per KV head × a 32-token window (128 query rows), D = 128.
//
// The quantity is the one every scorer of this library computes (KVMem
// "Query-conditioned retrieval"; ActKV §7.1 aggregation): for a unit (layer
// l, KV head h, session r) and query row (g, w),
//   z[g,w,b] = q[g,w]·meank[b]/sqrt(D),   LSE[g,w] = log Σ_b e^z,
//   score[b] = (1/W) Σ_w max_g exp(z[g,w,b] − LSE[g,w]).
//
// Design (Mean-K read from HBM once):
//   * A cluster of C ≤ 8 CTAs (one per SM) owns a unit; CTA `rank` takes the
//     unit's 256-block tiles rank, rank + C, …  A tile is one tcgen05.mma
//     product D[ρ][b] (M = 128 query rows, N = 256 blocks, K = 128) into one
//     of two 256-column TMEM buffers.  (N = 256 runs the tensor pipe about
//     2.3 times faster per block than two N = 128 products.)
//   * The query rows are loaded by a 5-D tensor map in the order
//     ρ = g_l + 2·w_l + 8·g_h + 16·w_h (g = 2·g_h + g_l, w = 4·w_h + w_l): in
//     each 16-lane half of TMEM, lanes ρ and ρ + 8 hold query heads g and
//     g + 2 of one window position.
//   * Pass 1 (per lane = query row): online (max, Σ2^(z−max)) over the tile's
//     blocks.  The logits of a CTA's last (up to) two tiles stay in TMEM.
//   * The CTAs of the cluster exchange their row partials with st.async into
//     each other's shared memory, and every CTA forms the row LSEs.
//   * Pass 2 reads the kept logits again with the 16x256b TMEM shape, which
//     gives a thread two rows (lanes t/4 and t/4 + 8 of a 16-lane half): the
//     heads g_l and g_l + 2 of window position t/8.  x = z·log2e/√D − LSE; the
//     max over those two heads in the thread, over g_l with lane t^4, one ex2
//     per (w, b), the sum over the half's four window positions with lanes
//     t^8 and t^16 (each stage halving the columns a lane carries), the two
//     halves added in the thread, and the warp quarters through shared
//     memory in a fixed order.
//   * Four epilogue warpgroups split every tile: group e takes its columns
//     64e … 64e + 63, so each step of the chain above has 16 warps on it.
//   * A CTA with more than two tiles multiplies its first tiles again after
//     the exchange (they are still in L2); the last two are never reloaded.
//     Jobs run in the order A(u) R(u−1) B(u) (A = first multiplications of
//     the reloaded tiles, R = their second, B = kept tiles), so the next
//     unit's first tiles stream in during a unit's exchange and pass 2.
// Every wait is bounded (1 s of %globaltimer) and records KVC_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <atomic>

#include "kvc_internal.cuh"
#include "tc_ptx.cuh"

namespace kvc {
namespace {

using namespace tc;

constexpr int kFG = 4;           // query heads per KV head
constexpr int kFW = 32;          // window positions
constexpr int kFD = 128;         // head dim
constexpr int kFTB = 256;        // Mean-K blocks per tile (MMA N)
constexpr int kFNS = 2;          // Mean-K ring stages (64 KB each)
constexpr int kFQB = 2;          // query-row buffers (32 KB each)
constexpr int kFNBUF = 2;        // TMEM buffers of 256 columns
constexpr int kFKeep = kFNBUF;   // tiles whose logits stay in TMEM
constexpr int kFTarget = 4;      // tiles per CTA of a mean-length unit the cluster aims at
constexpr int kFNEG = 4;         // epilogue warpgroups
constexpr int kFCols = kFTB / kFNEG;  // columns of every tile a group takes (64)
constexpr int kFNCH = kFCols / 32;    // their 32-column chunks
constexpr int kFMaxC = 8;        // CTAs per cluster
constexpr int kFThreads = 64 + 128 * kFNEG;
constexpr uint32_t kFTile = kFTB * kFD * 2;  // 64 KB
constexpr uint32_t kFQ = 128 * kFD * 2;      // 32 KB

struct FusedArgs {
  float *scores;
  const int64_t *blk_off;
  int32_t *status;
  int L, H, n_sess;
  int max_tiles;  // longest session accepted, in tiles
  int64_t nb_total;
  float zscale;  // log2(e)/sqrt(D)
  uint32_t idesc;
};

struct FusedSmem {
  uint8_t *ring, *q;
  uint64_t *full, *empty, *tfull, *tempty, *qfull, *qempty, *recv;
  uint32_t *tmem_holder;
  volatile int *failed;
  float2 *egpart;  // [kFNEG][128] per-group row partials
  float2 *rbuf;    // [2 parities][kFMaxC ranks][128] received partials
  float *lse;      // [128] row LSE (base 2)
  float *red;      // [kFNEG][2 parities][4 quarters][kFCols] pass-2 column sums
  __device__ explicit FusedSmem(uint8_t *raw) {
    uint8_t *p = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    ring = p;
    p += kFNS * kFTile;
    q = p;
    p += kFQB * kFQ;
    uint64_t *b = reinterpret_cast<uint64_t *>(p);
    full = b;
    empty = full + kFNS;
    tfull = empty + kFNS;
    tempty = tfull + kFNBUF;
    qfull = tempty + kFNBUF;
    qempty = qfull + kFQB;
    recv = qempty + kFQB;
    tmem_holder = reinterpret_cast<uint32_t *>(recv + 2);
    failed = reinterpret_cast<volatile int *>(tmem_holder + 1);
    egpart = reinterpret_cast<float2 *>(tmem_holder + 4);  // 16-byte aligned
    rbuf = egpart + kFNEG * 128;
    lse = reinterpret_cast<float *>(rbuf + 2 * kFMaxC * 128);
    red = lse + 128;
  }
  static constexpr size_t bytes() {
    return 1024 + (size_t)kFNS * kFTile + (size_t)kFQB * kFQ +
           (2 * kFNS + 2 * kFNBUF + 2 * kFQB + 2) * 8 + 16 +
           (size_t)(kFNEG + 2 * kFMaxC) * 128 * 8 + 128 * 4 + (size_t)kFNEG * 2 * 4 * kFCols * 4;
  }
};

struct FUnit {
  int l, h, r, nb, n_tiles, my_tiles, n_rec, mk_row0, q_unit;
  int64_t b0;
};

// A unit and this CTA's share of it: my_tiles tiles, of which the first
// n_rec are multiplied twice (before and after the exchange).
__device__ __forceinline__ FUnit funit(const FusedArgs &a, int unit, int C, int rank) {
  FUnit u;
  u.r = unit % a.n_sess;
  const int lh = unit / a.n_sess;
  u.h = lh % a.H;
  u.l = lh / a.H;
  const int64_t b0 = a.blk_off[u.r], b1 = a.blk_off[u.r + 1];
  const bool ok =
      b0 >= 0 && b1 > b0 && b1 <= a.nb_total && b1 - b0 <= (int64_t)a.max_tiles * kFTB;
  u.b0 = ok ? b0 : 0;
  u.nb = ok ? (int)(b1 - b0) : 0;
  u.n_tiles = (u.nb + kFTB - 1) / kFTB;
  u.my_tiles = u.n_tiles > rank ? (u.n_tiles - rank + C - 1) / C : 0;
  u.n_rec = u.my_tiles > kFKeep ? u.my_tiles - kFKeep : 0;
  u.mk_row0 = (int)(((int64_t)u.l * a.H + u.h) * a.nb_total + u.b0);
  u.q_unit = (u.l * a.n_sess + u.r) * a.H + u.h;
  return u;
}

// Remote 8-byte store into a peer's shared memory that counts its bytes on
// the peer's mbarrier when it lands (no fence or separate arrive).
__device__ __forceinline__ void st_async_f2(uint32_t raddr, float2 v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
               ::"r"(raddr), "f"(v.x), "f"(v.y), "r"(rbar)
               : "memory");
}

__device__ __forceinline__ void merge_lse(float &m, float &s, float m2, float s2) {
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

// Pass 1 of this group's columns of one tile for this lane's query row:
// (max, Σ2^(z·zs − max)) over the `valid` blocks, 32 columns at a time.
// Column j adds into accumulator j mod 8 (held as four packed pairs).
__device__ __forceinline__ void fused_pass1(uint32_t taddr, int valid, float zs, float &pm,
                                            float &ps) {
  pm = -INFINITY;
  ps = 0.f;
  const uint64_t zs2 = pk2(zs, zs);
#pragma unroll 1
  for (int c = 0; c < kFNCH && 32 * c < valid; c++) {
    uint32_t r[32];
    tmem_issue32(taddr + (uint32_t)(32 * c), r);
    tmem_wait32(r);
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; j++) v[j] = __uint_as_float(r[j]);
    const int nv = valid - 32 * c;
    if (nv < 32) {
#pragma unroll
      for (int j = 0; j < 32; j++)
        if (j >= nv) v[j] = -INFINITY;
    }
    float m0 = max3(v[0], v[1], v[2]), m1 = max3(v[3], v[4], v[5]);
    float m2 = max3(v[6], v[7], v[8]), m3 = max3(v[9], v[10], v[11]);
#pragma unroll
    for (int j = 12; j < 28; j += 8) {
      m0 = max3(m0, v[j], v[j + 1]);
      m1 = max3(m1, v[j + 2], v[j + 3]);
      m2 = max3(m2, v[j + 4], v[j + 5]);
      m3 = max3(m3, v[j + 6], v[j + 7]);
    }
    m0 = max3(m0, v[28], v[29]);
    m1 = max3(m1, v[30], v[31]);
    const float mn = fmaxf(pm, fmaxf(max3(m0, m1, m2), m3) * zs);
    const uint64_t nmn2 = pk2(-mn, -mn);
    uint64_t acc[4];
    acc[0] = pk2((pm == -INFINITY) ? 0.f : ps * ex2(pm - mn), 0.f);
#pragma unroll
    for (int k = 1; k < 4; k++) acc[k] = pk2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
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

// 16 lanes × 32 columns of TMEM with the 16x256b shape: register 4k + j of
// thread t holds lane (t/4 + 8·(j ≥ 2)), column 8k + 2·(t%4) + (j & 1).
__device__ __forceinline__ void tmem_ld16x256x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Pass 2 of one tile for this warp's 32 query rows (TMEM lanes 32q … 32q+31 =
// two 16-lane halves; `taddr` points at lane 32q and this group's columns).
// Rows are ordered so that in half h, lane 2·w_l + g_l + 8·g_h is window
// position w = 4·(2q + h) + w_l and query head g = 2·g_h + g_l: the 16x256b
// load gives thread t heads g_l and g_l + 2 (g_l = bit 2 of t) of window
// position w_l = t/8.  Per 32 columns and half: x = z·zs − LSE; max over g_h
// in the thread, over g_l with lane t^4 (each stage halving the columns a
// lane carries), one ex2, the sum over w_l with lanes t^8 and t^16; the two
// halves are added in the thread.  Lane t ends with column
// 16·b2 + 8·b3 + 2·(t%4) + b4 (b_i = bit i of t).
__device__ __forceinline__ void fused_pass2(uint32_t taddr, const float *lse_q, float zs, int lane,
                                            float *red_q) {
  const bool b2 = lane & 4, b3 = lane & 8, b4 = lane & 16;
  const int col_in_chunk = 16 * (int)b2 + 8 * (int)b3 + 2 * (lane & 3) + (int)b4;
  const uint64_t zs2 = pk2(zs, zs);
  uint64_t nl2[2][2];  // [half][g_h]: −LSE of this thread's two rows, paired
#pragma unroll
  for (int h = 0; h < 2; h++)
#pragma unroll
    for (int gh = 0; gh < 2; gh++) {
      const float l = lse_q[16 * h + (lane >> 2) + 8 * gh];
      nl2[h][gh] = pk2(-l, -l);
    }
#pragma unroll 1
  for (int c = 0; c < kFNCH; c++) {
    float sum = 0.f;
#pragma unroll
    for (int h = 0; h < 2; h++) {
      uint32_t r[16];
      tmem_ld16x256x4(taddr + ((uint32_t)(16 * h) << 16) + (uint32_t)(32 * c), r);
      float v[8];  // [2k + e]: column 8k + 2·(t%4) + e, max over g_h
#pragma unroll
      for (int k = 0; k < 4; k++) {
        float x0, x1, y0, y1;
        upk2(fma2(pk2(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1])), zs2, nl2[h][0]),
             x0, x1);
        upk2(fma2(pk2(__uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3])), zs2,
                  nl2[h][1]),
             y0, y1);
        v[2 * k] = fmaxf(x0, y0);
        v[2 * k + 1] = fmaxf(x1, y1);
      }
      float e[4];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const float keep = b2 ? v[4 + i] : v[i], send = b2 ? v[i] : v[4 + i];
        e[i] = ex2(fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 4)));
      }
      float s2[2];
#pragma unroll
      for (int i = 0; i < 2; i++) {
        const float keep = b3 ? e[2 + i] : e[i], send = b3 ? e[i] : e[2 + i];
        s2[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
      }
      const float keep = b4 ? s2[1] : s2[0], send = b4 ? s2[0] : s2[1];
      sum += keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    }
    red_q[32 * c + col_in_chunk] = sum;
  }
}

__global__ void __launch_bounds__(kFThreads, 1)
k_score_fused(const __grid_constant__ CUtensorMap tm_mk, const __grid_constant__ CUtensorMap tm_q,
              FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  FusedSmem sm(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = (int)cluster_nrank(), rank = (int)cluster_rank();
  const int cluster_id = blockIdx.x / C, n_clusters = gridDim.x / C;
  const int n_units = a.L * a.H * a.n_sess;

  if (threadIdx.x == 0) {
    *sm.failed = 0;
    for (int i = 0; i < kFNS; i++) {
      mbar_init(smem_u32(sm.full + i), 1);
      mbar_init(smem_u32(sm.empty + i), 1);
    }
    for (int i = 0; i < kFNBUF; i++) {
      mbar_init(smem_u32(sm.tfull + i), 1);
      mbar_init(smem_u32(sm.tempty + i), 4 * kFNEG);  // every epilogue warp reads every tile
    }
    for (int i = 0; i < kFQB; i++) {
      mbar_init(smem_u32(sm.qfull + i), 1);
      mbar_init(smem_u32(sm.qempty + i), 1);
    }
    // each receive barrier: one local arrival that arms it for the bytes of
    // the C − 1 peers' row partials
    for (int i = 0; i < 2; i++) {
      mbar_init(smem_u32(sm.recv + i), 1);
      if (C > 1) mbar_expect_tx(smem_u32(sm.recv + i), (uint32_t)(C - 1) * 128 * 8);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) alloc_tmem_cols(sm.tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (C > 1) cluster_sync_all();  // peers' barriers exist before any remote arrive
  const uint32_t tmem = *sm.tmem_holder;

  // Job order of a CTA (the same for all three roles).  With A(u) = the
  // tiles of unit u multiplied twice (first n_rec), B(u) = the tiles whose
  // logits stay in TMEM and R(u) = the second multiplication of A(u):
  //   A(u0) B(u0) | A(u1) R(u0) B(u1) | A(u2) R(u1) B(u2) | … | R(u_last)
  // A job waits for the TMEM buffer of the job four places earlier, so the
  // next unit's first tiles stream in while this unit's exchange and pass 2
  // run, and R(u) follows them out of L2.
  if (warp == 0) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t s = 0, qi = 0;
      bool ok = true;
      int prev_unit = -1;
      // tiles multiplied twice stay in L2 until their second read (evict
      // last); second reads and the kept tiles are the last use (evict first)
      const uint64_t keep = l2_evict_last(), drop = l2_evict_first();
      auto load_tile = [&](int row0, int i, uint64_t pol) -> bool {
        const int slot = s % kFNS;
        if (!wait_or_abort(smem_u32(sm.empty + slot), ((s / kFNS) & 1) ^ 1, sm.failed))
          return false;
        mbar_expect_tx(smem_u32(sm.full + slot), kFTile);
        for (int kb = 0; kb < 2; kb++)
          tma_load_2d_hint(smem_u32(sm.ring + slot * kFTile + kb * (kFTile / 2)), &tm_mk, kb * 64,
                           row0 + (rank + i * C) * kFTB, smem_u32(sm.full + slot), pol);
        s++;
        return true;
      };
      for (int unit = cluster_id; ok; unit += n_clusters) {
        const bool last = unit >= n_units;
        FUnit u{};
        if (!last) {
          u = funit(a, unit, C, rank);
          if (u.nb == 0 && rank == 0) record_error(a.status, KVC_ERR_BOUNDS);
          if (u.my_tiles > 0) {
            const int qb = qi % kFQB;
            if (!(ok = wait_or_abort(smem_u32(sm.qempty + qb), ((qi / kFQB) & 1) ^ 1,
                                     sm.failed)))
              break;
            mbar_expect_tx(smem_u32(sm.qfull + qb), kFQ);
            for (int kb = 0; kb < 2; kb++)
              tma_load_5d(smem_u32(sm.q + qb * kFQ + kb * (kFQ / 2)), &tm_q, kb * 64, 0, 0,
                          2 * u.q_unit, 0, smem_u32(sm.qfull + qb));
            qi++;
          }
        }
        for (int i = 0; i < u.n_rec && ok; i++) ok = load_tile(u.mk_row0, i, keep);  // A(u)
        if (prev_unit >= 0) {
          const FUnit prev = funit(a, prev_unit, C, rank);
          for (int i = 0; i < prev.n_rec && ok; i++)
            ok = load_tile(prev.mk_row0, i, drop);                                    // R(prev)
        }
        for (int i = u.n_rec; i < u.my_tiles && ok; i++)
          ok = load_tile(u.mk_row0, i, drop);                                         // B(u)
        if (last) break;
        prev_unit = unit;
      }
      if (!ok) *sm.failed = 1;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t s = 0, t = 0, qi = 0;
      bool ok = true;
      int prev_nrec = 0, prev_qb = -1;
      auto mma_job = [&](int qb) -> bool {
        const int slot = s % kFNS, buf = t % kFNBUF;
        if (!wait_or_abort(smem_u32(sm.full + slot), (s / kFNS) & 1, sm.failed)) return false;
        if (!wait_or_abort(smem_u32(sm.tempty + buf), ((t / kFNBUF) & 1) ^ 1, sm.failed))
          return false;
        tc_fence_after();
        const uint32_t qa = smem_u32(sm.q + qb * kFQ), ma = smem_u32(sm.ring + slot * kFTile);
        const uint32_t d = tmem + (uint32_t)(buf * kFTB);
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint32_t k32 = (uint32_t)(kk & 3) * 32u;
          mma_bf16(d, smem_desc(qa + (kk >> 2) * (kFQ / 2) + k32),
                   smem_desc(ma + (kk >> 2) * (kFTile / 2) + k32), a.idesc, kk > 0);
        }
        mma_commit(smem_u32(sm.empty + slot));
        mma_commit(smem_u32(sm.tfull + buf));
        s++;
        t++;
        return true;
      };
      for (int unit = cluster_id; ok; unit += n_clusters) {
        const bool last = unit >= n_units;
        FUnit u{};
        int qb = -1;
        if (!last) {
          u = funit(a, unit, C, rank);
          if (u.my_tiles > 0) {
            qb = qi % kFQB;
            if (!(ok = wait_or_abort(smem_u32(sm.qfull + qb), (qi / kFQB) & 1, sm.failed)))
              break;
            qi++;
          }
        }
        for (int i = 0; i < u.n_rec && ok; i++) ok = mma_job(qb);                  // A(u)
        if (prev_qb >= 0) {
          for (int i = 0; i < prev_nrec && ok; i++) ok = mma_job(prev_qb);         // R(prev)
          if (ok) mma_commit(smem_u32(sm.qempty + prev_qb));  // prev's last MMA issued
        }
        for (int i = u.n_rec; i < u.my_tiles && ok; i++) ok = mma_job(qb);        // B(u)
        if (last) break;
        prev_nrec = u.n_rec;
        prev_qb = qb;
      }
      if (!ok) *sm.failed = 1;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- epilogue
    const int eg = (warp - 2) >> 2;          // this thread's group
    const int quarter = warp & 3;            // TMEM lane quarter of this warp
    const int row = 32 * quarter + lane;     // this thread's TMEM lane (query row)
    const int gt = ((warp - 2) & 3) * 32 + lane;  // 0 … 127 within the group
    const int et = (warp - 2) * 32 + lane;        // 0 … 128·kFNEG − 1
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    const float zs = a.zscale, invW = 1.f / (float)kFW;
    float *red = sm.red + eg * 2 * 4 * kFCols;
    uint32_t t = 0, ui = 0, rp = 0;
    bool ok = true;
    int prev_unit = -1;
    // pass 2 of one job of unit w (local tile i); the row LSEs are in sm.lse
    // (a unit's reloaded tiles run before the next exchange, whose first
    // barrier every group passes only after them)
    auto pass2_job = [&](const FUnit &w, int i, uint32_t job, bool wait_full) {
      const uint32_t buf = job % kFNBUF;
      if (wait_full)
        ok = __all_sync(0xFFFFFFFFu, ok && wait_or_abort(smem_u32(sm.tfull + buf),
                                                          (job / kFNBUF) & 1, sm.failed));
      const int tile = rank + i * C;
      const int valid = min(kFCols, w.nb - tile * kFTB - eg * kFCols);  // this group's columns
      float *rq = red + (rp & 1) * 4 * kFCols;
      if (ok && valid > 0) {
        tc_fence_after();
        fused_pass2(tmem + lane_base + buf * kFTB + eg * kFCols, sm.lse + 32 * quarter, zs,
                    lane, rq + quarter * kFCols);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(sm.tempty + buf));
      named_sync(4 + eg, 128);
      if (ok && gt < valid) {
        float *out = a.scores + ((int64_t)w.l * a.H + w.h) * a.nb_total + w.b0 + tile * kFTB +
                     eg * kFCols;
        out[gt] = ((rq[gt] + rq[kFCols + gt]) + (rq[2 * kFCols + gt] + rq[3 * kFCols + gt])) * invW;
      }
      rp++;
    };
    // pass 1 of one job of unit w (local tile i); releases the buffer unless kept
    auto pass1_job = [&](const FUnit &w, int i, uint32_t job, float &pm, float &ps) {
      const uint32_t buf = job % kFNBUF;
      ok = __all_sync(0xFFFFFFFFu, ok && wait_or_abort(smem_u32(sm.tfull + buf),
                                                        (job / kFNBUF) & 1, sm.failed));
      const int valid = min(kFCols, w.nb - (rank + i * C) * kFTB - eg * kFCols);
      if (ok && valid > 0) {  // this group's columns of the tile
        tc_fence_after();
        float qm, qs;
        fused_pass1(tmem + lane_base + buf * kFTB + eg * kFCols, valid, zs, qm, qs);
        merge_lse(pm, ps, qm, qs);
      }
      if (i < w.n_rec) {  // not kept: the buffer goes back to the MMA warp
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(sm.tempty + buf));
      }
    };
    for (int unit = cluster_id;; unit += n_clusters) {
      const bool last = unit >= n_units;
      FUnit u{};
      if (!last) u = funit(a, unit, C, rank);
      // a group merges its columns of the unit's tiles in tile order, and the
      // groups merge in group order, so the result depends only on the unit
      float pm = -INFINITY, ps = 0.f;
      for (int i = 0; i < u.n_rec; i++, t++) pass1_job(u, i, t, pm, ps);         // A(u)
      if (prev_unit >= 0) {
        const FUnit prev = funit(a, prev_unit, C, rank);
        for (int i = 0; i < prev.n_rec; i++, t++) pass2_job(prev, i, t, true);  // R(prev)
      }
      const uint32_t tB = t;
      for (int i = u.n_rec; i < u.my_tiles; i++, t++) pass1_job(u, i, t, pm, ps);  // B(u)
      if (last) break;
      if (C > 1 || u.my_tiles > 0) {
        // exchange: group partials → CTA partial → every CTA of the cluster
        const int par = ui & 1;
        sm.egpart[eg * 128 + row] = make_float2(pm, ps);
        named_sync(2, 128 * kFNEG);
        if (eg == 0) {
          // group 0: this row's CTA partial to every peer, then (once the
          // peers' partials are in) the row's LSE; the other groups go on to
          // the barrier below
          float m = pm, s2 = ps;
          for (int g2 = 1; g2 < kFNEG; g2++) {
            const float2 o = sm.egpart[g2 * 128 + row];
            merge_lse(m, s2, o.x, o.y);
          }
          const float2 v = make_float2(m, s2);
          float2 *mine = sm.rbuf + (par * kFMaxC + rank) * 128 + row;
          *mine = v;
          const uint32_t a_mine = smem_u32(mine), a_bar = smem_u32(sm.recv + par);
          for (int p = 1; p < C; p++) {
            const uint32_t peer = (uint32_t)((rank + p) % C);
            st_async_f2(mapa_u32(a_mine, peer), v, mapa_u32(a_bar, peer));
          }
          if (C > 1) {
            ok = __all_sync(0xFFFFFFFFu, ok && wait_or_abort(smem_u32(sm.recv + par),
                                                              (ui >> 1) & 1, sm.failed, true));
            // re-arm this parity for the unit after next: no peer can send that
            // unit's partials before it has received this CTA's next ones
            if (et == 0) mbar_expect_tx(smem_u32(sm.recv + par), (uint32_t)(C - 1) * 128 * 8);
          }
          float mm = -INFINITY, ss = 0.f;
          for (int c = 0; c < C; c++) {
            const float2 w = sm.rbuf[(par * kFMaxC + c) * 128 + row];
            merge_lse(mm, ss, w.x, w.y);
          }
          sm.lse[row] = (mm == -INFINITY) ? INFINITY : mm + log2f(ss);
        }
        named_sync(2, 128 * kFNEG);
        ui++;
        for (int i = u.n_rec; i < u.my_tiles; i++)                               // pass 2 of B(u)
          pass2_job(u, i, tB + (uint32_t)(i - u.n_rec), false);
      }
      prev_unit = unit;
      if (!ok) {
        *sm.failed = 1;
        if (et == 0) record_error(a.status, KVC_ERR_TIMEOUT);
      }
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
    for (int i = 0; i < kFNS; i++) {
      mbar_drain(smem_u32(sm.full + i), 0);
      mbar_drain(smem_u32(sm.full + i), 1);
    }
    for (int i = 0; i < kFNBUF; i++) {
      mbar_drain(smem_u32(sm.tfull + i), 0);
      mbar_drain(smem_u32(sm.tfull + i), 1);
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

// Clusters of C that can be resident at once (0: the kernel cannot run),
// cached per device; −1 marks an entry not yet queried (two host threads
// that race on one entry both run the same query and store the same value).
int fused_clusters(int C) {
  using Row = std::atomic<int>[kFMaxC + 1];
  static Row *const cached = [] {  // initialised once, thread-safely
    Row *rows = new Row[64];
    for (int d = 0; d < 64; d++)
      for (int c = 0; c <= kFMaxC; c++) rows[d][c].store(-1, std::memory_order_relaxed);
    return rows;
  }();
  if (C < 1 || C > kFMaxC) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int have = cached[dev][C].load(std::memory_order_acquire);
  if (have >= 0) return have;
  const size_t smem = FusedSmem::bytes();
  int n = 0;
  if (cudaFuncSetAttribute(k_score_fused, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, k_score_fused, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  cached[dev][C].store(n, std::memory_order_release);
  return n;
}

// CTAs per cluster: about kFTarget tiles of a mean-length session per CTA
// (twice that when the longest session is 1.5× the mean or more),
// rounded down to a power of two (at most eight), and smaller while the
// size cannot be scheduled.  A tile multiplied twice is reloaded about one
// round (its CTA's share of a unit, plus the next unit's first tiles) after
// its first read; with four tiles per CTA that is ~50 MB across the GPU, so
// the reload still hits L2 (eight tiles per CTA measured 1.57× the
// algorithmic DRAM reads).
int fused_cluster(int64_t nb_total, int n_sess, int nb_max) {
  const int64_t mean = (nb_total + n_sess - 1) / (n_sess > 0 ? n_sess : 1);
  // Sessions of very different lengths: twice the tiles per CTA.  Short
  // sessions then leave fewer CTAs of their cluster idle and every session
  // pays half the exchanges; measured on 128 sessions of 2–32 tiles, 11.6 ms
  // against 12.9 ms for four tiles per CTA.
  const int target = 2 * (int64_t)nb_max >= 3 * mean ? 2 * kFTarget : kFTarget;
  const int64_t want = ((mean + kFTB - 1) / kFTB + target - 1) / target;
  int c = 1;
  while (2 * c <= want && 2 * c <= kFMaxC) c *= 2;
  while (c > 1 && fused_clusters(c) == 0) c /= 2;
  return c;
}

// q rows [units][G = 4][W = 32][D] seen as five dimensions (d, g_l, w_l,
// g_h + 2·unit, w_h) with g = 2·g_h + g_l and w = 4·w_h + w_l; g_h and the unit
// share one dimension because the unit stride is twice the g_h stride.  A box
// (64 columns, 2, 4, 2, 8) at (·, 0, 0, 2·unit, 0) lands in shared memory as
// rows ρ = g_l + 2·w_l + 8·g_h + 16·w_h: within each 16-row half, rows ρ and
// ρ + 8 are query heads g and g + 2 of one window position (the pairs the
// 16x256b TMEM load gives one thread in pass 2).
bool make_q_rows_map(CUtensorMap *m, const void *q, uint64_t q_units) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t row = (cuuint64_t)kFD * 2;  // bytes per (g, w) row
  cuuint64_t dims[5] = {(cuuint64_t)kFD, 2, 4, 2 * q_units, (cuuint64_t)kFW / 4};
  cuuint64_t strides[4] = {(cuuint64_t)kFW * row, row, 2 * (cuuint64_t)kFW * row, 4 * row};
  cuuint32_t box[5] = {64, 2, 4, 2, (cuuint32_t)kFW / 4};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool score_fused_supported(int G, int D, int W, int nb_max) {
  return G == kFG && D == kFD && W == kFW && nb_max > 0 && fused_clusters(1) > 0;
}

cudaError_t launch_score_fused(const uint16_t *q, const uint16_t *meank, float *scores, int L,
                               int H, int Hq, int D, int W, const int64_t *blk_off, int n_sess,
                               int64_t nb_total, int nb_max, int32_t *status, cudaStream_t s) {
  if (H <= 0 || Hq != kFG * H || !score_fused_supported(Hq / H, D, W, nb_max))
    return cudaErrorNotSupported;
  const int C = fused_cluster(nb_total, n_sess, nb_max), nc = fused_clusters(C);
  const int n_units = L * H * n_sess;
  CUtensorMap mk_map, q_map;
  if (!make_map(&mk_map, meank, (uint64_t)L * H * nb_total, D, kFTB) ||
      !make_q_rows_map(&q_map, q, (uint64_t)L * n_sess * H))
    return cudaErrorNotSupported;
  FusedArgs a{};
  a.scores = scores;
  a.blk_off = blk_off;
  a.status = status;
  a.L = L;
  a.H = H;
  a.n_sess = n_sess;
  a.max_tiles = (nb_max + kFTB - 1) / kFTB;
  a.nb_total = nb_total;
  a.zscale = 1.4426950408889634f / sqrtf((float)D);
  a.idesc = make_idesc(128, kFTB);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((nc < n_units ? nc : n_units) * C);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = FusedSmem::bytes();
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_score_fused, mk_map, q_map, a);
}

}  // namespace kvc
