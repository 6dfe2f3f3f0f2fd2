// pack.cu — execution-view pack with re-RoPE, and the RoPE table.
//
// KVMem, "Tiered movement": an execution view holds only the selected
// blocks, packed into contiguous logical positions; the position-independent
// raw K is re-RoPEd at the new positions and V is copied as-is.
//
// One CTA owns one view block (32 tokens) of one (layer, session) and walks
// the KV heads: every head of the view block sits at the same 32 positions,
// so the CTA loads its cos/sin values once and reuses them for all heads.
// Thread layout: token = tid / (D/16), chunk c = tid % (D/16); a thread
// rotates the 8 pairs (j, j + D/2) for j ∈ [8c, 8c+8) with two 16-byte K
// loads, copies 32 bytes of V, and keeps two heads' loads in flight.  All
// K/V traffic is 16-byte, coalesced and streaming (touched once).
//
// The tiered variant (KVMem "Tiered movement", with step-to-step overlap
// reuse) keeps the raw K/V history in host memory: blocks the previous step
// already had in its view are taken from device memory, the others are read
// by the kernel itself from pinned host memory over NVLink-C2C (no CPU
// gather, no staging copy), and the view's raw K is kept for the next step.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

__global__ void __launch_bounds__(256)
k_rope_table(float *__restrict__ tab, int n_pos, int pos0, int half, int D,
             double theta) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)n_pos * half) return;
  int i = (int)(t / half), j = (int)(t - (int64_t)i * half);
  // angle = p · theta^(−2j/D), in fp64
  double freq = pow(theta, -2.0 * (double)j / (double)D);
  double a = (double)(pos0 + i) * freq;
  double sa, ca;
  sincos(a, &sa, &ca);
  reinterpret_cast<float2 *>(tab)[t] = make_float2((float)ca, (float)sa);
}

struct PackArgs {
  const uint16_t *kraw, *vraw;
  const int32_t *kept, *kept_count;
  const int64_t *tok_off;
  const float *rope_tab;
  uint16_t *kview, *vview;
  int32_t *status;
  int L, H, n_sess, budget;
  int64_t n_tok;
};

template <int D>
__device__ __forceinline__ void rotate8(const uint4 &lo, const uint4 &hi,
                                        const float (&c)[8], const float (&s)[8],
                                        uint4 &olo, uint4 &ohi) {
  const uint32_t xl[4] = {lo.x, lo.y, lo.z, lo.w};
  const uint32_t xh[4] = {hi.x, hi.y, hi.z, hi.w};
  uint32_t rl[4], rh[4];
#pragma unroll
  for (int e = 0; e < 4; e++) {
    float x0 = bf16_lo(xl[e]), x1 = bf16_hi(xl[e]);
    float y0 = bf16_lo(xh[e]), y1 = bf16_hi(xh[e]);
    float c0 = c[2 * e], s0 = s[2 * e], c1 = c[2 * e + 1], s1 = s[2 * e + 1];
    rl[e] = pack_bf16x2(fmaf(x0, c0, -y0 * s0), fmaf(x1, c1, -y1 * s1));
    rh[e] = pack_bf16x2(fmaf(y0, c0, x0 * s0), fmaf(y1, c1, x1 * s1));
  }
  olo = make_uint4(rl[0], rl[1], rl[2], rl[3]);
  ohi = make_uint4(rh[0], rh[1], rh[2], rh[3]);
}

template <int D>
__global__ void __launch_bounds__(2 * D)
k_pack_rerope(PackArgs a) {
  constexpr int TPT = D / 16;  // threads per token
  constexpr int HALF = D / 2;
  const int tok = threadIdx.x / TPT, c = threadIdx.x % TPT;
  const int i = blockIdx.x;           // view block
  const int lr = blockIdx.y;          // (layer, session), session fastest
  const int r = lr % a.n_sess, l = lr / a.n_sess;

  const int64_t t0 = a.tok_off[r], t1 = a.tok_off[r + 1];
  const bool sess_ok = t0 >= 0 && t1 >= t0 && t1 <= a.n_tok && (t0 % kBlock) == 0 &&
                       ((t1 - t0) % kBlock) == 0;
  const int64_t nb = sess_ok ? (t1 - t0) / kBlock : 0;

  // cos/sin of view position 32·i + tok for pairs 8c … 8c+7
  float cs[8], sn[8];
  {
    const float4 *tb = reinterpret_cast<const float4 *>(
        a.rope_tab + ((int64_t)(i * kBlock + tok) * HALF + 8 * c) * 2);
#pragma unroll
    for (int e = 0; e < 4; e++) {
      float4 v = __ldg(tb + e);
      cs[2 * e] = v.x;
      sn[2 * e] = v.y;
      cs[2 * e + 1] = v.z;
      sn[2 * e + 1] = v.w;
    }
  }

  const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll 2
  for (int h = 0; h < a.H; h++) {
    const int64_t seg = ((int64_t)l * a.H + h) * a.n_sess + r;
    const int64_t dst = ((seg * a.budget + i) * kBlock + tok) * D;
    int cnt = a.kept_count[seg];
    bool live = i < cnt && cnt <= a.budget;
    int64_t src = 0;
    if (live) {
      int kb = a.kept[seg * a.budget + i];
      if (kb < 0 || kb >= nb) {
        if (threadIdx.x == 0) record_error(a.status, KVC_ERR_BOUNDS);
        live = false;
      } else {
        src = (((int64_t)l * a.H + h) * a.n_tok + t0 + (int64_t)kb * kBlock + tok) * D;
      }
    } else if (cnt > a.budget && threadIdx.x == 0) {
      record_error(a.status, KVC_ERR_BOUNDS);
    }
    if (!live) {
      st_stream(a.kview + dst + 8 * c, zero);
      st_stream(a.kview + dst + HALF + 8 * c, zero);
      st_stream(a.vview + dst + 8 * c, zero);
      st_stream(a.vview + dst + HALF + 8 * c, zero);
      continue;
    }
    uint4 klo = ld_stream(a.kraw + src + 8 * c);
    uint4 khi = ld_stream(a.kraw + src + HALF + 8 * c);
    uint4 vlo = ld_stream(a.vraw + src + 8 * c);
    uint4 vhi = ld_stream(a.vraw + src + HALF + 8 * c);
    uint4 olo, ohi;
    rotate8<D>(klo, khi, cs, sn, olo, ohi);
    st_stream(a.kview + dst + 8 * c, olo);
    st_stream(a.kview + dst + HALF + 8 * c, ohi);
    st_stream(a.vview + dst + 8 * c, vlo);
    st_stream(a.vview + dst + HALF + 8 * c, vhi);
  }
}

// ------------------------------------------------------------ tiered

struct TieredArgs {
  const uint16_t *kraw_host, *vraw_host;     // [L][H][n_tok][D], host memory; with
                                             // host_slot: slot arenas, see below
  const int32_t *host_slot;  // NULL, or [L][H][n_tok / 32]: host slot of each unit
  int64_t slot_elems;        // elements from one slot to the next
  int32_t n_slots;
  const int32_t *kept_prev, *kept_count_prev;
  const uint16_t *kcache_prev, *vview_prev;  // [L][H][n_sess][32·budget][D]
  const int32_t *kept, *kept_count;
  const int64_t *tok_off;
  const float *rope_tab;
  uint16_t *kcache, *kview, *vview;
  int32_t *n_hits, *status;
  int L, H, n_sess, budget;
  int64_t n_tok;
};

// Position of block kb in the previous ascending kept list, or −1.
__device__ __forceinline__ int find_prev(const int32_t *list, int n, int kb) {
  int lo = 0, hi = n - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int v = __ldg(list + mid);
    if (v == kb) return mid;
    if (v < kb) lo = mid + 1;
    else hi = mid - 1;
  }
  return -1;
}

// As k_pack_rerope, but each kept block's raw K and V come either from the
// previous step's view (a block kept by both steps: its raw K from the
// previous raw-K cache, its V from the previous V view, both in HBM) or, for
// a miss, straight from host memory over the CPU–GPU link.  The block's raw
// K also goes to this step's raw-K cache, so the next step can reuse it.
// With a slot table, host memory holds only some units (layer, head,
// block): unit (l, h, g) (g counted over the whole history) sits in slot
// host_slot[(l·H + h)·(n_tok/32) + g], its K rows at
// kraw_host + slot·slot_elems + t·D (V likewise); a unit without a slot is
// recorded as KVC_ERR_BOUNDS and packed as zeros.
template <int D>
__global__ void __launch_bounds__(2 * D)
k_pack_tiered(TieredArgs a) {
  constexpr int TPT = D / 16;
  constexpr int HALF = D / 2;
  const int tok = threadIdx.x / TPT, c = threadIdx.x % TPT;
  const int i = blockIdx.x;
  const int lr = blockIdx.y;
  const int r = lr % a.n_sess, l = lr / a.n_sess;

  const int64_t t0 = a.tok_off[r], t1 = a.tok_off[r + 1];
  const bool sess_ok = t0 >= 0 && t1 >= t0 && t1 <= a.n_tok && (t0 % kBlock) == 0 &&
                       ((t1 - t0) % kBlock) == 0;
  const int64_t nb = sess_ok ? (t1 - t0) / kBlock : 0;

  float cs[8], sn[8];
  {
    const float4 *tb = reinterpret_cast<const float4 *>(
        a.rope_tab + ((int64_t)(i * kBlock + tok) * HALF + 8 * c) * 2);
#pragma unroll
    for (int e = 0; e < 4; e++) {
      float4 v = __ldg(tb + e);
      cs[2 * e] = v.x;
      sn[2 * e] = v.y;
      cs[2 * e + 1] = v.z;
      sn[2 * e + 1] = v.w;
    }
  }

  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int h = 0; h < a.H; h++) {
    const int64_t seg = ((int64_t)l * a.H + h) * a.n_sess + r;
    const int64_t row0 = seg * a.budget * kBlock;  // first view row of the segment
    const int64_t dst = (row0 + (int64_t)i * kBlock + tok) * D;
    const int cnt = a.kept_count[seg];
    bool live = i < cnt && cnt <= a.budget;
    int kb = -1;
    if (live) {
      kb = a.kept[seg * a.budget + i];
      if (kb < 0 || kb >= nb) {
        if (threadIdx.x == 0) record_error(a.status, KVC_ERR_BOUNDS);
        live = false;
      }
    } else if (cnt > a.budget && threadIdx.x == 0) {
      record_error(a.status, KVC_ERR_BOUNDS);
    }
    if (!live) {
      st_stream(a.kview + dst + 8 * c, zero);
      st_stream(a.kview + dst + HALF + 8 * c, zero);
      st_stream(a.vview + dst + 8 * c, zero);
      st_stream(a.vview + dst + HALF + 8 * c, zero);
      st_stream(a.kcache + dst + 8 * c, zero);
      st_stream(a.kcache + dst + HALF + 8 * c, zero);
      continue;
    }
    int ip = -1;
    if (a.kept_prev) {
      const int cp = min(max(a.kept_count_prev[seg], 0), a.budget);
      ip = find_prev(a.kept_prev + seg * a.budget, cp, kb);
    }
    const uint16_t *ksrc, *vsrc;
    if (ip >= 0) {
      const int64_t src = (row0 + (int64_t)ip * kBlock + tok) * D;
      ksrc = a.kcache_prev + src;
      vsrc = a.vview_prev + src;
    } else if (a.host_slot) {
      const int32_t sl =
          __ldg(a.host_slot + ((int64_t)l * a.H + h) * (a.n_tok / kBlock) + t0 / kBlock + kb);
      if (sl < 0 || sl >= a.n_slots) {
        if (threadIdx.x == 0) record_error(a.status, KVC_ERR_BOUNDS);
        st_stream(a.kview + dst + 8 * c, zero);
        st_stream(a.kview + dst + HALF + 8 * c, zero);
        st_stream(a.vview + dst + 8 * c, zero);
        st_stream(a.vview + dst + HALF + 8 * c, zero);
        st_stream(a.kcache + dst + 8 * c, zero);
        st_stream(a.kcache + dst + HALF + 8 * c, zero);
        continue;
      }
      const int64_t src = (int64_t)sl * a.slot_elems + (int64_t)tok * D;
      ksrc = a.kraw_host + src;
      vsrc = a.vraw_host + src;
    } else {
      const int64_t src = (((int64_t)l * a.H + h) * a.n_tok + t0 + (int64_t)kb * kBlock + tok) * D;
      ksrc = a.kraw_host + src;
      vsrc = a.vraw_host + src;
    }
    if (a.n_hits && ip >= 0 && threadIdx.x == 0) atomicAdd(a.n_hits, 1);
    const uint4 klo = ld_stream(ksrc + 8 * c);
    const uint4 khi = ld_stream(ksrc + HALF + 8 * c);
    const uint4 vlo = ld_stream(vsrc + 8 * c);
    const uint4 vhi = ld_stream(vsrc + HALF + 8 * c);
    uint4 olo, ohi;
    rotate8<D>(klo, khi, cs, sn, olo, ohi);
    st_stream(a.kview + dst + 8 * c, olo);
    st_stream(a.kview + dst + HALF + 8 * c, ohi);
    st_stream(a.vview + dst + 8 * c, vlo);
    st_stream(a.vview + dst + HALF + 8 * c, vhi);
    st_stream(a.kcache + dst + 8 * c, klo);
    st_stream(a.kcache + dst + HALF + 8 * c, khi);
  }
}

}  // namespace

cudaError_t launch_pack_tiered(const uint16_t *kraw_host, const uint16_t *vraw_host,
                               const int32_t *host_slot, int64_t slot_elems, int32_t n_slots,
                               const int32_t *kept_prev, const int32_t *kept_count_prev,
                               const uint16_t *kcache_prev, const uint16_t *vview_prev,
                               const int32_t *kept, const int32_t *kept_count, int L, int H,
                               int D, const int64_t *tok_off, int n_sess, int64_t n_tok,
                               int budget, const float *rope_tab, uint16_t *kcache,
                               uint16_t *kview, uint16_t *vview, int32_t *n_hits,
                               int32_t *status, cudaStream_t s) {
  TieredArgs a{};
  a.kraw_host = kraw_host;
  a.vraw_host = vraw_host;
  a.host_slot = host_slot;
  a.slot_elems = slot_elems;
  a.n_slots = n_slots;
  a.kept_prev = kept_prev;
  a.kept_count_prev = kept_count_prev;
  a.kcache_prev = kcache_prev;
  a.vview_prev = vview_prev;
  a.kept = kept;
  a.kept_count = kept_count;
  a.tok_off = tok_off;
  a.rope_tab = rope_tab;
  a.kcache = kcache;
  a.kview = kview;
  a.vview = vview;
  a.n_hits = n_hits;
  a.status = status;
  a.L = L;
  a.H = H;
  a.n_sess = n_sess;
  a.budget = budget;
  a.n_tok = n_tok;
  dim3 grid(budget, L * n_sess);
  if (D == 128)
    k_pack_tiered<128><<<grid, 256, 0, s>>>(a);
  else
    k_pack_tiered<64><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float *tab, int n_pos, int pos0, int D,
                              double theta, cudaStream_t s) {
  int half = D / 2;
  int64_t n = (int64_t)n_pos * half;
  k_rope_table<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(tab, n_pos, pos0, half,
                                                          D, theta);
  return cudaGetLastError();
}

cudaError_t launch_pack_rerope(const uint16_t *kraw, const uint16_t *vraw,
                               const int32_t *kept, const int32_t *kept_count,
                               int L, int H, int D, const int64_t *tok_off,
                               int n_sess, int64_t n_tok, int budget,
                               const float *rope_tab, uint16_t *kview,
                               uint16_t *vview, int32_t *status,
                               cudaStream_t s) {
  PackArgs a{kraw, vraw, kept, kept_count, tok_off, rope_tab, kview, vview,
             status, L, H, n_sess, budget, n_tok};
  dim3 grid(budget, L * n_sess);
  if (D == 128)
    k_pack_rerope<128><<<grid, 256, 0, s>>>(a);
  else
    k_pack_rerope<64><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvc
