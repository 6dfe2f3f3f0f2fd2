// redirect.cu — slot-map redirection to the dead slot and alias-aware free.
//
// IntentKV §4 "Redirect": S_r[j] ← s† for every dropped position j; kept
// positions and every K/V row stay where they are.  IntentKV §4 check 6 and
// §7: a dropped slot u is returned to the allocator only if j is outside
// the protected prefix, u ≠ s†, and no remaining reference (a sibling
// session's, or an alias inside the same map) still holds u.  Every map
// entry holds one count of its slot, so "no remaining reference" is "the
// count reached zero".
//
// The result equals visiting positions in (session, position) order; the
// GPU gets there without serialising:
//   k_redirect_drop   one thread per position: dropped entries decrement
//                     their slot's count atomically, are redirected, and
//                     publish their flat position p = r·N + j into
//                     last[u] with atomicMax (the slot's last dropper in
//                     visiting order);
//   k_redirect_count  a position frees u iff it is u's last dropper, u's
//                     count is now zero and j ≥ prefix_len — per-block
//                     counts of such positions;
//   k_redirect_scan   one CTA turns the counts into offsets (and n_freed);
//   k_redirect_emit   each block writes its freed slots at its offset, in
//                     position order — the list order of the sequential
//                     definition, deterministic.
// Scratch: last[n_slots], orig[n_sess·N] and the per-block counts.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kRThreads = 1024;

struct RArgs {
  int32_t *slot_map;
  const uint32_t *keepmask;
  int32_t *refcnt;
  int32_t *freed;
  int32_t *n_freed;
  int32_t *last;   // [n_slots]
  int32_t *orig;   // [n_sess·N]: dropped slot or −1
  int32_t *bsum;   // [n_blocks]
  int32_t *status;
  int n_sess, N, words, prefix_len, sentinel, freed_cap, n_blocks;
  int64_t n_slots, n_pos;
};

__global__ void __launch_bounds__(256)
k_redirect_drop(RArgs a) {
  int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= a.n_pos) return;
  int r = (int)(p / a.N), j = (int)(p - (int64_t)r * a.N);
  uint32_t word = a.keepmask[(int64_t)r * a.words + (j >> 5)];
  int32_t out = -1;
  if (!((word >> (j & 31)) & 1u)) {
    int32_t u = a.slot_map[p];
    if (u != a.sentinel) {
      if (u < 0 || u >= a.n_slots) {
        record_error(a.status, KVC_ERR_BOUNDS);
      } else {
        int32_t old = atomicSub(&a.refcnt[u], 1);
        if (old < 1) {
          atomicAdd(&a.refcnt[u], 1);
          record_error(a.status, KVC_ERR_BOUNDS);
        } else {
          a.slot_map[p] = a.sentinel;
          atomicMax(&a.last[u], (int32_t)p);
          out = u;
        }
      }
    }
  }
  a.orig[p] = out;
}

__device__ __forceinline__ bool frees(const RArgs &a, int64_t p) {
  if (p >= a.n_pos) return false;
  int32_t u = a.orig[p];
  if (u < 0) return false;
  int j = (int)(p % a.N);
  return j >= a.prefix_len && a.refcnt[u] == 0 && a.last[u] == (int32_t)p;
}

__device__ __forceinline__ int block_excl_scan(int v, int *total, int *warp_tot) {
  int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int n_warps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < n_warps ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  int excl = x - v + (warp > 0 ? warp_tot[warp - 1] : 0);
  *total = warp_tot[n_warps - 1];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(kRThreads)
k_redirect_count(RArgs a) {
  __shared__ int warp_tot[32];
  int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int tot;
  block_excl_scan(frees(a, p) ? 1 : 0, &tot, warp_tot);
  if (threadIdx.x == 0) a.bsum[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(kRThreads)
k_redirect_scan(RArgs a) {
  __shared__ int warp_tot[32];
  int carry = 0;
  for (int base = 0; base < a.n_blocks; base += blockDim.x) {
    int i = base + threadIdx.x;
    int v = i < a.n_blocks ? a.bsum[i] : 0;
    int tot;
    int ex = block_excl_scan(v, &tot, warp_tot);
    if (i < a.n_blocks) a.bsum[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) {
    *a.n_freed = carry;
    if (carry > a.freed_cap) record_error(a.status, KVC_ERR_CAPACITY);
  }
}

__global__ void __launch_bounds__(kRThreads)
k_redirect_emit(RArgs a) {
  __shared__ int warp_tot[32];
  int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  bool f = frees(a, p);
  int tot;
  int rank = block_excl_scan(f ? 1 : 0, &tot, warp_tot);
  int pos = a.bsum[blockIdx.x] + rank;
  if (f && pos < a.freed_cap) a.freed[pos] = a.orig[p];
}

struct WsLayout {
  size_t last, orig, bsum, total;
};

WsLayout ws_layout(int n_sess, int N, int64_t n_slots) {
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  int64_t n_pos = (int64_t)n_sess * N;
  int64_t n_blocks = (n_pos + kRThreads - 1) / kRThreads;
  WsLayout w;
  w.last = 0;
  w.orig = al((size_t)n_slots * 4);
  w.bsum = w.orig + al((size_t)n_pos * 4);
  w.total = w.bsum + al((size_t)n_blocks * 4);
  return w;
}

}  // namespace

size_t redirect_free_ws_bytes(int n_sess, int N, int64_t n_slots) {
  return ws_layout(n_sess, N, n_slots).total;
}

cudaError_t launch_redirect_free(int32_t *slot_map, const uint32_t *keepmask,
                                 int n_sess, int N, int32_t *refcnt,
                                 int64_t n_slots, int prefix_len,
                                 int32_t sentinel, int32_t *freed,
                                 int freed_cap, int32_t *n_freed, void *ws,
                                 int32_t *status, cudaStream_t s) {
  WsLayout w = ws_layout(n_sess, N, n_slots);
  char *base = static_cast<char *>(ws);
  RArgs a;
  a.slot_map = slot_map;
  a.keepmask = keepmask;
  a.refcnt = refcnt;
  a.freed = freed;
  a.n_freed = n_freed;
  a.last = reinterpret_cast<int32_t *>(base + w.last);
  a.orig = reinterpret_cast<int32_t *>(base + w.orig);
  a.bsum = reinterpret_cast<int32_t *>(base + w.bsum);
  a.status = status;
  a.n_sess = n_sess;
  a.N = N;
  a.words = (N + 31) / 32;
  a.prefix_len = prefix_len;
  a.sentinel = sentinel;
  a.freed_cap = freed_cap;
  a.n_slots = n_slots;
  a.n_pos = (int64_t)n_sess * N;
  a.n_blocks = (int)((a.n_pos + kRThreads - 1) / kRThreads);
  cudaError_t e = cudaMemsetAsync(a.last, 0xFF, (size_t)n_slots * 4, s);  // −1
  if (e != cudaSuccess) return e;
  k_redirect_drop<<<(unsigned)((a.n_pos + 255) / 256), 256, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_redirect_count<<<a.n_blocks, kRThreads, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_redirect_scan<<<1, kRThreads, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_redirect_emit<<<a.n_blocks, kRThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvc
