// repo.cu — the repository view of the raw K/V history (KVMem, "Tiered
// movement"): which tier holds each unit (layer, KV head, 32-token block),
// the host-RAM tier as a slot arena, the NVMe tier as a backing file, the
// placement policy (units used most often keep their host slots) and the
// bulk reads of a step's misses.  Host code only; the GPU reads the arena
// through kvc_pack_tiered_slots.
#include <errno.h>
#include <fcntl.h>
#include <limits.h>
#include <stdlib.h>
#include <string.h>
#include <sys/stat.h>
#include <sys/uio.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <new>
#include <stdexcept>
#include <thread>
#include <vector>

#include "kvc.h"

struct kvc_repo {
  int fd = -1;
  bool direct = false;
  int64_t n_blocks = 0;   // blocks of the history
  int64_t n_units = 0;    // L·H·n_blocks
  int L = 0, H = 0, D = 0;
  int64_t rec_elems = 0;  // 2·32·D (K rows, then V rows)
  int64_t rec_bytes = 0;
  int32_t n_slots = 0;
  uint16_t *arena = nullptr;
  int io_threads = 1;
  std::vector<int32_t> slot_of;    // unit → host slot, −1
  std::vector<int64_t> block_in;   // slot → unit, −1
  std::vector<uint8_t> stored;     // unit written to the file
  std::vector<int64_t> uses;       // unit → steps that kept it
  std::vector<int64_t> last;       // unit → last step that kept it
  std::vector<uint8_t> pinned;     // scratch: needed by the current step
  std::vector<int32_t> free_slots;
  std::vector<int64_t> chg_unit;   // the last step's slot changes: unit …
  std::vector<int32_t> chg_slot;   // … and its new slot (−1: evicted)
  kvc_repo_stats st{};
};

namespace {

constexpr int kTok = KVC_BLOCK_TOKENS;

// One vectored write of consecutive records, repeated on a short write until
// every byte is out (iov is advanced in place).
bool pwritev_all(int fd, std::vector<iovec> &iov, int64_t off) {
  size_t first = 0;
  while (first < iov.size()) {
    const int cnt = (int)std::min<size_t>(iov.size() - first, IOV_MAX);
    const ssize_t w = pwritev(fd, iov.data() + first, cnt, (off_t)off);
    if (w < 0 && errno == EINTR) continue;
    if (w <= 0) return false;
    off += w;
    size_t done = (size_t)w;
    while (done > 0 && first < iov.size()) {
      if (done >= iov[first].iov_len) {
        done -= iov[first].iov_len;
        first++;
      } else {
        iov[first].iov_base = static_cast<char *>(iov[first].iov_base) + done;
        iov[first].iov_len -= done;
        done = 0;
      }
    }
  }
  return true;
}

// One vectored read of consecutive records into their slots, repeated on a
// short read until every byte is in (iov is advanced in place).
bool preadv_all(int fd, std::vector<iovec> &iov, int64_t off) {
  size_t first = 0;
  while (first < iov.size()) {
    const int cnt = (int)std::min<size_t>(iov.size() - first, IOV_MAX);
    const ssize_t r = preadv(fd, iov.data() + first, cnt, (off_t)off);
    if (r < 0 && errno == EINTR) continue;
    if (r <= 0) return false;
    off += r;
    size_t got = (size_t)r;
    while (got > 0 && first < iov.size()) {
      if (got >= iov[first].iov_len) {
        got -= iov[first].iov_len;
        first++;
      } else {
        iov[first].iov_base = static_cast<char *>(iov[first].iov_base) + got;
        iov[first].iov_len -= got;
        got = 0;
      }
    }
  }
  return true;
}

// The record of unit u = (l·H + h)·n_blocks + g gathered from
// [L][H][n_tok][D] arrays into dst ([2][32][D]: the unit's K rows, then its
// V rows; both contiguous in the source).
void gather_record(const kvc_repo *r, int64_t u, const uint16_t *kraw, const uint16_t *vraw,
                   int64_t n_tok, uint16_t *dst) {
  const int64_t lh = u / r->n_blocks, g = u % r->n_blocks;
  const int64_t rows = (int64_t)kTok * r->D;
  const int64_t src = (lh * n_tok + g * kTok) * r->D;
  memcpy(dst, kraw + src, (size_t)rows * 2);
  memcpy(dst + rows, vraw + src, (size_t)rows * 2);
}

// Position of kb in an ascending list of n, or −1 (the tiered pack's own
// search, so that the plan's misses are exactly the kernel's).
int find_in(const int32_t *list, int n, int kb) {
  int lo = 0, hi = n - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int v = list[mid];
    if (v == kb) return mid;
    if (v < kb) lo = mid + 1;
    else hi = mid - 1;
  }
  return -1;
}

// kvc_repo_put's body.  Slots go to the put units in order (layer, head,
// block) while free ones remain; then the io_threads threads take the
// (layer, head) rows in turn and write each row's records as vectored writes
// of up to kPutChunk consecutive records, gathering every record into its
// slot or, for a unit without one, into the thread's own staging records.
constexpr int64_t kPutChunk = 64;

kvc_status repo_put(kvc_repo *r, int64_t b0, int64_t nb, const kvc_bf16 *kraw,
                    const kvc_bf16 *vraw, int64_t n_tok) {
  const int64_t rows = (int64_t)r->L * r->H;
  const int nt = (int)std::max<int64_t>(1, std::min<int64_t>(r->io_threads, rows));
  const int64_t chunk = std::min(kPutChunk, nb);
  // allocations first: staging records and the iovec lists of every thread
  uint16_t *staging = nullptr;
  if (posix_memalign(reinterpret_cast<void **>(&staging), 4096,
                     (size_t)(nt * chunk * r->rec_bytes)) != 0)
    return KVC_ERR_NOMEM;
  struct Free {
    void *p;
    ~Free() { free(p); }
  } free_staging{staging};
  std::vector<std::vector<iovec>> iovs((size_t)nt);
  for (auto &v : iovs) v.reserve((size_t)chunk);
  // ---- from here on nothing allocates
  for (int64_t lh = 0; lh < rows; lh++)
    for (int64_t g = b0; g < b0 + nb; g++) {
      const int64_t u = lh * r->n_blocks + g;
      if (r->slot_of[(size_t)u] < 0 && !r->free_slots.empty()) {
        const int32_t slot = r->free_slots.back();
        r->free_slots.pop_back();
        r->slot_of[(size_t)u] = slot;
        r->block_in[(size_t)slot] = u;
      }
    }
  std::atomic<bool> io_ok{true};
  auto worker = [&](int t) {
    std::vector<iovec> &iov = iovs[(size_t)t];
    uint16_t *mine = staging + (int64_t)t * chunk * r->rec_elems;
    for (int64_t lh = t; lh < rows && io_ok; lh += nt)
      for (int64_t g0 = b0; g0 < b0 + nb && io_ok; g0 += chunk) {
        const int64_t n = std::min(chunk, b0 + nb - g0);
        iov.clear();
        for (int64_t i = 0; i < n; i++) {
          const int64_t u = lh * r->n_blocks + g0 + i;
          const int32_t slot = r->slot_of[(size_t)u];
          uint16_t *dst = slot >= 0 ? r->arena + (int64_t)slot * r->rec_elems
                                    : mine + i * r->rec_elems;
          gather_record(r, u, kraw, vraw, n_tok, dst);
          iov.push_back(iovec{dst, (size_t)r->rec_bytes});
        }
        if (!pwritev_all(r->fd, iov, (lh * r->n_blocks + g0) * r->rec_bytes)) {
          io_ok = false;
          break;
        }
        for (int64_t i = 0; i < n; i++) r->stored[(size_t)(lh * r->n_blocks + g0 + i)] = 1;
      }
  };
  std::thread pool[64];
  int started = 0;
  for (int t = 1; t < nt; t++) {
    try {
      pool[started] = std::thread(worker, t);
      started++;
    } catch (...) {
      worker(t);  // no thread to be had: this thread writes that share too
    }
  }
  worker(0);
  for (int t = 0; t < started; t++) pool[t].join();
  if (!io_ok) return KVC_ERR_IO;
  r->st.bytes_written += rows * nb * r->rec_bytes;
  return KVC_OK;
}

kvc_status repo_plan(const int32_t *kept, const int32_t *kept_count, const int32_t *kept_prev,
                     const int32_t *kept_count_prev, int32_t L, int32_t H, int32_t n_sess,
                     int32_t budget, const int64_t *tok_off, int64_t n_blocks, int64_t *used,
                     int64_t *n_used, int64_t *need, int64_t *n_need) {
  // collected per kept entry, then sorted and made unique: the work grows
  // with the kept lists, not with the history
  std::vector<int64_t> vu, vn;
  for (int64_t seg = 0; seg < (int64_t)L * H * n_sess; seg++) {
    const int r = (int)(seg % n_sess);
    const int64_t ubase = (seg / n_sess) * n_blocks;  // unit of (l, h, block 0)
    const int64_t t0 = tok_off[r], t1 = tok_off[r + 1];
    if (t0 < 0 || t1 < t0 || t0 % kTok || (t1 - t0) % kTok || t1 / kTok > n_blocks)
      return KVC_ERR_INVALID_ARG;
    const int64_t nb = (t1 - t0) / kTok, g0 = t0 / kTok;
    const int cnt = kept_count[seg];
    if (cnt < 0 || cnt > budget) return KVC_ERR_BOUNDS;
    const int32_t *list = kept + seg * budget;
    const int32_t *prev = kept_prev ? kept_prev + seg * budget : nullptr;
    const int cp = prev ? std::min(std::max(kept_count_prev[seg], 0), budget) : 0;
    for (int i = 0; i < cnt; i++) {
      const int kb = list[i];
      if (kb < 0 || kb >= nb) return KVC_ERR_BOUNDS;
      vu.push_back(ubase + g0 + kb);
      if (!prev || find_in(prev, cp, kb) < 0) vn.push_back(ubase + g0 + kb);
    }
  }
  for (auto *v : {&vu, &vn}) {
    std::sort(v->begin(), v->end());
    v->erase(std::unique(v->begin(), v->end()), v->end());
  }
  std::copy(vu.begin(), vu.end(), used);
  std::copy(vn.begin(), vn.end(), need);
  *n_used = (int64_t)vu.size();
  *n_need = (int64_t)vn.size();
  return KVC_OK;
}

// kvc_repo_step's body.  Everything it allocates is allocated before the
// repository changes, so an allocation failure (an exception, turned into
// KVC_ERR_NOMEM by the caller) leaves the repository as it was.
kvc_status repo_step(kvc_repo *r, const int64_t *used, int64_t n_used, const int64_t *need,
                     int64_t n_need, int32_t *host_slot) {
  // the step's needed units, once each
  std::vector<int64_t> want;
  std::vector<int64_t> fetch;
  want.reserve((size_t)n_need);
  fetch.reserve((size_t)n_need);
  for (int64_t i = 0; i < n_need; i++)
    if (!r->pinned[(size_t)need[i]]) {
      r->pinned[(size_t)need[i]] = 1;
      want.push_back(need[i]);
    }
  struct Unpin {  // the pins are scratch of this call, whatever happens
    kvc_repo *r;
    const std::vector<int64_t> &want;
    ~Unpin() {
      for (int64_t g : want) r->pinned[(size_t)g] = 0;
    }
  } unpin{r, want};
  if ((int64_t)want.size() > r->n_slots) return KVC_ERR_CAPACITY;
  for (int64_t g : want)
    if (r->slot_of[(size_t)g] < 0) fetch.push_back(g);
  std::sort(fetch.begin(), fetch.end());
  // slots for the fetched units: free ones first, then k taken from others
  const size_t n_free = std::min(fetch.size(), r->free_slots.size());
  const size_t k = fetch.size() - n_free;  // want fits the slots, so k candidates exist
  // runs of consecutive units (consecutive blocks of one layer and head):
  // one vectored read each (at most 1 GiB)
  struct Run {
    int64_t off;
    size_t first, n;
    std::vector<iovec> iov;
  };
  std::vector<Run> runs;
  const size_t max_run = (size_t)std::max<int64_t>(1, (1LL << 30) / r->rec_bytes);
  for (size_t i = 0; i < fetch.size(); i++) {
    if (i == 0 || fetch[i] != fetch[i - 1] + 1 || runs.back().n >= max_run)
      runs.push_back(Run{fetch[i] * r->rec_bytes, i, 0, {}});
    runs.back().n++;
  }
  for (Run &run : runs) run.iov.reserve(run.n);
  std::vector<int32_t> dest, cand;
  dest.reserve(fetch.size());
  if (k > 0) cand.reserve((size_t)r->n_slots);
  std::vector<int64_t> chg_unit;
  std::vector<int32_t> chg_slot;
  chg_unit.reserve(fetch.size() + k);
  chg_slot.reserve(fetch.size() + k);

  // ---- from here on nothing allocates: the repository changes
  r->st.steps++;
  const int64_t step = r->st.steps;
  for (int64_t i = 0; i < n_used; i++) {
    r->uses[(size_t)used[i]]++;
    r->last[(size_t)used[i]] = step;
  }
  r->st.needed += (int64_t)want.size();
  r->st.host_hits += (int64_t)(want.size() - fetch.size());
  for (size_t i = 0; i < n_free; i++) dest.push_back(r->free_slots[r->free_slots.size() - 1 - i]);
  r->free_slots.resize(r->free_slots.size() - n_free);
  if (k > 0) {
    // the slots of the least-used units the step does not need (ties: the
    // least recently used, then the lowest index), with this step's uses counted
    for (int32_t s = 0; s < r->n_slots; s++) {
      const int64_t b = r->block_in[(size_t)s];
      if (b >= 0 && !r->pinned[(size_t)b]) cand.push_back(s);
    }
    auto colder = [&](int32_t x, int32_t y) {
      const int64_t bx = r->block_in[(size_t)x], by = r->block_in[(size_t)y];
      if (r->uses[(size_t)bx] != r->uses[(size_t)by])
        return r->uses[(size_t)bx] < r->uses[(size_t)by];
      if (r->last[(size_t)bx] != r->last[(size_t)by]) return r->last[(size_t)bx] < r->last[(size_t)by];
      return bx < by;
    };
    std::nth_element(cand.begin(), cand.begin() + (ptrdiff_t)(k - 1), cand.end(), colder);
    for (size_t i = 0; i < k; i++) {
      const int32_t s = cand[i];
      const int64_t old = r->block_in[(size_t)s];
      r->slot_of[(size_t)old] = -1;
      r->block_in[(size_t)s] = -1;
      chg_unit.push_back(old);
      chg_slot.push_back(-1);
      r->st.evictions++;
      dest.push_back(s);
    }
  }
  for (size_t i = 0; i < fetch.size(); i++) {
    r->slot_of[(size_t)fetch[i]] = dest[i];
    r->block_in[(size_t)dest[i]] = fetch[i];
    chg_unit.push_back(fetch[i]);
    chg_slot.push_back(dest[i]);
  }
  for (Run &run : runs)
    for (size_t i = run.first; i < run.first + run.n; i++)
      run.iov.push_back(iovec{r->arena + (int64_t)dest[i] * r->rec_elems, (size_t)r->rec_bytes});
  r->chg_unit.swap(chg_unit);
  r->chg_slot.swap(chg_slot);

  std::atomic<bool> io_ok{true};
  auto worker = [&](int t, int nt) {
    for (size_t j = (size_t)t; j < runs.size(); j += (size_t)nt)
      if (!preadv_all(r->fd, runs[j].iov, runs[j].off)) io_ok = false;
  };
  const int nt = (int)std::min<size_t>((size_t)r->io_threads, runs.size());
  if (nt <= 1) {
    worker(0, 1);
  } else {
    std::thread pool[64];
    int started = 0;
    for (int t = 1; t < nt; t++) {
      try {
        pool[started] = std::thread(worker, t, nt);
        started++;
      } catch (...) {
        worker(t, nt);  // no thread to be had: this thread reads that share too
      }
    }
    worker(0, nt);
    for (int t = 0; t < started; t++) pool[t].join();
  }
  if (!io_ok) {
    // the fetched units' slots hold nothing valid: give them back (the free
    // list's capacity is n_slots, so this does not allocate)
    for (int64_t g : fetch) {
      const int32_t s = r->slot_of[(size_t)g];
      r->slot_of[(size_t)g] = -1;
      r->block_in[(size_t)s] = -1;
      r->free_slots.push_back(s);
    }
    // the evictions stand: report them, and the fetched units as slotless
    for (size_t i = 0; i < r->chg_slot.size(); i++)
      if (r->chg_slot[i] >= 0) r->chg_slot[i] = -1;
    return KVC_ERR_IO;
  }
  r->st.fetched += (int64_t)fetch.size();
  r->st.read_calls += (int64_t)runs.size();
  r->st.bytes_read += (int64_t)fetch.size() * r->rec_bytes;
  if (host_slot)
    for (int64_t u = 0; u < r->n_units; u++) host_slot[u] = r->slot_of[(size_t)u];
  return KVC_OK;
}

}  // namespace

extern "C" {

kvc_status kvc_repo_create(const char *path, int64_t n_blocks, int32_t L, int32_t H, int32_t D,
                           int32_t n_slots, kvc_bf16 *arena, int32_t io_threads, int32_t flags,
                           kvc_repo **out) {
  if (!path || !arena || !out || n_blocks < 1 || L < 1 || H < 1 || n_slots < 1 ||
      io_threads < 1 || io_threads > 64 || (flags & ~KVC_REPO_DIRECT_IO))
    return KVC_ERR_INVALID_ARG;
  *out = nullptr;
  if (D != 64 && D != 128) return KVC_ERR_SHAPE;
  const bool direct = (flags & KVC_REPO_DIRECT_IO) != 0;
  if (direct && (reinterpret_cast<uintptr_t>(arena) & 4095u)) return KVC_ERR_ALIGN;
  kvc_repo *r = new (std::nothrow) kvc_repo;
  if (!r) return KVC_ERR_NOMEM;
  r->direct = direct;
  r->n_blocks = n_blocks;
  r->n_units = (int64_t)L * H * n_blocks;
  r->L = L;
  r->H = H;
  r->D = D;
  r->rec_elems = 2LL * kTok * D;
  r->rec_bytes = r->rec_elems * 2;  // 8 or 16 KB: direct I/O sizes are aligned
  r->n_slots = n_slots;
  r->arena = arena;
  r->io_threads = io_threads;
  int oflags = O_RDWR | O_CREAT | O_TRUNC;
#ifdef O_DIRECT
  if (direct) oflags |= O_DIRECT;
#else
  if (direct) {
    delete r;
    return KVC_ERR_IO;
  }
#endif
  r->fd = open(path, oflags, 0600);
  if (r->fd < 0 || ftruncate(r->fd, (off_t)(r->n_units * r->rec_bytes)) != 0) {
    if (r->fd >= 0) close(r->fd);
    delete r;
    return KVC_ERR_IO;
  }
  try {
    r->slot_of.assign((size_t)r->n_units, -1);
    r->stored.assign((size_t)r->n_units, 0);
    r->uses.assign((size_t)r->n_units, 0);
    r->last.assign((size_t)r->n_units, 0);
    r->pinned.assign((size_t)r->n_units, 0);
    r->block_in.assign((size_t)n_slots, -1);
    // the free list's capacity stays n_slots for the repository's life, so
    // giving slots back never allocates
    r->free_slots.resize((size_t)n_slots);
  } catch (const std::exception &) {  // std::bad_alloc, std::length_error
    close(r->fd);
    delete r;
    return KVC_ERR_NOMEM;
  }
  for (int32_t i = 0; i < n_slots; i++) r->free_slots[(size_t)i] = n_slots - 1 - i;
  *out = r;
  return KVC_OK;
}

kvc_status kvc_repo_put(kvc_repo *r, int64_t b0, int64_t nb, const kvc_bf16 *kraw,
                        const kvc_bf16 *vraw, int64_t n_tok) {
  if (!r || !kraw || !vraw || b0 < 0 || nb < 1 || n_tok < 1 || b0 + nb > r->n_blocks ||
      (b0 + nb) * kTok > n_tok)
    return KVC_ERR_INVALID_ARG;
  try {
    return repo_put(r, b0, nb, kraw, vraw, n_tok);
  } catch (const std::exception &) {  // std::bad_alloc, std::length_error
    return KVC_ERR_NOMEM;
  }
}

kvc_status kvc_repo_plan(const int32_t *kept, const int32_t *kept_count,
                         const int32_t *kept_prev, const int32_t *kept_count_prev, int32_t L,
                         int32_t H, int32_t n_sess, int32_t budget, const int64_t *tok_off,
                         int64_t n_blocks, int64_t *used, int64_t *n_used, int64_t *need,
                         int64_t *n_need) {
  if (!kept || !kept_count || !tok_off || !used || !n_used || !need || !n_need || L < 1 ||
      H < 1 || n_sess < 1 || budget < 1 || n_blocks < 1 || (kept_prev && !kept_count_prev))
    return KVC_ERR_INVALID_ARG;
  try {
    return repo_plan(kept, kept_count, kept_prev, kept_count_prev, L, H, n_sess, budget, tok_off,
                     n_blocks, used, n_used, need, n_need);
  } catch (const std::exception &) {  // std::bad_alloc, std::length_error
    return KVC_ERR_NOMEM;
  }
}


kvc_status kvc_repo_step(kvc_repo *r, const int64_t *used, int64_t n_used, const int64_t *need,
                         int64_t n_need, int32_t *host_slot) {
  if (!r || n_used < 0 || n_need < 0 || (n_used && !used) || (n_need && !need))
    return KVC_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n_used; i++)
    if (used[i] < 0 || used[i] >= r->n_units) return KVC_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n_need; i++)
    if (need[i] < 0 || need[i] >= r->n_units || !r->stored[(size_t)need[i]])
      return KVC_ERR_INVALID_ARG;
  try {
    return repo_step(r, used, n_used, need, n_need, host_slot);
  } catch (const std::exception &) {  // std::bad_alloc, std::length_error
    return KVC_ERR_NOMEM;
  }
}

kvc_status kvc_repo_slots(const kvc_repo *r, int32_t *host_slot) {
  if (!r || !host_slot) return KVC_ERR_INVALID_ARG;
  for (int64_t u = 0; u < r->n_units; u++) host_slot[u] = r->slot_of[(size_t)u];
  return KVC_OK;
}

int64_t kvc_repo_changes(const kvc_repo *r, int64_t *units, int32_t *slots, int64_t cap) {
  if (!r || cap < 0 || (cap > 0 && (!units || !slots))) return -1;
  const int64_t n = (int64_t)r->chg_unit.size();
  for (int64_t i = 0; i < std::min(n, cap); i++) {
    units[i] = r->chg_unit[(size_t)i];
    slots[i] = r->chg_slot[(size_t)i];
  }
  return n;
}

int32_t kvc_repo_where(const kvc_repo *r, int64_t u) {
  if (!r || u < 0 || u >= r->n_units) return -1;
  if (!r->stored[(size_t)u]) return 0;
  return r->slot_of[(size_t)u] >= 0 ? 1 : 2;
}

kvc_status kvc_repo_get_stats(const kvc_repo *r, kvc_repo_stats *out) {
  if (!r || !out) return KVC_ERR_INVALID_ARG;
  *out = r->st;
  return KVC_OK;
}

void kvc_repo_destroy(kvc_repo *r) {
  if (!r) return;
  if (r->fd >= 0) close(r->fd);
  delete r;
}

}  // extern "C"
