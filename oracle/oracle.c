/*
 * oracle.c — plain, slow, obviously-correct CPU reference of the
 * query-conditioned KV compression event.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file, and this file includes nothing of the product: the two
 * share no code.  Only the test-suite, the package smoke check and the CPU
 * baseline leg of the benchmark load it.
 *
 * Every function is the plain definition of one step, written in scalar C
 * with fp64 arithmetic, in the order the pages state it; no blocking, no
 * fusion, no reordering.  Each cites the page and section it follows:
 *   [ActKV]   ActKV: Efficient LLM Agents through Action-Guided KV Cache
 *             Management
 *   [IntentKV] IntentKV: Cross-Turn Intent-Aware KV Cache Pruning for Agent
 *             Inference
 *   [KVMem]   KVMem: Virtualizing Million-Token Agent Workspaces on a
 *             Consumer GPU
 * Where the pages leave a step open, the reading taken is stated at the
 * function.  All functions return 0 on success and a positive code on a bad
 * argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BLOCK 32 /* [KVMem] "Query-conditioned retrieval": 32-token blocks */

/* ---------------------------------------------------------------- bf16 */

/* bf16 bit pattern → exact fp64 value. */
double orc_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* fp64 → bf16 with one round-to-nearest-even step (no double rounding
 * through fp32): keep 8 significant bits of the normalised significand; in
 * the subnormal range the spacing is 2^-133. */
uint16_t orc_f64_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0u;
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double a = fabs(x);
  if (a == 0.0) return sign;
  double r;
  if (a < ldexp(1.0, -126)) {
    r = ldexp(nearbyint(ldexp(a, 133)), -133);
  } else {
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, 0.5 <= m < 1 */
    r = ldexp(nearbyint(ldexp(m, 8)), e - 8);
  }
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

/* ------------------------------------------------------------ Mean-K */

/* [KVMem] "Query-conditioned retrieval": one RoPE-stripped mean key per
 * (layer, KV head, 32-token block).  kraw is [rows][n_tok][D] pre-RoPE keys
 * (rows = layers × KV heads); meank is [rows][n_tok/32][D].
 * Reading: the mean is the exact fp64 mean rounded once to bf16. */
int orc_meank(const uint16_t *kraw, uint16_t *meank, int64_t rows,
              int64_t n_tok, int D) {
  if (!kraw || !meank || rows < 1 || n_tok < ORC_BLOCK || D < 1) return 1;
  if (n_tok % ORC_BLOCK) return 2;
  int64_t nb = n_tok / ORC_BLOCK;
  for (int64_t r = 0; r < rows; r++)
    for (int64_t b = 0; b < nb; b++)
      for (int d = 0; d < D; d++) {
        double sum = 0.0;
        for (int t = 0; t < ORC_BLOCK; t++)
          sum += orc_bf16_to_f64(
              kraw[(r * n_tok + b * ORC_BLOCK + t) * D + d]);
        meank[(r * nb + b) * D + d] = orc_f64_to_bf16(sum / ORC_BLOCK);
      }
  return 0;
}

/* ------------------------------------------------------------- score */

/* Score of one (session, layer, KV head) unit in Mean-K mode.
 * [KVMem] "Query-conditioned retrieval": blocks are scored in the model's
 * own attention space, q · MeanKᵀ / sqrt(D) with the pre-RoPE query, and
 * turned into attention mass by a softmax over the history blocks.
 * [ActKV] §7.1 (Algorithm 3): the per-KV-head score is the maximum over the
 * query heads of the GQA group and the mean over the query tokens.
 *   q      [G][W][D] bf16: the G query heads of this KV head, W tokens each
 *   meank  [Nb][D] bf16
 *   score  [Nb] fp32 out
 * z[w,g,b] = q[g,w]·meank[b]/sqrt(D);  LSE[w,g] = log Σ_b e^z (max-shifted);
 * score[b] = (1/W) Σ_w max_g exp(z[w,g,b] − LSE[w,g]), rounded to fp32. */
int orc_score_unit(const uint16_t *q, const uint16_t *meank, int G, int W,
                   int D, int64_t nb, float *score) {
  if (!q || !meank || !score || G < 1 || W < 1 || D < 1 || nb < 1) return 1;
  double *z = (double *)malloc(sizeof(double) * (size_t)G * W * nb);
  double *lse = (double *)malloc(sizeof(double) * (size_t)G * W);
  if (!z || !lse) {
    free(z);
    free(lse);
    return 3;
  }
  double inv_sqrt_d = 1.0 / sqrt((double)D);
  for (int g = 0; g < G; g++)
    for (int w = 0; w < W; w++) {
      const uint16_t *qr = q + ((int64_t)g * W + w) * D;
      double *zr = z + ((int64_t)g * W + w) * nb;
      for (int64_t b = 0; b < nb; b++) {
        double dot = 0.0;
        for (int d = 0; d < D; d++)
          dot += orc_bf16_to_f64(qr[d]) * orc_bf16_to_f64(meank[b * D + d]);
        zr[b] = dot * inv_sqrt_d;
      }
      double m = -INFINITY;
      for (int64_t b = 0; b < nb; b++)
        if (zr[b] > m) m = zr[b];
      double s = 0.0;
      for (int64_t b = 0; b < nb; b++) s += exp(zr[b] - m);
      lse[g * W + w] = m + log(s);
    }
  for (int64_t b = 0; b < nb; b++) {
    double acc = 0.0;
    for (int w = 0; w < W; w++) {
      double best = 0.0;
      for (int g = 0; g < G; g++) {
        double p = exp(z[((int64_t)g * W + w) * nb + b] - lse[g * W + w]);
        if (p > best) best = p;
      }
      acc += best;
    }
    score[b] = (float)(acc / W);
  }
  free(z);
  free(lse);
  return 0;
}

/* ------------------------------------------------------- QueryMemory */

/* [IntentKV] §4 "Memory recurrence" and §7 item 1: M_t = e^{-λ} M_{t-1} +
 * Enc(q_t), then renormalised to unit norm along the head dimension.
 * Reading: Enc(q_t) = gain · (mean over the turn's T query tokens), with
 * decay = e^{-λ}; a zero vector is left at zero by the renormalisation.
 *   M  [rows][D] fp32 in/out (rows = sessions × layers × query heads)
 *   q  [rows][T][D] bf16 */
int orc_qmem_update(float *M, const uint16_t *q, int64_t rows, int T, int D,
                    double decay, double gain, int renorm) {
  if (!M || !q || rows < 1 || T < 1 || D < 1) return 1;
  double *v = (double *)malloc(sizeof(double) * (size_t)D);
  if (!v) return 3;
  for (int64_t r = 0; r < rows; r++) {
    for (int d = 0; d < D; d++) {
      double mean = 0.0;
      for (int t = 0; t < T; t++)
        mean += orc_bf16_to_f64(q[(r * T + t) * D + d]);
      mean /= T;
      v[d] = decay * (double)M[r * D + d] + gain * mean;
    }
    if (renorm) {
      double n2 = 0.0;
      for (int d = 0; d < D; d++) n2 += v[d] * v[d];
      double n = sqrt(n2);
      if (n > 0.0)
        for (int d = 0; d < D; d++) v[d] /= n;
    }
    for (int d = 0; d < D; d++) M[r * D + d] = (float)v[d];
  }
  free(v);
  return 0;
}

/* Rule score of one session (QueryMemory mode).
 * [IntentKV] §4 "Rule score": rule_j = Σ_{l,h} softmax_j(M[l,h]·K[l,h,j]/√D),
 * with §4 check 1: GQA KV heads expanded to the query heads (query head hq
 * reads KV head hq / G).  K is read through the paged slot map ([ActKV] §2:
 * a logical position resolves to a physical slot).
 * Reading: positions whose slot is the dead slot are no longer history; they
 * are left out of every softmax and get rule = -1.
 *   M         [L][Hq][D] fp32
 *   kpool     [L][n_slots][H][D] bf16
 *   slot_map  [N] int32
 *   rule      [N] fp32 out */
int orc_rule_session(const float *M, const uint16_t *kpool, int64_t n_slots,
                     const int32_t *slot_map, int N, int L, int H, int Hq,
                     int D, int32_t sentinel, float *rule) {
  if (!M || !kpool || !slot_map || !rule || N < 1 || L < 1 || H < 1 ||
      Hq < H || Hq % H || D < 1)
    return 1;
  int G = Hq / H;
  for (int j = 0; j < N; j++)
    if (slot_map[j] != sentinel && (slot_map[j] < 0 || slot_map[j] >= n_slots))
      return 4;
  double *acc = (double *)calloc((size_t)N, sizeof(double));
  double *z = (double *)malloc(sizeof(double) * (size_t)N);
  if (!acc || !z) {
    free(acc);
    free(z);
    return 3;
  }
  double inv_sqrt_d = 1.0 / sqrt((double)D);
  int n_live = 0;
  for (int j = 0; j < N; j++) n_live += slot_map[j] != sentinel;
  for (int l = 0; l < L; l++)
    for (int hq = 0; hq < Hq; hq++) {
      int h = hq / G;
      const float *m = M + ((int64_t)l * Hq + hq) * D;
      double zmax = -INFINITY;
      for (int j = 0; j < N; j++) {
        if (slot_map[j] == sentinel) continue;
        const uint16_t *k =
            kpool + (((int64_t)l * n_slots + slot_map[j]) * H + h) * D;
        double dot = 0.0;
        for (int d = 0; d < D; d++) dot += (double)m[d] * orc_bf16_to_f64(k[d]);
        z[j] = dot * inv_sqrt_d;
        if (z[j] > zmax) zmax = z[j];
      }
      if (n_live == 0) continue;
      double s = 0.0;
      for (int j = 0; j < N; j++)
        if (slot_map[j] != sentinel) s += exp(z[j] - zmax);
      double lse = zmax + log(s);
      for (int j = 0; j < N; j++)
        if (slot_map[j] != sentinel) acc[j] += exp(z[j] - lse);
    }
  for (int j = 0; j < N; j++)
    rule[j] = slot_map[j] == sentinel ? -1.0f : (float)acc[j];
  free(acc);
  free(z);
  return 0;
}

/* ------------------------------------------------------------ select */

typedef struct {
  float key;
  int32_t idx;
} orc_item;

/* (score descending, index ascending); -0.0 == +0.0 under C's ==. */
static int orc_item_cmp(const void *a, const void *b) {
  const orc_item *x = (const orc_item *)a, *y = (const orc_item *)b;
  if (x->key > y->key) return -1;
  if (x->key < y->key) return 1;
  return (x->idx > y->idx) - (x->idx < y->idx);
}

static int orc_int_cmp(const void *a, const void *b) {
  int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
  return (x > y) - (x < y);
}

/* One segment of the budgeted top-k with a forced set.
 * [IntentKV] §4 "Top-k selection": K* = F ∪ argtop_{|K|=C*} Σ_{j∈K} s_j —
 * the maximum-sum C*-subset of the non-forced items, i.e. the C* largest
 * scores, always keeping the forced set F.
 * [KVMem] "Query-conditioned retrieval": sink and recent blocks are always
 * kept (F), the rest of the budget is filled by score, and the survivors are
 * restored in chronological order (ascending index).
 * [ActKV] §3.3: the eviction output is a Boolean keep mask.
 * Readings: the budget counts F (C* = budget − |F|); F is the union of the
 * first n_sink and the last n_recent items, clipped to the segment; if
 * n ≤ budget every item is kept; equal scores keep the lower index; NaN
 * scores are rejected (return 5).
 *   kept  [budget] int32 out: ascending indices, -1 past *count
 *   mask  [ceil(n/32)] uint32 out or NULL */
int orc_select(const float *scores, int n, int budget, int n_sink,
               int n_recent, int32_t *kept, int32_t *count, uint32_t *mask) {
  if (!scores || !kept || !count || n < 1 || budget < 1 || n_sink < 0 ||
      n_recent < 0)
    return 1;
  if (n_sink + n_recent > budget) return 2;
  for (int i = 0; i < n; i++)
    if (isnan(scores[i])) return 5;
  char *keep = (char *)calloc((size_t)n, 1);
  orc_item *items = (orc_item *)malloc(sizeof(orc_item) * (size_t)n);
  if (!keep || !items) {
    free(keep);
    free(items);
    return 3;
  }
  if (n <= budget) {
    for (int i = 0; i < n; i++) keep[i] = 1;
  } else {
    int n_forced = 0;
    for (int i = 0; i < n; i++)
      if (i < n_sink || i >= n - n_recent) {
        keep[i] = 1;
        n_forced++;
      }
    int m = 0;
    for (int i = 0; i < n; i++)
      if (!keep[i]) {
        items[m].key = scores[i];
        items[m].idx = i;
        m++;
      }
    qsort(items, (size_t)m, sizeof(orc_item), orc_item_cmp);
    int take = budget - n_forced;
    for (int t = 0; t < take && t < m; t++) keep[items[t].idx] = 1;
  }
  int c = 0;
  for (int i = 0; i < n; i++)
    if (keep[i]) kept[c++] = i;
  qsort(kept, (size_t)c, sizeof(int32_t), orc_int_cmp); /* already sorted */
  for (int i = c; i < budget; i++) kept[i] = -1;
  *count = c;
  if (mask) {
    int words = (n + 31) / 32;
    for (int w = 0; w < words; w++) mask[w] = 0;
    for (int i = 0; i < n; i++)
      if (keep[i]) mask[i / 32] |= 1u << (i % 32);
  }
  free(keep);
  free(items);
  return 0;
}

/* -------------------------------------------------------------- RoPE */

/* Rotary embedding of one vector at one position, in fp64 throughout.
 * Reading (the pages name Qwen-family models but print no formula): NeoX
 * rotate-half, element j paired with j + D/2, angle = pos · theta^(−2j/D),
 *   (x_j, x_{j+D/2}) → (x_j cos − x_{j+D/2} sin, x_{j+D/2} cos + x_j sin). */
int orc_rope_f64(const double *x, double *out, int D, double pos,
                 double theta) {
  if (!x || !out || D < 2 || D % 2) return 1;
  int half = D / 2;
  for (int j = 0; j < half; j++) {
    double freq = pow(theta, -2.0 * (double)j / (double)D);
    double a = pos * freq;
    double c = cos(a), s = sin(a);
    out[j] = x[j] * c - x[j + half] * s;
    out[j + half] = x[j + half] * c + x[j] * s;
  }
  return 0;
}

/* Execution-view pack of one (session, layer, KV head) unit.
 * [KVMem] "Tiered movement": the selected blocks are packed into contiguous
 * logical positions; raw (position-independent) K is re-RoPEd at the new
 * positions and V is copied as-is.
 * View token i (< 32·count) comes from history token 32·kept[i/32] + i%32 and
 * sits at position pos0 + i; view tokens past 32·count are zero.
 *   kraw, vraw    [n_tok][D] bf16 (pre-RoPE K, V of this unit)
 *   kview, vview  [32·budget][D] bf16 out
 * K is rotated in fp64 from the bf16 input and rounded once to bf16. */
int orc_pack_unit(const uint16_t *kraw, const uint16_t *vraw, int64_t n_tok,
                  int D, const int32_t *kept, int count, int budget,
                  int64_t pos0, double theta, uint16_t *kview,
                  uint16_t *vview) {
  if (!kraw || !vraw || !kept || !kview || !vview || D < 2 || D % 2 ||
      count < 0 || count > budget || n_tok % ORC_BLOCK)
    return 1;
  int64_t nb = n_tok / ORC_BLOCK;
  for (int i = 0; i < count; i++)
    if (kept[i] < 0 || kept[i] >= nb) return 4;
  double *x = (double *)malloc(sizeof(double) * (size_t)D);
  double *y = (double *)malloc(sizeof(double) * (size_t)D);
  if (!x || !y) {
    free(x);
    free(y);
    return 3;
  }
  int64_t n_view = (int64_t)ORC_BLOCK * budget;
  for (int64_t i = 0; i < n_view; i++) {
    uint16_t *ko = kview + i * D, *vo = vview + i * D;
    if (i >= (int64_t)ORC_BLOCK * count) {
      for (int d = 0; d < D; d++) ko[d] = vo[d] = 0;
      continue;
    }
    int64_t src = (int64_t)ORC_BLOCK * kept[i / ORC_BLOCK] + i % ORC_BLOCK;
    for (int d = 0; d < D; d++) x[d] = orc_bf16_to_f64(kraw[src * D + d]);
    orc_rope_f64(x, y, D, (double)(pos0 + i), theta);
    for (int d = 0; d < D; d++) ko[d] = orc_f64_to_bf16(y[d]);
    memcpy(vo, vraw + src * D, sizeof(uint16_t) * (size_t)D);
  }
  free(x);
  free(y);
  return 0;
}

/* ---------------------------------------------------- paged addressing */

/* [ActKV] §2 (paged KV background): a block table maps logical blocks to
 * physical blocks of BS slots; logical position p lives in slot
 * block_table[p / BS] · BS + p % BS.  Fills slot_map[0 .. seqused-1]. */
int orc_slot_map(const int32_t *block_table, int n_blocks, int BS,
                 int seqused, int32_t *slot_map) {
  if (!block_table || !slot_map || BS < 1 || seqused < 0 ||
      seqused > n_blocks * BS)
    return 1;
  for (int p = 0; p < seqused; p++)
    slot_map[p] = block_table[p / BS] * BS + p % BS;
  return 0;
}

/* ------------------------------------------------- redirect and free */

/* Slot-map redirection with alias-aware freeing, all sessions of one event.
 * [IntentKV] §4 "Redirect": S_r[j] ← s† for every dropped j (kept positions
 * and all K/V rows stay where they are).
 * [IntentKV] §4 check 6 and §7: a dropped slot u = S_r[j] is freed only if
 * (a) j is outside the protected prefix, (b) u ≠ s†, (c) no remaining
 * reference holds u (siblings' and earlier redirects' aliases included).
 * Reading: every slot-map entry holds one count in refcnt and (c) is "the
 * count reaches zero"; positions are visited in (session, position) order,
 * so the freed list is ordered by each slot's last dropping reference, and
 * (a) is judged at that reference.
 *   slot_map [n_sess][N] in/out;  keepmask [n_sess][ceil(N/32)]
 *   refcnt [n_slots] in/out;  freed [cap] out;  *n_freed out
 * Returns 4 on a slot out of range or a count below zero, 6 on overflow of
 * cap (the list is truncated). */
int orc_redirect_free(int32_t *slot_map, const uint32_t *keepmask, int n_sess,
                      int N, int32_t *refcnt, int64_t n_slots, int prefix_len,
                      int32_t sentinel, int32_t *freed, int cap,
                      int32_t *n_freed) {
  if (!slot_map || !keepmask || !refcnt || !freed || !n_freed || n_sess < 1 ||
      N < 1 || cap < 0)
    return 1;
  int words = (N + 31) / 32;
  int nf = 0, rc = 0;
  for (int r = 0; r < n_sess; r++)
    for (int j = 0; j < N; j++) {
      int kept = (keepmask[(int64_t)r * words + j / 32] >> (j % 32)) & 1u;
      if (kept) continue;
      int32_t *e = slot_map + (int64_t)r * N + j;
      int32_t u = *e;
      if (u == sentinel) continue;
      if (u < 0 || u >= n_slots || refcnt[u] < 1) {
        rc = 4;
        continue;
      }
      *e = sentinel;
      refcnt[u] -= 1;
      if (refcnt[u] == 0 && j >= prefix_len) {
        if (nf < cap)
          freed[nf] = u;
        else
          rc = rc ? rc : 6;
        nf++;
      }
    }
  *n_freed = nf;
  return rc;
}

/* ------------------------------------------------ LSE-recovery scoring */

/* The attention backend's by-product: for one request's query rows q
 * [L][Hq][D] (bf16, the current decode step) against its first seq_len
 * cached keys (paged: position p in slot block_table[p / BS]·BS + p % BS of
 * kpool [L][n_slots][H][D]), lse[l][hq] = ln Σ_p exp(q·k/√D), query head hq
 * reading KV head hq / G.  [ActKV] §7.1: the LSE of the softmax
 * normalisation over the keys the query attends to. */
int orc_attention_lse(const uint16_t *q, const uint16_t *kpool, int64_t n_slots,
                      const int32_t *block_table, int BS, int seq_len, int L, int H,
                      int Hq, int D, double *lse) {
  if (!q || !kpool || !block_table || !lse || BS < 1 || seq_len < 1 || L < 1 ||
      H < 1 || Hq < H || Hq % H || D < 1)
    return 1;
  const int G = Hq / H;
  const double inv_sqrt_d = 1.0 / sqrt((double)D);
  double *s = (double *)malloc(sizeof(double) * (size_t)seq_len);
  if (!s) return 3;
  for (int l = 0; l < L; l++)
    for (int hq = 0; hq < Hq; hq++) {
      const int h = hq / G;
      double mx = -INFINITY;
      for (int p = 0; p < seq_len; p++) {
        const int64_t slot = (int64_t)block_table[p / BS] * BS + p % BS;
        if (slot < 0 || slot >= n_slots) {
          free(s);
          return 4;
        }
        const uint16_t *k = kpool + (((int64_t)l * n_slots + slot) * H + h) * D;
        const uint16_t *qq = q + ((int64_t)l * Hq + hq) * D;
        double dot = 0.0;
        for (int d = 0; d < D; d++) dot += orc_bf16_to_f64(qq[d]) * orc_bf16_to_f64(k[d]);
        s[p] = dot * inv_sqrt_d;
        if (s[p] > mx) mx = s[p];
      }
      double sum = 0.0;
      for (int p = 0; p < seq_len; p++) sum += exp(s[p] - mx);
      lse[l * Hq + hq] = mx + log(sum);
    }
  free(s);
  return 0;
}

/* One decode step of the action score of one request.
 * [ActKV] §7.1 (Algorithm 3): for each cached key, the attention
 * probability of the current query token is recovered from the backend's
 * LSE as exp(q·k/√D − LSE); the maximum is taken over the query heads of
 * the key's GQA group, and a running mean over the action tokens is
 * updated in place (no past queries are kept); the state restarts at the
 * first token of an action region.
 * Readings: a token's score sums that group maximum over the layers and KV
 * heads (a slot holds every layer's KV of one token, so eviction on paged
 * memory is per token); keys at positions ≥ seq_len are not visible to the
 * query and contribute 0; the mean is state ← state + (x − state)/count,
 * with count the number of action tokens so far, this one included
 * (count = 1 restarts it: state ← x).
 *   q [L][Hq][D] bf16;  lse [L][Hq] (natural log);  kpool [L][n_slots][H][D]
 *   block_table [n_blocks];  state [n_blocks·BS] in/out */
int orc_recover_step(const uint16_t *q, const double *lse, const uint16_t *kpool,
                     int64_t n_slots, const int32_t *block_table, int n_blocks, int BS,
                     int seq_len, int count, int L, int H, int Hq, int D, double *state) {
  if (!q || !lse || !kpool || !block_table || !state || BS < 1 || n_blocks < 1 ||
      seq_len < 0 || seq_len > n_blocks * BS || count < 1 || L < 1 || H < 1 || Hq < H ||
      Hq % H || D < 1)
    return 1;
  const int G = Hq / H;
  const double inv_sqrt_d = 1.0 / sqrt((double)D);
  for (int p = 0; p < n_blocks * BS; p++) {
    double x = 0.0;
    if (p < seq_len) {
      const int64_t slot = (int64_t)block_table[p / BS] * BS + p % BS;
      if (slot < 0 || slot >= n_slots) return 4;
      for (int l = 0; l < L; l++)
        for (int h = 0; h < H; h++) {
          const uint16_t *k = kpool + (((int64_t)l * n_slots + slot) * H + h) * D;
          double best = 0.0;
          for (int g = 0; g < G; g++) {
            const int hq = h * G + g;
            const uint16_t *qq = q + ((int64_t)l * Hq + hq) * D;
            double dot = 0.0;
            for (int d = 0; d < D; d++) dot += orc_bf16_to_f64(qq[d]) * orc_bf16_to_f64(k[d]);
            const double prob = exp(dot * inv_sqrt_d - lse[l * Hq + hq]);
            if (prob > best) best = prob;
          }
          x += best;
        }
    }
    state[p] = count == 1 ? x : state[p] + (x - state[p]) / count;
  }
  return 0;
}

/* ------------------------------------------------- tail compaction plan */

/* Conflict-free slot plan of one request.  [ActKV] §7.2 (Algorithm 4):
 * after eviction, every retained entry is compacted into the last X logical
 * blocks of the request; destinations are the evicted slots inside that
 * tail region, sources the retained entries outside it, and the two sets
 * are disjoint, so one pass of copies needs no buffer; the blocks before
 * the region are returned.
 * Readings (the region's formula is lost on the page): with Y = ⌈n/BS⌉
 * blocks holding the request's n tokens and m retained tokens, X = ⌈m/BS⌉
 * and the region is logical blocks [Y−X, Y); a destination is any slot of
 * the region not holding a retained token (slots past n in the last block
 * included); the k-th source in position order goes to the k-th
 * destination in position order; logical slots are translated to physical
 * ones through the block table.
 *   keepmask [⌈n/32⌉] (bit p%32 of word p/32: token p retained)
 *   src, dst [≤ m] physical slots;  *n_pairs
 *   *X;  freed [Y] the physical blocks given back, in logical order; *n_freed
 *   new_table [X] the region's physical blocks;  tail_mask [⌈X·BS/32⌉]
 *   (bit i: slot i of the region holds a retained token afterwards) */
int orc_tail_plan(const uint32_t *keepmask, int n, const int32_t *block_table, int BS,
                  int32_t *src, int32_t *dst, int *n_pairs, int *X, int32_t *freed,
                  int *n_freed, int32_t *new_table, uint32_t *tail_mask) {
  if (!keepmask || !block_table || !src || !dst || !n_pairs || !X || !freed || !n_freed ||
      !new_table || !tail_mask || BS < 1 || n < 0)
    return 1;
  const int Y = (n + BS - 1) / BS;
  int m = 0;
  for (int p = 0; p < n; p++) m += (keepmask[p / 32] >> (p % 32)) & 1u;
  const int x = (m + BS - 1) / BS;
  const int start = (Y - x) * BS;
  *X = x;
  /* sources: retained tokens before the region, in position order */
  int ns = 0;
  for (int p = 0; p < start; p++)
    if ((keepmask[p / 32] >> (p % 32)) & 1u) src[ns++] = p;
  /* destinations: region slots not holding a retained token, in order */
  int nd = 0;
  for (int p = start; p < Y * BS && nd < ns; p++) {
    const int kept = p < n && ((keepmask[p / 32] >> (p % 32)) & 1u);
    if (!kept) dst[nd++] = p;
  }
  if (nd != ns) return 5; /* cannot happen: the region has ≥ m − (kept inside) holes */
  for (int i = 0; i < (x * BS + 31) / 32; i++) tail_mask[i] = 0u;
  for (int p = start; p < Y * BS; p++)
    if (p < n && ((keepmask[p / 32] >> (p % 32)) & 1u))
      tail_mask[(p - start) / 32] |= 1u << ((p - start) % 32);
  for (int k = 0; k < ns; k++) {
    const int t = dst[k] - start;
    tail_mask[t / 32] |= 1u << (t % 32);
    src[k] = block_table[src[k] / BS] * BS + src[k] % BS;
    dst[k] = block_table[dst[k] / BS] * BS + dst[k] % BS;
  }
  *n_pairs = ns;
  for (int b = 0; b < Y - x; b++) freed[b] = block_table[b];
  *n_freed = Y - x;
  for (int b = 0; b < x; b++) new_table[b] = block_table[Y - x + b];
  return 0;
}

/* ---------------------------------------------------- LRFU keep score */

struct orc_mass_item {
  double m;
  int i;
};

static int orc_mass_desc(const void *a, const void *b) {
  const struct orc_mass_item *x = (const struct orc_mass_item *)a;
  const struct orc_mass_item *y = (const struct orc_mass_item *)b;
  if (x->m > y->m) return -1;
  if (x->m < y->m) return 1;
  return (x->i > y->i) - (x->i < y->i);
}

/* [ActKV] §5.2 (attention-aware LRFU, Algorithm 1): after an action region
 * each entry's keep score decays by λ and gains the entry's action-region
 * attention score when the entry is a hit, a hit being membership of the
 * top-p set of that region's scores (p = 90% on the page).
 * Readings (the update's equation is lost on the page):
 *   KS_t = λ·KS_{t−1} + hit_t·s_t — recency only at λ = 0, an undecayed sum
 *   (frequency) at λ = 1, the two limits the page describes;
 *   the top-p set is the shortest prefix of the entries ordered by score
 *   (descending, lower index first among equal scores) whose score mass
 *   reaches p·Σ s; an entry whose score is not a positive finite number
 *   (≤ 0, NaN, ±∞) has no mass and is never a hit.
 * KS is computed in fp64 from the fp32 inputs and rounded once to fp32.
 *   scores [n];  ks [n] in/out;  hits [n] out (0/1) */
int orc_lrfu_update(const float *scores, int n, double p, double lambda, float *ks,
                    uint8_t *hits) {
  if (!scores || !ks || !hits || n < 0 || !(p >= 0.0 && p <= 1.0) ||
      !(lambda >= 0.0 && lambda <= 1.0))
    return 1;
  struct orc_mass_item *it =
      (struct orc_mass_item *)malloc(sizeof(struct orc_mass_item) * (size_t)(n > 0 ? n : 1));
  if (!it) return 3;
  double total = 0.0;
  for (int i = 0; i < n; i++) {
    const double s = (double)scores[i];
    it[i].m = (s > 0.0 && isfinite(s)) ? s : 0.0; /* NaN compares false: no mass */
    it[i].i = i;
    total += it[i].m;
    hits[i] = 0;
  }
  qsort(it, (size_t)n, sizeof(struct orc_mass_item), orc_mass_desc);
  const double target = p * total;
  double cum = 0.0;
  for (int k = 0; k < n && cum < target && it[k].m > 0.0; k++) {
    hits[it[k].i] = 1;
    cum += it[k].m;
  }
  for (int i = 0; i < n; i++) {
    const double s = (double)scores[i];
    ks[i] = (float)(lambda * (double)ks[i] + (hits[i] ? s : 0.0));
  }
  free(it);
  return 0;
}

/* ------------------------------------------------- confidence monitor */

static int orc_f64_desc(const void *a, const void *b) {
  const double x = *(const double *)a, y = *(const double *)b;
  return (x < y) - (x > y);
}

static int orc_f64_asc(const void *a, const void *b) {
  const double x = *(const double *)a, y = *(const double *)b;
  return (x > y) - (x < y);
}

/* [ActKV] §6.1 "Token-level confidence": the negative average
 * log-probability of the k most probable tokens of the predicted
 * distribution P = softmax(logits):
 *   C = −(1/k) Σ_{j ≤ k} log P(j) = LSE − (1/k) Σ_{j ≤ k} logit(j),
 * with LSE = log Σ_v exp(logit_v).  fp64 throughout.
 *   logits [V] (fp32);  *conf out */
int orc_token_confidence(const float *logits, int V, int k, double *conf) {
  if (!logits || !conf || V < 1 || k < 1 || k > V) return 1;
  double mx = -INFINITY;
  for (int v = 0; v < V; v++)
    if ((double)logits[v] > mx) mx = (double)logits[v];
  double sum = 0.0;
  for (int v = 0; v < V; v++) sum += exp((double)logits[v] - mx);
  const double lse = mx + log(sum);
  double *sorted = (double *)malloc(sizeof(double) * (size_t)V);
  if (!sorted) return 3;
  for (int v = 0; v < V; v++) sorted[v] = (double)logits[v];
  qsort(sorted, (size_t)V, sizeof(double), orc_f64_desc);
  double top = 0.0;
  for (int j = 0; j < k; j++) top += sorted[j] - lse; /* log P(j) */
  *conf = -top / (double)k;
  free(sorted);
  return 0;
}

/* [ActKV] §6.1 "Trace-level confidence" and "Trend detection".
 *   R'_m = min{C_i : m·s ≤ i < m·s + w}, m = 0 … ⌊(L − w)/s⌋ (windows of w
 *          tokens, stride s; no window if L < w);
 *   Q_b  = the b-th percentile of R' (linear interpolation between the
 *          order statistics at rank (b/100)·(n − 1), the common definition);
 *   R    = the entries of R' with value ≤ Q_b, kept at their window index m;
 *   slope = the least-squares slope of R against m (0 if R has fewer than
 *          two distinct window indices).
 * Readings: the percentile's interpolation and the time axis of the fit are
 * not given on the page; these are the plainest choices.
 *   conf [L];  *slope, *n_windows, *n_kept out */
int orc_conf_trend(const double *conf, int L, int w, int s, double b, double *slope,
                   int *n_windows, int *n_kept) {
  if (!conf || !slope || !n_windows || !n_kept || L < 0 || w < 1 || s < 1 ||
      !(b >= 0.0 && b <= 100.0))
    return 1;
  *slope = 0.0;
  *n_windows = 0;
  *n_kept = 0;
  if (L < w) return 0;
  const int n = (L - w) / s + 1;
  double *rp = (double *)malloc(sizeof(double) * (size_t)n);
  double *srt = (double *)malloc(sizeof(double) * (size_t)n);
  if (!rp || !srt) {
    free(rp);
    free(srt);
    return 3;
  }
  for (int m = 0; m < n; m++) {
    double mn = INFINITY;
    for (int i = m * s; i < m * s + w; i++)
      if (conf[i] < mn) mn = conf[i];
    rp[m] = mn;
    srt[m] = mn;
  }
  qsort(srt, (size_t)n, sizeof(double), orc_f64_asc);
  const double pos = b / 100.0 * (double)(n - 1);
  const int lo = (int)floor(pos);
  const int hi = lo + 1 < n ? lo + 1 : lo;
  const double q = srt[lo] + (pos - (double)lo) * (srt[hi] - srt[lo]);
  double sx = 0.0, sy = 0.0, sxx = 0.0, sxy = 0.0;
  int cnt = 0;
  for (int m = 0; m < n; m++)
    if (rp[m] <= q) {
      sx += m;
      sy += rp[m];
      sxx += (double)m * m;
      sxy += (double)m * rp[m];
      cnt++;
    }
  const double den = cnt * sxx - sx * sx;
  *slope = (cnt >= 2 && den > 0.0) ? (cnt * sxy - sx * sy) / den : 0.0;
  *n_windows = n;
  *n_kept = cnt;
  free(rp);
  free(srt);
  return 0;
}

/* [ActKV] §6.2, Algorithm 2 (confidence-driven adaptive budget): start
 * small; when the confidence trend is falling (slope < 0) raise the
 * budget; when it is flat or recovering keep it — it is never lowered.
 * Reading: the page gives no increment; the budget grows by `step`, capped
 * at `max_budget`. */
int orc_adapt_budget(double slope, int budget, int step, int max_budget) {
  if (slope < 0.0) {
    const int nb = budget + step;
    return nb < max_budget ? nb : (budget > max_budget ? budget : max_budget);
  }
  return budget;
}
