/*
 * kvc.h — C ABI of the query-conditioned KV compression event (sm_103a).
 *
 * One compression event runs once per agent step, after prefill and before
 * decode (KVMem: Virtualizing Million-Token Agent Workspaces on a Consumer
 * GPU, "Step-level scheduling").  It follows the three primitives of
 * ActKV: Efficient LLM Agents through Action-Guided KV Cache Management,
 * §3.3 ("unified workflow": attention calculation → entry eviction with a
 * Boolean keep mask → cache compaction):
 *
 *   score   kvc_score        Mean-K block scoring (KVMem, "Query-conditioned
 *                            retrieval"), or
 *           kvc_score_qmem   QueryMemory rule score (IntentKV: Cross-Turn
 *                            Intent-Aware KV Cache Pruning for Agent
 *                            Inference, §4 "Rule score")
 *   select  kvc_select       budgeted top-k with a forced set, chronological
 *                            output + keep mask (IntentKV §4 "Top-k
 *                            selection"; KVMem "Query-conditioned retrieval")
 *   layout  kvc_pack_rerope  execution view: gather + re-RoPE K, copy V
 *                            (KVMem, "Tiered movement"), or
 *           kvc_redirect_free slot-map redirection to a dead slot with
 *                            alias/refcount-aware freeing (IntentKV §4
 *                            "Redirect", §4 check 6, §7)
 *
 * Conventions (all entry points):
 *  - Every pointer named "device" is CUDA device memory owned by the caller.
 *    The library never allocates or frees memory and keeps no state between
 *    calls.  Scratch space ("ws") is passed in; its size comes from the
 *    matching *_workspace_size() query.
 *  - bf16 tensors are passed as kvc_bf16 (the raw 16-bit bf16 bit pattern).
 *  - All work is enqueued asynchronously on `stream`.  The return value
 *    reports host-side validation only; it is returned before any launch.
 *    Errors found on the device (an out-of-range index, a NaN score) are
 *    recorded in the caller's `dev_status` word (first error wins, written
 *    with an atomic compare-and-swap; a NULL dev_status disables the record
 *    but not the bounds checks: a bad index is skipped, never dereferenced).
 *    Read it with kvc_device_status() after the stream has been synchronised.
 *    No kernel traps, asserts or spins without a bound.
 *  - Sizes are element counts unless a name ends in _bytes.  Layouts are
 *    row-major with the last dimension contiguous.
 *  - KV blocks are KVC_BLOCK_TOKENS = 32 tokens (KVMem's default block
 *    size).  Histories are multiples of 32 tokens; head_dim D ∈ {64, 128}.
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVC_BLOCK_TOKENS 32
/* bf16 of -1e4 rounded to nearest even = -9984.0 (bit pattern 0xC61C):
 * the dead-slot key (IntentKV §2 "Layout": K set to -10^4, V set to 0). */
#define KVC_SENTINEL_K_BITS 0xC61Cu
/* Longest segment kvc_select stages in shared memory; a launch whose
 * max_seg_len is larger reads the scores from global memory on every pass
 * instead (same result, one CTA per segment either way). */
#define KVC_SELECT_STAGED_SEG 49152
/* Longest segment kvc_select accepts (KVMem's 10M-token workspace is 312,500
 * blocks per layer and KV head; token-level sessions run longer). */
#define KVC_SELECT_MAX_SEG (1 << 30)
/* Longest segment kvc_lrfu_update accepts (its keys are staged in shared
 * memory). */
#define KVC_LRFU_MAX_SEG 49152
/* Widest query-row set (W * G) kvc_score accepts for one KV head. */
#define KVC_SCORE_MAX_ROWS 256

typedef uint16_t kvc_bf16;

typedef enum {
  KVC_OK = 0,
  KVC_ERR_INVALID_ARG = 1, /* NULL pointer, negative or zero size            */
  KVC_ERR_SHAPE = 2,       /* unsupported D, history not a multiple of 32 …  */
  KVC_ERR_BUDGET = 3,      /* budget < 1 or sink + recent > budget           */
  KVC_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned               */
  KVC_ERR_WORKSPACE = 5,   /* ws_bytes smaller than the size query returned  */
  KVC_ERR_CUDA = 6,        /* a CUDA launch or query failed                  */
  KVC_ERR_BOUNDS = 7,      /* device: an index or offset was out of range    */
  KVC_ERR_NAN = 8,         /* device: a NaN score reached kvc_select         */
  KVC_ERR_TIMEOUT = 9,     /* device: a bounded wait gave up                 */
  KVC_ERR_CAPACITY = 10,   /* device: the freed-slot list overflowed; host:
                              more blocks needed at once than repository slots */
  KVC_ERR_IO = 11,         /* host: the repository's backing file failed     */
  KVC_ERR_NOMEM = 12       /* host: the repository's tables or scratch could
                              not be allocated (nothing changed)             */
} kvc_status;

/* Kernel choice for the entry points that have more than one kernel for the
 * same arithmetic (a diagnostic of this library, no counterpart on the
 * pages).  The plain entry points (kvc_score, kvc_score_qmem,
 * kvc_recover_score) choose by shape and device, which is KVC_KERNEL_AUTO;
 * their _ex variants take the choice as an argument so that a test or a
 * profile can run one particular kernel.  A kernel that does not cover the
 * call's sizes is refused with KVC_ERR_SHAPE before any launch; a value that
 * does not belong to the entry point is KVC_ERR_INVALID_ARG.  Every kernel of
 * one entry point computes the same quantity within the accuracy that entry
 * point states. */
typedef enum {
  KVC_KERNEL_AUTO = 0,
  /* kvc_score_ex (Mean-K scoring) */
  KVC_KERNEL_SCORE_FUSED = 1,   /* tcgen05, Mean-K read once; G = 4, W = 32, D = 128 */
  KVC_KERNEL_SCORE_RING = 2,    /* tcgen05, two passes in a CTA-cluster ring          */
  KVC_KERNEL_SCORE_PERSIST = 3, /* tcgen05, persistent grid, L2 exchange              */
  KVC_KERNEL_SCORE_SPLIT = 4,   /* tcgen05, two launches                              */
  KVC_KERNEL_SCORE_CC = 5,      /* CUDA cores, two launches; any shape                */
  KVC_KERNEL_SCORE_GROUP = 6,   /* tcgen05, two passes, CTA groups exchanging through
                                   L2; 129–192 query rows, D = 128                   */
  /* kvc_score_qmem_ex (rule score) */
  KVC_KERNEL_QMEM_TC = 16,      /* tcgen05 logits (8 KV heads, G ∈ {2, 4}), rule
                                   phase in the same kernel from L2                  */
  KVC_KERNEL_QMEM_CC = 17,      /* CUDA-core logits; any shape                        */
  KVC_KERNEL_QMEM_TC_SPILL = 18, /* tcgen05 logits (8 KV heads, G ∈ {2, 4, 8})
                                    spilled to the workspace, rule phase in a
                                    second kernel                                 */
  /* kvc_recover_score_ex (LSE-recovery score) */
  KVC_KERNEL_RECOVER_TC = 32,   /* tcgen05 page tiles (H 8, block 16, G ∈ {2, 4, 8})  */
  KVC_KERNEL_RECOVER_CC = 33    /* CUDA cores; any shape                              */
} kvc_kernel;

/* Static, never-NULL description of a status code. */
const char *kvc_status_string(kvc_status s);

/* Copies *dev_status (device int32) to *host_out, synchronously (this call
 * blocks until all prior work on the device is done).  Returns KVC_ERR_CUDA
 * if the copy fails. */
kvc_status kvc_device_status(const int32_t *dev_status, int32_t *host_out);

/* Library version, "major.minor.patch". */
const char *kvc_version(void);

/* Self-test of the bounded waits (a diagnostic of this library; no
 * counterpart on the pages).  Launches one CTA whose first thread waits on a
 * shared-memory mbarrier that nothing arrives on.  The wait is the same
 * bounded wait the tensor-core kernels use: it polls against %globaltimer and
 * gives up after one second.  The kernel then records KVC_ERR_TIMEOUT in
 * *dev_status and returns.  The launch takes about a second; no fault or trap
 * is raised, and the context stays usable.
 * Errors: KVC_ERR_INVALID_ARG (dev_status NULL), KVC_ERR_CUDA (launch). */
kvc_status kvc_selftest_bounded_wait(int32_t *dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Index maintenance (not part of the timed event).
 *
 * kvc_build_meank — KVMem, "Query-conditioned retrieval": one RoPE-stripped
 * mean key per (layer, KV head, 32-token block).
 *   kraw   device bf16 [L][H][n_tok][D]   raw (pre-RoPE) keys
 *   meank  device bf16 [L][H][n_tok/32][D] out: block means
 * Each output element is the exact mean of the 32 inputs rounded once to
 * bf16 (round-to-nearest-even).  The kernel sums in fp32 with Knuth's
 * TwoSum, which keeps every rounding error of the running sum, so the sum is
 * exact while a guard holds over each thread's 8 columns: all inputs zero,
 * or 32·max|x| in [2^-60, 2^100) with min|x| > 2^-29·max|x| (no zero,
 * subnormal, NaN or infinity next to normal values).  Columns outside the
 * guard are summed in fp64 in token order, which is exact whenever their
 * magnitudes span less than about 2^40 (NaN gives the quiet NaN 0x7FC0).
 * Errors: KVC_ERR_INVALID_ARG (NULL, sizes < 1), KVC_ERR_SHAPE (n_tok % 32,
 * D ∉ {64,128}), KVC_ERR_ALIGN (pointers not 16-byte aligned).
 * ---------------------------------------------------------------------- */
kvc_status kvc_build_meank(const kvc_bf16 *kraw, kvc_bf16 *meank, int32_t L,
                           int32_t H, int32_t D, int64_t n_tok,
                           int32_t *dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 1 (score), Mean-K mode.
 * KVMem, "Query-conditioned retrieval" (score blocks in the model's own
 * attention space against RoPE-stripped Mean-K), with the GQA aggregation of
 * ActKV §7.1 (Algorithm 3: max over the query heads of a group, mean over
 * the query tokens):
 *   z[w,g,b]   = q[l, h*G+g, w] · meank[l,h,b] / sqrt(D)
 *   LSE[w,g]   = log Σ_b exp z[w,g,b]          (over the session's blocks)
 *   score[l,h,b] = (1/W) Σ_w max_g exp(z[w,g,b] − LSE[w,g])
 *   q        device bf16 [L][n_sess][Hq][W][D]  pre-RoPE query window
 *   meank    device bf16 [L][H][nb_total][D]
 *   blk_off  device int64 [n_sess+1]  session r owns blocks
 *            [blk_off[r], blk_off[r+1]) of every (l, h) row; blk_off[0] = 0,
 *            blk_off[n_sess] = nb_total, each session non-empty and at most
 *            nb_max blocks (violations: KVC_ERR_BOUNDS in dev_status, the
 *            session is skipped)
 *   scores   device fp32 [L][H][nb_total]  out
 *   ws       device scratch of kvc_score_workspace_size() bytes
 * G = Hq/H; W*G ≤ KVC_SCORE_MAX_ROWS.
 * Accuracy: products accumulate in fp32 and exponentials are taken in base 2
 * in fp32; each score lies within 1e-3 relative of the exact value for the
 * same bf16 inputs.  Repeating a call, or scoring some layers in a call of
 * their own, gives bit-identical scores.
 * Errors: KVC_ERR_INVALID_ARG, KVC_ERR_SHAPE (Hq % H, D, W*G too wide),
 * KVC_ERR_ALIGN, KVC_ERR_WORKSPACE.
 * ---------------------------------------------------------------------- */
size_t kvc_score_workspace_size(int32_t L, int32_t H, int32_t Hq, int32_t W,
                                int32_t n_sess, int32_t nb_max, int64_t nb_total);
kvc_status kvc_score(const kvc_bf16 *q, const kvc_bf16 *meank, float *scores,
                     int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t W,
                     const int64_t *blk_off, int32_t n_sess, int64_t nb_total,
                     int32_t nb_max, void *ws, size_t ws_bytes,
                     int32_t *dev_status, cudaStream_t stream);
/* kvc_score with the kernel named by `kernel` (KVC_KERNEL_AUTO or one of
 * KVC_KERNEL_SCORE_*; see kvc_kernel).  Same arguments, result and errors. */
kvc_status kvc_score_ex(const kvc_bf16 *q, const kvc_bf16 *meank, float *scores,
                        int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t W,
                        const int64_t *blk_off, int32_t n_sess, int64_t nb_total,
                        int32_t nb_max, void *ws, size_t ws_bytes,
                        int32_t *dev_status, kvc_kernel kernel, cudaStream_t stream);

/* kvc_score for callers that cannot allocate device memory (no counterpart
 * on the pages; this is a convenience of the library).  Some hosts cannot
 * pass a workspace: a serving runtime that carves all of HBM into its own
 * pool at start-up and forbids device allocations afterwards, or a plugin
 * inside such a runtime that receives tensors but no allocator.  This call
 * takes the same inputs and outputs as kvc_score and computes the same
 * scores, but its scratch is a fixed array of KVC_SCORE_STATIC_SCRATCH_BYTES
 * compiled into the library (held by every GPU that loads the library until
 * the process exits); it calls no cudaMalloc/cudaFree.
 *  - Sizes whose scratch (kvc_score_workspace_size) exceeds the array are
 *    rejected with KVC_ERR_WORKSPACE before anything is launched; the 8B-
 *    class 128K-token event (36 layers, 8/32 heads, W 32) needs about 5 MB.
 *  - kvc_score's own argument, shape and alignment errors are reported
 *    first, exactly as kvc_score reports them.
 *  - The first call on a device looks up the array's device address (once
 *    per device, with that device current) and keeps it; make that first
 *    call before any stream capture on the device.  The kept address belongs
 *    to the context current at that call: a call under another context of
 *    the device (one the caller created and made current) repeats the
 *    look-up, so make such a call before capture too.  Do not call this
 *    entry point again after a cudaDeviceReset in the same process: the
 *    reset unloads the array, and the library does not track resets.
 *  - Every call shares the one array per device: calls whose kernels overlap
 *    on the GPU (different streams, no ordering between them) race and give
 *    undefined scores.  Serialise them (one stream, or events).
 * Errors: those of kvc_score, plus KVC_ERR_WORKSPACE as above and
 * KVC_ERR_CUDA if the device address cannot be obtained. */
#define KVC_SCORE_STATIC_SCRATCH_BYTES (8u << 20)
/* KVC_SCORE_STATIC_SCRATCH_BYTES as compiled into this library (bindings
 * read the limit from here rather than repeat the constant). */
size_t kvc_score_static_scratch_bytes(void);
kvc_status kvc_score_static(const kvc_bf16 *q, const kvc_bf16 *meank, float *scores,
                            int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t W,
                            const int64_t *blk_off, int32_t n_sess, int64_t nb_total,
                            int32_t nb_max, int32_t *dev_status, cudaStream_t stream);

/* Number of kernels one kvc_score call with these sizes launches on this
 * device (1: tensor-core scorer with a thread-block-cluster LSE exchange;
 * 2: two-launch scoring), 0 for invalid sizes.  Host-only query. */
int32_t kvc_score_launches(int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t W,
                           int32_t n_sess, int32_t nb_max);

/* ------------------------------------------------------------------------
 * QueryMemory update (IntentKV §4 "Memory recurrence", §7 item 1):
 *   M ← decay·M + gain·mean_t q_turn[t];  then, if renorm, M ← M/‖M‖₂ along D
 *   (a zero vector stays zero).
 *   M       device fp32 [n_sess][L][Hq][D]  in/out (start from zeros)
 *   q_turn  device bf16 [n_sess][L][Hq][T][D]  the turn's pre-RoPE queries
 * Errors: KVC_ERR_INVALID_ARG, KVC_ERR_SHAPE (D), KVC_ERR_ALIGN.
 * ---------------------------------------------------------------------- */
kvc_status kvc_qmem_update(float *M, const kvc_bf16 *q_turn, int32_t n_sess,
                           int32_t L, int32_t Hq, int32_t D, int32_t T,
                           float decay, float gain, int32_t renorm,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 1 (score), QueryMemory mode (IntentKV §4 "Rule score", §4 check 1:
 * GQA KV heads expanded to the Hq query heads):
 *   z[l,hq,j]  = M[r,l,hq] · kpool[l, slot_map[r,j], hq/G] / sqrt(D)
 *   rule[r,j]  = Σ_{l,hq} exp(z[l,hq,j] − LSE[l,hq]),  LSE over the live j
 * A position whose slot is `sentinel` (redirected by an earlier event) is
 * dead: it is left out of every softmax and gets rule = -1, below any live
 * score.
 *   M        device fp32 [n_sess][L][Hq][D]
 *   kpool    device bf16 [L][n_slots][H][D]   paged K pool, one row per slot
 *   slot_map device int32 [n_sess][N]         logical position → slot
 *   rule     device fp32 [n_sess][N]          out
 *   ws       device scratch of kvc_score_qmem_workspace_size() bytes
 * A slot outside [0, n_slots) is recorded as KVC_ERR_BOUNDS and treated as
 * dead.  Shapes: D ∈ {64, 128}; H divides 32; Hq a multiple of H with
 * G = Hq/H ≤ 8.  Errors: KVC_ERR_INVALID_ARG, KVC_ERR_SHAPE, KVC_ERR_ALIGN,
 * KVC_ERR_WORKSPACE.
 * ---------------------------------------------------------------------- */
size_t kvc_score_qmem_workspace_size(int32_t n_sess, int32_t L, int32_t Hq,
                                     int32_t N);
kvc_status kvc_score_qmem(const float *M, const kvc_bf16 *kpool,
                          const int32_t *slot_map, int32_t sentinel,
                          float *rule, int32_t n_sess, int32_t L, int32_t H,
                          int32_t Hq, int32_t D, int32_t N, int64_t n_slots,
                          void *ws, size_t ws_bytes, int32_t *dev_status,
                          cudaStream_t stream);
/* kvc_score_qmem with the logits kernel named by `kernel` (KVC_KERNEL_AUTO,
 * KVC_KERNEL_QMEM_TC, KVC_KERNEL_QMEM_TC_SPILL or KVC_KERNEL_QMEM_CC).  AUTO
 * takes QMEM_TC where it applies, then QMEM_TC_SPILL, then QMEM_CC. */
kvc_status kvc_score_qmem_ex(const float *M, const kvc_bf16 *kpool,
                             const int32_t *slot_map, int32_t sentinel,
                             float *rule, int32_t n_sess, int32_t L, int32_t H,
                             int32_t Hq, int32_t D, int32_t N, int64_t n_slots,
                             void *ws, size_t ws_bytes, int32_t *dev_status,
                             kvc_kernel kernel, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 2 (select): budgeted top-k with a forced set (IntentKV §4 "Top-k
 * selection": K* = F ∪ argtop_{C*} s), sink and recent always kept and the
 * result restored in chronological order (KVMem, "Query-conditioned
 * retrieval"), plus the Boolean keep mask (ActKV §3.3).
 * Per segment s of length n = seg_off[s+1] − seg_off[s]:
 *   F = {0 … n_sink−1} ∪ {n−n_recent … n−1}  (clipped to the segment)
 *   if n ≤ budget: keep all n; otherwise keep F plus the budget − |F|
 *   non-forced items ranked by (score descending, index ascending);
 *   −0.0 ranks equal to +0.0.
 *   scores     device fp32, segment s at [seg_off[s], seg_off[s+1])
 *   seg_off    device int64 [n_seg+1], non-decreasing, each n ≤ max_seg_len
 *   kept       device int32 [n_seg][budget] out: ascending segment-local
 *              indices; entries past kept_count[s] are set to -1
 *   kept_count device int32 [n_seg] out: min(budget, n)
 *   keepmask   device uint32 [n_seg][ceil(max_seg_len/32)] out, may be NULL:
 *              bit (i%32) of word i/32 is 1 iff item i is kept; bits at or
 *              past n are 0
 * A NaN score is recorded as KVC_ERR_NAN and ranks below every number.
 * Launches with max_seg_len ≤ KVC_SELECT_STAGED_SEG stage each segment's
 * keys in shared memory; longer ones read them from global memory on each of
 * the search's passes (the result is the same).
 * Errors: KVC_ERR_INVALID_ARG, KVC_ERR_BUDGET (budget < 1, n_sink < 0,
 * n_recent < 0, n_sink + n_recent > budget), KVC_ERR_SHAPE (max_seg_len >
 * KVC_SELECT_MAX_SEG), KVC_ERR_ALIGN.
 * ---------------------------------------------------------------------- */
kvc_status kvc_select(const float *scores, const int64_t *seg_off,
                      int32_t n_seg, int32_t max_seg_len, int32_t budget,
                      int32_t n_sink, int32_t n_recent, int32_t *kept,
                      int32_t *kept_count, uint32_t *keepmask,
                      int32_t *dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * RoPE table for the execution view (NeoX rotate-half convention):
 *   tab[i][j] = (cos a, sin a),  a = (pos0 + i) · theta^(−2j/D),  j < D/2
 * computed in fp64 and rounded to fp32.
 *   tab  device fp32 [n_pos][D/2][2]
 * Errors: KVC_ERR_INVALID_ARG, KVC_ERR_SHAPE (D), KVC_ERR_ALIGN.
 * ---------------------------------------------------------------------- */
kvc_status kvc_rope_table(float *tab, int32_t n_pos, int32_t pos0, int32_t D,
                          double theta, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 3a (layout): execution-view pack (KVMem, "Tiered movement": selected
 * blocks packed into contiguous logical positions, raw K re-RoPEd at the
 * new positions, V copied as-is).  For view token i of segment (l,h,r)
 * with i < 32·kept_count:
 *   src         = tok_off[r] + 32·kept[(l,h,r)][i/32] + i%32
 *   kview[i]    = RoPE(kraw[l,h,src], position of table row i)
 *   vview[i]    = vraw[l,h,src]   (bit copy)
 * View tokens at or past 32·kept_count are written as zeros.
 *   kraw, vraw  device bf16 [L][H][n_tok][D]   (pre-RoPE K, V)
 *   kept, kept_count  as written by kvc_select over segments ordered
 *               (l, h, r) with r fastest: [L][H][n_sess][budget], [L][H][n_sess]
 *   tok_off     device int64 [n_sess+1], multiples of 32, tok_off[n_sess] = n_tok
 *   rope_tab    device fp32 [32·budget][D/2][2] from kvc_rope_table
 *   kview, vview device bf16 [L][H][n_sess][32·budget][D] out
 * RoPE pairs element j with j + D/2:
 *   (x_j, x_{j+D/2}) → (x_j·c − x_{j+D/2}·s, x_{j+D/2}·c + x_j·s),
 * computed in fp32 and rounded to bf16 (nearest even).
 * A kept index outside the session's blocks is recorded as KVC_ERR_BOUNDS;
 * its view block is zero-filled.
 * Errors: KVC_ERR_INVALID_ARG, KVC_ERR_SHAPE, KVC_ERR_BUDGET, KVC_ERR_ALIGN.
 * ---------------------------------------------------------------------- */
kvc_status kvc_pack_rerope(const kvc_bf16 *kraw, const kvc_bf16 *vraw,
                           const int32_t *kept, const int32_t *kept_count,
                           int32_t L, int32_t H, int32_t D,
                           const int64_t *tok_off, int32_t n_sess,
                           int64_t n_tok, int32_t budget,
                           const float *rope_tab, kvc_bf16 *kview,
                           kvc_bf16 *vview, int32_t *dev_status,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 3a, tiered (KVMem, "Tiered movement": the raw history lives in host
 * memory, the GPU holds only the execution view; missed blocks are brought
 * in and re-RoPEd, and blocks shared by consecutive steps stay on the GPU).
 * Same output as kvc_pack_rerope for the same kept lists (bit for bit), but
 * the source of each kept block's raw K and V is
 *   - the previous step's view, when the block is also in the previous kept
 *     list of its (l, h, r): raw K from kcache_prev, V from vview_prev
 *     (device memory);
 *   - otherwise kraw_host / vraw_host, read by the kernel directly from
 *     host memory (which must be pinned and device-accessible, e.g.
 *     cudaHostAlloc, so that the same address works on the device; on
 *     GB300 the reads go over NVLink-C2C).
 * The kernel also writes this step's raw-K cache (kcache[i] = the raw K of
 * view block i) for the next step.  Callers alternate two sets of
 * (kcache, vview) buffers between steps; the outputs must not overlap the
 * previous step's buffers.
 *   kraw_host, vraw_host  host bf16 [L][H][n_tok][D], page-locked and mapped
 *                 (cudaHostAlloc / cudaHostRegister); the call translates them
 *                 with cudaHostGetDevicePointer and returns
 *                 KVC_ERR_INVALID_ARG for memory that is not
 *   kept_prev, kept_count_prev  the previous step's kvc_select output, or
 *                 NULL (first step: every block is a miss)
 *   kcache_prev, vview_prev, kcache, kview, vview
 *                 device bf16 [L][H][n_sess][32·budget][D]
 *   n_hits        device int32 [1], may be NULL: incremented once per
 *                 (view block, l, h) found in the previous view
 * Other arguments as kvc_pack_rerope.
 * Errors: those of kvc_pack_rerope; KVC_ERR_INVALID_ARG if kept_prev is
 * given without kept_count_prev, kcache_prev or vview_prev.
 * ---------------------------------------------------------------------- */
kvc_status kvc_pack_tiered(const kvc_bf16 *kraw_host, const kvc_bf16 *vraw_host,
                           const int32_t *kept_prev, const int32_t *kept_count_prev,
                           const kvc_bf16 *kcache_prev, const kvc_bf16 *vview_prev,
                           const int32_t *kept, const int32_t *kept_count, int32_t L,
                           int32_t H, int32_t D, const int64_t *tok_off, int32_t n_sess,
                           int64_t n_tok, int32_t budget, const float *rope_tab,
                           kvc_bf16 *kcache, kvc_bf16 *kview, kvc_bf16 *vview, int32_t *n_hits,
                           int32_t *dev_status, cudaStream_t stream);

/* kvc_pack_tiered with only some of the history in host memory (the
 * repository view below holds the rest in its backing file).  The unit
 * (l, h, g) — layer, KV head and block g of the history (tokens 32g …
 * 32g + 31, counted over all sessions) — sits in host slot
 * s = host_slot[(l·H + h)·(n_tok/32) + g]; its raw K rows are at
 *   kslots_host + s·slot_elems + t·D   (t < 32),
 * its V rows likewise from vslots_host.  Only misses read host memory; a
 * missed unit whose slot is outside [0, n_slots) is recorded as
 * KVC_ERR_BOUNDS and packed as zeros.
 *   kslots_host, vslots_host  host bf16, page-locked and mapped (as for
 *                 kvc_pack_tiered), slot_elems ≥ 32·D apart
 *   host_slot     device int32 [L][H][n_tok / 32]
 * Other arguments, outputs and errors as kvc_pack_tiered, plus
 * KVC_ERR_INVALID_ARG for a NULL host_slot, n_slots < 1 or slot_elems too
 * small, and KVC_ERR_ALIGN when slot_elems·2 is not a multiple of 16. */
kvc_status kvc_pack_tiered_slots(const kvc_bf16 *kslots_host, const kvc_bf16 *vslots_host,
                                 int64_t slot_elems, int32_t n_slots, const int32_t *host_slot,
                                 const int32_t *kept_prev, const int32_t *kept_count_prev,
                                 const kvc_bf16 *kcache_prev, const kvc_bf16 *vview_prev,
                                 const int32_t *kept, const int32_t *kept_count, int32_t L,
                                 int32_t H, int32_t D, const int64_t *tok_off, int32_t n_sess,
                                 int64_t n_tok, int32_t budget, const float *rope_tab,
                                 kvc_bf16 *kcache, kvc_bf16 *kview, kvc_bf16 *vview,
                                 int32_t *n_hits, int32_t *dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Repository view (KVMem, "Tiered movement": a repository view tracks where
 * each block lives; the execution view holds only the selected blocks;
 * blocks recalled often prefer host RAM over NVMe; misses move in bulk).
 * Host code only: no GPU work, no CUDA call.  Not thread-safe: one thread
 * at a time per repository.
 *
 * The unit of placement is what one (layer, KV head) selects: 32 tokens of
 * raw K and V of one layer and head, one record [2][32][D] bf16 (K rows,
 * then V rows).  Unit u = (l·H + h)·n_blocks + g.  Every unit put is
 * written to the backing file (the NVMe tier) at offset u·record_bytes.
 * Host RAM holds at most n_slots units, in the caller's arena
 * [n_slots][2][32][D] (page-locked and mapped when kvc_pack_tiered_slots
 * reads it: pass kslots_host = arena, vslots_host = arena + 32·D,
 * slot_elems = 2·32·D).  The GPU tier is the previous execution view, which
 * kvc_pack_tiered_slots reuses by itself.
 *
 * Placement: a unit counts one use per step in which its (layer, head) keeps
 * its block for some session.  When a step needs units that are not in host
 * RAM, they take free slots first, then the slots of the units with the
 * fewest uses (ties: the least recently used, then the lowest index) among
 * those the step does not need; units are immutable once put, so an
 * eviction writes nothing.  Units read from the file are grouped into runs of
 * consecutive units (consecutive blocks of one layer and head), one vectored
 * read per run, the runs spread over io_threads threads.
 * ---------------------------------------------------------------------- */
typedef struct kvc_repo kvc_repo;

typedef struct {
  int64_t steps;          /* kvc_repo_step calls                              */
  int64_t needed;         /* units needed from host RAM, summed over steps     */
  int64_t host_hits;      /* of those, already in host RAM                     */
  int64_t fetched;        /* read from the backing file                        */
  int64_t read_calls;     /* vectored reads issued for them                    */
  int64_t bytes_read;
  int64_t evictions;      /* host slots taken from another block               */
  int64_t bytes_written;  /* by kvc_repo_put                                   */
} kvc_repo_stats;

/* flags of kvc_repo_create: read and write the backing file around the
 * operating system's page cache (O_DIRECT), so that reads come from the
 * device; the arena must then be 4096-byte aligned (page-locked allocations
 * are), and file systems without direct I/O refuse the file (KVC_ERR_IO). */
#define KVC_REPO_DIRECT_IO 1

/* Creates (or truncates) the backing file at `path`, sized for L·H·n_blocks
 * records.  arena: host memory for n_slots records, owned by the caller and
 * kept alive until kvc_repo_destroy.  io_threads in [1, 64].  Errors:
 * KVC_ERR_INVALID_ARG, KVC_ERR_SHAPE (D ∉ {64, 128}), KVC_ERR_ALIGN (direct
 * I/O with an arena not 4096-byte aligned), KVC_ERR_IO, KVC_ERR_NOMEM. */
kvc_status kvc_repo_create(const char *path, int64_t n_blocks, int32_t L, int32_t H, int32_t D,
                           int32_t n_slots, kvc_bf16 *arena, int32_t io_threads, int32_t flags,
                           kvc_repo **out);

/* Puts blocks b0 … b0 + nb − 1 of every layer and head, taken from host
 * bf16 [L][H][n_tok][D] arrays (block g = tokens 32g … 32g + 31): each unit
 * is written to the backing file and, while free slots remain, kept in host
 * RAM (slots taken layer-major, then head, then block).  The (layer, head)
 * rows are spread over io_threads threads, each writing up to 64 consecutive
 * records per vectored write.  Putting a unit again overwrites it.  Errors:
 * KVC_ERR_INVALID_ARG (range outside the history or the repository),
 * KVC_ERR_IO (units whose write failed are not marked as put),
 * KVC_ERR_NOMEM. */
kvc_status kvc_repo_put(kvc_repo *repo, int64_t b0, int64_t nb, const kvc_bf16 *kraw,
                        const kvc_bf16 *vraw, int64_t n_tok);

/* The units one step uses and the ones it misses (work in proportion to the
 * kept entries, not to the history), from its kept lists and the previous
 * step's (host int32 copies of kvc_select's outputs for the L
 * packed layers, [L][H][n_sess][budget] and [L][H][n_sess]; kept_prev NULL
 * on the first step): kept index kb of (l, h, r) is unit
 * (l·H + h)·n_blocks + tok_off[r]/32 + kb.  used: every kept unit; need: the
 * kept units whose (l, h, r) did not keep them last step (the reads
 * kvc_pack_tiered_slots makes from host memory).  Both come out sorted and
 * unique; each array holds L·H·n_blocks entries.  Errors:
 * KVC_ERR_INVALID_ARG, KVC_ERR_BOUNDS (a kept index outside its session),
 * KVC_ERR_NOMEM. */
kvc_status kvc_repo_plan(const int32_t *kept, const int32_t *kept_count,
                         const int32_t *kept_prev, const int32_t *kept_count_prev, int32_t L,
                         int32_t H, int32_t n_sess, int32_t budget, const int64_t *tok_off,
                         int64_t n_blocks, int64_t *used, int64_t *n_used, int64_t *need,
                         int64_t *n_need);

/* One step: counts a use of every unit in `used`, brings every unit of
 * `need` into host RAM (reading the missing ones from the backing file) and,
 * if host_slot is not NULL, writes host_slot[u] (host int32 [L·H·n_blocks])
 * = the slot of unit u, or −1.  The slots that changed are also kept for
 * kvc_repo_changes, so that a caller holding the table elsewhere (on the
 * GPU) can update only those entries.  Every unit of `need` must have been
 * put.  Errors: KVC_ERR_INVALID_ARG (an index out of range or never put),
 * KVC_ERR_CAPACITY (more units in `need` than slots; nothing changes),
 * KVC_ERR_IO (the step's evictions stand and its fetched units have no slot,
 * both listed by kvc_repo_changes; host_slot is not written), KVC_ERR_NOMEM
 * (scratch for the step could not be allocated; nothing changes). */
kvc_status kvc_repo_step(kvc_repo *repo, const int64_t *used, int64_t n_used,
                         const int64_t *need, int64_t n_need, int32_t *host_slot);

/* The whole slot table now: host_slot[u] (host int32 [L·H·n_blocks]) = the
 * slot of unit u, or −1 (for a first copy of the table elsewhere). */
kvc_status kvc_repo_slots(const kvc_repo *repo, int32_t *host_slot);

/* The last kvc_repo_step's slot changes: units[i] now has slot slots[i]
 * (−1: evicted).  Writes at most cap entries and returns how many there are
 * (−1 for a bad handle or arguments). */
int64_t kvc_repo_changes(const kvc_repo *repo, int64_t *units, int32_t *slots, int64_t cap);

/* Where unit u lives: 0 not put, 1 host RAM (and the file), 2 the file only;
 * −1 for a bad handle or index. */
int32_t kvc_repo_where(const kvc_repo *repo, int64_t u);

kvc_status kvc_repo_get_stats(const kvc_repo *repo, kvc_repo_stats *out);

/* Closes the backing file (which stays on disk) and frees the repository. */
void kvc_repo_destroy(kvc_repo *repo);

/* ------------------------------------------------------------------------
 * Dead slot (IntentKV §2 "Layout", §4 check 3): writes K = bf16(−1e4) =
 * −9984 (0xC61C) into every element and V = +0.0 into slot `sentinel` of
 * every layer and head.
 *   kpool, vpool  device bf16 [L][n_slots][H][D]; vpool may be NULL
 * Errors: KVC_ERR_INVALID_ARG (sentinel outside [0, n_slots)), KVC_ERR_SHAPE.
 * ---------------------------------------------------------------------- */
kvc_status kvc_init_sentinel(kvc_bf16 *kpool, kvc_bf16 *vpool, int32_t L,
                             int32_t H, int32_t D, int64_t n_slots,
                             int32_t sentinel, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 3b (layout): slot-map redirection and alias-aware free (IntentKV §4
 * "Redirect": S_r[j] ← s† for every dropped j; §4 check 6 and §7 "alias-
 * aware deallocation": a dropped slot u is freed only if j is outside the
 * protected prefix, u ≠ s†, and no remaining reference holds u).
 * Every slot-map entry holds one count in refcnt (the sentinel's count is
 * never touched).  Semantics are those of visiting (r, j) in row-major
 * order: for each position with keep bit 0 and u = slot_map[r,j] ≠ sentinel,
 *   slot_map[r,j] ← sentinel;  refcnt[u] −= 1;
 *   if refcnt[u] reaches 0 and j ≥ prefix_len: append u to `freed`.
 * The freed list is therefore ordered by the (r, j) of each slot's last
 * dropping reference.  Kept positions and the K/V pools are not touched.
 *   slot_map  device int32 [n_sess][N]   in/out
 *   keepmask  device uint32 [n_sess][ceil(N/32)]  from kvc_select
 *   refcnt    device int32 [n_slots]     in/out
 *   freed     device int32 [freed_cap]   out
 *   n_freed   device int32 [1]           out: list length
 *   ws        device scratch of kvc_redirect_free_workspace_size() bytes
 * A slot outside [0, n_slots) or a count that would go below zero is
 * recorded as KVC_ERR_BOUNDS and that position is left as it was; a list
 * longer than freed_cap is recorded as KVC_ERR_CAPACITY (the first
 * freed_cap entries are written).
 * Errors: KVC_ERR_INVALID_ARG, KVC_ERR_SHAPE, KVC_ERR_ALIGN,
 * KVC_ERR_WORKSPACE.
 * ---------------------------------------------------------------------- */
size_t kvc_redirect_free_workspace_size(int32_t n_sess, int32_t N,
                                        int64_t n_slots);
kvc_status kvc_redirect_free(int32_t *slot_map, const uint32_t *keepmask,
                             int32_t n_sess, int32_t N, int32_t *refcnt,
                             int64_t n_slots, int32_t prefix_len,
                             int32_t sentinel, int32_t *freed,
                             int32_t freed_cap, int32_t *n_freed, void *ws,
                             size_t ws_bytes, int32_t *dev_status,
                             cudaStream_t stream);

/* ========================================================================
 * ActKV paged primitives (ActKV: Efficient LLM Agents through Action-Guided
 * KV Cache Management, §3.3 workflow on the paged layout of §2): the same
 * score → keep mask → compaction sequence, for a serving engine whose KV
 * cache lives in pages.  Layout (§2 "Background"): a K pool and a V pool of
 * [L][n_slots][H][D] bf16, one H·D row per (layer, physical slot); request
 * r's logical position p lives in slot block_table[r][p / block_size] ·
 * block_size + p % block_size (the page's worked example: block_size 2,
 * block_table [17, 9], 3 tokens → slots 34, 35, 18).
 * ====================================================================== */

/* Longest request (max_blocks · block_size) kvc_tail_plan accepts. */
#define KVC_TAIL_MAX_TOKENS (1 << 20)

/* ------------------------------------------------------------------------
 * LSE-recovery action score, one decode step (ActKV §7.1, Algorithm 3).
 * The attention backend has already produced, for the current query token
 * of each request, lse[r][l][hq] = ln Σ_p exp(q·k_p/√D) over the keys it
 * attended to; each probability is recovered as exp(q·k/√D − LSE) without
 * materialising the attention matrix.  For request r with count[r] ≥ 1 and
 * every position p < max_blocks·block_size:
 *   x[p] = Σ_l Σ_h max_{g<G} exp(q[r,l,hG+g]·K[l, slot(p), h]/√D − lse[r,l,hG+g])
 *          for p < seqused_k[r] (the keys visible to the query), else 0;
 *   state[r][p] ← x[p]                               if count[r] == 1
 *   state[r][p] ← state + (x[p] − state)/count[r]    otherwise
 * i.e. the running mean over the action tokens of the region (count[r] = the
 * index of this action token, 1 at the region's first token, which restarts
 * the state).  Requests with count[r] < 1 are not generating an action and
 * are left untouched.  A slot holds every layer's KV of one token, so one
 * score per position sums over layers and KV heads.
 *   q            device bf16 [n_req][L][Hq][D]   the current query token
 *   lse          device fp32 [n_req][L][Hq]      natural-log LSE per head
 *   kpool        device bf16 [L][n_slots][H][D]
 *   block_table  device int32 [n_req][max_blocks] physical block ids
 *   seqused_k    device int32 [n_req]  keys visible (≤ max_blocks·block_size)
 *   count        device int32 [n_req]  action-token index (< 1: skip)
 *   state        device fp32 [n_req][max_blocks·block_size]  in/out
 * G = Hq/H.  Arithmetic: fp32 products and sums, exp as 2^(log2 e·(…)) with
 * the hardware ex2, the group maximum taken before the exponential.
 * Shapes with H = 8, block_size = 16, G ∈ {2, 4, 8} run on the tensor cores
 * (one 128-row page tile per MMA, brought in by TMA from the block table);
 * any other shape runs on a CUDA-core kernel (kvc_recover_tensor_core tells
 * which).  ws is optional scratch (NULL, or ws_bytes from
 * kvc_recover_score_workspace_size): when a few requests' pages cannot fill
 * the GPU, the tensor-core path then splits the layers into groups, writes
 * each group's partial sums to ws and adds them in group order in a second
 * kernel (the result is deterministic either way; without ws, or when the
 * size query returns 0, one kernel and no scratch).  A visible position whose block id is outside the pool, or a
 * seqused_k outside [0, max_blocks·block_size], is recorded as
 * KVC_ERR_BOUNDS: the page scores 0 (the request is skipped).
 * Errors: KVC_ERR_INVALID_ARG, KVC_ERR_SHAPE (D ∉ {64,128}, Hq % H,
 * Hq > 256, block_size > 64), KVC_ERR_ALIGN (q, kpool, lse, state).
 * ---------------------------------------------------------------------- */
size_t kvc_recover_score_workspace_size(int32_t n_req, int32_t max_blocks, int32_t L, int32_t H,
                                        int32_t Hq, int32_t D, int32_t block_size);
kvc_status kvc_recover_score(const kvc_bf16 *q, const float *lse, const kvc_bf16 *kpool,
                             int64_t n_slots, const int32_t *block_table, int32_t max_blocks,
                             const int32_t *seqused_k, const int32_t *count, int32_t n_req,
                             int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t block_size,
                             float *state, void *ws, size_t ws_bytes, int32_t *dev_status,
                             cudaStream_t stream);
/* kvc_recover_score with the kernel named by `kernel` (KVC_KERNEL_AUTO,
 * KVC_KERNEL_RECOVER_TC or KVC_KERNEL_RECOVER_CC). */
kvc_status kvc_recover_score_ex(const kvc_bf16 *q, const float *lse, const kvc_bf16 *kpool,
                                int64_t n_slots, const int32_t *block_table, int32_t max_blocks,
                                const int32_t *seqused_k, const int32_t *count, int32_t n_req,
                                int32_t L, int32_t H, int32_t Hq, int32_t D, int32_t block_size,
                                float *state, void *ws, size_t ws_bytes, int32_t *dev_status,
                                kvc_kernel kernel, cudaStream_t stream);

/* 1 if kvc_recover_score runs these sizes on the tensor cores, else 0. */
int32_t kvc_recover_tensor_core(int32_t H, int32_t Hq, int32_t D, int32_t block_size);

/* ------------------------------------------------------------------------
 * LRFU keep score (ActKV §5.2, attention-aware LRFU, Algorithm 1): after an
 * action region, every entry's keep score decays and gains its action-
 * region attention score when the entry is a hit, so an entry is evicted
 * only after it has not drawn high attention for a while.  Per segment s
 * (one request's entries [seg_off[s], seg_off[s+1])):
 *   hit_i  ⇔ i is in the shortest prefix of the entries ordered by score
 *            (descending, lower index first among equal scores) whose score
 *            mass reaches top_p · Σ scores (p = 0.9 on the page);
 *   keep_score[i] ← fma(lambda, keep_score[i], hit_i ? scores[i] : 0).
 * lambda = 0 keeps only the latest region (recency), lambda = 1 sums every
 * region (frequency).  Scores that are not positive finite numbers carry no
 * mass and never hit (a NaN is recorded as KVC_ERR_NAN).  The masses are
 * summed in fp64; the boundary entry is exact up to that rounding.
 *   scores      device fp32 (e.g. kvc_recover_score's state at the end of the
 *               region)
 *   seg_off     device int64 [n_seg+1], each segment ≤ max_seg_len
 *   keep_score  device fp32, same layout as scores, in/out
 *   hitmask     device uint32 [n_seg][⌈max_seg_len/32⌉] out, may be NULL
 * Entries with the highest keep scores are then retained with kvc_select.
 * Errors: KVC_ERR_INVALID_ARG (top_p or lambda outside [0, 1]),
 * KVC_ERR_SHAPE (max_seg_len > KVC_LRFU_MAX_SEG).
 * ---------------------------------------------------------------------- */
kvc_status kvc_lrfu_update(const float *scores, const int64_t *seg_off, int32_t n_seg,
                           int32_t max_seg_len, float top_p, float lambda, float *keep_score,
                           uint32_t *hitmask, int32_t *dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Confidence monitor (ActKV §6.1): token-level confidence of each predicted
 * distribution, the negative average log-probability of its top-k tokens,
 *   conf[t] = −(1/k) Σ_{j ≤ k} log P_t(j) = LSE_t − (1/k) Σ_{j ≤ k} logit_t(j)
 * (P_t = softmax of row t; ties at the k-th logit count once per copy).
 *   logits  device fp32 [n_tok][V]  (the model's output rows)
 *   conf    device fp32 [n_tok] out
 * fp32 arithmetic (LSE from per-thread online max/sum merged in a fixed
 * order); the top-k set is exact.  A NaN logit is recorded as KVC_ERR_NAN.
 * Errors: KVC_ERR_INVALID_ARG (sizes, top_k > V).
 * ---------------------------------------------------------------------- */
kvc_status kvc_token_confidence(const float *logits, int32_t n_tok, int32_t V, int32_t top_k,
                                float *conf, int32_t *dev_status, cudaStream_t stream);

/* Largest number of windows kvc_conf_trend_budget takes per trace. */
#define KVC_CONF_MAX_WINDOWS 8192

/* ------------------------------------------------------------------------
 * Trace confidence, trend and adaptive budget (ActKV §6.1 "Trace-level
 * confidence", "Trend detection"; §6.2 Algorithm 2).  For each trace t (one
 * request's token confidences conf[trace_off[t] … trace_off[t+1])):
 *   R'_m   = min of the window [m·stride, m·stride + window), m = 0 …
 *            ⌊(L − window)/stride⌋ (no window if L < window);
 *   Q      = the bottom_pct-th percentile of R' (linear interpolation between
 *            the order statistics at rank bottom_pct/100·(n − 1));
 *   slope[t] = least-squares slope of the windows with R'_m ≤ Q against m
 *            (fp64; 0 with fewer than two such windows); n_kept[t] = their
 *            number;
 *   budget[t] ← max(budget[t], min(budget[t] + budget_step, max_budget)) if
 *            slope < 0, else unchanged — the budget starts small and is never
 *            lowered (one already above max_budget is kept).
 *   conf       device fp32; trace_off device int64 [n_trace+1]
 *   slope      device fp64 [n_trace] out; budget device int32 [n_trace]
 *              in/out; n_kept device int32 [n_trace] out
 * Errors: KVC_ERR_INVALID_ARG, KVC_ERR_SHAPE (more than KVC_CONF_MAX_WINDOWS
 * windows), KVC_ERR_ALIGN (slope not 8-byte aligned).
 * ---------------------------------------------------------------------- */
kvc_status kvc_conf_trend_budget(const float *conf, const int64_t *trace_off, int32_t n_trace,
                                 int32_t max_trace_len, int32_t window, int32_t stride,
                                 float bottom_pct, int32_t budget_step, int32_t max_budget,
                                 double *slope, int32_t *budget, int32_t *n_kept,
                                 int32_t *dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Conflict-free tail slot plan (ActKV §7.2, Algorithm 4, planning step).
 * Request r holds n = seqused_k[r] tokens in Y = ⌈n/block_size⌉ logical
 * blocks, m of them retained (keep-mask bits).  All retained tokens are
 * consolidated into the last X = ⌈m/block_size⌉ logical blocks [Y−X, Y):
 *   sources       retained positions before the region, ascending;
 *   destinations  positions of the region that hold no retained token
 *                 (including the unused slots past n), ascending;
 * the k-th source goes to the k-th destination, so the two sets are
 * disjoint and all copies can run at once without a buffer.  Logical
 * positions are translated to physical slots through the block table.
 *   keepmask      device uint32 [n_req][mask_words]: bit p%32 of word p/32
 *                 = position p retained (bits at or past n are ignored)
 *   src_slot, dst_slot  device int32 [n_req][max_blocks·block_size] out:
 *                 the pairs, then −1
 *   n_pairs       device int32 [n_req] out
 *   n_tail_blocks device int32 [n_req] out: X
 *   freed_blocks  device int32 [n_req][max_blocks] out: block_table[r][0 …
 *                 Y−X−1] (returned to the allocator), then −1
 *   n_freed       device int32 [n_req] out: Y − X
 *   new_table     device int32 [n_req][max_blocks] out: block_table[r][Y−X
 *                 … Y−1], then −1
 *   tail_mask     device uint32 [n_req][⌈max_blocks·block_size/32⌉] out:
 *                 bit i = slot i of the region holds a retained token after
 *                 the copies
 * The result is unique and exact (integer work only).  A seqused_k outside
 * [0, max_blocks·block_size] or longer than mask_words·32 is recorded as
 * KVC_ERR_BOUNDS and that request gets an empty plan; a block id outside
 * the pool is recorded and its slot written as −1.
 * Errors: KVC_ERR_INVALID_ARG, KVC_ERR_SHAPE (max_blocks·block_size >
 * KVC_TAIL_MAX_TOKENS).
 * ---------------------------------------------------------------------- */
kvc_status kvc_tail_plan(const uint32_t *keepmask, int32_t mask_words,
                         const int32_t *seqused_k, const int32_t *block_table,
                         int32_t max_blocks, int32_t n_req, int32_t block_size, int64_t n_slots,
                         int32_t *src_slot, int32_t *dst_slot, int32_t *n_pairs,
                         int32_t *n_tail_blocks, int32_t *freed_blocks, int32_t *n_freed,
                         int32_t *new_table, uint32_t *tail_mask, int32_t *dev_status,
                         cudaStream_t stream);

/* ------------------------------------------------------------------------
 * One-shot in-place compaction (ActKV §7.2, Algorithm 4, copy step): for
 * every request r, pair k < n_pairs[r] and layer l,
 *   kpool[l][dst_slot[r][k]] ← kpool[l][src_slot[r][k]]   (H·D elements)
 *   vpool[l][dst_slot[r][k]] ← vpool[l][src_slot[r][k]]
 * as bit copies, all at once.  The pairs must come from kvc_tail_plan (or
 * any plan whose sources and destinations are disjoint); with overlapping
 * pairs the result is undefined.
 *   kpool, vpool  device bf16 [L][n_slots][H][D]  in/out
 *   src_slot, dst_slot  device int32 [n_req][pair_cap]; n_pairs device
 *                 int32 [n_req] (clamped to [0, pair_cap])
 * A slot outside [0, n_slots) is recorded as KVC_ERR_BOUNDS and that pair
 * is skipped.
 * Errors: KVC_ERR_INVALID_ARG, KVC_ERR_SHAPE (D, n_req > 65535),
 * KVC_ERR_ALIGN (pools).
 * ---------------------------------------------------------------------- */
kvc_status kvc_tail_compact(kvc_bf16 *kpool, kvc_bf16 *vpool, int64_t n_slots, int32_t L,
                            int32_t H, int32_t D, const int32_t *src_slot,
                            const int32_t *dst_slot, const int32_t *n_pairs, int32_t pair_cap,
                            int32_t n_req, int32_t *dev_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H_ */
