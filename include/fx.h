/*
 * fx.h -- C ABI of libfx: importance-scored KV-cache token selection feeding sparse GQA decode
 * attention, for one NVIDIA GB300 (sm_103a).
 *
 * What the calls compute follows three pages:
 *   [FastOCR]  "FastOCR: Dynamic Visual Fixation via KV Cache Pruning for Efficient Document Parsing",
 *              Methodology: Focal-Guided Pruning (focal layers attend over the whole cache and keep
 *              the top-attended image tokens at a kept ratio; the selection is propagated to the
 *              non-focal layers, which attend only to the pruned set) and Cross-Step Fixation Reuse
 *              (the deepest focal layer's set from the previous step warm-starts the next step).
 *   [FastKV]   "FastKV: Decoupling of Context Reduction and KV Cache Compression for Prefill-Decoding
 *              Acceleration", 2.A Token-Selective Propagation (saliency = attention weights from a
 *              recent window of queries to every context token) and 2.B Decoupled KV Retention (a
 *              chosen subset of KV entries is kept for decoding).
 *   [HPD]      "HPD-Parsing -- Hierarchical Parallel Document Parsing", method part 2 (branches reuse
 *              the shared visual + layout prefix KV zero-copy and each attends only to that prefix,
 *              its own prefix and its own history) and part 3 P-MTP (each branch drafts several
 *              tokens and verifies them in one step).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library allocates no device
 *     memory; calls that need scratch take a caller-provided workspace sized by the matching
 *     fx_*_workspace_bytes() query.  A workspace must be zero-filled once before its first use
 *     (fx_workspace_init does that); every call leaves it ready for the next one.  A workspace may be
 *     used by one stream at a time.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Calls only
 *     enqueue work; none synchronises the host, so they can be captured into CUDA graphs.
 *   - bf16 tensors are passed as fx_bf16 (the 16-bit storage of a bfloat16).  Head dimension d must
 *     be 128.  Rows of 128 bf16 values (256 bytes) must start on 16-byte boundaries: base pointers
 *     16-byte aligned and every row stride a multiple of 8 elements.
 *   - GQA grouping: with G = Hq / Hkv, query head g belongs to KV head g / G.
 *   - q and out tensors are laid out [batch, Hq, Mq, 128] (contiguous).  Outputs are fp32.
 *   - `flags` (the argument before `stream` of every compute call) is a bit set of FX_LAUNCH_*:
 *       FX_LAUNCH_PDL            launch as a programmatic dependent of the kernel enqueued just before
 *                                it on the same stream: the call's kernels may start while that kernel
 *                                is still running and wait for it on the device before reading or
 *                                writing anything it could have produced.  Back-to-back calls (layer
 *                                after layer) then overlap one call's start with the previous one's end.
 *       FX_LAUNCH_INPUTS_READY   (with FX_LAUNCH_PDL) the caller guarantees that the lengths, the index
 *                                lists and the K/V rows the call reads were written by the host or by
 *                                a kernel enqueued two or more launches earlier -- not by the kernel
 *                                immediately before.  The call may then read them, and start its K/V
 *                                loads, before that kernel finishes.  Queries, outputs and workspace
 *                                are still touched only after it finishes.
 *     0 gives ordinary stream-ordered launches.
 *   - The library keeps a little state per device (the address of its device error word, the SM count,
 *     and for the no-allocation call the address of its scratch array), looked up on the first call on
 *     each device.  A cudaDeviceReset invalidates it: make no library call on a device after resetting
 *     it in the same process.
 *   - Host-side argument errors return a status and set a thread-local message (fx_last_error);
 *     nothing is enqueued then.  Data that only the device can see (lengths, indices, offsets) is
 *     checked by the kernels: a bad value is clamped or skipped -- never dereferenced -- and a bit is
 *     set in a per-device error word that fx_device_errors() reads and clears.
 */
#ifndef FX_H
#define FX_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FX_API __attribute__((visibility("default")))
#else
#define FX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t fx_bf16; /* storage of one bfloat16 value */

typedef enum {
    FX_OK = 0,
    FX_ERR_INVALID_ARG = 1, /* a null pointer, an out-of-range size or a misaligned pointer/stride */
    FX_ERR_UNSUPPORTED = 2, /* a shape the kernels do not implement (d != 128, too many query rows) */
    FX_ERR_WORKSPACE = 3,   /* workspace missing, too small or not 256-byte aligned */
    FX_ERR_CUDA = 4,        /* a CUDA runtime call failed; fx_last_error() has its message */
    FX_ERR_DEVICE = 5       /* fx_device_errors(): a kernel saw bad device-side data */
} fx_status;

/* Launch flags (see the conventions above). */
#define FX_LAUNCH_PDL 1u
#define FX_LAUNCH_INPUTS_READY 2u

/* Bits of the device error word (fx_device_errors). */
#define FX_DEVERR_LEN 1u      /* a length outside [0, capacity]; it was clamped */
#define FX_DEVERR_INDEX 2u    /* a token index outside [0, len); that entry was skipped */
#define FX_DEVERR_OFFSETS 4u  /* branch suffix offsets decreasing or past the suffix rows; branch suffix skipped */
#define FX_DEVERR_CAPACITY 8u /* a compacted cache would exceed its capacity; extra rows not written */
#define FX_DEVERR_TIMEOUT 16u /* a bounded wait for an asynchronous copy gave up; that call's output is invalid */

/*
 * One layer's KV cache, read-only.  Element (b, h, t, c) of K is at k[b*stride_b + h*stride_h +
 * t*stride_t + c] (strides in elements), likewise V with the same strides.  Rows t < len[b] are
 * valid; len is a device array of B int32 values with 0 <= len[b] <= Tcap.
 */
typedef struct {
    const fx_bf16* k;
    const fx_bf16* v;
    const int32_t* len;
    int64_t stride_b, stride_h, stride_t;
    int32_t B, Hkv, Tcap, d;
} fx_kv_desc;

/* A writable KV cache (destination of fx_kv_compact); len receives the new lengths. */
typedef struct {
    fx_bf16* k;
    fx_bf16* v;
    int32_t* len;
    int64_t stride_b, stride_h, stride_t;
    int32_t B, Hkv, Tcap, d;
} fx_kv_out_desc;

/* Last host-side error message of the calling thread ("" if none). */
FX_API const char* fx_last_error(void);

/* ABI version of this header (incremented on any incompatible change). */
FX_API int fx_abi_version(void);

/*
 * Synchronises `stream`, then reads and clears the device error word of the current device.
 * *bits receives the FX_DEVERR_* bits seen since the last read.  Returns FX_ERR_DEVICE when any bit
 * was set, FX_OK otherwise.
 */
FX_API fx_status fx_device_errors(unsigned* bits, void* stream);

/* Zero-fills a workspace before its first use (an asynchronous memset on `stream`). */
FX_API fx_status fx_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------- */
/* fx_focal_attn_scores -- a focal layer: full attention over the whole cache plus per-token
 * importance.  [FastOCR] Focal-Guided Pruning; [FastKV] 2.A window saliency.
 *
 * For each sequence b, KV head h and query row (gi, i) (query head h*G + gi, query position i):
 *   p_j = softmax_j(scale * q . k_j) over the visible tokens j < len[b] -- and, when q_pos0 >= 0,
 *         only j <= q_pos0 + i (query position i sits at token position q_pos0 + i: causal window);
 *   out[b, h*G+gi, i, :] = sum_j p_j v_j                              (written when out != NULL)
 *   scores[b, h, j - cand_lo] = sum over the group's G*Mq rows of p_j,  cand_lo <= j < cand_hi
 *                                                                     (written when scores != NULL)
 * The softmax always runs over every visible token; the candidate range only selects which token
 * importances are reported (tokens j >= len[b] report 0).  Scores of one row sum to G*Mq over the
 * full range.  An empty row (len[b] == 0) gives out = 0.
 *
 *   kv      cache, as above                    q      [B, Hq, Mq, 128] bf16
 *   Hq      query heads (multiple of Hkv)      Mq     query positions per sequence (>= 1)
 *   q_pos0  -1: no causal limit; >= 0: position of query 0
 *   scale   logit scale (use 1/sqrt(128) for plain attention)
 *   out     [B, Hq, Mq, 128] fp32 or NULL      scores [B, Hkv, cand_hi - cand_lo] fp32 or NULL
 *   G*Mq must be <= 64.  0 <= cand_lo <= cand_hi <= Tcap.
 * Workspace: fx_focal_workspace_bytes(B, Hkv, Hq, Mq, Tcap) bytes.
 * A call without output rows (out == NULL) and with G*Mq > 8 runs on the tensor cores when K admits a
 * tensor map (row strides multiples of 8 elements and nonzero head and token strides; a batch stride
 * of 0 is allowed), the cache has at most 2 x (SM count) x 128 x (128 / N) rows (N = 16, 32 or 64,
 * the rows rounded up) and B*Hkv*(1 + 2*G*Mq) <= 262140 (its counters live in the workspace's fixed
 * counter region): the logits stay in tensor memory, so K is read once and no logits are written.
 * The result agrees with the other route within the score tolerance.  Its persistent CTAs (one per
 * SM) each allocate all 512 tensor-memory columns of the SM, and the allocation waits, without a limit,
 * for them to be free: run no other kernel that holds tensor memory concurrently on another stream.
 */
FX_API size_t fx_focal_workspace_bytes(int B, int Hkv, int Hq, int Mq, int Tcap);
FX_API fx_status fx_focal_attn_scores(const fx_kv_desc* kv, const fx_bf16* q, int Hq, int Mq, int q_pos0,
                               float scale, int cand_lo, int cand_hi, float* out, float* scores,
                               void* ws, size_t ws_bytes, unsigned flags, void* stream);

/* ------------------------------------------------------------------------------------------- */
/* fx_topk_select -- keep the k most important tokens of each row.  [FastOCR] Focal-Guided Pruning
 * (top-attended tokens at kept ratio tau) and Cross-Step Fixation Reuse (warm start).
 *
 * For each of `rows` rows of n fp32 scores (row r at scores + r*n): the k entries that come first in
 * the order (score descending, index ascending) -- so ties go to the lower index -- written to
 * idx_out[r*k .. r*k+k) in ascending index order.  Scores are compared as floats (-0.0 < +0.0; NaN
 * must not occur).
 * prev_idx (NULL or [rows, k] distinct indices in [0, n)) is the previous step's set: it only speeds
 * the search up (every score at least the smallest score over prev_idx is a candidate) and never
 * changes the result.  An index of prev_idx outside [0, n) sets FX_DEVERR_INDEX and that row runs
 * without the warm start.  Under FX_LAUNCH_INPUTS_READY, prev_idx is the index list read before the
 * preceding kernel finishes; the scores are always read after it.
 * 1 <= k <= n.  No workspace.
 */
FX_API fx_status fx_topk_select(const float* scores, int rows, int n, int k, const int32_t* prev_idx,
                         int32_t* idx_out, unsigned flags, void* stream);

/* ------------------------------------------------------------------------------------------- */
/* Focal-layer selection by warm-up profiling.  [FastOCR] Focal-Guided Pruning, Focal Layer Selection
 * (during w warm-up steps, profile each layer's image-attention ratio; the C layers with the highest
 * ratio become the focal layers).
 *
 * fx_focal_mass: for each row r (one (b, KV head)) of scores [rows, n] from fx_focal_attn_scores with
 * the image tokens as candidates,
 *   mass[r] = (accumulate ? mass[r] : 0) + (sum_j scores[r, j]) / R
 * which is the mean share of attention the group's R query rows put on the image tokens (a value in
 * [0, 1]).  A layer's image-attention ratio is the mean of mass over its rows and the warm-up steps.
 *   scores [rows, n] fp32; mass [rows] fp32 (read when accumulate != 0, then written).  No workspace.
 *
 * fx_choose_focal_layers (host only, no GPU): the C layers with the largest ratio[l] (ties go to the
 * lower layer), written to layers_out[0..C) in ascending order.  1 <= C <= n_layers.
 */
FX_API fx_status fx_focal_mass(const float* scores, int rows, int n, int R, int accumulate, float* mass,
                        unsigned flags, void* stream);
FX_API fx_status fx_choose_focal_layers(const float* ratio, int n_layers, int C, int32_t* layers_out);

/* ------------------------------------------------------------------------------------------- */
/* fx_csfr_schedule -- which index set every layer of one decode step attends over (host only, no GPU).
 * [FastOCR] Focal-Guided Pruning (a focal layer refreshes the set; the layers after it, down to the next
 * focal layer, attend only to that set) and Cross-Step Fixation Reuse (the layers before the first
 * focal layer reuse the previous step's set of the deepest focal layer).
 *
 * focal_layers: the C focal layers, strictly ascending, each in [0, n_layers).  first_step != 0: no
 * previous step exists (its layers before the first focal layer attend densely).  For each layer l:
 *   kind[l] = FX_CSFR_FOCAL     l is focal: fx_focal_attn_scores + fx_topk_select make its set; src[l] = l
 *             FX_CSFR_CURRENT   attend over this step's set of focal layer src[l] (the nearest above l)
 *             FX_CSFR_PREVIOUS  attend over the previous step's set of focal layer src[l] (the deepest)
 *             FX_CSFR_DENSE     attend over the whole cache (first step, before the first focal layer);
 *                               src[l] = -1
 * kind, src: host arrays of n_layers entries.
 */
#define FX_CSFR_FOCAL 0
#define FX_CSFR_CURRENT 1
#define FX_CSFR_PREVIOUS 2
#define FX_CSFR_DENSE 3
FX_API fx_status fx_csfr_schedule(int n_layers, const int32_t* focal_layers, int C, int first_step, int32_t* kind,
                                  int32_t* src);

/* ------------------------------------------------------------------------------------------- */
/* fx_sparse_gqa_decode -- a non-focal layer: decode attention over the selected tokens only.
 * [FastOCR] Focal-Guided Pruning (non-focal layers attend only to the pruned set; the full cache
 * stays intact); [FastKV] 2.B (decoding over the retained entries).
 *
 * One query position per sequence.  For each b and query head g (KV head h = g / G):
 *   S = { idx[b, h, 0..k) } followed by the dense tail { tail_lo .. len[b]-1 }
 *   out[b, g, 0, :] = sum_{j in S} softmax_S(scale * q . k_j) v_j   (softmax renormalised over S)
 * idx entries are token positions in [0, len[b]); an entry outside that range sets FX_DEVERR_INDEX
 * and is skipped.  A listed token that is also in the tail counts twice (callers keep idx < tail_lo).
 * k = 0 with tail_lo = 0 is plain dense decode over the whole cache; an empty S gives out = 0.
 *
 *   q    [B, Hq, 1, 128] bf16         idx  [B, Hkv, k] int32 (NULL when k == 0)
 *   out  [B, Hq, 1, 128] fp32         G = Hq / Hkv must be <= 64
 * Workspace: fx_sparse_workspace_bytes(B, Hkv, Hq, k, tail_lo, Tcap) bytes.
 */
FX_API size_t fx_sparse_workspace_bytes(int B, int Hkv, int Hq, int k, int tail_lo, int Tcap);
FX_API fx_status fx_sparse_gqa_decode(const fx_kv_desc* kv, const fx_bf16* q, int Hq, const int32_t* idx,
                               int k, int tail_lo, float scale, float* out, void* ws,
                               size_t ws_bytes, unsigned flags, void* stream);

/* ------------------------------------------------------------------------------------------- */
/* fx_kv_compact -- decoupled KV retention: copy the retained rows of n_layers layers into a
 * contiguous cache, once, after prefill.  [FastKV] 2.B.
 *
 * For every layer l < n_layers, b and h, destination row r of
 *   S = idx_l[b, h, 0..k) followed by tail_lo .. len[b]-1,   idx_l = idx + l*idx_stride_layer
 * receives source row S[r] (K and V, bit-exact copies), so the kept rows stay in the order given
 * (ascending when idx is ascending and below tail_lo).  dst->len[b] = k + max(0, len[b] - tail_lo).
 * Layer l of the source starts at element offset l*src_stride_layer from src->k / src->v, layer l of
 * the destination at l*dst_stride_layer; all layers share src->len.  Rows past the new length are
 * not touched.  An idx entry outside [0, len[b]) sets FX_DEVERR_INDEX and its row is not written; a
 * new length above dst->Tcap sets FX_DEVERR_CAPACITY and only dst->Tcap rows are written (dst->len
 * is then clamped to dst->Tcap).
 *   idx [B, Hkv, k] int32 per layer (NULL when k == 0); idx_stride_layer (elements) = 0: one set
 *   for every layer (a selection made at one layer), B*Hkv*k for a [n_layers, B, Hkv, k] array of
 *   per-layer sets (FastKV's per-layer KV retention).  src and dst must agree on B, Hkv and d.
 * No workspace.
 */
FX_API fx_status fx_kv_compact(const fx_kv_desc* src, int64_t src_stride_layer, const int32_t* idx,
                        int64_t idx_stride_layer, int k, int tail_lo, const fx_kv_out_desc* dst,
                        int64_t dst_stride_layer, int n_layers, unsigned flags, void* stream);

/*
 * Decode-step append: the new token's key and value rows of every layer join that layer's cache.
 * [FastKV] 3.2 decodes over the compacted cache and [FastOCR] decodes over the visual + text cache;
 * in both, every decoding step adds one row per (layer, sequence, KV head).
 *
 * For every layer l < n_layers, b < cache->B and h < cache->Hkv:
 *   K_l[b, h, pos[b], :] = k_new[l, b, h, :]   and   V_l[b, h, pos[b], :] = v_new[l, b, h, :]
 * as bit-exact copies, where layer l of the cache starts at element offset l*stride_layer from
 * cache->k / cache->v.
 *   k_new, v_new  bf16 [n_layers, B, Hkv, 128], contiguous (device).
 *   pos           int32 [B] (device): the row each sequence writes, normally its current length.  A
 *                 position outside [0, cache->Tcap) sets FX_DEVERR_LEN and that sequence's rows are
 *                 not written.
 * cache->len is neither read nor written (lengths stay the caller's).  No workspace.
 */
FX_API fx_status fx_kv_append(const fx_kv_out_desc* cache, int64_t stride_layer, int n_layers,
                              const fx_bf16* k_new, const fx_bf16* v_new, const int32_t* pos, unsigned flags,
                              void* stream);

/* ------------------------------------------------------------------------------------------- */
/* fx_kv_retain_per_layer -- FastKV decoupled KV retention with its own selection at every layer.
 * [FastKV] 2.A (saliency: attention of a window of recent queries to all context tokens) and 2.B
 * (KV retention rate: how many entries each layer keeps for decoding).
 *
 * For every layer l < n_layers (layer l of the cache at element offset l*src_stride_layer from
 * kv->k / kv->v; all layers share kv->len):
 *   scores_l = fx_focal_attn_scores(layer l, window queries q_l, q_pos0, scale, candidates [0, cand_hi))
 *              (scores only: no output rows, V is not read)
 *   idx_l    = fx_topk_select(scores_l, keep_k)  -> idx_out + l*B*Hkv*keep_k
 * then fx_kv_compact of all n_layers layers with the per-layer sets idx_l followed by the tail
 * [tail_lo, len[b]) (the window), into dst (layer l at l*dst_stride_layer; dst->len = new lengths).
 *   q        [n_layers, B, Hq, Mq, 128] bf16 (contiguous): layer l's window queries
 *   idx_out  [n_layers, B, Hkv, keep_k] int32, written (ascending per row)
 *   1 <= keep_k <= cand_hi <= Tcap.  Results equal those of the individual calls.
 * Workspace: fx_retain_workspace_bytes(B, Hkv, Hq, Mq, Tcap, cand_hi) bytes: the scoring scratch and
 * the scores of up to 32 layers.  Layers are taken 32 at a time; with more than 8 query rows per KV
 * head a batch is scored by one launch of the tensor-core scoring kernel (otherwise by one focal call
 * per layer), and each batch is selected by one top-k call over all its rows.  A K layout that admits
 * no tensor map (strides not multiples of 16 bytes) takes the per-layer calls.
 */
FX_API size_t fx_retain_workspace_bytes(int B, int Hkv, int Hq, int Mq, int Tcap, int cand_hi);
FX_API fx_status fx_kv_retain_per_layer(const fx_kv_desc* kv, int64_t src_stride_layer, int n_layers,
                                 const fx_bf16* q, int Hq, int Mq, int q_pos0, float scale, int cand_hi,
                                 int keep_k, int tail_lo, int32_t* idx_out, const fx_kv_out_desc* dst,
                                 int64_t dst_stride_layer, void* ws, size_t ws_bytes, unsigned flags,
                                 void* stream);

/* ------------------------------------------------------------------------------------------- */
/* fx_shared_prefix_decode -- parallel draft verification over a shared prefix.  [HPD] parts 2
 * (shared-prefix KV reuse with context isolation) and 3 (P-MTP parallel verification).
 *
 * Br branches share one prefix KV; branch b sees its first P_b rows (P_b = len[b], the branch's fork
 * position, or P when len == NULL) -- zero-copy reuse of the context visible where it forked.  It
 * owns suffix rows off[b] .. off[b]+L_b-1 and Mq draft rows.  For branch b, KV head h and query row
 * (gi, i) (query head h*G + gi, draft position i):
 *   S = prefix rows 0..P_b-1 (or prefix_idx[b, h, 0..kp) when prefix_idx != NULL)
 *       ++ the branch's suffix rows ++ the branch's draft rows 0..i         (causal inside the draft)
 *   out[b, h*G+gi, i, :] = sum_{j in S} softmax_S(scale * q . k_j) v_j
 *
 *   prefix      rows (h, t) at k + h*stride_h + t*stride_t, t < P (k and v non-NULL even when P == 0);
 *               len: NULL or device [Br] int32 in [0, P] (outside: FX_DEVERR_LEN, clamped)
 *   suffix      rows (h, t) at suf_k + h*suf_stride_h + t*suf_stride_t, t < suf_rows
 *   suf_off     suf_len == NULL: device [Br + 1] int32, non-decreasing, L_b = suf_off[b+1] - suf_off[b];
 *               suf_len != NULL: device [Br] starts and L_b = suf_len[b] (ranges anywhere, e.g. fixed
 *               slots of a branch pool); every range must lie in [0, suf_rows) and L_b <= max_suffix
 *               (else FX_DEVERR_OFFSETS: an out-of-range suffix is skipped, a long one cut)
 *   draft       rows (b, i, h) at draft_k + b*draft_stride_b + i*draft_stride_i + h*draft_stride_h
 *   q           [Br, Hq, Mq, 128] bf16;  out [Br, Hq, Mq, 128] fp32;  G*Mq <= 64
 *   prefix_idx  NULL (dense prefix) or [Br, Hkv, kp] int32 prefix positions in [0, P_b) (others set
 *               FX_DEVERR_INDEX and are skipped)
 * Workspace: fx_shared_prefix_workspace_bytes(Br, Hkv, Hq, Mq, np, max_suffix) bytes, where np is
 * P (dense) or kp (sparse).
 * A dense prefix of at least 128 rows with Br*G*Mq >= 128 query rows per KV head runs on the tensor
 * cores (128-row x 128-key tiles, bf16 products with fp32 accumulation, the probabilities as bf16
 * hi + lo parts): two launches, the prefix partials held in the workspace (included in the size
 * above) and folded into the verify kernel's merge.  The result agrees with the single-kernel route
 * within the same output tolerance.  Each CTA of that route allocates all 512 columns of its SM's
 * tensor memory and the allocation waits, without a limit, for them to be free: run no other kernel
 * that holds tensor memory concurrently on another stream.
 */
typedef struct {
    const fx_bf16* k;
    const fx_bf16* v;
    int64_t stride_h, stride_t;
    int32_t P, Hkv, d;
    const int32_t* len;   /* [Br] visible prefix rows per branch (fork positions), or NULL: all P */
} fx_prefix_desc;

typedef struct {
    const fx_bf16* suf_k;
    const fx_bf16* suf_v;
    int64_t suf_stride_h, suf_stride_t;
    const int32_t* suf_off;
    int32_t suf_rows, max_suffix;
    const fx_bf16* draft_k;
    const fx_bf16* draft_v;
    int64_t draft_stride_b, draft_stride_i, draft_stride_h;
    int32_t Br, Mq;
    const int32_t* suf_len;   /* [Br] suffix rows per branch (suf_off then holds starts), or NULL */
} fx_branch_desc;

FX_API size_t fx_shared_prefix_workspace_bytes(int Br, int Hkv, int Hq, int Mq, int np, int max_suffix);
FX_API fx_status fx_shared_prefix_decode(const fx_prefix_desc* prefix, const fx_branch_desc* branches,
                                  const fx_bf16* q, int Hq, const int32_t* prefix_idx, int kp,
                                  float scale, float* out, void* ws, size_t ws_bytes, unsigned flags,
                                  void* stream);

/* ------------------------------------------------------------------------------------------- */
/* Branch pool -- host-side bookkeeping for layout-coordinated parallel decoding.  [HPD] part 2
 * (content branches fork at <FORK>, reuse the shared prefix KV visible at the fork position without a
 * copy, and the shared KV is released by reference count when every child is done).
 *
 * One shared prefix of at most prefix_cap rows (the parent's context; it grows as the layout branch
 * decodes) and at most max_branches content branches, each owning the fixed slot of suffix rows
 * [id*slot_rows, (id+1)*slot_rows) of a caller-owned suffix buffer.  The pool does no GPU work and
 * owns no device memory: it hands out rows and fills the branch arrays of fx_shared_prefix_decode.
 * Calls returning int give -1 on error (message in fx_last_error); the pool is thread-safe.
 *   create           NULL on bad sizes
 *   extend_prefix    the parent appends n prefix rows: first new row (-1 past prefix_cap)
 *   fork             a new branch whose fork position is the current prefix length: its id (= slot),
 *                    -1 when every slot is taken; the prefix gains a reference
 *   append           reserve n more suffix rows of branch id: the first row to write (-1 when the
 *                    slot would overflow or the branch is not live)
 *   release          branch id done: its slot is free; returns the prefix references left
 *   release_parent   the parent is done (no more extend/fork); returns the references left -- at 0
 *                    the prefix buffer may be freed
 *   batch            the live branches in ascending id order: ids, suffix starts (suf_off with
 *                    suf_len), suffix lengths and fork positions (fx_prefix_desc.len), host arrays of
 *                    max_branches entries; returns how many
 */
typedef struct fx_branch_pool fx_branch_pool;
FX_API fx_branch_pool* fx_branch_pool_create(int prefix_cap, int max_branches, int slot_rows);
FX_API void fx_branch_pool_destroy(fx_branch_pool* pool);
FX_API int fx_branch_pool_extend_prefix(fx_branch_pool* pool, int n);
FX_API int fx_branch_pool_fork(fx_branch_pool* pool);
FX_API int fx_branch_pool_append(fx_branch_pool* pool, int branch, int n);
FX_API int fx_branch_pool_release(fx_branch_pool* pool, int branch);
FX_API int fx_branch_pool_release_parent(fx_branch_pool* pool);
FX_API int fx_branch_pool_prefix_refs(fx_branch_pool* pool);
FX_API int fx_branch_pool_prefix_len(fx_branch_pool* pool);
FX_API int fx_branch_pool_batch(fx_branch_pool* pool, int32_t* ids, int32_t* suf_start, int32_t* suf_len,
                         int32_t* prefix_len);

/* ------------------------------------------------------------------------------------------- */
/* fx_test_stall_wait -- testing hook for the device-side failure path; the pages have no counterpart.
 *
 * Every wait of a kernel on an mbarrier (copies landing, pushed partials arriving) gives up after a
 * fixed number of polls, sets FX_DEVERR_TIMEOUT and lets the kernel finish, so a wait that can never
 * complete leaves the context usable instead of hanging the GPU.  With polls > 0, every later
 * decode-shaped fx_sparse_gqa_decode call (G <= 8 query heads per KV head) adds one such wait, of
 * `polls` polls, on a barrier that nothing arrives on, after its results are complete: the call
 * returns, its output is still correct, and fx_device_errors() then reports FX_DEVERR_TIMEOUT.
 * polls = 0 (the default) turns the extra wait off.  Process-wide; not for production use.
 */
FX_API void fx_test_stall_wait(unsigned polls);

/* ------------------------------------------------------------------------------------------- */
/* fx_focal_attn_scores_noalloc -- fx_focal_attn_scores for callers that cannot allocate device
 * memory.  The pages have no counterpart for this call; it is a convenience of this library.
 *
 * Who needs it: code that runs while a CUDA graph is being captured (allocating there is refused or
 * forces a device-wide synchronisation that breaks the capture), real-time loops that allow no
 * allocator calls after start-up, and hosts that reach the GPU only through this C interface.
 *
 * Same arguments and results as fx_focal_attn_scores, without ws / ws_bytes: the scratch is one
 * fixed device array inside the library, fx_noalloc_scratch_bytes() = 16 MiB, which every GPU that
 * loads the library holds until the process exits.  A call whose fx_focal_workspace_bytes() exceeds
 * that size returns FX_ERR_UNSUPPORTED and launches nothing.  The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress), so make that first call before any stream
 * capture.  All calls on a device share the one array and leave their data in it; nothing in it has
 * to start at zero.  Calls that can overlap on the GPU (for example on two streams) race on the
 * array: the caller must order them.  The call allocates nothing.
 */
FX_API size_t fx_noalloc_scratch_bytes(void);
FX_API fx_status fx_focal_attn_scores_noalloc(const fx_kv_desc* kv, const fx_bf16* q, int Hq, int Mq,
                                              int q_pos0, float scale, int cand_lo, int cand_hi,
                                              float* out, float* scores, unsigned flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FX_H */
