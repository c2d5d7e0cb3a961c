/*
 * kvsel.h - attention-guided KV selection on one NVIDIA GB300 (sm_103a).
 *
 * C ABI of libkvsel.so.  Every entry point validates its arguments on the
 * host, then enqueues hand-written CUDA kernels on the caller's stream and
 * returns without synchronising.  Conventions shared by all calls:
 *
 *  - Pointers are DEVICE pointers owned by the caller unless stated
 *    otherwise.  The library allocates no device memory: scratch comes from
 *    a caller-provided workspace whose size the matching *_workspace()
 *    function returns.
 *  - Every workspace starts with a device status word and the counters the
 *    kernels synchronise on.  A workspace must be zero when first used
 *    (allocate it zeroed); afterwards the library keeps it consistent.
 *    After a KVSEL_ERR_TIMEOUT status, zero the whole workspace again.  Kernels that detect a problem on the device
 *    (a block-table entry outside the pool, a bounded wait that ran out)
 *    record a kvsel_status there and carry on without faulting;
 *    kvsel_read_status() returns it.
 *  - Host-detectable errors (NULL where a buffer is required, unsupported
 *    head_dim / page_size / group size, a budget smaller than sinks +
 *    window, a workspace that is too small) return immediately with no
 *    launch, and kvsel_last_error_string() describes them.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *  - CUDA graphs: calls of kvsel_decode_attn, kvsel_h2o_evict,
 *    kvsel_snapkv_select and kvsel_block_priority (with their input and
 *    output copies) have been captured and replayed, the first two with
 *    results identical to the same calls made eagerly; kvsel_sparse_decode
 *    must not be captured (see its notes); the other entry points have not
 *    been tried in a graph.
 *  - No C++ exception crosses this interface.
 *
 * Paged KV layout (the paged cache of "From sliding window to
 * attention-guided eviction" §5, blocks of 16 or 256 tokens): K and V pools
 * are separate bf16 arrays [num_pages][num_kv_heads][page_size][head_dim]; a
 * sequence owns the pages listed in its row of an int32 block table
 * [batch][max_pages]; token slot t of sequence b lives in page
 * block_table[b][t / page_size], row t % page_size.  Supported here:
 * head_dim = 128; num_q_heads / num_kv_heads <= 16 for the decode step
 * (and its block signal), the sparse decode and Quest, <= 8 for SnapKV;
 * and page_size 16, 32, 64, 128 or 256 for the decode step, the H2O evict,
 * the keep-list compaction, the sparse decode and Quest (the kernels
 * address a page in 16-token tiles); SnapKV and the decode step's block
 * signal take page_size 16 only (else KVSEL_ERR_UNSUPPORTED).
 */
#ifndef KVSEL_H
#define KVSEL_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVSEL_API __attribute__((visibility("default")))
#else
#define KVSEL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvsel_status {
  KVSEL_OK = 0,
  KVSEL_ERR_INVALID_ARG = 1, /* rejected on the host; nothing was launched       */
  KVSEL_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels implement */
  KVSEL_ERR_CUDA = 3,        /* a CUDA runtime call failed (launch, attribute)   */
  KVSEL_ERR_TIMEOUT = 4,     /* device: a bounded wait ran out                   */
  KVSEL_ERR_BAD_INDEX = 5    /* device: a block-table entry outside the pool     */
} kvsel_status;

typedef enum kvsel_dtype { KVSEL_BF16 = 0, KVSEL_F32 = 1 } kvsel_dtype;

typedef struct kvsel_paged_kv {
  void* k_pool;          /* bf16 [num_pages][num_kv_heads][page_size][head_dim] */
  void* v_pool;          /* bf16, same layout                                   */
  int32_t num_pages;
  int32_t num_kv_heads;
  int32_t num_q_heads;   /* q head h reads kv head h / (num_q_heads/num_kv_heads) */
  int32_t head_dim;      /* 128                                                 */
  int32_t page_size;     /* 16, 32, 64, 128 or 256 (see above for which calls)  */
} kvsel_paged_kv;

/* Human-readable reason for the last non-OK status returned on this thread. */
KVSEL_API const char* kvsel_last_error_string(void);

/* Zero the status word of `workspace` (async on `stream`); the
 * synchronisation counters are left alone. */
KVSEL_API kvsel_status kvsel_clear_status(void* workspace, void* stream);

/* Synchronise `stream`, return the device status recorded in `workspace`
 * since it was last cleared, and clear it. */
KVSEL_API kvsel_status kvsel_read_status(void* workspace, void* stream);

/* Bound the waits on other CTAs of the kernels that use `workspace` (the
 * decode step's per-pair readiness counters, the block-priority sort's grid
 * barriers) at `spins` short sleeps (tens of ns each) instead of the default
 * of a few seconds; 0 restores the default.  Enqueued on `stream`; the value
 * sits in the workspace's status block and stays until changed or the
 * workspace is zeroed.  A wait that runs out records KVSEL_ERR_TIMEOUT and
 * the kernel finishes without hanging: the decode step's results are then
 * unspecified (every access stays in bounds), the sort stops before its
 * scatter.  Waits inside one CTA (TMA stages) keep their own fixed bound.
 * Failure-detection tests use a short limit with a wait that nothing ends. */
KVSEL_API kvsel_status kvsel_set_wait_limit(void* workspace, unsigned spins, void* stream);

/* Launch tracing for profiling.  While tracing is on for the calling thread,
 * every kernel the library launches from that thread records
 * events[2i] just before and events[2i+1] just after launch i, on the launch
 * stream.  `events` holds 2*capacity cudaEvent_t handles created by the
 * caller; launches past `capacity` are not recorded. */
KVSEL_API kvsel_status kvsel_trace_start(void* const* events, int capacity);
/* Stop tracing.  Returns the number of launches recorded and, when `names`
 * is non-NULL, stores up to `capacity` static kernel-name strings there. */
KVSEL_API int kvsel_trace_stop(const char** names, int capacity);

/* ---------------------------------------------------------------------------
 * Score-emitting decode attention (append + split-K attention + H2O update).
 *
 * Defines ("From sliding window to attention-guided eviction" §3.1 and §4.2
 * step 1; "Long context, KV eviction and sparse attention", sparse-selection
 * section, for the d^-1/2 scale and the q-head -> kv-head grouping):
 *   for each sequence b (live length S_b after the optional append) and
 *   q head h with kv head g = h / G:
 *     s_j  = scale * q_h . K_g[j]            for j < S_b
 *     p_hj = exp(s_j - max s) / sum exp(s - max s)
 *     o_h  = sum_j p_hj V_g[j]
 *     cum[b][g][j] += sum_{h in group g} p_hj      (the H2O cumulative score)
 *
 * Arguments:
 *   kv           paged pools (read; the appended token is written).
 *   block_table  int32 [batch][max_pages], read only.
 *   seq_lens     int32 [batch]: in, live length before the append; out, +1
 *                when k_new/v_new are given (written by the last kernel).
 *   q            bf16 [batch][num_q_heads][head_dim].
 *   k_new,v_new  bf16 [batch][num_kv_heads][head_dim], or both NULL (no
 *                append).  The new token goes to slot seq_lens[b] and is
 *                attended in the same call.
 *   pos_map      int32 [batch][num_kv_heads][max_len] or NULL: slot -> original
 *                token position; the appended slot gets next_pos[b].
 *   next_pos     int32 [batch] or NULL: original position of the next token;
 *                incremented with the append.  Required if pos_map is given.
 *   scale        logit scale (head_dim^-1/2 for standard attention).
 *   out          [batch][num_q_heads][head_dim], bf16 or fp32 per out_dtype.
 *   probs        fp32 [batch][num_q_heads][max_len] or NULL: p_hj at slot j;
 *                entries j >= S_b are not written.
 *   h2o_cum      fp32 [batch][num_kv_heads][max_len] or NULL: updated in
 *                place; the appended slot starts from 0.
 *   max_len      capacity in slots of probs / h2o_cum / pos_map rows;
 *                every S_b (after the append) must be <= max_len and
 *                <= max_pages * page_size, else KVSEL_ERR_BAD_INDEX is
 *                recorded on the device and nothing is computed.
 *   batch        at most 1024 sequences.
 *   num_ctas     how many CTAs share the work: the pages of all (sequence,
 *                kv head) pairs are cut into num_ctas equal contiguous ranges
 *                (0 = every co-resident CTA slot, the fastest choice; at most
 *                that many, and at most 1024).  Results do not depend on it
 *                beyond fp32 rounding.
 *   workspace    >= kvsel_decode_attn_workspace(...) bytes, status word zeroed.
 *   h2o_link     NULL, or the workspace of the kvsel_h2o_evict call(s) that
 *                follow this step for the same batch and kv heads, with
 *                h2o_link_bytes its size (at least the part that
 *                kvsel_h2o_link_bytes(batch, num_kv_heads) gives; else
 *                KVSEL_ERR_INVALID_ARG).  Used only with h2o_cum: the step
 *                then also lists, per (sequence, kv head), the slots whose new
 *                score is at or above the threshold that the last evict call
 *                found for that row, and the next evict call selects among
 *                those alone when the list allows it.  Selections are
 *                identical with or without it.  The list is valid until the
 *                next call that changes the scores.
 * Returns KVSEL_OK once the kernels are enqueued.
 */
KVSEL_API size_t kvsel_decode_attn_workspace(const kvsel_paged_kv* kv, int batch, int max_len,
                                   int with_probs);
KVSEL_API kvsel_status kvsel_decode_attn(const kvsel_paged_kv* kv, const int32_t* block_table,
                               int max_pages, int32_t* seq_lens, int batch, const void* q,
                               const void* k_new, const void* v_new, int32_t* pos_map,
                               int32_t* next_pos, float scale, void* out, int out_dtype,
                               float* probs, float* h2o_cum, int max_len, int num_ctas,
                               void* workspace, size_t ws_bytes, void* h2o_link,
                               size_t h2o_link_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Decode step that also emits the step's top-k block signal ("Sparse
 * attention x KV-cache offloading: eight questions" §5.1: each block keeps an
 * fp32 score accumulator and an int32 last-update step, and every decode
 * step accumulates each request's top-k blocks, k = 512 in the page's
 * estimate) from the same launch.
 *
 * Defines, on top of kvsel_decode_attn: for sequence b (S_b keys after the
 * append) and block (page) j < ceil(S_b / 16),
 *   mass[b][j] = the step's attention probability summed over every q head
 *                and the block's keys
 *   chosen[b]  = the topk_blocks blocks of largest mass, ties to the lower
 *                block (every block when there are no more), ascending
 *   for j in chosen[b], phys = block_table[b][j]:
 *                block_score[phys] += mass[b][j];  block_step[phys] = step
 * Other blocks' metadata is left untouched.  A sequence with no keys gets no
 * signal (its topk_out row is -1).
 *
 * signal (host pointer; NULL: exactly kvsel_decode_attn):
 *   topk_blocks   >= 1.
 *   step          the value stamped into block_step.
 *   block_score   fp32 [num_pages], block_step int32 [num_pages]: per
 *                 physical block, read-modify-written (device pointers).
 *   topk_out      int32 [batch][topk_blocks] or NULL: chosen[b], -1 padded.
 *   mass_out      fp32 [batch][ceil(max_len / 16)] or NULL: mass[b][j].
 * workspace       >= kvsel_decode_attn_ex_workspace(kv, batch, max_len,
 *                 probs != NULL, signal != NULL) bytes, zeroed before first
 *                 use.
 * The signal runs in the kernel's last phase, on the CTA that completes a
 * sequence's last (sequence, kv head) pair.
 */
typedef struct kvsel_block_signal {
  int topk_blocks;
  int32_t step;
  float* block_score;
  int32_t* block_step;
  int32_t* topk_out;
  float* mass_out;
} kvsel_block_signal;
KVSEL_API size_t kvsel_decode_attn_ex_workspace(const kvsel_paged_kv* kv, int batch, int max_len,
                                                int with_probs, int with_signal);
KVSEL_API kvsel_status kvsel_decode_attn_ex(const kvsel_paged_kv* kv, const int32_t* block_table,
                                            int max_pages, int32_t* seq_lens, int batch, const void* q,
                                            const void* k_new, const void* v_new, int32_t* pos_map,
                                            int32_t* next_pos, float scale, void* out, int out_dtype,
                                            float* probs, float* h2o_cum, int max_len, int num_ctas,
                                            const kvsel_block_signal* signal, void* workspace,
                                            size_t ws_bytes, void* h2o_link, size_t h2o_link_bytes,
                                            void* stream);
/* Bytes at the start of an H2O evict workspace that kvsel_decode_attn uses as
 * h2o_link (0 for invalid arguments). */
KVSEL_API size_t kvsel_h2o_link_bytes(int batch, int num_kv_heads);

/* Invalidate the decode -> select hand-off kept in an H2O evict workspace
 * (async on `stream`): every row's candidate list and last threshold are
 * cleared, so the next kvsel_h2o_evict ranks each row's full scores and the
 * decode step after it collects candidates again from the new thresholds.
 * Call it after writing h2o_cum by other means (seeding it from
 * kvsel_snapkv_select_ex's seed_out, adding a prefill seed, restoring a
 * checkpoint): a list built before such a write does not hold a slot that
 * the write lifted above the row's threshold.
 *   workspace  the H2O evict workspace (256-byte aligned), for batch x
 *              num_kv_heads rows.
 * Returns KVSEL_ERR_INVALID_ARG for a NULL or misaligned workspace or
 * non-positive sizes. */
KVSEL_API kvsel_status kvsel_h2o_link_reset(void* workspace, int batch, int num_kv_heads, void* stream);

/* Allocation-free kvsel_decode_attn.  The pages have no counterpart: this is
 * for callers that cannot allocate device memory (a runtime without a device
 * allocator, a plug-in whose host owns all allocations, code that must not
 * call the allocator in the middle of a step).  It takes the same arguments
 * as kvsel_decode_attn minus the workspace and the H2O link, and computes
 * the same results;
 * its scratch is a fixed 8 MiB array inside this library that every GPU
 * loading the library keeps until the process exits.
 *  - The first call on a device looks up that array's device address (with
 *    the device current); make that first call before any stream capture.
 *  - Calls that need more scratch than 8 MiB are rejected with
 *    KVSEL_ERR_INVALID_ARG: about (1024 + batch * num_kv_heads) * 64 bytes
 *    + batch * num_kv_heads * 12 bytes + batch * num_q_heads * 512 bytes (an
 *    fp32 O accumulator), plus batch * num_q_heads * max_len * 4 bytes when
 *    probs is not given (the kernel keeps its logits there).
 *  - Every call uses the same array, so calls that overlap on the GPU (other
 *    streams, other threads) race and corrupt each other; serialise them.
 *    Each call clears the array's status word, counters and O accumulator
 *    first.
 *  - Device-side problems (a block-table entry outside the pool) are not
 *    reported back: there is no workspace to read them from.
 * Nothing here calls cudaMalloc, cudaFree or any allocating library routine. */
KVSEL_API kvsel_status kvsel_decode_attn_noalloc(const kvsel_paged_kv* kv, const int32_t* block_table,
                                                 int max_pages, int32_t* seq_lens, int batch,
                                                 const void* q, const void* k_new, const void* v_new,
                                                 int32_t* pos_map, int32_t* next_pos, float scale,
                                                 void* out, int out_dtype, float* probs,
                                                 float* h2o_cum, int max_len, int num_ctas,
                                                 void* stream);

/* ---------------------------------------------------------------------------
 * H2O heavy-hitter selection with StreamingLLM sinks + window, optional
 * in-place compaction.
 *
 * Defines ("From sliding window to attention-guided eviction" §4.1 and the
 * §4.2 pseudocode; "Long context, KV eviction and sparse attention",
 * StreamingLLM section): for each sequence b and kv head g with live length
 * S = seq_lens[b]:
 *   if S <= budget nothing is evicted; otherwise
 *   keep = [0, n_sink) U HH U [S - window, S), where HH is the
 *   (budget - n_sink - window) slots of [n_sink, S - window) with the
 *   largest h2o_cum[b][g][.], ties to the lower slot.
 * With budget = n_sink + window this is StreamingLLM; with n_sink = 0 as
 * well it is the sliding window.
 *
 * Arguments:
 *   kv, block_table  pools and table; modified only when compact != 0.
 *   seq_lens     int32 [batch]; when compact != 0 set to min(S, budget).
 *   h2o_cum      fp32 [batch][num_kv_heads][max_len] (read; compacted).
 *   pos_map      int32 [batch][num_kv_heads][max_len] or NULL (compacted).
 *   budget, n_sink, window   budget >= n_sink + window, n_sink,window >= 0.
 *   compact      0: select only.  1: also move the kept K/V rows, scores and
 *                positions to slots 0..n_keep-1 in order, set block-table
 *                entries from ceil(n_keep/page_size) up to the old page count
 *                to -1 and list those page ids in freed_pages.
 *   keep_out     int32 [batch][num_kv_heads][budget] or NULL: kept original
 *                positions (pos_map applied; slot indices if pos_map is
 *                NULL), ascending, padded with -1.
 *   freed_pages  int32 [batch][max_pages] or NULL: released page ids, -1 padded.
 *   workspace    >= kvsel_h2o_evict_workspace(...) bytes, status word zeroed.
 */
KVSEL_API size_t kvsel_h2o_evict_workspace(const kvsel_paged_kv* kv, int batch, int budget);
KVSEL_API kvsel_status kvsel_h2o_evict(const kvsel_paged_kv* kv, int32_t* block_table, int max_pages,
                             int32_t* seq_lens, int batch, float* h2o_cum, int32_t* pos_map,
                             int max_len, int budget, int n_sink, int window, int compact,
                             int32_t* keep_out, int32_t* freed_pages, void* workspace,
                             size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Keep-list compaction of the paged cache: move each row's kept slots to the
 * front, release the pages past them, shorten the sequence.
 *
 * Defines ("From sliding window to attention-guided eviction": the §4.2
 * pseudocode evicts every slot outside the keep set; §4.3 step 6 continues
 * generation with only the kept KV): for sequence b with live length
 * S = seq_lens[b] and kv head g, with keep row r = keep[b][g][0..n):
 *   K_g[i], V_g[i]  <- K_g[r[i]], V_g[r[i]]     for i < n, in place
 *   scores[b][g][i] <- scores[b][g][r[i]]       (optional, e.g. the H2O score)
 *   pos_map[b][g][i]<- pos_map[b][g][r[i]]      (optional)
 *   block_table[b][p] = -1 for ceil(n/16) <= p < ceil(S/16), those page ids
 *   listed in freed_pages[b] (-1 padded); seq_lens[b] = n.
 * After kvsel_snapkv_select[_ex] (group-sum mode) this is the compaction of
 * the prompt cache: pass the layer block table as [num_layers][max_pages],
 * seq_lens = S per layer, keep = keep_out with keep_stride = its capacity and
 * keep_count from the options (positions equal slots in a fresh prompt).  The
 * seeds kvsel_snapkv_select_ex writes are already in kept order.
 *
 * Arguments (device pointers unless noted):
 *   kv            both pools (read and written in place).
 *   block_table   int32 [batch][max_pages]; seq_lens int32 [batch] (in/out).
 *   keep          int32 [batch][num_kv_heads][keep_stride]: each row's kept
 *                 SLOTS, strictly ascending, each < S.
 *   keep_count    int32 [batch][num_kv_heads], or NULL: a row's count is then
 *                 the number of entries before its first negative one.
 *                 Every kv head of a sequence must keep the same count (one
 *                 block table serves them all), so the per-head counts of
 *                 SnapKV's union mode are rejected when they differ.
 *   scores        fp32 [batch][num_kv_heads][max_len] or NULL.
 *   pos_map       int32 [batch][num_kv_heads][max_len] or NULL.
 *   max_len       row length of scores / pos_map (>= S when either is given).
 *   freed_pages   int32 [batch][max_pages] or NULL.
 *   workspace     >= kvsel_kv_compact_workspace(batch, num_kv_heads) bytes,
 *                 status word zeroed.
 * Device-detected problems (a count or slot out of range, a row not strictly
 * ascending, counts that differ between kv heads, S beyond the table or
 * max_len) record KVSEL_ERR_BAD_INDEX and leave that sequence untouched; a
 * block-table entry outside the pool records it too and skips that row.
 * Launches: check (one CTA per sequence), move (one per (sequence, kv head)),
 * truncate (one per sequence).
 */
KVSEL_API size_t kvsel_kv_compact_workspace(int batch, int num_kv_heads);
KVSEL_API kvsel_status kvsel_kv_compact(const kvsel_paged_kv* kv, int32_t* block_table, int max_pages,
                                        int32_t* seq_lens, int batch, const int32_t* keep, int keep_stride,
                                        const int32_t* keep_count, float* scores, int32_t* pos_map,
                                        int max_len, int32_t* freed_pages, void* workspace, size_t ws_bytes,
                                        void* stream);

/* ---------------------------------------------------------------------------
 * Block offload priority: decay aging, token -> block fold, per-request
 * percentile, global eviction order.
 *
 * Defines ("Sparse attention x KV-cache offloading: eight questions" §2.1
 * exponential decay, §3.1 token -> block aggregation, §3.2 per-request
 * percentile normalisation, §5.1 fp32 score per block):
 *   if increment: score[t] = fmaf(decay, score[t], increment[t]) (in place)
 *   block i of request r covers tokens [i*block_size, (i+1)*block_size) of r,
 *   valid ones only; its score is the max, the mean, or (TOPP) the mean of
 *   the ceil(top_p * n) largest (top_p * n as an fp32 product) of its n
 *   valid tokens;
 *   PERCENTILE: rank q of the block in its request by (score asc, block asc),
 *   key = fp32(2q + 1) / fp32(2n_r) (correctly rounded); NONE: key = score;
 *   order = all blocks sorted by (key asc, request asc, block asc); the first
 *   ceil(evict_frac * N) (evaluated in double) are written as
 *   (request << 32) | block.
 *
 * Arguments (device pointers unless noted):
 *   token_scores  fp32 [total tokens], requests laid out back to back (CSR).
 *   increment     fp32, same layout, or NULL (no update).
 *   req_offsets   int64 [num_requests + 1] token offsets, non-decreasing.
 *   block_size    1..256 tokens; at most 2^30 blocks per request.  With the
 *                 percentile, requests of up to 16384 blocks are ranked in
 *                 shared memory, larger ones by one CTA sorting the request
 *                 through the workspace (about 12 us per 8192 blocks and
 *                 digit pass, four passes: meant for token-level blocks).
 *   agg           KVSEL_AGG_MAX / _MEAN / _TOPP;  norm  KVSEL_NORM_*.
 *   block_score_out  fp32 [max_total_blocks] or NULL: block scores in
 *                 (request, block) order.
 *   max_total_blocks  host-side upper bound on the total block count N.
 *   order_out     int64 [order_capacity]; entries past the evict count are
 *                 not written.
 *   n_out         int64 [2]: the evict count and N (-1 if the lengths were
 *                 rejected on the device).
 * Device-detected problems: N > max_total_blocks or a negative length ->
 * KVSEL_ERR_BAD_INDEX; more than 2^30 blocks in one request ->
 * KVSEL_ERR_UNSUPPORTED; in both cases nothing else is computed.
 */
typedef enum kvsel_block_agg {
  KVSEL_AGG_MAX = 0,
  KVSEL_AGG_MEAN = 1,
  KVSEL_AGG_TOPP = 2,
  KVSEL_AGG_FRAC_HOT = 3, /* fraction of the block's valid tokens with score >= threshold */
  KVSEL_AGG_ALL_COLD = 4  /* the max; only blocks whose max is < threshold may be evicted */
} kvsel_block_agg;
typedef enum kvsel_block_norm { KVSEL_NORM_NONE = 0, KVSEL_NORM_PERCENTILE = 1 } kvsel_block_norm;
KVSEL_API size_t kvsel_block_priority_workspace(int num_requests, int64_t max_total_blocks);
KVSEL_API kvsel_status kvsel_block_priority(float* token_scores, const float* increment, float decay,
                                            const int64_t* req_offsets, int num_requests,
                                            int block_size, int agg, float top_p, int norm,
                                            float evict_frac, float* block_score_out,
                                            int64_t max_total_blocks, int64_t* order_out,
                                            int64_t order_capacity, int64_t* n_out, void* workspace,
                                            size_t ws_bytes, void* stream);

/* Temporal aggregation and block policies beyond kvsel_block_priority
 * ("Sparse attention x KV-cache offloading: eight questions" §2.1: sliding-
 * window average, exponential decay, max pooling over steps; "From sliding
 * window to attention-guided eviction" §5.1: order blocks by their fraction
 * of important tokens, or evict only blocks whose tokens are all cold).
 * kvsel_block_priority_ex takes the arguments of kvsel_block_priority plus
 * `opt` (host pointer; NULL = decay update, threshold unused):
 *   update   KVSEL_UPDATE_DECAY: score[t] = fmaf(decay, score[t], increment[t]);
 *            KVSEL_UPDATE_MAX:   score[t] = max(score[t], increment[t]);
 *            KVSEL_UPDATE_WINDOW: the sum of the last `window` increments,
 *            kept exactly: slot = step % window, score[t] += increment[t] -
 *            history[slot][t], history[slot][t] = increment[t] (the window
 *            average is score / window, which orders blocks the same way).
 *            Every update mode needs `increment`; without it no update runs.
 *   history  fp32 [window][history_tokens] (device), zero before step 0.
 *   window   >= 1; step >= 0; history_tokens >= the total token count, else
 *            KVSEL_ERR_BAD_INDEX is recorded on the device and nothing is
 *            computed.
 *   threshold  AGG_FRAC_HOT / AGG_ALL_COLD: a token is hot when its score is
 *            >= threshold.  With AGG_ALL_COLD the order holds evictable
 *            blocks only and n_out[0] = min(ceil(evict_frac * N), their
 *            count); block_score_out holds the max. */
typedef enum kvsel_score_update {
  KVSEL_UPDATE_DECAY = 0,
  KVSEL_UPDATE_MAX = 1,
  KVSEL_UPDATE_WINDOW = 2
} kvsel_score_update;
typedef struct kvsel_bp_options {
  int update;
  float* history;
  int window;
  int64_t step;
  int64_t history_tokens;
  float threshold;
} kvsel_bp_options;
KVSEL_API kvsel_status kvsel_block_priority_ex(float* token_scores, const float* increment, float decay,
                                               const int64_t* req_offsets, int num_requests,
                                               int block_size, int agg, float top_p, int norm,
                                               float evict_frac, float* block_score_out,
                                               int64_t max_total_blocks, int64_t* order_out,
                                               int64_t order_capacity, int64_t* n_out, void* workspace,
                                               size_t ws_bytes, const kvsel_bp_options* opt, void* stream);

/* ---------------------------------------------------------------------------
 * DSA-style sparse decode: indexer scores, top-k, attention over the
 * selected keys.
 *
 * Defines ("Long context, KV eviction and sparse attention": the DSA
 * paragraph and the sparse-selection section's masked softmax), with S_b the
 * live length after the optional append:
 *   I[b][s]  = sum_j idx_w[b][j] * max(0, idx_q[b][j] . idx_k[b][s]),  s < S_b
 *   sel_b    = the top_k positions by I (ties to the lower position; all of
 *              them when S_b <= top_k), ascending
 *   out[b][h]= softmax_{s in sel_b}(scale * q[b][h] . K_{h/G}[s]) V_{h/G}[s]
 * One selected set per sequence, shared by every q head.
 *
 * Arguments (device pointers):
 *   kv, block_table, max_pages, seq_lens, batch, q, k_new, v_new  as for
 *                 kvsel_decode_attn (seq_lens += 1 when appending).
 *   idx_q         bf16 [batch][num_idx_heads][idx_dim];  idx_w fp32
 *                 [batch][num_idx_heads].
 *   idx_k         bf16 [batch][max_len][idx_dim]: one indexer key per token;
 *                 the appended token's key (idx_k_new, bf16 [batch][idx_dim])
 *                 is written at slot seq_lens[b].  k_new, v_new, idx_k_new are
 *                 all given or all NULL.
 *   num_idx_heads 1..8;  idx_dim 64.
 *   top_k         >= 1;  max_len <= 2^28 (UNSUPPORTED beyond).
 *   out           [batch][num_q_heads][128], bf16 or fp32 (out_dtype).
 *   topk_out      int32 [batch][top_k] or NULL: sel_b, padded with -1.
 *   scores_out    fp32 [batch][max_len] or NULL: I (entries >= S_b untouched).
 *   workspace     >= kvsel_sparse_decode_workspace(kv, batch, max_len, top_k,
 *                 scores_out != NULL) bytes, status word zeroed.
 * Launches: the indexer; the top-k (one 8-CTA thread-block cluster of 1024
 * threads per sequence when max_len <= 262144, 16K-position slices and a
 * final CTA per sequence above that); the attention (the splits of a
 * (sequence, kv head) one cluster).  Each may start while its predecessor
 * finishes and waits for it before reading its results.
 * CUDA graphs: do not capture this call.  Captured with its input and output
 * copies and replayed, these launches have ended in an illegal memory access
 * whose cause is not known; called on a stream, they have not.
 */
KVSEL_API size_t kvsel_sparse_decode_workspace(const kvsel_paged_kv* kv, int batch, int max_len,
                                               int top_k, int with_scores_out);
KVSEL_API kvsel_status kvsel_sparse_decode(const kvsel_paged_kv* kv, const int32_t* block_table,
                                           int max_pages, int32_t* seq_lens, int batch, const void* q,
                                           const void* k_new, const void* v_new, const void* idx_q,
                                           const float* idx_w, void* idx_k, const void* idx_k_new,
                                           int num_idx_heads, int idx_dim, int max_len, int top_k,
                                           float scale, void* out, int out_dtype, int32_t* topk_out,
                                           float* scores_out, void* workspace, size_t ws_bytes,
                                           void* stream);

/* ---------------------------------------------------------------------------
 * SnapKV prefill selection, all layers of one prompt in one call.
 *
 * Defines ("From sliding window to attention-guided eviction" §4.3 steps
 * 2-5): per layer and kv head, the G*W observation rows (the last W prompt
 * queries of each of the kv head's G q heads; window query i is at position
 * S - W + i and attends causally to keys 0..S-W+i) vote for every prefix
 * key j < S - W with the sum of their softmax weights (scale * q . k logits);
 * the votes are max-pooled with a stride-1 window of pool_kernel positions
 * clipped to the prefix; keep = the keep_k best pooled positions (ties to
 * the lower position) followed by the window S-W..S-1, ascending.
 *
 * Arguments (device pointers):
 *   kv            K pool (V is not read); num_q_heads / num_kv_heads = G.
 *   block_table   int32 [num_layers][max_pages]: layer l's prompt pages.
 *   seq_len       prompt length S (host value), obs_window W <= S.
 *   q_obs         bf16 [num_layers][num_q_heads][W][128].
 *   scale         logit scale, > 0 (head_dim^-1/2); else KVSEL_ERR_INVALID_ARG.
 *   pool_kernel   odd, 1..33 (7 in SnapKV).
 *   keep_out      int32 [num_layers][num_kv_heads][keep_k + W]; when
 *                 S - W <= keep_k every position 0..S-1 is kept, -1 padded.
 *   vote_out      fp32 [num_layers][num_kv_heads][S - W] or NULL (raw votes).
 * Limits: G * W <= 256, S < 2^28 (UNSUPPORTED beyond).
 */
KVSEL_API size_t kvsel_snapkv_select_workspace(const kvsel_paged_kv* kv, int num_layers, int seq_len,
                                               int obs_window, int with_vote_out);
KVSEL_API kvsel_status kvsel_snapkv_select(const kvsel_paged_kv* kv, const int32_t* block_table,
                                           int max_pages, int num_layers, int seq_len,
                                           const void* q_obs, int obs_window, float scale,
                                           int pool_kernel, int keep_k, int32_t* keep_out,
                                           float* vote_out, void* workspace, size_t ws_bytes,
                                           void* stream);

/* ---------------------------------------------------------------------------
 * SnapKV selection with the GQA-union keep mode and cold-start seeds.
 *
 * Defines (same section, "KV sharing under GQA", and §2.3 "cold start", the
 * option of prefill attention as the seed score):
 *   KVSEL_SNAP_GROUP_SUM   the selection above (one summed vote per kv head).
 *   KVSEL_SNAP_HEAD_UNION  every q head h votes alone (the sum over its own W
 *                          rows), pools its vote and picks its own keep_k;
 *                          the kv head keeps the union of its G heads' picks
 *                          (ascending), then the window S-W..S-1.
 *   seed of key j (either mode) = the sum over the group's G*W window rows of
 *                          their causal softmax weight on key j, for every
 *                          j < S (window keys included: row i sees keys up to
 *                          S-W+i).  It is the H2O accumulated score the kv
 *                          head would hold had the last W prompt tokens been
 *                          decoded one by one with the same queries, so it can
 *                          initialise H2O's cum or block_priority's token
 *                          scores for the kept cache.
 *
 * Arguments as for kvsel_snapkv_select, plus:
 *   opt           NULL (group sum, no seeds, no counts) or:
 *     mode        kvsel_snap_mode.
 *     keep_count  int32 [num_layers][num_kv_heads] or NULL: valid entries of
 *                 each keep row (keep_k + W, or S when S - W <= keep_k; the
 *                 union's size + W).
 *     seed_out    fp32 or NULL: entry i of (layer l, kv head h) at
 *                 seed_out[l * seed_layer_stride + h * seed_head_stride + i]
 *                 = the seed of position keep[l][h][i] for i < keep_count,
 *                 0 for the padding up to the keep capacity.  The strides
 *                 (elements) must give each row the keep capacity:
 *                 head stride >= capacity, layer stride >= head stride *
 *                 num_kv_heads when num_layers > 1 (else INVALID_ARG).
 *                 Pointing it at a cum buffer seeds the compacted cache.
 *   keep_out      int32 [num_layers][num_kv_heads][capacity], capacity =
 *                 keep_k + W (group sum) or G * keep_k + W (union); -1 padded.
 *   vote_out      group sum: fp32 [num_layers][num_kv_heads][S - W];
 *                 union: fp32 [num_layers][num_q_heads][S - W] (per-head votes).
 *   workspace     >= kvsel_snapkv_select_ex_workspace(kv, num_layers, seq_len,
 *                 obs_window, vote_out != NULL, mode) bytes, status zeroed.
 * Launches: statistics, votes (also the window keys when seeding), pool and
 * select (per q head for the union), plus one union launch.
 */
typedef enum kvsel_snap_mode { KVSEL_SNAP_GROUP_SUM = 0, KVSEL_SNAP_HEAD_UNION = 1 } kvsel_snap_mode;
typedef struct kvsel_snap_options {
  int mode;
  int32_t* keep_count;
  float* seed_out;
  int64_t seed_layer_stride;
  int64_t seed_head_stride;
} kvsel_snap_options;
KVSEL_API size_t kvsel_snapkv_select_ex_workspace(const kvsel_paged_kv* kv, int num_layers, int seq_len,
                                                  int obs_window, int with_vote_out, int mode);
KVSEL_API kvsel_status kvsel_snapkv_select_ex(const kvsel_paged_kv* kv, const int32_t* block_table,
                                              int max_pages, int num_layers, int seq_len,
                                              const void* q_obs, int obs_window, float scale,
                                              int pool_kernel, int keep_k, const kvsel_snap_options* opt,
                                              int32_t* keep_out, float* vote_out, void* workspace,
                                              size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Quest page selection for decode ("Long context, KV eviction and sparse
 * attention", sparse-selection section: a page's logit is bounded by the
 * elementwise min and max of its keys, and the best-bounded pages are kept).
 *
 * Defines, for sequence b (S_b keys once the new token is appended) and q
 * head h (kv head h / G), with Quest pages of 16 tokens whatever the pool's
 * page_size (a pool page of P tokens holds P / 16 of them):
 *   bound[b][h][p] = sum_d max(q_d * kmin[p]_d, q_d * kmax[p]_d), for every
 *                    full page p < S_b / 16 (kmin / kmax over its 16 keys)
 *   pages[b][h]    = the budget_pages largest bounds, ties to the lower page
 *                    (every full page when there are no more), ascending
 *   out[b][h]      = softmax(scale * q . k) V over the tokens of pages[b][h]
 *                    and those of the trailing partial page (always kept)
 * Each q head chooses alone.
 *
 * Page metadata (both calls): page_meta bf16
 * [num_pages][num_kv_heads][page_size / 16][2][128] indexed by PHYSICAL pool
 * page, then the Quest page within it: the min row, then the max row, of that
 * Quest page's keys (its valid keys for a partial page).  kvsel_quest_page_meta fills it for
 * every page 0..ceil(seq_lens[b] / 16) - 1 of each sequence (after a prefill);
 * kvsel_quest_decode keeps it current as it appends.
 *
 * kvsel_quest_page_meta arguments (device pointers): kv (K pool), block_table
 * int32 [batch][max_pages], seq_lens int32 [batch] (not modified), page_meta,
 * status_word: an int32 the kernel records KVSEL_ERR_BAD_INDEX in for a bad
 * length or block-table entry (e.g. the start of a zeroed workspace).
 *
 * kvsel_quest_decode arguments (device pointers):
 *   kv, block_table, max_pages, seq_lens, batch, q, k_new, v_new  as for
 *                 kvsel_decode_attn (k_new / v_new both given or both NULL;
 *                 seq_lens += 1 when appending, published at the end).
 *   page_meta     as above; updated for the appended token's page.
 *   budget_pages  >= 1 full Quest pages per q head (budget / 16 tokens).
 *   out           [batch][num_q_heads][128], bf16 or fp32 (out_dtype).
 *   pages_out     int32 [batch][num_q_heads][budget_pages] or NULL: pages[b][h]
 *                 (Quest page indices), -1 padded.
 *   bounds_out    fp32 [batch][num_q_heads][max_pages * page_size / 16] or
 *                 NULL: bound[b][h][p] for p < S_b / 16 (the rest untouched).
 *   workspace     >= kvsel_quest_decode_workspace(kv, batch, max_pages,
 *                 budget_pages, bounds_out != NULL, pages_out != NULL) bytes,
 *                 zeroed before its first use (it carries counters and page
 *                 masks that every call leaves at zero).
 * Limits: head_dim 128, page_size 16, 32, 64, 128 or 256, G <= 16 (else
 * UNSUPPORTED); max_pages * page_size and num_pages * num_kv_heads *
 * page_size < 2^31.
 * Launches: bounds (+ append), per-head top-k (+ the kv head's page list),
 * attention over the listed pages.
 */
KVSEL_API kvsel_status kvsel_quest_page_meta(const kvsel_paged_kv* kv, const int32_t* block_table,
                                             int max_pages, const int32_t* seq_lens, int batch,
                                             void* page_meta, void* status_word, void* stream);
KVSEL_API size_t kvsel_quest_decode_workspace(const kvsel_paged_kv* kv, int batch, int max_pages,
                                              int budget_pages, int with_bounds_out, int with_pages_out);
KVSEL_API kvsel_status kvsel_quest_decode(const kvsel_paged_kv* kv, const int32_t* block_table,
                                          int max_pages, int32_t* seq_lens, int batch, const void* q,
                                          const void* k_new, const void* v_new, void* page_meta,
                                          int budget_pages, float scale, void* out, int out_dtype,
                                          int32_t* pages_out, float* bounds_out, void* workspace,
                                          size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVSEL_H */
