/*
 * bsattn.h - block-sparse decode attention over a paged KV cache (C ABI).
 *
 * One decode step of one attention layer, for every unit u = (sequence b, KV head
 * h_kv), u = b * n_kv_heads + h_kv:
 *
 *   bs_build_block_summaries  sub-block mean keys kept current as tokens are appended
 *   bs_score_blocks           block scores: mean-key dot products max-pooled over the
 *                             sub-blocks of a block and reduced over the GQA group
 *   bs_select_topk            per-unit block selection: forced sink/local blocks,
 *                             query-aware top-k, NOSA's eviction-driven dual selection
 *   bs_sparse_decode_attn     split-KV flash-decode over the selected blocks only
 *   bs_block_setdiff          blocks added to / removed from the selection since the
 *                             previous step
 *   bs_decode_step            all five for one layer in two launches
 *   bs_block_swap             moves the blocks that the set-difference adds from host
 *                             memory into a GPU block cache (the offload path)
 *   bs_cpu_sparse_attn,       attention of a block subset on the host cores, and the
 *   bs_lse_merge              GPU merge of two partial results (CPU/GPU split)
 *
 * Method sources: "Technisches Resümee: NOSA: Native und Offloadable Sparse
 * Attention" (section Methodik: "1. Algorithmus: NOSA" and "2. System: NOSI") and
 * "Technische Samenvatting: Fluxion" (sections Probleemstelling, Kerninzichten,
 * Systeemcomponenten).
 *
 * Conventions shared by every call
 * --------------------------------
 * Ownership. The caller allocates and owns every buffer. The library allocates
 *   nothing and keeps no state between calls; the persistent state of a decode loop
 *   (summaries, alive mask, previous selection) lives in caller buffers.
 * Memory spaces. Struct arguments (bs_dims, bs_kv, bs_head_cfg) are HOST structs
 *   passed by pointer; every array they point to, and every array argument, is
 *   DEVICE memory unless the parameter says otherwise.
 * Asynchrony. Each call validates its host-visible arguments, enqueues kernels on
 *   `stream` and returns. Nothing waits for the GPU.
 * Errors. Host-detected problems (null pointers, bad shapes, misalignment, a too
 *   small workspace) return a non-zero bs_status before anything is enqueued.
 *   A failed launch returns BS_ERR_CUDA. Problems only the device can see (a page
 *   index outside the pool, a per-unit configuration that breaks a rule below, a
 *   capacity overflow, a bounded wait that ran out) store the first such code into
 *   `*dev_status` (an int32 device word the caller zeroes; atomicCAS from 0) and the
 *   offending unit's work is skipped, never performed out of bounds. Read it after
 *   synchronising.
 * Determinism. Results are bitwise reproducible run to run (no floating-point
 *   atomics; partials merge in a fixed order). Selections never depend on the other
 *   units of the batch; attention outputs depend on them only through the attention's
 *   plan (bs_sparse_decode_attn), in the last bits.
 *
 * Data layout (dims below are the fields of bs_dims)
 * ----------------------------------------------------
 *   K, V pools     [n_pages][page_size=16][head_dim], kv_dtype; 16-byte aligned base.
 *   page_table     int32 [units][max_pages_per_unit]; entry p of unit u is the
 *                  physical page holding tokens [16p, 16p+16) of that unit.
 *   seq_lens       int32 [batch]; T = tokens in the cache including the current
 *                  decode token, which sits at position T-1.
 *   q              [batch][n_q_heads][head_dim], q_dtype; query heads
 *                  [h_kv*G, (h_kv+1)*G) share KV head h_kv (G = n_q_heads/n_kv_heads).
 *   summaries      float32; unit u's sub-block j occupies
 *                  summaries[sum_off[u] + j*head_dim ... + head_dim).
 *   scores         float32 [units][max_blocks_per_unit].
 *   evict_logits   float32 [units][max_blocks_per_unit] (dual units only).
 *   alive          uint8   [units][max_blocks_per_unit] (dual units only; start at 1).
 *   sel_idx        int32   [units][max_sel_per_unit], ascending, padded with -1.
 *   sel_cnt        int32   [units].
 *   out            float32 [batch][n_q_heads][head_dim];  lse float32 [batch][n_q_heads].
 */
#ifndef BSATTN_H_
#define BSATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. NULL selects the legacy default stream. */
typedef struct CUstream_st *bs_stream_t;

typedef enum {
  BS_OK = 0,
  BS_ERR_INVALID_ARG = 1,   /* null pointer, value out of its documented range */
  BS_ERR_SHAPE = 2,         /* unsupported head_dim, group size or page size */
  BS_ERR_ALIGN = 3,         /* a pointer or offset breaks its alignment rule */
  BS_ERR_CAPACITY = 4,      /* a buffer or row is too small for the data */
  BS_ERR_CUDA = 5,          /* a CUDA launch failed */
  BS_ERR_DEVICE_BOUNDS = 6, /* (device) a page index outside the pool or table */
  BS_ERR_TIMEOUT = 7        /* (device) a bounded wait ran out */
} bs_status;

typedef enum { BS_BF16 = 0, BS_FP32 = 1 } bs_dtype;

/* Head classes (Fluxion, Kerninzichten item 2: streaming vs retrieval heads;
 * NOSA, Dual-Selection-Mechanismus: query-aware plus query-agnostic selection). */
typedef enum { BS_STREAMING = 0, BS_RETRIEVAL = 1, BS_DUAL = 2 } bs_head_class;

/* How the G query heads of a group combine their max-pooled block scores
 * (Fluxion, Systeemcomponenten: GQA handled at group level). */
typedef enum { BS_GROUP_MAX = 0, BS_GROUP_MEAN = 1 } bs_group_reduce;

/* Shapes and capacities, host struct. Supported: head_dim 64 or 128, page_size 16,
 * G = n_q_heads / n_kv_heads in 1..8, max_blocks_per_unit <= 16384, and pools of at
 * most (2^31 - 1) / 16 pages (pool rows are signed 32-bit tensor-map coordinates);
 * larger values return BS_ERR_CAPACITY. */
typedef struct {
  int32_t batch, n_q_heads, n_kv_heads, head_dim, page_size;
  int32_t max_pages_per_unit;        /* page-table row length */
  int32_t max_blocks_per_unit;       /* row length of scores / evict_logits / alive */
  int32_t max_sel_per_unit;          /* row length of sel_idx and of setdiff outputs */
  int32_t max_subs_per_unit;         /* upper bound on ceil(T/s) over units (grid sizing) */
  int32_t max_gather_pages_per_unit; /* upper bound on pages covered by a selection */
  int64_t n_pages;                   /* pages in each of the K and V pools */
  bs_dtype kv_dtype, q_dtype;
} bs_dims;

/* Paged KV cache: device pointers. */
typedef struct {
  const void *k_pool, *v_pool;
  const int32_t *page_table;
  const int32_t *seq_lens;
} bs_kv;

/* Per-unit head properties, struct of arrays of length batch * n_kv_heads, device
 * memory (host memory for bs_check_head_cfg only). These are the outputs of the
 * pages' head-property predictor and granularity-budget selector, taken as inputs.
 * Rules (checked by bs_check_head_cfg on the host and by every kernel on the device):
 *   cls in {STREAMING, RETRIEVAL, DUAL};  g % 16 == 0;  g % s == 0 and g/s a power
 *   of two <= 64;  k >= 0;  0 <= k_e <= k (k_e used by DUAL units only);
 *   sink_tokens >= 0;  local_tokens >= 1 (the current token is always attended);
 *   sum_off % 4 == 0 (16-byte aligned summary rows); sum_rows >= ceil(T/s).
 * Selection: forced blocks F = [0, ceil(sink/g)) U [floor(max(0,T-local)/g), ceil(T/g));
 * candidates C = complete blocks outside F; streaming: S = F; retrieval: S = F plus
 * the k best of C; dual: S = F plus Gamma_e (k_e best alive blocks of C by eviction
 * logit) plus Gamma_q (k - k_e best of C minus Gamma_e by score). Ties go to the
 * lower block index. */
typedef struct {
  const int32_t *cls, *block_tokens, *sub_tokens, *k_total, *k_evict;
  const int32_t *sink_tokens, *local_tokens;
  const int64_t *sum_off;   /* float offset of unit u's first summary row */
  const int32_t *sum_rows;  /* summary rows reserved for unit u */
} bs_head_cfg;

/* Host-side check of a head configuration whose nine arrays are in HOST memory.
 * `seq_lens_host` (length batch) are the largest lengths the caller will use.
 * Returns BS_OK or the first rule broken (BS_ERR_INVALID_ARG, BS_ERR_ALIGN,
 * BS_ERR_CAPACITY). Launches nothing. */
bs_status bs_check_head_cfg(const bs_dims *dims, const bs_head_cfg *cfg_host,
                            const int32_t *seq_lens_host);

/* a1. Sub-block key summaries.
 * NOSA, "Blockweise Implementierung": mean pooling inside sub-blocks is the first
 * stage of the two-stage pooling; NOSI fuses the pooling with the KV write.
 * For each unit of sequence b, recomputes every sub-block j that holds a token of
 * [tok_begin[b], seq_lens[b]): kbar_j = (1/n_j) sum of K[t] over the n_j tokens of
 * [j*s, min((j+1)*s, T)), summed in token order in fp32. A decode step passes
 * tok_begin = T-1 (one sub-block per unit); a prefill passes 0. The result does not
 * depend on how the range was split across calls.
 * tok_begin: device int32 [batch]. max_new_tokens (host): an upper bound on
 * seq_lens[b] - tok_begin[b], used only to size the grid. */
bs_status bs_build_block_summaries(const bs_dims *dims, const bs_kv *kv, const bs_head_cfg *cfg,
                                   const int32_t *tok_begin, int32_t max_new_tokens,
                                   float *summaries, int32_t *dev_status, bs_stream_t stream);

/* a2. Block scores.
 * NOSA, "Blockweise Implementierung": max pooling at block level over the sub-block
 * means; Fluxion, "Granularity-Budget Selector": one selection per GQA group.
 * For every retrieval or dual unit and every candidate block c:
 *   S[c] = reduce_{h in group} max_{j in sub-blocks of c} (q_h . kbar_j) / sqrt(d),
 * reduce = max (BS_GROUP_MAX) or mean (BS_GROUP_MEAN). Entries of the row outside
 * the candidate range are written as -inf; rows of streaming units are not touched. */
bs_status bs_score_blocks(const bs_dims *dims, const void *q, const bs_head_cfg *cfg,
                          const int32_t *seq_lens, const float *summaries,
                          bs_group_reduce group_reduce, float *scores, int32_t *dev_status,
                          bs_stream_t stream);

/* a3. Block selection.
 * Fluxion, Kerninzichten item 2 (streaming vs retrieval heads, per-head budget and
 * granularity); NOSA, Dual-Selection-Mechanismus (Gamma_q, Gamma_e and the strict
 * eviction rule: a block of C that is not in Gamma_e is marked dead in `alive` and
 * never enters Gamma_e again) and ED-DMA (selection on pre-exponential logits).
 * Writes S of every unit, ascending, into sel_idx (padded with -1) and |S| into
 * sel_cnt. evict_logits and alive may be NULL when no unit is DUAL (a DUAL unit
 * with NULL arrays reports BS_ERR_INVALID_ARG on the device). Scores and logits are
 * compared exactly as float32 order keys. */
bs_status bs_select_topk(const bs_dims *dims, const bs_head_cfg *cfg, const int32_t *seq_lens,
                         const float *scores, const float *evict_logits, uint8_t *alive,
                         int32_t *sel_idx, int32_t *sel_cnt, int32_t *dev_status,
                         bs_stream_t stream);

/* a4. Sparse decode attention.
 * Fluxion, Probleemstelling item 1 (sparse attention over the selected KV blocks)
 * and Kerninzichten item 3 (bound by data movement). For each query head h of unit
 * u, over the tokens U of the selected blocks (each clipped to t < T):
 *   out_h = sum_t softmax_t(x_h(t)) V[t],  lse_h = log sum_t exp(x_h(t)),
 *   x_h(t) = q_h . K[t] / sqrt(d) + e[u][t / g]  (e = 0 when evict_bias is NULL).
 * evict_bias (device fp32 [units][max_blocks_per_unit], or NULL for plain softmax)
 * is the ED-DMA variant (NOSA, "ED-DMA": blocks are chosen on the eviction head's
 * pre-exponential logits and the exponential is applied only in the attention; here
 * read as each block's logit added to the attention logit of each of its tokens, so
 * exp(e) weights the block's tokens). Entries must be finite or -inf; a block at -inf
 * drops out, and a unit whose tokens all drop out gets a zero row and lse = -inf. Only
 * the entries of selected blocks are read.
 * Split-KV: a unit's gathered pages are cut into contiguous pieces; each piece keeps an
 * fp32 online softmax and the partials are merged by log-sum-exp in a fixed order, so
 * the result does not depend on timing. Two plans, chosen from the dims:
 *   - cluster mode (max_gather_pages_per_unit <= 1024 with at most 19 units, at least
 *     304 units, or max_gather_pages_per_unit <= 256): every unit gets S splits, S the
 *     largest power of two <= 16 with units * S <= two CTAs per SM; the S CTAs of a
 *     unit form one thread-block cluster and merge through distributed shared memory;
 *     split j takes pages [j*p, (j+1)*p), p = ceil(pages / S);
 *   - workspace mode (the rest): each unit's splits are sized by its own page count,
 *     p = max(4 * ceil(pages / 128), m) pages per split (m = 24, or 4 when
 *     max_gather_pages_per_unit > 1024), so at most 32 splits; partials go through the
 *     workspace and the last split to finish merges them. In the fused step
 *     (bs_decode_step) only the splits that can hold pages take part: at most
 *     ceil(min(n_blk, |forced| + k_total) * block_tokens / 16 / m) when m = 24 (the
 *     others leave at once; the merge is the same, as their records were empty).
 * A unit's plan depends on its own sizes only, so a sub-batch launched with the same S
 * gives bitwise the same per-unit results as the full batch.
 * workspace: device scratch of at least bs_workspace_size(dims) bytes, 16-byte
 * aligned. It starts with four int32 words per unit (padded to 16 bytes): the fused
 * step's selection tickets, the attention's arrival tickets, the fused step's published
 * selections and the epochs of the last ones taken. These must be zero before the first
 * call: zero the workspace once after allocating it. Every call that completes leaves
 * the tickets zero again; after a call that reported BS_ERR_TIMEOUT, zero the workspace
 * again. Then, by mode: cluster mode the fused step's page lists (int32 [units]
 * [max_gather_pages_per_unit]); workspace mode 32 split records of G * (head_dim + 4)
 * floats per unit. The rest is overwritten per call.
 * Calls that share a workspace must not run concurrently. */
bs_status bs_sparse_decode_attn(const bs_dims *dims, const void *q, const bs_kv *kv,
                                const bs_head_cfg *cfg, const int32_t *sel_idx,
                                const int32_t *sel_cnt, const float *evict_bias, float *out, float *lse,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                bs_stream_t stream);

/* a4, without a workspace argument. The pages have no counterpart of this call; it
 * exists for callers that cannot allocate device memory for a workspace: a plugin
 * inside a host engine that owns every allocation and offers no allocator, or a
 * serving loop that may not call cudaMalloc once it runs (the call synchronises the
 * device and can fail under memory pressure). Same inputs, outputs and results as
 * bs_sparse_decode_attn, but the workspace it would take (arrival counters and, for
 * selections above 1024 pages per unit, split partials) lives in a fixed 8 MiB array
 * inside this library's device memory, which every GPU that loads the library keeps
 * until the process exits.
 * Limit: bs_workspace_size(dims) must not exceed 8 MiB; larger dims return
 * BS_ERR_CAPACITY before anything is enqueued. In workspace mode the split records
 * take 67.6 KB per unit at head_dim 128, G = 4: at most 124 units (62 at G = 8); in
 * cluster mode (counters and page lists, 16 + 4 * max_gather_pages_per_unit bytes per
 * unit) 2,040 units at 1024 pages per unit.
 * The first call on each device looks up the array's device address with that device
 * current and caches it; make that first call before any stream capture. The cached
 * address belongs to the device's context at that time: after cudaDeviceReset (or
 * anything else that destroys and re-creates the device's primary context) it is stale,
 * so do not call this entry point again in that process.
 * Every call clears the arrival counters on `stream` before its kernel. All calls
 * share the one array per device, so calls whose kernels overlap on the GPU (on
 * different streams, or from different threads) race and corrupt each other's
 * results; serialise them. Allocates nothing: no cudaMalloc, cudaFree or allocating
 * library routine. */
bs_status bs_sparse_decode_attn_noalloc(const bs_dims *dims, const void *q, const bs_kv *kv,
                                        const bs_head_cfg *cfg, const int32_t *sel_idx,
                                        const int32_t *sel_cnt, const float *evict_bias, float *out,
                                        float *lse, int32_t *dev_status, bs_stream_t stream);

/* a5. Set-difference of selections.
 * NOSA, "2. System: NOSI": set-difference kernels drive block swapping.
 * added = cur \ prev and removed = prev \ cur per unit, both ascending, padded with
 * -1 to max_sel_per_unit; counts in added_cnt / removed_cnt. prev_cnt[u] = 0 gives
 * added = cur (first step). Input lists must be ascending and duplicate-free. */
bs_status bs_block_setdiff(const bs_dims *dims, const int32_t *prev_idx, const int32_t *prev_cnt,
                           const int32_t *cur_idx, const int32_t *cur_cnt, int32_t *added,
                           int32_t *added_cnt, int32_t *removed, int32_t *removed_cnt,
                           int32_t *dev_status, bs_stream_t stream);

/* Buffers of one decode step of one layer for bs_decode_step (device pointers). */
typedef struct {
  const void *q;              /* [batch][n_q_heads][head_dim], q_dtype */
  float *summaries;           /* as for bs_build_block_summaries; the sub-block holding T-1 is rewritten */
  float *scores;              /* [units][max_blocks_per_unit] scratch: this step's candidate scores */
  const float *evict_logits;  /* [units][max_blocks_per_unit]; may be NULL when no unit is DUAL */
  uint8_t *alive;             /* [units][max_blocks_per_unit], in/out; may be NULL when no unit is DUAL */
  const float *evict_bias;    /* the attention's ED-DMA block logits, as for bs_sparse_decode_attn (NULL:
                                 plain softmax); may be evict_logits itself */
  const int32_t *prev_idx, *prev_cnt;  /* previous step's selection (prev_cnt 0 at the first step) */
  int32_t *cur_idx, *cur_cnt;          /* this step's selection (written); must not alias prev */
  int32_t *added, *added_cnt, *removed, *removed_cnt;  /* set-difference (written) */
  float *out, *lse;           /* attention output (written) */
  void *workspace;            /* as for bs_sparse_decode_attn: bs_workspace_size bytes, counters zeroed once */
  size_t workspace_bytes;
  int32_t *dev_status;
} bs_step_io;

/* One decode step of one layer: a1, a2, a3, a4 and a5 in two launches (three in the
 * attention's workspace mode when a unit can have more than 2048 candidate blocks;
 * bs_decode_step_launches says which).
 * The results are those of bs_score_blocks, bs_select_topk, bs_sparse_decode_attn and
 * bs_block_setdiff called in that order, plus the a1 update of the one sub-block that
 * holds token T-1 (call bs_build_block_summaries first if more than one token was
 * appended since the last step). Only the order of fp32 additions inside the
 * attention may differ from the separate calls (streaming units split their pages
 * differently), which stays within rounding.
 * Launch 1 scores every candidate tile (one or several 64-row tiles per CTA); the
 * unit's first CTA also updates a1 (that sub-block lies in the forced tail block,
 * which no score of this step reads); the unit's CTA that finishes last (an arrival
 * ticket) selects, publishes the selection (once the row and the page list are
 * written, cur_cnt receives the count and the unit's published word in the workspace
 * receives (epoch << 16) | count with a release store, the epoch one past the one the
 * attention last took, so a count left from an earlier step can never be taken for
 * this step's) and writes the set-difference. Launch 2 is the attention, launched as a
 * programmatic dependent: streaming units' pages need no selection and are attended
 * before launch 1 ends; the others wait, bounded, for their unit's published word.
 * With three launches: launch 1 scores the tiles of all units as one stream in equal
 * shares over a persistent grid; launch 2 runs one 1024-thread CTA per unit that
 * updates a1, waits for launch 1 (streaming units do not wait), selects, publishes and
 * writes the set-difference; launch 3 is the attention as above.
 * The launches may begin before the work ahead of them in `stream` has finished;
 * before waiting for it they read only the per-unit head configuration (cfg arrays),
 * so those must not be written by the kernel immediately before this call. Everything
 * else is read after that work has finished. Requires max_sel_per_unit <= 4096.
 * Errors as for the separate calls; after BS_ERR_TIMEOUT zero the workspace again. */
bs_status bs_decode_step(const bs_dims *dims, const bs_kv *kv, const bs_head_cfg *cfg, const bs_step_io *io,
                         bs_group_reduce group_reduce, bs_stream_t stream);

/* ------------------------------------------------------------------------------
 * Set-difference-driven block swap into a GPU block cache ("Technisches Resümee:
 * NOSA", Methodik / 2. System: NOSI: the KV cache in minimal block units, set-
 * difference kernels for block swapping, host-to-device transfer kernels over
 * Unified Virtual Addressing; Lokalitätsgarantie: blocks kept from one step to the
 * next stay in the GPU cache).
 *
 * The full KV lives in host memory; the GPU holds, per unit, `slots_per_unit` block
 * slots of `pages_per_slot` pages each (pages_per_slot >= g/16 of every unit). A
 * block is resident exactly while it is selected: after the swap of a step, the
 * cached blocks of unit u are that step's selection.
 * ------------------------------------------------------------------------------ */

/* Host-resident paged KV. The pools must be pinned host memory that the device can
 * read (under unified addressing the host pointer of cudaHostAlloc / cudaHostRegister
 * memory is that device pointer); `page_table` is DEVICE memory. */
typedef struct {
  const void *k_pool, *v_pool;   /* [n_pages][16][head_dim], kv_dtype, 16-byte aligned */
  const int32_t *page_table;     /* [units][max_pages_per_unit]: host page of each logical page */
  int64_t n_pages;
} bs_host_kv;

/* GPU block cache (all device memory). Slot s of unit u owns device pages
 * (u * slots_per_unit + s) * pages_per_slot + p, p < pages_per_slot, in `k_pool` and
 * `v_pool` ([units * slots_per_unit * pages_per_slot][16][head_dim]). `page_table`
 * ([units][max_pages_per_unit]) maps each logical page of a cached block to its
 * device page and every other entry to -1; with it and the cache pools, bs_kv
 * describes the cache for bs_sparse_decode_attn. slot_block / block_slot are the
 * cache state (in/out; start with all -1). */
typedef struct {
  void *k_pool, *v_pool;
  int32_t *page_table;          /* [units][max_pages_per_unit] */
  int32_t *slot_block;          /* [units][slots_per_unit]: block held by a slot, -1 free */
  int32_t *block_slot;          /* [units][max_blocks_per_unit]: slot of a block, -1 not cached */
  int32_t slots_per_unit;       /* 1..4096, at least the largest selection */
  int32_t pages_per_slot;       /* >= g/16 of every unit */
} bs_block_cache;

/* One step's swap for every unit: first every block of `removed` leaves the cache
 * (its slot is freed, its page-table entries become -1); then the blocks of `added`
 * (ascending) take the free slots in ascending slot order, their page-table entries
 * are set, and the pages of each added block that hold tokens (< T) are copied, K and
 * V, from the host pools into the block's slot (16-byte loads over the host link, no
 * staging copy). The page holding token T-1 (the token appended this step) is copied
 * and mapped too when its block was already cached, so the cache stays current as the
 * tail block grows. `added` / `removed` and their counts are bs_block_setdiff's output
 * (or bs_decode_step's); seq_lens (device, [batch]) give T. Two launches: the
 * bookkeeping (one CTA per unit), then the copies (one CTA per added block and one
 * per unit for the appended token's page).
 * Device-side errors: a block index outside [0, max_blocks_per_unit) or a host page
 * outside the host pool sets BS_ERR_DEVICE_BOUNDS (that block is skipped); more added
 * blocks than free slots sets BS_ERR_CAPACITY (the excess is not cached). */
bs_status bs_block_swap(const bs_dims *dims, const bs_head_cfg *cfg, const int32_t *seq_lens,
                        const bs_host_kv *host, const bs_block_cache *cache, const int32_t *added,
                        const int32_t *added_cnt, const int32_t *removed, const int32_t *removed_cnt,
                        int32_t *dev_status, bs_stream_t stream);

/* ------------------------------------------------------------------------------
 * CPU/GPU split attention ("Technische Samenvatting: Fluxion", Kerninzichten item 3:
 * sparse attention is bound by data movement; Systeemcomponenten: the CPU and the GPU
 * serve one step in parallel). A unit's selection may be split into two block subsets:
 * one attended on the GPU (bs_sparse_decode_attn, e.g. over the block cache), the
 * other on the host cores over host-resident KV (bs_cpu_sparse_attn); bs_lse_merge
 * combines the two partial results into the attention over the union.
 * ------------------------------------------------------------------------------ */

/* Host copies of the tables the CPU side reads (all HOST memory). */
typedef struct {
  const int32_t *page_table;    /* [units][max_pages_per_unit]: host page of each logical page */
  const int32_t *seq_lens;      /* [batch]: T */
  const int32_t *block_tokens;  /* [units]: g */
  const float *evict_bias;      /* NULL, or the ED-DMA block logits [units][max_blocks_per_unit] as for
                                   bs_sparse_decode_attn */
  int32_t max_blocks_per_unit;  /* row length of evict_bias (used only when it is set) */
} bs_host_tables;

/* Attention of each unit's listed blocks (tokens clipped to T) on the host cores,
 * fp32 arithmetic, units spread over n_threads threads; synchronous. Everything is
 * HOST memory: q ([batch][n_q_heads][head_dim], q_dtype), the pools of `kv` (its
 * page_table field is not used; `tables` gives the host page table), sel_idx
 * ([units][max_sel_per_unit], ascending), sel_cnt ([units]), out ([batch][n_q_heads]
 * [head_dim] fp32) and lse ([batch][n_q_heads] fp32, natural log; -inf and a zero row
 * for a unit with nothing to attend). Returns BS_ERR_DEVICE_BOUNDS (after finishing
 * the other units) if a block or page index is out of range. */
bs_status bs_cpu_sparse_attn(const bs_dims *dims, const void *q, const bs_host_kv *kv, const bs_host_tables *tables,
                             const int32_t *sel_idx, const int32_t *sel_cnt, float *out, float *lse,
                             int n_threads);

/* out, lse = the log-sum-exp merge of two partial attention results over disjoint
 * token sets of every query head (device memory, layout of out / lse above): with
 * M = max(lse_a, lse_b), w = exp(lse - M), out = (w_a o_a + w_b o_b) / (w_a + w_b) and
 * lse = M + log(w_a + w_b); a side with lse = -inf contributes nothing, and two
 * empty sides give a zero row and -inf. out / lse may be out_a / lse_a (in place). */
bs_status bs_lse_merge(const bs_dims *dims, const float *out_a, const float *lse_a, const float *out_b,
                       const float *lse_b, float *out, float *lse, bs_stream_t stream);

/* Bytes of workspace bs_sparse_decode_attn needs for these dims (0 on bad dims). */
size_t bs_workspace_size(const bs_dims *dims);

/* Kernels one bs_decode_step call launches for these dims (each a programmatic
 * dependent of the one before), or 0 on bad dims. Host only; launches nothing. */
int bs_decode_step_launches(const bs_dims *dims);

/* Every wait inside a kernel (for a bulk copy to land, for the fused step's selection
 * to be published) gives up after a wall-clock limit, reports BS_ERR_TIMEOUT in the
 * status word and lets the kernel finish. This sets that limit, in nanoseconds, for the
 * kernels launched from now on (those already captured in a CUDA graph keep the limit
 * they were captured with); 1000 ns .. 60 s, default one second. Returns
 * BS_ERR_INVALID_ARG (and keeps the old limit) outside that range. Process-wide; host
 * only. */
bs_status bs_set_wait_limit_ns(uint64_t limit_ns);

/* The current limit of device-side waits, in nanoseconds. */
uint64_t bs_wait_limit_ns(void);

/* Static text for a status code. */
const char *bs_status_string(bs_status status);

#ifdef __cplusplus
}
#endif

#endif /* BSATTN_H_ */
