/*
 * fi.h -- C ABI of the GB300 (sm_103a) paged serving-attention library.
 *
 * The library computes attention over a block-sparse-row (BSR) paged KV-cache
 * for batch decode and ragged causal prefill, under a deterministic
 * load-balanced split-KV plan whose partial attention states (O, LSE) are
 * merged in-kernel.  Source: page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎"
 * (digest of the MLSys 2025 FlashInfer paper), sections cited per call below.
 *
 * Conventions for every call
 *   - Plain C types only.  `stream` is a cudaStream_t passed as void*
 *     (NULL = the legacy default stream).
 *   - Device pointers point to memory of the current CUDA device; host
 *     pointers to ordinary or pinned host memory, as stated per argument.
 *   - bf16 tensors are IEEE bfloat16 bit patterns (2 bytes each), row-major,
 *     densely packed:
 *        q, o       [total_q, num_qo_heads, head_dim]       (ragged rows, qo_indptr)
 *        k_pages,
 *        v_pages    [num_pages, num_kv_heads, page_size, head_dim]   ("HND")
 *        lse        float32 [total_q, num_qo_heads], natural log, includes the
 *                   softmax scale: lse = log sum_j exp(q.k_j / sqrt(head_dim)).
 *     Query head h reads KV head h / (num_qo_heads / num_kv_heads).
 *   - Every call returns an fi_status; 0 is success.  Nothing aborts,
 *     throws or exits across this boundary.  On a host-side error no output
 *     and no workspace state is changed.
 *   - head_dim must be 128.
 *   - One workspace holds exactly one plan at a time: fi_plan and
 *     fi_plan_composable replace it (a composable plan's shared and
 *     per-request parts are one plan with one reduction map).  The plan, its
 *     page-index copy, split counters and partial-output slots live in the
 *     workspace's fixed segments, so a launch captured in a CUDA graph keeps
 *     valid pointers across re-plans (核心机制 7, App. D.1); a second live plan
 *     would need a second set of segments.  A caller that keeps several plans
 *     live (e.g. the prefill and the decode batch of one step) creates one
 *     workspace per plan.
 */
#ifndef FI_H_
#define FI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fi_status {
  FI_OK = 0,
  FI_ERR_INVALID_ARG = 1, /* malformed indptr / lengths / pointers / sizes */
  FI_ERR_CAPACITY = 2,    /* batch, tokens or pages exceed the workspace's capacity */
  FI_ERR_UNSUPPORTED = 3, /* head_dim != 128, heads not divisible, page size the path can't tile */
  FI_ERR_CUDA = 4,        /* a CUDA runtime call failed (the message is in fi_last_error_message) */
  FI_ERR_DEVICE = 5,      /* a device-side check tripped (see fi_get_error) */
  FI_ERR_NO_PLAN = 6      /* fi_run before a successful fi_plan on this workspace */
} fi_status;

/* Page layouts of k_pages / v_pages (fi_workspace_set_variant). */
#define FI_KV_LAYOUT_HND 0 /* [num_pages, num_kv_heads, page_size, head_dim] */
#define FI_KV_LAYOUT_NHD 1 /* [num_pages, page_size, num_kv_heads, head_dim] */

/* Element types of k_pages / v_pages (fi_workspace_set_kv_dtype). */
#define FI_KV_DTYPE_BF16 0 /* bfloat16 */
#define FI_KV_DTYPE_E4M3 1 /* fp8 e4m3 codes (1 byte), one scale per tensor */

/* Device-side error bits reported by fi_get_error. */
#define FI_DEVERR_PAGE_OOB 0x1     /* a page index >= num_pages was skipped */
#define FI_DEVERR_WAIT_TIMEOUT 0x2 /* a pipeline wait gave up after its iteration limit */
#define FI_DEVERR_TMEM 0x4         /* tensor-memory allocation returned an unusable address */

typedef struct fi_workspace fi_workspace;

/*
 * fi_workspace_create -- allocate the workspace once, at maximum capacity.
 *
 * Source: 核心机制 7 "CUDAGraph 兼容的静态化手段" (paper App. D.1, D.3): the
 * workspace is sized for the largest batch up front and its segments keep
 * fixed offsets, so a captured fi_run keeps valid pointers; the number of
 * partial-output tiles is bounded by 2 * #CTA.
 *
 *   max_batch       most requests one plan may hold (>= 1)
 *   max_total_q     most query tokens one plan may hold (>= 1)
 *   max_kv_pages    most entries kv_indices may hold (>= 1)
 *   num_qo_heads, num_kv_heads, head_dim   fixed for the workspace
 *   num_sms         SM budget of the attention kernels; 0 selects every SM of
 *                   the device (App. E: the SMs attention may use are given by
 *                   the user).  Each path runs k persistent CTAs per SM
 *                   (App. D.3: #CTA = k * #SM): k = 1 for decode tiles and for
 *                   the 256-row tensor-core tiles (one CTA holds all 512 TMEM
 *                   columns).
 *   out             receives the handle (owned by the caller; release with
 *                   fi_workspace_destroy)
 *
 * Allocates one device buffer (plan segments, page-index copy, split
 * counters, partial-output slots) and one pinned host buffer of the plan
 * segments, on the current device.  Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
int fi_workspace_create(int max_batch, int max_total_q, int max_kv_pages, int num_qo_heads, int num_kv_heads,
                        int head_dim, int num_sms, fi_workspace** out);

/* Release a workspace (synchronises with its last plan copy first). NULL is a no-op. */
int fi_workspace_destroy(fi_workspace* ws);

/*
 * fi_workspace_set_cost_model -- parameters of the scheduler's tile cost and chunk bound.
 *
 * Source: 核心机制 6 "负载均衡调度" (paper §3.3.1, Alg. 1): cost(l_q, l_kv) =
 * alpha * l_q + beta * l_kv.  l_min is the smallest KV chunk the plan cuts
 * (tokens).  Defaults: alpha = beta = 1, l_min = 256.  Takes effect at the
 * next fi_plan.  Errors: INVALID_ARG (alpha < 0, beta < 1, l_min < 1).
 */
int fi_workspace_set_cost_model(fi_workspace* ws, int64_t alpha, int64_t beta, int32_t l_min);

/*
 * fi_workspace_set_variant -- attention variant for the following fi_plan.
 *
 * Source: 问题背景 挑战二 (paper §1) names sliding-window masks and Grok's logit
 * soft-cap among the variants a serving library must carry, and 核心机制 5
 * (paper §3.2-3.2.3) treats masks, logits transforms and the KV layout as
 * inputs of one attention template.
 *
 *   window_left      -1 for none; else a causal plan's query token t, aligned
 *                    at key position p = l_kv - l_q + t, sees keys p - window_left
 *                    .. p.  The plan reads only the keys windows reach.
 *   logits_soft_cap  0 for none; else the scaled logit x = scale * q.k becomes
 *                    cap * tanh(x / cap) before the softmax.
 *   kv_layout        FI_KV_LAYOUT_HND or FI_KV_LAYOUT_NHD.
 *
 * The variant is fixed into the plan at fi_plan; fi_run uses the plan's.  A
 * window on a non-causal batch makes fi_plan return UNSUPPORTED; so does NHD
 * decode unless the page size is a power of two and num_kv_heads is 1, 2, 4,
 * 8 or 16.  A captured fi_run keeps
 * the variant it was captured with.  Default: none, none, HND.
 * Errors: INVALID_ARG.
 */
int fi_workspace_set_variant(fi_workspace* ws, int32_t window_left, float logits_soft_cap, int32_t kv_layout);

/*
 * fi_workspace_set_kv_dtype -- element type of the KV pages for the following fi_plan.
 *
 * Source: 核心机制 8 (paper App. F): a mixed-precision kernel keeps queries and
 * outputs in 16-bit floats and stores the KV-cache in fp8.  Reading: e4m3
 * codes with one scale per tensor, K = k_scale * code and V = v_scale * code.
 *
 *   kv_dtype          FI_KV_DTYPE_BF16 (default) or FI_KV_DTYPE_E4M3
 *   k_scale, v_scale  > 0; used with e4m3 pages
 *
 * With e4m3, k_pages / v_pages hold one byte per element in the workspace's
 * layout (HND or NHD) and q and o stay bf16.  Decode tiles compute in f16 MMAs
 * with fp32 accumulation and need a power-of-two page size (NHD pages, as for
 * bf16, also a power-of-two H_kv of at most 16).  Tensor-core tiles widen the
 * codes to f16 in shared memory (exactly), convert q to f16 there and run f16
 * MMAs; they take the page sizes of bf16 pages.  Composable plans (fi_plan_composable) take
 * e4m3 HND pages of a power-of-two size.  fi_plan returns UNSUPPORTED
 * otherwise.  NaN codes in the pages give undefined rows.  Errors: INVALID_ARG.
 */
int fi_workspace_set_kv_dtype(fi_workspace* ws, int32_t kv_dtype, float k_scale, float v_scale);

/*
 * fi_plan -- inspector step: compute the work plan for one batch on the CPU.
 *
 * Source: 核心机制 6 (paper §3.3.1, Alg. 1, Fig. 6) and 核心机制 7 (App. D):
 * per generation step the CPU derives lengths, picks the tile, bounds the KV
 * chunk L_kv = sum ceil(l_qo/T_q) * l_kv / #CTA, cuts long work into chunks
 * (short work writes the output directly), sorts work longest-first and
 * hands it out through a CTA priority queue, and records the reduction map of
 * split rows.  The plan is computed into pinned host memory and copied to the
 * workspace with cudaMemcpyAsync on `stream`.  The plan depends only on the
 * lengths, never on kv_indices values: identical lengths give a bit-identical
 * plan.  It may be reused by any number of fi_run calls (e.g. every layer).
 *
 *   qo_indptr      HOST int32 [batch + 1], qo_indptr[0] = 0, non-decreasing
 *   kv_indptr      HOST int32 [batch + 1], kv_indptr[0] = 0, non-decreasing;
 *                  request i owns pages kv_indices[kv_indptr[i] .. kv_indptr[i+1])
 *   kv_indices     HOST int32 [kv_indptr[batch]], page ids >= 0
 *   last_page_len  HOST int32 [batch]; in [1, page_size] for requests with pages
 *   causal         0 = full attention; 1 = query token t of request i sees keys
 *                  j <= l_kv - l_q + t (mask aligned to the end of the KV)
 *   stream         stream of the plan copy; fi_run on another stream must be
 *                  ordered after it by the caller
 *
 * The index arrays are copied: the caller may free or reuse them on return.
 * A new fi_plan replaces the previous plan of the workspace.  Not capturable
 * in a CUDA graph (it waits for the previous plan's copy to finish before
 * reusing the pinned buffer).
 * Errors: INVALID_ARG, CAPACITY, UNSUPPORTED, CUDA.
 */
int fi_plan(fi_workspace* ws, const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
            const int32_t* last_page_len, int batch, int num_qo_heads, int num_kv_heads, int head_dim,
            int page_size, int causal, void* stream);

/*
 * fi_plan_composable -- inspector step for a batch given in composable formats: a shared
 * sub-matrix plus per-request rows, planned together with one reduction map.
 *
 * Source: 核心机制 2 "可组合格式" (paper §3.1.2, Fig. 3): a KV-cache whose requests share a
 * prefix is the sum of two block-sparse matrices over the same query rows: the shared part, whose
 * block rows span all query tokens of a group (Br = the group's tokens), and the per-request part
 * (Br = 1); their attention states combine with ⊕ (术语与记号 "Attention State 与 ⊕", §2.2).
 * 核心机制 6-7 (§3.3.1, App. D): both parts are cut into chunks and queued as one plan whose
 * reduction map spans both formats.
 *
 *   shared_*       HOST int32, as for fi_plan: block row i covers query tokens
 *                  shared_qo_indptr[i] .. shared_qo_indptr[i+1] - 1 (the same token numbering as
 *                  qo_indptr; shared_qo_indptr[shared_batch] <= qo_indptr[batch]) and owns pages
 *                  shared_kv_indices[shared_kv_indptr[i] .. shared_kv_indptr[i+1]).  Every key of a
 *                  block row is visible to all of its tokens.
 *   qo_indptr .. last_page_len, batch, causal   the per-request part, as for fi_plan (causal masks
 *                  align to the end of each request's own KV)
 *
 * Output row t is (state of t over its block row's shared keys) ⊕ (state over its own keys).  The
 * shared part takes 256-row tensor-core tiles and writes every chunk to a partial slot; the
 * per-request part takes decode tiles (every request must have at most 8 rows = query tokens x group
 * size, else UNSUPPORTED), and each of its rows merges its own chunks and the shared slots that hold
 * its rows, in the plan's fixed order.  fi_run then makes two launches, the second chained to the
 * first by programmatic dependent launch.  The workspace's variant must be the default (bf16 HND
 * pages, no window, no soft-cap), else UNSUPPORTED; fi_run_merge with a given state is UNSUPPORTED
 * for these plans.  fi_plan_info reports path 2.  Other behaviour and errors as fi_plan.
 */
int fi_plan_composable(fi_workspace* ws, const int32_t* shared_qo_indptr, const int32_t* shared_kv_indptr,
                       const int32_t* shared_kv_indices, const int32_t* shared_last_page_len, int shared_batch,
                       const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
                       const int32_t* last_page_len, int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                       int page_size, int causal, void* stream);

/*
 * fi_run -- executor step: one persistent kernel (attention + merge of split rows).
 *
 * Source: 核心机制 6-7 (paper §3.3.1, App. D): attention and the contraction
 * of partial outputs run in one persistent kernel of fixed grid; partial
 * states of a split row go to workspace slots and are merged in the order
 * the plan fixed (no atomic aggregation), so outputs are bit-identical from
 * run to run.  Decode tiles (<= 8 rows) run warp-level MMAs with the KV tokens
 * on the MMA's 16-row side (power-of-two page sizes) or CUDA cores (other page
 * sizes); larger requests run 256-row tiles (two 128-row tcgen05 MMA tiles
 * sharing each K/V tile) on the tensor cores (核心机制 4, paper §3.2.2).
 * A decode split row is merged by the last of its chunks to finish; a
 * tensor-core split row by a contraction kernel chained to the attention
 * launch (programmatic dependent launch, one warp per row).  Both sum the
 * chunks in the plan's slot order.
 *
 *   q          DEVICE bf16 [total_q, num_qo_heads, 128]
 *   k_pages    DEVICE bf16 [num_pages, num_kv_heads, page_size, 128]
 *   v_pages    DEVICE bf16, same shape as k_pages
 *   num_pages  rows of the page pool; every planned page id must be below it
 *   o          DEVICE bf16 [total_q, num_qo_heads, 128]   (written)
 *   lse        DEVICE float32 [total_q, num_qo_heads]     (written)
 *
 * Slots of a request's last page past its last token may hold anything (NaN
 * included): no kernel lets them reach an output.
 *
 * Every row of o/lse that the plan covers is written; a row that sees no key
 * gets o = 0, lse = -inf.  Asynchronous on `stream`.  A decode-tile launch is
 * made a programmatic dependent of the previous kernel on the stream: its CTAs
 * may set up shared memory while that kernel drains, and read no global memory
 * before it has completed.  Capturable in a CUDA
 * graph, and a captured launch stays valid for later plans of the same
 * workspace that keep the same path and tile (fi_plan_info header[1..3]) and
 * page size; on the tensor-core path they must also keep the total query count
 * (the launch holds a TMA descriptor of q whose extent is the plan's total_q).
 * Launches over pages of 8 or more tokens hold TMA descriptors of k_pages and
 * v_pages built from the call's pointers, num_pages and page size.
 * Calls that share a workspace must not overlap on the GPU.
 * Errors: NO_PLAN, INVALID_ARG (null pointers, q / k_pages / v_pages not
 * 16-byte aligned, page id >= num_pages), CUDA.
 */
int fi_run(fi_workspace* ws, const void* q, const void* k_pages, const void* v_pages, int num_pages, void* o,
           float* lse, void* stream);

/*
 * fi_run_merge -- fi_run, with each output row merged (⊕) into a given state.
 *
 * Source: 核心机制 2 "可组合格式" (paper §3.1.2, Fig. 3) and 术语与记号
 * "Attention State 与 ⊕" (paper §2.2): the attention of one block-sparse
 * sub-matrix (e.g. per-request suffixes, Br = 1) is combined with the state of
 * another over a disjoint key set (e.g. the shared prefix, Br = #requests).
 * Here the combination is done by the kernel that writes the rows, so no
 * separate merge launch runs.
 *
 *   o_prev    DEVICE bf16 [total_q, num_qo_heads, 128]: the other state's O
 *   lse_prev  DEVICE float32 [total_q, num_qo_heads]: its LSE (natural log;
 *             -inf for a row that saw no key)
 *   o, lse    written with (state of this plan) ⊕ (o_prev, lse_prev); they may
 *             be the same buffers as o_prev / lse_prev (in place)
 * Other arguments, behaviour and errors as fi_run; o_prev and lse_prev are
 * both null (plain fi_run) or both set (else INVALID_ARG).
 */
int fi_run_merge(fi_workspace* ws, const void* q, const void* k_pages, const void* v_pages, int num_pages,
                 const void* o_prev, const float* lse_prev, void* o, float* lse, void* stream);

/*
 * fi_merge_states -- (O, LSE) of two disjoint KV sets merged into one.
 *
 * Source: 术语与记号 "Attention State 与 ⊕" (paper §2.2) and 核心机制 2
 * "可组合格式" (paper §3.1.2, Fig. 3): states over disjoint key sets combine
 * with an associative, commutative operator, so a shared-prefix sub-matrix
 * and a per-request suffix sub-matrix can be computed separately and merged:
 *   s = log(e^s_a + e^s_b),  O = e^(s_a - s) O_a + e^(s_b - s) O_b,
 * with (0, -inf) as the identity.
 *
 *   o_a, o_b, o   DEVICE bf16 [rows, heads, head_dim]   (o may alias o_a or o_b)
 *   lse_a, lse_b, lse   DEVICE float32 [rows, heads], natural log
 * Asynchronous on `stream`.  Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
int fi_merge_states(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o, float* lse,
                    int rows, int heads, int head_dim, void* stream);

/*
 * fi_get_error -- read and clear the workspace's device-side error word
 * (FI_DEVERR_* bits).  Synchronises the device.  Errors: INVALID_ARG, CUDA.
 */
int fi_get_error(fi_workspace* ws, int32_t* err_bits);

/*
 * fi_plan_info -- copy the current plan's 16-int32 header to host memory:
 *   [0] magic 0x46495031  [1] path (0 decode tiles, 1 tensor-core tiles, 2 composable: the
 *                         remaining fields are those of the per-request part)
 *   [2] tokens per tile   [3] rows per tile  [4] group size g  [5] #CTA
 *   [6] work items  [7] split rows  [8] partial slots  [9] L_kv (tokens)
 *   [10] page_size  [11] causal  [12] num_qo_heads  [13] num_kv_heads
 *   [14] head_dim   [15] batch
 * Errors: INVALID_ARG, NO_PLAN.
 */
int fi_plan_info(const fi_workspace* ws, int32_t* header16);

/*
 * fi_plan_compute -- the planner alone, on the host, with no device work.
 *
 * Same inputs and rules as fi_plan (kv_indices is not an input: plans never
 * depend on it), plus the SM budget (num_sms, as for fi_workspace_create), the
 * cost model and the sliding window (window_left, as for
 * fi_workspace_set_variant; -1 for none).  Writes the plan as one
 * flat int32 array:
 *   header[16] | cta_indptr[num_ctas + 1] | items[n_items][8] (queue order)
 *   | split rows[n_split][8] | slot_to_split_row[n_slots]
 * item = {page_base, q_start, q_len, kv_head, kv_lo, kv_hi, diag, slot(-1 = direct)},
 * split row = {first_slot, n_chunks, q_start, q_len, kv_head, 0, 0, 0}.
 *   out       HOST int32 buffer of `capacity` elements (may be NULL to query)
 *   out_len   receives the number of elements the plan needs
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY (out too small; out_len is set).
 */
int fi_plan_compute(const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* last_page_len, int batch,
                    int num_qo_heads, int num_kv_heads, int head_dim, int page_size, int causal, int num_sms,
                    int64_t alpha, int64_t beta, int32_t l_min, int32_t window_left, int32_t* out,
                    int64_t capacity, int64_t* out_len);

/*
 * fi_plan_composable_compute -- the composable planner alone, on the host, with no device work.
 *
 * Inputs as fi_plan_composable (no page ids), with the SM budget and the default cost model.
 * Writes the shared part's plan (as fi_plan_compute lays a plan out, every unit listed), then the
 * per-request part's plan (its header's slot count covers both parts' slots; slot_to_split_row has
 * -1 for the shared slots; unit fields 5 and 6 are the unit's first ext entry and count), then the
 * ext list: per entry {shared slot, (row offset + 512) | (rows of the shared tile << 16)}.  An item
 * whose slot field is -(2 + u) writes its rows directly after merging unit u's ext entries.
 *   out, capacity, out_len   as fi_plan_compute
 * Errors: INVALID_ARG, UNSUPPORTED, CAPACITY.
 */
int fi_plan_composable_compute(const int32_t* shared_qo_indptr, const int32_t* shared_kv_indptr,
                               const int32_t* shared_last_page_len, int shared_batch, const int32_t* qo_indptr,
                               const int32_t* kv_indptr, const int32_t* last_page_len, int batch, int num_qo_heads,
                               int num_kv_heads, int head_dim, int page_size, int causal, int num_sms, int32_t* out,
                               int64_t capacity, int64_t* out_len);

/*
 * fi_decode_noalloc -- the CUDA-core decode path without any allocation.
 *
 * The paper has no counterpart to this call; it exists for callers that
 * cannot allocate device memory or let a library do so (for example a serving
 * runtime that hands the whole GPU to its own memory pool up front, or a
 * plugin host whose allocator the library must not touch).  It plans and runs
 * one batch like fi_plan + fi_run, but needs no workspace: its plan, page-index
 * copy, split counters and partial slots live in one file-scope device array
 * of FI_NOALLOC_SCRATCH_BYTES (4 MiB) that every GPU loading the library holds
 * until the process exits, and the plan is built in static host storage.  It
 * calls no cudaMalloc, cudaFree, cudaHostAlloc or other allocating routine.
 *
 *   index arrays   HOST int32, as for fi_plan (copied; free on return)
 *   q, k_pages, v_pages, o, lse   DEVICE, as for fi_run
 *   stream         the plan copy, the counter reset and the kernel run on it
 *
 * The plan is the one fi_plan makes for the same lengths with the default cost
 * model and every SM of the device (the same planner code, run over static
 * storage), so it is bit-identical to fi_plan's and accepts the same inputs.
 * All calls share the array: calls that overlap on the GPU (different streams
 * without ordering) race; host calls are serialised.  The array keeps the last
 * call's contents, so each call clears its split counters.  Its first 256 bytes
 * hold a device-side error word (FI_DEVERR_* bits) that calls only add to: read
 * and clear it with fi_decode_noalloc_get_error.
 * The first call on a device looks up the array's device address and sets the
 * kernel attribute (with that device current).
 * Errors: INVALID_ARG (also for q / k_pages / v_pages that are not
 * 16-byte aligned), CAPACITY (plan + page indices + slots do not
 * fit in the array), UNSUPPORTED (the batch needs tensor-core tiles, i.e. some
 * request has more than 8 rows = query tokens x group size, or a KV length
 * above 2^30), CUDA.
 */
#define FI_NOALLOC_SCRATCH_BYTES (4u << 20)
int fi_decode_noalloc(const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
                      const int32_t* last_page_len, int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                      int page_size, int causal, const void* q, const void* k_pages, const void* v_pages,
                      int num_pages, void* o, float* lse, void* stream);

/*
 * fi_decode_noalloc_get_error -- read and clear the error word of fi_decode_noalloc's array on the
 * current device (FI_DEVERR_* bits set by every call since the last read; 0 if none).
 * Synchronises the device.  Allocates nothing.  Errors: INVALID_ARG, CUDA.
 */
int fi_decode_noalloc_get_error(int32_t* err_bits);

/* Number of SMs of the current device (the default SM budget). Errors: CUDA. */
int fi_device_sm_count(int* out);

/* Static text for a status code. */
const char* fi_status_string(int status);

/* Text of the last CUDA failure seen by this thread (empty if none). */
const char* fi_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* FI_H_ */
