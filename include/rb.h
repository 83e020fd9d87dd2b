/*
 * rb.h — C ABI of the ragged mixed-batch step library (librb.so), NVIDIA GB300 / sm_103a.
 *
 * One flattened, unpadded forward step over a mixed batch of full prefills, chunked-prefill
 * segments and decodes, for ONE attention layer:
 *
 *   rb_prepare_inputs   persistent batch arrays -> flat step inputs + attention metadata
 *   rb_kv_write         this step's new K/V rows -> paged KV cache (by slot_mapping)
 *   rb_paged_attention  varlen causal GQA attention through the page table
 *   rb_gather_rows      hidden rows at logits_indices (the rows the LM head needs)
 *   rb_step             all four in one call (one memset and two launches)
 *   rb_step_host        rb_step with the caller's host-to-device and device-to-host copies
 *   rb_step_host_async  the same with the copies on streams of their own (pipelined steps)
 *
 * and, before rb_prepare_inputs, the runner's per-step merge of scheduler deltas into the
 * persistent batch:
 *
 *   rb_batch_apply_update  remove, append, install and condense rows on the device
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer named d_* is DEVICE memory on the current CUDA device; the caller owns it,
 *    allocates it and keeps it alive until the work queued on `stream` has finished.  The
 *    library allocates no device memory and never synchronises: each call only enqueues
 *    kernels (and, for rb_prepare_inputs, one 4-byte memset) on `stream`, a cudaStream_t passed
 *    as void* (NULL = the legacy default stream); rb_step_host and rb_step_host_async also
 *    enqueue the caller's copies, the latter on the caller's copy streams with event records
 *    and waits between them.  The one exception to "no device memory" is
 *    the 64 MiB scratch array of rb_paged_attention_static_ws: a static device array of the
 *    library's module, so every GPU that loads the library holds it until the process exits.
 *  - All index arrays are int32.  bf16 tensors are passed as void* holding IEEE bfloat16 bits.
 *  - Host-side checks (null pointers, sizes, alignment, unsupported shapes) run before anything
 *    is enqueued and return a status other than RB_OK; nothing is enqueued then.
 *  - Device-side checks never trap and never spin without limit: a violated precondition sets a
 *    bit (RB_EBIT_*) in a caller-owned int32 error word with atomicOr, the offending access is
 *    skipped or redirected to the null page, and the kernel carries on.  The caller zeroes the
 *    word when it wants a fresh reading (rb_prepare_inputs zeroes its own) and reads it after
 *    the step.  Results are unspecified where a bit was set.
 *  - RB_ERR_CUDA means a CUDA runtime call failed (for example a launch error); the failing
 *    call's cudaError_t can be read with cudaGetLastError().
 *
 * Page layout (per layer, K and V separate tensors): [num_blocks * block_size, nkv, head_dim]
 * bf16, i.e. row `slot` holds the K (or V) of one token for all kv heads; slot =
 * page_id * block_size + offset ("vLLM 源码完全拆解（五）…", "Block table 是逐请求的页表";
 * nano-vLLM's per-layer cache [num_blocks, block_size, kv_heads, head_dim]).
 */
#ifndef RB_H_
#define RB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rb_status {
  RB_OK = 0,
  RB_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size, misaligned buffer */
  RB_ERR_CAPACITY = 2,    /* a size exceeds a capacity given in rb_dims or the workspace */
  RB_ERR_CUDA = 4,        /* a CUDA runtime call failed */
  RB_ERR_UNSUPPORTED = 5  /* a shape this build has no kernel for */
} rb_status;

/* Device error-word bits (atomicOr'ed; see the conventions above). */
#define RB_EBIT_NUM_SCHEDULED 0x001 /* a real request has num_scheduled < 1 */
#define RB_EBIT_NUM_COMPUTED 0x002  /* a real request has num_computed < 0 */
#define RB_EBIT_SEQ_LEN 0x004       /* num_computed + num_scheduled > max_model_len, or it
                                       needs more pages than max_blocks_per_req */
#define RB_EBIT_TOKEN_SUM 0x008     /* sum of num_scheduled != num_tokens */
#define RB_EBIT_BLOCK_ID 0x010      /* a page id read for a real token is outside
                                       [0, num_blocks) or is the null page */
#define RB_EBIT_SLOT 0x020          /* rb_kv_write: slot >= num_blocks * block_size */
#define RB_EBIT_ROW_INDEX 0x040     /* rb_gather_rows: index outside [0, num_hidden_rows) */
#define RB_EBIT_ATTN_META 0x080     /* rb_paged_attention: query_start_loc not monotone, last
                                       entry != num_tokens, seq_len < query length, or seq_len
                                       beyond max_blocks_per_req pages */
#define RB_EBIT_TIMEOUT 0x100       /* a bounded wait on an asynchronous copy gave up */

/* Static sizes of the persistent batch and of one layer's paged KV pool. */
typedef struct rb_dims {
  int32_t block_size;         /* B: tokens per KV page */
  int32_t num_q_heads;        /* nh */
  int32_t num_kv_heads;       /* nkv; nh % nkv == 0, query head h reads kv head h / (nh/nkv) */
  int32_t head_dim;           /* hd */
  int32_t max_num_reqs;       /* rows of the token table and of the page table */
  int32_t max_model_len;      /* M: columns of the token table */
  int32_t max_blocks_per_req; /* MB: columns of the page table */
  int32_t num_blocks;         /* physical pages in the pool, the null page included */
  int32_t null_block;         /* reserved page id that receives every padding token */
  int32_t kernel_blocks_per_manager_block; /* r: page-table entries are manager blocks of
                                 r * block_size tokens ("vLLM 源码完全拆解（五）…", "混合 KV
                                 Cache：一条请求不止一张页表": a 32-token manager block seen by a
                                 16-token kernel expands into two kernel pages, manager ids
                                 [0, 1, 2] -> kernel ids [0 .. 5]); manager id m covers kernel
                                 pages m*r .. m*r + r - 1, so logical kernel page j of a row is
                                 block_table[i, j / r] * r + j % r.  1 (or 0) = the table holds
                                 kernel pages.  With r > 1: num_blocks and null_block are in
                                 kernel pages and multiples of r, max_blocks_per_req counts
                                 table entries (a row spans max_blocks_per_req * r kernel pages)
                                 and the whole manager block null_block / r is reserved. */
} rb_dims;

/* Human-readable name of a status code (static string). */
const char* rb_status_string(int32_t status);

/* Number of kernels this library has enqueued since it was loaded (all devices, all calls). */
uint64_t rb_kernel_launch_count(void);

/*
 * rb_debug_attention_wait_limit — test hook of the attention launch's bounded waits; the pages
 * have no counterpart.  Every wait of the fused attention launch on an asynchronous copy, an
 * MMA or another role gives up after `wait_limit_ns` (default 1 s; 0 restores it), sets
 * RB_EBIT_TIMEOUT, lets the copies and MMAs it already issued complete, frees its tensor memory
 * and returns.  With `withhold_first_unit` = 1 the producer of CTA 0 stops before handing its
 * first prefill unit to the other roles (no copy or MMA of that unit is ever issued), so their
 * waits for it run out: a test of the timeout path that faults nothing.  Process-wide, read at
 * each attention call's set-up; not for production use.  RB_ERR_INVALID_ARG for a limit
 * outside [100 us, 10 s] (other than 0) or a flag other than 0 / 1.
 */
rb_status rb_debug_attention_wait_limit(uint64_t wait_limit_ns, int32_t withhold_first_unit);

/*
 * rb_pad_for_graph — host function; smallest entry of `capture_sizes` (sorted ascending,
 * `num_sizes` entries) that is >= num_tokens; num_tokens itself when it exceeds the largest size
 * (the step then runs unpadded), and -1 for invalid arguments (null sizes with num_sizes > 0,
 * num_sizes < 0, num_tokens < 0, unsorted sizes).
 * Source: "第8章 ModelRunner：从 SchedulerOutput 到 GPU Kernel", "8.5 pad_for_cudagraph" and
 * "8.5.0.5 pad_for_cudagraph 的实现" (bisect_left over sorted sizes); "04 · 模型执行与 CUDA Graph",
 * "4.4 派发" (beyond the largest captured size the step runs eager).
 */
int32_t rb_pad_for_graph(const int32_t* capture_sizes, int32_t num_sizes, int32_t num_tokens);

/*
 * rb_prepare_inputs — flatten one step of the persistent batch.
 * Source: "vLLM 源码完全拆解（五）：GPUModelRunner 如何把动态请求拼成一次 GPU 前向", sections
 * "第一步" (query_start_loc = exclusive prefix sum of num_scheduled), "第二步" (positions =
 * num_computed + offset in the request; seq_lens = num_computed + num_scheduled), "第三步"
 * (input ids gathered from row i, columns c_i .. c_i+q_i-1 of the token table), "第四步"
 * (logits_indices = query_start_loc[1:] - 1), "Block table 是逐请求的页表" (slot_mapping) and
 * "固定地址与动态有效长度如何共存" (padding to a captured size); "04 · 模型执行与 CUDA Graph",
 * "5. 关键细节与坑" (padding tokens use the null page).
 *
 * Inputs (device, int32):
 *   d_token_table   [max_num_reqs, max_model_len]       row i = token history of batch row i
 *   d_num_computed  [num_reqs]                          tokens already in the cache (c_i)
 *   d_num_scheduled [num_reqs]                          tokens scheduled this step (q_i >= 1)
 *   d_block_table   [max_num_reqs, max_blocks_per_req]  physical page ids of each row
 * Sizes: 0 <= num_reqs <= num_reqs_padded <= max_num_reqs; num_tokens = sum(q_i) (checked on the
 *   device); num_tokens <= num_tokens_padded; num_tokens_padded >= 1 when num_reqs_padded >= 1.
 * Outputs (device, int32, written in full):
 *   d_input_ids, d_positions, d_slot_mapping  [num_tokens_padded]
 *   d_query_start_loc                          [num_reqs_padded + 1]
 *   d_seq_lens, d_logits_indices               [num_reqs_padded]
 *   d_scalars [4] = {max_query_len, max_seq_len, num_actual_tokens (= num_tokens), error word}
 * Optional phase flags ("Chunked Prefill：query 很长，但仍只是一段区间", "第四步"): when
 *   d_is_prefilling and d_discard_request_mask [num_reqs_padded] (int32 0/1) are given (both,
 *   with d_num_prompt [num_reqs] = prompt lengths whenever num_reqs > 0) they receive
 *   is_prefilling = num_computed < num_prompt (not "query length 1 means decode") and
 *   discard_request_mask = num_computed + num_scheduled < num_prompt (the chunk ends inside the
 *   prompt, so the token sampled from its last position is not an output); padded requests get
 *   0 and 1.  With both flag pointers NULL nothing is written and d_num_prompt is ignored.
 * Padding: request i >= num_reqs gets the empty interval at the end (query_start_loc = N),
 *   seq_len 0 and logits index max(N-1, 0); token t >= N gets input id 0, position 0 and slot
 *   null_block * B + (t - N) % B, so padding only ever touches the null page.
 * Errors: host -> RB_ERR_INVALID_ARG / RB_ERR_CAPACITY / RB_ERR_UNSUPPORTED (num_reqs > 16384);
 *   device -> bits NUM_SCHEDULED, NUM_COMPUTED, SEQ_LEN, TOKEN_SUM, BLOCK_ID in d_scalars[3]
 *   (zeroed by this call); a token whose page id is invalid gets a null-page slot.
 */
rb_status rb_prepare_inputs(const rb_dims* dims, int32_t num_reqs, int32_t num_reqs_padded,
                            int32_t num_tokens, int32_t num_tokens_padded,
                            const int32_t* d_token_table, const int32_t* d_num_computed,
                            const int32_t* d_num_scheduled, const int32_t* d_block_table,
                            int32_t* d_input_ids, int32_t* d_positions,
                            int32_t* d_query_start_loc, int32_t* d_seq_lens,
                            int32_t* d_slot_mapping, int32_t* d_logits_indices,
                            int32_t* d_scalars, const int32_t* d_num_prompt,
                            int32_t* d_is_prefilling, int32_t* d_discard_request_mask,
                            void* stream);

/*
 * rb_kv_write — scatter this step's K and V rows into the paged cache.
 * Source: "vLLM 源码完全拆解（五）…", "3. 物理 KV 槽位" (row t goes to slot_mapping[t]);
 * "变长批处理与一次混合前向", runner.py (the write happens before attention reads the context);
 * "Nano-VLLM全代码解析笔记(4)-model_runner" (a slot of -1 is skipped).
 *
 *   d_k, d_v        [num_tokens_padded, nkv, hd] bf16, rows contiguous, 16-byte aligned
 *   d_slot_mapping  [num_tokens_padded] int32; slot < 0 -> row skipped
 *   d_k_cache, d_v_cache  [num_blocks * B, nkv, hd] bf16, 16-byte aligned (updated in place)
 *   d_error_word    int32 or NULL; bit SLOT for slot >= num_blocks * B (row skipped)
 * Two real tokens must not share a slot (then the surviving row is unspecified).
 */
rb_status rb_kv_write(const rb_dims* dims, int32_t num_tokens_padded, const void* d_k,
                      const void* d_v, const int32_t* d_slot_mapping, void* d_k_cache,
                      void* d_v_cache, int32_t* d_error_word, void* stream);

/*
 * Workspace bytes rb_paged_attention needs for batches of at most max_num_reqs requests and
 * max_num_tokens real tokens (0 on invalid arguments).  The workspace is caller-owned device
 * memory, at least 256-byte aligned; its contents need no initialisation and are scratch.
 */
size_t rb_paged_attention_workspace_size(const rb_dims* dims, int32_t max_num_reqs,
                                         int32_t max_num_tokens);

/*
 * rb_paged_attention — varlen causal GQA attention of a mixed batch through the page table.
 * Source: "vLLM 源码完全拆解（五）…", "4. 注意力读取边界" (query j of request i reads only its
 * own request, keys 0 .. c_i + j, c_i = seq_len - query length) and "为什么不显式构造巨大
 * Attention Mask" (bounds from query_start_loc, seq_lens, causal=True); "变长批处理与一次混合前向",
 * runner.py (scale 1/sqrt(hd); new K/V written first, then the whole context is read);
 * "Nano-VLLM全代码解析笔记(4)-model_runner" (cu_seqlens_q / seq lens / block tables).
 *
 *   d_q               [num_tokens_padded, nh, hd] bf16 (this step's queries, flat order)
 *   d_k_cache/v_cache [num_blocks * B, nkv, hd] bf16 — must already hold this step's rows
 *   d_block_table     [max_num_reqs, max_blocks_per_req] int32
 *   d_query_start_loc [num_reqs + 1] int32, d_seq_lens [num_reqs] int32
 *   softmax_scale     multiplier of q.k (normally 1/sqrt(hd))
 *   d_out             [num_tokens_padded, nh, hd] bf16; rows >= num_tokens are written as 0
 *   d_workspace       rb_paged_attention_workspace_size(dims, >= num_reqs, >= num_tokens) bytes
 *   d_error_word      int32 or NULL; bits ATTN_META, BLOCK_ID, TIMEOUT
 * Supported: block_size 16, head_dim 64 or 128, nh/nkv <= 16; base pointers 16-byte aligned.
 * Decodes and short queries (query length x nh/nkv <= 8) run a split-KV streaming kernel; longer
 * queries run a tensor-core tile kernel; all requests of the batch are handled by one call.
 */
rb_status rb_paged_attention(const rb_dims* dims, int32_t num_reqs, int32_t num_tokens,
                             int32_t num_tokens_padded, const void* d_q, const void* d_k_cache,
                             const void* d_v_cache, const int32_t* d_block_table,
                             const int32_t* d_query_start_loc, const int32_t* d_seq_lens,
                             float softmax_scale, void* d_out, void* d_workspace,
                             size_t workspace_bytes, int32_t* d_error_word, void* stream);

/*
 * rb_paged_attention_profiled — rb_paged_attention that also records caller-created CUDA events
 * (cudaEvent_t passed as void*) on `stream` between its launches, for per-kernel timing:
 * events[0] after the planner, events[1] after the decode kernel, events[2] after the prefill
 * kernel; only the first num_events (<= 3) are used and NULL entries are skipped.  While
 * `stream` is being captured into a CUDA graph the records are made as external event nodes, so
 * they are recorded on every replay.  Same
 * arguments, results and errors as rb_paged_attention otherwise; RB_ERR_INVALID_ARG if
 * num_events < 0 or events is NULL with num_events > 0.
 */
rb_status rb_paged_attention_profiled(const rb_dims* dims, int32_t num_reqs, int32_t num_tokens,
                                      int32_t num_tokens_padded, const void* d_q,
                                      const void* d_k_cache, const void* d_v_cache,
                                      const int32_t* d_block_table,
                                      const int32_t* d_query_start_loc,
                                      const int32_t* d_seq_lens, float softmax_scale, void* d_out,
                                      void* d_workspace, size_t workspace_bytes,
                                      int32_t* d_error_word, void* stream, void* const* events,
                                      int32_t num_events);

/*
 * rb_paged_attention_static_ws — rb_paged_attention without a caller-provided workspace.
 * The pages have no counterpart: this entry point exists for callers that cannot allocate
 * device memory, such as code whose host framework owns every device byte (a raw cudaMalloc
 * would escape its accounting) or a step loop where cudaMalloc/cudaFree would synchronise the
 * device.  It allocates nothing.  Its scratch is a fixed 64 MiB array compiled into the library,
 * held by every GPU that loads it until the process exits.
 *
 * Arguments, layouts, results and device error bits are those of rb_paged_attention.
 * Errors: RB_ERR_CAPACITY when rb_paged_attention_workspace_size(dims, num_reqs, num_tokens)
 * exceeds 64 MiB (at 8 kv heads and head_dim 128: more than 991 requests); RB_ERR_CUDA if the
 * array's device address cannot be obtained.  The first call on a device looks that address
 * up with the device current and keeps it for later calls; make it before any stream capture.
 * The kept address belongs to the device's primary context (the one the CUDA runtime uses):
 * after cudaDeviceReset, or from a context the caller made itself with the driver API, it is
 * not valid, so such callers must not use this entry point.  All calls on a device share
 * the array: calls whose work overlaps on the GPU (e.g. two streams at once) race on it, so
 * serialise them.  Nothing in the array needs clearing between calls: the planner launch
 * rewrites every field the later launches read.
 */
rb_status rb_paged_attention_static_ws(const rb_dims* dims, int32_t num_reqs, int32_t num_tokens,
                                       int32_t num_tokens_padded, const void* d_q,
                                       const void* d_k_cache, const void* d_v_cache,
                                       const int32_t* d_block_table,
                                       const int32_t* d_query_start_loc,
                                       const int32_t* d_seq_lens, float softmax_scale,
                                       void* d_out, int32_t* d_error_word, void* stream);

/*
 * rb_cascade_prefix_len — host function; the shared-prefix length a cascade call may use:
 * min(shared_prefix_tokens, min_i num_computed[i]) rounded down to a multiple of block_size
 * (pass the page-table entry's token count, block_size * kernel_blocks_per_manager_block).
 * Source: "第8章 ModelRunner…", "8.3.2.5 Cascade Attention 的 "最小 num_computed_tokens - 1"
 * 规则" (the printed rule: cap by the smallest num_computed, then align to the block size, so
 * no request's query sees a key of the prefix that it must not see).  num_computed is HOST
 * memory [num_reqs].  0 for num_reqs = 0; -1 for invalid arguments (negative values, NULL
 * num_computed with num_reqs > 0, block_size < 1).
 */
int32_t rb_cascade_prefix_len(int32_t shared_prefix_tokens, const int32_t* num_computed,
                              int32_t num_reqs, int32_t block_size);

/* Workspace bytes of rb_paged_attention_cascade (the ordinary workspace plus the prefix pass's
   fp32 outputs [max_num_tokens, nh, head_dim] and log-sum-exps); 0 for invalid arguments. */
size_t rb_paged_attention_cascade_workspace_size(const rb_dims* dims, int32_t max_num_reqs,
                                                 int32_t max_num_tokens);

/*
 * rb_paged_attention_cascade — rb_paged_attention when every request shares its first
 * common_prefix_len tokens (the same page-table entries): the prefix keys are read once for
 * all query rows, then each request's own keys.  Same result up to rounding.
 * Source: "第8章 ModelRunner…", "8.3.2.5 Cascade Attention" (a shared-prefix pass and a
 * per-request suffix pass).
 *
 *   pass 1: every query row of the batch against keys [0, P) of row 0's pages, no mask (P is
 *           at most every request's cached length, so each query sees all of them) -> fp32
 *           output and log-sum-exp per (token, head) in the workspace;
 *   pass 2: the ordinary causal attention over keys [P, seq_len) of each request, whose
 *           epilogue merges the pass-1 row by log-sum-exp before rounding to bf16.
 * Arguments as rb_paged_attention, plus common_prefix_len = P (rb_cascade_prefix_len gives
 * it); the workspace is rb_paged_attention_cascade_workspace_size(dims, num_reqs, num_tokens).
 * P = 0 (or an empty batch) is rb_paged_attention.
 * Errors: host -> as rb_paged_attention, RB_ERR_INVALID_ARG when P is not a multiple of
 *   block_size * kernel_blocks_per_manager_block or spans more than max_blocks_per_req entries,
 *   RB_ERR_UNSUPPORTED for P > 0 on shapes without the tcgen05 path (head group not a power of
 *   two, head_dim not 64 or 128); device -> bit ATTN_META when a request caches fewer than P
 *   tokens or its first P / (block_size * r) entries differ from row 0's (results unspecified).
 */
rb_status rb_paged_attention_cascade(const rb_dims* dims, int32_t num_reqs, int32_t num_tokens,
                                     int32_t num_tokens_padded, int32_t common_prefix_len,
                                     const void* d_q, const void* d_k_cache,
                                     const void* d_v_cache, const int32_t* d_block_table,
                                     const int32_t* d_query_start_loc, const int32_t* d_seq_lens,
                                     float softmax_scale, void* d_out, void* d_workspace,
                                     size_t workspace_bytes, int32_t* d_error_word, void* stream);

/*
 * rb_gather_rows — out[i, :] = hidden[indices[i], :] for i < num_rows.
 * Source: "vLLM 源码完全拆解（五）…", "第四步：只在必要位置计算 logits"; "04 · 模型执行与
 * CUDA Graph", step ⑤ (hidden_states[logits_indices]).
 *
 *   d_hidden  [num_hidden_rows, hidden_size] bf16;  d_indices [num_rows] int32
 *   d_out     [num_rows, hidden_size] bf16
 *   d_error_word int32 or NULL; bit ROW_INDEX for an index outside [0, num_hidden_rows), whose
 *   output row is written as zeros.
 * hidden_size * 2 must be a multiple of 16 bytes and both base pointers 16-byte aligned.
 */
rb_status rb_gather_rows(int32_t num_rows, int32_t hidden_size, int32_t num_hidden_rows,
                         const void* d_hidden, const int32_t* d_indices, void* d_out,
                         int32_t* d_error_word, void* stream);

/*
 * rb_step — the whole step in one call: rb_prepare_inputs, rb_kv_write (the step's K/V at
 * slot_mapping), rb_paged_attention and rb_gather_rows (hidden rows at logits_indices), with
 * the same results bit for bit, enqueued as one memset and two launches instead of five
 * launches: one preparation kernel writes the metadata, copies the K/V rows, gathers the hidden
 * rows and plans the attention; the attention launch follows.  Sources: those of the four
 * calls.  Arguments are those of the four calls, gathered in one struct (all device pointers
 * but `dims`; the scalars' error word collects every call's bits and is zeroed here).
 * Errors: the host checks of the four calls; device bits as the four calls set them.
 */
typedef struct rb_step_args {
  const rb_dims* dims;
  int32_t num_reqs, num_reqs_padded, num_tokens, num_tokens_padded;
  int32_t hidden_size;      /* columns of d_hidden / d_rows_out */
  int32_t num_hidden_rows;  /* rows of d_hidden (normally num_tokens_padded) */
  float softmax_scale;
  /* persistent batch (rb_prepare_inputs) */
  const int32_t* d_token_table;
  const int32_t* d_num_computed;
  const int32_t* d_num_scheduled;
  const int32_t* d_block_table;
  const int32_t* d_num_prompt; /* optional, with the two flag outputs */
  /* this step's activations and the paged cache */
  const void* d_q;      /* [num_tokens_padded, nh, hd] bf16 */
  const void* d_k;      /* [num_tokens_padded, nkv, hd] bf16 */
  const void* d_v;
  const void* d_hidden; /* [num_hidden_rows, hidden_size] bf16 */
  void* d_k_cache;      /* [num_blocks * block_size, nkv, hd] bf16 */
  void* d_v_cache;
  /* outputs */
  int32_t* d_input_ids;
  int32_t* d_positions;
  int32_t* d_query_start_loc;
  int32_t* d_seq_lens;
  int32_t* d_slot_mapping;
  int32_t* d_logits_indices;
  int32_t* d_scalars;
  int32_t* d_is_prefilling;         /* optional */
  int32_t* d_discard_request_mask;  /* optional */
  void* d_attn_out;  /* [num_tokens_padded, nh, hd] bf16 */
  void* d_rows_out;  /* [num_reqs_padded, hidden_size] bf16 */
  /* attention workspace: rb_paged_attention_workspace_size(dims, num_reqs, num_tokens) */
  void* d_workspace;
  size_t workspace_bytes;
} rb_step_args;

rb_status rb_step(const rb_step_args* args, void* stream);

/*
 * rb_step_profiled — rb_step with caller-owned CUDA events recorded between its launches, for
 * per-kernel timing of a step: events[0] after the preparation launch, events[1] after the
 * attention launch (cudaEvent_t passed as void*, created by the caller; null slots and slots
 * past num_events are skipped).  Inside a stream capture the records become external event
 * nodes.  Sources, arguments, results and errors are those of rb_step, plus RB_ERR_INVALID_ARG
 * for num_events < 0 or a null `events` with num_events > 0, and RB_ERR_CUDA if a record fails.
 */
rb_status rb_step_profiled(const rb_step_args* args, void* const* events, int32_t num_events,
                           void* stream);

/*
 * rb_host_copy — one contiguous copy between caller-owned host memory and caller-owned device
 * memory: `bytes` bytes from `src` to `dst` (both null only when `bytes` is 0).  Page-locked
 * host memory makes the copy asynchronous; pageable memory works but the copy then blocks the
 * calling thread.
 */
typedef struct rb_host_copy {
  void* dst;
  const void* src;
  size_t bytes;
} rb_host_copy;

/*
 * rb_step_host — rb_step with its inputs brought in from host memory and its results returned
 * to it: after every host check of rb_step passes, enqueues on `stream` the `num_in` host-to-
 * device copies `in` (typically the token and page tables, the counters, q / k / v and the
 * hidden states, into the device buffers `args` points at), then the step exactly as rb_step,
 * then the `num_out` device-to-host copies `out` (typically the attention output, the gathered
 * rows and the scalars with the error word).  One cudaMemcpyAsync per copy, in array order;
 * nothing else is allocated or synchronised.  The step's inputs and outputs are what the
 * caller names: the library does not check that the copies cover them.
 * Errors: RB_ERR_INVALID_ARG for a null `args`, negative counts, a null array with a nonzero
 * count or a null pointer in a copy of nonzero size; the host checks of rb_step; all returned
 * before anything is enqueued.  RB_ERR_CUDA if enqueueing a copy or a launch fails (what was
 * enqueued before stays enqueued).  Device bits as rb_step sets them.
 */
rb_status rb_step_host(const rb_step_args* args, const rb_host_copy* in, int32_t num_in,
                       const rb_host_copy* out, int32_t num_out, void* stream);

/*
 * rb_step_host_async — rb_step_host with its copies on streams of their own, so that the
 * copies of consecutive steps overlap the steps themselves (the host link and the GPU work at
 * once): enqueues the `num_in` host-to-device copies on `in_stream` and records `in_done`
 * there; makes `stream` wait for `in_done`, enqueues the step exactly as rb_step on `stream`
 * and records `step_done` there; makes `out_stream` wait for `step_done` and enqueues the
 * `num_out` device-to-host copies on it.  `in_done` and `step_done` are caller-created
 * cudaEvent_t (passed as void*); streams may be null (the legacy default stream).
 * The caller keeps the buffers of steps in flight apart (for example two sets of input and
 * output buffers used by alternate steps) and orders their reuse: the in-copies of a later
 * step into a set after the step that read the set (`in_stream` waiting on that step's
 * `step_done`), a later step's writes to an output set after the out-copies of the step
 * before (`stream` waiting on an event recorded on `out_stream`).  One cudaMemcpyAsync per
 * copy; nothing is allocated or synchronised.
 * Errors: those of rb_step_host, plus RB_ERR_INVALID_ARG for a null `in_done` or
 * `step_done`, all returned before anything is enqueued; RB_ERR_CUDA if enqueueing a copy, a
 * record, a wait or a launch fails (what was enqueued before stays enqueued).
 */
rb_status rb_step_host_async(const rb_step_args* args, const rb_host_copy* in, int32_t num_in,
                             const rb_host_copy* out, int32_t num_out, void* stream,
                             void* in_stream, void* out_stream, void* in_done,
                             void* step_done);

/*
 * Persistent batch — one row per resident request, every column device-resident and
 * caller-owned ("vLLM 源码完全拆解（五）…", "行号是一种短生命周期地址": the row is the common key
 * of the request's token history, counters and page row; a move must carry every column).
 * The live rows are always the prefix [0, *d_num_rows).  Contents past a row's d_num_tokens /
 * d_num_blocks, and rows at or past *d_num_rows, are not state and may hold anything.  Start
 * an empty batch with *d_num_rows = 0 (the other columns need no initial values).
 */
typedef struct rb_batch {
  int32_t max_num_reqs;       /* rows (<= 4096) */
  int32_t max_model_len;      /* M: token-table columns */
  int32_t max_blocks_per_req; /* MB: page-table columns */
  int32_t reserved;           /* 0 */
  int64_t* d_req_id;          /* [max_num_reqs] request id of each live row (ids are >= 0) */
  int32_t* d_token_table;     /* [max_num_reqs, M] token history of each row */
  int32_t* d_num_tokens;      /* [max_num_reqs] valid history length of each row */
  int32_t* d_num_prompt;      /* [max_num_reqs] prompt length */
  int32_t* d_num_computed;    /* [max_num_reqs] tokens already in the KV cache */
  int32_t* d_block_table;     /* [max_num_reqs, MB] page ids of each row */
  int32_t* d_num_blocks;      /* [max_num_reqs] valid page-table entries of each row */
  int32_t* d_num_rows;        /* [1] live rows */
} rb_batch;

/*
 * One step's scheduler output in request-id terms ("第8章 ModelRunner…", "8.2.2 三种变更操作";
 * "vLLM 源码完全拆解（五）…", "新请求建立完整状态" and "驻留请求只合并差量").  All arrays are
 * device memory (typically slices of one buffer filled by a single host-to-device copy);
 * offsets arrays have count + 1 non-decreasing entries indexing the payload that follows them.
 */
typedef struct rb_batch_update {
  int32_t num_scheduled;             /* S: requests scheduled this step (new ones included) */
  int32_t num_new;                   /* NN */
  int32_t num_cached;                /* NC */
  int32_t reserved;                  /* 0 */
  const int64_t* d_sched_req_id;     /* [S] */
  const int32_t* d_sched_num_tokens; /* [S] tokens scheduled for each */
  const int64_t* d_new_req_id;       /* [NN] requests entering the batch, whole state: */
  const int32_t* d_new_num_computed; /* [NN] */
  const int32_t* d_new_num_prompt;   /* [NN] */
  const int32_t* d_new_token_start;  /* [NN + 1] -> d_new_tokens: each request's history */
  const int32_t* d_new_tokens;
  const int32_t* d_new_block_start;  /* [NN + 1] -> d_new_blocks: each request's page ids */
  const int32_t* d_new_blocks;
  const int64_t* d_cached_req_id;      /* [NC] resident requests that changed: */
  const int32_t* d_cached_num_computed;/* [NC] new num_computed */
  const int32_t* d_cached_replace;     /* [NC] 1: resumed from preemption, the page row is
                                          replaced by the given ids; 0: they are appended */
  const int32_t* d_cached_token_start; /* [NC + 1] -> d_cached_tokens: appended to the history */
  const int32_t* d_cached_tokens;
  const int32_t* d_cached_block_start; /* [NC + 1] -> d_cached_blocks */
  const int32_t* d_cached_blocks;
} rb_batch_update;

#define RB_EBIT_BATCH_ID 0x200    /* rb_batch_apply_update: a negative or repeated request id, a
                                     new request that is not scheduled, a delta for a request
                                     that is not resident, or a scheduled request that is
                                     neither resident nor new */
#define RB_EBIT_BATCH_SIZE 0x400  /* rb_batch_apply_update: decreasing offsets, a history longer
                                     than M or a page row longer than MB */

/* Workspace bytes rb_batch_apply_update needs for a batch of `max_num_reqs` rows. */
rb_status rb_batch_update_workspace_size(int32_t max_num_reqs, size_t* bytes);

/*
 * rb_batch_apply_update — merge one step's scheduler output into the persistent batch, in the
 * order the runner does it, then write this step's per-row scheduled counts.
 * Source: "vLLM 源码完全拆解（五）…", "先删除完成和本轮未调度的请求", "新请求建立完整状态",
 * "驻留请求只合并差量", "最后压紧并刷新派生 metadata" and "行号是一种短生命周期地址" (A B C D, B
 * finishes, D moves to row 1); "第8章 ModelRunner…", "8.2.2.5 _update_states 的真实四段执行"
 * (removals first; new requests take the freed rows) and "8.2.2.6" (an id that is finished and
 * scheduled as new again names a new request); "04 · 模型执行与 CUDA Graph", "4.2 块表" (append_row).
 *
 *  1. a live row is removed unless its request is scheduled and not announced again as new;
 *  2. each resident request in the cached list sets num_computed, appends its tokens after its
 *     history, and appends its page ids (or, with replace, makes them its whole page row);
 *  3. new requests, in list order, take the freed rows in ascending order, then the rows after
 *     the old end of the batch, each with its whole history, counters and page row;
 *  4. condense: the highest live row moves (all columns) into the lowest remaining hole, the
 *     next highest into the next, until the live rows are [0, S).
 * Outputs: the batch (columns and *d_num_rows = S); d_num_scheduled [max_num_reqs] int32 =
 *   tokens scheduled for each row (0 for rows >= S), the d_num_scheduled input of
 *   rb_prepare_inputs with num_reqs = S; d_row_of_sched [S] int32 (or NULL) = the row of each
 *   scheduled request.
 * Work: a one-block planner (request-id hash, hole scan, pairing, counters) and a grid of
 *   16-byte copies of the moved and installed token and page rows.
 * Errors: host -> RB_ERR_INVALID_ARG (null pointers, negative counts, NN or NC > S),
 *   RB_ERR_CAPACITY (S > max_num_reqs, small workspace), RB_ERR_UNSUPPORTED (max_num_reqs >
 *   4096); device -> RB_EBIT_BATCH_ID / RB_EBIT_BATCH_SIZE in *d_error_word (not zeroed here),
 *   and then the batch is left exactly as it was and the two outputs are unspecified.
 */
rb_status rb_batch_apply_update(const rb_batch* batch, const rb_batch_update* update,
                                int32_t* d_num_scheduled, int32_t* d_row_of_sched,
                                void* d_workspace, size_t workspace_bytes,
                                int32_t* d_error_word, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RB_H_ */
