// rb_step: one whole step of the hot path — metadata, KV write, attention and the last-token
// row gather — in one memset and two launches.
//
// The four separate calls (rb_prepare_inputs, rb_kv_write, rb_paged_attention, rb_gather_rows)
// cost five launches, each of which waits for cold metadata before it can start.  Here one
// preparation launch does everything that only needs the batch's metadata:
//   - every CTA recomputes the prefix sum of num_scheduled in shared memory (as
//     rb_prepare_inputs does), so each knows the owner of any token and any request's last row;
//   - CTA 0 runs the attention planner (from its scan and num_computed) while the last CTA
//     writes the per-request outputs;
//   - one warp per token writes its input id, position and slot and copies the token's K and V
//     rows into that slot (16-byte accesses, lanes over the row);
//   - one warp per request copies the hidden row at its logits index.
// The attention launch (fused decode + prefill, or decode and prefill) follows on the stream.
// Results are those of the four calls in order, bit for bit.
//
// Sources: "vLLM 源码完全拆解（五）…" 第一步 .. 第四步, "Block table 是逐请求的页表",
// "3. 物理 KV 槽位", "4. 注意力读取边界"; "变长批处理与一次混合前向", runner.py (write K/V, then
// attend); "04 · 模型执行与 CUDA Graph", step ⑤ (hidden_states[logits_indices]).
#include "attn_plan.cuh"
#include "prep_common.cuh"

namespace rb {
namespace {

constexpr int kWarps = prep::kThreads / 32;

struct StepArgs {
  prep::PrepArgs p;
  attn::AttnArgs at;
  int head_dim;
  const int4* k;
  const int4* v;
  int4* kc;
  int4* vc;
  int kv_chunks;  // 16-byte chunks per token row of K (or V)
  long long num_slots;
  const int4* hidden;
  int4* rows_out;
  int hid_chunks;  // 16-byte chunks per hidden row
  int num_hidden_rows;
};

// One warp copies `chunks` 16-byte chunks of row pair (s0 -> d0, s1 -> d1); each batch's loads
// are issued before its stores (the compiler must assume a store may alias a later load, so a
// load-store loop would wait one memory round trip per chunk).  s1 / d1 may be null.
template <int kBatch>
__device__ __forceinline__ void warp_copy_rows(int4* d0, const int4* s0, int4* d1,
                                               const int4* s1, int chunks, int lane) {
  for (int c0 = 0; c0 < chunks; c0 += 32 * kBatch) {
    int4 x0[kBatch], x1[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int c = c0 + u * 32 + lane;
      const bool in = c < chunks;
      x0[u] = in && s0 != nullptr ? __ldg(s0 + c) : make_int4(0, 0, 0, 0);
      x1[u] = in && s1 != nullptr ? __ldg(s1 + c) : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < chunks) {
        d0[c] = x0[u];
        if (d1 != nullptr) d1[c] = x1[u];
      }
    }
  }
}

__global__ void __launch_bounds__(prep::kThreads) step_prep_kernel(StepArgs s) {
  using namespace prep;
  extern __shared__ int32_t s_qsl[];  // [R + 1]
  const PrepArgs& a = s.p;
  int32_t* err = a.scalars + 3;
  block_scan_scheduled(a, s_qsl);
  const int total = s_qsl[a.R];
  // CTA 0 plans the attention from its own scan and num_computed (the values the request
  // outputs hold); the last CTA writes the request outputs, then helps with the tokens
  if (blockIdx.x == 0) {
    if (gridDim.x == 1) request_outputs(a, s_qsl, total, err);
    attn::plan_body(s.at, s.head_dim, attn::ReqSrc{s_qsl, nullptr, a.num_computed});
  } else if (blockIdx.x == gridDim.x - 1) {
    request_outputs(a, s_qsl, total, err);
  }
  // CTA 0 carries the planner on the launch's critical path: the other CTAs take the tokens
  // and rows when there are any
  const int lane = threadIdx.x & 31;
  const int skip = gridDim.x > 1 ? 1 : 0;
  if (static_cast<int>(blockIdx.x) < skip) return;
  const int gw = (blockIdx.x - skip) * kWarps + (threadIdx.x >> 5);
  const int nw = (gridDim.x - skip) * kWarps;
  const int n_real = min(a.N, total);
  constexpr int kPre = 4;  // chunks per lane of each row fetched before the token's metadata
  for (int t = gw; t < a.N_pad; t += nw) {
    // the token's K and V rows need no metadata: their loads are in flight while the owner,
    // position and slot are looked up
    const long long src = static_cast<long long>(t) * s.kv_chunks;
    int4 xk[kPre], xv[kPre];
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int c = u * 32 + lane;
      xk[u] = c < s.kv_chunks ? __ldg(s.k + src + c) : make_int4(0, 0, 0, 0);
      xv[u] = c < s.kv_chunks ? __ldg(s.v + src + c) : make_int4(0, 0, 0, 0);
    }
    int r = -1;
    const TokMeta m = token_meta(a, s_qsl, n_real, t, r);
    int bits = m.bits;
    if (m.slot >= s.num_slots) bits |= RB_EBIT_SLOT;
    if (lane == 0) {
      a.input_ids[t] = m.id;
      a.positions[t] = m.pos;
      a.slots[t] = m.slot;
      if (bits) raise_error(err, bits);
    }
    if (m.slot < 0 || m.slot >= s.num_slots) continue;
    const long long dst = static_cast<long long>(m.slot) * s.kv_chunks;
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int c = u * 32 + lane;
      if (c < s.kv_chunks) {
        s.kc[dst + c] = xk[u];
        s.vc[dst + c] = xv[u];
      }
    }
    if (s.kv_chunks > 32 * kPre)  // wider rows: the rest in batches
      warp_copy_rows<4>(s.kc + dst + 32 * kPre, s.k + src + 32 * kPre, s.vc + dst + 32 * kPre,
                        s.v + src + 32 * kPre, s.kv_chunks - 32 * kPre, lane);
  }
  for (int i = gw; i < a.R_pad; i += nw) {
    const int row = i < a.R ? s_qsl[i + 1] - 1 : max(a.N - 1, 0);
    const bool ok = row >= 0 && row < s.num_hidden_rows;
    if (!ok && lane == 0) raise_error(err, RB_EBIT_ROW_INDEX);
    int4* dst = s.rows_out + static_cast<long long>(i) * s.hid_chunks;
    const int4* src = ok ? s.hidden + static_cast<long long>(row) * s.hid_chunks : nullptr;
    warp_copy_rows<8>(dst, src, nullptr, nullptr, s.hid_chunks, lane);
  }
}

}  // namespace
}  // namespace rb

namespace rb {
namespace {

// Every host check of rb_step, and the launch arguments it builds; nothing is enqueued.
rb_status step_build(const rb_step_args& x, StepArgs* out_sa, attn::AttnSetup* out_su) {
  const rb_dims& d = *x.dims;
  prep::PrepArgs p;
  rb_status st = prep::prep_args_of(
      d, x.num_reqs, x.num_reqs_padded, x.num_tokens, x.num_tokens_padded, x.d_token_table,
      x.d_num_computed, x.d_num_scheduled, x.d_block_table, x.d_input_ids, x.d_positions,
      x.d_query_start_loc, x.d_seq_lens, x.d_slot_mapping, x.d_logits_indices, x.d_scalars,
      x.d_num_prompt, x.d_is_prefilling, x.d_discard_request_mask, &p);
  if (st != RB_OK) return st;
  // KV write and gather operands
  const long long row_bytes = 2LL * d.num_kv_heads * d.head_dim;
  if (row_bytes % 16 != 0 || (2LL * x.hidden_size) % 16 != 0) return RB_ERR_UNSUPPORTED;
  if (x.hidden_size < 1 || x.num_hidden_rows < 0) return RB_ERR_INVALID_ARG;
  if (x.num_tokens_padded > 0 && (x.d_k == nullptr || x.d_v == nullptr)) return RB_ERR_INVALID_ARG;
  if (x.num_reqs_padded > 0 && (x.d_hidden == nullptr || x.d_rows_out == nullptr))
    return RB_ERR_INVALID_ARG;
  if (!aligned16(x.d_k) || !aligned16(x.d_v) || !aligned16(x.d_hidden) ||
      !aligned16(x.d_rows_out))
    return RB_ERR_INVALID_ARG;
  attn::AttnSetup& su = *out_su;
  st = attn::attn_setup(x.dims, x.num_reqs, x.num_tokens, x.num_tokens_padded, x.d_q,
                        x.d_k_cache, x.d_v_cache, x.d_block_table, x.d_query_start_loc,
                        x.d_seq_lens, x.softmax_scale, x.d_attn_out, x.d_workspace,
                        x.workspace_bytes, x.d_scalars + 3, &su);
  if (st != RB_OK) return st;
  st = attn::attn_encode_maps(&su);
  if (st != RB_OK) return st;

  StepArgs& sa = *out_sa;
  sa.p = p;
  sa.at = su.a;
  sa.head_dim = d.head_dim;
  sa.k = static_cast<const int4*>(x.d_k);
  sa.v = static_cast<const int4*>(x.d_v);
  sa.kc = static_cast<int4*>(x.d_k_cache);
  sa.vc = static_cast<int4*>(x.d_v_cache);
  sa.kv_chunks = static_cast<int>(row_bytes / 16);
  sa.num_slots = static_cast<long long>(d.num_blocks) * d.block_size;
  sa.hidden = static_cast<const int4*>(x.d_hidden);
  sa.rows_out = static_cast<int4*>(x.d_rows_out);
  sa.hid_chunks = static_cast<int>(2LL * x.hidden_size / 16);
  sa.num_hidden_rows = x.num_hidden_rows;
  return RB_OK;
}

// Records event i of a profiled call (none when i >= n or the slot is null); inside a stream
// capture the record becomes a graph node.
struct StepMarks {
  void* const* events;
  int n;
  bool record(int i, cudaStream_t s) const {
    if (i >= n || events[i] == nullptr) return true;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return false;
    return cudaEventRecordWithFlags(static_cast<cudaEvent_t>(events[i]), s,
                                    cap == cudaStreamCaptureStatusActive
                                        ? cudaEventRecordExternal
                                        : cudaEventRecordDefault) == cudaSuccess;
  }
};

// The step's memset and two launches on stream `s`; `marks` (optional) records its events
// after the preparation launch and after the attention launch.
rb_status step_enqueue(const rb_step_args& x, const StepArgs& sa, const attn::AttnSetup& su,
                       cudaStream_t s, const StepMarks& marks = StepMarks{nullptr, 0}) {
  if (cudaMemsetAsync(x.d_scalars + 3, 0, sizeof(int32_t), s) != cudaSuccess) return RB_ERR_CUDA;
  const size_t smem = static_cast<size_t>(x.num_reqs + 1) * sizeof(int32_t);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(step_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return RB_ERR_CUDA;
  const int sms = max(1, device_sm_count());
  const int want = (max(x.num_tokens_padded, x.num_reqs_padded) + kWarps - 1) / kWarps;
  const int grid = max(1, min(want, 2 * sms)) + (want > 0 ? 1 : 0);  // + the planner's CTA
  step_prep_kernel<<<grid, prep::kThreads, smem, s>>>(sa);
  if (last_launch_status() != RB_OK) return RB_ERR_CUDA;
  note_launches(1);
  if (!marks.record(0, s)) return RB_ERR_CUDA;
  const rb_status st = attn::attn_main(su, s);
  if (st != RB_OK) return st;
  return marks.record(1, s) ? RB_OK : RB_ERR_CUDA;
}

}  // namespace
}  // namespace rb

extern "C" rb_status rb_step(const rb_step_args* args, void* stream) {
  rb::CallRange range_("rb_step");
  using namespace rb;
  if (args == nullptr || args->dims == nullptr) return RB_ERR_INVALID_ARG;
  StepArgs sa;
  attn::AttnSetup su;
  const rb_status st = step_build(*args, &sa, &su);
  if (st != RB_OK) return st;
  return step_enqueue(*args, sa, su, static_cast<cudaStream_t>(stream));
}

extern "C" rb_status rb_step_profiled(const rb_step_args* args, void* const* events,
                                      int32_t num_events, void* stream) {
  rb::CallRange range_("rb_step_profiled");
  using namespace rb;
  if (args == nullptr || args->dims == nullptr || num_events < 0 ||
      (num_events > 0 && events == nullptr))
    return RB_ERR_INVALID_ARG;
  StepArgs sa;
  attn::AttnSetup su;
  const rb_status st = step_build(*args, &sa, &su);
  if (st != RB_OK) return st;
  return step_enqueue(*args, sa, su, static_cast<cudaStream_t>(stream),
                      StepMarks{events, num_events});
}

namespace rb {
namespace {

rb_status check_host_copies(const rb_step_args* args, const rb_host_copy* in, int32_t num_in,
                            const rb_host_copy* out, int32_t num_out) {
  if (args == nullptr || args->dims == nullptr || num_in < 0 || num_out < 0 ||
      (num_in > 0 && in == nullptr) || (num_out > 0 && out == nullptr))
    return RB_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_in; ++i)
    if (in[i].bytes > 0 && (in[i].dst == nullptr || in[i].src == nullptr))
      return RB_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_out; ++i)
    if (out[i].bytes > 0 && (out[i].dst == nullptr || out[i].src == nullptr))
      return RB_ERR_INVALID_ARG;
  return RB_OK;
}

rb_status enqueue_copies(const rb_host_copy* c, int32_t n, cudaMemcpyKind kind, cudaStream_t s) {
  for (int32_t i = 0; i < n; ++i)
    if (c[i].bytes > 0 && cudaMemcpyAsync(c[i].dst, c[i].src, c[i].bytes, kind, s) != cudaSuccess)
      return RB_ERR_CUDA;
  return RB_OK;
}

}  // namespace
}  // namespace rb

extern "C" rb_status rb_step_host(const rb_step_args* args, const rb_host_copy* in,
                                  int32_t num_in, const rb_host_copy* out, int32_t num_out,
                                  void* stream) {
  rb::CallRange range_("rb_step_host");
  using namespace rb;
  rb_status st = check_host_copies(args, in, num_in, out, num_out);
  if (st != RB_OK) return st;
  StepArgs sa;
  attn::AttnSetup su;
  st = step_build(*args, &sa, &su);
  if (st != RB_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = enqueue_copies(in, num_in, cudaMemcpyHostToDevice, s)) != RB_OK) return st;
  if ((st = step_enqueue(*args, sa, su, s)) != RB_OK) return st;
  return enqueue_copies(out, num_out, cudaMemcpyDeviceToHost, s);
}

extern "C" rb_status rb_step_host_async(const rb_step_args* args, const rb_host_copy* in,
                                        int32_t num_in, const rb_host_copy* out,
                                        int32_t num_out, void* stream, void* in_stream,
                                        void* out_stream, void* in_done, void* step_done) {
  rb::CallRange range_("rb_step_host_async");
  using namespace rb;
  rb_status st = check_host_copies(args, in, num_in, out, num_out);
  if (st != RB_OK) return st;
  if (in_done == nullptr || step_done == nullptr) return RB_ERR_INVALID_ARG;
  StepArgs sa;
  attn::AttnSetup su;
  st = step_build(*args, &sa, &su);
  if (st != RB_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t si = static_cast<cudaStream_t>(in_stream);
  cudaStream_t so = static_cast<cudaStream_t>(out_stream);
  cudaEvent_t ei = static_cast<cudaEvent_t>(in_done), es = static_cast<cudaEvent_t>(step_done);
  if ((st = enqueue_copies(in, num_in, cudaMemcpyHostToDevice, si)) != RB_OK) return st;
  if (cudaEventRecord(ei, si) != cudaSuccess || cudaStreamWaitEvent(s, ei, 0) != cudaSuccess)
    return RB_ERR_CUDA;
  if ((st = step_enqueue(*args, sa, su, s)) != RB_OK) return st;
  if (cudaEventRecord(es, s) != cudaSuccess || cudaStreamWaitEvent(so, es, 0) != cudaSuccess)
    return RB_ERR_CUDA;
  return enqueue_copies(out, num_out, cudaMemcpyDeviceToHost, so);
}
