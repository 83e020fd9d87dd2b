// rb_paged_attention: varlen causal GQA attention of a mixed batch through the page table.
//
// What it computes ("vLLM 源码完全拆解（五）…", "4. 注意力读取边界"; "变长批处理与一次混合前向",
// runner.py): for request i with c_i = seq_len_i - q_i cached tokens, query j (position c_i + j)
// and query head h reading kv head h / (nh/nkv):
//     o = softmax(scale * q . K[0 .. c_i + j]) . V[0 .. c_i + j]
// over the request's own pages only.
//
// One call enqueues its kernels on the caller's stream, with no host round trip (the host
// only knows num_reqs and the token counts):
//   1. plan     (1 CTA)  validates the metadata, classifies requests (decode-like when
//                        query_len * group <= 8), splits the CTAs between decode and prefill
//                        work, sizes KV splits, writes per-request unit offsets, zeroes padding;
//   2. one persistent launch: every CTA runs decode units (split-KV, one warp per (request, kv
//      head, split); the last split of a (request, kv head) merges the partials) and prefill
//      units (tcgen05 tiles of 128 / group whole tokens), starting with the kind the planner
//      assigned it and then helping with the other, so HBM-bound and tensor-bound work overlap.
#include "attn_plan.cuh"

namespace rb {
namespace attn {
namespace {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) attn_plan_kernel(AttnArgs a, int head_dim) {
  plan_body(a, head_dim, ReqSrc{a.qsl, a.seq_lens, nullptr});
}

// Cascade: checks the shared prefix, writes the suffix pass's sequence lengths (seq_len - P)
// and sets the header up for the prefix pass (its units only; no decode units).
__global__ void __launch_bounds__(kPlanThreads)
    cascade_prepare_kernel(AttnArgs a, int prefix_len, int prefix_entries, int32_t* lens_out) {
  const int tid = threadIdx.x;
  int bits = 0;
  if (tid == 0 && (a.qsl[0] != 0 || a.qsl[a.R] != a.N)) bits |= RB_EBIT_ATTN_META;
  for (int r = tid; r < a.R; r += kPlanThreads) {
    const int q = a.qsl[r + 1] - a.qsl[r], L = a.seq_lens[r];
    // every query must see the whole prefix: P <= cached length (the 8.3.2.5 cap)
    if (q < 0 || L - q < prefix_len) bits |= RB_EBIT_ATTN_META;
    lens_out[r] = L - prefix_len;
  }
  // every request's first page-table entries must be the shared ones (those of row 0)
  const long long total = static_cast<long long>(a.R) * prefix_entries;
  for (long long i = tid; i < total; i += kPlanThreads) {
    const int r = static_cast<int>(i / prefix_entries), e = static_cast<int>(i % prefix_entries);
    if (a.block_table[static_cast<size_t>(r) * a.MB + e] != a.block_table[e])
      bits |= RB_EBIT_ATTN_META;
  }
  if (tid == 0) {
    a.header[kHNumDecodeUnits] = 0;
    a.header[kHNumPrefillUnits] =
        a.nkv * ((a.N + 2 * a.tile_tokens - 1) / (2 * a.tile_tokens)) * a.prefix_splits;
    a.header[kHDecodeNext] = 0;
    a.header[kHPrefillNext] = 0;
    a.header[kHSplitPages] = kMinSplitPages;
    a.header[kHDecodeCtas] = 0;
    a.header[kHRoleNext] = 0;
  }
  if (bits) raise_error(a.err, bits);
}

}  // namespace
}  // namespace attn
}  // namespace rb

extern "C" size_t rb_paged_attention_workspace_size(const rb_dims* dims, int32_t max_num_reqs,
                                                    int32_t max_num_tokens) {
  if (dims == nullptr || max_num_reqs < 0 || max_num_tokens < 0 || dims->num_kv_heads < 1 ||
      dims->head_dim < 1)
    return 0;
  return rb::attn::ws_layout(dims->head_dim, dims->num_kv_heads, max_num_reqs, max_num_tokens)
      .total;
}

namespace rb {
namespace attn {

rb_status attn_setup(const rb_dims* dims, int32_t num_reqs, int32_t num_tokens,
                     int32_t num_tokens_padded, const void* d_q, const void* d_k_cache,
                     const void* d_v_cache, const int32_t* d_block_table,
                     const int32_t* d_query_start_loc, const int32_t* d_seq_lens,
                     float softmax_scale, void* d_out, void* d_workspace, size_t workspace_bytes,
                     int32_t* d_error_word, AttnSetup* su) {
  if (dims == nullptr) return RB_ERR_INVALID_ARG;
  const rb_dims& d = *dims;
  if (d.block_size != kPage) return RB_ERR_UNSUPPORTED;
  if (d.head_dim != 64 && d.head_dim != 128) return RB_ERR_UNSUPPORTED;
  if (d.num_kv_heads < 1 || d.num_q_heads < 1 || d.num_q_heads % d.num_kv_heads != 0)
    return RB_ERR_INVALID_ARG;
  if (d.num_q_heads / d.num_kv_heads > 16) return RB_ERR_UNSUPPORTED;
  PageGeom g;
  if (page_geom_of(d, &g) != RB_OK || d.max_num_reqs < 0) return RB_ERR_INVALID_ARG;
  if (static_cast<long long>(d.num_blocks) * kPage > 0x7fffffffLL) return RB_ERR_CAPACITY;
  if (num_reqs < 0 || num_tokens < 0 || num_tokens_padded < num_tokens) return RB_ERR_INVALID_ARG;
  if (num_reqs > d.max_num_reqs) return RB_ERR_CAPACITY;
  if (!std::isfinite(softmax_scale)) return RB_ERR_INVALID_ARG;
  if (d_q == nullptr || d_k_cache == nullptr || d_v_cache == nullptr || d_block_table == nullptr ||
      d_query_start_loc == nullptr || d_seq_lens == nullptr || d_out == nullptr ||
      d_workspace == nullptr)
    return RB_ERR_INVALID_ARG;
  if (!aligned16(d_q) || !aligned16(d_k_cache) || !aligned16(d_v_cache) || !aligned16(d_out) ||
      (reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0)
    return RB_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(d.head_dim, d.num_kv_heads, num_reqs, num_tokens);
  if (workspace_bytes < w.total) return RB_ERR_CAPACITY;

  const int group = d.num_q_heads / d.num_kv_heads;
  su->g = g;
  su->head_dim = d.head_dim;
  su->k_cache = d_k_cache;
  su->v_cache = d_v_cache;
  su->num_kv_heads = d.num_kv_heads;
  su->num_slots = static_cast<long long>(d.num_blocks) * kPage;
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  AttnArgs& a = su->a;
  a = AttnArgs{};
  a.q = static_cast<const __nv_bfloat16*>(d_q);
  a.out = static_cast<__nv_bfloat16*>(d_out);
  a.block_table = d_block_table;
  a.qsl = d_query_start_loc;
  a.seq_lens = d_seq_lens;
  a.header = reinterpret_cast<int32_t*>(ws + w.header);
  a.dec_off = reinterpret_cast<int32_t*>(ws + w.dec_off);
  a.pre_off = reinterpret_cast<int32_t*>(ws + w.pre_off);
  a.done = reinterpret_cast<int32_t*>(ws + w.done);
  a.pre_list = reinterpret_cast<int32_t*>(ws + w.pre_list);
  a.part_ml = reinterpret_cast<float2*>(ws + w.part_ml);
  a.part_o = reinterpret_cast<float*>(ws + w.part_o);
  a.R = num_reqs;
  a.N = num_tokens;
  a.N_pad = num_tokens_padded;
  a.nh = d.num_q_heads;
  a.nkv = d.num_kv_heads;
  a.group = group;
  a.MB = d.max_blocks_per_req;
  a.num_blocks = d.num_blocks;
  a.null_block = d.null_block;
  a.ratio = g.ratio;
  a.kp_cap = static_cast<long long>(d.max_blocks_per_req) * g.ratio;
  const int sms = max(1, device_sm_count());
  a.target_units = min(kMaxTargetUnits, 32 * sms);
  a.tile_tokens = 128 / group;  // a tcgen05 unit is a pair of 128-row tiles of whole tokens
  a.fused_ctas = sms;
  a.decode_warps_per_cta = 8;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.err = d_error_word;
  debug_wait_settings(&a.wait_limit_ns, &a.withhold_first_unit);
  return RB_OK;
}

rb_status attn_encode_maps(AttnSetup* su) {
  const AttnArgs& a = su->a;
  if (!encode_kv_tensor_map(&su->kmap, su->k_cache, su->head_dim, su->num_kv_heads,
                            su->num_slots) ||
      !encode_kv_tensor_map(&su->vmap, su->v_cache, su->head_dim, su->num_kv_heads,
                            su->num_slots))
    return RB_ERR_CUDA;
  if (a.N_pad > 0 && !encode_q_tensor_map(&su->qmap, a.q, su->head_dim, a.nh, a.N_pad, a.group))
    return RB_ERR_CUDA;
  return RB_OK;
}

template <class Mark>
rb_status attn_main_impl(const AttnSetup& su, cudaStream_t s, const Mark& mark) {
  const AttnArgs& a = su.a;
  rb_status st = RB_OK;
  // one launch runs decode and prefill units side by side
  if (!mark(1)) return RB_ERR_CUDA;
  if (a.R > 0) st = launch_prefill_tc(a, su.head_dim, su.qmap, su.kmap, su.vmap, s);
  if (st != RB_OK) return st;
  if (!mark(2)) return RB_ERR_CUDA;
  return RB_OK;
}

rb_status attn_main(const AttnSetup& su, cudaStream_t s) {
  return attn_main_impl(su, s, [](int) { return true; });
}

}  // namespace attn
}  // namespace rb

namespace {

// Event marks between the launches of one call (profiling); inside a stream capture the
// records become graph nodes.
struct Marks {
  void* const* events;
  int n;
  cudaStream_t s;
  bool capturing;
  bool operator()(int i) const {
    return i >= n || events[i] == nullptr ||
           cudaEventRecordWithFlags(static_cast<cudaEvent_t>(events[i]), s,
                                    capturing ? cudaEventRecordExternal
                                              : cudaEventRecordDefault) == cudaSuccess;
  }
};

rb_status paged_attention_impl(const rb_dims* dims, int32_t num_reqs, int32_t num_tokens,
                               int32_t num_tokens_padded, const void* d_q, const void* d_k_cache,
                               const void* d_v_cache, const int32_t* d_block_table,
                               const int32_t* d_query_start_loc, const int32_t* d_seq_lens,
                               float softmax_scale, void* d_out, void* d_workspace,
                               size_t workspace_bytes, int32_t* d_error_word, void* stream,
                               void* const* events, int32_t num_events,
                               int32_t prefix_len = 0) {
  using namespace rb;
  using namespace rb::attn;
  AttnSetup su;
  rb_status st = attn_setup(dims, num_reqs, num_tokens, num_tokens_padded, d_q, d_k_cache,
                            d_v_cache, d_block_table, d_query_start_loc, d_seq_lens,
                            softmax_scale, d_out, d_workspace, workspace_bytes, d_error_word,
                            &su);
  if (st != RB_OK) return st;
  const rb_dims& d = *dims;
  const PageGeom& g = su.g;
  AttnArgs& a = su.a;
  // cascade: P page-aligned in whole page-table entries, within a row
  if (prefix_len < 0 || prefix_len % (kPage * g.ratio) != 0 ||
      prefix_len / (kPage * g.ratio) > d.max_blocks_per_req)
    return RB_ERR_INVALID_ARG;
  if (num_reqs == 0 || num_tokens == 0) prefix_len = 0;  // nothing shares anything
  const CascadeLayout cl =
      cascade_layout(d.head_dim, d.num_q_heads, d.num_kv_heads, num_reqs, num_tokens);
  if (prefix_len > 0 && workspace_bytes < cl.total) return RB_ERR_CAPACITY;
  st = attn_encode_maps(&su);
  if (st != RB_OK) return st;

  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (prefix_len > 0) {
    // "8.3.2.5 Cascade Attention": the shared prefix once for every query row, then the
    // ordinary causal pass over each request's own keys [P, seq_len), merged per row
    const int entries = prefix_len / (kPage * g.ratio);
    int32_t* lens = reinterpret_cast<int32_t*>(ws + cl.lens);
    a.pre_lse = reinterpret_cast<float*>(ws + cl.lse);
    a.pre_o = reinterpret_cast<float*>(ws + cl.o);
    // cut the prefix keys into ranges so the prefix pass has a few units per SM (each range
    // at least 4 key tiles); the suffix epilogues merge one partial per range
    const int tiles = (prefix_len + 127) / 128;
    const int base_units = d.num_kv_heads * ((num_tokens + 2 * a.tile_tokens - 1) /
                                             (2 * a.tile_tokens));
    const int sms = max(1, device_sm_count());
    int splits = (4 * sms + base_units - 1) / base_units;
    splits = max(1, min(splits, min(kMaxPrefixSplits, tiles / 4)));
    const int split_keys = (tiles + splits - 1) / splits * 128;
    splits = (prefix_len + split_keys - 1) / split_keys;
    a.prefix_splits = splits;
    a.prefix_split_keys = split_keys;
    AttnArgs ap = a;
    ap.cascade = kPrefixPass;
    ap.prefix_len = prefix_len;
    cascade_prepare_kernel<<<1, kPlanThreads, 0, s>>>(ap, prefix_len, entries, lens);
    if (last_launch_status() != RB_OK) return RB_ERR_CUDA;
    note_launches(1);
    st = launch_prefill_tc(ap, d.head_dim, su.qmap, su.kmap, su.vmap, s);
    if (st != RB_OK) return st;
    a.cascade = kSuffixPass;
    a.seq_lens = lens;
    a.block_table = d_block_table + entries;  // every row starts at its entry `entries`
    a.kp_cap = static_cast<long long>(d.max_blocks_per_req - entries) * g.ratio;
  }
  cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
  if (num_events > 0 && cudaStreamIsCapturing(s, &capturing) != cudaSuccess) return RB_ERR_CUDA;
  const Marks mark{events, num_events, s, capturing == cudaStreamCaptureStatusActive};
  attn_plan_kernel<<<1, kPlanThreads, 0, s>>>(a, d.head_dim);
  if (last_launch_status() != RB_OK) return RB_ERR_CUDA;
  note_launches(1);
  if (!mark(0)) return RB_ERR_CUDA;
  return attn_main_impl(su, s, mark);
}

}  // namespace

extern "C" rb_status rb_paged_attention(const rb_dims* dims, int32_t num_reqs, int32_t num_tokens,
                                        int32_t num_tokens_padded, const void* d_q,
                                        const void* d_k_cache, const void* d_v_cache,
                                        const int32_t* d_block_table,
                                        const int32_t* d_query_start_loc,
                                        const int32_t* d_seq_lens, float softmax_scale,
                                        void* d_out, void* d_workspace, size_t workspace_bytes,
                                        int32_t* d_error_word, void* stream) {
  rb::CallRange range_("rb_paged_attention");
  return paged_attention_impl(dims, num_reqs, num_tokens, num_tokens_padded, d_q, d_k_cache,
                              d_v_cache, d_block_table, d_query_start_loc, d_seq_lens,
                              softmax_scale, d_out, d_workspace, workspace_bytes, d_error_word,
                              stream, nullptr, 0);
}

extern "C" rb_status rb_paged_attention_profiled(
    const rb_dims* dims, int32_t num_reqs, int32_t num_tokens, int32_t num_tokens_padded,
    const void* d_q, const void* d_k_cache, const void* d_v_cache, const int32_t* d_block_table,
    const int32_t* d_query_start_loc, const int32_t* d_seq_lens, float softmax_scale, void* d_out,
    void* d_workspace, size_t workspace_bytes, int32_t* d_error_word, void* stream,
    void* const* events, int32_t num_events) {
  rb::CallRange range_("rb_paged_attention_profiled");
  if (num_events < 0 || (num_events > 0 && events == nullptr)) return RB_ERR_INVALID_ARG;
  return paged_attention_impl(dims, num_reqs, num_tokens, num_tokens_padded, d_q, d_k_cache,
                              d_v_cache, d_block_table, d_query_start_loc, d_seq_lens,
                              softmax_scale, d_out, d_workspace, workspace_bytes, d_error_word,
                              stream, events, num_events);
}

extern "C" size_t rb_paged_attention_cascade_workspace_size(const rb_dims* dims,
                                                            int32_t max_num_reqs,
                                                            int32_t max_num_tokens) {
  if (dims == nullptr || max_num_reqs < 0 || max_num_tokens < 0 || dims->num_kv_heads < 1 ||
      dims->num_q_heads < 1 || dims->head_dim < 1)
    return 0;
  return rb::attn::cascade_layout(dims->head_dim, dims->num_q_heads, dims->num_kv_heads,
                                  max_num_reqs, max_num_tokens)
      .total;
}

extern "C" rb_status rb_paged_attention_cascade(
    const rb_dims* dims, int32_t num_reqs, int32_t num_tokens, int32_t num_tokens_padded,
    int32_t common_prefix_len, const void* d_q, const void* d_k_cache, const void* d_v_cache,
    const int32_t* d_block_table, const int32_t* d_query_start_loc, const int32_t* d_seq_lens,
    float softmax_scale, void* d_out, void* d_workspace, size_t workspace_bytes,
    int32_t* d_error_word, void* stream) {
  rb::CallRange range_("rb_paged_attention_cascade");
  return paged_attention_impl(dims, num_reqs, num_tokens, num_tokens_padded, d_q, d_k_cache,
                              d_v_cache, d_block_table, d_query_start_loc, d_seq_lens,
                              softmax_scale, d_out, d_workspace, workspace_bytes, d_error_word,
                              stream, nullptr, 0, common_prefix_len);
}

extern "C" int32_t rb_cascade_prefix_len(int32_t shared_prefix_tokens,
                                         const int32_t* num_computed, int32_t num_reqs,
                                         int32_t block_size) {
  if (shared_prefix_tokens < 0 || num_reqs < 0 || block_size < 1 ||
      (num_reqs > 0 && num_computed == nullptr))
    return -1;
  if (num_reqs == 0) return 0;
  int32_t p = shared_prefix_tokens;
  for (int32_t i = 0; i < num_reqs; ++i) {
    if (num_computed[i] < 0) return -1;
    p = num_computed[i] < p ? num_computed[i] : p;
  }
  return p / block_size * block_size;
}
