// Shared definitions of the paged-attention kernels (planner, split-KV decode, prefill tiles,
// split combine).  Not part of the C ABI.
#pragma once

#include "rb_internal.cuh"

namespace rb {
namespace attn {

constexpr int kMaxCols = 8;          // decode columns: (query token, head of the group) pairs
constexpr int kMaxTargetUnits = 8192;
constexpr int kMinSplitPages = 8;
constexpr int kPage = 16;            // tokens per KV page (the only page size these kernels take)

enum HeaderField : int {
  kHNumDecodeUnits = 0,
  kHNumPrefillUnits = 1,
  kHDecodeNext = 2,
  kHPrefillNext = 3,
  kHSplitPages = 4,
  kHDecodeCtas = 5,  // fused kernel: CTAs that start on decode units
  kHRoleNext = 6,    // fused kernel: role ticket counter
  kHeaderInts = 32
};

// Workspace: [header][decode unit offsets R+1][prefill unit offsets R+1]
//            [finished-split counters R x nkv][prefill pair list][partial (m, l)][partial o]
struct WsLayout {
  size_t header, dec_off, pre_off, done, pre_list, part_ml, part_o, total;
  long long max_units;
};

// Prefill (request, tile pair) entries a batch can have: a pair covers 2 * (128 / group) >= 16
// query tokens for groups up to 16, so sum over requests of ceil(q_i / pair tokens)
// <= N / 16 + R.
__host__ __device__ inline long long max_prefill_pairs(int num_reqs, int num_tokens) {
  return static_cast<long long>(num_tokens) / 16 + num_reqs + 1;
}

inline WsLayout ws_layout(int head_dim, int num_kv_heads, int num_reqs, int num_tokens) {
  WsLayout w{};
  size_t off = 0;
  auto take = [&off](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~static_cast<size_t>(255);
    return o;
  };
  w.max_units = kMaxTargetUnits + static_cast<long long>(num_kv_heads) * num_reqs;
  w.header = take(kHeaderInts * sizeof(int32_t));
  w.dec_off = take(static_cast<size_t>(num_reqs + 1) * sizeof(int32_t));
  w.pre_off = take(static_cast<size_t>(num_reqs + 1) * sizeof(int32_t));
  w.done = take(static_cast<size_t>(num_reqs) * num_kv_heads * sizeof(int32_t));
  w.pre_list = take(static_cast<size_t>(max_prefill_pairs(num_reqs, num_tokens)) * sizeof(int32_t));
  w.part_ml = take(static_cast<size_t>(w.max_units) * kMaxCols * sizeof(float2));
  w.part_o = take(static_cast<size_t>(w.max_units) * kMaxCols * head_dim * sizeof(float));
  w.total = off;
  return w;
}

// Cascade attention ("第8章 ModelRunner…", "8.3.2.5 Cascade Attention"): a prefix pass runs every
// query row against the P keys all requests share (no mask: P <= every request's cached
// length), a suffix pass runs the ordinary causal attention over keys [P, seq_len) and merges
// the prefix result into each row by log-sum-exp before the single bf16 rounding.
enum CascadePass : int { kNoCascade = 0, kPrefixPass = 1, kSuffixPass = 2 };
constexpr int kMaxPrefixSplits = 4;  // the prefix keys may be cut into this many ranges

// Extra workspace of a cascade call, after the ordinary layout: shifted sequence lengths and,
// per prefix key range, the prefix pass's normalised outputs (fp32) with their log2-domain
// log-sum-exp.
struct CascadeLayout {
  size_t lens, lse, o, total;
};

inline CascadeLayout cascade_layout(int head_dim, int num_q_heads, int num_kv_heads, int num_reqs,
                                    int num_tokens) {
  CascadeLayout c{};
  size_t off = ws_layout(head_dim, num_kv_heads, num_reqs, num_tokens).total;
  auto take = [&off](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~static_cast<size_t>(255);
    return o;
  };
  c.lens = take(static_cast<size_t>(num_reqs) * sizeof(int32_t));
  c.lse = take(static_cast<size_t>(kMaxPrefixSplits) * num_tokens * num_q_heads * sizeof(float));
  c.o = take(static_cast<size_t>(kMaxPrefixSplits) * num_tokens * num_q_heads * head_dim *
             sizeof(float));
  c.total = off;
  return c;
}

struct AttnArgs {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const int32_t* block_table;
  const int32_t* qsl;
  const int32_t* seq_lens;
  int32_t* header;
  int32_t* dec_off;
  int32_t* pre_off;
  int32_t* done;  // per (request, kv head): decode splits finished so far
  int32_t* pre_list;  // tcgen05 prefill (request, pair) entries, longest first: r * 65536 + pair
  float2* part_ml;
  float* part_o;
  int R, N, N_pad, nh, nkv, group, MB, num_blocks, null_block;
  int ratio;  // kernel pages per page-table entry (manager block)
  int target_units;
  int tile_tokens;  // query tokens per 128-row tcgen05 tile: 128 / group (whole tokens only)
  int fused_ctas;  // > 0: decode and prefill share one launch of this many CTAs (one per SM)
  int decode_warps_per_cta;  // decode warps per CTA in the launch that runs decode units
  float scale_log2;
  int32_t* err;
  long long kp_cap;   // kernel pages a row may span (max_blocks_per_req * ratio, less a shift)
  int cascade;        // CascadePass
  int prefix_len;     // prefix pass: the shared keys [0, P) of row 0
  int prefix_splits;  // key ranges of the prefix pass (1 .. kMaxPrefixSplits)
  int prefix_split_keys;  // keys per range (a multiple of 128)
  float* pre_o;       // [splits, N, nh, HD] prefix-pass outputs per key range, normalised
  float* pre_lse;     // [splits, N, nh] their log-sum-exp (log2 units of the scaled scores)
  // limit of the fused launch's bounded waits, and (tests only) CTA 0's producer withholding
  // the arrival of its first prefill unit so that the waits for it run out
  unsigned long long wait_limit_ns;
  int withhold_first_unit;
};

// Test hook behind rb_debug_attention_wait_limit: the wait limit and withhold flag of every
// later attention call (process-wide).
void debug_wait_settings(unsigned long long* limit_ns, int* withhold);

// Weights that merge a suffix-pass row (accumulator relative to running max m, sum l; log2
// units) with the prefix-pass rows of the same (token, head) (one per key range: log-sum-exp
// lse_s, normalised o_s): out = acc * (return value) + sum_s o_s * w[s].
__device__ __forceinline__ float cascade_weights(const AttnArgs& a, size_t row, float m, float l,
                                                 float* w) {
  const size_t stride = static_cast<size_t>(a.N) * a.nh;
  float lse[kMaxPrefixSplits];
  float mx = l > 0.f ? m : -INFINITY;
#pragma unroll
  for (int s = 0; s < kMaxPrefixSplits; ++s) {
    lse[s] = s < a.prefix_splits ? __ldg(a.pre_lse + s * stride + row) : -INFINITY;
    mx = fmaxf(mx, lse[s]);
  }
  if (mx == -INFINITY) {
#pragma unroll
    for (int s = 0; s < kMaxPrefixSplits; ++s) w[s] = 0.f;
    return 0.f;
  }
  const float wa = l > 0.f ? fast_exp2(m - mx) : 0.f;
  float den = l * wa;
#pragma unroll
  for (int s = 0; s < kMaxPrefixSplits; ++s) {
    w[s] = lse[s] == -INFINITY ? 0.f : fast_exp2(lse[s] - mx);
    den += w[s];
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
  for (int s = 0; s < kMaxPrefixSplits; ++s) w[s] *= inv;
  return wa * inv;
}

// Prefix-pass output row of key range s for (token, head) row `row`.
template <int HD>
__device__ __forceinline__ const float* cascade_row(const AttnArgs& a, int s, size_t row) {
  return a.pre_o + (static_cast<size_t>(s) * a.N * a.nh + row) * HD;
}

// Request classes shared by the planner and the kernels.
__host__ __device__ inline bool is_decode_class(int q, int group) {
  return q >= 1 && q * group <= kMaxCols;
}

// Host side of one attention call: checked arguments, kernel arguments and TMA descriptors.
struct AttnSetup {
  AttnArgs a;
  PageGeom g;
  int head_dim, num_kv_heads;
  const void* k_cache;
  const void* v_cache;
  long long num_slots;
  CUtensorMap qmap, kmap, vmap;
};

// Host checks and kernel arguments of rb_paged_attention (no launch, no driver call).
rb_status attn_setup(const rb_dims* dims, int32_t num_reqs, int32_t num_tokens,
                     int32_t num_tokens_padded, const void* d_q, const void* d_k_cache,
                     const void* d_v_cache, const int32_t* d_block_table,
                     const int32_t* d_query_start_loc, const int32_t* d_seq_lens,
                     float softmax_scale, void* d_out, void* d_workspace, size_t workspace_bytes,
                     int32_t* d_error_word, AttnSetup* su);
// Encodes the TMA descriptors of a set-up call.
rb_status attn_encode_maps(AttnSetup* su);
// Enqueues what follows the planner: the fused decode + prefill launch.
rb_status attn_main(const AttnSetup& su, cudaStream_t s);

rb_status launch_prefill_tc(const AttnArgs& a, int head_dim, const CUtensorMap& qmap,
                            const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t s);

}  // namespace attn
}  // namespace rb
