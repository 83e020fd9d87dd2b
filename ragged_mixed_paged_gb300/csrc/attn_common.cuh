// Shared definitions of the paged-attention kernels (planner, split-KV decode, prefill tiles,
// split combine).  Not part of the C ABI.
#pragma once

#include "rb_internal.cuh"

namespace rb {
namespace attn {

constexpr int kMaxCols = 8;          // decode columns: (query token, head of the group) pairs
constexpr int kPrefillTileM = 64;    // query rows per mma.sync prefill tile
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
//            [finished-split counters R x nkv][partial (m, l)][partial o]
struct WsLayout {
  size_t header, dec_off, pre_off, done, part_ml, part_o, total;
  long long max_units;
};

inline WsLayout ws_layout(int head_dim, int num_kv_heads, int num_reqs) {
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
  w.part_ml = take(static_cast<size_t>(w.max_units) * kMaxCols * sizeof(float2));
  w.part_o = take(static_cast<size_t>(w.max_units) * kMaxCols * head_dim * sizeof(float));
  w.total = off;
  return w;
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
  float2* part_ml;
  float* part_o;
  int R, N, N_pad, nh, nkv, group, MB, num_blocks, null_block;
  int ratio;  // kernel pages per page-table entry (manager block)
  int target_units;
  int tile_m;  // query rows per prefill unit (256 on the tcgen05 path, 64 on the mma.sync path)
  int fused_ctas;  // > 0: decode and prefill share one launch of this many CTAs (one per SM)
  int decode_warps_per_cta;  // decode warps per CTA in the launch that runs decode units
  float scale_log2;
  int32_t* err;
};

// Request classes shared by the planner and the kernels.
__host__ __device__ inline bool is_decode_class(int q, int group) {
  return q >= 1 && q * group <= kMaxCols;
}

rb_status launch_decode(const AttnArgs& a, int head_dim, const CUtensorMap& kmap,
                        const CUtensorMap& vmap, cudaStream_t s);
rb_status launch_prefill(const AttnArgs& a, int head_dim, const CUtensorMap& kmap,
                         const CUtensorMap& vmap, cudaStream_t s);
bool prefill_tc_supported(int head_dim, int group);
rb_status launch_prefill_tc(const AttnArgs& a, int head_dim, const CUtensorMap& qmap,
                            const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t s);

}  // namespace attn
}  // namespace rb
