// rb_prepare_inputs: flat step inputs and attention metadata of one mixed batch, one kernel.
//
// What it computes: see prep_common.cuh ("vLLM 源码完全拆解（五）…", 第一步 .. 第四步).
//
// Design: the per-request arrays are tiny, so every CTA recomputes the prefix sum of
// num_scheduled in shared memory (warp-shuffle scan) instead of waiting on a second launch;
// then each thread expands 4 consecutive tokens (binary search for the owner of the first,
// linear advance for the rest) and writes them with 16-byte stores.  CTA 0 also writes the
// per-request outputs and the scalar reductions.
#include "prep_common.cuh"

namespace rb {
namespace prep {

rb_status prep_args_of(const rb_dims& d, int32_t num_reqs, int32_t num_reqs_padded,
                       int32_t num_tokens, int32_t num_tokens_padded,
                       const int32_t* d_token_table, const int32_t* d_num_computed,
                       const int32_t* d_num_scheduled, const int32_t* d_block_table,
                       int32_t* d_input_ids, int32_t* d_positions, int32_t* d_query_start_loc,
                       int32_t* d_seq_lens, int32_t* d_slot_mapping, int32_t* d_logits_indices,
                       int32_t* d_scalars, const int32_t* d_num_prompt, int32_t* d_is_prefilling,
                       int32_t* d_discard_request_mask, PrepArgs* a) {
  if (d_query_start_loc == nullptr || d_scalars == nullptr) return RB_ERR_INVALID_ARG;
  PageGeom g;
  if (d.block_size < 1 || d.max_num_reqs < 0 || d.max_model_len < 1 ||
      page_geom_of(d, &g) != RB_OK)
    return RB_ERR_INVALID_ARG;
  if (static_cast<long long>(d.num_blocks) * d.block_size > 0x7fffffffLL) return RB_ERR_CAPACITY;
  if (num_reqs < 0 || num_reqs_padded < num_reqs || num_tokens < 0 ||
      num_tokens_padded < num_tokens)
    return RB_ERR_INVALID_ARG;
  if (num_reqs_padded > d.max_num_reqs) return RB_ERR_CAPACITY;
  if (num_reqs_padded > 0 && num_tokens_padded < 1) return RB_ERR_INVALID_ARG;
  if (num_reqs > kMaxReqs) return RB_ERR_UNSUPPORTED;
  if (num_reqs > 0 && (d_token_table == nullptr || d_num_computed == nullptr ||
                       d_num_scheduled == nullptr || d_block_table == nullptr))
    return RB_ERR_INVALID_ARG;
  if (num_reqs_padded > 0 && (d_seq_lens == nullptr || d_logits_indices == nullptr))
    return RB_ERR_INVALID_ARG;
  if (num_tokens_padded > 0 &&
      (d_input_ids == nullptr || d_positions == nullptr || d_slot_mapping == nullptr))
    return RB_ERR_INVALID_ARG;
  // phase flags are written when both flag outputs are given (prompt lengths then needed)
  const bool flags = d_is_prefilling != nullptr || d_discard_request_mask != nullptr;
  if (flags && (d_is_prefilling == nullptr || d_discard_request_mask == nullptr ||
                (num_reqs > 0 && d_num_prompt == nullptr)))
    return RB_ERR_INVALID_ARG;
  *a = PrepArgs{num_reqs, num_reqs_padded, num_tokens, num_tokens_padded, d.block_size,
                d.max_model_len, d.max_blocks_per_req, d.num_blocks, d.null_block, g.ratio,
                d_token_table, d_num_computed, d_num_scheduled, d_block_table, d_input_ids,
                d_positions, d_query_start_loc, d_seq_lens, d_slot_mapping, d_logits_indices,
                d_scalars, d_num_prompt, d_is_prefilling, d_discard_request_mask};
  return RB_OK;
}

namespace {

constexpr int kTokPerThread = 4;
constexpr int kTokPerCta = kThreads * kTokPerThread;

__global__ void __launch_bounds__(kThreads) prepare_inputs_kernel(PrepArgs a) {
  extern __shared__ int32_t s_qsl[];  // [R + 1]
  int32_t* err = a.scalars + 3;
  block_scan_scheduled(a, s_qsl);
  const int total = s_qsl[a.R];
  if (blockIdx.x == 0) request_outputs(a, s_qsl, total, err);

  // ---- per-token expansion ----
  const int t0 = blockIdx.x * kTokPerCta + threadIdx.x * kTokPerThread;
  if (t0 >= a.N_pad) return;
  int ids[kTokPerThread], pos[kTokPerThread], slot[kTokPerThread];
  int bits = 0;
  const int n_real = min(a.N, total);
  int r = -1;
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) {
    const int t = t0 + k;
    ids[k] = pos[k] = slot[k] = 0;
    if (t >= a.N_pad) continue;
    const TokMeta m = token_meta(a, s_qsl, n_real, t, r);
    ids[k] = m.id;
    pos[k] = m.pos;
    slot[k] = m.slot;
    bits |= m.bits;
  }
  if (bits) raise_error(err, bits);
  const bool vec = (t0 + kTokPerThread <= a.N_pad) && aligned16(a.input_ids) &&
                   aligned16(a.positions) && aligned16(a.slots);
  if (vec) {
    *reinterpret_cast<int4*>(a.input_ids + t0) = make_int4(ids[0], ids[1], ids[2], ids[3]);
    *reinterpret_cast<int4*>(a.positions + t0) = make_int4(pos[0], pos[1], pos[2], pos[3]);
    *reinterpret_cast<int4*>(a.slots + t0) = make_int4(slot[0], slot[1], slot[2], slot[3]);
  } else {
#pragma unroll
    for (int k = 0; k < kTokPerThread; ++k) {
      if (t0 + k < a.N_pad) {
        a.input_ids[t0 + k] = ids[k];
        a.positions[t0 + k] = pos[k];
        a.slots[t0 + k] = slot[k];
      }
    }
  }
}

}  // namespace
}  // namespace prep
}  // namespace rb

extern "C" rb_status rb_prepare_inputs(const rb_dims* dims, int32_t num_reqs,
                                       int32_t num_reqs_padded, int32_t num_tokens,
                                       int32_t num_tokens_padded, const int32_t* d_token_table,
                                       const int32_t* d_num_computed,
                                       const int32_t* d_num_scheduled,
                                       const int32_t* d_block_table, int32_t* d_input_ids,
                                       int32_t* d_positions, int32_t* d_query_start_loc,
                                       int32_t* d_seq_lens, int32_t* d_slot_mapping,
                                       int32_t* d_logits_indices, int32_t* d_scalars,
                                       const int32_t* d_num_prompt, int32_t* d_is_prefilling,
                                       int32_t* d_discard_request_mask, void* stream) {
  rb::CallRange range_("rb_prepare_inputs");
  using namespace rb;
  using namespace rb::prep;
  if (dims == nullptr) return RB_ERR_INVALID_ARG;
  PrepArgs a;
  const rb_status st = prep_args_of(
      *dims, num_reqs, num_reqs_padded, num_tokens, num_tokens_padded, d_token_table,
      d_num_computed, d_num_scheduled, d_block_table, d_input_ids, d_positions,
      d_query_start_loc, d_seq_lens, d_slot_mapping, d_logits_indices, d_scalars, d_num_prompt,
      d_is_prefilling, d_discard_request_mask, &a);
  if (st != RB_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(d_scalars + 3, 0, sizeof(int32_t), s) != cudaSuccess) return RB_ERR_CUDA;
  const size_t smem = static_cast<size_t>(num_reqs + 1) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(prepare_inputs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return RB_ERR_CUDA;
  }
  const int grid = max(1, (num_tokens_padded + kTokPerCta - 1) / kTokPerCta);
  prepare_inputs_kernel<<<grid, kThreads, smem, s>>>(a);
  if (last_launch_status() != RB_OK) return RB_ERR_CUDA;
  note_launches(1);
  return RB_OK;
}
