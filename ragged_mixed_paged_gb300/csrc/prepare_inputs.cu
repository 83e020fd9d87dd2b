// rb_prepare_inputs: flat step inputs and attention metadata of one mixed batch, one kernel.
//
// What it computes ("vLLM 源码完全拆解（五）：GPUModelRunner 如何把动态请求拼成一次 GPU 前向",
// sections 第一步 .. 第四步, "Block table 是逐请求的页表", "固定地址与动态有效长度如何共存"):
//   query_start_loc = exclusive prefix sum of num_scheduled (tail = N for padded requests)
//   seq_lens[i]     = num_computed[i] + num_scheduled[i]           (0 for padded requests)
//   positions[t]    = num_computed[r] + (t - query_start_loc[r])   (r = owner of token t)
//   input_ids[t]    = token_table[r, positions[t]]
//   slot_mapping[t] = page(r, pos / B) * B + pos % B                  (padding -> null page)
//                     page(r, j) = block_table[r, j / ratio] * ratio + j % ratio: the table
//                     may hold manager blocks of `ratio` kernel pages ("混合 KV Cache：一条请求
//                     不止一张页表"); ratio 1 reads kernel pages directly
//   logits_indices  = query_start_loc[1:] - 1
//   is_prefilling   = num_computed < num_prompt, discard_request_mask = seq_len < num_prompt
//                     (optional; "Chunked Prefill：query 很长，但仍只是一段区间")
//
// Design: the per-request arrays are tiny, so every CTA recomputes the prefix sum of
// num_scheduled in shared memory (warp-shuffle scan) instead of waiting on a second launch;
// then each thread expands 4 consecutive tokens (binary search for the owner of the first,
// linear advance for the rest) and writes them with 16-byte stores.  CTA 0 also writes the
// per-request outputs and the scalar reductions.
#include "rb_internal.cuh"

namespace rb {
namespace {

constexpr int kThreads = 256;
constexpr int kTokPerThread = 4;
constexpr int kTokPerCta = kThreads * kTokPerThread;
constexpr int kMaxReqs = 16384;

struct PrepArgs {
  int R, R_pad, N, N_pad, B, M, MB, num_blocks, null_block, ratio;
  const int32_t* __restrict__ token_table;
  const int32_t* __restrict__ num_computed;
  const int32_t* __restrict__ num_scheduled;
  const int32_t* __restrict__ block_table;
  int32_t* input_ids;
  int32_t* positions;
  int32_t* qsl;
  int32_t* seq_lens;
  int32_t* slots;
  int32_t* logits;
  int32_t* scalars;
  const int32_t* __restrict__ num_prompt;  // optional: phase flags below
  int32_t* is_prefilling;
  int32_t* discard;
};

// Exclusive prefix sum of num_scheduled[0..R) into s_qsl[0..R] (s_qsl[R] = total).
__device__ void block_scan_scheduled(const PrepArgs& a, int32_t* s_qsl) {
  __shared__ int32_t s_warp[kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (a.R + kThreads - 1) / kThreads;
  const int lo = min(tid * per, a.R), hi = min(lo + per, a.R);
  uint32_t sum = 0;
  for (int i = lo; i < hi; ++i) sum += static_cast<uint32_t>(a.num_scheduled[i]);
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[warp] = static_cast<int32_t>(incl);
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kThreads / 32 ? static_cast<uint32_t>(s_warp[lane]) : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    if (lane < kThreads / 32) s_warp[lane] = static_cast<int32_t>(w);
  }
  __syncthreads();
  uint32_t run = incl - sum + (warp > 0 ? static_cast<uint32_t>(s_warp[warp - 1]) : 0u);
  for (int i = lo; i < hi; ++i) {
    s_qsl[i] = static_cast<int32_t>(run);
    run += static_cast<uint32_t>(a.num_scheduled[i]);
  }
  if (tid == 0) s_qsl[a.R] = s_warp[kThreads / 32 - 1];
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) prepare_inputs_kernel(PrepArgs a) {
  extern __shared__ int32_t s_qsl[];  // [R + 1]
  __shared__ int32_t s_max_q, s_max_len;
  int32_t* err = a.scalars + 3;
  block_scan_scheduled(a, s_qsl);
  const int total = s_qsl[a.R];
  const int tid = threadIdx.x;

  // ---- per-request outputs and scalar reductions (CTA 0) ----
  if (blockIdx.x == 0) {
    if (tid == 0) { s_max_q = 0; s_max_len = 0; }
    __syncthreads();
    int my_q = 0, my_len = 0, bits = 0;
    for (int i = tid; i < a.R_pad + 1; i += kThreads) a.qsl[i] = i <= a.R ? s_qsl[i] : a.N;
    for (int i = tid; i < a.R_pad; i += kThreads) {
      if (i < a.R) {
        const int c = a.num_computed[i], q = a.num_scheduled[i];
        const long long len = static_cast<long long>(c) + q;
        if (q < 1) bits |= RB_EBIT_NUM_SCHEDULED;
        if (c < 0) bits |= RB_EBIT_NUM_COMPUTED;
        if (len > a.M || (len + a.B - 1) / a.B > static_cast<long long>(a.MB) * a.ratio)
          bits |= RB_EBIT_SEQ_LEN;
        a.seq_lens[i] = static_cast<int32_t>(len);
        a.logits[i] = s_qsl[i + 1] - 1;
        my_q = max(my_q, q);
        my_len = max(my_len, static_cast<int>(len));
        if (a.is_prefilling != nullptr) {  // "Chunked Prefill": phase from computed vs prompt
          const int p = a.num_prompt[i];
          a.is_prefilling[i] = c < p ? 1 : 0;
          a.discard[i] = len < p ? 1 : 0;
        }
      } else {
        a.seq_lens[i] = 0;
        a.logits[i] = max(a.N - 1, 0);
        if (a.is_prefilling != nullptr) {
          a.is_prefilling[i] = 0;
          a.discard[i] = 1;
        }
      }
    }
    if (tid == 0 && total != a.N) bits |= RB_EBIT_TOKEN_SUM;
    if (bits) raise_error(err, bits);
    atomicMax(&s_max_q, my_q);
    atomicMax(&s_max_len, my_len);
    __syncthreads();
    if (tid == 0) {
      a.scalars[0] = s_max_q;
      a.scalars[1] = s_max_len;
      a.scalars[2] = a.N;
    }
  }

  // ---- per-token expansion ----
  const int t0 = blockIdx.x * kTokPerCta + tid * kTokPerThread;
  if (t0 >= a.N_pad) return;
  int ids[kTokPerThread], pos[kTokPerThread], slot[kTokPerThread];
  int bits = 0;
  const int n_real = min(a.N, total);
  int r = -1;
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) {
    const int t = t0 + k;
    ids[k] = 0;
    pos[k] = 0;
    slot[k] = a.null_block * a.B + ((t - a.N) % a.B + a.B) % a.B;
    if (t >= a.N_pad) continue;
    if (t >= a.N) continue;  // padding token -> null page
    if (t >= n_real) {       // sum(num_scheduled) < N: no owner
      bits |= RB_EBIT_TOKEN_SUM;
      slot[k] = a.null_block * a.B;
      continue;
    }
    if (r < 0) {
      r = upper_bound_i32(s_qsl, a.R + 1, t) - 1;
    } else {
      while (r + 1 <= a.R && s_qsl[r + 1] <= t) ++r;
    }
    if (r < 0 || r >= a.R) { bits |= RB_EBIT_NUM_SCHEDULED; r = -1; slot[k] = a.null_block * a.B; continue; }
    const int j = t - s_qsl[r];
    const int c = a.num_computed[r];
    const long long p = static_cast<long long>(c) + j;
    if (j < 0 || p < 0 || p >= a.M || p / a.B >= static_cast<long long>(a.MB) * a.ratio) {
      bits |= RB_EBIT_SEQ_LEN;
      slot[k] = a.null_block * a.B;
      continue;
    }
    const int pp = static_cast<int>(p);
    pos[k] = pp;
    ids[k] = a.token_table[static_cast<size_t>(r) * a.M + pp];
    const int blk = kernel_page(a.block_table + static_cast<size_t>(r) * a.MB, pp / a.B,
                                a.ratio, a.num_blocks, a.null_block);
    if (blk < 0) {
      bits |= RB_EBIT_BLOCK_ID;
      slot[k] = a.null_block * a.B + pp % a.B;
    } else {
      slot[k] = blk * a.B + pp % a.B;
    }
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
  using namespace rb;
  if (dims == nullptr || d_query_start_loc == nullptr || d_scalars == nullptr)
    return RB_ERR_INVALID_ARG;
  const rb_dims& d = *dims;
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

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(d_scalars + 3, 0, sizeof(int32_t), s) != cudaSuccess) return RB_ERR_CUDA;
  PrepArgs a{num_reqs, num_reqs_padded, num_tokens, num_tokens_padded, d.block_size,
             d.max_model_len, d.max_blocks_per_req, d.num_blocks, d.null_block, g.ratio,
             d_token_table, d_num_computed, d_num_scheduled, d_block_table, d_input_ids,
             d_positions, d_query_start_loc, d_seq_lens, d_slot_mapping, d_logits_indices,
             d_scalars, d_num_prompt, d_is_prefilling, d_discard_request_mask};
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
