// Shared device code of the step-preparation kernels (rb_prepare_inputs and the fused step):
// the in-CTA prefix sum of num_scheduled, the per-request outputs and the per-token expansion.
// Not part of the C ABI.
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
#pragma once

#include "rb_internal.cuh"

namespace rb {
namespace prep {

constexpr int kThreads = 256;  // every preparation CTA
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
__device__ __forceinline__ void block_scan_scheduled(const PrepArgs& a, int32_t* s_qsl) {
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

// Per-request outputs and the scalar reductions (one CTA, all of its threads).
__device__ __forceinline__ void request_outputs(const PrepArgs& a, const int32_t* s_qsl,
                                                int total, int32_t* err) {
  __shared__ int32_t s_max_q, s_max_len;
  const int tid = threadIdx.x;
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
  __syncthreads();
}

struct TokMeta {
  int id, pos, slot, bits;
};

// Input id, position, slot and error bits of flat token t.  `r` is the owner found for the
// previous token this thread expanded (-1: none yet); tokens must come in increasing order.
__device__ __forceinline__ TokMeta token_meta(const PrepArgs& a, const int32_t* s_qsl,
                                              int n_real, int t, int& r) {
  TokMeta m{0, 0, a.null_block * a.B + ((t - a.N) % a.B + a.B) % a.B, 0};
  if (t >= a.N) return m;  // padding token -> null page
  if (t >= n_real) {       // sum(num_scheduled) < N: no owner
    m.bits = RB_EBIT_TOKEN_SUM;
    m.slot = a.null_block * a.B;
    return m;
  }
  if (r < 0) {
    r = upper_bound_i32(s_qsl, a.R + 1, t) - 1;
  } else {
    while (r + 1 <= a.R && s_qsl[r + 1] <= t) ++r;
  }
  if (r < 0 || r >= a.R) {
    m.bits = RB_EBIT_NUM_SCHEDULED;
    r = -1;
    m.slot = a.null_block * a.B;
    return m;
  }
  const int j = t - s_qsl[r];
  const int c = a.num_computed[r];
  const long long p = static_cast<long long>(c) + j;
  if (j < 0 || p < 0 || p >= a.M || p / a.B >= static_cast<long long>(a.MB) * a.ratio) {
    m.bits = RB_EBIT_SEQ_LEN;
    m.slot = a.null_block * a.B;
    return m;
  }
  const int pp = static_cast<int>(p);
  m.pos = pp;
  m.id = a.token_table[static_cast<size_t>(r) * a.M + pp];
  const int blk = kernel_page(a.block_table + static_cast<size_t>(r) * a.MB, pp / a.B, a.ratio,
                              a.num_blocks, a.null_block);
  if (blk < 0) {
    m.bits = RB_EBIT_BLOCK_ID;
    m.slot = a.null_block * a.B + pp % a.B;
  } else {
    m.slot = blk * a.B + pp % a.B;
  }
  return m;
}

// Host-side checks shared by rb_prepare_inputs and rb_step; fills `a` (outputs included).
rb_status prep_args_of(const rb_dims& d, int32_t num_reqs, int32_t num_reqs_padded,
                       int32_t num_tokens, int32_t num_tokens_padded,
                       const int32_t* d_token_table, const int32_t* d_num_computed,
                       const int32_t* d_num_scheduled, const int32_t* d_block_table,
                       int32_t* d_input_ids, int32_t* d_positions, int32_t* d_query_start_loc,
                       int32_t* d_seq_lens, int32_t* d_slot_mapping, int32_t* d_logits_indices,
                       int32_t* d_scalars, const int32_t* d_num_prompt, int32_t* d_is_prefilling,
                       int32_t* d_discard_request_mask, PrepArgs* a);

}  // namespace prep
}  // namespace rb
