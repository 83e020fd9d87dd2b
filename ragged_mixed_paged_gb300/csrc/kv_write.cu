// rb_kv_write: scatter this step's K/V rows into the paged cache by slot_mapping.
//
// "vLLM 源码完全拆解（五）…", "3. 物理 KV 槽位": the t-th new K/V goes to slot_mapping[t] and the
// write needs no request id; "Nano-VLLM全代码解析笔记(4)-model_runner": slot -1 is skipped.
//
// Pure data movement, bound by HBM: each token row (nkv * hd bf16, 2 KiB for 8 x 128) is copied
// with 16-byte vector loads and stores, one 16-byte chunk per thread and iteration, K and V in
// the same thread, grid sized to a multiple of the SM count.
#include "rb_internal.cuh"

namespace rb {
namespace {

constexpr int kThreads = 256;

template <int kChunks>  // 16-byte chunks per token row (0 = runtime value)
__global__ void __launch_bounds__(kThreads)
    kv_write_kernel(int n_tokens, int chunks_rt, long long num_slots, const int4* __restrict__ k,
                    const int4* __restrict__ v, const int32_t* __restrict__ slots,
                    int4* __restrict__ kc, int4* __restrict__ vc, int32_t* err) {
  const int chunks = kChunks > 0 ? kChunks : chunks_rt;
  const long long total = static_cast<long long>(n_tokens) * chunks;
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += stride) {
    const int t = static_cast<int>(i / chunks);
    const int ch = static_cast<int>(i - static_cast<long long>(t) * chunks);
    const int s = __ldg(slots + t);
    if (s < 0) continue;
    if (s >= num_slots) {
      if (ch == 0) raise_error(err, RB_EBIT_SLOT);
      continue;
    }
    const int4 kk = __ldg(k + i);
    const int4 vv = __ldg(v + i);
    const long long dst = static_cast<long long>(s) * chunks + ch;
    kc[dst] = kk;
    vc[dst] = vv;
  }
}

}  // namespace
}  // namespace rb

extern "C" rb_status rb_kv_write(const rb_dims* dims, int32_t num_tokens_padded, const void* d_k,
                                 const void* d_v, const int32_t* d_slot_mapping, void* d_k_cache,
                                 void* d_v_cache, int32_t* d_error_word, void* stream) {
  rb::CallRange range_("rb_kv_write");
  using namespace rb;
  if (dims == nullptr || num_tokens_padded < 0) return RB_ERR_INVALID_ARG;
  const rb_dims& d = *dims;
  if (d.block_size < 1 || d.num_kv_heads < 1 || d.head_dim < 1 || d.num_blocks < 1)
    return RB_ERR_INVALID_ARG;
  const long long row_bytes = 2LL * d.num_kv_heads * d.head_dim;
  if (row_bytes % 16 != 0) return RB_ERR_UNSUPPORTED;
  if (num_tokens_padded == 0) return RB_OK;
  if (d_k == nullptr || d_v == nullptr || d_slot_mapping == nullptr || d_k_cache == nullptr ||
      d_v_cache == nullptr)
    return RB_ERR_INVALID_ARG;
  if (!aligned16(d_k) || !aligned16(d_v) || !aligned16(d_k_cache) || !aligned16(d_v_cache))
    return RB_ERR_INVALID_ARG;
  const int chunks = static_cast<int>(row_bytes / 16);
  const long long num_slots = static_cast<long long>(d.num_blocks) * d.block_size;
  const long long total = static_cast<long long>(num_tokens_padded) * chunks;
  const int sms = max(1, device_sm_count());
  const long long want = (total + kThreads - 1) / kThreads;
  const int grid = static_cast<int>(want < 16LL * sms ? want : 16LL * sms);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* k = static_cast<const int4*>(d_k);
  auto* v = static_cast<const int4*>(d_v);
  auto* kc = static_cast<int4*>(d_k_cache);
  auto* vc = static_cast<int4*>(d_v_cache);
  if (chunks == 128)
    kv_write_kernel<128><<<grid, kThreads, 0, s>>>(num_tokens_padded, chunks, num_slots, k, v,
                                                   d_slot_mapping, kc, vc, d_error_word);
  else
    kv_write_kernel<0><<<grid, kThreads, 0, s>>>(num_tokens_padded, chunks, num_slots, k, v,
                                                 d_slot_mapping, kc, vc, d_error_word);
  if (last_launch_status() != RB_OK) return RB_ERR_CUDA;
  note_launches(1);
  return RB_OK;
}
