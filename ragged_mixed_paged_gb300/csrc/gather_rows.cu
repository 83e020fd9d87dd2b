// rb_gather_rows: out[i, :] = hidden[indices[i], :] — the rows the LM head needs.
//
// "vLLM 源码完全拆解（五）…", "第四步：只在必要位置计算 logits"; "04 · 模型执行与 CUDA Graph",
// step ⑤ (hidden_states[logits_indices]).  A 16-byte vectorised row copy, bound by HBM.
#include "rb_internal.cuh"

namespace rb {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    gather_rows_kernel(int num_rows, int chunks, int num_hidden_rows,
                       const int4* __restrict__ hidden, const int32_t* __restrict__ idx,
                       int4* __restrict__ out, int32_t* err) {
  const long long total = static_cast<long long>(num_rows) * chunks;
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += stride) {
    const int row = static_cast<int>(i / chunks);
    const int ch = static_cast<int>(i - static_cast<long long>(row) * chunks);
    const int src = __ldg(idx + row);
    int4 val = make_int4(0, 0, 0, 0);
    if (src < 0 || src >= num_hidden_rows) {
      if (ch == 0) raise_error(err, RB_EBIT_ROW_INDEX);
    } else {
      val = __ldg(hidden + static_cast<long long>(src) * chunks + ch);
    }
    out[i] = val;
  }
}

}  // namespace
}  // namespace rb

extern "C" rb_status rb_gather_rows(int32_t num_rows, int32_t hidden_size, int32_t num_hidden_rows,
                                    const void* d_hidden, const int32_t* d_indices, void* d_out,
                                    int32_t* d_error_word, void* stream) {
  rb::CallRange range_("rb_gather_rows");
  using namespace rb;
  if (num_rows < 0 || hidden_size < 1 || num_hidden_rows < 0) return RB_ERR_INVALID_ARG;
  if ((2LL * hidden_size) % 16 != 0) return RB_ERR_UNSUPPORTED;
  if (num_rows == 0) return RB_OK;
  if (d_hidden == nullptr || d_indices == nullptr || d_out == nullptr) return RB_ERR_INVALID_ARG;
  if (!aligned16(d_hidden) || !aligned16(d_out)) return RB_ERR_INVALID_ARG;
  const int chunks = static_cast<int>(2LL * hidden_size / 16);
  const long long total = static_cast<long long>(num_rows) * chunks;
  const int sms = max(1, device_sm_count());
  const long long want = (total + kThreads - 1) / kThreads;
  const int grid = static_cast<int>(want < 8LL * sms ? want : 8LL * sms);
  gather_rows_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      num_rows, chunks, num_hidden_rows, static_cast<const int4*>(d_hidden), d_indices,
      static_cast<int4*>(d_out), d_error_word);
  if (last_launch_status() != RB_OK) return RB_ERR_CUDA;
  note_launches(1);
  return RB_OK;
}
