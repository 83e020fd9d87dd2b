// rb_paged_attention_static_ws: rb_paged_attention for callers that cannot allocate device
// memory.  Such callers include code embedded in a host framework whose allocator owns every
// device byte (raw cudaMalloc would bypass its accounting), and step loops where a cudaMalloc
// or cudaFree would synchronise the device.  The attention workspace (planner header, unit
// offsets, split-KV partials) lives in a fixed array compiled into this library instead.
//
// The array is kStaticScratchBytes per device.  Every GPU that loads the library holds it until
// the process exits.  Every call on a device shares it, so calls whose work overlaps on the GPU
// (for example on two streams at once) race on it; calls must be serialised, e.g. on one stream.
// Nothing in it needs clearing between calls: the planner kernel rewrites every field the
// later kernels read.
#include <mutex>

#include "rb_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = 64ull << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_attention_scratch[kStaticScratchBytes];

// Device address of the array on the current device.  Looked up once per device, on the first
// call made with that device current; that first call should come before any stream capture.
// A symbol's address belongs to a CUDA context: the one kept here is the device's primary
// context's (the runtime's), so it does not survive cudaDeviceReset and does not hold in a
// context the caller created with the driver API.
void* scratch_for_current_device() {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attention_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" rb_status rb_paged_attention_static_ws(
    const rb_dims* dims, int32_t num_reqs, int32_t num_tokens, int32_t num_tokens_padded,
    const void* d_q, const void* d_k_cache, const void* d_v_cache, const int32_t* d_block_table,
    const int32_t* d_query_start_loc, const int32_t* d_seq_lens, float softmax_scale,
    void* d_out, int32_t* d_error_word, void* stream) {
  rb::CallRange range_("rb_paged_attention_static_ws");
  if (dims == nullptr || num_reqs < 0 || num_tokens < 0) return RB_ERR_INVALID_ARG;
  const size_t need = rb_paged_attention_workspace_size(dims, num_reqs, num_tokens);
  if (need == 0) return RB_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return RB_ERR_CAPACITY;
  void* scratch = scratch_for_current_device();
  if (scratch == nullptr) return RB_ERR_CUDA;
  return rb_paged_attention(dims, num_reqs, num_tokens, num_tokens_padded, d_q, d_k_cache,
                            d_v_cache, d_block_table, d_query_start_loc, d_seq_lens,
                            softmax_scale, d_out, scratch, kStaticScratchBytes, d_error_word,
                            stream);
}
