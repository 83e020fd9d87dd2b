// Host-side pieces of librb: status strings, launch counting, SM counts, TMA descriptors and
// rb_pad_for_graph.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "rb_internal.cuh"

namespace rb {

static std::atomic<uint64_t> g_launches{0};

// rb_debug_attention_wait_limit's settings (defaults: 1 s, nothing withheld)
constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;
static std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
static std::atomic<int> g_withhold{0};

void note_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }

namespace attn {
void debug_wait_settings(unsigned long long* limit_ns, int* withhold) {
  *limit_ns = g_wait_limit_ns.load();
  *withhold = g_withhold.load();
}
}  // namespace attn

int device_sm_count() {
  static std::mutex mu;
  static int counts[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      counts[dev] = n;
  }
  return counts[dev];
}

rb_status last_launch_status() {
  return cudaGetLastError() == cudaSuccess ? RB_OK : RB_ERR_CUDA;
}

rb_status page_geom_of(const rb_dims& d, PageGeom* g) {
  const int r = d.kernel_blocks_per_manager_block == 0 ? 1 : d.kernel_blocks_per_manager_block;
  if (r < 1 || r > 64 || d.num_blocks < 1 || d.null_block < 0 || d.null_block >= d.num_blocks ||
      d.num_blocks % r != 0 || d.null_block % r != 0 || d.max_blocks_per_req < 1 ||
      static_cast<long long>(d.max_blocks_per_req) * r > 0x7fffffffLL)
    return RB_ERR_INVALID_ARG;
  g->ratio = r;
  g->num_blocks = d.num_blocks;
  g->null_block = d.null_block;
  return RB_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_kv_tensor_map(CUtensorMap* map, const void* base, int head_dim, int num_kv_heads,
                          long long num_slots) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim),
                              static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(num_slots)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                 static_cast<cuuint64_t>(head_dim) * num_kv_heads * 2};
  const cuuint32_t box[3] = {64, 1, 16};
  const cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_q_tensor_map(CUtensorMap* map, const void* base, int head_dim, int num_q_heads,
                         long long num_tokens, int group) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr || group < 1 || group > 128) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim),
                              static_cast<cuuint64_t>(num_q_heads),
                              static_cast<cuuint64_t>(num_tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                 static_cast<cuuint64_t>(head_dim) * num_q_heads * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group),
                             static_cast<cuuint32_t>(128 / group)};
  const cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace rb

extern "C" {

const char* rb_status_string(int32_t status) {
  switch (status) {
    case RB_OK: return "ok";
    case RB_ERR_INVALID_ARG: return "invalid argument";
    case RB_ERR_CAPACITY: return "capacity exceeded";
    case RB_ERR_CUDA: return "CUDA runtime error";
    case RB_ERR_UNSUPPORTED: return "unsupported shape";
    default: return "unknown status";
  }
}

uint64_t rb_kernel_launch_count(void) { return rb::g_launches.load(); }

rb_status rb_debug_attention_wait_limit(uint64_t wait_limit_ns, int32_t withhold_first_unit) {
  if (withhold_first_unit < 0 || withhold_first_unit > 1) return RB_ERR_INVALID_ARG;
  if (wait_limit_ns != 0 && (wait_limit_ns < 100000ull || wait_limit_ns > 10000000000ull))
    return RB_ERR_INVALID_ARG;
  rb::g_wait_limit_ns.store(wait_limit_ns == 0 ? rb::kDefaultWaitLimitNs : wait_limit_ns);
  rb::g_withhold.store(withhold_first_unit);
  return RB_OK;
}

int32_t rb_pad_for_graph(const int32_t* capture_sizes, int32_t num_sizes, int32_t num_tokens) {
  if (num_sizes < 0 || num_tokens < 0 || (num_sizes > 0 && capture_sizes == nullptr)) return -1;
  for (int32_t i = 1; i < num_sizes; ++i)
    if (capture_sizes[i] < capture_sizes[i - 1]) return -1;
  if (num_sizes == 0 || num_tokens > capture_sizes[num_sizes - 1]) return num_tokens;
  int32_t lo = 0, hi = num_sizes;  // first size >= num_tokens
  while (lo < hi) {
    const int32_t mid = lo + (hi - lo) / 2;
    if (capture_sizes[mid] < num_tokens) lo = mid + 1; else hi = mid;
  }
  return capture_sizes[lo];
}

}  // extern "C"
