// Split-KV decode attention (requests whose query_len * group <= 8), HBM-streaming.
//
// Work unit = (request, kv head, split of pages); one warp per unit, units pulled from an
// atomic counter by a persistent grid.  Each warp owns a ring of shared-memory stages; lane 0
// issues TMA loads (3-D tensor map, one {64 dims x 16 slots} box per 128-byte half of a page,
// 128B swizzle) and the warp waits on the stage's mbarrier with a bounded wait.
//
// The contraction runs transposed so a 16-token page is one MMA tile:
//   S^T[16 keys, 8 cols] = K[16, hd] . Q^T[hd, 8]     cols = (query token, head of the group)
//   O^T[hd, 8 cols]     += V^T[hd, 16] . P^T[16, 8]
// with mma.sync m16n8k16 (bf16 in, fp32 accumulate).  P^T's fragments come from S^T's with a
// register transpose (movmatrix), so each page costs 2 x hd/16 MMAs and every K/V byte is read
// once per kv head, shared by the whole query-head group.  Softmax statistics are per column,
// reduced with warp shuffles; a unit with several splits leaves (m, l, o) partials and the last
// split of its (request, kv head) to finish merges them; a single-split unit writes the
// normalised bf16 output directly.
#include "attn_decode_warp.cuh"

namespace rb {
namespace attn {
namespace {

template <int HD>
__global__ void __launch_bounds__(DecCfg<HD>::kWarps * 32)
    attn_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  using C = DecCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[C::kWarps][C::kStages];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  const uint32_t wbase = base_u32 + warp * C::kStages * C::kStageBytes;
  uint8_t* wbase_ptr = smem_raw + (wbase - raw_u32);
  if (lane == 0) {
    for (int s = 0; s < C::kStages; ++s) mbar_init(&bars[warp][s], 1);
    fence_barrier_init();
  }
  __syncwarp();
  decode_warp<HD>(&kmap, &vmap, a, bars[warp], wbase, wbase_ptr, -1);
}

template <int HD>
rb_status launch_decode_hd(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           cudaStream_t s) {
  using C = DecCfg<HD>;
  static int blocks_per_sm[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RB_ERR_CUDA;
  if (blocks_per_sm[dev] == 0) {
    if (cudaFuncSetAttribute(attn_decode_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return RB_ERR_CUDA;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_decode_kernel<HD>, C::kWarps * 32,
                                                      C::kSmemBytes) != cudaSuccess ||
        n < 1)
      return RB_ERR_CUDA;
    blocks_per_sm[dev] = n;
  }
  const int grid = max(1, device_sm_count()) * blocks_per_sm[dev];
  attn_decode_kernel<HD><<<grid, C::kWarps * 32, C::kSmemBytes, s>>>(kmap, vmap, a);
  if (last_launch_status() != RB_OK) return RB_ERR_CUDA;
  note_launches(1);
  return RB_OK;
}

}  // namespace

rb_status launch_decode(const AttnArgs& a, int head_dim, const CUtensorMap& kmap,
                        const CUtensorMap& vmap, cudaStream_t s) {
  return head_dim == 128 ? launch_decode_hd<128>(a, kmap, vmap, s)
                         : launch_decode_hd<64>(a, kmap, vmap, s);
}

}  // namespace attn
}  // namespace rb
