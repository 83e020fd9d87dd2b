// Prefill / chunk attention tiles (requests whose query_len * group > 8).
//
// Work unit = (request, kv head, tile of 64 query rows); rows are (query token, head of the
// group) pairs, token-major, so one K/V tile in shared memory serves every query head of the
// group.  A persistent grid pulls units from an atomic counter, most expensive tile of each
// request first.  Thread 0 issues the TMA loads of a 64-key K/V tile (4 pages x 128-byte boxes,
// 128B swizzle) into a 2-stage ring guarded by mbarriers; 4 warps each own 16 rows and run
// S = Q K^T and O += P V on the tensor cores with fp32 accumulation and an online softmax.
// Only tiles that reach past a row's causal limit pay for the mask.
#include "attn_common.cuh"

namespace rb {
namespace attn {
namespace {

template <int HD>
struct PreCfg {
  static constexpr int kWarps = 4;
  static constexpr int kTileM = kPrefillTileM;  // 16 rows per warp
  static constexpr int kTileN = 64;             // keys per K/V tile
  static constexpr int kPagesPerTile = kTileN / kPage;
  static constexpr int kStages = 2;
  static constexpr int kBoxes = HD / 64;
  static constexpr int kBoxBytes = kPage * 128;
  static constexpr int kTileBytes = kPagesPerTile * kBoxes * kBoxBytes;  // K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
  static constexpr int kKS = HD / 16;  // k-steps over head_dim
  static constexpr int kND = HD / 8;   // n-tiles over head_dim
  static constexpr int kNT = kTileN / 8;
};

// byte offset of (key in tile, 16-byte chunk of head_dim) inside a K or V tile
template <int HD>
__device__ __forceinline__ uint32_t tile_off(int key, int chunk) {
  using C = PreCfg<HD>;
  return static_cast<uint32_t>(((key >> 4) * C::kBoxes + (chunk >> 3)) * C::kBoxBytes) +
         swz128(key & 15, chunk & 7);
}

template <int HD>
__global__ void __launch_bounds__(PreCfg<HD>::kWarps * 32)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  using C = PreCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[C::kStages];
  __shared__ int s_unit;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base_u32 - raw_u32);
  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  const int n_units = a.header[kHNumPrefillUnits];
  uint32_t it = 0;  // K/V tiles consumed by this CTA (selects stage and phase)

  while (true) {
    if (tid == 0) s_unit = atomicAdd(a.header + kHPrefillNext, 1);
    __syncthreads();
    const int u = s_unit;
    __syncthreads();
    if (u >= n_units) break;
    const int r = upper_bound_i32(a.pre_off, a.R + 1, u) - 1;
    const int first = a.pre_off[r];
    const int tiles_r = (a.pre_off[r + 1] - first) / a.nkv;
    const int local = u - first;
    const int h = local % a.nkv;
    const int tile = tiles_r - 1 - local / a.nkv;
    const int t0 = a.qsl[r], q = a.qsl[r + 1] - t0, L = a.seq_lens[r];
    const int c = L - q, rows_total = q * a.group, pages_r = (L + kPage - 1) / kPage;
    const int row0 = tile * C::kTileM;
    const int jmax = (min(row0 + C::kTileM, rows_total) - 1) / a.group;
    const int kv_end = c + jmax + 1;  // keys [0, kv_end) are visible to some row of the tile
    const int n_kt = (kv_end + C::kTileN - 1) / C::kTileN;
    const int32_t* bt_row = a.block_table + static_cast<size_t>(r) * a.MB;

    // my two rows: ra = warp*16 + lane/4, rb = ra + 8
    const int ra = row0 + warp * 16 + (lane >> 2), rb = ra + 8;
    const bool va = ra < rows_total, vb_ = rb < rows_total;
    const int ja = va ? ra / a.group : 0, jb = vb_ ? rb / a.group : 0;
    const int ha = va ? ra - ja * a.group : 0, hb = vb_ ? rb - jb * a.group : 0;
    const int lim_a = c + ja, lim_b = c + jb;
    const int lim_min = c + (row0 / a.group);

    uint32_t aq[C::kKS][4];
    {
      const uint32_t* qa = reinterpret_cast<const uint32_t*>(
          a.q + (static_cast<size_t>(t0 + ja) * a.nh + h * a.group + ha) * HD);
      const uint32_t* qb = reinterpret_cast<const uint32_t*>(
          a.q + (static_cast<size_t>(t0 + jb) * a.nh + h * a.group + hb) * HD);
#pragma unroll
      for (int ks = 0; ks < C::kKS; ++ks) {
        const int d = ks * 16 + 2 * (lane & 3);
        aq[ks][0] = va ? __ldg(qa + (d >> 1)) : 0u;
        aq[ks][1] = vb_ ? __ldg(qb + (d >> 1)) : 0u;
        aq[ks][2] = va ? __ldg(qa + ((d + 8) >> 1)) : 0u;
        aq[ks][3] = vb_ ? __ldg(qb + ((d + 8) >> 1)) : 0u;
      }
    }
    float o[C::kND][4];
#pragma unroll
    for (int nd = 0; nd < C::kND; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    auto issue = [&](int kt, uint32_t stage) {  // thread 0 only
      uint64_t* bar = &bars[stage];
      mbar_arrive_expect_tx(bar, C::kStageBytes);
      const uint32_t kdst = base_u32 + stage * C::kStageBytes;
      const uint32_t vdst = kdst + C::kTileBytes;
#pragma unroll
      for (int pi = 0; pi < C::kPagesPerTile; ++pi) {
        const int pg = kt * C::kPagesPerTile + pi;
        int id = a.null_block;  // pages past the sequence: any valid page, zeroed below
        if (pg < pages_r) {
          id = kernel_page(bt_row, pg, a.ratio, a.num_blocks, a.null_block);
          if (id < 0 || id >= a.num_blocks || id == a.null_block) {
            raise_error(a.err, RB_EBIT_BLOCK_ID);
            id = a.null_block;
          }
        }
#pragma unroll
        for (int b = 0; b < C::kBoxes; ++b) {
          const uint32_t off = (pi * C::kBoxes + b) * C::kBoxBytes;
          tma_load_3d(kdst + off, &kmap, bar, b * 64, h, id * kPage);
          tma_load_3d(vdst + off, &vmap, bar, b * 64, h, id * kPage);
        }
      }
    };

    if (tid == 0)
      for (int i = 0; i < C::kStages && i < n_kt; ++i) issue(i, (it + i) % C::kStages);

    for (int kt = 0; kt < n_kt; ++kt) {
      const uint32_t stage = it % C::kStages, phase = (it / C::kStages) & 1u;
      const bool ok = mbar_wait_bounded(&bars[stage], phase);
      if (__syncthreads_or(!ok)) {
        if (tid == 0) raise_error(a.err, RB_EBIT_TIMEOUT);
        for (int k = 0; k < C::kStages && kt + k < n_kt; ++k) {
          const uint32_t it2 = it + k;
          mbar_wait_bounded(&bars[it2 % C::kStages], (it2 / C::kStages) & 1u);
        }
        return;
      }
      const uint32_t kb = base_u32 + stage * C::kStageBytes;
      const uint32_t vbuf = kb + C::kTileBytes;
      const int key_base = kt * C::kTileN;
      if (key_base + C::kTileN > L) {  // rows past the sequence may hold anything: zero V
        const int kmin = max(L - key_base, 0);
        uint8_t* vptr = base_ptr + stage * C::kStageBytes + C::kTileBytes;
        constexpr int kPerRow = HD / 8;
        for (int x = tid; x < (C::kTileN - kmin) * kPerRow; x += C::kWarps * 32) {
          const int key = kmin + x / kPerRow, ch = x % kPerRow;
          *reinterpret_cast<uint4*>(vptr + ((key >> 4) * C::kBoxes + (ch >> 3)) * C::kBoxBytes +
                                    (key & 15) * 128 + (ch & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncthreads();
      }

      // S = Q K^T : 16 rows x 64 keys per warp
      float sacc[C::kNT][4];
#pragma unroll
      for (int nt = 0; nt < C::kNT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
      {
        const int mi = lane >> 3;
#pragma unroll
        for (int ks = 0; ks < C::kKS; ++ks) {
#pragma unroll
          for (int np = 0; np < C::kNT / 2; ++np) {
            const int key = (np * 2 + (mi >> 1)) * 8 + (lane & 7);
            const int ch = ks * 2 + (mi & 1);
            uint32_t bf[4];
            ldsm_x4(bf, kb + tile_off<HD>(key, ch));
            mma_16816(sacc[np * 2], aq[ks], bf[0], bf[1]);
            mma_16816(sacc[np * 2 + 1], aq[ks], bf[2], bf[3]);
          }
        }
      }
      // mask (only where the tile reaches past the smallest limit of the tile), online softmax
      const bool need_mask = key_base + C::kTileN - 1 > lim_min;
      float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < C::kNT; ++nt) {
        const int k0 = key_base + nt * 8 + 2 * (lane & 3);
        float s0 = sacc[nt][0] * a.scale_log2, s1 = sacc[nt][1] * a.scale_log2;
        float s2 = sacc[nt][2] * a.scale_log2, s3 = sacc[nt][3] * a.scale_log2;
        if (need_mask) {
          s0 = k0 <= lim_a ? s0 : -INFINITY;
          s1 = k0 + 1 <= lim_a ? s1 : -INFINITY;
          s2 = k0 <= lim_b ? s2 : -INFINITY;
          s3 = k0 + 1 <= lim_b ? s3 : -INFINITY;
        }
        sacc[nt][0] = s0; sacc[nt][1] = s1; sacc[nt][2] = s2; sacc[nt][3] = s3;
        mx_a = fmaxf(mx_a, fmaxf(s0, s1));
        mx_b = fmaxf(mx_b, fmaxf(s2, s3));
      }
#pragma unroll
      for (int o2 = 1; o2 < 4; o2 <<= 1) {
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, o2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, o2));
      }
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      const float ms_a = mn_a == -INFINITY ? 0.f : mn_a, ms_b = mn_b == -INFINITY ? 0.f : mn_b;
      const float al_a = fast_exp2(m_a - ms_a), al_b = fast_exp2(m_b - ms_b);
      m_a = mn_a;
      m_b = mn_b;
      float rs_a = 0.f, rs_b = 0.f;
      uint32_t pf[C::kNT][2];
#pragma unroll
      for (int nt = 0; nt < C::kNT; ++nt) {
        const float p0 = fast_exp2(sacc[nt][0] - ms_a), p1 = fast_exp2(sacc[nt][1] - ms_a);
        const float p2 = fast_exp2(sacc[nt][2] - ms_b), p3 = fast_exp2(sacc[nt][3] - ms_b);
        rs_a += p0 + p1;
        rs_b += p2 + p3;
        pf[nt][0] = pack_bf16x2(p0, p1);
        pf[nt][1] = pack_bf16x2(p2, p3);
      }
      l_a = l_a * al_a + rs_a;
      l_b = l_b * al_b + rs_b;
#pragma unroll
      for (int nd = 0; nd < C::kND; ++nd) {
        o[nd][0] *= al_a; o[nd][1] *= al_a; o[nd][2] *= al_b; o[nd][3] *= al_b;
      }
      // O += P V
      {
        const int mi = lane >> 3;
#pragma unroll
        for (int kk = 0; kk < C::kTileN / 16; ++kk) {
          const uint32_t pa[4] = {pf[2 * kk][0], pf[2 * kk][1], pf[2 * kk + 1][0], pf[2 * kk + 1][1]};
#pragma unroll
          for (int nd2 = 0; nd2 < C::kND / 2; ++nd2) {
            const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
            const int ch = nd2 * 2 + (mi >> 1);
            uint32_t bf[4];
            ldsm_x4_t(bf, vbuf + tile_off<HD>(key, ch));
            mma_16816(o[nd2 * 2], pa, bf[0], bf[1]);
            mma_16816(o[nd2 * 2 + 1], pa, bf[2], bf[3]);
          }
        }
      }
      __syncthreads();  // every warp is done with this stage
      if (tid == 0 && kt + C::kStages < n_kt) issue(kt + C::kStages, stage);
      ++it;
    }

#pragma unroll
    for (int o2 = 1; o2 < 4; o2 <<= 1) {
      l_a += __shfl_xor_sync(0xffffffffu, l_a, o2);
      l_b += __shfl_xor_sync(0xffffffffu, l_b, o2);
    }
    const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f, inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
    uint32_t* oa = reinterpret_cast<uint32_t*>(
        a.out + (static_cast<size_t>(t0 + ja) * a.nh + h * a.group + ha) * HD);
    uint32_t* ob = reinterpret_cast<uint32_t*>(
        a.out + (static_cast<size_t>(t0 + jb) * a.nh + h * a.group + hb) * HD);
#pragma unroll
    for (int nd = 0; nd < C::kND; ++nd) {
      const int d = nd * 8 + 2 * (lane & 3);
      if (va) oa[d >> 1] = pack_bf16x2(o[nd][0] * inv_a, o[nd][1] * inv_a);
      if (vb_) ob[d >> 1] = pack_bf16x2(o[nd][2] * inv_b, o[nd][3] * inv_b);
    }
  }
}

template <int HD>
rb_status launch_prefill_hd(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t s) {
  using C = PreCfg<HD>;
  static int blocks_per_sm[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RB_ERR_CUDA;
  if (blocks_per_sm[dev] == 0) {
    if (cudaFuncSetAttribute(attn_prefill_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return RB_ERR_CUDA;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_prefill_kernel<HD>,
                                                      C::kWarps * 32, C::kSmemBytes) != cudaSuccess ||
        n < 1)
      return RB_ERR_CUDA;
    blocks_per_sm[dev] = n;
  }
  const int grid = max(1, device_sm_count()) * blocks_per_sm[dev];
  attn_prefill_kernel<HD><<<grid, C::kWarps * 32, C::kSmemBytes, s>>>(kmap, vmap, a);
  if (last_launch_status() != RB_OK) return RB_ERR_CUDA;
  note_launches(1);
  return RB_OK;
}

}  // namespace

rb_status launch_prefill(const AttnArgs& a, int head_dim, const CUtensorMap& kmap,
                         const CUtensorMap& vmap, cudaStream_t s) {
  return head_dim == 128 ? launch_prefill_hd<128>(a, kmap, vmap, s)
                         : launch_prefill_hd<64>(a, kmap, vmap, s);
}

}  // namespace attn
}  // namespace rb
