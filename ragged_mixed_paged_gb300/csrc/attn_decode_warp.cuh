// Split-KV decode warp of the fused attention kernel (its decode units).  Not part of the C ABI.
//
// Work unit = (request, kv head, split of pages); one warp per unit, units pulled from an atomic
// counter (or handed out statically to decode-first CTAs).  Each warp owns a ring of
// shared-memory stages; lane 0 issues TMA loads (3-D tensor map, one {64 dims x 16 slots} box
// per 128-byte half of a page, 128B swizzle) and the warp waits on the stage's mbarrier with a
// bounded wait.
//
// The contraction runs transposed so a 16-token page is one MMA tile:
//   S^T[16 keys, 8 cols] = K[16, hd] . Q^T[hd, 8]     cols = (query token, head of the group)
//   O^T[hd, 8 cols]     += V^T[hd, 16] . P^T[16, 8]
// with mma.sync m16n8k16 (bf16 in, fp32 accumulate): its contraction per page is 16 keys by at
// most 8 columns, far below a tcgen05 tile, and the unit is bound by HBM, not by the tensor
// pipe.  P^T's fragments come from S^T's with a register transpose (movmatrix), so each page
// costs 2 x hd/16 MMAs and every K/V byte is read once per kv head, shared by the whole
// query-head group.  Softmax statistics are per column: exponents are taken against a
// reference maximum that is re-reduced with warp shuffles (and O rescaled) only on the pages
// where a score climbs well above it; a unit with several splits leaves (m, l, o) partials
// and the last split of its (request, kv head) to finish merges them; a single-split unit
// writes the normalised bf16 output directly.
#pragma once

#include "attn_common.cuh"

namespace rb {
namespace attn {

template <int HD>
struct DecCfg {
  static constexpr int kStages = 3;  // per warp
  static constexpr int kBoxes = HD / 64;                 // 128-byte halves of a token row
  static constexpr int kBoxBytes = kPage * 128;          // one TMA box: 16 rows x 128 bytes
  static constexpr int kPageBytes = kBoxes * kBoxBytes;  // one page of one kv head (K or V)
  static constexpr int kStageBytes = 2 * kPageBytes;
  static constexpr int kKS = HD / 16;
};

// Log-sum-exp merge of the split partials of one (request, kv head) by one warp: 4 lanes per
// column (8 columns), each lane owning a quarter of head_dim; the split maxima are also spread
// over the 4 lanes.  Partials written by other SMs are read through L2 (ld.global.cg).
template <int HD>
__device__ void combine_splits(const AttnArgs& a, int h, int first, int nsplit, int t0,
                               int cols) {
  constexpr int kLanesPerCol = 4;
  constexpr int kPer = HD / kLanesPerCol;  // values of one column per lane
  const int lane = threadIdx.x & 31;
  const int col = lane / kLanesPerCol, part = lane % kLanesPerCol;
  const bool active = col < cols;
  const int c = active ? col : 0;
  float mx = -INFINITY;
  for (int sp = part; sp < nsplit; sp += kLanesPerCol)
    mx = fmaxf(mx, __ldcg(&a.part_ml[static_cast<size_t>(first + sp * a.nkv + h) * kMaxCols + c].x));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  if (mx == -INFINITY) mx = 0.f;
  float acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  float lsum = 0.f;
#pragma unroll 2
  for (int sp = 0; sp < nsplit; ++sp) {
    const size_t u = static_cast<size_t>(first + sp * a.nkv + h);
    const float2 ml = __ldcg(a.part_ml + u * kMaxCols + c);
    const float w = fast_exp2(ml.x - mx);
    lsum += w * ml.y;
    const float4* o = reinterpret_cast<const float4*>(a.part_o + (u * kMaxCols + c) * HD +
                                                      part * kPer);
#pragma unroll
    for (int v = 0; v < kPer / 4; ++v) {
      const float4 x = __ldcg(o + v);
      acc[4 * v + 0] += w * x.x;
      acc[4 * v + 1] += w * x.y;
      acc[4 * v + 2] += w * x.z;
      acc[4 * v + 3] += w * x.w;
    }
  }
  if (!active) return;
  const int j = col / a.group, hh = col - j * a.group;
  const size_t row = static_cast<size_t>(t0 + j) * a.nh + h * a.group + hh;
  float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  if (a.cascade == kSuffixPass) {  // fold in the shared-prefix rows (acc and lsum are at mx)
    float wp[kMaxPrefixSplits];
    const float wa = cascade_weights(a, row, mx, lsum, wp);
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc[k] *= wa;
#pragma unroll
    for (int ps = 0; ps < kMaxPrefixSplits; ++ps) {
      if (ps >= a.prefix_splits) break;
      const float4* o1 = reinterpret_cast<const float4*>(cascade_row<HD>(a, ps, row) + part * kPer);
#pragma unroll
      for (int v = 0; v < kPer / 4; ++v) {
        const float4 x = __ldg(o1 + v);
        acc[4 * v + 0] += x.x * wp[ps];
        acc[4 * v + 1] += x.y * wp[ps];
        acc[4 * v + 2] += x.z * wp[ps];
        acc[4 * v + 3] += x.w * wp[ps];
      }
    }
    inv = 1.f;
  }
  uint4* dst = reinterpret_cast<uint4*>(a.out + row * HD + part * kPer);
#pragma unroll
  for (int v = 0; v < kPer / 8; ++v) {
    uint4 wv;
    wv.x = pack_bf16x2(acc[8 * v + 0] * inv, acc[8 * v + 1] * inv);
    wv.y = pack_bf16x2(acc[8 * v + 2] * inv, acc[8 * v + 3] * inv);
    wv.z = pack_bf16x2(acc[8 * v + 4] * inv, acc[8 * v + 5] * inv);
    wv.w = pack_bf16x2(acc[8 * v + 6] * inv, acc[8 * v + 7] * inv);
    dst[v] = wv;
  }
}

// One decode warp: pulls (request, kv head, split) units from the shared counter until none
// are left.  `bars` are this warp's kStages mbarriers (initialised, count 1) and `wbase` /
// `wbase_ptr` the shared-memory address / pointer of its kStages stages (1024-byte aligned).
// `first_unit` >= 0: the warp's first unit, handed out statically (the counter then starts
// past every statically handed unit), which saves the first atomic's round trip.
template <int HD>
__device__ void decode_warp(const CUtensorMap* kmap_p, const CUtensorMap* vmap_p,
                            const AttnArgs& a, uint64_t* bars, uint32_t wbase,
                            uint8_t* wbase_ptr, int first_unit) {
  using C = DecCfg<HD>;
  const int lane = threadIdx.x & 31;
  const int n_units = a.header[kHNumDecodeUnits];
  const int sp = a.header[kHSplitPages];
  uint32_t it = 0;  // pages this warp has consumed (selects stage and phase)

  int next_static = first_unit;
  while (true) {
    int u = next_static;
    if (u < 0) {
      if (lane == 0) u = atomicAdd(a.header + kHDecodeNext, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
    }
    next_static = -1;
    if (u >= n_units) break;
    const int r = warp_upper_bound_i32(a.dec_off, a.R + 1, u) - 1;
    const int first = a.dec_off[r];
    const int nsplit = (a.dec_off[r + 1] - first) / a.nkv;
    const int local = u - first;
    const int split = local / a.nkv, h = local - split * a.nkv;
    const int t0 = a.qsl[r], q = a.qsl[r + 1] - t0, L = a.seq_lens[r];
    const int c = L - q, cols = q * a.group, pages = (L + kPage - 1) / kPage;
    const int p_begin = split * sp, p_end = min(p_begin + sp, pages);
    const int n_pages = p_end - p_begin;

    // Q^T fragments (B operand: k = head dim, n = column)
    uint32_t bq[C::kKS][2];
    {
      const int col = lane >> 2;
      const bool valid = col < cols;
      const int j = valid ? col / a.group : 0;
      const int hh = valid ? col - j * a.group : 0;
      const uint32_t* qp = reinterpret_cast<const uint32_t*>(
          a.q + (static_cast<size_t>(t0 + j) * a.nh + h * a.group + hh) * HD);
#pragma unroll
      for (int ks = 0; ks < C::kKS; ++ks) {
        const int d = ks * 16 + 2 * (lane & 3);
        bq[ks][0] = valid ? __ldg(qp + (d >> 1)) : 0u;
        bq[ks][1] = valid ? __ldg(qp + ((d + 8) >> 1)) : 0u;
      }
    }
    const int c0 = 2 * (lane & 3), c1 = c0 + 1;
    const int lim0 = c0 < cols ? c + c0 / a.group : c;
    const int lim1 = c1 < cols ? c + c1 / a.group : c;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[C::kKS][4];
#pragma unroll
    for (int mt = 0; mt < C::kKS; ++mt)
      acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

    // page ids of pages [win, win + 32) held one per lane, the next window prefetched
    const int32_t* bt_row = a.block_table + static_cast<size_t>(r) * a.MB;
    int win = p_begin;
    auto page = [&](int pg) {
      return pg < p_end ? kernel_page(bt_row, pg, a.ratio, a.num_blocks, a.null_block)
                        : a.null_block;
    };
    int bid = page(win + lane);
    int bid_next = page(win + 32 + lane);

    auto issue = [&](int pg, uint32_t stage) {  // called by the whole warp
      if (pg - win >= 32) {
        win += 32;
        bid = bid_next;
        bid_next = page(win + 32 + lane);
      }
      int id = __shfl_sync(0xffffffffu, bid, pg - win);
      if (lane == 0) {
        if (id < 0 || id >= a.num_blocks || id == a.null_block) {
          raise_error(a.err, RB_EBIT_BLOCK_ID);
          id = a.null_block;
        }
        uint64_t* bar = &bars[stage];
        mbar_arrive_expect_tx(bar, C::kStageBytes);
        const uint32_t kdst = wbase + stage * C::kStageBytes;
        const uint32_t vdst = kdst + C::kPageBytes;
#pragma unroll
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(kdst + b * C::kBoxBytes, kmap_p, bar, b * 64, h, id * kPage);
#pragma unroll
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(vdst + b * C::kBoxBytes, vmap_p, bar, b * 64, h, id * kPage);
      }
    };

    for (int i = 0; i < C::kStages && i < n_pages; ++i)
      issue(p_begin + i, (it + i) % C::kStages);

    bool dead = false;
    for (int i = 0; i < n_pages; ++i) {
      const int pg = p_begin + i;
      const uint32_t stage = it % C::kStages, phase = (it / C::kStages) & 1u;
      const bool ok = mbar_wait_bounded(&bars[stage], phase);
      if (__any_sync(0xffffffffu, !ok)) {
        // give up: flag it, let the copies already issued land, leave the kernel
        if (lane == 0) raise_error(a.err, RB_EBIT_TIMEOUT);
        for (int k = 0; k < C::kStages && i + k < n_pages; ++k) {
          const uint32_t it2 = it + k;
          mbar_wait_bounded(&bars[it2 % C::kStages], (it2 / C::kStages) & 1u);
        }
        dead = true;
        break;
      }
      const uint32_t kb = wbase + stage * C::kStageBytes;
      const uint32_t vb = kb + C::kPageBytes;

      // S^T = K . Q^T  (16 keys x 8 cols), even and odd 16-dim steps in two accumulators so
      // the MMAs form two dependency chains instead of one (+3 % per CTA on this GPU)
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      {
        float s2[4] = {0.f, 0.f, 0.f, 0.f};
        const int mi = lane >> 3, rr = lane & 7;
        const int key = ((mi & 1) << 3) + rr;
#pragma unroll
        for (int ks = 0; ks < C::kKS; ++ks) {
          const int chunk = ks * 2 + (mi >> 1);
          uint32_t af[4];
          ldsm_x4(af, kb + (chunk >> 3) * C::kBoxBytes + swz128(key, chunk & 7));
          if (ks & 1) mma_16816(s2, af, bq[ks][0], bq[ks][1]);
          else mma_16816(s, af, bq[ks][0], bq[ks][1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i] += s2[i];
      }
      // causal mask per column, then the softmax per column (log2 domain)
      const int key0 = pg * kPage + (lane >> 2), key1 = key0 + 8;
      const float x0 = key0 <= lim0 ? s[0] * a.scale_log2 : -INFINITY;
      const float x1 = key0 <= lim1 ? s[1] * a.scale_log2 : -INFINITY;
      const float x2 = key1 <= lim0 ? s[2] * a.scale_log2 : -INFINITY;
      const float x3 = key1 <= lim1 ? s[3] * a.scale_log2 : -INFINITY;
      // The exponents are taken against a reference m per column that moves only when a score
      // exceeds it by more than kGrowth (log2 units): then the column maxima are reduced and
      // O and l rescaled, as an online softmax does on every page.  Otherwise the page costs
      // no shuffles and no rescale; every term stays below 2^kGrowth and the result, O / l, is
      // the same (the partials' (m, l) are relative to the same m, which the merge accounts for).
      constexpr float kGrowth = 8.f;
      const float g0 = fmaxf(x0, x2), g1 = fmaxf(x1, x3);
      if (__any_sync(0xffffffffu, g0 > m0 + kGrowth || g1 > m1 + kGrowth)) {
        float mx0 = g0, mx1 = g1;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = fast_exp2(m0 - (mn0 == -INFINITY ? 0.f : mn0));
        const float al1 = fast_exp2(m1 - (mn1 == -INFINITY ? 0.f : mn1));
        l0 *= al0;
        l1 *= al1;
#pragma unroll
        for (int mt = 0; mt < C::kKS; ++mt) {
          acc[mt][0] *= al0; acc[mt][1] *= al1; acc[mt][2] *= al0; acc[mt][3] *= al1;
        }
        m0 = mn0;
        m1 = mn1;
      }
      const float ms0 = m0 == -INFINITY ? 0.f : m0, ms1 = m1 == -INFINITY ? 0.f : m1;
      const float p0 = fast_exp2(x0 - ms0), p1 = fast_exp2(x1 - ms1);
      const float p2 = fast_exp2(x2 - ms0), p3 = fast_exp2(x3 - ms1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      // rows past the end of the sequence may hold anything: zero their V before P.V
      if (pg * kPage + kPage > L) {
        const int kmin = L - pg * kPage;
        uint8_t* vptr = wbase_ptr + stage * C::kStageBytes + C::kPageBytes;
        const int per_row = C::kBoxes * 8;
        for (int x = lane; x < (kPage - kmin) * per_row; x += 32) {
          const int row = kmin + x / per_row, rest = x % per_row;
          *reinterpret_cast<uint4*>(vptr + (rest >> 3) * C::kBoxBytes + row * 128 +
                                    (rest & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      // P^T fragments from S^T's by a register transpose
      const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
      const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));
      {
        const int mi = lane >> 3, rr = lane & 7;
        const int key = ((mi >> 1) << 3) + rr;
#pragma unroll
        for (int mt = 0; mt < C::kKS; ++mt) {
          const int chunk = mt * 2 + (mi & 1);
          uint32_t af[4];
          ldsm_x4_t(af, vb + (chunk >> 3) * C::kBoxBytes + swz128(key, chunk & 7));
          mma_16816(acc[mt], af, pb0, pb1);
        }
      }
      __syncwarp();
      if (i + C::kStages < n_pages) issue(pg + C::kStages, stage);
      ++it;
    }
    if (dead) return;

#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    const int dlo = lane >> 2;
    if (nsplit == 1 && a.cascade != kSuffixPass) {
      // (in a cascade suffix pass even an unsplit unit goes through the merge below, which
      // also folds in the shared-prefix rows)
      const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
      __nv_bfloat16* o0 = nullptr;
      __nv_bfloat16* o1 = nullptr;
      if (c0 < cols) {
        const int j = c0 / a.group, hh = c0 - j * a.group;
        o0 = a.out + (static_cast<size_t>(t0 + j) * a.nh + h * a.group + hh) * HD;
      }
      if (c1 < cols) {
        const int j = c1 / a.group, hh = c1 - j * a.group;
        o1 = a.out + (static_cast<size_t>(t0 + j) * a.nh + h * a.group + hh) * HD;
      }
#pragma unroll
      for (int mt = 0; mt < C::kKS; ++mt) {
        const int d0 = mt * 16 + dlo, d1 = d0 + 8;
        if (o0) { o0[d0] = __float2bfloat16_rn(acc[mt][0] * inv0); o0[d1] = __float2bfloat16_rn(acc[mt][2] * inv0); }
        if (o1) { o1[d0] = __float2bfloat16_rn(acc[mt][1] * inv1); o1[d1] = __float2bfloat16_rn(acc[mt][3] * inv1); }
      }
    } else {
      float* po = a.part_o + static_cast<size_t>(u) * kMaxCols * HD;
#pragma unroll
      for (int mt = 0; mt < C::kKS; ++mt) {
        const int d0 = mt * 16 + dlo, d1 = d0 + 8;
        po[c0 * HD + d0] = acc[mt][0];
        po[c0 * HD + d1] = acc[mt][2];
        po[c1 * HD + d0] = acc[mt][1];
        po[c1 * HD + d1] = acc[mt][3];
      }
      if (lane < 4) {
        a.part_ml[static_cast<size_t>(u) * kMaxCols + c0] = make_float2(m0, l0);
        a.part_ml[static_cast<size_t>(u) * kMaxCols + c1] = make_float2(m1, l1);
      }
      // the last split of this (request, kv head) to finish merges all partials
      __threadfence();
      __syncwarp();
      int prev = 0;
      if (lane == 0) prev = atomicAdd(a.done + r * a.nkv + h, 1);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev == nsplit - 1) {
        __threadfence();
        combine_splits<HD>(a, h, first, nsplit, t0, cols);
      }
    }
  }
}

}  // namespace attn
}  // namespace rb
