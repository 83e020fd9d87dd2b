// The attention planner as a device function, shared by the planner launch of
// rb_paged_attention and the fused step kernel.  Not part of the C ABI.
#pragma once

#include "attn_common.cuh"

namespace rb {
namespace attn {

// Block-wide exclusive scan of two int32 values per thread; returns totals via *tot.
__device__ __forceinline__ void block_scan2(int v0, int v1, int* ex0, int* ex1, int* tot0, int* tot1) {
  __shared__ int s0[32], s1[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int i0 = v0, i1 = v1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, i0, o);
    const int b = __shfl_up_sync(0xffffffffu, i1, o);
    if (lane >= o) { i0 += a; i1 += b; }
  }
  if (lane == 31) { s0[warp] = i0; s1[warp] = i1; }
  __syncthreads();
  if (warp == 0) {
    int w0 = lane < nw ? s0[lane] : 0, w1 = lane < nw ? s1[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, w0, o);
      const int b = __shfl_up_sync(0xffffffffu, w1, o);
      if (lane >= o) { w0 += a; w1 += b; }
    }
    s0[lane] = w0;
    s1[lane] = w1;
  }
  __syncthreads();
  *ex0 = i0 - v0 + (warp > 0 ? s0[warp - 1] : 0);
  *ex1 = i1 - v1 + (warp > 0 ? s1[warp - 1] : 0);
  *tot0 = s0[nw - 1];
  *tot1 = s1[nw - 1];
  __syncthreads();
}

struct ReqInfo {
  bool ok;
  int q, L, pages;
};

__device__ __forceinline__ ReqInfo req_info(const AttnArgs& a, int r) {
  ReqInfo x;
  const int s = a.qsl[r], e = a.qsl[r + 1];
  x.q = e - s;
  x.L = a.seq_lens[r];
  x.pages = (x.L + kPage - 1) / kPage;
  x.ok = s >= 0 && x.q >= 0 && e <= a.N && x.L >= x.q && x.pages <= a.kp_cap;
  return x;
}

// The planner, run by one whole CTA of any size: validates the metadata, classifies requests,
// splits the CTAs of a fused launch between decode and prefill work, sizes the KV splits,
// writes per-request unit offsets and the header, clears the split counters and writes the
// padding rows of the output as zeros.
__device__ __forceinline__ void plan_body(const AttnArgs& a, int head_dim) {
  __shared__ unsigned long long s_pages;
  __shared__ float s_flops;
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int per = (a.R + nthreads - 1) / nthreads;
  const int lo = min(tid * per, a.R), hi = min(lo + per, a.R);
  int bits = 0;
  if (tid == 0) {
    s_pages = 0;
    s_flops = 0.f;
    if (a.qsl[0] != 0 || a.qsl[a.R] != a.N) bits |= RB_EBIT_ATTN_META;
  }
  __syncthreads();
  unsigned long long my_pages = 0;
  float my_flops = 0.f;  // prefill work: 4 * nh * hd * visible keys
  for (int r = lo; r < hi; ++r) {
    const ReqInfo x = req_info(a, r);
    if (!x.ok) { bits |= RB_EBIT_ATTN_META; continue; }
    if (is_decode_class(x.q, a.group)) {
      my_pages += static_cast<unsigned long long>(x.pages);
    } else {
      const float c = static_cast<float>(x.L - x.q), q = static_cast<float>(x.q);
      my_flops += 4.f * a.nh * head_dim * (q * c + 0.5f * q * (q + 1.f));
    }
  }
  if (my_pages) atomicAdd(&s_pages, my_pages);
  if (my_flops > 0.f) atomicAdd(&s_flops, my_flops);
  __syncthreads();
  const long long page_heads = static_cast<long long>(s_pages) * a.nkv;
  // Fused launch: split the CTAs between decode (HBM-bound) and prefill (tensor-bound) so both
  // finish together; CTAs that run out of their own work then help with the other kind.
  // Rates per SM: ~80 GB/s of paged K/V for decode, ~7 TFLOP/s for prefill tiles.  Splits are
  // sized for every CTA of the launch (all of them may end up helping with decode), so the
  // decode tail stays short.
  int decode_ctas = 0;
  int target = a.target_units;
  if (a.fused_ctas > 0) {
    const float dec_bytes = static_cast<float>(page_heads) * (2.f * kPage * head_dim * 2.f);
    const float t_dec = dec_bytes / 80e3f;   // microseconds on one SM
    const float t_pre = s_flops / 7e6f;
    if (t_dec > 0.f) {
      const float share = t_pre > 0.f ? t_dec / (t_dec + t_pre) : 1.f;
      decode_ctas = max(1, min(a.fused_ctas, static_cast<int>(share * a.fused_ctas + 0.5f)));
    }
    target = min(kMaxTargetUnits, 4 * a.decode_warps_per_cta * a.fused_ctas);
  }
  const int sp = static_cast<int>(max(static_cast<long long>(kMinSplitPages),
                                      (page_heads + target - 1) / target));
  int my_d = 0, my_p = 0;
  for (int r = lo; r < hi; ++r) {
    const ReqInfo x = req_info(a, r);
    if (!x.ok || x.q == 0) continue;
    if (is_decode_class(x.q, a.group)) my_d += (x.pages + sp - 1) / sp * a.nkv;
    else my_p += (x.q * a.group + a.tile_m - 1) / a.tile_m * a.nkv;
  }
  int ex_d, ex_p, tot_d, tot_p;
  block_scan2(my_d, my_p, &ex_d, &ex_p, &tot_d, &tot_p);
  for (int r = lo; r < hi; ++r) {
    const ReqInfo x = req_info(a, r);
    a.dec_off[r] = ex_d;
    a.pre_off[r] = ex_p;
    if (!x.ok || x.q == 0) continue;
    if (is_decode_class(x.q, a.group)) ex_d += (x.pages + sp - 1) / sp * a.nkv;
    else ex_p += (x.q * a.group + a.tile_m - 1) / a.tile_m * a.nkv;
  }
  if (tid == 0) {
    a.dec_off[a.R] = tot_d;
    a.pre_off[a.R] = tot_p;
    a.header[kHNumDecodeUnits] = tot_d;
    a.header[kHNumPrefillUnits] = tot_p;
    a.header[kHDecodeNext] = 0;
    a.header[kHPrefillNext] = 0;
    a.header[kHSplitPages] = sp;
    a.header[kHDecodeCtas] = decode_ctas;
    a.header[kHRoleNext] = 0;
  }
  for (int i = tid; i < a.R * a.nkv; i += nthreads) a.done[i] = 0;
  // rows of padding tokens are written as zeros
  const long long row16 = static_cast<long long>(a.nh) * head_dim * 2 / 16;
  int4* out = reinterpret_cast<int4*>(a.out);
  const long long first = static_cast<long long>(a.N) * row16;
  const long long last = static_cast<long long>(a.N_pad) * row16;
  for (long long i = first + tid; i < last; i += nthreads) out[i] = make_int4(0, 0, 0, 0);
  if (bits) raise_error(a.err, bits);
}

}  // namespace attn
}  // namespace rb
