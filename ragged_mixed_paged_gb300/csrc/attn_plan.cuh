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

// Where the planner reads request metadata: query_start_loc (global, or a shared-memory copy)
// and either the sequence lengths or, with `computed`, num_computed (seq_len = num_computed + q,
// as the preparation step writes it).
struct ReqSrc {
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* computed;
};

__device__ __forceinline__ ReqInfo req_info(const AttnArgs& a, const ReqSrc& src, int r) {
  ReqInfo x;
  const int s = src.qsl[r], e = src.qsl[r + 1];
  x.q = e - s;
  x.L = src.computed != nullptr
            ? static_cast<int32_t>(static_cast<long long>(src.computed[r]) + x.q)
            : src.seq_lens[r];
  x.pages = (x.L + kPage - 1) / kPage;
  x.ok = s >= 0 && x.q >= 0 && e <= a.N && x.L >= x.q && x.pages <= a.kp_cap;
  return x;
}

// Query-token pairs of tiles a prefill request of q tokens is cut into (tile_tokens tokens per
// 128-row tile, two tiles per unit).
__device__ __forceinline__ int prefill_pairs(int q, int tile_tokens) {
  return (q + 2 * tile_tokens - 1) / (2 * tile_tokens);
}

// Key tiles (128 keys) of tcgen05 prefill unit `pair` (query tokens [2 T pair, 2 T pair + 2 T)
// of a request with c cached tokens and q new ones, T = tile_tokens): the tiles its last query
// token sees, the larger of its two tiles' counts.
__device__ __forceinline__ int pair_key_tiles(int c, int q, int tile_tokens, int pair) {
  const int last_tok = min((pair + 1) * 2 * tile_tokens, q) - 1;
  return (c + last_tok + 1 + 127) / 128;
}

// Finish-time model of the fused launch (microseconds, this GPU, cold caches; fitted to per-unit
// timestamps and whole-launch times): a decode unit of p pages takes about 6 + 0.6 p on one
// warp, a CTA streams at most ~73 GB/s of paged K/V and all of them together ~6.4 TB/s; a
// tcgen05 prefill unit of n key tiles takes about 8 + 2.3 n on one CTA.
constexpr float kDecUnitUs = 6.f, kDecPageUs = 0.6f, kDecBytesPerUsPerCta = 73e3f;
constexpr float kHbmBytesPerUs = 6.4e6f;
constexpr float kPreUnitUs = 8.f, kPreTileUs = 2.3f;
constexpr int kTileBins = 512;  // histogram bins of prefill units by key tiles (longer: last bin)

// The planner, run by one whole CTA of any size: validates the metadata, classifies requests,
// sizes the KV splits, writes per-request unit offsets, lists the tcgen05 prefill units
// longest first, splits the CTAs of a fused launch between decode and prefill work, writes the
// header, clears the split counters and writes the padding rows of the output as zeros.
// `src`: defaults to the call's query_start_loc and seq_lens in global memory; the fused step
// passes its shared-memory scan and num_computed, so the planner need not wait for (and read
// back) the request outputs the same launch writes.
__device__ __forceinline__ void plan_body(const AttnArgs& a, int head_dim, ReqSrc src) {
  __shared__ unsigned long long s_pages;
  const int tid = threadIdx.x, nthreads = blockDim.x, lane = tid & 31;
  const int per = (a.R + nthreads - 1) / nthreads;  // the same for every thread
  const int lo = min(tid * per, a.R), hi = min(lo + per, a.R);
  // Each request's metadata is read once: a thread keeps its first kCache requests in a local
  // array for the later passes (a pass over global metadata costs an L2 round trip).  The loops
  // stay rolled: the planner runs once per step, from a cold instruction cache, and its time
  // follows its code size more than its arithmetic.
  constexpr int kCache = 4;
  ReqInfo cache[kCache];
#pragma unroll 1
  for (int k = 0; k < kCache; ++k)
    cache[k] = lo + k < hi ? req_info(a, src, lo + k) : ReqInfo{false, 0, 0, 0};
  auto get = [&](int k) { return k < kCache ? cache[k] : req_info(a, src, lo + k); };
  auto each = [&](auto&& fn) {  // fn(r, info) over this thread's requests, in order
#pragma unroll 1
    for (int k = 0; lo + k < hi; ++k) fn(lo + k, get(k));
  };
  int bits = 0;
  if (tid == 0) {
    s_pages = 0;
    if (src.qsl[0] != 0 || src.qsl[a.R] != a.N) bits |= RB_EBIT_ATTN_META;
  }
  __syncthreads();
  unsigned long long my_pages = 0;
  each([&](int, const ReqInfo& x) {
    if (!x.ok) bits |= RB_EBIT_ATTN_META;
    else if (is_decode_class(x.q, a.group)) my_pages += static_cast<unsigned long long>(x.pages);
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) my_pages += __shfl_xor_sync(0xffffffffu, my_pages, o);
  if (lane == 0 && my_pages) atomicAdd(&s_pages, my_pages);
  __syncthreads();
  const long long page_heads = static_cast<long long>(s_pages) * a.nkv;
  // Fused launch: splits are sized for every CTA of the launch (all of them may end up helping
  // with decode), so the decode tail stays short.
  const int target = a.fused_ctas > 0
                         ? min(kMaxTargetUnits, 4 * a.decode_warps_per_cta * a.fused_ctas)
                         : a.target_units;
  const int sp = static_cast<int>(max(static_cast<long long>(kMinSplitPages),
                                      (page_heads + target - 1) / target));
  auto units_of = [&](const ReqInfo& x, int* d, int* p) {
    if (!x.ok || x.q == 0) return;
    if (is_decode_class(x.q, a.group)) *d += (x.pages + sp - 1) / sp * a.nkv;
    else *p += prefill_pairs(x.q, a.tile_tokens) * a.nkv;
  };
  int my_d = 0, my_p = 0;
  each([&](int, const ReqInfo& x) { units_of(x, &my_d, &my_p); });
  int ex_d, ex_p, tot_d, tot_p;
  block_scan2(my_d, my_p, &ex_d, &ex_p, &tot_d, &tot_p);
  each([&](int r, const ReqInfo& x) {
    a.dec_off[r] = ex_d;
    a.pre_off[r] = ex_p;
    units_of(x, &ex_d, &ex_p);
  });

  // tcgen05 prefill units in one global longest-first order: a counting sort of the (request,
  // pair) entries by key tiles, so the long units start first whatever request they belong to.
  // The pairs of each prefill request are spread over the lanes of its thread's warp.
  __shared__ int s_bin[kTileBins];
  __shared__ float s_pre_us;
  __shared__ int s_pre_max;
  const bool fused = a.fused_ctas > 0;
  auto warp_pairs = [&](auto&& body) {  // body(r, c, q, pair) for every pair, warp-cooperative
    auto one = [&](int r, const ReqInfo& x, bool has) {
      const bool pre = has && x.ok && x.q > 0 && !is_decode_class(x.q, a.group);
      const int pairs = pre ? prefill_pairs(x.q, a.tile_tokens) : 0;
      unsigned m = __ballot_sync(0xffffffffu, pairs > 0);
      while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const int rr = __shfl_sync(0xffffffffu, r, src);
        const int q = __shfl_sync(0xffffffffu, x.q, src);
        const int c = __shfl_sync(0xffffffffu, x.L - x.q, src);
        const int np = __shfl_sync(0xffffffffu, pairs, src);
        for (int p = lane; p < np; p += 32) body(rr, c, q, p);
      }
    };
#pragma unroll 1
    for (int k = 0; k < per; ++k) {  // uniform: every thread has the same `per`
      const int r = lo + k;
      one(r, r < hi ? get(k) : ReqInfo{false, 0, 0, 0}, r < hi);
    }
  };
  if (fused) {
    for (int i = tid; i < kTileBins; i += nthreads) s_bin[i] = 0;
    if (tid == 0) {
      s_pre_us = 0.f;
      s_pre_max = 0;
    }
    __syncthreads();
    float my_us = 0.f;
    int my_max = 0;
    warp_pairs([&](int, int c, int q, int p) {
      const int n = pair_key_tiles(c, q, a.tile_tokens, p);
      atomicAdd(&s_bin[min(n, kTileBins - 1)], 1);
      my_us += kPreUnitUs + kPreTileUs * n;
      my_max = max(my_max, n);
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      my_us += __shfl_xor_sync(0xffffffffu, my_us, o);
      my_max = max(my_max, __shfl_xor_sync(0xffffffffu, my_max, o));
    }
    if (lane == 0 && my_us > 0.f) atomicAdd(&s_pre_us, my_us);
    if (lane == 0 && my_max > 0) atomicMax(&s_pre_max, my_max);
    __syncthreads();
    // bins in descending tile order: start position of each bin in the list
    const int per_bin = (kTileBins + nthreads - 1) / nthreads;
    int cnt = 0;
    for (int i = 0; i < per_bin; ++i) {
      const int b = kTileBins - 1 - (tid * per_bin + i);
      if (b >= 0) cnt += s_bin[b];
    }
    int start, total, dummy0, dummy1;
    block_scan2(cnt, 0, &start, &dummy0, &total, &dummy1);
    for (int i = 0; i < per_bin; ++i) {
      const int b = kTileBins - 1 - (tid * per_bin + i);
      if (b < 0) continue;
      const int c = s_bin[b];
      s_bin[b] = start;
      start += c;
    }
    __syncthreads();
    warp_pairs([&](int r, int c, int q, int p) {
      const int n = pair_key_tiles(c, q, a.tile_tokens, p);
      a.pre_list[atomicAdd(&s_bin[min(n, kTileBins - 1)], 1)] = r * 65536 + p;
    });
  }

  // Decode-first CTAs: the count that minimises the later of the two finish times under the
  // model above (CTAs that run out of their own kind then help with the other kind); every
  // thread scores a few counts, the best (time, count) wins.
  __shared__ unsigned long long s_best;
  if (tid == 0) s_best = ~0ull;
  __syncthreads();
  if (fused) {
    const int C = a.fused_ctas;
    const float dec_bytes = static_cast<float>(page_heads) * (2.f * kPage * head_dim * 2.f);
    const float t_unit = kDecUnitUs + kDecPageUs * sp;
    const float pre_total = s_pre_us * a.nkv, pre_long = kPreUnitUs + kPreTileUs * s_pre_max;
    auto t_dec = [&](int d) {
      if (tot_d == 0) return 0.f;
      const int waves = (tot_d + a.decode_warps_per_cta * d - 1) / (a.decode_warps_per_cta * d);
      return fmaxf(waves * t_unit, dec_bytes / fminf(d * kDecBytesPerUsPerCta, kHbmBytesPerUs));
    };
    auto t_pre = [&](int p) { return tot_p == 0 ? 0.f : fmaxf(pre_long, pre_total / p); };
    auto key = [](float t, int d) {
      return (static_cast<unsigned long long>(__float_as_uint(t)) << 32) |
             static_cast<unsigned>(d);
    };
    // d = C: everything decodes first, then prefills (also the only choice without prefill).
    // A split must beat it by 10 %: split CTAs also contend for HBM and L2, which the model
    // leaves out, and the decode-first pass measured faster whenever the two were close.
    unsigned long long best =
        tid == 0 ? key(0.9f * (t_dec(C) + t_pre(C)), tot_d > 0 ? C : 0) : ~0ull;
    // d = 0: everything prefills first, so the longest units start at once, and the decode
    // units fill the CTAs as they run out of prefill units (the last, partial wave of prefill
    // units leaves CTAs idle otherwise).  Only for decode work that is bandwidth-heavy next to
    // one decode unit's latency: a few short decode units run after the prefill as a tail of
    // their own.  Measured against decode-first: long context (decode HBM time 9.5 unit
    // latencies) 6.27 -> 6.05 ms; the same batch at 1/8 of its lengths (5.8) 0.99 -> 1.13 ms
    // and the padding example (0.9) 65 -> 77 us, both slower; hence the threshold of 8.
    const float dec_stream = dec_bytes / kHbmBytesPerUs;
    if (tid == 1 && tot_d > 0 && tot_p > 0 && dec_stream > 8.f * t_unit)
      best = key(0.9f * fmaxf(pre_long, pre_total / C + dec_stream), 0);
    if (tot_d > 0 && tot_p > 0)
      for (int d = 1 + tid; d < C; d += nthreads)
        best = min(best, key(fmaxf(t_dec(d), t_pre(C - d)), d));
    atomicMin(&s_best, best);
  }
  __syncthreads();

  if (tid == 0) {
    const int decode_ctas = fused ? static_cast<int>(s_best & 0xffffffffu) : 0;
    a.dec_off[a.R] = tot_d;
    a.pre_off[a.R] = tot_p;
    a.header[kHNumDecodeUnits] = tot_d;
    a.header[kHNumPrefillUnits] = tot_p;
    // decode-first CTAs of a fused launch take their warps' first units statically
    a.header[kHDecodeNext] = decode_ctas * a.decode_warps_per_cta;
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
