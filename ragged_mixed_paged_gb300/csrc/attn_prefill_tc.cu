// Prefill / chunk attention tiles on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Work unit = (request, kv head, tile of 128 query rows); rows are (query token, head of the
// group) pairs, token-major, so every K/V tile serves the whole query-head group.  One CTA per
// SM (persistent; units pulled from an atomic counter, the most expensive tile of each request
// first), 6 warps with fixed roles:
//   warp 4     TMA producer: fetches units into a 4-entry ring, loads the Q tile once per unit
//              (3-D box {64 dims, group heads, 128/group tokens}) and each 128-key K and V
//              tile (8 pages x 128-byte boxes, 128B swizzle, one page per lane) into separate
//              3-stage rings, V one tile behind K (K is released as soon as S is done);
//   warp 5     allocates 512 TMEM columns; one thread issues the MMAs:
//              S_j = Q K_j^T  (M=128, N=128, K=hd; A, B K-major from shared memory) into one of
//              two S buffers, then O += P_{j-1} V_{j-1}  (M=128, N=hd, K=128; A = P read from
//              TMEM, B = V MN-major from shared memory), so S_{j+1} runs while P_j is made;
//   warps 0-3  softmax, thread t = query row t: reads its S row from TMEM, masks causally,
//              keeps a running max and sum in the log2 domain, writes P (bf16) back over the
//              S columns, and rescales the O row in TMEM only when the max grows by more than
//              2^8 (exact either way: P and the sum share the same reference).  The epilogue
//              reads O, divides by the sum and stores bf16 rows.
// All mbarrier waits are bounded; a timeout sets RB_EBIT_TIMEOUT, every role stops, in-flight
// copies and MMAs are drained with bounded waits and TMEM is freed before the CTA exits.
#include "attn_common.cuh"
#include "tc_ptx.cuh"

namespace rb {
namespace attn {
namespace {

template <int HD>
struct TcCfg {
  static constexpr int kM = 128;                          // query rows per tile
  static constexpr int kN = 128;                          // keys per K/V tile
  static constexpr int kPagesPerTile = kN / kPage;        // 8
  static constexpr int kHalves = HD / 64;                 // 128-byte swizzle atoms per row
  static constexpr int kHalfBytes = kN * 128;             // one 64-dim half of a K or V tile
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  static constexpr int kQHalfBytes = kM * 128;
  static constexpr int kQBytes = kHalves * kQHalfBytes;
  static constexpr int kStagesK = 3;                      // K freed when S is done
  static constexpr int kStagesV = 3;                      // V freed when P V is done
  static constexpr int kVOffset = kStagesK * kTileBytes;
  static constexpr int kQOffset = kVOffset + kStagesV * kTileBytes;
  static constexpr int kUsed = kQOffset + kQBytes;
  // at least 120 KB keeps one CTA per SM (each CTA holds all 512 TMEM columns)
  static constexpr int kSmemBytes = (kUsed + 1024) > 120 * 1024 ? (kUsed + 1024) : 120 * 1024;
  static constexpr int kThreads = 192;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;                  // S0 at 0, S1 at 128, O at 256
  static constexpr int kRing = 4;
};

struct TcUnit {
  int r, h, row0, t0, q, L, c, rows_total, n_kt, pages, valid;
};

struct TcShared {
  uint64_t unit_full[4], unit_empty[4];
  uint64_t q_full, q_empty;
  uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done, o_free, drain;
  TcUnit units[4];
  uint32_t tmem_base;
  int abort;
};

constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t phase, volatile int* abort,
                                        int32_t* err) {
#pragma unroll 1
  for (int i = 0; i < 128; ++i)
    if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  while (true) {
    if (mbar_try_wait(bar, phase)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      if (atomicExch(const_cast<int*>(abort), 1) == 0) raise_error(err, RB_EBIT_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ TcUnit decode_unit(const AttnArgs& a, int u) {
  TcUnit un{};
  const int r = upper_bound_i32(a.pre_off, a.R + 1, u) - 1;
  const int first = a.pre_off[r];
  const int tiles_r = (a.pre_off[r + 1] - first) / a.nkv;
  const int local = u - first;
  un.r = r;
  un.h = local % a.nkv;
  const int tile = tiles_r - 1 - local / a.nkv;
  un.t0 = a.qsl[r];
  un.q = a.qsl[r + 1] - un.t0;
  un.L = a.seq_lens[r];
  un.c = un.L - un.q;
  un.rows_total = un.q * a.group;
  un.row0 = tile * 128;
  const int jmax = (min(un.row0 + 128, un.rows_total) - 1) / a.group;
  un.n_kt = (un.c + jmax + 1 + 127) / 128;
  un.pages = (un.L + kPage - 1) / kPage;
  un.valid = 1;
  return un;
}

template <int HD>
__device__ void producer(const AttnArgs& a, TcShared& sh, uint32_t smem_base,
                         const CUtensorMap* qmap, const CUtensorMap* kmap,
                         const CUtensorMap* vmap) {
  // The whole warp: page ids are held one per lane (a 32-page window, the next one prefetched)
  // and lanes 0..7 each issue the boxes of one page of a tile.  V runs one tile behind K.
  using C = TcCfg<HD>;
  volatile int* abort = &sh.abort;
  const int lane = threadIdx.x & 31;
  const int n_units = a.header[kHNumPrefillUnits];
  uint32_t it = 0, q_armed = 0, k_armed[3] = {0, 0, 0}, v_armed[3] = {0, 0, 0};
  auto lane0_wait = [&](uint64_t* bar, uint32_t phase) -> bool {
    int ok = 1;
    if (lane == 0) ok = tc_wait(bar, phase, abort, a.err) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  for (int k = 0;; ++k) {
    const int slot = k % C::kRing;
    if (!lane0_wait(&sh.unit_empty[slot], ((k / C::kRing) & 1) ^ 1)) break;
    if (lane == 0) {
      const int u = atomicAdd(a.header + kHPrefillNext, 1);
      TcUnit un{};
      if (u < n_units) un = decode_unit(a, u);
      sh.units[slot] = un;
      tc::mbar_arrive(&sh.unit_full[slot]);
    }
    __syncwarp();
    const TcUnit un = sh.units[slot];
    if (!un.valid) break;
    if (!lane0_wait(&sh.q_empty, (k & 1) ^ 1)) break;
    if (lane == 0) {
      mbar_arrive_expect_tx(&sh.q_full, C::kQBytes);
      ++q_armed;
#pragma unroll
      for (int hf = 0; hf < C::kHalves; ++hf)
        tma_load_3d(smem_base + C::kQOffset + hf * C::kQHalfBytes, qmap, &sh.q_full, hf * 64,
                    un.h * a.group, un.t0 + un.row0 / a.group);
    }
    const int32_t* bt_row = a.block_table + static_cast<size_t>(un.r) * a.MB;
    int win = 0;
    int bid = lane < un.pages ? __ldg(bt_row + lane) : a.null_block;
    int bid_next = 32 + lane < un.pages ? __ldg(bt_row + 32 + lane) : a.null_block;
    int ids[2] = {a.null_block, a.null_block};  // page id of this lane for tiles j and j-1
    bool ok = true;
    for (int j = 0; j <= un.n_kt; ++j) {
      if (j < un.n_kt) {  // K of tile j
        const int first = j * C::kPagesPerTile;
        if (first - win >= 32) {
          win += 32;
          bid = bid_next;
          bid_next = win + 32 + lane < un.pages ? __ldg(bt_row + win + 32 + lane) : a.null_block;
        }
        int id = __shfl_sync(0xffffffffu, bid, first + (lane & 7) - win);
        const int pg = first + (lane & 7);
        if (pg >= un.pages) {
          id = a.null_block;  // past the sequence: any valid page (masked, V zeroed)
        } else if (id < 0 || id >= a.num_blocks || id == a.null_block) {
          if (lane < C::kPagesPerTile) raise_error(a.err, RB_EBIT_BLOCK_ID);
          id = a.null_block;
        }
        ids[j & 1] = id;
        const uint32_t itk = it + j, st = itk % C::kStagesK;
        if (!lane0_wait(&sh.k_empty[st], ((itk / C::kStagesK) & 1) ^ 1)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&sh.k_full[st], C::kTileBytes);
          ++k_armed[st];
        }
        __syncwarp();
        if (lane < C::kPagesPerTile) {
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(smem_base + st * C::kTileBytes + hf * C::kHalfBytes + lane * (kPage * 128),
                        kmap, &sh.k_full[st], hf * 64, un.h, id * kPage);
        }
      }
      if (j >= 1) {  // V of tile j-1
        const uint32_t itv = it + j - 1, st = itv % C::kStagesV;
        if (!lane0_wait(&sh.v_empty[st], ((itv / C::kStagesV) & 1) ^ 1)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&sh.v_full[st], C::kTileBytes);
          ++v_armed[st];
        }
        __syncwarp();
        if (lane < C::kPagesPerTile) {
          const int id = ids[(j - 1) & 1];
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(smem_base + C::kVOffset + st * C::kTileBytes + hf * C::kHalfBytes +
                            lane * (kPage * 128),
                        vmap, &sh.v_full[st], hf * 64, un.h, id * kPage);
        }
      }
    }
    if (!ok) break;
    it += un.n_kt;
  }
  if (lane == 0 && *abort) {  // let every copy already issued land before the CTA can exit
    if (q_armed) mbar_wait_bounded(&sh.q_full, (q_armed - 1) & 1, 100000000ull);
    for (int b = 0; b < 3; ++b) {
      if (k_armed[b]) mbar_wait_bounded(&sh.k_full[b], (k_armed[b] - 1) & 1, 100000000ull);
      if (v_armed[b]) mbar_wait_bounded(&sh.v_full[b], (v_armed[b] - 1) & 1, 100000000ull);
    }
  }
}

template <int HD>
__device__ void mma_issuer(const AttnArgs& a, TcShared& sh, uint32_t tmem, uint32_t smem_base) {
  using C = TcCfg<HD>;
  volatile int* abort = &sh.abort;
  constexpr uint32_t idesc_s = tc::make_idesc(128, 128, false);
  constexpr uint32_t idesc_o = tc::make_idesc(128, HD, true);
  const uint32_t qs = smem_base + C::kQOffset;
  uint32_t it = 0;
  bool issued = false;
  auto issue_pv = [&](uint32_t itp, bool first_of_unit, int k) -> bool {
    const uint32_t sb = itp & 1u, st = itp % C::kStagesV;
    if (!tc_wait(&sh.p_full[sb], (itp >> 1) & 1, abort, a.err)) return false;
    if (!tc_wait(&sh.v_full[st], (itp / C::kStagesV) & 1, abort, a.err)) return false;
    if (first_of_unit && k > 0 && !tc_wait(&sh.o_free, (k - 1) & 1, abort, a.err)) return false;
    tc::fence_after_sync();
    const uint32_t vb = smem_base + C::kVOffset + st * C::kTileBytes;
#pragma unroll
    for (int kk = 0; kk < C::kN / 16; ++kk) {
      const uint64_t bdesc = tc::sdesc_sw128(vb + kk * (16 * 128), C::kHalfBytes, 1024);
      tc::mma_ts(tmem + C::kColO, tmem + sb * 128 + kk * 8, bdesc, idesc_o,
                 (first_of_unit && kk == 0) ? 0u : 1u);
    }
    tc::commit(&sh.o_done);
    tc::commit(&sh.v_empty[st]);
    return true;
  };
  for (int k = 0;; ++k) {
    const int slot = k % C::kRing;
    if (!tc_wait(&sh.unit_full[slot], (k / C::kRing) & 1, abort, a.err)) break;
    const TcUnit un = sh.units[slot];
    if (!un.valid) break;
    if (!tc_wait(&sh.q_full, k & 1, abort, a.err)) break;
    tc::fence_after_sync();
    bool ok = true;
    for (int j = 0; j < un.n_kt && ok; ++j) {
      const uint32_t itg = it + j, st = itg % C::kStagesK, sb = itg & 1u;
      if (!tc_wait(&sh.k_full[st], (itg / C::kStagesK) & 1, abort, a.err)) { ok = false; break; }
      tc::fence_after_sync();
      const uint32_t kb = smem_base + st * C::kTileBytes;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
        const uint32_t off = (ks >> 2) * C::kQHalfBytes + (ks & 3) * 32;
        const uint64_t adesc = tc::sdesc_sw128(qs + off, 16, 1024);
        const uint64_t bdesc = tc::sdesc_sw128(kb + (ks >> 2) * C::kHalfBytes + (ks & 3) * 32,
                                               16, 1024);
        tc::mma_ss(tmem + sb * 128, adesc, bdesc, idesc_s, ks > 0 ? 1u : 0u);
      }
      issued = true;
      tc::commit(&sh.s_full[sb]);
      tc::commit(&sh.k_empty[st]);
      if (j == un.n_kt - 1) tc::commit(&sh.q_empty);
      if (j > 0) ok = issue_pv(itg - 1, j == 1, k);
    }
    if (ok) ok = issue_pv(it + un.n_kt - 1, un.n_kt == 1, k);
    if (!ok) break;
    tc::mbar_arrive(&sh.unit_empty[slot]);
    it += un.n_kt;
  }
  if (issued) {  // every MMA and every commit-arrival lands before TMEM and smem are released
    tc::commit(&sh.drain);
    mbar_wait_bounded(&sh.drain, 0, 100000000ull);
  }
}

template <int HD>
__device__ void softmax_wg(const AttnArgs& a, TcShared& sh, uint32_t tmem, uint8_t* smem_ptr) {
  using C = TcCfg<HD>;
  volatile int* abort = &sh.abort;
  const int t = threadIdx.x;  // 0..127: query row within the tile and TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>((t >> 5) * 32) << 16;
  uint32_t it = 0, pv_seen = 0;
  auto wait_all = [&](uint64_t* bar, uint32_t phase) -> bool {
    const bool ok = tc_wait(bar, phase, abort, a.err);
    return !__any_sync(0xffffffffu, !ok);
  };
  auto catch_up = [&](uint32_t target) -> bool {  // consume o_done phases up to `target`
    while (pv_seen < target) {
      if (!wait_all(&sh.o_done, pv_seen & 1)) return false;
      ++pv_seen;
    }
    return true;
  };
  for (int k = 0;; ++k) {
    const int slot = k % C::kRing;
    if (!wait_all(&sh.unit_full[slot], (k / C::kRing) & 1)) break;
    const TcUnit un = sh.units[slot];
    if (!un.valid) break;
    const int row = un.row0 + t;
    const bool valid = row < un.rows_total;
    const int jt = valid ? row / a.group : 0;
    const int hh = valid ? row - jt * a.group : 0;
    const int lim = un.c + jt;
    const int lim_min = un.c + un.row0 / a.group;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < un.n_kt; ++j) {
      const uint32_t itg = it + j, sb = itg & 1u, sv = itg % C::kStagesV;
      if (!wait_all(&sh.s_full[sb], (itg >> 1) & 1)) { ok = false; break; }
      tc::fence_after_sync();
      float s[128];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tc::ld32(tmem + lane_off + sb * 128 + 0, r0);
        tc::ld32(tmem + lane_off + sb * 128 + 32, r1);
        tc::ld32(tmem + lane_off + sb * 128 + 64, r2);
        tc::ld32(tmem + lane_off + sb * 128 + 96, r3);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(r0[i]) * a.scale_log2;
          s[32 + i] = __uint_as_float(r1[i]) * a.scale_log2;
          s[64 + i] = __uint_as_float(r2[i]) * a.scale_log2;
          s[96 + i] = __uint_as_float(r3[i]) * a.scale_log2;
        }
      }
      const int kv_base = j * C::kN;
      if (kv_base + C::kN - 1 > lim_min) {
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = (kv_base + i <= lim) ? s[i] : -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
      for (int i = 8; i < 128; ++i) mx[i & 7] = fmaxf(mx[i & 7], s[i]);
      const float m_tile = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const bool need = m_tile > m_ref + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? m_tile : m_ref;
        const float alpha = fast_exp2(m_ref - m_new);
        if (j > 0) {
          if (!catch_up(itg)) { ok = false; break; }  // O must hold P_{j-1} V_{j-1}
          tc::fence_after_sync();
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            tc::ld32(tmem + lane_off + C::kColO + c * 32, r);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tc::st32(tmem + lane_off + C::kColO + c * 32, r);
          }
          tc::wait_st();
        }
        l *= alpha;
        m_ref = m_new;
      }
      // keys at or past the end of the sequence may hold anything: zero their V rows
      if (kv_base + C::kN > un.L) {
        if (!wait_all(&sh.v_full[sv], (itg / C::kStagesV) & 1)) { ok = false; break; }
        const int kmin = max(un.L - kv_base, 0);
        if (t >= kmin) {
          uint8_t* vrow = smem_ptr + C::kVOffset + sv * C::kTileBytes + t * 128;
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(vrow + hf * C::kHalfBytes + c * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
        }
      }
      const float mu = m_ref == -INFINITY ? 0.f : m_ref;
      float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = fast_exp2(s[c * 64 + 2 * i] - mu);
          const float p1 = fast_exp2(s[c * 64 + 2 * i + 1] - mu);
          rs[i & 7] += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tc::st32(tmem + lane_off + sb * 128 + c * 32, pk);
      }
      tc::wait_st();
      l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      // observe P_{j-1} V_{j-1} before P_j lets the next one start: o_done then never runs more
      // than one phase ahead of pv_seen, so its parity waits stay unambiguous
      if (!catch_up(itg)) { ok = false; break; }
      tc::fence_before_sync();
      tc::mbar_arrive(&sh.p_full[sb]);
    }
    if (!ok) break;
    it += un.n_kt;
    if (!catch_up(it)) break;  // every P V of this unit has landed in O
    tc::fence_after_sync();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(
        a.out + (static_cast<size_t>(un.t0 + jt) * a.nh + un.h * a.group + hh) * HD);
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      uint32_t r[32];
      tc::ld32(tmem + lane_off + C::kColO + c * 32, r);
      tc::wait_ld();
      if (valid) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv, __uint_as_float(r[8 * v + 1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv, __uint_as_float(r[8 * v + 3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv, __uint_as_float(r[8 * v + 5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv, __uint_as_float(r[8 * v + 7]) * inv);
          dst[c * 4 + v] = w;
        }
      }
    }
    tc::fence_before_sync();
    tc::mbar_arrive(&sh.o_free);
    tc::mbar_arrive(&sh.unit_empty[slot]);
  }
}

template <int HD>
__global__ void __launch_bounds__(TcCfg<HD>::kThreads, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                           const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  using C = TcCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ TcShared sh;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);

  if (tid == 0) {
    for (int i = 0; i < C::kRing; ++i) {
      mbar_init(&sh.unit_full[i], 1);
      mbar_init(&sh.unit_empty[i], 1 + 128);
    }
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&sh.k_full[i], 1);
      mbar_init(&sh.k_empty[i], 1);
      mbar_init(&sh.v_full[i], 1);
      mbar_init(&sh.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.p_full[i], 128);
    }
    mbar_init(&sh.o_done, 1);
    mbar_init(&sh.o_free, 128);
    mbar_init(&sh.drain, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(&sh.tmem_base, C::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 4) {
    producer<HD>(a, sh, base, &qmap, &kmap, &vmap);
  } else if (warp == 5) {
    if ((tid & 31) == 0) mma_issuer<HD>(a, sh, tmem, base);
  } else {
    softmax_wg<HD>(a, sh, tmem, base_ptr);
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 5) {
    __syncwarp();
    tc::tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int HD>
rb_status launch_hd(const AttnArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                    const CUtensorMap& vmap, cudaStream_t s) {
  using C = TcCfg<HD>;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RB_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(attn_prefill_tc_kernel<HD>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return RB_ERR_CUDA;
    configured[dev] = true;
  }
  const int grid = max(1, device_sm_count());
  attn_prefill_tc_kernel<HD><<<grid, C::kThreads, C::kSmemBytes, s>>>(qmap, kmap, vmap, a);
  if (last_launch_status() != RB_OK) return RB_ERR_CUDA;
  note_launches(1);
  return RB_OK;
}

}  // namespace

bool prefill_tc_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

rb_status launch_prefill_tc(const AttnArgs& a, int head_dim, const CUtensorMap& qmap,
                            const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t s) {
  return head_dim == 128 ? launch_hd<128>(a, qmap, kmap, vmap, s)
                         : launch_hd<64>(a, qmap, kmap, vmap, s);
}

}  // namespace attn
}  // namespace rb
