// Prefill / chunk attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// The same persistent launch also runs the split-KV decode units (attn_decode_warp.cuh): the
// planner assigns each CTA a first kind of work (decode or prefill) so HBM-bound and
// tensor-bound units run side by side; a CTA whose queue empties helps with the other one.
//
// Prefill unit = (request, kv head, pair of 128-row query tiles A and B); rows are (query token,
// head of the group) pairs, token-major, so every K/V tile serves the whole query-head group
// and both tiles of the pair.  A tile holds T = 128 / group whole tokens (T * group rows; for a
// group that does not divide 128 the last rows hold no query and are masked out).  One CTA per
// SM (persistent; units pulled from an atomic counter, the most expensive pair of each request
// first), 12 warps with fixed roles (the single-thread MMA issuer is warp 0, the oldest warp of
// its SM sub-partition, which shares that scheduler with one softmax warp of each tile):
//   warp 1     TMA producer of units, Q and K: fetches units into a 4-entry ring, loads Q_A and
//              Q_B once per unit (3-D boxes {64 dims, group heads, T tokens}) and each 128-key
//              K tile (8 pages x 128-byte boxes, 128B swizzle, one page per lane) into a
//              2-stage K ring (K is freed once S is done);
//   warp 2     TMA producer of V: the same boxes into a 3-stage V ring;
//   warp 0     allocates all 512 TMEM columns (S_A, S_B, O_A, O_B); one thread issues the MMAs
//              in the order S_A(0) S_B(0) | PV_A(0) S_A(1) | PV_B(0) S_B(1) | PV_A(1) ...
//              S = Q K^T: M=128, N=128, K=hd, both operands K-major in shared memory;
//              O += P V:  M=128, N=hd,  K=128, P read from TMEM, V MN-major in shared memory;
//              so one tile's softmax runs while the tensor core works on the other tile;
//   warps 4-7  softmax of tile A, warps 8-11 softmax of tile B; thread t = query row t: reads its
//              S row from TMEM, masks causally, takes exponents against a running reference
//              (log2 domain) and keeps their sum, writes P (bf16) back over the S columns.  The
//              reference is the row's first-tile maximum and moves (O rescaled in TMEM, the
//              tile's exponents taken again) only when a tile's sum exceeds 2^20 (exact either
//              way: P and the sum share the reference), so a common tile takes no row maximum.
//              The epilogue reads O, divides by the sum, stores bf16 rows.  The side that reads
//              every K/V tile of the unit (B, or A alone) hands the Q, K and V slots back to the
//              producers as its S tiles land, so the issuer commits only S, O and its drain.
// All mbarrier waits are bounded; a timeout sets RB_EBIT_TIMEOUT, every role stops, in-flight
// copies and MMAs are drained with bounded waits and TMEM is freed before the CTA exits.
#include "attn_common.cuh"
#include "attn_decode_warp.cuh"
#include "tc_ptx.cuh"

namespace rb {
namespace attn {
namespace {

template <int HD>
struct TcCfg {
  static constexpr int kM = 128;                          // query rows per tile (2 per unit)
  static constexpr int kN = 128;                          // keys per K/V tile
  static constexpr int kPagesPerTile = kN / kPage;        // 8
  static constexpr int kHalves = HD / 64;                 // 128-byte swizzle atoms per row
  static constexpr int kHalfBytes = kN * 128;             // one 64-dim half of a K or V tile
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  static constexpr int kQHalfBytes = kM * 128;
  static constexpr int kQBytes = kHalves * kQHalfBytes;   // one Q tile
  // V tile j is read by the first block of step j, K tile j + 1 by the second half of it, and
  // both slots free at the same point (S of tile j - 1 landing): the deeper ring goes to V
  static constexpr int kStagesK = 2;
  static constexpr int kStagesV = 3;
  static constexpr int kVOffset = kStagesK * kTileBytes;
  static constexpr int kQOffset = kVOffset + kStagesV * kTileBytes;  // Q_A then Q_B
  static constexpr int kUsed = kQOffset + 2 * kQBytes;
  static_assert(8 * DecCfg<HD>::kStages * DecCfg<HD>::kStageBytes <= kUsed,
                "the decode phase's stages must fit in the prefill phase's shared memory");
  // at least 120 KB keeps one CTA per SM (each CTA holds all 512 TMEM columns)
  static constexpr int kSmemBytes = (kUsed + 1024) > 120 * 1024 ? (kUsed + 1024) : 120 * 1024;
  // 3 warpgroups launched at 168 registers per thread (the 64-bit-register pool of one SM for
  // 384 threads); the softmax warpgroups then take 216 and the producer/MMA warpgroup keeps 72:
  // 2 x 128 x 216 + 128 x 72 = 384 x 168.
  static constexpr int kThreads = 384;
  static constexpr int kLaunchRegs = 168;
  static constexpr int kSoftmaxRegs = 216;
  static constexpr int kControlRegs = 72;
  static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
  static constexpr int kMmaWarp = 0;
  static constexpr int kProducerWarp = 1;   // units, Q and K
  static constexpr int kProducerVWarp = 2;  // V (warp 3 only completes the first warpgroup)
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0;                   // S_A at 0, S_B at 128
  static constexpr uint32_t kColO0 = 256;                 // O_A at 256, O_B at 256 + HD
  static constexpr int kRing = 4;
  __device__ static constexpr uint32_t col_s(int x) { return kColS0 + 128u * x; }
  __device__ static constexpr uint32_t col_o(int x) { return kColO0 + static_cast<uint32_t>(HD) * x; }
};

// A unit of work: query tokens [tok0, tok0 + 2T) of the request's q (tile A the first T, tile
// B the next T), T = tile_tokens.  In a cascade prefix pass `r` holds the unit's prefix key
// range (the pages are row 0's), the tokens are the whole batch's, key indices are relative to
// the range's first key and no row is masked causally: every row sees keys [0, c].
struct TcUnit {
  int r, h, tok0, t0, q, L, c, n[2], n_kt, pages, valid;
};

// First page of a unit's keys and the page-table row they are read from.
__device__ __forceinline__ int unit_first_page(const AttnArgs& a, const TcUnit& un) {
  return a.cascade == kPrefixPass ? un.r * (a.prefix_split_keys / kPage) : 0;
}
__device__ __forceinline__ int unit_table_row(const AttnArgs& a, const TcUnit& un) {
  return a.cascade == kPrefixPass ? 0 : un.r;
}

struct TcShared {
  uint64_t unit_full[4], unit_empty[4];
  uint64_t q_full, q_empty;
  uint64_t k_full[TcCfg<128>::kStagesK], k_empty[TcCfg<128>::kStagesK];
  uint64_t v_full[TcCfg<128>::kStagesV], v_empty[TcCfg<128>::kStagesV];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t drain;
  uint64_t dec_bars[8][DecCfg<128>::kStages];  // decode phase: one ring per warp 0..7
  TcUnit units[4];
  uint32_t tmem_base;
  int abort;
  int decode_first;
  int role_rank;  // order in which this CTA took its role: decode-first CTAs are ranks 0..D-1
};

// Bounded wait (a.wait_limit_ns, 1 s unless a test shortened it) that also gives up as soon as
// another role has aborted.  `Relaxed`: for the MMA issuer (see mma_issuer).
template <bool Relaxed = false>
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t phase, volatile int* abort,
                                        const AttnArgs& a) {
  int32_t* err = a.err;
  auto test = [&]() { return Relaxed ? mbar_try_wait_relaxed(bar, phase) : mbar_try_wait(bar, phase); };
#pragma unroll 1
  for (int i = 0; i < 128; ++i)
    if (test()) return true;
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  while (true) {
    if (test()) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > a.wait_limit_ns) {
      if (atomicExch(const_cast<int*>(abort), 1) == 0) raise_error(err, RB_EBIT_TIMEOUT);
      return false;
    }
  }
}

// Largest sum of one tile's exponents (128 keys of one row) taken against a lagging reference:
// P <= 2^20 keeps P V and the row sum far inside fp32 and bf16 range.
constexpr float kSumLimit = 1048576.f;

__device__ __forceinline__ int tiles_for(int c, int jmax) { return (c + jmax + 1 + 127) / 128; }
constexpr int kKeysPerTile = 128;  // keys per K/V tile

__device__ __forceinline__ TcUnit decode_unit(const AttnArgs& a, int u) {
  TcUnit un{};
  const int T = a.tile_tokens;
  if (a.cascade == kPrefixPass) {
    // (key range, kv head, 2T query tokens of the whole batch) against one range of the shared
    // keys [0, P) of row 0; key indices are relative to the range's first key
    const int per_split = a.nkv * ((a.N + 2 * T - 1) / (2 * T));
    const int split = u / per_split, rem = u - split * per_split;
    const int k0 = split * a.prefix_split_keys;
    const int k1 = min(a.prefix_len, k0 + a.prefix_split_keys);
    un.r = split;
    un.h = rem % a.nkv;
    un.tok0 = (rem / a.nkv) * 2 * T;
    un.t0 = 0;
    un.q = a.N;
    un.L = k1 - k0;
    un.c = un.L - 1;
    const int nk = (un.L + kKeysPerTile - 1) / kKeysPerTile;
    un.n[0] = nk;
    un.n[1] = un.tok0 + T < un.q ? nk : 0;
    un.n_kt = nk;
    un.pages = (un.L + kPage - 1) / kPage;
    un.valid = 1;
    return un;
  }
  // the planner lists the (request, pair) entries longest first; the kv heads of one entry
  // are consecutive units
  const int entry = __ldg(a.pre_list + u / a.nkv);
  const int r = entry >> 16, pair = entry & 0xffff;
  un.r = r;
  un.h = u % a.nkv;
  un.t0 = a.qsl[r];
  un.q = a.qsl[r + 1] - un.t0;
  un.L = a.seq_lens[r];
  un.c = un.L - un.q;
  un.tok0 = pair * 2 * T;
  un.n[0] = tiles_for(un.c, min(un.tok0 + T, un.q) - 1);
  un.n[1] = un.tok0 + T < un.q ? tiles_for(un.c, min(un.tok0 + 2 * T, un.q) - 1) : 0;
  un.n_kt = max(un.n[0], un.n[1]);
  un.pages = (un.L + kPage - 1) / kPage;
  un.valid = 1;
  return un;
}

// Page ids of a unit's K/V tiles for one warp: a 32-page window of the unit's block-table row
// held one id per lane, the next window prefetched; lane l & 7 takes page l & 7 of a tile.
struct PageWindow {
  const AttnArgs& a;
  const int32_t* bt_row;
  int page0, pages, win, bid, bid_next, lane;
  __device__ PageWindow(const AttnArgs& a_, const TcUnit& un, int lane_)
      : a(a_),
        bt_row(a_.block_table + static_cast<size_t>(unit_table_row(a_, un)) * a_.MB),
        page0(unit_first_page(a_, un)),
        pages(un.pages),
        win(0),
        lane(lane_) {
    bid = page(lane);
    bid_next = page(32 + lane);
  }
  __device__ int page(int pg) const {
    return pg < pages ? kernel_page(bt_row, page0 + pg, a.ratio, a.num_blocks, a.null_block)
                      : a.null_block;
  }
  // This lane's page id for tile j (tiles are taken in order).  Pages past the sequence read
  // the null page (masked; V rows zeroed); an invalid id is reported when `report` and replaced
  // by the null page.
  __device__ int tile_page(int j, bool report) {
    const int first = j * kKeysPerTile / kPage;
    if (first - win >= 32) {
      win += 32;
      bid = bid_next;
      bid_next = page(win + 32 + lane);
    }
    int id = __shfl_sync(0xffffffffu, bid, first + (lane & 7) - win);
    const int pg = first + (lane & 7);
    if (pg >= pages) {
      id = a.null_block;
    } else if (id < 0 || id >= a.num_blocks || id == a.null_block) {
      if (report && lane < kKeysPerTile / kPage) raise_error(a.err, RB_EBIT_BLOCK_ID);
      id = a.null_block;
    }
    return id;
  }
};

// Producer of units, Q and K (warp 1, whole warp).  It takes units from the global counter
// into the 4-entry unit ring, loads Q_A and Q_B once per unit and each K tile into the K
// ring; lanes 0..7 each issue the boxes of one page of a tile.
template <int HD>
__device__ void producer_qk(const AttnArgs& a, TcShared& sh, uint32_t smem_base,
                            const CUtensorMap* qmap, const CUtensorMap* kmap) {
  using C = TcCfg<HD>;
  volatile int* abort = &sh.abort;
  const int lane = threadIdx.x & 31;
  const int n_units = a.header[kHNumPrefillUnits];
  uint32_t it = 0, q_armed = 0, k_armed[C::kStagesK] = {};
  // the unit ring guards plain shared memory (the unit descriptors): acquiring wait
  auto lane0_wait = [&](uint64_t* bar, uint32_t phase) -> bool {
    int ok = 1;
    if (lane == 0) ok = tc_wait(bar, phase, abort, a) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  // Q and K slots are read only by tcgen05.mma and written only by TMA: a relaxed test first
  // (an acquiring wait on a long-complete phase cost this warp a few hundred cycles per tile)
  auto slot_wait = [&](uint64_t* bar, uint32_t phase) -> bool {
    int ok = 1;
    if (lane == 0)
      ok = (mbar_test_relaxed(bar, phase) || tc_wait<true>(bar, phase, abort, a)) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  for (int k = 0;; ++k) {
    const int slot = k % C::kRing;
    if (!lane0_wait(&sh.unit_empty[slot], ((k / C::kRing) & 1) ^ 1)) break;
    int withhold = 0;
    if (lane == 0) {
      const int u = atomicAdd(a.header + kHPrefillNext, 1);
      TcUnit un{};
      if (u < n_units) un = decode_unit(a, u);
      sh.units[slot] = un;
      // test hook: CTA 0 stops before its first unit reaches the other roles, so their waits
      // for it run out while nothing of that unit has been issued
      withhold = a.withhold_first_unit && blockIdx.x == 0 && k == 0 && un.valid;
      if (!withhold) tc::mbar_arrive(&sh.unit_full[slot]);
    }
    if (__shfl_sync(0xffffffffu, withhold, 0)) break;
    __syncwarp();
    const TcUnit un = sh.units[slot];
    if (!un.valid) break;
    if (!slot_wait(&sh.q_empty, (k & 1) ^ 1)) break;
    if (lane == 0) {
      // one box per 64-dim half of a tile: T tokens x group heads = T * group rows of 128 bytes
      const int nq = un.n[1] > 0 ? 2 : 1;
      mbar_arrive_expect_tx(&sh.q_full, nq * C::kHalves * a.tile_tokens * a.group * 128);
      ++q_armed;
      for (int x = 0; x < nq; ++x)
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(smem_base + C::kQOffset + x * C::kQBytes + hf * C::kQHalfBytes, qmap,
                      &sh.q_full, hf * 64, un.h * a.group, un.t0 + un.tok0 + a.tile_tokens * x);
    }
    PageWindow pw(a, un, lane);
    bool ok = true;
    for (int j = 0; j < un.n_kt; ++j) {
      const int id = pw.tile_page(j, true);
      const uint32_t itk = it + j, st = itk % C::kStagesK;
      if (!slot_wait(&sh.k_empty[st], ((itk / C::kStagesK) & 1) ^ 1)) { ok = false; break; }
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
    if (!ok) break;
    it += un.n_kt;
  }
  if (lane == 0 && *abort) {  // let every copy already issued land before the CTA can exit
    if (q_armed) mbar_wait_bounded(&sh.q_full, (q_armed - 1) & 1, 100000000ull);
    for (int b = 0; b < C::kStagesK; ++b)
      if (k_armed[b]) mbar_wait_bounded(&sh.k_full[b], (k_armed[b] - 1) & 1, 100000000ull);
  }
}

// Producer of V (warp 2, whole warp): follows the unit ring like the other consumers and loads
// each V tile into the V ring.  A warp of its own, so that V tiles are issued as soon as their
// slot frees, not after the next K tile (one warp issuing both took about a whole key-tile step
// for the TMA issue and waits alone, and left V late).
template <int HD>
__device__ void producer_v(const AttnArgs& a, TcShared& sh, uint32_t smem_base,
                           const CUtensorMap* vmap) {
  using C = TcCfg<HD>;
  volatile int* abort = &sh.abort;
  const int lane = threadIdx.x & 31;
  uint32_t it = 0, v_armed[C::kStagesV] = {};
  auto lane0_wait = [&](uint64_t* bar, uint32_t phase) -> bool {
    int ok = 1;
    if (lane == 0) ok = tc_wait(bar, phase, abort, a) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  auto slot_wait = [&](uint64_t* bar, uint32_t phase) -> bool {
    int ok = 1;
    if (lane == 0)
      ok = (mbar_test_relaxed(bar, phase) || tc_wait<true>(bar, phase, abort, a)) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  for (int k = 0;; ++k) {
    const int slot = k % C::kRing;
    if (!lane0_wait(&sh.unit_full[slot], (k / C::kRing) & 1)) break;
    const TcUnit un = sh.units[slot];
    if (!un.valid) break;
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&sh.unit_empty[slot]);  // the descriptor is in registers
    PageWindow pw(a, un, lane);
    bool ok = true;
    for (int j = 0; j < un.n_kt; ++j) {
      const int id = pw.tile_page(j, false);
      const uint32_t itv = it + j, st = itv % C::kStagesV;
      if (!slot_wait(&sh.v_empty[st], ((itv / C::kStagesV) & 1) ^ 1)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(&sh.v_full[st], C::kTileBytes);
        ++v_armed[st];
      }
      __syncwarp();
      if (lane < C::kPagesPerTile) {
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(smem_base + C::kVOffset + st * C::kTileBytes + hf * C::kHalfBytes +
                          lane * (kPage * 128),
                      vmap, &sh.v_full[st], hf * 64, un.h, id * kPage);
      }
    }
    if (!ok) break;
    it += un.n_kt;
  }
  if (lane == 0 && *abort) {
    for (int b = 0; b < C::kStagesV; ++b)
      if (v_armed[b]) mbar_wait_bounded(&sh.v_full[b], (v_armed[b] - 1) & 1, 100000000ull);
  }
}

template <int HD>
__device__ void mma_issuer(const AttnArgs& a, TcShared& sh, uint32_t tmem, uint32_t smem_base) {
  using C = TcCfg<HD>;
  volatile int* abort = &sh.abort;
  constexpr uint32_t idesc_s = tc::make_idesc(128, 128, false);
  constexpr uint32_t idesc_o = tc::make_idesc(128, HD, true);
  uint32_t itk = 0;                       // K/V tiles consumed
  uint32_t tcount[2] = {0, 0};            // S (= P V) tiles per side
  uint32_t ucount[2] = {0, 0};            // units per side that used O
  bool issued = false;
  // Every barrier of the loop below guards data that only tcgen05.mma reads (P and O in tensor
  // memory, Q, K and V that TMA wrote to shared memory), and each wait is followed by
  // tcgen05.fence::after_thread_sync before the MMAs that read it, so the waits are relaxed: an
  // acquiring try_wait behind queued MMAs left the tensor pipe idle ~140 cycles per wait on this
  // GPU, a relaxed one costs nothing.  The unit descriptor is plain shared memory written by the
  // producer warp: its barrier keeps the acquiring wait.
  auto wait = [&](uint64_t* bar, uint32_t phase) { return tc_wait<true>(bar, phase, abort, a); };
  // A wait whose result decides a branch costs the issuing thread a few hundred cycles even when
  // the phase is long complete; so every barrier of one step is first tested at once (the tests
  // issue back to back, one branch on their conjunction) and only a step that finds one not yet
  // complete takes the bounded waits one by one.
  auto test = [](uint64_t* bar, uint32_t phase) { return mbar_test_relaxed(bar, phase); };
  // Shared-memory descriptors are built once: a k-step moves the start address by 32 bytes
  // within a 128-byte swizzle atom, a 64-dim half by a half tile, a stage or a Q tile by whole
  // tiles.  All of these only add to the address field in the descriptor's low word (which no
  // step carries out of), so the MMAs take the two 32-bit halves and add to the low one.
  const uint64_t q_desc0 = tc::sdesc_sw128(smem_base + C::kQOffset, 16, 1024);
  const uint64_t k_desc0 = tc::sdesc_sw128(smem_base, 16, 1024);
  const uint64_t v_desc0 = tc::sdesc_sw128(smem_base + C::kVOffset, C::kHalfBytes, 1024);
  const uint32_t q_lo = static_cast<uint32_t>(q_desc0), k_lo = static_cast<uint32_t>(k_desc0),
                 v_lo = static_cast<uint32_t>(v_desc0);
  const uint32_t q_hi = static_cast<uint32_t>(q_desc0 >> 32),
                 k_hi = static_cast<uint32_t>(k_desc0 >> 32),
                 v_hi = static_cast<uint32_t>(v_desc0 >> 32);
  auto step = [](int ks, uint32_t half_bytes) -> uint32_t {
    return ((ks >> 2) * half_bytes + (ks & 3) * 32) >> 4;
  };
  auto issue_s = [&](int x, uint32_t kt) {  // S_x = Q_x K^T into S_x
    const uint32_t kd = k_lo + (((kt % C::kStagesK) * C::kTileBytes) >> 4);
    const uint32_t qd = q_lo + ((x * C::kQBytes) >> 4);
    const uint32_t d = tmem + C::col_s(x);
    tc::mma_ss_lh(d, qd, q_hi, kd, k_hi, idesc_s, 0u);
#pragma unroll
    for (int ks = 1; ks < HD / 16; ++ks)
      tc::mma_ss_lh_acc(d, qd + step(ks, C::kQHalfBytes), q_hi, kd + step(ks, C::kHalfBytes),
                        k_hi, idesc_s);
    tc::commit(&sh.s_full[x]);
    issued = true;
  };
  // O_x (+)= P_x V.  Only the side's last P V of a unit is committed on its own (o_done): an
  // earlier one is covered by the commit of the S issued after it.
  auto issue_pv = [&](int x, uint32_t kt, bool first, bool last) {
    const uint32_t vd = v_lo + (((kt % C::kStagesV) * C::kTileBytes) >> 4);
    const uint32_t d = tmem + C::col_o(x), p = tmem + C::col_s(x);
    tc::mma_ts_lh(d, p, vd, v_hi, idesc_o, first ? 0u : 1u);
#pragma unroll
    for (int kk = 1; kk < C::kN / 16; ++kk)
      tc::mma_ts_lh_acc(d, p + kk * 8, vd + ((kk * 16 * 128) >> 4), v_hi, idesc_o);
    if (last) tc::commit(&sh.o_done[x]);
  };
  for (int k = 0;; ++k) {
    const int slot = k % C::kRing;
    if (!tc_wait(&sh.unit_full[slot], (k / C::kRing) & 1, abort, a)) break;
    const TcUnit un = sh.units[slot];
    if (!un.valid) break;
    const bool q_k = test(&sh.q_full, k & 1) & test(&sh.k_full[itk % C::kStagesK], (itk / C::kStagesK) & 1);
    if (!q_k && (!wait(&sh.q_full, k & 1) ||
                 !wait(&sh.k_full[itk % C::kStagesK], (itk / C::kStagesK) & 1)))
      break;
    tc::fence_after_sync();
    issue_s(0, itk);
    if (un.n[1] > 0) issue_s(1, itk);
    bool ok = true;
    for (int j = 0; j < un.n_kt && ok; ++j) {
      const uint32_t kt = itk + j;
      bool k_ready = false, v_ready = false;
#pragma unroll
      for (int x = 0; x < 2; ++x) {  // unrolled: the per-side counters stay in registers
        if (j >= un.n[x]) continue;
        // every wait of this side's step first, then one fence before its MMAs
        const bool next_s = j + 1 < un.n[x];
        const bool need_v = !v_ready, need_o = j == 0 && ucount[x] > 0, need_k = next_s && !k_ready;
        const uint32_t ph_p = (tcount[x] + j) & 1, ph_v = (kt / C::kStagesV) & 1,
                       ph_o = (ucount[x] - 1) & 1, ph_k = ((kt + 1) / C::kStagesK) & 1;
        uint64_t* bar_v = &sh.v_full[kt % C::kStagesV];
        uint64_t* bar_k = &sh.k_full[(kt + 1) % C::kStagesK];
        const bool ready = test(&sh.p_full[x], ph_p) & (!need_v || test(bar_v, ph_v)) &
                           (!need_o || test(&sh.o_free[x], ph_o)) & (!need_k || test(bar_k, ph_k));
        if (!ready && (!wait(&sh.p_full[x], ph_p) || (need_v && !wait(bar_v, ph_v)) ||
                       (need_o && !wait(&sh.o_free[x], ph_o)) || (need_k && !wait(bar_k, ph_k)))) {
          ok = false;
          break;
        }
        k_ready = k_ready || next_s;
        v_ready = true;
        tc::fence_after_sync();
        issue_pv(x, kt, j == 0, !next_s);
        if (next_s) issue_s(x, kt + 1);
      }
      if (!ok) break;
    }
    if (!ok) break;
    tc::mbar_arrive(&sh.unit_empty[slot]);
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      tcount[x] += un.n[x];
      if (un.n[x] > 0) ++ucount[x];
    }
    itk += un.n_kt;
  }
  if (issued) {  // every MMA and every commit-arrival lands before TMEM and smem are released
    tc::commit(&sh.drain);
    mbar_wait_bounded(&sh.drain, 0, 100000000ull);
  }
}

// Softmax and epilogue of tile x (0 = A, 1 = B); thread t = row t of the tile = TMEM lane t.
template <int HD>
__device__ void softmax_wg(const AttnArgs& a, TcShared& sh, uint32_t tmem, uint8_t* smem_ptr,
                           int x) {
  using C = TcCfg<HD>;
  volatile int* abort = &sh.abort;
  const int t = threadIdx.x & 127;
  const uint32_t lane_off = static_cast<uint32_t>((t >> 5) * 32) << 16;
  const uint32_t col_s = tmem + lane_off + C::col_s(x), col_o = tmem + lane_off + C::col_o(x);
  uint32_t tc_x = 0, itk = 0, uc_x = 0;  // S tiles, K/V tiles and units (with n > 0) of this side
  auto wait_all = [&](uint64_t* bar, uint32_t phase) -> bool {
    const bool ok = tc_wait(bar, phase, abort, a);
    return !__any_sync(0xffffffffu, !ok);
  };
  // One lane of each warp arrives for the warp: 128 arrivals on one barrier load the barrier
  // unit that the MMA issuer's waits go through.
  const bool lane0 = (t & 31) == 0;
  auto arrive_warp = [&](uint64_t* bar) {
    __syncwarp();
    if (lane0) tc::mbar_arrive(bar);
  };
  // s_full of tile j tracks every MMA issued before S_j, P V of tile j - 1 among them; o_done
  // completes once per unit of this side, after its last P V.
  for (int k = 0;; ++k) {
    const int slot = k % C::kRing;
    if (!wait_all(&sh.unit_full[slot], (k / C::kRing) & 1)) break;
    const TcUnit un = sh.units[slot];
    if (!un.valid) break;
    const int n = un.n[x];
    // row t of this tile: token tok_base + t / group, head t % group of the kv head's group;
    // rows past T * group (a group that does not divide 128) or past the last token hold no
    // query: every key is masked for them and they are never stored
    const int tok_base = un.tok0 + a.tile_tokens * x;
    const int rows_used = a.tile_tokens * a.group;
    const int jt_in = t / a.group;
    const bool valid = t < rows_used && tok_base + jt_in < un.q;
    const int jt = valid ? tok_base + jt_in : 0;
    const int hh = valid ? t - jt_in * a.group : 0;
    const bool causal = a.cascade != kPrefixPass;
    const int lim = !valid ? -1 : (causal ? un.c + jt : un.c);
    const int lim_min = causal ? un.c + tok_base : un.c;
    const bool partial = rows_used < C::kM || tok_base + a.tile_tokens > un.q;
    // The side that reads every K/V tile of the unit (B, or A when B is empty: B's rows come
    // later, so it sees at least A's keys) hands the Q, K and V slots back to the producers:
    // its S of tile j landing means every MMA issued before that S has completed, S_A of tile
    // j and both P V of tile j - 1 among them; its last P V landing (o_done) frees the last V.
    // This keeps those arrivals off the MMA issuer, whose commits are its critical path.
    const bool releases = x == (un.n[1] > 0 ? 1 : 0);
    // running reference (log2 domain) and sum; a row without a query starts at 0, so that only
    // rows with visible keys take the first tile's maximum
    float m_ref = valid ? -INFINITY : 0.f, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const uint32_t tj = tc_x + j;
      if (!wait_all(&sh.s_full[x], tj & 1)) { ok = false; break; }
      if (releases && t == 0) {
        const uint32_t kt = itk + j;
        tc::mbar_arrive(&sh.k_empty[kt % C::kStagesK]);
        if (j > 0) tc::mbar_arrive(&sh.v_empty[(kt - 1) % C::kStagesV]);
        if (j + 1 == n) tc::mbar_arrive(&sh.q_empty);
      }
      tc::fence_after_sync();
      float s[128];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tc::ld32(col_s + 0, r0);
        tc::ld32(col_s + 32, r1);
        tc::ld32(col_s + 64, r2);
        tc::ld32(col_s + 96, r3);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(r0[i]);
          s[32 + i] = __uint_as_float(r1[i]);
          s[64 + i] = __uint_as_float(r2[i]);
          s[96 + i] = __uint_as_float(r3[i]);
        }
      }
      const int kv_base = j * C::kN;
      if (partial || kv_base + C::kN - 1 > lim_min) {
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = (kv_base + i <= lim) ? s[i] : -INFINITY;
      }
      // The exponents are taken against the running reference m_ref, not against this tile's
      // maximum: any reference gives the same softmax, since P and the sum share it.  The row
      // maximum is taken only (a) on the first tile of a row and (b) when the tile's sum of
      // exponents shows the reference lagging the row's maximum by more than log2 of
      // kSumLimit (or overflowing); then O and the sum are rescaled to the new reference and
      // the tile's exponents are taken again.  So P <= kSumLimit always, and the common tile
      // skips the maximum over its 128 columns.
      auto take_tile_max = [&]() {
        // eight running maxima over the 16 groups of 8 columns, three-input max instructions
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = fmax3(s[k], s[8 + k], s[16 + k]);
#pragma unroll
        for (int g = 3; g + 1 < 16; g += 2)
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], s[8 * g + k], s[8 * g + 8 + k]);
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], s[120 + k]);
        // scores are scaled inside the exponent: max and mask commute with a positive scale
        const float m_tile = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                   fmaxf(mx[6], mx[7])) *
                             a.scale_log2;
        const bool need = m_tile > m_ref;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? m_tile : m_ref;
          const float alpha = fast_exp2(m_ref - m_new);
          if (j > 0) {  // O holds P_{j-1} V_{j-1}: S_j, issued after it, has landed
            uint32_t r[32];
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
              tc::ld32(col_o + c * 32, r);
              tc::wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
              tc::st32(col_o + c * 32, r);
            }
            tc::wait_st();
          }
          l *= alpha;
          m_ref = m_new;
        }
      };
      if (__any_sync(0xffffffffu, m_ref == -INFINITY)) take_tile_max();
      // keys at or past the end of the sequence may hold anything: zero their V rows (only the
      // unit's last K/V tile can reach them; tile A zeroes it when it uses that tile)
      if (kv_base + C::kN > un.L && (x == 0 || j >= un.n[0])) {
        const uint32_t kt = itk + j, sv = kt % C::kStagesV;
        if (!wait_all(&sh.v_full[sv], (kt / C::kStagesV) & 1)) { ok = false; break; }
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
      // exponents and the row sum two columns at a time with the paired fp32 FMA / add
      // instructions; P (bf16) goes over the S columns
      auto exponents = [&]() -> float {
        const float mu = m_ref == -INFINITY ? 0.f : m_ref;
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2), nmu2 = make_float2(-mu, -mu);
        float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 e = __ffma2_rn(make_float2(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]),
                                        sc2, nmu2);
            const float2 p = make_float2(fast_exp2(e.x), fast_exp2(e.y));
            rs[i & 3] = __fadd2_rn(rs[i & 3], p);
            pk[i] = pack_bf16x2(p.x, p.y);
          }
          tc::st16(col_s + c * 16, pk);
        }
        const float2 rs01 = __fadd2_rn(rs[0], rs[1]), rs23 = __fadd2_rn(rs[2], rs[3]);
        const float2 rsum = __fadd2_rn(rs01, rs23);
        return rsum.x + rsum.y;
      };
      float rsum = exponents();
      if (__any_sync(0xffffffffu, !(rsum <= kSumLimit))) {  // rare: re-reference this tile
        tc::wait_st();
        take_tile_max();
        rsum = exponents();
      }
      tc::wait_st();
      // P_j overwrites the S columns P_{j-1} V_{j-1} read: that product is done, since S_j (the
      // MMA after it) has landed
      tc::fence_before_sync();
      arrive_warp(&sh.p_full[x]);
      l += rsum;
    }
    if (!ok) break;
    const uint32_t kt_last = itk + un.n_kt - 1;
    itk += un.n_kt;
    if (n > 0) {
      if (!wait_all(&sh.o_done[x], uc_x & 1)) break;  // the unit's last P V is in O
      if (releases && t == 0) tc::mbar_arrive(&sh.v_empty[kt_last % C::kStagesV]);
      ++uc_x;
      tc_x += n;
      tc::fence_after_sync();
      // the whole O row into registers at once; O is then free for the next unit's P V while
      // this row is scaled and stored
      uint32_t o[HD];
#pragma unroll
      for (int c = 0; c < HD / 32; ++c)
        tc::ld32(col_o + c * 32, *reinterpret_cast<uint32_t(*)[32]>(o + c * 32));
      tc::wait_ld();
      tc::fence_before_sync();
      arrive_warp(&sh.o_free[x]);
      const size_t orow = static_cast<size_t>(un.t0 + jt) * a.nh + un.h * a.group + hh;
      // rows are written with 32-byte stores when the output is 32-byte aligned (a warp's
      // rows are scattered: fewer, whole-sector stores), else 16-byte ones
      if (a.cascade == kPrefixPass) {
        // shared-prefix row: normalised fp32 output and its log-sum-exp, merged later
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t prow = static_cast<size_t>(un.r) * a.N * a.nh + orow;
        float* dst = a.pre_o + prow * HD;
        if (valid) {
#pragma unroll
          for (int i = 0; i < HD; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * inv);
          if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
#pragma unroll
            for (int v = 0; v < HD / 8; ++v)
              st_global_v8(dst + 8 * v, o[8 * v], o[8 * v + 1], o[8 * v + 2], o[8 * v + 3],
                           o[8 * v + 4], o[8 * v + 5], o[8 * v + 6], o[8 * v + 7]);
          } else {
#pragma unroll
            for (int v = 0; v < HD / 4; ++v)
              reinterpret_cast<uint4*>(dst)[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
          }
          a.pre_lse[prow] = l > 0.f ? m_ref + __log2f(l) : -INFINITY;
        }
      } else if (valid) {
        // out = O * wa + sum over prefix key ranges of (shared-prefix row) * wp (cascade only)
        float wa = 1.f / l;
        float wp[kMaxPrefixSplits];
        const bool cas = a.cascade == kSuffixPass;
        if (cas) wa = cascade_weights(a, orow, m_ref, l, wp);
        else if (!(l > 0.f)) wa = 0.f;
#pragma unroll
        for (int i = 0; i < HD; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * wa);
        if (cas) {
#pragma unroll
          for (int ps = 0; ps < kMaxPrefixSplits; ++ps) {
            if (ps >= a.prefix_splits) break;
            const float4* o1 = reinterpret_cast<const float4*>(cascade_row<HD>(a, ps, orow));
#pragma unroll
            for (int v = 0; v < HD / 4; ++v) {
              const float4 e = __ldg(o1 + v);
              o[4 * v + 0] = __float_as_uint(__uint_as_float(o[4 * v + 0]) + e.x * wp[ps]);
              o[4 * v + 1] = __float_as_uint(__uint_as_float(o[4 * v + 1]) + e.y * wp[ps]);
              o[4 * v + 2] = __float_as_uint(__uint_as_float(o[4 * v + 2]) + e.z * wp[ps]);
              o[4 * v + 3] = __float_as_uint(__uint_as_float(o[4 * v + 3]) + e.w * wp[ps]);
            }
          }
        }
        uint32_t pk[HD / 2];
#pragma unroll
        for (int i = 0; i < HD / 2; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]));
        __nv_bfloat16* dst = a.out + orow * HD;
        if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
#pragma unroll
          for (int v = 0; v < HD / 16; ++v)
            st_global_v8(dst + 16 * v, pk[8 * v], pk[8 * v + 1], pk[8 * v + 2], pk[8 * v + 3],
                         pk[8 * v + 4], pk[8 * v + 5], pk[8 * v + 6], pk[8 * v + 7]);
        } else {
#pragma unroll
          for (int v = 0; v < HD / 8; ++v)
            reinterpret_cast<uint4*>(dst)[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
    }
    arrive_warp(&sh.unit_empty[slot]);
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
  if (tid == 32) {  // the three descriptors every role's first copies use
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  if (tid == 0) {
    for (int i = 0; i < C::kRing; ++i) {
      mbar_init(&sh.unit_full[i], 1);
      // the issuer, one lane of each softmax warp and the V producer
      mbar_init(&sh.unit_empty[i], 1 + 8 + 1);
    }
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    for (int i = 0; i < C::kStagesK; ++i) {
      mbar_init(&sh.k_full[i], 1);
      mbar_init(&sh.k_empty[i], 1);
    }
    for (int i = 0; i < C::kStagesV; ++i) {
      mbar_init(&sh.v_full[i], 1);
      mbar_init(&sh.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.p_full[i], 4);  // one lane of each softmax warp
      mbar_init(&sh.o_done[i], 1);
      mbar_init(&sh.o_free[i], 4);
    }
    mbar_init(&sh.drain, 1);
    for (int w = 0; w < 8; ++w)
      for (int st = 0; st < DecCfg<128>::kStages; ++st) mbar_init(&sh.dec_bars[w][st], 1);
    sh.abort = 0;
    sh.role_rank = atomicAdd(a.header + kHRoleNext, 1);
    sh.decode_first = sh.role_rank < a.header[kHDecodeCtas];
    fence_barrier_init();
  }
  if (warp == C::kMmaWarp) {
    tc::tmem_alloc(&sh.tmem_base, C::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  // Two phases: the kind of work the planner assigned this CTA first, then the other kind
  // until its queue is empty too.  The decode phase runs on warps 4-11, each with its own ring of
  // decode stages in the same shared memory the prefill phase uses.  Each register class keeps
  // its own loop so the code after setmaxnreg stays within that class's budget.
  const bool decode_first = sh.decode_first != 0;
  auto phase_end = [] {
    fence_proxy_async_smem();  // generic smem traffic of this phase before the next one's TMA
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  };
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kControlRegs));
    for (int phase = 0; phase < 2; ++phase) {
      if ((phase == 0) != decode_first) {
        if (warp == C::kProducerWarp) {
          producer_qk<HD>(a, sh, base, &qmap, &kmap);
        } else if (warp == C::kProducerVWarp) {
          producer_v<HD>(a, sh, base, &vmap);
        } else if (warp == C::kMmaWarp) {
          if ((tid & 31) == 0) mma_issuer<HD>(a, sh, tmem, base);
        }
      }
      phase_end();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kSoftmaxRegs));
    for (int phase = 0; phase < 2; ++phase) {
      if ((phase == 0) == decode_first) {
        using D = DecCfg<HD>;
        const int w = warp - 4;
        // a decode-first CTA's warps start on units rank x 8 + w without the counter
        decode_warp<HD>(&kmap, &vmap, a, sh.dec_bars[w], base + w * D::kStages * D::kStageBytes,
                        base_ptr + w * D::kStages * D::kStageBytes,
                        decode_first ? sh.role_rank * a.decode_warps_per_cta + w : -1);
      } else {
        softmax_wg<HD>(a, sh, tmem, base_ptr, (warp >> 2) - 1);
      }
      phase_end();
    }
  }
  if (warp == C::kMmaWarp) {
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

rb_status launch_prefill_tc(const AttnArgs& a, int head_dim, const CUtensorMap& qmap,
                            const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t s) {
  return head_dim == 128 ? launch_hd<128>(a, qmap, kmap, vmap, s)
                         : launch_hd<64>(a, qmap, kmap, vmap, s);
}

}  // namespace attn
}  // namespace rb
