// Internal helpers shared by the librb kernels (sm_103a).  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "rb.h"

#ifdef RB_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace rb {

// One NVTX range around each C-ABI call, for timelines in a profiler.  Compiled in only with
// -DRB_NVTX (build.py: RB_NVTX=1 in the environment); otherwise it costs nothing.
struct CallRange {
#ifdef RB_NVTX
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
#else
  explicit CallRange(const char*) {}
#endif
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
void note_launches(int n);          // adds to rb_kernel_launch_count()

// Page-table geometry shared by the entry points that read a page table.
struct PageGeom {
  int ratio;        // kernel pages per page-table entry (manager block), >= 1
  int num_blocks;   // kernel pages in the pool
  int null_block;   // kernel page of the null page
};

// Validates the page-table fields of rb_dims; fills `g`.  RB_OK or RB_ERR_INVALID_ARG.
rb_status page_geom_of(const rb_dims& d, PageGeom* g);
int device_sm_count();              // SM count of the current device (cached per device)
rb_status last_launch_status();     // RB_ERR_CUDA if the previous launch failed

__host__ __device__ inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Encodes a 3-D TMA descriptor over a paged cache [num_slots, nkv, hd] bf16 with a box of
// {64 dims, 1 head, 16 slots} and 128-byte swizzle.  Returns false if the driver refuses it.
bool encode_kv_tensor_map(CUtensorMap* map, const void* base, int head_dim, int num_kv_heads,
                          long long num_slots);
// 3-D TMA descriptor over queries [num_tokens, nh, hd] bf16 with a box of {64 dims, `group`
// heads, 128 / group (rounded down) tokens} and 128-byte swizzle: one box = up to 128 (token,
// head) rows x 128 bytes.
bool encode_q_tensor_map(CUtensorMap* map, const void* base, int head_dim, int num_q_heads,
                         long long num_tokens, int group);

// ---------------------------------------------------------------------------------------------
// device side
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void raise_error(int32_t* err, int32_t bit) {
  if (err != nullptr) atomicOr(err, bit);
}

// Kernel page holding logical kernel page `pg` of a row whose page-table entries are manager
// blocks of `ratio` kernel pages: entry pg / ratio, page pg % ratio inside it.  Returns -1 when
// the entry is outside the pool or is the manager block that holds the null page, so callers
// treat it like any invalid page id.
__device__ __forceinline__ int kernel_page(const int32_t* bt_row, int pg, int ratio,
                                           int num_blocks, int null_block) {
  if (ratio == 1) {
    const int id = __ldg(bt_row + pg);
    return (id < 0 || id >= num_blocks || id == null_block) ? -1 : id;
  }
  const int m = __ldg(bt_row + pg / ratio);
  if (m < 0 || m >= num_blocks / ratio || m == null_block / ratio) return -1;
  return m * ratio + pg % ratio;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}
// 32-byte global store (sm_100 family); `p` must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, uint32_t r0, uint32_t r1, uint32_t r2,
                                             uint32_t r3, uint32_t r4, uint32_t r5, uint32_t r6,
                                             uint32_t r7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(r0),
               "r"(r1), "r"(r2), "r"(r3), "r"(r4), "r"(r5), "r"(r6), "r"(r7)
               : "memory");
}

// Non-blocking test of a phase, relaxed (see mbar_try_wait_relaxed).  Several of these issued
// back to back, their results combined before one branch, overlap their latencies.
__device__ __forceinline__ bool mbar_test_relaxed(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.relaxed.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}
// The same test with relaxed semantics: no acquire ordering of this thread's later memory
// accesses.  For a thread whose only consumers of the awaited data are asynchronous tcgen05
// operations ordered after the wait by tcgen05.fence::after_thread_sync.
__device__ __forceinline__ bool mbar_try_wait_relaxed(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.relaxed.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for `phase` of `bar` to complete; gives up after ~`limit_ns` and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t phase,
                                                  uint64_t limit_ns = 200000000ull) {
#pragma unroll 1
  for (int i = 0; i < 64; ++i)
    if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  while (true) {
    if (mbar_try_wait(bar, phase)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Fetch a tensor map (a __grid_constant__ kernel parameter) into the TMA unit's descriptor cache
// ahead of its first use.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled TMA load into shared memory, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst_smem, const CUtensorMap* map,
                                            uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst_smem),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transposes an 8x8 b16 matrix held one fragment row-pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// max(a, b, c) in one instruction (PTX three-input max.f32; a NaN input is ignored like fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// 2^x on the SFU (PTX ex2.approx.ftz.f32).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// First index i in [0, n) with a[i] > x (a sorted ascending), or n.
__device__ __forceinline__ int upper_bound_i32(const int32_t* a, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// The same, by a whole converged warp: each round the 32 lanes test 32 evenly spaced entries
// at once, so a search takes ceil(log32 n) dependent loads instead of log2 n.
__device__ __forceinline__ int warp_upper_bound_i32(const int32_t* a, int n, int32_t x) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = n;  // the answer lies in [lo, hi]
  while (lo < hi) {
    const int stride = (hi - lo + 31) / 32;
    const int idx = lo + lane * stride;
    const bool above = idx < hi && a[idx] > x;
    const unsigned valid = __ballot_sync(0xffffffffu, idx < hi);
    const unsigned hit = __ballot_sync(0xffffffffu, above);
    if (hit & 1u) return lo;  // a[lo] > x
    const int f = hit ? __ffs(hit) - 1 : 32 - __clz(valid);  // first lane above (or past the last valid)
    const int prev = lo + (f - 1) * stride;                  // a[prev] <= x
    if (hit) hi = lo + f * stride;
    lo = prev + 1;
    if (stride == 1) return hit ? hi : lo;
  }
  return lo;
}

// Byte offset of (row, 16-byte chunk) in a TMA box of 16 rows x 128 bytes with 128B swizzle.
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

}  // namespace rb
