// rb_batch_apply_update: the runner's per-step merge of scheduler deltas into the persistent
// batch, on the device.
//
// "vLLM 源码完全拆解（五）…": "先删除完成和本轮未调度的请求", "新请求建立完整状态",
// "驻留请求只合并差量", "最后压紧并刷新派生 metadata", "行号是一种短生命周期地址";
// "第8章 ModelRunner…": "8.2.2.5" (removals first, new requests take the freed rows) and
// "8.2.2.6" (an id scheduled as new again names a new request); "04 · 模型执行与 CUDA Graph",
// "4.2 块表" (append_row).
//
// Two launches.  A one-block planner reads the request ids of the live rows, the schedule and
// the delta lists, validates all of it, and only then writes: the counter columns of every
// final row, the cleared rows past the new end, d_num_scheduled / d_row_of_sched, and a list of
// copy descriptors (token and page rows that move or arrive) in the workspace.  A grid of
// 256-thread blocks then performs the copies in 16 KiB chunks with 16-byte accesses.  Sources
// of the copies are rows past the new end (which nothing writes any more) and the update's
// payload, destinations are rows below the new end, so the copies never overlap.  If the
// planner finds an error it writes nothing but the status, and the copy kernel does nothing.
#include "rb_internal.cuh"

namespace rb {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kCopyThreads = 256;
constexpr int kChunk = 4096;            // int32 elements per copy chunk (16 KiB)
constexpr int kMaxRows = 4096;
constexpr long long kEmpty = -1;
constexpr int kUnset = -0x7fffffff;     // final_src of a row nothing was assigned to

enum : int { kSrcTok = 0, kSrcBlk = 1, kSrcNewTok = 2, kSrcNewBlk = 3, kSrcCachedTok = 4,
             kSrcCachedBlk = 5 };

struct CopyDesc {
  long long src;   // element offset into the source array
  long long dst;   // element offset into the token table (dst_blk == 0) or the page table
  int count;       // int32 elements
  int kinds;       // source kind | (dst_blk << 8)
};

struct WsLayoutB {
  size_t header, desc, chunk_start, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayoutB ws_layout(int max_rows) {
  WsLayoutB w;
  const size_t max_desc = 4 * static_cast<size_t>(max_rows);
  w.header = 0;
  w.desc = 64;
  w.chunk_start = align_up(w.desc + max_desc * sizeof(CopyDesc), 16);
  w.total = align_up(w.chunk_start + (max_desc + 1) * sizeof(int), 256);
  return w;
}

struct PlanArgs {
  rb_batch b;
  rb_batch_update u;
  int32_t* num_sched_out;
  int32_t* row_of_sched;
  int32_t* err;
  unsigned char* ws;
  int hash_cap;  // power of two >= 2 * S
};

__device__ __forceinline__ unsigned hash_id(long long key, int cap) {
  unsigned long long x = static_cast<unsigned long long>(key);
  x ^= x >> 33;
  x *= 0xff51afd7ed558ccdULL;
  x ^= x >> 33;
  return static_cast<unsigned>(x) & static_cast<unsigned>(cap - 1);
}

__device__ int hash_find(const long long* keys, const int* vals, int cap, long long key) {
  unsigned h = hash_id(key, cap);
  for (int it = 0; it < cap; ++it) {
    const long long k = keys[h];
    if (k == key) return vals[h];
    if (k == kEmpty) return -1;
    h = (h + 1) & static_cast<unsigned>(cap - 1);
  }
  return -1;
}

// Exclusive prefix sum over the block (kPlanThreads threads); *total gets the block's sum.
__device__ int block_exclusive_scan(int v, int* warp_tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tmp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_tmp[lane] = w;  // inclusive sums of the warps
  }
  __syncthreads();
  const int before = (warp == 0 ? 0 : warp_tmp[warp - 1]) + x - v;
  *total = warp_tmp[31];
  __syncthreads();
  return before;
}

__device__ void emit(CopyDesc* desc, int* n_desc, int src_kind, bool dst_blk, long long src,
                     long long dst, int count) {
  if (count <= 0) return;
  const int slot = atomicAdd(n_desc, 1);
  CopyDesc d;
  d.src = src;
  d.dst = dst;
  d.count = count;
  d.kinds = src_kind | (dst_blk ? 256 : 0);
  desc[slot] = d;
}

__global__ void __launch_bounds__(kPlanThreads) batch_plan_kernel(PlanArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_err, s_n_desc, s_holes, s_above;
  __shared__ int warp_tmp[32];
  const rb_batch& b = a.b;
  const rb_batch_update& u = a.u;
  const int NR = b.max_num_reqs, M = b.max_model_len, MB = b.max_blocks_per_req;
  const int S = u.num_scheduled, NN = u.num_new, NC = u.num_cached, H = a.hash_cap;
  const int tid = threadIdx.x;
  long long* hkey = reinterpret_cast<long long*>(smem);  // [H] request ids of the schedule
  int* hval = reinterpret_cast<int*>(hkey + H);          // [H] their index in the schedule
  int* row_sched = hval + H;                             // [NR] schedule index kept in row r
  int* aux = row_sched + NR;                             // [NR] freed rows, ascending
  int* final_src = aux + NR;                             // [NR] source of final row f
  int* sched_row = final_src + NR;                       // [S] old row of a resident request
  int* sched_new = sched_row + S;                        // [S] index in the new list
  int* sched_cached = sched_new + S;                     // [S] index in the delta list
  int* header = reinterpret_cast<int*>(a.ws);
  CopyDesc* desc = reinterpret_cast<CopyDesc*>(a.ws + ws_layout(NR).desc);
  int* chunk_start = reinterpret_cast<int*>(a.ws + ws_layout(NR).chunk_start);

  if (tid == 0) {
    s_err = 0;
    s_n_desc = 0;
  }
  for (int i = tid; i < H; i += kPlanThreads) hkey[i] = kEmpty;
  for (int i = tid; i < NR; i += kPlanThreads) {
    row_sched[i] = -1;
    final_src[i] = kUnset;
  }
  for (int i = tid; i < S; i += kPlanThreads) sched_row[i] = sched_new[i] = sched_cached[i] = -1;
  const int old_n = *b.d_num_rows;
  __syncthreads();
  if (old_n < 0 || old_n > NR) {
    if (tid == 0) atomicOr(&s_err, RB_EBIT_BATCH_SIZE);
  }

  // the schedule, keyed by request id
  for (int s = tid; s < S; s += kPlanThreads) {
    const long long key = u.d_sched_req_id[s];
    if (key < 0) {
      atomicOr(&s_err, RB_EBIT_BATCH_ID);
      continue;
    }
    unsigned h = hash_id(key, H);
    for (int it = 0; it < H; ++it) {
      const long long prev = static_cast<long long>(
          atomicCAS(reinterpret_cast<unsigned long long*>(hkey + h),
                    static_cast<unsigned long long>(kEmpty), static_cast<unsigned long long>(key)));
      if (prev == kEmpty) {
        hval[h] = s;
        break;
      }
      if (prev == key) {  // scheduled twice
        atomicOr(&s_err, RB_EBIT_BATCH_ID);
        break;
      }
      h = (h + 1) & static_cast<unsigned>(H - 1);
    }
  }
  __syncthreads();

  // new requests: scheduled, announced once, payload sizes within the row
  for (int k = tid; k < NN; k += kPlanThreads) {
    const int s = hash_find(hkey, hval, H, u.d_new_req_id[k]);
    if (s < 0 || atomicExch(sched_new + s, k) != -1) atomicOr(&s_err, RB_EBIT_BATCH_ID);
    const int t0 = u.d_new_token_start[k], t1 = u.d_new_token_start[k + 1];
    const int b0 = u.d_new_block_start[k], b1 = u.d_new_block_start[k + 1];
    if (t0 < 0 || t1 < t0 || t1 - t0 > M || b0 < 0 || b1 < b0 || b1 - b0 > MB)
      atomicOr(&s_err, RB_EBIT_BATCH_SIZE);
  }
  __syncthreads();

  // live rows: kept iff scheduled and not announced again as new (step 1)
  if (s_err == 0) {
    for (int r = tid; r < old_n; r += kPlanThreads) {
      const long long id = b.d_req_id[r];
      const int s = id < 0 ? -1 : hash_find(hkey, hval, H, id);
      if (s < 0 || sched_new[s] >= 0) continue;
      if (atomicExch(sched_row + s, r) != -1) atomicOr(&s_err, RB_EBIT_BATCH_ID);
      row_sched[r] = s;
      const int nt = b.d_num_tokens[r], nb = b.d_num_blocks[r];
      if (nt < 0 || nt > M || nb < 0 || nb > MB) atomicOr(&s_err, RB_EBIT_BATCH_SIZE);
    }
  }
  __syncthreads();

  // deltas of resident requests (step 2 is applied below, at the request's final row)
  if (s_err == 0) {
    for (int c = tid; c < NC; c += kPlanThreads) {
      const int s = hash_find(hkey, hval, H, u.d_cached_req_id[c]);
      if (s < 0 || sched_row[s] < 0 || atomicExch(sched_cached + s, c) != -1) {
        atomicOr(&s_err, RB_EBIT_BATCH_ID);
        continue;
      }
      const int r = sched_row[s];
      const int t0 = u.d_cached_token_start[c], t1 = u.d_cached_token_start[c + 1];
      const int b0 = u.d_cached_block_start[c], b1 = u.d_cached_block_start[c + 1];
      const int base = u.d_cached_replace[c] ? 0 : b.d_num_blocks[r];
      if (t0 < 0 || t1 < t0 || b0 < 0 || b1 < b0 ||
          static_cast<long long>(b.d_num_tokens[r]) + (t1 - t0) > M ||
          static_cast<long long>(base) + (b1 - b0) > MB)
        atomicOr(&s_err, RB_EBIT_BATCH_SIZE);
    }
    for (int s = tid; s < S; s += kPlanThreads)
      if (sched_row[s] < 0 && sched_new[s] < 0) atomicOr(&s_err, RB_EBIT_BATCH_ID);
  }
  __syncthreads();
  if (s_err != 0) {
    if (tid == 0) {
      header[0] = s_err;
      header[1] = header[2] = 0;
      atomicOr(a.err, s_err);
    }
    return;
  }

  // freed rows below the old end, ascending
  for (int base = 0; base < old_n; base += kPlanThreads) {
    const int r = base + tid;
    const int hole = (r < old_n && row_sched[r] < 0) ? 1 : 0;
    int tile_total;
    const int rank = block_exclusive_scan(hole, warp_tmp, &tile_total);
    const int before = base == 0 ? 0 : s_holes;
    if (hole) aux[before + rank] = r;
    __syncthreads();
    if (tid == 0) s_holes = before + tile_total;
    __syncthreads();
  }
  if (old_n == 0 && tid == 0) s_holes = 0;
  __syncthreads();
  const int holes = s_holes;
  const int F = old_n - holes + NN;  // == S: every scheduled request is resident or new

  // kept rows below F stay; new request k takes the k-th freed row, then the tail (step 3)
  for (int r = tid; r < min(F, old_n); r += kPlanThreads)
    if (row_sched[r] >= 0) final_src[r] = r;
  for (int k = tid; k < NN; k += kPlanThreads)
    final_src[k < holes ? aux[k] : old_n + (k - holes)] = -2 - k;
  // condense (step 4): the j-th highest kept row at or past F fills the j-th remaining hole
  for (int base = F; base < old_n; base += kPlanThreads) {
    const int r = base + tid;
    const int kept = (r < old_n && row_sched[r] >= 0) ? 1 : 0;
    int tile_total;
    const int rank = block_exclusive_scan(kept, warp_tmp, &tile_total);
    const int before = base == F ? 0 : s_above;
    if (kept) aux[NR - 1 - (before + rank)] = r;  // ascending from the top of aux
    __syncthreads();
    if (tid == 0) s_above = before + tile_total;
    __syncthreads();
  }
  if (tid == 0 && F >= old_n) s_above = 0;
  __syncthreads();
  const int above = s_above;
  // aux[0, holes) (freed rows) and aux[NR - above, NR) (kept rows >= F) never overlap:
  // holes + above <= old_n <= NR.  The holes below F are aux[0, NN + above).
  for (int j = tid; j < above; j += kPlanThreads) {
    const int src = aux[NR - 1 - (above - 1 - j)];  // j-th highest
    final_src[aux[NN + j]] = src;
  }
  __syncthreads();

  // every final row: counters now, copies as descriptors
  for (int f = tid; f < F; f += kPlanThreads) {
    const int src = final_src[f];
    if (src == kUnset) {  // every row below F has a source; this only guards the indexing
      atomicOr(a.err, RB_EBIT_BATCH_ID);
      continue;
    }
    long long id;
    int s, nt, nb, prompt, computed;
    bool replace = false;
    int c = -1;
    if (src >= 0) {
      s = row_sched[src];
      id = b.d_req_id[src];
      nt = b.d_num_tokens[src];
      nb = b.d_num_blocks[src];
      prompt = b.d_num_prompt[src];
      computed = b.d_num_computed[src];
      c = sched_cached[s];
      replace = c >= 0 && u.d_cached_replace[c] != 0;
      if (src != f) {
        emit(desc, &s_n_desc, kSrcTok, false, static_cast<long long>(src) * M,
             static_cast<long long>(f) * M, nt);
        if (!replace)
          emit(desc, &s_n_desc, kSrcBlk, true, static_cast<long long>(src) * MB,
               static_cast<long long>(f) * MB, nb);
      }
    } else {
      const int k = -2 - src;
      id = u.d_new_req_id[k];
      s = hash_find(hkey, hval, H, id);
      const int t0 = u.d_new_token_start[k], b0 = u.d_new_block_start[k];
      nt = u.d_new_token_start[k + 1] - t0;
      nb = u.d_new_block_start[k + 1] - b0;
      prompt = u.d_new_num_prompt[k];
      computed = u.d_new_num_computed[k];
      emit(desc, &s_n_desc, kSrcNewTok, false, t0, static_cast<long long>(f) * M, nt);
      emit(desc, &s_n_desc, kSrcNewBlk, true, b0, static_cast<long long>(f) * MB, nb);
    }
    if (c >= 0) {
      const int t0 = u.d_cached_token_start[c], b0 = u.d_cached_block_start[c];
      const int m = u.d_cached_token_start[c + 1] - t0;
      const int nbl = u.d_cached_block_start[c + 1] - b0;
      emit(desc, &s_n_desc, kSrcCachedTok, false, t0, static_cast<long long>(f) * M + nt, m);
      nt += m;
      const int base = replace ? 0 : nb;
      emit(desc, &s_n_desc, kSrcCachedBlk, true, b0, static_cast<long long>(f) * MB + base, nbl);
      nb = base + nbl;
      computed = u.d_cached_num_computed[c];
    }
    b.d_req_id[f] = id;
    b.d_num_tokens[f] = nt;
    b.d_num_blocks[f] = nb;
    b.d_num_prompt[f] = prompt;
    b.d_num_computed[f] = computed;
    a.num_sched_out[f] = u.d_sched_num_tokens[s];
    if (a.row_of_sched != nullptr) a.row_of_sched[s] = f;
  }
  __syncthreads();  // rows past F were read above; clear them only now

  for (int r = F + tid; r < old_n; r += kPlanThreads) {
    b.d_req_id[r] = -1;
    b.d_num_tokens[r] = 0;
    b.d_num_blocks[r] = 0;
    b.d_num_prompt[r] = 0;
    b.d_num_computed[r] = 0;
  }
  for (int r = F + tid; r < NR; r += kPlanThreads) a.num_sched_out[r] = 0;
  if (tid == 0) *b.d_num_rows = F;

  // chunk offsets of the descriptors
  const int n_desc = s_n_desc;
  int running = 0;
  for (int base = 0; base < n_desc; base += kPlanThreads) {
    const int i = base + tid;
    const int ch = i < n_desc ? (desc[i].count + kChunk - 1) / kChunk : 0;
    int tile_total;
    const int rank = block_exclusive_scan(ch, warp_tmp, &tile_total);
    if (i < n_desc) chunk_start[i] = running + rank;
    running += tile_total;
  }
  if (tid == 0) {
    chunk_start[n_desc] = running;
    header[0] = 0;
    header[1] = n_desc;
    header[2] = running;
  }
}

struct CopyArgs {
  const int* header;
  const CopyDesc* desc;
  const int* chunk_start;
  const int32_t* src[6];
  int32_t* tok;
  int32_t* blk;
};

__global__ void __launch_bounds__(kCopyThreads) batch_copy_kernel(CopyArgs a) {
  if (a.header[0] != 0) return;
  const int n_desc = a.header[1], total = a.header[2];
  const int tid = threadIdx.x;
  for (int g = blockIdx.x; g < total; g += gridDim.x) {
    int lo = 0, hi = n_desc - 1;  // last descriptor whose first chunk is <= g
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.chunk_start[mid] <= g) lo = mid;
      else hi = mid - 1;
    }
    const CopyDesc d = a.desc[lo];
    const long long begin = static_cast<long long>(g - a.chunk_start[lo]) * kChunk;
    const int n = static_cast<int>(min(static_cast<long long>(kChunk), d.count - begin));
    const int32_t* base;
    switch (d.kinds & 255) {
      case kSrcTok: base = a.src[kSrcTok]; break;
      case kSrcBlk: base = a.src[kSrcBlk]; break;
      case kSrcNewTok: base = a.src[kSrcNewTok]; break;
      case kSrcNewBlk: base = a.src[kSrcNewBlk]; break;
      case kSrcCachedTok: base = a.src[kSrcCachedTok]; break;
      default: base = a.src[kSrcCachedBlk]; break;
    }
    const int32_t* src = base + d.src + begin;
    int32_t* dst = ((d.kinds >> 8) ? a.blk : a.tok) + d.dst + begin;
    const uintptr_t sa = reinterpret_cast<uintptr_t>(src), da = reinterpret_cast<uintptr_t>(dst);
    if (((sa ^ da) & 15u) == 0) {
      const int head = min(n, static_cast<int>(((16u - (sa & 15u)) & 15u) >> 2));
      if (tid < head) dst[tid] = src[tid];
      const int body = (n - head) >> 2;
      const int4* s4 = reinterpret_cast<const int4*>(src + head);
      int4* d4 = reinterpret_cast<int4*>(dst + head);
      for (int i = tid; i < body; i += kCopyThreads) d4[i] = __ldg(s4 + i);
      for (int i = head + 4 * body + tid; i < n; i += kCopyThreads) dst[i] = src[i];
    } else {
      for (int i = tid; i < n; i += kCopyThreads) dst[i] = __ldg(src + i);
    }
  }
}

size_t plan_smem_bytes(int max_rows, int S, int cap) {
  return static_cast<size_t>(cap) * (sizeof(long long) + sizeof(int)) +
         static_cast<size_t>(max_rows) * 3 * sizeof(int) + static_cast<size_t>(S) * 3 * sizeof(int);
}

}  // namespace
}  // namespace rb

extern "C" rb_status rb_batch_update_workspace_size(int32_t max_num_reqs, size_t* bytes) {
  using namespace rb;
  if (bytes == nullptr || max_num_reqs < 1) return RB_ERR_INVALID_ARG;
  if (max_num_reqs > kMaxRows) return RB_ERR_UNSUPPORTED;
  *bytes = ws_layout(max_num_reqs).total;
  return RB_OK;
}

extern "C" rb_status rb_batch_apply_update(const rb_batch* batch, const rb_batch_update* update,
                                           int32_t* d_num_scheduled, int32_t* d_row_of_sched,
                                           void* d_workspace, size_t workspace_bytes,
                                           int32_t* d_error_word, void* stream) {
  rb::CallRange range_("rb_batch_apply_update");
  using namespace rb;
  if (batch == nullptr || update == nullptr) return RB_ERR_INVALID_ARG;
  const rb_batch& b = *batch;
  const rb_batch_update& u = *update;
  if (b.max_num_reqs < 1 || b.max_model_len < 1 || b.max_blocks_per_req < 1 || b.reserved != 0)
    return RB_ERR_INVALID_ARG;
  if (b.max_num_reqs > kMaxRows) return RB_ERR_UNSUPPORTED;
  if (!b.d_req_id || !b.d_token_table || !b.d_num_tokens || !b.d_num_prompt ||
      !b.d_num_computed || !b.d_block_table || !b.d_num_blocks || !b.d_num_rows)
    return RB_ERR_INVALID_ARG;
  const int S = u.num_scheduled, NN = u.num_new, NC = u.num_cached;
  if (S < 0 || NN < 0 || NC < 0 || NN > S || NC > S || u.reserved != 0) return RB_ERR_INVALID_ARG;
  if (S > b.max_num_reqs) return RB_ERR_CAPACITY;
  if (S > 0 && (!u.d_sched_req_id || !u.d_sched_num_tokens)) return RB_ERR_INVALID_ARG;
  if (NN > 0 && (!u.d_new_req_id || !u.d_new_num_computed || !u.d_new_num_prompt ||
                 !u.d_new_token_start || !u.d_new_tokens || !u.d_new_block_start ||
                 !u.d_new_blocks))
    return RB_ERR_INVALID_ARG;
  if (NC > 0 && (!u.d_cached_req_id || !u.d_cached_num_computed || !u.d_cached_replace ||
                 !u.d_cached_token_start || !u.d_cached_tokens || !u.d_cached_block_start ||
                 !u.d_cached_blocks))
    return RB_ERR_INVALID_ARG;
  if (d_num_scheduled == nullptr || d_error_word == nullptr || d_workspace == nullptr ||
      !aligned16(d_workspace))
    return RB_ERR_INVALID_ARG;
  const WsLayoutB ws = ws_layout(b.max_num_reqs);
  if (workspace_bytes < ws.total) return RB_ERR_CAPACITY;

  int cap = 64;
  while (cap < 2 * S) cap <<= 1;
  const size_t smem = plan_smem_bytes(b.max_num_reqs, S, cap);
  // opt in once per device to the largest planner footprint (4096 rows, all scheduled)
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return RB_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(batch_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(plan_smem_bytes(kMaxRows, kMaxRows, 2 * kMaxRows))) !=
        cudaSuccess)
      return RB_ERR_CUDA;
    configured[dev] = true;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PlanArgs pa;
  pa.b = b;
  pa.u = u;
  pa.num_sched_out = d_num_scheduled;
  pa.row_of_sched = d_row_of_sched;
  pa.err = d_error_word;
  pa.ws = static_cast<unsigned char*>(d_workspace);
  pa.hash_cap = cap;
  batch_plan_kernel<<<1, kPlanThreads, smem, st>>>(pa);
  if (last_launch_status() != RB_OK) return RB_ERR_CUDA;
  note_launches(1);

  CopyArgs ca;
  ca.header = reinterpret_cast<const int*>(pa.ws + ws.header);
  ca.desc = reinterpret_cast<const CopyDesc*>(pa.ws + ws.desc);
  ca.chunk_start = reinterpret_cast<const int*>(pa.ws + ws.chunk_start);
  ca.src[kSrcTok] = b.d_token_table;
  ca.src[kSrcBlk] = b.d_block_table;
  ca.src[kSrcNewTok] = u.d_new_tokens;
  ca.src[kSrcNewBlk] = u.d_new_blocks;
  ca.src[kSrcCachedTok] = u.d_cached_tokens;
  ca.src[kSrcCachedBlk] = u.d_cached_blocks;
  ca.tok = b.d_token_table;
  ca.blk = b.d_block_table;
  // chunks per final row: at most two token copies and two page copies
  const long long per_row = 2LL * ((b.max_model_len + kChunk - 1) / kChunk) +
                            2LL * ((b.max_blocks_per_req + kChunk - 1) / kChunk);
  const long long bound = per_row * b.max_num_reqs;
  const int sms = max(1, device_sm_count());
  const int grid = static_cast<int>(bound < 2LL * sms ? bound : 2LL * sms);
  batch_copy_kernel<<<grid, kCopyThreads, 0, st>>>(ca);
  if (last_launch_status() != RB_OK) return RB_ERR_CUDA;
  note_launches(1);
  return RB_OK;
}
