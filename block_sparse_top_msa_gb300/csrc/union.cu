// Query-tile union metadata ("flashinfer.msa_ops.msa_sparse_attention":
// query tokens are processed in tiles, each running one online softmax over
// the union of the blocks its tokens selected; the union metadata is built
// from q2k_indices).
//
// One CTA per (query tile, KV head). The tile's W*topk ids are filtered to
// the usable ones, sorted (bitonic, in shared memory) and deduplicated into
// the ascending union list; each token's membership bitmask over union
// positions is then set by binary search. Output format: see msa_build_union
// in include/msa.h.
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "tile_map.cuh"

namespace msa {
namespace {

constexpr int kUnionThreads = 256;

__global__ void __launch_bounds__(kUnionThreads)
    build_union_kernel(UnionArgs a) {
  extern __shared__ int smem_i[];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int tile = blockIdx.x, h = blockIdx.y;
  const int n = a.tile_tokens * a.topk;
  int P = 1;
  while (P < n) P <<= 1;
  int* scratch = smem_i;                       // nt + 2
  int* keys = scratch + nt + 2;                // P
  int* ulist = keys + P;                       // cap
  uint32_t* mem = reinterpret_cast<uint32_t*>(ulist + a.cap);  // W * words
  uint32_t* bmem = mem + a.tile_tokens * a.words;              // cap (block_members only)
  __shared__ int s_ulen;

  grid_dependents_launch();
  if (a.item_counter != nullptr && tile == 0 && h == 0 && tid == 0) *a.item_counter = 0;
  int b = 0, t0 = 0;
  const bool live = locate_tile(a.cu_q, a.batch, a.tile_tokens, tile, scratch, &b, &t0);
  const size_t base = (size_t)h * a.max_tiles + tile;
  if (!live) {
    if (tid == 0) a.union_len[base] = 0;
    for (int j = tid; j < a.cap; j += nt) a.union_blocks[base * a.cap + j] = -1;
    for (int j = tid; j < a.tile_tokens * a.words; j += nt)
      a.member[base * a.tile_tokens * a.words + j] = 0u;
    if (a.block_members != nullptr)
      for (int j = tid; j < a.cap; j += nt) a.block_members[base * a.cap + j] = 0u;
    if (a.tile_info != nullptr && h == 0 && tid < 2) a.tile_info[2 * tile + tid] = -1;
    return;
  }
  const int end = a.cu_q[b + 1];
  const int lq = end - a.cu_q[b];
  const int lk = a.seqused_k ? a.seqused_k[b] : a.cu_k[b + 1] - a.cu_k[b];
  int nblk = (lk + kBlk - 1) / kBlk;
  if (a.seqused_k && nblk > a.max_pages) nblk = a.max_pages;
  const int nw = min(a.tile_tokens, end - t0);
  if (a.block_members != nullptr)
    for (int j = tid; j < a.cap; j += nt) bmem[j] = 0u;

  // Usable ids of the tile's rows; everything else sorts to the end.
  for (int i = tid; i < P; i += nt) {
    int key = INT_MAX;
    if (i < n) {
      const int w = i / a.topk;
      if (w < nw) {
        const int id = a.q2k[((size_t)h * a.total_q + t0 + w) * a.topk + (i % a.topk)];
        const long long pos = (long long)lk - lq + (t0 + w - a.cu_q[b]);
        if (id >= 0 && id < nblk && (!a.causal || (long long)id * kBlk <= pos)) key = id;
      }
    }
    keys[i] = key;
  }
  for (int j = tid; j < a.tile_tokens * a.words; j += nt) mem[j] = 0u;
  __syncthreads();
  // Bitonic sort, ascending.
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P; i += nt) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const int x = keys[i], y = keys[ixj];
          const bool up = (i & k) == 0;
          if ((x > y) == up) {
            keys[i] = y;
            keys[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  // Deduplicate: position of each first occurrence = number of distinct
  // smaller keys. Done by a block scan over chunks of nt elements.
  int carry = 0;
  for (int c0 = 0; c0 < P; c0 += nt) {
    const int i = c0 + tid;
    int flag = 0;
    int key = INT_MAX;
    if (i < P) {
      key = keys[i];
      flag = key != INT_MAX && (i == 0 || keys[i - 1] != key);
    }
    scratch[tid] = flag;
    __syncthreads();
    for (int off = 1; off < nt; off <<= 1) {
      const int add = tid >= off ? scratch[tid - off] : 0;
      __syncthreads();
      scratch[tid] += add;
      __syncthreads();
    }
    if (flag) ulist[carry + scratch[tid] - 1] = key;
    const int tot = scratch[nt - 1];
    __syncthreads();
    carry += tot;
  }
  if (tid == 0) s_ulen = carry;
  __syncthreads();
  const int ulen = s_ulen;

  // Membership bits.
  for (int i = tid; i < nw * a.topk; i += nt) {
    const int w = i / a.topk;
    const int id = a.q2k[((size_t)h * a.total_q + t0 + w) * a.topk + (i % a.topk)];
    const long long pos = (long long)lk - lq + (t0 + w - a.cu_q[b]);
    if (id < 0 || id >= nblk || (a.causal && (long long)id * kBlk > pos)) continue;
    int lo = 0, hi = ulen - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (ulist[mid] < id) lo = mid + 1; else hi = mid;
    }
    atomicOr(&mem[w * a.words + (lo >> 5)], 1u << (lo & 31));
    if (a.block_members != nullptr) atomicOr(&bmem[lo], 1u << w);
  }
  __syncthreads();
  if (tid == 0) a.union_len[base] = ulen;
  for (int j = tid; j < a.cap; j += nt) a.union_blocks[base * a.cap + j] = j < ulen ? ulist[j] : -1;
  for (int j = tid; j < a.tile_tokens * a.words; j += nt)
    a.member[base * a.tile_tokens * a.words + j] = mem[j];
  if (a.block_members != nullptr)
    for (int j = tid; j < a.cap; j += nt) a.block_members[base * a.cap + j] = bmem[j];
  if (a.tile_info != nullptr && h == 0 && tid == 0) {
    a.tile_info[2 * tile] = t0;
    a.tile_info[2 * tile + 1] = b;
  }
}

// Fast path for W * topk <= 1024: one key per thread (blockDim.x = P, a power
// of two >= 32), bitonic sort in registers with warp shuffles for strides
// below 32 and shared memory for the larger ones, ballot-based compaction.
__global__ void __launch_bounds__(1024) build_union_small_kernel(UnionArgs a) {
  extern __shared__ int smem_i[];
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, wid = tid >> 5;
  const int tile = blockIdx.x, h = blockIdx.y;
  int* scratch = smem_i;             // nt + 2 (tile lookup), then nt (sort exchange)
  int* ulist = scratch + nt + 2;     // cap
  uint32_t* mem = reinterpret_cast<uint32_t*>(ulist + a.cap);  // W * words
  uint32_t* bmem = mem + a.tile_tokens * a.words;              // cap (block_members only)
  __shared__ int s_warp[32];
  __shared__ int s_ulen;

  grid_dependents_launch();
  if (a.item_counter != nullptr && tile == 0 && h == 0 && tid == 0) *a.item_counter = 0;
  int b = 0, t0 = 0;
  const bool live = locate_tile(a.cu_q, a.batch, a.tile_tokens, tile, scratch, &b, &t0);
  const size_t base = (size_t)h * a.max_tiles + tile;
  if (!live) {
    if (tid == 0) a.union_len[base] = 0;
    for (int j = tid; j < a.cap; j += nt) a.union_blocks[base * a.cap + j] = -1;
    for (int j = tid; j < a.tile_tokens * a.words; j += nt)
      a.member[base * a.tile_tokens * a.words + j] = 0u;
    if (a.block_members != nullptr)
      for (int j = tid; j < a.cap; j += nt) a.block_members[base * a.cap + j] = 0u;
    if (a.tile_info != nullptr && h == 0 && tid < 2) a.tile_info[2 * tile + tid] = -1;
    return;
  }
  const int end = a.cu_q[b + 1];
  const int lq = end - a.cu_q[b];
  const int lk = a.seqused_k ? a.seqused_k[b] : a.cu_k[b + 1] - a.cu_k[b];
  int nblk = (lk + kBlk - 1) / kBlk;
  if (a.seqused_k && nblk > a.max_pages) nblk = a.max_pages;
  const int nw = min(a.tile_tokens, end - t0);
  const int n = a.tile_tokens * a.topk;
  if (a.block_members != nullptr)
    for (int j = tid; j < a.cap; j += nt) bmem[j] = 0u;

  // This thread's id (usable ids only; the rest sort to the end).
  int key = INT_MAX;
  int my_id = -1, my_w = 0;
  if (tid < n) {
    my_w = tid / a.topk;
    if (my_w < nw) {
      const int id = a.q2k[((size_t)h * a.total_q + t0 + my_w) * a.topk + (tid % a.topk)];
      const long long pos = (long long)lk - lq + (t0 + my_w - a.cu_q[b]);
      if (id >= 0 && id < nblk && (!a.causal || (long long)id * kBlk <= pos)) {
        key = id;
        my_id = id;
      }
    }
  }
  for (int j = tid; j < a.tile_tokens * a.words; j += nt) mem[j] = 0u;
  int* xchg = scratch;  // reused: the tile lookup is done
  __syncthreads();
  for (int k = 2; k <= nt; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      int other;
      if (j >= 32) {
        xchg[tid] = key;
        __syncthreads();
        other = xchg[tid ^ j];
        __syncthreads();
      } else {
        other = __shfl_xor_sync(0xffffffffu, key, j);
      }
      const bool up = (tid & k) == 0, lower = (tid & j) == 0;
      key = (lower == up) ? min(key, other) : max(key, other);
    }
  }
  // First occurrence of each distinct usable id.
  xchg[tid] = key;
  __syncthreads();
  const int prev = tid > 0 ? xchg[tid - 1] : INT_MIN;
  const bool flag = key != INT_MAX && key != prev;
  const unsigned ball = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) s_warp[wid] = __popc(ball);
  __syncthreads();
  if (wid == 0) {
    const int nwarps = nt >> 5;
    int v = lane < nwarps ? s_warp[lane] : 0;
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += u;
    }
    if (lane < nwarps) s_warp[lane] = v;  // inclusive
    if (lane == 31) s_ulen = v;
  }
  __syncthreads();
  const int before = (wid > 0 ? s_warp[wid - 1] : 0) + __popc(ball & ((1u << lane) - 1u));
  if (flag) ulist[before] = key;
  const int ulen = s_ulen;
  __syncthreads();
  // Membership bits: binary search of this thread's original id.
  if (my_id >= 0) {
    int lo = 0, hi = ulen - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (ulist[mid] < my_id) lo = mid + 1; else hi = mid;
    }
    atomicOr(&mem[my_w * a.words + (lo >> 5)], 1u << (lo & 31));
    if (a.block_members != nullptr) atomicOr(&bmem[lo], 1u << my_w);
  }
  __syncthreads();
  if (tid == 0) a.union_len[base] = ulen;
  for (int j = tid; j < a.cap; j += nt) a.union_blocks[base * a.cap + j] = j < ulen ? ulist[j] : -1;
  for (int j = tid; j < a.tile_tokens * a.words; j += nt)
    a.member[base * a.tile_tokens * a.words + j] = mem[j];
  if (a.block_members != nullptr)
    for (int j = tid; j < a.cap; j += nt) a.block_members[base * a.cap + j] = bmem[j];
  if (a.tile_info != nullptr && h == 0 && tid == 0) {
    a.tile_info[2 * tile] = t0;
    a.tile_info[2 * tile + 1] = b;
  }
}

__global__ void __launch_bounds__(32) reset_counter_kernel(int32_t* counter) {
  grid_dependents_launch();
  if (threadIdx.x == 0) *counter = 0;
  // Completes only after the grids it depends on (if launched as a
  // dependent), so its completion implies theirs.
  grid_dependency_wait();
}

}  // namespace

cudaError_t launch_reset_counter(int32_t* counter, cudaStream_t s) {
  reset_counter_kernel<<<1, 32, 0, s>>>(counter);
  return cudaGetLastError();
}

cudaError_t launch_build_union(const UnionArgs& a, cudaStream_t s) {
  if (a.block_members != nullptr && a.tile_tokens > 32) return cudaErrorInvalidValue;
  const int n = a.tile_tokens * a.topk;
  int P = 1;
  while (P < n) P <<= 1;
  if (P <= 1024) {
    const int nt = P < 32 ? 32 : P;
    const size_t smem = sizeof(int) * ((size_t)nt + 2 + a.cap + (size_t)a.tile_tokens * a.words +
                                       (a.block_members != nullptr ? (size_t)a.cap : 0));
    cudaError_t e = set_smem_limit((const void*)build_union_small_kernel, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.max_tiles, a.num_kv_heads);
    build_union_small_kernel<<<grid, nt, smem, s>>>(a);
    return cudaGetLastError();
  }
  const size_t smem =
      sizeof(int) * ((size_t)kUnionThreads + 2 + P + a.cap + (size_t)a.tile_tokens * a.words +
                     (a.block_members != nullptr ? (size_t)a.cap : 0));
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = set_smem_limit((const void*)build_union_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_tiles, a.num_kv_heads);
  build_union_kernel<<<grid, kUnionThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace msa
