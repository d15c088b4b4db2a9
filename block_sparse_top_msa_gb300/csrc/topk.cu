// Top-k block selection over proxy scores (consumer of
// "flashinfer.msa_ops.msa_proxy_score"; produces q2k_indices in the layout of
// "flashinfer.msa_ops.msa_sparse_attention": ascending, -1 padded).
//
// One thread per (query, score head), 128 queries per CTA. Scores are laid out
// (head, tile, query) with the query fastest, so the CTA streams its 128-query
// column band through shared memory in chunks of kChunk block rows: every
// thread issues several coalesced 16-byte loads per chunk (double-buffered
// with cp.async), then walks its own column from shared memory. Each thread
// keeps its current best `topk` (score, id) pairs in registers, sorted by
// score; ids arrive in ascending order, so requiring a strictly larger score to
// displace an entry breaks ties toward the lower block id. -inf and NaN never
// enter.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace msa {
namespace {

constexpr int kTopkThreads = 128;  // queries per CTA
constexpr int kChunk = 32;         // block rows per shared-memory chunk

MSA_DEV void cp_async16(void* dst, const void* src, bool valid) {
  const int bytes = valid ? 16 : 0;  // zero-fill outside the tensor
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(bytes)
               : "memory");
}
MSA_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
MSA_DEV void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
MSA_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

template <int K>
__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const float* __restrict__ scores, int num_score_heads, int T, int total_q,
                int topk, int hkv_out, int32_t* __restrict__ q2k) {
  __shared__ __align__(16) float band[2][kChunk][kTopkThreads];
  const int tid = threadIdx.x;
  const int q0 = blockIdx.x * kTopkThreads;
  const int q = q0 + tid;
  const int sh = blockIdx.y;
  const float* base = scores + (size_t)sh * T * total_q;
  // 16-byte copies need 16-byte aligned rows; otherwise scalar loads.
  const bool vec = (total_q % 4) == 0 && (reinterpret_cast<uintptr_t>(scores) & 15) == 0;

  auto load_chunk = [&](int c, int buf) {
    const int t0 = c * kChunk;
    if (vec) {
      // kChunk rows x 32 float4 per row, 8 copies per thread. Zero-filled
      // copies (past T or past total_q) are never read as candidates: rows
      // past T are not walked and columns past total_q belong to no thread
      // that writes a result.
#pragma unroll
      for (int j = 0; j < kChunk / 4; ++j) {
        const int idx = tid + j * kTopkThreads;
        const int r = idx / (kTopkThreads / 4), c4 = idx % (kTopkThreads / 4);
        const int t = t0 + r, qq = q0 + c4 * 4;
        const bool ok = t < T && qq < total_q;
        cp_async16(&band[buf][r][c4 * 4], ok ? base + (size_t)t * total_q + qq : base, ok);
      }
    } else {
      for (int r = 0; r < kChunk; ++r) {
        const int t = t0 + r;
        band[buf][r][tid] = (t < T && q < total_q) ? __ldg(base + (size_t)t * total_q + q)
                                                   : -INFINITY;
      }
    }
    cp_async_commit();
  };

  float v[K];
  int id[K];
#pragma unroll
  for (int i = 0; i < K; ++i) {
    v[i] = -INFINITY;
    id[i] = -1;
  }
  float thr = -INFINITY;  // score of the last live slot, v[topk - 1]
  const int nchunks = (T + kChunk - 1) / kChunk;
  load_chunk(0, 0);
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunks) {
      load_chunk(c + 1, buf ^ 1);
      cp_async_wait_one();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
    const int rows = min(kChunk, T - c * kChunk);
    for (int r = 0; r < rows; ++r) {
      const float s = band[buf][r][tid];
      if (s > thr) {  // rejects NaN and -inf
        const int t = c * kChunk + r;
#pragma unroll
        for (int i = K - 1; i >= 0; --i) {
          if (i < topk) {
            const bool above_prev = i > 0 && s > v[i > 0 ? i - 1 : 0];
            const bool above_cur = s > v[i];
            if (above_prev) {
              v[i] = v[i > 0 ? i - 1 : 0];
              id[i] = id[i > 0 ? i - 1 : 0];
            } else if (above_cur) {
              v[i] = s;
              id[i] = t;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < K; ++i)
          if (i == topk - 1) thr = v[i];
      }
    }
    __syncthreads();  // buffer `buf` is refilled by the next iteration's prefetch
  }
  if (q >= total_q) return;
  // Sort the chosen ids ascending; unused slots (-1) go last.
#pragma unroll
  for (int i = 0; i < K; ++i)
    if (id[i] < 0) id[i] = 0x7fffffff;
  // Odd-even transposition sort (K rounds of fixed compare-exchanges).
#pragma unroll
  for (int p = 0; p < K; ++p) {
#pragma unroll
    for (int j = p & 1; j + 1 < K; j += 2) {
      const int x = id[j], y = id[j + 1];
      id[j] = min(x, y);
      id[j + 1] = max(x, y);
    }
  }
  const int h0 = num_score_heads == 1 ? 0 : sh;
  const int h1 = num_score_heads == 1 ? hkv_out : sh + 1;
  for (int h = h0; h < h1; ++h) {
    int32_t* dst = q2k + ((size_t)h * total_q + q) * topk;
#pragma unroll
    for (int i = 0; i < K; ++i)
      if (i < topk) dst[i] = id[i] == 0x7fffffff ? -1 : id[i];
  }
}

// Buffered selection for topk <= 16. Each thread still owns one query, but a
// row only costs a compare and, for a score above the current threshold, an
// append to the thread's candidate buffer in shared memory. When some lane's
// buffer holds kBuf entries, the warp merges every lane's buffer into its
// sorted list with fixed networks (bitonic sort of the buffer, elementwise
// best against the reversed list, bitonic clean-up), and the threshold becomes
// the list's last score. Order: larger score first, equal scores by lower id.
constexpr int kBuf = 16;
constexpr int kChunkB = 16;  // block rows per shared-memory chunk
constexpr int kStagesB = 4;  // chunks in flight (cp.async ring)
constexpr size_t kBufferedSmem =
    sizeof(float) * kStagesB * kChunkB * kTopkThreads + (sizeof(float) + sizeof(int)) * kBuf * kTopkThreads;

struct Cand {
  float s;
  int id;
};
// a ranks before b
MSA_DEV bool better(const Cand& a, const Cand& b) { return a.s > b.s || (a.s == b.s && a.id < b.id); }
MSA_DEV void cex(Cand& a, Cand& b) {  // a <- the better one
  const bool sw = better(b, a);
  const Cand x = a;
  a = sw ? b : a;
  b = sw ? x : b;
}

template <int K>
MSA_DEV void merge_buffer(Cand (&lst)[K], const float* cv, const int* ci, int cnt, int tid) {
  Cand b[kBuf];
#pragma unroll
  for (int j = 0; j < kBuf; ++j) {
    b[j].s = j < cnt ? cv[j * kTopkThreads + tid] : -INFINITY;
    b[j].id = j < cnt ? ci[j * kTopkThreads + tid] : 0x7fffffff;
  }
  // Bitonic sort of the buffer, best first.
#pragma unroll
  for (int k = 2; k <= kBuf; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < kBuf; ++i) {
        const int l = i ^ j;
        if (l > i) {
          if ((i & k) == 0) cex(b[i], b[l]);
          else cex(b[l], b[i]);
        }
      }
    }
  }
  // The best K of both sorted runs: elementwise best of lst[i] and b[K-1-i]
  // (a bitonic sequence), then a bitonic clean-up, best first.
#pragma unroll
  for (int i = 0; i < K; ++i)
    if (better(b[K - 1 - i], lst[i])) lst[i] = b[K - 1 - i];
#pragma unroll
  for (int j = K >> 1; j > 0; j >>= 1) {
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const int l = i ^ j;
      if (l > i) cex(lst[i], lst[l]);
    }
  }
}

template <int K>
__global__ void __launch_bounds__(kTopkThreads)
    topk_buffered_kernel(const float* __restrict__ scores, int num_score_heads, int T, int total_q,
                         int topk, int hkv_out, int32_t* __restrict__ q2k) {
  static_assert(K <= kBuf, "the merge takes the best K of K + kBuf entries");
  constexpr int kChunk = kChunkB;
  extern __shared__ __align__(16) float dyn[];
  float (*band)[kChunk][kTopkThreads] = reinterpret_cast<float (*)[kChunk][kTopkThreads]>(dyn);
  float (*cv)[kTopkThreads] =
      reinterpret_cast<float (*)[kTopkThreads]>(dyn + kStagesB * kChunk * kTopkThreads);
  int (*ci)[kTopkThreads] = reinterpret_cast<int (*)[kTopkThreads]>(cv + kBuf);
  const int tid = threadIdx.x;
  const int q0 = blockIdx.x * kTopkThreads;
  const int q = q0 + tid;
  const int sh = blockIdx.y;
  const float* base = scores + (size_t)sh * T * total_q;
  const bool vec = (total_q % 4) == 0 && (reinterpret_cast<uintptr_t>(scores) & 15) == 0;

  auto load_chunk = [&](int c, int buf) {
    const int t0 = c * kChunk;
    if (vec) {
#pragma unroll
      for (int j = 0; j < kChunk / 4; ++j) {
        const int idx = tid + j * kTopkThreads;
        const int r = idx / (kTopkThreads / 4), c4 = idx % (kTopkThreads / 4);
        const int t = t0 + r, qq = q0 + c4 * 4;
        const bool ok = t < T && qq < total_q;
        cp_async16(&band[buf][r][c4 * 4], ok ? base + (size_t)t * total_q + qq : base, ok);
      }
    } else {
      for (int r = 0; r < kChunk; ++r) {
        const int t = t0 + r;
        band[buf][r][tid] = (t < T && q < total_q) ? __ldg(base + (size_t)t * total_q + q)
                                                   : -INFINITY;
      }
    }
    cp_async_commit();
  };

  Cand lst[K];
#pragma unroll
  for (int i = 0; i < K; ++i) lst[i] = Cand{-INFINITY, 0x7fffffff};
  // A score must exceed thr to be a candidate: the list's K-th score (-inf
  // until K live scores have been merged). The list keeps the best K >= topk,
  // so this bound is exact for topk == K and safe (looser) below it.
  float thr = -INFINITY;
  int cnt = 0;
  const int nchunks = (T + kChunk - 1) / kChunk;
  // One commit group per chunk (empty past the end), so that after issuing
  // chunk c + kStagesB - 1, at most kStagesB - 1 groups newer than c pend.
  for (int c = 0; c < kStagesB - 1; ++c) {
    if (c < nchunks) load_chunk(c, c);
    else cp_async_commit();
  }
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c % kStagesB;
    const int nx = c + kStagesB - 1;
    if (nx < nchunks) load_chunk(nx, nx % kStagesB);
    else cp_async_commit();
    asm volatile("cp.async.wait_group %0;" ::"n"(kStagesB - 1) : "memory");
    __syncthreads();
    const int rows = min(kChunk, T - c * kChunk);
    for (int r0 = 0; r0 < rows; r0 += 4) {
#pragma unroll
      for (int r = r0; r < r0 + 4; ++r) {
        if (r < rows) {
          const float s = band[buf][r][tid];
          if (s > thr) {  // rejects NaN and -inf
            cv[cnt][tid] = s;
            ci[cnt][tid] = c * kChunk + r;
            ++cnt;
          }
        }
      }
      // A lane enters a group of 4 rows with at most kBuf - 4 candidates, so
      // the buffer (kBuf slots) never overflows.
      if (__any_sync(0xffffffffu, cnt > kBuf - 4)) {
        merge_buffer<K>(lst, &cv[0][0], &ci[0][0], cnt, tid);
        cnt = 0;
        thr = lst[K - 1].s;
      }
    }
    __syncthreads();  // slot `buf` is refilled by a later iteration's prefetch
  }
  if (__any_sync(0xffffffffu, cnt > 0)) merge_buffer<K>(lst, &cv[0][0], &ci[0][0], cnt, tid);
  if (q >= total_q) return;
  int id[K];
#pragma unroll
  for (int i = 0; i < K; ++i) id[i] = i < topk ? lst[i].id : 0x7fffffff;
  // Ascending ids, unused slots (-1) last.
#pragma unroll
  for (int p = 0; p < K; ++p) {
#pragma unroll
    for (int j = p & 1; j + 1 < K; j += 2) {
      const int x = id[j], y = id[j + 1];
      id[j] = min(x, y);
      id[j + 1] = max(x, y);
    }
  }
  const int h0 = num_score_heads == 1 ? 0 : sh;
  const int h1 = num_score_heads == 1 ? hkv_out : sh + 1;
  for (int h = h0; h < h1; ++h) {
    int32_t* dst = q2k + ((size_t)h * total_q + q) * topk;
#pragma unroll
    for (int i = 0; i < K; ++i)
      if (i < topk) dst[i] = id[i] == 0x7fffffff ? -1 : id[i];
  }
}

template <int K>
cudaError_t launch_k(const TopkArgs& a, cudaStream_t s) {
  dim3 grid((a.total_q + kTopkThreads - 1) / kTopkThreads, a.num_score_heads);
  topk_kernel<K><<<grid, kTopkThreads, 0, s>>>(a.scores, a.num_score_heads, a.max_k_tiles,
                                                a.total_q, a.topk, a.num_kv_heads_out, a.q2k);
  return cudaGetLastError();
}

}  // namespace

template <int K>
cudaError_t launch_buffered(const TopkArgs& a, cudaStream_t s) {
  dim3 grid((a.total_q + kTopkThreads - 1) / kTopkThreads, a.num_score_heads);
  cudaError_t e = set_smem_limit((const void*)topk_buffered_kernel<K>, (int)kBufferedSmem);
  if (e != cudaSuccess) return e;
  topk_buffered_kernel<K><<<grid, kTopkThreads, kBufferedSmem, s>>>(a.scores, a.num_score_heads, a.max_k_tiles,
                                                         a.total_q, a.topk, a.num_kv_heads_out, a.q2k);
  return cudaGetLastError();
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
  if (a.total_q == 0) return cudaSuccess;
  if (a.topk <= 8) return launch_buffered<8>(a, s);
  if (a.topk <= 16) return launch_buffered<16>(a, s);
  if (a.topk <= 32) return launch_k<32>(a, s);
  return launch_k<64>(a, s);
}

}  // namespace msa
