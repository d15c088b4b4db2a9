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

template <int K>
cudaError_t launch_k(const TopkArgs& a, cudaStream_t s) {
  dim3 grid((a.total_q + kTopkThreads - 1) / kTopkThreads, a.num_score_heads);
  topk_kernel<K><<<grid, kTopkThreads, 0, s>>>(a.scores, a.num_score_heads, a.max_k_tiles,
                                                a.total_q, a.topk, a.num_kv_heads_out, a.q2k);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
  if (a.total_q == 0) return cudaSuccess;
  if (a.topk <= 8) return launch_k<8>(a, s);
  if (a.topk <= 16) return launch_k<16>(a, s);
  if (a.topk <= 32) return launch_k<32>(a, s);
  return launch_k<64>(a, s);
}

}  // namespace msa
