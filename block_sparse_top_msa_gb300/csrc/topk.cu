// Top-k block selection over proxy scores (consumer of
// "flashinfer.msa_ops.msa_proxy_score"; produces q2k_indices in the layout of
// "flashinfer.msa_ops.msa_sparse_attention": ascending, -1 padded).
//
// One thread per (query, score head). Scores are laid out (head, tile, query)
// with the query fastest, so a warp reading column t of 32 consecutive
// queries issues one coalesced 128-byte load. Each thread keeps its current
// best `topk` (score, id) pairs in registers, sorted by score; ids arrive in
// ascending order, so requiring a strictly larger score to displace an entry
// breaks ties toward the lower block id. -inf and NaN never enter.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace msa {
namespace {

constexpr int kTopkThreads = 128;

template <int K>
__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const float* __restrict__ scores, int num_score_heads, int T, int total_q,
                int topk, int hkv_out, int32_t* __restrict__ q2k) {
  const int q = blockIdx.x * blockDim.x + threadIdx.x;
  const int sh = blockIdx.y;
  if (q >= total_q) return;
  float v[K];
  int id[K];
#pragma unroll
  for (int i = 0; i < K; ++i) {
    v[i] = -INFINITY;
    id[i] = -1;
  }
  const float* col = scores + (size_t)sh * T * total_q + q;
  float thr = -INFINITY;  // score of the last live slot, v[topk - 1]
  float next = T > 0 ? __ldg(col) : -INFINITY;
  for (int t = 0; t < T; ++t) {
    const float s = next;
    if (t + 1 < T) next = __ldg(col + (size_t)(t + 1) * total_q);
    if (!(s > thr)) continue;  // also rejects NaN and -inf
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
  // Sort the chosen ids ascending; unused slots (-1) go last.
#pragma unroll
  for (int i = 0; i < K; ++i)
    if (id[i] < 0) id[i] = 0x7fffffff;
#pragma unroll
  for (int i = 0; i < K; ++i) {
#pragma unroll
    for (int j = 0; j + 1 < K - i; ++j) {
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
