// Whole-tensor E4M3 -> bf16 decode of flat K/V ("flashinfer.msa_ops.
// msa_sparse_attention", FP8 K/V route). Prefill-sized forwards run the
// attention kernel over a bf16 copy that this pass writes into the
// workspace: one read of the E4M3 bytes and one write of the bf16 values,
// HBM-bound, after which every K/V block the attention kernel reads (many
// times, from L2 and HBM) is already in the MMA's operand format. Decoding is
// exact (E4M3 -> f16 -> bf16 loses nothing; NaN stays NaN), so the result is
// the one the in-kernel conversion gives.
//
// Each thread moves 16 E4M3 codes (one 16-byte load) to 16 bf16 values (two
// 16-byte stores) per step, grid-striding over K then V.
#include "common.cuh"
#include "internal.h"

namespace msa {
namespace {

constexpr int kDecodeThreads = 256;
constexpr int kDecodeCtasPerSM = 8;
constexpr int kDecodeSMs = 152;

__global__ void __launch_bounds__(kDecodeThreads)
    kv_e4m3_to_bf16_kernel(const uint4* __restrict__ k8, const uint4* __restrict__ v8,
                           uint4* __restrict__ k16, uint4* __restrict__ v16, size_t n16) {
  const size_t stride = (size_t)gridDim.x * kDecodeThreads;
  for (size_t i = (size_t)blockIdx.x * kDecodeThreads + threadIdx.x; i < 2 * n16; i += stride) {
    const bool second = i >= n16;
    const size_t j = second ? i - n16 : i;
    const uint4 raw = __ldcs((second ? v8 : k8) + j);
    uint4 lo, hi;
    e4m3x4_to_bf16(raw.x, lo.x, lo.y);
    e4m3x4_to_bf16(raw.y, lo.z, lo.w);
    e4m3x4_to_bf16(raw.z, hi.x, hi.y);
    e4m3x4_to_bf16(raw.w, hi.z, hi.w);
    uint4* dst = (second ? v16 : k16) + 2 * j;
    dst[0] = lo;
    dst[1] = hi;
  }
}

}  // namespace

cudaError_t launch_kv_decode(const KvDecodeArgs& a, cudaStream_t s) {
  if (a.n16 == 0) return cudaSuccess;
  const size_t want = (2 * a.n16 + kDecodeThreads - 1) / kDecodeThreads;
  const unsigned grid =
      (unsigned)(want < (size_t)kDecodeSMs * kDecodeCtasPerSM ? want
                                                              : (size_t)kDecodeSMs * kDecodeCtasPerSM);
  kv_e4m3_to_bf16_kernel<<<grid, kDecodeThreads, 0, s>>>(
      static_cast<const uint4*>(a.k8), static_cast<const uint4*>(a.v8), static_cast<uint4*>(a.k16),
      static_cast<uint4*>(a.v16), a.n16);
  return cudaGetLastError();
}

}  // namespace msa
