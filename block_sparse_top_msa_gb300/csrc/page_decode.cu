// Page-pool decode for prefill-sized paged calls with E4M3 or packed NVFP4
// K/V ("flashinfer.msa_ops.msa_sparse_attention": paged K/V, fp8 and the
// packed-NVFP4 paged route). Every page a request can read is decoded once
// into a bf16 page pool in the workspace, at pool page b * max_pages + t for
// request b's block t, and the page table is renumbered to match (-1 where
// the request has no block t or its page is unmapped). The bf16 attention
// kernel then streams bf16 tiles, which on tensor-bound calls beats
// converting every block visit inside the attention kernel.
//
// One CTA per (request, block), a 1-D grid of batch * max_pages CTAs: K then
// V of every KV head, 16 elements (16 bytes of E4M3, or 8 bytes of E2M1 pairs
// and their block scale) per step. NVFP4 values are exact in bf16 (see fp4x16_to_bf16); the global
// scales are applied by the attention kernel as on the in-kernel route.
#include "common.cuh"
#include "internal.h"

namespace msa {
namespace {

constexpr int kPageThreads = 256;

__global__ void __launch_bounds__(kPageThreads) pages_to_bf16_kernel(const PageDecodeArgs a) {
  const size_t slot = blockIdx.x;  // request b's block t: slot b * max_pages + t
  const int b = (int)(slot / (size_t)a.max_pages);
  const int t = (int)(slot - (size_t)b * a.max_pages);
  int nblk = (a.seqused_k[b] + kBlk - 1) / kBlk;
  if (nblk > a.max_pages) nblk = a.max_pages;
  const int p = t < nblk ? a.page_table[slot] : -1;
  const bool valid = p >= 0 && p < a.num_pages;
  if (threadIdx.x == 0) a.pt_out[slot] = valid ? (int32_t)slot : -1;
  if (!valid) return;
  const int units = 2 * a.hkv * 1024;  // (side, head, token, 16-element chunk)
  for (int i = threadIdx.x; i < units; i += kPageThreads) {
    const int side = i / (a.hkv * 1024);
    const int rem = i - side * a.hkv * 1024;
    const int h = rem >> 10, r = (rem >> 3) & 127, c = rem & 7;
    uint32_t w[8];
    if (a.mode == 1) {
      const uint8_t* src = (side == 0 ? a.k8 : a.v8) + ((size_t)p * a.hkv + h) * (kBlk * kHeadDim);
      const uint4 raw = *reinterpret_cast<const uint4*>(src + r * kHeadDim + c * 16);
      e4m3x4_to_bf16(raw.x, w[0], w[1]);
      e4m3x4_to_bf16(raw.y, w[2], w[3]);
      e4m3x4_to_bf16(raw.z, w[4], w[5]);
      e4m3x4_to_bf16(raw.w, w[6], w[7]);
    } else {
      const size_t page = (size_t)p * a.fp4_page_stride;
      const uint8_t* codes = (side == 0 ? a.fp4_k : a.fp4_v) + page + (size_t)h * kFp4Data;
      const uint8_t* scales =
          (side == 0 ? a.fp4_k_scale : a.fp4_v_scale) + page + (size_t)h * kFp4Scales;
      fp4x16_to_bf16(*reinterpret_cast<const uint2*>(codes + r * 64 + c * 8),
                     scales[fp4_scale_offset(side == 1, r, c)], w);
    }
    uint16_t* dst = (side == 0 ? a.k16 : a.v16) + ((slot * a.hkv + h) * kBlk + r) * kHeadDim + c * 16;
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

}  // namespace

cudaError_t launch_page_decode(const PageDecodeArgs& a, cudaStream_t s) {
  if (a.mode == 0 || a.batch <= 0 || a.max_pages <= 0) return cudaSuccess;
  const unsigned long long slots = (unsigned long long)a.batch * (unsigned long long)a.max_pages;
  if (slots > 0x7fffffffull) return cudaErrorInvalidConfiguration;  // one CTA per slot
  pages_to_bf16_kernel<<<(unsigned)slots, kPageThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace msa
