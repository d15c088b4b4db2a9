// Paged decode without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// decode: inference engines that plan every byte of device memory up front and
// hand kernels no scratch, plugin hosts whose kernel interface has no
// workspace argument, and code running where calling cudaMalloc is not
// allowed. For them this entry point runs msa_sparse_attention_fwd itself
// (the same kernels, the same result bits) with its workspace placed in a
// fixed array that is part of the library's device image instead of a
// caller-provided buffer.
//
// The array is shared by every call on a device and keeps the contents the
// last call left; the forward needs no initialised workspace (the union pass
// writes every field the attention pass reads). Two calls whose work overlaps
// on the GPU (different streams, or host threads racing) use the same array
// and race; callers must order them.
#include <mutex>

#include "../../include/msa.h"
#include "internal.h"

namespace msa {
namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB per device, held until exit

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device. Looked up once
// per device (with that device current) and cached; nullptr on failure.
unsigned char* scratch_on_current_device() {
  static std::mutex mu;
  static unsigned char* addr[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned char*>(p);
  }
  return addr[dev];
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" size_t msa_sparse_decode_noalloc_scratch_limit(void) { return kNoAllocScratchBytes; }

extern "C" msa_status_t msa_sparse_decode_noalloc(
    const void* q, const void* k, const void* v, const int32_t* q2k_indices, int topk,
    const int32_t* cu_seqlens_q, const int32_t* page_table, int max_pages, int num_pages,
    const int32_t* seqused_k, int batch, int total_q, int num_qo_heads, int num_kv_heads,
    int head_dim, int max_seqlen_q, int causal, float softmax_scale, void* out, float* lse,
    cudaStream_t stream) {
  if (page_table == nullptr || seqused_k == nullptr) return MSA_INVALID_ARG;
  // Decided on the host, before any device call: the forward's workspace for
  // this call must fit the array. Sizes the forward rejects give no size; the
  // forward then returns its own status without touching the device.
  const size_t need = msa_sparse_attention_workspace_size(
      batch, total_q, num_qo_heads, num_kv_heads, head_dim, topk, max_seqlen_q, 1);
  if (need > kNoAllocScratchBytes) return MSA_WORKSPACE_TOO_SMALL;
  // The array is passed whenever the sizes are valid (need > 0), also for an
  // empty call (total_q == 0), which the forward accepts and returns MSA_OK for
  // without launching anything.
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (need > 0) {
    ws = scratch_on_current_device();
    if (ws == nullptr) return MSA_CUDA_ERROR;
    ws_bytes = kNoAllocScratchBytes;
  }
  return msa_sparse_attention_fwd(q, MSA_BF16, k, v, MSA_BF16, q2k_indices, topk, cu_seqlens_q,
                                  nullptr, page_table, max_pages, num_pages, seqused_k, batch,
                                  total_q, 0, num_qo_heads, num_kv_heads, head_dim, max_seqlen_q,
                                  causal, softmax_scale, out, lse, ws, ws_bytes, stream);
}
