// Paged decode without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// decode: inference engines that plan every byte of device memory up front and
// hand kernels no scratch, plugin hosts whose kernel interface has no
// workspace argument, and code running where calling cudaMalloc is not
// allowed. For them this entry point runs the same split-KV decode kernel as
// msa_sparse_attention_fwd, but keeps its scratch (per-split partial results
// and one completion ticket per (request, KV head)) in a fixed array that is
// part of the library's device image instead of a caller-provided workspace.
//
// The array is shared by every call on a device and keeps the contents the
// last call left. The tickets are cleared on the stream before each launch;
// the partials are always written before they are read. Two calls whose work
// overlaps on the GPU (different streams, or host threads racing) use the same
// array and race; callers must order them.
#include <mutex>

#include "../../include/msa.h"
#include "internal.h"
#include "tmap.h"

namespace msa {
namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB per device, held until exit

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

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

bool rows_map(CUtensorMap* m, const void* base, int H, long long T, uint32_t box_h,
              uint32_t box_t) {
  const uint64_t dims[3] = {128, (uint64_t)H, (uint64_t)(T > 0 ? T : 1)};
  const uint64_t strides[2] = {256ull, 256ull * H};
  const uint32_t box[3] = {64u, box_h, box_t};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box);
}

bool pages_map(CUtensorMap* m, const void* base, int H, int pages) {
  const uint64_t dims[4] = {128, 128, (uint64_t)H, (uint64_t)pages};
  const uint64_t strides[3] = {256ull, 256ull * 128, 256ull * 128 * H};
  const uint32_t box[4] = {64u, 128u, 1u, 1u};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box);
}

bool aligned_to(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
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
  if (q == nullptr || k == nullptr || v == nullptr || q2k_indices == nullptr ||
      cu_seqlens_q == nullptr || page_table == nullptr || seqused_k == nullptr || out == nullptr)
    return MSA_INVALID_ARG;
  if (batch < 1 || total_q < 0 || num_qo_heads < 1 || num_kv_heads < 1 || max_pages < 1 ||
      num_pages < 1 || num_qo_heads % num_kv_heads != 0 || max_seqlen_q < 1)
    return MSA_INVALID_ARG;
  if (!aligned_to(q, 16) || !aligned_to(k, 16) || !aligned_to(v, 16) || !aligned_to(out, 16) ||
      !aligned_to(q2k_indices, 4) || !aligned_to(cu_seqlens_q, 4) || !aligned_to(page_table, 4) ||
      !aligned_to(seqused_k, 4) || (lse != nullptr && !aligned_to(lse, 4)))
    return MSA_INVALID_ARG;
  const int G = num_qo_heads / num_kv_heads;
  if (head_dim != 128 || topk < 1 || topk > 64 || max_seqlen_q > 4 || G > 16)
    return MSA_UNSUPPORTED;
  if (total_q == 0) return MSA_OK;

  // Scratch layout, the same as the workspace the forward's decode route uses.
  const int rows = G * max_seqlen_q;
  const int R = rows <= 16 ? 16 : (rows <= 32 ? 32 : 64);
  const int pps = decode_pages_per_split(rows);
  const int splits = (max_seqlen_q * topk + pps - 1) / pps;
  const size_t parts = (size_t)batch * num_kv_heads * splits;
  const size_t off_ml = round256(parts * R * 128 * sizeof(float));
  const size_t off_tickets = off_ml + round256(parts * R * 2 * sizeof(float));
  const size_t need = off_tickets + round256((size_t)batch * num_kv_heads * sizeof(int));
  if (need > kNoAllocScratchBytes) return MSA_WORKSPACE_TOO_SMALL;

  unsigned char* scratch = scratch_on_current_device();
  unsigned* fault = fault_word();
  if (scratch == nullptr || fault == nullptr) return MSA_CUDA_ERROR;

  DecodeArgs a{};
  a.fault = fault;
  if (!rows_map(&a.tmap_q, q, num_qo_heads, total_q, (uint32_t)G, (uint32_t)max_seqlen_q) ||
      !pages_map(&a.tmap_k, k, num_kv_heads, num_pages) ||
      !pages_map(&a.tmap_v, v, num_kv_heads, num_pages))
    return MSA_CUDA_ERROR;
  const float scale = softmax_scale > 0.f ? softmax_scale : 0.08838834764831845f;  // 128^-0.5
  a.q2k = q2k_indices;
  a.topk = topk;
  a.cu_q = cu_seqlens_q;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.seqused_k = seqused_k;
  a.batch = batch;
  a.total_q = total_q;
  a.num_qo_heads = num_qo_heads;
  a.num_kv_heads = num_kv_heads;
  a.sq_max = max_seqlen_q;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  a.lse = lse;
  a.pages_per_split = pps;
  a.splits = splits;
  a.part_o = reinterpret_cast<float*>(scratch);
  a.part_ml = reinterpret_cast<float*>(scratch + off_ml);
  a.tickets = reinterpret_cast<int*>(scratch + off_tickets);
  // Tickets must start at zero; the array still holds the previous call's values.
  if (cudaMemsetAsync(a.tickets, 0, (size_t)batch * num_kv_heads * sizeof(int), stream) !=
      cudaSuccess)
    return MSA_CUDA_ERROR;
  return launch_decode(a, stream) == cudaSuccess ? MSA_OK : MSA_CUDA_ERROR;
}
