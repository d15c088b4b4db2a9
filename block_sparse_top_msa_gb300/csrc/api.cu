// C ABI of libmsa: host-side validation, workspace layout, tensor-map
// encoding and kernel launches. No allocation, no host synchronisation
// (except msa_read_device_fault, which exists to synchronise).
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <cmath>
#include <mutex>
#include <new>
#include <tuple>
#include <vector>

#include "../../include/msa.h"
#include "internal.h"
#include "tmap.h"

namespace msa {

__device__ unsigned g_msa_fault_word;

unsigned* fault_word() {
  static std::mutex mu;
  static unsigned* addr[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_msa_fault_word) == cudaSuccess) addr[dev] = static_cast<unsigned*>(p);
  }
  return addr[dev];
}

namespace {

constexpr int kMaxTopk = 64;
// Packed-NVFP4 calls with at most this many query tokens per request (and
// G <= 16) take the decode kernel when the workspace holds its lists.
constexpr int kFp4DecodeMaxSeqQ = 16;
bool fp4_decode_route(int num_qo_heads, int num_kv_heads, int max_seqlen_q) {
  return num_qo_heads / num_kv_heads <= 16 && max_seqlen_q <= kFp4DecodeMaxSeqQ;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

int tile_tokens_for(int hq, int hkv) {
  if (hkv <= 0 || hq <= 0) return 0;
  const int G = hq / hkv;
  return G >= 128 ? 1 : 128 / G;
}

// Work planning for the persistent attention kernel assumes a 152-SM GB300
// (device-independent, so the workspace size query needs no device).
constexpr int kPlanSMs = 152;
constexpr int kMinSplitBlocks = 4;
constexpr int kProxyFewTiles = 2;    // proxy tiles per SM below which columns are split
constexpr int kProxyCtasPerSM = 16;  // proxy CTAs per SM aimed at when tiles are few
constexpr int kProxyMinSlice = 16;   // fewest block columns per proxy CTA

struct PrefillLayout {
  int W, max_tiles, cap, words;
  int whole_units, tail_units, splits, pps, rows_part, num_items;
  size_t off_info, off_len, off_blocks, off_member, off_part_o, off_part_ml, off_counter, total;
};

PrefillLayout prefill_layout(int batch, int total_q, int hq, int hkv, int topk, int max_seqlen_q) {
  PrefillLayout L{};
  // Tiles never span sequences, so capping W at the longest query run changes
  // no tile; it only shrinks the union arrays and the Q tile of short runs.
  L.W = tile_tokens_for(hq, hkv);
  const int sq = max_seqlen_q < 1 ? 1 : max_seqlen_q;
  if (sq < L.W) L.W = sq;
  // Tile count bound: sum_b ceil(Lq_b / W) <= ceil(total_q / W) + batch, a tile
  // has at least one token, and with W >= every Lq a sequence has one tile.
  long long mt = ((long long)total_q + L.W - 1) / L.W + batch;
  if (total_q > 0 && mt > total_q) mt = total_q;
  if (L.W >= sq && mt > batch) mt = batch;
  if (mt < 1) mt = 1;
  L.max_tiles = (int)mt;
  L.cap = L.W * topk;
  L.words = (L.cap + 31) / 32;
  const int G = hq / hkv;
  const long long units = (long long)hkv * L.max_tiles;
  // Longest union a tile can have: its tokens' selections, at most cap.
  const long long bound_ll = (long long)L.W * topk;
  const int bound = (int)(bound_ll < L.cap ? bound_ll : L.cap);
  // Whole units fill complete rounds of the SMs; the remainder ("tail") is
  // split so the last round is spread over all SMs.
  L.whole_units = (int)units;
  L.tail_units = 0;
  L.splits = 1;
  L.pps = L.cap;
  // The split count minimises the tail's length in blocks: rounds of pieces
  // over the SMs times the piece size, plus one block per item for its start
  // and hand-over (pieces are dealt round-robin, one per SM and round).
  const long long rem = units % kPlanSMs;
  if (rem > 0) {
    long long best_cost = ((rem + kPlanSMs - 1) / kPlanSMs) * (long long)(bound + 1);
    for (int S = 2; S <= bound; ++S) {
      int pps = (bound + S - 1) / S;
      if (pps < kMinSplitBlocks) pps = kMinSplitBlocks;
      const int s_eff = (bound + pps - 1) / pps;
      if (s_eff < 2) continue;
      const long long rounds = (rem * s_eff + kPlanSMs - 1) / kPlanSMs;
      const long long cost = rounds * (pps + 1);
      if (cost < best_cost) {
        best_cost = cost;
        L.splits = s_eff;
        L.pps = pps;
        L.tail_units = (int)rem;
        L.whole_units = (int)(units - rem);
      }
    }
  }
  L.rows_part = 0;
  if (L.tail_units > 0) {
    const int rows = L.W * G;
    L.rows_part = rows >= 128 ? 128 : ((rows + 15) / 16) * 16;
  }
  L.num_items = L.whole_units + L.tail_units * L.splits;
  const size_t parts = (size_t)L.tail_units * L.splits;
  size_t off = 0;
  L.off_info = off;
  off += up256((size_t)L.max_tiles * 2 * sizeof(int32_t));
  L.off_len = off;
  off += up256((size_t)units * sizeof(int32_t));
  L.off_blocks = off;
  off += up256((size_t)units * L.cap * sizeof(int32_t));
  L.off_member = off;
  off += up256((size_t)units * L.W * L.words * sizeof(uint32_t));
  L.off_part_o = off;
  off += up256(parts * L.rows_part * 128 * sizeof(float));
  L.off_part_ml = off;
  off += up256(parts * L.rows_part * 2 * sizeof(float));
  L.off_counter = off;
  off += 256;
  L.total = off;
  return L;
}

// Layout of the swapped-orientation prefill kernel: query tiles of W tokens
// with W * G <= 256 rows (W <= 32, so a tile's member tokens fit one 32-bit
// mask per union block), no splits, and the per-block member masks.
struct SwappedLayout {
  bool usable;  // G a multiple of 8 and at most 64
  int W, max_tiles, cap, words, num_items;
  size_t off_info, off_len, off_blocks, off_member, off_bmem, off_counter, total;
};

SwappedLayout swapped_layout(int batch, int total_q, int hq, int hkv, int topk,
                             int max_seqlen_q) {
  SwappedLayout L{};
  const int G = hkv > 0 ? hq / hkv : 0;
  L.usable = G >= 8 && G <= 64 && G % 8 == 0;
  if (!L.usable) return L;
  L.W = 256 / G < 32 ? 256 / G : 32;
  const int sq = max_seqlen_q < 1 ? 1 : max_seqlen_q;
  if (sq < L.W) L.W = sq;
  long long mt = ((long long)total_q + L.W - 1) / L.W + batch;
  if (total_q > 0 && mt > total_q) mt = total_q;
  if (L.W >= sq && mt > batch) mt = batch;
  if (mt < 1) mt = 1;
  L.max_tiles = (int)mt;
  L.cap = L.W * topk;
  L.words = (L.cap + 31) / 32;
  const size_t units = (size_t)hkv * L.max_tiles;
  L.num_items = (int)units;
  size_t off = 0;
  L.off_info = off;
  off += up256((size_t)L.max_tiles * 2 * sizeof(int32_t));
  L.off_len = off;
  off += up256(units * sizeof(int32_t));
  L.off_blocks = off;
  off += up256(units * L.cap * sizeof(int32_t));
  L.off_member = off;
  off += up256(units * L.W * L.words * sizeof(uint32_t));
  L.off_bmem = off;
  off += up256(units * L.cap * sizeof(uint32_t));
  L.off_counter = off;
  off += 256;
  L.total = off;
  return L;
}

// Forward route: 0 chooses by measured speed (the union-tile kernel, for
// now, on every workload measured), 1 always the union-tile kernel, 2 the
// swapped kernel wherever it applies (msa_set_prefill_route).
int g_route = 0;

bool use_swapped(const SwappedLayout& S, int esize, int max_seqlen_q) {
  (void)max_seqlen_q;
  return S.usable && esize == 2 && g_route == 2;
}

// Flat E4M3 K/V on a prefill-sized call (at least as many query rows x query
// heads as key rows x KV heads) is decoded to bf16 once, into the workspace,
// and attended with the bf16 kernel: the attention kernel is tensor-bound
// there, and converting in the kernel costs it more than the HBM-bound
// decode pass does. Decode-sized calls (few query rows over long contexts)
// read each selected block about once, so they keep the E4M3 bytes and
// convert in the kernel.
bool kv_decode_route(msa_dtype_t kv_dtype, bool paged, long long total_q, int hq,
                     long long total_k, int hkv) {
  return kv_dtype == MSA_FP8_E4M3 && !paged && total_k > 0 &&
         total_q * hq >= total_k * hkv;
}
// Bytes of one bf16 copy of a flat (total_k, hkv, 128) tensor, 256-aligned.
size_t kv_copy_bytes(long long total_k, int hkv) {
  return up256((size_t)total_k * (size_t)hkv * 128 * 2);
}

// Paged E4M3 / NVFP4 K/V on a prefill-sized call (query rows x query heads at
// least the page table's key capacity x KV heads) is decoded into a bf16 page
// pool (batch * max_pages pages) with a renumbered page table, for the same
// reason as the flat copy above.
bool paged_copy_route(long long total_q, int hq, int batch, int max_pages, int hkv) {
  return batch > 0 && max_pages > 0 &&
         total_q * hq >= (long long)batch * max_pages * 128 * hkv;
}
// Bytes of the bf16 K and V page pools and the renumbered table.
size_t page_pool_bytes(int batch, int max_pages, int hkv) {
  const size_t pages = (size_t)batch * max_pages;
  return 2 * up256(pages * hkv * 128 * 128 * 2) + up256(pages * sizeof(int32_t));
}
// Places the pools after the first `need` bytes of the workspace.
void place_page_pool(PageDecodeArgs* pd, uint8_t* ws, size_t need, int batch, int max_pages,
                     int hkv) {
  const size_t pages = (size_t)batch * max_pages;
  const size_t side = up256(pages * hkv * 128 * 128 * 2);
  pd->k16 = reinterpret_cast<uint16_t*>(ws + need);
  pd->v16 = reinterpret_cast<uint16_t*>(ws + need + side);
  pd->pt_out = reinterpret_cast<int32_t*>(ws + need + 2 * side);
  pd->batch = batch;
  pd->max_pages = max_pages;
  pd->hkv = hkv;
}

// (d, H, T) map over a (T, H, d) tensor; element size 2 (bf16) or 1 (e4m3).
bool map_rows(CUtensorMap* m, const void* base, int esize, int H, long long T, uint32_t box_h,
              uint32_t box_t) {
  const uint64_t dims[3] = {128, (uint64_t)H, (uint64_t)(T > 0 ? T : 1)};
  const uint64_t strides[2] = {128ull * esize, 128ull * esize * H};
  const uint32_t box[3] = {esize == 2 ? 64u : 128u, box_h, box_t};  // 128-byte inner box
  return encode_tiled(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                      3, base, dims, strides, box);
}

// (d, 128, H, pages) map over a (pages, H, 128, d) paged cache.
bool map_pages(CUtensorMap* m, const void* base, int esize, int H, int pages) {
  const uint64_t dims[4] = {128, 128, (uint64_t)H, (uint64_t)pages};
  const uint64_t strides[3] = {128ull * esize, 128ull * 128 * esize, 128ull * 128 * esize * H};
  const uint32_t box[4] = {esize == 2 ? 64u : 128u, 128u, 1u, 1u};
  return encode_tiled(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                      4, base, dims, strides, box);
}

// (64 bytes, 128, H, pages) map over the packed-NVFP4 code slices of a planar
// page pool (slice (p, h) at p * page_stride + h * 8192), 64-byte swizzle.
bool map_fp4_codes(CUtensorMap* m, const void* base, int H, int pages, long long page_stride) {
  const uint64_t dims[4] = {64, 128, (uint64_t)H, (uint64_t)pages};
  const uint64_t strides[3] = {64, 64ull * 128, (uint64_t)page_stride};
  const uint32_t box[4] = {64u, 128u, 1u, 1u};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_64B);
}

msa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_CUDA_ERROR; }

cudaEvent_t g_timing[3] = {nullptr, nullptr, nullptr};
bool g_timing_on = false;

void mark(int i, cudaStream_t s) {
  if (g_timing_on) cudaEventRecord(g_timing[i], s);
}

}  // namespace

cudaError_t set_smem_limit(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::vector<std::tuple<const void*, int, int>> done;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const auto& t : done)
      if (std::get<0>(t) == kernel && std::get<1>(t) == dev && std::get<2>(t) >= bytes)
        return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) {
    std::lock_guard<std::mutex> lk(mu);
    done.emplace_back(kernel, dev, bytes);
  }
  return e;
}

int device_smem_optin() {
  static int cache[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  if (cache[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return 0;
    cache[dev] = v;
  }
  return cache[dev];
}

}  // namespace msa

using namespace msa;

extern "C" {

const char* msa_status_string(msa_status_t s) {
  switch (s) {
    case MSA_OK: return "MSA_OK";
    case MSA_INVALID_ARG: return "MSA_INVALID_ARG";
    case MSA_UNSUPPORTED: return "MSA_UNSUPPORTED";
    case MSA_WORKSPACE_TOO_SMALL: return "MSA_WORKSPACE_TOO_SMALL";
    case MSA_CUDA_ERROR: return "MSA_CUDA_ERROR";
  }
  return "MSA_UNKNOWN_STATUS";
}

int msa_union_tile_tokens(int num_qo_heads, int num_kv_heads) {
  return tile_tokens_for(num_qo_heads, num_kv_heads);
}

size_t msa_sparse_attention_workspace_size(int batch, int total_q, int num_qo_heads,
                                           int num_kv_heads, int head_dim, int topk,
                                           int max_seqlen_q, int paged) {
  if (batch < 1 || total_q < 0 || num_qo_heads < 1 || num_kv_heads < 1 ||
      num_qo_heads % num_kv_heads != 0 || head_dim != 128 || topk < 1 || topk > kMaxTopk ||
      num_qo_heads / num_kv_heads > 128)
    return 0;
  (void)paged;
  const size_t a =
      prefill_layout(batch, total_q, num_qo_heads, num_kv_heads, topk, max_seqlen_q).total;
  const SwappedLayout S =
      swapped_layout(batch, total_q, num_qo_heads, num_kv_heads, topk, max_seqlen_q);
  return S.usable && S.total > a ? S.total : a;
}

size_t msa_sparse_attention_workspace_size_kv(int batch, int total_q, int num_qo_heads,
                                              int num_kv_heads, int head_dim, int topk,
                                              int max_seqlen_q, int paged, msa_dtype_t kv_dtype,
                                              int total_k) {
  const size_t base = msa_sparse_attention_workspace_size(
      batch, total_q, num_qo_heads, num_kv_heads, head_dim, topk, max_seqlen_q, paged);
  if (base == 0 || total_k < 0) return 0;
  if (paged != 0) {  // total_k carries the page table width
    if (kv_dtype != MSA_FP8_E4M3 || !paged_copy_route(total_q, num_qo_heads, batch, total_k,
                                                      num_kv_heads))
      return base;
    return base + page_pool_bytes(batch, total_k, num_kv_heads);
  }
  if (!kv_decode_route(kv_dtype, paged != 0, total_q, num_qo_heads, total_k, num_kv_heads))
    return base;
  return base + 2 * kv_copy_bytes(total_k, num_kv_heads);
}

size_t msa_sparse_attention_nvfp4_workspace_size(int batch, int total_q, int num_qo_heads,
                                                 int num_kv_heads, int head_dim, int topk,
                                                 int max_seqlen_q, int max_pages) {
  const size_t base = msa_sparse_attention_workspace_size(
      batch, total_q, num_qo_heads, num_kv_heads, head_dim, topk, max_seqlen_q, 1);
  if (base == 0 || max_pages < 1) return 0;
  if (paged_copy_route(total_q, num_qo_heads, batch, max_pages, num_kv_heads))
    return base + page_pool_bytes(batch, max_pages, num_kv_heads);
  if (fp4_decode_route(num_qo_heads, num_kv_heads, max_seqlen_q))
    return base + fp4_decode_workspace_bytes((long long)total_q * num_kv_heads, topk);
  return base;
}

}  // extern "C"

namespace msa {
namespace {

// Everything a forward launch needs, decided and encoded on the host.
struct ForwardPlan {
  bool empty = true;  // total_q == 0: nothing to launch
  KvDecodeArgs dq{};    // n16 > 0: E4M3 K/V decoded to bf16 before the union kernel
  PageDecodeArgs pd{};  // mode > 0: paged E4M3 / NVFP4 pages decoded to a bf16 pool first
  UnionArgs u{};
  PrefillArgs a{};
  bool swapped = false;  // the swapped-orientation prefill kernel, else the union-tile kernel
  bool skip_union = false;  // direct mode: the attention kernel builds one-token unions itself
  bool fp4_decode = false;  // packed-NVFP4 decode-shaped call: fp4_decode_kernel alone
  Fp4DecodeArgs f4{};
};

// The swapped-kernel part of a forward plan (arguments already checked).
msa_status_t build_swapped(const void* q, msa_dtype_t q_dtype, const void* k, const void* v,
                           const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
                           const int32_t* cu_seqlens_k, const int32_t* page_table, int max_pages,
                           int num_pages, const int32_t* seqused_k, int batch, int total_q,
                           int total_k, int num_qo_heads, int num_kv_heads, int causal,
                           float scale_log2, void* out, float* lse, uint8_t* ws,
                           const SwappedLayout& S, unsigned* fault, ForwardPlan* plan) {
  const bool paged = page_table != nullptr;
  const int G = num_qo_heads / num_kv_heads;
  plan->swapped = true;
  UnionArgs& u = plan->u;
  u.q2k = q2k_indices;
  u.topk = topk;
  u.cu_q = cu_seqlens_q;
  u.cu_k = cu_seqlens_k;
  u.seqused_k = seqused_k;
  u.max_pages = max_pages;
  u.batch = batch;
  u.total_q = total_q;
  u.num_kv_heads = num_kv_heads;
  u.causal = causal ? 1 : 0;
  u.tile_tokens = S.W;
  u.max_tiles = S.max_tiles;
  u.cap = S.cap;
  u.words = S.words;
  u.union_len = reinterpret_cast<int32_t*>(ws + S.off_len);
  u.union_blocks = reinterpret_cast<int32_t*>(ws + S.off_blocks);
  u.member = reinterpret_cast<uint32_t*>(ws + S.off_member);
  u.block_members = reinterpret_cast<uint32_t*>(ws + S.off_bmem);
  u.tile_info = reinterpret_cast<int32_t*>(ws + S.off_info);
  u.item_counter = reinterpret_cast<int32_t*>(ws + S.off_counter);
  PrefillArgs& a = plan->a;
  a.fault = fault;
  bool ok = map_rows(&a.tmap_q, q, 2, num_qo_heads, total_q, (uint32_t)G, (uint32_t)S.W) &&
            map_rows(&a.tmap_q1, q, 2, num_qo_heads, total_q, (uint32_t)G, 1u);
  if (paged) {
    ok = ok && map_pages(&a.tmap_k, k, 2, num_kv_heads, num_pages) &&
         map_pages(&a.tmap_v, v, 2, num_kv_heads, num_pages);
  } else {
    ok = ok && map_rows(&a.tmap_k, k, 2, num_kv_heads, total_k, 1, 128) &&
         map_rows(&a.tmap_v, v, 2, num_kv_heads, total_k, 1, 128);
  }
  if (!ok) return MSA_CUDA_ERROR;
  a.paged = paged ? 1 : 0;
  a.kv_fp8 = 0;
  a.kv_fp4 = 0;
  a.out_scale = 1.f;
  a.f16 = q_dtype == MSA_FP16 ? 1 : 0;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.seqused_k = seqused_k;
  a.batch = batch;
  a.total_q = total_q;
  a.num_qo_heads = num_qo_heads;
  a.num_kv_heads = num_kv_heads;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale_log2;
  a.tile_tokens = S.W;
  a.max_tiles = S.max_tiles;
  a.cap = S.cap;
  a.words = S.words;
  a.union_len = u.union_len;
  a.union_blocks = u.union_blocks;
  a.member = u.member;
  a.block_members = u.block_members;
  a.tile_info = u.tile_info;
  a.out = out;
  a.lse = lse;
  a.whole_units = S.num_items;
  a.tail_units = 0;
  a.splits = 1;
  a.pps = S.cap;
  a.rows_part = 0;
  a.num_items = S.num_items;
  a.part_o = nullptr;
  a.part_ml = nullptr;
  a.item_counter = u.item_counter;
  return MSA_OK;
}

msa_status_t build_forward(
    const void* q, msa_dtype_t q_dtype, const void* k, const void* v, msa_dtype_t kv_dtype,
    const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, const int32_t* page_table, int max_pages, int num_pages,
    const int32_t* seqused_k, int batch, int total_q, int total_k, int num_qo_heads,
    int num_kv_heads, int head_dim, int max_seqlen_q, int causal, float softmax_scale, void* out,
    float* lse, void* workspace, size_t workspace_bytes, ForwardPlan* plan) {
  // ---- argument checks (host only; nothing is read from the device) ----
  const bool paged = page_table != nullptr;
  if (cu_seqlens_k != nullptr && paged) return MSA_INVALID_ARG;   // two length sources
  if (cu_seqlens_k == nullptr && !paged) return MSA_INVALID_ARG;  // no length source
  if (paged && (seqused_k == nullptr || max_pages < 1 || num_pages < 1)) return MSA_INVALID_ARG;
  if (!paged && seqused_k != nullptr) return MSA_INVALID_ARG;
  if (q == nullptr || k == nullptr || v == nullptr || q2k_indices == nullptr ||
      cu_seqlens_q == nullptr || out == nullptr)
    return MSA_INVALID_ARG;
  if (batch < 1 || total_q < 0 || num_qo_heads < 1 || num_kv_heads < 1) return MSA_INVALID_ARG;
  if (num_qo_heads % num_kv_heads != 0) return MSA_INVALID_ARG;
  if (!paged && total_k < 1) return MSA_INVALID_ARG;
  if (total_q > 0 && max_seqlen_q < 1) return MSA_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(q2k_indices, 4) || !aligned(cu_seqlens_q, 4) ||
      (cu_seqlens_k && !aligned(cu_seqlens_k, 4)) || (page_table && !aligned(page_table, 4)) ||
      (seqused_k && !aligned(seqused_k, 4)) || (lse && !aligned(lse, 4)) ||
      (workspace && !aligned(workspace, 256)))
    return MSA_INVALID_ARG;
  if (head_dim != 128) return MSA_UNSUPPORTED;
  // bf16 q with bf16 or E4M3 K/V, or fp16 q with fp16 K/V.
  if (q_dtype == MSA_FP16 ? kv_dtype != MSA_FP16
                          : (q_dtype != MSA_BF16 || (kv_dtype != MSA_BF16 && kv_dtype != MSA_FP8_E4M3)))
    return MSA_UNSUPPORTED;
  if (topk < 1 || topk > kMaxTopk) return MSA_UNSUPPORTED;
  const int G = num_qo_heads / num_kv_heads;
  if (G > 128) return MSA_UNSUPPORTED;
  const size_t need = msa_sparse_attention_workspace_size(
      batch, total_q, num_qo_heads, num_kv_heads, head_dim, topk, max_seqlen_q, paged ? 1 : 0);
  if (workspace_bytes < need || (need > 0 && workspace == nullptr)) return MSA_WORKSPACE_TOO_SMALL;
  plan->empty = total_q == 0;
  if (plan->empty) return MSA_OK;
  unsigned* fault = fault_word();
  if (fault == nullptr) return MSA_CUDA_ERROR;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)head_dim);
  const float scale_log2 = scale * 1.4426950408889634f;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // E4M3 on a prefill-sized call: the flat copy or the paged page pool goes
  // after the layout's regions when the workspace holds it; with a smaller
  // workspace the attention kernel converts E4M3 itself.
  const size_t copy = kv_copy_bytes(total_k, num_kv_heads);
  if (kv_decode_route(kv_dtype, paged, total_q, num_qo_heads, total_k, num_kv_heads) &&
      workspace_bytes >= need + 2 * copy) {
    plan->dq.k8 = k;
    plan->dq.v8 = v;
    plan->dq.k16 = ws + need;
    plan->dq.v16 = ws + need + copy;
    plan->dq.n16 = (size_t)total_k * num_kv_heads * 128 / 16;
    k = plan->dq.k16;
    v = plan->dq.v16;
    kv_dtype = MSA_BF16;
  } else if (kv_dtype == MSA_FP8_E4M3 && paged &&
             paged_copy_route(total_q, num_qo_heads, batch, max_pages, num_kv_heads) &&
             workspace_bytes >= need + page_pool_bytes(batch, max_pages, num_kv_heads)) {
    PageDecodeArgs& pd = plan->pd;
    place_page_pool(&pd, ws, need, batch, max_pages, num_kv_heads);
    pd.mode = 1;
    pd.page_table = page_table;
    pd.seqused_k = seqused_k;
    pd.num_pages = num_pages;
    pd.k8 = static_cast<const uint8_t*>(k);
    pd.v8 = static_cast<const uint8_t*>(v);
    k = pd.k16;
    v = pd.v16;
    kv_dtype = MSA_BF16;
    page_table = pd.pt_out;
    num_pages = batch * max_pages;
  }
  const int esize = kv_dtype == MSA_FP8_E4M3 ? 1 : 2;

  const SwappedLayout S =
      swapped_layout(batch, total_q, num_qo_heads, num_kv_heads, topk, max_seqlen_q);
  if (use_swapped(S, esize, max_seqlen_q))
    return build_swapped(q, q_dtype, k, v, q2k_indices, topk, cu_seqlens_q, cu_seqlens_k,
                         page_table, max_pages, num_pages, seqused_k, batch, total_q, total_k,
                         num_qo_heads, num_kv_heads, causal, scale_log2, out, lse, ws, S, fault,
                         plan);
  const PrefillLayout L =
      prefill_layout(batch, total_q, num_qo_heads, num_kv_heads, topk, max_seqlen_q);
  UnionArgs& u = plan->u;
  u.q2k = q2k_indices;
  u.topk = topk;
  u.cu_q = cu_seqlens_q;
  u.cu_k = cu_seqlens_k;
  u.seqused_k = seqused_k;
  u.max_pages = max_pages;
  u.batch = batch;
  u.total_q = total_q;
  u.num_kv_heads = num_kv_heads;
  u.causal = causal ? 1 : 0;
  u.tile_tokens = L.W;
  u.max_tiles = L.max_tiles;
  u.cap = L.cap;
  u.words = L.words;
  u.union_len = reinterpret_cast<int32_t*>(ws + L.off_len);
  u.union_blocks = reinterpret_cast<int32_t*>(ws + L.off_blocks);
  u.member = reinterpret_cast<uint32_t*>(ws + L.off_member);
  u.tile_info = reinterpret_cast<int32_t*>(ws + L.off_info);
  u.item_counter = reinterpret_cast<int32_t*>(ws + L.off_counter);
  PrefillArgs& a = plan->a;
  a.fault = fault;
  bool ok = map_rows(&a.tmap_q, q, 2, num_qo_heads, total_q, (uint32_t)G, (uint32_t)L.W);
  if (paged) {
    ok = ok && map_pages(&a.tmap_k, k, esize, num_kv_heads, num_pages) &&
         map_pages(&a.tmap_v, v, esize, num_kv_heads, num_pages);
  } else {
    ok = ok && map_rows(&a.tmap_k, k, esize, num_kv_heads, total_k, 1, 128) &&
         map_rows(&a.tmap_v, v, esize, num_kv_heads, total_k, 1, 128);
  }
  if (!ok) return MSA_CUDA_ERROR;
  a.paged = paged ? 1 : 0;
  a.kv_fp8 = esize == 1 ? 1 : 0;
  a.kv_fp4 = 0;
  a.out_scale = 1.f;
  a.f16 = q_dtype == MSA_FP16 ? 1 : 0;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.seqused_k = seqused_k;
  a.batch = batch;
  a.total_q = total_q;
  a.num_qo_heads = num_qo_heads;
  a.num_kv_heads = num_kv_heads;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale_log2;
  a.tile_tokens = L.W;
  a.max_tiles = L.max_tiles;
  a.cap = L.cap;
  a.words = L.words;
  a.union_len = u.union_len;
  a.union_blocks = u.union_blocks;
  a.member = u.member;
  a.tile_info = u.tile_info;
  a.out = out;
  a.lse = lse;
  a.whole_units = L.whole_units;
  a.tail_units = L.tail_units;
  a.splits = L.splits;
  a.pps = L.pps;
  a.rows_part = L.rows_part;
  a.num_items = L.num_items;
  a.part_o = reinterpret_cast<float*>(ws + L.off_part_o);
  a.part_ml = reinterpret_cast<float*>(ws + L.off_part_ml);
  a.item_counter = u.item_counter;
  a.q2k = q2k_indices;
  a.topk = topk;
  // One-token tiles (decode with seqlen_q 1, or G >= 128): the attention
  // kernel derives each tile's union from the token's own row (bf16 / fp16
  // instance; the E4M3 / NVFP4 converter instance keeps the union kernel).
  a.direct = (L.W == 1 && topk <= 32 && esize == 2) ? 1 : 0;
  plan->skip_union = a.direct != 0;
  // The counter reset before a direct launch is an ordinary launch, so every
  // earlier kernel (a decode pass included) has completed when it starts.
  a.wait_late = a.direct;
  return MSA_OK;
}

// The packed-NVFP4 paged route: the E4M3 kernel instance (converter warps),
// fed by bulk copies of each page's K and V slices and block scales, with
// the K global scale folded into the softmax scale and the V global scale
// into the output.
msa_status_t build_forward_fp4(
    const void* q, msa_dtype_t q_dtype, const void* k, const void* k_scale, const void* v,
    const void* v_scale, long long page_stride, float k_global_scale, float v_global_scale,
    const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q, const int32_t* page_table,
    int max_pages, int num_pages, const int32_t* seqused_k, int batch, int total_q,
    int num_qo_heads, int num_kv_heads, int head_dim, int max_seqlen_q, float softmax_scale,
    void* out, float* lse, void* workspace, size_t workspace_bytes, ForwardPlan* plan) {
  if (k == nullptr || k_scale == nullptr || v == nullptr || v_scale == nullptr ||
      page_table == nullptr)
    return MSA_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(k_scale, 16) || !aligned(v, 16) || !aligned(v_scale, 16) ||
      page_stride <= 0 || page_stride % 16 != 0)
    return MSA_INVALID_ARG;
  if (!(k_global_scale > 0.f) || !(v_global_scale > 0.f) || !std::isfinite(k_global_scale) ||
      !std::isfinite(v_global_scale))
    return MSA_INVALID_ARG;
  if (q_dtype != MSA_BF16) return MSA_UNSUPPORTED;
  // Prefill-sized calls given the larger workspace: decode the pages into a
  // bf16 pool and run the bf16 attention kernel on it.
  const size_t need = msa_sparse_attention_workspace_size(
      batch, total_q, num_qo_heads, num_kv_heads, head_dim, topk, max_seqlen_q, 1);
  if (need > 0 && total_q > 0 && workspace != nullptr && aligned(workspace, 256) &&
      paged_copy_route(total_q, num_qo_heads, batch, max_pages, num_kv_heads) &&
      workspace_bytes >= need + page_pool_bytes(batch, max_pages, num_kv_heads)) {
    PageDecodeArgs pd{};
    place_page_pool(&pd, static_cast<uint8_t*>(workspace), need, batch, max_pages,
                    num_kv_heads);
    pd.mode = 2;
    pd.page_table = page_table;
    pd.seqused_k = seqused_k;
    pd.num_pages = num_pages;
    pd.fp4_k = static_cast<const uint8_t*>(k);
    pd.fp4_k_scale = static_cast<const uint8_t*>(k_scale);
    pd.fp4_v = static_cast<const uint8_t*>(v);
    pd.fp4_v_scale = static_cast<const uint8_t*>(v_scale);
    pd.fp4_page_stride = page_stride;
    const msa_status_t sc = build_forward(
        q, q_dtype, pd.k16, pd.v16, MSA_BF16, q2k_indices, topk, cu_seqlens_q, nullptr,
        pd.pt_out, max_pages, batch * max_pages, seqused_k, batch, total_q, 0, num_qo_heads,
        num_kv_heads, head_dim, max_seqlen_q, 1, softmax_scale, out, lse, workspace,
        workspace_bytes, plan);
    if (sc != MSA_OK || plan->empty) return sc;
    plan->pd = pd;
    plan->a.scale_log2 *= k_global_scale;
    plan->a.out_scale = v_global_scale;
    return MSA_OK;
  }
  // The checks and plan of the E4M3 paged route (the tensor maps it encodes
  // over the code bytes are never used by this route).
  const msa_status_t st = build_forward(
      q, q_dtype, k, v, MSA_FP8_E4M3, q2k_indices, topk, cu_seqlens_q, nullptr, page_table,
      max_pages, num_pages, seqused_k, batch, total_q, 0, num_qo_heads, num_kv_heads, head_dim,
      max_seqlen_q, 1, softmax_scale, out, lse, workspace, workspace_bytes, plan);
  if (st != MSA_OK || plan->empty) return st;
  PrefillArgs& a = plan->a;
  a.kv_fp4 = 1;
  a.fp4_k = static_cast<const uint8_t*>(k);
  a.fp4_k_scale = static_cast<const uint8_t*>(k_scale);
  a.fp4_v = static_cast<const uint8_t*>(v);
  a.fp4_v_scale = static_cast<const uint8_t*>(v_scale);
  a.fp4_page_stride = page_stride;
  a.scale_log2 *= k_global_scale;
  a.out_scale = v_global_scale;
  // Decode-shaped calls (G <= 16, a few query tokens per request), given the
  // workspace for their block lists: one unit per (token, KV head) in the
  // register-dequantizing decode kernel.
  const int G = num_qo_heads / num_kv_heads;
  const long long units = (long long)total_q * num_kv_heads;
  if (fp4_decode_route(num_qo_heads, num_kv_heads, max_seqlen_q) && workspace != nullptr &&
      aligned(workspace, 256) && workspace_bytes >= need + fp4_decode_workspace_bytes(units, topk)) {
    Fp4DecodeArgs& f = plan->f4;
    place_fp4_decode_workspace(&f, static_cast<uint8_t*>(workspace) + need, units, topk);
    if (!map_fp4_codes(&f.tmap_kc, k, num_kv_heads, num_pages, page_stride) ||
        !map_fp4_codes(&f.tmap_vc, v, num_kv_heads, num_pages, page_stride))
      return MSA_CUDA_ERROR;
    f.fault = a.fault;
    f.q = static_cast<const uint16_t*>(q);
    f.q2k = q2k_indices;
    f.topk = topk;
    f.cu_q = cu_seqlens_q;
    f.page_table = page_table;
    f.max_pages = max_pages;
    f.num_pages = num_pages;
    f.seqused_k = seqused_k;
    f.k_scale = static_cast<const uint8_t*>(k_scale);
    f.v_scale = static_cast<const uint8_t*>(v_scale);
    f.page_stride = page_stride;
    f.batch = batch;
    f.total_q = total_q;
    f.num_qo_heads = num_qo_heads;
    f.num_kv_heads = num_kv_heads;
    f.G = G;
    f.scale_log2 = a.scale_log2;
    f.out_scale = v_global_scale;
    f.out = static_cast<uint16_t*>(out);
    f.lse = lse;
    plan->fp4_decode = true;
  }
  return MSA_OK;
}

msa_status_t launch_forward(const ForwardPlan& p, cudaStream_t stream) {
  if (p.empty) return MSA_OK;
  mark(0, stream);
  if (p.fp4_decode) {
    mark(1, stream);
    const cudaError_t e = launch_fp4_decode(p.f4, stream);
    mark(2, stream);
    return from_cuda(e);
  }
  cudaError_t e = launch_kv_decode(p.dq, stream);
  if (e != cudaSuccess) return MSA_CUDA_ERROR;
  e = launch_page_decode(p.pd, stream);
  if (e != cudaSuccess) return MSA_CUDA_ERROR;
  e = p.skip_union ? launch_reset_counter(p.a.item_counter, stream)
                   : launch_build_union(p.u, stream);
  if (e != cudaSuccess) return MSA_CUDA_ERROR;
  mark(1, stream);
  e = p.swapped ? launch_prefill_swapped(p.a, stream) : launch_prefill(p.a, stream);
  mark(2, stream);
  return from_cuda(e);
}

}  // namespace
}  // namespace msa

struct msa_attention_plan {
  msa::ForwardPlan p;
};

extern "C" {

#define MSA_FWD_ARGS                                                                           \
  q, q_dtype, k, v, kv_dtype, q2k_indices, topk, cu_seqlens_q, cu_seqlens_k, page_table,    \
      max_pages, num_pages, seqused_k, batch, total_q, total_k, num_qo_heads, num_kv_heads, \
      head_dim, max_seqlen_q, causal, softmax_scale, out, lse, workspace, workspace_bytes

msa_status_t msa_sparse_attention_fwd(
    const void* q, msa_dtype_t q_dtype, const void* k, const void* v, msa_dtype_t kv_dtype,
    const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, const int32_t* page_table, int max_pages, int num_pages,
    const int32_t* seqused_k, int batch, int total_q, int total_k, int num_qo_heads,
    int num_kv_heads, int head_dim, int max_seqlen_q, int causal, float softmax_scale, void* out,
    float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  msa::ForwardPlan p;
  const msa_status_t st = msa::build_forward(MSA_FWD_ARGS, &p);
  if (st != MSA_OK) return st;
  return msa::launch_forward(p, stream);
}

msa_status_t msa_sparse_attention_prepare(
    const void* q, msa_dtype_t q_dtype, const void* k, const void* v, msa_dtype_t kv_dtype,
    const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, const int32_t* page_table, int max_pages, int num_pages,
    const int32_t* seqused_k, int batch, int total_q, int total_k, int num_qo_heads,
    int num_kv_heads, int head_dim, int max_seqlen_q, int causal, float softmax_scale, void* out,
    float* lse, void* workspace, size_t workspace_bytes, msa_attention_plan_t** plan_out) {
  if (plan_out == nullptr) return MSA_INVALID_ARG;
  *plan_out = nullptr;
  msa_attention_plan_t* plan = new (std::nothrow) msa_attention_plan_t;
  if (plan == nullptr) return MSA_CUDA_ERROR;
  const msa_status_t st = msa::build_forward(MSA_FWD_ARGS, &plan->p);
  if (st != MSA_OK) {
    delete plan;
    return st;
  }
  *plan_out = plan;
  return MSA_OK;
}

msa_status_t msa_sparse_attention_run(const msa_attention_plan_t* plan, cudaStream_t stream) {
  if (plan == nullptr) return MSA_INVALID_ARG;
  return msa::launch_forward(plan->p, stream);
}

void msa_sparse_attention_plan_free(msa_attention_plan_t* plan) { delete plan; }

#undef MSA_FWD_ARGS

#define MSA_FP4_ARGS                                                                        \
  q, q_dtype, k, k_scale, v, v_scale, page_stride_bytes, k_global_scale, v_global_scale,  \
      q2k_indices, topk, cu_seqlens_q, page_table, max_pages, num_pages, seqused_k, batch, \
      total_q, num_qo_heads, num_kv_heads, head_dim, max_seqlen_q, softmax_scale, out, lse, \
      workspace, workspace_bytes

msa_status_t msa_sparse_attention_nvfp4_paged(
    const void* q, msa_dtype_t q_dtype, const void* k, const void* k_scale, const void* v,
    const void* v_scale, long long page_stride_bytes, float k_global_scale,
    float v_global_scale, const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
    const int32_t* page_table, int max_pages, int num_pages, const int32_t* seqused_k,
    int batch, int total_q, int num_qo_heads, int num_kv_heads, int head_dim,
    int max_seqlen_q, float softmax_scale, void* out, float* lse, void* workspace,
    size_t workspace_bytes, cudaStream_t stream) {
  msa::ForwardPlan p;
  const msa_status_t st = msa::build_forward_fp4(MSA_FP4_ARGS, &p);
  if (st != MSA_OK) return st;
  return msa::launch_forward(p, stream);
}

msa_status_t msa_sparse_attention_nvfp4_prepare(
    const void* q, msa_dtype_t q_dtype, const void* k, const void* k_scale, const void* v,
    const void* v_scale, long long page_stride_bytes, float k_global_scale,
    float v_global_scale, const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
    const int32_t* page_table, int max_pages, int num_pages, const int32_t* seqused_k,
    int batch, int total_q, int num_qo_heads, int num_kv_heads, int head_dim,
    int max_seqlen_q, float softmax_scale, void* out, float* lse, void* workspace,
    size_t workspace_bytes, msa_attention_plan_t** plan_out) {
  if (plan_out == nullptr) return MSA_INVALID_ARG;
  *plan_out = nullptr;
  msa_attention_plan_t* plan = new (std::nothrow) msa_attention_plan_t;
  if (plan == nullptr) return MSA_CUDA_ERROR;
  const msa_status_t st = msa::build_forward_fp4(MSA_FP4_ARGS, &plan->p);
  if (st != MSA_OK) {
    delete plan;
    return st;
  }
  *plan_out = plan;
  return MSA_OK;
}

#undef MSA_FP4_ARGS



msa_status_t msa_proxy_score(const void* q, msa_dtype_t q_dtype, const void* k,
                             msa_dtype_t k_dtype, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_k, const int32_t* page_table, int max_pages,
                             const int32_t* seqused_k, int batch, int total_q, int total_k,
                             int num_qo_heads, int num_kv_heads, int head_dim, int max_seqlen_q,
                             int max_k_tiles, int causal, int reduce_heads, float* output,
                             cudaStream_t stream) {
  const bool paged = page_table != nullptr;
  const int num_pages = paged ? total_k : 0;  // paged: total_k counts the pool's pages
  if (cu_seqlens_k != nullptr && paged) return MSA_INVALID_ARG;   // two length sources
  if (cu_seqlens_k == nullptr && !paged) return MSA_INVALID_ARG;  // no length source
  if (paged && (seqused_k == nullptr || max_pages < 1 || num_pages < 1)) return MSA_INVALID_ARG;
  if (!paged && seqused_k != nullptr) return MSA_INVALID_ARG;
  if (q == nullptr || k == nullptr || cu_seqlens_q == nullptr || output == nullptr)
    return MSA_INVALID_ARG;
  if (batch < 1 || total_q < 0 || total_k < 1 || num_qo_heads < 1 ||
      num_kv_heads < 1 || num_qo_heads % num_kv_heads != 0 || max_k_tiles < 1)
    return MSA_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(output, 4) || !aligned(cu_seqlens_q, 4) ||
      (cu_seqlens_k && !aligned(cu_seqlens_k, 4)) || (page_table && !aligned(page_table, 4)) ||
      (seqused_k && !aligned(seqused_k, 4)))
    return MSA_INVALID_ARG;
  // q bf16 or fp16; K of q's type, or E4M3 (upconverted to q's type in the kernel).
  if (head_dim != 128 || (q_dtype != MSA_BF16 && q_dtype != MSA_FP16) ||
      (k_dtype != q_dtype && k_dtype != MSA_FP8_E4M3))
    return MSA_UNSUPPORTED;
  const int k_esize = k_dtype == MSA_FP8_E4M3 ? 1 : 2;
  const int G = num_qo_heads / num_kv_heads;
  if (G > 128) return MSA_UNSUPPORTED;
  if (reduce_heads && (G > 32 || (G & (G - 1)) != 0)) return MSA_UNSUPPORTED;
  if (total_q == 0) return MSA_OK;
  ProxyArgs a{};
  a.fault = fault_word();
  if (a.fault == nullptr) return MSA_CUDA_ERROR;
  const int Wm = tile_tokens_for(num_qo_heads, num_kv_heads);
  bool ok = map_rows(&a.tmap_q, q, 2, num_qo_heads, total_q, (uint32_t)G, (uint32_t)Wm);
  ok = ok && (paged ? map_pages(&a.tmap_k, k, k_esize, num_kv_heads, num_pages)
                    : map_rows(&a.tmap_k, k, k_esize, num_kv_heads, total_k, 1, 128));
  if (!ok) return MSA_CUDA_ERROR;
  a.f16 = q_dtype == MSA_FP16 ? 1 : 0;
  a.k_fp8 = k_esize == 1 ? 1 : 0;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.paged = paged ? 1 : 0;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.seqused_k = seqused_k;
  a.batch = batch;
  a.total_q = total_q;
  a.num_qo_heads = num_qo_heads;
  a.num_kv_heads = num_kv_heads;
  a.max_k_tiles = max_k_tiles;
  a.causal = causal ? 1 : 0;
  a.reduce_heads = reduce_heads ? 1 : 0;
  a.tile_tokens = Wm;
  // Query tiles of one M tile when max_seqlen_q (a bound on every Lq) says no
  // sequence has more than Wm query tokens, else of two.
  a.one_m = (max_seqlen_q > 0 && max_seqlen_q <= Wm) ? 1 : 0;
  const int TQ = (a.one_m ? 1 : 2) * Wm;
  a.max_tiles = (total_q + TQ - 1) / TQ + batch;
  // Few tiles (decode-sized problems, under kProxyFewTiles per SM): split
  // each tile's block columns into slices so that there are about
  // kProxyCtasPerSM CTAs per SM, at least kProxyMinSlice columns each and at
  // most what one pass over the groups holds (the running-max buffer / TQ columns).
  const long long cap_cols = (a.k_fp8 ? 14336 : 16384) / TQ;  // the kernel's running-max buffer
  long long sc = max_k_tiles;
  const long long target = (long long)kProxyCtasPerSM * kPlanSMs;
  if ((long long)a.max_tiles < (long long)kProxyFewTiles * kPlanSMs) {
    sc = ((long long)max_k_tiles * a.max_tiles + target - 1) / target;
    if (sc < kProxyMinSlice) sc = kProxyMinSlice;
  }
  if (sc > cap_cols) sc = cap_cols;
  if (sc > max_k_tiles) sc = max_k_tiles;
  a.slice_cols = (int)sc;
  a.slices = (int)((max_k_tiles + sc - 1) / sc);
  a.out = output;
  return from_cuda(launch_proxy(a, stream));
}

msa_status_t msa_topk_select(const float* scores, int num_score_heads, int max_k_tiles,
                             int total_q, int topk, int num_kv_heads_out, int32_t* q2k_indices,
                             cudaStream_t stream) {
  if (scores == nullptr || q2k_indices == nullptr) return MSA_INVALID_ARG;
  if (num_score_heads < 1 || max_k_tiles < 1 || total_q < 0 || num_kv_heads_out < 1)
    return MSA_INVALID_ARG;
  if (num_score_heads != 1 && num_score_heads != num_kv_heads_out) return MSA_INVALID_ARG;
  if (!aligned(scores, 4) || !aligned(q2k_indices, 4)) return MSA_INVALID_ARG;
  if (topk < 1 || topk > kMaxTopk) return MSA_UNSUPPORTED;
  if (total_q == 0) return MSA_OK;
  TopkArgs a{scores, num_score_heads, max_k_tiles, total_q, topk, num_kv_heads_out, q2k_indices};
  return from_cuda(launch_topk(a, stream));
}

msa_status_t msa_build_union(const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_k, const int32_t* seqused_k, int max_pages,
                             int batch, int total_q, int num_kv_heads, int causal, int tile_tokens,
                             int max_tiles, int32_t* union_len, int32_t* union_blocks,
                             uint32_t* member, int32_t* tile_info, cudaStream_t stream) {
  if (q2k_indices == nullptr || cu_seqlens_q == nullptr || union_len == nullptr ||
      union_blocks == nullptr || member == nullptr)
    return MSA_INVALID_ARG;
  if ((cu_seqlens_k == nullptr) == (seqused_k == nullptr)) return MSA_INVALID_ARG;
  if (seqused_k != nullptr && max_pages < 1) return MSA_INVALID_ARG;
  if (batch < 1 || total_q < 0 || num_kv_heads < 1 || max_tiles < 0) return MSA_INVALID_ARG;
  if (tile_tokens < 1 || tile_tokens > 128) return MSA_INVALID_ARG;
  if (topk < 1 || topk > kMaxTopk) return MSA_UNSUPPORTED;
  if (max_tiles == 0) return MSA_OK;
  UnionArgs u{};
  u.q2k = q2k_indices;
  u.topk = topk;
  u.cu_q = cu_seqlens_q;
  u.cu_k = cu_seqlens_k;
  u.seqused_k = seqused_k;
  u.max_pages = max_pages;
  u.batch = batch;
  u.total_q = total_q;
  u.num_kv_heads = num_kv_heads;
  u.causal = causal ? 1 : 0;
  u.tile_tokens = tile_tokens;
  u.max_tiles = max_tiles;
  u.cap = tile_tokens * topk;
  u.words = (u.cap + 31) / 32;
  u.union_len = union_len;
  u.union_blocks = union_blocks;
  u.member = member;
  u.tile_info = tile_info;
  return from_cuda(launch_build_union(u, stream));
}

msa_status_t msa_build_union_block_members(
    const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, const int32_t* seqused_k, int max_pages, int batch, int total_q,
    int num_kv_heads, int causal, int tile_tokens, int max_tiles, int32_t* union_len,
    int32_t* union_blocks, uint32_t* member, uint32_t* block_members, int32_t* tile_info,
    cudaStream_t stream) {
  if (block_members == nullptr || tile_tokens > 32) return MSA_INVALID_ARG;
  if (q2k_indices == nullptr || cu_seqlens_q == nullptr || union_len == nullptr ||
      union_blocks == nullptr || member == nullptr)
    return MSA_INVALID_ARG;
  if ((cu_seqlens_k == nullptr) == (seqused_k == nullptr)) return MSA_INVALID_ARG;
  if (seqused_k != nullptr && max_pages < 1) return MSA_INVALID_ARG;
  if (batch < 1 || total_q < 0 || num_kv_heads < 1 || max_tiles < 0) return MSA_INVALID_ARG;
  if (tile_tokens < 1) return MSA_INVALID_ARG;
  if (topk < 1 || topk > kMaxTopk) return MSA_UNSUPPORTED;
  if (max_tiles == 0) return MSA_OK;
  UnionArgs u{};
  u.q2k = q2k_indices;
  u.topk = topk;
  u.cu_q = cu_seqlens_q;
  u.cu_k = cu_seqlens_k;
  u.seqused_k = seqused_k;
  u.max_pages = max_pages;
  u.batch = batch;
  u.total_q = total_q;
  u.num_kv_heads = num_kv_heads;
  u.causal = causal ? 1 : 0;
  u.tile_tokens = tile_tokens;
  u.max_tiles = max_tiles;
  u.cap = tile_tokens * topk;
  u.words = (u.cap + 31) / 32;
  u.union_len = union_len;
  u.union_blocks = union_blocks;
  u.member = member;
  u.block_members = block_members;
  u.tile_info = tile_info;
  return from_cuda(launch_build_union(u, stream));
}

msa_status_t msa_set_prefill_route(int route) {
  if (route < 0 || route > 2) return MSA_INVALID_ARG;
  g_route = route;
  return MSA_OK;
}

int msa_prefill_tile_tokens(int batch, int total_q, int num_qo_heads, int num_kv_heads,
                            int topk, int max_seqlen_q, msa_dtype_t kv_dtype) {
  if (batch < 1 || num_qo_heads < 1 || num_kv_heads < 1 || num_qo_heads % num_kv_heads != 0 ||
      topk < 1 || topk > kMaxTopk)
    return 0;
  const SwappedLayout S =
      swapped_layout(batch, total_q, num_qo_heads, num_kv_heads, topk, max_seqlen_q);
  if (use_swapped(S, kv_dtype == MSA_FP8_E4M3 ? 1 : 2, max_seqlen_q)) return S.W;
  return prefill_layout(batch, total_q, num_qo_heads, num_kv_heads, topk, max_seqlen_q).W;
}

msa_status_t msa_set_timing_events(void* const* events, int count) {
  if (count == 0) {
    g_timing_on = false;
    return MSA_OK;
  }
  if (count != 3 || events == nullptr) return MSA_INVALID_ARG;
  for (int i = 0; i < 3; ++i) {
    if (events[i] == nullptr) return MSA_INVALID_ARG;
    g_timing[i] = static_cast<cudaEvent_t>(events[i]);
  }
  g_timing_on = true;
  return MSA_OK;
}

msa_status_t msa_read_device_fault(unsigned int* fault, cudaStream_t stream) {
  if (fault == nullptr) return MSA_INVALID_ARG;
  unsigned* dev = fault_word();
  if (dev == nullptr) return MSA_CUDA_ERROR;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MSA_CUDA_ERROR;
  unsigned host = 0;
  if (cudaMemcpy(&host, dev, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MSA_CUDA_ERROR;
  const unsigned zero = 0;
  if (cudaMemcpy(dev, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return MSA_CUDA_ERROR;
  *fault = host;
  return MSA_OK;
}

}  // extern "C"
