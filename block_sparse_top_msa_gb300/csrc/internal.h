// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
// Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace msa {

// Device address of the library's fault word on the current device (host).
unsigned* fault_word();

struct UnionArgs {
  const int32_t* q2k;
  int topk;
  const int32_t* cu_q;
  const int32_t* cu_k;       // flat lengths, or NULL
  const int32_t* seqused_k;  // paged lengths, or NULL
  int max_pages;
  int batch;
  int total_q;
  int num_kv_heads;
  int causal;
  int tile_tokens;  // W
  int max_tiles;
  int cap;          // W * topk
  int words;        // ceil(cap / 32)
  int32_t* union_len;
  int32_t* union_blocks;
  uint32_t* member;
  int32_t* tile_info;  // may be NULL
  int32_t* item_counter;  // may be NULL: set to 0 (the attention kernel's work counter)
  // May be NULL (only for tile_tokens <= 32): per union position, a mask of
  // the tile's tokens that selected it (bit w = token w of the tile), i.e.
  // the membership bits transposed; (num_kv_heads, max_tiles, cap) uint32.
  uint32_t* block_members;
};
cudaError_t launch_build_union(const UnionArgs& a, cudaStream_t s);
// Zeroes the attention kernel's work counter in a one-thread kernel that
// lets its programmatic dependent start at once.
cudaError_t launch_reset_counter(int32_t* counter, cudaStream_t s);

struct TopkArgs {
  const float* scores;
  int num_score_heads;
  int max_k_tiles;
  int total_q;
  int topk;
  int num_kv_heads_out;
  int32_t* q2k;
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s);


struct PrefillArgs {
  unsigned* fault;      // device fault word (bounded-wait expiry, capacity)
  CUtensorMap tmap_q;   // (d, Hq, Tq) bf16, box (64, G, W)
  CUtensorMap tmap_k;   // flat (d or d bytes, Hkv, Tk) / paged (.., 128, Hkv, pages)
  CUtensorMap tmap_v;
  int paged;
  int kv_fp8;           // E4M3 K/V, or packed NVFP4 K/V (kv_fp4), converted in the kernel
  int f16;              // q, k, v and out are fp16 (else bf16; E4M3 K/V only with bf16)
  // Packed NVFP4 paged K/V: per page (fp4_page_stride bytes apart) and KV
  // head, 128 x 64 bytes of E2M1 pairs and 128 x 8 E4M3 block scales for K
  // (scales token-major) and for V (scales in 4 x 4 tiles, scale-index major).
  int kv_fp4;
  const uint8_t* fp4_k;
  const uint8_t* fp4_k_scale;
  const uint8_t* fp4_v;
  const uint8_t* fp4_v_scale;
  long long fp4_page_stride;
  float out_scale;      // multiplies every output (the NVFP4 V global scale; else 1)
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* page_table;
  int max_pages;
  int num_pages;
  const int32_t* seqused_k;
  int batch;
  int total_q;
  int num_qo_heads;
  int num_kv_heads;
  int causal;
  float scale_log2;
  int tile_tokens;
  int max_tiles;
  int cap;
  int words;
  // Union metadata (written by the union kernel, or in direct mode by this
  // kernel's item setup).
  int32_t* union_len;
  int32_t* union_blocks;
  const uint32_t* member;
  int32_t* tile_info;
  void* out;
  float* lse;
  // Work items, handed out dynamically to a persistent grid. Units are (query tile, KV head)
  // pairs, head-major with the heaviest tiles first within a head. The first whole_units units are one item each and
  // write out/lse directly. Each remaining ("tail") unit is split into
  // `splits` items, item s taking union entries [s*pps, (s+1)*pps); a tail
  // unit whose union needs more than one split writes fp32 partials
  // (rows_part rows per item), combined by a second kernel.
  // Splitting only the tail evens out the last round of work across the SMs.
  int whole_units;
  int tail_units;
  int splits;
  int pps;
  int rows_part;
  int num_items;
  float* part_o;        // (tail_units*splits, rows_part, 128)
  float* part_ml;       // (tail_units*splits, rows_part, 2)
  int* item_counter;    // items handed out beyond the first round; 0 at launch
  // Swapped-orientation prefill kernel only: per union position, the mask of
  // the tile's tokens that selected it (bit w = token w), and a q map whose
  // box is one token's G query heads, (64, G, 1).
  const uint32_t* block_members;
  CUtensorMap tmap_q1;
  // One-token tiles (tile_tokens == 1, topk <= 32) may skip the union
  // kernel: with `direct` set, the attention kernel's item setup filters,
  // sorts and deduplicates the token's own q2k row (every union entry is
  // then a member) and writes union_len, union_blocks and tile_info itself.
  const int32_t* q2k;
  int topk;
  int direct;
  // The preceding kernel only zeroes item_counter (launch_reset_counter, an
  // ordinary launch, so every other input was complete before it began): the
  // attention kernel waits for it only before its first claim from the
  // counter.
  int wait_late;
};
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);
// The swapped-orientation prefill kernel (bf16 / fp16 K/V, G a multiple of 8
// and at most 64, tile_tokens * G <= 256, tile_tokens <= 32, no splits).
cudaError_t launch_prefill_swapped(const PrefillArgs& a, cudaStream_t s);
int device_sm_count();
// Raises `kernel`'s dynamic shared-memory limit to at least `bytes` on the
// current device; the driver call is made once per (kernel, device, size).
cudaError_t set_smem_limit(const void* kernel, int bytes);
// The current device's per-block shared-memory limit (opt-in), cached.
int device_smem_optin();

struct ProxyArgs {
  unsigned* fault;      // device fault word (bounded-wait expiry, capacity)
  CUtensorMap tmap_q;   // (d, Hq, Tq) 16-bit, box (64, G, Wm)
  CUtensorMap tmap_k;   // flat (d, Hkv, Tk) / paged (d, 128, Hkv, pages), 128-key box of
                        // 128 bytes (64 16-bit values, or 128 E4M3 codes)
  const int32_t* cu_q;
  const int32_t* cu_k;        // flat lengths, or NULL when paged
  int paged;
  const int32_t* page_table;  // (B, max_pages), paged only
  int max_pages;
  int num_pages;
  const int32_t* seqused_k;   // (B), paged only
  int batch;
  int total_q;
  int num_qo_heads;
  int num_kv_heads;
  int max_k_tiles;
  int causal;
  int reduce_heads;
  int tile_tokens;      // tokens per M-tile (128 / G)
  int max_tiles;        // upper bound on query tiles of 2 M-tiles each
  int one_m;            // query tiles of tile_tokens tokens (one M tile), else 2 * tile_tokens
  int slice_cols;       // block columns per CTA: CTA (tile, s) takes [s, s + 1) * slice_cols
  int slices;           // column slices per tile
  float* out;
  int f16;              // q (and 16-bit K) are fp16, else bf16
  int k_fp8;            // K is E4M3, upconverted in the kernel to q's type
};
cudaError_t launch_proxy(const ProxyArgs& a, cudaStream_t s);

// Flat E4M3 K and V (n16 16-byte groups each) decoded to bf16 copies.
struct KvDecodeArgs {
  const void* k8 = nullptr;
  const void* v8 = nullptr;
  void* k16 = nullptr;
  void* v16 = nullptr;
  size_t n16 = 0;
};
cudaError_t launch_kv_decode(const KvDecodeArgs& a, cudaStream_t s);

// Paged E4M3 (mode 1: (pages, Hkv, 128, 128) bytes) or packed NVFP4 (mode 2:
// planar pages) K/V decoded into a bf16 pool of batch * max_pages pages, with
// the renumbered page table written to pt_out (batch, max_pages).
struct PageDecodeArgs {
  int mode = 0;  // 0: nothing to do
  const int32_t* page_table = nullptr;
  const int32_t* seqused_k = nullptr;
  int max_pages = 0, num_pages = 0, batch = 0, hkv = 0;
  const uint8_t* k8 = nullptr;
  const uint8_t* v8 = nullptr;
  const uint8_t* fp4_k = nullptr;
  const uint8_t* fp4_k_scale = nullptr;
  const uint8_t* fp4_v = nullptr;
  const uint8_t* fp4_v_scale = nullptr;
  long long fp4_page_stride = 0;
  uint16_t* k16 = nullptr;
  uint16_t* v16 = nullptr;
  int32_t* pt_out = nullptr;
};
cudaError_t launch_page_decode(const PageDecodeArgs& a, cudaStream_t s);

// Packed-NVFP4 paged decode: one work unit per (query token, KV head) whose
// G <= 16 query heads form the 16 rows of warp-level MMAs; each unit attends
// over its token's own selected blocks. A list launch writes the units' block
// lists; the decode launch splits the list positions evenly over its CTAs.
constexpr int kFp4DecodeMaxCtas = 1024;  // partial slots in the workspace
struct Fp4DecodeArgs {
  unsigned* fault = nullptr;
  CUtensorMap tmap_kc;  // K codes (64 bytes, 128, Hkv, pages), 64-byte swizzle, box (64, 128, 1, 1)
  CUtensorMap tmap_vc;  // V codes, the same
  const uint16_t* q = nullptr;  // bf16 (total_q, Hq, 128)
  const int32_t* q2k = nullptr;  // (Hkv, total_q, topk)
  int topk = 0;
  const int32_t* cu_q = nullptr;
  const int32_t* page_table = nullptr;
  int max_pages = 0, num_pages = 0;
  const int32_t* seqused_k = nullptr;
  const uint8_t* k_scale = nullptr;  // (page, head) slice at p * page_stride + h * 1024
  const uint8_t* v_scale = nullptr;
  long long page_stride = 0;
  int batch = 0, total_q = 0, num_qo_heads = 0, num_kv_heads = 0, G = 0;
  float scale_log2 = 0.f;  // softmax scale * log2(e) * K global scale
  float out_scale = 1.f;   // V global scale
  uint16_t* out = nullptr;  // bf16 (total_q, Hq, 128)
  float* lse = nullptr;     // (total_q, Hq) or NULL
  // workspace (place_fp4_decode_workspace)
  int2* list = nullptr;      // (units, topk) of (page, visible keys); page -1: none
  int32_t* arrive = nullptr;  // (units): segments of the unit finished
  float* part_ml = nullptr;  // (max CTAs, 2, 16, 2): a segment's (m, l) per row
  float* part_o = nullptr;   // (max CTAs, 2, 16, 128): a segment's unnormalised O
};
size_t fp4_decode_workspace_bytes(long long units, int topk);
void place_fp4_decode_workspace(Fp4DecodeArgs* a, uint8_t* ws, long long units, int topk);
cudaError_t launch_fp4_decode(const Fp4DecodeArgs& a, cudaStream_t s);

}  // namespace msa
