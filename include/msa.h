/*
 * libmsa — MiniMax Sparse Attention (MSA) forward for NVIDIA GB300 (sm_103a).
 *
 * C ABI. Every pointer argument marked "device" is a CUDA device pointer the
 * caller allocated and owns; the library allocates no memory, never
 * synchronises the host with the device, and enqueues all work on the
 * caller's stream. All tensors are dense and contiguous (row-major, last
 * dimension fastest) in the layouts stated below, which are those of the
 * FlashInfer MSA documentation pages ("flashinfer.msa_ops.msa_sparse_attention",
 * "flashinfer.msa_ops.msa_proxy_score", "prepare_msa_nvfp4_sparse_decode").
 *
 * Errors: every entry point validates its arguments on the host before any
 * launch and returns a status. Index values and cu_seqlens contents are caller
 * contracts and are never copied back to the host; kernels mask out-of-range
 * block ids and page ids instead of faulting. Device pointers must be 16-byte
 * aligned.
 *
 * Sizes used below: Tq = total_q, Tk = total_k, Hq = num_qo_heads,
 * Hkv = num_kv_heads, G = Hq / Hkv, d = head_dim (128), B = batch,
 * BLK = 128 (KV block = page size in tokens).
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MSA_OK = 0,
  MSA_INVALID_ARG = 1,          /* malformed or conflicting arguments */
  MSA_UNSUPPORTED = 2,          /* valid but not supported by this library (dtype, head_dim, sizes) */
  MSA_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below the size query's answer */
  MSA_CUDA_ERROR = 4            /* a CUDA runtime/driver call failed at launch */
} msa_status_t;

typedef enum { MSA_BF16 = 0, MSA_FP16 = 1, MSA_FP8_E4M3 = 2 } msa_dtype_t;

/* Human-readable name of a status code (static storage). */
const char* msa_status_string(msa_status_t status);

/*
 * Workspace bytes msa_sparse_attention_fwd needs for these sizes
 * ("msa_sparse_attention", workspace: caller-owned storage). paged != 0 when
 * K/V come with a page table. Returns 0 for sizes the forward would reject.
 */
size_t msa_sparse_attention_workspace_size(int batch, int total_q, int num_qo_heads,
                                           int num_kv_heads, int head_dim, int topk,
                                           int max_seqlen_q, int paged);

/*
 * Workspace bytes for the forward's fastest route with these K/V: the size
 * above, plus, for MSA_FP8_E4M3 K/V on a prefill-sized call, room for a bf16
 * copy of K and V:
 *   flat (paged == 0; total_k = key rows): when total_q * num_qo_heads >=
 *     total_k * num_kv_heads, 2 * 256-byte-rounded total_k * num_kv_heads *
 *     head_dim * 2 bytes;
 *   paged (paged != 0; total_k = max_pages, the page table's width): when
 *     total_q * num_qo_heads >= batch * max_pages * 128 * num_kv_heads, a bf16
 *     page pool of batch * max_pages pages for K and for V plus a renumbered
 *     page table (each 256-byte rounded).
 * Given that much, the forward decodes E4M3 into the copy with one HBM-bound
 * pass and runs the attention kernel on bf16 operands; given only the size
 * above, the attention kernel converts E4M3 itself (same results, slower on
 * tensor-bound calls). Equals the size above for every other case. Returns 0
 * where the size above does or total_k < 0.
 */
size_t msa_sparse_attention_workspace_size_kv(int batch, int total_q, int num_qo_heads,
                                              int num_kv_heads, int head_dim, int topk,
                                              int max_seqlen_q, int paged, msa_dtype_t kv_dtype,
                                              int total_k);

/*
 * Sparse attention forward ("flashinfer.msa_ops.msa_sparse_attention").
 *
 * Each query token t and query head h attends only to the keys of the 128-token
 * KV blocks listed in q2k_indices[h / G, t, :] (batch-local block ids,
 * ascending, -1 padded), with right-aligned causal masking when causal != 0
 * (query i of a sequence with Lq queries and Lk keys sits at key position
 * Lk - Lq + i) and query head h reading KV head h / G (GQA; "prepare_msa_nvfp4_
 * sparse_decode", q). The result equals per-query softmax attention over that
 * query's own blocks: out = softmax(scale * q k^T) v over the selected visible
 * keys; lse = natural log of the softmax normaliser. A row with no visible
 * selected key gets out = 0 and lse = -inf. Query tokens are processed in
 * tiles that each run one online softmax over the union of their tokens'
 * blocks; the union metadata is built into the workspace.
 *
 *   q            device, (Tq, Hq, d), q_dtype MSA_BF16 or MSA_FP16
 *   k, v         device; flat (Tk, Hkv, d) when page_table == NULL, else
 *                paged (num_pages, Hkv, BLK, d); kv_dtype: with bf16 q,
 *                MSA_BF16 or MSA_FP8_E4M3 (E4M3 "fn", decoded exactly to
 *                bf16: by a pass into the workspace when it holds
 *                msa_sparse_attention_workspace_size_kv(...) bytes, else in
 *                the attention kernel); with fp16 q, MSA_FP16
 *   q2k_indices  device int32 (Hkv, Tq, topk); 1 <= topk <= 64
 *   cu_seqlens_q device int32 (B+1), cumulative query lengths
 *   cu_seqlens_k device int32 (B+1) for flat K/V; must be NULL when paged
 *   page_table   device int32 (B, max_pages) mapping batch-local block -> page,
 *                or NULL for flat K/V; requires seqused_k
 *   seqused_k    device int32 (B), valid keys per sequence (paged only)
 *   max_seqlen_q host bound on every Lq; with the tile count it decides how
 *                the work is split: when there are fewer (tile, KV head) units
 *                than the GPU has room for (decode-sized problems), each
 *                tile's union list is split across several work items whose
 *                partial results are merged on the device
 *   softmax_scale  <= 0 selects head_dim^-0.5
 *   out          device, (Tq, Hq, d), dtype of q; fully written
 *   lse          device float32 (Tq, Hq) or NULL
 *   workspace    device scratch of at least
 *                msa_sparse_attention_workspace_size(...) bytes (or the
 *                larger msa_sparse_attention_workspace_size_kv(...), see
 *                there), 256-byte aligned; its contents need no
 *                initialisation, and calls that share one workspace must be
 *                ordered on the device.
 * Every route, decode-sized paged calls (seqlen_q <= 4) included, takes any
 * G = Hq / Hkv up to 128: a query tile holds floor(128 / G) tokens (at least
 * one), so a larger G only means fewer tokens per tile.
 * Returns MSA_INVALID_ARG when both or neither of cu_seqlens_k and page_table
 * are given (paged length comes only from seqused_k, per the page's rule of
 * declining two possibly disagreeing length sources), when Hq % Hkv != 0, or
 * when a pointer is NULL or misaligned; MSA_UNSUPPORTED for head_dim != 128,
 * G > 128, a dtype pair other than those above, or topk outside [1, 64].
 */
msa_status_t msa_sparse_attention_fwd(
    const void* q, msa_dtype_t q_dtype, const void* k, const void* v, msa_dtype_t kv_dtype,
    const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, const int32_t* page_table, int max_pages, int num_pages,
    const int32_t* seqused_k, int batch, int total_q, int total_k, int num_qo_heads,
    int num_kv_heads, int head_dim, int max_seqlen_q, int causal, float softmax_scale, void* out,
    float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Prepared forward: msa_sparse_attention_prepare takes exactly the arguments
 * of msa_sparse_attention_fwd (without the stream), checks them with the same
 * rules and statuses, and binds them: the work split, the workspace layout
 * and the TMA descriptors are decided once, on the host, with no device
 * access. msa_sparse_attention_run then launches that forward on `stream`
 * with no allocation, no host synchronisation and no argument processing;
 * it can be captured into a CUDA graph. The bound device buffers must stay
 * allocated while the plan is used; their contents may change between runs
 * (each run reads them afresh). A plan is host memory owned by the caller,
 * released with msa_sparse_attention_plan_free (NULL is accepted). (The
 * prepare / runner split follows the interface the pages give for
 * "prepare_msa_nvfp4_sparse_decode"; here it serves the bf16, fp16 and E4M3
 * routes of msa_sparse_attention_fwd.)
 */
typedef struct msa_attention_plan msa_attention_plan_t;
msa_status_t msa_sparse_attention_prepare(
    const void* q, msa_dtype_t q_dtype, const void* k, const void* v, msa_dtype_t kv_dtype,
    const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, const int32_t* page_table, int max_pages, int num_pages,
    const int32_t* seqused_k, int batch, int total_q, int total_k, int num_qo_heads,
    int num_kv_heads, int head_dim, int max_seqlen_q, int causal, float softmax_scale, void* out,
    float* lse, void* workspace, size_t workspace_bytes, msa_attention_plan_t** plan);
msa_status_t msa_sparse_attention_run(const msa_attention_plan_t* plan, cudaStream_t stream);
void msa_sparse_attention_plan_free(msa_attention_plan_t* plan);

/*
 * Packed NVFP4 paged K/V forward ("flashinfer.msa_ops.msa_sparse_attention":
 * the packed-NVFP4 paged route, parameters k, k_scale, v_scale,
 * k_global_scale, v_global_scale, page_table, seqused_k;
 * "prepare_msa_nvfp4_sparse_decode": k, k_scale, v_scale and the global
 * scales). Computes what msa_sparse_attention_fwd computes (causal, paged)
 * with K = e2m1 * block scale * k_global_scale and V = e2m1 * block scale *
 * v_global_scale:
 *   k, v          device uint8 views of a planar page pool: page p's slice for
 *                 KV head h starts at p * page_stride_bytes + h * 8192 and holds
 *                 128 tokens x 64 bytes of E2M1 pairs (element 2i in the low
 *                 nibble of byte i, 2i + 1 in the high nibble);
 *   k_scale,      device E4M3 block scales, one per 16 elements: (page, head)
 *   v_scale       slice at p * page_stride_bytes + h * 1024, 128 x 8 bytes; K
 *                 scales token-major (token t, scale s at 8 t + s), V scales in
 *                 4 x 4 (token, scale) tiles, row-major over tiles, each tile
 *                 scale-index major (t, s at 32 (t/4) + 16 (s/4) + 4 (s%4) +
 *                 t%4). The pages' planar page is [K data | K scales | V data
 *                 | V scales]; any stride multiple of 16 bytes is accepted;
 *   k_global_scale, v_global_scale  positive, finite; the K one folds into the
 *                 softmax scale, the V one into the output;
 *   q             bf16 only; other arguments as msa_sparse_attention_fwd with
 *                 cu_seqlens_k = NULL and causal = 1;
 *   workspace     at least msa_sparse_attention_workspace_size(..., paged = 1)
 *                 bytes. msa_sparse_attention_nvfp4_workspace_size adds, for
 *                 prefill-sized calls (total_q * num_qo_heads >= batch *
 *                 max_pages * 128 * num_kv_heads), a bf16 page pool and a
 *                 renumbered page table: given that much, the pages the batch
 *                 can read are decoded to bf16 once and the attention kernel
 *                 runs on bf16 operands. For decode-shaped calls (G <= 16 and
 *                 max_seqlen_q <= 16) it adds the per-(token, KV head) block
 *                 lists, one merge counter per unit and fixed partial slots
 *                 (about 17 MB): given that much, a decode kernel that
 *                 dequantizes K and V in registers runs. With only the plain
 *                 size the attention kernel decodes NVFP4 in-kernel (same
 *                 results within the stated tolerance; every route computes
 *                 S and O in fp32).
 * Unmapped pages (page id outside [0, num_pages)) are neither read nor used.
 * Returns MSA_INVALID_ARG for a NULL or misaligned pointer, a page stride not
 * a positive multiple of 16, or a global scale that is not positive and
 * finite; MSA_UNSUPPORTED for non-bf16 q; otherwise as the bf16 forward.
 * msa_sparse_attention_nvfp4_prepare binds the same call into a plan that
 * msa_sparse_attention_run launches (the pages' prepare / runner interface).
 */
size_t msa_sparse_attention_nvfp4_workspace_size(int batch, int total_q, int num_qo_heads,
                                                 int num_kv_heads, int head_dim, int topk,
                                                 int max_seqlen_q, int max_pages);
msa_status_t msa_sparse_attention_nvfp4_paged(
    const void* q, msa_dtype_t q_dtype, const void* k, const void* k_scale, const void* v,
    const void* v_scale, long long page_stride_bytes, float k_global_scale,
    float v_global_scale, const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
    const int32_t* page_table, int max_pages, int num_pages, const int32_t* seqused_k,
    int batch, int total_q, int num_qo_heads, int num_kv_heads, int head_dim,
    int max_seqlen_q, float softmax_scale, void* out, float* lse, void* workspace,
    size_t workspace_bytes, cudaStream_t stream);
msa_status_t msa_sparse_attention_nvfp4_prepare(
    const void* q, msa_dtype_t q_dtype, const void* k, const void* k_scale, const void* v,
    const void* v_scale, long long page_stride_bytes, float k_global_scale,
    float v_global_scale, const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
    const int32_t* page_table, int max_pages, int num_pages, const int32_t* seqused_k,
    int batch, int total_q, int num_qo_heads, int num_kv_heads, int head_dim,
    int max_seqlen_q, float softmax_scale, void* out, float* lse, void* workspace,
    size_t workspace_bytes, msa_attention_plan_t** plan);

/*
 * Dense proxy pass, MSA stage 1 ("flashinfer.msa_ops.msa_proxy_score").
 *
 * output[h, t, q] = max over the keys j of KV block t of the UNSCALED logit
 * <q[q, h, :], k[j, h / G, :]>, with j < Lk and, when causal, j <= Lk - Lq + i
 * (right-aligned, applied before the max); -inf when block t holds no such key
 * (beyond the sequence or wholly above the causal limit). With
 * reduce_heads != 0 the max is also taken over all query heads and the output
 * has one head.
 *
 *   q            device, (Tq, Hq, 128), MSA_BF16 or MSA_FP16
 *   k            device, q's dtype or MSA_FP8_E4M3 (E4M3 "fn", upconverted
 *                exactly to q's type in the kernel); flat (Tk, Hkv, 128) when
 *                page_table is NULL, else a paged pool (num_pages, Hkv, 128,
 *                128) of k's element size
 *   cu_seqlens_q device int32 (B+1)
 *   cu_seqlens_k device int32 (B+1) for flat K; must be NULL when paged
 *   page_table   device int32 (B, max_pages) mapping batch-local block ->
 *                page, or NULL for flat K; requires seqused_k. A block whose
 *                entry is negative or >= num_pages holds no key (-inf).
 *   seqused_k    device int32 (B), keys per sequence (paged only)
 *   total_k      keys in flat K, or num_pages, the pool's page count, when paged
 *   max_seqlen_q host bound on every Lq, or 0 when unknown; a bound <= 128/G
 *                lets query tiles hold one M=128 tile instead of two
 *   max_k_tiles  number of block columns; blocks >= ceil(Lk/128) read -inf
 *   output       device float32 (reduce_heads ? 1 : Hq, max_k_tiles, Tq),
 *                query fastest; fully written
 * Decode-sized calls (few query tiles over long contexts) split each tile's
 * block columns across many CTAs; a block's max needs no merge.
 * Returns MSA_INVALID_ARG when both or neither of cu_seqlens_k and
 * page_table are given, when a paged call lacks seqused_k or max_pages, or as
 * for msa_sparse_attention_fwd; MSA_UNSUPPORTED for head_dim != 128, another
 * dtype pair (e.g. bf16 q with fp16 K), or reduce_heads with G = Hq / Hkv not
 * a power of two <= 32.
 */
msa_status_t msa_proxy_score(const void* q, msa_dtype_t q_dtype, const void* k,
                             msa_dtype_t k_dtype, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_k, const int32_t* page_table, int max_pages,
                             const int32_t* seqused_k, int batch, int total_q, int total_k,
                             int num_qo_heads, int num_kv_heads, int head_dim, int max_seqlen_q,
                             int max_k_tiles, int causal, int reduce_heads, float* output,
                             cudaStream_t stream);

/*
 * Top-k block selection from proxy scores (the consumer named by
 * "msa_proxy_score", Returns; output contract of q2k_indices in
 * "msa_sparse_attention" and "prepare_msa_nvfp4_sparse_decode").
 *
 * For each query q, the topk largest scores among its max_k_tiles columns;
 * equal scores go to the lower block id; -inf and NaN are never chosen. The
 * chosen ids are written ascending and -1 padded.
 *
 *   scores       device float32 (num_score_heads, max_k_tiles, Tq)
 *   num_score_heads  1 (broadcast to all num_kv_heads_out heads) or
 *                num_kv_heads_out (one selection per head)
 *   q2k_indices  device int32 (num_kv_heads_out, Tq, topk); 1 <= topk <= 64
 */
msa_status_t msa_topk_select(const float* scores, int num_score_heads, int max_k_tiles,
                             int total_q, int topk, int num_kv_heads_out, int32_t* q2k_indices,
                             cudaStream_t stream);

/*
 * Query-tile union metadata ("msa_sparse_attention": "the union metadata is
 * built internally from q2k_indices"), exported so it can be checked on its
 * own. Tiles are tile_tokens consecutive queries of one sequence, numbered in
 * sequence order; tile tau of KV head h:
 *   union_len[h, tau]              number of distinct usable ids
 *   union_blocks[h, tau, 0:cap]    those ids ascending, -1 filled
 *   member[h, tau, w, 0:words]     bit j set iff union_blocks[h, tau, j] is in
 *                                  the row of the tile's token w
 *   tile_info[tau, 0:2]            (first packed query row, sequence), or
 *                                  (-1, -1) past the last tile; may be NULL
 * with cap = tile_tokens * topk and words = ceil(cap / 32). An id is usable for
 * a token iff 0 <= id < ceil(Lk/128) (and id < max_pages when paged) and, when
 * causal, its block holds a key at or before the token's position. Rows past a
 * sequence end are zero. Arrays are sized for max_tiles tiles, which must be
 * at least the number of tiles, sum_b ceil(Lq_b / tile_tokens); tiles past
 * the last get length 0.
 *   cu_seqlens_k (flat) or seqused_k (paged): exactly one is non-NULL.
 * tile_tokens must lie in [1, 128].
 */
msa_status_t msa_build_union(const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_k, const int32_t* seqused_k, int max_pages,
                             int batch, int total_q, int num_kv_heads, int causal, int tile_tokens,
                             int max_tiles, int32_t* union_len, int32_t* union_blocks,
                             uint32_t* member, int32_t* tile_info, cudaStream_t stream);

/* Tokens per query tile for Hq/Hkv: floor(128 / G), at least 1. The forward
 * uses min(this, max_seqlen_q), which forms the same tiles (tiles never span
 * sequences). */
int msa_union_tile_tokens(int num_qo_heads, int num_kv_heads);

/*
 * msa_build_union with one more output, for tile_tokens <= 32:
 *   block_members[h, tau, 0:cap]   device uint32; bit w set iff the tile's
 *                                  token w has union_blocks[h, tau, j] usable
 *                                  in its row (the member bits transposed);
 *                                  0 past union_len
 * This is the union metadata of the forward's swapped-orientation kernel
 * (see msa_prefill_tile_tokens), which walks each union block's member
 * tokens. Same arguments and errors as msa_build_union otherwise;
 * tile_tokens > 32 or a NULL block_members is MSA_INVALID_ARG.
 */
msa_status_t msa_build_union_block_members(
    const int32_t* q2k_indices, int topk, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, const int32_t* seqused_k, int max_pages, int batch, int total_q,
    int num_kv_heads, int causal, int tile_tokens, int max_tiles, int32_t* union_len,
    int32_t* union_blocks, uint32_t* member, uint32_t* block_members, int32_t* tile_info,
    cudaStream_t stream);

/*
 * Tokens per query tile of the attention kernel msa_sparse_attention_fwd
 * uses for these sizes and K/V dtype under the current route (see
 * msa_set_prefill_route; an E4M3 call on its bf16-copy route counts as
 * MSA_BF16). Two kernels compute the same result:
 *   - the union-tile kernel: floor(128 / G) tokens per tile (128 rows = one
 *     MMA tile), each tile's rows walking its whole union; every call by
 *     default;
 *   - the swapped-orientation kernel: min(32, 256 / G) tokens per tile, the
 *     MMAs' N being only the member rows of each union block; 16-bit K/V and
 *     G a multiple of 8 up to 64, when route 2 is set.
 * Both are capped at max_seqlen_q. Returns 0 for invalid sizes.
 */
int msa_prefill_tile_tokens(int batch, int total_q, int num_qo_heads, int num_kv_heads, int topk,
                            int max_seqlen_q, msa_dtype_t kv_dtype);

/*
 * Testing and benchmarking: which attention kernel later forward calls use.
 * 0 (the default) the faster one as measured (at present the union-tile
 * kernel everywhere); 1 always the union-tile kernel; 2 the
 * swapped-orientation kernel wherever it applies (16-bit K/V, G a multiple
 * of 8 up to 64). Process-wide, not thread-safe. Other values:
 * MSA_INVALID_ARG.
 */
msa_status_t msa_set_prefill_route(int route);

/*
 * Waits for `stream`, then returns and clears the library's device fault word
 * of the current device in *fault (0 = none). Kernels never trap: a wait that
 * exceeds its time limit (2 s), or an internal capacity check, sets a bit here
 * and the kernel unwinds and returns. Bits: 1 a TMA copy never landed, 2 an
 * MMA completion never came, 4 the softmax warps never released a buffer,
 * 8 a capacity check failed, 16 another wait expired. Synchronises the host:
 * for tests and diagnostics.
 */
msa_status_t msa_read_device_fault(unsigned int* fault, cudaStream_t stream);

/*
 * Diagnostics: launches one CTA that waits, with a limit of timeout_us
 * microseconds (1 .. 1000000), on a barrier nothing arrives at. The wait
 * expires, fault bit 16 is set, and the kernel returns: the same path every
 * bounded wait of the library takes instead of hanging.
 */
msa_status_t msa_selftest_wait_timeout(unsigned int timeout_us, cudaStream_t stream);

/*
 * Paged decode for callers that cannot allocate device memory (no counterpart
 * on the documentation pages; it is an addition of this library).
 *
 * Engines that plan all device memory ahead of time, plugin interfaces that
 * give a kernel no workspace, and code running where cudaMalloc may not be
 * called cannot provide the workspace msa_sparse_attention_fwd needs. This
 * entry point is msa_sparse_attention_fwd for a paged call with bf16 q and
 * K/V (arguments as there; same kernels, same result bits), with the
 * workspace taken from a fixed 16 MiB array inside the library's device
 * image, which every GPU that loads the library holds until the process
 * exits. It allocates nothing. Calls whose workspace
 * (msa_sparse_attention_workspace_size with paged = 1) exceeds the array are
 * rejected with MSA_WORKSPACE_TOO_SMALL before anything is launched;
 * msa_sparse_decode_noalloc_scratch_limit() returns the array size.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it for the life of the process; make that first
 * call before any stream capture, and do not use the library across a
 * cudaDeviceReset of that device (the cached address would be stale). All calls share the one array and it keeps the previous call's
 * contents (the forward needs no initialised workspace); calls whose work
 * overlaps on the GPU race on the array, so callers must order them.
 */
msa_status_t msa_sparse_decode_noalloc(
    const void* q, const void* k, const void* v, const int32_t* q2k_indices, int topk,
    const int32_t* cu_seqlens_q, const int32_t* page_table, int max_pages, int num_pages,
    const int32_t* seqused_k, int batch, int total_q, int num_qo_heads, int num_kv_heads,
    int head_dim, int max_seqlen_q, int causal, float softmax_scale, void* out, float* lse,
    cudaStream_t stream);
size_t msa_sparse_decode_noalloc_scratch_limit(void);

/*
 * Diagnostics: timing events for msa_sparse_attention_fwd. When `events`
 * points to three cudaEvent_t handles (count == 3), every later forward call
 * records events[0] before its first launch, events[1] after the metadata
 * step (union kernel, or the decode ticket reset) and events[2] after the
 * attention kernel, all on the call's stream. count == 0 turns it off. The
 * handles are owned by the caller and must outlive their use. Not
 * thread-safe; meant for benchmarks.
 */
msa_status_t msa_set_timing_events(void* const* events, int count);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* MSA_H_ */
