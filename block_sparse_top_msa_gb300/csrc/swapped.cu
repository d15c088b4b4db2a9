// MSA sparse attention prefill for sm_103a in the swapped orientation
// ("flashinfer.msa_ops.msa_sparse_attention": each query attends only the
// top-K KV blocks selected in q2k_indices; query tokens are processed in
// tiles, each running one online softmax over the union of its tokens'
// blocks. "prepare_msa_nvfp4_sparse_decode" describes running both MMAs of
// its decode kernel in a swapped orientation, keys as the MMA's M).
//
// Why this kernel exists: with randomly chosen blocks, a query tile's union
// is several times longer than any one token's selection, so an M=128 row
// tile over the union computes mostly masked products. Here the roles are
// swapped: for each union block, the MMA's M is the block's 128 keys (QK) or
// the 128 head dimensions (PV), and N is only the query rows that selected
// the block (member rows, gathered), 16 to 64 per MMA. The MMA work then
// follows the member rows, and a tile holds more tokens (32 x 8 heads = 256
// rows), so each K/V block brought in from L2 serves more rows.
//
// Work item: a query tile of W tokens (W * G <= 256 rows, row r = token
// r / G, head r % G of the KV head's group) and a KV head. Its stream of
// chunks: per union block with member tokens M_u, chunks of at most 64
// member rows. Roles:
//   K / V warps  : TMA the block's K and V tiles into two-slot rings (flat
//                  rows cu_k[b] + 128 id, or page page_table[b, id]); the K
//                  warp also hands out the work items;
//   Q warp       : walks the chunk stream, publishes each chunk's record
//                  and column table (row and key limit per column) in
//                  shared memory, and TMA-gathers the member tokens' G query
//                  rows into a K-major buffer QB (N = 16 * ceil(rows / 16));
//   MMA warp     : follows the records; each step issues S^T = K_u QB^T of
//                  chunk g + 2 (M = 128 keys, fp32 in TMEM) and D = V_u^T P
//                  of chunk g (M = 128 dims, A and B MN-major) with their K
//                  steps interleaved;
//   softmax warps: two teams of four (one warp per key quarter = TMEM lane
//                  quarter) take alternate chunks: mask keys past each
//                  column's limit, column maxima by shuffle transposes and an
//                  exchange across the quarters, the running max per row
//                  (updated in chunk order, handed between the teams per
//                  quarter; O rescaled lazily, only when the max grows by
//                  more than 2^8), P = 2^(s * scale * log2 e - m) written
//                  as bf16 / fp16 over QB, and per-quarter column sums;
//   merge warps  : thread = head dimension; O^T[:, row] = alpha * O^T[:, row]
//                  + D[:, column] for each member row and l[row] = alpha *
//                  l[row] + column sum, O^T (d x 256 rows, fp32) resident in
//                  TMEM for the whole item; at the end of the item out = O / l
//                  and the natural-log LSE.
// Rows whose token did not select a block get nothing from it, so each
// row's result is exactly its own blocks' softmax attention.
//
// Measured on the flat varlen prefill (2 x 32768, 64/8 heads, top-16) it
// takes 24 ms against 17.9 ms for the union-tile kernel (prefill.cu): per
// chunk of about 32 member rows the softmax team needs about 3400 cycles
// from S^T to P, and with QK two chunks ahead that latency sets the pace,
// although the MMAs and the K/V loads per chunk would take about a third of
// it. The forward therefore runs the union-tile kernel unless route 2 is
// chosen (msa_set_prefill_route).
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tmem_wide.cuh"

namespace msa {
namespace {

constexpr int kSwBuf = 4;          // S/D TMEM buffers and QB/P buffers (chunk g uses g % 4)
constexpr int kSwItems = 8;        // work items handed from the K warp to the other roles
constexpr int kSwClaimAhead = 4;   // the K warp claims its next item this many blocks early
constexpr int kChunkN = 64;        // member rows per chunk (MMA N <= 64)
constexpr uint32_t kColS = 256;    // first TMEM column of the S/D buffers (O^T: 0..255)
constexpr int kHalfQB = kChunkN * 128;  // one 64-column half of a QB/P buffer
constexpr float kSwRescale = 8.0f;
constexpr int kColSlots = 8;       // column tables (chunk g uses g % 8; read until merge(g))

// Warp roles.
constexpr int kSmWarps = 8;        // softmax: key quarter q = warp & 3, team warp >> 2
constexpr int kMergeWarp0 = 8;     // four merge warps (quarter = warp & 3)
constexpr int kKWarp = 12;         // K loads; claims and publishes the work items
constexpr int kVWarp = 13;         // V loads
constexpr int kQWarp = 14;         // member-row Q gathers
constexpr int kMmaWarp = 15;
constexpr int kSwWarps = 16;
constexpr int kSwThreads = kSwWarps * 32;
// Readers of the item ring: the merge, V and Q warps (the MMA and softmax
// warps follow the Q warp's chunk records instead).
constexpr int kSwItemReaders = 4 + 1 + 1;

struct SwItem {
  int tile, h, t0, b, n_union, seq_q0, lq, lk, kv0;
};

// One chunk of the CTA's stream, published by the Q warp in slot g % 8 with
// its column table (and completed with qb_full): the MMA width N, member
// tokens, the block ordinal j, flags and the ordinal of its item among the
// CTA's non-empty items.
constexpr int kRecFirst = 1;      // first chunk of its block
constexpr int kRecLast = 2;       // last chunk of its block
constexpr int kRecItemEnd = 4;    // last chunk of its item
constexpr int kRecStreamEnd = 8;  // no chunk: the stream has ended
struct ChunkRec {
  int N, ntok, j, flags, item;
};

struct __align__(1024) SwSmem {
  uint8_t kv[4][2][16384];              // K slots 0, 1 and V slots 2, 3 (two 64-column halves)
  uint8_t qb[kSwBuf][2][kHalfQB];       // gathered Q rows, then P (K-major, 128-byte swizzle)
  // Running max per tile row (log2 units), one copy per key quarter: each
  // quarter's two warps (one per team) read and write only their own, in
  // chunk order (state_done). The running sum l lives with the merge warps.
  float m_ref[4][256];
  float l_row[256];
  float alpha[kSwBuf][kChunkN];         // rescale factor per chunk column, for the merge
  float psum[kSwBuf][4][kChunkN];       // per key quarter column sums of P, for the merge
  float xch[2][2][2][4][32];            // [team][slot][pass][quarter][lane]: column maxima
  float bc_off[kSmWarps][kChunkN];      // per-warp broadcast of the column offsets
  // Per chunk (slot g % 8), written by the Q warp: each column's tile row
  // (-1 past the member rows) and last visible key relative to the block's
  // first (127: none masked; -1: an unmapped page).
  int col_row[kColSlots][kChunkN];
  int col_rel[kColSlots][kChunkN];
  ChunkRec rec[kColSlots];
  float inv_l[256];
  uint64_t kv_full[4], kv_empty[4];
  uint64_t qb_full[kSwBuf], qb_free[kSwBuf];
  uint64_t qk_done[kSwBuf], p_full[kSwBuf], pv_done[kSwBuf], d_free[kSwBuf];
  uint64_t state_free;
  uint64_t state_done[4];               // per key quarter: the row max of chunk g is written
  uint64_t drain;
  uint64_t item_full[kSwItems], item_empty[kSwItems];
  int item_idx[kSwItems];
  SwItem item_ring[kSwItems];
  uint32_t tmem_base;
  int abort;
};

MSA_DEV float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Named barrier `id` over `n` threads; returns the AND of p over them.
MSA_DEV bool bar_and(int id, int n, bool p) {
  int r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.s32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\tselp.s32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((int)p), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Bit position of the s-th (from 0) set bit of m.
MSA_DEV int nth_set_bit(uint32_t m, int s) {
  for (int i = 0; i < s; ++i) m &= m - 1u;
  return __ffs(m) - 1;
}

// Column reduction over the warp's 32 lanes (keys): on entry every lane
// holds its values of C columns; on exit lane j holds the reduction of
// column j & (C - 1) over all 32 lanes. Butterfly transpose: at each stage
// a lane keeps one half of its columns and trades the other half with its
// partner, so the values per lane halve while the lanes covered double.
template <int C, bool MAX>
MSA_DEV float lane_reduce(float (&v)[C], int lane) {
#pragma unroll
  for (int o = C / 2; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = C; o < 32; o <<= 1) {
    const float x = __shfl_xor_sync(0xffffffffu, r, o);
    r = MAX ? fmaxf(r, x) : r + x;
  }
  return r;
}

// Zeroes 32 columns of this warp's lane quarter.
MSA_DEV void tmem_zero32(uint32_t taddr) {
  const uint32_t z = 0u;
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, "
      "%1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1, %1};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(z)
      : "memory");
}

template <int C>
MSA_DEV void tmem_ld_cols(uint32_t taddr, float (&v)[C]) {
  if constexpr (C == 8) tmem_ld8(taddr, v);
  else if constexpr (C == 16) tmem_ld16(taddr, v);
  else tmem_ld32(taddr, v);
}

MSA_DEV SwItem sw_item_at(const PrefillArgs& a, int i) {
  SwItem it;
  // Head-major: all tiles of one KV head (later, heavier tiles first) before
  // the next head, so the items in flight share one head's K/V in L2.
  it.h = i / a.max_tiles;
  it.tile = a.max_tiles - 1 - (i - it.h * a.max_tiles);
  const int2 ti = __ldg(reinterpret_cast<const int2*>(a.tile_info) + it.tile);
  it.t0 = ti.x;
  it.b = ti.y;
  it.n_union = 0;
  it.seq_q0 = it.lq = it.lk = it.kv0 = 0;
  if (it.t0 >= 0) {
    it.n_union = __ldg(a.union_len + (size_t)it.h * a.max_tiles + it.tile);
    it.seq_q0 = __ldg(a.cu_q + it.b);
    it.lq = __ldg(a.cu_q + it.b + 1) - it.seq_q0;
    if (a.paged) {
      it.lk = __ldg(a.seqused_k + it.b);
    } else {
      it.kv0 = __ldg(a.cu_k + it.b);
      it.lk = __ldg(a.cu_k + it.b + 1) - it.kv0;
    }
  }
  return it;
}

// Walks an item's chunks: union blocks with at least one member token, each
// split into chunks of at most `tpc` member tokens (lowest tokens first).
// g counts chunks and j counts blocks over the CTA's whole stream. Called
// by all 32 lanes of a warp: the union list is read 32 blocks at a time,
// one block per lane, and handed out by shuffles.
struct Chunks {
  const uint32_t* bm;
  const int32_t* ul;
  int n_union, u, wbase;
  uint32_t w_bm;   // this lane's block of the current window
  int w_ul;
  uint32_t rest;  // members of block u not yet in a chunk
  uint32_t cm;    // the current chunk's member tokens
  int ntok, N, blk;
  bool first, last;
  int g, j;
};

MSA_DEV void chunks_item(Chunks& c, const PrefillArgs& a, const SwItem& it) {
  const size_t unit = (size_t)it.h * a.max_tiles + it.tile;
  c.bm = a.block_members + unit * a.cap;
  c.ul = a.union_blocks + unit * a.cap;
  c.n_union = it.n_union;
  c.u = -1;
  c.wbase = -32;
  c.rest = 0u;
}

MSA_DEV bool chunks_next(Chunks& c, int tpc, int G) {
  c.first = false;
  while (c.rest == 0u) {
    if (++c.u >= c.n_union) return false;
    if (c.u >= c.wbase + 32) {
      c.wbase = c.u;
      const int v = c.u + (int)(threadIdx.x & 31);
      c.w_bm = v < c.n_union ? __ldg(c.bm + v) : 0u;
      c.w_ul = v < c.n_union ? __ldg(c.ul + v) : 0;
    }
    c.rest = __shfl_sync(0xffffffffu, c.w_bm, c.u - c.wbase);
    if (c.rest != 0u) {
      c.blk = __shfl_sync(0xffffffffu, c.w_ul, c.u - c.wbase);
      c.first = true;
      ++c.j;
    }
  }
  uint32_t m = c.rest, cm = 0u;
  for (int i = 0; i < tpc && m != 0u; ++i) {
    const uint32_t low = m & (0u - m);
    cm |= low;
    m ^= low;
  }
  c.rest = m;
  c.cm = cm;
  c.ntok = __popc(cm);
  c.N = ((c.ntok * G + 15) / 16) * 16;
  c.last = m == 0u;
  ++c.g;
  return true;
}

// Per-thread context of the softmax warps.
struct SmCtx {
  uint32_t lane_base;  // TMEM address of this warp's lane quarter, column 0
  int q4, team, warp, lane;
  float scale_log2;
};

// Phase 1 of one pass over C (16 or 32) columns col0 .. col0 + C - 1 of a
// chunk: load S^T, mask keys past each column's limit, and return this
// lane's column maximum over the warp's 32 keys (lane j: column col0 + j).
template <int C>
MSA_DEV void load_masked(const SwSmem& sm, const SmCtx& x, int buf, int ts, int col0, float (&s)[C]) {
  tmem_ld_cols<C>(x.lane_base + kColS + (uint32_t)(buf * 64 + col0), s);
  const int my_rel = sm.col_rel[ts][col0 + (x.lane & (C - 1))];
  if (__any_sync(0xffffffffu, my_rel < 127)) {
    const int key = x.q4 * 32 + x.lane;
#pragma unroll
    for (int i = 0; i < C; i += 4) {
      const int4 r4 = *reinterpret_cast<const int4*>(&sm.col_rel[ts][col0 + i]);
      if (key > r4.x) s[i] = -INFINITY;
      if (key > r4.y) s[i + 1] = -INFINITY;
      if (key > r4.z) s[i + 2] = -INFINITY;
      if (key > r4.w) s[i + 3] = -INFINITY;
    }
  }
}

template <int C>
MSA_DEV float pass_max(const SwSmem& sm, const SmCtx& x, int buf, int ts, int col0, float (&s)[C]) {
  load_masked<C>(sm, x, buf, ts, col0, s);
  float t[C];
#pragma unroll
  for (int i = 0; i < C; ++i) t[i] = s[i];
  return lane_reduce<C, true>(t, x.lane);
}

// Phase 3 of one pass: P = 2^(s * scale_log2 - offset) for the pass's
// columns, stored MN-major over the chunk's QB buffer (the PV's B operand:
// key k's 64 columns form one 128-byte row, rows of 8 keys 1 KB apart,
// 16-byte chunk c at position c ^ (k % 8)), and this quarter's column sums.
template <int C, bool F16>
MSA_DEV void pass_exp(SwSmem& sm, const SmCtx& x, int buf, int col0, const float (&s)[C]) {
  const int key = x.q4 * 32 + x.lane;
  uint8_t* prow = &sm.qb[buf][0][0] + (key >> 3) * 1024 + (key & 7) * 128;
  float p[C];
#pragma unroll
  for (int i = 0; i < C; i += 8) {
    const float4 o0 = *reinterpret_cast<const float4*>(&sm.bc_off[x.warp][col0 + i]);
    const float4 o1 = *reinterpret_cast<const float4*>(&sm.bc_off[x.warp][col0 + i + 4]);
    const float oo[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
    uint32_t pk[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      p[i + e] = ex2f(fmaf(s[i + e], x.scale_log2, -oo[e]));
      p[i + e + 1] = ex2f(fmaf(s[i + e + 1], x.scale_log2, -oo[e + 1]));
      pk[e >> 1] = pack_x2<F16>(p[i + e], p[i + e + 1]);
    }
    const int c16 = (col0 + i) >> 3;
    *reinterpret_cast<uint4*>(prow + ((c16 ^ (key & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  const float sum = lane_reduce<C, false>(p, x.lane);
  if (x.lane < C) sm.psum[buf][x.q4][col0 + x.lane] = sum;
}

// Phase 2 for the pass's columns: the running max of each column's row
// (lazy: it moves only when it grows by more than 2^8), the factor alpha
// that rescales the row's O and l, and the offset of this chunk's P
// (broadcast to the warp through bc_off). Quarter 0 hands alpha to the merge.
template <int C>
MSA_DEV void pass_state(SwSmem& sm, const SmCtx& x, int buf, int ts, int col0, int nvalid,
                        float mx) {
  const int n = col0 + x.lane;
  float off = INFINITY;
  if (x.lane < C && n < nvalid) {
    const int row = sm.col_row[ts][n];
    const float m_old = sm.m_ref[x.q4][row];
    float m_new = m_old;
    if (mx != -INFINITY) {
      const float ms = mx * x.scale_log2;
      if (m_old == -INFINITY || ms > m_old + kSwRescale) m_new = ms;
    }
    off = m_new == -INFINITY ? 0.f : m_new;
    sm.m_ref[x.q4][row] = m_new;
    if (x.q4 == 0) sm.alpha[buf][n] = m_old == -INFINITY ? 0.f : ex2f(m_old - m_new);
  }
  if (x.lane < C) sm.bc_off[x.warp][n] = off;
}

template <bool F16>
__global__ void __launch_bounds__(kSwThreads, 1)
    prefill_swapped_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  {
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (pad + sizeof(SwSmem) > dyn) {
      if (threadIdx.x == 0) atomicOr(a.fault, (unsigned)kFaultCapacity);
      return;
    }
  }
  SwSmem& sm = *reinterpret_cast<SwSmem*>(smem_raw + pad);
  unsigned* fault = a.fault;
  volatile int* abort = &sm.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.num_qo_heads / a.num_kv_heads;
  const int W = a.tile_tokens;
  const int tpc = kChunkN / G;  // member tokens per chunk

  auto read_item = [&](int n, bool& okr, SwItem& it) -> int {
    const int slot = n % kSwItems;
    if (!mbar_wait_sleep(&sm.item_full[slot], (n / kSwItems) & 1, fault, kFaultWaitOther, abort)) {
      okr = false;
      return -1;
    }
    const int idx = *reinterpret_cast<volatile int*>(&sm.item_idx[slot]);
    if (idx >= 0) it = sm.item_ring[slot];
    return idx;
  };
  auto release_item = [&](int n) { mbar_arrive(&sm.item_empty[n % kSwItems]); };

  if (tid == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int s = 0; s < kSwBuf; ++s) {
      mbar_init(&sm.qb_full[s], 1);
      mbar_init(&sm.qb_free[s], 1);
      mbar_init(&sm.qk_done[s], 1);
      mbar_init(&sm.p_full[s], 4);  // the four warps of the chunk's team
      mbar_init(&sm.pv_done[s], 1);
      mbar_init(&sm.d_free[s], 4);
    }
    mbar_init(&sm.state_free, 4);
    for (int q = 0; q < 4; ++q) mbar_init(&sm.state_done[q], 1);
    mbar_init(&sm.drain, 1);
    for (int s = 0; s < kSwItems; ++s) {
      mbar_init(&sm.item_full[s], 1);
      mbar_init(&sm.item_empty[s], kSwItemReaders);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < 256; i += kSwThreads) {
#pragma unroll
    for (int q = 0; q < 4; ++q) sm.m_ref[q][i] = -INFINITY;
    sm.l_row[i] = 0.f;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  grid_dependency_wait();
  grid_dependents_launch();

  if (warp == kKWarp || warp == kVWarp) {
    // ------------------------------------------------------------ K / V loads
    if (lane == 0) {
      const bool kw = warp == kKWarp;
      tma_prefetch_desc(kw ? (const void*)&a.tmap_k : (const void*)&a.tmap_v);
      int last_j = -1;  // last block loaded (it and the one before are drained on abort)
      bool ok = true;
      int j = -1;
      int claim = blockIdx.x;
      for (int ni = 0; ok; ++ni) {
        SwItem it{};
        int i = -1;
        if (kw) {
          // Hand out the work: the first item is blockIdx.x, later ones come
          // from the launch-wide counter, claimed kSwClaimAhead blocks before
          // the current item's end (faster SMs take more items).
          while (claim < a.num_items) {
            it = sw_item_at(a, claim);
            if (it.t0 >= 0) {
              i = claim;
              break;
            }
            claim = (int)gridDim.x + atomicAdd(a.item_counter, 1);
          }
          const int slot = ni % kSwItems;
          if (ni >= kSwItems && !mbar_wait_sleep(&sm.item_empty[slot], ((ni / kSwItems) - 1) & 1, fault,
                                           kFaultWaitOther, abort)) {
            ok = false;
            break;
          }
          sm.item_idx[slot] = i;
          if (i >= 0) sm.item_ring[slot] = it;
          mbar_arrive(&sm.item_full[slot]);
          if (i < 0) break;
          if (it.n_union <= kSwClaimAhead) claim = (int)gridDim.x + atomicAdd(a.item_counter, 1);
        } else {
          i = read_item(ni, ok, it);
          if (!ok) break;
          release_item(ni);
          if (i < 0) break;
        }
        const size_t unit = (size_t)it.h * a.max_tiles + it.tile;
        const uint32_t* bm = a.block_members + unit * a.cap;
        const int32_t* ul = a.union_blocks + unit * a.cap;
        for (int u = 0; u < it.n_union; ++u) {
          if (kw && it.n_union > kSwClaimAhead && u == it.n_union - kSwClaimAhead)
            claim = (int)gridDim.x + atomicAdd(a.item_counter, 1);
          if (__ldg(bm + u) == 0u) continue;  // no member: not a block of the stream
          ++j;
          const int blk = __ldg(ul + u);
          const int s = (kw ? 0 : 2) + (j & 1);
          if (j >= 2 && !mbar_wait_sleep(&sm.kv_empty[s], ((j >> 1) - 1) & 1, fault, kFaultWaitMma, abort)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&sm.kv_full[s], 2u * 16384u);
          const CUtensorMap* map = kw ? &a.tmap_k : &a.tmap_v;
          if (a.paged) {
            int page = __ldg(a.page_table + (size_t)it.b * a.max_pages + blk);
            // An unmapped page reads as zeros (out-of-range box) and is masked.
            if (page < 0 || page >= a.num_pages) page = a.num_pages;
            for (int c = 0; c < 2; ++c) tma_load_4d(sm.kv[s][c], map, &sm.kv_full[s], c * 64, 0, it.h, page);
          } else {
            const int row = it.kv0 + blk * kBlk;
            for (int c = 0; c < 2; ++c) tma_load_3d(sm.kv[s][c], map, &sm.kv_full[s], c * 64, it.h, row);
          }
          last_j = j;
        }
      }
      if (!ok) {
        for (int jj = last_j - 1; jj <= last_j; ++jj)
          if (jj >= 0)
            mbar_wait_sleep(&sm.kv_full[(kw ? 0 : 2) + (jj & 1)], (jj >> 1) & 1, fault, kFaultWaitTma);
      }
    }
  } else if (warp == kQWarp) {
    // ------------------------------------------------------------ Q gathers
    // Walks the chunk stream and publishes each chunk: its record and column
    // table (the whole warp; lane j fills columns j and j + 32), and, from
    // lane 0, the gathers of the member tokens' query rows into the chunk's
    // QB buffer. Two end records close the stream (one for each softmax team).
    if (lane == 0) tma_prefetch_desc(&a.tmap_q1);
    Chunks c{};
    c.g = c.j = -1;
    int last_g = -1;  // last chunk gathered (it and the three before are drained on abort)
    int item = -1;
    bool ok = true;
    auto take_buffer = [&](int g) -> bool {
      const int buf = g & (kSwBuf - 1);
      return g < kSwBuf ||
             mbar_wait_sleep(&sm.qb_free[buf], ((g >> 2) - 1) & 1, fault, kFaultWaitMma, abort);
    };
    for (int ni = 0; ok; ++ni) {
      SwItem it{};
      const int i = read_item(ni, ok, it);
      __syncwarp();
      if (!ok) break;
      if (lane == 0) release_item(ni);
      if (i < 0) break;
      if (it.n_union == 0) continue;
      ++item;
      chunks_item(c, a, it);
      while (chunks_next(c, tpc, G)) {
        const int buf = c.g & (kSwBuf - 1), ts = c.g & (kColSlots - 1);
        // Last chunk of the item: the last chunk of its last union block
        // (every union block has a member token: the union holds exactly the
        // ids some token of the tile can use).
        const bool item_end = c.rest == 0u && c.u == c.n_union - 1;
        if (!take_buffer(c.g)) {
          ok = false;
          break;
        }
        bool page_ok = true;
        if (a.paged) {
          const int pg = __ldg(a.page_table + (size_t)it.b * a.max_pages + c.blk);
          page_ok = pg >= 0 && pg < a.num_pages;
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int n = lane + 32 * h2;
          int row = -1, rel = 127;
          if (n < c.ntok * G) {
            const int sl = n / G, gh = n - sl * G;
            const int w = nth_set_bit(c.cm, sl);
            row = w * G + gh;
            const long long pos = (long long)it.lk - it.lq + (it.t0 + w - it.seq_q0);
            long long lastk = (long long)it.lk - 1;
            if (a.causal && pos < lastk) lastk = pos;
            const long long r = lastk - (long long)c.blk * kBlk;
            rel = page_ok ? (r > 127 ? 127 : (int)r) : -1;
          }
          sm.col_row[ts][n] = row;
          sm.col_rel[ts][n] = rel;
        }
        if (lane == 0) {
          ChunkRec r;
          r.N = c.N;
          r.ntok = c.ntok;
          r.j = c.j;
          r.flags = (c.first ? kRecFirst : 0) | (c.last ? kRecLast : 0) | (item_end ? kRecItemEnd : 0);
          r.item = item;
          sm.rec[ts] = r;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_expect_tx(&sm.qb_full[buf], (uint32_t)(c.ntok * G * 256));
          uint32_t m = c.cm;
          for (int sl = 0; m != 0u; ++sl) {
            const int w = __ffs(m) - 1;
            m &= m - 1u;
            for (int h2 = 0; h2 < 2; ++h2)
              tma_load_3d(&sm.qb[buf][h2][sl * G * 128], &a.tmap_q1, &sm.qb_full[buf], h2 * 64,
                          it.h * G, it.t0 + w);
          }
        }
        last_g = c.g;
      }
    }
    for (int e = 0; ok && e < 2; ++e) {
      const int g = ++c.g;
      if (!take_buffer(g)) break;
      if (lane == 0) {
        ChunkRec r{};
        r.flags = kRecStreamEnd;
        sm.rec[g & (kColSlots - 1)] = r;
        mbar_arrive(&sm.qb_full[g & (kSwBuf - 1)]);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) {
      for (int q = 0; q < kSwBuf; ++q)
        if (last_g - q >= 0)
          mbar_wait_sleep(&sm.qb_full[(last_g - q) & (kSwBuf - 1)], ((last_g - q) >> 2) & 1, fault,
                          kFaultWaitTma);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Follows the chunk records. Each step issues QK of chunk gq = gp + 2 and
    // PV of chunk gp with their K steps interleaved (two independent
    // accumulators in flight), then commits both.
    if (lane == 0) {
      constexpr uint32_t kSlot16 = (2 * 16384) >> 4;  // one K or V slot
      constexpr uint32_t kHalfKV16 = 16384 >> 4;      // second 64-column half of a slot
      constexpr uint32_t kBuf16 = (2 * kHalfQB) >> 4;  // one QB/P buffer
      constexpr uint32_t kHalfQB16 = kHalfQB >> 4;
      const uint64_t dk0 = sdesc_sw128(smem_u32(&sm.kv[0][0][0]), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(&sm.kv[2][0][0]), 16384, 1024);
      const uint64_t dq0 = sdesc_sw128(smem_u32(&sm.qb[0][0][0]), 16, 1024);
      // P as the PV's B operand: MN-major, one 64-column atom, 8-key groups 1 KB apart.
      const uint64_t dp0 = sdesc_sw128(smem_u32(&sm.qb[0][0][0]), 16384, 1024);
      bool ok = true;
      int gq = 0, gp = 0, gend = 0x7fffffff;
      // Waits for chunk g's record; false when a wait gave up.
      auto get_rec = [&](int g, ChunkRec& r) -> bool {
        if (!mbar_wait_sleep(&sm.qb_full[g & (kSwBuf - 1)], (g >> 2) & 1, fault, kFaultWaitTma, abort))
          return false;
        r = sm.rec[g & (kColSlots - 1)];
        return true;
      };
      // Inputs of QK(g): the block's K (first chunk of a block), the S/D
      // buffer released by the merge of chunk g - 4.
      auto qk_ready = [&](int g, const ChunkRec& r) -> bool {
        const int buf = g & (kSwBuf - 1);
        if ((r.flags & kRecFirst) &&
            !mbar_wait_sleep(&sm.kv_full[r.j & 1], (r.j >> 1) & 1, fault, kFaultWaitTma, abort))
          return false;
        if (g >= kSwBuf &&
            !mbar_wait_sleep(&sm.d_free[buf], ((g >> 2) - 1) & 1, fault, kFaultWaitSoftmax, abort))
          return false;
        return true;
      };
      // Inputs of PV(g): P from the softmax, the block's V (first chunk).
      auto pv_ready = [&](int g, const ChunkRec& r) -> bool {
        if (!mbar_wait_sleep(&sm.p_full[g & (kSwBuf - 1)], (g >> 2) & 1, fault, kFaultWaitSoftmax, abort))
          return false;
        if ((r.flags & kRecFirst) &&
            !mbar_wait_sleep(&sm.kv_full[2 + (r.j & 1)], (r.j >> 1) & 1, fault, kFaultWaitTma, abort))
          return false;
        return true;
      };
      auto qk_mma = [&](int g, const ChunkRec& r, int kk) {
        const int buf = g & (kSwBuf - 1);
        const uint32_t id = idesc_16bit_f32(128, r.N, false, false, F16);
        const uint64_t dk = dk0 + (r.j & 1) * kSlot16, dq = dq0 + buf * kBuf16;
        mma_ss(tbase + kColS + (uint32_t)(buf * 64), dk + (kk >> 2) * kHalfKV16 + (kk & 3) * 2,
               dq + (kk >> 2) * kHalfQB16 + (kk & 3) * 2, id, kk > 0 ? 1u : 0u);
      };
      auto pv_mma = [&](int g, const ChunkRec& r, int kk) {
        const int buf = g & (kSwBuf - 1);
        const uint32_t id = idesc_16bit_f32(128, r.N, true, true, F16);
        const uint64_t dv = dv0 + (r.j & 1) * kSlot16, dp = dp0 + buf * kBuf16;
        mma_ss(tbase + kColS + (uint32_t)(buf * 64), dv + kk * 128, dp + kk * 128, id,
               kk > 0 ? 1u : 0u);
      };
      auto qk_commit = [&](int g, const ChunkRec& r) {
        mma_commit(&sm.qk_done[g & (kSwBuf - 1)]);
        if (r.flags & kRecLast) mma_commit(&sm.kv_empty[r.j & 1]);
      };
      auto pv_commit = [&](int g, const ChunkRec& r) {
        const int buf = g & (kSwBuf - 1);
        mma_commit(&sm.pv_done[buf]);
        mma_commit(&sm.qb_free[buf]);
        if (r.flags & kRecLast) mma_commit(&sm.kv_empty[2 + (r.j & 1)]);
      };
      // Prologue: QK of the first two chunks.
      for (int k = 0; ok && k < 2 && gq < gend; ++k) {
        ChunkRec r;
        ok = get_rec(gq, r);
        if (!ok) break;
        if (r.flags & kRecStreamEnd) {
          gend = gq;
          break;
        }
        ok = qk_ready(gq, r);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) qk_mma(gq, r, kk);
        qk_commit(gq, r);
        ++gq;
      }
      while (ok && gp < gend) {
        const ChunkRec rp = sm.rec[gp & (kColSlots - 1)];  // waited for by the QK step
        ChunkRec rq{};
        bool have_q = false;
        if (gq < gend) {
          ok = get_rec(gq, rq);
          if (!ok) break;
          if (rq.flags & kRecStreamEnd) gend = gq;
          else have_q = true;
        }
        ok = pv_ready(gp, rp) && (!have_q || qk_ready(gq, rq));
        if (!ok) break;
        tc_fence_after();
        if (have_q) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            qk_mma(gq, rq, kk);
            pv_mma(gp, rp, kk);
          }
          qk_commit(gq, rq);
          ++gq;
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) pv_mma(gp, rp, kk);
        }
        pv_commit(gp, rp);
        ++gp;
      }
      mma_commit(&sm.drain);
      mbar_wait_sleep(&sm.drain, 0, fault, kFaultWaitMma);
    }
  } else if (warp < kSmWarps) {
    // ------------------------------------------------------------ softmax
    // Two teams of four warps (one per key quarter) take alternate chunks,
    // so two chunks are in flight; each warp covers all of its chunk's
    // columns for its 32 keys, in passes of 32 (or 16) columns.
    SmCtx x;
    x.q4 = warp & 3;
    x.team = warp >> 2;
    x.warp = warp;
    x.lane = lane;
    x.scale_log2 = a.scale_log2;
    x.lane_base = tbase + ((uint32_t)(x.q4 * 32) << 16);
    const int bar_team = 1 + x.team;
    bool ok = true;
    int item = -1, xslot = 0;
    for (int g = x.team;; g += 2) {
      const int buf = g & (kSwBuf - 1), ts = g & (kColSlots - 1);
      const uint32_t ph = (g >> 2) & 1;
      // qb_full: the chunk's record and column table are written (and, for
      // a real chunk, its Q rows have landed).
      ok = ok && mbar_wait_sleep(&sm.qb_full[buf], ph, fault, kFaultWaitTma, abort);
      ok = bar_and(bar_team, 128, ok);
      if (!ok) break;
      const ChunkRec r = sm.rec[ts];
      if (r.flags & kRecStreamEnd) break;
      // The row state is reset by the merge warps after the previous item's
      // epilogue.
      if (r.item != item) {
        if (r.item > 0)
          ok = mbar_wait_sleep(&sm.state_free, (r.item - 1) & 1, fault, kFaultWaitOther, abort);
        item = r.item;
      }
      ok = ok && mbar_wait_sleep(&sm.qk_done[buf], ph, fault, kFaultWaitMma, abort);
      ok = !__any_sync(0xffffffffu, !ok);
      tc_fence_after();
      const int nvalid = r.ntok * G;
      const int npass = (r.N + 31) >> 5;  // passes of 32 columns (the last may run past N)
      float* xs = &sm.xch[x.team][xslot][0][0][0];
      // Phase 1: column maxima over this warp's keys, exchanged in the team.
#pragma unroll 1
      for (int ps = 0; ps < npass; ++ps) {
        float s0[32];
        xs[(ps * 4 + x.q4) * 32 + lane] = pass_max<32>(sm, x, buf, ts, ps * 32, s0);
      }
      ok = bar_and(bar_team, 128, ok);
      float mx[2];
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        mx[ps] = xs[(ps * 4) * 32 + lane];
#pragma unroll
        for (int q = 1; q < 4; ++q) mx[ps] = fmaxf(mx[ps], xs[(ps * 4 + q) * 32 + lane]);
      }
      xslot ^= 1;
      // Phase 2, in chunk order per key quarter: the previous chunk (the
      // other team's) has written its row maxima.
      if (g > 0)
        ok = ok && mbar_wait_sleep(&sm.state_done[x.q4], (g - 1) & 1, fault, kFaultWaitSoftmax, abort);
      pass_state<32>(sm, x, buf, ts, 0, nvalid, mx[0]);
      if (npass > 1) pass_state<32>(sm, x, buf, ts, 32, nvalid, mx[1]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.state_done[x.q4]);
      // Phase 3: P and column sums (S^T reloaded from TMEM and masked again).
      // Columns past N get P too, in QB columns the PV's N never reaches.
#pragma unroll 1
      for (int ps = 0; ps < npass; ++ps) {
        float s0[32];
        load_masked<32>(sm, x, buf, ts, ps * 32, s0);
        pass_exp<32, F16>(sm, x, buf, ps * 32, s0);
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[buf]);
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ merge + epilogue
    const int q4 = warp & 3;
    const int mt = tid - kMergeWarp0 * 32;  // 0..127
    const uint32_t lane_base = tbase + ((uint32_t)(q4 * 32) << 16);
    const int dcol = q4 * 32 + lane;  // this thread's head dimension
    const int R = W * G;
    for (int c0 = 0; c0 < 256; c0 += 32) tmem_zero32(lane_base + (uint32_t)c0);
    int g = 0;
    bool ok = true;
    for (int ni = 0; ok; ++ni) {
      SwItem it{};
      const int cur = read_item(ni, ok, it);
      __syncwarp();
      if (ok && lane == 0) release_item(ni);
      ok = bar_and(3, 128, ok);
      if (!ok || cur < 0) break;
      const int nw = min(W, it.seq_q0 + it.lq - it.t0);
      const size_t orow0 = (size_t)it.t0 * a.num_qo_heads + (size_t)it.h * G;
      if (it.n_union == 0) {
        // No usable block at all: out = 0, lse = -inf.
        for (int r = 0; r < nw * G; ++r) {
          const int w = r / G;
          const size_t orow = orow0 + (size_t)w * a.num_qo_heads + (r - w * G);
          reinterpret_cast<uint16_t*>(a.out)[orow * 128 + dcol] = 0;
        }
        for (int r = mt; r < nw * G; r += 128) {
          const int w = r / G;
          if (a.lse != nullptr) a.lse[orow0 + (size_t)w * a.num_qo_heads + (r - w * G)] = -INFINITY;
        }
        continue;
      }
      for (;; ++g) {
        const int buf = g & (kSwBuf - 1), ts = g & (kColSlots - 1);
        const uint32_t ph = (g >> 2) & 1;
        ok = mbar_wait_sleep(&sm.pv_done[buf], ph, fault, kFaultWaitMma, abort) &&
             mbar_wait_sleep(&sm.p_full[buf], ph, fault, kFaultWaitSoftmax, abort);
        ok = bar_and(3, 128, ok);  // the four merge warps give up together
        if (!ok) break;
        tc_fence_after();
        const ChunkRec r = sm.rec[ts];
        const int nvalid = r.ntok * G;
        // l[row] = alpha * l[row] + the column's sum of P over all 128 keys;
        // rows repeat across chunks, and the barrier above orders the updates.
        if (mt < nvalid) {
          const int row = sm.col_row[ts][mt];
          sm.l_row[row] = sm.alpha[buf][mt] * sm.l_row[row] + sm.psum[buf][0][mt] +
                          sm.psum[buf][1][mt] + sm.psum[buf][2][mt] + sm.psum[buf][3][mt];
        }
        // O^T[:, row] = alpha * O^T[:, row] + D[:, column] for each member row,
        // in groups of 8 columns (one token's 8 heads; G is a multiple of 8),
        // four groups per TMEM round trip.
        const int ngrp = nvalid >> 3;
        for (int g0 = 0; g0 < ngrp; g0 += 4) {
          uint32_t dv[4][8], ov[4][8];
          int orow[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            orow[e] = g0 + e < ngrp ? sm.col_row[ts][(g0 + e) * 8] : 0;
            if (g0 + e < ngrp) {
              tmem_ld8_nowait(lane_base + kColS + (uint32_t)(buf * 64 + (g0 + e) * 8), dv[e]);
              tmem_ld8_nowait(lane_base + (uint32_t)orow[e], ov[e]);
            }
          }
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (g0 + e < ngrp) {
              const float4 a0 = *reinterpret_cast<const float4*>(&sm.alpha[buf][(g0 + e) * 8]);
              const float4 a1 = *reinterpret_cast<const float4*>(&sm.alpha[buf][(g0 + e) * 8 + 4]);
              const float al[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
              for (int k = 0; k < 8; ++k)
                ov[e][k] = __float_as_uint(
                    fmaf(al[k], __uint_as_float(ov[e][k]), __uint_as_float(dv[e][k])));
              tmem_st8_nowait(lane_base + (uint32_t)orow[e], ov[e]);
            }
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.d_free[buf]);
        if (r.flags & kRecItemEnd) {
          ++g;
          break;
        }
      }
      if (!ok) break;
      // ---------------------------------------------------- item epilogue
      // The row state for this item is final: every chunk's p_full has been
      // waited for above (the softmax writes m before it), and the l
      // updates are this group's own, ordered by the barrier below.
      ok = bar_and(3, 128, ok);
      if (!ok) break;
      for (int r = mt; r < R; r += 128) {
        const float l = sm.l_row[r];
        sm.inv_l[r] = l > 0.f ? a.out_scale / l : 0.f;
        const int w = r / G;
        if (w < nw && a.lse != nullptr)
          a.lse[orow0 + (size_t)w * a.num_qo_heads + (r - w * G)] =
              l > 0.f ? (sm.m_ref[0][r] + log2f(l)) * 0.69314718055994531f : -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q) sm.m_ref[q][r] = -INFINITY;
        sm.l_row[r] = 0.f;
      }
      ok = bar_and(3, 128, ok);
      if (!ok) break;
      // out = O^T[:, row] / l per row, eight columns (one token, eight
      // heads) per TMEM load; O^T is zeroed for the next item.
      for (int c0 = 0; c0 < R; c0 += 8) {
        float o[8];
        tmem_ld8(lane_base + (uint32_t)c0, o);
        const int w = c0 / G, gh0 = c0 - w * G;
        if (w < nw) {
          const size_t orow = orow0 + (size_t)w * a.num_qo_heads + gh0;
          uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + orow * 128 + dcol;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[(size_t)i * 128] = (uint16_t)(pack_x2<F16>(o[i] * sm.inv_l[c0 + i], 0.f) & 0xFFFFu);
        }
      }
      for (int c0 = 0; c0 < R; c0 += 32) tmem_zero32(lane_base + (uint32_t)c0);
      tc_fence_before();
      ok = bar_and(3, 128, ok);  // inv_l and the row state are free again
      if (!ok) break;
      if (lane == 0) mbar_arrive(&sm.state_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <class Kernel>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       const PrefillArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <bool F16>
cudaError_t launch_sw(const PrefillArgs& a, cudaStream_t s) {
  const int optin = device_smem_optin();
  if (optin <= 0) return cudaErrorInvalidDevice;
  size_t smem = sizeof(SwSmem) + 1024;
  if (smem > (size_t)optin) smem = (size_t)optin;
  cudaError_t e = set_smem_limit((const void*)prefill_swapped_kernel<F16>, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = a.num_items < device_sm_count() ? a.num_items : device_sm_count();
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(prefill_swapped_kernel<F16>, dim3(grid), dim3(kSwThreads), smem, s, a);
}

}  // namespace

cudaError_t launch_prefill_swapped(const PrefillArgs& a, cudaStream_t s) {
  return a.f16 ? launch_sw<true>(a, s) : launch_sw<false>(a, s);
}

}  // namespace msa
