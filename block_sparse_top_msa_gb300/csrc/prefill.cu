// MSA sparse attention for sm_103a, prefill and paged decode
// ("flashinfer.msa_ops.msa_sparse_attention": each query attends only the
// top-K KV blocks selected in q2k_indices; query tokens are processed in
// tiles, each running one online softmax over the union of the blocks its
// tokens selected).
//
// A persistent grid (one CTA per SM) walks work items: a query tile of
// W = 128 / G consecutive tokens of one sequence (128 rows (token w, query
// head g) = one tcgen05 M=128 tile, row r in TMEM lane r), a KV head, and a
// slice of the tile's union list (whole lists, except for the last round of
// decode-sized launches, whose lists are split and merged afterwards by
// merge_splits_kernel). Roles per CTA, for each union block u:
//   K producer    : claims the CTA's next item from a launch-wide counter,
//                   publishes it to the other roles, loads the item's Q tile
//                   and TMA-gathers K_u (flat rows cu_k[b] + 128 id, or page
//                   page_table[b, id]) into a three-deep ring;
//   V producer    : the same for V_u (bf16 / fp16 K/V);
//   MMA warp      : S_u = Q K_u^T (fp32, TMEM, three S buffers, QK running
//                   two blocks ahead), then O += P_u V_u with P read from TMEM;
//   softmax warps : two warpgroups split each S row by columns; a thread
//                   masks its row's keys by block membership of its token,
//                   causality (key <= Lk - Lq + i) and the sequence end,
//                   updates the running max (rescaling O only when the max
//                   grows by more than 2^8), writes P = 2^(s*scale*log2e - m)
//                   into TMEM, and at the end of an item writes O / l and the
//                   natural-log LSE (or fp32 partials of a split item).
// E4M3 and packed NVFP4 K/V (the FP8 instance): one softmax warpgroup, and
// the producer fills a staging ring (TMA for E4M3, bulk copies of the
// planar page's code and scale slices for NVFP4) that six converter warps
// decode exactly to bf16 in the MMA's swizzled layout.
// Rows whose token did not select block u get P = 0 for it, so each row's
// result is exactly its own blocks' softmax attention.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tmem_wide.cuh"

namespace msa {
namespace {

constexpr int kF8Stages = 2;    // E4M3 staging ring (K and V bytes of one block)
constexpr int kSBuf = 3;        // S/P buffers in TMEM: QK runs two blocks ahead of PV
constexpr int kPV = 3;          // PV completion barriers (block g uses g % kPV)
constexpr int kItemRing = 4;    // work items handed from the K producer to the other roles
constexpr int kClaimAhead = 4;  // the K producer claims its next item this many blocks early
static_assert(kPV == kSBuf, "the MMA issuer walks S buffers and PV barriers with one ring");
constexpr int kTile = 16384;    // bytes of one 128-row x 128-byte swizzled tile
constexpr float kRescaleLog2 = 8.0f;

// TMEM column map (512 columns allocated): S_b at 128*b for b = 0..2, O at
// 384. P (packed bf16 pairs) overwrites S_b once the softmax has read it: the
// P of S columns 64j..64j+63 goes to columns 64j..64j+31, inside the column
// group its softmax warpgroup owns.
constexpr uint32_t kColO = 384;

// Shared memory holds one Q tile, a three-deep K ring and a three-deep V ring
// (bf16). STREAM: layout for memory-bound launches (decode-sized problems
// split into many short items, at most 64 real Q rows): two Q slots share the
// one 32 KiB Q region, slot j starting j * rows * 128 bytes in, so the next
// item's Q loads while the current one runs; each slot's real rows stay clear
// of the other's, and the rows an M=128 MMA reads past them (other slots, or
// the K ring) only feed S rows no token owns.
//
// Completion barriers: qk_done[g % 3] completes when QK(g) (and every MMA
// issued before it) has completed: S_g is readable and the K slot of block g
// is free. pv_done[g % 3] likewise for PV(g): O holds block g and its V slot
// is free. One commit per MMA group keeps the issuing thread's overhead low.
// One work item: a (query tile, KV head, split) triple and its slice of the
// tile's union list. Every role derives the same items in the same order.
struct Item {
  int tile, h, split, t0, b, n_union, p_begin, n;
  int tail;                 // index among the split (tail) units, or -1 for a whole unit
  int seq_q0, lq, lk, kv0;  // the tile's sequence (valid when t0 >= 0)
};

// Warp roles. The softmax runs in kSoftmaxWG warpgroups; with two, warps q
// and q + 4 share TMEM lanes 32q..32q+31 and split each S row by columns
// (0..63 and 64..127), exchanging their partial row maxima every block. The
// E4M3 / NVFP4 variant keeps one warpgroup and spends the registers on six
// converter warps (12 warps at 168 registers); its conversion is latency-
// bound, and four converters were measured 5-7% slower.
template <bool FP8>
struct Roles {
  static constexpr int kSoftmaxWG = FP8 ? 1 : 2;
  static constexpr int kSoftmaxWarps = 4 * kSoftmaxWG;
  static constexpr int kProducerWarp = kSoftmaxWarps;              // Q and K (E4M3: K and V)
  static constexpr int kMmaWarp = kSoftmaxWarps + 1;
  static constexpr int kVProducerWarp = FP8 ? -1 : kSoftmaxWarps + 2;  // V (bf16 only)
  static constexpr int kConvWarp0 = kSoftmaxWarps + 2;              // E4M3 / NVFP4 converters
  static constexpr int kConvWarps = 6;
  static constexpr int kWarps = kSoftmaxWarps + 2 + (FP8 ? kConvWarps : 1);
  // Readers of the item ring (the K producer writes it): V producer (bf16),
  // the MMA issuer's two cursors, every softmax warp, every converter warp.
  static constexpr int kItemReaders = (FP8 ? 0 : 1) + 2 + kSoftmaxWarps + (FP8 ? kConvWarps : 0);
  static constexpr int kThreads = kWarps * 32;
};

template <bool FP8, bool STREAM = false>
struct __align__(1024) PrefillSmem {
  static constexpr int kXch = Roles<FP8>::kSoftmaxWG == 2 ? 2 * 2 * 128 : 1;
  static constexpr int kQBuf = STREAM ? 2 : 1;   // Q tiles of consecutive items
  static constexpr int kQRegions = 1;
  static constexpr int kKStages = FP8 ? 2 : 3;   // K ring (a slot frees when its QK completes)
  static constexpr int kVStages = FP8 ? 2 : 3;   // V ring (a slot frees when its PV completes)
  static_assert(kKStages <= kSBuf && kVStages <= kPV, "ring deeper than its completion barriers");
  uint8_t q[kQRegions][2][kTile];
  uint8_t k[kKStages][2][kTile];
  uint8_t v[kVStages][2][kTile];
  uint8_t k8[FP8 ? kF8Stages : 1][FP8 ? kTile : 16];
  uint8_t v8[FP8 ? kF8Stages : 1][FP8 ? kTile : 16];
  uint64_t q_full[kQBuf];
  uint64_t q_empty[kQBuf];
  uint64_t k_full[kKStages];
  uint64_t v_full[kVStages];
  uint64_t f8_full[kF8Stages];
  uint64_t f8_empty[kF8Stages];
  int f8_valid[kF8Stages];  // NVFP4: the staged block's page is mapped (else it is zero)
  uint64_t qk_done[kSBuf];
  uint64_t p_full[kSBuf];
  uint64_t pv_done[kPV];
  uint64_t o_free;
  uint64_t drain;
  uint64_t item_full[kItemRing];
  uint64_t item_empty[kItemRing];
  int item_idx[kItemRing];
  Item item_ring[kItemRing];
  uint32_t tmem_base;
  int abort;
  float xch[kXch];  // [slot][warpgroup][row] values exchanged between the softmax warpgroups
};

MSA_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Named barrier of softmax warps q and q + 4 (64 threads, barrier q + 1);
// returns the AND of p over both warps. Both warps of a pair take the same
// branches (their decisions are made from exchanged values), so each arrives.
MSA_DEV bool pair_barrier_and(int q, bool p) {
  int r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.s32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, 64, pi;\n\tselp.s32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((int)p), "r"(q + 1)
      : "memory");
  return r != 0;
}

MSA_DEV float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Max of 64 values with four independent three-input chains.
MSA_DEV float row_max64(const float* v) {
  float m0 = v[0], m1 = v[1], m2 = v[2], m3 = v[3];
#pragma unroll
  for (int c = 4; c + 8 <= 64; c += 8) {
    m0 = fmax3(m0, v[c], v[c + 1]);
    m1 = fmax3(m1, v[c + 2], v[c + 3]);
    m2 = fmax3(m2, v[c + 4], v[c + 5]);
    m3 = fmax3(m3, v[c + 6], v[c + 7]);
  }
  m0 = fmax3(m0, v[60], v[61]);
  m1 = fmax3(m1, v[62], v[63]);
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// Running-max update of one row for a block whose raw max logit is mx. The
// reference max only moves when the new max exceeds it by more than 2^8, so
// O is rescaled rarely; P stays <= 2^8, exact enough for bf16 and fp32 sums.
MSA_DEV void update_max(bool mem, float mx, float scale_log2, float& m_ref, float& l,
                        float& alpha, bool& rescale) {
  if (!mem) return;
  const float m_new = mx * scale_log2;
  if (m_ref == -INFINITY || m_new > m_ref + kRescaleLog2) {
    if (m_ref != -INFINITY) {
      alpha = ex2(m_ref - m_new);
      rescale = true;
      l *= alpha;
    }
    m_ref = m_new;
  }
}

// P = 2^(s * scale_log2 + neg_m) for N columns, packed to 16-bit pairs (the
// type of V) and stored to TMEM at pcol (N/2 columns); the fp32 values are
// summed into acc. P <= 2^8, well inside the f16 range.
template <int N, bool F16 = false>
MSA_DEV void exp_pack_store(const float* sv, float2 sc2, float neg_m, float2& acc, uint32_t pcol) {
  uint32_t pk[N / 2];
  const float2 nm2 = make_float2(neg_m, neg_m);
#pragma unroll
  for (int c = 0; c < N; c += 2) {
    const float2 x = __ffma2_rn(make_float2(sv[c], sv[c + 1]), sc2, nm2);
    const float p0 = ex2(x.x), p1 = ex2(x.y);
    acc = __fadd2_rn(acc, make_float2(p0, p1));
    pk[c >> 1] = pack_x2<F16>(p0, p1);
  }
  if (N == 64) tmem_st32(pcol, pk);
}

// Upconverts one 128x128 E4M3 tile (TMA SWIZZLE_128B image, 128-byte rows)
// into the two 64-column bf16 halves the MMA reads, with kThreads threads.
template <int kThreads>
MSA_DEV void convert_tile(const uint8_t* src, uint8_t* dst_half0, int t) {
#pragma unroll 2
  for (int i = t; i < 1024; i += kThreads) {
    const int r = i >> 3, c = i & 7;
    const uint4 raw = *reinterpret_cast<const uint4*>(src + sw128_offset(r, c));
    uint32_t outw[8];
    e4m3x4_to_bf16(raw.x, outw[0], outw[1]);
    e4m3x4_to_bf16(raw.y, outw[2], outw[3]);
    e4m3x4_to_bf16(raw.z, outw[4], outw[5]);
    e4m3x4_to_bf16(raw.w, outw[6], outw[7]);
    uint8_t* dst = dst_half0 + (c >> 2) * kTile;
    const int c16 = (c & 3) * 2;
    *reinterpret_cast<uint4*>(dst + sw128_offset(r, c16)) =
        make_uint4(outw[0], outw[1], outw[2], outw[3]);
    *reinterpret_cast<uint4*>(dst + sw128_offset(r, c16 + 1)) =
        make_uint4(outw[4], outw[5], outw[6], outw[7]);
  }
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to shared memory, completing on `bar`.
MSA_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Converts one staged NVFP4 slice (kFp4Data code bytes, then kFp4Scales
// scales) into the two 64-column bf16 halves the MMA reads (SWIZZLE_128B
// image), or writes zeros when the slice's page is unmapped.
template <int kThreads>
MSA_DEV void convert_fp4_tile(const uint8_t* src, bool v_order, bool valid, uint8_t* dst_half0,
                              int t) {
#pragma unroll 2
  for (int i = t; i < 1024; i += kThreads) {
    const int r = i >> 3, c = i & 7;  // token r, elements 16c .. 16c + 15
    uint32_t outw[8];
    if (valid) {
      const uint2 codes = *reinterpret_cast<const uint2*>(src + r * 64 + c * 8);
      fp4x16_to_bf16(codes, src[kFp4Data + fp4_scale_offset(v_order, r, c)], outw);
    } else {
#pragma unroll
      for (int w = 0; w < 8; ++w) outw[w] = 0u;
    }
    uint8_t* dst = dst_half0 + (c >> 2) * kTile;
    const int c16 = (c & 3) * 2;
    *reinterpret_cast<uint4*>(dst + sw128_offset(r, c16)) =
        make_uint4(outw[0], outw[1], outw[2], outw[3]);
    *reinterpret_cast<uint4*>(dst + sw128_offset(r, c16 + 1)) =
        make_uint4(outw[4], outw[5], outw[6], outw[7]);
  }
}

// The (t0, b) pair of item i's tile, the one field that needs a load before
// the rest can be fetched (and that the softmax warps fetch one item ahead).
MSA_DEV int2 item_tile_info(const PrefillArgs& a, int i) {
  const int unit = i < a.whole_units ? i : a.whole_units + (i - a.whole_units) / a.splits;
  const int h = unit / a.max_tiles;
  const int tile = a.max_tiles - 1 - (unit - h * a.max_tiles);
  return __ldg(reinterpret_cast<const int2*>(a.tile_info) + tile);
}

MSA_DEV Item item_at(const PrefillArgs& a, int i, int2 ti) {
  Item it;
  int unit;
  if (i < a.whole_units) {
    unit = i;
    it.split = 0;
    it.tail = -1;
  } else {
    const int j = i - a.whole_units;
    it.tail = j / a.splits;
    it.split = j - it.tail * a.splits;
    unit = a.whole_units + it.tail;
  }
  // Head-major: all tiles of one KV head (later, heavier tiles first) before
  // the next head, so the items in flight share one head's K/V in L2.
  it.h = unit / a.max_tiles;
  const int tile_idx = unit - it.h * a.max_tiles;
  it.tile = a.max_tiles - 1 - tile_idx;
  it.t0 = ti.x;
  it.b = ti.y;
  it.p_begin = it.tail < 0 ? 0 : it.split * a.pps;
  it.n_union = 0;
  it.n = 0;
  it.seq_q0 = it.lq = it.lk = it.kv0 = 0;
  if (it.t0 >= 0) {
    it.n_union = __ldg(a.union_len + (size_t)it.h * a.max_tiles + it.tile);
    it.n = it.tail < 0 ? it.n_union : max(0, min(it.n_union, it.p_begin + a.pps) - it.p_begin);
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

// Union metadata load: read-only path when the union kernel wrote it before
// the launch, L2 when this launch's own item setup wrote it (direct mode).
MSA_DEV int32_t meta_ld(const int32_t* p, bool direct) { return direct ? __ldcg(p) : __ldg(p); }
MSA_DEV uint32_t meta_ld(const uint32_t* p, bool direct) { return direct ? __ldcg(p) : __ldg(p); }

// Sequence holding packed query row t: the b with cu_q[b] <= t < cu_q[b + 1],
// returned with those two offsets. The first probe assumes equal query
// lengths (exact for a decode batch); otherwise a binary search for the last
// b with cu_q[b] <= t.
MSA_DEV int find_sequence(const int32_t* cu_q, int batch, int total_q, int t, int& q0, int& q1) {
  const int g = min(batch - 1, (int)((long long)t * batch / max(total_q, 1)));
  q0 = __ldcg(cu_q + g);
  q1 = __ldcg(cu_q + g + 1);
  if (q0 <= t && t < q1) return g;
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldcg(cu_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  q0 = __ldcg(cu_q + lo);
  q1 = __ldcg(cu_q + lo + 1);
  return lo;
}

// Work item i of a one-token-tile launch without the union kernel (direct
// mode): the tile is query row t0 = tile, and its union is that token's own
// selection: the ids of its q2k row (KV head h) that are usable (0 <= id <
// number of blocks, and id * 128 <= the token's position when causal),
// ascending and without repeats, the set the union kernel would produce for a
// one-token tile. The list, its length and the tile's (t0, b) are written to
// the union arrays for the other roles (which read them after the item is
// published) and the merge kernel; every split of a unit writes the same
// values. One thread; two dependent rounds of loads (the row with the
// sequence probe, then the sequence's key length).
MSA_DEV Item direct_item(const PrefillArgs& a, int i) {
  constexpr int kN = 32;  // topk <= 32
  Item it;
  int unit;
  if (i < a.whole_units) {
    unit = i;
    it.split = 0;
    it.tail = -1;
  } else {
    const int j = i - a.whole_units;
    it.tail = j / a.splits;
    it.split = j - it.tail * a.splits;
    unit = a.whole_units + it.tail;
  }
  it.h = unit / a.max_tiles;
  it.tile = a.max_tiles - 1 - (unit - it.h * a.max_tiles);
  it.t0 = it.tile;
  it.p_begin = it.tail < 0 ? 0 : it.split * a.pps;
  const int32_t* row = a.q2k + ((size_t)it.h * a.total_q + it.t0) * a.topk;
  int key[kN];
#pragma unroll
  for (int j = 0; j < kN; ++j) key[j] = j < a.topk ? __ldcg(row + j) : -1;
  int q1;
  it.b = find_sequence(a.cu_q, a.batch, a.total_q, it.t0, it.seq_q0, q1);
  it.lq = q1 - it.seq_q0;
  int nblk;
  if (a.paged) {
    it.kv0 = 0;
    it.lk = __ldcg(a.seqused_k + it.b);
    nblk = min((it.lk + kBlk - 1) / kBlk, a.max_pages);
  } else {
    it.kv0 = __ldcg(a.cu_k + it.b);
    it.lk = __ldcg(a.cu_k + it.b + 1) - it.kv0;
    nblk = (it.lk + kBlk - 1) / kBlk;
  }
  const long long pos = (long long)it.lk - it.lq + (it.t0 - it.seq_q0);
  bool sorted = true;
#pragma unroll
  for (int j = 0; j < kN; ++j) {
    const int id = key[j];
    key[j] = (id < 0 || id >= nblk || (a.causal && (long long)id * kBlk > pos)) ? INT_MAX : id;
    if (j > 0) sorted = sorted && key[j - 1] <= key[j];
  }
  if (!sorted) {
    // Bitonic sorting network, ascending.
#pragma unroll
    for (int k = 2; k <= kN; k <<= 1) {
#pragma unroll
      for (int s = k >> 1; s > 0; s >>= 1) {
#pragma unroll
        for (int x = 0; x < kN; ++x) {
          const int y = x ^ s;
          if (y > x) {
            const int lo = min(key[x], key[y]), hi = max(key[x], key[y]);
            const bool up = (x & k) == 0;
            key[x] = up ? lo : hi;
            key[y] = up ? hi : lo;
          }
        }
      }
    }
  }
  // The union arrays are indexed (KV head, tile), like the union kernel's.
  const size_t slot = (size_t)it.h * a.max_tiles + it.tile;
  int32_t* dst = a.union_blocks + slot * a.cap;
  int n = 0;
#pragma unroll
  for (int j = 0; j < kN; ++j) {
    if (key[j] != INT_MAX && (j == 0 || key[j] != key[j - 1])) dst[n++] = key[j];
  }
  a.union_len[slot] = n;
  int32_t* ti = a.tile_info + 2 * it.tile;
  ti[0] = it.t0;
  ti[1] = it.b;
  it.n_union = n;
  it.n = it.tail < 0 ? n : max(0, min(n, it.p_begin + a.pps) - it.p_begin);
  return it;
}

// Slot index and phase parity of a position in a ring of N slots, advanced
// one step at a time (no divisions on the MMA issue path).
template <int N>
struct RingPos {
  int idx = 0;
  uint32_t phase = 0;
  MSA_DEV void next() {
    if (++idx == N) {
      idx = 0;
      phase ^= 1u;
    }
  }
};

// Position in the CTA's stream of blocks: n items read from the item ring,
// block u inside the current item, ordinal k of the item among non-empty
// items, and global block ordinal g.
struct Cursor {
  int n, u, k, g;
  bool valid;
  Item it;
};

template <bool FP8, bool STREAM, bool F16>
__global__ void __launch_bounds__(Roles<FP8>::kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillArgs a) {
  static_assert(!(FP8 && F16), "E4M3 K/V are upconverted to bf16");
  using R = Roles<FP8>;
  using Smem = PrefillSmem<FP8, STREAM>;
  // 16-bit prefill layout (long items): an item's epilogue is deferred until
  // the next item's first block has published its P.
  constexpr bool kDeferEpilogue = !STREAM && !FP8;
  constexpr int kQBuf = Smem::kQBuf;
  constexpr int kKStages = Smem::kKStages;
  constexpr int kVStages = Smem::kVStages;
  extern __shared__ uint8_t smem_raw[];
  // The swizzled tiles need a 1024-byte aligned base; the launch reserves up
  // to 1 KiB of slack for it when the limit leaves room. A launch whose slack
  // does not cover the base's actual offset reports and does nothing.
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  {
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (pad + sizeof(Smem) > dyn) {
      if (threadIdx.x == 0) atomicOr(a.fault, (unsigned)kFaultCapacity);
      return;
    }
  }
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw + pad);
  unsigned* fault = a.fault;
  volatile int* abort = &sm.abort;
  // Waits until QK(j) / PV(j), the j-th block's MMA group of this CTA, has
  // completed. Block j - 3 used the same barrier one phase earlier, and every
  // caller has already seen it complete (MMAs complete in issue order, and
  // each caller waits for blocks in increasing order; the softmax and the
  // epilogue wait for QK(gg) first, which is issued after PV(gg - 3)), so the
  // parity names the right phase. No barrier can run a phase ahead of a
  // waiter either: QK(j + 3) and PV(j + 3) need data the waiter has not
  // released yet.
  auto qk_wait = [&](int j) {
    return mbar_wait(&sm.qk_done[j % kSBuf], (j / kSBuf) & 1, fault, kFaultWaitMma, abort);
  };
  auto pv_wait = [&](int j) {
    return mbar_wait(&sm.pv_done[j % kPV], (j / kPV) & 1, fault, kFaultWaitMma, abort);
  };
  // The n-th work item of this CTA (index -1 once there are none left) and
  // its fields, published by the K producer in slot n % kItemRing. A reader
  // copies the item and releases the slot at once (release_item, one arrival
  // per reader), so the publisher only ever waits on reads, not on progress.
  auto read_item = [&](int n, bool& okr, Item& it) -> int {
    const int slot = n % kItemRing;
    if (!mbar_wait(&sm.item_full[slot], (n / kItemRing) & 1, fault, kFaultWaitOther, abort)) {
      okr = false;
      return -1;
    }
    const int idx = *reinterpret_cast<volatile int*>(&sm.item_idx[slot]);
    if (idx >= 0) it = sm.item_ring[slot];
    return idx;
  };
  auto release_item = [&](int n) { mbar_arrive(&sm.item_empty[n % kItemRing]); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.num_qo_heads / a.num_kv_heads;
  const int W = a.tile_tokens;
  // Shared-memory address of half c of Q slot qb.
  auto q_addr = [&](int qb, int c) -> uint8_t* {
    if (STREAM) return &sm.q[0][c][0] + (size_t)qb * (W * G) * 128;
    return &sm.q[qb][c][0];
  };

  if (tid == 0) {
    for (int s = 0; s < kQBuf; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&sm.k_full[s], FP8 ? R::kConvWarps : 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&sm.v_full[s], FP8 ? R::kConvWarps : 1);
    }
    for (int s = 0; s < kF8Stages; ++s) {
      mbar_init(&sm.f8_full[s], 1);
      mbar_init(&sm.f8_empty[s], R::kConvWarps);
    }
    for (int s = 0; s < kSBuf; ++s) {
      mbar_init(&sm.qk_done[s], 1);
      mbar_init(&sm.p_full[s], R::kSoftmaxWarps);
    }
    for (int s = 0; s < kPV; ++s) mbar_init(&sm.pv_done[s], 1);
    mbar_init(&sm.o_free, R::kSoftmaxWarps);
    mbar_init(&sm.drain, 1);
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(&sm.item_full[s], 1);
      mbar_init(&sm.item_empty[s], R::kItemReaders);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == R::kMmaWarp) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  // Everything above overlaps the tail of the union-metadata kernel; its
  // results are read only after this wait (programmatic dependent launch).
  // With wait_late, the kernel before this one only zeroes the work counter
  // (all other inputs were complete before it started): only the K producer
  // waits, before its first claim from the counter.
  if (!a.wait_late) grid_dependency_wait();
  grid_dependents_launch();

  if (warp == R::kProducerWarp || warp == R::kVProducerWarp) {
    // ------------------------------------------------------------ producers
    // One thread issues the Q tiles and the K blocks (for E4M3: both K and V
    // bytes into the staging ring); for bf16 a second warp issues the V
    // blocks, so that a K load never queues behind a V slot still in use.
    if (lane == 0) {
      const bool kq = warp == R::kProducerWarp;
      tma_prefetch_desc(&a.tmap_q);
      tma_prefetch_desc(&a.tmap_k);
      tma_prefetch_desc(&a.tmap_v);
      // Last block issued into each slot, to drain copies in flight on abort.
      int last_k[kKStages], last_v[kVStages], last_8[kF8Stages];
      for (int s = 0; s < kKStages; ++s) last_k[s] = -1;
      for (int s = 0; s < kVStages; ++s) last_v[s] = -1;
      for (int s = 0; s < kF8Stages; ++s) last_8[s] = -1;
      bool ok = true;
      int g = 0, k = 0;  // blocks issued, non-empty items seen
      // The K producer hands out the work: its first item is blockIdx.x, each
      // later one comes from the launch-wide counter (in increasing order,
      // heaviest first), claimed kClaimAhead blocks before the current item
      // ends, so SMs that run faster take more items. Items with nothing to do
      // are skipped, except a tile's first split when the tile has no usable
      // block (its rows are written as empty by the softmax warps).
      // Launches that wait late (direct mode) take their first item before
      // the kernel that zeroes the counter has been waited for.
      int claim = blockIdx.x;
      // The claimed next item is set up (its loads) while this item's last
      // blocks are in flight, right after a block's copies are issued.
      Item pend{};
      int pend_idx = -1;
      bool want_pend = false;
      // Loads item x's Q tile as the kk-th non-empty item's (slot kk % kQBuf).
      auto load_q = [&](int kk, const Item& x) -> bool {
        const int qb = kk % kQBuf;
        if (kk >= kQBuf &&
            !mbar_wait(&sm.q_empty[qb], ((kk / kQBuf) - 1) & 1, fault, kFaultWaitMma, abort))
          return false;
        mbar_expect_tx(&sm.q_full[qb], 2u * 128u * (uint32_t)(G * W));
        for (int c = 0; c < 2; ++c)
          tma_load_3d(q_addr(qb, c), &a.tmap_q, &sm.q_full[qb], c * 64, x.h * G, x.t0);
        return true;
      };
      bool dep_waited = !a.wait_late;
      auto next_claim = [&](int) {
        if (!dep_waited) {
          grid_dependency_wait();
          dep_waited = true;
        }
        return (int)gridDim.x + atomicAdd(a.item_counter, 1);
      };
      for (int ni = 0; ok; ++ni) {
        Item it{};
        int i = -1;
        if (kq) {
          while (claim < a.num_items) {
            const int cand = claim;
            if (cand == pend_idx) it = pend;
            else it = a.direct ? direct_item(a, cand) : item_at(a, cand, item_tile_info(a, cand));
            if (it.t0 >= 0 && (it.n > 0 || (it.split == 0 && it.n_union == 0))) {
              i = cand;
              break;
            }
            claim = next_claim(claim);
          }
          const int slot = ni % kItemRing;
          if (ni >= kItemRing && !mbar_wait(&sm.item_empty[slot], ((ni / kItemRing) - 1) & 1, fault,
                                            kFaultWaitOther, abort)) {
            ok = false;
            break;
          }
          sm.item_idx[slot] = i;
          if (i >= 0) sm.item_ring[slot] = it;
          mbar_arrive(&sm.item_full[slot]);
          if (i < 0) break;
          if (it.n <= kClaimAhead) {
            claim = next_claim(claim);
            want_pend = true;
          }
        } else {
          i = read_item(ni, ok, it);
          if (!ok) break;
          release_item(ni);
          if (i < 0) break;
        }
        if (it.n == 0) continue;
        if (kq && !load_q(k, it)) {
          ok = false;
          break;
        }
        const int32_t* ulist =
            a.union_blocks + ((size_t)it.h * a.max_tiles + it.tile) * a.cap + it.p_begin;
        // Union entries two blocks ahead, page entries one block ahead, so a
        // block's copies never wait on a load chain.
        const int32_t* prow = a.paged ? a.page_table + (size_t)it.b * a.max_pages : nullptr;
        int id1 = meta_ld(ulist, a.direct);
        int id2 = it.n > 1 ? meta_ld(ulist + 1, a.direct) : 0;
        int pg1 = a.paged ? prow[id1] : 0;
        for (int u = 0; u < it.n; ++u, ++g) {
          if (kq && it.n > kClaimAhead && u == it.n - kClaimAhead) {
            claim = next_claim(claim);
            want_pend = true;
          }
          const int blk = id1;
          int page = pg1;
          id1 = id2;
          if (u + 2 < it.n) id2 = meta_ld(ulist + u + 2, a.direct);
          if (a.paged && u + 1 < it.n) pg1 = prow[id1];
          if (a.paged) {
            // An unmapped page reads as zeros (out-of-range TMA box) and is masked.
            if (page < 0 || page >= a.num_pages) page = a.num_pages;
          }
          const int row = it.kv0 + blk * kBlk;
          if (FP8) {
            const int s8 = g % kF8Stages;
            if (g >= kF8Stages && !mbar_wait(&sm.f8_empty[s8], ((g / kF8Stages) - 1) & 1, fault,
                                             kFaultWaitOther, abort)) {
              ok = false;
              break;
            }
            if (a.kv_fp4) {
              // Bulk copies of the page's K and V slices; an unmapped page is
              // not read, and the converters write zeros for it.
              const bool valid = page < a.num_pages;
              sm.f8_valid[s8] = valid ? 1 : 0;
              if (valid) {
                const long long off = (long long)page * a.fp4_page_stride;
                const size_t slice = (size_t)it.h * kFp4Data, sslice = (size_t)it.h * kFp4Scales;
                uint8_t* kst = &sm.k8[s8][0];  // kTile bytes in the E4M3 instance
                uint8_t* vst = &sm.v8[s8][0];
                mbar_expect_tx(&sm.f8_full[s8], 2 * (kFp4Data + kFp4Scales));
                bulk_load(kst, a.fp4_k + off + slice, kFp4Data, &sm.f8_full[s8]);
                bulk_load(kst + kFp4Data, a.fp4_k_scale + off + sslice, kFp4Scales, &sm.f8_full[s8]);
                bulk_load(vst, a.fp4_v + off + slice, kFp4Data, &sm.f8_full[s8]);
                bulk_load(vst + kFp4Data, a.fp4_v_scale + off + sslice, kFp4Scales, &sm.f8_full[s8]);
              } else {
                mbar_arrive(&sm.f8_full[s8]);
              }
            } else if (a.paged) {
              mbar_expect_tx(&sm.f8_full[s8], 2 * kTile);
              tma_load_4d(sm.k8[s8], &a.tmap_k, &sm.f8_full[s8], 0, 0, it.h, page);
              tma_load_4d(sm.v8[s8], &a.tmap_v, &sm.f8_full[s8], 0, 0, it.h, page);
            } else {
              mbar_expect_tx(&sm.f8_full[s8], 2 * kTile);
              tma_load_3d(sm.k8[s8], &a.tmap_k, &sm.f8_full[s8], 0, it.h, row);
              tma_load_3d(sm.v8[s8], &a.tmap_v, &sm.f8_full[s8], 0, it.h, row);
            }
            last_8[s8] = g;
          } else if (kq) {
            const int ks = g % kKStages;
            if (g >= kKStages && !qk_wait(g - kKStages)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&sm.k_full[ks], 2 * kTile);
            for (int c = 0; c < 2; ++c) {
              if (a.paged) tma_load_4d(sm.k[ks][c], &a.tmap_k, &sm.k_full[ks], c * 64, 0, it.h, page);
              else tma_load_3d(sm.k[ks][c], &a.tmap_k, &sm.k_full[ks], c * 64, it.h, row);
            }
            last_k[ks] = g;
            if (want_pend) {
              want_pend = false;
              if (claim < a.num_items) {
                pend = a.direct ? direct_item(a, claim) : item_at(a, claim, item_tile_info(a, claim));
                pend_idx = claim;
              }
            }
          } else {
            const int vs = g % kVStages;
            if (g >= kVStages && !pv_wait(g - kVStages)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&sm.v_full[vs], 2 * kTile);
            for (int c = 0; c < 2; ++c) {
              if (a.paged) tma_load_4d(sm.v[vs][c], &a.tmap_v, &sm.v_full[vs], c * 64, 0, it.h, page);
              else tma_load_3d(sm.v[vs][c], &a.tmap_v, &sm.v_full[vs], c * 64, it.h, row);
            }
            last_v[vs] = g;
          }
        }
        ++k;
      }
      if (!ok) {
        // Let copies already in flight land before the CTA's shared memory is released.
        for (int s = 0; s < kKStages; ++s)
          if (last_k[s] >= 0) mbar_wait(&sm.k_full[s], (last_k[s] / kKStages) & 1, fault, kFaultWaitTma);
        for (int s = 0; s < kVStages; ++s)
          if (last_v[s] >= 0) mbar_wait(&sm.v_full[s], (last_v[s] / kVStages) & 1, fault, kFaultWaitTma);
        for (int s = 0; s < kF8Stages; ++s)
          if (last_8[s] >= 0) mbar_wait(&sm.f8_full[s], (last_8[s] / kF8Stages) & 1, fault, kFaultWaitTma);
      }
    }
  } else if (warp == R::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Walks the block stream twice: QK runs two blocks ahead of PV, across
    // item boundaries, so the softmax of block g overlaps PV(g-1) and QK(g+1).
    if (lane == 0) {
      const uint32_t idS = idesc_16bit_f32(128, 128, false, false, F16);
      const uint32_t idO = idesc_16bit_f32(128, 128, false, true, F16);
      bool ok = true;
      // Descriptors of slot 0; a slot or K step only moves the start-address
      // field (16-byte units), so the issue path adds constants.
      constexpr uint32_t kSlot16 = (2 * kTile) >> 4;  // one K or V slot
      constexpr uint32_t kHalf16 = kTile >> 4;        // second 64-column half
      const uint64_t dq0 = sdesc_sw128(smem_u32(q_addr(0, 0)), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(&sm.k[0][0][0]), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(&sm.v[0][0][0]), kTile, 1024);
      const uint32_t qslot16 = STREAM ? ((uint32_t)(W * G) * 128u) >> 4 : 0u;
      // Ring positions of the QK stream and of the PV stream.
      RingPos<kQBuf> rq;
      RingPos<kKStages> rk;
      RingPos<kSBuf> rs;
      RingPos<kVStages> rv;
      RingPos<kSBuf> rp;
      uint32_t ofree_phase = 0;
      auto issue_qk = [&](const Cursor& c) -> bool {
        if (c.u == 0 && !mbar_wait(&sm.q_full[rq.idx], rq.phase, fault, kFaultWaitTma, abort))
          return false;
        if (!mbar_wait(&sm.k_full[rk.idx], rk.phase, fault, kFaultWaitTma, abort)) return false;
        tc_fence_after();
        const uint64_t dq = dq0 + rq.idx * qslot16, dk = dk0 + rk.idx * kSlot16;
        const uint32_t ts = tbase + rs.idx * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf16 + (kk & 3) * 2;
          mma_ss(ts, dq + off, dk + off, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&sm.qk_done[rs.idx]);
        if (c.u == c.it.n - 1) {
          mma_commit(&sm.q_empty[rq.idx]);
          rq.next();
        }
        rk.next();
        rs.next();
        return true;
      };
      auto issue_pv = [&](const Cursor& c) -> bool {
        // A new item's first PV overwrites O: its previous epilogue must have read it.
        if (c.u == 0 && c.k > 0) {
          if (!mbar_wait(&sm.o_free, ofree_phase, fault, kFaultWaitSoftmax, abort)) return false;
          ofree_phase ^= 1u;
        }
        if (!mbar_wait(&sm.p_full[rp.idx], rp.phase, fault, kFaultWaitSoftmax, abort)) return false;
        if (!mbar_wait(&sm.v_full[rv.idx], rv.phase, fault, kFaultWaitTma, abort)) return false;
        tc_fence_after();
        const uint64_t dv = dv0 + rv.idx * kSlot16;
        const uint32_t tp = tbase + rp.idx * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tbase + kColO, tp + (kk >> 2) * 64 + (kk & 3) * 8, dv + kk * 128, idO,
                 (c.u > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&sm.pv_done[rp.idx]);
        rv.next();
        rp.next();
        return true;
      };
      // Moves a cursor to the next block, reading new items from the ring as
      // it passes item boundaries; false if a read gave up.
      auto cursor_next = [&](Cursor& c) -> bool {
        ++c.g;
        ++c.u;
        while (c.u >= c.it.n) {
          bool okr = true;
          const int i = read_item(c.n, okr, c.it);
          if (!okr) return false;
          release_item(c.n);
          ++c.n;
          if (i < 0) {
            c.valid = false;
            return true;
          }
          c.u = 0;
          if (c.it.n > 0) ++c.k;
        }
        c.valid = true;
        return true;
      };
      Cursor qc, pc;
      qc.n = pc.n = 0;
      qc.u = pc.u = 0;
      qc.k = pc.k = -1;
      qc.g = pc.g = -1;
      qc.it.n = pc.it.n = 0;
      ok = cursor_next(qc) && cursor_next(pc);
      for (int j = 0; ok && j < 2 && qc.valid; ++j) ok = issue_qk(qc) && cursor_next(qc);
      while (ok && pc.valid) {
        if (qc.valid) {
          ok = issue_qk(qc) && cursor_next(qc);
          if (!ok) break;
        }
        ok = issue_pv(pc) && cursor_next(pc);
      }
      // Nothing may be in flight when TMEM is released.
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, fault, kFaultWaitMma);
    }
  } else if (FP8 && warp >= R::kConvWarp0 && warp < R::kConvWarp0 + R::kConvWarps) {
    // ------------------------------------------------------------ E4M3 -> bf16
    const int ct = tid - R::kConvWarp0 * 32;
    int g = 0;
    bool ok = true;
    for (int ni = 0; ok; ++ni) {
      Item it{};
      const int i = read_item(ni, ok, it);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) release_item(ni);
      if (i < 0) break;
      for (int u = 0; u < it.n; ++u, ++g) {
        const int s8 = g % kF8Stages, ks = g % kKStages, vs = g % kVStages;
        if (!mbar_wait(&sm.f8_full[s8], (g / kF8Stages) & 1, fault, kFaultWaitTma, abort) ||
            (g >= kKStages && !qk_wait(g - kKStages))) {
          ok = false;
          break;
        }
        const bool fp4_valid = a.kv_fp4 && sm.f8_valid[s8] != 0;
        if (a.kv_fp4) convert_fp4_tile<R::kConvWarps * 32>(sm.k8[s8], false, fp4_valid, sm.k[ks][0], ct);
        else convert_tile<R::kConvWarps * 32>(sm.k8[s8], sm.k[ks][0], ct);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.k_full[ks]);
        if (g >= kVStages && !pv_wait(g - kVStages)) {
          ok = false;
          break;
        }
        if (a.kv_fp4) convert_fp4_tile<R::kConvWarps * 32>(sm.v8[s8], true, fp4_valid, sm.v[vs][0], ct);
        else convert_tile<R::kConvWarps * 32>(sm.v8[s8], sm.v[vs][0], ct);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sm.v_full[vs]);
          mbar_arrive(&sm.f8_empty[s8]);
        }
      }
    }
  } else if (warp < R::kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax + epilogue
    constexpr int NW = R::kSoftmaxWG;
    constexpr int kHalves = 2 / NW;   // 64-column halves of S and O per warp
    const int q4 = warp & 3;          // TMEM lane quarter
    const int wg = warp >> 2;         // column group (with NW == 2: columns 64*wg..64*wg+63)
    const int row = q4 * 32 + lane;   // TMEM lane
    const int w = row / G, gh = row - w * G;
    const uint32_t lane_base = tbase + ((uint32_t)(q4 * 32) << 16);
    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
    bool ok = true;
    int g = 0;   // blocks consumed
    int xi = 0;  // exchanges with the partner warp so far (two alternating slots)
    // Publishes v to the partner warp (same lanes, other column group) and
    // returns the partner's value; okv becomes the AND over both warps. A
    // slot is rewritten two exchanges later, after the partner has passed the
    // barrier that follows its read.
    auto exchange = [&](float v, bool& okv) -> float {
      float* slot = sm.xch + (xi & 1) * 256;
      slot[wg * 128 + row] = v;
      okv = pair_barrier_and(q4, okv);
      ++xi;
      return slot[(1 - wg) * 128 + row];
    };
    // Item epilogue: out = O / l and the natural-log LSE (or the fp32
    // partials of a split item). It is deferred until the next item's first
    // block has published its P, so that the next item's first PV (which
    // overwrites O) waits only for O to be read, not for a whole softmax
    // pass as well.
    struct Epi {
      bool valid;
      int glast, tail, split, nsplit;
      float m_ref, l;
      bool active;
      size_t orow;
    };
    Epi pe{};
    pe.valid = false;
    constexpr bool kDefer = kDeferEpilogue;
    auto run_epilogue = [&](const Epi& e) -> bool {
      bool okk = pv_wait(e.glast);
      okk = !__any_sync(0xffffffffu, !okk);
      float lt = e.l;  // the row's full sum
      if constexpr (NW == 2) lt += exchange(e.l, okk);
      if (!okk) return false;
      tc_fence_after();
      const size_t part = ((size_t)(e.tail < 0 ? 0 : e.tail) * a.splits + e.split) * a.rows_part;
      const bool has = lt > 0.f;
      const float os = a.out_scale;  // output scale (the NVFP4 V global scale; else 1)
      const float inv = has ? os / lt : 0.f;
      auto store_half = [&](int half, const float* o) {
        if (!e.active) return;
        if (e.nsplit == 1) {
          uint4* dst =
              reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + e.orow * 128);
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
            uint4 v4 = make_uint4(0u, 0u, 0u, 0u);
            if (has)
              v4 = make_uint4(pack_x2<F16>(o[c] * inv, o[c + 1] * inv),
                              pack_x2<F16>(o[c + 2] * inv, o[c + 3] * inv),
                              pack_x2<F16>(o[c + 4] * inv, o[c + 5] * inv),
                              pack_x2<F16>(o[c + 6] * inv, o[c + 7] * inv));
            dst[(half * 64 + c) >> 3] = v4;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(a.part_o + (part + row) * 128 + half * 64);
#pragma unroll
          for (int c = 0; c < 64; c += 4)
            dst[c >> 2] = make_float4(o[c] * os, o[c + 1] * os, o[c + 2] * os, o[c + 3] * os);
        }
      };
      // O is released (the next item's first PV may overwrite it) as soon as
      // this warp's columns are in registers, before the global stores.
      {
        float o[64];
        tmem_ld64(lane_base + kColO + wg * kHalves * 64, o);
        if (kHalves == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.o_free);
        }
        store_half(wg * kHalves, o);
      }
      if (kHalves == 2) {
        float o[64];
        tmem_ld64(lane_base + kColO + 64, o);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.o_free);
        store_half(1, o);
      }
      if (e.nsplit == 1) {
        if (e.active && wg == 0 && a.lse != nullptr)
          a.lse[e.orow] = has ? (e.m_ref + log2f(lt)) * 0.69314718055994531f : -INFINITY;
        return true;
      }
      if (e.active && wg == 0) {
        a.part_ml[(part + row) * 2] = e.m_ref;
        a.part_ml[(part + row) * 2 + 1] = lt;
      }
      // The unit's splits are combined by merge_splits_kernel after this launch.
      return true;
    };
    // Both warps of a pair agree on each read's outcome before going on
    // (they meet at paired barriers below).
    for (int ni = 0;; ++ni) {
      Item it{};
      const int cur = read_item(ni, ok, it);
      __syncwarp();
      if (ok && lane == 0) release_item(ni);
      if (NW == 2) ok = pair_barrier_and(q4, ok);
      if (!ok || cur < 0) break;
      if (it.t0 < 0) continue;
      const int nw = min(W, it.seq_q0 + it.lq - it.t0);
      const bool active = row < W * G && w < nw;
      const size_t orow = (size_t)(it.t0 + w) * a.num_qo_heads + (size_t)it.h * G + gh;
      // Items holding blocks of this unit (a whole unit is a single item).
      const int nsplit = it.tail < 0 ? 1 : (it.n_union + a.pps - 1) / a.pps;
      if (it.n == 0) {
        // A tile with no usable block at all: out = 0, lse = -inf.
        if (it.split == 0 && it.n_union == 0 && active) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + orow * 128);
#pragma unroll
          for (int c = 0; c < 8 * kHalves; ++c) dst[wg * 8 * kHalves + c] = make_uint4(0u, 0u, 0u, 0u);
          if (wg == 0 && a.lse != nullptr) a.lse[orow] = -INFINITY;
        }
        continue;
      }
      const long long pos = (long long)it.lk - it.lq + (it.t0 + w - it.seq_q0);
      const size_t unit = (size_t)it.h * a.max_tiles + it.tile;
      const uint32_t* mrow = a.member + (unit * W + (active ? w : 0)) * a.words;
      const int32_t* ulist = a.union_blocks + unit * a.cap + it.p_begin;
      float m_ref = -INFINITY, l = 0.f;  // l: sum over this warp's columns
      // Per-block metadata, loaded ahead so that no load waits on another in
      // the block loop: union entries two blocks ahead, page entries one block
      // ahead (kept raw until used). Direct mode: every union entry is the
      // token's own (usable) block.
      uint32_t mword = !active ? 0u : a.direct ? ~0u : __ldg(mrow + (it.p_begin >> 5));
      const int32_t* prow = a.paged ? a.page_table + (size_t)it.b * a.max_pages : nullptr;
      int id1 = meta_ld(ulist, a.direct);
      int id2 = it.n > 1 ? meta_ld(ulist + 1, a.direct) : 0;
      int pg1 = a.paged ? __ldg(prow + id1) : 0;
      for (int u = 0; u < it.n; ++u) {
        const int gg = g + u, bb = gg % kSBuf;
        const int upos = it.p_begin + u;  // position in the tile's union list
        const int blk = id1;
        const int pg = pg1;
        id1 = id2;
        if (u + 2 < it.n) id2 = meta_ld(ulist + u + 2, a.direct);
        if (a.paged && u + 1 < it.n) pg1 = __ldg(prow + id1);
        const bool page_ok = !a.paged || (pg >= 0 && pg < a.num_pages);
        bool mem = active && ((mword >> (upos & 31)) & 1u) && page_ok;
        if (u + 1 < it.n && ((upos + 1) & 31) == 0 && active && !a.direct)
          mword = __ldg(mrow + ((upos + 1) >> 5));
        int lim = 127;
        if (mem) {
          long long last = (long long)it.lk - 1;
          if (a.causal && pos < last) last = pos;
          last -= (long long)blk * kBlk;
          if (last < 0) mem = false;
          else if (last < 127) lim = (int)last;
        }
        // QK(gg) done: S is readable, and every PV up to gg-3 (the last user
        // of this P buffer) has completed.
        ok = qk_wait(gg);
        ok = !__any_sync(0xffffffffu, !ok);
        if (NW == 1 && !ok) break;
        tc_fence_after();
        const bool warp_mem = __any_sync(0xffffffffu, mem);
        const bool warp_masked = __any_sync(0xffffffffu, mem && lim < 127);
        const uint32_t scol = lane_base + bb * 128;  // S_b; P_b in columns 0..31 and 64..95
        float alpha = 1.f;
        bool rescale = false;
        float2 acc = make_float2(0.f, 0.f);
        if constexpr (NW == 2) {
          const uint32_t gcol = scol + wg * 64;  // this warp's 64 S columns; its P: the first 32
          float sv[64];
          float mx = -INFINITY;
          if (ok && warp_mem) {
            tmem_ld64(gcol, sv);
            if (warp_masked) {
#pragma unroll
              for (int c = 0; c < 64; ++c)
                if (wg * 64 + c > lim) sv[c] = -INFINITY;
            }
            mx = row_max64(sv);
          }
          mx = fmaxf(mx, exchange(mx, ok));
          if (!ok) break;
          if (warp_mem) {
            update_max(mem, mx, a.scale_log2, m_ref, l, alpha, rescale);
            // Non-member rows use -inf as their offset, so every P entry is 0.
            const float neg_m = mem ? -m_ref : -INFINITY;
            exp_pack_store<64, F16>(sv, sc2, neg_m, acc, gcol);
          } else {
            // QK(gg) overwrote this buffer: P must be rewritten (zeros) every block.
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = 0u;
            tmem_st32(gcol, pk);
          }
        } else {
          if (warp_mem) {
            float mx = -INFINITY;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float sv[64];
              tmem_ld64(scol + half * 64, sv);
              if (warp_masked) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                  if (half * 64 + c > lim) sv[c] = -INFINITY;
              }
              mx = fmaxf(mx, row_max64(sv));
            }
            update_max(mem, mx, a.scale_log2, m_ref, l, alpha, rescale);
            const float neg_m = mem ? -m_ref : -INFINITY;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float sv[64];
              tmem_ld64(scol + half * 64, sv);
              if (warp_masked) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                  if (half * 64 + c > lim) sv[c] = -INFINITY;
              }
              // Written over columns of this half that were just read.
              exp_pack_store<64, F16>(sv, sc2, neg_m, acc, scol + half * 64);
            }
          } else {
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = 0u;
            tmem_st32(scol, pk);
            tmem_st32(scol + 64, pk);
          }
        }
        if (mem) l += acc.x + acc.y;
        // Rows rescale identically in both warps of a pair (same maxima).
        if (__any_sync(0xffffffffu, rescale)) {
          // O must hold every PV of this item up to gg-1 before it is rescaled.
          ok = pv_wait(gg - 1);
          ok = !__any_sync(0xffffffffu, !ok);
          if (NW == 2) ok = pair_barrier_and(q4, ok);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int hh = 0; hh < kHalves; ++hh) {
            const uint32_t ocol = lane_base + kColO + (wg * kHalves + hh) * 64;
            float o[64];
            tmem_ld64(ocol, o);
            uint32_t ow[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) ow[c] = __float_as_uint(o[c] * alpha);
            tmem_st64(ocol, ow);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[bb]);
        if (kDefer && u == 0 && pe.valid) {
          ok = run_epilogue(pe);
          pe.valid = false;
          if (!ok) break;
        }
      }
      if (!ok) break;
      if constexpr (kDefer) {
        // This item's epilogue runs once the next item's first block has
        // published its P (or after the last item).
        pe.valid = true;
        pe.glast = g + it.n - 1;
        pe.tail = it.tail;
        pe.split = it.split;
        pe.nsplit = nsplit;
        pe.m_ref = m_ref;
        pe.l = l;
        pe.active = active;
        pe.orow = orow;
        g += it.n;
      } else {
        // Decode layout: the epilogue in line at the item's end (the same
        // work as run_epilogue; the deferred form measured slower there).
        // ---------------------------------------------------- item epilogue
        const int glast = g + it.n - 1;
        ok = pv_wait(glast);
        ok = !__any_sync(0xffffffffu, !ok);
        float lt = l;  // the row's full sum
        if constexpr (NW == 2) lt += exchange(l, ok);
        if (!ok) break;
        tc_fence_after();
        const size_t part = ((size_t)(it.tail < 0 ? 0 : it.tail) * a.splits + it.split) * a.rows_part;
        const bool has = lt > 0.f;
        const float os = a.out_scale;  // output scale (the NVFP4 V global scale; else 1)
        const float inv = has ? os / lt : 0.f;
        auto store_half = [&](int half, const float* o) {
          if (!active) return;
          if (nsplit == 1) {
            uint4* dst =
                reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + orow * 128);
  #pragma unroll
            for (int c = 0; c < 64; c += 8) {
              uint4 v4 = make_uint4(0u, 0u, 0u, 0u);
              if (has)
                v4 = make_uint4(pack_x2<F16>(o[c] * inv, o[c + 1] * inv),
                                pack_x2<F16>(o[c + 2] * inv, o[c + 3] * inv),
                                pack_x2<F16>(o[c + 4] * inv, o[c + 5] * inv),
                                pack_x2<F16>(o[c + 6] * inv, o[c + 7] * inv));
              dst[(half * 64 + c) >> 3] = v4;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(a.part_o + (part + row) * 128 + half * 64);
  #pragma unroll
            for (int c = 0; c < 64; c += 4)
              dst[c >> 2] = make_float4(o[c] * os, o[c + 1] * os, o[c + 2] * os, o[c + 3] * os);
          }
        };
        // O is released (the next item's first PV may overwrite it) as soon as
        // this warp's columns are in registers, before the global stores.
        {
          float o[64];
          tmem_ld64(lane_base + kColO + wg * kHalves * 64, o);
          if (kHalves == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.o_free);
          }
          store_half(wg * kHalves, o);
        }
        if (kHalves == 2) {
          float o[64];
          tmem_ld64(lane_base + kColO + 64, o);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.o_free);
          store_half(1, o);
        }
        g += it.n;
        if (nsplit == 1) {
          if (active && wg == 0 && a.lse != nullptr)
            a.lse[orow] = has ? (m_ref + log2f(lt)) * 0.69314718055994531f : -INFINITY;
          continue;
        }
        if (active && wg == 0) {
          a.part_ml[(part + row) * 2] = m_ref;
          a.part_ml[(part + row) * 2 + 1] = lt;
        }
        // The unit's splits are combined by merge_splits_kernel after this launch.
      }
    }
    if (kDefer && ok && pe.valid) ok = run_epilogue(pe);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}


// Launches `kernel` so that it may start while the previous kernel on the
// stream is finishing (programmatic dependent launch); the kernel itself
// waits with grid_dependency_wait() before reading that kernel's results.
template <class Kernel>
cudaError_t launch_dependent(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
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

// Combines the fp32 partials of the tail units whose union was split across
// several work items: for each such unit and active row, with
// M = max_s m_s, L = sum_s 2^(m_s - M) l_s, out = sum_s 2^(m_s - M) O_s / L and
// lse = (M + log2 L) ln 2 (m in log2 units of the scaled logits), M taken
// as a running maximum over groups of four splits whose loads are issued
// together. A split with no visible key (m = -inf) contributes nothing. One
// warp per (tail unit, row); each lane owns four of the 128 dims.
__global__ void __launch_bounds__(256) merge_splits_kernel(const __grid_constant__ PrefillArgs a) {
  // The union metadata read below is final before this launch may begin: the
  // attention kernel lets it launch only after waiting for the union kernel.
  // Only the partials need the wait, so it comes after the metadata loads.
  // In direct mode the attention kernel writes the metadata; a one-token tile
  // is its own query row (t0 = tile, one token), so only the union length is
  // read, after the wait, together with the first splits' partials.
  constexpr int kU = 4;
  const int warp_global = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp_global >= a.tail_units * a.rows_part) return;
  const int t = warp_global / a.rows_part, row = warp_global - t * a.rows_part;
  const int unit = a.whole_units + t;
  const int h = unit / a.max_tiles;  // same head-major order as item_at
  const int tile = a.max_tiles - 1 - (unit - h * a.max_tiles);
  const int G = a.num_qo_heads / a.num_kv_heads;
  const int w = row / G, gh = row - w * G;
  if (row >= a.tile_tokens * G) return;
  int t0 = tile, n_union = 0;
  if (!a.direct) {
    t0 = __ldg(a.tile_info + 2 * tile);
    if (t0 < 0) return;
    n_union = __ldg(a.union_len + (size_t)h * a.max_tiles + tile);
    if ((n_union + a.pps - 1) / a.pps <= 1) return;  // written directly by the attention kernel
    const int b = __ldg(a.tile_info + 2 * tile + 1);
    if (w >= min(a.tile_tokens, __ldg(a.cu_q + b + 1) - t0)) return;
  }
  const size_t p0 = (size_t)t * a.splits * a.rows_part + row;
  grid_dependency_wait();  // partials (and, in direct mode, metadata) of the attention kernel
  if (a.direct) n_union = __ldcg(a.union_len + (size_t)h * a.max_tiles + tile);
  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  // Loads of a group run ahead of the union length (bounded by the launch's
  // split count); splits past the unit's own count are ignored.
  for (int s0 = 0; s0 < a.splits; s0 += kU) {
    float2 ml[kU];
    float4 ov[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const size_t pr = p0 + (size_t)min(s0 + j, a.splits - 1) * a.rows_part;
      ml[j] = __ldcg(reinterpret_cast<const float2*>(a.part_ml) + pr);
      ov[j] = __ldcg(reinterpret_cast<const float4*>(a.part_o + pr * 128) + lane);
    }
    const int nsplit = (n_union + a.pps - 1) / a.pps;
    if (nsplit <= 1) return;  // direct mode: written directly by the attention kernel
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      if (s0 + j >= nsplit || ml[j].x == -INFINITY) continue;
      if (ml[j].x > M) {
        const float r = ex2(M - ml[j].x);  // 0 while M is -inf (L and acc are 0 then)
        L *= r;
        acc.x *= r;
        acc.y *= r;
        acc.z *= r;
        acc.w *= r;
        M = ml[j].x;
      }
      const float f = ex2(ml[j].x - M);
      L += f * ml[j].y;
      acc.x += f * ov[j].x;
      acc.y += f * ov[j].y;
      acc.z += f * ov[j].z;
      acc.w += f * ov[j].w;
    }
    if (s0 + kU >= nsplit) break;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const size_t orow = (size_t)(t0 + w) * a.num_qo_heads + (size_t)h * G + gh;
  uint2* dst = reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + orow * 128) + lane;
  *dst = a.f16 ? make_uint2(pack_f16x2(acc.x * inv, acc.y * inv), pack_f16x2(acc.z * inv, acc.w * inv))
               : make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (lane == 0 && a.lse != nullptr)
    a.lse[orow] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

template <bool FP8, bool STREAM, bool F16>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
  // Up to 1 KiB of slack for aligning the base, within the per-block limit
  // (the kernel checks that the slack it got covers its base's offset).
  const int optin = device_smem_optin();
  if (optin <= 0) return cudaErrorInvalidDevice;
  size_t smem = sizeof(PrefillSmem<FP8, STREAM>) + 1024;
  if (smem > (size_t)optin) smem = (size_t)optin;
  cudaError_t e = set_smem_limit((const void*)prefill_kernel<FP8, STREAM, F16>, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = a.num_items < device_sm_count() ? a.num_items : device_sm_count();
  if (grid <= 0) return cudaSuccess;
  e = launch_dependent(prefill_kernel<FP8, STREAM, F16>, dim3(grid), dim3(Roles<FP8>::kThreads),
                       smem, s, a);
  if (e != cudaSuccess || a.splits <= 1 || a.tail_units == 0) return e;
  const long long warps = (long long)a.tail_units * a.rows_part;
  return launch_dependent(merge_splits_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s,
                          a);
}

}  // namespace

int device_sm_count() {
  static int cache[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  if (a.kv_fp8) return launch_t<true, false, false>(a, s);
  // Split launches are the memory-bound, decode-sized ones; their Q slots
  // share a region when a tile has at most 64 rows (whole 8-row groups).
  const int rows = a.tile_tokens * (a.num_qo_heads / a.num_kv_heads);
  const bool stream = a.splits > 1 && a.tail_units > 0 && rows <= 64 && rows % 8 == 0;
  if (a.f16) return stream ? launch_t<false, true, true>(a, s) : launch_t<false, false, true>(a, s);
  return stream ? launch_t<false, true, false>(a, s) : launch_t<false, false, false>(a, s);
}

}  // namespace msa
