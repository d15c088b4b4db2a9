// Packed-NVFP4 paged sparse decode ("flashinfer.msa_ops.msa_sparse_attention",
// the packed-NVFP4 paged route; "prepare_msa_nvfp4_sparse_decode", parameters
// k, k_scale, v_scale and the global scales).
//
// One unit is (query token, KV head): the G <= 16 query heads of the token
// that share the KV head are the 16 rows of warp-level m16n8k16 MMAs, and the
// unit attends over the blocks of the token's own q2k row (usable ids only,
// each once). Two launches:
//
// fp4_list_kernel, one warp per unit, writes the unit's block list to the
// workspace: topk slots of (page, visible keys), the usable blocks first in
// row order, then holes (page -1); and zeroes the unit's merge counter.
//
// fp4_decode_kernel: CTAs of four warps, three per SM. The units' list slots,
// taken in order, form V = units * topk positions; CTA i takes the contiguous
// range [i V / n, (i + 1) V / n), so every CTA gets the same number of blocks
// to within one (holes are skipped). The range cuts units into segments; a
// segment that is a whole unit writes the unit's output, the others write
// (m, l, O) partials and the last of a unit's segments to finish (a counter
// per unit) combines them.
//
// Per block, TMA brings the K and V code slices (64-byte swizzled, so every
// shared-memory read below is conflict-free) and bulk copies bring the scale
// slices into a three-stage ring. Inside a segment, PV of block j - 1 runs
// together with QK^T of block j, so at the first barrier of block j every warp
// is done with block j - 1, and block j + 2 is issued into its stage. A
// segment's q rows arrive by bulk copy into one of two slots, one segment
// ahead. The block is dequantized in registers on its way into the MMAs,
// never written back:
//   E2M1 pair -> f16 pair (cvt), times the E4M3 block scale (exact in f16:
//   at most 6 significant bits, magnitude 2^-10 .. 2688).
// q (bf16) enters the MMAs as f16 scaled by a power of two per row (exact for
// every bf16 value of the row down to 2^-28 of its largest magnitude), and
// that power of two is taken back out of the fp32 scores with the softmax
// scale, log2(e) and the K global scale. P is rounded to f16 (11 significant
// bits) for the PV MMA; S and O accumulate in fp32; the V global scale
// multiplies the output.
//
// Warp w computes S for tokens 32w .. 32w + 31 of a block, the four warps
// agree on the block's row maxima through shared memory, each publishes its
// P fragments, and warp w then computes O for dims 32w .. 32w + 31 over all
// 128 tokens. QK^T takes its contraction dims in a permuted order: thread
// (n, c) of a fragment holds dims 32c .. 32c + 31 of a K row (one 16-byte
// load), and q is loaded in the same order, so a k-step pairs the same dims on
// both sides. PV takes its B fragments from ldmatrix.trans over 8 tokens x 32
// dims; a thread receives dims 4n .. 4n + 3 of two tokens, and byte permutes
// form the (token, token) pairs of one dim. Output column n of n-tile i is dim
// 32w + 4n + i.
#include <cuda_fp16.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace msa {
namespace {

constexpr uint32_t kOffVc = kFp4Data;                    // V codes
constexpr uint32_t kOffKs = 2 * kFp4Data;                // K scales (token-major)
constexpr uint32_t kOffVs = 2 * kFp4Data + kFp4Scales;   // V scales (4 x 4 tiles)
constexpr uint32_t kF4StageBytes = 2 * kFp4Data + 2 * kFp4Scales;  // 18432, a multiple of 1024
constexpr uint32_t kF4HalfBytes = kFp4Data + kFp4Scales;           // one side of a block
constexpr int kF4Threads = 128;
// Three CTAs per SM (154 registers a thread, no spills) measured 4% faster
// than four (128 registers, the compiler's cap at four).
constexpr int kF4CtasPerSm = 3;
constexpr int kF4Stages = 3;

struct F4Smem {
  // Block b in stage b % 3: K codes | V codes | K scales | V scales. Once
  // every warp has finished QK^T of the block, its P fragments ([k-step][lane]:
  // the A operand of one PV k-step, 4 KB) overwrite the start of the K codes.
  uint8_t stage[kF4Stages][kF4StageBytes];
  uint16_t q[2][16 * kHeadDim];  // bf16 q rows of segment s in slot s % 2 (G rows used)
  float rmax[16][4];  // [row][warp]: per-warp block row maxima
  float lsum[16][4];  // [row][warp]: per-warp row sums at the end of a segment
  int last;           // this CTA combines the current unit's segments
  int abort;
  uint64_t kfull[kF4Stages], vfull[kF4Stages], qfull[2];
};

MSA_DEV void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

MSA_DEV void tma_4d(uint32_t dst, const void* map, uint64_t* bar, int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

MSA_DEV void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

MSA_DEV void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

MSA_DEV uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
MSA_DEV uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return v;
}
MSA_DEV void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// The four bytes of w (two E2M1 codes each, element 2i in the low nibble) as
// four f16 pairs, byte k in d[k]. The bytes are taken apart by one vector
// move, which measured 30% faster than a shift per byte.
MSA_DEV void e2m1x8_f16x2(uint32_t w, uint32_t (&d)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(w));
}
// Two E4M3 codes (low byte first) as an f16 pair.
MSA_DEV uint32_t e4m3x2_f16x2(uint32_t two) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)two));
  return d;
}
MSA_DEV uint32_t hmul2_u(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
MSA_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
MSA_DEV float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
MSA_DEV float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Request b holding query token t (cu_q ascending, empty requests allowed).
MSA_DEV int request_of(const int32_t* cu_q, int batch, int total_q, int t, int& q0, int& q1) {
  const int guess = min(batch - 1, (int)((long long)t * batch / max(total_q, 1)));
  q0 = __ldcg(cu_q + guess);
  q1 = __ldcg(cu_q + guess + 1);
  if (q0 <= t && t < q1) return guess;
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldcg(cu_q + mid) <= t) lo = mid; else hi = mid - 1;
  }
  q0 = __ldcg(cu_q + lo);
  q1 = __ldcg(cu_q + lo + 1);
  return lo;
}

// The V list positions are cut into n ranges [i V / n, (i + 1) V / n): the
// start of range i, and the range holding position x.
MSA_DEV long long range_start(int i, long long V, int n) { return (long long)i * V / n; }
MSA_DEV int range_of(long long x, long long V, int n) { return (int)(((x + 1) * n - 1) / V); }

// ------------------------------------------------------------ block lists
__global__ void __launch_bounds__(256) fp4_list_kernel(const __grid_constant__ Fp4DecodeArgs a) {
  grid_dependents_launch();
  grid_dependency_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hkv = a.num_kv_heads;
  const long long u = (long long)blockIdx.x * 8 + warp;
  if (u >= (long long)a.total_q * hkv) return;
  const int tk = (int)(u / hkv), h = (int)(u - (long long)tk * hkv);
  int q0, q1;
  const int b = request_of(a.cu_q, a.batch, a.total_q, tk, q0, q1);
  const int lk = __ldcg(a.seqused_k + b);
  const long long pos = (long long)lk - (q1 - q0) + (tk - q0);  // last visible key
  const int nblk = min((lk + kBlk - 1) / kBlk, a.max_pages);
  const int32_t* row = a.q2k + ((size_t)h * a.total_q + tk) * a.topk;
  const int id0 = lane < a.topk ? __ldcg(row + lane) : -1;
  const int id1 = lane + 32 < a.topk ? __ldcg(row + lane + 32) : -1;
  bool v0 = id0 >= 0 && id0 < nblk && (long long)id0 * kBlk <= pos;
  bool v1 = id1 >= 0 && id1 < nblk && (long long)id1 * kBlk <= pos;
  // keep the first occurrence of each id
  for (int j = 0; j < a.topk; ++j) {
    const int idj = __shfl_sync(0xffffffffu, j < 32 ? id0 : id1, j & 31);
    if (j < lane && idj == id0) v0 = false;
    if (j < lane + 32 && idj == id1) v1 = false;
  }
  int pg0 = -1, pg1 = -1;
  if (v0) {
    pg0 = __ldcg(a.page_table + (size_t)b * a.max_pages + id0);
    v0 = pg0 >= 0 && pg0 < a.num_pages;  // an unmapped page holds no key
  }
  if (v1) {
    pg1 = __ldcg(a.page_table + (size_t)b * a.max_pages + id1);
    v1 = pg1 >= 0 && pg1 < a.num_pages;
  }
  const unsigned m0 = __ballot_sync(0xffffffffu, v0), m1 = __ballot_sync(0xffffffffu, v1);
  const unsigned below = (1u << lane) - 1u;
  const int n0 = __popc(m0), n = n0 + __popc(m1);
  int2* list = a.list + (size_t)u * a.topk;
  if (v0)
    list[__popc(m0 & below)] = make_int2(pg0, (int)min(128LL, pos - (long long)id0 * kBlk + 1));
  if (v1)
    list[n0 + __popc(m1 & below)] =
        make_int2(pg1, (int)min(128LL, pos - (long long)id1 * kBlk + 1));
  if (lane >= n && lane < a.topk) list[lane] = make_int2(-1, 0);
  if (lane + 32 >= n && lane + 32 < a.topk) list[lane + 32] = make_int2(-1, 0);
  if (lane == 0) a.arrive[u] = 0;
}

// A window of 32 consecutive list positions, one per lane (warp-uniform use).
struct ListWindow {
  long long base;
  int page, cnt;
};

MSA_DEV void window_load(ListWindow& w, const int2* list, long long b, long long end) {
  w.base = b;
  const long long x = b + (threadIdx.x & 31);
  int2 e = make_int2(-1, 0);
  if (x < end) e = __ldcg(list + x);
  w.page = e.x;
  w.cnt = e.y;
}

// The first position in [x, lim) holding a usable block, or lim.
MSA_DEV long long next_valid(ListWindow& w, const int2* list, long long x, long long lim,
                             long long end) {
  while (x < lim) {
    if (x < w.base || x >= w.base + 32) window_load(w, list, x, end);
    const unsigned valid = __ballot_sync(0xffffffffu, w.page >= 0);
    const unsigned rest = valid & (0xffffffffu << (int)(x - w.base));
    if (rest != 0u) {
      const long long y = w.base + __ffs(rest) - 1;
      return y < lim ? y : lim;
    }
    x = w.base + 32;
  }
  return lim;
}

// Rows g and g + 8 of a unit's output (dims 32 wg + 8c .. + 7, the fragment
// order of this kernel's PV) as bf16 O / L times the output scale, and their
// LSE (natural log); rows past G are padding and are not stored.
MSA_DEV void store_rows_bf16(const Fp4DecodeArgs& a, const float (&o)[4][4], const float (&M)[2],
                             const float (&L)[2], long long tk, long long h, int g, int c, int wg,
                             int G, int hq, float os) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = g + 8 * r;
    if (row >= G) continue;
    const size_t orow = (size_t)tk * hq + (size_t)h * G + row;
    const float inv = L[r] > 0.f ? os / L[r] : 0.f;
    uint4 v;
    v.x = pack_bf16x2(o[0][2 * r] * inv, o[1][2 * r] * inv);
    v.y = pack_bf16x2(o[2][2 * r] * inv, o[3][2 * r] * inv);
    v.z = pack_bf16x2(o[0][2 * r + 1] * inv, o[1][2 * r + 1] * inv);
    v.w = pack_bf16x2(o[2][2 * r + 1] * inv, o[3][2 * r + 1] * inv);
    *reinterpret_cast<uint4*>(a.out + orow * kHeadDim + 32 * wg + 8 * c) = v;
    if (wg == 0 && c == 0 && a.lse != nullptr)
      a.lse[orow] = L[r] > 0.f ? (M[r] + log2f(L[r])) * 0.69314718055994531f : -INFINITY;
  }
}

// ------------------------------------------------------------ decode
__global__ void __launch_bounds__(kF4Threads, kF4CtasPerSm)
    fp4_decode_kernel(const __grid_constant__ Fp4DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  F4Smem& sm = *reinterpret_cast<F4Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  const int wg = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kF4Stages; ++s) {
      mbar_init(&sm.kfull[s], 1);
      mbar_init(&sm.vfull[s], 1);
    }
    mbar_init(&sm.qfull[0], 1);
    mbar_init(&sm.qfull[1], 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int hkv = a.num_kv_heads, topk = a.topk, G = a.G, hq = a.num_qo_heads;
  const long long V = (long long)a.total_q * hkv * topk;
  const int ng = gridDim.x, gid = blockIdx.x;
  const long long start = range_start(gid, V, ng), end = range_start(gid + 1, V, ng);
  volatile int* abort = &sm.abort;
  const bool issuer = threadIdx.x == 0;
  if (issuer) {
    tma_prefetch_desc(&a.tmap_kc);
    tma_prefetch_desc(&a.tmap_vc);
  }
  grid_dependency_wait();  // the block lists (and, through their launch, every input)
  if (start >= end) return;
  const int2* list = a.list;
  const long long u_first = start / topk, u_last = (end - 1) / topk;

  // ---- issuer: warp 0 walks the range, thread 0 issues block b's K and V
  // into stage b % 3 (blocks 0 .. 2 up front, block b + 2 at the first
  // barrier of block b, when stage (b + 2) % 3 is no longer read).
  ListWindow iw;
  iw.base = -64;
  iw.page = -1;
  iw.cnt = 0;
  long long ix = start;
  uint32_t nis = 0;  // blocks issued
  auto issue_next = [&]() {  // warp 0, uniform
    const long long y = next_valid(iw, list, ix, end, end);
    if (y >= end) {
      ix = end;
      return;
    }
    const int page = __shfl_sync(0xffffffffu, iw.page, (int)(y - iw.base));
    ix = y + 1;
    if (issuer) {
      // the stage was last written by this CTA's P stores (generic proxy)
      fence_async_smem();
      const int st = nis % kF4Stages;
      const int h = (int)((y / topk) % hkv);
      const uint32_t dst = smem_u32(sm.stage[st]);
      const long long off = (long long)page * a.page_stride + (long long)h * kFp4Scales;
      mbar_expect_tx(&sm.kfull[st], kF4HalfBytes);
      tma_4d(dst, &a.tmap_kc, &sm.kfull[st], 0, 0, h, page);
      bulk_g2s(dst + kOffKs, a.k_scale + off, kFp4Scales, &sm.kfull[st]);
      mbar_expect_tx(&sm.vfull[st], kF4HalfBytes);
      tma_4d(dst + kOffVc, &a.tmap_vc, &sm.vfull[st], 0, 0, h, page);
      bulk_g2s(dst + kOffVs, a.v_scale + off, kFp4Scales, &sm.vfull[st]);
    }
    ++nis;
  };
  if (wg == 0)
    for (int i = 0; i < kF4Stages; ++i) issue_next();
  // q rows of segment s (unit u_first + s) into slot s % 2: segments 0 and 1
  // up front, segment s + 1 when segment s starts (every warp has then
  // converted segment s - 1's rows).
  const uint32_t qbytes = (uint32_t)G * kHeadDim * 2;
  long long nq = 0;  // segments whose q was issued (thread 0)
  auto issue_q = [&](long long sg) {
    const long long uu = u_first + sg;
    const long long tq = uu / hkv, hh = uu - tq * hkv;
    fence_async_smem();  // the slot was last read by this CTA's generic loads
    mbar_expect_tx(&sm.qfull[sg & 1], qbytes);
    bulk_g2s(smem_u32(sm.q[sg & 1]), a.q + ((size_t)tq * hq + (size_t)hh * G) * kHeadDim, qbytes,
             &sm.qfull[sg & 1]);
    nq = sg + 1;
  };
  if (issuer) {
    issue_q(0);
    if (u_last > u_first) issue_q(1);
  }

  // ---- per-warp pieces of a block
  uint32_t j = 0;      // blocks consumed (the one whose S is being computed)
  uint32_t qa[2][16] = {};  // q rows g, g + 8, dims 32c .. 32c + 31, f16 pairs (scaled by 2^e)
  float rs[2];         // 2^-e times the softmax scale, log2(e) and the K global scale
  float acc[4][4];     // S of this warp's 32 tokens (n-tiles of 8)
  float o[4][4];       // O of this warp's 32 dims
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  uint4 kw[4];
  uint32_t sA[4], sB[4];
  const int grp = 2 * wg + (g >> 2);  // V scale index of dims 32 wg + 4g .. + 3

  // QK^T of a block: load this warp's K rows and scales, zero S.
  auto qk_load = [&](uint32_t sbase) {
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int t = 32 * wg + 8 * jj + g;
      kw[jj] = lds128(sbase + t * 64 + 16 * (c ^ ((t >> 1) & 3)));
      const uint32_t s2 = e4m3x2_f16x2(lds16(sbase + kOffKs + t * 8 + 2 * c));
      sA[jj] = prmt(s2, s2, 0x1010u);  // scale of dims 32c .. 32c + 15
      sB[jj] = prmt(s2, s2, 0x3232u);  // scale of dims 32c + 16 .. 32c + 31
#pragma unroll
      for (int y = 0; y < 4; ++y) acc[jj][y] = 0.f;
    }
  };
  // k-steps 2q, 2q + 1 of QK^T: word q of each K row (dims 32c + 8q .. + 7).
  auto qk_part = [&](int q) {
    const uint32_t a0[4] = {qa[0][4 * q], qa[1][4 * q], qa[0][4 * q + 1], qa[1][4 * q + 1]};
    const uint32_t a1[4] = {qa[0][4 * q + 2], qa[1][4 * q + 2], qa[0][4 * q + 3],
                            qa[1][4 * q + 3]};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const uint32_t w = q == 0 ? kw[jj].x : q == 1 ? kw[jj].y : q == 2 ? kw[jj].z : kw[jj].w;
      const uint32_t sc = q < 2 ? sA[jj] : sB[jj];
      uint32_t d4[4];
      e2m1x8_f16x2(w, d4);
      const uint32_t b0 = hmul2_u(d4[0], sc), b1 = hmul2_u(d4[1], sc);
      const uint32_t b2 = hmul2_u(d4[2], sc), b3 = hmul2_u(d4[3], sc);
      mma_f16(acc[jj], a0, b0, b1);
      mma_f16(acc[jj], a1, b2, b3);
    }
  };
  // PV k-steps 2q, 2q + 1 (tokens 32q .. 32q + 31) for this warp's 32 dims;
  // P of the block is in its stage's K-code region.
  auto pv_part = [&](int q, uint32_t sbase, int cnt) {
    uint32_t vr[4];
    {
      const int mi = lane >> 3;
      const int T = 32 * q + 16 * (mi >> 1) + 8 * (mi & 1) + (lane & 7);
      ldsm_x4_trans(sbase + kOffVc + T * 64 + 16 * (wg ^ ((T >> 1) & 3)), vr);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int ss = 2 * q + hh;
      const uint4 af4 = lds128(sbase + (ss * 32 + lane) * 16);
      const uint32_t af[4] = {af4.x, af4.y, af4.z, af4.w};
      uint32_t bb[2][4];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int t0 = 16 * ss + 8 * half + 2 * c;
        uint32_t s2 =
            lds16(sbase + kOffVs + 32 * (t0 >> 2) + 16 * (grp >> 2) + 4 * (grp & 3) + (t0 & 3));
        if (cnt < kBlk) {  // keys past the visible ones weigh nothing
          if (t0 >= cnt) s2 &= 0xff00u;
          if (t0 + 1 >= cnt) s2 &= 0x00ffu;
        }
        const uint32_t sc = e4m3x2_f16x2(s2);
        const uint32_t r = vr[2 * hh + half];
        uint32_t d4[4];  // token t0: d4[0], d4[1]; token t0 + 1: d4[2], d4[3]
        e2m1x8_f16x2(r, d4);
        const uint32_t x0 = d4[0], x1 = d4[1], y0 = d4[2], y1 = d4[3];
        bb[half][0] = hmul2_u(prmt(x0, y0, 0x5410u), sc);
        bb[half][1] = hmul2_u(prmt(x0, y0, 0x7632u), sc);
        bb[half][2] = hmul2_u(prmt(x1, y1, 0x5410u), sc);
        bb[half][3] = hmul2_u(prmt(x1, y1, 0x7632u), sc);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) mma_f16(o[i], af, bb[0][i], bb[1][i]);
    }
  };
  // Block j's S (in acc) to P: the four warps agree on the block's row
  // maxima, block j + 2 is issued, O and l are rescaled, and each warp puts
  // its P fragments (the A operands of PV k-steps 2 wg, 2 wg + 1) into the
  // block's K-code region, whose K every warp has finished reading.
  auto softmax_phase = [&](uint32_t sbase, int cnt) {
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        float v = acc[jj][y] * rs[y >> 1];
        if (cnt < kBlk && 32 * wg + 8 * jj + 2 * c + (y & 1) >= cnt) v = -INFINITY;
        acc[jj][y] = v;
        mx[y >> 1] = fmaxf(mx[y >> 1], v);
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    if (c == 0) {
      sm.rmax[g][wg] = mx[0];
      sm.rmax[g + 8][wg] = mx[1];
    }
    __syncthreads();
    // block j + 2 goes into the stage of block j - 1, which every warp has
    // finished (its PV came before this barrier); blocks 0 .. 2 went up front
    if (wg == 0 && nis < j + kF4Stages) issue_next();
    float al[2], mu[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float4 rm = *reinterpret_cast<const float4*>(&sm.rmax[g + 8 * r][0]);
      const float mn = fmaxf(m[r], fmaxf(fmaxf(rm.x, rm.y), fmaxf(rm.z, rm.w)));
      mu[r] = mn == -INFINITY ? 0.f : mn;  // reference while nothing is visible yet
      al[r] = ex2f(m[r] - mu[r]);
      m[r] = mn;
    }
    float ps[2] = {0.f, 0.f};
    uint32_t pk[4][2];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const float e0 = ex2f(acc[jj][0] - mu[0]), e1 = ex2f(acc[jj][1] - mu[0]);
      const float e2 = ex2f(acc[jj][2] - mu[1]), e3 = ex2f(acc[jj][3] - mu[1]);
      ps[0] += e0 + e1;
      ps[1] += e2 + e3;
      const __half2 h01 = __floats2half2_rn(e0, e1), h23 = __floats2half2_rn(e2, e3);
      pk[jj][0] = *reinterpret_cast<const uint32_t*>(&h01);
      pk[jj][1] = *reinterpret_cast<const uint32_t*>(&h23);
    }
    l[0] = l[0] * al[0] + ps[0];
    l[1] = l[1] * al[1] + ps[1];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[i][0] *= al[0];
      o[i][1] *= al[0];
      o[i][2] *= al[1];
      o[i][3] *= al[1];
    }
    sts128(sbase + ((2 * wg) * 32 + lane) * 16, make_uint4(pk[0][0], pk[0][1], pk[1][0], pk[1][1]));
    sts128(sbase + ((2 * wg + 1) * 32 + lane) * 16,
           make_uint4(pk[2][0], pk[2][1], pk[3][0], pk[3][1]));
    __syncthreads();
  };

  ListWindow cw;
  cw.base = -64;
  cw.page = -1;
  cw.cnt = 0;
  const float os = a.out_scale;
  for (long long u = u_first; u <= u_last; ++u) {
    const long long p0 = max(start, u * topk), p1 = min(end, (u + 1) * topk);
    const long long tk = u / hkv, h = u - tk * hkv;
    __syncthreads();  // every warp is past the previous segment (q slot, lsum reuse)
    const long long sg = u - u_first;
    if (issuer && sg >= 1 && u + 1 <= u_last) issue_q(sg + 1);
    mbar_wait(&sm.qfull[sg & 1], (uint32_t)(sg >> 1) & 1u, a.fault, kFaultWaitTma, abort);
    // q rows g and g + 8 as f16 pairs scaled by 2^e per row; rs = the fp32
    // factor back to log2 units of the scaled logits.
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = g + 8 * r;
      uint4 raw[4];
      if (row < G) {
#pragma unroll
        for (int v = 0; v < 4; ++v)
          raw[v] = lds128(smem_u32(&sm.q[sg & 1][row * kHeadDim + 32 * c + 8 * v]));
      } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) raw[v] = make_uint4(0u, 0u, 0u, 0u);
      }
      float amax = 0.f;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint32_t w[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w[i] & 0xffffu)),
                                   fabsf(bf16_bits_to_float(w[i] >> 16))));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      int e = 0;
      if (amax > 0.f && amax <= 3.0e38f) {
        int E;
        frexpf(amax, &E);                 // amax = f * 2^E, f in [0.5, 1)
        e = min(max(15 - E, -100), 100);  // largest scaled magnitude below 2^15
      }
      const float up = ldexpf(1.f, e);
      rs[r] = ldexpf(a.scale_log2, -e);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint32_t w[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 hv = __floats2half2_rn(bf16_bits_to_float(w[i] & 0xffffu) * up,
                                               bf16_bits_to_float(w[i] >> 16) * up);
          qa[r][4 * v + i] = *reinterpret_cast<const uint32_t*>(&hv);
        }
      }
    }
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int y = 0; y < 4; ++y) o[i][y] = 0.f;

    // Blocks of the segment: S of the first alone, then PV of block i - 1
    // together with S of block i, then PV of the last.
    long long x = next_valid(cw, list, p0, p1, end);
    if (x < p1) {
      int cnt = __shfl_sync(0xffffffffu, cw.cnt, (int)(x - cw.base));
      uint32_t sbase = smem_u32(sm.stage[j % kF4Stages]);
      mbar_wait(&sm.kfull[j % kF4Stages], (j / kF4Stages) & 1u, a.fault, kFaultWaitTma, abort);
      qk_load(sbase);
#pragma unroll
      for (int q = 0; q < 4; ++q) qk_part(q);
      softmax_phase(sbase, cnt);
      while (true) {
        x = next_valid(cw, list, x + 1, p1, end);
        const uint32_t jp = j;  // the block whose PV is pending
        const uint32_t pbase = sbase;
        const int pcnt = cnt;
        mbar_wait(&sm.vfull[jp % kF4Stages], (jp / kF4Stages) & 1u, a.fault, kFaultWaitTma, abort);
        ++j;
        if (x >= p1) {
#pragma unroll
          for (int q = 0; q < 4; ++q) pv_part(q, pbase, pcnt);
          break;
        }
        cnt = __shfl_sync(0xffffffffu, cw.cnt, (int)(x - cw.base));
        sbase = smem_u32(sm.stage[j % kF4Stages]);
        mbar_wait(&sm.kfull[j % kF4Stages], (j / kF4Stages) & 1u, a.fault, kFaultWaitTma, abort);
        qk_load(sbase);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          qk_part(q);
          pv_part(q, pbase, pcnt);
        }
        softmax_phase(sbase, cnt);
      }
    }

    // ---- the segment's rows: L = the sum of the warps' partial sums
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
    }
    if (c == 0) {
      sm.lsum[g][wg] = l[0];
      sm.lsum[g + 8][wg] = l[1];
    }
    __syncthreads();
    float L[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float4 ls = *reinterpret_cast<const float4*>(&sm.lsum[g + 8 * r][0]);
      L[r] = (ls.x + ls.y) + (ls.z + ls.w);
    }
    const int g_first = range_of(u * topk, V, ng), g_last = range_of(u * topk + topk - 1, V, ng);
    if (g_first == g_last) {  // the whole unit is this CTA's
      store_rows_bf16(a, o, m, L, tk, h, g, c, wg, G, hq, os);
      continue;
    }
    // The segment's partial: slot 0 when the segment opens this CTA's range,
    // else slot 1 (it closes the range). O unnormalised, by (row, dim).
    const int slot = start >= u * topk ? 0 : 1;
    float* po = a.part_o + ((size_t)gid * 2 + slot) * 16 * kHeadDim;
    float* pml = a.part_ml + ((size_t)gid * 2 + slot) * 16 * 2;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = g + 8 * r;
      __stcg(reinterpret_cast<float4*>(po + row * kHeadDim + 32 * wg + 8 * c),
             make_float4(o[0][2 * r], o[1][2 * r], o[2][2 * r], o[3][2 * r]));
      __stcg(reinterpret_cast<float4*>(po + row * kHeadDim + 32 * wg + 8 * c + 4),
             make_float4(o[0][2 * r + 1], o[1][2 * r + 1], o[2][2 * r + 1], o[3][2 * r + 1]));
      if (wg == 0 && c == 0) {
        __stcg(pml + row * 2, m[r]);
        __stcg(pml + row * 2 + 1, L[r]);
      }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) sm.last = atomicAdd(a.arrive + u, 1) == g_last - g_first ? 1 : 0;
    __syncthreads();
    if (sm.last == 0) continue;
    __threadfence();
    // This CTA finished the unit's last segment: M = max m, L = sum 2^(m - M) l,
    // O = sum 2^(m - M) O_s over every segment's partial.
    float MM[2] = {-INFINITY, -INFINITY};
    for (int gi = g_first; gi <= g_last; ++gi) {
      const int sl = range_start(gi, V, ng) >= u * topk ? 0 : 1;
      const float* ml = a.part_ml + ((size_t)gi * 2 + sl) * 16 * 2;
#pragma unroll
      for (int r = 0; r < 2; ++r) MM[r] = fmaxf(MM[r], __ldcg(ml + (g + 8 * r) * 2));
    }
    float LL[2] = {0.f, 0.f};
    float oo[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int y = 0; y < 4; ++y) oo[i][y] = 0.f;
    for (int gi = g_first; gi <= g_last; ++gi) {
      const int sl = range_start(gi, V, ng) >= u * topk ? 0 : 1;
      const float* ml = a.part_ml + ((size_t)gi * 2 + sl) * 16 * 2;
      const float* op = a.part_o + ((size_t)gi * 2 + sl) * 16 * kHeadDim;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = g + 8 * r;
        const float f = MM[r] == -INFINITY ? 0.f : ex2f(__ldcg(ml + row * 2) - MM[r]);
        LL[r] += f * __ldcg(ml + row * 2 + 1);
        const float4 lo =
            __ldcg(reinterpret_cast<const float4*>(op + row * kHeadDim + 32 * wg + 8 * c));
        const float4 hi =
            __ldcg(reinterpret_cast<const float4*>(op + row * kHeadDim + 32 * wg + 8 * c + 4));
        oo[0][2 * r] += f * lo.x;
        oo[1][2 * r] += f * lo.y;
        oo[2][2 * r] += f * lo.z;
        oo[3][2 * r] += f * lo.w;
        oo[0][2 * r + 1] += f * hi.x;
        oo[1][2 * r + 1] += f * hi.y;
        oo[2][2 * r + 1] += f * hi.z;
        oo[3][2 * r + 1] += f * hi.w;
      }
    }
    store_rows_bf16(a, oo, MM, LL, tk, h, g, c, wg, G, hq, os);
  }

  // No copy may still be landing when the CTA exits (every one was consumed
  // unless a wait gave up): wait for the last fill of each stage.
  if (issuer) {
    for (uint32_t st = 0; st < (uint32_t)kF4Stages && st < nis; ++st) {
      const uint32_t last = nis - 1 - ((nis - 1 - st) % kF4Stages);
      mbar_wait(&sm.kfull[st], (last / kF4Stages) & 1u, a.fault, kFaultWaitTma);
      mbar_wait(&sm.vfull[st], (last / kF4Stages) & 1u, a.fault, kFaultWaitTma);
    }
    for (long long sl = 0; sl < 2 && sl < nq; ++sl) {
      const long long last = nq - 1 - ((nq - 1 - sl) % 2);
      mbar_wait(&sm.qfull[sl], (uint32_t)(last >> 1) & 1u, a.fault, kFaultWaitTma);
    }
  }
}

}  // namespace

size_t fp4_decode_workspace_bytes(long long units, int topk) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  return up((size_t)units * topk * sizeof(int2)) + up((size_t)units * sizeof(int32_t)) +
         up((size_t)kFp4DecodeMaxCtas * 2 * 16 * 2 * sizeof(float)) +
         up((size_t)kFp4DecodeMaxCtas * 2 * 16 * kHeadDim * sizeof(float));
}

void place_fp4_decode_workspace(Fp4DecodeArgs* a, uint8_t* ws, long long units, int topk) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  size_t off = 0;
  a->list = reinterpret_cast<int2*>(ws + off);
  off += up((size_t)units * topk * sizeof(int2));
  a->arrive = reinterpret_cast<int32_t*>(ws + off);
  off += up((size_t)units * sizeof(int32_t));
  a->part_ml = reinterpret_cast<float*>(ws + off);
  off += up((size_t)kFp4DecodeMaxCtas * 2 * 16 * 2 * sizeof(float));
  a->part_o = reinterpret_cast<float*>(ws + off);
}

cudaError_t launch_fp4_decode(const Fp4DecodeArgs& a, cudaStream_t s) {
  const long long units = (long long)a.total_q * a.num_kv_heads;
  if (units <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((units + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, fp4_list_kernel, a);
  if (e != cudaSuccess) return e;
  const int smem = (int)sizeof(F4Smem) + 1024;
  e = set_smem_limit((const void*)fp4_decode_kernel, smem);
  if (e != cudaSuccess) return e;
  // Several CTAs per SM need the largest shared-memory carveout (set once per
  // device; a repeated set is harmless).
  {
    static std::atomic<unsigned long long> carveout_set{0};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if ((carveout_set.load() & bit) == 0) {
      e = cudaFuncSetAttribute((const void*)fp4_decode_kernel,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      carveout_set.fetch_or(bit);
    }
  }
  const long long V = units * a.topk;
  long long grid = (long long)kF4CtasPerSm * device_sm_count();
  if (grid > kFp4DecodeMaxCtas) grid = kFp4DecodeMaxCtas;
  if (grid > V) grid = V;
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kF4Threads);
  cfg.dynamicSmemBytes = smem;
  return cudaLaunchKernelEx(&cfg, fp4_decode_kernel, a);
}

}  // namespace msa
