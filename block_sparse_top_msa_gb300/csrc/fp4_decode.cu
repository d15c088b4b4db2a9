// Packed-NVFP4 paged sparse decode ("flashinfer.msa_ops.msa_sparse_attention",
// the packed-NVFP4 paged route; "prepare_msa_nvfp4_sparse_decode", parameters
// k, k_scale, v_scale and the global scales).
//
// One work unit is (query token, KV head): the G <= 16 query heads of the
// token that share the KV head are the 16 rows of warp-level m16n8k16 MMAs,
// and the unit attends over the blocks of the token's own q2k row (usable ids
// only, each once). Per block, TMA brings the K and V code slices (64-byte
// swizzled, so every shared-memory read below is conflict-free) and bulk
// copies bring both scale slices into one ring stage; the block is then
// dequantized in registers on its way into the MMAs, never written back:
//   E2M1 pair -> f16 pair (cvt), times the E4M3 block scale (exact in f16:
//   at most 6 significant bits, magnitude 2^-10 .. 2688).
// q (bf16) enters the MMAs as f16 scaled by a power of two per row (exact for
// every bf16 value of the row down to 2^-28 of its largest magnitude), and
// that power of two is taken back out of the fp32 scores with the softmax
// scale, log2(e) and the K global scale. P is rounded to f16 (11 significant
// bits) for the PV MMA; S and O accumulate in fp32; the V global scale
// multiplies the output.
//
// A CTA has two groups of four consumer warps and one producer warp. The
// groups take alternate blocks of a unit. Within a group, warp w computes S
// for tokens 32w .. 32w + 31 of the block, the group agrees on the block's row
// maxima through shared memory, each warp publishes its P fragments, and warp
// w then computes O for dims 32w .. 32w + 31 over all 128 tokens. At the end
// of a unit the two groups' (m, l, O) are combined.
//
// QK^T takes its contraction dims in a permuted order: thread (n, c) of a
// fragment holds dims 32c .. 32c + 31 of a K row (one 16-byte load), and q is
// loaded in the same order, so a k-step pairs the same dims on both sides.
// PV takes its B fragments from ldmatrix.trans over 8 tokens x 32 dims; a
// thread receives dims 4n .. 4n + 3 of two tokens, and byte permutes form the
// (token, token) pairs of one dim. Output column n of n-tile i is dim
// 32w + 4n + i.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace msa {
namespace {

constexpr int kF4Stages = 5;
constexpr uint32_t kOffVc = kFp4Data;                    // V codes
constexpr uint32_t kOffKs = 2 * kFp4Data;                // K scales (token-major)
constexpr uint32_t kOffVs = 2 * kFp4Data + kFp4Scales;   // V scales (4 x 4 tiles)
constexpr uint32_t kF4StageBytes = 2 * kFp4Data + 2 * kFp4Scales;  // 18432, a multiple of 1024
constexpr int kF4Consumers = 8;
constexpr int kF4Threads = (kF4Consumers + 1) * 32;
constexpr int kF4MaxTopk = 64;
constexpr int kBarUnit = 5;  // named barrier of all consumer warps (1..4: the groups' own)

struct F4Smem {
  uint8_t stage[kF4Stages][kF4StageBytes];
  // P fragments [group][k-step][lane]: the A operand of one PV k-step as
  // four f16 pairs per lane. One buffer per group suffices: a warp writes the
  // next block's P only after the group's first barrier of that block, which
  // every warp of the group reaches after its last read of this block's P.
  // At the end of a unit the whole array is the buffer through which group 1
  // hands its O to group 0.
  uint4 pfrag[2][8][32];
  float rmax[2][16][4];     // [group][row][warp]: per-warp block row maxima
  float lpart[2][4][16];    // [group][warp][row]: partial row sums at the end of a unit
  float mrun[2][16];        // [group][row]: running maxima at the end of a unit
  int32_t list_page[kF4MaxTopk];  // producer: the unit's pages, in list order
  int32_t list_cnt[kF4MaxTopk];   // producer: visible keys of each listed block
  int32_t unit_n[2];              // listed blocks of the unit in slot k % 2
  int32_t n_agreed;               // the count every consumer warp uses for the unit
  int32_t stage_cnt[kF4Stages];   // visible keys of the block in a stage
  uint64_t full[kF4Stages];
  uint64_t empty[kF4Stages];
  uint64_t ufull[2];
  uint64_t uempty[2];
  int abort;
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

// Byte `k` of w (two E2M1 codes, element 2i in the low nibble) as an f16 pair.
MSA_DEV uint32_t e2m1x2_f16x2(uint32_t w, int k) {
  uint32_t d;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(d)
      : "r"(w >> (8 * k)));
  return d;
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
MSA_DEV void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
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

__global__ void __maxnreg__(112)
    fp4_decode_kernel(const __grid_constant__ Fp4DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  F4Smem& sm = *reinterpret_cast<F4Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kF4Stages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.ufull[i], 1);
      mbar_init(&sm.uempty[i], kF4Consumers);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();
  volatile int* abort = &sm.abort;
  const int hkv = a.num_kv_heads;
  const int units = a.total_q * hkv;

  if (warp == kF4Consumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&a.tmap_kc);
      tma_prefetch_desc(&a.tmap_vc);
    }
    uint32_t seq = 0;
    int k = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++k) {
      if (*abort) break;
      const int tk = u / hkv, h = u - tk * hkv;
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
      if (v0) {
        const int e = __popc(m0 & below);
        sm.list_page[e] = pg0;
        sm.list_cnt[e] = (int)min(128LL, pos - (long long)id0 * kBlk + 1);
      }
      if (v1) {
        const int e = n0 + __popc(m1 & below);
        sm.list_page[e] = pg1;
        sm.list_cnt[e] = (int)min(128LL, pos - (long long)id1 * kBlk + 1);
      }
      __syncwarp();
      const int slot = k & 1;
      if (lane == 0) {
        if (k >= 2) mbar_wait(&sm.uempty[slot], ((k >> 1) - 1) & 1, a.fault, kFaultWaitOther, abort);
        sm.unit_n[slot] = n;
        mbar_arrive(&sm.ufull[slot]);
        for (int e = 0; e < n; ++e, ++seq) {
          const int st = (int)(seq % kF4Stages);
          const uint32_t round = seq / kF4Stages;
          if (round > 0 &&
              !mbar_wait(&sm.empty[st], (round - 1) & 1, a.fault, kFaultWaitOther, abort))
            break;
          const int page = sm.list_page[e];
          sm.stage_cnt[st] = sm.list_cnt[e];
          const uint32_t dst = smem_u32(sm.stage[st]);
          mbar_expect_tx(&sm.full[st], kF4StageBytes);
          tma_4d(dst, &a.tmap_kc, &sm.full[st], 0, 0, h, page);
          tma_4d(dst + kOffVc, &a.tmap_vc, &sm.full[st], 0, 0, h, page);
          const long long off = (long long)page * a.page_stride + (long long)h * kFp4Scales;
          bulk_g2s(dst + kOffKs, a.k_scale + off, kFp4Scales, &sm.full[st]);
          bulk_g2s(dst + kOffVs, a.v_scale + off, kFp4Scales, &sm.full[st]);
        }
      }
      seq = __shfl_sync(0xffffffffu, seq, 0);
      __syncwarp();
    }
    // No copy may still be landing when the CTA exits: wait for the last
    // fill of every stage (already complete unless the consumers gave up).
    if (lane == 0) {
      for (int st = 0; st < kF4Stages; ++st) {
        if ((uint32_t)st >= seq) break;
        const uint32_t last = seq - 1 - ((seq - 1 - st) % kF4Stages);  // last sequence number on st
        mbar_wait(&sm.full[st], (last / kF4Stages) & 1, a.fault, kFaultWaitTma);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int gp = warp >> 2, wg = warp & 3;
  const int g = lane >> 2, c = lane & 3;
  const int G = a.G;
  const int hq = a.num_qo_heads;
  const float os = a.out_scale;
  uint32_t seq_base = 0;
  int k = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x, ++k) {
    const int tk = u / hkv, h = u - tk * hkv;
    const int slot = k & 1;
    mbar_wait(&sm.ufull[slot], (k >> 1) & 1, a.fault, kFaultWaitOther, abort);
    if (warp == 0 && lane == 0) sm.n_agreed = min(max(sm.unit_n[slot], 0), kF4MaxTopk);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.uempty[slot]);
    named_bar(kBarUnit, kF4Consumers * 32);
    const int n = sm.n_agreed;

    // q rows g and g + 8 (heads h * G + row), dims 32c .. 32c + 31, as f16
    // pairs scaled by 2^e per row; rs = the fp32 factor back to log2 units.
    uint32_t qa[2][16];
    float rs[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = g + 8 * r;
      uint4 raw[4];
      if (row < G) {
        const uint4* src = reinterpret_cast<const uint4*>(
            a.q + ((size_t)tk * hq + (size_t)h * G + row) * kHeadDim + 32 * c);
#pragma unroll
        for (int v = 0; v < 4; ++v) raw[v] = __ldg(src + v);
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
        frexpf(amax, &E);               // amax = f * 2^E, f in [0.5, 1)
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

    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int x = 0; x < 4; ++x) o[i][x] = 0.f;

    for (int e = gp; e < n; e += 2) {
      const uint32_t sq = seq_base + (uint32_t)e;
      const int st = (int)(sq % kF4Stages);
      mbar_wait(&sm.full[st], (sq / kF4Stages) & 1, a.fault, kFaultWaitTma, abort);
      const int cnt = sm.stage_cnt[st];
      const uint32_t sbase = smem_u32(sm.stage[st]);

      // ---- S = q K^T for tokens 32 wg .. 32 wg + 31 (n-tiles j: 8 tokens each)
      float acc[4][4];
      uint4 kw[4];
      uint32_t sA[4], sB[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int t = 32 * wg + 8 * j + g;
        kw[j] = lds128(sbase + t * 64 + 16 * (c ^ ((t >> 1) & 3)));
        const uint32_t s2 = e4m3x2_f16x2(lds16(sbase + kOffKs + t * 8 + 2 * c));
        sA[j] = prmt(s2, s2, 0x1010u);  // scale of dims 32c .. 32c + 15
        sB[j] = prmt(s2, s2, 0x3232u);  // scale of dims 32c + 16 .. 32c + 31
#pragma unroll
        for (int x = 0; x < 4; ++x) acc[j][x] = 0.f;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t a0[4] = {qa[0][4 * q], qa[1][4 * q], qa[0][4 * q + 1], qa[1][4 * q + 1]};
        const uint32_t a1[4] = {qa[0][4 * q + 2], qa[1][4 * q + 2], qa[0][4 * q + 3],
                                qa[1][4 * q + 3]};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w = q == 0 ? kw[j].x : q == 1 ? kw[j].y : q == 2 ? kw[j].z : kw[j].w;
          const uint32_t sc = q < 2 ? sA[j] : sB[j];
          const uint32_t p0 = hmul2_u(e2m1x2_f16x2(w, 0), sc);
          const uint32_t p1 = hmul2_u(e2m1x2_f16x2(w, 1), sc);
          const uint32_t p2 = hmul2_u(e2m1x2_f16x2(w, 2), sc);
          const uint32_t p3 = hmul2_u(e2m1x2_f16x2(w, 3), sc);
          mma_f16(acc[j], a0, p0, p1);
          mma_f16(acc[j], a1, p2, p3);
        }
      }

      // ---- block row maxima, agreed across the group's four warps
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int t = 32 * wg + 8 * j + 2 * c + (x & 1);
          const float v = t < cnt ? acc[j][x] * rs[x >> 1] : -INFINITY;
          acc[j][x] = v;
          mx[x >> 1] = fmaxf(mx[x >> 1], v);
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      }
      if (c == 0) {
        sm.rmax[gp][g][wg] = mx[0];
        sm.rmax[gp][g + 8][wg] = mx[1];
      }
      named_bar(1 + 2 * gp, 128);
      float al[2], mu[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float4 rm = *reinterpret_cast<const float4*>(&sm.rmax[gp][g + 8 * r][0]);
        const float mn = fmaxf(m[r], fmaxf(fmaxf(rm.x, rm.y), fmaxf(rm.z, rm.w)));
        mu[r] = mn == -INFINITY ? 0.f : mn;  // reference while nothing is visible yet
        al[r] = ex2f(m[r] - mu[r]);
        m[r] = mn;
      }
      float ps[2] = {0.f, 0.f};
      uint32_t pk[4][2];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float p0 = ex2f(acc[j][0] - mu[0]), p1 = ex2f(acc[j][1] - mu[0]);
        const float p2 = ex2f(acc[j][2] - mu[1]), p3 = ex2f(acc[j][3] - mu[1]);
        ps[0] += p0 + p1;
        ps[1] += p2 + p3;
        const __half2 h01 = __floats2half2_rn(p0, p1), h23 = __floats2half2_rn(p2, p3);
        pk[j][0] = *reinterpret_cast<const uint32_t*>(&h01);
        pk[j][1] = *reinterpret_cast<const uint32_t*>(&h23);
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
      // n-tiles (0, 1) are the A operand of PV k-step 2 wg, (2, 3) of 2 wg + 1
      const uint32_t pbase = smem_u32(&sm.pfrag[gp][0][0]);
      sts128(pbase + ((2 * wg) * 32 + lane) * 16, make_uint4(pk[0][0], pk[0][1], pk[1][0], pk[1][1]));
      sts128(pbase + ((2 * wg + 1) * 32 + lane) * 16,
             make_uint4(pk[2][0], pk[2][1], pk[3][0], pk[3][1]));
      named_bar(2 + 2 * gp, 128);

      // ---- O += P V for dims 32 wg .. 32 wg + 31 over the block's 128 tokens
      const int grp = 2 * wg + (g >> 2);  // V scale index of dims 32 wg + 4g .. + 3
#pragma unroll
      for (int sp = 0; sp < 8; sp += 2) {
        uint32_t vr[4];
        {
          const int mi = lane >> 3;
          const int T = 16 * (sp + (mi >> 1)) + 8 * (mi & 1) + (lane & 7);
          ldsm_x4_trans(sbase + kOffVc + T * 64 + 16 * (wg ^ ((T >> 1) & 3)), vr);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int ss = sp + hh;
          const uint4 af4 = lds128(pbase + (ss * 32 + lane) * 16);
          const uint32_t af[4] = {af4.x, af4.y, af4.z, af4.w};
          uint32_t bb[2][4];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int t0 = 16 * ss + 8 * half + 2 * c;
            uint32_t s2 = lds16(sbase + kOffVs + 32 * (t0 >> 2) + 16 * (grp >> 2) + 4 * (grp & 3) +
                                (t0 & 3));
            if (cnt < kBlk) {  // keys past the visible ones weigh nothing
              if (t0 >= cnt) s2 &= 0xff00u;
              if (t0 + 1 >= cnt) s2 &= 0x00ffu;
            }
            const uint32_t sc = e4m3x2_f16x2(s2);
            const uint32_t r = vr[2 * hh + half];
            const uint32_t x0 = e2m1x2_f16x2(r, 0), x1 = e2m1x2_f16x2(r, 1);
            const uint32_t y0 = e2m1x2_f16x2(r, 2), y1 = e2m1x2_f16x2(r, 3);
            bb[half][0] = hmul2_u(prmt(x0, y0, 0x5410u), sc);
            bb[half][1] = hmul2_u(prmt(x0, y0, 0x7632u), sc);
            bb[half][2] = hmul2_u(prmt(x1, y1, 0x5410u), sc);
            bb[half][3] = hmul2_u(prmt(x1, y1, 0x7632u), sc);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) mma_f16(o[i], af, bb[0][i], bb[1][i]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[st]);
    }

    // ---- combine the two groups: M = max m, L = sum 2^(m - M) l
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
    }
    if (c == 0) {
      sm.lpart[gp][wg][g] = l[0];
      sm.lpart[gp][wg][g + 8] = l[1];
      if (wg == 0) {
        sm.mrun[gp][g] = m[0];
        sm.mrun[gp][g + 8] = m[1];
      }
    }
    named_bar(kBarUnit, kF4Consumers * 32);
    float f[2], L[2], M[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = g + 8 * r;
      const float ma = sm.mrun[0][row], mb = sm.mrun[1][row];
      float la = 0.f, lb = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        la += sm.lpart[0][w][row];
        lb += sm.lpart[1][w][row];
      }
      M[r] = fmaxf(ma, mb);
      if (M[r] == -INFINITY) {
        f[r] = 0.f;
        L[r] = 0.f;
      } else {
        const float fa = ex2f(ma - M[r]), fb = ex2f(mb - M[r]);
        f[r] = gp == 0 ? fa : fb;
        L[r] = fa * la + fb * lb;
      }
    }
    // Both groups' P buffers are free here (every PV of the unit is done) and
    // stay free until group 0 has read them: group 1 next writes P after the
    // barrier that opens the next unit.
    const uint32_t xo = smem_u32(&sm.pfrag[0][0][0]) + (wg * 32 + lane) * 64;
    if (gp == 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        sts128(xo + 16 * i, make_uint4(__float_as_uint(o[i][0] * f[0]), __float_as_uint(o[i][1] * f[0]),
                                       __float_as_uint(o[i][2] * f[1]), __float_as_uint(o[i][3] * f[1])));
    }
    named_bar(kBarUnit, kF4Consumers * 32);
    if (gp == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 x = lds128(xo + 16 * i);
        o[i][0] = o[i][0] * f[0] + __uint_as_float(x.x);
        o[i][1] = o[i][1] * f[0] + __uint_as_float(x.y);
        o[i][2] = o[i][2] * f[1] + __uint_as_float(x.z);
        o[i][3] = o[i][3] * f[1] + __uint_as_float(x.w);
      }
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
    seq_base += (uint32_t)n;
  }
}

}  // namespace

cudaError_t launch_fp4_decode(const Fp4DecodeArgs& a, cudaStream_t s) {
  const long long units = (long long)a.total_q * a.num_kv_heads;
  if (units <= 0) return cudaSuccess;
  const int smem = (int)sizeof(F4Smem) + 1024;
  cudaError_t e = set_smem_limit((const void*)fp4_decode_kernel, smem);
  if (e != cudaSuccess) return e;
  const long long slots = 2LL * device_sm_count();
  const int grid = (int)(units < slots ? units : slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kF4Threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fp4_decode_kernel, a);
}

}  // namespace msa
