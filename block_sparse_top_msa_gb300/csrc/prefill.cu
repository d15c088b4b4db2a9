// MSA sparse attention prefill for sm_103a ("flashinfer.msa_ops.msa_sparse_attention":
// each query attends only the top-K KV blocks selected in q2k_indices; query
// tokens are processed in tiles, each running one online softmax over the
// union of the blocks its tokens selected, writing the final output directly).
//
// One CTA per (query tile, KV head). A tile is W = 128 / G consecutive query
// tokens of one sequence, i.e. 128 rows (token w, query head g) = one
// tcgen05 M=128 tile; row r lives in TMEM lane r. For each block u of the
// tile's union list:
//   producer warp : TMA-gathers K_u and V_u (128 tokens x 128 dims) into a
//                   two-stage shared-memory ring (flat rows cu_k[b] + 128*id,
//                   or page page_table[b, id]); for E4M3 K/V the bytes land in
//                   a staging ring and converter warps upconvert them exactly
//                   to bf16 in the MMA's swizzled layout;
//   MMA warp      : S_u = Q K_u^T (fp32, TMEM, double-buffered), then, once
//                   the softmax has produced P_{u-1}, O += P_{u-1} V_{u-1}
//                   with P read from TMEM;
//   softmax warps : thread r loads its S row, masks keys by block membership
//                   of its token, causality (key <= Lk - Lq + i) and the
//                   sequence end, updates the running max (rescaling O only
//                   when the max grows by more than 2^8), writes P = 2^(s*scale*log2e - m)
//                   as bf16 into TMEM, and at the end writes O / l and the
//                   natural-log LSE.
// Rows whose token did not select block u get P = 0 for it, so each row's
// result is exactly its own blocks' softmax attention.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tmem_wide.cuh"

namespace msa {
namespace {

constexpr int kStages = 2;      // bf16 K/V ring
constexpr int kF8Stages = 2;    // E4M3 staging ring
constexpr int kTile = 16384;    // bytes of one 128-row x 128-byte swizzled tile
constexpr float kRescaleLog2 = 8.0f;

// TMEM column map (512 columns allocated).
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP0 = 384, kColP1 = 448;

template <bool FP8>
struct __align__(1024) PrefillSmem {
  uint8_t q[2][kTile];
  uint8_t k[kStages][2][kTile];
  uint8_t v[kStages][2][kTile];
  uint8_t k8[FP8 ? kF8Stages : 1][FP8 ? kTile : 16];
  uint8_t v8[FP8 ? kF8Stages : 1][FP8 ? kTile : 16];
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t f8_full[kF8Stages];
  uint64_t f8_empty[kF8Stages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <bool FP8>
struct Roles {
  static constexpr int kSoftmaxWarps = 4;
  static constexpr int kProducerWarp = 4;
  static constexpr int kMmaWarp = 5;
  static constexpr int kConvWarp0 = 6;
  static constexpr int kWarps = FP8 ? 10 : 6;
  static constexpr int kThreads = kWarps * 32;
};

MSA_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Upconverts one 128x128 E4M3 tile (TMA SWIZZLE_128B image, 128-byte rows)
// into the two 64-column bf16 halves the MMA reads. 128 threads.
MSA_DEV void convert_tile(const uint8_t* src, uint8_t* dst_half0, int t) {
#pragma unroll 2
  for (int j = 0; j < 8; ++j) {
    const int i = t + j * 128;
    const int r = i >> 3, c = i & 7;
    const uint4 raw = *reinterpret_cast<const uint4*>(src + sw128_offset(r, c));
    const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t outw[8];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
#pragma unroll
      for (int y = 0; y < 2; ++y) {
        const uint16_t pair = (uint16_t)(words[x] >> (16 * y));
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
        const __half2 hh = *reinterpret_cast<const __half2*>(&h2);
        const float2 f = __half22float2(hh);
        outw[x * 2 + y] = pack_bf16x2(f.x, f.y);
      }
    }
    uint8_t* dst = dst_half0 + (c >> 2) * kTile;
    const int c16 = (c & 3) * 2;
    *reinterpret_cast<uint4*>(dst + sw128_offset(r, c16)) =
        make_uint4(outw[0], outw[1], outw[2], outw[3]);
    *reinterpret_cast<uint4*>(dst + sw128_offset(r, c16 + 1)) =
        make_uint4(outw[4], outw[5], outw[6], outw[7]);
  }
}

template <bool FP8>
__global__ void __launch_bounds__(Roles<FP8>::kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillArgs a) {
  using R = Roles<FP8>;
  using Smem = PrefillSmem<FP8>;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  unsigned* fault = a.fault;
  volatile int* abort = &sm.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = a.max_tiles - 1 - (int)blockIdx.x;  // heavier (later) tiles first
  const int h = blockIdx.y;
  const int G = a.num_qo_heads / a.num_kv_heads;
  const int W = a.tile_tokens;

  const int t0 = a.tile_info[2 * tile];
  if (t0 < 0) return;  // past the last tile (uniform over the CTA)
  const int b = a.tile_info[2 * tile + 1];
  const size_t ubase = (size_t)h * a.max_tiles + tile;
  const int n = a.union_len[ubase];
  const int32_t* ulist = a.union_blocks + ubase * a.cap;
  const int seq_q0 = a.cu_q[b];
  const int lq = a.cu_q[b + 1] - seq_q0;
  const int lk = a.paged ? a.seqused_k[b] : a.cu_k[b + 1] - a.cu_k[b];
  const int nw = min(W, seq_q0 + lq - t0);

  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], FP8 ? 4 : 1);
      mbar_init(&sm.v_full[s], FP8 ? 4 : 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int s = 0; s < kF8Stages; ++s) {
      mbar_init(&sm.f8_full[s], 1);
      mbar_init(&sm.f8_empty[s], 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.p_full[s], 4);
      mbar_init(&sm.o_done[s], 1);
    }
    mbar_init(&sm.drain, 1);
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

  if (warp == R::kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&a.tmap_q);
      tma_prefetch_desc(&a.tmap_k);
      tma_prefetch_desc(&a.tmap_v);
      mbar_expect_tx(&sm.q_full, 2u * 128u * (uint32_t)(G * W));
      for (int c = 0; c < 2; ++c) tma_load_3d(sm.q[c], &a.tmap_q, &sm.q_full, c * 64, h * G, t0);
      const int kv0 = a.paged ? 0 : a.cu_k[b];
      int last_issue[kStages > kF8Stages ? kStages : kF8Stages];
      for (int s = 0; s < (kStages > kF8Stages ? kStages : kF8Stages); ++s) last_issue[s] = -1;
      bool ok = true;
      for (int u = 0; u < n; ++u) {
        const int blk = ulist[u];
        int page = 0;
        if (a.paged) {
          page = a.page_table[(size_t)b * a.max_pages + blk];
          // An unmapped page reads as zeros (out-of-range TMA box) and is masked.
          if (page < 0 || page >= a.num_pages) page = a.num_pages;
        }
        if (!FP8) {
          const int st = u % kStages;
          if (u >= kStages &&
              !mbar_wait(&sm.kv_empty[st], ((u / kStages) - 1) & 1, fault, kFaultWaitMma, abort)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&sm.k_full[st], 2 * kTile);
          for (int c = 0; c < 2; ++c) {
            if (a.paged) tma_load_4d(sm.k[st][c], &a.tmap_k, &sm.k_full[st], c * 64, 0, h, page);
            else tma_load_3d(sm.k[st][c], &a.tmap_k, &sm.k_full[st], c * 64, h, kv0 + blk * kBlk);
          }
          mbar_expect_tx(&sm.v_full[st], 2 * kTile);
          for (int c = 0; c < 2; ++c) {
            if (a.paged) tma_load_4d(sm.v[st][c], &a.tmap_v, &sm.v_full[st], c * 64, 0, h, page);
            else tma_load_3d(sm.v[st][c], &a.tmap_v, &sm.v_full[st], c * 64, h, kv0 + blk * kBlk);
          }
          last_issue[st] = u;
        } else {
          const int s8 = u % kF8Stages;
          if (u >= kF8Stages &&
              !mbar_wait(&sm.f8_empty[s8], ((u / kF8Stages) - 1) & 1, fault, kFaultWaitOther,
                         abort)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&sm.f8_full[s8], 2 * kTile);
          if (a.paged) {
            tma_load_4d(sm.k8[s8], &a.tmap_k, &sm.f8_full[s8], 0, 0, h, page);
            tma_load_4d(sm.v8[s8], &a.tmap_v, &sm.f8_full[s8], 0, 0, h, page);
          } else {
            tma_load_3d(sm.k8[s8], &a.tmap_k, &sm.f8_full[s8], 0, h, kv0 + blk * kBlk);
            tma_load_3d(sm.v8[s8], &a.tmap_v, &sm.f8_full[s8], 0, h, kv0 + blk * kBlk);
          }
          last_issue[s8] = u;
        }
      }
      if (!ok) {
        // Let copies already in flight land before the CTA's shared memory is released.
        for (int s = 0; s < (FP8 ? kF8Stages : kStages); ++s) {
          const int u = last_issue[s];
          if (u < 0) continue;
          if (FP8) {
            mbar_wait(&sm.f8_full[s], (u / kF8Stages) & 1, fault, kFaultWaitTma);
          } else {
            mbar_wait(&sm.k_full[s], (u / kStages) & 1, fault, kFaultWaitTma);
            mbar_wait(&sm.v_full[s], (u / kStages) & 1, fault, kFaultWaitTma);
          }
        }
      }
    }
  } else if (warp == R::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      const uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      const uint32_t idO = idesc_bf16_f32(128, 128, false, true);
      bool ok = mbar_wait(&sm.q_full, 0, fault, kFaultWaitTma, abort);
      auto pv = [&](int u) -> bool {
        const int bb = u & 1, st = u % kStages;
        if (!mbar_wait(&sm.p_full[bb], (u >> 1) & 1, fault, kFaultWaitSoftmax, abort)) return false;
        if (!mbar_wait(&sm.v_full[st], (u / kStages) & 1, fault, kFaultWaitTma, abort)) return false;
        tc_fence_after();
        const uint32_t pcol = bb ? kColP1 : kColP0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t bd = sdesc_sw128(smem_u32(sm.v[st][0]) + k * 2048, kTile, 1024);
          mma_ts(tbase + kColO, tbase + pcol + k * 8, bd, idO, (u > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&sm.o_done[bb]);
        mma_commit(&sm.kv_empty[st]);
        return true;
      };
      for (int u = 0; ok && u < n; ++u) {
        const int bb = u & 1, st = u % kStages;
        ok = mbar_wait(&sm.k_full[st], (u / kStages) & 1, fault, kFaultWaitTma, abort);
        if (!ok) break;
        tc_fence_after();
        const uint32_t scol = bb ? kColS1 : kColS0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t ad = sdesc_sw128(smem_u32(sm.q[k >> 2]) + (k & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(smem_u32(sm.k[st][k >> 2]) + (k & 3) * 32, 16, 1024);
          mma_ss(tbase + scol, ad, bd, idS, k > 0 ? 1u : 0u);
        }
        mma_commit(&sm.s_full[bb]);
        if (u >= 1) ok = pv(u - 1);
      }
      if (ok) ok = pv(n - 1);
      // Nothing may be in flight when TMEM is released.
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, fault, kFaultWaitMma);
    }
  } else if (FP8 && warp >= R::kConvWarp0) {
    // ------------------------------------------------------------ E4M3 -> bf16
    const int ct = tid - R::kConvWarp0 * 32;
    for (int u = 0; u < n; ++u) {
      const int s8 = u % kF8Stages, st = u % kStages;
      if (!mbar_wait(&sm.f8_full[s8], (u / kF8Stages) & 1, fault, kFaultWaitTma, abort)) break;
      if (u >= kStages &&
          !mbar_wait(&sm.kv_empty[st], ((u / kStages) - 1) & 1, fault, kFaultWaitMma, abort))
        break;
      convert_tile(sm.k8[s8], sm.k[st][0], ct);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.k_full[st]);
      convert_tile(sm.v8[s8], sm.v[st][0], ct);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.v_full[st]);
        mbar_arrive(&sm.f8_empty[s8]);
      }
    }
  } else if (warp < R::kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax
    const int row = tid;  // TMEM lane
    const int w = row / G, g = row - w * G;
    const bool active = row < W * G && w < nw;
    const long long pos = (long long)lk - lq + (t0 + w - seq_q0);
    const uint32_t* mrow = a.member + (ubase * W + (active ? w : 0)) * a.words;
    const uint32_t lane_base = tbase + ((uint32_t)(warp * 32) << 16);
    float m_ref = -INFINITY, l = 0.f;
    uint32_t mword = 0;
    bool pzero[2] = {false, false};
    bool ok = true;
    for (int u = 0; u < n; ++u) {
      const int bb = u & 1;
      if ((u & 31) == 0 && active) mword = __ldg(mrow + (u >> 5));
      bool mem = active && ((mword >> (u & 31)) & 1u);
      int lim = 127;
      if (mem) {
        const int blk = __ldg(ulist + u);
        if (a.paged) {
          const int page = __ldg(a.page_table + (size_t)b * a.max_pages + blk);
          if (page < 0 || page >= a.num_pages) mem = false;
        }
        long long last = (long long)lk - 1;
        if (a.causal && pos < last) last = pos;
        last -= (long long)blk * kBlk;
        if (last < 0) mem = false;
        else if (last < 127) lim = (int)last;
      }
      ok = mbar_wait(&sm.s_full[bb], (u >> 1) & 1, fault, kFaultWaitMma, abort);
      if (__any_sync(0xffffffffu, !ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool warp_mem = __any_sync(0xffffffffu, mem);
      const uint32_t scol = lane_base + (bb ? kColS1 : kColS0);
      const uint32_t pcol = lane_base + (bb ? kColP1 : kColP0);
      float alpha = 1.f;
      bool rescale = false;
      if (warp_mem) {
        // Pass 1: masked row max over the two 64-column halves of S.
        float mx = -INFINITY;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float s[64];
          tmem_ld64(scol + half * 64, s);
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (lim >= 127 || half * 64 + c <= lim) mx = fmaxf(mx, s[c]);
        }
        if (mem) {
          const float mrow_max = mx * a.scale_log2;
          if (m_ref == -INFINITY || mrow_max > m_ref + kRescaleLog2) {
            if (m_ref != -INFINITY) {
              alpha = ex2(m_ref - mrow_max);
              rescale = true;
              l *= alpha;
            }
            m_ref = mrow_max;
          }
        }
        // Pass 2: P = 2^(s*scale*log2e - m) as bf16 pairs (0 for masked keys
        // and for rows whose token did not select this block). QK(u) having
        // completed implies PV(u-2) completed, so P buffer bb is free.
        const float neg_m = mem ? -m_ref : 0.f;
        float sum = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float s[64];
          tmem_ld64(scol + half * 64, s);
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const int key = half * 64 + c;
            float p0 = ex2(fmaf(s[c], a.scale_log2, neg_m));
            float p1 = ex2(fmaf(s[c + 1], a.scale_log2, neg_m));
            if (!mem || (lim < 127 && key > lim)) p0 = 0.f;
            if (!mem || (lim < 127 && key + 1 > lim)) p1 = 0.f;
            sum += p0 + p1;
            pk[c >> 1] = pack_bf16x2(p0, p1);
          }
          tmem_st32(pcol + half * 32, pk);
        }
        if (mem) l += sum;
        pzero[bb] = false;
      } else if (!pzero[bb]) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = 0u;
        tmem_st32(pcol, pk);
        tmem_st32(pcol + 32, pk);
        pzero[bb] = true;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O must hold every PV up to u-1 before it is rescaled.
        ok = mbar_wait(&sm.o_done[(u - 1) & 1], ((u - 1) >> 1) & 1, fault, kFaultWaitMma, abort);
        if (__any_sync(0xffffffffu, !ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float o[64];
          tmem_ld64(lane_base + kColO + half * 64, o);
          uint32_t ow[64];
#pragma unroll
          for (int c = 0; c < 64; ++c) ow[c] = __float_as_uint(o[c] * alpha);
          tmem_st64(lane_base + kColO + half * 64, ow);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[bb]);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n > 0) {
      ok = mbar_wait(&sm.o_done[(n - 1) & 1], ((n - 1) >> 1) & 1, fault, kFaultWaitMma, abort);
      ok = !__any_sync(0xffffffffu, !ok);
    }
    const bool has = ok && n > 0 && l > 0.f;
    const size_t orow = (size_t)(t0 + w) * a.num_qo_heads + (size_t)h * G + g;
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + orow * 128);
    const float inv = has ? 1.f / l : 0.f;
    if (ok && n > 0) tc_fence_after();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float o[64];
      if (ok && n > 0) tmem_ld64(lane_base + kColO + half * 64, o);
      if (active && ok) {
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          uint4 v4 = make_uint4(0u, 0u, 0u, 0u);
          if (has)
            v4 = make_uint4(pack_bf16x2(o[c] * inv, o[c + 1] * inv),
                            pack_bf16x2(o[c + 2] * inv, o[c + 3] * inv),
                            pack_bf16x2(o[c + 4] * inv, o[c + 5] * inv),
                            pack_bf16x2(o[c + 6] * inv, o[c + 7] * inv));
          dst[(half * 64 + c) >> 3] = v4;
        }
      }
    }
    if (active && ok && a.lse != nullptr)
      a.lse[orow] = has ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <bool FP8>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(PrefillSmem<FP8>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<FP8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_tiles, a.num_kv_heads);
  prefill_kernel<FP8><<<grid, Roles<FP8>::kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  return a.kv_fp8 ? launch_t<true>(a, s) : launch_t<false>(a, s);
}

}  // namespace msa
