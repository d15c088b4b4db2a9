// MSA stage 1, the dense proxy pass ("flashinfer.msa_ops.msa_proxy_score":
// max_score[h, t, q] is the max over the 128 keys of KV block t of the
// unscaled, causally masked q.k logits; blocks beyond the sequence or wholly
// above the causal limit give -inf; reduce_heads takes the max over query
// heads as well).
//
// One CTA per (query tile of 2 * Wm tokens, slice of its block columns),
// Wm = 128 / G: two tcgen05 M=128 tiles of (token, head-in-group) rows (the
// second skipped when the tile has at most Wm tokens). A block column's max
// needs no other slice, so decode-sized problems (few tokens, long contexts)
// spread each tile's columns over many CTAs. K is flat or paged (one page
// per block; an unmapped page gives -inf). Loop order: KV group g outer, KV
// block t inner. For each (g, t) the producer warp TMA-loads K of block t
// (128 x 128 bf16) into a two-stage ring; the MMA warp computes both tiles'
// S = Q_g K_t^T into TMEM (double-buffered, 4 x 128 columns); eight epilogue
// warps (two per TMEM lane quadrant, one per M tile) take each row's masked
// max over the 128 keys and then the max over the G heads of the token
// (warp shuffles). With reduce_heads the running max over groups lives in
// shared memory per (block, token) and is written once, coalesced, per block
// column; the per-head buffer of the reference design is never materialised.
// q and K are bf16 or fp16 (the MMA takes q's type); E4M3 K ("fn") is loaded
// by TMA into a two-stage staging ring and upconverted exactly to q's type in
// the MMA's swizzled layout by the eight epilogue warps, which convert block
// t + 1 before taking the maxima of block t.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tile_map.cuh"
#include "tmem_wide.cuh"

namespace msa {
namespace {

constexpr int kPxStages = 2;
constexpr int kPxTile = 16384;
constexpr int kPxEpiWarps = 8;
constexpr int kPxProducerWarp = 8;
constexpr int kPxMmaWarp = 9;
constexpr int kPxThreads = 10 * 32;

// F8K: an E4M3 staging ring, paid for with a smaller running-max buffer.
template <bool F8K>
struct __align__(1024) ProxySmem {
  static constexpr int kRed = F8K ? 14336 : 16384;  // floats of running max (block column x token)
  uint8_t q[2][2][kPxTile];            // [M tile][d half]
  uint8_t k[kPxStages][2][kPxTile];
  uint8_t k8[F8K ? kPxStages : 1][F8K ? kPxTile : 16];  // E4M3 K as loaded (F8K)
  float red[kRed];                     // running max per (block column, token)
  uint64_t q_full, q_empty;
  uint64_t k_full[kPxStages], k_empty[kPxStages];
  uint64_t f8_full[kPxStages], f8_empty[kPxStages];
  uint64_t s_full[2], s_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int scan[kPxThreads + 2];
  int abort;
};

// One 128 x 128 E4M3 K tile (TMA SWIZZLE_128B image, 128-byte rows) to the
// two 64-column 16-bit halves the MMA reads, by the 256 epilogue threads.
template <bool F16>
MSA_DEV void px_convert_tile(const uint8_t* src, uint8_t* dst_half0, int t) {
#pragma unroll 2
  for (int i = t; i < 1024; i += kPxEpiWarps * 32) {
    const int r = i >> 3, c = i & 7;
    const uint4 raw = *reinterpret_cast<const uint4*>(src + sw128_offset(r, c));
    uint32_t w[8];
    if (F16) {
      e4m3x4_to_f16(raw.x, w[0], w[1]);
      e4m3x4_to_f16(raw.y, w[2], w[3]);
      e4m3x4_to_f16(raw.z, w[4], w[5]);
      e4m3x4_to_f16(raw.w, w[6], w[7]);
    } else {
      e4m3x4_to_bf16(raw.x, w[0], w[1]);
      e4m3x4_to_bf16(raw.y, w[2], w[3]);
      e4m3x4_to_bf16(raw.z, w[4], w[5]);
      e4m3x4_to_bf16(raw.w, w[6], w[7]);
    }
    uint8_t* dst = dst_half0 + (c >> 2) * kPxTile;
    const int c16 = (c & 3) * 2;
    *reinterpret_cast<uint4*>(dst + sw128_offset(r, c16)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(dst + sw128_offset(r, c16 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// PAGED: K from a page pool. ONE_M: query tiles of Wm tokens, one M tile
// (decode-sized calls, where no sequence has more than Wm query tokens).
// F8K: E4M3 K, upconverted by the epilogue warps.
template <bool PAGED, bool ONE_M, bool F8K>
__global__ void __launch_bounds__(kPxThreads, 1) proxy_kernel(const __grid_constant__ ProxyArgs a) {
  constexpr int MT = ONE_M ? 1 : 2;  // M tiles computed
  using Smem = ProxySmem<F8K>;
  constexpr int kPxRed = Smem::kRed;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned* fault = a.fault;
  volatile int* abort = &sm.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.num_qo_heads / a.num_kv_heads;
  const int Wm = a.tile_tokens;  // tokens per M tile
  const int TQ = MT * Wm;        // tokens per query tile
  const int tile = a.max_tiles - 1 - (int)(blockIdx.x / a.slices);
  const int slice = (int)(blockIdx.x % a.slices);

  int b = 0, t0 = 0;
  if (!locate_tile(a.cu_q, a.batch, TQ, tile, sm.scan, &b, &t0)) return;
  const int seq_q0 = a.cu_q[b];
  const int lq = a.cu_q[b + 1] - seq_q0;
  const int lk = PAGED ? a.seqused_k[b] : a.cu_k[b + 1] - a.cu_k[b];
  const int kv0 = PAGED ? 0 : a.cu_k[b];
  const int ntok = min(TQ, seq_q0 + lq - t0);
  int nblk = (lk + kBlk - 1) / kBlk;
  if (nblk > a.max_k_tiles) nblk = a.max_k_tiles;
  if (PAGED && nblk > a.max_pages) nblk = a.max_pages;
  // Last block any token of the tile can see.
  int t_hi = nblk - 1;
  if (a.causal) {
    const long long pmax = (long long)lk - lq + (t0 + ntok - 1 - seq_q0);
    const long long lim = pmax < 0 ? -1 : pmax / kBlk;
    if (lim < t_hi) t_hi = (int)lim;
  }
  const int ncols = t_hi + 1;  // block columns with visible keys; the rest are -inf
  // This CTA's columns [c_lo, c_lo + ncs); slice 0 also writes the -inf rest.
  const int c_lo = min(ncols, slice * a.slice_cols);
  const int ncs = min(ncols, c_lo + a.slice_cols) - c_lo;
  if (ncs == 0 && slice > 0) return;
  const int CH = kPxRed / TQ;  // block columns per pass over the groups
  const int nchunks = (ncs + CH - 1) / CH;
  const int nsteps = nchunks * a.num_kv_heads;  // (chunk, group) passes

  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int s = 0; s < kPxStages; ++s) {
      mbar_init(&sm.k_full[s], F8K ? kPxEpiWarps : 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.f8_full[s], 1);
      mbar_init(&sm.f8_empty[s], kPxEpiWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.s_free[s], kPxEpiWarps);
    }
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == kPxMmaWarp) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  // Columns in chunk c: c_lo + [c * CH, min(ncs, (c + 1) * CH)).
  auto chunk_cols = [&](int c) { return min(CH, ncs - c * CH); };

  if (warp == kPxProducerWarp) {
    if (lane == 0 && ncs > 0) {
      tma_prefetch_desc(&a.tmap_q);
      tma_prefetch_desc(&a.tmap_k);
      int it = 0;  // global K-tile counter
      bool ok = true;
      int last_k[kPxStages] = {-1, -1};
      for (int p = 0; ok && p < nsteps; ++p) {
        const int c = p / a.num_kv_heads, g = p % a.num_kv_heads;
        if (p > 0 && !mbar_wait(&sm.q_empty, (p - 1) & 1, fault, kFaultWaitMma, abort)) {
          ok = false;
          break;
        }
        mbar_expect_tx(&sm.q_full, (uint32_t)MT * 2u * 128u * (uint32_t)(G * Wm));
        for (int m = 0; m < MT; ++m)
          for (int hh = 0; hh < 2; ++hh)
            tma_load_3d(sm.q[m][hh], &a.tmap_q, &sm.q_full, hh * 64, g * G, t0 + m * Wm);
        const int nc = chunk_cols(c);
        for (int j = 0; j < nc; ++j, ++it) {
          const int st = it % kPxStages;
          // E4M3: the staging slot is free once its tile is converted; the
          // converters themselves wait for the 16-bit slot.
          uint64_t* free_bar = F8K ? &sm.f8_empty[st] : &sm.k_empty[st];
          if (it >= kPxStages &&
              !mbar_wait(free_bar, ((it / kPxStages) - 1) & 1, fault,
                         F8K ? kFaultWaitSoftmax : kFaultWaitMma, abort)) {
            ok = false;
            break;
          }
          const int t = c_lo + c * CH + j;
          if (F8K) {
            mbar_expect_tx(&sm.f8_full[st], kPxTile);
            if (PAGED) {
              int page = a.page_table[(size_t)b * a.max_pages + t];
              if (page < 0 || page >= a.num_pages) page = a.num_pages;
              tma_load_4d(sm.k8[st], &a.tmap_k, &sm.f8_full[st], 0, 0, g, page);
            } else {
              tma_load_3d(sm.k8[st], &a.tmap_k, &sm.f8_full[st], 0, g, kv0 + t * kBlk);
            }
            last_k[st] = it;
            continue;
          }
          mbar_expect_tx(&sm.k_full[st], 2 * kPxTile);
          if (PAGED) {
            int page = a.page_table[(size_t)b * a.max_pages + t];
            // An unmapped page reads as zeros (out-of-range box); the epilogue gives it -inf.
            if (page < 0 || page >= a.num_pages) page = a.num_pages;
            for (int hh = 0; hh < 2; ++hh)
              tma_load_4d(sm.k[st][hh], &a.tmap_k, &sm.k_full[st], hh * 64, 0, g, page);
          } else {
            for (int hh = 0; hh < 2; ++hh)
              tma_load_3d(sm.k[st][hh], &a.tmap_k, &sm.k_full[st], hh * 64, g, kv0 + t * kBlk);
          }
          last_k[st] = it;
        }
      }
      if (!ok) {
        for (int s = 0; s < kPxStages; ++s)
          if (last_k[s] >= 0)
            mbar_wait(F8K ? &sm.f8_full[s] : &sm.k_full[s], (last_k[s] / kPxStages) & 1, fault,
                      kFaultWaitTma);
      }
    }
  } else if (warp == kPxMmaWarp) {
    if (lane == 0 && ncs > 0) {
      const uint32_t idS = idesc_16bit_f32(128, 128, false, false, a.f16 != 0);
      int it = 0;
      bool ok = true;
      for (int p = 0; ok && p < nsteps; ++p) {
        const int c = p / a.num_kv_heads;
        if (!mbar_wait(&sm.q_full, p & 1, fault, kFaultWaitTma, abort)) {
          ok = false;
          break;
        }
        const int nc = chunk_cols(c);
        for (int j = 0; j < nc; ++j, ++it) {
          const int st = it % kPxStages, bb = it & 1;
          if (!mbar_wait(&sm.k_full[st], (it / kPxStages) & 1, fault, kFaultWaitTma, abort) ||
              (it >= 2 && !mbar_wait(&sm.s_free[bb], ((it >> 1) - 1) & 1, fault,
                                     kFaultWaitSoftmax, abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint32_t dcol = (uint32_t)(bb * 256 + m * 128);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t ad = sdesc_sw128(smem_u32(sm.q[m][k >> 2]) + (k & 3) * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(smem_u32(sm.k[st][k >> 2]) + (k & 3) * 32, 16, 1024);
              mma_ss(tbase + dcol, ad, bd, idS, k > 0 ? 1u : 0u);
            }
          }
          mma_commit(&sm.s_full[bb]);
          mma_commit(&sm.k_empty[st]);
        }
        mma_commit(&sm.q_empty);
      }
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, fault, kFaultWaitMma);
    }
  } else {
    // ------------------------------------------------------------ epilogue (8 warps)
    // Thread (M tile m, lane quadrant, lane) owns row r of tile m. With
    // reduce_heads the head-0 thread of each token keeps the token's running
    // max over groups in sm.red and writes it during the last group's pass.
    const int m = warp >> 2, quad = warp & 3;
    const int r = quad * 32 + lane;                 // row inside M tile m
    const int w = r / G, gg = r - w * G;
    const int tw = m * Wm + w;                      // token inside the tile
    const bool active = r < Wm * G && tw < ntok;
    const long long pos = (long long)lk - lq + (t0 + tw - seq_q0);
    const uint32_t taddr_lane = tbase + ((uint32_t)(quad * 32) << 16);
    int it = 0;
    bool ok = true;
    // E4M3: tile x (in the order the producer loads them) from staging slot
    // x % 2 into 16-bit slot x % 2, once QK(x - 2) has released that slot.
    const int ntiles = ncs * a.num_kv_heads;
    auto convert = [&](int x) -> bool {
      const int st = x % kPxStages;
      bool okc = mbar_wait(&sm.f8_full[st], (x / kPxStages) & 1, fault, kFaultWaitTma, abort) &&
                 (x < kPxStages ||
                  mbar_wait(&sm.k_empty[st], ((x / kPxStages) - 1) & 1, fault, kFaultWaitMma, abort));
      if (__any_sync(0xffffffffu, !okc)) return false;
      if (a.f16) px_convert_tile<true>(sm.k8[st], sm.k[st][0], tid);
      else px_convert_tile<false>(sm.k8[st], sm.k[st][0], tid);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.f8_empty[st]);
        mbar_arrive(&sm.k_full[st]);
      }
      return true;
    };
    if (F8K && ntiles > 0) ok = convert(0);
    for (int p = 0; ok && p < nsteps; ++p) {
      const int c = p / a.num_kv_heads, g = p % a.num_kv_heads;
      const int nc = chunk_cols(c);
      for (int j = 0; j < nc; ++j, ++it) {
        const int bb = it & 1;
        const int t = c_lo + c * CH + j;
        if (F8K && it + 1 < ntiles && !convert(it + 1)) {
          ok = false;
          break;
        }
        ok = mbar_wait(&sm.s_full[bb], (it >> 1) & 1, fault, kFaultWaitMma, abort);
        if (__any_sync(0xffffffffu, !ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // (With ONE_M, tile 1's columns are read unwritten and ignored: none
        // of its rows is active.)
        float s[128];
        tmem_ld128(taddr_lane + (uint32_t)(bb * 256 + m * 128), s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.s_free[bb]);
        float mx = -INFINITY;
        bool page_ok = true;
        if (PAGED) {
          const int pg = __ldg(a.page_table + (size_t)b * a.max_pages + t);
          page_ok = pg >= 0 && pg < a.num_pages;
        }
        if (active && page_ok) {
          long long last = (long long)lk - 1;
          if (a.causal && pos < last) last = pos;
          last -= (long long)t * kBlk;
          if (last >= 127) {
#pragma unroll
            for (int i = 0; i < 128; ++i) mx = fmaxf(mx, s[i]);
          } else if (last >= 0) {
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (i <= last) mx = fmaxf(mx, s[i]);
          }
        }
        if (a.reduce_heads) {
          // Rows of one token are G consecutive lanes (G a power of two <= 32).
          for (int off = 1; off < G; off <<= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          if (active && gg == 0) {
            float& slot = sm.red[j * TQ + tw];
            const float v = g == 0 ? mx : fmaxf(slot, mx);
            if (g == a.num_kv_heads - 1) a.out[(size_t)t * a.total_q + t0 + tw] = v;
            else slot = v;
          }
        } else if (active) {
          const int hq = g * G + gg;
          a.out[((size_t)hq * a.max_k_tiles + t) * a.total_q + t0 + tw] = mx;
        }
      }
    }
    // Columns no token of the tile can see (written by the tile's slice 0).
    const int heads_out = a.reduce_heads ? 1 : a.num_qo_heads;
    const int rest = slice == 0 ? a.max_k_tiles - ncols : 0;
    for (long long i = tid; i < (long long)heads_out * rest * ntok; i += kPxEpiWarps * 32) {
      const int tt = (int)(i % ntok);
      const long long q2 = i / ntok;
      const int t = ncols + (int)(q2 % rest);
      const int hq = (int)(q2 / rest);
      a.out[((size_t)hq * a.max_k_tiles + t) * a.total_q + t0 + tt] = -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kPxMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <bool F8K>
cudaError_t launch_proxy_t(const ProxyArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(ProxySmem<F8K>) + 1024;
  cudaError_t e = cudaSuccess;
  for (auto k : {proxy_kernel<false, false, F8K>, proxy_kernel<false, true, F8K>,
                 proxy_kernel<true, false, F8K>, proxy_kernel<true, true, F8K>})
    if (e == cudaSuccess) e = set_smem_limit((const void*)k, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((long long)a.max_tiles * a.slices));
  if (a.paged) {
    if (a.one_m) proxy_kernel<true, true, F8K><<<grid, kPxThreads, smem, s>>>(a);
    else proxy_kernel<true, false, F8K><<<grid, kPxThreads, smem, s>>>(a);
  } else {
    if (a.one_m) proxy_kernel<false, true, F8K><<<grid, kPxThreads, smem, s>>>(a);
    else proxy_kernel<false, false, F8K><<<grid, kPxThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_proxy(const ProxyArgs& a, cudaStream_t s) {
  return a.k_fp8 ? launch_proxy_t<true>(a, s) : launch_proxy_t<false>(a, s);
}

}  // namespace msa
