// Paged split-KV decode for short query runs (seqlen_q <= 4 per request).
//
// Follows "flashinfer.msa_ops.msa_sparse_attention" (paged K/V with
// page_table + seqused_k; q2k_indices) and "prepare_msa_nvfp4_sparse_decode"
// (request b owns query rows [b*s_q, (b+1)*s_q); token i sits at key position
// seqused_k[b] - s_q + i; at most 16 query heads per KV head; split-KV
// partials merged, completion counters reset after every merge).
//
// Work unit: (request b, KV head h). Its rows are the request's s_q tokens x
// G query heads (<= 64). The unit's pages are the union of its tokens'
// selected, visible blocks; each CTA of the unit takes `pages_per_split`
// consecutive union entries, streams each page's K and V (32 KiB each) into
// shared memory by TMA (two-stage ring), and runs the online softmax with
// warp-level bf16 MMAs. Each CTA writes an fp32 partial (O, m, l); the last
// CTA of the unit to finish (atomic ticket, no waiting) merges the partials
// and writes out/lse. The kernel is bound by HBM: every selected page of
// every (request, KV head) is read exactly once.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace msa {
namespace {

constexpr int kDecThreads = 128;
constexpr int kDecStages = 2;
constexpr int kMaxUnion = 256;      // s_q (<= 4) * topk (<= 64)
constexpr int kHalf = 128 * 128;    // bytes of one 64-column half of a 128-row bf16 tile

struct __align__(1024) DecodeSmem {
  uint8_t kv[kDecStages][4][kHalf];   // [stage][K half0, K half1, V half0, V half1]
  uint8_t q[2][64 * 128];             // Q halves, up to 64 rows
  uint64_t full[kDecStages];
  uint64_t qbar;
  int ulist[kMaxUnion];
  uint32_t tokmask[4][kMaxUnion / 32];  // union membership per token
  int sort_keys[kMaxUnion];
  int scan[kDecThreads + 2];
  int page_of_stage[kDecStages];
  int ulen;
  int last;
  float comb_m[4][16];
  float comb_l[4][16];
};

MSA_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
MSA_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
MSA_DEV void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Address of the 16-byte chunk holding column `col` (multiple of 8) of `row`
// in a 128-column bf16 tile stored as two 128B-swizzled 64-column halves.
MSA_DEV uint32_t tile_addr(uint32_t base, uint32_t half_bytes, int row, int col) {
  return base + (uint32_t)(col >> 6) * half_bytes + sw128_offset(row, (col & 63) >> 3);
}

// RG: 16-row groups (1, 2 or 4); KG = 4 / RG warps split the 128 keys of a page.
template <int RG>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int KG = 4 / RG;
  constexpr int KEYS = 128 / KG;  // keys per warp per page
  constexpr int NT = KEYS / 8;    // 8-key MMA tiles per warp
  constexpr int ROWS = RG * 16;
  extern __shared__ uint8_t smem_raw[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned* fault = a.fault;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, unit = blockIdx.y;
  const int b = unit / a.num_kv_heads, h = unit % a.num_kv_heads;
  const int G = a.num_qo_heads / a.num_kv_heads;
  const int row0 = a.cu_q[b];
  int sq = a.cu_q[b + 1] - row0;
  if (sq > a.sq_max) {
    if (tid == 0) atomicOr(fault, kFaultCapacity);
    sq = a.sq_max;
  }
  const int rows = sq * G;
  const int lk = a.seqused_k[b];
  int nblk = (lk + kBlk - 1) / kBlk;
  if (nblk > a.max_pages) nblk = a.max_pages;

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) mbar_init(&sm.full[s], 1);
    mbar_init(&sm.qbar, 1);
    fence_mbar_init();
  }
  // ---- union of the request's selections (sorted, unique) ----
  const int n = sq * a.topk;
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = tid; i < P; i += kDecThreads) {
    int key = 0x7fffffff;
    if (i < n) {
      const int tok = i / a.topk;
      const int id = a.q2k[((size_t)h * a.total_q + row0 + tok) * a.topk + (i % a.topk)];
      const long long pos = (long long)lk - sq + tok;
      if (id >= 0 && id < nblk && (!a.causal || (long long)id * kBlk <= pos)) key = id;
    }
    sm.sort_keys[i] = key;
  }
  for (int i = tid; i < 4 * (kMaxUnion / 32); i += kDecThreads) (&sm.tokmask[0][0])[i] = 0u;
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P; i += kDecThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const int x = sm.sort_keys[i], y = sm.sort_keys[ixj];
          if ((x > y) == ((i & k) == 0)) {
            sm.sort_keys[i] = y;
            sm.sort_keys[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  {
    int carry = 0;
    for (int c0 = 0; c0 < P; c0 += kDecThreads) {
      const int i = c0 + tid;
      int key = 0x7fffffff, flag = 0;
      if (i < P) {
        key = sm.sort_keys[i];
        flag = key != 0x7fffffff && (i == 0 || sm.sort_keys[i - 1] != key);
      }
      sm.scan[tid] = flag;
      __syncthreads();
      for (int off = 1; off < kDecThreads; off <<= 1) {
        const int add = tid >= off ? sm.scan[tid - off] : 0;
        __syncthreads();
        sm.scan[tid] += add;
        __syncthreads();
      }
      if (flag) sm.ulist[carry + sm.scan[tid] - 1] = key;
      const int tot = sm.scan[kDecThreads - 1];
      __syncthreads();
      carry += tot;
    }
    if (tid == 0) sm.ulen = carry;
    __syncthreads();
  }
  const int ulen = sm.ulen;
  for (int i = tid; i < n; i += kDecThreads) {
    const int tok = i / a.topk;
    const int id = a.q2k[((size_t)h * a.total_q + row0 + tok) * a.topk + (i % a.topk)];
    const long long pos = (long long)lk - sq + tok;
    if (id < 0 || id >= nblk || (a.causal && (long long)id * kBlk > pos)) continue;
    int lo = 0, hi = ulen - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sm.ulist[mid] < id) lo = mid + 1; else hi = mid;
    }
    atomicOr(&sm.tokmask[tok][lo >> 5], 1u << (lo & 31));
  }
  const int p_begin = split * a.pages_per_split;
  const int p_end = min(ulen, p_begin + a.pages_per_split);
  const int npages = max(0, p_end - p_begin);
  __syncthreads();

  // ---- TMA producer (thread 0): Q, then the first stages ----
  auto issue_page = [&](int i) {
    const int st = i % kDecStages;
    const int blk = sm.ulist[p_begin + i];
    int page = a.page_table[(size_t)b * a.max_pages + blk];
    // An unmapped page is fetched as an out-of-range box (zeros) and masked.
    sm.page_of_stage[st] = (page >= 0 && page < a.num_pages) ? page : -1;
    if (page < 0 || page >= a.num_pages) page = a.num_pages;
    mbar_expect_tx(&sm.full[st], 4 * kHalf);
    for (int c = 0; c < 2; ++c) {
      tma_load_4d(sm.kv[st][c], &a.tmap_k, &sm.full[st], c * 64, 0, h, page);
      tma_load_4d(sm.kv[st][2 + c], &a.tmap_v, &sm.full[st], c * 64, 0, h, page);
    }
  };
  if (tid == 0 && npages > 0) {
    tma_prefetch_desc(&a.tmap_k);
    tma_prefetch_desc(&a.tmap_v);
    mbar_expect_tx(&sm.qbar, 2 * 128 * G * a.sq_max);
    for (int c = 0; c < 2; ++c)
      tma_load_3d(sm.q[c], &a.tmap_q, &sm.qbar, c * 64, h * G, row0);
    for (int i = 0; i < kDecStages && i < npages; ++i) issue_page(i);
  }

  const int rg = warp % RG, kg = warp / RG;
  const int gid = lane >> 2, tig = lane & 3;
  const int r_lo = rg * 16 + gid, r_hi = r_lo + 8;
  const int tok_lo = r_lo / G, tok_hi = r_hi / G;
  const bool act_lo = r_lo < rows, act_hi = r_hi < rows;
  const long long pos_lo = (long long)lk - sq + tok_lo, pos_hi = (long long)lk - sq + tok_hi;

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  uint32_t qf[8][4];
  bool ok = true;

  if (npages > 0) {
    ok = mbar_wait(&sm.qbar, 0, fault, kFaultWaitTma);
    if (__syncthreads_or(!ok)) ok = false;
    if (ok) {
      const uint32_t qbase = smem_u32(sm.q[0]);
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        const int row = rg * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int col = kc * 16 + ((lane >> 4) & 1) * 8;
        ldsm_x4(tile_addr(qbase, 64 * 128, row, col), qf[kc][0], qf[kc][1], qf[kc][2], qf[kc][3]);
      }
    }
  }

  for (int i = 0; ok && i < npages; ++i) {
    const int st = i % kDecStages;
    ok = mbar_wait(&sm.full[st], (i / kDecStages) & 1, fault, kFaultWaitTma);
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    const int upos = p_begin + i;
    const int blk = sm.ulist[upos];
    const bool page_ok = sm.page_of_stage[st] >= 0;
    // Last visible key offset inside this block per row, or -1.
    auto limit_of = [&](bool act, int tok, long long pos) -> int {
      if (!act || !page_ok) return -1;
      if (!((sm.tokmask[tok][upos >> 5] >> (upos & 31)) & 1u)) return -1;
      long long lim = (long long)lk - 1;
      if (a.causal && pos < lim) lim = pos;
      lim -= (long long)blk * kBlk;
      return lim < 0 ? -1 : (lim > 127 ? 127 : (int)lim);
    };
    const int lim_lo = limit_of(act_lo, tok_lo, pos_lo);
    const int lim_hi = limit_of(act_hi, tok_hi, pos_hi);
    const bool any = __any_sync(0xffffffffu, (lim_lo >= kg * KEYS) || (lim_hi >= kg * KEYS));
    if (any) {
      const uint32_t kbase = smem_u32(sm.kv[st][0]);
      const uint32_t vbase = smem_u32(sm.kv[st][2]);
      float s[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
          const int key = kg * KEYS + j * 8 + (lane & 7) + ((lane >> 4) & 1) * 8;
          const int col = kc * 16 + ((lane >> 3) & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(tile_addr(kbase, kHalf, key, col), b0, b1, b2, b3);
          mma16816(s[j], qf[kc], b0, b1);
          mma16816(s[j + 1], qf[kc], b2, b3);
        }
      }
      // Mask, scale to log2 units, row max.
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = kg * KEYS + j * 8 + tig * 2 + e;
          s[j][e] = key <= lim_lo ? s[j][e] * a.scale_log2 : -INFINITY;
          s[j][2 + e] = key <= lim_hi ? s[j][2 + e] * a.scale_log2 : -INFINITY;
          mx_lo = fmaxf(mx_lo, s[j][e]);
          mx_hi = fmaxf(mx_hi, s[j][2 + e]);
        }
      }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float use_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
      const float use_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
      const float al_lo = exp2f(m_lo - use_lo), al_hi = exp2f(m_hi - use_hi);
      m_lo = mn_lo;
      m_hi = mn_hi;
      l_lo *= al_lo;
      l_hi *= al_hi;
#pragma unroll
      for (int dt = 0; dt < 16; ++dt) {
        o[dt][0] *= al_lo;
        o[dt][1] *= al_lo;
        o[dt][2] *= al_hi;
        o[dt][3] *= al_hi;
      }
      uint32_t pf[NT / 2][4];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const float p0 = exp2f(s[j][0] - use_lo), p1 = exp2f(s[j][1] - use_lo);
        const float p2 = exp2f(s[j][2] - use_hi), p3 = exp2f(s[j][3] - use_hi);
        l_lo += p0 + p1;
        l_hi += p2 + p3;
        pf[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(p0, p1);
        pf[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(p2, p3);
      }
#pragma unroll
      for (int kc = 0; kc < NT / 2; ++kc) {
        const uint32_t afr[4] = {pf[kc][0], pf[kc][1], pf[kc][2], pf[kc][3]};
#pragma unroll
        for (int dt = 0; dt < 16; dt += 2) {
          const int key = kg * KEYS + kc * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int col = dt * 8 + ((lane >> 4) & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(tile_addr(vbase, kHalf, key, col), b0, b1, b2, b3);
          mma16816(o[dt], afr, b0, b1);
          mma16816(o[dt + 1], afr, b2, b3);
        }
      }
    }
    __syncthreads();  // stage `st` fully consumed
    if (tid == 0 && i + kDecStages < npages) issue_page(i + kDecStages);
  }

  // ---- combine key-group warps through shared memory, write the partial ----
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  __syncthreads();
  float* obuf = reinterpret_cast<float*>(&sm.kv[0][0][0]);  // [warp][16][128]
  {
    float* ow = obuf + warp * 16 * 128;
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      const int c = dt * 8 + tig * 2;
      ow[gid * 128 + c] = o[dt][0];
      ow[gid * 128 + c + 1] = o[dt][1];
      ow[(gid + 8) * 128 + c] = o[dt][2];
      ow[(gid + 8) * 128 + c + 1] = o[dt][3];
    }
    if (tig == 0) {
      sm.comb_m[warp][gid] = m_lo;
      sm.comb_m[warp][gid + 8] = m_hi;
      sm.comb_l[warp][gid] = l_lo;
      sm.comb_l[warp][gid + 8] = l_hi;
    }
  }
  __syncthreads();
  const size_t part = (size_t)unit * a.splits + split;
  for (int idx = tid; idx < ROWS * 128; idx += kDecThreads) {
    const int r = idx >> 7, c = idx & 127;
    if (r >= rows) break;
    const int rgr = r >> 4, rr = r & 15;
    float M = -INFINITY;
#pragma unroll
    for (int g2 = 0; g2 < KG; ++g2) M = fmaxf(M, sm.comb_m[g2 * RG + rgr][rr]);
    float acc = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int g2 = 0; g2 < KG; ++g2) {
        const int w = g2 * RG + rgr;
        const float mw = sm.comb_m[w][rr];
        if (mw == -INFINITY) continue;
        const float f = exp2f(mw - M);
        acc += f * obuf[w * 16 * 128 + rr * 128 + c];
        L += f * sm.comb_l[w][rr];
      }
    }
    a.part_o[(part * ROWS + r) * 128 + c] = acc;
    if (c == 0) {
      a.part_ml[(part * ROWS + r) * 2] = M;
      a.part_ml[(part * ROWS + r) * 2 + 1] = L;
    }
  }

  // ---- last CTA of the unit merges ----
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&a.tickets[unit], 1);
    sm.last = prev == a.splits - 1;
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  const float ln2 = 0.69314718055994531f;
  for (int r = warp; r < rows; r += kDecThreads / 32) {
    float M = -INFINITY;
    for (int s = 0; s < a.splits; ++s)
      M = fmaxf(M, __ldcg(&a.part_ml[(((size_t)unit * a.splits + s) * ROWS + r) * 2]));
    float L = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (M != -INFINITY) {
      for (int s = 0; s < a.splits; ++s) {
        const size_t ps = ((size_t)unit * a.splits + s) * ROWS + r;
        const float ms = __ldcg(&a.part_ml[ps * 2]);
        if (ms == -INFINITY) continue;
        const float f = exp2f(ms - M);
        L += f * __ldcg(&a.part_ml[ps * 2 + 1]);
        const float4 ov = __ldcg(reinterpret_cast<const float4*>(&a.part_o[ps * 128 + lane * 4]));
        acc[0] += f * ov.x;
        acc[1] += f * ov.y;
        acc[2] += f * ov.z;
        acc[3] += f * ov.w;
      }
    }
    const int tok = r / G, g = r % G;
    const size_t orow = (size_t)(row0 + tok) * a.num_qo_heads + (size_t)h * G + g;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + orow * 128 + lane * 4;
    const uint32_t w0 = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    const uint32_t w1 = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(out) = make_uint2(w0, w1);
    if (a.lse != nullptr && lane == 0)
      a.lse[orow] = L > 0.f ? (M + log2f(L)) * ln2 : -INFINITY;
  }
  if (tid == 0) a.tickets[unit] = 0;
}

template <int RG>
cudaError_t launch_rg(const DecodeArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(DecodeSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<RG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.splits, a.batch * a.num_kv_heads);
  decode_kernel<RG><<<grid, kDecThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int decode_pages_per_split(int rows) { return rows <= 16 ? 4 : 8; }

size_t decode_workspace_bytes(int batch, int num_kv_heads, int rows_max, int splits) {
  const int ROWS = rows_max <= 16 ? 16 : (rows_max <= 32 ? 32 : 64);
  const size_t parts = (size_t)batch * num_kv_heads * splits;
  size_t bytes = parts * ROWS * 128 * sizeof(float);
  bytes += parts * ROWS * 2 * sizeof(float);
  bytes += (size_t)batch * num_kv_heads * sizeof(int);
  return bytes;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  const int G = a.num_qo_heads / a.num_kv_heads;
  const int rows = G * a.sq_max;
  if (rows <= 16) return launch_rg<1>(a, s);
  if (rows <= 32) return launch_rg<2>(a, s);
  return launch_rg<4>(a, s);
}

}  // namespace msa
