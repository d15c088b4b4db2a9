// MSA reference oracle: plain, slow, fp64 CPU implementation.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
// this file; only the tests, the smoke check and the CPU-baseline leg of the
// benchmark use it. It shares no code, header or constant with the CUDA path.
//
// Every function follows the plain definition of what the method computes, as
// stated on the FlashInfer documentation pages for MiniMax Sparse Attention:
//   * "flashinfer.msa_ops.msa_sparse_attention" (description and the
//     Parameters list: q, k, v, q2k_indices, cu_seqlens_*, causal,
//     softmax_scale, page_table, seqused_k, return_softmax_lse; Returns);
//   * "flashinfer.msa_ops.msa_proxy_score" (description; Parameters causal,
//     max_k_tiles, reduce_heads; Returns);
//   * "prepare_msa_nvfp4_sparse_decode" (q: GQA head mapping; seqlen_q:
//     right-aligned causal positions; out/lse: natural-log normaliser).
// The union tile of the attention page is a scheduling device; the result it
// must reach is per-query softmax attention over that query's own blocks, and
// that is what is written out here, one query row and one head at a time.
//
// Readings taken where the pages are silent (each is also listed in the
// design notes):
//   R1 block id t of sequence b covers keys [128 t, 128 t + 127] of b
//      (batch-local, "maps batch-local KV block indices to pages");
//   R2 query i of a sequence with Lq queries and Lk keys sits at key position
//      Lk - Lq + i (right-aligned causal); a negative position sees nothing;
//   R3 a row with no visible selected key has out = 0 and lse = -inf;
//   R4 indices are a set: duplicates count once, any negative value is padding;
//   R5 an id >= ceil(Lk/128), >= max_pages, or mapping to a page outside
//      [0, num_pages) contributes no keys;
//   R6 lse is the natural log of the sum of exp(scaled logits);
//   R8 E4M3 is the "fn" variant: bias 7, no infinities, S.1111.111 is NaN;
//   R9 the proxy block max runs over visible keys only, -inf when none;
//   R11 a NaN score is never selected by top-k; ties go to the lower block id;
//   R12 packed NVFP4: element 2i of a row is the low nibble of byte i and
//      element 2i + 1 the high nibble;
//   R13 NVFP4 block scales: one E4M3 scale per 16 consecutive elements of a
//      token's row; K scales linear (token-major); the V scales' "(4, 4)
//      swizzle inside (token, scale index)" read as 4 x 4 tiles of (token,
//      scale index) stored in row-major tile order, each tile scale-index
//      major: (t, s) at byte 4 (d / 16) (t / 4) + 16 (s / 4) + 4 (s % 4) + t % 4
//      of the (page, head)'s scale region (32 (t / 4) + ... for d = 128).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <set>
#include <thread>
#include <utility>
#include <vector>

namespace {

constexpr int kBlock = 128;  // KV block = page = 128 tokens (attention page, k parameter)
constexpr double kNegInf = -std::numeric_limits<double>::infinity();

enum { DT_BF16 = 0, DT_FP16 = 1, DT_E4M3 = 2, DT_F64 = 3 };

// bf16 is the top half of an IEEE binary32.
double bf16_value(uint16_t bits) {
  uint32_t u = uint32_t(bits) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return double(f);
}

// IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits.
double fp16_value(uint16_t h) {
  const int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = std::ldexp(double(m), -24);
  else if (e == 31) v = m ? std::numeric_limits<double>::quiet_NaN()
                          : std::numeric_limits<double>::infinity();
  else v = std::ldexp(double(1024 + m), e - 25);
  return s ? -v : v;
}

// OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
// subnormals at exponent 0, no infinities, S.1111.111 is NaN.
double e4m3_value(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) v = std::numeric_limits<double>::quiet_NaN();
  else if (e == 0) v = std::ldexp(double(m), -9);        // (m/8) * 2^-6
  else v = std::ldexp(double(8 + m), e - 10);            // (1 + m/8) * 2^(e-7)
  return s ? -v : v;
}

// OCP FP4 E2M1, the element format of NVFP4: 1 sign, 2 exponent (bias 1),
// 1 mantissa bit; exponent 0 is subnormal (m / 2); no infinities, no NaN.
double e2m1_value(uint8_t c) {
  const int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  const double v = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

double element(const void* base, int dtype, long long idx) {
  switch (dtype) {
    case DT_BF16: return bf16_value(static_cast<const uint16_t*>(base)[idx]);
    case DT_FP16: return fp16_value(static_cast<const uint16_t*>(base)[idx]);
    case DT_F64: return static_cast<const double*>(base)[idx];
    default: return e4m3_value(static_cast<const uint8_t*>(base)[idx]);
  }
}

// Sequence b owning packed row t: cu[b] <= t < cu[b+1]. Empty sequences are skipped.
int owning_sequence(const int32_t* cu, int batch, long long t) {
  int lo = 0, hi = batch;  // answer in [0, batch)
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (cu[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

// Where the keys live: flat (total_k, Hkv, d) with cu_seqlens_k, or paged
// (num_pages, Hkv, 128, d) with page_table (batch, max_pages) and seqused_k.
struct KeySource {
  const void* k;
  const void* v;
  int dtype;
  const int32_t* cu_k;
  const int32_t* page_table;
  int max_pages;
  int num_pages;
  const int32_t* seqused_k;
  int Hkv;
  int d;

  long long length(int b) const {
    return page_table ? (long long)seqused_k[b] : (long long)cu_k[b + 1] - cu_k[b];
  }
  // Element offset of key j (batch-local) of sequence b, KV head kh; -1 if the
  // block holding it maps to no page (reading R5).
  long long offset(int b, int kh, long long j) const {
    if (page_table) {
      const long long t = j / kBlock;
      if (t >= max_pages) return -1;
      const int p = page_table[(long long)b * max_pages + t];
      if (p < 0 || p >= num_pages) return -1;
      return (((long long)p * Hkv + kh) * kBlock + j % kBlock) * d;
    }
    return ((long long)(cu_k[b] + j) * Hkv + kh) * d;
  }
};

// Query row geometry: sequence, length, right-aligned position (reading R2).
struct RowPos {
  int b;
  long long Lq, Lk, pos;
};

RowPos locate(const int32_t* cu_q, int batch, const KeySource& ks, long long t) {
  RowPos r;
  r.b = owning_sequence(cu_q, batch, t);
  r.Lq = (long long)cu_q[r.b + 1] - cu_q[r.b];
  r.Lk = ks.length(r.b);
  r.pos = r.Lk - r.Lq + (t - cu_q[r.b]);
  return r;
}

template <class F>
void parallel_rows(long long n, int threads, F&& fn) {
  if (threads < 1) threads = 1;
  if (threads > n) threads = int(std::max<long long>(1, n));
  std::vector<std::thread> pool;
  for (int w = 0; w < threads; ++w) {
    pool.emplace_back([&, w]() {
      for (long long r = w; r < n; r += threads) fn(r);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Decode n E4M3 codes to fp64 (reading R8).
void oracle_e4m3_decode(const uint8_t* codes, long long n, double* out) {
  for (long long i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
}

void oracle_bf16_decode(const uint16_t* bits, long long n, double* out) {
  for (long long i = 0; i < n; ++i) out[i] = bf16_value(bits[i]);
}

// Decode n IEEE binary16 bit patterns to fp64 (the fp16 q / K / V of the
// attention page's Parameters).
void oracle_fp16_decode(const uint16_t* bits, long long n, double* out) {
  for (long long i = 0; i < n; ++i) out[i] = fp16_value(bits[i]);
}

// Decode n E2M1 codes (low nibble of each byte) to fp64.
void oracle_e2m1_decode(const uint8_t* codes, long long n, double* out) {
  for (long long i = 0; i < n; ++i) out[i] = e2m1_value(codes[i] & 15);
}

// NVFP4 paged K/V pool to fp64 K and V of shape (num_pages, Hkv, 128, d)
// ("msa_sparse_attention": k, k_scale, v_scale, k_global_scale,
// v_global_scale; "prepare_msa_nvfp4_sparse_decode": k, k_scale, v_scale).
// Page p starts at byte p * page_stride and is planar:
//   [K data (Hkv, 128, d/2) | K scales (Hkv, 128, d/16) | V data | V scales].
// Value of element c of token t, head h: e2m1(nibble) * e4m3(its block
// scale) * global scale (the K global scale folds into the softmax scale and
// the V one into the output: the same product). Readings R12, R13.
void oracle_nvfp4_dequant(const uint8_t* pool, long long page_stride, int num_pages, int Hkv,
                          int d, double k_global, double v_global, double* k_out, double* v_out) {
  const long long data = (long long)Hkv * kBlock * (d / 2);
  const long long scales = (long long)Hkv * kBlock * (d / 16);
  for (int p = 0; p < num_pages; ++p) {
    const uint8_t* page = pool + (long long)p * page_stride;
    for (int side = 0; side < 2; ++side) {
      const uint8_t* dat = page + side * (data + scales);
      const uint8_t* sc = dat + data;
      const double global = side == 0 ? k_global : v_global;
      double* dst = side == 0 ? k_out : v_out;
      for (int h = 0; h < Hkv; ++h)
        for (int t = 0; t < kBlock; ++t)
          for (int c = 0; c < d; ++c) {
            const uint8_t byte = dat[((long long)h * kBlock + t) * (d / 2) + c / 2];
            const uint8_t code = (c % 2 == 0) ? (byte & 15) : (byte >> 4);
            const int s = c / 16;
            long long at;
            if (side == 0) {
              at = ((long long)h * kBlock + t) * (d / 16) + s;
            } else {
              at = (long long)h * kBlock * (d / 16) + 4 * (d / 16) * (t / 4) + 16 * (s / 4) +
                   4 * (s % 4) + t % 4;
            }
            dst[(((long long)p * Hkv + h) * kBlock + t) * d + c] =
                e2m1_value(code) * e4m3_value(sc[at]) * global;
          }
    }
  }
}

// Sparse attention forward, plain definition ("msa_sparse_attention":
// description, q2k_indices, causal, softmax_scale, return_softmax_lse).
//
// For query row t (packed index) and query head h, with KV head
// kh = h / (Hq / Hkv) (GQA, "prepare_msa_nvfp4_sparse_decode", q):
//   S = set of non-negative ids in q2k[kh, t, :]
//   J = { keys j of blocks in S : j < Lk, and j <= pos when causal }
//   s_j = scale * <q, k_j>;  out = sum_j softmax(s)_j v_j;  lse = ln sum_j e^{s_j}
// rows[0:n_rows] lists the packed query rows to evaluate (NULL = all rows,
// n_rows = total_q). out is (n_rows, Hq, d), lse is (n_rows, Hq); both fp64.
int oracle_sparse_attention(const void* q, int q_dtype, const void* k, const void* v, int kv_dtype,
                            const int32_t* q2k, int topk, const int32_t* cu_q, const int32_t* cu_k,
                            const int32_t* page_table, int max_pages, int num_pages,
                            const int32_t* seqused_k, int batch, int total_q, int Hq, int Hkv, int d,
                            int causal, double scale, const int32_t* rows, int n_rows, double* out,
                            double* lse, int threads) {
  if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || topk <= 0 || batch <= 0) return 1;
  const int G = Hq / Hkv;
  KeySource ks{k, v, kv_dtype, cu_k, page_table, max_pages, num_pages, seqused_k, Hkv, d};
  parallel_rows(n_rows, threads, [&](long long r) {
    const long long t = rows ? rows[r] : r;
    const RowPos rp = locate(cu_q, batch, ks, t);
    const long long nblk = (rp.Lk + kBlock - 1) / kBlock;
    std::vector<double> qrow(d), acc(d);
    std::vector<double> logit;
    std::vector<long long> where;
    for (int h = 0; h < Hq; ++h) {
      const int kh = h / G;
      std::set<int> selected;  // reading R4
      for (int c = 0; c < topk; ++c) {
        const int id = q2k[((long long)kh * total_q + t) * topk + c];
        if (id >= 0) selected.insert(id);
      }
      for (int c = 0; c < d; ++c) qrow[c] = element(q, q_dtype, (t * Hq + h) * (long long)d + c);
      logit.clear();
      where.clear();
      for (int id : selected) {
        if (id >= nblk) continue;  // reading R5
        for (long long j = (long long)id * kBlock; j < std::min<long long>((long long)(id + 1) * kBlock, rp.Lk); ++j) {
          if (causal && j > rp.pos) break;
          const long long off = ks.offset(rp.b, kh, j);
          if (off < 0) break;  // the whole block maps to no page
          double dot = 0.0;
          for (int c = 0; c < d; ++c) dot += qrow[c] * element(k, kv_dtype, off + c);
          logit.push_back(scale * dot);
          where.push_back(off);
        }
      }
      double* o = out + (r * Hq + h) * (long long)d;
      if (logit.empty()) {  // reading R3
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        if (lse) lse[r * Hq + h] = kNegInf;
        continue;
      }
      double m = kNegInf;
      for (double s : logit) m = std::max(m, s);
      double l = 0.0;
      std::fill(acc.begin(), acc.end(), 0.0);
      for (size_t n = 0; n < logit.size(); ++n) {
        const double p = std::exp(logit[n] - m);
        l += p;
        for (int c = 0; c < d; ++c) acc[c] += p * element(v, kv_dtype, where[n] + c);
      }
      for (int c = 0; c < d; ++c) o[c] = acc[c] / l;
      if (lse) lse[r * Hq + h] = m + std::log(l);  // reading R6
    }
  });
  return 0;
}

// Proxy score ("msa_proxy_score"): max over the keys of block tt of the
// unscaled, causally masked logit <q_{t,h}, k_{j, h/G}>; -inf when the block
// has no visible key (beyond the sequence, or entirely above the causal limit).
// With reduce_heads, the max is also taken over h.
// out is (Hq or 1, max_k_tiles, n_rows), query fastest.
int oracle_proxy_score(const void* q, int q_dtype, const void* k, int k_dtype, const int32_t* cu_q,
                       const int32_t* cu_k, const int32_t* page_table, int max_pages, int num_pages,
                       const int32_t* seqused_k, int batch, int total_q, int Hq, int Hkv, int d,
                       int max_k_tiles, int causal, int reduce_heads, const int32_t* rows, int n_rows,
                       double* out, int threads) {
  (void)total_q;
  if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || batch <= 0 || max_k_tiles <= 0) return 1;
  const int G = Hq / Hkv;
  KeySource ks{k, nullptr, k_dtype, cu_k, page_table, max_pages, num_pages, seqused_k, Hkv, d};
  const int out_heads = reduce_heads ? 1 : Hq;
  for (long long i = 0; i < (long long)out_heads * max_k_tiles * n_rows; ++i) out[i] = kNegInf;
  parallel_rows(n_rows, threads, [&](long long r) {
    const long long t = rows ? rows[r] : r;
    const RowPos rp = locate(cu_q, batch, ks, t);
    std::vector<double> qrow(d);
    for (int h = 0; h < Hq; ++h) {
      const int kh = h / G;
      for (int c = 0; c < d; ++c) qrow[c] = element(q, q_dtype, (t * Hq + h) * (long long)d + c);
      for (int tt = 0; tt < max_k_tiles; ++tt) {
        double best = kNegInf;
        for (long long j = (long long)tt * kBlock; j < std::min<long long>((long long)(tt + 1) * kBlock, rp.Lk); ++j) {
          if (causal && j > rp.pos) break;
          const long long off = ks.offset(rp.b, kh, j);
          if (off < 0) break;
          double dot = 0.0;
          for (int c = 0; c < d; ++c) dot += qrow[c] * element(k, k_dtype, off + c);
          best = std::max(best, dot);
        }
        double& slot = out[((long long)(reduce_heads ? 0 : h) * max_k_tiles + tt) * n_rows + r];
        slot = std::max(slot, best);
      }
    }
  });
  return 0;
}

// Top-k block selection (the consumer of the proxy score, "msa_topk_select"
// contract as stated on the proxy and decode pages): for each query, the topk
// highest selectable scores of its max_k_tiles columns, ties to the lower
// block id, returned ascending and -1 padded. -inf and NaN are never selected
// (reading R11). scores is (num_score_heads, max_k_tiles, total_q) fp32; with
// one score head the selection is broadcast to all num_kv_heads_out heads,
// otherwise num_score_heads must equal num_kv_heads_out (one per head).
// q2k is (num_kv_heads_out, n_rows, topk).
int oracle_topk_select(const float* scores, int num_score_heads, int max_k_tiles, int total_q, int topk,
                       int num_kv_heads_out, const int32_t* rows, int n_rows, int32_t* q2k) {
  if (num_score_heads != 1 && num_score_heads != num_kv_heads_out) return 1;
  for (int h = 0; h < num_kv_heads_out; ++h) {
    const int sh = num_score_heads == 1 ? 0 : h;
    for (long long r = 0; r < n_rows; ++r) {
      const long long t = rows ? rows[r] : r;
      std::vector<std::pair<double, int>> cand;
      for (int tt = 0; tt < max_k_tiles; ++tt) {
        const double s = scores[((long long)sh * max_k_tiles + tt) * total_q + t];
        if (std::isnan(s) || s == kNegInf) continue;
        cand.emplace_back(s, tt);
      }
      std::sort(cand.begin(), cand.end(), [](const std::pair<double, int>& a, const std::pair<double, int>& b) {
        if (a.first != b.first) return a.first > b.first;
        return a.second < b.second;
      });
      std::vector<int> chosen;
      for (size_t i = 0; i < cand.size() && (int)i < topk; ++i) chosen.push_back(cand[i].second);
      std::sort(chosen.begin(), chosen.end());
      int32_t* dst = q2k + ((long long)h * n_rows + r) * topk;
      for (int c = 0; c < topk; ++c) dst[c] = c < (int)chosen.size() ? chosen[c] : -1;
    }
  }
  return 0;
}

// Union metadata ("msa_sparse_attention" description: query tokens are
// processed in tiles, each over the union of the blocks its tokens selected).
// Tiles are tile_tokens consecutive queries of one sequence, numbered in
// sequence order. For tile tau of KV head h:
//   union_len[h, tau]             number of distinct usable ids in the tile
//   union_blocks[h, tau, 0:cap]   those ids ascending, -1 filled
//   member[h, tau, w, 0:cap/32]   bit j set iff union_blocks[j] is in token w's row
// An id is usable for token w iff 0 <= id < ceil(Lk/128) (and < max_pages when
// paged) and, when causal, the block holds a key <= pos(w). Rows past the
// sequence end are zero. num_tiles must equal the sum of ceil(Lq_b/tile_tokens).
int oracle_build_union(const int32_t* q2k, int topk, const int32_t* cu_q, const int32_t* cu_k,
                       const int32_t* seqused_k, int max_pages, int batch, int total_q, int Hkv,
                       int causal, int tile_tokens, int cap, int num_tiles, int32_t* union_len,
                       int32_t* union_blocks, uint32_t* member) {
  const int words = (cap + 31) / 32;
  const bool paged = seqused_k != nullptr;
  int tau = 0;
  std::vector<std::pair<long long, int>> tiles;  // (first packed row, sequence)
  for (int b = 0; b < batch; ++b) {
    for (long long s = cu_q[b]; s < cu_q[b + 1]; s += tile_tokens) tiles.emplace_back(s, b);
  }
  if ((int)tiles.size() != num_tiles) return 1;
  for (int h = 0; h < Hkv; ++h) {
    for (tau = 0; tau < num_tiles; ++tau) {
      const long long t0 = tiles[tau].first;
      const int b = tiles[tau].second;
      const long long Lq = (long long)cu_q[b + 1] - cu_q[b];
      const long long Lk = paged ? (long long)seqused_k[b] : (long long)cu_k[b + 1] - cu_k[b];
      long long nblk = (Lk + kBlock - 1) / kBlock;
      if (paged) nblk = std::min<long long>(nblk, max_pages);
      std::vector<std::set<int>> rowsets(tile_tokens);
      std::set<int> all;
      for (int w = 0; w < tile_tokens; ++w) {
        const long long t = t0 + w;
        if (t >= cu_q[b + 1]) break;
        const long long pos = Lk - Lq + (t - cu_q[b]);
        for (int c = 0; c < topk; ++c) {
          const int id = q2k[((long long)h * total_q + t) * topk + c];
          if (id < 0 || id >= nblk) continue;
          if (causal && (long long)id * kBlock > pos) continue;
          rowsets[w].insert(id);
          all.insert(id);
        }
      }
      if ((int)all.size() > cap) return 2;
      const long long base = (long long)h * num_tiles + tau;
      union_len[base] = (int32_t)all.size();
      std::vector<int> ulist(all.begin(), all.end());
      for (int j = 0; j < cap; ++j) union_blocks[base * cap + j] = j < (int)ulist.size() ? ulist[j] : -1;
      for (int w = 0; w < tile_tokens; ++w) {
        uint32_t* mw = member + (base * tile_tokens + w) * words;
        for (int x = 0; x < words; ++x) mw[x] = 0u;
        for (int j = 0; j < (int)ulist.size(); ++j) {
          if (rowsets[w].count(ulist[j])) mw[j / 32] |= 1u << (j % 32);
        }
      }
    }
  }
  return 0;
}

}  // extern "C"
