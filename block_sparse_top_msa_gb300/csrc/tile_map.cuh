// Query-tile numbering shared by the kernels that walk query tiles: tiles are
// `W` consecutive queries of one sequence, numbered sequence by sequence.
// A CTA maps its tile number to (sequence, first packed row) with a chunked
// block-wide scan over the per-sequence tile counts, so no host-side or
// precomputed schedule is needed.
#pragma once

#include "common.cuh"

namespace msa {

// All threads of the block must call this. Returns false when `tile` lies past
// the last tile. `scratch` needs blockDim.x + 2 ints of shared memory.
__device__ __forceinline__ bool locate_tile(const int32_t* cu_q, int batch, int W, int tile,
                                            int* scratch, int* seq, int* first_row) {
  const int tid = threadIdx.x, nt = blockDim.x;
  int carry = 0;
  if (tid == 0) scratch[nt] = -1;
  __syncthreads();
  for (int base = 0; base < batch; base += nt) {
    const int b = base + tid;
    int cnt = 0, start = 0;
    if (b < batch) {
      start = cu_q[b];
      const int lq = cu_q[b + 1] - start;
      cnt = lq > 0 ? (lq + W - 1) / W : 0;
    }
    scratch[tid] = cnt;
    __syncthreads();
    // Inclusive Hillis-Steele scan over the chunk.
    for (int off = 1; off < nt; off <<= 1) {
      int add = tid >= off ? scratch[tid - off] : 0;
      __syncthreads();
      scratch[tid] += add;
      __syncthreads();
    }
    const int incl = scratch[tid];
    const int excl = incl - cnt;
    const int total = scratch[nt - 1];
    if (b < batch && cnt > 0 && tile >= carry + excl && tile < carry + incl) {
      scratch[nt] = b;
      scratch[nt + 1] = start + (tile - carry - excl) * W;
    }
    __syncthreads();
    const int found = scratch[nt];
    carry += total;
    __syncthreads();
    if (found >= 0) break;
  }
  const int found = scratch[nt];
  if (found < 0) return false;
  *seq = found;
  *first_row = scratch[nt + 1];
  return true;
}

}  // namespace msa
