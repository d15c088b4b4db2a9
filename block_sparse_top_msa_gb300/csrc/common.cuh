// Device helpers shared by the MSA kernels: mbarriers with bounded waits, TMA
// tensor loads, tcgen05 (TMEM allocation, MMA, loads/stores) and descriptor
// encoders for sm_103a. Every wait is bounded by wall-clock time; on expiry a
// bit is set in the library's fault word and the caller unwinds.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MSA_DEV __device__ __forceinline__

namespace msa {

constexpr int kBlk = 128;   // KV block / page size in tokens
constexpr int kHeadDim = 128;

// Fault bits reported through msa_read_device_fault.
enum FaultBits : unsigned {
  kFaultWaitTma = 1u << 0,
  kFaultWaitMma = 1u << 1,
  kFaultWaitSoftmax = 1u << 2,
  kFaultCapacity = 1u << 3,
  kFaultWaitOther = 1u << 4,
};

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait

MSA_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MSA_DEV unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
MSA_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
MSA_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

MSA_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
MSA_DEV void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
MSA_DEV bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed. Gives up after
// kWaitLimitNs (or as soon as *abort is set by another warp of the CTA),
// recording `code` in the fault word; returns false in that case.
MSA_DEV bool mbar_wait_for(uint64_t* bar, uint32_t parity, unsigned* fault, unsigned code,
                           unsigned long long limit_ns, volatile int* abort = nullptr) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_test(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (global_ns() - t0 > limit_ns) {
      if (fault) atomicOr(fault, code);
      if (abort) *abort = 1;
      return false;
    }
  }
}
MSA_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* fault, unsigned code,
                       volatile int* abort = nullptr) {
  return mbar_wait_for(bar, parity, fault, code, kWaitLimitNs, abort);
}

// try_wait with a suspend-time hint: the thread is suspended by the hardware
// until the phase completes or `hint_ns` elapses, so a waiting warp takes no
// issue slots from the warps doing the work.
MSA_DEV bool mbar_test_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// mbar_wait whose polls sleep (up to 100 us each) instead of spinning; the
// same 2 s limit, abort flag and fault report.
MSA_DEV bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, unsigned* fault, unsigned code,
                             volatile int* abort = nullptr) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_test_hint(bar, parity, 100000u)) return true;
    if (abort != nullptr && *abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      if (fault) atomicOr(fault, code);
      if (abort) *abort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
MSA_DEV void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
MSA_DEV void tma_load_3d(void* dst, const void* map, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
MSA_DEV void tma_load_4d(void* dst, const void* map, uint64_t* bar, int c0, int c1, int c2,
                         int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
// Generic-proxy shared-memory writes become visible to the async proxy
// (tensor core operand reads) after this fence.
MSA_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05
MSA_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
MSA_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MSA_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
MSA_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MSA_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D(tmem) (+)= A(smem desc) * B(smem desc)
MSA_DEV void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem desc)
MSA_DEV void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every MMA this thread issued before has completed.
MSA_DEV void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (tile base 1024-byte
// aligned; the start address may advance by 32-byte steps along K inside a
// swizzle row). lbo/sbo in bytes.
MSA_DEV uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
// a_mn / b_mn: operand stored MN-major (else K-major).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                          // D format: f32
         | (1u << 7)                        // A format: bf16
         | (1u << 10)                       // B format: bf16
         | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17)         // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}
// The same with A and B both f16 (format code 0) when f16, else both bf16.
__host__ __device__ constexpr uint32_t idesc_16bit_f32(int M, int N, bool a_mn, bool b_mn,
                                                       bool f16) {
  return f16 ? (idesc_bf16_f32(M, N, a_mn, b_mn) & ~((1u << 7) | (1u << 10)))
             : idesc_bf16_f32(M, N, a_mn, b_mn);
}

// 32 lanes x 32 bits x 16 columns: thread i of the warp reads lane (base + i),
// columns [col, col + 16). Load and wait in one statement, so the registers are
// valid when the statement retires.
MSA_DEV void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

MSA_DEV void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32 bits x 16 columns store, completed before the statement retires.
MSA_DEV void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// 32 lanes x 32 bits x 8 columns load / store without the completion wait
// (several may be issued, then one tmem_wait_ld / tmem_wait_st).
MSA_DEV void tmem_ld8_nowait(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
}
MSA_DEV void tmem_st8_nowait(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
MSA_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
MSA_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 bits x 8 columns, waited.
MSA_DEV void tmem_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  tmem_ld8_nowait(taddr, r);
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

MSA_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
MSA_DEV uint32_t pack_f16x2(float lo, float hi) {
  __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
// Two floats as a packed pair of the 16-bit type of the operands (lo first).
template <bool F16>
MSA_DEV uint32_t pack_x2(float lo, float hi) {
  return F16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

// Four E4M3 ("fn") codes, lowest byte first, to four bf16 values (two packed
// pairs), exactly: E4M3 -> f16 is exact, and so is f16 -> bf16 for every
// E4M3 value (NaN stays NaN). (An integer-only decode that scales the placed
// bits by 2^120 was measured slower than these conversions.)
MSA_DEV void e4m3x4_to_bf16(uint32_t w, uint32_t& lo, uint32_t& hi) {
#pragma unroll
  for (int y = 0; y < 2; ++y) {
    const uint16_t pair = (uint16_t)(w >> (16 * y));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
    (y == 0 ? lo : hi) = pack_bf16x2(f.x, f.y);
  }
}

// Four E4M3 ("fn") codes, lowest byte first, to four f16 values (two packed
// pairs), exactly (every E4M3 value is an f16 value).
MSA_DEV void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((uint16_t)(w & 0xffffu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((uint16_t)(w >> 16)));
}

// Bytes of one (page, KV head) slice of packed NVFP4: 128 tokens x 64 bytes of
// E2M1 pairs, and 128 x 8 E4M3 block scales (one per 16 elements).
constexpr uint32_t kFp4Data = 128 * 64;
constexpr uint32_t kFp4Scales = 128 * 8;

// Byte offset of token r's block scale s (0..7) in a slice's scale region:
// token-major for K; for V, 4 x 4 tiles of (token, scale index) in row-major
// tile order, each tile scale-index major.
MSA_DEV int fp4_scale_offset(bool v_order, int r, int s) {
  return v_order ? 32 * (r >> 2) + 16 * (s >> 2) + 4 * (s & 3) + (r & 3) : r * 8 + s;
}

// Sixteen E2M1 codes (eight bytes, element 2i in the low nibble of byte i)
// times their E4M3 block scale, as eight packed bf16 pairs. Exact: E2M1 and
// E4M3 are exact in f16, their product (at most 6 significant bits, magnitude
// 2^-10 .. 2688) is exact in f16 and in bf16.
MSA_DEV void fp4x16_to_bf16(uint2 codes, uint8_t scale, uint32_t (&out)[8]) {
  uint32_t sc2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(sc2) : "h"((uint16_t)(scale | (scale << 8))));
  const __half2 s2 = *reinterpret_cast<const __half2*>(&sc2);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t word = i < 4 ? codes.x : codes.y;
    const uint16_t byte = (uint16_t)((word >> (8 * (i & 3))) & 0xFFu);
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h2)
        : "h"(byte));
    const __half2 v2 = __hmul2(*reinterpret_cast<const __half2*>(&h2), s2);
    const float2 f = __half22float2(v2);
    out[i] = pack_bf16x2(f.x, f.y);
  }
}

// Byte offset of the 16-byte chunk `c16` (0..7) of row `row` inside a
// 128-byte-swizzled tile whose rows are 128 bytes (the TMA SWIZZLE_128B image).
MSA_DEV uint32_t sw128_offset(uint32_t row, uint32_t c16) {
  return row * 128u + ((c16 ^ (row & 7u)) << 4);
}

MSA_DEV int elect_lane0() { return (threadIdx.x & 31) == 0; }

// Programmatic dependent launch: block until the grid launched before this
// one on the stream has completed and its writes are visible. A no-op when
// the kernel was launched without the programmatic-serialization attribute.
MSA_DEV void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel on the stream (launched with programmatic
// serialization) start its prologue now; it still waits for this grid's
// completion before reading its results.
MSA_DEV void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace msa
