// pkv_common.cuh -- device helpers shared by the libpkv kernels (sm_103a).
//
// Inline PTX for the pieces CUDA C++ does not expose directly: mbarrier
// waits with a time limit, 1-D bulk (TMA) copies of K/V rows into shared
// memory, ldmatrix / movmatrix fragment loads, mma.sync on bf16/f16 with fp32
// accumulation, and the e4m3 <-> f16/f32 conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// Bits of the device error word (see pkv_device_errors in pkv.h).
enum : unsigned int {
  kErrSlotRange = 1u,    // slot at or beyond num_blocks * block_size
  kErrBlockRange = 2u,   // block id outside [0, num_blocks)
  kErrLengths = 4u,      // q_s < 0, q_s > N_s or N_s beyond the block table
  kErrWaitTimeout = 8u,  // a bounded wait gave up
  kErrPlan = 16u,        // the workspace holds no plan for this call's shapes
};

// A bounded wait gives up after this many SM clock cycles (about 2 s).
constexpr long long kWaitLimitCycles = 4000000000LL;

// Logical tiling.  Every tile and split boundary is a logical token position
// so that the result does not depend on block_size or page placement.
constexpr int kChunkBaseShift = 7;    // smallest split-KV chunk: 128 tokens ...
constexpr int kChunkBaseShiftFp8 = 8; // ... 256 with an e4m3 cache (the same bytes per chunk)
constexpr int kMaxChunks = 512;       // a sequence is split into at most this many chunks
constexpr int kPrefillRows = 64;      // (query token, head) rows per prefill tile

// Chunk length of a decoding sequence of n keys: the smallest 2^base * 2^k
// that splits it into at most kMaxChunks chunks, as a shift (chunk =
// 1 << shift).  Depends on n (and the cache format) only.
__host__ __device__ inline int chunk_shift(int n, int base = kChunkBaseShift) {
  int k = base;
  while ((((unsigned)n + (1u << k) - 1u) >> k) > (unsigned)kMaxChunks) ++k;
  return k;
}
__host__ __device__ inline int chunk_tokens(int n, int base = kChunkBaseShift) { return 1 << chunk_shift(n, base); }

// Chunks of the longest sequence a block table of max_ctx tokens can hold
// (with the smallest base: a bound for every format).
__host__ __device__ inline int max_chunks_for(int64_t max_ctx) {
  if (max_ctx <= 0) return 1;
  const int n = max_ctx > 0x7fffffff ? 0x7fffffff : static_cast<int>(max_ctx);
  const int c = chunk_tokens(n);
  return (n + c - 1) / c;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase of the given parity to complete; gives up after
// kWaitLimitCycles, records kErrWaitTimeout and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) {
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
  return true;
}

// mbar_wait by every lane of a warp with one result for the whole warp, so
// that no lane goes on while another gives up (warp-collective instructions
// after the wait need every lane).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, unsigned int* err) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, err));
}

// 1-D bulk copy global -> shared, completion counted in bytes on an mbarrier.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// The same with an L2 cache policy (createpolicy): data read once, such as
// the K/V rows of a decode step, is marked evict-first, so that it does
// not push out what the next kernels read again (tables, work lists,
// split-KV partials).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel in the stream runs;
// grid_dep_wait() blocks until that kernel has completed and its writes are
// visible.  launch_dependents() lets the next kernel start early.  Both are
// no-ops for a kernel launched normally.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Named barrier over the first `threads` threads (consumer warps only).
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- fragments
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Transpose of an 8x8 b16 matrix held one pair per thread in the mma
// fragment layout (row lane/4, columns 2*(lane%4) and +1).
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// D += A(16x16, row) * B(16x8, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- conversions
// Two fp32 -> bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// Split p into a bf16 pair hi + lo with hi = bf16(p), lo = bf16(p - hi):
// hi + lo carries about 16 significant bits of p.
__device__ __forceinline__ void split_bf16(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(p0, p1);
  lo = pack_bf16(p0 - bf16_lo(hi), p1 - bf16_hi(hi));
}

// Two e4m3 codes (low byte first) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// Four e4m3 codes in a word -> two f16x2 (bytes 0,1 and bytes 2,3).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& r01, uint32_t& r23) {
  r01 = e4m3x2_to_f16x2(static_cast<uint16_t>(w & 0xFFFFu));
  r23 = e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16));
}

// Two fp32 -> two e4m3 codes (lo in the low byte): round to nearest even,
// saturate to +-448, NaN to NaN.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// bf16 pair -> f16 pair (round to nearest even; exact for |x| in the f16
// normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
  return pack_f16(bf16_lo(x), bf16_hi(x));
}

__device__ __forceinline__ float warp_max_xor(float v, int m) {
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
}

// Output element stores.
__device__ __forceinline__ void store2(float* p, float a, float b) {
  *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
__device__ __forceinline__ void store2(__nv_bfloat16* p, float a, float b) {
  *reinterpret_cast<uint32_t*>(p) = pack_bf16(a, b);
}
__device__ __forceinline__ void store1(float* p, float a) { *p = a; }
__device__ __forceinline__ void store1(__nv_bfloat16* p, float a) { *p = __float2bfloat16_rn(a); }

// Index of the last entry of the non-decreasing prefix array off[0..n] that
// is <= x (off[0] = 0 <= x < off[n]).
__device__ __forceinline__ int upper_index(const int32_t* off, int n, int x) {
  int lo = 0, hi = n;  // off[lo] <= x < off[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (__ldg(off + mid) <= x)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

}  // namespace pkv
