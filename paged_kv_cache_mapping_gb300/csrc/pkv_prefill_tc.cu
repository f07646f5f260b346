// pkv_prefill_tc.cu -- causal prefill attention on the fifth-generation
// tensor cores: tcgen05 MMAs with the accumulators in tensor memory (TMEM),
// operands staged by TMA tensor copies with 128-byte swizzle.
//
// nanoserve, "Architecture" step 3 and its chunked-prefill notes: the query
// tokens of a prefill chunk attend causally over the cached prefix and the
// chunk itself, in the same packed step as the decodes.  A tile of 128 query
// rows (whole tokens x the G query heads of one KV head) against a tile of
// 128 keys is a dense contraction, run here as
//     S = Q K^T      (M 128, N 128 keys, K = D; bf16 in, fp32 in TMEM)
//     O += P V       (M 128, N = D, K 128 keys; P split into bf16 hi + lo)
// with an online softmax (base 2) between them, two threads per query row.
// P never leaves tensor memory: the softmax threads overwrite their row of S
// with the hi and lo bf16 parts of P (64 packed columns each) and the P V
// MMAs read their A operand from there.  The softmax arithmetic runs as
// packed f32x2 operations where it can: the MMA-issuing warp shares a
// scheduler with two softmax warps, and a dense stream of FMA-pipe
// instructions there delays its MMA issues.  An M 128 x N 128 x K 16 MMA keeps
// the tensor core at its full rate; N 64 would run at about two thirds.
//
// e4m3 caches ("How Easy Is It to Start Serving LLMs?", the FP8 KV cache
// setting): the MMAs take f16 operands.  A K or V tile's codes land at the
// end of its stage and the producer warp converts them in place to f16
// (exact), in the swizzled layout a bf16 tile has; the softmax warps convert
// each unit's Q tile from bf16 to f16 in place; P is one f16 part (P V runs
// once).  The scales are folded into the exponent and the output, as in the
// decode kernel.
//
// CTA (one per SM, persistent over tiles), 11 warps:
//   warp 0   TMA producer: claims work units, loads the Q tile of each (two
//            Q buffers: the next unit's Q arrives while this unit runs) and
//            its K tiles of 128 keys (boxes of 16 consecutive slots of one
//            head per d half, or of 8 for block sizes that are 8 mod 16, so
//            that a box lies in one block) into a 2-stage ring.
//   warp 2   TMA producer of the V tiles, in its own 2-stage ring.
//            Keys past the sequence and bad block ids read out of bounds,
//            which TMA fills with zeros.
//   warp 1   MMA issuer (one thread) and owner of the TMEM allocation
//            (S / P double-buffered in columns 0-255, O double-buffered in
//            256-511: a unit's O is read out after the next unit's first tile).
//            MMAs issued by one thread run in issue order, so the Q K^T that
//            overwrites an S buffer is issued after the P V that reads it.
//   warps 3-10  softmax, two threads per query row (a warp may only reach
//            the TMEM lanes of its quarter, so warps w and w + 4 share rows;
//            the first takes keys 0-63 of each tile, the second 64-127).
//            Each thread loads its half row of S from TMEM, masks it (only
//            on tiles that cut a row's visible range), trades its partial
//            max with its partner through shared memory, writes its half of
//            P in place and, only when the row's max grows by more than 2^8,
//            waits for the previous P V and rescales its half of the row of
//            O in TMEM; at the end the partners add their sums and each
//            writes half of O / l.  Q K^T of the next tile and P V of the
//            previous one run on the tensor core meanwhile.
// Block sizes must be multiples of 8.
#include <cuda.h>

#include <mutex>

#include "pkv_kernels.h"

namespace pkv {
namespace {

constexpr int kTcRows = 128;    // query rows per tile (MMA M)
constexpr int kTcKeys = 128;    // keys per key tile (MMA N of Q K^T, K of P V)
constexpr int kKStages = 2;     // K ring depth
constexpr int kVStages = 2;     // V ring depth
constexpr int kQBufs = 2;       // Q tiles: the next unit's Q is loaded while this unit runs
constexpr int kTcThreads = 352;  // 11 warps
constexpr int kSoftmaxWarp0 = 3; // warps 3-10: two per TMEM lane quarter
// A row's reference max moves only when a tile's max exceeds it by more than
// this (log2 units), so p = 2^(x - m_ref) stays below 2^8 and O needs a
// rescale in TMEM only then.
constexpr float kTcTau = 8.f;

template <int D>
struct TcGeom {
  static constexpr int kHalves = D / 64;                     // 128-byte atoms along d
  static constexpr int kQBytes = kHalves * kTcRows * 128;
  static constexpr int kKVBytes = kHalves * kTcKeys * 128;   // one K or V tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBufs * kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kKVBytes;
  static constexpr int kOffBar = kOffV + kVStages * kKVBytes;
  static constexpr int kOffX = kOffBar + 512;                 // row max / sum exchange [2][2][kTcRows]
  static constexpr int kSmem = kOffX + 4 * kTcRows * 4 + 1024; // + 1024-byte alignment slack
  static constexpr uint32_t kTmemCols = 512;                  // S / P 2 x 128 columns, O 2 x 128 columns
  static constexpr uint32_t kColO = 2 * kTcKeys;              // O of unit parity b at kColO + 128 b
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(kColO + 128 + D <= kTmemCols, "tensor memory");
};

// ---- tcgen05 / TMA wrappers
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  // shared-memory matrix descriptor: start >> 4, leading and stride byte
  // offsets >> 4, descriptor version 1, 128-byte swizzle
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// instruction descriptor, kind::f16: fp32 accumulator, A and B both bf16
// (f16 = false) or both f16, K-major A, B K-major (b_mn = 0) or MN-major
// (b_mn = 1), M = 128, N = n
__host__ __device__ constexpr uint32_t umma_idesc(int n, int b_mn, bool f16 = false) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcRows >> 4) << 24);
}

// The MMA and commit wrappers are executed by the whole (converged) warp
// and issue from one lane chosen by elect.sync: the operands are then the
// same in every lane and stay in the uniform datapath.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// the same with A read from tensor memory: row r of A in lane r, column c
// holding elements 2c (low half) and 2c + 1 (high half) of the row
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define PKV_R32(x) \
  "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]), "=r"(x[8]), \
      "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15]), "=r"(x[16]), \
      "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]), "=r"(x[24]), \
      "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
#define PKV_W32(x) \
  "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]), "r"(x[8]), "r"(x[9]), \
      "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]), "r"(x[15]), "r"(x[16]), "r"(x[17]), "r"(x[18]), \
      "r"(x[19]), "r"(x[20]), "r"(x[21]), "r"(x[22]), "r"(x[23]), "r"(x[24]), "r"(x[25]), "r"(x[26]), "r"(x[27]), \
      "r"(x[28]), "r"(x[29]), "r"(x[30]), "r"(x[31])
#define PKV_ARGS32                                                                                                \
  "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, " \
  "%24, %25, %26, %27, %28, %29, %30, %31}"

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&x)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " PKV_ARGS32 ", [%32];" : PKV_R32(x) : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&x)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
               "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::
                   "r"(taddr),
               PKV_W32(x));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of fp32 (sm_100 f32x2 arithmetic): one instruction does two
// lanes' worth of the FMA-pipe work, which leaves more issue slots to the
// MMA-issuing warp that shares a scheduler with softmax warps.
// three-input max (sm_100): exact, like two fmaxf
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ unsigned long long pk2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void up2(unsigned long long v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Work unit u: prefill tile u / Hkv (tokens r0 .. r1-1 of its sequence,
// the last tokens first), KV head u % Hkv.  Key tiles are numbered across
// the CTA's units (g); tile g uses K/V stage g % 3 and S / P buffer g % 2,
// and signals o_done[g % 2] when its P V has finished.
template <int D>
__device__ __forceinline__ unsigned char* tc_smem() {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  return smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
}

// What warp 0 reads once the previous kernel has completed, in one round
// trip: the plan check and the prefill CTA count.
struct TcStart {
  int ok, active, n_units, pad;  // n_units: written by active CTAs after the check
};

// The barrier area (8-byte slots from Geo::kOffBar): mbarriers, the TMEM
// address, the abort flag, the unit ring and its descriptors, the start
// record.
enum : int {
  kBarQFull = 0, kBarQEmpty = 2, kBarKFull = 4, kBarKEmpty = 6, kBarVFull = 8, kBarVEmpty = 10,
  kBarSFull = 12, kBarPFull = 14, kBarODone = 16, kBarDrain = 18, kSlotTmem = 19, kSlotAbort = 20,
  kBarUnitFull = 21, kBarUnitEmpty = 23, kSlotUnitRing = 25, kBarX = 26, kBarOFree = 34,
  kBarKsFull = 36, kBarVsFull = 38, kBarQConv = 40,  // e4m3 caches: tile copies landed, Q converted
  kOffUnitDesc = 384,  // bytes: PrefillDesc[2]
  kOffStart = 448,     // bytes: TcStart
};

// Barriers, set up before the dependency wait (no global memory access),
// and the tensor maps prefetched.
template <int D>
__device__ __forceinline__ void prefill_tc_setup(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                                 const CUtensorMap& tm_v) {
  using Geo = TcGeom<D>;
  unsigned char* smem = tc_smem<D>();
  const uint32_t b0 = smem_u32(smem + Geo::kOffBar);
  auto bar = [&](int i) -> uint32_t { return b0 + 8 * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < kQBufs; ++b) {
      mbar_init(bar(kBarQFull + b), 1);
      mbar_init(bar(kBarQEmpty + b), 1);
      mbar_init(bar(kBarQConv + b), 8);  // the softmax warps
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarSFull + b), 1);
      mbar_init(bar(kBarPFull + b), 8);
      mbar_init(bar(kBarODone + b), 1);
      mbar_init(bar(kBarOFree + b), 8);
      mbar_init(bar(kBarUnitFull + b), 1);
      mbar_init(bar(kBarUnitEmpty + b), 10);  // the V producer, the MMA warp and the 8 softmax warps
    }
    mbar_init(bar(kBarDrain), 1);
    for (int s = 0; s < kKStages; ++s) mbar_init(bar(kBarKsFull + s), 1);
    for (int s = 0; s < kVStages; ++s) mbar_init(bar(kBarVsFull + s), 1);
    for (int q = 0; q < 4; ++q) {
      mbar_init(bar(kBarX + 2 * q), 2);
      mbar_init(bar(kBarX + 2 * q + 1), 2);
    }
    *reinterpret_cast<volatile int*>(smem + Geo::kOffBar + 8 * kSlotAbort) = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane < 3) {
    const CUtensorMap* m = lane == 0 ? &tm_q : lane == 1 ? &tm_k : &tm_v;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
  }
}

template <int D, typename OutT, bool KV8>
__device__ __forceinline__ void prefill_tc_body(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                                const CUtensorMap& tm_v, int active, int n_units,
                                                int first_word) {
  using Geo = TcGeom<D>;
  unsigned char* smem = tc_smem<D>();
  const uint32_t sQ = smem_u32(smem + Geo::kOffQ);
  const uint32_t sK = smem_u32(smem + Geo::kOffK);
  const uint32_t sV = smem_u32(smem + Geo::kOffV);
  const uint32_t b0 = smem_u32(smem + Geo::kOffBar);
  auto bar = [&](int i) -> uint32_t { return b0 + 8 * i; };
  // Q buffer b of unit parity b: filled (q_full), read by the unit's last
  // Q K^T (q_empty)
  auto q_full = [&](int b) { return bar(kBarQFull + b); };
  auto q_empty = [&](int b) { return bar(kBarQEmpty + b); };
  auto q_buf = [&](int b) { return sQ + b * Geo::kQBytes; };
  const uint32_t drain = bar(kBarDrain);
  auto k_full = [&](int s) { return bar(kBarKFull + s); };
  auto k_empty = [&](int s) { return bar(kBarKEmpty + s); };
  auto v_full = [&](int s) { return bar(kBarVFull + s); };
  auto v_empty = [&](int s) { return bar(kBarVEmpty + s); };
  auto s_full = [&](int b) { return bar(kBarSFull + b); };
  auto p_full = [&](int b) { return bar(kBarPFull + b); };
  auto o_done = [&](int b) { return bar(kBarODone + b); };
  auto o_free = [&](int b) { return bar(kBarOFree + b); };  // O buffer b read out by the epilogue
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Geo::kOffBar + 8 * kSlotTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Geo::kOffBar + 8 * kSlotAbort);
  // work units: the TMA warp claims them and passes each index, with its
  // descriptor, to the other warps through a 2-slot ring (no warp reads a
  // descriptor from global memory on its way into a unit)
  auto unit_full = [&](int b) { return bar(kBarUnitFull + b); };
  auto unit_empty = [&](int b) { return bar(kBarUnitEmpty + b); };
  volatile int* unit_ring = reinterpret_cast<volatile int*>(smem + Geo::kOffBar + 8 * kSlotUnitRing);
  PrefillDesc* unit_desc = reinterpret_cast<PrefillDesc*>(smem + Geo::kOffBar + kOffUnitDesc);  // [2]
  // the two softmax warps of TMEM lane quarter q trade per-row values
  // through buffer b of xval, paired by barrier xbar(q, b)
  auto xbar = [&](int q, int b) { return bar(kBarX + 2 * q + b); };
  // e4m3 caches: a K / V tile's copies land in stage s (ks_full / vs_full)
  // before its codes are converted; the MMAs wait for Q in f16 (q_conv)
  auto ks_full = [&](int s) { return bar(kBarKsFull + s); };
  auto vs_full = [&](int s) { return bar(kBarVsFull + s); };
  auto q_conv = [&](int b) { return bar(kBarQConv + b); };
  float* xval = reinterpret_cast<float*>(smem + Geo::kOffX);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the abort flag as one value for the whole warp (another warp may set it
  // between two lanes' reads)
  auto aborted = [&]() -> bool { return __any_sync(0xffffffffu, *abort_flag != 0); };
  const uint32_t tmem = *tslot;
  const uint32_t tO = tmem + Geo::kColO;  // S / P buffers: columns 0 .. 2 * kTcKeys - 1; O buffers from here

  const int G = p.G, Hkv = p.Hkv;
  const int tq = p.pf_tq;  // query tokens per tile
  const uint32_t q_box_bytes = (uint32_t)(Geo::kHalves * G * tq * 128);

  // Key tiles of a unit: from the first tile any of its rows sees (a sliding
  // window skips the ones before) to the tile of its last row's last key.
  auto unit_tiles = [&](const PrefillDesc& e, int& kt0, int& n_kt) {
    const int first = p.window_left >= 0 ? max(0, e.n - e.q_s + e.r0 - p.window_left) : 0;
    kt0 = first / kTcKeys;
    n_kt = (e.kv_end + kTcKeys - 1) / kTcKeys - kt0;
  };
  // e4m3 caches: a tile's codes (kTcKeys rows of D bytes) land at the end of
  // its f16 stage and are converted in place into the 128-byte-swizzled
  // layout the bf16 tiles have (16-byte chunk c of key r's row in d half h
  // at h * kTcKeys * 128 + r * 128 + ((c ^ (r % 8)) * 16)); e4m3 -> f16 is
  // exact.  Lane l reads 16 codes of one key (d 16 j .. 16 j + 15) and
  // writes the two f16 chunks they make.  A written chunk only covers code
  // rows read by this or an earlier loop step: with D = 128 a key's codes
  // sit where its own d half 1 goes; with D = 64 output row r covers code
  // rows 2 r - 128 and 2 r - 127 (r >= 64), never past the rows read so far.
  constexpr int kStage8 = Geo::kKVBytes - kTcKeys * D;  // codes' offset in a stage
  auto convert_kv = [&](uint32_t stage) {
    constexpr int kCpr = D / 16;         // 16-code chunks per key
    constexpr int kKeysPer = 32 / kCpr;  // keys per loop step
    const int j = lane % kCpr, rr = lane / kCpr;
    const int hh = j / 4, c0 = 2 * (j % 4);  // d half and first chunk of the 16 codes
#pragma unroll 4
    for (int r0 = 0; r0 < kTcKeys; r0 += kKeysPer) {
      const int r = r0 + rr;
      uint4 w;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                   : "r"(stage + kStage8 + r * D + 16 * j));
      __syncwarp();
      uint32_t f[8];
      e4m3x4_to_f16(w.x, f[0], f[1]);
      e4m3x4_to_f16(w.y, f[2], f[3]);
      e4m3x4_to_f16(w.z, f[4], f[5]);
      e4m3x4_to_f16(w.w, f[6], f[7]);
      const uint32_t row = stage + hh * kTcKeys * 128 + r * 128;
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((c0 ^ (r & 7)) << 4)), "r"(f[0]),
                   "r"(f[1]), "r"(f[2]), "r"(f[3])
                   : "memory");
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (((c0 + 1) ^ (r & 7)) << 4)), "r"(f[4]),
                   "r"(f[5]), "r"(f[6]), "r"(f[7])
                   : "memory");
      __syncwarp();
    }
  };
  // K or V tiles of one unit, one TMA box per issuing lane (bx keys x one d
  // half, or bx keys x D e4m3 codes; bx = 16, or 8 for block sizes that are
  // 8 mod 16, so that a box never crosses a block); the block-table entry of
  // the next tile is loaded while this one is issued.  e4m3 tiles are
  // converted one tile behind their copies.  claim: called (by the K
  // producer) after the tile kt_claim is issued.
  auto stream_kv = [&](const PrefillDesc& e, int hk, int& g, bool is_v, int kt_claim, auto&& claim) -> bool {
    const int64_t n_slots = p.num_blocks * p.bs;
    const int32_t* bt_row = p.bt + (int64_t)e.s * p.bt_stride;
    int kt0, n_kt;
    unit_tiles(e, kt0, n_kt);
    const int bx = (p.bs & 15) == 0 ? 16 : 8;
    const int n_box = kTcKeys / bx;                       // boxes per d half (per tile for e4m3)
    const int bi = lane % n_box;                          // keys bx bi .. bx bi + bx - 1 of the tile
    const bool issuer = lane < n_box * (KV8 ? 1 : Geo::kHalves);
    constexpr int32_t kPast = INT32_MIN;  // a block past the sequence
    const CUtensorMap* map = is_v ? &tm_v : &tm_k;
    const uint32_t base = is_v ? sV : sK;
    const int ns = is_v ? kVStages : kKStages;
    auto load_blk = [&](int kt) -> int32_t {
      const int key0 = (kt0 + kt) * kTcKeys + bx * bi;
      int32_t v = kPast;
      if (key0 < e.n) v = __ldg(bt_row + (p.bs_shift >= 0 ? (key0 >> p.bs_shift) : (key0 / p.bs)));
      return v;
    };
    // e4m3: convert tile gg (waits for its copies), then hand it to the MMAs
    auto convert = [&](int gg) -> bool {
      const int st = gg % ns, ph = (gg / ns) & 1;
      if (!mbar_wait_warp(is_v ? vs_full(st) : ks_full(st), ph, p.err)) return false;
      convert_kv(base + st * Geo::kKVBytes);
      fence_proxy_async_smem();  // the MMAs read the f16 tile through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(is_v ? v_full(st) : k_full(st));
      return true;
    };
    int32_t blk = load_blk(0);
    for (int kt = 0; kt < n_kt; ++kt, ++g) {
      int32_t nxt = kPast;
      if (kt + 1 < n_kt) nxt = load_blk(kt + 1);
      const int key0 = (kt0 + kt) * kTcKeys + bx * bi;
      int slot = (int)n_slots;  // out of bounds: TMA fills zeros
      if ((uint32_t)blk < (uint32_t)p.num_blocks) {
        const int lb = p.bs_shift >= 0 ? (key0 >> p.bs_shift) : (key0 / p.bs);
        slot = blk * p.bs + (key0 - lb * p.bs);
      } else if (blk != kPast) {
        atomicOr(p.err, kErrBlockRange);
      }
      const int st = g % ns, ph = (g / ns) & 1;
      const uint32_t empty = is_v ? v_empty(st) : k_empty(st);
      if (!mbar_wait_warp(empty, ph ^ 1, p.err)) return false;
      if constexpr (KV8) {
        const uint32_t landed = is_v ? vs_full(st) : ks_full(st);
        if (lane == 0) mbar_arrive_expect_tx(landed, kTcKeys * D);
        __syncwarp();
        if (issuer) tma_load_3d(base + st * Geo::kKVBytes + kStage8 + bi * bx * D, map, 0, hk, slot, landed);
      } else {
        const uint32_t full = is_v ? v_full(st) : k_full(st);
        if (lane == 0) mbar_arrive_expect_tx(full, Geo::kKVBytes);
        __syncwarp();
        const int h = lane / n_box;  // d half
        if (issuer) tma_load_3d(base + st * Geo::kKVBytes + h * kTcKeys * 128 + bi * bx * 128, map, h * 64, hk, slot,
                                full);
      }
      if (kt == kt_claim) claim();
      if (KV8 && kt > 0 && !convert(g - 1)) return false;
      blk = nxt;
    }
    if (KV8 && n_kt > 0 && !convert(g - 1)) return false;
    return true;
  };
  // giving up: let the copies a producer warp issued land before the CTA exits
  auto drain_copies = [&](int g, bool is_v) {
    const int ns = is_v ? kVStages : kKStages;
    for (int k = g - 1; k >= 0 && k >= g - ns; --k) {
      const int st = k % ns, ph = (k / ns) & 1;
      if (KV8)
        mbar_wait_warp(is_v ? vs_full(st) : ks_full(st), ph, p.err);
      else
        mbar_wait_warp(is_v ? v_full(st) : k_full(st), ph, p.err);
    }
  };

  if (warp == 0) {
    // ======================= TMA producer: units, Q and K =======================
    int g = 0, q_it = 0, ui = 0;
    // hands unit index x (>= n_units: no more units) and its descriptor to
    // the other warps
    auto publish = [&](int x, const PrefillDesc& e) -> bool {
      if (!mbar_wait_warp(unit_empty(ui & 1), ((ui >> 1) & 1) ^ 1, p.err)) return false;
      if (lane == 0) {
        unit_ring[ui & 1] = x;
        unit_desc[ui & 1] = e;
        mbar_arrive(unit_full(ui & 1));
      }
      __syncwarp();
      ++ui;
      return true;
    };
    // the first unit of a CTA is fixed; later ones are claimed in order, the
    // longest first, when this warp has three K tiles of the current unit
    // left to issue (its first tile, for shorter units): late enough that
    // CTAs finishing early take more of the remaining units, early enough
    // that the claim's round trip is over when the next unit's Q and K tiles
    // are due
    int u = blockIdx.x;
    for (; !aborted(); ++q_it) {
      PrefillDesc e{};
      if (q_it == 0) {  // word i of the first unit's descriptor is in lane i
#pragma unroll
        for (int i = 0; i < 8; ++i)
          reinterpret_cast<int32_t*>(&e)[i] = __shfl_sync(0xffffffffu, first_word, i);
      } else if (u < n_units) {
        e = p.ws.pf_desc[u / Hkv];
      }
      if (!publish(u, e)) { *abort_flag = 1; break; }
      if (u >= n_units) break;
      // claim c of the plan's runs names unit c mod n_units (see Workspace)
      unsigned long long c = 0;
      auto claim = [&]() {
        if (lane == 0) c = atomicAdd(p.ws.pf_work, 1ull);
      };
      int kt0, n_kt;
      unit_tiles(e, kt0, n_kt);
      const int hk = u - (u / Hkv) * Hkv;
      const int qb = q_it & 1;  // this unit's Q buffer
      if (!mbar_wait_warp(q_empty(qb), ((q_it >> 1) & 1) ^ 1, p.err)) { *abort_flag = 1; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full(qb), q_box_bytes);
        for (int h = 0; h < Geo::kHalves; ++h)
          tma_load_3d(q_buf(qb) + h * kTcRows * 128, &tm_q, h * 64, hk * G, e.t0 + e.r0, q_full(qb));
      }
      if (!stream_kv(e, hk, g, false, max(0, n_kt - 3), claim)) { *abort_flag = 1; break; }
      int next = 0;
      if (lane == 0) next = static_cast<int>(active + c % static_cast<unsigned long long>(n_units));
      u = __shfl_sync(0xffffffffu, next, 0);
    }
    if (aborted()) drain_copies(g, false);
  } else if (warp == 2) {
    // ======================= TMA producer: V =======================
    // runs on its own so that K tiles are not held back by the V ring
    int g = 0, ui = 0;
    while (!aborted()) {
      if (!mbar_wait_warp(unit_full(ui & 1), (ui >> 1) & 1, p.err)) { *abort_flag = 1; break; }
      const int u = unit_ring[ui & 1];
      const PrefillDesc e = unit_desc[ui & 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(unit_empty(ui & 1));
      ++ui;
      if (u >= n_units) break;
      if (!stream_kv(e, u - (u / Hkv) * Hkv, g, true, -1, [] {})) { *abort_flag = 1; break; }
    }
    if (aborted()) drain_copies(g, true);
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    constexpr uint32_t kIdQK = umma_idesc(kTcKeys, 0, KV8);
    constexpr uint32_t kIdPV = umma_idesc(D, 1, KV8);
    int g = 0, ui = 0;
    bool ok = true;
    // S[gg % 2] = Q K^T for key tile gg (global numbering) against Q buffer qb
    auto issue_qk = [&](int gg, int qb) -> bool {
      const int st = gg % kKStages, ph = (gg / kKStages) & 1, sb = gg & 1;
      // S buffer sb last held P of tile gg - 2, whose P V was issued before
      // this Q K^T (issue order is execution order)
      if (!mbar_wait_warp(k_full(st), ph, p.err)) return false;
      tc_fence_after();
      {
        // a descriptor's start address is its low field (bytes >> 4): the
        // k steps add constant offsets to one base descriptor per operand
        const uint64_t dq = umma_desc(q_buf(qb), 16, 1024), dk = umma_desc(sK + st * Geo::kKVBytes, 16, 1024);
#pragma unroll
        for (int kb = 0; kb < D / 16; ++kb) {
          const uint32_t kq = ((kb >> 2) * kTcRows * 128 + (kb & 3) * 32) >> 4;
          const uint32_t kk = ((kb >> 2) * kTcKeys * 128 + (kb & 3) * 32) >> 4;
          umma_bf16(tmem + sb * kTcKeys, dq + kq, dk + kk, kIdQK, kb > 0);
        }
        umma_commit(s_full(sb));
        umma_commit(k_empty(st));
      }
      __syncwarp();
      return true;
    };
    // unit number q_it from the ring (u >= n_units: none left) and, for a
    // real one, its Q tile ready in buffer q_it % 2
    auto next_unit = [&](int q_it, int& u, PrefillDesc& e) -> bool {
      u = n_units;
      if (!mbar_wait_warp(unit_full(ui & 1), (ui >> 1) & 1, p.err)) return false;
      u = unit_ring[ui & 1];
      e = unit_desc[ui & 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(unit_empty(ui & 1));
      ++ui;
      if (u >= n_units) return true;
      const int qb = q_it & 1;
      return mbar_wait_warp(KV8 ? q_conv(qb) : q_full(qb), (q_it >> 1) & 1, p.err);
    };
    int u = n_units;
    PrefillDesc e{};
    ok = next_unit(0, u, e);
    if (ok && u < n_units) ok = issue_qk(0, 0);  // the first unit's first tile (every unit has one)
    for (int q_it = 0; ok && u < n_units && !aborted(); ++q_it) {
      int kt0, n_kt;
      unit_tiles(e, kt0, n_kt);
      const int ob = q_it & 1;  // O buffer of this unit (the epilogue may still read the other)
      const int qb = q_it & 1;  // its Q buffer
      const uint32_t tOu = tO + ob * 128;
      int u2 = n_units;
      PrefillDesc e2{};
      for (int t = 0; t < n_kt && ok; ++t) {
        const int gg = g + t;
        if (t + 1 < n_kt) {
          ok = issue_qk(gg + 1, qb);
        } else {
          umma_commit(q_empty(qb));  // the unit's Q is no longer read
          // the next unit's first Q K^T goes ahead of this unit's last P V,
          // as within a unit, so that the softmax warps find its S ready
          // (not with e4m3 caches: that Q is converted by the softmax warps
          // after this unit's last P, which the P V below waits for)
          if (!KV8) {
            ok = next_unit(q_it + 1, u2, e2);
            if (ok && u2 < n_units) ok = issue_qk(gg + 1, (q_it + 1) & 1);
          }
        }
        if (!ok) break;
        const int st = gg % kVStages, ph = (gg / kVStages) & 1, pb = gg & 1;
        ok = mbar_wait_warp(p_full(pb), (gg >> 1) & 1, p.err) && mbar_wait_warp(v_full(st), ph, p.err) &&
             (t > 0 || mbar_wait_warp(o_free(ob), ((q_it >> 1) & 1) ^ 1, p.err));
        if (!ok) break;
        tc_fence_after();
        {
          // P hi in columns 0-63 of the buffer, P lo in 64-127 (e4m3 caches:
          // P in f16, columns 0-63): 16 keys are 8 columns; V is MN-major, 16
          // keys = 2048 bytes of each d half
          const uint32_t tp = tmem + pb * kTcKeys;
          const uint64_t dv = umma_desc(sV + st * Geo::kKVBytes, kTcKeys * 128, 1024);
          const uint32_t acc0 = t > 0;
#pragma unroll
          for (int kk = 0; kk < kTcKeys / 16; ++kk) {
            umma_bf16_ta(tOu, tp + kk * 8, dv + kk * 128, kIdPV, kk > 0 ? 1u : acc0);  // P (hi)
            if (!KV8) umma_bf16_ta(tOu, tp + kTcKeys / 2 + kk * 8, dv + kk * 128, kIdPV, 1);  // P lo
          }
          umma_commit(o_done(pb));
          umma_commit(v_empty(st));
        }
        __syncwarp();
      }
      g += n_kt;
      if (KV8 && ok) {
        ok = next_unit(q_it + 1, u2, e2);
        if (ok && u2 < n_units) ok = issue_qk(g, (q_it + 1) & 1);
      }
      u = u2;
      e = e2;
    }
    if (!ok || aborted()) {
      // giving up: every MMA issued so far must finish before TMEM is freed
      *abort_flag = 1;
      umma_commit(drain);
      __syncwarp();
      mbar_wait_warp(drain, 0, p.err);
    }
  } else {
    // ======================= softmax / epilogue (warps 3-10) =======================
    const int quarter = warp & 3;                        // TMEM lanes 32 * quarter ..
    const int half = (warp - kSoftmaxWarp0) >> 2;        // keys 64 half .. of each tile
    const int r = 32 * quarter + lane;                   // this thread's query row
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    constexpr int kHalfKeys = kTcKeys / 2;
    constexpr int kHalfD = D / 2;
    int g = 0, ui = 0, xj = 0, uc = 0;  // uc: units begun (O buffer parity)
    bool ok = true;
    // The epilogue of a unit, run after the next unit's first tile (or at
    // the end): wait for the unit's last P V, then write this thread's half
    // of its row of O / l and hand the O buffer back.  The last P V's
    // barrier cannot have moved on meanwhile: the next P V on that barrier
    // needs a P that this warp writes only after the epilogue.
    bool pend = false, pend_valid = false;
    int pend_lg = 0, pend_ob = 0;
    float pend_inv = 0.f;
    OutT* pend_dst = nullptr;
    auto epilogue = [&]() -> bool {
      pend = false;
      if (!mbar_wait_warp(o_done(pend_lg & 1), (pend_lg >> 1) & 1, p.err)) return false;
      tc_fence_after();
      const uint32_t to = tO + pend_ob * 128 + lane_off;
      const float inv = pend_inv;
#pragma unroll 1
      for (int c = kHalfD * half; c < kHalfD * (half + 1); c += 32) {
        uint32_t v[32];
        tmem_ld32(to + c, v);
        tmem_wait_ld();
        if (pend_valid) {
          OutT* d = pend_dst + c;
          if ((reinterpret_cast<uintptr_t>(d) & 15u) == 0) {  // 16-byte stores (same rounding as store2)
            constexpr int kPer = 16 / (int)sizeof(OutT);     // elements per store
#pragma unroll
            for (int j = 0; j < 32; j += kPer) {
              uint4 w;
              uint32_t* wu = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if constexpr (sizeof(OutT) == 2) {
                  wu[e] = pack_bf16(__uint_as_float(v[j + 2 * e]) * inv, __uint_as_float(v[j + 2 * e + 1]) * inv);
                } else {
                  wu[e] = __float_as_uint(__uint_as_float(v[j + e]) * inv);
                }
              }
              *reinterpret_cast<uint4*>(d + j) = w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; j += 2)
              store2(d + j, __uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free(pend_ob));
      return true;
    };
    // gives this thread's value for its row to the partner thread and
    // returns the partner's (double-buffered; the partner makes the same
    // sequence of calls)
    auto trade = [&](float mine, float& theirs) -> bool {
      const int b = xj & 1;
      const uint32_t par = (uint32_t)(xj >> 1) & 1u;
      ++xj;
      xval[(b * 2 + half) * kTcRows + r] = mine;
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar(quarter, b));
      if (!mbar_wait_warp(xbar(quarter, b), par, p.err)) return false;
      theirs = xval[(b * 2 + (half ^ 1)) * kTcRows + r];
      return true;
    };
    while (ok && !aborted()) {
      int u = n_units;
      PrefillDesc e{};
      ok = mbar_wait_warp(unit_full(ui & 1), (ui >> 1) & 1, p.err);
      if (ok) {
        u = unit_ring[ui & 1];
        e = unit_desc[ui & 1];
        __syncwarp();
        if (lane == 0) mbar_arrive(unit_empty(ui & 1));
      }
      ++ui;
      if (!ok || u >= n_units) break;
      const int hk = u - (u / Hkv) * Hkv;
      const int ob = uc & 1;  // this unit's O buffer
      const uint32_t tOu = tO + ob * 128;
      if constexpr (KV8) {
        // the MMAs take f16 operands: Q (bf16, as its copy left it) to f16 in
        // place, 16 bytes per step, before the unit's first Q K^T
        const int qb = uc & 1;
        if (!mbar_wait_warp(q_full(qb), (uc >> 1) & 1, p.err)) { ok = false; break; }
        const int tid = static_cast<int>(threadIdx.x) - 32 * kSoftmaxWarp0;
#pragma unroll 2
        for (int i = tid; i < Geo::kQBytes / 16; i += 32 * 8) {
          uint4 w;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                       : "r"(q_buf(qb) + 16 * i));
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(q_buf(qb) + 16 * i), "r"(bf16x2_to_f16x2(w.x)),
                       "r"(bf16x2_to_f16x2(w.y)), "r"(bf16x2_to_f16x2(w.z)), "r"(bf16x2_to_f16x2(w.w))
                       : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_conv(qb));
      }
      ++uc;
      int kt0, n_kt;
      unit_tiles(e, kt0, n_kt);
      const int tok = r / G, hj = r - tok * G;
      const int i = e.r0 + tok;                          // query index in the sequence
      const bool valid = tok < tq && i < e.r1;
      const int pos = e.n - e.q_s + i;                   // absolute position: keys 0 .. pos
      float m = -INFINITY, l = 0.f;                      // reference max (base 2), this half's sum
      for (int t = 0; t < n_kt; ++t) {
        const int gg = g + t, sb = gg & 1;
        const uint32_t ts = tmem + sb * kTcKeys + lane_off;  // this row of S, then of P
        if (!mbar_wait_warp(s_full(sb), (gg >> 1) & 1, p.err)) { ok = false; break; }
        tc_fence_after();
        float x[kHalfKeys];  // this half row of S; x * xs is the base-2 logit
        {
          uint32_t u0[32], u1[32];
          tmem_ld32(ts + kHalfKeys * half, u0);
          tmem_ld32(ts + kHalfKeys * half + 32, u1);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            x[j] = __uint_as_float(u0[j]);
            x[32 + j] = __uint_as_float(u1[j]);
          }
        }
        // with a positive scale the max is taken on the raw scores and the
        // scale folds into the exponent's FMA; a soft cap (or another scale)
        // turns the row into logits first
        const bool raw_max = p.soft_cap <= 0.f && p.qk_scale_log2 > 0.f;
        const float xs = raw_max ? p.qk_scale_log2 : 1.f;
        if (!raw_max) {
          if (p.soft_cap > 0.f) {  // soft cap: cap * tanh(s / cap), in base 2
#pragma unroll
            for (int c = 0; c < kHalfKeys; ++c) x[c] = p.cap_post * tanhf(x[c] * p.cap_pre);
          } else {
#pragma unroll
            for (int c = 0; c < kHalfKeys; ++c) x[c] *= p.qk_scale_log2;
          }
        }
        {  // columns lo_c .. lim of this half are visible (lo_c <= 0 without
           // a window); a half tile inside every row's visible range needs no mask
          const int kbase = (kt0 + t) * kTcKeys + kHalfKeys * half;
          const int lim = valid ? pos - kbase : -1;
          const int lo_c = p.window_left >= 0 ? pos - p.window_left - kbase : INT32_MIN;
          if (__any_sync(0xffffffffu, lim < kHalfKeys - 1 || lo_c > 0)) {
#pragma unroll
            for (int c = 0; c < kHalfKeys; ++c) x[c] = c <= lim && c >= lo_c ? x[c] : -INFINITY;
          }
        }
        float mx;
        {  // tree reduction over this half, then the partner's half
          float t8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) t8[j] = x[j];
          static_assert(kHalfKeys == 64, "the reduction below covers 64 keys");
#pragma unroll
          for (int c = 8; c < 56; c += 16)  // keys 8 .. 55, two per step
#pragma unroll
            for (int j = 0; j < 8; ++j) t8[j] = fmax3(t8[j], x[c + j], x[c + 8 + j]);
#pragma unroll
          for (int j = 0; j < 8; ++j) t8[j] = fmaxf(t8[j], x[56 + j]);  // keys 56 .. 63
          mx = fmax3(fmax3(t8[0], t8[1], t8[2]), fmax3(t8[3], t8[4], t8[5]), fmaxf(t8[6], t8[7]));
          float other;
          if (!trade(mx, other)) { ok = false; break; }
          mx = fmaxf(mx, other) * xs;
        }
        // move the reference max only when this tile exceeds it by more than
        // tau (both partners see the same mx, m and so decide alike)
        const bool need = mx > m + kTcTau;
        if (__any_sync(0xffffffffu, need)) {
          const float mn = need ? mx : m;
          const float alpha = mn == -INFINITY ? 1.f : ex2_approx(m - mn);
          if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            // O holds every P V of the unit so far: wait for the last, rescale
            // this thread's half of the row
            const int pg = gg - 1;
            if (!mbar_wait_warp(o_done(pg & 1), (pg >> 1) & 1, p.err)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c = kHalfD * half; c < kHalfD * (half + 1); c += 32) {
              uint32_t v[32];
              tmem_ld32(tOu + lane_off + c, v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
              tmem_st32(tOu + lane_off + c, v);
            }
            tmem_wait_st();
          }
          l *= alpha;
          m = mn;
        }
        // P = 2^(x - m) over the S columns the tile came from: hi parts of
        // keys 2c, 2c + 1 in column c, lo parts 64 columns further.  The P V
        // of tile gg - 2 that read this buffer finished before its Q K^T ran.
        const float ms = m == -INFINITY ? 0.f : m;
        {
          // keys 2w, 2w + 1 as one packed pair: exponent argument, row sum
          // and the lo residual each take one f32x2 instruction per pair.
          // hi keeps the upper 16 bits of each p (bf16 by truncation), lo the
          // upper 16 bits of the exact remainder p - hi: hi + lo carries about
          // 16 significant bits.  Key 2w in the low halves.
          const unsigned long long xs2 = pk2(xs, xs), nms2 = pk2(-ms, -ms);
          unsigned long long s2[2] = {pk2(0.f, 0.f), pk2(0.f, 0.f)};  // partial sums, kept apart for latency
          uint32_t hi[32], lo[32];
#pragma unroll
          for (int w = 0; w < 32; ++w) {
            float a0, a1;
            up2(fma2(pk2(x[2 * w], x[2 * w + 1]), xs2, nms2), a0, a1);
            const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
            const unsigned long long pp = pk2(p0, p1);
            s2[w & 1] = add2(s2[w & 1], pp);
            if constexpr (KV8) {
              hi[w] = pack_f16(p0, p1);  // f16 P (the e4m3 path's V is f16): nearest even
            } else {
              const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
              hi[w] = __byte_perm(u0, u1, 0x7632);
              float r0, r1;  // p - hi exactly: the truncated-away low bits
              up2(sub2(pp, pk2(__uint_as_float(u0 & 0xFFFF0000u), __uint_as_float(u1 & 0xFFFF0000u))), r0, r1);
              lo[w] = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
            }
          }
          tmem_st32(ts + 32 * half, hi);
          if (!KV8) tmem_st32(ts + kHalfKeys + 32 * half, lo);
          float t0, t1, t2, t3;
          up2(s2[0], t0, t1);
          up2(s2[1], t2, t3);
          l += (t0 + t1) + (t2 + t3);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(sb));
        if (t == 0 && pend && !epilogue()) { ok = false; break; }  // the previous unit's
      }
      if (!ok) break;
      // the row's sum: the partners add their halves; the epilogue (O / l)
      // follows the next unit's first tile, so that its TMEM loads and
      // global stores overlap that tile's MMAs
      float l_other;
      if (!trade(l, l_other)) { ok = false; break; }
      const float lt = l + l_other;
      pend = true;
      pend_lg = g + n_kt - 1;
      pend_ob = ob;
      pend_valid = valid;
      pend_inv = valid && lt > 0.f ? p.v_scale / lt : 0.f;
      pend_dst = static_cast<OutT*>(p.out) + (int64_t)(e.t0 + i) * p.o_st + (int64_t)(hk * G + hj) * p.o_sh;
      g += n_kt;
    }
    if (ok && pend && !epilogue()) ok = false;  // the last unit's
    if (!ok) *abort_flag = 1;
  }
}

template <int D, typename OutT, bool KV8>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using Geo = TcGeom<D>;
  unsigned char* smem = tc_smem<D>();
  prefill_tc_setup<D>(tm_q, tm_k, tm_v);
  // launched with programmatic dependent launch: wait for the previous
  // kernel (every thread, before any global access), then let the decode
  // kernel that follows launch and set up on the SMs this grid frees
  grid_dep_wait();
  launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  TcStart* start = reinterpret_cast<TcStart*>(smem + Geo::kOffBar + kOffStart);
  if (warp == 0) {
    // one load per lane: the plan's signature (lanes 0 .. kPlanSig - 1) and
    // its prefill CTA count (16); every CTA of every run reads these, so
    // they are usually in L2
    int32_t sig[kPlanSig];
    plan_signature(p, sig);
    int32_t want = 0;
#pragma unroll
    for (int i = 0; i < kPlanSig; ++i) want = lane == i ? sig[i] : want;
    int32_t v = 0;
    if (lane < kPlanSig) {
      v = __ldcg(p.ws.sig + lane);
    } else if (lane == 16) {
      v = __ldcg(p.ws.pf_ctas);
    }
    const bool ok = __all_sync(0xffffffffu, lane >= kPlanSig || v == want);
    const int n_ctas = __shfl_sync(0xffffffffu, v, 16);
    if (lane == 0) {
      start->ok = ok;
      // the plan gives the prefill part of the SMs (the decode kernel takes
      // the rest): the CTAs past that many leave at once
      start->active = min(static_cast<int>(gridDim.x), n_ctas);
    }
  }
  __syncthreads();
  const int ok = start->ok, active = start->active;
  if (!ok) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrPlan);
    return;
  }
  // the CTAs past the prefill's share leave at once (their SMs go to the
  // decode kernel); the others allocate TMEM and take the units (first
  // unit = CTA index, then claims)
  if (static_cast<int>(blockIdx.x) >= active) return;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Geo::kOffBar + 8 * kSlotTmem);
  // the unit count and the first unit's descriptor (unit = CTA index; the
  // tile list has room for every CTA of the grid, whatever the plan holds)
  // come in while TMEM is allocated
  int first_word = 0, n_units = 0;
  if (warp == 0) {
    if (lane < 8) first_word = __ldcg(reinterpret_cast<const int32_t*>(p.ws.pf_desc + blockIdx.x / p.Hkv) + lane);
    if (lane == 8) n_units = __ldcg(p.ws.pf_off + p.B) * p.Hkv;
    n_units = __shfl_sync(0xffffffffu, n_units, 8);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(Geo::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (warp == 0 && lane == 0) start->n_units = n_units;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  n_units = start->n_units;
  prefill_tc_body<D, OutT, KV8>(p, tm_q, tm_k, tm_v, active, n_units, first_word);
  // ---- teardown: every MMA of this CTA has completed (its results were
  // waited for, or the MMA warp drained them), then free TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*tslot), "r"(Geo::kTmemCols));
  }
}

// ---- host: tensor maps
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
  });
  return fn;
}

// 3-D bf16 map {d, heads, rows} with a {64, box_h, box_r} box, 128-byte swizzle
bool encode_3d(CUtensorMap* m, const void* base, uint64_t d, uint64_t heads, uint64_t rows, uint64_t head_stride_b,
               uint64_t row_stride_b, uint32_t box_h, uint32_t box_r) {
  EncodeTiled fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {d, heads, rows};
  const cuuint64_t strides[2] = {head_stride_b, row_stride_b};
  const cuuint32_t box[3] = {64, box_h, box_r};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map of e4m3 codes {d, heads, rows} with a {D, 1, box_r} box (whole
// rows of one head), no swizzle: the kernel converts them into the swizzled
// f16 layout itself
bool encode_3d_codes(CUtensorMap* m, const void* base, uint64_t d, uint64_t heads, uint64_t rows,
                     uint64_t head_stride_b, uint64_t row_stride_b, uint32_t box_r) {
  EncodeTiled fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {d, heads, rows};
  const cuuint64_t strides[2] = {head_stride_b, row_stride_b};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 1, box_r};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, typename OutT, bool KV8>
cudaError_t launch_tc(const AttnParams& p, int64_t max_units, int num_sms, cudaStream_t st) {
  using Geo = TcGeom<D>;
  CUtensorMap mq, mk, mv;
  const uint64_t n_slots = (uint64_t)p.num_blocks * (uint64_t)p.bs;
  const uint32_t bx = p.bs % 16 == 0 ? 16 : 8;  // keys per box: a box stays inside one block
  if (!encode_3d(&mq, p.q, D, p.Hq, p.T, (uint64_t)p.q_sh * 2, (uint64_t)p.q_st * 2, p.G, p.pf_tq))
    return cudaErrorInvalidValue;
  const bool kv_ok =
      KV8 ? encode_3d_codes(&mk, p.k_cache, D, p.Hkv, n_slots, (uint64_t)D, (uint64_t)p.Hkv * D, bx) &&
                encode_3d_codes(&mv, p.v_cache, D, p.Hkv, n_slots, (uint64_t)D, (uint64_t)p.Hkv * D, bx)
          : encode_3d(&mk, p.k_cache, D, p.Hkv, n_slots, (uint64_t)D * 2, (uint64_t)p.Hkv * D * 2, 1, bx) &&
                encode_3d(&mv, p.v_cache, D, p.Hkv, n_slots, (uint64_t)D * 2, (uint64_t)p.Hkv * D * 2, 1, bx);
  if (!kv_ok) return cudaErrorInvalidValue;
  auto kern = prefill_tc_kernel<D, OutT, KV8>;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern), Geo::kSmem);
  if (e != cudaSuccess) return e;
  int64_t grid = num_sms;
  if (grid > max_units) grid = max_units;
  if (grid < 1) return cudaSuccess;
  return launch_ex(kern, dim3((unsigned)grid), dim3(kTcThreads), Geo::kSmem, st, true, p, mq, mk, mv);
}

}  // namespace

bool prefill_tc_supported(int kv, int64_t D, int64_t bs, int64_t G) {
  return (kv == 1 || kv == 2) && (D == 64 || D == 128) && bs % 8 == 0 && G >= 1 && G <= kTcRows;
}

int prefill_tc_tokens_per_tile(int64_t G) { return (int)(kTcRows / G); }

cudaError_t launch_prefill_tc(const AttnParams& p, int out_kind, int64_t max_units, int num_sms, cudaStream_t st) {
#define PKV_TC(D, KV8)                                                          \
  (out_kind ? launch_tc<D, __nv_bfloat16, KV8>(p, max_units, num_sms, st) \
            : launch_tc<D, float, KV8>(p, max_units, num_sms, st))
  if (p.kv_esize == 1) return p.D == 128 ? PKV_TC(128, true) : PKV_TC(64, true);
  return p.D == 128 ? PKV_TC(128, false) : PKV_TC(64, false);
#undef PKV_TC
}

}  // namespace pkv
