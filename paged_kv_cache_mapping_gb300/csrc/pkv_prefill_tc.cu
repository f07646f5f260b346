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
// with an online softmax (base 2) between them, one thread per query row.
//
// CTA (one per SM, persistent over tiles), 6 warps:
//   warp 0   TMA producer: the Q tile of a work unit, then K and V tiles of
//            128 keys (8 boxes of 16 consecutive slots of one head per d
//            half) into 2-stage rings.  Keys past the sequence and bad block
//            ids read out of bounds, which TMA fills with zeros.
//   warp 1   MMA issuer (one thread) and owner of the TMEM allocation
//            (S: columns 0-127, O: columns 128-127+D).
//   warps 2-5  softmax: each thread loads its row of S from TMEM, masks,
//            updates the running max and sum, writes its row of P (hi and lo
//            bf16 parts) into shared memory, rescales its row of O in TMEM
//            when the max grows, and at the end writes O / l.
// Block sizes must be multiples of 16 (a box of 16 keys lies in one block).
#include <cuda.h>

#include <mutex>

#include "pkv_kernels.h"

namespace pkv {
namespace {

constexpr int kTcRows = 128;  // query rows per tile (MMA M)
constexpr int kTcKeys = 128;  // keys per key tile
constexpr int kTcThreads = 192;

template <int D>
struct TcGeom {
  static constexpr int kHalves = D / 64;                     // 128-byte atoms along d
  static constexpr int kQBytes = kHalves * kTcRows * 128;
  static constexpr int kKVBytes = kHalves * kTcKeys * 128;   // one K or V tile
  static constexpr int kPBytes = (kTcKeys / 64) * kTcRows * 128;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;              // 2 stages
  static constexpr int kOffV = kOffK + 2 * kKVBytes;         // 2 stages
  static constexpr int kOffP = kOffV + 2 * kKVBytes;         // hi, then lo
  static constexpr int kOffBar = kOffP + 2 * kPBytes;
  static constexpr int kSmem = kOffBar + 256 + 1024;          // barriers, 1024-byte alignment slack
  static constexpr uint32_t kTmemCols = 256;                  // S 128 + O D, rounded to a power of 2
};

// ---- tcgen05 / TMA wrappers
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  // shared-memory matrix descriptor: start >> 4, leading and stride byte
  // offsets >> 4, descriptor version 1, 128-byte swizzle
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B,
// K-major A, B K-major (b_mn = 0) or MN-major (b_mn = 1), M = 128, N = n
__host__ __device__ constexpr uint32_t umma_idesc(int n, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(kTcRows >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
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

// byte offset of element (row r, column c) in a K-major, 128-byte-swizzled
// tile of `rows` rows of 16-bit elements (64 columns per atom)
__device__ __forceinline__ uint32_t sw128_off(int r, int c, int rows) {
  return (uint32_t)((c >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) +
                    ((c & 7) << 1));
}

// Work unit u: prefill tile u / Hkv (tokens r0 .. r1-1 of its sequence,
// the last tokens first), KV head u % Hkv.
template <int D, typename OutT>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using Geo = TcGeom<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const uint32_t sQ = smem_u32(smem + Geo::kOffQ);
  const uint32_t sK = smem_u32(smem + Geo::kOffK);
  const uint32_t sV = smem_u32(smem + Geo::kOffV);
  const uint32_t sP = smem_u32(smem + Geo::kOffP);
  unsigned char* pbase = smem + Geo::kOffP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Geo::kOffBar);
  const uint32_t b0 = smem_u32(bars);
  const uint32_t q_full = b0, q_empty = b0 + 8;
  const uint32_t k_full = b0 + 16, k_empty = b0 + 32, v_full = b0 + 48, v_empty = b0 + 64;  // [2] each
  const uint32_t s_full = b0 + 80, s_empty = b0 + 88, p_full = b0 + 96, o_done = b0 + 104, o_free = b0 + 112;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 15);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 16);
  const uint32_t drain = b0 + 136;  // the MMA warp's last commit when the CTA gives up
  // the abort flag as one value for the whole warp (another warp may set it
  // between two lanes' reads)
  auto aborted = [&]() -> bool { return __any_sync(0xffffffffu, *abort_flag != 0); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(k_full + 8 * i, 1);
      mbar_init(k_empty + 8 * i, 1);
      mbar_init(v_full + 8 * i, 1);
      mbar_init(v_empty + 8 * i, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 4);
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(o_free, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(Geo::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tS = tmem, tO = tmem + 128;

  const int G = p.G, Hkv = p.Hkv;
  const int tq = p.pf_tq;  // query tokens per tile
  const int n_units = p.ws.pf_off[p.B] * Hkv;
  const uint32_t q_box_bytes = (uint32_t)(Geo::kHalves * G * tq * 128);

  if (warp == 0) {
    // ======================= TMA producer =======================
    const int64_t n_slots = p.num_blocks * p.bs;
    int kv_it = 0, q_it = 0;
    for (int u = blockIdx.x; u < n_units && !aborted(); u += gridDim.x, ++q_it) {
      const PrefillDesc e = p.ws.pf_desc[u / Hkv];
      const int g = u - (u / Hkv) * Hkv;
      if (!mbar_wait_warp(q_empty, (q_it & 1) ^ 1, p.err)) { *abort_flag = 1; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, q_box_bytes);
        for (int h = 0; h < Geo::kHalves; ++h)
          tma_load_3d(sQ + h * kTcRows * 128, &tm_q, h * 64, g * G, e.t0 + e.r0, q_full);
      }
      const int32_t* bt_row = p.bt + (int64_t)e.s * p.bt_stride;
      const int n_kt = (e.kv_end + kTcKeys - 1) / kTcKeys;
      bool failed = false;
      for (int kt = 0; kt < n_kt; ++kt, ++kv_it) {
        const int st = kv_it & 1, ph = (kv_it >> 1) & 1;
        // lane l: key block l % 8 of the tile (16 keys), d half l / 8
        const int bi = lane & 7, h = (lane >> 3) & 1;
        const int key0 = kt * kTcKeys + 16 * bi;
        int slot = (int)n_slots;  // out of bounds: zero fill
        if (key0 < e.n) {
          const int lb = p.bs_shift >= 0 ? (key0 >> p.bs_shift) : (key0 / p.bs);
          const int32_t blk = __ldg(bt_row + lb);
          if ((uint32_t)blk < (uint32_t)p.num_blocks)
            slot = blk * p.bs + (key0 - lb * p.bs);
          else
            atomicOr(p.err, kErrBlockRange);
        }
        const bool issuer = lane < 8 * Geo::kHalves;
        if (!mbar_wait_warp(k_empty + 8 * st, ph ^ 1, p.err)) { failed = true; break; }
        if (lane == 0) mbar_arrive_expect_tx(k_full + 8 * st, Geo::kKVBytes);
        __syncwarp();
        if (issuer)
          tma_load_3d(sK + st * Geo::kKVBytes + h * kTcKeys * 128 + bi * 2048, &tm_k, h * 64, g, slot,
                      k_full + 8 * st);
        if (!mbar_wait_warp(v_empty + 8 * st, ph ^ 1, p.err)) { failed = true; break; }
        if (lane == 0) mbar_arrive_expect_tx(v_full + 8 * st, Geo::kKVBytes);
        __syncwarp();
        if (issuer)
          tma_load_3d(sV + st * Geo::kKVBytes + h * kTcKeys * 128 + bi * 2048, &tm_v, h * 64, g, slot,
                      v_full + 8 * st);
      }
      if (failed) { *abort_flag = 1; break; }
    }
    if (aborted() && kv_it > 0) {
      // giving up: let the copies this warp issued land before the CTA exits
      for (int k = kv_it - 1; k >= 0 && k >= kv_it - 2; --k) {
        mbar_wait_warp(k_full + 8 * (k & 1), (k >> 1) & 1, p.err);
        mbar_wait_warp(v_full + 8 * (k & 1), (k >> 1) & 1, p.err);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    constexpr uint32_t kIdQK = umma_idesc(kTcKeys, 0);
    constexpr uint32_t kIdPV = umma_idesc(D, 1);
    int kv_it = 0, q_it = 0, s_it = 0, p_it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok && !aborted(); u += gridDim.x, ++q_it) {
      const PrefillDesc e = p.ws.pf_desc[u / Hkv];
      const int n_kt = (e.kv_end + kTcKeys - 1) / kTcKeys;
      ok = mbar_wait_warp(q_full, q_it & 1, p.err);
      // S = Q K^T for key tile kt (K stage of kv_it + kt)
      auto issue_qk = [&](int kt) -> bool {
        const int it = kv_it + kt, st = it & 1, ph = (it >> 1) & 1;
        if (!mbar_wait_warp(k_full + 8 * st, ph, p.err)) return false;
        if (!mbar_wait_warp(s_empty, (s_it & 1) ^ 1, p.err)) return false;
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kb = 0; kb < D / 16; ++kb) {
            const uint32_t ko = (kb >> 2) * kTcRows * 128 + (kb & 3) * 32;
            const uint32_t kk = (kb >> 2) * kTcKeys * 128 + (kb & 3) * 32;
            umma_bf16(tS, umma_desc(sQ + ko, 16, 1024), umma_desc(sK + st * Geo::kKVBytes + kk, 16, 1024), kIdQK,
                      kb > 0);
          }
          umma_commit(s_full);
          umma_commit(k_empty + 8 * st);
        }
        __syncwarp();
        ++s_it;
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int kt = 0; kt < n_kt && ok; ++kt) {
        if (kt + 1 < n_kt) ok = issue_qk(kt + 1);
        if (kt + 1 == n_kt && ok && lane == 0) umma_commit(q_empty);  // Q no longer read
        if (!ok) break;
        const int it = kv_it + kt, st = it & 1, ph = (it >> 1) & 1;
        ok = mbar_wait_warp(p_full, p_it & 1, p.err) && mbar_wait_warp(v_full + 8 * st, ph, p.err) &&
             (kt > 0 || mbar_wait_warp(o_free, (q_it & 1) ^ 1, p.err));
        if (!ok) break;
        ++p_it;
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < kTcKeys / 16; ++kk) {
            const uint32_t pa = (kk >> 2) * kTcRows * 128 + (kk & 3) * 32;
            const uint64_t vd = umma_desc(sV + st * Geo::kKVBytes + kk * 2048, kTcKeys * 128, 1024);
            umma_bf16(tO, umma_desc(sP + pa, 16, 1024), vd, kIdPV, kt > 0 || kk > 0);
            umma_bf16(tO, umma_desc(sP + Geo::kPBytes + pa, 16, 1024), vd, kIdPV, 1);
          }
          umma_commit(o_done);
          umma_commit(v_empty + 8 * st);
        }
        __syncwarp();
      }
      kv_it += n_kt;
    }
    if (!ok || aborted()) {
      // giving up: every MMA issued so far must finish before TMEM is freed
      *abort_flag = 1;
      if (lane == 0) umma_commit(drain);
      __syncwarp();
      mbar_wait_warp(drain, 0, p.err);
    }
  } else {
    // ======================= softmax / epilogue (warps 2-5) =======================
    const int quarter = warp & 3;             // TMEM lanes 32 * quarter ..
    const int r = 32 * quarter + lane;        // this thread's query row
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    int s_it = 0, o_it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok && !aborted(); u += gridDim.x) {
      const PrefillDesc e = p.ws.pf_desc[u / Hkv];
      const int g = u - (u / Hkv) * Hkv;
      const int n_kt = (e.kv_end + kTcKeys - 1) / kTcKeys;
      const int tok = r / G, hj = r - tok * G;
      const int i = e.r0 + tok;                          // query index in the sequence
      const bool valid = tok < tq && i < e.r1;
      const int pos = e.n - e.q_s + i;                   // absolute position: keys 0 .. pos
      float m = -INFINITY, l = 0.f;
      for (int kt = 0; kt < n_kt; ++kt) {
        if (!mbar_wait_warp(s_full, s_it & 1, p.err)) { ok = false; break; }
        ++s_it;
        tc_fence_after();
        float x[kTcKeys];
#pragma unroll
        for (int c = 0; c < kTcKeys; c += 32) {
          uint32_t v[32];
          tmem_ld32(tS + lane_off + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) x[c + j] = __uint_as_float(v[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty);
        // mask and running max (base 2)
        const int lim = valid ? pos - kt * kTcKeys : -1;  // columns 0 .. lim are visible
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTcKeys; ++c) {
          x[c] = c <= lim ? x[c] * p.qk_scale_log2 : -INFINITY;
          mx = fmaxf(mx, x[c]);
        }
        const float mn = fmaxf(m, mx);
        const float ms = mn == -INFINITY ? 0.f : mn;
        const float alpha = exp2f(m - ms);
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < kTcKeys; ++c) {
          x[c] = exp2f(x[c] - ms);
          sum += x[c];
        }
        l = l * alpha + sum;
        m = mn;
        // the previous tile's P V must be done before P and O are touched
        if (kt > 0) {
          if (!mbar_wait_warp(o_done, o_it & 1, p.err)) { ok = false; break; }
          ++o_it;
          tc_fence_after();
        }
        // P row: hi = bf16(p), lo = bf16(p - hi), 16-byte chunks in swizzled order
#pragma unroll
        for (int c = 0; c < kTcKeys; c += 8) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) split_bf16(x[c + 2 * j], x[c + 2 * j + 1], hi[j], lo[j]);
          const uint32_t off = sw128_off(r, c, kTcRows);
          *reinterpret_cast<uint4*>(pbase + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(pbase + Geo::kPBytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        // rescale the rows of O whose max grew; the TMEM loads and stores are
        // warp-collective, so the whole warp takes the branch together
        if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t v[32];
            tmem_ld32(tO + lane_off + c, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            tmem_st32(tO + lane_off + c, v);
          }
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (!ok) break;
      // epilogue: O / l for valid rows
      if (!mbar_wait_warp(o_done, o_it & 1, p.err)) { ok = false; break; }
      ++o_it;
      tc_fence_after();
      const float inv = valid && l > 0.f ? p.v_scale / l : 0.f;
      OutT* dst = static_cast<OutT*>(p.out) + (int64_t)(e.t0 + i) * p.o_st + (int64_t)(g * G + hj) * p.o_sh;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t v[32];
        tmem_ld32(tO + lane_off + c, v);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) store2(dst + c + j, __uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
    }
    if (!ok) *abort_flag = 1;
  }
  // ---- teardown: every MMA this CTA issued has completed (the MMA warp's
  // last commits were waited on above, or the CTA gave up), then free TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Geo::kTmemCols));
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

template <int D, typename OutT>
cudaError_t launch_tc(const AttnParams& p, int64_t max_units, int num_sms, cudaStream_t st) {
  using Geo = TcGeom<D>;
  CUtensorMap mq, mk, mv;
  const uint64_t n_slots = (uint64_t)p.num_blocks * (uint64_t)p.bs;
  if (!encode_3d(&mq, p.q, D, p.Hq, p.T, (uint64_t)p.q_sh * 2, (uint64_t)p.q_st * 2, p.G, p.pf_tq) ||
      !encode_3d(&mk, p.k_cache, D, p.Hkv, n_slots, (uint64_t)D * 2, (uint64_t)p.Hkv * D * 2, 1, 16) ||
      !encode_3d(&mv, p.v_cache, D, p.Hkv, n_slots, (uint64_t)D * 2, (uint64_t)p.Hkv * D * 2, 1, 16))
    return cudaErrorInvalidValue;
  auto kern = prefill_tc_kernel<D, OutT>;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern), Geo::kSmem);
  if (e != cudaSuccess) return e;
  int64_t grid = num_sms;
  if (grid > max_units) grid = max_units;
  if (grid < 1) return cudaSuccess;
  kern<<<(unsigned)grid, kTcThreads, Geo::kSmem, st>>>(p, mq, mk, mv);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(int kv, int64_t D, int64_t bs, int64_t G) {
  return kv == 1 && (D == 64 || D == 128) && bs % 16 == 0 && G >= 1 && G <= kTcRows;
}

int prefill_tc_tokens_per_tile(int64_t G) { return (int)(kTcRows / G); }

cudaError_t launch_prefill_tc(const AttnParams& p, int out_kind, int64_t max_units, int num_sms, cudaStream_t st) {
  if (p.D == 128)
    return out_kind ? launch_tc<128, __nv_bfloat16>(p, max_units, num_sms, st)
                    : launch_tc<128, float>(p, max_units, num_sms, st);
  return out_kind ? launch_tc<64, __nv_bfloat16>(p, max_units, num_sms, st)
                  : launch_tc<64, float>(p, max_units, num_sms, st);
}

}  // namespace pkv
