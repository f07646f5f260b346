// pkv_prefill.cu -- causal attention of multi-token query chunks (chunked
// prefill) over paged K/V, on the tensor cores.
//
// What it computes: query row i of a sequence with q_s new tokens and N_s
// keys sits at position p = N_s - q_s + i and attends to keys 0..p: the
// cached prefix plus the chunk's own earlier tokens (nanoserve, "Chunked
// prefill" bullet and "Architecture" step 3; "How to design an LLM serving
// system (a vLLM deep dive)", "Latency and scaling knobs": chunked prefill).
// Prefill is compute-bound ("How to design an LLM serving system", "Two
// phases and the KV cache"), so both products are dense MMAs.
//
// Design: persistent CTAs; a work item is (sequence, tile of 64 query rows,
// KV head), a query row being a (token, head-of-the-group) pair, so one K/V
// stage serves the whole GQA group.  The same producer warp and staging ring
// as the decode kernel stream the keys 0 .. max position of the tile; four
// consumer warps own 16 rows each and run S = Q K^T and O += P V as
// mma.sync m16n8k16 with an online softmax per row (the query rows are the M
// dimension).  P enters PV as a bf16 hi + lo pair; with an e4m3 cache, K and
// V are converted exactly to f16 and P is f16.
#include "pkv_pipeline.cuh"

namespace pkv {

template <int KV, int D>
struct PrefillCfg {
  static constexpr int kEsz = KV == 2 ? 1 : 2;
  static constexpr int kRowB = D * kEsz;
  static constexpr int kRowS = kRowB + 16;
  static constexpr int kNW = 4;
  static constexpr int kST = 64;             // keys per stage
  static constexpr int kNS = KV == 2 ? 4 : 3;
  static constexpr int kStageB = 2 * kST * kRowS;
  static constexpr int kKS = D / 16;         // k-steps over d
  static constexpr int kND = D / 8;          // 8-wide output tiles over d
  static constexpr int kThreads = (kNW + 1) * 32;
  static constexpr size_t kSmem = (size_t)kNS * kStageB + 2 * kNS * 8 + 64;
  static_assert(kPrefillRows == 16 * kNW, "a tile is 16 rows per consumer warp");
};

struct PrefillItem {
  int s, g, q_s, n, r0, r1;  // rows r0 .. r1-1 of q_s * G
  int kv_end;                // keys 0 .. kv_end-1 are visible to some row
  int64_t t0;                // packed index of the sequence's first query token
};

__device__ __forceinline__ bool prefill_item(const AttnParams& p, int n_items, int w, PrefillItem& it) {
  if (w >= n_items) return false;
  const PrefillDesc e = p.ws.pf_desc[w / p.Hkv];
  it.g = w % p.Hkv;
  it.s = e.s;
  it.t0 = e.t0;
  it.q_s = e.q_s;
  it.n = e.n;
  it.r0 = e.r0;
  it.r1 = e.r1;
  it.kv_end = e.kv_end;
  return true;
}

template <int KV, int D, typename OutT>
__global__ void __launch_bounds__(PrefillCfg<KV, D>::kThreads, 2) prefill_kernel(AttnParams p) {
  using C = PrefillCfg<KV, D>;
  using R = Ring<C::kRowB, C::kRowS, C::kST, C::kNS>;
  if (!plan_matches_warp(p)) {  // the same answer in every thread
    if (threadIdx.x == 0) atomicOr(p.err, kErrPlan);
    return;
  }
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)C::kNS * C::kStageB);
  volatile int* flags = reinterpret_cast<volatile int*>(bars + 2 * C::kNS);  // [0] abort
  R ring;
  ring.base = smem;
  ring.base_s = smem_u32(smem);
  ring.full0 = smem_u32(bars);
  ring.empty0 = smem_u32(bars + C::kNS);
  if (threadIdx.x == 0) flags[0] = 0;
  init_ring_barriers<C::kNS>(ring.full0, ring.empty0, C::kNW);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = __ldg(p.ws.pf_off + p.B) * p.Hkv;
  if (warp == C::kNW) {
    // ======================= producer warp =======================
    const char* kbase = static_cast<const char*>(p.k_cache);
    const char* vbase = static_cast<const char*>(p.v_cache);
    int fill = 0;
    PrefillItem it;
    for (int w = blockIdx.x; prefill_item(p, n_items, w, it); w += gridDim.x) {
      const int32_t* bt_row = p.bt + (int64_t)it.s * p.bt_stride;
      for (int j0 = 0; j0 < it.kv_end; j0 += C::kST) {
        if (flags[0]) break;
        if (!ring.produce(p, fill, bt_row, it.g, j0, min(C::kST, it.kv_end - j0), kbase, vbase, lane)) {
          flags[0] = 1;
          break;
        }
        ++fill;
      }
      if (flags[0]) break;
    }
    ring.drain(p, fill);
    return;
  }

  // ======================= consumer warps =======================
  const int g4 = lane >> 2, t4 = lane & 3;
  int cons = 0;
  PrefillItem it;
  for (int w = blockIdx.x; prefill_item(p, n_items, w, it); w += gridDim.x) {
    // rows of this thread: A = 16*warp + g4, B = A + 8 (tile-relative)
    const int rA = it.r0 + 16 * warp + g4, rB = rA + 8;
    const bool vA = rA < it.r1, vB = rB < it.r1;
    const int iA = vA ? rA / p.G : 0, iB = vB ? rB / p.G : 0;
    const int hA = it.g * p.G + (vA ? rA - iA * p.G : 0), hB = it.g * p.G + (vB ? rB - iB * p.G : 0);
    const int posA = vA ? it.n - it.q_s + iA : -1, posB = vB ? it.n - it.q_s + iB : -1;
    const int64_t tA = it.t0 + iA, tB = it.t0 + iB;
    // ---- Q fragments (A operand: rows = query rows, k = d)
    uint32_t qa[C::kKS][4];
    {
      const __nv_bfloat16* qA = static_cast<const __nv_bfloat16*>(p.q) + tA * p.q_st + (int64_t)hA * p.q_sh;
      const __nv_bfloat16* qB = static_cast<const __nv_bfloat16*>(p.q) + tB * p.q_st + (int64_t)hB * p.q_sh;
#pragma unroll
      for (int ks = 0; ks < C::kKS; ++ks) {
        if constexpr (KV == 2) {
          const uint2 a = vA ? *reinterpret_cast<const uint2*>(qA + 16 * ks + 4 * t4) : make_uint2(0, 0);
          const uint2 b = vB ? *reinterpret_cast<const uint2*>(qB + 16 * ks + 4 * t4) : make_uint2(0, 0);
          qa[ks][0] = bf16x2_to_f16x2(a.x);
          qa[ks][2] = bf16x2_to_f16x2(a.y);
          qa[ks][1] = bf16x2_to_f16x2(b.x);
          qa[ks][3] = bf16x2_to_f16x2(b.y);
        } else {
          qa[ks][0] = vA ? *reinterpret_cast<const uint32_t*>(qA + 16 * ks + 2 * t4) : 0u;
          qa[ks][2] = vA ? *reinterpret_cast<const uint32_t*>(qA + 16 * ks + 2 * t4 + 8) : 0u;
          qa[ks][1] = vB ? *reinterpret_cast<const uint32_t*>(qB + 16 * ks + 2 * t4) : 0u;
          qa[ks][3] = vB ? *reinterpret_cast<const uint32_t*>(qB + 16 * ks + 2 * t4 + 8) : 0u;
        }
      }
    }
    float acc[C::kND][4];
#pragma unroll
    for (int i = 0; i < C::kND; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    const int warp_pos_max = max(posA, posB);  // per thread; stage skip below is warp-uniform
    int wmax = warp_pos_max;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));

    for (int j0 = 0; j0 < it.kv_end; j0 += C::kST, ++cons) {
      if (!flags[0] && !ring.wait_full(p, cons)) flags[0] = 1;
      if (j0 <= wmax && !flags[0]) {
        const uint32_t sK = ring.k_rows(cons), sV = ring.v_rows(cons);
        // ---- S = Q K^T : 16 rows x 64 keys (8 tiles of 8 keys)
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        const uint32_t aK = sK + (lane & 7) * C::kRowS + (lane >> 3) * 16;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
          for (int kq = 0; kq < C::kKS / (KV == 2 ? 4 : 2); ++kq) {
            uint32_t w0, w1, w2, w3;
            ldsm_x4(aK + 8 * nt * C::kRowS + 64 * kq, w0, w1, w2, w3);
            if constexpr (KV == 2) {
              // four 16-byte chunks = four k-steps, d permuted as in Q
              const uint32_t wv[4] = {w0, w1, w2, w3};
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                uint32_t b0, b1;
                e4m3x4_to_f16(wv[c], b0, b1);
                mma_f16(s[nt], qa[4 * kq + c], b0, b1);
              }
            } else {
              mma_bf16(s[nt], qa[2 * kq], w0, w1);
              mma_bf16(s[nt], qa[2 * kq + 1], w2, w3);
            }
          }
        }
        // ---- causal mask and online softmax (base 2), per row
        float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int j = j0 + 8 * nt + 2 * t4;
          s[nt][0] = j <= posA ? s[nt][0] * p.qk_scale_log2 : -INFINITY;
          s[nt][1] = j + 1 <= posA ? s[nt][1] * p.qk_scale_log2 : -INFINITY;
          s[nt][2] = j <= posB ? s[nt][2] * p.qk_scale_log2 : -INFINITY;
          s[nt][3] = j + 1 <= posB ? s[nt][3] * p.qk_scale_log2 : -INFINITY;
          mxA = fmaxf(mxA, fmaxf(s[nt][0], s[nt][1]));
          mxB = fmaxf(mxB, fmaxf(s[nt][2], s[nt][3]));
        }
        mxA = warp_max_xor(mxA, 1); mxA = warp_max_xor(mxA, 2);
        mxB = warp_max_xor(mxB, 1); mxB = warp_max_xor(mxB, 2);
        const float mnA = fmaxf(mA, mxA), mnB = fmaxf(mB, mxB);
        const float msA = mnA == -INFINITY ? 0.f : mnA, msB = mnB == -INFINITY ? 0.f : mnB;
        const float alA = exp2f(mA - msA), alB = exp2f(mB - msB);
        mA = mnA;
        mB = mnB;
        float sumA = 0.f, sumB = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          s[nt][0] = exp2f(s[nt][0] - msA);
          s[nt][1] = exp2f(s[nt][1] - msA);
          s[nt][2] = exp2f(s[nt][2] - msB);
          s[nt][3] = exp2f(s[nt][3] - msB);
          sumA += s[nt][0] + s[nt][1];
          sumB += s[nt][2] + s[nt][3];
        }
        lA = lA * alA + sumA;
        lB = lB * alB + sumB;
#pragma unroll
        for (int i = 0; i < C::kND; ++i) {
          acc[i][0] *= alA;
          acc[i][1] *= alA;
          acc[i][2] *= alB;
          acc[i][3] *= alB;
        }
        // ---- O += P V : k = 16 keys per step
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t aV = sV + (16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8) * C::kRowS + (lane >> 4) * 16;
          if constexpr (KV == 2) {
            uint32_t a[4];
            a[0] = pack_f16(s[2 * kk][0], s[2 * kk][1]);
            a[1] = pack_f16(s[2 * kk][2], s[2 * kk][3]);
            a[2] = pack_f16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            a[3] = pack_f16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int cp = 0; cp < C::kRowB / 32; ++cp) {
              uint32_t w0, w1, w2, w3;  // (top, bottom) keys x chunks 2cp, 2cp+1
              ldsm_x4(aV + 32 * cp, w0, w1, w2, w3);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                uint32_t x0t, x1t, x0b, x1b;
                e4m3x4_to_f16(hh ? w2 : w0, x0t, x1t);
                e4m3x4_to_f16(hh ? w3 : w1, x0b, x1b);
                const int c = 2 * cp + hh;  // 16-byte chunk = 16 values of d
                mma_f16(acc[2 * c], a, movm_t(x0t), movm_t(x0b));
                mma_f16(acc[2 * c + 1], a, movm_t(x1t), movm_t(x1b));
              }
            }
          } else {
            uint32_t ah[4], al[4];
            split_bf16(s[2 * kk][0], s[2 * kk][1], ah[0], al[0]);
            split_bf16(s[2 * kk][2], s[2 * kk][3], ah[1], al[1]);
            split_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1], ah[2], al[2]);
            split_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3], ah[3], al[3]);
#pragma unroll
            for (int np = 0; np < C::kND / 2; ++np) {
              uint32_t b0, b1, b2, b3;  // d tiles 2np (b0, b1) and 2np+1 (b2, b3)
              ldsm_x4_t(aV + 32 * np, b0, b1, b2, b3);
              mma_bf16(acc[2 * np], ah, b0, b1);
              mma_bf16(acc[2 * np], al, b0, b1);
              mma_bf16(acc[2 * np + 1], ah, b2, b3);
              mma_bf16(acc[2 * np + 1], al, b2, b3);
            }
          }
        }
      }
      ring.release(cons, lane);
    }
    // ---- normalise and store
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    OutT* oA = static_cast<OutT*>(p.out) + tA * p.o_st + (int64_t)hA * p.o_sh;
    OutT* oB = static_cast<OutT*>(p.out) + tB * p.o_st + (int64_t)hB * p.o_sh;
#pragma unroll
    for (int nd = 0; nd < C::kND; ++nd) {
      int d;
      if constexpr (KV == 2)
        d = 16 * (nd >> 1) + 4 * t4 + 2 * (nd & 1);  // permuted d of the e4m3 path
      else
        d = 8 * nd + 2 * t4;
      if (vA) store2(oA + d, acc[nd][0] / lA * p.v_scale, acc[nd][1] / lA * p.v_scale);
      if (vB) store2(oB + d, acc[nd][2] / lB * p.v_scale, acc[nd][3] / lB * p.v_scale);
    }
  }
}

template <int KV, int D, typename OutT>
static cudaError_t launch_prefill_t(const AttnParams& p, int64_t max_items, int num_sms, cudaStream_t st) {
  using C = PrefillCfg<KV, D>;
  auto kern = prefill_kernel<KV, D, OutT>;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern), C::kSmem);
  if (e != cudaSuccess) return e;
  int occ = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::kThreads, C::kSmem);
  if (occ < 1) occ = 1;
  int64_t grid = (int64_t)num_sms * occ;
  if (grid > max_items) grid = max_items;
  if (grid < 1) return cudaSuccess;
  kern<<<(unsigned)grid, C::kThreads, C::kSmem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const AttnParams& p, int kv, int out_kind, int64_t max_items, int num_sms,
                           cudaStream_t st) {
#define PKV_PF(KV, D) \
  (out_kind ? launch_prefill_t<KV, D, __nv_bfloat16>(p, max_items, num_sms, st) \
            : launch_prefill_t<KV, D, float>(p, max_items, num_sms, st))
  if (kv == 1) return p.D == 128 ? PKV_PF(1, 128) : PKV_PF(1, 64);
  return p.D == 128 ? PKV_PF(2, 128) : PKV_PF(2, 64);
#undef PKV_PF
}

}  // namespace pkv
