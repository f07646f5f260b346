// pkv_decode.cu -- paged decode attention (one query token per sequence),
// split-KV chunks and their log-sum-exp merge, plus the device-side plan.
//
// What it computes: for a decoding sequence s (q_s = 1, N_s keys) and query
// head h, o = sum_j softmax_j(scale * q.k_j) v_j over j < N_s, K/V read
// straight from the pages named by the block table (nanoserve, "Triton
// paged-attention decode kernel" bullet; "How Easy Is It to Start Serving
// LLMs?", "1. Block-sparse KV memory").
//
// Design (GB300):
//   * Persistent CTAs, one work item = (sequence, logical chunk, KV head).
//     The chunk length depends only on N_s (512 * 2^k tokens, at most 32
//     chunks), so results do not depend on the batch or the page layout
//     ("How Easy Is It to Start Serving LLMs?", "3. Load balancing": long
//     requests are split into chunks and a merge step stitches them).
//   * One producer warp copies each K and V row (one token, one KV head,
//     D elements) from its page into shared memory with a 1-D bulk copy
//     (TMA) that completes on an mbarrier; stages of 64 logical tokens form
//     a ring.  Every page is read once for all Hq/Hkv query heads.
//   * Four consumer warps each take 16 tokens of a stage.  S = K q^T and
//     O^T += V^T P run on the tensor cores (mma.sync m16n8k16): the keys are
//     the M dimension and the group's query heads the N dimension, so the
//     softmax statistics of a head live in one lane column.  P is fed to
//     the PV product as a bf16 hi + lo pair (two MMAs), which keeps it to
//     about 16 significant bits; with an e4m3 cache, K and V are converted
//     exactly to f16 and P is f16.
//   * Each warp keeps its own running max and sum; the four are combined at
//     the end of the chunk in a fixed order.  A sequence of one chunk writes
//     its output directly; otherwise each chunk writes its normalised output
//     and log2-sum-exp2 to the workspace, and the CTA that finishes the last
//     chunk of a (sequence, KV head) merges them (no separate merge launch).
#include "pkv_pipeline.cuh"

namespace pkv {

// ---------------------------------------------------------------- plan
// One block: per-sequence work counts, their exclusive prefix sums, and the
// merge counters reset.  Reads device lengths; no host round trip.
__global__ void __launch_bounds__(1024) plan_kernel(AttnParams p) {
  __shared__ int warp_d[32], warp_p[32];
  const int tid = threadIdx.x, nth = blockDim.x;
  const int B = p.B;
  const int per = (B + nth - 1) / nth;
  const int s0 = min(tid * per, B), s1 = min(s0 + per, B);
  auto counts = [&](int s, int& dec, int& pf) {
    const int c0 = __ldg(p.cu_q + s), c1 = __ldg(p.cu_q + s + 1);
    const int q_s = c1 - c0;
    const int n = __ldg(p.seq_lens + s);
    dec = pf = 0;
    if (q_s == 0) return;
    if (q_s < 0 || q_s > n || (int64_t)n > (int64_t)p.max_blocks * p.bs || c0 < 0 || c1 > p.T) {
      atomicOr(p.err, kErrLengths);
      return;
    }
    if (q_s == 1 && p.G <= p.decode_max_g) {
      const int c = chunk_tokens(n);
      dec = (n + c - 1) / c;
    } else {
      pf = (int)(((int64_t)q_s * p.G + kPrefillRows - 1) / kPrefillRows);
    }
  };
  int dsum = 0, psum = 0;
  for (int s = s0; s < s1; ++s) {
    int d, f;
    counts(s, d, f);
    dsum += d;
    psum += f;
  }
  // block-wide exclusive scan of (dsum, psum)
  const int lane = tid & 31, warp = tid >> 5;
  int xd = dsum, xp = psum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int yd = __shfl_up_sync(0xffffffffu, xd, o), yp = __shfl_up_sync(0xffffffffu, xp, o);
    if (lane >= o) {
      xd += yd;
      xp += yp;
    }
  }
  if (lane == 31) {
    warp_d[warp] = xd;
    warp_p[warp] = xp;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = nth >> 5;
    int vd = lane < nw ? warp_d[lane] : 0, vp = lane < nw ? warp_p[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yd = __shfl_up_sync(0xffffffffu, vd, o), yp = __shfl_up_sync(0xffffffffu, vp, o);
      if (lane >= o) {
        vd += yd;
        vp += yp;
      }
    }
    if (lane < nw) {
      warp_d[lane] = vd;
      warp_p[lane] = vp;
    }
  }
  __syncthreads();
  int run_d = xd - dsum + (warp > 0 ? warp_d[warp - 1] : 0);
  int run_p = xp - psum + (warp > 0 ? warp_p[warp - 1] : 0);
  for (int s = s0; s < s1; ++s) {
    int d, f;
    counts(s, d, f);
    p.ws.dec_off[s] = run_d;
    p.ws.pf_off[s] = run_p;
    run_d += d;
    run_p += f;
  }
  if (s1 == B && s0 < s1) {
    p.ws.dec_off[B] = run_d;
    p.ws.pf_off[B] = run_p;
  }
  if (B == 0 && tid == 0) {
    p.ws.dec_off[0] = 0;
    p.ws.pf_off[0] = 0;
  }
  for (int i = tid; i < B * p.Hkv; i += nth) p.ws.counters[i] = 0;
}

// ---------------------------------------------------------------- decode
template <int KV, int D>
struct DecodeCfg {
  static constexpr int kEsz = KV == 2 ? 1 : 2;       // bytes per cache element
  static constexpr int kRowB = D * kEsz;              // bytes per K/V row
  static constexpr int kRowS = kRowB + 16;            // padded smem row stride
  static constexpr int kNW = 4;                       // consumer warps
  static constexpr int kST = 16 * kNW;                // tokens per stage
  static constexpr int kNS = KV == 2 ? 6 : 4;         // stages in the ring
  static constexpr int kStageB = 2 * kST * kRowS;     // K rows then V rows
  static constexpr int kMT = D / 16;                  // 16-wide d tiles
  static constexpr int kThreads = (kNW + 1) * 32;
  // combine area: m[kNW][8], l[kNW][8], o[kNW][8][D], merge weights [8][kMaxChunks]
  static constexpr int kCombFloats = kNW * 8 * 2 + kNW * 8 * D + 8 * kMaxChunks;
  static constexpr size_t kSmem = (size_t)kNS * kStageB + kCombFloats * 4 + 2 * kNS * 8 + 64;
};

struct DecodeItem {
  int s, c, g, nchunks, k0, k1, u;
  int64_t t;
};

__device__ __forceinline__ bool decode_item(const AttnParams& p, int w, DecodeItem& it) {
  const int units = __ldg(p.ws.dec_off + p.B);
  if (w >= units * p.Hkv) return false;
  it.u = w / p.Hkv;
  it.g = w - it.u * p.Hkv;
  it.s = upper_index(p.ws.dec_off, p.B, it.u);
  it.c = it.u - __ldg(p.ws.dec_off + it.s);
  const int n = __ldg(p.seq_lens + it.s);
  const int ct = chunk_tokens(n);
  it.nchunks = (n + ct - 1) / ct;
  it.k0 = it.c * ct;
  it.k1 = min(it.k0 + ct, n);
  it.t = __ldg(p.cu_q + it.s);
  return true;
}

// Output column d of accumulator tile mt, half (0: row g, 1: row g + 8).
template <int KV>
__device__ __forceinline__ int acc_d(int mt, int half, int g) {
  if constexpr (KV == 2)
    return 16 * mt + 4 * (g >> 1) + (g & 1) + 2 * half;  // permuted d of the e4m3 path
  else
    return 16 * mt + g + 8 * half;
}

template <int KV, int D, typename OutT>
__global__ void __launch_bounds__(DecodeCfg<KV, D>::kThreads, 1) decode_kernel(AttnParams p) {
  using C = DecodeCfg<KV, D>;
  using R = Ring<C::kRowB, C::kRowS, C::kST, C::kNS>;
  extern __shared__ __align__(128) unsigned char smem[];
  float* cm = reinterpret_cast<float*>(smem + (size_t)C::kNS * C::kStageB);
  float* cl = cm + C::kNW * 8;
  float* co = cl + C::kNW * 8;
  float* cw = co + C::kNW * 8 * D;
  uint64_t* bars = reinterpret_cast<uint64_t*>(cw + 8 * kMaxChunks);
  volatile int* flags = reinterpret_cast<volatile int*>(bars + 2 * C::kNS);  // [0] abort, [1] last
  R ring;
  ring.base = smem;
  ring.base_s = smem_u32(smem);
  ring.full0 = smem_u32(bars);
  ring.empty0 = smem_u32(bars + C::kNS);
  if (threadIdx.x == 0) flags[0] = flags[1] = 0;
  init_ring_barriers<C::kNS>(ring.full0, ring.empty0, C::kNW);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == C::kNW) {
    // ======================= producer warp =======================
    const char* kbase = static_cast<const char*>(p.k_cache);
    const char* vbase = static_cast<const char*>(p.v_cache);
    int fill = 0;
    DecodeItem it;
    for (int w = blockIdx.x; decode_item(p, w, it); w += gridDim.x) {
      const int32_t* bt_row = p.bt + (int64_t)it.s * p.bt_stride;
      for (int j0 = it.k0; j0 < it.k1; j0 += C::kST) {
        if (flags[0]) break;
        if (!ring.produce(p, fill, bt_row, it.g, j0, min(C::kST, it.k1 - j0), kbase, vbase, lane)) {
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
  const int g4 = lane >> 2, t4 = lane & 3;  // fragment row / column-pair index
  const int nthr = C::kNW * 32;
  int cons = 0;
  DecodeItem it;
  for (int w = blockIdx.x; decode_item(p, w, it); w += gridDim.x) {
    // ---- query fragments (B operand: k = d, n = query head of the group)
    uint32_t qb[C::kMT][2];
    {
      const bool hv = g4 < p.G;
      const int h = it.g * p.G + (hv ? g4 : 0);
      const __nv_bfloat16* qrow =
          static_cast<const __nv_bfloat16*>(p.q) + it.t * p.q_st + (int64_t)h * p.q_sh;
#pragma unroll
      for (int ks = 0; ks < C::kMT; ++ks) {
        if constexpr (KV == 2) {
          const uint2 v = hv ? *reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * t4) : make_uint2(0, 0);
          qb[ks][0] = bf16x2_to_f16x2(v.x);
          qb[ks][1] = bf16x2_to_f16x2(v.y);
        } else {
          qb[ks][0] = hv ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t4) : 0u;
          qb[ks][1] = hv ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t4 + 8) : 0u;
        }
      }
    }
    float acc[C::kMT][4];
#pragma unroll
    for (int i = 0; i < C::kMT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int j0 = it.k0; j0 < it.k1; j0 += C::kST, ++cons) {
      if (!flags[0] && !ring.wait_full(p, cons)) flags[0] = 1;
      const int base = j0 + 16 * warp;  // first token of this warp
      if (base < it.k1 && !flags[0]) {
        const uint32_t sK = ring.k_rows(cons) + (16 * warp) * C::kRowS;
        const uint32_t sV = ring.v_rows(cons) + (16 * warp) * C::kRowS;
        // ---- S = K q^T : rows = 16 tokens, cols = heads
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (KV == 2) {
          const uint32_t aK = sK + ((lane & 7) + ((lane >> 3) & 1) * 8) * C::kRowS + (lane >> 4) * 16;
#pragma unroll
          for (int kp = 0; kp < C::kMT / 2; ++kp) {
            uint32_t w0, w1, w2, w3;
            ldsm_x4(aK + 32 * kp, w0, w1, w2, w3);
            uint32_t a[4];
            e4m3x4_to_f16(w0, a[0], a[2]);
            e4m3x4_to_f16(w1, a[1], a[3]);
            mma_f16(s, a, qb[2 * kp][0], qb[2 * kp][1]);
            e4m3x4_to_f16(w2, a[0], a[2]);
            e4m3x4_to_f16(w3, a[1], a[3]);
            mma_f16(s, a, qb[2 * kp + 1][0], qb[2 * kp + 1][1]);
          }
        } else {
          const uint32_t aK = sK + ((lane & 7) + ((lane >> 3) & 1) * 8) * C::kRowS + ((lane >> 4) & 1) * 16;
#pragma unroll
          for (int ks = 0; ks < C::kMT; ++ks) {
            uint32_t a[4];
            ldsm_x4(aK + 32 * ks, a[0], a[1], a[2], a[3]);
            mma_bf16(s, a, qb[ks][0], qb[ks][1]);
          }
        }
        // ---- online softmax (base 2) per head column
        const bool v0 = base + g4 < it.k1, v1 = base + g4 + 8 < it.k1;
        const float x0 = v0 ? s[0] * p.qk_scale_log2 : -INFINITY;
        const float x1 = v0 ? s[1] * p.qk_scale_log2 : -INFINITY;
        const float x2 = v1 ? s[2] * p.qk_scale_log2 : -INFINITY;
        const float x3 = v1 ? s[3] * p.qk_scale_log2 : -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
        mx0 = warp_max_xor(mx0, 4); mx0 = warp_max_xor(mx0, 8); mx0 = warp_max_xor(mx0, 16);
        mx1 = warp_max_xor(mx1, 4); mx1 = warp_max_xor(mx1, 8); mx1 = warp_max_xor(mx1, 16);
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = exp2f(m0 - ms0), al1 = exp2f(m1 - ms1);
        const float p0 = exp2f(x0 - ms0), p1 = exp2f(x1 - ms1);
        const float p2 = exp2f(x2 - ms0), p3 = exp2f(x3 - ms1);
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int i = 0; i < C::kMT; ++i) {
          acc[i][0] *= al0;
          acc[i][1] *= al1;
          acc[i][2] *= al0;
          acc[i][3] *= al1;
        }
        // ---- O^T += V^T P : rows = d, cols = heads, k = tokens
        if constexpr (KV == 2) {
          const uint32_t b0 = movm_t(pack_f16(p0, p1)), b1 = movm_t(pack_f16(p2, p3));
          const uint32_t aV = sV + ((lane & 7) + ((lane >> 3) & 1) * 8) * C::kRowS + (lane >> 4) * 16;
#pragma unroll
          for (int cp = 0; cp < C::kMT / 2; ++cp) {
            uint32_t w0, w1, w2, w3;
            ldsm_x4(aV + 32 * cp, w0, w1, w2, w3);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t wt = hh ? w2 : w0, wb = hh ? w3 : w1;
              uint32_t x0t, x1t, x0b, x1b;
              e4m3x4_to_f16(wt, x0t, x1t);
              e4m3x4_to_f16(wb, x0b, x1b);
              const uint32_t a[4] = {movm_t(x0t), movm_t(x1t), movm_t(x0b), movm_t(x1b)};
              mma_f16(acc[2 * cp + hh], a, b0, b1);
            }
          }
        } else {
          uint32_t hi0, lo0, hi1, lo1;
          split_bf16(p0, p1, hi0, lo0);
          split_bf16(p2, p3, hi1, lo1);
          const uint32_t bh0 = movm_t(hi0), bh1 = movm_t(hi1), bl0 = movm_t(lo0), bl1 = movm_t(lo1);
          const uint32_t aV = sV + ((lane & 7) + ((lane >> 4) & 1) * 8) * C::kRowS + ((lane >> 3) & 1) * 16;
#pragma unroll
          for (int mt = 0; mt < C::kMT; ++mt) {
            uint32_t a[4];
            ldsm_x4_t(aV + 32 * mt, a[0], a[1], a[2], a[3]);
            mma_bf16(acc[mt], a, bh0, bh1);
            mma_bf16(acc[mt], a, bl0, bl1);
          }
        }
      }
      ring.release(cons, lane);
    }

    // ---- combine the four warps (fixed order) -------------------------
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    if (lane < 4) {
      cm[warp * 8 + 2 * lane] = m0;
      cm[warp * 8 + 2 * lane + 1] = m1;
      cl[warp * 8 + 2 * lane] = l0;
      cl[warp * 8 + 2 * lane + 1] = l1;
    }
    named_sync(1, nthr);
    {
      const int c0 = 2 * t4, c1 = c0 + 1;
      float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
      for (int v = 0; v < C::kNW; ++v) {
        M0 = fmaxf(M0, cm[v * 8 + c0]);
        M1 = fmaxf(M1, cm[v * 8 + c1]);
      }
      const float f0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M0);
      const float f1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M1);
      float* cow = co + warp * 8 * D;
#pragma unroll
      for (int mt = 0; mt < C::kMT; ++mt) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int d = acc_d<KV>(mt, half, g4);
          cow[c0 * D + d] = acc[mt][2 * half] * f0;
          cow[c1 * D + d] = acc[mt][2 * half + 1] * f1;
        }
      }
    }
    named_sync(1, nthr);
    const int hq0 = it.g * p.G;
    const bool single = it.nchunks == 1;
    for (int e = threadIdx.x; e < p.G * D; e += nthr) {
      const int col = e / D, d = e - col * D;
      float M = -INFINITY;
#pragma unroll
      for (int v = 0; v < C::kNW; ++v) M = fmaxf(M, cm[v * 8 + col]);
      float L = 0.f, o = 0.f;
#pragma unroll
      for (int v = 0; v < C::kNW; ++v) {
        const float mv = cm[v * 8 + col];
        L += (mv == -INFINITY ? 0.f : exp2f(mv - M)) * cl[v * 8 + col];
        o += co[(v * 8 + col) * D + d];
      }
      const float val = o / L * p.v_scale;
      const int h = hq0 + col;
      if (single) {
        store1(static_cast<OutT*>(p.out) + it.t * p.o_st + (int64_t)h * p.o_sh + d, val);
      } else {
        p.ws.part_o[((int64_t)it.u * p.Hq + h) * D + d] = val;
        if (d == 0) p.ws.part_lse[(int64_t)it.u * p.Hq + h] = M + log2f(L);
      }
    }
    if (!single) {
      // ---- last chunk of (s, g) to finish merges all of them -----------
      __threadfence();
      named_sync(1, nthr);
      if (threadIdx.x == 0) {
        const int done = atomicAdd(p.ws.counters + it.s * p.Hkv + it.g, 1);
        flags[1] = done == it.nchunks - 1;
      }
      named_sync(1, nthr);
      if (flags[1]) {
        __threadfence();
        const int u0 = __ldg(p.ws.dec_off + it.s);
        // chunk weights 2^(lse_c - max) per head column
        for (int e = threadIdx.x; e < p.G * it.nchunks; e += nthr) {
          const int col = e / it.nchunks, c = e - col * it.nchunks;
          cw[col * kMaxChunks + c] = __ldcg(p.ws.part_lse + (int64_t)(u0 + c) * p.Hq + hq0 + col);
        }
        named_sync(1, nthr);
        for (int e = threadIdx.x; e < p.G * D; e += nthr) {
          const int col = e / D, d = e - col * D;
          float M = -INFINITY;
          for (int c = 0; c < it.nchunks; ++c) M = fmaxf(M, cw[col * kMaxChunks + c]);
          float L = 0.f, o = 0.f;
          for (int c = 0; c < it.nchunks; ++c) {
            const float wgt = exp2f(cw[col * kMaxChunks + c] - M);
            L += wgt;
            o += wgt * __ldcg(p.ws.part_o + ((int64_t)(u0 + c) * p.Hq + hq0 + col) * D + d);
          }
          store1(static_cast<OutT*>(p.out) + it.t * p.o_st + (int64_t)(hq0 + col) * p.o_sh + d, o / L);
        }
      }
    }
    named_sync(1, nthr);  // the combine area is reused by the next item
  }
}

// ---------------------------------------------------------------- launch
template <int KV, int D, typename OutT>
static cudaError_t launch_decode_t(const AttnParams& p, int64_t max_items, int num_sms, cudaStream_t st) {
  using C = DecodeCfg<KV, D>;
  auto kern = decode_kernel<KV, D, OutT>;
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

cudaError_t launch_plan(const AttnParams& p, cudaStream_t st) {
  plan_kernel<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode(const AttnParams& p, int kv, int out_kind, int64_t max_items, int num_sms,
                          cudaStream_t st) {
#define PKV_DEC(KV, D) \
  (out_kind ? launch_decode_t<KV, D, __nv_bfloat16>(p, max_items, num_sms, st) \
            : launch_decode_t<KV, D, float>(p, max_items, num_sms, st))
  if (kv == 1) return p.D == 128 ? PKV_DEC(1, 128) : PKV_DEC(1, 64);
  return p.D == 128 ? PKV_DEC(2, 128) : PKV_DEC(2, 64);
#undef PKV_DEC
}

}  // namespace pkv
