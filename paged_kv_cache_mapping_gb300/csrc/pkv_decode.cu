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
//   * A work item is (sequence, logical chunk, group of HP KV heads).  The
//     chunk length depends only on N_s (256 * 2^k tokens, at most 128
//     chunks), so results depend neither on the batch nor on the page layout
//     ("How Easy Is It to Start Serving LLMs?", "3. Load balancing": long
//     requests are split into chunks and a merge step stitches them).  The
//     plan kernel lists the chunks once per call; persistent CTAs (one per
//     SM) claim items from a global counter, so every SM stays busy to the
//     end.
//   * One producer warp per CTA stages the chunk 16 logical tokens at a time:
//     a token's K row for all HP heads of the group is HP * D contiguous
//     elements of the cache (2 KB at D = 128, bf16, HP = 8), fetched with one
//     1-D bulk copy (TMA) that completes on the stage's mbarrier; V likewise.
//     Whole-token copies keep the number of TMA requests low, which is what
//     limits a TMA gather of small rows.  Block ids are fetched a stage
//     ahead; the item's descriptor and query rows go through a two-slot item
//     ring.  Every page is read once for all Hq/Hkv query heads.
//   * Consumer warp h owns KV head h of the group for the whole chunk: S =
//     K q^T and O^T += V^T P run on the tensor cores (mma.sync m16n8k16)
//     with the 16 keys of a stage as M and the head's G query heads as N, so
//     a head's softmax statistics live in one lane column and need no
//     cross-warp combine.  P enters the PV product as a bf16 hi + lo pair
//     (two MMAs; about 16 significant bits); with an e4m3 cache K and V are
//     converted exactly to f16 and P is f16.
//   * A sequence of one chunk writes its output directly.  Otherwise each
//     chunk writes its normalised output and log2-sum-exp2 to the workspace,
//     and the warp that finishes the last chunk of a (sequence, KV head)
//     merges them in chunk order (no separate merge launch, no CTA-wide
//     synchronisation).
#include "pkv_pipeline.cuh"

namespace pkv {

// ---------------------------------------------------------------- plan
// One block: per-sequence work counts, their exclusive prefix sums, the
// descriptor lists of decode chunks and prefill tiles, and the merge
// counters reset.  Reads device lengths; no host round trip.
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
    const int n = __ldg(p.seq_lens + s);
    const int t0 = __ldg(p.cu_q + s);
    if (d > 0) {
      const int ct = chunk_tokens(n);
      for (int c = 0; c < d; ++c) {
        DecodeDesc e;
        e.s = s;
        e.k0 = c * ct;
        e.k1 = min(e.k0 + ct, n);
        e.t = t0;
        e.nchunks = d;
        e.u0 = run_d;
        e.c = c;
        e.pad = 0;
        p.ws.dec_desc[run_d + c] = e;
      }
    }
    if (f > 0) {
      const int q_s = __ldg(p.cu_q + s + 1) - t0;
      for (int qt = 0; qt < f; ++qt) {
        PrefillDesc e;
        e.s = s;
        e.t0 = t0;
        e.q_s = q_s;
        e.n = n;
        e.r0 = qt * kPrefillRows;
        e.r1 = min(e.r0 + kPrefillRows, q_s * p.G);
        e.kv_end = n - q_s + (e.r1 - 1) / p.G + 1;
        e.pad = 0;
        p.ws.pf_desc[run_p + qt] = e;
      }
    }
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
  if (tid == 0) *p.ws.work = 0;
}

// ---------------------------------------------------------------- decode
template <int KV, int D>
struct DecodeGeom {
  static constexpr int kRowB = D * (KV == 2 ? 1 : 2);  // one head's K (or V) row
  static constexpr int kST = 16;                        // tokens per stage
  static constexpr int kMT = D / 16;                    // 16-wide tiles over d
  static constexpr int kQRowB = D * 2;                  // one bf16 query row
  static constexpr int kMaxHP = 8;
  static constexpr int kThreads = (kMaxHP + 1) * 32;
};

__host__ __device__ inline int align16(int v) { return (v + 15) & ~15; }

// Shared memory of a decode CTA: the stage ring, the item ring, mbarriers.
template <int KV, int D>
__host__ __device__ inline int decode_tok_stride(int hp) { return hp * DecodeGeom<KV, D>::kRowB + 16; }
template <int KV, int D>
__host__ __device__ inline int decode_stage_bytes(int hp) { return 2 * DecodeGeom<KV, D>::kST * decode_tok_stride<KV, D>(hp); }
template <int KV, int D>
__host__ __device__ inline int decode_item_bytes(int hp, int G) {
  return align16(hp * G * DecodeGeom<KV, D>::kQRowB + 64);
}
template <int KV, int D>
__host__ __device__ inline size_t decode_smem(int hp, int ns, int G) {
  return (size_t)ns * decode_stage_bytes<KV, D>(hp) + 2 * decode_item_bytes<KV, D>(hp, G) + (2 * ns + 4) * 8 + 16;
}

// Output column d of accumulator tile mt, half (0: row g, 1: row g + 8).
template <int KV>
__device__ __forceinline__ int acc_d(int mt, int half, int g) {
  if constexpr (KV == 2)
    return 16 * mt + 4 * (g >> 1) + (g & 1) + 2 * half;  // permuted d of the e4m3 path
  else
    return 16 * mt + g + 8 * half;
}

// Byte offset, within a cache, of the HP-head row of logical token j of a
// sequence, or -1 if its block id is out of range (recorded).
__device__ __forceinline__ int64_t token_row(const AttnParams& p, const int32_t* bt_row, int j, int hg,
                                             int row_bytes) {
  const int lb = p.bs_shift >= 0 ? (j >> p.bs_shift) : (j / p.bs);
  const int32_t blk = __ldg(bt_row + lb);
  if (blk < 0 || blk >= p.num_blocks) {
    atomicOr(p.err, kErrBlockRange);
    return -1;
  }
  return (((int64_t)blk * p.bs + (j - lb * p.bs)) * p.Hkv + (int64_t)hg * p.hp) * (int64_t)row_bytes;
}

template <int KV, int D, typename OutT>
__global__ void __launch_bounds__(DecodeGeom<KV, D>::kThreads, 1) decode_kernel(AttnParams p) {
  using Geo = DecodeGeom<KV, D>;
  constexpr int RowB = Geo::kRowB, ST = Geo::kST, MT = Geo::kMT, QRowB = Geo::kQRowB;
  const int HP = p.hp, NS = p.ns, G = p.G;
  const int tokS = decode_tok_stride<KV, D>(HP);
  const int stageB = decode_stage_bytes<KV, D>(HP);
  const int itemB = decode_item_bytes<KV, D>(HP, G);
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* items = smem + (size_t)NS * stageB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(items + 2 * itemB);
  const uint32_t stage0 = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * NS;
  const uint32_t ifull0 = empty0 + 8 * NS, iempty0 = ifull0 + 16;
  volatile int* flags = reinterpret_cast<volatile int*>(bars + 2 * NS + 4);  // [0] abort
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, HP);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(ifull0 + 8 * i, 1);
      mbar_init(iempty0 + 8 * i, HP);
    }
    flags[0] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp > HP) return;  // launched with (HP + 1) warps; nothing else to do
  const int HG = p.Hkv / HP;
  const int n_items = __ldg(p.ws.dec_off + p.B) * HG;

  if (warp == HP) {
    // ======================= producer warp =======================
    const char* kbase = static_cast<const char*>(p.k_cache);
    const char* vbase = static_cast<const char*>(p.v_cache);
    const int tok = lane & 15;
    const bool is_v = lane >= 16;
    const int copy_b = HP * RowB;
    int slot = 0, phase = 0, islot = 0, iphase = 0, fills = 0;
    int w = 0;
    if (lane == 0) w = atomicAdd(p.ws.work, 1);
    w = __shfl_sync(0xffffffffu, w, 0);
    while (w < n_items && !flags[0]) {
      int wn = 0;
      if (lane == 0) wn = atomicAdd(p.ws.work, 1);  // the next item, claimed ahead
      const DecodeDesc d = p.ws.dec_desc[w / HG];
      const int hg = w - (w / HG) * HG;
      // ---- publish the item: descriptor and the group's query rows
      if (!mbar_wait(iempty0 + 8 * islot, iphase ^ 1, p.err)) {
        flags[0] = 1;
        break;
      }
      unsigned char* it = items + islot * itemB;
      const int q_rows = HP * G;
      if (lane == 0) {
        int* meta = reinterpret_cast<int*>(it + q_rows * QRowB);
        meta[0] = d.s;
        meta[1] = d.k0;
        meta[2] = d.k1;
        meta[3] = d.t;
        meta[4] = d.nchunks;
        meta[5] = d.u0 + d.c;
        meta[6] = hg;
        meta[7] = d.u0;
        mbar_arrive_expect_tx(ifull0 + 8 * islot, q_rows * QRowB);
      }
      __syncwarp();
      {
        const __nv_bfloat16* q0 = static_cast<const __nv_bfloat16*>(p.q) + (int64_t)d.t * p.q_st +
                                  (int64_t)hg * q_rows * p.q_sh;
        if (p.q_sh == D) {
          if (lane == 0) bulk_g2s(smem_u32(it), q0, q_rows * QRowB, ifull0 + 8 * islot);
        } else {
          for (int r = lane; r < q_rows; r += 32)
            bulk_g2s(smem_u32(it + r * QRowB), q0 + (int64_t)r * p.q_sh, QRowB, ifull0 + 8 * islot);
        }
      }
      if (++islot == 2) {
        islot = 0;
        iphase ^= 1;
      }
      // ---- K/V stages: lanes 0-15 copy K rows, lanes 16-31 V rows
      const int32_t* bt_row = p.bt + (int64_t)d.s * p.bt_stride;
      int64_t row_next = d.k0 + tok < d.k1 ? token_row(p, bt_row, d.k0 + tok, hg, RowB) : -1;
      for (int j0 = d.k0; j0 < d.k1; j0 += ST) {
        const int64_t row = row_next;
        const int jn = j0 + ST + tok;
        row_next = jn < d.k1 ? token_row(p, bt_row, jn, hg, RowB) : -1;  // a stage ahead
        if (!mbar_wait(empty0 + 8 * slot, phase ^ 1, p.err)) {
          flags[0] = 1;
          break;
        }
        unsigned char* dst = smem + (size_t)slot * stageB + (is_v ? ST * tokS : 0) + tok * tokS;
        if (row < 0) {  // past the chunk or a bad block id: this token adds nothing
          uint4* z = reinterpret_cast<uint4*>(dst);
          for (int i = 0; i < copy_b / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
        }
        if (__any_sync(0xffffffffu, row < 0)) fence_proxy_async_smem();
        const unsigned valid = __ballot_sync(0xffffffffu, row >= 0);
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * slot, __popc(valid) * copy_b);
        __syncwarp();
        if (row >= 0) bulk_g2s(smem_u32(dst), (is_v ? vbase : kbase) + row, copy_b, full0 + 8 * slot);
        ++fills;
        if (++slot == NS) {
          slot = 0;
          phase ^= 1;
        }
      }
      w = __shfl_sync(0xffffffffu, wn, 0);
    }
    // ---- no more items: tell the consumers, then let the last copies land
    if (!flags[0] && mbar_wait(iempty0 + 8 * islot, iphase ^ 1, p.err)) {
      if (lane == 0) {
        reinterpret_cast<int*>(items + islot * itemB + HP * G * QRowB)[0] = -1;
        mbar_arrive(ifull0 + 8 * islot);
      }
    } else {
      flags[0] = 1;
    }
    for (int f = 0; f < NS && f < fills; ++f) {
      // stage slots hold the last min(NS, fills) fills; wait for each
      int sl = slot - 1 - f, ph = phase;
      if (sl < 0) {
        sl += NS;
        ph ^= 1;
      }
      if (!mbar_wait(full0 + 8 * sl, ph, p.err)) break;
    }
    return;
  }

  // ======================= consumer warp h = warp =======================
  const int h = warp;
  const int g4 = lane >> 2, t4 = lane & 3;  // fragment row / column-pair index
  int slot = 0, phase = 0, islot = 0, iphase = 0;
  for (;;) {
    if (!mbar_wait(ifull0 + 8 * islot, iphase, p.err)) {
      flags[0] = 1;
      return;
    }
    const unsigned char* it = items + islot * itemB;
    const int* meta = reinterpret_cast<const int*>(it + HP * G * QRowB);
    const int s = meta[0];
    if (s < 0) return;  // no more items
    const int k0 = meta[1], k1 = meta[2], t = meta[3], nchunks = meta[4], u = meta[5], hg = meta[6];
    const int u0 = meta[7];
    const int g = hg * HP + h;  // KV head of this warp
    // ---- query fragments (B operand: k = d, n = query head of the group)
    uint32_t qb[MT][2];
    {
      const bool hv = g4 < G;
      const unsigned char* qrow = it + (h * G + (hv ? g4 : 0)) * QRowB;
#pragma unroll
      for (int ks = 0; ks < MT; ++ks) {
        if constexpr (KV == 2) {
          const uint2 v = hv ? *reinterpret_cast<const uint2*>(qrow + 2 * (16 * ks + 4 * t4)) : make_uint2(0, 0);
          qb[ks][0] = bf16x2_to_f16x2(v.x);
          qb[ks][1] = bf16x2_to_f16x2(v.y);
        } else {
          qb[ks][0] = hv ? *reinterpret_cast<const uint32_t*>(qrow + 2 * (16 * ks + 2 * t4)) : 0u;
          qb[ks][1] = hv ? *reinterpret_cast<const uint32_t*>(qrow + 2 * (16 * ks + 2 * t4 + 8)) : 0u;
        }
      }
    }
    float acc[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int j0 = k0; j0 < k1; j0 += ST) {
      if (!mbar_wait(full0 + 8 * slot, phase, p.err)) {
        flags[0] = 1;
        return;
      }
      const uint32_t sK = stage0 + slot * stageB + h * RowB;
      const uint32_t sV = sK + ST * tokS;
      // ---- S = K q^T : rows = 16 tokens, cols = heads
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (KV == 2) {
        const uint32_t aK = sK + ((lane & 7) + ((lane >> 3) & 1) * 8) * tokS + (lane >> 4) * 16;
#pragma unroll
        for (int kp = 0; kp < MT / 2; ++kp) {
          uint32_t w0, w1, w2, w3;
          ldsm_x4(aK + 32 * kp, w0, w1, w2, w3);
          uint32_t a[4];
          e4m3x4_to_f16(w0, a[0], a[2]);
          e4m3x4_to_f16(w1, a[1], a[3]);
          mma_f16(sc, a, qb[2 * kp][0], qb[2 * kp][1]);
          e4m3x4_to_f16(w2, a[0], a[2]);
          e4m3x4_to_f16(w3, a[1], a[3]);
          mma_f16(sc, a, qb[2 * kp + 1][0], qb[2 * kp + 1][1]);
        }
      } else {
        const uint32_t aK = sK + ((lane & 7) + ((lane >> 3) & 1) * 8) * tokS + ((lane >> 4) & 1) * 16;
#pragma unroll
        for (int ks = 0; ks < MT; ++ks) {
          uint32_t a[4];
          ldsm_x4(aK + 32 * ks, a[0], a[1], a[2], a[3]);
          mma_bf16(sc, a, qb[ks][0], qb[ks][1]);
        }
      }
      // ---- online softmax (base 2) per head column
      const bool v0 = j0 + g4 < k1, v1 = j0 + g4 + 8 < k1;
      const float x0 = v0 ? sc[0] * p.qk_scale_log2 : -INFINITY;
      const float x1 = v0 ? sc[1] * p.qk_scale_log2 : -INFINITY;
      const float x2 = v1 ? sc[2] * p.qk_scale_log2 : -INFINITY;
      const float x3 = v1 ? sc[3] * p.qk_scale_log2 : -INFINITY;
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
      for (int i = 0; i < MT; ++i) {
        acc[i][0] *= al0;
        acc[i][1] *= al1;
        acc[i][2] *= al0;
        acc[i][3] *= al1;
      }
      // ---- O^T += V^T P : rows = d, cols = heads, k = tokens
      if constexpr (KV == 2) {
        const uint32_t b0 = movm_t(pack_f16(p0, p1)), b1 = movm_t(pack_f16(p2, p3));
        const uint32_t aV = sV + ((lane & 7) + ((lane >> 3) & 1) * 8) * tokS + (lane >> 4) * 16;
#pragma unroll
        for (int cp = 0; cp < MT / 2; ++cp) {
          uint32_t w0, w1, w2, w3;
          ldsm_x4(aV + 32 * cp, w0, w1, w2, w3);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t x0t, x1t, x0b, x1b;
            e4m3x4_to_f16(hh ? w2 : w0, x0t, x1t);
            e4m3x4_to_f16(hh ? w3 : w1, x0b, x1b);
            const uint32_t a[4] = {movm_t(x0t), movm_t(x1t), movm_t(x0b), movm_t(x1b)};
            mma_f16(acc[2 * cp + hh], a, b0, b1);
          }
        }
      } else {
        uint32_t hi0, lo0, hi1, lo1;
        split_bf16(p0, p1, hi0, lo0);
        split_bf16(p2, p3, hi1, lo1);
        const uint32_t bh0 = movm_t(hi0), bh1 = movm_t(hi1), bl0 = movm_t(lo0), bl1 = movm_t(lo1);
        const uint32_t aV = sV + ((lane & 7) + ((lane >> 4) & 1) * 8) * tokS + ((lane >> 3) & 1) * 16;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t a[4];
          ldsm_x4_t(aV + 32 * mt, a[0], a[1], a[2], a[3]);
          mma_bf16(acc[mt], a, bh0, bh1);
          mma_bf16(acc[mt], a, bl0, bl1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);
      if (++slot == NS) {
        slot = 0;
        phase ^= 1;
      }
    }

    // ---- epilogue of this warp's head
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    const int c0 = 2 * t4, c1 = c0 + 1;  // this thread's head columns
    const float r0 = p.v_scale / l0, r1 = p.v_scale / l1;
    const int hq0 = g * G;
    if (nchunks == 1) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int dd = acc_d<KV>(mt, half, g4);
          if (c0 < G) store1(static_cast<OutT*>(p.out) + (int64_t)t * p.o_st + (int64_t)(hq0 + c0) * p.o_sh + dd,
                             acc[mt][2 * half] * r0);
          if (c1 < G) store1(static_cast<OutT*>(p.out) + (int64_t)t * p.o_st + (int64_t)(hq0 + c1) * p.o_sh + dd,
                             acc[mt][2 * half + 1] * r1);
        }
      }
    } else {
      float* po = p.ws.part_o + (int64_t)u * p.Hq * D;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int dd = acc_d<KV>(mt, half, g4);
          if (c0 < G) po[(int64_t)(hq0 + c0) * D + dd] = acc[mt][2 * half] * r0;
          if (c1 < G) po[(int64_t)(hq0 + c1) * D + dd] = acc[mt][2 * half + 1] * r1;
        }
      }
      if (g4 == 0) {
        if (c0 < G) p.ws.part_lse[(int64_t)u * p.Hq + hq0 + c0] = m0 + log2f(l0);
        if (c1 < G) p.ws.part_lse[(int64_t)u * p.Hq + hq0 + c1] = m1 + log2f(l1);
      }
      // ---- the warp that finishes the last chunk of (s, g) merges them
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        __threadfence();  // cumulative over the warp's writes ordered by __syncwarp
        last = atomicAdd(p.ws.counters + s * p.Hkv + g, 1) == nchunks - 1;
        if (last) __threadfence();
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        for (int col = 0; col < G; ++col) {
          const float* lse = p.ws.part_lse + (int64_t)u0 * p.Hq + hq0 + col;
          float M = -INFINITY;
          for (int c = lane; c < nchunks; c += 32) M = fmaxf(M, __ldcg(lse + (int64_t)c * p.Hq));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
          float L = 0.f, o[D / 32];
#pragma unroll
          for (int k = 0; k < D / 32; ++k) o[k] = 0.f;
          for (int c = 0; c < nchunks; ++c) {
            const float wgt = exp2f(__ldcg(lse + (int64_t)c * p.Hq) - M);
            L += wgt;
            const float* src = p.ws.part_o + ((int64_t)(u0 + c) * p.Hq + hq0 + col) * D;
#pragma unroll
            for (int k = 0; k < D / 32; ++k) o[k] += wgt * __ldcg(src + lane + 32 * k);
          }
          OutT* dst = static_cast<OutT*>(p.out) + (int64_t)t * p.o_st + (int64_t)(hq0 + col) * p.o_sh;
#pragma unroll
          for (int k = 0; k < D / 32; ++k) store1(dst + lane + 32 * k, o[k] / L);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(iempty0 + 8 * islot);
    if (++islot == 2) {
      islot = 0;
      iphase ^= 1;
    }
  }
}

// ---------------------------------------------------------------- launch
// Decode geometry for a head count: HP KV heads per item (a divisor of Hkv,
// at most 8) and as many stages as fit in shared memory.
template <int KV, int D>
static bool decode_geometry(int Hkv, int G, int& hp, int& ns) {
  const size_t budget = 227 * 1024;
  for (hp = 8; hp >= 1; --hp) {
    if (Hkv % hp) continue;
    for (ns = 8; ns >= 3; --ns)
      if (decode_smem<KV, D>(hp, ns, G) <= budget) return true;
  }
  return false;
}

template <int KV, int D, typename OutT>
static cudaError_t launch_decode_t(AttnParams p, int64_t max_items, int num_sms, cudaStream_t st) {
  using Geo = DecodeGeom<KV, D>;
  int hp = 1, ns = 3;
  if (!decode_geometry<KV, D>(p.Hkv, p.G, hp, ns)) return cudaErrorInvalidConfiguration;
  p.hp = hp;
  p.ns = ns;
  const size_t smem = decode_smem<KV, D>(hp, ns, p.G);
  auto kern = decode_kernel<KV, D, OutT>;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern), 227 * 1024);
  if (e != cudaSuccess) return e;
  const int threads = (hp + 1) * 32;
  int occ = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
  if (occ < 1) occ = 1;
  int64_t grid = (int64_t)num_sms * occ;
  const int64_t items = (max_items + hp - 1) / hp;  // max_items counts (unit, KV head) pairs
  if (grid > items) grid = items;
  if (grid < 1) return cudaSuccess;
  (void)Geo::kThreads;
  kern<<<(unsigned)grid, threads, smem, st>>>(p);
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
