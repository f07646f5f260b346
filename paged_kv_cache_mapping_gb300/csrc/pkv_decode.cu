// pkv_decode.cu -- paged decode attention (one query token per sequence),
// split-KV chunks and their log-sum-exp merge.  The work lists it consumes
// come from the plan kernel (pkv_plan.cu).
//
// What it computes: for a decoding sequence s (q_s = 1, N_s keys) and query
// head h, o = sum_j softmax_j(scale * q.k_j) v_j over j < N_s, K/V read
// straight from the pages named by the block table (nanoserve, "Triton
// paged-attention decode kernel" bullet; "How Easy Is It to Start Serving
// LLMs?", "1. Block-sparse KV memory").
//
// Design (GB300):
//   * A work item is (sequence, logical chunk, group of HP KV heads).  The
//     chunk length depends only on N_s (128 * 2^k tokens, 256 * 2^k with an
//     e4m3 cache, at most 512 chunks), so results depend neither on the
//     batch nor on the page layout
//     ("How Easy Is It to Start Serving LLMs?", "3. Load balancing": long
//     requests are split into chunks and a merge step stitches them).  The
//     plan lists the chunks once per model step, full chunks first (larger
//     sizes first), ragged ones last; persistent CTAs (one per SM) claim
//     items from a global counter, so every SM stays busy to the end.
//   * A copy warp stages the chunk 16 logical tokens at a time: a token's K
//     row for all HP heads of the group is HP * D contiguous elements (2 KB
//     at D = 128, bf16, HP = 8), and two adjacent rows of one block go as one
//     1-D bulk copy (TMA) that completes on the stage's mbarrier; V likewise.
//     Few, large copies keep the number of TMA requests low, which is what
//     bounds an SM's rate.  A scheduler warp fetches block ids a group of 16
//     stages ahead; the item's descriptor and query rows go through a
//     two-slot item ring.  Every page is read once for all Hq/Hkv query heads.
//   * Consumer warp h owns KV head h of the group for the whole chunk: S =
//     K q^T and O^T += V^T P run on the tensor cores (mma.sync m16n8k16)
//     with the 16 keys of a stage as M and the head's G query heads as N, so
//     a head's softmax statistics live in one lane column and need no
//     cross-warp combine.  P enters the PV product as a bf16 hi + lo pair
//     (two MMAs; about 16 significant bits); with an e4m3 cache K and V are
//     converted exactly to f16 (V's codes come transposed from a byte-matrix
//     load) and P is f16.
//   * A sequence of one chunk writes its output directly.  Otherwise each
//     chunk writes its normalised output and log2-sum-exp2 to the workspace;
//     once all the decode items are handed out, the same queue hands out the
//     merge items of each split sequence (query-head slices of a head group,
//     R warps per head over ranges of the chunks), which wait until the other
//     CTAs report the sequence's chunks finished and combine them in chunk
//     order -- CTAs that run out of chunks merge while the others finish.
#include <algorithm>

#include "pkv_pipeline.cuh"

namespace pkv {

// ---------------------------------------------------------------- decode
template <int KV, int D>
struct DecodeGeom {
  static constexpr int kRowB = D * (KV == 2 ? 1 : 2);  // one head's K (or V) row
  static constexpr int kST = 16;                        // tokens per stage
  static constexpr int kMT = D / 16;                    // 16-wide tiles over d
  static constexpr int kQRowB = D * 2;                  // one bf16 query row
  static constexpr int kMaxHP = 8;
  static constexpr int kRecs = 16;  // stage records between the scheduler and the copy warp
  static constexpr int kThreads = (kMaxHP + 2) * 32;
};

__host__ __device__ inline int align16(int v) { return (v + 15) & ~15; }

// One stage as the scheduler warp hands it to the copy warp: the cache slot
// of each of its 16 tokens (-1: nothing to copy), the first KV head of the
// item (-1: no more stages) and the tokens that start a block (bit t).
struct StageRec {
  int32_t slot[16];
  int32_t head_off;
  uint32_t block_start;
  int32_t pad[2];
};

// Shared memory of a decode CTA: the stage ring, the item ring, mbarriers.
// Tokens are staged in pairs, the two rows of a pair back to back (one bulk
// copy of two adjacent slots fetches both: the per-copy cost, not the bytes,
// bounded an SM's rate with one copy per token row) and 16 bytes of padding
// between pairs.
template <int KV, int D>
__host__ __device__ inline int decode_pair_stride(int hp) { return 2 * hp * DecodeGeom<KV, D>::kRowB + 16; }
template <int KV, int D>
__host__ __device__ inline int decode_half_bytes(int hp) {  // the K (or V) half of a stage
  return (DecodeGeom<KV, D>::kST / 2) * decode_pair_stride<KV, D>(hp);
}
template <int KV, int D>
__host__ __device__ inline int decode_stage_bytes(int hp) { return 2 * decode_half_bytes<KV, D>(hp); }
// An item slot: the item's query rows (a decode item) or the exchange of the
// partial merges (a merge item: per consumer warp M, L and D values), then
// the item's descriptor.
template <int KV, int D>
__host__ __device__ inline int decode_item_data_bytes(int hp, int G) {
  const int q = hp * G * DecodeGeom<KV, D>::kQRowB, ex = hp * (D + 4) * 4;
  return align16(q > ex ? q : ex);
}
template <int KV, int D>
__host__ __device__ inline int decode_item_bytes(int hp, int G) {
  return decode_item_data_bytes<KV, D>(hp, G) + 64;
}
template <int KV, int D>
__host__ __device__ inline size_t decode_smem(int hp, int ns, int G) {
  return (size_t)ns * decode_stage_bytes<KV, D>(hp) + 2 * decode_item_bytes<KV, D>(hp, G) +
         DecodeGeom<KV, D>::kRecs * sizeof(StageRec) + (2 * ns + 6 + 2 * DecodeGeom<KV, D>::kRecs) * 8 + 16;
}

// Two 16 x 16 byte matrices, transposed on the way: lanes 0-15 give the
// addresses of matrix 0's rows, lanes 16-31 those of matrix 1.  Lane 4g + t
// receives, of matrix 0, column g of rows 4t .. 4t+3 (r0, row 4t in the low
// byte) and column g + 8 of the same rows (r1); r2, r3 likewise of matrix 1.
__device__ __forceinline__ void ldsm_b8_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                             uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Output column d of accumulator tile mt, half (0: row g, 1: row g + 8).
__device__ __forceinline__ int acc_d(int mt, int half, int g) {
  return 16 * mt + g + 8 * half;
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct MergePart {
  float M, L;
  float4 acc;
};

// A warp merges the results of chunks c0 .. c1-1 of query head hq of a split
// sequence (unit u0 + c holds chunk c): lane l accumulates output elements
// 4l .. 4l+3.  Returns, in every lane, the range's reference max M (log2
// units) and L = sum_c 2^(lse_c - M), and in lane l its part of
// acc = sum_c 2^(lse_c - M) o_c, chunks in order.  The range is taken in
// blocks of 128 chunks (one, up to 128 chunks per warp): lane k holds the
// weights of chunks k, k + 32, .. of a block, and the loads of sixteen
// chunks are issued together before they are used; a later block with a
// larger max rescales what came before.
template <int D>
__device__ __forceinline__ MergePart merge_range(const AttnParams& p, int u0, int c0, int c1, int hq, int lane) {
  constexpr int kQ = 4;   // chunks per lane in a block
  constexpr int kB = 16;  // chunks per batch of loads
  const float* lse = p.ws.part_lse + (int64_t)u0 * p.Hq + hq;
  const bool act = lane * 4 < D;
  const float4* base = reinterpret_cast<const float4*>(p.ws.part_o + (int64_t)u0 * p.Hq * D) +
                       (int64_t)hq * (D / 4) + lane;
  const int64_t cstep = (int64_t)p.Hq * D / 4;  // float4s between chunks
  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int b0 = c0; b0 < c1; b0 += 32 * kQ) {
    const int n = min(c1 - b0, 32 * kQ);
    float wv[kQ], lv[kQ];
    float Mb = M;
#pragma unroll
    for (int k = 0; k < kQ; ++k) {
      const int c = lane + 32 * k;
      lv[k] = c < n ? __ldcg(lse + (int64_t)(b0 + c) * p.Hq) : -INFINITY;
      Mb = fmaxf(Mb, lv[k]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Mb = fmaxf(Mb, __shfl_xor_sync(0xffffffffu, Mb, o));
    if (Mb != M) {  // the blocks before were weighted against the old max (none for the first)
      const float a = M == -INFINITY ? 0.f : exp2f(M - Mb);
      L *= a;
      acc.x *= a;
      acc.y *= a;
      acc.z *= a;
      acc.w *= a;
      M = Mb;
    }
    float l = 0.f;
#pragma unroll
    for (int k = 0; k < kQ; ++k) {
      wv[k] = lane + 32 * k < n ? exp2f(lv[k] - M) : 0.f;
      l += wv[k];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    L += l;
#pragma unroll
    for (int k = 0; k < kQ; ++k) {
      if (32 * k >= n) break;
#pragma unroll
      for (int cb = 0; cb < 32; cb += kB) {
        if (32 * k + cb >= n) break;
        float4 v[kB];
#pragma unroll
        for (int b = 0; b < kB; ++b) {
          const int c = 32 * k + cb + b;
          v[b] = act && c < n ? __ldcg(base + (int64_t)(b0 + c) * cstep) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int b = 0; b < kB; ++b) {
          const float wc = __shfl_sync(0xffffffffu, wv[k], cb + b);  // 0 past n
          acc.x += wc * v[b].x;
          acc.y += wc * v[b].y;
          acc.z += wc * v[b].z;
          acc.w += wc * v[b].w;
        }
      }
    }
  }
  return MergePart{M, L, acc};
}

// A warp merges all the chunk results of query head hq of a split sequence
// of n <= 128 chunks and writes the output row (the merge items whose
// heads each take one warp): lane c holds the weights of chunks c, c + 32,
// ..; lane l accumulates output elements 4l .. 4l+3.  The first sixteen
// chunks' loads go out with the log-sum-exp loads, the others sixteen at a
// time.  o = sum_c 2^(lse_c - M) o_c / sum_c 2^(lse_c - M), chunks in order.
template <typename OutT, int D>
__device__ __noinline__ void merge_head(const AttnParams& p, int u0, int n, int hq, int t, int lane) {
  constexpr int kQ = 4;   // chunks per lane
  constexpr int kB = 16;  // chunks per batch of loads
  const bool act = lane * 4 < D;
  const float4* base = reinterpret_cast<const float4*>(p.ws.part_o + (int64_t)u0 * p.Hq * D) +
                       (int64_t)hq * (D / 4) + lane;
  const int64_t cstep = (int64_t)p.Hq * D / 4;  // float4s between chunks
  float4 v[kB];
#pragma unroll
  for (int b = 0; b < kB; ++b) v[b] = act && b < n ? __ldcg(base + b * cstep) : make_float4(0.f, 0.f, 0.f, 0.f);
  float wv[kQ], lv[kQ];
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kQ; ++k) {
    const int c = lane + 32 * k;
    lv[k] = c < n ? __ldcg(p.ws.part_lse + (int64_t)(u0 + c) * p.Hq + hq) : -INFINITY;
    M = fmaxf(M, lv[k]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f;
#pragma unroll
  for (int k = 0; k < kQ; ++k) {
    wv[k] = lane + 32 * k < n ? exp2f(lv[k] - M) : 0.f;
    L += wv[k];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kQ; ++k) {
    if (32 * k >= n) break;
#pragma unroll
    for (int cb = 0; cb < 32; cb += kB) {
      if (32 * k + cb >= n) break;
      if (k + cb > 0) {
#pragma unroll
        for (int b = 0; b < kB; ++b) {
          const int c = 32 * k + cb + b;
          v[b] = act && c < n ? __ldcg(base + c * cstep) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const float wc = __shfl_sync(0xffffffffu, wv[k], cb + b);  // 0 past n
        acc.x += wc * v[b].x;
        acc.y += wc * v[b].y;
        acc.z += wc * v[b].z;
        acc.w += wc * v[b].w;
      }
    }
  }
  if (!act) return;
  const float inv_l = 1.f / L;
  OutT* dst = static_cast<OutT*>(p.out) + (int64_t)t * p.o_st + (int64_t)hq * p.o_sh + 4 * lane;
  store2(dst, acc.x * inv_l, acc.y * inv_l);
  store2(dst + 2, acc.z * inv_l, acc.w * inv_l);
}

// Stores lane l's elements 4l .. 4l+3 of query head hq of row t: acc / L.
template <typename OutT, int D>
__device__ __forceinline__ void store_merged(const AttnParams& p, int t, int hq, int lane, float L, float4 acc) {
  if (lane * 4 >= D) return;
  const float inv_l = 1.f / L;
  OutT* dst = static_cast<OutT*>(p.out) + (int64_t)t * p.o_st + (int64_t)hq * p.o_sh + 4 * lane;
  store2(dst, acc.x * inv_l, acc.y * inv_l);
  store2(dst + 2, acc.z * inv_l, acc.w * inv_l);
}

// Item descriptor as published in the item ring.
enum : int { kItemDecode = 0, kItemMerge = 1 };
// u: the chunk of a decode item, the first query head (within the group) of
// a merge item; a merge item's k0 holds the done count it waits for (the
// sequence's chunks of every run of the plan so far, this one included) and
// its k1 holds H | (R << 8) (see MergeDesc).
struct ItemMeta {
  int s, k0, k1, t, nchunks, u, hg, u0, kind;
};

// Consumer warp h's part of merge item m: H query heads from m.u of the
// group's HP * G, each merged by R warps over R ranges of the chunks
// (H * R = HP); warp h takes head m.u + h / R and range h % R.  With R > 1
// the partial merges of a head meet in the item slot's data area (warp h:
// M, L, then its D values), exchanged through the slot's barrier mb (phase
// mph), and the warp of range 0 combines them:
// o = sum_r 2^(M_r - M*) acc_r / sum_r 2^(M_r - M*) L_r.  Out of line, so
// that the decode loop's code stays as it is.  Returns false if the wait for
// the other warps gave up.
template <typename OutT, int D>
__device__ __noinline__ bool merge_item(const AttnParams& p, int u0, int n, int hq0, int t, int k1, int h, int lane,
                                        unsigned char* it, uint32_t mb, int mph, int ready) {
  const int R = k1 >> 8;
  const int r = h % R;
  const int hq = hq0 + h / R;
  MergePart mp{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  if (ready) mp = merge_range<D>(p, u0, r * n / R, (r + 1) * n / R, hq, lane);
  if (R == 1) {
    if (ready) store_merged<OutT, D>(p, t, hq, lane, mp.L, mp.acc);
    return true;
  }
  float* ex = reinterpret_cast<float*>(it) + h * (D + 4);
  if (lane == 0) {
    ex[0] = mp.M;
    ex[1] = mp.L;
  }
  if (lane * 4 < D) *reinterpret_cast<float4*>(ex + 4 + 4 * lane) = mp.acc;
  __syncwarp();
  if (lane == 0) mbar_arrive(mb);
  if (r != 0) return true;
  if (!mbar_wait_warp(mb, mph, p.err)) return false;
  if (!ready) return true;
  const float* e0 = reinterpret_cast<const float*>(it) + h * (D + 4);
  float Ms = -INFINITY;
  for (int q = 0; q < R; ++q) Ms = fmaxf(Ms, e0[q * (D + 4)]);
  float Ls = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q = 0; q < R; ++q) {
    const float* e = e0 + q * (D + 4);
    const float wq = exp2f(e[0] - Ms);
    Ls += wq * e[1];
    if (lane * 4 < D) {
      const float4 v = *reinterpret_cast<const float4*>(e + 4 + 4 * lane);
      a.x += wq * v.x;
      a.y += wq * v.y;
      a.z += wq * v.z;
      a.w += wq * v.w;
    }
  }
  store_merged<OutT, D>(p, t, hq, lane, Ls, a);
  return true;
}


template <int KV, int D, typename OutT>
__device__ __forceinline__ void decode_body(const AttnParams& p) {
  using Geo = DecodeGeom<KV, D>;
  constexpr int RowB = Geo::kRowB, ST = Geo::kST, MT = Geo::kMT, QRowB = Geo::kQRowB;
  const int HP = p.hp, NS = p.ns, G = p.G;
  const int pairS = decode_pair_stride<KV, D>(HP);
  // e4m3: MMA rows 8-15 take the odd tokens of pairs rot, rot + 1, .. (mod
  // 8), so that the byte-matrix V loads below read eight different bank
  // groups per eight rows; rot = 4 where a pair's two rows sit a multiple
  // of 128 bytes apart (their banks coincide), else 0
  const int rot = KV == 2 && ((HP * RowB) & 127) == 0 ? 4 : 0;
  const int halfB = decode_half_bytes<KV, D>(HP);
  const int stageB = decode_stage_bytes<KV, D>(HP);
  const int itemB = decode_item_bytes<KV, D>(HP, G);
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* items = smem + (size_t)NS * stageB;
  constexpr int NR = Geo::kRecs;
  StageRec* recs = reinterpret_cast<StageRec*>(items + 2 * itemB);
  uint64_t* bars = reinterpret_cast<uint64_t*>(recs + NR);
  const uint32_t stage0 = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * NS;
  const uint32_t ifull0 = empty0 + 8 * NS, iempty0 = ifull0 + 16;
  const uint32_t rfull0 = iempty0 + 16, rempty0 = rfull0 + 8 * NR;
  const uint32_t mex0 = rempty0 + 8 * NR;  // [2] partial merges of the item in slot i written
  volatile int* flags = reinterpret_cast<volatile int*>(bars + 2 * NS + 6 + 2 * NR);  // [0] abort
  const int itemD = decode_item_data_bytes<KV, D>(HP, G);  // the descriptor's offset in a slot
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
    for (int i = 0; i < NR; ++i) {
      mbar_init(rfull0 + 8 * i, 32);
      mbar_init(rempty0 + 8 * i, 32);
    }
    mbar_init(mex0, HP);
    mbar_init(mex0 + 8, HP);
    flags[0] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // the plan kernel's lists are complete after this wait; beside the
  // tensor-core prefill the wait is at the end (see decode_kernel)
  if (!p.dec_concurrent) grid_dep_wait();
  if (warp > HP + 1) return;  // launched with (HP + 2) warps; nothing else to do
  const int HG = p.Hkv / HP;

  if (warp == HP) {
    // ======================= copy warp =======================
    // Issues the K/V copies of each stage record, all HP heads of the item
    // per token row, 16-byte-aligned bulk copies: lane l < 16 copies token
    // pair l % 8 (K on lanes 0-7, V on 8-15), both rows in one copy when
    // they are adjacent slots of one block (block size 1: never).  Otherwise, with a bf16 cache
    // lane l copies the pair's first row and lane l + 16 its second; with an
    // e4m3 cache lane l copies both (the arrangement that measured fastest
    // for each format).  It reads no global memory itself, so nothing but a
    // free stage slot holds it up.
    const char* kbase = static_cast<const char*>(p.k_cache);
    const char* vbase = static_cast<const char*>(p.v_cache);
    const int copy_b = HP * RowB;
    const uint64_t pol = l2_evict_first_policy();  // each K/V row is read once per call
    int rec = 0, rphase = 0, slot = 0, phase = 0, fills = 0;
    for (;;) {
      if (!mbar_wait(rfull0 + 8 * rec, rphase, p.err)) {
        flags[0] = 1;
        break;
      }
      const int q = lane & 7;
      const bool pv = ((lane >> 3) & 1) != 0;
      const int32_t sl_a = recs[rec].slot[2 * q], sl_b = recs[rec].slot[2 * q + 1];
      const int head_off = recs[rec].head_off;
      const uint32_t starts = recs[rec].block_start;
      mbar_arrive(rempty0 + 8 * rec);
      if (++rec == NR) {
        rec = 0;
        rphase ^= 1;
      }
      if (head_off < 0) break;  // no more stages
      if (!mbar_wait(empty0 + 8 * slot, phase ^ 1, p.err)) {
        flags[0] = 1;
        break;
      }
      const char* src = pv ? vbase : kbase;
      unsigned char* dst = smem + (size_t)slot * stageB + (pv ? halfB : 0) + q * pairS;
      // adjacent slots of one block, for an item covering every KV head, are
      // one contiguous run; slots of adjacent blocks are not joined, so that
      // the copies a stage takes do not depend on where its blocks lie
      const bool joint = sl_a >= 0 && sl_b == sl_a + 1 && !((starts >> (2 * q + 1)) & 1u) && HP == p.Hkv;
      int bytes = 0;
      bool zeroed = false;
      auto zero_row = [&](unsigned char* row) {  // a token that adds nothing: zeros keep the MMA inputs finite
        uint4* z = reinterpret_cast<uint4*>(row);
        for (int k = 0; k < copy_b / 16; ++k) z[k] = make_uint4(0, 0, 0, 0);
        zeroed = true;
      };
      if constexpr (KV == 2) {
        // lanes 0-15: the pair, or both of its rows one by one
        const bool act = lane < 16;
        if (act && !joint) {
          if (sl_a < 0) zero_row(dst); else bytes += copy_b;
          if (sl_b < 0) zero_row(dst + copy_b); else bytes += copy_b;
        } else if (act) {
          bytes = 2 * copy_b;
        }
        if (__any_sync(0xffffffffu, zeroed)) fence_proxy_async_smem();
        const unsigned total = __reduce_add_sync(0xffffffffu, (unsigned)bytes);
        if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * slot, total);
        __syncwarp();
        if (act && joint) {
          bulk_g2s_hint(smem_u32(dst), src + ((int64_t)sl_a * p.Hkv + head_off) * RowB, 2 * copy_b,
                        full0 + 8 * slot, pol);
        } else if (act) {
          if (sl_a >= 0)
            bulk_g2s_hint(smem_u32(dst), src + ((int64_t)sl_a * p.Hkv + head_off) * RowB, copy_b, full0 + 8 * slot,
                          pol);
          if (sl_b >= 0)
            bulk_g2s_hint(smem_u32(dst + copy_b), src + ((int64_t)sl_b * p.Hkv + head_off) * RowB, copy_b,
                          full0 + 8 * slot, pol);
        }
      } else {
        // lanes 0-15: the pair or its first row; lanes 16-31: the second row
        // of a pair that is not joint
        const bool second = lane >= 16;
        const bool act = !(second && joint);
        const int32_t sl = second ? sl_b : sl_a;
        if (second) dst += copy_b;
        if (act) {
          if (sl < 0) zero_row(dst); else bytes = joint ? 2 * copy_b : copy_b;
        }
        if (__any_sync(0xffffffffu, zeroed)) fence_proxy_async_smem();
        const unsigned total = __reduce_add_sync(0xffffffffu, (unsigned)bytes);
        if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * slot, total);
        __syncwarp();
        if (bytes > 0)
          bulk_g2s_hint(smem_u32(dst), src + ((int64_t)sl * p.Hkv + head_off) * RowB, (uint32_t)bytes,
                        full0 + 8 * slot, pol);
      }
      ++fills;
      if (++slot == NS) {
        slot = 0;
        phase ^= 1;
      }
    }
    // let the last copies land before the CTA can exit
    for (int f = 0; f < NS && f < fills; ++f) {
      int sl = slot - 1 - f, ph = phase;
      if (sl < 0) {
        sl += NS;
        ph ^= 1;
      }
      if (!mbar_wait(full0 + 8 * sl, ph, p.err)) break;
    }
    return;
  }

  if (warp == HP + 1) {
    // ======================= scheduler warp =======================
    // Claims items, publishes each to the consumers (descriptor and query
    // rows) and turns its keys into stage records for the copy warp.  Every
    // global load on the path (work counter, descriptors, block tables) is
    // taken here, up to kRecs stages ahead of the copies, so that their
    // latency never stalls the copy stream.  When the consumers hand an item
    // slot back, a split chunk they finished is reported to the merge items
    // through the sequence's done counter.
    // the plan's sizes (the other warps do not need them); a workspace
    // planned for other shapes gives no work
    const bool planned = plan_matches_warp(p);
    int32_t sz = 0;
    if (lane == 0) sz = __ldcg(p.ws.dec_off + p.B);
    if (lane == 1) sz = __ldcg(p.ws.n_merge);
    const int dec_units = __shfl_sync(0xffffffffu, sz, 0), merges = __shfl_sync(0xffffffffu, sz, 1);
    if (!planned && lane == 0) atomicOr(p.err, kErrPlan);
    const int n_dec = planned ? dec_units * HG : 0;             // decode items, then
    const int n_items = planned ? n_dec + merges : 0;           // merge items
    constexpr int GS = 16;  // stages whose block-table entries are loaded together
    constexpr int32_t kPast = INT32_MIN;
    const int tok = lane & 15, half = lane >> 4;
    int rec = 0, rphase = 0;
    int islot = 0, iphase = 0;
    int pub0 = 0, pub1 = 0;      // items published into item slot 0 / 1
    int done0 = -1, done1 = -1;  // done-counter index of a split chunk held by slot 0 / 1
    auto retire = [&](int x) {
      const int di = x ? done1 : done0;
      if (di >= 0 && lane == 0) {
        __threadfence();  // the consumers' partial writes (seen through the slot's mbarrier) first
        atomicAdd(p.ws.done + di, 1);
      }
      if (x) done1 = -1; else done0 = -1;
    };
    // Publishes item x (descriptor e) into the next item slot, or the end
    // marker when x >= n_items, once the consumers have handed the slot back.
    // run: how many runs of the plan came before this one (merge items).
    auto publish = [&](int x, const DecodeDesc& e, int run) -> bool {
      if (!mbar_wait(iempty0 + 8 * islot, iphase ^ 1, p.err)) return false;
      retire(islot);
      unsigned char* it = items + islot * itemB;
      const int q_rows = HP * G;
      ItemMeta* mp = reinterpret_cast<ItemMeta*>(it + itemD);
      if (x >= n_items) {
        if (lane == 0) {
          mp->s = -1;
          mbar_arrive(ifull0 + 8 * islot);
        }
      } else if (x < n_dec) {
        const int hg = x - (x / HG) * HG;
        if (e.nchunks > 1) {
          if (islot) done1 = e.s * HG + hg; else done0 = e.s * HG + hg;
        }
        if (lane == 0) {
          *mp = ItemMeta{e.s, e.k0, e.k1, e.t, e.nchunks, e.u0 + e.c, hg, e.u0, kItemDecode};
          mbar_arrive_expect_tx(ifull0 + 8 * islot, q_rows * QRowB);
        }
        __syncwarp();
        const __nv_bfloat16* q0 = static_cast<const __nv_bfloat16*>(p.q) + (int64_t)e.t * p.q_st +
                                  (int64_t)hg * q_rows * p.q_sh;
        if (p.q_sh == D) {
          if (lane == 0) bulk_g2s(smem_u32(it), q0, q_rows * QRowB, ifull0 + 8 * islot);
        } else {
          for (int r = lane; r < q_rows; r += 32)
            bulk_g2s(smem_u32(it + r * QRowB), q0 + (int64_t)r * p.q_sh, QRowB, ifull0 + 8 * islot);
        }
      } else {
        const int4* mdp = reinterpret_cast<const int4*>(p.ws.merge_desc + (x - n_dec));
        const int4 md0 = __ldcg(mdp), md1 = __ldcg(mdp + 1);  // s, hg, h0, hr | nchunks, u0, t
        // the counts wrap modulo 2^32 on both sides
        const int need = static_cast<int>((static_cast<unsigned>(run) + 1u) * static_cast<unsigned>(md1.x));
        const ItemMeta mm{md0.x, need, md0.w, md1.z, md1.x, md0.z, md0.y, md1.y, kItemMerge};
        if (lane == 0) {
          *mp = mm;
          mbar_arrive(ifull0 + 8 * islot);
        }
      }
      __syncwarp();
      if (islot) ++pub1; else ++pub0;
      if (++islot == 2) {
        islot = 0;
        iphase ^= 1;
      }
      return true;
    };
    // Hands one record to the copy warp; every lane arrives, releasing its
    // own writes to the record.
    auto put_record = [&](int tok_slot, bool writer, int head_off, uint32_t starts) -> bool {
      if (!mbar_wait(rempty0 + 8 * rec, rphase ^ 1, p.err)) return false;
      if (writer) recs[rec].slot[tok] = tok_slot;
      if (lane == 0) {
        recs[rec].head_off = head_off;
        recs[rec].block_start = starts;
      }
      mbar_arrive(rfull0 + 8 * rec);
      if (++rec == NR) {
        rec = 0;
        rphase ^= 1;
      }
      return true;
    };
    bool ok = true;
    int w = blockIdx.x;
    // Claims.  Alone, a CTA's first item is its index and each item it
    // processes claims the next: a run makes n_items claims, and claim c of
    // the run's base .. base + n_items - 1 names item gridDim.x + c - base.
    // Beside the prefill, CTAs start at different times (some only when a
    // prefill CTA leaves its SM), so every item is claimed, the first one
    // too: a run makes n_items + gridDim.x claims (each CTA one past the
    // end), and claim c names item c - base.  base is a multiple of the run's
    // claim count, found once from the first claim (lane 0 only).
    const bool claim_all = p.dec_concurrent != 0;
    const unsigned long long run_claims =
        static_cast<unsigned long long>(n_items) + (claim_all ? gridDim.x : 0u);
    unsigned long long base = ~0ull;
    int run = 0;
    auto find_base = [&](unsigned long long c) {
      if (base == ~0ull) {
        run = static_cast<int>(c / run_claims);
        base = c - c % run_claims;
      }
    };
    if (claim_all) {
      w = n_items;
      if (n_items > 0) {
        int first = 0;
        if (lane == 0) {
          const unsigned long long c = atomicAdd(p.ws.work, 1ull);
          find_base(c);
          first = static_cast<int>(c - base);
        }
        w = __shfl_sync(0xffffffffu, first, 0);
      }
    }
    while (ok && w < n_items && !flags[0]) {
      // the next item (read at the end of the iteration)
      unsigned long long c = 0;
      if (lane == 0) c = atomicAdd(p.ws.work, 1ull);
      DecodeDesc d{};
      const bool is_dec = w < n_dec;
      int item_run = 0;
      if (is_dec) {
        const int4* dp = reinterpret_cast<const int4*>(p.ws.dec_desc + w / HG);
        const int4 d0 = __ldcg(dp), d1 = __ldcg(dp + 1);
        d = DecodeDesc{d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
      } else {  // a merge item needs the run number
        if (lane == 0) find_base(c);
        item_run = __shfl_sync(0xffffffffu, run, 0);
      }
      ok = publish(w, d, item_run);
      if (ok && is_dec) {
        const int head_off = (w - (w / HG) * HG) * HP;
        const int32_t* bt_row = p.bt + (int64_t)d.s * p.bt_stride;
        for (int gb = d.k0; gb < d.k1 && ok; gb += ST * GS) {
          // lane (tok, half) resolves token tok of stages half, half + 2, ..
          int32_t blk[GS / 2], off[GS / 2];
#pragma unroll
          for (int k = 0; k < GS / 2; ++k) {
            const int j = gb + ST * (2 * k + half) + tok;
            blk[k] = kPast;
            off[k] = 0;
            if (j < d.k1) {
              const int lb = p.bs_shift >= 0 ? (j >> p.bs_shift) : (j / p.bs);
              off[k] = j - lb * p.bs;
              blk[k] = __ldcg(bt_row + lb);
            }
          }
          int32_t sl[GS / 2];
#pragma unroll
          for (int k = 0; k < GS / 2; ++k) {
            const bool valid = (uint32_t)blk[k] < (uint32_t)p.num_blocks;
            if (!valid && blk[k] != kPast) atomicOr(p.err, kErrBlockRange);
            sl[k] = valid ? blk[k] * p.bs + off[k] : -1;
          }
#pragma unroll
          for (int i = 0; i < GS; ++i) {
            if (gb + ST * i >= d.k1) break;
            // the stage's tokens at offset 0 of their block
            const uint32_t m = __ballot_sync(0xffffffffu, off[i >> 1] == 0) >> (16 * (i & 1));
            if (!put_record(sl[i >> 1], half == (i & 1), head_off, m & 0xffffu)) {
              ok = false;
              break;
            }
          }
        }
      }
      int next = 0;
      if (lane == 0) {
        find_base(c);
        next = static_cast<int>((claim_all ? 0u : gridDim.x) + (c - base));
      }
      w = __shfl_sync(0xffffffffu, next, 0);
    }
    // ---- the end: the consumers' end marker, the copy warp's end record,
    // and the last item's split chunk reported once its slot comes back
    if (ok && !flags[0]) ok = publish(n_items, DecodeDesc{}, 0);
    if (!put_record(-1, true, -1, 0u)) ok = false;
    if (ok && !flags[0]) {
      const int n_last = islot ? pub1 : pub0;  // the slot published before the end marker
      if (n_last > 0 && mbar_wait(iempty0 + 8 * islot, (n_last - 1) & 1, p.err)) retire(islot);
    } else {
      flags[0] = 1;
    }
    return;
  }

  // ======================= consumer warp h = warp =======================
  const int h = warp;
  const int g4 = lane >> 2, t4 = lane & 3;  // fragment row / column-pair index
  int slot = 0, phase = 0, islot = 0, iphase = 0;
  int mphase = 0;  // bit i: the phase of slot i's exchange barrier
  for (;;) {
    if (!mbar_wait(ifull0 + 8 * islot, iphase, p.err)) {
      flags[0] = 1;
      return;
    }
    unsigned char* it = items + islot * itemB;
    const ItemMeta m = *reinterpret_cast<const ItemMeta*>(it + itemD);
    if (m.s < 0) return;  // no more items
    const int g = m.hg * HP + h;  // KV head of this warp
    const int hq0 = g * G;
    if (m.kind == kItemMerge) {
      // ---- merge a split sequence's chunks once every chunk is finished
      int ready = 1;
      if (lane == 0) {
        const int32_t* cnt = p.ws.done + m.s * HG + m.hg;
        // done counts run on (modulo 2^32): compare the difference
        auto short_of = [&]() { return static_cast<int>(static_cast<unsigned>(ld_acquire(cnt)) -
                                                        static_cast<unsigned>(m.k0)) < 0; };
        if (short_of()) {
          const long long t0 = clock64();
          while (short_of()) {
            __nanosleep(200);
            if (clock64() - t0 > kWaitLimitCycles) {
              atomicOr(p.err, kErrWaitTimeout);
              ready = 0;
              break;
            }
          }
        }
      }
      ready = __shfl_sync(0xffffffffu, ready, 0);
      __syncwarp();
      const int R = m.k1 >> 8;
      if (R == 1 && m.nchunks <= 128) {  // one warp per head
        if (ready) merge_head<OutT, D>(p, m.u0, m.nchunks, m.hg * HP * G + m.u + h, m.t, lane);
      } else if (!merge_item<OutT, D>(p, m.u0, m.nchunks, m.hg * HP * G + m.u, m.t, m.k1, h, lane, it,
                                      mex0 + 8 * islot, (mphase >> islot) & 1, ready)) {
        flags[0] = 1;
      }
      if (R > 1) mphase ^= 1 << islot;
      __syncwarp();
      if (lane == 0) mbar_arrive(iempty0 + 8 * islot);
      if (++islot == 2) {
        islot = 0;
        iphase ^= 1;
      }
      continue;
    }
    const int k0 = m.k0, k1 = m.k1;
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
      const uint32_t sV = sK + halfB;
      // ---- S = K q^T : rows = 16 tokens, cols = heads
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (KV == 2) {
        // MMA row r < 8 holds token 2r, row 8 + r the odd token of pair
        // (r + rot) % 8: each 8-row matrix reads 8 different pairs, in 8
        // different bank groups
        const int kodd = (lane >> 3) & 1;
        const uint32_t aK = sK + (((lane & 7) + kodd * rot) & 7) * pairS + kodd * (HP * RowB) + (lane >> 4) * 16;
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
        // MMA row r holds token 2 (r % 8) + r / 8 (the e4m3 order with rot 0)
        const uint32_t aK = sK + (lane & 7) * pairS + ((lane >> 3) & 1) * (HP * RowB) + ((lane >> 4) & 1) * 16;
#pragma unroll
        for (int ks = 0; ks < MT; ++ks) {
          uint32_t a[4];
          ldsm_x4(aK + 32 * ks, a[0], a[1], a[2], a[3]);
          mma_bf16(sc, a, qb[ks][0], qb[ks][1]);
        }
      }
      // ---- online softmax (base 2) per head column
      // the tokens of accumulator rows g4 and g4 + 8
      const int tr0 = 2 * g4, tr1 = 2 * ((g4 + rot) & 7) + 1;
      const bool v0 = j0 + tr0 < k1, v1 = j0 + tr1 < k1;
      if (p.soft_cap > 0.f) {  // soft cap: cap * tanh(s / cap), in base 2
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = p.cap_post * tanhf(sc[e] * p.cap_pre);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] *= p.qk_scale_log2;
      }
      const float x0 = v0 ? sc[0] : -INFINITY;
      const float x1 = v0 ? sc[1] : -INFINITY;
      const float x2 = v1 ? sc[2] : -INFINITY;
      const float x3 = v1 ? sc[3] : -INFINITY;
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
      // the running max moves in few stages: most skip the rescale (a
      // factor of exactly 1 leaves acc as it is)
      if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          acc[i][0] *= al0;
          acc[i][1] *= al1;
          acc[i][2] *= al0;
          acc[i][3] *= al1;
        }
      }
      // ---- O^T += V^T P : rows = d, cols = heads, k = tokens
      if constexpr (KV == 2) {
        // k positions 2t, 2t + 1 of the product are the tokens of MMA rows
        // 2t, 2t + 1 (tokens 4t, 4t + 2) and k positions 2t + 8, 2t + 9 those
        // of rows 2t + 8, 2t + 9 (the odd tokens of pairs 2t + rot, 2t + 1 +
        // rot, mod 8), as the transposed P below has them; a transposing
        // byte load of the V rows of those four tokens, in that order, as
        // source rows 4t .. 4t + 3 gives each lane its codes in k order,
        // d = 16 mt + g (and + 8) down the rows
        const uint32_t b0 = movm_t(pack_f16(p0, p1)), b1 = movm_t(pack_f16(p2, p3));
        const int vr = lane & 15, vb = vr & 3, vt = vr >> 2;
        const int vpair = vb < 2 ? 2 * vt + vb : (2 * vt + vb - 2 + rot) & 7;
        const uint32_t aV = sV + vpair * pairS + (vb >> 1) * (HP * RowB) + (lane >> 4) * 16;
#pragma unroll
        for (int cp = 0; cp < MT / 2; ++cp) {
          uint32_t w0, w1, w2, w3;
          ldsm_b8_x2_t(aV + 32 * cp, w0, w1, w2, w3);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t a[4];
            e4m3x4_to_f16(hh ? w2 : w0, a[0], a[2]);
            e4m3x4_to_f16(hh ? w3 : w1, a[1], a[3]);
            mma_f16(acc[2 * cp + hh], a, b0, b1);
          }
        }
      } else {
        uint32_t hi0, lo0, hi1, lo1;
        split_bf16(p0, p1, hi0, lo0);
        split_bf16(p2, p3, hi1, lo1);
        const uint32_t bh0 = movm_t(hi0), bh1 = movm_t(hi1), bl0 = movm_t(lo0), bl1 = movm_t(lo1);
        // k position j of the product is token 2 (j % 8) + j / 8, as in S
        const uint32_t aV = sV + (lane & 7) * pairS + ((lane >> 4) & 1) * (HP * RowB) + ((lane >> 3) & 1) * 16;
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
    const int t = m.t, u = m.u;
    if (m.nchunks == 1) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int dd = acc_d(mt, half, g4);
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
          const int dd = acc_d(mt, half, g4);
          if (c0 < G) po[(int64_t)(hq0 + c0) * D + dd] = acc[mt][2 * half] * r0;
          if (c1 < G) po[(int64_t)(hq0 + c1) * D + dd] = acc[mt][2 * half + 1] * r1;
        }
      }
      if (g4 == 0) {
        if (c0 < G) p.ws.part_lse[(int64_t)u * p.Hq + hq0 + c0] = m0 + log2f(l0);
        if (c1 < G) p.ws.part_lse[(int64_t)u * p.Hq + hq0 + c1] = m1 + log2f(l1);
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

template <int KV, int D, typename OutT>
__global__ void __launch_bounds__(DecodeGeom<KV, D>::kThreads, 1) decode_kernel(AttnParams p) {
  // the kernel that follows (the next layer's append or run) may launch and
  // set up on the SMs this grid leaves; it waits for this grid to complete
  launch_dependents();
  decode_body<KV, D, OutT>(p);
  // Beside the tensor-core prefill (dec_concurrent) this grid is launched as
  // soon as every prefill CTA has passed its own dependency wait, which
  // comes after the plan's kernel completed; so the plan's lists, and
  // everything written before the plan, are in place when the decode CTAs
  // start, and they read them through L2 (no stale L1 lines).  The prefill
  // writes nothing the decode kernel reads.  CTA 0 waits for the prefill
  // before it exits, which makes this grid -- the last of the call --
  // complete only after the prefill has; the other CTAs leave as soon as
  // their items are done, so that the next kernel's CTAs can take their SMs.
  if (p.dec_concurrent && blockIdx.x == 0) grid_dep_wait();
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
static cudaError_t launch_decode_t(AttnParams p, int64_t max_items, int num_sms, cudaStream_t st, bool pdl) {
  int hp = 1, ns = 3;
  if (!decode_geometry<KV, D>(p.Hkv, p.G, hp, ns) || hp != p.hp) return cudaErrorInvalidConfiguration;
  p.ns = ns;
  const size_t smem = decode_smem<KV, D>(hp, ns, p.G);
  auto kern = decode_kernel<KV, D, OutT>;
  cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(kern), 227 * 1024);
  if (e != cudaSuccess) return e;
  const int threads = (hp + 2) * 32;
  int occ = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
  if (occ < 1) occ = 1;
  int64_t grid = (int64_t)num_sms * occ;
  const int64_t items = (max_items + hp - 1) / hp + (int64_t)p.B * p.Hq;  // chunks + merges
  if (grid > items) grid = items;
  if (grid < 1) return cudaSuccess;
  return launch_ex(kern, dim3((unsigned)grid), dim3(threads), smem, st, pdl, p);
}

int decode_heads_per_item(int kv, int D, int Hkv, int G) {
  int hp = 0, ns = 0;
  bool ok;
  if (kv == 1)
    ok = D == 128 ? decode_geometry<1, 128>(Hkv, G, hp, ns) : decode_geometry<1, 64>(Hkv, G, hp, ns);
  else
    ok = D == 128 ? decode_geometry<2, 128>(Hkv, G, hp, ns) : decode_geometry<2, 64>(Hkv, G, hp, ns);
  return ok ? hp : 0;
}

cudaError_t launch_decode(const AttnParams& p, int kv, int out_kind, int64_t max_items, int num_sms,
                          cudaStream_t st, bool pdl) {
#define PKV_DEC(KV, D) \
  (out_kind ? launch_decode_t<KV, D, __nv_bfloat16>(p, max_items, num_sms, st, pdl) \
            : launch_decode_t<KV, D, float>(p, max_items, num_sms, st, pdl))
  if (kv == 1) return p.D == 128 ? PKV_DEC(1, 128) : PKV_DEC(1, 64);
  return p.D == 128 ? PKV_DEC(2, 128) : PKV_DEC(2, 64);
#undef PKV_DEC
}

}  // namespace pkv
