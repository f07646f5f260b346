// pkv_plan.cu -- the device-side plan of one attention call: per-sequence
// work counts, their prefix sums and the work lists of the decode and
// prefill kernels, built from the device lengths with no host round trip.
//
// Decode rows are cut into chunks whose length depends only on the
// sequence's visible key count (128 * 2^k tokens, 256 * 2^k with an e4m3
// cache, at most 512 chunks), so
// results depend neither on the batch nor on the page layout ("How Easy Is
// It to Start Serving LLMs?", "3. Load balancing": long requests are split
// into chunks and a merge step stitches them).  Prefill rows are cut into
// tiles of query tokens, the last tokens (most keys) first.
#include "pkv_pipeline.cuh"

namespace pkv {

// ---------------------------------------------------------------- plan
// Block-wide exclusive scan of K counts per thread (warp shuffles, then one
// warp over the warp totals).  off[] = the thread's offsets, totals[] = the
// block totals.
template <int K>
__device__ __forceinline__ void block_scan(const int (&v)[K], int (&off)[K], int (&totals)[K]) {
  __shared__ int wsum[32][K];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x[K];
#pragma unroll
  for (int k = 0; k < K; ++k) x[k] = v[k];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int y = __shfl_up_sync(0xffffffffu, x[k], o);
      if (lane >= o) x[k] += y;
    }
  }
  if (lane == 31)
#pragma unroll
    for (int k = 0; k < K; ++k) wsum[warp][k] = x[k];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      int y = lane < nw ? wsum[lane][k] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int z = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) y += z;
      }
      if (lane < nw) wsum[lane][k] = y;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    off[k] = x[k] - v[k] + (warp > 0 ? wsum[warp - 1][k] : 0);
    totals[k] = wsum[nw - 1][k];
  }
}

// Smallest decode chunk (as a shift): a chunk of an e4m3 cache holds twice
// the tokens, so that its bytes, and the work an item carries against its
// fixed costs (descriptor, query rows, partial result), stay the same.
__device__ __forceinline__ int decode_chunk_base(const AttnParams& p) {
  return p.kv_esize == 1 ? kChunkBaseShiftFp8 : kChunkBaseShift;
}

// First key a decoding query (position n - 1) sees.
__device__ __forceinline__ int decode_first_key(const AttnParams& p, int n) {
  return p.window_left >= 0 && n - 1 - p.window_left > 0 ? n - 1 - p.window_left : 0;
}

// Work counts of sequence s: decode chunks (all, full, ragged last) or
// prefill tiles.  Inconsistent lengths give no work (and are recorded).
struct SeqCounts {
  int dec, full, tail, pf;  // decode chunks (all, full, ragged last), prefill tiles
  int n, t0, q_s;           // the lengths they came from
  int cls;                  // size class of the decode chunks (0: the smallest chunk)
  int mi;                   // merge items (split sequences)
};

// How the merge of a sequence of n chunks is cut: R consumer warps (a
// divisor of HP) share each query head, each merging at most 64 chunks where
// it can, so an item carries H = HP / R heads.  Depends on n and HP only.
__device__ __forceinline__ void merge_split(int n, int hp, int& H, int& R) {
  R = hp;
  for (int r = 1; r <= hp; ++r) {
    if (hp % r == 0 && 64 * r >= n) {
      R = r;
      break;
    }
  }
  H = hp / R;
}

// The full chunks of the decode list are ordered by size, the largest first
// (sequences of one size in order), so that the longest items start first.
constexpr int kChunkClasses = 16;

__device__ __forceinline__ SeqCounts seq_counts(const AttnParams& p, int s, bool record) {
  // L2 loads: the lengths may have been written by the previous kernel
  const int c0 = __ldcg(p.cu_q + s), c1 = __ldcg(p.cu_q + s + 1);
  const int q_s = c1 - c0;
  const int n = __ldcg(p.seq_lens + s);
  SeqCounts c{0, 0, 0, 0, n, c0, q_s, 0, 0};
  if (q_s == 0) return c;
  if (q_s < 0 || q_s > n || (int64_t)n > (int64_t)p.max_blocks * p.bs || c0 < 0 || c1 > p.T) {
    if (record) atomicOr(p.err, kErrLengths);
    return c;
  }
  if (q_s == 1 && p.G <= p.decode_max_g) {
    // the visible keys [lo, n) are cut into chunks of 2^k from lo
    const int lo = decode_first_key(p, n);
    const int k = chunk_shift(n - lo, decode_chunk_base(p));
    c.dec = (int)(((unsigned)(n - lo) + (1u << k) - 1u) >> k);
    c.full = (n - lo) >> k;
    c.tail = c.dec - c.full;
    c.cls = min(k - decode_chunk_base(p), kChunkClasses - 1);
    if (c.dec > 1) {
      int H, R;
      merge_split(c.dec, p.hp, H, R);
      c.mi = (p.Hkv / p.hp) * R * p.G;
    }
  } else {
    c.pf = p.pf_tq > 0 ? (q_s + p.pf_tq - 1) / p.pf_tq
                       : (int)(((int64_t)q_s * p.G + kPrefillRows - 1) / kPrefillRows);
  }
  return c;
}

// Descriptor of decode chunk ch of sequence s: off0 is the sequence's first
// entry in the per-sequence chunk numbering, off1 / off2 its first full /
// ragged chunk in the work list, where all full chunks (tot_full of them)
// come before the ragged ones.
__device__ __forceinline__ void write_dec_desc(const AttnParams& p, int s, const SeqCounts& c, int off0, int off1,
                                               int off2, int tot_full, int ch) {
  const int first = decode_first_key(p, c.n);
  const int k = chunk_shift(c.n - first, decode_chunk_base(p));
  const int k0 = first + (ch << k);
  int4* dst = reinterpret_cast<int4*>(p.ws.dec_desc + (ch < c.full ? off1 + ch : tot_full + off2));
  dst[0] = make_int4(s, k0, min(k0 + (1 << k), c.n), c.t0);
  dst[1] = make_int4(c.dec, off0, ch, 0);
}

// Descriptor of merge item k of split sequence s (its items start at off4):
// head group k / (R G), heads (k mod R G) * H .. + H - 1 of the group.
__device__ __forceinline__ void write_merge_desc(const AttnParams& p, int s, const SeqCounts& c, int off0, int off4,
                                                 int k) {
  int H, R;
  merge_split(c.dec, p.hp, H, R);
  const int per = R * p.G;
  int4* dst = reinterpret_cast<int4*>(p.ws.merge_desc + off4 + k);
  dst[0] = make_int4(s, k / per, (k % per) * H, H | (R << 8));
  dst[1] = make_int4(c.dec, off0, c.t0, 0);
}

// Descriptor of prefill tile qt of sequence s (its tiles start at off3).
__device__ __forceinline__ void write_pf_desc(const AttnParams& p, int s, const SeqCounts& c, int off3, int qt) {
  int4* dst = reinterpret_cast<int4*>(p.ws.pf_desc + off3 + qt);
  dst[0] = make_int4(s, c.t0, c.q_s, c.n);
  if (p.pf_tq > 0) {  // query tokens r0 .. r1-1, the last tokens (most keys) first
    const int r1 = c.q_s - qt * p.pf_tq, r0 = max(0, r1 - p.pf_tq);
    dst[1] = make_int4(r0, r1, c.n - c.q_s + r1, 0);
  } else {  // (token, head) rows r0 .. r1-1
    const int r0 = qt * kPrefillRows, r1 = min(r0 + kPrefillRows, c.q_s * p.G);
    dst[1] = make_int4(r0, r1, c.n - c.q_s + (r1 - 1) / p.G + 1, 0);
  }
}

// Batches up to this size write their lists one warp per sequence (one lane
// per chunk or tile); larger ones one thread per sequence.
constexpr int kPlanSeqs = 512;

// Key tiles (of the tensor-core prefill's 128 keys) that the prefill units
// of sequence s cover, summed over its query tiles.
__device__ __forceinline__ long long prefill_key_tiles(const AttnParams& p, const SeqCounts& c) {
  long long n = 0;
  for (int qt = 0; qt < c.pf; ++qt) {
    const int r1 = c.q_s - qt * p.pf_tq, r0 = max(0, r1 - p.pf_tq);
    const int kv_end = c.n - c.q_s + r1;
    const int first = p.window_left >= 0 ? max(0, c.n - c.q_s + r0 - p.window_left) : 0;
    n += (kv_end + 127) / 128 - first / 128;
  }
  return n;
}

// Measured rates on GB300 (sm_103a) that split the SMs of a call between the
// tensor-core prefill and the decode kernel running beside it: a prefill
// unit costs about kPfTileUs per 128-key tile (D = 128; half at D = 64)
// plus kPfUnitUs of start and epilogue, a decode CTA streams about
// kDecSmBytesPerUs of K/V (bf16; kDecSmBytesPerUsFp8 with an e4m3 cache,
// whose consumers do more work per byte), and all of them together at most
// kHbmBytesPerUs.
constexpr float kPfTileUs = 1.3f;
constexpr float kPfUnitUs = 3.5f;
constexpr float kDecSmBytesPerUs = 55e3f;
constexpr float kDecSmBytesPerUsFp8 = 45e3f;
constexpr float kHbmBytesPerUs = 6.0e6f;

// Prefill CTAs for a call with the given prefill key tiles (per KV head) and
// decode bytes: the split that gives the two kernels the shortest common
// time.  Called by a whole warp; lane l tries l + 1, l + 33, ..
__device__ inline int prefill_cta_split(const AttnParams& p, long long pf_tiles, int pf_units,
                                        long long dec_bytes) {
  const int S = p.num_sms, lane = threadIdx.x & 31;
  if (dec_bytes == 0 || S < 2) return S;
  const float pf = (float)pf_tiles * (float)p.Hkv * kPfTileUs * (p.D / 128.f) + (float)pf_units * kPfUnitUs;
  const float rate = p.kv_esize == 1 ? kDecSmBytesPerUsFp8 : kDecSmBytesPerUs;
  const float dec = (float)dec_bytes / rate, hbm = (float)dec_bytes / kHbmBytesPerUs;
  int best = S;
  float best_t = INFINITY;
  for (int P = lane + 1; P < S; P += 32) {
    const float t = fmaxf(__fdividef(pf, (float)P), fmaxf(__fdividef(dec, (float)(S - P)), hbm));
    if (t < best_t) {
      best_t = t;
      best = P;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {  // the smallest time, the fewest CTAs on a tie
    const float ot = __shfl_xor_sync(0xffffffffu, best_t, o);
    const int op = __shfl_xor_sync(0xffffffffu, best, o);
    if (ot < best_t || (ot == best_t && op < best)) {
      best_t = ot;
      best = op;
    }
  }
  return best;
}

// One block: per-sequence work counts and their prefix sums, the decode
// work list (every full chunk first, the largest chunks first, then the
// ragged last chunks, so that the small pieces come last), the list of split sequences, the prefill
// tile list, the claim and done counters of the runs zeroed, and the
// plan's signature.  Reads device lengths; no host round trip.  A plan
// serves any number of runs (one per layer) over the same lengths: the
// counters run on from one run to the next (see Workspace).
__global__ void __launch_bounds__(1024) plan_kernel(AttnParams p) {
  launch_dependents();  // the next kernel may start its set-up now
  // launched with programmatic dependent launch: the lengths may come from
  // the previous kernel, and the workspace may still be read by the previous
  // run's kernels until that kernel has completed
  grid_dep_wait();
  const int tid = threadIdx.x, nth = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nth >> 5;
  const int B = p.B;
  const int per = (B + nth - 1) / nth;
  const int s0 = min(tid * per, B), s1 = min(s0 + per, B);
  // First pass, counts and their prefix sums; with the tensor-core prefill,
  // also the work that decides how the SMs are split between the kernels
  __shared__ unsigned long long s_pf_tiles, s_dec_keys;
  if (tid == 0) s_pf_tiles = s_dec_keys = 0ull;
  __syncthreads();
  SeqCounts first{};  // the thread's first sequence, kept for the second pass
  int sum[5] = {0, 0, 0, 0, 0};
  int cls[kChunkClasses];  // full chunks per size class
#pragma unroll
  for (int j = 0; j < kChunkClasses; ++j) cls[j] = 0;
  long long pf_tiles = 0, dec_keys = 0;
  for (int s = s0; s < s1; ++s) {
    const SeqCounts c = seq_counts(p, s, true);
    if (s == s0) first = c;
#pragma unroll
    for (int j = 0; j < kChunkClasses; ++j) cls[j] += j == c.cls ? c.full : 0;
    sum[0] += c.dec;
    sum[1] += c.full;
    sum[2] += c.tail;
    sum[3] += c.pf;
    sum[4] += c.mi;
    if (p.path == 2) {
      pf_tiles += prefill_key_tiles(p, c);
      if (c.dec > 0) dec_keys += c.n - decode_first_key(p, c.n);
    }
  }
  if (p.path == 2) {
    atomicAdd(&s_pf_tiles, (unsigned long long)pf_tiles);
    atomicAdd(&s_dec_keys, (unsigned long long)dec_keys);
  }
  int off[5], tot[5];
  block_scan<5>(sum, off, tot);  // its barriers order the additions above
  // full chunks: class j starts after every larger class.  When every
  // sequence's chunks have one size (the usual case), that is the order of
  // the sequences, which the scan above already gives.
  int cls_off[kChunkClasses], cls_tot[kChunkClasses];
  bool one_class = true;
#pragma unroll
  for (int j = 1; j < kChunkClasses; ++j) one_class = one_class && cls[j] == 0;
  if (__syncthreads_and(one_class)) {
#pragma unroll
    for (int j = 0; j < kChunkClasses; ++j) cls_off[j] = j == 0 ? off[1] : 0;
  } else {
    block_scan<kChunkClasses>(cls, cls_off, cls_tot);
    int base = 0;
#pragma unroll
    for (int j = kChunkClasses - 1; j >= 0; --j) {
      cls_off[j] += base;
      base += cls_tot[j];
    }
  }
  __shared__ int4 sq_cnt[kPlanSeqs];  // dec, full, pf, n
  __shared__ int4 sq_off[kPlanSeqs];  // off[0..3]
  __shared__ int4 sq_len[kPlanSeqs];  // t0, q_s, mi, off[4]
  const bool by_warp = B <= kPlanSeqs;
  for (int s = s0; s < s1; ++s) {
    const SeqCounts c = s == s0 ? first : seq_counts(p, s, false);
    p.ws.dec_off[s] = off[0];
    p.ws.pf_off[s] = off[3];
    int full_off = 0;  // the sequence's first full chunk in the list
#pragma unroll
    for (int j = 0; j < kChunkClasses; ++j) {
      if (j == c.cls) {
        full_off = cls_off[j];
        cls_off[j] += c.full;
      }
    }
    if (by_warp) {
      sq_cnt[s] = make_int4(c.dec, c.full, c.pf, c.n);
      sq_off[s] = make_int4(off[0], full_off, off[2], off[3]);
      sq_len[s] = make_int4(c.t0, c.q_s, c.mi, off[4]);
    } else {
      for (int ch = 0; ch < c.dec; ++ch) write_dec_desc(p, s, c, off[0], full_off, off[2], tot[1], ch);
      for (int qt = 0; qt < c.pf; ++qt) write_pf_desc(p, s, c, off[3], qt);
      for (int k = 0; k < c.mi; ++k) write_merge_desc(p, s, c, off[0], off[4], k);
    }
    off[0] += c.dec;
    off[1] += c.full;
    off[2] += c.tail;
    off[3] += c.pf;
    off[4] += c.mi;
  }
  if (by_warp) {
    __syncthreads();
    for (int s = warp; s < B; s += nw) {
      const int4 cn = sq_cnt[s], of = sq_off[s];
      const int4 ln = sq_len[s];
      const SeqCounts c{cn.x, cn.y, cn.x - cn.y, cn.z, cn.w, ln.x, ln.y, 0, ln.z};
      for (int ch = lane; ch < c.dec; ch += 32) write_dec_desc(p, s, c, of.x, of.y, of.z, tot[1], ch);
      for (int qt = lane; qt < c.pf; qt += 32) write_pf_desc(p, s, c, of.w, qt);
      for (int k = lane; k < c.mi; k += 32) write_merge_desc(p, s, c, of.x, ln.w, k);
    }
  }
  if (warp == 0) {
    const int pf_ctas = p.path == 2 ? prefill_cta_split(p, (long long)s_pf_tiles, tot[3] * p.Hkv,
                                                        (long long)s_dec_keys * p.Hkv * p.D * p.kv_esize * 2)
                                    : p.num_sms;
    if (lane == 0) {
      p.ws.dec_off[B] = tot[0];
      p.ws.pf_off[B] = tot[3];
      *p.ws.work = 0ull;
      *p.ws.pf_work = 0ull;
      *p.ws.n_merge = tot[4];
      *p.ws.pf_ctas = pf_ctas;
    }
  }
  if (tid < kPlanSig) {
    int32_t sig[kPlanSig];
    plan_signature(p, sig);
    p.ws.sig[tid] = sig[tid];
  }
  for (int i = tid; i < B * p.Hkv; i += nth) p.ws.done[i] = 0;
}

cudaError_t launch_plan(const AttnParams& p, cudaStream_t st) {
  return launch_ex(plan_kernel, dim3(1), dim3(1024), 0, st, true, p);
}

}  // namespace pkv
