// pkv_kernels.h -- parameter blocks and launchers shared between the host
// side of libpkv (pkv_api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <utility>

#include "pkv.h"
#include "pkv_common.cuh"

namespace pkv {

// ---------------------------------------------------------------- append
struct AppendParams {
  const void* k;
  const void* v;
  int64_t k_st, k_sh, v_st, v_sh;  // row strides (elements) of k and v
  const void* slots;               // int32 or int64 [T]
  void* k_cache;
  void* v_cache;
  int64_t T;
  int32_t Hkv, D;
  int64_t num_slots;  // num_blocks * block_size
  float k_inv_scale, v_inv_scale;
  unsigned int* err;
};

cudaError_t launch_slot_mapping(const int32_t* cu_q, const int32_t* seq_lens, const int32_t* bt,
                                int64_t bt_stride, int32_t max_blocks, int32_t B, int32_t bs, void* slots,
                                bool slots_i64, int64_t T, unsigned int* err, cudaStream_t stream);

cudaError_t launch_csr_tables(const int32_t* indptr, const int32_t* indices, int64_t nnz, int32_t* bt,
                              int64_t bt_stride, int32_t max_blocks, int32_t B, unsigned int* err,
                              cudaStream_t stream);

// src_kind: 0 = f32 rows, 1 = bf16 rows.
cudaError_t launch_append(const AppendParams& p, int src_kind, bool fp8, bool slots_i64,
                          cudaStream_t stream);

// ---------------------------------------------------------------- attention
// Device workspace of one attention call (all offsets 256-byte aligned).
// One decode unit: a logical chunk of one sequence (all KV heads share it).
struct DecodeDesc {
  int32_t s;        // sequence
  int32_t k0, k1;   // keys k0 .. k1-1
  int32_t t;        // packed row of the sequence's query token
  int32_t nchunks;  // chunks of the sequence
  int32_t u0;       // unit index of the sequence's first chunk
  int32_t c;        // chunk index
  int32_t pad;
};

// One merge item: H query heads (h0 .. h0+H-1 of head group hg's HP * G) of a
// split sequence, each merged by R consumer warps over R ranges of its
// nchunks chunks (H * R = HP), the R partial merges then combined in shared
// memory.
struct MergeDesc {
  int32_t s;        // sequence
  int32_t hg;       // head group
  int32_t h0;       // first query head of the item within the group
  int32_t hr;       // H | (R << 8)
  int32_t nchunks;  // chunks of the sequence
  int32_t u0;       // unit of its first chunk
  int32_t t;        // packed row of its query token
  int32_t pad;
};

// One prefill tile: 64 consecutive (token, head-of-group) rows of a sequence.
struct PrefillDesc {
  int32_t s;
  int32_t t0;       // packed row of the sequence's first query token
  int32_t q_s, n;   // query rows and keys of the sequence
  int32_t r0, r1;   // rows r0 .. r1-1 of q_s * G
  int32_t kv_end;   // keys 0 .. kv_end-1 are visible to some row
  int32_t pad;
};

struct Workspace {
  int32_t* dec_off;      // [B+1] prefix sums of decode chunk units (unit u0 + c = chunk c)
  int32_t* pf_off;       // [B+1] prefix sums of prefill row tiles
  // Claim counters.  Every run of a plan claims exactly as many decode
  // items (prefill units) as the plan lists, one claim per item processed,
  // so at the start of the k-th run after the plan a counter holds k times
  // that number: a claim c names item c mod n of run c / n, and no run has
  // to reset anything when it ends.  The plan zeroes them.
  unsigned long long* work;     // [1] decode item claims
  unsigned long long* pf_work;  // [1] tensor-core prefill unit claims
  int32_t* n_merge;      // [1] merge items
  int32_t* pf_ctas;      // [1] CTAs the tensor-core prefill runs on beside the decode kernel
  int32_t* sig;          // [kPlanSig] what the plan was made for (plan_signature)
  MergeDesc* merge_desc;  // [B * Hq] merge items, in sequence order
  int32_t* done;         // [B * Hkv] finished chunks per (sequence, head group), summed over runs
  DecodeDesc* dec_desc;  // [B * max_chunks] decode work: full chunks first, then ragged tails
  PrefillDesc* pf_desc;  // [max prefill tiles] prefill tiles in order
  float* part_o;         // [B * max_chunks, Hq, D] chunk outputs (normalised)
  float* part_lse;       // [B * max_chunks, Hq] chunk log2-sum-exp2
};

struct AttnParams {
  // query rows and output
  const void* q;
  int64_t q_st, q_sh;  // strides (elements)
  void* out;
  int64_t o_st, o_sh;
  // sequences
  int64_t T;  // packed query rows (host-side count; cu_seqlens_q must stay within it)
  const int32_t* cu_q;
  const int32_t* seq_lens;
  const int32_t* bt;
  int64_t bt_stride;
  int32_t max_blocks;
  int32_t B;
  // caches [num_blocks, bs, Hkv, D]
  const void* k_cache;
  const void* v_cache;
  int64_t num_blocks;
  int32_t bs;
  int32_t bs_shift;  // log2(bs) when bs is a power of two, else -1
  int32_t Hq, Hkv, G, D;
  float qk_scale_log2;  // scale * k_scale * log2(e)
  float v_scale;        // applied to the output (e4m3 caches), else 1
  int32_t decode_max_g;  // sequences with q_s == 1 and G <= this take the decode path
  int32_t hp;            // decode: KV heads per work item (consumer warps), divides Hkv, <= 8
  int32_t ns;            // decode: stages in the staging ring
  int32_t pf_tq;         // tensor-core prefill: query tokens per tile (0: the mma.sync prefill tiles)
  int32_t path;          // prefill kernel of the call: 0 none, 1 mma.sync, 2 tensor-core (tcgen05)
  int32_t num_sms;       // SMs of the device (the plan splits them between prefill and decode)
  int32_t kv_esize;      // bytes per cache element
  int32_t dec_concurrent;  // decode kernel launched beside the tensor-core prefill (see decode_kernel)
  // variants: soft_cap > 0 turns a score s into soft_cap * tanh(s / soft_cap);
  // the kernels take x = cap_post * tanh(raw * cap_pre) in base 2, raw being
  // the q.k dot product of the stored values.  window_left >= 0: the query
  // at position p sees keys p - window_left .. p.
  float soft_cap, cap_pre, cap_post;
  int32_t window_left;
  Workspace ws;
  unsigned int* err;
};

// The shapes and choices a plan depends on, written by the plan kernel into
// the workspace and checked by every kernel of a run before it reads the
// plan's lists: a run whose call disagrees with the plan in the workspace
// does no work and records kErrPlan.
constexpr int kPlanSig = 13;
constexpr int32_t kPlanMagic = 0x504b5631;  // "PKV1"
__host__ __device__ inline void plan_signature(const AttnParams& p, int32_t (&sig)[kPlanSig]) {
  sig[0] = kPlanMagic;
  sig[1] = p.B;
  sig[2] = static_cast<int32_t>(p.T);
  sig[3] = p.Hkv;
  sig[4] = p.G;
  sig[5] = p.D;
  sig[6] = p.bs;
  sig[7] = p.max_blocks;
  sig[8] = p.pf_tq;
  sig[9] = p.path;
  sig[10] = p.window_left;
  sig[11] = p.decode_max_g;
  sig[12] = p.hp;
}

// The check by a whole warp after its dependency wait (the signature is
// written by the plan kernel and not changed by a run): lane i < kPlanSig
// compares word i, so that a warp makes kPlanSig loads, not 32 times as
// many (every CTA of a grid reads the same few words).
__device__ __forceinline__ bool plan_matches_warp(const AttnParams& p) {
  const int lane = threadIdx.x & 31;
  int32_t sig[kPlanSig];
  plan_signature(p, sig);
  int32_t want = 0;
#pragma unroll
  for (int i = 0; i < kPlanSig; ++i) want = lane == i ? sig[i] : want;
  const bool ok = lane >= kPlanSig || __ldcg(p.ws.sig + lane) == want;
  return __all_sync(0xffffffffu, ok);
}

// Launchers.  out_kind: 0 = f32, 1 = bf16.  kv: 0 = f32, 1 = bf16, 2 = e4m3.
// Prefill tiles of a call are at most ceil(T * G / 64) + B; decode chunks at
// most B * max_chunks_for(max_blocks * block_size).
size_t attention_workspace_bytes(int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t D, int64_t max_ctx);

// Launch with an optional programmatic-dependent-launch attribute (the
// kernel may start while the previous kernel of the stream finishes; it
// must call grid_dep_wait() before reading that kernel's results).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raises a kernel's dynamic shared memory limit once per device.
cudaError_t set_smem_attr(const void* kernel, size_t bytes);

cudaError_t launch_plan(const AttnParams& p, cudaStream_t st);
// KV heads per decode item (the decode kernel's consumer warps) for a
// cache format and head shape; 0 if the decode kernel cannot be built for it.
int decode_heads_per_item(int kv, int D, int Hkv, int G);
cudaError_t launch_decode(const AttnParams& p, int kv, int out_kind, int64_t max_items, int num_sms,
                          cudaStream_t st, bool pdl);

cudaError_t launch_prefill(const AttnParams& p, int kv, int out_kind, int64_t max_items, int num_sms,
                           cudaStream_t st);
cudaError_t launch_f32(const AttnParams& p, int out_kind, int64_t T, cudaStream_t st);

// Tensor-core (tcgen05) prefill: bf16 or e4m3 caches, D 64 or 128, block
// size a multiple of 8, G <= 128.
bool prefill_tc_supported(int kv, int64_t D, int64_t bs, int64_t G);
int prefill_tc_tokens_per_tile(int64_t G);
cudaError_t launch_prefill_tc(const AttnParams& p, int out_kind, int64_t max_units, int num_sms, cudaStream_t st);

// Records msg as the calling thread's pkv_last_error() and returns st.
pkv_status record_failure(pkv_status st, const std::string& msg);

}  // namespace pkv
