// pkv_append.cu -- slot computation and the slot-mapped KV append.
//
// Slot computation: nanoserve, "Architecture", step 2 ("Prepare": each new
// token's cache slot is computed from its block table); "How to design an
// LLM serving system (a vLLM deep dive)", "PagedAttention (vLLM KV manager)"
// (block table, slot_mapping).  slot = table[p / bs] * bs + p % bs for the
// token at position p = N_s - q_s + i.
//
// Append: nanoserve, "Architecture", step 3 ("Forward": each layer writes
// this step's K/V into the paged cache before attending).  One warp moves
// one (token, KV head) row of K and of V with 16-byte loads; the cache row
// of slot s for head h starts at element (s * Hkv + h) * D.  An e4m3 cache
// stores cvt.rn.satfinite(x * inv_scale) with the product in fp32 ("How Easy
// Is It to Start Serving LLMs?", "What each setting does to performance").
#include "pkv_kernels.h"

namespace pkv {

template <typename SlotT>
__global__ void slot_mapping_kernel(const int32_t* __restrict__ cu_q, const int32_t* __restrict__ seq_lens,
                                    const int32_t* __restrict__ bt, int64_t bt_stride, int32_t max_blocks,
                                    int32_t B, int32_t bs, SlotT* __restrict__ slots, int64_t T,
                                    unsigned int* err) {
  // launched with programmatic dependent launch: let the next kernel set up,
  // then wait for the previous one (every thread, before any early return,
  // so that this grid completes only after its predecessor)
  launch_dependents();
  grid_dep_wait();
  int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int32_t total = __ldg(cu_q + B);
  SlotT slot = -1;
  if (t < total) {
    const int s = upper_index(cu_q, B, static_cast<int>(t));
    const int32_t c0 = __ldg(cu_q + s);
    const int32_t q_s = __ldg(cu_q + s + 1) - c0;
    const int32_t n_s = __ldg(seq_lens + s);
    if (q_s < 0 || q_s > n_s || (int64_t)n_s > (int64_t)max_blocks * bs || t < c0 || t - c0 >= q_s) {
      atomicOr(err, kErrLengths);
    } else {
      const int64_t p = (int64_t)n_s - q_s + (t - c0);
      const int32_t blk = __ldg(bt + s * bt_stride + p / bs);
      if (blk < 0) {
        atomicOr(err, kErrBlockRange);
      } else {
        slot = static_cast<SlotT>((int64_t)blk * bs + p % bs);
      }
    }
  } else {
    atomicOr(err, kErrLengths);  // T disagrees with cu_seqlens_q[B]
  }
  slots[t] = slot;
}

// ---------------------------------------------------------------- append
// Elements per 16-byte source vector.
template <typename SrcT> struct Vec16;
template <> struct Vec16<float> { static constexpr int n = 4; };
template <> struct Vec16<__nv_bfloat16> { static constexpr int n = 8; };

__device__ __forceinline__ void store_vec(float* dst, uint4 v) { *reinterpret_cast<uint4*>(dst) = v; }
__device__ __forceinline__ void store_vec(__nv_bfloat16* dst, uint4 v) { *reinterpret_cast<uint4*>(dst) = v; }

// 8 bf16 -> 8 e4m3 codes (8 bytes) of x * inv_scale.
__device__ __forceinline__ uint2 quant8(uint4 v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint16_t a = f32x2_to_e4m3x2(bf16_lo(w[2 * i]) * inv, bf16_hi(w[2 * i]) * inv);
    const uint16_t b = f32x2_to_e4m3x2(bf16_lo(w[2 * i + 1]) * inv, bf16_hi(w[2 * i + 1]) * inv);
    o[i] = static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
  }
  return make_uint2(o[0], o[1]);
}

// 4 f32 -> 4 e4m3 codes (4 bytes).
__device__ __forceinline__ uint32_t quant4(uint4 v, float inv) {
  const uint16_t a = f32x2_to_e4m3x2(__uint_as_float(v.x) * inv, __uint_as_float(v.y) * inv);
  const uint16_t b = f32x2_to_e4m3x2(__uint_as_float(v.z) * inv, __uint_as_float(v.w) * inv);
  return static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
}

// One warp per (token, KV head) row; lanes split the K row and the V row
// into 16-byte source vectors.
template <typename SrcT, bool kFp8, typename SlotT>
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
  launch_dependents();  // as in slot_mapping_kernel
  grid_dep_wait();
  constexpr int kVec = Vec16<SrcT>::n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x * (int64_t)(blockDim.x >> 5) + warp;
  if (row >= p.T * p.Hkv) return;
  const int64_t t = row / p.Hkv;
  const int h = static_cast<int>(row - t * p.Hkv);
  const int64_t slot = static_cast<int64_t>(reinterpret_cast<const SlotT*>(p.slots)[t]);
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (lane == 0) atomicOr(p.err, kErrSlotRange);
    return;
  }
  const int vecs = p.D / kVec;  // vectors per row
  for (int c = lane; c < 2 * vecs; c += 32) {
    const bool is_v = c >= vecs;
    const int e = (is_v ? c - vecs : c) * kVec;  // element offset in the row
    const SrcT* src = reinterpret_cast<const SrcT*>(is_v ? p.v : p.k) +
                      t * (is_v ? p.v_st : p.k_st) + h * (is_v ? p.v_sh : p.k_sh) + e;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(src));
    const int64_t dst_el = (slot * p.Hkv + h) * p.D + e;
    if constexpr (kFp8) {
      uint8_t* dst = reinterpret_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache) + dst_el;
      const float inv = is_v ? p.v_inv_scale : p.k_inv_scale;
      if constexpr (kVec == 8) {
        *reinterpret_cast<uint2*>(dst) = quant8(x, inv);
      } else {
        *reinterpret_cast<uint32_t*>(dst) = quant4(x, inv);
      }
    } else {
      store_vec(reinterpret_cast<SrcT*>(is_v ? p.v_cache : p.k_cache) + dst_el, x);
    }
  }
}

// Block tables from the CSR page-list form: request b reads the pages
// kv_indices[kv_indptr[b] .. kv_indptr[b+1]-1] in order ("How Easy Is It to
// Start Serving LLMs?", "1. Block-sparse KV memory").  One block per request
// row; a bad row (decreasing or out-of-range offsets, more pages than
// max_blocks) is filled with -1 and recorded.
__global__ void __launch_bounds__(128) csr_tables_kernel(const int32_t* __restrict__ indptr,
                                                         const int32_t* __restrict__ indices, int64_t nnz,
                                                         int32_t* __restrict__ bt, int64_t bt_stride,
                                                         int32_t max_blocks, int32_t B, unsigned int* err) {
  launch_dependents();
  grid_dep_wait();
  const int b = blockIdx.x;
  if (b >= B) return;
  const int32_t a0 = __ldg(indptr + b), a1 = __ldg(indptr + b + 1);
  const bool bad = a0 < 0 || a1 < a0 || (int64_t)a1 > nnz || a1 - a0 > max_blocks;
  if (bad && threadIdx.x == 0) atomicOr(err, kErrLengths);
  int32_t* row = bt + (int64_t)b * bt_stride;
  const int32_t n = bad ? 0 : a1 - a0;
  for (int i = threadIdx.x; i < max_blocks; i += blockDim.x) row[i] = i < n ? __ldg(indices + a0 + i) : -1;
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_slot_mapping(const int32_t* cu_q, const int32_t* seq_lens, const int32_t* bt,
                                int64_t bt_stride, int32_t max_blocks, int32_t B, int32_t bs, void* slots,
                                bool slots_i64, int64_t T, unsigned int* err, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = static_cast<unsigned>((T + threads - 1) / threads);
  if (slots_i64)
    return launch_ex(slot_mapping_kernel<int64_t>, dim3(blocks), dim3(threads), 0, stream, true, cu_q, seq_lens, bt,
                     bt_stride, max_blocks, B, bs, static_cast<int64_t*>(slots), T, err);
  return launch_ex(slot_mapping_kernel<int32_t>, dim3(blocks), dim3(threads), 0, stream, true, cu_q, seq_lens, bt,
                   bt_stride, max_blocks, B, bs, static_cast<int32_t*>(slots), T, err);
}

cudaError_t launch_csr_tables(const int32_t* indptr, const int32_t* indices, int64_t nnz, int32_t* bt,
                              int64_t bt_stride, int32_t max_blocks, int32_t B, unsigned int* err,
                              cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  return launch_ex(csr_tables_kernel, dim3((unsigned)B), dim3(128), 0, stream, true, indptr, indices, nnz, bt,
                   bt_stride, max_blocks, B, err);
}

cudaError_t launch_append(const AppendParams& p, int src_kind, bool fp8, bool slots_i64,
                          cudaStream_t stream) {
  const int64_t rows = p.T * p.Hkv;
  if (rows == 0) return cudaSuccess;
  const int threads = 256, rows_per_block = threads / 32;
  const unsigned blocks = static_cast<unsigned>((rows + rows_per_block - 1) / rows_per_block);
#define PKV_APPEND(SRC, FP8, SLOT) \
  return launch_ex(append_kernel<SRC, FP8, SLOT>, dim3(blocks), dim3(threads), 0, stream, true, p)
  if (src_kind == 0) {  // f32 rows
    if (fp8) {
      if (slots_i64) PKV_APPEND(float, true, int64_t); else PKV_APPEND(float, true, int32_t);
    } else {
      if (slots_i64) PKV_APPEND(float, false, int64_t); else PKV_APPEND(float, false, int32_t);
    }
  } else {  // bf16 rows
    if (fp8) {
      if (slots_i64) PKV_APPEND(__nv_bfloat16, true, int64_t); else PKV_APPEND(__nv_bfloat16, true, int32_t);
    } else {
      if (slots_i64) PKV_APPEND(__nv_bfloat16, false, int64_t); else PKV_APPEND(__nv_bfloat16, false, int32_t);
    }
  }
#undef PKV_APPEND
  return cudaGetLastError();
}

}  // namespace pkv
