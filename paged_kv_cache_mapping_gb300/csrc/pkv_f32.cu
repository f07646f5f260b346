// pkv_f32.cu -- paged attention for fp32 queries and fp32 caches.
//
// The same computation as the tensor-core kernels -- causal GQA attention of
// each packed query row over its sequence's pages, the pages reached through
// the block table ("How to design an LLM serving system (a vLLM deep dive)",
// "PagedAttention (vLLM KV manager)"; nanoserve, "Architecture" step 3) --
// for the fp32 variant, on the CUDA cores in fp32 with an online softmax.
// One CTA per (query token, KV head); warp w serves query heads w, w+4, ...
// of the group, each lane holding D/32 elements of q and of the output.
#include "pkv_kernels.h"

namespace pkv {

template <typename OutT>
__global__ void __launch_bounds__(128) f32_attention_kernel(AttnParams p, int64_t T) {
  const int64_t t = blockIdx.x;
  const int g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = __ldg(p.cu_q + p.B);
  if (t >= total) return;
  const int s = upper_index(p.cu_q, p.B, static_cast<int>(t));
  const int c0 = __ldg(p.cu_q + s);
  const int q_s = __ldg(p.cu_q + s + 1) - c0;
  const int n = __ldg(p.seq_lens + s);
  if (q_s < 0 || q_s > n || (int64_t)n > (int64_t)p.max_blocks * p.bs || t < c0 || t - c0 >= q_s) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrLengths);
    return;
  }
  const int pos = n - q_s + static_cast<int>(t - __ldg(p.cu_q + s));
  const int per = p.D / 32;  // elements per lane, <= 8
  const float* kc = static_cast<const float*>(p.k_cache);
  const float* vc = static_cast<const float*>(p.v_cache);
  const int32_t* bt_row = p.bt + (int64_t)s * p.bt_stride;
  for (int hh = warp; hh < p.G; hh += blockDim.x >> 5) {
    const int h = g * p.G + hh;
    const float* qrow = static_cast<const float*>(p.q) + t * p.q_st + (int64_t)h * p.q_sh;
    float qv[8], o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      qv[k] = k < per ? qrow[lane + 32 * k] : 0.f;
      o[k] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j <= pos; ++j) {
      const int lb = p.bs_shift >= 0 ? (j >> p.bs_shift) : (j / p.bs);
      const int32_t blk = __ldg(bt_row + lb);
      if (blk < 0 || blk >= p.num_blocks) {
        if (lane == 0) atomicOr(p.err, kErrBlockRange);
        continue;
      }
      const int64_t row = (((int64_t)blk * p.bs + (j - lb * p.bs)) * p.Hkv + g) * p.D;
      float dot = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < per) dot = fmaf(qv[k], __ldg(kc + row + lane + 32 * k), dot);
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o2);
      const float x = dot * p.qk_scale_log2;
      const float mn = fmaxf(m, x);
      const float alpha = exp2f(m - mn), w = exp2f(x - mn);
      l = l * alpha + w;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < per) o[k] = fmaf(w, __ldg(vc + row + lane + 32 * k), o[k] * alpha);
      m = mn;
    }
    OutT* orow = static_cast<OutT*>(p.out) + t * p.o_st + (int64_t)h * p.o_sh;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < per) store1(orow + lane + 32 * k, o[k] / l);
  }
}

cudaError_t launch_f32(const AttnParams& p, int out_kind, int64_t T, cudaStream_t st) {
  if (T == 0 || p.Hkv == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(T), static_cast<unsigned>(p.Hkv));
  if (out_kind)
    f32_attention_kernel<__nv_bfloat16><<<grid, 128, 0, st>>>(p, T);
  else
    f32_attention_kernel<float><<<grid, 128, 0, st>>>(p, T);
  return cudaGetLastError();
}

}  // namespace pkv
