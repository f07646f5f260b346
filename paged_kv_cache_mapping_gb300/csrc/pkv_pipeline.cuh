// pkv_pipeline.cuh -- the producer side of the K/V staging ring shared by the
// decode and prefill kernels.
//
// A stage holds kST consecutive logical tokens of one KV head: kST K rows,
// then kST V rows, each row padded to kRowS bytes (the 16-byte pad puts 8
// consecutive rows on 8 distinct bank groups for ldmatrix).  Each row is
// fetched from its page -- block_tables[s][j / bs], offset j % bs -- with a
// 1-D bulk copy that completes on the stage's "full" mbarrier.  Rows past
// the range, and rows whose block id is out of range, are zero-filled
// instead, so they add exactly nothing to the softmax sums.
#pragma once

#include "pkv_kernels.h"

namespace pkv {

template <int kRowB, int kRowS, int kST, int kNS>
struct Ring {
  static constexpr int kStageB = 2 * kST * kRowS;

  unsigned char* base;  // generic pointer to stage 0
  uint32_t base_s;      // shared-window address of stage 0
  uint32_t full0, empty0;

  // Producer warp: fill stage number `fill` (ring slot fill % kNS) with
  // tokens j0 .. j0 + nvalid - 1 of KV head g of the sequence whose block
  // table row is bt_row.  Returns false if a wait gave up.
  __device__ __forceinline__ bool produce(const AttnParams& p, int fill, const int32_t* bt_row, int g,
                                          int j0, int nvalid, const char* kbase, const char* vbase,
                                          int lane) const {
    const int slot = fill % kNS;
    const uint32_t full = full0 + 8 * slot, empty = empty0 + 8 * slot;
    // row addresses first: the block-table loads overlap the wait below
    int64_t src[kST / 32];  // byte offset of the row in the cache, -1 = none
    uint32_t bytes = 0;
#pragma unroll
    for (int r = 0; r < kST / 32; ++r) {
      const int jj = lane + 32 * r;
      src[r] = -1;
      if (jj < nvalid) {
        const int j = j0 + jj;
        const int lb = p.bs_shift >= 0 ? (j >> p.bs_shift) : (j / p.bs);
        const int off = j - lb * p.bs;
        const int32_t blk = __ldg(bt_row + lb);
        if (blk >= 0 && blk < p.num_blocks) {
          src[r] = (((int64_t)blk * p.bs + off) * p.Hkv + g) * (int64_t)kRowB;
          bytes += 2 * kRowB;
        } else {
          atomicOr(p.err, kErrBlockRange);
        }
      }
    }
    if (!mbar_wait(empty, ((fill / kNS) & 1) ^ 1, p.err)) return false;
    const uint32_t sK = base_s + slot * kStageB, sV = sK + kST * kRowS;
    bool zeroed = false;
#pragma unroll
    for (int r = 0; r < kST / 32; ++r) {
      if (src[r] < 0) {
        const int jj = lane + 32 * r;
        uint4* zk = reinterpret_cast<uint4*>(base + slot * kStageB + jj * kRowS);
        uint4* zv = reinterpret_cast<uint4*>(base + slot * kStageB + (kST + jj) * kRowS);
#pragma unroll
        for (int i = 0; i < kRowB / 16; ++i) {
          zk[i] = make_uint4(0, 0, 0, 0);
          zv[i] = make_uint4(0, 0, 0, 0);
        }
        zeroed = true;
      }
    }
    if (__any_sync(0xffffffffu, zeroed)) fence_proxy_async_smem();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(full, bytes);
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kST / 32; ++r) {
      if (src[r] >= 0) {
        const int jj = lane + 32 * r;
        bulk_g2s(sK + jj * kRowS, kbase + src[r], kRowB, full);
        bulk_g2s(sV + jj * kRowS, vbase + src[r], kRowB, full);
      }
    }
    return true;
  }

  // Producer warp, before exit: the copies of the last stages must land
  // while the CTA still owns its shared memory.
  __device__ __forceinline__ void drain(const AttnParams& p, int fill) const {
    for (int f = fill > kNS ? fill - kNS : 0; f < fill; ++f) {
      if (!mbar_wait(full0 + 8 * (f % kNS), (f / kNS) & 1, p.err)) break;
    }
  }

  // Consumer warp: wait until stage number `cons` is full.
  __device__ __forceinline__ bool wait_full(const AttnParams& p, int cons) const {
    return mbar_wait(full0 + 8 * (cons % kNS), (cons / kNS) & 1, p.err);
  }

  // Consumer warp: hand stage number `cons` back to the producer.
  __device__ __forceinline__ void release(int cons, int lane) const {
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * (cons % kNS));
  }

  __device__ __forceinline__ uint32_t k_rows(int cons) const { return base_s + (cons % kNS) * kStageB; }
  __device__ __forceinline__ uint32_t v_rows(int cons) const { return k_rows(cons) + kST * kRowS; }
};

// Barrier set-up by thread 0, then a CTA-wide barrier.
template <int kNS>
__device__ __forceinline__ void init_ring_barriers(uint32_t full0, uint32_t empty0, int consumers) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, consumers);
    }
    fence_barrier_init();
  }
  __syncthreads();
}

}  // namespace pkv
