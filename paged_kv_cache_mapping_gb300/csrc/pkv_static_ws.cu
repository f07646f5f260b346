// pkv_static_ws.cu -- pkv_attention_static_workspace: the attention call with
// its scratch taken from a fixed array inside the library, for callers that
// cannot allocate device memory (declared in include/pkv.h).
//
// The array below is the scratch of every call on a device.  It is set up
// once per device, the first time the call runs with that device current:
// cudaGetSymbolAddress gives the array's address in that device's context,
// which is cached and handed to the unchanged pkv_attention as its
// workspace.  That first call makes runtime calls of its own, so it belongs
// before any stream capture starts.
//
// The array keeps whatever the previous call left in it.  Nothing in the
// workspace is read before the call writes it, with two exceptions -- the
// decode work counter and the per-(sequence, head group) done counters --
// and the plan kernel, which every call launches first on its stream,
// resets both before any other kernel of the call reads them.
//
// Calls whose GPU work can overlap (different streams, or host threads
// without ordering between them) share the one array and race on it.
//
// The cached address belongs to the context that was current at the first
// call on the device: the device's primary context, which the CUDA runtime
// uses.  After cudaDeviceReset, or under another context made current with
// the driver API, that address is stale; the call is not for such use.
#include <mutex>
#include <string>

#include "pkv.h"
#include "pkv_kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[PKV_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices];

pkv_status static_workspace_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return pkv::record_failure(PKV_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  }
  if (dev < 0 || dev >= kMaxDevices) return pkv::record_failure(PKV_ERR_UNSUPPORTED, "device index beyond 63");
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress((void**)&ptr, g_static_ws);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return pkv::record_failure(PKV_ERR_CUDA, std::string("cudaGetSymbolAddress(static workspace): ") +
                                                   cudaGetErrorString(e));
    }
    if ((reinterpret_cast<uintptr_t>(ptr) & 255) != 0)
      return pkv::record_failure(PKV_ERR_CUDA, "static workspace is not 256-byte aligned");
    g_static_ptr[dev] = ptr;
  }
  *out = g_static_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_attention_static_workspace(const pkv_tensor* q, const pkv_tensor* cu_seqlens_q,
                                                     const pkv_tensor* seq_lens, const pkv_tensor* block_tables,
                                                     const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                                                     float scale, float k_scale, float v_scale,
                                                     int32_t max_q_len, pkv_tensor* out, void* stream) {
  // the batch the call would run is seq_lens' B; a block table of another
  // height is the argument error pkv_attention reports, not a size error
  if (seq_lens == nullptr || seq_lens->ndim != 1 || block_tables == nullptr || block_tables->ndim != 2 ||
      block_tables->shape[0] != seq_lens->shape[0])
    return pkv::record_failure(PKV_ERR_INVALID_ARGUMENT,
                               "pkv_attention_static_workspace: seq_lens must be [B] and block_tables [B, max_blocks]");
  size_t need = 0;
  pkv_status st = pkv_attention_workspace_size(q, block_tables, k_cache, &need);
  if (st != PKV_OK) return st;
  if (need > static_cast<size_t>(PKV_STATIC_WORKSPACE_BYTES))
    return pkv::record_failure(
        PKV_ERR_WORKSPACE_TOO_SMALL,
        "pkv_attention_static_workspace: this call needs " + std::to_string(need) +
            " bytes of scratch (B = " + std::to_string(seq_lens->shape[0]) +
            ", T = " + std::to_string(q->shape[0]) + ", Hq = " + std::to_string(q->shape[1]) +
            ", max context = " + std::to_string(block_tables->shape[1] * k_cache->shape[1]) +
            " tokens) but the library's static array holds " + std::to_string(PKV_STATIC_WORKSPACE_BYTES) +
            "; use pkv_attention with a caller-provided workspace");
  void* ws = nullptr;
  st = static_workspace_address(&ws);
  if (st != PKV_OK) return st;
  return pkv_attention(q, cu_seqlens_q, seq_lens, block_tables, k_cache, v_cache, scale, k_scale, v_scale,
                       max_q_len, out, ws, PKV_STATIC_WORKSPACE_BYTES, stream);
}
