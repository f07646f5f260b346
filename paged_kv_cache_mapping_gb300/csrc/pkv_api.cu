// pkv_api.cu -- the C ABI of libpkv.so (declared in include/pkv.h): host-side
// validation of every tensor, the launch plan, and status reporting.
//
// The library allocates no device memory: the caller passes the caches, the
// outputs and the attention workspace.  Its one piece of static device
// state is the error word below, which the kernels OR bits into when they
// meet an out-of-range index instead of faulting.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>

#include "pkv.h"
#include "pkv_kernels.h"

namespace {

__device__ unsigned int g_pkv_error_word;

thread_local std::string t_last_error;

pkv_status fail(pkv_status st, const std::string& msg) {
  t_last_error = msg;
  return st;
}

pkv_status cuda_fail(cudaError_t e, const char* where) {
  cudaGetLastError();  // clear a sticky launch error of this thread
  return fail(PKV_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_err_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];
std::atomic<uint64_t> g_attr_set_mask[256];  // per kernel slot: devices configured

bool check_mode() {
  static const bool on = [] {
    const char* v = getenv("PKV_CHECK");
    return v != nullptr && v[0] != '\0' && strcmp(v, "0") != 0;
  }();
  return on;
}

// Per-device address of the error word and the SM count, with that device
// current.  cudaGetSymbolAddress gives the device address of the __device__
// variable in the current device's context.
pkv_status device_state(unsigned int** err, int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device index beyond 63");
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_pkv_error_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    g_num_sms[dev] = sms;
    g_err_ptr[dev] = static_cast<unsigned int*>(ptr);
  }
  *err = g_err_ptr[dev];
  *num_sms = g_num_sms[dev];
  return PKV_OK;
}

// After the launches of a call: in check mode, wait for the stream and turn
// a recorded device error into a status.
pkv_status finish(cudaStream_t st, const char* what) {
  if (!check_mode()) return PKV_OK;
  uint32_t flags = 0;
  pkv_status s = pkv_device_errors(st, &flags);
  if (s != PKV_OK) return s;
  if (flags)
    return fail(PKV_ERR_DEVICE_CHECK,
                std::string(what) + ": device check failed, flags 0x" + std::to_string(flags) +
                    " (1 slot range, 2 block id range, 4 lengths, 8 wait timeout, 16 no matching plan)");
  return PKV_OK;
}

// ---------------------------------------------------------------- validation
const char* dtype_name(pkv_dtype d) {
  switch (d) {
    case PKV_F32: return "f32";
    case PKV_BF16: return "bf16";
    case PKV_FP8_E4M3: return "fp8_e4m3";
    case PKV_I32: return "i32";
    case PKV_I64: return "i64";
  }
  return "?";
}

int esize(pkv_dtype d) {
  switch (d) {
    case PKV_F32: return 4;
    case PKV_BF16: return 2;
    case PKV_FP8_E4M3: return 1;
    case PKV_I32: return 4;
    case PKV_I64: return 8;
  }
  return 0;
}

std::string describe(const char* name, const pkv_tensor* t) {
  std::string s = std::string(name) + " (" + dtype_name(t->dtype) + ", shape [";
  for (int i = 0; i < t->ndim; ++i) s += (i ? ", " : "") + std::to_string(t->shape[i]);
  return s + "])";
}

pkv_status need(bool ok, const std::string& msg) {
  return ok ? PKV_OK : fail(PKV_ERR_INVALID_ARGUMENT, msg);
}

#define PKV_TRY(expr)                 \
  do {                                \
    pkv_status _s = (expr);           \
    if (_s != PKV_OK) return _s;      \
  } while (0)

pkv_status check_tensor(const char* name, const pkv_tensor* t, int ndim) {
  if (t == nullptr) return fail(PKV_ERR_INVALID_ARGUMENT, std::string(name) + " is NULL");
  if (t->ndim != ndim)
    return fail(PKV_ERR_INVALID_ARGUMENT,
                describe(name, t) + ": expected " + std::to_string(ndim) + " dimensions");
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0) return fail(PKV_ERR_INVALID_ARGUMENT, describe(name, t) + ": negative extent");
  int64_t n = 1;
  for (int i = 0; i < ndim; ++i) n *= t->shape[i];
  if (n > 0 && t->data == nullptr) return fail(PKV_ERR_INVALID_ARGUMENT, std::string(name) + ": data is NULL");
  return PKV_OK;
}

bool contiguous(const pkv_tensor* t) {
  int64_t expect = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] != 1 && t->stride[i] != expect) return false;
    expect *= t->shape[i];
  }
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pkv_status check_vector_i32(const char* name, const pkv_tensor* t, int64_t len) {
  PKV_TRY(check_tensor(name, t, 1));
  PKV_TRY(need(t->dtype == PKV_I32, describe(name, t) + ": must be i32"));
  PKV_TRY(need(t->shape[0] == len, describe(name, t) + ": expected length " + std::to_string(len)));
  PKV_TRY(need(t->shape[0] <= 1 || t->stride[0] == 1, describe(name, t) + ": must be contiguous"));
  return PKV_OK;
}

pkv_status check_block_tables(const pkv_tensor* bt, int64_t B) {
  PKV_TRY(check_tensor("block_tables", bt, 2));
  PKV_TRY(need(bt->dtype == PKV_I32, describe("block_tables", bt) + ": must be i32"));
  PKV_TRY(need(bt->shape[0] == B, describe("block_tables", bt) + ": first extent must be B = " +
                                     std::to_string(B)));
  PKV_TRY(need(bt->shape[1] >= 1, describe("block_tables", bt) + ": needs at least one column"));
  PKV_TRY(need(bt->shape[1] <= 1 || bt->stride[1] == 1, "block_tables: column stride must be 1"));
  PKV_TRY(need(bt->shape[0] <= 1 || bt->stride[0] >= bt->shape[1], "block_tables: rows overlap"));
  return PKV_OK;
}

pkv_status check_caches(const pkv_tensor* kc, const pkv_tensor* vc) {
  PKV_TRY(check_tensor("k_cache", kc, 4));
  PKV_TRY(check_tensor("v_cache", vc, 4));
  PKV_TRY(need(kc->dtype == vc->dtype, "k_cache and v_cache dtypes differ"));
  for (int i = 0; i < 4; ++i)
    PKV_TRY(need(kc->shape[i] == vc->shape[i], "k_cache and v_cache shapes differ"));
  PKV_TRY(need(kc->dtype == PKV_F32 || kc->dtype == PKV_BF16 || kc->dtype == PKV_FP8_E4M3,
               describe("k_cache", kc) + ": cache dtype must be f32, bf16 or fp8_e4m3"));
  PKV_TRY(need(contiguous(kc) && contiguous(vc), "caches must be contiguous [num_blocks, block_size, Hkv, D]"));
  PKV_TRY(need(kc->shape[1] >= 1, "block_size must be >= 1"));
  PKV_TRY(need(kc->shape[2] >= 1 && kc->shape[3] >= 1, "Hkv and D must be >= 1"));
  PKV_TRY(need(kc->shape[0] <= INT32_MAX, "num_blocks beyond int32"));
  PKV_TRY(need(aligned(kc->data, 16) && aligned(vc->data, 16), "cache data must be 16-byte aligned"));
  return PKV_OK;
}

int log2_exact(int64_t v) {
  if (v <= 0 || (v & (v - 1))) return -1;
  int k = 0;
  while ((int64_t(1) << k) < v) ++k;
  return k;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

namespace pkv {

cudaError_t set_smem_attr(const void* kernel, size_t bytes) {
  // small open-addressing table keyed by the kernel's address
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uintptr_t key = reinterpret_cast<uintptr_t>(kernel);
  static std::atomic<uintptr_t> keys[256];
  size_t i = (key >> 4) % 256;
  for (size_t probe = 0; probe < 256; ++probe, i = (i + 1) % 256) {
    uintptr_t k = keys[i].load();
    if (k == 0) {
      uintptr_t expected = 0;
      if (!keys[i].compare_exchange_strong(expected, key) && expected != key) continue;
      k = key;
    }
    if (k != key) continue;
    const uint64_t bit = uint64_t(1) << (dev & 63);
    if (g_attr_set_mask[i].load() & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess) g_attr_set_mask[i].fetch_or(bit);
    return e;
  }
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

int64_t max_prefill_tiles(int64_t B, int64_t T, int64_t G) {
  return (T * G + kPrefillRows - 1) / kPrefillRows + B;
}

struct WsLayout {
  size_t dec_off, pf_off, work, merge_desc, done, dec_desc, pf_desc, part_o, part_lse, total;
};

static WsLayout ws_layout(int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t D, int64_t max_ctx) {
  const int64_t G = Hkv > 0 ? Hq / Hkv : 1;
  const int64_t units = B * max_chunks_for(max_ctx);
  WsLayout L{};
  size_t n = 0;
  L.dec_off = n;  n += align_up(sizeof(int32_t) * (B + 1), 256);
  L.pf_off = n;   n += align_up(sizeof(int32_t) * (B + 1), 256);
  L.work = n;     n += 256;  // claim counters, merge count, plan signature
  L.merge_desc = n; n += align_up(sizeof(MergeDesc) * B * Hq, 256);
  L.done = n;     n += align_up(sizeof(int32_t) * B * Hkv, 256);
  L.dec_desc = n; n += align_up(sizeof(DecodeDesc) * units, 256);
  L.pf_desc = n;  n += align_up(sizeof(PrefillDesc) * max_prefill_tiles(B, T, G), 256);
  L.part_o = n;   n += align_up(sizeof(float) * units * Hq * D, 256);
  L.part_lse = n; n += align_up(sizeof(float) * units * Hq, 256);
  L.total = n;
  return L;
}

size_t attention_workspace_bytes(int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t D, int64_t max_ctx) {
  return ws_layout(B, T, Hq, Hkv, D, max_ctx).total;
}

pkv_status record_failure(pkv_status st, const std::string& msg) { return fail(st, msg); }

}  // namespace pkv

// ======================================================================
extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARGUMENT: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE_CHECK: return "device index check failed";
    case PKV_ERR_OUT_OF_BLOCKS: return "out of cache blocks";
  }
  return "unknown status";
}

const char* pkv_last_error(void) { return t_last_error.c_str(); }

const char* pkv_version(void) { return "0.1.0"; }

pkv_status pkv_device_errors(void* stream, uint32_t* flags) {
  if (flags == nullptr) return fail(PKV_ERR_INVALID_ARGUMENT, "flags is NULL");
  unsigned int* err = nullptr;
  int sms = 0;
  PKV_TRY(device_state(&err, &sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_pkv_error_word, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_pkv_error_word, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  *flags = v;
  return PKV_OK;
}

pkv_status pkv_slot_mapping(const pkv_tensor* cu_seqlens_q, const pkv_tensor* seq_lens,
                            const pkv_tensor* block_tables, int32_t block_size, pkv_tensor* slot_mapping,
                            void* stream) {
  PKV_TRY(check_tensor("seq_lens", seq_lens, 1));
  const int64_t B = seq_lens->shape[0];
  PKV_TRY(need(B <= INT32_MAX - 1, "B beyond int32"));
  PKV_TRY(check_vector_i32("seq_lens", seq_lens, B));
  PKV_TRY(check_vector_i32("cu_seqlens_q", cu_seqlens_q, B + 1));
  PKV_TRY(check_block_tables(block_tables, B));
  PKV_TRY(need(block_size >= 1, "block_size must be >= 1"));
  PKV_TRY(need(block_tables->shape[1] * (int64_t)block_size <= INT32_MAX, "max_blocks * block_size beyond int32"));
  PKV_TRY(check_tensor("slot_mapping", slot_mapping, 1));
  PKV_TRY(need(slot_mapping->dtype == PKV_I32 || slot_mapping->dtype == PKV_I64, "slot_mapping must be i32 or i64"));
  PKV_TRY(need(slot_mapping->shape[0] <= 1 || slot_mapping->stride[0] == 1, "slot_mapping must be contiguous"));
  const int64_t T = slot_mapping->shape[0];
  unsigned int* err = nullptr;
  int sms = 0;
  PKV_TRY(device_state(&err, &sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (B == 0 || T == 0) return PKV_OK;
  cudaError_t e = pkv::launch_slot_mapping(
      static_cast<const int32_t*>(cu_seqlens_q->data), static_cast<const int32_t*>(seq_lens->data),
      static_cast<const int32_t*>(block_tables->data), block_tables->stride[0],
      static_cast<int32_t>(block_tables->shape[1]), static_cast<int32_t>(B), block_size, slot_mapping->data,
      slot_mapping->dtype == PKV_I64, T, err, st);
  if (e != cudaSuccess) return cuda_fail(e, "slot mapping launch");
  return finish(st, "pkv_slot_mapping");
}

pkv_status pkv_csr_to_block_tables(const pkv_tensor* kv_indptr, const pkv_tensor* kv_indices,
                                   pkv_tensor* block_tables, void* stream) {
  PKV_TRY(check_tensor("kv_indptr", kv_indptr, 1));
  const int64_t B = kv_indptr->shape[0] - 1;
  PKV_TRY(need(B >= 0 && B <= INT32_MAX - 1, "kv_indptr must have B + 1 entries"));
  PKV_TRY(check_vector_i32("kv_indptr", kv_indptr, B + 1));
  PKV_TRY(check_tensor("kv_indices", kv_indices, 1));
  PKV_TRY(need(kv_indices->dtype == PKV_I32, "kv_indices must be int32"));
  PKV_TRY(need(kv_indices->shape[0] <= 1 || kv_indices->stride[0] == 1, "kv_indices must be contiguous"));
  PKV_TRY(check_block_tables(block_tables, B));
  PKV_TRY(need(block_tables->shape[1] <= INT32_MAX, "max_blocks beyond int32"));
  unsigned int* err = nullptr;
  int sms = 0;
  PKV_TRY(device_state(&err, &sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (B == 0 || block_tables->shape[1] == 0) return PKV_OK;
  cudaError_t e = pkv::launch_csr_tables(static_cast<const int32_t*>(kv_indptr->data),
                                         static_cast<const int32_t*>(kv_indices->data), kv_indices->shape[0],
                                         static_cast<int32_t*>(block_tables->data), block_tables->stride[0],
                                         static_cast<int32_t>(block_tables->shape[1]), static_cast<int32_t>(B), err, st);
  if (e != cudaSuccess) return cuda_fail(e, "csr table launch");
  return finish(st, "pkv_csr_to_block_tables");
}

pkv_status pkv_append(const pkv_tensor* k, const pkv_tensor* v, const pkv_tensor* slot_mapping,
                      pkv_tensor* k_cache, pkv_tensor* v_cache, float k_scale, float v_scale, void* stream) {
  PKV_TRY(check_tensor("k", k, 3));
  PKV_TRY(check_tensor("v", v, 3));
  PKV_TRY(check_caches(k_cache, v_cache));
  const int64_t T = k->shape[0], Hkv = k_cache->shape[2], D = k_cache->shape[3];
  for (int i = 0; i < 3; ++i) PKV_TRY(need(k->shape[i] == v->shape[i], "k and v shapes differ"));
  PKV_TRY(need(k->dtype == v->dtype, "k and v dtypes differ"));
  PKV_TRY(need(k->shape[1] == Hkv && k->shape[2] == D,
               describe("k", k) + " does not match cache [.., .., Hkv, D] = [" + std::to_string(Hkv) + ", " +
                   std::to_string(D) + "]"));
  PKV_TRY(check_tensor("slot_mapping", slot_mapping, 1));
  PKV_TRY(need(slot_mapping->dtype == PKV_I32 || slot_mapping->dtype == PKV_I64, "slot_mapping must be i32 or i64"));
  PKV_TRY(need(slot_mapping->shape[0] == T, "slot_mapping length must equal T"));
  PKV_TRY(need(T <= 1 || slot_mapping->stride[0] == 1, "slot_mapping must be contiguous"));
  const bool fp8 = k_cache->dtype == PKV_FP8_E4M3;
  int src_kind;
  if (k->dtype == PKV_F32 && (k_cache->dtype == PKV_F32 || fp8))
    src_kind = 0;
  else if (k->dtype == PKV_BF16 && (k_cache->dtype == PKV_BF16 || fp8))
    src_kind = 1;
  else
    return fail(PKV_ERR_UNSUPPORTED, std::string("append ") + dtype_name(k->dtype) + " rows into a " +
                                         dtype_name(k_cache->dtype) + " cache");
  PKV_TRY(need(D % 8 == 0 && D <= 256, "append needs D a multiple of 8, at most 256"));
  if (src_kind == 0) PKV_TRY(need(D % 4 == 0, "f32 rows need D % 4 == 0"));
  const int es = esize(k->dtype);
  for (const pkv_tensor* x : {k, v}) {
    PKV_TRY(need(x->stride[2] == 1 || x->shape[2] == 1, "k/v must have unit stride in D"));
    PKV_TRY(need(aligned(x->data, 16) && (x->stride[0] * es) % 16 == 0 && (x->stride[1] * es) % 16 == 0,
                 "k/v rows must be 16-byte aligned (data and strides)"));
  }
  if (fp8) {
    PKV_TRY(need(k_scale > 0.f && v_scale > 0.f && k_scale == k_scale && v_scale == v_scale,
                 "fp8 scales must be positive and finite"));
  }
  unsigned int* err = nullptr;
  int sms = 0;
  PKV_TRY(device_state(&err, &sms));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) return PKV_OK;
  pkv::AppendParams p{};
  p.k = k->data;
  p.v = v->data;
  p.k_st = k->stride[0];
  p.k_sh = k->stride[1];
  p.v_st = v->stride[0];
  p.v_sh = v->stride[1];
  p.slots = slot_mapping->data;
  p.k_cache = k_cache->data;
  p.v_cache = v_cache->data;
  p.T = T;
  p.Hkv = static_cast<int32_t>(Hkv);
  p.D = static_cast<int32_t>(D);
  p.num_slots = k_cache->shape[0] * k_cache->shape[1];
  p.k_inv_scale = fp8 ? 1.0f / k_scale : 1.0f;  // IEEE fp32 division on the host
  p.v_inv_scale = fp8 ? 1.0f / v_scale : 1.0f;
  p.err = err;
  cudaError_t e = pkv::launch_append(p, src_kind, fp8, slot_mapping->dtype == PKV_I64, st);
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return finish(st, "pkv_append");
}

pkv_status pkv_attention_workspace_size(const pkv_tensor* q, const pkv_tensor* block_tables,
                                        const pkv_tensor* k_cache, size_t* bytes) {
  PKV_TRY(check_tensor("q", q, 3));
  PKV_TRY(check_tensor("block_tables", block_tables, 2));
  PKV_TRY(check_tensor("k_cache", k_cache, 4));
  PKV_TRY(need(bytes != nullptr, "bytes is NULL"));
  PKV_TRY(need(k_cache->shape[2] >= 1, "Hkv must be >= 1"));
  *bytes = pkv::attention_workspace_bytes(block_tables->shape[0], q->shape[0], q->shape[1], k_cache->shape[2],
                                          q->shape[2], block_tables->shape[1] * k_cache->shape[1]);
  return PKV_OK;
}

}  // extern "C"

namespace {

// One attention call, validated: the kernel parameters and the choices the
// host makes from the shapes alone.
struct Call {
  pkv::AttnParams p;
  int kv;           // 0 f32, 1 bf16, 2 e4m3 caches
  int out_kind;     // 0 f32, 1 bf16 output
  bool prefill;     // a prefill kernel runs (max_q_len > 1, unknown, or G beyond the decode kernel)
  bool tc;          // ... the tensor-core one
  int64_t max_ctx;  // tokens a block table can hold
  int sms;
  cudaStream_t st;
};

// Validates the arguments of an attention call and fills c.  The plan call
// passes no v_cache and no out (NULL): it needs only the shapes, the lengths
// and the workspace.
pkv_status prepare(const pkv_tensor* q, const pkv_tensor* cu_seqlens_q, const pkv_tensor* seq_lens,
                   const pkv_tensor* block_tables, const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                   float scale, float k_scale, float v_scale, int32_t max_q_len, const pkv_tensor* out,
                   float soft_cap, int32_t window_left, void* workspace, size_t workspace_bytes, void* stream,
                   Call& c) {
  const bool plan_only = out == nullptr;
  if (plan_only) v_cache = k_cache;
  PKV_TRY(check_tensor("q", q, 3));
  if (!plan_only) PKV_TRY(check_tensor("out", out, 3));
  PKV_TRY(check_tensor("seq_lens", seq_lens, 1));
  const int64_t B = seq_lens->shape[0];
  PKV_TRY(need(B <= (1 << 24), "B beyond 2^24 sequences"));
  PKV_TRY(check_vector_i32("seq_lens", seq_lens, B));
  PKV_TRY(check_vector_i32("cu_seqlens_q", cu_seqlens_q, B + 1));
  PKV_TRY(check_block_tables(block_tables, B));
  PKV_TRY(check_caches(k_cache, v_cache));
  const int64_t T = q->shape[0], Hq = q->shape[1], D = q->shape[2];
  const int64_t NB = k_cache->shape[0], bs = k_cache->shape[1], Hkv = k_cache->shape[2];
  PKV_TRY(need(k_cache->shape[3] == D, "q and cache head dims differ"));
  PKV_TRY(need(Hq >= 1 && Hq % Hkv == 0, "Hq must be a positive multiple of Hkv"));
  if (!plan_only) {
    PKV_TRY(need(out->shape[0] == T && out->shape[1] == Hq && out->shape[2] == D,
                 describe("out", out) + " must have q's shape"));
    PKV_TRY(need(out->dtype == PKV_F32 || out->dtype == PKV_BF16, "out must be f32 or bf16"));
  }
  PKV_TRY(need(block_tables->shape[1] * bs <= INT32_MAX, "max_blocks * block_size beyond int32"));
  PKV_TRY(need(T <= INT32_MAX, "T beyond int32"));
  if (NB * bs > INT32_MAX)
    return fail(PKV_ERR_UNSUPPORTED, "num_blocks * block_size beyond int32 (slots are 32-bit in attention)");
  int kv;
  if (q->dtype == PKV_F32 && k_cache->dtype == PKV_F32)
    kv = 0;
  else if (q->dtype == PKV_BF16 && k_cache->dtype == PKV_BF16)
    kv = 1;
  else if (q->dtype == PKV_BF16 && k_cache->dtype == PKV_FP8_E4M3)
    kv = 2;
  else
    return fail(PKV_ERR_UNSUPPORTED, std::string("q ") + dtype_name(q->dtype) + " with a " +
                                         dtype_name(k_cache->dtype) + " cache");
  if (kv == 0)
    PKV_TRY(need(D % 32 == 0 && D <= 256, "f32 attention needs D a multiple of 32, at most 256"));
  else if (D != 64 && D != 128)
    return fail(PKV_ERR_UNSUPPORTED, "bf16/fp8 attention is built for D = 64 and D = 128");
  PKV_TRY(need(q->stride[2] == 1 || D == 1, "q must have unit stride in D"));
  const int qes = esize(q->dtype);
  PKV_TRY(need(aligned(q->data, 16) && (q->stride[0] * qes) % 16 == 0 && (q->stride[1] * qes) % 16 == 0,
               "q rows must be 16-byte aligned (data and strides)"));
  if (!plan_only) {
    PKV_TRY(need(out->stride[2] == 1 || D == 1, "out must have unit stride in D"));
    const int oes = esize(out->dtype);
    PKV_TRY(need(aligned(out->data, 16) && (out->stride[0] * oes) % 8 == 0 && (out->stride[1] * oes) % 8 == 0,
                 "out rows must be 8-byte aligned (data and strides)"));
    if (kv == 2)
      PKV_TRY(need(k_scale > 0.f && v_scale > 0.f && k_scale == k_scale && v_scale == v_scale,
                   "fp8 scales must be positive and finite"));
    PKV_TRY(need(scale == scale, "scale is NaN"));
  }
  const int64_t max_ctx = block_tables->shape[1] * bs;
  const size_t ws_need = pkv::attention_workspace_bytes(B, T, Hq, Hkv, D, max_ctx);
  if (kv != 0) {
    if (workspace_bytes < ws_need)
      return fail(PKV_ERR_WORKSPACE_TOO_SMALL, "workspace needs " + std::to_string(ws_need) + " bytes, got " +
                                                   std::to_string(workspace_bytes));
    PKV_TRY(need(workspace != nullptr && aligned(workspace, 256), "workspace must be 256-byte aligned"));
  }
  c.st = static_cast<cudaStream_t>(stream);
  c.kv = kv;
  c.out_kind = !plan_only && out->dtype == PKV_BF16 ? 1 : 0;
  c.max_ctx = max_ctx;

  pkv::AttnParams& p = c.p;
  p = pkv::AttnParams{};
  p.q = q->data;
  p.q_st = q->stride[0];
  p.q_sh = q->stride[1];
  p.out = plan_only ? nullptr : out->data;
  p.T = T;
  p.o_st = plan_only ? 0 : out->stride[0];
  p.o_sh = plan_only ? 0 : out->stride[1];
  p.cu_q = static_cast<const int32_t*>(cu_seqlens_q->data);
  p.seq_lens = static_cast<const int32_t*>(seq_lens->data);
  p.bt = static_cast<const int32_t*>(block_tables->data);
  p.bt_stride = block_tables->stride[0];
  p.max_blocks = static_cast<int32_t>(block_tables->shape[1]);
  p.B = static_cast<int32_t>(B);
  p.k_cache = k_cache->data;
  p.v_cache = v_cache->data;
  p.num_blocks = NB;
  p.bs = static_cast<int32_t>(bs);
  p.bs_shift = log2_exact(bs);
  p.Hq = static_cast<int32_t>(Hq);
  p.Hkv = static_cast<int32_t>(Hkv);
  p.G = static_cast<int32_t>(Hq / Hkv);
  p.D = static_cast<int32_t>(D);
  const float kLog2e = 1.4426950408889634f;
  p.qk_scale_log2 = scale * (kv == 2 ? k_scale : 1.0f) * kLog2e;
  p.soft_cap = soft_cap > 0.f ? soft_cap : 0.f;
  p.cap_pre = p.soft_cap > 0.f ? scale * (kv == 2 ? k_scale : 1.0f) / soft_cap : 0.f;
  p.cap_post = p.soft_cap > 0.f ? soft_cap * kLog2e : 0.f;
  p.window_left = window_left >= 0 ? window_left : -1;
  p.v_scale = kv == 2 ? v_scale : 1.0f;
  p.decode_max_g = 8;
  p.kv_esize = esize(k_cache->dtype);
  if (kv == 0) {
    if (p.soft_cap > 0.f || p.window_left >= 0)
      return fail(PKV_ERR_UNSUPPORTED, "a soft cap or sliding window is built for bf16 and e4m3 caches");
    c.prefill = c.tc = false;
    return device_state(&p.err, &c.sms);
  }
  // workspace carve-up
  {
    const pkv::WsLayout L = pkv::ws_layout(B, T, Hq, Hkv, D, max_ctx);
    char* w = static_cast<char*>(workspace);
    p.ws.dec_off = reinterpret_cast<int32_t*>(w + L.dec_off);
    p.ws.pf_off = reinterpret_cast<int32_t*>(w + L.pf_off);
    p.ws.work = reinterpret_cast<unsigned long long*>(w + L.work);
    p.ws.pf_work = p.ws.work + 1;
    p.ws.n_merge = reinterpret_cast<int32_t*>(w + L.work + 16);
    p.ws.pf_ctas = reinterpret_cast<int32_t*>(w + L.work + 20);
    p.ws.sig = reinterpret_cast<int32_t*>(w + L.work + 32);
    p.ws.merge_desc = reinterpret_cast<pkv::MergeDesc*>(w + L.merge_desc);
    p.ws.done = reinterpret_cast<int32_t*>(w + L.done);
    p.ws.dec_desc = reinterpret_cast<pkv::DecodeDesc*>(w + L.dec_desc);
    p.ws.pf_desc = reinterpret_cast<pkv::PrefillDesc*>(w + L.pf_desc);
    p.ws.part_o = reinterpret_cast<float*>(w + L.part_o);
    p.ws.part_lse = reinterpret_cast<float*>(w + L.part_lse);
  }
  const int G = p.G;
  c.prefill = (max_q_len > 1) || (max_q_len <= 0 && T >= 2) || G > p.decode_max_g;
  c.tc = c.prefill && pkv::prefill_tc_supported(kv, D, bs, G);
  const bool variant = p.soft_cap > 0.f || p.window_left >= 0;
  if (variant && c.prefill && !c.tc)
    return fail(PKV_ERR_UNSUPPORTED, "a soft cap or sliding window needs decode rows, or prefill rows on bf16 "
                                     "or e4m3 caches with block sizes a multiple of 8 (max_q_len > 1 here)");
  p.pf_tq = c.tc ? pkv::prefill_tc_tokens_per_tile(G) : 0;
  p.path = !c.prefill ? 0 : (c.tc ? 2 : 1);
  // the decode kernel's KV heads per item: the plan cuts merge items by it
  p.hp = G <= p.decode_max_g ? pkv::decode_heads_per_item(kv, D, Hkv, G) : 1;
  if (p.hp < 1) return fail(PKV_ERR_UNSUPPORTED, "no decode kernel geometry for these heads");
  // every argument is valid: the device's error word and SM count
  PKV_TRY(device_state(&p.err, &c.sms));
  p.num_sms = c.sms;
  return PKV_OK;
}

pkv_status launch_plan(const Call& c) {
  if (c.kv == 0 || c.p.T == 0 || c.p.B == 0) return PKV_OK;
  cudaError_t e = pkv::launch_plan(c.p, c.st);
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");
  return PKV_OK;
}

// The kernels of one run over the plan in the workspace: the prefill kernel
// (if any), then the decode kernel.
pkv_status launch_run(const Call& c) {
  const pkv::AttnParams& p = c.p;
  if (p.T == 0 || p.B == 0) return PKV_OK;
  cudaError_t e;
  if (c.kv == 0) {
    e = pkv::launch_f32(p, c.out_kind, p.T, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "f32 attention launch");
    return PKV_OK;
  }
  if (c.prefill) {
    const int64_t tiles = pkv::max_prefill_tiles(p.B, p.T, p.G);
    e = c.tc ? pkv::launch_prefill_tc(p, c.out_kind, tiles * p.Hkv, c.sms, c.st)
             : pkv::launch_prefill(p, c.kv, c.out_kind, tiles * p.Hkv, c.sms, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  }
  if (p.G <= p.decode_max_g) {
    const int64_t dec_seqs = std::min<int64_t>(p.B, p.T);
    // programmatic launch after the plan or the previous kernel of the
    // stream (the decode kernel waits for it before reading anything), and
    // after the tensor-core prefill, beside which it runs (it waits for the
    // prefill only before it exits); after the mma.sync prefill it is a
    // plain launch
    pkv::AttnParams pd = p;
    pd.dec_concurrent = c.tc ? 1 : 0;
    e = pkv::launch_decode(pd, c.kv, c.out_kind, dec_seqs * pkv::max_chunks_for(c.max_ctx) * p.Hkv, c.sms, c.st,
                           !c.prefill || c.tc);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  }
  return PKV_OK;
}

pkv_status variant_args(const pkv_attention_variant* variant, float& cap, int32_t& window) {
  cap = 0.f;
  window = -1;
  if (variant != nullptr) {
    PKV_TRY(need(variant->logits_soft_cap >= 0.f && variant->logits_soft_cap < INFINITY,
                 "logits_soft_cap must be finite and >= 0 (0: off)"));
    cap = variant->logits_soft_cap;
    window = variant->window_left < 0 ? -1 : variant->window_left;
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_attention(const pkv_tensor* q, const pkv_tensor* cu_seqlens_q, const pkv_tensor* seq_lens,
                         const pkv_tensor* block_tables, const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                         float scale, float k_scale, float v_scale, int32_t max_q_len, pkv_tensor* out,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return pkv_attention_ex(q, cu_seqlens_q, seq_lens, block_tables, k_cache, v_cache, scale, k_scale, v_scale,
                          max_q_len, out, nullptr, workspace, workspace_bytes, stream);
}

pkv_status pkv_attention_ex(const pkv_tensor* q, const pkv_tensor* cu_seqlens_q, const pkv_tensor* seq_lens,
                            const pkv_tensor* block_tables, const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                            float scale, float k_scale, float v_scale, int32_t max_q_len, pkv_tensor* out,
                            const pkv_attention_variant* variant, void* workspace, size_t workspace_bytes,
                            void* stream) {
  float cap;
  int32_t window;
  PKV_TRY(variant_args(variant, cap, window));
  PKV_TRY(need(out != nullptr, "out is NULL"));
  Call c;
  PKV_TRY(prepare(q, cu_seqlens_q, seq_lens, block_tables, k_cache, v_cache, scale, k_scale, v_scale, max_q_len,
                  out, cap, window, workspace, workspace_bytes, stream, c));
  PKV_TRY(launch_plan(c));
  PKV_TRY(launch_run(c));
  return finish(c.st, "pkv_attention");
}

pkv_status pkv_attention_plan(const pkv_tensor* q, const pkv_tensor* cu_seqlens_q, const pkv_tensor* seq_lens,
                              const pkv_tensor* block_tables, const pkv_tensor* k_cache, int32_t max_q_len,
                              const pkv_attention_variant* variant, void* workspace, size_t workspace_bytes,
                              void* stream) {
  float cap;
  int32_t window;
  PKV_TRY(variant_args(variant, cap, window));
  Call c;
  PKV_TRY(prepare(q, cu_seqlens_q, seq_lens, block_tables, k_cache, nullptr, 1.f, 1.f, 1.f, max_q_len, nullptr,
                  cap, window, workspace, workspace_bytes, stream, c));
  PKV_TRY(launch_plan(c));
  return finish(c.st, "pkv_attention_plan");
}

pkv_status pkv_attention_run(const pkv_tensor* q, const pkv_tensor* cu_seqlens_q, const pkv_tensor* seq_lens,
                             const pkv_tensor* block_tables, const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                             float scale, float k_scale, float v_scale, int32_t max_q_len, pkv_tensor* out,
                             const pkv_attention_variant* variant, void* workspace, size_t workspace_bytes,
                             void* stream) {
  float cap;
  int32_t window;
  PKV_TRY(variant_args(variant, cap, window));
  PKV_TRY(need(out != nullptr, "out is NULL"));
  Call c;
  PKV_TRY(prepare(q, cu_seqlens_q, seq_lens, block_tables, k_cache, v_cache, scale, k_scale, v_scale, max_q_len,
                  out, cap, window, workspace, workspace_bytes, stream, c));
  PKV_TRY(launch_run(c));
  return finish(c.st, "pkv_attention_run");
}

}  // extern "C"
