/*
 * pkv.h -- C ABI of libpkv.so: paged KV cache append and attention for one
 * GB300 (sm_103a) GPU.
 *
 * The problem, as the pages state it:
 *   - "How to design an LLM serving system (a vLLM deep dive)", section
 *     "PagedAttention (vLLM KV manager)": the KV cache is a pool of fixed
 *     physical blocks of block_size tokens; each request's block table maps
 *     its logical positions to non-contiguous physical blocks; slot_mapping
 *     tells the kernel which physical slot each token's K/V goes to.
 *   - nanoserve, section "Architecture" (one engine step): all new tokens of
 *     a step are packed into one [T] dimension, each token's cache slot is
 *     computed from its block table (step 2), and each layer writes this
 *     step's K/V into the paged cache, then attends over the full context
 *     through the block table (step 3); decodes and prefill chunks share a
 *     step ("Chunked prefill", "Packed batches").
 *   - "How Easy Is It to Start Serving LLMs?", section "1. Block-sparse KV
 *     memory": the page table is all the attention kernel needs; pages may
 *     sit anywhere in the pool and may be shared.
 *
 * Layouts (row-major, innermost last):
 *   q, out        [T, Hq, D]        packed query rows of all sequences
 *   k, v          [T, Hkv, D]       this step's new K/V rows
 *   k_cache,
 *   v_cache       [num_blocks, block_size, Hkv, D]   one layer, contiguous
 *   block_tables  [B, max_blocks]   int32 physical block ids
 *   cu_seqlens_q  [B+1]             int32, rows of sequence s are
 *                                   cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1
 *   seq_lens      [B]               int32, N_s = keys of sequence s, this
 *                                   step's new tokens included
 *   slot_mapping  [T]               int32 or int64 flat slot per new row
 *
 * Semantics (every function):
 *   - Query row i of sequence s (q_s = cu_seqlens_q[s+1]-cu_seqlens_q[s]
 *     rows) sits at position p = N_s - q_s + i and attends, causally, to
 *     keys 0..p; a decode is the q_s = 1 case.  Query head h reads KV head
 *     h / (Hq / Hkv).
 *   - The flat slot of position p is
 *     block_tables[s][p / block_size] * block_size + p % block_size, and
 *     slot = block * block_size + offset addresses
 *     cache[block][offset][head][:].
 *   - fp8 caches hold OCP e4m3 codes of x / scale (per-tensor scales).
 *
 * Ownership and execution: the caller owns every buffer (device memory,
 * e.g. from PyTorch) and the stream.  The library allocates no memory and
 * never synchronises, except in check mode (environment PKV_CHECK=1).  A
 * PKV_OK return means the work was enqueued on the stream.  Pointers are
 * device pointers unless stated.  Device-resident indices (slots, block
 * ids, lengths) are bounds-checked by the kernels: an out-of-range index
 * is skipped (no write, zero contribution) and recorded; check mode, or
 * pkv_device_errors(), reports it.  No kernel traps or faults on bad
 * indices.
 *
 * Kernels of this library are launched with programmatic dependent launch:
 * each may begin (and set up) while the previous kernel in the stream is
 * still running, and waits for that kernel to complete, with its writes
 * visible, before it reads or writes any memory.  Inputs written by the
 * previous kernel of the stream, the lengths included, are therefore safe.
 *
 * The library keeps, per device, the addresses of its own device variables
 * (the error word, the static workspace), looked up at the first call on
 * the device in the runtime's primary context.  It is not for use after
 * cudaDeviceReset or under another context made current through the
 * driver API.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the library are exported; everything else in it is hidden. */
#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARGUMENT = 1,    /* shapes, dtypes, strides or values disagree */
  PKV_ERR_UNSUPPORTED = 2,         /* a valid request outside the built variants */
  PKV_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below the size required */
  PKV_ERR_CUDA = 4,                /* a CUDA call failed; pkv_last_error() says which */
  PKV_ERR_DEVICE_CHECK = 5,        /* check mode: a kernel met an out-of-range index */
  PKV_ERR_OUT_OF_BLOCKS = 6        /* block manager: the pool cannot hold the request */
} pkv_status;

typedef enum {
  PKV_F32 = 0,
  PKV_BF16 = 1,
  PKV_FP8_E4M3 = 2,
  PKV_I32 = 3,
  PKV_I64 = 4
} pkv_dtype;

/* A strided view of caller-owned memory.  Strides are in elements. */
typedef struct {
  void* data;
  pkv_dtype dtype;
  int32_t ndim;
  int64_t shape[4];
  int64_t stride[4];
} pkv_tensor;

/*
 * pkv_slot_mapping -- the flat cache slot of every new row of a step.
 * nanoserve, "Architecture", step 2 ("Prepare": compute each token's cache
 * slot from its block table); "How to design an LLM serving system (a vLLM
 * deep dive)", "PagedAttention" (slot_mapping).
 *
 *   cu_seqlens_q  [B+1] int32 (device)
 *   seq_lens      [B]   int32 (device), N_s after this step's rows
 *   block_tables  [B, max_blocks] int32 (device), unit column stride
 *   block_size    tokens per block, >= 1
 *   slot_mapping  [T] int32 or int64 (device, written), T = cu_seqlens_q[B]
 *                 is the caller's host-side row count (shape[0])
 *
 * Rows of a sequence whose lengths are inconsistent (q_s < 0, q_s > N_s or
 * N_s > max_blocks * block_size) or whose block id is negative get slot -1
 * and are recorded as a device error.
 */
PKV_API pkv_status pkv_slot_mapping(const pkv_tensor* cu_seqlens_q, const pkv_tensor* seq_lens,
                            const pkv_tensor* block_tables, int32_t block_size,
                            pkv_tensor* slot_mapping, void* stream);

/*
 * pkv_csr_to_block_tables -- block tables from the CSR page-list form.
 * "How Easy Is It to Start Serving LLMs?", "1. Block-sparse KV memory:
 * scattered pages cost nothing": a batch's pages as a sparse matrix with one
 * row per request; request i reads pages kv_indices[kv_indptr[i] ..
 * kv_indptr[i+1]-1] in order, and requests sharing a prompt list the same
 * page ids.
 *
 *   kv_indptr     [B+1] int32 (device), non-decreasing, kv_indptr[0] = 0
 *   kv_indices    [nnz] int32 (device), physical block ids, contiguous
 *   block_tables  [B, max_blocks] int32 (device, written), unit column
 *                 stride: row i holds request i's pages, then -1
 *
 * The sequence lengths stay the caller's (seq_lens of pkv_attention).  A
 * row with offsets that decrease or leave [0, nnz], or with more than
 * max_blocks pages, is filled with -1 and recorded as a device error (bit 4).
 */
PKV_API pkv_status pkv_csr_to_block_tables(const pkv_tensor* kv_indptr, const pkv_tensor* kv_indices,
                                           pkv_tensor* block_tables, void* stream);

/*
 * pkv_append -- scatter this step's K/V rows into their slots.
 * nanoserve, "Architecture", step 3 ("Forward": each layer writes this
 * step's K/V into the paged cache, then attends); "How to design an LLM
 * serving system (a vLLM deep dive)", "PagedAttention" (slot_mapping).
 *
 *   k, v          [T, Hkv, D], unit stride in D, 16-byte aligned rows
 *   slot_mapping  [T] int32 or int64; a negative slot skips the row
 *   k_cache,
 *   v_cache       [num_blocks, block_size, Hkv, D], contiguous
 *   k_scale,
 *   v_scale       per-tensor scales, used only when the cache is e4m3:
 *                 the stored code is e4m3_rn_satfinite(x * (1.0f / scale)),
 *                 the product taken in fp32 ("How Easy Is It to Start
 *                 Serving LLMs?", "What each setting does to performance":
 *                 FP8 KV cache)
 *
 * Supported: f32 -> f32, bf16 -> bf16, bf16 or f32 -> e4m3; D a multiple of
 * 8 up to 256.  Same-format rows are copied bit for bit.  Slots at or beyond
 * num_blocks * block_size are skipped and recorded.  Two rows with the same
 * non-negative slot in one call leave that slot unspecified.
 */
PKV_API pkv_status pkv_append(const pkv_tensor* k, const pkv_tensor* v, const pkv_tensor* slot_mapping,
                      pkv_tensor* k_cache, pkv_tensor* v_cache, float k_scale, float v_scale,
                      void* stream);

/*
 * pkv_attention_workspace_size -- bytes of device workspace pkv_attention
 * needs for these shapes (a host-side bound; no device access).
 *   q [T, Hq, D], block_tables [B, max_blocks], k_cache [NB, bs, Hkv, D].
 */
PKV_API pkv_status pkv_attention_workspace_size(const pkv_tensor* q, const pkv_tensor* block_tables,
                                        const pkv_tensor* k_cache, size_t* bytes);

/*
 * pkv_attention -- causal GQA attention of the packed query rows over each
 * sequence's pages.
 * nanoserve, "Architecture" step 3 and the "Triton paged-attention decode
 * kernel" bullet (K/V read straight from the block table with an online
 * softmax, decodes and prefill chunks in one step); "How Easy Is It to Start
 * Serving LLMs?", "3. Load balancing: keep every SM busy" (long requests are
 * split into chunks and a merge step stitches them back together).
 *
 *   q             [T, Hq, D] bf16 or f32, unit stride in D
 *   cu_seqlens_q  [B+1] int32
 *   seq_lens      [B] int32 (N_s includes this step's rows)
 *   block_tables  [B, max_blocks] int32, unit column stride; entries past
 *                 ceil(N_s / block_size) are never read
 *   k_cache,
 *   v_cache       [num_blocks, block_size, Hkv, D] contiguous; bf16 or e4m3
 *                 with bf16 q, f32 with f32 q
 *   scale         softmax scale (e.g. 1/sqrt(D))
 *   k_scale,
 *   v_scale       e4m3 dequantisation scales (value = code * scale); ignored
 *                 for bf16/f32 caches
 *   max_q_len     a host-side upper bound on q_s (1 for a pure decode batch;
 *                 <= 0 means "unknown", taken as T).  With max_q_len == 1
 *                 only the decode path is launched.
 *   out           [T, Hq, D] f32 or bf16 (written), unit stride in D
 *   workspace     device scratch of workspace_bytes, at least
 *                 pkv_attention_workspace_size(); 256-byte aligned
 *
 * The result for a row depends only on its own sequence (lengths, pages'
 * contents, query), never on the block size, the physical placement of
 * pages, or the other sequences of the batch: all tiling and splitting is
 * in logical token positions.  A bf16 output equals the f32 output rounded
 * to nearest even.
 *
 * Supported: Hq % Hkv == 0; D in {64, 128} for bf16/e4m3 caches, D a
 * multiple of 32 up to 256 for f32 caches; any block_size >= 1; q_s = 0
 * sequences produce no rows.
 */
PKV_API pkv_status pkv_attention(const pkv_tensor* q, const pkv_tensor* cu_seqlens_q,
                         const pkv_tensor* seq_lens, const pkv_tensor* block_tables,
                         const pkv_tensor* k_cache, const pkv_tensor* v_cache, float scale,
                         float k_scale, float v_scale, int32_t max_q_len, pkv_tensor* out,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * pkv_attention_ex -- pkv_attention with two of the variants a kernel
 * family is built for ("How Easy Is It to Start Serving LLMs?", "2. JIT
 * compilation: one template, a kernel per variant": logit soft-capping and
 * sliding windows).
 *
 *   logits_soft_cap  > 0: every scaled score s = scale * q.k becomes
 *                    logits_soft_cap * tanh(s / logits_soft_cap) before the
 *                    softmax; 0 turns it off.  Must be finite.
 *   window_left      >= 0: the query at position p attends to keys
 *                    max(0, p - window_left) .. p; < 0 turns it off.
 *
 * Built for decode rows and for prefill rows on caches whose block size is
 * a multiple of 8 (bf16 and e4m3 caches alike); other cases (f32 caches,
 * prefill rows on other block sizes) return PKV_ERR_UNSUPPORTED.
 * variant == NULL is pkv_attention.  With a window, a decode reads only the
 * blocks its window touches.
 */
typedef struct {
  float logits_soft_cap;
  int32_t window_left;
} pkv_attention_variant;

PKV_API pkv_status pkv_attention_ex(const pkv_tensor* q, const pkv_tensor* cu_seqlens_q,
                                    const pkv_tensor* seq_lens, const pkv_tensor* block_tables,
                                    const pkv_tensor* k_cache, const pkv_tensor* v_cache, float scale,
                                    float k_scale, float v_scale, int32_t max_q_len, pkv_tensor* out,
                                    const pkv_attention_variant* variant, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * pkv_attention_plan / pkv_attention_run -- pkv_attention in two parts, so
 * that one plan serves every layer of a model step.
 * "How Easy Is It to Start Serving LLMs?", "3. Load balancing: keep every SM
 * busy": the work of a decode step is planned once from the sequence
 * lengths, kept in a fixed GPU buffer, and reused by the attention of every
 * layer; scheduling then costs almost nothing per layer and stays
 * CUDA-graph friendly.
 *
 * pkv_attention_plan reads cu_seqlens_q and seq_lens on the device (no
 * device-to-host copy) and writes the work lists of the call into the
 * workspace, with a record of the shapes they were made for.  Arguments as
 * pkv_attention_ex; q's and k_cache's data are not read (only their shapes
 * and dtypes), block_tables' contents are not read, and of variant only
 * window_left matters (it decides which keys a decode reads).
 *
 * pkv_attention_run runs the attention of one layer over the plan in the
 * workspace: arguments, results and errors as pkv_attention_ex, which is
 * plan + run.  Between the plan and its runs the caller must keep
 * cu_seqlens_q, seq_lens, the shapes of q, block_tables and the caches, the
 * cache dtype, max_q_len and window_left unchanged; q, the caches' contents,
 * the block tables' contents, out, scale, k_scale, v_scale and the soft cap
 * may change from run to run.  A run leaves the plan intact, so runs may
 * follow each other on the stream without limit; a new plan replaces the
 * old one.  A run on a workspace whose plan was made for other shapes or
 * choices does no work and records bit 16 in the device error word
 * (pkv_device_errors); a run given other lengths than its plan's is not
 * detected and gives unspecified rows.  The runs of a plan keep count of
 * the work they claim in the workspace; after a run that recorded a wait
 * timeout (bit 8) those counts are off, so make a new plan.  Runs that share a workspace must not
 * overlap on the GPU (keep them on one stream).  With f32 caches the plan is
 * empty and a run is the whole call.
 */
PKV_API pkv_status pkv_attention_plan(const pkv_tensor* q, const pkv_tensor* cu_seqlens_q,
                                      const pkv_tensor* seq_lens, const pkv_tensor* block_tables,
                                      const pkv_tensor* k_cache, int32_t max_q_len,
                                      const pkv_attention_variant* variant, void* workspace,
                                      size_t workspace_bytes, void* stream);

PKV_API pkv_status pkv_attention_run(const pkv_tensor* q, const pkv_tensor* cu_seqlens_q,
                                     const pkv_tensor* seq_lens, const pkv_tensor* block_tables,
                                     const pkv_tensor* k_cache, const pkv_tensor* v_cache, float scale,
                                     float k_scale, float v_scale, int32_t max_q_len, pkv_tensor* out,
                                     const pkv_attention_variant* variant, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* Size of the scratch array inside the library that
 * pkv_attention_static_workspace uses on each device (16 MiB). */
#define PKV_STATIC_WORKSPACE_BYTES (16u << 20)

/*
 * pkv_attention_static_workspace -- pkv_attention without a workspace
 * argument: the scratch is a fixed 16 MiB array inside the library, one per
 * device, so the call allocates no device memory at all.  The method's
 * description has no counterpart to this call; it exists for callers that
 * cannot allocate: a runtime that has already handed every byte of HBM to
 * its own pools (weights, KV block pool), plain C code with no device
 * allocator of its own, or code that must not call cudaMalloc/cudaFree in
 * the middle of its work because those calls can synchronise the device.
 *
 * Arguments, layouts, results and errors are those of pkv_attention.  In
 * addition:
 *   - a call whose pkv_attention_workspace_size() exceeds
 *     PKV_STATIC_WORKSPACE_BYTES is rejected with
 *     PKV_ERR_WORKSPACE_TOO_SMALL before anything is launched, and
 *     pkv_last_error() names the size it needed (as a guide: 16 sequences
 *     with Hq = 32, D = 128 and up to 4096 tokens of context fit; 64 such
 *     sequences do not);
 *   - the first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call
 *     before starting any stream capture;
 *   - every call on a device uses the same array, and the array keeps what
 *     the last call left in it (each call resets the counters it needs on
 *     the stream before using them).  Calls whose GPU work can overlap --
 *     issued on different streams, or from host threads with no ordering
 *     between them -- race on the array and corrupt each other's results:
 *     keep such calls on one stream or order them with events.
 *   - the array's 16 MiB of device memory are reserved when the CUDA runtime
 *     loads the library's code for this call on a device (at the first call
 *     under lazy module loading);
 *   - the cached address is that of the device's primary context: after
 *     cudaDeviceReset, or with another context current, it is stale.
 */
PKV_API pkv_status pkv_attention_static_workspace(const pkv_tensor* q, const pkv_tensor* cu_seqlens_q,
                                                  const pkv_tensor* seq_lens,
                                                  const pkv_tensor* block_tables,
                                                  const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                                                  float scale, float k_scale, float v_scale,
                                                  int32_t max_q_len, pkv_tensor* out, void* stream);

/*
 * pkv_device_errors -- synchronise the stream, then return (in *flags) and
 * clear the record of out-of-range indices the kernels met on the current
 * device since the last call.  Bits: 1 = slot beyond the pool, 2 = block id
 * out of range, 4 = inconsistent lengths, 8 = a bounded wait gave up, 16 =
 * an attention run found no plan for its shapes in the workspace.
 */
PKV_API pkv_status pkv_device_errors(void* stream, uint32_t* flags);

/* Static description of a status code. */
PKV_API const char* pkv_status_string(pkv_status status);

/* Detail of the last failure on the calling thread ("" if none). */
PKV_API const char* pkv_last_error(void);

/* Library version, "major.minor.patch". */
PKV_API const char* pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
