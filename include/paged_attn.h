/*
 * paged_attn.h -- C ABI of libpagedattn.so: paged (block-table) KV-cache
 * append and attention on one NVIDIA GB300 (sm_103a).
 *
 * The operations follow the I/O contract of onnxruntime/mobius PR #395
 * "Add paged / block-table KV cache export" (sections "How it works (per
 * attention layer)" and "ONNX I/O contract"): new K/V rows are scattered
 * into a per-layer page pool at slot_mapping (ScatterND), and attention
 * reads a sequence's pages through block_table (Gather) with causal and
 * padding masking given by nonpad_kv_seqlen (here: seq_lens).  The batched,
 * row-padded block_table, seq_lens and query_start_loc follow the vLLM-shaped
 * metadata of ROCm/maxtext PR #93 "[Draft] kv paged kernels" (the
 * attention='gpu_paged' commit).
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor arguments are DEVICE pointers on the current CUDA device,
 *   owned by the caller.  The library allocates no device memory and keeps
 *   no per-call state.  Its state: one device-side error word per device
 *   (see paged_device_error); a process-wide note of whether the runtime
 *   accepts the decode kernel's cooperative launch (learnt on the first eager
 *   decode launch); and, for paged_attention_decode_cascade only, one extra
 *   stream and two events per (host thread, device), created by the first
 *   cascade call on that thread and kept for the thread's life.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream).  Host-side argument checks run before any launch; on a
 *   non-PA_OK return nothing was launched.
 * - Pool layout (NHD): key_pool and value_pool are each
 *   [num_pages, page_size, num_kv_heads, head_dim], contiguous, element type
 *   `dtype`.  The flat slot s = page_id * page_size + offset addresses row s
 *   of the pool viewed as [num_pages * page_size, num_kv_heads, head_dim].
 * - GQA/MQA: num_q_heads must be a multiple of num_kv_heads; query head h
 *   reads KV head h / (num_q_heads / num_kv_heads).
 * - The softmax scale is a required argument (there is no default 1/sqrt(d)):
 *   a query that already carries its scale is passed with scale = 1.0.
 * - There is no attention-bias, ALiBi or sliding-window argument: those are
 *   unsupported, not silently ignored.
 * - Device-side checks: a block_table entry outside [0, num_pages), a slot
 *   >= num_pages * page_size, or a seq_len outside [0, max_blocks_per_seq *
 *   page_size] is recorded in the device error word and the offending read
 *   or write is skipped (no trap, no hang).
 */
#ifndef PAGED_ATTN_H_
#define PAGED_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ABI_VERSION 2

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_NULL = 1,         /* a required pointer is NULL                        */
  PA_ERR_SHAPE = 2,        /* inconsistent or negative sizes                    */
  PA_ERR_DTYPE = 3,        /* unknown dtype                                     */
  PA_ERR_RANGE = 4,        /* a size is beyond what the kernels index (int32)   */
  PA_ERR_UNSUPPORTED = 5,  /* valid but not implemented (head_dim, page_size)   */
  PA_ERR_CUDA = 6,         /* a CUDA runtime call failed (launch, attribute)    */
  PA_ERR_WORKSPACE = 7,    /* workspace missing or smaller than required        */
  PA_ERR_ALIGN = 8         /* a pointer is not aligned as the dtype requires    */
} pa_status;

typedef enum pa_dtype {
  PA_DTYPE_F32 = 0,        /* float32 pool, q and out                           */
  PA_DTYPE_BF16 = 1,       /* bfloat16 pool, q and out; fp32 accumulation       */
  PA_DTYPE_FP8_E4M3 = 2    /* e4m3 pool with k_scale / v_scale; bf16 q, out and
                              appended rows                                     */
} pa_dtype;

/* One layer's KV page pool (mobius PR #395 "ONNX I/O contract":
 * key_pool.{i} / value_pool.{i}).  All fields are read-only to the library
 * except the pool contents, which paged_kv_append updates in place. */
typedef struct pa_kv_pool {
  void* key_pool;          /* device [num_pages, page_size, num_kv_heads, head_dim] */
  void* value_pool;        /* device, same shape and dtype                           */
  int64_t num_pages;       /* > 0; num_pages * page_size < 2^31                      */
  int32_t page_size;       /* tokens per page, > 0                                   */
  int32_t num_kv_heads;    /* > 0                                                    */
  int32_t head_dim;        /* > 0                                                    */
  int32_t dtype;           /* pa_dtype                                               */
  /* e4m3 pools only (ignored otherwise): a stored code c stands for
   * e4m3(c) * scale; finite and > 0.  The pages name an fp8 KV cache (mobius
   * build features, maxtext pool-sizing table) without a scheme; one scale per
   * pool and tensor is the plainest one. */
  float k_scale;
  float v_scale;
} pa_kv_pool;

/*
 * paged_kv_append -- the ScatterND write (mobius PR #395, "How it works",
 * step 1; the aiter AppendKvJA step of maxtext PR #93).
 *
 *   for t in [0, num_tokens):  if slot_mapping[t] >= 0:
 *       key_pool.flat[slot_mapping[t]]   = key[t]
 *       value_pool.flat[slot_mapping[t]] = value[t]
 *
 * key, value    device [num_tokens, num_kv_heads, head_dim], pool dtype
 *               (bf16 for an e4m3 pool, 16-byte aligned: each element x is
 *               stored as e4m3_rn_satfinite(float32(x) / float32(scale)) --
 *               round to nearest even, magnitudes past 448 saturate, NaN
 *               stays NaN -- with the pool's k_scale / v_scale).
 * slot_mapping  device int64 [num_tokens]; entry = page_id * page_size +
 *               offset.  A negative entry marks a padding token (skipped).
 *               Entries must be unique within one call (otherwise which
 *               row lands is unspecified).  An entry >= num_pages*page_size
 *               is recorded in the device error word and skipped.
 * num_tokens    >= 0; 0 launches nothing.
 * The write is a bit copy (for f32 / bf16 pools): the pool afterwards is
 * bit-identical to the ScatterND result.
 */
pa_status paged_kv_append(const pa_kv_pool* pool, const void* key, const void* value,
                          const int64_t* slot_mapping, int64_t num_tokens, void* stream);

/*
 * paged_attention_decode -- one query token per sequence, attending to all
 * seq_lens[b] keys of its pages (mobius PR #395: Gather(pool, block_table)
 * then Attention with nonpad_kv_seqlen; decode is the one-token case).
 *
 *   out[b, h] = sum_j softmax_j(scale * q[b,h] . K_b[j, h/G]) V_b[j, h/G],
 *   j in [0, seq_lens[b]),  K_b[j] = key_pool[block_table[b, j / page_size],
 *                                             j % page_size]
 *
 * q, out        device [batch, num_q_heads, head_dim], pool dtype.  out may
 *               not alias q.  A sequence with seq_lens[b] == 0 gets out = 0.
 * block_table   device int32 [batch, max_blocks_per_seq], row-padded; entries
 *               past ceil(seq_lens[b] / page_size) are never read.
 * seq_lens      device int32 [batch], the KV length including this step's
 *               appended token (append first, then attend).
 * max_seq_len   host upper bound of seq_lens (used to size the launch).
 * workspace     device scratch of at least
 *               paged_attention_decode_workspace_size(...) bytes (may be NULL
 *               when that size is 0), 16-byte aligned, owned by the caller and
 *               not shared by calls in flight at the same time.  Its
 *               contents need no initialisation: each call writes every
 *               partial it reads, and the per-segment arrival counters that
 *               schedule the merge of a segment cut across CTAs carry a tag
 *               derived from a per-launch epoch kept at the workspace's start
 *               (each launch reads it and stores the next), so a word left by
 *               any earlier launch, a CUDA graph replay included, or never
 *               written counts as zero.  The merge runs inside the one
 *               decode kernel (no second launch).
 * The decode kernel is a persistent grid of at most one CTA per SM, launched
 * cooperatively (all CTAs resident at once: the CTAs that computed the parts
 * of a cut segment each merge a slice of it), so its start can wait for SMs
 * held by kernels on other streams.  Where the runtime refuses that launch,
 * the CTA that counts a segment's last part merges the whole segment.
 * bf16 path (tensor cores): page_size a power of two >= 8, head_dim in
 * {64, 128}, at most 32 query heads per KV head, q 16-byte aligned, at most
 * 2^31 - 1 slots (num_pages * page_size) per pool and batch *
 * ceil(max_seq_len / 16) below 2^31 (PA_ERR_RANGE beyond);
 * e4m3 pools: the bf16 limits; q and out are bf16; the attention is that of
 * the values the codes stand for (scale * k_scale * q . e4m3(K), outputs
 * times v_scale), computed with f16 products (every e4m3 value is an f16);
 * CUDA-core path (fp32 arithmetic, one key at a time; correct, not fast):
 * f32 pools, and bf16 pools of any other page_size (1, 2, 4, or not a power
 * of two); head_dim <= 256, no workspace used.
 */
size_t paged_attention_decode_workspace_size(int32_t batch, int32_t num_q_heads,
                                             int32_t num_kv_heads, int32_t head_dim,
                                             int32_t dtype);

pa_status paged_attention_decode(const pa_kv_pool* pool, const void* q, void* out,
                                 int32_t batch, int32_t num_q_heads,
                                 const int32_t* block_table, int32_t max_blocks_per_seq,
                                 const int32_t* seq_lens, int32_t max_seq_len, float scale,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * CSR page tables.  paged_attention_decode_csr / paged_attention_prefill_csr
 * are paged_attention_decode / paged_attention_prefill with each sequence's
 * pages given in the compressed form of NVIDIA/recsys-examples PR #400
 * (KVCacheMetadata: kv_indices, kv_indptr, kv_last_page_len) instead of a
 * row-padded block_table and seq_lens:
 *
 *   pages of sequence b = kv_indices[kv_indptr[b] .. kv_indptr[b+1]),
 *   L_b = (kv_indptr[b+1] - kv_indptr[b] - 1) * page_size + kv_last_page_len[b]
 *         (0 when the sequence has no page),
 *
 * i.e. the last page holds kv_last_page_len[b] tokens, 1 .. page_size.
 *
 * kv_indptr         device int32 [batch + 1], non-decreasing, kv_indptr[0] >= 0,
 *                   kv_indptr[batch] <= num_kv_indices.
 * kv_indices        device int32 [num_kv_indices], physical page ids.
 * kv_last_page_len  device int32 [batch].
 * max_seq_len       host upper bound of every L_b.
 * Device contents the host cannot check: a slice of kv_indptr outside
 * [0, num_kv_indices] or running backwards is treated as an empty sequence and
 * a kv_last_page_len outside [1, page_size] is clamped; both are recorded in
 * the device error word (code 3, see paged_device_error).  Every other argument, and the
 * workspace of the decode call (paged_attention_decode_workspace_size), is as
 * for the row-padded calls.
 */
pa_status paged_attention_decode_csr(const pa_kv_pool* pool, const void* q, void* out,
                                     int32_t batch, int32_t num_q_heads,
                                     const int32_t* kv_indptr, const int32_t* kv_indices,
                                     int64_t num_kv_indices, const int32_t* kv_last_page_len,
                                     int32_t max_seq_len, float scale, void* workspace,
                                     size_t workspace_bytes, void* stream);

pa_status paged_attention_prefill_csr(const pa_kv_pool* pool, const void* q, void* out,
                                      int32_t batch, int32_t num_q_heads,
                                      const int32_t* query_start_loc, int64_t total_q,
                                      int32_t max_q_len, const int32_t* kv_indptr,
                                      const int32_t* kv_indices, int64_t num_kv_indices,
                                      const int32_t* kv_last_page_len, int32_t max_seq_len,
                                      float scale, void* stream);

/*
 * paged_attention_decode_cascade -- decode for a batch whose sequences all
 * begin with the same prefix on the same physical pages (block tables that
 * alias the pages of a common prompt prefix: the RadixAttention case of
 * mobius PR #395, summary; the page-granular prefix index of ROCm/maxtext
 * PR #93, prefix cache (M5) commit).  Sequence b attends to
 *
 *   the prefix_len tokens on prefix_block_ids, then
 *   its own seq_lens[b] tokens on block_table[b, ...],
 *
 * i.e. exactly paged_attention_decode over the concatenated key lists.  The
 * prefix is read once for all B query rows (one tensor-core pass with its keys
 * cut into chunks, fp32 partials) instead of once per sequence; each sequence's
 * own tokens go through the split-KV decode, and the partials of both are
 * merged per row.  The prefix pass runs on a second stream of the library's,
 * forked from `stream` and joined back to it with events (so stream order and
 * stream capture hold); that stream is created by the first cascade call on a
 * host thread, which must therefore come before any stream capture there.
 *
 * prefix_block_ids  device int32 [ceil(prefix_len / page_size)], the shared
 *                   pages in order (the prefix may end inside its last page).
 * prefix_len        tokens of the shared prefix, >= 0; 0 runs plain decode.
 * block_table, seq_lens, max_blocks_per_seq, max_seq_len
 *                   the sequences' OWN pages and token counts (excluding the
 *                   prefix); a sequence with seq_lens[b] == 0 attends to the
 *                   prefix alone.
 * q, out, scale     as for paged_attention_decode.
 * workspace         device scratch of at least
 *                   paged_attention_decode_cascade_workspace_size(...) bytes,
 *                   16-byte aligned; contents need no initialisation.
 * bf16 pools only (PA_ERR_UNSUPPORTED for f32), with the tensor-core limits
 * of paged_attention_decode (a page_size that is not a power of two >= 8
 * gives PA_ERR_UNSUPPORTED when prefix_len > 0).
 */
size_t paged_attention_decode_cascade_workspace_size(int32_t batch, int32_t num_q_heads,
                                                     int32_t num_kv_heads, int32_t head_dim,
                                                     int32_t dtype);

pa_status paged_attention_decode_cascade(const pa_kv_pool* pool, const void* q, void* out,
                                         int32_t batch, int32_t num_q_heads,
                                         const int32_t* prefix_block_ids, int32_t prefix_len,
                                         const int32_t* block_table, int32_t max_blocks_per_seq,
                                         const int32_t* seq_lens, int32_t max_seq_len, float scale,
                                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * paged_attention_decode_append -- one decode step in one launch: the append
 * of this step's K/V rows (paged_kv_append with one token per sequence) and
 * the decode that attends to them (mobius PR #395, "How it works (per
 * attention layer)": step 1 writes the new rows, step 2 attends).  The
 * result equals paged_kv_append(pool, key, value, slot_mapping, batch)
 * followed by paged_attention_decode(...) with the same arguments, provided
 *   (a) slot_mapping[b] >= 0 is the slot of sequence b's last key, position
 *       seq_lens[b] - 1 (block_table[b][(L-1)/page_size] * page_size +
 *       (L-1) % page_size) -- the new token of a decode step; and
 *   (b) no slot written by the call is a key of another sequence.
 * The new rows are written to the pool and, for each sequence, attended to
 * straight from key/value (the pool row is not read back).  An entry
 * breaking (a) is recorded in the device error word (code 2, detail = the
 * slot) and that sequence's output then attends to the new row in place of
 * its last key.  slot_mapping[b] < 0: sequence b has no new token (its keys
 * are all in the pool already).
 *
 * key, value    device [batch, num_kv_heads, head_dim] bf16 (f32 for f32
 *               pools), 16-byte aligned; e4m3 pools store their codes
 *               (quantised as paged_kv_append does).
 * slot_mapping  device int64 [batch], 8-byte aligned.
 * Every other argument, limit and the workspace are those of
 * paged_attention_decode.  The CUDA-core path (f32 pools, bf16 pools of
 * other page sizes) runs the append and the decode as two launches.
 */
pa_status paged_attention_decode_append(const pa_kv_pool* pool, const void* key, const void* value,
                                        const int64_t* slot_mapping, const void* q, void* out,
                                        int32_t batch, int32_t num_q_heads,
                                        const int32_t* block_table, int32_t max_blocks_per_seq,
                                        const int32_t* seq_lens, int32_t max_seq_len, float scale,
                                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * paged_attention_decode_static_scratch -- paged_attention_decode without a
 * caller-provided workspace.  The pages have no counterpart of this call: it
 * exists for callers that cannot allocate device memory, such as a plugin in
 * an inference runtime that owns all device memory and hands its plugins no
 * allocator, or a latency-critical serving loop that may not take
 * cudaMalloc's implicit synchronisation mid-step.
 *
 * The split-KV partials go to a file-scope device array of
 * PA_DECODE_STATIC_SCRATCH_BYTES that the library holds on every GPU that
 * loads it, until the process exits.  The call allocates nothing (no
 * cudaMalloc, no cudaFree, no allocating library routine).
 * - The first call on a device looks up the array's device address with
 *   that device current (cudaGetSymbolAddress); make that first call before
 *   any stream capture on the device.
 * - All calls share the one array, which keeps the last call's contents;
 *   calls whose kernels overlap on the GPU (different streams, or unordered
 *   host threads) race on it.  No part of it needs to start zeroed.
 * - The stream must belong to the current device (the array's address is
 *   that device's); a stream of another device gives PA_ERR_CUDA and nothing
 *   is launched.
 * - bf16 and e4m3 pools only (PA_ERR_UNSUPPORTED for f32, whose decode needs no
 *   workspace anyway).  A call whose partials would not fit, i.e. when
 *   paged_attention_decode_workspace_size(...) exceeds
 *   PA_DECODE_STATIC_SCRATCH_BYTES, returns PA_ERR_WORKSPACE and launches
 *   nothing.
 * Arguments, layout and results are those of paged_attention_decode.
 */
#define PA_DECODE_STATIC_SCRATCH_BYTES (8u << 20)

pa_status paged_attention_decode_static_scratch(const pa_kv_pool* pool, const void* q, void* out,
                                                int32_t batch, int32_t num_q_heads,
                                                const int32_t* block_table,
                                                int32_t max_blocks_per_seq,
                                                const int32_t* seq_lens, int32_t max_seq_len,
                                                float scale, void* stream);

/*
 * paged_attention_prefill -- varlen causal attention for a packed batch of
 * new tokens (query_start_loc layout of maxtext PR #93's vLLM-shaped
 * metadata; causal + padding masks from is_causal=1 and nonpad_kv_seqlen of
 * mobius PR #395).
 *
 * Sequence b owns packed rows [query_start_loc[b], query_start_loc[b+1]) of
 * q; with n_b rows and L_b = seq_lens[b], its row i is the token at absolute
 * position p = L_b - n_b + i and attends to keys 0..p of its pages (the new
 * tokens are the last n_b of the sequence, already appended).  A row with
 * p < 0 gets out = 0.
 *
 * q, out           device [total_q, num_q_heads, head_dim], pool dtype.
 * query_start_loc  device int32 [batch + 1], non-decreasing, [0] = 0,
 *                  [batch] = total_q.
 * max_q_len        host upper bound of n_b (sizes the launch).
 * block_table, seq_lens, max_seq_len, scale: as for decode.
 * bf16 path (tensor cores): page_size a power of two >= 8, head_dim in
 * {64, 128}, at most 32 query heads per KV head;
 * e4m3 pools: the bf16 limits, q 16-byte aligned; q and out are bf16; the
 * attention is that of the values the codes stand for (scale * k_scale *
 * q . e4m3(K), outputs times v_scale), computed with f16 products: q is
 * rounded to f16 (exact for bf16 values of magnitude 2^-14 .. 65504), the
 * codes are exact in f16, and the softmax weights are rounded to f16;
 * CUDA-core path (fp32 arithmetic): f32 pools, and bf16 pools of any other
 * page_size; head_dim <= 256.
 */
pa_status paged_attention_prefill(const pa_kv_pool* pool, const void* q, void* out,
                                  int32_t batch, int32_t num_q_heads,
                                  const int32_t* query_start_loc, int64_t total_q,
                                  int32_t max_q_len, const int32_t* block_table,
                                  int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  int32_t max_seq_len, float scale, void* stream);

/*
 * paged_device_error -- read and clear the device error word of the current
 * device.  Synchronises the device.  *code = 0 when no violation was seen,
 * else 1 = block_table / kv_indices entry out of range, 2 = slot out of
 * range, 3 = seq_len (or CSR kv_indptr / kv_last_page_len) out of range,
 * 4 = query_start_loc inconsistent, 5 = a bounded wait inside a kernel gave
 * up; *detail holds the offending value.  Either pointer may be NULL.
 */
pa_status paged_device_error(int64_t* code, int64_t* detail);

/*
 * pa_testing_decode_part_wait -- TEST HOOK, not for production use: the pages
 * have no counterpart.  paged_attention_decode (bf16 and e4m3 pools, same
 * arguments, same workspace) with the one wait inside the decode kernel that
 * depends on other CTAs -- a CTA holding part of a sequence's keys waits for
 * the other CTAs' parts before merging its slice of the rows -- given the
 * limit `wait_ns` (1 us .. 2 s; every public call uses 2 s) and
 * `extra_parts` (0 .. 1024) parts added to the count each such wait expects.
 * With extra_parts > 0 those parts never arrive, so every such wait runs out
 * after wait_ns: the kernel records code 5 (a bounded wait gave up) in the
 * device error word, finishes without those parts and returns; the outputs
 * of the affected sequences are then unspecified.  It exists so that the
 * failure path of the bounded wait can be exercised without a fault or a
 * hang; a later call on the same workspace is unaffected.  PA_ERR_RANGE for
 * a limit or count outside the ranges above.
 */
pa_status pa_testing_decode_part_wait(const pa_kv_pool* pool, const void* q, void* out,
                                      int32_t batch, int32_t num_q_heads,
                                      const int32_t* block_table, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t max_seq_len, float scale,
                                      void* workspace, size_t workspace_bytes, uint64_t wait_ns,
                                      int32_t extra_parts, void* stream);

/* Human-readable name of a status code (static storage). */
const char* pa_status_string(int32_t status);

/* PA_ABI_VERSION of the loaded library. */
int32_t pa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H_ */
