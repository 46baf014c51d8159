// Launch-side declarations shared between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Geometry of one layer's pool, as the kernels see it.
struct PoolGeom {
  const void* key_pool;
  const void* value_pool;
  int64_t num_pages;
  int32_t page_size;
  int32_t page_shift;     // log2(page_size) when page_size is a power of two, else -1
  int32_t num_kv_heads;
  int32_t head_dim;
};

// ---- append ---------------------------------------------------------------
struct AppendParams {
  void* key_pool;
  void* value_pool;
  const void* key;
  const void* value;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  int64_t num_slots;      // num_pages * page_size
  int64_t row_bytes;      // num_kv_heads * head_dim * elem_size (of the pool)
  unsigned long long* err;
  // e4m3 pools: key / value rows are bf16 and are quantised on the way in
  int32_t kv8;
  float k_scale, v_scale;
};
cudaError_t launch_append(const AppendParams& p, int vec_bytes, int num_sms, cudaStream_t s);

// ---- decode (bf16, split-KV over a balanced partition of 16-key blocks) ---
struct DecodeParams {
  PoolGeom pool;
  const void* q;          // [B, Hq, D] bf16
  void* out;              // [B, Hq, D] bf16
  const int32_t* block_table;      // dense rows, or kv_indices in the CSR form
  const int32_t* seq_lens;         // dense form
  const int32_t* kv_indptr;        // CSR form (nullptr: dense), see page_list_start / seq_keys
  const int32_t* kv_last_page_len; // CSR form
  int64_t kv_len;                  // CSR form: entries of kv_indices
  float* part_o;          // [slots, G, D] fp32 unnormalised partial outputs
  float2* part_ml;        // [slots, G] (running max in log2 units, denominator)
  // launch epoch word + grid arrival counter (2 words at a fixed place, the
  // workspace's start): every launch reads the epoch E, and the last of its
  // CTAs to have read it stores E + 1, so E differs between consecutive
  // launches on one workspace (CUDA graph replays included) whatever the
  // words held before
  unsigned long long* launch_epoch;
  // fused append + decode: this step's rows (bf16 [B, Hkv, D]) and their
  // slots (int64 [B]); new_k == nullptr for a plain decode.  The kernel writes
  // them to the pool (e4m3 pools: codes with k_quant / v_quant) and attends
  // to each sequence's new row from the input, not from the pool.
  const void* new_k;
  const void* new_v;
  const int64_t* new_slots;
  float k_quant;
  float v_quant;
  // 1: the grid is co-resident (cooperative launch), so every CTA that holds a
  // part of a cut segment waits for the segment's last part and merges its own
  // slice of the rows; 0: the CTA counting the last part merges all of them
  int32_t slice_merge;
  // [B * Hkv] arrival counters of segments cut across CTAs, tagged with E
  // (any other contents read as zero): the last CTA to finish its part of a
  // segment merges the segment's partials
  unsigned long long* seg_count;
  // Limit (ns) of a CTA's wait for the other parts of a cut segment (0: the
  // default limit of every bounded wait), and parts added to every cut
  // segment's expected count.  Both are 0 in every public call; the
  // wait-expiry test hook (pa_testing_decode_part_wait) sets them so that the
  // wait runs out within a short limit.
  unsigned long long part_wait_ns;
  int32_t test_extra_parts;
  int32_t heads_per_box;  // HB: KV heads loaded per TMA box (power of two <= 8)
  int32_t smem_budget;    // dynamic shared memory the stage ring is sized against
  int32_t batch;
  int32_t num_q_heads;
  int32_t group;          // G = Hq / Hkv
  int32_t max_blocks;     // block_table row length
  int32_t num_ctas;       // CTAs of the split kernel (partition count)
  float scale_log2;       // scale * log2(e)
  unsigned long long* err;
  // cascade decode: the keys of every sequence start with a shared prefix whose
  // partials (one set per key chunk) are merged in by the combine kernel; the
  // split kernel then never finalises a row itself.  pre_chunks == 0: plain decode.
  // e4m3 pools: K/V codes (k_scale is folded into scale_log2 on the host);
  // every finished row is multiplied by v_scale (1 for bf16 pools)
  int32_t kv8;
  float v_scale;
  const float* pre_o;     // [pre_chunks, B, Hq, D] fp32 unnormalised
  const float2* pre_ml;   // [pre_chunks, B, Hq] (reference max in log2 units, denominator)
  int32_t pre_chunks;
  // 32-row groups, and 16-row groups of few long sequences (the WC
  // instantiations, chosen when this is > 0): the weight of a segment
  // (sequence x head box) in the cut of the units into CTA ranges, in 16-key
  // blocks of the box (decode_segment_penalty).  0 for cascade decode, whose
  // combine kernel recomputes the plain cut.
  int32_t seg_penalty;
};
// Number of partial slots the split kernel may write for this launch.
int decode_heads_per_box(int32_t num_kv_heads, int32_t group, int32_t page_size);
int decode_segment_penalty(int32_t head_dim, int32_t heads_per_box, int32_t group, bool kv8, int32_t batch,
                           int32_t num_kv_heads, int32_t num_ctas);
int64_t decode_partial_slots(int32_t batch, int32_t num_kv_heads, int32_t num_ctas, int32_t heads_per_box);
int decode_num_ctas(int num_sms, int32_t batch, int32_t num_kv_heads, int32_t max_seq_len, int32_t heads_per_box);
// Launch the fused (append + decode) split kernel (decode_fused.cu).
cudaError_t launch_split_fused(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rt,
                               cudaStream_t s);
cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t s);
// Cascade: split kernel on s, then the combine after `prefix_done` (an event
// recorded once the prefix partials are written) has completed.
cudaError_t launch_decode_cascade_bf16(const DecodeParams& p, cudaStream_t s, cudaEvent_t prefix_done);
// Dynamic shared memory the bf16 decode split kernel needs.
// (size_t)-1 when no stage ring of >= 2 stages fits the budget.
size_t decode_smem_bytes(int head_dim, int group, int batch, int heads_per_box, int budget, bool kv8);

// TMA descriptor of a bf16 pool viewed as {64, rows, num_kv_heads,
// head_dim/64} (strides num_kv_heads*head_dim*2, head_dim*2 and 128 bytes),
// box {64, box_rows, box_heads, box_slabs}, 128-byte swizzle: a box lands as
// [slab][head][row][128 B].  False if the driver refuses it.
bool encode_pool_tmap(CUtensorMap* map, const void* base, int64_t rows, int num_kv_heads, int head_dim,
                      int box_rows, int box_heads, int box_slabs);
// The same pool as a 5-D tensor {64 dims, 8 slots, head_dim/64 slabs,
// slots/8 blocks, heads}: one box {64, 8, head_dim/64, box_blocks, 1} lands as
// [block][slab][8 slots][128 B] (128-byte swizzle), so 8-slot row groups sit at
// a uniform stride of head_dim*16 bytes whatever the page size.  Needs
// slots % 8 == 0.
bool encode_pool_tmap_blocked(CUtensorMap* map, const void* base, int64_t rows, int num_kv_heads, int head_dim,
                              int box_blocks);
// An e4m3 pool as a 3-D tensor {head_dim codes, slots, heads}: one box
// {head_dim, box_rows, box_heads} lands as [head][row][head_dim B], with
// `swizzle` each row's 16-byte chunks swizzled (128-byte swizzle for head_dim
// 128, 64-byte for 64), else rows plainly one after another.
bool encode_pool_tmap_u8(CUtensorMap* map, const void* base, int64_t rows, int num_kv_heads, int head_dim,
                         int box_rows, int box_heads, bool swizzle);

// ---- prefill (bf16) ------------------------------------------------------
struct PrefillParams {
  PoolGeom pool;
  const void* q;          // [T, Hq, D] bf16
  void* out;              // [T, Hq, D] bf16
  const int32_t* query_start_loc;
  const int32_t* block_table;      // dense rows, or kv_indices in the CSR form
  const int32_t* seq_lens;         // dense form
  const int32_t* kv_indptr;        // CSR form (nullptr: dense)
  const int32_t* kv_last_page_len; // CSR form
  int64_t kv_len;                  // CSR form: entries of kv_indices
  int64_t total_q;
  int32_t batch;
  int32_t num_q_heads;
  int32_t group;
  int32_t max_blocks;
  int32_t max_q_len;
  float scale_log2;
  unsigned long long* err;
  // Shared-prefix pass of cascade decode (part_o != nullptr): one sequence of
  // prefix_len keys on block_table row 0, queried by the batch's `batch_rows`
  // decode rows of q [batch_rows, Hq, D], none of them causal; key tiles are
  // cut into chunks of chunk_tiles (blockIdx.z = chunk) and every chunk writes
  // unnormalised partials instead of out.
  float* part_o;          // [chunks, batch_rows, Hq, D] fp32
  float2* part_ml;        // [chunks, batch_rows, Hq] (reference max in log2 units, denominator)
  int32_t batch_rows;
  int32_t prefix_len;
  int32_t chunk_tiles;
  // e4m3 pools: K/V codes, k_scale folded into scale_log2 on the host, every
  // output row multiplied by v_scale (1 for bf16 pools)
  int32_t kv8;
  float v_scale;
};
cudaError_t launch_prefill_bf16(const PrefillParams& p, cudaStream_t s);

// ---- fp32 path (decode = prefill with one row per sequence) --------------
// The CUDA-core path (attn_f32.cu): f32 pools, and bf16 pools whose page
// size the TMA boxes of the tensor-core kernels cannot take.
struct AttnF32Params {
  PoolGeom pool;
  const void* q;          // [rows, Hq, D], the pool's element type
  void* out;              // [rows, Hq, D], the pool's element type
  int32_t bf16;           // 1: q, pools and out are bf16 (fp32 arithmetic); 0: f32
  const int32_t* query_start_loc;  // null for decode (row b = sequence b, n_b = 1)
  const int32_t* block_table;      // dense rows, or kv_indices in the CSR form
  const int32_t* seq_lens;         // dense form
  const int32_t* kv_indptr;        // CSR form (nullptr: dense)
  const int32_t* kv_last_page_len; // CSR form
  int64_t kv_len;                  // CSR form: entries of kv_indices
  int64_t rows;
  int32_t batch;
  int32_t num_q_heads;
  int32_t group;
  int32_t max_blocks;
  float scale;
  unsigned long long* err;
};
cudaError_t launch_attn_f32(const AttnF32Params& p, int num_sms, cudaStream_t s);

}  // namespace pa
