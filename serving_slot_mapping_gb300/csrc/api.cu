// C ABI of libpagedattn.so (declared in include/paged_attn.h): host-side
// argument checks, launch-shape choices and dispatch to the kernels.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "../../include/paged_attn.h"
#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;

// One error word per device, written by kernels on a range violation.
__device__ unsigned long long g_error_word;

std::atomic<unsigned long long*> g_err_ptr[kMaxDevices];
std::atomic<int> g_num_sms[kMaxDevices];

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

unsigned long long* error_word() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  unsigned long long* p = g_err_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 1;
  int n = g_num_sms[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    g_num_sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int max_smem_optin() {
  const int dev = current_device();
  int v = 0;
  if (dev < 0 || cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  return v;
}

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t elem_size(int32_t dtype) { return dtype == PA_DTYPE_F32 ? 4 : (dtype == PA_DTYPE_FP8_E4M3 ? 1 : 2); }

bool kv8(const pa_kv_pool* pool) { return pool->dtype == PA_DTYPE_FP8_E4M3; }

// Pages the TMA boxes of the tensor-core kernels take: whole 8-slot blocks.
bool tma_pages(const pa_kv_pool* pool) { return is_pow2(pool->page_size) && pool->page_size >= 8; }

// The CUDA-core attention path (attn_f32.cu): f32 pools, and bf16 pools of
// other page sizes (1, 2, 4, or not a power of two).
bool core_path(const pa_kv_pool* pool) {
  return pool->dtype == PA_DTYPE_F32 || (pool->dtype == PA_DTYPE_BF16 && !tma_pages(pool));
}

pa_status check_pool(const pa_kv_pool* pool) {
  if (pool == nullptr || pool->key_pool == nullptr || pool->value_pool == nullptr) return PA_ERR_NULL;
  if (pool->dtype != PA_DTYPE_F32 && pool->dtype != PA_DTYPE_BF16 && pool->dtype != PA_DTYPE_FP8_E4M3)
    return PA_ERR_DTYPE;
  if (kv8(pool) && !(std::isfinite(pool->k_scale) && pool->k_scale > 0.f && std::isfinite(pool->v_scale) &&
                     pool->v_scale > 0.f))
    return PA_ERR_RANGE;
  if (pool->num_pages <= 0 || pool->page_size <= 0 || pool->num_kv_heads <= 0 || pool->head_dim <= 0)
    return PA_ERR_SHAPE;
  if (pool->num_pages > INT32_MAX) return PA_ERR_RANGE;
  const size_t es = elem_size(pool->dtype);
  if (!aligned(pool->key_pool, es) || !aligned(pool->value_pool, es)) return PA_ERR_ALIGN;
  return PA_OK;
}

pa::PoolGeom geom(const pa_kv_pool* pool) {
  pa::PoolGeom g;
  g.key_pool = pool->key_pool;
  g.value_pool = pool->value_pool;
  g.num_pages = pool->num_pages;
  g.page_size = pool->page_size;
  g.page_shift = is_pow2(pool->page_size) ? pa::ilog2_pow2(pool->page_size) : -1;
  g.num_kv_heads = pool->num_kv_heads;
  g.head_dim = pool->head_dim;
  return g;
}

// Shape checks common to decode and prefill.
pa_status check_attention(const pa_kv_pool* pool, int32_t batch, int32_t num_q_heads,
                          int32_t max_blocks_per_seq, int32_t max_seq_len, float scale) {
  pa_status st = check_pool(pool);
  if (st != PA_OK) return st;
  if (batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0) return PA_ERR_SHAPE;
  if (num_q_heads % pool->num_kv_heads != 0) return PA_ERR_SHAPE;
  if ((int64_t)max_blocks_per_seq * pool->page_size > INT32_MAX) return PA_ERR_RANGE;
  if ((int64_t)max_seq_len > (int64_t)max_blocks_per_seq * pool->page_size) return PA_ERR_SHAPE;
  if (!std::isfinite(scale)) return PA_ERR_RANGE;
  if (!core_path(pool)) {  // bf16 and e4m3: the TMA / tensor-core paths
    if (pool->head_dim != 64 && pool->head_dim != 128) return PA_ERR_UNSUPPORTED;
    // page-sized TMA boxes of 8-slot blocks (e4m3 pools have no other path)
    if (!tma_pages(pool)) return PA_ERR_UNSUPPORTED;
    if (num_q_heads / pool->num_kv_heads > 32) return PA_ERR_UNSUPPORTED;
    if (!aligned(pool->key_pool, 16) || !aligned(pool->value_pool, 16)) return PA_ERR_ALIGN;
  } else {
    if (pool->head_dim > 256) return PA_ERR_UNSUPPORTED;
  }
  return PA_OK;
}

constexpr double kLog2e = 1.4426950408889634;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t decode_ws_bytes(int32_t batch, int32_t hq, int32_t hkv, int32_t d, int ctas, int hb) {
  if (batch <= 0 || hq <= 0 || hkv <= 0 || d <= 0) return 0;
  const int64_t slots = pa::decode_partial_slots(batch, hkv, ctas, hb);
  const int64_t g = hq / hkv;
  // [launch epoch, grid counter | pad] [partial o] [partial (m, l)] [segment counters]
  return 256 + align_up((size_t)(slots * g * d * 4), 256) + align_up((size_t)(slots * g * 8), 256) +
         align_up((size_t)batch * hkv * 8, 256);
}

}  // namespace

extern "C" {

int32_t pa_abi_version(void) { return PA_ABI_VERSION; }

const char* pa_status_string(int32_t status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULL: return "PA_ERR_NULL: a required pointer is NULL";
    case PA_ERR_SHAPE: return "PA_ERR_SHAPE: inconsistent or negative sizes";
    case PA_ERR_DTYPE: return "PA_ERR_DTYPE: unknown dtype";
    case PA_ERR_RANGE: return "PA_ERR_RANGE: a value is outside the supported range";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: head_dim/page_size/group not implemented";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: a CUDA runtime call failed";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN: a pointer is misaligned";
    default: return "unknown pa_status";
  }
}

pa_status paged_kv_append(const pa_kv_pool* pool, const void* key, const void* value,
                          const int64_t* slot_mapping, int64_t num_tokens, void* stream) {
  pa_status st = check_pool(pool);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (key == nullptr || value == nullptr || slot_mapping == nullptr) return PA_ERR_NULL;
  if (!aligned(slot_mapping, 8)) return PA_ERR_ALIGN;
  const size_t es = elem_size(pool->dtype);
  pa::AppendParams p{};
  p.key_pool = pool->key_pool;
  p.value_pool = pool->value_pool;
  p.key = key;
  p.value = value;
  p.slot_mapping = slot_mapping;
  p.num_tokens = num_tokens;
  p.num_slots = pool->num_pages * (int64_t)pool->page_size;
  p.row_bytes = (int64_t)pool->num_kv_heads * pool->head_dim * (int64_t)es;
  p.err = error_word();
  if (kv8(pool)) {  // bf16 rows in, e4m3 codes out, 8 elements per step
    if (p.row_bytes % 8 != 0) return PA_ERR_UNSUPPORTED;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(pool->key_pool, 8) || !aligned(pool->value_pool, 8))
      return PA_ERR_ALIGN;
    p.kv8 = 1;
    p.k_scale = pool->k_scale;
    p.v_scale = pool->v_scale;
    cudaError_t e = pa::launch_append(p, 8, num_sms(), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  int vec = 16;
  while (vec > (int)es && ((p.row_bytes % vec) != 0 || !aligned(key, vec) || !aligned(value, vec) ||
                           !aligned(pool->key_pool, vec) || !aligned(pool->value_pool, vec)))
    vec >>= 1;
  if (!aligned(key, es) || !aligned(value, es)) return PA_ERR_ALIGN;
  cudaError_t e = pa::launch_append(p, vec, num_sms(), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t paged_attention_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_dim, int32_t dtype) {
  if (dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_FP8_E4M3) return 0;
  if (num_kv_heads <= 0 || num_q_heads <= 0) return 0;
  // heads per box for page_size >= 16 is an upper bound for every page size
  const int hb = pa::decode_heads_per_box(num_kv_heads, num_q_heads / num_kv_heads, 16);
  return decode_ws_bytes(batch, num_q_heads, num_kv_heads, head_dim, num_sms(), hb);
}

namespace {

// Host view of the page-table arguments: the dense form (block_table rows +
// seq_lens) or the CSR form (kv_indptr slices of kv_indices +
// kv_last_page_len); the kernels read either through page_list_start /
// seq_keys.
struct Table {
  const int32_t* ids = nullptr;       // block_table, or kv_indices
  const int32_t* seq_lens = nullptr;  // dense
  const int32_t* indptr = nullptr;    // CSR
  const int32_t* last = nullptr;      // CSR
  int64_t kv_len = 0;                 // CSR: entries of kv_indices
  int32_t max_blocks = 0;             // dense row length (CSR: ceil(max_seq_len / page_size))
};

pa_status check_table(const Table& t) {
  if (t.ids == nullptr) return PA_ERR_NULL;
  if (t.indptr == nullptr ? t.seq_lens == nullptr : t.last == nullptr) return PA_ERR_NULL;
  if (!aligned(t.ids, 4) || !aligned(t.seq_lens, 4) || !aligned(t.indptr, 4) || !aligned(t.last, 4))
    return PA_ERR_ALIGN;
  if (t.indptr != nullptr && t.kv_len < 0) return PA_ERR_SHAPE;
  return PA_OK;
}

Table dense_table(const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens) {
  Table t;
  t.ids = block_table;
  t.seq_lens = seq_lens;
  t.max_blocks = max_blocks;
  return t;
}

// Launch parameters of the bf16 split-KV decode (shared by plain and cascade
// decode); the partials take the first bytes of the workspace.
pa_status bf16_decode_params(const pa_kv_pool* pool, const void* q, void* out, int32_t batch,
                             int32_t num_q_heads, const Table& t, int32_t max_seq_len, float scale, void* workspace,
                             size_t workspace_bytes, pa::DecodeParams* p, int reserved_sms = 0) {
  const int32_t group = num_q_heads / pool->num_kv_heads;
  // the decode kernel's TMA boxes address a pool row (slot) with a 32-bit
  // coordinate: at most 2^31 - 1 slots per pool
  if (pool->num_pages * (int64_t)pool->page_size > INT32_MAX) return PA_ERR_RANGE;
  // ... and counts the batch's 16-key blocks (shared pages counted per
  // sequence) in 32 bits
  if ((int64_t)batch * (((int64_t)max_seq_len + 15) / 16) > INT32_MAX) return PA_ERR_RANGE;
  if (!aligned(q, 16) || !aligned(out, 4)) return PA_ERR_ALIGN;
  const int hb = pa::decode_heads_per_box(pool->num_kv_heads, group, pool->page_size);
  const int sms = num_sms() - reserved_sms;
  const int ctas = pa::decode_num_ctas(sms < 1 ? 1 : sms, batch, pool->num_kv_heads, max_seq_len, hb);
  const size_t need = decode_ws_bytes(batch, num_q_heads, pool->num_kv_heads, pool->head_dim, ctas, hb);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return PA_ERR_ALIGN;
  const int budget = max_smem_optin();
  if (pa::decode_smem_bytes(pool->head_dim, group, batch, hb, budget, kv8(pool)) > (size_t)budget)
    return PA_ERR_UNSUPPORTED;
  const int64_t slots = pa::decode_partial_slots(batch, pool->num_kv_heads, ctas, hb);
  *p = pa::DecodeParams{};
  p->pool = geom(pool);
  p->q = q;
  p->out = out;
  p->block_table = t.ids;
  p->seq_lens = t.seq_lens;
  p->kv_indptr = t.indptr;
  p->kv_last_page_len = t.last;
  p->kv_len = t.kv_len;
  char* ws = static_cast<char*>(workspace);
  p->launch_epoch = reinterpret_cast<unsigned long long*>(ws);
  p->part_o = reinterpret_cast<float*>(ws + 256);
  const size_t o_bytes = align_up((size_t)(slots * group * pool->head_dim * 4), 256);
  p->part_ml = reinterpret_cast<float2*>(ws + 256 + o_bytes);
  p->seg_count = reinterpret_cast<unsigned long long*>(ws + 256 + o_bytes + align_up((size_t)(slots * group * 8), 256));
  p->batch = batch;
  p->num_q_heads = num_q_heads;
  p->group = group;
  p->max_blocks = t.max_blocks;
  p->num_ctas = ctas;
  p->heads_per_box = hb;
  p->smem_budget = budget;
  // e4m3 pools: S = scale * k_scale * q . e4m3(K), O = v_scale * softmax(S) e4m3(V)
  p->kv8 = kv8(pool) ? 1 : 0;
  p->scale_log2 = (float)((double)scale * (kv8(pool) ? (double)pool->k_scale : 1.0) * kLog2e);
  p->v_scale = kv8(pool) ? pool->v_scale : 1.f;
  // segment changes weigh in the cut (32-row groups; 16-row groups of few long
  // sequences); positions are counted in 32 bits
  const int pen = pa::decode_segment_penalty(pool->head_dim, hb, group, kv8(pool), batch, pool->num_kv_heads, ctas);
  const int64_t max_keys = std::max<int64_t>(max_seq_len, (int64_t)t.max_blocks * pool->page_size);
  p->seg_penalty = (int64_t)batch * ((max_keys + 15) / 16 + pen) <= INT32_MAX ? pen : 0;
  p->err = error_word();
  return PA_OK;
}

// Cascade decode, prefix pass: key chunks per (row tile, KV head), an upper
// bound on the chunk count.  The prefix pass runs beside the split kernel
// (which leaves it the SMs it needs), so it takes about a quarter of the SMs
// (num_SMs / 4 CTAs in all); fewer chunks also mean fewer fp32 partials
// (B*Hq*D*4 bytes each) for the combine kernel to read back.
int cascade_chunk_target(int32_t batch, int32_t group, int32_t num_kv_heads) {
  const int64_t row_ctas = ((int64_t)batch * group + 255) / 256;
  const int64_t t = num_sms() / (4 * row_ctas * num_kv_heads);
  return (int)(t < 1 ? 1 : t);
}

// A second stream per (host thread, device) on which the cascade's prefix pass
// runs beside the split kernel: forked from and joined back to the caller's
// stream with events, so the order is kept and stream capture records a fork
// and a join.  Created on first use (make the first cascade call on a thread
// before capturing) and kept for the life of the thread.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

SideStream* side_stream() {
  constexpr int kMaxDev = 64;
  thread_local SideStream side[kMaxDev];
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDev) return nullptr;
  SideStream& ss = side[dev];
  if (ss.stream == nullptr) {
    if (cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
  }
  return &ss;
}

size_t cascade_prefix_bytes(int chunks, int32_t batch, int32_t num_q_heads, int32_t head_dim) {
  const size_t rows = (size_t)chunks * batch * num_q_heads;
  return align_up(rows * head_dim * 4, 256) + align_up(rows * 8, 256);
}

}  // namespace

namespace {

pa_status decode_impl(const pa_kv_pool* pool, const void* q, void* out, int32_t batch, int32_t num_q_heads,
                      const Table& t, int32_t max_seq_len, float scale, void* workspace, size_t workspace_bytes,
                      void* stream) {
  pa_status st = check_attention(pool, batch, num_q_heads, t.max_blocks, max_seq_len, scale);
  if (st != PA_OK) return st;
  if (batch == 0) return PA_OK;
  if (q == nullptr || out == nullptr) return PA_ERR_NULL;
  st = check_table(t);
  if (st != PA_OK) return st;
  if (q == out) return PA_ERR_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (core_path(pool)) {
    if (!aligned(q, elem_size(pool->dtype)) || !aligned(out, elem_size(pool->dtype))) return PA_ERR_ALIGN;
    pa::AttnF32Params p{};
    p.pool = geom(pool);
    p.q = q;
    p.out = out;
    p.bf16 = pool->dtype == PA_DTYPE_BF16 ? 1 : 0;
    p.query_start_loc = nullptr;
    p.block_table = t.ids;
    p.seq_lens = t.seq_lens;
    p.kv_indptr = t.indptr;
    p.kv_last_page_len = t.last;
    p.kv_len = t.kv_len;
    p.rows = batch;
    p.batch = batch;
    p.num_q_heads = num_q_heads;
    p.group = num_q_heads / pool->num_kv_heads;
    p.max_blocks = t.max_blocks;
    p.scale = scale;
    p.err = error_word();
    return pa::launch_attn_f32(p, num_sms(), s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  pa::DecodeParams p;
  st = bf16_decode_params(pool, q, out, batch, num_q_heads, t, max_seq_len, scale, workspace, workspace_bytes, &p);
  if (st != PA_OK) return st;
  return pa::launch_decode_bf16(p, s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status prefill_impl(const pa_kv_pool* pool, const void* q, void* out, int32_t batch, int32_t num_q_heads,
                       const int32_t* query_start_loc, int64_t total_q, int32_t max_q_len, const Table& t,
                       int32_t max_seq_len, float scale, void* stream) {
  pa_status st = check_attention(pool, batch, num_q_heads, t.max_blocks, max_seq_len, scale);
  if (st != PA_OK) return st;
  if (total_q < 0 || max_q_len < 0 || total_q > INT32_MAX) return PA_ERR_SHAPE;
  if (batch == 0 || total_q == 0) return PA_OK;
  if (max_q_len == 0) return PA_ERR_SHAPE;
  if (q == nullptr || out == nullptr || query_start_loc == nullptr) return PA_ERR_NULL;
  st = check_table(t);
  if (st != PA_OK) return st;
  if (q == out) return PA_ERR_SHAPE;
  if (!aligned(query_start_loc, 4)) return PA_ERR_ALIGN;
  if (!aligned(q, 4) || !aligned(out, 4)) return PA_ERR_ALIGN;
  if (kv8(pool) && !aligned(q, 16)) return PA_ERR_ALIGN;  // e4m3 pools: q rows read 16 bytes at a time
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const pa::PoolGeom g = geom(pool);
  const int32_t group = num_q_heads / pool->num_kv_heads;
  if (core_path(pool)) {
    pa::AttnF32Params p{};
    p.pool = g;
    p.q = q;
    p.out = out;
    p.bf16 = pool->dtype == PA_DTYPE_BF16 ? 1 : 0;
    p.query_start_loc = query_start_loc;
    p.block_table = t.ids;
    p.seq_lens = t.seq_lens;
    p.kv_indptr = t.indptr;
    p.kv_last_page_len = t.last;
    p.kv_len = t.kv_len;
    p.rows = total_q;
    p.batch = batch;
    p.num_q_heads = num_q_heads;
    p.group = group;
    p.max_blocks = t.max_blocks;
    p.scale = scale;
    p.err = error_word();
    return pa::launch_attn_f32(p, num_sms(), s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  if (batch > 65535 || pool->num_kv_heads > 65535) return PA_ERR_RANGE;  // grid y/z limits
  // a sequence's packed rows (token x G heads of one KV head) are 32-bit in the kernel
  if ((int64_t)max_q_len * group > INT32_MAX / 2) return PA_ERR_RANGE;
  pa::PrefillParams p{};
  p.pool = g;
  p.q = q;
  p.out = out;
  p.query_start_loc = query_start_loc;
  p.block_table = t.ids;
  p.seq_lens = t.seq_lens;
  p.kv_indptr = t.indptr;
  p.kv_last_page_len = t.last;
  p.kv_len = t.kv_len;
  p.total_q = total_q;
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.group = group;
  p.max_blocks = t.max_blocks;
  p.max_q_len = max_q_len;
  // e4m3 pools: S = scale * k_scale * q . e4m3(K), O = v_scale * softmax(S) e4m3(V)
  p.kv8 = kv8(pool) ? 1 : 0;
  p.scale_log2 = (float)((double)scale * (kv8(pool) ? (double)pool->k_scale : 1.0) * kLog2e);
  p.v_scale = kv8(pool) ? pool->v_scale : 1.f;
  p.err = error_word();
  return pa::launch_prefill_bf16(p, s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// The CSR form as a Table; max_seq_len bounds every sequence's keys.
pa_status csr_table(const pa_kv_pool* pool, const int32_t* kv_indptr, const int32_t* kv_indices, int64_t kv_len,
                    const int32_t* kv_last_page_len, int32_t max_seq_len, Table* t) {
  if (pool == nullptr || pool->page_size <= 0) return PA_ERR_NULL;
  if (kv_indptr == nullptr) return PA_ERR_NULL;
  if (max_seq_len < 0 || kv_len < 0) return PA_ERR_SHAPE;
  *t = Table{};
  t->ids = kv_indices;
  t->indptr = kv_indptr;
  t->last = kv_last_page_len;
  t->kv_len = kv_len;
  const int64_t mb = ((int64_t)max_seq_len + pool->page_size - 1) / pool->page_size;
  t->max_blocks = (int32_t)(mb < 1 ? 1 : mb);
  return PA_OK;
}

}  // namespace

pa_status paged_attention_decode(const pa_kv_pool* pool, const void* q, void* out, int32_t batch,
                                 int32_t num_q_heads, const int32_t* block_table,
                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 int32_t max_seq_len, float scale, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return decode_impl(pool, q, out, batch, num_q_heads, dense_table(block_table, max_blocks_per_seq, seq_lens),
                     max_seq_len, scale, workspace, workspace_bytes, stream);
}

pa_status pa_testing_decode_part_wait(const pa_kv_pool* pool, const void* q, void* out, int32_t batch,
                                      int32_t num_q_heads, const int32_t* block_table,
                                      int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len,
                                      float scale, void* workspace, size_t workspace_bytes, uint64_t wait_ns,
                                      int32_t extra_parts, void* stream) {
  if (pool == nullptr) return PA_ERR_NULL;
  if (pool->dtype != PA_DTYPE_BF16 && pool->dtype != PA_DTYPE_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  if (!tma_pages(pool)) return PA_ERR_UNSUPPORTED;  // the CUDA-core path has no wait
  // a short limit (1 us .. 2 s) and a bounded count: the hook can only
  // shorten a wait, never lengthen one
  if (wait_ns < 1000u || wait_ns > 2000000000u || extra_parts < 0 || extra_parts > 1024) return PA_ERR_RANGE;
  const Table t = dense_table(block_table, max_blocks_per_seq, seq_lens);
  pa_status st = check_attention(pool, batch, num_q_heads, t.max_blocks, max_seq_len, scale);
  if (st != PA_OK) return st;
  if (batch == 0) return PA_OK;
  if (q == nullptr || out == nullptr) return PA_ERR_NULL;
  st = check_table(t);
  if (st != PA_OK) return st;
  if (q == out) return PA_ERR_SHAPE;
  pa::DecodeParams p;
  st = bf16_decode_params(pool, q, out, batch, num_q_heads, t, max_seq_len, scale, workspace, workspace_bytes, &p);
  if (st != PA_OK) return st;
  p.part_wait_ns = wait_ns;
  p.test_extra_parts = extra_parts;
  return pa::launch_decode_bf16(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status paged_attention_decode_append(const pa_kv_pool* pool, const void* key, const void* value,
                                        const int64_t* slot_mapping, const void* q, void* out, int32_t batch,
                                        int32_t num_q_heads, const int32_t* block_table,
                                        int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                        int32_t max_seq_len, float scale, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  const Table t = dense_table(block_table, max_blocks_per_seq, seq_lens);
  pa_status st = check_attention(pool, batch, num_q_heads, t.max_blocks, max_seq_len, scale);
  if (st != PA_OK) return st;
  if (batch == 0) return PA_OK;
  if (q == nullptr || out == nullptr || key == nullptr || value == nullptr || slot_mapping == nullptr)
    return PA_ERR_NULL;
  st = check_table(t);
  if (st != PA_OK) return st;
  if (q == out) return PA_ERR_SHAPE;
  if (!aligned(slot_mapping, 8)) return PA_ERR_ALIGN;
  if (core_path(pool)) {  // the CUDA-core path: append and decode as two launches
    st = paged_kv_append(pool, key, value, slot_mapping, batch, stream);
    if (st != PA_OK) return st;
    return decode_impl(pool, q, out, batch, num_q_heads, t, max_seq_len, scale, workspace, workspace_bytes, stream);
  }
  if (!aligned(key, 16) || !aligned(value, 16)) return PA_ERR_ALIGN;  // 8 bf16 elements per access
  pa::DecodeParams p;
  st = bf16_decode_params(pool, q, out, batch, num_q_heads, t, max_seq_len, scale, workspace, workspace_bytes, &p);
  if (st != PA_OK) return st;
  p.new_k = key;
  p.new_v = value;
  p.new_slots = slot_mapping;
  p.k_quant = kv8(pool) ? pool->k_scale : 1.f;
  p.v_quant = kv8(pool) ? pool->v_scale : 1.f;
  return pa::launch_decode_bf16(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status paged_attention_decode_csr(const pa_kv_pool* pool, const void* q, void* out, int32_t batch,
                                     int32_t num_q_heads, const int32_t* kv_indptr, const int32_t* kv_indices,
                                     int64_t num_kv_indices, const int32_t* kv_last_page_len,
                                     int32_t max_seq_len, float scale, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  Table t;
  const pa_status st = csr_table(pool, kv_indptr, kv_indices, num_kv_indices, kv_last_page_len, max_seq_len, &t);
  if (st != PA_OK) return st;
  return decode_impl(pool, q, out, batch, num_q_heads, t, max_seq_len, scale, workspace, workspace_bytes, stream);
}

size_t paged_attention_decode_cascade_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                                     int32_t head_dim, int32_t dtype) {
  if (dtype != PA_DTYPE_BF16) return 0;
  if (num_kv_heads <= 0 || num_q_heads <= 0 || batch <= 0 || num_q_heads % num_kv_heads != 0) return 0;
  const int target = cascade_chunk_target(batch, num_q_heads / num_kv_heads, num_kv_heads);
  return paged_attention_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, dtype) +
         cascade_prefix_bytes(target, batch, num_q_heads, head_dim);
}

pa_status paged_attention_decode_cascade(const pa_kv_pool* pool, const void* q, void* out, int32_t batch,
                                         int32_t num_q_heads, const int32_t* prefix_block_ids, int32_t prefix_len,
                                         const int32_t* block_table, int32_t max_blocks_per_seq,
                                         const int32_t* seq_lens, int32_t max_seq_len, float scale,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  pa_status st = check_attention(pool, batch, num_q_heads, max_blocks_per_seq, max_seq_len, scale);
  if (st != PA_OK) return st;
  if (pool->dtype != PA_DTYPE_BF16) return PA_ERR_UNSUPPORTED;
  if (prefix_len < 0) return PA_ERR_SHAPE;
  if (batch == 0) return PA_OK;
  if (prefix_len == 0)  // nothing shared: plain decode (its workspace is a prefix of this one's)
    return paged_attention_decode(pool, q, out, batch, num_q_heads, block_table, max_blocks_per_seq, seq_lens,
                                  max_seq_len, scale, workspace, workspace_bytes, stream);
  if (!tma_pages(pool)) return PA_ERR_UNSUPPORTED;  // the prefix pass is the tensor-core kernel
  if (q == nullptr || out == nullptr || block_table == nullptr || seq_lens == nullptr ||
      prefix_block_ids == nullptr)
    return PA_ERR_NULL;
  if (q == out) return PA_ERR_SHAPE;
  if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(prefix_block_ids, 4)) return PA_ERR_ALIGN;
  if ((int64_t)batch * (num_q_heads / pool->num_kv_heads) > INT32_MAX / 2) return PA_ERR_RANGE;
  if (pool->num_kv_heads > 65535) return PA_ERR_RANGE;  // grid y
  const int32_t group = num_q_heads / pool->num_kv_heads;
  const size_t dec_bound =
      paged_attention_decode_workspace_size(batch, num_q_heads, pool->num_kv_heads, pool->head_dim, PA_DTYPE_BF16);
  const int target = cascade_chunk_target(batch, group, pool->num_kv_heads);
  const size_t need = dec_bound + cascade_prefix_bytes(target, batch, num_q_heads, pool->head_dim);
  if (workspace == nullptr || workspace_bytes < need) return PA_ERR_WORKSPACE;
  // prefix pass: the B decode rows against the shared pages, one set of
  // partials per key chunk, placed after the decode partials
  const int nt = (prefix_len + 127) / 128;
  const int chunk_tiles = (nt + target - 1) / target;
  const int chunks = (nt + chunk_tiles - 1) / chunk_tiles;
  const int prefix_ctas = (int)(((int64_t)batch * group + 255) / 256) * pool->num_kv_heads * chunks;
  pa::DecodeParams p;
  st = bf16_decode_params(pool, q, out, batch, num_q_heads, dense_table(block_table, max_blocks_per_seq, seq_lens),
                          max_seq_len, scale, workspace, dec_bound, &p, prefix_ctas);
  if (st != PA_OK) return st;
  float* pre_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + dec_bound);
  const size_t pre_rows = (size_t)chunks * batch * num_q_heads;
  float2* pre_ml = reinterpret_cast<float2*>(reinterpret_cast<char*>(pre_o) +
                                             align_up(pre_rows * pool->head_dim * 4, 256));
  pa::PrefillParams pp{};
  pp.pool = p.pool;
  pp.q = q;
  pp.out = nullptr;
  pp.block_table = prefix_block_ids;
  pp.total_q = batch;
  pp.batch = 1;
  pp.num_q_heads = num_q_heads;
  pp.group = group;
  pp.max_blocks = (prefix_len + pool->page_size - 1) / pool->page_size;
  pp.max_q_len = batch;
  pp.scale_log2 = p.scale_log2;
  pp.err = p.err;
  pp.part_o = pre_o;
  pp.part_ml = pre_ml;
  pp.batch_rows = batch;
  pp.prefix_len = prefix_len;
  pp.chunk_tiles = chunk_tiles;
  pp.v_scale = 1.f;
  p.pre_o = pre_o;
  p.pre_ml = pre_ml;
  p.pre_chunks = chunks;
  p.seg_penalty = 0;  // the combine kernel recomputes the plain cut of the units
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SideStream* side = side_stream();
  if (side == nullptr) return PA_ERR_CUDA;
  // fork: the prefix pass starts after everything already queued on s
  if (cudaEventRecord(side->fork, s) != cudaSuccess || cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess)
    return PA_ERR_CUDA;
  if (pa::launch_prefill_bf16(pp, side->stream) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaEventRecord(side->join, side->stream) != cudaSuccess) return PA_ERR_CUDA;
  // the split kernel runs meanwhile on s; the combine waits for both
  return pa::launch_decode_cascade_bf16(p, s, side->join) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status paged_attention_prefill(const pa_kv_pool* pool, const void* q, void* out, int32_t batch,
                                  int32_t num_q_heads, const int32_t* query_start_loc, int64_t total_q,
                                  int32_t max_q_len, const int32_t* block_table,
                                  int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  int32_t max_seq_len, float scale, void* stream) {
  return prefill_impl(pool, q, out, batch, num_q_heads, query_start_loc, total_q, max_q_len,
                      dense_table(block_table, max_blocks_per_seq, seq_lens), max_seq_len, scale, stream);
}

pa_status paged_attention_prefill_csr(const pa_kv_pool* pool, const void* q, void* out, int32_t batch,
                                      int32_t num_q_heads, const int32_t* query_start_loc, int64_t total_q,
                                      int32_t max_q_len, const int32_t* kv_indptr, const int32_t* kv_indices,
                                      int64_t num_kv_indices, const int32_t* kv_last_page_len,
                                      int32_t max_seq_len, float scale, void* stream) {
  Table t;
  const pa_status st = csr_table(pool, kv_indptr, kv_indices, num_kv_indices, kv_last_page_len, max_seq_len, &t);
  if (st != PA_OK) return st;
  return prefill_impl(pool, q, out, batch, num_q_heads, query_start_loc, total_q, max_q_len, t, max_seq_len, scale,
                      stream);
}

pa_status paged_device_error(int64_t* code, int64_t* detail) {
  if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
  unsigned long long w = 0;
  if (cudaMemcpyFromSymbol(&w, g_error_word, sizeof(w)) != cudaSuccess) return PA_ERR_CUDA;
  const unsigned long long zero = 0;
  if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return PA_ERR_CUDA;
  if (code) *code = (int64_t)(w >> 56);
  if (detail) {
    int64_t d = (int64_t)(w & ((1ull << 56) - 1));
    if (d & (1ll << 55)) d -= (1ll << 56);  // sign-extend the 56-bit field
    *detail = d;
  }
  return PA_OK;
}

}  // extern "C"
