// paged_attention_decode_static_scratch: the bf16 decode call for callers that
// cannot allocate device memory.
//
// Some callers of a decode step are not allowed to call cudaMalloc or any
// allocating library routine: a plugin inside an inference runtime that owns
// every byte of device memory and gives its plugins no allocator, or a
// latency-critical serving loop that may not take cudaMalloc's implicit
// device-wide synchronisation in the middle of a step.  For them this entry
// point keeps the split-KV partials in a file-scope __device__ array that
// the library owns, so the caller passes only inputs and outputs.
//
// The array is PA_DECODE_STATIC_SCRATCH_BYTES (8 MiB) and exists on every
// GPU that loads the library, until the process exits.  Host code may not
// use the array's name as a device address; the address is looked up once
// per device with cudaGetSymbolAddress, with that device current, by the
// first call on that device.  Every call shares the array: two calls whose
// kernels overlap on the GPU (on different streams, or on one device from
// several host threads without ordering) race on it.  Nothing in it needs to
// start zeroed: every partial a call reads is written earlier in the same
// launch, and the arrival counters carry a tag derived from a per-launch
// epoch word kept at the array's start (each launch reads it and stores the
// next), so counts left by an earlier call read as zero.
//
// The stream must belong to the current device: the array's address is the
// current device's, so a call whose stream is on another GPU is refused
// (PA_ERR_CUDA) before anything is launched.
#include <atomic>

#include "../../include/paged_attn.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[PA_DECODE_STATIC_SCRATCH_BYTES];

std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_decode_scratch on the current device (looked up once).
pa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return PA_OK;
}

}  // namespace

extern "C" pa_status paged_attention_decode_static_scratch(
    const pa_kv_pool* pool, const void* q, void* out, int32_t batch, int32_t num_q_heads,
    const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
    int32_t max_seq_len, float scale, void* stream) {
  if (pool == nullptr) return PA_ERR_NULL;
  if (pool->dtype != PA_DTYPE_BF16 && pool->dtype != PA_DTYPE_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  const size_t need = paged_attention_decode_workspace_size(batch, num_q_heads, pool->num_kv_heads,
                                                            pool->head_dim, pool->dtype);
  if (need > (size_t)PA_DECODE_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  // the scratch address below is the current device's: the kernel must run there
  int cur = -1, sdev = -1;
  if (cudaGetDevice(&cur) != cudaSuccess ||
      cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess || sdev != cur)
    return PA_ERR_CUDA;
  void* scratch = nullptr;
  const pa_status st = scratch_address(&scratch);
  if (st != PA_OK) return st;
  return paged_attention_decode(pool, q, out, batch, num_q_heads, block_table, max_blocks_per_seq,
                                seq_lens, max_seq_len, scale, scratch,
                                (size_t)PA_DECODE_STATIC_SCRATCH_BYTES, stream);
}
