// CUDA-core path of paged_attention_decode / paged_attention_prefill: fp32
// pools, and bf16 pools whose page size is not a power of two >= 8 (the TMA
// boxes of the tensor-core kernels take whole 8-slot blocks of a page).
//
// Same operation as the tensor-core kernels (onnxruntime/mobius PR #395 "Add
// paged / block-table KV cache export", "How it works": Gather through
// block_table, then attention with is_causal + nonpad_kv_seqlen masking),
// computed in fp32 on CUDA cores, so that an fp32 pool keeps fp32 accuracy end
// to end.  One warp owns one (query row, query head); lanes split head_dim (up
// to 256), keys are visited one at a time with an online softmax.  This path
// serves small fp32 models, page sizes 1 to 4 (and other page sizes) of bf16
// pools and correctness runs, not the hot path.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pa {

namespace {

constexpr int kMaxPerLane = 8;  // head_dim <= 256

__device__ __forceinline__ float ld_elem(const float* x, int64_t i) { return x[i]; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* x, int64_t i) { return __bfloat162float(x[i]); }
__device__ __forceinline__ void st_elem(float* x, int64_t i, float v) { x[i] = v; }
__device__ __forceinline__ void st_elem(__nv_bfloat16* x, int64_t i, float v) { x[i] = __float2bfloat16_rn(v); }

// T: the element type of q, the pools and out
template <typename T>
__global__ void __launch_bounds__(256) attn_f32_kernel(AttnF32Params p) {
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  const int64_t nwarps = (int64_t)gridDim.x * warps_per_block;
  const int D = p.pool.head_dim, Hq = p.num_q_heads, Hkv = p.pool.num_kv_heads;
  const int ps = p.pool.page_size;
  const int max_len = p.max_blocks * ps;
  const int64_t total = p.rows * Hq;
  const T* kpool = static_cast<const T*>(p.pool.key_pool);
  const T* vpool = static_cast<const T*>(p.pool.value_pool);
  for (int64_t w = (int64_t)blockIdx.x * warps_per_block + (threadIdx.x >> 5); w < total; w += nwarps) {
    const int64_t r = w / Hq;
    const int h = (int)(w - r * Hq);
    const int hk = h / p.group;
    int b, n, i;
    if (p.query_start_loc == nullptr) {
      b = (int)r; n = 1; i = 0;
    } else {
      int lo = 0, hi = p.batch;  // largest b with query_start_loc[b] <= r
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.query_start_loc + mid) <= r) lo = mid; else hi = mid;
      }
      b = lo;
      const int s0 = __ldg(p.query_start_loc + b);
      n = __ldg(p.query_start_loc + b + 1) - s0;
      i = (int)(r - s0);
    }
    const int L = seq_keys(p.seq_lens, p.kv_indptr, p.kv_last_page_len, p.kv_len, b, ps, max_len, lane == 0 ? p.err : nullptr);
    const int pos = L - n + i;
    const T* qrow = static_cast<const T*>(p.q) + (r * Hq + h) * (int64_t)D;
    float qv[kMaxPerLane], ov[kMaxPerLane];
#pragma unroll
    for (int t = 0; t < kMaxPerLane; ++t) {
      const int d = lane + 32 * t;
      qv[t] = d < D ? ld_elem(qrow, d) : 0.f;
      ov[t] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const int32_t* bt = p.block_table + page_list_start(p.kv_indptr, p.max_blocks, b);
    for (int j = 0; j <= pos; ++j) {
      const int page = __ldg(bt + j / ps);
      if (page < 0 || page >= p.pool.num_pages) {
        if (lane == 0) record_error(p.err, ERR_BLOCK_TABLE, page);
        continue;
      }
      const int64_t off = ((int64_t)page * ps + j % ps) * Hkv * D + (int64_t)hk * D;
      float s = 0.f;
#pragma unroll
      for (int t = 0; t < kMaxPerLane; ++t) {
        const int d = lane + 32 * t;
        if (d < D) s = fmaf(qv[t], ld_elem(kpool, off + d), s);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      s *= p.scale;
      const float mn = fmaxf(m, s);
      const float a = expf(m - mn);
      const float e = expf(s - mn);
      l = l * a + e;
#pragma unroll
      for (int t = 0; t < kMaxPerLane; ++t) {
        const int d = lane + 32 * t;
        if (d < D) ov[t] = fmaf(ov[t], a, e * ld_elem(vpool, off + d));
      }
      m = mn;
    }
    T* orow = static_cast<T*>(p.out) + (r * Hq + h) * (int64_t)D;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int t = 0; t < kMaxPerLane; ++t) {
      const int d = lane + 32 * t;
      if (d < D) st_elem(orow, d, ov[t] * inv);
    }
  }
}

}  // namespace

cudaError_t launch_attn_f32(const AttnF32Params& p, int num_sms, cudaStream_t s) {
  const int64_t total = p.rows * p.num_q_heads;
  if (total <= 0) return cudaSuccess;
  const int threads = 256, wpb = threads / 32;
  int64_t blocks = (total + wpb - 1) / wpb;
  if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
  if (p.bf16)
    attn_f32_kernel<__nv_bfloat16><<<(int)blocks, threads, 0, s>>>(p);
  else
    attn_f32_kernel<float><<<(int)blocks, threads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
