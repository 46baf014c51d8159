// paged_kv_append: the ScatterND write of new K/V rows into the page pool
// (onnxruntime/mobius PR #395 "Add paged / block-table KV cache export",
// "How it works (per attention layer)", step 1).
//
// One warp per token row: the K row and the V row (num_kv_heads * head_dim
// elements each, contiguous in both source and pool) are copied with
// 16-byte vector loads/stores when alignment allows.  The loads bypass L1
// (read once); the stores keep the default policy so that the attention
// kernel that runs next finds the fresh rows in L2.  An e4m3 pool takes bf16
// rows and stores their codes (quantize8).
#include "common.cuh"
#include "internal.h"

namespace pa {

template <typename V>
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
  // The attention kernel that follows may start its prologue now; it waits
  // (griddepcontrol.wait) for this grid before reading the pool.
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int64_t nvec = p.row_bytes / (int64_t)sizeof(V);
  for (int64_t t = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5); t < p.num_tokens;
       t += (int64_t)gridDim.x * warps) {
    const int64_t slot = __ldg(p.slot_mapping + t);
    if (slot < 0) continue;  // padding token
    if (slot >= p.num_slots) {
      if (lane == 0) record_error(p.err, ERR_SLOT, slot);
      continue;
    }
    const V* ks = reinterpret_cast<const V*>(static_cast<const char*>(p.key) + t * p.row_bytes);
    const V* vs =
        reinterpret_cast<const V*>(static_cast<const char*>(p.value) + t * p.row_bytes);
    V* kd = reinterpret_cast<V*>(static_cast<char*>(p.key_pool) + slot * p.row_bytes);
    V* vd = reinterpret_cast<V*>(static_cast<char*>(p.value_pool) + slot * p.row_bytes);
    int64_t i = lane;
    // Four vectors of K and four of V in flight per lane per iteration.
    for (; i + 96 < nvec; i += 128) {
      V a0 = __ldcs(ks + i), a1 = __ldcs(ks + i + 32), a2 = __ldcs(ks + i + 64),
        a3 = __ldcs(ks + i + 96);
      V b0 = __ldcs(vs + i), b1 = __ldcs(vs + i + 32), b2 = __ldcs(vs + i + 64),
        b3 = __ldcs(vs + i + 96);
      kd[i] = a0; kd[i + 32] = a1; kd[i + 64] = a2; kd[i + 96] = a3;
      vd[i] = b0; vd[i + 32] = b1; vd[i + 64] = b2; vd[i + 96] = b3;
    }
    for (; i < nvec; i += 32) {
      V a = __ldcs(ks + i);
      V b = __ldcs(vs + i);
      kd[i] = a;
      vd[i] = b;
    }
  }
}

__global__ void __launch_bounds__(256) append_e4m3_kernel(AppendParams p) {
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int64_t n8 = p.row_bytes / 8;  // groups of 8 elements (row_bytes = elements)
  for (int64_t t = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5); t < p.num_tokens;
       t += (int64_t)gridDim.x * warps) {
    const int64_t slot = __ldg(p.slot_mapping + t);
    if (slot < 0) continue;  // padding token
    if (slot >= p.num_slots) {
      if (lane == 0) record_error(p.err, ERR_SLOT, slot);
      continue;
    }
    const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const char*>(p.key) + t * p.row_bytes * 2);
    const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const char*>(p.value) + t * p.row_bytes * 2);
    uint2* kd = reinterpret_cast<uint2*>(static_cast<char*>(p.key_pool) + slot * p.row_bytes);
    uint2* vd = reinterpret_cast<uint2*>(static_cast<char*>(p.value_pool) + slot * p.row_bytes);
    for (int64_t i = lane; i < n8; i += 32) {
      const uint4 a = __ldcs(ks + i), b = __ldcs(vs + i);
      kd[i] = quantize8(a, p.k_scale);
      vd[i] = quantize8(b, p.v_scale);
    }
  }
}

cudaError_t launch_append(const AppendParams& p, int vec_bytes, int num_sms, cudaStream_t s) {
  if (p.num_tokens <= 0) return cudaSuccess;
  const int threads = 256, warps = threads / 32;
  int64_t blocks = (p.num_tokens + warps - 1) / warps;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (p.kv8) {
    append_e4m3_kernel<<<(int)blocks, threads, 0, s>>>(p);
    return cudaGetLastError();
  }
  switch (vec_bytes) {
    case 16: append_kernel<uint4><<<(int)blocks, threads, 0, s>>>(p); break;
    case 8: append_kernel<uint2><<<(int)blocks, threads, 0, s>>>(p); break;
    case 4: append_kernel<uint32_t><<<(int)blocks, threads, 0, s>>>(p); break;
    default: append_kernel<unsigned short><<<(int)blocks, threads, 0, s>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace pa
