// Host-side TMA descriptors (CUtensorMap) for the page pools.
//
// A pool [num_pages, page_size, num_kv_heads, head_dim] (bf16) is described as
// a 4-D tensor {64 dims, num_pages * page_size slots, num_kv_heads,
// head_dim / 64 slabs} with strides (slot: num_kv_heads*head_dim*2 B, head:
// head_dim*2 B, slab: 128 B).  One box {64, rows, heads, slabs} then lands in
// shared memory as [slab][head][row][128 B] with the 128-byte swizzle: per
// slab, `heads` tiles of `rows` x 128 B, each one KV head of consecutive
// slots, the layout an ldmatrix of one head reads without bank conflicts.
// Fewer, larger boxes matter: each TMA issue costs the issuing warp a fixed
// time, so 2 KB boxes cannot keep HBM busy while 4-32 KB boxes can.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <atomic>

#include "internal.h"

namespace pa {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<void*> fn{nullptr};
  void* p = fn.load(std::memory_order_acquire);
  if (p == nullptr) {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
      return nullptr;
    fn.store(p, std::memory_order_release);
  }
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
}

}  // namespace

bool encode_pool_tmap(CUtensorMap* map, const void* base, int64_t rows, int num_kv_heads, int head_dim,
                      int box_rows, int box_heads, int box_slabs) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return false;
  // dims: 64 dims of a slab, slots, heads, slabs of 64 dims
  cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)num_kv_heads, (cuuint64_t)(head_dim / 64)};
  cuuint64_t strides[3] = {(cuuint64_t)num_kv_heads * head_dim * 2, (cuuint64_t)head_dim * 2, 128};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_heads, (cuuint32_t)box_slabs};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_pool_tmap_blocked(CUtensorMap* map, const void* base, int64_t rows, int num_kv_heads, int head_dim,
                              int box_blocks) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr || rows % 8 != 0) return false;
  const cuuint64_t slot_stride = (cuuint64_t)num_kv_heads * head_dim * 2;
  // dims: 64 dims of a slab, slot within an 8-slot block, slabs, blocks, heads
  cuuint64_t dims[5] = {64, 8, (cuuint64_t)(head_dim / 64), (cuuint64_t)(rows / 8), (cuuint64_t)num_kv_heads};
  cuuint64_t strides[4] = {slot_stride, 128, 8 * slot_stride, (cuuint64_t)head_dim * 2};
  cuuint32_t box[5] = {64, 8, (cuuint32_t)(head_dim / 64), (cuuint32_t)box_blocks, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_pool_tmap_u8(CUtensorMap* map, const void* base, int64_t rows, int num_kv_heads, int head_dim,
                         int box_rows, int box_heads, bool swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)rows, (cuuint64_t)num_kv_heads};
  cuuint64_t strides[2] = {(cuuint64_t)num_kv_heads * head_dim, (cuuint64_t)head_dim};
  cuuint32_t box[3] = {(cuuint32_t)head_dim, (cuuint32_t)box_rows, (cuuint32_t)box_heads};
  cuuint32_t estr[3] = {1, 1, 1};
  // a row of head_dim codes is one swizzle span: 128-byte rows (head_dim 128)
  // take the 128-byte swizzle, 64-byte rows the 64-byte one
  if (head_dim != 64 && head_dim != 128) return false;
  const CUtensorMapSwizzle sw = !swizzle ? CU_TENSOR_MAP_SWIZZLE_NONE
                                         : (head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace pa
