// Host-side TMA descriptors (CUtensorMap) for the page pools.
//
// A pool [num_pages, page_size, num_kv_heads, head_dim] (bf16) is described as
// a 3-D tensor {head_dim, num_pages * page_size, num_kv_heads} whose slot
// stride (num_kv_heads*head_dim*2 B) is larger than its head stride
// (head_dim*2 B).  One box {64, rows, heads} then lands in shared memory as
// `heads` tiles of `rows` x 128 B, each tile one KV head of consecutive slots
// with the 128-byte swizzle, i.e. the layout an ldmatrix of one head reads
// without bank conflicts.
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
                      int box_rows, int box_heads) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)rows, (cuuint64_t)num_kv_heads};
  cuuint64_t strides[2] = {(cuuint64_t)num_kv_heads * head_dim * 2, (cuuint64_t)head_dim * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_heads};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace pa
