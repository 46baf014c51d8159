// Device helpers shared by the paged-attention kernels (sm_103a).
// Inline PTX wrappers for cp.async, ldmatrix and the warp-level bf16 MMA,
// plus the device error word.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace pa {

// Device error word: high 8 bits = code, low 56 bits = detail.  The first
// violation wins; later ones are dropped.  Never traps.
enum : unsigned long long {
  ERR_BLOCK_TABLE = 1,
  ERR_SLOT = 2,
  ERR_SEQ_LEN = 3,
  ERR_QUERY_LOC = 4,
};

__device__ __forceinline__ void record_error(unsigned long long* err, unsigned long long code,
                                             long long detail) {
  if (err == nullptr) return;
  unsigned long long packed = (code << 56) | ((unsigned long long)detail & ((1ull << 56) - 1));
  atomicCAS(err, 0ull, packed);
}

// ---------------------------------------------------------------------------
// cp.async (16-byte, L2-only) with zero fill when src_bytes == 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ---------------------------------------------------------------------------
// ldmatrix / mma.sync m16n8k16 bf16 -> fp32
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The same warp-level MMA with f16 operands (used where K/V come from e4m3
// codes, which f16 holds exactly).
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// A bf16 pair (low element first) as an f16 pair.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Two e4m3 codes as an f16 pair (first code in the low half), exact: every
// e4m3 value, NaN included, is an f16.  _lo takes bytes 0-1 of w, _hi 2-3.
__device__ __forceinline__ uint32_t e4m3x2_lo_to_f16x2(uint32_t w) {
  uint32_t d;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n}\n" : "=r"(d) : "r"(w));
  return d;
}
__device__ __forceinline__ uint32_t e4m3x2_hi_to_f16x2(uint32_t w) {
  uint32_t d;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.f16x2.e4m3x2 %0, hi;\n}\n" : "=r"(d) : "r"(w));
  return d;
}

// Two floats (first in the low byte) as e4m3 codes: round to nearest even,
// finite magnitudes past 448 saturate, NaN stays NaN.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// e4m3 pools: eight bf16 elements (one 16-byte load) become eight codes (one
// 8-byte store); code = e4m3_rn_satfinite(x / scale) with an IEEE division.
__device__ __forceinline__ uint2 quantize8(uint4 v, float scale) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    c[j] = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w[j] << 16), scale),
                           __fdiv_rn(__uint_as_float(w[j] & 0xFFFF0000u), scale));
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// ---- page tables --------------------------------------------------------------
// A sequence's pages come from one of two forms:
//  * dense: a row-padded block_table [B, max_blocks] and seq_lens [B];
//  * CSR:   kv_indptr [B+1] into kv_indices (passed as block_table) and
//           kv_last_page_len [B]: sequence b's pages are
//           kv_indices[kv_indptr[b] .. kv_indptr[b+1]) and its last page holds
//           kv_last_page_len[b] tokens (the page-table metadata of
//           NVIDIA/recsys-examples PR #400, KVCacheMetadata), so it has
//           (n_pages - 1) * page_size + kv_last_page_len[b] keys.
// Offset of sequence b's first entry in block_table / kv_indices.
__device__ __forceinline__ int64_t page_list_start(const int32_t* kv_indptr, int max_blocks, int b) {
  return kv_indptr != nullptr ? (int64_t)__ldg(kv_indptr + b) : (int64_t)b * max_blocks;
}

// Keys of sequence b.  Dense: seq_lens[b], clamped to [0, max_len].  CSR: from
// the page count and the last page's fill, which is clamped to [1, page_size];
// a slice of kv_indptr outside [0, kv_len] or running backwards counts as no
// page (so nothing past kv_indices is ever read).  Out-of-range inputs are
// recorded when err is given.
__device__ __forceinline__ int seq_keys(const int32_t* seq_lens, const int32_t* kv_indptr,
                                        const int32_t* kv_last_page_len, int64_t kv_len, int b, int page_size,
                                        int max_len, unsigned long long* err) {
  if (kv_indptr == nullptr) {
    int L = __ldg(seq_lens + b);
    if (L < 0 || L > max_len) {
      if (err != nullptr) record_error(err, ERR_SEQ_LEN, L);
      L = L < 0 ? 0 : max_len;
    }
    return L;
  }
  const int s0 = __ldg(kv_indptr + b), s1 = __ldg(kv_indptr + b + 1);
  if (s0 < 0 || s1 < s0 || (int64_t)s1 > kv_len) {
    if (err != nullptr) record_error(err, ERR_SEQ_LEN, s1);
    return 0;
  }
  const int n = s1 - s0;
  if (n == 0) return 0;
  int last = __ldg(kv_last_page_len + b);
  if (last < 1 || last > page_size) {
    if (err != nullptr) record_error(err, ERR_SEQ_LEN, last);
    last = last < 1 ? 1 : page_size;
  }
  return (n - 1) * page_size + last;
}

// 2^x by the SFU's approximate base-2 exponential (PTX ex2.approx.ftz.f32):
// results below 2^-126 flush to zero, which changes no attention weight that
// survives the bf16 / fp32 sums.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Swizzled byte offset of 16-byte chunk `chunk` of row `row` in a tile whose
// rows are `row_bytes` long (row_bytes a multiple of 128): the chunk index is
// XOR-ed with (row % 8) so that 8 rows read at one logical chunk hit 8
// distinct bank groups (ldmatrix is then conflict-free).
__device__ __forceinline__ uint32_t swz(int row, int chunk, int row_bytes) {
  return row * row_bytes + ((chunk ^ (row & 7)) << 4);
}

// Programmatic dependent launch.  griddep_wait blocks until the grids this
// one depends on have completed and their memory is visible (a no-op when
// the kernel was not launched as a programmatic dependent);
// griddep_launch_dependents lets the next kernel on the stream start its
// prologue early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Launch with programmatic stream serialization allowed (see griddep_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// launch_pdl with every CTA of the grid resident at once (cooperative launch),
// for kernels whose CTAs wait on one another.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_coop(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

__host__ __device__ __forceinline__ int ilog2_pow2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

}  // namespace pa
