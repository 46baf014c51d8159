// paged_attention_prefill, bf16 path (warp-level MMA version).
//
// Varlen causal attention for packed new tokens (query_start_loc layout of
// ROCm/maxtext PR #93 "[Draft] kv paged kernels", the gpu_paged commit),
// masked by is_causal + nonpad_kv_seqlen as in onnxruntime/mobius PR #395
// "Add paged / block-table KV cache export" ("How it works", step 3).  Token
// i of sequence b sits at absolute position p = L_b - n_b + i and sees keys
// 0..p, read from the pages listed in block_table.
//
// Tiling: a CTA owns 64 packed rows of one (sequence, KV head): row r is
// query token r / G, query head hk*G + r % G, so each K/V tile staged in
// shared memory serves all G heads that read it.  Keys come in tiles of 64
// (four 16-key page blocks), double-buffered with cp.async through
// block_table; rows at or past L_b are zero-filled.  Each warp computes 16
// rows: S = Q K^T and O += P V with mma.sync m16n8k16 (bf16 in, fp32
// accumulate), online softmax in the log2 domain.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pa {

namespace {

constexpr int kBM = 64;   // packed rows per CTA
constexpr int kBN = 64;   // keys per tile
constexpr int kThreads = 128;

template <int D>
__global__ void __launch_bounds__(kThreads) prefill_mma_kernel(PrefillParams p) {
  constexpr int kRowBytes = D * 2;
  constexpr int kChunks = D / 8;
  constexpr int kTileBytes = kBN * kRowBytes;
  constexpr int kCopies = 2 * kBN * kChunks / kThreads;
  extern __shared__ __align__(1024) unsigned char smem[];

  const int b = blockIdx.z, hk = blockIdx.y;
  const int G = p.group, Hq = p.num_q_heads, Hkv = p.pool.num_kv_heads;
  const int qs = __ldg(p.query_start_loc + b);
  const int qe = __ldg(p.query_start_loc + b + 1);
  const int n = qe - qs;
  const int ps = p.pool.page_size, pshift = p.pool.page_shift;
  const int max_len = p.max_blocks * ps;
  int L = __ldg(p.seq_lens + b);
  if (L < 0 || L > max_len) {
    if (threadIdx.x == 0 && hk == 0 && blockIdx.x == 0) record_error(p.err, ERR_SEQ_LEN, L);
    L = L < 0 ? 0 : max_len;
  }
  if (n < 0 || qs < 0 || (int64_t)qe > p.total_q) {
    if (threadIdx.x == 0 && hk == 0 && blockIdx.x == 0) record_error(p.err, ERR_QUERY_LOC, qs);
    return;
  }
  if (n > p.max_q_len && threadIdx.x == 0 && hk == 0 && blockIdx.x == 0)
    record_error(p.err, ERR_QUERY_LOC, n);  // rows past the launch bound are not computed
  const int rows_total = n * G;
  const int tiles = (rows_total + kBM - 1) / kBM;
  const int tile = gridDim.x - 1 - blockIdx.x;  // heaviest (latest) tiles first
  if (tile >= tiles) return;
  const int row0 = tile * kBM;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int first = L - n;  // absolute position of new token 0
  const int last_row = min(row0 + kBM, rows_total) - 1;
  const int pos_max = first + last_row / G;
  const int pos_min = first + row0 / G;

  // rows of this thread: rA = lane/4, rB = rA + 8 within the warp's 16
  const int RA = row0 + warp * 16 + (lane >> 2), RB = RA + 8;
  const bool vA = RA < rows_total, vB = RB < rows_total;
  const int posA = vA ? first + RA / G : pos_max;
  const int posB = vB ? first + RB / G : pos_max;
  const int warp_pos_max = min(pos_max, first + min(row0 + warp * 16 + 15, last_row) / G);

  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(p.q);
  auto row_ptr = [&](int R) {  // packed row -> element offset of q/out row
    const int i = R / G, g = R - (R / G) * G;
    return ((int64_t)(qs + i) * Hq + (int64_t)hk * G + g) * D;
  };

  if (pos_max < 0) {  // no row of this tile sees any key (invalid input): zeros
    for (int idx = tid; idx < kBM * D; idx += kThreads) {
      const int R = row0 + idx / D;
      if (R < rows_total) outp[row_ptr(R) + idx % D] = __float2bfloat16_rn(0.f);
    }
    return;
  }

  uint32_t qf[D / 16][4];
  {
    const uint32_t* qa = reinterpret_cast<const uint32_t*>(qp + (vA ? row_ptr(RA) : 0));
    const uint32_t* qb = reinterpret_cast<const uint32_t*>(qp + (vB ? row_ptr(RB) : 0));
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int d0 = kk * 16 + (lane & 3) * 2;
      qf[kk][0] = vA ? __ldg(qa + d0 / 2) : 0u;
      qf[kk][1] = vB ? __ldg(qb + d0 / 2) : 0u;
      qf[kk][2] = vA ? __ldg(qa + (d0 + 8) / 2) : 0u;
      qf[kk][3] = vB ? __ldg(qb + (d0 + 8) / 2) : 0u;
    }
  }

  const __nv_bfloat16* kpool = static_cast<const __nv_bfloat16*>(p.pool.key_pool);
  const __nv_bfloat16* vpool = static_cast<const __nv_bfloat16*>(p.pool.value_pool);
  const int64_t row_elems = (int64_t)Hkv * D;
  const int32_t* bt = p.block_table + (int64_t)b * p.max_blocks;

  auto load_tile = [&](int kt, int slot) {
    unsigned char* st = smem + slot * 2 * kTileBytes;
#pragma unroll
    for (int i = 0; i < kCopies; ++i) {
      const int idx = tid + i * kThreads;
      const int row = idx / kChunks, ch = idx % kChunks;  // row in [0, 2*kBN): [tensor][key]
      const int tensor = row / kBN, r = row % kBN;
      const int j = kt * kBN + r;
      bool ok = j < L;
      const __nv_bfloat16* src = kpool;
      if (ok) {
        const int page = __ldg(bt + (j >> pshift));
        if (page < 0 || page >= p.pool.num_pages) {
          record_error(p.err, ERR_BLOCK_TABLE, page);
          ok = false;
        } else {
          src = (tensor ? vpool : kpool) + (((int64_t)page << pshift) + (j & (ps - 1))) * row_elems +
                (int64_t)hk * D + ch * 8;
        }
      }
      cp_async_16(smem_u32(st + tensor * kTileBytes + swz(r, ch, kRowBytes)), src, ok ? 16 : 0);
    }
  };

  float o[D / 8][4];
#pragma unroll
  for (int n8 = 0; n8 < D / 8; ++n8) o[n8][0] = o[n8][1] = o[n8][2] = o[n8][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sl2 = p.scale_log2;
  const int ntiles = pos_max / kBN + 1;
  const int mi = lane >> 3, rr = lane & 7;

  load_tile(0, 0);
  cp_async_commit();
#pragma unroll 1
  for (int kt = 0; kt < ntiles; ++kt) {
    if (kt + 1 < ntiles) load_tile(kt + 1, (kt + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int key0 = kt * kBN;
    if (key0 <= warp_pos_max) {
      const uint32_t kbase = smem_u32(smem + (kt & 1) * 2 * kTileBytes);
      const uint32_t vbase = kbase + kTileBytes;
      float s[kBN / 8][4];
#pragma unroll
      for (int t = 0; t < kBN / 8; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int t2 = 0; t2 < kBN / 16; ++t2) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kbase + swz(t2 * 16 + (mi >> 1) * 8 + rr, kk * 2 + (mi & 1), kRowBytes), b0, b1,
                      b2, b3);
          mma_bf16_16816(s[2 * t2], qf[kk], b0, b1);
          mma_bf16_16816(s[2 * t2 + 1], qf[kk], b2, b3);
        }
      }
      const bool need_mask = key0 + kBN - 1 > pos_min;
#pragma unroll
      for (int t = 0; t < kBN / 8; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = key0 + t * 8 + (lane & 3) * 2 + (e & 1);
          const int pos = e < 2 ? posA : posB;
          s[t][e] = (!need_mask || key <= pos) ? s[t][e] * sl2 : -INFINITY;
        }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int t = 0; t < kBN / 8; ++t) {
        mx0 = fmaxf(mx0, fmaxf(s[t][0], s[t][1]));
        mx1 = fmaxf(mx1, fmaxf(s[t][2], s[t][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      // a row that has seen no key yet keeps a -inf max: use 0 as the base
      const float b0s = mn0 == -INFINITY ? 0.f : mn0, b1s = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = fast_exp2(m0 - b0s), al1 = fast_exp2(m1 - b1s);
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int t = 0; t < kBN / 8; ++t) {
        s[t][0] = fast_exp2(s[t][0] - b0s);
        s[t][1] = fast_exp2(s[t][1] - b0s);
        s[t][2] = fast_exp2(s[t][2] - b1s);
        s[t][3] = fast_exp2(s[t][3] - b1s);
        rs0 += s[t][0] + s[t][1];
        rs1 += s[t][2] + s[t][3];
      }
      l0 = l0 * al0 + rs0;
      l1 = l1 * al1 + rs1;
      if (__any_sync(0xffffffffu, (al0 != 1.f) | (al1 != 1.f))) {
#pragma unroll
        for (int n8 = 0; n8 < D / 8; ++n8) {
          o[n8][0] *= al0; o[n8][1] *= al0;
          o[n8][2] *= al1; o[n8][3] *= al1;
        }
      }
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int ks = 0; ks < kBN / 16; ++ks) {
        uint32_t pa[4];
        pa[0] = pack_bf16(s[2 * ks][0], s[2 * ks][1]);
        pa[1] = pack_bf16(s[2 * ks][2], s[2 * ks][3]);
        pa[2] = pack_bf16(s[2 * ks + 1][0], s[2 * ks + 1][1]);
        pa[3] = pack_bf16(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(vbase + swz(ks * 16 + (mi & 1) * 8 + rr, 2 * j + (mi >> 1), kRowBytes), b0,
                            b1, b2, b3);
          mma_bf16_16816(o[2 * j], pa, b0, b1);
          mma_bf16_16816(o[2 * j + 1], pa, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  float la = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
  la += __shfl_xor_sync(0xffffffffu, la, 2);
  float lb = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
  lb += __shfl_xor_sync(0xffffffffu, lb, 2);
  const float ia = la > 0.f ? 1.f / la : 0.f, ib = lb > 0.f ? 1.f / lb : 0.f;
  uint32_t* oa = reinterpret_cast<uint32_t*>(outp + (vA ? row_ptr(RA) : 0));
  uint32_t* ob = reinterpret_cast<uint32_t*>(outp + (vB ? row_ptr(RB) : 0));
#pragma unroll
  for (int n8 = 0; n8 < D / 8; ++n8) {
    const int col = n8 * 8 + (lane & 3) * 2;
    if (vA) oa[col / 2] = pack_bf16(o[n8][0] * ia, o[n8][1] * ia);
    if (vB) ob[col / 2] = pack_bf16(o[n8][2] * ib, o[n8][3] * ib);
  }
}

template <int D>
cudaError_t launch_prefill_mma(const PrefillParams& p, cudaStream_t s) {
  const size_t smem = 2 * 2 * (size_t)kBN * D * 2;
  auto kern = prefill_mma_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = ((int64_t)p.max_q_len * p.group + kBM - 1) / kBM;
  dim3 grid((unsigned)tiles, (unsigned)p.pool.num_kv_heads, (unsigned)p.batch);
  kern<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bf16(const PrefillParams& p, cudaStream_t s) {
  if (p.max_q_len <= 0 || p.batch <= 0) return cudaSuccess;
  return p.pool.head_dim == 128 ? launch_prefill_mma<128>(p, s) : launch_prefill_mma<64>(p, s);
}

}  // namespace pa
