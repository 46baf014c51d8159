// paged_attention_prefill, bf16 path: tcgen05 / TMEM varlen causal attention.
//
// What is computed: varlen causal attention for packed new tokens
// (query_start_loc layout of ROCm/maxtext PR #93 "[Draft] kv paged kernels",
// the gpu_paged commit), masked by is_causal + nonpad_kv_seqlen as in
// onnxruntime/mobius PR #395 "Add paged / block-table KV cache export" ("How
// it works", step 3).  Token i of sequence b sits at absolute position
// p = L_b - n_b + i and sees keys 0..p, read from the pages in block_table.
//
// Tiling (GB300-first): a CTA owns 128 packed rows of one (sequence, KV head)
// -- row r is query token r / G, query head hk*G + r % G -- so every K/V tile
// in shared memory serves all G heads that read it.  Keys come in tiles of
// 128 (eight 16-key pages).
// * 4 loader warps stage Q once and K/V tiles (2-stage ring) with 16-byte
//   cp.async through block_table into the 128-byte-swizzled UMMA layout;
//   rows at or past L_b are zero-filled.  Pages are scattered, so a K tile's
//   rows cannot come from one TMA box, and per-page boxes are too small to
//   keep up with the tensor core.
// * 1 MMA warp issues tcgen05.mma: S = Q K^T (M 128, N 128, fp32 in TMEM,
//   double-buffered so S(j+1) overlaps the softmax of S(j)) and O += P V
//   (M 128, N head_dim, fp32 in TMEM), each committed to an mbarrier.
// * 4 softmax warps own one TMEM lane (= one row) per thread: tcgen05.ld of S,
//   causal mask, online softmax in the log2 domain with a lazily updated
//   reference max (O and l are rescaled in TMEM only when the row max grows by
//   more than 2^8), P written to shared memory as bf16 in the UMMA A layout,
//   and at the end O / l written to global as bf16.
// Fully masked key tiles are never loaded or multiplied.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace pa {

namespace {

constexpr int kBM = 128;             // packed query rows per CTA (TMEM lanes)
constexpr int kBN = 128;             // keys per tile
constexpr int kNS = 2;               // K/V ring stages
constexpr int kSoftmaxWarps = 4;     // warps 0..3 (TMEM lane quarters 0..3)
constexpr int kMmaWarp = 4;
constexpr int kLoadWarp0 = 5;        // warps 5..8
constexpr int kLoadThreads = 128;
constexpr int kThreads = 32 * 9;
constexpr int kSlab = kBM * 128;     // one 64-column slab of a 128-row tile (16 KB)
constexpr float kRescaleThreshold = 8.f;  // log2 units

template <int D>
struct PCfg {
  static constexpr int kSlabs = D / 64;
  static constexpr int kQBytes = kSlabs * kSlab;
  static constexpr int kKVTile = kSlabs * kSlab;       // K or V tile (128 keys)
  static constexpr int kStageBytes = 2 * kKVTile;
  static constexpr int kPBytes = 2 * kSlab;            // P: 128 rows x 128 keys
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQBytes;
  static constexpr int kPOff = kKVOff + kNS * kStageBytes;
  static constexpr int kBarOff = kPOff + kPBytes;
  static constexpr int kSmem = kBarOff + 16 * 8 + 16 + 1024;  // barriers, TMEM base, alignment slack
  static constexpr uint32_t kTmemCols = 512;           // S0 | S1 | O
  static constexpr uint32_t kOCol = 256;
};

// barriers
enum { B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = 1 + kNS, B_SFULL = 1 + 2 * kNS, B_PFULL = 3 + 2 * kNS, B_PVDONE = 4 + 2 * kNS,
       B_COUNT = 5 + 2 * kNS };

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(PrefillParams p) {
  using C = PCfg<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int b = blockIdx.z, hk = blockIdx.y;
  const int G = p.group, Hq = p.num_q_heads, Hkv = p.pool.num_kv_heads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qs = __ldg(p.query_start_loc + b);
  const int qe = __ldg(p.query_start_loc + b + 1);
  const int n = qe - qs;
  const int ps = p.pool.page_size, pshift = p.pool.page_shift;
  const int max_len = p.max_blocks * ps;
  int L = __ldg(p.seq_lens + b);
  if (L < 0 || L > max_len) {
    if (tid == 0 && hk == 0 && blockIdx.x == 0) record_error(p.err, ERR_SEQ_LEN, L);
    L = L < 0 ? 0 : max_len;
  }
  if (n < 0 || qs < 0 || (int64_t)qe > p.total_q) {
    if (tid == 0 && hk == 0 && blockIdx.x == 0) record_error(p.err, ERR_QUERY_LOC, qs);
    return;
  }
  if (n > p.max_q_len && tid == 0 && hk == 0 && blockIdx.x == 0) record_error(p.err, ERR_QUERY_LOC, n);
  const int rows_total = n * G;
  const int tiles = (rows_total + kBM - 1) / kBM;
  const int tile = gridDim.x - 1 - blockIdx.x;  // heaviest (latest) tiles first
  if (tile >= tiles) return;
  const int row0 = tile * kBM;
  const int first = L - n;  // absolute position of new token 0
  const int last_row = min(row0 + kBM, rows_total) - 1;
  const int pos_max = first + last_row / G;
  const int pos_min = first + row0 / G;
  const int nt = pos_max >= 0 ? pos_max / kBN + 1 : 0;  // key tiles with a visible key

  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(p.q);
  auto row_off = [&](int R) {  // packed row -> element offset of its q / out row
    const int i = R / G, g = R - (R / G) * G;
    return ((int64_t)(qs + i) * Hq + (int64_t)hk * G + g) * D;
  };
  griddep_launch_dependents();
  if (nt == 0) {  // no row of this tile sees any key (invalid input): zeros
    griddep_wait();
    for (int idx = tid; idx < kBM * D; idx += kThreads) {
      const int R = row0 + idx / D;
      if (R < rows_total) outp[row_off(R) + idx % D] = __float2bfloat16_rn(0.f);
    }
    return;
  }

  unsigned char* q_s = smem + C::kQOff;
  unsigned char* kv_s = smem + C::kKVOff;
  unsigned char* p_s = smem + C::kPOff;
  const uint32_t bars = smem_u32(smem + C::kBarOff);
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOff + 16 * 8);

  if (tid == 0) {
    mbar_init(bar(B_QFULL), kLoadThreads);
    for (int s = 0; s < kNS; ++s) {
      mbar_init(bar(B_KVFULL + s), kLoadThreads);
      mbar_init(bar(B_KVEMPTY + s), 1);
    }
    mbar_init(bar(B_SFULL + 0), 1);
    mbar_init(bar(B_SFULL + 1), 1);
    mbar_init(bar(B_PFULL), 32 * kSoftmaxWarps);
    mbar_init(bar(B_PVDONE), 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const float sl2 = p.scale_log2;
  bool alive = true;

  if (warp >= kLoadWarp0) {
    // ======================= loaders (cp.async) =======================
    const int lt = tid - 32 * kLoadWarp0;
    griddep_wait();  // the pool rows of this step were written by the append kernel
    constexpr int kChunks = D / 8;  // 16-byte chunks per row
    // Q: 128 packed rows
#pragma unroll 4
    for (int idx = lt; idx < kBM * kChunks; idx += kLoadThreads) {
      const int r = idx / kChunks, c = idx % kChunks;
      const int R = row0 + r;
      const bool ok = R < rows_total;
      const __nv_bfloat16* src = ok ? qp + row_off(R) + c * 8 : qp;
      cp_async_16(smem_u32(q_s + (c >> 3) * kSlab + r * 128 + (((c & 7) ^ (r & 7)) << 4)), src, ok ? 16 : 0);
    }
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async_smem();  // generic-proxy (cp.async) writes -> visible to the tensor core
    mbar_arrive(bar(B_QFULL));
    const __nv_bfloat16* kpool = static_cast<const __nv_bfloat16*>(p.pool.key_pool);
    const __nv_bfloat16* vpool = static_cast<const __nv_bfloat16*>(p.pool.value_pool);
    const int64_t row_elems = (int64_t)Hkv * D;
    const int32_t* bt = p.block_table + (int64_t)b * p.max_blocks;
    for (int j = 0; j < nt; ++j) {
      const int s = j % kNS;
      if (j > 0) {
        // publish tile j-1 before blocking on the ring: the MMA warp may need it
        // (S(j-1)) before it can free the stage tile j goes to
        cp_async_wait<0>();
        fence_proxy_async_smem();
        mbar_arrive(bar(B_KVFULL + (j - 1) % kNS));
      }
      if (j >= kNS && alive) alive = mbar_wait(bar(B_KVEMPTY + s), (uint32_t)(((j / kNS) - 1) & 1), p.err);
      unsigned char* st = kv_s + s * C::kStageBytes;
      // thread lt copies 16-byte chunk (lt % kChunks) of rows r = lt / kChunks + kRowStep * i of
      // both K and V: one block_table lookup per row, shared by the two tensors
      constexpr int kRowStep = kLoadThreads / kChunks;
      const int c = lt % kChunks;
#pragma unroll 4
      for (int r = lt / kChunks; r < kBN; r += kRowStep) {
        const int key = j * kBN + r;
        const uint32_t dst = smem_u32(st + (c >> 3) * kSlab + r * 128 + (((c & 7) ^ (r & 7)) << 4));
        int64_t off = -1;
        if (key < L) {
          const int page = __ldg(bt + (key >> pshift));
          if (page < 0 || page >= p.pool.num_pages) record_error(p.err, ERR_BLOCK_TABLE, page);
          else off = (((int64_t)page << pshift) + (key & (ps - 1))) * row_elems + (int64_t)hk * D + c * 8;
        }
        cp_async_16(dst, off >= 0 ? kpool + off : kpool, off >= 0 ? 16 : 0);
        cp_async_16(dst + C::kKVTile, off >= 0 ? vpool + off : vpool, off >= 0 ? 16 : 0);
      }
      cp_async_commit();
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    mbar_arrive(bar(B_KVFULL + (nt - 1) % kNS));
  }

  if (warp == kMmaWarp && lane == 0) {
    // ======================= MMA issuer =======================
    const uint32_t q_addr = smem_u32(q_s);
    const uint32_t kv_addr = smem_u32(kv_s);
    const uint32_t p_addr = smem_u32(p_s);
    constexpr uint32_t idesc_s = umma_idesc_bf16(kBM, kBN, false);
    constexpr uint32_t idesc_o = umma_idesc_bf16(kBM, D, true);
    auto issue_s = [&](int j) {  // S[j & 1] = Q K_j^T
      const uint32_t k_addr = kv_addr + (j % kNS) * C::kStageBytes;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kSlab + (kk & 3) * 32;
        umma_bf16(tmem + (j & 1) * kBN, umma_desc_sw128(q_addr + off, 16, 1024),
                  umma_desc_sw128(k_addr + off, 16, 1024), idesc_s, kk > 0);
      }
      umma_commit(bar(B_SFULL + (j & 1)));
    };
    if (alive) alive = mbar_wait(bar(B_QFULL), 0, p.err);
    for (int j = 0; j < nt; ++j) {
      if (j == 0) {
        if (alive) alive = mbar_wait(bar(B_KVFULL), 0, p.err);
        tc_fence_after();
        issue_s(0);
      }
      if (j + 1 < nt) {
        if (alive) alive = mbar_wait(bar(B_KVFULL + (j + 1) % kNS), (uint32_t)(((j + 1) / kNS) & 1), p.err);
        tc_fence_after();
        issue_s(j + 1);
      }
      if (alive) alive = mbar_wait(bar(B_PFULL), (uint32_t)(j & 1), p.err);
      tc_fence_after();
      const uint32_t v_addr = kv_addr + (j % kNS) * C::kStageBytes + C::kKVTile;
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk) {  // O += P V over 16-key steps
        umma_bf16(tmem + C::kOCol, umma_desc_sw128(p_addr + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024),
                  umma_desc_sw128(v_addr + kk * 16 * 128, kSlab, 1024), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(bar(B_PVDONE));
      umma_commit(bar(B_KVEMPTY + j % kNS));
    }
  }

  if (warp < kSoftmaxWarps) {
    // ======================= softmax: one TMEM lane (row) per thread =======================
    const int r = tid;  // row within the tile == TMEM lane
    const int R = row0 + r;
    const bool valid_row = R < rows_total;
    const int pos = valid_row ? first + R / G : pos_max;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float m_ref = -INFINITY, l = 0.f;
    for (int j = 0; j < nt; ++j) {
      if (alive) alive = mbar_wait(bar(B_SFULL + (j & 1)), (uint32_t)((j >> 1) & 1), p.err);
      tc_fence_after();
      const uint32_t s_addr = lane_base + (j & 1) * kBN;
      const int key0 = j * kBN;
      const bool need_mask = key0 + kBN - 1 > pos_min;
      // pass 1: row max of this tile
      float tmax = -INFINITY;
#pragma unroll
      for (int cb = 0; cb < kBN / 32; ++cb) {
        uint32_t v[32];
        tmem_ld32(s_addr + cb * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float sv = __uint_as_float(v[e]) * sl2;
          const bool vis = !need_mask || key0 + cb * 32 + e <= pos;
          tmax = fmaxf(tmax, vis ? sv : -INFINITY);
        }
      }
      // reference max: moved only when the row max grows by more than 2^8
      float alpha = 1.f;
      bool rescale = false;
      if (tmax > m_ref + kRescaleThreshold) {
        alpha = fast_exp2(m_ref - tmax);  // 0 when m_ref is -inf
        m_ref = tmax;
        l *= alpha;
        rescale = j > 0;
      }
      const float mbase = m_ref == -INFINITY ? 0.f : m_ref;
      if (j > 0) {  // PV(j-1) must be done before O is touched and P is overwritten
        if (alive) alive = mbar_wait(bar(B_PVDONE), (uint32_t)((j - 1) & 1), p.err);
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t v[32];
          tmem_ld32(lane_base + C::kOCol + cb * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st32(lane_base + C::kOCol + cb * 32, v);
        }
        tmem_wait_st();
      }
      // pass 2: P = exp2(s - m) as bf16 into the UMMA A layout (K-major, 128-byte swizzle)
      float rsum = 0.f;
#pragma unroll
      for (int cb = 0; cb < kBN / 32; ++cb) {
        uint32_t v[32];
        tmem_ld32(s_addr + cb * 32, v);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int k0 = key0 + cb * 32 + e;
          const bool v0 = !need_mask || k0 <= pos, v1 = !need_mask || k0 + 1 <= pos;
          const float p0 = v0 ? fast_exp2(fmaf(__uint_as_float(v[e]), sl2, -mbase)) : 0.f;
          const float p1 = v1 ? fast_exp2(fmaf(__uint_as_float(v[e + 1]), sl2, -mbase)) : 0.f;
          rsum += p0 + p1;
          pk[e >> 1] = pack_bf16(p0, p1);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // four 16-byte chunks: keys cb*32 + 8q .. +7
          const int key = cb * 32 + q * 8;
          const int slab = key >> 6, chunk = (key & 63) >> 3;
          *reinterpret_cast<uint4*>(p_s + slab * kSlab + r * 128 + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      l += rsum;
      fence_proxy_async_smem();  // P stores -> visible to the tensor core
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
    }
    // ---- epilogue: O / l -> bf16 ----
    if (alive) alive = mbar_wait(bar(B_PVDONE), (uint32_t)((nt - 1) & 1), p.err);
    tc_fence_after();
    griddep_wait();  // before the first global write
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* orow = outp + (valid_row ? row_off(R) : 0);
#pragma unroll
    for (int cb = 0; cb < D / 32; ++cb) {
      uint32_t v[32];
      tmem_ld32(lane_base + C::kOCol + cb * 32, v);
      tmem_wait_ld();
      if (valid_row) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(v[8 * q + 0]) * inv, __uint_as_float(v[8 * q + 1]) * inv);
          w.y = pack_bf16(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv);
          w.z = pack_bf16(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv);
          w.w = pack_bf16(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv);
          *reinterpret_cast<uint4*>(orow + cb * 32 + q * 8) = w;
        }
      }
    }
  }

  // ---- teardown: every warp reaches this point; TMEM is freed by its allocator warp ----
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

template <int D>
cudaError_t launch_prefill_tc(const PrefillParams& p, cudaStream_t s) {
  using C = PCfg<D>;
  auto kern = prefill_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = ((int64_t)p.max_q_len * p.group + kBM - 1) / kBM;
  return launch_pdl(kern, dim3((unsigned)tiles, (unsigned)p.pool.num_kv_heads, (unsigned)p.batch), dim3(kThreads),
                    (size_t)C::kSmem, s, p);
}

}  // namespace

cudaError_t launch_prefill_bf16(const PrefillParams& p, cudaStream_t s) {
  if (p.max_q_len <= 0 || p.batch <= 0) return cudaSuccess;
  return p.pool.head_dim == 128 ? launch_prefill_tc<128>(p, s) : launch_prefill_tc<64>(p, s);
}

}  // namespace pa
