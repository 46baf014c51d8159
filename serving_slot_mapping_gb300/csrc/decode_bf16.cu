// paged_attention_decode, bf16 path: split-KV online-softmax decode over the
// page pool plus a combine kernel.
//
// What is computed (onnxruntime/mobius PR #395 "Add paged / block-table KV
// cache export", "How it works": Gather(pool, block_table) then Attention
// masked to nonpad_kv_seqlen; decode is the one-query-token case):
//   out[b, h] = softmax_j(scale * q[b,h] . K_b[j, h/G]) V_b[j, h/G],  j < L_b
//
// Work decomposition (GB300-first, not from the pages):
// * The unit of work is a 16-key block of one (sequence, KV head) pair.  All
//   units of the batch are laid out in one list, sequence-major, and the
//   list is cut into `num_ctas` equal contiguous ranges (one persistent CTA
//   per SM).  Every CTA streams the same number of KV bytes whatever the mix
//   of context lengths, so there is no tail of idle SMs.
// * A CTA walks its range pair by pair ("segments").  NWK warps take NWK
//   consecutive blocks per pipeline stage; RT row-tiles of 16 query heads
//   cover the G heads that share the KV head, so each page is read from HBM
//   once for all G heads (GQA/MQA reuse).
// * Pages are staged with 16-byte cp.async into an XOR-swizzled smem ring of
//   STAGES stages, following block_table per key row.  Rows at or past L_b
//   are zero-filled and masked, so stale or NaN-poisoned slots never reach
//   the arithmetic.
// * QK^T and PV use mma.sync m16n8k16 bf16 with fp32 accumulation; the
//   softmax is online in the log2 domain (scale * log2(e) folded in).  The
//   output rescale is skipped when no running max moved.
// * A segment that covers a whole pair writes the bf16 output directly.  A
//   pair cut by a range boundary leaves one fp32 partial (m, l, o) per CTA
//   in the workspace, and the combine kernel merges them with
//   o = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pa {

namespace {

constexpr int kNWK = 4;  // warps along keys (blocks per stage)

__device__ __forceinline__ int nblk_of(const int32_t* seq_lens, int b, int max_len,
                                       unsigned long long* err) {
  int L = __ldg(seq_lens + b);
  if (L < 0 || L > max_len) {
    record_error(err, ERR_SEQ_LEN, L);
    L = L < 0 ? 0 : max_len;
  }
  return (L + 15) >> 4;
}

__device__ __forceinline__ int seq_len_of(const int32_t* seq_lens, int b, int max_len) {
  int L = __ldg(seq_lens + b);
  return L < 0 ? 0 : (L > max_len ? max_len : L);
}

// CTA that owns unit u when U units are cut into n ranges [c*U/n, (c+1)*U/n).
__device__ __forceinline__ int cta_of_unit(int64_t u, int64_t U, int n) {
  return (int)(((u + 1) * (int64_t)n - 1) / U);
}

// True when CTA c owns no unit (more CTAs than units): it writes no partial.
__device__ __forceinline__ bool cta_range_empty(int c, int64_t U, int n) {
  return (int64_t)c * U / n == (int64_t)(c + 1) * U / n;
}

struct Cursor {
  int b, hk, k, nblk, L;
  int64_t u;
};

template <int D, int RT, int STAGES>
struct Cfg {
  static constexpr int kThreads = 32 * RT * kNWK;
  static constexpr int kRowBytes = D * 2;
  static constexpr int kChunks = D / 8;                 // 16-byte chunks per row
  static constexpr int kBlockBytes = 16 * kRowBytes;    // one 16-key K or V tile
  static constexpr int kStageBytes = kNWK * 2 * kBlockBytes;
  static constexpr int kRowsPerStage = kNWK * 2 * 16;
  static constexpr int kCopiesPerThread = kRowsPerStage * kChunks / kThreads;
};

template <int D, int RT, int STAGES>
__global__ void __launch_bounds__(32 * RT * kNWK, 1) decode_split_kernel(DecodeParams p) {
  using C = Cfg<D, RT, STAGES>;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int G = p.group;
  const int B = p.batch;
  const int Hkv = p.pool.num_kv_heads;
  const int Hq = p.num_q_heads;
  unsigned char* ring = smem;
  float* mrg_o = reinterpret_cast<float*>(smem + STAGES * C::kStageBytes);  // [NWK][G][D]
  float* mrg_ml = mrg_o + kNWK * G * D;                                      // [NWK][G][2]
  int* prefix = reinterpret_cast<int*>(mrg_ml + kNWK * G * 2);               // [B+1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wk = warp % kNWK;
  const int rt = warp / kNWK;
  const int ps = p.pool.page_size, pshift = p.pool.page_shift;
  const int max_len = p.max_blocks * ps;

  // ---- prefix sum of 16-key block counts over the batch ----
  for (int b = tid; b < B; b += C::kThreads) prefix[b + 1] = nblk_of(p.seq_lens, b, max_len, p.err);
  if (tid == 0) prefix[0] = 0;
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < B; base += 32) {
      int idx = base + lane;
      int v = idx < B ? prefix[idx + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (idx < B) prefix[idx + 1] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();

  const int64_t NB = prefix[B];
  const int64_t U = NB * Hkv;
  const int n = p.num_ctas, c = blockIdx.x;
  const int64_t u0 = (int64_t)c * U / n, u1 = (int64_t)(c + 1) * U / n;
  if (u0 >= u1) return;

  auto locate = [&](int64_t u) {
    Cursor cur;
    const int x = (int)(u / Hkv);
    int lo = 0, hi = B;  // largest b in [0, B) with prefix[b] <= x
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (prefix[mid] <= x) lo = mid; else hi = mid;
    }
    cur.b = lo;
    cur.nblk = prefix[lo + 1] - prefix[lo];
    const int r = (int)(u - (int64_t)Hkv * prefix[lo]);
    cur.hk = r / cur.nblk;
    cur.k = r - cur.hk * cur.nblk;
    cur.L = seq_len_of(p.seq_lens, cur.b, max_len);
    cur.u = u;
    return cur;
  };
  auto stage_len = [&](const Cursor& cur) {
    int64_t left = u1 - cur.u;
    int nb = cur.nblk - cur.k;
    if (nb > kNWK) nb = kNWK;
    if (left < nb) nb = (int)left;
    return nb;
  };
  auto advance = [&](Cursor& cur, int nb) {
    cur.u += nb;
    cur.k += nb;
    if (cur.k == cur.nblk) {
      cur.k = 0;
      if (++cur.hk == Hkv) {
        cur.hk = 0;
        do { ++cur.b; } while (cur.b < B && prefix[cur.b + 1] == prefix[cur.b]);
        if (cur.b < B) {
          cur.nblk = prefix[cur.b + 1] - prefix[cur.b];
          cur.L = seq_len_of(p.seq_lens, cur.b, max_len);
        }
      }
    }
  };

  const __nv_bfloat16* kpool = static_cast<const __nv_bfloat16*>(p.pool.key_pool);
  const __nv_bfloat16* vpool = static_cast<const __nv_bfloat16*>(p.pool.value_pool);
  const int64_t row_elems = (int64_t)Hkv * D;

  // Issue the cp.async copies of one stage (nb blocks of pair cur) into ring slot `slot`.
  auto load_stage = [&](const Cursor& cur, int nb, int slot) {
    unsigned char* st = ring + slot * C::kStageBytes;
    const int32_t* bt = p.block_table + (int64_t)cur.b * p.max_blocks;
#pragma unroll
    for (int i = 0; i < C::kCopiesPerThread; ++i) {
      const int idx = tid + i * C::kThreads;
      const int row = idx / C::kChunks;       // [w][tensor][r]
      const int ch = idx % C::kChunks;
      const int w = row >> 5, tensor = (row >> 4) & 1, r = row & 15;
      const int j = (cur.k + w) * 16 + r;
      bool ok = (w < nb) && (j < cur.L);
      const __nv_bfloat16* src = kpool;
      if (ok) {
        const int page = __ldg(bt + (j >> pshift));
        if (page < 0 || page >= p.pool.num_pages) {
          record_error(p.err, ERR_BLOCK_TABLE, page);
          ok = false;
        } else {
          const int64_t slot_row = ((int64_t)page << pshift) + (j & (ps - 1));
          src = (tensor ? vpool : kpool) + slot_row * row_elems + (int64_t)cur.hk * D + ch * 8;
        }
      }
      cp_async_16(smem_u32(st + (w * 2 + tensor) * C::kBlockBytes + swz(r, ch, C::kRowBytes)),
                  src, ok ? 16 : 0);
    }
  };

  // ---- prologue: fill STAGES-1 stages ----
  Cursor pc = locate(u0);
  int pslot = 0;
#pragma unroll 1
  for (int s = 0; s < STAGES - 1; ++s) {
    if (pc.u < u1) {
      const int nb = stage_len(pc);
      load_stage(pc, nb, pslot);
      advance(pc, nb);
    }
    cp_async_commit();
    pslot = (pslot + 1) % STAGES;
  }

  Cursor cc = locate(u0);
  int cslot = 0;
  bool seg_start = true;
  int seg_first_k = cc.k;

  // per-warp state: two rows per thread (g = lane/4 and g + 8 of this row tile)
  uint32_t qf[D / 16][4];
  float o[D / 8][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int rA = rt * 16 + (lane >> 2), rB = rA + 8;
  const float sl2 = p.scale_log2;

#pragma unroll 1
  while (cc.u < u1) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    // refill the slot consumed in the previous iteration
    if (pc.u < u1) {
      const int nb = stage_len(pc);
      load_stage(pc, nb, pslot);
      advance(pc, nb);
    }
    cp_async_commit();
    pslot = (pslot + 1) % STAGES;

    const int nb = stage_len(cc);
    if (seg_start) {
      seg_start = false;
      seg_first_k = cc.k;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
#pragma unroll
      for (int n8 = 0; n8 < D / 8; ++n8) o[n8][0] = o[n8][1] = o[n8][2] = o[n8][3] = 0.f;
      const uint32_t* qb = reinterpret_cast<const uint32_t*>(
          static_cast<const __nv_bfloat16*>(p.q) + ((int64_t)cc.b * Hq + (int64_t)cc.hk * G) * D);
      const int cpair = (lane & 3);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int d0 = kk * 16 + cpair * 2;
        qf[kk][0] = rA < G ? __ldg(qb + (rA * D + d0) / 2) : 0u;
        qf[kk][1] = rB < G ? __ldg(qb + (rB * D + d0) / 2) : 0u;
        qf[kk][2] = rA < G ? __ldg(qb + (rA * D + d0 + 8) / 2) : 0u;
        qf[kk][3] = rB < G ? __ldg(qb + (rB * D + d0 + 8) / 2) : 0u;
      }
    }

    if (wk < nb) {
      const unsigned char* kt = ring + cslot * C::kStageBytes + (wk * 2) * C::kBlockBytes;
      const unsigned char* vt = kt + C::kBlockBytes;
      const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
      float s[2][4];
#pragma unroll
      for (int t = 0; t < 2; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kbase + swz((mi >> 1) * 8 + rr, kk * 2 + (mi & 1), C::kRowBytes), b0, b1, b2, b3);
        mma_bf16_16816(s[0], qf[kk], b0, b1);
        mma_bf16_16816(s[1], qf[kk], b2, b3);
      }
      const int valid = cc.L - (cc.k + wk) * 16;  // >= 1
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = t * 8 + (lane & 3) * 2 + (e & 1);
          s[t][e] = key < valid ? s[t][e] * sl2 : -INFINITY;
        }
      float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
      float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
      float p_[2][4];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        p_[t][0] = fast_exp2(s[t][0] - mn0);
        p_[t][1] = fast_exp2(s[t][1] - mn0);
        p_[t][2] = fast_exp2(s[t][2] - mn1);
        p_[t][3] = fast_exp2(s[t][3] - mn1);
      }
      l0 = l0 * al0 + (p_[0][0] + p_[0][1] + p_[1][0] + p_[1][1]);
      l1 = l1 * al1 + (p_[0][2] + p_[0][3] + p_[1][2] + p_[1][3]);
      if (__any_sync(0xffffffffu, (al0 != 1.f) | (al1 != 1.f))) {
#pragma unroll
        for (int n8 = 0; n8 < D / 8; ++n8) {
          o[n8][0] *= al0; o[n8][1] *= al0;
          o[n8][2] *= al1; o[n8][3] *= al1;
        }
      }
      m0 = mn0;
      m1 = mn1;
      uint32_t pa[4];
      pa[0] = pack_bf16(p_[0][0], p_[0][1]);
      pa[1] = pack_bf16(p_[0][2], p_[0][3]);
      pa[2] = pack_bf16(p_[1][0], p_[1][1]);
      pa[3] = pack_bf16(p_[1][2], p_[1][3]);
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vbase + swz((mi & 1) * 8 + rr, 2 * j + (mi >> 1), C::kRowBytes), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * j], pa, b0, b1);
        mma_bf16_16816(o[2 * j + 1], pa, b2, b3);
      }
    }

    const bool pair_end = (cc.k + nb == cc.nblk);
    const bool seg_end = pair_end || (cc.u + nb == u1);
    if (seg_end) {
      // ---- merge the NWK warps' partial softmax states of this segment ----
      float la = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
      la += __shfl_xor_sync(0xffffffffu, la, 2);
      float lb = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
      lb += __shfl_xor_sync(0xffffffffu, lb, 2);
      if ((lane & 3) == 0) {
        if (rA < G) { mrg_ml[(wk * G + rA) * 2] = m0; mrg_ml[(wk * G + rA) * 2 + 1] = la; }
        if (rB < G) { mrg_ml[(wk * G + rB) * 2] = m1; mrg_ml[(wk * G + rB) * 2 + 1] = lb; }
      }
#pragma unroll
      for (int n8 = 0; n8 < D / 8; ++n8) {
        const int col = n8 * 8 + (lane & 3) * 2;
        if (rA < G) {
          mrg_o[(wk * G + rA) * D + col] = o[n8][0];
          mrg_o[(wk * G + rA) * D + col + 1] = o[n8][1];
        }
        if (rB < G) {
          mrg_o[(wk * G + rB) * D + col] = o[n8][2];
          mrg_o[(wk * G + rB) * D + col + 1] = o[n8][3];
        }
      }
      __syncthreads();
      const bool complete = (seg_first_k == 0) && pair_end;
      const int64_t pair = (int64_t)cc.b * Hkv + cc.hk;
      const int64_t pslot_idx = pair + c;
      __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out) + ((int64_t)cc.b * Hq + (int64_t)cc.hk * G) * D;
      for (int idx = tid; idx < G * D; idx += C::kThreads) {
        const int g = idx / D, d = idx - (idx / D) * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kNWK; ++w) M = fmaxf(M, mrg_ml[(w * G + g) * 2]);
        float acc = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < kNWK; ++w) {
          const float mw = mrg_ml[(w * G + g) * 2];
          const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
          acc += f * mrg_o[(w * G + g) * D + d];
          den += f * mrg_ml[(w * G + g) * 2 + 1];
        }
        if (complete) {
          outp[idx] = __float2bfloat16_rn(den > 0.f ? acc / den : 0.f);
        } else {
          p.part_o[(pslot_idx * G + g) * D + d] = acc;
          if (d == 0) p.part_ml[pslot_idx * G + g] = make_float2(M, den);
        }
      }
      __syncthreads();
      seg_start = true;
    }
    advance(cc, nb);
    cslot = (cslot + 1) % STAGES;
  }
  cp_async_wait<0>();
}

// Merge the partials of pairs that were cut across CTAs; zero-fill empty sequences.
__global__ void __launch_bounds__(128) decode_combine_kernel(DecodeParams p, int D) {
  const int Hkv = p.pool.num_kv_heads;
  const int G = p.group;
  const int pair = blockIdx.x;
  const int b = pair / Hkv, hk = pair - (pair / Hkv) * Hkv;
  const int max_len = p.max_blocks * p.pool.page_size;
  __shared__ long long red[2][4];
  long long before = 0, total = 0;
  for (int i = threadIdx.x; i < p.batch; i += blockDim.x) {
    const int nb = (seq_len_of(p.seq_lens, i, max_len) + 15) >> 4;
    total += nb;
    if (i < b) before += nb;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  if ((threadIdx.x & 31) == 0) { red[0][threadIdx.x >> 5] = before; red[1][threadIdx.x >> 5] = total; }
  __syncthreads();
  before = red[0][0] + red[0][1] + red[0][2] + red[0][3];
  total = red[1][0] + red[1][1] + red[1][2] + red[1][3];
  const int nblk = (seq_len_of(p.seq_lens, b, max_len) + 15) >> 4;
  __nv_bfloat16* outp =
      static_cast<__nv_bfloat16*>(p.out) + ((int64_t)b * p.num_q_heads + (int64_t)hk * G) * D;
  if (nblk == 0) {
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) outp[idx] = __float2bfloat16_rn(0.f);
    return;
  }
  const int64_t U = total * Hkv;
  const int64_t us = before * Hkv + (int64_t)hk * nblk, ue = us + nblk;
  const int c0 = cta_of_unit(us, U, p.num_ctas), c1 = cta_of_unit(ue - 1, U, p.num_ctas);
  if (c0 == c1) return;  // written by the split kernel
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int g = idx / D, d = idx - (idx / D) * D;
    float M = -INFINITY;
    for (int cc = c0; cc <= c1; ++cc) {
      if (cta_range_empty(cc, U, p.num_ctas)) continue;  // wrote no partial
      M = fmaxf(M, p.part_ml[((int64_t)pair + cc) * G + g].x);
    }
    float acc = 0.f, den = 0.f;
    for (int cc = c0; cc <= c1; ++cc) {
      if (cta_range_empty(cc, U, p.num_ctas)) continue;
      const int64_t sidx = (int64_t)pair + cc;
      const float2 ml = p.part_ml[sidx * G + g];
      const float f = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
      acc += f * p.part_o[(sidx * G + g) * D + d];
      den += f * ml.y;
    }
    outp[idx] = __float2bfloat16_rn(den > 0.f ? acc / den : 0.f);
  }
}

template <int D, int RT, int STAGES>
size_t split_smem_bytes(int G, int B) {
  using C = Cfg<D, RT, STAGES>;
  return (size_t)STAGES * C::kStageBytes + (size_t)kNWK * G * (D + 2) * 4 + (size_t)(B + 1) * 4;
}

template <int D, int RT, int STAGES>
cudaError_t launch_split(const DecodeParams& p, cudaStream_t s) {
  using C = Cfg<D, RT, STAGES>;
  const size_t smem = split_smem_bytes<D, RT, STAGES>(p.group, p.batch);
  auto kern = decode_split_kernel<D, RT, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<p.num_ctas, C::kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

int64_t decode_partial_slots(int32_t batch, int32_t num_kv_heads, int32_t num_ctas) {
  return (int64_t)batch * num_kv_heads + num_ctas;
}

int decode_num_ctas(int num_sms, int32_t batch, int32_t num_kv_heads, int32_t max_seq_len,
                    int32_t head_dim, int32_t group) {
  (void)head_dim;
  (void)group;
  const int64_t ubound = (int64_t)batch * num_kv_heads * (((int64_t)max_seq_len + 15) / 16);
  int64_t n = num_sms;
  if (ubound < n) n = ubound;
  if (n < 1) n = 1;
  return (int)n;
}

cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t s) {
  const int D = p.pool.head_dim;
  const int RT = p.group <= 16 ? 1 : 2;
  cudaError_t e;
  if (D == 128) {
    e = RT == 1 ? launch_split<128, 1, 4>(p, s) : launch_split<128, 2, 4>(p, s);
  } else {
    e = RT == 1 ? launch_split<64, 1, 8>(p, s) : launch_split<64, 2, 8>(p, s);
  }
  if (e != cudaSuccess) return e;
  const int pairs = p.batch * p.pool.num_kv_heads;
  decode_combine_kernel<<<pairs, 128, 0, s>>>(p, D);
  return cudaGetLastError();
}

}  // namespace pa
