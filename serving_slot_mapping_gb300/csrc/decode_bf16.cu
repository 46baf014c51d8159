// paged_attention_decode, bf16 path: split-KV online-softmax decode over the
// page pool plus a combine kernel, chained by programmatic dependent launch.
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
// * Inside a CTA a producer warp walks the range and, for each block,
//   follows block_table to the page and issues TMA tensor copies of the K and
//   V rows of that KV head into a ring of mbarrier-guarded stages (128 KB of
//   KV in flight per SM).  The ring is split among the consumer key groups;
//   each slot has one issuing lane and one consuming group, both in order,
//   and the lanes issue concurrently.  A second producer warp bulk-copies,
//   per pair ("segment"), the G query rows that share the KV head.
// * Consumer warps (key groups x row tiles of 16 query heads) take blocks
//   round-robin: S = Q K^T and O += P V with mma.sync m16n8k16 (bf16 in,
//   fp32 accumulate), online softmax in the log2 domain, output rescale
//   skipped when no running max moved.  Each page is read from HBM once for
//   all G heads (GQA/MQA reuse).
// * Keys at or past L_b are masked in S, and their V rows are zeroed in
//   shared memory, so stale or NaN-poisoned slots never reach the output.
// * At a segment end the key groups merge in shared memory.  A segment that
//   covers a whole pair writes the bf16 output directly; a pair cut by a
//   range boundary leaves one fp32 partial (m, l, o) per CTA in the
//   workspace, and the combine kernel merges them with
//   o = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i.
// * Both kernels are launched with programmatic stream serialization: the
//   split kernel's prologue (barriers, the seq_len prefix, block-table reads)
//   runs while the preceding append kernel finishes, and the combine kernel's
//   launch and prologue overlap the split kernel's tail.  Every access to data
//   an earlier kernel may write comes after griddepcontrol.wait.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace pa {

namespace {

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

template <int D, int RT>
struct Cfg {
  static constexpr int kNWK = RT == 1 ? 8 : 4;            // key groups
  static constexpr int kConsumers = kNWK * RT;            // consumer warps
  static constexpr int kThreads = 32 * (kConsumers + 2);  // + KV producer warp + Q producer warp
  static constexpr int kSlabs = D / 64;                   // 128-byte swizzle slabs per row
  static constexpr int kSlabBytes = 16 * 128;             // one slab of a 16-key tile
  static constexpr int kTileBytes = kSlabs * kSlabBytes;  // one 16-key K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = D == 128 ? 16 : 32;      // 128 KB of KV in flight per SM
  static constexpr int kSPG = kStages / kNWK;             // ring slots owned by one key group
  static constexpr int kQRows = 16 * RT;
  static constexpr int kQSlotBytes = kQRows * D * 2;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kBarOffset = kRingBytes + 2 * kQSlotBytes;
  static constexpr int kNumBars = 2 * kStages + 4;        // full[], empty[], qfull[2], qempty[2]
  static constexpr int kMergeOffset = kBarOffset + kNumBars * 8;
};

template <int D, int RT>
size_t split_smem_bytes(int G, int B) {
  using C = Cfg<D, RT>;
  return 1024 /* alignment slack */ + (size_t)C::kMergeOffset + (size_t)C::kNWK * G * (D + 2) * 4 +
         (size_t)(B + 1) * 4;
}

template <int D, int RT>
__global__ void __launch_bounds__(Cfg<D, RT>::kThreads, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                        DecodeParams p) {
  using C = Cfg<D, RT>;
  constexpr int S = C::kStages;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int G = p.group;
  const int B = p.batch;
  const int Hkv = p.pool.num_kv_heads;
  const int Hq = p.num_q_heads;
  unsigned char* ring = smem;
  unsigned char* qring = smem + C::kRingBytes;
  const uint32_t bars = smem_u32(smem + C::kBarOffset);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto qfull_bar = [&](int s) { return bars + 8u * (2 * S + s); };
  auto qempty_bar = [&](int s) { return bars + 8u * (2 * S + 2 + s); };
  float* mrg_o = reinterpret_cast<float*>(smem + C::kMergeOffset);  // [NWK][G][D]
  float* mrg_ml = mrg_o + C::kNWK * G * D;                           // [NWK][G][2]
  int* prefix = reinterpret_cast<int*>(mrg_ml + C::kNWK * G * 2);    // [B+1] 16-key blocks before b

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ps = p.pool.page_size, pshift = p.pool.page_shift;
  const int max_len = p.max_blocks * ps;

  // ---- set-up: barriers, zeroed Q slots (rows >= G stay zero), block prefix ----
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), RT);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(qfull_bar(s), 1);
      mbar_init(qempty_bar(s), C::kConsumers);
    }
    fence_mbar_init();
  }
  for (int i = tid; i < 2 * C::kQSlotBytes / 16; i += C::kThreads)
    reinterpret_cast<uint4*>(qring)[i] = make_uint4(0, 0, 0, 0);
  for (int b = tid; b < B; b += C::kThreads) prefix[b + 1] = nblk_of(p.seq_lens, b, max_len, p.err);
  if (tid == 0) prefix[0] = 0;
  fence_proxy_async_smem();
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < B; base += 32) {
      const int idx = base + lane;
      int v = idx < B ? prefix[idx + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
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
  griddep_launch_dependents();
  if (warp < C::kConsumers) griddep_wait();  // before any output write
  // sequences with no key (seq_len 0) get out = 0; CTA b % n writes them
  for (int b = c; b < B; b += n) {
    if (prefix[b + 1] != prefix[b]) continue;
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out) + (int64_t)b * Hq * D;
    if (warp < C::kConsumers)
      for (int idx = tid; idx < Hq * D; idx += C::kConsumers * 32) ob[idx] = __float2bfloat16_rn(0.f);
  }
  if (u0 >= u1) return;

  auto locate = [&](int64_t u) {
    Cursor cur;
    const int x = (int)(u / Hkv);
    int lo = 0, hi = B;  // largest b in [0, B) with prefix[b] <= x
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
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

  const __nv_bfloat16* qglob = static_cast<const __nv_bfloat16*>(p.q);

  if (warp == C::kConsumers + 1) {
    // ======================= Q producer =======================
    // Walks the CTA's segments (pairs) in order and bulk-copies each pair's
    // G query rows into a 2-slot ring; in-order issue keeps every parity wait
    // at most one phase ahead of the barrier.
    if (lane != 0) return;
    Cursor cur = locate(u0);
    bool alive = true;
    griddep_wait();
    for (int seg = 0; cur.u < u1; ++seg) {
      const int qs = seg & 1;
      if (seg >= 2 && alive) alive = mbar_wait(qempty_bar(qs), ((seg >> 1) - 1) & 1, p.err);
      const uint32_t qbytes = (uint32_t)(G * D * 2);
      mbar_arrive_expect_tx(qfull_bar(qs), qbytes);
      bulk_load(smem_u32(qring + qs * C::kQSlotBytes), qglob + ((int64_t)cur.b * Hq + (int64_t)cur.hk * G) * D,
                qbytes, qfull_bar(qs));
      advance(cur, (int)min((int64_t)(cur.nblk - cur.k), u1 - cur.u));
    }
    return;
  }

  if (warp == C::kConsumers) {
    // ======================= KV producer =======================
    // Ring slot l belongs to key group g = l / kSPG, which consumes its blocks
    // in order; lane l issues that group's blocks t = r, r + kSPG, ... (r =
    // l % kSPG), so each slot has one in-order writer and one in-order reader.
    // The lanes issue concurrently: measured on GB300, one thread issuing 2 KB
    // TMA boxes back to back streams only ~2.6 TB/s, sixteen lanes ~5.5 TB/s.
    if (lane >= S) return;
    const int g = lane / C::kSPG, r = lane % C::kSPG;
    const int slot = lane;
    const int R = ps < 16 ? ps : 16;  // rows per TMA box (page_size >= 8)
    Cursor cur = locate(u0);
    int64_t tcount = 0;  // blocks of group g before the current segment
    bool alive = true;
    griddep_wait();
    while (cur.u < u1) {
      const int nb_seg = (int)min((int64_t)(cur.nblk - cur.k), u1 - cur.u);
      const int cnt = nb_seg > g ? (nb_seg - g + C::kNWK - 1) / C::kNWK : 0;
      int64_t t = tcount + (((r - tcount) % C::kSPG) + C::kSPG) % C::kSPG;  // first t >= tcount, t % kSPG == r
      const int32_t* bt = p.block_table + (int64_t)cur.b * p.max_blocks;
      for (; t < tcount + cnt; t += C::kSPG) {
        const int j = g + (int)(t - tcount) * C::kNWK;  // block within the segment
        if (t >= C::kSPG && alive)
          alive = mbar_wait(empty_bar(slot), (uint32_t)(((t / C::kSPG) - 1) & 1), p.err);
        const int key0 = (cur.k + j) * 16;
        int rows[2] = {-1, -1};
        int nbox = 0;
        for (int q = 0; q < 16 / R; ++q) {
          const int kk = key0 + q * R;
          if (kk >= cur.L) break;
          const int page = __ldg(bt + (kk >> pshift));
          if (page < 0 || page >= p.pool.num_pages) {
            record_error(p.err, ERR_BLOCK_TABLE, page);
            continue;
          }
          rows[q] = page * ps + (kk & (ps - 1));
          ++nbox;
        }
        mbar_arrive_expect_tx(full_bar(slot), (uint32_t)(nbox * 2 * C::kSlabs * R * 128));
        const uint32_t kdst = smem_u32(ring + slot * C::kStageBytes);
        const uint32_t vdst = kdst + C::kTileBytes;
        for (int q = 0; q < 16 / R; ++q) {
          if (rows[q] < 0) continue;
#pragma unroll
          for (int sl = 0; sl < C::kSlabs; ++sl) {
            tma_load_3d(kdst + sl * C::kSlabBytes + q * R * 128, &tmap_k, sl * 64, cur.hk, rows[q], full_bar(slot));
            tma_load_3d(vdst + sl * C::kSlabBytes + q * R * 128, &tmap_v, sl * 64, cur.hk, rows[q], full_bar(slot));
          }
        }
      }
      tcount += cnt;
      advance(cur, nb_seg);
    }
    return;
  }

  // ======================= consumer warps =======================
  const int rt = warp / C::kNWK;  // row tile: query heads rt*16 .. rt*16+15 of the group
  const int wk = warp % C::kNWK;  // key group: blocks j with j % kNWK == wk
  const int rA = rt * 16 + (lane >> 2), rB = rA + 8;
  const float sl2 = p.scale_log2;
  const int mi = lane >> 3, rr = lane & 7;
  Cursor cc = locate(u0);
  int seg = -1;
  int64_t tg = 0;  // blocks this key group has consumed so far
  bool alive = true;
  while (cc.u < u1) {
    ++seg;
    const int nb_seg = (int)min((int64_t)(cc.nblk - cc.k), u1 - cc.u);
    const int first_k = cc.k;
    // ---- the pair's query rows (A fragments of m16n8k16) ----
    uint32_t qf[D / 16][4];
    {
      const int qs = seg & 1;
      if (alive) alive = mbar_wait(qfull_bar(qs), (seg >> 1) & 1, p.err);
      const uint32_t* qsm = reinterpret_cast<const uint32_t*>(qring + qs * C::kQSlotBytes);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int d0 = kk * 16 + (lane & 3) * 2;
        qf[kk][0] = qsm[(rA * D + d0) >> 1];
        qf[kk][1] = qsm[(rB * D + d0) >> 1];
        qf[kk][2] = qsm[(rA * D + d0 + 8) >> 1];
        qf[kk][3] = qsm[(rB * D + d0 + 8) >> 1];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty_bar(qs));
    }
    float o[D / 8][4];
#pragma unroll
    for (int n8 = 0; n8 < D / 8; ++n8) o[n8][0] = o[n8][1] = o[n8][2] = o[n8][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int j = wk; j < nb_seg; j += C::kNWK, ++tg) {
      const int slot = wk * C::kSPG + (int)(tg % C::kSPG);
      if (alive) alive = mbar_wait(full_bar(slot), (uint32_t)((tg / C::kSPG) & 1), p.err);
      unsigned char* kt = ring + slot * C::kStageBytes;
      unsigned char* vt = kt + C::kTileBytes;
      const int valid = cc.L - (first_k + j) * 16;  // >= 1
      if (valid < 16) {
        // rows past L_b may hold stale or poisoned data: zero them in V (K is masked below)
        for (int e = lane; e < (16 - valid) * C::kSlabs * 8; e += 32) {
          const int row = valid + e / (C::kSlabs * 8);
          const int rem = e % (C::kSlabs * 8);
          *reinterpret_cast<uint4*>(vt + (rem >> 3) * C::kSlabBytes + row * 128 + (rem & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
      float s[2][4];
#pragma unroll
      for (int t = 0; t < 2; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kbase + sw128((mi >> 1) * 8 + rr, kk * 2 + (mi & 1), C::kSlabBytes), b0, b1, b2, b3);
        mma_bf16_16816(s[0], qf[kk], b0, b1);
        mma_bf16_16816(s[1], qf[kk], b2, b3);
      }
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
      for (int jj = 0; jj < D / 16; ++jj) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vbase + sw128((mi & 1) * 8 + rr, 2 * jj + (mi >> 1), C::kSlabBytes), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * jj], pa, b0, b1);
        mma_bf16_16816(o[2 * jj + 1], pa, b2, b3);
      }
      if (valid < 16) fence_proxy_async_smem();  // our zero stores precede the next TMA into this slot
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(slot));
    }

    // ---- merge the key groups' partial softmax states of this segment ----
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
      if (rA < G) *reinterpret_cast<float2*>(&mrg_o[(wk * G + rA) * D + col]) = make_float2(o[n8][0], o[n8][1]);
      if (rB < G) *reinterpret_cast<float2*>(&mrg_o[(wk * G + rB) * D + col]) = make_float2(o[n8][2], o[n8][3]);
    }
    named_barrier(1, C::kConsumers * 32);
    const bool complete = (first_k == 0) && (first_k + nb_seg == cc.nblk);
    const int64_t pair = (int64_t)cc.b * Hkv + cc.hk;
    const int64_t pslot = pair + c;
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out) + ((int64_t)cc.b * Hq + (int64_t)cc.hk * G) * D;
    for (int idx = tid; idx < G * D; idx += C::kConsumers * 32) {
      const int g = idx / D, d = idx - (idx / D) * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::kNWK; ++w) M = fmaxf(M, mrg_ml[(w * G + g) * 2]);
      float acc = 0.f, den = 0.f;
#pragma unroll
      for (int w = 0; w < C::kNWK; ++w) {
        const float mw = mrg_ml[(w * G + g) * 2];
        const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
        acc += f * mrg_o[(w * G + g) * D + d];
        den += f * mrg_ml[(w * G + g) * 2 + 1];
      }
      if (complete) {
        outp[idx] = __float2bfloat16_rn(den > 0.f ? acc / den : 0.f);
      } else {
        p.part_o[(pslot * G + g) * D + d] = acc;
        if (d == 0) p.part_ml[pslot * G + g] = make_float2(M, den);
      }
    }
    named_barrier(1, C::kConsumers * 32);
    advance(cc, nb_seg);
  }
}

// Merge the partials of pairs that were cut across CTAs.
__global__ void __launch_bounds__(128) decode_combine_kernel(DecodeParams p, int D) {
  const int Hkv = p.pool.num_kv_heads;
  const int G = p.group;
  const int pair = blockIdx.x;
  const int b = pair / Hkv, hk = pair - (pair / Hkv) * Hkv;
  const int max_len = p.max_blocks * p.pool.page_size;
  // The prologue reads only seq_lens and overlaps the split kernel's tail;
  // partials are read after the split grid has completed.
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
  griddep_wait();
  if (nblk == 0) return;  // zeroed by the split kernel
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

template <int D, int RT>
cudaError_t launch_split(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  using C = Cfg<D, RT>;
  const size_t smem = split_smem_bytes<D, RT>(p.group, p.batch);
  auto kern = decode_split_kernel<D, RT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(p.num_ctas), dim3(C::kThreads), smem, s, tk, tv, p);
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

size_t decode_smem_bytes(int head_dim, int group, int batch) {
  const int RT = group <= 16 ? 1 : 2;
  if (head_dim == 128)
    return RT == 1 ? split_smem_bytes<128, 1>(group, batch) : split_smem_bytes<128, 2>(group, batch);
  return RT == 1 ? split_smem_bytes<64, 1>(group, batch) : split_smem_bytes<64, 2>(group, batch);
}

cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t s) {
  const int D = p.pool.head_dim;
  const int RT = p.group <= 16 ? 1 : 2;
  const int R = p.pool.page_size < 16 ? p.pool.page_size : 16;
  const int64_t rows = p.pool.num_pages * (int64_t)p.pool.page_size;
  CUtensorMap tk, tv;
  if (!encode_pool_tmap(&tk, p.pool.key_pool, rows, p.pool.num_kv_heads, D, R) ||
      !encode_pool_tmap(&tv, p.pool.value_pool, rows, p.pool.num_kv_heads, D, R))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (D == 128) {
    e = RT == 1 ? launch_split<128, 1>(p, tk, tv, s) : launch_split<128, 2>(p, tk, tv, s);
  } else {
    e = RT == 1 ? launch_split<64, 1>(p, tk, tv, s) : launch_split<64, 2>(p, tk, tv, s);
  }
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_combine_kernel, dim3(p.batch * p.pool.num_kv_heads), dim3(128), 0, s, p, D);
}

}  // namespace pa
