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
// 128.
// * 1 TMA warp stages K/V tiles (3-stage rings) page by page: its lanes look
//   up one page each in block_table and issue one box per page (a whole
//   128-key tile when pages hold >= 128 slots), so a tile costs 128 /
//   min(page_size, 128) copies.  The 5-D view of the pool lands each box as
//   [8-slot block][64-dim slab][8 slots][128 B], i.e. 8-key row groups at one
//   uniform stride: exactly a K-major UMMA operand for K and an MN-major one
//   for V.  Slots at or past L_b in the last tile are zeroed in V.
// * 1 MMA thread issues tcgen05.mma: S = Q K^T (M 128, N 128, fp32 in TMEM,
//   double-buffered so S(j+1) overlaps the softmax of S(j)) and O += P V
//   (M 128, N head_dim, fp32 in TMEM, P from TMEM), each committed to
//   mbarriers.  It
//   issues whichever of the next S and the next PV is ready first.
// * 4 softmax warps own one TMEM lane (= one row) per thread: they stage their
//   own Q row once (cp.async), then per key tile tcgen05.ld the row of S,
//   apply the causal mask, run the online softmax in the log2 domain with a
//   lazily updated reference max (O and l are rescaled in TMEM only when the
//   row max grows by more than 2^8), write P as bf16 back to TMEM (double
//   buffered; PV reads its A operand from there), and at the end write O / l
//   to global as bf16.
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
constexpr int kNSK = 3;              // K ring stages
constexpr int kNSV = 3;              // V ring stages
constexpr int kSoftmaxWarps = 4;     // warps 0..3 (TMEM lane quarters 0..3)
constexpr int kMmaWarp = 4;
constexpr int kTmaWarp = 5;
// 6 warps: at most 2 per SM sub-partition, so each thread may hold 255
// registers (the softmax keeps a whole 128-column row of S in registers)
constexpr int kThreads = 32 * 6;
constexpr int kSlab = kBM * 128;     // one 64-column slab of the 128-row Q tile (16 KB)
constexpr float kRescaleThreshold = 8.f;  // log2 units

constexpr int kBarSlots = 24;

template <int D>
struct PCfg {
  static constexpr int kSlabs = D / 64;
  static constexpr int kRowBlock = kSlabs * 1024;      // one 8-key block of a K/V tile, all slabs
  static constexpr int kQBytes = kSlabs * kSlab;
  static constexpr int kKVTile = kBN * D * 2;          // K or V tile (128 keys)
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + kNSK * kKVTile;
  static constexpr int kPageOff = kVOff + kNSV * kKVTile;  // [8 tiles][32 lanes] page ids seen by the TMA warp
  static constexpr int kBarOff = kPageOff + 8 * 32 * 4;
  static constexpr int kSmem = kBarOff + kBarSlots * 8 + 16 + 1024;  // barriers, TMEM base, alignment slack
  static constexpr uint32_t kTmemCols = 512;           // S0 | S1 | O | P0 | P1
  static constexpr uint32_t kOCol = 256;
  static constexpr uint32_t kPCol = 384;               // P(j) as bf16 pairs: 64 columns at kPCol + (j & 1) * 64
};

// barriers: K and V stages are filled and freed separately (K(j) is free once
// S(j) is done, V(j) once PV(j) is done); S, P and PV-done each have one
// barrier per TMEM buffer (tile j uses j & 1), which keeps every parity
// waiter within one phase of its barrier: S(j+2) is issued only after PV(j),
// and PV(j+1) only after P(j+1).  B_VLAST completes the copies of a last V
// tile that the TMA warp still has to zero past L before publishing it.
enum { B_QFULL = 0, B_KFULL = 1, B_KEMPTY = B_KFULL + kNSK, B_VFULL = B_KEMPTY + kNSK, B_VEMPTY = B_VFULL + kNSV,
       B_SFULL = B_VEMPTY + kNSV, B_PFULL = B_SFULL + 2, B_PVDONE = B_PFULL + 2, B_VLAST = B_PVDONE + 2,
       B_COUNT = B_VLAST + 1 };
static_assert(B_COUNT <= kBarSlots, "barrier slots");

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                      PrefillParams p) {
  using C = PCfg<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int b = blockIdx.z, hk = blockIdx.y;
  const int G = p.group, Hq = p.num_q_heads;
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
  const uint32_t k_base = smem_u32(smem + C::kKOff);
  const uint32_t v_base = smem_u32(smem + C::kVOff);
  const uint32_t bars = smem_u32(smem + C::kBarOff);
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOff + kBarSlots * 8);

  if (tid == 0) {
    mbar_init(bar(B_QFULL), 32 * kSoftmaxWarps);
    for (int s = 0; s < kNSK; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < kNSV; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    mbar_init(bar(B_SFULL + 0), 1);
    mbar_init(bar(B_SFULL + 1), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_PFULL + i), 32 * kSoftmaxWarps);
      mbar_init(bar(B_PVDONE + i), 1);
    }
    mbar_init(bar(B_VLAST), 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const float sl2 = p.scale_log2;
  bool alive = true;

  if (warp == kTmaWarp) {
    // ======================= TMA producer (one warp) =======================
    // Per tile each lane < ops copies one page box (keys lane*kpo .. +kpo-1 of
    // the tile); lane 0 posts the byte count of the boxes actually issued.  K
    // and V are issued independently, each as soon as its ring slot is free
    // (polled by lane 0, the result shared with the warp so that all lanes take
    // the same path).  The page ids of tile j+1 are read while tile j is
    // issued, and a V tile reuses the ids its K tile looked up.
    griddep_wait();  // the pool rows of this step were written by the append kernel
    const int kpo = ps < kBN ? ps : kBN;  // keys per box
    const int ops = kBN / kpo;
    const uint32_t box_bytes = (uint32_t)kpo * D * 2;
    const int32_t* bt = p.block_table + (int64_t)b * p.max_blocks;
    int* page_ring = reinterpret_cast<int*>(smem + C::kPageOff);
    auto fetch = [&](int j) {  // raw block_table entry of this lane's box in tile j, -1 if none
      const int key = j * kBN + lane * kpo;
      return (j < nt && lane < ops && key < L) ? __ldg(bt + (key >> pshift)) : -1;
    };
    auto issue = [&](const CUtensorMap* map, uint32_t dst, int j, int page, uint32_t full) {
      const bool ok = page >= 0;
      const int cnt = __popc(__ballot_sync(0xffffffffu, ok));
      if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)cnt * box_bytes);
      __syncwarp();
      if (ok) {
        const int64_t slot = ((int64_t)page << pshift) + ((j * kBN + lane * kpo) & (ps - 1));
        tma_load_5d(dst + (uint32_t)(lane * (kpo / 8)) * C::kRowBlock, map, 0, 0, 0, (int)(slot >> 3), hk, full);
      }
    };
    auto slot_free = [&](int i) {  // lane 0 polls, the warp agrees
      int t = 0;
      if (lane == 0) t = mbar_test(bar(i >> 1), (uint32_t)(i & 1)) ? 1 : 0;
      return __shfl_sync(0xffffffffu, t, 0) != 0;
    };
    int jk = 0, jv = 0;
    int raw = fetch(0);
    unsigned long long t_last = global_ns();
    while (jv < nt && alive) {
      bool progressed = false;
      if (jk < nt && (jk < kNSK || slot_free(((B_KEMPTY + jk % kNSK) << 1) | (((jk / kNSK) - 1) & 1)))) {
        int page = raw;
        if (lane < ops && jk * kBN + lane * kpo < L) {
          if (page < 0 || page >= p.pool.num_pages) {
            record_error(p.err, ERR_BLOCK_TABLE, page);
            page = -1;
          }
        } else {
          page = -1;
        }
        page_ring[(jk & 7) * 32 + lane] = page;
        issue(&tmap_k, k_base + (jk % kNSK) * C::kKVTile, jk, page, bar(B_KFULL + jk % kNSK));
        ++jk;
        raw = fetch(jk);
        progressed = true;
      }
      if (jv < jk && (jv < kNSV || slot_free(((B_VEMPTY + jv % kNSV) << 1) | (((jv / kNSV) - 1) & 1)))) {
        const int s = jv % kNSV;
        const int page = page_ring[(jv & 7) * 32 + lane];
        const uint32_t vdst = v_base + s * C::kKVTile;
        const int valid = L - jv * kBN;  // keys of this tile below L (>= 1)
        if (valid >= kBN) {
          issue(&tmap_v, vdst, jv, page, bar(B_VFULL + s));
        } else {
          // last tile: slots valid..127 must hold zeros (they meet P = 0, and
          // the pool there may hold anything, NaN included)
          issue(&tmap_v, vdst, jv, page, bar(B_VLAST));
          alive = __all_sync(0xffffffffu, mbar_wait(bar(B_VLAST), 0, p.err));
          unsigned char* vt = smem + C::kVOff + s * C::kKVTile;
          const int chunks = (kBN - valid) * (D / 8);  // 16-byte chunks to clear
          for (int idx = lane; idx < chunks; idx += 32) {
            const int k = valid + idx / (D / 8), c = idx % (D / 8);
            *reinterpret_cast<uint4*>(vt + (k >> 3) * C::kRowBlock + (c >> 3) * 1024 + (k & 7) * 128 +
                                      (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_VFULL + s));
        }
        ++jv;
        progressed = true;
      }
      int give_up = 0;
      if (lane == 0) {
        const unsigned long long now = global_ns();
        if (progressed) {
          t_last = now;
        } else if (now - t_last > kWaitLimitNs) {
          record_error(p.err, ERR_TIMEOUT, jv);
          give_up = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, give_up, 0)) alive = false;
      if (!progressed) __nanosleep(64);
    }
  }

  if (warp == kMmaWarp && lane == 0) {
    // ======================= MMA issuer =======================
    // S(ns) may be issued once K(ns) is loaded and ns <= np + 1 (its TMEM
    // buffer held S(ns-2), whose softmax PV(ns-2) has consumed); PV(np) once
    // V(np) is loaded and P(np) is written.  Whichever is ready goes first.
    const uint32_t q_addr = smem_u32(q_s);
    constexpr uint32_t idesc_s = umma_idesc_bf16(kBM, kBN, false);
    constexpr uint32_t idesc_o = umma_idesc_bf16(kBM, D, true);
    if (alive) alive = mbar_wait(bar(B_QFULL), 0, p.err);
    int ns = 0, np = 0;
    unsigned long long t_last = global_ns();
    while (np < nt) {
      bool progressed = false;
      if (ns < nt && ns <= np + 1 &&
          (!alive || mbar_test(bar(B_KFULL + ns % kNSK), (uint32_t)((ns / kNSK) & 1)))) {
        tc_fence_after();
        const uint32_t k_addr = k_base + (ns % kNSK) * C::kKVTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // S[ns & 1] = Q K^T over 16-dim steps
          umma_bf16(tmem + (ns & 1) * kBN, umma_desc_sw128(q_addr + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024),
                    umma_desc_sw128(k_addr + (kk >> 2) * 1024 + (kk & 3) * 32, 16, C::kRowBlock), idesc_s, kk > 0);
        }
        umma_commit(bar(B_SFULL + (ns & 1)));
        umma_commit(bar(B_KEMPTY + ns % kNSK));
        ++ns;
        progressed = true;
      }
      if (np < ns && (!alive || (mbar_test(bar(B_PFULL + (np & 1)), (uint32_t)((np >> 1) & 1)) &&
                                 mbar_test(bar(B_VFULL + np % kNSV), (uint32_t)((np / kNSV) & 1))))) {
        tc_fence_after();
        const uint32_t v_addr = v_base + (np % kNSV) * C::kKVTile;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {  // O += P V over 16-key steps (two 8-key blocks each)
          umma_bf16_ts(tmem + C::kOCol, tmem + C::kPCol + (np & 1) * 64 + kk * 8,
                       umma_desc_sw128(v_addr + kk * 2 * C::kRowBlock, 1024, C::kRowBlock), idesc_o,
                       (np > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_PVDONE + (np & 1)));
        umma_commit(bar(B_VEMPTY + np % kNSV));
        ++np;
        progressed = true;
      }
      const unsigned long long now = global_ns();
      if (progressed) {
        t_last = now;
      } else if (alive && now - t_last > kWaitLimitNs) {
        record_error(p.err, ERR_TIMEOUT, np);
        alive = false;  // finish without waiting (results are garbage, recorded)
      } else {
        __nanosleep(32);
      }
    }
  }

  if (warp < kSoftmaxWarps) {
    // ======================= softmax: one TMEM lane (row) per thread =======================
    const int r = tid;  // row within the tile == TMEM lane
    const int R = row0 + r;
    const bool valid_row = R < rows_total;
    {  // this thread's Q row into the UMMA A layout (K-major, 128-byte swizzle); zeros past the last row
      const __nv_bfloat16* src = qp + (valid_row ? row_off(R) : 0);
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        cp_async_16(smem_u32(q_s + (c >> 3) * kSlab + r * 128 + (((c & 7) ^ (r & 7)) << 4)), src + c * 8,
                    valid_row ? 16 : 0);
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(bar(B_QFULL));
    }
    const int pos = valid_row ? first + R / G : pos_max;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float m_ref = -INFINITY, l = 0.f;
    for (int j = 0; j < nt; ++j) {
      if (alive) alive = mbar_wait(bar(B_SFULL + (j & 1)), (uint32_t)((j >> 1) & 1), p.err);
      tc_fence_after();
      const uint32_t s_addr = lane_base + (j & 1) * kBN;
      const int key0 = j * kBN;
      // the whole row of S(j): 128 fp32 in registers, scaled to log2 units in place
      uint32_t v[kBN / 32][32];
#pragma unroll
      for (int cb = 0; cb < kBN / 32; ++cb) tmem_ld32(s_addr + cb * 32, v[cb]);
      tmem_wait_ld();
      if (key0 + kBN - 1 > pos_min) {  // a diagonal tile: column c is visible iff c <= pos - key0
        const int lim = pos - key0;
#pragma unroll
        for (int cb = 0; cb < kBN / 32; ++cb)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            v[cb][e] = __float_as_uint(cb * 32 + e <= lim ? __uint_as_float(v[cb][e]) * sl2 : -INFINITY);
      } else {
#pragma unroll
        for (int cb = 0; cb < kBN / 32; ++cb)
#pragma unroll
          for (int e = 0; e < 32; ++e) v[cb][e] = __float_as_uint(__uint_as_float(v[cb][e]) * sl2);
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
      for (int cb = 0; cb < kBN / 32; ++cb)
#pragma unroll
        for (int e = 0; e < 32; ++e) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(v[cb][e]));
      const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // reference max: moved only when the row max grows by more than 2^8
      float alpha = 1.f;
      bool rescale = false;
      if (tmax > m_ref + kRescaleThreshold) {
        alpha = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - tmax);
        m_ref = tmax;
        l *= alpha;
        rescale = j > 0;
      }
      const float mbase = m_ref == -INFINITY ? 0.f : m_ref;
      // P = exp2(x - m) packed as bf16 pairs (in place of S); masked x = -inf gives 0
      float rs[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) rs[i] = 0.f;
#pragma unroll
      for (int cb = 0; cb < kBN / 32; ++cb)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = fast_exp2(__uint_as_float(v[cb][e]) - mbase);
          const float p1 = fast_exp2(__uint_as_float(v[cb][e + 1]) - mbase);
          rs[(e >> 1) & 7] += p0 + p1;
          v[cb][e >> 1] = pack_bf16(p0, p1);
        }
      const float rsum = ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      // O is rescaled in place only when some row of the warp moved its
      // reference max; PV(j-1) must have finished with O first.  (S(j) being
      // complete already implies PV(j-2) is, so P's buffer j & 1 is free.)
      if (__any_sync(0xffffffffu, rescale)) {
        if (alive) alive = mbar_wait(bar(B_PVDONE + ((j - 1) & 1)), (uint32_t)(((j - 1) >> 1) & 1), p.err);
        tc_fence_after();
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t o[32];
          tmem_ld32(lane_base + C::kOCol + cb * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(lane_base + C::kOCol + cb * 32, o);
        }
      }
      // P(j) into TMEM as the A operand of PV(j): 64 keys per 32 columns
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          w[i] = v[2 * h][i];
          w[16 + i] = v[2 * h + 1][i];
        }
        tmem_st32(lane_base + C::kPCol + (j & 1) * 64 + h * 32, w);
      }
      tmem_wait_st();
      l += rsum;
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + (j & 1)));
    }
    // ---- epilogue: O / l -> bf16 ----
    if (alive) alive = mbar_wait(bar(B_PVDONE + ((nt - 1) & 1)), (uint32_t)(((nt - 1) >> 1) & 1), p.err);
    tc_fence_after();
    griddep_wait();  // before the first global write
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* orow = outp + (valid_row ? row_off(R) : 0);
#pragma unroll
    for (int cb = 0; cb < D / 32; ++cb) {
      uint32_t o[32];
      tmem_ld32(lane_base + C::kOCol + cb * 32, o);
      tmem_wait_ld();
      if (valid_row) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
          w.y = pack_bf16(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
          w.z = pack_bf16(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
          w.w = pack_bf16(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
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
  const int ps = p.pool.page_size;
  if (ps < 8 || p.pool.page_shift < 0) return cudaErrorInvalidValue;
  const int kpo = ps < kBN ? ps : kBN;  // keys per TMA box
  const int64_t rows = p.pool.num_pages * (int64_t)ps;
  CUtensorMap tk, tv;
  if (!encode_pool_tmap_blocked(&tk, p.pool.key_pool, rows, p.pool.num_kv_heads, D, kpo / 8) ||
      !encode_pool_tmap_blocked(&tv, p.pool.value_pool, rows, p.pool.num_kv_heads, D, kpo / 8))
    return cudaErrorInvalidValue;
  auto kern = prefill_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = ((int64_t)p.max_q_len * p.group + kBM - 1) / kBM;
  return launch_pdl(kern, dim3((unsigned)tiles, (unsigned)p.pool.num_kv_heads, (unsigned)p.batch), dim3(kThreads),
                    (size_t)C::kSmem, s, tk, tv, p);
}

}  // namespace

cudaError_t launch_prefill_bf16(const PrefillParams& p, cudaStream_t s) {
  if (p.max_q_len <= 0 || p.batch <= 0) return cudaSuccess;
  return p.pool.head_dim == 128 ? launch_prefill_tc<128>(p, s) : launch_prefill_tc<64>(p, s);
}

}  // namespace pa
