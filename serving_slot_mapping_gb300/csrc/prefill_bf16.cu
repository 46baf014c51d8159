// paged_attention_prefill, bf16 path: tcgen05 / TMEM varlen causal attention.
//
// What is computed: varlen causal attention for packed new tokens
// (query_start_loc layout of ROCm/maxtext PR #93 "[Draft] kv paged kernels",
// the gpu_paged commit), masked by is_causal + nonpad_kv_seqlen as in
// onnxruntime/mobius PR #395 "Add paged / block-table KV cache export" ("How
// it works", step 3).  Token i of sequence b sits at absolute position
// p = L_b - n_b + i and sees keys 0..p, read from the pages in block_table.
//
// Tiling (GB300-first): a CTA owns 256 packed rows of one (sequence, KV head)
// -- row r is query token r / G, query head hk*G + r % G -- as two 128-row
// query tiles A and B that share every K/V tile staged in shared memory, so
// each byte brought in feeds twice the tensor-core work (the copies, not the
// tensor core, bound a single-tile CTA: with ~2 us of loaded L2 latency, the
// bytes a CTA can keep in flight cap its tile rate).  Keys come in tiles of
// 128.
// * 1 TMA warp stages K/V tiles (3- and 2-stage rings) page by page: its
//   lanes look up one page each in block_table and issue one box per page (a
//   whole 128-key tile when pages hold >= 128 slots).  The 5-D view of the
//   pool lands each box as [8-slot block][64-dim slab][8 slots][128 B], i.e.
//   8-key row groups at one uniform stride: exactly a K-major UMMA operand
//   for K and an MN-major one for V.  Slots at or past L_b in the last tile
//   are zeroed in V.
// * 1 MMA thread issues tcgen05.mma in a fixed order, S_A(0) S_B(0), then per
//   key tile j: PV_A(j) S_A(j+1) PV_B(j) S_B(j+1), so the tensor core works
//   on one query tile while the other tile's softmax runs.  S = Q K^T and
//   O += P V are M 128 with fp32 accumulators in TMEM; P is bf16 in TMEM,
//   written over the columns of S it came from, and read by PV as its A
//   operand.  (tcgen05 operations of one thread execute in issue order, so
//   S(j+1) overwrites P(j) only after PV(j) has read it.)
// * 2 softmax warpgroups, one per query tile, own one TMEM lane (= one row)
//   per thread: they stage their own Q row once (cp.async), then per key tile
//   read the row of S from TMEM twice (the max, then exp2 and P), apply the
//   causal mask, run the online softmax in the log2 domain with a lazily
//   updated reference max (O and l are rescaled in TMEM only when the row
//   max grows by more than 2^8), and at the end write O / l as bf16.
// Fully masked key tiles are never loaded or multiplied.
//
// e4m3 pools (KV8): the TMA lands each page's codes ([keys][D B], unswizzled)
// in the upper half of the K or V ring slot, and two more warps (one for K,
// one for V, so that neither ring waits on the other's conversions) convert
// the tile in place into the f16 layout above (cvt e4m3x2 -> f16x2 is exact:
// every e4m3 value is an f16), zeroing rows at or past L_b.  Q is staged and P
// written as f16, so both products are kind::f16 with f16 operands; k_scale is
// folded into the softmax scale and v_scale into the final normalisation.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace pa {

namespace {

constexpr int kBM = 128;             // packed query rows per query tile (TMEM lanes)
constexpr int kQT = 2;               // query tiles per CTA
constexpr int kBN = 128;             // keys per tile
constexpr int kNSK = 3;              // K ring stages
constexpr int kNSV = 2;              // V ring stages
constexpr int kMmaWarp = 8;          // warps 0..7: softmax of query tile (warp / 4)
constexpr int kTmaWarp = 9;
constexpr int kCvtWarp = 10;         // e4m3 pools: warp 10 converts landed K tiles to f16, warp 11 V tiles
// 10 warps (12 for e4m3 pools): at most 3 on an SM sub-partition, so at most
// 168 registers a thread; the softmax holds half a row of S (64 fp32) at a time
constexpr int kSlab = kBM * 128;     // one 64-column slab of a 128-row Q tile (16 KB)
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr int kBarSlots = 24;

template <int D, bool KV8 = false>
struct PCfg {
  static constexpr int kThreads = 32 * (KV8 ? 12 : 10);
  static constexpr int kSlabs = D / 64;
  static constexpr int kRowBlock = kSlabs * 1024;      // one 8-key block of a K/V tile, all slabs
  static constexpr int kQBytes = kSlabs * kSlab;       // one Q tile
  static constexpr int kKVTile = kBN * D * 2;          // K or V tile (128 keys)
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQT * kQBytes;
  static constexpr int kVOff = kKOff + kNSK * kKVTile;
  static constexpr int kPageOff = kVOff + kNSV * kKVTile;  // [8 tiles][32 lanes] page ids seen by the TMA warp
  static constexpr int kBarOff = kPageOff + 8 * 32 * 4;
  static constexpr int kSmem = kBarOff + kBarSlots * 8 + 16 + 1024;  // barriers, TMEM base, alignment slack
  static constexpr uint32_t kTmemCols = 512;           // S_A | S_B | O_A | O_B
  static constexpr uint32_t kSCol = 0;                 // S of query tile t at kSCol + 128 t (P over its first 64)
  static constexpr uint32_t kOCol = 256;               // O of query tile t at kOCol + 128 t
};

// barriers.  K and V stages are filled and freed separately (K(j) is free
// once both S(j) are done, V(j) once both PV(j) are).  S, P and O-done have
// one barrier per query tile.  Every parity waiter stays within one phase of
// its barrier: S_t(j+1) is issued only after PV_t(j), which needs P_t(j).
// B_VLAST completes the copies of a last V tile that the TMA warp still has
// to zero past L before publishing it.
// e4m3 pools: K/V FULL means the codes landed, K/V READY that the converter
// has written the f16 tile (the MMA waits for READY).
enum { B_QFULL = 0, B_KFULL = 1, B_KEMPTY = B_KFULL + kNSK, B_VFULL = B_KEMPTY + kNSK, B_VEMPTY = B_VFULL + kNSV,
       B_SFULL = B_VEMPTY + kNSV, B_PFULL = B_SFULL + kQT, B_ODONE = B_PFULL + kQT, B_VLAST = B_ODONE + kQT,
       B_KREADY = B_VLAST + 1, B_VREADY = B_KREADY + kNSK, B_COUNT = B_VREADY + kNSV };
static_assert(B_COUNT <= kBarSlots, "barrier slots");

// e4m3 pools: one warp turns the codes of a landed tile ([kBN keys][D B] in
// the upper half of its ring slot) into f16 in the UMMA layout over the whole
// slot ([8-key block][slab][8 keys][128 B], 128-byte swizzle), rows at or past
// `valid` set to zero.  The 8-key blocks go in order, four at a time with all
// loads of the four before any store: block k's f16 bytes overlay the codes of
// blocks 2k - 16 and 2k - 15 only, which are converted by then or in the same
// four.
template <int D>
__device__ __forceinline__ void convert_tile_e4m3(unsigned char* slot, int valid, int lane) {
  constexpr int kChunks = D / 16;            // 16-code chunks of one key's row
  constexpr int kKeysPerLoad = 32 / kChunks;  // keys one warp-wide load covers (4 or 8)
  constexpr int kLoads = 8 / kKeysPerLoad;    // loads per lane per 8-key block (2 or 1)
  constexpr int kRowBlock = (D / 64) * 1024;  // bytes of one 8-key block in f16
  const unsigned char* codes = slot + kBN * D;
  // lane -> (key r0 of the load's keys, 16-code chunk m).  D = 128: each
  // quarter-warp takes chunks 0..3 of one key and 4..7 of the key beside it
  // (key rows 8 apart in r0 & 1), so a quarter's 16-byte loads hit 8 bank
  // groups and so do its f16 stores (even and odd chunks XOR key % 8 of two
  // keys of different parity); D = 64: chunk lane % 4 of key lane / 4 does both.
  const int q4 = lane >> 3, j8 = lane & 7;
  const int m = D == 128 ? (j8 & 3) + 4 * (j8 >> 2) : lane % kChunks;
  const int r0 = D == 128 ? 2 * (q4 >> 1) + ((j8 >> 2) ^ (q4 & 1)) : lane / kChunks;
#pragma unroll 1
  for (int k0 = 0; k0 < kBN / 8; k0 += 4) {
    uint4 raw[4][kLoads];
#pragma unroll
    for (int kb = 0; kb < 4; ++kb)
#pragma unroll
      for (int x = 0; x < kLoads; ++x)
        raw[kb][x] = *reinterpret_cast<const uint4*>(codes + ((k0 + kb) * 8 + r0 + x * kKeysPerLoad) * D + m * 16);
    __syncwarp();
#pragma unroll
    for (int kb = 0; kb < 4; ++kb)
#pragma unroll
      for (int x = 0; x < kLoads; ++x) {
        const int key = (k0 + kb) * 8 + r0 + x * kKeysPerLoad, kr = key & 7;
        const uint4 w = raw[kb][x];
        uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;  // dims 16m .. 16m+7 and 16m+8 .. 16m+15
        if (key < valid) {
          lo = make_uint4(e4m3x2_lo_to_f16x2(w.x), e4m3x2_hi_to_f16x2(w.x), e4m3x2_lo_to_f16x2(w.y),
                          e4m3x2_hi_to_f16x2(w.y));
          hi = make_uint4(e4m3x2_lo_to_f16x2(w.z), e4m3x2_hi_to_f16x2(w.z), e4m3x2_lo_to_f16x2(w.w),
                          e4m3x2_hi_to_f16x2(w.w));
        }
        unsigned char* blk = slot + (key >> 3) * kRowBlock + kr * 128;
        const int c0 = 2 * m, c1 = 2 * m + 1;  // 8-dim chunks over D
        *reinterpret_cast<uint4*>(blk + (c0 >> 3) * 1024 + (((c0 & 7) ^ kr) << 4)) = lo;
        *reinterpret_cast<uint4*>(blk + (c1 >> 3) * 1024 + (((c1 & 7) ^ kr) << 4)) = hi;
      }
    __syncwarp();
  }
}

template <int D, bool KV8>
__global__ void __launch_bounds__(PCfg<D, KV8>::kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                      PrefillParams p) {
  using C = PCfg<D, KV8>;
  constexpr int kThreads = C::kThreads;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // shared-prefix pass of cascade decode: one non-causal sequence (the prefix)
  // queried by every decode row; blockIdx.z is then the key chunk
  const bool pre = p.part_o != nullptr;
  const int b = pre ? 0 : blockIdx.z, hk = blockIdx.y;
  const int G = p.group, Hq = p.num_q_heads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qs = pre ? 0 : __ldg(p.query_start_loc + b);
  const int qe = pre ? p.batch_rows : __ldg(p.query_start_loc + b + 1);
  const int n = qe - qs;
  const int ps = p.pool.page_size, pshift = p.pool.page_shift;
  const int max_len = p.max_blocks * ps;
  const int L = pre ? p.prefix_len
                    : seq_keys(p.seq_lens, p.kv_indptr, p.kv_last_page_len, p.kv_len, b, ps, max_len,
                               (tid == 0 && hk == 0 && blockIdx.x == 0) ? p.err : nullptr);
  if (n < 0 || qs < 0 || (int64_t)qe > p.total_q) {
    if (tid == 0 && hk == 0 && blockIdx.x == 0) record_error(p.err, ERR_QUERY_LOC, qs);
    return;
  }
  if (n > p.max_q_len && tid == 0 && hk == 0 && blockIdx.x == 0) record_error(p.err, ERR_QUERY_LOC, n);
  const int rows_total = n * G;
  const int tiles = (rows_total + kQT * kBM - 1) / (kQT * kBM);
  const int tile = gridDim.x - 1 - blockIdx.x;  // heaviest (latest) tiles first
  if (tile >= tiles) return;
  // causal: new token i sits at position first + i; the prefix pass is not
  // causal (every row sees keys 0..L-1, as a row at position L-1 would)
  const int first = L - n;  // absolute position of new token 0
  // per query tile t: rows from row0_t, key tiles [jb, nt_t) with a visible key
  // (nt_t <= jb if the tile has no row)
  int row0_t[kQT], pmin_t[kQT], nt_t[kQT];
#pragma unroll
  for (int t = 0; t < kQT; ++t) {
    row0_t[t] = (tile * kQT + t) * kBM;
    const int last_row = min(row0_t[t] + kBM, rows_total) - 1;
    pmin_t[t] = pre ? L - 1 : first + row0_t[t] / G;
    const int pmax = pre ? L - 1 : first + last_row / G;
    nt_t[t] = (row0_t[t] < rows_total && pmax >= 0) ? pmax / kBN + 1 : 0;
  }
  // the key tiles this CTA covers: all of them, or one chunk in the prefix pass
  const int jb = pre ? (int)blockIdx.z * p.chunk_tiles : 0;
  if (pre) {
#pragma unroll
    for (int t = 0; t < kQT; ++t) nt_t[t] = min(nt_t[t], jb + p.chunk_tiles);
  }
  const int nt = max(nt_t[0], nt_t[1]);  // end (exclusive) of the key tiles the CTA loads

  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out);
  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(p.q);
  auto row_off = [&](int R) {  // packed row -> element offset of its q / out row
    const int i = R / G, g = R - (R / G) * G;
    return ((int64_t)(qs + i) * Hq + (int64_t)hk * G + g) * D;
  };
  griddep_launch_dependents();
  if (nt <= jb) {  // no row of this CTA sees any key (invalid input): zeros
    if (pre) return;  // the launch covers every chunk with keys
    griddep_wait();
    const int r0 = row0_t[0];
    for (int idx = tid; idx < kQT * kBM * D; idx += kThreads) {
      const int R = r0 + idx / D;
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
    mbar_init(bar(B_QFULL), 32 * 8);
    for (int s = 0; s < kNSK; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < kNSV; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int t = 0; t < kQT; ++t) {
      mbar_init(bar(B_SFULL + t), 1);
      mbar_init(bar(B_PFULL + t), 32 * 4);
      mbar_init(bar(B_ODONE + t), 1);
    }
    mbar_init(bar(B_VLAST), 1);
    for (int s = 0; s < kNSK; ++s) mbar_init(bar(B_KREADY + s), 1);
    for (int s = 0; s < kNSV; ++s) mbar_init(bar(B_VREADY + s), 1);
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
    const int kpo = ps < kBN ? ps : kBN;  // keys per box
    const int ops = kBN / kpo;
    const uint32_t box_bytes = (uint32_t)kpo * D * (KV8 ? 1 : 2);
    const int32_t* bt = p.block_table + (pre ? 0 : page_list_start(p.kv_indptr, p.max_blocks, b));
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
        if (KV8)  // codes in the slot's upper half, [keys][D B]
          tma_load_3d(dst + (uint32_t)(kBN * D + lane * kpo * D), map, 0, (int)slot, hk, full);
        else
          tma_load_5d(dst + (uint32_t)(lane * (kpo / 8)) * C::kRowBlock, map, 0, 0, 0, (int)(slot >> 3), hk, full);
      }
    };
    auto slot_free = [&](int i) {  // lane 0 polls, the warp agrees
      int t = 0;
      if (lane == 0) t = mbar_test(bar(i >> 1), (uint32_t)(i & 1)) ? 1 : 0;
      return __shfl_sync(0xffffffffu, t, 0) != 0;
    };
    int jk = jb, jv = jb;  // next K / V tile to issue (absolute); ring slots count from jb
    int raw = fetch(jb);  // block_table is an input, not written by the append kernel
    griddep_wait();      // the pool rows of this step were written by the append kernel
    unsigned long long t_last = global_ns();
    while (jv < nt && alive) {
      bool progressed = false;
      const int jkl = jk - jb, jvl = jv - jb;
      if (jk < nt && (jkl < kNSK || slot_free(((B_KEMPTY + jkl % kNSK) << 1) | (((jkl / kNSK) - 1) & 1)))) {
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
        issue(&tmap_k, k_base + (jkl % kNSK) * C::kKVTile, jk, page, bar(B_KFULL + jkl % kNSK));
        ++jk;
        raw = fetch(jk);
        progressed = true;
      }
      if (jv < jk && (jvl < kNSV || slot_free(((B_VEMPTY + jvl % kNSV) << 1) | (((jvl / kNSV) - 1) & 1)))) {
        const int s = jvl % kNSV;
        const int page = page_ring[(jv & 7) * 32 + lane];
        const uint32_t vdst = v_base + s * C::kKVTile;
        const int valid = L - jv * kBN;  // keys of this tile below L (>= 1)
        if (KV8 || valid >= kBN) {  // (e4m3: the converter zeroes the rows past L)
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


  if (KV8 && (warp == kCvtWarp || warp == kCvtWarp + 1)) {
    // ======================= e4m3 -> f16 converters (K: warp 10, V: warp 11) =======================
    // Each converts its ring's tiles in order, as they land.
    const bool isv = warp == kCvtWarp + 1;
    const int nslots = isv ? kNSV : kNSK;
    for (int j = jb; j < nt && alive; ++j) {
      const int jl = j - jb, valid = min(L - j * kBN, kBN), sl = jl % nslots;
      alive = __all_sync(0xffffffffu,
                         mbar_wait(bar((isv ? B_VFULL : B_KFULL) + sl), (uint32_t)((jl / nslots) & 1), p.err));
      convert_tile_e4m3<D>(smem + (isv ? C::kVOff : C::kKOff) + sl * C::kKVTile, valid, lane);
      fence_proxy_async_smem();  // the f16 tile before the tensor core reads it
      __syncwarp();
      if (lane == 0) mbar_arrive(bar((isv ? B_VREADY : B_KREADY) + sl));
    }
  }

  if (warp == kMmaWarp && lane == 0) {
    // ======================= MMA issuer =======================
    // Fixed order S_A(0) S_B(0), then per key tile j: PV_A(j) S_A(j+1)
    // PV_B(j) S_B(j+1), skipping the key tiles a query tile does not see: the
    // two query tiles alternate on the tensor core, each one's softmax running
    // while the other's products do.  The first S of a key tile waits for K,
    // the first PV for V; the last S (PV) of a key tile frees its K (V) stage.
    constexpr uint32_t idesc_s = KV8 ? umma_idesc_f16(kBM, kBN, false) : umma_idesc_bf16(kBM, kBN, false);
    constexpr uint32_t idesc_o = KV8 ? umma_idesc_f16(kBM, D, true) : umma_idesc_bf16(kBM, D, true);
    constexpr int kKWait = KV8 ? B_KREADY : B_KFULL, kVWait = KV8 ? B_VREADY : B_VFULL;
    // descriptors at the base of each operand; a K step adds its byte offset / 16
    // to the start-address field (every address stays below 256 KB, so no carry)
    const uint64_t q_desc = umma_desc_sw128(smem_u32(q_s), 16, 1024);
    const uint64_t k_desc = umma_desc_sw128(k_base, 16, C::kRowBlock);
    const uint64_t v_desc = umma_desc_sw128(v_base, 1024, C::kRowBlock);
    if (alive) alive = mbar_wait(bar(B_QFULL), 0, p.err);
    const int nt0 = nt_t[0], nt1 = nt_t[1];
    auto issue_s = [&](int t, int j) {
      const int jl = j - jb;
      const int sk = jl % kNSK;
      if (t == 0 || j >= nt0) {  // first S of key tile j
        if (alive) alive = mbar_wait(bar(kKWait + sk), (uint32_t)((jl / kNSK) & 1), p.err);
        tc_fence_after();
      }
      const uint64_t qd = q_desc + (uint64_t)((t * C::kQBytes) >> 4);
      const uint64_t kd = k_desc + (uint64_t)((sk * C::kKVTile) >> 4);
      const uint32_t s_tm = tmem + C::kSCol + t * 128;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)  // S_t = Q_t K^T over 16-dim steps
        umma_bf16(s_tm, qd + (uint64_t)(((kk >> 2) * kSlab + (kk & 3) * 32) >> 4),
                  kd + (uint64_t)(((kk >> 2) * 1024 + (kk & 3) * 32) >> 4), idesc_s, kk > 0);
      umma_commit(bar(B_SFULL + t));
      if (t == 1 || j >= nt1) umma_commit(bar(B_KEMPTY + sk));  // last S of key tile j
    };
    auto issue_pv = [&](int t, int j) {
      const int jl = j - jb;
      const int sv = jl % kNSV;
      if (alive) alive = mbar_wait(bar(B_PFULL + t), (uint32_t)(jl & 1), p.err);
      if (t == 0 || j >= nt0) {  // first PV of key tile j
        if (alive) alive = mbar_wait(bar(kVWait + sv), (uint32_t)((jl / kNSV) & 1), p.err);
      }
      tc_fence_after();
      const uint64_t vd = v_desc + (uint64_t)((sv * C::kKVTile) >> 4);
      const uint32_t s_tm = tmem + C::kSCol + t * 128;
      const uint32_t o_tm = tmem + C::kOCol + t * 128;
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk)  // O_t += P_t V over 16-key steps (two 8-key blocks each)
        umma_bf16_ts(o_tm, s_tm + kk * 8, vd + (uint64_t)((kk * 2 * C::kRowBlock) >> 4), idesc_o,
                     (j > jb || kk > 0) ? 1u : 0u);
      if (j == (t ? nt1 : nt0) - 1) umma_commit(bar(B_ODONE + t));
      if (t == 1 || j >= nt1) umma_commit(bar(B_VEMPTY + sv));  // last PV of key tile j
    };
    if (nt0 > jb) issue_s(0, jb);
    if (nt1 > jb) issue_s(1, jb);
    for (int j = jb; j < nt; ++j) {
      if (j < nt0) issue_pv(0, j);
      if (j + 1 < nt0) issue_s(0, j + 1);
      if (j < nt1) issue_pv(1, j);
      if (j + 1 < nt1) issue_s(1, j + 1);
    }
  }

  if (warp < 4 * kQT) {
    // ======================= softmax: one TMEM lane (row) per thread =======================
    const int t = warp >> 2;                 // query tile
    const int r = tid & (kBM - 1);           // row within the tile == TMEM lane
    const int R = (t ? row0_t[1] : row0_t[0]) + r;
    const bool valid_row = R < rows_total;
    const int ntt = t ? nt_t[1] : nt_t[0];
    const int pmin = t ? pmin_t[1] : pmin_t[0];
    {  // this thread's Q row into the UMMA A layout (K-major, 128-byte swizzle); zeros past the last row
      unsigned char* qt = q_s + t * C::kQBytes;
      const __nv_bfloat16* src = qp + (valid_row ? row_off(R) : 0);
      if (KV8) {  // f16 operands: bf16 -> f16 on the way in
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (valid_row) {
            v = __ldg(reinterpret_cast<const uint4*>(src) + c);
            v = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
          }
          *reinterpret_cast<uint4*>(qt + (c >> 3) * kSlab + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
        }
      } else {
#pragma unroll
        for (int c = 0; c < D / 8; ++c)
          cp_async_16(smem_u32(qt + (c >> 3) * kSlab + r * 128 + (((c & 7) ^ (r & 7)) << 4)), src + c * 8,
                      valid_row ? 16 : 0);
        cp_async_commit();
        cp_async_wait<0>();
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(B_QFULL));
    }
    const int pos = valid_row ? (pre ? L - 1 : first + R / G) : -1;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = lane_base + C::kSCol + t * 128;
    const uint32_t o_col = lane_base + C::kOCol + t * 128;
    float m_ref = -INFINITY, l = 0.f;
    for (int j = jb; j < ntt; ++j) {
      if (alive) alive = mbar_wait(bar(B_SFULL + t), (uint32_t)((j - jb) & 1), p.err);
      tc_fence_after();
      const int key0 = j * kBN;
      const bool diag = key0 + kBN - 1 > pmin;  // some key of the tile lies past some row's position
      const int lim = pos - key0;                    // column c is visible iff c <= lim
      // x = s * scale * log2(e), -inf where masked.  Off the diagonal with a
      // positive scale (the common case) the max is taken over raw S and
      // exp2 takes one fused multiply-add: no mask, no separate scaling.
      const bool plain = !diag && sl2 > 0.f;
      auto scaled = [&](uint32_t raw, int c) {
        const float x = __uint_as_float(raw) * sl2;
        return (!diag || c <= lim) ? x : -INFINITY;
      };
      // pass 1: the row max, 64 columns at a time
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
      if (plain) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[2][32];
          tmem_ld32(s_col + h * 64, v[0]);
          tmem_ld32(s_col + h * 64 + 32, v[1]);
          tmem_wait_ld();
#pragma unroll
          for (int cb = 0; cb < 2; ++cb)
#pragma unroll
            for (int e = 0; e < 32; ++e) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(v[cb][e]));
        }
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[2][32];
          tmem_ld32(s_col + h * 64, v[0]);
          tmem_ld32(s_col + h * 64 + 32, v[1]);
          tmem_wait_ld();
#pragma unroll
          for (int cb = 0; cb < 2; ++cb)
#pragma unroll
            for (int e = 0; e < 32; ++e) mx[e & 7] = fmaxf(mx[e & 7], scaled(v[cb][e], h * 64 + cb * 32 + e));
        }
      }
      float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                         fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      if (plain) tmax *= sl2;
      // reference max: moved only when the row max grows by more than 2^8
      float alpha = 1.f;
      bool rescale = false;
      if (tmax > m_ref + kRescaleThreshold) {
        alpha = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - tmax);
        m_ref = tmax;
        l *= alpha;
        rescale = j > jb;
      }
      const float mbase = m_ref == -INFINITY ? 0.f : m_ref;
      // pass 2: P = exp2(x - m) as bf16 pairs, written over the S columns just read
      float rs[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) rs[i] = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[2][32];
        tmem_ld32(s_col + h * 64, v[0]);
        tmem_ld32(s_col + h * 64 + 32, v[1]);
        tmem_wait_ld();
        uint32_t w[32];
        if (plain) {
#pragma unroll
          for (int cb = 0; cb < 2; ++cb)
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float p0 = fast_exp2(fmaf(__uint_as_float(v[cb][e]), sl2, -mbase));
              const float p1 = fast_exp2(fmaf(__uint_as_float(v[cb][e + 1]), sl2, -mbase));
              rs[(e >> 1) & 7] += p0 + p1;
              w[cb * 16 + (e >> 1)] = KV8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
            }
        } else {
#pragma unroll
          for (int cb = 0; cb < 2; ++cb)
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float p0 = fast_exp2(scaled(v[cb][e], h * 64 + cb * 32 + e) - mbase);
              const float p1 = fast_exp2(scaled(v[cb][e + 1], h * 64 + cb * 32 + e + 1) - mbase);
              rs[(e >> 1) & 7] += p0 + p1;
              w[cb * 16 + (e >> 1)] = KV8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
            }
        }
        tmem_st32(s_col + h * 32, w);
      }
      l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      // O is rescaled in place only when some row of the warp moved its
      // reference max.  PV_t(j-1) is complete: S_t(j) was issued after it.
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t o[32];
          tmem_ld32(o_col + cb * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(o_col + cb * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + t));
    }
    // ---- epilogue: O / l -> bf16 (zeros for a tile that sees no key) ----
    const bool has = ntt > jb;
    if (has) {
      if (alive) alive = mbar_wait(bar(B_ODONE + t), 0, p.err);
      tc_fence_after();
    }
    griddep_wait();  // before the first global write
    if (pre && has) {
      // unnormalised partial of this key chunk: O and (reference max, l); the
      // whole warp takes part in each tcgen05.ld, valid rows store
      const int64_t pr =
          valid_row ? ((int64_t)blockIdx.z * n + R / G) * Hq + (int64_t)hk * G + (R - (R / G) * G) : 0;
      float* po = p.part_o + pr * D;
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t o[32];
        tmem_ld32(o_col + cb * 32, o);
        tmem_wait_ld();
        if (valid_row) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(po + cb * 32 + q * 4) =
                make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
      }
      if (valid_row) p.part_ml[pr] = make_float2(m_ref, l);
    }
    const float inv = l > 0.f ? p.v_scale / l : 0.f;  // v_scale: 1 for bf16 pools
    __nv_bfloat16* orow = outp + (valid_row ? row_off(R) : 0);
#pragma unroll
    for (int cb = 0; cb < D / 32 && !pre; ++cb) {
      uint32_t o[32];
      if (has) {
        tmem_ld32(o_col + cb * 32, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
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

template <int D, bool KV8>
cudaError_t launch_prefill_tc(const PrefillParams& p, cudaStream_t s) {
  using C = PCfg<D, KV8>;
  const int ps = p.pool.page_size;
  if (ps < 8 || p.pool.page_shift < 0) return cudaErrorInvalidValue;
  if (KV8 && p.part_o != nullptr) return cudaErrorInvalidValue;  // the cascade prefix pass: bf16 pools
  const int kpo = ps < kBN ? ps : kBN;  // keys per TMA box
  const int64_t rows = p.pool.num_pages * (int64_t)ps;
  CUtensorMap tk, tv;
  if (KV8) {
    if (!encode_pool_tmap_u8(&tk, p.pool.key_pool, rows, p.pool.num_kv_heads, D, kpo, 1, false) ||
        !encode_pool_tmap_u8(&tv, p.pool.value_pool, rows, p.pool.num_kv_heads, D, kpo, 1, false))
      return cudaErrorInvalidValue;
  } else if (!encode_pool_tmap_blocked(&tk, p.pool.key_pool, rows, p.pool.num_kv_heads, D, kpo / 8) ||
             !encode_pool_tmap_blocked(&tv, p.pool.value_pool, rows, p.pool.num_kv_heads, D, kpo / 8)) {
    return cudaErrorInvalidValue;
  }
  auto kern = prefill_tc_kernel<D, KV8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = ((int64_t)p.max_q_len * p.group + kQT * kBM - 1) / (kQT * kBM);
  unsigned gz = (unsigned)p.batch;
  if (p.part_o != nullptr) {  // prefix pass of cascade decode: z = key chunk
    if (p.chunk_tiles <= 0 || p.prefix_len <= 0) return cudaErrorInvalidValue;
    const int nt = (p.prefix_len + kBN - 1) / kBN;
    gz = (unsigned)((nt + p.chunk_tiles - 1) / p.chunk_tiles);
  }
  return launch_pdl(kern, dim3((unsigned)tiles, (unsigned)p.pool.num_kv_heads, gz), dim3(C::kThreads),
                    (size_t)C::kSmem, s, tk, tv, p);
}

}  // namespace

cudaError_t launch_prefill_bf16(const PrefillParams& p, cudaStream_t s) {
  if (p.max_q_len <= 0 || p.batch <= 0) return cudaSuccess;
  if (p.kv8) return p.pool.head_dim == 128 ? launch_prefill_tc<128, true>(p, s) : launch_prefill_tc<64, true>(p, s);
  return p.pool.head_dim == 128 ? launch_prefill_tc<128, false>(p, s) : launch_prefill_tc<64, false>(p, s);
}

}  // namespace pa
