// The split-KV decode kernel of paged_attention_decode (bf16 and e4m3 pools),
// templated on the shape (head_dim, heads per box, row tiles), the pool
// element type and FUSED (paged_attention_decode_append: the kernel also
// writes the step's new K/V rows and attends to them from its input) and WC
// (the weighted cut below for 16-row groups).  The plain instantiations are
// compiled in decode_bf16.cu, the fused ones in decode_fused.cu, the WC ones in
// decode_weighted.cu, so a plain decode carries none of the fused code.
//
// What is computed (onnxruntime/mobius PR #395 "Add paged / block-table KV
// cache export", "How it works": Gather(pool, block_table) then Attention
// masked to nonpad_kv_seqlen; decode is the one-query-token case):
//   out[b, h] = softmax_j(scale * q[b,h] . K_b[j, h/G]) V_b[j, h/G],  j < L_b
//
// Work decomposition (GB300-first, not from the pages):
// * The unit of work is one 16-key block of one sequence for a box of HB KV
//   heads (HB = the largest power of two <= 8 dividing num_kv_heads; 1 for
//   page_size 8).  All units are laid out sequence-major and cut into
//   `num_ctas` equal contiguous ranges, one persistent CTA per SM, so every
//   CTA streams the same number of KV bytes whatever the context-length mix.
//   For 32-row groups, where a segment change costs a CTA ~5 us, each segment
//   also weighs seg_penalty blocks in the cut, and a publisher warp counts the
//   CTA's cut segments off the consumer path; the WC instantiations do the same
//   for 16-row groups of long sequences (each cut across several CTAs).
// * Two producer warps (even and odd stages) follow block_table and load each
//   stage (NBS blocks x HB heads of K and V) with TMA tensor copies through a
//   4-D view of the pool {64 dims, slots, kv_heads, slabs}: one box
//   {64, 16, HB, D/64} lands as HB tiles of 16 rows x 128 B per slab with the
//   128-byte swizzle.  For 8 KV heads a box is a 32 KB slice of one page.
//   Measured on GB300 (random pages streamed into a shared ring, one CTA per
//   SM): 32 KB boxes reach 7.2 TB/s and 4 KB boxes 7.0 TB/s when the 32 lanes
//   of a warp issue them, one issuing thread only 2.9 TB/s; so the producer
//   lanes issue a stage's boxes together.  A third warp bulk-copies, per
//   segment, the query rows.
// * Eight consumer warps map to (head in box, block in stage, row tile of 16
//   query heads): S = Q K^T and O += P V with mma.sync m16n8k16 (bf16 in,
//   fp32 accumulate), online softmax in the log2 domain, output rescale
//   skipped when no running max moved.  Each page is read from HBM once for
//   all G query heads of its KV head (GQA/MQA reuse).  Every consumer waits
//   on every stage in order, so no mbarrier parity wait can run a phase ahead.
// * e4m3 pools (KV8): a box brings D code bytes per row (128- or 64-byte
//   swizzle); ldmatrix reads the codes as 16-bit pairs and cvt turns them into
//   the f16 B fragments of mma.sync m16n8k16 f16 (Q's dims and the output
//   columns are permuted to match); k_scale is folded into the softmax scale,
//   v_scale into the final normalisation.
// * Keys at or past L_b are masked in S and their V rows are zeroed in shared
//   memory, so stale or NaN-poisoned slots never reach the output.
// * At a segment (sequence x head box) end, warps that shared a head merge in
//   shared memory; a segment covering the whole sequence writes bf16 output,
//   a segment cut by a range boundary leaves one fp32 partial (m, l, o) per
//   CTA.  Parts are counted in workspace words tagged with a per-launch epoch;
//   after its range every CTA holding a part waits until all are counted and
//   merges a slice of the segment's rows (the grid is launched cooperatively,
//   so all CTAs are resident; without that launch the CTA counting the last
//   part merges the whole segment), with
//   o = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i.
//   Cascade decode instead leaves every segment's partials to the combine
//   kernel in decode_bf16.cu.
// * The kernel uses programmatic stream serialization: its prologue runs
//   while the preceding kernel (the append) finishes.  Every access to data
//   an earlier kernel may write comes after griddepcontrol.wait.
#pragma once
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace pa {

namespace {

// keys of sequence b (either page-table form), with / without recording bad input
__device__ __forceinline__ int nblk_of(const DecodeParams& p, int b, int max_len) {
  return (seq_keys(p.seq_lens, p.kv_indptr, p.kv_last_page_len, p.kv_len, b, p.pool.page_size, max_len, p.err) + 15) >> 4;
}

__device__ __forceinline__ int seq_len_of(const DecodeParams& p, int b, int max_len) {
  return seq_keys(p.seq_lens, p.kv_indptr, p.kv_last_page_len, p.kv_len, b, p.pool.page_size, max_len, nullptr);
}

// CTA that owns unit u when U units are cut into n ranges [c*U/n, (c+1)*U/n)
// (the same for a position of the weighted cut below, with W positions).
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

// Count one more arrival on a counter word holding (tag << 16) | arrivals in
// this launch; a word with another tag (an earlier launch's, or uninitialised
// memory) counts as 0.  Returns the arrivals before this one.  Once the word
// carries this launch's tag an arrival is one atomicAdd; only a stale word
// takes a compare-and-swap, which exactly one arrival wins (a loser re-reads
// and adds), so each arrival makes at most three atomic operations.  The
// bound only guards against a broken counter (then a bounded-wait error is
// recorded and the caller acts as a non-last arrival).
__device__ __forceinline__ unsigned arrive_part(unsigned long long* cnt, unsigned long long tag,
                                                unsigned long long* err) {
  unsigned long long w = *reinterpret_cast<volatile unsigned long long*>(cnt);
  for (int it = 0; it < 8; ++it) {
    if ((w >> 16) == tag) {
      if ((w & 0xFFFFu) == 0xFFFFu) break;  // a full count field: not a live counter
      const unsigned long long old = atomicAdd(cnt, 1ull);
      if ((old >> 16) == tag && (old & 0xFFFFu) != 0xFFFFu) return (unsigned)(old & 0xFFFFu);
      break;
    }
    const unsigned long long got = atomicCAS(cnt, w, (tag << 16) | 1ull);
    if (got == w) return 0u;
    w = got;
  }
  record_error(err, ERR_TIMEOUT, -1);
  return 0xFFFFFFFFu;
}

// Acquire-release fence at GPU scope (lighter than the sequentially
// consistent fence of __threadfence; release and acquire patterns need no more).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;\n" ::: "memory"); }

// Load with acquire semantics at GPU scope: later reads of this thread (and,
// through a barrier, of its CTA) see what was published before the value.
__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* ptr) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(ptr) : "memory");
  return v;
}

// One warp merges query row (head h of the box, row g) of segment `seg`, cut
// into parts by CTAs c0 .. c0 + nparts - 1 (a CTA that owns no unit, only
// possible when U < n, wrote nothing and weighs 0), and writes the bf16
// result to outrow: o = v_scale * sum_q 2^(m_q - M) o_q / sum_q 2^(m_q - M) l_q.
// Lane q holds part q's (m, l); each lane accumulates 4 dims.  The first 8
// parts' rows are loaded together with the (m, l) (one round trip), later
// parts one by one.
__device__ __noinline__ void merge_segment_row(const DecodeParams& p, int64_t seg, int HB, int G, int h, int g,
                                               int c0, int nparts, int64_t U, int n, int D,
                                               __nv_bfloat16* outrow) {
  const int lane = threadIdx.x & 31;
  const bool some_empty = U < n;
  const bool dims = 4 * lane < D;
  auto absent = [&](int q) { return some_empty && cta_range_empty(c0 + q, U, n); };
  auto row = [&](int q) {
    return __ldcg(reinterpret_cast<const float4*>(p.part_o + (((seg + c0 + q) * HB + h) * G + g) * D) + lane);
  };
  auto ml_of = [&](int q) {
    return absent(q) ? make_float2(-INFINITY, 0.f) : __ldcg(p.part_ml + ((seg + c0 + q) * HB + h) * G + g);
  };
  constexpr int kRegParts = 8;
  float4 vr[kRegParts];
#pragma unroll
  for (int q = 0; q < kRegParts; ++q)
    vr[q] = (q < nparts && dims && !absent(q)) ? row(q) : make_float4(0.f, 0.f, 0.f, 0.f);
  const float2 ml_mine = lane < nparts ? ml_of(lane) : make_float2(-INFINITY, 0.f);
  float M = ml_mine.x;
  for (int q = lane + 32; q < nparts; q += 32) M = fmaxf(M, ml_of(q).x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float f_mine = (ml_mine.x == -INFINITY) ? 0.f : fast_exp2(ml_mine.x - M);
  float den = f_mine * ml_mine.y;
  for (int q = lane + 32; q < nparts; q += 32) {
    const float2 ml = ml_of(q);
    den += (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M) * ml.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const float inv = den > 0.f ? p.v_scale / den : 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int q = 0; q < kRegParts; ++q) {
    const float f = __shfl_sync(0xffffffffu, f_mine, q);
    acc.x += f * vr[q].x; acc.y += f * vr[q].y; acc.z += f * vr[q].z; acc.w += f * vr[q].w;
  }
  for (int q = kRegParts; q < nparts; ++q) {
    float f = __shfl_sync(0xffffffffu, f_mine, q & 31);
    if (q >= 32) {
      const float2 ml = ml_of(q);
      f = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
    }
    if (f != 0.f && dims) {
      const float4 v = row(q);
      acc.x += f * v.x; acc.y += f * v.y; acc.z += f * v.z; acc.w += f * v.w;
    }
  }
  if (dims) {
    uint2 packed;
    packed.x = pack_bf16(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(outrow + 4 * lane) = packed;
  }
}

// The consumer threads (nthreads, ids tid) merge every query row of segment
// (b, head box hkb), cut into parts by CTAs c0 .. c0 + span - 1, into the bf16
// output.  A part's partials are contiguous ([HB*G rows][D] fp32 and
// [HB*G] (m, l)), so each part is copied whole into shared memory (the idle
// stage ring, `scratch`) with 16-byte cp.async -- one round trip for all
// parts -- and every thread then merges 4 dims of a row:
//   o = v_scale * sum_q 2^(m_q - M) o_q / sum_q 2^(m_q - M) l_q.
// Parts that do not fit in the ring are merged warp by warp from global memory.
template <int D>
__device__ __noinline__ void merge_segment(const DecodeParams& p, int b, int hkb, int c0, int span, int HB, int Hg,
                                           int64_t U, int n, int row_lo, int row_hi, unsigned char* scratch,
                                           int scratch_bytes, int tid, int nthreads, int bar_id) {
  const int G = p.group;
  const int all_rows = HB * G;  // a part's rows (h, g), contiguous
  const int rows = row_hi - row_lo;  // the rows merged here
  if (rows <= 0) return;
  const int64_t seg = (int64_t)b * Hg + hkb;
  const int64_t Hq = p.num_q_heads;
  __nv_bfloat16* out =
      static_cast<__nv_bfloat16*>(p.out) + ((int64_t)b * Hq + (int64_t)hkb * HB * G + row_lo) * D;
  const int o_bytes = rows * D * 4;
  if ((int64_t)span * (o_bytes + rows * 8) > scratch_bytes) {
    const int warp = tid >> 5;
    for (int t = warp; t < rows; t += nthreads / 32) {
      const int r = row_lo + t;
      merge_segment_row(p, seg, HB, G, r / G, r - (r / G) * G, c0, span, U, n, D, out + (int64_t)t * D);
    }
    return;
  }
  float* so = reinterpret_cast<float*>(scratch);                            // [span][rows][D]
  float2* sml = reinterpret_cast<float2*>(scratch + (size_t)span * o_bytes);  // [span][rows]
  const bool some_empty = U < n;
  // flat loops over (part, chunk) and (part, row): every copy and load of a
  // thread is independent, so all are in flight at once
  const int chunks = o_bytes / 16;  // 16-byte chunks of one part's rows
  const uint32_t so_u32 = smem_u32(so);
  for (int i = tid; i < span * chunks; i += nthreads) {
    const int q = i / chunks, k = i - q * chunks;
    if (some_empty && cta_range_empty(c0 + q, U, n)) continue;
    cp_async_16(so_u32 + (uint32_t)i * 16u, p.part_o + ((seg + c0 + q) * all_rows + row_lo) * D + 4 * k, 16);
  }
#pragma unroll 4
  for (int i = tid; i < span * rows; i += nthreads) {
    const int q = i / rows, r = i - q * rows;
    sml[i] = (some_empty && cta_range_empty(c0 + q, U, n)) ? make_float2(-INFINITY, 0.f)
                                                          : __ldcg(p.part_ml + (seg + c0 + q) * all_rows + row_lo + r);
  }
  cp_async_commit();
  cp_async_wait<0>();
  named_barrier(bar_id, nthreads);
  for (int x = tid; x < rows * (D / 4); x += nthreads) {
    const int r = x / (D / 4), c4 = x - r * (D / 4);
    float M = -INFINITY;
    for (int q = 0; q < span; ++q) M = fmaxf(M, sml[q * rows + r].x);
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < span; ++q) {
      const float2 ml = sml[q * rows + r];
      if (ml.x == -INFINITY) continue;
      const float f = fast_exp2(ml.x - M);
      const float4 v = reinterpret_cast<const float4*>(so + ((size_t)q * rows + r) * D)[c4];
      den += f * ml.y;
      acc.x += f * v.x; acc.y += f * v.y; acc.z += f * v.z; acc.w += f * v.w;
    }
    const float inv = den > 0.f ? p.v_scale / den : 0.f;
    uint2 packed;
    packed.x = pack_bf16(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(out + (int64_t)r * D + 4 * c4) = packed;
  }
}

// Compile-time shape of one configuration: HB heads per box, RT row tiles,
// WC the weighted cut and publisher warp for 16-row groups.
template <int D, int HB, int RT, bool KV8 = false, bool WC = false>
struct Cfg {
  static constexpr int kConsumers = 8;
  // 16-key blocks a consumer warp takes per stage: two for 32-row groups, so
  // each of those warps (latency-bound, one per row tile) carries twice the
  // keys through one softmax step and has independent MMA chains to overlap
  static constexpr int BPW = RT;
  static constexpr int NBS = kConsumers * BPW / (HB * RT);  // blocks per stage
  static constexpr int NW = NBS / BPW;                      // consumer warps per (head, row tile)
  static constexpr int kKvProducers = 2;                  // KV producer warps, alternating stages
  // 32-row groups: a segment change costs a CTA ~5 us (the NW warps' chained
  // merge, the part's write and count), so the cut of the units weighs
  // segment changes (seg_penalty) and a publisher warp does each cut
  // segment's fence and count off the consumer path; with WC, 16-row groups
  // whose sequences each span several CTAs too (the CTAs holding two cut
  // segments, two counts and two merges, set the call's time)
  static constexpr bool kCostlyChange = RT == 2 || WC;
  // + the Q producer warp (+ the publisher warp)
  static constexpr int kThreads = 32 * (kConsumers + kKvProducers + 1 + (kCostlyChange ? 1 : 0));
  static constexpr int kBars = kCostlyChange ? 7 : 4;  // mbarriers after the ring's two per stage
  // bf16 pools land as 128-byte-swizzled slabs of 64 dims; e4m3 pools land a
  // whole row of D codes per slot, swizzled over its D bytes (see sw_e4m3)
  static constexpr int kSlabs = KV8 ? 1 : D / 64;          // TMA slabs per row
  static constexpr int kRowBytes = KV8 ? D : 128;         // bytes of one slot row of one slab
  static constexpr int kHeadTile = 16 * kRowBytes;        // one head, 16 rows, one slab
  static constexpr int kBoxBytes = HB * kHeadTile;        // one {row, 16, HB} box
  static constexpr int kTensorBytes = NBS * kSlabs * kBoxBytes;
  static constexpr int kStageBytes = 2 * kTensorBytes;    // K then V
};

// Most ring stages a CTA keeps (small e4m3 / MQA stages reach it).
constexpr int kMaxStages = 12;

// Byte offset of 16-byte chunk `chunk` of row `row` in one head's e4m3 tile
// ([16 rows][D B]) as TMA lands it: the 128-byte swizzle (D = 128: chunk XOR
// row % 8) or the 64-byte one (D = 64: chunk XOR (row / 2) % 4).  Eight rows
// of one chunk then sit in eight distinct bank groups.
template <int D>
__device__ __forceinline__ uint32_t sw_e4m3(int row, int chunk) {
  if (D == 128) return row * 128 + ((chunk ^ (row & 7)) << 4);
  return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
}

// Runtime shared-memory layout (stage count depends on G and B).
struct Layout {
  int stages, qslot, bar_off, mrg_off, prefix_off, total;
};

template <int D, int HB, int RT, bool KV8 = false, bool WC = false>
__host__ __device__ inline Layout make_layout(int G, int B, int budget) {
  using C = Cfg<D, HB, RT, KV8, WC>;
  Layout L;
  L.qslot = ((HB * G * D * 2) + 127) / 128 * 128;
  const int merge = C::NW > 1 ? HB * G * (D + 2) * 4 : 0;  // one slot: the chained merge below
  const int prefix = ((B + 1) * 4 + 127) / 128 * 128;
  const int fixed = 2 * L.qslot + (2 * kMaxStages + C::kBars) * 8 + 128 + merge + prefix + 128 + 1024;
  int s = (budget - fixed) / C::kStageBytes;
  if (s > kMaxStages) s = kMaxStages;
  L.stages = s;
  L.bar_off = s * C::kStageBytes + 2 * L.qslot;
  L.mrg_off = L.bar_off + (2 * s + C::kBars) * 8 + 128;  // + the pending-merge list
  L.prefix_off = L.mrg_off + merge;
  L.total = L.prefix_off + prefix + 1024;
  return L;
}

template <int D, int HB, int RT, bool KV8, bool FUSED, bool WC = false>
__global__ void __launch_bounds__(Cfg<D, HB, RT, KV8, WC>::kThreads, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                        DecodeParams p) {
  using C = Cfg<D, HB, RT, KV8, WC>;
  constexpr int NBS = C::NBS, BPW = C::BPW, NW = C::NW;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int G = p.group;
  const int B = p.batch;
  const int Hkv = p.pool.num_kv_heads;
  const int Hg = Hkv / HB;  // head boxes per sequence
  const int Hq = p.num_q_heads;
  const Layout lay = make_layout<D, HB, RT, KV8, WC>(G, B, p.smem_budget);
  const int S = lay.stages;
  unsigned char* ring = smem;
  unsigned char* qring = smem + S * C::kStageBytes;
  const uint32_t bars = smem_u32(smem + lay.bar_off);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto qfull_bar = [&](int s) { return bars + 8u * (2 * S + s); };
  auto qempty_bar = [&](int s) { return bars + 8u * (2 * S + 2 + s); };
  // (kCostlyChange) cut segment e (0, 1) of this range: its partial is
  // written (consumers -> publisher); every cut segment is published
  // (publisher -> consumers)
  auto pub_bar = [&](int e) { return bars + 8u * (2 * S + 4 + e); };
  const uint32_t pubd_bar = bars + 8u * (2 * S + 6);
  float* mrg_o = reinterpret_cast<float*>(smem + lay.mrg_off);       // [HB][G][D]
  float* mrg_ml = mrg_o + HB * G * D;                                 // [HB][G][2]
  int* prefix = reinterpret_cast<int*>(smem + lay.prefix_off);        // [B+1] 16-key blocks before b
  // segments this CTA merges (some of) after its range: [0] = count, then
  // kPend ints each (b, head box, c0, span, parts, this CTA's part index);
  // bytes 96..103 hold this launch's counter tag
  constexpr int kPend = 6;
  volatile int* pending = reinterpret_cast<volatile int*>(smem + lay.bar_off + (2 * S + C::kBars) * 8);  // [24]
  volatile unsigned long long* tag_slot = reinterpret_cast<volatile unsigned long long*>(pending + 24);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ps = p.pool.page_size, pshift = p.pool.page_shift;
  const int max_len = p.max_blocks * ps;

  // ---- set-up: barriers and the per-sequence block prefix (reads seq_lens only) ----
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), C::kConsumers);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(qfull_bar(s), 1);
      mbar_init(qempty_bar(s), C::kConsumers);
    }
    if constexpr (C::kCostlyChange) {
      mbar_init(pub_bar(0), 1);
      mbar_init(pub_bar(1), 1);
      mbar_init(pubd_bar, 1);
    }
    fence_mbar_init();
  }
  const int n = p.num_ctas, c = blockIdx.x;
  // Units: (b, head box hg, 16-key block k), sequence-major, cut into one
  // range per CTA.  Plainly, the U units in n equal ranges.  With
  // kCostlyChange they are laid out on a line of positions on which each
  // segment (sequence x head box with keys) takes P header positions and then
  // one per block (P = seg_penalty: a segment change's time in blocks), the W
  // positions are cut into n equal ranges and a CTA takes the units whose
  // positions fall in its range, so CTAs whose ranges hold more segment
  // changes get fewer blocks.  Every range is kept longer than a header (else
  // P = 0), so with P > 0 every CTA owns a unit.  prefix[b] counts the
  // positions (blocks, plus P per segment) before sequence b.
  int P = 0;
  for (int pass = 0; pass < 2; ++pass) {
    if constexpr (C::kCostlyChange) {
      if (pass == 0) P = p.seg_penalty;
      else __syncthreads();  // every thread has read the first pass's total
    }
    for (int b = tid; b < B; b += C::kThreads) {
      const int nb = nblk_of(p, b, max_len);
      prefix[b + 1] = C::kCostlyChange && nb > 0 ? nb + P : nb;
    }
    if (tid == 0) prefix[0] = 0;
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
    if (!C::kCostlyChange || P == 0 || (int64_t)prefix[B] * Hg >= (int64_t)n * (P + 1)) break;
    P = 0;
  }
  const int64_t W = (int64_t)prefix[B] * Hg;  // positions (units when P = 0)
  const int64_t u0 = (int64_t)c * W / n, u1 = (int64_t)(c + 1) * W / n;
  griddep_launch_dependents();
  // Counter tag of this launch, kept by thread 0 (the only thread that counts
  // arrivals) in shared memory: read the epoch E, then count this CTA on the grid counter; the
  // n-th CTA (every CTA has read E by then) stores E + 1.  The tag is the top
  // 48 bits of (E + 1) times an odd constant (the 64-bit golden-ratio
  // multiplier), so memory filled with a repeated byte or word does not read
  // as a matching tag, and E and E + 1 give different tags.
  if (warp < C::kConsumers) {
    griddep_wait();  // before any output write, and before the epoch is read
    if (tid == 0) {
      pending[0] = 0;
      const unsigned long long e = *reinterpret_cast<volatile unsigned long long*>(p.launch_epoch);
      const unsigned long long tag = ((e + 1) * 0x9E3779B97F4A7C15ull) >> 16;
      *tag_slot = tag;
      __threadfence();
      if (arrive_part(p.launch_epoch + 1, tag, p.err) == (unsigned)(n - 1))
        *reinterpret_cast<volatile unsigned long long*>(p.launch_epoch) = e + 1;
    }
  }
  if (FUSED && warp < C::kConsumers) {
    // fused append: CTA c writes the new rows of tokens c, c + n, ... into the
    // pool.  No CTA of this launch reads them back from the pool: each
    // sequence's new row reaches its attention from the input (below).
    const int64_t num_slots = p.pool.num_pages * (int64_t)ps;
    const int row_elems = Hkv * D;  // one slot: contiguous in the input and the pool
    for (int b = c; b < B; b += n) {
      const int64_t slot = __ldg(p.new_slots + b);
      if (slot < 0) continue;  // no new token for sequence b
      if (slot >= num_slots) {
        if (tid == 0) record_error(p.err, ERR_SLOT, slot);
        continue;
      }
      if (tid == 0) {  // the new token must be b's last key: position seq_lens[b] - 1
        const int L = seq_len_of(p, b, max_len);
        const int32_t* bt = p.block_table + page_list_start(p.kv_indptr, p.max_blocks, b);
        if (L < 1 || (int64_t)__ldg(bt + ((L - 1) >> pshift)) * ps + ((L - 1) & (ps - 1)) != slot)
          record_error(p.err, ERR_SLOT, slot);
      }
      const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.new_k) + (int64_t)b * row_elems);
      const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.new_v) + (int64_t)b * row_elems);
      if (KV8) {
        uint2* kd = reinterpret_cast<uint2*>(static_cast<unsigned char*>(const_cast<void*>(p.pool.key_pool)) + slot * row_elems);
        uint2* vd = reinterpret_cast<uint2*>(static_cast<unsigned char*>(const_cast<void*>(p.pool.value_pool)) + slot * row_elems);
        for (int i = tid; i < row_elems / 8; i += C::kConsumers * 32) {
          kd[i] = quantize8(__ldg(ks + i), p.k_quant);
          vd[i] = quantize8(__ldg(vs + i), p.v_quant);
        }
      } else {
        uint4* kd = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(const_cast<void*>(p.pool.key_pool)) + slot * row_elems);
        uint4* vd = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(const_cast<void*>(p.pool.value_pool)) + slot * row_elems);
        for (int i = tid; i < row_elems / 8; i += C::kConsumers * 32) {
          kd[i] = __ldg(ks + i);
          vd[i] = __ldg(vs + i);
        }
      }
    }
  }
  // sequences with no key (seq_len 0) get out = 0; CTA b % n writes them
  for (int b = c; b < B; b += n) {
    if (prefix[b + 1] != prefix[b]) continue;
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.out) + (int64_t)b * Hq * D;
    if (warp < C::kConsumers)
      for (int idx = tid; idx < Hq * D; idx += C::kConsumers * 32) ob[idx] = __float2bfloat16_rn(0.f);
  }
  if (u0 >= u1) return;

  // the first unit at position u or after it (u in a header: the segment's
  // first unit); cur.u is the unit's position
  auto locate = [&](int64_t u) {
    Cursor cur;
    const int x = (int)(u / Hg);
    int lo = 0, hi = B;  // largest b in [0, B) with prefix[b] <= x
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= x) lo = mid; else hi = mid;
    }
    cur.b = lo;
    const int r = (int)(u - (int64_t)Hg * prefix[lo]);
    if constexpr (C::kCostlyChange) {
      const int seg = prefix[lo + 1] - prefix[lo];  // positions of one head box's segment
      cur.nblk = seg - P;
      cur.hk = r / seg;
      const int off = r - cur.hk * seg;
      cur.k = off >= P ? off - P : 0;
      cur.u = (int64_t)Hg * prefix[lo] + (int64_t)cur.hk * seg + P + cur.k;
    } else {
      cur.nblk = prefix[lo + 1] - prefix[lo];
      cur.hk = r / cur.nblk;  // head box index
      cur.k = r - cur.hk * cur.nblk;
      cur.u = u;
    }
    cur.L = seq_len_of(p, cur.b, max_len);
    return cur;
  };
  auto advance = [&](Cursor& cur, int nb) {
    cur.u += nb;
    cur.k += nb;
    if (cur.k == cur.nblk) {
      cur.k = 0;
      if constexpr (C::kCostlyChange) cur.u += P;  // the next segment's header
      if (++cur.hk == Hg) {
        cur.hk = 0;
        do { ++cur.b; } while (cur.b < B && prefix[cur.b + 1] == prefix[cur.b]);
        if (cur.b < B) {
          cur.nblk = prefix[cur.b + 1] - prefix[cur.b] - (C::kCostlyChange ? P : 0);
          cur.L = seq_len_of(p, cur.b, max_len);
        }
      }
    }
  };
  // blocks in the stage that starts at cur (a stage never crosses a segment)
  auto stage_blocks = [&](const Cursor& cur) {
    int64_t nb = cur.nblk - cur.k;
    if (nb > NBS) nb = NBS;
    if (nb > u1 - cur.u) nb = u1 - cur.u;
    return (int)nb;
  };

  const __nv_bfloat16* qglob = static_cast<const __nv_bfloat16*>(p.q);

  if (warp == C::kConsumers + C::kKvProducers) {
    // ======================= Q producer =======================
    // Segment by segment, in order, the HB*G query rows of the head box go to a
    // 2-slot ring (in-order issue keeps each parity wait one phase ahead at most).
    if (lane != 0) return;
    Cursor cur = locate(u0);
    bool alive = true;
    griddep_wait();
    for (int seg = 0; cur.u < u1; ++seg) {
      const int qs = seg & 1;
      if (seg >= 2 && alive) alive = mbar_wait(qempty_bar(qs), ((seg >> 1) - 1) & 1, p.err);
      const uint32_t qbytes = (uint32_t)(HB * G * D * 2);
      mbar_arrive_expect_tx(qfull_bar(qs), qbytes);
      bulk_load(smem_u32(qring + qs * lay.qslot), qglob + ((int64_t)cur.b * Hq + (int64_t)cur.hk * HB * G) * D,
                qbytes, qfull_bar(qs));
      advance(cur, (int)min((int64_t)(cur.nblk - cur.k), u1 - cur.u));
    }
    return;
  }

  if constexpr (C::kCostlyChange) {
    if (warp == C::kConsumers + C::kKvProducers + 1) {
      // ======================= part publisher =======================
      // For each segment of this range cut across CTAs (plain decode: a range
      // cuts at most two, its first and its last), wait until the consumers
      // have written this CTA's partial of it, then publish it: a GPU-scope
      // release fence (cumulative over the consumers' writes, which the
      // mbarrier's release/acquire orders before it) and a count on the
      // segment's counter; note the merge this CTA then takes part in.  Done
      // here, the fence's wait for the partial writes and the counter's round
      // trip hold up no consumer warp, so no stage of the ring is freed late.
      if (lane != 0) return;
      if (p.pre_chunks == 0) {
        Cursor cur = locate(u0);
        bool alive = true;
        for (int e = 0; cur.u < u1;) {
          const int seg_blocks = (int)min((int64_t)(cur.nblk - cur.k), u1 - cur.u);
          if (!(cur.k == 0 && seg_blocks == cur.nblk)) {
            if (alive) alive = mbar_wait(pub_bar(e), 0, p.err);
            const int64_t seg_id = (int64_t)cur.b * Hg + cur.hk;
            // positions of the segment's first and last units
            const int64_t us = (int64_t)Hg * prefix[cur.b] + (int64_t)cur.hk * (cur.nblk + P) + P;
            const int c0 = cta_of_unit(us, W, n), c1 = cta_of_unit(us + cur.nblk - 1, W, n);
            int arrivals = c1 - c0 + 1, mine = c - c0;  // CTAs c0 .. c1 own the segment's units ...
            if (W < n) {  // ... except those without a unit, which took no part (only when P = 0)
              arrivals = mine = 0;
              for (int x = c0; x <= c1; ++x) {
                const int part = cta_range_empty(x, W, n) ? 0 : 1;
                arrivals += part;
                if (x < c) mine += part;
              }
            }
            fence_acq_rel_gpu();  // release: the partials, then the count
            const bool last = arrive_part(p.seg_count + seg_id, *tag_slot, p.err) == (unsigned)(arrivals - 1);
            if (p.slice_merge || last) {
              const int pe = pending[0];
              volatile int* ent = pending + 1 + kPend * pe;
              ent[0] = cur.b;
              ent[1] = cur.hk;
              ent[2] = c0;
              ent[3] = c1 - c0 + 1;  // the merge walks the CTA span (empty CTAs weigh 0)
              ent[4] = p.slice_merge ? arrivals + p.test_extra_parts : 1;
              ent[5] = p.slice_merge ? mine : 0;
              pending[0] = pe + 1;
            }
            ++e;
          }
          advance(cur, seg_blocks);
        }
      }
      mbar_arrive(pubd_bar);
      return;
    }
  }

  if (warp >= C::kConsumers && warp < C::kConsumers + C::kKvProducers) {
    // ======================= KV producers =======================
    // Producer w issues stages w, w + 2, w + 4, ...: lane 0 claims the ring
    // slot, then the lanes issue the stage's boxes concurrently.  A producer's
    // serial work per stage caps the rate of small stages (32 KB for MQA), so
    // two share them, and each keeps its part short: the block_table entries of
    // its next stage are read while the current one waits for its slot, and the
    // per-lane box geometry of a full stage is computed once.  (Consumers free
    // stages in order, so a producer waiting for stage i - S to be freed has
    // seen stage i - 2 - S freed: it is never two phases ahead of a slot.)
    const int pw = warp - C::kConsumers;
    const int R = ps < 16 ? ps : 16;  // rows per box (page_size >= 8)
    // page_size >= 16: one box per (tensor, block) covers every slab; page_size
    // 8: one box per (tensor, block, slab, 8-row half) so rows land at 16-row pitch
    const int slabs_per_op = R == 16 ? C::kSlabs : 1;
    const int boxes_per_block = (16 / R) * (C::kSlabs / slabs_per_op);
    constexpr int kOpsPerLane = 2;  // at most 2 tensors x 8 blocks x 4 boxes = 64 ops a stage
    static_assert(2 * NBS * 2 * (D / 64) <= 32 * kOpsPerLane, "ops per stage");
    // op -> (block jj, first row q*R of the box) and its shared-memory offset in
    // the stage; tensor TT = K or V, slab sl
    struct OpGeom {
      int jj, q, TT, sl;
      uint32_t off;
      bool on;
    };
    auto geom = [&](int nbs, int op) {
      OpGeom g;
      g.on = op < 2 * nbs * boxes_per_block;
      const int sub = op % boxes_per_block;
      g.q = sub % (16 / R);
      g.sl = sub / (16 / R);
      g.jj = (op / boxes_per_block) % nbs;
      g.TT = op / (boxes_per_block * nbs);
      g.off = (uint32_t)(((g.TT * NBS + g.jj) * C::kSlabs + g.sl) * C::kBoxBytes + g.q * R * C::kRowBytes);
      return g;
    };
    // every stage but a segment's last has NBS blocks: its geometry is fixed per lane
    OpGeom full_geom[kOpsPerLane];
#pragma unroll
    for (int x = 0; x < kOpsPerLane; ++x) full_geom[x] = geom(NBS, lane + 32 * x);
    // raw block_table entries of this lane's ops in the stage at cu (loads only)
    auto fetch = [&](const Cursor& cu, int nbs, int (&pg)[kOpsPerLane]) {
      const int32_t* bt = p.block_table + page_list_start(p.kv_indptr, p.max_blocks, cu.b);
#pragma unroll
      for (int x = 0; x < kOpsPerLane; ++x) {
        const OpGeom g = nbs == NBS ? full_geom[x] : geom(nbs, lane + 32 * x);
        const int kk = (cu.k + g.jj) * 16 + g.q * R;
        pg[x] = (g.on && nbs > 0 && kk < cu.L) ? __ldg(bt + (kk >> pshift)) : 0;
      }
    };
    // the stage after the one at (c, nb); nb = 0 past the CTA's range
    auto next_stage = [&](Cursor& c, int& nb) {
      if (nb == 0) return;
      advance(c, nb);
      nb = c.u < u1 ? stage_blocks(c) : 0;
    };
    Cursor cur = locate(u0);
    bool alive = true;
    int nbs = stage_blocks(cur);
    // this producer's next stage index i, kept as ring slot + wrap count
    // (no division in the loop): slot = i % S, lap = i / S
    int slot = 0, lap = 0;
    if (pw == 1) {
      next_stage(cur, nbs);
      slot = 1;  // S >= 2
    }
    // page ids of the current and the next stage; the loop is unrolled by two
    // with the buffers swapped, so no register holding a load in flight is
    // ever copied (a copy would wait for the load)
    int pga[kOpsPerLane], pgb[kOpsPerLane];
    fetch(cur, nbs, pga);  // block_table is an input, not written by the append kernel
    griddep_wait();        // the pool rows of this step were written by the append kernel
    auto stage = [&](int (&pg)[kOpsPerLane], int (&pg_n)[kOpsPerLane]) {
      Cursor nx = cur;
      int nbs_n = nbs;
      next_stage(nx, nbs_n);
      next_stage(nx, nbs_n);  // this producer's next stage: two ahead
      fetch(nx, nbs_n, pg_n);
      // this stage's rows first (its page ids were read an iteration ago), so
      // a slot is refilled the moment it is freed
      const uint32_t sbase = smem_u32(ring + slot * C::kStageBytes);
      int row[kOpsPerLane];
      uint32_t dst[kOpsPerLane];
      int mine = 0;
#pragma unroll
      for (int x = 0; x < kOpsPerLane; ++x) {
        const OpGeom g = nbs == NBS ? full_geom[x] : geom(nbs, lane + 32 * x);
        const int kk = (cur.k + g.jj) * 16 + g.q * R;
        row[x] = -1;
        dst[x] = sbase + g.off;
        if (g.on && kk < cur.L) {
          const int page = pg[x];
          if (page < 0 || page >= p.pool.num_pages) {
            if (g.sl == 0 && g.TT == 0) record_error(p.err, ERR_BLOCK_TABLE, page);
          } else {
            row[x] = page * ps + (kk & (ps - 1));
            ++mine;
          }
        }
      }
      const int issued = __reduce_add_sync(0xffffffffu, mine);
      if (lane == 0 && lap > 0 && alive) alive = mbar_wait(empty_bar(slot), (uint32_t)((lap - 1) & 1), p.err);
      alive = __shfl_sync(0xffffffffu, alive ? 1 : 0, 0) != 0;
      if (lane == 0) mbar_arrive_expect_tx(full_bar(slot), (uint32_t)(issued * R * C::kRowBytes * HB * slabs_per_op));
      __syncwarp();
#pragma unroll
      for (int x = 0; x < kOpsPerLane; ++x) {
        if (row[x] < 0) continue;
        const OpGeom g = nbs == NBS ? full_geom[x] : geom(nbs, lane + 32 * x);
        if (KV8)
          tma_load_3d(dst[x], g.TT ? &tmap_v : &tmap_k, 0, row[x], cur.hk * HB, full_bar(slot));
        else
          tma_load_4d(dst[x], g.TT ? &tmap_v : &tmap_k, 0, row[x], cur.hk * HB, g.sl, full_bar(slot));
      }
      cur = nx;
      nbs = nbs_n;
      slot += C::kKvProducers;  // kKvProducers <= S
      if (slot >= S) {
        slot -= S;
        ++lap;
      }
    };
    while (nbs > 0) {
      stage(pga, pgb);
      if (nbs == 0) break;
      stage(pgb, pga);
    }
    return;
  }

  // ======================= consumer warps =======================
  const int h = warp % HB;               // head within the box
  const int jw = (warp / HB) % NW;       // blocks jw * BPW .. jw * BPW + BPW - 1 of each stage
  const int rt = warp / (HB * NW);       // row tile: query heads rt*16 .. rt*16+15 of the group
  const int rA = rt * 16 + (lane >> 2), rB = rA + 8;
  const float sl2 = p.scale_log2;
  const int mi = lane >> 3, rr = lane & 7;
  Cursor cc = locate(u0);
  int ncut = 0;        // (kCostlyChange) cut segments handed to the publisher so far
  int slot = 0;        // ring slot of the next stage (stage index % S)
  uint32_t phase = 0;  // its full-barrier parity ((stage index / S) & 1)
  bool alive = true;
  for (int seg = 0; cc.u < u1; ++seg) {
    const int seg_blocks = (int)min((int64_t)(cc.nblk - cc.k), u1 - cc.u);
    const int first_k = cc.k;
    const int hk = cc.hk * HB + h;  // this warp's KV head
    // ---- query rows of head hk (A fragments of m16n8k16; rows >= G are zero) ----
    uint32_t qf[D / 16][4];
    {
      const int qs = seg & 1;
      if (alive) alive = mbar_wait(qfull_bar(qs), (seg >> 1) & 1, p.err);
      const uint32_t* qsm = reinterpret_cast<const uint32_t*>(qring + qs * lay.qslot) + (h * G * D) / 2;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        if (KV8) {
          // f16, dims permuted to match the e4m3 K fragments: within a 16-dim
          // step, MMA k = 2c, 2c + 1 are dims 4c, 4c + 1 and k = 2c + 8, 2c + 9
          // are dims 4c + 2, 4c + 3 (c = lane % 4)
          const int d0 = kk * 16 + (lane & 3) * 4;
          qf[kk][0] = rA < G ? bf16x2_to_f16x2(qsm[(rA * D + d0) >> 1]) : 0u;
          qf[kk][1] = rB < G ? bf16x2_to_f16x2(qsm[(rB * D + d0) >> 1]) : 0u;
          qf[kk][2] = rA < G ? bf16x2_to_f16x2(qsm[(rA * D + d0 + 2) >> 1]) : 0u;
          qf[kk][3] = rB < G ? bf16x2_to_f16x2(qsm[(rB * D + d0 + 2) >> 1]) : 0u;
        } else {
          const int d0 = kk * 16 + (lane & 3) * 2;
          qf[kk][0] = rA < G ? qsm[(rA * D + d0) >> 1] : 0u;
          qf[kk][1] = rB < G ? qsm[(rB * D + d0) >> 1] : 0u;
          qf[kk][2] = rA < G ? qsm[(rA * D + d0 + 8) >> 1] : 0u;
          qf[kk][3] = rB < G ? qsm[(rB * D + d0 + 8) >> 1] : 0u;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty_bar(qs));
    }
    float o[D / 8][4];
#pragma unroll
    for (int n8 = 0; n8 < D / 8; ++n8) o[n8][0] = o[n8][1] = o[n8][2] = o[n8][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int done = 0; done < seg_blocks;) {
      const int nbs = min(NBS, seg_blocks - done);
      // fused append: one of this warp's blocks may be the sequence's last,
      // whose row L_b - 1 is the new token; fetch this lane's 8 elements of
      // the new K / V row of head hk before the wait (lanes 0 .. D/8 - 1: K,
      // then V)
      const int last_jb = cc.nblk - 1 - (first_k + done);  // the last block's index in this stage
      const int new_bb = (FUSED && last_jb >= jw * BPW && last_jb < jw * BPW + BPW && last_jb < nbs &&
                          __ldg(p.new_slots + cc.b) >= 0)
                             ? last_jb - jw * BPW
                             : -1;
      constexpr int kRowChunks = D / 8;  // lanes per tensor
      uint4 nr = make_uint4(0, 0, 0, 0);
      if (new_bb >= 0 && lane < 2 * kRowChunks) {
        const int T = lane / kRowChunks, e8 = lane - T * kRowChunks;
        nr = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(T ? p.new_v : p.new_k) +
                                                  ((int64_t)cc.b * Hkv + hk) * D) + e8);
      }
      if (alive) alive = mbar_wait(full_bar(slot), phase, p.err);
      if (jw * BPW < nbs) {
        unsigned char* st = ring + slot * C::kStageBytes;
        float s[2 * BPW][4];
        int valid[BPW];
        uint32_t vbase[BPW];
        bool touched = false;  // shared-memory stores this warp made into the stage
#pragma unroll
        for (int bb = 0; bb < BPW; ++bb) {
          const int jb = jw * BPW + bb;  // block within the stage
          s[2 * bb][0] = s[2 * bb][1] = s[2 * bb][2] = s[2 * bb][3] = 0.f;
          s[2 * bb + 1][0] = s[2 * bb + 1][1] = s[2 * bb + 1][2] = s[2 * bb + 1][3] = 0.f;
          valid[bb] = jb < nbs ? cc.L - (first_k + done + jb) * 16 : 0;  // >= 1 for a block of the stage
          unsigned char* kt = st + (jb * C::kSlabs) * C::kBoxBytes + h * C::kHeadTile;
          unsigned char* vt = st + ((NBS + jb) * C::kSlabs) * C::kBoxBytes + h * C::kHeadTile;
          vbase[bb] = smem_u32(vt);
          if (jb >= nbs) continue;
          if (valid[bb] < 16) {
            // rows past L_b may hold stale or poisoned data (NaN would survive
            // P = 0): zero them in V; K is masked below.  A row's chunks stay in
            // the row under either swizzle.
            constexpr int kCh = C::kRowBytes / 16;  // 16-byte chunks of a row of one slab
            for (int e = lane; e < (16 - valid[bb]) * C::kSlabs * kCh; e += 32) {
              const int row = valid[bb] + e / (C::kSlabs * kCh);
              const int rem = e % (C::kSlabs * kCh);
              *reinterpret_cast<uint4*>(vt + (rem / kCh) * C::kBoxBytes + row * C::kRowBytes + (rem % kCh) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
            touched = true;
          }
          if (bb == new_bb) {
            // the new token's K and V rows (row L_b - 1 of this block) come from
            // the input: the pool row may still be in flight from the append above
            const int r = valid[bb] - 1;
            if (lane < 2 * kRowChunks) {
              const int T = lane / kRowChunks, e8 = lane - T * kRowChunks;  // elements 8*e8 .. 8*e8 + 7
              unsigned char* tile = T ? vt : kt;
              if (KV8)  // 8 codes: half of 16-byte chunk e8 / 2 (a chunk stays contiguous under the swizzle)
                *reinterpret_cast<uint2*>(tile + sw_e4m3<D>(r, e8 >> 1) + (e8 & 1) * 8) =
                    quantize8(nr, T ? p.v_quant : p.k_quant);
              else
                *reinterpret_cast<uint4*>(tile + sw128(r, e8, C::kBoxBytes)) = nr;
            }
            __syncwarp();
            touched = true;
          }
          const uint32_t kbase = smem_u32(kt);
          if (KV8) {
            // e4m3 K as 16-bit pairs: matrix m = keys (m & 1) * 8 .. + 7 of
            // 16-dim chunk 2 * q2 + (m >> 1); lane gets 4 codes of key lane / 4,
            // dims 4c .. 4c + 3: the first two are B register 0, the last two 1
#pragma unroll
            for (int q2 = 0; q2 < D / 32; ++q2) {
              uint32_t r0, r1, r2, r3;
              ldmatrix_x4(kbase + sw_e4m3<D>((mi & 1) * 8 + rr, 2 * q2 + (mi >> 1)), r0, r1, r2, r3);
              mma_f16_16816(s[2 * bb], qf[2 * q2], e4m3x2_lo_to_f16x2(r0), e4m3x2_hi_to_f16x2(r0));
              mma_f16_16816(s[2 * bb + 1], qf[2 * q2], e4m3x2_lo_to_f16x2(r1), e4m3x2_hi_to_f16x2(r1));
              mma_f16_16816(s[2 * bb], qf[2 * q2 + 1], e4m3x2_lo_to_f16x2(r2), e4m3x2_hi_to_f16x2(r2));
              mma_f16_16816(s[2 * bb + 1], qf[2 * q2 + 1], e4m3x2_lo_to_f16x2(r3), e4m3x2_hi_to_f16x2(r3));
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              uint32_t b0, b1, b2, b3;
              ldmatrix_x4(kbase + sw128((mi >> 1) * 8 + rr, kk * 2 + (mi & 1), C::kBoxBytes), b0, b1, b2, b3);
              mma_bf16_16816(s[2 * bb], qf[kk], b0, b1);
              mma_bf16_16816(s[2 * bb + 1], qf[kk], b2, b3);
            }
          }
        }
#pragma unroll
        for (int t = 0; t < 2 * BPW; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = (t & 1) * 8 + (lane & 3) * 2 + (e & 1);
            s[t][e] = key < valid[t >> 1] ? s[t][e] * sl2 : -INFINITY;
          }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int t = 0; t < 2 * BPW; ++t) {
          mx0 = fmaxf(mx0, fmaxf(s[t][0], s[t][1]));
          mx1 = fmaxf(mx1, fmaxf(s[t][2], s[t][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
        float p_[2 * BPW][4];
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int t = 0; t < 2 * BPW; ++t) {
          p_[t][0] = fast_exp2(s[t][0] - mn0);
          p_[t][1] = fast_exp2(s[t][1] - mn0);
          p_[t][2] = fast_exp2(s[t][2] - mn1);
          p_[t][3] = fast_exp2(s[t][3] - mn1);
          rs0 += p_[t][0] + p_[t][1];
          rs1 += p_[t][2] + p_[t][3];
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
        for (int bb = 0; bb < BPW; ++bb) {
          if (jw * BPW + bb >= nbs) continue;
          uint32_t pa[4];
          if (KV8) {
            pa[0] = pack_f16(p_[2 * bb][0], p_[2 * bb][1]);
            pa[1] = pack_f16(p_[2 * bb][2], p_[2 * bb][3]);
            pa[2] = pack_f16(p_[2 * bb + 1][0], p_[2 * bb + 1][1]);
            pa[3] = pack_f16(p_[2 * bb + 1][2], p_[2 * bb + 1][3]);
          } else {
            pa[0] = pack_bf16(p_[2 * bb][0], p_[2 * bb][1]);
            pa[1] = pack_bf16(p_[2 * bb][2], p_[2 * bb][3]);
            pa[2] = pack_bf16(p_[2 * bb + 1][0], p_[2 * bb + 1][1]);
            pa[3] = pack_bf16(p_[2 * bb + 1][2], p_[2 * bb + 1][3]);
          }
          if (KV8) {
            // e4m3 V, transposed as 16-bit pairs: lane gets keys 2c, 2c + 1 of
            // dims 2j, 2j + 1 (j = lane / 4) of a 16-dim chunk, regrouped to key
            // pairs per dim; the even dims form output tile 2 * chunk, the odd
            // ones tile 2 * chunk + 1, so o[t] column n is dim (t / 2) * 16 + 2n + t % 2
#pragma unroll
            for (int q2 = 0; q2 < D / 32; ++q2) {
              uint32_t r0, r1, r2, r3;
              ldmatrix_x4_trans(vbase[bb] + sw_e4m3<D>((mi & 1) * 8 + rr, 2 * q2 + (mi >> 1)), r0, r1, r2, r3);
              r0 = __byte_perm(r0, 0u, 0x3120);  // (key 2c, key 2c+1) of dim 2j | same of dim 2j+1
              r1 = __byte_perm(r1, 0u, 0x3120);
              r2 = __byte_perm(r2, 0u, 0x3120);
              r3 = __byte_perm(r3, 0u, 0x3120);
              mma_f16_16816(o[4 * q2], pa, e4m3x2_lo_to_f16x2(r0), e4m3x2_lo_to_f16x2(r1));
              mma_f16_16816(o[4 * q2 + 1], pa, e4m3x2_hi_to_f16x2(r0), e4m3x2_hi_to_f16x2(r1));
              mma_f16_16816(o[4 * q2 + 2], pa, e4m3x2_lo_to_f16x2(r2), e4m3x2_lo_to_f16x2(r3));
              mma_f16_16816(o[4 * q2 + 3], pa, e4m3x2_hi_to_f16x2(r2), e4m3x2_hi_to_f16x2(r3));
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < D / 16; ++jj) {
              uint32_t b0, b1, b2, b3;
              ldmatrix_x4_trans(vbase[bb] + sw128((mi & 1) * 8 + rr, 2 * jj + (mi >> 1), C::kBoxBytes), b0, b1, b2,
                                b3);
              mma_bf16_16816(o[2 * jj], pa, b0, b1);
              mma_bf16_16816(o[2 * jj + 1], pa, b2, b3);
            }
          }
        }
        if (touched) fence_proxy_async_smem();  // our stores precede the next TMA into this slot
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(slot));
      done += nbs;
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
    }

    // ---- segment end: normalise / merge / write ----
    // Output pair x (0 .. D/8 - 1) of this lane, for rows rA (half 0) / rB
    // (half 1): two adjacent dims starting at out_col(x).  bf16 tiles hold
    // dims t * 8 + 2c, 2c + 1; the e4m3 path's tiles 2k, 2k + 1 hold the even
    // and odd dims of chunk k, so a lane's adjacent pairs mix the two.
    auto out_col = [&](int x) {
      const int k = x >> 1, pi = x & 1, c = lane & 3;
      return KV8 ? k * 16 + 4 * c + 2 * pi : k * 16 + 8 * pi + 2 * c;
    };
    auto out_pair = [&](const float (&acc)[D / 8][4], int x, int half) {
      const int k = x >> 1, pi = x & 1;
      return KV8 ? make_float2(acc[2 * k][2 * half + pi], acc[2 * k + 1][2 * half + pi])
                 : make_float2(acc[2 * k + pi][2 * half], acc[2 * k + pi][2 * half + 1]);
    };
    float la = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
    la += __shfl_xor_sync(0xffffffffu, la, 2);
    float lb = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
    lb += __shfl_xor_sync(0xffffffffu, lb, 2);
    // a segment whole in this CTA is finished here, unless a cascade's prefix
    // partials still have to be merged in (then the combine kernel finishes it)
    const bool complete = (first_k == 0) && (seg_blocks == cc.nblk) && p.pre_chunks == 0;
    const int64_t seg_id = (int64_t)cc.b * Hg + cc.hk;
    const int64_t pslot = (seg_id + c) * HB + h;  // unique per (segment, CTA, head)
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out) + ((int64_t)cc.b * Hq + (int64_t)hk * G) * D;
    if (NW > 1) {
      // NW warps share each head and row tile, each with the state of its
      // blocks of every stage: chained through one shared-memory slot, warp
      // NW - 1 hands its state to warp NW - 2, ... down to warp 0 (one slot
      // instead of NW leaves room for another stage of the ring).
      // o_w = 2^(m_w - M) o_w + 2^(m_x - M) o_x, the same for l, M = max(m_w, m_x).
      float* mo = mrg_o + (h * G) * D;
      float* mml = mrg_ml + (h * G) * 2;
      auto set_pair = [&](int x, int half, float2 v) {
        const int k = x >> 1, pi = x & 1;
        if (KV8) {
          o[2 * k][2 * half + pi] = v.x;
          o[2 * k + 1][2 * half + pi] = v.y;
        } else {
          o[2 * k + pi][2 * half] = v.x;
          o[2 * k + pi][2 * half + 1] = v.y;
        }
      };
#pragma unroll 1
      for (int w = NW - 1; w >= 1; --w) {
        if (jw == w) {
          if ((lane & 3) == 0) {
            if (rA < G) { mml[rA * 2] = m0; mml[rA * 2 + 1] = la; }
            if (rB < G) { mml[rB * 2] = m1; mml[rB * 2 + 1] = lb; }
          }
#pragma unroll
          for (int x = 0; x < D / 8; ++x) {
            const int col = out_col(x);
            if (rA < G) *reinterpret_cast<float2*>(&mo[rA * D + col]) = out_pair(o, x, 0);
            if (rB < G) *reinterpret_cast<float2*>(&mo[rB * D + col]) = out_pair(o, x, 1);
          }
        }
        named_barrier(1, C::kConsumers * 32);
        if (jw == w - 1) {
          float fa = 1.f, ga = 0.f, fb = 1.f, gb = 0.f;  // weights of mine / the handed-over state
          if (rA < G) {
            const float mx = mml[rA * 2], M = fmaxf(m0, mx);
            fa = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M);
            ga = mx == -INFINITY ? 0.f : fast_exp2(mx - M);
            la = la * fa + mml[rA * 2 + 1] * ga;
            m0 = M;
          }
          if (rB < G) {
            const float mx = mml[rB * 2], M = fmaxf(m1, mx);
            fb = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M);
            gb = mx == -INFINITY ? 0.f : fast_exp2(mx - M);
            lb = lb * fb + mml[rB * 2 + 1] * gb;
            m1 = M;
          }
#pragma unroll
          for (int x = 0; x < D / 8; ++x) {
            const int col = out_col(x);
            float2 va = out_pair(o, x, 0), vb = out_pair(o, x, 1);
            if (rA < G) {
              const float2 t = *reinterpret_cast<const float2*>(&mo[rA * D + col]);
              va = make_float2(va.x * fa + t.x * ga, va.y * fa + t.y * ga);
            }
            if (rB < G) {
              const float2 t = *reinterpret_cast<const float2*>(&mo[rB * D + col]);
              vb = make_float2(vb.x * fb + t.x * gb, vb.y * fb + t.y * gb);
            }
            set_pair(x, 0, va);
            set_pair(x, 1, vb);
          }
        }
        named_barrier(1, C::kConsumers * 32);
      }
    }
    if (jw == 0) {
      // this warp holds its rows' whole segment state: write it
      // v_scale: e4m3 V codes stand for code * v_scale (1 for bf16 pools)
      const float ia = la > 0.f ? p.v_scale / la : 0.f, ib = lb > 0.f ? p.v_scale / lb : 0.f;
#pragma unroll
      for (int x = 0; x < D / 8; ++x) {
        const int col = out_col(x);
        const float2 va = out_pair(o, x, 0), vb = out_pair(o, x, 1);
        if (complete) {
          if (rA < G) *reinterpret_cast<uint32_t*>(outp + rA * D + col) = pack_bf16(va.x * ia, va.y * ia);
          if (rB < G) *reinterpret_cast<uint32_t*>(outp + rB * D + col) = pack_bf16(vb.x * ib, vb.y * ib);
        } else {
          if (rA < G) *reinterpret_cast<float2*>(p.part_o + (pslot * G + rA) * D + col) = va;
          if (rB < G) *reinterpret_cast<float2*>(p.part_o + (pslot * G + rB) * D + col) = vb;
        }
      }
      if (!complete && (lane & 3) == 0) {
        if (rA < G) p.part_ml[pslot * G + rA] = make_float2(m0, la);
        if (rB < G) p.part_ml[pslot * G + rB] = make_float2(m1, lb);
      }
    }
    if (!complete && p.pre_chunks == 0) {
      // This CTA's part of a segment cut across CTAs is written.  Publish and
      // count it: the consumer barrier orders every consumer thread's partial
      // writes before the publishing thread's fence (cumulative) and count
      // (thread 0, or the publisher warp after thread 0's CTA-scope release on
      // an mbarrier).  The segment is merged after the CTAs' ranges, with the
      // stage rings idle: by each CTA holding a part, a slice of the rows each
      // (co-resident grid), or else by the CTA that counts the last part.  No
      // consumer waits here.
      named_barrier(2, C::kConsumers * 32);
      if constexpr (C::kCostlyChange) {
        if (tid == 0) mbar_arrive(pub_bar(ncut));
        ++ncut;
      } else if (tid == 0) {
        const int64_t us = (int64_t)Hg * prefix[cc.b] + (int64_t)cc.hk * cc.nblk;
        const int c0 = cta_of_unit(us, W, n), c1 = cta_of_unit(us + cc.nblk - 1, W, n);
        int arrivals = c1 - c0 + 1, mine = c - c0;  // CTAs c0 .. c1 own the segment's units ...
        if (W < n) {  // ... except those without a unit, which took no part
          arrivals = mine = 0;
          for (int x = c0; x <= c1; ++x) {
            const int part = cta_range_empty(x, W, n) ? 0 : 1;
            arrivals += part;
            if (x < c) mine += part;
          }
        }
        fence_acq_rel_gpu();  // release: the partials above, then the count
        const bool last = arrive_part(p.seg_count + seg_id, *tag_slot, p.err) == (unsigned)(arrivals - 1);
        if (p.slice_merge || last) {
          const int e = pending[0];  // a CTA range cuts at most 2 segments
          volatile int* ent = pending + 1 + kPend * e;
          ent[0] = cc.b;
          ent[1] = cc.hk;
          ent[2] = c0;
          ent[3] = c1 - c0 + 1;  // the merge walks the CTA span (empty CTAs weigh 0)
          ent[4] = p.slice_merge ? arrivals + p.test_extra_parts : 1;
          ent[5] = p.slice_merge ? mine : 0;
          pending[0] = e + 1;
        }
      }
    }
    advance(cc, seg_blocks);
  }
  if (p.pre_chunks == 0) {
    if constexpr (C::kCostlyChange) {
      if (tid == 0 && alive) alive = mbar_wait(pubd_bar, 0, p.err);  // every part of this CTA published
    }
    named_barrier(2, C::kConsumers * 32);  // every count of this CTA recorded; the ring is idle
    const int npend = pending[0];
    // A range cuts at most two segments, its first and its last.  With two to
    // merge, the consumer warps split in halves that wait for and merge one
    // segment each at the same time (each with half the idle ring as scratch
    // and its own named barrier), so the later merge does not queue behind
    // the earlier one.
    const int groups = npend == 2 ? 2 : 1;
    const int gsize = C::kConsumers * 32 / groups;
    const int grp = tid / gsize, gtid = tid - grp * gsize;
    const int bar_id = groups == 2 ? 3 + grp : 2;
    const int scratch_bytes = S * C::kStageBytes / groups;
    for (int e = grp; e < npend; e += groups) {
      volatile int* ent = pending + 1 + kPend * e;
      const int b = ent[0], hkb = ent[1], c0 = ent[2], span = ent[3], parts = ent[4], mine = ent[5];
      if (gtid == 0) {
        if (p.slice_merge) {
          // wait for the segment's last part (its CTAs are all resident and
          // run to their range ends without waiting on anyone); the acquire
          // load that sees the full count orders the parts' partials (each
          // published by a fence and a count) before this group's reads
          const unsigned long long tag = *tag_slot;
          const unsigned long long* cnt = p.seg_count + (int64_t)b * Hg + hkb;
          const unsigned long long limit = p.part_wait_ns != 0 ? p.part_wait_ns : kWaitLimitNs;
          const unsigned long long t0 = global_ns();
          for (;;) {
            const unsigned long long w = ld_acquire_gpu(cnt);
            if ((w >> 16) == tag && (int)(w & 0xFFFFu) >= parts) break;
            if (global_ns() - t0 > limit) {
              record_error(p.err, ERR_TIMEOUT, -2);
              break;
            }
            __nanosleep(128);
          }
        } else {
          fence_acq_rel_gpu();  // this CTA counted the last part: the others' partials before its reads
        }
      }
      named_barrier(bar_id, gsize);
      // merge rows [mine, mine + 1) * rows / parts of the segment
      const int rows = HB * p.group;
      merge_segment<D>(p, b, hkb, c0, span, HB, Hg, W, n, mine * rows / parts, (mine + 1) * rows / parts,
                       ring + grp * scratch_bytes, scratch_bytes, gtid, gsize, bar_id);
      named_barrier(bar_id, gsize);  // before a next merge reuses the scratch
    }
  }
}

}  // namespace

// Cooperative launch with programmatic serialization: 0 not tried yet, 1
// accepted, -1 refused (decode_bf16.cu).
int coop_launch_state();
void set_coop_launch_state(int v);

// head_dim 128, 8 heads per box, 16-row groups, seg_penalty > 0: the WC
// instantiations (decode_weighted.cu)
cudaError_t launch_split_weighted(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, bool kv8,
                                  bool fused, cudaStream_t s);

namespace {

template <int D, int HB, int RT, bool KV8, bool FUSED, bool WC = false>
cudaError_t launch_split(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  using C = Cfg<D, HB, RT, KV8, WC>;
  const Layout lay = make_layout<D, HB, RT, KV8, WC>(p.group, p.batch, p.smem_budget);
  if (lay.stages < 2) return cudaErrorInvalidConfiguration;
  auto kern = decode_split_kernel<D, HB, RT, KV8, FUSED, WC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total);
  if (e != cudaSuccess) return e;
  // Plain decode: a co-resident (cooperative) grid lets every CTA of a cut
  // segment merge a slice of it.  Whether the runtime takes a cooperative
  // launch with programmatic serialization is learnt from the first eager
  // launch (never tried inside a stream capture); otherwise the CTA counting
  // a segment's last part merges it whole.
  if (p.pre_chunks == 0 && coop_launch_state() >= 0) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess &&
        (cs == cudaStreamCaptureStatusNone || coop_launch_state() > 0)) {
      DecodeParams pc = p;
      pc.slice_merge = 1;
      e = launch_pdl_coop(kern, dim3(p.num_ctas), dim3(C::kThreads), (size_t)lay.total, s, tk, tv, pc);
      if (e == cudaSuccess) {
        set_coop_launch_state(1);
        return e;
      }
      (void)cudaGetLastError();
      if (cs != cudaStreamCaptureStatusNone) return e;  // the capture is lost: report it
      set_coop_launch_state(-1);
    }
  }
  return launch_pdl(kern, dim3(p.num_ctas), dim3(C::kThreads), (size_t)lay.total, s, tk, tv, p);
}

template <int D, bool KV8, bool FUSED>
cudaError_t launch_split_d(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rt,
                           cudaStream_t s) {
  switch (p.heads_per_box * 10 + rt) {
    case 81:
      // 16-row groups in boxes of 8 heads with a segment penalty: the WC
      // instantiation (decode_weighted.cu)
      if constexpr (D == 128)
        if (p.seg_penalty > 0) return launch_split_weighted(p, tk, tv, KV8, FUSED, s);
      return launch_split<D, 8, 1, KV8, FUSED>(p, tk, tv, s);
    case 41: return launch_split<D, 4, 1, KV8, FUSED>(p, tk, tv, s);
    case 21: return launch_split<D, 2, 1, KV8, FUSED>(p, tk, tv, s);
    case 11: return launch_split<D, 1, 1, KV8, FUSED>(p, tk, tv, s);
    case 42: return launch_split<D, 4, 2, KV8, FUSED>(p, tk, tv, s);
    case 22: return launch_split<D, 2, 2, KV8, FUSED>(p, tk, tv, s);
    case 12: return launch_split<D, 1, 2, KV8, FUSED>(p, tk, tv, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

}  // namespace pa
