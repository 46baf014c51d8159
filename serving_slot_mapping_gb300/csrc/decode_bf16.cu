// paged_attention_decode, bf16 and e4m3 paths: the host side of the split-KV
// decode (launch geometry, shared-memory layout, tensor maps) and, for
// cascade decode only, the combine kernel that merges the split kernel's
// partials with the shared prefix's.  The split kernel itself is in
// decode_split.cuh (see there for the work decomposition).
#include <atomic>

#include "decode_split.cuh"

namespace pa {

namespace {

// Cascade decode: merge each (sequence, KV head) pair's own-key partials
// (those of every CTA that owns a part of the sequence; none if it has no key
// of its own) with the shared prefix's partials, one per key chunk.  One CTA
// per pair; warp w merges rows g = w, w + 4, ... of the pair's G query heads:
// lanes load the partials' (m, l) in parallel and reduce with shuffles, then
// each lane accumulates 4 dims with float4 loads, 8 partials in flight.
__global__ void __launch_bounds__(128) decode_combine_kernel(DecodeParams p, int D) {
  const int Hkv = p.pool.num_kv_heads;
  const int HB = p.heads_per_box;
  const int Hg = Hkv / HB;
  const int G = p.group;
  const int pair = blockIdx.x;
  const int b = pair / Hkv, hk = pair - (pair / Hkv) * Hkv;
  const int hg = hk / HB, h = hk - (hk / HB) * HB;
  const int max_len = p.max_blocks * p.pool.page_size;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // The prologue reads only seq_lens and overlaps the split kernel's tail;
  // partials are read after the split grid has completed.
  __shared__ long long red[2][4];
  long long before = 0, total = 0;
  for (int i = threadIdx.x; i < p.batch; i += blockDim.x) {
    const int nb = (seq_len_of(p, i, max_len) + 15) >> 4;
    total += nb;
    if (i < b) before += nb;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  if (lane == 0) { red[0][warp] = before; red[1][warp] = total; }
  __syncthreads();
  before = red[0][0] + red[0][1] + red[0][2] + red[0][3];
  total = red[1][0] + red[1][1] + red[1][2] + red[1][3];
  const int nblk = (seq_len_of(p, b, max_len) + 15) >> 4;
  griddep_wait();
  const int n = p.num_ctas;
  int c0 = 0, nparts = 0;
  bool some_empty = false;
  int64_t U = 0;
  if (nblk > 0) {
    U = total * Hg;
    const int64_t us = before * Hg + (int64_t)hg * nblk, ue = us + nblk;
    c0 = cta_of_unit(us, U, n);
    nparts = cta_of_unit(ue - 1, U, n) - c0 + 1;
    some_empty = U < n;
  }
  const int64_t seg = (int64_t)b * Hg + hg;
  const int nparts_all = nparts + p.pre_chunks;
  const int64_t Hq = p.num_q_heads;
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(p.out) + ((int64_t)b * Hq + (int64_t)hk * G) * D;
  for (int g = warp; g < G; g += 4) {
    const int64_t hq = (int64_t)hk * G + g;
    auto ml_of = [&](int q) {  // q < nparts: own-key partial q; else prefix chunk q - nparts
      if (q < nparts) {
        if (some_empty && cta_range_empty(c0 + q, U, n)) return make_float2(-INFINITY, 0.f);
        return __ldcg(p.part_ml + ((seg + c0 + q) * HB + h) * G + g);
      }
      return __ldcg(p.pre_ml + ((int64_t)(q - nparts) * p.batch + b) * Hq + hq);
    };
    auto row_of = [&](int q) {
      if (q < nparts)
        return reinterpret_cast<const float4*>(p.part_o + (((seg + c0 + q) * HB + h) * G + g) * D);
      return reinterpret_cast<const float4*>(p.pre_o + (((int64_t)(q - nparts) * p.batch + b) * Hq + hq) * D);
    };
    // (m, l): lane q holds partial q (the first 32), later ones are looped over
    const float2 ml_mine = lane < nparts_all ? ml_of(lane) : make_float2(-INFINITY, 0.f);
    float M = ml_mine.x;
    for (int q = lane + 32; q < nparts_all; q += 32) M = fmaxf(M, ml_of(q).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float f_mine = (ml_mine.x == -INFINITY) ? 0.f : fast_exp2(ml_mine.x - M);
    float den = f_mine * ml_mine.y;
    for (int q = lane + 32; q < nparts_all; q += 32) {
      const float2 ml = ml_of(q);
      den += (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M) * ml.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    const float inv = den > 0.f ? p.v_scale / den : 0.f;
    // weighted rows, 8 partials at a time with all their loads in flight; a
    // partial of weight 0 (empty, or negligible) is not read
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const bool dims = 4 * lane < D;
    for (int q0 = 0; q0 < nparts_all; q0 += 8) {
      float f[8];
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int q = q0 + u;
        f[u] = __shfl_sync(0xffffffffu, f_mine, q & 31);
        if (q >= 32 && q < nparts_all) {
          const float2 ml = ml_of(q);
          f[u] = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
        }
        if (q >= nparts_all) f[u] = 0.f;
        v[u] = (dims && f[u] != 0.f) ? __ldcg(row_of(q) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x += f[u] * v[u].x; acc.y += f[u] * v[u].y; acc.z += f[u] * v[u].z; acc.w += f[u] * v[u].w;
      }
    }
    if (dims) {
      uint2 packed;
      packed.x = pack_bf16(acc.x * inv, acc.y * inv);
      packed.y = pack_bf16(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(outp + (int64_t)g * D + 4 * lane) = packed;
    }
  }
}

}  // namespace

namespace {
std::atomic<int> g_coop_state{0};
}  // namespace

int coop_launch_state() { return g_coop_state.load(std::memory_order_relaxed); }
void set_coop_launch_state(int v) { g_coop_state.store(v, std::memory_order_relaxed); }

int decode_heads_per_box(int32_t num_kv_heads, int32_t group, int32_t page_size) {
  const int rt = group <= 16 ? 1 : 2;
  if (page_size < 16) return 1;
  int hb = 1;
  while (hb * 2 <= 8 / rt && num_kv_heads % (hb * 2) == 0) hb *= 2;
  return hb;
}

// 32-row groups (two row tiles): a CTA loses ~5 us at each segment change of
// its range (measured on GB300 with per-CTA global-timer stamps: the NW
// consumer warps' chained merge, the part's write and count, the next
// segment's query rows).  In 16-key blocks of one head box that is the
// change's time over one block's: its K and V bytes at ~46 GB/s (an SM's share
// of HBM) or its MMA work at ~0.35 ns per query-key pair, whichever is longer.
// 16-row groups in boxes of 8 heads of 128 dims whose segments (sequence x
// head box) number at most a quarter of the CTAs, so that each is cut across
// four or more CTA ranges on average: the WC instantiations, 8 blocks (bf16)
// or 12 (e4m3).  There the CTAs whose ranges hold two cut segments (two
// counts, two merges) finish last; per-CTA stamps put them ~2.6 us per extra
// segment behind.  The weights were set by measurement on GB300 (batch 32 of
// 512-4096 keys, 32/8 heads, weights 4 to 12 tried: bf16 63.2 -> 60.7 us at
// 8, e4m3 47.6 -> 45.0 us at 12).  Other shapes cut the units plainly (0).
int decode_segment_penalty(int32_t head_dim, int32_t heads_per_box, int32_t group, bool kv8, int32_t batch,
                           int32_t num_kv_heads, int32_t num_ctas) {
  if (group <= 16) {
    if (head_dim != 128 || heads_per_box != 8) return 0;
    const int64_t segments = (int64_t)batch * (num_kv_heads / heads_per_box);
    return 4 * segments <= num_ctas ? (kv8 ? 12 : 8) : 0;
  }
  const double bytes_ns = 2.0 * 16 * heads_per_box * head_dim * (kv8 ? 1 : 2) / 46.0;
  const double mma_ns = 16.0 * heads_per_box * group * 0.35;
  return (int)(5000.0 / (bytes_ns > mma_ns ? bytes_ns : mma_ns) + 0.5);
}

int64_t decode_partial_slots(int32_t batch, int32_t num_kv_heads, int32_t num_ctas, int32_t heads_per_box) {
  // (segment + CTA) * HB + head over segments (b, head box): B*Hkv + n*HB at most
  return (int64_t)batch * num_kv_heads + (int64_t)num_ctas * heads_per_box;
}

int decode_num_ctas(int num_sms, int32_t batch, int32_t num_kv_heads, int32_t max_seq_len, int32_t heads_per_box) {
  const int64_t ubound = (int64_t)batch * (num_kv_heads / heads_per_box) * (((int64_t)max_seq_len + 15) / 16);
  int64_t n = num_sms;
  if (ubound < n) n = ubound;
  if (n < 1) n = 1;
  return (int)n;
}

size_t decode_smem_bytes(int head_dim, int group, int batch, int heads_per_box, int budget, bool kv8) {
  const int rt = group <= 16 ? 1 : 2;
  Layout L;
#define PA_LAYOUT(DD, HH, RR) \
  L = kv8 ? make_layout<DD, HH, RR, true>(group, batch, budget) : make_layout<DD, HH, RR, false>(group, batch, budget)
  const int key = (head_dim == 128 ? 1000 : 0) + heads_per_box * 10 + rt;
  switch (key) {
    case 1081: PA_LAYOUT(128, 8, 1); break;
    case 1041: PA_LAYOUT(128, 4, 1); break;
    case 1021: PA_LAYOUT(128, 2, 1); break;
    case 1011: PA_LAYOUT(128, 1, 1); break;
    case 1042: PA_LAYOUT(128, 4, 2); break;
    case 1022: PA_LAYOUT(128, 2, 2); break;
    case 1012: PA_LAYOUT(128, 1, 2); break;
    case 81: PA_LAYOUT(64, 8, 1); break;
    case 41: PA_LAYOUT(64, 4, 1); break;
    case 21: PA_LAYOUT(64, 2, 1); break;
    case 11: PA_LAYOUT(64, 1, 1); break;
    case 42: PA_LAYOUT(64, 4, 2); break;
    case 22: PA_LAYOUT(64, 2, 2); break;
    case 12: PA_LAYOUT(64, 1, 2); break;
    default: return (size_t)-1;
  }
#undef PA_LAYOUT
  return L.stages >= 2 ? (size_t)L.total : (size_t)-1;
}

namespace {

cudaError_t launch_split_only(const DecodeParams& p, cudaStream_t s) {
  const int D = p.pool.head_dim;
  const int RT = p.group <= 16 ? 1 : 2;
  const int R = p.pool.page_size < 16 ? p.pool.page_size : 16;
  const int64_t rows = p.pool.num_pages * (int64_t)p.pool.page_size;
  CUtensorMap tk, tv;
  if (p.kv8) {
    if (!encode_pool_tmap_u8(&tk, p.pool.key_pool, rows, p.pool.num_kv_heads, D, R, p.heads_per_box, true) ||
        !encode_pool_tmap_u8(&tv, p.pool.value_pool, rows, p.pool.num_kv_heads, D, R, p.heads_per_box, true))
      return cudaErrorInvalidValue;
    if (p.new_k != nullptr) return launch_split_fused(p, tk, tv, RT, s);
    return D == 128 ? launch_split_d<128, true, false>(p, tk, tv, RT, s)
                    : launch_split_d<64, true, false>(p, tk, tv, RT, s);
  }
  const int box_slabs = R == 16 ? D / 64 : 1;
  if (!encode_pool_tmap(&tk, p.pool.key_pool, rows, p.pool.num_kv_heads, D, R, p.heads_per_box, box_slabs) ||
      !encode_pool_tmap(&tv, p.pool.value_pool, rows, p.pool.num_kv_heads, D, R, p.heads_per_box, box_slabs))
    return cudaErrorInvalidValue;
  if (p.new_k != nullptr) return launch_split_fused(p, tk, tv, RT, s);
  return D == 128 ? launch_split_d<128, false, false>(p, tk, tv, RT, s)
                  : launch_split_d<64, false, false>(p, tk, tv, RT, s);
}

}  // namespace

cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t s) {
  // segments cut across CTAs are merged inside the split kernel
  return launch_split_only(p, s);
}


cudaError_t launch_decode_cascade_bf16(const DecodeParams& p, cudaStream_t s, cudaEvent_t prefix_done) {
  cudaError_t e = launch_split_only(p, s);
  if (e != cudaSuccess) return e;
  e = cudaStreamWaitEvent(s, prefix_done, 0);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_combine_kernel, dim3(p.batch * p.pool.num_kv_heads), dim3(128), 0, s, p, p.pool.head_dim);
}

}  // namespace pa
