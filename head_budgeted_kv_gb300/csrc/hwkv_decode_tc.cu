// Stream-K split-K decode attention over per-head paged rings (block_size % 16 == 0, head_dim
// 64 or 128), optionally fused with the append of the step's new token: tile work on the
// tensor cores for bf16 pools (up to 16 query heads per KV head), on the CUDA cores for fp32
// pools (up to 4).
//
// "HeadWiseKV: Budgeted Per-Head Cache Residency for Hybrid Long-Context Language Models",
// abstract and section "Grouped-Cache Runtime": attention reads only the materialised window
// of each KV head (the last min(w, len) tokens), through the head's block table.
//
// Work decomposition ("stream-K"): every (seq, kv head) group contributes the 16-token ring
// tiles that hold resident tokens -- a cyclic run of tiles starting at the tile of the oldest
// resident slot.  Numbering those tiles group after group gives one line of T equal-cost
// tiles; the persistent grid of N CTAs splits it into N equal contiguous ranges, so every
// CTA streams the same number of bytes whatever the windows and lengths are.  A CTA walks its
// range group by group ("segments"); its 4 warps take the segment's tiles round-robin, each
// through its own TMA + mbarrier pipeline that runs on across segment boundaries.  At the end
// of a segment the warps' online-softmax states are merged in shared memory; a group held by
// one CTA is written out directly, otherwise the CTA stores a partial (m, l, acc) and bumps
// the group's arrival counter, and the CTA that arrives last merges all partials of the group
// and writes the output (no CTA ever waits for another).  After a CTA's last tile its stage
// buffers are free, and a merge there fetches the whole partial block with one bulk copy.
// The sequence lengths are staged in shared memory once, so crossing into the next group
// costs no global round trip.
//
// Per tile (16 tokens), per warp, bf16 (hwkv_decode_tile.cuh, consume_tile), with the GQA
// group (G <= 16 query heads, zero-padded to one or two 8-column n-tiles) on the N side of
// mma.sync.m16n8k16 bf16 -> fp32:
//   S[16 tok][8 q] = K_tile . Q^T over head_dim per n-tile (K tile loaded once with ldmatrix
//   from the 128-byte-swizzled TMA tile and shared by the n-tiles), masked to resident slots,
//   online softmax in fp32 in the log2 domain; P is moved from the accumulator layout to the
//   operand layout with movmatrix.trans; O^T[D][8 q] = alpha * O^T + V_tile^T . P (V tile
//   loaded once with ldmatrix.trans).
// fp32 (consume_tile_f32): lanes own consecutive dims; the tile's 16 x 4 dot products are summed
// over the warp by a butterfly transpose-reduction, P goes through shared memory for the FMAs.
//
// Waits are bounded (~2 s); a timeout records HWKV_DEVERR_WAIT_TIMEOUT and the warp stops.
#include "hwkv_decode_tile.cuh"

namespace hwkv {
namespace {

constexpr int kFlatMerge = 24;  // most contributors one CTA merges directly

// Line positions charged for each group's boundary.  A group with tiles spans kGapTiles
// positions that hold no tile, then its tiles; a CTA whose range takes in a group's start thus
// streams kGapTiles fewer tiles, which pays for what a boundary costs it (the warps' merge,
// publishing a partial, the next group's q), so CTAs with boundaries do not end last.
constexpr int kGapTiles = 24;

// Tiles per warp pulled into L2 while the CTA waits for the preceding grid (early reads only),
// when its range holds at least kL2PrefetchMin positions.  Short ranges (small batches) skip it:
// there the preceding grid's last streams and merges, which the prefetch would slow, are most of
// what the wait is for.  Depth swept on the full geometry with the dependent-launch trigger at
// kernel entry: head_dim 128, 0 -> 957, 2 -> 969, 4 -> 982, 6 -> 989, 8 -> 988 tokens/s; head_dim
// 64 (three CTAs per SM, half the bytes per tile), GQA 4: 0 -> 0.828, 2 -> 0.836, 4 -> 0.819,
// 6 -> 0.807 of the copy peak.
template <int D>
__host__ __device__ constexpr int l2_prefetch() {
  return D == 128 ? 6 : 2;
}
constexpr int kL2PrefetchMin = 64;

__device__ __forceinline__ int group_span(const Group& gr) { return gr.tiles > 0 ? gr.tiles + kGapTiles : 0; }

// Writes a merged (M, L, acc) of query head q, columns 4*d4 .. 4*d4 + 3: normalised to the
// output `out_grp` (bf16 or fp32) when it is non-null, else unnormalised to partial slot `dst_slot`.
template <typename T, int D>
__device__ __forceinline__ void store_merged(float M, float L, float4 acc, int q, int d4, int G, T* out_grp,
                                             float* dst_acc, float* dst_ml, long long dst_slot) {
  if (out_grp != nullptr) {
    const float inv = L > 0.f ? 1.f / L : 0.f;
    if constexpr (sizeof(T) == 4) {
      *reinterpret_cast<float4*>(out_grp + (int64_t)q * D + d4 * 4) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t*>(&lo);
      packed.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(out_grp + (int64_t)q * D + d4 * 4) = packed;
    }
  } else {
    const long long slot = dst_slot * G + q;
    reinterpret_cast<float4*>(dst_acc + slot * D)[d4] = acc;
    if (d4 == 0) reinterpret_cast<float2*>(dst_ml)[slot] = make_float2(M, L);
  }
}
// Folds `count` consecutive partial slots [first, first + count) of a partial buffer out of
// registers, with exactly the arithmetic of the shared-memory merge below: first the maximum
// M = max_i m_i, then, slot after slot, w_i = 2^(m_i - M), L = fma(l_i, w_i, L) and
// acc = fma(acc_i, w_i, acc).  Whichever path a group's last arriver takes, the output is the
// same bit for bit.  Each thread owns 4 consecutive output columns of one query head and keeps
// 8 slots' loads in flight.  Output as store_merged.  `live(i)` tells whether slot first + i
// holds a partial.
template <typename T, int D, typename Live>
__device__ __forceinline__ void merge_slots_regs(const float* src_acc, const float* src_ml, long long first,
                                                 int count, int G, Live live, T* out_grp,
                                                 float* dst_acc, float* dst_ml, long long dst_slot) {
  constexpr int kV = D / 4;  // float4 columns per query head
  constexpr int kBatch = 8;
  for (int e = threadIdx.x; e < G * kV; e += blockDim.x) {
    const int q = e / kV, d4 = e - (e / kV) * kV;
    float M = kNegInf;
    for (int i0 = 0; i0 < count; i0 += kBatch) {
      float m[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j;
        m[j] = i < count && live(i) ? __ldcg(src_ml + ((first + i) * G + q) * 2) : kNegInf;
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) M = fmaxf(M, m[j]);
    }
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < count; i0 += kBatch) {
      float2 ml[kBatch];
      float4 v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j;
        if (i < count && live(i)) {
          const long long slot = (first + i) * G + q;
          ml[j] = __ldcg(reinterpret_cast<const float2*>(src_ml) + slot);
          v[j] = __ldcg(reinterpret_cast<const float4*>(src_acc + slot * D) + d4);
        } else {
          ml[j] = make_float2(kNegInf, 0.f);
          v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (i0 + j < count && live(i0 + j)) {
          const float w = M == kNegInf ? 0.f : ex2(ml[j].x - M);
          L = fmaf(ml[j].y, w, L);
          acc.x = fmaf(v[j].x, w, acc.x);
          acc.y = fmaf(v[j].y, w, acc.y);
          acc.z = fmaf(v[j].z, w, acc.z);
          acc.w = fmaf(v[j].w, w, acc.w);
        }
      }
    }
    store_merged<T, D>(M, L, acc, q, d4, G, out_grp, dst_acc, dst_ml, dst_slot);
  }
}
constexpr uint32_t kBulkChunk = 16384;  // bytes per bulk copy of a partial block

// Shared-memory resources a merge may use: the stage buffers (free once the CTA has consumed
// its last tile), two mbarriers for bulk copies into them and the phases they are at.
struct MergeStage {
  float* buf;               // null: not available
  uint32_t bytes;
  uint64_t* bar0;           // copies into the whole buffer or its first half ...
  uint64_t* bar1;           // ... and into its second half
  uint32_t phase0, phase1;  // completed uses of bar0 / bar1 (uniform in the CTA)
  int stuck0, stuck1;       // parity of a use that may still be in flight after a timeout, else -1
};

// Folds `count` consecutive partial slots [first, first + count) into the output or partial
// slot of store_merged.  When every slot holds a partial (`dense`), the stage buffers are free
// and the accumulators fit them and the (m, l) of every (slot, head) fit `s_ml` (2 * count * G
// <= ml_cap floats), the accumulators are fetched in one bulk copy while those (m, l) are read
// into `s_ml`; each thread then forms its head's maximum M = max_i m_i and, slot after slot,
// w_i = 2^(m_i - M), L = fma(l_i, w_i, L) and the sum of w_i * acc_i over its 4 columns out of
// shared memory (the threads of a warp share a head, so the reads are broadcasts).  The whole
// merge waits for about one round trip to L2.  Otherwise the register merge above runs, with
// the same arithmetic, so an output does not depend on which path its last arriver took.
// `live(i)` tells whether slot first + i holds a partial.
template <typename T, int D, typename Live>
__device__ __forceinline__ void merge_slots_one(const float* src_acc, const float* src_ml, long long first, int count,
                                            int G, Live live, bool dense, T* out_grp, float* dst_acc,
                                            float* dst_ml, long long dst_slot, float* s_ml, int ml_cap,
                                            MergeStage& ms, int32_t* err) {
  const uint32_t bytes = (uint32_t)count * (uint32_t)G * D * 4u;
  if (!dense || ms.buf == nullptr || 2 * count * G > ml_cap || bytes > ms.bytes) {
    merge_slots_regs<T, D>(src_acc, src_ml, first, count, G, live, out_grp, dst_acc, dst_ml, dst_slot);
    return;
  }
  if (threadIdx.x == 0) {
    // the partials were written and acquired, and the buffer last read, through the generic proxy
    fence_proxy_async_all();
    mbar_arrive_expect_tx(ms.bar0, bytes);
    const char* src = reinterpret_cast<const char*>(src_acc + first * G * D);
    for (uint32_t off = 0; off < bytes; off += kBulkChunk)
      bulk_load(smem_addr(ms.buf) + off, src + off, bytes - off < kBulkChunk ? bytes - off : kBulkChunk, ms.bar0);
  }
  for (int p = threadIdx.x; p < count * G; p += blockDim.x) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(src_ml) + first * G + p);
    s_ml[p] = ml.x;
    s_ml[count * G + p] = ml.y;
  }
  __syncthreads();
  const bool landed = mbar_wait_bounded(ms.bar0, ms.phase0 & 1u);
  ++ms.phase0;
  if (!landed && threadIdx.x == 0) atomicOr(err, HWKV_DEVERR_WAIT_TIMEOUT);
  constexpr int kV = D / 4;  // float4 columns per query head
  const float4* sacc = reinterpret_cast<const float4*>(ms.buf);
  for (int e = threadIdx.x; e < G * kV; e += blockDim.x) {
    const int q = e / kV, d4 = e - (e / kV) * kV;
    float M = kNegInf;
    for (int i = 0; i < count; ++i) M = fmaxf(M, s_ml[i * G + q]);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < count; ++i) {
      const float w = M == kNegInf ? 0.f : ex2(s_ml[i * G + q] - M);
      L = fmaf(s_ml[count * G + i * G + q], w, L);
      if (landed) {
        const float4 v = sacc[(i * G + q) * kV + d4];
        acc.x = fmaf(v.x, w, acc.x);
        acc.y = fmaf(v.y, w, acc.y);
        acc.z = fmaf(v.z, w, acc.z);
        acc.w = fmaf(v.w, w, acc.w);
      }
    }
    store_merged<T, D>(M, L, acc, q, d4, G, out_grp, dst_acc, dst_ml, dst_slot);
  }
  if (!landed) {  // a copy may still be in flight: no later merge reuses the buffer
    ms.stuck0 = (int)((ms.phase0 - 1u) & 1u);
    ms.buf = nullptr;
  }
}

// Folds `count` consecutive partial slots [first, first + count) into the output or partial
// slot of store_merged.  When every slot holds a partial (`dense`), the stage buffers are free
// and the accumulators fit them and the (m, l) of every (slot, head) fit `s_ml` (2 * count * G
// <= ml_cap floats), the accumulators are fetched in one bulk copy while those (m, l) are read
// into `s_ml`; each thread then forms its head's maximum M = max_i m_i and, slot after slot,
// w_i = 2^(m_i - M), L = fma(l_i, w_i, L) and the sum of w_i * acc_i over its 4 columns out of
// shared memory (the threads of a warp share a head, so the reads are broadcasts).  The whole
// merge waits for about one round trip to L2.  Accumulators larger than the buffers (large GQA
// groups: 8 KB per partial at 16 query heads) are merged in passes over subsets of the query
// heads, one bulk copy per slot and pass, the next pass landing in one half of the buffers
// while the previous one is summed out of the other.  Otherwise the register merge above runs.
// Every path has the same arithmetic, so an output does not depend on which one its last
// arriver took.  `live(i)` tells whether slot first + i holds a partial.
template <typename T, int D, typename Live>
__device__ __forceinline__ void merge_slots_passes(const float* src_acc, const float* src_ml, long long first, int count,
                                            int G, Live live, bool dense, T* out_grp, float* dst_acc,
                                            float* dst_ml, long long dst_slot, float* s_ml, int ml_cap,
                                            MergeStage& ms, int32_t* err) {
  constexpr int kV = D / 4;  // float4 columns per query head
  const uint32_t bytes = (uint32_t)count * (uint32_t)G * D * 4u;
  const bool one = bytes <= ms.bytes;
  // heads per pass when the accumulators exceed the buffers: the largest power of two dividing
  // G whose pass fits half the buffers and gives every column its own thread
  int hp = one ? G : 0;
  if (!one)
    for (int h = G; h >= 1; h >>= 1)
      if (G % h == 0 && (uint32_t)count * (uint32_t)h * D * 4u <= ms.bytes / 2u && h * kV <= (int)blockDim.x) {
        hp = h;
        break;
      }
  if (!dense || ms.buf == nullptr || 2 * count * G > ml_cap || hp == 0) {
    merge_slots_regs<T, D>(src_acc, src_ml, first, count, G, live, out_grp, dst_acc, dst_ml, dst_slot);
    return;
  }
  const int passes = G / hp;
  const uint32_t pass_bytes = (uint32_t)count * (uint32_t)hp * D * 4u;
  // pass p: heads [p hp, (p + 1) hp) of every slot, into half p % 2 (the whole buffer with one pass)
  auto issue = [&](int p) {
    uint64_t* bar = (p & 1) ? ms.bar1 : ms.bar0;
    // the partials were written and acquired, and the buffer last read, through the generic proxy
    fence_proxy_async_all();
    mbar_arrive_expect_tx(bar, pass_bytes);
    const uint32_t dst = smem_addr(ms.buf) + (uint32_t)(p & 1) * (ms.bytes / 2u);
    if (one) {
      const char* src = reinterpret_cast<const char*>(src_acc + first * G * D);
      for (uint32_t off = 0; off < pass_bytes; off += kBulkChunk)
        bulk_load(dst + off, src + off, pass_bytes - off < kBulkChunk ? pass_bytes - off : kBulkChunk, bar);
    } else {
      const uint32_t row = (uint32_t)hp * D * 4u;
      for (int i = 0; i < count; ++i)
        bulk_load(dst + (uint32_t)i * row, src_acc + ((first + i) * G + (long long)p * hp) * D, row, bar);
    }
  };
  const uint32_t base0 = ms.phase0, base1 = ms.phase1;
  if (threadIdx.x == 0) {
    issue(0);
    if (passes > 1) issue(1);
  }
  for (int p = threadIdx.x; p < count * G; p += blockDim.x) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(src_ml) + first * G + p);
    s_ml[p] = ml.x;
    s_ml[count * G + p] = ml.y;
  }
  __syncthreads();
  ms.phase0 = base0 + (uint32_t)((passes + 1) / 2);
  ms.phase1 = base1 + (uint32_t)(passes / 2);
  // the weighted sum of heads [p hp, (p + 1) hp) out of the buffer half holding pass p
  auto sum_pass = [&](int p, bool landed) {
    const float4* sacc = reinterpret_cast<const float4*>(ms.buf) + (size_t)(p & 1) * (ms.bytes / 32u);
    for (int e = threadIdx.x; e < hp * kV; e += blockDim.x) {
      const int ql = e / kV, d4 = e - (e / kV) * kV;
      const int q = p * hp + ql;
      float M = kNegInf;
      for (int i = 0; i < count; ++i) M = fmaxf(M, s_ml[i * G + q]);
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = 0; i < count; ++i) {
        const float w = M == kNegInf ? 0.f : ex2(s_ml[i * G + q] - M);
        L = fmaf(s_ml[count * G + i * G + q], w, L);
        if (landed) {
          const float4 v = sacc[(i * hp + ql) * kV + d4];
          acc.x = fmaf(v.x, w, acc.x);
          acc.y = fmaf(v.y, w, acc.y);
          acc.z = fmaf(v.z, w, acc.z);
          acc.w = fmaf(v.w, w, acc.w);
        }
      }
      store_merged<T, D>(M, L, acc, q, d4, G, out_grp, dst_acc, dst_ml, dst_slot);
    }
  };
  if (one) {  // every thread waits for the one copy itself: no CTA barrier on the merge chain
    const bool landed = mbar_wait_bounded(ms.bar0, base0 & 1u);
    if (!landed && threadIdx.x == 0) atomicOr(err, HWKV_DEVERR_WAIT_TIMEOUT);
    sum_pass(0, landed);
    if (!landed) {  // a copy may still be in flight: no later merge reuses the buffer
      ms.stuck0 = (int)(base0 & 1u);
      ms.buf = nullptr;
    }
    return;
  }
  bool ok = true;
  for (int p = 0; p < passes; ++p) {
    const int h = p & 1;
    const uint32_t parity = ((h ? base1 : base0) + (uint32_t)(p >> 1)) & 1u;
    ok = __syncthreads_and(ok && mbar_wait_bounded(h ? ms.bar1 : ms.bar0, parity));
    sum_pass(p, ok);
    if (!ok) {  // copies of this and the next pass may still be in flight: no later merge reuses the buffer
      if (threadIdx.x == 0) atomicOr(err, HWKV_DEVERR_WAIT_TIMEOUT);
      const int next = p + 1 < passes ? (int)(((h ? base0 : base1) + (uint32_t)((p + 1) >> 1)) & 1u) : -1;
      if (h) {
        ms.stuck1 = (int)parity;
        ms.stuck0 = next;
      } else {
        ms.stuck0 = (int)parity;
        ms.stuck1 = next;
      }
      ms.buf = nullptr;
      break;
    }
    __syncthreads();  // half h is read: the copy of pass p + 2 may land there
    if (threadIdx.x == 0 && p + 2 < passes) issue(p + 2);
  }
}

// The merge of a group's partials: instances holding 16 query-head columns may meet partials
// larger than the stage buffers and take the head-pass merge; the others the one-copy merge.
template <typename T, int D, int GP, typename Live>
__device__ __forceinline__ void merge_slots(const float* src_acc, const float* src_ml, long long first, int count,
                                            int G, Live live, bool dense, T* out_grp, float* dst_acc,
                                            float* dst_ml, long long dst_slot, float* s_ml, int ml_cap,
                                            MergeStage& ms, int32_t* err) {
  if constexpr (GP == 16)
    merge_slots_passes<T, D>(src_acc, src_ml, first, count, G, live, dense, out_grp, dst_acc, dst_ml, dst_slot, s_ml,
                             ml_cap, ms, err);
  else
    merge_slots_one<T, D>(src_acc, src_ml, first, count, G, live, dense, out_grp, dst_acc, dst_ml, dst_slot, s_ml,
                          ml_cap, ms, err);
}

// Bumps an arrival counter and tells the whole CTA whether it arrived last; the last arriver
// resets the counter to 0 for the next launch.  Call after the CTA's partial is written (by any
// of its threads): the barrier orders those writes before thread 0's atomic, whose release
// half makes them visible device-wide before the count moves, and whose acquire half (with
// the second barrier) lets the last arriver's threads read every other contributor's partial.
__device__ __forceinline__ bool arrive_last(uint32_t* counter, int expected, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    *s_flag = old + 1u == (unsigned)expected;
    if (*s_flag) *counter = 0u;
  }
  __syncthreads();
  return *s_flag != 0;
}

// Query heads whose warp states meet in shared memory per merge pass: a whole 8-column n-tile,
// except at head_dim 128 with 8 or 16 columns, where passes of 4 keep the scratch at 8 KB so two
// CTAs fit an SM.
template <int D, int GP>
__host__ __device__ constexpr int merge_heads() {
  return GP < 8 ? GP : (D == 128 ? 4 : 8);
}

// CTAs per SM: bf16 two at head_dim 128, three at 64 (4 stages of half-size tiles fit three in
// shared memory, and the per-tile instruction chain, twice as long per byte there, needs the
// warps); fp32 tiles are twice the bytes: one at 128, two at 64.
template <typename T, int D>
__host__ __device__ constexpr int sk_min_ctas() {
  return sizeof(T) == 2 ? (D == 64 ? 3 : 2) : (D == 64 ? 2 : 1);
}

template <typename Elem, int D, int GP, int NS>
__global__ void __launch_bounds__(kWarps * 32, sk_min_ctas<Elem, D>())
    decode_sk_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ DecodeArgs a) {
  using State = WarpState<Elem, D, GP>;
  constexpr int W = kWarps;
  constexpr int kEB = (int)sizeof(Elem);
  constexpr int kTileBytes = kTile * D * kEB;  // 16 rows
  constexpr int kStageBytes = 2 * kTileBytes;  // K tile + V tile
  constexpr int NT = State::NT;                // 8-column groups of query heads
  constexpr int SG = merge_heads<D, GP>();      // query heads merged per pass in shared memory
  constexpr int kPasses = GP < 8 ? 1 : 8 / SG;  // passes per 8-column group

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  float* sc_acc = reinterpret_cast<float*>(smem + W * NS * kStageBytes);  // [W][SG][D]
  __shared__ __align__(8) uint64_t bars[W * NS];
  __shared__ float sc_m[W * SG], sc_l[W * SG];
  __shared__ __align__(8) uint64_t merge_bar[2];  // bulk copies of partial blocks
  // the partial merge's (m, l) scratch reuses the warps' merge area: 2 * slots * G floats
  constexpr int kMlCap = W * SG * D;
  __shared__ long long s_scan[W];
  __shared__ long long s_start[2];
  __shared__ int s_last;
  __shared__ int s_lens_buf[kLensCache];
  __shared__ __align__(16) float s_p[kEB == 4 ? W * 64 : 4];  // fp32 tiles: each warp's P

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.pv.kv_heads;
  const int B = a.pv.num_seqs;
  const int ngroups = B * H;
  const int nctas = gridDim.x, cta = blockIdx.x;
  const int G = a.group;
  const int Hq = H * G;
  const int bs = a.pv.block_size;
  Elem* const out = static_cast<Elem*>(a.out);

  // The next grid in the stream may start at once: its CTAs take the slots this grid's CTAs
  // free, run their own early reads, and wait for this grid before anything else (with the
  // trigger at the end of each CTA's stream instead, they started only after the slowest
  // stream: full workload 961 -> 971 tokens/s, batch 1 unchanged).
  griddep_launch_dependents();
  // the descriptor is a kernel parameter, so it may be fetched before the wait below
  if (threadIdx.x == 0) prefetch_tensormap(&tmap);
  // Launched as a programmatic dependent.  By default everything waits for the grids this one
  // depends on.  With a.early the caller guarantees that the lengths, the block table and this
  // layer's pool were written before the preceding grid in the stream started, so the schedule
  // and the first tile loads run before the wait; q, k_new / v_new and every write of this
  // grid come after it.
  if (!a.early) griddep_wait();

  if (cta == 0) {
    for (int s = threadIdx.x; s < B; s += W * 32)
      if (__ldcg(a.lens + s) + a.len_add < 0) atomicOr(a.pv.err, HWKV_DEVERR_NEG_LENGTH);
  }
  // the lengths are staged once, so crossing into the next group never waits on global memory
  const int* s_lens = B <= kLensCache ? s_lens_buf : nullptr;
  if (s_lens != nullptr) {
    for (int s = threadIdx.x; s < B; s += W * 32) s_lens_buf[s] = seq_len(a, s);
    __syncthreads();
  }

  // ---- schedule: needed tiles per group, their prefix sums, this CTA's range ----------
  if (threadIdx.x == 0) s_start[0] = -1;
  const int per = (ngroups + W * 32 - 1) / (W * 32);
  const int g_lo = min(ngroups, (int)threadIdx.x * per), g_hi = min(ngroups, g_lo + per);
  long long mine = 0;
  for (int g = g_lo; g < g_hi; ++g) mine += group_span(load_group(a, s_lens, g));
  long long T;
  const long long excl = block_exclusive_scan<W>(mine, s_scan, T);
  const long long t_lo = range_start(T, cta, nctas), t_hi = range_start(T, cta + 1, nctas);
  if (t_lo < t_hi && excl <= t_lo && t_lo < excl + mine) {
    long long pre = excl;
    for (int g = g_lo; g < g_hi; ++g) {
      const int c = group_span(load_group(a, s_lens, g));
      if (t_lo < pre + c) {
        s_start[0] = g;
        s_start[1] = pre;
        break;
      }
      pre += c;
    }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < W * NS; ++i) mbar_init(&bars[i], 1);
    mbar_init(&merge_bar[0], 1);
    mbar_init(&merge_bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  // the range holds a tile unless it lies within one group's gap
  const bool has_range =
      t_lo < t_hi && s_start[0] >= 0 && t_hi > (t_lo > s_start[1] + kGapTiles ? t_lo : s_start[1] + kGapTiles);
  const int g_start = has_range ? (int)s_start[0] : 0;
  const long long pre_start = has_range ? s_start[1] : 0;

  // ---- per-warp TMA pipeline ---------------------------------------------------------
  uint64_t* wbar = bars + warp * NS;
  const uint32_t wstage = smem_addr(smem + warp * NS * kStageBytes);
  const uint64_t policy = evict_first_policy();

  int ig = g_start;            // issue cursor: group, its first tile on the line, the group
  long long ipre = pre_start;
  Group igr = load_group(a, s_lens, ig);
  long long j_issue = t_lo + warp;
  int issued = 0;
  auto issue_next = [&](int issuer) {
    // this warp's next position that holds a tile: past a group's end go to the next group,
    // within its gap step on; nothing is issued once the range is done
    for (;;) {
      if (j_issue >= t_hi) return;
      if (j_issue >= ipre + group_span(igr)) {
        ipre += group_span(igr);
        igr = load_group(a, s_lens, ++ig);
      } else if (j_issue < ipre + kGapTiles) {
        j_issue += W;
      } else {
        break;
      }
    }
    if (lane == issuer) {
      const int st = issued % NS;
      // the first stages may be issued before the dependent-launch wait: read through L2
      issue_tile<kEB, D>(&tmap, a, igr, tile_slot(igr, j_issue - ipre - kGapTiles), wstage + st * kStageBytes,
                         &wbar[st], policy, issued < NS);
    }
    j_issue += W;
    ++issued;
  };
  // the first stages are issued by different lanes so their table lookups overlap
  if (has_range)
    for (int i = 0; i < NS && j_issue < t_hi; ++i) issue_next(i);
  if (a.early && has_range && lane < l2_prefetch<D>() && t_hi - t_lo >= kL2PrefetchMin) {
    // Until the wait below ends, the preceding grid only merges and completes and the memory
    // system is nearly idle: pull the tiles this warp takes after its staged ones into L2
    // (lane i: the position i steps on; a position inside a gap is skipped).
    const long long p = j_issue + (long long)lane * W;
    if (p < t_hi) {
      int g = ig;
      long long pre = ipre;
      Group gr = igr;
      while (p >= pre + group_span(gr)) {
        pre += group_span(gr);
        gr = load_group(a, s_lens, ++g);
      }
      if (p >= pre + kGapTiles) {
        const int t0 = tile_slot(gr, p - pre - kGapTiles);
        const int jb = t0 / bs;
        const int32_t blk = __ldcg(gr.tbl + jb);
        if (blk >= 0 && (int64_t)blk < a.pv.total_blocks) {
          const char* rows = static_cast<const char*>(a.pv.pool) + ((int64_t)blk * 2 * bs + (t0 - jb * bs)) * D * kEB;
          prefetch_l2_bulk(rows, kTileBytes);                         // K rows of the tile
          prefetch_l2_bulk(rows + (int64_t)bs * D * kEB, kTileBytes);  // V rows
        }
      }
    }
  }
  if (a.early) griddep_wait();
  // groups with nothing resident (length 0) get a zero output, each from one CTA
  for (int g = cta; g < ngroups; g += nctas) {
    const Group gr = load_group(a, s_lens, g);
    if (gr.tiles == 0)
      for (int e = threadIdx.x; e < G * D; e += W * 32)
        store_out<Elem>(out + ((int64_t)gr.s * Hq + gr.h * G + e / D) * D + e % D, 0.f);
  }
  if (!has_range) return;

  int sg = g_start;            // segment cursor (uniform in the CTA)
  long long spre = pre_start;
  Group sgr = load_group(a, s_lens, sg);
  long long j_cons = t_lo + warp;
  int consumed = 0;
  int drain_from = -1;         // set when a wait timed out
  bool patched_stage = false;  // a generic-proxy write went into the stage just released
  MergeStage ms{nullptr, (uint32_t)(W * NS * kStageBytes), &merge_bar[0], &merge_bar[1], 0u, 0u, -1, -1};

  for (;;) {
    // the segment: the group's tiles within the range
    const long long seg_begin = t_lo > spre + kGapTiles ? t_lo : spre + kGapTiles;
    const long long seg_end = t_hi < spre + group_span(sgr) ? t_hi : spre + group_span(sgr);
    // another segment follows when the next group's first tile is within the range
    const bool more = spre + group_span(sgr) + kGapTiles < t_hi;
    while (j_cons < seg_begin) j_cons += W;  // over the group's gap

    State ws;
    ws.begin(a, sgr, G, lane);
    const int new_slot = (a.k_new != nullptr) ? (sgr.len - 1) % sgr.rs.C : -1;

    while (j_cons < seg_end) {
      const int st = consumed % NS;
      if (drain_from < 0 && !mbar_wait_bounded(&wbar[st], (uint32_t)(consumed / NS) & 1u)) {
        drain_from = consumed;
        if (lane == 0) atomicOr(a.pv.err, HWKV_DEVERR_WAIT_TIMEOUT);
      }
      if (drain_from < 0) {
        const uint32_t sK = wstage + st * kStageBytes;
        const int t0 = tile_slot(sgr, j_cons - spre - kGapTiles);
        if (ws.consume(a, sgr, t0, new_slot, sK, sK + kTileBytes, s_p + warp * 64, lane)) patched_stage = true;
      }
      __syncwarp();
      ++consumed;
      if (drain_from < 0 && j_issue < t_hi) {
        if (patched_stage) {  // every lane orders its shared-memory writes before the next TMA
          fence_proxy_async_smem();
          __syncwarp();
        }
        issue_next(0);
      }
      patched_stage = false;
      j_cons += W;
    }

    // ---- end of segment: merge the warps, then store output or partial -----------------
    ws.finish();
    const bool whole = seg_begin == spre + kGapTiles && seg_end == spre + group_span(sgr);
    const long long slot = (long long)sg + cta;  // unique per (group, CTA) along the line
    // pass (nt, hh): the warps' states of query heads [8*nt + hh*SG, 8*nt + (hh+1)*SG) meet in
    // shared memory and are folded into the output or this CTA's partial
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int hh = 0; hh < kPasses; ++hh) {
      if (nt > 0 || hh > 0) __syncthreads();  // the previous pass has read the scratch
      ws.template publish<SG>(nt, hh, warp, lane, sc_m, sc_l, sc_acc);
      __syncthreads();
      const int g0 = 8 * nt + hh * SG;
      const int ng = min(SG, G - g0);  // real query heads of this pass
      for (int e = threadIdx.x; e < ng * D; e += W * 32) {
        const int gl = e / D, d = e - (e / D) * D;
        const int g = g0 + gl;
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, sc_m[w * SG + gl]);
        float Ls = 0.f, A = 0.f;
        if (M != kNegInf) {
#pragma unroll
          for (int w = 0; w < W; ++w) {
            const float f = ex2(sc_m[w * SG + gl] - M);
            Ls += sc_l[w * SG + gl] * f;
            A += sc_acc[(w * SG + gl) * D + d] * f;
          }
        }
        if (whole) {
          store_out<Elem>(out + ((int64_t)sgr.s * Hq + sgr.h * G + g) * D + d, Ls > 0.f ? A / Ls : 0.f);
        } else {
          a.part_acc[(slot * G + g) * D + d] = A;
          if (d == 0) {
            a.part_ml[(slot * G + g) * 2 + 0] = M;
            a.part_ml[(slot * G + g) * 2 + 1] = Ls;
          }
        }
      }
    }
    if (!whole) {
      // The partial is published; count arrivals.  Up to kFlatMerge contributors: the last
      // CTA of the group merges them all.  More (long windows at small batch): blocks of
      // kMergeBlock consecutive contributors are merged by their last arriver into a second-
      // level partial, and the last of those merges the blocks (one level of ~100 partials,
      // streamed through the stage buffers in chunks by one CTA, was slower at batch 1: 877
      // against 955 tokens/s; it moves ~200 KB through one SM where the tree spreads it).
      // After the last segment no copy is in flight (unless a wait timed out): merges may
      // stage partial blocks in the stage buffers.
      if (!more) ms.buf = __syncthreads_or(drain_from >= 0) ? nullptr : reinterpret_cast<float*>(smem);
      const int c_lo = cta_of(spre + kGapTiles, T, nctas), c_hi = cta_of(spre + group_span(sgr) - 1, T, nctas);
      const bool all_live = T >= nctas;  // then no CTA range is empty
      const int k = c_hi - c_lo + 1;
      Elem* const out_grp = out + ((int64_t)sgr.s * Hq + sgr.h * G) * D;
      if (!all_live || k <= kFlatMerge) {
        int expected = k;
        if (!all_live) {
          expected = 0;
          for (int c = c_lo; c <= c_hi; ++c) expected += range_start(T, c + 1, nctas) > range_start(T, c, nctas);
        }
        if (arrive_last(&a.counters[sg], expected, &s_last)) {
          auto live = [&](int i) {
            return all_live || range_start(T, c_lo + i + 1, nctas) > range_start(T, c_lo + i, nctas);
          };
          merge_slots<Elem, D, GP>(a.part_acc, a.part_ml, (long long)sg + c_lo, k, G, live, all_live, out_grp, nullptr,
                         nullptr, 0, sc_acc, kMlCap, ms, a.pv.err);
        }
      } else {
        auto live = [](int) { return true; };
        const int nb = (k + kMergeBlock - 1) / kMergeBlock;
        const int b = (cta - c_lo) / kMergeBlock;
        const int b_lo = c_lo + b * kMergeBlock;
        const int b_n = min(kMergeBlock, c_hi - b_lo + 1);
        const long long slot2 = (long long)sg * a.merge_blocks + b;
        if (arrive_last(&a.counters1[slot2], b_n, &s_last)) {
          merge_slots<Elem, D, GP>(a.part_acc, a.part_ml, (long long)sg + b_lo, b_n, G, live, true, (Elem*)nullptr, a.part2_acc,
                         a.part2_ml, slot2, sc_acc, kMlCap, ms, a.pv.err);
          if (arrive_last(&a.counters[sg], nb, &s_last))
            merge_slots<Elem, D, GP>(a.part2_acc, a.part2_ml, (long long)sg * a.merge_blocks, nb, G, live, true, out_grp,
                           nullptr, nullptr, 0, sc_acc, kMlCap, ms, a.pv.err);
        }
      }
    }
    __syncthreads();  // the merge scratch is rewritten by the next segment
    if (!more) break;
    do {
      spre += group_span(sgr);
      sgr = load_group(a, s_lens, ++sg);
    } while (sgr.tiles == 0);
  }

  if (drain_from >= 0) {
    // let copies still in flight land before the shared memory is released
    for (int c = drain_from; c < issued; ++c)
      if (!mbar_wait_bounded(&wbar[c % NS], (uint32_t)(c / NS) & 1u)) break;
  }
  if (ms.stuck0 >= 0) mbar_wait_bounded(&merge_bar[0], (uint32_t)ms.stuck0);
  if (ms.stuck1 >= 0) mbar_wait_bounded(&merge_bar[1], (uint32_t)ms.stuck1);
}

template <typename T, int D, int GP, int NS>
constexpr int sk_smem_bytes() {
  // stages + merge scratch (merge_heads query heads per pass) + align slack
  return kWarps * NS * (2 * kTile * D * (int)sizeof(T)) + kWarps * merge_heads<D, GP>() * D * 4 + 1024;
}

// pipeline depth: bf16 3 (head_dim 128) or 4 (head_dim 64) stages of 16 tokens per warp; at 64
// the same bytes stay in flight per SM with three CTAs (4 stages: D64 decode 0.75 -> 0.81 of
// the copy peak against 6 stages and two CTAs).  fp32: 3 stages (192 KB at 128, one CTA per
// SM; 96 KB at 64, two).
template <typename T, int D>
constexpr int stages() {
  return sizeof(T) == 2 && D == 64 ? 4 : 3;
}

template <typename T, int D, int GP>
cudaError_t configure_one(int* ctas_per_sm) {
  constexpr int NS = stages<T, D>();
  cudaError_t e = cudaFuncSetAttribute(decode_sk_kernel<T, D, GP, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       sk_smem_bytes<T, D, GP, NS>());
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, decode_sk_kernel<T, D, GP, NS>, kWarps * 32,
                                                       sk_smem_bytes<T, D, GP, NS>());
}

template <typename T, int D, int GP>
cudaError_t launch_one(const DecodeArgs& a, const CUtensorMap* tmap, int ctas, cudaStream_t st) {
  constexpr int NS = stages<T, D>();
  // programmatic dependent launch: the CTAs may become resident while the previous kernel in
  // the stream finishes; they wait for it (griddepcontrol.wait) before reading anything
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = sk_smem_bytes<T, D, GP, NS>();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_sk_kernel<T, D, GP, NS>, *tmap, a);
  count_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D>
cudaError_t configure_dim(int dtype, int ctas_per_sm[kGroupPads]) {
  cudaError_t e;
  if (dtype == HWKV_F32) {  // fp32: one instance, up to 4 query heads per KV head
    ctas_per_sm[1] = ctas_per_sm[2] = 0;
    return configure_one<float, D, 4>(&ctas_per_sm[0]);
  }
  if ((e = configure_one<__nv_bfloat16, D, 4>(&ctas_per_sm[0])) != cudaSuccess) return e;
  if ((e = configure_one<__nv_bfloat16, D, 8>(&ctas_per_sm[1])) != cudaSuccess) return e;
  return configure_one<__nv_bfloat16, D, 16>(&ctas_per_sm[2]);
}

template <typename T, int D>
cudaError_t launch_dim(const DecodeArgs& a, const CUtensorMap* tmap, int ctas, cudaStream_t st) {
  if constexpr (sizeof(T) == 4) {
    return a.group <= 4 ? launch_one<T, D, 4>(a, tmap, ctas, st) : cudaErrorInvalidValue;
  } else {
    switch (decode_tc_group_pad(a.group)) {
      case 4: return launch_one<T, D, 4>(a, tmap, ctas, st);
      case 8: return launch_one<T, D, 8>(a, tmap, ctas, st);
      default: return launch_one<T, D, 16>(a, tmap, ctas, st);
    }
  }
}

}  // namespace

int decode_tc_group_pad(int group) { return group <= 4 ? 4 : group <= 8 ? 8 : 16; }

int decode_tc_pad_index(int group) { return group <= 4 ? 0 : group <= 8 ? 1 : 2; }

cudaError_t configure_decode_tc(int head_dim, int dtype, int ctas_per_sm[kGroupPads]) {
  if (head_dim == 128) return configure_dim<128>(dtype, ctas_per_sm);
  if (head_dim == 64) return configure_dim<64>(dtype, ctas_per_sm);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap* tmap, int ctas, cudaStream_t st) {
  const bool f32 = a.pv.elem_bytes == 4;
  if (a.pv.head_dim == 128) return f32 ? launch_dim<float, 128>(a, tmap, ctas, st) : launch_dim<__nv_bfloat16, 128>(a, tmap, ctas, st);
  if (a.pv.head_dim == 64) return f32 ? launch_dim<float, 64>(a, tmap, ctas, st) : launch_dim<__nv_bfloat16, 64>(a, tmap, ctas, st);
  return cudaErrorInvalidValue;
}

}  // namespace hwkv
