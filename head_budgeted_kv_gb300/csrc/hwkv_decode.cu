// Split-K decode attention over per-head paged rings, and the split-K combine.
//
// "HeadWiseKV: Budgeted Per-Head Cache Residency for Hybrid Long-Context Language Models",
// abstract and section "Grouped-Cache Runtime": attention reads only the materialised
// window of each KV head (the last min(w, len) tokens), through the head's block table.
//
// Work decomposition (one launch per layer, static shape so it can be graph-captured):
//   item = (seq s, kv head h, chunk c); chunk c covers ring slots [c*S, min(C, (c+1)*S)),
//   S = split_tokens.  Each CTA streams the resident slots of its chunk once and emits
//   (m, l, acc[D]) per query head of the GQA group: m = running max of scale*log2(e)*<q,k>,
//   l = sum of 2^(score - m), acc = sum of 2^(score - m) * v.  Heads whose ring is one
//   chunk write the normalised output directly; the others are merged by combine_kernel.
//
// Tensor-core kernel (bf16, block_size % 16 == 0, head_dim 64 or 128):
//   - every warp owns NS shared-memory stages of 16 tokens (K tile + V tile) and streams
//     its tiles with TMA (cp.async.bulk.tensor.2d, 128-byte swizzle) completing on an
//     mbarrier; lane 0 re-issues a stage as soon as the warp has consumed it;
//   - the GQA group (G <= 8 query heads, zero-padded to 8) is the N side of
//     mma.sync.m16n8k16 bf16 -> fp32: S[16 tok][8 q] = K_tile . Q^T over D, then
//     O^T[D][8 q] += V_tile^T . P with P moved from the accumulator layout to the operand
//     layout by movmatrix.trans;
//   - online softmax in fp32 in the log2 domain (ex2.approx), warp-shuffle max reduction;
//   - the CTA's warps are merged through shared memory at the end.
// CUDA-core kernel (fp32 pools, or shapes the tensor-core kernel does not take):
//   one token per warp iteration, lanes split head_dim, warp-shuffle dot products.
//
// No wait in this file is unbounded: an mbarrier wait gives up after ~2 s, records
// HWKV_DEVERR_WAIT_TIMEOUT and the warp stops.
#include <cuda_bf16.h>

#include "hwkv_internal.h"
#include "../../include/hwkv.h"

namespace hwkv {
namespace {

constexpr int kTile = 16;          // tokens per mma row tile / per pipeline stage
constexpr float kNegInf = -__builtin_huge_valf();

// ------------------------------------------------------------------------------------
// small PTX helpers
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity; false after ~2 s (never spins forever).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && global_timer_ns() - t0 > 2000000000ull) return false;
  }
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// C[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------------------------
// work items and resident-slot tests
// ------------------------------------------------------------------------------------
struct Item {
  int s, h, c;      // seq, kv head, chunk
  int C, w;         // ring capacity and window of the head
  int nchunks;
};

__device__ __forceinline__ Item decode_item(const DecodeArgs& a, int item) {
  const int per_seq = a.chunk_prefix[a.pv.kv_heads];
  Item it;
  it.s = item / per_seq;
  const int r = item - it.s * per_seq;
  int h = 0;
  while (a.chunk_prefix[h + 1] <= r) ++h;
  it.h = h;
  it.c = r - a.chunk_prefix[h];
  it.nchunks = a.chunk_prefix[h + 1] - a.chunk_prefix[h];
  it.C = (a.g.nblk_prefix[h + 1] - a.g.nblk_prefix[h]) * a.pv.block_size;
  it.w = a.g.window[h];
  return it;
}

// The resident window of a head at length len: the n = min(w, len) newest positions,
// which occupy the n ring slots starting at slot (len - n) mod C (cyclically).
struct Resident {
  int n, first_slot, C;
};

__device__ __forceinline__ Resident resident(int len, int w, int C) {
  Resident r;
  r.n = w < len ? w : len;
  r.first_slot = (len - r.n) % C;
  r.C = C;
  return r;
}

__device__ __forceinline__ bool slot_valid(const Resident& r, int t) {
  int d = t - r.first_slot;
  if (d < 0) d += r.C;
  return d < r.n;
}

// Does the tile of kTile slots starting at t0 (t0 + kTile <= C) hold a resident slot?
__device__ __forceinline__ bool tile_needed(const Resident& r, int t0) {
  if (r.n <= 0) return false;
  int d = t0 - r.first_slot;
  if (d < 0) d += r.C;
  return d < r.n || d > r.C - kTile;
}

template <typename T>
__device__ __forceinline__ void store_out(T* p, float x);
template <>
__device__ __forceinline__ void store_out<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename T>
__device__ __forceinline__ float load_in(const T* p);
template <>
__device__ __forceinline__ float load_in<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_in<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// Merges W per-warp states (smem, canonical layout m/l: [W][8], acc: warp w at acc_of(w),
// [8][D]) and stores either the final output (single-chunk heads) or the item's partial.
template <typename T, int D, int W, typename AccOf>
__device__ __forceinline__ void merge_and_store(const DecodeArgs& a, const Item& it, int item, const float* sm_m,
                                                const float* sm_l, AccOf acc_of) {
  const int G = a.group;
  const int Hq = a.pv.kv_heads * G;
  for (int e = threadIdx.x; e < G * D; e += W * 32) {
    const int g = e / D, d = e - (e / D) * D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, sm_m[w * 8 + g]);
    float Ls = 0.f, A = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float f = ex2(sm_m[w * 8 + g] - M);
        Ls += sm_l[w * 8 + g] * f;
        A += acc_of(w)[g * D + d] * f;
      }
    }
    if (it.nchunks == 1) {
      T* out = static_cast<T*>(a.out) + ((int64_t)it.s * Hq + it.h * G + g) * D + d;
      store_out<T>(out, Ls > 0.f ? A / Ls : 0.f);
    } else {
      a.part_acc[((int64_t)item * G + g) * D + d] = A;
      if (d == 0) {
        a.part_ml[((int64_t)item * G + g) * 2 + 0] = M;
        a.part_ml[((int64_t)item * G + g) * 2 + 1] = Ls;
      }
    }
  }
}

// ------------------------------------------------------------------------------------
// tensor-core kernel
// ------------------------------------------------------------------------------------
// Byte offset of element (row, d) of a 16-row tile loaded as D/64 boxes of [16 rows][64
// elems] with the 128-byte swizzle: box hf = d / 64 at hf * 2048; inside a box, row r is
// the 128-byte line r and its 16-byte chunk c lands at chunk c ^ (r % 8).
__device__ __forceinline__ uint32_t swz(int row, int d) {
  return (uint32_t)((d >> 6) * 2048 + row * 128 + ((((d & 63) >> 3) ^ (row & 7)) << 4) + (d & 7) * 2);
}

template <int D, int W, int NS>
__global__ void __launch_bounds__(W * 32) decode_tc_kernel(const __grid_constant__ CUtensorMap tmap,
                                                           const __grid_constant__ DecodeArgs a) {
  constexpr int kHalves = D / 64;
  constexpr int kTileBytes = kTile * D * 2;          // 16 rows of bf16
  constexpr int kStageBytes = 2 * kTileBytes;        // K tile + V tile
  constexpr int kSteps = D / 16;                     // k-steps of QK, m-tiles of PV
  static_assert(8 * D * 4 <= NS * kStageBytes, "merge scratch must fit in a warp's stages");

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bars[W * NS];
  __shared__ float sm_m[W * 8], sm_l[W * 8];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x;
  const Item it = decode_item(a, item);
  int len = a.lens[it.s];
  if (len < 0) {
    if (threadIdx.x == 0) atomicOr(a.pv.err, HWKV_DEVERR_NEG_LENGTH);
    len = 0;
  }
  const Resident rs = resident(len, it.w, it.C);
  const int bs = a.pv.block_size;
  const int t_begin = it.c * a.split_tokens;
  const int t_end = min(it.C, t_begin + a.split_tokens);
  const int ntiles = (t_end - t_begin) / kTile;
  const int32_t* tbl_row =
      a.pv.tbl + a.g.tbl_base + (int64_t)it.s * a.g.tbl_seq_stride + a.g.nblk_prefix[it.h];

  if (threadIdx.x == 0) {
    for (int i = 0; i < W * NS; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  uint64_t* wbar = bars + warp * NS;
  uint8_t* wstage = smem + warp * NS * kStageBytes;
  const uint32_t wstage_s = smem_addr(wstage);

  // Q of the GQA group as the B operand of S = K . Q^T: lane holds q[g][16i + 2(lane%4) + {0,1}]
  // and the same +8, g = lane/4; rows g >= G are zero.
  const int gq = lane >> 2, q4 = lane & 3;
  const int G = a.group;
  uint32_t qf[kSteps][2];
  {
    const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(a.q) +
                                ((int64_t)it.s * (a.pv.kv_heads * G) + it.h * G + gq) * D;
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {
      if (gq < G) {
        qf[i][0] = *reinterpret_cast<const uint32_t*>(qrow + 16 * i + 2 * q4);
        qf[i][1] = *reinterpret_cast<const uint32_t*>(qrow + 16 * i + 2 * q4 + 8);
      } else {
        qf[i][0] = 0u;
        qf[i][1] = 0u;
      }
    }
  }

  float acc[kSteps][4];
#pragma unroll
  for (int j = 0; j < kSteps; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;   // columns g = 2*q4, 2*q4 + 1
  const float sl2 = a.scale_log2;
  const uint64_t policy = evict_first_policy();

  auto next_needed = [&](int k) {
    while (k < ntiles && !tile_needed(rs, t_begin + k * kTile)) k += W;
    return k;
  };
  auto issue = [&](int k, int st) {  // lane 0 only
    const int t0 = t_begin + k * kTile;
    const int j = t0 / bs;
    const int r0 = t0 - j * bs;
    int32_t blk = tbl_row[j];
    if (blk < 0 || (int64_t)blk >= a.pv.total_blocks) {
      atomicOr(a.pv.err, HWKV_DEVERR_BAD_BLOCK);
      blk = 0;  // keep the barrier accounting intact; the result is flagged as invalid
    }
    const int row_k = blk * 2 * bs + r0;
    const int row_v = row_k + bs;
    const uint32_t dst = wstage_s + st * kStageBytes;
    mbar_arrive_expect_tx(&wbar[st], kStageBytes);
#pragma unroll
    for (int hf = 0; hf < kHalves; ++hf) {
      tma_load_2d(dst + hf * 2048, &tmap, hf * 64, row_k, &wbar[st], policy);
      tma_load_2d(dst + kTileBytes + hf * 2048, &tmap, hf * 64, row_v, &wbar[st], policy);
    }
  };

  int kq = next_needed(warp);
  int issued = 0;
  for (int st = 0; st < NS; ++st) {
    if (kq < ntiles) {
      if (lane == 0) issue(kq, st);
      ++issued;
      kq = next_needed(kq + W);
    }
  }

  // ldmatrix lane roles: matrix mi = lane/8, row rr = lane%8
  const int mi = lane >> 3, rr = lane & 7;
  const int a_row = rr + ((mi & 1) << 3);     // K tile (non-transposed A): token row
  const int a_dof = (mi >> 1) << 3;           //                            +8 dims
  const int v_row = rr + ((mi >> 1) << 3);    // V tile (transposed A): token row
  const int v_dof = (mi & 1) << 3;            //                        +8 dims

  int kc = next_needed(warp);
  int consumed = 0;
  bool timed_out = false;
  while (kc < ntiles) {
    const int st = consumed % NS;
    if (!mbar_wait_bounded(&wbar[st], (uint32_t)(consumed / NS) & 1u)) {
      timed_out = true;
      break;
    }
    const uint32_t sK = wstage_s + st * kStageBytes;
    const uint32_t sV = sK + kTileBytes;

    // S[16 tok][8 q] = K_tile . Q^T (two accumulation chains)
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {
      uint32_t af[4];
      ldsm_x4(af, sK + swz(a_row, 16 * i + a_dof));
      if (i & 1) mma_bf16(sb, af, qf[i][0], qf[i][1]);
      else mma_bf16(sa, af, qf[i][0], qf[i][1]);
    }
    const int t0 = t_begin + kc * kTile;
    const bool v0 = slot_valid(rs, t0 + gq), v1 = slot_valid(rs, t0 + gq + 8);
    const float s0 = v0 ? sa[0] + sb[0] : kNegInf;
    const float s1 = v0 ? sa[1] + sb[1] : kNegInf;
    const float s2 = v1 ? sa[2] + sb[2] : kNegInf;
    const float s3 = v1 ? sa[3] + sb[3] : kNegInf;
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(m0, mx0 * sl2), n1 = fmaxf(m1, mx1 * sl2);
    const float b0 = n0 == kNegInf ? 0.f : n0, b1 = n1 == kNegInf ? 0.f : n1;
    const float al0 = ex2(m0 - b0), al1 = ex2(m1 - b1);
    const float p0 = ex2(fmaf(s0, sl2, -b0)), p1 = ex2(fmaf(s1, sl2, -b1));
    const float p2 = ex2(fmaf(s2, sl2, -b0)), p3 = ex2(fmaf(s3, sl2, -b1));
    l0 = fmaf(l0, al0, p0 + p2);
    l1 = fmaf(l1, al1, p1 + p3);
    m0 = n0;
    m1 = n1;
    const uint32_t pb0 = movmatrix_trans(pack_bf16(p0, p1));
    const uint32_t pb1 = movmatrix_trans(pack_bf16(p2, p3));

    // O^T[D][8 q] = alpha * O^T + V_tile^T . P
#pragma unroll
    for (int j = 0; j < kSteps; ++j) {
      acc[j][0] *= al0;
      acc[j][1] *= al1;
      acc[j][2] *= al0;
      acc[j][3] *= al1;
      uint32_t af[4];
      ldsm_x4_trans(af, sV + swz(v_row, 16 * j + v_dof));
      mma_bf16(acc[j], af, pb0, pb1);
    }

    __syncwarp();
    ++consumed;
    if (kq < ntiles) {
      if (lane == 0) issue(kq, st);
      ++issued;
      kq = next_needed(kq + W);
    }
    kc = next_needed(kc + W);
  }

  if (timed_out) {
    if (lane == 0) atomicOr(a.pv.err, HWKV_DEVERR_WAIT_TIMEOUT);
    // let copies still in flight land before the shared memory is released
    for (int c = consumed; c < issued; ++c) {
      if (!mbar_wait_bounded(&wbar[c % NS], (uint32_t)(c / NS) & 1u)) break;
    }
  }

  // full per-column sums over the 16 token rows held by the 8 lanes of a column
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  float* wacc = reinterpret_cast<float*>(wstage);  // [8][D], own stages are idle now
  if (lane < 4) {
    sm_m[warp * 8 + 2 * q4] = m0;
    sm_m[warp * 8 + 2 * q4 + 1] = m1;
    sm_l[warp * 8 + 2 * q4] = l0;
    sm_l[warp * 8 + 2 * q4 + 1] = l1;
  }
#pragma unroll
  for (int j = 0; j < kSteps; ++j) {
    const int d = 16 * j + gq;
    wacc[(2 * q4) * D + d] = acc[j][0];
    wacc[(2 * q4 + 1) * D + d] = acc[j][1];
    wacc[(2 * q4) * D + d + 8] = acc[j][2];
    wacc[(2 * q4 + 1) * D + d + 8] = acc[j][3];
  }
  __syncthreads();
  merge_and_store<__nv_bfloat16, D, W>(a, it, item, sm_m, sm_l, [&](int w) {
    return reinterpret_cast<const float*>(smem + w * NS * kStageBytes);
  });
}

// ------------------------------------------------------------------------------------
// CUDA-core kernel
// ------------------------------------------------------------------------------------
constexpr int kSimtWarps = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kSimtWarps * 32) decode_simt_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int W = kSimtWarps;
  constexpr int PER = D / 32;
  __shared__ float sm_m[W * 8], sm_l[W * 8];
  __shared__ float sm_acc[W * 8 * D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x;
  const Item it = decode_item(a, item);
  int len = a.lens[it.s];
  if (len < 0) {
    if (threadIdx.x == 0) atomicOr(a.pv.err, HWKV_DEVERR_NEG_LENGTH);
    len = 0;
  }
  const Resident rs = resident(len, it.w, it.C);
  const int bs = a.pv.block_size;
  const int t_begin = it.c * a.split_tokens;
  const int t_end = min(it.C, t_begin + a.split_tokens);
  const int32_t* tbl_row =
      a.pv.tbl + a.g.tbl_base + (int64_t)it.s * a.g.tbl_seq_stride + a.g.nblk_prefix[it.h];
  const int G = a.group;
  const float sl2 = a.scale_log2;

  float qv[kMaxGroup][PER];
  float m[kMaxGroup], l[kMaxGroup], acc[kMaxGroup][PER];
  const T* qbase = static_cast<const T*>(a.q) + ((int64_t)it.s * (a.pv.kv_heads * G) + it.h * G) * D;
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    m[g] = kNegInf;
    l[g] = 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      qv[g][k] = g < G ? load_in<T>(qbase + g * D + lane + 32 * k) : 0.f;
      acc[g][k] = 0.f;
    }
  }

  for (int t = t_begin + warp; t < t_end; t += W) {
    if (!slot_valid(rs, t)) continue;
    const int j = t / bs;
    int32_t blk = tbl_row[j];
    if (blk < 0 || (int64_t)blk >= a.pv.total_blocks) {
      if (lane == 0) atomicOr(a.pv.err, HWKV_DEVERR_BAD_BLOCK);
      continue;
    }
    const T* krow = static_cast<const T*>(a.pv.pool) + ((int64_t)blk * 2 * bs + (t - j * bs)) * D;
    const T* vrow = krow + (int64_t)bs * D;
    float kv[PER], vv[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      kv[k] = load_in<T>(krow + lane + 32 * k);
      vv[k] = load_in<T>(vrow + lane + 32 * k);
    }
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) {
      if (g < G) {
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < PER; ++k) dot = fmaf(qv[g][k], kv[k], dot);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float sc = dot * sl2;
        const float mn = fmaxf(m[g], sc);
        const float al = ex2(m[g] - mn);
        const float p = ex2(sc - mn);
        l[g] = fmaf(l[g], al, p);
#pragma unroll
        for (int k = 0; k < PER; ++k) acc[g][k] = fmaf(acc[g][k], al, p * vv[k]);
        m[g] = mn;
      }
    }
  }

#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    if (lane == 0) {
      sm_m[warp * 8 + g] = m[g];
      sm_l[warp * 8 + g] = l[g];
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) sm_acc[(warp * 8 + g) * D + lane + 32 * k] = acc[g][k];
  }
  __syncthreads();
  merge_and_store<T, D, W>(a, it, item, sm_m, sm_l, [&](int w) { return sm_acc + w * 8 * D; });
}

// ------------------------------------------------------------------------------------
// split-K combine: one CTA per (seq, kv head) whose ring spans several chunks
// ------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ DecodeArgs a) {
  const int H = a.pv.kv_heads;
  const int s = blockIdx.x / H, h = blockIdx.x - (blockIdx.x / H) * H;
  const int nch = a.chunk_prefix[h + 1] - a.chunk_prefix[h];
  if (nch <= 1) return;
  const int G = a.group;
  const int64_t item0 = (int64_t)s * a.chunk_prefix[H] + a.chunk_prefix[h];
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int g = e / D, d = e - (e / D) * D;
    float M = kNegInf;
    for (int c = 0; c < nch; ++c) M = fmaxf(M, a.part_ml[((item0 + c) * G + g) * 2]);
    float Ls = 0.f, A = 0.f;
    if (M != kNegInf) {
      for (int c = 0; c < nch; ++c) {
        const int64_t ig = (item0 + c) * G + g;
        const float f = ex2(a.part_ml[ig * 2] - M);
        Ls += a.part_ml[ig * 2 + 1] * f;
        A += a.part_acc[ig * D + d] * f;
      }
    }
    T* out = static_cast<T*>(a.out) + ((int64_t)s * H * G + h * G + g) * D + d;
    store_out<T>(out, Ls > 0.f ? A / Ls : 0.f);
  }
}

template <int D, int W, int NS>
constexpr int tc_smem_bytes() {
  return W * NS * (2 * kTile * D * 2) + 1024;  // stages + slack to align them to 1024 B
}

template <int D, int W, int NS>
cudaError_t configure_tc() {
  return cudaFuncSetAttribute(decode_tc_kernel<D, W, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              tc_smem_bytes<D, W, NS>());
}

template <int D, int W, int NS>
cudaError_t launch_tc(const DecodeArgs& a, const CUtensorMap* tmap, int items, cudaStream_t st) {
  decode_tc_kernel<D, W, NS><<<items, W * 32, tc_smem_bytes<D, W, NS>(), st>>>(*tmap, a);
  count_launches(1);
  return cudaGetLastError();
}

// tile pipeline shapes: 4 warps per CTA, 3 (D = 128) or 6 (D = 64) stages of 16 tokens per
// warp, ~97 KB of shared memory so that two CTAs share an SM
constexpr int kTcWarps = 4;
constexpr int kTcStages128 = 3;
constexpr int kTcStages64 = 6;

}  // namespace

cudaError_t configure_decode_tc(int head_dim) {
  if (head_dim == 128) return configure_tc<128, kTcWarps, kTcStages128>();
  if (head_dim == 64) return configure_tc<64, kTcWarps, kTcStages64>();
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap* tmap, int items, cudaStream_t st) {
  if (a.pv.head_dim == 128) return launch_tc<128, kTcWarps, kTcStages128>(a, tmap, items, st);
  if (a.pv.head_dim == 64) return launch_tc<64, kTcWarps, kTcStages64>(a, tmap, items, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_simt(const DecodeArgs& a, int dtype, int items, cudaStream_t st) {
  const int D = a.pv.head_dim;
  if (dtype == HWKV_F32 && D == 64) decode_simt_kernel<float, 64><<<items, kSimtWarps * 32, 0, st>>>(a);
  else if (dtype == HWKV_F32 && D == 128) decode_simt_kernel<float, 128><<<items, kSimtWarps * 32, 0, st>>>(a);
  else if (dtype == HWKV_BF16 && D == 64) decode_simt_kernel<__nv_bfloat16, 64><<<items, kSimtWarps * 32, 0, st>>>(a);
  else if (dtype == HWKV_BF16 && D == 128) decode_simt_kernel<__nv_bfloat16, 128><<<items, kSimtWarps * 32, 0, st>>>(a);
  else return cudaErrorInvalidValue;
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_combine(const DecodeArgs& a, int dtype, cudaStream_t st) {
  const int blocks = a.pv.num_seqs * a.pv.kv_heads;
  const int D = a.pv.head_dim;
  if (dtype == HWKV_F32 && D == 64) combine_kernel<float, 64><<<blocks, 256, 0, st>>>(a);
  else if (dtype == HWKV_F32 && D == 128) combine_kernel<float, 128><<<blocks, 256, 0, st>>>(a);
  else if (dtype == HWKV_BF16 && D == 64) combine_kernel<__nv_bfloat16, 64><<<blocks, 256, 0, st>>>(a);
  else if (dtype == HWKV_BF16 && D == 128) combine_kernel<__nv_bfloat16, 128><<<blocks, 256, 0, st>>>(a);
  else return cudaErrorInvalidValue;
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace hwkv
