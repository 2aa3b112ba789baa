// Tile-level pieces of the tensor-core decode kernel (hwkv_decode_tc.cu): the (seq, kv head)
// group of a step, the ring tiles it needs, the layout of a TMA tile in shared memory, the
// loads of one tile, and the work of one warp on one 16-token tile.
//
// "HeadWiseKV: Budgeted Per-Head Cache Residency for Hybrid Long-Context Language Models",
// abstract and section "Grouped-Cache Runtime": attention reads only the materialised window
// of each KV head (the last min(w, len) tokens) through the head's block table.
#pragma once

#include "hwkv_device.cuh"

namespace hwkv {
namespace {

constexpr int kWarps = 4;

// One (seq, kv head) group at this step: its resident window and needed tiles.
struct Group {
  int s, h;
  int len;         // length after the append
  Resident rs;     // resident slots
  int C16;         // ring capacity in tiles
  int t_first;     // tile of the oldest resident slot
  int tiles;       // needed tiles, cyclically from t_first
  const int32_t* tbl;
};

constexpr int kLensCache = 256;  // sequence lengths a CTA stages in shared memory

// length of sequence s after the append, clamped at 0
__device__ __forceinline__ int seq_len(const DecodeArgs& a, int s) {
  const int len = __ldcg(a.lens + s) + a.len_add;  // L2: may be read before the dependent-launch wait
  return len < 0 ? 0 : len;
}

// Group g; its sequence length comes from `s_lens` (shared memory) when that is non-null.
__device__ __forceinline__ Group load_group(const DecodeArgs& a, const int* s_lens, int g) {
  Group gr;
  const int H = a.pv.kv_heads;
  gr.s = g / H;
  gr.h = g - gr.s * H;
  gr.len = s_lens != nullptr ? s_lens[gr.s] : seq_len(a, gr.s);
  const int C = (a.g.nblk_prefix[gr.h + 1] - a.g.nblk_prefix[gr.h]) * a.pv.block_size;
  gr.rs = resident(gr.len, a.g.window[gr.h], C);
  gr.C16 = C >> 4;
  gr.t_first = gr.rs.first_slot >> 4;
  if (gr.rs.n > 0) {
    const uint32_t last = (uint32_t)gr.rs.first_slot + (uint32_t)gr.rs.n - 1u;
    gr.tiles = min(gr.C16, (int)(last >> 4) - gr.t_first + 1);
  } else {
    gr.tiles = 0;
  }
  gr.tbl = a.pv.tbl + a.g.tbl_base + (int64_t)gr.s * a.g.tbl_seq_stride + a.g.nblk_prefix[gr.h];
  return gr;
}

// ring slot of the first token of the i-th needed tile of a group
__device__ __forceinline__ int tile_slot(const Group& gr, long long i) {
  int t = gr.t_first + (int)i;
  if (t >= gr.C16) t -= gr.C16;
  return t << 4;
}

// first item of part c when T items are split over n parts
__device__ __forceinline__ long long range_start(long long T, int c, int n) { return T * c / n; }

// part whose range holds item t
__device__ __forceinline__ int cta_of(long long t, long long T, int n) { return (int)(((t + 1) * n - 1) / T); }

// Byte offset of element (row, d) of a 16-row tile stored as D/64 TMA boxes of [16 rows][64
// elements] with the 128-byte swizzle: box hf = d / 64 at hf * 2048; inside a box row r is
// the 128-byte line r and its 16-byte chunk c sits at chunk c ^ (r % 8).
__device__ __forceinline__ uint32_t swz(int row, int d) {
  return (uint32_t)((d >> 6) * 2048 + row * 128 + ((((d & 63) >> 3) ^ (row & 7)) << 4) + (d & 7) * 2);
}

template <int W>
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* s_warp, long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  long long base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    const long long sw = s_warp[w];
    if (w < warp) base += sw;
    tot += sw;
  }
  total = tot;
  __syncthreads();
  return base + x - v;
}

// Q of group `gr` as the B operand of S = K . Q^T: in n-tile nt the lane holds
// q[g][16i + 2*q4 + {0,1}] and the same +8, g = 8*nt + lane/4; heads g >= G are zero.
template <int D, int NT>
__device__ __forceinline__ void load_q_frags(const DecodeArgs& a, const Group& gr, int G, int lane,
                                             uint32_t (&qf)[NT][D / 16][2]) {
  const int gq = lane >> 2, q4 = lane & 3;
  const int Hq = a.pv.kv_heads * G;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int g = 8 * nt + gq;
    const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(a.q) + ((int64_t)gr.s * Hq + gr.h * G + g) * D;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      qf[nt][i][0] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * i + 2 * q4) : 0u;
      qf[nt][i][1] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * i + 2 * q4 + 8) : 0u;
    }
  }
}

// One warp's work on one 16-token tile of group `gr` whose first token sits in ring slot t0,
// staged at sK (K rows) and sV (V rows):
//   * fused append: when the tile holds the new token's slot, that row's copy in shared memory
//     is replaced by k_new / v_new and the row is written to the pool (no other CTA reads this
//     tile in the launch); returns true then (the caller fences before TMA refills the stage);
//   * S[16 tok][8 q] = K_tile . Q^T per n-tile (two accumulation chains), masked to resident
//     slots, online softmax in fp32 in the log2 domain;
//   * O^T[D][8 q] = alpha * O^T + V_tile^T . P per n-tile.
template <int D, int NT>
__device__ __forceinline__ bool consume_tile(const DecodeArgs& a, const Group& gr, int t0, int new_slot,
                                             uint32_t sK, uint32_t sV, const uint32_t (&qf)[NT][D / 16][2],
                                             float (&acc)[D / 16][NT][4], float (&mx)[NT][2], float (&ls)[NT][2],
                                             int lane) {
  constexpr int kSteps = D / 16;
  constexpr int kRowVecs = D * 2 / 16;  // 16-byte vectors per row
  const int bs = a.pv.block_size;
  const int H = a.pv.kv_heads;
  // ldmatrix lane roles: matrix mi = lane/8, row rr = lane%8
  const int mi = lane >> 3, rr = lane & 7;
  const int a_row = rr + ((mi & 1) << 3);   // K tile (non-transposed A operand): token row
  const int a_dof = (mi >> 1) << 3;         //                                    +8 dims
  const int v_row = rr + ((mi >> 1) << 3);  // V tile (transposed A operand): token row
  const int v_dof = (mi & 1) << 3;          //                                +8 dims
  const int gq = lane >> 2;                 // accumulator roles: token/dim row
  const float sl2 = a.scale_log2;

  bool patched = false;
  if (new_slot >= t0 && new_slot < t0 + kTile) {
    const int r = new_slot - t0;
    const int jb = new_slot / bs;
    const int32_t blk = gr.tbl[jb];
    const bool blk_ok = blk >= 0 && (int64_t)blk < a.pv.total_blocks;
    const int64_t src = ((int64_t)gr.s * H + gr.h) * D * 2;
    char* dstk = static_cast<char*>(a.pv.pool) + ((int64_t)(blk_ok ? blk : 0) * 2 * bs + (new_slot - jb * bs)) * D * 2;
    for (int i = lane; i < 2 * kRowVecs; i += 32) {
      const int kv = i / kRowVecs, c = i - kv * kRowVecs;
      const uint4 val =
          *reinterpret_cast<const uint4*>(static_cast<const char*>(kv ? a.v_new : a.k_new) + src + c * 16);
      const uint32_t sa = (kv ? sV : sK) + swz(r, c * 8);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sa), "r"(val.x), "r"(val.y), "r"(val.z),
                   "r"(val.w)
                   : "memory");
      if (blk_ok) *reinterpret_cast<uint4*>(dstk + (int64_t)kv * bs * D * 2 + c * 16) = val;
    }
    __syncwarp();
    patched = true;
  }

  float sa[NT][4], sb[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) sa[nt][e] = sb[nt][e] = 0.f;
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    uint32_t af[4];
    ldsm_x4(af, sK + swz(a_row, 16 * i + a_dof));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (i & 1) mma_bf16(sb[nt], af, qf[nt][i][0], qf[nt][i][1]);
      else mma_bf16(sa[nt], af, qf[nt][i][0], qf[nt][i][1]);
    }
  }
  const bool v0 = slot_valid(gr.rs, t0 + gq), v1 = slot_valid(gr.rs, t0 + gq + 8);
  float al[NT][2];
  uint32_t pb[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float s0 = v0 ? sa[nt][0] + sb[nt][0] : kNegInf;
    const float s1 = v0 ? sa[nt][1] + sb[nt][1] : kNegInf;
    const float s2 = v1 ? sa[nt][2] + sb[nt][2] : kNegInf;
    const float s3 = v1 ? sa[nt][3] + sb[nt][3] : kNegInf;
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(mx[nt][0], mx0 * sl2), n1 = fmaxf(mx[nt][1], mx1 * sl2);
    const float b0 = n0 == kNegInf ? 0.f : n0, b1 = n1 == kNegInf ? 0.f : n1;
    al[nt][0] = ex2(mx[nt][0] - b0);
    al[nt][1] = ex2(mx[nt][1] - b1);
    const float p0 = ex2(fmaf(s0, sl2, -b0)), p1 = ex2(fmaf(s1, sl2, -b1));
    const float p2 = ex2(fmaf(s2, sl2, -b0)), p3 = ex2(fmaf(s3, sl2, -b1));
    ls[nt][0] = fmaf(ls[nt][0], al[nt][0], p0 + p2);
    ls[nt][1] = fmaf(ls[nt][1], al[nt][1], p1 + p3);
    mx[nt][0] = n0;
    mx[nt][1] = n1;
    pb[nt][0] = movmatrix_trans(pack_bf16(p0, p1));
    pb[nt][1] = movmatrix_trans(pack_bf16(p2, p3));
  }

#pragma unroll
  for (int j = 0; j < kSteps; ++j) {
    uint32_t af[4];
    ldsm_x4_trans(af, sV + swz(v_row, 16 * j + v_dof));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      acc[j][nt][0] *= al[nt][0];
      acc[j][nt][1] *= al[nt][1];
      acc[j][nt][2] *= al[nt][0];
      acc[j][nt][3] *= al[nt][1];
      mma_bf16(acc[j][nt], af, pb[nt][0], pb[nt][1]);
    }
  }
  return patched;
}

// Issues the TMA loads of one 16-token tile (K rows and V rows of ring slot t0 of group `gr`)
// into the stage at `dst`, completing on `bar`.  `through_l2`: read the table entry with an
// L2 load (before the dependent-launch wait).  A bad table entry is flagged and block 0 read,
// so the barrier accounting stays intact.
template <int D>
__device__ __forceinline__ void issue_tile(const CUtensorMap* tmap, const DecodeArgs& a, const Group& gr, int t0,
                                           uint32_t dst, uint64_t* bar, uint64_t policy, bool through_l2) {
  constexpr int kHalves = D / 64;
  constexpr int kTileBytes = kTile * D * 2;
  const int bs = a.pv.block_size;
  const int jb = t0 / bs;
  const int r0 = t0 - jb * bs;
  int32_t blk = through_l2 ? __ldcg(gr.tbl + jb) : gr.tbl[jb];
  if (blk < 0 || (int64_t)blk >= a.pv.total_blocks) {
    atomicOr(a.pv.err, HWKV_DEVERR_BAD_BLOCK);
    blk = 0;
  }
  const int row_k = blk * 2 * bs + r0;
  const int row_v = row_k + bs;
  mbar_arrive_expect_tx(bar, 2 * kTileBytes);
#pragma unroll
  for (int hf = 0; hf < kHalves; ++hf) {
    tma_load_2d(dst + hf * 2048, tmap, hf * 64, row_k, bar, policy);
    tma_load_2d(dst + kTileBytes + hf * 2048, tmap, hf * 64, row_v, bar, policy);
  }
}

}  // namespace
}  // namespace hwkv
