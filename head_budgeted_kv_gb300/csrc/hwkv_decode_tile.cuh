// Tile-level pieces of the stream-K decode kernel (hwkv_decode_tc.cu): the (seq, kv head) group
// of a step, the ring tiles it needs, the layout of a TMA tile in shared memory, the loads of
// one tile, and the work of one warp on one 16-token tile -- on the tensor cores for bf16
// pools, on the CUDA cores for fp32 pools.
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

// Byte offset of element (row, d) of a 16-row tile of EB-byte elements stored as TMA boxes of
// [16 rows][128 bytes] with the 128-byte swizzle: box hf = d * EB / 128 at hf * 2048; inside a
// box row r is the 128-byte line r and its 16-byte chunk c sits at chunk c ^ (r % 8).
template <int EB>
__device__ __forceinline__ uint32_t swz_e(int row, int d) {
  const int b = d * EB;
  return (uint32_t)((b >> 7) * 2048 + row * 128 + ((((b & 127) >> 4) ^ (row & 7)) << 4) + (b & 15));
}

__device__ __forceinline__ uint32_t swz(int row, int d) { return swz_e<2>(row, d); }

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

// Fused append: when the 16-token tile starting at ring slot t0 holds the new token's slot,
// that row's copy in shared memory (sK / sV, EB-byte elements, 128-byte swizzle) is replaced
// by k_new / v_new and the row is written to the pool; no other CTA reads this tile in the
// launch.  Returns true then (the caller fences before TMA refills the stage).
template <int EB, int D>
__device__ __forceinline__ bool patch_new_row(const DecodeArgs& a, const Group& gr, int t0, int new_slot, uint32_t sK,
                                              uint32_t sV, int lane) {
  if (new_slot < t0 || new_slot >= t0 + kTile) return false;
  constexpr int kRowBytes = D * EB;
  constexpr int kRowVecs = kRowBytes / 16;  // 16-byte vectors per row
  const int bs = a.pv.block_size;
  const int r = new_slot - t0;
  const int jb = new_slot / bs;
  const int32_t blk = gr.tbl[jb];
  const bool blk_ok = blk >= 0 && (int64_t)blk < a.pv.total_blocks;
  const int64_t src = ((int64_t)gr.s * a.pv.kv_heads + gr.h) * kRowBytes;
  char* dstk =
      static_cast<char*>(a.pv.pool) + ((int64_t)(blk_ok ? blk : 0) * 2 * bs + (new_slot - jb * bs)) * kRowBytes;
  for (int i = lane; i < 2 * kRowVecs; i += 32) {
    const int kv = i / kRowVecs, c = i - kv * kRowVecs;
    const uint4 val = *reinterpret_cast<const uint4*>(static_cast<const char*>(kv ? a.v_new : a.k_new) + src + c * 16);
    const uint32_t sa = (kv ? sV : sK) + swz_e<EB>(r, c * (16 / EB));
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sa), "r"(val.x), "r"(val.y), "r"(val.z), "r"(val.w)
                 : "memory");
    if (blk_ok) *reinterpret_cast<uint4*>(dstk + (int64_t)kv * bs * kRowBytes + c * 16) = val;
  }
  __syncwarp();
  return true;
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
  // ldmatrix lane roles: matrix mi = lane/8, row rr = lane%8
  const int mi = lane >> 3, rr = lane & 7;
  const int a_row = rr + ((mi & 1) << 3);   // K tile (non-transposed A operand): token row
  const int a_dof = (mi >> 1) << 3;         //                                    +8 dims
  const int v_row = rr + ((mi >> 1) << 3);  // V tile (transposed A operand): token row
  const int v_dof = (mi & 1) << 3;          //                                +8 dims
  const int gq = lane >> 2;                 // accumulator roles: token/dim row
  const float sl2 = a.scale_log2;

  const bool patched = patch_new_row<2, D>(a, gr, t0, new_slot, sK, sV, lane);

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
// of EB-byte elements into the stage at `dst`, completing on `bar`: D * EB / 128 boxes of
// [16 rows][128 bytes] per K or V tile.  `through_l2`: read the table entry with an L2 load
// (before the dependent-launch wait).  A bad table entry is flagged and block 0 read, so the
// barrier accounting stays intact.
template <int EB, int D>
__device__ __forceinline__ void issue_tile(const CUtensorMap* tmap, const DecodeArgs& a, const Group& gr, int t0,
                                           uint32_t dst, uint64_t* bar, uint64_t policy, bool through_l2) {
  constexpr int kBoxes = D * EB / 128;
  constexpr int kBoxElems = 128 / EB;
  constexpr int kTileBytes = kTile * D * EB;
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
  for (int hf = 0; hf < kBoxes; ++hf) {
    tma_load_2d(dst + hf * 2048, tmap, hf * kBoxElems, row_k, bar, policy);
    tma_load_2d(dst + kTileBytes + hf * 2048, tmap, hf * kBoxElems, row_v, bar, policy);
  }
}

// fp32 query, key and value rows: one warp's work on one 16-token tile of group `gr`, on the
// CUDA cores (fp32 keeps full precision: no tensor-core rounding of the operands).  Lane l holds
// dims [DPL*l, DPL*l + DPL) of every row (DPL = D / 32) and of q and of the accumulator of each
// of the G <= 4 query heads; m, l (log2 units) are kept in every lane.
//   * the 16 x 4 partial dot products of the tile are summed over the 32 lanes by a butterfly
//     that halves the values a lane holds each round (62 shuffles for the tile, not 5 per dot):
//     lane l ends with the scores of token l / 2, heads 2 (l % 2) and 2 (l % 2) + 1;
//   * per head: tile maximum and, after exponentiation, tile sum over the 16 lanes of that
//     parity, the online-softmax update (alpha = 2^(m_old - m_new));
//   * P (16 x 4 fp32) goes through the warp's 64 floats of `p_s`, and O += P^T . V as FMAs.
template <int D>
__device__ __forceinline__ bool consume_tile_f32(const DecodeArgs& a, const Group& gr, int t0, int new_slot,
                                                 uint32_t sK, uint32_t sV, const float (&q)[4][D / 32],
                                                 float (&acc)[4][D / 32], float (&m)[4], float (&l)[4],
                                                 float* p_s, int lane) {
  constexpr int DPL = D / 32;
  const bool patched = patch_new_row<4, D>(a, gr, t0, new_slot, sK, sV, lane);
  float v[64];  // partial <q_g, k_t> over this lane's dims, index t * 4 + g
#pragma unroll
  for (int t = 0; t < kTile; ++t) {
    float k[DPL];
    const uint32_t ad = sK + swz_e<4>(t, lane * DPL);
    if constexpr (DPL == 4) {
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(k[0]), "=f"(k[1]), "=f"(k[2]), "=f"(k[3]) : "r"(ad));
    } else {
      asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(k[0]), "=f"(k[1]) : "r"(ad));
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float d = q[g][0] * k[0];
#pragma unroll
      for (int j = 1; j < DPL; ++j) d = fmaf(q[g][j], k[j], d);
      v[t * 4 + g] = d;
    }
  }
  // butterfly: at distance 16, 8, 4, 2, 1 a lane keeps the lower or upper half of its values
  // (by that bit of its lane index) and adds the partner's copy of the same half
#pragma unroll
  for (int r = 0; r < 5; ++r) {
    const int k = 16 >> r, half = 32 >> r;
    const bool upper = (lane & k) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[half + i];
      const float keep = upper ? v[half + i] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, k);
    }
  }
  const int par = lane & 1;  // this lane's heads: 2 par, 2 par + 1
  const bool valid = slot_valid(gr.rs, t0 + (lane >> 1));
  const float sl2 = a.scale_log2;
  const float s0 = valid ? v[0] * sl2 : kNegInf, s1 = valid ? v[1] * sl2 : kNegInf;
  float x0 = s0, x1 = s1;
#pragma unroll
  for (int off = 2; off < 32; off <<= 1) {
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
  }
  const float y0 = __shfl_xor_sync(0xffffffffu, x0, 1), y1 = __shfl_xor_sync(0xffffffffu, x1, 1);
  const float tmax[4] = {par ? y0 : x0, par ? y1 : x1, par ? x0 : y0, par ? x1 : y1};
  float base[4], alpha[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const float mn = fmaxf(m[g], tmax[g]);
    base[g] = mn == kNegInf ? 0.f : mn;
    alpha[g] = ex2(m[g] - base[g]);
    m[g] = mn;
  }
  const float p0 = ex2(s0 - (par ? base[2] : base[0])), p1 = ex2(s1 - (par ? base[3] : base[1]));
  float u0 = p0, u1 = p1;
#pragma unroll
  for (int off = 2; off < 32; off <<= 1) {
    u0 += __shfl_xor_sync(0xffffffffu, u0, off);
    u1 += __shfl_xor_sync(0xffffffffu, u1, off);
  }
  const float w0 = __shfl_xor_sync(0xffffffffu, u0, 1), w1 = __shfl_xor_sync(0xffffffffu, u1, 1);
  const float tsum[4] = {par ? w0 : u0, par ? w1 : u1, par ? u0 : w0, par ? u1 : w1};
#pragma unroll
  for (int g = 0; g < 4; ++g) l[g] = fmaf(l[g], alpha[g], tsum[g]);
  p_s[2 * lane] = p0;  // index t * 4 + g with t = lane / 2, g = 2 (lane % 2)
  p_s[2 * lane + 1] = p1;
  __syncwarp();
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[g][j] *= alpha[g];
  const uint32_t ps_addr = smem_addr(p_s);
#pragma unroll
  for (int t = 0; t < kTile; ++t) {
    float p[4], vv[DPL];
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(p[0]), "=f"(p[1]), "=f"(p[2]), "=f"(p[3])
                 : "r"(ps_addr + t * 16));
    const uint32_t ad = sV + swz_e<4>(t, lane * DPL);
    if constexpr (DPL == 4) {
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(vv[0]), "=f"(vv[1]), "=f"(vv[2]), "=f"(vv[3])
                   : "r"(ad));
    } else {
      asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(vv[0]), "=f"(vv[1]) : "r"(ad));
    }
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
      for (int j = 0; j < DPL; ++j) acc[g][j] = fmaf(p[g], vv[j], acc[g][j]);
  }
  __syncwarp();  // p_s is rewritten by the next tile
  return patched;
}

// The state one warp carries through a segment, by element type.
template <typename T, int D, int GP>
struct WarpState;

// bf16: the GQA group on the N side of mma.sync (GP columns in 8-column n-tiles), fp32
// accumulators in the mma layout; ls holds this lane's partial row sums until finish().
template <int D, int GP>
struct WarpState<__nv_bfloat16, D, GP> {
  static constexpr int NT = (GP + 7) / 8;
  static constexpr int kEB = 2;
  uint32_t qf[NT][D / 16][2];
  float acc[D / 16][NT][4];
  float mx[NT][2], ls[NT][2];

  __device__ __forceinline__ void begin(const DecodeArgs& a, const Group& gr, int G, int lane) {
    load_q_frags<D, NT>(a, gr, G, lane, qf);
#pragma unroll
    for (int j = 0; j < D / 16; ++j)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[j][nt][0] = acc[j][nt][1] = acc[j][nt][2] = acc[j][nt][3] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mx[nt][0] = mx[nt][1] = kNegInf, ls[nt][0] = ls[nt][1] = 0.f;
  }
  __device__ __forceinline__ bool consume(const DecodeArgs& a, const Group& gr, int t0, int new_slot, uint32_t sK,
                                          uint32_t sV, float*, int lane) {
    return consume_tile<D, NT>(a, gr, t0, new_slot, sK, sV, qf, acc, mx, ls, lane);
  }
  __device__ __forceinline__ void finish() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        ls[nt][0] += __shfl_xor_sync(0xffffffffu, ls[nt][0], off);
        ls[nt][1] += __shfl_xor_sync(0xffffffffu, ls[nt][1], off);
      }
  }
  // this warp's states of query heads [8 nt + hh SG, 8 nt + (hh + 1) SG) into the merge scratch
  template <int SG>
  __device__ __forceinline__ void publish(int nt, int hh, int warp, int lane, float* sc_m, float* sc_l,
                                          float* sc_acc) const {
    const int gq = lane >> 2, q4 = lane & 3;
    const int c0 = 2 * q4 - hh * SG;  // this lane's first column within the pass
    if (c0 < 0 || c0 >= SG) return;
    if (gq == 0) {
      sc_m[warp * SG + c0] = mx[nt][0];
      sc_m[warp * SG + c0 + 1] = mx[nt][1];
      sc_l[warp * SG + c0] = ls[nt][0];
      sc_l[warp * SG + c0 + 1] = ls[nt][1];
    }
    float* wacc = sc_acc + warp * SG * D;
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      const int d = 16 * j + gq;
      wacc[c0 * D + d] = acc[j][nt][0];
      wacc[(c0 + 1) * D + d] = acc[j][nt][1];
      wacc[c0 * D + d + 8] = acc[j][nt][2];
      wacc[(c0 + 1) * D + d + 8] = acc[j][nt][3];
    }
  }
};

// fp32: CUDA-core tile work (consume_tile_f32), up to 4 query heads.
template <int D, int GP>
struct WarpState<float, D, GP> {
  static_assert(GP == 4, "fp32 tile decode holds 4 query-head columns");
  static constexpr int NT = 1;
  static constexpr int kEB = 4;
  static constexpr int DPL = D / 32;
  float q[4][DPL], acc[4][DPL], m[4], l[4];

  __device__ __forceinline__ void begin(const DecodeArgs& a, const Group& gr, int G, int lane) {
    const int Hq = a.pv.kv_heads * G;
    const float* qrow = static_cast<const float*>(a.q) + ((int64_t)gr.s * Hq + gr.h * G) * D + lane * DPL;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
#pragma unroll
      for (int j = 0; j < DPL; ++j) {
        q[g][j] = g < G ? qrow[g * D + j] : 0.f;
        acc[g][j] = 0.f;
      }
      m[g] = kNegInf;
      l[g] = 0.f;
    }
  }
  __device__ __forceinline__ bool consume(const DecodeArgs& a, const Group& gr, int t0, int new_slot, uint32_t sK,
                                          uint32_t sV, float* p_s, int lane) {
    return consume_tile_f32<D>(a, gr, t0, new_slot, sK, sV, q, acc, m, l, p_s, lane);
  }
  __device__ __forceinline__ void finish() {}
  template <int SG>
  __device__ __forceinline__ void publish(int, int, int warp, int lane, float* sc_m, float* sc_l,
                                          float* sc_acc) const {
    static_assert(SG == 4, "one merge pass of 4 query heads");
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        sc_m[warp * SG + g] = m[g];
        sc_l[warp * SG + g] = l[g];
      }
    }
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
      for (int j = 0; j < DPL; ++j) sc_acc[(warp * SG + g) * D + lane * DPL + j] = acc[g][j];
  }
};

}  // namespace
}  // namespace hwkv
