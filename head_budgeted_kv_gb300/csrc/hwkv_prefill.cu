// Chunked prefill over the per-head paged rings: windowed causal attention for a chunk of new
// tokens on the sm_100-family tensor cores (tcgen05, accumulators in tensor memory), then the
// chunk's K/V written into the rings.
//
// "HeadWiseKV: Budgeted Per-Head Cache Residency for Hybrid Long-Context Language Models",
// abstract and section "Grouped-Cache Runtime": each KV head keeps only a static window w of
// its newest tokens.  A new token at position p therefore attends, per KV head, to positions
// [max(0, p + 1 - w), p]: the part before the chunk is read from the head's ring in the pool
// (the last min(w, p0) positions before the chunk start p0), the rest from the chunk's own
// K/V rows.  Appending the chunk then overwrites ring slots that earlier queries of the same
// chunk still read, so the append is a second launch after the attention.
//
// prefill_kernel<D> (bf16, block_size % 16 == 0, head_dim 64 or 128, GQA group 1 <= G <= 16):
//   CTA = (seq, kv head, two query tiles of 128 rows); a tile holds floor(128 / G) tokens x G
//   query heads (row r = token r / G, head r % G; rows past the last whole token idle).  Keys
//   stream in stages of 64 (four 16-token ring or chunk tiles) through a ring of shared-memory
//   stages filled by TMA (pool tiles through the block table, chunk tiles through a tensor map
//   of the chunk).  Warp roles:
//     warp 0      TMA producer (one lane),
//     warp 1      tensor-memory owner; one lane issues S = Q . K^T per stage and query tile
//                 (M 128, N 64, K = D; both operands in shared memory) into tensor memory,
//     warp 2      one lane issues O += P . V (M 128, N = D, K 64; P read from tensor memory,
//                 V from shared memory MN-major), O accumulated in tensor memory (two issuers,
//                 so one's waits for P or for data are covered by the other's queued work),
//     warps 4-7   softmax of query tile 0, warps 8-11 of tile 1: thread i owns row i, loads
//                 its S row from tensor memory, masks it (causal, window, resident slots),
//                 runs the online softmax in fp32 (log2 domain) and writes its P row as bf16
//                 back over the first half of the S columns it came from.
//   S is double-buffered per tile: the S of stage j + 2 is issued once the P . V of stage j,
//   which reads the same columns, has completed.
//   The running maximum used for P is raised only when a row's maximum grows by more than
//   2^8 (then the row of O in tensor memory and its sum are rescaled), so P stays <= 256 and
//   O is rarely touched between stages.  Every wait is bounded (~2 s); a timeout records
//   HWKV_DEVERR_WAIT_TIMEOUT and all roles stop.
#include <algorithm>

#include "hwkv_tcgen05.cuh"

namespace hwkv {
namespace {

constexpr int kPfM = 128;                  // query rows per tile (MMA M)
constexpr int kPfKeys = 64;                // keys per stage (MMA N of S, K of P . V)
constexpr int kPfSub = kPfKeys / kTile;    // ring / chunk tiles per stage
constexpr int kPfThreads = 12 * 32;

template <int D>
struct PfCfg {
  static constexpr int kHalves = D / 64;              // 128-byte column blocks of a row
  static constexpr int kQBytes = kPfM * D * 2;        // one query tile
  static constexpr int kKBytes = kPfKeys * D * 2;     // K (or V) of one stage
  static constexpr int kStageBytes = 2 * kKBytes;
  static constexpr int kStages = D == 128 ? 5 : 8;
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = 2 * kQBytes;
  static constexpr int kSmem = kStageOff + kStages * kStageBytes + 1024;
  // tensor-memory columns: S (then P, in its first 32 columns) of query tile x in buffer b at
  // (2x + b) * 64 (two buffers per tile, so the next stage's S is computed while the softmax
  // works on this one), O of tile x at 256 + x * D
  static constexpr uint32_t kCols = 512;
  static constexpr uint32_t kColO = 4 * kPfKeys;
};

__device__ __forceinline__ void tma_load_2d_l2(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Waits for a phase; gives up when another role has given up (`abort`) or after ~2 s, which
// it records and announces.
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > 2000000000ull) {
        *abort = 1;
        atomicOr(err, HWKV_DEVERR_WAIT_TIMEOUT);
        return false;
      }
    }
  }
}

// The key tiles one CTA streams: first the ring tiles holding the prior context its queries
// may see, then the chunk tiles up to its last query.
struct PfTiles {
  Resident rs;        // resident positions before the chunk
  int prior_first;    // ring tile of the oldest prior position needed
  int prior_tiles;    // number of ring tiles (cyclic from prior_first)
  int C16;
  int p_oldest;       // position held by ring slot rs.first_slot
  int chunk_first;    // chunk rows [16 * chunk_first, ...)
  int chunk_tiles;
};

// How the producer copies one stage (see the producer).
struct PfCopy {
  int mode;          // 0 one pool box, 1 one chunk box, 2 per tile
  int a, b;          // mode 0: row in block, first block; mode 1: first chunk row
  int row[4];        // mode 2: pool row of tile u, or -1 - chunk row
};

// Where the keys of one 16-token tile of the stream come from.
struct PfKeyTile {
  int kind;  // 0 ring, 1 chunk, 2 padding (no keys)
  int a;     // ring: ring distance of the tile's first slot from the oldest resident slot;
             // chunk: chunk row of the tile's first key
};

__device__ __forceinline__ PfKeyTile key_tile(const PfTiles& tl, int t, int C) {
  PfKeyTile k;
  if (t < tl.prior_tiles) {
    int tile = tl.prior_first + t;
    if (tile >= tl.C16) tile -= tl.C16;
    int d = (tile << 4) - tl.rs.first_slot;
    if (d < 0) d += C;
    k.kind = 0;
    k.a = d;
  } else if (t < tl.prior_tiles + tl.chunk_tiles) {
    k.kind = 1;
    k.a = (tl.chunk_first + t - tl.prior_tiles) << 4;
  } else {
    k.kind = 2;
    k.a = 0;
  }
  return k;
}

// Whether every key of stream stage j is visible to every live row of a query tile whose live
// tokens sit at positions [pq_lo, pq_hi]: all four tiles full (resident ring slots or chunk
// rows) and every key position in (pq_hi - w, pq_lo].  Such a stage needs no mask.
__device__ __forceinline__ bool stage_clean(const PfTiles& tl, int j, int C, int p0, int n, int w, int pq_lo,
                                            int pq_hi) {
  bool clean = pq_lo <= pq_hi;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const PfKeyTile kt = key_tile(tl, j * 4 + u, C);
    int k_lo = 0;
    if (kt.kind == 0) {
      clean = clean && kt.a + kTile - 1 < tl.rs.n;
      k_lo = tl.p_oldest + kt.a;
    } else if (kt.kind == 1) {
      clean = clean && kt.a + kTile - 1 < n;
      k_lo = p0 + kt.a;
    } else {
      clean = false;
    }
    clean = clean && k_lo + kTile - 1 <= pq_lo && k_lo > pq_hi - w;
  }
  return clean;
}

// bits lo .. hi (inclusive, clamped to 0 .. 15) of a 16-key tile
__device__ __forceinline__ uint32_t range_bits(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 15);
  return lo > hi ? 0u : ((0xFFFFu >> (15 - hi)) & (0xFFFFu << lo));
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap pool_map,
                                                               const __grid_constant__ CUtensorMap stage_map,
                                                               const __grid_constant__ CUtensorMap knew_map,
                                                               const __grid_constant__ CUtensorMap vnew_map,
                                                               const __grid_constant__ CUtensorMap knew64_map,
                                                               const __grid_constant__ CUtensorMap vnew64_map,
                                                               const __grid_constant__ CUtensorMap q_map,
                                                               const __grid_constant__ PrefillArgs a) {
  using Cfg = PfCfg<D>;
  constexpr int NS = Cfg::kStages;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t kv_full[NS], kv_empty[NS];
  // per query tile x and stage parity b (a phase of each barrier is one stage of that parity,
  // so no waiter can fall two phases behind, which a parity wait could not detect)
  __shared__ __align__(8) uint64_t q_full, s_full[2][2], p_full[2][2], o_done[2][2], o_final[2], drain[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ PfCopy s_copy[32];  // copy plan of the producer's next 32 stages
  // bit jj: stage jj of this CTA needs no mask for query tile x (set by warp 3 ahead of the
  // softmax; a bit not yet set only costs the masked path, which is exact for any stage)
  constexpr int kCleanWords = 48;
  __shared__ uint32_t s_clean[2][kCleanWords];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {  // the TMA descriptors, ahead of their first use
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&stage_map);
    prefetch_tensormap(&pool_map);
    prefetch_tensormap(&knew64_map);
    prefetch_tensormap(&vnew64_map);
    prefetch_tensormap(&knew_map);
    prefetch_tensormap(&vnew_map);
  }
  const int H = a.pv.kv_heads;
  const int G = a.group;
  const int QT = kPfM / G;  // tokens per query tile
  const int Hq = H * G;
  const int bs = a.pv.block_size;

  // work item: heads in the host's order (longest CTAs first), then sequences, tile pairs,
  // then the splits of the pair's key stream
  int hi = 0;
  while (hi + 1 < H && (int)blockIdx.x >= a.head_ctas[hi + 1]) ++hi;
  const int h = a.head_order[hi];
  const int sp = a.splits[hi];
  const int item = ((int)blockIdx.x - a.head_ctas[hi]) / sp;
  const int piece = ((int)blockIdx.x - a.head_ctas[hi]) - item * sp;
  const int s = item / a.q_tiles;
  const int qt = item - s * a.q_tiles;

  const int p0 = a.pos0[s];
  const int n = a.nlen[s];
  if (p0 < 0 || n < 0 || n > a.n_max) {
    if (threadIdx.x == 0 && h == a.head_order[0] && qt == 0) atomicOr(a.pv.err, HWKV_DEVERR_NEG_LENGTH);
    return;
  }
  const int qa = qt * 2 * QT;  // first chunk row of this CTA
  if (qa >= n) return;
  const int qb = min(n, qa + 2 * QT);  // one past the last chunk row
  const int w = a.g.window[h];
  const int C = (a.g.nblk_prefix[h + 1] - a.g.nblk_prefix[h]) * bs;
  const int32_t* tbl = a.pv.tbl + a.g.tbl_base + (int64_t)s * a.g.tbl_seq_stride + a.g.nblk_prefix[h];

  // key tiles: prior positions [lo, p0) with lo = max(0, p0 + qa + 1 - w), chunk rows [clo, qb)
  PfTiles tl;
  tl.rs = resident(p0, w, C);
  tl.C16 = C >> 4;
  tl.p_oldest = p0 - tl.rs.n;
  {
    const int lo = max(0, p0 + qa + 1 - w);
    const int need = p0 - lo;  // prior positions the first query may see (<= rs.n)
    if (need > 0) {
      const int first_slot = lo % C;
      tl.prior_first = first_slot >> 4;
      const uint32_t last = (uint32_t)first_slot + (uint32_t)need - 1u;
      tl.prior_tiles = min(tl.C16, (int)(last >> 4) - tl.prior_first + 1);
    } else {
      tl.prior_first = 0;
      tl.prior_tiles = 0;
    }
    const int clo = max(0, qa + 1 - w);
    tl.chunk_first = clo >> 4;
    tl.chunk_tiles = ((qb - 1) >> 4) - tl.chunk_first + 1;
  }
  const int ntiles = tl.prior_tiles + tl.chunk_tiles;
  const int nst = (ntiles + kPfSub - 1) / kPfSub;
  // the stage holding chunk rows past n, if any (only the stream's last tile can)
  const int vz_stage =
      (tl.chunk_tiles > 0 && ((tl.chunk_first + tl.chunk_tiles) << 4) > n) ? (ntiles - 1) / kPfSub : -1;
  // this CTA's stages [j0, j0 + nloc) of the stream; a split stream leaves a partial per CTA
  const bool split = sp > 1;
  const int j0 = split ? piece * a.split_stages[hi] : 0;
  const int nloc = split ? min(nst, j0 + a.split_stages[hi]) - j0 : nst;
  if (nloc <= 0) {  // nothing of the stream left for this split: an empty partial
    float2* ml = reinterpret_cast<float2*>(a.part_ml) + (size_t)blockIdx.x * 2 * kPfM;
    for (int r = threadIdx.x; r < 2 * kPfM; r += blockDim.x) ml[r] = make_float2(kNegInf, 0.f);
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(&q_full, 1);
    for (int x = 0; x < 2; ++x) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&s_full[x][b], 1);
        mbar_init(&p_full[x][b], 4);
        mbar_init(&o_done[x][b], 1);
      }
      mbar_init(&o_final[x], 1);
    }
    for (int i = 0; i < 2 * kCleanWords; ++i) s_clean[i / kCleanWords][i % kCleanWords] = 0u;
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, Cfg::kCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;
  const uint32_t sbase = smem_addr(smem);
  volatile int* abort = &s_abort;

  if (warp == 0) {
    // ---- TMA producer (whole warp) ----------------------------------------------------
    {
      if (lane == 0) {
        // both query tiles: box of G heads x QT tokens x 64 columns per column block
        mbar_arrive_expect_tx(&q_full, 2 * Cfg::kHalves * QT * G * 128);
        for (int x = 0; x < 2; ++x)
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tma_load_3d(sbase + Cfg::kQOff + x * Cfg::kQBytes + hf * (kPfM * 128), &q_map, hf * 64, h * G,
                        s * a.n_max + qa + x * QT, &q_full);
      }
      int issued = 0;
      // Copy plan of 32 stages at a time, one stage per lane (table lookups and index math in
      // parallel), then lane 0 issues the copies.  mode 0: one 64-key box of the pool per K / V
      // and column block (the ring tiles lie in consecutive blocks as a stage_map box covers
      // them); 1: one 64-row box of the chunk; 2: per 16-row tile (rows: pool row, or -1 - chunk
      // row for a chunk tile).
      for (int c0 = 0; c0 < nloc; c0 += 32) {
        if (__shfl_sync(0xffffffffu, (int)*abort, 0)) break;  // the same decision in every lane
        {
          const int jj = c0 + lane;
          if (jj < nloc) {
            const int j = j0 + jj;
            int kind[kPfSub], blk[kPfSub], r0[kPfSub], row[kPfSub];
            bool blk_ok = true;
#pragma unroll
            for (int u = 0; u < kPfSub; ++u) {
              const int t = j * kPfSub + u;
              kind[u] = t < tl.prior_tiles ? 0 : (t < ntiles ? 1 : 2);
              blk[u] = 0;
              r0[u] = 0;
              if (kind[u] == 0) {
                int tile = tl.prior_first + t;
                if (tile >= tl.C16) tile -= tl.C16;
                const int t0 = tile << 4;
                const int jb = a.bs_log2 >= 0 ? t0 >> a.bs_log2 : t0 / bs;
                blk[u] = __ldg(tbl + jb);
                r0[u] = t0 - jb * bs;
              }
            }
#pragma unroll
            for (int u = 0; u < kPfSub; ++u) {
              if (kind[u] == 0) {
                if (blk[u] < 0 || (int64_t)blk[u] >= a.pv.total_blocks) {
                  atomicOr(a.pv.err, HWKV_DEVERR_BAD_BLOCK);
                  blk[u] = 0;  // keep the barrier accounting intact; the result is flagged
                  blk_ok = false;
                }
                row[u] = blk[u] * 2 * bs + r0[u];
              } else if (kind[u] == 1) {
                row[u] = -1 - ((tl.chunk_first + j * kPfSub + u - tl.prior_tiles) << 4);
              } else {
                row[u] = 0;  // padding: pool row 0 (finite, masked)
              }
            }
            const int tb = a.stage_tb;
            bool ring_stage = tb > 0 && blk_ok && kind[0] == 0 && kind[kPfSub - 1] == 0 && r0[0] + tb <= bs;
#pragma unroll
            for (int u = 1; u < kPfSub; ++u)
              ring_stage = ring_stage && kind[u] == 0 && r0[u] == r0[0] + ((kTile * u) & (tb - 1)) &&
                           blk[u] == blk[0] + (kTile * u) / max(tb, 1);
            const bool chunk_stage = kind[0] == 1 && kind[kPfSub - 1] == 1;
            PfCopy& cp = s_copy[lane];
            cp.mode = ring_stage ? 0 : (chunk_stage ? 1 : 2);
            cp.a = ring_stage ? r0[0] : (chunk_stage ? -1 - row[0] : 0);
            cp.b = ring_stage ? blk[0] : 0;
#pragma unroll
            for (int u = 0; u < kPfSub; ++u) cp.row[u] = row[u];
          }
        }
        __syncwarp();
        if (lane == 0) {
          for (int l = 0; l < 32 && c0 + l < nloc; ++l) {
            const int jj = c0 + l;
            const int st = jj % NS;
            const PfCopy cp = s_copy[l];
            if (jj >= NS && !pf_wait(&kv_empty[st], (uint32_t)((jj / NS) - 1) & 1u, abort, a.pv.err)) break;
            const uint32_t kdst = sbase + Cfg::kStageOff + st * Cfg::kStageBytes;
            const uint32_t vdst = kdst + Cfg::kKBytes;
            mbar_arrive_expect_tx(&kv_full[st], Cfg::kStageBytes);
            if (cp.mode == 0) {
#pragma unroll
              for (int hf = 0; hf < Cfg::kHalves; ++hf) {
                tma_load_3d(kdst + hf * (kPfKeys * 128), &stage_map, hf * 64, cp.a, cp.b, &kv_full[st]);
                tma_load_3d(vdst + hf * (kPfKeys * 128), &stage_map, hf * 64, bs + cp.a, cp.b, &kv_full[st]);
              }
            } else if (cp.mode == 1) {
              const int z = s * a.n_max + cp.a;
#pragma unroll
              for (int hf = 0; hf < Cfg::kHalves; ++hf) {
                tma_load_3d(kdst + hf * (kPfKeys * 128), &knew64_map, hf * 64, h, z, &kv_full[st]);
                tma_load_3d(vdst + hf * (kPfKeys * 128), &vnew64_map, hf * 64, h, z, &kv_full[st]);
              }
            } else {
#pragma unroll
              for (int u = 0; u < kPfSub; ++u) {
#pragma unroll
                for (int hf = 0; hf < Cfg::kHalves; ++hf) {
                  const uint32_t off = hf * (kPfKeys * 128) + u * (kTile * 128);
                  if (cp.row[u] < 0) {
                    const int z = s * a.n_max + (-1 - cp.row[u]);
                    tma_load_3d(kdst + off, &knew_map, hf * 64, h, z, &kv_full[st]);
                    tma_load_3d(vdst + off, &vnew_map, hf * 64, h, z, &kv_full[st]);
                  } else {
                    tma_load_2d_l2(kdst + off, &pool_map, hf * 64, cp.row[u], &kv_full[st]);
                    tma_load_2d_l2(vdst + off, &pool_map, hf * 64, cp.row[u] + bs, &kv_full[st]);
                  }
                }
              }
            }
            ++issued;
          }
        }
        __syncwarp();
      }
      if (lane == 0 && *abort) {  // let the copies in flight land before the shared memory is released
        for (int j = max(0, issued - NS); j < issued; ++j)
          if (!mbar_wait_bounded(&kv_full[j % NS], (uint32_t)(j / NS) & 1u)) break;
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ---- MMA issuers: warp 1 the S of every stage, warp 2 the P . V of every stage ------
    if (lane == 0) {
      constexpr uint32_t idS = umma_idesc_bf16(kPfM, kPfKeys, false, false);
      constexpr uint32_t idO = umma_idesc_bf16(kPfM, D, false, true);
      // Descriptors are built once; an operand's start address moves by adding its offset in
      // 16-byte units to the low field (shared addresses stay below 2^18 bytes, so the
      // 14-bit field does not carry).
      const uint64_t dq = umma_desc_sw128(sbase + Cfg::kQOff, 16, 1024);
      const uint64_t dk = umma_desc_sw128(sbase + Cfg::kStageOff, 16, 1024);
      const uint64_t dv = umma_desc_sw128(sbase + Cfg::kStageOff + Cfg::kKBytes, kPfKeys * 128, 1024);
      bool ok = true;
      if (warp == 1) {
        // S_x = Q_x . K^T of stage j into buffer j % 2, once the P . V of stage j - 2 (which
        // read the P written there) has completed
        ok = pf_wait(&q_full, 0, abort, a.pv.err);
        for (int j = 0; ok && j < nloc; ++j) {
          const int st = j % NS, b = j & 1;
          ok = pf_wait(&kv_full[st], (uint32_t)(j / NS) & 1u, abort, a.pv.err);
          if (!ok) break;
          tc_fence_after_sync();
          const uint64_t dks = dk + (uint64_t)((st * Cfg::kStageBytes) >> 4);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (j >= 2) {
              ok = pf_wait(&o_done[x][b], (uint32_t)((j - 2) >> 1) & 1u, abort, a.pv.err);
              if (!ok) break;
              tc_fence_after_sync();
            }
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
              constexpr int kQRow = kPfM * 128, kKRow = kPfKeys * 128;
              umma_bf16(tmem + (2 * x + b) * kPfKeys,
                        dq + (uint64_t)((x * Cfg::kQBytes + (i >> 2) * kQRow + (i & 3) * 32) >> 4),
                        dks + (uint64_t)(((i >> 2) * kKRow + (i & 3) * 32) >> 4), idS, i > 0 ? 1u : 0u);
            }
            umma_commit(&s_full[x][b]);
          }
        }
      } else {
        // O_x += P_x . V of stage j, once the softmax has written P_x into tensor memory; the
        // stage is free once this completes (its S was complete before P was written)
        for (int j = 0; ok && j < nloc; ++j) {
          const int st = j % NS, b = j & 1;
          const uint64_t dvs = dv + (uint64_t)((st * Cfg::kStageBytes) >> 4);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            ok = pf_wait(&p_full[x][b], (uint32_t)(j >> 1) & 1u, abort, a.pv.err);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t pcol = tmem + (2 * x + b) * kPfKeys;
#pragma unroll
            for (int i = 0; i < kPfKeys / 16; ++i)
              umma_bf16_tmem_a(tmem + Cfg::kColO + x * D, pcol + i * 8, dvs + (uint64_t)((i * 16 * 128) >> 4), idO,
                               (j > 0 || i > 0) ? 1u : 0u);
            umma_commit(&o_done[x][b]);
            if (j == nloc - 1) umma_commit(&o_final[x]);
          }
          if (!ok) break;
          umma_commit(&kv_empty[st]);
        }
      }
      umma_commit(&drain[warp - 1]);  // every MMA this lane issued completes before tensor memory is freed
      mbar_wait_bounded(&drain[warp - 1], 0);
    }
  } else if (warp == 3) {
    // ---- which stages are clean, 32 at a time ------------------------------------------
    int pql[2], pqh[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      pql[x] = p0 + qa + x * QT;
      pqh[x] = p0 + min(n, qa + (x + 1) * QT) - 1;
    }
    for (int c0 = 0; c0 < nloc && c0 < 32 * kCleanWords; c0 += 32) {
      const int jj = c0 + lane;
      const bool in = jj < nloc;
      const bool c_0 = in && stage_clean(tl, j0 + jj, C, p0, n, w, pql[0], pqh[0]);
      const bool c_1 = in && stage_clean(tl, j0 + jj, C, p0, n, w, pql[1], pqh[1]);
      const uint32_t b0 = __ballot_sync(0xffffffffu, c_0), b1 = __ballot_sync(0xffffffffu, c_1);
      if (lane == 0) {
        reinterpret_cast<volatile uint32_t*>(s_clean[0])[c0 >> 5] = b0;
        reinterpret_cast<volatile uint32_t*>(s_clean[1])[c0 >> 5] = b1;
      }
    }
  } else if (warp >= 4) {
    // ---- softmax of query tile x: thread = row ----------------------------------------
    const int x = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row of the tile = tensor-memory lane
    const int tok = qa + x * QT + r / G;
    const bool live = r < QT * G && tok < n;
    const int pq = p0 + tok;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t colO = Cfg::kColO + x * D;
    const float sl2 = a.scale_log2;
    // with a positive scale the row maximum is taken on raw scores and scale-and-subtract is
    // one packed FMA; masked scores become -inf before scaling (+inf for a negative scale)
    const bool pos_scale = sl2 > 0.f;
    const float masked = pos_scale ? kNegInf : -kNegInf;
    float m_ref = kNegInf, l = 0.f;
    bool ok = true;
    // clean-stage bits of stages [32 * k, 32 * k + 32), read once per 32 stages: a shared-memory
    // load waits behind the tensor cores' operand reads (hundreds of cycles while an S product
    // runs), so it is kept off the per-stage path
    uint32_t clean_word = 0u;
    for (int jj = 0; jj < nloc; ++jj) {
      const int j = j0 + jj;  // stage of the stream; jj counts this CTA's stages (barrier phases)
      const int b = jj & 1;
      ok = __all_sync(0xffffffffu, pf_wait(&s_full[x][b], (uint32_t)(jj >> 1) & 1u, abort, a.pv.err));
      if (!ok) break;
      tc_fence_after_sync();
      float sv[kPfKeys];
      tmem_ld64(lane_base + (2 * x + b) * kPfKeys, sv);

      // a "clean" stage needs no mask for any live row (precomputed by warp 3; a bit it has not
      // set yet only costs the masked path, which is exact for any stage)
      if ((jj & 31) == 0)
        clean_word = jj < 32 * kCleanWords ? reinterpret_cast<volatile uint32_t*>(s_clean[x])[jj >> 5] : 0u;
      const bool clean = (clean_word >> (jj & 31)) & 1u;
      if (!clean) {
        PfKeyTile kt[kPfSub];
#pragma unroll
        for (int u = 0; u < kPfSub; ++u) kt[u] = key_tile(tl, j * kPfSub + u, C);
        // visible keys of this row per 16-key tile: position in (pq - w, pq], resident or in
        // the chunk, as intervals of the tile's key index
#pragma unroll
        for (int u = 0; u < kPfSub; ++u) {
          uint32_t vis = 0;
          const int ka = kt[u].a;
          if (kt[u].kind == 0) {
            // ring distance d = ka + i (wrapping at C) holds position p_oldest + d
            const int dlo = max(0, pq - w + 1 - tl.p_oldest), dhi = min(tl.rs.n - 1, pq - tl.p_oldest);
            vis = range_bits(dlo - ka, min(dhi - ka, C - 1 - ka));
            if (ka + kTile > C) vis |= range_bits(max(dlo - ka + C, C - ka), dhi - ka + C);
          } else if (kt[u].kind == 1) {
            vis = range_bits(pq - w + 1 - p0 - ka, min(n - 1 - ka, pq - p0 - ka));
          }
          if (!live) vis = 0;
#pragma unroll
          for (int i = 0; i < kTile; ++i) sv[u * kTile + i] = (vis >> i) & 1u ? sv[u * kTile + i] : masked;
        }
      }
      // row maximum in log2 units
      float mx;
      if (pos_scale) {
        // a tree of three-input maxima (64 -> 22 -> 8 -> 3 -> 1), not a dependent chain
        float t1[22], t2[8], t3[3];
#pragma unroll
        for (int i = 0; i < 21; ++i) t1[i] = fmax3(sv[3 * i], sv[3 * i + 1], sv[3 * i + 2]);
        t1[21] = sv[63];
#pragma unroll
        for (int i = 0; i < 7; ++i) t2[i] = fmax3(t1[3 * i], t1[3 * i + 1], t1[3 * i + 2]);
        t2[7] = t1[21];
        t3[0] = fmax3(t2[0], t2[1], t2[2]);
        t3[1] = fmax3(t2[3], t2[4], t2[5]);
        t3[2] = fmaxf(t2[6], t2[7]);
        const float m3 = fmax3(t3[0], t3[1], t3[2]);
        mx = m3 == kNegInf ? kNegInf : m3 * sl2;
      } else {
        mx = kNegInf;
#pragma unroll
        for (int c = 0; c < kPfKeys; ++c) {
          sv[c] = sv[c] == -kNegInf ? kNegInf : sv[c] * sl2;
          mx = fmaxf(mx, sv[c]);
        }
      }
      const float m_new = fmaxf(m_ref, mx);
      const bool grow = m_new > m_ref + 8.f;
      // O may be rescaled once the previous P . V into it has completed
      if (jj > 0 && __any_sync(0xffffffffu, grow)) {
        ok = __all_sync(0xffffffffu, pf_wait(&o_done[x][(jj - 1) & 1], (uint32_t)((jj - 1) >> 1) & 1u, abort, a.pv.err));
        if (!ok) break;
        tc_fence_after_sync();
        {
          const float f = grow ? ex2(m_ref - m_new) : 1.f;
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            float o[32];
            tmem_ld32(lane_base + colO + c, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= f;
            tmem_st32(lane_base + colO + c, o);
          }
        }
      }
      if (grow) {
        l *= ex2(m_ref - m_new);
        m_ref = m_new;
      }
      const float bm = m_ref == kNegInf ? 0.f : m_ref;

      // V rows past the chunk are zeroed: their P is 0, but 0 times a non-finite value is not.
      // Only the stream's last tile, a chunk tile, can hold such rows.
      if (x == 0 && j == vz_stage) {
        PfKeyTile kt[kPfSub];
#pragma unroll
        for (int u = 0; u < kPfSub; ++u) kt[u] = key_tile(tl, j * kPfSub + u, C);
        {
          ok = __all_sync(0xffffffffu, pf_wait(&kv_full[jj % NS], (uint32_t)(jj / NS) & 1u, abort, a.pv.err));
          if (!ok) break;
          const uint32_t vst = sbase + Cfg::kStageOff + (jj % NS) * Cfg::kStageBytes + Cfg::kKBytes;
#pragma unroll
          for (int u = 0; u < kPfSub; ++u) {
            if (kt[u].kind == 1 && kt[u].a + kTile > n) {
              const int i0 = max(0, n - kt[u].a);
              const int nvec = (kTile - i0) * Cfg::kHalves * 8;
              for (int e = r; e < nvec; e += kPfM) {
                const int rr = i0 + e / (Cfg::kHalves * 8);
                const int rem2 = e % (Cfg::kHalves * 8);
                const uint32_t adr = vst + (rem2 >> 3) * (kPfKeys * 128) + (u * kTile + rr) * 128 + (rem2 & 7) * 16;
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(adr), "r"(0u) : "memory");
              }
            }
          }
          fence_proxy_async_smem();  // before the P . V reads the stage
        }
      }

      // P row (bf16 pairs) over the S columns it came from: p = 2^(s * scale_log2 - m_ref)
      const float2 sl2v = make_float2(pos_scale ? sl2 : 1.f, pos_scale ? sl2 : 1.f);
      const float2 nb = make_float2(-bm, -bm);
      float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      float pk[kPfKeys / 2];
#pragma unroll
      for (int c = 0; c < kPfKeys / 2; ++c) {
        const float2 t = ffma2(make_float2(sv[2 * c], sv[2 * c + 1]), sl2v, nb);
        const float2 pp = make_float2(ex2(t.x), ex2(t.y));
        ls[c & 3] = fadd2(ls[c & 3], pp);
        pk[c] = __uint_as_float(pack_bf16(pp.x, pp.y));
      }
      l += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
      tmem_st32(lane_base + (2 * x + b) * kPfKeys, pk);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[x][b]);
    }
    // the last P . V into O
    if (ok) ok = __all_sync(0xffffffffu, pf_wait(&o_final[x], 0u, abort, a.pv.err));
    if (ok && split) {
      // partial of a split stream: O not normalised, with the row's reference maximum and sum
      tc_fence_after_sync();
      const size_t prow = (size_t)blockIdx.x * 2 * kPfM + x * kPfM + r;
      float* po = a.part_o + prow * D;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        float o[32];
        tmem_ld32(lane_base + colO + c, o);
        if (live) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4*>(po + c + 4 * k) = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        }
      }
      if (live) reinterpret_cast<float2*>(a.part_ml)[prow] = make_float2(m_ref, l);
    } else if (ok) {
      // normalise and store the row
      tc_fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                            (((int64_t)s * a.n_max + (live ? tok : 0)) * Hq + h * G + r % G) * D;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        float o[32];
        tmem_ld32(lane_base + colO + c, o);
        if (live) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16(o[8 * k + 0] * inv, o[8 * k + 1] * inv);
            v.y = pack_bf16(o[8 * k + 2] * inv, o[8 * k + 3] * inv);
            v.z = pack_bf16(o[8 * k + 4] * inv, o[8 * k + 5] * inv);
            v.w = pack_bf16(o[8 * k + 6] * inv, o[8 * k + 7] * inv);
            *reinterpret_cast<uint4*>(orow + c + 8 * k) = v;
          }
        }
      }
    }
  }

  // teardown: every tensor-memory access has completed (loads wait, the issuer drained)
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Cfg::kCols);
  }
}

// Appends the chunk to the rings: chunk row i of (seq, head) is position p0 + i and goes to
// slot (p0 + i) mod C; only the last min(C, n) rows are written (the earlier ones would be
// overwritten by later rows of the same chunk), so every slot is written at most once.
// grid.x: groups of 8 rows, grid.y: seq * H + head; one warp per row.
__global__ void __launch_bounds__(256) chunk_append_kernel(const __grid_constant__ PrefillArgs a, int row_bytes) {
  const int H = a.pv.kv_heads;
  const int s = blockIdx.y / H, h = blockIdx.y - (blockIdx.y / H) * H;
  const int p0 = a.pos0[s], n = a.nlen[s];
  if (p0 < 0 || n < 0 || n > a.n_max) return;  // flagged by the attention kernel
  const int bs = a.pv.block_size;
  const int C = (a.g.nblk_prefix[h + 1] - a.g.nblk_prefix[h]) * bs;
  const int first = n > C ? n - C : 0;
  const int i = first + blockIdx.x * 8 + (threadIdx.x >> 5);
  if (i >= n) return;
  const int lane = threadIdx.x & 31;
  const uint32_t slot = (uint32_t)(p0 + i) % (uint32_t)C;
  const int jb = (int)(slot / (uint32_t)bs);
  const int32_t blk = a.pv.tbl[a.g.tbl_base + (int64_t)s * a.g.tbl_seq_stride + a.g.nblk_prefix[h] + jb];
  if (blk < 0 || (int64_t)blk >= a.pv.total_blocks) {
    if (lane == 0) atomicOr(a.pv.err, HWKV_DEVERR_BAD_BLOCK);
    return;
  }
  char* dk = static_cast<char*>(a.pv.pool) + ((int64_t)blk * 2 * bs + (slot - (uint32_t)jb * bs)) * row_bytes;
  char* dv = dk + (int64_t)bs * row_bytes;
  const int64_t src = (((int64_t)s * a.n_max + i) * H + h) * row_bytes;
  const int nvec = row_bytes / 16;
  for (int v = lane; v < 2 * nvec; v += 32) {
    if (v < nvec) reinterpret_cast<uint4*>(dk)[v] = reinterpret_cast<const uint4*>(static_cast<const char*>(a.k_new) + src)[v];
    else reinterpret_cast<uint4*>(dv)[v - nvec] = reinterpret_cast<const uint4*>(static_cast<const char*>(a.v_new) + src)[v - nvec];
  }
}

// Merges the partials of split key streams: per (seq, head, tile pair) whose stream was split,
// each live row's output is the online-softmax merge of its splits' (O, reference maximum m,
// sum l): out = sum_i O_i 2^(m_i - M) / sum_i l_i 2^(m_i - M), M = max_i m_i.  A CTA takes
// kCombineRows rows of one tile pair and a warp a quarter of those, one row at a time: lane i
// holds split i's (m, l) and split i + 32's, so the maximum is one warp reduction and every
// weight is known before the partial rows (lanes over head_dim) stream in, kCombineAhead splits
// per batch of loads.  The sums run in split order.
constexpr int kCombineRows = 32;
constexpr int kCombineAhead = 8;

template <int C>
struct CombineVec;
template <>
struct CombineVec<4> {
  using T = float4;
};
template <>
struct CombineVec<2> {
  using T = float2;
};

template <int D>
__global__ void __launch_bounds__(256) prefill_combine_kernel(const __grid_constant__ PrefillArgs a) {
  constexpr int kC = D / 32;  // columns per lane
  constexpr int kSlabs = 2 * kPfM / kCombineRows;
  using Vec = typename CombineVec<kC>::T;
  const int per_head = a.pv.num_seqs * a.q_tiles;
  const int unit = blockIdx.x / kSlabs, slab = blockIdx.x - unit * kSlabs;
  const int hi = unit / per_head;
  const int item = unit - hi * per_head;
  const int sp = a.splits[hi];
  if (sp <= 1) return;
  const int h = a.head_order[hi];
  const int s = item / a.q_tiles, qt = item - (item / a.q_tiles) * a.q_tiles;
  const int p0 = a.pos0[s], n = a.nlen[s];
  if (p0 < 0 || n < 0 || n > a.n_max) return;
  const int G = a.group, QT = kPfM / G, Hq = a.pv.kv_heads * G;
  const int qa = qt * 2 * QT;
  if (qa >= n) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t slot0 = (size_t)a.head_ctas[hi] + (size_t)item * sp;
  const float2* part_ml = reinterpret_cast<const float2*>(a.part_ml);
  const size_t split_stride = (size_t)2 * kPfM * D;  // floats from one split's row to the next's
  for (int k = 0; k < kCombineRows / 8; ++k) {
    const int row = slab * kCombineRows + warp * (kCombineRows / 8) + k;
    const int x = row / kPfM, r = row - x * kPfM;
    const int tok = qa + x * QT + r / G;
    if (r >= QT * G || tok >= n) continue;
    float2 e0 = make_float2(kNegInf, 0.f), e1 = e0;
    if (lane < sp) e0 = part_ml[(slot0 + lane) * 2 * kPfM + row];
    if (lane + 32 < sp) e1 = part_ml[(slot0 + lane + 32) * 2 * kPfM + row];
    float M = fmaxf(e0.x, e1.x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f, acc[kC];
#pragma unroll
    for (int c = 0; c < kC; ++c) acc[c] = 0.f;
    if (M != kNegInf) {
      const float f0 = e0.x == kNegInf ? 0.f : ex2(e0.x - M);
      const float f1 = e1.x == kNegInf ? 0.f : ex2(e1.x - M);
      const float* po = a.part_o + (slot0 * 2 * kPfM + row) * D + lane * kC;
      for (int i0 = 0; i0 < sp; i0 += kCombineAhead) {
        Vec v[kCombineAhead];
#pragma unroll
        for (int j = 0; j < kCombineAhead; ++j)
          if (i0 + j < sp) v[j] = *reinterpret_cast<const Vec*>(po + (size_t)(i0 + j) * split_stride);
#pragma unroll
        for (int j = 0; j < kCombineAhead; ++j) {
          const int i = i0 + j;
          if (i >= sp) break;
          const bool lo = i < 32;
          const float mi = __shfl_sync(0xffffffffu, lo ? e0.x : e1.x, i & 31);
          const float li = __shfl_sync(0xffffffffu, lo ? e0.y : e1.y, i & 31);
          const float fi = __shfl_sync(0xffffffffu, lo ? f0 : f1, i & 31);
          if (mi == kNegInf) continue;  // an empty partial
          L = fmaf(li, fi, L);
          const float* vf = reinterpret_cast<const float*>(&v[j]);
#pragma unroll
          for (int c = 0; c < kC; ++c) acc[c] = fmaf(vf[c], fi, acc[c]);
        }
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + (((int64_t)s * a.n_max + tok) * Hq + h * G + r % G) * D;
#pragma unroll
    for (int c = 0; c < kC; c += 2)
      *reinterpret_cast<uint32_t*>(orow + lane * kC + c) = pack_bf16(acc[c] * inv, acc[c + 1] * inv);
  }
}

template <int D>
cudaError_t launch_pf(const PrefillArgs& a, const CUtensorMap* pm, const CUtensorMap* sm, const CUtensorMap* km,
                      const CUtensorMap* vm, const CUtensorMap* km64, const CUtensorMap* vm64, const CUtensorMap* qm,
                      int items, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, PfCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  prefill_kernel<D><<<items, kPfThreads, PfCfg<D>::kSmem, st>>>(*pm, *sm, *km, *vm, *km64, *vm64, *qm, a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

int prefill_tokens_per_cta(int group) { return 2 * (kPfM / group); }

int prefill_max_stages(int window, int ring_capacity, int group, int n_max) {
  // ring tiles: at most the window's (or the ring's) 16-token tiles plus one for alignment;
  // chunk tiles: the pair's tokens plus the window reaching back into the chunk
  const int qt2 = 2 * (kPfM / group);
  const int64_t prior = std::min<int64_t>(ring_capacity / 16, (window + 15) / 16 + 1);
  const int64_t chunk = std::min<int64_t>((n_max + 15) / 16 + 1, (qt2 + (int64_t)window + 15) / 16 + 1);
  return (int)((prior + chunk + kPfSub - 1) / kPfSub);
}

int prefill_tile_tokens(int group) { return kPfM / group; }

int prefill_stages_estimate(int window, int ring_capacity, int group, int n_max, int qa) {
  // the kernel's key tiles (prior positions [lo, p0), chunk rows [clo, qb)) for p0 = 2 C
  const int qt2 = 2 * (kPfM / group);
  const int qb = std::min(n_max, qa + qt2);
  if (qa >= qb) return 0;
  const int64_t C = ring_capacity, p0 = 2 * C;
  const int64_t lo = std::max<int64_t>(0, p0 + qa + 1 - window);
  const int64_t need = p0 - lo;
  int64_t prior = 0;
  if (need > 0) {
    const int64_t first = lo % C;
    prior = std::min<int64_t>(C / 16, (first + need - 1) / 16 - first / 16 + 1);
  }
  const int clo = std::max(0, qa + 1 - window);
  const int64_t chunk = (qb - 1) / 16 - clo / 16 + 1;
  return (int)((prior + chunk + kPfSub - 1) / kPfSub);
}

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap* pool_map, const CUtensorMap* stage_map,
                           const CUtensorMap* knew_map, const CUtensorMap* vnew_map, const CUtensorMap* knew64_map,
                           const CUtensorMap* vnew64_map, const CUtensorMap* q_map, cudaStream_t st) {
  const int items = a.head_ctas[a.pv.kv_heads];
  if (a.group < 1 || a.group > kMaxGroup) return cudaErrorInvalidValue;
  if (a.pv.head_dim == 128)
    return launch_pf<128>(a, pool_map, stage_map, knew_map, vnew_map, knew64_map, vnew64_map, q_map, items, st);
  if (a.pv.head_dim == 64)
    return launch_pf<64>(a, pool_map, stage_map, knew_map, vnew_map, knew64_map, vnew64_map, q_map, items, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_combine(const PrefillArgs& a, cudaStream_t st) {
  // CTAs for the work-order positions up to the last split head (the others return at once)
  int split_heads = 0;
  for (int i = 0; i < a.pv.kv_heads; ++i)
    if (a.splits[i] > 1) split_heads = i + 1;
  const int blocks = split_heads * a.pv.num_seqs * a.q_tiles * (2 * kPfM / kCombineRows);
  if (blocks == 0) return cudaSuccess;
  if (a.pv.head_dim == 128) prefill_combine_kernel<128><<<blocks, 256, 0, st>>>(a);
  else if (a.pv.head_dim == 64) prefill_combine_kernel<64><<<blocks, 256, 0, st>>>(a);
  else return cudaErrorInvalidValue;
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_chunk_append(const PrefillArgs& a, int max_rows, cudaStream_t st) {
  const int row_bytes = a.pv.head_dim * 2;
  const dim3 grid((unsigned)((max_rows + 7) / 8), (unsigned)(a.pv.num_seqs * a.pv.kv_heads));
  chunk_append_kernel<<<grid, 256, 0, st>>>(a, row_bytes);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace hwkv
