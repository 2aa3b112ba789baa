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
//     warp 1      tensor-memory owner and MMA issuer (one lane): per stage and query tile
//                 S = Q . K^T (M 128, N 64, K = D) into tensor memory, and O += P . V
//                 (M 128, N = D, K 64; V read MN-major) accumulated in tensor memory,
//     warps 4-7   softmax of query tile 0, warps 8-11 of tile 1: thread i owns row i, loads
//                 its S row from tensor memory, masks it (causal, window, resident slots),
//                 runs the online softmax in fp32 (log2 domain) and writes its P row as bf16
//                 to shared memory in the 128-byte-swizzled K-major layout the MMA reads.
//   The running maximum used for P is raised only when a row's maximum grows by more than
//   2^8 (then the row of O in tensor memory and its sum are rescaled), so P stays <= 256 and
//   O is rarely touched between stages.  Every wait is bounded (~2 s); a timeout records
//   HWKV_DEVERR_WAIT_TIMEOUT and all roles stop.
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
  static constexpr int kStages = D == 128 ? 4 : 6;
  static constexpr int kPBytes = kPfM * kPfKeys * 2;  // P of one query tile
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = 2 * kQBytes;
  static constexpr int kPOff = kStageOff + kStages * kStageBytes;
  static constexpr int kSmem = kPOff + 2 * kPBytes + 1024;
  // tensor-memory columns: S of tiles 0 / 1 (64 each), O of tiles 0 / 1 (D each)
  static constexpr uint32_t kCols = D == 128 ? 512 : 256;
  static constexpr uint32_t kColS = 0, kColO = 2 * kPfKeys;
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

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap pool_map,
                                                               const __grid_constant__ CUtensorMap knew_map,
                                                               const __grid_constant__ CUtensorMap vnew_map,
                                                               const __grid_constant__ CUtensorMap q_map,
                                                               const __grid_constant__ PrefillArgs a) {
  using Cfg = PfCfg<D>;
  constexpr int NS = Cfg::kStages;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t kv_full[NS], kv_empty[NS];
  __shared__ __align__(8) uint64_t q_full, s_full[2], s_free[2], p_full[2], o_done[2], drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.pv.kv_heads;
  const int G = a.group;
  const int QT = kPfM / G;  // tokens per query tile
  const int Hq = H * G;
  const int bs = a.pv.block_size;

  // work item: heads in the host's order (longest windows first), then sequences, tile pairs
  const int per_head = a.pv.num_seqs * a.q_tiles;
  const int h = a.head_order[blockIdx.x / per_head];
  const int rem = blockIdx.x % per_head;
  const int s = rem / a.q_tiles;
  const int qt = rem % a.q_tiles;

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

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(&q_full, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&s_free[x], 4);
      mbar_init(&p_full[x], 4);
      mbar_init(&o_done[x], 1);
    }
    mbar_init(&drain, 1);
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
    // ---- TMA producer -----------------------------------------------------------------
    if (lane == 0) {
      // both query tiles: box of G heads x QT tokens x 64 columns per column block
      mbar_arrive_expect_tx(&q_full, 2 * Cfg::kHalves * QT * G * 128);
      for (int x = 0; x < 2; ++x)
        for (int hf = 0; hf < Cfg::kHalves; ++hf)
          tma_load_3d(sbase + Cfg::kQOff + x * Cfg::kQBytes + hf * (kPfM * 128), &q_map, hf * 64, h * G,
                      s * a.n_max + qa + x * QT, &q_full);
      int issued = 0;
      for (int j = 0; j < nst; ++j) {
        const int st = j % NS;
        // pool rows of the stage's ring tiles (looked up before waiting for the slot); chunk
        // tiles are -1; padding tiles past the stream read pool row 0 (finite, masked)
        int row[kPfSub];
#pragma unroll
        for (int u = 0; u < kPfSub; ++u) {
          const int t = j * kPfSub + u;
          row[u] = 0;
          if (t < tl.prior_tiles) {
            int tile = tl.prior_first + t;
            if (tile >= tl.C16) tile -= tl.C16;
            const int t0 = tile << 4;
            const int jb = t0 / bs;
            int32_t blk = tbl[jb];
            if (blk < 0 || (int64_t)blk >= a.pv.total_blocks) {
              atomicOr(a.pv.err, HWKV_DEVERR_BAD_BLOCK);
              blk = 0;
            }
            row[u] = blk * 2 * bs + (t0 - jb * bs);
          } else if (t < ntiles) {
            row[u] = -1;
          }
        }
        if (j >= NS && !pf_wait(&kv_empty[st], (uint32_t)((j / NS) - 1) & 1u, abort, a.pv.err)) break;
        const uint32_t kdst = sbase + Cfg::kStageOff + st * Cfg::kStageBytes;
        const uint32_t vdst = kdst + Cfg::kKBytes;
        mbar_arrive_expect_tx(&kv_full[st], Cfg::kStageBytes);
#pragma unroll
        for (int u = 0; u < kPfSub; ++u) {
#pragma unroll
          for (int hf = 0; hf < Cfg::kHalves; ++hf) {
            const uint32_t off = hf * (kPfKeys * 128) + u * (kTile * 128);
            if (row[u] < 0) {
              const int z = s * a.n_max + ((tl.chunk_first + j * kPfSub + u - tl.prior_tiles) << 4);
              tma_load_3d(kdst + off, &knew_map, hf * 64, h, z, &kv_full[st]);
              tma_load_3d(vdst + off, &vnew_map, hf * 64, h, z, &kv_full[st]);
            } else {
              tma_load_2d_l2(kdst + off, &pool_map, hf * 64, row[u], &kv_full[st]);
              tma_load_2d_l2(vdst + off, &pool_map, hf * 64, row[u] + bs, &kv_full[st]);
            }
          }
        }
        ++issued;
      }
      if (*abort) {  // let the copies in flight land before the shared memory is released
        for (int j = max(0, issued - NS); j < issued; ++j)
          if (!mbar_wait_bounded(&kv_full[j % NS], (uint32_t)(j / NS) & 1u)) break;
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer -------------------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t idS = umma_idesc_bf16(kPfM, kPfKeys, false, false);
      constexpr uint32_t idO = umma_idesc_bf16(kPfM, D, false, true);
      bool ok = pf_wait(&q_full, 0, abort, a.pv.err);
      for (int j = 0; ok && j <= nst; ++j) {
        if (j < nst) {
          // S_x = Q_x . K^T for both query tiles, as soon as each softmax has read its last S
          const int st = j % NS;
          ok = pf_wait(&kv_full[st], (uint32_t)(j / NS) & 1u, abort, a.pv.err);
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t kaddr = sbase + Cfg::kStageOff + st * Cfg::kStageBytes;
          for (int x = 0; x < 2 && ok; ++x) {
            if (j > 0) {
              ok = pf_wait(&s_free[x], (uint32_t)(j - 1) & 1u, abort, a.pv.err);
              if (!ok) break;
              tc_fence_after_sync();
            }
            const uint32_t qaddr = sbase + Cfg::kQOff + x * Cfg::kQBytes;
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
              const uint32_t qo = (i >> 2) * (kPfM * 128) + (i & 3) * 32;
              const uint32_t ko = (i >> 2) * (kPfKeys * 128) + (i & 3) * 32;
              umma_bf16(tmem + Cfg::kColS + x * kPfKeys, umma_desc_sw128(qaddr + qo, 16, 1024),
                        umma_desc_sw128(kaddr + ko, 16, 1024), idS, i > 0 ? 1u : 0u);
            }
            umma_commit(&s_full[x]);
          }
          if (!ok) break;
        }
        if (j > 0) {
          // O_x += P_x . V of the previous stage, once each softmax has written its P
          const int jp = j - 1, stp = jp % NS;
          const uint32_t vaddr = sbase + Cfg::kStageOff + stp * Cfg::kStageBytes + Cfg::kKBytes;
          for (int x = 0; x < 2 && ok; ++x) {
            ok = pf_wait(&p_full[x], (uint32_t)jp & 1u, abort, a.pv.err);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t paddr = sbase + Cfg::kPOff + x * Cfg::kPBytes;
#pragma unroll
            for (int i = 0; i < kPfKeys / 16; ++i)
              umma_bf16(tmem + Cfg::kColO + x * D, umma_desc_sw128(paddr + i * 32, 16, 1024),
                        umma_desc_sw128(vaddr + i * (16 * 128), kPfKeys * 128, 1024), idO,
                        (jp > 0 || i > 0) ? 1u : 0u);
            umma_commit(&o_done[x]);
          }
          if (!ok) break;
          umma_commit(&kv_empty[stp]);
        }
      }
      umma_commit(&drain);  // every MMA issued above completes before tensor memory is freed
      mbar_wait_bounded(&drain, 0);
    }
  } else if (warp >= 4) {
    // ---- softmax of query tile x: thread = row ----------------------------------------
    const int x = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row of the tile = tensor-memory lane
    const int tok = qa + x * QT + r / G;
    const bool live = r < QT * G && tok < n;
    const int pq = p0 + tok;
    const int t_first = qa + x * QT, t_last = min(n, qa + (x + 1) * QT) - 1;  // live tokens of the tile
    const int pq_lo = p0 + t_first, pq_hi = p0 + t_last;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t colS = Cfg::kColS + x * kPfKeys, colO = Cfg::kColO + x * D;
    const uint32_t prow = sbase + Cfg::kPOff + x * Cfg::kPBytes + r * 128;
    const float sl2 = a.scale_log2;
    float m_ref = kNegInf, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nst; ++j) {
      ok = __all_sync(0xffffffffu, pf_wait(&s_full[x], (uint32_t)j & 1u, abort, a.pv.err));
      if (!ok) break;
      tc_fence_after_sync();
      float sv[kPfKeys];
      tmem_ld32(lane_base + colS, sv);
      tmem_ld32(lane_base + colS + 32, sv + 32);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[x]);

      // where the stage's keys come from; a "clean" stage needs no mask for any live row
      PfKeyTile kt[kPfSub];
      bool clean = t_first <= t_last;
#pragma unroll
      for (int u = 0; u < kPfSub; ++u) {
        kt[u] = key_tile(tl, j * kPfSub + u, C);
        int k_lo = 0;
        if (kt[u].kind == 0) {
          clean = clean && kt[u].a + kTile - 1 < tl.rs.n;
          k_lo = tl.p_oldest + kt[u].a;
        } else if (kt[u].kind == 1) {
          clean = clean && kt[u].a + kTile - 1 < n;
          k_lo = p0 + kt[u].a;
        } else {
          clean = false;
        }
        clean = clean && k_lo + kTile - 1 <= pq_lo && k_lo > pq_hi - w;
      }
      float mx = kNegInf;
      if (clean) {
#pragma unroll
        for (int c = 0; c < kPfKeys; ++c) {
          sv[c] *= sl2;
          mx = fmaxf(mx, sv[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kPfKeys; ++c) {
          const int u = c >> 4, i = c & 15;
          bool okk = false;
          int kp = 0;
          if (kt[u].kind == 0) {
            int d = kt[u].a + i;
            if (d >= C) d -= C;
            okk = d < tl.rs.n;
            kp = tl.p_oldest + d;
          } else if (kt[u].kind == 1) {
            const int rr = kt[u].a + i;
            okk = rr < n;
            kp = p0 + rr;
          }
          okk = okk && live && kp <= pq && kp > pq - w;
          sv[c] = okk ? sv[c] * sl2 : kNegInf;
          mx = fmaxf(mx, sv[c]);
        }
      }
      const float m_new = fmaxf(m_ref, mx);
      const bool grow = m_new > m_ref + 8.f;
      // P buffer and O are this tile's to touch once the previous P . V has completed
      if (j > 0) {
        ok = __all_sync(0xffffffffu, pf_wait(&o_done[x], (uint32_t)(j - 1) & 1u, abort, a.pv.err));
        if (!ok) break;
        tc_fence_after_sync();
        if (__any_sync(0xffffffffu, grow)) {
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
      const float b = m_ref == kNegInf ? 0.f : m_ref;

      // V rows past the chunk are zeroed: their P is 0, but 0 times a non-finite value is not
      if (x == 0) {
        bool need = false;
#pragma unroll
        for (int u = 0; u < kPfSub; ++u) need = need || (kt[u].kind == 1 && kt[u].a + kTile > n);
        if (need) {
          ok = __all_sync(0xffffffffu, pf_wait(&kv_full[j % NS], (uint32_t)(j / NS) & 1u, abort, a.pv.err));
          if (!ok) break;
          const uint32_t vst = sbase + Cfg::kStageOff + (j % NS) * Cfg::kStageBytes + Cfg::kKBytes;
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
        }
      }

      // P row (bf16) in the 128-byte-swizzled K-major layout
      float ls = 0.f;
#pragma unroll
      for (int k = 0; k < kPfKeys / 8; ++k) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pa = ex2(sv[8 * k + 2 * e] - b), pb = ex2(sv[8 * k + 2 * e + 1] - b);
          ls += pa + pb;
          pk[e] = pack_bf16(pa, pb);
        }
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(prow + ((k ^ (r & 7)) << 4)), "r"(pk[0]),
                     "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                     : "memory");
      }
      l += ls;
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[x]);
    }
    if (ok) ok = __all_sync(0xffffffffu, pf_wait(&o_done[x], (uint32_t)(nst - 1) & 1u, abort, a.pv.err));
    if (ok) {
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

template <int D>
cudaError_t launch_pf(const PrefillArgs& a, const CUtensorMap* pm, const CUtensorMap* km, const CUtensorMap* vm,
                      const CUtensorMap* qm, int items, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, PfCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  prefill_kernel<D><<<items, kPfThreads, PfCfg<D>::kSmem, st>>>(*pm, *km, *vm, *qm, a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

int prefill_tokens_per_cta(int group) { return 2 * (kPfM / group); }

int prefill_tile_tokens(int group) { return kPfM / group; }

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap* pool_map, const CUtensorMap* knew_map,
                           const CUtensorMap* vnew_map, const CUtensorMap* q_map, cudaStream_t st) {
  const int items = a.pv.kv_heads * a.pv.num_seqs * a.q_tiles;
  if (a.group < 1 || a.group > kMaxGroup) return cudaErrorInvalidValue;
  if (a.pv.head_dim == 128) return launch_pf<128>(a, pool_map, knew_map, vnew_map, q_map, items, st);
  if (a.pv.head_dim == 64) return launch_pf<64>(a, pool_map, knew_map, vnew_map, q_map, items, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_chunk_append(const PrefillArgs& a, int max_rows, cudaStream_t st) {
  const int row_bytes = a.pv.head_dim * 2;
  const dim3 grid((unsigned)((max_rows + 7) / 8), (unsigned)(a.pv.num_seqs * a.pv.kv_heads));
  chunk_append_kernel<<<grid, 256, 0, st>>>(a, row_bytes);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace hwkv
