// Chunked prefill over the per-head paged rings: windowed causal attention for a chunk of new
// tokens, then the chunk's K/V written into the rings.
//
// "HeadWiseKV: Budgeted Per-Head Cache Residency for Hybrid Long-Context Language Models",
// abstract and section "Grouped-Cache Runtime": each KV head keeps only a static window w of
// its newest tokens.  A new token at position p therefore attends, per KV head, to positions
// [max(0, p + 1 - w), p]: the part before the chunk is read from the head's ring in the pool
// (the last min(w, p0) positions before the chunk start p0), the rest from the chunk's own
// K/V rows.  Appending the chunk then overwrites ring slots that earlier queries of the same
// chunk still read, so the append is a second launch after the attention.
//
// prefill_kernel (bf16, block_size % 16 == 0, head_dim 64 or 128, GQA group 1 <= G <= 16):
//   CTA = (seq, kv head, query tile of 64 rows = floor(64/G) tokens x G query heads, the rows
//   past the last whole token idle); 4 consumer
//   warps own 16 rows each, a producer warp streams 16-token K/V tiles into a 4-stage ring of
//   shared memory with TMA (pool tiles through the block table, chunk tiles through a tensor
//   map of the chunk).  Per tile and warp: S[16 rows][16 keys] = Q K^T and O += P V with
//   mma.sync.m16n8k16 bf16 -> fp32 (FlashAttention-2 register reuse of P), causal + window
//   mask per row, online softmax in fp32 (log2 domain).  Waits are bounded (~2 s).
#include "hwkv_device.cuh"

namespace hwkv {
namespace {

constexpr int kPfConsumers = 4;            // consumer warps (16 query rows each)
constexpr int kPfThreads = (kPfConsumers + 1) * 32;
constexpr int kPfStages = 4;
constexpr int kPfRows = kPfConsumers * 16;  // query rows per CTA

__device__ __forceinline__ uint32_t swz(int row, int d) {
  return (uint32_t)((d >> 6) * 2048 + row * 128 + ((((d & 63) >> 3) ^ (row & 7)) << 4) + (d & 7) * 2);
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

// The key tiles one CTA streams: first the ring tiles holding the prior context its queries
// may see, then the chunk tiles up to its last query.
struct PfTiles {
  // prior part (ring of the head at length p0)
  Resident rs;        // resident positions before the chunk
  int prior_first;    // ring tile of the oldest prior position needed
  int prior_tiles;    // number of ring tiles (cyclic from prior_first)
  int C16;
  int p_oldest;       // position held by ring slot rs.first_slot
  // chunk part: chunk rows [16 * chunk_first, ...)
  int chunk_first;
  int chunk_tiles;
};

template <int D>
__global__ void __launch_bounds__(kPfThreads) prefill_kernel(const __grid_constant__ CUtensorMap pool_map,
                                                            const __grid_constant__ CUtensorMap knew_map,
                                                            const __grid_constant__ CUtensorMap vnew_map,
                                                            const __grid_constant__ PrefillArgs a) {
  constexpr int kHalves = D / 64;
  constexpr int kTileBytes = kTile * D * 2;
  constexpr int kStageBytes = 2 * kTileBytes;
  constexpr int kSteps = D / 16;  // k-steps of QK
  constexpr int kDTiles = D / 8;  // n-tiles of PV

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kPfStages], empty[kPfStages];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.pv.kv_heads;
  const int G = a.group;
  const int QT = kPfRows / G;  // tokens per CTA
  const int Hq = H * G;
  const int bs = a.pv.block_size;

  // work item: heads in the host's order (longest windows first), then sequences, query tiles
  const int per_head = a.pv.num_seqs * a.q_tiles;
  const int h = a.head_order[blockIdx.x / per_head];
  const int rem = blockIdx.x % per_head;
  const int s = rem / a.q_tiles;
  const int qt = rem % a.q_tiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kPfConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int p0 = a.pos0[s];
  const int n = a.nlen[s];
  if (p0 < 0 || n < 0 || n > a.n_max) {
    if (threadIdx.x == 0 && h == a.head_order[0] && qt == 0) atomicOr(a.pv.err, HWKV_DEVERR_NEG_LENGTH);
    return;
  }
  const int qa = qt * QT;  // first chunk row of this CTA
  if (qa >= n) return;
  const int qb = min(n, qa + QT);  // one past the last chunk row
  const int w = a.g.window[h];
  const int C = (a.g.nblk_prefix[h + 1] - a.g.nblk_prefix[h]) * bs;
  const int32_t* tbl = a.pv.tbl + a.g.tbl_base + (int64_t)s * a.g.tbl_seq_stride + a.g.nblk_prefix[h];

  // tiles: prior positions [lo, p0) with lo = max(0, p0 + qa + 1 - w), chunk rows [clo, qb)
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

  if (warp == kPfConsumers) {
    // ---- producer: one lane streams the tiles -----------------------------------------
    if (lane == 0) {
      const uint64_t policy = evict_first_policy();
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kPfStages;
        if (t >= kPfStages && !mbar_wait_bounded(&empty[st], (uint32_t)((t / kPfStages) - 1) & 1u)) {
          atomicOr(a.pv.err, HWKV_DEVERR_WAIT_TIMEOUT);
          break;
        }
        const uint32_t dst = smem_addr(smem) + st * kStageBytes;
        mbar_arrive_expect_tx(&full[st], kStageBytes);
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
          const int row_k = blk * 2 * bs + (t0 - jb * bs);
#pragma unroll
          for (int hf = 0; hf < kHalves; ++hf) {
            tma_load_2d(dst + hf * 2048, &pool_map, hf * 64, row_k, &full[st], policy);
            tma_load_2d(dst + kTileBytes + hf * 2048, &pool_map, hf * 64, row_k + bs, &full[st], policy);
          }
        } else {
          const int z = s * a.n_max + ((tl.chunk_first + t - tl.prior_tiles) << 4);
#pragma unroll
          for (int hf = 0; hf < kHalves; ++hf) {
            tma_load_3d(dst + hf * 2048, &knew_map, hf * 64, h, z, &full[st]);
            tma_load_3d(dst + kTileBytes + hf * 2048, &vnew_map, hf * 64, h, z, &full[st]);
          }
        }
      }
    }
    return;
  }

  // ---- consumers: 16 query rows per warp; row r -> token qa + r / G, head r % G ----------
  const int gq = lane >> 2, q4 = lane & 3;
  const int row0 = warp * 16 + gq, row1 = row0 + 8;
  const int tok0 = qa + row0 / G, tok1 = qa + row1 / G;  // chunk rows of the lane's two rows
  const int pq0 = p0 + tok0, pq1 = p0 + tok1;            // their positions
  // rows holding a real query: inside the CTA's whole tokens and the chunk
  const bool ok0 = row0 < QT * G && tok0 < n, ok1 = row1 < QT * G && tok1 < n;
  // Q as the A operand: lane holds rows row0/row1, dims 16i + 2*q4 + {0,1} and +8
  uint32_t qf[kSteps][4];
  {
    const __nv_bfloat16* qbase = static_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* q0 = qbase + (((int64_t)s * a.n_max + (ok0 ? tok0 : 0)) * Hq + h * G + row0 % G) * D;
    const __nv_bfloat16* q1 = qbase + (((int64_t)s * a.n_max + (ok1 ? tok1 : 0)) * Hq + h * G + row1 % G) * D;
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {
      const int d = 16 * i + 2 * q4;
      qf[i][0] = ok0 ? *reinterpret_cast<const uint32_t*>(q0 + d) : 0u;
      qf[i][1] = ok1 ? *reinterpret_cast<const uint32_t*>(q1 + d) : 0u;
      qf[i][2] = ok0 ? *reinterpret_cast<const uint32_t*>(q0 + d + 8) : 0u;
      qf[i][3] = ok1 ? *reinterpret_cast<const uint32_t*>(q1 + d + 8) : 0u;
    }
  }
  float o[kDTiles][4];
#pragma unroll
  for (int j = 0; j < kDTiles; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;  // rows row0, row1
  const float sl2 = a.scale_log2;
  const int mi = lane >> 3, rr = lane & 7;
  const int k_key = rr + ((mi >> 1) << 3), k_dof = (mi & 1) << 3;  // K (B operand, non-transposed)
  const int v_key = rr + ((mi & 1) << 3), v_dof = (mi >> 1) << 3;  // V (B operand, transposed)

  for (int t = 0; t < ntiles; ++t) {
    const int st = t % kPfStages;
    if (!mbar_wait_bounded(&full[st], (uint32_t)(t / kPfStages) & 1u)) {
      if (lane == 0) atomicOr(a.pv.err, HWKV_DEVERR_WAIT_TIMEOUT);
      break;
    }
    const uint32_t sK = smem_addr(smem) + st * kStageBytes;
    const uint32_t sV = sK + kTileBytes;

    // positions of the lane's four keys (columns 2*q4, 2*q4 + 1 of each 8-key half)
    int kp[4];
    bool kv_ok[4];
    if (t < tl.prior_tiles) {
      int tile = tl.prior_first + t;
      if (tile >= tl.C16) tile -= tl.C16;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int slot = (tile << 4) + (c >> 1) * 8 + 2 * q4 + (c & 1);
        int d = slot - tl.rs.first_slot;
        if (d < 0) d += C;
        kv_ok[c] = d < tl.rs.n;
        kp[c] = tl.p_oldest + d;
      }
    } else {
      const int r0 = (tl.chunk_first + t - tl.prior_tiles) << 4;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int r = r0 + (c >> 1) * 8 + 2 * q4 + (c & 1);
        kv_ok[c] = r < n;
        kp[c] = p0 + r;
      }
    }

    // S[16 rows][16 keys] = Q . K^T
    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {
      uint32_t b[4];
      ldsm_x4(b, sK + swz(k_key, 16 * i + k_dof));
      const uint32_t a4[4] = {qf[i][0], qf[i][1], qf[i][2], qf[i][3]};
      mma_bf16(sc[0], a4, b[0], b[1]);
      mma_bf16(sc[1], a4, b[2], b[3]);
    }
    // mask: key position in [pq - w + 1, pq] of its row, and holding a real token
    float x[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = nt * 2 + (e & 1);
        const int pq = (e < 2) ? pq0 : pq1;
        const bool ok = kv_ok[c] && kp[c] <= pq && kp[c] > pq - w;
        x[nt][e] = ok ? sc[nt][e] : kNegInf;
      }
    }
    float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
    float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(m0, mx0 * sl2), n1 = fmaxf(m1, mx1 * sl2);
    const float b0 = n0 == kNegInf ? 0.f : n0, b1 = n1 == kNegInf ? 0.f : n1;
    const float al0 = ex2(m0 - b0), al1 = ex2(m1 - b1);
    float p[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      p[nt][0] = ex2(fmaf(x[nt][0], sl2, -b0));
      p[nt][1] = ex2(fmaf(x[nt][1], sl2, -b0));
      p[nt][2] = ex2(fmaf(x[nt][2], sl2, -b1));
      p[nt][3] = ex2(fmaf(x[nt][3], sl2, -b1));
    }
    l0 = fmaf(l0, al0, p[0][0] + p[0][1] + p[1][0] + p[1][1]);
    l1 = fmaf(l1, al1, p[0][2] + p[0][3] + p[1][2] + p[1][3]);
    m0 = n0;
    m1 = n1;
    // P as the A operand of O += P . V (16 rows x 16 keys)
    const uint32_t pa[4] = {pack_bf16(p[0][0], p[0][1]), pack_bf16(p[0][2], p[0][3]), pack_bf16(p[1][0], p[1][1]),
                            pack_bf16(p[1][2], p[1][3])};
#pragma unroll
    for (int j = 0; j < kDTiles; j += 2) {
      uint32_t b[4];
      ldsm_x4_trans(b, sV + swz(v_key, 8 * j + v_dof));
      o[j][0] *= al0;
      o[j][1] *= al0;
      o[j][2] *= al1;
      o[j][3] *= al1;
      o[j + 1][0] *= al0;
      o[j + 1][1] *= al0;
      o[j + 1][2] *= al1;
      o[j + 1][3] *= al1;
      mma_bf16(o[j], pa, b[0], b[1]);
      mma_bf16(o[j + 1], pa, b[2], b[3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // normalise and store the lane's two rows (row sums over the 4 lanes of a row)
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
  __nv_bfloat16* obase = static_cast<__nv_bfloat16*>(a.out);
  if (ok0) {
    __nv_bfloat16* o0 = obase + (((int64_t)s * a.n_max + tok0) * Hq + h * G + row0 % G) * D;
#pragma unroll
    for (int j = 0; j < kDTiles; ++j)
      *reinterpret_cast<uint32_t*>(o0 + 8 * j + 2 * q4) = pack_bf16(o[j][0] * i0, o[j][1] * i0);
  }
  if (ok1) {
    __nv_bfloat16* o1 = obase + (((int64_t)s * a.n_max + tok1) * Hq + h * G + row1 % G) * D;
#pragma unroll
    for (int j = 0; j < kDTiles; ++j)
      *reinterpret_cast<uint32_t*>(o1 + 8 * j + 2 * q4) = pack_bf16(o[j][2] * i1, o[j][3] * i1);
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
constexpr int pf_smem() {
  return kPfStages * 2 * kTile * D * 2 + 1024;
}

template <int D>
cudaError_t launch_pf(const PrefillArgs& a, const CUtensorMap* pm, const CUtensorMap* km, const CUtensorMap* vm,
                      int items, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, pf_smem<D>());
  if (e != cudaSuccess) return e;
  prefill_kernel<D><<<items, kPfThreads, pf_smem<D>(), st>>>(*pm, *km, *vm, a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

int prefill_tokens_per_cta(int group) { return kPfRows / group; }

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap* pool_map, const CUtensorMap* knew_map,
                           const CUtensorMap* vnew_map, cudaStream_t st) {
  const int items = a.pv.kv_heads * a.pv.num_seqs * a.q_tiles;
  if (a.group < 1 || a.group > kMaxGroup) return cudaErrorInvalidValue;
  if (a.pv.head_dim == 128) return launch_pf<128>(a, pool_map, knew_map, vnew_map, items, st);
  if (a.pv.head_dim == 64) return launch_pf<64>(a, pool_map, knew_map, vnew_map, items, st);
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
