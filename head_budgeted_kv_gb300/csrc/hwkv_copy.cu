// Append and materialise: the two kernels that write the per-head paged pool.
//
// "HeadWiseKV: Budgeted Per-Head Cache Residency for Hybrid Long-Context Language Models",
// abstract and section "Grouped-Cache Runtime": each KV head keeps a static window w in
// ceil(w / bs) blocks; the runtime materialises that residency instead of masking a full
// cache.  A head's blocks form a ring of C = nblk * bs slots: position p lives in slot
// p mod C, so a fixed number of blocks holds a sliding window without reallocation.
//
// Both kernels are HBM copies: 16-byte vector loads and stores, one physical-block lookup
// per row.  They never fault on bad lengths or table entries: those are recorded in the
// device error word and the row is skipped.
#include "hwkv_device.cuh"
#include "hwkv_internal.h"
#include "../../include/hwkv.h"

namespace hwkv {
namespace {

struct RowPtr {
  char* k;   // K row of the slot; the V row is block_size rows further
  bool ok;
};

// Pool address of the K row holding position p of (seq s, kv head h).
__device__ __forceinline__ RowPtr slot_row(const PoolView& pv, const LayerGeom& g, int s, int h,
                                           uint32_t p, uint32_t row_bytes) {
  const uint32_t bs = (uint32_t)pv.block_size;
  const uint32_t C = (uint32_t)(g.nblk_prefix[h + 1] - g.nblk_prefix[h]) * bs;
  const uint32_t slot = p % C;
  const uint32_t j = slot / bs;
  const uint32_t r = slot - j * bs;
  const int32_t blk = pv.tbl[g.tbl_base + (int64_t)s * g.tbl_seq_stride + g.nblk_prefix[h] + j];
  RowPtr out;
  out.ok = blk >= 0 && (int64_t)blk < pv.total_blocks;
  out.k = (char*)pv.pool + ((int64_t)(out.ok ? blk : 0) * 2 * bs + r) * (int64_t)row_bytes;
  return out;
}

// One warp per (seq, kv head): copies the new token's K and V rows into slot pos mod C.
__global__ void __launch_bounds__(128) append_kernel(const __grid_constant__ CopyArgs a, uint32_t row_bytes) {
  const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int H = a.pv.kv_heads;
  if (warp >= a.pv.num_seqs * H) return;
  const int s = warp / H, h = warp - (warp / H) * H;
  const int32_t p = a.lens[s];
  if (p < 0) {
    if (lane == 0) atomicOr(a.pv.err, HWKV_DEVERR_NEG_LENGTH);
    return;
  }
  const RowPtr dst = slot_row(a.pv, a.g, s, h, (uint32_t)p, row_bytes);
  if (!dst.ok) {
    if (lane == 0) atomicOr(a.pv.err, HWKV_DEVERR_BAD_BLOCK);
    return;
  }
  const int nvec = (int)(row_bytes / 16);
  const int64_t src_off = ((int64_t)s * H + h) * row_bytes;
  const uint4* sk = reinterpret_cast<const uint4*>((const char*)a.k + src_off);
  const uint4* sv = reinterpret_cast<const uint4*>((const char*)a.v + src_off);
  uint4* dk = reinterpret_cast<uint4*>(dst.k);
  uint4* dv = reinterpret_cast<uint4*>(dst.k + (int64_t)a.pv.block_size * row_bytes);
  for (int i = lane; i < 2 * nvec; i += 32) {
    if (i < nvec) dk[i] = sk[i];
    else dv[i - nvec] = sv[i - nvec];
  }
}

constexpr int kMatThreads = 256;
constexpr int kMatRows = 64;  // rows (positions) of one (seq, head) per CTA

// grid.x: chunks of kMatRows positions of the resident window, grid.y: seq * H + head.
// NVEC = 16-byte vectors per row.  Each thread issues all its loads before its stores.
template <int NVEC>
__global__ void __launch_bounds__(kMatThreads) materialize_kernel(const __grid_constant__ CopyArgs a) {
  constexpr uint32_t kRowBytes = NVEC * 16;
  constexpr int kRowsPerPass = kMatThreads / NVEC;
  constexpr int kPasses = kMatRows / kRowsPerPass;
  const int H = a.pv.kv_heads;
  const int s = blockIdx.y / H, h = blockIdx.y - (blockIdx.y / H) * H;
  const int32_t L = a.lens[s];
  if (L < 0 || (int64_t)L > a.max_len) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0)
      atomicOr(a.pv.err, L < 0 ? HWKV_DEVERR_NEG_LENGTH : HWKV_DEVERR_SRC_RANGE);
    return;
  }
  const int32_t w = a.g.window[h];
  const int32_t n = w < L ? w : L;         // resident positions: [L - n, L)
  const int32_t r0 = (int32_t)blockIdx.x * kMatRows;
  if (r0 >= n) return;
  const int32_t first = L - n;
  const int c = threadIdx.x % NVEC;
  const int rr = threadIdx.x / NVEC;
  const int64_t src_off = (a.seq_stride * s + a.head_stride * h) * (int64_t)a.pv.elem_bytes;
  const char* kbase = (const char*)a.k + src_off;
  const char* vbase = (const char*)a.v + src_off;

  uint4 kb[kPasses], vb[kPasses];
  char* dst[kPasses];
  bool live[kPasses];
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const int32_t r = r0 + i * kRowsPerPass + rr;
    live[i] = r < n;
    dst[i] = nullptr;
    if (live[i]) {
      const int32_t p = first + r;
      const int64_t off = (int64_t)p * kRowBytes + c * 16;
      kb[i] = __ldcs(reinterpret_cast<const uint4*>(kbase + off));
      vb[i] = __ldcs(reinterpret_cast<const uint4*>(vbase + off));
      const RowPtr rp = slot_row(a.pv, a.g, s, h, (uint32_t)p, kRowBytes);
      if (!rp.ok) {
        atomicOr(a.pv.err, HWKV_DEVERR_BAD_BLOCK);
        live[i] = false;
      }
      dst[i] = rp.k + c * 16;
    }
  }
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    if (live[i]) {
      *reinterpret_cast<uint4*>(dst[i]) = kb[i];
      *reinterpret_cast<uint4*>(dst[i] + (int64_t)a.pv.block_size * kRowBytes) = vb[i];
    }
  }
}

// One thread per sequence: out[s] = in[s] + delta, in unsigned arithmetic (a wrapped value is
// negative and flagged by the kernels that read it as a length or position).
__global__ void __launch_bounds__(256) advance_positions_kernel(const int32_t* in, int32_t* out, int n, int32_t delta) {
  const int i = (int)(blockIdx.x * blockDim.x + threadIdx.x);
  if (i < n) out[i] = (int32_t)((uint32_t)in[i] + (uint32_t)delta);
}

// The bounded wait every kernel of the library uses, run on its own: a phase that has
// completed (one arrival, no bytes) must be seen at once, a phase nothing will complete must be
// given up after limit_ns.  out[0]: the error bits recorded (HWKV_DEVERR_WAIT_TIMEOUT when the
// second wait gave up), out[1]: 1 when the first wait succeeded, out[2]: microseconds the
// second wait took.
__global__ void __launch_bounds__(32) wait_selftest_kernel(int32_t* out, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar[2];
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar[1], 0);
    const bool seen = mbar_wait_bounded(&bar[1], 0, limit_ns);
    const uint64_t t0 = global_timer_ns();
    const bool never = mbar_wait_bounded(&bar[0], 0, limit_ns);
    const uint64_t t1 = global_timer_ns();
    out[0] = never ? 0 : HWKV_DEVERR_WAIT_TIMEOUT;
    out[1] = seen ? 1 : 0;
    const uint64_t us = (t1 - t0) / 1000ull;
    out[2] = us > 0x7FFFFFFFull ? 0x7FFFFFFF : (int32_t)us;
  }
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t* out, uint32_t limit_us, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(out, (uint64_t)limit_us * 1000ull);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_advance_positions(const int32_t* in, int32_t* out, int n, int32_t delta, cudaStream_t st) {
  advance_positions_kernel<<<(n + 255) / 256, 256, 0, st>>>(in, out, n, delta);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_append(const CopyArgs& a, int dtype, cudaStream_t st) {
  const uint32_t row_bytes = (uint32_t)a.pv.head_dim * (dtype == HWKV_F32 ? 4u : 2u);
  const int warps = a.pv.num_seqs * a.pv.kv_heads;
  const int blocks = (warps + 3) / 4;
  append_kernel<<<blocks, 128, 0, st>>>(a, row_bytes);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_materialize(const CopyArgs& a, int dtype, int max_rows, cudaStream_t st) {
  const uint32_t row_bytes = (uint32_t)a.pv.head_dim * (dtype == HWKV_F32 ? 4u : 2u);
  const dim3 grid((unsigned)(((int64_t)max_rows + kMatRows - 1) / kMatRows), (unsigned)(a.pv.num_seqs * a.pv.kv_heads));
  switch (row_bytes / 16) {
    case 8: materialize_kernel<8><<<grid, kMatThreads, 0, st>>>(a); break;
    case 16: materialize_kernel<16><<<grid, kMatThreads, 0, st>>>(a); break;
    case 32: materialize_kernel<32><<<grid, kMatThreads, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace hwkv
