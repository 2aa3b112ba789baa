// CUDA-core split-K decode attention and its combine: the path for fp32 pools and for
// shapes the tensor-core kernel does not take (block_size not a multiple of 16).
//
// "HeadWiseKV: Budgeted Per-Head Cache Residency for Hybrid Long-Context Language Models",
// abstract and section "Grouped-Cache Runtime": attention reads only the materialised window
// of each KV head (the last min(w, len) tokens), through the head's block table.
//
// item = (seq s, kv head h, chunk c); chunk c covers ring slots [c*S, min(C, (c+1)*S)),
// S = split_tokens.  Each CTA streams the resident slots of its chunk once, one token per
// warp iteration, lanes splitting head_dim, and emits (m, l, acc[D]) per query head of the
// GQA group: m = running max of scale*log2(e)*<q,k>, l = sum of 2^(score - m),
// acc = sum of 2^(score - m) * v.  Heads whose ring is one chunk write the normalised
// output directly; the others are merged by combine_kernel.  A CTA holds at most 8 query heads:
// larger GQA groups are split over grid.y (each slice streams the chunk again).
#include "hwkv_device.cuh"

namespace hwkv {
namespace {

struct Item {
  int s, h, c;  // seq, kv head, chunk
  int C, w;     // ring capacity and window of the head
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

constexpr int kSimtWarps = 4;
constexpr int kSimtHeads = 8;  // query heads per CTA

template <typename T, int D>
__global__ void __launch_bounds__(kSimtWarps * 32) decode_simt_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int W = kSimtWarps;
  constexpr int PER = D / 32;
  constexpr int GH = kSimtHeads;
  __shared__ float sm_m[W * GH], sm_l[W * GH];
  __shared__ float sm_acc[W * GH * D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x;
  const Item it = decode_item(a, item);
  int len = a.lens[it.s] + a.len_add;
  if (len < 0) {
    if (threadIdx.x == 0 && it.h == 0 && it.c == 0) atomicOr(a.pv.err, HWKV_DEVERR_NEG_LENGTH);
    len = 0;
  }
  const Resident rs = resident(len, it.w, it.C);
  const int bs = a.pv.block_size;
  const int t_begin = it.c * a.split_tokens;
  const int t_end = min(it.C, t_begin + a.split_tokens);
  const int32_t* tbl_row =
      a.pv.tbl + a.g.tbl_base + (int64_t)it.s * a.g.tbl_seq_stride + a.g.nblk_prefix[it.h];
  const int G = a.group;
  const int Hq = a.pv.kv_heads * G;
  const float sl2 = a.scale_log2;
  const int g0 = blockIdx.y * GH;      // first query head of this CTA's slice
  const int ng = min(GH, G - g0);      // query heads of the slice

  float qv[GH][PER];
  float m[GH], l[GH], acc[GH][PER];
  const T* qbase = static_cast<const T*>(a.q) + ((int64_t)it.s * Hq + it.h * G + g0) * D;
#pragma unroll
  for (int g = 0; g < GH; ++g) {
    m[g] = kNegInf;
    l[g] = 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      qv[g][k] = g < ng ? load_in<T>(qbase + g * D + lane + 32 * k) : 0.f;
      acc[g][k] = 0.f;
    }
  }

  for (int t = t_begin + warp; t < t_end; t += W) {
    if (!slot_valid(rs, t)) continue;
    const int j = t / bs;
    const int32_t blk = tbl_row[j];
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
    for (int g = 0; g < GH; ++g) {
      if (g < ng) {
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
  for (int g = 0; g < GH; ++g) {
    if (lane == 0) {
      sm_m[warp * GH + g] = m[g];
      sm_l[warp * GH + g] = l[g];
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) sm_acc[(warp * GH + g) * D + lane + 32 * k] = acc[g][k];
  }
  __syncthreads();

  // merge the warps; single-chunk heads write the output, the others their partial
  for (int e = threadIdx.x; e < ng * D; e += W * 32) {
    const int gl = e / D, d = e - (e / D) * D;
    const int g = g0 + gl;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, sm_m[w * GH + gl]);
    float Ls = 0.f, A = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float f = ex2(sm_m[w * GH + gl] - M);
        Ls += sm_l[w * GH + gl] * f;
        A += sm_acc[(w * GH + gl) * D + d] * f;
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

// split-K combine: one CTA per (seq, kv head) whose ring spans several chunks
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

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, int dtype, int items, cudaStream_t st) {
  const int D = a.pv.head_dim;
  const dim3 grid((unsigned)items, (unsigned)((a.group + kSimtHeads - 1) / kSimtHeads));
  if (dtype == HWKV_F32 && D == 64) decode_simt_kernel<float, 64><<<grid, kSimtWarps * 32, 0, st>>>(a);
  else if (dtype == HWKV_F32 && D == 128) decode_simt_kernel<float, 128><<<grid, kSimtWarps * 32, 0, st>>>(a);
  else if (dtype == HWKV_BF16 && D == 64) decode_simt_kernel<__nv_bfloat16, 64><<<grid, kSimtWarps * 32, 0, st>>>(a);
  else if (dtype == HWKV_BF16 && D == 128) decode_simt_kernel<__nv_bfloat16, 128><<<grid, kSimtWarps * 32, 0, st>>>(a);
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
