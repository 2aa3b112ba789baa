// Internal declarations shared by the host side of the C ABI (hwkv_host.cpp) and the
// sm_103a kernels (hwkv_copy.cu, hwkv_decode.cu).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

struct hwkv_pool;

namespace hwkv {

constexpr int kMaxKvHeads = 32;
constexpr int kMergeBlock = 8;   // CTAs whose partials one first-level merge folds
constexpr int kMaxGroup = 16;  // query heads per KV head (GQA group)
constexpr int kGroupPads = 3;   // tensor-core decode instances: 4, 8 or 16 query-head columns

// Geometry of one layer, passed by value to every kernel of that layer.
//   table entry of (seq s, kv head h, logical block j) = tbl[tbl_base + s*tbl_seq_stride
//                                                          + nblk_prefix[h] + j]
struct LayerGeom {
  int64_t tbl_base;
  int32_t tbl_seq_stride;                 // sum_h nblk[h]
  int32_t nblk_prefix[kMaxKvHeads + 1];   // prefix sums of nblk over heads
  int32_t window[kMaxKvHeads];            // static window w per head
};

struct PoolView {
  void* pool;              // physical blocks [total_blocks][2][bs][D]
  const int32_t* tbl;      // flat block table
  int32_t* err;            // device error word
  int64_t total_blocks;
  int32_t block_size;
  int32_t head_dim;
  int32_t kv_heads;
  int32_t num_seqs;
  int32_t elem_bytes;      // 4 (f32) or 2 (bf16)
};

struct CopyArgs {
  PoolView pv;
  LayerGeom g;
  const void* k;           // materialise: full prefill; append: new token rows
  const void* v;
  int64_t seq_stride;      // elements (materialise only)
  int64_t head_stride;     // elements (materialise only)
  int64_t max_len;         // rows per (s, h) in the source (materialise only)
  const int32_t* lens;     // materialise: prefill lengths; append: positions
  int32_t rows_per_cta;    // materialise only
};

struct DecodeArgs {
  PoolView pv;
  LayerGeom g;
  const void* q;           // [B][Hq][D]
  void* out;               // [B][Hq][D]
  const int32_t* lens;     // [B]; length after the append = lens[s] + len_add
  int32_t len_add;         // 0: lens are lengths after the append; 1: positions (fused append)
  int32_t early;           // schedule and first tile loads may run before the dependent-launch wait
  const void* k_new;       // fused append: new K / V rows [B][H][D], else null
  const void* v_new;
  float* part_acc;         // [slots][G][D]   unnormalised split accumulators
  float* part_ml;          // [slots][G][2]   (running max in log2 units, sum of weights)
  uint32_t* counters;      // [B*H] arrival counters of this layer (tensor-core kernel), all 0
  uint32_t* counters1;     // [B*H][merge_blocks] first-level arrival counters, all 0
  float* part2_acc;        // [B*H*merge_blocks][G][D] second-level partials
  float* part2_ml;         // [B*H*merge_blocks][G][2]
  int32_t merge_blocks;    // first-level merge blocks per head: ceil(CTAs / kMergeBlock) + 1
  float scale_log2;        // scale * log2(e)
  int32_t group;           // G = Hq / H
  int32_t split_tokens;    // CUDA-core kernel: tokens per split-K chunk (power of two)
  int32_t chunk_prefix[kMaxKvHeads + 1];  // CUDA-core kernel: prefix over heads of ceil(C_h / split)
};

struct PrefillArgs {
  PoolView pv;
  LayerGeom g;
  const void* q;           // [B][n_max][Hq][D]
  const void* k_new;       // [B][n_max][H][D] chunk keys / values
  const void* v_new;
  void* out;               // [B][n_max][Hq][D]
  const int32_t* pos0;     // [B] lengths before the chunk
  const int32_t* nlen;     // [B] chunk lengths (<= n_max)
  int32_t n_max;
  int32_t group;           // G = Hq / H
  int32_t q_tiles;         // query-tile pairs per (seq, head): ceil(n_max / chunk tokens per pair)
  float scale_log2;
  int32_t bs_log2;         // log2(block_size), or -1 when it is not a power of two
  int32_t stage_tb;        // rows of one block in a 64-key pool copy (16, 32, 64), 0: per-tile copies only
  int32_t head_order[kMaxKvHeads];  // heads in work order (longest CTAs first)
  // split of long key streams: head order position i has splits[i] CTAs per (seq, tile pair),
  // each streaming split_stages[i] stages; its CTAs are [head_ctas[i], head_ctas[i + 1])
  int32_t splits[kMaxKvHeads];
  int32_t split_stages[kMaxKvHeads];
  int32_t head_ctas[kMaxKvHeads + 1];
  float* part_o;           // [CTA][256 rows][D] unnormalised partial outputs of split streams
  float* part_ml;          // [CTA][256 rows][2] (reference maximum in log2 units, sum)
};

// Counts every kernel launch the library makes (read by hwkv_kernel_launches).
void count_launches(uint64_t n);

// Records a message for hwkv_last_error() on this thread and returns `code`.
int set_error(int code, const char* fmt, ...);

// HWKV_OK when the pool's device is the current one, else an error (message recorded).
int check_pool_device(const struct ::hwkv_pool* p);

// Launchers (hwkv_copy.cu, hwkv_decode.cu).  dtype: 0 = f32, 1 = bf16.
cudaError_t launch_append(const CopyArgs& a, int dtype, cudaStream_t st);
// out[i] = in[i] + delta for i < n (in == out allowed)
cudaError_t launch_advance_positions(const int32_t* in, int32_t* out, int n, int32_t delta, cudaStream_t st);
// the bounded wait of every kernel, on a phase that completes and one that never does
cudaError_t launch_wait_selftest(int32_t* out, uint32_t limit_us, cudaStream_t st);
// max_rows: the most positions any (seq, head) of the layer copies, min(max window, max_len)
cudaError_t launch_materialize(const CopyArgs& a, int dtype, int max_rows, cudaStream_t st);
// once per device before the first launch; returns resident CTAs per SM of the instances
// for 4, 8 and 16 query-head columns (fp32 pools: 4 only, the others 0)
cudaError_t configure_decode_tc(int head_dim, int dtype, int ctas_per_sm[kGroupPads]);
// stream-K kernel (tensor cores for bf16, CUDA cores for fp32 with group <= 4): `ctas`
// persistent CTAs split the resident tiles of the layer evenly
cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap* tmap, int ctas, cudaStream_t st);
int decode_tc_group_pad(int group);  // query-head columns the kernel instance holds (4, 8 or 16)
int decode_tc_pad_index(int group);  // 0, 1, 2 for 4, 8, 16 columns
cudaError_t launch_decode_simt(const DecodeArgs& a, int dtype, int items, cudaStream_t st);
cudaError_t launch_combine(const DecodeArgs& a, int dtype, cudaStream_t st);
// chunked prefill (hwkv_prefill.cu): attention, then the chunk appended to the rings
int prefill_tokens_per_cta(int group);  // chunk tokens one CTA answers (two query tiles)
int prefill_tile_tokens(int group);     // chunk tokens of one 128-row query tile
// pool_map: 16-row tiles of the pool; stage_map: 64 keys of consecutive blocks (see
// hwkv_pool::stage_map); knew/vnew maps: 16-row and 64-row boxes of the chunk
cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap* pool_map, const CUtensorMap* stage_map,
                           const CUtensorMap* knew_map, const CUtensorMap* vnew_map, const CUtensorMap* knew64_map,
                           const CUtensorMap* vnew64_map, const CUtensorMap* q_map, cudaStream_t st);
cudaError_t launch_chunk_append(const PrefillArgs& a, int max_rows, cudaStream_t st);
// merge of the partials of split key streams (after launch_prefill)
cudaError_t launch_prefill_combine(const PrefillArgs& a, cudaStream_t st);
// upper bound on the 64-key stages of one prefill CTA's key stream for a head
int prefill_max_stages(int window, int ring_capacity, int group, int n_max);
// the 64-key stages the tile pair starting at chunk row qa streams when the context before the
// chunk is longer than the ring and the chunk holds n_max rows (work estimate for planning)
int prefill_stages_estimate(int window, int ring_capacity, int group, int n_max, int qa);

}  // namespace hwkv
