/*
 * hwkv -- per-head budgeted KV residency on one GB300 (sm_103a).
 *
 * C ABI of the grouped-cache runtime described in "HeadWiseKV: Budgeted Per-Head Cache
 * Residency for Hybrid Long-Context Language Models" (blog summary):
 *
 *   - abstract: every physical KV head of a residual global-attention layer gets a static
 *     history window w; the runtime MATERIALISES that residency (it keeps only the window)
 *     instead of masking a full cache, so the cache footprint is exact before serving;
 *   - section "Grouped-Cache Runtime": a paged block table gives each head
 *     ceil(w / block_size) KV blocks, pre-allocated before serving.
 *
 * Terms used below
 *   L  layers (global-attention layers only), H kv heads, Hq query heads (Hq = G * H),
 *   D  head_dim, bs block_size, B num_seqs, eb element bytes (4 for F32, 2 for BF16).
 *   nblk[l][h] = ceil(w[l][h] / bs);  ring capacity C[l][h] = nblk[l][h] * bs tokens.
 *   Token position p of (seq, layer, head) lives in ring slot p mod C; slot t is row
 *   t mod bs of logical block t / bs, which the block table maps to a physical block.
 *   A physical block is [2][bs][D] elements: bs K rows, then bs V rows (2*bs*D*eb bytes).
 *   Query head q reads kv head q / G (consecutive groups).
 *   Decode attention at length len covers positions [max(0, len - w), len): the last
 *   min(w, len) tokens, including the one appended in the same step.
 *
 * Conventions
 *   - Every function returns an int status (HWKV_OK or a negative HWKV_ERR_*); on error
 *     hwkv_last_error() (thread-local) describes it.  Argument errors are reported before
 *     anything is launched.
 *   - Pointers named *_dev and every tensor argument are DEVICE pointers on the current
 *     CUDA device; the caller owns them (e.g. torch tensors).  `stream` is a cudaStream_t
 *     (NULL = legacy default stream).  Calls that take a stream are asynchronous on it.
 *   - Lengths and positions live on the device so that a captured CUDA graph stays valid
 *     across decode steps; kernels check them and record problems in a device error word
 *     that hwkv_check_device_errors() reads.  Kernels never trap or spin without bound.
 *   - Inputs must be finite: a masked pool row that holds Inf/NaN bits can still poison
 *     a result (0 * Inf), as in any attention kernel.
 */
#ifndef HWKV_H
#define HWKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HWKV_ABI_VERSION 3

/* status codes */
#define HWKV_OK 0
#define HWKV_ERR_INVALID_ARG (-1)
#define HWKV_ERR_ALIGNMENT (-2)
#define HWKV_ERR_POOL_TOO_SMALL (-3)
#define HWKV_ERR_CUDA (-4)
#define HWKV_ERR_DEVICE_CHECK (-5)
#define HWKV_ERR_UNSUPPORTED (-6)
#define HWKV_ERR_WORKSPACE_TOO_SMALL (-7)
#define HWKV_ERR_BUDGET (-8)

/* element types of the pool and of every tensor passed with it */
#define HWKV_F32 0
#define HWKV_BF16 1

/* decode kernel selection for hwkv_set_decode_config */
#define HWKV_KERNEL_AUTO 0   /* stream-K kernel where supported, else the split kernel       */
#define HWKV_KERNEL_TENSOR 1 /* stream-K kernel: tensor cores for bf16, CUDA cores for fp32
                                (fp32: up to 4 query heads per KV head); bs % 16 == 0 only  */
#define HWKV_KERNEL_SIMT 2   /* split-K CUDA-core kernel, any supported shape                  */

/* bits of the device error word */
#define HWKV_DEVERR_NEG_LENGTH 1     /* a length / position below 0                    */
#define HWKV_DEVERR_BAD_BLOCK 2      /* a block-table entry outside the pool            */
#define HWKV_DEVERR_SRC_RANGE 4      /* materialise length above max_len               */
#define HWKV_DEVERR_WAIT_TIMEOUT 8   /* a pipeline wait gave up (work was skipped)      */

typedef struct hwkv_pool* hwkv_pool_t;

/* ABI / layout version (kernel-ABI compatibility check of the cache layout).  Returns
 * HWKV_ABI_VERSION of the loaded library. */
int hwkv_abi_version(void);

/* Thread-local description of the last error on this thread ("" if none). */
const char* hwkv_last_error(void);

/* Short constant name of a status code. */
const char* hwkv_status_string(int status);

/* Pre-serving footprint prediction ("Grouped-Cache Runtime": ceil(w / bs) blocks per head;
 * abstract: demand known exactly before serving).  Pure host, needs no GPU.
 *   windows: host int32 [layers][kv_heads], each >= 1.
 *   out_bytes = num_seqs * sum_{l,h} ceil(w[l][h]/bs) * bs * head_dim * 2 * eb.
 * Supported: 1 <= kv_heads <= 32, head_dim in {64, 128}, block_size >= 1, dtype F32/BF16,
 * every ring capacity below 2^31 tokens and at most 2^31 - 1 blocks in total.
 * Errors: HWKV_ERR_INVALID_ARG, HWKV_ERR_UNSUPPORTED. */
int hwkv_pool_bytes(int layers, int kv_heads, int head_dim, int block_size, const int32_t* windows,
                    int num_seqs, int dtype, uint64_t* out_bytes);

/* Binds a caller-owned device buffer as the per-head paged pool ("Grouped-Cache Runtime").
 *   dev_pool: device pointer, 256-byte aligned, dev_pool_bytes >= hwkv_pool_bytes().
 *   The pool is zero-filled on `stream`.  The block table starts as the identity map with
 *   physical ids handed out in (layer, seq, kv head, logical block) order.
 *   The library allocates its own small device metadata (block table, error word) and
 *   frees it in hwkv_pool_destroy; the pool buffer itself is never freed by the library.
 *   Synchronises `stream` before returning.
 * Errors: HWKV_ERR_INVALID_ARG, HWKV_ERR_UNSUPPORTED, HWKV_ERR_ALIGNMENT (pool pointer),
 *         HWKV_ERR_POOL_TOO_SMALL (checked before anything is written), HWKV_ERR_CUDA. */
int hwkv_pool_create(int layers, int kv_heads, int head_dim, int block_size, const int32_t* windows,
                     int num_seqs, int dtype, void* dev_pool, uint64_t dev_pool_bytes, void* stream,
                     hwkv_pool_t* out);

/* Frees the library-owned metadata.  The caller must make sure no work using the pool is
 * still in flight.  NULL is accepted. */
int hwkv_pool_destroy(hwkv_pool_t pool);

/* Geometry of a created pool: bytes, physical block count, bytes per block. */
int hwkv_pool_geometry(hwkv_pool_t pool, uint64_t* pool_bytes, int64_t* total_blocks, int64_t* block_bytes);

/* Copies the physical block ids of (seq, layer, kv_head) -- nblk of them, logical block
 * order -- into host_out[0 .. cap).  *n receives nblk.  Host copy of the library's table. */
int hwkv_block_table(hwkv_pool_t pool, int seq, int layer, int kv_head, int32_t* host_out, int cap, int* n);

/* Replaces the whole block table (the cache manager above the runtime chooses physical
 * blocks).  host_table: int32 [total_blocks] in (layer, seq, kv head, logical block) order;
 * it must be a permutation of 0 .. total_blocks-1 (checked; HWKV_ERR_INVALID_ARG otherwise).
 * The pool bytes are NOT moved.  Copies on `stream` and synchronises it. */
int hwkv_set_block_table(hwkv_pool_t pool, const int32_t* host_table, int64_t n, void* stream);

/* Materialise ("Grouped-Cache Runtime", abstract): compacts one layer of a contiguous full
 * prefill KV into the pool.  For every seq s and kv head h, the last min(w, L_s) positions
 * p of the prefill are copied to ring slot p mod C (K and V rows); nothing else is written.
 *   k_full, v_full: device, element (s, h, p, d) at s*seq_stride + h*head_stride + p*D + d
 *                   (strides in elements; rows contiguous), 16-byte aligned, strides*eb
 *                   multiples of 16.
 *   max_len: rows available per (s, h) in the source; lens_dev[s] must be in [0, max_len]
 *            (checked on the device: HWKV_DEVERR_NEG_LENGTH / HWKV_DEVERR_SRC_RANGE, the
 *            sequence is skipped).
 *   lens_dev: device int32 [num_seqs] prefill lengths L_s.
 * max_len == 0 is an empty prefill: nothing is read or written and the pointers may be NULL. */
int hwkv_materialize(hwkv_pool_t pool, int layer, const void* k_full, const void* v_full,
                     int64_t seq_stride, int64_t head_stride, int64_t max_len, const int32_t* lens_dev,
                     void* stream);

/* Append: writes the new token of every (seq, kv head) of one layer into its ring slot
 * pos mod C (the slot of the oldest token, which has just left the window when C == w).
 *   k_new, v_new: device [num_seqs][kv_heads][D], 16-byte aligned.
 *   pos_dev: device int32 [num_seqs], the length BEFORE the append (position of the new
 *            token); negative values are flagged (HWKV_DEVERR_NEG_LENGTH) and skipped. */
int hwkv_append(hwkv_pool_t pool, int layer, const void* k_new, const void* v_new, const int32_t* pos_dev,
                void* stream);

/* Position bookkeeping of a serving loop, on the device: out_dev[s] = pos_dev[s] + delta for the
 * pool's num_seqs sequences (int32, wrapping; out_dev may be pos_dev).  It lets a decode step
 * captured in a CUDA graph advance its positions after the step (delta 1), or form the lengths
 * after the append from the positions before it, without a kernel from outside this library.
 * The pages have no counterpart: this is a service of this library, not a step of the method.
 *   pos_dev, out_dev: device int32 [num_seqs], 4-byte aligned.  One kernel on `stream`. */
int hwkv_advance_positions(hwkv_pool_t pool, const int32_t* pos_dev, int32_t* out_dev, int32_t delta, void* stream);

/* Check of the bounded waits (a service of this library; the pages have no counterpart).
 * Every wait of every kernel here gives up after a time limit (~2 s) and records
 * HWKV_DEVERR_WAIT_TIMEOUT in the error word instead of spinning forever.  This runs that same
 * wait loop on its own, in one warp, so a host can see the path work without faulting or
 * hanging a GPU: first on an mbarrier phase that has completed, then on one that nothing will
 * complete, given up after limit_us microseconds.
 *   out_dev: device int32 [3], 4-byte aligned, written by the kernel: [0] the error bits it
 *            recorded (HWKV_DEVERR_WAIT_TIMEOUT when the second wait gave up), [1] 1 when the
 *            first wait returned true, [2] the microseconds the second wait took.
 *   limit_us: 1 .. 2 000 000 (HWKV_ERR_INVALID_ARG otherwise).
 * One kernel on `stream`, on the current device; HWKV_ERR_CUDA if it cannot be launched. */
int hwkv_wait_selftest(uint32_t limit_us, int32_t* out_dev, void* stream);

/* Bytes of scratch hwkv_decode_attn / hwkv_append_decode_attn need for the current decode
 * configuration (fp32 split-K partials; maximum over layers). */
int hwkv_decode_workspace_bytes(hwkv_pool_t pool, int q_heads, uint64_t* out);

/* Split-K decode attention over the resident window of one layer (abstract: attention reads
 * the materialised window, never a masked full cache).  For query head q of seq s, with
 * h = q / G and w = w[layer][h]:
 *     out[s][q] = sum_{p in [max(0,len_s-w), len_s)} softmax_p(scale * <q, k_p>) v_p
 * computed with fp32 accumulation and an online softmax; out has the pool's dtype.
 *   q, out: device [num_seqs][q_heads][D], 16-byte aligned; q_heads = G * kv_heads, G <= 16
 *           (the stream-K kernel pads the group to 4, 8 or 16 query-head columns on the
 *           tensor cores for bf16 pools, to 4 on the CUDA cores for fp32 pools).
 *   lens_dev: device int32 [num_seqs], lengths AFTER this step's append.  len 0 gives 0s.
 *   workspace: device scratch of >= hwkv_decode_workspace_bytes(), 16-byte aligned; its
 *              contents need no initialisation and are clobbered.  Launches that may run
 *              at the same time need distinct workspaces.
 * The stream-K kernel splits the layer's resident tiles evenly over a persistent grid and
 * merges partial results through per-(seq, head) arrival counters that the library keeps in
 * its own device memory (one set per layer); concurrent launches of the SAME layer race.
 * Other shapes (block_size not a multiple of 16, fp32 groups above 4) take the split-K
 * CUDA-core kernel and a merge kernel.
 * Errors: HWKV_ERR_INVALID_ARG, HWKV_ERR_ALIGNMENT, HWKV_ERR_WORKSPACE_TOO_SMALL,
 *         HWKV_ERR_UNSUPPORTED, HWKV_ERR_CUDA (launch failure). */
int hwkv_decode_attn(hwkv_pool_t pool, int layer, const void* q, int q_heads, float scale,
                     const int32_t* lens_dev, void* out, void* workspace, uint64_t workspace_bytes,
                     void* stream);

/* One decode step of one layer: hwkv_append followed by hwkv_decode_attn, with the same
 * results.  pos_dev holds the lengths BEFORE the append; attention runs at pos + 1.  On the
 * tensor-core path this is a single kernel: the CTA that streams the tile holding the new
 * token's slot takes the new rows from k_new / v_new and also writes them into the pool. */
int hwkv_append_decode_attn(hwkv_pool_t pool, int layer, const void* q, int q_heads, float scale,
                            const void* k_new, const void* v_new, const int32_t* pos_dev, void* out,
                            void* workspace, uint64_t workspace_bytes, void* stream);

/* Flags of hwkv_decode_attn_ex. */
#define HWKV_DECODE_EARLY_READS 1

/* hwkv_decode_attn (k_new = v_new = NULL; lens_dev = lengths after the append) or
 * hwkv_append_decode_attn (k_new, v_new given; lens_dev = positions before the append), with
 * flags:
 *   HWKV_DECODE_EARLY_READS  the caller guarantees that lens_dev, the block table and this
 *     layer's pool were last written by work that completed before the kernel that immediately
 *     precedes this call in `stream` started (e.g. lengths set once per step before layer 0,
 *     and a previous layer's attention just before).  The tensor-core kernel then computes its
 *     schedule and issues its first K/V loads while that kernel is still finishing (it is
 *     launched as a programmatic dependent), and waits for it only before it reads q, k_new,
 *     v_new or writes anything.  Same results as without the flag.  Do not set it on the call
 *     that follows the kernel which updates the lengths.  Ignored by the CUDA-core kernel.
 * Errors as hwkv_decode_attn; HWKV_ERR_INVALID_ARG for unknown flags. */
int hwkv_decode_attn_ex(hwkv_pool_t pool, int layer, const void* q, int q_heads, float scale, const void* k_new,
                        const void* v_new, const int32_t* lens_dev, void* out, void* workspace,
                        uint64_t workspace_bytes, int flags, void* stream);

/* Bytes of the static scratch array behind hwkv_decode_attn_noalloc. */
#define HWKV_NOALLOC_SCRATCH_BYTES (4u << 20)

/* hwkv_decode_attn without a workspace argument, for callers that cannot allocate device
 * memory where they run attention (during CUDA graph capture, under an allocator that owns
 * all device memory, inside hosts that forbid allocation after start-up).  The pages have
 * no counterpart: this is a service of this library, not a step of the method.
 *   Results are those of hwkv_decode_attn with the same arguments, bit for bit.  The split-K
 *   scratch is a fixed array of HWKV_NOALLOC_SCRATCH_BYTES (4 MiB) inside the library; the
 *   call allocates nothing (no cudaMalloc / cudaFree, no allocating library routine).
 *   A configuration whose scratch (hwkv_decode_workspace_bytes) exceeds the array is
 *   rejected with HWKV_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 *   The pool's device must be current (HWKV_ERR_INVALID_ARG otherwise).  The first call on a
 *   device looks up the array's device address there; under CUDA's default lazy module
 *   loading that lookup also loads the module holding the array and commits its 4 MiB on
 *   that device, which then stay committed until the process exits.  Make that first call
 *   before any stream capture.
 *   All calls share the one array and it keeps the last call's contents; nothing in it has
 *   to start at zero.  Calls whose kernels overlap on the GPU (other streams, other threads)
 *   race on the array: serialise them. */
int hwkv_decode_attn_noalloc(hwkv_pool_t pool, int layer, const void* q, int q_heads, float scale,
                             const int32_t* lens_dev, void* out, void* stream);

/* Chunked prefill of one layer ("Grouped-Cache Runtime": every head keeps only its window):
 * for each sequence s, a chunk of n_s new tokens at positions pos_s .. pos_s + n_s - 1 attends
 * causally, per KV head h, to the positions [max(0, p + 1 - w_h), p] of each token p -- the
 * ones before the chunk read from the head's ring in the pool, the others from the chunk --
 * and the chunk is then appended to the rings (slot p mod C; the last min(C, n_s) tokens are
 * written).  The result equals appending the tokens one by one and decoding each.
 *   q, out: device bf16 [num_seqs][n_max][q_heads][D]; k_new, v_new: [num_seqs][n_max][kv_heads][D];
 *   all 16-byte aligned.  pos_dev / n_dev: device int32 [num_seqs], lengths before the chunk
 *   and chunk lengths (0 <= n_s <= n_max, checked on the device; a bad sequence is skipped and
 *   flagged HWKV_DEVERR_NEG_LENGTH).  Rows of out at or past n_s are left untouched.
 *   workspace: device scratch of hwkv_prefill_workspace_bytes() bytes (16-byte aligned) that lets
 *   the library split long key streams over several CTAs and merge their fp32 partials; NULL or
 *   a smaller size runs one CTA per stream (same results up to rounding, slower for long windows
 *   at small batch).  Contents need no initialisation and are clobbered.
 * Needs a bf16 pool with block_size % 16 == 0 and q_heads = G * kv_heads with G <= 16
 * (HWKV_ERR_UNSUPPORTED otherwise).  Two or three kernels on `stream` (attention, the merge of
 * split streams, the append). */
int hwkv_prefill_attn(hwkv_pool_t pool, int layer, const void* q, int q_heads, float scale, const void* k_new,
                      const void* v_new, int n_max, const int32_t* pos_dev, const int32_t* n_dev, void* out,
                      void* workspace, uint64_t workspace_bytes, void* stream);

/* Bytes of workspace hwkv_prefill_attn uses to split the key streams of `layer` for chunks of up
 * to n_max tokens and q_heads query heads (0 when nothing would be split).  Host only; depends on
 * the geometry, the GPU's SM count and hwkv_set_prefill_config. */
int hwkv_prefill_workspace_bytes(hwkv_pool_t pool, int layer, int q_heads, int n_max, uint64_t* out);

/* The launch plan hwkv_prefill_attn uses for `layer` (host only: no pool, no device).  The
 * geometry arguments are those of hwkv_pool_create (bf16); num_sms is the GPU's SM count and
 * max_stages the cap of hwkv_set_prefill_config (0 = automatic).  For launch position
 * i < kv_heads: head_order[i] is the KV head, splits[i] its CTAs per (sequence, query-tile pair)
 * and split_stages[i] the 64-key stages each of them streams (CTA k of a split stream takes
 * stages [k * split_stages[i], (k + 1) * split_stages[i]) of it, so splits[i] * split_stages[i]
 * covers the longest stream of the head).  *workspace_bytes is what hwkv_prefill_workspace_bytes
 * returns for a pool of this geometry on such a GPU (0 when nothing is split).  The arrays hold
 * kv_heads entries each and are caller-owned.  Errors as hwkv_pool_bytes and
 * hwkv_prefill_attn's argument checks. */
int hwkv_prefill_plan(int layers, int kv_heads, int head_dim, int block_size, const int32_t* windows, int num_seqs,
                      int layer, int q_heads, int n_max, int num_sms, int max_stages, int32_t* head_order,
                      int32_t* splits, int32_t* split_stages, uint64_t* workspace_bytes);

/* Prefill configuration: max_stages caps the 64-key stages one CTA streams before its stream is
 * split, the same cap for every head (0 = automatic: a cap of about three waves of one CTA per
 * SM, then, for launches of at most 2048 unsplit CTAs, split counts refined per head against a
 * time model of the launch, planned once per (layer, q_heads, n_max) and kept).  Results differ
 * only by rounding. */
int hwkv_set_prefill_config(hwkv_pool_t pool, int max_stages);

/* Decode configuration.  kernel = HWKV_KERNEL_*.  split_tokens: tokens of one split-K chunk of
 * the CUDA-core kernel (0 = automatic; else a power of two in [16, 65536]).  workers: CTAs of
 * the tensor-core kernel's persistent grid (0 = automatic: every SM, as many CTAs as fit; 95% of
 * that when a layer's ring capacity is under 128 16-token tiles per CTA, so the next launch's
 * first CTAs find free slots).
 * Changes the workspace size.  Results differ between configurations only by rounding. */
int hwkv_set_decode_config(hwkv_pool_t pool, int split_tokens, int workers, int kernel);

/* Number of kernels this library has launched in this process (all pools, all devices).
 * Lets a caller count the launches inside a timed region. */
int hwkv_kernel_launches(uint64_t* out);

/* Distortion of a candidate window vector, supplied by the caller (e.g. measured with a
 * model).  windows: [kv_heads] candidate of `layer`; chosen: [layer][kv_heads] window vectors
 * already chosen for layers 0 .. layer-1 (execution order), so the distortion may depend on
 * them.  Return the distortion; smaller is better. */
typedef double (*hwkv_distortion_fn)(void* user, int layer, const int32_t* windows, const int32_t* chosen);

/* Host-side policy search of "HeadWiseKV: Budgeted Per-Head Cache Residency for Hybrid
 * Long-Context Language Models", section "SeqCalib": layers are visited in execution order;
 * for each layer the candidate window vector of smallest distortion whose cost fits the
 * remaining budget is chosen (ties: the first such candidate), and its cost is taken off the
 * budget.  The cost of a vector is its exact pool footprint, the bytes hwkv_pool_bytes predicts:
 * num_seqs * sum_h ceil(w_h / block_size) * block_size * head_dim * 2 * eb.
 *   candidates: host int32 [layers][num_candidates][kv_heads], every window >= 1.
 *   out_windows: host int32 [layers][kv_heads] (may be the windows argument of pool_create);
 *   out_choice: host int32 [layers] chosen candidate index; out_bytes: total pool bytes.
 * Pure host, needs no GPU.  Errors: HWKV_ERR_INVALID_ARG, HWKV_ERR_UNSUPPORTED, HWKV_ERR_BUDGET
 * (no candidate of some layer fits what is left of the budget; the message names the layer). */
int hwkv_seqcalib(int layers, int kv_heads, int head_dim, int block_size, int num_seqs, int dtype,
                  int num_candidates, const int32_t* candidates, hwkv_distortion_fn distortion, void* user,
                  uint64_t budget_bytes, int32_t* out_windows, int32_t* out_choice, uint64_t* out_bytes);

/* Synchronises `stream`, reads and clears the device error word.  *out_bits receives the
 * HWKV_DEVERR_* bits seen since the last call.  Returns HWKV_ERR_DEVICE_CHECK if any bit
 * was set, HWKV_OK otherwise. */
int hwkv_check_device_errors(hwkv_pool_t pool, void* stream, int32_t* out_bits);

#ifdef __cplusplus
}
#endif

#endif /* HWKV_H */
