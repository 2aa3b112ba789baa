// Host side of the hwkv C ABI: argument checks, pool geometry and block tables, the
// tensor map of the pool, decode planning, and the launches.
//
// Geometry follows "HeadWiseKV: Budgeted Per-Head Cache Residency for Hybrid Long-Context
// Language Models", section "Grouped-Cache Runtime" (ceil(w / block_size) blocks per head,
// pre-allocated before serving) and abstract (the footprint is exact before serving).
// Physical block ids start as the identity in (layer, seq, kv head, logical block) order.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <limits>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <tuple>
#include <vector>

#include "hwkv_internal.h"
#include "../../include/hwkv.h"

using namespace hwkv;

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return HWKV_OK;
}

// NVTX range of one library call, in the "hwkv" domain, with the layer as its payload, so a
// profile of a serving step attributes each append / decode / prefill launch to its call.
// Without a profiler attached a push or pop is a check of one function pointer.
nvtxDomainHandle_t nvtx_domain() {
  static nvtxDomainHandle_t d = nvtxDomainCreateA("hwkv");
  return d;
}

struct NvtxRange {
  explicit NvtxRange(const char* name, int layer) {
    nvtxEventAttributes_t ev;
    std::memset(&ev, 0, sizeof ev);
    ev.version = NVTX_VERSION;
    ev.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    ev.messageType = NVTX_MESSAGE_TYPE_ASCII;
    ev.message.ascii = name;
    ev.payloadType = NVTX_PAYLOAD_TYPE_INT32;
    ev.payload.iValue = layer;
    nvtxDomainRangePushEx(nvtx_domain(), &ev);
  }
  ~NvtxRange() { nvtxDomainRangePop(nvtx_domain()); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

#define HWKV_CUDA_TRY(expr, what)                                                           \
  do {                                                                                     \
    cudaError_t e_ = (expr);                                                               \
    if (e_ != cudaSuccess) return fail(HWKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e_)); \
  } while (0)

struct Geometry {
  int layers = 0, kv_heads = 0, head_dim = 0, block_size = 0, num_seqs = 0, dtype = 0, eb = 0;
  std::vector<int32_t> windows, nblk;   // [layers * kv_heads]
  std::vector<int64_t> tbl_base;        // [layers] table offset of (layer, seq 0, head 0)
  std::vector<int32_t> seq_stride;      // [layers] sum_h nblk
  int64_t total_blocks = 0;
  uint64_t pool_bytes = 0;
};

constexpr int64_t kInt32Max = std::numeric_limits<int32_t>::max();

int plan_geometry(int layers, int kv_heads, int head_dim, int block_size, const int32_t* windows, int num_seqs,
                  int dtype, Geometry* g) {
  if (layers < 1) return fail(HWKV_ERR_INVALID_ARG, "layers must be >= 1 (got %d)", layers);
  if (kv_heads < 1 || kv_heads > kMaxKvHeads)
    return fail(HWKV_ERR_UNSUPPORTED, "kv_heads must be in [1, %d] (got %d)", kMaxKvHeads, kv_heads);
  if (head_dim != 64 && head_dim != 128)
    return fail(HWKV_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", head_dim);
  if (block_size < 1) return fail(HWKV_ERR_INVALID_ARG, "block_size must be >= 1 (got %d)", block_size);
  if (num_seqs < 1) return fail(HWKV_ERR_INVALID_ARG, "num_seqs must be >= 1 (got %d)", num_seqs);
  if (dtype != HWKV_F32 && dtype != HWKV_BF16) return fail(HWKV_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  if (!windows) return fail(HWKV_ERR_INVALID_ARG, "windows is NULL");
  g->layers = layers;
  g->kv_heads = kv_heads;
  g->head_dim = head_dim;
  g->block_size = block_size;
  g->num_seqs = num_seqs;
  g->dtype = dtype;
  g->eb = dtype == HWKV_F32 ? 4 : 2;
  g->windows.assign(windows, windows + (size_t)layers * kv_heads);
  g->nblk.resize(g->windows.size());
  g->tbl_base.resize(layers);
  g->seq_stride.resize(layers);
  int64_t blocks = 0;
  for (int l = 0; l < layers; ++l) {
    int64_t per_seq = 0;
    for (int h = 0; h < kv_heads; ++h) {
      const int64_t w = g->windows[(size_t)l * kv_heads + h];
      if (w < 1) return fail(HWKV_ERR_INVALID_ARG, "window of layer %d head %d must be >= 1 (got %lld)", l, h, (long long)w);
      const int64_t nb = (w + block_size - 1) / block_size;  // ceil(w / block_size)
      if (nb * block_size > kInt32Max)
        return fail(HWKV_ERR_UNSUPPORTED, "ring of layer %d head %d exceeds 2^31 tokens", l, h);
      g->nblk[(size_t)l * kv_heads + h] = (int32_t)nb;
      per_seq += nb;
    }
    if (per_seq > kInt32Max) return fail(HWKV_ERR_UNSUPPORTED, "layer %d has more than 2^31 blocks per sequence", l);
    g->tbl_base[l] = blocks;
    g->seq_stride[l] = (int32_t)per_seq;
    blocks += per_seq * num_seqs;
    if (blocks * 2 * (int64_t)block_size > kInt32Max)
      return fail(HWKV_ERR_UNSUPPORTED, "pool exceeds 2^31 rows (blocks x 2 x block_size)");
  }
  g->total_blocks = blocks;
  g->pool_bytes = (uint64_t)blocks * 2u * (uint64_t)block_size * (uint64_t)head_dim * (uint64_t)g->eb;
  return HWKV_OK;
}

struct LayerPlan {
  int32_t split = 0;
  int32_t items = 0;
  bool multi_chunk = false;
  int32_t chunk_prefix[kMaxKvHeads + 1] = {};
};

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

void hwkv::count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int hwkv::set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

struct hwkv_pool {
  Geometry g;
  char* dev_pool = nullptr;
  void* d_meta = nullptr;
  int32_t* d_tbl = nullptr;
  int32_t* d_err = nullptr;
  // arrival counters of the tensor-core kernel, all kept at 0 between launches:
  // [layers][groups] final counters, then [layers][groups][merge_blocks] first-level ones
  uint32_t* d_counters = nullptr;
  int counter_merge_blocks = 0;
  std::vector<int32_t> h_tbl;
  int device = 0;
  int num_sms = 0;
  int ctas_per_sm[kGroupPads] = {0, 0, 0};  // tensor-core decode instances, by group pad
  int split_override = 0;
  int workers_override = 0;
  int64_t max_layer_tiles = 0;  // most 16-token ring tiles of one layer (all sequences and heads)
  int kernel_choice = HWKV_KERNEL_AUTO;
  std::vector<LayerPlan> plans;
  bool has_tmap = false;       // the pool's 2-D tensor map (16-row tiles)
  bool has_stage_map = false;  // bf16: the 3-D stage map of the prefill
  alignas(64) CUtensorMap tmap;
  // the pool as (head_dim, 2 * block_size rows, block): one box of stage_tb rows of 64 / stage_tb
  // consecutive blocks is 64 keys (K or V) of a prefill stage
  alignas(64) CUtensorMap stage_map;
  int stage_tb = 0;
  int prefill_max_stages = 0;  // cap on a prefill CTA's key stages (0 = automatic)
  // automatic prefill split counts per head, by (layer, group, chunk size)
  mutable std::map<std::tuple<int, int, int>, std::vector<int>> prefill_plans;
  mutable std::mutex prefill_plans_mu;
};

namespace {

// The stream-K decode kernel takes bf16 pools (tensor cores) and fp32 pools (CUDA cores, up to
// 4 query heads per KV head) whose block size is a multiple of 16 (one TMA box of 16 rows).
bool tc_eligible(const hwkv_pool* p) {
  return (p->g.dtype == HWKV_BF16 || p->g.dtype == HWKV_F32) && p->g.block_size % 16 == 0 && p->has_tmap;
}

bool tc_group_ok(const hwkv_pool* p, int group) { return p->g.dtype == HWKV_BF16 || group <= 4; }

bool use_tc(const hwkv_pool* p, int group) {
  if (p->kernel_choice == HWKV_KERNEL_SIMT) return false;
  return tc_eligible(p) && tc_group_ok(p, group);
}

// chunked prefill: bf16 pools with the 3-D stage map
bool prefill_eligible(const hwkv_pool* p) { return p->g.dtype == HWKV_BF16 && tc_eligible(p) && p->has_stage_map; }

void plan_decode(hwkv_pool* p) {
  const Geometry& g = p->g;
  p->plans.assign(g.layers, LayerPlan());
  for (int l = 0; l < g.layers; ++l) {
    LayerPlan& lp = p->plans[l];
    int64_t tokens = 0;
    for (int h = 0; h < g.kv_heads; ++h) tokens += (int64_t)g.nblk[(size_t)l * g.kv_heads + h] * g.block_size;
    tokens *= g.num_seqs;
    p->max_layer_tiles = std::max<int64_t>(p->max_layer_tiles, tokens / 16);
    int32_t split = p->split_override;
    if (split == 0) {
      // about four waves of two CTAs per SM; powers of two so the level-set windows
      // (1K .. 64K) split into equal chunks
      const int64_t want = tokens / std::max<int64_t>(1, 8LL * std::max(1, p->num_sms));
      split = 256;
      while (split < want && split < 2048) split <<= 1;
    }
    lp.split = split;
    lp.chunk_prefix[0] = 0;
    for (int h = 0; h < g.kv_heads; ++h) {
      const int64_t C = (int64_t)g.nblk[(size_t)l * g.kv_heads + h] * g.block_size;
      const int32_t n = (int32_t)((C + split - 1) / split);
      lp.chunk_prefix[h + 1] = lp.chunk_prefix[h] + n;
      if (n > 1) lp.multi_chunk = true;
    }
    lp.items = lp.chunk_prefix[g.kv_heads] * g.num_seqs;
  }
}

// Time model of a prefill launch for choosing its split, in units of one 64-key stage of one
// CTA (0.853 us on GB300, the same on every geometry measured).  A CTA costs its stages plus a
// fixed cost (tensor-memory and barrier setup, the Q load and first stage, the epilogue: ~7.2 us
// unsplit, ~8.8 us when it stores fp32 partials) and ~0.6 us before the next CTA starts on its
// SM; each split CTA adds ~0.047 us to the merge kernel.  CTAs are handed to SMs in launch order
// (one CTA per SM), each to the SM that frees first.  Measured per CTA with %globaltimer stamps:
// the model reproduces the spans of four long and full-geometry launches within 1%.
constexpr double kPfFixed = 8.4, kPfFixedSplit = 10.3, kPfGap = 0.7, kPfMergePerCta = 0.055, kPfEmptyCta = 1.2;
// the split search runs only for launches of at most this many unsplit CTAs (beyond that, many
// CTAs per SM balance well as they are)
constexpr int64_t kPfSearchMaxCtas = 2048;

struct PfHead {
  int h, window, maxst;
  std::vector<int> stages;  // estimated stages of each tile pair's key stream
};

// Launch order of the heads for splits sp (indexed like hd): longest CTAs first (the classic
// longest-processing-time order), then longer windows, then head index.
std::vector<int> prefill_launch_order(const std::vector<PfHead>& hd, const std::vector<int>& sp) {
  std::vector<int> order(hd.size());
  for (size_t i = 0; i < hd.size(); ++i) order[i] = (int)i;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
    const int cx = (hd[x].maxst + sp[x] - 1) / sp[x], cy = (hd[y].maxst + sp[y] - 1) / sp[y];
    if (cx != cy) return cx > cy;
    return hd[x].window > hd[y].window;
  });
  return order;
}

double predict_prefill(const std::vector<PfHead>& hd, const std::vector<int>& sp, int seqs, int sms) {
  std::vector<double> free_at((size_t)std::max(1, sms), 0.0);  // min-heap of SM free times
  double merge = 0.0;
  for (int i : prefill_launch_order(hd, sp)) {
    const PfHead& e = hd[(size_t)i];
    const int ss = (e.maxst + sp[i] - 1) / sp[i];
    for (int s = 0; s < seqs; ++s)
      for (int nst : e.stages)
        for (int k = 0; k < sp[i]; ++k) {
          const int nloc = std::min(nst, (k + 1) * ss) - k * ss;
          const double d = nloc > 0 ? nloc + (sp[i] > 1 ? kPfFixedSplit : kPfFixed) + kPfGap : kPfEmptyCta;
          std::pop_heap(free_at.begin(), free_at.end(), std::greater<double>());
          free_at.back() += d;
          std::push_heap(free_at.begin(), free_at.end(), std::greater<double>());
        }
    if (sp[i] > 1) merge += kPfMergePerCta * seqs * (double)e.stages.size() * sp[i];
  }
  return *std::max_element(free_at.begin(), free_at.end()) + merge;
}

// Work plan of one prefill launch.  A head whose key stream (upper bound over lengths) is much
// longer than an even share of the work (about three waves of one CTA per SM, or the configured
// stage cap) is split over several CTAs per (seq, query-tile pair), whose fp32 partials a merge
// kernel combines.  In the automatic mode the split counts are then refined per head by a
// coordinate search on the time model above, and the heads launch longest CTAs first; the plan
// is kept per (layer, group, chunk size).  Returns the workspace bytes the split needs (0 when
// nothing is split).  allow_split = false plans one CTA per stream.
uint64_t plan_prefill(const hwkv_pool* p, int layer, int G, int n_max, bool allow_split, PrefillArgs& a) {
  const Geometry& g = p->g;
  const int H = g.kv_heads;
  const int* win = &g.windows[(size_t)layer * H];
  const int per_pair = prefill_tokens_per_cta(G);
  const int pairs = (n_max + per_pair - 1) / per_pair;
  const int64_t items = (int64_t)g.num_seqs * pairs;
  std::vector<PfHead> hd((size_t)H);
  int64_t work = 0;
  for (int h = 0; h < H; ++h) {
    const int C = g.nblk[(size_t)layer * H + h] * g.block_size;
    hd[(size_t)h].h = h;
    hd[(size_t)h].window = win[h];
    hd[(size_t)h].maxst = prefill_max_stages(win[h], C, G, n_max);
    work += items * hd[(size_t)h].maxst;
  }
  std::vector<int> sp((size_t)H, 1);
  std::vector<int> order;
  if (allow_split) {
    const bool automatic = p->prefill_max_stages <= 0;
    const int64_t target = !automatic ? p->prefill_max_stages
                                      : std::max<int64_t>(16, (work + 3LL * p->num_sms - 1) / (3LL * p->num_sms));
    for (int h = 0; h < H; ++h)
      if (hd[(size_t)h].maxst > target)
        sp[(size_t)h] = (int)std::min<int64_t>(64, (hd[(size_t)h].maxst + target - 1) / target);
    if (automatic && items * H <= kPfSearchMaxCtas) {
      std::lock_guard<std::mutex> lock(p->prefill_plans_mu);
      const auto key = std::make_tuple(layer, G, n_max);
      auto it = p->prefill_plans.find(key);
      if (it == p->prefill_plans.end()) {
        for (int h = 0; h < H; ++h) {
          const int C = g.nblk[(size_t)layer * H + h] * g.block_size;
          for (int qt = 0; qt < pairs; ++qt)
            hd[(size_t)h].stages.push_back(prefill_stages_estimate(win[h], C, G, n_max, qt * per_pair));
        }
        const double start = predict_prefill(hd, sp, g.num_seqs, p->num_sms);
        std::vector<int> best = sp;
        double best_t = start;
        for (int round = 0; round < 6; ++round) {
          bool improved = false;
          for (int h = 0; h < H; ++h)
            for (int d : {-1, 1, 2}) {
              std::vector<int> t = best;
              t[(size_t)h] += d;
              if (t[(size_t)h] < 1 || t[(size_t)h] > 64) continue;
              const double v = predict_prefill(hd, t, g.num_seqs, p->num_sms);
              if (v < best_t - 1e-9) {
                best_t = v;
                best = t;
                improved = true;
              }
            }
          if (!improved) break;
        }
        // keep the plain rule unless the model predicts a clear gain
        if (best_t > 0.98 * start) best = sp;
        it = p->prefill_plans.emplace(key, best).first;
      }
      sp = it->second;
      order = prefill_launch_order(hd, sp);
    }
  }
  if (order.empty()) {  // heads by decreasing window
    order.resize((size_t)H);
    for (int h = 0; h < H; ++h) order[(size_t)h] = h;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return win[x] > win[y]; });
  }
  int64_t ctas = 0;
  bool any = false;
  for (int i = 0; i < H; ++i) {
    const int h = order[(size_t)i];
    const int n_sp = sp[(size_t)h];
    a.head_order[i] = h;
    a.splits[i] = n_sp;
    a.split_stages[i] = (hd[(size_t)h].maxst + n_sp - 1) / n_sp;
    a.head_ctas[i] = (int32_t)ctas;
    ctas += items * n_sp;
    any = any || n_sp > 1;
  }
  a.head_ctas[H] = (int32_t)ctas;
  a.q_tiles = pairs;
  return any ? (uint64_t)ctas * 2 * 128 * ((uint64_t)g.head_dim + 2) * sizeof(float) : 0;
}

// Persistent CTAs of the tensor-core kernel: every resident slot, except for small layers
// (under 128 tiles of ring capacity per slot, a small batch): there about 5% of the slots stay
// free, so the next launch's first CTAs run their schedule and first loads while this launch
// finishes (batch 1 at 161K: +3% tokens/s; larger layers gain nothing and lose a little).
int tc_workers(const hwkv_pool* p, int group) {
  if (p->workers_override > 0) return p->workers_override;
  const int per_sm = p->ctas_per_sm[decode_tc_pad_index(group)];
  const int full = std::max(1, p->num_sms * std::max(1, per_sm));
  if (p->max_layer_tiles < 128LL * full) return std::max(1, full * 95 / 100);
  return full;
}

// first-level merge blocks per head for a grid of `workers` CTAs
int merge_blocks_for(int workers) { return (workers + kMergeBlock - 1) / kMergeBlock + 1; }

int max_tc_workers(const hwkv_pool* p) { return std::max({tc_workers(p, 4), tc_workers(p, 8), tc_workers(p, 16)}); }

// Workspace regions (each 256-byte aligned): partials [slots][G][D] floats, their (m, l)
// [slots][G][2]; for the tensor-core kernel also the second-level partials and (m, l).
// Partial slots: CUDA-core kernel one per chunk item; tensor-core kernel one per (group, CTA)
// pair along the tile line (at most groups + CTAs), second level groups x merge blocks.
struct WorkspaceLayout {
  int64_t slots1 = 0, slots2 = 0;
  uint64_t acc1 = 0, ml1 = 0, acc2 = 0, ml2 = 0, total = 0;
};

uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

WorkspaceLayout workspace_layout(const hwkv_pool* p, int group) {
  WorkspaceLayout w;
  const int64_t groups = (int64_t)p->g.num_seqs * p->g.kv_heads;
  if (use_tc(p, group)) {
    w.slots1 = groups + tc_workers(p, group);
    w.slots2 = groups * merge_blocks_for(tc_workers(p, group));
  } else {
    for (const LayerPlan& lp : p->plans)
      if (lp.multi_chunk) w.slots1 = std::max<int64_t>(w.slots1, lp.items);
  }
  const uint64_t D = (uint64_t)p->g.head_dim;
  w.acc1 = 0;
  w.ml1 = align256(w.acc1 + (uint64_t)w.slots1 * group * D * 4);
  w.acc2 = align256(w.ml1 + (uint64_t)w.slots1 * group * 2 * 4);
  w.ml2 = align256(w.acc2 + (uint64_t)w.slots2 * group * D * 4);
  w.total = w.slots1 + w.slots2 > 0 ? align256(w.ml2 + (uint64_t)w.slots2 * group * 2 * 4) : 0;
  return w;
}

uint64_t workspace_bytes(const hwkv_pool* p, int group) { return workspace_layout(p, group).total; }

// (Re)allocates the arrival counters for the current grid size, zeroed.
int ensure_counters(hwkv_pool* p) {
  const int mb = merge_blocks_for(max_tc_workers(p));
  if (p->d_counters && mb <= p->counter_merge_blocks) return HWKV_OK;
  const size_t groups = (size_t)p->g.num_seqs * p->g.kv_heads;
  const size_t n = (size_t)p->g.layers * groups * (1 + (size_t)mb);
  uint32_t* c = nullptr;
  HWKV_CUDA_TRY(cudaMalloc(&c, n * sizeof(uint32_t)), "cudaMalloc of the arrival counters");
  cudaError_t e = cudaMemset(c, 0, n * sizeof(uint32_t));
  if (e != cudaSuccess) {
    cudaFree(c);
    return fail(HWKV_ERR_CUDA, "cudaMemset of the arrival counters: %s", cudaGetErrorString(e));
  }
  if (p->d_counters) {
    cudaDeviceSynchronize();  // no launch may still use the old counters
    cudaFree(p->d_counters);
  }
  p->d_counters = c;
  p->counter_merge_blocks = mb;
  return HWKV_OK;
}

size_t counter_count(const hwkv_pool* p) {
  return (size_t)p->g.layers * p->g.num_seqs * p->g.kv_heads * (1 + (size_t)p->counter_merge_blocks);
}

int check_device(const hwkv_pool* p) {
  int dev = -1;
  HWKV_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev != p->device) return fail(HWKV_ERR_INVALID_ARG, "pool lives on device %d but device %d is current", p->device, dev);
  return HWKV_OK;
}

}  // namespace

int hwkv::check_pool_device(const hwkv_pool* p) { return check_device(p); }

namespace {

PoolView pool_view(const hwkv_pool* p) {
  PoolView v;
  v.pool = p->dev_pool;
  v.tbl = p->d_tbl;
  v.err = p->d_err;
  v.total_blocks = p->g.total_blocks;
  v.block_size = p->g.block_size;
  v.head_dim = p->g.head_dim;
  v.kv_heads = p->g.kv_heads;
  v.num_seqs = p->g.num_seqs;
  v.elem_bytes = p->g.eb;
  return v;
}

LayerGeom layer_geom(const hwkv_pool* p, int layer) {
  const Geometry& g = p->g;
  LayerGeom lg;
  std::memset(&lg, 0, sizeof lg);
  lg.tbl_base = g.tbl_base[layer];
  lg.tbl_seq_stride = g.seq_stride[layer];
  lg.nblk_prefix[0] = 0;
  for (int h = 0; h < g.kv_heads; ++h) {
    lg.nblk_prefix[h + 1] = lg.nblk_prefix[h] + g.nblk[(size_t)layer * g.kv_heads + h];
    lg.window[h] = g.windows[(size_t)layer * g.kv_heads + h];
  }
  return lg;
}

}  // namespace

extern "C" {

int hwkv_abi_version(void) { return HWKV_ABI_VERSION; }

const char* hwkv_last_error(void) { return g_last_error.c_str(); }

const char* hwkv_status_string(int status) {
  switch (status) {
    case HWKV_OK: return "HWKV_OK";
    case HWKV_ERR_INVALID_ARG: return "HWKV_ERR_INVALID_ARG";
    case HWKV_ERR_ALIGNMENT: return "HWKV_ERR_ALIGNMENT";
    case HWKV_ERR_POOL_TOO_SMALL: return "HWKV_ERR_POOL_TOO_SMALL";
    case HWKV_ERR_CUDA: return "HWKV_ERR_CUDA";
    case HWKV_ERR_DEVICE_CHECK: return "HWKV_ERR_DEVICE_CHECK";
    case HWKV_ERR_UNSUPPORTED: return "HWKV_ERR_UNSUPPORTED";
    case HWKV_ERR_WORKSPACE_TOO_SMALL: return "HWKV_ERR_WORKSPACE_TOO_SMALL";
    case HWKV_ERR_BUDGET: return "HWKV_ERR_BUDGET";
    default: return "HWKV_ERR_UNKNOWN";
  }
}

int hwkv_pool_bytes(int layers, int kv_heads, int head_dim, int block_size, const int32_t* windows, int num_seqs,
                    int dtype, uint64_t* out_bytes) {
  if (!out_bytes) return fail(HWKV_ERR_INVALID_ARG, "out_bytes is NULL");
  Geometry g;
  const int rc = plan_geometry(layers, kv_heads, head_dim, block_size, windows, num_seqs, dtype, &g);
  if (rc != HWKV_OK) return rc;
  *out_bytes = g.pool_bytes;
  return ok();
}

int hwkv_pool_create(int layers, int kv_heads, int head_dim, int block_size, const int32_t* windows, int num_seqs,
                     int dtype, void* dev_pool, uint64_t dev_pool_bytes, void* stream, hwkv_pool_t* out) {
  if (!out) return fail(HWKV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  Geometry g;
  int rc = plan_geometry(layers, kv_heads, head_dim, block_size, windows, num_seqs, dtype, &g);
  if (rc != HWKV_OK) return rc;
  if (!dev_pool) return fail(HWKV_ERR_INVALID_ARG, "dev_pool is NULL");
  if (!aligned(dev_pool, 256)) return fail(HWKV_ERR_ALIGNMENT, "dev_pool must be 256-byte aligned");
  if (dev_pool_bytes < g.pool_bytes)
    return fail(HWKV_ERR_POOL_TOO_SMALL, "pool buffer holds %llu bytes, the windows need %llu",
                (unsigned long long)dev_pool_bytes, (unsigned long long)g.pool_bytes);
  int dev = 0;
  HWKV_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
  cudaPointerAttributes attr;
  HWKV_CUDA_TRY(cudaPointerGetAttributes(&attr, dev_pool), "cudaPointerGetAttributes");
  if ((attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) || attr.device != dev)
    return fail(HWKV_ERR_INVALID_ARG, "dev_pool is not device memory of the current device %d", dev);

  hwkv_pool* p = new (std::nothrow) hwkv_pool();
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "out of host memory");
  p->g = std::move(g);
  p->dev_pool = static_cast<char*>(dev_pool);
  p->device = dev;
  cudaError_t e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    delete p;
    return fail(HWKV_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  }
  const size_t tbl_bytes = ((size_t)p->g.total_blocks * sizeof(int32_t) + 255) & ~(size_t)255;
  e = cudaMalloc(&p->d_meta, tbl_bytes + 256);
  if (e != cudaSuccess) {
    delete p;
    return fail(HWKV_ERR_CUDA, "cudaMalloc of the block table: %s", cudaGetErrorString(e));
  }
  p->d_tbl = static_cast<int32_t*>(p->d_meta);
  p->d_err = reinterpret_cast<int32_t*>(static_cast<char*>(p->d_meta) + tbl_bytes);
  p->h_tbl.resize((size_t)p->g.total_blocks);
  for (int64_t i = 0; i < p->g.total_blocks; ++i) p->h_tbl[(size_t)i] = (int32_t)i;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto cleanup_fail = [&](const char* what, cudaError_t err) {
    cudaStreamSynchronize(st);
    cudaFree(p->d_meta);
    delete p;
    return fail(HWKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
  };
  if ((e = cudaMemcpyAsync(p->d_tbl, p->h_tbl.data(), (size_t)p->g.total_blocks * sizeof(int32_t),
                           cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return cleanup_fail("upload of the block table", e);
  if ((e = cudaMemsetAsync(p->d_err, 0, 256, st)) != cudaSuccess) return cleanup_fail("cudaMemsetAsync", e);
  if ((e = cudaMemsetAsync(p->dev_pool, 0, p->g.pool_bytes, st)) != cudaSuccess)
    return cleanup_fail("zero-fill of the pool", e);
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cleanup_fail("cudaStreamSynchronize", e);

  if (p->g.dtype == HWKV_F32 && p->g.block_size % 16 == 0) {
    // fp32: boxes of 16 rows x 32 elements (128 bytes), the decode kernel's tiles
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode) {
      const int64_t rows = p->g.total_blocks * 2 * p->g.block_size;
      cuuint64_t dims[2] = {(cuuint64_t)p->g.head_dim, (cuuint64_t)rows};
      cuuint64_t strides[1] = {(cuuint64_t)p->g.head_dim * 4};
      cuuint32_t box[2] = {32, 16};
      cuuint32_t estr[2] = {1, 1};
      CUresult cr = encode(&p->tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p->dev_pool, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      p->has_tmap = cr == CUDA_SUCCESS;
    }
  }
  if (p->g.dtype == HWKV_BF16 && p->g.block_size % 16 == 0) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode) {
      const int64_t rows = p->g.total_blocks * 2 * p->g.block_size;
      cuuint64_t dims[2] = {(cuuint64_t)p->g.head_dim, (cuuint64_t)rows};
      cuuint64_t strides[1] = {(cuuint64_t)p->g.head_dim * 2};
      cuuint32_t box[2] = {64, 16};
      cuuint32_t estr[2] = {1, 1};
      CUresult cr = encode(&p->tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p->dev_pool, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      const int bs = p->g.block_size;
      const int tb = bs == 16 ? 16 : bs == 32 ? 32 : (bs % 64 == 0 ? 64 : 16);
      cuuint64_t sdims[3] = {(cuuint64_t)p->g.head_dim, (cuuint64_t)(2 * bs), (cuuint64_t)p->g.total_blocks};
      cuuint64_t sstrides[2] = {(cuuint64_t)p->g.head_dim * 2, (cuuint64_t)2 * bs * p->g.head_dim * 2};
      cuuint32_t sbox[3] = {64, (cuuint32_t)tb, (cuuint32_t)(64 / tb)};
      cuuint32_t sestr[3] = {1, 1, 1};
      CUresult cr2 = encode(&p->stage_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p->dev_pool, sdims, sstrides, sbox, sestr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      p->stage_tb = (bs == 16 || bs == 32 || bs % 64 == 0) ? tb : 0;
      p->has_tmap = cr == CUDA_SUCCESS && cr2 == CUDA_SUCCESS;
      p->has_stage_map = p->has_tmap;
    }
  }
  if (p->has_tmap) {
    e = configure_decode_tc(p->g.head_dim, p->g.dtype, p->ctas_per_sm);
    if (e != cudaSuccess) return cleanup_fail("cudaFuncSetAttribute", e);
  }
  plan_decode(p);
  if (p->has_tmap) {
    const int crc = ensure_counters(p);
    if (crc != HWKV_OK) {
      const std::string msg = g_last_error;
      cudaFree(p->d_meta);
      delete p;
      return fail(crc, "%s", msg.c_str());
    }
  }
  *out = p;
  return ok();
}

int hwkv_pool_destroy(hwkv_pool_t p) {
  if (!p) return ok();
  if (p->d_counters) cudaFree(p->d_counters);
  cudaError_t e = cudaFree(p->d_meta);
  delete p;
  if (e != cudaSuccess) return fail(HWKV_ERR_CUDA, "cudaFree: %s", cudaGetErrorString(e));
  return ok();
}

int hwkv_pool_geometry(hwkv_pool_t p, uint64_t* pool_bytes, int64_t* total_blocks, int64_t* block_bytes) {
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "pool is NULL");
  if (pool_bytes) *pool_bytes = p->g.pool_bytes;
  if (total_blocks) *total_blocks = p->g.total_blocks;
  if (block_bytes) *block_bytes = 2LL * p->g.block_size * p->g.head_dim * p->g.eb;
  return ok();
}

int hwkv_block_table(hwkv_pool_t p, int seq, int layer, int kv_head, int32_t* host_out, int cap, int* n) {
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "pool is NULL");
  const Geometry& g = p->g;
  if (seq < 0 || seq >= g.num_seqs || layer < 0 || layer >= g.layers || kv_head < 0 || kv_head >= g.kv_heads)
    return fail(HWKV_ERR_INVALID_ARG, "seq/layer/kv_head out of range");
  const int32_t nb = g.nblk[(size_t)layer * g.kv_heads + kv_head];
  if (n) *n = nb;
  if (!host_out && cap > 0) return fail(HWKV_ERR_INVALID_ARG, "host_out is NULL");
  int64_t off = g.tbl_base[layer] + (int64_t)seq * g.seq_stride[layer];
  for (int h = 0; h < kv_head; ++h) off += g.nblk[(size_t)layer * g.kv_heads + h];
  for (int j = 0; j < nb && j < cap; ++j) host_out[j] = p->h_tbl[(size_t)(off + j)];
  return ok();
}

int hwkv_set_block_table(hwkv_pool_t p, const int32_t* host_table, int64_t n, void* stream) {
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "pool is NULL");
  if (!host_table) return fail(HWKV_ERR_INVALID_ARG, "host_table is NULL");
  if (n != p->g.total_blocks)
    return fail(HWKV_ERR_INVALID_ARG, "table has %lld entries, the pool %lld blocks", (long long)n,
                (long long)p->g.total_blocks);
  std::vector<char> seen((size_t)n, 0);
  for (int64_t i = 0; i < n; ++i) {
    const int32_t b = host_table[i];
    if (b < 0 || b >= n || seen[(size_t)b])
      return fail(HWKV_ERR_INVALID_ARG, "table entry %lld (%d) is out of range or repeated", (long long)i, b);
    seen[(size_t)b] = 1;
  }
  int rc = check_device(p);
  if (rc != HWKV_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  HWKV_CUDA_TRY(cudaMemcpyAsync(p->d_tbl, host_table, (size_t)n * sizeof(int32_t), cudaMemcpyHostToDevice, st),
                "upload of the block table");
  HWKV_CUDA_TRY(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  p->h_tbl.assign(host_table, host_table + n);
  return ok();
}

int hwkv_materialize(hwkv_pool_t p, int layer, const void* k_full, const void* v_full, int64_t seq_stride,
                     int64_t head_stride, int64_t max_len, const int32_t* lens_dev, void* stream) {
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "pool is NULL");
  const Geometry& g = p->g;
  if (layer < 0 || layer >= g.layers) return fail(HWKV_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (seq_stride < 0 || head_stride < 0 || max_len < 0) return fail(HWKV_ERR_INVALID_ARG, "negative stride or max_len");
  if (max_len == 0) return ok();  // an empty prefill: nothing is read or written
  if (!k_full || !v_full || !lens_dev) return fail(HWKV_ERR_INVALID_ARG, "NULL tensor argument");
  if (!aligned(k_full, 16) || !aligned(v_full, 16) || !aligned(lens_dev, 4))
    return fail(HWKV_ERR_ALIGNMENT, "k_full / v_full must be 16-byte aligned, lens 4-byte aligned");
  if ((seq_stride * g.eb) % 16 != 0 || (head_stride * g.eb) % 16 != 0)
    return fail(HWKV_ERR_ALIGNMENT, "seq_stride and head_stride must be multiples of 16 bytes");
  if (max_len > kInt32Max) return fail(HWKV_ERR_INVALID_ARG, "max_len must be below 2^31");
  int rc = check_device(p);
  if (rc != HWKV_OK) return rc;
  NvtxRange range_("hwkv_materialize", layer);
  CopyArgs a;
  std::memset(&a, 0, sizeof a);
  a.pv = pool_view(p);
  a.g = layer_geom(p, layer);
  a.k = k_full;
  a.v = v_full;
  a.seq_stride = seq_stride;
  a.head_stride = head_stride;
  a.max_len = max_len;
  a.lens = lens_dev;
  int64_t max_rows = 0;
  for (int h = 0; h < g.kv_heads; ++h) max_rows = std::max<int64_t>(max_rows, a.g.window[h]);
  max_rows = std::min<int64_t>(max_rows, max_len);
  if (max_rows == 0) return ok();
  HWKV_CUDA_TRY(launch_materialize(a, g.dtype, (int)max_rows, static_cast<cudaStream_t>(stream)), "materialize launch");
  return ok();
}

int hwkv_append(hwkv_pool_t p, int layer, const void* k_new, const void* v_new, const int32_t* pos_dev, void* stream) {
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "pool is NULL");
  const Geometry& g = p->g;
  if (layer < 0 || layer >= g.layers) return fail(HWKV_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (!k_new || !v_new || !pos_dev) return fail(HWKV_ERR_INVALID_ARG, "NULL tensor argument");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(pos_dev, 4))
    return fail(HWKV_ERR_ALIGNMENT, "k_new / v_new must be 16-byte aligned, pos 4-byte aligned");
  int rc = check_device(p);
  if (rc != HWKV_OK) return rc;
  NvtxRange range_("hwkv_append", layer);
  CopyArgs a;
  std::memset(&a, 0, sizeof a);
  a.pv = pool_view(p);
  a.g = layer_geom(p, layer);
  a.k = k_new;
  a.v = v_new;
  a.lens = pos_dev;
  HWKV_CUDA_TRY(launch_append(a, g.dtype, static_cast<cudaStream_t>(stream)), "append launch");
  return ok();
}

int hwkv_advance_positions(hwkv_pool_t p, const int32_t* pos_dev, int32_t* out_dev, int32_t delta, void* stream) {
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "pool is NULL");
  if (!pos_dev || !out_dev) return fail(HWKV_ERR_INVALID_ARG, "NULL tensor argument");
  if (!aligned(pos_dev, 4) || !aligned(out_dev, 4)) return fail(HWKV_ERR_ALIGNMENT, "positions must be 4-byte aligned");
  int rc = check_device(p);
  if (rc != HWKV_OK) return rc;
  HWKV_CUDA_TRY(launch_advance_positions(pos_dev, out_dev, p->g.num_seqs, delta, static_cast<cudaStream_t>(stream)),
                "advance-positions launch");
  return ok();
}

int hwkv_wait_selftest(uint32_t limit_us, int32_t* out_dev, void* stream) {
  if (limit_us < 1 || limit_us > 2000000u) return fail(HWKV_ERR_INVALID_ARG, "limit_us must be in [1, 2000000]");
  if (!out_dev) return fail(HWKV_ERR_INVALID_ARG, "NULL output");
  if (!aligned(out_dev, 4)) return fail(HWKV_ERR_ALIGNMENT, "out_dev must be 4-byte aligned");
  HWKV_CUDA_TRY(launch_wait_selftest(out_dev, limit_us, static_cast<cudaStream_t>(stream)), "wait self-test launch");
  return ok();
}

int hwkv_decode_workspace_bytes(hwkv_pool_t p, int q_heads, uint64_t* out) {
  if (!p || !out) return fail(HWKV_ERR_INVALID_ARG, "NULL argument");
  if (q_heads < p->g.kv_heads || q_heads % p->g.kv_heads != 0 || q_heads / p->g.kv_heads > kMaxGroup)
    return fail(HWKV_ERR_UNSUPPORTED, "q_heads must be G * kv_heads with 1 <= G <= %d", kMaxGroup);
  *out = workspace_bytes(p, q_heads / p->g.kv_heads);
  return ok();
}

}  // extern "C"

namespace {

// Shared body of hwkv_decode_attn (len_add 0, no new rows) and hwkv_append_decode_attn
// (len_add 1: lens are the positions before the append, k_new / v_new are appended).
int decode_common(hwkv_pool_t p, int layer, const void* q, int q_heads, float scale, const int32_t* lens_dev,
                  int len_add, const void* k_new, const void* v_new, void* out, void* workspace, uint64_t ws_bytes,
                  int flags, void* stream) {
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "pool is NULL");
  if (flags & ~HWKV_DECODE_EARLY_READS) return fail(HWKV_ERR_INVALID_ARG, "unknown decode flags %#x", flags);
  const Geometry& g = p->g;
  if (layer < 0 || layer >= g.layers) return fail(HWKV_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (q_heads < g.kv_heads || q_heads % g.kv_heads != 0 || q_heads / g.kv_heads > kMaxGroup)
    return fail(HWKV_ERR_UNSUPPORTED, "q_heads must be G * kv_heads with 1 <= G <= %d (got %d)", kMaxGroup, q_heads);
  if (!(scale == scale) || scale == std::numeric_limits<float>::infinity() ||
      scale == -std::numeric_limits<float>::infinity())
    return fail(HWKV_ERR_INVALID_ARG, "scale must be finite");
  if (!q || !out || !lens_dev) return fail(HWKV_ERR_INVALID_ARG, "NULL tensor argument");
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(lens_dev, 4))
    return fail(HWKV_ERR_ALIGNMENT, "q / out must be 16-byte aligned, lens 4-byte aligned");
  if (len_add) {
    if (!k_new || !v_new) return fail(HWKV_ERR_INVALID_ARG, "NULL k_new / v_new");
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return fail(HWKV_ERR_ALIGNMENT, "k_new / v_new must be 16-byte aligned");
  }
  const int G = q_heads / g.kv_heads;
  const LayerPlan& lp = p->plans[layer];
  const bool tc = use_tc(p, G);
  const uint64_t need = workspace_bytes(p, G);
  if (tc || lp.multi_chunk) {
    if (!workspace || ws_bytes < need)
      return fail(HWKV_ERR_WORKSPACE_TOO_SMALL, "workspace holds %llu bytes, decode needs %llu",
                  (unsigned long long)ws_bytes, (unsigned long long)need);
    if (!aligned(workspace, 16)) return fail(HWKV_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  }
  int rc = check_device(p);
  if (rc != HWKV_OK) return rc;
  NvtxRange range_(len_add ? "hwkv_append_decode_attn" : "hwkv_decode_attn", layer);
  if (p->kernel_choice == HWKV_KERNEL_TENSOR && !(tc_eligible(p) && tc_group_ok(p, G)))
    return fail(HWKV_ERR_UNSUPPORTED,
                "the stream-K decode needs block_size % 16 == 0, and up to 4 query heads per KV head for fp32");

  DecodeArgs a;
  std::memset(&a, 0, sizeof a);
  a.pv = pool_view(p);
  a.g = layer_geom(p, layer);
  a.q = q;
  a.out = out;
  a.lens = lens_dev;
  a.len_add = len_add;
  a.early = (flags & HWKV_DECODE_EARLY_READS) ? 1 : 0;
  const WorkspaceLayout wl = workspace_layout(p, G);
  char* ws = static_cast<char*>(workspace);
  a.part_acc = ws ? reinterpret_cast<float*>(ws + wl.acc1) : nullptr;
  a.part_ml = ws ? reinterpret_cast<float*>(ws + wl.ml1) : nullptr;
  a.part2_acc = ws ? reinterpret_cast<float*>(ws + wl.acc2) : nullptr;
  a.part2_ml = ws ? reinterpret_cast<float*>(ws + wl.ml2) : nullptr;
  if (tc) {
    const int64_t groups = (int64_t)g.num_seqs * g.kv_heads;
    a.merge_blocks = merge_blocks_for(tc_workers(p, G));
    a.counters = p->d_counters + (int64_t)layer * groups;
    a.counters1 = p->d_counters + (int64_t)g.layers * groups + (int64_t)layer * groups * p->counter_merge_blocks;
  }
  a.scale_log2 = scale * 1.4426950408889634f;
  a.group = G;
  a.split_tokens = lp.split;
  std::memcpy(a.chunk_prefix, lp.chunk_prefix, sizeof a.chunk_prefix);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (tc) {
    a.k_new = len_add ? k_new : nullptr;  // appended inside the kernel
    a.v_new = len_add ? v_new : nullptr;
    HWKV_CUDA_TRY(launch_decode_tc(a, &p->tmap, tc_workers(p, G), st), "decode launch");
    return ok();
  }
  if (len_add) {
    CopyArgs c;
    std::memset(&c, 0, sizeof c);
    c.pv = a.pv;
    c.g = a.g;
    c.k = k_new;
    c.v = v_new;
    c.lens = lens_dev;
    HWKV_CUDA_TRY(launch_append(c, g.dtype, st), "append launch");
  }
  HWKV_CUDA_TRY(launch_decode_simt(a, g.dtype, lp.items, st), "decode launch");
  if (lp.multi_chunk) HWKV_CUDA_TRY(launch_combine(a, g.dtype, st), "combine launch");
  return ok();
}

}  // namespace

extern "C" {

int hwkv_decode_attn(hwkv_pool_t p, int layer, const void* q, int q_heads, float scale, const int32_t* lens_dev,
                     void* out, void* workspace, uint64_t ws_bytes, void* stream) {
  return decode_common(p, layer, q, q_heads, scale, lens_dev, 0, nullptr, nullptr, out, workspace, ws_bytes, 0,
                       stream);
}

int hwkv_decode_attn_ex(hwkv_pool_t p, int layer, const void* q, int q_heads, float scale, const void* k_new,
                        const void* v_new, const int32_t* lens_dev, void* out, void* workspace, uint64_t ws_bytes,
                        int flags, void* stream) {
  const bool fused = k_new != nullptr || v_new != nullptr;
  return decode_common(p, layer, q, q_heads, scale, lens_dev, fused ? 1 : 0, k_new, v_new, out, workspace, ws_bytes,
                       flags, stream);
}

int hwkv_append_decode_attn(hwkv_pool_t p, int layer, const void* q, int q_heads, float scale, const void* k_new,
                            const void* v_new, const int32_t* pos_dev, void* out, void* workspace, uint64_t ws_bytes,
                            void* stream) {
  return decode_common(p, layer, q, q_heads, scale, pos_dev, 1, k_new, v_new, out, workspace, ws_bytes, 0, stream);
}

int hwkv_prefill_workspace_bytes(hwkv_pool_t p, int layer, int q_heads, int n_max, uint64_t* out) {
  if (!p || !out) return fail(HWKV_ERR_INVALID_ARG, "NULL argument");
  const Geometry& g = p->g;
  if (layer < 0 || layer >= g.layers) return fail(HWKV_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (q_heads < g.kv_heads || q_heads % g.kv_heads != 0 || q_heads / g.kv_heads > kMaxGroup)
    return fail(HWKV_ERR_UNSUPPORTED, "q_heads must be G * kv_heads with 1 <= G <= %d", kMaxGroup);
  if (n_max < 1) return fail(HWKV_ERR_INVALID_ARG, "n_max must be >= 1");
  PrefillArgs a;
  std::memset(&a, 0, sizeof a);
  *out = plan_prefill(p, layer, q_heads / g.kv_heads, n_max, true, a);
  return ok();
}

int hwkv_prefill_plan(int layers, int kv_heads, int head_dim, int block_size, const int32_t* windows, int num_seqs,
                      int layer, int q_heads, int n_max, int num_sms, int max_stages, int32_t* head_order,
                      int32_t* splits, int32_t* split_stages, uint64_t* workspace_bytes) {
  if (!head_order || !splits || !split_stages || !workspace_bytes) return fail(HWKV_ERR_INVALID_ARG, "NULL output");
  hwkv_pool p;  // host fields only: geometry, SM count, stage cap, plan cache
  const int rc = plan_geometry(layers, kv_heads, head_dim, block_size, windows, num_seqs, HWKV_BF16, &p.g);
  if (rc != HWKV_OK) return rc;
  if (block_size % 16 != 0) return fail(HWKV_ERR_UNSUPPORTED, "prefill needs block_size % 16 == 0");
  if (layer < 0 || layer >= layers) return fail(HWKV_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (q_heads < kv_heads || q_heads % kv_heads != 0 || q_heads / kv_heads > kMaxGroup)
    return fail(HWKV_ERR_UNSUPPORTED, "q_heads must be G * kv_heads with 1 <= G <= %d", kMaxGroup);
  if (n_max < 1) return fail(HWKV_ERR_INVALID_ARG, "n_max must be >= 1");
  if (num_sms < 1) return fail(HWKV_ERR_INVALID_ARG, "num_sms must be >= 1");
  if (max_stages < 0) return fail(HWKV_ERR_INVALID_ARG, "max_stages must be >= 0");
  p.num_sms = num_sms;
  p.prefill_max_stages = max_stages;
  PrefillArgs a;
  std::memset(&a, 0, sizeof a);
  *workspace_bytes = plan_prefill(&p, layer, q_heads / kv_heads, n_max, true, a);
  for (int i = 0; i < kv_heads; ++i) {
    head_order[i] = a.head_order[i];
    splits[i] = a.splits[i];
    split_stages[i] = a.split_stages[i];
  }
  return ok();
}

int hwkv_set_prefill_config(hwkv_pool_t p, int max_stages) {
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "pool is NULL");
  if (max_stages < 0) return fail(HWKV_ERR_INVALID_ARG, "max_stages must be >= 0");
  p->prefill_max_stages = max_stages;
  return ok();
}

int hwkv_prefill_attn(hwkv_pool_t p, int layer, const void* q, int q_heads, float scale, const void* k_new,
                      const void* v_new, int n_max, const int32_t* pos_dev, const int32_t* n_dev, void* out,
                      void* workspace, uint64_t workspace_bytes, void* stream) {
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "pool is NULL");
  const Geometry& g = p->g;
  if (layer < 0 || layer >= g.layers) return fail(HWKV_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (!prefill_eligible(p)) return fail(HWKV_ERR_UNSUPPORTED, "prefill needs a bf16 pool with block_size % 16 == 0");
  if (q_heads < g.kv_heads || q_heads % g.kv_heads != 0)
    return fail(HWKV_ERR_UNSUPPORTED, "q_heads must be a multiple of kv_heads");
  const int G = q_heads / g.kv_heads;
  if (G > kMaxGroup) return fail(HWKV_ERR_UNSUPPORTED, "q_heads must be G * kv_heads with 1 <= G <= %d", kMaxGroup);
  if (!(scale == scale) || scale == std::numeric_limits<float>::infinity() ||
      scale == -std::numeric_limits<float>::infinity())
    return fail(HWKV_ERR_INVALID_ARG, "scale must be finite");
  if (n_max < 1) return fail(HWKV_ERR_INVALID_ARG, "n_max must be >= 1");
  if ((int64_t)g.num_seqs * n_max > kInt32Max) return fail(HWKV_ERR_UNSUPPORTED, "num_seqs * n_max must be below 2^31");
  if (!q || !k_new || !v_new || !out || !pos_dev || !n_dev) return fail(HWKV_ERR_INVALID_ARG, "NULL tensor argument");
  if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(out, 16) || !aligned(pos_dev, 4) ||
      !aligned(n_dev, 4) || !aligned(workspace, 16))
    return fail(HWKV_ERR_ALIGNMENT, "tensors and workspace must be 16-byte aligned, lengths 4-byte aligned");
  int rc = check_device(p);
  if (rc != HWKV_OK) return rc;
  NvtxRange range_("hwkv_prefill_attn", layer);
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return fail(HWKV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  // the chunk as a 3-D tensor (head_dim, kv_heads, seq * n_max + row): boxes of 16 and of 64
  // rows of one head
  alignas(64) CUtensorMap kmap, vmap, kmap64, vmap64, qmap;
  const cuuint64_t dims[3] = {(cuuint64_t)g.head_dim, (cuuint64_t)g.kv_heads, (cuuint64_t)g.num_seqs * n_max};
  const cuuint64_t strides[2] = {(cuuint64_t)g.head_dim * 2, (cuuint64_t)g.kv_heads * g.head_dim * 2};
  const cuuint32_t box[3] = {64, 1, 16}, box64[3] = {64, 1, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  for (int kv = 0; kv < 4; ++kv) {
    CUtensorMap* m = kv == 0 ? &kmap : kv == 1 ? &vmap : kv == 2 ? &kmap64 : &vmap64;
    CUresult cr = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>((kv & 1) ? v_new : k_new), dims,
                         strides, kv < 2 ? box : box64, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return fail(HWKV_ERR_CUDA, "tensor map of the chunk could not be encoded (%d)", (int)cr);
  }
  {
    // the queries as (head_dim, q_heads, seq * n_max + row): a box of the G heads of one KV head
    // for the tokens of one 128-row query tile
    const int tt = prefill_tile_tokens(G);
    const cuuint64_t qdims[3] = {(cuuint64_t)g.head_dim, (cuuint64_t)q_heads, (cuuint64_t)g.num_seqs * n_max};
    const cuuint64_t qstrides[2] = {(cuuint64_t)g.head_dim * 2, (cuuint64_t)q_heads * g.head_dim * 2};
    const cuuint32_t qbox[3] = {64, (cuuint32_t)G, (cuuint32_t)tt};
    CUresult cr = encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), qdims, qstrides, qbox, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return fail(HWKV_ERR_CUDA, "tensor map of the queries could not be encoded (%d)", (int)cr);
  }
  PrefillArgs a;
  std::memset(&a, 0, sizeof a);
  a.pv = pool_view(p);
  a.g = layer_geom(p, layer);
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.out = out;
  a.pos0 = pos_dev;
  a.nlen = n_dev;
  a.n_max = n_max;
  a.group = G;
  // split long key streams when the workspace holds their partials, else one CTA per stream
  uint64_t need = plan_prefill(p, layer, G, n_max, true, a);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) need = plan_prefill(p, layer, G, n_max, false, a);
  if (need > 0) {
    a.part_o = static_cast<float*>(workspace);
    a.part_ml = a.part_o + (size_t)a.head_ctas[g.kv_heads] * 2 * 128 * g.head_dim;
  }
  a.scale_log2 = scale * 1.4426950408889634f;
  a.bs_log2 = -1;
  for (int b = 0; b < 31; ++b)
    if ((1 << b) == g.block_size) a.bs_log2 = b;
  a.stage_tb = p->stage_tb;
  int max_c = 0;
  for (int h = 0; h < g.kv_heads; ++h) max_c = std::max(max_c, a.g.nblk_prefix[h + 1] - a.g.nblk_prefix[h]);
  max_c *= g.block_size;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  HWKV_CUDA_TRY(launch_prefill(a, &p->tmap, &p->stage_map, &kmap, &vmap, &kmap64, &vmap64, &qmap, st),
                "prefill launch");
  if (need > 0) HWKV_CUDA_TRY(launch_prefill_combine(a, st), "prefill combine launch");
  HWKV_CUDA_TRY(launch_chunk_append(a, std::min(n_max, max_c), st), "chunk append launch");
  return ok();
}

int hwkv_set_decode_config(hwkv_pool_t p, int split_tokens, int workers, int kernel) {
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "pool is NULL");
  if (workers < 0 || workers > (1 << 20)) return fail(HWKV_ERR_INVALID_ARG, "workers must be in [0, 2^20]");
  if (split_tokens != 0 &&
      (split_tokens < 16 || split_tokens > 65536 || (split_tokens & (split_tokens - 1)) != 0))
    return fail(HWKV_ERR_INVALID_ARG, "split_tokens must be 0 or a power of two in [16, 65536]");
  if (kernel != HWKV_KERNEL_AUTO && kernel != HWKV_KERNEL_TENSOR && kernel != HWKV_KERNEL_SIMT)
    return fail(HWKV_ERR_INVALID_ARG, "unknown kernel %d", kernel);
  if (kernel == HWKV_KERNEL_TENSOR && !tc_eligible(p))
    return fail(HWKV_ERR_UNSUPPORTED, "the stream-K decode needs block_size % 16 == 0");
  p->split_override = split_tokens;
  p->workers_override = workers;
  p->kernel_choice = kernel;
  plan_decode(p);
  if (p->has_tmap) {
    const int rc = ensure_counters(p);
    if (rc != HWKV_OK) return rc;
  }
  return ok();
}

int hwkv_seqcalib(int layers, int kv_heads, int head_dim, int block_size, int num_seqs, int dtype,
                  int num_candidates, const int32_t* candidates, hwkv_distortion_fn distortion, void* user,
                  uint64_t budget_bytes, int32_t* out_windows, int32_t* out_choice, uint64_t* out_bytes) {
  if (num_candidates < 1) return fail(HWKV_ERR_INVALID_ARG, "num_candidates must be >= 1");
  if (!candidates || !distortion || !out_windows) return fail(HWKV_ERR_INVALID_ARG, "NULL argument");
  // every candidate must be a valid window vector; its cost is the one-layer pool footprint
  std::vector<uint64_t> cost((size_t)layers * num_candidates);
  for (int l = 0; l < layers; ++l) {
    for (int c = 0; c < num_candidates; ++c) {
      const int32_t* w = candidates + ((size_t)l * num_candidates + c) * kv_heads;
      Geometry g;
      const int rc = plan_geometry(1, kv_heads, head_dim, block_size, w, num_seqs, dtype, &g);
      if (rc != HWKV_OK) return rc;
      cost[(size_t)l * num_candidates + c] = g.pool_bytes;
    }
  }
  std::vector<int32_t> chosen((size_t)layers * kv_heads);
  uint64_t remaining = budget_bytes, total = 0;
  for (int l = 0; l < layers; ++l) {
    int best = -1;
    double best_d = std::numeric_limits<double>::infinity();
    for (int c = 0; c < num_candidates; ++c) {
      const int32_t* w = candidates + ((size_t)l * num_candidates + c) * kv_heads;
      const double d = distortion(user, l, w, chosen.data());
      if (cost[(size_t)l * num_candidates + c] <= remaining && d < best_d) {
        best = c;
        best_d = d;
      }
    }
    if (best < 0)
      return fail(HWKV_ERR_BUDGET, "no candidate window vector of layer %d fits the remaining budget of %llu bytes", l,
                  (unsigned long long)remaining);
    const uint64_t cb = cost[(size_t)l * num_candidates + best];
    remaining -= cb;
    total += cb;
    std::memcpy(&chosen[(size_t)l * kv_heads], candidates + ((size_t)l * num_candidates + best) * kv_heads,
                sizeof(int32_t) * (size_t)kv_heads);
    if (out_choice) out_choice[l] = best;
  }
  std::memcpy(out_windows, chosen.data(), sizeof(int32_t) * chosen.size());
  if (out_bytes) *out_bytes = total;
  return ok();
}

int hwkv_kernel_launches(uint64_t* out) {
  if (!out) return fail(HWKV_ERR_INVALID_ARG, "out is NULL");
  *out = g_launches.load(std::memory_order_relaxed);
  return ok();
}

int hwkv_check_device_errors(hwkv_pool_t p, void* stream, int32_t* out_bits) {
  if (!p) return fail(HWKV_ERR_INVALID_ARG, "pool is NULL");
  int rc = check_device(p);
  if (rc != HWKV_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t bits = 0;
  HWKV_CUDA_TRY(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  HWKV_CUDA_TRY(cudaMemcpy(&bits, p->d_err, sizeof bits, cudaMemcpyDeviceToHost), "read of the error word");
  HWKV_CUDA_TRY(cudaMemset(p->d_err, 0, sizeof bits), "reset of the error word");
  if (out_bits) *out_bits = bits;
  if (bits != 0) {
    // an aborted launch can leave arrival counters behind: start the next launch from zero
    if (p->d_counters)
      HWKV_CUDA_TRY(cudaMemset(p->d_counters, 0, counter_count(p) * sizeof(uint32_t)), "reset of the arrival counters");
    return fail(HWKV_ERR_DEVICE_CHECK, "device error bits 0x%x", bits);
  }
  return ok();
}

}  // extern "C"
