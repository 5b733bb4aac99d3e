// C ABI of the Barnes-Hut library: context, scratch management and the
// per-call orchestration of the GPU stages.  No physics here; every step of
// the path runs in the kernels of k_keys_sort.cu, k_build.cu, k_walk.cu and
// k_direct.cu.
//
// The stage order is the GASPHiA tree-code page's (section "计算核函数":
// computeBoundingBox -> buildTree -> computeCenterOfMass -> computeGravity),
// with the spatial sort of the tree page's "实现步骤" section in front of the
// build.  Unlike the page (a host synchronisation and error check after
// every stage), the whole call is enqueued on one stream with no host
// synchronisation, so it can be captured in a CUDA graph; kernels report
// failures through a device status word read by bh_sync_status.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <new>
#include <string>
#include <vector>

#include "bh_internal.h"

using namespace bh;

struct bh_ctx {
  int device = 0;
  int num_sms = 1;
  float theta = 0.5f, G = 1.f, eps = 0.f;
  int bits = 21, leaf_cap = 16, opening = BH_OPEN_VOTE, timing = 0, group = 0;
  int tbits = 10;                   // BH_OPT_TARGET_KEY_BITS
  int estimator = BH_EST_BARNES_HUT, samples = 1, strata_level = 2;
  int pipeline = 1;
  int order = BH_ORDER_RADIX;
  int order_factor = 2;             // insertion-tree pool: nodes per row
  int shards = 1, shard = 0;        // walk only shard `shard` of `shards`
  int schedule = 1;                 // BH_OPT_SCHEDULE
  unsigned long long seed = 0;
  // group schedule: the last walk's terms per group, and the order built
  // from them; `sched_groups` groups of `sched_gs` targets are valid
  unsigned int *gcost = nullptr, *gorder = nullptr;
  long long cap_groups = 0, sched_groups = -1;
  int sched_gs = 0;
  bool sched_now = false;           // this call walks in the scheduled order
  long long last_groups = 0;        // groups of the last call's walk,
  bool last_costs = false, last_ordered = false;   // costs recorded / order used
  int *strata = nullptr;
  int strata_cap = 0;
  // neighbour search scratch
  NbNode *nb_nodes = nullptr;
  float *nb_h = nullptr;
  unsigned long long *nb_scan = nullptr;
  long long nb_cap_n = 0, nb_cap_nodes = 0;
  unsigned spin_limit = 1u << 22;
  std::string err;

  DevCtrl *ctrl = nullptr;
  float4 *partials = nullptr;
  int bbox_blocks = 0;

  long long cap_n = 0, cap_m = 0, cap_nodes = 0;
  int cap_tiles_sort = 0, cap_tiles_build = 0;
  SortBufs sort{}, sort_t{};
  unsigned long long *status = nullptr;
  float4 *spm = nullptr, *stm = nullptr;
  BuildBufs build{};
  OrderBufs order_bufs{};           // insertion tree of BH_ORDER_TREE

  double *dpartial = nullptr;
  long long dpartial_cap = 0;

  float4 *stage_in = nullptr, *stage_tgt = nullptr, *stage_out = nullptr;
  long long stage_n = 0, stage_m = 0, stage_o = 0;

  cudaEvent_t ev[BH_NUM_STAGES + 1] = {};
  bool stage_ran[BH_NUM_STAGES] = {};
  bool timed = false;

  WalkArgs last_walk{};
  long long last_n = 0, last_m = 0;

  // CUDA graph of the whole step, replayed when a call repeats exactly.
  struct Key {
    const void *pm, *tg;
    void *out;
    long long n, m, cap_n, cap_m, cap_order, cap_groups;   // capacities: buffers reallocated
    float theta, G, eps;
    int bits, tbits, leaf_cap, opening, group;
    unsigned spin;
    int estimator, samples, strata_level, pipeline, order, shards, shard, schedule, sched;
    unsigned long long seed;
    bool operator==(const Key &o) const { return memcmp(this, &o, sizeof(Key)) == 0; }
  };
  int use_graph = 1;
  cudaStream_t cap_stream = nullptr;
  cudaGraphExec_t gexec = nullptr;
  Key gkey{}, prev_key{};
  bool has_prev = false;
  int g_fb = 0, g_fbt = 0;
  WalkArgs g_walk{};
  int last_fb = 0, last_fbt = 0;
  bool last_self = true, last_valid = false;
};

namespace {

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev)
      cudaSetDevice(prev);
  }
};

int fail(bh_ctx *c, int code, const std::string &msg) {
  if (c) c->err = msg;
  return code;
}

int cuda_fail(bh_ctx *c, cudaError_t e, const char *where) {
  return fail(c, BH_ECUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

template <typename T>
void free_dev(T *&p) {
  if (p) cudaFree(p);
  p = nullptr;
}

template <typename T>
bool alloc_dev(T *&p, long long count) {
  free_dev(p);
  if (count <= 0) count = 1;
  return cudaMalloc((void **)&p, sizeof(T) * (size_t)count) == cudaSuccess;
}

long long node_bound(long long n, int leaf_cap, int bits) {
  // leaves <= n; nodes with >= 2 children < leaves; single-child internal
  // cells hold > leaf_cap particles and are disjoint within each level below
  // `bits`, so at most n/(leaf_cap+1) of them per level.
  return 2 * n + (long long)bits * (n / (leaf_cap + 1) + 1) + 8;
}

void free_sources(bh_ctx *c) {
  for (int k = 0; k < 2; ++k) { free_dev(c->sort.keys[k]); free_dev(c->sort.idx[k]); }
  free_dev(c->spm);
  free_dev(c->build.topo); free_dev(c->build.parent); free_dev(c->build.level);
  free_dev(c->build.arrive); free_dev(c->build.pq); free_dev(c->build.rec);
  free_dev(c->build.tile_counts); free_dev(c->build.tile_q); free_dev(c->build.facts);
  c->cap_n = 0; c->cap_nodes = 0;
}

void free_order(bh_ctx *c) {
  OrderBufs &b = c->order_bufs;
  free_dev(b.child); free_dev(b.offs); free_dev(b.parent);
  free_dev(b.count); free_dev(b.arrive); free_dev(b.nchn);
  free_dev(b.dir); free_dev(b.hist);
  b.cap_nodes = 0;
}

// The insertion tree's pool: order_factor x rows + 64 nodes (factor 2 at
// first).  A node is a Morton (or index) digit prefix that two or more rows
// share; the measured workloads need 0.25-0.72 nodes per row, but rows that
// agree on long prefixes (near duplicates) can need more, which the build
// reports as BH_ETREE_OVERFLOW; bh_sync_status then raises the factor 4x for
// the next call, up to 32 -- enough for any input: with 31 digit levels the
// tree has at most 1 + 31 (rows - 1) nodes.
int ensure_order(bh_ctx *c, long long rows) {
  const long long want = (long long)c->order_factor * rows + 64;
  if (want <= c->order_bufs.cap_nodes) return BH_OK;
  cudaDeviceSynchronize();
  free_order(c);
  OrderBufs &b = c->order_bufs;
  bool ok = alloc_dev(b.child, want * 8) && alloc_dev(b.offs, want * 8) &&
            alloc_dev(b.parent, want) && alloc_dev(b.count, want) &&
            alloc_dev(b.arrive, want) && alloc_dev(b.nchn, want) &&
            alloc_dev(b.dir, 8 + 64 + 512 + 4096) && alloc_dev(b.hist, 4096);
  if (!ok) {
    free_order(c);
    return fail(c, BH_ENOMEM, "insertion tree allocation failed");
  }
  b.cap_nodes = want;
  return BH_OK;
}

void free_targets(bh_ctx *c) {
  for (int k = 0; k < 2; ++k) { free_dev(c->sort_t.keys[k]); free_dev(c->sort_t.idx[k]); }
  free_dev(c->stm);
  c->cap_m = 0;
}

int ensure_status(bh_ctx *c, long long n) {
  long long tiles = (n + kSortTile - 1) / kSortTile;
  if (tiles <= c->cap_tiles_sort && c->status) return BH_OK;
  long long want = tiles + tiles / 4 + 1;
  if (!alloc_dev(c->status, want * 256)) return fail(c, BH_ENOMEM, "look-back slots");
  // the tag in every slot must not match a live call: start from zero and
  // the epoch (which starts at 1 after the first bbox) never tags zero slots
  cudaMemset(c->status, 0, sizeof(unsigned long long) * (size_t)want * 256);
  c->cap_tiles_sort = (int)want;
  c->sort.status = c->sort_t.status = c->status;
  c->sort.cap_tiles = c->sort_t.cap_tiles = (int)want;
  return BH_OK;
}

int ensure_sources(bh_ctx *c, long long n) {
  const long long need_nodes = node_bound(n, c->leaf_cap, c->bits);
  if (n <= c->cap_n && need_nodes <= c->cap_nodes) return ensure_status(c, n);
  cudaDeviceSynchronize();
  free_sources(c);
  long long cap = n + n / 8 + 1024;
  long long nodes = node_bound(cap, c->leaf_cap, c->bits);
  if (nodes > (1LL << 31) - 1) return fail(c, BH_EINVAL, "too many particles for int32 node indices");
  bool ok = true;
  for (int k = 0; k < 2; ++k) {
    ok = ok && alloc_dev(c->sort.keys[k], cap);
    ok = ok && alloc_dev(c->sort.idx[k], cap);
  }
  ok = ok && alloc_dev(c->spm, cap);
  ok = ok && alloc_dev(c->build.topo, nodes);
  ok = ok && alloc_dev(c->build.parent, nodes);
  ok = ok && alloc_dev(c->build.level, nodes);
  ok = ok && alloc_dev(c->build.arrive, nodes);
  ok = ok && alloc_dev(c->build.pq, 8 * nodes);
  ok = ok && alloc_dev(c->build.rec, nodes);
  ok = ok && alloc_dev(c->build.facts, 2 * cap);
  long long btiles = (cap + 1 + kBuildTile - 1) / kBuildTile;
  ok = ok && alloc_dev(c->build.tile_counts, btiles * kMaxLevels);
  ok = ok && alloc_dev(c->build.tile_q, 4 * btiles);
  if (!ok) {
    free_sources(c);
    return fail(c, BH_ENOMEM, "source scratch allocation failed");
  }
  c->cap_n = cap;
  c->cap_nodes = nodes;
  c->build.cap_nodes = nodes;
  c->build.cap_tiles = (int)btiles;
  return ensure_status(c, cap);
}

int ensure_targets(bh_ctx *c, long long m) {
  if (m <= c->cap_m) return ensure_status(c, m);
  cudaDeviceSynchronize();
  free_targets(c);
  long long cap = m + m / 8 + 1024;
  bool ok = true;
  for (int k = 0; k < 2; ++k) {
    ok = ok && alloc_dev(c->sort_t.keys[k], cap);
    ok = ok && alloc_dev(c->sort_t.idx[k], cap);
  }
  ok = ok && alloc_dev(c->stm, cap);
  if (!ok) {
    free_targets(c);
    return fail(c, BH_ENOMEM, "target scratch allocation failed");
  }
  c->cap_m = cap;
  return ensure_status(c, cap);
}

// Targets per walk group: the stochastic estimator's 32; else BH_OPT_GROUP,
// or by default 64, or 32 when the targets fill fewer groups of 64 than the
// walk has warps taking groups (16 per SM): then the smaller groups walk in
// parallel what the larger ones would walk one after the other.
long long walk_group_size(const bh_ctx *c, long long m) {
  if (c->estimator == BH_EST_STOCHASTIC) return 32;
  if (c->group) return c->group;
  return (m + 63) / 64 < 16LL * c->num_sms ? 32 : 64;
}

// Per-group cost and order buffers for m targets (groups of >= 32).  A new
// allocation holds no costs, so the schedule starts over.
int ensure_sched(bh_ctx *c, long long m) {
  const long long need = (m + 31) / 32;
  if (need <= c->cap_groups) return BH_OK;
  cudaDeviceSynchronize();
  free_dev(c->gcost);
  free_dev(c->gorder);
  c->cap_groups = 0;
  c->sched_groups = -1;
  const long long cap = need + need / 8 + 64;
  if (!alloc_dev(c->gcost, cap) || !alloc_dev(c->gorder, cap)) {
    free_dev(c->gcost);
    free_dev(c->gorder);
    return fail(c, BH_ENOMEM, "group schedule buffers");
  }
  c->cap_groups = cap;
  return BH_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

int check_rows(bh_ctx *c, const float *p, size_t rows, const char *name) {
  if (rows == 0) return BH_OK;
  if (!p) return fail(c, BH_EINVAL, std::string(name) + " is NULL");
  if (!aligned16(p)) return fail(c, BH_EINVAL, std::string(name) + " is not 16-byte aligned");
  if (rows > (size_t)(1LL << 30)) return fail(c, BH_EINVAL, std::string(name) + " has too many rows");
  return BH_OK;
}

void record(bh_ctx *c, int i, cudaStream_t s) {
  if (c->timing) cudaEventRecord(c->ev[i], s);
}

}  // namespace

namespace {

// Spatial sort of n rows whose keys are in sb.keys[0] (caller order): the
// sorted keys and indices land in sb.keys[*fb] / sb.idx[*fb] and the rows in
// key order in `sorted`.  Radix sort then gather, or (BH_ORDER_TREE) the
// insertion tree's depth-first order, which writes the rows itself.  Event
// `rec` (if >= 0) is recorded between ordering and placement.
cudaError_t enqueue_order(bh_ctx *c, const float4 *pm, long long n, int bits, SortBufs &sb,
                          float4 *sorted, int which, int rec, int *fb, cudaStream_t s) {
  cudaError_t e;
  if (c->order == BH_ORDER_TREE) {
    *fb = 1;
    e = launch_order_tree(pm, sb.keys[0], n, bits, c->order_bufs, sb.keys[1], sb.idx[1],
                          sorted, c->ctrl, c->num_sms, s);
    if (rec >= 0) record(c, rec, s);
    if (e == cudaSuccess)
      e = launch_order_place(pm, sb.keys[0], n, bits, c->order_bufs, sb.keys[1],
                             sb.idx[1], sorted, c->ctrl, c->num_sms, s);
  } else {
    const unsigned int *gather_skip = nullptr;
    e = launch_sort(sb, n, bits, c->ctrl, which, c->spin_limit, pm, sorted, fb,
                    &gather_skip, s);
    if (rec >= 0) record(c, rec, s);
    if (e == cudaSuccess) e = launch_gather(pm, sb.idx[*fb], n, sorted, gather_skip, s);
  }
  return e;
}

// Enqueue every stage of one step on `s` (no host synchronisation).
cudaError_t enqueue_step(bh_ctx *c, const float4 *pm, long long N,
                         const float4 *tg, long long M, float4 *out, bool self,
                         cudaStream_t s, int *fb_out, int *fbt_out,
                         WalkArgs *walk_out) {
  cudaError_t e = cudaMemsetAsync(&c->ctrl->step, 0, sizeof(StepCtrl), s);
  if (e != cudaSuccess) return e;
  record(c, 0, s);
  int fb = 0, fbt = 0;
  e = launch_bbox(pm, N, c->partials, c->bbox_blocks, c->ctrl, 0, c->bits, true, s);
  record(c, 1, s);
  if (e == cudaSuccess) e = launch_keys(pm, N, c->sort.keys[0], c->ctrl, 0, c->bits, s);
  record(c, 2, s);
  if (e == cudaSuccess) e = enqueue_order(c, pm, N, c->bits, c->sort, c->spm, 0, 3, &fb, s);
  else record(c, 3, s);
  record(c, 4, s);
  if (e == cudaSuccess) e = launch_build(c->sort.keys[fb], c->spm, N, c->bits, c->leaf_cap, c->build, c->ctrl, s);
  record(c, 5, s);
  if (e == cudaSuccess) e = launch_com(c->spm, c->sort.keys[fb], N, c->bits, c->theta, c->build, c->ctrl, s);
  record(c, 6, s);
  if (!self) {
    if (e == cudaSuccess) e = launch_bbox(tg, M, c->partials, c->bbox_blocks, c->ctrl, 1, c->tbits, false, s);
    if (e == cudaSuccess) e = launch_keys(tg, M, c->sort_t.keys[0], c->ctrl, 1, c->tbits, s);
    if (e == cudaSuccess) e = enqueue_order(c, tg, M, c->tbits, c->sort_t, c->stm, 1, -1, &fbt, s);
  }
  record(c, 7, s);
  WalkArgs a;
  a.spm = c->spm;
  a.n = N;
  a.rec = c->build.rec;
  a.tpos = self ? c->spm : c->stm;
  a.tperm = self ? c->sort.idx[fb] : c->sort_t.idx[fbt];
  a.m = M;
  a.out = out;
  a.eps2 = c->eps * c->eps;
  a.G = c->G;
  a.self_mode = self ? 1 : 0;
  a.opening = c->opening;
  a.group = c->group ? c->group : ((M + 63) / 64 < 16LL * c->num_sms ? 32 : 64);
  a.num_sms = c->num_sms;
  a.pipelined = c->pipeline;
  const long long gs = walk_group_size(c, M);
  const long long ng = (M + gs - 1) / gs;
  // the walk order's groups, split into `shards` contiguous ranges
  a.g_begin = ng * c->shard / c->shards;
  a.g_end = ng * (c->shard + 1) / c->shards;
  // whole calls of the deterministic walk record their groups' costs; the
  // next call over the same groups takes them heaviest first
  const bool record_costs = c->schedule && c->shards == 1 &&
                            c->estimator != BH_EST_STOCHASTIC && ng <= c->cap_groups;
  a.gcost = record_costs ? c->gcost : nullptr;
  a.gorder = (record_costs && c->sched_now) ? c->gorder : nullptr;
  if (e == cudaSuccess && a.gorder)
    e = launch_group_order(c->gcost, ng, c->gorder, c->ctrl, c->num_sms, s);
  if (c->estimator == BH_EST_STOCHASTIC) {
    SbhArgs b;
    b.spm = c->spm;
    b.n = N;
    b.rec = c->build.rec;
    b.topo = c->build.topo;
    b.nodes = c->build.cap_nodes;
    b.strata = c->strata;
    b.tpos = a.tpos;
    b.tperm = a.tperm;
    b.m = M;
    b.out = out;
    b.eps2 = a.eps2;
    b.G = c->G;
    b.self_mode = a.self_mode;
    b.strata_level = c->strata_level;
    b.samples = c->samples;
    b.num_sms = c->num_sms;
    b.seed = c->seed;
    b.g_begin = a.g_begin;
    b.g_end = a.g_end;
    if (e == cudaSuccess) e = launch_sbh(b, c->strata, c->strata_cap, c->ctrl, s);
  } else if (e == cudaSuccess) {
    e = launch_walk(a, c->ctrl, s);
    if (a.gcost) {
      c->sched_groups = ng;
      c->sched_gs = (int)gs;
    }
  }
  record(c, 8, s);
  *fb_out = fb;
  *fbt_out = fbt;
  *walk_out = a;
  return e;
}

}  // namespace

extern "C" {

int bh_create(bh_ctx **out, int device, size_t max_sources, size_t max_targets) {
  if (!out) return BH_EINVAL;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
    return BH_EINVAL;
  bh_ctx *c = new (std::nothrow) bh_ctx();
  if (!c) return BH_ENOMEM;
  c->device = device;
  DeviceGuard g(device);
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device);
  if (c->num_sms < 1) c->num_sms = 1;
  c->bbox_blocks = c->num_sms * 4;
  bool ok = alloc_dev(c->ctrl, 1) && alloc_dev(c->partials, 2LL * c->bbox_blocks);
  if (ok) ok = cudaMemset(c->ctrl, 0, sizeof(DevCtrl)) == cudaSuccess;
  for (int i = 0; ok && i <= BH_NUM_STAGES; ++i)
    ok = cudaEventCreate(&c->ev[i]) == cudaSuccess;
  if (ok && max_sources) ok = ensure_sources(c, (long long)max_sources) == BH_OK;
  if (ok && max_targets) ok = ensure_targets(c, (long long)max_targets) == BH_OK;
  if (ok) ok = ensure_status(c, 1) == BH_OK;
  if (ok) ok = cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking) == cudaSuccess;
  if (!ok) {
    bh_destroy(c);
    return BH_ENOMEM;
  }
  *out = c;
  return BH_OK;
}

int bh_destroy(bh_ctx *c) {
  if (!c) return BH_OK;
  {
    DeviceGuard g(c->device);
    cudaDeviceSynchronize();
    free_sources(c);
    free_targets(c);
    free_order(c);
    free_dev(c->status);
    free_dev(c->strata);
    free_dev(c->nb_nodes);
    free_dev(c->nb_h);
    free_dev(c->nb_scan);
    free_dev(c->ctrl);
    free_dev(c->partials);
    free_dev(c->dpartial);
    free_dev(c->stage_in);
    free_dev(c->stage_tgt);
    free_dev(c->stage_out);
    free_dev(c->gcost);
    free_dev(c->gorder);
    for (int i = 0; i <= BH_NUM_STAGES; ++i)
      if (c->ev[i]) cudaEventDestroy(c->ev[i]);
    if (c->gexec) cudaGraphExecDestroy(c->gexec);
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
  }
  delete c;
  return BH_OK;
}

int bh_set_params(bh_ctx *c, float theta, float G, float eps) {
  if (!c) return BH_EINVAL;
  if (!(theta >= 0.f) || !isfinite(theta)) return fail(c, BH_EINVAL, "theta must be finite and >= 0");
  if (!isfinite(G)) return fail(c, BH_EINVAL, "G must be finite");
  if (!(eps >= 0.f) || !isfinite(eps)) return fail(c, BH_EINVAL, "eps must be finite and >= 0");
  c->theta = theta;
  c->G = G;
  c->eps = eps;
  return BH_OK;
}

int bh_set_option(bh_ctx *c, int key, long long v) {
  if (!c) return BH_EINVAL;
  switch (key) {
    case BH_OPT_KEY_BITS:
      if (v != 21 && v != 10) return fail(c, BH_EINVAL, "key bits must be 21 or 10");
      c->bits = (int)v;
      return BH_OK;
    case BH_OPT_LEAF_CAP:
      if (v < 1 || v > kMaxLeafCap) return fail(c, BH_EINVAL, "leaf capacity must be in 1..64");
      c->leaf_cap = (int)v;
      return BH_OK;
    case BH_OPT_OPENING:
      if (v != BH_OPEN_VOTE && v != BH_OPEN_BOX) return fail(c, BH_EINVAL, "unknown opening rule");
      c->opening = (int)v;
      return BH_OK;
    case BH_OPT_TIMING:
      c->timing = v ? 1 : 0;
      return BH_OK;
    case BH_OPT_GRAPH:
      c->use_graph = v ? 1 : 0;
      return BH_OK;
    case BH_OPT_GROUP:
      if (v != 0 && v != 32 && v != 64) return fail(c, BH_EINVAL, "group must be 0, 32 or 64");
      c->group = (int)v;
      return BH_OK;
    case BH_OPT_ESTIMATOR:
      if (v != BH_EST_BARNES_HUT && v != BH_EST_STOCHASTIC)
        return fail(c, BH_EINVAL, "unknown estimator");
      c->estimator = (int)v;
      return BH_OK;
    case BH_OPT_SEED:
      c->seed = (unsigned long long)v;
      return BH_OK;
    case BH_OPT_SAMPLES:
      if (v < 1 || v > 1024) return fail(c, BH_EINVAL, "samples must be in 1..1024");
      c->samples = (int)v;
      return BH_OK;
    case BH_OPT_PIPELINE:
      c->pipeline = v ? 1 : 0;
      return BH_OK;
    case BH_OPT_SHARDS:
      if (v < 1 || v > (1 << 20)) return fail(c, BH_EINVAL, "shards must be in 1..2^20");
      c->shards = (int)v;
      if (c->shard >= c->shards) c->shard = 0;
      return BH_OK;
    case BH_OPT_SHARD:
      if (v < 0 || v >= c->shards) return fail(c, BH_EINVAL, "shard must be in 0..shards-1");
      c->shard = (int)v;
      return BH_OK;
    case BH_OPT_TARGET_KEY_BITS:
      if (v != 21 && v != 10) return fail(c, BH_EINVAL, "target key bits must be 21 or 10");
      c->tbits = (int)v;
      return BH_OK;
    case BH_OPT_SCHEDULE:
      if (v < 0 || v > 2) return fail(c, BH_EINVAL, "schedule must be 0, 1 or 2");
      c->schedule = (int)v;
      return BH_OK;
    case BH_OPT_ORDER:
      if (v != BH_ORDER_RADIX && v != BH_ORDER_TREE) return fail(c, BH_EINVAL, "unknown order");
      c->order = (int)v;
      return BH_OK;
    case BH_OPT_STRATA_LEVEL:
      if (v < 0 || v > 6) return fail(c, BH_EINVAL, "strata level must be in 0..6");
      c->strata_level = (int)v;
      return BH_OK;
    default:
      return fail(c, BH_EINVAL, "unknown option");
  }
}

int bh_set_debug(bh_ctx *c, int key, long long v) {
  if (!c) return BH_EINVAL;
  if (key == BH_DBG_SPIN_LIMIT) {
    if (v < 0 || v > (1LL << 30)) return fail(c, BH_EINVAL, "spin limit out of range");
    c->spin_limit = (unsigned)v;
    return BH_OK;
  }
  return fail(c, BH_EINVAL, "unknown debug key");
}

int bh_compute(bh_ctx *c, const float *pos_mass, size_t n, const float *targets,
               size_t m, float *acc_pot, void *stream) {
  if (!c) return BH_EINVAL;
  c->err.clear();
  const bool self = targets == nullptr;
  const long long N = (long long)n, M = self ? N : (long long)m;
  int rc;
  if ((rc = check_rows(c, pos_mass, n, "pos_mass")) != BH_OK) return rc;
  if (!self && (rc = check_rows(c, targets, m, "targets")) != BH_OK) return rc;
  if ((rc = check_rows(c, acc_pot, (size_t)M, "acc_pot")) != BH_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  DeviceGuard g(c->device);
  c->last_valid = false;
  if (M == 0) return BH_OK;
  if (N == 0) {
    cudaError_t e = cudaMemsetAsync(acc_pot, 0, sizeof(float4) * (size_t)M, s);
    return e == cudaSuccess ? BH_OK : cuda_fail(c, e, "memset");
  }
  if ((rc = ensure_sources(c, N)) != BH_OK) return rc;
  if (!self && (rc = ensure_targets(c, M)) != BH_OK) return rc;
  if (c->order == BH_ORDER_TREE &&
      (rc = ensure_order(c, c->cap_n > c->cap_m ? c->cap_n : c->cap_m)) != BH_OK)
    return rc;
  if ((rc = ensure_sched(c, M)) != BH_OK) return rc;
  const long long walk_gs = walk_group_size(c, M);
  const long long walk_ng = (M + walk_gs - 1) / walk_gs;
  const bool costs = c->schedule && c->shards == 1 && c->estimator != BH_EST_STOCHASTIC;
  // with no more groups than the walk has warps taking them (16 per SM) every
  // group starts at once and the order cannot matter (unless forced)
  c->sched_now = costs && c->sched_groups == walk_ng && c->sched_gs == walk_gs &&
                 (c->schedule == 2 || walk_ng > 16LL * c->num_sms);
  if (c->estimator == BH_EST_STOCHASTIC && !c->strata) {
    // strata of level s <= 6 number at most 8^6
    if (!alloc_dev(c->strata, 1LL << 18)) return fail(c, BH_ENOMEM, "strata list");
    c->strata_cap = 1 << 18;
  }

  const float4 *pm = reinterpret_cast<const float4 *>(pos_mass);
  const float4 *tg = reinterpret_cast<const float4 *>(targets);
  float4 *out = reinterpret_cast<float4 *>(acc_pot);
  for (int i = 0; i < BH_NUM_STAGES; ++i) c->stage_ran[i] = false;
  int fb = 0, fbt = 0;
  WalkArgs walk{};
  cudaError_t e = cudaSuccess;

  // Repeated identical calls replay one CUDA graph of the whole step: the
  // second identical call captures it on an internal stream, later ones
  // launch it.  Not while stage timing is on or while the caller's stream
  // is itself being captured.
  bh_ctx::Key key;
  memset(&key, 0, sizeof(key));
  key.pm = pm; key.tg = tg; key.out = out; key.n = N; key.m = M;
  key.cap_n = c->cap_n; key.cap_m = c->cap_m;
  key.cap_order = c->order_bufs.cap_nodes;
  key.theta = c->theta; key.G = c->G; key.eps = c->eps;
  key.bits = c->bits; key.tbits = c->tbits; key.leaf_cap = c->leaf_cap;
  key.opening = c->opening;
  key.group = c->group; key.spin = c->spin_limit;
  key.estimator = c->estimator; key.samples = c->samples;
  key.strata_level = c->strata_level; key.seed = c->seed; key.pipeline = c->pipeline;
  key.order = c->order;
  key.shards = c->shards; key.shard = c->shard;
  key.cap_groups = c->cap_groups;
  key.schedule = c->schedule; key.sched = c->sched_now ? 1 : 0;
  bool graph = c->use_graph && !c->timing && c->cap_stream;
  if (graph) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
      graph = false;
  }
  bool done = false;
  if (graph && c->gexec && key == c->gkey) {
    e = cudaGraphLaunch(c->gexec, s);
    fb = c->g_fb; fbt = c->g_fbt; walk = c->g_walk;
    done = true;
  } else if (graph && c->has_prev && key == c->prev_key) {
    cudaGraph_t gr = nullptr;
    cudaError_t ec = cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal);
    if (ec == cudaSuccess) {
      ec = enqueue_step(c, pm, N, tg, M, out, self, c->cap_stream, &fb, &fbt, &walk);
      cudaError_t ee = cudaStreamEndCapture(c->cap_stream, &gr);
      if (ec == cudaSuccess) ec = ee;
    }
    cudaGraphExec_t ex = nullptr;
    if (ec == cudaSuccess && gr) ec = cudaGraphInstantiate(&ex, gr, 0);
    if (gr) cudaGraphDestroy(gr);
    if (ec == cudaSuccess && ex) {
      if (c->gexec) cudaGraphExecDestroy(c->gexec);
      c->gexec = ex;
      c->gkey = key;
      c->g_fb = fb; c->g_fbt = fbt; c->g_walk = walk;
      e = cudaGraphLaunch(ex, s);
      done = true;
    } else {
      cudaGetLastError();          // capture unsupported here: run directly
      c->use_graph = 0;
    }
  }
  if (!done) e = enqueue_step(c, pm, N, tg, M, out, self, s, &fb, &fbt, &walk);
  c->prev_key = key;
  c->has_prev = true;
  c->last_walk = walk;
  if (e != cudaSuccess) return cuda_fail(c, e, "launch");
  for (int i = 0; i < BH_NUM_STAGES; ++i) c->stage_ran[i] = true;
  c->stage_ran[BH_STAGE_TARGETS] = !self;
  c->timed = c->timing != 0;
  c->last_n = N;
  c->last_m = M;
  c->last_fb = fb;
  c->last_fbt = fbt;
  c->last_self = self;
  c->last_groups = walk_ng;
  c->last_costs = costs;
  c->last_ordered = c->sched_now;
  c->last_valid = true;
  return BH_OK;
}

int bh_sync_status(bh_ctx *c, void *stream) {
  if (!c) return BH_EINVAL;
  DeviceGuard g(c->device);
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "stream synchronize");
  unsigned err = 0;
  e = cudaMemcpy(&err, &c->ctrl->keep.err, sizeof(unsigned), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(c, e, "status read");
  if (err) {
    cudaMemset(&c->ctrl->keep.err, 0, sizeof(unsigned));
    // a row left out of the insertion tree: the next call gets a larger pool
    unsigned order_fail = 0;
    if (err == BH_ETREE_OVERFLOW && c->order == BH_ORDER_TREE &&
        cudaMemcpy(&order_fail, &c->ctrl->step.order_fail, sizeof(unsigned),
                   cudaMemcpyDeviceToHost) == cudaSuccess &&
        order_fail && c->order_factor < 32)
      c->order_factor = c->order_factor * 4 < 32 ? c->order_factor * 4 : 32;
    const char *what = err == BH_EINVAL ? "non-finite input"
                       : err == BH_ETIMEOUT ? "a device wait timed out"
                       : err == BH_ETREE_OVERFLOW ? "node pool or walk stack overflow"
                                                  : "device error";
    return fail(c, (int)err, what);
  }
  return BH_OK;
}

int bh_compute_host(bh_ctx *c, const float *pos_mass, size_t n, const float *targets,
                    size_t m, float *acc_pot, void *stream) {
  if (!c) return BH_EINVAL;
  const bool self = targets == nullptr;
  const long long N = (long long)n, M = self ? N : (long long)m;
  if (N > 0 && !pos_mass) return fail(c, BH_EINVAL, "pos_mass is NULL");
  if (M > 0 && !acc_pot) return fail(c, BH_EINVAL, "acc_pot is NULL");
  if (!self && M > 0 && !targets) return fail(c, BH_EINVAL, "targets is NULL");
  DeviceGuard g(c->device);
  cudaStream_t s = (cudaStream_t)stream;
  if (N > c->stage_n) {
    cudaDeviceSynchronize();
    if (!alloc_dev(c->stage_in, N + N / 8 + 64)) return fail(c, BH_ENOMEM, "staging");
    c->stage_n = N + N / 8 + 64;
  }
  if (!self && M > c->stage_m) {
    cudaDeviceSynchronize();
    if (!alloc_dev(c->stage_tgt, M + M / 8 + 64)) return fail(c, BH_ENOMEM, "staging");
    c->stage_m = M + M / 8 + 64;
  }
  // Page-locked (pinned) output memory is device-accessible: the kernels then
  // write the results straight into it over the host link while they run,
  // instead of a device buffer copied back afterwards.
  float *dev_out = nullptr;
  {
    cudaPointerAttributes at;
    if (M > 0 && cudaPointerGetAttributes(&at, acc_pot) == cudaSuccess &&
        at.type == cudaMemoryTypeHost && at.devicePointer)
      dev_out = reinterpret_cast<float *>(at.devicePointer);
    else
      cudaGetLastError();
  }
  if (!dev_out && M > c->stage_o) {
    cudaDeviceSynchronize();
    if (!alloc_dev(c->stage_out, M + M / 8 + 64)) return fail(c, BH_ENOMEM, "staging");
    c->stage_o = M + M / 8 + 64;
  }
  cudaError_t e = cudaSuccess;
  if (N > 0) e = cudaMemcpyAsync(c->stage_in, pos_mass, sizeof(float4) * (size_t)N, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && !self && M > 0)
    e = cudaMemcpyAsync(c->stage_tgt, targets, sizeof(float4) * (size_t)M, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(c, e, "host to device copy");
  int rc = bh_compute(c, (const float *)c->stage_in, n,
                      self ? nullptr : (const float *)c->stage_tgt, m,
                      dev_out ? dev_out : (float *)c->stage_out, stream);
  if (rc != BH_OK) return rc;
  if (M > 0 && !dev_out) {
    e = cudaMemcpyAsync(acc_pot, c->stage_out, sizeof(float4) * (size_t)M, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(c, e, "device to host copy");
  }
  return bh_sync_status(c, stream);
}

int bh_direct(bh_ctx *c, const float *pos_mass, size_t n, const float *targets,
              size_t m, float *acc_pot, void *stream) {
  if (!c) return BH_EINVAL;
  c->err.clear();
  const bool self = targets == nullptr;
  const long long N = (long long)n, M = self ? N : (long long)m;
  int rc;
  if ((rc = check_rows(c, pos_mass, n, "pos_mass")) != BH_OK) return rc;
  if (!self && (rc = check_rows(c, targets, m, "targets")) != BH_OK) return rc;
  if ((rc = check_rows(c, acc_pot, (size_t)M, "acc_pot")) != BH_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  DeviceGuard g(c->device);
  if (M == 0) return BH_OK;
  if (N == 0) {
    cudaError_t e = cudaMemsetAsync(acc_pot, 0, sizeof(float4) * (size_t)M, s);
    return e == cudaSuccess ? BH_OK : cuda_fail(c, e, "memset");
  }
  long long want = 4 * M * 64;
  if (want > (1LL << 25)) want = 4 * M > (1LL << 25) ? 4 * M : (1LL << 25);
  if (c->dpartial_cap < 4 * M) {
    cudaDeviceSynchronize();
    if (!alloc_dev(c->dpartial, want)) {
      c->dpartial_cap = 0;
      return fail(c, BH_ENOMEM, "direct-sum partials");
    }
    c->dpartial_cap = want;
  }
  cudaError_t e = launch_direct(reinterpret_cast<const float4 *>(pos_mass), N,
                                reinterpret_cast<const float4 *>(self ? pos_mass : targets),
                                M, self, c->eps, c->G, c->dpartial, c->dpartial_cap,
                                reinterpret_cast<float4 *>(acc_pot), c->num_sms, s);
  if (e != cudaSuccess) return cuda_fail(c, e, "direct launch");
  return BH_OK;
}

int bh_neighbors(bh_ctx *c, const float *pos_mass, const float *h, size_t n,
                 float kappa, int mode, unsigned int *counts,
                 unsigned long long *offsets, unsigned int *list, size_t list_cap,
                 void *stream) {
  if (!c) return BH_EINVAL;
  c->err.clear();
  int rc;
  if ((rc = check_rows(c, pos_mass, n, "pos_mass")) != BH_OK) return rc;
  if (n && !h) return fail(c, BH_EINVAL, "h is NULL");
  if (n && !counts) return fail(c, BH_EINVAL, "counts is NULL");
  if (list && !offsets) return fail(c, BH_EINVAL, "a list needs offsets");
  if (!(kappa > 0.f) || !isfinite(kappa)) return fail(c, BH_EINVAL, "kappa must be finite and > 0");
  if (mode != BH_NB_GATHER && mode != BH_NB_SYMMETRIC) return fail(c, BH_EINVAL, "unknown neighbour mode");
  if (n > 0xffffffffULL) return fail(c, BH_EINVAL, "too many particles for 32-bit indices");
  cudaStream_t s = (cudaStream_t)stream;
  DeviceGuard g(c->device);
  c->last_valid = false;
  const long long N = (long long)n;
  if (N == 0) {
    if (offsets) {
      cudaError_t e = cudaMemsetAsync(offsets, 0, sizeof(unsigned long long), s);
      if (e != cudaSuccess) return cuda_fail(c, e, "memset");
    }
    return BH_OK;
  }
  if ((rc = ensure_sources(c, N)) != BH_OK) return rc;
  if (c->order == BH_ORDER_TREE && (rc = ensure_order(c, c->cap_n)) != BH_OK) return rc;
  if (c->nb_cap_n < c->cap_n || c->nb_cap_nodes < c->cap_nodes) {
    cudaDeviceSynchronize();
    free_dev(c->nb_nodes); free_dev(c->nb_h); free_dev(c->nb_scan);
    c->nb_cap_n = c->nb_cap_nodes = 0;
    if (!alloc_dev(c->nb_nodes, c->cap_nodes) || !alloc_dev(c->nb_h, c->cap_n) ||
        !alloc_dev(c->nb_scan, c->cap_n / 1024 + 2))
      return fail(c, BH_ENOMEM, "neighbour search scratch");
    c->nb_cap_n = c->cap_n;
    c->nb_cap_nodes = c->cap_nodes;
  }
  const float4 *pm = reinterpret_cast<const float4 *>(pos_mass);
  int fb = 0;
  cudaError_t e = cudaMemsetAsync(&c->ctrl->step, 0, sizeof(StepCtrl), s);
  if (e == cudaSuccess) e = launch_bbox(pm, N, c->partials, c->bbox_blocks, c->ctrl, 0, c->bits, true, s);
  if (e == cudaSuccess) e = launch_keys(pm, N, c->sort.keys[0], c->ctrl, 0, c->bits, s);
  if (e == cudaSuccess) e = enqueue_order(c, pm, N, c->bits, c->sort, c->spm, 0, -1, &fb, s);
  if (e == cudaSuccess) e = launch_build(c->sort.keys[fb], c->spm, N, c->bits, c->leaf_cap, c->build, c->ctrl, s);
  NbArgs a;
  a.spm = c->spm;
  a.sh = c->nb_h;
  a.n = N;
  a.topo = c->build.topo;
  a.nodes = c->nb_nodes;
  a.nodes_cap = c->build.cap_nodes;
  a.perm = c->sort.idx[fb];
  a.kappa = kappa;
  a.symmetric = mode == BH_NB_SYMMETRIC ? 1 : 0;
  a.counts = counts;
  a.offsets = offsets;
  a.list = list;
  a.list_cap = list ? (unsigned long long)list_cap : 0ull;
  a.num_sms = c->num_sms;
  if (e == cudaSuccess)
    e = launch_neighbors(a, h, c->build.parent, c->build.arrive, c->nb_scan, c->ctrl, s);
  if (e != cudaSuccess) return cuda_fail(c, e, "neighbour search launch");
  return BH_OK;
}

int bh_fp32_probe(bh_ctx *c, int packed, int iters, double *flops, void *stream) {
  if (!c) return BH_EINVAL;
  c->err.clear();
  if ((packed != 0 && packed != 1) || iters < 1 || iters > (1 << 24))
    return fail(c, BH_EINVAL, "fp32 probe: packed must be 0 or 1, iters in 1..2^24");
  DeviceGuard g(c->device);
  const int nsink = 4 * 2 * c->bbox_blocks;   // floats of c->partials, never written
  cudaError_t e = launch_fma_probe(packed == 1, iters, c->num_sms,
                                   reinterpret_cast<float *>(c->partials), nsink,
                                   (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "fp32 probe launch");
  if (flops) *flops = (double)fma_probe_flops(packed == 1, iters, c->num_sms);
  return BH_OK;
}

int bh_get_stage_times(bh_ctx *c, float *ms, int n) {
  if (!c || !ms || n < 0 || n > BH_NUM_STAGES) return BH_EINVAL;
  if (!c->timed) return fail(c, BH_EINVAL, "no timed call (set BH_OPT_TIMING)");
  DeviceGuard g(c->device);
  cudaError_t e = cudaEventSynchronize(c->ev[BH_NUM_STAGES]);
  if (e != cudaSuccess) return cuda_fail(c, e, "event synchronize");
  for (int i = 0; i < n; ++i) {
    float t = 0.f;
    if (c->stage_ran[i]) cudaEventElapsedTime(&t, c->ev[i], c->ev[i + 1]);
    ms[i] = t;
  }
  return BH_OK;
}

int bh_get_counters(bh_ctx *c, unsigned long long *executed, unsigned long long *groups) {
  if (!c) return BH_EINVAL;
  DeviceGuard g(c->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(c, e, "synchronize");
  StepCtrl st;
  e = cudaMemcpy(&st, &c->ctrl->step, sizeof(StepCtrl), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(c, e, "counter read");
  if (executed) *executed = st.executed;
  if (groups) *groups = st.groups;
  return BH_OK;
}

int bh_debug_export(bh_ctx *c, int what, void *dst, size_t bytes) {
  if (!c || !dst) return BH_EINVAL;
  if (!c->last_valid) return fail(c, BH_EINVAL, "no completed bh_compute to export");
  DeviceGuard g(c->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(c, e, "synchronize");
  StepCtrl st;
  e = cudaMemcpy(&st, &c->ctrl->step, sizeof(StepCtrl), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(c, e, "control read");
  long long nodes = 0;
  for (int l = 0; l <= c->bits; ++l) nodes += st.level_total[l];
  if (nodes > c->cap_nodes) nodes = c->cap_nodes;
  auto need = [&](size_t b) { return bytes >= b; };
  switch (what) {
    case BH_EXPORT_CUBE: {
      if (!need(16)) return fail(c, BH_EINVAL, "buffer too small");
      e = cudaMemcpy(dst, &c->ctrl->keep.cube[0], 16, cudaMemcpyDeviceToHost);
      break;
    }
    case BH_EXPORT_KEYS:
      if (!need(8 * (size_t)c->last_n)) return fail(c, BH_EINVAL, "buffer too small");
      e = cudaMemcpy(dst, c->sort.keys[c->last_fb], 8 * (size_t)c->last_n, cudaMemcpyDeviceToHost);
      break;
    case BH_EXPORT_PERM:
      if (!need(4 * (size_t)c->last_n)) return fail(c, BH_EINVAL, "buffer too small");
      e = cudaMemcpy(dst, c->sort.idx[c->last_fb], 4 * (size_t)c->last_n, cudaMemcpyDeviceToHost);
      break;
    case BH_EXPORT_TARGET_PERM:
      if (c->last_self) return fail(c, BH_EINVAL, "last call had no separate targets");
      if (!need(4 * (size_t)c->last_m)) return fail(c, BH_EINVAL, "buffer too small");
      e = cudaMemcpy(dst, c->sort_t.idx[c->last_fbt], 4 * (size_t)c->last_m, cudaMemcpyDeviceToHost);
      break;
    case BH_EXPORT_GROUP_COST:
    case BH_EXPORT_GROUP_ORDER: {
      const bool cost = what == BH_EXPORT_GROUP_COST;
      if (cost ? !c->last_costs : !c->last_ordered)
        return fail(c, BH_EINVAL, cost ? "last call recorded no group costs"
                                       : "last call walked its groups in Morton order");
      if (!need(4 * (size_t)c->last_groups)) return fail(c, BH_EINVAL, "buffer too small");
      e = cudaMemcpy(dst, cost ? c->gcost : c->gorder, 4 * (size_t)c->last_groups,
                     cudaMemcpyDeviceToHost);
      break;
    }
    case BH_EXPORT_WALK_STATS:
      if (!need(32)) return fail(c, BH_EINVAL, "buffer too small");
      memcpy(dst, st.walk_stats, 32);
      break;
    case BH_EXPORT_SORT_PATH:
      if (!need(8)) return fail(c, BH_EINVAL, "buffer too small");
      memcpy(dst, st.bucket_sort, 8);
      break;
    case BH_EXPORT_NODE_COUNT:
      if (!need(8)) return fail(c, BH_EINVAL, "buffer too small");
      memcpy(dst, &nodes, 8);
      break;
    case BH_EXPORT_NODES: {
      if (!need(24 * (size_t)nodes)) return fail(c, BH_EINVAL, "buffer too small");
      std::vector<int4> topo((size_t)nodes);
      std::vector<int> par((size_t)nodes);
      std::vector<unsigned char> lv((size_t)nodes);
      e = cudaMemcpy(topo.data(), c->build.topo, sizeof(int4) * (size_t)nodes, cudaMemcpyDeviceToHost);
      if (e == cudaSuccess) e = cudaMemcpy(par.data(), c->build.parent, sizeof(int) * (size_t)nodes, cudaMemcpyDeviceToHost);
      if (e == cudaSuccess) e = cudaMemcpy(lv.data(), c->build.level, (size_t)nodes, cudaMemcpyDeviceToHost);
      if (e != cudaSuccess) break;
      int *o = (int *)dst;
      for (long long k = 0; k < nodes; ++k) {
        const int4 t = topo[(size_t)k];
        o[6 * k + 0] = lv[(size_t)k];
        o[6 * k + 1] = t.x;
        o[6 * k + 2] = t.y - t.x;
        o[6 * k + 3] = t.z;
        o[6 * k + 4] = t.z >= 0 ? t.w - t.z : 0;
        o[6 * k + 5] = par[(size_t)k];
      }
      break;
    }
    case BH_EXPORT_COM: {
      if (!need(16 * (size_t)nodes)) return fail(c, BH_EINVAL, "buffer too small");
      std::vector<NodeRec> rec((size_t)nodes);
      e = cudaMemcpy(rec.data(), c->build.rec, sizeof(NodeRec) * (size_t)nodes, cudaMemcpyDeviceToHost);
      if (e != cudaSuccess) break;
      float *o = (float *)dst;
      for (long long k = 0; k < nodes; ++k) {
        o[4 * k + 0] = rec[(size_t)k].com.x;
        o[4 * k + 1] = rec[(size_t)k].com.y;
        o[4 * k + 2] = rec[(size_t)k].com.z;
        o[4 * k + 3] = rec[(size_t)k].com.w;
      }
      break;
    }
    default:
      return fail(c, BH_EINVAL, "unknown export key");
  }
  if (e != cudaSuccess) return cuda_fail(c, e, "export copy");
  return BH_OK;
}

int bh_count_interactions(bh_ctx *c, unsigned int *counts,
                          unsigned long long *total, void *stream) {
  if (!c) return BH_EINVAL;
  if (!c->last_valid) return fail(c, BH_EINVAL, "no completed bh_compute to count");
  DeviceGuard g(c->device);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_count(c->last_walk, counts, c->ctrl, s);
  if (e != cudaSuccess) return cuda_fail(c, e, "count launch");
  if (total) {
    e = cudaStreamSynchronize(s);
    if (e == cudaSuccess)
      e = cudaMemcpy(total, &c->ctrl->step.useful, sizeof(unsigned long long),
                     cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(c, e, "count read");
  }
  return BH_OK;
}

int bh_leapfrog(bh_ctx *c, float *pos_mass, float *vel, size_t n,
                float *acc_pot, float dt, int nsteps, int flags, void *stream) {
  if (!c) return BH_EINVAL;
  c->err.clear();
  int rc;
  if ((rc = check_rows(c, pos_mass, n, "pos_mass")) != BH_OK) return rc;
  if ((rc = check_rows(c, vel, n, "vel")) != BH_OK) return rc;
  if ((rc = check_rows(c, acc_pot, n, "acc_pot")) != BH_OK) return rc;
  if (!isfinite(dt) || nsteps < 0) return fail(c, BH_EINVAL, "dt must be finite and nsteps >= 0");
  if (n == 0) return BH_OK;
  DeviceGuard g(c->device);
  cudaStream_t s = (cudaStream_t)stream;
  float4 *pm = reinterpret_cast<float4 *>(pos_mass);
  float4 *v = reinterpret_cast<float4 *>(vel);
  float4 *a = reinterpret_cast<float4 *>(acc_pot);
  const long long N = (long long)n;
  if (!(flags & BH_LF_ACC_VALID)) {
    if ((rc = bh_compute(c, pos_mass, n, nullptr, 0, acc_pot, stream)) != BH_OK) return rc;
  }
  const float half = 0.5f * dt;
  for (int k = 0; k < nsteps; ++k) {
    cudaError_t e = launch_kick_drift(pm, v, a, N, half, dt, c->num_sms, s);
    if (e != cudaSuccess) return cuda_fail(c, e, "kick-drift launch");
    if ((rc = bh_compute(c, pos_mass, n, nullptr, 0, acc_pot, stream)) != BH_OK) return rc;
    e = launch_kick(v, a, N, half, c->num_sms, s);
    if (e != cudaSuccess) return cuda_fail(c, e, "kick launch");
  }
  return BH_OK;
}

const char *bh_last_error(const bh_ctx *c) {
  return c ? c->err.c_str() : "null context";
}

}  // extern "C"
