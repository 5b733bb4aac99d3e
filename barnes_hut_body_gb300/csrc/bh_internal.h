// Internal declarations shared by the CUDA translation units of libbh.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "bh.h"

namespace bh {

// Host-side memo of a per-device launch property (SM count, resident blocks
// per SM, a kernel's shared-memory opt-in).  Such properties belong to one
// device, and one process may drive several devices through separate
// contexts, so each device (the current one at the call) gets its own slot;
// `make` runs once per device and must return a nonzero value.
constexpr int kMaxDevices = 64;
template <class F>
inline int per_device(std::atomic<int> (&memo)[kMaxDevices], F make) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return make();
  int v = memo[d].load(std::memory_order_relaxed);
  if (v == 0) {
    v = make();
    memo[d].store(v, std::memory_order_relaxed);
  }
  return v;
}

// Launch a kernel and return the status of that launch alone (not the
// thread's last error, which may belong to an earlier, unrelated call).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

// Number of SMs of the current device (at least 1).
inline int sm_count() {
  static std::atomic<int> memo[kMaxDevices];
  return per_device(memo, [] {
    int dev = 0, c = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
    return c > 0 ? c : 1;
  });
}

// Octree levels 0..21 (21 bits per axis of a 63-bit Morton key).
constexpr int kMaxBits = 21;
constexpr int kMaxLevels = kMaxBits + 1;
constexpr int kMaxPasses = 8;           // 8-bit radix digits of a 63-bit key

// Radix sort tiles: 256 threads x 16 keys (4096) once there are more
// 3072-key tiles than resident blocks (at 2^20 keys every block then sorts
// exactly one tile per pass), 256 x 12 keys below that (shorter tiles when
// each block has one anyway).  Look-back slots are sized for the smaller.
constexpr int kSortThreads = 256;
constexpr int kSortItemsSmall = 12;
constexpr int kSortItemsLarge = 16;
constexpr int kSortTile = kSortThreads * kSortItemsSmall;

// Tree build tile: 256 threads x 4 positions.
constexpr int kBuildThreads = 256;
constexpr int kBuildIters = 4;
constexpr int kBuildTile = kBuildThreads * kBuildIters;
constexpr int kMaxLeafCap = 64;

// Reciprocal square root of the softened squared distance: the hardware
// approximation with denormals flushed (PTX rsqrt.approx.ftz.f32).  The
// argument is >= eps^2, a normal number for every eps > 0, where it equals
// rsqrtf; without the flush, rsqrtf pays a range check and rescaling around
// every approximation (measured: ~3 extra instructions per call, 16% of the
// walk's instructions).  With eps = 0 a pair closer than ~1e-19, whose
// force overflows fp32 anyway, gets rsqrt(0) = inf instead of a huge finite.
__device__ __forceinline__ float rsqrt_ftz(float x) {
  float y;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32x2 arithmetic (Blackwell's f32x2 instructions): two fp32
// values per 64-bit register, one instruction for both, each rounded as the
// scalar operation would be.
typedef unsigned long long f2;
__device__ __forceinline__ f2 pk(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk(f2 v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
  f2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Device status word values mirror the public codes.
constexpr unsigned kErrNonFinite = BH_EINVAL;
constexpr unsigned kErrTimeout = BH_ETIMEOUT;
constexpr unsigned kErrOverflow = BH_ETREE_OVERFLOW;

// Per-call control block, zeroed by one cudaMemsetAsync at the start of
// every bh_compute (so no kernel relies on state left by an earlier call).
struct StepCtrl {
  unsigned int hist[2][kMaxPasses][256];   // digit histograms: sources, targets
  unsigned int hist_top[2][256];           // 63-bit keys: histogram of bits 55..62
  unsigned int tile_ctr[2][kMaxPasses + 1];  // radix tile tickets per pass (+ the
                                           // top-digit pass)
  unsigned int bucket_sort[2];             // 1: every top-digit bucket fits one
                                           // block, the bucket sort ordered the keys
  unsigned int bbox_done[2];               // blocks finished in the bbox pass
  unsigned int work_ctr;                   // traversal group tickets
  int strata;                              // stochastic walk: strata found
  unsigned long long executed;             // source terms evaluated
  unsigned long long groups;               // groups walked
  unsigned long long useful;               // per-target interaction count
  unsigned long long walk_stats[4];        // rounds, nodes tested, nodes put
                                           // to the vote, leaf chunks
  int level_total[kMaxLevels];             // nodes per level (build scan)
  unsigned int fill_ctr;                   // group tickets of a second walk
  unsigned int trie_nodes;                 // insertion tree: nodes allocated
  unsigned int order_fail;                 // insertion tree: a row left out
  int pad1;
  unsigned int sched_cnt[33];              // group schedule: groups per cost class
  unsigned int sched_fill[33];             //   and positions handed out per class
};

// Control block kept across calls.
struct PersistCtrl {
  unsigned int err;          // first device error code of the call
  unsigned int epoch;        // bumped once per call; tags look-back slots
  unsigned int pad[2];
  float4 cube[2];            // (lo_x, lo_y, lo_z, L): sources, targets
  float scale[2];            // 2^bits / L, fp32 IEEE division
  float pad2[2];
  int qexp[2][2];            // fixed-point moments: 2^k_m scales a mass,
                             // 2^k_x a mass x (coordinate - lo); chosen so
                             // that n * max|m| fits in 2^62 (0, 0: no mass)
};

struct DevCtrl {
  StepCtrl step;
  PersistCtrl keep;
};

// Nodes of the current tree: the level totals summed over every level (the
// step's control block starts zeroed and the build writes levels 0..bits
// only), with all the loads in flight at once.
__device__ __forceinline__ long long node_total(const DevCtrl *ctrl) {
  long long t = 0;
#pragma unroll
  for (int l = 0; l < kMaxLevels; ++l) t += ctrl->step.level_total[l];
  return t;
}

// One traversal record per node, 32 bytes: (com.xyz, mass) and
// (ropen2 = w^2/theta^2, link, count, flags).  link = first child for an
// internal node, first particle (sorted index) for a leaf; count = children
// or particles.  flags bit 0 = leaf; bits 8..15 = level.
struct alignas(16) NodeRec {
  float4 com;
  float ropen2;
  int link;
  int count;
  int flags;
};

struct SortBufs {
  unsigned long long *keys[2];
  unsigned int *idx[2];
  unsigned long long *status;   // look-back slots, (tiles x 256)
  int cap_tiles;
};

// --- launchers (each enqueues on `s`, returns cudaGetLastError()) ---------
cudaError_t launch_bbox(const float4 *pm, long long n, float4 *partials,
                        int max_blocks, DevCtrl *ctrl, int which, int bits,
                        bool bump_epoch, cudaStream_t s);
cudaError_t launch_keys(const float4 *pm, long long n, unsigned long long *keys,
                        DevCtrl *ctrl, int which, int bits, cudaStream_t s);
// Sorts keys[0] (with implicit iota values); the result lands in
// keys[final]/idx[final], final returned through *final_buf.
// Sort the keys in sb.keys[0] (ties by index) into sb.keys[*final_buf] and
// the permutation into sb.idx[*final_buf].  63-bit keys may take the bucket
// path, which also writes the gathered rows (pm in key order) to `sorted`;
// the gather must then be told to skip through *gather_skip (a device flag,
// or NULL when the gather always runs).
cudaError_t launch_sort(SortBufs &b, long long n, int bits, DevCtrl *ctrl,
                        int which, unsigned spin_limit, const float4 *pm, float4 *sorted,
                        int *final_buf, const unsigned int **gather_skip,
                        cudaStream_t s);
cudaError_t launch_gather(const float4 *in, const unsigned int *perm,
                          long long n, float4 *out, const unsigned int *skip_if,
                          cudaStream_t s);

// Tree-topology order (k_order.cu): an insertion tree over the Morton digits
// then the index digits of every particle; its depth-first slot order is the
// stable (key, index) order.
struct OrderBufs {
  int *child;            // 8 slots per node: EMPTY, LOCKED, -3 - particle, node
  int *offs;             // 8 per node: start of each slot's range in the node's
  int *parent;
  int *count;            // particles below the node
  int *arrive;           // children that finished counting
  int *nchn;             // slots holding nodes
  int *dir;              // node of each cell of depths 1..4 (or -1)
  unsigned *hist;        // rows per depth-4 cell
  long long cap_nodes;
};
// Builds the tree over keys[0..n) (caller order) and counts it.
cudaError_t launch_order_tree(const float4 *pm, const unsigned long long *keys, long long n,
                              int bits, OrderBufs &b, unsigned long long *skeys,
                              unsigned int *sidx, float4 *spm, DevCtrl *ctrl, int num_sms,
                              cudaStream_t s);
// Writes every particle's key, index and row at its depth-first rank.
cudaError_t launch_order_place(const float4 *pm, const unsigned long long *keys, long long n,
                               int bits, OrderBufs &b, unsigned long long *skeys,
                               unsigned int *sidx, float4 *spm, DevCtrl *ctrl, int num_sms,
                               cudaStream_t s);

struct BuildBufs {
  int4 *topo;            // (first, end, first_child | -1, child_end)
  int *parent;
  unsigned char *level;
  int *arrive;
  long long *pq;         // per node 8 x int64: the fixed-point moment prefix
                         // (m, m x, m y, m z) at the node's first particle,
                         // then at one past its last, each relative to the
                         // start of the build tile holding that position
  NodeRec *rec;
  signed char *facts;          // [position][2]: the first level at which the
                               // position starts a cell, and its leaf level
                               // (the count pass's, for the write pass)
  unsigned int *tile_counts;   // [level][tile]
  long long *tile_q;           // [tile][4]: the tile's moment sums, then the
                               // prefix before the tile
  long long cap_nodes;
  int cap_tiles;
};

cudaError_t launch_build(const unsigned long long *skeys, const float4 *spm,
                         long long n, int bits, int leaf_cap, BuildBufs &b,
                         DevCtrl *ctrl, cudaStream_t s);
cudaError_t launch_com(const float4 *spm, const unsigned long long *skeys,
                       long long n, int bits, float theta, BuildBufs &b,
                       DevCtrl *ctrl, cudaStream_t s);

struct WalkArgs {
  const float4 *spm;          // sorted sources
  long long n;                // number of sources
  const NodeRec *rec;
  const float4 *tpos;         // targets in walk order
  const unsigned int *tperm;  // walk order -> caller index
  long long m;                // number of targets
  float4 *out;                // caller order
  float eps2, G;
  int self_mode;              // targets are the sorted sources
  int opening;                // BH_OPEN_*
  int group;                  // 32 or 64
  int num_sms;
  int pipelined;              // producer/consumer warps (groups of 64)
  long long g_begin, g_end;   // the groups this call walks (a shard of them)
  unsigned int *gcost;        // if set: per group, the terms its walk evaluates
  const unsigned int *gorder; // if set: ticket k walks group gorder[k] (a
                              // permutation of [0, g_end); g_begin is 0)
};
cudaError_t launch_walk(const WalkArgs &a, DevCtrl *ctrl, cudaStream_t s);
// Heaviest first: order[] = the groups [0, ngroups) by descending power-of-two
// class of cost[] (the previous walk's terms per group).  Two grid passes
// (class counts, then placement) on counters in ctrl->step.
cudaError_t launch_group_order(const unsigned int *cost, long long ngroups,
                               unsigned int *order, DevCtrl *ctrl, int num_sms,
                               cudaStream_t s);

// Stochastic Barnes-Hut walk (one warp per 32 Morton-ordered queries).
struct SbhArgs {
  const float4 *spm;          // sorted sources
  long long n;
  const NodeRec *rec;
  const int4 *topo;           // (first, end, first child, child end) per node
  long long nodes;            // node pool capacity (bounds every node index)
  const int *strata;          // filled by the strata pass
  const float4 *tpos;         // targets in walk order
  const unsigned int *tperm;  // walk order -> caller index
  long long m;
  float4 *out;                // caller order
  float eps2, G;
  int self_mode;
  int strata_level;
  int samples;
  int num_sms;
  unsigned long long seed;
  long long g_begin, g_end;   // groups of 32 queries this call walks
};
cudaError_t launch_sbh(const SbhArgs &a, int *strata, int strata_cap,
                       DevCtrl *ctrl, cudaStream_t s);

// Neighbour search: per node the particles' bounding box and largest
// smoothing length, 32 bytes.
struct alignas(16) NbNode {
  float4 lo_h;               // (lo.x, lo.y, lo.z, max h)
  float4 hi;                 // (hi.x, hi.y, hi.z, unused)
};
struct NbArgs {
  const float4 *spm;         // sorted particles
  float *sh;                 // sorted smoothing lengths (written)
  long long n;
  const int4 *topo;
  NbNode *nodes;
  long long nodes_cap;
  const unsigned int *perm;  // sorted -> caller index
  float kappa;
  int symmetric;
  unsigned int *counts;      // caller order
  unsigned long long *offsets;   // caller order, n + 1, or null
  unsigned int *list;        // or null
  unsigned long long list_cap;
  int num_sms;
};
cudaError_t launch_neighbors(const NbArgs &a, const float *h, const int *parent,
                             int *arrive, unsigned long long *scan_tmp,
                             DevCtrl *ctrl, cudaStream_t s);
cudaError_t launch_count(const WalkArgs &a, unsigned int *counts, DevCtrl *ctrl,
                         cudaStream_t s);

cudaError_t launch_direct(const float4 *src, long long n, const float4 *tgt,
                          long long m, bool self_mode, float eps, float G,
                          double *partial, long long partial_cap, float4 *out,
                          int num_sms, cudaStream_t s);

// fp32 throughput probe (k_peak.cu): flops one launch performs, and the
// launch (8 blocks of 256 threads per SM; `sink` is never written).
long long fma_probe_flops(bool packed, int iters, int num_sms);
cudaError_t launch_fma_probe(bool packed, int iters, int num_sms, float *sink,
                             int nsink, cudaStream_t s);

cudaError_t launch_kick_drift(float4 *pm, float4 *vel, const float4 *acc,
                              long long n, float hk, float dt, int num_sms,
                              cudaStream_t s);
cudaError_t launch_kick(float4 *vel, const float4 *acc, long long n, float hk,
                        int num_sms, cudaStream_t s);

}  // namespace bh
