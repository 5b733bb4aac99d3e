// SPH neighbour search on the octree ("树结构（基于根据 Burtscher 和 Pingali
// 的研究）", sections 粒子领域搜索 and 树遍历计算: visit the cells within the
// kernel scale of the query and test their particles; GASPHiA keeps a
// per-node maximum smoothing length, d_node_hmax, for the same search).
//
// Particle j != i is a neighbour of i iff |x_i - x_j|^2 < (kappa H)^2 with
// H = max(h_i, h_j) (symmetric) or H = h_i (gather), the test in fp32 with
// every operation rounded as written, so the lists are exact.
//
// Per node, a bottom-up pass stores the particles' bounding box and maximum
// smoothing length (the last child to arrive combines its siblings, as the
// centre-of-mass pass does).  One warp serves 32 consecutive sorted particles
// (groups taken by atomic tickets): it tests up to 32 nodes per round (one per
// lane) against the group's bounding box and largest smoothing length and,
// when the group is spread wider than its largest search radius, against
// each particle's own sphere -- both with a margin that makes the pruning
// conservative under fp32 rounding -- pushes the child ranges of opened cells
// on a shared-memory stack, and tests the particles of the round's opened
// leaves, loaded 32 at a time, against each lane's own particle.  A counting
// walk gives the counts, a scan gives the offsets, and an identical second
// walk writes the lists.
#include <climits>

#include "bh_internal.h"

namespace bh {
namespace {

constexpr int kNbThreads = 128;
constexpr int kNbWarps = kNbThreads / 32;
// Child ranges per warp.  A round takes up to 32 nodes from the top ranges
// (deepest first) and pushes at most 32, the ranges of the cells it opened,
// the deepest on top, so levels never decrease towards the top.  A round
// that takes level-l nodes has first consumed every range above them, all
// deeper than l; so the level-(l+1) ranges on the stack all come from one
// round: at most 32 per level, 32 * 22 + 32 = 736 < 768.
constexpr int kNbStack = 768;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void set_err(DevCtrl *c, unsigned code) {
  atomicCAS(&c->keep.err, 0u, code);
}

// h into sorted order; negative or non-finite h is an argument error.
__global__ void gather_h_kernel(const float *__restrict__ h,
                                const unsigned int *__restrict__ perm, long long n,
                                float *__restrict__ sh, DevCtrl *ctrl) {
  bool bad = false;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x; r < n; r += stride) {
    const unsigned p = perm[r];
    const float v = p < n ? h[p] : 0.f;
    if (!(v >= 0.f) || !isfinite(v)) bad = true;
    sh[r] = v;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) set_err(ctrl, kErrNonFinite);
}

__device__ __forceinline__ void finish(long long c, const float4 &lo, const float4 &hi,
                                       NbNode *nodes) {
  NbNode r;
  r.lo_h = lo;
  r.hi = hi;
  nodes[c] = r;
}

// Bounding box and maximum h per node, leaves first, parents by the last
// child to arrive (arrival counters zeroed by the build for internal nodes).
__global__ void __launch_bounds__(256)
nb_node_kernel(const float4 *__restrict__ spm, const float *__restrict__ sh,
               long long n, const int4 *__restrict__ topo,
               const int *__restrict__ parent, int *arrive, NbNode *nodes,
               DevCtrl *ctrl, long long cap_nodes) {
  const long long total = node_total(ctrl);
  if (total > cap_nodes) return;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total;
       c += stride) {
    const int4 t = topo[c];
    if (t.z >= 0) continue;                        // internal: done by a child
    long long f = t.x < 0 ? 0 : t.x, e = t.y;
    if (f > n) f = n;
    if (e > n) e = n;
    float4 lo = make_float4(INFINITY, INFINITY, INFINITY, 0.f);
    float4 hi = make_float4(-INFINITY, -INFINITY, -INFINITY, 0.f);
    for (long long j = f; j < e; ++j) {
      const float4 p = spm[j];
      lo.x = fminf(lo.x, p.x); lo.y = fminf(lo.y, p.y); lo.z = fminf(lo.z, p.z);
      hi.x = fmaxf(hi.x, p.x); hi.y = fmaxf(hi.y, p.y); hi.z = fmaxf(hi.z, p.z);
      lo.w = fmaxf(lo.w, sh[j]);
    }
    finish(c, lo, hi, nodes);
    long long node = c;
    for (int guard = 0; guard <= kMaxLevels; ++guard) {
      const int p = parent[node];
      if (p < 0 || p >= total) break;
      __threadfence();
      const int4 tp = topo[p];
      const int nch = tp.w - tp.z;
      if (tp.z < 0 || nch < 1 || nch > 8 || tp.w > total) break;
      if (atomicAdd(arrive + p, 1) != nch - 1) break;
      __threadfence();
      float4 a = make_float4(INFINITY, INFINITY, INFINITY, 0.f);
      float4 b = make_float4(-INFINITY, -INFINITY, -INFINITY, 0.f);
      for (int k = tp.z; k < tp.w; ++k) {
        const float4 l = __ldcg(&nodes[k].lo_h), u = __ldcg(&nodes[k].hi);
        a.x = fminf(a.x, l.x); a.y = fminf(a.y, l.y); a.z = fminf(a.z, l.z);
        a.w = fmaxf(a.w, l.w);
        b.x = fmaxf(b.x, u.x); b.y = fmaxf(b.y, u.y); b.z = fmaxf(b.z, u.z);
      }
      finish(p, a, b, nodes);
      node = p;
    }
  }
}

// Can a particle in [lo, hi] with smoothing length h reach the node (true
// also for some that cannot: the test is conservative under fp32 rounding,
// a pair's rounded r^2 being >= d2 (1 - 2^-21))?
__device__ __forceinline__ bool reaches(float lx, float ly, float lz, float hx, float hy,
                                        float hz, float h, const NbNode &nd, float kappa,
                                        bool sym) {
  const float dx = fmaxf(0.f, fmaxf(__fsub_rn(nd.lo_h.x, hx), __fsub_rn(lx, nd.hi.x)));
  const float dy = fmaxf(0.f, fmaxf(__fsub_rn(nd.lo_h.y, hy), __fsub_rn(ly, nd.hi.y)));
  const float dz = fmaxf(0.f, fmaxf(__fsub_rn(nd.lo_h.z, hz), __fsub_rn(lz, nd.hi.z)));
  float d2 = __fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy));
  d2 = __fadd_rn(d2, __fmul_rn(dz, dz));
  const float H = sym ? fmaxf(h, nd.lo_h.w) : h;
  const float s = __fmul_rn(kappa, H);
  return __fmul_rn(d2, 1.f - 0x1p-20f) < __fmul_rn(s, s);
}

// The exact pair test (fp32, rounded as written).
__device__ __forceinline__ bool pair_in(const float4 &qi, float hi, const float4 &pj,
                                        float hj, float kappa, bool sym) {
  const float dx = __fsub_rn(qi.x, pj.x), dy = __fsub_rn(qi.y, pj.y),
              dz = __fsub_rn(qi.z, pj.z);
  float r2 = __fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy));
  r2 = __fadd_rn(r2, __fmul_rn(dz, dz));
  const float H = sym ? fmaxf(hi, hj) : hi;
  const float s = __fmul_rn(kappa, H);
  return r2 < __fmul_rn(s, s);
}

// Per-warp shared memory: a stack of node ranges [first, end) (children of
// opened cells, at most 8 each), and the particle ranges of the leaves opened
// in one round with their running offsets.
struct NbWarp {
  int2 stack[kNbStack];
  int leaf_f[32];
  int leaf_pre[33];
};

// kFill = false: counts; true: lists at offs (caller order).
template <bool kSym, bool kFill>
__global__ void __launch_bounds__(kNbThreads)
nb_walk_kernel(const float4 *__restrict__ spm, const float *__restrict__ sh,
               long long n, const int4 *__restrict__ topo,
               const NbNode *__restrict__ nodes, long long nnodes_cap,
               const unsigned int *__restrict__ perm, float kappa,
               unsigned int *counts, const unsigned long long *__restrict__ offs,
               unsigned int *list, unsigned long long list_cap, DevCtrl *ctrl) {
  __shared__ NbWarp smem[kNbWarps];
  NbWarp &W = smem[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;
  long long nnodes = node_total(ctrl);
  if (nnodes > nnodes_cap) nnodes = nnodes_cap;
  const long long ngroups = (n + 31) / 32;
  unsigned int *ticket = kFill ? &ctrl->step.fill_ctr : &ctrl->step.work_ctr;
  for (;;) {
    unsigned gg = 0;
    if (lane == 0) gg = atomicAdd(ticket, 1u);
    const long long g = __shfl_sync(kFull, gg, 0);
    if (g >= ngroups) break;
    const long long qi = g * 32 + lane;
    const bool valid = qi < n;
    const float4 q = spm[valid ? qi : n - 1];
    const float hq = valid ? sh[qi] : 0.f;
    // the group's bounding box and largest smoothing length
    float glo_x = q.x, glo_y = q.y, glo_z = q.z, ghi_x = q.x, ghi_y = q.y, ghi_z = q.z;
    float ghq = hq;
    for (int o = 16; o > 0; o >>= 1) {
      glo_x = fminf(glo_x, __shfl_xor_sync(kFull, glo_x, o));
      glo_y = fminf(glo_y, __shfl_xor_sync(kFull, glo_y, o));
      glo_z = fminf(glo_z, __shfl_xor_sync(kFull, glo_z, o));
      ghi_x = fmaxf(ghi_x, __shfl_xor_sync(kFull, ghi_x, o));
      ghi_y = fmaxf(ghi_y, __shfl_xor_sync(kFull, ghi_y, o));
      ghi_z = fmaxf(ghi_z, __shfl_xor_sync(kFull, ghi_z, o));
      ghq = fmaxf(ghq, __shfl_xor_sync(kFull, ghq, o));
    }
    // a group is spread out when its box is wider than half its largest
    // search radius; then the per-particle node test pays for itself.  (At
    // the full radius a group in the sparse outskirts whose box is just
    // under its one huge sphere -- h ~ 0.46 in a 2^18 Plummer sphere -- opened
    // a large part of the halo and walked 1.2M pair tests on one warp,
    // setting the time of the whole kernel.)
    const float ext = fmaxf(fmaxf(ghi_x - glo_x, ghi_y - glo_y), ghi_z - glo_z);
    const bool spread = ext > 0.5f * kappa * ghq;
    unsigned cnt = 0, tests = 0;
    unsigned long long base = 0;
    const unsigned dst = valid ? perm[qi] : 0u;
    if (kFill && valid && dst < n) base = offs[dst];
    if (lane == 0 && nnodes > 0) W.stack[0] = make_int2(0, 1);
    int sp = nnodes > 0 ? 1 : 0;
    __syncwarp();
    long long rounds = 0;
    while (sp > 0) {
      if (++rounds > nnodes + 1) {            // only a corrupt tree gets here
        set_err(ctrl, kErrOverflow);
        break;
      }
      // up to 32 nodes from the top ranges, one per lane
      int node = -1, got = 0;
      while (got < 32 && sp > 0) {
        const int2 r = W.stack[sp - 1];
        const int len = r.y - r.x;
        const int take = len < 32 - got ? len : 32 - got;
        if (lane >= got && lane < got + take) node = r.x + (lane - got);
        got += take;
        __syncwarp();
        if (take >= len) {
          --sp;
        } else if (lane == 0) {
          W.stack[sp - 1].x = r.x + take;
        }
        __syncwarp();
      }
      bool open = false, leaf = false;
      int4 t = make_int4(0, 0, -1, -1);
      NbNode nd;
      if (node >= 0 && node < nnodes) {
        t = topo[node];
        nd = nodes[node];
        // first against the group's box and largest h
        open = reaches(glo_x, glo_y, glo_z, ghi_x, ghi_y, ghi_z, ghq, nd, kappa, kSym);
        leaf = t.z < 0;
      }
      // then, where the group is spread out, against each particle's own
      // sphere: a node is opened only if some particle of the group can
      // reach it
      if (spread && __any_sync(kFull, open)) {
        bool any = false;
        for (int k = 0; k < 32; ++k) {
          const float x = __shfl_sync(kFull, q.x, k), y = __shfl_sync(kFull, q.y, k),
                      z = __shfl_sync(kFull, q.z, k), hk = __shfl_sync(kFull, hq, k);
          const bool vk = __shfl_sync(kFull, valid, k);
          if (open && vk && !any) any = reaches(x, y, z, x, y, z, hk, nd, kappa, kSym);
        }
        open = any;
      }
      // push the child range of each opened cell; children lie after their
      // parent in the breadth-first order and only such links are followed,
      // so every walk ends
      const bool push = open && !leaf && t.z > node && t.w > t.z && t.w <= nnodes &&
                        t.w - t.z <= 8;
      // lane 0 holds the deepest node taken; pushing in reverse lane order
      // keeps levels non-decreasing towards the top of the stack
      const unsigned pb = __ballot_sync(kFull, push);
      if (push) {
        const int at = sp + __popc(pb >> lane) - 1;
        if (at < kNbStack) W.stack[at] = make_int2(t.z, t.w);
        else set_err(ctrl, kErrOverflow);
      }
      sp += __popc(pb);
      if (sp > kNbStack) sp = kNbStack;
      // the particles of the opened leaves, 32 at a time (one load each)
      const bool lf = open && leaf;
      long long f = t.x < 0 ? 0 : t.x, e = t.y > n ? n : t.y;
      int len = lf && e > f ? (int)(e - f) : 0;
      int pre = len;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, pre, o);
        if (lane >= o) pre += y;
      }
      const int ptot = __shfl_sync(kFull, pre, 31);
      W.leaf_f[lane] = (int)f;
      W.leaf_pre[lane + 1] = pre;
      if (lane == 0) W.leaf_pre[0] = 0;
      __syncwarp();
      for (int c0 = 0; c0 < ptot; c0 += 32) {
        // lane l loads particle c0 + l of the concatenated leaf ranges
        const int pos = c0 + lane;
        int j = -1;
        float4 pj = make_float4(0.f, 0.f, 0.f, 0.f);
        float hj = 0.f;
        if (pos < ptot) {
          int lo = 0, hi = 31;                  // last leaf with pre <= pos
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (W.leaf_pre[mid] <= pos) lo = mid; else hi = mid - 1;
          }
          j = W.leaf_f[lo] + (pos - W.leaf_pre[lo]);
          pj = spm[j];
          hj = sh[j];
        }
        const int m = ptot - c0 < 32 ? ptot - c0 : 32;
        for (int k = 0; k < m; ++k) {
          const int jk = __shfl_sync(kFull, j, k);
          float4 pk;
          pk.x = __shfl_sync(kFull, pj.x, k);
          pk.y = __shfl_sync(kFull, pj.y, k);
          pk.z = __shfl_sync(kFull, pj.z, k);
          const float hk = __shfl_sync(kFull, hj, k);
          tests += valid;
          if (valid && jk != qi && pair_in(q, hq, pk, hk, kappa, kSym)) {
            if (kFill) {
              const unsigned long long at = base + cnt;
              if (at < list_cap) list[at] = perm[jk];
            }
            ++cnt;
          }
        }
      }
      __syncwarp();
    }
    if (valid && dst < n) {
      if (kFill) {
        if (base + cnt > list_cap) set_err(ctrl, kErrOverflow);
      } else {
        counts[dst] = cnt;
      }
    }
    if (!kFill) {                           // pair tests of the counting walk
      unsigned long long tt = tests;
      for (int o = 16; o > 0; o >>= 1) tt += __shfl_xor_sync(kFull, tt, o);
      if (lane == 0 && tt) atomicAdd(&ctrl->step.executed, tt);
    }
  }
}

// Exclusive scan of n u32 counts into n + 1 u64 offsets: block sums, a scan
// of the block sums by one block, then per-block scans.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
scan_block_sums(const unsigned int *__restrict__ x, long long n,
                unsigned long long *__restrict__ bsum) {
  __shared__ unsigned long long ws[32];
  const long long i = (long long)blockIdx.x * kScanThreads + threadIdx.x;
  unsigned long long v = i < n ? x[i] : 0ull;
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0;
    for (int k = 0; k < kScanThreads / 32; ++k) t += ws[k];
    bsum[blockIdx.x] = t;
  }
}

__global__ void __launch_bounds__(kScanThreads)
scan_sums(unsigned long long *bsum, long long nb) {
  __shared__ unsigned long long ws[32];
  __shared__ unsigned long long carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (long long b0 = 0; b0 < nb; b0 += kScanThreads) {
    const long long i = b0 + threadIdx.x;
    const unsigned long long v = i < nb ? bsum[i] : 0ull;
    unsigned long long x = v;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) ws[w] = x;
    __syncthreads();
    unsigned long long pre = carry, tot = 0;
    for (int k = 0; k < kScanThreads / 32; ++k) {
      if (k < w) pre += ws[k];
      tot += ws[k];
    }
    if (i < nb) bsum[i] = pre + x - v;
    __syncthreads();
    if (threadIdx.x == 0) carry += tot;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kScanThreads)
scan_apply(const unsigned int *__restrict__ x, long long n,
           const unsigned long long *__restrict__ bsum,
           unsigned long long *__restrict__ out) {
  __shared__ unsigned long long ws[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const long long i = (long long)blockIdx.x * kScanThreads + threadIdx.x;
  const unsigned long long v = i < n ? x[i] : 0ull;
  unsigned long long s = v;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(kFull, s, o);
    if (lane >= o) s += y;
  }
  if (lane == 31) ws[w] = s;
  __syncthreads();
  unsigned long long pre = bsum[blockIdx.x];
  for (int k = 0; k < w; ++k) pre += ws[k];
  if (i < n) out[i] = pre + s - v;
  if (i == n - 1) out[n] = pre + s;
}

template <bool kSym, bool kFill>
cudaError_t launch_walk_t(const NbArgs &a, DevCtrl *ctrl, cudaStream_t s) {
  static std::atomic<int> memo[kMaxDevices];
  const int per_sm = per_device(memo, [] {
    int b = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, nb_walk_kernel<kSym, kFill>,
                                                  kNbThreads, 0);
    return b > 0 ? b : 1;
  });
  const long long ngroups = (a.n + 31) / 32;
  long long blocks = (ngroups + kNbWarps - 1) / kNbWarps;
  const long long cap = (long long)a.num_sms * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  nb_walk_kernel<kSym, kFill><<<(unsigned)blocks, kNbThreads, 0, s>>>(
      a.spm, a.sh, a.n, a.topo, a.nodes, a.nodes_cap, a.perm, a.kappa, a.counts,
      a.offsets, a.list, a.list_cap, ctrl);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_neighbors(const NbArgs &a, const float *h, const int *parent,
                             int *arrive, unsigned long long *scan_tmp,
                             DevCtrl *ctrl, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  long long blocks = (a.n + 255) / 256;
  if (blocks > (long long)a.num_sms * 8) blocks = (long long)a.num_sms * 8;
  gather_h_kernel<<<(unsigned)blocks, 256, 0, s>>>(h, a.perm, a.n, a.sh, ctrl);
  nb_node_kernel<<<(unsigned)blocks, 256, 0, s>>>(a.spm, a.sh, a.n, a.topo, parent,
                                                  arrive, a.nodes, ctrl, a.nodes_cap);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = a.symmetric ? launch_walk_t<true, false>(a, ctrl, s)
                  : launch_walk_t<false, false>(a, ctrl, s);
  if (e != cudaSuccess || !a.offsets) return e;
  const long long nb = (a.n + kScanThreads - 1) / kScanThreads;
  scan_block_sums<<<(unsigned)nb, kScanThreads, 0, s>>>(a.counts, a.n, scan_tmp);
  scan_sums<<<1, kScanThreads, 0, s>>>(scan_tmp, nb);
  scan_apply<<<(unsigned)nb, kScanThreads, 0, s>>>(a.counts, a.n, scan_tmp, a.offsets);
  e = cudaGetLastError();
  if (e != cudaSuccess || !a.list) return e;
  return a.symmetric ? launch_walk_t<true, true>(a, ctrl, s)
                     : launch_walk_t<false, true>(a, ctrl, s);
}

}  // namespace bh
