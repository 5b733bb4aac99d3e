// Octree build over sorted Morton keys, and the bottom-up centre-of-mass pass.
//
// The tree is the one the tree page after Burtscher & Pingali builds by
// inserting particles and subdividing a cell until its particles separate
// (section "构建树结构"), restated on integer key prefixes so the result does
// not depend on insertion order: a cell of level l is a run of sorted keys
// sharing their top 3*l bits; it exists iff its parent holds more than the
// leaf capacity B; it is internal iff it holds more than B and l < bits.
// The page's builder locks child slots with atomicCAS and allocates nodes
// with a global counter (its "稠密存储" section); on GB300 the build is instead
// three data-parallel passes over the keys, no locks and no waits:
//
//   count  -- per position j: the first level at which j starts a cell
//             (one past the common-prefix length with key j-1) and the level
//             of its leaf (one past the deepest level whose cell holds more
//             than B keys, found from lcp(key_i, key_{i+B}) over the B+1
//             windows containing j).  Warp ballots count, per tile and per
//             level, how many cells start in the tile.
//   scan   -- one block per level turns the tile counts into tile offsets.
//   write  -- the same ballots give each cell its breadth-first index
//             (level offset + rank among the level's cells in key order).
//             The thread at a cell's first key writes (first, level, first
//             child, parent); the thread at the position just past its last
//             key writes (end, one-past-last child).
//
// Nodes come out breadth first with the children of a node contiguous and in
// octant order, so the walk reads a node's children as one coalesced block.
//
// Centre of mass (GASPHiA page, section "计算核函数": computeCenterOfMass):
// every leaf sums its particles; a child that finishes bumps its parent's
// arrival counter and the child that arrives last sums the parent's children
// (in index order, so the result is deterministic) and carries on upward.
// No thread ever waits for another.
#include <cuda_runtime.h>
#include <stdint.h>

#include "bh_internal.h"

namespace bh {

namespace {

__device__ __forceinline__ void set_err(DevCtrl *c, unsigned code) {
  atomicCAS(&c->keep.err, 0u, code);
}

// Common prefix of two keys in whole 3-bit levels (bits for equal keys).
__device__ __forceinline__ int lcp_levels(unsigned long long a,
                                          unsigned long long b, int bits) {
  unsigned long long x = a ^ b;
  if (x == 0ull) return bits;
  return (__clzll((long long)x) - (64 - 3 * bits)) / 3;
}

constexpr int kHalo = kMaxLeafCap + 1;

struct TileGeom {
  // keys of positions [tb - B - 1, tb + kBuildTile + B]
  unsigned long long k[kBuildTile + 2 * kHalo + 2];
  signed char lam[kBuildTile + kHalo + 1];   // lcp(key_i, key_{i+B})
  signed char D[kBuildTile + 1];             // deepest over-full level at j
};

// Fill the tile geometry for positions j in [tb, tb + kBuildTile).
__device__ void load_geom(TileGeom &g, const unsigned long long *skeys,
                          long long n, long long tb, int B, int bits) {
  const long long k0 = tb - B - 1;
  const int nk = kBuildTile + 2 * B + 2;
  for (int x = threadIdx.x; x < nk; x += blockDim.x) {
    long long i = k0 + x;
    g.k[x] = (i >= 0 && i < n) ? skeys[i] : 0ull;
  }
  __syncthreads();
  // lam[y] for i = k0 + y, y in [0, kBuildTile + B + 1)
  for (int y = threadIdx.x; y < kBuildTile + B + 1; y += blockDim.x) {
    long long i = k0 + y;
    signed char v = -1;
    if (i >= 0 && i + B <= n - 1) v = (signed char)lcp_levels(g.k[y], g.k[y + B], bits);
    g.lam[y] = v;
  }
  __syncthreads();
  // D[z] for j = tb - 1 + z: max lam over i in [j - B, j]  (lam index i - k0)
  for (int z = threadIdx.x; z < kBuildTile + 1; z += blockDim.x) {
    int m = -1;
    for (int q = 0; q <= B; ++q) {
      int v = g.lam[z + q];            // i = j - B + q  ->  y = z + q
      m = v > m ? v : m;
    }
    g.D[z] = (signed char)m;
  }
  __syncthreads();
}

// Leaf level from D: one past the deepest over-full level, capped at bits.
__device__ __forceinline__ int leaf_level(int D, int bits) {
  int l = D + 1;
  return l < bits ? l : bits;
}

constexpr int kLvWarps = kBuildThreads / 32;

// Per-position facts for position j of this tile.
__device__ __forceinline__ void position_facts(const TileGeom &g, long long n,
                                               long long tb, long long j,
                                               int B, int bits, int &s, int &L,
                                               int &e, int &Lp) {
  const long long k0 = tb - B - 1;
  s = bits + 1; L = -1; e = bits + 1; Lp = -1;
  if (j < 0 || j > n) return;
  const int z = (int)(j - (tb - 1));      // D index of j
  if (j < n) {
    L = (n > B) ? leaf_level(g.D[z], bits) : 0;
    if (j == 0) s = 0;
    else s = lcp_levels(g.k[j - 1 - k0], g.k[j - k0], bits) + 1;
  }
  if (j >= 1) {
    Lp = (n > B) ? leaf_level(g.D[z - 1], bits) : 0;
    e = (j == n) ? -1 : lcp_levels(g.k[j - 1 - k0], g.k[j - k0], bits);
  }
}

// ---------------------------------------------------------------------------
// count pass: per tile, per level, number of cells that start in the tile
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBuildThreads)
build_count_kernel(const unsigned long long *__restrict__ skeys, long long n,
                   int B, int bits, unsigned int *tile_counts, int ntiles) {
  __shared__ TileGeom g;
  __shared__ unsigned s_cnt[kMaxLevels];
  const long long tb = (long long)blockIdx.x * kBuildTile;
  if (threadIdx.x < kMaxLevels) s_cnt[threadIdx.x] = 0;
  load_geom(g, skeys, n, tb, B, bits);
  const int lane = threadIdx.x & 31;
  unsigned mine = 0;   // lane l accumulates level l
  for (int it = 0; it < kBuildIters; ++it) {
    long long j = tb + it * kBuildThreads + threadIdx.x;
    int s, L, e, Lp;
    position_facts(g, n, tb, j, B, bits, s, L, e, Lp);
    // only the levels some position of this warp starts a cell at
    const int lo = (int)__reduce_min_sync(0xffffffffu, (unsigned)(s <= L ? s : bits + 1));
    const int hi = __reduce_max_sync(0xffffffffu, L < 0 ? 0 : L);
    for (int l = lo; l <= hi; ++l) {
      unsigned b = __ballot_sync(0xffffffffu, s <= l && l <= L);
      if (lane == l) mine += __popc(b);
    }
  }
  if (lane <= bits && mine) atomicAdd(&s_cnt[lane], mine);
  __syncthreads();
  if (threadIdx.x <= bits)
    tile_counts[(long long)threadIdx.x * ntiles + blockIdx.x] = s_cnt[threadIdx.x];
}

// ---------------------------------------------------------------------------
// scan pass: block l scans the tile counts of level l (exclusive, in place)
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
build_scan_kernel(unsigned int *tile_counts, int ntiles, DevCtrl *ctrl) {
  __shared__ unsigned s_warp[kScanThreads / 32];
  __shared__ unsigned s_carry;
  const int l = blockIdx.x;
  unsigned *row = tile_counts + (long long)l * ntiles;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < ntiles; base += kScanThreads) {
    int t = base + threadIdx.x;
    unsigned v = t < ntiles ? row[t] : 0u;
    unsigned x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      unsigned y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[w] = x;
    __syncthreads();
    unsigned off = 0, tot = 0;
    for (int k = 0; k < kScanThreads / 32; ++k) {
      unsigned c = s_warp[k];
      if (k < w) off += c;
      tot += c;
    }
    unsigned carry = s_carry;
    if (t < ntiles) row[t] = carry + off + x - v;
    __syncthreads();
    if (threadIdx.x == 0) s_carry = carry + tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) ctrl->step.level_total[l] = (int)s_carry;
}

// ---------------------------------------------------------------------------
// write pass
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBuildThreads)
build_write_kernel(const unsigned long long *__restrict__ skeys, long long n,
                   int B, int bits, const unsigned int *__restrict__ tile_off,
                   int ntiles, DevCtrl *ctrl, int4 *topo, int *parent,
                   unsigned char *level, int *arrive, long long cap_nodes) {
  __shared__ TileGeom g;
  __shared__ unsigned s_cnt[kBuildIters][kLvWarps][kMaxLevels];
  __shared__ long long s_base[kMaxLevels + 1];
  __shared__ int s_ok;
  const long long tb = (long long)blockIdx.x * kBuildTile;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    long long off = 0;
    for (int l = 0; l <= bits; ++l) {
      s_base[l] = off + tile_off[(long long)l * ntiles + blockIdx.x];
      off += ctrl->step.level_total[l];
    }
    s_base[bits + 1] = off;
    s_ok = off <= cap_nodes;
    if (!s_ok && blockIdx.x == 0) set_err(ctrl, kErrOverflow);
  }
  for (int k = threadIdx.x; k < kBuildIters * kLvWarps * kMaxLevels; k += blockDim.x)
    (&s_cnt[0][0][0])[k] = 0u;
  load_geom(g, skeys, n, tb, B, bits);
  if (!s_ok) return;
  // phase A: per (iteration, warp, level) counts, over the warp's levels only
  int s[kBuildIters], L[kBuildIters], e[kBuildIters], Lp[kBuildIters];
#pragma unroll
  for (int it = 0; it < kBuildIters; ++it) {
    long long j = tb + it * kBuildThreads + threadIdx.x;
    position_facts(g, n, tb, j, B, bits, s[it], L[it], e[it], Lp[it]);
    const int lo = (int)__reduce_min_sync(0xffffffffu, (unsigned)(s[it] <= L[it] ? s[it] : bits + 1));
    const int hi = __reduce_max_sync(0xffffffffu, L[it] < 0 ? 0 : L[it]);
    for (int l = lo; l <= hi; ++l) {
      unsigned b = __ballot_sync(0xffffffffu, s[it] <= l && l <= L[it]);
      if (lane == 0) s_cnt[it][w][l] = __popc(b);
    }
  }
  __syncthreads();
  // phase B: exclusive offsets in (iteration, warp) order, per level
  if (threadIdx.x <= bits) {
    const int l = threadIdx.x;
    unsigned run = 0;
    for (int it = 0; it < kBuildIters; ++it)
      for (int k = 0; k < kLvWarps; ++k) {
        unsigned c = s_cnt[it][k][l];
        s_cnt[it][k][l] = run;
        run += c;
      }
  }
  __syncthreads();
  // phase C: ranks by ballot, level by level with a window of three levels
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int it = 0; it < kBuildIters; ++it) {
    const long long j = tb + it * kBuildThreads + threadIdx.x;
    const int sj = s[it], Lj = L[it], ej = e[it], Lpj = Lp[it];
    // r[l] = number of level-l cells that start before j (global index
    // offset included); st[l] = whether one starts at j.
    long long r_m1 = 0, r_0 = 0;
    bool st_m1 = false, st_0 = false;
    // Levels with a write in this warp: starts in [s, L], ends in (e, Lp].
    const int wlo = (int)__reduce_min_sync(
        0xffffffffu, (unsigned)min(sj <= Lj ? sj : bits + 1, ej + 1 <= Lpj ? ej + 1 : bits + 1));
    const int whi = __reduce_max_sync(0xffffffffu, (unsigned)max(max(Lj, Lpj), 0));
    const int l_first = wlo > 0 ? wlo - 1 : 0;
    const int l_last = whi + 1 < bits + 1 ? whi + 1 : bits + 1;
    for (int l = l_first; l <= l_last; ++l) {
      long long r_p1 = 0;
      bool st_p1 = false;
      if (l <= bits) {
        bool pred = sj <= l && l <= Lj;
        unsigned b = __ballot_sync(0xffffffffu, pred);
        r_p1 = s_base[l] + s_cnt[it][w][l] + __popc(b & lt);
        st_p1 = pred;
      }
      // handle level lv = l - 1 using ranks of lv - 1 (r_m1), lv (r_0), lv + 1 (r_p1)
      const int lv = l - 1;
      if (lv >= wlo && lv >= 0) {
        if (st_0) {                              // a cell of level lv starts at j
          long long idx = r_0;
          if (idx >= 0 && idx < cap_nodes) {
            int fc = (lv < Lj) ? (int)r_p1 : -1;   // first child starts at j too
            int par = -1;
            if (lv > 0) par = (int)(r_m1 + (st_m1 ? 0 : -1));
            topo[idx].x = (int)j;
            topo[idx].z = fc;
            parent[idx] = par;
            level[idx] = (unsigned char)lv;
            if (fc >= 0) arrive[idx] = 0;
          }
        }
        if (lv > ej && lv <= Lpj) {            // the cell holding j-1 ends at j
          long long idx = r_0 - 1;
          if (idx >= 0 && idx < cap_nodes) {
            topo[idx].y = (int)j;
            topo[idx].w = (lv < Lpj) ? (int)r_p1 : -1;
          }
        }
      }
      r_m1 = r_0; st_m1 = st_0;
      r_0 = r_p1; st_0 = st_p1;
    }
  }
}

// ---------------------------------------------------------------------------
// centre of mass, bottom up
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned compact3(unsigned long long key, int axis) {
  unsigned q = 0;
  for (int k = 0; k < kMaxBits; ++k)
    q |= (unsigned)((key >> (3 * k + axis)) & 1ull) << k;
  return q;
}

__device__ void finish_node(long long c, float4 sum, int lvl, int link,
                            int count, bool leaf, float4 cube, float theta,
                            int bits, const unsigned long long *skeys,
                            int first_particle, float4 *msum, NodeRec *rec) {
  msum[c] = sum;
  NodeRec r;
  const float w = ldexpf(cube.w, -lvl);            // full cell edge
  if (sum.w != 0.f) {
    const float inv = __frcp_rn(sum.w);
    r.com = make_float4(sum.x * inv, sum.y * inv, sum.z * inv, sum.w);
  } else {                                          // massless: cell centre
    unsigned long long key = skeys[first_particle];
    const int sh = bits - lvl;
    float ctr[3];
    const float lo[3] = {cube.x, cube.y, cube.z};
    for (int a = 0; a < 3; ++a) {
      unsigned cell = compact3(key, a) >> sh;
      ctr[a] = lo[a] + ((float)cell + 0.5f) * w;
    }
    r.com = make_float4(ctr[0], ctr[1], ctr[2], 0.f);
  }
  r.ropen2 = __fdiv_rn(__fmul_rn(w, w), __fmul_rn(theta, theta));
  r.link = link;
  r.count = count;
  r.flags = (leaf ? 1 : 0) | (lvl << 8);
  rec[c] = r;
}

__global__ void __launch_bounds__(256)
com_kernel(const float4 *__restrict__ spm, const unsigned long long *skeys,
           long long n, int bits, float theta, const int4 *__restrict__ topo,
           const int *__restrict__ parent, const unsigned char *__restrict__ level,
           int *arrive, float4 *msum, NodeRec *rec, DevCtrl *ctrl,
           long long cap_nodes) {
  long long total = 0;
  for (int l = 0; l <= bits; ++l) total += ctrl->step.level_total[l];
  if (total > cap_nodes) return;
  const float4 cube = ctrl->keep.cube[0];
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x;
       c < total; c += stride) {
    int4 t = topo[c];
    if (t.z >= 0) continue;                       // internal: done by a child
    long long f = t.x < 0 ? 0 : t.x;
    if (f > n) f = n;
    long long e = t.y < f ? f : t.y;
    if (e > n) e = n;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    long long j = f;
    for (; j + 4 <= e; j += 4) {          // four loads in flight
      float4 p[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) p[u] = __ldg(spm + j + u);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        s.x = fmaf(p[u].w, p[u].x, s.x);
        s.y = fmaf(p[u].w, p[u].y, s.y);
        s.z = fmaf(p[u].w, p[u].z, s.z);
        s.w += p[u].w;
      }
    }
    for (; j < e; ++j) {
      float4 p = __ldg(spm + j);
      s.x = fmaf(p.w, p.x, s.x);
      s.y = fmaf(p.w, p.y, s.y);
      s.z = fmaf(p.w, p.z, s.z);
      s.w += p.w;
    }
    int lvl = level[c];
    finish_node(c, s, lvl, (int)f, (int)(e - f), true, cube, theta, bits,
                skeys, (int)(f < n ? f : 0), msum, rec);
    // climb while this thread is the last child to finish
    long long node = c;
    for (int guard = 0; guard <= kMaxLevels; ++guard) {
      int p = parent[node];
      if (p < 0 || p >= total) break;
      __threadfence();
      int4 tp = topo[p];
      int nch = tp.w - tp.z;
      if (tp.z < 0 || nch < 1 || nch > 8 || tp.w > total) break;
      int old = atomicAdd(arrive + p, 1);
      if (old != nch - 1) break;
      __threadfence();
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = tp.z; k < tp.w; ++k) {
        float4 q = __ldcg(msum + k);
        a.x += q.x; a.y += q.y; a.z += q.z; a.w += q.w;
      }
      int plv = level[p];
      long long pf = tp.x < 0 ? 0 : (tp.x < n ? tp.x : 0);
      finish_node(p, a, plv, tp.z, nch, false, cube, theta, bits, skeys,
                  (int)pf, msum, rec);
      node = p;
    }
  }
}

}  // namespace

cudaError_t launch_build(const unsigned long long *skeys, long long n, int bits,
                         int leaf_cap, BuildBufs &b, DevCtrl *ctrl,
                         cudaStream_t s) {
  const long long ntiles = (n + 1 + kBuildTile - 1) / kBuildTile;  // positions 0..n
  if (ntiles > b.cap_tiles) return cudaErrorInvalidValue;
  build_count_kernel<<<(unsigned)ntiles, kBuildThreads, 0, s>>>(
      skeys, n, leaf_cap, bits, b.tile_counts, (int)ntiles);
  build_scan_kernel<<<bits + 1, kScanThreads, 0, s>>>(b.tile_counts, (int)ntiles,
                                                      ctrl);
  build_write_kernel<<<(unsigned)ntiles, kBuildThreads, 0, s>>>(
      skeys, n, leaf_cap, bits, b.tile_counts, (int)ntiles, ctrl, b.topo,
      b.parent, b.level, b.arrive, b.cap_nodes);
  return cudaGetLastError();
}

cudaError_t launch_com(const float4 *spm, const unsigned long long *skeys,
                       long long n, int bits, float theta, BuildBufs &b,
                       DevCtrl *ctrl, cudaStream_t s) {
  int blocks = sm_count() * 8;
  com_kernel<<<blocks, 256, 0, s>>>(spm, skeys, n, bits, theta, b.topo,
                                    b.parent, b.level, b.arrive, b.msum, b.rec,
                                    ctrl, b.cap_nodes);
  return cudaGetLastError();
}

}  // namespace bh
