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
//             windows containing j), stored for the write pass.  Warp
//             ballots count, per tile and per level, how many cells start in
//             the tile.
//   scan   -- one block per level turns the tile counts into tile offsets.
//   write  -- from the stored levels (no keys needed), the same ballots
//             give each cell its breadth-first index
//             (level offset + rank among the level's cells in key order).
//             The thread at a cell's first key writes (first, level, first
//             child, parent); the thread at the position just past its last
//             key writes (end, one-past-last child).
//
// Nodes come out breadth first with the children of a node contiguous and in
// octant order, so the walk reads a node's children as one coalesced block.
//
// Centre of mass (GASPHiA page, section "计算核函数": computeCenterOfMass):
// a cell's mass and mass moments are sums over a contiguous range of the
// sorted particles, so they are differences of two prefix sums.  The prefix
// sums are kept exactly: every particle's mass m and moments m (x - lo)
// (per axis, lo = the cube's corner) are scaled by powers of two chosen from
// the largest |m|, the cube and n, and rounded to 64-bit integers (the
// product m (x - lo) is formed exactly from the two 24-bit mantissas, so the
// only rounding is the final one, to half a unit of 2^-k), which makes the
// sums exact and independent of the order they are formed in.  The write
// pass forms them for its tile: the thread at a cell's first key records the
// prefix there and the thread one past its last key the prefix at the end,
// both relative to their tile, and the tile's sums go out; one block turns
// the tiles' sums into tile prefixes.  Every node then takes mass =
// difference of the mass prefixes and com = lo + (difference of the moment
// prefixes) / mass, on its own: no pass waits for its children.
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
constexpr int kLamLen = kBuildTile + kHalo + 1;

struct TileGeom {
  // keys of positions [tb - B - 1, tb + kBuildTile + B]
  unsigned long long k[kBuildTile + 2 * kHalo + 2];
  signed char lam[2][kLamLen];               // lcp(key_i, key_{i+B}), and
                                             // window maxima built from it
  signed char D[kBuildTile + 1];             // deepest over-full level at j
};

// The tile's keys (with the halos) into shared memory, every load issued
// before the first store; no barrier.
constexpr int kKeyLoads = (kBuildTile + 2 * kHalo + 2 + kBuildThreads - 1) / kBuildThreads;

__device__ __forceinline__ void load_keys(TileGeom &g, const unsigned long long *skeys,
                                          long long n, long long tb, int B) {
  const long long k0 = tb - B - 1;
  const int nk = kBuildTile + 2 * B + 2;
  unsigned long long v[kKeyLoads];
#pragma unroll
  for (int u = 0; u < kKeyLoads; ++u) {
    const int x = threadIdx.x + u * kBuildThreads;
    const long long i = k0 + x;
    v[u] = (x < nk && i >= 0 && i < n) ? __ldg(skeys + i) : 0ull;
  }
#pragma unroll
  for (int u = 0; u < kKeyLoads; ++u) {
    const int x = threadIdx.x + u * kBuildThreads;
    if (x < nk) g.k[x] = v[u];
  }
}

// Fill the tile geometry for positions j in [tb, tb + kBuildTile).
// D_j = max of lam over the B + 1 windows [i, i + B] that contain j; the
// maximum over B + 1 consecutive values comes from a sparse table: the
// maxima of runs of 2^s values by doubling, then two overlapping runs.
__device__ void load_geom(TileGeom &g, const unsigned long long *skeys,
                          long long n, long long tb, int B, int bits) {
  load_keys(g, skeys, n, tb, B);
  const long long k0 = tb - B - 1;
  __syncthreads();
  // lam[y] for i = k0 + y, y in [0, kBuildTile + B + 1)
  const int nl = kBuildTile + B + 1;
  for (int y = threadIdx.x; y < nl; y += blockDim.x) {
    long long i = k0 + y;
    signed char v = -1;
    if (i >= 0 && i + B <= n - 1) v = (signed char)lcp_levels(g.k[y], g.k[y + B], bits);
    g.lam[0][y] = v;
  }
  __syncthreads();
  // runs of p = 2^s values: run[y] = max lam[y .. y + p - 1]
  const int W = B + 1;
  int p = 1, cur = 0;
  while (2 * p <= W) {
    for (int y = threadIdx.x; y + p < nl; y += blockDim.x) {
      const signed char a = g.lam[cur][y], b = g.lam[cur][y + p];
      g.lam[cur ^ 1][y] = a > b ? a : b;
    }
    __syncthreads();
    cur ^= 1;
    p *= 2;
  }
  // D[z] for j = tb - 1 + z: windows i in [j - B, j] -> lam index z .. z + B
  for (int z = threadIdx.x; z < kBuildTile + 1; z += blockDim.x) {
    const signed char a = g.lam[cur][z], b = g.lam[cur][z + W - p];
    g.D[z] = a > b ? a : b;
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
// fixed-point moments of one particle: (m, m dx, m dy, m dz) scaled by
// 2^k_m and 2^k_x, d = coordinate - lo rounded once in fp32
// ---------------------------------------------------------------------------
struct Q4 {
  long long m, x, y, z;
};

// A float as mantissa 2^(e - 150): the 24-bit mantissa with its hidden bit
// (none for a subnormal, whose e is then 1) and the biased exponent e.
__device__ __forceinline__ unsigned split_float(float v, int &e) {
  const unsigned u = __float_as_uint(v);
  e = (int)((u >> 23) & 0xffu);
  const unsigned mant = u & 0x7fffffu;
  if (e) return mant | 0x800000u;
  e = 1;
  return mant;
}

// P 2^s rounded to the nearest integer (ties away from zero); the result
// must be below 2^63.  ((P >> (t - 1)) + 1) >> 1 is (P + 2^(t-1)) >> t
// without the overflow.
__device__ __forceinline__ unsigned long long shift_round(unsigned long long P, int s) {
  const int sl = s < 0 ? 0 : (s > 63 ? 63 : s);
  const int t = -s < 1 ? 1 : (-s > 64 ? 64 : -s);
  const unsigned long long left = P << sl;
  const unsigned long long right = ((P >> (t - 1)) + 1ull) >> 1;
  return s >= 0 ? left : right;
}

// Moments of one particle, exact up to the final rounding to an integer:
// m 2^k_m, and m d 2^k_x per axis with d = coordinate - lo (rounded once in
// fp32, >= 0), the product m d formed exactly as (M D) 2^(e_m + e_d - 300)
// from the two mantissas.
__device__ __forceinline__ Q4 moments(float4 p, float4 cube, int km, int kx) {
  int em;
  const unsigned M = split_float(p.w, em);
  const bool neg = __float_as_uint(p.w) >> 31;
  const float d[3] = {__fsub_rn(p.x, cube.x), __fsub_rn(p.y, cube.y),
                      __fsub_rn(p.z, cube.z)};
  long long v[4];
  v[0] = (long long)shift_round(M, em - 150 + km);
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    int ed;
    const unsigned D = split_float(d[a], ed);
    v[1 + a] = (long long)shift_round((unsigned long long)M * D, em + ed - 300 + kx);
  }
  Q4 q;
  q.m = neg ? -v[0] : v[0];
  q.x = neg ? -v[1] : v[1];
  q.y = neg ? -v[2] : v[2];
  q.z = neg ? -v[3] : v[3];
  return q;
}

__device__ __forceinline__ void q_add(Q4 &a, const Q4 &b) {
  a.m += b.m; a.x += b.x; a.y += b.y; a.z += b.z;
}

__device__ __forceinline__ Q4 q_shfl_xor(const Q4 &a, int o) {
  Q4 r;
  r.m = __shfl_xor_sync(0xffffffffu, a.m, o);
  r.x = __shfl_xor_sync(0xffffffffu, a.x, o);
  r.y = __shfl_xor_sync(0xffffffffu, a.y, o);
  r.z = __shfl_xor_sync(0xffffffffu, a.z, o);
  return r;
}

__device__ __forceinline__ Q4 q_shfl_up(const Q4 &a, int o) {
  Q4 r;
  r.m = __shfl_up_sync(0xffffffffu, a.m, o);
  r.x = __shfl_up_sync(0xffffffffu, a.x, o);
  r.y = __shfl_up_sync(0xffffffffu, a.y, o);
  r.z = __shfl_up_sync(0xffffffffu, a.z, o);
  return r;
}

// Moments of the kQPer consecutive positions tb + kQPer * threadIdx.x + u of
// this tile (0 past the last particle); `each` receives them one by one.
constexpr int kQPer = kBuildTile / kBuildThreads;

__device__ __forceinline__ void thread_moments(const float4 *__restrict__ spm, long long n,
                                               long long tb, float4 cube, int km, int kx,
                                               Q4 (&each)[kQPer]) {
  const long long j0 = tb + (long long)kQPer * threadIdx.x;
  float4 p[kQPer];
#pragma unroll
  for (int u = 0; u < kQPer; ++u)
    p[u] = (j0 + u < n) ? __ldg(spm + j0 + u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int u = 0; u < kQPer; ++u) each[u] = moments(p[u], cube, km, kx);
}

// ---------------------------------------------------------------------------
// count pass: per tile, per level, number of cells that start in the tile
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kBuildThreads)
build_count_kernel(const unsigned long long *__restrict__ skeys, long long n,
                   int B, int bits, unsigned int *tile_counts, int ntiles,
                   signed char *__restrict__ facts) {
  __shared__ TileGeom g;
  __shared__ unsigned s_cnt[kMaxLevels];
  const long long tb = (long long)blockIdx.x * kBuildTile;
  if (threadIdx.x < kMaxLevels) s_cnt[threadIdx.x] = 0;
  const int lane = threadIdx.x & 31;
  load_geom(g, skeys, n, tb, B, bits);       // synchronises the block
  unsigned mine = 0;   // lane l accumulates level l
  for (int it = 0; it < kBuildIters; ++it) {
    long long j = tb + it * kBuildThreads + threadIdx.x;
    int s, L, e, Lp;
    position_facts(g, n, tb, j, B, bits, s, L, e, Lp);
    // the write pass takes (s, L) from here instead of the keys
    if (j < n) reinterpret_cast<char2 *>(facts)[j] = make_char2((signed char)s, (signed char)L);
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

// Exclusive scan, in place, of vals[0], vals[stride], ..., vals[(count-1)
// stride] by one block; returns the total.  Each thread takes kScanPer
// consecutive values per chunk (one chunk covers 4096 values: 4M keys).
constexpr int kScanPer = 4;

template <typename T>
__device__ long long block_scan_column(T *vals, long long stride, int count) {
  __shared__ long long s_warp[kScanThreads / 32];
  __shared__ long long s_carry, s_chunk;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < count; base += kScanThreads * kScanPer) {
    const int t0 = base + threadIdx.x * kScanPer;
    long long v[kScanPer];
    long long run = 0;                       // this thread's values
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      v[u] = t0 + u < count ? (long long)vals[stride * (t0 + u)] : 0;
      run += v[u];
    }
    long long x = run;                       // inclusive over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[w] = x;
    __syncthreads();
    if (w == 0) {                            // the warps' totals, exclusive
      const long long tw = s_warp[lane];
      long long xw = tw;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, xw, o);
        if (lane >= o) xw += y;
      }
      s_warp[lane] = xw - tw;
      if (lane == 31) s_chunk = xw;
    }
    __syncthreads();
    long long acc = s_carry + s_warp[w] + (x - run);
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      if (t0 + u < count) vals[stride * (t0 + u)] = (T)acc;
      acc += v[u];
    }
    __syncthreads();
    if (threadIdx.x == 0) s_carry += s_chunk;
    __syncthreads();
  }
  return s_carry;
}

__global__ void __launch_bounds__(kScanThreads)
build_scan_kernel(unsigned int *tile_counts, int ntiles, DevCtrl *ctrl) {
  const int l = blockIdx.x;
  const long long tot = block_scan_column(tile_counts + (long long)l * ntiles, 1, ntiles);
  if (threadIdx.x == 0) ctrl->step.level_total[l] = (int)tot;
}

// ---------------------------------------------------------------------------
// write pass
// ---------------------------------------------------------------------------
// Dynamic shared memory of the write pass: the moment prefix at each of the
// tile's positions.
constexpr size_t kWriteDynSmem = sizeof(long long) * 4 * kBuildTile;
// Writes, per node, the moment prefixes at its first particle and one past
// its last, each relative to the start of the tile holding that position
// (the tile's own prefix is added by the centre-of-mass pass), and the
// tile's moment sums to tile_q[4 tile ..].
__global__ void __launch_bounds__(kBuildThreads, 4)
build_write_kernel(const signed char *__restrict__ facts,
                   const float4 *__restrict__ spm, long long n,
                   int B, int bits, const unsigned int *__restrict__ tile_off,
                   long long *tile_q, int ntiles, DevCtrl *ctrl, int4 *topo,
                   int *parent, unsigned char *level, int *arrive, long long *pq,
                   long long cap_nodes) {
  __shared__ unsigned s_cnt[kBuildIters][kLvWarps][kMaxLevels];
  __shared__ long long s_base[kMaxLevels + 1];
  __shared__ long long s_wq[kBuildThreads / 32][4];
  __shared__ int s_ok;
  extern __shared__ longlong2 s_P[];       // [kBuildTile][2]: (m, x), (y, z)
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int tile = blockIdx.x;
  const long long tb = (long long)tile * kBuildTile;
  // per position j, as the count pass found them: the first level at which
  // j starts a cell and its leaf level, and the leaf level at j - 1; loaded
  // with the particles, packed one byte each until the moments are done
  unsigned packed[kBuildIters];
#pragma unroll
  for (int it = 0; it < kBuildIters; ++it) {
    const long long j = tb + it * kBuildThreads + threadIdx.x;
    unsigned sl = 0xffffu & (unsigned)((bits + 1) | (0xff << 8));   // s = bits + 1, L = -1
    unsigned lp = 0xffu;                                            // Lp = -1
    if (j < n) sl = __ldg(reinterpret_cast<const unsigned short *>(facts) + j);
    if (j >= 1 && j <= n) lp = (unsigned char)__ldg(facts + 2 * (j - 1) + 1);
    packed[it] = sl | (lp << 16);
  }
  // the tile's moments: local exclusive prefix at positions
  // tb + kQPer * threadIdx.x + u, and the tile's sums
  {
    Q4 each[kQPer];
    thread_moments(spm, n, tb, ctrl->keep.cube[0], ctrl->keep.qexp[0][0],
                   ctrl->keep.qexp[0][1], each);
    Q4 t = each[0];
#pragma unroll
    for (int u = 1; u < kQPer; ++u) q_add(t, each[u]);
    Q4 x = t;                                  // inclusive over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      Q4 y = q_shfl_up(x, o);
      if (lane >= o) q_add(x, y);
    }
    if (lane == 31) {
      s_wq[w][0] = x.m; s_wq[w][1] = x.x; s_wq[w][2] = x.y; s_wq[w][3] = x.z;
    }
    __syncthreads();
    if (threadIdx.x < 4) {
      long long agg = 0;
      for (int k = 0; k < kBuildThreads / 32; ++k) agg += s_wq[k][threadIdx.x];
      tile_q[4LL * tile + threadIdx.x] = agg;
    }
    Q4 run;
    run.m = x.m - t.m; run.x = x.x - t.x; run.y = x.y - t.y; run.z = x.z - t.z;
    for (int k = 0; k < w; ++k) {
      run.m += s_wq[k][0]; run.x += s_wq[k][1]; run.y += s_wq[k][2]; run.z += s_wq[k][3];
    }
#pragma unroll
    for (int u = 0; u < kQPer; ++u) {
      const int pos = kQPer * threadIdx.x + u;
      s_P[2 * pos] = make_longlong2(run.m, run.x);
      s_P[2 * pos + 1] = make_longlong2(run.y, run.z);
      q_add(run, each[u]);
    }
  }
  if (w == 0) {
    // level l's first index in this tile: the nodes of the levels above it
    // (a scan across lanes) plus the tile offset within the level; all the
    // loads in flight at once
    const bool in = lane <= bits;
    const long long tot = in ? ctrl->step.level_total[lane] : 0;
    const long long toff = in ? tile_off[(long long)lane * ntiles + tile] : 0;
    long long x = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (in) s_base[lane] = x - tot + toff;
    const long long all = __shfl_sync(0xffffffffu, x, 31);
    if (lane == 0) {
      s_base[bits + 1] = all;
      s_ok = all <= cap_nodes;
      if (!s_ok && tile == 0) set_err(ctrl, kErrOverflow);
    }
  }
  for (int k = threadIdx.x; k < kBuildIters * kLvWarps * kMaxLevels; k += blockDim.x)
    (&s_cnt[0][0][0])[k] = 0u;
  __syncthreads();                           // counts zeroed, bases set
  if (!s_ok) return;
  // s: first level at which j starts a cell, L: its leaf level; e: the cells
  // of levels above e that hold j - 1 end at j (lcp(key j-1, key j) = s - 1;
  // -1 at j = n), Lp: the leaf level at j - 1; out of range nothing starts
  // or ends
  int s[kBuildIters], L[kBuildIters], e[kBuildIters], Lp[kBuildIters];
#pragma unroll
  for (int it = 0; it < kBuildIters; ++it) {
    const long long j = tb + it * kBuildThreads + threadIdx.x;
    s[it] = (signed char)(packed[it] & 0xffu);
    L[it] = (signed char)((packed[it] >> 8) & 0xffu);
    Lp[it] = (signed char)((packed[it] >> 16) & 0xffu);
    e[it] = (j >= 1 && j < n) ? s[it] - 1 : (j == n ? -1 : bits + 1);
  }
  // phase A: per (iteration, warp, level) counts, over the warp's levels only
#pragma unroll
  for (int it = 0; it < kBuildIters; ++it) {
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
            longlong2 *d = reinterpret_cast<longlong2 *>(pq + 8 * idx);
            d[0] = s_P[2 * (j - tb)];
            d[1] = s_P[2 * (j - tb) + 1];
          }
        }
        if (lv > ej && lv <= Lpj) {            // the cell holding j-1 ends at j
          long long idx = r_0 - 1;
          if (idx >= 0 && idx < cap_nodes) {
            topo[idx].y = (int)j;
            topo[idx].w = (lv < Lpj) ? (int)r_p1 : -1;
            longlong2 *d = reinterpret_cast<longlong2 *>(pq + 8 * idx + 4);
            d[0] = s_P[2 * (j - tb)];
            d[1] = s_P[2 * (j - tb) + 1];
          }
        }
      }
      r_m1 = r_0; st_m1 = st_0;
      r_0 = r_p1; st_0 = st_p1;
    }
  }
}

// ---------------------------------------------------------------------------
// the tiles' moment sums -> exclusive prefixes (one block, exact integers)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kScanThreads)
tile_prefix_kernel(long long *tile_q, int ntiles) {
  block_scan_column(tile_q + blockIdx.x, 4, ntiles);    // one column per block
}

// ---------------------------------------------------------------------------
// centre of mass: every node on its own, from its two moment prefixes
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned compact3(unsigned long long key, int axis) {
  unsigned q = 0;
  for (int k = 0; k < kMaxBits; ++k)
    q |= (unsigned)((key >> (3 * k + axis)) & 1ull) << k;
  return q;
}

// Centre of mass and mass of node c from its two moment prefixes (every
// operation explicitly rounded, so any thread computing a node gets the
// same bits); a massless node takes its cell's centre.
__device__ __forceinline__ float4 node_com(long long c, const unsigned long long *skeys,
                                           long long n, int bits, const int4 *topo,
                                           const unsigned char *level, const long long *pq,
                                           const long long *tile_pre, float4 cube, int km,
                                           int kx, int4 &t, int &lvl) {
  t = topo[c];
  lvl = level[c];
  const long long first = t.x < 0 ? 0 : (t.x > n ? n : t.x);
  const long long end = t.y < first ? first : (t.y > n ? n : t.y);
  // prefixes at first and end: the node's tile-relative values plus the
  // prefix before the tile each position falls in
  const longlong2 *q = reinterpret_cast<const longlong2 *>(pq + 8 * c);
  const longlong2 *tf = reinterpret_cast<const longlong2 *>(tile_pre + 4 * (first / kBuildTile));
  const longlong2 *te = reinterpret_cast<const longlong2 *>(tile_pre + 4 * (end / kBuildTile));
  longlong2 f0 = q[0], f1 = q[1], e0 = q[2], e1 = q[3];
  const longlong2 tf0 = tf[0], tf1 = tf[1], te0 = te[0], te1 = te[1];
  f0.x += tf0.x; f0.y += tf0.y; f1.x += tf1.x; f1.y += tf1.y;
  e0.x += te0.x; e0.y += te0.y; e1.x += te1.x; e1.y += te1.y;
  const long long dm = e0.x - f0.x;
  if (dm != 0) {
    // com - lo = (sum m d 2^kx) / (sum m 2^km) * 2^(km - kx)
    const float fm = __ll2float_rn(dm);
    const int sc = km - kx;
    return make_float4(
        __fadd_rn(cube.x, ldexpf(__fdiv_rn(__ll2float_rn(e0.y - f0.y), fm), sc)),
        __fadd_rn(cube.y, ldexpf(__fdiv_rn(__ll2float_rn(e1.x - f1.x), fm), sc)),
        __fadd_rn(cube.z, ldexpf(__fdiv_rn(__ll2float_rn(e1.y - f1.y), fm), sc)),
        ldexpf(fm, -km));
  }
  const float w = ldexpf(cube.w, -lvl);                 // massless: cell centre
  const unsigned long long key = skeys[first < n ? first : 0];
  const int sh = bits - lvl;
  float ctr[3];
  const float lo[3] = {cube.x, cube.y, cube.z};
  for (int a = 0; a < 3; ++a) {
    const unsigned cell = compact3(key, a) >> sh;
    ctr[a] = __fadd_rn(lo[a], __fmul_rn(__fadd_rn((float)cell, 0.5f), w));
  }
  return make_float4(ctr[0], ctr[1], ctr[2], 0.f);
}

// Per internal node, the factor F that lets the walk accept all children at
// once: with r the largest distance from the node's centre of mass to a
// child's, every child's centre lies at least d - r from a target box that
// is d from the node's (distance to a set is 1-Lipschitz), and a child's
// opening test w_c^2/theta^2 < d_c^2 (w_c = w/2) then holds whenever
// d^2 > (w^2/theta^2) (1/2 + theta r / w)^2.  F = that factor times 1 + 1e-4
// (so fp32 rounding of either test cannot part them), rounded up to a
// multiple of 2^-16 and stored as F 2^16 in flags bits 16..31 when F < 1;
// 0 = never (an opened node has d^2 <= w^2/theta^2, so F >= 1 cannot hold).
__device__ __forceinline__ unsigned children_factor(float r2max, float w, float theta) {
  const float rho = __fdiv_ru(__fsqrt_ru(r2max), w);
  const float f = __fmaf_ru(theta, rho, 0.5f);
  const float F = __fmul_ru(__fmul_ru(f, f), 1.0001f);
  if (!(F < 1.f)) return 0u;
  const float q = ceilf(__fmul_ru(F, 65536.f));
  return q >= 65535.f ? 0u : (unsigned)q;
}

__global__ void __launch_bounds__(256, 5)
com_kernel(const unsigned long long *__restrict__ skeys, long long n, int bits,
           float theta, const int4 *__restrict__ topo,
           const unsigned char *__restrict__ level, const long long *__restrict__ pq,
           const long long *__restrict__ tile_pre, NodeRec *__restrict__ rec,
           const DevCtrl *__restrict__ ctrl, long long cap_nodes) {
  const long long total = node_total(ctrl);
  if (total > cap_nodes) return;
  const float4 cube = ctrl->keep.cube[0];
  const int km = ctrl->keep.qexp[0][0], kx = ctrl->keep.qexp[0][1];
  const float th2 = __fmul_rn(theta, theta);
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x;
       c < total; c += stride) {
    int4 t;
    int lvl;
    NodeRec r;
    r.com = node_com(c, skeys, n, bits, topo, level, pq, tile_pre, cube, km, kx, t, lvl);
    const bool leaf = t.z < 0;
    const long long first = t.x < 0 ? 0 : (t.x > n ? n : t.x);
    const long long end = t.y < first ? first : (t.y > n ? n : t.y);
    const float w = ldexpf(cube.w, -lvl);            // full cell edge
    r.ropen2 = __fdiv_rn(__fmul_rn(w, w), th2);
    if (leaf) {
      r.link = (int)first;
      r.count = (int)(end - first);
    } else {
      const int nch = t.w - t.z;
      const bool ok = nch >= 1 && nch <= 8 && t.w <= total && t.z > c;
      r.link = t.z;
      r.count = ok ? nch : 0;
    }
    r.flags = (leaf ? 1 : 0) | (lvl << 8);
    rec[c] = r;
  }
}

// Per internal node, from the finished records: the largest distance from
// its centre of mass to a child's, turned into the children factor (flags
// bits 16..31).  Only the node's own thread writes its flags; other threads
// read only centres of mass, which no thread writes here.
__global__ void __launch_bounds__(256)
children_factor_kernel(NodeRec *rec, int bits, float theta,
                       const DevCtrl *__restrict__ ctrl, long long cap_nodes) {
  const float L = ctrl->keep.cube[0].w;
  const long long total = node_total(ctrl);
  if (total > cap_nodes || !(theta > 0.f)) return;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x;
       c < total; c += stride) {
    const int4 q = *reinterpret_cast<const int4 *>(&rec[c].ropen2);  // (ro2, link, count, flags)
    const int flags = q.w, link = q.y, count = q.z;
    if ((flags & 1) || count < 1 || count > 8 || link <= c || link + count > total) continue;
    const float4 cp = __ldg(reinterpret_cast<const float4 *>(rec + c));
    float4 ck[8];                            // all children's loads in flight
#pragma unroll
    for (int k = 0; k < 8; ++k)
      ck[k] = __ldg(reinterpret_cast<const float4 *>(rec + link + (k < count ? k : 0)));
    float r2max = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float dx = __fsub_rn(ck[k].x, cp.x), dy = __fsub_rn(ck[k].y, cp.y),
                  dz = __fsub_rn(ck[k].z, cp.z);
      r2max = fmaxf(r2max, __fadd_ru(__fadd_ru(__fmul_ru(dx, dx), __fmul_ru(dy, dy)),
                                     __fmul_ru(dz, dz)));
    }
    const float w = ldexpf(L, -((flags >> 8) & 255));
    rec[c].flags = flags | (int)(children_factor(r2max, w, theta) << 16);
  }
}

}  // namespace

cudaError_t launch_build(const unsigned long long *skeys, const float4 *spm,
                         long long n, int bits, int leaf_cap, BuildBufs &b,
                         DevCtrl *ctrl, cudaStream_t s) {
  const long long ntiles = (n + 1 + kBuildTile - 1) / kBuildTile;  // positions 0..n
  if (ntiles > b.cap_tiles) return cudaErrorInvalidValue;
  // the write pass's moment prefix takes it past the 48 KB default
  static std::atomic<int> memo[kMaxDevices];
  const int opted = per_device(memo, [] {
    return cudaFuncSetAttribute(build_write_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kWriteDynSmem) == cudaSuccess ? 1 : -1;
  });
  if (opted < 0) return cudaErrorInvalidValue;
  {
    const cudaError_t le = launch_k(build_count_kernel, dim3((unsigned)ntiles), dim3(kBuildThreads), 0, s,
      skeys, n, leaf_cap, bits, b.tile_counts, (int)ntiles, b.facts);
    if (le != cudaSuccess) return le;
  }
  {
    const cudaError_t le = launch_k(build_scan_kernel, dim3(bits + 1), dim3(kScanThreads), 0, s,
                                    b.tile_counts, (int)ntiles, ctrl);
    if (le != cudaSuccess) return le;
  }
  {
    const cudaError_t le = launch_k(build_write_kernel, dim3((unsigned)ntiles), dim3(kBuildThreads), kWriteDynSmem, s,
      b.facts, spm, n, leaf_cap, bits, b.tile_counts, b.tile_q, (int)ntiles, ctrl,
      b.topo, b.parent, b.level, b.arrive, b.pq, b.cap_nodes);
    if (le != cudaSuccess) return le;
  }
  {
    const cudaError_t le = launch_k(tile_prefix_kernel, dim3(4), dim3(kScanThreads), 0, s,
                                    b.tile_q, (int)ntiles);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

cudaError_t launch_com(const float4 *spm, const unsigned long long *skeys,
                       long long n, int bits, float theta, BuildBufs &b,
                       DevCtrl *ctrl, cudaStream_t s) {
  (void)spm;
  int blocks = sm_count() * 8;
  {
    const cudaError_t le = launch_k(com_kernel, dim3(blocks), dim3(256), 0, s,
                                    skeys, n, bits, theta, b.topo, b.level, b.pq,
                                    b.tile_q, b.rec, ctrl, b.cap_nodes);
    if (le != cudaSuccess) return le;
  }
  {
    const cudaError_t le = launch_k(children_factor_kernel, dim3(blocks), dim3(256), 0, s,
                                    b.rec, bits, theta, ctrl, b.cap_nodes);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

}  // namespace bh
