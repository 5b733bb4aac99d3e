// Stochastic Barnes-Hut ("Stochastic Barnes-Hut Approximation for Fast
// Summation on the GPU", section 方法, key designs 1-4).
//
// The exact sum over the sources is a telescoping sum along each source's
// root-to-leaf path: refining a cell T replaces its monopole by its children's,
//   Delta_T(q) = sum_{c child of T} m_c f(p_c, q) - m_T f(p_T, q).
// Per stratum R (the octree's cells at level s, plus leaves above s) a query
// takes R's monopole and one random path per sample: the path index I is
// uniform among R's particles, each step continues with probability
// p = min(1, max(1, beta_T) / beta_c) (beta = distance to the centre of mass
// over the cell edge; a leaf's children are its particles, of size half the
// leaf edge), and a surviving step adds Delta_T * (n_R / n_T) / P(reach it).
//
// GPU layout: one warp per group of 32 consecutive Morton-ordered queries,
// one query per lane.  The random numbers belong to the group (the page
// shares seeds across a warp), so every lane follows the same path I and
// the node loads are warp-uniform; lanes differ only in where their roulette
// stops.  Random numbers: Philox4x64-10 with key (seed, 0) and counter
// (group, stratum, sample, block); block 0 word 0 gives I, roulette step k
// reads block 1 + k/4, word k%4.  The 32 lanes compute the 8 blocks of 4
// (stratum, sample) pairs at once.  The roulette decision is taken in fp32
// on squared distances with every operation rounded as written (no
// contraction), so it depends only on the inputs and the tree.
#include <climits>

#include "bh_internal.h"

namespace bh {
namespace {

constexpr int kSbhThreads = 256;
constexpr int kRngBlocks = 8;                       // Philox blocks per path
constexpr int kMaxSteps = 4 * (kRngBlocks - 1);     // 28 >= 22 steps of any path
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void set_err(DevCtrl *c, unsigned code) {
  atomicCAS(&c->keep.err, 0u, code);
}

// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC 2011).
__device__ __forceinline__ void philox4x64_10(unsigned long long c0,
                                              unsigned long long c1,
                                              unsigned long long c2,
                                              unsigned long long c3,
                                              unsigned long long k0,
                                              unsigned long long k1,
                                              unsigned long long o[4]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const unsigned long long h0 = __umul64hi(0xD2E7470EE14C6C93ull, c0);
    const unsigned long long l0 = 0xD2E7470EE14C6C93ull * c0;
    const unsigned long long h1 = __umul64hi(0xCA5A826395121157ull, c2);
    const unsigned long long l1 = 0xCA5A826395121157ull * c2;
    c0 = h1 ^ c1 ^ k0;
    c1 = l1;
    c2 = h0 ^ c3 ^ k1;
    c3 = l0;
    k0 += 0x9E3779B97F4A7C15ull;
    k1 += 0xBB67AE8584CAA73Bull;
  }
  o[0] = c0; o[1] = c1; o[2] = c2; o[3] = c3;
}

// |q - p|^2, each operation rounded to fp32 in this order.
__device__ __forceinline__ float dist2_rn(const float4 &q, float px, float py, float pz) {
  const float dx = __fsub_rn(q.x, px), dy = __fsub_rn(q.y, py),
              dz = __fsub_rn(q.z, pz);
  const float d2 = __fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy));
  return __fadd_rn(d2, __fmul_rn(dz, dz));
}

// The roulette.  The continue probability min(1, max(1, beta_T) / beta_c),
// beta = r / w, with the child's edge w_T / 2, is min(1, max(w_T, r_T) /
// (2 r_c)); the draw u survives iff (4 (u u)) r_c^2 < max(w_T w_T, r_T^2),
// every operation rounded to fp32 as written.
__device__ __forceinline__ bool survives(float u, float wT, float dT2, float dc2) {
  const float lhs = __fmul_rn(__fmul_rn(4.f, __fmul_rn(u, u)), dc2);
  const float rhs = fmaxf(__fmul_rn(wT, wT), dT2);
  return lhs < rhs;
}

// Its probability, for the path weight only.
__device__ __forceinline__ float survival_prob(float wT, float dT2, float dc2) {
  if (!(dc2 > 0.f)) return 1.f;
  const float p = sqrtf(fmaxf(wT * wT, dT2) / (4.f * dc2));
  return p < 1.f ? p : 1.f;
}

// w = L * 2^-level, exact for the levels of a 21-bit tree.
__device__ __forceinline__ float edge(float L, int level) {
  return L * __int_as_float((127 - level) << 23);
}

// One softened monopole term of mass m at s on query q: (a, phi) / G.
__device__ __forceinline__ float4 mono(const float4 &q, float sx, float sy,
                                       float sz, float m, float eps2) {
  const float dx = sx - q.x, dy = sy - q.y, dz = sz - q.z;
  const float r2 = fmaf(dx, dx, fmaf(dy, dy, fmaf(dz, dz, eps2)));
  const float inv = r2 > 0.f ? rsqrt_ftz(r2) : 0.f;
  const float mi = m * inv;
  const float mi3 = mi * inv * inv;
  return make_float4(mi3 * dx, mi3 * dy, mi3 * dz, -mi);
}

__device__ __forceinline__ void axpy(float4 &acc, float w, const float4 &t) {
  acc.x = fmaf(w, t.x, acc.x);
  acc.y = fmaf(w, t.y, acc.y);
  acc.z = fmaf(w, t.z, acc.z);
  acc.w = fmaf(w, t.w, acc.w);
}

// Strata: nodes at level s and leaves above it, in node order.  Levels
// ascend along the breadth-first node array, so they all lie in the first
// sum_{l <= s} level_total[l] nodes.  One block, ordered compaction.
__global__ void __launch_bounds__(1024) strata_kernel(const NodeRec *__restrict__ rec,
                                                      long long nodes_cap, int s, int cap,
                                                      int *strata, DevCtrl *ctrl) {
  __shared__ unsigned warp_cnt[32];
  __shared__ int base_s;
  long long prefix = 0;
  for (int l = 0; l <= s && l < kMaxLevels; ++l) prefix += ctrl->step.level_total[l];
  if (prefix > nodes_cap) prefix = nodes_cap;       // never read past the pool
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) base_s = 0;
  __syncthreads();
  for (long long c0 = 0; c0 < prefix; c0 += blockDim.x) {
    const long long c = c0 + threadIdx.x;
    bool take = false;
    if (c < prefix) {
      const int fl = rec[c].flags;
      const int lv = (fl >> 8) & 255;
      take = lv == s || (lv < s && (fl & 1));
    }
    const unsigned bal = __ballot_sync(kFull, take);
    if (lane == 0) warp_cnt[w] = __popc(bal);
    __syncthreads();
    int off = base_s;
    for (int k = 0; k < w; ++k) off += warp_cnt[k];
    const int pos = off + __popc(bal & ((1u << lane) - 1u));
    if (take) {
      if (pos < cap) strata[pos] = (int)c;
      else set_err(ctrl, kErrOverflow);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int k = 0; k < (int)(blockDim.x >> 5); ++k) tot += warp_cnt[k];
      base_s += tot;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) ctrl->step.strata = base_s < cap ? base_s : cap;
}

// Per-warp staging in shared memory: the Philox blocks of a batch of four
// (stratum, sample) pairs (lane 8j + b holds block b of pair j), the four
// strata, and eight child slots per pair (the stratum's children, then the
// children of the current cell on its path).  Reads are warp-uniform
// broadcasts.
struct SbhWarp {
  unsigned long long rng[32][4];
  NodeRec strat[4];
  int2 srange[4];            // (first, end) particles of each stratum
  NodeRec child[32];
  int2 crange[32];           // (first, end) particles of each child
};

template <bool kSelf>
__global__ void __launch_bounds__(kSbhThreads) sbh_kernel(SbhArgs a, DevCtrl *ctrl) {
  __shared__ SbhWarp smem[kSbhThreads / 32];
  SbhWarp &W = smem[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;
  const float L = ctrl->keep.cube[0].w;
  const long long ns = ctrl->step.strata;
  const long long S = a.samples;
  const long long npairs = ns * S;
  const long long gend = a.g_end;       // groups [g_begin, g_end) of this call
  const float inv_s = 1.f / (float)S;
  unsigned long long useful = 0, groups = 0;
  for (;;) {
    unsigned g = 0;
    if (lane == 0) g = atomicAdd(&ctrl->step.work_ctr, 1u);
    g = __shfl_sync(kFull, g, 0) + (unsigned)a.g_begin;
    if ((long long)g >= gend) break;
    ++groups;
    const long long qi = (long long)g * 32 + lane;
    const bool valid = qi < a.m;
    const float4 q = a.tpos[valid ? qi : a.m - 1];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    unsigned nterm = 0;
    for (long long t0 = 0; t0 < npairs; t0 += 4) {
      {
        // lane 8j + b: Philox block b of pair t0 + j, and child b of that
        // pair's stratum (so the first step of all four paths is loaded)
        const long long tl = t0 + (lane >> 3);
        const int b = lane & 7;
        const bool pair_ok = tl < npairs;
        const long long rl = pair_ok ? tl / S : 0;
        unsigned long long o[4];
        philox4x64_10((unsigned long long)g, (unsigned long long)rl,
                      (unsigned long long)(tl - rl * S), (unsigned long long)b,
                      a.seed, 0ull, o);
        W.rng[lane][0] = o[0]; W.rng[lane][1] = o[1];
        W.rng[lane][2] = o[2]; W.rng[lane][3] = o[3];
        const int Rl = a.strata[rl];
        const NodeRec srec = a.rec[Rl];
        const int4 stop = a.topo[Rl];
        if (b == 0) {
          W.strat[lane >> 3] = srec;
          W.srange[lane >> 3] = make_int2(stop.x, stop.y);
        }
        const int snc = (srec.flags & 1) ? 0 : (srec.count < 8 ? srec.count : 8);
        if (pair_ok && b < snc && srec.link >= 0 && (long long)srec.link + b < a.nodes) {
          W.child[lane] = a.rec[srec.link + b];
          const int4 ct = a.topo[srec.link + b];
          W.crange[lane] = make_int2(ct.x, ct.y);
        }
        __syncwarp();
      }
      const int jn = npairs - t0 < 4 ? (int)(npairs - t0) : 4;
      for (int j = 0; j < jn; ++j) {
        const long long smp = (t0 + j) % S;
        const int cb = 8 * j;
        const NodeRec recR = W.strat[j];
        const int2 rngR = W.srange[j];
        const long long nR = (long long)rngR.y - rngR.x;
        float4 fpar = mono(q, recR.com.x, recR.com.y, recR.com.z, recR.com.w, a.eps2);
        if (smp == 0) {                      // the stratum's monopole, once
          axpy(acc, 1.f, fpar);
          nterm += 1;
        }
        long long J = rngR.x + (long long)__umul64hi(W.rng[cb][0], (unsigned long long)nR);
        if (J < 0 || J >= a.n) J = 0;         // only a corrupt tree gets here
        // the current cell T, warp-uniform
        float4 tcom = recR.com;
        int tlink = recR.link, tcount = recR.count, tflags = recR.flags;
        long long nT = nR;
        float P = 1.f;
        bool active = valid;
        for (int k = 0; k < kMaxSteps; ++k) {
          const bool leaf = tflags & 1;
          const int lv = (tflags >> 8) & 255;
          const float wT = edge(L, lv);
          const int nc = leaf ? 0 : (tcount < 8 ? tcount : 8);
          int ci = 0;
          float cx, cy, cz;
          if (leaf) {
            const float4 pj = a.spm[J];
            cx = pj.x; cy = pj.y; cz = pj.z;
          } else {
            const bool ok = tlink >= 0 && (long long)tlink + nc <= a.nodes;
            if (k > 0) {                      // T's children into the slots
              if (lane < nc && ok) {
                W.child[cb + lane] = a.rec[tlink + lane];
                const int4 ct = a.topo[tlink + lane];
                W.crange[cb + lane] = make_int2(ct.x, ct.y);
              }
              __syncwarp();
            }
            // the path child: the last child whose first particle is <= J
            const unsigned bal = __ballot_sync(
                kFull, ok && lane < nc && (long long)W.crange[cb + lane].x <= J);
            if (bal == 0u) break;             // only a corrupt tree gets here
            ci = 31 - __clz(bal);
            const float4 cc = W.child[cb + ci].com;
            cx = cc.x; cy = cc.y; cz = cc.z;
          }
          const float dT2 = dist2_rn(q, tcom.x, tcom.y, tcom.z);
          const float dc2 = dist2_rn(q, cx, cy, cz);
          const float u = __ull2float_rn(W.rng[cb + 1 + (k >> 2)][k & 3] >> 40) * 0x1p-24f;
          const bool go = active && survives(u, wT, dT2, dc2);
          if (!__any_sync(kFull, go)) break;
          if (go) P *= survival_prob(wT, dT2, dc2);
          const float wgt = go ? __fdividef((float)nR * inv_s, (float)nT * P) : 0.f;
          float4 fnext = make_float4(0.f, 0.f, 0.f, 0.f);
          if (leaf) {
            // a leaf at the deepest level may hold any number of particles
            const long long j0 = tlink < 0 ? 0 : tlink;
            long long j1 = j0 + (tcount < 0 ? 0 : tcount);
            if (j1 > a.n) j1 = a.n;
            for (long long jj = j0; jj < j1; ++jj) {
              const float4 pj = a.spm[jj];
              if (kSelf && jj == qi) continue;
              axpy(acc, wgt, mono(q, pj.x, pj.y, pj.z, pj.w, a.eps2));
              nterm += go;
            }
          } else {
            for (int c = 0; c < nc; ++c) {
              const float4 cc = W.child[cb + c].com;
              const float4 tc = mono(q, cc.x, cc.y, cc.z, cc.w, a.eps2);
              axpy(acc, wgt, tc);
              if (c == ci) fnext = tc;
            }
            nterm += go ? (unsigned)nc : 0u;
          }
          axpy(acc, -wgt, fpar);
          nterm += go;
          active = go;
          if (leaf) break;
          const NodeRec nx = W.child[cb + ci];
          const int2 nr = W.crange[cb + ci];
          tcom = nx.com;
          tlink = nx.link;
          tcount = nx.count;
          tflags = nx.flags;
          nT = (long long)nr.y - nr.x;
          fpar = fnext;
          __syncwarp();                       // slots read before reuse
        }
      }
      __syncwarp();                           // batch data read before reuse
    }
    if (valid) {
      float4 res;
      res.x = a.G * acc.x; res.y = a.G * acc.y; res.z = a.G * acc.z; res.w = a.G * acc.w;
      const unsigned dst = a.tperm[qi];
      if (dst < a.m) a.out[dst] = res;
      useful += nterm;
    }
  }
  for (int o = 16; o > 0; o >>= 1) useful += __shfl_xor_sync(kFull, useful, o);
  if (lane == 0) {
    if (useful) atomicAdd(&ctrl->step.executed, useful);
    if (groups) atomicAdd(&ctrl->step.groups, groups);
  }
}

}  // namespace

cudaError_t launch_sbh(const SbhArgs &a, int *strata, int strata_cap,
                       DevCtrl *ctrl, cudaStream_t s) {
  if (a.m <= 0) return cudaSuccess;
  strata_kernel<<<1, 1024, 0, s>>>(a.rec, a.nodes, a.strata_level, strata_cap, strata, ctrl);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  static std::atomic<int> memo[2][kMaxDevices];
  const bool self = a.self_mode != 0;
  const int per_sm = per_device(memo[self ? 1 : 0], [self] {
    int b = 0;
    if (self)
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, sbh_kernel<true>, kSbhThreads, 0);
    else
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, sbh_kernel<false>, kSbhThreads, 0);
    return b > 0 ? b : 1;
  });
  const long long ngroups = a.g_end - a.g_begin;
  long long blocks = (long long)a.num_sms * per_sm;
  const long long need = (ngroups + kSbhThreads / 32 - 1) / (kSbhThreads / 32);
  if (blocks > need) blocks = need;
  if (blocks < 1) blocks = 1;
  if (a.self_mode)
    sbh_kernel<true><<<(unsigned)blocks, kSbhThreads, 0, s>>>(a, ctrl);
  else
    sbh_kernel<false><<<(unsigned)blocks, kSbhThreads, 0, s>>>(a, ctrl);
  return cudaGetLastError();
}

}  // namespace bh
