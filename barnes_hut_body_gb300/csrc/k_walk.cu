// Warp-cooperative Barnes-Hut walk.
//
// The GASPHiA tree-code page (section "性能瓶颈分析") walks the tree per
// particle and lets a warp skip a cell only when the opening test
// w_sq/theta_sq < r_sq holds for all 32 lanes (__all_sync); if any lane
// fails, the whole warp descends.  Its section "排序算法" shows that the walk
// only pays off when the 32 particles of a warp are close in space, which
// the Morton sort guarantees here.
//
// GB300 design, one warp per group of 32*T consecutive targets in Morton
// order (T targets per lane):
//  * Lane-parallel over nodes.  A shared-memory stack holds child ranges
//    (first child, count <= 8).  Each round the warp pops ranges until it has
//    up to 32 candidate nodes, one per lane, and loads their 32-byte records
//    (children are contiguous, so a range is one coalesced read).
//  * Opening decision.  Every lane first tests its node against the group's
//    bounding box: if w^2/theta^2 < d^2 with d the distance from the centre
//    of mass to the box, the test holds for every target, so the node is
//    accepted.  In BH_OPEN_VOTE mode the undecided nodes are then resolved
//    one by one with the page's rule: each lane evaluates its own targets
//    and the warp accepts only if all of them pass (__all_sync).  BH_OPEN_BOX
//    keeps the box answer.
//  * Accepted nodes (centre of mass + mass) and the particles of opened
//    leaves are appended to a per-warp interaction list in shared memory;
//    opened internal nodes push their child range.  Whenever 64 entries are
//    waiting, the warp evaluates them for all its targets: each entry is one
//    broadcast shared-memory read followed by 3 sub, 3 FMA, 1 rsqrt, 3 mul,
//    3 FMA and 1 add per target -- no divergence, no per-lane branching.
//  * Self mode: a target's own particle, when it comes through an opened
//    leaf, adds exactly m*rsqrt(eps^2) to its potential and nothing to its
//    acceleration; the walk records which targets saw their own particle and
//    removes that term at the end (with eps = 0 a zero-distance pair is
//    skipped in the inner loop instead).
//  * Persistent grid (SM count x resident blocks); warps take groups from an
//    atomic ticket so dense regions do not leave SMs idle.
#include <cuda_runtime.h>
#include <stdint.h>

#include "bh_internal.h"

namespace bh {

namespace {

constexpr int kWalkWarps = 8;
constexpr int kWalkThreads = kWalkWarps * 32;
constexpr int kStackCap = 736;   // >= 28 * 22 + 32: pops >= 1 range of <= 8
                                 // per round, pushes <= 32, depth <= 22
constexpr int kListCap = 96;
constexpr int kFlushAt = 64;

struct WarpSmem {
  float4 list[kListCap];
  unsigned int stack[kStackCap];
};

__device__ __forceinline__ void set_err(DevCtrl *c, unsigned code) {
  atomicCAS(&c->keep.err, 0u, code);
}

template <int T, bool kEps0>
__device__ __forceinline__ void interact(const float4 e, const float (&px)[T],
                                         const float (&py)[T],
                                         const float (&pz)[T], float eps2,
                                         float (&ax)[T], float (&ay)[T],
                                         float (&az)[T], float (&ph)[T]) {
#pragma unroll
  for (int k = 0; k < T; ++k) {
    float dx = e.x - px[k];
    float dy = e.y - py[k];
    float dz = e.z - pz[k];
    float r2 = fmaf(dx, dx, fmaf(dy, dy, fmaf(dz, dz, eps2)));
    float inv = rsqrtf(r2);
    if (kEps0) inv = (r2 > 0.f) ? inv : 0.f;
    float minv = e.w * inv;
    float minv3 = minv * (inv * inv);
    ax[k] = fmaf(dx, minv3, ax[k]);
    ay[k] = fmaf(dy, minv3, ay[k]);
    az[k] = fmaf(dz, minv3, az[k]);
    ph[k] -= minv;
  }
}

template <int T, bool kEps0>
__device__ __forceinline__ void flush_full(const float4 *list,
                                           const float (&px)[T],
                                           const float (&py)[T],
                                           const float (&pz)[T], float eps2,
                                           float (&ax)[T], float (&ay)[T],
                                           float (&az)[T], float (&ph)[T]) {
#pragma unroll 8
  for (int j = 0; j < kFlushAt; ++j)
    interact<T, kEps0>(list[j], px, py, pz, eps2, ax, ay, az, ph);
}

template <int T, bool kEps0>
__device__ __forceinline__ void flush_part(const float4 *list, int cnt,
                                           const float (&px)[T],
                                           const float (&py)[T],
                                           const float (&pz)[T], float eps2,
                                           float (&ax)[T], float (&ay)[T],
                                           float (&az)[T], float (&ph)[T]) {
#pragma unroll 4
  for (int j = 0; j < cnt; ++j)
    interact<T, kEps0>(list[j], px, py, pz, eps2, ax, ay, az, ph);
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

template <int T, bool kVote, bool kEps0, bool kSelf>
__global__ void __launch_bounds__(kWalkThreads, 2)
walk_kernel(WalkArgs a, DevCtrl *ctrl) {
  __shared__ WarpSmem smem[kWalkWarps];
  const int lane = threadIdx.x & 31;
  WarpSmem &S = smem[threadIdx.x >> 5];
  const unsigned lt = (1u << lane) - 1u;
  constexpr int GS = 32 * T;
  const long long ngroups = (a.m + GS - 1) / GS;
  unsigned long long executed = 0, ngroup_done = 0;
  long long nnodes = 0;
  for (int l = 0; l < kMaxLevels; ++l) nnodes += ctrl->step.level_total[l];

  for (;;) {
    unsigned long long g = 0;
    if (lane == 0) g = atomicAdd(&ctrl->step.work_ctr, 1u);
    g = __shfl_sync(0xffffffffu, g, 0);
    if ((long long)g >= ngroups) break;
    const long long t0 = (long long)g * GS;
    const int nvalid = (int)((a.m - t0) < GS ? (a.m - t0) : GS);

    float px[T], py[T], pz[T], ax[T], ay[T], az[T], ph[T];
    bool valid[T], selfhit[T];
    float bl0 = INFINITY, bl1 = INFINITY, bl2 = INFINITY;
    float bh0 = -INFINITY, bh1 = -INFINITY, bh2 = -INFINITY;
#pragma unroll
    for (int k = 0; k < T; ++k) {
      const long long t = t0 + k * 32 + lane;
      valid[k] = t < a.m;
      float4 p = __ldg(a.tpos + (valid[k] ? t : t0));
      px[k] = p.x; py[k] = p.y; pz[k] = p.z;
      ax[k] = ay[k] = az[k] = ph[k] = 0.f;
      selfhit[k] = false;
      bl0 = fminf(bl0, p.x); bh0 = fmaxf(bh0, p.x);
      bl1 = fminf(bl1, p.y); bh1 = fmaxf(bh1, p.y);
      bl2 = fminf(bl2, p.z); bh2 = fmaxf(bh2, p.z);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      bl0 = fminf(bl0, __shfl_xor_sync(0xffffffffu, bl0, o));
      bl1 = fminf(bl1, __shfl_xor_sync(0xffffffffu, bl1, o));
      bl2 = fminf(bl2, __shfl_xor_sync(0xffffffffu, bl2, o));
      bh0 = fmaxf(bh0, __shfl_xor_sync(0xffffffffu, bh0, o));
      bh1 = fmaxf(bh1, __shfl_xor_sync(0xffffffffu, bh1, o));
      bh2 = fmaxf(bh2, __shfl_xor_sync(0xffffffffu, bh2, o));
    }

    int sp = 1;                     // stack: the root as a range of one
    if (lane == 0) S.stack[0] = 0u;
    int nl = 0;                     // entries waiting in the list
    __syncwarp();

    while (sp > 0) {
      // ---- pop ranges until up to 32 nodes ----------------------------
      unsigned ent = 0;
      int cnt = 0;
      if (lane < sp) {
        ent = S.stack[sp - 1 - lane];
        cnt = (int)(ent & 7u) + 1;
      }
      const int pre = warp_incl_scan(cnt, lane);
      const bool take = lane < sp && pre <= 32;
      const unsigned tmask = __ballot_sync(0xffffffffu, take);
      const int ntake = __popc(tmask);
      const int total = __shfl_sync(0xffffffffu, pre, ntake - 1);
      sp -= ntake;
      const int excl = pre - cnt;
      const unsigned starts =
          __reduce_or_sync(0xffffffffu, take ? (1u << excl) : 0u);
      bool has = lane < total;
      int e = __popc(starts & ((2u << lane) - 1u)) - 1;
      e = e < 0 ? 0 : e;
      const unsigned ebase = __shfl_sync(0xffffffffu, ent >> 3, e);
      const int eexcl = __shfl_sync(0xffffffffu, excl, e);
      const unsigned node = ebase + (unsigned)(lane - eexcl);
      __syncwarp();

      // ---- load the candidate's record and test it ---------------------
      float4 c4 = make_float4(0.f, 0.f, 0.f, 0.f);
      float ro2 = 0.f;
      int link = 0, count = 0, flags = 0;
      bool acc = false;
      if (has && node >= nnodes) {     // only after a failed earlier stage
        has = false;
        set_err(ctrl, kErrOverflow);
      }
      if (has) {
        const float4 *r = reinterpret_cast<const float4 *>(a.rec + node);
        c4 = __ldg(r);
        float4 q = __ldg(r + 1);
        ro2 = q.x;
        link = __float_as_int(q.y);
        count = __float_as_int(q.z);
        flags = __float_as_int(q.w);
        float dx = fmaxf(fmaxf(bl0 - c4.x, c4.x - bh0), 0.f);
        float dy = fmaxf(fmaxf(bl1 - c4.y, c4.y - bh1), 0.f);
        float dz = fmaxf(fmaxf(bl2 - c4.z, c4.z - bh2), 0.f);
        acc = ro2 < fmaf(dx, dx, fmaf(dy, dy, dz * dz));
      }
      if (kVote) {
        unsigned cand = __ballot_sync(0xffffffffu, has && !acc);
        unsigned accm = 0;
        while (cand) {
          const int c = __ffs(cand) - 1;
          cand &= cand - 1u;
          const float cx = __shfl_sync(0xffffffffu, c4.x, c);
          const float cy = __shfl_sync(0xffffffffu, c4.y, c);
          const float cz = __shfl_sync(0xffffffffu, c4.z, c);
          const float r2o = __shfl_sync(0xffffffffu, ro2, c);
          bool ok = true;
#pragma unroll
          for (int k = 0; k < T; ++k) {
            float dx = cx - px[k], dy = cy - py[k], dz = cz - pz[k];
            float r2 = fmaf(dx, dx, fmaf(dy, dy, dz * dz));
            ok = ok && (!valid[k] || r2o < r2);
          }
          if (__all_sync(0xffffffffu, ok)) accm |= 1u << c;
        }
        acc = acc || ((accm >> lane) & 1u);
      }
      const bool leaf = (flags & 1) != 0;
      // Children always sit at larger indices (breadth-first order), so
      // pushing only forward links bounds every path, even over a tree left
      // inconsistent by a failed earlier stage.
      const bool open_int = has && !acc && !leaf && count >= 1 && count <= 8 &&
                            (unsigned)link > node &&
                            (long long)link + count <= nnodes;
      const bool open_leaf = has && !acc && leaf && link >= 0 && link <= a.n;
      if (open_leaf && count > a.n - link) count = (int)(a.n - link);

      // ---- accepted nodes -> interaction list ---------------------------
      const unsigned am = __ballot_sync(0xffffffffu, has && acc);
      if (has && acc) S.list[nl + __popc(am & lt)] = c4;
      nl += __popc(am);

      // ---- opened internal nodes -> stack -------------------------------
      const unsigned om = __ballot_sync(0xffffffffu, open_int);
      const int npush = __popc(om);
      if (sp + npush <= kStackCap) {
        if (open_int)
          S.stack[sp + __popc(om & lt)] =
              ((unsigned)link << 3) | (unsigned)(count - 1);
        sp += npush;
      } else if (npush) {
        if (lane == 0) set_err(ctrl, kErrOverflow);
      }
      __syncwarp();
      if (nl >= kFlushAt) {
        flush_full<T, kEps0>(S.list, px, py, pz, a.eps2, ax, ay, az, ph);
        executed += (unsigned long long)kFlushAt * nvalid;
        nl -= kFlushAt;
        __syncwarp();
        if (lane < nl) S.list[lane] = S.list[kFlushAt + lane];
        __syncwarp();
      }

      // ---- opened leaves -> their particles -----------------------------
      const unsigned lm = __ballot_sync(0xffffffffu, open_leaf);
      if (lm) {
        const int pc = open_leaf ? (count > 0 ? count : 0) : 0;
        const int ppre = warp_incl_scan(pc, lane);
        const int ptotal = __shfl_sync(0xffffffffu, ppre, 31);
        const int pexcl = ppre - pc;
        if (kSelf) {
          // which targets of the group see their own particle
          unsigned long long msk = 0ull;
          if (open_leaf && pc > 0) {
            long long lo = (long long)link - t0, hi = lo + pc;
            if (lo < 0) lo = 0;
            if (hi > GS) hi = GS;
            if (lo < hi) {
              unsigned long long upper =
                  (hi >= 64) ? ~0ull : ((1ull << hi) - 1ull);
              msk = upper & ~((1ull << lo) - 1ull);
            }
          }
          const unsigned m0 = __reduce_or_sync(0xffffffffu, (unsigned)msk);
          const unsigned m1 =
              __reduce_or_sync(0xffffffffu, (unsigned)(msk >> 32));
#pragma unroll
          for (int k = 0; k < T; ++k)
            selfhit[k] = selfhit[k] || (((k == 0 ? m0 : m1) >> lane) & 1u);
        }
        for (int base = 0; base < ptotal; base += 32) {
          const int q = base + lane;
          int lo = 0;
#pragma unroll
          for (int s = 16; s >= 1; s >>= 1) {
            int v = __shfl_sync(0xffffffffu, ppre, lo + s - 1);
            if (v <= q) lo += s;
          }
          const int owner = lo > 31 ? 31 : lo;
          const int of = __shfl_sync(0xffffffffu, link, owner);
          const int oe = __shfl_sync(0xffffffffu, pexcl, owner);
          if (q < ptotal) S.list[nl + lane] = __ldg(a.spm + of + (q - oe));
          nl += (ptotal - base < 32) ? (ptotal - base) : 32;
          __syncwarp();
          if (nl >= kFlushAt) {
            flush_full<T, kEps0>(S.list, px, py, pz, a.eps2, ax, ay, az, ph);
            executed += (unsigned long long)kFlushAt * nvalid;
            nl -= kFlushAt;
            __syncwarp();
            if (lane < nl) S.list[lane] = S.list[kFlushAt + lane];
            __syncwarp();
          }
        }
      }
    }
    if (nl > 0) {
      flush_part<T, kEps0>(S.list, nl, px, py, pz, a.eps2, ax, ay, az, ph);
      executed += (unsigned long long)nl * nvalid;
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < T; ++k) {
      if (!valid[k]) continue;
      const long long t = t0 + k * 32 + lane;
      if (kSelf && !kEps0 && selfhit[k]) {
        // undo the self pair: it added m * rsqrt(eps^2) to -phi
        const float m_self = __ldg(a.tpos + t).w;
        ph[k] += m_self * rsqrtf(a.eps2);
      }
      const unsigned ci = a.tperm ? a.tperm[t] : (unsigned)t;
      if (ci < (unsigned long long)a.m)
        a.out[ci] = make_float4(a.G * ax[k], a.G * ay[k], a.G * az[k], a.G * ph[k]);
    }
    ++ngroup_done;
  }
  if (lane == 0) {
    atomicAdd(&ctrl->step.executed, executed);
    atomicAdd(&ctrl->step.groups, ngroup_done);
  }
}


// Per-target interaction count: the number of terms a walk that decides the
// opening test per target (no group vote) evaluates -- accepted cells plus
// particle pairs of opened leaves, the own pair excluded.  One thread per
// target, depth-first with a private stack; used to report useful work.
constexpr int kCountStack = 8 * kMaxLevels + 8;

__global__ void __launch_bounds__(256)
count_kernel(const NodeRec *__restrict__ rec, const float4 *__restrict__ tpos,
             const unsigned int *__restrict__ tperm, long long m, long long n,
             int self_mode, unsigned int *counts, DevCtrl *ctrl) {
  long long nnodes = 0;
  for (int l = 0; l < kMaxLevels; ++l) nnodes += ctrl->step.level_total[l];
  unsigned long long local = 0;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < m;
       t += stride) {
    const float4 p = __ldg(tpos + t);
    unsigned stack[kCountStack];
    int sp = 0;
    stack[sp++] = 0;
    unsigned long long terms = 0;
    while (sp > 0) {
      const unsigned c = stack[--sp];
      if (c >= nnodes) continue;
      const float4 *r = reinterpret_cast<const float4 *>(rec + c);
      const float4 cm = __ldg(r);
      const float4 q = __ldg(r + 1);
      const int link = __float_as_int(q.y), count = __float_as_int(q.z);
      const bool leaf = (__float_as_int(q.w) & 1) != 0;
      const float dx = cm.x - p.x, dy = cm.y - p.y, dz = cm.z - p.z;
      if (q.x < fmaf(dx, dx, fmaf(dy, dy, dz * dz))) {
        ++terms;
      } else if (leaf) {
        long long cnt = count < 0 ? 0 : count;
        if (self_mode && t >= link && t < link + cnt) --cnt;
        terms += (unsigned long long)cnt;
      } else if (count >= 1 && count <= 8 && (unsigned)link > c &&
                 sp + count <= kCountStack) {
        for (int k = count - 1; k >= 0; --k) stack[sp++] = (unsigned)link + k;
      } else if (count >= 1) {
        set_err(ctrl, kErrOverflow);
      }
    }
    local += terms;
    if (counts) {
      const unsigned ci = tperm ? tperm[t] : (unsigned)t;
      if (ci < (unsigned long long)m) counts[ci] = (unsigned)terms;
    }
  }
  for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
  if ((threadIdx.x & 31) == 0) atomicAdd(&ctrl->step.useful, local);
}

template <int T, bool kVote, bool kEps0, bool kSelf>
cudaError_t launch_one(const WalkArgs &a, DevCtrl *ctrl, cudaStream_t s) {
  static int per_sm = 0;
  if (per_sm == 0) {
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, walk_kernel<T, kVote, kEps0, kSelf>, kWalkThreads, 0);
    if (per_sm < 1) per_sm = 1;
  }
  const long long ngroups = (a.m + 32 * T - 1) / (32 * T);
  long long blocks = (long long)a.num_sms * per_sm;
  long long need = (ngroups + kWalkWarps - 1) / kWalkWarps;
  if (blocks > need) blocks = need;
  if (blocks < 1) blocks = 1;
  walk_kernel<T, kVote, kEps0, kSelf><<<(unsigned)blocks, kWalkThreads, 0, s>>>(a, ctrl);
  return cudaGetLastError();
}

template <int T>
cudaError_t launch_t(const WalkArgs &a, DevCtrl *ctrl, cudaStream_t s) {
  const bool vote = a.opening == BH_OPEN_VOTE;
  const bool eps0 = a.eps2 == 0.f;
  const bool self = a.self_mode != 0;
  if (vote) {
    if (eps0) return self ? launch_one<T, true, true, true>(a, ctrl, s)
                          : launch_one<T, true, true, false>(a, ctrl, s);
    return self ? launch_one<T, true, false, true>(a, ctrl, s)
                : launch_one<T, true, false, false>(a, ctrl, s);
  }
  if (eps0) return self ? launch_one<T, false, true, true>(a, ctrl, s)
                        : launch_one<T, false, true, false>(a, ctrl, s);
  return self ? launch_one<T, false, false, true>(a, ctrl, s)
              : launch_one<T, false, false, false>(a, ctrl, s);
}

}  // namespace

cudaError_t launch_count(const WalkArgs &a, unsigned int *counts, DevCtrl *ctrl,
                         cudaStream_t s) {
  if (a.m <= 0) return cudaSuccess;
  long long blocks = (a.m + 255) / 256;
  if (blocks > (long long)a.num_sms * 16) blocks = (long long)a.num_sms * 16;
  cudaMemsetAsync(&ctrl->step.useful, 0, sizeof(unsigned long long), s);
  count_kernel<<<(unsigned)blocks, 256, 0, s>>>(a.rec, a.tpos, a.tperm, a.m, a.n,
                                                 a.self_mode, counts, ctrl);
  return cudaGetLastError();
}

cudaError_t launch_walk(const WalkArgs &a, DevCtrl *ctrl, cudaStream_t s) {
  if (a.m <= 0) return cudaSuccess;
  return a.group == 32 ? launch_t<1>(a, ctrl, s) : launch_t<2>(a, ctrl, s);
}

}  // namespace bh
