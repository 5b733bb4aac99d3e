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
//    up to 32 candidate nodes, one per lane, and stages their 32-byte
//    records in shared memory with one TMA bulk copy (cp.async.bulk) per
//    range -- children are contiguous records -- completing on a per-warp
//    mbarrier; the wait is bounded.
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
//    waiting, the warp evaluates them (while the round's record copies are
//    in flight) for all its targets with Blackwell's
//    packed fp32x2 instructions: two entries per 64-bit operand, so a pair of
//    entries costs two broadcast shared-memory reads and, per target, 13
//    packed ops (3 sub, 3 fma, 3 mul, 3 fma, 1 sub) plus 2 rsqrt -- no
//    divergence, no per-lane branching.
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
constexpr int kListCap = 96;    // entries; stored as pairs (see below)
constexpr int kFlushAt = 64;
constexpr int kProbesPerSlot = 4;   // probe targets per 32-target slot

// The interaction list holds entries (x, y, z, m) two by two, each pair as
// two 16-byte words: (x_j, x_j+1, y_j, y_j+1) and (z_j, z_j+1, m_j, m_j+1).
// One broadcast 16-byte shared load then yields two packed fp32x2 operands.
struct alignas(128) WarpSmem {
  float4 rec[32][2];                  // the round's node records (TMA target)
  ulonglong2 list[kListCap / 2][2];
  float4 cand[32];                    // candidates put to the vote
  float4 probe[8];                    // probe targets of the group
  unsigned int stack[kStackCap];
  unsigned long long bar;             // completion of the record copies
};
constexpr unsigned kRecWaitLimit = 1u << 26;   // polls; a copy takes microseconds

__device__ __forceinline__ unsigned smem_addr(const void *p) {
  return (unsigned)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void set_err(DevCtrl *c, unsigned code) {
  atomicCAS(&c->keep.err, 0u, code);
}

// Append entry j (x, y, z, m) to the paired list.
__device__ __forceinline__ void list_put(WarpSmem &S, int j, float4 v) {
  float *w = reinterpret_cast<float *>(&S.list[j >> 1][0]);
  const int h = j & 1;
  w[h] = v.x;
  w[2 + h] = v.y;
  w[4 + h] = v.z;
  w[6 + h] = v.w;
}

// Whether all children of an opened node pass the box test: the node's box
// distance d2 against its opening radius times the factor the build stored
// in flags bits 16..31 (0 = never).
__device__ __forceinline__ bool children_accepted(float d2, float ro2, int flags) {
  const unsigned f = (unsigned)flags >> 16;
  return f != 0u && ro2 * __uint2float_rn(f) * (1.f / 65536.f) < d2;
}

// A list entry (x, y, z, m): particle j, or the centre of mass of node j.
__device__ __forceinline__ float4 entry_source(const WalkArgs &a, bool node, long long j) {
  return node ? __ldg(reinterpret_cast<const float4 *>(a.rec + j)) : __ldg(a.spm + j);
}

// Targets are held duplicated in both fp32 lanes (P = (p, p)); a pair of
// entries then gives two interactions per packed instruction.  Per pair and
// target: 3 sub, 3 fma, 2 rsqrt, 3 mul, 3 fma, 1 sub (13 packed + 2 MUFU).
template <int T, bool kEps0>
struct Acc {
  f2 px[T], py[T], pz[T];     // targets, duplicated in both lanes
  f2 ax[T], ay[T], az[T], ph[T];
  f2 eps2;

  __device__ __forceinline__ void pair(const ulonglong2 a, const ulonglong2 b) {
    // a = (xx, yy), b = (zz, mm)
#pragma unroll
    for (int k = 0; k < T; ++k) {
      f2 dx = sub2(a.x, px[k]);
      f2 dy = sub2(a.y, py[k]);
      f2 dz = sub2(b.x, pz[k]);
      f2 r2 = fma2(dx, dx, fma2(dy, dy, fma2(dz, dz, eps2)));
      float r0, r1;
      upk(r2, r0, r1);
      float i0 = rsqrt_ftz(r0), i1 = rsqrt_ftz(r1);
      if (kEps0) {
        i0 = (r0 > 0.f) ? i0 : 0.f;
        i1 = (r1 > 0.f) ? i1 : 0.f;
      }
      f2 inv = pk(i0, i1);
      f2 minv = mul2(b.y, inv);
      f2 minv3 = mul2(minv, mul2(inv, inv));
      ax[k] = fma2(dx, minv3, ax[k]);
      ay[k] = fma2(dy, minv3, ay[k]);
      az[k] = fma2(dz, minv3, az[k]);
      ph[k] = sub2(ph[k], minv);
    }
  }

  // Evaluate list pairs [0, npairs).
  __device__ __forceinline__ void run(const WarpSmem &S, int npairs) {
#pragma unroll 2
    for (int p = 0; p < npairs; ++p) pair(S.list[p][0], S.list[p][1]);
  }
  // unrolled 4 deep (2 with eps = 0, whose zero-distance guard would spill)
  __device__ __forceinline__ void run_full(const WarpSmem &S) {
    if constexpr (kEps0) {
#pragma unroll 2
      for (int p = 0; p < kFlushAt / 2; ++p) pair(S.list[p][0], S.list[p][1]);
    } else {
#pragma unroll 4
      for (int p = 0; p < kFlushAt / 2; ++p) pair(S.list[p][0], S.list[p][1]);
    }
  }
  // the same over a bare list of entry pairs
  __device__ __forceinline__ void run_list(const ulonglong2 (*list)[2], int npairs) {
#pragma unroll 2
    for (int p = 0; p < npairs; ++p) pair(list[p][0], list[p][1]);
  }
  // a full list of NPAIRS entry pairs
  template <int NPAIRS>
  __device__ __forceinline__ void run_full_list(const ulonglong2 (*list)[2]) {
#pragma unroll 4
    for (int p = 0; p < NPAIRS; ++p) pair(list[p][0], list[p][1]);
  }
};

// Evaluate the first kFlushAt list entries and move the rest to the front.
template <int T, bool kEps0>
__device__ __forceinline__ void flush_front(WarpSmem &S, Acc<T, kEps0> &accum,
                                            int &nl, int nvalid,
                                            unsigned long long &executed) {
  const int lane = threadIdx.x & 31;
  accum.run_full(S);
  executed += (unsigned long long)kFlushAt * nvalid;
  nl -= kFlushAt;
  __syncwarp();
  if (lane < (nl + 1) / 2) {
    S.list[lane][0] = S.list[kFlushAt / 2 + lane][0];
    S.list[lane][1] = S.list[kFlushAt / 2 + lane][1];
  }
  __syncwarp();
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
  const long long gend = a.g_end;       // groups [g_begin, g_end) of this call
  unsigned long long executed = 0, ngroup_done = 0;
  unsigned long long st_rounds = 0, st_tested = 0, st_voted = 0, st_chunks = 0;
  const long long nnodes = node_total(ctrl);
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&S.bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  unsigned rec_phase = 0;

  for (;;) {
    unsigned long long g = 0;
    if (lane == 0) g = atomicAdd(&ctrl->step.work_ctr, 1u);
    g = __shfl_sync(0xffffffffu, g, 0) + (unsigned long long)a.g_begin;
    if ((long long)g >= gend) break;
    if (a.gorder) {
      g = a.gorder[g];
      if ((long long)g >= gend) {        // not a permutation: skip, flag
        if (lane == 0) set_err(ctrl, kErrOverflow);
        continue;
      }
    }
    const unsigned long long exec0 = executed;
    const long long t0 = (long long)g * GS;
    const int nvalid = (int)((a.m - t0) < GS ? (a.m - t0) : GS);

    float px[T], py[T], pz[T];
    Acc<T, kEps0> accum;
    accum.eps2 = pk(a.eps2, a.eps2);
    bool valid[T], selfhit[T];
    float bl0 = INFINITY, bl1 = INFINITY, bl2 = INFINITY;
    float bh0 = -INFINITY, bh1 = -INFINITY, bh2 = -INFINITY;
#pragma unroll
    for (int k = 0; k < T; ++k) {
      const long long t = t0 + k * 32 + lane;
      valid[k] = t < a.m;
      float4 p = __ldg(a.tpos + (valid[k] ? t : t0));
      px[k] = p.x; py[k] = p.y; pz[k] = p.z;
      accum.px[k] = pk(p.x, p.x);
      accum.py[k] = pk(p.y, p.y);
      accum.pz[k] = pk(p.z, p.z);
      if ((lane & (32 / kProbesPerSlot - 1)) == 0)
        S.probe[k * kProbesPerSlot + lane / (32 / kProbesPerSlot)] = make_float4(p.x, p.y, p.z, 0.f);
      accum.ax[k] = accum.ay[k] = accum.az[k] = accum.ph[k] = 0ull;
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
      ++st_rounds;
      st_tested += (unsigned)total;

      // ---- stage the candidates' records with TMA bulk copies -------------
      // one copy per popped range (children are contiguous records); a
      // range outside the node pool only follows a failed earlier stage
      const unsigned rbase = ent >> 3;
      const bool rok = take && (long long)rbase + cnt <= nnodes;
      if (take && !rok) set_err(ctrl, kErrOverflow);
      const unsigned okm = __ballot_sync(0xffffffffu, rok);
      unsigned bytes = rok ? (unsigned)cnt * 32u : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
      // the previous round's generic reads of S.rec before the async writes
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     ::"r"(smem_addr(&S.bar)), "r"(bytes) : "memory");
      __syncwarp();
      if (rok)
        asm volatile(
            "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
            ::"r"(smem_addr(&S.rec[excl][0])), "l"(a.rec + rbase), "r"((unsigned)cnt * 32u),
              "r"(smem_addr(&S.bar)) : "memory");
      {   // lanes whose range was refused hold no node
        const int er = __shfl_sync(0xffffffffu, (int)rok, e);
        if (has && (!er || !((okm >> e) & 1u))) has = false;
      }
      // ---- evaluate a full list while the copies are in flight ------------
      if (nl >= kFlushAt) flush_front(S, accum, nl, nvalid, executed);
      {
        bool done = false;
        for (unsigned it = 0; it < kRecWaitLimit && !done; ++it) {
          unsigned ok;
          asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                       " selp.u32 %0, 1, 0, p;\n}\n"
                       : "=r"(ok) : "r"(smem_addr(&S.bar)), "r"(rec_phase) : "memory");
          done = ok != 0;
        }
        rec_phase ^= 1u;
        if (!__all_sync(0xffffffffu, done)) {
          // give up on this launch: flag it, let the copies land, leave
          if (lane == 0) set_err(ctrl, kErrTimeout);
          for (unsigned it = 0; it < kRecWaitLimit; ++it) {
            unsigned ok;
            asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                         " selp.u32 %0, 1, 0, p;\n}\n"
                         : "=r"(ok) : "r"(smem_addr(&S.bar)), "r"(rec_phase ^ 1u) : "memory");
            if (ok) break;
          }
          return;
        }
      }
      float4 c4 = make_float4(0.f, 0.f, 0.f, 0.f);
      float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
      if (has) {
        c4 = S.rec[lane][0];
        q = S.rec[lane][1];
      }

      // ---- opening test ---------------------------------------------------
      const float ro2 = q.x;
      const int link = __float_as_int(q.y);
      int count = __float_as_int(q.z);
      const int flags = __float_as_int(q.w);
      bool acc = false;
      float d2 = 0.f;
      if (has) {
        float dx = fmaxf(fmaxf(bl0 - c4.x, c4.x - bh0), 0.f);
        float dy = fmaxf(fmaxf(bl1 - c4.y, c4.y - bh1), 0.f);
        float dz = fmaxf(fmaxf(bl2 - c4.z, c4.z - bh2), 0.f);
        d2 = fmaf(dx, dx, fmaf(dy, dy, dz * dz));
        acc = ro2 < d2;
      }
      if (kVote) {
        // Probe pre-test: if one of the probe targets (real targets of the
        // group) fails the opening test, the vote fails; same arithmetic as
        // the vote, so the outcome is identical, only cheaper.
        bool und = has && !acc;
        if (__any_sync(0xffffffffu, und)) {
#pragma unroll
          for (int k = 0; k < kProbesPerSlot * T; ++k) {
            const float4 pr = S.probe[k];
            float dx = c4.x - pr.x, dy = c4.y - pr.y, dz = c4.z - pr.z;
            float r2 = fmaf(dx, dx, fmaf(dy, dy, dz * dz));
            und = und && (ro2 < r2);
          }
        }
        unsigned cand = __ballot_sync(0xffffffffu, und);
        st_voted += __popc(cand);
        if (und) S.cand[lane] = make_float4(c4.x, c4.y, c4.z, ro2);
        __syncwarp();
        unsigned accm = 0;
        while (cand) {
          const int c = __ffs(cand) - 1;
          cand &= cand - 1u;
          const float4 cd = S.cand[c];
          bool ok = true;
#pragma unroll
          for (int k = 0; k < T; ++k) {
            float dx = cd.x - px[k], dy = cd.y - py[k], dz = cd.z - pz[k];
            float r2 = fmaf(dx, dx, fmaf(dy, dy, dz * dz));
            ok = ok && (!valid[k] || cd.w < r2);
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
      // an opened node whose children all pass the box test: its children
      // go to the list without being tested
      const bool kids = open_int && children_accepted(d2, ro2, flags);

      // ---- accepted nodes -> interaction list ---------------------------
      const unsigned am = __ballot_sync(0xffffffffu, has && acc);
      if (has && acc) list_put(S, nl + __popc(am & lt), c4);
      nl += __popc(am);

      // ---- opened internal nodes -> stack -------------------------------
      const bool push = open_int && !kids;
      const unsigned om = __ballot_sync(0xffffffffu, push);
      const int npush = __popc(om);
      if (sp + npush <= kStackCap) {
        if (push)
          S.stack[sp + __popc(om & lt)] =
              ((unsigned)link << 3) | (unsigned)(count - 1);
        sp += npush;
      } else if (npush) {
        if (lane == 0) set_err(ctrl, kErrOverflow);
      }
      __syncwarp();

      // ---- opened leaves -> their particles; accepted children ----------
      const bool expand = open_leaf || kids;
      const unsigned lm = __ballot_sync(0xffffffffu, expand);
      if (lm) {
        const int pc = expand ? (count > 0 ? count : 0) : 0;
        const int ppre = warp_incl_scan(pc, lane);
        const int ptotal = __shfl_sync(0xffffffffu, ppre, 31);
        const int pexcl = ppre - pc;
        // which targets of the group see their own particle (only leaves
        // holding some of the group's own targets can)
        const bool mine = kSelf && open_leaf && pc > 0 && (long long)link < t0 + GS &&
                          (long long)link + pc > t0;
        if (kSelf && __any_sync(0xffffffffu, mine)) {
          unsigned long long msk = 0ull;
          if (mine) {
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
          ++st_chunks;
          const int qi = base + lane;
          int lo = 0;
#pragma unroll
          for (int s = 16; s >= 1; s >>= 1) {
            int v = __shfl_sync(0xffffffffu, ppre, lo + s - 1);
            if (v <= qi) lo += s;
          }
          const int owner = lo > 31 ? 31 : lo;
          const int of = __shfl_sync(0xffffffffu, link, owner);
          const int oe = __shfl_sync(0xffffffffu, pexcl, owner);
          const bool okid = __shfl_sync(0xffffffffu, (int)kids, owner) != 0;
          float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
          if (qi < ptotal) pv = entry_source(a, okid, of + (qi - oe));
          if (nl >= kFlushAt) flush_front(S, accum, nl, nvalid, executed);
          if (qi < ptotal) list_put(S, nl + lane, pv);
          nl += (ptotal - base < 32) ? (ptotal - base) : 32;
          __syncwarp();
        }
      }
    }
    if (nl >= kFlushAt) flush_front(S, accum, nl, nvalid, executed);
    if (nl > 0) {
      if ((nl & 1) && lane == 0) list_put(S, nl, make_float4(0.f, 0.f, 0.f, 0.f));
      __syncwarp();
      accum.run(S, (nl + 1) / 2);
      executed += (unsigned long long)nl * nvalid;
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < T; ++k) {
      if (!valid[k]) continue;
      const long long t = t0 + k * 32 + lane;
      float x0, x1, y0, y1, z0, z1, p0, p1;
      upk(accum.ax[k], x0, x1);
      upk(accum.ay[k], y0, y1);
      upk(accum.az[k], z0, z1);
      upk(accum.ph[k], p0, p1);
      float ph = p0 + p1;
      if (kSelf && !kEps0 && selfhit[k]) {
        // undo the self pair: it added m * rsqrt(eps^2) to -phi
        const float m_self = __ldg(a.tpos + t).w;
        ph += m_self * rsqrt_ftz(a.eps2);
      }
      const unsigned ci = a.tperm ? a.tperm[t] : (unsigned)t;
      if (ci < (unsigned long long)a.m)
        a.out[ci] = make_float4(a.G * (x0 + x1), a.G * (y0 + y1), a.G * (z0 + z1),
                                a.G * ph);
    }
    if (a.gcost && lane == 0) {
      const unsigned long long c = executed - exec0;
      a.gcost[g] = c < 0xffffffffull ? (unsigned)c : 0xffffffffu;
    }
    ++ngroup_done;
  }
  if (lane == 0) {
    atomicAdd(&ctrl->step.executed, executed);
    atomicAdd(&ctrl->step.groups, ngroup_done);
    atomicAdd(&ctrl->step.walk_stats[0], st_rounds);
    atomicAdd(&ctrl->step.walk_stats[1], st_tested);
    atomicAdd(&ctrl->step.walk_stats[2], st_voted);
    atomicAdd(&ctrl->step.walk_stats[3], st_chunks);
  }
}


// ---------------------------------------------------------------------------
// Pipelined walk: the same traversal and arithmetic as walk_kernel, split
// between two warps per group.  The producer warp traverses (pops, record
// loads, box/probe/vote tests, leaf gathers) and fills 128-entry list buffers;
// the consumer warp evaluates full buffers for the group's targets.  Four
// buffers per pair circulate through two mbarriers each (full: producer ->
// consumer, empty: consumer -> producer); every wait is bounded.  The
// traversal (latency- and control-bound) and the evaluation (FMA-bound) of
// different groups then overlap within an SM instead of alternating inside
// one warp.  Split this way each warp needs fewer registers (64: four blocks
// of eight warps per SM, twice the fused walk's warps), which is what makes
// it the faster form.
// ---------------------------------------------------------------------------
constexpr int kWsPairs = 4;
constexpr int kWsThreads = kWsPairs * 64;
constexpr int kWsBufs = 4;
constexpr int kWsEntries = 128;   // per buffer: fewer hand-offs than 64 (-1..2%)
constexpr unsigned kWsWaitLimit = 1u << 26;   // polls; a buffer takes microseconds

struct WsHdr {
  long long group;           // -1: no more groups
  int n;                     // entries in the buffer
  int last;                  // last buffer of the group
  unsigned self0, self1;     // targets whose own particle was evaluated
};

struct WsPairSmem {
  ulonglong2 list[kWsBufs][kWsEntries / 2][2];
  WsHdr hdr[kWsBufs];
  unsigned long long full[kWsBufs], empty[kWsBufs];
  float4 cand[32];
  float4 probe[8];
  unsigned int stack[kStackCap];
};

__device__ __forceinline__ unsigned su32(const void *p) {
  return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mb_init(unsigned long long *b, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mb_arrive(unsigned long long *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mb_try(unsigned long long *b, unsigned parity) {
  unsigned ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
               " selp.u32 %0, 1, 0, p;\n}\n"
               : "=r"(ok) : "r"(su32(b)), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait by every lane; false (for the whole warp) on timeout.
__device__ __forceinline__ bool mb_wait(unsigned long long *b, unsigned parity) {
  bool ok = false;
  for (unsigned i = 0; i < kWsWaitLimit && !ok; ++i) ok = mb_try(b, parity);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void ws_put(ulonglong2 (*list)[2], int j, float4 v) {
  float *w = reinterpret_cast<float *>(&list[j >> 1][0]);
  const int h = j & 1;
  w[h] = v.x;
  w[2 + h] = v.y;
  w[4 + h] = v.z;
  w[6 + h] = v.w;
}

template <int T, bool kVote, bool kEps0, bool kSelf>
__device__ __forceinline__ void ws_producer(const WalkArgs &a, DevCtrl *ctrl, WsPairSmem &S,
                                            long long nnodes) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  constexpr int GS = 32 * T;
  const long long gend = a.g_end;       // groups [g_begin, g_end) of this call
  unsigned st_rounds = 0, st_tested = 0, st_voted = 0, st_chunks = 0, done = 0;
  unsigned eph = 0;              // parity of the next wait on each empty barrier
  int b = 0, nl = 0;
  bool alive = mb_wait(&S.empty[0], 0);
  eph ^= 1u;
  // hand buffer b (nl entries) to the consumer and take the next one
  auto hand_off = [&](long long g, int n, int last, unsigned s0, unsigned s1) {
    if (lane == 0) {
      WsHdr h;
      h.group = g; h.n = n; h.last = last; h.self0 = s0; h.self1 = s1;
      S.hdr[b] = h;
    }
    __syncwarp();
    mb_arrive(&S.full[b]);
    b = (b + 1) % kWsBufs;
    alive = alive && mb_wait(&S.empty[b], (eph >> b) & 1u);
    eph ^= 1u << b;
  };

  while (alive) {
    unsigned long long gg = 0;
    if (lane == 0) gg = atomicAdd(&ctrl->step.work_ctr, 1u);
    long long g = (long long)__shfl_sync(0xffffffffu, gg, 0) + a.g_begin;
    if (g >= gend) break;
    if (a.gorder) {
      g = a.gorder[g];
      if (g >= gend) {                    // not a permutation: skip, flag
        if (lane == 0) set_err(ctrl, kErrOverflow);
        continue;
      }
    }
    const long long t0 = g * GS;

    float px[T], py[T], pz[T];
    bool valid[T], selfhit[T];
    float bl0 = INFINITY, bl1 = INFINITY, bl2 = INFINITY;
    float bh0 = -INFINITY, bh1 = -INFINITY, bh2 = -INFINITY;
#pragma unroll
    for (int k = 0; k < T; ++k) {
      const long long t = t0 + k * 32 + lane;
      valid[k] = t < a.m;
      const float4 p = __ldg(a.tpos + (valid[k] ? t : t0));
      px[k] = p.x; py[k] = p.y; pz[k] = p.z;
      if ((lane & (32 / kProbesPerSlot - 1)) == 0)
        S.probe[k * kProbesPerSlot + lane / (32 / kProbesPerSlot)] = make_float4(p.x, p.y, p.z, 0.f);
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
    int sp = 1;
    if (lane == 0) S.stack[0] = 0u;
    __syncwarp();

    // append `cnt` entries (this lane's at rank r if put), spilling into the
    // next buffer when the current one fills
    auto append = [&](bool put, int r, int cnt, float4 v) {
      if (nl + cnt > kWsEntries) {
        const int first = kWsEntries - nl;      // entries that still fit
        if (put && r < first) ws_put(S.list[b], nl + r, v);
        hand_off(g, kWsEntries, 0, 0u, 0u);
        if (put && r >= first) ws_put(S.list[b], r - first, v);
        nl = cnt - first;
      } else {
        if (put) ws_put(S.list[b], nl + r, v);
        nl += cnt;
      }
    };

    while (sp > 0 && alive) {
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
      const unsigned starts = __reduce_or_sync(0xffffffffu, take ? (1u << excl) : 0u);
      bool has = lane < total;
      int e = __popc(starts & ((2u << lane) - 1u)) - 1;
      e = e < 0 ? 0 : e;
      const unsigned ebase = __shfl_sync(0xffffffffu, ent >> 3, e);
      const int eexcl = __shfl_sync(0xffffffffu, excl, e);
      const unsigned node = ebase + (unsigned)(lane - eexcl);
      __syncwarp();
      ++st_rounds;
      st_tested += (unsigned)total;
      if (has && node >= nnodes) {
        has = false;
        set_err(ctrl, kErrOverflow);
      }
      float4 c4 = make_float4(0.f, 0.f, 0.f, 0.f);
      float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
      if (has) {
        const float4 *r = reinterpret_cast<const float4 *>(a.rec + node);
        c4 = __ldg(r);
        q = __ldg(r + 1);
      }
      const float ro2 = q.x;
      const int link = __float_as_int(q.y);
      int count = __float_as_int(q.z);
      const int flags = __float_as_int(q.w);
      bool acc = false;
      float d2 = 0.f;
      if (has) {
        float dx = fmaxf(fmaxf(bl0 - c4.x, c4.x - bh0), 0.f);
        float dy = fmaxf(fmaxf(bl1 - c4.y, c4.y - bh1), 0.f);
        float dz = fmaxf(fmaxf(bl2 - c4.z, c4.z - bh2), 0.f);
        d2 = fmaf(dx, dx, fmaf(dy, dy, dz * dz));
        acc = ro2 < d2;
      }
      if (kVote) {
        bool und = has && !acc;
        if (__any_sync(0xffffffffu, und)) {
#pragma unroll
          for (int k = 0; k < kProbesPerSlot * T; ++k) {
            const float4 pr = S.probe[k];
            float dx = c4.x - pr.x, dy = c4.y - pr.y, dz = c4.z - pr.z;
            float r2 = fmaf(dx, dx, fmaf(dy, dy, dz * dz));
            und = und && (ro2 < r2);
          }
        }
        unsigned cand = __ballot_sync(0xffffffffu, und);
        st_voted += __popc(cand);
        if (und) S.cand[lane] = make_float4(c4.x, c4.y, c4.z, ro2);
        __syncwarp();
        unsigned accm = 0;
        while (cand) {
          const int c = __ffs(cand) - 1;
          cand &= cand - 1u;
          const float4 cd = S.cand[c];
          bool ok = true;
#pragma unroll
          for (int k = 0; k < T; ++k) {
            float dx = cd.x - px[k], dy = cd.y - py[k], dz = cd.z - pz[k];
            float r2 = fmaf(dx, dx, fmaf(dy, dy, dz * dz));
            ok = ok && (!valid[k] || cd.w < r2);
          }
          if (__all_sync(0xffffffffu, ok)) accm |= 1u << c;
        }
        acc = acc || ((accm >> lane) & 1u);
      }
      const bool leaf = (flags & 1) != 0;
      const bool open_int = has && !acc && !leaf && count >= 1 && count <= 8 &&
                            (unsigned)link > node && (long long)link + count <= nnodes;
      const bool open_leaf = has && !acc && leaf && link >= 0 && link <= a.n;
      if (open_leaf && count > a.n - link) count = (int)(a.n - link);
      // an opened node whose children all pass the box test (children_factor
      // of the build): its children go to the list without being tested
      const bool kids = open_int && children_accepted(d2, ro2, flags);

      // accepted nodes -> list
      const unsigned am = __ballot_sync(0xffffffffu, has && acc);
      append(has && acc, __popc(am & lt), __popc(am), c4);

      // opened internal nodes -> stack
      const bool push = open_int && !kids;
      const unsigned om = __ballot_sync(0xffffffffu, push);
      const int npush = __popc(om);
      if (sp + npush <= kStackCap) {
        if (push)
          S.stack[sp + __popc(om & lt)] = ((unsigned)link << 3) | (unsigned)(count - 1);
        sp += npush;
      } else if (npush) {
        if (lane == 0) set_err(ctrl, kErrOverflow);
      }
      __syncwarp();

      // opened leaves -> their particles; accepted children -> their records
      const bool expand = open_leaf || kids;
      const unsigned lm = __ballot_sync(0xffffffffu, expand);
      if (lm) {
        const int pc = expand ? (count > 0 ? count : 0) : 0;
        const int ppre = warp_incl_scan(pc, lane);
        const int ptotal = __shfl_sync(0xffffffffu, ppre, 31);
        const int pexcl = ppre - pc;
        const bool mine = kSelf && open_leaf && pc > 0 && (long long)link < t0 + GS &&
                          (long long)link + pc > t0;
        if (kSelf && __any_sync(0xffffffffu, mine)) {
          unsigned long long msk = 0ull;
          if (mine) {
            long long lo = (long long)link - t0, hi = lo + pc;
            if (lo < 0) lo = 0;
            if (hi > GS) hi = GS;
            if (lo < hi) {
              unsigned long long upper = (hi >= 64) ? ~0ull : ((1ull << hi) - 1ull);
              msk = upper & ~((1ull << lo) - 1ull);
            }
          }
          const unsigned m0 = __reduce_or_sync(0xffffffffu, (unsigned)msk);
          const unsigned m1 = __reduce_or_sync(0xffffffffu, (unsigned)(msk >> 32));
#pragma unroll
          for (int k = 0; k < T; ++k)
            selfhit[k] = selfhit[k] || (((k == 0 ? m0 : m1) >> lane) & 1u);
        }
        for (int base = 0; base < ptotal && alive; base += 32) {
          ++st_chunks;
          const int qi = base + lane;
          int lo = 0;
#pragma unroll
          for (int s = 16; s >= 1; s >>= 1) {
            int v = __shfl_sync(0xffffffffu, ppre, lo + s - 1);
            if (v <= qi) lo += s;
          }
          const int owner = lo > 31 ? 31 : lo;
          const int of = __shfl_sync(0xffffffffu, link, owner);
          const int oe = __shfl_sync(0xffffffffu, pexcl, owner);
          const bool okid = __shfl_sync(0xffffffffu, (int)kids, owner) != 0;
          float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
          if (qi < ptotal) pv = entry_source(a, okid, of + (qi - oe));
          const int nput = (ptotal - base < 32) ? (ptotal - base) : 32;
          append(qi < ptotal, lane, nput, pv);
          __syncwarp();
        }
      }
    }
    if (!alive) break;
    // the group's last buffer: pad to a pair, record the self hits
    if ((nl & 1) && lane == 0) ws_put(S.list[b], nl, make_float4(0.f, 0.f, 0.f, 0.f));
    const unsigned s0 = __ballot_sync(0xffffffffu, selfhit[0]);
    const unsigned s1 = T > 1 ? __ballot_sync(0xffffffffu, selfhit[T - 1]) : 0u;
    hand_off(g, nl, 1, s0, s1);
    nl = 0;
    ++done;
  }
  // no more groups: tell the consumer
  if (alive) {
    if (lane == 0) {
      WsHdr h;
      h.group = -1; h.n = 0; h.last = 1; h.self0 = h.self1 = 0u;
      S.hdr[b] = h;
    }
    __syncwarp();
    mb_arrive(&S.full[b]);
  } else if (lane == 0) {
    set_err(ctrl, kErrTimeout);
  }
  if (lane == 0) {
    atomicAdd(&ctrl->step.groups, done);
    atomicAdd(&ctrl->step.walk_stats[0], st_rounds);
    atomicAdd(&ctrl->step.walk_stats[1], st_tested);
    atomicAdd(&ctrl->step.walk_stats[2], st_voted);
    atomicAdd(&ctrl->step.walk_stats[3], st_chunks);
  }
}

template <int T, bool kEps0, bool kSelf>
__device__ __forceinline__ void ws_consumer(const WalkArgs &a, DevCtrl *ctrl, WsPairSmem &S) {
  const int lane = threadIdx.x & 31;
  constexpr int GS = 32 * T;
  unsigned long long executed = 0, exec0 = 0;
  // all buffers start empty
#pragma unroll
  for (int k = 0; k < kWsBufs; ++k) mb_arrive(&S.empty[k]);
  unsigned fph = 0;
  int b = 0;
  long long cur = -2;
  int nvalid = 0;
  Acc<T, kEps0> accum;
  accum.eps2 = pk(a.eps2, a.eps2);
  for (;;) {
    if (!mb_wait(&S.full[b], (fph >> b) & 1u)) {
      if (lane == 0) set_err(ctrl, kErrTimeout);
      break;
    }
    fph ^= 1u << b;
    const WsHdr h = S.hdr[b];
    if (h.group < 0) break;
    if (h.group != cur) {                 // first buffer of a new group
      cur = h.group;
      exec0 = executed;
      const long long t0 = cur * GS;
      nvalid = (int)((a.m - t0) < GS ? (a.m - t0) : GS);
#pragma unroll
      for (int k = 0; k < T; ++k) {
        const long long t = t0 + k * 32 + lane;
        const float4 p = __ldg(a.tpos + (t < a.m ? t : t0));
        accum.px[k] = pk(p.x, p.x);
        accum.py[k] = pk(p.y, p.y);
        accum.pz[k] = pk(p.z, p.z);
        accum.ax[k] = accum.ay[k] = accum.az[k] = accum.ph[k] = 0ull;
      }
    }
    if (h.n > 0) {
      if (h.n == kWsEntries) accum.template run_full_list<kWsEntries / 2>(S.list[b]);
      else accum.run_list(S.list[b], (h.n + 1) / 2);
      executed += (unsigned long long)h.n * nvalid;
    }
    if (h.last) {
      const long long t0 = cur * GS;
      if (a.gcost && lane == 0) {
        const unsigned long long c = executed - exec0;
        a.gcost[cur] = c < 0xffffffffull ? (unsigned)c : 0xffffffffu;
      }
#pragma unroll
      for (int k = 0; k < T; ++k) {
        const long long t = t0 + k * 32 + lane;
        if (t >= a.m) continue;
        float x0, x1, y0, y1, z0, z1, p0, p1;
        upk(accum.ax[k], x0, x1);
        upk(accum.ay[k], y0, y1);
        upk(accum.az[k], z0, z1);
        upk(accum.ph[k], p0, p1);
        float ph = p0 + p1;
        const bool sh = (((k == 0 ? h.self0 : h.self1) >> lane) & 1u) != 0;
        if (kSelf && !kEps0 && sh) {
          const float m_self = __ldg(a.tpos + t).w;
          ph += m_self * rsqrt_ftz(a.eps2);
        }
        const unsigned ci = a.tperm ? a.tperm[t] : (unsigned)t;
        if (ci < (unsigned long long)a.m)
          a.out[ci] = make_float4(a.G * (x0 + x1), a.G * (y0 + y1), a.G * (z0 + z1),
                                  a.G * ph);
      }
    }
    __syncwarp();
    mb_arrive(&S.empty[b]);
    b = (b + 1) % kWsBufs;
  }
  if (lane == 0) atomicAdd(&ctrl->step.executed, executed);
}

template <int T, bool kVote, bool kEps0, bool kSelf>
__global__ void __launch_bounds__(kWsThreads, 4)
walk_ws_kernel(WalkArgs a, DevCtrl *ctrl) {
  __shared__ WsPairSmem smem[kWsPairs];
  const int w = threadIdx.x >> 5;
  WsPairSmem &S = smem[w >> 1];
  if (threadIdx.x < kWsPairs * kWsBufs) {
    const int p = threadIdx.x / kWsBufs, k = threadIdx.x % kWsBufs;
    mb_init(&smem[p].full[k], 32);
    mb_init(&smem[p].empty[k], 32);
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();
  const long long nnodes = node_total(ctrl);
  if (w & 1) ws_consumer<T, kEps0, kSelf>(a, ctrl, S);
  else ws_producer<T, kVote, kEps0, kSelf>(a, ctrl, S, nnodes);
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
  const long long nnodes = node_total(ctrl);
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
cudaError_t launch_ws(const WalkArgs &a, DevCtrl *ctrl, cudaStream_t s) {
  static std::atomic<int> memo[kMaxDevices];
  const int per_sm = per_device(memo, [] {
    int b = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &b, walk_ws_kernel<T, kVote, kEps0, kSelf>, kWsThreads, 0);
    return b > 0 ? b : 1;
  });
  const long long ngroups = a.g_end - a.g_begin;
  long long blocks = (long long)a.num_sms * per_sm;
  const long long need = (ngroups + kWsPairs - 1) / kWsPairs;
  if (blocks > need) blocks = need;
  if (blocks < 1) blocks = 1;
  {
    const cudaError_t le = launch_k(walk_ws_kernel<T, kVote, kEps0, kSelf>, dim3((unsigned)blocks), dim3(kWsThreads), 0, s,
                                    a, ctrl);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

template <int T, bool kVote, bool kEps0, bool kSelf>
cudaError_t launch_one(const WalkArgs &a, DevCtrl *ctrl, cudaStream_t s) {
  // groups of 32 always run as producer/consumer pairs: with twice the
  // traversal per target, the fused form was 19-25% slower for them
  if constexpr (T == 1) {
    return launch_ws<T, kVote, kEps0, kSelf>(a, ctrl, s);
  } else {
    if (a.pipelined) return launch_ws<T, kVote, kEps0, kSelf>(a, ctrl, s);
  }
  static std::atomic<int> memo[kMaxDevices];
  const int per_sm = per_device(memo, [] {
    int b = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &b, walk_kernel<T, kVote, kEps0, kSelf>, kWalkThreads, 0);
    return b > 0 ? b : 1;
  });
  const long long ngroups = a.g_end - a.g_begin;
  long long blocks = (long long)a.num_sms * per_sm;
  long long need = (ngroups + kWalkWarps - 1) / kWalkWarps;
  if (blocks > need) blocks = need;
  if (blocks < 1) blocks = 1;
  {
    const cudaError_t le = launch_k(walk_kernel<T, kVote, kEps0, kSelf>, dim3((unsigned)blocks), dim3(kWalkThreads), 0, s,
                                    a, ctrl);
    if (le != cudaSuccess) return le;
  }
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

// ---------------------------------------------------------------------------
// Group schedule.  Groups differ in cost by an order of magnitude (a group of
// Morton-consecutive targets that straddles a high-level cell boundary, or
// sits next to a dense clump, opens far more of the tree), and tickets
// handed out in Morton order leave the heaviest ones to start last: the walk
// ends with a tail of a few long groups while most SMs idle.  Handing the
// heaviest out first (largest-first list scheduling) shortens that tail; the
// costs come from the previous call's walk over the same groups.  Only the
// order in which groups are taken changes, so every result is unchanged.
// ---------------------------------------------------------------------------
constexpr int kOrderThreads = 256;
constexpr int kCostClasses = 33;      // 0 and the 32 powers of two of a u32

// class of a cost by its leading bit, heaviest first: [2^31, 2^32) -> 0,
// [2^30, 2^31) -> 1, ..., 1 -> 31, 0 -> 32
__device__ __forceinline__ int cost_class(unsigned c) { return __clz(c); }

// Groups per class.  Lanes of one class (match.any) add with one atomic.
__global__ void __launch_bounds__(kOrderThreads)
group_class_count_kernel(const unsigned int *__restrict__ cost, long long ngroups,
                         unsigned int *cnt) {
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * kOrderThreads;
  for (long long base = (long long)blockIdx.x * kOrderThreads; base < ngroups; base += stride) {
    const long long g = base + threadIdx.x;
    const int cls = g < ngroups ? cost_class(cost[g]) : kCostClasses;
    const unsigned peers = __match_any_sync(0xffffffffu, cls);
    if (cls < kCostClasses && (peers & ((1u << lane) - 1u)) == 0u)
      atomicAdd(&cnt[cls], (unsigned)__popc(peers));
  }
}

// Placement: class k owns positions [start_k, start_k + cnt_k) with the
// classes in order; each group takes the next free position of its class.
// Every class hands out exactly cnt_k positions, so order[] is a
// permutation of [0, ngroups) (the order within a class is arbitrary).
__global__ void __launch_bounds__(kOrderThreads)
group_place_kernel(const unsigned int *__restrict__ cost, long long ngroups,
                   const unsigned int *__restrict__ cnt, unsigned int *fill,
                   unsigned int *__restrict__ order) {
  __shared__ unsigned int start[kCostClasses];
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  if (threadIdx.x == 0) {
    unsigned run = 0;
    for (int k = 0; k < kCostClasses; ++k) {
      start[k] = run;
      run += cnt[k];
    }
  }
  __syncthreads();
  const long long stride = (long long)gridDim.x * kOrderThreads;
  for (long long base = (long long)blockIdx.x * kOrderThreads; base < ngroups; base += stride) {
    const long long g = base + threadIdx.x;
    const int cls = g < ngroups ? cost_class(cost[g]) : kCostClasses;
    const unsigned peers = __match_any_sync(0xffffffffu, cls);
    const int leader = __ffs(peers) - 1;
    unsigned at = 0;
    if (cls < kCostClasses && lane == leader) at = atomicAdd(&fill[cls], (unsigned)__popc(peers));
    at = __shfl_sync(0xffffffffu, at, leader) + (unsigned)__popc(peers & lt);
    if (cls < kCostClasses && at < cnt[cls]) order[start[cls] + at] = (unsigned)g;
  }
}

cudaError_t launch_group_order(const unsigned int *cost, long long ngroups,
                               unsigned int *order, DevCtrl *ctrl, int num_sms,
                               cudaStream_t s) {
  if (ngroups <= 0) return cudaSuccess;
  long long blocks = (ngroups + kOrderThreads - 1) / kOrderThreads;
  if (blocks > 4LL * num_sms) blocks = 4LL * num_sms;
  {
    const cudaError_t le = launch_k(group_class_count_kernel, dim3((unsigned)blocks), dim3(kOrderThreads), 0, s,
                                    cost, ngroups,
                                                                        ctrl->step.sched_cnt);
    if (le != cudaSuccess) return le;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    const cudaError_t le = launch_k(group_place_kernel, dim3((unsigned)blocks), dim3(kOrderThreads), 0, s,
      cost, ngroups, ctrl->step.sched_cnt, ctrl->step.sched_fill, order);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

cudaError_t launch_walk(const WalkArgs &a, DevCtrl *ctrl, cudaStream_t s) {
  if (a.m <= 0 || a.g_end <= a.g_begin) return cudaSuccess;
  return a.group == 32 ? launch_t<1>(a, ctrl, s) : launch_t<2>(a, ctrl, s);
}

}  // namespace bh
