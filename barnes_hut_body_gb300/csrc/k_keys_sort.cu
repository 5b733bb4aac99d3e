// Bounding cube, Morton keys and the on-device radix sort.
//
// Stages 1-3 of the pipeline of the GASPHiA tree-code page (section
// "计算核函数": computeBoundingBox) and of the tree page after Burtscher &
// Pingali (section "实现步骤": bounding box by reduction, then Morton /
// Z-order keys and a spatial sort so that the 32 threads of a warp hold
// spatially close particles -- the page's "排序算法" section shows the walk
// is 10-15x slower without it).
//
// GB300 design:
//  * bbox: one pass of 16-byte loads, grid sized to the SM count; the last
//    block to finish (ticket counter, no waiting) reduces the block partials
//    and writes the cube and the quantisation scale.
//  * keys: fixed fp32 op sequence (round-to-nearest sub, mul; clamp;
//    truncate) so the integer codes are reproducible bit for bit; the same
//    pass builds the digit histograms of every radix pass.
//  * sort: least-significant-digit radix sort, 8-bit digits, one kernel per
//    digit ("one sweep"): each tile ranks its keys with warp ballots, learns
//    its global offset by decoupled look-back over the tiles before it (a
//    bounded wait that flags BH_ETIMEOUT instead of hanging), then scatters
//    through shared memory so that global writes come out in runs.  Stable,
//    so equal keys keep the original index order.
#include <cuda_runtime.h>
#include <stdint.h>

#include "bh_internal.h"

namespace bh {

namespace {

__device__ __forceinline__ void set_err(DevCtrl *c, unsigned code) {
  atomicCAS(&c->keep.err, 0u, code);
}

// The top digit of a 63-bit key (bit 63 is always 0): bits 55..62, the
// octree's first two levels and two bits of the third.
constexpr int kTopShift = 55;
// The bucket sort: one block of kBucketThreads threads holds a bucket of up
// to kBucketCap keys (kBucketItems per thread) in shared memory.
constexpr int kBucketThreads = 512;
constexpr int kBucketItems = 9;
constexpr int kBucketCap = kBucketThreads * kBucketItems;   // 4608 keys

__device__ __forceinline__ bool finite4(float4 p) {
  return isfinite(p.x) && isfinite(p.y) && isfinite(p.z) && isfinite(p.w);
}

// ---------------------------------------------------------------------------
// Bounding cube
// ---------------------------------------------------------------------------
constexpr int kBboxThreads = 256;

__global__ void __launch_bounds__(kBboxThreads)
bbox_kernel(const float4 *__restrict__ pm, long long n, float4 *partials,
            DevCtrl *ctrl, int which, int bits, int bump_epoch) {
  float lo0 = INFINITY, lo1 = INFINITY, lo2 = INFINITY;
  float hi0 = -INFINITY, hi1 = -INFINITY, hi2 = -INFINITY;
  float mm = 0.f;                       // largest |mass|
  bool bad = false;
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  // four independent 16-byte loads in flight per thread
  for (; i + 3 * stride < n; i += 4 * stride) {
    float4 p[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) p[u] = __ldg(pm + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      bad |= !finite4(p[u]);
      mm = fmaxf(mm, fabsf(p[u].w));
      lo0 = fminf(lo0, p[u].x); hi0 = fmaxf(hi0, p[u].x);
      lo1 = fminf(lo1, p[u].y); hi1 = fmaxf(hi1, p[u].y);
      lo2 = fminf(lo2, p[u].z); hi2 = fmaxf(hi2, p[u].z);
    }
  }
  for (; i < n; i += stride) {
    float4 p = __ldg(pm + i);
    bad |= !finite4(p);
    mm = fmaxf(mm, fabsf(p.w));
    lo0 = fminf(lo0, p.x); hi0 = fmaxf(hi0, p.x);
    lo1 = fminf(lo1, p.y); hi1 = fmaxf(hi1, p.y);
    lo2 = fminf(lo2, p.z); hi2 = fmaxf(hi2, p.z);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo0 = fminf(lo0, __shfl_xor_sync(0xffffffffu, lo0, o));
    lo1 = fminf(lo1, __shfl_xor_sync(0xffffffffu, lo1, o));
    lo2 = fminf(lo2, __shfl_xor_sync(0xffffffffu, lo2, o));
    hi0 = fmaxf(hi0, __shfl_xor_sync(0xffffffffu, hi0, o));
    hi1 = fmaxf(hi1, __shfl_xor_sync(0xffffffffu, hi1, o));
    hi2 = fmaxf(hi2, __shfl_xor_sync(0xffffffffu, hi2, o));
    mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
  }
  bad = __any_sync(0xffffffffu, bad);
  __shared__ float s[7][kBboxThreads / 32];
  __shared__ int s_bad[kBboxThreads / 32];
  __shared__ bool s_last;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s[0][w] = lo0; s[1][w] = lo1; s[2][w] = lo2;
    s[3][w] = hi0; s[4][w] = hi1; s[5][w] = hi2;
    s[6][w] = mm;
    s_bad[w] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float4 a = make_float4(s[0][0], s[1][0], s[2][0], 0.f);
    float4 b = make_float4(s[3][0], s[4][0], s[5][0], s[6][0]);
    int anybad = s_bad[0];
    for (int k = 1; k < kBboxThreads / 32; ++k) {
      a.x = fminf(a.x, s[0][k]); a.y = fminf(a.y, s[1][k]); a.z = fminf(a.z, s[2][k]);
      b.x = fmaxf(b.x, s[3][k]); b.y = fmaxf(b.y, s[4][k]); b.z = fmaxf(b.z, s[5][k]);
      b.w = fmaxf(b.w, s[6][k]);
      anybad |= s_bad[k];
    }
    a.w = anybad ? 1.f : 0.f;
    partials[2 * blockIdx.x] = a;
    partials[2 * blockIdx.x + 1] = b;
    __threadfence();
    unsigned t = atomicAdd(&ctrl->step.bbox_done[which], 1u);
    s_last = (t == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  // Last block: reduce the partials of every block.
  __threadfence();
  lo0 = lo1 = lo2 = INFINITY;
  hi0 = hi1 = hi2 = -INFINITY;
  mm = 0.f;
  bad = false;
  for (int k = threadIdx.x; k < (int)gridDim.x; k += blockDim.x) {
    float4 a = __ldcg(partials + 2 * k), b = __ldcg(partials + 2 * k + 1);
    lo0 = fminf(lo0, a.x); lo1 = fminf(lo1, a.y); lo2 = fminf(lo2, a.z);
    hi0 = fmaxf(hi0, b.x); hi1 = fmaxf(hi1, b.y); hi2 = fmaxf(hi2, b.z);
    mm = fmaxf(mm, b.w);
    bad |= (a.w != 0.f);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo0 = fminf(lo0, __shfl_xor_sync(0xffffffffu, lo0, o));
    lo1 = fminf(lo1, __shfl_xor_sync(0xffffffffu, lo1, o));
    lo2 = fminf(lo2, __shfl_xor_sync(0xffffffffu, lo2, o));
    hi0 = fmaxf(hi0, __shfl_xor_sync(0xffffffffu, hi0, o));
    hi1 = fmaxf(hi1, __shfl_xor_sync(0xffffffffu, hi1, o));
    hi2 = fmaxf(hi2, __shfl_xor_sync(0xffffffffu, hi2, o));
    mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
  }
  bad = __any_sync(0xffffffffu, bad);
  __syncthreads();
  if (lane == 0) {
    s[0][w] = lo0; s[1][w] = lo1; s[2][w] = lo2;
    s[3][w] = hi0; s[4][w] = hi1; s[5][w] = hi2;
    s[6][w] = mm;
    s_bad[w] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float l[3] = {s[0][0], s[1][0], s[2][0]}, h[3] = {s[3][0], s[4][0], s[5][0]};
    int anybad = s_bad[0];
    float mmax = s[6][0];
    for (int k = 1; k < kBboxThreads / 32; ++k) {
      for (int a = 0; a < 3; ++a) {
        l[a] = fminf(l[a], s[a][k]);
        h[a] = fmaxf(h[a], s[3 + a][k]);
      }
      mmax = fmaxf(mmax, s[6][k]);
      anybad |= s_bad[k];
    }
    // Cube side: the largest extent (fp32 subtraction); 1 if all coincide.
    float L = 0.f;
    for (int a = 0; a < 3; ++a) L = fmaxf(L, __fsub_rn(h[a], l[a]));
    if (L == 0.f) L = 1.f;
    ctrl->keep.cube[which] = make_float4(l[0], l[1], l[2], L);
    ctrl->keep.scale[which] = __fdiv_rn((float)(1u << bits), L);
    // Fixed-point moment scales (powers of two): with |m| < 2^(e_m + 1),
    // (coordinate - lo) < 2^(e_L + 1) and n <= 2^c, a sum over all particles
    // of m 2^k_m or of m (coordinate - lo) 2^k_x stays below 2^62.
    int km = 0, kx = 0;
    if (mmax > 0.f && isfinite(mmax)) {
      const int c = n > 1 ? 64 - __clzll((unsigned long long)(n - 1)) : 0;
      const int em = ilogbf(mmax), eL = ilogbf(L);
      km = 61 - c - em;
      kx = 60 - c - em - eL;
    }
    ctrl->keep.qexp[which][0] = km;
    ctrl->keep.qexp[which][1] = kx;
    if (anybad) set_err(ctrl, kErrNonFinite);
    if (bump_epoch) ctrl->keep.epoch += 1u;
    ctrl->step.bbox_done[which] = 0;
  }
}

// ---------------------------------------------------------------------------
// Morton keys + digit histograms
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long spread3(unsigned int v) {
  // Insert two zero bits after each of the low 21 bits (Z-order interleave).
  unsigned long long x = v & 0x1fffffu;
  x = (x | x << 32) & 0x1f00000000ffffull;
  x = (x | x << 16) & 0x1f0000ff0000ffull;
  x = (x | x << 8) & 0x100f00f00f00f00full;
  x = (x | x << 4) & 0x10c30c30c30c30c3ull;
  x = (x | x << 2) & 0x1249249249249249ull;
  return x;
}

__device__ __forceinline__ unsigned int quantise(float x, float lo, float s,
                                                 float top) {
  // (x - lo) * s in round-to-nearest fp32, clamped to [0, 2^bits - 1]
  // (fmaxf maps NaN, e.g. 0 * inf, to 0), then truncated.
  float v = __fmul_rn(__fsub_rn(x, lo), s);
  return __float2uint_rz(fminf(fmaxf(v, 0.f), top));
}

constexpr int kKeysThreads = 256;

__global__ void __launch_bounds__(kKeysThreads)
keys_kernel(const float4 *__restrict__ pm, long long n,
            unsigned long long *__restrict__ keys, DevCtrl *ctrl, int which,
            int bits) {
  __shared__ unsigned int h[kMaxPasses + 1][256];   // + bits 55..62 of 63-bit keys
  for (int k = threadIdx.x; k < (kMaxPasses + 1) * 256; k += blockDim.x)
    (&h[0][0])[k] = 0u;
  __syncthreads();
  const float4 cube = ctrl->keep.cube[which];
  const float s = ctrl->keep.scale[which];
  const float top = (float)((1u << bits) - 1u);
  const int passes = (3 * bits + 7) / 8;
  const int hists = passes + (bits == kMaxBits ? 1 : 0);
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long base = (long long)blockIdx.x * blockDim.x; base < n;
       base += stride) {
    long long i = base + threadIdx.x;
    bool valid = i < n;
    unsigned long long key = 0;
    if (valid) {
      float4 p = __ldg(pm + i);
      unsigned qx = quantise(p.x, cube.x, s, top);
      unsigned qy = quantise(p.y, cube.y, s, top);
      unsigned qz = quantise(p.z, cube.z, s, top);
      key = spread3(qx) | (spread3(qy) << 1) | (spread3(qz) << 2);
      keys[i] = key;
    }
    // Spatially ordered input makes whole warps share the high digits: add
    // those with one atomic; otherwise every lane adds its own.
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    for (int ps = 0; ps < hists; ++ps) {
      const unsigned d = (unsigned)(key >> (ps < passes ? 8 * ps : kTopShift)) & 255u;
      const unsigned d0 = __shfl_sync(0xffffffffu, d, 0);
      if (__all_sync(0xffffffffu, !valid || d == d0)) {
        if (lane == 0) atomicAdd(&h[ps][d0], (unsigned)__popc(vmask));
      } else if (valid) {
        atomicAdd(&h[ps][d], 1u);
      }
    }
  }
  __syncthreads();
  unsigned int *gh = &ctrl->step.hist[which][0][0];
  for (int k = threadIdx.x; k < passes * 256; k += blockDim.x) {
    unsigned v = (&h[0][0])[k];
    if (v) atomicAdd(gh + k, v);
  }
  if (hists > passes)
    for (int k = threadIdx.x; k < 256; k += blockDim.x) {
      unsigned v = h[passes][k];
      if (v) atomicAdd(&ctrl->step.hist_top[which][k], v);
    }
}

// ---------------------------------------------------------------------------
// One radix pass (8-bit digit at `shift`)
// ---------------------------------------------------------------------------
constexpr unsigned long long kFlagAgg = 1ull << 30;
constexpr unsigned long long kFlagPrefix = 2ull << 30;
constexpr unsigned long long kValMask = (1ull << 30) - 1ull;
constexpr int kLookback = 8;     // predecessor slots read per round trip

__device__ __forceinline__ unsigned long long ld_volatile(
    const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_volatile(unsigned long long *p,
                                            unsigned long long v) {
  asm volatile("st.volatile.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Exclusive block scan of one value per thread (256 threads).
__device__ __forceinline__ unsigned block_excl_scan256(unsigned v,
                                                       unsigned *s_warp,
                                                       unsigned *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[w] = x;
  __syncthreads();
  unsigned off = 0, tot = 0;
#pragma unroll
  for (int k = 0; k < kSortThreads / 32; ++k) {
    unsigned c = s_warp[k];
    if (k < w) off += c;
    tot += c;
  }
  __syncthreads();
  if (total) *total = tot;
  return off + x - v;
}

// ---- TMA bulk copies into shared memory, completion on an mbarrier -------
__device__ __forceinline__ unsigned smem_u32(const void *p) {
  return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned long long *bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long *bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, unsigned parity) {
  unsigned ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
               " selp.u32 %0, 1, 0, p;\n}\n"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_load(void *dst, const void *src, unsigned bytes,
                                          unsigned long long *bar) {
  asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// Rank of this lane's digit d among the warp's keys of the same digit so far:
// lanes holding d (found with eight ballots) count before it in lane order,
// on top of the warp's running count `row[d]`, which the lowest such lane
// then advances.  Keys ranked one item after another keep their order, so
// the sort is stable.
__device__ __forceinline__ unsigned warp_rank(unsigned d, unsigned *row, unsigned lt) {
  unsigned peers = 0xffffffffu;
#pragma unroll
  for (int bt = 0; bt < 8; ++bt) {
    unsigned bit = (d >> bt) & 1u;
    unsigned bal = __ballot_sync(0xffffffffu, bit);
    peers &= bit ? bal : ~bal;
  }
  const unsigned before = row[d];
  const unsigned r = before + __popc(peers & lt);
  __syncwarp();
  if ((peers & lt) == 0u) row[d] = before + __popc(peers);
  __syncwarp();
  return r;
}

constexpr unsigned kTmaWaitLimit = 1u << 26;   // polls; a bulk copy takes microseconds

template <int ITEMS>
struct SortSmem {
  // Two input stages (keys, then indices).  A stage's data is read into
  // registers, then the stage is reused to stage the scatter.
  alignas(128) unsigned long long k[2][kSortThreads * ITEMS];
  alignas(128) unsigned int v[2][kSortThreads * ITEMS];
  unsigned int whist[kSortThreads / 32][256];
  unsigned int dig_excl[256];
  unsigned int glob[256];
  unsigned int gofs[256];
  unsigned int warp[kSortThreads / 32];
  alignas(8) unsigned long long bar[2];
  long long tile[2];
};

// Persistent pass: each block takes tile tickets in order, one ahead, and
// prefetches the next tile with TMA bulk copies while it ranks, looks back
// and scatters the current one.
template <bool kFirst, int ITEMS>
__global__ void __launch_bounds__(kSortThreads, 2)
sort_pass_kernel(const unsigned long long *__restrict__ kin,
                 const unsigned int *__restrict__ vin,
                 unsigned long long *__restrict__ kout,
                 unsigned int *__restrict__ vout, long long n, long long ntiles,
                 int shift, const unsigned int *__restrict__ hist,
                 unsigned int *tile_ctr, unsigned long long *status,
                 unsigned int tag_base, DevCtrl *ctrl,
                 unsigned int spin_limit, const unsigned int *skip_if,
                 unsigned int *decide) {
  extern __shared__ __align__(128) unsigned char sort_smem_raw[];
  constexpr int kTile = kSortThreads * ITEMS;
  SortSmem<ITEMS> &S = *reinterpret_cast<SortSmem<ITEMS> *>(sort_smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  // a regular digit pass has nothing to do once the bucket sort ran
  if (skip_if && *skip_if) return;
  if (decide) {
    // the top-digit pass runs only if every bucket fits one block of the
    // bucket sort; every block finds the same answer, block 0 publishes it
    unsigned mx = __reduce_max_sync(0xffffffffu, hist[tid]);
    if (lane == 0) S.warp[w] = mx;
    __syncthreads();
    mx = 0;
    for (int k = 0; k < kSortThreads / 32; ++k) mx = S.warp[k] > mx ? S.warp[k] : mx;
    __syncthreads();
    const bool fits = mx <= (unsigned)kBucketCap;
    if (blockIdx.x == 0 && tid == 0) *decide = fits ? 1u : 0u;
    if (!fits) return;
  }
  const unsigned long long tag =
      (unsigned long long)(tag_base + ctrl->keep.epoch * 32u) << 32;

  auto issue = [&](int b, long long t) {
    // keys (and indices) of tile t into stage b; sizes rounded up to 16
    // bytes (the buffers are padded past n)
    const long long base = t * kTile;
    const long long cnt = n - base < kTile ? n - base : kTile;
    const unsigned kb = (unsigned)((cnt * 8 + 15) & ~15LL);
    const unsigned vb = kFirst ? 0u : (unsigned)((cnt * 4 + 15) & ~15LL);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_expect_tx(&S.bar[b], kb + vb);
    bulk_load(&S.k[b][0], kin + base, kb, &S.bar[b]);
    if (!kFirst) bulk_load(&S.v[b][0], vin + base, vb, &S.bar[b]);
  };

  if (tid == 0) {
    mbar_init(&S.bar[0]);
    mbar_init(&S.bar[1]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    S.tile[0] = atomicAdd(tile_ctr, 1u);
  }
  // global start of each digit = exclusive scan of this pass's histogram
  S.gofs[tid] = block_excl_scan256(hist[tid], S.warp, nullptr);
  __syncthreads();
  if (tid == 0 && S.tile[0] < ntiles) issue(0, S.tile[0]);
  unsigned parity[2] = {0u, 0u};
  int b = 0;
  const unsigned lt = (1u << lane) - 1u;

  for (;;) {
    __syncthreads();                       // previous tile fully written out
    const long long tile = S.tile[b];
    if (tile >= ntiles) break;
    if (tid == 0) {
      const long long tn = atomicAdd(tile_ctr, 1u);
      S.tile[b ^ 1] = tn;
      if (tn < ntiles) issue(b ^ 1, tn);
    }
    for (int k = tid; k < (kSortThreads / 32) * 256; k += kSortThreads)
      (&S.whist[0][0])[k] = 0u;
    {
      unsigned spins = 0;
      while (!mbar_try_wait(&S.bar[b], parity[b])) {
        if (++spins > kTmaWaitLimit) {
          set_err(ctrl, kErrTimeout);
          break;
        }
      }
      parity[b] ^= 1u;
    }
    const long long base = tile * kTile;
    const int wbase = w * (ITEMS * 32);

    unsigned long long key[ITEMS];
    unsigned int val[ITEMS];
    unsigned int rnk[ITEMS];
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int j = wbase + i * 32 + lane;
      const bool valid = base + j < n;
      key[i] = valid ? S.k[b][j] : ~0ull;
      if (kFirst) val[i] = (unsigned)(base + j);
      else val[i] = valid ? S.v[b][j] : 0u;
    }
    __syncthreads();                       // whist zeroed
#pragma unroll
    for (int i = 0; i < ITEMS; ++i)
      rnk[i] = warp_rank((unsigned)(key[i] >> shift) & 255u, S.whist[w], lt);
    __syncthreads();
    // per digit: offsets of the warps within the tile, and the tile's count
    const unsigned d = tid;
    unsigned run = 0;
#pragma unroll
    for (int k = 0; k < kSortThreads / 32; ++k) {
      unsigned c = S.whist[k][d];
      S.whist[k][d] = run;
      run += c;
    }
    const unsigned total = run;
    // decoupled look-back over the tiles before this one: publish this
    // tile's counts, issue the first window of predecessor reads, and do the
    // block-local scatter (which needs no global offset) while they fly
    unsigned long long *slot = status + tile * 256 + d;
    st_volatile(slot, tag | (tile == 0 ? kFlagPrefix : kFlagAgg) |
                          (unsigned long long)total);
    long long t = tile - 1;
    unsigned long long wv[kLookback];
#pragma unroll
    for (int k = 0; k < kLookback; ++k)
      wv[k] = (t - k >= 0) ? ld_volatile(status + (t - k) * 256 + d) : (tag | kFlagPrefix);
    S.dig_excl[d] = block_excl_scan256(total, S.warp, nullptr);
    __syncthreads();
    // scatter into the stage in digit order
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      unsigned dd = (unsigned)(key[i] >> shift) & 255u;
      unsigned pos = S.dig_excl[dd] + S.whist[w][dd] + rnk[i];
      S.k[b][pos] = key[i];
      S.v[b][pos] = val[i];
    }
    unsigned excl = 0;
    if (tile > 0) {
      unsigned spins = 0;
      bool done = false;
      for (;;) {
        int used = 0;
#pragma unroll
        for (int k = 0; k < kLookback; ++k) {
          if (done || used < k) break;
          const unsigned long long sv = wv[k];
          if ((sv & 0xffffffff00000000ull) != tag) break;   // not published yet
          if (t - k >= 0) excl += (unsigned)(sv & kValMask);
          used = k + 1;
          if ((sv & kFlagPrefix) || t - k <= 0) done = true;
        }
        t -= used;
        if (done || t < 0) break;
        if (used == 0) {
          if (++spins > spin_limit) {
            set_err(ctrl, kErrTimeout);
            break;
          }
          if (spins > 64) __nanosleep(32);
        }
#pragma unroll
        for (int k = 0; k < kLookback; ++k)
          wv[k] = (t - k >= 0) ? ld_volatile(status + (t - k) * 256 + d) : (tag | kFlagPrefix);
      }
      st_volatile(slot, tag | kFlagPrefix |
                            ((unsigned long long)(excl + total) & kValMask));
    }
    S.glob[d] = S.gofs[d] + excl;
    __syncthreads();
    // write out: consecutive slots of one digit go to consecutive addresses
    const long long nvalid = n - base < kTile ? n - base : kTile;
    for (int j = tid; j < nvalid; j += kSortThreads) {
      unsigned long long k = S.k[b][j];
      unsigned dd = (unsigned)(k >> shift) & 255u;
      unsigned long long g = (unsigned long long)S.glob[dd] + (j - S.dig_excl[dd]);
      if (g < (unsigned long long)n) {
        kout[g] = k;
        vout[g] = S.v[b][j];
      }
    }
    b ^= 1;
  }
}

// ---------------------------------------------------------------------------
// Short arrays: the whole sort in one block.  At a few thousand keys each
// tile pass above is one tile and costs its launch and ramp (~8 us, 8 passes
// ~64 us at 4096 keys); here every digit pass ranks, scans and scatters in
// shared memory, one launch for all of them.  Same ranking (warp_rank, keys
// handled in index order), so the same stable permutation.
// ---------------------------------------------------------------------------
constexpr int kSmallSortThreads = 1024;
constexpr int kSmallSortItems = 4;
constexpr int kSmallSortWarps = kSmallSortThreads / 32;
constexpr int kSmallSortN = kSmallSortThreads * kSmallSortItems;   // 4096 keys
constexpr int kSmallRow = 257;   // padded warp-count rows: the per-digit scan
                                 // reads one column without bank conflicts

struct SmallSortSmem {
  alignas(16) unsigned long long k[2][kSmallSortN];
  alignas(16) unsigned int v[2][kSmallSortN];
  unsigned int whist[kSmallSortWarps * kSmallRow];
  unsigned int dig[256];
};

__global__ void __launch_bounds__(kSmallSortThreads, 1)
sort_small_kernel(const unsigned long long *__restrict__ kin, long long n, int passes,
                  unsigned long long *__restrict__ kout, unsigned int *__restrict__ vout) {
  extern __shared__ __align__(128) unsigned char small_sort_raw[];
  SmallSortSmem &S = *reinterpret_cast<SmallSortSmem *>(small_sort_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const int wbase = w * (kSmallSortItems * 32);
  // padding keys (all ones, larger than any 63-bit key) sort after the real ones
  for (int j = tid; j < kSmallSortN; j += kSmallSortThreads) {
    S.k[0][j] = j < n ? kin[j] : ~0ull;
    S.v[0][j] = (unsigned)j;
  }
  int cur = 0;
  for (int p = 0; p < passes; ++p) {
    const int shift = 8 * p;
    for (int k = tid; k < kSmallSortWarps * kSmallRow; k += kSmallSortThreads) S.whist[k] = 0u;
    __syncthreads();                       // counts zeroed (and the first stage loaded)
    unsigned long long key[kSmallSortItems];
    unsigned int val[kSmallSortItems], rnk[kSmallSortItems];
#pragma unroll
    for (int i = 0; i < kSmallSortItems; ++i) {
      const int j = wbase + i * 32 + lane;
      key[i] = S.k[cur][j];
      val[i] = S.v[cur][j];
    }
#pragma unroll
    for (int i = 0; i < kSmallSortItems; ++i)
      rnk[i] = warp_rank((unsigned)(key[i] >> shift) & 255u, &S.whist[w * kSmallRow], lt);
    __syncthreads();
    // per digit, the offsets of the warps (lane = warp) and the digit total:
    // warp w takes digits 8w .. 8w+7
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int d = w * 8 + q;
      const unsigned c = S.whist[lane * kSmallRow + d];
      unsigned x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      S.whist[lane * kSmallRow + d] = x - c;
      if (lane == 31) S.dig[d] = x;
    }
    __syncthreads();
    // start of each digit: exclusive scan of the 256 totals (8 per lane)
    if (w == 0) {
      unsigned t[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { t[q] = S.dig[lane * 8 + q]; sum += t[q]; }
      unsigned x = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      unsigned run = x - sum;
#pragma unroll
      for (int q = 0; q < 8; ++q) { S.dig[lane * 8 + q] = run; run += t[q]; }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kSmallSortItems; ++i) {
      const unsigned d = (unsigned)(key[i] >> shift) & 255u;
      const unsigned pos = S.dig[d] + S.whist[w * kSmallRow + d] + rnk[i];
      S.k[cur ^ 1][pos] = key[i];
      S.v[cur ^ 1][pos] = val[i];
    }
    cur ^= 1;
    __syncthreads();                       // counts read by every warp's scatter
  }
  for (int j = tid; j < n; j += kSmallSortThreads) {
    kout[j] = S.k[cur][j];
    vout[j] = S.v[cur][j];
  }
}

// ---------------------------------------------------------------------------
// Bucket sort: after one pass on the top digit (bits 55..62), the keys sit
// in 256 buckets, each already in index order.  When every bucket holds at
// most kBucketCap keys, one block per bucket sorts its keys on bits 0..54 in
// shared memory (7 digit passes, the same warp-ballot ranking, so the same
// stable order) and writes the final keys, indices and gathered rows -- one
// kernel in place of seven global passes and the gather.
// ---------------------------------------------------------------------------
constexpr int kBucketWarps = kBucketThreads / 32;
constexpr int kBucketPasses = 7;

struct BucketSmem {
  alignas(16) unsigned long long k[kBucketCap];
  alignas(16) unsigned int v[kBucketCap];
  unsigned int whist[kBucketWarps * kSmallRow];
  unsigned int dig[256];
  unsigned int warp[kBucketWarps];
  unsigned int off;
};

// One stable 8-bit digit pass over the bucket in shared memory (key bits
// shift .. shift + 7): warp-ballot ranks, the warps' offsets per digit, the
// digit starts (left in S.dig), the scatter.  Warp-items wholly past `live`
// are padding in every pass (padding keys are the largest and start last,
// so a stable pass leaves them where they are): neither ranked nor moved.
__device__ __forceinline__ void bucket_pass(BucketSmem &S, int shift, int live, int wbase,
                                            int tid, int lane, int w, unsigned lt) {
  for (int k = tid; k < kBucketWarps * kSmallRow; k += kBucketThreads) S.whist[k] = 0u;
  __syncthreads();                         // counts zeroed, keys in place
  unsigned long long key[kBucketItems];
  unsigned int val[kBucketItems], rnk[kBucketItems];
#pragma unroll
  for (int i = 0; i < kBucketItems; ++i) {
    const int j = wbase + i * 32 + lane;
    key[i] = S.k[j];
    val[i] = S.v[j];
  }
#pragma unroll
  for (int i = 0; i < kBucketItems; ++i)
    if (wbase + i * 32 < live)
      rnk[i] = warp_rank((unsigned)(key[i] >> shift) & 255u, &S.whist[w * kSmallRow], lt);
  __syncthreads();                         // every warp holds its keys: the buffer is free
  // per digit (thread d < 256): the warps' offsets and the digit's total
  if (tid < 256) {
    unsigned run = 0;
#pragma unroll
    for (int k = 0; k < kBucketWarps; ++k) {
      const unsigned c = S.whist[k * kSmallRow + tid];
      S.whist[k * kSmallRow + tid] = run;
      run += c;
    }
    S.dig[tid] = run;
  }
  __syncthreads();
  // start of each digit: exclusive scan of the 256 totals (8 per lane)
  if (w == 0) {
    unsigned t[8], sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) { t[q] = S.dig[lane * 8 + q]; sum += t[q]; }
    unsigned x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    unsigned run = x - sum;
#pragma unroll
    for (int q = 0; q < 8; ++q) { S.dig[lane * 8 + q] = run; run += t[q]; }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kBucketItems; ++i) {
    if (wbase + i * 32 < live) {
      const unsigned d = (unsigned)(key[i] >> shift) & 255u;
      const unsigned pos = S.dig[d] + S.whist[w * kSmallRow + d] + rnk[i];
      S.k[pos] = key[i];
      S.v[pos] = val[i];
    }
  }
  __syncthreads();                         // scattered; the counts may be cleared
}

// The bucket's keys share bits 55..62; a first pass on bits 47..54 splits
// it into 256 sub-buckets whose keys share bits 47..62.  When none holds
// more than kSubCap keys, each warp sorts whole sub-buckets on the
// composite (bits 0..46 of the key, position in the sub-bucket) -- unique,
// and in index order for equal keys, since the passes so far are stable and
// the bucket started in index order: by counting up to 32 keys (rank =
// number of smaller composites), by a bitonic network up to 64.  Otherwise
// the bucket takes the seven digit passes on bits 0..55 (LSD from the
// current order, which is stable so far, is still the stable sort).
constexpr int kSubShift = 47;
constexpr int kSubCap = 64;

__device__ __forceinline__ unsigned long long umin64(unsigned long long a, unsigned long long b) {
  return a < b ? a : b;
}
__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a < b ? b : a;
}

// Sort sub-bucket [st, st + sz) (2 <= sz <= kSubCap) of the shared arrays by
// one warp, in place.
__device__ __forceinline__ void sort_sub_bucket(BucketSmem &S, int st, int sz, int lane) {
  constexpr unsigned long long kLow = (1ull << kSubShift) - 1ull;
  unsigned long long a0 = lane < sz ? ((S.k[st + lane] & kLow) << 6) | (unsigned)lane : ~0ull;
  unsigned long long a1 = lane + 32 < sz
                              ? ((S.k[st + lane + 32] & kLow) << 6) | (unsigned)(lane + 32)
                              : ~0ull;
  int r0 = lane, r1 = lane + 32;           // ranks of a0, a1 in the sorted sub-bucket
  if (sz <= 32) {
    int r = 0;
    for (int t = 0; t < sz; ++t) r += __shfl_sync(0xffffffffu, a0, t) < a0 ? 1 : 0;
    r0 = r;
  } else {
    // bitonic network over the 64 slots e = lane (a0) and e = lane + 32 (a1)
#pragma unroll
    for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        if (j == 32) {
          const unsigned long long lo = umin64(a0, a1), hi = umax64(a0, a1);
          a0 = lo;
          a1 = hi;
        } else {
          const unsigned long long v0 = __shfl_xor_sync(0xffffffffu, a0, j);
          const unsigned long long v1 = __shfl_xor_sync(0xffffffffu, a1, j);
          const bool lower = (lane & j) == 0;
          const bool asc0 = (lane & k) == 0, asc1 = ((lane + 32) & k) == 0;
          a0 = (lower == asc0) ? umin64(a0, v0) : umax64(a0, v0);
          a1 = (lower == asc1) ? umin64(a1, v1) : umax64(a1, v1);
        }
      }
    }
  }
  // counting: this lane's entry goes to rank r0; bitonic: slot e holds rank e
  unsigned long long k0 = 0, k1 = 0;
  unsigned v0 = 0, v1 = 0;
  int i0 = -1, i1 = -1;                    // source positions of what this lane writes
  if (sz <= 32) {
    if (lane < sz) i0 = lane;
  } else {
    if (lane < sz) i0 = (int)(a0 & 63ull);
    if (lane + 32 < sz) i1 = (int)(a1 & 63ull);
  }
  if (i0 >= 0) { k0 = S.k[st + i0]; v0 = S.v[st + i0]; }
  if (i1 >= 0) { k1 = S.k[st + i1]; v1 = S.v[st + i1]; }
  __syncwarp();
  if (i0 >= 0) { S.k[st + r0] = k0; S.v[st + r0] = v0; }
  if (i1 >= 0) { S.k[st + r1] = k1; S.v[st + r1] = v1; }
  __syncwarp();
}

__global__ void __launch_bounds__(kBucketThreads, 2)
bucket_sort_kernel(const unsigned long long *__restrict__ kin,
                   const unsigned int *__restrict__ vin, long long n,
                   const unsigned int *__restrict__ hist_top,
                   const unsigned int *__restrict__ go,
                   unsigned long long *__restrict__ kout, unsigned int *__restrict__ vout,
                   const float4 *__restrict__ pm, float4 *__restrict__ sorted) {
  if (!*go) return;
  extern __shared__ __align__(128) unsigned char bucket_raw[];
  BucketSmem &S = *reinterpret_cast<BucketSmem *>(bucket_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const int b = blockIdx.x;
  // this bucket's start: the counts of the buckets before it
  {
    unsigned c = tid < b ? hist_top[tid] : 0u;   // b < 256 <= kBucketThreads
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) S.warp[w] = c;
    __syncthreads();
    if (tid == 0) {
      unsigned o = 0;
      for (int k = 0; k < kBucketWarps; ++k) o += S.warp[k];
      S.off = o;
    }
    __syncthreads();
  }
  const long long off = S.off;
  const int cnt = (int)hist_top[b];
  if (cnt == 0 || off + cnt > n || cnt > kBucketCap) return;
  // padding keys (all ones) sort after the real ones; every load is issued
  // before the first store so the bucket arrives in one memory latency
  {
    unsigned long long kk[kBucketItems];
    unsigned int vv[kBucketItems];
#pragma unroll
    for (int i = 0; i < kBucketItems; ++i) {
      const int j = i * kBucketThreads + tid;
      kk[i] = j < cnt ? kin[off + j] : ~0ull;
      vv[i] = j < cnt ? vin[off + j] : 0u;
    }
#pragma unroll
    for (int i = 0; i < kBucketItems; ++i) {
      S.k[i * kBucketThreads + tid] = kk[i];
      S.v[i * kBucketThreads + tid] = vv[i];
    }
  }
  const int live = (cnt + 31) & ~31;
  const int wbase = w * (kBucketItems * 32);
  bucket_pass(S, kSubShift, live, wbase, tid, lane, w, lt);
  // the largest sub-bucket (real keys only: the padding is digit 255, last)
  if (tid < 256) {
    const int st = (int)S.dig[tid];
    int en = tid < 255 ? (int)S.dig[tid + 1] : live;
    en = en < cnt ? en : cnt;
    const unsigned mx = __reduce_max_sync(0xffffffffu, (unsigned)(en > st ? en - st : 0));
    if (lane == 0) S.warp[w] = mx;
  }
  __syncthreads();
  unsigned mx = 0;
#pragma unroll
  for (int k = 0; k < 256 / 32; ++k) mx = S.warp[k] > mx ? S.warp[k] : mx;
  if (mx <= (unsigned)kSubCap) {
    for (int d = w; d < 256; d += kBucketWarps) {
      const int st = (int)S.dig[d];
      int en = d < 255 ? (int)S.dig[d + 1] : live;
      en = en < cnt ? en : cnt;
      if (en - st >= 2) sort_sub_bucket(S, st, en - st, lane);
    }
    __syncthreads();
  } else {
    // all seven passes, the last on bits 48..55: LSD from the current order
    // (stable so far) is the stable sort
    for (int p = 0; p < kBucketPasses; ++p)
      bucket_pass(S, 8 * p, live, wbase, tid, lane, w, lt);
  }
  // write out: all row loads in flight at once
  {
    unsigned int vv[kBucketItems];
    float4 rr[kBucketItems];
#pragma unroll
    for (int i = 0; i < kBucketItems; ++i) {
      const int j = i * kBucketThreads + tid;
      vv[i] = S.v[j];
      rr[i] = (j < cnt && vv[i] < (unsigned long long)n) ? __ldg(pm + vv[i])
                                                         : make_float4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kBucketItems; ++i) {
      const int j = i * kBucketThreads + tid;
      if (j < cnt) {
        kout[off + j] = S.k[j];
        vout[off + j] = vv[i];
        sorted[off + j] = rr[i];
      }
    }
  }
}

__global__ void gather_kernel(const float4 *__restrict__ in,
                              const unsigned int *__restrict__ perm,
                              long long n, float4 *__restrict__ out,
                              const unsigned int *__restrict__ skip_if) {
  if (skip_if && *skip_if) return;         // the bucket sort wrote the rows
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x; r < n;
       r += stride) {
    unsigned p = perm[r];
    out[r] = (p < (unsigned long long)n) ? __ldg(in + p) : make_float4(0, 0, 0, 0);
  }
}

}  // namespace

cudaError_t launch_bbox(const float4 *pm, long long n, float4 *partials,
                        int max_blocks, DevCtrl *ctrl, int which, int bits,
                        bool bump_epoch, cudaStream_t s) {
  long long want = (n + kBboxThreads * 4 - 1) / (kBboxThreads * 4);
  int blocks = (int)(want < max_blocks ? want : max_blocks);
  if (blocks < 1) blocks = 1;
  {
    const cudaError_t le = launch_k(bbox_kernel, dim3(blocks), dim3(kBboxThreads), 0, s,
                                    pm, n, partials, ctrl, which,
                                               bits, bump_epoch ? 1 : 0);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

cudaError_t launch_keys(const float4 *pm, long long n, unsigned long long *keys,
                        DevCtrl *ctrl, int which, int bits, cudaStream_t s) {
  // Every block merges its shared-memory digit counts (up to 8 x 256) into
  // the global histograms with atomics.  From 2^21 keys on, 8 blocks per SM
  // (more histogram copies to spread the shared atomics, more loads in
  // flight) are faster (keys stage 4M 0.049 -> 0.046 ms, 16M 0.180 ->
  // 0.161); below, the extra merges cost more than they gain (1M 0.021 ->
  // 0.024), so 4.
  long long want = (n + kKeysThreads - 1) / kKeysThreads;
  long long cap = (long long)sm_count() * (n >= (1LL << 21) ? 8 : 4);
  int blocks = (int)(want < cap ? want : cap);
  if (blocks < 1) blocks = 1;
  {
    const cudaError_t le = launch_k(keys_kernel, dim3(blocks), dim3(kKeysThreads), 0, s,
                                    pm, n, keys, ctrl, which, bits);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

// the digit-pass kernels' shared-memory opt-in, once per device
template <int ITEMS>
void pass_attributes() {
  static std::atomic<int> attr[kMaxDevices];
  const size_t smem = sizeof(SortSmem<ITEMS>);
  per_device(attr, [smem] {
    cudaFuncSetAttribute(sort_pass_kernel<true, ITEMS>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaFuncSetAttribute(sort_pass_kernel<false, ITEMS>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return 1;
  });
}

template <int ITEMS>
cudaError_t sort_passes(SortBufs &b, long long n, int passes, DevCtrl *ctrl, int which,
                        unsigned spin_limit, int *final_buf, const unsigned int *skip_if,
                        cudaStream_t s) {
  pass_attributes<ITEMS>();
  const size_t smem = sizeof(SortSmem<ITEMS>);
  constexpr long long kTile = (long long)kSortThreads * ITEMS;
  const long long tiles = (n + kTile - 1) / kTile;
  long long grid = (long long)sm_count() * 2;
  if (grid > tiles) grid = tiles;
  if (grid < 1) grid = 1;
  int cur = 0;
  for (int p = 0; p < passes; ++p) {
    const unsigned *hist = &ctrl->step.hist[which][p][0];
    unsigned *ctr = &ctrl->step.tile_ctr[which][p];
    unsigned tag = (unsigned)(which * 16 + p);
    if (p == 0)
      {
        const cudaError_t le = launch_k(sort_pass_kernel<true, ITEMS>, dim3((unsigned)grid), dim3(kSortThreads), smem, s,
          b.keys[cur], nullptr, b.keys[cur ^ 1], b.idx[cur ^ 1], n, tiles, 8 * p,
          hist, ctr, b.status, tag, ctrl, spin_limit, skip_if, nullptr);
        if (le != cudaSuccess) return le;
      }
    else
      {
        const cudaError_t le = launch_k(sort_pass_kernel<false, ITEMS>, dim3((unsigned)grid), dim3(kSortThreads), smem, s,
          b.keys[cur], b.idx[cur], b.keys[cur ^ 1], b.idx[cur ^ 1], n, tiles, 8 * p,
          hist, ctr, b.status, tag, ctrl, spin_limit, skip_if, nullptr);
        if (le != cudaSuccess) return le;
      }
    cur ^= 1;
  }
  *final_buf = cur;
  return cudaSuccess;
}

// 63-bit keys: the top-digit pass into buffer 1, then the bucket sort back
// into buffer 0 (with the rows gathered); both do nothing unless every
// top-digit bucket fits one block, which the top pass decides on the device.
// (A graph conditional node choosing between this and the digit passes
// measured slower than letting the idle kernels return at once.)
template <int ITEMS>
cudaError_t top_pass(SortBufs &b, long long n, DevCtrl *ctrl, int which,
                     unsigned spin_limit, cudaStream_t s) {
  pass_attributes<ITEMS>();
  const size_t smem = sizeof(SortSmem<ITEMS>);
  constexpr long long kTile = (long long)kSortThreads * ITEMS;
  const long long tiles = (n + kTile - 1) / kTile;
  long long grid = (long long)sm_count() * 2;
  if (grid > tiles) grid = tiles;
  if (grid < 1) grid = 1;
  return launch_k(sort_pass_kernel<true, ITEMS>, dim3((unsigned)grid),
                  dim3(kSortThreads), smem, s, b.keys[0], nullptr, b.keys[1],
                  b.idx[1], n, tiles, kTopShift, &ctrl->step.hist_top[which][0],
                  &ctrl->step.tile_ctr[which][kMaxPasses], b.status,
                  (unsigned)(which * 16 + kMaxPasses), ctrl, spin_limit, nullptr,
                  &ctrl->step.bucket_sort[which]);
}

cudaError_t bucket_sort(SortBufs &b, long long n, DevCtrl *ctrl, int which,
                        const float4 *pm, float4 *sorted, cudaStream_t s) {
  static std::atomic<int> attr[kMaxDevices];
  per_device(attr, [] {
    cudaFuncSetAttribute(bucket_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sizeof(BucketSmem));
    return 1;
  });
  return launch_k(bucket_sort_kernel, dim3(256), dim3(kBucketThreads), sizeof(BucketSmem), s,
                  b.keys[1], b.idx[1], n, &ctrl->step.hist_top[which][0],
                  &ctrl->step.bucket_sort[which], b.keys[0], b.idx[0], pm, sorted);
}

cudaError_t launch_sort(SortBufs &b, long long n, int bits, DevCtrl *ctrl,
                        int which, unsigned spin_limit, const float4 *pm, float4 *sorted,
                        int *final_buf, const unsigned int **gather_skip,
                        cudaStream_t s) {
  const int passes = (3 * bits + 7) / 8;
  *gather_skip = nullptr;
  if (n <= kSmallSortN) {
    static std::atomic<int> attr[kMaxDevices];
    per_device(attr, [] {
      cudaFuncSetAttribute(sort_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sizeof(SmallSortSmem));
      return 1;
    });
    {
      const cudaError_t le = launch_k(sort_small_kernel, dim3(1), dim3(kSmallSortThreads), sizeof(SmallSortSmem), s,
        b.keys[0], n, passes, b.keys[1], b.idx[1]);
      if (le != cudaSuccess) return le;
    }
    *final_buf = 1;
    return cudaGetLastError();
  }
  const long long tiles_small = (n + kSortTile - 1) / kSortTile;
  if (tiles_small > b.cap_tiles) return cudaErrorInvalidValue;
  // 4096-key tiles once 3072-key tiles outnumber the resident blocks
  const bool large = tiles_small > 2LL * sm_count();
  const unsigned *skip = nullptr;
  // with more than 256 * kBucketCap keys some bucket must overflow
  if (bits == kMaxBits && n <= 256LL * kBucketCap) {
    // the bucket path first; the digit passes and the gather then do
    // nothing if it ran (same final buffer either way)
    cudaError_t e = large ? top_pass<kSortItemsLarge>(b, n, ctrl, which, spin_limit, s)
                          : top_pass<kSortItemsSmall>(b, n, ctrl, which, spin_limit, s);
    if (e == cudaSuccess) e = bucket_sort(b, n, ctrl, which, pm, sorted, s);
    if (e != cudaSuccess) return e;
    skip = &ctrl->step.bucket_sort[which];
    *gather_skip = skip;
  }
  if (large)
    return sort_passes<kSortItemsLarge>(b, n, passes, ctrl, which, spin_limit, final_buf, skip, s);
  return sort_passes<kSortItemsSmall>(b, n, passes, ctrl, which, spin_limit, final_buf, skip, s);
}

cudaError_t launch_gather(const float4 *in, const unsigned int *perm,
                          long long n, float4 *out, const unsigned int *skip_if,
                          cudaStream_t s) {
  long long want = (n + 255) / 256;
  long long cap = (long long)sm_count() * 16;
  int blocks = (int)(want < cap ? want : cap);
  if (blocks < 1) blocks = 1;
  {
    const cudaError_t le = launch_k(gather_kernel, dim3(blocks), dim3(256), 0, s,
                                    in, perm, n, out, skip_if);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

}  // namespace bh
