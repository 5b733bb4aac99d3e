// Brute-force double loop: every source acts on every target.
//
// The GASPHiA tree-code page uses a 暴力双循环 (brute-force double loop) as the
// accuracy and speed reference for its tree walk (section "精度与加速比验证").
//
// GB300 design: a block of 256 threads holds 2 targets per thread; sources
// stream through shared memory in tiles of 1024 rows (coalesced 16-byte
// loads), stored two by two as (x_j, x_j+1, y_j, y_j+1) and (z_j, z_j+1,
// m_j, m_j+1), so one pair of broadcast 16-byte loads feeds Blackwell's
// packed fp32x2 instructions: per pair of sources and target, 13 packed
// operations (3 sub, 3 fma, 3 mul, 3 fma, 1 sub) and 2 reciprocal square
// roots give two interactions.  Sums are kept in fp32 within a tile and in
// fp64 across tiles, which keeps the relative error near 1e-6 at 2^20
// sources.
// When there are too few targets to fill the GPU the sources are split over
// blockIdx.y; every split writes its fp64 partial sums and a second kernel
// adds the splits in a fixed order (deterministic).
// Self mode: a block's 512 targets lie inside one 1024-row source tile; for
// that tile alone the loop compares source and target indices and gives the
// own pair no term at all (its reciprocal distance set to zero), so the
// large m/eps of a small softening never enters a sum that must later
// cancel it.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>
#include <tuple>
#include <utility>

#include "bh_internal.h"

namespace bh {

namespace {

constexpr int kDirThreads = 256;
constexpr int kDirT = 2;
constexpr int kDirTile = 1024;

// One tile's sums for this thread's targets.  kMask: a source row equal to
// a target's own row gets a zero reciprocal distance (no term).
template <bool kMask, bool kEps0>
__device__ __forceinline__ void tile_sum(const ulonglong2 (*tile)[2], int npairs,
                                         const f2 *px, const f2 *py, const f2 *pz,
                                         f2 e2, const long long *ti, long long b,
                                         f2 *fx, f2 *fy, f2 *fz, f2 *fp) {
#pragma unroll 4
  for (int q = 0; q < npairs; ++q) {
    const ulonglong2 a = tile[q][0], c = tile[q][1];    // (xx, yy), (zz, mm)
#pragma unroll
    for (int k = 0; k < kDirT; ++k) {
      const f2 dx = sub2(a.x, px[k]), dy = sub2(a.y, py[k]), dz = sub2(c.x, pz[k]);
      const f2 r2 = fma2(dx, dx, fma2(dy, dy, fma2(dz, dz, e2)));
      float r0, r1;
      upk(r2, r0, r1);
      float i0 = rsqrt_ftz(r0), i1 = rsqrt_ftz(r1);
      if (kEps0) {
        i0 = (r0 > 0.f) ? i0 : 0.f;
        i1 = (r1 > 0.f) ? i1 : 0.f;
      }
      if (kMask) {
        const long long j = b + 2 * q;
        i0 = (ti[k] == j) ? 0.f : i0;
        i1 = (ti[k] == j + 1) ? 0.f : i1;
      }
      const f2 inv = pk(i0, i1);
      const f2 minv = mul2(c.y, inv);
      const f2 minv3 = mul2(minv, mul2(inv, inv));
      fx[k] = fma2(dx, minv3, fx[k]);
      fy[k] = fma2(dy, minv3, fy[k]);
      fz[k] = fma2(dz, minv3, fz[k]);
      fp[k] = sub2(fp[k], minv);
    }
  }
}

template <bool kSelf, bool kEps0>
__global__ void __launch_bounds__(kDirThreads)
direct_kernel(const float4 *__restrict__ src, long long n,
              const float4 *__restrict__ tgt, long long m, float eps2,
              long long chunk, double *__restrict__ partial) {
  __shared__ ulonglong2 tile[kDirTile / 2][2];   // source pairs
  const long long tbase = (long long)blockIdx.x * (kDirThreads * kDirT);
  const long long s0 = (long long)blockIdx.y * chunk;
  long long s1 = s0 + chunk;
  if (s1 > n) s1 = n;
  f2 px[kDirT], py[kDirT], pz[kDirT];   // targets, duplicated in both halves
  long long ti[kDirT];
  double acc[kDirT][4];
  const f2 e2 = pk(eps2, eps2);
#pragma unroll
  for (int k = 0; k < kDirT; ++k) {
    ti[k] = tbase + k * kDirThreads + threadIdx.x;
    float4 p = __ldg(tgt + (ti[k] < m ? ti[k] : 0));
    px[k] = pk(p.x, p.x); py[k] = pk(p.y, p.y); pz[k] = pk(p.z, p.z);
    acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = 0.0;
  }
  for (long long b = s0; b < s1; b += kDirTile) {
    const int cnt = (int)((s1 - b) < kDirTile ? (s1 - b) : kDirTile);
    const int npairs = (cnt + 1) / 2;
    __syncthreads();
    for (int q = threadIdx.x; q < npairs; q += kDirThreads) {
      // an odd tile's last pair is completed by a massless source at the
      // first one's position (it adds exactly 0)
      const float4 u = __ldg(src + b + 2 * q);
      float4 v = 2 * q + 1 < cnt ? __ldg(src + b + 2 * q + 1) : make_float4(u.x, u.y, u.z, 0.f);
      tile[q][0] = make_ulonglong2(pk(u.x, v.x), pk(u.y, v.y));
      tile[q][1] = make_ulonglong2(pk(u.z, v.z), pk(u.w, v.w));
    }
    __syncthreads();
    f2 fx[kDirT], fy[kDirT], fz[kDirT], fp[kDirT];
#pragma unroll
    for (int k = 0; k < kDirT; ++k) fx[k] = fy[k] = fz[k] = fp[k] = 0ull;
    // the tile holding this block's own rows (self mode, eps > 0)
    const bool own = kSelf && !kEps0 && tbase < b + cnt &&
                     b < tbase + kDirThreads * kDirT;
    if (own)
      tile_sum<true, kEps0>(tile, npairs, px, py, pz, e2, ti, b, fx, fy, fz, fp);
    else
      tile_sum<false, kEps0>(tile, npairs, px, py, pz, e2, ti, b, fx, fy, fz, fp);
#pragma unroll
    for (int k = 0; k < kDirT; ++k) {
      float x0, x1, y0, y1, z0, z1, p0, p1;
      upk(fx[k], x0, x1);
      upk(fy[k], y0, y1);
      upk(fz[k], z0, z1);
      upk(fp[k], p0, p1);
      acc[k][0] += x0 + x1; acc[k][1] += y0 + y1;
      acc[k][2] += z0 + z1; acc[k][3] += p0 + p1;
    }
  }
#pragma unroll
  for (int k = 0; k < kDirT; ++k) {
    if (ti[k] >= m) continue;
    double *o = partial + ((long long)blockIdx.y * m + ti[k]) * 4;
    o[0] = acc[k][0]; o[1] = acc[k][1]; o[2] = acc[k][2]; o[3] = acc[k][3];
  }
}

__global__ void direct_finish_kernel(const double *__restrict__ partial,
                                     int splits, long long m, float G,
                                     float4 *__restrict__ out) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < m;
       t += stride) {
    double s[4] = {0.0, 0.0, 0.0, 0.0};
    for (int y = 0; y < splits; ++y) {
      const double *p = partial + ((long long)y * m + t) * 4;
      s[0] += p[0]; s[1] += p[1]; s[2] += p[2]; s[3] += p[3];
    }
    out[t] = make_float4((float)(G * s[0]), (float)(G * s[1]),
                         (float)(G * s[2]), (float)(G * s[3]));
  }
}

// Launch with the status of this launch alone (cudaLaunchKernel returns it),
// instead of reading the thread's last error, which may belong to an
// earlier, unrelated call.
template <typename... KArgs, size_t... I>
cudaError_t launch_tuple(void (*k)(KArgs...), dim3 g, dim3 b, cudaStream_t s,
                         std::tuple<KArgs...> &t, std::index_sequence<I...>) {
  void *p[] = {(void *)&std::get<I>(t)...};
  return cudaLaunchKernel((const void *)k, g, b, p, 0, s);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_checked(void (*k)(KArgs...), dim3 g, dim3 b, cudaStream_t s,
                           Args... args) {
  std::tuple<KArgs...> t(args...);
  return launch_tuple(k, g, b, s, t, std::index_sequence_for<KArgs...>{});
}

}  // namespace

cudaError_t launch_direct(const float4 *src, long long n, const float4 *tgt,
                          long long m, bool self_mode, float eps, float G,
                          double *partial, long long partial_cap, float4 *out,
                          int num_sms, cudaStream_t s) {
  if (m <= 0) return cudaSuccess;
  const long long bx = (m + kDirThreads * kDirT - 1) / (kDirThreads * kDirT);
  long long splits = (4LL * num_sms + bx - 1) / bx;
  long long max_by_src = (n + kDirTile - 1) / kDirTile;
  if (splits > max_by_src) splits = max_by_src;
  if (splits > 64) splits = 64;
  while (splits > 1 && splits * m * 4 > partial_cap) --splits;
  if (splits < 1) splits = 1;
  if (m * 4 > partial_cap) return cudaErrorInvalidValue;
  long long chunk = (n + splits - 1) / splits;
  chunk = ((chunk + kDirTile - 1) / kDirTile) * kDirTile;
  splits = (n + chunk - 1) / chunk;
  if (splits < 1) splits = 1;
  const float eps2 = eps * eps;
  dim3 grid((unsigned)bx, (unsigned)splits);
  const bool eps0 = eps2 == 0.f;
  auto k = self_mode ? (eps0 ? direct_kernel<true, true> : direct_kernel<true, false>)
                     : (eps0 ? direct_kernel<false, true> : direct_kernel<false, false>);
  cudaError_t e = launch_checked(k, grid, dim3(kDirThreads), s, src, n, tgt, m, eps2,
                                 chunk, partial);
  if (e != cudaSuccess) return e;
  long long fb = (m + 255) / 256;
  if (fb > (long long)num_sms * 16) fb = (long long)num_sms * 16;
  return launch_checked(direct_finish_kernel, dim3((unsigned)fb), dim3(256), s,
                        (const double *)partial, (int)splits, m, G, out);
}

// ---------------------------------------------------------------------------
// Allocation-free entry point
//
// bh_direct_static serves callers that cannot allocate device memory when
// they need forces: code running while a CUDA graph is being captured
// (cudaMalloc is not allowed there), loops that must never synchronise the
// device (cudaMalloc and cudaFree can), and host programs that hand all GPU
// memory to their own pool at start-up.  It needs no context: its only
// scratch -- the fp64 partial sums of the source splits -- lives in a
// file-scope device array that every GPU loading the library keeps until
// the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr long long kStaticScratchDoubles = 1LL << 20;   // 8 MiB
constexpr int kStaticMaxDevices = 64;

static __device__ __align__(256) double g_static_partial[kStaticScratchDoubles];

std::mutex g_static_mu;
double *g_static_addr[kStaticMaxDevices] = {};
int g_static_sms[kStaticMaxDevices] = {};

}  // namespace

}  // namespace bh

extern "C" int bh_direct_static(const float *pos_mass, size_t n,
                                const float *targets, size_t m, float G,
                                float eps, float *acc_pot, void *stream) {
  using namespace bh;
  const bool self = targets == nullptr;
  const long long N = (long long)n, M = self ? N : (long long)m;
  auto bad_rows = [](const float *p, long long rows) {
    return rows > 0 && (p == nullptr || ((uintptr_t)p & 15u) != 0);
  };
  if (bad_rows(pos_mass, N) || (!self && bad_rows(targets, M)) || bad_rows(acc_pot, M))
    return BH_EINVAL;
  if (!isfinite(G) || !(eps >= 0.f) || !isfinite(eps)) return BH_EINVAL;
  if (M == 0) return BH_OK;
  if (4 * M > kStaticScratchDoubles) return BH_EINVAL;   // > 262,144 targets
  cudaStream_t s = (cudaStream_t)stream;
  if (N == 0)
    return cudaMemsetAsync(acc_pot, 0, sizeof(float4) * (size_t)M, s) == cudaSuccess
               ? BH_OK : BH_ECUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStaticMaxDevices)
    return BH_ECUDA;
  double *scratch = nullptr;
  int sms = 1;
  {
    // Set-up, once per device with that device current: the host name of
    // g_static_partial is only a stand-in, the kernels need its device
    // address.  The first call on a device does this, so it should come
    // before any stream capture.
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_static_partial) != cudaSuccess || !p)
        return BH_ECUDA;
      int c = 0;
      if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return BH_ECUDA;
      g_static_sms[dev] = c > 0 ? c : 1;
      g_static_addr[dev] = static_cast<double *>(p);
    }
    scratch = g_static_addr[dev];
    sms = g_static_sms[dev];
  }
  cudaError_t e = launch_direct(reinterpret_cast<const float4 *>(pos_mass), N,
                                reinterpret_cast<const float4 *>(self ? pos_mass : targets),
                                M, self, eps, G, scratch, kStaticScratchDoubles,
                                reinterpret_cast<float4 *>(acc_pot), sms, s);
  return e == cudaSuccess ? BH_OK : BH_ECUDA;
}

