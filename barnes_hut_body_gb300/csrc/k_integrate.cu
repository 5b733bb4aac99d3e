// Leapfrog time integration around the Barnes-Hut forces.
//
// The GASPHiA tree-code page opens with a 5M-particle galaxy collision run
// as a pure N-body simulation: the gravity of every step is followed by a
// position/velocity update.  The pages print no integrator; this is the
// plainest symplectic one, kick-drift-kick:
//     v += a dt/2;   x += v dt;   a = gravity(x);   v += a dt/2.
// Both updates are streaming kernels (16-byte loads/stores, HBM bound); the
// gravity between them is a full bh_compute, so the tree is rebuilt from the
// drifted positions every step.
#include <cuda_runtime.h>
#include <stdint.h>

#include "bh_internal.h"

namespace bh {

namespace {

// v += a * hk ;  x += v * dt   (masses untouched)
__global__ void kick_drift_kernel(float4 *__restrict__ pm, float4 *__restrict__ vel,
                                  const float4 *__restrict__ acc, long long n,
                                  float hk, float dt) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const float4 a = __ldg(acc + i);
    float4 v = vel[i];
    float4 p = pm[i];
    v.x = fmaf(a.x, hk, v.x);
    v.y = fmaf(a.y, hk, v.y);
    v.z = fmaf(a.z, hk, v.z);
    p.x = fmaf(v.x, dt, p.x);
    p.y = fmaf(v.y, dt, p.y);
    p.z = fmaf(v.z, dt, p.z);
    vel[i] = v;
    pm[i] = p;
  }
}

// v += a * hk
__global__ void kick_kernel(float4 *__restrict__ vel,
                            const float4 *__restrict__ acc, long long n,
                            float hk) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const float4 a = __ldg(acc + i);
    float4 v = vel[i];
    v.x = fmaf(a.x, hk, v.x);
    v.y = fmaf(a.y, hk, v.y);
    v.z = fmaf(a.z, hk, v.z);
    vel[i] = v;
  }
}

int grid_for(long long n, int num_sms) {
  long long want = (n + 255) / 256;
  long long cap = (long long)num_sms * 8;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_kick_drift(float4 *pm, float4 *vel, const float4 *acc,
                              long long n, float hk, float dt, int num_sms,
                              cudaStream_t s) {
  kick_drift_kernel<<<grid_for(n, num_sms), 256, 0, s>>>(pm, vel, acc, n, hk, dt);
  return cudaGetLastError();
}

cudaError_t launch_kick(float4 *vel, const float4 *acc, long long n, float hk,
                        int num_sms, cudaStream_t s) {
  kick_kernel<<<grid_for(n, num_sms), 256, 0, s>>>(vel, acc, n, hk);
  return cudaGetLastError();
}

}  // namespace bh
