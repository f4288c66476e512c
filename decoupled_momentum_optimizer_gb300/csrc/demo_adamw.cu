// Decoupled AdamW shard step: each replica keeps its own first and second
// moments (never synchronised); the replicas' AdamW directions are averaged
// densely (full synchronisation) and applied with decoupled weight decay.
//
// "DeToNATION: Decoupled Torch Network-Aware Training on Interlinked Online
// Nodes" (Paper-Notes, AAAI 2026), method section, "4. Decoupled AdamW"; the
// ViT-B bandwidth table runs it with full synchronisation.  AdamW itself is
// Loshchilov & Hutter's (bias-corrected moments, decoupled weight decay).
//
// The step is elementwise, so it is a plain grid-stride loop over groups of
// four parameters: per group every replica's g, m, v are read with one
// 16-byte load each (8 bytes for bf16 g), m and v are written back, and theta
// is read and written once.  All accesses are fully coalesced, and all of a
// group's loads are in flight together.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "demo_launch.h"

namespace demo {

constexpr int kAdamThreads = 256;

__device__ __forceinline__ float4 load_grad4(const void* g, long long i, bool bf16) {
  if (!bf16) return reinterpret_cast<const float4*>(g)[i];
  const uint2 w = reinterpret_cast<const uint2*>(g)[i];
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u), __uint_as_float(w.y << 16),
                     __uint_as_float(w.y & 0xffff0000u));
}

struct AdamLane {
  float b1, b2, omb1, omb2, rbc1, rbc2, eps;

  // One replica's moments for one parameter; returns its AdamW direction.
  __device__ __forceinline__ float update(float g, float& m, float& v) const {
    m = __fmaf_rn(b1, m, omb1 * g);
    v = __fmaf_rn(b2, v, omb2 * (g * g));
    return (m * rbc1) / (sqrtf(v * rbc2) + eps);
  }
};

// One group of four parameters.  Every load of the group (each replica's g, m
// and v, and theta) is issued before any store: the stores to m and v could
// alias the next replica's inputs as far as the compiler knows, so a loop that
// stored as it went would wait for memory once per replica.  NR > 0 fixes the
// replica count at compile time; NR = 0 handles any R in batches of four.
template <bool BF16, int NR>
__device__ __forceinline__ void adamw_group(const AdamWParams& p, const AdamLane& a, long long i) {
  constexpr int B = NR > 0 ? NR : 4;
  const float4 th0 = reinterpret_cast<const float4*>(p.theta)[i];
  float4 U = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  const int R = NR > 0 ? NR : p.R;
  for (int r0 = 0; r0 < R; r0 += B) {
    float4 g[B], m[B], v[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (NR > 0 || r0 + b < R) {
        g[b] = load_grad4(p.g[r0 + b], i, BF16);
        m[b] = reinterpret_cast<const float4*>(p.m[r0 + b])[i];
        v[b] = reinterpret_cast<const float4*>(p.v[r0 + b])[i];
      }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (NR > 0 || r0 + b < R) {
        U.x += a.update(g[b].x, m[b].x, v[b].x);
        U.y += a.update(g[b].y, m[b].y, v[b].y);
        U.z += a.update(g[b].z, m[b].z, v[b].z);
        U.w += a.update(g[b].w, m[b].w, v[b].w);
        reinterpret_cast<float4*>(p.m[r0 + b])[i] = m[b];
        reinterpret_cast<float4*>(p.v[r0 + b])[i] = v[b];
      }
    }
  }
  float4 th = th0;
  th.x = __fmaf_rn(-p.lr, __fmaf_rn(p.wd, th.x, U.x * p.rcpR), th.x);
  th.y = __fmaf_rn(-p.lr, __fmaf_rn(p.wd, th.y, U.y * p.rcpR), th.y);
  th.z = __fmaf_rn(-p.lr, __fmaf_rn(p.wd, th.z, U.z * p.rcpR), th.z);
  th.w = __fmaf_rn(-p.lr, __fmaf_rn(p.wd, th.w, U.w * p.rcpR), th.w);
  reinterpret_cast<float4*>(p.theta)[i] = th;
}

template <bool BF16, int NR>
__global__ void __launch_bounds__(kAdamThreads) adamw_kernel(const __grid_constant__ AdamWParams p) {
  const AdamLane a{p.beta1, p.beta2, p.omb1, p.omb2, p.rbc1, p.rbc2, p.eps};
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.n4; i += stride)
    adamw_group<BF16, NR>(p, a, i);
}

template <bool BF16>
static cudaError_t launch_adamw_t(const cudaLaunchConfig_t& cfg, const AdamWParams& p) {
  switch (p.R) {
    case 1: return cudaLaunchKernelEx(&cfg, adamw_kernel<BF16, 1>, p);
    case 2: return cudaLaunchKernelEx(&cfg, adamw_kernel<BF16, 2>, p);
    case 3: return cudaLaunchKernelEx(&cfg, adamw_kernel<BF16, 3>, p);
    case 4: return cudaLaunchKernelEx(&cfg, adamw_kernel<BF16, 4>, p);
    default: return cudaLaunchKernelEx(&cfg, adamw_kernel<BF16, 0>, p);
  }
}

cudaError_t launch_adamw(const AdamWParams& p, bool bf16, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kAdamThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  return bf16 ? launch_adamw_t<true>(cfg, p) : launch_adamw_t<false>(cfg, p);
}

}  // namespace demo
