// Dense decode: the DiLoCo sync step's receiver, theta <- theta - lr * mean_r(v_r).
//
// "DeToNATION: Decoupled Torch Network-Aware Training on Interlinked Online
// Nodes" (Paper-Notes, AAAI 2026), "2. Replication Schemes" table (DiLoCo: full
// synchronisation every n steps) and "1. FlexDeMo" Algorithm 1 (the parameter update).
//
// On a sync step every replica sends its whole momentum, so Q = Y and the update is
// elementwise.  A grid-stride loop over groups of four parameters reads every
// replica's four values (one 16-byte load for float32, 8 bytes for 16-bit formats,
// the tile's bit-plane words for the ternary format), all of a group's loads before
// any arithmetic, and updates theta with one 16-byte load and store.  The sum runs
// over the replicas in order from 0, then is scaled by 1/R and applied with one FMA,
// exactly as the fused step does, so the two stay bit-identical.
#include "demo_common.cuh"
#include "demo_launch.h"

namespace demo {

constexpr int kDenseThreads = 256;

// The four values of replica payload `v` for parameters 4i .. 4i + 3 (chunk c = 4i / 32,
// positions j .. j + 3 within it), as the receiver decodes them.
__device__ __forceinline__ float4 dense_values(const void* v, int wire, long long i) {
  if (wire == kWireF32) return reinterpret_cast<const float4*>(v)[i];
  if (wire == kWireTernary) {
    const long long e = 4 * i;
    const long long c = e >> 5;
    const int j = static_cast<int>(e & 31);
    const int bit = static_cast<int>(c & 31);
    // words [tile][32 positions][2]: nonzero and negative bit-planes, bit = chunk within the tile
    const uint4 w01 = reinterpret_cast<const uint4*>(v)[((c >> 5) * 32 + j) / 2];
    const uint4 w23 = reinterpret_cast<const uint4*>(v)[((c >> 5) * 32 + j) / 2 + 1];
    auto val = [bit](uint32_t nz, uint32_t ng) {
      return ((nz >> bit) & 1u) ? (((ng >> bit) & 1u) ? -1.0f : 1.0f) : 0.0f;
    };
    return make_float4(val(w01.x, w01.y), val(w01.z, w01.w), val(w23.x, w23.y), val(w23.z, w23.w));
  }
  const uint2 h = reinterpret_cast<const uint2*>(v)[i];
  return make_float4(wire_from_bits16(h.x & 0xffffu, wire), wire_from_bits16(h.x >> 16, wire),
                     wire_from_bits16(h.y & 0xffffu, wire), wire_from_bits16(h.y >> 16, wire));
}

template <int MAXR>
__global__ void __launch_bounds__(kDenseThreads) dense_decode_kernel(const __grid_constant__ DenseParams<MAXR> p) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.n4; i += stride) {
    const float4 th0 = reinterpret_cast<const float4*>(p.theta)[i];
    float4 s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int r0 = 0; r0 < p.R; r0 += 4) {
      float4 v[4];
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (r0 + b < p.R) v[b] = dense_values(p.vals[r0 + b], p.wire, i);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (r0 + b < p.R) {
          s.x += v[b].x;
          s.y += v[b].y;
          s.z += v[b].z;
          s.w += v[b].w;
        }
      }
    }
    float4 th = th0;
    th.x = __fmaf_rn(-p.lr, s.x * p.rcpR, th.x);
    th.y = __fmaf_rn(-p.lr, s.y * p.rcpR, th.y);
    th.z = __fmaf_rn(-p.lr, s.z * p.rcpR, th.z);
    th.w = __fmaf_rn(-p.lr, s.w * p.rcpR, th.w);
    reinterpret_cast<float4*>(p.theta)[i] = th;
  }
}

// DiLoCo between syncs ("2. Replication Schemes" table: the momentum accumulates locally and
// nothing is sent; Algorithm 1's momentum accumulation alone): m_r <- beta m_r + g_r, one FMA per element as
// the tile kernels compute it, so the result is bit-identical to theirs.  Every replica's
// loads for a group of four parameters (in batches of four replicas) are issued before any
// store, so the compiler need not order them against stores that might alias.
__device__ __forceinline__ float4 grad4(const void* g, long long i, bool bf16) {
  if (!bf16) return reinterpret_cast<const float4*>(g)[i];
  const uint2 h = reinterpret_cast<const uint2*>(g)[i];
  return make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xffff0000u), __uint_as_float(h.y << 16),
                     __uint_as_float(h.y & 0xffff0000u));
}

template <int MAXR, bool BF16>
__global__ void __launch_bounds__(kDenseThreads) momentum_kernel(const __grid_constant__ MomentumParams<MAXR> p) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.n4; i += stride) {
    for (int r0 = 0; r0 < p.R; r0 += 4) {
      float4 g[4], m[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (r0 + b < p.R) {
          g[b] = grad4(p.g[r0 + b], i, BF16);
          m[b] = reinterpret_cast<const float4*>(p.m[r0 + b])[i];
        }
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (r0 + b < p.R) {
          float4 x;
          x.x = __fmaf_rn(p.beta, m[b].x, g[b].x);
          x.y = __fmaf_rn(p.beta, m[b].y, g[b].y);
          x.z = __fmaf_rn(p.beta, m[b].z, g[b].z);
          x.w = __fmaf_rn(p.beta, m[b].w, g[b].w);
          reinterpret_cast<float4*>(p.m[r0 + b])[i] = x;
        }
      }
    }
  }
}

cudaError_t launch_momentum_small(const MomentumParams<kSmallReplicas>& p, bool bf16, int grid, cudaStream_t st) {
  if (bf16)
    momentum_kernel<kSmallReplicas, true><<<grid, kDenseThreads, 0, st>>>(p);
  else
    momentum_kernel<kSmallReplicas, false><<<grid, kDenseThreads, 0, st>>>(p);
  return cudaPeekAtLastError();
}

cudaError_t launch_momentum_large(const MomentumParams<kMaxReplicas>& p, bool bf16, int grid, cudaStream_t st) {
  if (bf16)
    momentum_kernel<kMaxReplicas, true><<<grid, kDenseThreads, 0, st>>>(p);
  else
    momentum_kernel<kMaxReplicas, false><<<grid, kDenseThreads, 0, st>>>(p);
  return cudaPeekAtLastError();
}

cudaError_t launch_dense_small(const DenseParams<kSmallReplicas>& p, int grid, cudaStream_t st) {
  dense_decode_kernel<kSmallReplicas><<<grid, kDenseThreads, 0, st>>>(p);
  return cudaPeekAtLastError();
}

cudaError_t launch_dense_large(const DenseParams<kMaxReplicas>& p, int grid, cudaStream_t st) {
  dense_decode_kernel<kMaxReplicas><<<grid, kDenseThreads, 0, st>>>(p);
  return cudaPeekAtLastError();
}

}  // namespace demo
