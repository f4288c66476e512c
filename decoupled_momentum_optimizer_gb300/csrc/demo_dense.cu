// Dense decode: the DiLoCo sync step's receiver, theta <- theta - lr * mean_r(v_r).
//
// "DeToNATION: Decoupled Torch Network-Aware Training on Interlinked Online
// Nodes" (Paper-Notes, AAAI 2026), "2. Replication Schemes" table (DiLoCo: full
// synchronisation every n steps) and "1. FlexDeMo" Algorithm 1 (the parameter update).
//
// On a sync step every replica sends its whole momentum, so Q = Y and the update is
// elementwise.  The sum runs over the replicas in order from 0, then is scaled by 1/R and
// applied with one FMA, exactly as the fused step does, so the two stay bit-identical.
//
// All kernels here are grid-stride loops (over groups of four parameters per lane, or over
// tiles per warp for the ternary format), launched with as many CTAs as are resident at once:
// one wave, with no CTAs that start late and set the end (the float32 decode at 2^26, R = 2:
// 164 -> 154 us against eight CTAs per SM).  Each lane issues all its loads of a batch of
// replicas before any arithmetic or store.
#include "demo_common.cuh"
#include "demo_launch.h"

namespace demo {

constexpr int kDenseThreads = 256;
constexpr int kDenseWarps = kDenseThreads / 32;

// One wave of resident CTAs, or one CTA per eight units of work where that is at most two
// waves: on a small shard every lane then runs a single iteration, and the CTAs of the second
// wave start as soon as the first ones end (momentum pass, 2^20 parameters, 64 replicas:
// 138 us with one wave of two iterations per lane, 131 us with this).
int one_wave(int per_sm, int sms, long long units) {
  const long long want = (units + kDenseWarps - 1) / kDenseWarps;
  const long long wave = static_cast<long long>(per_sm) * sms;
  const long long g = want <= 2 * wave ? want : wave;
  return static_cast<int>(g > 0 ? g : 1);
}

// The four values of replica payload `v` for parameters 4i .. 4i + 3 (float32 or 16-bit
// formats): one 16-byte or 8-byte load.
__device__ __forceinline__ float4 dense_values(const void* v, int wire, long long i) {
  if (wire == kWireF32) return reinterpret_cast<const float4*>(v)[i];
  const uint2 h = reinterpret_cast<const uint2*>(v)[i];
  return make_float4(wire_from_bits16(h.x & 0xffffu, wire), wire_from_bits16(h.x >> 16, wire),
                     wire_from_bits16(h.y & 0xffffu, wire), wire_from_bits16(h.y >> 16, wire));
}

// Float32 and 16-bit payloads: a grid-stride loop over groups of four parameters, each lane's
// theta load and its batch of replicas' payload loads issued before any arithmetic.  (Two or
// four groups per lane, which hold more bytes in flight but need more registers, measured
// slower: bfloat16 payloads, R = 2, 2^26 parameters: 125 us with one group, 236 with two.)
template <int MAXR>
__global__ void __launch_bounds__(kDenseThreads) dense_decode_kernel(const __grid_constant__ DenseParams<MAXR> p) {
  constexpr int kBatch = 4;  // replicas whose loads are in flight together
  const long long stride = static_cast<long long>(gridDim.x) * kDenseThreads;
  float4* theta = reinterpret_cast<float4*>(p.theta);
  for (long long i = static_cast<long long>(blockIdx.x) * kDenseThreads + threadIdx.x; i < p.n4; i += stride) {
    const float4 th0 = theta[i];
    float4 s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int r0 = 0; r0 < p.R; r0 += kBatch) {
      float4 v[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
        if (r0 + b < p.R) v[b] = dense_values(p.vals[r0 + b], p.wire, i);
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
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
    theta[i] = th;
  }
}

// Ternary payloads (bit-planes over the 32 chunks of a tile, two words per position: nonzero,
// then negative).  A warp's unit is one tile with lane = position: each lane reads its
// position's two words once per replica (a coalesced 256-byte row per warp) and theta moves in
// 32 coalesced 128-byte rows, one per chunk.
//
// The per-chunk sums of +1, -1 and 0 are counted with SIMD-within-a-word arithmetic, the
// words' chunk bits sorted by chunk mod 4: field word h holds, in its nibble j, the count of
// chunk 4j + h.  A replica adds its positive bits and subtracts its negative bits (masked to
// the low bit of each nibble); nibbles start at 8, so over up to seven replicas none leaves
// 1 .. 15 and nothing carries or borrows between them.  Every seven replicas the nibbles are
// added into byte counters (even and odd nibbles apart) that start at 128 and stay within
// 128 +- R (R <= 64).  The float sum of the same values in replica order is exactly the
// integer count, so theta is bit-identical to the sum taken value by value.
template <int MAXR>
__global__ void __launch_bounds__(kDenseThreads) dense_ternary_kernel(const __grid_constant__ DenseParams<MAXR> p) {
  constexpr int kGroup = 7;  // replicas per nibble pass
  constexpr uint32_t kLow = 0x11111111u;
  const int lane = threadIdx.x & 31;
  const long long nc = p.n4 / 8;
  const long long ntiles = (nc + 31) / 32;
  const long long nwarps = static_cast<long long>(gridDim.x) * kDenseWarps;
  for (long long t = static_cast<long long>(blockIdx.x) * kDenseWarps + (threadIdx.x >> 5); t < ntiles; t += nwarps) {
    const long long c0 = t * 32;
    const int rows = nc - c0 < 32 ? static_cast<int>(nc - c0) : 32;
    float* th_row = p.theta + c0 * 32 + lane;
    float th[32];
#pragma unroll
    for (int cc = 0; cc < 32; ++cc) th[cc] = cc < rows ? th_row[cc * 32] : 0.0f;
    uint32_t even[4], odd[4];  // byte b: the count of chunk 4 (2b) + h, resp. 4 (2b + 1) + h
#pragma unroll
    for (int h = 0; h < 4; ++h) even[h] = odd[h] = 0x80808080u;
    for (int r0 = 0; r0 < p.R; r0 += kGroup) {
      uint2 w[kGroup];
#pragma unroll
      for (int b = 0; b < kGroup; ++b)
        if (r0 + b < p.R) w[b] = reinterpret_cast<const uint2*>(p.vals[r0 + b])[t * 32 + lane];
      uint32_t f[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) f[h] = 0x88888888u;
#pragma unroll
      for (int b = 0; b < kGroup; ++b) {
        if (r0 + b < p.R) {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const uint32_t nz = w[b].x >> h, ng = w[b].y >> h;
            f[h] += (nz & ~ng & kLow) - (nz & ng & kLow);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        even[h] += (f[h] & 0x0f0f0f0fu) - 0x08080808u;
        odd[h] += ((f[h] >> 4) & 0x0f0f0f0fu) - 0x08080808u;
      }
    }
#pragma unroll
    for (int cc = 0; cc < 32; ++cc) {
      if (cc < rows) {
        const int j = cc >> 2;
        const uint32_t word = (j & 1) ? odd[cc & 3] : even[cc & 3];
        const int cnt = static_cast<int>((word >> (8 * (j >> 1))) & 0xffu) - 128;
        th_row[cc * 32] = __fmaf_rn(-p.lr, static_cast<float>(cnt) * p.rcpR, th[cc]);
      }
    }
  }
}

// DiLoCo between syncs ("2. Replication Schemes" table: the momentum accumulates locally and
// nothing is sent; Algorithm 1's momentum accumulation alone): m_r <- beta m_r + g_r, one FMA
// per element as the tile kernels compute it, so the result is bit-identical to theirs.  A
// grid-stride loop over groups of four parameters, G groups (one grid stride apart) per lane
// and iteration; every load of a batch of replicas is issued before any store, so the compiler
// need not order them against stores that might alias.
__device__ __forceinline__ float4 grad4(const void* g, long long i, bool bf16) {
  if (!bf16) return reinterpret_cast<const float4*>(g)[i];
  const uint2 h = reinterpret_cast<const uint2*>(g)[i];
  return make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xffff0000u), __uint_as_float(h.y << 16),
                     __uint_as_float(h.y & 0xffff0000u));
}

template <int MAXR, bool BF16, int G>
__global__ void __launch_bounds__(kDenseThreads) momentum_kernel(const __grid_constant__ MomentumParams<MAXR> p) {
  constexpr int kBatch = G >= 2 ? 2 : 4;
  const long long stride = static_cast<long long>(gridDim.x) * kDenseThreads;
  for (long long i0 = static_cast<long long>(blockIdx.x) * kDenseThreads + threadIdx.x; i0 < p.n4; i0 += G * stride) {
    for (int r0 = 0; r0 < p.R; r0 += kBatch) {
      float4 g[kBatch][G], m[kBatch][G];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
#pragma unroll
        for (int q = 0; q < G; ++q) {
          const long long i = i0 + q * stride;
          if (r0 + b < p.R && (q == 0 || i < p.n4)) {
            g[b][q] = grad4(p.g[r0 + b], i, BF16);
            m[b][q] = reinterpret_cast<const float4*>(p.m[r0 + b])[i];
          }
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
#pragma unroll
        for (int q = 0; q < G; ++q) {
          const long long i = i0 + q * stride;
          if (r0 + b < p.R && (q == 0 || i < p.n4)) {
            float4 x;
            x.x = __fmaf_rn(p.beta, m[b][q].x, g[b][q].x);
            x.y = __fmaf_rn(p.beta, m[b][q].y, g[b][q].y);
            x.z = __fmaf_rn(p.beta, m[b][q].z, g[b][q].z);
            x.w = __fmaf_rn(p.beta, m[b][q].w, g[b][q].w);
            reinterpret_cast<float4*>(p.m[r0 + b])[i] = x;
          }
        }
      }
    }
  }
}

// Groups of four parameters per lane and iteration of the momentum pass: two for a single
// replica with bfloat16 gradients, whose one group holds too few bytes in flight (2^26
// parameters: 120 -> 105 us); with float32 gradients one group measured faster (122 us against
// 126 with two), and for R >= 2 the batch of replicas already keeps enough in flight.
int momentum_rows(int R, bool bf16) { return bf16 && R == 1 ? 2 : 1; }

// Resident CTAs per SM of each instantiation at kDenseThreads threads, found once when the
// library is initialised rather than at launch (a launch may be inside a stream capture).
template <int MAXR>
int dense_per_sm = 1;
template <int MAXR>
int ternary_per_sm = 1;
template <int MAXR, bool BF16, int G>
int momentum_per_sm = 1;

template <typename Kernel>
cudaError_t ctas_per_sm(Kernel kernel, int* out) {
  int b = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kDenseThreads, 0);
  if (e == cudaSuccess) *out = b > 0 ? b : 1;
  return e;
}

template <int MAXR>
cudaError_t prepare_dense_replicas() {
  const cudaError_t e[] = {
      ctas_per_sm(dense_decode_kernel<MAXR>, &dense_per_sm<MAXR>),
      ctas_per_sm(dense_ternary_kernel<MAXR>, &ternary_per_sm<MAXR>),
      ctas_per_sm(momentum_kernel<MAXR, false, 1>, &momentum_per_sm<MAXR, false, 1>),
      ctas_per_sm(momentum_kernel<MAXR, false, 2>, &momentum_per_sm<MAXR, false, 2>),
      ctas_per_sm(momentum_kernel<MAXR, true, 1>, &momentum_per_sm<MAXR, true, 1>),
      ctas_per_sm(momentum_kernel<MAXR, true, 2>, &momentum_per_sm<MAXR, true, 2>),
  };
  for (cudaError_t x : e)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

template <int MAXR>
cudaError_t launch_dense(const DenseParams<MAXR>& p, int sms, cudaStream_t st) {
  if (p.wire == kWireTernary) {
    const int grid = one_wave(ternary_per_sm<MAXR>, sms, (p.n4 / 8 + 31) / 32);
    dense_ternary_kernel<MAXR><<<grid, kDenseThreads, 0, st>>>(p);
  } else {
    const int grid = one_wave(dense_per_sm<MAXR>, sms, (p.n4 + 31) / 32);
    dense_decode_kernel<MAXR><<<grid, kDenseThreads, 0, st>>>(p);
  }
  return cudaPeekAtLastError();
}

template <int MAXR, bool BF16, int G>
cudaError_t launch_momentum_rows(const MomentumParams<MAXR>& p, int sms, cudaStream_t st) {
  const int grid = one_wave(momentum_per_sm<MAXR, BF16, G>, sms, (p.n4 + 32 * G - 1) / (32 * G));
  momentum_kernel<MAXR, BF16, G><<<grid, kDenseThreads, 0, st>>>(p);
  return cudaPeekAtLastError();
}

template <int MAXR>
cudaError_t launch_momentum(const MomentumParams<MAXR>& p, bool bf16, int sms, cudaStream_t st) {
  const bool two = momentum_rows(p.R, bf16) == 2;
  if (bf16)
    return two ? launch_momentum_rows<MAXR, true, 2>(p, sms, st) : launch_momentum_rows<MAXR, true, 1>(p, sms, st);
  return two ? launch_momentum_rows<MAXR, false, 2>(p, sms, st) : launch_momentum_rows<MAXR, false, 1>(p, sms, st);
}

cudaError_t prepare_dense_kernels() {
  // The table is the same on every device the library accepts (one architecture): it is filled
  // once, so a later device's initialisation never writes it while launches read it.  The
  // caller (demo_init) holds the library's lock.
  static bool filled = false;
  if (filled) return cudaSuccess;
  cudaError_t e = prepare_dense_replicas<kSmallReplicas>();
  if (e == cudaSuccess) e = prepare_dense_replicas<kMaxReplicas>();
  if (e == cudaSuccess) filled = true;
  return e;
}

cudaError_t launch_momentum_small(const MomentumParams<kSmallReplicas>& p, bool bf16, int sms, cudaStream_t st) {
  return launch_momentum(p, bf16, sms, st);
}

cudaError_t launch_momentum_large(const MomentumParams<kMaxReplicas>& p, bool bf16, int sms, cudaStream_t st) {
  return launch_momentum(p, bf16, sms, st);
}

cudaError_t launch_dense_small(const DenseParams<kSmallReplicas>& p, int sms, cudaStream_t st) {
  return launch_dense(p, sms, st);
}

cudaError_t launch_dense_large(const DenseParams<kMaxReplicas>& p, int sms, cudaStream_t st) {
  return launch_dense(p, sms, st);
}

}  // namespace demo
