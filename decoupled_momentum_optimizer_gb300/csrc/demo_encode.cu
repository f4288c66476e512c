// Split-path encode: one replica's Algorithm 1 steps 3-5 and its payload (the
// buffer the real system would hand to the inter-node all_gather / all-reduce).
//
// "DeToNATION: Decoupled Torch Network-Aware Training on Interlinked Online
// Nodes" (Paper-Notes, AAAI 2026), method section, "1. FlexDeMo" Algorithm 1
// steps 3-5, "2. Replication Schemes" table, "3. Sign function" subsection.
//
// Same warp/tile organisation as the fused step: per warp, tiles of 32 chunks
// stream through a two-slot TMA ring; each lane encodes its chunk in registers;
// the new momentum leaves through the tile's own slot with coalesced stores and
// the slot is refilled at once.  The payload of chunk c is written to
// vals[c*k .. c*k+k) (and idx for DeMo) by the lane that owns c, as one vector
// store when k is 1, 2, 4 or 8.
#include "demo_common.cuh"
#include "demo_params.h"

namespace demo {

struct alignas(1024) EncWarpSmem {
  float gbuf[2][1024];  // g tile, then a [i][lane] scratch column per lane
  float mbuf[2][1024];  // m tile, then the new m on its way out
};

constexpr int kEncWarps = kStepWarps;
constexpr int kEncThreads = kEncWarps * 32;
constexpr size_t kEncSmem = 1024 + kEncWarps * sizeof(EncWarpSmem) + kEncWarps * 16;

// Store k payload values (and index bytes) of one chunk; k in {1, 2, 4, 8} uses one vector store each.
__device__ __forceinline__ void store_payload(float* vrow, uint8_t* irow, const float (&pv)[8], uint32_t ilo,
                                              uint32_t ihi, int k) {
  switch (k) {
    case 1:
      vrow[0] = pv[0];
      if (irow) irow[0] = static_cast<uint8_t>(ilo);
      break;
    case 2:
      *reinterpret_cast<float2*>(vrow) = make_float2(pv[0], pv[1]);
      if (irow) *reinterpret_cast<uint16_t*>(irow) = static_cast<uint16_t>(ilo);
      break;
    case 4:
      *reinterpret_cast<float4*>(vrow) = make_float4(pv[0], pv[1], pv[2], pv[3]);
      if (irow) *reinterpret_cast<uint32_t*>(irow) = ilo;
      break;
    default:  // 8
      reinterpret_cast<float4*>(vrow)[0] = make_float4(pv[0], pv[1], pv[2], pv[3]);
      reinterpret_cast<float4*>(vrow)[1] = make_float4(pv[4], pv[5], pv[6], pv[7]);
      if (irow) *reinterpret_cast<uint2*>(irow) = make_uint2(ilo, ihi);
      break;
  }
}

__device__ __forceinline__ bool vector_k(int k) { return k == 1 || k == 2 || k == 4 || k == 8; }

template <int MODE, bool BF16>
__global__ void __launch_bounds__(kEncThreads, 1) encode_kernel(const __grid_constant__ EncodeParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  EncWarpSmem& ws = reinterpret_cast<EncWarpSmem*>(base)[warp];
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kEncWarps * sizeof(EncWarpSmem)) + 2 * warp;

  const long long gw = static_cast<long long>(blockIdx.x) * kEncWarps + warp;
  const long long TW = static_cast<long long>(gridDim.x) * kEncWarps;
  if (gw >= p.ntiles) return;
  const long long nitems = (p.ntiles - 1 - gw) / TW + 1;

  if (lane == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto issue = [&](long long item) {
    if (item >= nitems) return;
    const int s = static_cast<int>(item & 1);
    const int y = static_cast<int>((gw + item * TW) * 32);
    mbar_expect_tx(&bars[s], (BF16 ? kTileBytesBF16 : kTileBytesF32) + kTileBytesF32);
    tma_load_2d(ws.gbuf[s], &p.g, &bars[s], 0, y);
    tma_load_2d(ws.mbuf[s], &p.m, &bars[s], 0, y);
  };
  if (lane == 0) {
    issue(0);
    issue(1);
  }

  for (long long item = 0; item < nitems; ++item) {
    const int s = static_cast<int>(item & 1);
    const uint32_t par = static_cast<uint32_t>((item >> 1) & 1);
    const long long row0 = (gw + item * TW) * 32;
    const long long c = row0 + lane;
    const bool valid = c < p.nc;

    const bool ok = mbar_wait_bounded(&bars[s], par);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) {
        atomicOr(p.fault, kFaultLoadTimeout);
        for (long long it = item; it < item + 2 && it < nitems; ++it)
          mbar_wait_bounded(&bars[it & 1], static_cast<uint32_t>((it >> 1) & 1));
      }
      __syncwarp();
      return;
    }

    float x[32], gv[32];
    load_row_grad<BF16>(ws.gbuf[s], lane, gv);
    load_row_f32(ws.mbuf[s], lane, x);
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __fmaf_rn(p.beta, x[i], gv[i]);
    __syncwarp();  // every lane has read its g row: the g tile becomes a scratch
    float* scratch = ws.gbuf[s];

    if constexpr (MODE == kModeDemo) {
      float X[32], Xs[32];
      dct32_forward(x, X);
      const uint32_t M = topk_select(X, p.k, Xs);
#pragma unroll
      for (int u = 0; u < 32; ++u) scratch[u * 32 + lane] = Xs[u];
      float* vrow = p.vals + c * p.k;
      uint8_t* irow = p.idx + c * p.k;
      uint32_t mm = M;
      if (vector_k(p.k)) {
        float pv[8];
        uint32_t ilo = 0, ihi = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          pv[j] = 0.0f;
          if (j < p.k) {
            const int u = __ffs(mm) - 1;
            mm &= mm - 1;
            const float v = scratch[u * 32 + lane];
            pv[j] = p.sign ? sign3(v) : v;
            if (j < 4) ilo |= static_cast<uint32_t>(u) << (8 * j);
            else ihi |= static_cast<uint32_t>(u) << (8 * (j - 4));
          }
        }
        if (valid) store_payload(vrow, irow, pv, ilo, ihi, p.k);
      } else {
        for (int j = 0; j < p.k; ++j) {
          const int u = __ffs(mm) - 1;
          mm &= mm - 1;
          float v = scratch[u * 32 + lane];
          if (p.sign) v = sign3(v);
          if (valid) {
            vrow[j] = v;
            irow[j] = static_cast<uint8_t>(u);
          }
        }
      }
      float q[32];
      dct32_inverse(Xs, q);
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] -= q[i];
    } else if constexpr (MODE == kModeDiloco) {
      if (p.sync) {
        if (valid) {
          float4* vrow = reinterpret_cast<float4*>(p.vals + c * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float4 v = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
            if (p.sign) v = make_float4(sign3(v.x), sign3(v.y), sign3(v.z), sign3(v.w));
            vrow[j] = v;
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = 0.0f;
      }
    } else {
      // Random / Striding: values at the selected positions, in draw order.
#pragma unroll
      for (int i = 0; i < 32; ++i) scratch[i * 32 + lane] = x[i];
      float* vrow = p.vals + c * p.k;
      uint32_t P;
      if (vector_k(p.k)) {
        float pv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) pv[j] = 0.0f;
        auto emit = [&](int j, int pos) {
          const float v = scratch[pos * 32 + lane];
          const float w = p.sign ? sign3(v) : v;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) pv[jj] = (jj == j) ? w : pv[jj];
        };
        if constexpr (MODE == kModeRandom) {
          P = random_draws(p.hbase, static_cast<uint64_t>(c), p.k, emit);
        } else {
          for (int j = 0; j < p.k; ++j) emit(j, stride_position(p.stride_o, p.stride_ns, j));
          P = p.stride_mask;
        }
        if (valid) store_payload(vrow, nullptr, pv, 0, 0, p.k);
      } else {
        auto emit = [&](int j, int pos) {
          float v = scratch[pos * 32 + lane];
          if (p.sign) v = sign3(v);
          if (valid) vrow[j] = v;
        };
        if constexpr (MODE == kModeRandom) {
          P = random_draws(p.hbase, static_cast<uint64_t>(c), p.k, emit);
        } else {
          for (int j = 0; j < p.k; ++j) emit(j, stride_position(p.stride_o, p.stride_ns, j));
          P = p.stride_mask;
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = ((P >> i) & 1u) ? 0.0f : x[i];
    }

    store_tile_coalesced(ws.mbuf[s], lane, x, p.m_ptr, row0, p.nc);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) issue(item + 2);
  }
}

cudaError_t launch_encode(const EncodeParams& p, int mode, bool bf16, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kEncThreads);
  cfg.dynamicSmemBytes = kEncSmem;
  cfg.stream = st;
#define DEMO_LAUNCH(M, B) \
  if (mode == M && bf16 == B) return cudaLaunchKernelEx(&cfg, encode_kernel<M, B>, p);
  DEMO_LAUNCH(kModeDemo, false)
  DEMO_LAUNCH(kModeDemo, true)
  DEMO_LAUNCH(kModeRandom, false)
  DEMO_LAUNCH(kModeRandom, true)
  DEMO_LAUNCH(kModeStride, false)
  DEMO_LAUNCH(kModeStride, true)
  DEMO_LAUNCH(kModeDiloco, false)
  DEMO_LAUNCH(kModeDiloco, true)
#undef DEMO_LAUNCH
  return cudaErrorInvalidValue;
}

cudaError_t prepare_encode_kernels() {
  cudaError_t e = cudaSuccess;
#define DEMO_ATTR(M, B)                                                                      \
  if (e == cudaSuccess)                                                                      \
    e = cudaFuncSetAttribute(encode_kernel<M, B>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             static_cast<int>(kEncSmem));
  DEMO_ATTR(kModeDemo, false)
  DEMO_ATTR(kModeDemo, true)
  DEMO_ATTR(kModeRandom, false)
  DEMO_ATTR(kModeRandom, true)
  DEMO_ATTR(kModeStride, false)
  DEMO_ATTR(kModeStride, true)
  DEMO_ATTR(kModeDiloco, false)
  DEMO_ATTR(kModeDiloco, true)
#undef DEMO_ATTR
  return e;
}

}  // namespace demo
