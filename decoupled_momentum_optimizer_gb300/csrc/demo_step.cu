// Fused DeMo shard step: every replica's encode (momentum, selection, error
// feedback, payload) and the decode (scatter-mean, inverse transform, theta
// update) in one pass over HBM.  The payloads never leave the SM.
//
// "DeToNATION: Decoupled Torch Network-Aware Training on Interlinked Online
// Nodes" (Paper-Notes, AAAI 2026), method section, "1. FlexDeMo", Algorithm 1
// (momentum accumulation through the parameter update), with the replication
// group R simulated by R resident replicas.
//
// Per warp, a tile is 32 chunks (one per lane) and is visited as R + 1 items:
// item r < R streams g_r and m_r through TMA into a two-slot ring, computes the
// replica's encode in registers and writes m_r back; the last item streams
// theta, turns the accumulated payloads into Q and writes theta back.  Results
// leave through the item's own slot: each lane writes its row into the
// swizzled tile, the warp reads it back transposed and issues 512-byte
// coalesced stores, and the slot is immediately refilled with the load for
// item i + 2.  Shared memory per warp is 20 KB (two 8 KB slots and a 4 KB
// payload accumulator), so up to 11 warps fit on an SM; the kernel is built for
// 6, 8 and 11 and the launch takes the fewest that cover the item's compute
// (step_warps).  With a 16-bit wire format the accumulated values are rounded
// exactly as the split path's receiver rounds them, so fused and split results
// stay bit-identical.
#include "demo_common.cuh"
#include "demo_params.h"

namespace demo {

struct alignas(1024) StepWarpSmem {
  float gbuf[2][1024];  // slot s: g_r tile (f32 or bf16), later the stash of kept coefficients; or theta
  float mbuf[2][1024];  // slot s: m_r tile, later the new m_r on its way out
  float acc[32 * 32];   // DeMo: per-lane payload sums [u][lane]
};

// Dynamic shared memory of a CTA of `warps` warps: alignment slack, the warps'
// tiles, their two mbarriers each, and the replica-count reciprocal table.
constexpr size_t step_smem(int warps) { return 1024 + warps * sizeof(StepWarpSmem) + warps * 16 + 272; }
static_assert(step_smem(kStepWarps) <= 232448, "shared memory per CTA");

// KV > 0 (DeMo, k in {1, 2, 4, 8}): k is KV at compile time, so the top-k and the payload
// loop unroll; KV = 0: k is the runtime value.
template <int MODE, bool BF16, int MAXR, int WARPS, int KV>
__global__ void __launch_bounds__(WARPS * 32, 1) step_kernel(const __grid_constant__ StepParams<MAXR> p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned start (the TMA swizzle patterns are relative to 1024-byte boundaries),
  // derived by pointer arithmetic on the shared array so every access stays a shared-memory one
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  StepWarpSmem& ws = reinterpret_cast<StepWarpSmem*>(base)[warp];
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + WARPS * sizeof(StepWarpSmem)) + 2 * warp;
  float* rcp = reinterpret_cast<float*>(base + WARPS * sizeof(StepWarpSmem) + WARPS * 16);
  griddep_launch_dependents();
  for (int i = threadIdx.x; i <= kMaxReplicas; i += blockDim.x) rcp[i] = p.rcp_tab[i];
  for (int i = threadIdx.x; i <= 2 * p.R; i += blockDim.x)
    prefetch_tmap(i == 0 ? &p.theta : (i <= p.R ? &p.g[i - 1] : &p.m[i - 1 - p.R]));
  __syncthreads();

  // The launch may run fewer warps than the shared-memory layout holds (WARPS is the most
  // the build's registers allow): warps are counted from the block size.
  const int nw = static_cast<int>(blockDim.x >> 5);
  const long long gw = static_cast<long long>(blockIdx.x) * nw + warp;
  const long long TW = static_cast<long long>(gridDim.x) * nw;
  if (gw >= p.ntiles) return;
  const long long ntw = (p.ntiles - 1 - gw) / TW + 1;
  const bool theta_item = !(MODE == kModeDiloco && !p.sync);
  const int ipt = theta_item ? p.R + 1 : p.R;
  const long long nitems = ntw * ipt;

  if (lane == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if constexpr (MODE == kModeDemo) {
#pragma unroll
    for (int u = 0; u < 32; ++u) ws.acc[u * 32 + lane] = 0.0f;
  }
  __syncwarp();

  // Items are loaded strictly in order, so the loads keep their own (tile, kind)
  // cursor instead of dividing item numbers by the items per tile.
  long long ld_t = gw, ld_item = 0;
  int ld_kind = 0, ld_slot = 0;
  auto issue = [&]() {
    if (ld_t >= p.ntiles) return;
    const int y = static_cast<int>(ld_t * 32);
    uint64_t* bar = &bars[ld_slot];
    const uint32_t extra = stall_extra(p.stall_at, gw, ld_item++);
    if (ld_kind < p.R) {
      mbar_expect_tx(bar, (BF16 ? kTileBytesBF16 : kTileBytesF32) + kTileBytesF32 + extra);
      tma_load_2d(ws.gbuf[ld_slot], &p.g[ld_kind], bar, 0, y);
      tma_load_2d(ws.mbuf[ld_slot], &p.m[ld_kind], bar, 0, y);
    } else {
      mbar_expect_tx(bar, kTileBytesF32 + extra);
      tma_load_2d(ws.gbuf[ld_slot], &p.theta, bar, 0, y);
    }
    ld_slot ^= 1;
    if (++ld_kind == ipt) {
      ld_kind = 0;
      ld_t += TW;
    }
  };
  griddep_wait();  // the previous kernel's writes (m, theta) are visible from here on
  if (lane == 0) {
    issue();
    issue();
  }

  uint32_t P = 0;       // Random / Striding / DiLoCo: positions sent from this lane's chunk
  float accr[32];       // Random / Striding / DiLoCo: per-position payload sums
  uint32_t cnt8[8];     // DeMo: byte (u & 3) of cnt8[u >> 2] counts the replicas that sent slot u
#pragma unroll
  for (int i = 0; i < 32; ++i) accr[i] = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) cnt8[i] = 0u;

  long long t = gw;
  int kind = 0;
  for (long long item = 0; item < nitems; ++item) {
    const int s = static_cast<int>(item & 1);
    const uint32_t par = static_cast<uint32_t>((item >> 1) & 1);
    const long long row0 = t * 32;
    const long long c = row0 + lane;

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

    if (kind == 0) {
      if constexpr (MODE == kModeRandom) P = random_mask(p.hbase, static_cast<uint64_t>(c), p.k);
      if constexpr (MODE == kModeStride) P = p.stride_mask;
      if constexpr (MODE == kModeDiloco) P = 0xffffffffu;
      if constexpr (MODE == kModeDemo) {
#pragma unroll
        for (int i = 0; i < 8; ++i) cnt8[i] = 0u;
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) accr[i] = 0.0f;
      }
    }

    if (kind < p.R) {
      // ---- one replica: m <- beta m + g; select q; m <- m - q; payload -> accumulators
      float x[32], gv[32];
      load_row_grad<BF16>(ws.gbuf[s], lane, gv);
      load_row_f32(ws.mbuf[s], lane, x);
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = __fmaf_rn(p.beta, x[i], gv[i]);

      if constexpr (MODE == kModeDemo) {
        float X[32], Xs[32];
        dct32_forward(x, X);
        const int kk = KV > 0 ? KV : p.k;
        const uint32_t M = topk_select(X, kk, Xs);
        __syncwarp();  // every lane has read its g row: the g tile becomes the stash
        float* stash = ws.gbuf[s];
#pragma unroll
        for (int u = 0; u < 32; ++u) stash[u * 32 + lane] = Xs[u];
        uint32_t mm = M;
        if (p.wire >= kWireBF16) {
#pragma unroll
          for (int j = 0; j < kk; ++j) {  // payload in ascending u, rounded as the wire format rounds it
            const int u = __ffs(mm) - 1;
            mm &= mm - 1;
            float v = stash[u * 32 + lane];
            if (p.sign) v = sign3(v);
            ws.acc[u * 32 + lane] += wire_round(v, p.wire);
          }
        } else {
#pragma unroll
          for (int j = 0; j < kk; ++j) {  // payload in ascending u
            const int u = __ffs(mm) - 1;
            mm &= mm - 1;
            float v = stash[u * 32 + lane];
            if (p.sign) v = sign3(v);
            ws.acc[u * 32 + lane] += v;
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) cnt8[i] += (((M >> (4 * i)) & 0xfu) * 0x204081u) & 0x01010101u;
        float q[32];
        dct32_inverse(Xs, q);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] -= q[i];
      } else if constexpr (MODE == kModeDiloco) {
        if (p.sync) {
          if (p.wire >= kWireBF16) {
#pragma unroll
            for (int i = 0; i < 32; ++i) accr[i] += wire_round(p.sign ? sign3(x[i]) : x[i], p.wire);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) accr[i] += p.sign ? sign3(x[i]) : x[i];
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = 0.0f;
        }
      } else {
        if (p.wire >= kWireBF16) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const bool in = (P >> i) & 1u;
            accr[i] += in ? wire_round(p.sign ? sign3(x[i]) : x[i], p.wire) : 0.0f;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const bool in = (P >> i) & 1u;
            accr[i] += in ? (p.sign ? sign3(x[i]) : x[i]) : 0.0f;
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = ((P >> i) & 1u) ? 0.0f : x[i];
      }
      store_tile_coalesced(ws.mbuf[s], lane, x, p.m_ptr[kind], row0, p.nc);
    } else {
      // ---- decode: Q from the accumulated payloads, theta <- theta - lr Q
      float th[32];
      load_row_f32(ws.gbuf[s], lane, th);
      float Q[32];
      if constexpr (MODE == kModeDemo) {
        float Y[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const uint32_t cnt = (cnt8[u >> 2] >> (8 * (u & 3))) & 0xffu;
          Y[u] = ws.acc[u * 32 + lane] * rcp[cnt];
          ws.acc[u * 32 + lane] = 0.0f;
        }
        dct32_inverse(Y, Q);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) Q[i] = accr[i] * p.rcpR;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) th[i] = __fmaf_rn(-p.lr, Q[i], th[i]);
      __syncwarp();  // every lane has read its theta row
      store_tile_coalesced(ws.gbuf[s], lane, th, p.theta_ptr, row0, p.nc);
    }

    // The slot has been read and written back: refill it with item + 2.
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) issue();
    if (++kind == ipt) {
      kind = 0;
      t += TW;
    }
  }
}

// Resident warps per SM for one step, from the compute per item (measured on
// 2^26 to 2^29-parameter shards, R = 2 and 8, float32 and bfloat16 gradients):
// Striding and DiLoCo sync items are a multiply-add per element; Random adds
// k hashes per chunk once per tile, i.e. shared by R + 1 items; DeMo adds the
// transforms and k - 1 top-k rounds per replica, and from k = 7 on it needs
// all eleven warps to keep HBM busy.  (DiLoCo steps between syncs are sent to
// the elementwise momentum kernel by the host; their rule here is kept for the
// kernel's own generality.)
int step_warps(int mode, int k, bool bf16, int R, bool sync) {
  if (mode == kModeStride) return kStepWarpsLight;
  if (mode == kModeDiloco) return sync ? kStepWarpsLight : kStepWarpsMid;
  if (mode == kModeRandom) return k <= R + 1 ? kStepWarpsLight : kStepWarpsMid;
  if (k == 1 && !bf16) return kStepWarpsLight;
  if (k == 8 && !bf16) return kStepWarpsMid;  // the step compiled for k = 8 (float32 gradients)
  return k <= 6 ? kStepWarpsMid : kStepWarps;
}

template <int MAXR, int WARPS, bool BF16>
static cudaError_t launch_step_demo(const cudaLaunchConfig_t& cfg, const StepParams<MAXR>& p, int kv) {
  switch (kv) {
    case 1: return cudaLaunchKernelEx(&cfg, step_kernel<kModeDemo, BF16, MAXR, WARPS, 1>, p);
    case 2: return cudaLaunchKernelEx(&cfg, step_kernel<kModeDemo, BF16, MAXR, WARPS, 2>, p);
    case 4: return cudaLaunchKernelEx(&cfg, step_kernel<kModeDemo, BF16, MAXR, WARPS, 4>, p);
    case 8: return cudaLaunchKernelEx(&cfg, step_kernel<kModeDemo, BF16, MAXR, WARPS, 8>, p);
    default: return cudaLaunchKernelEx(&cfg, step_kernel<kModeDemo, BF16, MAXR, WARPS, 0>, p);
  }
}

template <int MAXR, int WARPS>
static cudaError_t launch_step_w(const StepParams<MAXR>& p, int mode, bool bf16, int kv, int active, int grid,
                                 cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(active * 32);
  cfg.dynamicSmemBytes = persistent_smem(step_smem(WARPS));
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (mode == kModeDemo)
    return bf16 ? launch_step_demo<MAXR, WARPS, true>(cfg, p, kv) : launch_step_demo<MAXR, WARPS, false>(cfg, p, kv);
#define DEMO_LAUNCH(M, B) \
  if (mode == M && bf16 == B) return cudaLaunchKernelEx(&cfg, step_kernel<M, B, MAXR, WARPS, 0>, p);
  DEMO_LAUNCH(kModeRandom, false)
  DEMO_LAUNCH(kModeRandom, true)
  DEMO_LAUNCH(kModeStride, false)
  DEMO_LAUNCH(kModeStride, true)
  DEMO_LAUNCH(kModeDiloco, false)
  DEMO_LAUNCH(kModeDiloco, true)
#undef DEMO_LAUNCH
  return cudaErrorInvalidValue;
}

template <int MAXR>
static cudaError_t launch_step_t(const StepParams<MAXR>& p, int mode, bool bf16, int warps, int kv, int active,
                                 int grid, cudaStream_t st) {
  if (active < 1 || active > warps) return cudaErrorInvalidValue;
  if (warps == kStepWarpsLight) return launch_step_w<MAXR, kStepWarpsLight>(p, mode, bf16, kv, active, grid, st);
  if (warps == kStepWarpsMid) return launch_step_w<MAXR, kStepWarpsMid>(p, mode, bf16, kv, active, grid, st);
  if (warps == kStepWarps) return launch_step_w<MAXR, kStepWarps>(p, mode, bf16, kv, active, grid, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_step_small(const StepParams<kSmallReplicas>& p, int mode, bool bf16, int warps, int kv, int active,
                              int grid, cudaStream_t st) {
  return launch_step_t(p, mode, bf16, warps, kv, active, grid, st);
}

cudaError_t launch_step_large(const StepParams<kMaxReplicas>& p, int mode, bool bf16, int warps, int kv, int active,
                              int grid, cudaStream_t st) {
  return launch_step_t(p, mode, bf16, warps, kv, active, grid, st);
}

template <int MAXR, int WARPS>
static cudaError_t prepare_w() {
  cudaError_t e = cudaSuccess;
#define DEMO_ATTR(M, B, KV)                                                                                  \
  if (e == cudaSuccess)                                                                                      \
    e = cudaFuncSetAttribute(step_kernel<M, B, MAXR, WARPS, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             static_cast<int>(persistent_smem(step_smem(WARPS))));
  DEMO_ATTR(kModeDemo, false, 0)
  DEMO_ATTR(kModeDemo, false, 1)
  DEMO_ATTR(kModeDemo, false, 2)
  DEMO_ATTR(kModeDemo, false, 4)
  DEMO_ATTR(kModeDemo, false, 8)
  DEMO_ATTR(kModeDemo, true, 0)
  DEMO_ATTR(kModeDemo, true, 1)
  DEMO_ATTR(kModeDemo, true, 2)
  DEMO_ATTR(kModeDemo, true, 4)
  DEMO_ATTR(kModeDemo, true, 8)
  DEMO_ATTR(kModeRandom, false, 0)
  DEMO_ATTR(kModeRandom, true, 0)
  DEMO_ATTR(kModeStride, false, 0)
  DEMO_ATTR(kModeStride, true, 0)
  DEMO_ATTR(kModeDiloco, false, 0)
  DEMO_ATTR(kModeDiloco, true, 0)
#undef DEMO_ATTR
  return e;
}

template <int MAXR>
static cudaError_t prepare_t() {
  cudaError_t e = prepare_w<MAXR, kStepWarpsLight>();
  if (e == cudaSuccess) e = prepare_w<MAXR, kStepWarpsMid>();
  if (e == cudaSuccess) e = prepare_w<MAXR, kStepWarps>();
  return e;
}

cudaError_t prepare_step_kernels() {
  cudaError_t e = prepare_t<kSmallReplicas>();
  if (e == cudaSuccess) e = prepare_t<kMaxReplicas>();
  return e;
}

}  // namespace demo
