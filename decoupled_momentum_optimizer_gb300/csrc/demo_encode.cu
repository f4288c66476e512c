// Split-path encode: one replica's momentum accumulation, extraction and error
// feedback (Algorithm 1) and its payload (the
// buffer the real system would hand to the inter-node all_gather / all-reduce).
//
// "DeToNATION: Decoupled Torch Network-Aware Training on Interlinked Online
// Nodes" (Paper-Notes, AAAI 2026), method section, "1. FlexDeMo" Algorithm 1
// (accumulation, extraction, removal), "2. Replication Schemes" table, "3. Sign
// function" subsection.
//
// Same warp/tile organisation as the fused step: per warp, tiles of 32 chunks
// stream through a two-slot TMA ring; each lane encodes its chunk in registers;
// the new momentum leaves through the tile's own slot with coalesced stores and
// the slot is refilled at once.  The payload is written in the requested wire
// format: float32 / 16-bit values of chunk c at vals[c*k .. c*k+k) (and uint8
// indices for DeMo) by the lane that owns c, as one vector store when k is 1, 2,
// 4 or 8; or ternary bit-planes, one 32-bit word per warp tile and value slot
// built with warp ballots.
#include "demo_common.cuh"
#include "demo_launch.h"

namespace demo {

struct alignas(1024) EncWarpSmem {
  float gbuf[2][1024];  // g tile, then a [i][lane] scratch column per lane
  float mbuf[2][1024];  // m tile, then the new m on its way out
};

// Dynamic shared memory of a CTA of `warps` warps: alignment slack, tiles, mbarriers.
constexpr size_t enc_smem(int warps) { return 1024 + warps * sizeof(EncWarpSmem) + warps * 16; }
static_assert(enc_smem(kStepWarps) <= 232448, "shared memory per CTA");

__device__ __forceinline__ bool vector_k(int k) { return k == 1 || k == 2 || k == 4 || k == 8; }

// Collects one chunk's payload entries (slot j: value v, index u) and writes
// them in the wire format.  put() must be called by all 32 lanes of the warp
// for the same j (the ternary format packs the warp's chunks with ballots).
struct PayloadOut {
  void* vals;
  void* idx;       // nullptr unless DeMo
  long long c;     // this lane's chunk
  long long tile;  // the warp's tile (chunks 32 tile .. 32 tile + 31)
  int lane, k, wire;
  bool valid, vec;
  float pv[8];
  uint32_t ilo, ihi;
  bool tern;  // wire == kWireTernary (a constant false in the k-specialised DeMo kernels)

  __device__ __forceinline__ void put(int j, int u, float v) {
    if (tern) {
      const uint32_t nz = __ballot_sync(0xffffffffu, valid && v != 0.0f);
      const uint32_t ng = __ballot_sync(0xffffffffu, valid && v < 0.0f);
      uint32_t* vw = static_cast<uint32_t*>(vals) + (tile * k + j) * 2;
      if (lane == 0) {
        vw[0] = nz;
        vw[1] = ng;
      }
      if (idx) {
        uint32_t* iw = static_cast<uint32_t*>(idx) + (tile * k + j) * 5;
#pragma unroll
        for (int b = 0; b < 5; ++b) {
          const uint32_t w = __ballot_sync(0xffffffffu, valid && ((u >> b) & 1));
          if (lane == 0) iw[b] = w;
        }
      }
      return;
    }
    if (vec) {
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) pv[jj] = (jj == j) ? v : pv[jj];
      if (j < 4) ilo |= static_cast<uint32_t>(u) << (8 * j);
      else ihi |= static_cast<uint32_t>(u) << (8 * (j - 4));
      return;
    }
    if (!valid) return;
    if (wire == kWireF32) static_cast<float*>(vals)[c * k + j] = v;
    else static_cast<uint16_t*>(vals)[c * k + j] = static_cast<uint16_t>(wire_bits16(v, wire));
    if (idx) static_cast<uint8_t*>(idx)[c * k + j] = static_cast<uint8_t>(u);
  }

  // Vector store of the collected entries (k in {1, 2, 4, 8}, value formats other than ternary).
  __device__ __forceinline__ void finish() {
    if (tern || !vec || !valid) return;
    uint8_t* irow = idx ? static_cast<uint8_t*>(idx) + c * k : nullptr;
    if (wire == kWireF32) {
      float* vrow = static_cast<float*>(vals) + c * k;
      switch (k) {
        case 1: vrow[0] = pv[0]; break;
        case 2: *reinterpret_cast<float2*>(vrow) = make_float2(pv[0], pv[1]); break;
        case 4: *reinterpret_cast<float4*>(vrow) = make_float4(pv[0], pv[1], pv[2], pv[3]); break;
        default:
          reinterpret_cast<float4*>(vrow)[0] = make_float4(pv[0], pv[1], pv[2], pv[3]);
          reinterpret_cast<float4*>(vrow)[1] = make_float4(pv[4], pv[5], pv[6], pv[7]);
      }
    } else {
      uint32_t h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = wire_bits16(pv[2 * i], wire) | (wire_bits16(pv[2 * i + 1], wire) << 16);
      uint16_t* vrow = static_cast<uint16_t*>(vals) + c * k;
      switch (k) {
        case 1: vrow[0] = static_cast<uint16_t>(h[0]); break;
        case 2: *reinterpret_cast<uint32_t*>(vrow) = h[0]; break;
        case 4: *reinterpret_cast<uint2*>(vrow) = make_uint2(h[0], h[1]); break;
        default: *reinterpret_cast<uint4*>(vrow) = make_uint4(h[0], h[1], h[2], h[3]);
      }
    }
    if (irow) {
      switch (k) {
        case 1: irow[0] = static_cast<uint8_t>(ilo); break;
        case 2: *reinterpret_cast<uint16_t*>(irow) = static_cast<uint16_t>(ilo); break;
        case 4: *reinterpret_cast<uint32_t*>(irow) = ilo; break;
        default: *reinterpret_cast<uint2*>(irow) = make_uint2(ilo, ihi);
      }
    }
  }
};

// Ternary bit-planes of a DeMo tile for k = K known at compile time: each ballot word is kept
// by the lane with its index in the tile's block (value words [K][2], index words [K][5]), and
// the block leaves with coalesced stores instead of one single-lane store per word.  put()
// must be called by all 32 lanes for the same j, with j a compile-time index.
template <int K>
struct TernaryOut {
  static constexpr int kIdxRegs = (5 * K + 31) / 32;
  uint32_t* vw;  // the tile's value words
  uint32_t* iw;  // the tile's index words
  int lane;
  bool valid;
  uint32_t v_word, i_word[kIdxRegs];

  __device__ __forceinline__ void put(int j, int u, float v) {
    const uint32_t nz = __ballot_sync(0xffffffffu, valid && v != 0.0f);
    const uint32_t ng = __ballot_sync(0xffffffffu, valid && v < 0.0f);
    v_word = lane == 2 * j ? nz : (lane == 2 * j + 1 ? ng : v_word);
#pragma unroll
    for (int b = 0; b < 5; ++b) {
      const uint32_t w = __ballot_sync(0xffffffffu, valid && ((u >> b) & 1));
      const int at = 5 * j + b;
      i_word[at / 32] = lane == at % 32 ? w : i_word[at / 32];
    }
  }

  __device__ __forceinline__ void finish() {
    if (lane < 2 * K) vw[lane] = v_word;
#pragma unroll
    for (int q = 0; q < kIdxRegs; ++q)
      if (32 * q + lane < 5 * K) iw[32 * q + lane] = i_word[q];
  }
};

// DiLoCo sync step: the whole row of 32 values of this lane's chunk, in the wire format.
__device__ __forceinline__ void put_row(void* vals, int wire, long long c, long long tile, int lane, bool valid,
                                        const float (&v)[32]) {
  if (wire == kWireTernary) {
    uint32_t my_nz = 0, my_ng = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint32_t nz = __ballot_sync(0xffffffffu, valid && v[j] != 0.0f);
      const uint32_t ng = __ballot_sync(0xffffffffu, valid && v[j] < 0.0f);
      my_nz = (lane == j) ? nz : my_nz;
      my_ng = (lane == j) ? ng : my_ng;
    }
    reinterpret_cast<uint2*>(static_cast<uint32_t*>(vals) + tile * 64)[lane] = make_uint2(my_nz, my_ng);
    return;
  }
  if (!valid) return;
  if (wire == kWireF32) {
    float4* row = reinterpret_cast<float4*>(static_cast<float*>(vals) + c * 32);
#pragma unroll
    for (int j = 0; j < 8; ++j) row[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  } else {
    uint4* row = reinterpret_cast<uint4*>(static_cast<uint16_t*>(vals) + c * 32);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        h[i] = wire_bits16(v[8 * j + 2 * i], wire) | (wire_bits16(v[8 * j + 2 * i + 1], wire) << 16);
      row[j] = make_uint4(h[0], h[1], h[2], h[3]);
    }
  }
}

// KV > 0 (DeMo, a float32 or 16-bit format, k in {1, 2, 4, 8}): k is KV at compile
// time, so the payload loop unrolls, each entry goes straight to its register and the
// vector store needs no dispatch on k; KV < 0 (DeMo, the ternary format, k = -KV in
// {1, 2, 4, 8}): the same for the tile's bit-plane words (TernaryOut); KV = 0: k is the
// runtime value.
template <int MODE, bool BF16, int WARPS, int KV>
__global__ void __launch_bounds__(WARPS * 32, 1) encode_kernel(const __grid_constant__ EncodeParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned start (the TMA swizzle patterns are relative to 1024-byte boundaries),
  // derived by pointer arithmetic on the shared array so every access stays a shared-memory one
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  EncWarpSmem& ws = reinterpret_cast<EncWarpSmem*>(base)[warp];
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + WARPS * sizeof(EncWarpSmem)) + 2 * warp;
  // Programmatic launch.  By default the kernel lets the next one start at once and waits for
  // the previous one before its first global access.  With defer_wait (set by the host only
  // inside a sequence of its own launches whose kernels share no buffers), the loads and the
  // work overlap the previous kernel's tail and the wait moves to the end, so this grid still
  // completes after the previous one and every event recorded behind it covers both; the next
  // kernel is let start only once this one's own wait has passed when it does wait first, so
  // a deferred successor never starts ahead of the work before the sequence.
  if (p.defer_wait) griddep_launch_dependents();

  // The launch may run fewer warps than the shared-memory layout holds: warps are counted
  // from the block size.
  const int nw = static_cast<int>(blockDim.x >> 5);
  const long long gw = static_cast<long long>(blockIdx.x) * nw + warp;
  const long long TW = static_cast<long long>(gridDim.x) * nw;
  if (gw >= p.ntiles) {
    if (!p.defer_wait) {
      griddep_wait();
      griddep_launch_dependents();
    }
    return;
  }
  const long long nitems = (p.ntiles - 1 - gw) / TW + 1;

  if (lane == 0) {
    prefetch_tmap(&p.g);
    prefetch_tmap(&p.m);
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (!p.defer_wait) {
    griddep_wait();  // the previous kernel's writes (m, an earlier payload's readers) are done
    griddep_launch_dependents();
  }

  auto issue = [&](long long item) {
    if (item >= nitems) return;
    const int s = static_cast<int>(item & 1);
    const int y = static_cast<int>((gw + item * TW) * 32);
    mbar_expect_tx(&bars[s], (BF16 ? kTileBytesBF16 : kTileBytesF32) + kTileBytesF32 + stall_extra(p.stall_at, gw, item));
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
      if (p.defer_wait) griddep_wait();
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
      const uint32_t M = topk_select(X, KV < 0 ? -KV : p.k, Xs);
#pragma unroll
      for (int u = 0; u < 32; ++u) scratch[u * 32 + lane] = Xs[u];
      const bool tern = KV != 0 ? false : p.wire == kWireTernary;
      PayloadOut out{p.vals, p.idx, c, row0 >> 5, lane, KV > 0 ? KV : p.k, p.wire, valid,
                     KV > 0 ? true : vector_k(p.k) && !tern, {0, 0, 0, 0, 0, 0, 0, 0}, 0u, 0u, tern};
      uint32_t mm = M;
      auto entry = [&](int j) {  // payload in ascending u
        const int u = __ffs(mm) - 1;
        mm &= mm - 1;
        const float v = scratch[u * 32 + lane];
        out.put(j, u, p.sign ? sign3(v) : v);
      };
      if constexpr (KV < 0) {
        constexpr int K = -KV;
        const long long tile = row0 >> 5;
        TernaryOut<K> tw{static_cast<uint32_t*>(p.vals) + tile * K * 2, static_cast<uint32_t*>(p.idx) + tile * K * 5,
                         lane, valid, 0u, {}};
#pragma unroll
        for (int j = 0; j < K; ++j) {
          const int u = __ffs(mm) - 1;
          mm &= mm - 1;
          const float v = scratch[u * 32 + lane];
          tw.put(j, u, p.sign ? sign3(v) : v);
        }
        tw.finish();
      } else {
        if constexpr (KV > 0) {
#pragma unroll
          for (int j = 0; j < KV; ++j) entry(j);
        } else {
          for (int j = 0; j < p.k; ++j) entry(j);
        }
        out.finish();
      }
      float q[32];
      dct32_inverse(Xs, q);
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] -= q[i];
    } else if constexpr (MODE == kModeDiloco) {
      if (p.sync) {
        float sv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[i] = p.sign ? sign3(x[i]) : x[i];
        if (p.wire == kWireF32) {
          // a float32 payload row has the momentum's layout: it leaves through the (free) g slot
          // with the same coalesced stores (2^27 encode: 355 -> 328 us, 89% -> 97% of the copy
          // peak, against each lane storing its own row)
          store_tile_coalesced(ws.gbuf[s], lane, sv, static_cast<float*>(p.vals), row0, p.nc);
        } else {
          put_row(p.vals, p.wire, c, row0 >> 5, lane, valid, sv);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = 0.0f;
      }
    } else {
      // Random / Striding: values at the selected positions, in draw order.
#pragma unroll
      for (int i = 0; i < 32; ++i) scratch[i * 32 + lane] = x[i];
      PayloadOut out{p.vals, nullptr, c, row0 >> 5, lane, p.k, p.wire, valid,
                     vector_k(p.k) && p.wire != kWireTernary, {0, 0, 0, 0, 0, 0, 0, 0}, 0u, 0u,
                     p.wire == kWireTernary};
      auto emit = [&](int j, int pos) {
        const float v = scratch[pos * 32 + lane];
        out.put(j, pos, p.sign ? sign3(v) : v);
      };
      uint32_t P;
      if constexpr (MODE == kModeRandom) {
        P = random_draws(p.hbase, static_cast<uint64_t>(c + p.chunk0), p.k, emit);
      } else {
        for (int j = 0; j < p.k; ++j) emit(j, stride_position(p.stride_o, p.stride_ns, j));
        P = p.stride_mask;
      }
      out.finish();
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = ((P >> i) & 1u) ? 0.0f : x[i];
    }

    store_tile_coalesced(ws.mbuf[s], lane, x, p.m_ptr, row0, p.nc);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) issue(item + 2);
  }
  if (p.defer_wait) griddep_wait();  // complete only after the previous kernel
}

// Resident warps per SM for one encode, and whether DeMo runs the kernel compiled for
// its k (*kv = k) or the runtime-k one (*kv = 0), from its compute per tile (measured
// jointly on the T5-base shard with float32 and the OLMo-shaped shard with bfloat16
// gradients): as in the fused step, fewer warps run faster once HBM is saturated,
// unless the selection needs them (DeMo from k = 7 on, the ternary format's ballots).
// The k-compiled kernel issues fewer instructions and so wants fewer warps; bfloat16
// gradients bring less data per tile for the same compute and want more.
// The k-specialised ternary DeMo encode: warps per CTA by gradient dtype (float32, bfloat16)
// and k (1, 2, 4, 8).  Measured on a 2^27 shard with float32 gradients: k = 1 6 warps 255 us
// (runtime k, 11 warps: 284), k = 2 6 warps 244 us (8: 274), k = 4 8 warps 266 us (11: 286),
// k = 8 11 warps 275 us (8: 300, runtime k: 354); with bfloat16 gradients k = 1, 2 8 warps
// 222 / 219 us (6: 220 / 234, 11: 237 / 239), k = 4 11 warps 215 us (8: 222).  The seven
// ballots per entry at k = 8 want the most warps in flight.
constexpr int kTernaryEncodeWarps[2][4] = {{kStepWarpsLight, kStepWarpsLight, kStepWarpsMid, kStepWarps},
                                           {kStepWarpsMid, kStepWarpsMid, kStepWarps, kStepWarps}};

int encode_warps(int mode, int k, int wire, bool bf16, int* kv) {
  *kv = 0;
  if (mode == kModeDemo) {
    if (wire == kWireTernary) {
      if (k != 1 && k != 2 && k != 4 && k != 8) return kStepWarps;
      *kv = -k;
      return kTernaryEncodeWarps[bf16 ? 1 : 0][k == 1 ? 0 : k == 2 ? 1 : k == 4 ? 2 : 3];
    }
    if (k == 1 || k == 2 || k == 4 || k == 8) {
      if (!bf16 && k <= 2) {
        *kv = k;
        return kStepWarpsLight;
      }
      if (bf16 ? k >= 2 : k == 8) *kv = k;
      return kStepWarpsMid;
    }
    if (bf16) return k == 1 ? kStepWarpsMid : kStepWarps;
    return k <= 6 ? kStepWarpsMid : kStepWarps;
  }
  // Random with float32 gradients: k <= 4 draws per chunk are light enough for six warps
  // (k <= 2: 1-3% faster than eight on 2^26-2^28 shards and the ViT-B shard; k = 4 on a 2^27
  // shard 247 us against 282 us with eight); k = 8 wants eight (six: 363 us, eight: 276).
  // With bfloat16 gradients k <= 2 take six (201 / 206 us against 216 / 225 with eleven), k = 4
  // eight (222 against 243), k = 8 eleven (241; eight: 275).
  if (mode == kModeRandom) {
    if (bf16) return k <= 2 ? kStepWarpsLight : k == 4 ? kStepWarpsMid : kStepWarps;
    return k <= 4 ? kStepWarpsLight : kStepWarpsMid;
  }
  // Striding with float32 gradients: eleven warps, but six for k = 8 (2^27: 277 us against 285).
  if (mode == kModeStride) return bf16 ? kStepWarpsLight : (k == 8 ? kStepWarpsLight : kStepWarps);
  return bf16 ? kStepWarpsLight : kStepWarpsMid;
}

template <int WARPS, bool BF16>
static cudaError_t launch_encode_demo(const cudaLaunchConfig_t& cfg, const EncodeParams& p, int kv) {
  switch (kv) {
    case 1: return cudaLaunchKernelEx(&cfg, encode_kernel<kModeDemo, BF16, WARPS, 1>, p);
    case 2: return cudaLaunchKernelEx(&cfg, encode_kernel<kModeDemo, BF16, WARPS, 2>, p);
    case 4: return cudaLaunchKernelEx(&cfg, encode_kernel<kModeDemo, BF16, WARPS, 4>, p);
    case 8: return cudaLaunchKernelEx(&cfg, encode_kernel<kModeDemo, BF16, WARPS, 8>, p);
    case -1: return cudaLaunchKernelEx(&cfg, encode_kernel<kModeDemo, BF16, WARPS, -1>, p);
    case -2: return cudaLaunchKernelEx(&cfg, encode_kernel<kModeDemo, BF16, WARPS, -2>, p);
    case -4: return cudaLaunchKernelEx(&cfg, encode_kernel<kModeDemo, BF16, WARPS, -4>, p);
    case -8: return cudaLaunchKernelEx(&cfg, encode_kernel<kModeDemo, BF16, WARPS, -8>, p);
    default: return cudaLaunchKernelEx(&cfg, encode_kernel<kModeDemo, BF16, WARPS, 0>, p);
  }
}

template <int WARPS>
static cudaError_t launch_encode_w(const EncodeParams& p, int mode, bool bf16, int kv, int active, int grid,
                                   cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(active * 32);
  cfg.dynamicSmemBytes = persistent_smem(enc_smem(WARPS));
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (mode == kModeDemo)
    return bf16 ? launch_encode_demo<WARPS, true>(cfg, p, kv) : launch_encode_demo<WARPS, false>(cfg, p, kv);
#define DEMO_LAUNCH(M, B) \
  if (mode == M && bf16 == B) return cudaLaunchKernelEx(&cfg, encode_kernel<M, B, WARPS, 0>, p);
  DEMO_LAUNCH(kModeRandom, false)
  DEMO_LAUNCH(kModeRandom, true)
  DEMO_LAUNCH(kModeStride, false)
  DEMO_LAUNCH(kModeStride, true)
  DEMO_LAUNCH(kModeDiloco, false)
  DEMO_LAUNCH(kModeDiloco, true)
#undef DEMO_LAUNCH
  return cudaErrorInvalidValue;
}

cudaError_t launch_encode(const EncodeParams& p, int mode, bool bf16, int warps, int kv, int active, int grid,
                          cudaStream_t st) {
  if (active < 1 || active > warps) return cudaErrorInvalidValue;
  if (warps == kStepWarpsLight) return launch_encode_w<kStepWarpsLight>(p, mode, bf16, kv, active, grid, st);
  if (warps == kStepWarpsMid) return launch_encode_w<kStepWarpsMid>(p, mode, bf16, kv, active, grid, st);
  if (warps == kStepWarps) return launch_encode_w<kStepWarps>(p, mode, bf16, kv, active, grid, st);
  return cudaErrorInvalidValue;
}

template <int WARPS>
static cudaError_t prepare_encode_w() {
  cudaError_t e = cudaSuccess;
#define DEMO_ATTR(M, B, KV)                                                                             \
  if (e == cudaSuccess)                                                                                 \
    e = cudaFuncSetAttribute(encode_kernel<M, B, WARPS, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             static_cast<int>(persistent_smem(enc_smem(WARPS))));
  DEMO_ATTR(kModeDemo, false, 0)
  DEMO_ATTR(kModeDemo, false, 1)
  DEMO_ATTR(kModeDemo, false, 2)
  DEMO_ATTR(kModeDemo, false, 4)
  DEMO_ATTR(kModeDemo, false, 8)
  DEMO_ATTR(kModeDemo, false, -1)
  DEMO_ATTR(kModeDemo, false, -2)
  DEMO_ATTR(kModeDemo, false, -4)
  DEMO_ATTR(kModeDemo, false, -8)
  DEMO_ATTR(kModeDemo, true, 0)
  DEMO_ATTR(kModeDemo, true, 1)
  DEMO_ATTR(kModeDemo, true, 2)
  DEMO_ATTR(kModeDemo, true, 4)
  DEMO_ATTR(kModeDemo, true, 8)
  DEMO_ATTR(kModeDemo, true, -1)
  DEMO_ATTR(kModeDemo, true, -2)
  DEMO_ATTR(kModeDemo, true, -4)
  DEMO_ATTR(kModeDemo, true, -8)
  DEMO_ATTR(kModeRandom, false, 0)
  DEMO_ATTR(kModeRandom, true, 0)
  DEMO_ATTR(kModeStride, false, 0)
  DEMO_ATTR(kModeStride, true, 0)
  DEMO_ATTR(kModeDiloco, false, 0)
  DEMO_ATTR(kModeDiloco, true, 0)
#undef DEMO_ATTR
  return e;
}

cudaError_t prepare_encode_kernels() {
  cudaError_t e = prepare_encode_w<kStepWarpsLight>();
  if (e == cudaSuccess) e = prepare_encode_w<kStepWarpsMid>();
  if (e == cudaSuccess) e = prepare_encode_w<kStepWarps>();
  return e;
}

}  // namespace demo
