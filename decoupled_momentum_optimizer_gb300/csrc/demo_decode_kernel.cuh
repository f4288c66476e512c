// The split-path decode kernel (see demo_decode.cu), its helpers and its launch and
// set-up templates, shared by the translation units that compile its staging flavours.
#pragma once

#include "demo_common.cuh"
#include "demo_launch.h"

namespace demo {

// One slot's running sum and number of received entries.
struct alignas(8) SumCount {
  float sum;
  uint32_t cnt;
};

template <int STAGE>
struct alignas(1024) DecWarpSmem {
  float tbuf[2][1024];                    // theta tiles (and the theta rows on their way out)
  SumCount acc[32 * 32];                  // DeMo: [u][lane]; others: [i][lane].sum = Q scratch
  unsigned char stage[2][STAGE];          // slot s: staged payload spans, replica r at r * (vspan + ispan)
};

// Dynamic shared memory of a decode CTA of `warps` warps (see dec_stage_bytes).
constexpr size_t dec_smem(int warps) {
  return 1024 + warps * (2 * 4096 + 8 * 1024 + 2 * dec_stage_bytes(warps)) + warps * 16 + 272;
}
template <int W>
constexpr bool dec_shape_fits() {
  return sizeof(DecWarpSmem<dec_stage_bytes(W)>) == 2 * 4096 + 8 * 1024 + 2 * dec_stage_bytes(W) &&
         dec_smem(W) <= 232448;
}
static_assert(dec_shape_fits<11>() && dec_shape_fits<10>() && dec_shape_fits<9>() && dec_shape_fits<8>(),
              "decode shapes: layout and shared memory per CTA");

__device__ __forceinline__ bool vector_kd(int k) { return k == 1 || k == 2 || k == 4 || k == 8; }

// Per-lane asynchronous 16-byte copies from global to shared memory (both addresses
// 16-byte aligned), cached in L2 only.  Each lane's copies since its last commit form one
// group; waiting for all but the newest N groups makes the older ones' data visible to the
// lane, and a warp barrier after it to the whole warp.
__device__ __forceinline__ void lane_copy16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
// The same for a 4-byte unit (both addresses 4-byte aligned), cached in L1 and L2.
__device__ __forceinline__ void lane_copy4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void lane_copy_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void lane_copy_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Value j of chunk c (tile `tile`, lane `lane`) of a payload with kv values per chunk.
__device__ __forceinline__ float payload_value(const void* vals, int wire, long long c, long long tile, int lane,
                                               int kv, int j) {
  if (wire == kWireF32) return static_cast<const float*>(vals)[c * kv + j];
  if (wire == kWireTernary) {
    const uint2 w = reinterpret_cast<const uint2*>(vals)[tile * kv + j];
    const uint32_t nz = (w.x >> lane) & 1u, ng = (w.y >> lane) & 1u;
    return nz ? (ng ? -1.0f : 1.0f) : 0.0f;
  }
  return wire_from_bits16(static_cast<const uint16_t*>(vals)[c * kv + j], wire);
}

// Bit `lane` of plane word w moved to bit b, masked to that bit.  ROT: one funnel-shift rotation
// right by lane - b and a masked OR per bit; measured faster where the words are loaded one or
// two at a time (2^26 decode, R = 64 in groups: k = 4 936 -> 878 us; k = 1, 2 at every R) and
// slower beside the 16-byte vector reads of k >= 4 (R = 16, k = 4: 246 -> 253 us).
template <bool ROT>
__device__ __forceinline__ uint32_t plane_bit(uint32_t w, int lane, int b) {
  if constexpr (ROT) return __funnelshift_r(w, w, static_cast<uint32_t>(lane - b) & 31u) & (1u << b);
  return ((w >> lane) & 1u) << b;
}

// Index j of chunk c in a DeMo payload (uint8, or 5 ternary bit-planes); used modulo 32.
__device__ __forceinline__ int payload_index(const void* idx, int wire, long long c, long long tile, int lane, int k,
                                             int j) {
  if (wire == kWireTernary) {
    const uint32_t* w = static_cast<const uint32_t*>(idx) + (tile * k + j) * 5;
    int u = 0;
#pragma unroll
    for (int b = 0; b < 5; ++b) u |= static_cast<int>(plane_bit<true>(w[b], lane, b));
    return u;
  }
  return static_cast<const uint8_t*>(idx)[c * k + j] & 31;
}

// Vector load of one chunk's k values (k in {1, 2, 4, 8}; float32 or 16-bit wire) and its index bytes.
__device__ __forceinline__ void load_payload(const void* vals, const void* idx, int wire, long long c, int k,
                                             float (&pv)[8], uint32_t& ilo, uint32_t& ihi) {
  ilo = ihi = 0;
  if (wire == kWireF32) {
    const float* vrow = static_cast<const float*>(vals) + c * k;
    switch (k) {
      case 1: pv[0] = vrow[0]; break;
      case 2: { const float2 v = *reinterpret_cast<const float2*>(vrow); pv[0] = v.x; pv[1] = v.y; break; }
      case 4: {
        const float4 v = *reinterpret_cast<const float4*>(vrow);
        pv[0] = v.x; pv[1] = v.y; pv[2] = v.z; pv[3] = v.w;
        break;
      }
      default: {
        const float4 a = reinterpret_cast<const float4*>(vrow)[0];
        const float4 b = reinterpret_cast<const float4*>(vrow)[1];
        pv[0] = a.x; pv[1] = a.y; pv[2] = a.z; pv[3] = a.w;
        pv[4] = b.x; pv[5] = b.y; pv[6] = b.z; pv[7] = b.w;
      }
    }
  } else {
    const uint16_t* vrow = static_cast<const uint16_t*>(vals) + c * k;
    uint32_t h[4] = {0, 0, 0, 0};
    switch (k) {
      case 1: h[0] = vrow[0]; break;
      case 2: h[0] = *reinterpret_cast<const uint32_t*>(vrow); break;
      case 4: { const uint2 v = *reinterpret_cast<const uint2*>(vrow); h[0] = v.x; h[1] = v.y; break; }
      default: {
        const uint4 v = *reinterpret_cast<const uint4*>(vrow);
        h[0] = v.x; h[1] = v.y; h[2] = v.z; h[3] = v.w;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      pv[2 * i] = wire_from_bits16(h[i] & 0xffffu, wire);
      pv[2 * i + 1] = wire_from_bits16(h[i] >> 16, wire);
    }
  }
  if (idx) {
    const uint8_t* irow = static_cast<const uint8_t*>(idx) + c * k;
    switch (k) {
      case 1: ilo = irow[0]; break;
      case 2: ilo = *reinterpret_cast<const uint16_t*>(irow); break;
      case 4: ilo = *reinterpret_cast<const uint32_t*>(irow); break;
      default: { const uint2 w = *reinterpret_cast<const uint2*>(irow); ilo = w.x; ihi = w.y; }
    }
  }
}

// One chunk's KV values of a float32 or 16-bit payload (KV in {1, 2, 4, 8}), one vector load.
template <int KV>
__device__ __forceinline__ void load_values(const void* vals, int wire, long long c, float (&v)[KV]) {
  if (wire == kWireF32) {
    const float* row = static_cast<const float*>(vals) + c * KV;
    if constexpr (KV == 1) {
      v[0] = row[0];
    } else if constexpr (KV == 2) {
      const float2 a = *reinterpret_cast<const float2*>(row);
      v[0] = a.x;
      v[1] = a.y;
    } else {
#pragma unroll
      for (int q = 0; q < KV / 4; ++q) {
        const float4 a = reinterpret_cast<const float4*>(row)[q];
        v[4 * q] = a.x;
        v[4 * q + 1] = a.y;
        v[4 * q + 2] = a.z;
        v[4 * q + 3] = a.w;
      }
    }
  } else {
    const uint16_t* row = static_cast<const uint16_t*>(vals) + c * KV;
    uint32_t h[(KV + 1) / 2];
    if constexpr (KV == 1) {
      h[0] = row[0];
    } else if constexpr (KV == 2) {
      h[0] = *reinterpret_cast<const uint32_t*>(row);
    } else if constexpr (KV == 4) {
      const uint2 a = *reinterpret_cast<const uint2*>(row);
      h[0] = a.x;
      h[1] = a.y;
    } else {
      const uint4 a = *reinterpret_cast<const uint4*>(row);
      h[0] = a.x;
      h[1] = a.y;
      h[2] = a.z;
      h[3] = a.w;
    }
#pragma unroll
    for (int i = 0; i < KV; ++i) v[i] = wire_from_bits16((h[i / 2] >> (16 * (i & 1))) & 0xffffu, wire);
  }
}

// Adds one replica's entries for chunk c (sum and count per slot u) to acc.
// vals / idx address either the payload buffers (chunk c of tile `tile`) or a
// staged copy of the tile's spans (c = lane, tile = 0).  `valid`: the chunk
// exists; `reads`: the lane may read (per-chunk formats only for chunks that
// exist; the ternary words belong to the whole tile and every lane reads them).
// KV > 0: k is KV, known at compile time (a float32 or 16-bit format with k in
// {1, 2, 4, 8}), so the vector load needs no dispatch on k and the entry loop runs
// exactly k times; KV = 0: k is the runtime value.
template <int KV>
__device__ __forceinline__ void demo_accumulate(SumCount* acc, int lane, const void* vals, const void* idx, int wire,
                                                int k_runtime, long long c, long long tile, bool valid, bool reads) {
  const int k = KV > 0 ? KV : k_runtime;
  if (KV > 0 || (wire != kWireTernary && vector_kd(k))) {
    if (valid) {
      float pv[8];
      uint32_t ilo, ihi;
      load_payload(vals, idx, wire, c, k, pv, ilo, ihi);
      constexpr int kMaxEntries = KV > 0 ? KV : 8;
      int uu[kMaxEntries];
#pragma unroll
      for (int j = 0; j < kMaxEntries; ++j) uu[j] = ((j < 4 ? ilo >> (8 * j) : ihi >> (8 * (j - 4)))) & 31;
      bool ascending = false;
      if constexpr (KV > 1) {
        ascending = true;
#pragma unroll
        for (int j = 1; j < KV; ++j) ascending = ascending && uu[j] > uu[j - 1];
      }
      if (ascending) {
        // A valid payload lists distinct slots in ascending order: read all k slots,
        // then update and write them, instead of a chain of k dependent updates.
        SumCount a[kMaxEntries];
#pragma unroll
        for (int j = 0; j < kMaxEntries; ++j) a[j] = acc[uu[j] * 32 + lane];
#pragma unroll
        for (int j = 0; j < kMaxEntries; ++j) {
          a[j].sum += pv[j];
          a[j].cnt += 1u;
        }
#pragma unroll
        for (int j = 0; j < kMaxEntries; ++j) acc[uu[j] * 32 + lane] = a[j];
      } else {
#pragma unroll
        for (int j = 0; j < kMaxEntries; ++j) {
          if (KV > 0 || j < k) {
            SumCount a = acc[uu[j] * 32 + lane];
            a.sum += pv[j];
            a.cnt += 1u;
            acc[uu[j] * 32 + lane] = a;
          }
        }
      }
    }
  } else {
    for (int j = 0; j < k; ++j) {
      const int u = reads ? payload_index(idx, wire, c, tile, lane, k, j) : 0;
      const float v = reads ? payload_value(vals, wire, c, tile, lane, k, j) : 0.0f;
      if (valid) {
        SumCount a = acc[u * 32 + lane];
        a.sum += v;
        a.cnt += 1u;
        acc[u * 32 + lane] = a;
      }
    }
  }
}

// One replica's entries for this lane's chunk, read and decoded, for a k known at
// compile time: KV < 0 is -k for the ternary format (KV > 0, k for a float32 or 16-bit
// format, is also readable this way, but demo_accumulate serves those: reading ahead
// measured 1-2% slower there).  For the ternary format every entry takes seven bit-plane
// words, and reading the next replica's entries before adding this replica's lets those
// loads overlap the shared-memory updates (the updates themselves stay in replica order).
template <int KV>
struct DemoEntries {
  static constexpr int K = KV < 0 ? -KV : KV;
  float pv[K];
  int uu[K];
};

// VEC: read the ternary words of k >= 4 as 16-byte vectors where aligned.  Measured faster
// except in the group flavours (2^26: R = 8 k = 4 164 -> 156 us, R = 2 k = 8 (2^27) 230 -> 223
// us; grouped, R = 64: 939 -> 980 us), which read them one or two words at a time.
template <int KV, bool VEC = false>
__device__ __forceinline__ void demo_read(DemoEntries<KV>& e, const void* vals, const void* idx, int wire,
                                          long long c, long long tile, int lane) {
  constexpr int K = DemoEntries<KV>::K;
  if constexpr (KV < 0) {
    // the tile's bit-planes: value words [K][2] (nonzero, negative), index words [K][5]; this
    // lane's chunk is bit `lane` of each word
    const uint32_t* vw = static_cast<const uint32_t*>(vals) + tile * K * 2;
    const uint32_t* iw = static_cast<const uint32_t*>(idx) + tile * K * 5;
    if constexpr (K >= 4 && VEC) {
      // k >= 4: a tile's 2k value words and 5k index words are whole 16-byte vectors when the
      // buffers are 16-byte aligned (staged spans always are): 7k / 4 vector loads instead of
      // 6k loads of one or two words
      if (((reinterpret_cast<uintptr_t>(vw) | reinterpret_cast<uintptr_t>(iw)) & 15u) == 0) {
        uint32_t vwd[2 * K], iwd[5 * K];
#pragma unroll
        for (int q = 0; q < K / 2; ++q) {
          const uint4 t = reinterpret_cast<const uint4*>(vw)[q];
          vwd[4 * q] = t.x;
          vwd[4 * q + 1] = t.y;
          vwd[4 * q + 2] = t.z;
          vwd[4 * q + 3] = t.w;
        }
#pragma unroll
        for (int q = 0; q < 5 * K / 4; ++q) {
          const uint4 t = reinterpret_cast<const uint4*>(iw)[q];
          iwd[4 * q] = t.x;
          iwd[4 * q + 1] = t.y;
          iwd[4 * q + 2] = t.z;
          iwd[4 * q + 3] = t.w;
        }
#pragma unroll
        for (int j = 0; j < K; ++j) {
          const uint32_t nz = (vwd[2 * j] >> lane) & 1u, ng = (vwd[2 * j + 1] >> lane) & 1u;
          e.pv[j] = nz ? (ng ? -1.0f : 1.0f) : 0.0f;
          int u = 0;
#pragma unroll
          for (int b = 0; b < 5; ++b) u |= static_cast<int>(plane_bit<false>(iwd[5 * j + b], lane, b));
          e.uu[j] = u;
        }
        return;
      }
    }
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const uint2 w = reinterpret_cast<const uint2*>(vw)[j];
      const uint32_t nz = (w.x >> lane) & 1u, ng = (w.y >> lane) & 1u;
      e.pv[j] = nz ? (ng ? -1.0f : 1.0f) : 0.0f;
      int u = 0;
#pragma unroll
      for (int b = 0; b < 5; ++b) u |= static_cast<int>(plane_bit<true>(iw[5 * j + b], lane, b));
      e.uu[j] = u;
    }
  } else {
    float pv[8];
    uint32_t ilo, ihi;
    load_payload(vals, idx, wire, c, K, pv, ilo, ihi);
#pragma unroll
    for (int j = 0; j < K; ++j) {
      e.pv[j] = pv[j];
      e.uu[j] = ((j < 4 ? ilo >> (8 * j) : ihi >> (8 * (j - 4)))) & 31;
    }
  }
}

template <int KV>
__device__ __forceinline__ void demo_add(SumCount* acc, int lane, const DemoEntries<KV>& e) {
  constexpr int K = DemoEntries<KV>::K;
  bool ascending = false;
  if constexpr (K > 1) {
    ascending = true;
#pragma unroll
    for (int j = 1; j < K; ++j) ascending = ascending && e.uu[j] > e.uu[j - 1];
  }
  if (ascending) {
    // A valid payload lists distinct slots in ascending order: read all k slots, then update
    // and write them, instead of a chain of k dependent updates.
    SumCount a[K];
#pragma unroll
    for (int j = 0; j < K; ++j) a[j] = acc[e.uu[j] * 32 + lane];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      a[j].sum += e.pv[j];
      a[j].cnt += 1u;
    }
#pragma unroll
    for (int j = 0; j < K; ++j) acc[e.uu[j] * 32 + lane] = a[j];
  } else {
#pragma unroll
    for (int j = 0; j < K; ++j) {
      SumCount a = acc[e.uu[j] * 32 + lane];
      a.sum += e.pv[j];
      a.cnt += 1u;
      acc[e.uu[j] * 32 + lane] = a;
    }
  }
}

// Replicas [r_begin, r_end) added in order, each replica's entries read before the previous
// replica's are added.  `at(r, e)` reads replica r's entries; `adds`: this lane's chunk exists.
template <int KV, class At>
__device__ __forceinline__ void demo_add_replicas(SumCount* acc, int lane, int r_begin, int r_end, bool adds, At&& at) {
  if (r_begin >= r_end) return;
  DemoEntries<KV> cur;
  at(r_begin, cur);
  for (int r = r_begin; r < r_end; ++r) {
    DemoEntries<KV> nxt = cur;
    if (r + 1 < r_end) at(r + 1, nxt);
    if (adds) demo_add<KV>(acc, lane, cur);
    cur = nxt;
  }
}

// Unstaged DeMo replicas of the float32 / 16-bit formats are read F replicas at a time,
// their loads in flight together: F = 32 / k in the kernels for many replicas (about 160
// bytes of entries per lane), 4 in those for R <= 4.
constexpr int kFlight = 4;

template <int MODE, int MAXR, int WARPS, int KV, int FLAV>
__global__ void __launch_bounds__(WARPS * 32, 1) decode_kernel(const __grid_constant__ DecodeParams<MAXR> p) {
  using WarpSmem = DecWarpSmem<dec_stage_bytes(WARPS)>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned start (the TMA swizzle patterns are relative to 1024-byte boundaries),
  // derived by pointer arithmetic on the shared array so every access stays a shared-memory one
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WarpSmem& ws = reinterpret_cast<WarpSmem*>(base)[warp];
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + WARPS * sizeof(WarpSmem)) + 2 * warp;
  float* rcp = reinterpret_cast<float*>(base + WARPS * sizeof(WarpSmem) + WARPS * 16);
  griddep_launch_dependents();
  for (int i = threadIdx.x; i <= kMaxReplicas; i += blockDim.x) rcp[i] = p.rcp_tab[i];
  if (threadIdx.x == 0) prefetch_tmap(&p.theta);
  __syncthreads();

  // The launch may run fewer warps than the shared-memory layout holds: warps are counted
  // from the block size.
  const int nw = static_cast<int>(blockDim.x >> 5);
  const long long gw = static_cast<long long>(blockIdx.x) * nw + warp;
  const long long TW = static_cast<long long>(gridDim.x) * nw;
  if (gw >= p.ntiles) return;
  const long long ntw = (p.ntiles - 1 - gw) / TW + 1;  // tiles of this warp
  // Items: one per tile, or (group > 0) one per group of replicas on full tiles.
  const int G = (FLAV & kFlavGroups) ? p.group : 0;
  const int ngf = G > 0 ? (p.R + G - 1) / G : 1;  // items of a full tile
  const bool own_ragged = (p.nc & 31) != 0 && (p.ntiles - 1 - gw) % TW == 0;
  const long long nitems = ntw * ngf - (own_ragged ? ngf - 1 : 0);
  auto full = [&](long long t) { return (t + 1) * 32 <= p.nc; };
  // Replicas staged by item g of tile t: [r0, r1).  The last item of a tile also holds
  // the theta tile and reads the replicas [r1, R) directly (none when grouped).
  auto staged_range = [&](long long t, int g, int& r0, int& r1) {
    if (!full(t)) {
      r0 = r1 = 0;
    } else if (G > 0) {
      r0 = g * G;
      r1 = r0 + G < p.R ? r0 + G : p.R;
    } else {
      r0 = 0;
      r1 = p.nstaged;
    }
  };

  if (lane == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
#pragma unroll
  for (int u = 0; u < 32; ++u) ws.acc[u * 32 + lane] = SumCount{0.0f, 0u};
  __syncwarp();

  const uint32_t span = p.vspan + p.ispan;  // staged bytes per replica
  const uint32_t stride = p.sstride;         // their distance in the staging area (span rounded up to 16)
  constexpr bool lane_copy = (FLAV & kFlavLaneCopy) != 0;
  constexpr bool kVecWords = (FLAV & kFlavGroups) == 0;  // ternary words as vectors (see demo_read)
  // Lane copies: the staged spans of an item are units of US bytes (16, or 4 for the ternary
  // spans that are not 16-byte multiples) u = 0, 1, ... (replica u / P, byte US (u % P) of its
  // span, stored at that replica's stride); lane l copies the units l, l + 32, ...
  const int US = p.lane_unit;
  const int P = US > 0 ? static_cast<int>(span) / US : 0;
  const int step_r = P ? 32 / P : 0, step_o = P ? (32 % P) * US : 0;
  const int lane_r = P ? lane / P : 0, lane_o = P ? (lane % P) * US : 0;
  // Items are loaded strictly in order: the loads keep their own (tile, item) cursor.  The
  // whole warp runs issue(); lane 0 starts the theta tile's copy (and, without lane copies,
  // the spans' bulk copies) on the slot's barrier.  With lane copies every call commits one
  // copy group, empty past the last item: when item i is consumed, groups up to i + 1 are
  // committed, and waiting for all but the newest one completes item i's.
  long long ld_t = gw, ld_item = 0;
  int ld_g = 0, ld_slot = 0;
  auto issue = [&]() {
    if (ld_t < p.ntiles) {
      const int items = full(ld_t) ? ngf : 1;
      const bool last = ld_g == items - 1;
      int r0, r1;
      staged_range(ld_t, ld_g, r0, r1);
      uint64_t* bar = &bars[ld_slot];
      if (lane == 0) {
        const uint32_t staged = lane_copy ? 0u : (r1 - r0) * span;
        mbar_expect_tx(bar, (last ? kTileBytesF32 : 0) + staged + stall_extra(p.stall_at, gw, ld_item));
        if (last) tma_load_2d(ws.tbuf[ld_slot], &p.theta, bar, 0, static_cast<int>(ld_t * 32));
        if (!lane_copy) {
          for (int r = r0; r < r1; ++r) {
            unsigned char* d = ws.stage[ld_slot] + (r - r0) * stride;
            bulk_load(d, static_cast<const unsigned char*>(p.vals[r]) + ld_t * p.vspan, p.vspan, bar);
            if (p.ispan)
              bulk_load(d + p.vspan, static_cast<const unsigned char*>(p.idx[r]) + ld_t * p.ispan, p.ispan, bar);
          }
        }
      }
      if (lane_copy) {
        const int units = (r1 - r0) * P;
        int rr = lane_r, o = lane_o;
        for (int u = lane; u < units; u += 32) {
          const int r = r0 + rr;
          const unsigned char* src =
              o < static_cast<int>(p.vspan)
                  ? static_cast<const unsigned char*>(p.vals[r]) + ld_t * p.vspan + o
                  : static_cast<const unsigned char*>(p.idx[r]) + ld_t * p.ispan + (o - static_cast<int>(p.vspan));
          unsigned char* dst = ws.stage[ld_slot] + rr * stride + o;
          if (US == 16) {
            lane_copy16(dst, src);
          } else {
            lane_copy4(dst, src);
          }
          rr += step_r;
          o += step_o;
          if (o >= static_cast<int>(span)) {
            o -= static_cast<int>(span);
            ++rr;
          }
        }
      }
      ++ld_item;
      ld_slot ^= 1;
      if (++ld_g == items) {
        ld_g = 0;
        ld_t += TW;
      }
    }
    if (lane_copy) lane_copy_commit();
  };
  griddep_wait();  // the payloads the previous kernels wrote are visible from here on
  issue();
  issue();

  // Random / Striding, k <= 8: one replica's k values for a chunk, padded with zeros to 8
  // (a vector load where the format allows), and the running sums per draw over the items
  // of the current tile.
  const bool vec_draws = p.wire != kWireTernary && vector_kd(p.k);
  auto load_draws = [&](const void* vbase, long long cc, long long tl, float (&pv)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) pv[j] = 0.0f;
    if (vec_draws) {
      uint32_t ilo, ihi;
      load_payload(vbase, nullptr, p.wire, cc, p.k, pv, ilo, ihi);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < p.k) pv[j] = payload_value(vbase, p.wire, cc, tl, lane, p.k, j);
    }
  };
  float rsum[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) rsum[j] = 0.0f;

  long long t = gw;
  int g = 0;
  for (long long item = 0; item < nitems; ++item) {
    const int s = static_cast<int>(item & 1);
    const uint32_t par = static_cast<uint32_t>((item >> 1) & 1);
    const long long row0 = t * 32;
    const long long c = row0 + lane;
    const bool valid = c < p.nc;
    const int items = full(t) ? ngf : 1;
    const bool last = g == items - 1;
    int r0, ns;  // replicas staged by this item: [r0, ns)
    staged_range(t, g, r0, ns);

    const bool ok = mbar_wait_bounded(&bars[s], par);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) {
        atomicOr(p.fault, kFaultLoadTimeout);
        for (long long it = item; it < item + 2 && it < nitems; ++it)
          mbar_wait_bounded(&bars[it & 1], static_cast<uint32_t>((it >> 1) & 1));
      }
      if (lane_copy) lane_copy_wait<0>();
      __syncwarp();
      return;
    }
    if (lane_copy) {
      lane_copy_wait<1>();  // this item's group (the newer one is the next item's)
      __syncwarp();
    }

    if constexpr (MODE != kModeDemo) {
      // Random / Striding with k <= 8 in groups: the staged replicas of this item join the
      // running per-draw sums (the replicas of a tile's items in order)
      if (G > 0 && p.k <= 8) {
        for (int r = r0; r < ns; ++r) {
          float pv[8];
          load_draws(ws.stage[s] + (r - r0) * stride, lane, 0, pv);
#pragma unroll
          for (int j = 0; j < 8; ++j) rsum[j] += pv[j];
        }
      }
    }
    if constexpr (MODE == kModeDemo) {
      if constexpr (KV < 0) {
        demo_add_replicas<KV>(ws.acc, lane, r0, ns, true, [&](int r, DemoEntries<KV>& e) {
          const unsigned char* sv = ws.stage[s] + (r - r0) * stride;
          demo_read<KV, kVecWords>(e, sv, sv + p.vspan, p.wire, lane, 0, lane);
        });
      } else {
        for (int r = r0; r < ns; ++r) {
          const unsigned char* sv = ws.stage[s] + (r - r0) * stride;
          demo_accumulate<KV>(ws.acc, lane, sv, sv + p.vspan, p.wire, p.k, lane, 0, true, true);
        }
      }
    }
    if (!last) {
      // a group of replicas only: the slot is read, refill it with the load two items on
      fence_proxy_async_smem();
      __syncwarp();
      issue();
      ++g;
      continue;
    }

    float th[32];
    load_row_f32(ws.tbuf[s], lane, th);

    float Q[32];
    if constexpr (MODE == kModeDemo) {
      const long long tile = row0 >> 5;
      const bool reads = valid || p.wire == kWireTernary;
      if constexpr (KV < 0) {
        // the ternary words belong to the whole tile and every lane reads them
        demo_add_replicas<KV>(ws.acc, lane, ns, p.R, valid, [&](int r, DemoEntries<KV>& e) {
          if (reads) demo_read<KV, kVecWords>(e, p.vals[r], p.idx[r], p.wire, c, tile, lane);
        });
      } else if constexpr (KV > 0) {
        // replicas not staged, read from global memory F at a time (their loads in flight
        // together), then added in replica order
        constexpr int F = MAXR > kSmallReplicas ? 32 / KV : kFlight;
        int r = ns;
        for (; r + F <= p.R; r += F) {
          DemoEntries<KV> e[F];
#pragma unroll
          for (int q = 0; q < F; ++q)
            if (valid) demo_read<KV>(e[q], p.vals[r + q], p.idx[r + q], p.wire, c, tile, lane);
          if (valid) {
#pragma unroll
            for (int q = 0; q < F; ++q) demo_add<KV>(ws.acc, lane, e[q]);
          }
        }
        for (; r < p.R; ++r)
          demo_accumulate<KV>(ws.acc, lane, p.vals[r], p.idx[r], p.wire, p.k, c, tile, valid, valid);
      } else {
        for (int r = ns; r < p.R; ++r)
          demo_accumulate<KV>(ws.acc, lane, p.vals[r], p.idx[r], p.wire, p.k, c, tile, valid, reads);
      }
      if (p.R * p.k > kMaxReplicas) {
        // Valid payloads count at most R entries per slot; a malformed one (an index
        // repeated within a chunk) can count more than the reciprocal table covers.
        // Such a slot is replaced by its mean and a count of one (rcp[1] = 1), the
        // reciprocal rounded as the table's entries are.
        uint32_t most = 0;
#pragma unroll
        for (int u = 0; u < 32; ++u) most = umax32(most, ws.acc[u * 32 + lane].cnt);
        if (__any_sync(0xffffffffu, most > kMaxReplicas)) {
#pragma unroll 1
          for (int u = 0; u < 32; ++u) {
            const SumCount a = ws.acc[u * 32 + lane];
            if (a.cnt > kMaxReplicas)
              ws.acc[u * 32 + lane] = SumCount{a.sum * __frcp_rn(static_cast<float>(a.cnt)), 1u};
          }
        }
      }
      float Y[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const SumCount a = ws.acc[u * 32 + lane];
        Y[u] = a.sum * rcp[a.cnt];
      }
#pragma unroll
      for (int u = 0; u < 32; ++u) ws.acc[u * 32 + lane] = SumCount{0.0f, 0u};
      dct32_inverse(Y, Q);
    } else {
      // Random / Striding: every replica sent the same positions; Q = mean at those positions.
      float* qs = reinterpret_cast<float*>(ws.acc);  // [i][lane] scratch (first 4 KB)
#pragma unroll
      for (int i = 0; i < 32; ++i) qs[i * 32 + lane] = 0.0f;
      const long long tile = row0 >> 5;
      if (p.k <= 8) {
        // k <= 8: sum the replicas' k values per draw (replicas in order: the staged ones from
        // shared memory, item by item, then the others from global memory, four replicas'
        // loads in flight at a time; one vector load per replica where the format allows),
        // then place each sum at its draw's position, with the draws unrolled.
        float (&sum)[8] = rsum;
        auto& load_one = load_draws;
        if (G == 0) {
          for (int r = 0; r < ns; ++r) {
            float pv[8];
            load_one(ws.stage[s] + r * stride, lane, 0, pv);
#pragma unroll
            for (int j = 0; j < 8; ++j) sum[j] += pv[j];
          }
        }
        const bool reads = valid || p.wire == kWireTernary;  // rows past the end read nothing
        int r = ns;
        if constexpr (KV > 0) {
          // k compiled (the receiver of many replicas, none staged): 32 / k replicas' vector
          // loads in flight together, k sums
          constexpr int F = 32 / KV;
          for (; r + F <= p.R; r += F) {
            float pv[F][KV];
#pragma unroll
            for (int q = 0; q < F; ++q) {
              if (reads) {
                load_values<KV>(p.vals[r + q], p.wire, c, pv[q]);
              } else {
#pragma unroll
                for (int j = 0; j < KV; ++j) pv[q][j] = 0.0f;
              }
            }
#pragma unroll
            for (int q = 0; q < F; ++q)
#pragma unroll
              for (int j = 0; j < KV; ++j) sum[j] += pv[q][j];
          }
        } else {
          for (; r + 4 <= p.R; r += 4) {
            float pv[4][8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (reads) {
                load_one(p.vals[r + q], c, tile, pv[q]);
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) pv[q][j] = 0.0f;
              }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int j = 0; j < 8; ++j) sum[j] += pv[q][j];
          }
        }
        for (; r < p.R; ++r) {
          float pv[8];
          if (reads) {
            load_one(p.vals[r], c, tile, pv);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) pv[j] = 0.0f;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) sum[j] += pv[j];
        }
        uint64_t hc = 0;
        uint32_t free_mask = 0xffffffffu;
        if constexpr (MODE == kModeRandom) hc = splitmix64(p.hbase ^ static_cast<uint64_t>(c + p.chunk0));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j < p.k) {
            int pos;
            if constexpr (MODE == kModeRandom) {
              pos = random_draw(hc, j, free_mask);
            } else {
              pos = stride_position(p.stride_o, p.stride_ns, j);
            }
            qs[pos * 32 + lane] = sum[j] * p.rcpR;
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) sum[j] = 0.0f;
      } else {
        const bool reads = valid || p.wire == kWireTernary;  // as in the DeMo branch
        auto take = [&](int j, int pos) {
          float sum = 0.0f;
          for (int r = 0; r < ns; ++r) sum += payload_value(ws.stage[s] + r * stride, p.wire, lane, 0, lane, p.k, j);
          for (int r = ns; r < p.R; ++r) sum += reads ? payload_value(p.vals[r], p.wire, c, tile, lane, p.k, j) : 0.0f;
          if (valid) qs[pos * 32 + lane] = sum * p.rcpR;
        };
        if constexpr (MODE == kModeRandom) {
          random_draws(p.hbase, static_cast<uint64_t>(c + p.chunk0), p.k, take);
        } else {
          for (int j = 0; j < p.k; ++j) take(j, stride_position(p.stride_o, p.stride_ns, j));
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) Q[i] = qs[i * 32 + lane];
    }

#pragma unroll
    for (int i = 0; i < 32; ++i) th[i] = __fmaf_rn(-p.lr, Q[i], th[i]);
    __syncwarp();  // every lane has read its theta row
    store_tile_coalesced(ws.tbuf[s], lane, th, p.theta_ptr, row0, p.nc);
    fence_proxy_async_smem();
    __syncwarp();
    issue();
    g = 0;
    t += TW;
  }
}

// Random and Striding decodes compiled for k (kv in {1, 2, 4, 8}, float32 or 16-bit values)
// exist only where they run: the many-replica kernels of the 11-warp plain shape, whose
// replicas are all read directly; every other kernel takes k at run time (kv = 0).
template <int MAXR, int WARPS, int FLAV>
constexpr bool kSchemeKV = MAXR > kSmallReplicas && WARPS == kDecShapes[0] && FLAV == kFlavPlain;

template <int MAXR, int WARPS, int FLAV>
static cudaError_t launch_decode_w(const DecodeParams<MAXR>& p, int mode, int kv, int active, int grid,
                                   cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(active * 32);
  cfg.dynamicSmemBytes = persistent_smem(dec_smem(WARPS));
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (mode) {
    case kModeDemo:
      switch (kv) {
        case 1: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, MAXR, WARPS, 1, FLAV>, p);
        case 2: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, MAXR, WARPS, 2, FLAV>, p);
        case 4: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, MAXR, WARPS, 4, FLAV>, p);
        case 8: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, MAXR, WARPS, 8, FLAV>, p);
        case -1: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, MAXR, WARPS, -1, FLAV>, p);
        case -2: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, MAXR, WARPS, -2, FLAV>, p);
        case -4: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, MAXR, WARPS, -4, FLAV>, p);
        case -8: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, MAXR, WARPS, -8, FLAV>, p);
        default: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, MAXR, WARPS, 0, FLAV>, p);
      }
    case kModeRandom:
      if constexpr (kSchemeKV<MAXR, WARPS, FLAV>) {
        switch (kv) {
          case 1: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeRandom, MAXR, WARPS, 1, FLAV>, p);
          case 2: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeRandom, MAXR, WARPS, 2, FLAV>, p);
          case 4: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeRandom, MAXR, WARPS, 4, FLAV>, p);
          case 8: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeRandom, MAXR, WARPS, 8, FLAV>, p);
          default: break;
        }
      }
      return cudaLaunchKernelEx(&cfg, decode_kernel<kModeRandom, MAXR, WARPS, 0, FLAV>, p);
    case kModeStride:
      if constexpr (kSchemeKV<MAXR, WARPS, FLAV>) {
        switch (kv) {
          case 1: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeStride, MAXR, WARPS, 1, FLAV>, p);
          case 2: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeStride, MAXR, WARPS, 2, FLAV>, p);
          case 4: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeStride, MAXR, WARPS, 4, FLAV>, p);
          case 8: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeStride, MAXR, WARPS, 8, FLAV>, p);
          default: break;
        }
      }
      return cudaLaunchKernelEx(&cfg, decode_kernel<kModeStride, MAXR, WARPS, 0, FLAV>, p);
    default: return cudaErrorInvalidValue;
  }
}

// Every CTA shape of one flavour.
template <int MAXR, int FLAV>
static cudaError_t launch_decode_shapes(const DecodeParams<MAXR>& p, int mode, int warps, int kv, int active,
                                        int grid, cudaStream_t st) {
  if (active < 1 || active > warps) return cudaErrorInvalidValue;
  if (warps == 11) return launch_decode_w<MAXR, 11, FLAV>(p, mode, kv, active, grid, st);
  if (warps == 10) return launch_decode_w<MAXR, 10, FLAV>(p, mode, kv, active, grid, st);
  if (warps == 9) return launch_decode_w<MAXR, 9, FLAV>(p, mode, kv, active, grid, st);
  if (warps == 8) return launch_decode_w<MAXR, 8, FLAV>(p, mode, kv, active, grid, st);
  return cudaErrorInvalidValue;
}

template <class K>
static cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int MAXR, int WARPS, int FLAV>
static cudaError_t prepare_decode_w() {
  const int bytes = static_cast<int>(persistent_smem(dec_smem(WARPS)));
  cudaError_t e = set_smem(decode_kernel<kModeDemo, MAXR, WARPS, 0, FLAV>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeDemo, MAXR, WARPS, 1, FLAV>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeDemo, MAXR, WARPS, 2, FLAV>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeDemo, MAXR, WARPS, 4, FLAV>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeDemo, MAXR, WARPS, 8, FLAV>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeDemo, MAXR, WARPS, -1, FLAV>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeDemo, MAXR, WARPS, -2, FLAV>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeDemo, MAXR, WARPS, -4, FLAV>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeDemo, MAXR, WARPS, -8, FLAV>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeRandom, MAXR, WARPS, 0, FLAV>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeStride, MAXR, WARPS, 0, FLAV>, bytes);
  if constexpr (kSchemeKV<MAXR, WARPS, FLAV>) {
    if (e == cudaSuccess) e = set_smem(decode_kernel<kModeRandom, MAXR, WARPS, 1, FLAV>, bytes);
    if (e == cudaSuccess) e = set_smem(decode_kernel<kModeRandom, MAXR, WARPS, 2, FLAV>, bytes);
    if (e == cudaSuccess) e = set_smem(decode_kernel<kModeRandom, MAXR, WARPS, 4, FLAV>, bytes);
    if (e == cudaSuccess) e = set_smem(decode_kernel<kModeRandom, MAXR, WARPS, 8, FLAV>, bytes);
    if (e == cudaSuccess) e = set_smem(decode_kernel<kModeStride, MAXR, WARPS, 1, FLAV>, bytes);
    if (e == cudaSuccess) e = set_smem(decode_kernel<kModeStride, MAXR, WARPS, 2, FLAV>, bytes);
    if (e == cudaSuccess) e = set_smem(decode_kernel<kModeStride, MAXR, WARPS, 4, FLAV>, bytes);
    if (e == cudaSuccess) e = set_smem(decode_kernel<kModeStride, MAXR, WARPS, 8, FLAV>, bytes);
  }
  return e;
}

template <int MAXR, int FLAV>
static cudaError_t prepare_decode_shapes() {
  cudaError_t e = prepare_decode_w<MAXR, 11, FLAV>();
  if (e == cudaSuccess) e = prepare_decode_w<MAXR, 10, FLAV>();
  if (e == cudaSuccess) e = prepare_decode_w<MAXR, 9, FLAV>();
  if (e == cudaSuccess) e = prepare_decode_w<MAXR, 8, FLAV>();
  return e;
}

// The many-replica flavours, compiled in their own translation units.
cudaError_t launch_decode_lane_copy(const DecodeParams<kMaxReplicas>& p, int mode, int warps, int kv, int active,
                                    int grid, cudaStream_t st);
cudaError_t launch_decode_groups(const DecodeParams<kMaxReplicas>& p, int mode, int warps, int kv, int flavor,
                                 int active, int grid, cudaStream_t st);
cudaError_t launch_decode_lane_copy_small(const DecodeParams<kSmallReplicas>& p, int mode, int warps, int kv,
                                          int active, int grid, cudaStream_t st);
cudaError_t prepare_decode_lane_copy();
cudaError_t prepare_decode_groups();

}  // namespace demo
