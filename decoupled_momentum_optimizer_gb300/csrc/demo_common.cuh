// Device building blocks shared by the DeMo shard-step kernels (sm_103a).
//
// Layout on chip: one warp owns a tile of 32 chunks; lane i owns chunk i of
// the tile (32 consecutive float32 values = one 128-byte row).  Tiles of g, m
// and theta arrive through TMA (cp.async.bulk.tensor, 2-D, 128-byte swizzle
// for float32 rows, 64-byte swizzle for bfloat16 rows), so that each lane can
// read its own row with conflict-free 16-byte shared-memory loads.  All
// per-chunk arithmetic (momentum, 32-point DCT, top-k, feedback, update) runs
// in the lane's registers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dct32_factors.cuh"

namespace demo {

constexpr int kChunk = 32;
constexpr int kTileBytesF32 = 32 * 128;  // 32 rows x 32 float32
constexpr int kTileBytesBF16 = 32 * 64;  // 32 rows x 32 bfloat16
constexpr unsigned kFaultLoadTimeout = 1u;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait

enum { kModeDemo = 0, kModeRandom = 1, kModeStride = 2, kModeDiloco = 3 };
enum { kWireF32 = 0, kWireTernary = 1, kWireBF16 = 2, kWireF16 = 3 };

// The value a receiver decodes from v sent in `wire` (nearest-even 16-bit rounding).
__device__ __forceinline__ float wire_round(float v, int wire) {
  if (wire == kWireBF16) return __bfloat162float(__float2bfloat16_rn(v));
  if (wire == kWireF16) return __half2float(__float2half_rn(v));
  return v;
}

__device__ __forceinline__ uint32_t wire_bits16(float v, int wire) {
  if (wire == kWireBF16) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return __half_as_ushort(__float2half_rn(v));
}

__device__ __forceinline__ float wire_from_bits16(uint32_t b, int wire) {
  if (wire == kWireBF16) return __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(b)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
}

// ----------------------------------------------------------------------------
// PTX wrappers: shared-memory addresses, mbarriers, TMA, proxy fences
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar`; gives up after kWaitLimitNs and reports it.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Test hook of the give-up path above: when stall_at = 1 + i (0 = off), the load of item i of
// global warp 0 announces kStallBytes more than it delivers, so its barrier never completes
// and the warp's bounded wait runs out, exactly as for a copy that never lands.  Every copy
// still lands; the warp reports the fault, waits (bounded) for its copies and returns.
constexpr uint32_t kStallBytes = 16;
__device__ __forceinline__ uint32_t stall_extra(long long stall_at, long long gw, long long item) {
  return (stall_at != 0 && gw == 0 && item + 1 == stall_at) ? kStallBytes : 0u;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
      : "memory");
}

// 1-D bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to shared memory, counted on `bar`'s transaction count.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch.  A tile kernel launched with programmatic stream
// serialisation may start while the previous kernel of its stream is still running:
// griddep_launch_dependents lets the next kernel's CTAs start their prologue on the SMs
// this grid frees, and griddep_wait blocks until the previous grid has completed and its
// memory operations are visible.  Each tile kernel waits before its first global-memory
// access, so every read and write stays ordered after the previous kernel, and since every
// kernel in the chain waits, after all earlier ones.  (The one exception is an encode the
// host marks as sharing no buffers with the kernels around it: it waits only before exiting,
// see encode_kernel.)  Without the launch attribute both are no-ops.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------------------
// Swizzled row access.  TMA's 128-byte swizzle stores 16-byte unit j of row r
// at unit j ^ (r & 7) (tile base 1024-byte aligned); the 64-byte swizzle of a
// 64-byte row stores unit j at j ^ ((r >> 1) & 3).
// ----------------------------------------------------------------------------

__device__ __forceinline__ void load_row_f32(const float* tile, int row, float (&v)[32]) {
  const char* base = reinterpret_cast<const char*>(tile) + row * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 q = *reinterpret_cast<const float4*>(base + ((j ^ (row & 7)) << 4));
    v[4 * j + 0] = q.x;
    v[4 * j + 1] = q.y;
    v[4 * j + 2] = q.z;
    v[4 * j + 3] = q.w;
  }
}

__device__ __forceinline__ void store_row_f32(float* tile, int row, const float (&v)[32]) {
  char* base = reinterpret_cast<char*>(tile) + row * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    *reinterpret_cast<float4*>(base + ((j ^ (row & 7)) << 4)) =
        make_float4(v[4 * j + 0], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }
}

// Write the warp's tile (row `lane` held by each lane in v) to rows [row0, row0 + 32)
// of a row-major [nrows][32] float array.  The rows go through the swizzled
// 4 KB shared tile `buf` and are read back transposed, so every 16-byte global
// store instruction covers 512 contiguous bytes.  Rows at or past nrows are not
// written.  `buf` may be reused as soon as the call returns and the warp has
// synchronised.
__device__ __forceinline__ void store_tile_coalesced(float* buf, int lane, const float (&v)[32], float* gbase,
                                                     long long row0, long long nrows) {
  store_row_f32(buf, lane, v);
  __syncwarp();
  const char* b = reinterpret_cast<const char*>(buf);
  const int j = lane & 7;
  float4* dst = reinterpret_cast<float4*>(gbase + row0 * 32) + (lane >> 3) * 8 + j;
  const int live = nrows - row0 >= 32 ? 32 : static_cast<int>(nrows - row0);  // rows of the tile inside the array
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int r = q * 4 + (lane >> 3);
    const float4 val = *reinterpret_cast<const float4*>(b + r * 128 + ((j ^ (r & 7)) << 4));
    if (r < live) dst[q * 32] = val;
  }
}

__device__ __forceinline__ void load_row_bf16(const void* tile, int row, float (&v)[32]) {
  const char* base = reinterpret_cast<const char*>(tile) + row * 64;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 q = *reinterpret_cast<const uint4*>(base + ((j ^ ((row >> 1) & 3)) << 4));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[8 * j + 2 * e + 0] = __uint_as_float(w[e] << 16);
      v[8 * j + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  }
}

template <bool BF16>
__device__ __forceinline__ void load_row_grad(const void* tile, int row, float (&v)[32]) {
  if constexpr (BF16) {
    load_row_bf16(tile, row, v);
  } else {
    load_row_f32(reinterpret_cast<const float*>(tile), row, v);
  }
}

// ----------------------------------------------------------------------------
// Orthonormal 32-point DCT-II (forward) and its transpose DCT-III (inverse),
// by the recursive even/odd split: the odd outputs of a size-N stage are the
// DCT-IV (size N/2) of the differences x_n - x_{N-1-n}, the even outputs the
// size-N/2 DCT-II of the sums.  All DCT-IV blocks carry the 1/4 orthonormal
// factor; the DC and the 2-point stage use sqrt(1/32).  404 flops per chunk.
// ----------------------------------------------------------------------------

__device__ __forceinline__ void dct32_forward(const float (&x)[32], float (&X)[32]) {
  float s16[16], d16[16], o16[16];
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    s16[n] = x[n] + x[31 - n];
    d16[n] = x[n] - x[31 - n];
  }
  demo_dct4_16(d16, o16);
#pragma unroll
  for (int j = 0; j < 16; ++j) X[2 * j + 1] = o16[j];

  float s8[8], d8[8], o8[8];
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    s8[n] = s16[n] + s16[15 - n];
    d8[n] = s16[n] - s16[15 - n];
  }
  demo_dct4_8(d8, o8);
#pragma unroll
  for (int j = 0; j < 8; ++j) X[4 * j + 2] = o8[j];

  float s4[4], d4[4], o4[4];
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    s4[n] = s8[n] + s8[7 - n];
    d4[n] = s8[n] - s8[7 - n];
  }
  demo_dct4_4(d4, o4);
#pragma unroll
  for (int j = 0; j < 4; ++j) X[8 * j + 4] = o4[j];

  float s2[2], d2[2], o2[2];
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    s2[n] = s4[n] + s4[3 - n];
    d2[n] = s4[n] - s4[3 - n];
  }
  demo_dct4_2(d2, o2);
  X[8] = o2[0];
  X[24] = o2[1];
  X[0] = (s2[0] + s2[1]) * DEMO_DCT_C0;
  X[16] = (s2[0] - s2[1]) * DEMO_DCT_C0;
}

__device__ __forceinline__ void dct32_inverse(const float (&Y)[32], float (&q)[32]) {
  float e2[2];
  e2[0] = (Y[0] + Y[16]) * DEMO_DCT_C0;
  e2[1] = (Y[0] - Y[16]) * DEMO_DCT_C0;

  float z2[2] = {Y[8], Y[24]}, o2[2];
  demo_dct4_2(z2, o2);
  float e4[4];
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    e4[n] = e2[n] + o2[n];
    e4[3 - n] = e2[n] - o2[n];
  }

  float z4[4], o4[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) z4[j] = Y[8 * j + 4];
  demo_dct4_4(z4, o4);
  float e8[8];
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    e8[n] = e4[n] + o4[n];
    e8[7 - n] = e4[n] - o4[n];
  }

  float z8[8], o8[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) z8[j] = Y[4 * j + 2];
  demo_dct4_8(z8, o8);
  float e16[16];
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    e16[n] = e8[n] + o8[n];
    e16[15 - n] = e8[n] - o8[n];
  }

  float z16[16], o16[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) z16[j] = Y[2 * j + 1];
  demo_dct4_16(z16, o16);
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    q[n] = e16[n] + o16[n];
    q[31 - n] = e16[n] - o16[n];
  }
}

// ----------------------------------------------------------------------------
// Exact top-k of |X| with ties to the lowest index.
//
// Keys are the IEEE bits of |X_u| (monotone as unsigned integers).  Fast path:
// k-1 rounds each find the largest key strictly below the previous threshold
// (a wrapped subtraction maps "key < T" to the upper half of the unsigned
// range, so one max does the filtering); the mask {key >= T_k} is the answer
// whenever it has exactly k members.  Otherwise some keys tie and an exact
// k-round scan (strictly greater wins, so the lowest index wins ties) decides.
// Returns the mask of kept slots and Xs = X on the kept slots, 0 elsewhere.
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t umax32(uint32_t a, uint32_t b) { return a > b ? a : b; }

// Largest of 32 unsigned keys: a tree of 3-input maxima.
__device__ __forceinline__ uint32_t max_tree(const uint32_t (&v)[32]) {
  uint32_t a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = __vimax3_u32(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  a[10] = umax32(v[30], v[31]);
  const uint32_t b0 = __vimax3_u32(a[0], a[1], a[2]);
  const uint32_t b1 = __vimax3_u32(a[3], a[4], a[5]);
  const uint32_t b2 = __vimax3_u32(a[6], a[7], a[8]);
  const uint32_t b3 = umax32(a[9], a[10]);
  return __vimax3_u32(b0, b1, umax32(b2, b3));
}

// Largest key strictly below T, as T + max_u (key_u - T) over the wrapped
// differences: keys below T map to [2^32 - T, 2^32), all others to [0, 2^31),
// so one add-and-max per key filters and maximises at once.  Returns T itself
// when no key is below T.
__device__ __forceinline__ uint32_t next_below(const uint32_t (&key)[32], uint32_t T) {
  const uint32_t negT = 0u - T;
  uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
#pragma unroll
  for (int u = 0; u < 32; u += 4) {
    m0 = __viaddmax_u32(key[u + 0], negT, m0);
    m1 = __viaddmax_u32(key[u + 1], negT, m1);
    m2 = __viaddmax_u32(key[u + 2], negT, m2);
    m3 = __viaddmax_u32(key[u + 3], negT, m3);
  }
  const uint32_t best = __vimax3_u32(m0, m1, umax32(m2, m3));
  return best >= 0x80000000u ? best + T : T;
}

__device__ __forceinline__ uint32_t topk_select(const float (&X)[32], int k, float (&Xs)[32]) {
  if (k >= 32) {
#pragma unroll
    for (int u = 0; u < 32; ++u) Xs[u] = X[u];
    return 0xffffffffu;
  }
  uint32_t key[32];
#pragma unroll
  for (int u = 0; u < 32; ++u) key[u] = __float_as_uint(X[u]) & 0x7fffffffu;

  uint32_t T = max_tree(key);
  for (int r = 1; r < k; ++r) T = next_below(key, T);
  uint32_t M = 0;
#pragma unroll
  for (int u = 0; u < 32; ++u) M |= static_cast<uint32_t>(key[u] >= T) << u;

  if (__popc(M) != k) {
    // Exact ties decide the selection: k rounds of "largest not yet taken".
    M = 0;
    for (int r = 0; r < k; ++r) {
      uint32_t best = 0;
      int bu = -1;
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const bool take = !((M >> u) & 1u) && (bu < 0 || key[u] > best);
        best = take ? key[u] : best;
        bu = take ? u : bu;
      }
      M |= 1u << bu;
    }
  }
#pragma unroll
  for (int u = 0; u < 32; ++u) Xs[u] = ((M >> u) & 1u) ? X[u] : 0.0f;
  return M;
}

// Ternary sign: -1, 0 or +1 (NaN -> 0).
__device__ __forceinline__ float sign3(float v) { return v > 0.0f ? 1.0f : (v < 0.0f ? -1.0f : 0.0f); }

// ----------------------------------------------------------------------------
// Counter-based positions (Random and Striding schemes)
// ----------------------------------------------------------------------------

// splitmix64 output function of state z (Steele, Lea & Flood 2014; Vigna).
__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Position of the r-th (0-based) set bit of v; v must have more than r set bits.
__device__ __forceinline__ int nth_set_bit(uint32_t v, int r) {
  int pos = 0;
  int c = __popc(v & 0xffffu);
  if (r >= c) { r -= c; v >>= 16; pos += 16; }
  c = __popc(v & 0xffu);
  if (r >= c) { r -= c; v >>= 8; pos += 8; }
  c = __popc(v & 0xfu);
  if (r >= c) { r -= c; v >>= 4; pos += 4; }
  c = __popc(v & 0x3u);
  if (r >= c) { r -= c; v >>= 2; pos += 2; }
  c = static_cast<int>(v & 1u);
  if (r >= c) pos += 1;
  return pos;
}

// Random scheme: k draws for global chunk c by partial Fisher-Yates.  hbase is
// sm(sm(seed) ^ step), hoisted to the host.  Calls f(j, position) for each draw
// j in order and returns the mask of the k positions.
// Draw j of a chunk whose hash is hc: the r-th still free position, r uniform
// in [0, 32 - j); the position is taken out of free_mask.
__device__ __forceinline__ int random_draw(uint64_t hc, int j, uint32_t& free_mask) {
  const uint64_t h = splitmix64(hc ^ static_cast<uint64_t>(j));
  const uint32_t r = static_cast<uint32_t>(((h >> 32) * static_cast<uint64_t>(32 - j)) >> 32);
  const int p = nth_set_bit(free_mask, static_cast<int>(r));
  free_mask &= ~(1u << p);
  return p;
}

template <class F>
__device__ __forceinline__ uint32_t random_draws(uint64_t hbase, uint64_t c, int k, F&& f) {
  const uint64_t hc = splitmix64(hbase ^ c);
  uint32_t free_mask = 0xffffffffu, sel = 0;
  for (int j = 0; j < k; ++j) {
    const int p = random_draw(hc, j, free_mask);
    sel |= 1u << p;
    f(j, p);
  }
  return sel;
}

__device__ __forceinline__ uint32_t random_mask(uint64_t hbase, uint64_t c, int k) {
  return random_draws(hbase, c, k, [](int, int) {});
}

// Striding scheme: positions o + ns * j, ns = 32 / k, o = step mod ns.
__device__ __forceinline__ int stride_position(int o, int ns, int j) { return o + ns * j; }

}  // namespace demo
