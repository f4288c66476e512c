// C ABI of the DeMo shard step: argument checks, TMA tensor maps, launches.
// The operations and their sources are described in include/demo.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/demo.h"
#include "demo_common.cuh"
#include "demo_launch.h"

namespace {

using namespace demo;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxN = int64_t(1) << 35;  // keeps every row coordinate within int32

constexpr int kMaxBlocks = 64;  // blocks of the pipelined step

struct DeviceState {
  std::atomic<bool> ready{false};  // set last by demo_init (release), read by every call (acquire)
  int sms = 0;
  unsigned int* fault = nullptr;
  cudaEvent_t ev_enc[kMaxBlocks];  // block b encoded (compute stream)
  cudaEvent_t ev_xch[kMaxBlocks];  // block b exchanged (communication stream)
  // Held while one pipelined call enqueues its work: the event pool is shared, and a
  // wait takes the event's last record at the time it is enqueued, so calls from
  // several host threads stay correct when their enqueue sequences do not interleave.
  std::mutex pipeline_mu;
  // Test hook of the kernels' bounded waits (demo_test_stall_next_launch): 1 + the item whose
  // load the next tile-kernel launch makes stall, 0 = none; taken (and cleared) by that launch.
  std::atomic<long long> stall_at{0};
};

DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
std::mutex g_mu;

__device__ unsigned int g_fault_word;

// splitmix64 output function (Steele, Lea & Flood 2014; Vigna's splitmix64.c).
uint64_t splitmix64_host(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

int check_shape(int64_t n, int chunk, int k, int mode, int diloco_period) {
  if (chunk != DEMO_CHUNK) return DEMO_EINVAL;
  if (n <= 0 || n % DEMO_CHUNK != 0 || n > kMaxN) return DEMO_EINVAL;
  if (mode < DEMO_MODE_DEMO || mode > DEMO_MODE_DILOCO) return DEMO_EINVAL;
  if (mode == DEMO_MODE_DILOCO) {
    if (diloco_period < 1) return DEMO_EINVAL;
  } else {
    if (k < 1 || k > DEMO_CHUNK) return DEMO_EINVAL;
    if (mode == DEMO_MODE_STRIDE && DEMO_CHUNK % k != 0) return DEMO_EINVAL;
  }
  return DEMO_OK;
}

bool valid_wire(int wire) { return wire >= DEMO_WIRE_F32 && wire <= DEMO_WIRE_F16; }

int current_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DEMO_ENOTINIT;
  }
  if (dev < 0 || dev >= kMaxDevices || !g_dev[dev].ready.load(std::memory_order_acquire)) return DEMO_ENOTINIT;
  *out = &g_dev[dev];
  return DEMO_OK;
}

bool diloco_sync(uint64_t step, int period) { return (step + 1) % static_cast<uint64_t>(period) == 0; }

// [nc rows x 32 columns] view of a flat shard; boxes of 32 x 32 elements.
bool make_map(CUtensorMap* map, const void* ptr, int64_t nc, bool bf16) {
  const cuuint64_t dims[2] = {32, static_cast<cuuint64_t>(nc)};
  const cuuint64_t strides[1] = {bf16 ? 64ull : 128ull};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                              const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              bf16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Launch shape of a tile kernel: the build (`inst` warps: its shared-memory layout and
// register budget), the warps that run per CTA (`active`) and the grid.
struct TileShape {
  int inst, active, grid;
};

// Most tiles per warp for which a shard counts as small (see tile_shape).
constexpr int64_t kLatencyTilesPerWarp = 3;

// Large shards stream HBM: one CTA of `warps` warps per SM, the fewest warps that cover
// the compute per item (chosen per mode), so that fewer requests are in flight once HBM is
// saturated.  A small shard is a few tiles per warp, and its time is the longest chain of
// tiles any warp walks (each tile is R + 1 dependent items).  There every SM gets a CTA and
// each warp m = ceil(ntiles / (SMs * inst)) tiles, with the fewest warps per CTA that reach
// m: they share the SM's issue slots with the fewest other warps.  Any warp count up to the
// build's fits its registers, so `inst` is the widest build (11 warps for the fused step
// and the encode; the decode keeps the build its payload staging needs).
TileShape tile_shape(int warps, int widest, int64_t ntiles, const DeviceState* st) {
  const int64_t S = st->sms;
  const int64_t m = (ntiles + S * widest - 1) / (S * widest);
  if (m <= kLatencyTilesPerWarp) {
    const int active = static_cast<int>((ntiles + m * S - 1) / (m * S));
    const int64_t grid = (ntiles + active - 1) / active;
    return {widest, active, static_cast<int>(grid < S ? grid : S)};
  }
  const int64_t want = (ntiles + warps - 1) / warps;
  return {warps, warps, static_cast<int>(want < S ? want : S)};
}

template <class P>
void fill_selection(P& p, int mode, int k, uint64_t seed, uint64_t step) {
  p.hbase = splitmix64_host(splitmix64_host(seed) ^ step);
  p.stride_o = 0;
  p.stride_ns = 1;
  if (mode == DEMO_MODE_STRIDE) {
    p.stride_ns = DEMO_CHUNK / k;
    p.stride_o = static_cast<int>(step % static_cast<uint64_t>(p.stride_ns));
  }
}

template <class P>
void fill_rcp(P& p) {
  p.rcp_tab[0] = 0.0f;
  for (int c = 1; c <= kMaxReplicas; ++c) p.rcp_tab[c] = 1.0f / static_cast<float>(c);
}

unsigned int stride_mask(int o, int ns, int k) {
  unsigned int m = 0;
  for (int j = 0; j < k; ++j) m |= 1u << (o + ns * j);
  return m;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? DEMO_OK : DEMO_ECUDA; }

// DiLoCo between syncs: only the momenta move, m_r <- beta m_r + g_r, an elementwise pass
// with no tiles (the tile kernels would compute the same FMA per element).
template <int MAXR>
int run_momentum(DeviceState* st, int64_t n, float beta, int R, const void* const* g, int grad_dtype,
                 float* const* m, cudaStream_t stream) {
  MomentumParams<MAXR> p;
  std::memset(&p, 0, sizeof(p));
  for (int r = 0; r < R; ++r) {
    p.g[r] = g[r];
    p.m[r] = m[r];
  }
  p.n4 = n / 4;
  p.R = R;
  p.beta = beta;
  const bool bf16 = grad_dtype == DEMO_GRAD_BF16;
  cudaError_t e;
  if constexpr (MAXR == kSmallReplicas) {
    e = launch_momentum_small(p, bf16, st->sms, stream);
  } else {
    e = launch_momentum_large(p, bf16, st->sms, stream);
  }
  return to_status(e);
}

// DeMo's fused step compiled for k (the top-k and the payload loop unrolled), where it measured
// faster than the runtime-k kernel: every k in {1, 2, 4, 8} with bfloat16 gradients (2^28,
// R = 2: k = 4 1160 -> 1096 us, k = 8 1287 -> 1187; 2^26, R = 8: k = 4 1005 -> 891), and k = 1
// and k = 8 with float32 gradients (k = 8 with eight warps: 1288 -> 1251 us).  With float32
// gradients and k = 2 or 4 the compiled kernel was 2-4% slower on large shards and is used only
// on small ones (at most kLatencyTilesPerWarp tiles per warp), where its fewer instructions win
// (2^21, R = 8, k = 4: 47.1 -> 43.9 us).
bool step_kv(int mode, int k, bool bf16, bool small) {
  return mode == DEMO_MODE_DEMO && (k == 1 || k == 2 || k == 4 || k == 8) && (bf16 || small || k == 1 || k == 8);
}

template <int MAXR>
int run_step(DeviceState* st, float* theta, int64_t n, int k, float beta, float lr, int mode, int sign, int R,
             const void* const* g, int grad_dtype, float* const* m, int diloco_period, uint64_t seed, uint64_t step,
             int wire, cudaStream_t stream) {
  static_assert(sizeof(StepParams<MAXR>) < 32000, "kernel parameter block too large");
  if (mode == DEMO_MODE_DILOCO && !diloco_sync(step, diloco_period))
    return run_momentum<MAXR>(st, n, beta, R, g, grad_dtype, m, stream);
  StepParams<MAXR> p;
  std::memset(&p, 0, sizeof(p));
  const int64_t nc = n / DEMO_CHUNK;
  const bool bf16 = grad_dtype == DEMO_GRAD_BF16;
  if (!make_map(&p.theta, theta, nc, false)) return DEMO_ECUDA;
  p.theta_ptr = theta;
  for (int r = 0; r < R; ++r) {
    if (!make_map(&p.g[r], g[r], nc, bf16)) return DEMO_ECUDA;
    if (!make_map(&p.m[r], m[r], nc, false)) return DEMO_ECUDA;
    p.m_ptr[r] = m[r];
  }
  p.nc = nc;
  p.ntiles = (nc + 31) / 32;
  p.R = R;
  p.k = (mode == DEMO_MODE_DILOCO) ? DEMO_CHUNK : k;
  p.sign = sign;
  p.sync = (mode == DEMO_MODE_DILOCO) ? diloco_sync(step, diloco_period) : 1;
  fill_selection(p, mode, p.k, seed, step);
  p.stride_mask = (mode == DEMO_MODE_STRIDE) ? stride_mask(p.stride_o, p.stride_ns, k) : 0u;
  p.beta = beta;
  p.lr = lr;
  p.rcpR = 1.0f / static_cast<float>(R);
  fill_rcp(p);
  p.wire = wire;
  p.fault = st->fault;
  p.stall_at = st->stall_at.exchange(0);
  const TileShape sh = tile_shape(step_warps(mode, p.k, bf16, R, p.sync != 0), kStepWarps, p.ntiles, st);
  // DeMo with k in {1, 2, 4, 8} runs the step compiled for its k
  // small shards (at most kLatencyTilesPerWarp tiles per warp of the widest build) are bound by
  // the issue rate of a few warps, not by HBM
  const bool small = (p.ntiles + st->sms * kStepWarps - 1) / (st->sms * kStepWarps) <= kLatencyTilesPerWarp;
  const int kv = step_kv(mode, k, bf16, small) ? k : 0;
  cudaError_t e;
  if constexpr (MAXR == kSmallReplicas) {
    e = launch_step_small(p, mode, bf16, sh.inst, kv, sh.active, sh.grid, stream);
  } else {
    e = launch_step_large(p, mode, bf16, sh.inst, kv, sh.active, sh.grid, stream);
  }
  return to_status(e);
}

// Which replicas' payloads the decode kernel stages through shared memory, the CTA shape
// that goes with it (returns its warp count) and the kernel flavour.  The spans of one
// 32-chunk tile must be 16-byte multiples (so every tile's span starts 16-byte aligned in a
// 16-byte aligned buffer).  The shape with the most warps whose staging holds every
// replica is taken (measured faster than staging only some with more warps).  When none
// holds them all (the receiver of an all_gather over many replicas), the replicas are
// staged a group at a time (the decode visits each full tile as one item per group; Random
// and Striding for k <= 8 only), or, for DeMo with k in {1, 2, 4, 8} and long spans, read
// directly.  DiLoCo payloads (4 KB of float32 per tile and replica) are always read
// directly.
// How the spans move (measured on 2^24 and 2^26 shards with 8 to 64 replicas): with more
// than four replicas, lane copies for spans up to 320 bytes (192 in the 11-warp shape), bulk
// copies for longer ones.  Payloads that no shape holds whole are read directly, F = 32 / k
// replicas at a time, when k is 1, 2, 4 or 8 with a float32 or 16-bit format: DeMo's from
// 256-byte spans on (staged in groups below), Random's and Striding's always (2^26, R = 64:
// 1.1-2.2x faster than groups).
constexpr size_t kLaneCopyMaxSpan = 320;
constexpr size_t kLaneCopyMaxSpanWide = 192;
constexpr size_t kDirectMinSpan = 256;

// Whether a decode of R <= 4 staged replicas is light enough per tile to run best with the
// fewest warps (measured over every scheme, k in {1, 4, 8}, R in {2, 4} and every wire format;
// DeMo only for k = 4 with float32 payloads and two replicas, 2^27: 197 -> 190 us; its other
// cases measured 3-15% slower with eight warps).
bool few_warps_decode(int mode, int k, int wire, int R) {
  if (mode == DEMO_MODE_STRIDE) return wire != DEMO_WIRE_TERNARY || R <= 2;
  if (mode == DEMO_MODE_RANDOM) return (wire == DEMO_WIRE_F32 && k <= 4) || (k == 1 && R <= 2);
  return k == 4 && wire == DEMO_WIRE_F32 && R <= 2;
}

template <class P>
int stage_payloads(P& p, int mode, int k, int wire, int R, int* flavor) {
  p.nstaged = 0;
  p.group = 0;
  p.vspan = p.ispan = 0;
  p.sstride = 0;
  p.lane_unit = 16;
  *flavor = kFlavPlain;
  if (mode == DEMO_MODE_DILOCO) return kDecShapes[0];
  const bool demo = mode == DEMO_MODE_DEMO;
  size_t vs, is;
  if (wire == DEMO_WIRE_TERNARY) {
    vs = 8 * static_cast<size_t>(k);                // [tile][k][2] words
    is = demo ? 20 * static_cast<size_t>(k) : 0;    // [tile][k][5] words
  } else {
    vs = 32 * static_cast<size_t>(k) * (wire == DEMO_WIRE_F32 ? 4 : 2);
    is = demo ? 32 * static_cast<size_t>(k) : 0;    // uint8 [chunk][k]
  }
  const bool kv_path = demo && (k == 1 || k == 2 || k == 4 || k == 8);
  const bool ternary = wire == DEMO_WIRE_TERNARY;
  const size_t span = vs + is;
  // Ternary spans that are not 16-byte multiples (odd k, and DeMo's index planes for k = 1, 2)
  // are 4-byte multiples: lane copies of 4-byte units stage them, each replica at a 16-byte
  // aligned stride (2^26 decode, DeMo k = 1: R = 2 112 -> 88 us, R = 64 1365 -> 375 us, against
  // reading their words directly on each tile).  The float32 and 16-bit spans are always
  // 16-byte multiples.
  const bool units4 = ternary && (vs % 16 || is % 16);
  const size_t stride = (span + 15) / 16 * 16;
  const size_t small = static_cast<size_t>(dec_stage_bytes(kDecShapes[0]));
  if ((!units4 && (vs % 16 || is % 16)) || vs % 4 || is % 4 || stride > small) return kDecShapes[0];
  int aligned = 0;  // leading replicas with 16-byte aligned buffers
  while (aligned < R && aligned16(p.vals[aligned]) && (!demo || aligned16(p.idx[aligned]))) ++aligned;
  int warps = kDecShapes[0];
  int ns = static_cast<int>(std::min<size_t>(aligned, small / stride));
  if (ns < R && aligned == R) {
    for (int w : kDecShapes) {
      if (R * stride <= static_cast<size_t>(dec_stage_bytes(w))) {
        warps = w;
        ns = R;
        break;
      }
    }
    if (ns < R) {
      // Payloads that no shape holds whole (the receiver of an all_gather over many
      // replicas): stage them a group at a time, one item per group, with the largest
      // staging area (8 warps, 6 KB), so that each item moves as much as it can.  Random
      // and Striding keep per-draw sums across the items for k <= 8 only.
      const bool pow2 = k == 1 || k == 2 || k == 4 || k == 8;
      const bool direct = kv_path ? (!ternary && span >= kDirectMinSpan) : (!demo && pow2 && !ternary);
      if (direct) {
        ns = 0;
      } else if (demo || k <= 8) {
        warps = kDecShapes[3];
        p.group = static_cast<int>(static_cast<size_t>(dec_stage_bytes(warps)) / stride);
        ns = 0;
      }
    }
  }
  p.nstaged = ns;
  const bool staged = ns > 0 || p.group > 0;
  const bool lane_copy = staged && (units4 || (R > kSmallReplicas &&
                                               span <= (warps == kDecShapes[0] ? kLaneCopyMaxSpanWide : kLaneCopyMaxSpan)));
  p.sstride = static_cast<unsigned int>(stride);
  p.lane_unit = units4 ? 4 : 16;
  *flavor = (p.group > 0 ? kFlavGroups : kFlavPlain) | (lane_copy ? kFlavLaneCopy : kFlavPlain);
  p.vspan = static_cast<unsigned int>(vs);
  p.ispan = static_cast<unsigned int>(is);
  return warps;
}

// The DiLoCo sync step's decode is elementwise (every replica sends its whole
// momentum): one grid-stride pass over the parameters.
template <int MAXR>
int run_dense_decode(DeviceState* st, float* theta, int64_t n, float lr, int R, const void* const* vals, int wire,
                     cudaStream_t stream) {
  DenseParams<MAXR> p;
  std::memset(&p, 0, sizeof(p));
  p.theta = theta;
  for (int r = 0; r < R; ++r) p.vals[r] = vals[r];
  p.n4 = n / 4;
  p.R = R;
  p.wire = wire;
  p.lr = lr;
  p.rcpR = 1.0f / static_cast<float>(R);
  cudaError_t e;
  if constexpr (MAXR == kSmallReplicas) {
    e = launch_dense_small(p, st->sms, stream);
  } else {
    e = launch_dense_large(p, st->sms, stream);
  }
  return to_status(e);
}

template <int MAXR>
int run_decode(DeviceState* st, float* theta, int64_t n, int k, float lr, int mode, int R,
               const void* const* vals, const void* const* idx, uint64_t seed, uint64_t step, int wire,
               cudaStream_t stream, int64_t chunk0 = 0) {
  if (mode == DEMO_MODE_DILOCO) return run_dense_decode<MAXR>(st, theta, n, lr, R, vals, wire, stream);
  DecodeParams<MAXR> p;
  std::memset(&p, 0, sizeof(p));
  const int64_t nc = n / DEMO_CHUNK;
  if (!make_map(&p.theta, theta, nc, false)) return DEMO_ECUDA;
  p.theta_ptr = theta;
  for (int r = 0; r < R; ++r) {
    p.vals[r] = vals[r];
    p.idx[r] = (mode == DEMO_MODE_DEMO) ? idx[r] : nullptr;
  }
  p.nc = nc;
  p.ntiles = (nc + 31) / 32;
  p.chunk0 = chunk0;
  p.R = R;
  p.k = (mode == DEMO_MODE_DILOCO) ? DEMO_CHUNK : k;
  fill_selection(p, mode, p.k, seed, step);
  p.lr = lr;
  p.rcpR = 1.0f / static_cast<float>(R);
  fill_rcp(p);
  p.wire = wire;
  p.fault = st->fault;
  p.stall_at = st->stall_at.exchange(0);
  int flavor;
  int warps = stage_payloads(p, mode, k, wire, R, &flavor);
  // Receivers of at most four replicas, all staged, on large shards: the shape with the fewest
  // warps (and the largest staging, so every span still fits) where the per-tile work is light,
  // and the widest where the Random draws or the ternary bit extraction are heavy (2^27, R = 2,
  // 11 -> 8 warps: Striding k = 4 f32 200 -> 190 us, bf16 190 -> 176, ternary 176 -> 162;
  // Random k = 1 f32 182 -> 167, k = 4 207 -> 184; but Random k = 8 f32 202 -> 242 and Random
  // k = 4 ternary 174 -> 203).  Below 16 tiles per warp of the widest shape the fewer warps hide
  // less latency (2^24, DeMo k = 4: 99.8 -> 102.4 us for the split step).
  const bool many_tiles = p.ntiles >= 16LL * st->sms * kDecShapes[0];
  if (many_tiles && p.nstaged == R && R <= kSmallReplicas && k <= 8 && few_warps_decode(mode, k, wire, R))
    warps = kDecShapes[3];
  const TileShape sh = tile_shape(warps, warps, p.ntiles, st);
  // DeMo with k in {1, 2, 4, 8} runs the decode compiled for its k: kv = k for the float32 and
  // 16-bit formats, kv = -k for the ternary one
  const bool kv_ok = mode == DEMO_MODE_DEMO && (k == 1 || k == 2 || k == 4 || k == 8);
  // Random and Striding with many replicas, none staged (read directly, F at a time), and k in
  // {1, 2, 4, 8} with a float32 or 16-bit format run the decode compiled for k as well
  const bool scheme_kv = (mode == DEMO_MODE_RANDOM || mode == DEMO_MODE_STRIDE) && R > kSmallReplicas &&
                         (k == 1 || k == 2 || k == 4 || k == 8) && wire != DEMO_WIRE_TERNARY && p.nstaged == 0 &&
                         p.group == 0;
  const int kv = kv_ok ? (wire == DEMO_WIRE_TERNARY ? -k : k) : (scheme_kv ? k : 0);
  cudaError_t e;
  if constexpr (MAXR == kSmallReplicas) {
    e = launch_decode_small(p, mode, sh.inst, kv, flavor, sh.active, sh.grid, stream);
  } else {
    e = launch_decode_large(p, mode, sh.inst, kv, flavor, sh.active, sh.grid, stream);
  }
  return to_status(e);
}

// Deferred grid-dependency waits for the encodes after the first of demo_step_pipelined and
// demo_encode_replicas (EncodeParams::defer_wait).  T5-base shard, DeMo k = 4, R = 2, pipelined:
// 16 blocks 1.616 -> 1.534 ms, 8 blocks 1.401 -> 1.342, 4 blocks 1.342 -> 1.310; the same for the
// pipelined decodes measured no change (each follows a wait on the exchange's event, which
// orders it fully).
constexpr bool kDeferEncodeWait = true;

// One replica's encode over n elements whose first chunk is chunk0 of the shard (arguments checked).
int run_encode(DeviceState* st, const void* g, int grad_dtype, float* m, int64_t n, int k, float beta, int mode,
               int sign, bool sends, uint64_t seed, uint64_t step, int wire, void* vals, void* idx, int64_t chunk0,
               cudaStream_t stream, bool defer_wait = false) {
  if (mode == DEMO_MODE_DILOCO && !sends) {
    const void* gs[1] = {g};
    float* ms[1] = {m};
    return run_momentum<kSmallReplicas>(st, n, beta, 1, gs, grad_dtype, ms, stream);
  }
  EncodeParams p;
  std::memset(&p, 0, sizeof(p));
  const int64_t nc = n / DEMO_CHUNK;
  const bool bf16 = grad_dtype == DEMO_GRAD_BF16;
  if (!make_map(&p.g, g, nc, bf16) || !make_map(&p.m, m, nc, false)) return DEMO_ECUDA;
  p.m_ptr = m;
  p.vals = vals;
  p.idx = idx;
  p.nc = nc;
  p.ntiles = (nc + 31) / 32;
  p.chunk0 = chunk0;
  p.k = (mode == DEMO_MODE_DILOCO) ? DEMO_CHUNK : k;
  p.sign = sign;
  p.sync = (mode == DEMO_MODE_DILOCO) ? (sends ? 1 : 0) : 1;
  p.wire = wire;
  fill_selection(p, mode, p.k, seed, step);
  p.stride_mask = (mode == DEMO_MODE_STRIDE) ? stride_mask(p.stride_o, p.stride_ns, k) : 0u;
  p.beta = beta;
  p.fault = st->fault;
  p.stall_at = st->stall_at.exchange(0);
  p.defer_wait = defer_wait ? 1 : 0;
  int kv = 0;
  const TileShape sh = tile_shape(encode_warps(mode, p.k, wire, bf16, &kv), kStepWarps, p.ntiles, st);
  return to_status(launch_encode(p, mode, bf16, sh.inst, kv, sh.active, sh.grid, stream));
}

// Byte offset of the payload of the block starting at chunk c0 (tile t0 = c0 / 32) in a wire-format buffer.
struct PayloadLayout {
  size_t val_per_chunk = 0, idx_per_chunk = 0;  // float32 / 16-bit formats
  size_t val_per_tile = 0, idx_per_tile = 0;    // ternary format
  size_t vals_at(int64_t c0) const { return val_per_tile ? (c0 / 32) * val_per_tile : c0 * val_per_chunk; }
  size_t idx_at(int64_t c0) const { return idx_per_tile ? (c0 / 32) * idx_per_tile : c0 * idx_per_chunk; }
  // end of the payload of chunks before c1 (a partial last tile counts whole)
  size_t vals_end(int64_t c1) const { return val_per_tile ? ((c1 + 31) / 32) * val_per_tile : c1 * val_per_chunk; }
  size_t idx_end(int64_t c1) const { return idx_per_tile ? ((c1 + 31) / 32) * idx_per_tile : c1 * idx_per_chunk; }
};

// Argument checks of one replica's encode (demo_encode_wire); *sends tells whether the step
// sends a payload.
int check_encode(const void* g, int grad_dtype, const float* m, int64_t n, int chunk, int k, float beta, int mode,
                 int sign, int diloco_period, uint64_t step, int wire, const void* vals, const void* idx,
                 bool* sends_out) {
  const int s = check_shape(n, chunk, k, mode, diloco_period);
  if (s != DEMO_OK) return s;
  if (grad_dtype != DEMO_GRAD_F32 && grad_dtype != DEMO_GRAD_BF16) return DEMO_EINVAL;
  if (sign != 0 && sign != 1) return DEMO_EINVAL;
  if (!valid_wire(wire) || (wire == DEMO_WIRE_TERNARY && !sign)) return DEMO_EINVAL;
  if (!std::isfinite(beta)) return DEMO_EINVAL;
  const bool sends = mode != DEMO_MODE_DILOCO || diloco_sync(step, diloco_period);
  *sends_out = sends;
  if (g == nullptr || m == nullptr) return DEMO_EINVAL;
  if (sends && vals == nullptr) return DEMO_EINVAL;
  if (mode == DEMO_MODE_DEMO && idx == nullptr) return DEMO_EINVAL;
  if (!aligned16(g) || !aligned16(m)) return DEMO_EALIGN;
  if (sends && !aligned16(vals)) return DEMO_EALIGN;
  if (mode == DEMO_MODE_DEMO && !aligned16(idx)) return DEMO_EALIGN;
  const size_t gb = static_cast<size_t>(n) * (grad_dtype == DEMO_GRAD_BF16 ? 2 : 4);
  const size_t fb = static_cast<size_t>(n) * 4;
  if (overlap(g, gb, m, fb)) return DEMO_EINVAL;
  if (sends) {
    // the payload is written: it may overlap neither the gradient, the momentum nor itself
    size_t ib = 0;
    const size_t vb = demo_payload_bytes_wire(mode, n, DEMO_CHUNK, k, step, diloco_period, wire, &ib);
    if (overlap(vals, vb, g, gb) || overlap(vals, vb, m, fb)) return DEMO_EINVAL;
    if (mode == DEMO_MODE_DEMO && (overlap(idx, ib, g, gb) || overlap(idx, ib, m, fb) || overlap(idx, ib, vals, vb)))
      return DEMO_EINVAL;
  }
  return DEMO_OK;
}

PayloadLayout payload_layout(int mode, int k, int wire) {
  PayloadLayout L;
  const size_t kv = mode == DEMO_MODE_DILOCO ? DEMO_CHUNK : static_cast<size_t>(k);
  if (wire == DEMO_WIRE_TERNARY) {
    L.val_per_tile = kv * 8;
    L.idx_per_tile = mode == DEMO_MODE_DEMO ? static_cast<size_t>(k) * 20 : 0;
  } else {
    L.val_per_chunk = kv * (wire == DEMO_WIRE_F32 ? 4 : 2);
    L.idx_per_chunk = mode == DEMO_MODE_DEMO ? static_cast<size_t>(k) : 0;
  }
  return L;
}

}  // namespace

extern "C" {

const char* demo_status_string(int status) {
  switch (status) {
    case DEMO_OK: return "DEMO_OK";
    case DEMO_EINVAL: return "DEMO_EINVAL: invalid argument";
    case DEMO_EALIGN: return "DEMO_EALIGN: device pointer not 16-byte aligned";
    case DEMO_ENODEV: return "DEMO_ENODEV: no sm_103 device";
    case DEMO_ECUDA: return "DEMO_ECUDA: CUDA call or launch failed";
    case DEMO_ENOTINIT: return "DEMO_ENOTINIT: demo_init was not called for the current device";
    case DEMO_ENOSPACE: return "DEMO_ENOSPACE: the payloads need more than the library's fixed scratch";
    default: return "DEMO_UNKNOWN";
  }
}

int demo_init(int device) {
  std::lock_guard<std::mutex> lock(g_mu);
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count <= 0) {
    cudaGetLastError();
    return DEMO_ENODEV;
  }
  if (device < 0 || device >= count || device >= kMaxDevices) return DEMO_ENODEV;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
    return DEMO_ECUDA;
  if (major != 10 || minor != 3) return DEMO_ENODEV;
  if (cudaSetDevice(device) != cudaSuccess) return DEMO_ECUDA;
  DeviceState& st = g_dev[device];
  if (st.ready.load(std::memory_order_acquire)) return DEMO_OK;
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return DEMO_ECUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0)
    return DEMO_ECUDA;
  if (prepare_step_kernels() != cudaSuccess || prepare_encode_kernels() != cudaSuccess ||
      prepare_decode_kernels() != cudaSuccess || prepare_dense_kernels() != cudaSuccess)
    return DEMO_ECUDA;
  void* fault = nullptr;
  if (cudaGetSymbolAddress(&fault, g_fault_word) != cudaSuccess) return DEMO_ECUDA;
  if (cudaMemset(fault, 0, sizeof(unsigned int)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
    return DEMO_ECUDA;
  for (int b = 0; b < kMaxBlocks; ++b) {
    if (cudaEventCreateWithFlags(&st.ev_enc[b], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&st.ev_xch[b], cudaEventDisableTiming) != cudaSuccess)
      return DEMO_ECUDA;
  }
  st.sms = sms;
  st.fault = static_cast<unsigned int*>(fault);
  st.ready.store(true, std::memory_order_release);
  return DEMO_OK;
}

size_t demo_payload_bytes_wire(int mode, int64_t n, int chunk, int k, uint64_t step, int diloco_period, int wire,
                               size_t* idx_bytes) {
  if (idx_bytes) *idx_bytes = 0;
  if (check_shape(n, chunk, k, mode, diloco_period) != DEMO_OK || !valid_wire(wire)) return 0;
  const size_t nc = static_cast<size_t>(n / DEMO_CHUNK);
  const size_t T = (nc + 31) / 32;
  size_t kv;
  if (mode == DEMO_MODE_DILOCO) {
    if (!diloco_sync(step, diloco_period)) return 0;
    kv = DEMO_CHUNK;
  } else {
    kv = static_cast<size_t>(k);
  }
  if (wire == DEMO_WIRE_TERNARY) {
    if (idx_bytes && mode == DEMO_MODE_DEMO) *idx_bytes = T * static_cast<size_t>(k) * 20;
    return T * kv * 8;
  }
  if (idx_bytes && mode == DEMO_MODE_DEMO) *idx_bytes = nc * static_cast<size_t>(k);
  return nc * kv * (wire == DEMO_WIRE_F32 ? 4 : 2);
}

size_t demo_payload_bytes(int mode, int64_t n, int chunk, int k, uint64_t step, int diloco_period,
                          size_t* idx_bytes) {
  return demo_payload_bytes_wire(mode, n, chunk, k, step, diloco_period, DEMO_WIRE_F32, idx_bytes);
}

int demo_encode_wire(const void* g, int grad_dtype, float* m, int64_t n, int chunk, int k, float beta, int mode,
                     int sign, int diloco_period, uint64_t seed, uint64_t step, int wire, void* vals, void* idx,
                     void* stream) {
  bool sends = false;
  int s = check_encode(g, grad_dtype, m, n, chunk, k, beta, mode, sign, diloco_period, step, wire, vals, idx, &sends);
  if (s != DEMO_OK) return s;
  DeviceState* st = nullptr;
  s = current_state(&st);
  if (s != DEMO_OK) return s;
  return run_encode(st, g, grad_dtype, m, n, k, beta, mode, sign, sends, seed, step, wire, vals, idx, 0,
                    static_cast<cudaStream_t>(stream));
}

int demo_encode_replicas(const void* const* g, int grad_dtype, float* const* m, int64_t n, int chunk, int k,
                         float beta, int mode, int sign, int R, int diloco_period, uint64_t seed, uint64_t step,
                         int wire, void* const* vals, void* const* idx, void* stream) {
  if (R < 1 || R > DEMO_MAX_REPLICAS || g == nullptr || m == nullptr) return DEMO_EINVAL;
  bool sends = false;
  const bool demo = mode == DEMO_MODE_DEMO;
  for (int r = 0; r < R; ++r) {
    void* v = vals ? vals[r] : nullptr;
    void* ix = idx ? idx[r] : nullptr;
    const int s = check_encode(g[r], grad_dtype, m[r], n, chunk, k, beta, mode, sign, diloco_period, step, wire, v,
                               ix, &sends);
    if (s != DEMO_OK) return s;
  }
  // every m, vals and idx is written: none may overlap another replica's buffers (each replica's
  // own were checked above)
  const size_t fb = static_cast<size_t>(n) * 4;
  const size_t gb = static_cast<size_t>(n) * (grad_dtype == DEMO_GRAD_BF16 ? 2 : 4);
  size_t ib = 0;
  const size_t vb = sends ? demo_payload_bytes_wire(mode, n, DEMO_CHUNK, k, step, diloco_period, wire, &ib) : 0;
  for (int r = 0; r < R; ++r) {
    for (int q = 0; q < R; ++q) {
      if (q == r) continue;
      if (overlap(m[r], fb, m[q], fb) || overlap(m[r], fb, g[q], gb)) return DEMO_EINVAL;
      if (sends) {
        if (overlap(vals[r], vb, g[q], gb) || overlap(vals[r], vb, m[q], fb) || overlap(vals[r], vb, vals[q], vb))
          return DEMO_EINVAL;
        if (demo && (overlap(idx[r], ib, g[q], gb) || overlap(idx[r], ib, m[q], fb) ||
                     overlap(idx[r], ib, vals[q], vb) || overlap(idx[r], ib, idx[q], ib)))
          return DEMO_EINVAL;
      }
    }
  }
  DeviceState* st = nullptr;
  int s = current_state(&st);
  if (s != DEMO_OK) return s;
  // DiLoCo between syncs: only the momenta move, all R in one elementwise pass
  if (!sends) {
    return R <= kSmallReplicas
               ? run_momentum<kSmallReplicas>(st, n, beta, R, g, grad_dtype, m, static_cast<cudaStream_t>(stream))
               : run_momentum<kMaxReplicas>(st, n, beta, R, g, grad_dtype, m, static_cast<cudaStream_t>(stream));
  }
  // The replicas share no buffers, so every encode after the first may start while the previous
  // one finishes and wait for it only before exiting (EncodeParams::defer_wait).
  for (int r = 0; r < R; ++r) {
    s = run_encode(st, g[r], grad_dtype, m[r], n, k, beta, mode, sign, true, seed, step, wire, vals[r],
                   demo ? idx[r] : nullptr, 0, static_cast<cudaStream_t>(stream), kDeferEncodeWait && r > 0);
    if (s != DEMO_OK) return s;
  }
  return DEMO_OK;
}

int demo_encode(const void* g, int grad_dtype, float* m, int64_t n, int chunk, int k, float beta, int mode,
                int sign, int diloco_period, uint64_t seed, uint64_t step, float* vals, uint8_t* idx,
                void* stream) {
  return demo_encode_wire(g, grad_dtype, m, n, chunk, k, beta, mode, sign, diloco_period, seed, step,
                          DEMO_WIRE_F32, vals, idx, stream);
}

int demo_decode_update_wire(float* theta, int64_t n, int chunk, int k, float lr, int mode, int R,
                            const void* const* vals, const void* const* idx, int diloco_period, uint64_t seed,
                            uint64_t step, int wire, void* stream) {
  int s = check_shape(n, chunk, k, mode, diloco_period);
  if (s != DEMO_OK) return s;
  if (R < 1 || R > DEMO_MAX_REPLICAS) return DEMO_EINVAL;
  if (!valid_wire(wire)) return DEMO_EINVAL;
  if (!std::isfinite(lr)) return DEMO_EINVAL;
  if (theta == nullptr || vals == nullptr) return DEMO_EINVAL;
  if (mode == DEMO_MODE_DEMO && idx == nullptr) return DEMO_EINVAL;
  const bool sends = mode != DEMO_MODE_DILOCO || diloco_sync(step, diloco_period);
  for (int r = 0; r < R && sends; ++r) {
    if (vals[r] == nullptr) return DEMO_EINVAL;
    if (mode == DEMO_MODE_DEMO && idx[r] == nullptr) return DEMO_EINVAL;
  }
  if (!aligned16(theta)) return DEMO_EALIGN;
  for (int r = 0; r < R && sends; ++r) {
    if (!aligned16(vals[r])) return DEMO_EALIGN;
    if (mode == DEMO_MODE_DEMO && !aligned16(idx[r])) return DEMO_EALIGN;
  }
  if (sends) {
    // theta is written while the payloads are read: no payload may overlap it (payloads are
    // read only and may be shared between replicas)
    size_t ib = 0;
    const size_t vb = demo_payload_bytes_wire(mode, n, DEMO_CHUNK, k, step, diloco_period, wire, &ib);
    const size_t fb = static_cast<size_t>(n) * 4;
    for (int r = 0; r < R; ++r) {
      if (overlap(theta, fb, vals[r], vb)) return DEMO_EINVAL;
      if (mode == DEMO_MODE_DEMO && overlap(theta, fb, idx[r], ib)) return DEMO_EINVAL;
    }
  }
  DeviceState* st = nullptr;
  s = current_state(&st);
  if (s != DEMO_OK) return s;
  if (!sends) return DEMO_OK;  // DiLoCo between syncs: theta does not move
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return R <= kSmallReplicas
             ? run_decode<kSmallReplicas>(st, theta, n, k, lr, mode, R, vals, idx, seed, step, wire, cs)
             : run_decode<kMaxReplicas>(st, theta, n, k, lr, mode, R, vals, idx, seed, step, wire, cs);
}

int demo_decode_update(float* theta, int64_t n, int chunk, int k, float lr, int mode, int R,
                       const float* const* vals, const uint8_t* const* idx, int diloco_period, uint64_t seed,
                       uint64_t step, void* stream) {
  return demo_decode_update_wire(theta, n, chunk, k, lr, mode, R, reinterpret_cast<const void* const*>(vals),
                                 reinterpret_cast<const void* const*>(idx), diloco_period, seed, step, DEMO_WIRE_F32,
                                 stream);
}

int demo_step_wire(float* theta, int64_t n, int chunk, int k, float beta, float lr, int mode, int sign, int R,
                   const void* const* g, int grad_dtype, float* const* m, int diloco_period, uint64_t seed,
                   uint64_t step, int wire, void* stream) {
  int s = check_shape(n, chunk, k, mode, diloco_period);
  if (s != DEMO_OK) return s;
  if (R < 1 || R > DEMO_MAX_REPLICAS) return DEMO_EINVAL;
  if (grad_dtype != DEMO_GRAD_F32 && grad_dtype != DEMO_GRAD_BF16) return DEMO_EINVAL;
  if (sign != 0 && sign != 1) return DEMO_EINVAL;
  if (!valid_wire(wire) || (wire == DEMO_WIRE_TERNARY && !sign)) return DEMO_EINVAL;
  if (!std::isfinite(beta) || !std::isfinite(lr)) return DEMO_EINVAL;
  if (theta == nullptr || g == nullptr || m == nullptr) return DEMO_EINVAL;
  for (int r = 0; r < R; ++r)
    if (g[r] == nullptr || m[r] == nullptr) return DEMO_EINVAL;
  if (!aligned16(theta)) return DEMO_EALIGN;
  for (int r = 0; r < R; ++r)
    if (!aligned16(g[r]) || !aligned16(m[r])) return DEMO_EALIGN;
  // m_r and theta are written: none may overlap another buffer (the g_r are
  // read only and may be shared between replicas).
  const size_t fb = static_cast<size_t>(n) * 4;
  const size_t gb = static_cast<size_t>(n) * (grad_dtype == DEMO_GRAD_BF16 ? 2 : 4);
  for (int r = 0; r < R; ++r) {
    if (overlap(m[r], fb, theta, fb)) return DEMO_EINVAL;
    for (int q = 0; q < R; ++q) {
      if (q != r && overlap(m[r], fb, m[q], fb)) return DEMO_EINVAL;
      if (overlap(m[r], fb, g[q], gb)) return DEMO_EINVAL;
    }
    if (overlap(theta, fb, g[r], gb)) return DEMO_EINVAL;
  }
  DeviceState* st = nullptr;
  s = current_state(&st);
  if (s != DEMO_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return R <= kSmallReplicas
             ? run_step<kSmallReplicas>(st, theta, n, k, beta, lr, mode, sign, R, g, grad_dtype, m, diloco_period,
                                        seed, step, wire, cs)
             : run_step<kMaxReplicas>(st, theta, n, k, beta, lr, mode, sign, R, g, grad_dtype, m, diloco_period,
                                      seed, step, wire, cs);
}

int demo_step(float* theta, int64_t n, int chunk, int k, float beta, float lr, int mode, int sign, int R,
              const void* const* g, int grad_dtype, float* const* m, int diloco_period, uint64_t seed,
              uint64_t step, void* stream) {
  return demo_step_wire(theta, n, chunk, k, beta, lr, mode, sign, R, g, grad_dtype, m, diloco_period, seed, step,
                        DEMO_WIRE_F32, stream);
}

int demo_step_pipelined(float* theta, int64_t n, int chunk, int k, float beta, float lr, int mode, int sign, int R,
                        const void* const* g, int grad_dtype, float* const* m, int diloco_period, uint64_t seed,
                        uint64_t step, int wire, void* const* send_vals, void* const* send_idx,
                        void* const* recv_vals, void* const* recv_idx, int blocks, void* compute_stream,
                        void* comm_stream) {
  int s = check_shape(n, chunk, k, mode, diloco_period);
  if (s != DEMO_OK) return s;
  if (R < 1 || R > DEMO_MAX_REPLICAS || blocks < 1 || blocks > kMaxBlocks) return DEMO_EINVAL;
  if (grad_dtype != DEMO_GRAD_F32 && grad_dtype != DEMO_GRAD_BF16) return DEMO_EINVAL;
  if (sign != 0 && sign != 1) return DEMO_EINVAL;
  if (!valid_wire(wire) || (wire == DEMO_WIRE_TERNARY && !sign)) return DEMO_EINVAL;
  if (!std::isfinite(beta) || !std::isfinite(lr)) return DEMO_EINVAL;
  if (theta == nullptr || g == nullptr || m == nullptr) return DEMO_EINVAL;
  const bool sends = mode != DEMO_MODE_DILOCO || diloco_sync(step, diloco_period);
  const bool demo = mode == DEMO_MODE_DEMO;
  if (sends && (send_vals == nullptr || recv_vals == nullptr)) return DEMO_EINVAL;
  if (sends && demo && (send_idx == nullptr || recv_idx == nullptr)) return DEMO_EINVAL;
  for (int r = 0; r < R; ++r) {
    if (g[r] == nullptr || m[r] == nullptr) return DEMO_EINVAL;
    if (sends && (send_vals[r] == nullptr || recv_vals[r] == nullptr)) return DEMO_EINVAL;
    if (sends && demo && (send_idx[r] == nullptr || recv_idx[r] == nullptr)) return DEMO_EINVAL;
  }
  if (!aligned16(theta)) return DEMO_EALIGN;
  for (int r = 0; r < R; ++r) {
    if (!aligned16(g[r]) || !aligned16(m[r])) return DEMO_EALIGN;
    if (sends && (!aligned16(send_vals[r]) || !aligned16(recv_vals[r]))) return DEMO_EALIGN;
    if (sends && demo && (!aligned16(send_idx[r]) || !aligned16(recv_idx[r]))) return DEMO_EALIGN;
  }
  const size_t fb = static_cast<size_t>(n) * 4;
  const size_t gb = static_cast<size_t>(n) * (grad_dtype == DEMO_GRAD_BF16 ? 2 : 4);
  for (int r = 0; r < R; ++r) {
    if (overlap(m[r], fb, theta, fb)) return DEMO_EINVAL;
    for (int q = 0; q < R; ++q) {
      if (q != r && overlap(m[r], fb, m[q], fb)) return DEMO_EINVAL;
      if (overlap(m[r], fb, g[q], gb)) return DEMO_EINVAL;
    }
    if (overlap(theta, fb, g[r], gb)) return DEMO_EINVAL;
  }
  if (sends) {
    // every send and receive buffer is written: each must be apart from theta, every m and g,
    // and every other payload buffer
    size_t ib = 0;
    const size_t vb = demo_payload_bytes_wire(mode, n, DEMO_CHUNK, k, step, diloco_period, wire, &ib);
    const int nbuf = demo ? 4 : 2;
    auto buf = [&](int r, int j) -> const void* {
      const void* const* a[4] = {send_vals, recv_vals, send_idx, recv_idx};
      return a[j][r];
    };
    auto len = [&](int j) { return j < 2 ? vb : ib; };
    for (int r = 0; r < R; ++r) {
      for (int j = 0; j < nbuf; ++j) {
        const void* b = buf(r, j);
        if (overlap(b, len(j), theta, fb)) return DEMO_EINVAL;
        for (int q = 0; q < R; ++q) {
          if (overlap(b, len(j), m[q], fb) || overlap(b, len(j), g[q], gb)) return DEMO_EINVAL;
          for (int i = 0; i < nbuf; ++i)
            if ((q != r || i != j) && overlap(b, len(j), buf(q, i), len(i))) return DEMO_EINVAL;
        }
      }
    }
  }
  DeviceState* st = nullptr;
  s = current_state(&st);
  if (s != DEMO_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
  cudaStream_t xs = static_cast<cudaStream_t>(comm_stream);
  std::lock_guard<std::mutex> enqueue(st->pipeline_mu);

  // blocks of whole 32-chunk tiles, so every wire format's payload splits at block boundaries
  const int64_t nc = n / DEMO_CHUNK;
  const int64_t T = (nc + 31) / 32;
  const int64_t tpb = (T + blocks - 1) / blocks;
  const int B = static_cast<int>((T + tpb - 1) / tpb);
  const PayloadLayout L = payload_layout(mode, k, wire);
  auto chunk_lo = [&](int b) { return std::min<int64_t>(static_cast<int64_t>(b) * tpb * 32, nc); };
  auto chunk_hi = [&](int b) { return std::min<int64_t>(static_cast<int64_t>(b + 1) * tpb * 32, nc); };
  auto at = [](const void* p, size_t off) { return static_cast<char*>(const_cast<void*>(p)) + off; };

  auto decode_block = [&](int b) -> int {
    const int64_t c0 = chunk_lo(b), c1 = chunk_hi(b);
    const void* v[DEMO_MAX_REPLICAS];
    const void* ix[DEMO_MAX_REPLICAS];
    for (int r = 0; r < R; ++r) {
      v[r] = at(recv_vals[r], L.vals_at(c0));
      ix[r] = demo ? at(recv_idx[r], L.idx_at(c0)) : nullptr;
    }
    float* th = theta + c0 * DEMO_CHUNK;
    const int64_t nb = (c1 - c0) * DEMO_CHUNK;
    return R <= kSmallReplicas
               ? run_decode<kSmallReplicas>(st, th, nb, k, lr, mode, R, v, ix, seed, step, wire, cs, c0)
               : run_decode<kMaxReplicas>(st, th, nb, k, lr, mode, R, v, ix, seed, step, wire, cs, c0);
  };

  // Every encode after the first follows one of this call's own encodes or decodes, which
  // touch none of its buffers (each reads and writes its own block of g_r, m_r and the send
  // buffers; the decodes read the receive buffers and theta): it may load and work while the
  // previous kernel finishes and wait for it only before exiting.
  // DiLoCo between syncs sends nothing: the step is the momenta alone, one elementwise pass
  if (!sends) {
    return R <= kSmallReplicas ? run_momentum<kSmallReplicas>(st, n, beta, R, g, grad_dtype, m, cs)
                               : run_momentum<kMaxReplicas>(st, n, beta, R, g, grad_dtype, m, cs);
  }
  for (int b = 0; b < B; ++b) {
    const int64_t c0 = chunk_lo(b), c1 = chunk_hi(b);
    const int64_t nb = (c1 - c0) * DEMO_CHUNK;
    for (int r = 0; r < R; ++r) {
      const void* gb_ptr = at(g[r], static_cast<size_t>(c0) * DEMO_CHUNK * (grad_dtype == DEMO_GRAD_BF16 ? 2 : 4));
      s = run_encode(st, gb_ptr, grad_dtype, m[r] + c0 * DEMO_CHUNK, nb, k, beta, mode, sign, true, seed, step, wire,
                     at(send_vals[r], L.vals_at(c0)), demo ? at(send_idx[r], L.idx_at(c0)) : nullptr, c0, cs,
                     kDeferEncodeWait && (b > 0 || r > 0));
      if (s != DEMO_OK) return s;
    }
    // the exchange of block b: a loopback copy of every replica's payload block on the communication stream
    if (cudaEventRecord(st->ev_enc[b], cs) != cudaSuccess || cudaStreamWaitEvent(xs, st->ev_enc[b], 0) != cudaSuccess)
      return DEMO_ECUDA;
    for (int r = 0; r < R; ++r) {
      if (cudaMemcpyAsync(at(recv_vals[r], L.vals_at(c0)), at(send_vals[r], L.vals_at(c0)),
                          L.vals_end(c1) - L.vals_at(c0), cudaMemcpyDeviceToDevice, xs) != cudaSuccess)
        return DEMO_ECUDA;
      if (demo && cudaMemcpyAsync(at(recv_idx[r], L.idx_at(c0)), at(send_idx[r], L.idx_at(c0)),
                                  L.idx_end(c1) - L.idx_at(c0), cudaMemcpyDeviceToDevice, xs) != cudaSuccess)
        return DEMO_ECUDA;
    }
    if (cudaEventRecord(st->ev_xch[b], xs) != cudaSuccess) return DEMO_ECUDA;
    // decode the previous block while this block's exchange is in flight
    if (b >= 1) {
      if (cudaStreamWaitEvent(cs, st->ev_xch[b - 1], 0) != cudaSuccess) return DEMO_ECUDA;
      s = decode_block(b - 1);
      if (s != DEMO_OK) return s;
    }
  }
  if (cudaStreamWaitEvent(cs, st->ev_xch[B - 1], 0) != cudaSuccess) return DEMO_ECUDA;
  return decode_block(B - 1);
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Fixed scratch for demo_step_pipelined_static (callers that cannot allocate)
// ----------------------------------------------------------------------------

namespace {

constexpr size_t kStaticHalfBytes = size_t(32) << 20;  // send half and receive half, 32 MiB each
static __device__ __align__(256) unsigned char g_static_scratch[2 * kStaticHalfBytes];
void* g_static_scratch_addr[kMaxDevices] = {};

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace

extern "C" {

int demo_step_pipelined_static(float* theta, int64_t n, int chunk, int k, float beta, float lr, int mode, int sign,
                               int R, const void* const* g, int grad_dtype, float* const* m, int diloco_period,
                               uint64_t seed, uint64_t step, int wire, int blocks, void* compute_stream,
                               void* comm_stream) {
  if (R < 1 || R > DEMO_MAX_REPLICAS) return DEMO_EINVAL;
  size_t ib = 0;
  const size_t vb = demo_payload_bytes_wire(mode, n, chunk, k, step, diloco_period, wire, &ib);
  const size_t per_replica = round256(vb) + round256(ib);
  if (per_replica * static_cast<size_t>(R) > kStaticHalfBytes) return DEMO_ENOSPACE;

  // Device address of the array on the current device, looked up once per device.
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return DEMO_ENOTINIT;
  }
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_static_scratch_addr[dev] == nullptr) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_static_scratch) != cudaSuccess || addr == nullptr) return DEMO_ECUDA;
      g_static_scratch_addr[dev] = addr;
    }
    base = g_static_scratch_addr[dev];
  }

  void* send_vals[DEMO_MAX_REPLICAS];
  void* send_idx[DEMO_MAX_REPLICAS];
  void* recv_vals[DEMO_MAX_REPLICAS];
  void* recv_idx[DEMO_MAX_REPLICAS];
  char* send = static_cast<char*>(base);
  char* recv = send + kStaticHalfBytes;
  for (int r = 0; r < R; ++r) {
    const size_t off = static_cast<size_t>(r) * per_replica;
    send_vals[r] = send + off;
    recv_vals[r] = recv + off;
    send_idx[r] = ib ? send + off + round256(vb) : nullptr;
    recv_idx[r] = ib ? recv + off + round256(vb) : nullptr;
  }
  const bool payload = vb > 0;
  return demo_step_pipelined(theta, n, chunk, k, beta, lr, mode, sign, R, g, grad_dtype, m, diloco_period, seed, step,
                             wire, payload ? send_vals : nullptr, ib ? send_idx : nullptr,
                             payload ? recv_vals : nullptr, ib ? recv_idx : nullptr, blocks, compute_stream,
                             comm_stream);
}

int demo_validate_payload(int64_t n, int chunk, int k, int wire, const void* idx_host, int64_t* first_bad) {
  if (first_bad) *first_bad = -1;
  if (check_shape(n, chunk, k, DEMO_MODE_DEMO, 1) != DEMO_OK || !valid_wire(wire) || idx_host == nullptr)
    return DEMO_EINVAL;
  const int64_t nc = n / DEMO_CHUNK;
  for (int64_t c = 0; c < nc; ++c) {
    int prev = -1;
    bool ok = true;
    for (int j = 0; j < k && ok; ++j) {
      int u;
      if (wire == DEMO_WIRE_TERNARY) {
        const uint32_t* w = static_cast<const uint32_t*>(idx_host) + ((c / 32) * k + j) * 5;
        u = 0;
        for (int b = 0; b < 5; ++b) u |= static_cast<int>((w[b] >> (c % 32)) & 1u) << b;
      } else {
        u = static_cast<const uint8_t*>(idx_host)[c * k + j];
      }
      ok = u < DEMO_CHUNK && u > prev;
      prev = u;
    }
    if (!ok) {
      if (first_bad) *first_bad = c;
      return DEMO_EINVAL;
    }
  }
  return DEMO_OK;
}

int demo_adamw_step(float* theta, int64_t n, float beta1, float beta2, float eps, float lr, float weight_decay,
                    int R, const void* const* g, int grad_dtype, float* const* m, float* const* v, uint64_t step,
                    void* stream) {
  if (n <= 0 || n % DEMO_CHUNK != 0 || n > kMaxN) return DEMO_EINVAL;
  if (R < 1 || R > DEMO_MAX_REPLICAS) return DEMO_EINVAL;
  if (grad_dtype != DEMO_GRAD_F32 && grad_dtype != DEMO_GRAD_BF16) return DEMO_EINVAL;
  if (!std::isfinite(beta1) || !std::isfinite(beta2) || !std::isfinite(eps) || !std::isfinite(lr) ||
      !std::isfinite(weight_decay))
    return DEMO_EINVAL;
  if (beta1 < 0.0f || beta1 >= 1.0f || beta2 < 0.0f || beta2 >= 1.0f || !(eps > 0.0f)) return DEMO_EINVAL;
  if (theta == nullptr || g == nullptr || m == nullptr || v == nullptr) return DEMO_EINVAL;
  for (int r = 0; r < R; ++r)
    if (g[r] == nullptr || m[r] == nullptr || v[r] == nullptr) return DEMO_EINVAL;
  if (!aligned16(theta)) return DEMO_EALIGN;
  for (int r = 0; r < R; ++r)
    if (!aligned16(g[r]) || !aligned16(m[r]) || !aligned16(v[r])) return DEMO_EALIGN;
  // written buffers (theta, every m_r and v_r) must not overlap anything else
  const size_t fb = static_cast<size_t>(n) * 4;
  const size_t gb = static_cast<size_t>(n) * (grad_dtype == DEMO_GRAD_BF16 ? 2 : 4);
  for (int r = 0; r < R; ++r) {
    if (overlap(theta, fb, g[r], gb) || overlap(theta, fb, m[r], fb) || overlap(theta, fb, v[r], fb))
      return DEMO_EINVAL;
    for (int q = 0; q < R; ++q) {
      if (overlap(m[r], fb, g[q], gb) || overlap(v[r], fb, g[q], gb) || overlap(m[r], fb, v[q], fb))
        return DEMO_EINVAL;
      if (q != r && (overlap(m[r], fb, m[q], fb) || overlap(v[r], fb, v[q], fb))) return DEMO_EINVAL;
    }
  }
  DeviceState* st = nullptr;
  const int s = current_state(&st);
  if (s != DEMO_OK) return s;
  AdamWParams p;
  std::memset(&p, 0, sizeof(p));
  p.theta = theta;
  for (int r = 0; r < R; ++r) {
    p.g[r] = g[r];
    p.m[r] = m[r];
    p.v[r] = v[r];
  }
  p.n4 = n / 4;
  p.R = R;
  p.beta1 = beta1;
  p.beta2 = beta2;
  p.omb1 = static_cast<float>(1.0 - static_cast<double>(beta1));
  p.omb2 = static_cast<float>(1.0 - static_cast<double>(beta2));
  const double t = static_cast<double>(step) + 1.0;
  p.rbc1 = static_cast<float>(1.0 / (1.0 - std::pow(static_cast<double>(beta1), t)));
  p.rbc2 = static_cast<float>(1.0 / (1.0 - std::pow(static_cast<double>(beta2), t)));
  p.eps = eps;
  p.lr = lr;
  p.wd = weight_decay;
  p.rcpR = 1.0f / static_cast<float>(R);
  const int64_t want = (p.n4 + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * st->sms ? want : 8LL * st->sms);
  return to_status(launch_adamw(p, grad_dtype == DEMO_GRAD_BF16, grid, static_cast<cudaStream_t>(stream)));
}

int demo_test_stall_next_launch(long long item) {
  DeviceState* st = nullptr;
  const int s = current_state(&st);
  if (s != DEMO_OK) return s;
  st->stall_at.store(item >= 0 ? item + 1 : 0);
  return DEMO_OK;
}

int demo_device_fault(unsigned int* code) {
  if (code == nullptr) return DEMO_EINVAL;
  DeviceState* st = nullptr;
  const int s = current_state(&st);
  if (s != DEMO_OK) return s;
  unsigned int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return DEMO_ECUDA;
  if (cudaMemcpy(&v, st->fault, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DEMO_ECUDA;
  if (cudaMemset(st->fault, 0, sizeof(v)) != cudaSuccess) return DEMO_ECUDA;
  *code = v;
  return DEMO_OK;
}

}  // extern "C"
