// C ABI of the DeMo shard step: argument checks, TMA tensor maps, launches.
// The operations and their sources are described in include/demo.h.
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/demo.h"
#include "demo_common.cuh"
#include "demo_params.h"

namespace {

using namespace demo;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxN = int64_t(1) << 35;  // keeps every row coordinate within int32

struct DeviceState {
  bool ready = false;
  int sms = 0;
  unsigned int* fault = nullptr;
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
  if (dev < 0 || dev >= kMaxDevices || !g_dev[dev].ready) return DEMO_ENOTINIT;
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

int grid_for(int64_t ntiles, const DeviceState* st, int warps_per_cta = kStepWarps) {
  const int64_t want = (ntiles + warps_per_cta - 1) / warps_per_cta;
  return static_cast<int>(want < st->sms ? want : st->sms);
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

template <int MAXR>
int run_step(DeviceState* st, float* theta, int64_t n, int k, float beta, float lr, int mode, int sign, int R,
             const void* const* g, int grad_dtype, float* const* m, int diloco_period, uint64_t seed, uint64_t step,
             int wire, cudaStream_t stream) {
  static_assert(sizeof(StepParams<MAXR>) < 32000, "kernel parameter block too large");
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
  const int grid = grid_for(p.ntiles, st);
  cudaError_t e;
  if constexpr (MAXR == kSmallReplicas) {
    e = launch_step_small(p, mode, bf16, grid, stream);
  } else {
    e = launch_step_large(p, mode, bf16, grid, stream);
  }
  return to_status(e);
}

template <int MAXR>
int run_decode(DeviceState* st, float* theta, int64_t n, int k, float lr, int mode, int R,
               const void* const* vals, const void* const* idx, uint64_t seed, uint64_t step, int wire,
               cudaStream_t stream) {
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
  p.R = R;
  p.k = (mode == DEMO_MODE_DILOCO) ? DEMO_CHUNK : k;
  fill_selection(p, mode, p.k, seed, step);
  p.lr = lr;
  p.rcpR = 1.0f / static_cast<float>(R);
  fill_rcp(p);
  p.wire = wire;
  p.fault = st->fault;
  const int grid = grid_for(p.ntiles, st);
  cudaError_t e;
  if constexpr (MAXR == kSmallReplicas) {
    e = launch_decode_small(p, mode, grid, stream);
  } else {
    e = launch_decode_large(p, mode, grid, stream);
  }
  return to_status(e);
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
  if (st.ready) return DEMO_OK;
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
      prepare_decode_kernels() != cudaSuccess)
    return DEMO_ECUDA;
  void* fault = nullptr;
  if (cudaGetSymbolAddress(&fault, g_fault_word) != cudaSuccess) return DEMO_ECUDA;
  if (cudaMemset(fault, 0, sizeof(unsigned int)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
    return DEMO_ECUDA;
  st.sms = sms;
  st.fault = static_cast<unsigned int*>(fault);
  st.ready = true;
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
  int s = check_shape(n, chunk, k, mode, diloco_period);
  if (s != DEMO_OK) return s;
  if (grad_dtype != DEMO_GRAD_F32 && grad_dtype != DEMO_GRAD_BF16) return DEMO_EINVAL;
  if (sign != 0 && sign != 1) return DEMO_EINVAL;
  if (!valid_wire(wire) || (wire == DEMO_WIRE_TERNARY && !sign)) return DEMO_EINVAL;
  if (!std::isfinite(beta)) return DEMO_EINVAL;
  const bool sends = mode != DEMO_MODE_DILOCO || diloco_sync(step, diloco_period);
  if (g == nullptr || m == nullptr) return DEMO_EINVAL;
  if (sends && vals == nullptr) return DEMO_EINVAL;
  if (mode == DEMO_MODE_DEMO && idx == nullptr) return DEMO_EINVAL;
  if (!aligned16(g) || !aligned16(m)) return DEMO_EALIGN;
  if (sends && !aligned16(vals)) return DEMO_EALIGN;
  if (mode == DEMO_MODE_DEMO && !aligned16(idx)) return DEMO_EALIGN;
  const size_t gb = static_cast<size_t>(n) * (grad_dtype == DEMO_GRAD_BF16 ? 2 : 4);
  if (overlap(g, gb, m, static_cast<size_t>(n) * 4)) return DEMO_EINVAL;
  DeviceState* st = nullptr;
  s = current_state(&st);
  if (s != DEMO_OK) return s;

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
  p.k = (mode == DEMO_MODE_DILOCO) ? DEMO_CHUNK : k;
  p.sign = sign;
  p.sync = (mode == DEMO_MODE_DILOCO) ? (sends ? 1 : 0) : 1;
  p.wire = wire;
  fill_selection(p, mode, p.k, seed, step);
  p.stride_mask = (mode == DEMO_MODE_STRIDE) ? stride_mask(p.stride_o, p.stride_ns, k) : 0u;
  p.beta = beta;
  p.fault = st->fault;
  return to_status(launch_encode(p, mode, bf16, grid_for(p.ntiles, st), static_cast<cudaStream_t>(stream)));
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
