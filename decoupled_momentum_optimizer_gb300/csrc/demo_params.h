// Kernel parameter blocks and launcher declarations of the DeMo shard step.
// Tensor maps travel by value as __grid_constant__ kernel parameters.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace demo {

constexpr int kMaxReplicas = 64;
constexpr int kSmallReplicas = 4;  // parameter blocks for R <= 4 stay small

template <int MAXR>
struct StepParams {
  CUtensorMap theta;
  CUtensorMap g[MAXR];
  CUtensorMap m[MAXR];
  float* theta_ptr;  // the same buffers as raw pointers, for the coalesced stores
  float* m_ptr[MAXR];
  long long nc;      // chunks in the shard
  long long ntiles;  // ceil(nc / 32)
  int R, k, sign;
  int sync;          // DiLoCo: this step sends the full momentum
  int stride_o, stride_ns;
  unsigned int stride_mask;
  float beta, lr, rcpR;
  unsigned long long hbase;  // sm(sm(seed) ^ step) for the Random scheme
  float rcp_tab[kMaxReplicas + 1];  // float32(1/c), entry 0 = 0
  int wire;                         // payload wire format the on-chip values are rounded to
  unsigned int* fault;
};

struct EncodeParams {
  CUtensorMap g;
  CUtensorMap m;
  float* m_ptr;
  void* vals;  // wire-format payload values
  void* idx;   // DeMo indices (uint8 [nc][k], or uint32 bit-planes for the ternary format)
  long long nc, ntiles;
  long long chunk0;  // shard index of the first chunk (the Random scheme hashes shard chunk indices)
  int k, sign, sync, wire;
  int stride_o, stride_ns;
  unsigned int stride_mask;
  float beta;
  unsigned long long hbase;
  unsigned int* fault;
};

template <int MAXR>
struct DecodeParams {
  CUtensorMap theta;
  float* theta_ptr;
  const void* vals[MAXR];
  const void* idx[MAXR];
  long long nc, ntiles;
  long long chunk0;  // shard index of the first chunk
  int R, k, wire;
  int stride_o, stride_ns;
  // Payload staging: replicas 0..nstaged-1 have their per-tile spans (vspan bytes
  // of values, ispan bytes of indices at tile t * span) copied to shared memory
  // with the theta tile; the others, and a ragged last tile, are read directly.
  int nstaged;
  unsigned int vspan, ispan;
  float lr, rcpR;
  unsigned long long hbase;
  float rcp_tab[kMaxReplicas + 1];
  unsigned int* fault;
};

// Shared-memory staging per decode slot for the replicas' payload spans: 2 KB
// with 11 warps per SM, or 3 KB with 10 warps when the replicas fit only that.
constexpr int kDecStageBytes = 2048;
constexpr int kDecStageBytesWide = 3072;
constexpr int kDecWarpsWide = 10;

// Decoupled AdamW (elementwise, grid-stride over groups of four parameters).
struct AdamWParams {
  float* theta;
  const void* g[kMaxReplicas];
  float* m[kMaxReplicas];
  float* v[kMaxReplicas];
  long long n4;  // n / 4
  int R;
  float beta1, beta2, omb1, omb2;  // beta and 1 - beta (exact in float32)
  float rbc1, rbc2;                // 1 / (1 - beta^t), t = step + 1
  float eps, lr, wd, rcpR;
};

cudaError_t launch_adamw(const AdamWParams& p, bool bf16, int grid, cudaStream_t st);

// Launchers (one per translation unit).  `grid` CTAs of W warps (kStepWarps for
// the encode and decode kernels); each warp walks the tiles gw, gw + W * grid, ...
//
// The fused step kernel is built for three resident warp counts per SM.  Its
// data stream per item is fixed, its compute per item is not (Striding and
// DiLoCo do almost none, DeMo's top-k grows with k), and once HBM is saturated
// more resident warps only add memory requests in flight, which lowers the
// DRAM rate.  step_warps() takes the fewest warps that still cover the item's
// compute.
constexpr int kStepWarps = 11;
constexpr int kStepWarpsMid = 8;
constexpr int kStepWarpsLight = 6;
int step_warps(int mode, int k, bool bf16, int R, bool sync);
cudaError_t launch_step_small(const StepParams<kSmallReplicas>& p, int mode, bool bf16, int warps, int grid,
                              cudaStream_t st);
cudaError_t launch_step_large(const StepParams<kMaxReplicas>& p, int mode, bool bf16, int warps, int grid,
                              cudaStream_t st);
int encode_warps(int mode, int k, int wire);
cudaError_t launch_encode(const EncodeParams& p, int mode, bool bf16, int warps, int grid, cudaStream_t st);
cudaError_t launch_decode_small(const DecodeParams<kSmallReplicas>& p, int mode, int warps, int grid,
                                cudaStream_t st);
cudaError_t launch_decode_large(const DecodeParams<kMaxReplicas>& p, int mode, int warps, int grid,
                                cudaStream_t st);

// Set the dynamic shared-memory limit of every kernel instantiation.
cudaError_t prepare_step_kernels();
cudaError_t prepare_encode_kernels();
cudaError_t prepare_decode_kernels();

}  // namespace demo
