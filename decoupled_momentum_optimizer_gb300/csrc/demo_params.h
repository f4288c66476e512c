// The fused step kernel's parameter block and launchers, and the constants all
// kernels share.  Tensor maps travel by value as __grid_constant__ kernel
// parameters.  The split-path and AdamW kernels' blocks are in demo_launch.h.
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
  long long stall_at;  // test hook of the bounded waits: 1 + the item whose load stalls (warp 0), 0 = off
};

// Launchers (one per translation unit; the other kernels' are in demo_launch.h).
// `grid` CTAs of W warps; each warp walks the tiles gw, gw + W * grid, ...
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
// `warps` picks the build (its shared-memory layout and register budget); `active` warps
// (1..warps) run in each CTA.  kv: DeMo's k when the step is compiled for it (1, 2, 4 or 8),
// else 0.
cudaError_t launch_step_small(const StepParams<kSmallReplicas>& p, int mode, bool bf16, int warps, int kv, int active,
                              int grid, cudaStream_t st);
cudaError_t launch_step_large(const StepParams<kMaxReplicas>& p, int mode, bool bf16, int warps, int kv, int active,
                              int grid, cudaStream_t st);

// The tile kernels are persistent: each assumes one CTA per SM (its grid is at most one CTA
// per SM and its warps walk their tiles statically).  A CTA that asks for more than half of
// an SM's shared memory (228 KB) can never share the SM with another CTA of the same kernel
// -- not even when a programmatically dependent launch places its CTAs while the previous
// kernel still holds some SMs -- so every launch asks for at least this much.
constexpr size_t kOneCtaPerSmSmem = 116 * 1024;
constexpr size_t persistent_smem(size_t bytes) { return bytes > kOneCtaPerSmSmem ? bytes : kOneCtaPerSmSmem; }

// Set the dynamic shared-memory limit of every step kernel instantiation.
cudaError_t prepare_step_kernels();

}  // namespace demo
