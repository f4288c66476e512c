// Split-path decode, group flavours for many replicas: payloads that no staging area
// holds whole are staged a group of replicas at a time, each full tile visited as one item
// per group, with the 8-warp shape (6 KB of staging per slot); the spans of a group move by
// bulk copies or, for short spans, by lane copies.  The kernel is in demo_decode_kernel.cuh.
#include "demo_decode_kernel.cuh"

namespace demo {

cudaError_t launch_decode_groups(const DecodeParams<kMaxReplicas>& p, int mode, int warps, int kv, int flavor,
                                 int active, int grid, cudaStream_t st) {
  if (warps != kDecShapes[3] || active < 1 || active > warps) return cudaErrorInvalidValue;
  if (flavor == kFlavGroups) return launch_decode_w<kMaxReplicas, kDecShapes[3], kFlavGroups>(p, mode, kv, active, grid, st);
  if (flavor == kFlavGroupsLaneCopy)
    return launch_decode_w<kMaxReplicas, kDecShapes[3], kFlavGroupsLaneCopy>(p, mode, kv, active, grid, st);
  return cudaErrorInvalidValue;
}

cudaError_t prepare_decode_groups() {
  cudaError_t e = prepare_decode_w<kMaxReplicas, kDecShapes[3], kFlavGroups>();
  if (e == cudaSuccess) e = prepare_decode_w<kMaxReplicas, kDecShapes[3], kFlavGroupsLaneCopy>();
  return e;
}

}  // namespace demo
