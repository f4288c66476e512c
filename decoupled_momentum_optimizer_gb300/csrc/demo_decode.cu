// Split-path decode of the DeMo, Random and Striding schemes: scatter-mean of R
// replicas' payloads, inverse transform, theta <- theta - lr Q.  (The DiLoCo sync
// step's decode is elementwise and lives in demo_dense.cu.)
//
// "DeToNATION: Decoupled Torch Network-Aware Training on Interlinked Online
// Nodes" (Paper-Notes, AAAI 2026), method section, "1. FlexDeMo" Algorithm 1
// (synchronisation and the parameter update with Q_t), "2. Replication Schemes" table.
//
// Per warp, theta tiles of 32 chunks stream through a two-slot TMA ring.  With
// each theta tile the replicas' payload spans for the same 32 chunks (contiguous
// in every wire format) are staged in shared memory two items ahead, so their
// latency overlaps the work on earlier tiles: all of them, the leading ones that
// fit, or (many replicas) a group per item.  Replicas that are not staged, spans
// that are not 16-byte multiples and a ragged last tile are read directly.  Lane i combines
// the payload entries of its chunk (replicas in order 0..R-1, read in the
// payload's wire format) in shared-memory accumulators, forms Q and updates its
// theta row, which leaves through the tile's own slot with coalesced stores.
// The arithmetic matches the fused step operation by operation, so split and
// fused results are bit-identical.
//
// The kernel lives in demo_decode_kernel.cuh; this unit compiles the plain flavour (lane 0's
// bulk copies, one item per tile) for every replica count, demo_decode_lanes.cu the
// lane-copy flavour and demo_decode_groups.cu the two group flavours for many replicas.
#include "demo_decode_kernel.cuh"

namespace demo {

cudaError_t launch_decode_small(const DecodeParams<kSmallReplicas>& p, int mode, int warps, int kv, int flavor,
                                int active, int grid, cudaStream_t st) {
  if (flavor == kFlavLaneCopy) return launch_decode_lane_copy_small(p, mode, warps, kv, active, grid, st);
  if (flavor != kFlavPlain) return cudaErrorInvalidValue;
  return launch_decode_shapes<kSmallReplicas, kFlavPlain>(p, mode, warps, kv, active, grid, st);
}

cudaError_t launch_decode_large(const DecodeParams<kMaxReplicas>& p, int mode, int warps, int kv, int flavor,
                                int active, int grid, cudaStream_t st) {
  switch (flavor) {
    case kFlavPlain: return launch_decode_shapes<kMaxReplicas, kFlavPlain>(p, mode, warps, kv, active, grid, st);
    case kFlavLaneCopy: return launch_decode_lane_copy(p, mode, warps, kv, active, grid, st);
    case kFlavGroups:
    case kFlavGroupsLaneCopy: return launch_decode_groups(p, mode, warps, kv, flavor, active, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t prepare_decode_kernels() {
  cudaError_t e = prepare_decode_shapes<kSmallReplicas, kFlavPlain>();
  if (e == cudaSuccess) e = prepare_decode_shapes<kMaxReplicas, kFlavPlain>();
  if (e == cudaSuccess) e = prepare_decode_lane_copy();
  if (e == cudaSuccess) e = prepare_decode_groups();
  return e;
}

}  // namespace demo
