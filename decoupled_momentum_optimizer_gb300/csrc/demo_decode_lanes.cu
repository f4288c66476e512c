// Split-path decode, lane-copy flavour for many replicas (R > 4): the staged payload
// spans of a tile (all replicas, or the leading ones that fit) are copied by all 32 lanes
// of the warp with 16-byte asynchronous copies, which moves short spans (up to a few
// hundred bytes per replica) faster than one bulk copy per span.  The kernel is in
// demo_decode_kernel.cuh.
#include "demo_decode_kernel.cuh"

namespace demo {

cudaError_t launch_decode_lane_copy(const DecodeParams<kMaxReplicas>& p, int mode, int warps, int kv, int active,
                                    int grid, cudaStream_t st) {
  return launch_decode_shapes<kMaxReplicas, kFlavLaneCopy>(p, mode, warps, kv, active, grid, st);
}

cudaError_t prepare_decode_lane_copy() { return prepare_decode_shapes<kMaxReplicas, kFlavLaneCopy>(); }

}  // namespace demo
