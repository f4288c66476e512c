// Split-path decode, lane-copy flavour: the staged payload spans of a tile (all replicas, or
// the leading ones that fit) are copied by all 32 lanes of the warp with asynchronous copies,
// which moves short spans (up to a few hundred bytes per replica) faster than one bulk copy
// per span, and stages the ternary spans that are not 16-byte multiples (4-byte units), which
// bulk copies cannot.  Many replicas (R > 4): every kernel; R <= 4: the ternary cases only.
// The kernel is in demo_decode_kernel.cuh.
#include "demo_decode_kernel.cuh"

namespace demo {

cudaError_t launch_decode_lane_copy(const DecodeParams<kMaxReplicas>& p, int mode, int warps, int kv, int active,
                                    int grid, cudaStream_t st) {
  return launch_decode_shapes<kMaxReplicas, kFlavLaneCopy>(p, mode, warps, kv, active, grid, st);
}

// R <= 4: only ternary spans that are not 16-byte multiples are staged by lane copies (4-byte
// units); the kernels are those such payloads can reach: DeMo compiled for k = 1 or 2 or
// taking k at run time, and Random and Striding.
template <int WARPS>
static cudaError_t launch_small_w(const DecodeParams<kSmallReplicas>& p, int mode, int kv, int active, int grid,
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
  constexpr int R4 = kSmallReplicas, LC = kFlavLaneCopy;
  switch (mode) {
    case kModeDemo:
      if (kv == -1) return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, R4, WARPS, -1, LC>, p);
      if (kv == -2) return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, R4, WARPS, -2, LC>, p);
      return cudaLaunchKernelEx(&cfg, decode_kernel<kModeDemo, R4, WARPS, 0, LC>, p);
    case kModeRandom: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeRandom, R4, WARPS, 0, LC>, p);
    case kModeStride: return cudaLaunchKernelEx(&cfg, decode_kernel<kModeStride, R4, WARPS, 0, LC>, p);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_lane_copy_small(const DecodeParams<kSmallReplicas>& p, int mode, int warps, int kv,
                                          int active, int grid, cudaStream_t st) {
  if (active < 1 || active > warps) return cudaErrorInvalidValue;
  if (warps == 11) return launch_small_w<11>(p, mode, kv, active, grid, st);
  if (warps == 10) return launch_small_w<10>(p, mode, kv, active, grid, st);
  if (warps == 9) return launch_small_w<9>(p, mode, kv, active, grid, st);
  if (warps == 8) return launch_small_w<8>(p, mode, kv, active, grid, st);
  return cudaErrorInvalidValue;
}

template <int WARPS>
static cudaError_t prepare_small_w() {
  const int bytes = static_cast<int>(persistent_smem(dec_smem(WARPS)));
  constexpr int R4 = kSmallReplicas, LC = kFlavLaneCopy;
  cudaError_t e = set_smem(decode_kernel<kModeDemo, R4, WARPS, -1, LC>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeDemo, R4, WARPS, -2, LC>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeDemo, R4, WARPS, 0, LC>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeRandom, R4, WARPS, 0, LC>, bytes);
  if (e == cudaSuccess) e = set_smem(decode_kernel<kModeStride, R4, WARPS, 0, LC>, bytes);
  return e;
}

cudaError_t prepare_decode_lane_copy() {
  cudaError_t e = prepare_decode_shapes<kMaxReplicas, kFlavLaneCopy>();
  if (e == cudaSuccess) e = prepare_small_w<11>();
  if (e == cudaSuccess) e = prepare_small_w<10>();
  if (e == cudaSuccess) e = prepare_small_w<9>();
  if (e == cudaSuccess) e = prepare_small_w<8>();
  return e;
}

}  // namespace demo
