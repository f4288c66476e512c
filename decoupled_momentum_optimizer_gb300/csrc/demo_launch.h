// Parameter blocks and launchers of the split-path kernels (encode, decode) and
// of the Decoupled AdamW step.
#pragma once

#include "demo_params.h"

namespace demo {

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
  long long stall_at;  // test hook of the bounded waits (see stall_extra), 0 = off
  // 1: the previous kernel of the stream is one of this library's encodes or decodes that
  // touches none of this kernel's buffers; wait for it only before exiting (see encode_kernel)
  int defer_wait;
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
  // Staged replica r of an item sits at r * sstride in the staging area: vspan + ispan rounded
  // up to 16 bytes (equal to it for bulk copies, which need 16-byte multiples).  Lane copies
  // move lane_unit bytes per copy: 16, or 4 for ternary spans that are not 16-byte multiples.
  unsigned int sstride;
  int lane_unit;
  // More replicas than a staging area holds: each full tile is visited as ceil(R / group)
  // items, item i staging replicas [i * group, (i + 1) * group) and the last one also the
  // theta tile; 0 = one item per tile.
  int group;
  float lr, rcpR;
  unsigned long long hbase;
  float rcp_tab[kMaxReplicas + 1];
  unsigned int* fault;
  long long stall_at;  // test hook of the bounded waits (see stall_extra), 0 = off
};

// Decode CTA shapes: warps per SM and the shared-memory staging per slot for the
// replicas' payload spans (each shape fills the SM's shared memory).  The launch
// takes the shape with the most warps whose staging holds every replica's span;
// when none does, 11 warps stage the replicas that fit 2 KB.
__host__ __device__ constexpr int dec_stage_bytes(int warps) {
  return warps >= 11 ? 2048 : warps == 10 ? 3072 : warps == 9 ? 4608 : 6144;
}
constexpr int kDecShapes[] = {11, 10, 9, 8};

// Staging flavours of the decode kernel, each compiled separately so that no kernel
// carries the code of a staging method it does not use.  Bit 0: the staged spans are
// copied by all 32 lanes of a warp with 16-byte asynchronous copies (one copy group per
// item) instead of lane 0's 1-D bulk copies on the item's barrier; bit 1: one item per
// group of replicas (DecodeParams::group > 0, the 8-warp shape only).  The kernels for
// R <= 4 are plain only.
constexpr int kFlavPlain = 0;
constexpr int kFlavLaneCopy = 1;
constexpr int kFlavGroups = 2;
constexpr int kFlavGroupsLaneCopy = kFlavGroups | kFlavLaneCopy;

// Dense decode (the DiLoCo sync step's receiver; elementwise over groups of four).  The
// launchers of it and of the momentum pass size their grid themselves (one wave of resident
// CTAs on `sms` SMs).
template <int MAXR>
struct DenseParams {
  float* theta;
  const void* vals[MAXR];  // each replica's whole momentum in the wire format
  long long n4;            // n / 4
  int R, wire;
  float lr, rcpR;
};

cudaError_t launch_dense_small(const DenseParams<kSmallReplicas>& p, int sms, cudaStream_t st);
cudaError_t launch_dense_large(const DenseParams<kMaxReplicas>& p, int sms, cudaStream_t st);

// Momentum only (DiLoCo between syncs): m_r <- beta m_r + g_r for every replica.
template <int MAXR>
struct MomentumParams {
  const void* g[MAXR];  // float32 or bfloat16 [n]
  float* m[MAXR];       // float32 [n]
  long long n4;         // n / 4
  int R;
  float beta;
};

cudaError_t launch_momentum_small(const MomentumParams<kSmallReplicas>& p, bool bf16, int sms, cudaStream_t st);
cudaError_t launch_momentum_large(const MomentumParams<kMaxReplicas>& p, bool bf16, int sms, cudaStream_t st);

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

// The encode and decode kernels run kStepWarps warps per CTA unless their own
// selection says otherwise (encode_warps, and the decode's staging shape).
int encode_warps(int mode, int k, int wire, bool bf16, int* kv);
// kv: DeMo's k when the encode is specialised for it (1, 2, 4 or 8 with a float32 or
// 16-bit format; -1, -2, -4 or -8 for those k with the ternary format), else 0.
// `warps` picks the build (shared-memory layout, register budget); `active` warps (1..warps)
// run in each CTA.
cudaError_t launch_encode(const EncodeParams& p, int mode, bool bf16, int warps, int kv, int active, int grid,
                          cudaStream_t st);
// kv: DeMo's k when the decode is specialised for it (1, 2, 4 or 8 with a float32 or
// 16-bit format; -1, -2, -4 or -8 for those k with the ternary format), else 0.
cudaError_t launch_decode_small(const DecodeParams<kSmallReplicas>& p, int mode, int warps, int kv, int flavor,
                                int active, int grid, cudaStream_t st);
cudaError_t launch_decode_large(const DecodeParams<kMaxReplicas>& p, int mode, int warps, int kv, int flavor,
                                int active, int grid, cudaStream_t st);

// Set the dynamic shared-memory limit of every encode and decode kernel instantiation.
cudaError_t prepare_encode_kernels();
cudaError_t prepare_decode_kernels();
// Find the resident CTAs per SM of the dense decode and momentum kernels (their grids).
cudaError_t prepare_dense_kernels();

}  // namespace demo
