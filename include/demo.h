/*
 * demo.h -- C ABI of the GB300 decoupled-momentum (DeMo / FlexDeMo) shard step.
 *
 * The library runs, on one GPU, the data-parallel optimizer step of FlexDeMo
 * for ONE flat float32 parameter shard and R replicas of it ("DeToNATION:
 * Decoupled Torch Network-Aware Training on Interlinked Online Nodes",
 * Paper-Notes AAAI 2026, section on the method, "1. FlexDeMo" Algorithm 1,
 * from the momentum accumulation to the parameter update; "DeMo: Decoupled
 * Momentum Optimization", abstract):
 *
 *   per replica r:  m_r <- beta m_r + g_r                 (momentum accumulation)
 *                   split m_r into 32-element chunks; select        (extraction)
 *                   q_r = the selected component; m_r <- m_r - q_r     (removal)
 *                   payload_r = q_r's values (ternary sign if asked)
 *   all replicas:   Y = per-slot mean of the payloads (scatter-mean)      (sync)
 *                   Q = inverse transform of Y, theta <- theta - lr Q   (update)
 *
 * Selection ("replication scheme", same page, "2. Replication Schemes" table):
 *   DEMO_MODE_DEMO    orthonormal DCT-II of the chunk, keep the k coefficients
 *                     of largest magnitude (exact ties: lowest index u); the
 *                     payload carries k values and k uint8 indices per chunk,
 *                     in ascending u order.  Q = inverse DCT (DCT-III) of Y.
 *   DEMO_MODE_RANDOM  k positions per chunk drawn from the shared seed (no
 *                     indices sent): draw j of chunk c at step t uses
 *                     h = H(seed, t, c, j), H(s,t,c,j) = sm(sm(sm(sm(s)^t)^c)^j),
 *                     sm = the splitmix64 output function, r_j = (h>>32)*(32-j)>>32,
 *                     position = the r_j-th still-free position (partial
 *                     Fisher-Yates).  Payload: k values in draw order.  Q = Y.
 *   DEMO_MODE_STRIDE  positions o + (32/k) j, o = step mod (32/k); k must
 *                     divide 32.  Payload: k values in j order.  Q = Y.
 *   DEMO_MODE_DILOCO  on steps with (step+1) mod diloco_period == 0 the whole
 *                     momentum is sent (32 values per chunk) and m is zeroed;
 *                     on other steps only the momentum accumulates and theta
 *                     is untouched.
 * The sign flag replaces every sent value by sign(v) in {-1, 0, +1} (same page,
 * "3. Sign function" subsection); m always subtracts the unsigned q.
 * The mean of a slot divides by the number of replicas that sent that slot.
 *
 * Conventions shared by every entry point:
 *   - Pointers named as device pointers are caller-owned device memory of the
 *     current device, 16-byte aligned.  A buffer a call writes may overlap no
 *     other buffer of the call (DEMO_EINVAL); buffers it only reads may be
 *     shared (one gradient for several replicas, one payload for several).
 *     Pointer ARRAYS (g, m, vals, idx) are host arrays of R device pointers.
 *   - n is the shard length, a positive multiple of 32; chunk must be 32.
 *   - Calls enqueue on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and return without synchronising.  The library allocates no memory in
 *     these calls and keeps no per-shard state.
 *   - Argument errors are found on the host before anything is launched and
 *     return a negative status; nothing is printed.  A launch failure returns
 *     DEMO_ECUDA.  A device-side wait that gives up (a copy that never lands)
 *     sets a device fault word read by demo_device_fault().
 *   - Same inputs and (seed, step) give bit-identical outputs; replicas are
 *     combined in the fixed order r = 0..R-1 (no floating-point atomics).
 *   - Non-finite inputs produce unspecified values, never out-of-bounds
 *     accesses.
 *   - Calls may come from several host threads once demo_init has returned
 *     for the device.  demo_step_pipelined enqueues each call's work under a
 *     per-device lock (it shares a pool of events); the kernels of calls that
 *     overlap on the GPU are ordered only by the caller's streams.
 *   - demo_encode(_wire), demo_encode_replicas, demo_decode_update(_wire), demo_step(_wire),
 *     demo_step_pipelined and demo_adamw_step make only kernel launches, event
 *     records and waits and asynchronous device copies on the given streams, so
 *     they may be captured into a CUDA graph (after demo_init).  A captured call
 *     keeps the arguments it was captured with, step and seed included: each
 *     replay repeats that step on the buffers' contents at replay time.
 *     demo_init and demo_device_fault synchronise and must not be captured.
 */
#ifndef DEMO_GB300_H
#define DEMO_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DEMO_CHUNK 32
#define DEMO_MAX_REPLICAS 64

enum demo_mode {
  DEMO_MODE_DEMO = 0,
  DEMO_MODE_RANDOM = 1,
  DEMO_MODE_STRIDE = 2,
  DEMO_MODE_DILOCO = 3
};

enum demo_grad_dtype {
  DEMO_GRAD_F32 = 0,  /* float32 gradients */
  DEMO_GRAD_BF16 = 1  /* bfloat16 gradients, widened exactly to float32 */
};

/*
 * Wire formats of the payload (what the split path writes and reads):
 *   DEMO_WIRE_F32      values float32 [n/32][kv]; DeMo indices uint8 [n/32][k].
 *   DEMO_WIRE_TERNARY  sign must be 1.  Chunks are grouped in tiles of 32 (chunk c
 *                      is bit c mod 32 of tile c / 32; T = ceil(n/32 / 32) tiles).
 *                      Values: uint32 [T][kv][2]; word 0 has bit l set when value j
 *                      of chunk 32t+l is nonzero, word 1 when it is negative.  DeMo
 *                      indices: uint32 [T][k][5]; word b holds bit b of index j of
 *                      every chunk of the tile.  Bits of chunks past the end are 0.
 *                      2 bits per value and 5 per index instead of 32 and 8.
 *   DEMO_WIRE_BF16     values rounded to nearest-even bfloat16, [n/32][kv] 16-bit
 *                      words; indices as DEMO_WIRE_F32.
 *   DEMO_WIRE_F16      values rounded to nearest-even float16, likewise.
 * kv = k for DeMo, Random and Striding and 32 for DiLoCo.  The receiver decodes
 * the rounded values; the ternary format is lossless for signed payloads.  The
 * ternary values come from the sign subsection of the DeToNATION notes ("3. Sign
 * function and hyper-parameters"), which also compares fp32 with fp16 payloads.
 */
enum demo_wire {
  DEMO_WIRE_F32 = 0,
  DEMO_WIRE_TERNARY = 1,
  DEMO_WIRE_BF16 = 2,
  DEMO_WIRE_F16 = 3
};

enum demo_status {
  DEMO_OK = 0,
  DEMO_EINVAL = -1,   /* an argument is out of range or a pointer is NULL */
  DEMO_EALIGN = -2,   /* a device pointer is not 16-byte aligned */
  DEMO_ENODEV = -3,   /* no device, or the device is not an sm_103 GPU */
  DEMO_ECUDA = -4,    /* a CUDA runtime call or a launch failed */
  DEMO_ENOTINIT = -5, /* demo_init() was not called for the current device */
  DEMO_ENOSPACE = -6  /* the request needs more than the library's fixed scratch */
};

/*
 * demo_init -- prepare the library for `device` and make it current.
 * Checks that the device is compute capability 10.3 (GB300), resolves the
 * tensor-map encoder from the CUDA driver and sets the kernels' shared-memory
 * limits.  Idempotent; call it once per device before the other calls (and
 * before any stream capture).  Returns DEMO_OK, DEMO_ENODEV or DEMO_ECUDA.
 */
int demo_init(int device);

/*
 * demo_payload_bytes -- bytes ONE replica sends for one step (host only).
 * Returns the value bytes (float32); *idx_bytes (if not NULL) receives the
 * index bytes (uint8, DeMo only).  DeMo: n/32*k*4 values + n/32*k indices;
 * Random, Striding: n/32*k*4; DiLoCo: 4n on sync steps, else 0.  Returns 0 for
 * invalid arguments.  Source: "2. Replication Schemes" table, whether a scheme
 * transmits indices.
 */
size_t demo_payload_bytes(int mode, int64_t n, int chunk, int k, uint64_t step,
                          int diloco_period, size_t* idx_bytes);

/*
 * demo_encode -- one replica's accumulation, extraction and removal, plus its
 * payload (the send buffer).
 *   g       device, n elements of grad_dtype (read only)
 *   m       device float32 [n], momentum, updated in place to beta m + g - q
 *   vals    device float32: [n/32][k] (DeMo, Random, Striding) or [n] (DiLoCo
 *           sync step); may be NULL on DiLoCo non-sync steps
 *   idx     device uint8 [n/32][k] for DeMo (ascending u per chunk); NULL for
 *           the other modes
 *   k       1..32 (Striding: a divisor of 32; ignored by DiLoCo)
 *   beta    finite float; sign: 0 or 1; diloco_period >= 1 (DiLoCo only)
 *   seed, step: the shared index seed and the 0-based step counter
 * vals and idx (of demo_payload_bytes' sizes) may overlap neither g, m nor
 * each other (DEMO_EINVAL), nor may m overlap g.
 */
int demo_encode(const void* g, int grad_dtype, float* m, int64_t n, int chunk, int k,
                float beta, int mode, int sign, int diloco_period, uint64_t seed,
                uint64_t step, float* vals, uint8_t* idx, void* stream);

/*
 * demo_decode_update -- the synchronisation (scatter-mean of R payloads) and the
 * parameter update.
 *   theta   device float32 [n], updated in place to theta - lr Q
 *   R       1..64 payloads, vals[r] / idx[r] laid out as demo_encode writes
 *           them (idx only for DeMo; pass NULL otherwise)
 *   lr      finite float
 * DiLoCo on a non-sync step leaves theta untouched and launches nothing.
 * A DeMo index byte is used modulo 32 (it never addresses outside the chunk);
 * an index repeated within a chunk is counted once per entry, as every
 * received entry enters the scatter-mean.  The payloads are read only and may
 * be shared between replicas, but none may overlap theta (DEMO_EINVAL).
 */
int demo_decode_update(float* theta, int64_t n, int chunk, int k, float lr, int mode, int R,
                       const float* const* vals, const uint8_t* const* idx,
                       int diloco_period, uint64_t seed, uint64_t step, void* stream);

/*
 * demo_step -- the fused step: demo_encode for every replica followed by
 * demo_decode_update, in one pass over memory; the payloads stay on chip.
 *   theta   device float32 [n], updated in place
 *   g[r]    device [n] of grad_dtype, r = 0..R-1 (read only)
 *   m[r]    device float32 [n], updated in place
 * Same arguments and limits as the split calls; results are bit-identical to
 * demo_encode (r = 0..R-1) followed by demo_decode_update.
 */
int demo_step(float* theta, int64_t n, int chunk, int k, float beta, float lr, int mode,
              int sign, int R, const void* const* g, int grad_dtype, float* const* m,
              int diloco_period, uint64_t seed, uint64_t step, void* stream);

/*
 * Wire-format variants of the calls above.  `vals` / `idx` point to buffers laid
 * out as the wire format states (device memory, 16-byte aligned); the other
 * arguments are those of the plain calls, which equal these with DEMO_WIRE_F32.
 * demo_step_wire rounds the values it accumulates on chip exactly as the split
 * path's receiver would, so fused and split results stay bit-identical for
 * every format.  DEMO_WIRE_TERNARY with sign == 0 returns DEMO_EINVAL.
 */
size_t demo_payload_bytes_wire(int mode, int64_t n, int chunk, int k, uint64_t step, int diloco_period,
                               int wire, size_t* idx_bytes);
int demo_encode_wire(const void* g, int grad_dtype, float* m, int64_t n, int chunk, int k, float beta,
                     int mode, int sign, int diloco_period, uint64_t seed, uint64_t step, int wire,
                     void* vals, void* idx, void* stream);
int demo_decode_update_wire(float* theta, int64_t n, int chunk, int k, float lr, int mode, int R,
                            const void* const* vals, const void* const* idx, int diloco_period,
                            uint64_t seed, uint64_t step, int wire, void* stream);

/*
 * demo_encode_replicas -- demo_encode_wire for every replica r = 0..R-1 of the
 * replication group (1 <= R <= 64) in one call, enqueued in that order on `stream`
 * ("1. FlexDeMo", Algorithm 1, steps 3-5, which each member of the group runs).
 *   g[r], m[r], vals[r], idx[r]   replica r's buffers, each as demo_encode_wire
 *                                 takes them (vals / idx may be NULL where that
 *                                 call allows it: the whole array, or entries)
 * Results are bit-identical to R calls of demo_encode_wire.  Every m, vals and
 * idx is written, so none may overlap another replica's buffers (DEMO_EINVAL; the
 * gradients, read only, may be shared).  Because the replicas share no buffers,
 * each encode kernel after the first starts while the previous one finishes and
 * waits for it only before exiting; separate calls cannot, as the library cannot
 * know that successive calls touch different buffers.
 */
int demo_encode_replicas(const void* const* g, int grad_dtype, float* const* m, int64_t n, int chunk,
                         int k, float beta, int mode, int sign, int R, int diloco_period, uint64_t seed,
                         uint64_t step, int wire, void* const* vals, void* const* idx, void* stream);
int demo_step_wire(float* theta, int64_t n, int chunk, int k, float beta, float lr, int mode, int sign,
                   int R, const void* const* g, int grad_dtype, float* const* m, int diloco_period,
                   uint64_t seed, uint64_t step, int wire, void* stream);

/*
 * demo_step_pipelined -- the split path with its exchange overlapped: the shard
 * is cut into `blocks` blocks of whole 32-chunk tiles (1 <= blocks <= 64); for
 * each block every replica's encode runs on `compute_stream` into send_vals /
 * send_idx, the block's payloads are copied (the loopback of the replication
 * group's all_gather / all-reduce) to recv_vals / recv_idx on `comm_stream`,
 * and the block is decoded from the receive buffers on `compute_stream` while
 * the next block's exchange is in flight (an overlap the DeToNATION notes list
 * as not yet exploited, "limitations": CUDA-stream overlap of communication and
 * computation).  Send and receive buffers are laid out as demo_encode_wire
 * writes a whole shard; results are bit-identical to demo_step_wire.  The
 * Random scheme hashes shard chunk indices, so blocks draw the same positions
 * as a single call.  The call only enqueues work; on return the compute stream
 * holds the whole step.  Events are taken from a pool created by demo_init.
 * Every send and receive buffer is written, so each must be apart from theta,
 * every g[r] and m[r] and every other payload buffer (DEMO_EINVAL).
 */
int demo_step_pipelined(float* theta, int64_t n, int chunk, int k, float beta, float lr, int mode, int sign, int R,
                        const void* const* g, int grad_dtype, float* const* m, int diloco_period, uint64_t seed,
                        uint64_t step, int wire, void* const* send_vals, void* const* send_idx,
                        void* const* recv_vals, void* const* recv_idx, int blocks, void* compute_stream,
                        void* comm_stream);

/*
 * demo_step_pipelined_static -- demo_step_pipelined without caller-provided
 * payload buffers and without any allocation.  The pages have no counterpart:
 * this exists for callers that cannot allocate device memory when they step --
 * for example a framework whose caching allocator already holds the device's
 * memory, or a runtime that forbids allocation after start-up -- and so cannot
 * provide the send / receive buffers demo_step_pipelined needs.
 *
 * The payload send and receive buffers live in one fixed array of 64 MiB of
 * device memory inside the library (32 MiB for the R replicas' send payloads,
 * 32 MiB for the receive payloads, each replica's buffers rounded up to 256
 * bytes; demo_payload_bytes_wire gives the sizes).  Every GPU that loads the
 * library holds that array until the process exits.  A request that does not
 * fit returns DEMO_ENOSPACE and launches nothing.  The call allocates nothing:
 * no cudaMalloc, no cudaFree, no library routine that allocates.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  Every call
 * shares the one array and leaves the last step's payloads in it: each step's
 * encode overwrites every payload word its decode reads, so nothing has to start
 * at zero, but calls whose work overlaps on the GPU (on different streams, or
 * different threads) race on the array.  Arguments and results are those of
 * demo_step_pipelined, which this call runs with buffers inside the array.
 */
int demo_step_pipelined_static(float* theta, int64_t n, int chunk, int k, float beta, float lr, int mode,
                               int sign, int R, const void* const* g, int grad_dtype, float* const* m,
                               int diloco_period, uint64_t seed, uint64_t step, int wire, int blocks,
                               void* compute_stream, void* comm_stream);

/*
 * demo_validate_payload -- host-side check of one replica's DeMo indices
 * (host memory, wire layout as above): every chunk must list k distinct indices
 * in [0, 32) in ascending order.  Returns DEMO_OK, or DEMO_EINVAL with
 * *first_bad (if not NULL) set to the first offending chunk.  A receiver can run
 * it on a payload from an untrusted link; the decode kernels themselves only
 * use an index modulo 32, so a corrupt index never addresses outside its chunk.
 */
int demo_validate_payload(int64_t n, int chunk, int k, int wire, const void* idx_host, int64_t* first_bad);

/*
 * demo_adamw_step -- one Decoupled AdamW step over R replicas ("DeToNATION"
 * notes, method section, "4. Decoupled AdamW": the first and second moments
 * stay local to each replica; the ViT-B bandwidth table runs it with full
 * synchronisation).  With t = step + 1 and every replica r:
 *   m_r <- beta1 m_r + (1 - beta1) g_r,   v_r <- beta2 v_r + (1 - beta2) g_r^2
 *   u_r  = (m_r / (1 - beta1^t)) / (sqrt(v_r / (1 - beta2^t)) + eps)
 * then U = mean_r u_r (the dense sync) and theta <- theta - lr (U + weight_decay theta)
 * (Loshchilov & Hutter's AdamW).  theta, m[r], v[r]: device float32 [n], updated
 * in place; g[r]: device [n] of grad_dtype.  0 <= beta < 1, eps > 0, all finite;
 * n a positive multiple of 32; 1 <= R <= 64.  Same error conventions as above.
 */
int demo_adamw_step(float* theta, int64_t n, float beta1, float beta2, float eps, float lr, float weight_decay,
                    int R, const void* const* g, int grad_dtype, float* const* m, float* const* v, uint64_t step,
                    void* stream);

/* demo_status_string -- a static, human-readable name for a status code. */
const char* demo_status_string(int status);

/*
 * demo_device_fault -- read and clear the fault word of the current device.
 * Synchronises the device.  *code receives 0 when no kernel gave up on a wait
 * since the last call, else a bit set (1: a tile load never completed).
 * Returns DEMO_OK, DEMO_ENOTINIT or DEMO_ECUDA.
 */
int demo_device_fault(unsigned int* code);

/*
 * demo_test_stall_next_launch -- test hook for the failure path of the kernels'
 * device-side waits (failure detection without a GPU fault); the pages have no
 * counterpart.  The next launch of a tile kernel on the current device (the one
 * demo_step, demo_encode or demo_decode_update runs, or their _wire / pipelined
 * variants; not the elementwise DiLoCo and AdamW kernels) makes its first warp
 * announce 16 bytes more than the load of that warp's item `item` (0-based)
 * delivers.  That load's barrier then never completes: the warp's bounded wait
 * gives up after its limit (2 s), the warp sets bit 1 of the fault word, waits
 * (again bounded) for the copies it has in flight and returns, leaving its
 * remaining tiles unprocessed.  Every copy still lands, nothing faults or hangs,
 * and the context stays usable.  A negative item cancels a pending request; a
 * request stays pending until a tile kernel launches.  Returns DEMO_OK or
 * DEMO_ENOTINIT.
 */
int demo_test_stall_next_launch(long long item);

#ifdef __cplusplus
}
#endif

#endif /* DEMO_GB300_H */
