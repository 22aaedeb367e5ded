/*
 * boost_block.h -- C ABI of the GB300 (sm_103a) low-rank bottleneck block.
 *
 * The operation is the CoLA-style bottleneck of "BOOST: BOttleneck-Optimized
 * Scalable Training Framework for Low-Rank Large Language Models"
 * (arXiv 2512.12131; technical summary on gist.science, §2.1-§2.2):
 *
 *     s      = (mean_j x[t,j]^2 + eps)^-1/2              (RMSNorm statistics)
 *     z      = s * (x @ (gamma (.) A))                  (grouped down-projection,
 *                                                        1/rms deferred to the GEMM)
 *     a      = act(z)                                   (bottleneck nonlinearity)
 *     y[i]   = a[:, i*r:(i+1)*r] @ B[i],  i < k         (batched up-projection)
 *
 * forward and backward, bf16 storage with fp32 accumulation.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensors are dense, row-major, bf16 (passed as raw 16-bit storage,
 *   `const void*` / `void*`) unless stated; fp32 tensors are `float*`.
 *   Device pointers must be device memory of the current device; host
 *   pointers are marked "host".
 * - The caller owns every buffer. The library allocates no device memory,
 *   keeps no per-call state between calls, and writes only to the outputs and
 *   the workspace. It holds a few per-device resources for the life of the
 *   process, created on first use: a second stream and two events that let one
 *   GEMM run as two concurrent launches over disjoint rows or columns
 *   ("co-scheduling": a launch of 8-CTA clusters plus a CTA-pair launch on the
 *   SMs no cluster fits); two more streams and three events on which the backward,
 *   when the environment sets BOOST_FORK_STREAMS=1 (off by default),
 *   runs its dB and dA GEMMs concurrently with dx; and cached cluster-occupancy
 *   counts (boost_rmsnorm_rstd_noalloc adds its fixed array, below).
 * - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 *   stream): work on the library's other streams is forked from `stream` and
 *   joined back to it with events, so everything a call enqueues is ordered after
 *   earlier work on `stream` and before later work on it. Calls may be captured into
 *   CUDA graphs (the fork and join become part of the capture). Kernels are launched
 *   as programmatic dependent launches (unless the environment sets BOOST_PDL=0):
 *   each may start its prologue while the kernel before it on the stream finishes,
 *   but waits for that kernel's completion before it reads or writes global memory,
 *   so the ordering above holds for any earlier work. Every argument
 *   is validated on the host before anything is enqueued: a call that returns
 *   BOOST_ERR_INVALID_ARG, _UNSUPPORTED_SHAPE, _ALIGNMENT or _WORKSPACE has
 *   enqueued nothing; BOOST_ERR_CUDA (a launch refused by the runtime) may
 *   leave the first steps of the call enqueued.
 * - Device pointers must be 16-byte aligned. d, k*r, n (and r) must be
 *   multiples of 8 so that every row starts on a 16-byte boundary.
 * - Errors found on the device (a bounded wait that ran out) are recorded in
 *   the workspace's error word and reported by boost_block_check().
 * - Thread safety: calls on different workspaces may run concurrently; the
 *   fork/launch/join sequences on the library's streams are serialised
 *   internally. Two threads capturing graphs on different streams at the same
 *   time would both capture those streams: do not overlap such captures.
 */
#ifndef BOOST_BLOCK_H
#define BOOST_BLOCK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BOOST_OK = 0,
    BOOST_ERR_INVALID_ARG = 1,       /* NULL where a tensor is required, bad enum, negative size */
    BOOST_ERR_UNSUPPORTED_SHAPE = 2, /* d % S != 0, dims not multiples of 8, sizes over limits */
    BOOST_ERR_ALIGNMENT = 3,         /* a pointer is not 16-byte aligned */
    BOOST_ERR_WORKSPACE = 4,         /* workspace NULL, misaligned or smaller than required */
    BOOST_ERR_CUDA = 5,              /* a CUDA runtime call failed (no device, launch failure) */
    BOOST_ERR_TIMEOUT = 6,           /* a kernel's bounded wait ran out (device-side) */
    BOOST_ERR_DEVICE_CHECK = 7       /* a kernel recorded an internal consistency failure */
} boost_status;

typedef enum { BOOST_ACT_IDENTITY = 0, BOOST_ACT_SILU = 1 } boost_act;

/*
 * Shape of one bottleneck block.
 *   T        tokens (rows of x), >= 0
 *   d        input width (the hidden size of the pages' [b,s,d] activations)
 *   r        bottleneck rank per group (the pages' low-rank dimension r)
 *   k        number of grouped projections sharing x (3 for Q/K/V, 2 for gate/up)
 *   n        output width of each up-projection
 *   S        number of column shards of d whose sum-of-squares partials are
 *            computed separately and combined once (Online-RMSNorm, §2.2);
 *            1 <= S and d % S == 0. Only used when has_norm != 0.
 *   eps      RMSNorm epsilon, added to the mean square inside the sqrt
 *   act      boost_act: SiLU (CoLA) or identity (SVD-style bottleneck)
 *   has_norm 1: the block starts with RMSNorm (gamma, rstd, dgamma used);
 *            0: no norm (s == 1, gamma/rstd/dgamma must be NULL)
 */
typedef struct {
    int64_t T, d, r, k, n;
    int32_t S;
    float eps;
    int32_t act;
    int32_t has_norm;
} boost_block_desc;

/* Size in bytes of the workspace boost_block_fwd and boost_block_bwd need for
 * `desc` (the larger of the two; 0 for an invalid desc). The workspace is
 * caller-owned device memory, 256-byte aligned, reusable across calls with the
 * same or a smaller desc; its first 256 bytes hold the error word. */
size_t boost_block_workspace_bytes(const boost_block_desc* desc);

/* Clear the workspace's error word (asynchronous, on `stream`). */
boost_status boost_block_ws_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Forward of one block (technical summary §2.2: Online-RMSNorm, linear-layer
 * grouping).
 *   x      [T, d]          input activations
 *   gamma  [d]             RMSNorm weight (NULL iff has_norm == 0)
 *   A      [d, k*r]        concatenated down-projection weights; group i is
 *                          columns [i*r, (i+1)*r)
 *   B      [k, r, n]       up-projection weights, one [r, n] matrix per group
 *   y      [k, T, n]       out: y[i] = act(s * x @ (gamma (.) A))[:, group i] @ B[i]
 *   rstd   [T] fp32        out, optional (NULL to skip): the row scale s,
 *                          which boost_block_bwd may take back instead of
 *                          recomputing it. Must be NULL when has_norm == 0.
 *   ws     workspace of boost_block_workspace_bytes(desc) bytes or more
 * Steps enqueued: sharded row statistics with one combine; gamma folded into
 * A (bf16); one tensor-core GEMM over all k groups with s and act applied in
 * its epilogue (the normalised x is never written); one batched tensor-core
 * GEMM for the k up-projections.
 */
boost_status boost_block_fwd(const boost_block_desc* desc,
                             const void* x, const void* gamma, const void* A, const void* B,
                             void* y, float* rstd,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * Forward of the gate/up bottleneck of a LLaMA MLP (k == 2: group 0 = gate,
 * group 1 = up) with the SwiGLU forward fused into the up-projection: one
 * tensor-core kernel accumulates the gate and the up group of an output tile in
 * two TMEM accumulators and its epilogue writes gate = y[0] and up = y[1] (the
 * backward needs them) and h = silu(gate) * up, formed from the bf16 gate and up
 * values, so no separate pass reads gate and up back. Workload of the technical
 * summary §4 (LLaMA-2 MLP); the fusion is this library's.
 *   x, gamma, A, B, rstd, ws  as in boost_block_fwd; desc->k must be 2
 *   y      [2, T, n]  out: gate and up
 *   h      [T, n]     out: silu(gate) * up (may be NULL only when T == 0)
 * Errors: as boost_block_fwd, plus BOOST_ERR_INVALID_ARG for k != 2 or a NULL h.
 */
boost_status boost_block_fwd_swiglu(const boost_block_desc* desc,
                                    const void* x, const void* gamma, const void* A,
                                    const void* B, void* y, void* h, float* rstd,
                                    void* ws, size_t ws_bytes, void* stream);

/*
 * Forward of one block with one output group (desc->k == 1) and a residual added
 * in the up-projection's epilogue: y = res + block(x), for a transformer layer's
 * residual connection around a block (the O projection, the MLP's down
 * projection). The sum is formed as a separate add pass would form it: the block's
 * output rounded to bf16, plus res, rounded to bf16. It is bitwise equal to
 * boost_block_fwd followed by boost_add, without writing and reading the block's
 * own output. The residual connection belongs to the LLaMA-2 layer (technical
 * summary §4); the fusion is this library's.
 *   x, gamma, A, B, rstd, ws  as in boost_block_fwd
 *   res    [T, n]     the residual (device, bf16, 16-byte aligned; disjoint from y, or y
 *                     itself); may be NULL only when T == 0
 *   y      [1, T, n]  out: res + block(x)
 * Errors: as boost_block_fwd, plus BOOST_ERR_INVALID_ARG for k != 1, a NULL res or a
 * res that overlaps y without being y, BOOST_ERR_ALIGNMENT for a misaligned res. The up-projection always uses its
 * plain-store epilogue here (no TMA stores).
 */
boost_status boost_block_fwd_residual(const boost_block_desc* desc,
                                      const void* x, const void* gamma, const void* A,
                                      const void* B, const void* res, void* y, float* rstd,
                                      void* ws, size_t ws_bytes, void* stream);

/*
 * Backward of one block with recompute (technical summary §2.2,
 * communication-free low-rank activation checkpointing: only x is kept; the
 * r-wide activation is regenerated inside the block).
 *   x, gamma, A, B   as in boost_block_fwd
 *   rstd   [T] fp32  s from the forward, or NULL to recompute it from x
 *   dy     [k, T, n] upstream gradient of y
 *   dx     [T, d]    out: gradient of x (through the RMSNorm Jacobian)
 *   dgamma [d]       out: gradient of gamma (NULL iff has_norm == 0)
 *   dA     [d, k*r]  out: gradient of A
 *   dB     [k, r, n] out: gradient of B
 * Steps enqueued: (stats if rstd is NULL), fold, one tensor-core kernel with
 * two TMEM accumulators per tile (z recomputed from x, and dy_i @ B_i^T)
 * whose epilogue writes a, dzs = s * act'(z) * (dy B^T) and per-row partials
 * of sum_m dz*z; dB = a^T dy and G = x^T dzs (split-K when too few tiles);
 * dA = gamma (.) G and dgamma_j = sum_m A_jm G_jm; dx = dzs @ A'^T minus the
 * RMSNorm row term (s^2/d) (sum_m dz z) x, applied in the GEMM epilogue.
 */
boost_status boost_block_bwd(const boost_block_desc* desc,
                             const void* x, const void* gamma, const void* A, const void* B,
                             const float* rstd, const void* dy,
                             void* dx, void* dgamma, void* dA, void* dB,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * Backward of one block whose input gradient is added to a residual gradient in
 * the dx epilogue: dx = res + (the block's input gradient). This is the gradient of x
 * through a residual connection x + block(x), with res the gradient arriving by the
 * skip path. Formed as a separate add pass would form it: dx rounded to bf16, plus
 * res, rounded to bf16. It is bitwise equal to boost_block_bwd followed by boost_add.
 *   x, gamma, A, B, rstd, dy, dgamma, dA, dB, ws  as in boost_block_bwd
 *   res    [T, d]  the residual gradient (device, bf16, 16-byte aligned; disjoint from
 *                  dx, or dx itself); may be NULL only when T == 0
 *   dx     [T, d]  out: res + the block's input gradient
 * Errors: as boost_block_bwd, plus BOOST_ERR_INVALID_ARG for a NULL res or a res that
 * overlaps dx without being dx, BOOST_ERR_ALIGNMENT for a misaligned res.
 */
boost_status boost_block_bwd_residual(const boost_block_desc* desc,
                                      const void* x, const void* gamma, const void* A,
                                      const void* B, const float* rstd, const void* dy,
                                      const void* res, void* dx, void* dgamma, void* dA,
                                      void* dB, void* ws, size_t ws_bytes, void* stream);

/*
 * Backward of the down bottleneck of a LLaMA MLP (no norm) whose input is
 * h = silu(gate) * up, with the SwiGLU backward fused into the dgrad epilogue: the
 * block's input gradient dh (rounded to bf16) never reaches HBM; the epilogue reads
 * gate and up and writes dgate = dh * up * silu'(gate) and dup = dh * silu(gate).
 * Workload of the technical summary §4 (LLaMA-2 MLP); fusion is this library's.
 *   h          [T, d]  the block's input (d = the MLP's hidden width)
 *   A, B, dy   as in boost_block_bwd (desc->has_norm must be 0)
 *   gate, up   [T, d]  the gate and up projections h was formed from
 *   dgate, dup [T, d]  out (may be the two halves of one [2, T, d] buffer)
 *   dA, dB             out, as in boost_block_bwd
 */
boost_status boost_block_bwd_swiglu(const boost_block_desc* desc, const void* h, const void* A,
                                    const void* B, const void* dy, const void* gate,
                                    const void* up, void* dgate, void* dup, void* dA, void* dB,
                                    void* ws, size_t ws_bytes, void* stream);

/*
 * Online-RMSNorm statistics alone (technical summary §2.2): per-shard sums of
 * squares and their single combine.
 *   x     [T, d]
 *   ssq   [S, T] fp32 out: ssq[s, t] = sum over columns [s*d/S, (s+1)*d/S) of x[t,j]^2
 *   rstd  [T] fp32   out: (sum_s ssq[s,t] / d + eps)^-1/2, shards summed in index order
 * desc->has_norm must be 1.
 */
boost_status boost_rmsnorm_stats(const boost_block_desc* desc, const void* x,
                                 float* ssq, float* rstd, void* stream);

/*
 * Row scales without any device allocation. The paper has no counterpart to this
 * entry point; it exists for callers that cannot call cudaMalloc, such as code
 * running inside a host framework whose caching allocator owns all device memory
 * (a direct allocation would bypass its accounting or fail under its memory cap)
 * and plugins that are handed only their input and output buffers.
 *   x     [T, d]   input activations (device)
 *   rstd  [T] fp32 out: (sum_s ssq[s,t] / d + eps)^-1/2, shards summed in index
 *                  order; equal to boost_rmsnorm_stats's rstd up to fp32 rounding
 *                  (its kernels split a row among threads differently, so the
 *                  partial sums are added in another order); desc->has_norm must be 1
 * The S x T per-shard partials live in one fixed array of 2^20 floats (4 MiB)
 * inside the library, reserved on every GPU that loads it and held until the
 * process exits. Limit: S*T <= 1048576, else BOOST_ERR_UNSUPPORTED_SHAPE and
 * nothing is enqueued. No call allocates or frees memory. The first call on a
 * device looks up the array's device address with that device current; make that
 * first call before any stream capture. All calls share the array (each call
 * writes every partial it reads, so nothing is cleared and the array keeps the
 * last call's values): calls whose kernels overlap on the GPU race, so serialise
 * them (one stream, or events between streams).
 */
boost_status boost_rmsnorm_rstd_noalloc(const boost_block_desc* desc, const void* x,
                                        float* rstd, void* stream);

/*
 * The batched up-projection alone, from a caller-provided bottleneck activation:
 * y[i] = a[:, group i] @ B[i]; with h non-NULL (k == 2: gate and up groups) the
 * gate/up form of boost_block_fwd_swiglu, also writing h = silu(y[0]) * y[1]. For
 * the checkpoint cut at the bottleneck (technical summary §2.2, low-rank activation
 * checkpointing; §2.1 places the tensor-parallel block boundary at the r-wide
 * activations): a caller that kept only a from the forward regenerates the d-wide
 * section in backward. Bitwise equal to the up-projection inside the block forward.
 *   a   [T, k*r]  bottleneck activation (the block forward's act(z))
 *   B   [k, r, n] up-projection weights
 *   y   [k, T, n] out
 *   h   [T, n]    out, optional (NULL: plain up-projection)
 *   ws  workspace as for boost_block_fwd (its error word is used)
 */
boost_status boost_block_up(const boost_block_desc* desc, const void* a, const void* B,
                            void* y, void* h, void* ws, size_t ws_bytes, void* stream);

/*
 * Forward of one block with the down-projection run as an explicit emulation of
 * the bottleneck-aware tensor-parallel exchange (technical summary §2.1: the
 * down-projection is row-parallel over d, and one all-reduce of the narrow [T, k*r]
 * activations replaces one of d-wide ones; §2.2: the Online-RMSNorm statistics ride
 * on the same exchange). The S column shards of d stand for S ranks:
 *   1. per shard s, the unscaled partial product x[:, shard s] @ A'[shard s, :]
 *      (one split-K tensor-core GEMM whose splits are the shards) and, for a normed
 *      block, the shard's per-row sums of squares: the payload each rank sends;
 *   2. the reduction over the shards in shard order (standing in for the
 *      all-reduce), the row scale from the summed sums of squares (full-d mean) and
 *      a = act(s * z);
 *   3. the batched up-projection, as in boost_block_fwd.
 * Arguments as boost_block_fwd, plus
 *   payload  device fp32 [S*T*k*r + has_norm*S*T], caller-owned, written: the
 *            partial products [S, T, k*r], then (normed blocks) the sums of squares
 *            [S, T]; the values S ranks would contribute to the exchange.
 * y equals boost_block_fwd's up to fp32 summation order (the shard partials are
 * summed after rounding to fp32). Requires d % S == 0 and d / S a multiple of 64
 * (whole k-blocks per shard), else BOOST_ERR_UNSUPPORTED_SHAPE. The fused path
 * (boost_block_fwd) computes the same block without materialising the payload; this
 * entry exists to measure the exchange the pages' design performs.
 */
boost_status boost_block_fwd_btp(const boost_block_desc* desc,
                                 const void* x, const void* gamma, const void* A, const void* B,
                                 void* y, float* rstd, float* payload,
                                 void* ws, size_t ws_bytes, void* stream);

/*
 * Exact bookkeeping of the shard and group partition (host only, no CUDA).
 *   shard_off       host [S+1]: shard s covers columns [shard_off[s], shard_off[s+1]) of d
 *   group_col_off   host [k+1]: group i covers columns [off[i], off[i+1]) of A
 *   exchange_elems  host [1]: values in the one exchange that carries the
 *                   bottleneck partials plus the statistics, T*(k*r+1)
 *                   (technical summary §2.1: payload [b,s,r] instead of [b,s,d])
 * Any output pointer may be NULL.
 */
boost_status boost_block_layout(const boost_block_desc* desc, int64_t* shard_off,
                                int64_t* group_col_off, int64_t* exchange_elems);

/* Byte offsets, inside a workspace for `desc`, of the tensors the block keeps there
 * between its kernels (host only): a [T, k*r] bf16 (the bottleneck activation,
 * written by the forward and again by the backward's recompute), dzs [T, k*r]
 * bf16, the folded weight A' [d, k*r] bf16 and rstd [T] fp32 (used when the
 * caller passes no rstd). Any output pointer may be NULL. For tests and
 * inspection; the contents are only meaningful after the producing call. */
boost_status boost_block_ws_layout(const boost_block_desc* desc, size_t* off_a, size_t* off_dzs,
                                   size_t* off_Ap, size_t* off_rstd);

/* Synchronise `stream`, then read and clear the workspace's error word.
 * Returns BOOST_OK, BOOST_ERR_TIMEOUT / BOOST_ERR_DEVICE_CHECK recorded by a
 * kernel, or BOOST_ERR_CUDA if the stream reports an error. */
boost_status boost_block_check(void* ws, void* stream);

/* Static description of a status code (never NULL). */
const char* boost_status_string(boost_status status);

/*
 * SwiGLU between the gate/up bottleneck and the down bottleneck of the LLaMA
 * MLP shape the pages evaluate (technical summary §4):
 *   h = silu(gate) * up, elementwise over [T, n].
 */
boost_status boost_swiglu_fwd(int64_t T, int64_t n, const void* gate, const void* up,
                              void* h, void* stream);

/* Backward of boost_swiglu_fwd: dgate = dh * up * silu'(gate), dup = dh * silu(gate).
 * dgate and dup may be the two halves of one [2, T, n] buffer. */
boost_status boost_swiglu_bwd(int64_t T, int64_t n, const void* gate, const void* up,
                              const void* dh, void* dgate, void* dup, void* stream);

/* Residual add out = a + b over `count` bf16 elements (count % 8 == 0);
 * out may alias a or b. */
boost_status boost_add(int64_t count, const void* a, const void* b, void* out, void* stream);

/*
 * Debug write counting, the tile-coverage check that stands in for a memory
 * checker (the pages define nothing of the kind). boost_debug_count_writes(counts,
 * capacity) starts recording: every tensor-core GEMM enqueued afterwards (by any
 * entry point, on any stream) is given its own plane of `counts`, shaped like its
 * output, and its epilogues atomically add 1 for each output element they write;
 * boost_debug_count_writes(NULL, 0) stops. counts: device int32 [capacity], zeroed by
 * the caller, 16-byte aligned. boost_debug_count_log(log, max_ops) returns the
 * number of GEMM operations recorded (or -1 if `capacity` ran out, after which
 * operations were left unrecorded) and copies up to max_ops entries of 8 int64 to
 * host `log`: plane offset in counts, M, N, leading dimension, planes per split,
 * splits, plane stride, split stride. Element (s, p, m, c) of an operation sits at
 * offset + s*split_stride + p*plane_stride + m*ld + c; a correct tiling leaves 1 at
 * every m < M, c < N and 0 in the padding c >= N. Process-wide; for tests.
 */
boost_status boost_debug_count_writes(int32_t* counts, int64_t capacity);
int64_t boost_debug_count_log(int64_t* log, int64_t max_ops);

/*
 * Self-test of the bounded wait every kernel uses (failure detection without a
 * GPU fault): launches one tiny kernel that waits on an mbarrier nothing
 * arrives on, with a wait limit of `limit_us` microseconds (1..10^6). The
 * kernel gives up, records BOOST_ERR_TIMEOUT in the workspace's error word and
 * returns; boost_block_check() then reports it and the context stays usable.
 */
boost_status boost_debug_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us,
                                      void* stream);

/*
 * Per-kernel timing of the library's own launches (measurement support; the
 * pages define no such interface). While enabled, each launch is bracketed by
 * two CUDA events on its stream and its algorithmic work (flops, bytes: every
 * operand read once, every output written once) is accumulated per kernel.
 *   boost_profile_enable(1) clears the counters and starts recording,
 *   boost_profile_enable(0) stops; both first collect pending events.
 *   boost_profile_kernel_count() is the number of kernel ids.
 *   boost_profile_read(id, ...) synchronises the pending events and returns the
 *   kernel's static name, launch count, summed event time in milliseconds and
 *   summed algorithmic flops and bytes. Any output pointer may be NULL. A
 *   "launch" here is one timed operation: a GEMM whose rows are split over two
 *   concurrent kernels (the co-scheduled launch shape) counts once, its time
 *   spanning both.
 *   boost_profile_read_kernels(id, &kernels) returns the number of kernels those
 *   operations launched (>= the launch count). kernels must not be NULL.
 * While the stream is being captured into a CUDA graph, the events become the
 * graph's event-record nodes: launch such a graph once, then read the counters
 * (reading returns the events to a pool that later operations reuse, so a graph
 * launched again after that no longer times its own operations).
 * boost_profile_only(id) restricts the timing to the operations of kernel id (-1:
 * every kernel, the default): each bracketing event pair makes the stream wait for
 * the operation before it, which on the LLaMA-2 7B MLP step costs about 3% of the
 * step when every operation is timed, so a measurement that needs one kernel's time
 * inside an otherwise undisturbed step times that kernel alone. Returns
 * BOOST_ERR_INVALID_ARG for an id outside [-1, boost_profile_kernel_count()).
 * Process-wide; intended for one measuring thread.
 */
boost_status boost_profile_enable(int on);
boost_status boost_profile_only(int id);
int boost_profile_kernel_count(void);
boost_status boost_profile_read(int id, const char** name, int64_t* launches, double* total_ms,
                                double* total_flops, double* total_bytes);
boost_status boost_profile_read_kernels(int id, int64_t* kernels);

#ifdef __cplusplus
}
#endif

#endif /* BOOST_BLOCK_H */
