/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention forward library.
 *
 * Operation (per sequence and value head hv, independently):
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 * q_t and k_t come from key head hv / (HV / H) (grouped value heads).  This is
 * the recurrence that the chunked listing `naive_chunk_kda` evaluates (page
 * "手撕KDA", section "1 Naive": argument list, shapes, GVA expansion by
 * repeat_interleave, chunk loop).  g is a natural-log decay (<= 0 in practice),
 * beta is used as given (no sigmoid), q and k are used as given (no L2
 * normalisation): those pre-stages are not part of this operation.
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers to contiguous row-major arrays,
 *    16-byte aligned (beta and cu_seqlens: 4-byte aligned).  The caller allocates and owns every buffer; the library
 *    never allocates or frees device memory and never synchronises the device.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream)
 *    and runs asynchronously.  The device that is current at the call must be
 *    the one that holds the tensors and owns `stream`: launches, tensor maps and
 *    per-device set-up follow the current device.
 *  - Arguments are validated on the host before anything is enqueued; on any
 *    error nothing is launched and nothing is written.
 *  - cu_seqlens is not read on the host (that would need a device sync); each
 *    block checks the bounds of its own sequence on the device and reports a
 *    violation through the device status word in the workspace.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_F32 = 0,   /* fp32 q, k, v, o */
  KDA_BF16 = 1   /* bf16 q, k, v, o */
} kda_dtype;

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,     /* bad shape, null required pointer, HV % H != 0, ... */
  KDA_ERR_UNSUPPORTED = 2,     /* valid but not compiled: K or V outside {64, 128} */
  KDA_ERR_ALIGNMENT = 3,       /* a pointer is not 16-byte aligned */
  KDA_ERR_CUDA = 4,            /* a CUDA runtime call failed (launch, attribute, ...) */
  KDA_ERR_DEVICE_TIMEOUT = 5,  /* device status: a bounded on-chip wait gave up */
  KDA_ERR_WORKSPACE = 6,       /* workspace missing or smaller than required */
  KDA_ERR_DEVICE_BOUNDS = 7,   /* device status: cu_seqlens out of order or out of range */
  KDA_ERR_STATIC_SCRATCH = 8,  /* problem larger than kda_chunk_fwd_static_scratch can hold */
  KDA_ERR_DECAY_RANGE = 9      /* device status: g decays faster than the chunk kernels support */
} kda_status;

typedef struct {
  int B;          /* batch (must be 1 when cu_seqlens is given)                  */
  int T;          /* tokens per sequence, or packed total with cu_seqlens         */
  int H;          /* key heads (q, k)                                              */
  int HV;         /* value heads (v, g, beta, state); HV % H == 0                 */
  int K;          /* key dim; 64 or 128                                            */
  int V;          /* value dim; 64 or 128                                          */
  int num_seqs;   /* N when cu_seqlens is given, else 0                            */
  kda_dtype io_dtype;  /* dtype of q, k, v and out; g, beta and states are fp32 */
} kda_shape;

/*
 * Chunked forward (the hot path).  Page "手撕KDA", section "1 Naive"
 * (naive_chunk_kda) defines the operation; the chunked evaluation (within-chunk
 * cumsum of g, decayed keys and queries, strictly lower-triangular L, inverse of
 * (I + L), W/U, serial state carry, intra-chunk output) follows that listing.
 *
 *   q, k          [B, T, H, K]   io_dtype
 *   v             [B, T, HV, V]  io_dtype
 *   g             [B, T, HV, K]  fp32, log-space decay (natural log, <= 0).  The
 *                 tensor-core kernels form every decay factor relative to a point
 *                 inside the 16-token block it spans, so they are exact for any
 *                 decay whose sum over each 16-token block of a sequence (tokens
 *                 16 j .. 16 j + 15 from the sequence start), per key dimension, is
 *                 >= -83; the bounded gate g >= -5 per token satisfies this.  A
 *                 block outside that range sets KDA_ERR_DECAY_RANGE in the device
 *                 status (its outputs are then not meaningful); the
 *                 token-recurrent kernel has no such limit.
 *   beta          [B, T, HV]     fp32
 *   scale         > 0 and finite (the listing's default is K^-0.5; pass it)
 *   initial_state [NS, HV, K, V] fp32 or NULL (zeros); NS = B, or num_seqs
 *   cu_seqlens    [num_seqs + 1] int32 or NULL; cu[0] = 0, non-decreasing,
 *                 cu[num_seqs] = T; sequences are packed along T
 *   out           [B, T, HV, V]  io_dtype; must not alias an input
 *   final_state   [NS, HV, K, V] fp32 or NULL (not written); may alias
 *                 initial_state (each state slice is read before it is written)
 *   workspace     device scratch of at least kda_chunk_fwd_workspace_size()
 *                 bytes, owned by the caller: the device status word and, for
 *                 the tensor-core kernels, record flags and a ring of per-chunk
 *                 records for each (sequence, value head) (16 x 73 KiB each).
 *                 Nothing in it needs initialising.  Calls that share a
 *                 workspace must be ordered on one stream.
 * Returns KDA_OK when the work was enqueued.  T = 0 (or all sequences empty)
 * copies initial_state (or zeros) to final_state.
 * bf16 with K = V = 128 runs a tensor-core chunk kernel; fp32 I/O and other
 * supported sizes run the token-recurrent CUDA-core kernel (same operation).
 * Of the two tensor-core kernels, the split kernel (one CTA per (sequence,
 * value head) carrying the state, the other SMs preparing chunk records) runs
 * when there are at most 40 such units and they fill at most a quarter of the
 * SMs; otherwise the cluster kernel (4 CTAs per unit) runs.  The environment
 * variable KDA_CHUNK_SPLIT=0 or 1, read at each call, forces one of them (1
 * only where the split kernel can hold the units).  Either kernel gives the
 * same results up to rounding order.
 */
KDA_API kda_status kda_chunk_fwd(const kda_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, float scale,
                         const float* initial_state, const int32_t* cu_seqlens, void* out,
                         float* final_state, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Gate activations of kda_chunk_fwd_gated. */
typedef enum {
  KDA_GATE_BOUNDED = 0,   /* g = lower_bound * sigmoid(exp(A_log[hv]) * (g_raw + dt_bias[hv, d])) */
  KDA_GATE_SOFTPLUS = 1   /* g = -exp(A_log[hv]) * softplus(g_raw + dt_bias[hv, d])            */
} kda_gate_kind;

typedef struct {
  kda_gate_kind kind;
  const float* A_log;     /* [HV] fp32, device                                       */
  const float* dt_bias;   /* [HV, K] fp32, device                                    */
  float lower_bound;      /* bounded gate only: < 0 (the pages use -5)               */
} kda_gate;

/*
 * kda_chunk_fwd with the pre-stage fused into the chunk kernels: the raw
 * projections go in, the activations are applied where the chunks are prepared
 * (page "手撕KDA", section 2: l2norm, beta sigmoid and gate activation before the
 * chunk computation; section 5 and page "KDA源码剖析之FlashKDA（上）", part 7: the
 * bounded gate, computed in the kernel that builds the chunk):
 *
 *   q, k      [B, T, H, K]  bf16, raw: each row is scaled by 1 / sqrt(|row|^2 + 1e-6)
 *   v         [B, T, HV, V] bf16
 *   g_raw     [B, T, HV, K] bf16: the gate input (half the bytes of an fp32 g)
 *   beta_raw  [B, T, HV]    fp32: beta = sigmoid(beta_raw)
 *   gate      the activation and its parameters (per value head)
 * and everything else as kda_chunk_fwd (same workspace size).  Requires bf16 I/O
 * and K = V = 128 (the tensor-core kernels); other shapes return
 * KDA_ERR_UNSUPPORTED.  The decay range of kda_chunk_fwd applies to the activated
 * g; the bounded gate with lower_bound >= -5 always meets it.
 */
KDA_API kda_status kda_chunk_fwd_gated(const kda_shape* shape, const void* q, const void* k, const void* v,
                                       const void* g_raw, const float* beta_raw, const kda_gate* gate,
                                       float scale, const float* initial_state, const int32_t* cu_seqlens,
                                       void* out, float* final_state, void* workspace, size_t workspace_bytes,
                                       void* stream);

/*
 * The forward in two passes, through the per-chunk states.  The chunked form carries
 * the state from chunk to chunk and, given the state entering a chunk, computes that
 * chunk's output on its own (page "手撕KDA", section "1 Naive": the chunk loop; section
 * 1.1, the C++ port, keeps the state entering every chunk):
 *
 *   kda_chunk_states: the serial state scan only.  h [B, HV, NT, K, V] bf16 receives
 *     the state entering each chunk (NT = ceil(T / 64); h[.., 0] is the initial state),
 *     final_state (optional) the state after the last token; no output.  Same
 *     workspace as kda_chunk_fwd.  The states are also what a backward pass reads.
 *   kda_chunk_output: o [B, T, HV, V] from h, every chunk in parallel
 *     (o_n = qd_n h[n] + Aqk_n (U_n - W_n h[n])); workspace: the 256-byte status word.
 *
 * Both take bf16 I/O, K = V = 128 and fixed-length sequences (num_seqs = 0); other
 * shapes return KDA_ERR_UNSUPPORTED.  kda_chunk_states_size gives the bytes of h.
 */
KDA_API size_t kda_chunk_states_size(const kda_shape* shape);
KDA_API kda_status kda_chunk_states(const kda_shape* shape, const void* q, const void* k, const void* v,
                                    const float* g, const float* beta, const float* initial_state, void* h,
                                    float* final_state, void* workspace, size_t workspace_bytes, void* stream);
KDA_API kda_status kda_chunk_output(const kda_shape* shape, const void* q, const void* k, const void* v,
                                    const float* g, const float* beta, float scale, const void* h, void* out,
                                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward: the gradients of the loss sum_t <d_out_t, o_t> + <d_final_state, S_final>
 * with respect to every input of kda_chunk_fwd (same shapes and conventions; the
 * method's recurrence, page "手撕KDA" section "1 Naive"), in the chunk form of that
 * page's sections 2 and 4: per 64-token chunk the forward's products are recomputed,
 * the states entering the chunks and the state gradients leaving them are carried by
 * two chains (S' = Q S + R forward, dS = Q^T dS' + B backward), and every chunk's
 * gradients follow in parallel; five launches.  Every product splits each operand into
 * high and low parts and sums three tensor-core products (fp32-level accuracy): tcgen05
 * with bf16 parts for the two chains (K = 128), the value-side gradients and the
 * K x K / K x V products (K = V = 128), warp-level TF32 products elsewhere.  Blocks of
 * 16 tokens whose decay passes about -80 (natural log) per key dimension set status
 * bit 4, as the forward's chunk kernels do; a wait on the kernels' own copies or
 * products that passes the wait limit sets the timeout bit (the call still completes).
 *
 *   d_out          [B, T, HV, V]  io_dtype
 *   d_final_state  [NS, HV, K, V] fp32 or NULL (zeros)
 *   dq, dk         [B, T, H, K]   fp32: summed over the value heads sharing a key head
 *   dv             [B, T, HV, V]  fp32;   dg [B, T, HV, K] fp32;   dbeta [B, T, HV] fp32
 *   d_initial_state [NS, HV, K, V] fp32 or NULL (not written)
 *   workspace      at least kda_backward_workspace_size() bytes: the status word and a
 *                  slot of fp32 intermediates per (chunk, value head) (about 457 KB at
 *                  K = V = 128; with cu_seqlens, ceil(T / 64) + NS chunks are reserved)
 * Any io_dtype and K, V in {64, 128}.  The gradients must not overlap each other or
 * any input.  With the environment variable KDA_BACKWARD=recurrent (read at each call)
 * the same gradients come from reverse mode through the token recurrence instead (fp32
 * on CUDA cores, one CTA per 32 value columns; slower), which the workspace size also
 * covers.
 */
KDA_API size_t kda_backward_workspace_size(const kda_shape* shape);
KDA_API kda_status kda_backward(const kda_shape* shape, const void* q, const void* k, const void* v,
                                const float* g, const float* beta, float scale, const float* initial_state,
                                const int32_t* cu_seqlens, const void* d_out, const float* d_final_state,
                                float* dq, float* dk, float* dv, float* dg, float* dbeta, float* d_initial_state,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Token-recurrent forward: the defining recurrence evaluated token by token on
 * CUDA cores in fp32 (same arguments and results as kda_chunk_fwd; its
 * workspace needs only the 256-byte status word).  Kept as the
 * exact-precision path and as a cross-check for the chunked kernel.
 */
KDA_API kda_status kda_recurrent_fwd(const kda_shape* shape, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, float scale,
                             const float* initial_state, const int32_t* cu_seqlens, void* out,
                             float* final_state, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * Recurrent step for inference: T (typically 1) new tokens of each of B sequences
 * against their resident states, which are updated in place.  The same recurrence
 * as kda_chunk_fwd (page "手撕KDA", section "1 Naive"; its section 5 validates the
 * chunked kernels against this recurrent form), evaluated token by token on CUDA
 * cores in fp32 with the state held in registers for the call's tokens:
 *
 *   q, k    [B, T, H, K]   io_dtype          v  [B, T, HV, V]  io_dtype
 *   g       [B, T, HV, K]  fp32              beta [B, T, HV]   fp32
 *   state   [B, HV, K, V]  fp32, required: read, then overwritten with the state
 *           after the T tokens (must not overlap any other argument)
 *   out     [B, T, HV, V]  io_dtype
 * shape->num_seqs must be 0 (no packing: every sequence advances by T tokens);
 * K and V in {64, 128}.  No workspace, no device-side status: every check is on
 * the host.  At T = 1 and K = V = 128 a call moves 128 KiB of state per
 * (sequence, value head) and is bound by HBM bandwidth.
 */
KDA_API kda_status kda_decode(const kda_shape* shape, const void* q, const void* k, const void* v,
                              const float* g, const float* beta, float scale, float* state, void* out,
                              void* stream);

/* Bytes of device workspace kda_chunk_fwd needs for `shape` (>= 256; also
 * enough for kda_recurrent_fwd).  Depends on the number of sequences and value
 * heads, not on T. */
KDA_API size_t kda_chunk_fwd_workspace_size(const kda_shape* shape);

/*
 * Read the device status word a previous call left in `workspace`: enqueues a
 * 4-byte device-to-host copy on `stream` and waits for that stream.  Returns
 * KDA_OK, KDA_ERR_DEVICE_TIMEOUT, KDA_ERR_DEVICE_BOUNDS or KDA_ERR_DECAY_RANGE (diagnostics only;
 * not for the hot loop).  With several bits set the first of timeout, bounds,
 * decay range is reported.
 */
KDA_API kda_status kda_read_device_status(const void* workspace, void* stream);

/* Static string for a status code. */
KDA_API const char* kda_status_string(kda_status status);

/* Chunk size used by the tensor-core kernel (tokens per chunk). */
KDA_API int kda_chunk_size(void);

/*
 * Name of the kernel kda_chunk_fwd launches for `shape` on the current device
 * (a static string; host-only, enqueues nothing): "kda_chunk_split_kernel",
 * "kda_chunk_fused_kernel", "recurrent_fwd_kernel", or "none" when there is no
 * work (or the shape is malformed).  For diagnostics and benchmarks.
 */
KDA_API const char* kda_chunk_fwd_kernel_name(const kda_shape* shape);

/*
 * How many times kda_chunk_fwd launches that kernel for `shape` (0 when there is no
 * work; host-only).  The split kernel gives every (sequence, value head) unit of a
 * launch its own SM for the serial state scan, at most 38 units per launch on a 152-SM
 * GB300 (three quarters of the SMs prepare chunks).  Problems with more units and at
 * least 16 chunks per sequence (on average) run as several launches of whole sequences,
 * stream-ordered on the caller's stream (packed sequences only when a launch holds one
 * sequence, i.e. more than 19 value heads); other problems with more units run the
 * cluster kernel once.
 */
KDA_API int kda_chunk_fwd_kernel_launches(const kda_shape* shape);

/*
 * kda_chunk_fwd without a caller-provided workspace.  (Not part of the method
 * on the pages: it is a convenience of this library.)
 *
 * Some callers cannot allocate device memory at the point where they run the
 * forward: a host framework that owns every device allocation through its own
 * pool and exposes none of it, a plugin called from code that must not pay
 * for cudaMalloc's implicit device synchronisation, or a latency-critical
 * loop that forbids allocation after start-up.  For them this entry point
 * takes the same inputs and outputs as kda_chunk_fwd but keeps its scratch
 * (the device status word and the chunk kernel's record rings) in one
 * fixed-size array compiled into the library, on every device that loads the
 * library, for the life of the process: about 36.5 MiB
 * (KDA_STATIC_SCRATCH_MAX_UNITS record rings + 16 KiB of status word and
 * record flags).
 *
 *   - Capacity: at most KDA_STATIC_SCRATCH_MAX_UNITS (sequence, value head)
 *     pairs per call (num_seqs or B, times HV); larger problems return
 *     KDA_ERR_STATIC_SCRATCH before anything is enqueued.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *     The first call on each device looks up that device's copy of the array
 *     (cudaGetSymbolAddress) and caches it; make that first call outside any
 *     stream capture.  Later calls only enqueue a memset of the status word
 *     (with the split kernel, also of its record flags: 4 KiB + 128 bytes per
 *     unit) and the kernel.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; the status word (and the split kernel's flags) are cleared at
 *     the start of each call and the rings need no clearing.  Calls whose work overlaps on the GPU (other
 *     streams, other host threads) race on the array and corrupt each other:
 *     order them on one stream.
 *   - status_word: if not NULL, receives the device address of the status
 *     word, to pass to kda_read_device_status().
 */
#define KDA_STATIC_SCRATCH_MAX_UNITS 32
KDA_API kda_status kda_chunk_fwd_static_scratch(const kda_shape* shape, const void* q, const void* k,
                                                const void* v, const float* g, const float* beta,
                                                float scale, const float* initial_state,
                                                const int32_t* cu_seqlens, void* out,
                                                float* final_state, void* stream,
                                                void** status_word);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
