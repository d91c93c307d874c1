/*
 * kda.h -- C ABI of libkda.so: the chunk-parallel forward pass of Kimi Delta
 * Attention (KDA) on one NVIDIA GB300 (sm_103a).
 *
 * The operation (per sequence s and head h, tokens t of that sequence):
 *
 *   g_t = g_min * sigmoid(theta_t)                               (dk vector)
 *   S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *   o_t = S_t^T q_t
 *
 * The bounded gate is eq. 1 of "Architecture Deep Dive: Kimi K3's MoE, Linear
 * Attention, and Long-Context Engineering" (sec. 3.2, gamma_min = -5) and the
 * scaled-sigmoid log-decay of "Kimi K3 Deep Dive" (section "The Design").  The
 * recurrence is the gated delta rule with channel-wise forgetting that the
 * "Kimi K3" explainer (section "Across the sequence") describes: a fixed-size
 * state S in R^{dk x dv} that each token reads, selectively forgets and writes.
 * The library evaluates it chunk by chunk (16-token chunks, "Kimi K3 Deep
 * Dive", section "The Problem"), every tile through dense products; the
 * tcgen05 path (KDA_PATH_TC) pairs two chunks into one 32-token state step
 * whose decay factors are anchored at the boundary between the two chunks,
 * so every factor stays within e^{+-80} as in a single 16-token chunk.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers are DEVICE pointers on the current CUDA device.  The caller owns
 * every buffer; the library allocates nothing per call.  Inputs are read
 * only; out and final_state are overwritten.  All calls are asynchronous on
 * `stream` and return as soon as the work is queued.
 *
 * Layouts (row-major, contiguous):
 *   fixed length (cu_seqlens == NULL):
 *     q, k, theta  [B, T, H, dk]      v, out  [B, T, H, dv]      beta [B, T, H]
 *     init_state, final_state  fp32 [B, H, dk, dv]   (row i = key channel)
 *   packed variable length (cu_seqlens != NULL):
 *     B is the number of sequences and T the total number of tokens; the
 *     tensors are [1, T, H, .]; cu_seqlens is int32 [B + 1] on the device with
 *     cu_seqlens[0] = 0, cu_seqlens[B] = T, non-decreasing; sequence s is the
 *     tokens [cu_seqlens[s], cu_seqlens[s+1]).  States are [B, H, dk, dv].
 *     The state restarts from init_state[s] (or zero) at every sequence start.
 *   init_state == NULL: every sequence starts from the zero state.
 *   final_state == NULL: the final state is not written.
 *   Lengths need not be multiples of 16: the last chunk of a sequence is
 *   masked (exactly as if padded with k = v = beta = 0, theta = -inf).
 *   The kernels check the packing table on the device, each block for the
 *   sequence it runs (cu_seqlens[0] = 0, cu_seqlens[B] = T, 0 <= start <= end
 *   <= T): a block whose check fails stores nothing and records
 *   KDA_ERR_BAD_SEQLENS in the status word (kda_device_status); no store ever
 *   leaves the rows [0, T) of the tensors.
 *
 * Semantics: no scaling of q and no normalisation of q or k is applied (the
 * caller normalises); beta is used as given (already in (0, 1)); g_min must be
 * negative.  o_t is read after the token-t update.
 *
 * Shapes: dk, dv in {16, 32, 64, 128}; B, H >= 1; T >= 0.
 * Alignment: every tensor pointer 16-byte aligned.
 *
 * Errors: every entry point returns KDA_OK (0) or a negative KDA_ERR_* code
 * and never throws.  Argument errors are found on the host before anything
 * is queued.  A device-side wait that runs out (the tensor-core paths bound
 * every wait) records KDA_ERR_DEVICE_TIMEOUT in a per-device status word that
 * kda_device_status() reads after the caller has synchronised.
 *
 * Threads: every entry point may be called from several host threads at
 * once.  The only state the library keeps is per device and written once:
 * the device check, the kernels' shared-memory attributes, the status-word
 * and scratch-area addresses; and a launch counter of the wrapped schedule
 * (below).  Calls that share an output buffer, a workspace or the no-alloc
 * scratch area must not overlap.
 *
 * Wrapped schedule: a register-resident forward call (KDA_PATH_MMA, the AUTO
 * choice for bf16 at dk = dv = 128) on a fixed-length batch with more
 * (sequence, head) chains than CTAs that can be resident on the device at
 * once (and not a multiple of that number), with final_state != NULL, runs
 * as equal windows of 16-token chunk steps, one per resident CTA, over the
 * chains laid end to end: no SM idles in a last, partial wave.  A chain cut
 * by a window boundary runs its first chunks in one CTA and the rest in
 * another; its fp32 state passes between them through the chain's own
 * final_state slot (overwritten with the true final state at the end) and a
 * flag in static device memory, so the results equal those of one chain
 * per CTA bit for bit.  The launch is cooperative (every CTA resident).  The
 * flags sit in a ring of 64 per-launch regions: up to 64 such calls may be
 * in flight on one device at once; beyond that, overlapping calls may wait
 * for each other's flags until their bounded wait runs out
 * (KDA_ERR_DEVICE_TIMEOUT).  init_state and final_state may be the same
 * buffer.  Without final_state the call runs one chain per CTA.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

/* status codes */
#define KDA_OK 0
#define KDA_ERR_INVALID_ARG (-1)        /* null pointer, bad size, bad g_min, bad enum   */
#define KDA_ERR_MISALIGNED (-2)         /* a tensor pointer not 16-byte aligned          */
#define KDA_ERR_UNSUPPORTED_DEVICE (-3) /* current device is not compute capability 10.3 */
#define KDA_ERR_LAUNCH (-4)             /* the CUDA launch itself failed                 */
#define KDA_ERR_DEVICE_TIMEOUT (-5)     /* a bounded device wait ran out (status word)   */
#define KDA_ERR_CUDA (-6)               /* another CUDA runtime error                    */
#define KDA_ERR_UNSUPPORTED_SHAPE (-7)  /* dk/dv outside {16,32,64,128} for this path    */
#define KDA_ERR_SCRATCH_TOO_SMALL (-8)  /* the fixed scratch area cannot hold the call   */
#define KDA_ERR_BAD_SEQLENS (-9)        /* device status: cu_seqlens not a valid packing  */

/* kernel path selection for kda_chunk_fwd_ex */
#define KDA_PATH_AUTO 0     /* KDA_PATH_MMA for bf16 with dk = dv = 128, else SIMT          */
#define KDA_PATH_SIMT 1     /* fp32 CUDA-core path (any supported dtype/shape)              */
#define KDA_PATH_TC 2       /* tcgen05/TMEM path, state stepped per 32 tokens (bf16, 128)   */
#define KDA_PATH_MMA 3      /* register-resident mma.sync path, 16-token steps (bf16, 128)  */
#define KDA_PATH_TC_SPLIT 4 /* KDA_PATH_TC with the state's bf16 copy as a high/low pair    */
#define KDA_PATH_MMA_TC 5   /* KDA_PATH_MMA with the intra-chunk A, P on tcgen05 (TMEM)     */

/* gate parameterisation (kda_fwd_args.gate) */
#define KDA_GATE_SIGMOID 0   /* g = g_min * sigmoid(theta): the bounded gate (default)     */
#define KDA_GATE_LOG_DECAY 1 /* theta holds the log-decay g <= 0 itself; g_min is ignored  */

/* element types of q, k, v, theta, beta and out */
#define KDA_DTYPE_BF16 0
#define KDA_DTYPE_F32 1

/*
 * kda_chunk_fwd -- bf16 q, k, v, theta and beta; fp32 out; fp32 states.
 * fp32 arithmetic in the gate, the cumulative sums and the state; bf16
 * tensor-core operands with fp32 accumulation in the chunk products (the
 * register-resident path, KDA_PATH_MMA).  kda_chunk_fwd_ex selects the
 * tcgen05 path (KDA_PATH_TC), whose products use tf32 operands for the
 * decayed Gram tile and bf16 high/low pairs for the chunk-local factors
 * (U, P, and the decayed keys of the last state update): more accurate when
 * the decay is slow, at a higher cost per token.
 * `out` is fp32 because the outputs of this operator are heavy-tailed (the
 * largest |o| is typically 14-18 times the RMS of o), so rounding even an
 * exact result to bf16 already moves the largest entries by about 4e-2 of
 * the RMS; an fp32 output keeps the error at the arithmetic's own level.
 * (The pages keep attention outputs in FP32 too: "Kimi K3" explainer,
 * section "Across the sequence".)  kda_chunk_fwd_ex can write bf16 instead.
 * Arguments as in the header comment above.  Returns KDA_OK or KDA_ERR_*.
 */
KDA_API int kda_chunk_fwd(const void* q, const void* k, const void* v, const void* theta,
                          const void* beta, float g_min, const float* init_state, float* out,
                          float* final_state, const int32_t* cu_seqlens, int B, int H, int T,
                          int dk, int dv, cudaStream_t stream);

/*
 * kda_chunk_fwd_f32 -- identical argument list with fp32 q, k, v, theta, beta
 * and out.  Computed entirely in fp32 on CUDA cores (no reduced-precision
 * operands), for callers that need fp32 accuracy.
 */
KDA_API int kda_chunk_fwd_f32(const float* q, const float* k, const float* v, const float* theta,
                              const float* beta, float g_min, const float* init_state, float* out,
                              float* final_state, const int32_t* cu_seqlens, int B, int H, int T,
                              int dk, int dv, cudaStream_t stream);

/* Extended call: the same operation with the element types and the kernel
 * path chosen explicitly.  `dtype` (KDA_DTYPE_*) is the type of q, k, v,
 * theta and beta; `out_dtype` that of out (KDA_DTYPE_F32, or KDA_DTYPE_BF16
 * to halve the output bytes at the cost of bf16 rounding of o; fp32 inputs
 * require an fp32 out).  `path` is KDA_PATH_*; KDA_PATH_TC, KDA_PATH_TC_SPLIT
 * and KDA_PATH_MMA require bf16 inputs and dk = dv = 128 (else
 * KDA_ERR_UNSUPPORTED_SHAPE).  KDA_PATH_TC_SPLIT is KDA_PATH_TC with the
 * state's bf16 copy kept as a high/low pair in the state read-out products:
 * more accurate when many channels decay slowly (the state then carries
 * many chunks), at the cost of a second read-out product per 32 tokens.
 * `gate` selects how theta becomes the log-decay.  KDA_GATE_SIGMOID is the
 * bounded gate of the pages, under which every in-chunk factor e^{-G} stays
 * at or below e^{80}.  KDA_GATE_LOG_DECAY takes g from theta as given (any
 * g <= 0, for instance -softplus of a logit) with no bound.  The
 * register-resident path (KDA_PATH_MMA, the AUTO choice for bf16 at
 * dk = dv = 128) then forms the tiles of every 16-token chunk whose sum of
 * |g| passes 126 ln 2 (about 87.3) position by position, from per-pair
 * factors e^{G_r - G_s} <= 1, so its results stay finite for any g <= 0; such
 * chunks cost several times a dense chunk.  The tcgen05 paths and the SIMT
 * path have no such fallback: they need the sum of |g| over every 16-token
 * chunk (chunks counted from the sequence start) to stay below about 88
 * (fp32 and bf16 overflow of e^{-G}), else their results are not finite. */
typedef struct kda_fwd_args {
  const void* q;
  const void* k;
  const void* v;
  const void* theta;
  const void* beta;
  float g_min;
  const float* init_state;
  void* out;
  float* final_state;
  const int32_t* cu_seqlens;
  int B, H, T, dk, dv;
  int dtype;
  int out_dtype;
  int path;
  int gate; /* KDA_GATE_*; zero-initialised structs get the bounded gate */
} kda_fwd_args;

KDA_API int kda_chunk_fwd_ex(const kda_fwd_args* args, cudaStream_t stream);

/* Device workspace the fused forward entry points (kda_chunk_fwd, _f32, _ex)
 * need: always 0 -- every intermediate of the chunked form lives in shared
 * memory, registers or tensor memory.  Kept so that callers can size a
 * workspace the same way for every entry point (the segmented forward and
 * the backward do need one). */
KDA_API size_t kda_chunk_fwd_workspace_size(int B, int H, int T, int dk, int dv);

/*
 * kda_chunk_fwd_segmented -- the operation of kda_chunk_fwd_ex, cut along the
 * sequence for batches with fewer (sequence, head) chains than SMs (a few
 * very long sequences).  The recurrence is affine in the state, so over any
 * segment S_end = Phi S_start + S_loc, with S_loc the end state from a zero
 * start and Phi (dk x dk) the end state with v = 0 from the identity; each
 * chain is cut into `segments` pieces of whole 32-token units, the pieces'
 * (Phi, S_loc) are computed in parallel, chained in fp32, and every piece is
 * then run from its start state.  The pieces are of equal length, or the
 * first is twice as long as the others when a model of the two launches on
 * the device's SMs says that finishes first (the first piece then runs beside
 * two rounds of the others' (Phi, S_loc) work).  Work grows by about
 * (2P - 3) / P for P segments and runs on otherwise idle SMs.  Results equal
 * the unsegmented call up to rounding order; the workspace size does not
 * depend on the split.
 * Requires bf16 inputs, dk = dv = 128 and a fixed-length batch (cu_seqlens
 * NULL; else KDA_ERR_UNSUPPORTED_SHAPE / KDA_ERR_INVALID_ARG) with B * T
 * below 2^31.  args->path picks the kernel that runs the pieces:
 * KDA_PATH_MMA the register-resident one, KDA_PATH_TC_SPLIT the tcgen05 one
 * with the split state copy, any other value the tcgen05 one.  segments = 1
 * runs the plain path.
 * `workspace`: device memory of at least kda_segmented_workspace_size(B, H, T,
 * dk, dv, segments) bytes, 256-byte aligned, owned by the caller, contents
 * need not be initialised; it is scratch until the stream has passed this
 * call, so calls that may overlap must not share one.  The library allocates
 * nothing.  Returns KDA_OK or KDA_ERR_*.
 */
KDA_API size_t kda_segmented_workspace_size(int B, int H, int T, int dk, int dv, int segments);
/* Test hook (host only, no counterpart on the pages): the plan of a
 * segmented call on a device with `sms` SMs (0: equal pieces) -- out[0] the
 * number of segments, out[1] the tokens of segment 0, out[2] the tokens of
 * each later segment (the last may be shorter).  KDA_OK or
 * KDA_ERR_INVALID_ARG. */
KDA_API int kda_debug_segment_plan(int B, int H, int T, int segments, int sms, int64_t* out);
KDA_API int kda_chunk_fwd_segmented(const kda_fwd_args* args, int segments, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream);

/*
 * kda_chunk_bwd -- gradients of kda_chunk_fwd's outputs and final state with
 * respect to q, k, v, theta, beta and the initial state (the reverse pass of
 * the recurrence of "Kimi K3 Deep Dive", section "Core Innovation 1"), in fp32
 * on CUDA cores, in chunked (WY) form: a forward pass that stores the state at
 * every 16-token chunk start and a reverse pass that carries the state
 * gradient and stores it at every chunk end, then one item per chunk for the
 * remaining gradients, all in one persistent kernel launch on `stream` whose
 * CTAs take the recurrences first and then the chunk items of the chains
 * whose recurrences are done.
 * Requires dk = dv = 128 and a fixed-length batch.  Layouts as kda_chunk_fwd:
 * q, k, theta, dq, dk, dtheta [B,T,H,dk]; v, d_out, dv [B,T,H,dv]; beta,
 * dbeta [B,T,H]; init_state, d_final, d_init [B,H,dk,dv] fp32 (each of the
 * three may be NULL: a zero initial state, no final-state gradient, not
 * written).  `dtype` (KDA_DTYPE_*) is the type of q, k, v, theta, beta; every
 * gradient and d_out/d_final are fp32.  `gate` as kda_fwd_args.gate.
 * `workspace`: device memory of kda_chunk_bwd_workspace_size(B, H, T, dk, dv)
 * bytes (B * H * ceil(T / 16) * 152 KB: two fp32 128 x 128 states and three
 * 16 x 128 fp32 tiles per chunk; then a work queue of 256 bytes plus one int
 * per (sequence, head) chain rounded up to 256 bytes), 16-byte aligned,
 * caller-owned, scratch until the stream has passed the call; it needs no
 * initial contents (the call clears the queue with a memset on `stream`
 * before its kernel launch).  The library allocates nothing.  A given
 * log-decay (KDA_GATE_LOG_DECAY) has the forward
 * pass's limit: the in-chunk sum of |g| below about 88.  Returns KDA_OK or
 * KDA_ERR_*.
 */
typedef struct kda_bwd_args {
  const void* q;
  const void* k;
  const void* v;
  const void* theta;
  const void* beta;
  float g_min;
  const float* init_state;
  const float* d_out;
  const float* d_final;
  float* dq;
  float* dk;
  float* dv;
  float* dtheta;
  float* dbeta;
  float* d_init;
  int B, H, T, dk_dim, dv_dim;
  int dtype;
  int gate;
} kda_bwd_args;

KDA_API size_t kda_chunk_bwd_workspace_size(int B, int H, int T, int dk, int dv);
KDA_API int kda_chunk_bwd(const kda_bwd_args* args, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/*
 * kda_selftest_withheld_handoff -- test hook for the failure path (no
 * counterpart on the pages).  Runs one kernel on the first (sequence, head)
 * chain of `args` (bf16, dk = dv = 128, fixed length, T >= 16): the
 * register-resident kernel if args->path is KDA_PATH_MMA, else the tcgen05
 * kernel, with the producer side withholding the hand-off of the first
 * chunk, and every bounded wait limited to `wait_limit_ns` (> 0).  The
 * consumer's wait runs out, the kernel stops all its roles, and the device
 * status word reads KDA_ERR_DEVICE_TIMEOUT after the stream is synchronised
 * (kda_device_status); the context stays usable.  Nothing is faulted or hung.
 * `workspace`: 256 bytes of caller device memory (the job descriptor).
 * Outputs are left incomplete.  Returns KDA_OK if the launch was made.
 */
KDA_API int kda_selftest_withheld_handoff(const kda_fwd_args* args, long long wait_limit_ns,
                                          void* workspace, size_t workspace_bytes,
                                          cudaStream_t stream);

/*
 * kda_debug_fwd_stages -- test hook (no counterpart on the pages): runs the
 * tcgen05 path (KDA_PATH_TC, or KDA_PATH_TC_SPLIT if args->path says so) on
 * `args` exactly as kda_chunk_fwd_ex does, and in addition writes the
 * intermediate stages of the first (sequence, head) chain -- rank 0 of the
 * launch -- for its first `nsc` 32-token units into `dump` (device, fp32,
 * 16-byte aligned, nsc * kda_debug_stage_floats() floats, caller-owned).
 * Per 32-token unit, in this order (row-major):
 *   A [32][32]   beta_r * (decayed k_r . k_s) for s < r, else 0
 *   P [32][32]   decayed q_t . k_s for s < t, else 0
 *   T [32][32]   (I + A)^{-1} (lower triangular)
 *   W [32][128]  T Diag(beta) (K e^{G}), G the cumulative log-decay from the
 *                unit's start
 *   U [32][128]  T Diag(beta) V - W S (S the state at the unit's start)
 *   eG [128]     e^{G} at the unit's last token
 *   qk [32]      q_t . k_t
 * Requires bf16 inputs and dk = dv = 128.  Returns KDA_OK or KDA_ERR_*.
 */
KDA_API int kda_debug_fwd_stages(const kda_fwd_args* args, float* dump, int nsc,
                                 cudaStream_t stream);
KDA_API int kda_debug_stage_floats(void);

/* Bytes of the scratch area built into the library for
 * kda_chunk_fwd_segmented_noalloc (24 MiB per device). */
#define KDA_NOALLOC_SCRATCH_BYTES (24u << 20)

/*
 * kda_chunk_fwd_segmented_noalloc -- kda_chunk_fwd_segmented over a scratch
 * area that is part of the library itself, for callers that cannot provide
 * a workspace (no allocation of any kind at call time: no cudaMalloc, no
 * allocating library).  The pages have no counterpart of this entry point; it
 * is an interface convenience of this library.
 * - Limit: a call needs kda_segmented_workspace_size(B, H, T, 128, 128,
 *   segments) bytes; above KDA_NOALLOC_SCRATCH_BYTES it returns
 *   KDA_ERR_SCRATCH_TOO_SMALL before anything is queued (use the workspace
 *   entry point then).  Example: B=1, H=32 fits up to segments = 5.
 * - Nothing in the area needs to start at zero; every call writes the parts
 *   it reads.
 * - There is one area per device: calls on the same device whose execution
 *   may overlap (other streams, other host threads) race on it and must be
 *   serialised by the caller.
 * - The area's device address is looked up by the first call made with that
 *   device current (a failed lookup is retried by the next call); make that
 *   first call before any stream capture on that device.  cudaDeviceReset
 *   discards the area: do not call this entry point on a device after
 *   resetting it in the same process.
 * - B * T must stay below 2^31 (KDA_ERR_INVALID_ARG).
 * Arguments, requirements and results otherwise as kda_chunk_fwd_segmented.
 */
KDA_API int kda_chunk_fwd_segmented_noalloc(const kda_fwd_args* args, int segments,
                                            cudaStream_t stream);

/*
 * kda_decode_step -- one recurrent step per (sequence, head): a single new
 * token against a resident fp32 state, which is updated in place.  The same
 * recurrence as kda_chunk_fwd for T = 1 ("Kimi K3 Deep Dive", section "Core
 * Innovation 1"; the fixed-size state of the "Kimi K3" explainer, section
 * "Across the sequence"):
 *   g = g_min * sigmoid(theta),  S <- Diag(e^g) S,
 *   S <- S + beta k (v - S^T k)^T,  o = S^T q.
 * Layouts (contiguous, row-major): q, k, theta [N, H, dk]; v [N, H, dv];
 * beta [N, H]; state [N, H, dk, dv] fp32 (dk rows); out [N, H, dv] fp32.
 * `dtype` (KDA_DTYPE_BF16 or KDA_DTYPE_F32) is the type of q, k, v, theta and
 * beta; the arithmetic is fp32.  All pointers are device pointers, 16-byte
 * aligned, owned by the caller; `state` is read and overwritten, `out` fully
 * written, the inputs only read.  N = 0 is a no-op.  Errors as for
 * kda_chunk_fwd (returned before anything is queued).  Asynchronous on
 * `stream`; the library allocates nothing.
 */
KDA_API int kda_decode_step(const void* q, const void* k, const void* v, const void* theta,
                            const void* beta, float g_min, float* state, float* out, int N, int H,
                            int dk, int dv, int dtype, cudaStream_t stream);

/* Reads the current device's status word (KDA_OK, KDA_ERR_DEVICE_TIMEOUT or
 * KDA_ERR_BAD_SEQLENS).
 * Synchronous with respect to the device's prior work only through the copy:
 * call after synchronising the streams that ran the forward pass.  A nonzero
 * `clear` resets the word to KDA_OK. */
KDA_API int kda_device_status(int clear);

/* The kernel path kda_chunk_fwd_ex would take for these arguments with
 * KDA_PATH_AUTO (KDA_PATH_MMA or KDA_PATH_SIMT), or a negative KDA_ERR_*. */
KDA_API int kda_select_path(int dtype, int dk, int dv);

/* Human-readable text for a status code (static storage, never NULL). */
KDA_API const char* kda_strerror(int code);

/* Library version as 10000*major + 100*minor + patch. */
KDA_API int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
