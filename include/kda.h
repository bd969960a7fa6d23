/*
 * kda.h -- C ABI of libkda, a GB300 (sm_103a) implementation of the
 * Kimi Delta Attention (KDA) token mixer.
 *
 * What the library computes (per sequence n and head h, tokens in order):
 *
 *     S_bar_t = Diag(alpha_t) S_{t-1}                 forget each key channel
 *     e_t     = beta_t (v_t - S_bar_t^T k_t)          correct the prediction
 *     S_t     = S_bar_t + k_t e_t^T                   rank-one delta write
 *     o_t     = S_t^T (scale * q_t)                   read after the write
 *
 * with S a d_k x d_v fp32 matrix (row i = key channel i) and
 * alpha_t = exp(log_alpha_t).  Sources: "Kimi Unveils Delta Attention and K3
 * Architecture Updates", sec. 4 (KDA) and sec. 4.1 (the d_k x d_v five-line
 * form); "Kimi Delta Attention: Channel-Wise Memory Control", "Change one
 * piece of Gated DeltaNet" (key-by-value orientation, o_t = S_t^T q_t).
 *
 * Memory contract shared by every entry point:
 *   - All tensor arguments are DEVICE pointers (HOST pointers for
 *     kda_chunk_fwd_host), contiguous and row-major in the layouts given
 *     below.  q, k, v, out and the states must be 16-byte
 *     aligned; log_alpha, beta and cu_seqlens 4-byte aligned.  The caller
 *     owns every buffer.
 *   - Calls are asynchronous with respect to the host; all work is enqueued
 *     on `stream` (0 = the legacy default stream).
 *   - Host-detectable errors are returned before anything is launched, and
 *     then no output is written.  A launch failure returns KDA_ERR_CUDA.
 *   - Outputs must not overlap inputs, except where stated.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_SUCCESS = 0,
    KDA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or flag   */
    KDA_ERR_UNSUPPORTED = 2,   /* valid request outside the support matrix     */
    KDA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed         */
    KDA_ERR_TIMEOUT = 4        /* a bounded device-side wait gave up           */
} kdaStatus_t;

typedef enum {
    KDA_DTYPE_BF16 = 0,        /* q, k, v and out are bfloat16 */
    KDA_DTYPE_F32 = 1          /* q, k, v and out are float32  */
} kdaDtype_t;

typedef enum {
    KDA_ENGINE_AUTO = 0,       /* tensor-core engine where supported, else SIMT */
    KDA_ENGINE_TENSOR = 1,     /* tcgen05/TMEM chunk engine (bf16, d = 128, C = 64) */
    KDA_ENGINE_SIMT = 2        /* fp32 CUDA-core chunk engine (any supported shape) */
} kdaEngine_t;

/* Problem description: int32 fields and, last, two pointers, so the struct
   has the same layout from C, C++ and ctypes on 64-bit hosts. */
typedef struct {
    int32_t num_seqs;      /* N >= 1: packed sequences (chunk_fwd) / batch (step) */
    int32_t total_tokens;  /* T >= 0: packed tokens (chunk_fwd); must equal N (step) */
    int32_t num_heads;     /* H >= 1 */
    int32_t d_k;           /* key width; d_k == d_v in {16, 32, 64, 128} */
    int32_t d_v;           /* value width */
    int32_t dtype;         /* kdaDtype_t of q, k, v, out */
    int32_t chunk_size;    /* chunk_fwd: 0 = default (64 for d >= 64, else 16),
                              or 16 / 32 / 64; ignored by the step */
    int32_t engine;        /* chunk_fwd: kdaEngine_t; ignored by the step */
    int32_t out_f32;       /* 0: out has the dtype of q; 1: out is float32
                              (bf16 inputs, fp32 results: no output rounding) */
    int32_t num_v_heads;   /* HV: 0 = H.  Otherwise a multiple of H: value
                              heads in groups of HV / H sharing one q/k head
                              (value head j reads q/k head j / (HV / H));
                              v, log_alpha, beta, out and the states carry HV
                              heads, q and k carry H */
    int32_t prologue;      /* kdaPrologue_t bits applied in-kernel to the
                              inputs; 0: q, k, beta, log_alpha used as given */
    const float *gate_bias;   /* [HV, d_k] float32, with KDA_PROLOGUE_GATE */
    const float *gate_A_log;  /* [HV] float32, with KDA_PROLOGUE_GATE */
} kdaShape_t;

/*
 * The fused input prologue ("Linear Attention, From Scratch to Kimi 3",
 * sec. 6 "Exactly how K3 computes the forget values" and sec. 7 "Q/K
 * normalization and query scaling"), applied by every kernel as it loads its
 * inputs, so the raw projections cross HBM once:
 *   KDA_PROLOGUE_L2NORM_QK   q and k are L2-normalised per head,
 *                            x / sqrt(sum x^2 + 1e-6) (the tensor-core
 *                            engine rounds the normalised rows to fp16,
 *                            the precision of its operands)
 *   KDA_PROLOGUE_BETA_LOGITS beta holds logits: beta = sigmoid(beta)
 *   KDA_PROLOGUE_GATE        log_alpha holds the gate projection g:
 *                            log_alpha = -5 sigmoid(exp(A_log[h]) (g + b[h, j]))
 *                            with b = gate_bias, A_log = gate_A_log (the
 *                            page strips this formula; this is the reading
 *                            its stated range, ingredients and sigmoid leave)
 * The scale argument still applies to q after normalisation.
 */
typedef enum {
    KDA_PROLOGUE_L2NORM_QK = 1,
    KDA_PROLOGUE_BETA_LOGITS = 2,
    KDA_PROLOGUE_GATE = 4
} kdaPrologue_t;

/*
 * kda_chunk_fwd -- chunkwise prefill over packed variable-length sequences.
 *
 * Defines: the recurrence above, evaluated chunk by chunk as in "Kimi Unveils
 * Delta Attention and K3 Architecture Updates", sec. 6 (chunk-local cumulative
 * log decay, the causal key-key system and its triangular solve, the WY form
 * of the corrected writes, the single inter-chunk state scan, and the causal
 * outputs).  Chunks restart at every sequence start ("Linear Attention, From
 * Scratch to Kimi 3", sec. 9, cu_seqlens); the last chunk of a sequence may be
 * shorter.  Results do not depend on the chunk size beyond rounding.
 *
 *   q, k          [T, H, d_k]  dtype        (used as given unless
 *                                            KDA_PROLOGUE_L2NORM_QK: then
 *                                            normalised in-kernel)
 *   v             [T, HV, d_v] dtype        HV = shape->num_v_heads, or H
 *   log_alpha     [T, HV, d_k] float32      finite and <= 0 (log retention;
 *                                            gate logits with KDA_PROLOGUE_GATE);
 *                                            16-byte aligned for the tensor-core
 *                                            engine
 *   beta          [T, HV]      float32      finite write strength
 *   scale                      host float   applied to q (pass d_k^-1/2 for
 *                                            the usual 1/sqrt(d_k) read)
 *   initial_state [N, HV, d_k, d_v] float32 or NULL for zero states
 *   cu_seqlens    [N + 1]      int32        device; cu[0] = 0, non-decreasing,
 *                                            cu[N] = T.  NULL means one
 *                                            sequence (then N must be 1).
 *   out           [T, HV, d_v] dtype (float32 if shape->out_f32)
 *                                            written for every token
 *   final_state   [N, HV, d_k, d_v] float32 or NULL (not written).  May be
 *                                            the same buffer as initial_state
 *                                            (in-place resume).
 *
 * Value-head groups (shape->num_v_heads = HV, a multiple of H): value head j
 * runs the recurrence with its own v, log_alpha, beta and state and with q/k
 * head j / (HV / H), as the pages' recurrent launch grid over value heads
 * ("Kimi Unveils Delta Attention and K3 Architecture Updates", sec. 5).
 *
 * cu_seqlens contents are not validated on the host (they live on the
 * device); the kernels clamp every sequence to [0, T], so out-of-range
 * offsets give wrong results but never an out-of-bounds access.
 * Scratch: up to kda_chunk_fwd_workspace_size() bytes, taken with
 * cudaMallocAsync/cudaFreeAsync on `stream` (stream-ordered, pooled by the
 * driver).  Use kda_chunk_fwd_ws to pass caller-owned scratch instead.
 *
 * Kernel overlap: the tensor-core engine launches, in stream order, a chunk
 * table, the chunk-parallel prep, the serial state scan and the output pass.
 * When the scan needs at most half of the SMs, the prep is a persistent grid
 * whose CTAs are all running before the scan is launched; the scan follows
 * the prep's results, and the output pass the prep's and the scan's, through
 * flags in the scratch.  No kernel ever waits on a kernel launched after
 * it, so the call completes under any schedule (a profiler that runs one
 * kernel at a time, other work on other streams holding SMs): the overlap
 * only changes how long it takes.  The results are bit-identical to the
 * sequential order, which calls with more scan CTAs use, and which
 * KDA_LAUNCH_ORDER=sequential forces.  Every wait inside the kernels is
 * bounded (~1 s); a wait that gives up (a hardware fault, not a schedule)
 * leaves KDA_ERR_TIMEOUT in the device status word (kda_device_status).
 *
 * Decayed products: a chunk whose cumulative log decay spans more than 80
 * about its middle token, or about the middle of either half, is evaluated
 * in a slower form (see kda_chunk_path_counts); any finite log_alpha <= 0
 * is accepted.
 *
 * Ranges (tensor-core engine): the state entering each chunk, beta * v and
 * the chunk's folded factors enter its MMAs as fp16 (11-bit significand,
 * largest finite value 65504); the state itself is carried in fp32.  Entries
 * of the state or of beta * v beyond +-65504 overflow to inf in those
 * operands and the results are invalid; tests cover states up to 1e4 in
 * magnitude, keys from a rank-4 subspace and repeated keys with beta = 1.
 * The pages give beta in (0, 1] ("Kimi Unveils Delta Attention and K3
 * Architecture Updates", sec. 2.1 and 3); the library accepts any finite
 * beta, but with unit keys the recurrence itself only stays bounded for
 * beta in [0, 2].  For inputs outside these ranges use KDA_ENGINE_SIMT
 * (fp32 throughout).
 */
kdaStatus_t kda_chunk_fwd(const void *q, const void *k, const void *v,
                          const float *log_alpha, const float *beta, float scale,
                          const float *initial_state, const int32_t *cu_seqlens,
                          void *out, float *final_state, const kdaShape_t *shape,
                          cudaStream_t stream);

/*
 * kda_chunk_fwd_workspace_size -- bytes of device scratch kda_chunk_fwd_ws
 * needs for `shape` (0 for the SIMT engine).  *bytes is written on success.
 */
kdaStatus_t kda_chunk_fwd_workspace_size(const kdaShape_t *shape, size_t *bytes);

/*
 * kda_chunk_fwd_ws -- kda_chunk_fwd with caller-owned scratch: `workspace` is
 * a device buffer of at least kda_chunk_fwd_workspace_size() bytes, 256-byte
 * aligned, not used by anything else until the work on `stream` is done.
 * Allocates nothing.
 */
kdaStatus_t kda_chunk_fwd_ws(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta, float scale,
                             const float *initial_state, const int32_t *cu_seqlens,
                             void *out, float *final_state, const kdaShape_t *shape,
                             void *workspace, size_t workspace_bytes,
                             cudaStream_t stream);

/*
 * kda_chunk_fwd_ws_timed -- kda_chunk_fwd_ws that also records CUDA events
 * on `stream` around its kernels, for measuring each stage on the device:
 * events[0] just before the first launch and events[i] right after launch i,
 * while i < max_events.  *n_recorded (if not NULL) receives the number of
 * events recorded, i.e. launches + 1; stage i spans events[i] -> events[i+1].
 * The events must have been created by the caller (cudaEventCreate or an
 * already-recorded framework event).  Stage order: tensor-core engine =
 * chunk table, intra-chunk prep, state scan, outputs; SIMT engine = one
 * fused kernel.  With events recorded the tensor-core engine runs its
 * kernels one after another (its default order runs the scan and the
 * outputs beside the prep), so the stage times add up to more than the
 * plain call takes.
 */
kdaStatus_t kda_chunk_fwd_ws_timed(const void *q, const void *k, const void *v,
                                   const float *log_alpha, const float *beta, float scale,
                                   const float *initial_state, const int32_t *cu_seqlens,
                                   void *out, float *final_state, const kdaShape_t *shape,
                                   void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream, cudaEvent_t *events,
                                   int32_t max_events, int32_t *n_recorded);

/*
 * kda_chunk_fwd_ws_diag -- a diagnostic form of kda_chunk_fwd_ws for tests of
 * the failure path (no page counterpart).  It forces the tensor-core
 * engine's overlapped order (flags between the kernels) and limits every
 * bounded wait inside the kernels to `wait_cycles` SM clocks (<= 0: the
 * default, ~1 s).  With withhold_prep != 0 it launches the chunk table and
 * the state scan only: the scan's first operand flag is then never
 * published, its waits run out after `wait_cycles`, it sets KDA_ERR_TIMEOUT
 * in the device status word and returns without writing final_state; out is
 * not written.  Arguments otherwise as kda_chunk_fwd_ws; KDA_ERR_UNSUPPORTED
 * unless the problem runs on the tensor-core engine.
 */
kdaStatus_t kda_chunk_fwd_ws_diag(const void *q, const void *k, const void *v,
                                  const float *log_alpha, const float *beta, float scale,
                                  const float *initial_state, const int32_t *cu_seqlens,
                                  void *out, float *final_state, const kdaShape_t *shape,
                                  void *workspace, size_t workspace_bytes,
                                  int32_t withhold_prep, int64_t wait_cycles,
                                  cudaStream_t stream);

/*
 * kda_chunk_path_counts -- how the tensor-core engine evaluated the decayed
 * products exp(G_i - G_j) of "Kimi Unveils Delta Attention and K3
 * Architecture Updates", sec. 6.3 and 6.5, per (chunk, head), summed over the
 * calls on the current device since the last read: counts[0] with one
 * reference token in the middle of the chunk (tensor cores); counts[1] with
 * one reference per half chunk and a third product for the block that spans
 * both halves (tensor cores, used when the decay over half a chunk exceeds
 * e^-80, as K3-range gates down to -5 per token reach); counts[2] with
 * every exponential taken directly on CUDA cores (decays stronger than
 * e^-80 within a quarter chunk).  Synchronises `stream`, then reads and
 * clears the counters.
 */
kdaStatus_t kda_chunk_path_counts(uint64_t counts[3], cudaStream_t stream);

/*
 * kda_chunk_fwd_host_scratch_size -- bytes of device scratch that
 * kda_chunk_fwd_host needs for `shape`: device copies of every input and
 * output plus the engine's workspace.  *bytes is written on success.
 */
kdaStatus_t kda_chunk_fwd_host_scratch_size(const kdaShape_t *shape, size_t *bytes);

/*
 * kda_chunk_fwd_host -- kda_chunk_fwd on HOST buffers: the same operation
 * (chunkwise form, "Kimi Unveils Delta Attention and K3 Architecture
 * Updates", sec. 6) with q, k, v, log_alpha, beta, initial_state, cu_seqlens,
 * out and final_state (and, with KDA_PROLOGUE_GATE, shape->gate_bias and
 * shape->gate_A_log) all in host memory, in the layouts kda_chunk_fwd
 * documents.  On `stream` the call enqueues the host-to-device copies of the
 * inputs, the prefill, and the device-to-host copies of out and final_state,
 * then returns: the results are in the host buffers once the stream's work
 * up to this point is done (cudaStreamSynchronize).  With page-locked host
 * buffers (cudaHostAlloc / cudaHostRegister) the copies are asynchronous,
 * so calls on two streams with two scratch buffers overlap one call's copies
 * with the other's kernels; with pageable buffers the copies block the host.
 *
 * device_scratch: a device buffer of at least
 * kda_chunk_fwd_host_scratch_size() bytes, 256-byte aligned, owned by this
 * call until its work on `stream` is done.  The host buffers must stay valid
 * (and out / final_state untouched) until then too.  Allocates nothing.
 * Errors: as kda_chunk_fwd, plus KDA_ERR_INVALID_ARG for a missing, short or
 * misaligned scratch buffer.
 */
kdaStatus_t kda_chunk_fwd_host(const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, float scale,
                               const float *initial_state, const int32_t *cu_seqlens,
                               void *out, float *final_state, const kdaShape_t *shape,
                               void *device_scratch, size_t scratch_bytes,
                               cudaStream_t stream);

/*
 * kda_chunk_fwd_static -- kda_chunk_fwd for callers that cannot allocate
 * device memory.  No page describes it; it exists for users of this library.
 *
 * Some callers are not allowed to allocate device memory when they run
 * prefill: code inside a host framework that owns every allocation, code on a
 * latency-critical path where an allocation could synchronise the device, or
 * services that must keep a fixed footprint after start-up.  This entry point
 * allocates nothing.  It takes the same arguments as kda_chunk_fwd and runs
 * the same kernels, with scratch taken from a fixed device array of
 * KDA_STATIC_SCRATCH_BYTES that the library reserves when it is loaded.
 *
 *   - The array is held on every GPU that loads the library, until exit.
 *   - Problems whose scratch (kda_chunk_fwd_workspace_size) exceeds
 *     KDA_STATIC_SCRATCH_BYTES are rejected with KDA_ERR_UNSUPPORTED before
 *     anything runs.  With H heads that is about (T/64 + N + 1) * H > 620
 *     (chunk, head) pairs, e.g. more than ~2,300 tokens of one 16-head
 *     sequence.
 *   - All calls share the one array: calls whose GPU work overlaps (other
 *     streams, other host threads) race on it and give wrong results, so
 *     serialise them.  The array keeps the previous call's contents; nothing
 *     in it needs clearing, because the kernels write every byte they read.
 *   - The first call on each device looks up the array's device address
 *     (with that device current).  Make that first call before any stream
 *     capture begins.
 */
#define KDA_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
kdaStatus_t kda_chunk_fwd_static(const void *q, const void *k, const void *v,
                                 const float *log_alpha, const float *beta, float scale,
                                 const float *initial_state, const int32_t *cu_seqlens,
                                 void *out, float *final_state, const kdaShape_t *shape,
                                 cudaStream_t stream);

/*
 * kda_recurrent_step -- one decode token for each of N independent sequences.
 *
 * Defines: one step of the recurrence above ("Kimi Unveils Delta Attention
 * and K3 Architecture Updates", sec. 4.1 five-line form and sec. 5, the fused
 * recurrent schedule for decode; "Kimi Delta Attention: Channel-Wise Memory
 * Control", "The core update in a few lines").  The state streams through
 * once: it is read, decayed, corrected and written back in place.
 *
 *   q, k       [N, H, d_k]  dtype
 *   v          [N, HV, d_v] dtype (HV = shape->num_v_heads, or H; groups as
 *                           for kda_chunk_fwd)
 *   log_alpha  [N, HV, d_k] float32, finite and <= 0
 *   beta       [N, HV]      float32
 *   scale                   host float applied to q
 *   state      [N, HV, d_k, d_v] float32, read and updated in place
 *   out        [N, HV, d_v] dtype (float32 if shape->out_f32)
 *
 * shape->total_tokens must equal shape->num_seqs (one token per sequence);
 * chunk_size and engine are ignored.  Allocates nothing.
 */
kdaStatus_t kda_recurrent_step(const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, float scale,
                               float *state, void *out, const kdaShape_t *shape,
                               cudaStream_t stream);

/*
 * kda_recurrent_fwd -- the token-by-token recurrence over packed sequences of
 * any length, each against its own slot of a state pool (short prefills,
 * multi-token decode and speculative verification, serving batches whose
 * states live in a cache).
 *
 * Defines: the recurrence above applied to every token of every sequence in
 * order ("Kimi Unveils Delta Attention and K3 Architecture Updates", sec. 4.1
 * and sec. 5, the fused recurrent kernel; "Linear Attention, From Scratch to
 * Kimi 3", sec. 9, whose fused kernel loops over the tokens of each
 * cu_seqlens sequence).  Each (sequence, head) state is read from its slot
 * once, carried through the sequence's tokens on chip and written back once,
 * in place.
 *
 *   q, k, v, log_alpha, beta, scale, out   as for kda_chunk_fwd ([T, H or HV, d])
 *   cu_seqlens     int32 [N + 1] device, non-decreasing, 0 .. T; NULL when
 *                  N == 1 (one sequence of T tokens)
 *   state_pool     float32 [num_slots, HV, d_k, d_v], read and updated in place
 *   state_indices  int32 [N] device: the pool slot of each sequence; a
 *                  negative index skips the sequence (its outputs are not
 *                  written, no slot is touched).  NULL: sequence s uses slot s
 *                  (num_slots >= N).  Two sequences must not share a slot.
 *   num_slots      number of slots in the pool; an index >= num_slots makes
 *                  the kernel skip that sequence and set the device status
 *                  word to KDA_ERR_INVALID_ARG (see kda_device_status)
 *
 * shape: num_seqs N, total_tokens T, num_heads H, d_k == d_v in {16, 32, 64,
 * 128}, dtype, out_f32; chunk_size and engine are ignored.  Alignment as for
 * kda_chunk_fwd (state_pool 16 bytes, state_indices 4).  Allocates nothing.
 * Errors detectable on the host return before any launch.
 *
 * This entry has no counterpart on the pages beyond the fused kernel itself:
 * the slot indirection is the serving-side state indexing of a state cache.
 */
kdaStatus_t kda_recurrent_fwd(const void *q, const void *k, const void *v,
                              const float *log_alpha, const float *beta, float scale,
                              const int32_t *cu_seqlens, float *state_pool,
                              const int32_t *state_indices, int32_t num_slots, void *out,
                              const kdaShape_t *shape, cudaStream_t stream);

/*
 * The short causal convolution that precedes the mixer in each KDA layer
 * ("Linear Attention, From Scratch to Kimi 3", sec. 7, "The short
 * convolution is temporal, not channel mixing"): every channel c owns a
 * W-tap filter over time, nothing mixes channels, and each sequence keeps a
 * cache of its W most recent pre-convolution inputs for decode.  q, k and v
 * each take their own call (own weights, own cache).  The tap formula is not
 * in the page text; this library computes, for token t of a sequence,
 *
 *     y[t, c] = act( sum_{i<W} weight[c, i] * x[t - W + 1 + i, c] + bias[c] )
 *
 * act = identity or SiLU (z * sigmoid(z)); inputs before a sequence's first
 * token come from its cache (slot W - 1 the most recent) or are zero.
 */
typedef struct {
    int32_t num_seqs;      /* N >= 1 */
    int32_t total_tokens;  /* T >= 0 packed tokens (prefill; ignored by the step) */
    int32_t channels;      /* C >= 1, a multiple of 8 */
    int32_t width;         /* W: taps, 2 .. 8 (4 in the K3 layer) */
    int32_t dtype;         /* kdaDtype_t of x, y and the caches */
    int32_t activation;    /* 0: none, 1: SiLU */
} kdaConvShape_t;

/*
 * kda_short_conv_fwd -- prefill over packed sequences.
 *
 *   x          [T, C] dtype, 16-byte aligned
 *   weight     [C, W] float32;  bias [C] float32 or NULL (both 16-byte aligned)
 *   cu_seqlens [N + 1] int32 device (NULL when N == 1); sequences never see
 *              each other's tokens
 *   cache_in   [N, C, W] dtype or NULL (zeros): each sequence's inputs before
 *              its first token, oldest first
 *   cache_out  [N, C, W] dtype or NULL: each sequence's W most recent inputs
 *              after the call (may be the same buffer as cache_in)
 *   y          [T, C] dtype, 16-byte aligned, not x
 *
 * Allocates nothing; errors detectable on the host return before any launch.
 */
kdaStatus_t kda_short_conv_fwd(const void *x, const float *weight, const float *bias,
                               const int32_t *cu_seqlens, const void *cache_in, void *cache_out,
                               void *y, const kdaConvShape_t *shape, cudaStream_t stream);

/*
 * kda_short_conv_step -- one decode token per sequence: each cache [N, C, W]
 * shifts by one, takes x [N, C] as its newest slot (in place), and y [N, C]
 * is the filter over it.  shape->total_tokens is ignored.
 */
kdaStatus_t kda_short_conv_step(const void *x, const float *weight, const float *bias,
                                void *cache, void *y, const kdaConvShape_t *shape,
                                cudaStream_t stream);

/*
 * kda_recurrent_bwd -- gradients of kda_chunk_fwd / kda_recurrent_fwd's
 * outputs and final states with respect to every input (training).
 *
 * Defines: reverse-mode differentiation of the recurrence above ("Kimi
 * Unveils Delta Attention and K3 Architecture Updates", sec. 4.1; the pages
 * say the chunkwise form serves training but derive no gradients, so this
 * library derives them from the token recurrence, step by step).  Inputs as
 * for kda_chunk_fwd, plus
 *
 *   d_out            [T, H, d_v] dtype of q, or NULL (zero)
 *   d_final_state    [N, H, d_k, d_v] float32, or NULL (zero)
 *
 * and outputs, all float32 whatever the input dtype:
 *
 *   dq, dk [T, H, d_k];  dv [T, H, d_v];  dlog_alpha [T, H, d_k];
 *   dbeta [T, H];  d_initial_state [N, H, d_k, d_v] or NULL (not written)
 *
 * One CTA per (sequence, head, column tile) carries its columns of the state
 * and of its gradient through the sequence: a forward sweep checkpoints the
 * state every 8 tokens, and the reverse sweep recomputes each 8-token chunk
 * from its checkpoint.  The tiles are 16 columns wide when the (sequence,
 * head) pairs alone would leave most SMs idle (fewer than two per SM), else
 * the whole width.  Scratch (checkpoints and one chunk of states per
 * (sequence, head), about (T / 8 + N) * H * d_k * d_v * 4 +
 * N * H * 8 * d_k * d_v * 4 bytes, plus, with 16-column tiles, the per-tile
 * partial sums of dq, dk, dlog_alpha and dbeta, (d_v / 16) * T * H *
 * (3 * d_k + 1) * 4 bytes) is taken with cudaMallocAsync / cudaFreeAsync on
 * `stream`.  Value-head groups and
 * the input prologue are not supported here (KDA_ERR_UNSUPPORTED).
 */
kdaStatus_t kda_recurrent_bwd(const void *q, const void *k, const void *v,
                              const float *log_alpha, const float *beta, float scale,
                              const float *initial_state, const int32_t *cu_seqlens,
                              const void *d_out, const float *d_final_state, float *dq, float *dk,
                              float *dv, float *dlog_alpha, float *dbeta, float *d_initial_state,
                              const kdaShape_t *shape, cudaStream_t stream);

/*
 * kda_chunk_bwd -- the same gradients as kda_recurrent_bwd, through the
 * chunkwise form (bf16, d_k = d_v = 128; no prologue, no value-head groups:
 * KDA_ERR_UNSUPPORTED otherwise).
 *
 * Defines: the chunk form of "Kimi Unveils Delta Attention and K3
 * Architecture Updates", sec. 6, differentiated by reverse mode.  Its one
 * serial part is the forward scan transposed on the same per-chunk factors,
 *     dS_c = Diag(exp(G_last)) dS_{c+1} - M'^T dS_{c+1} + Q'^T dO_c,
 * with M' = K_end^T W and Q' = s Gamma Q - A^qk W as in kda_chunk_fwd; it
 * runs on the tensor cores with bf16 operands and an fp32 state (the
 * gradients keep fp32 range).  With
 * the state entering every chunk (from the forward engine) and the gradient
 * leaving it, each 64-token chunk's gradients are computed independently, as
 * tensor-core products of the chunk form's factors (tf32 wherever a gradient
 * is an operand) and, where the decay across half a chunk exceeds e^-80,
 * direct exponents for the decayed products.  Arguments, layouts and outputs
 * as for kda_recurrent_bwd; q, k, v and log_alpha must be 16-byte aligned.
 * Scratch (the forward engine's images and states, the per-chunk factors,
 * the state gradients at every chunk boundary and the first gradient
 * kernel's operand images for the second: about (T / 64 + N + 1) * H *
 * 450 KB) is taken with cudaMallocAsync / cudaFreeAsync on `stream`; use
 * kda_chunk_bwd_ws to pass caller-owned scratch instead.
 */
kdaStatus_t kda_chunk_bwd(const void *q, const void *k, const void *v,
                          const float *log_alpha, const float *beta, float scale,
                          const float *initial_state, const int32_t *cu_seqlens,
                          const void *d_out, const float *d_final_state, float *dq, float *dk,
                          float *dv, float *dlog_alpha, float *dbeta, float *d_initial_state,
                          const kdaShape_t *shape, cudaStream_t stream);

/*
 * kda_chunk_bwd_workspace_size -- bytes of device scratch kda_chunk_bwd_ws
 * needs for `shape` (the shape kda_chunk_bwd accepts).  *bytes is written on
 * success; unsupported shapes return KDA_ERR_UNSUPPORTED.
 */
kdaStatus_t kda_chunk_bwd_workspace_size(const kdaShape_t *shape, size_t *bytes);

/*
 * kda_chunk_bwd_ws -- kda_chunk_bwd with caller-owned scratch: `workspace` is
 * a device buffer of at least kda_chunk_bwd_workspace_size() bytes, 256-byte
 * aligned, not used by anything else until the work on `stream` is done
 * (KDA_ERR_INVALID_ARG otherwise).  Allocates nothing.
 */
kdaStatus_t kda_chunk_bwd_ws(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta, float scale,
                             const float *initial_state, const int32_t *cu_seqlens,
                             const void *d_out, const float *d_final_state, float *dq,
                             float *dk, float *dv, float *dlog_alpha, float *dbeta,
                             float *d_initial_state, const kdaShape_t *shape, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *kda_status_string(kdaStatus_t status);

/*
 * kda_device_status -- synchronises `stream`, then reads and clears the
 * library's device-side status word on the current device: KDA_SUCCESS,
 * KDA_ERR_TIMEOUT if a bounded wait inside a kernel gave up since the last
 * call (that kernel's outputs are then invalid), or KDA_ERR_INVALID_ARG if
 * kda_recurrent_fwd met a state index >= num_slots (that sequence was
 * skipped).  Returns KDA_ERR_CUDA if the synchronisation itself fails.
 */
kdaStatus_t kda_device_status(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
