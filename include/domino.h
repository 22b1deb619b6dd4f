/*
 * domino.h -- C ABI of the GB300 (sm_103a) sliced tensor-parallel MLP library.
 *
 * The operation
 * -------------
 * The transformer MLP block  Y = act(X A) B  (GeLU), or
 *                            Y = (silu(X Wg) * (X Wu)) Wd  (SwiGLU),
 * computed the way Domino slices a tensor-parallel layer ("Domino: Eliminating
 * Communication in LLM Training via Generic Tensor Slicing and Overlapping",
 * Abstract: the data dependency of one batch is broken into independent pieces
 * whose communication overlaps the next piece's computation):
 *
 *   - the hidden dimension F is split into P tensor-parallel shards (the
 *     Megatron-LM column-parallel / row-parallel MLP, listed under "Builds on" on
 *     the Domino page): shard p owns columns [p F/P, (p+1) F/P) of A (of Wg and
 *     Wu) and the same rows of B;
 *   - the tokens X are split into mu independent row chunks;
 *   - the output columns can be split into out_slices column slices, a
 *     decomposition finer than a shard ("Design Space Exploration of DMA based
 *     Finer-Grain Compute Communication Overlap", Abstract);
 *   - each shard's row-parallel product is materialised as a partial output and
 *     a separate memory-bound shard-sum adds the P partials -- the stand-in, on
 *     one GPU, for the tensor-parallel all-reduce.  The shard-sum of chunk k
 *     overlaps the GEMMs of chunk k+1.
 *
 * All P shards live on the calling GPU as separate buffers; there are no peers
 * and no collectives.  The result equals the unsharded block up to rounding.
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Arrays are row-major, bf16 unless stated, in device memory of the current
 *    CUDA device.  Weights use the nn.Linear layout (out-features x in-features),
 *    which makes both forward contractions K-major:
 *        A_shards[p]  GeLU/identity: A_p^T  [F_p, d]
 *                     SwiGLU:        [2 F_p, d] = Wg_p^T rows then Wu_p^T rows
 *        B_shards[p]  B_p^T [d, F_p]   (B = Wd for SwiGLU)
 *    with F_p = F / P.  A_shards and B_shards themselves are HOST arrays of P
 *    device pointers.
 *  - Every device pointer must be 16-byte aligned (TMA); the workspace 256-byte.
 *  - The caller owns every buffer.  The library allocates no device memory.
 *  - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  Internally the library may fork work onto its own
 *    streams; it always joins them back into `stream` before returning.
 *  - One call in flight per workspace.
 *  - Argument, shape, alignment and workspace errors are detected on the host,
 *    before anything is launched, and returned as a status.  Device-side waits
 *    are bounded by desc->timeout_ns; a wait that runs out records
 *    DOMINO_ERR_TIMEOUT in the workspace's status word, which
 *    domino_query_device_status() reads.  No C++ exception crosses this ABI.
 */
#ifndef DOMINO_H
#define DOMINO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DOMINO_API __attribute__((visibility("default")))
#else
#define DOMINO_API
#endif

#define DOMINO_MAX_SHARDS 16
#define DOMINO_MAX_PIECES 64 /* mu * out_slices */

typedef enum domino_status {
  DOMINO_OK = 0,
  DOMINO_ERR_INVALID_ARG = 1, /* null pointer, negative size, unknown enum          */
  DOMINO_ERR_UNSUPPORTED = 2, /* shape outside what the kernels handle (see below)   */
  DOMINO_ERR_ALIGNMENT = 3,   /* pointer or leading dimension not 16-byte aligned    */
  DOMINO_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required          */
  DOMINO_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed                   */
  DOMINO_ERR_TIMEOUT = 6,     /* a device-side wait exceeded timeout_ns              */
  DOMINO_ERR_DEVICE = 7       /* current device is not sm_103 (GB300)                */
} domino_status_t;

typedef enum domino_act {
  DOMINO_ACT_GELU = 0,      /* exact GeLU  x * Phi(x)                         */
  DOMINO_ACT_GELU_TANH = 1, /* tanh approximation of GeLU                     */
  DOMINO_ACT_SWIGLU = 2,    /* silu(x Wg) * (x Wu)                            */
  DOMINO_ACT_IDENTITY = 3   /* no activation (used by tests)                  */
} domino_act_t;

typedef enum domino_partial_dtype {
  DOMINO_PARTIAL_F32 = 0, /* each shard's partial output kept in fp32         */
  DOMINO_PARTIAL_BF16 = 1 /* ... rounded to bf16 before the shard-sum         */
} domino_partial_dtype_t;

typedef enum domino_schedule {
  DOMINO_SCHEDULE_SERIAL = 0, /* GEMMs and shard-sums in order on one stream: no overlap  */
  DOMINO_SCHEDULE_STREAMS = 1, /* shard-sum of piece (k,s) on a second stream, released by
                                  an event after its GEMM, overlapping the next piece      */
  DOMINO_SCHEDULE_FUSED = 2    /* forward: GEMM1, GEMM2 and the shard-sum of every chunk in
                                  one persistent cooperative launch; the shard-sum of each
                                  128x256 output tile starts as soon as its P partials are
                                  stored, on the same SMs that keep running GEMM tiles.
                                  backward: dH, then the partial input gradients of every
                                  chunk and their shard-sum in one such launch, then the
                                  weight gradients (STREAMS if the device cannot run the
                                  paired cooperative launch).  Results are bit-identical to
                                  the other schedules; out_slices does not change the work
                                  (the pieces are already tiles).                          */
} domino_schedule_t;

/* desc->flags */
#define DOMINO_FLAG_KERNEL_TIMES 1u /* record CUDA events around every launch; read them
                                       back with domino_kernel_times()                  */
#define DOMINO_FLAG_ONE_CTA 2u      /* SERIAL/STREAMS schedules (and the backward) run their
                                       GEMMs as 2-CTA clusters computing 256x256 tiles with
                                       paired tensor-core MMAs (tcgen05 cta_group::2); this
                                       flag selects one-CTA 128x256 tiles instead          */

typedef struct domino_mlp_desc {
  int64_t M;              /* tokens (rows of X and Y), >= 0                      */
  int64_t d;              /* model width, > 0, multiple of 8                     */
  int64_t F;              /* hidden width (per gate/up for SwiGLU), > 0          */
  int32_t P;              /* shards, 1..DOMINO_MAX_SHARDS, P | F, (F/P) % 8 == 0  */
  int32_t mu;             /* row chunks, >= 1, mu | M                            */
  int32_t out_slices;     /* output column slices, >= 1, out_slices | d,
                             (d / out_slices) % 8 == 0                          */
  int32_t act;            /* domino_act_t                                        */
  int32_t partial_dtype;  /* domino_partial_dtype_t                              */
  int32_t schedule;       /* domino_schedule_t                                   */
  uint32_t flags;         /* DOMINO_FLAG_*                                       */
  int32_t reserve_sms;    /* SMs the library's kernels leave free for work that  */
                          /* runs beside them (a collective, another stream):    */
                          /* persistent grids are sized for (SM count -          */
                          /* reserve_sms) SMs; 0 = all; >= 0 and at most the SM  */
                          /* count - 2 (else DOMINO_ERR_INVALID_ARG)              */
  uint64_t timeout_ns;    /* bound on each device-side wait; 0 = 2 seconds       */
} domino_mlp_desc_t;

/* Bytes of device workspace domino_mlp_fwd/bwd need for this problem
 * (0 for an invalid descriptor).  Layout, all owned by the library while a call
 * runs: the device status words (bytes 0-15), the fused kernel's timeline (bytes
 * 64-87) and, from byte 128, the fused schedule's tile counters (one memset
 * clears timeline and counters before a fused call); then the hidden activations
 * [P][M][F_p] bf16 (unless `saved` is given to fwd) and the P partial outputs
 * [P][M][d] in the partial dtype, each 256-byte aligned.  with_bwd != 0 adds
 * what the backward pass needs (the gradient of the hidden layer). */
DOMINO_API size_t domino_mlp_workspace_size(const domino_mlp_desc_t* desc, int32_t with_bwd);

/* Bytes of the `saved` buffer that fwd fills for bwd (0 if invalid):
 * per shard p, [M][F_p] pre-activation g (and u for SwiGLU, as [M][2 F_p] = g|u)
 * followed by the activation H [M][F_p], all bf16. */
DOMINO_API size_t domino_mlp_saved_size(const domino_mlp_desc_t* desc);

/* Forward pass.  X [M,d]; A_shards/B_shards as above; Y [M,d] written (bf16).
 * M == 0 returns DOMINO_OK after checking the descriptor, touching nothing
 * (every pointer may then be NULL).
 * saved: NULL, or domino_mlp_saved_size() bytes that receive the
 * pre-activations and H for domino_mlp_bwd.
 * Steps per chunk k (and slice s): GEMM1 H_{k,p} = act(X_k A_p) for all p in one
 * launch, fused activation epilogue; GEMM2 Z_{k,p,s} = H_{k,p} B_p[:, s] into
 * shard p's partial buffer; shard-sum Y_k[:, s] = sum_{p=0}^{P-1} Z_{k,p,s}
 * accumulated in fp32 in shard order and rounded once to bf16. */
DOMINO_API domino_status_t domino_mlp_fwd(const domino_mlp_desc_t* desc, const void* X, const void* const* A_shards,
                               const void* const* B_shards, void* Y, void* saved, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Forward pass up to the exchange: the row-parallel partials of every shard,
 * without the sum over shards.  The Domino page ("Domino: Eliminating
 * Communication in LLM Training via Generic Tensor Slicing and Overlapping",
 * Abstract) overlaps each piece's communication with the next piece's
 * computation; on tensor-parallel ranks that communication is the all-reduce of
 * these partials, so this is the computation one rank holds (P = 1: its own
 * shard A_p, B_p) when the all-reduce runs outside this library.
 *  - Z_shards[p]: [M,d] row-major in desc->partial_dtype, 16-byte aligned,
 *    caller-owned; receives Z_p = act(X A_p) B_p (each (k, s) piece exactly as
 *    domino_mlp_fwd computes it before its shard-sum, bit for bit).
 *  - piece_events: NULL, or mu * out_slices cudaEvent_t handles created by the
 *    caller.  Event k * out_slices + s is recorded on `stream` as soon as piece
 *    (k, s) of every Z_p is written (SERIAL / STREAMS: right after that piece's
 *    row-parallel GEMM, so a collective on another stream can start on it while
 *    the next chunk computes; FUSED: after the one launch, which writes all).
 *  - X, A_shards, B_shards, saved, workspace, stream, errors: as domino_mlp_fwd
 *    (the workspace is sized by domino_mlp_workspace_size; its partial buffers
 *    are not used).  Y is not touched. */
DOMINO_API domino_status_t domino_mlp_fwd_partials(const domino_mlp_desc_t* desc, const void* X,
                                                   const void* const* A_shards, const void* const* B_shards,
                                                   void* const* Z_shards, void* const* piece_events, void* saved,
                                                   void* workspace, size_t workspace_bytes, void* stream);

/* Backward pass of the same block (chain rule), sliced the same way: the Domino
 * page ("Domino: Eliminating Communication in LLM Training via Generic Tensor
 * Slicing and Overlapping", Abstract) slices the data dependency of a whole
 * training step, and the backward's exchange is the all-reduce of the input
 * gradient's row-parallel partials, which the shard-sum stands in for here.
 * dY [M,d] in; dX [M,d] out; dA_shards[p] / dB_shards[p] out (bf16, the same
 * layouts as A_shards[p] / B_shards[p]).  `saved` must hold what domino_mlp_fwd
 * wrote for the same X and weights.  workspace: domino_mlp_workspace_size(desc, 1)
 * bytes.  First, over all M in one launch (it exchanges nothing):
 *   dH_p = dY B_p^T, with the activation derivative fused into the
 *     epilogue: dG = dH * act'(g) (SwiGLU: dg = dH * u * silu'(g),
 *     du = dH * silu(g)), from the saved pre-activations.
 * Then per chunk k (and slice s):
 *   the partial input gradient of shard p, dG_{k,p} A_p^T, into shard p's partial
 *     buffer, then dX_k[:, s] = sum over p of the partials (the shard-sum, in fp32,
 *     shard order; it overlaps the next chunk's GEMMs);
 * then, over all M: dA_p = dG_p^T X and dB_p = dY^T H_p (they overlap the last
 * chunk's shard-sum).  With DOMINO_SCHEDULE_FUSED the partial input gradients
 * of every chunk and their shard-sum run as one cooperative launch in which each
 * 128x256 tile of dX is summed as soon as its P partials are stored (the weight
 * gradients follow it).  M == 0 writes zero weight gradients and touches nothing
 * else (X, dY, saved, dX and workspace may then be NULL). */
DOMINO_API domino_status_t domino_mlp_bwd(const domino_mlp_desc_t* desc, const void* X, const void* const* A_shards,
                               const void* const* B_shards, const void* dY, const void* saved, void* dX,
                               void* const* dA_shards, void* const* dB_shards, void* workspace,
                               size_t workspace_bytes, void* stream);

/* The shard-sum alone, the stand-in on one GPU for the tensor-parallel all-reduce
 * whose cost the Domino page (Abstract) hides behind computation:
 * Y[r, c] = bf16( sum_{p=0}^{P-1} partials[p][r, c] ),
 * fp32 accumulation in shard order, one round-to-nearest-even at the end.
 * partials: HOST array of P device pointers to [rows, cols] matrices with leading
 * dimension ld_partial (elements) in `partial_dtype`; Y [rows, cols] bf16 with
 * leading dimension ld_y.  cols, ld_partial and ld_y must be multiples of 8
 * (else DOMINO_ERR_ALIGNMENT), and rows * cols / 8 (the 16-byte vectors of Y,
 * counted with 32-bit indices) below 2^32 (else DOMINO_ERR_UNSUPPORTED). */
DOMINO_API domino_status_t domino_shard_sum(const void* const* partials, int32_t P, int32_t partial_dtype, int64_t rows,
                                 int64_t cols, int64_t ld_partial, void* Y, int64_t ld_y, void* stream);

/* Device-side timeline of the last DOMINO_SCHEDULE_FUSED cooperative launch made
 * with this workspace (the forward, or the backward's partial input gradients;
 * %globaltimer nanoseconds): when its first CTA started, when the
 * last GEMM tile's epilogue finished, and when the last shard-sum finished.
 * reduce_end_ns - gemm_end_ns (if positive) is the reduction time left exposed.
 * Synchronises `stream`; `out` is host memory. */
typedef struct domino_timeline {
  uint64_t start_ns;
  uint64_t gemm_end_ns;
  uint64_t reduce_end_ns;
} domino_timeline_t;
DOMINO_API domino_status_t domino_read_timeline(const void* workspace, void* stream, domino_timeline_t* out);

/* Synchronises `stream`, returns the first device-side error recorded in the
 * workspace's status word since the last query (DOMINO_OK if none) and clears it.
 * The pages have no counterpart: every device-side wait of the library is bounded
 * (desc->timeout_ns), and a wait that runs out records DOMINO_ERR_TIMEOUT here
 * instead of hanging the GPU. */
DOMINO_API domino_status_t domino_query_device_status(void* workspace, void* stream);

/* Self-test of the bounded device-side waits: launches one block that waits, with
 * the same bounded wait the kernels use, for a flag in the workspace header that
 * nothing sets.  After timeout_ns the wait gives up and records
 * DOMINO_ERR_TIMEOUT in the workspace's status words (read them with
 * domino_query_device_status); the context stays usable.  workspace: at least
 * 256 bytes (the header).  Returns the launch status. */
DOMINO_API domino_status_t domino_selftest_wait_timeout(void* workspace, uint64_t timeout_ns, void* stream);

/* Static, NUL-terminated name of a status code. */
DOMINO_API const char* domino_status_string(domino_status_t status);

/* Human-readable detail of the last error returned on the calling host thread. */
DOMINO_API const char* domino_last_error(void);

/* Forward pass without a caller-provided workspace, for callers that cannot
 * allocate device memory when they run the layer (allocation-free real-time
 * loops, hosts that hand out all device memory themselves, runtimes that forbid
 * allocation after start-up).  No counterpart on the pages: this is a packaging
 * of domino_mlp_fwd, not a step of the method.
 *
 * Same arguments and result as domino_mlp_fwd with saved = NULL, but the scratch
 * (hidden activations and shard partials) lives in a fixed array of
 * DOMINO_NOALLOC_SCRATCH_BYTES of device memory inside the library, which every
 * GPU that loads the library holds until the process exits.  The call allocates
 * nothing: no cudaMalloc, no cudaFree, no stream or event creation.
 *  - Runs the SERIAL schedule on `stream` whatever desc->schedule says; desc->flags
 *    must be 0.
 *  - A problem whose workspace (domino_mlp_workspace_size(desc, 0)) exceeds
 *    DOMINO_NOALLOC_SCRATCH_BYTES is rejected with DOMINO_ERR_WORKSPACE.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any stream
 *    capture.
 *  - Every call on a device shares the one array and leaves its contents behind:
 *    calls that overlap on the GPU (other streams, other host threads) race, so
 *    serialise them.
 *  - Device-side waits are bounded as in domino_mlp_fwd.  A wait that runs out
 *    records DOMINO_ERR_TIMEOUT in status words at the start of the array (Y is
 *    then incomplete); read them with domino_mlp_fwd_noalloc_status before the
 *    next call on the device, which clears them. */
#define DOMINO_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB */
DOMINO_API domino_status_t domino_mlp_fwd_noalloc(const domino_mlp_desc_t* desc, const void* X,
                                                  const void* const* A_shards, const void* const* B_shards, void* Y,
                                                  void* stream);

/* Device status of the most recent domino_mlp_fwd_noalloc call on the current
 * device: synchronises `stream`, returns DOMINO_OK or the error a device-side
 * wait recorded (DOMINO_ERR_TIMEOUT; detail in domino_last_error) and clears it.
 * If `header` is non-NULL it receives the device address of the array's
 * 256-byte header (status words at bytes 0-15), which can be handed to
 * domino_selftest_wait_timeout as its workspace to exercise this report.  Does
 * the per-device set-up of domino_mlp_fwd_noalloc if no call has done it yet;
 * allocates nothing. */
DOMINO_API domino_status_t domino_mlp_fwd_noalloc_status(void* stream, void** header);

/* Kernel launch timing.  Every call made with DOMINO_FLAG_KERNEL_TIMES records a
 * CUDA event before and after each of its kernel launches, on the stream the
 * kernel is launched on, and appends one record per launch to a process-wide
 * log (events are pooled; the log holds at most DOMINO_MAX_TIMED_LAUNCHES
 * records, further launches are not recorded). */
#define DOMINO_MAX_TIMED_LAUNCHES 262144

typedef enum domino_kernel_kind {
  DOMINO_KERNEL_GEMM1 = 0,     /* column-parallel GEMM + activation, all shards        */
  DOMINO_KERNEL_GEMM2 = 1,     /* row-parallel GEMM into the partial buffers           */
  DOMINO_KERNEL_SHARD_SUM = 2, /* sum of the P partials                                */
  DOMINO_KERNEL_BWD_DH = 3,    /* backward: dH and the activation derivative           */
  DOMINO_KERNEL_BWD_DX = 4,    /* backward: partial input gradients                    */
  DOMINO_KERNEL_BWD_DW = 5,    /* backward: weight gradients                           */
  DOMINO_KERNEL_FUSED = 6,     /* the fused forward kernel (whole call)                */
  DOMINO_KERNEL_ATTN = 7,      /* attention core of the attention block                */
  DOMINO_KERNEL_BWD_DX_FUSED = 8, /* backward, FUSED schedule: the partial input gradients of
                                     every chunk and their shard-sum in one launch          */
  DOMINO_KERNEL_ATTN_OUT_FUSED = 9 /* attention block, FUSED schedule: one chunk's output
                                     projection and its shard-sum in one launch            */
} domino_kernel_kind_t;

typedef struct domino_kernel_time {
  int32_t call;     /* index of the timed call since the last reset (0-based)          */
  int32_t kind;     /* domino_kernel_kind_t                                            */
  int32_t chunk;    /* k                                                               */
  int32_t slice;    /* s (0 for kernels that cover all slices)                         */
  int32_t stream;   /* 0: the caller's stream, 1: the library's reduction stream       */
  float start_ms;   /* event before the launch, relative to the call's first event     */
  float end_ms;     /* event after the launch, same origin                             */
} domino_kernel_time_t;

/* Waits for the recorded events and copies up to max_records records (oldest
 * first) into `out` (host memory; may be NULL to only count).  Returns the
 * number of records logged since the last reset. */
DOMINO_API int32_t domino_kernel_times(domino_kernel_time_t* out, int32_t max_records);

/* Empties the log (the pooled events are kept for reuse). */
DOMINO_API void domino_kernel_times_reset(void);

/* The sliced tensor-parallel attention block, the other half of the layer
 * (Domino page, Abstract: the whole layer is sliced into independent pieces;
 * Megatron-LM's split, titles under "Builds on" on that page):
 *   Q | K | V = X Wqkv                              column-parallel, by heads
 *   O_h = softmax(Q_h K_h^T / sqrt(dh) + causal mask) V_h    per sequence, head
 *   Y = [O_0 | ... | O_{H-1}] Wo                    row-parallel, by heads
 * X holds B sequences of S tokens ([B S, d] bf16, sequence b = rows b S ..
 * (b+1) S - 1); token t attends to tokens 0..t of its own sequence.  The H heads
 * are split into P shards of Hp = H / P heads (shard p: heads p Hp .. (p+1) Hp -
 * 1), the sequences into mu chunks of B / mu whole sequences.  Per chunk k: the
 * projection of every shard (one grouped GEMM launch), the attention core of
 * every (shard, sequence, head, 128-query tile) (one launch, flash-style on the
 * tensor cores: scores and P V in tensor memory, online softmax, no score matrix
 * in global memory), the output projection of every shard into its partial
 * buffer (one launch), and the shard-sum of the chunk -- on the library's
 * reduction stream with DOMINO_SCHEDULE_STREAMS, so it overlaps chunk k+1;
 * DOMINO_SCHEDULE_FUSED does the same for every chunk but the last, whose output
 * projection and shard-sum -- which no later chunk could hide -- are one
 * cooperative launch in which each 128x256 tile of Y is summed as soon as its P
 * partials are stored (the separate launches if the device cannot run it).
 * Weights, nn.Linear layout, per shard:
 *   Wqkv_shards[p]  [3 Hp dh, d]: shard p's query heads' rows, then its key
 *                   heads', then its value heads' (head h: rows h dh .. (h+1) dh)
 *   Wo_shards[p]    Wo_p^T [d, Hp dh]
 * Supported: dh = 128, S a multiple of 128, P | H, mu | B, d % 8 == 0; any
 * schedule (FUSED: mu <= 8).  Other shapes: DOMINO_ERR_UNSUPPORTED
 * (ALIGNMENT for d).  Softmax in fp32; Q, K, V, P and O rounded to bf16. */
typedef struct domino_attn_desc {
  int64_t B;              /* sequences, >= 0                                     */
  int64_t S;              /* tokens per sequence, multiple of 128                */
  int64_t d;              /* model width, multiple of 8                          */
  int32_t H;              /* heads, P | H                                        */
  int32_t dh;             /* head width: 128                                     */
  int32_t P;              /* shards, 1..DOMINO_MAX_SHARDS                        */
  int32_t mu;             /* chunks of whole sequences, mu | B, <= DOMINO_MAX_PIECES */
  int32_t partial_dtype;  /* domino_partial_dtype_t                              */
  int32_t schedule;       /* domino_schedule_t                                   */
  uint32_t flags;         /* DOMINO_FLAG_KERNEL_TIMES, DOMINO_FLAG_ONE_CTA       */
  uint32_t reserved;      /* must be 0                                           */
  uint64_t timeout_ns;    /* bound on each device-side wait; 0 = 2 seconds       */
} domino_attn_desc_t;

/* Workspace bytes of domino_attn_fwd (0 for an invalid descriptor): a 256-byte
 * header (device status at bytes 0-15; with DOMINO_SCHEDULE_FUSED, the last
 * chunk k's timeline -- 3 words as in domino_read_timeline -- at byte 64 + 24 k), the
 * counters of one fused output-projection launch, Q|K|V per shard
 * [P][B S][3 Hp dh] bf16, the attention output per shard [P][B S][Hp dh] bf16,
 * the partials [P][B S][d]. */
DOMINO_API size_t domino_attn_workspace_size(const domino_attn_desc_t* desc);

/* Forward pass: X [B S, d] -> Y [B S, d] bf16.  B == 0 returns DOMINO_OK having
 * touched nothing.  Kernel kinds in the timing log: GEMM1 (projection), ATTN
 * (attention core), GEMM2 (output projection), SHARD_SUM. */
DOMINO_API domino_status_t domino_attn_fwd(const domino_attn_desc_t* desc, const void* X,
                                           const void* const* Wqkv_shards, const void* const* Wo_shards, void* Y,
                                           void* workspace, size_t workspace_bytes, void* stream);

/* Strand interleaving: the forward of one micro-batch (strand a) and the
 * backward of another (strand b) of the same layer in one call, their launches
 * interleaved so that the shard-sums of each strand run beside the other
 * strand's GEMMs (the DHelix review page, "Hiding Communication Cost in
 * Distributed LLM Training via Micro-batch Co-execution": two strands co-run so
 * that one strand's communication hides under the other's computation).
 * Order on `stream`: strand b's dH over all M; then for k = 0..mu-1 strand a's
 * chunk k (GEMM1, GEMM2 per slice) and strand b's chunk k (dX partials per
 * slice); then strand b's weight gradients.  Every shard-sum goes to the
 * reduction stream after an event behind its GEMM (schedule STREAMS) or runs in
 * order (SERIAL); DOMINO_SCHEDULE_FUSED is rejected with
 * DOMINO_ERR_UNSUPPORTED.  Results are bit-identical to domino_mlp_fwd(strand a)
 * and domino_mlp_bwd(strand b) with the same descriptor.
 * Arguments as for those two calls: A_shards/B_shards shared; Xa -> Ya (and
 * saved_a, may be NULL); Xb, dYb, saved_b (what the forward of strand b saved)
 * -> dXb, dA_shards, dB_shards.  workspace: domino_mlp_interleaved_workspace_size()
 * bytes; device errors are reported in its first header (read it with
 * domino_query_device_status). */
DOMINO_API size_t domino_mlp_interleaved_workspace_size(const domino_mlp_desc_t* desc);
DOMINO_API domino_status_t domino_mlp_fwd_bwd_interleaved(const domino_mlp_desc_t* desc, const void* const* A_shards,
                                                          const void* const* B_shards, const void* Xa, void* Ya,
                                                          void* saved_a, const void* Xb, const void* dYb,
                                                          const void* saved_b, void* dXb, void* const* dA_shards,
                                                          void* const* dB_shards, void* workspace,
                                                          size_t workspace_bytes, void* stream);

/* Schedule selection.  The FiCCO page ("Design Space Exploration of DMA based
 * Finer-Grain Compute Communication Overlap", Abstract) picks a decomposition
 * for each operator from its sizes with heuristics, because finer pieces cost
 * GEMM efficiency; this entry point does that for the number of row chunks mu
 * and the schedule.  The rule (host arithmetic only):
 *   - schedule: DOMINO_SCHEDULE_FUSED when the fused cooperative forward can be
 *     launched, else DOMINO_SCHEDULE_STREAMS;
 *   - candidates: mu in {1, 2, 4, ...} with mu | M and mu * out_slices <=
 *     DOMINO_MAX_PIECES; a candidate "fills" the GPU when one chunk's GEMM1 has
 *     at least one paired 256 x 256 tile per 2-CTA cluster (num_sms / 2);
 *   - mu = the smallest filling candidate whose chunk of hidden activations,
 *     (M / mu) * F * 2 bytes over all shards, fits in 9/10 of the L2 (GEMM2 then
 *     reads H from L2); if none fits, the largest filling candidate; if none
 *     fills, mu = 1.
 * problem: M, d, F, P, out_slices, act, partial_dtype as for domino_mlp_fwd (mu,
 * schedule and flags are ignored).  hw: hardware figures; NULL, or a field <= 0
 * (fused_available < 0), means "ask the current CUDA device".  out: the choice.
 * Errors: DOMINO_ERR_INVALID_ARG / UNSUPPORTED / ALIGNMENT for a problem
 * domino_mlp_fwd would reject (with mu = 1), DOMINO_ERR_CUDA when a device query
 * fails.  Launches nothing and allocates nothing. */
typedef struct domino_plan_hw {
  int32_t num_sms;          /* streaming multiprocessors                            */
  int32_t fused_available;  /* 1 / 0: the fused forward can / cannot be launched    */
  int64_t l2_bytes;         /* L2 cache size in bytes                               */
} domino_plan_hw_t;

typedef enum domino_plan_reason {
  DOMINO_PLAN_FITS_L2 = 0,        /* smallest filling mu whose chunk of H fits the budget */
  DOMINO_PLAN_LARGEST_FILLING = 1,/* no filling mu fits: the largest filling one          */
  DOMINO_PLAN_SMALL = 2           /* no mu fills the GPU: mu = 1                          */
} domino_plan_reason_t;

typedef struct domino_plan {
  int32_t mu;                  /* chosen row chunks                                  */
  int32_t schedule;            /* chosen domino_schedule_t                           */
  int32_t reason;              /* domino_plan_reason_t                               */
  int32_t gemm1_tiles_per_chunk; /* paired GEMM1 tiles of one chunk at the chosen mu */
  int64_t chunk_h_bytes;       /* (M / mu) * F * 2 at the chosen mu                  */
  int64_t l2_budget_bytes;     /* 9/10 of the L2 it was compared with                */
} domino_plan_t;

DOMINO_API domino_status_t domino_mlp_plan(const domino_mlp_desc_t* problem, const domino_plan_hw_t* hw,
                                           domino_plan_t* out);

/* The same selection for the attention block (domino_attn_fwd), whose chunks
 * are mu groups of B / mu whole sequences:
 *   - schedule: always DOMINO_SCHEDULE_STREAMS (its output projection writes
 *     the partials at close to the memory's rate, so a shard-sum folded into
 *     that launch contends with it rather than hiding behind it);
 *   - candidates: mu in {1, 2, 4, ...} with mu | B and mu <= DOMINO_MAX_PIECES;
 *     a candidate fills the GPU when one chunk's Q|K|V projection has at least
 *     one paired 256 x 256 tile per 2-CTA cluster;
 *   - mu = the smallest filling candidate whose chunk of Q|K|V, (B / mu) S 3 H
 *     dh 2 bytes, fits in 9/10 of the L2; else the largest filling candidate;
 *     else mu = 1.  (The Q|K|V size stands in for how much work each chunk's
 *     launches get against the shard-sum that chunking hides; on the GPT- and
 *     Llama-style blocks it picks the fastest mu of 1, 2 and 4.)
 * problem: as for domino_attn_fwd (mu, schedule and flags are ignored).  hw: as
 * for domino_mlp_plan (fused_available is not consulted).  out: the choice,
 * with gemm1_tiles_per_chunk = the projection's paired tiles of one chunk and
 * chunk_h_bytes = one chunk's Q|K|V bytes.  Errors: as domino_attn_fwd would
 * reject the problem with mu = 1, or DOMINO_ERR_CUDA when a device query fails.
 * Launches nothing and allocates nothing. */
DOMINO_API domino_status_t domino_attn_plan(const domino_attn_desc_t* problem, const domino_plan_hw_t* hw,
                                            domino_plan_t* out);

/* Tensor-core rate probe: the dense bf16 throughput of this GPU's tcgen05 MMAs
 * on their own, the ceiling the GEMM main loops approach.  Each 2-CTA cluster
 * (one CTA per SM) issues `mmas_per_cluster` back-to-back paired MMAs of
 * 256 x 256 x 16 (bf16 operands already in shared memory, fp32 accumulators in
 * tensor memory); there are no loads, stores or epilogue.  The kernel also
 * counts SM cycles and nanoseconds around the MMA stream of cluster 0, so the
 * rate per SM per clock follows without an outside clock reading.
 * mmas_per_cluster: 1 .. DOMINO_TENSOR_PEAK_MAX_MMAS.  clusters: 2-CTA
 * clusters to launch, <= 0 for the most that can be co-resident (the paired
 * GEMMs' grid); more than that is rejected with DOMINO_ERR_UNSUPPORTED.
 * workspace: >= DOMINO_TENSOR_PEAK_WS_BYTES bytes of device memory, 256-byte
 * aligned, its status words zero (as after domino_query_device_status).
 * timeout_ns: bound on the wait for the MMAs to finish (0: 5 s).  stream: the
 * launch stream; the call synchronises on it and returns the measurement in
 * *out.  Errors: DOMINO_ERR_INVALID_ARG / ALIGNMENT for bad arguments (before
 * any CUDA call), DOMINO_ERR_CUDA, DOMINO_ERR_TIMEOUT when the wait gave up. */
#define DOMINO_TENSOR_PEAK_MAX_MMAS (1 << 22)
#define DOMINO_TENSOR_PEAK_WS_BYTES 256

typedef struct domino_tensor_peak {
  double tflops;            /* flops / kernel duration, in TFLOP/s                     */
  double flops;             /* 2 * 256 * 256 * 16 * mmas_per_cluster * clusters        */
  double ms;                /* kernel duration (CUDA events on `stream`)               */
  double sm_mhz;            /* SM clock during cluster 0's MMA stream (cycles / ns)    */
  double flops_per_clk_sm;  /* cluster 0's flops / its cycles / 2 SMs                  */
  int32_t clusters;         /* 2-CTA clusters launched                                 */
  int32_t num_sms;          /* SMs of the device                                       */
} domino_tensor_peak_t;

DOMINO_API domino_status_t domino_tensor_peak(int64_t mmas_per_cluster, int32_t clusters, void* workspace,
                                              size_t workspace_bytes, uint64_t timeout_ns, void* stream,
                                              domino_tensor_peak_t* out);

#ifdef __cplusplus
}
#endif

#endif /* DOMINO_H */
