/*
 * libkda -- Kimi Delta Attention (KDA) chunked forward pass for one NVIDIA
 * GB300 (sm_103a).  Plain C ABI: device pointers, sizes, a CUDA stream.
 *
 * The operation (per sequence n and head h, state S in R^{V x K}, row =
 * value index, column = key index):
 *     a_t = gate(g_t + dt_bias[h])        per key channel, natural log, <= 0
 *     S   = S * Diag(exp(a_t))
 *     S   = S + beta_t (v_t - S k_t) k_t^T,   beta_t = sigmoid(beta logit)
 *     o_t = scale * S q_t
 * with q, k optionally L2-normalised per token (q / sqrt(|q|^2 + 1e-6)).
 * Gate forms (flash-linear-attention skills, fla-kda SKILL.md, "Gate
 * contracts"; fla-kda skill page):
 *     safe   : a = lower_bound * sigmoid(exp(A_log[h]) * z), -5 <= lb < 0,
 *              A_log may be NULL (multiplier 1)
 *     unsafe : a = -exp(A_log[h]) * softplus(z), A_log required
 * Argument table and constraints follow the flashkda.fwd table of the
 * FlashKDA page ("Core Kernel API flashkda.fwd"): K == V == 128, bf16 q/k/v/g
 * and beta logits, fp32 A_log [H] and dt_bias [H, K], states [N, H, V, K] in
 * fp32 or bf16 (same dtype when both given), int64 cu_seqlens [N+1] with
 * B == 1 ("Variable-Length (Packed) Batching").  Chaining final_state into
 * the next call's initial_state continues a stream ("Stateful Inference").
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (every violation is reported before any launch) ---- */
#define KDA_OK 0
#define KDA_ERR_NULL_ARG 1        /* a required pointer is NULL */
#define KDA_ERR_HEAD_DIM 2        /* K or V is not 128 */
#define KDA_ERR_SHAPE 3           /* negative size, or N inconsistent with B */
#define KDA_ERR_GATE_FLAGS 4      /* not exactly one of KDA_GATE_SAFE / _UNSAFE / _LOGSPACE,
                                     or an unknown flag bit */
#define KDA_ERR_LOWER_BOUND 5     /* safe gate with lower_bound outside [-5, 0) */
#define KDA_ERR_A_LOG_REQUIRED 6  /* unsafe gate with A_log == NULL */
#define KDA_ERR_STATE_DTYPE 7     /* state_dtype not KDA_DTYPE_F32 / KDA_DTYPE_BF16 */
#define KDA_ERR_VARLEN_BATCH 8    /* cu_seqlens given with B != 1 */
#define KDA_ERR_ALIGNMENT 9       /* a tensor pointer is not 16-byte aligned */
#define KDA_ERR_WORKSPACE 10      /* workspace NULL, misaligned or too small */
#define KDA_ERR_LAUNCH 11         /* a CUDA launch failed (cudaGetLastError) */
#define KDA_ERR_NOALLOC_LIMIT 12  /* kda_fwd_noalloc: problem needs more scratch than built in */
#define KDA_ERR_DEVICE_TIMEOUT 13 /* (device status) a kernel gave up waiting for its operands */
#define KDA_ERR_BAD_SEQLENS 14    /* (device status) cu_seqlens values inconsistent (see kda_fwd_args) */

/* ---- flags ---- */
#define KDA_GATE_SAFE 0x1u   /* lower_bound * sigmoid(exp(A_log) * (g + dt_bias)) */
#define KDA_GATE_UNSAFE 0x2u /* -exp(A_log) * softplus(g + dt_bias) */
#define KDA_QK_L2NORM 0x4u   /* L2-normalise q and k per token inside the kernel */
/* g already holds the log-space decay a_t (natural log, <= 0 expected; values
 * are not checked): chunk_kda without the in-kernel gate (fla-kda SKILL.md,
 * "Gate contracts").  A_log, dt_bias and lower_bound are not used. */
#define KDA_GATE_LOGSPACE 0x8u
/* beta already holds beta in [0, 1] (no sigmoid applied): the beta-activation
 * mode named in the same page's correctness checklist. */
#define KDA_BETA_PROB 0x10u
/* g is fp32 [B, T, H, 128] instead of bf16, with any gate form; meant for the
 * caller-gated mode, whose log decays the pages pass in fp32 (fla-kda SKILL.md,
 * "Gate contracts": chunk_kda with use_gate_in_kernel=False). */
#define KDA_G_FP32 0x20u

/* ---- state dtypes ---- */
#define KDA_DTYPE_F32 0
#define KDA_DTYPE_BF16 1

/*
 * Arguments of one forward call.  All tensors are dense, row-major and live
 * in device memory owned by the caller; the library never allocates device
 * memory and keeps no pointer after the call returns (work is asynchronous
 * on the given stream, so buffers must stay valid until it completes).
 *
 *  q, k, g : bf16 [B, T, H, 128]      v, out : bf16 [B, T, H, 128]
 *            (g fp32 with KDA_G_FP32)
 *  beta    : bf16 [B, T, H]  (logits, sigmoid applied inside; with KDA_BETA_PROB
 *            beta itself)
 *  g       : raw gate logits, or with KDA_GATE_LOGSPACE the log decays a_t
 *  out     : written completely for every token of every sequence
 *  q, k, v, g, beta, out may be NULL when B * T == 0 (no tokens: only the
 *            final state, equal to the initial state, is written)
 *  A_log   : fp32 [H]       (NULL only with KDA_GATE_SAFE -> multiplier 1)
 *  dt_bias : fp32 [H, 128]  (NULL -> 0)
 *  initial_state, final_state : [N, H, 128(V), 128(K)] in state_dtype, or
 *            NULL (initial NULL -> zero state; final NULL -> not written).
 *            bf16 final states are rounded to nearest-even from fp32.
 *  cu_seqlens : int64 [N+1] device array or NULL.  With it B must be 1, T is
 *            the packed token total, cu[0] = 0, non-decreasing, cu[N] = T.
 *            The values are not read on the host; the kernels check them and
 *            any violation sets the device status to KDA_ERR_BAD_SEQLENS.
 *            Then kda_fwd (and kda_fwd_noalloc) process no sequence at all
 *            (out untouched, every final state = its initial state), since
 *            overlapping sequences could need more workspace than was sized;
 *            kda_fwd_recurrent skips only the sequences whose bounds leave
 *            [0, T] or decrease.
 *            Without it N must equal B and sequence n is batch row n.
 *  All sizes are int64; tensor pointers must be 16-byte aligned.
 */
typedef struct kda_fwd_args {
  const void *q, *k, *v, *g, *beta;
  float scale;
  void *out;
  const float *A_log;
  const float *dt_bias;
  float lower_bound;
  const void *initial_state;
  void *final_state;
  int32_t state_dtype;
  const int64_t *cu_seqlens;
  int64_t B, T, H, N;
  int64_t K, V;
  uint32_t flags;
} kda_fwd_args;

/*
 * Device scratch (bytes) that kda_fwd needs for these arguments: per-chunk
 * intermediates of the WY form (W, U, gated queries, end-decayed keys, the
 * intra-chunk read-out matrix and the chunk decay) plus the chunk index of
 * packed sequences.  For a dense call with very few sequence-heads (N*H at
 * most 7 on 152 SMs: all 2G - 1 runs of four CTAs each fit on the GPU at once
 * for some G >= 3) and at least 64 chunks per segment, kda_fwd cuts the state
 * stage's chain into G segments (the sequence split): the fp32 transition
 * buffers add (3G - 3) * N*H*64 KiB.  Depends on sizes, on whether cu_seqlens
 * is given and on the current device; size the workspace on the device that
 * runs the call.
 * Returns 0 for argument sets that kda_fwd would reject.
 */
size_t kda_fwd_workspace_bytes(const kda_fwd_args *args);

/*
 * Enqueue the forward pass on `stream` (a cudaStream_t; NULL = legacy default
 * stream).  `workspace` is caller-owned device memory of at least
 * kda_fwd_workspace_bytes(args) bytes, 256-byte aligned; its contents need no
 * initialisation and are garbage afterwards.  Calls that share a workspace
 * must be ordered on the device.  Returns KDA_OK or an error code; on an
 * argument error nothing is launched and nothing is written; KDA_ERR_LAUNCH
 * (a failed launch, event or tensor-map set-up) may follow launches already
 * made by the same call.  The call only enqueues work, so it may be captured
 * into a CUDA graph: the tensor maps of the inputs travel with the launch as
 * parameters (tested bit-identical to eager calls).  Every kernel of a call
 * runs on `stream`, one after another.  The first call on a device, which sets
 * up kernel attributes, is best made outside a capture.  The per-device set-up
 * is kept for the life of the process: do not use the library across
 * cudaDeviceReset.
 */
int kda_fwd(const kda_fwd_args *args, void *workspace, size_t workspace_bytes, void *stream);

/*
 * kda_fwd, additionally recording three caller-created CUDA events
 * (cudaEvent_t, each may be NULL) on `stream`: events[0] before the first
 * launch, events[1] after the intra-chunk stage (chunk index + per-chunk WY
 * quantities), events[2] after the recurrent stage.  For measurement only;
 * the computation is identical to kda_fwd.
 */
int kda_fwd_profiled(const kda_fwd_args *args, void *workspace, size_t workspace_bytes,
                     void *stream, void *const events[3]);

/*
 * The same forward pass token by token: the fused_recurrent_kda entry point of
 * the fla KDA code (fla-kda SKILL.md names chunk_kda and fused_recurrent_kda as
 * its public entry points).  For decoding, i.e. one or a few tokens per
 * sequence: each (sequence, head) streams its state from initial_state through
 * registers to final_state once, with no workspace (none is taken).
 * Arguments, flags, layouts and error codes as kda_fwd; final_state may be the
 * same buffer as initial_state (in-place state update).  Asynchronous on
 * `stream` (cudaStream_t or NULL); returns KDA_ERR_LAUNCH if the launch fails.
 * Cost grows with the tokens per sequence (a serial loop): prefer kda_fwd for
 * prefill.
 */
int kda_fwd_recurrent(const kda_fwd_args *args, void *stream);

/* Number of kernel launches kda_fwd makes for these arguments on the current
 * device (0 if none or if the arguments are invalid): 2 or 3 for one pass
 * (3 with cu_seqlens: the chunk index scan), 4 for the sequence split (see
 * kda_fwd_workspace_bytes). */
int kda_fwd_launches(const kda_fwd_args *args);

/*
 * kda_fwd without a caller-provided workspace.  No counterpart in the pages:
 * this exists for callers that cannot allocate device memory when they run
 * the forward pass (host callbacks or plugins without an allocator, code
 * that must not touch the owning framework's caching allocator, fixed
 * memory budgets that forbid runtime cudaMalloc).  The workspace comes from a
 * buffer of KDA_NOALLOC_SCRATCH_BYTES compiled into the library, held on every
 * GPU that loads the library until the process exits.  The call itself
 * allocates nothing.
 *
 *  - Limit: problems whose kda_fwd_workspace_bytes(args) exceeds
 *    KDA_NOALLOC_SCRATCH_BYTES are rejected with KDA_ERR_NOALLOC_LIMIT before
 *    anything runs (32 MiB holds 451 (64-token chunk, head) slots, e.g.
 *    T * H <= 28,864 token-heads for dense inputs).
 *  - Set-up: the first call on a device looks up the buffer's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address is kept for the life of the
 *    process: do not use the library across cudaDeviceReset.
 *  - Sharing: every call on a device uses the same buffer, which keeps the
 *    previous call's contents.  Nothing in it needs to start at zero, but
 *    calls that can overlap on the GPU (different streams, no ordering) race
 *    on it: order them.
 * Other arguments, ownership and errors are as for kda_fwd.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int kda_fwd_noalloc(const kda_fwd_args *args, void *stream);

/*
 * The forward pass end to end on HOST buffers: copy the inputs to the device,
 * run the same two stages as kda_fwd, copy the output (and final state) back.
 * No counterpart in the pages, whose entry point takes device tensors; this
 * is the call for callers whose data sit in host memory.  The transfers of one
 * call are pipelined with its kernels: dense inputs are cut along the token
 * axis into at most 64 pieces of whole 64-token chunks (about 32 MiB of
 * inputs each; the recurrent state passes from piece to piece in fp32 inside
 * device_buffer, so the result is that of kda_fwd on the same inputs), packed
 * inputs into groups of whole sequences; the copy in of piece p + 1, the
 * kernels of piece p and the copy back of piece p - 1 overlap.
 *
 *  - Arguments: as kda_fwd, except that every pointer in `args` (q, k, v, g,
 *    beta, out, A_log, dt_bias, initial_state, final_state, cu_seqlens) is
 *    host memory.  Page-locked memory (cudaHostAlloc / cudaHostRegister) is
 *    needed for the copies to be asynchronous and overlap; pageable memory
 *    gives the same results with the copies serialised.  cu_seqlens is read
 *    on the host and checked: cu[0] == 0, non-decreasing, cu[N] == T, else
 *    KDA_ERR_SHAPE.
 *  - device_buffer: caller-owned device memory of at least
 *    kda_fwd_host_device_bytes(args) bytes, 256-byte aligned, holding the
 *    device copies, the output, the carried state and the workspace; garbage
 *    afterwards.  Calls sharing it must be ordered.
 *  - Ordering: the call starts after the work already on `stream`
 *    (cudaStream_t or NULL) and `stream` waits for its last copy back, so
 *    `out` and `final_state` hold the results once `stream` has reached that
 *    point (e.g. after cudaStreamSynchronize(stream)).  The host buffers
 *    must stay valid until then.
 *  - Resources: on first use per device the library creates two non-blocking
 *    copy streams (one per direction) and 130 events, kept until the process
 *    exits; concurrent
 *    calls on one device enqueue one after another (a mutex).
 *  - Errors: as kda_fwd (checked before anything is enqueued); KDA_ERR_WORKSPACE
 *    for a missing, misaligned or short device_buffer; KDA_ERR_LAUNCH if a copy
 *    or launch fails to enqueue.
 */
size_t kda_fwd_host_device_bytes(const kda_fwd_args *args);
int kda_fwd_host(const kda_fwd_args *args, void *device_buffer, size_t device_bytes, void *stream);

/*
 * Backward pass: the gradients of L = <out, dout> + <final_state, dfinal_state>
 * with respect to every input of the forward call (the "chunk_bwd" stage of the
 * fla-kda code map, SKILL.md "Code map"; the pages' FlashKDA entry point itself
 * is forward-only).  Computed in fp32 from the bf16 inputs in chunked (WY / UT)
 * form over 64-token chunks: the chunk quantities of the forward are recomputed
 * per chunk, a forward pass over the chunks stores the state before each chunk,
 * a reverse pass stores the state gradient after each chunk, and every chunk's
 * input gradients are then formed independently (workspace).  All gradients are
 * fp32.
 *
 *  fwd            : the forward call's arguments (out and final_state unused;
 *                   every layout, flag and check as kda_fwd)
 *  dout           : bf16 [B, T, H, 128], dL/d out
 *  dfinal_state   : fp32 [N, H, 128, 128] or NULL (no final-state term)
 *  dq, dk, dv, dg : fp32 [B, T, H, 128], written completely (dg with respect to
 *                   the raw g: logits, or the log decays with KDA_GATE_LOGSPACE)
 *  dbeta          : fp32 [B, T, H] with respect to the raw beta (logits, or beta
 *                   itself with KDA_BETA_PROB)
 *  dA_log         : fp32 [H] or NULL; not written with KDA_GATE_LOGSPACE
 *  ddt_bias       : fp32 [H, 128] or NULL; not written with KDA_GATE_LOGSPACE
 *  dinitial_state : fp32 [N, H, 128, 128] or NULL
 * dA_log and ddt_bias are sums over tokens taken per chunk and then over the
 * chunks in order; every gradient is deterministic.  dA_log reads 0 for the safe
 * gate without A_log.  With cu_seqlens whose bounds are inconsistent, no chunk
 * is processed (zero token gradients, dinitial_state = dfinal_state) and the
 * stream's status word reads KDA_ERR_BAD_SEQLENS.
 */
typedef struct kda_bwd_args {
  kda_fwd_args fwd;
  const void *dout;
  const float *dfinal_state;
  float *dq, *dk, *dv, *dg;
  float *dbeta;
  float *dA_log;
  float *ddt_bias;
  float *dinitial_state;
} kda_bwd_args;

/* Device scratch for kda_bwd: one 559,872-byte item per (chunk slot, head),
 * holding the chunk's recomputed quantities, the state before the chunk and the
 * state gradient after it (fp32), for B * ceil(T / 64) chunk slots, or
 * ceil(T / 64) + N with cu_seqlens after a 256-byte-rounded header of
 * (N + 1) int64 chunk offsets; 0 if the forward arguments are invalid. */
size_t kda_bwd_workspace_bytes(const kda_bwd_args *args);

/* Enqueue the backward pass on `stream` (every launch and memset on that
 * stream, so a call can be captured into a CUDA graph once the library has
 * been used on the device).  Workspace as for kda_fwd (caller
 * owned, 256-byte aligned, at least kda_bwd_workspace_bytes).  Returns KDA_OK
 * or an error code before any launch (the kda_fwd checks; dout and the token
 * gradients must be given when B * T > 0; 16-byte alignment of the float
 * tensors), or KDA_ERR_LAUNCH. */
int kda_bwd(const kda_bwd_args *args, void *workspace, size_t workspace_bytes, void *stream);

/*
 * kda_bwd, additionally recording four caller-created CUDA events
 * (cudaEvent_t, each may be NULL) on `stream`: events[0] before the first
 * operation, events[1] after the recompute and forward state pass launches,
 * events[2] after the reverse state pass, events[3] after the chunk gradient
 * launches.  For measurement only; the computation is identical to kda_bwd.
 */
int kda_bwd_profiled(const kda_bwd_args *args, void *workspace, size_t workspace_bytes,
                     void *stream, void *const events[4]);

/*
 * Device-side status of the forward calls enqueued on `stream` (a cudaStream_t;
 * NULL = legacy default stream), the kda_get_status(cudaStream_t) of the
 * boundary: KDA_OK, KDA_ERR_DEVICE_TIMEOUT if a CTA of such a call gave up
 * waiting (bounded wait, about a second of SM cycles) for its asynchronous
 * operand copies and returned without finishing its work, or
 * KDA_ERR_BAD_SEQLENS if a call's cu_seqlens values were inconsistent.
 *
 *  - One status word per (device, stream): every kernel of a call reports into
 *    the word of the stream the call was enqueued on, so calls on different
 *    streams never see, overwrite or clear each other's codes.  The words come
 *    from a table of 1023 slots built into the library; a stream takes a slot
 *    on its first call and keeps it, and the streams beyond the 1023rd
 *    distinct handle on a device share one further slot.  Two host threads using the per-thread
 *    default stream handle (cudaStreamPerThread) share a word.
 *  - Sticky until read: the call synchronises `stream`, returns its word as it
 *    stands after all work enqueued on it so far (the last code set wins) and
 *    clears it.  Returns -1 if the read fails or `stream` is being captured
 *    into a CUDA graph (a captured call reports into the word of the stream it
 *    was captured on, whatever stream replays the graph).
 */
int kda_get_status(void *stream);

/*
 * Self-test of the failure path (no counterpart in the pages): launches one
 * block on `stream` that waits, with the same bounded mbarrier wait the state
 * kernel uses, on a barrier phase that nothing completes; after `cycles` SM
 * cycles (1 .. 2^31) it gives up, sets the device status word to
 * KDA_ERR_DEVICE_TIMEOUT in the status word of `stream` exactly as a real
 * timeout does, and returns.  The context stays usable.  Returns KDA_OK, KDA_ERR_SHAPE for a cycle count out
 * of range, or KDA_ERR_LAUNCH.
 */
int kda_selftest_wait_timeout(long long cycles, void *stream);

/* Human-readable text of a status code (static storage). */
const char *kda_error_string(int code);

/* Library version, e.g. 100 for 0.1.0. */
int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
