/*
 * lizard_attn.h -- C ABI of the Lizard hybrid attention operator on B300.
 *
 *     y_t = yg_t + alpha * ya_t
 *
 * "Lizard: An Efficient Linearization Framework for Large Language Models"
 * (gist.science/de), section 2 "Kernkomponenten der Architektur":
 *   item 1 "Gated Linear Attention (GLA) mit lernbarem Gate" -- the gate
 *          branch yg, a recurrence over a d_k x d_v state per head whose
 *          rows decay by sigmoid(g_t), the learnable data-dependent gate:
 *              S_t = diag(sigmoid(g_t)) S_{t-1} + k_t^T v_t ,   yg_t = q_t S_t
 *   item 2 "Anchor Window Attention" -- the anchor branch ya, softmax
 *          attention over the w most recent tokens (the current one
 *          included) plus m learnable meta-memory keys that act as attention
 *          sinks: they enter the softmax normaliser and carry value zero:
 *              ya_t = sum_s e^{q_t.k_s} v_s / (sum_s e^{q_t.k_s} + sum_j e^{q_t.mu_j})
 *   item 3 "Hybride Ausgabe" -- the combine y = yg + alpha * ya.
 * The same operator is described in gist.science/it section 2 "Architettura
 * Ibrida" and gist.science/pt section 2A "Arquitetura Hibrida".  No scale is
 * applied inside the softmax: callers pre-scale q (and k) as they wish.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library never allocates, frees or retains them past the call.
 *   - Tensors are dense, row-major, head-major: [B][H][L][d] with the last
 *     dimension contiguous.  Every pointer must be 16-byte aligned (the
 *     state's pos: 8-byte, see lizard_state).
 *   - Element type of q, k, v, g, meta keys, y and the ring buffer is the
 *     call's lizard_dtype (fp32 or bf16).  The recurrent state S is always
 *     fp32 and all accumulation is fp32.
 *   - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *     stream); a call returns once the work is enqueued.
 *   - Arguments are validated on the host before anything is launched; a
 *     rejected call launches nothing and touches no buffer.
 *   - Errors are returned as lizard_status.  Nothing aborts, throws or traps.
 *   - Scratch: a call that needs temporary device memory (a prompt run as
 *     sequence segments, the backward pass) takes it stream-ordered on
 *     `stream` from a memory pool the library owns (one per device) and
 *     frees it there.  Freed memory stays reserved in that pool for the
 *     library's later calls -- at most the largest scratch of any one call
 *     so far, e.g. about 810 MB for the backward of B4 H32 L4096 d128 --
 *     until lizard_scratch_trim returns it or the process exits; failure to
 *     allocate is LIZARD_ERR_CUDA (a prefill then runs unsegmented instead).
 *   - Supported shapes: d_k == d_v in {64, 128, 256}; 1 <= w <= LIZARD_MAX_WINDOW;
 *     0 <= m <= LIZARD_MAX_META.  d = 256 runs the exact CUDA-core kernels
 *     (prefill, continued prefill, decode; its backward is not built: the
 *     backward and the no-allocation prefill take d in {64, 128}); a decode
 *     step at d = 256 in fp32 stages its ring and meta keys in shared
 *     memory and is UNSUPPORTED where they do not fit (w > 99 with 16 meta
 *     keys, w > 107 with none).  Anything else in range but not built is
 *     LIZARD_ERR_UNSUPPORTED; anything meaningless is LIZARD_ERR_INVALID_ARG.
 */
#ifndef LIZARD_ATTN_H
#define LIZARD_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define LIZARD_API __attribute__((visibility("default")))
#else
#define LIZARD_API
#endif

/* cudaStream_t without pulling in the CUDA headers (same type). */
struct CUstream_st;
typedef struct CUstream_st *lizard_stream_t;

#define LIZARD_MAX_WINDOW 128
#define LIZARD_MAX_META 16

typedef enum {
    LIZARD_OK = 0,
    LIZARD_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or dtype */
    LIZARD_ERR_UNSUPPORTED = 2,   /* valid request outside the built shapes    */
    LIZARD_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed       */
    LIZARD_ERR_TIMEOUT = 4        /* a bounded device-side wait gave up         */
} lizard_status;

typedef enum { LIZARD_F32 = 0, LIZARD_BF16 = 1 } lizard_dtype;

/*
 * Recurrent state of B sequences x H heads: what constant-memory decoding
 * keeps between tokens (gist.science/de section 2 item 1, last bullet).
 *   S       [B][H][dk][dv] fp32   gate-branch state, row i = key dim i
 *   ring_k  [B][H][w][dk]  dtype  keys of the last w tokens, token p in slot p % w
 *   ring_v  [B][H][w][dv]  dtype  values, same slots
 *   pos     [B] int64             tokens consumed so far by each sequence
 * All four are caller-owned device buffers: S, ring_k and ring_v 16-byte
 * aligned, pos 8-byte aligned.  The batch is the outermost dim of each, so
 * sequences b0 .. b1-1 of a state form a state of their own (S + b0 H dk dv,
 * ring_k + b0 H w dk, ring_v + b0 H w dv, pos + b0, B = b1 - b0).
 */
typedef struct {
    float *S;
    void *ring_k;
    void *ring_v;
    int64_t *pos;
    int B, H, dk, dv, w;
    lizard_dtype dtype;
} lizard_state;

/*
 * Variants of the operator (the teachers' model shapes; the pages print
 * neither, so both are design variants).  Passed to the *_v entry points;
 * NULL there, or the plain entry points, mean neither.
 *   alpha_h  [H] fp32 device array: the anchor weight of each head (the
 *            combine y = yg + alpha_h[h] ya of gist.science/de section 2
 *            item 3, per head); NULL: the call's alpha for every head.
 *            4-byte aligned.
 *   Hkv      key/value heads, 0 meaning H.  H % Hkv == 0: query head h
 *            reads key/value head h / (H / Hkv) of its batch row, so k and
 *            v (and, in the backward, dk and dv) are [B][Hkv][L][d] (decode:
 *            [B][Hkv][d]).  The gate logits, the meta keys and the state
 *            stay per query head (the state's ring keeps each query head's
 *            window keys and values).
 * An invalid variant (Hkv not dividing H, negative) is LIZARD_ERR_INVALID_ARG.
 */
typedef struct {
    const float *alpha_h;
    int Hkv;
} lizard_variant;

/*
 * lizard_state_init: the empty state -- S = 0, ring = 0, pos = 0 -- for all
 * B x H units.  Enqueued on `stream`.  Errors: INVALID_ARG for a null state
 * or buffer, bad sizes or misaligned buffers; CUDA if the launch fails.
 */
LIZARD_API lizard_status lizard_state_init(const lizard_state *st, lizard_stream_t stream);

/*
 * lizard_attn_prefill: the operator over a whole prompt of L tokens per
 * sequence, starting from the empty state (no earlier tokens).
 *   q, k, g  [B][H][L][dk]  dtype   queries, keys, gate logits (gamma = sigmoid(g))
 *   v        [B][H][L][dv]  dtype   values
 *   meta_k   [H][m][dk]     dtype   meta-memory keys (may be NULL when m == 0)
 *   alpha                           weight of the anchor branch
 *   y        [B][H][L][dv]  dtype   output (written; may not alias an input)
 *   st       nullable.  When given, its dims/dtype must match the call and
 *            the prefill WRITES the state that follows the prompt: S after
 *            token L-1, the last min(L, w) keys/values into the ring, and
 *            pos[b] = L.  Its previous contents are ignored.
 * L == 0 or B*H == 0 is a valid empty call (only the state is written);
 * with L == 0 the token pointers (q, k, v, g, y) may be NULL.
 */
LIZARD_API lizard_status lizard_attn_prefill(const void *q, const void *k, const void *v, const void *g,
                                  const void *meta_k, float alpha,
                                  int B, int H, int L, int dk, int dv, int w, int m,
                                  lizard_dtype dtype, void *y, const lizard_state *st,
                                  lizard_stream_t stream);

/* lizard_attn_prefill with a variant (see lizard_variant). */
LIZARD_API lizard_status lizard_attn_prefill_v(const void *q, const void *k, const void *v, const void *g,
                                    const void *meta_k, float alpha, int B, int H, int L, int dk, int dv,
                                    int w, int m, lizard_dtype dtype, void *y, const lizard_state *st,
                                    const lizard_variant *var, lizard_stream_t stream);

/*
 * lizard_attn_prefill_continue: L more tokens of each of st->B sequences
 * and st->H heads, continuing from `st` (read, then updated in place) --
 * chunked prefill of a long prompt, or a prompt that follows decoded tokens.
 * The recurrence simply carries on (gist.science/de section 2 item 1: S
 * holds the whole past of the gate branch; item 2: the anchor window of a
 * token spans the w most recent tokens, earlier calls' included, which the
 * ring keeps).  For sequence b with p = pos[b] tokens consumed so far, the
 * new tokens are positions p .. p + L - 1:
 *   y_t = q_t S_t + alpha * ya_t,  S_t = diag(sigmoid(g_t)) S_{t-1} + k_t^T v_t
 * from S_{p-1} = st->S, and the window of position t is positions
 * max(0, t - w + 1) .. t, those before p read from ring slot (position % w).
 * Afterwards S is the state after position p + L - 1, ring slot
 * (position % w) holds the last min(L, w) new keys and values (older slots
 * are kept), and pos[b] = p + L.  A prefill of L1 tokens followed by a
 * continuation of L2 gives the y and state of one prefill of L1 + L2 tokens
 * (up to rounding); the sequences of one call may be at different p.
 *   q, k, g  [B][H][L][dk]  st->dtype;  v [B][H][L][dv];  meta_k [H][m][dk]
 *   y        [B][H][L][dv]  st->dtype   output (may not alias an input)
 * Shapes and paths as lizard_attn_prefill (dk == dv from st; H <= 16384).
 * Like lizard_attn_prefill it allocates only when a prompt runs as sequence
 * segments (few batch x head units, long L): then the segments' start
 * states and a copy of the first segment's S and window history live in
 * the library's scratch (see the conventions above).
 * L == 0 or B == 0 is a no-op.  Precondition: 0 <= pos[b] < 2^40 (a state
 * written by this library always is).  While the call runs, pos[b] carries
 * an arrival count in its high bits; it holds p + L again once the work is
 * done.  A pos outside that range is reported (lizard_check_device_status);
 * that sequence's y, S, ring and pos are then undefined, but every access
 * stays inside the caller's buffers.
 */
LIZARD_API lizard_status lizard_attn_prefill_continue(const void *q, const void *k, const void *v, const void *g,
                                           const void *meta_k, float alpha, int L, int m, void *y,
                                           const lizard_state *st, lizard_stream_t stream);

/* lizard_attn_prefill_continue with a variant (see lizard_variant). */
LIZARD_API lizard_status lizard_attn_prefill_continue_v(const void *q, const void *k, const void *v, const void *g,
                                             const void *meta_k, float alpha, int L, int m, void *y,
                                             const lizard_state *st, const lizard_variant *var,
                                             lizard_stream_t stream);

/*
 * lizard_attn_prefill_noalloc: lizard_attn_prefill for callers that must not
 * allocate device memory during a call -- for example a serving runtime
 * that reserves all device memory up front for its own pool, code that must
 * not touch the driver's allocator while other work is being captured or
 * timed, or an embedding that forbids run-time allocation.  (The paper has
 * no counterpart; this entry point is about memory management only.)
 *
 * Same arguments and results as lizard_attn_prefill; it covers the
 * tensor-core path (bf16 with dk == dv in {64, 128}), LIZARD_ERR_UNSUPPORTED
 * otherwise.  When a prompt runs as sequence segments (few batch x head
 * units, long L) the segments' start states need scratch.  This variant
 * keeps it in a fixed device array of LIZARD_NOALLOC_SCRATCH_BYTES (16 MiB)
 * that every GPU loading the library holds until the process exits, and
 * calls no cudaMalloc, cudaFree or allocating library routine.  A problem
 * whose segment states would not fit (units x (segments - 1) x 66048 bytes)
 * is rejected with LIZARD_ERR_UNSUPPORTED before anything is launched.
 *   - The first call on each device (and the first after a reset of that
 *     device, which gives it a new context) looks up the array's device
 *     address (cudaGetSymbolAddress) with that device current; make that
 *     first call before any stream capture on that device.
 *   - Every call shares the one array and overwrites what it reads (nothing
 *     in it needs to start at zero), so calls whose work overlaps on the GPU
 *     -- on different streams, or from different host threads -- race and
 *     must be serialised by the caller.
 */
#define LIZARD_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
LIZARD_API lizard_status lizard_attn_prefill_noalloc(const void *q, const void *k, const void *v, const void *g,
                                          const void *meta_k, float alpha,
                                          int B, int H, int L, int dk, int dv, int w, int m,
                                          lizard_dtype dtype, void *y, const lizard_state *st,
                                          lizard_stream_t stream);

/*
 * lizard_scratch_trim: hands the scratch the library's pool holds on the
 * current device back to the driver, keeping at most `keep_bytes` reserved
 * for later calls.  Memory of calls still running on the GPU is not
 * returned: synchronise the streams of earlier calls first.  A device that
 * never needed scratch has no pool: LIZARD_OK, nothing done.
 * Not part of the paper's operator; memory management only.
 */
LIZARD_API lizard_status lizard_scratch_trim(size_t keep_bytes);

/* lizard_scratch_reserved: bytes the library's scratch pool holds on the
 * current device (0 without a pool); *bytes must be a host pointer. */
LIZARD_API lizard_status lizard_scratch_reserved(size_t *bytes);

/*
 * lizard_attn_backward: gradients of a scalar loss through the operator over
 * a prompt that starts from the empty state (training), given dy = dLoss/dy.
 * The gate (gist.science/de section 2 item 1, gamma = sigmoid(g)), the
 * meta-memory keys (item 2) and alpha (item 3) are trained along with the
 * inputs, so every one of them gets a gradient:
 *   q, k, g, v, meta_k, alpha, B..m, dtype   as lizard_attn_prefill
 *   dy       [B][H][L][dv]  dtype   upstream gradient
 *   dq, dk, dg [B][H][L][dk] dtype, dv [B][H][L][dv] dtype   written
 *   dmeta_k  [H][m][dk]     fp32    written (summed over the batch); may be
 *                                   NULL when m == 0
 *   dalpha   one fp32 value         written (summed over everything); 4-byte
 *                                   aligned
 * Gradients are computed in fp32 from the stored input bits (every gate
 * value is handled: all exponents the kernel takes are <= 0) and rounded
 * to dtype once.  Scratch (see the conventions above) per (batch, head)
 * unit: for bf16 with dk == 128 and w <= 65 (tensor cores) the bf16 state
 * and state gradient at every 64-token chunk boundary plus 4 (L dk + 2 L)
 * bytes, otherwise 4 (L dk + 2 L + m dk + 1) bytes.
 * L == 0 or B == 0 writes zero dmeta_k and dalpha and nothing else.
 */
LIZARD_API lizard_status lizard_attn_backward(const void *q, const void *k, const void *v, const void *g,
                                   const void *meta_k, float alpha, int B, int H, int L, int dk, int dv,
                                   int w, int m, lizard_dtype dtype, const void *dy, void *dq, void *dk_out,
                                   void *dv_out, void *dg, float *dmeta_k, float *dalpha,
                                   lizard_stream_t stream);

/*
 * lizard_attn_backward with a variant (see lizard_variant).  With alpha_h,
 * dalpha has H entries, d alpha_h[h] (each summed over the batch); with
 * grouped key/value heads, dk and dv are [B][Hkv][L][d], each the sum over
 * its group's query heads (fp32 sum of the heads' values, rounded once).
 */
LIZARD_API lizard_status lizard_attn_backward_v(const void *q, const void *k, const void *v, const void *g,
                                     const void *meta_k, float alpha, int B, int H, int L, int dk, int dv,
                                     int w, int m, lizard_dtype dtype, const void *dy, void *dq, void *dk_out,
                                     void *dv_out, void *dg, float *dmeta_k, float *dalpha,
                                     const lizard_variant *var, lizard_stream_t stream);

/*
 * lizard_gate_projection: the gate logits the operator takes, from the layer
 * input -- the gate module Gamma = sigmoid(W_gamma x) of gist.science/de
 * section 2 item 1 sits directly ahead of the operator; this computes its
 * logits g = W_gamma x and writes them in the operator's head-major layout
 * (the operator applies the log-sigmoid itself):
 *   x        [B][L][dmodel]   bf16   layer input, row-major
 *   w_gamma  [H * dk][dmodel] bf16   gate weight (a linear layer's weight)
 *   g        [B][H][L][dk]    bf16   written: g[b][h][t][i] =
 *                                    sum_c x[b][t][c] w_gamma[h dk + i][c]
 * fp32 accumulation on the tensor cores, rounded to bf16 once.  Supported:
 * bf16, dk == 128, dmodel a multiple of 8 (LIZARD_ERR_UNSUPPORTED
 * otherwise).  B * L == 0 is a no-op.
 */
LIZARD_API lizard_status lizard_gate_projection(const void *x, const void *w_gamma, int B, int L, int dmodel,
                                     int H, int dk, lizard_dtype dtype, void *g, lizard_stream_t stream);

/*
 * lizard_attn_decode_step: one new token for each of st->B sequences and
 * st->H heads, continuing from `st` (updated in place).
 *   q, k, g  [B][H][dk]  st->dtype;  v [B][H][dv];  meta_k [H][m][dk]
 *   y        [B][H][dv]  st->dtype   output
 * At p = pos[b]: S <- diag(sigmoid(g)) S + k^T v; yg = q S; the window is the
 * current token plus tokens max(0, p-w+1) .. p-1 read from the ring; then
 * the current k, v go to ring slot p % w and pos[b] becomes p + 1.
 * Enqueues one kernel.  st->H < 2^20 (LIZARD_ERR_UNSUPPORTED otherwise:
 * the CTAs of a sequence count their arrivals in pos's high bits).
 * Precondition: 0 <= pos[b] < 2^40 (a state written by this library always
 * is).  While the kernel runs, pos[b] carries an
 * arrival count in its high bits; it holds p + 1 again once the step is
 * done.  A pos outside that range is reported (see
 * lizard_check_device_status); that sequence's y, S, ring and pos are then
 * undefined, but every access stays inside the caller's buffers.
 */
LIZARD_API lizard_status lizard_attn_decode_step(const void *q, const void *k, const void *v, const void *g,
                                      const void *meta_k, float alpha, int m, void *y,
                                      const lizard_state *st, lizard_stream_t stream);

/* lizard_attn_decode_step with a variant (see lizard_variant). */
LIZARD_API lizard_status lizard_attn_decode_step_v(const void *q, const void *k, const void *v, const void *g,
                                        const void *meta_k, float alpha, int m, void *y,
                                        const lizard_state *st, const lizard_variant *var,
                                        lizard_stream_t stream);

/*
 * Failure detection is testable without a GPU fault: with the environment
 * variable LIZARD_DEBUG_DECODE_FIRST_WAIT_POLLS=n set when a process first
 * decodes, every decode step of that process gives up its first wait (for
 * its input copies) after n polls, records a timeout and skips its work,
 * still waiting, with the normal limit, for its copies before it retires.
 * lizard_check_device_status then reports LIZARD_ERR_TIMEOUT and the
 * context stays usable.  For testing only; unset, the normal limit applies.
 */

/*
 * lizard_check_device_status: synchronises `stream`, then reads and clears
 * the library's device error word.  LIZARD_ERR_TIMEOUT if a kernel since the
 * last check abandoned a bounded wait (its outputs are then undefined),
 * LIZARD_ERR_INVALID_ARG if a decode step or a continued prefill found a pos
 * outside [0, 2^40), LIZARD_ERR_CUDA if
 * synchronising failed, LIZARD_OK otherwise.
 */
LIZARD_API lizard_status lizard_check_device_status(lizard_stream_t stream);

/* Human-readable name of a status code (static storage). */
LIZARD_API const char *lizard_status_string(lizard_status s);

#ifdef __cplusplus
}
#endif

#endif /* LIZARD_ATTN_H */
