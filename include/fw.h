/*
 * fw.h -- C ABI of the GB300 (sm_103a) fast-weight memory recurrence library
 * (libfw.so).
 *
 * The library computes the causal fast-weight memory recurrence of the
 * "Fast Weight Attention for Continual Learning" paper reading (Falcon-1,
 * §3.2 and §4.2): every token writes into a d_k x d_v fp32 state S with one
 * normalised gradient step on the instantaneous ridge loss
 *
 *     l_t(S) = 1/2 |S^T x_t - y_t|^2 + (lambda_t / 2) |S|_F^2,
 *     r_t    = y_t - S_{t-1}^T x_t,
 *     eta_t  = beta_t / (|x_t|^2 + lambda_t + eps),
 *     S_t    = (1 - eta_t lambda_t) S_{t-1} + eta_t x_t r_t^T,
 *
 * on the shifted training pair (x_t, y_t) = (phi(k_{t-1}), v_t) with the
 * boundary x_1 := 0, eta_1 := 0 (§4.1), and reads after the write,
 * o_t = S_t^T q_t (§1.4).  FW_FALCON1A is the same page's inner-product family
 * (§4.3): the write drops the residual, S_t = (1 - eta_t lambda_t) S_{t-1}
 * + eta_t x_t y_t^T, with Falcon-1's step, pairing and boundary.  FW_FALCON2 and
 * FW_FALCON2A take a step size per value channel (§4.2): beta is indexed by the
 * value column j as well, eta_{j,t} = beta_{j,t} / (|x_t|^2 + lambda_t + eps),
 * and column j of S takes its own scalar write.  FW_FALCON3 and FW_FALCON3A
 * (§4.2, §4.3; entry points fw_window_prefill / fw_window_step) write with one
 * gradient step on the average loss of the last W pairs (the window),
 *     S_t = (1 - eta_t lambda_t) S_{t-1}
 *           + (eta_t / B_t) sum_{j in window} x_j (y_j - S_{t-1}^T x_j)^T,
 *     eta_t = beta_t / (mu_t + lambda_t + eps),
 *     mu_t = largest eigenvalue of (1/B_t) sum_{j in window} x_j x_j^T,
 * where the window holds the pairs t-W+1 .. t that exist and B_t counts them
 * (eta_t = 0 when none does); FW_FALCON3A writes y_j in place of the
 * residual.  With W = 1 they are FW_FALCON1 and FW_FALCON1A.  Flags select
 * the other arms of the page's read / pairing design (§3.3, §4.1): reading
 * before the write and the same-step pair.  FW_LINATTN selects plain causal linear attention,
 * S_t = S_{t-1} + phi(k_t) v_t^T, o_t = S_t^T phi(q_t) ("Attention is also an
 * FFN" blog, §2.1 and §4.1), the special case without residual or decay.
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them.  Rows are contiguous, row-major.
 *     Its own workspace is taken only by the chunked prefill's two-segment
 *     form (few long chains; see fw_debug_segment_split), stream-ordered on the
 *     call's stream from a private pool that keeps its memory between calls.
 *   - q, k, v, o:  [B][H][T][d] (prefill) or [B][H][d] (step), element type
 *     FW_F32 (float) or FW_BF16 (bfloat16), d innermost.
 *   - beta, lambda: float [B][H][T] (prefill) or [B][H] (step); beta of
 *     FW_FALCON2 / FW_FALCON2A is float [B][H][T][d_v] (prefill) or [B][H][d_v]
 *     (step).  Ignored (may be NULL) in FW_LINATTN mode, required otherwise.
 *   - S0, S_T, S: float [B][H][d_k][d_v], S[i][j] = key row i, value column j,
 *     so a read is o_j = sum_i S[i][j] q_i (the blog's y = q @ S).
 *   - Pointers must be 16-byte aligned (vector and TMA loads).
 *   - Every call validates its arguments before any launch, enqueues its work
 *     on `stream` and returns without synchronising.  A non-zero return means
 *     nothing was launched (except FW_ERR_CUDA, see fw_last_cuda_error()).
 *   - Waits inside kernels are bounded; a wait that runs out sets a device
 *     error word instead of hanging.  fw_check() reads and clears it.
 *   - Inputs are never written (except S in fw_step, updated in place).
 */
#ifndef FW_H_
#define FW_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FW_VERSION 120 /* 1.2.0 */

typedef enum { FW_F32 = 0, FW_BF16 = 1 } fw_dtype;

/* FW_FALCON1: shifted pair, residual write, normalised step and decay.
 * FW_LINATTN: same-step pair, additive write S += phi(k) v^T, no eta/gamma.
 * FW_FALCON1A: Falcon-1's pair, step and decay with the additive write
 *              S = gamma S + eta x v^T (no residual).
 * FW_FALCON2, FW_FALCON2A: FW_FALCON1, FW_FALCON1A with a step size (and so a
 *              decay) per value channel; beta carries a trailing d_v index.
 * FW_FALCON3, FW_FALCON3A: the window modes, taken only by fw_window_prefill
 *              and fw_window_step (the other calls return FW_ERR_MODE). */
typedef enum {
    FW_FALCON1 = 0, FW_LINATTN = 1, FW_FALCON1A = 2, FW_FALCON2 = 3, FW_FALCON2A = 4,
    FW_FALCON3 = 5, FW_FALCON3A = 6
} fw_mode;

/* Largest window (number of pairs W) of FW_FALCON3 / FW_FALCON3A. */
#define FW_WINDOW_MAX 8

/* The pairs that a Falcon-3 window carries from one call to the next: the
 * newest W-1 training pairs of every chain, which the next token's window
 * still holds.  Device pointers owned by the caller.  For W = 1 nothing is
 * carried and the struct is not read. */
typedef struct {
    float *x;    /* [B][H][W-1][d_k] the pairs' keys, phi applied, oldest first */
    float *y;    /* [B][H][W-1][d_v] their targets (values), as fp32 */
    int32_t *n;  /* [B][H] how many pairs are held, in the newest n slots
                    (0 .. W-1); the other slots are ignored on input and
                    written as zeros */
} fw_window;

/* Flags (bitwise OR) of fw_prefill_ex and fw_step_ex.
 * FW_FLAG_RBW: read before the write, o_t = S_{t-1}^T q_t (every mode).
 * FW_FLAG_SAME_PAIR: FW_FALCON1 / FW_FALCON1A pair (phi(k_t), v_t) for every
 *   token, so the first token writes too and k_init is not used (prefill
 *   only; FW_LINATTN always pairs this way, and a step pairs whatever key it
 *   is given).  The pages name these arms without printing formulas; the
 *   readings above are the plainest ones. */
typedef enum { FW_FLAG_RBW = 1, FW_FLAG_SAME_PAIR = 2 } fw_flag;

/* Feature map phi.  FW_FALCON1 applies it to the key only (the read uses q as
 * given); FW_LINATTN applies it to both q and k, never to v.
 * FW_PHI_ELU1: elu(z) + 1 = z + 1 for z > 0, exp(z) for z <= 0. */
typedef enum { FW_PHI_IDENTITY = 0, FW_PHI_ELU1 = 1 } fw_phi;

/* Kernel choice for fw_prefill_ex.  FW_ALGO_AUTO picks a chunked tensor-core
 * kernel when one supports the call (bf16, d_k = d_v = 128; for FW_FALCON1,
 * FW_FALCON1A, FW_FALCON2 and FW_FALCON2A only with FW_PHI_IDENTITY): the
 * per-channel one for FW_FALCON2 / FW_FALCON2A, the shared-step one for the
 * other modes.  Otherwise FW_FALCON2 / FW_FALCON2A run on the staged per-token
 * kernel of the window family and the other modes on the plain per-token SIMT
 * recurrence.  FW_ALGO_CHUNKED insists on a chunked kernel; FW_ALGO_RECURRENT
 * forces the plain per-token recurrence. */
typedef enum { FW_ALGO_AUTO = 0, FW_ALGO_RECURRENT = 1, FW_ALGO_CHUNKED = 2 } fw_algo;

typedef struct {
    int64_t B;   /* batch, >= 1 */
    int64_t H;   /* heads, >= 1 */
    int64_t T;   /* tokens per chain; >= 1 for prefill, must be 1 for fw_step */
    int32_t d_k; /* key width, 64 or 128 */
    int32_t d_v; /* value width, equal to d_k */
} fw_shape;

enum {
    FW_OK = 0,
    FW_ERR_NULL = -1,        /* a required pointer is NULL */
    FW_ERR_SHAPE = -2,       /* B, H or T < 1, d_k not in {64,128}, d_v != d_k, T != 1 in a
                                step, window outside 1 .. FW_WINDOW_MAX */
    FW_ERR_DTYPE = -3,       /* unknown fw_dtype */
    FW_ERR_ALIGN = -4,       /* a pointer is not 16-byte aligned */
    FW_ERR_MODE = -5,        /* unknown fw_mode, fw_phi, fw_algo or flag bit, or a mode
                                the call does not take */
    FW_ERR_CUDA = -6,        /* a CUDA call failed; see fw_last_cuda_error() */
    FW_ERR_TIMEOUT = -7,     /* a bounded device wait ran out (reported by fw_check) */
    FW_ERR_UNSUPPORTED = -8, /* FW_ALGO_CHUNKED asked for a call it does not support */
    FW_ERR_ARG = -9,         /* eps negative or not finite, or o aliases an input */
    FW_ERR_DEVICE = -10,     /* the current device is not an sm_103 GPU */
    FW_ERR_SCRATCH = -11     /* fw_prefill_noalloc: the call needs more than FW_SCRATCH_BYTES */
};

/*
 * fw_prefill -- run the recurrence over T tokens for B*H independent chains.
 *
 * Passage: "Fast Weight Attention for Continual Learning" paper reading,
 * §3.2/§4.1/§4.2 (FW_FALCON1); "Attention is also an FFN" blog §2.1
 * (FW_LINATTN).  Chunked evaluation follows the same page's §4.4 (intra-chunk
 * triangular solve, short inter-chunk recurrence, parallel outputs).
 *
 *   q, k, v  in   [B][H][T][d] of `dtype`
 *   beta     in   float [B][H][T], or [B][H][T][d_v] for FW_FALCON2 /
 *                 FW_FALCON2A (not FW_LINATTN; beta in [0, 2) keeps the
 *                 regression write stable, other values are computed
 *                 literally)
 *   lambda   in   float [B][H][T]   (not FW_LINATTN; >= 0)
 *   S0       in   float [B][H][d][d] or NULL for a zero start state
 *   o        out  [B][H][T][d] of `dtype` (rounded to nearest even for bf16);
 *                 must not overlap any input
 *   S_T      out  float [B][H][d][d], the state after token T; may equal S0
 *   eps      in   >= 0, added to the step's denominator (not FW_LINATTN)
 * Returns FW_OK or a negative FW_ERR_* code.
 */
int fw_prefill(const void *q, const void *k, const void *v, const float *beta,
               const float *lambda, const float *S0, void *o, float *S_T,
               const fw_shape *shape, fw_dtype dtype, fw_mode mode, fw_phi phi, float eps,
               cudaStream_t stream);

/*
 * fw_prefill_ex -- fw_prefill with three more arguments.
 *   k_init  in  [B][H][d] of `dtype` or NULL.  FW_FALCON1 / FW_FALCON1A with
 *               the shifted pair: the key that precedes this call's first
 *               token (the last key of a previous prefill of the same
 *               sequence).  Given, the first token's pair is (phi(k_init), v_1)
 *               with the normal step; NULL keeps the boundary x_1 = 0,
 *               eta_1 = 0.  Ignored in FW_LINATTN mode and with
 *               FW_FLAG_SAME_PAIR.
 *   flags   in  0 or FW_FLAG_* bits (FW_ERR_MODE for unknown bits).
 *   algo    in  FW_ALGO_AUTO, or force one kernel (FW_ERR_UNSUPPORTED if the
 *               chunked kernel cannot take the call).
 */
int fw_prefill_ex(const void *q, const void *k, const void *v, const float *beta,
                  const float *lambda, const float *S0, const void *k_init, void *o,
                  float *S_T, const fw_shape *shape, fw_dtype dtype, fw_mode mode,
                  fw_phi phi, float eps, unsigned flags, fw_algo algo, cudaStream_t stream);

/*
 * fw_prefill_noalloc -- fw_prefill_ex for callers that want no device memory
 * allocated on their behalf.  The pages have no counterpart: this is a
 * deployment detail of this library, not part of the method.
 *
 * Same arguments, validation and kernels as fw_prefill_ex.  The only call
 * that needs workspace is the chunked prefill's two-segment form (few long
 * chains, see fw_debug_segment_split); here it takes that workspace from one
 * static device buffer of FW_SCRATCH_BYTES compiled into the library
 * (file-scope, 256-byte aligned) instead of the stream-ordered pool, and
 * nothing is allocated or freed.  A call whose two-segment form would need
 * more than FW_SCRATCH_BYTES (n_chains x (T - T/2) x 256 bytes plus
 * n_chains x 224 KiB) returns FW_ERR_SCRATCH and launches nothing; every
 * other call runs exactly as fw_prefill_ex would.
 *   - One buffer per device: calls that overlap on a device (two streams, two
 *     host threads) race on it; order them.
 *   - The first call on a device looks the buffer's address up
 *     (cudaGetSymbolAddress) and sets kernel attributes: make one call
 *     before capturing a stream.
 *   - Nothing in the buffer has to start at zero: the segment launch writes
 *     every byte the second kernel reads.
 *   - The buffer is reserved when the library's module holding it loads
 *     (with CUDA's default lazy loading, at the first call of this function).
 * Returns FW_OK or a negative FW_ERR_* code.
 */
#define FW_SCRATCH_BYTES (144u * 1024u * 1024u)
int fw_prefill_noalloc(const void *q, const void *k, const void *v, const float *beta,
                       const float *lambda, const float *S0, const void *k_init, void *o,
                       float *S_T, const fw_shape *shape, fw_dtype dtype, fw_mode mode,
                       fw_phi phi, float eps, unsigned flags, fw_algo algo,
                       cudaStream_t stream);

/*
 * fw_step -- one decode step for B*H independent states, S updated in place.
 *
 * Passage: the Falcon-1 write of "Fast Weight Attention for Continual
 * Learning" paper reading §3.2 with the pair (phi(k_prev), v) and the read
 * after the write; the blog's forward_step (§4.1) for FW_LINATTN, where
 * `k_prev` is the current token's key.  A step knows no position: to start a
 * sequence with steps pass beta = 0 (an empty first write).
 *
 *   q, k_prev, v  in      [B][H][d] of `dtype`
 *   beta, lambda  in      float [B][H] (beta [B][H][d_v] for FW_FALCON2 /
 *                         FW_FALCON2A; not used by FW_LINATTN)
 *   S             in/out  float [B][H][d][d]
 *   o             out     [B][H][d] of `dtype`, o = S_new^T q
 *   shape         T must be 1
 */
int fw_step(const void *q, const void *k_prev, const void *v, const float *beta,
            const float *lambda, float *S, void *o, const fw_shape *shape, fw_dtype dtype,
            fw_mode mode, fw_phi phi, float eps, cudaStream_t stream);

/*
 * fw_step_ex -- fw_step with flags: FW_FLAG_RBW reads before the write,
 * o = S_old^T q (FW_FLAG_SAME_PAIR has no effect on a step: the pair is
 * whatever key is passed as `k_prev`).  Unknown bits give FW_ERR_MODE.
 */
int fw_step_ex(const void *q, const void *k_prev, const void *v, const float *beta,
               const float *lambda, float *S, void *o, const fw_shape *shape, fw_dtype dtype,
               fw_mode mode, fw_phi phi, float eps, unsigned flags, cudaStream_t stream);

/*
 * fw_window_prefill -- FW_FALCON3 / FW_FALCON3A over T tokens for B*H chains,
 * with a window of `window` pairs (1 .. FW_WINDOW_MAX).
 *
 * Passage: "Fast Weight Attention for Continual Learning" paper reading,
 * §4.2 (Falcon-3, the sliding-window minibatch step) and §4.3 (Falcon-3A);
 * pairing, boundary and read as fw_prefill (§4.1, §1.4).  The pages give the
 * window no size and no start-of-sequence rule: the window holds the pairs
 * that exist (the first token's shifted pair does not, unless k_init is
 * given), B_t counts them, and a carried window supplies the pairs of an
 * earlier call.
 *
 *   q, k, v, beta, lambda, S0, k_init, o, S_T, eps
 *            as fw_prefill_ex (beta, lambda float [B][H][T]; phi applies to
 *            the key only; o must not overlap an input)
 *   win_in   in   the window carried from an earlier call of the same
 *                 sequences, or NULL (no pairs before this call)
 *   win_out  out  the window after token T, or NULL (not wanted); its arrays
 *                 must not overlap win_in's or any other argument
 *   window   W, 1 .. FW_WINDOW_MAX (FW_ERR_SHAPE otherwise)
 *   mode     FW_FALCON3 or FW_FALCON3A (FW_ERR_MODE otherwise)
 *   flags    FW_FLAG_RBW (read before the write), FW_FLAG_SAME_PAIR (pair
 *            (phi(k_t), v_t) for every token; k_init unused)
 * Evaluated by a per-token SIMT kernel in fp32.  Returns FW_OK or FW_ERR_*.
 */
int fw_window_prefill(const void *q, const void *k, const void *v, const float *beta,
                      const float *lambda, const float *S0, const void *k_init,
                      const fw_window *win_in, void *o, float *S_T, const fw_window *win_out,
                      const fw_shape *shape, int window, fw_dtype dtype, fw_mode mode,
                      fw_phi phi, float eps, unsigned flags, cudaStream_t stream);

/*
 * fw_window_step -- one FW_FALCON3 / FW_FALCON3A decode step for B*H states:
 * the window is the carried pairs plus the new pair (phi(k_prev), v); S is
 * updated in place and the carried window moves on by one pair.
 *
 * Passage: as fw_window_prefill; the step is the same write for one token.
 *
 *   q, k_prev, v, beta, lambda, S, o, eps   as fw_step (beta, lambda [B][H])
 *   win_in   in   the carried window, or NULL (empty)
 *   win_out  out  the window after this step, or NULL; it must not overlap
 *                 win_in (alternate two buffers from step to step)
 *   window, mode  as fw_window_prefill; flags: FW_FLAG_RBW only
 *   shape    T must be 1
 */
int fw_window_step(const void *q, const void *k_prev, const void *v, const float *beta,
                   const float *lambda, float *S, const fw_window *win_in, void *o,
                   const fw_window *win_out, const fw_shape *shape, int window, fw_dtype dtype,
                   fw_mode mode, fw_phi phi, float eps, unsigned flags, cudaStream_t stream);

/* Synchronise `stream`, then read and clear the device error word.
 * Returns FW_OK, FW_ERR_TIMEOUT, or FW_ERR_CUDA. */
int fw_check(cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *fw_status_string(int status);

/* FW_VERSION of the built library. */
int fw_version(void);

/* The cudaError_t of the last failed CUDA call in this thread (0 if none). */
int fw_last_cuda_error(void);

/* Wall-time limit of every bounded device wait, in microseconds (default
 * 2,000,000).  Values < 1 restore the default.  Applies to later calls. */
void fw_set_wait_limit_us(long long us);

/* Testing hook for the timeout path: while `on` is non-zero, chunked-kernel
 * launches first wait on a barrier that nothing arrives on, so the wait runs
 * out after the wait limit; the kernel then records FW_ERR_TIMEOUT (read by
 * fw_check), drains its copies in flight, frees its tensor memory and exits.
 * No GPU fault is involved. */
void fw_debug_force_timeout(int on);

/* Testing hook for the two-segment form of the chunked prefill (Falcon-1, 1A,
 * linear attention; bf16, d = 128).  With few chains and a long sequence the
 * chunked launch splits each chain at a chunk boundary near T/2 and runs, at
 * once, the first segment from S0, the second from a zero state, and the second
 * again from S = I with zero targets; since the state map of a segment is affine
 * in its initial state (S_t = Phi_t S_mid + S_t^0), a second kernel then adds
 * S_mid^T (Phi_t^T q_t) to the second segment's outputs and forms
 * S_T = Phi_T S_mid + S_T^0.  mode 0 (default): the launch decides (at most a
 * third of the SMs hold a chain and T >= 4096); 1: split whenever T spans two
 * chunks; -1: never.  Applies to later calls.  The split draws its workspace
 * (bf16 n_chains x (T - T/2) x 128 and fp32 3 x n_chains x 128 x 128) from a
 * stream-ordered pool; without it the call runs unsplit. */
void fw_debug_segment_split(int mode);

#ifdef __cplusplus
}
#endif
#endif /* FW_H_ */
