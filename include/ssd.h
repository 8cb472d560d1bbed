/*
 * ssd.h -- C ABI of libssd: the Mamba2 mixer core (conv1d + SiLU over xBC,
 * chunked SSD, causal segments with affine summaries, exclusive segment scan,
 * correction), forward and backward, on one GB300 (sm_103a).
 *
 * Method.  Megatron-LM PR #6808 "Add state-passing context parallelism for
 * Mamba2" (description): the SSD transform of one causal segment is affine in
 * its initial state, S_out = a_block * S_in + S_ext; every segment computes its
 * (S_ext, a_block) from a zero initial state, an exclusive causal scan over the
 * summaries recovers each segment's true initial state, and a correction pass
 * applies it; the conv halo is the previous segment's last d_conv-1 tokens;
 * backward mirrors this with a reverse boundary scan and recomputes everything
 * that scales with the sequence length.  Resets at packed-sequence boundaries
 * follow seq_idx derived from cu_seqlens (NeMo Automodel PR #1441 "feat:
 * context-parallel with nemotron v3", Key changes).  The per-token model is the
 * Mamba2 selective SSM:
 *     u      = SiLU(causal depthwise conv1d(xBC) + conv_b)      (x, B, C parts)
 *     dt_t   = softplus(dt_raw_t + dt_bias),  A = -exp(A_log)
 *     h_t    = exp(dt_t*A) * h_{t-1} + dt_t * x_t (outer) B_t    (P x N per head)
 *     y_t    = h_t . C_t + D * x_t
 * with the state zeroed where seq_idx changes and the conv taps masked there.
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or synchronises the host; every call only enqueues
 *    work on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *  - Arguments are validated before anything is launched.  A rejected call
 *    returns a negative ssd_status and launches nothing.  SSD_ERR_CUDA means a
 *    launch failed; the CUDA error is then also left for cudaGetLastError().
 *  - Activations (x, B, C, dt_raw, y, dy and their grads) use `dims.dtype`;
 *    parameters, states and parameter grads are fp32.  Arithmetic is fp32
 *    (bf16 tensor-core operands with fp32 accumulation on the bf16 path).
 *  - Shapes: b = batch, L = seqlen, H = nheads, P = headdim, N = dstate,
 *    G = ngroups (head h reads group h / (H/G)), Q = chunk, S = n_segments.
 *    Token-major layouts: element (b, t, c) of a tensor with token stride ts
 *    lives at ptr[(b*L + t)*ts + c].  Channels within a token are contiguous.
 */
#ifndef SSD_H
#define SSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ssd_stream_t; /* == cudaStream_t */

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_DIMS = -1,   /* a dimension is <= 0, H % G != 0, or d_conv != 4 */
  SSD_ERR_SEGMENT_ALIGN = -2,  /* L % (n_segments * chunk) != 0 */
  SSD_ERR_NULL_PTR = -3,       /* a required pointer is NULL */
  SSD_ERR_ALIGNMENT = -4,      /* pointer or token stride violates the alignment rules below */
  SSD_ERR_DTYPE = -5,          /* dims.dtype is not an ssd_dtype */
  SSD_ERR_WORKSPACE = -6,      /* workspace NULL or smaller than ssd_workspace_size() */
  SSD_ERR_UNSUPPORTED = -7,    /* valid but outside the supported envelope (see ssd_forward) */
  SSD_ERR_CUDA = -8,           /* a kernel launch failed */
  SSD_ERR_DEVICE_TIMEOUT = -9  /* a bounded device-side wait gave up (see ssd_device_status) */
} ssd_status;

typedef enum { SSD_BF16 = 0, SSD_F32 = 1 } ssd_dtype;

typedef struct {
  int32_t batch, seqlen, nheads, headdim, dstate, ngroups;
  int32_t d_conv;     /* must be 4 */
  int32_t chunk;      /* Q: SSD chunk length */
  int32_t n_segments; /* S: equal causal segments; each must be a multiple of chunk */
  int32_t dtype;      /* ssd_dtype of the activations */
  int32_t gated_norm; /* 1: y is the gated RMSNorm of the mixer output (needs z and
                         norm_weight in ssd_inputs; at most 4096 channels per group), 0: none */
} ssd_dims;

/* Pre-conv activations as laid out by the in-projection (zero-copy views into
 * one zxBCdt buffer are fine: pass each part's pointer and token stride).
 *   x  (b, L, H*P)  B (b, L, G*N)  C (b, L, G*N)  dt (b, L, H)
 * x, B, C: 16-byte aligned, token strides a multiple of 8 elements (bf16) or
 * 4 elements (fp32).  dt: element aligned, any token stride >= H.
 * Parameters (fp32, contiguous): dt_bias, A_log, D (H); conv_w (Cd, 4),
 * 16-byte aligned, where tap 3 multiplies the current token; conv_b (Cd);
 * Cd = H*P + 2*G*N and the conv channel order is [x | B | C].
 * seq_idx (b, L) int32, 16-byte aligned (the tensor-core kernels copy it into
 * shared memory in 16-byte units), non-decreasing within a row, or NULL (one
 * sequence per row).  The state and the conv taps are reset where it changes.
 * initial_states (b, H, P, N) fp32, 16-byte aligned, or NULL (zero): each row's
 * state before its first token, to which that token's decay applies (the
 * Mamba2 chunked-scan convention; the pages list initial states as not
 * supported yet: "Add state-passing context parallelism for Mamba2", "Not
 * supported yet").  With packed rows it seeds the row's first sequence only;
 * later sequences start from zero.  The exclusive segment scan starts from it.
 * Gated RMSNorm (dims.gated_norm = 1; else z and norm_weight must be NULL): the
 * step after the mixer core in a Mamba2 block, which the Megatron-LM PR keeps
 * outside its fused function (description); Mamba2's gated norm with one norm
 * group per B/C group of heads (H*P/G channels):
 *     g = y * silu(z),   out = g * norm_weight / sqrt(mean_group(g^2) + norm_eps)
 * z (b, L, H*P) activation dtype with its own token stride (a view into the
 * zxBCdt buffer), 16-byte aligned, stride a multiple of 8 (bf16) or 4 (fp32)
 * elements; norm_weight (H*P) fp32, 16-byte aligned; norm_eps >= 0. */
typedef struct {
  const void *x;  int64_t x_tok_stride;
  const void *B;  int64_t B_tok_stride;
  const void *C;  int64_t C_tok_stride;
  const void *dt; int64_t dt_tok_stride;
  const float *dt_bias, *A_log, *D, *conv_w, *conv_b;
  const int32_t *seq_idx;
  const float *initial_states;
  const void *z;  int64_t z_tok_stride;
  const float *norm_weight;
  float norm_eps;
} ssd_inputs;

/* Gradients, written (not accumulated).  dx, dB, dC, ddt have the layout and
 * alignment rules of x, B, C, dt, with their own token strides (they may be
 * views into one d(zxBCdt) buffer).  ddt_bias, dA_log, dD (H), dconv_w (Cd,4),
 * dconv_b (Cd) are fp32 and summed over batch and tokens.  dinitial_states
 * (b, H, P, N) fp32, 16-byte aligned: the gradient of the initial states, the
 * reverse segment scan carried one step past the first segment; written only
 * when the inputs have initial_states, and may be NULL.  With the gated norm:
 * dz (layout rules of z, its own token stride) and dnorm_weight (H*P) fp32,
 * both required. */
typedef struct {
  void *dx;  int64_t dx_tok_stride;
  void *dB;  int64_t dB_tok_stride;
  void *dC;  int64_t dC_tok_stride;
  void *ddt; int64_t ddt_tok_stride;
  float *ddt_bias, *dA_log, *dD, *dconv_w, *dconv_b;
  float *dinitial_states;
  void *dz;  int64_t dz_tok_stride;
  float *dnorm_weight;
} ssd_grads;

/* Bytes of device workspace ssd_forward (backward = 0) or ssd_backward
 * (backward = 1) needs for `dims`; 0 if dims are invalid.  The workspace is
 * scratch: its contents need not survive between calls. */
size_t ssd_workspace_size(const ssd_dims *dims, int backward);

/* Forward.  y (b, L, H*P) activation dtype, contiguous (with the gated norm: its
 * output; the mixer output itself is not written); final_state (b, H, P, N)
 * fp32 = the state after each row's last token (with packing: of the row's last
 * sequence), or NULL; seg_init_states (b, S, H, P, N) fp32 = each segment's true
 * initial state recovered by the exclusive scan (what ssd_backward may reuse),
 * or NULL.  Supported envelope: P and N multiples of 8 and <= 256, chunk a
 * multiple of 32 and <= 256, n_segments <= 1024; otherwise SSD_ERR_UNSUPPORTED. */
ssd_status ssd_forward(const ssd_dims *dims, const ssd_inputs *in, void *y, float *final_state,
                       float *seg_init_states, void *workspace, size_t ws_bytes, ssd_stream_t stream);

/* Forward of a packed row of sequences (THD layout, dims.batch = 1) that also
 * returns the state after every sequence's last token: seq_final_states
 * (nseq, H, P, N) fp32, 16-byte aligned, sequence s covering tokens
 * [cu_seqlens[s], cu_seqlens[s+1]) (cu_seqlens: nseq + 1 int32 device values, the
 * layout of "feat: context-parallel with nemotron v3", Key changes).  in->seq_idx
 * is required and must describe the same sequences (ssd_cu_seqlens_to_seq_idx
 * makes it; neither is checked against the other on the host).  Sequences
 * that are empty or fall outside [0, seqlen) get a zero state.  Everything else
 * as ssd_forward, same workspace size.  No gradient flows back through
 * seq_final_states (ssd_backward's dfinal_state is the row's last token's). */
ssd_status ssd_forward_varlen(const ssd_dims *dims, const ssd_inputs *in, void *y, float *final_state,
                              float *seg_init_states, const int32_t *cu_seqlens, int32_t nseq,
                              float *seq_final_states, void *workspace, size_t ws_bytes, ssd_stream_t stream);

/* Backward of  L = <dy, y> + <dfinal_state, final_state>  (y the forward's output:
 * with the gated norm, the normalised output; the mixer output is recomputed).
 * dy (b, L, H*P) activation dtype, contiguous; dfinal_state (b, H, P, N) fp32 or
 * NULL (zero); seg_init_states from ssd_forward on the same inputs, or NULL to
 * have them recomputed.  Everything that scales with L is recomputed. */
ssd_status ssd_backward(const ssd_dims *dims, const ssd_inputs *in, const void *dy, const float *dfinal_state,
                        const float *seg_init_states, const ssd_grads *grads, void *workspace, size_t ws_bytes,
                        ssd_stream_t stream);

/* Forward without any workspace argument, for callers that cannot allocate
 * device memory: code running inside a host framework that owns every device
 * allocation and forbids new ones after start-up (inference plugins, real-time
 * serving loops), or code for which a cudaMalloc would synchronise the device
 * and break its latency budget.  Same arguments, results and rules as
 * ssd_forward minus the workspace.  The scratch is one fixed array of
 * SSD_STATIC_SCRATCH_BYTES in the library's device memory (each GPU that loads
 * the library holds it until the process exits); problems whose forward needs
 * more (ssd_workspace_size(dims, 0) > SSD_STATIC_SCRATCH_BYTES) are rejected
 * with SSD_ERR_WORKSPACE before anything is launched.  The first call on each
 * device looks up the array's device address (make that first call before any
 * stream capture); no call allocates or frees memory.  All calls share the one
 * array, so calls whose GPU work may overlap (other streams, other host
 * threads) race on it and must be serialised by the caller.  The array's
 * status word (a device-side wait that gave up) is read with
 * ssd_device_status(NULL, stream).  This entry point has no counterpart in the
 * pages the method comes from. */
#define SSD_STATIC_SCRATCH_BYTES (32u << 20)
ssd_status ssd_forward_static(const ssd_dims *dims, const ssd_inputs *in, void *y, float *final_state,
                              float *seg_init_states, ssd_stream_t stream);

/* seq_idx[t] = i for cu_seqlens[i] <= t < cu_seqlens[i+1], t in [0, total_tokens)
 * (NeMo Automodel PR #1441, Key changes: seq_idx computed from cu_seqlens).
 * cu_seqlens (nseq + 1) int32 device array, non-decreasing, cu_seqlens[0] = 0 and
 * cu_seqlens[nseq] = total_tokens (not checked on the host: tokens outside every
 * range get seq_idx -1). */
ssd_status ssd_cu_seqlens_to_seq_idx(const int32_t *cu_seqlens, int32_t nseq, int32_t *seq_idx,
                                     int32_t total_tokens, ssd_stream_t stream);

/* Reads the device status word kept in `workspace` by the last call that used
 * it (synchronises `stream`): SSD_OK, or SSD_ERR_DEVICE_TIMEOUT if a bounded
 * device-side wait gave up (the outputs of that call are then garbage; the
 * context stays usable and the next call starts from a cleared word).
 * workspace = NULL reads the word of ssd_forward_static's fixed scratch array
 * on the current device instead.  Returns SSD_ERR_CUDA if the read fails. */
ssd_status ssd_device_status(const void *workspace, ssd_stream_t stream);

/* Failure detection.  Every wait of one role of a kernel on another (mbarrier
 * hand-offs inside the tensor-core kernels) gives up after this limit,
 * raises the status word that ssd_device_status reads and lets the kernel
 * finish: it drains the copies and tensor-core operations it started, frees
 * its tensor memory and returns, so the process can carry on.  Applies to the
 * calls made after it, from any host thread; returns the previous limit.  The
 * default, SSD_DEFAULT_WAIT_LIMIT_NS (1.5 s), is far above any real hand-off;
 * a limit of 0 makes every wait that is not already satisfied give up (a way
 * to exercise the failure path). */
#define SSD_DEFAULT_WAIT_LIMIT_NS 1500000000ull
uint64_t ssd_set_wait_limit_ns(uint64_t limit_ns);

/* Per-kernel timing for benchmarks.  After ssd_profile_begin(), every kernel
 * that ssd_forward / ssd_backward launch (from this host thread) is bracketed
 * by a pair of CUDA events recorded on the launch stream (events come from a
 * fixed pool created on the first begin; at most 65536 launches are recorded,
 * later ones run unrecorded).  ssd_profile_end() waits for the recorded events,
 * writes up to max_entries per-kernel totals (name, launches, summed
 * milliseconds) in first-launch order, stops recording and returns the number
 * of entries, or a negative ssd_status.  Not for use during stream capture. */
typedef struct {
  const char *name; /* static string */
  int32_t launches;
  float total_ms;
} ssd_kernel_time;

ssd_status ssd_profile_begin(void);
int32_t ssd_profile_end(ssd_kernel_time *out, int32_t max_entries);

/* Static description of a status code. */
const char *ssd_status_string(ssd_status status);

#ifdef __cplusplus
}
#endif
#endif /* SSD_H */
