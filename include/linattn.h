/*
 * linattn.h -- C ABI of the GB300 (sm_103a) causal kernelised linear
 * attention library (liblinattn.so).
 *
 * The operation, in the notation of the pages it follows:
 *
 *   feature map   phi(x) = elu(x) + 1  (alpha = 1; positive)
 *                 ["Linear Attention Kernel", section "Choice of phi";
 *                  "Efficient Attention Variants", section 4]
 *   causal state  S_t = S_{t-1} + phi(k_t) v_t^T,  z_t = z_{t-1} + phi(k_t),
 *                 S_0 = 0, z_0 = 0, write before read (token t sees itself)
 *   causal read   o_t = phi(q_t)^T S_t / phi(q_t)^T z_t
 *                 ["Efficient Attention Variants", section 5, prefix-sum
 *                  recurrence; "Linear Attention Kernel", section
 *                  "Recurrent form"]
 *   non-causal    S = phi(K)^T V, z = column sums of phi(K),
 *                 o_i = phi(q_i)^T S / phi(q_i)^T z
 *                 ["Linear Attention Kernel", section "Rewrite:
 *                  associativity"; "Efficient Attention Variants", section 4]
 *   scalar decay  S_t = gamma_h S_{t-1} + k_t v_t^T,  o_t = q_t^T S_t
 *                 (RetNet; no feature map, no normaliser)
 *                 ["Efficient Attention Variants", section 7.1]
 *   decode step   one iteration of the causal recurrence on a stored state,
 *                 with no KV cache ["Efficient Attention Variants",
 *                 sections 1 and 5; "Linear Attention and SSM", eq.
 *                 attn-linssm-recurrence]
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are DEVICE pointers on the current CUDA device,
 *    owned by the caller, contiguous row-major, 16-byte aligned (workspaces:
 *    256-byte aligned):
 *        q, k   [B, H, N, d]     (dtype: bf16 or fp32, see la_dtype)
 *        v      [B, H, N, dv]
 *        out    [B, H, N, dv]    always fp32
 *        S      [B, H, d, dv]    fp32, S[b,h,i,c] pairs key feature i with
 *                                value channel c
 *        z      [B, H, d]        fp32
 *    The feature dimension r of the pages equals d.
 *  - d and dv must each be 32, 64 or 128.  B, H >= 1.  N >= 0 (N = 0 is a
 *    no-op).  B*H <= 2^31 - 1.
 *  - gamma is a HOST pointer to H floats (per-head decay, 0 < gamma <= 1),
 *    read during the call and not retained, or NULL for no decay.  For
 *    normalised feature maps the decay weights numerator and denominator
 *    alike (mask gamma^(t-j)).  Decay is not defined for the non-causal form.
 *  - Every call only enqueues work on `stream` (NULL = legacy default stream)
 *    and returns; results are ready once the stream is synchronised.  No
 *    entry point allocates or frees memory on the compute path; scratch is
 *    the caller's `workspace`.
 *  - Argument errors are returned before anything is enqueued.  A status of
 *    LA_ERR_CUDA means a launch failed (the CUDA error is left for the
 *    caller's next runtime call).  Device-side checks (bounded waits, index
 *    checks) never trap: they record a code in a per-device status word that
 *    la_get_device_status() returns and clears.
 *  - Normalised reads divide by max(phi(q)^T z, FLT_MIN); for elu+1 the
 *    denominator is a sum of positive terms, so this only matters when every
 *    term underflows (the numerator is then zero too and o = 0).
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LA_API __attribute__((visibility("default")))
#else
#define LA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; kept opaque so this header needs no CUDA headers. */
typedef struct CUstream_st* la_stream_t;

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,   /* NULL / misaligned pointer, bad size or enum  */
    LA_ERR_UNSUPPORTED = 2,   /* valid request outside what is implemented   */
    LA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed        */
    LA_ERR_TIMEOUT = 4,       /* device: a bounded wait gave up              */
    LA_ERR_DEVICE_CHECK = 5,  /* device: an internal consistency check failed */
    LA_ERR_WORKSPACE = 6,     /* workspace missing or smaller than required  */
    LA_ERR_TOO_LARGE = 7      /* la_forward_noalloc: the sizes need more
                                 scratch than its fixed device array holds   */
} la_status;

typedef enum {
    LA_FM_ELU1 = 0,          /* phi = elu + 1, normalised read               */
    LA_FM_IDENTITY_NORM = 1, /* phi = identity, normalised read (the pages'
                                hand-worked examples give features directly) */
    LA_FM_NONE = 2           /* phi = identity, unnormalised (RetNet)        */
} la_feature_map;

typedef enum {
    LA_BF16 = 0,             /* q, k, v are bfloat16                          */
    LA_FP32 = 1              /* q, k, v are float                             */
} la_dtype;

/* Library version, major * 10000 + minor * 100 + patch. */
LA_API int la_version(void);

/* Static description of a status code; never NULL. */
LA_API const char* la_status_string(la_status status);

/*
 * Bytes of device workspace la_forward needs for these sizes (0 for N = 0).
 * The workspace holds per-chunk fp32 states and the chunk-scan flags; its
 * contents on entry do not matter and on exit are unspecified.
 */
LA_API size_t la_forward_workspace_size(int64_t B, int64_t H, int64_t N, int d, int dv, int causal,
                                 int dtype);

/*
 * Forward over B*H independent sequences of N tokens.
 *   causal = 1 : o_t reads the prefix state S_t (j <= t).
 *   causal = 0 : every o_i reads the full-sequence state (gamma must be NULL).
 *   feature_map: la_feature_map.  dtype: la_dtype of q, k, v.
 *   workspace  : device buffer of at least la_forward_workspace_size() bytes,
 *                256-byte aligned (cudaMalloc and PyTorch allocations are),
 *                owned by the caller; must not be used by another call that
 *                runs concurrently.  A missing, short or misaligned workspace
 *                returns LA_ERR_WORKSPACE before anything is enqueued.
 * Returns LA_OK once the work is enqueued on `stream`.
 */
LA_API la_status la_forward(const void* q, const void* k, const void* v, float* out, int64_t B,
                     int64_t H, int64_t N, int d, int dv, int causal, int feature_map,
                     const float* gamma, int dtype, void* workspace, size_t workspace_bytes,
                     la_stream_t stream);

/*
 * Causal forward continued from a given state and/or returning the final
 * state: the prefill of a long prompt in pieces, and the hand-off of a
 * prefill to la_decode_step at any point ("Efficient Attention Variants",
 * sections 1 and 5: the fixed-size state S_t, z_t is the whole summary of
 * the tokens before t).
 *   S0 [B,H,d,dv], z0 [B,H,d] : fp32 state before the first token, or both
 *                               NULL for S_0 = 0, z_0 = 0.  With decay, S0
 *                               and z0 are decayed like any earlier token.
 *   S_out, z_out              : fp32 buffers that receive the state after
 *                               the last token, or both NULL.  They may be
 *                               the same buffers as S0, z0 (in-place update).
 *   out                       : [B,H,N,dv] outputs, or NULL together with q
 *                               for a state-only call (then S_out is
 *                               required).
 * Every other argument is as for la_forward (causal form only); the
 * workspace must hold la_forward_workspace_size(B, H, N, d, dv, 1, dtype)
 * bytes.  With N = 0 the final state is S0, z0 (or zero).
 */
LA_API la_status la_forward_with_state(const void* q, const void* k, const void* v, float* out,
                                       const float* S0, const float* z0, float* S_out,
                                       float* z_out, int64_t B, int64_t H, int64_t N, int d,
                                       int dv, int feature_map, const float* gamma, int dtype,
                                       void* workspace, size_t workspace_bytes,
                                       la_stream_t stream);

/*
 * Diagnostic: the kernel path la_forward takes for these arguments --
 * "tcgen05" (the single-pass tensor-core kernel: bf16, d = dv = 64, causal,
 * no decay), "tcgen05_chunked" (the chunked tensor-core path: bf16, d and dv
 * in {64, 128}; decay only with LA_FM_NONE) or "simt" (CUDA cores, fp32,
 * every other case); "invalid" for arguments la_forward would reject.
 * has_decay: 1 if gamma will be non-NULL.  la_forward_with_state and
 * la_state take the chunked tensor-core path wherever its sizes and dtype
 * allow (la_state also with decay and a normalised map), else the CUDA-core
 * path.
 */
LA_API const char* la_forward_path(int64_t B, int64_t H, int64_t N, int d, int dv, int causal,
                                   int feature_map, int has_decay, int dtype);

/* Bytes of device workspace la_state needs (0 for N = 0); the workspace must be
 * 256-byte aligned, as for la_forward. */
LA_API size_t la_state_workspace_size(int64_t B, int64_t H, int64_t N, int d, int dv, int dtype);

/*
 * Final state of the causal recurrence after N tokens, starting from
 * S_0 = 0, z_0 = 0:  S [B,H,d,dv] and z [B,H,d] (fp32, overwritten).  This is
 * the prefill that hands a prompt to la_decode_step.  With N = 0 the outputs
 * are set to zero.  z is required for every feature map (for LA_FM_NONE it
 * receives the undecayed-or-decayed key sum and is simply unused by reads).
 */
LA_API la_status la_state(const void* k, const void* v, float* S, float* z, int64_t B, int64_t H,
                   int64_t N, int d, int dv, int feature_map, const float* gamma, int dtype,
                   void* workspace, size_t workspace_bytes, la_stream_t stream);

/*
 * One decode step for B*H sequences, one new token each:
 *   S <- gamma S + phi(k) v^T ;  z <- gamma z + phi(k) ;  o = phi(q)^T S / phi(q)^T z
 * (o = phi(q)^T S for LA_FM_NONE).  S [B,H,d,dv] and z [B,H,d] are updated in
 * place; q, k [B,H,d] and v [B,H,dv] are in `dtype`; out [B,H,dv] is fp32.
 * Needs no workspace.
 */
LA_API la_status la_decode_step(float* S, float* z, const void* q, const void* k, const void* v,
                         float* out, int64_t B, int64_t H, int d, int dv, int feature_map,
                         const float* gamma, int dtype, la_stream_t stream);

/*
 * Causal forward with a per-key-channel decay (GLA):
 *     S_t = diag(alpha_t) S_{t-1} + phi(k_t) v_t^T,  z_t = alpha_t o z_{t-1} + phi(k_t),
 *     o_t = phi(q_t)^T S_t / phi(q_t)^T z_t   (o_t = phi(q_t)^T S_t for LA_FM_NONE)
 * ["Efficient Attention Variants", section 7.2 GLA: alpha_t scales row i of
 * the state and is broadcast along the values].  alpha [B,H,N,d] is fp32
 * device memory with every entry in (0, 1] (data-dependent gates computed by
 * the caller; an exact 0 is not supported).  Runs on the CUDA cores in fp32;
 * workspace: la_gla_workspace_size() bytes, 256-byte aligned.  Other
 * arguments as for la_forward.
 */
LA_API size_t la_gla_workspace_size(int64_t B, int64_t H, int64_t N, int d, int dv);
LA_API la_status la_forward_gla(const void* q, const void* k, const void* v, const float* alpha,
                                float* out, int64_t B, int64_t H, int64_t N, int d, int dv,
                                int feature_map, int dtype, void* workspace,
                                size_t workspace_bytes, la_stream_t stream);

/*
 * One decode step with a per-key-channel decay alpha [B,H,d] (fp32, in
 * (0, 1]): S <- diag(alpha) S + phi(k) v^T, z <- alpha o z + phi(k), then the
 * read, as la_decode_step.
 */
LA_API la_status la_decode_step_gla(float* S, float* z, const void* q, const void* k,
                                    const void* v, const float* alpha, float* out, int64_t B,
                                    int64_t H, int d, int dv, int feature_map, int dtype,
                                    la_stream_t stream);

/*
 * The state before part `upto` of a sequence split into `nparts` consecutive
 * parts (sequence parallelism, "Linear Attention and SSM", LASP-2 section):
 * given each part's own final state from a zero start, U_p = (S_parts[p],
 * z_parts[p]) as la_state returns it, and the parts' token counts
 * part_len[p] (HOST array), computes
 *     P_0 = 0,   P_{p+1} = gamma^(part_len[p]) P_p + U_p,   out = P_upto
 * into S_out [B,H,d,dv] and z_out [B,H,d] (fp32).  S_parts is
 * [nparts][B,H,d,dv] and z_parts [nparts][B,H,d] (fp32, device), e.g. the
 * result of an all-gather of every rank's U_p.  la_forward_with_state from
 * (S_out, z_out) then gives the rank's outputs.  nparts <= 256; gamma as for
 * la_forward (host, H floats, or NULL).
 */
LA_API la_status la_state_prefix(const float* S_parts, const float* z_parts, int nparts,
                                 const int64_t* part_len, int upto, float* S_out, float* z_out,
                                 int64_t B, int64_t H, int d, int dv, const float* gamma,
                                 la_stream_t stream);

/*
 * Positive random features (Performer, FAVOR+): for each of `rows` rows u of
 * x [rows, d] (in_dtype) and the r rows w_j of w [r, d] (fp32, Gaussian,
 * drawn by the caller -- i.i.d. or in orthogonal blocks),
 *     x' = u / d^(1/4),   out[row, j] = exp(w_j . x' - |x'|^2 / 2) / sqrt(r)
 * written to out [rows, r] in out_dtype.  phi(q) . phi(k) is then an unbiased
 * estimate of exp(q . k / sqrt(d)) ["Efficient Attention Variants", section 6
 * Performer]; passing the features of q and k to la_forward with
 * LA_FM_IDENTITY_NORM (feature dimension r, r in {32, 64, 128}) gives
 * linear attention with that kernel.  d <= 128, r <= 256; all pointers are
 * device pointers, 16-byte aligned.
 */
LA_API la_status la_favor_features(const void* x, const float* w, void* out, int64_t rows, int d,
                                   int r, int in_dtype, int out_dtype, la_stream_t stream);

/*
 * la_forward without a workspace argument, for callers that cannot allocate
 * device memory (the pages have no counterpart: this is a deployment
 * convenience).  Typical such callers are a plugin running inside a host
 * application whose memory pool owns all device memory and forbids other
 * allocations, and latency-critical serving code that must not call
 * cudaMalloc / cudaFree because those calls can synchronise the whole device.
 *
 * Scratch comes from a fixed array of LA_NOALLOC_SCRATCH_BYTES compiled into
 * the library's device image; every GPU that loads the library keeps that
 * much memory reserved until the process exits.  Requests whose
 * la_forward_workspace_size() exceeds it return LA_ERR_TOO_LARGE before
 * anything is enqueued.  Nothing is allocated or freed by this call.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  All calls share the one array and it keeps
 * the previous call's contents (the forward clears what must start at zero
 * itself), so two calls whose work overlaps on the GPU -- on different
 * streams, or from different host threads -- race on it and give wrong
 * results: serialise them.  All other arguments and results are exactly
 * those of la_forward.
 */
#define LA_NOALLOC_SCRATCH_BYTES (64u << 20)
LA_API la_status la_forward_noalloc(const void* q, const void* k, const void* v, float* out,
                                    int64_t B, int64_t H, int64_t N, int d, int dv, int causal,
                                    int feature_map, const float* gamma, int dtype,
                                    la_stream_t stream);

/*
 * Diagnostic: total number of kernels this library has launched in this
 * process (all devices, all threads).  The difference across a region counts
 * the library's launches inside it.
 */
LA_API uint64_t la_launch_count(void);

/*
 * TEST HOOK, not for production use: exercises the give-up path of the
 * single-pass tensor-core forward, whose CTAs wait on one another's published
 * segment states.  wait_ns (> 0) replaces the 2 s limit of any single wait in
 * that kernel; withheld_segment (>= 0) is a segment ticket (the tickets of a
 * launch are numbered segment-major over the B*H sequences) whose aggregate
 * and exclusive prefix are computed but never published, so that the
 * look-backs of its successors run out of time; -1 withholds nothing.  The
 * setting applies to later launches on the current device until changed;
 * la_debug_set_tc_faults(2000000000, -1) restores the library's behaviour.
 * A launch whose waits ran out records LA_ERR_TIMEOUT (la_get_device_status),
 * every CTA drains its own copies and MMAs, frees its tensor memory and
 * exits; the context stays usable.
 */
LA_API la_status la_debug_set_tc_faults(uint64_t wait_ns, int withheld_segment);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word: LA_OK, LA_ERR_TIMEOUT or LA_ERR_DEVICE_CHECK (or LA_ERR_CUDA if the
 * synchronisation itself failed).
 */
LA_API la_status la_get_device_status(la_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */
