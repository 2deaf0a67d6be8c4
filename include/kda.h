/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention forward pass.
 *
 * The operation (one independent recurrence per sequence n and head h; the
 * state S is a K x V matrix, K = V = 128):
 *
 *   gate   gl[t,c] = lower_bound * sigmoid(exp(A_log[h]) * (g[t,h,c] + dt_bias[h,c]))
 *   decay  alpha_t = exp(gl[t,:])                  (per channel, in (exp(lower_bound), 1))
 *   write  b_t     = sigmoid(beta[t,h])
 *   state  S_t     = (I - b_t k_t k_t^T) Diag(alpha_t) S_{t-1} + b_t k_t v_t^T
 *   output o_t     = scale * S_t^T q_t
 *
 * Sources: "Moonshot AI Rilis FlashKDA" (captivela.com): the forward pass
 * takes q, k, v, the pre-activation gate g, beta logits, scale, out, A_log,
 * dt_bias and lower_bound; sigmoid is applied to beta inside the kernel;
 * initial and final states are optional and may be bf16 or fp32; q, k, v, g
 * are bf16 [B,T,H,K|V], beta bf16 [B,T,H], A_log / dt_bias / lower_bound fp32;
 * cu_seqlens selects variable-length batching; only K = V = 128.
 * "Moonshot AI Open-Sources FlashKDA" (alphasignal.ai), "Why KDA?": KDA is
 * Gated DeltaNet with channel-wise gating.  The pages print no formula: the
 * recurrence above is the gated delta rule with a diagonal decay, and the
 * gate formula is the reading that makes lower_bound the lower bound of the
 * per-token log-decay.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers (kda_fwd_host: HOST pointers),
 *     row-major with the last dimension contiguous, owned by the caller.
 *     The library keeps no pointer after a call returns.
 *   - Returns KDA_OK (0) or a negative kda_status.  Argument checks run on the
 *     host before anything is launched; a rejected call launches nothing and
 *     writes nothing.
 *   - kda_fwd is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronises.  Errors found on the device
 *     (a malformed cu_seqlens) are recorded in a per-device error word and
 *     reported by kda_fwd_get_error.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the optional recurrent states. */
typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_NULL = -1,            /* a required pointer is NULL                        */
    KDA_ERR_SHAPE = -2,           /* B, T, H, num_seqs inconsistent or out of range    */
    KDA_ERR_UNSUPPORTED_DIM = -3, /* K != 128 or V != 128                              */
    KDA_ERR_ALIGN = -4,           /* q, k, v, g or out not 16-byte aligned             */
    KDA_ERR_DTYPE = -5,           /* state dtype is neither KDA_BF16 nor KDA_F32       */
    KDA_ERR_LAUNCH = -6,          /* a kernel launch failed                            */
    KDA_ERR_DEVICE_TIMEOUT = -7,  /* a bounded device-side wait gave up                */
    KDA_ERR_BAD_SEQLENS = -8,     /* cu_seqlens not 0 .. T non-decreasing (device)     */
    KDA_ERR_ARCH = -9,            /* current device is not compute capability 10.3     */
    KDA_ERR_ALLOC = -10,          /* workspace allocation failed                       */
    KDA_ERR_CUDA = -11,           /* another CUDA runtime error                        */
    KDA_ERR_ARG = -12,            /* scale or lower_bound outside the supported range  */
    KDA_ERR_ALIAS = -13,          /* out overlaps an input, or states alias unsafely   */
    KDA_ERR_SCRATCH_LIMIT = -14,  /* kda_fwd_noalloc: num_seqs > KDA_NOALLOC_MAX_SEQS   */
    KDA_ERR_SEGMENTS = -15        /* kda_fwd_segments: num_segments not possible       */
} kda_status;

/*
 * kda_fwd -- KDA forward (prefill) pass.
 *
 *   q, k, g     bf16 [B, T, H, K]        v, out   bf16 [B, T, H, V]
 *               q and k are used as given (not normalised).  The kernel forms
 *               k * 2^-G with G down to 16 * lower_bound / ln 2 per chunk, so a
 *               key component must stay below 2^(128 + 16 * lower_bound / ln 2)
 *               in magnitude (about 10 at lower_bound = -5.4, 6,000 at -5)
 *               for that factor to stay finite; unit-norm keys always do.
 *               v enters a tensor-core product as fp16: its components must stay
 *               below 65,504 in magnitude.
 *   beta        bf16 [B, T, H]           logits; sigmoid is applied inside
 *   scale       multiplies the output    (finite)
 *   A_log       fp32 [H]                 dt_bias  fp32 [H, K]
 *   lower_bound fp32 scalar, in [-5.4, 0]: the per-token log-decay lies in
 *               [lower_bound, 0]; with 16-token chunks the in-chunk decay
 *               factors 2^(+-G) then stay within 2^124.6 of 1, inside the range
 *               of normal fp32 numbers (KDA_ERR_ARG outside it)
 *   initial_state  NULL (zero state) or [N, H, K, V] of initial_state_dtype
 *   final_state    NULL (not written) or [N, H, K, V] of final_state_dtype
 *               State element [n][h][i][j] is S[i][j]: row i = key channel,
 *               column j = value channel.  fp32 -> bf16 writes round to
 *               nearest even.  initial_state and final_state may be the
 *               same buffer if their dtypes match.
 *   cu_seqlens  NULL: B sequences of T tokens, N = B.
 *               Else int32 [num_seqs + 1] DEVICE array of token offsets,
 *               0 = cu[0] <= cu[1] <= ... <= cu[num_seqs] = T, with B == 1
 *               and N = num_seqs.  Zero-length sequences are allowed (their
 *               final state is their initial state).  Checked on the device:
 *               a malformed array sets KDA_ERR_BAD_SEQLENS in the error word
 *               and the call then writes neither out nor final_state.
 *   B, T, H     B >= 1, T >= 0, H >= 1; B*T*H*128 < 2^31
 *   K, V        must both be 128 (KDA_ERR_UNSUPPORTED_DIM otherwise)
 *   stream      cudaStream_t to run on
 *
 * q, k, v, g and out must be 16-byte aligned; out must not overlap any input.
 * kda_fwd is kda_fwd_segments with num_segments = 0: a long fixed-length call
 * whose B*H recurrences leave most SMs idle is cut into segments that run side
 * by side (see kda_fwd_segments); other calls run one pass.  A varlen call with
 * more (sequence, head) recurrences than SMs, whose sequences average at most 256
 * tokens, runs one persistent CTA per SM that takes the recurrences longest first
 * from a device counter and carries its pipeline from one to the next (results
 * bit-identical to one CTA per recurrence).  Varlen calls take
 * kda_fwd_workspace_bytes() of scratch (the longest-first sequence order, a
 * validity flag and that counter), and
 * split calls that many bytes of fp32 segment states, from the stream-ordered
 * allocator (cudaMallocAsync / cudaFreeAsync on `stream`); one-pass
 * fixed-length calls take none.  The call does not synchronise.  The first call on a device
 * raises the release threshold of that device's default memory pool to its
 * maximum, so that freed scratch stays in the pool instead of going back to
 * the driver at every synchronisation (a process-wide setting of that pool).
 */
int kda_fwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
            float scale, void* out, const float* A_log, const float* dt_bias,
            float lower_bound, const void* initial_state, int initial_state_dtype,
            void* final_state, int final_state_dtype, const int32_t* cu_seqlens,
            int num_seqs, int B, int T, int H, int K, int V, void* stream);

/*
 * kda_fwd_segments -- kda_fwd with the sequence split chosen by the caller.
 *
 * The recurrence is affine in the state: over a segment of tokens,
 * S_end = P S_start + B, with P the product of the segment's transitions
 * (I - b_t k_t k_t^T) Diag(alpha_t) and B the end state of the segment run from
 * a zero state.  A fixed-length call cut into s segments (the n = ceil(T / 16)
 * chunks of a sequence spread evenly: segment j holds chunks floor(j n / s) ..
 * floor((j + 1) n / s) - 1) runs in two windows of one segment's length:
 * window 0 runs segment 0 from the initial state and, for each middle segment,
 * its B (from a zero state) and its P (from the identity state with zero
 * values); a combine kernel chains S_start(j) = P_{j-1} S_start(j-1) + B_{j-1} in
 * fp32; window 1 runs segments 1 .. s-1 from their S_start.  That is 2s - 3
 * recurrences per (sequence, head) in window 0, s - 1 in window 1, for about
 * 2/s of the one-pass time when they fit on the SMs.  This is the chunk-parallel
 * stage of the pages' two-stage split ("Moonshot AI Open-Sources FlashKDA",
 * "What makes the kernel fast": the sequential stage has far less parallelism
 * than the token-parallel one), applied to whole segments.
 *
 *   num_segments  0: automatic -- the largest s whose window-0 recurrences,
 *                    (2s - 3) B H, fit on the device's SMs, with at least 1,024
 *                    tokens per segment; one pass when that gives s < 3
 *                 1: one pass (the same arithmetic as kda_fwd_noalloc)
 *                 s >= 2: s segments, at most ceil(T / 16) (KDA_ERR_SEGMENTS
 *                    otherwise, and for num_segments > 1 with cu_seqlens, which
 *                    always runs one pass)
 *
 * Other arguments, layouts and errors as kda_fwd.  Split and one-pass results
 * differ by rounding only (both are checked against the fp64 oracle); each is
 * deterministic.  Scratch: kda_fwd_workspace_bytes for the automatic choice;
 * for s segments 65,536 * B * H * (5s - 7) + 4,096 * H bytes, each of its four
 * parts rounded up to 256 (fp32 initial and end states of every segment's runs
 * and 16 zero rows of values).
 */
int kda_fwd_segments(const void* q, const void* k, const void* v, const void* g,
                     const void* beta, float scale, void* out, const float* A_log,
                     const float* dt_bias, float lower_bound, const void* initial_state,
                     int initial_state_dtype, void* final_state, int final_state_dtype,
                     const int32_t* cu_seqlens, int num_seqs, int B, int T, int H, int K,
                     int V, int num_segments, void* stream);

/*
 * kda_fwd_host -- the same operation on HOST buffers (end-to-end entry point).
 *
 * Same arguments and layouts as kda_fwd, except that every pointer
 * (cu_seqlens included) is a host pointer; pinned memory makes the copies
 * asynchronous.  The call allocates device buffers on `stream`, copies the
 * inputs host -> device, runs kda_fwd, copies out (and final_state)
 * device -> host, frees the buffers and synchronises `stream` before
 * returning, so the outputs are ready on return.  cu_seqlens is validated on
 * the host (KDA_ERR_BAD_SEQLENS) before anything is copied.  A fixed-length
 * call with B == 1 and T >= 2048 runs in token blocks (each half of the
 * tokens still left, in whole 16-token chunks, down to 256 tokens; the state
 * carried in fp32 on the device) so that the copies in and out overlap the
 * kernel on two extra streams; its results are bit-identical to one
 * one-pass call on the same data (kda_fwd_segments with num_segments = 1,
 * which is kda_fwd whenever kda_fwd does not split the sequence).
 */
int kda_fwd_host(const void* q, const void* k, const void* v, const void* g,
                 const void* beta, float scale, void* out, const float* A_log,
                 const float* dt_bias, float lower_bound, const void* initial_state,
                 int initial_state_dtype, void* final_state, int final_state_dtype,
                 const int32_t* cu_seqlens, int num_seqs, int B, int T, int H, int K, int V,
                 void* stream);

/*
 * kda_bwd -- the backward pass: gradients of a scalar loss L with respect to the
 * forward pass's inputs, given dL/d(out) and, optionally, dL/d(final state).
 *
 * No counterpart on the pages (the pages' library is forward-only: "Moonshot AI
 * Open-Sources FlashKDA", "Limitations before you integrate").  It differentiates
 * the recurrence above exactly (reverse order of its steps, token by token, in fp32):
 * with x = exp(A_log)(g + dt_bias), a = exp(lower_bound sigmoid(x)), b = sigmoid(beta),
 * S' = Diag(a) S, r = S'^T k, d = b (v - r), S = S' + k d^T, o = scale S^T q.
 *
 *   inputs      q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state
 *               (+ dtype), cu_seqlens, num_seqs, B, T, H, K, V: as kda_fwd
 *   d_out       bf16 [B, T, H, V]: dL/d(out)
 *   d_final_state  fp32 [N, H, K, V]: dL/d(final state), or NULL (zero)
 *   outputs (fp32): dq, dk, dg [B, T, H, K]; dv [B, T, H, V]; dbeta [B, T, H];
 *               dA_log [H]; ddt_bias [H, K] (summed over all sequences and tokens);
 *               d_initial_state [N, H, K, V] or NULL (not written); it is the
 *               gradient with respect to the initial state also when none is given.
 *
 * Outputs must not overlap the inputs or each other (KDA_ERR_ALIAS); q, k, v, g,
 * d_out, dv and d_initial_state must be 16-byte aligned.  Scratch:
 * kda_bwd_workspace_bytes() from the stream-ordered allocator (state checkpoints every
 * 8 tokens, each token's d and v - r, per-slice partial sums; about 21 KB per token
 * and head, so one call of more than ~12 M token-heads does not fit in a GB300's
 * memory and returns KDA_ERR_ALLOC; split such a call over the sequence with
 * d_final_state and d_initial_state carried between the parts).  Asynchronous on `stream`; a malformed cu_seqlens sets KDA_ERR_BAD_SEQLENS
 * in the error word and writes nothing.  Results are deterministic (fixed summation
 * order).  The work: 8 CTAs per (sequence, head), each owning 16 value columns of the
 * state, on CUDA cores; then a kernel that sums their partial dq, dk and decay
 * gradients and applies the activations, and one that sums dA_log and ddt_bias.
 */
int kda_bwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
            float scale, const float* A_log, const float* dt_bias, float lower_bound,
            const void* initial_state, int initial_state_dtype, const void* d_out,
            const float* d_final_state, float* dq, float* dk, float* dv, float* dg,
            float* dbeta, float* dA_log, float* ddt_bias, float* d_initial_state,
            const int32_t* cu_seqlens, int num_seqs, int B, int T, int H, int K, int V,
            void* stream);

/* Bytes of scratch kda_bwd takes from the stream-ordered allocator (host-only). */
size_t kda_bwd_workspace_bytes(int B, int T, int H, int num_seqs, int varlen);

/*
 * kda_fwd_get_error -- synchronise `stream`, then return and clear the current
 * device's error word: KDA_OK, KDA_ERR_BAD_SEQLENS or KDA_ERR_DEVICE_TIMEOUT
 * (or KDA_ERR_CUDA if the synchronisation itself failed).  There is one word
 * per device, shared by every call on it whatever its stream: it keeps the
 * first error any kernel recorded since the last read, and a call still
 * running on another stream may set it after this read.
 * KDA_ERR_DEVICE_TIMEOUT: a wait between the kernel's pipeline stages ran past
 * its bound (KDA_SPIN_LIMIT SM cycles, about 2 s with the default build); the
 * kernel then stops at its next wait, after its own asynchronous copies and
 * tensor-core operations have completed, and returns.  out and final_state are
 * then undefined for that call; the device and later calls are unaffected.
 */
int kda_fwd_get_error(void* stream);

/* Human-readable name of a kda_status value (static string, never NULL). */
const char* kda_status_string(int status);

/* The cudaError_t value (as an int) of the CUDA runtime failure behind the most
 * recent KDA_ERR_LAUNCH, KDA_ERR_ALLOC or KDA_ERR_CUDA returned to the calling
 * host thread (cudaGetErrorString gives its text); 0 if there was none.
 * Successful calls leave it unchanged.  Host-only, no CUDA call. */
int kda_last_cuda_error(void);

/* Bytes of scratch memory kda_fwd takes from the stream-ordered allocator for
 * the given problem (0 for an empty problem).  Varlen: host-only, no CUDA call.
 * Fixed length: reads the current device's SM count, on which the automatic
 * sequence split depends (0 when no device can be queried). */
size_t kda_fwd_workspace_bytes(int B, int T, int H, int num_seqs, int varlen);

/*
 * kda_fwd_noalloc -- kda_fwd for callers that cannot allocate device memory.
 *
 * No counterpart on the pages: this entry point exists for users of the
 * library whose device memory is not theirs to allocate from -- a serving
 * runtime or framework that reserves its whole memory budget up front and
 * owns every byte through its own allocator, or a hot loop that must not
 * pay for (or synchronise on) an allocation.  kda_fwd takes a small scratch
 * buffer from cudaMallocAsync on varlen calls; this variant takes it from a
 * fixed array in the library's own device memory instead, and calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * Same arguments, layouts and checks as kda_fwd (the caller still passes
 * every input and output buffer).  It always runs one pass, so its results are
 * those of kda_fwd_segments with num_segments = 1: kda_fwd's own, except on the
 * long fixed-length calls that kda_fwd splits into segments (whose scratch
 * would need an allocation).  Plus:
 *   - The scratch is a static device array sized for KDA_NOALLOC_MAX_SEQS
 *     sequences (about 256 KB).  Every GPU that loads this library holds one
 *     copy of it until the process exits.  Varlen calls with
 *     num_seqs > KDA_NOALLOC_MAX_SEQS return KDA_ERR_SCRATCH_LIMIT and launch
 *     nothing.  Fixed-length calls use no scratch.
 *   - The first varlen call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it.
 *   - All calls on a device share the one array.  Each call rewrites the part
 *     it uses before reading it (nothing needs to start at zero), but calls
 *     whose work overlaps on the GPU -- on different streams, or from
 *     different host threads -- race on it: order them on one stream or
 *     synchronise between them.
 */
#define KDA_NOALLOC_MAX_SEQS 65536
int kda_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                    const void* beta, float scale, void* out, const float* A_log,
                    const float* dt_bias, float lower_bound, const void* initial_state,
                    int initial_state_dtype, void* final_state, int final_state_dtype,
                    const int32_t* cu_seqlens, int num_seqs, int B, int T, int H, int K, int V,
                    void* stream);

/*
 * kda_decode -- one decode step: a single new token for each of N sequences,
 * applied to their states (the incremental decoding that the final state of a
 * prefill feeds: "FlashKDA" (productcool.com), "Main Features").  The result
 * equals kda_fwd on B = N sequences of T = 1 token with these states; per
 * (n, h) it reads the state once and writes it once, so its cost is the state
 * traffic (128 KB per (n, h) with fp32 states in and out).
 *
 *   q, k, g     bf16 [N, H, K]   (one token per sequence; [N, 1, H, K] in kda_fwd's layout)
 *   v, out      bf16 [N, H, V]
 *   beta        bf16 [N, H]      logits; sigmoid is applied inside
 *   scale, A_log, dt_bias, lower_bound   as for kda_fwd (same gate, same ranges)
 *   state_in    NULL (zero state) or [N, H, K, V] of state_in_dtype
 *   state_out   NULL (not written) or [N, H, K, V] of state_out_dtype; the
 *               usual call passes the same buffer as state_in (same dtype) to
 *               update the states in place
 *   N >= 0, H >= 1, N*H < 2^31; K = V = 128
 *
 * Device pointers, owned by the caller; q, k, v, g, out and both states must be
 * 16-byte aligned; out must not overlap an input or state_out, and state_in and
 * state_out must be the same buffer or disjoint.  Asynchronous on `stream`; no
 * scratch memory; argument errors as for kda_fwd (nothing is launched).
 */
int kda_decode(const void* q, const void* k, const void* v, const void* g, const void* beta,
               float scale, void* out, const float* A_log, const float* dt_bias,
               float lower_bound, const void* state_in, int state_in_dtype, void* state_out,
               int state_out_dtype, int N, int H, int K, int V, void* stream);

/* ---- launch accounting (for measurement; off by default) ------------------
 *
 * kda_profile_enable(1) makes every later kda_fwd, kda_fwd_noalloc and
 * kda_decode call (and the kda_fwd calls that kda_fwd_host makes) record a CUDA
 * event before and after each of its kernel launches, on the launch stream; enable(0)
 * stops recording.  Enabling clears the totals.  kda_profile_read
 * synchronises on the recorded events and returns, per kernel id
 * (KDA_KERNEL_*), the summed device time in milliseconds and the number of
 * launches since the last enable.  Arrays must hold KDA_NUM_KERNELS entries.
 * Returns KDA_OK, or KDA_ERR_CUDA. */
enum {
    KDA_KERNEL_SEQMAP = 0,
    KDA_KERNEL_FUSED = 1,
    KDA_KERNEL_DECODE = 2,
    KDA_KERNEL_COMBINE = 3,
    KDA_KERNEL_SEGPREP = 4,
    KDA_KERNEL_SEGFINAL = 5,
    KDA_KERNEL_BWD = 6,
    KDA_KERNEL_BWD_FINISH = 7,
    KDA_KERNEL_BWD_REDUCE = 8,
    KDA_NUM_KERNELS = 9
};
int kda_profile_enable(int on);
int kda_profile_read(double* total_ms, long long* launches);
const char* kda_kernel_name(int kernel_id);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H_ */
