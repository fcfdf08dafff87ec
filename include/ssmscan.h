/*
 * ssmscan.h -- C ABI of libssmscan, the Mamba2 selective-state scan on sm_103a.
 *
 * The operation (for every sequence i, head h, head-dim row p and token t of
 * the sequence, in token order; g(h) = h / (n_heads / n_groups)):
 *
 *     dA          = exp(dt[t,h] * A[h])
 *     S[h,p,:]    = dA * S[h,p,:] + dt[t,h] * x[t,h,p] * B[t,g(h),:]
 *     y[t,h,p]    = S[h,p,:] . C[t,g(h),:] + D[h] * x[t,h,p]
 *
 * S is the fp32 recurrent state of sequence i.  It lives in slot i of
 * state_slots and persists between calls.  Defined by:
 *   - "The llama journey", Day 14: the ssm_scan_f32_group kernel body (decay
 *     exp(dt*A) with a scalar A per head, input term B*x*dt, y = state . C
 *     from the state that already includes token t, one B/C per group of
 *     contiguous heads);
 *   - "The llama journey", Day 12: the SSM_SCAN tensor table (state
 *     [seq][head][dim][d_state]; x [token][head][dim]; dt [token][head];
 *     B, C [token][group][d_state]);
 *   - "keep the Mamba2 scan state in registers, stage tokens by chunk"
 *     (gllm PR 90), "What changes" and "Testing": batches mix fresh and
 *     resuming sequences; state is fp32 and moves between slot and registers.
 * The skip term D[h] * x[t,h,p] is part of the operation.  dt is used as given
 * (no softplus or bias is applied here).
 *
 * Memory and ownership (all calls):
 *   - Every pointer is CUDA device memory owned by the caller.  The library
 *     allocates nothing and never synchronises the stream; work is enqueued on
 *     `stream` (a cudaStream_t passed as void*; NULL = the legacy default
 *     stream) and its execution errors surface at the caller's next sync.
 *   - Tokens of all sequences are packed: sequence i owns tokens
 *     [seq_starts[i], seq_starts[i] + seq_lens[i]) of the n_tokens rows of
 *     x, dt, B, C and y.  Tokens owned by no sequence are neither read nor
 *     written.
 *   - resume_flags[i] != 0: start from slot i.  == 0: start from zero; the
 *     slot's old contents are never read (they may be NaN).  After the call
 *     slot i holds the state after the sequence's last token.  A zero-length
 *     sequence writes no y; a fresh one still leaves a zero slot.
 *   - Layouts (row-major, contiguous, fp32 unless stated):
 *       state_slots [n_seqs][n_heads][head_dim][d_state]   in/out
 *       x           [n_tokens][n_heads][head_dim]
 *       dt          [n_tokens][n_heads]
 *       A, D        [n_heads]
 *       B, C        [n_tokens][n_groups][d_state]
 *       y           [n_tokens][n_heads][head_dim]               out
 *       seq_starts, seq_lens, resume_flags   int32 [n_seqs], device memory
 *   - y must not overlap any input; inputs are read only.
 *   - Alignment: state_slots, B and C 16-byte aligned (the state moves as
 *     128-bit vectors); the others 4-byte aligned.
 *
 * Preconditions checked only on the device metadata's request: sequence
 * ranges must lie in [0, n_tokens) and not overlap.  With the environment
 * variable SSM_SCAN_CHECK=1 the library copies the metadata to the host,
 * synchronises and rejects bad ranges with SSM_ERR_INVALID_ARG (debug only).
 *
 * Errors: host-checkable faults return before any launch:
 *   SSM_ERR_INVALID_ARG  null pointer, negative size, n_heads % n_groups != 0,
 *                        misaligned pointer, bad tuning value;
 *   SSM_ERR_UNSUPPORTED  d_state not a multiple of 4, d_state > 1024;
 *   SSM_ERR_CUDA         a CUDA call or launch failed (cudaGetLastError);
 *   SSM_ERR_TIMEOUT      a bounded device wait gave up (the pipelined
 *                        tensor-core kernels: the segments' state pass and the
 *                        SSD chunk-state and output kernels).  Each such wait
 *                        polls an mbarrier a bounded number of times (seconds);
 *                        on giving up the kernel sets a status word in the
 *                        workspace, waits for its copies and products in
 *                        flight, frees its tensor memory and returns, so the
 *                        context stays usable.  The word is read back (and this
 *                        code returned) only under SSM_SCAN_CHECK=1; the library
 *                        never synchronises otherwise.  Without that check the
 *                        failure shows in the outputs instead:
 *                          - a segmented ssm_scan_* call: y is NaN for every
 *                            owned token and every slot keeps the contents it
 *                            had before the call;
 *                          - ssm_scan_ssd: when the chunk states gave up, y is
 *                            NaN for every owned token and the slots keep their
 *                            contents; when an output block gave up, y is NaN
 *                            over that block's chunk and heads (the slots hold
 *                            the final states).
 *                        SSM_SCAN_TEST_FAIL_WAITS=1 makes those waits give up
 *                        at once (tests of this path).
 * n_seqs == 0 is a successful no-op.
 */
#ifndef SSMSCAN_H
#define SSMSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = -1,
    SSM_ERR_UNSUPPORTED = -2,
    SSM_ERR_CUDA = -3,
    SSM_ERR_TIMEOUT = -4
} ssm_status;

/* Kernel path selection for ssm_scan_tuned. */
enum {
    SSM_PATH_AUTO = 0,           /* decode when n_tokens == n_seqs, else prefill */
    SSM_PATH_DECODE = 1,         /* warp-per-row kernel; correct for any lengths */
    SSM_PATH_PREFILL = 2,        /* chunk-staged kernel, decay-rescaled state with packed
                                    fp32x2 FMAs; correct for any lengths */
    SSM_PATH_PREFILL_DIRECT = 3  /* chunk-staged kernel stepping S itself (one multiply
                                    more per state element); correct for any lengths */
};

/*
 * Launch-shape overrides for ssm_scan_tuned.  Zero in any field means "pick
 * automatically".  Every combination that is accepted computes the same
 * result (up to float association); unsupported values give
 * SSM_ERR_INVALID_ARG.
 *   path             SSM_PATH_*
 *   lanes_per_row    lanes of a warp that share one state row: 1,2,4,8,16,32
 *   rows_per_thread  state rows each lane holds (a power of two, <= lanes_per_row:
 *                    up to 8 on SSM_PATH_PREFILL, up to 4 on the other paths;
 *                    automatic on SSM_PATH_PREFILL: about 16 state elements of a
 *                    row per lane and 4 rows)
 *   rows_per_cta     prefill: state rows per thread block (a multiple of the
 *                    rows one warp holds, at most 256 threads, 224 on
 *                    SSM_PATH_PREFILL, whose blocks add a producer warp except
 *                    where they are exactly four warps of 8 lanes x 4 rows: those
 *                    stage their own chunks, three blocks per SM); decode: ignored
 *   chunk_tokens     prefill: tokens staged in shared memory per chunk (1..256;
 *                    at most 32 on SSM_PATH_PREFILL, automatic 16 there, 32 on
 *                    SSM_PATH_PREFILL_DIRECT)
 *   ctas_per_sm      decode: if > 0, the grid is capped at this many blocks
 *                    per SM and warps loop over the remaining rows
 *   segment_tokens   SSM_PATH_PREFILL with a workspace (ssm_scan_ws): length of
 *                    the time segments long sequences are cut into (a multiple
 *                    of the chunk; an automatic chunk is the largest of 16, 8,
 *                    ... that divides it); 0 = automatic, < 0 = never segment
 *   segment_state    how the state pass of the time segments runs
 *                    (SSM_SEGMENT_STATE_*); ignored without segments
 */
enum {
    SSM_SEGMENT_STATE_AUTO = 0,   /* the tensor cores where d_state <= 128, head_dim <= 256 and
                                     a multiple of 4, and x 16-byte aligned; else the sequential
                                     kernel */
    SSM_SEGMENT_STATE_FP32 = 1,   /* the sequential kernel's state-only mode (fp32 FMAs) */
    SSM_SEGMENT_STATE_TENSOR = 2  /* the segment's state as a matrix product over its tokens on
                                     the tensor cores, operands split into two TF32 parts
                                     (hi*hi + hi*lo + lo*hi, fp32 accumulation: fp32-level
                                     accuracy); SSM_ERR_UNSUPPORTED where the shapes do not fit */
};
typedef struct {
    int path;
    int lanes_per_row;
    int rows_per_thread;
    int rows_per_cta;
    int chunk_tokens;
    int ctas_per_sm;
    int segment_tokens;
    int segment_state;
} ssm_scan_tuning;

/*
 * The scan.  Advances every sequence of the batch through its tokens, writes
 * y for each of them and leaves each sequence's final state in its slot.
 * n_tokens is the number of packed token rows of x, dt, B, C and y.
 */
int ssm_scan(float *state_slots, const float *x, const float *dt,
             const float *A, const float *B, const float *C, const float *D,
             float *y, const int32_t *seq_starts, const int32_t *seq_lens,
             const int32_t *resume_flags, int n_seqs, int n_tokens,
             int n_heads, int head_dim, int d_state, int n_groups,
             void *stream);

/* The same operation with explicit launch-shape choices (tests, tuning). */
int ssm_scan_tuned(float *state_slots, const float *x, const float *dt,
                   const float *A, const float *B, const float *C,
                   const float *D, float *y, const int32_t *seq_starts,
                   const int32_t *seq_lens, const int32_t *resume_flags,
                   int n_seqs, int n_tokens, int n_heads, int head_dim,
                   int d_state, int n_groups, const ssm_scan_tuning *tuning,
                   void *stream);

/*
 * Optional steps around the scan (all NULL / 0 = the plain scan).
 *   dt_bias, dt_softplus  Mamba2's discretisation of dt ("The llama journey",
 *       Day 14 kernel body; the decay-gate kernel of "ssm_gated_delta.cu"):
 *       v = dt[t,h] + dt_bias[h] (dt_bias NULL: no bias), then with dt_softplus
 *       nonzero the step is v for v > 20 and log1p(exp(v)) otherwise; that step
 *       replaces dt[t,h] everywhere in the recurrence above.  It is computed by
 *       a pass of its own into the first n_tokens*n_heads floats (rounded up to
 *       256 bytes) of the workspace, so these options need a workspace (see
 *       ssm_scan_ex_workspace_bytes); the scan kernels then read it as their
 *       step.  dt_bias: device, [n_heads] fp32, 4-byte aligned.
 *   state_snapshots  device, [n_tokens][n_heads][head_dim][d_state] fp32, out:
 *       row t receives the state right after token t for every token owned by a
 *       sequence, so accepting the first M tokens of a speculative run restores
 *       one contiguous [n_heads][head_dim][d_state] image (the rows of tokens
 *       owned by no sequence are not written).  16-byte aligned.
 *   gated_y, gate_z, norm_weight, norm_eps  Mamba2's gated RMSNorm after the
 *       scan, per (token, head) row of head_dim values:
 *       gated_y[t,h,p] = y[t,h,p] / sqrt(mean_p(y[t,h,:]^2) + norm_eps)
 *                        * norm_weight[p] * silu(gate_z[t,h,p]),
 *       silu(z) = z / (1 + exp(-z)), the weight shared by all heads (kernel 3
 *       of "ssm_gated_delta.cu").  gated_y, gate_z: device [n_tokens][n_heads]
 *       [head_dim] fp32; norm_weight: device [head_dim]; norm_eps > 0.  y is
 *       still written.  gated_y NULL: off (the other three are then ignored).
 *   launch_events, n_launch_events  timing of the call's kernels: an array of
 *       n_launch_events CUDA events (cudaEvent_t handles the caller created on
 *       the stream's device).  The call records launch_events[2k] on its stream
 *       right before its k-th kernel launch and launch_events[2k+1] right
 *       after it, while 2k+1 < n_launch_events, so cudaEventElapsedTime of a
 *       pair is that kernel's device time.  Launch order: the dt pass (with
 *       the dt options); then for ssm_scan_* the decode kernel, or the prefill
 *       kernel, or with time segments the plan, state-pass, combine and
 *       full-pass kernels; for ssm_scan_ssd the plan, chunk-state, state-pass
 *       and output kernels; then the gated RMSNorm (with gated_y), except
 *       where the rescaled prefill's last kernel writes it itself (its blocks
 *       then hold exactly one head each, as the automatic shape does at
 *       head_dim 64 and d_state 64 or 128, and z is 16-byte aligned).  NULL / 0:
 *       none; n_launch_events < 0, or > 0 with NULL events: SSM_ERR_INVALID_ARG;
 *       a failed record: SSM_ERR_CUDA.
 */
typedef struct {
    const float *dt_bias;
    int dt_softplus;
    float *state_snapshots;
    const float *gate_z;
    const float *norm_weight;
    float norm_eps;
    float *gated_y;
    void *const *launch_events;
    int n_launch_events;
} ssm_scan_options;

/*
 * The scan with tuning, options and workspace (each may be NULL / 0):
 * ssm_scan_ws plus the optional steps of ssm_scan_options.  With state
 * snapshots the call runs the decode kernel whatever the lengths (it steps
 * each sequence token by token with the state in registers and writes every
 * intermediate state; meant for the few tokens of a speculative verify step);
 * a tuning that asks for a prefill path then returns SSM_ERR_UNSUPPORTED.
 * Errors as for ssm_scan_ws, and SSM_ERR_INVALID_ARG for a misaligned option
 * pointer, norm_eps <= 0 with gated_y set, or dt options without a workspace
 * of at least the discretised step's bytes.  The workspace is used as by
 * ssm_scan_ws after that step's bytes.
 */
int ssm_scan_ex(float *state_slots, const float *x, const float *dt,
                const float *A, const float *B, const float *C, const float *D,
                float *y, const int32_t *seq_starts, const int32_t *seq_lens,
                const int32_t *resume_flags, int n_seqs, int n_tokens,
                int n_heads, int head_dim, int d_state, int n_groups,
                const ssm_scan_tuning *tuning, const ssm_scan_options *options,
                void *workspace, size_t workspace_bytes, void *stream);

/*
 * The scan with a caller-owned device workspace.  With a workspace the
 * prefill path may cut long sequences into time segments and run them in
 * parallel: a state-only pass per segment, a combine of the segment states
 * (S_in[k+1] = d_k S_in[k] + L_k, d_k the segment's decay prod exp(dt*A)),
 * then the full pass from each segment's incoming state.  This is the same
 * recurrence applied to whole segments; only float association changes.  The
 * state pass runs on the tensor cores where the shapes fit (see
 * tuning->segment_state): L_k unrolled into a sum over the segment's tokens,
 * sum_s dt_s exp(A sum_{r>s} dt_r) x_s B_s^T, with split TF32 operands.
 *   tuning          may be NULL
 *   workspace       device memory, 256-byte aligned, at least
 *                   ssm_scan_workspace_bytes(...) bytes for the same arguments
 *                   and tuning; NULL or too small: runs without segments
 *                   (SSM_ERR_INVALID_ARG if tuning->segment_tokens > 0)
 * The workspace is scratch: its contents are undefined afterwards and two
 * calls that overlap on the GPU must not share it.
 */
int ssm_scan_ws(float *state_slots, const float *x, const float *dt,
                const float *A, const float *B, const float *C, const float *D,
                float *y, const int32_t *seq_starts, const int32_t *seq_lens,
                const int32_t *resume_flags, int n_seqs, int n_tokens,
                int n_heads, int head_dim, int d_state, int n_groups,
                const ssm_scan_tuning *tuning, void *workspace,
                size_t workspace_bytes, void *stream);

/*
 * Bytes of workspace ssm_scan_ws uses for these sizes and tuning (NULL =
 * automatic) on the current device; 0 when it would not cut any sequence into
 * segments (for example decode batches) or the arguments are invalid.
 */
size_t ssm_scan_workspace_bytes(int n_seqs, int n_tokens, int n_heads,
                                int head_dim, int d_state, int n_groups,
                                const ssm_scan_tuning *tuning);

/*
 * The scan in chunked matrix form ("SSD") on the TF32 tensor cores.  The
 * gllm PR 90 page ("keep the Mamba2 scan state in registers, stage tokens by
 * chunk", "What changes" and "Not in this PR") names Mamba2's SSD
 * chunked-matmul algorithm as the way to parallelise prefill over time and
 * gives no algorithm; this form is the recurrence above unrolled over chunks
 * of `chunk` tokens of each sequence.  With a_t = sum_{s<=t in the chunk}
 * dt[s,h] A[h]:
 *     y_t   = exp(a_t) S_in.C_t + sum_{s<=t} exp(a_t - a_s) dt_s (C_t.B_s) x_s + D x_t
 *     S_out = exp(a_last) S_in + sum_s exp(a_last - a_s) dt_s x_s (x) B_s
 * and S_in of chunk k+1 is S_out of chunk k.  In exact arithmetic it equals
 * ssm_scan.  The contractions C B^T, (masked decay-weighted C B^T) x, S_in C^T
 * and x^T B round their operands to TF32 (10-bit mantissa, round to nearest)
 * and accumulate in fp32; the pass over chunks is fp32.  Expect
 * |y - y_exact| <= 5e-3 (1 + |y_exact|), not the 1e-4 of ssm_scan.
 *   chunk         tokens per chunk: 64 or 128 (0 = 128)
 *   workspace     device memory, 256-byte aligned, at least
 *                 ssm_scan_ssd_workspace_bytes(...) bytes for the same sizes
 *                 and chunk (chunk states [units][n_heads][head_dim][d_state]
 *                 fp32, units <= n_seqs + ceil(n_tokens / chunk), and room for
 *                 the discretised step of the dt options); scratch:
 *                 undefined afterwards, not shared by calls that overlap on
 *                 the GPU
 * Same arguments, layouts and metadata rules as ssm_scan, and also:
 *   - x and y 16-byte aligned;
 *   - head_dim a multiple of 16 and at most 128 (else SSM_ERR_UNSUPPORTED);
 *   - the chunk's shared-memory tiles must fit one block: SSM_ERR_UNSUPPORTED
 *     otherwise (for example d_state 1024; d_state up to 256 fits with
 *     chunk 64, up to 128 with chunk 128).
 * options: as for ssm_scan_ex (NULL = none); state snapshots are not
 * available in this form (SSM_ERR_UNSUPPORTED).
 * SSM_ERR_INVALID_ARG for a missing, misaligned or too small workspace or a
 * chunk other than 0, 64 or 128.
 */
int ssm_scan_ssd(float *state_slots, const float *x, const float *dt,
                 const float *A, const float *B, const float *C, const float *D,
                 float *y, const int32_t *seq_starts, const int32_t *seq_lens,
                 const int32_t *resume_flags, int n_seqs, int n_tokens,
                 int n_heads, int head_dim, int d_state, int n_groups,
                 int chunk, const ssm_scan_options *options, void *workspace,
                 size_t workspace_bytes, void *stream);

/*
 * Bytes of workspace ssm_scan_ex uses for these sizes, tuning and options
 * (NULL = none): the discretised step when dt options are set, plus what
 * ssm_scan_workspace_bytes reports (nothing with state snapshots); 0 for
 * invalid arguments or when none is needed.
 */
size_t ssm_scan_ex_workspace_bytes(int n_seqs, int n_tokens, int n_heads,
                                   int head_dim, int d_state, int n_groups,
                                   const ssm_scan_tuning *tuning,
                                   const ssm_scan_options *options);

/*
 * Bytes of workspace ssm_scan_ssd needs for these sizes and chunk (the same on
 * every device); 0 for invalid or unsupported arguments.
 */
size_t ssm_scan_ssd_workspace_bytes(int n_seqs, int n_tokens, int n_heads,
                                    int head_dim, int d_state, int n_groups,
                                    int chunk);

/*
 * Size of the scratch that ssm_scan_static keeps in device memory (32 MiB per
 * device, held from the library's load on that device until process exit).
 */
#define SSM_SCAN_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * The scan for callers that cannot allocate device memory (the pages have no
 * counterpart: it is a packaging choice of this library).  Some callers never
 * get to hand the library a workspace: a runtime without a device allocator,
 * a plugin whose host owns every allocation, a path that must not enter
 * cudaMalloc.  ssm_scan_static takes the same arguments as ssm_scan and runs
 * what ssm_scan_ws runs with an automatic plan, using instead a fixed scratch
 * array of SSM_SCAN_STATIC_SCRATCH_BYTES in device global memory that the
 * library owns.  It allocates nothing.
 *   - The first call on a device looks up the scratch's device address (a
 *     cudaGetSymbolAddress with that device current) and caches it; make that
 *     first call before any stream capture.  The cached address belongs to
 *     the device's context as it was then: a cudaDeviceReset while the
 *     library is loaded is not supported.
 *   - The stream must belong to the current device (SSM_ERR_INVALID_ARG
 *     otherwise), since the scratch address is looked up for that device.
 *   - When the automatic plan's segment states would not fit the scratch
 *     (very long or many long sequences, large states), the call runs with
 *     longer time segments (1024 tokens, doubled until they fit) or without
 *     segments (also when no such segment would be shorter than the longest
 *     sequence can be): the same results, less parallelism than ssm_scan_ws
 *     with a workspace of the size ssm_scan_workspace_bytes asks for.
 *   - Every call in the process shares the scratch, which keeps the last
 *     call's contents (nothing in it needs to start at zero).  Calls whose GPU
 *     work overlaps, on two streams or from two threads, race on it: the
 *     caller must serialise them.
 * Errors otherwise as for ssm_scan.
 */
int ssm_scan_static(float *state_slots, const float *x, const float *dt,
                    const float *A, const float *B, const float *C,
                    const float *D, float *y, const int32_t *seq_starts,
                    const int32_t *seq_lens, const int32_t *resume_flags,
                    int n_seqs, int n_tokens, int n_heads, int head_dim,
                    int d_state, int n_groups, void *stream);

/*
 * Causal depthwise conv1d + SiLU with a rolling conv-state slot, Mamba2's op in
 * front of the scan ("ssm_gated_delta.cu", kernel 2 and its batched variant;
 * the pages' kernel has no bias, the optional bias here is added before SiLU).
 * For sequence i (tokens packed as for ssm_scan) and channel c, the stream of
 * inputs is the slot's kernel_size-1 remembered inputs (oldest first; zeros
 * when resume_flags[i] == 0) followed by the sequence's tokens, and
 *     out[t, c] = silu(bias[c] + sum_{u < K} weight[c, u] * stream[t + u]),
 * silu(v) = v / (1 + exp(-v)), with stream[K-1+t] = x[t, c] (so weight[c, K-1]
 * multiplies the current token).  Afterwards slot i holds the stream's last
 * K-1 entries, and snapshot row t (optional) the slot image right after
 * token t.
 *   x, out      [n_tokens][channels] fp32, device (out written for owned tokens)
 *   weight      [channels][kernel_size] fp32, device
 *   bias        [channels] fp32, device, or NULL
 *   conv_state  [n_seqs][channels][kernel_size-1] fp32, device, in/out
 *   snapshots   [n_tokens][channels][kernel_size-1] fp32, device, or NULL
 *   kernel_size 1 .. 8
 * Ownership, metadata, stream and 4-byte alignment rules as for ssm_scan.
 * Errors: SSM_ERR_INVALID_ARG (sizes, NULL or misaligned pointers),
 * SSM_ERR_UNSUPPORTED (n_tokens * channels above 2^31), SSM_ERR_CUDA.
 */
int ssm_conv1d(const float *x, const float *weight, const float *bias,
               float *conv_state, float *out, const int32_t *seq_starts,
               const int32_t *seq_lens, const int32_t *resume_flags,
               int n_seqs, int n_tokens, int channels, int kernel_size,
               float *snapshots, void *stream);

/* Text for a status code (static storage; never NULL). */
const char *ssm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SSMSCAN_H */
