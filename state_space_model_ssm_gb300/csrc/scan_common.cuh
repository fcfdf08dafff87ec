// Shared definitions of the sm_103a scan kernels (device side and launchers).
//
// Operation (for sequence i, head h, head-dim row p, token t; g = h/(H/G)):
//   dA = exp(dt[t,h]*A[h]);  S[h,p,:] = dA*S[h,p,:] + dt[t,h]*x[t,h,p]*B[t,g,:];
//   y[t,h,p] = S[h,p,:].C[t,g,:] + D[h]*x[t,h,p]
// ("The llama journey", Day 14 kernel body; the D skip term is part of the
// operation here.)
//
// A "row" is one (head, head-dim) pair: its flattened index r = h*P + p is
// also its offset inside a token of x/y and inside a state slot (times N).
// Rows of one group are contiguous in that flattened order, so a run of rows
// inside one group shares B and C.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

struct ScanArgs {
    float *state;              // [n][H][P][N]
    const float *x;            // [T][H][P]
    const float *dt;           // [T][H]
    const float *A;            // [H]
    const float *B;            // [T][G][N]
    const float *C;            // [T][G][N]
    const float *D;            // [H]
    float *y;                  // [T][H][P]
    const int32_t *seq_starts; // [n]
    const int32_t *seq_lens;   // [n]
    const int32_t *resume;     // [n]
    int n_seqs, n_tokens, H, P, N, G;
    float *snaps;              // [T][H][P][N]: the state after each owned token, or null (decode kernel)
};

// Launch geometry of the chunk-staged prefill kernel.
struct PrefillGeom {
    int rows_per_group;  // (H/G)*P
    int runs_per_group;  // thread blocks per (sequence, group)
    int rows_per_cta;    // state rows a block owns
    int chunk;           // tokens staged per chunk
    int heads_cap;       // most heads one block's rows can touch
};

// Launch geometry of the warp-per-row decode kernel: grid.x covers the warps
// of one sequence, grid.y the sequences (blocks loop when n_seqs > grid.y).
struct DecodeGeom {
    int rows_per_warp;   // (32/LANES)*RPT
    int tasks_per_seq;   // warps per sequence: ceil(H*P / rows_per_warp)
};

constexpr unsigned kFullMask = 0xffffffffu;

template <int X>
struct Log2 { static constexpr int value = 1 + Log2<X / 2>::value; };
template <>
struct Log2<1> { static constexpr int value = 0; };

// Sum RPT per-row partial sums over the LANES lanes that share those rows.
// The first log2(RPT) butterfly levels also transpose: at each level a lane
// keeps half of its values and receives its partner's matching half, so the
// shuffle count is (RPT-1) + log2(LANES/RPT) instead of RPT*log2(LANES).
// On return every lane holds the full sum of row `reduced_row<LANES,RPT>(j)`.
template <int LANES, int RPT>
__device__ __forceinline__ float reduce_rows(float (&v)[RPT], int j)
{
    static_assert(RPT <= LANES, "more rows than lanes");
    constexpr int LV = Log2<RPT>::value;
#pragma unroll
    for (int level = 0, cnt = RPT, off = LANES / 2; level < LV; ++level, cnt /= 2, off /= 2) {
        const bool hi = (j & off) != 0;
#pragma unroll
        for (int m = 0; m < cnt / 2; ++m) {
            const float send = hi ? v[2 * m] : v[2 * m + 1];
            const float keep = hi ? v[2 * m + 1] : v[2 * m];
            v[m] = keep + __shfl_xor_sync(kFullMask, send, off);
        }
    }
    float s = v[0];
#pragma unroll
    for (int off = LANES / (2 * RPT); off >= 1; off /= 2)
        s += __shfl_xor_sync(kFullMask, s, off);
    return s;
}

// Which of the RPT rows lane j's reduced sum belongs to.
template <int LANES, int RPT>
__device__ __forceinline__ int reduced_row(int j)
{
    constexpr int LV = Log2<RPT>::value;
    constexpr int LL = Log2<LANES>::value;
    int r = 0;
#pragma unroll
    for (int k = 0; k < LV; ++k)
        r |= ((j >> (LL - 1 - k)) & 1) << k;
    return r;
}

// The first lane (of LANES) whose reduced sum is row r: the inverse of
// reduced_row for the lanes whose low bits are zero.
template <int LANES, int RPT>
__device__ __forceinline__ int reduced_lane(int r)
{
    constexpr int LV = Log2<RPT>::value;
    constexpr int LL = Log2<LANES>::value;
    int j = 0;
#pragma unroll
    for (int k = 0; k < LV; ++k)
        j |= ((r >> k) & 1) << (LL - 1 - k);
    return j;
}

// True for one lane per reduced row (the lane whose low bits are zero).
template <int LANES, int RPT>
__device__ __forceinline__ bool reduced_writer(int j)
{
    return (j & (LANES / RPT - 1)) == 0;
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialization (launch_pdl), so its blocks may be
// scheduled while the previous kernel on the stream drains.  griddep_entry()
// is the first statement of every kernel: it waits until the previous grid has
// completed and its writes are visible (griddepcontrol.wait; nothing of ours
// touches global memory before it), then lets the next kernel's blocks be
// scheduled as SMs free up (griddepcontrol.launch_dependents).  The result is
// the same as plain stream order; only launch latency and wave tails overlap.
__device__ __forceinline__ void griddep_entry()
{
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// True when a bounded device wait earlier in the same call gave up: the call's
// status word (zeroed by the call's first kernel) is nonzero.  The kernels
// that consume the products of such a wait then write NaN to y and leave the
// state slots as they were, so the failure shows in the outputs even when the
// host never reads the word back.
__device__ __forceinline__ bool call_failed(const int *status)
{
    return status != nullptr && *reinterpret_cast<const volatile int *>(status) != 0;
}

// NaN into rows [r0, r0 + nrows) of tokens [t0, t0 + len) of y ([T][H*P]);
// threads tid = 0 .. nthr-1 of the caller share the stores.
__device__ __forceinline__ void poison_y(float *y, long long HP, long long t0, int len, int r0, int nrows,
                                         int tid, int nthr)
{
    const long long n = (long long)len * nrows;
    for (long long i = tid; i < n; i += nthr) {
        const long long t = i / nrows;
        y[(t0 + t) * HP + r0 + (i - t * nrows)] = __int_as_float(0x7fc00000);
    }
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// kernel<<<grid, block, smem, stream>>>(args...) with programmatic stream
// serialization (see griddep_entry), then cudaGetLastError().
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// cudaFuncSetAttribute(kernel, MaxDynamicSharedMemorySize, bytes) on the
// current device, skipped when an earlier call already set at least `bytes`
// for that (device, kernel) pair (api.cu).  Thread-safe.
cudaError_t set_dynamic_smem(const void *kernel, size_t bytes);

// Host-side launchers (defined in prefill.cu / decode.cu).  Return a
// cudaError_t from the launch, or cudaErrorInvalidValue for a shape with no
// compiled kernel.
cudaError_t launch_prefill(const ScanArgs &a, const PrefillGeom &g, int lanes,
                           int vpl, int rpt, size_t smem_bytes, int sms,
                           cudaStream_t stream);
bool prefill_supported(int lanes, int vpl, int rpt);
size_t prefill_smem_bytes(const PrefillGeom &g, int N);

// Time segments of long sequences (the segment pass): work unit u is time
// segment units[u] = (sequence, segment) covering tokens [seg*seg_len,
// (seg+1)*seg_len) of the sequence.  units == nullptr: one unit per sequence.
struct SegmentPlan {
    const int2 *units;        // [max_units] (device), filled by the plan kernel
    const int *n_units;       // device count of valid units
    const int *unit_base;     // [n_seqs + 1] first unit of each sequence
    int seg_len;              // tokens per segment (a multiple of the chunk)
    float *seg_state;         // [max_units][H][P][N]: state pass output, then S_in of seg+1
    float *seg_decay;         // [max_units][H]: prod dA over the segment
    int *status;              // device word (may be null): zeroed by the plan kernel, nonzero
                              // when a bounded wait of the tensor-core state pass gave up
    int fail_waits;           // test hook: nonzero makes the pipeline's bounded waits give up at once
    int chunk_states;         // tensor-core state pass for the SSD form: every unit (each sequence's
                              // last too), no slot term, seg_decay = sum of dt*A (its log)
};
constexpr int kScanFull = 0;        // the scan with y
constexpr int kScanStateOnly = 1;   // one segment's state from zero, no y

// The gated RMSNorm output written by the full pass itself (see
// launch_gated_norm for the operation); out == nullptr: off.
struct GatedOut {
    const float *z;           // [T][H][P], 16-byte aligned
    const float *w;           // [P]
    float eps;
    float *out;               // [T][H][P], 16-byte aligned
};

cudaError_t launch_prefill_scaled(const ScanArgs &a, const PrefillGeom &g, int lanes, int vpl,
                                  int rpt, const SegmentPlan &plan, int mode, long long n_units,
                                  size_t smem_bytes, cudaStream_t stream, int epi = 0,
                                  const GatedOut *gated = nullptr);
cudaError_t launch_segment_plan(const ScanArgs &a, const SegmentPlan &plan, int max_units,
                                cudaStream_t stream);
cudaError_t launch_segment_combine(const ScanArgs &a, const SegmentPlan &plan, int max_units,
                                   cudaStream_t stream);
// The state pass on the tensor cores (segment_state_tc.cu): the same L_k and
// d_k as the kScanStateOnly mode, as a product over the segment's tokens with
// fp32 accuracy from split TF32 operands.  Grid (max_units, H).
// Its TMA descriptors of B and x (two CUtensorMap images) are encoded on the
// host before any launch; false when the driver cannot describe the tensors.
struct SegStateMaps {
    alignas(64) unsigned char b[128];
    alignas(64) unsigned char x[128];
};
bool segment_state_tc_supported(int N, int P, size_t smem_optin);
bool segment_state_tc_maps(const ScanArgs &a, SegStateMaps *maps);
cudaError_t launch_segment_state_tc(const ScanArgs &a, const SegmentPlan &plan, const SegStateMaps &maps,
                                    int max_units, cudaStream_t stream);
bool prefill_scaled_supported(int lanes, int vpl, int rpt);
// True for the shapes (and block sizes) whose full pass has the output-tile
// variants: y stored by the producer warp (epi 1), and also the gated output
// (epi 2).
bool prefill_scaled_tile_supported(int lanes, int vpl, int rpt, int rows_per_cta);
// True for the shapes (and block sizes) whose full pass has the self-staged
// variants (epi 5, and 4 with the gated output): no producer warp, four
// consumer warps stage the chunks themselves, three blocks per SM.
bool prefill_scaled_self_supported(int lanes, int vpl, int rpt, int rows_per_cta);
size_t prefill_scaled_smem_bytes(const PrefillGeom &g, int N, int lanes, int epi = 0);
constexpr int kScaledMaxChunk = 32;    // one warp lane per token in the coefficient pass

// The SSD chunked form (ssd.cu): work unit u is chunk units[u] = (sequence,
// k) covering tokens [k*chunk, (k+1)*chunk) of the sequence.
struct SsdPlan {
    const int2 *units;        // [max_units] (device), filled by the plan kernel
    const int *n_units;       // device count of valid units
    const int *unit_base;     // [n_seqs + 1] first unit of each sequence
    int chunk;                // tokens per chunk (64 or 128)
    float *chunk_state;       // [max_units][H][P][N]: chunk state, then the chunk's incoming state
    float *chunk_logdecay;    // [max_units][H]: sum of dt*A over the chunk
    int *status;              // device word: nonzero when a kernel's bounded wait gave up
    int fail_waits;           // test hook: nonzero makes the pipeline's bounded waits give up at once
};

// Shared-memory strides (floats) and launch shape of the SSD kernels.
struct SsdGeom {
    int n_pad;                // d_state rounded up to a multiple of 8
    int bs_stride;            // chunk-state kernel: B rows (== 8 mod 32)
    int xw_stride;            // chunk-state kernel: weighted x rows (== 8 mod 32)
    int cs_stride;            // output kernel: C, B and state rows (== 4 mod 32)
    int xs_stride;            // output kernel: x rows (== 4 mod 32)
    int heads_per_cta;        // heads of one group a block handles
    int use_tc;               // output kernel on tcgen05 (ssd_tc.cu) instead of mma.sync
    int tmem_cols;            // TMEM columns the tcgen05 output kernel allocates
    int state_buffers;        // chunk-state kernel: x tiles in flight (1 or 2)
    int out_buffers;          // output kernel: (x, S_in) tile pairs in flight (1 or 2)
    size_t smem_state, smem_out;
};

// Caller-supplied CUDA events recorded around a call's kernel launches, in
// launch order: ev[2k] right before the k-th launch, ev[2k + 1] right after
// it, while 2k + 1 < n (host side; a failed record makes the call fail).
struct LaunchTimer {
    void *const *ev = nullptr;
    int n = 0, k = 0;
    cudaStream_t stream = nullptr;
    bool failed = false;
    void before()
    {
        if (2 * k + 1 < n)
            failed |= cudaEventRecord(static_cast<cudaEvent_t>(ev[2 * k]), stream) != cudaSuccess;
    }
    void after()
    {
        if (2 * k + 1 < n)
            failed |= cudaEventRecord(static_cast<cudaEvent_t>(ev[2 * k + 1]), stream) != cudaSuccess;
        ++k;
    }
};

// The launch `launch()` (one kernel) bracketed by the timer's next event pair.
template <class F>
cudaError_t timed(LaunchTimer *tm, F &&launch)
{
    if (tm)
        tm->before();
    const cudaError_t e = launch();
    if (tm)
        tm->after();
    return e;
}

// The chunk-state, state-pass and output kernels, each bracketed by tm's events.
// With state_maps the chunk states run on the tensor-core state pass
// (segment_state_tc.cu), else on the mma.sync chunk-state kernel.
cudaError_t launch_ssd(const ScanArgs &a, const SsdPlan &plan, const SsdGeom &g, int max_units,
                       cudaStream_t stream, LaunchTimer *tm = nullptr, const SegStateMaps *state_maps = nullptr);
bool ssd_supported_chunk(int chunk);
int ssd_tc_buffers(int chunk, int n_pad, int P, size_t smem_optin);   // 0: not supported
int ssd_tc_tmem_cols(int n_pad, int P);
size_t ssd_tc_smem_bytes(int n_pad, int P, int nbuf);
cudaError_t launch_ssd_output_tc(const ScanArgs &a, const SsdPlan &plan, const SsdGeom &g, int max_units,
                                 cudaStream_t stream);
int ssd_max_head_dim();

// Mamba2's step for the owned tokens: out[t,h] = softplus(dt[t,h] + bias[h])
// (identity above 20; bias may be null, softplus optional), written once
// before the scan so that the scan kernels read a plain step (dt_prep.cu).
cudaError_t launch_dt_prep(const ScanArgs &a, const float *bias, int softplus, float *out, cudaStream_t stream);

// Causal depthwise conv1d + SiLU with a rolling conv-state slot (conv1d.cu).
cudaError_t launch_conv1d(const float *x, const float *w, const float *bias, float *state, float *out,
                          float *snaps, const int32_t *seq_starts, const int32_t *seq_lens,
                          const int32_t *resume, int n_seqs, int n_tokens, int C, int K, cudaStream_t stream);

// Gated RMSNorm of y per (token, head) row, after the scan (gated_norm.cu).
cudaError_t launch_gated_norm(const ScanArgs &a, const float *z, const float *w, float eps, float *out,
                              cudaStream_t stream);

cudaError_t launch_decode(const ScanArgs &a, const DecodeGeom &g, int lanes,
                          int vpl, int rpt, int grid_seqs, cudaStream_t stream);
bool decode_supported(int lanes, int vpl, int rpt);
constexpr int kDecodeWarps = 8;

}  // namespace ssm
