// Causal depthwise conv1d + SiLU with a rolling conv-state slot (sm_103a):
// Mamba2's op in front of the scan, after "ssm_gated_delta.cu", kernel 2 and
// its batched variant.  For every sequence i and channel c, the stream of
// inputs is the channel's k-1 remembered inputs (conv_state slot i, oldest
// first; zeros for a fresh sequence) followed by the sequence's tokens, and
//
//   out[t, c] = silu(bias[c] + sum_{u<k} w[c, u] * stream[t + u])
//
// (stream[k-1+t] is token t).  Afterwards the slot holds the stream's last k-1
// entries.  Snapshots (optional) hold stream[t+1 .. t+k-1], the slot image
// right after token t.
//
// Unlike the scan there is no recurrence through the outputs, so runs of
// tokens are computed independently: a thread owns 4 consecutive channels
// (128-bit loads and stores, contiguous across a warp) over a run of 16 tokens
// and keeps the last k-1 inputs in registers, so each input is read once plus
// a k-1 halo per run.  A complete run issues all 16 of its loads before any
// arithmetic (a quarter KiB per thread in flight; for kernel sizes 2..5
// registers are capped for three blocks per SM, so other blocks' loads overlap
// a block's arithmetic and stores), and SiLU takes the hardware
// exponential and an approximate division, v / (1 + exp(-v)) (about 1e-6
// relative), so the kernel stays bound by memory, not by the per-element
// arithmetic.  The slot update runs as a second launch so that no output reads
// a slot another thread has already rewritten.
#include "scan_common.cuh"

namespace ssm {

namespace {

constexpr int kConvThreads = 256;

struct ConvArgs {
    const float *x, *w, *bias;
    float *state, *out, *snaps;
    const int32_t *seq_starts, *seq_lens, *resume;
    int n_seqs, n_tokens, C, K;
};

// Entry i of a channel's stream: the slot's history before the sequence, then
// its tokens.
__device__ __forceinline__ float stream_at(const ConvArgs &a, const float *hist, bool fresh, long long t0,
                                           int c, int i)
{
    const int km1 = a.K - 1;
    if (i < km1)
        return fresh ? 0.f : hist[i];
    return __ldg(a.x + (t0 + i - km1) * a.C + c);
}

// Vector of CH consecutive channels.
template <int CH>
struct Lanes {
    float v[CH];
};

template <int CH>
__device__ __forceinline__ Lanes<CH> load_ch(const float *p)
{
    Lanes<CH> r;
    if constexpr (CH == 4) {
        const float4 q = __ldg(reinterpret_cast<const float4 *>(p));
        r.v[0] = q.x; r.v[1] = q.y; r.v[2] = q.z; r.v[3] = q.w;
    } else {
#pragma unroll
        for (int i = 0; i < CH; ++i)
            r.v[i] = __ldg(p + i);
    }
    return r;
}

template <int CH>
__device__ __forceinline__ void store_ch(float *p, const Lanes<CH> &r)
{
    if constexpr (CH == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(r.v[0], r.v[1], r.v[2], r.v[3]);
    } else {
#pragma unroll
        for (int i = 0; i < CH; ++i)
            p[i] = r.v[i];
    }
}

// Outputs (and snapshots) of a run of kConvRun tokens of one sequence for CH
// consecutive channels per thread.  The window of the last K-1 stream entries
// stays in registers, so every input is loaded once per run (plus K-1 entries
// of halo at the run's start).  grid: x = channel blocks, y = sequences,
// z strides over a sequence's runs.
constexpr int kConvRun = 16;

template <int CH, int K>
__global__ void __launch_bounds__(kConvThreads, (K >= 2 && K <= 5) ? 3 : 1)
conv1d_out_kernel(const ConvArgs a)
{
    griddep_entry();
    constexpr int KM1 = K - 1;
    const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * CH;
    if (c0 >= a.C)
        return;
    float w[K][CH], bias[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i) {
#pragma unroll
        for (int u = 0; u < K; ++u)
            w[u][i] = __ldg(a.w + (long long)(c0 + i) * K + u);
        bias[i] = a.bias ? __ldg(a.bias + c0 + i) : 0.f;
    }
    for (int seq = blockIdx.y; seq < a.n_seqs; seq += gridDim.y) {
        const long long t0 = a.seq_starts[seq];
        const int len = max(0, a.seq_lens[seq]);
        const bool fresh = a.resume[seq] == 0;
        for (int r0 = blockIdx.z * kConvRun; r0 < len; r0 += gridDim.z * kConvRun) {
            // window[u] = stream[r0 + u], u < K-1 (stream[K-1+t] is token t)
            float win[KM1 > 0 ? KM1 : 1][CH];
#pragma unroll
            for (int u = 0; u < KM1; ++u) {
                const int i = r0 + u;
                if (i < KM1) {
#pragma unroll
                    for (int q = 0; q < CH; ++q)
                        win[u][q] = fresh ? 0.f : a.state[((long long)seq * a.C + c0 + q) * KM1 + i];
                } else {
                    const Lanes<CH> xv = load_ch<CH>(a.x + (t0 + i - KM1) * a.C + c0);
#pragma unroll
                    for (int q = 0; q < CH; ++q)
                        win[u][q] = xv.v[q];
                }
            }
            const int rend = min(len, r0 + kConvRun);
            // token t of the run from its input xv and the window of the K-1 before it
            auto token = [&](int t, const Lanes<CH> &xv) {
                Lanes<CH> o;
#pragma unroll
                for (int q = 0; q < CH; ++q) {
                    float acc = fmaf(w[KM1][q], xv.v[q], bias[q]);
#pragma unroll
                    for (int u = 0; u < KM1; ++u)
                        acc = fmaf(w[u][q], win[u][q], acc);
                    o.v[q] = __fdividef(acc, 1.f + __expf(-acc));
                }
                store_ch<CH>(a.out + (t0 + t) * a.C + c0, o);
#pragma unroll
                for (int u = 0; u + 1 < KM1; ++u)
#pragma unroll
                    for (int q = 0; q < CH; ++q)
                        win[u][q] = win[u + 1][q];
                if constexpr (KM1 > 0) {
#pragma unroll
                    for (int q = 0; q < CH; ++q)
                        win[KM1 - 1][q] = xv.v[q];
                }
                if (a.snaps) {                                  // the slot image right after token t
#pragma unroll
                    for (int q = 0; q < CH; ++q) {
                        float *sn = a.snaps + ((t0 + t) * a.C + c0 + q) * KM1;
#pragma unroll
                        for (int u = 0; u < KM1; ++u)
                            sn[u] = win[u][q];
                    }
                }
            };
            if (rend - r0 == kConvRun) {                        // a complete run: every load first
                Lanes<CH> xs[kConvRun];
#pragma unroll
                for (int i = 0; i < kConvRun; ++i)
                    xs[i] = load_ch<CH>(a.x + (t0 + r0 + i) * a.C + c0);
#pragma unroll
                for (int i = 0; i < kConvRun; ++i)
                    token(r0 + i, xs[i]);
            } else {
                for (int t = r0; t < rend; ++t)
                    token(t, load_ch<CH>(a.x + (t0 + t) * a.C + c0));
            }
        }
    }
}

__global__ void __launch_bounds__(kConvThreads)
conv1d_state_kernel(const ConvArgs a)
{
    griddep_entry();
    const int km1 = a.K - 1;
    const long long e = (long long)blockIdx.x * kConvThreads + threadIdx.x;
    if (e >= (long long)a.n_seqs * a.C)
        return;
    const int seq = (int)(e / a.C), c = (int)(e - (long long)seq * a.C);
    const long long t0 = a.seq_starts[seq];
    const int len = max(0, a.seq_lens[seq]);
    const bool fresh = a.resume[seq] == 0;
    float *hist = a.state + ((long long)seq * a.C + c) * km1;
    float nh[8];
    for (int u = 0; u < km1; ++u)
        nh[u] = stream_at(a, hist, fresh, t0, c, len + u);   // read every entry before writing any
    for (int u = 0; u < km1; ++u)
        hist[u] = nh[u];
}

}  // namespace

namespace {

template <int CH, int K>
cudaError_t launch_out(const ConvArgs &a, int gz, cudaStream_t stream)
{
    const int per_block = kConvThreads * CH;
    const dim3 grid((unsigned)((a.C + per_block - 1) / per_block), (unsigned)(a.n_seqs < 65535 ? a.n_seqs : 65535),
                    (unsigned)gz);
    return launch_pdl(conv1d_out_kernel<CH, K>, grid, dim3(kConvThreads), 0, stream, a);
}

template <int CH>
cudaError_t launch_out_k(const ConvArgs &a, int gz, cudaStream_t stream)
{
    switch (a.K) {
    case 1: return launch_out<CH, 1>(a, gz, stream);
    case 2: return launch_out<CH, 2>(a, gz, stream);
    case 3: return launch_out<CH, 3>(a, gz, stream);
    case 4: return launch_out<CH, 4>(a, gz, stream);
    case 5: return launch_out<CH, 5>(a, gz, stream);
    case 6: return launch_out<CH, 6>(a, gz, stream);
    case 7: return launch_out<CH, 7>(a, gz, stream);
    case 8: return launch_out<CH, 8>(a, gz, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_conv1d(const float *x, const float *w, const float *bias, float *state, float *out,
                          float *snaps, const int32_t *seq_starts, const int32_t *seq_lens,
                          const int32_t *resume, int n_seqs, int n_tokens, int C, int K, cudaStream_t stream)
{
    ConvArgs a{x, w, bias, state, out, snaps, seq_starts, seq_lens, resume, n_seqs, n_tokens, C, K};
    if (n_tokens > 0) {
        // runs per sequence on average; the z blocks stride over a sequence's runs
        const long long runs = ((long long)n_tokens + (long long)n_seqs * kConvRun - 1) / ((long long)n_seqs * kConvRun);
        const int gz = (int)(runs < 1 ? 1 : (runs > 65535 ? 65535 : runs));
        const bool vec = C % 4 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                         (reinterpret_cast<uintptr_t>(out) & 15) == 0;
        const cudaError_t e = vec ? launch_out_k<4>(a, gz, stream) : launch_out_k<1>(a, gz, stream);
        if (e != cudaSuccess)
            return e;
    }
    if (K > 1) {
        const long long cells = (long long)n_seqs * C;
        return launch_pdl(conv1d_state_kernel, dim3((unsigned)((cells + kConvThreads - 1) / kConvThreads)),
                          dim3(kConvThreads), 0, stream, a);
    }
    return cudaSuccess;
}

}  // namespace ssm
