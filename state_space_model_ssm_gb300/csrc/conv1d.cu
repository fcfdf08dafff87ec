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
// Unlike the scan there is no recurrence through the outputs, so every
// (token, channel) output is computed independently, one thread each, with
// channels contiguous for coalesced loads and stores; the k reads of x per
// output hit L1/L2.  The slot update runs as a second launch so that no
// output reads a slot another thread has already rewritten.
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

__global__ void __launch_bounds__(kConvThreads)
conv1d_out_kernel(const ConvArgs a)
{
    const int km1 = a.K - 1;
    for (int seq = blockIdx.y; seq < a.n_seqs; seq += gridDim.y) {
        const long long t0 = a.seq_starts[seq];
        const long long n = (long long)max(0, a.seq_lens[seq]) * a.C;
        const bool fresh = a.resume[seq] == 0;
        for (long long e = (long long)blockIdx.x * kConvThreads + threadIdx.x; e < n;
             e += (long long)gridDim.x * kConvThreads) {
            const int t = (int)(e / a.C), c = (int)(e - (long long)t * a.C);
            const float *hist = a.state + ((long long)seq * a.C + c) * km1;
            const float *wc = a.w + (long long)c * a.K;
            float acc = a.bias ? __ldg(a.bias + c) : 0.f;
            for (int u = 0; u < a.K; ++u)
                acc = fmaf(__ldg(wc + u), stream_at(a, hist, fresh, t0, c, t + u), acc);
            a.out[(t0 + t) * a.C + c] = acc / (1.f + expf(-acc));
            if (a.snaps) {
                float *sn = a.snaps + ((t0 + t) * a.C + c) * km1;
                for (int u = 0; u < km1; ++u)
                    sn[u] = stream_at(a, hist, fresh, t0, c, t + 1 + u);
            }
        }
    }
}

__global__ void __launch_bounds__(kConvThreads)
conv1d_state_kernel(const ConvArgs a)
{
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

cudaError_t launch_conv1d(const float *x, const float *w, const float *bias, float *state, float *out,
                          float *snaps, const int32_t *seq_starts, const int32_t *seq_lens,
                          const int32_t *resume, int n_seqs, int n_tokens, int C, int K, cudaStream_t stream)
{
    ConvArgs a{x, w, bias, state, out, snaps, seq_starts, seq_lens, resume, n_seqs, n_tokens, C, K};
    if (n_tokens > 0) {
        const long long per_seq = ((long long)n_tokens * C + n_seqs - 1) / n_seqs;
        const long long gx = (per_seq + kConvThreads - 1) / kConvThreads;
        const dim3 grid((unsigned)(gx < 1 ? 1 : (gx > 8192 ? 8192 : gx)), (unsigned)(n_seqs < 65535 ? n_seqs : 65535));
        conv1d_out_kernel<<<grid, kConvThreads, 0, stream>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    if (K > 1) {
        const long long cells = (long long)n_seqs * C;
        conv1d_state_kernel<<<(unsigned)((cells + kConvThreads - 1) / kConvThreads), kConvThreads, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace ssm
