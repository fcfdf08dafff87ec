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
// Unlike the scan there is no recurrence through the outputs, so spans of
// tokens are computed independently: a thread owns 4 consecutive channels
// (128-bit loads and stores, contiguous across a warp) over a contiguous span
// of a sequence's tokens, walked in runs of 16, and keeps the last k-1 inputs in
// registers across the span, so each input is read once plus a k-1 halo per
// span.  The spans are sized so that the grid is about one wave of resident
// blocks with no block more than one run behind the others.  A complete run
// issues all 16 of its loads before any arithmetic (for kernel sizes 3..5
// registers are capped for three blocks per SM, so other blocks' loads overlap
// a block's arithmetic and stores), and SiLU takes the hardware
// exponential and an approximate division, v / (1 + exp(-v)) (about 1e-6
// relative), so the kernel stays bound by memory, not by the per-element
// arithmetic.  Only the block holding a sequence's first span reads its slot
// (later spans start past the k-1 history), so that block also rewrites the
// slot, after its own reads: no second launch.
#include <algorithm>
#include <atomic>

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

// Outputs (and snapshots) of a span of a sequence's tokens for CH consecutive
// channels per thread, in runs of kConvRun tokens.  The window of the last K-1
// stream entries stays in registers across the span, so every input is loaded
// once (plus K-1 entries of halo at the span's start).  grid: x = channel
// blocks, y = sequences, z = spans of span_runs runs each.
constexpr int kConvRun = 16;

template <int CH, int K>
__global__ void __launch_bounds__(kConvThreads, (K >= 3 && K <= 5) ? 3 : 1)
conv1d_out_kernel(const ConvArgs a, int span_runs)
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
        const int span = span_runs * kConvRun;
        for (int s0 = blockIdx.z * span; s0 < len; s0 += gridDim.z * span) {   // spans of the sequence (span > k-1)
            const int s1 = min(len, s0 + span);
            // window[u] = stream[s0 + u], u < K-1 (stream[K-1+t] is token t)
            float win[KM1 > 0 ? KM1 : 1][CH];
#pragma unroll
            for (int u = 0; u < KM1; ++u) {
                const int i = s0 + u;
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
            for (int r0 = s0; r0 < s1; r0 += kConvRun) {
                const int rend = min(s1, r0 + kConvRun);
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
        if constexpr (KM1 > 0) {
            if (blockIdx.z == 0) {
                // the slot after the sequence: the stream's last K-1 entries (old slot
                // entries or zeros when the sequence is shorter than K-1), written
                // after every read of the old slot by this thread (its channels only)
                float nh[KM1][CH];
#pragma unroll
                for (int u = 0; u < KM1; ++u) {
                    const int i = len + u;
                    if (i < KM1) {
#pragma unroll
                        for (int q = 0; q < CH; ++q)
                            nh[u][q] = fresh ? 0.f : a.state[((long long)seq * a.C + c0 + q) * KM1 + i];
                    } else {
                        const Lanes<CH> xv = load_ch<CH>(a.x + (t0 + i - KM1) * a.C + c0);
#pragma unroll
                        for (int q = 0; q < CH; ++q)
                            nh[u][q] = xv.v[q];
                    }
                }
#pragma unroll
                for (int q = 0; q < CH; ++q)
#pragma unroll
                    for (int u = 0; u < KM1; ++u)
                        a.state[((long long)seq * a.C + c0 + q) * KM1 + u] = nh[u][q];
            }
        }
    }
}

}  // namespace

namespace {

// Spans of about one wave: the blocks the device holds at once are spread over
// (channel blocks x sequences) and each sequence's average run count, so no
// block has more than one run more than another (with equal lengths).
template <int CH, int K>
cudaError_t launch_out(const ConvArgs &a, cudaStream_t stream)
{
    const int per_block = kConvThreads * CH;
    const int cblocks = (a.C + per_block - 1) / per_block;
    const int gy = a.n_seqs < 65535 ? a.n_seqs : 65535;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    // resident blocks per SM of this instantiation, asked once per device
    constexpr int kDevs = 64;
    static std::atomic<int> cached[kDevs];
    per_sm = dev < kDevs ? cached[dev].load(std::memory_order_relaxed) : 0;
    if (per_sm <= 0) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, conv1d_out_kernel<CH, K>, kConvThreads, 0);
        if (e != cudaSuccess)
            return e;
        if (dev < kDevs)
            cached[dev].store(per_sm, std::memory_order_relaxed);
    }
    const long long runs = ((long long)a.n_tokens + (long long)a.n_seqs * kConvRun - 1) /
                           ((long long)a.n_seqs * kConvRun);                   // per sequence, on average
    const long long resident = (long long)(per_sm > 0 ? per_sm : 1) * sms;
    const long long want_z = std::max(1LL, (resident + (long long)cblocks * gy - 1) / ((long long)cblocks * gy));
    const long long span_runs = std::max(1LL, (runs + want_z - 1) / want_z);
    const long long gz = std::min(65535LL, std::max(1LL, (runs + span_runs - 1) / span_runs));
    const dim3 grid((unsigned)cblocks, (unsigned)gy, (unsigned)gz);
    return launch_pdl(conv1d_out_kernel<CH, K>, grid, dim3(kConvThreads), 0, stream, a, (int)span_runs);
}

template <int CH>
cudaError_t launch_out_k(const ConvArgs &a, cudaStream_t stream)
{
    switch (a.K) {
    case 1: return launch_out<CH, 1>(a, stream);
    case 2: return launch_out<CH, 2>(a, stream);
    case 3: return launch_out<CH, 3>(a, stream);
    case 4: return launch_out<CH, 4>(a, stream);
    case 5: return launch_out<CH, 5>(a, stream);
    case 6: return launch_out<CH, 6>(a, stream);
    case 7: return launch_out<CH, 7>(a, stream);
    case 8: return launch_out<CH, 8>(a, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_conv1d(const float *x, const float *w, const float *bias, float *state, float *out,
                          float *snaps, const int32_t *seq_starts, const int32_t *seq_lens,
                          const int32_t *resume, int n_seqs, int n_tokens, int C, int K, cudaStream_t stream)
{
    ConvArgs a{x, w, bias, state, out, snaps, seq_starts, seq_lens, resume, n_seqs, n_tokens, C, K};
    if (n_seqs <= 0 || (n_tokens <= 0 && K <= 1))
        return cudaSuccess;                   // nothing to compute and no slot to roll
    // (with no tokens the launch still rolls the slots: a fresh sequence's slot becomes zeros)
    const bool vec = C % 4 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    return vec ? launch_out_k<4>(a, stream) : launch_out_k<1>(a, stream);
}

}  // namespace ssm
