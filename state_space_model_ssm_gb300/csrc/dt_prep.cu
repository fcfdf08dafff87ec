// Mamba2's discretisation step before the scan (sm_103a):
//
//   step[t,h] = v > 20 ? v : log1p(exp(v)),   v = dt[t,h] + dt_bias[h]
//
// ("The llama journey", Day 14 kernel body; the decay-gate kernel of
// "ssm_gated_delta.cu"), for the tokens owned by a sequence, into a buffer of
// the caller's workspace.  The scan kernels then read that buffer as their
// step.  Doing it here rather than at the kernels' own loads of dt keeps the
// option's code out of their hot loops (T*H floats: about 1 MB for 4096
// tokens at 64 heads, against the scan's hundreds).
#include "scan_common.cuh"

namespace ssm {

namespace {

constexpr int kDtThreads = 256;

__global__ void __launch_bounds__(kDtThreads)
dt_prep_kernel(const ScanArgs a, const float *bias, int softplus, float *out)
{
    griddep_entry();
    const int H = a.H;
    for (int seq = blockIdx.y; seq < a.n_seqs; seq += gridDim.y) {
        const long long t0 = a.seq_starts[seq];
        const long long n = (long long)max(0, a.seq_lens[seq]) * H;
        for (long long e = (long long)blockIdx.x * kDtThreads + threadIdx.x; e < n;
             e += (long long)gridDim.x * kDtThreads) {
            const long long i = t0 * H + e;            // element (t0 + e / H, e % H)
            float v = a.dt[i];
            if (bias)
                v += __ldg(bias + (int)(e % H));
            if (softplus && v <= 20.f)
                v = log1pf(expf(v));
            out[i] = v;
        }
    }
}

}  // namespace

cudaError_t launch_dt_prep(const ScanArgs &a, const float *bias, int softplus, float *out, cudaStream_t stream)
{
    if (a.n_seqs <= 0 || a.n_tokens <= 0)
        return cudaSuccess;
    const long long per_seq = ((long long)a.n_tokens * a.H + a.n_seqs - 1) / a.n_seqs;
    const long long gx = (per_seq + kDtThreads - 1) / kDtThreads;
    const dim3 grid((unsigned)(gx < 1 ? 1 : (gx > 4096 ? 4096 : gx)), (unsigned)(a.n_seqs < 65535 ? a.n_seqs : 65535));
    return launch_pdl(dt_prep_kernel, grid, dim3(kDtThreads), 0, stream, a, bias, softplus, out);
}

}  // namespace ssm
