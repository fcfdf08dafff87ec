// Gated RMSNorm after the scan (sm_103a): Mamba2's output gate, kernel 3 of
// "ssm_gated_delta.cu" applied to every (token, head) row of head_dim values:
//
//   gated_y[t,h,p] = y[t,h,p] / sqrt(mean_p(y[t,h,:]^2) + eps) * w[p] * silu(z[t,h,p])
//
// with silu(z) = z / (1 + exp(-z)) and w shared by all heads.  One warp per
// row: a strided pass for the sum of squares, a shuffle reduction, a second
// pass for the gated values (the row is re-read from L1/L2).  Only rows of
// tokens owned by a sequence are touched: grid.y walks the sequences and
// grid.x strides over a sequence's (token, head) rows.
#include "scan_common.cuh"

namespace ssm {

namespace {

constexpr int kNormWarps = 8;

__global__ void __launch_bounds__(32 * kNormWarps)
gated_norm_kernel(const ScanArgs a, const float *z, const float *w, float eps, float *out)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int P = a.P, H = a.H;
    for (int seq = blockIdx.y; seq < a.n_seqs; seq += gridDim.y) {
        const long long t0 = a.seq_starts[seq];
        const long long rows = (long long)max(0, a.seq_lens[seq]) * H;
        for (long long r = (long long)blockIdx.x * kNormWarps + warp; r < rows;
             r += (long long)gridDim.x * kNormWarps) {
            const long long off = (t0 * H + r) * P;       // row r = (token r / H, head r % H)
            const float *yr = a.y + off;
            float ss = 0.f;
            for (int p = lane; p < P; p += 32) {
                const float v = yr[p];
                ss = fmaf(v, v, ss);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                ss += __shfl_xor_sync(kFullMask, ss, o);
            const float inv = rsqrtf(ss / (float)P + eps);
            const float *zr = z + off;
            float *outr = out + off;
            for (int p = lane; p < P; p += 32) {
                const float zv = zr[p];
                outr[p] = yr[p] * inv * __ldg(w + p) * (zv / (1.f + expf(-zv)));
            }
        }
    }
}

}  // namespace

cudaError_t launch_gated_norm(const ScanArgs &a, const float *z, const float *w, float eps, float *out,
                              cudaStream_t stream)
{
    if (a.n_seqs <= 0)
        return cudaSuccess;
    const long long rows_per_seq = ((long long)a.n_tokens * a.H + a.n_seqs - 1) / a.n_seqs;
    const long long gx = (rows_per_seq + kNormWarps - 1) / kNormWarps;
    const dim3 grid((unsigned)(gx < 1 ? 1 : (gx > 4096 ? 4096 : gx)),
                    (unsigned)(a.n_seqs < 65535 ? a.n_seqs : 65535));
    gated_norm_kernel<<<grid, 32 * kNormWarps, 0, stream>>>(a, z, w, eps, out);
    return cudaGetLastError();
}

}  // namespace ssm
