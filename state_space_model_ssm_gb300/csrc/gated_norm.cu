// Gated RMSNorm after the scan (sm_103a): Mamba2's output gate, kernel 3 of
// "ssm_gated_delta.cu" applied to every (token, head) row of head_dim values:
//
//   gated_y[t,h,p] = y[t,h,p] / sqrt(mean_p(y[t,h,:]^2) + eps) * w[p] * silu(z[t,h,p])
//
// with silu(z) = z / (1 + exp(-z)) and w shared by all heads.  A row is shared
// by the lanes of a group (128-bit loads when head_dim is a multiple of 4, else
// one warp with scalar loads): the sum of squares is reduced by shuffles among
// the group's lanes and the row stays in registers for the gated pass.  Only rows of
// tokens owned by a sequence are touched: grid.y walks the sequences and
// grid.x strides over a sequence's (token, head) rows.
#include "scan_common.cuh"

namespace ssm {

namespace {

constexpr int kNormWarps = 8;

// silu(z) = z / (1 + e^-z) from the hardware exponential and an approximate
// division (about 1e-6 relative; the same form the prefill kernel's fused
// gated output uses).
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// Scalar path (any head_dim): one warp per row.
__global__ void __launch_bounds__(32 * kNormWarps)
gated_norm_kernel(const ScanArgs a, const float *z, const float *w, float eps, float *out)
{
    griddep_entry();
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
                outr[p] = yr[p] * inv * __ldg(w + p) * silu(zv);
            }
        }
    }
}

// Vector path (head_dim a multiple of 4, 16-byte aligned rows): a group of G
// lanes (a power of two, G float4 per pass) shares a row, 32/G rows per warp;
// the row's float4 are held in registers between the two passes (VPL per lane).
template <int G, int VPL>
__global__ void __launch_bounds__(32 * kNormWarps)
gated_norm_vec_kernel(const ScanArgs a, const float *z, const float *w, float eps, float *out)
{
    griddep_entry();
    constexpr int RPW = 32 / G;                       // rows per warp
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j = lane % G, sub = lane / G;
    const int P = a.P, P4 = P >> 2, H = a.H;
    for (int seq = blockIdx.y; seq < a.n_seqs; seq += gridDim.y) {
        const long long t0 = a.seq_starts[seq];
        const long long rows = (long long)max(0, a.seq_lens[seq]) * H;
        const long long step = (long long)gridDim.x * kNormWarps * RPW;
        for (long long rb = ((long long)blockIdx.x * kNormWarps + warp) * RPW; rb < rows; rb += step) {
            const long long r = rb + sub;
            const bool ok = r < rows;
            const long long off = (t0 * H + (ok ? r : rb)) * P;
            const float4 *yr = reinterpret_cast<const float4 *>(a.y + off);
            float4 v[VPL];
            float ss = 0.f;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int c = k * G + j;
                v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ok && c < P4)
                    v[k] = yr[c];
                ss = fmaf(v[k].x, v[k].x, fmaf(v[k].y, v[k].y, fmaf(v[k].z, v[k].z, fmaf(v[k].w, v[k].w, ss))));
            }
#pragma unroll
            for (int o = G / 2; o >= 1; o >>= 1)
                ss += __shfl_xor_sync(kFullMask, ss, o);
            const float inv = rsqrtf(ss / (float)P + eps);
            const float4 *zr = reinterpret_cast<const float4 *>(z + off);
            float4 *outr = reinterpret_cast<float4 *>(out + off);
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int c = k * G + j;
                if (ok && c < P4) {
                    const float4 zv = zr[c];
                    const float4 wv = __ldg(reinterpret_cast<const float4 *>(w) + c);
                    float4 o;
                    o.x = v[k].x * inv * wv.x * silu(zv.x);
                    o.y = v[k].y * inv * wv.y * silu(zv.y);
                    o.z = v[k].z * inv * wv.z * silu(zv.z);
                    o.w = v[k].w * inv * wv.w * silu(zv.w);
                    outr[c] = o;
                }
            }
        }
    }
}

template <int G, int VPL>
cudaError_t launch_vec(const ScanArgs &a, const float *z, const float *w, float eps, float *out, cudaStream_t st)
{
    const long long rows_per_seq = ((long long)a.n_tokens * a.H + a.n_seqs - 1) / a.n_seqs;
    const long long per_block = (long long)kNormWarps * (32 / G);
    const long long gx = (rows_per_seq + per_block - 1) / per_block;
    const dim3 grid((unsigned)(gx < 1 ? 1 : (gx > 8192 ? 8192 : gx)), (unsigned)(a.n_seqs < 65535 ? a.n_seqs : 65535));
    return launch_pdl(gated_norm_vec_kernel<G, VPL>, grid, dim3(32 * kNormWarps), 0, st, a, z, w, eps, out);
}

}  // namespace

cudaError_t launch_gated_norm(const ScanArgs &a, const float *z, const float *w, float eps, float *out,
                              cudaStream_t stream)
{
    if (a.n_seqs <= 0)
        return cudaSuccess;
    const int P4 = a.P / 4;
    const bool vec = a.P % 4 == 0 && ((reinterpret_cast<uintptr_t>(a.y) | reinterpret_cast<uintptr_t>(z) |
                                       reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(out)) & 15) == 0;
    if (vec) {                                        // lanes per row: the power of two covering P/4, up to 32
        if (P4 <= 1) return launch_vec<1, 1>(a, z, w, eps, out, stream);
        if (P4 <= 2) return launch_vec<2, 1>(a, z, w, eps, out, stream);
        if (P4 <= 4) return launch_vec<4, 1>(a, z, w, eps, out, stream);
        if (P4 <= 8) return launch_vec<8, 1>(a, z, w, eps, out, stream);
        if (P4 <= 16) return launch_vec<16, 1>(a, z, w, eps, out, stream);
        if (P4 <= 32) return launch_vec<32, 1>(a, z, w, eps, out, stream);
        if (P4 <= 64) return launch_vec<32, 2>(a, z, w, eps, out, stream);
        if (P4 <= 128) return launch_vec<32, 4>(a, z, w, eps, out, stream);
    }
    const long long rows_per_seq = ((long long)a.n_tokens * a.H + a.n_seqs - 1) / a.n_seqs;
    const long long gx = (rows_per_seq + kNormWarps - 1) / kNormWarps;
    const dim3 grid((unsigned)(gx < 1 ? 1 : (gx > 4096 ? 4096 : gx)),
                    (unsigned)(a.n_seqs < 65535 ? a.n_seqs : 65535));
    return launch_pdl(gated_norm_kernel, grid, dim3(32 * kNormWarps), 0, stream, a, z, w, eps, out);
}

}  // namespace ssm
