// Warp-per-row decode kernel of the Mamba2 scan (sm_103a).
//
// A decode step (one token per sequence) is almost all state traffic: every
// state row is read from its slot, updated once and written back ("keep the
// Mamba2 scan state in registers", gllm PR 90, "How the layout was chosen").
// So this kernel is laid out for HBM streaming rather than for token reuse:
//   - LANES lanes share one state row; lane j holds the row's float4 chunks
//     j, j+LANES, ... (VPL of them).  With LANES = 32 and d_state = 128 a warp
//     instruction moves one whole 512-byte row: fully coalesced 128-bit loads
//     and stores, no shared-memory tile;
//   - each lane group holds RPT rows and issues all of their slot loads before
//     any arithmetic, so RPT*512 bytes per warp are in flight;
//   - B and C (shared by the heads of a group) and the per-row scalars come
//     through the read-only path and hit in L1/L2 after the first warp.
// A warp's rows always belong to one sequence, so the token loop is uniform
// per warp.  The kernel is correct for any sequence lengths; it is meant for
// length 1.
#include "scan_common.cuh"

namespace ssm {

template <int LANES, int VPL, int RPT, bool EXACT>
__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_kernel(const ScanArgs a, const DecodeGeom geo)
{
    const int N = a.N, N4 = a.N >> 2, P = a.P, H = a.H;
    const int HP = H * P;
    const int heads_per_group = H / a.G;
    const int lane = threadIdx.x & 31;
    const int j = lane % LANES;
    const int lg = lane / LANES;
    const long long warp_id = (long long)blockIdx.x * kDecodeWarps + (threadIdx.x >> 5);
    const long long warp_stride = (long long)gridDim.x * kDecodeWarps;

    for (long long task = warp_id; task < geo.n_tasks; task += warp_stride) {
        const int seq = (int)(task / geo.tasks_per_seq);
        const int tr = (int)(task - (long long)seq * geo.tasks_per_seq);
        const int len = a.seq_lens[seq];
        const int tok_start = a.seq_starts[seq];
        const bool resume = a.resume[seq] != 0;

        int row[RPT], head[RPT];
        bool rvalid[RPT];
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            const int r = tr * geo.rows_per_warp + lg * RPT + q;
            rvalid[q] = r < HP;
            row[q] = rvalid[q] ? r : HP - 1;
            head[q] = row[q] / P;
        }

        // A2: all slot loads of this lane first (RPT*VPL float4 in flight).
        float4 s[RPT][VPL];
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            const float *slot = a.state + ((long long)seq * HP + row[q]) * N;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int c = k * LANES + j;
                s[q][k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (resume && rvalid[q] && (EXACT || c < N4))
                    s[q][k] = *reinterpret_cast<const float4 *>(slot + 4 * c);
            }
        }

        for (int t = 0; t < len; ++t) {
            const long long tok = (long long)tok_start + t;
            float dA[RPT], xdt[RPT], xv[RPT], part[RPT];
#pragma unroll
            for (int q = 0; q < RPT; ++q) {
                const float dtv = __ldg(a.dt + tok * H + head[q]);
                dA[q] = expf(dtv * __ldg(a.A + head[q]));          // A4
                xv[q] = __ldg(a.x + tok * HP + row[q]);
                xdt[q] = dtv * xv[q];
                part[q] = 0.f;
            }
#pragma unroll
            for (int q = 0; q < RPT; ++q) {
                const int g = head[q] / heads_per_group;
                const float *bt = a.B + (tok * a.G + g) * N;
                const float *ct = a.C + (tok * a.G + g) * N;
                float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
                for (int k = 0; k < VPL; ++k) {
                    const int c = k * LANES + j;
                    if (EXACT || c < N4) {
                        const float4 b = __ldg(reinterpret_cast<const float4 *>(bt) + c);
                        const float4 cc = __ldg(reinterpret_cast<const float4 *>(ct) + c);
                        s[q][k].x = fmaf(s[q][k].x, dA[q], xdt[q] * b.x);     // A5
                        s[q][k].y = fmaf(s[q][k].y, dA[q], xdt[q] * b.y);
                        s[q][k].z = fmaf(s[q][k].z, dA[q], xdt[q] * b.z);
                        s[q][k].w = fmaf(s[q][k].w, dA[q], xdt[q] * b.w);
                        acc0 = fmaf(s[q][k].x, cc.x, acc0);                  // A6
                        acc1 = fmaf(s[q][k].y, cc.y, acc1);
                        acc2 = fmaf(s[q][k].z, cc.z, acc2);
                        acc3 = fmaf(s[q][k].w, cc.w, acc3);
                    }
                }
                part[q] = (acc0 + acc1) + (acc2 + acc3);
            }
            const float ysum = reduce_rows<LANES, RPT>(part, j);
            const int qy = reduced_row<LANES, RPT>(j);
            float dxv = xv[0];
            int hy = head[0], ry = row[0];
            bool vy = rvalid[0];
#pragma unroll
            for (int q = 1; q < RPT; ++q)
                if (q == qy) { dxv = xv[q]; hy = head[q]; ry = row[q]; vy = rvalid[q]; }
            if (reduced_writer<LANES, RPT>(j) && vy)
                a.y[tok * HP + ry] = fmaf(__ldg(a.D + hy), dxv, ysum);
        }

        // A7: registers -> slot (coalesced 128-bit stores).
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            if (!rvalid[q])
                continue;
            float *slot = a.state + ((long long)seq * HP + row[q]) * N;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int c = k * LANES + j;
                if (EXACT || c < N4)
                    *reinterpret_cast<float4 *>(slot + 4 * c) = s[q][k];
            }
        }
    }
}

namespace {

template <int LANES, int VPL, int RPT>
cudaError_t launch_one(const ScanArgs &a, const DecodeGeom &g, int grid, cudaStream_t stream)
{
    const bool exact = (a.N / 4) == LANES * VPL;
    auto kern = exact ? decode_kernel<LANES, VPL, RPT, true> : decode_kernel<LANES, VPL, RPT, false>;
    kern<<<grid, kDecodeWarps * 32, 0, stream>>>(a, g);
    return cudaGetLastError();
}

}  // namespace

#define SSM_DECODE_SHAPES(X) \
    X(1, 1, 1) X(2, 1, 1) X(4, 1, 1) X(8, 1, 1) X(16, 1, 1) X(32, 1, 1) \
    X(32, 2, 1) X(32, 4, 1) X(32, 8, 1) \
    X(32, 1, 2) X(32, 1, 4) X(16, 1, 2) X(32, 2, 2) X(8, 1, 2) X(4, 1, 2) \
    X(16, 2, 1) X(16, 2, 2) X(8, 4, 1)

bool decode_supported(int lanes, int vpl, int rpt)
{
#define X(L, V, R) if (lanes == L && vpl == V && rpt == R) return true;
    SSM_DECODE_SHAPES(X)
#undef X
    return false;
}

cudaError_t launch_decode(const ScanArgs &a, const DecodeGeom &g, int lanes, int vpl, int rpt,
                          int grid, cudaStream_t stream)
{
#define X(L, V, R) if (lanes == L && vpl == V && rpt == R) return launch_one<L, V, R>(a, g, grid, stream);
    SSM_DECODE_SHAPES(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace ssm
