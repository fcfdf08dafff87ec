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
// per warp, and a lane group's RPT rows to one head, so dt, dA, B and C are
// loaded once per lane group and token.  The kernel is correct for any
// sequence lengths; it is meant for length 1, and for the short runs of a
// speculative verify step, where it can also write the state after every
// token (snapshots) straight from the registers.
#include "scan_common.cuh"

namespace ssm {

template <int LANES, int VPL, int RPT, bool EXACT>
__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_kernel(const ScanArgs a, const DecodeGeom geo)
{
    griddep_entry();
    const int N = a.N, N4 = a.N >> 2, P = a.P, H = a.H;
    const int HP = H * P;
    const int lane = threadIdx.x & 31;
    const int j = lane % LANES;
    const int lg = lane / LANES;
    const int task = blockIdx.x * kDecodeWarps + (threadIdx.x >> 5);   // warp within a sequence
    if (task >= geo.tasks_per_seq)
        return;                                                       // whole warp
    // The RPT rows of a lane group are consecutive and, because RPT divides P
    // (checked by the host), belong to one head and so to one group.
    const int row0 = task * geo.rows_per_warp + lg * RPT;
    const bool valid = row0 < HP;                                     // all RPT rows or none
    const int r0 = valid ? row0 : HP - RPT;
    const int head = r0 / P;
    const int grp = head / (H / a.G);
    const float Ah = __ldg(a.A + head);
    const float Dh = __ldg(a.D + head);

    for (int seq = blockIdx.y; seq < a.n_seqs; seq += gridDim.y) {
        const int len = a.seq_lens[seq];
        const int tok_start = a.seq_starts[seq];
        const bool resume = a.resume[seq] != 0;
        float *slot = a.state + ((long long)seq * HP + r0) * N;

        // A2: every slot load of this lane first (RPT*VPL float4 in flight).
        float4 s[RPT][VPL];
#pragma unroll
        for (int q = 0; q < RPT; ++q)
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int c = k * LANES + j;
                s[q][k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (resume && valid && (EXACT || c < N4))
                    s[q][k] = __ldcs(reinterpret_cast<const float4 *>(slot + (long long)q * N + 4 * c));
            }

        for (int t = 0; t < len; ++t) {
            const long long tok = (long long)tok_start + t;
            const float dtv = __ldg(a.dt + tok * H + head);
            const float dA = expf(dtv * Ah);                               // A4
            const float4 *bt = reinterpret_cast<const float4 *>(a.B + (tok * a.G + grp) * N);
            const float4 *ct = reinterpret_cast<const float4 *>(a.C + (tok * a.G + grp) * N);
            float xv[RPT], part[RPT];
#pragma unroll
            for (int q = 0; q < RPT; ++q)
                xv[q] = __ldg(a.x + tok * HP + r0 + q);
            float4 b[VPL], cc[VPL];
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int c = k * LANES + j;
                if (EXACT || c < N4) {
                    b[k] = __ldg(bt + c);
                    cc[k] = __ldg(ct + c);
                }
            }
#pragma unroll
            for (int q = 0; q < RPT; ++q) {
                const float xdt = dtv * xv[q];
                float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
                for (int k = 0; k < VPL; ++k) {
                    const int c = k * LANES + j;
                    if (EXACT || c < N4) {
                        s[q][k].x = fmaf(s[q][k].x, dA, xdt * b[k].x);          // A5
                        s[q][k].y = fmaf(s[q][k].y, dA, xdt * b[k].y);
                        s[q][k].z = fmaf(s[q][k].z, dA, xdt * b[k].z);
                        s[q][k].w = fmaf(s[q][k].w, dA, xdt * b[k].w);
                        acc0 = fmaf(s[q][k].x, cc[k].x, acc0);                  // A6
                        acc1 = fmaf(s[q][k].y, cc[k].y, acc1);
                        acc2 = fmaf(s[q][k].z, cc[k].z, acc2);
                        acc3 = fmaf(s[q][k].w, cc[k].w, acc3);
                    }
                }
                part[q] = (acc0 + acc1) + (acc2 + acc3);
            }
            const float ysum = reduce_rows<LANES, RPT>(part, j);
            const int qy = reduced_row<LANES, RPT>(j);
            float dxv = xv[0];
#pragma unroll
            for (int q = 1; q < RPT; ++q)
                if (q == qy) dxv = xv[q];
            if (reduced_writer<LANES, RPT>(j) && valid)
                a.y[tok * HP + r0 + qy] = fmaf(Dh, dxv, ysum);
            if (a.snaps && valid) {                                       // state after token t
                float *sn = a.snaps + (tok * HP + r0) * N;
#pragma unroll
                for (int q = 0; q < RPT; ++q)
#pragma unroll
                    for (int k = 0; k < VPL; ++k) {
                        const int c = k * LANES + j;
                        if (EXACT || c < N4)
                            __stcs(reinterpret_cast<float4 *>(sn + (long long)q * N + 4 * c), s[q][k]);
                    }
            }
        }

        // A7: registers -> slot (coalesced 128-bit stores).
        if (valid) {
#pragma unroll
            for (int q = 0; q < RPT; ++q)
#pragma unroll
                for (int k = 0; k < VPL; ++k) {
                    const int c = k * LANES + j;
                    if (EXACT || c < N4)
                        __stcs(reinterpret_cast<float4 *>(slot + (long long)q * N + 4 * c), s[q][k]);
                }
        }
    }
}

namespace {

template <int LANES, int VPL, int RPT>
cudaError_t launch_one(const ScanArgs &a, const DecodeGeom &g, int grid_seqs, cudaStream_t stream)
{
    const bool exact = (a.N / 4) == LANES * VPL;
    auto kern = exact ? decode_kernel<LANES, VPL, RPT, true> : decode_kernel<LANES, VPL, RPT, false>;
    const dim3 grid((unsigned)((g.tasks_per_seq + kDecodeWarps - 1) / kDecodeWarps), (unsigned)grid_seqs);
    return launch_pdl(kern, grid, dim3(kDecodeWarps * 32), 0, stream, a, g);
}

}  // namespace

#define SSM_DECODE_SHAPES(X) \
    X(1, 1, 1) X(2, 1, 1) X(4, 1, 1) X(8, 1, 1) X(16, 1, 1) X(32, 1, 1) \
    X(32, 2, 1) X(32, 4, 1) X(32, 8, 1) \
    X(32, 1, 2) X(32, 1, 4) X(16, 1, 2) X(32, 2, 2) X(8, 1, 2) X(4, 1, 2) \
    X(16, 2, 1) X(16, 2, 2) X(8, 4, 1) X(32, 1, 8)

bool decode_supported(int lanes, int vpl, int rpt)
{
#define X(L, V, R) if (lanes == L && vpl == V && rpt == R) return true;
    SSM_DECODE_SHAPES(X)
#undef X
    return false;
}

cudaError_t launch_decode(const ScanArgs &a, const DecodeGeom &g, int lanes, int vpl, int rpt,
                          int grid_seqs, cudaStream_t stream)
{
#define X(L, V, R) if (lanes == L && vpl == V && rpt == R) return launch_one<L, V, R>(a, g, grid_seqs, stream);
    SSM_DECODE_SHAPES(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace ssm
