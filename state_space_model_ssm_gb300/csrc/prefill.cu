// Chunk-staged prefill kernel of the Mamba2 scan (sm_103a).
//
// One thread block owns one sequence and a run of `rows_per_cta` contiguous
// state rows inside one group (so every row of the block uses the same B and
// C).  The rows' state stays in registers for the whole sequence:
//   - a row is split over LANES adjacent lanes; lane j of the row holds the
//     float4 chunks j, j+LANES, j+2*LANES, ... of the row's d_state elements
//     (VPL of them).  Interleaving at float4 granularity keeps the slot
//     load/store coalesced per instruction and makes the lanes of a row read
//     consecutive 16-byte words of a staged B/C row (no bank conflicts, no
//     padding);
//   - a lane holds RPT rows, which reuse each B/C value it reads from shared
//     memory.
// Tokens are processed in chunks of `chunk`: B, C and the block's x are
// copied to shared memory with cp.async one chunk ahead (double buffer); dt
// is read one chunk ahead into registers and turned into dA = exp(dt*A) once
// per (token, head).  y is a shuffle reduction over the lanes of a row, staged
// in shared memory and written back coalesced after each chunk.
//
// Prior art: the register-state, chunk-staged scan of gllm PR 90 ("What
// changes": contiguous 32-float lane slices with 4-float padding, 25 tokens
// per 32 KiB chunk).  Here the lane slices are interleaved float4 chunks
// instead (conflict-free without padding and coalesced in the slot), the
// chunk is sized for sm_103a's shared memory, and dA is hoisted out of the
// per-row loop (the TODO of "The llama journey", Day 13).
#include "scan_common.cuh"

namespace ssm {

namespace {

// Shared-memory carve-up: two staging buffers (B, C, x, dt, dA per buffer)
// followed by one y buffer.  Offsets are in floats.
struct PrefillSmem {
    float *base;
    int cb, cx, ch;     // floats per buffer of B (= C), x, dt (= dA)
    __device__ __forceinline__ float *B(int b) const { return base + b * cb; }
    __device__ __forceinline__ float *C(int b) const { return base + 2 * cb + b * cb; }
    __device__ __forceinline__ float *X(int b) const { return base + 4 * cb + b * cx; }
    __device__ __forceinline__ float *Dt(int b) const { return base + 4 * cb + 2 * cx + b * ch; }
    __device__ __forceinline__ float *DA(int b) const { return base + 4 * cb + 2 * cx + 2 * ch + b * ch; }
    __device__ __forceinline__ float *Y() const { return base + 4 * cb + 2 * cx + 4 * ch; }
};

__device__ __forceinline__ PrefillSmem carve(float *base, const PrefillGeom &g, int N)
{
    PrefillSmem s;
    s.base = base;
    s.cb = g.chunk * N;
    s.cx = g.chunk * g.rows_per_cta;
    s.ch = g.chunk * g.heads_cap;
    return s;
}

}  // namespace

size_t prefill_smem_bytes(const PrefillGeom &g, int N)
{
    const size_t per_buf = (size_t)g.chunk * (2 * (size_t)N + g.rows_per_cta + 2 * (size_t)g.heads_cap);
    return (2 * per_buf + (size_t)g.chunk * g.rows_per_cta) * sizeof(float);
}

template <int LANES, int VPL, int RPT, bool EXACT>
__global__ void __launch_bounds__(256, 1)
prefill_kernel(const ScanArgs a, const PrefillGeom geo)
{
    griddep_entry();
    extern __shared__ __align__(16) float smem[];
    const int N = a.N, N4 = a.N >> 2, P = a.P, H = a.H;
    const long long HP = (long long)H * P;
    const PrefillSmem sm = carve(smem, geo, N);

    // ---- work mapping: (sequence, group, run of rows) ----
    const int ctas_per_seq = a.G * geo.runs_per_group;
    const int seq = blockIdx.x / ctas_per_seq;
    const int rem = blockIdx.x - seq * ctas_per_seq;
    const int grp = rem / geo.runs_per_group;
    const int run = rem - grp * geo.runs_per_group;
    const int r0 = grp * geo.rows_per_group + run * geo.rows_per_cta;     // first row
    const int nrows = min(geo.rows_per_cta, geo.rows_per_group - run * geo.rows_per_cta);
    const int h0 = r0 / P;
    const int nheads = (r0 + nrows - 1) / P - h0 + 1;

    const int tok_start = a.seq_starts[seq];
    const int len = a.seq_lens[seq];
    const bool resume = a.resume[seq] != 0;

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int j = lane % LANES;                                   // lane within the row group
    const int lg = (warp * (32 / LANES)) + lane / LANES;          // row group within the block
    // RPT contiguous rows per lane group
    int rl[RPT], hl[RPT];
    bool rvalid[RPT];
    float Dv[RPT];
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
        const int r = lg * RPT + q;
        rvalid[q] = r < nrows;
        rl[q] = rvalid[q] ? r : (nrows - 1);
        hl[q] = (r0 + rl[q]) / P - h0;
        Dv[q] = a.D[h0 + hl[q]];
    }

    // ---- state load (A2): slot -> registers, or zero for a fresh sequence ----
    float4 s[RPT][VPL];
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
        const float *slot = a.state + ((long long)seq * HP + r0 + rl[q]) * N;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int c = k * LANES + j;
            s[q][k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (resume && rvalid[q] && (EXACT || c < N4))
                s[q][k] = *reinterpret_cast<const float4 *>(slot + 4 * c);
        }
    }

    const float *Bg = a.B + (long long)grp * N;
    const float *Cg = a.C + (long long)grp * N;
    const long long tokN = (long long)a.G * N;            // B/C token stride
    const float Ah_first = a.A[h0];

    // Stage chunk `c0` (tokens [c0*chunk, ...)) of B, C and x into buffer `buf`.
    auto stage = [&](int c0, int buf) {
        const int t0 = c0 * geo.chunk;
        const int cnt = min(geo.chunk, len - t0);
        const long long tok0 = (long long)tok_start + t0;
        // B and C: cnt rows of N4 float4
        {
            int t = tid / N4, v = tid - (tid / N4) * N4;
            const int dt_ = nthr / N4, dv = nthr - dt_ * N4;
            for (; t < cnt;) {
                const long long goff = (tok0 + t) * tokN + 4 * v;
                cp_async16(sm.B(buf) + t * N + 4 * v, Bg + goff);
                cp_async16(sm.C(buf) + t * N + 4 * v, Cg + goff);
                t += dt_;
                v += dv;
                if (v >= N4) { v -= N4; ++t; }
            }
        }
        // x: cnt rows of nrows floats
        {
            int t = tid / nrows, r = tid - (tid / nrows) * nrows;
            const int dt_ = nthr / nrows, dr = nthr - dt_ * nrows;
            for (; t < cnt;) {
                cp_async4(sm.X(buf) + t * geo.rows_per_cta + r, a.x + (tok0 + t) * HP + r0 + r);
                t += dt_;
                r += dr;
                if (r >= nrows) { r -= nrows; ++t; }
            }
        }
        cp_async_commit();
    };

    // dt of chunk c0 -> registers (one (token, head) pair per thread and pass).
    constexpr int kDtRegs = 4;
    float dtr[kDtRegs];
    auto load_dt = [&](int c0) {
        const int t0 = c0 * geo.chunk;
        const int cnt = min(geo.chunk, len - t0);
#pragma unroll
        for (int u = 0; u < kDtRegs; ++u) {
            const int idx = tid + u * nthr;
            dtr[u] = 0.f;
            if (idx < cnt * nheads) {
                const int t = idx / nheads, hh = idx - t * nheads;
                dtr[u] = a.dt[((long long)tok_start + t0 + t) * H + h0 + hh];
            }
        }
    };
    auto store_dt = [&](int c0, int buf) {
        const int t0 = c0 * geo.chunk;
        const int cnt = min(geo.chunk, len - t0);
#pragma unroll
        for (int u = 0; u < kDtRegs; ++u) {
            const int idx = tid + u * nthr;
            if (idx < cnt * nheads) {
                const int t = idx / nheads, hh = idx - t * nheads;
                const float Ah = (hh == 0) ? Ah_first : a.A[h0 + hh];
                sm.Dt(buf)[t * geo.heads_cap + hh] = dtr[u];
                sm.DA(buf)[t * geo.heads_cap + hh] = expf(dtr[u] * Ah);   // A4
            }
        }
    };

    const int n_chunks = (len + geo.chunk - 1) / geo.chunk;
    if (n_chunks > 0) {
        stage(0, 0);
        load_dt(0);
        store_dt(0, 0);
    }
    const int yrow_q = reduced_row<LANES, RPT>(j);
    const int yrow = lg * RPT + yrow_q;                       // block-local row of my reduced sum
    const bool ywriter = reduced_writer<LANES, RPT>(j) && yrow < nrows;

    for (int c = 0; c < n_chunks; ++c) {
        const int buf = c & 1;
        const bool more = (c + 1) < n_chunks;
        if (more) {
            stage(c + 1, buf ^ 1);     // A3: next chunk in flight during this one
            load_dt(c + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();               // chunk c visible to every thread

        const int cnt = min(geo.chunk, len - c * geo.chunk);
        const float *sB = sm.B(buf), *sC = sm.C(buf), *sX = sm.X(buf);
        const float *sDt = sm.Dt(buf), *sDA = sm.DA(buf);
#pragma unroll 4
        for (int tt = 0; tt < cnt; ++tt) {
            float dA[RPT], xdt[RPT], xv[RPT];
#pragma unroll
            for (int q = 0; q < RPT; ++q) {
                dA[q] = sDA[tt * geo.heads_cap + hl[q]];
                xv[q] = sX[tt * geo.rows_per_cta + rl[q]];
                xdt[q] = sDt[tt * geo.heads_cap + hl[q]] * xv[q];
            }
            float acc[RPT][4];
#pragma unroll
            for (int q = 0; q < RPT; ++q)
                acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
            const float *bt = sB + tt * N;
            const float *ct = sC + tt * N;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int cidx = k * LANES + j;
                if (EXACT || cidx < N4) {
                    const float4 b = *reinterpret_cast<const float4 *>(bt + 4 * cidx);
                    const float4 cc = *reinterpret_cast<const float4 *>(ct + 4 * cidx);
#pragma unroll
                    for (int q = 0; q < RPT; ++q) {          // A5 + A6 partial dot
                        s[q][k].x = fmaf(s[q][k].x, dA[q], xdt[q] * b.x);
                        s[q][k].y = fmaf(s[q][k].y, dA[q], xdt[q] * b.y);
                        s[q][k].z = fmaf(s[q][k].z, dA[q], xdt[q] * b.z);
                        s[q][k].w = fmaf(s[q][k].w, dA[q], xdt[q] * b.w);
                        acc[q][0] = fmaf(s[q][k].x, cc.x, acc[q][0]);
                        acc[q][1] = fmaf(s[q][k].y, cc.y, acc[q][1]);
                        acc[q][2] = fmaf(s[q][k].z, cc.z, acc[q][2]);
                        acc[q][3] = fmaf(s[q][k].w, cc.w, acc[q][3]);
                    }
                }
            }
            float part[RPT];
#pragma unroll
            for (int q = 0; q < RPT; ++q)
                part[q] = (acc[q][0] + acc[q][1]) + (acc[q][2] + acc[q][3]);
            const float ysum = reduce_rows<LANES, RPT>(part, j);
            if (ywriter) {
                float dxv = xv[0], dd = Dv[0];
#pragma unroll
                for (int q = 1; q < RPT; ++q)
                    if (q == yrow_q) { dxv = xv[q]; dd = Dv[q]; }
                sm.Y()[tt * geo.rows_per_cta + yrow] = fmaf(dd, dxv, ysum);
            }
        }
        if (more)
            store_dt(c + 1, buf ^ 1);
        __syncthreads();               // y of chunk c complete; buffer c free

        // y of chunk c: shared -> global, coalesced along the rows
        const long long tok0 = (long long)tok_start + c * geo.chunk;
        {
            int t = tid / nrows, r = tid - (tid / nrows) * nrows;
            const int dt_ = nthr / nrows, dr = nthr - dt_ * nrows;
            for (; t < cnt;) {
                a.y[(tok0 + t) * HP + r0 + r] = sm.Y()[t * geo.rows_per_cta + r];
                t += dt_;
                r += dr;
                if (r >= nrows) { r -= nrows; ++t; }
            }
        }
    }

    // ---- state store (A7): registers -> slot ----
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
        if (!rvalid[q])
            continue;
        float *slot = a.state + ((long long)seq * HP + r0 + rl[q]) * N;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int c = k * LANES + j;
            if (EXACT || c < N4)
                *reinterpret_cast<float4 *>(slot + 4 * c) = s[q][k];
        }
    }
}

// ---------------------------------------------------------------------------
// Host side: instantiated shapes and the launcher.

namespace {

template <int LANES, int VPL, int RPT>
cudaError_t launch_one(const ScanArgs &a, const PrefillGeom &g, size_t smem, cudaStream_t stream)
{
    const bool exact = (a.N / 4) == LANES * VPL;
    const int threads = (g.rows_per_cta / RPT) * LANES;
    const int ctas_per_seq = a.G * g.runs_per_group;
    const dim3 grid((unsigned)((long long)a.n_seqs * ctas_per_seq));
    auto kern = exact ? prefill_kernel<LANES, VPL, RPT, true> : prefill_kernel<LANES, VPL, RPT, false>;
    if (smem > 48 * 1024) {
        cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(kern), smem);
        if (e != cudaSuccess)
            return e;
    }
    return launch_pdl(kern, grid, dim3(threads), smem, stream, a, g);
}

}  // namespace

#define SSM_PREFILL_SHAPES(X) \
    X(1, 1, 1) X(1, 2, 1) X(1, 4, 1) X(1, 8, 1) \
    X(2, 8, 1) X(4, 8, 1) X(8, 8, 1) X(16, 8, 1) X(32, 8, 1) \
    X(8, 4, 1) X(16, 2, 1) X(32, 1, 1) \
    X(8, 4, 2) X(16, 2, 4) X(8, 2, 2) X(4, 8, 2)

bool prefill_supported(int lanes, int vpl, int rpt)
{
#define X(L, V, R) if (lanes == L && vpl == V && rpt == R) return true;
    SSM_PREFILL_SHAPES(X)
#undef X
    return false;
}

cudaError_t launch_prefill(const ScanArgs &a, const PrefillGeom &g, int lanes, int vpl, int rpt,
                           size_t smem, int /*sms*/, cudaStream_t stream)
{
#define X(L, V, R) if (lanes == L && vpl == V && rpt == R) return launch_one<L, V, R>(a, g, smem, stream);
    SSM_PREFILL_SHAPES(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace ssm
