// The scan in chunked matrix form on the TF32 tensor cores (sm_103a).
//
// The gllm PR 90 page ("keep the Mamba2 scan state in registers, stage tokens
// by chunk", "What changes" and "Not in this PR") names Mamba2's SSD
// chunked-matmul algorithm as the way to parallelise prefill over time but
// gives no algorithm.  This file derives it from the recurrence of "The llama
// journey", Day 14, by unrolling it inside a chunk of Q tokens of one
// sequence.  With a_t = sum_{s<=t} dt_s A[h] (chunk-local, inclusive):
//
//   S_t   = exp(a_t) S_in + sum_{s<=t} exp(a_t - a_s) dt_s x_s (x) B_s
//   y_t   = exp(a_t) S_in.C_t + sum_{s<=t} exp(a_t - a_s) dt_s (C_t.B_s) x_s + D x_t
//   S_out = exp(a_last) S_in + dS,   dS = sum_s exp(a_last - a_s) dt_s x_s (x) B_s
//
// The dense contractions (C B^T per group, the masked decay-weighted
// (C B^T) X, S_in C^T and X^T B) run as mma.sync m16n8k8 with TF32 operands
// (rounded to nearest) and fp32 accumulation; the pass over chunks,
// S_in[k+1] = exp(a_last,k) S_in[k] + dS_k, is serial and stays in fp32.
//
// Three kernels after the plan kernel of segments.cu (here with the chunk as
// the segment length):
//   chunk-state   dS_k and a_last,k per (chunk, head)       -> workspace
//   state pass    in place dS_k -> S_in[k]; final state     -> slot
//   output        y per (chunk, head) from S_in[k]          -> y
// A block of the chunk-state and output kernels handles one chunk, one group
// and a run of that group's heads, so B and C are staged (and C B^T formed)
// once for all of those heads.
#include "ssd_common.cuh"

namespace ssm {

namespace {

using namespace ssd;

constexpr int kStateThreads = 256;

// The chunk-state product for the items (16 head-dim rows x 4 column blocks)
// of one warp: dS[p][n] = sum_s Xw[s][p] Bs[s][n].  FULL: every item has its 4
// column blocks (d_state padded to a multiple of 32), so no per-block guard.
template <bool FULL>
__device__ __forceinline__ void state_items(const float *Xw, const float *Bs, int PS, int NS, float *dS0, int N,
                                            int items, int ngroups, int nblocks, int ksteps, int warp, int gq,
                                            int tq)
{
    for (int it = warp; it < items; it += kStateThreads / 32) {
        const int mb = it / ngroups, ng = it - mb * ngroups;
        const int jn = FULL ? 4 : min(4, nblocks - 4 * ng);
        float acc[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        const float *xr = Xw + tq * PS + 16 * mb + gq;
        const float *br = Bs + tq * NS + 32 * ng + gq;
#pragma unroll 2
        for (int ks = 0; ks < ksteps; ++ks, xr += 8 * PS, br += 8 * NS) {
            // A[m = p][k = s] = Xw[s][p];  B[k = s][n] = Bs[s][n]
            const uint32_t a0 = fb(xr[0]), a1 = fb(xr[8]), a2 = fb(xr[4 * PS]), a3 = fb(xr[4 * PS + 8]);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (FULL || j < jn)
                    mma_tf32(acc[j], a0, a1, a2, a3, fb(br[8 * j]), fb(br[4 * NS + 8 * j]));
        }
        float *dst = dS0 + (size_t)(16 * mb + gq) * N;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = 8 * (4 * ng + j) + 2 * tq;
            if (n < N) {
                *reinterpret_cast<float2 *>(dst + n) = make_float2(acc[j][0], acc[j][1]);
                *reinterpret_cast<float2 *>(dst + 8 * N + n) = make_float2(acc[j][2], acc[j][3]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Chunk-state kernel: dS[p][n] = sum_s w_s x_s[p] B_s[n] with
// w_s = exp(a_last - a_s) dt_s, as the product (w X)^T B (M = P, N = d_state,
// K = chunk tokens).  grid (unit, group, head run), 8 warps; a warp owns
// 16 head-dim rows x 32 state columns of dS per item.  B is staged once per
// block; the x tile of the next head is copied while this head's product runs
// (state_buffers == 2).
template <int Q>
__global__ void __launch_bounds__(kStateThreads)
ssd_chunk_state_kernel(const ScanArgs a, const SsdPlan p, const SsdGeom sg)
{
    griddep_entry();
    extern __shared__ float4 smem4[];
    const int NS = sg.bs_stride, PS = sg.xw_stride, nbuf = sg.state_buffers;
    float *Bs = reinterpret_cast<float *>(smem4);     // [Q][NS]     B_s[n] (tf32)
    float *Xw0 = Bs + Q * NS;                         // [Q][PS] x nbuf  w_s x_s[p] (tf32)
    float *wv = Xw0 + nbuf * Q * PS;                  // [2][Q]      w_s

    ChunkRange c;
    if (!chunk_of(a, p, blockIdx.x, c))
        return;
    const int g = blockIdx.y, hpg = a.H / a.G;
    const int hl0 = blockIdx.z * sg.heads_per_cta, hl1 = min(hpg, hl0 + sg.heads_per_cta);
    if (hl0 >= hl1)
        return;
    const int nh = hl1 - hl0;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    const int N = a.N, P = a.P, N4 = N >> 2, Np4 = sg.n_pad >> 2, P4 = P >> 2;

    if (c.len == 0) {                                 // empty sequence: dS = 0, a_last = 0
        for (int k = 0; k < nh; ++k) {
            const int h = g * hpg + hl0 + k;
            float4 *dst = reinterpret_cast<float4 *>(p.chunk_state + ((size_t)blockIdx.x * a.H + h) * (size_t)P * N);
            for (int i = tid; i < P * N4; i += kStateThreads)
                dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (tid == 0)
                p.chunk_logdecay[(size_t)blockIdx.x * a.H + h] = 0.f;
        }
        return;
    }

    const RowMap wB = row_map(Np4, lane, warp, kStateThreads / 32);
    const RowMap wX = row_map(P4, lane, warp, kStateThreads / 32);
    rows_copy(Bs, NS, a.B + ((size_t)c.t0 * a.G + g) * N, (size_t)a.G * N, Q, Np4, c.len, N4, wB);
    cp_async_commit();
    auto xbuf = [&](int k) { return Xw0 + ((nbuf == 2 && (k & 1)) ? Q * PS : 0); };
    auto issue = [&](int k) {
        const int h = g * hpg + hl0 + k;
        rows_copy(xbuf(k), PS, a.x + ((size_t)c.t0 * a.H + h) * P, (size_t)a.H * P, Q, P4, c.len, P4, wX);
        cp_async_commit();
    };
    issue(0);
    cp_async_wait<1>();
    rows_round(Bs, NS, Q, Np4, wB);

    const int mblocks = P >> 4, nblocks = sg.n_pad >> 3, ngroups = (nblocks + 3) >> 2;
    const int items = mblocks * ngroups, ksteps = (c.len + 7) >> 3;
    for (int k = 0; k < nh; ++k) {
        const int h = g * hpg + hl0 + k;
        float *Xw = xbuf(k);
        float *w = wv + (k & 1) * Q;
        if (warp == 0) {
            ChunkDecay<Q> cd;
            chunk_decay<Q>(a, c, h, lane, cd);
#pragma unroll
            for (int r = 0; r < ChunkDecay<Q>::R; ++r)
                w[lane * ChunkDecay<Q>::R + r] = expf(cd.last - cd.a[r]) * cd.d[r];
            if (lane == 0)
                p.chunk_logdecay[(size_t)blockIdx.x * a.H + h] = cd.last;
        }
        cp_async_wait<0>();
        __syncthreads();                              // w, rounded B, head k's x copies; head k-1 done
        rows_scale_round(Xw, PS, Q, P4, wX, w);
        if (nbuf == 2 && k + 1 < nh)
            issue(k + 1);
        __syncthreads();

        float *dS0 = p.chunk_state + ((size_t)blockIdx.x * a.H + h) * (size_t)P * N;
        if ((nblocks & 3) == 0)
            state_items<true>(Xw, Bs, PS, NS, dS0, N, items, ngroups, nblocks, ksteps, warp, gq, tq);
        else
            state_items<false>(Xw, Bs, PS, NS, dS0, N, items, ngroups, nblocks, ksteps, warp, gq, tq);
        if (nbuf == 1 && k + 1 < nh) {
            __syncthreads();                          // everyone done with the only x buffer
            issue(k + 1);
        }
    }
}

// ---------------------------------------------------------------------------
// State pass, in place over the units of each sequence:
//   S = slot (resume) or 0;  for k: tmp = dS_k; W_k = S; S = exp(a_last,k) S + tmp;
//   slot = S.
// W_k (the incoming state of chunk k) is stored rounded to TF32: the output
// kernels use it only as an operand of C S_in^T, whose operands are TF32, so
// they need not round it again; the chain itself runs on the unrounded S.
// One thread per float4 of a state slot.  The chain is serial in k but its
// loads are not: a thread copies the dS_k of up to kPassBatch chunks into its
// own column of shared memory with cp.async (no registers held while they fly)
// and only then runs the chain, so a sequence of 32 chunks waits on one memory
// latency, not 32.
constexpr int kPassThreads = 128;
constexpr int kPassBatch = 32;

__global__ void __launch_bounds__(kPassThreads)
ssd_state_pass_kernel(const ScanArgs a, const SsdPlan p, int max_units)
{
    griddep_entry();
    extern __shared__ float4 pass_buf[];               // [kPassBatch][kPassThreads]
    const int N4 = a.N >> 2;
    const long long slot4 = (long long)a.H * a.P * N4;
    const long long e = (long long)blockIdx.x * kPassThreads + threadIdx.x;
    if (e >= slot4 || call_failed(p.status))          // chunk states not valid: slots stay as they were
        return;
    const int head = (int)((e / N4) / a.P);
    float4 *W = reinterpret_cast<float4 *>(p.chunk_state);
    float4 *mine = pass_buf + threadIdx.x;
    for (int seq = blockIdx.y; seq < a.n_seqs; seq += gridDim.y) {
        const int b = p.unit_base[seq];
        const int nu = p.unit_base[seq + 1] - b;
        if (nu <= 0 || b < 0 || b + nu > max_units)
            continue;
        float4 *slot = reinterpret_cast<float4 *>(a.state) + (long long)seq * slot4 + e;
        float4 S = a.resume[seq] ? *slot : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k0 = 0; k0 < nu; k0 += kPassBatch) {
            const int n = min(kPassBatch, nu - k0);
            for (int j = 0; j < n; ++j)
                cp_async16(mine + j * kPassThreads, W + (long long)(b + k0 + j) * slot4 + e);
            cp_async_commit();
            float ld[kPassBatch];
#pragma unroll
            for (int j = 0; j < kPassBatch; ++j)
                ld[j] = j < n ? p.chunk_logdecay[(long long)(b + k0 + j) * a.H + head] : 0.f;
            cp_async_wait<0>();
#pragma unroll
            for (int j = 0; j < kPassBatch; ++j) {
                if (j < n) {
                    const float4 d = mine[j * kPassThreads];
                    W[(long long)(b + k0 + j) * slot4 + e] = ssd::tf32_round4(S);   // an operand only
                    const float f = expf(ld[j]);
                    S = make_float4(fmaf(f, S.x, d.x), fmaf(f, S.y, d.y), fmaf(f, S.z, d.z), fmaf(f, S.w, d.w));
                }
            }
        }
        *slot = S;
    }
}

// ---------------------------------------------------------------------------
// Per-warp pieces of the output kernel with compile-time trip counts, so the
// column blocks of a warp's causal row run as straight-line code.  Warp w of
// the output kernel owns rows 16w..16w+15: 2w column blocks left of the
// diagonal and the 1 or 2 diagonal ones (2 unless the chunk ends in row block w).

// G = C B^T for the warp's rows and its first NCB column blocks (NCB even).
template <int NCB, int QB>
__device__ __forceinline__ void form_g(float (&gacc)[QB][4], const float *a_base, const float *bb, int CS,
                                       int kn)
{
#pragma unroll 2
    for (int ks = 0; ks < kn; ++ks) {
        uint32_t af[4];
        ldsm_x4(af, a_base + 8 * ks);
#pragma unroll
        for (int cp = 0; cp < NCB / 2; ++cp) {
            uint32_t bf[4];
            ldsm_x4(bf, bb + 16 * cp * CS + 8 * ks);
            mma_tf32(gacc[2 * cp], af[0], af[1], af[2], af[3], bf[0], bf[1]);
            mma_tf32(gacc[2 * cp + 1], af[0], af[1], af[2], af[3], bf[2], bf[3]);
        }
    }
}

template <int QB, int W = 0>
__device__ __forceinline__ void form_g_warp(int warp, float (&gacc)[QB][4], const float *a_base,
                                            const float *bb, int CS, int kn)
{
    if constexpr (2 * W + 2 <= QB) {
        if (warp == W)
            form_g<2 * W + 2, QB>(gacc, a_base, bb, CS, kn);
        else
            form_g_warp<QB, W + 1>(warp, gacc, a_base, bb, CS, kn);
    }
}

// Decay values of a warp's two accumulator rows (log2 units: a_t log2(e)).
struct RowDecay {
    int tlo, thi;          // chunk rows of accumulator elements 0,1 and 2,3
    float aref;            // a at the warp's first row
    float alo, ahi;        // a at tlo, thi
    float elo, ehi;        // exp(a_t - a_ref)
};

// acc += M x over the warp's causal columns: NOFF blocks left of the
// diagonal, where exp(a_t - a_s) = e_t f_s (f_s = exp(a_ref - a_s)), then
// `ndiag` diagonal blocks with exp(a_t - a_s) taken directly and s > t masked.
// The m16n8 accumulator layout of G is used as the A operand with the k index
// permuted (logical k = tq <-> s = 2tq, k = tq+4 <-> s = 2tq+1); the x rows are
// read in the same order.
template <int NOFF, int QB, int NBY>
__device__ __forceinline__ void causal_mx(float (&yacc)[NBY][4], const float (&gacc)[QB][4], const float *alb,
                                          const float *dtb, const float *X, int XS, int tq, int gq,
                                          const RowDecay &rd, int ndiag)
{
#pragma unroll
    for (int cb = 0; cb < NOFF; ++cb) {
        const int s0 = 8 * cb + 2 * tq;
        const float2 as = *reinterpret_cast<const float2 *>(alb + s0);
        const float2 ds = *reinterpret_cast<const float2 *>(dtb + s0);
        const float f0 = ds.x * ex2(rd.aref - as.x), f1 = ds.y * ex2(rd.aref - as.y);
        const uint32_t a0 = tf32_bits(gacc[cb][0] * (f0 * rd.elo));
        const uint32_t a1 = tf32_bits(gacc[cb][2] * (f0 * rd.ehi));
        const uint32_t a2 = tf32_bits(gacc[cb][1] * (f1 * rd.elo));
        const uint32_t a3 = tf32_bits(gacc[cb][3] * (f1 * rd.ehi));
        const float *xr = X + s0 * XS + gq;
#pragma unroll
        for (int nb = 0; nb < NBY; ++nb)
            mma_tf32(yacc[nb], a0, a1, a2, a3, fb(xr[8 * nb]), fb(xr[XS + 8 * nb]));
    }
#pragma unroll
    for (int d = 0; d < 2; ++d) {
        if (d < ndiag) {
            const int cb = NOFF + d;
            const int s0 = 8 * cb + 2 * tq;
            const float2 as = *reinterpret_cast<const float2 *>(alb + s0);
            const float2 ds = *reinterpret_cast<const float2 *>(dtb + s0);
            const float m00 = s0 <= rd.tlo ? gacc[cb][0] * ds.x * ex2(rd.alo - as.x) : 0.f;
            const float m01 = s0 + 1 <= rd.tlo ? gacc[cb][1] * ds.y * ex2(rd.alo - as.y) : 0.f;
            const float m10 = s0 <= rd.thi ? gacc[cb][2] * ds.x * ex2(rd.ahi - as.x) : 0.f;
            const float m11 = s0 + 1 <= rd.thi ? gacc[cb][3] * ds.y * ex2(rd.ahi - as.y) : 0.f;
            const uint32_t a0 = tf32_bits(m00), a1 = tf32_bits(m10);
            const uint32_t a2 = tf32_bits(m01), a3 = tf32_bits(m11);
            const float *xr = X + s0 * XS + gq;
#pragma unroll
            for (int nb = 0; nb < NBY; ++nb)
                mma_tf32(yacc[nb], a0, a1, a2, a3, fb(xr[8 * nb]), fb(xr[XS + 8 * nb]));
        }
    }
}

template <int QB, int NBY, int W = 0>
__device__ __forceinline__ void causal_mx_warp(int warp, float (&yacc)[NBY][4], const float (&gacc)[QB][4],
                                               const float *alb, const float *dtb, const float *X, int XS,
                                               int tq, int gq, const RowDecay &rd, int ndiag)
{
    if constexpr (2 * W + 2 <= QB) {
        if (warp == W)
            causal_mx<2 * W, QB, NBY>(yacc, gacc, alb, dtb, X, XS, tq, gq, rd, ndiag);
        else
            causal_mx_warp<QB, NBY, W + 1>(warp, yacc, gacc, alb, dtb, X, XS, tq, gq, rd, ndiag);
    }
}

// ---------------------------------------------------------------------------
// Output kernel.  grid (unit, group, head run); Q/16 warps, warp w owns chunk
// rows 16w .. 16w+15.  Per block: G = C B^T (causal part of the warp's rows,
// K = d_state) into registers, once for all heads of the run.  Per head:
//   acc  = C S_in^T                (K = d_state)
//   acc *= exp(a_t)                (row scale)
//   acc += M x   M[t][s] = G[t][s] dt_s exp(a_t - a_s) for s <= t, else 0
//                                  (K = chunk tokens, causal)
//   y    = acc + D x
// M is formed from G's accumulator fragment directly: an m16n8 accumulator
// holds columns (2tq, 2tq+1) where an m16n8k8 A operand wants (tq, tq+4), so
// the k index of that product is permuted (logical k = tq <-> s = 2tq,
// k = tq+4 <-> s = 2tq+1) and the x rows are read in the same order.
// Shared memory: C | RB | RA | a log2(e) [2][Q] | dt [2][Q].  RB holds B until
// G is formed, then the (x, S_in) tiles of odd heads (of every head when
// out_buffers == 1); RA those of even heads, so the next head's tiles are in
// flight while this head's products run.
// NBY = head_dim / 8 exactly.
template <int Q, int NBY>
__global__ void __launch_bounds__(2 * Q)
ssd_output_kernel(const ScanArgs a, const SsdPlan p, const SsdGeom sg)
{
    griddep_entry();
    constexpr int QB = Q / 8;                         // 8-token column blocks per chunk
    constexpr int kThreads = 2 * Q;
    constexpr float kLog2e = 1.4426950408889634f;
    extern __shared__ float4 smem4[];
    const int CS = sg.cs_stride, XS = sg.xs_stride, P = a.P, N = a.N, nbuf = sg.out_buffers;
    const int buf_floats = Q * XS + P * CS;
    float *Cs = reinterpret_cast<float *>(smem4);     // [Q][CS]  C_t[n] (tf32)
    float *RB = Cs + Q * CS;
    float *RA = RB + max(Q * CS, buf_floats);
    float *al = RA + (nbuf == 2 ? buf_floats : 0);    // [2][Q]  a_t log2(e)
    float *dts = al + 2 * Q;                          // [2][Q]  dt_t

    ChunkRange c;
    if (!chunk_of(a, p, blockIdx.x, c) || c.len == 0)
        return;
    const int g = blockIdx.y, hpg = a.H / a.G;
    const int hl0 = blockIdx.z * sg.heads_per_cta, hl1 = min(hpg, hl0 + sg.heads_per_cta);
    if (hl0 >= hl1)
        return;
    const int nh = hl1 - hl0;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (call_failed(p.status)) {                      // the chunk states are not valid
        poison_y(a.y, (long long)a.H * a.P, c.t0, c.len, (g * hpg + hl0) * a.P, nh * a.P, tid, kThreads);
        return;
    }
    const int gq = lane >> 2, tq = lane & 3;
    const int lrow = lane & 7, lmat = lane >> 3;      // ldmatrix: tile and row this lane addresses
    const int N4 = N >> 2, Np4 = sg.n_pad >> 2, P4 = P >> 2;
    const RowMap wC = row_map(Np4, lane, warp, kThreads / 32);
    const RowMap wX = row_map(P4, lane, warp, kThreads / 32);

    auto head_buf = [&](int k) { return (nbuf == 2 && !(k & 1)) ? RA : RB; };
    auto issue = [&](int k) {
        const int h = g * hpg + hl0 + k;
        float *X = head_buf(k);
        rows_copy(X, XS, a.x + ((size_t)c.t0 * a.H + h) * P, (size_t)a.H * P, Q, P4, c.len, P4, wX);
        rows_copy(X + Q * XS, CS, p.chunk_state + ((size_t)blockIdx.x * a.H + h) * (size_t)P * N, N, P, Np4,
                  P, N4, wC);
        cp_async_commit();
    };

    const size_t bc_off = ((size_t)c.t0 * a.G + g) * N;
    rows_copy(Cs, CS, a.C + bc_off, (size_t)a.G * N, Q, Np4, c.len, N4, wC);
    rows_copy(RB, CS, a.B + bc_off, (size_t)a.G * N, Q, Np4, c.len, N4, wC);
    cp_async_commit();
    if (nbuf == 2) {
        issue(0);
        cp_async_wait<1>();
    } else {
        cp_async_wait<0>();
    }
    rows_round(Cs, CS, Q, Np4, wC);
    rows_round(RB, CS, Q, Np4, wC);
    __syncthreads();

    const int r0 = 16 * warp;
    const bool active = r0 < c.len;                   // the warp has rows to write
    const int cb_lim = active ? min(2 * warp + 1, (c.len - 1) >> 3) : -1;
    const int kn = sg.n_pad >> 3;
    // A fragments of C (rows r0..r0+15) at column 8*ks: a_base + 8*ks
    const float *a_base = Cs + (r0 + lrow + 8 * (lmat & 1)) * CS + 4 * (lmat >> 1);
    // B fragments of two 8-row blocks (rows 16*j ..) of an [rows][CS] tile
    const int b_off = (8 * (lmat >> 1) + lrow) * CS + 4 * (lmat & 1);

    float gacc[QB][4];
#pragma unroll
    for (int cb = 0; cb < QB; ++cb)
        gacc[cb][0] = gacc[cb][1] = gacc[cb][2] = gacc[cb][3] = 0.f;
    if (active)
        form_g_warp<QB>(warp, gacc, a_base, RB + b_off, CS, kn);
    if (nbuf == 1) {
        __syncthreads();                              // everyone done with B
        issue(0);
    }

    for (int k = 0; k < nh; ++k) {
        const int h = g * hpg + hl0 + k;
        const int b = k & 1;
        float *X = head_buf(k);
        float *S = X + Q * XS;
        float *alb = al + b * Q, *dtb = dts + b * Q;
        if (warp == 0) {
            ChunkDecay<Q> cd;
            chunk_decay<Q>(a, c, h, lane, cd);
#pragma unroll
            for (int r = 0; r < ChunkDecay<Q>::R; ++r) {
                alb[lane * ChunkDecay<Q>::R + r] = cd.a[r] * kLog2e;
                dtb[lane * ChunkDecay<Q>::R + r] = cd.d[r];
            }
        }
        cp_async_wait<0>();
        rows_round(X, XS, Q, P4, wX);
        rows_round(S, CS, P, Np4, wC);
        __syncthreads();                              // head k ready everywhere; head k-1 done
        if (nbuf == 2 && k + 1 < nh)
            issue(k + 1);

        if (active) {
            // x for the skip term, loaded now so the loads complete under the products
            const int tlo = r0 + gq, thi = tlo + 8;
            const size_t rs = (size_t)a.H * P;
            const float *xg = a.x + ((size_t)c.t0 * a.H + h) * P + 2 * tq;
            float2 xlo[NBY], xhi[NBY];
#pragma unroll
            for (int nb = 0; nb < NBY; ++nb) {
                xlo[nb] = tlo < c.len ? __ldg(reinterpret_cast<const float2 *>(xg + tlo * rs + 8 * nb))
                                      : make_float2(0.f, 0.f);
                xhi[nb] = thi < c.len ? __ldg(reinterpret_cast<const float2 *>(xg + thi * rs + 8 * nb))
                                      : make_float2(0.f, 0.f);
            }
            float yacc[NBY][4];
#pragma unroll
            for (int nb = 0; nb < NBY; ++nb)
                yacc[nb][0] = yacc[nb][1] = yacc[nb][2] = yacc[nb][3] = 0.f;
            const float *sb = S + b_off;
#pragma unroll 2
            for (int ks = 0; ks < kn; ++ks) {
                uint32_t af[4];
                ldsm_x4(af, a_base + 8 * ks);
#pragma unroll
                for (int np = 0; np < NBY / 2; ++np) {
                    uint32_t bf[4];
                    ldsm_x4(bf, sb + 16 * np * CS + 8 * ks);
                    mma_tf32(yacc[2 * np], af[0], af[1], af[2], af[3], bf[0], bf[1]);
                    mma_tf32(yacc[2 * np + 1], af[0], af[1], af[2], af[3], bf[2], bf[3]);
                }
            }
            RowDecay rd;
            rd.tlo = tlo;
            rd.thi = thi;
            rd.aref = alb[r0];
            rd.alo = alb[tlo];
            rd.ahi = alb[thi];
            const float Elo = ex2(rd.alo), Ehi = ex2(rd.ahi);
#pragma unroll
            for (int nb = 0; nb < NBY; ++nb) {
                yacc[nb][0] *= Elo;
                yacc[nb][1] *= Elo;
                yacc[nb][2] *= Ehi;
                yacc[nb][3] *= Ehi;
            }
            rd.elo = ex2(rd.alo - rd.aref);
            rd.ehi = ex2(rd.ahi - rd.aref);
            causal_mx_warp<QB, NBY>(warp, yacc, gacc, alb, dtb, X, XS, tq, gq, rd, cb_lim - 2 * warp + 1);

            const float Dh = a.D[h];
            float *yg = a.y + ((size_t)c.t0 * a.H + h) * P + 2 * tq;
#pragma unroll
            for (int nb = 0; nb < NBY; ++nb) {
                if (tlo < c.len)
                    __stcs(reinterpret_cast<float2 *>(yg + tlo * rs + 8 * nb),
                           make_float2(fmaf(Dh, xlo[nb].x, yacc[nb][0]), fmaf(Dh, xlo[nb].y, yacc[nb][1])));
                if (thi < c.len)
                    __stcs(reinterpret_cast<float2 *>(yg + thi * rs + 8 * nb),
                           make_float2(fmaf(Dh, xhi[nb].x, yacc[nb][2]), fmaf(Dh, xhi[nb].y, yacc[nb][3])));
            }
        }
        if (nbuf == 1 && k + 1 < nh) {
            __syncthreads();                          // everyone done with the only tile pair
            issue(k + 1);
        }
    }
}

template <int Q>
cudaError_t launch_ssd_q(const ScanArgs &a, const SsdPlan &plan, const SsdGeom &g, int max_units,
                         cudaStream_t stream, LaunchTimer *tm, const SegStateMaps *state_maps)
{
    const int hpg = a.H / a.G;
    const dim3 grid((unsigned)max_units, (unsigned)a.G, (unsigned)((hpg + g.heads_per_cta - 1) / g.heads_per_cta));

    cudaError_t e;
    if (state_maps) {
        // The chunk states on the tensor cores: the state pass of the time
        // segments with the chunk as segment, for every chunk (split TF32).
        SegmentPlan sp{};
        sp.units = plan.units;
        sp.n_units = plan.n_units;
        sp.unit_base = plan.unit_base;
        sp.seg_len = plan.chunk;
        sp.seg_state = plan.chunk_state;
        sp.seg_decay = plan.chunk_logdecay;
        sp.status = plan.status;
        sp.fail_waits = plan.fail_waits;
        sp.chunk_states = 1;
        e = timed(tm, [&] { return launch_segment_state_tc(a, sp, *state_maps, max_units, stream); });
    } else {
        auto state_k = ssd_chunk_state_kernel<Q>;
        e = set_dynamic_smem(reinterpret_cast<const void *>(state_k), g.smem_state);
        if (e != cudaSuccess)
            return e;
        e = timed(tm, [&] { return launch_pdl(state_k, grid, dim3(kStateThreads), g.smem_state, stream, a, plan, g); });
    }
    if (e != cudaSuccess)
        return e;

    const long long slot4 = (long long)a.H * a.P * (a.N >> 2);
    const dim3 pgrid((unsigned)((slot4 + kPassThreads - 1) / kPassThreads),
                     (unsigned)(a.n_seqs < 65535 ? a.n_seqs : 65535));
    const int pass_smem = kPassBatch * kPassThreads * (int)sizeof(float4);
    e = set_dynamic_smem(reinterpret_cast<const void *>(ssd_state_pass_kernel), (size_t)pass_smem);
    if (e != cudaSuccess)
        return e;
    e = timed(tm, [&] {
        return launch_pdl(ssd_state_pass_kernel, pgrid, dim3(kPassThreads), (size_t)pass_smem, stream, a, plan,
                          max_units);
    });
    if (e != cudaSuccess)
        return e;

    if (g.use_tc)
        return timed(tm, [&] { return launch_ssd_output_tc(a, plan, g, max_units, stream); });
    void (*out_k)(const ScanArgs, const SsdPlan, const SsdGeom) = nullptr;
    switch (a.P / 8) {
    case 2: out_k = ssd_output_kernel<Q, 2>; break;
    case 4: out_k = ssd_output_kernel<Q, 4>; break;
    case 6: out_k = ssd_output_kernel<Q, 6>; break;
    case 8: out_k = ssd_output_kernel<Q, 8>; break;
    case 10: out_k = ssd_output_kernel<Q, 10>; break;
    case 12: out_k = ssd_output_kernel<Q, 12>; break;
    case 14: out_k = ssd_output_kernel<Q, 14>; break;
    case 16: out_k = ssd_output_kernel<Q, 16>; break;
    default: return cudaErrorInvalidValue;
    }
    e = set_dynamic_smem(reinterpret_cast<const void *>(out_k), g.smem_out);
    if (e != cudaSuccess)
        return e;
    return timed(tm, [&] { return launch_pdl(out_k, grid, dim3(2 * Q), g.smem_out, stream, a, plan, g); });
}

}  // namespace

bool ssd_supported_chunk(int chunk) { return chunk == 64 || chunk == 128; }

int ssd_max_head_dim() { return 128; }

cudaError_t launch_ssd(const ScanArgs &a, const SsdPlan &plan, const SsdGeom &g, int max_units,
                       cudaStream_t stream, LaunchTimer *tm, const SegStateMaps *state_maps)
{
    if (a.P % 16 != 0 || a.P > ssd_max_head_dim())
        return cudaErrorInvalidValue;
    switch (plan.chunk) {
    case 64: return launch_ssd_q<64>(a, plan, g, max_units, stream, tm, state_maps);
    case 128: return launch_ssd_q<128>(a, plan, g, max_units, stream, tm, state_maps);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
