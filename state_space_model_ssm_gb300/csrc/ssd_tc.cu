// Output kernel of the chunked ("SSD") form on the 5th-generation tensor cores
// (tcgen05, sm_103a): the same per-chunk products as the mma.sync kernel of
// ssd.cu, issued by one thread per block with the accumulators (and C) in
// tensor memory (TMEM).
//
// One block per (chunk of 128 tokens, group, run of the group's heads), 8
// warps.  TMEM (one chunk row per lane) holds C itself, as the A operand of
// the two products with C, and three fp32 accumulators:
//   G  = C B^T              128 x 128   (once per block)
//   Yi = C S_in^T           128 x P     (per head)
//   Yx = M x                128 x P     (per head), M[t][s] = G[t][s] dt_s exp(a_t - a_s), s <= t
// and per head y = exp(a_t) Yi + Yx + D x.  Warp w reaches TMEM lanes
// 32 (w % 4) .. +31 (its chunk rows) and handles column half w / 4.
//
// Warps 8-11 copy global memory into shared memory one head ahead (two
// buffers for S_in and the staged x) and signal per-buffer mbarriers; the
// compute warps release a buffer through another mbarrier when its head is
// done.  Warp 12 issues every MMA (one thread) and forms each head's decay
// tables; it and the compute warps hand each other the head's steps through
// mbarriers (C and B ready, decay tables written, M and x^T written, products
// done, accumulators read), so C S_in^T of a head and the next head's decay
// tables run while the compute warps transpose x and form M.
//
// Shared-memory operands are K-major tiles without swizzle: 16-byte rows (4
// fp32 along K) in 8-row core matrices 128 bytes apart, consecutive 16-byte K
// chunks of the tile `lbo` bytes apart.  B and S_in arrive with 16-byte
// cp.async; x is needed with the token (contraction) index along K, so it is
// staged row-major and transposed through registers into a tile whose chunk
// stride is padded by 16 bytes (conflict-free 4-byte writes); M is written by
// the threads that form it from G.  Everything is rounded to TF32 (nearest)
// before the tensor core reads it.  S_in and the staged x of the next head are
// copied while the current head computes (two buffers where they fit).
#include "ssd_common.cuh"
#include "tc_common.cuh"

namespace ssm {

namespace {

using namespace ssd;
using namespace tc;

constexpr int kTcQ = 128;
constexpr int kTcThreads = 256;             // compute warps 0-7 (TMEM rows x column halves)
constexpr int kTcProducers = 4;             // warps 8-11 issue the global -> shared copies
constexpr int kTcMmaWarp = kTcThreads / 32 + kTcProducers;   // warp 12: the MMAs and the decay tables
constexpr int kTcBlock = kTcThreads + 32 * kTcProducers + 32;

// Barrier 2 over the compute warps and the MMA warp: the MMA warp has drained
// its products before the compute warps free TMEM.
__device__ __forceinline__ void mma_compute_sync() { asm volatile("bar.sync 2, 288;\n" ::: "memory"); }

// The same barrier, returning whether any compute thread passed `v` true.
__device__ __forceinline__ bool compute_sync_or(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 256, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}\n"
                 : "=r"(r) : "r"((uint32_t)v) : "memory");
    return r != 0;
}

// Shared-memory layout (bytes) of the block.
struct TcLayout {
    uint32_t BM, S[2], XR[2], XT, al, dts, fcol, bar, tslot, total;   // bar: 12 mbarriers
    uint32_t lc;      // k-chunk stride of the 128-row tiles (B, M)
    uint32_t ls;      // k-chunk stride of S_in (P rows)
    uint32_t lx;      // k-chunk stride of the transposed x tile (P rows + 16 bytes)
};

__host__ __device__ inline TcLayout tc_layout(int n_pad, int P, int nbuf)
{
    auto up = [](uint32_t v) { return (v + 1023u) & ~1023u; };
    TcLayout L;
    L.lc = kTcQ * 16;
    L.ls = (uint32_t)P * 16;
    L.lx = (uint32_t)P * 16 + 16;
    const uint32_t kbm = (uint32_t)(n_pad > kTcQ ? n_pad : kTcQ);
    const uint32_t sbytes = (uint32_t)P * n_pad * 4, xbytes = (uint32_t)kTcQ * P * 4;
    L.BM = 0;
    L.S[0] = up(L.BM + (uint32_t)kTcQ * kbm * 4);
    L.S[1] = nbuf == 2 ? up(L.S[0] + sbytes) : L.S[0];
    L.XR[0] = up(L.S[1] + sbytes);
    L.XR[1] = nbuf == 2 ? up(L.XR[0] + xbytes) : L.XR[0];
    L.XT = up(L.XR[1] + xbytes);
    L.al = up(L.XT + (uint32_t)(kTcQ / 4) * L.lx);
    L.dts = L.al + kTcQ * 4;
    L.fcol = L.dts + kTcQ * 4;
    L.bar = L.fcol + kTcQ * 4;
    L.tslot = L.bar + 96;
    L.total = L.tslot + 16;
    return L;
}

// TMEM columns: C (d_state rounded up to 32), G, Yi, Yx.
__host__ __device__ inline int tc_c_cols(int n_pad) { return (n_pad + 31) & ~31; }
__host__ __device__ inline int tc_tmem_need(int n_pad, int P) { return tc_c_cols(n_pad) + kTcQ + 2 * P; }

// A warp's walk over the cells (i, j) of an (ni x nj) grid in row-major order,
// starting at cell `warp` and stepping by the number of warps, with no
// division per step.
struct CellWalk {
    int i, j, di, dj;
};

__device__ __forceinline__ CellWalk cell_walk(int warp, int nj, int nwarps)
{
    CellWalk w;
    w.i = warp / nj;
    w.j = warp - w.i * nj;
    w.di = nwarps / nj;
    w.dj = nwarps - w.di * nj;
    return w;
}

__device__ __forceinline__ void cell_next(CellWalk &w, int nj)
{
    w.i += w.di;
    w.j += w.dj;
    if (w.j >= nj) {
        w.j -= nj;
        ++w.i;
    }
}

// 16-byte cells (row r, k-chunk j) of a `rows` x (4*w4) K-major tile: warp
// instruction covers 8 rows x 4 chunks (conflict-free 128-byte wavefronts).
// Global row r at g + r*gstride floats; rows >= vrows or chunks >= v4 zero.
__device__ __forceinline__ void kmajor_copy(char *tile, uint32_t lbo, const float *g, size_t gstride, int rows,
                                            int w4, int vrows, int v4, int warp, int lane, int nwarps)
{
    const int jgroups = (w4 + 3) >> 2;
    const int rlo = lane & 7, jlo = lane >> 3;
    for (CellWalk w = cell_walk(warp, jgroups, nwarps); w.i < (rows >> 3); cell_next(w, jgroups)) {
        const int r = 8 * w.i + rlo, j = 4 * w.j + jlo;
        if (j < w4) {
            const bool ok = r < vrows && j < v4;
            cp_async16_zfill(tile + j * lbo + r * 16, ok ? g + (size_t)r * gstride + 4 * j : g, ok ? 16 : 0);
        }
    }
}

__device__ __forceinline__ void kmajor_round(char *tile, uint32_t lbo, int rows, int w4, int warp, int lane)
{
    const int jgroups = (w4 + 3) >> 2;
    const int rlo = lane & 7, jlo = lane >> 3;
    for (CellWalk w = cell_walk(warp, jgroups, kTcThreads / 32); w.i < (rows >> 3); cell_next(w, jgroups)) {
        const int r = 8 * w.i + rlo, j = 4 * w.j + jlo;
        if (j < w4) {
            float4 *q = reinterpret_cast<float4 *>(tile + j * lbo + r * 16);
            *q = tf32_round4(*q);
        }
    }
}

// x of one head, staged row-major: token s, 16-byte chunk j (4 head-dim
// values) at xr + s*P*4 + (j ^ (s & 7))*16 (the XOR spreads a column of chunks
// over all banks).  Tokens >= len are zero.
__device__ __forceinline__ void xraw_copy(char *xr, const float *xh, size_t tstride, int P, int len, int warp,
                                          int lane, int nwarps)
{
    const int P4 = P >> 2;
    for (int i = warp * 32 + lane; i < kTcQ * P4; i += 32 * nwarps) {
        const int s = i / P4, j = i - s * P4;     // P4 is a multiple of 8: a shift and mask after inlining
        const bool ok = s < len;
        cp_async16_zfill(xr + s * P * 4 + ((j ^ (s & 7)) << 4), ok ? xh + (size_t)s * tstride + 4 * j : xh,
                         ok ? 16 : 0);
    }
}

// Transpose the staged x into the K-major operand (row p, token s along K) at
// xt + (s/4)*lx + p*16 + (s%4)*4, rounding to TF32.  Thread (s, half) moves
// the head-dim values of its half of token s: conflict-free 16-byte reads
// (the XOR) and 4-byte writes (lx = 16 mod 128 puts token s on bank s mod 32).
__device__ __forceinline__ void xraw_transpose(char *xt, uint32_t lx, const char *xr, int P, int tid)
{
    const int s = tid & (kTcQ - 1), half = tid >> 7;
    const int P4 = P >> 2, j0 = half * (P4 >> 1), j1 = j0 + (P4 >> 1);
    char *col = xt + (s >> 2) * lx + (s & 3) * 4;
    for (int j = j0; j < j1; ++j) {
        const float4 v = *reinterpret_cast<const float4 *>(xr + s * P * 4 + ((j ^ (s & 7)) << 4));
        *reinterpret_cast<float *>(col + (4 * j) * 16) = tf32_round(v.x);
        *reinterpret_cast<float *>(col + (4 * j + 1) * 16) = tf32_round(v.y);
        *reinterpret_cast<float *>(col + (4 * j + 2) * 16) = tf32_round(v.z);
        *reinterpret_cast<float *>(col + (4 * j + 3) * 16) = tf32_round(v.w);
    }
}

__global__ void __launch_bounds__(kTcBlock, 1)
ssd_output_tc_kernel(const ScanArgs a, const SsdPlan p, const SsdGeom sg)
{
    griddep_entry();
    extern __shared__ __align__(1024) unsigned char tc_smem[];
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
        poison_y(a.y, (long long)a.H * a.P, c.t0, c.len, (g * hpg + hl0) * a.P, nh * a.P, tid, kTcBlock);
        return;
    }
    const int P = a.P, N = a.N, N4 = N >> 2, Np4 = sg.n_pad >> 2;
    const int nbuf = sg.out_buffers;
    const TcLayout L = tc_layout(sg.n_pad, P, nbuf);
    char *sm = reinterpret_cast<char *>(tc_smem);
    char *BMt = sm + L.BM, *XTt = sm + L.XT;
    float *al = reinterpret_cast<float *>(sm + L.al);
    float *dts = reinterpret_cast<float *>(sm + L.dts);
    float *fcol = reinterpret_cast<float *>(sm + L.fcol);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bar);
    uint64_t *bar_g = bars, *bar_mma = bars + 1, *bar_b = bars + 2;
    uint64_t *full = bars + 3, *empty = bars + 5;      // per buffer
    uint64_t *drain = bars + 7;                       // all products issued so far done
    uint64_t *c_ready = bars + 8;                     // C in TMEM, B rounded
    uint64_t *m_ready = bars + 9;                     // per head: M and x^T written
    uint64_t *epi_done = bars + 10;                   // per head: its accumulators read
    uint64_t *dec_full = bars + 11;                   // per head: its decay tables written
    const long cap = p.fail_waits ? 0 : tc::kSpinLimit;   // polls of a pipeline wait
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L.tslot);
    constexpr float kLog2e = 1.4426950408889634f;
    const size_t bc_off = ((size_t)c.t0 * a.G + g) * N;

    if (warp == 0) {
        tmem_alloc(tslot, sg.tmem_cols);
    }
    if (tid == 0) {
        mbar_init(bar_g, 1);
        mbar_init(bar_mma, 1);
        mbar_init(drain, 1);
        mbar_init(bar_b, 32 * kTcProducers);
        for (int i = 0; i < 2; ++i) {
            mbar_init(full + i, 32 * kTcProducers);
            mbar_init(empty + i, kTcThreads);
        }
        mbar_init(c_ready, kTcThreads);
        mbar_init(m_ready, kTcThreads);
        mbar_init(epi_done, kTcThreads);
        mbar_init(dec_full, 32);
        mbar_init_fence();
    }
    __syncthreads();                                  // barriers and the TMEM address published

    // ---- producer warps: B, then S_in and the staged x of each head, one head
    // ahead of the compute warps (two buffers) ----
    if (warp >= kTcThreads / 32 && warp < kTcMmaWarp) {
        const int pw = warp - kTcThreads / 32;
        kmajor_copy(BMt, L.lc, a.B + bc_off, (size_t)a.G * N, kTcQ, Np4, c.len, N4, pw, lane, kTcProducers);
        cp_async_arrive(bar_b);
        for (int k = 0; k < nh; ++k) {
            const int b = nbuf == 2 ? (k & 1) : 0;
            if (k >= nbuf && !mbar_wait(empty + b, (uint32_t)((k / nbuf - 1) & 1), cap))
                break;                                // the compute warps gave up
            const int h = g * hpg + hl0 + k;
            kmajor_copy(sm + (b ? L.S[1] : L.S[0]), L.ls, p.chunk_state + ((size_t)blockIdx.x * a.H + h) * (size_t)P * N,
                        N, P, Np4, P, N4, pw, lane, kTcProducers);
            xraw_copy(sm + (b ? L.XR[1] : L.XR[0]), a.x + ((size_t)c.t0 * a.H + h) * P, (size_t)a.H * P, P, c.len,
                      pw, lane, kTcProducers);
            cp_async_arrive(full + b);
        }
        cp_async_wait<0>();                           // no copy lands after the block has gone
        return;
    }

    tc::fence_after();
    const uint32_t tmem = *tslot;
    const int ccols = tc_c_cols(sg.n_pad);
    const uint32_t tm_c = tmem, tm_g = tmem + ccols, tm_yi = tm_g + kTcQ, tm_yx = tm_yi + P;
    const int ksteps_n = sg.n_pad >> 3;

    // ---- MMA warp: G = C B^T once; per head Yi = C S_in^T as soon as S_in has
    // landed and the previous head's accumulators are read, Yx = M x once M and
    // x^T are written; between them the next head's decay tables ----
    if (warp == kTcMmaWarp) {
        // dt of the next head is loaded (scattered 4-byte reads) one head ahead
        float dt_next[ChunkDecay<kTcQ>::R];
        chunk_dt<kTcQ>(a, c, g * hpg + hl0, lane, dt_next);
        // a_t log2(e), dt_s and the column factors f_s of head k (see M below)
        auto decay_tables = [&](int k) {
            const int h = g * hpg + hl0 + k;
            ChunkDecay<kTcQ> cd;
            chunk_decay_from<kTcQ>(a.A[h], dt_next, lane, cd);
            if (k + 1 < nh)
                chunk_dt<kTcQ>(a, c, h + 1, lane, dt_next);
            // a of the last column of each 16-column piece (lane 4i+3 holds it)
            constexpr int R = ChunkDecay<kTcQ>::R;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int s = lane * R + r;
                const float ar = __shfl_sync(kFullMask, cd.a[R - 1], (s | 15) / R) * kLog2e;
                al[s] = cd.a[r] * kLog2e;
                dts[s] = cd.d[r];
                fcol[s] = cd.d[r] * ex2(ar - cd.a[r] * kLog2e);
            }
            mbar_arrive(dec_full);                    // every lane: its entries are written
        };
        decay_tables(0);
        // descriptors step by 2 K-chunks (8 tokens / state columns) per MMA
        bool mok = __all_sync(kFullMask, mbar_wait(c_ready, 0, cap));
        if (mok && lane == 0) {                       // G = C B^T
            tc::fence_after();
            const uint32_t id = idesc_tf32(kTcQ, kTcQ);
            const uint64_t db = smem_desc(smem_u32(BMt), L.lc, 128);
            for (int kk = 0; kk < ksteps_n; ++kk)
                tc::mma_ts(tm_g, tm_c + 8 * kk, db + (uint64_t)(kk * (2 * L.lc >> 4)), id, kk > 0);
            tc::commit(bar_g);
        }
        for (int k = 0; k < nh && mok; ++k) {
            const int b = nbuf == 2 ? (k & 1) : 0;
            bool got = mbar_wait(full + b, (uint32_t)((k / nbuf) & 1), cap);
            if (k > 0)
                got = mbar_wait(epi_done, (uint32_t)((k - 1) & 1), cap) && got;
            if (!__all_sync(kFullMask, got)) {
                mok = false;                          // a copy never landed or the compute warps gave up
                break;
            }
            if (lane == 0) {                          // Yi = C S_in^T (S_in arrives rounded to TF32)
                tc::fence_after();
                const uint32_t id = idesc_tf32(kTcQ, P);
                const uint64_t ds = smem_desc(smem_u32(sm + (b ? L.S[1] : L.S[0])), L.ls, 128);
                for (int kk = 0; kk < ksteps_n; ++kk)
                    tc::mma_ts(tm_yi, tm_c + 8 * kk, ds + (uint64_t)(kk * (2 * L.ls >> 4)), id, kk > 0);
            }
            if (!__all_sync(kFullMask, mbar_wait(m_ready, (uint32_t)(k & 1), cap))) {
                mok = false;
                break;
            }
            if (lane == 0) {                          // Yx = M x, over the chunk's tokens only
                tc::fence_after();
                const uint32_t id = idesc_tf32(kTcQ, P);
                const uint64_t dm = smem_desc(smem_u32(BMt), L.lc, 128);
                const uint64_t dx = smem_desc(smem_u32(XTt), L.lx, 128);
                const int ks = (c.len + 7) >> 3;
                for (int kk = 0; kk < ks; ++kk)
                    tc::mma(tm_yx, dm + (uint64_t)(kk * (2 * L.lc >> 4)), dx + (uint64_t)(kk * (2 * L.lx >> 4)), id,
                            kk > 0);
                tc::commit(bar_mma);                  // Yi and Yx of head k
            }
            __syncwarp();
            if (k + 1 < nh)
                decay_tables(k + 1);                  // the tables are free: M of head k is formed
        }
        if (lane == 0) {                              // every product issued so far done before TMEM is freed
            tc::commit(drain);
            mbar_wait(drain, 0);
        }
        __syncwarp();
        mma_compute_sync();
        return;
    }

    // ---- compute warps ----
    const int quad = warp & 3, half = warp >> 2;
    const int t = 32 * quad + lane;                   // chunk row (TMEM lane) of this thread
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;

    // C into TMEM: this thread's row t, its half of the (padded) columns (at
    // most 64: d_state <= 128).  Every load is issued before the first TMEM
    // store, so the setup waits on one memory latency, not one per 16 columns.
    {
        const bool row_ok = t < c.len;
        const float *crow = a.C + bc_off + (size_t)(row_ok ? t : 0) * a.G * N;
        const int cw = ccols >> 1, cbase = half * cw;
        float4 cv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            cv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (4 * i < cw && row_ok && cbase + 4 * i < N)
                cv[i] = __ldg(reinterpret_cast<const float4 *>(crow + cbase + 4 * i));
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            if (16 * cc < cw) {
                float v[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 w = cv[4 * cc + q];
                    v[4 * q] = tf32_round(w.x);
                    v[4 * q + 1] = tf32_round(w.y);
                    v[4 * q + 2] = tf32_round(w.z);
                    v[4 * q + 3] = tf32_round(w.w);
                }
                tmem_st16(tm_c + lane_off + cbase + 16 * cc, v);
            }
        }
        tmem_wait_st();
    }
    // every wait's outcome is taken per warp (__all_sync), so the warp-wide
    // tcgen05 loads and stores always run in whole warps
    bool ok = __all_sync(kFullMask, mbar_wait(bar_b, 0, cap));   // B landed
    if (ok) {
        kmajor_round(BMt, L.lc, kTcQ, Np4, warp, lane);
        fence_async_smem();
        tc::fence_before();
        mbar_arrive(c_ready);
    }

    for (int k = 0; k < nh && ok; ++k) {
        const int h = g * hpg + hl0 + k;
        const int b = nbuf == 2 ? (k & 1) : 0;
        const char *XRt = sm + (b ? L.XR[1] : L.XR[0]);
        if (!__all_sync(kFullMask, mbar_wait(full + b, (uint32_t)((k / nbuf) & 1), cap))) {
            ok = false;                               // S_in and x of head k never landed
            break;
        }
        // x^T of the previous head is no longer read: its products are done
        xraw_transpose(XTt, L.lx, XRt, P, tid);      // rounded to TF32 as it is transposed
        bool got = mbar_wait(dec_full, (uint32_t)(k & 1), cap);
        if (k == 0)
            got = mbar_wait(bar_g, 0, cap) && got;    // G formed; B's space is free for M
        if (!__all_sync(kFullMask, got)) {
            ok = false;
            break;
        }
        tc::fence_after();

        // M = G dt_s exp(a_t - a_s) for s <= t, into the A tile (reusing B's
        // space), in pieces of 16 columns.  A piece wholly left of the warp's
        // rows uses exp(a_t - a_s) = e_t f_s with the piece's last column r:
        // f_s = dt_s exp(a_r - a_s) (table `fcol`, built per head) and
        // e_t = exp(a_t - a_r), both <= 1 under decay; pieces that meet the
        // warp's diagonal take exp(a_t - a_s) per element and mask s > t.
        const float at = al[t];
        const int tmin_w = 32 * quad, tmax_w = 32 * quad + 31;
        for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 16) {
            float4 *mrow = reinterpret_cast<float4 *>(BMt + (c0 >> 2) * L.lc + t * 16);
            if (c0 > tmax_w) {                        // the whole piece is above the diagonal
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    mrow[q * (L.lc / 16)] = make_float4(0.f, 0.f, 0.f, 0.f);
                continue;
            }
            float gv[16];
            tmem_ld16(gv, tm_g + lane_off + c0);
            if (c0 + 15 < tmin_w) {                   // wholly below the diagonal
                const float et = ex2(at - al[c0 + 15]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 f = *reinterpret_cast<const float4 *>(fcol + c0 + 4 * q);
                    mrow[q * (L.lc / 16)] = make_float4(tf32_round(gv[4 * q] * (f.x * et)),
                                                        tf32_round(gv[4 * q + 1] * (f.y * et)),
                                                        tf32_round(gv[4 * q + 2] * (f.z * et)),
                                                        tf32_round(gv[4 * q + 3] * (f.w * et)));
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 as = *reinterpret_cast<const float4 *>(al + c0 + 4 * q);
                    const float4 ds = *reinterpret_cast<const float4 *>(dts + c0 + 4 * q);
                    const int s = c0 + 4 * q;
                    float4 m;
                    m.x = s <= t ? tf32_round(gv[4 * q] * ds.x * ex2(at - as.x)) : 0.f;
                    m.y = s + 1 <= t ? tf32_round(gv[4 * q + 1] * ds.y * ex2(at - as.y)) : 0.f;
                    m.z = s + 2 <= t ? tf32_round(gv[4 * q + 2] * ds.z * ex2(at - as.z)) : 0.f;
                    m.w = s + 3 <= t ? tf32_round(gv[4 * q + 3] * ds.w * ex2(at - as.w)) : 0.f;
                    mrow[q * (L.lc / 16)] = m;
                }
            }
        }
        tc::fence_before();
        fence_async_smem();
        mbar_arrive(m_ready);                         // M and x^T of head k written; the tables read

        if (!__all_sync(kFullMask, mbar_wait(bar_mma, (uint32_t)(k & 1), cap))) {
            ok = false;
            break;
        }
        tc::fence_after();

        // y = exp(a_t) Yi + Yx + D x for this thread's row and column half (every
        // lane takes part in the TMEM loads; rows past the chunk store nothing);
        // x comes from the staged (unrounded) tile
        {
            const float et = ex2(at), Dh = a.D[h];
            const bool row_ok = t < c.len;
            const size_t ro = ((size_t)(c.t0 + (row_ok ? t : 0)) * a.H + h) * P;
            const int cw = P >> 1;
            for (int c0 = half * cw; c0 < half * cw + cw; c0 += 16) {
                float yi[16], yx[16];
                tmem_ld16(yi, tm_yi + lane_off + c0);
                tmem_ld16(yx, tm_yx + lane_off + c0);
                if (row_ok) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = (c0 >> 2) + q;
                        const float4 xv = *reinterpret_cast<const float4 *>(XRt + t * P * 4 + ((j ^ (t & 7)) << 4));
                        float4 yv;
                        yv.x = fmaf(et, yi[4 * q], yx[4 * q]) + Dh * xv.x;
                        yv.y = fmaf(et, yi[4 * q + 1], yx[4 * q + 1]) + Dh * xv.y;
                        yv.z = fmaf(et, yi[4 * q + 2], yx[4 * q + 2]) + Dh * xv.z;
                        yv.w = fmaf(et, yi[4 * q + 3], yx[4 * q + 3]) + Dh * xv.w;
                        __stcs(reinterpret_cast<float4 *>(a.y + ro + c0 + 4 * q), yv);
                    }
                }
            }
        }
        tc::fence_before();
        mbar_arrive(epi_done);                        // Yi and Yx may be overwritten
        mbar_arrive(empty + b);                       // buffer b may be refilled
    }
    if (compute_sync_or(!ok)) {                       // a copy or product never completed
        if (tid == 0)
            atomicExch(p.status, 1);
        // this block's y is incomplete: NaN over its whole tile
        poison_y(a.y, (long long)a.H * P, c.t0, c.len, (g * hpg + hl0) * P, nh * P, tid, kTcThreads);
    }
    mma_compute_sync();                               // the MMA warp has drained its products
    if (warp == 0)
        tmem_dealloc(tmem, sg.tmem_cols);
}

}  // namespace

size_t ssd_tc_smem_bytes(int n_pad, int P, int nbuf) { return tc_layout(n_pad, P, nbuf).total; }

int ssd_tc_buffers(int chunk, int n_pad, int P, size_t smem_optin)
{
    if (chunk != kTcQ || n_pad > kTcQ || P % 32 != 0 || tc_tmem_need(n_pad, P) > 512)
        return 0;
    for (int nb = 2; nb >= 1; --nb)
        if (ssd_tc_smem_bytes(n_pad, P, nb) <= smem_optin)
            return nb;
    return 0;
}

int ssd_tc_tmem_cols(int n_pad, int P)
{
    int cols = 32;
    while (cols < tc_tmem_need(n_pad, P))
        cols <<= 1;
    return cols;
}

cudaError_t launch_ssd_output_tc(const ScanArgs &a, const SsdPlan &plan, const SsdGeom &g, int max_units,
                                 cudaStream_t stream)
{
    const int hpg = a.H / a.G;
    const dim3 grid((unsigned)max_units, (unsigned)a.G, (unsigned)((hpg + g.heads_per_cta - 1) / g.heads_per_cta));
    const size_t smem = ssd_tc_smem_bytes(g.n_pad, a.P, g.out_buffers);
    cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(ssd_output_tc_kernel), smem);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(ssd_output_tc_kernel, grid, dim3(kTcBlock), smem, stream, a, plan, g);
}

}  // namespace ssm
