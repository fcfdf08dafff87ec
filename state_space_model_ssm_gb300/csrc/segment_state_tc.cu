// State pass of the time segments on the 5th-generation tensor cores (sm_103a).
//
// The time segments of segments.cu need, for every segment k of a sequence but
// its last and every head h, the state the segment's tokens leave when the
// segment starts from zero, and the segment's decay.  Unrolling the recurrence
// ("The llama journey", Day 14: decay exp(dt A), input dt x B) over the
// segment's tokens s gives
//
//   L[p][n] = sum_s w_s x_s[p] B_s[n],   w_s = dt_s exp(A sum_{r > s} dt_r),
//   d       = exp(A sum_s dt_s),
//
// plus d S_slot[p][n] for the first segment of a resuming sequence.  L^T =
// B^T X_w is a matrix product over the segment's tokens: M = 128 state rows n
// (d_state padded with zero rows), N = the head dims of HB heads of one group
// side by side (head_dim padded to a multiple of 32), K = tokens.  B is the
// group's, so the heads of a block share its operand tile.  The sequential
// kernel's state-only mode computes the same values with one multiply-add
// chain per state element.
//
// fp32 accuracy from TF32 operands: each operand value v is split into hi =
// tf32(v) (nearest) and lo = v - hi (exact in fp32), and the products are
// accumulated as lo_a hi_b + hi_a lo_b + hi_a hi_b in fp32 (TMEM).  The
// dropped lo_a lo_b and the TF32 rounding of lo are each below 2^-21 of the
// product.
//
// A block owns one (segment, HB heads) and walks the segment's 16-token chunks
// from the last to the first, so that a token's decay exponent, the sum of
// dt A over the tokens after it, is a running suffix sum.  Three roles hand
// chunks to each other through mbarriers, so each runs ahead as far as its
// ring allows.  A loader warp brings the raw rows of B ([16][128] floats,
// d_state padded by the TMA's zero fill) and x ([16][HB][head_dim padded])
// into a ring of three stages with TMA, each chunk's load started as soon as
// the staging threads have read the chunk its stage held, and writes the
// chunk's token weights (lane = head * 16 + token, carrying each head's total;
// dt fetched with cp.async eight chunks ahead) beside it.  The 8 staging warps
// turn a staged chunk into operands.  B^T goes to TMEM, where the MMA takes its
// A operand from (row n in lane n, one token per column): each thread splits
// half of one row (8 tokens, conflict-free 4-byte reads) and writes its hi and
// lo parts with tcgen05.st, so the tensor core reads only X from shared
// memory.  X_w is a K-major shared-memory tile: the values of 4 consecutive
// tokens of one row form a 16-byte cell, written whole (consecutive rows
// across a warp).  Two operand buffers alternate.  Once a buffer is written the
// MMA warp issues the chunk's 6 MMAs (K = 8 each) and commits them to the
// buffer's mbarrier, which the staging warps wait on before they write that
// buffer again.  The epilogue reads the
// accumulator (warp w: state rows 32 (w % 4) .. +31, column half w / 4) and
// stores L with the state-slot layout, coalesced over n.
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "ssd_common.cuh"
#include "tc_common.cuh"

namespace ssm {

namespace {

using namespace tc;

constexpr int kSsQ = 16;                   // tokens per chunk (K of a chunk's products)
constexpr int kSsRows = 128;               // M: state rows n (d_state padded)
constexpr int kSsThreads = 256;           // warps 0-7 stage the operands
constexpr int kSsBlock = kSsThreads + 64;  // warp 8 issues the MMAs; warp 9 the TMA loads and the token weights
constexpr int kSsQuads = kSsQ / 4;         // 16-byte K cells per row and chunk
constexpr int kSsStages = 3;               // staged raw chunks
constexpr int kSsLead = kSsStages;         // chunks whose TMA is started before the one being staged
constexpr int kSsDtRing = 8;               // chunks of dt in flight or waiting in shared memory
constexpr int kSsBufs = 2;                 // operand buffers: staging of chunk j waits for chunk j - kSsBufs's products

// Shared memory (bytes), all offsets multiples of 1024: kSsBufs buffers of the
// X operand tiles (buffer b at b * buf; hi at 0, lo at x_lo), the staged raw
// chunks (stage s at raw + s * stage; B rows at 0, x rows at rx), mbarriers
// (full[] and empty[] per stage, written[] and mma[] per buffer, drain), the
// TMEM address, the token weights of each stage's chunk, the heads' decays and
// the dt ring.
struct SsLayout {
    uint32_t x_lo, buf;
    uint32_t raw, rx, stage;
    uint32_t bar, tslot, total;
    uint32_t wts, dec;        // weights of each stage's chunk [kSsStages][32] (lane = head * 16 + token);
                              // decays [HB], then their logs [HB] at dec + 16
    uint32_t dtr;             // dt of kSsDtRing chunks [kSsDtRing][32] (chunk j in row j % kSsDtRing)
    uint32_t lx;              // K-cell stride of the X tiles (nx rows)
};

__host__ __device__ constexpr SsLayout ss_layout(int nx)
{
    SsLayout L{};
    L.lx = (uint32_t)nx * 16;
    const uint32_t tx = L.lx * kSsQuads;
    L.x_lo = tx;
    L.buf = 2 * tx;
    L.raw = kSsBufs * L.buf;
    L.rx = kSsQ * kSsRows * 4;
    L.stage = L.rx + (uint32_t)(kSsQ * nx * 4);
    L.bar = L.raw + kSsStages * L.stage;
    L.tslot = L.bar + (uint32_t)((2 * kSsStages + 2 * kSsBufs + 2) / 2 * 2 * sizeof(uint64_t));
    L.wts = L.tslot + 16;
    L.dec = L.wts + kSsStages * 32 * 4;
    L.dtr = L.dec + 32;
    L.total = L.dtr + kSsDtRing * 32 * 4;
    return L;
}

// TMEM: the accumulator in columns [0, nx), then kSsBufs buffers of the B^T
// operand (buffer b at nx + 32 b: 16 hi columns, then 16 lo), one token per
// column, state row n in lane n.
__host__ __device__ constexpr uint32_t ss_tmem_cols(int nx)
{
    return nx + 32 * kSsBufs <= 128 ? 128u : nx + 32 * kSsBufs <= 256 ? 256u : 512u;
}

__device__ __forceinline__ float4 split_hi(float4 v, float4 &lo)
{
    const float4 hi = ssd::tf32_round4(v);
    lo = make_float4(v.x - hi.x, v.y - hi.y, v.z - hi.z, v.w - hi.w);
    return hi;
}

}  // namespace

namespace {

// X operand cells per staging thread, and whether the last round of them is partial.
template <int NX>
struct XCells {
    static constexpr int count = (NX * kSsQuads + kSsThreads - 1) / kSsThreads;
    static constexpr bool guard = (NX * kSsQuads) % kSsThreads != 0;
};

// One staged chunk (stage `raw`) into the operand buffers: this thread's half
// of B^T row `row` (tokens 8 half .. +7) into TMEM at `ta` (the buffer's hi
// columns of the warp's lanes) and its X cells (row xr[i] = head * p_pad + p,
// token quad xq[i]; xq < 0: none) into shared memory `buf`, X scaled by the
// chunk's weights `w` ([head * 16 + token]).  PARTIAL: tokens >= cnt read as
// zero (only the last chunk of a segment can be short).  No branch inside, so
// the loads, splits and stores of all cells interleave.
template <int XI, int HB, bool PARTIAL>
__device__ __forceinline__ void stage_chunk(const char *raw, char *buf, const float *w, uint32_t ta, int row,
                                            int half, const int (&xr)[XCells<32 * XI * HB>::count],
                                            const int (&xq)[XCells<32 * XI * HB>::count], int cnt)
{
    constexpr int p_pad = 32 * XI, nx = HB * p_pad;
    constexpr SsLayout L = ss_layout(nx);
    auto mask = [cnt](float4 v, int q) {
        if (PARTIAL) {
            v.x = 4 * q < cnt ? v.x : 0.f;
            v.y = 4 * q + 1 < cnt ? v.y : 0.f;
            v.z = 4 * q + 2 < cnt ? v.z : 0.f;
            v.w = 4 * q + 3 < cnt ? v.w : 0.f;
        }
        return v;
    };
    {
        const float *rb = reinterpret_cast<const float *>(raw) + row + 8 * half * kSsRows;
        float hi[8], lo[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float v = rb[k * kSsRows];
            if (PARTIAL)
                v = 8 * half + k < cnt ? v : 0.f;
            hi[k] = ssd::tf32_round(v);
            lo[k] = v - hi[k];
        }
        tmem_st8(ta + 8 * half, hi);
        tmem_st8(ta + 16 + 8 * half, lo);
    }
#pragma unroll
    for (int i = 0; i < XCells<nx>::count; ++i) {
        const int q = xq[i], r = xr[i];
        if (!XCells<nx>::guard || q >= 0) {
            const float4 w4 = *reinterpret_cast<const float4 *>(w + (r / p_pad) * 16 + 4 * q);
            const float *rx = reinterpret_cast<const float *>(raw + L.rx) + r;
            const float4 v = mask(make_float4(rx[(4 * q) * nx] * w4.x, rx[(4 * q + 1) * nx] * w4.y,
                                              rx[(4 * q + 2) * nx] * w4.z, rx[(4 * q + 3) * nx] * w4.w), q);
            float4 lo;
            const float4 hi = split_hi(v, lo);
            const uint32_t off = q * L.lx + r * 16;
            *reinterpret_cast<float4 *>(buf + off) = hi;
            *reinterpret_cast<float4 *>(buf + L.x_lo + off) = lo;
        }
    }
}

// XI: head_dim padded to 32 XI; HB: heads per block (1 or 2).
template <int XI, int HB>
__global__ void __launch_bounds__(kSsBlock, HB * XI <= 4 ? 2 : 1)
segment_state_tc_kernel(const ScanArgs a, const SegmentPlan plan, const __grid_constant__ CUtensorMap tm_b,
                        const __grid_constant__ CUtensorMap tm_x)
{
    griddep_entry();
    constexpr int p_pad = 32 * XI, nx = HB * p_pad;
    constexpr SsLayout L = ss_layout(nx);
    constexpr uint32_t kBoxBytes = (uint32_t)(kSsQ * (kSsRows + nx) * 4);   // both TMA boxes of a chunk
    extern __shared__ __align__(1024) unsigned char ss_smem[];
    const int unit = blockIdx.x, h0 = blockIdx.y * HB;
    if (unit >= *plan.n_units)
        return;
    const int2 us = plan.units[unit];
    const int seq = us.x, seg = us.y;
    const int seq_len = a.seq_lens[seq];
    const int nseg = max(1, (seq_len + plan.seg_len - 1) / plan.seg_len);
    if (seg >= nseg - 1 && !plan.chunk_states)
        return;                                       // the last segment needs no state pass
    const int len = min(plan.seg_len, seq_len - seg * plan.seg_len);
    const int nc = (len + kSsQ - 1) / kSsQ;
    const int tok0 = a.seq_starts[seq] + seg * plan.seg_len;
    const int P = a.P, N = a.N, H = a.H;
    if (nc <= 0) {                                    // an empty sequence (chunk states): state 0, sum 0
        for (int hb = 0; hb < HB; ++hb) {
            float *dst = plan.seg_state + ((size_t)unit * H + h0 + hb) * P * N;
            for (int i = threadIdx.x; i < P * N; i += kSsBlock)
                dst[i] = 0.f;
        }
        if (threadIdx.x < HB)
            plan.seg_decay[(size_t)unit * H + h0 + threadIdx.x] = plan.chunk_states ? 0.f : 1.f;
        return;
    }
    const int grp = h0 / (H / a.G);
    char *sm = reinterpret_cast<char *>(ss_smem);
    const uint32_t sbase = smem_u32(sm);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L.bar);     // per stage: TMA boxes landed, weights formed
    uint64_t *empty = full + kSsStages;                            // per stage: every staging thread read it
    uint64_t *written = empty + kSsStages;                         // per buffer: operands written
    uint64_t *mmab = written + kSsBufs;                            // per buffer: products done
    uint64_t *drain = mmab + kSsBufs;                              // after a failed wait: all products done
    const long cap = plan.fail_waits ? 0 : kSpinLimit;             // polls of a pipeline wait
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L.tslot);
    float *wts = reinterpret_cast<float *>(sm + L.wts);
    float *decs = reinterpret_cast<float *>(sm + L.dec);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr uint32_t cols = ss_tmem_cols(nx);

    if (warp == 0)
        tmem_alloc(tslot, cols);
    if (tid == 0) {
        for (int i = 0; i < kSsStages; ++i) {
            mbar_init(full + i, 1 + 32);              // the TMA's expect_tx, then the 32 weights lanes
            mbar_init(empty + i, kSsThreads);
        }
        for (int i = 0; i < kSsBufs; ++i) {
            mbar_init(written + i, kSsThreads);
            mbar_init(mmab + i, 1);
        }
        mbar_init(drain, 1);
        mbar_init_fence();
    }
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kSsThreads / 32) {
        // ---- MMA warp: a chunk's products once its operand buffer is written ----
        bool mok = true;
        if (lane == 0) {
            int b = 0;                                // operand buffer of chunk j
            for (int j = 0; j < nc; ++j) {
                if (!mbar_wait(written + b, (uint32_t)((j / kSsBufs) & 1), cap)) {
                    mok = false;                      // the staging warps gave up
                    break;
                }
                fence_after();
                constexpr uint32_t id = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(nx >> 3) << 17) |
                                        ((uint32_t)(kSsRows >> 4) << 24);        // idesc_tf32(128, nx)
                const uint32_t bx = sbase + b * L.buf;
                const uint32_t tah = tmem + nx + 32 * b, tal = tah + 16;         // B^T hi, lo in TMEM
#pragma unroll
                for (int kk = 0; kk < kSsQ / 8; ++kk) {
                    const uint64_t dxh = smem_desc(bx + 2 * kk * L.lx, L.lx, 128);
                    const uint64_t dxl = smem_desc(bx + L.x_lo + 2 * kk * L.lx, L.lx, 128);
                    mma_ts(tmem, tal + 8 * kk, dxh, id, (j > 0 || kk > 0) ? 1u : 0u);
                    mma_ts(tmem, tah + 8 * kk, dxl, id, 1u);
                    mma_ts(tmem, tah + 8 * kk, dxh, id, 1u);
                }
                commit(mmab + b);
                b = b == kSsBufs - 1 ? 0 : b + 1;
            }
        }
        __syncwarp();
        if (__syncthreads_or(!mok) && lane == 0) {   // a wait gave up: drain before TMEM is freed
            commit(drain);                            // arrives once every product issued so far is done
            mbar_wait(drain, 0);
        }
        __syncthreads();
        return;
    }
    if (warp == kSsThreads / 32 + 1) {
        // ---- loader warp: chunk j's TMA into stage j % kSsStages once the
        // staging threads have read the chunk that stage held, then its token
        // weights; at the end the heads' decays ----
        // chunk j of the walk (tokens [c * 16, c * 16 + 16) of the segment, c = nc - 1 - j)
        auto issue = [&](int j, int st) {
            const int t = tok0 + (nc - 1 - j) * kSsQ;
            char *raw = sm + L.raw + st * L.stage;
            mbar_expect_tx(full + st, kBoxBytes);
            tma_load_3d(raw, &tm_b, 0, grp, t, full + st);
            tma_load_3d(raw + L.rx, &tm_x, 0, h0, t, full + st);
        };
        constexpr float kLog2e = 1.4426950408889634f;
        const int wh = lane >> 4, ws = lane & 15;
        const float A2 = wh < HB ? a.A[h0 + wh] * kLog2e : 0.f;
        // dt of chunk j into ring row j % kSsDtRing, one cp.async group per chunk
        // (zeros past the segment)
        float *dtr = reinterpret_cast<float *>(sm + L.dtr);
        auto fetch_dt = [&](int j) {
            const int s = (nc - 1 - j) * kSsQ + ws;
            const bool in = j < nc && wh < HB && s < len;
            ssd::cp_async4_zfill(dtr + (j % kSsDtRing) * 32 + lane,
                                 in ? a.dt + (size_t)(tok0 + s) * H + h0 + wh : a.dt, in ? 4 : 0);
            cp_async_commit();
        };
        float carry = 0.f;                            // this lane's head: sum of dt A log2(e) walked so far
        // w_s = dt_s 2^(A2 * sum of dt over the tokens after s) of chunk j into the weights of stage st
        auto weights = [&](int j, int st) {
            const float dts = dtr[(j % kSsDtRing) * 32 + lane];
            float suf = dts * A2;                     // inclusive suffix sum within the 16 lanes
#pragma unroll
            for (int o = 1; o < kSsQ; o <<= 1) {
                const float t = __shfl_down_sync(kFullMask, suf, o);
                if (ws + o < kSsQ)
                    suf += t;
            }
            float after = __shfl_down_sync(kFullMask, suf, 1);
            if (ws == kSsQ - 1)
                after = 0.f;
            wts[st * 32 + lane] = dts * ssd::ex2(carry + after);
            carry += __shfl_sync(kFullMask, suf, lane & 16);
        };
        // dt (scattered 4-byte reads) is fetched kSsDtRing chunks ahead, so a
        // cold read's latency stays off the chunk chain; group g carries chunk g
#pragma unroll
        for (int j = 0; j < kSsDtRing; ++j)
            fetch_dt(j);
        bool lok = true;
        int issued = 0;                               // chunks whose TMA was started
        int st = 0;                                   // stage of chunk j
        for (int j = 0; j < nc; ++j) {
            if (j >= kSsStages &&                     // one decision for the warp (its shuffles need every lane)
                !__all_sync(kFullMask, mbar_wait(empty + st, (uint32_t)((j / kSsStages - 1) & 1), cap))) {
                lok = false;                          // the staging warps gave up
                break;
            }
            if (lane == 0)
                issue(j, st);
            issued = j + 1;
            cp_async_wait<kSsDtRing - 1>();           // group j (kSsDtRing + j committed)
            weights(j, st);
            mbar_arrive(full + st);                   // every lane: its weight is written
            fetch_dt(j + kSsDtRing);                  // into the row just read; a group every iteration
            st = st == kSsStages - 1 ? 0 : st + 1;
        }
        cp_async_wait<0>();
        const float cl = __shfl_sync(kFullMask, carry, 16 * (lane & 1));   // lane hb: head hb's log2 decay
        if (lane < HB) {
            decs[lane] = ssd::ex2(cl);
            decs[4 + lane] = cl * 0.6931471805599453f;   // the natural log: sum of dt A
        }
        if (__syncthreads_or(!lok) && lane == 0) {   // a wait gave up: each stage's last TMA lands
            for (int c = max(0, issued - kSsStages); c < issued; ++c)   // before the block exits
                mbar_wait(full + c % kSsStages, (uint32_t)((c / kSsStages) & 1));
        }
        __syncthreads();
        return;
    }

    // ---- staging warps ----
    const int quad = warp & 3, half = warp >> 2;
    const int row = 32 * quad + lane;                 // B^T row (TMEM lane) of this thread; tokens 8 half ..
    const uint32_t tlane = tmem + ((uint32_t)(32 * quad) << 16);
    int xr[XCells<nx>::count], xq[XCells<nx>::count];
#pragma unroll
    for (int i = 0; i < XCells<nx>::count; ++i) {
        const int it = tid + kSsThreads * i;
        xq[i] = it < nx * kSsQuads ? it / nx : -1;    // uniform across a warp (nx % 32 == 0)
        xr[i] = it - (it / nx) * nx;
    }

    bool ok = true;
    int last = -1;                                    // last chunk whose operands were written
    int st = 0;                                       // stage of chunk j
    int b = 0;                                        // operand buffer of chunk j
    for (int j = 0; j < nc; ++j) {
        const int cnt = min(kSsQ, len - (nc - 1 - j) * kSsQ);   // tokens of the chunk (16 but the first)
        ok = mbar_wait(full + st, (uint32_t)((j / kSsStages) & 1), cap);
        if (ok && j >= kSsBufs) {                     // buffer b: products of chunk j - kSsBufs done
            ok = mbar_wait(mmab + b, (uint32_t)((j / kSsBufs - 1) & 1), cap);
            fence_after();
        }
        if (!__all_sync(kFullMask, ok)) {            // one decision for the warp (tcgen05.st is warp-wide)
            ok = false;
            break;                                    // a wait gave up: write nothing more
        }
        const char *raw = sm + L.raw + st * L.stage;
        char *buf = sm + b * L.buf;
        const float *w = wts + st * 32;
        const uint32_t ta = tlane + nx + 32 * b;
        if (cnt < kSsQ)
            stage_chunk<XI, HB, true>(raw, buf, w, ta, row, half, xr, xq, cnt);
        else
            stage_chunk<XI, HB, false>(raw, buf, w, ta, row, half, xr, xq, cnt);
        mbar_arrive(empty + st);                      // this thread's reads of the stage are done
        tmem_wait_st();
        fence_before();
        fence_async_smem();
        mbar_arrive(written + b);
        last = j;
        st = st == kSsStages - 1 ? 0 : st + 1;
        b = b == kSsBufs - 1 ? 0 : b + 1;
    }

    if (ok && last == nc - 1)                         // every chunk's operands written: its products done
        ok = mbar_wait(mmab + last % kSsBufs, (uint32_t)((last / kSsBufs) & 1), cap);
    if (__syncthreads_or(!ok)) {                      // the MMA and loader warps drain the products and copies
        if (tid == 0 && plan.status)
            atomicExch(plan.status, 1);
    } else {
        fence_after();
        const uint32_t taddr = tlane;                 // state rows 32 quad .. +31 (row: this thread's)
        const bool from_slot = !plan.chunk_states && seg == 0 && a.resume[seq] != 0;
        constexpr int cw = nx / 2;
#pragma unroll
        for (int c0 = 0; c0 < cw; c0 += 16) {
            const int col = half * cw + c0;           // 16 columns of one head (16 | p_pad)
            const int hb = col / p_pad, p0 = col - hb * p_pad;
            const float d = decs[hb];
            float v[16];
            tmem_ld16(v, taddr + col);
            if (row < N && p0 < P) {
                const size_t hoff = ((size_t)h0 + hb) * P * N;
                float *dst = plan.seg_state + (size_t)unit * H * P * N + hoff;
                const float *src = from_slot ? a.state + (size_t)seq * H * P * N + hoff : nullptr;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int p = p0 + k;
                    if (p < P) {
                        float o = v[k];
                        if (src)
                            o = fmaf(d, src[(size_t)p * N + row], o);
                        dst[(size_t)p * N + row] = o;
                    }
                }
            }
        }
        if (tid < HB)
            plan.seg_decay[(size_t)unit * H + h0 + tid] = plan.chunk_states ? decs[4 + tid] : decs[tid];
    }
    fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tmem, cols);
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// fp32 [d2][d1][d0] tensor (d0 contiguous) read in boxes of b0 x b1 x b2.
bool encode_3d(CUtensorMap *tm, const float *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1,
               uint32_t b2)
{
    const auto fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * 4, d0 * d1 * 4};      // bytes, dims 1 and 2
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int XI, int HB>
cudaError_t launch_shape(const ScanArgs &a, const SegmentPlan &plan, const SegStateMaps &maps, int max_units,
                         cudaStream_t stream)
{
    constexpr size_t smem = ss_layout(HB * 32 * XI).total;
    CUtensorMap tm_b, tm_x;
    static_assert(sizeof(CUtensorMap) == sizeof(maps.b), "tensor map size");
    std::memcpy(&tm_b, maps.b, sizeof tm_b);
    std::memcpy(&tm_x, maps.x, sizeof tm_x);
    cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(segment_state_tc_kernel<XI, HB>), smem);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(segment_state_tc_kernel<XI, HB>, dim3((unsigned)max_units, (unsigned)(a.H / HB)),
                      dim3(kSsBlock), smem, stream, a, plan, tm_b, tm_x);
}

// Two heads per block where they share a group and their N (2 x head_dim
// padded) fits one product.
int heads_per_block(int H, int G, int P) { return ((H / G) % 2 == 0 && (P + 31) / 32 <= 4) ? 2 : 1; }

}  // namespace

bool segment_state_tc_supported(int N, int P, size_t smem_optin)
{
    if (N < 4 || N > kSsRows || N % 4 != 0 || P < 4 || P > 256 || P % 4 != 0 || !encode_fn())
        return false;
    return ss_layout(32 * ((P + 31) / 32)).total <= smem_optin;     // one head per block at most needs this
}

bool segment_state_tc_maps(const ScanArgs &a, SegStateMaps *maps)
{
    const int p_pad = 32 * ((a.P + 31) / 32), hb = heads_per_block(a.H, a.G, a.P);
    CUtensorMap tm_b, tm_x;
    if (a.n_tokens <= 0 ||
        !encode_3d(&tm_b, a.B, (uint64_t)a.N, (uint64_t)a.G, (uint64_t)a.n_tokens, kSsRows, 1, kSsQ) ||
        !encode_3d(&tm_x, a.x, (uint64_t)a.P, (uint64_t)a.H, (uint64_t)a.n_tokens, (uint32_t)p_pad, (uint32_t)hb,
                   kSsQ))
        return false;
    std::memcpy(maps->b, &tm_b, sizeof tm_b);
    std::memcpy(maps->x, &tm_x, sizeof tm_x);
    return true;
}

cudaError_t launch_segment_state_tc(const ScanArgs &a, const SegmentPlan &plan, const SegStateMaps &maps,
                                    int max_units, cudaStream_t stream)
{
    if (max_units <= 0 || a.n_tokens <= 0)
        return cudaSuccess;
    const int xi = (a.P + 31) / 32;
    if (heads_per_block(a.H, a.G, a.P) == 2) {
        switch (xi) {
        case 1: return launch_shape<1, 2>(a, plan, maps, max_units, stream);
        case 2: return launch_shape<2, 2>(a, plan, maps, max_units, stream);
        case 3: return launch_shape<3, 2>(a, plan, maps, max_units, stream);
        case 4: return launch_shape<4, 2>(a, plan, maps, max_units, stream);
        default: break;
        }
    }
    switch (xi) {
    case 1: return launch_shape<1, 1>(a, plan, maps, max_units, stream);
    case 2: return launch_shape<2, 1>(a, plan, maps, max_units, stream);
    case 3: return launch_shape<3, 1>(a, plan, maps, max_units, stream);
    case 4: return launch_shape<4, 1>(a, plan, maps, max_units, stream);
    case 5: return launch_shape<5, 1>(a, plan, maps, max_units, stream);
    case 6: return launch_shape<6, 1>(a, plan, maps, max_units, stream);
    case 7: return launch_shape<7, 1>(a, plan, maps, max_units, stream);
    case 8: return launch_shape<8, 1>(a, plan, maps, max_units, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
