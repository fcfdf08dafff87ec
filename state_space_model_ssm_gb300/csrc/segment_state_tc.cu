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
// B^T X_w is a matrix product over the segment's tokens (M = 128 state rows n,
// d_state padded with zero rows; N = head_dim padded to a multiple of 32;
// K = tokens), here on tcgen05.mma.  The sequential kernel's state-only mode
// computes the same values with one multiply-add chain per state element.
//
// fp32 accuracy from TF32 operands: each operand value v is split into hi =
// tf32(v) (nearest) and lo = v - hi (exact in fp32), and the products are
// accumulated as lo_a hi_b + hi_a lo_b + hi_a hi_b in fp32 (TMEM).  The
// dropped lo_a lo_b and the TF32 rounding of lo are each below 2^-21 of the
// product.
//
// A block (8 warps) owns one (segment, head).  It walks the segment's 32-token
// chunks from the last to the first, so that a token's decay exponent, the sum
// of dt A over the tokens after it, is a running suffix sum: each warp forms a
// chunk's weights in registers (lane = token) and carries the chunk's total.
// Each thread loads its cells of the next chunk's B and x into registers while
// it writes the current chunk into one of two operand buffers.  The token index
// is K, so the values of 4 consecutive tokens of one row form a 16-byte cell of
// the K-major tile, written whole (consecutive rows across a warp: no bank
// conflicts).  Thread 0 issues the chunk's 12 MMAs (K = 8 each) and commits
// them to the buffer's mbarrier, which the writers wait on two chunks later.
// The epilogue reads the accumulator (warp w: state rows 32 (w % 4) .. +31,
// column half w / 4) and stores L with the state-slot layout, coalesced over n.
#include "ssd_common.cuh"
#include "tc_common.cuh"

namespace ssm {

namespace {

using namespace tc;

constexpr int kSsQ = 32;                   // tokens per chunk (K of a chunk's products)
constexpr int kSsRows = 128;               // M: state rows n (d_state padded)
constexpr int kSsThreads = 256;
constexpr int kSsQuads = kSsQ / 4;         // 16-byte K cells per row and chunk
constexpr int kSsBCells = kSsRows * kSsQuads / kSsThreads;   // B cells per thread: 4

// Shared memory (bytes): two buffers of the four operand tiles, two mbarriers
// and the TMEM address.
struct SsLayout {
    uint32_t a_hi[2], a_lo[2], x_hi[2], x_lo[2], bar, tslot, total;
    uint32_t la, lx;          // K-cell strides of the B^T tiles (128 rows) and x_w tiles (p_pad rows)
};

__host__ __device__ inline SsLayout ss_layout(int p_pad)
{
    SsLayout L;
    L.la = kSsRows * 16;
    L.lx = (uint32_t)p_pad * 16;
    const uint32_t ta = L.la * kSsQuads, tx = L.lx * kSsQuads;
    uint32_t off = 0;
    for (int b = 0; b < 2; ++b) {
        L.a_hi[b] = off; off += ta;
        L.a_lo[b] = off; off += ta;
        L.x_hi[b] = off; off += tx;
        L.x_lo[b] = off; off += tx;
    }
    L.bar = off;   off += 2 * sizeof(uint64_t);
    L.tslot = off; off += 16;
    L.total = off;
    return L;
}

__host__ __device__ inline uint32_t ss_tmem_cols(int p_pad)
{
    return p_pad <= 32 ? 32u : p_pad <= 64 ? 64u : p_pad <= 128 ? 128u : 256u;
}

// One chunk's operand values in registers: B cells (row n, 4 tokens) and x
// cells (row p, 4 tokens) of this thread, and dt of token `lane`.
template <int XI>
struct ChunkRegs {
    float b[kSsBCells][4];
    float x[XI][4];
    float dt;
};

__device__ __forceinline__ float4 split_hi(float4 v, float4 &lo)
{
    const float4 hi = ssd::tf32_round4(v);
    lo = make_float4(v.x - hi.x, v.y - hi.y, v.z - hi.z, v.w - hi.w);
    return hi;
}

// Two blocks per SM where their shared memory fits (head_dim up to 96).
template <int XI>
__global__ void __launch_bounds__(kSsThreads, XI <= 3 ? 2 : 1)
segment_state_tc_kernel(const ScanArgs a, const SegmentPlan plan)
{
    extern __shared__ __align__(1024) unsigned char ss_smem[];
    const int unit = blockIdx.x, h = blockIdx.y;
    if (unit >= *plan.n_units)
        return;
    const int2 us = plan.units[unit];
    const int seq = us.x, seg = us.y;
    const int seq_len = a.seq_lens[seq];
    const int nseg = max(1, (seq_len + plan.seg_len - 1) / plan.seg_len);
    if (seg >= nseg - 1)
        return;                                       // the last segment needs no state pass
    const int len = min(plan.seg_len, seq_len - seg * plan.seg_len);
    const int nc = (len + kSsQ - 1) / kSsQ;
    const long long tok0 = (long long)a.seq_starts[seq] + (long long)seg * plan.seg_len;
    const int P = a.P, N = a.N, H = a.H;
    constexpr int p_pad = 32 * XI;
    const int grp = h / (H / a.G);
    const SsLayout L = ss_layout(p_pad);
    char *sm = reinterpret_cast<char *>(ss_smem);
    const uint32_t sbase = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L.tslot);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t cols = ss_tmem_cols(p_pad);
    constexpr float kLog2e = 1.4426950408889634f;
    const float A2 = a.A[h] * kLog2e;

    if (warp == 0)
        tmem_alloc(tslot, cols);
    if (tid == 0) {
        mbar_init(bars, 1);
        mbar_init(bars + 1, 1);
        mbar_init_fence();
    }
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tslot;

    // cells of this thread: B (row n, token quad qb + 2i), x (row px[i], quad qx[i])
    const int n = tid & (kSsRows - 1), qb = tid >> 7;
    int px[XI], qx[XI];
#pragma unroll
    for (int i = 0; i < XI; ++i) {
        const int it = tid + kSsThreads * i;
        qx[i] = it / p_pad;                           // uniform across a warp (p_pad % 32 == 0)
        px[i] = it - qx[i] * p_pad;
    }
    const size_t GN = (size_t)a.G * N, HP = (size_t)H * P;
    const float *Bg = a.B + ((size_t)tok0 * a.G + grp) * N;
    const float *xg = a.x + ((size_t)tok0 * H + h) * P;
    const float *dtg = a.dt + (size_t)tok0 * H + h;

    auto load = [&](int c, ChunkRegs<XI> &r) {
        const int s0 = c * kSsQ, cnt = min(kSsQ, len - s0);
#pragma unroll
        for (int i = 0; i < kSsBCells; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int s = 4 * (qb + 2 * i) + k;
                r.b[i][k] = (n < N && s < cnt) ? __ldg(Bg + (size_t)(s0 + s) * GN + n) : 0.f;
            }
#pragma unroll
        for (int i = 0; i < XI; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int s = 4 * qx[i] + k;
                r.x[i][k] = (px[i] < P && s < cnt) ? __ldg(xg + (size_t)(s0 + s) * HP + px[i]) : 0.f;
            }
        r.dt = lane < cnt ? __ldg(dtg + (size_t)(s0 + lane) * H) : 0.f;
    };

    ChunkRegs<XI> cur, nxt;
    load(nc - 1, cur);
    float carry = 0.f;                                // sum of dt A log2(e) over the tokens already walked
    bool ok = true;
    int last = -1;                                    // last chunk whose products were issued
    for (int j = 0; j < nc; ++j) {
        const int c = nc - 1 - j, b = j & 1;
        if (c > 0)
            load(c - 1, nxt);

        // w_s = dt_s 2^(A2 * sum of dt over the tokens after s), lane = token
        const float v = cur.dt * A2;
        float suf = v;                                // inclusive suffix sum within the chunk
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_down_sync(kFullMask, suf, o);
            if (lane + o < 32)
                suf += t;
        }
        float after = __shfl_down_sync(kFullMask, suf, 1);
        if (lane == 31)
            after = 0.f;
        const float w = cur.dt * ssd::ex2(carry + after);
        carry += __shfl_sync(kFullMask, suf, 0);

        if (j >= 2)                                   // buffer b: products of chunk j - 2 done
            ok = mbar_wait(bars + b, (uint32_t)(((j >> 1) - 1) & 1)) && ok;

        char *ah = sm + L.a_hi[b], *al = sm + L.a_lo[b], *xh = sm + L.x_hi[b], *xl = sm + L.x_lo[b];
#pragma unroll
        for (int i = 0; i < kSsBCells; ++i) {
            float4 lo;
            const float4 hi = split_hi(make_float4(cur.b[i][0], cur.b[i][1], cur.b[i][2], cur.b[i][3]), lo);
            const uint32_t off = (qb + 2 * i) * L.la + n * 16;
            *reinterpret_cast<float4 *>(ah + off) = hi;
            *reinterpret_cast<float4 *>(al + off) = lo;
        }
#pragma unroll
        for (int i = 0; i < XI; ++i) {
            const int q = qx[i];
            float4 xw;
            xw.x = cur.x[i][0] * __shfl_sync(kFullMask, w, 4 * q);
            xw.y = cur.x[i][1] * __shfl_sync(kFullMask, w, 4 * q + 1);
            xw.z = cur.x[i][2] * __shfl_sync(kFullMask, w, 4 * q + 2);
            xw.w = cur.x[i][3] * __shfl_sync(kFullMask, w, 4 * q + 3);
            float4 lo;
            const float4 hi = split_hi(xw, lo);
            const uint32_t off = q * L.lx + px[i] * 16;
            *reinterpret_cast<float4 *>(xh + off) = hi;
            *reinterpret_cast<float4 *>(xl + off) = lo;
        }
        fence_async_smem();
        if (__syncthreads_or(!ok))
            break;                                    // a wait gave up: issue nothing more
        if (tid == 0) {
            fence_after();
            const uint32_t id = idesc_tf32(kSsRows, p_pad);
#pragma unroll
            for (int kk = 0; kk < kSsQ / 8; ++kk) {
                const uint64_t dah = smem_desc(sbase + L.a_hi[b] + 2 * kk * L.la, L.la, 128);
                const uint64_t dal = smem_desc(sbase + L.a_lo[b] + 2 * kk * L.la, L.la, 128);
                const uint64_t dxh = smem_desc(sbase + L.x_hi[b] + 2 * kk * L.lx, L.lx, 128);
                const uint64_t dxl = smem_desc(sbase + L.x_lo[b] + 2 * kk * L.lx, L.lx, 128);
                mma(tmem, dal, dxh, id, (j > 0 || kk > 0) ? 1u : 0u);
                mma(tmem, dah, dxl, id, 1u);
                mma(tmem, dah, dxh, id, 1u);
            }
            commit(bars + b);
        }
        last = j;
        cur = nxt;
    }

    if (ok && last == nc - 1)                         // every product of the segment issued
        ok = mbar_wait(bars + (last & 1), (uint32_t)((last >> 1) & 1));
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            if (plan.status)
                atomicExch(plan.status, 1);
            if (last >= 0)                            // one more bounded wait for the products in flight
                mbar_wait(bars + (last & 1), (uint32_t)((last >> 1) & 1));
        }
    } else {
        fence_after();
        const float d = ssd::ex2(carry);
        const int quad = warp & 3, half = warp >> 2;
        const int row = 32 * quad + lane;             // state row n of this thread (TMEM lane)
        const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16);
        float *dst = plan.seg_state + ((size_t)unit * H + h) * P * N;
        const float *src = (seg == 0 && a.resume[seq] != 0) ? a.state + ((size_t)seq * H + h) * P * N : nullptr;
        constexpr int cw = p_pad / 2;
#pragma unroll
        for (int c0 = 0; c0 < cw; c0 += 16) {
            const int col = half * cw + c0;
            float v[16];
            tmem_ld16(v, taddr + col);
            if (row < N) {
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int p = col + k;
                    if (p < P) {
                        float o = v[k];
                        if (src)
                            o = fmaf(d, src[(size_t)p * N + row], o);
                        dst[(size_t)p * N + row] = o;
                    }
                }
            }
        }
        if (tid == 0)
            plan.seg_decay[(size_t)unit * H + h] = d;
    }
    fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tmem, cols);
}

template <int XI>
cudaError_t launch_xi(const ScanArgs &a, const SegmentPlan &plan, int max_units, cudaStream_t stream)
{
    const size_t smem = ss_layout(32 * XI).total;
    cudaError_t e = cudaFuncSetAttribute(segment_state_tc_kernel<XI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    segment_state_tc_kernel<XI><<<dim3((unsigned)max_units, (unsigned)a.H), kSsThreads, smem, stream>>>(a, plan);
    return cudaGetLastError();
}

}  // namespace

bool segment_state_tc_supported(int N, int P, size_t smem_optin)
{
    if (N < 1 || N > kSsRows || P < 1 || P > 256)
        return false;
    return ss_layout(32 * ((P + 31) / 32)).total <= smem_optin;
}

cudaError_t launch_segment_state_tc(const ScanArgs &a, const SegmentPlan &plan, int max_units, cudaStream_t stream)
{
    if (max_units <= 0)
        return cudaSuccess;
    switch ((a.P + 31) / 32) {
    case 1: return launch_xi<1>(a, plan, max_units, stream);
    case 2: return launch_xi<2>(a, plan, max_units, stream);
    case 3: return launch_xi<3>(a, plan, max_units, stream);
    case 4: return launch_xi<4>(a, plan, max_units, stream);
    case 5: return launch_xi<5>(a, plan, max_units, stream);
    case 6: return launch_xi<6>(a, plan, max_units, stream);
    case 7: return launch_xi<7>(a, plan, max_units, stream);
    case 8: return launch_xi<8>(a, plan, max_units, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
