// Device helpers shared by the chunked-form ("SSD") kernels: TF32 rounding,
// asynchronous tile copies, the chunk of a work unit and its cumulative decay.
#pragma once

#include "scan_common.cuh"

namespace ssm {
namespace ssd {

// Round a finite float to TF32 (10 mantissa bits), to nearest with ties away
// from zero: add half a unit of the 11th mantissa bit to the magnitude, then
// clear the 13 bits below the TF32 mantissa.  (Infinities stay infinite.)
__device__ __forceinline__ uint32_t tf32_bits(float v)
{
    return (__float_as_uint(v) + 0x1000u) & 0xffffe000u;
}

// 2^x with the special-function unit (relative error about 2^-22; results
// below the normal range flush to zero).
__device__ __forceinline__ float ex2(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float tf32_round(float v) { return __uint_as_float(tf32_bits(v)); }

__device__ __forceinline__ float4 tf32_round4(float4 v)
{
    return make_float4(tf32_round(v.x), tf32_round(v.y), tf32_round(v.z), tf32_round(v.w));
}

__device__ __forceinline__ uint32_t fb(float v) { return __float_as_uint(v); }

// d += A * B for one m16n8k8 tile: A 16x8 row-major fragment (a0..a3),
// B 8x8 column fragment (b0, b1), fp32 accumulators d0..d3.
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte cp.async; src_bytes == 0 writes 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async16_zfill(void *smem, const void *gmem, int src_bytes)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes)
                 : "memory");
}

// 4-byte cp.async through L1; src_bytes == 0 writes a zero word and reads nothing.
__device__ __forceinline__ void cp_async4_zfill(void *smem, const void *gmem, int src_bytes)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes)
                 : "memory");
}

// Four 8x8 tiles of 32-bit words (each row 16 bytes) from shared memory; lane
// l gives the row address of tile l/8, row l%8, and receives word (l%4) of
// row (l/4) of each tile: the m16n8k8 TF32 fragment layout.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const float *p)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s)
                 : "memory");
}

// Lane layout for row tiles `w4` float4 cells wide: `lanes` (a power of two,
// at least w4 unless w4 > 32) lanes share a row, so one warp instruction
// covers 32/lanes rows and a thread keeps a fixed column; no division per cell.
struct RowMap {
    int row0;    // first row of this thread
    int col;     // first float4 column of this thread
    int lanes;   // lanes per row (column step)
    int step;    // rows per pass of the block
};

__device__ __forceinline__ RowMap row_map(int w4, int lane, int warp, int nwarps)
{
    int lg = 0;
    while ((1 << lg) < w4 && lg < 5)
        ++lg;
    RowMap m;
    m.lanes = 1 << lg;
    const int rpi = 32 >> lg;                         // rows per warp instruction
    m.row0 = warp * rpi + (lane >> lg);
    m.col = lane & (m.lanes - 1);
    m.step = nwarps * rpi;
    return m;
}

// Asynchronous copy of a rows x w4 float4 tile: global row r at g + r*gstride
// floats, shared row r at s + r*sstride.  Cells with r >= vrows or column
// >= v4 are zero-filled without a global read (vrows >= 1, so g is a valid
// address).
__device__ __forceinline__ void rows_copy(float *s, int sstride, const float *g, size_t gstride, int rows,
                                          int w4, int vrows, int v4, const RowMap &m)
{
    for (int r = m.row0; r < rows; r += m.step) {
        const float *grow = g + (size_t)r * gstride;
        float *srow = s + r * sstride;
        for (int c = m.col; c < w4; c += m.lanes) {
            const bool ok = r < vrows && c < v4;
            cp_async16_zfill(srow + 4 * c, ok ? grow + 4 * c : g, ok ? 16 : 0);
        }
    }
}

// In place TF32 rounding of the cells this thread copied with the same map.
__device__ __forceinline__ void rows_round(float *s, int sstride, int rows, int w4, const RowMap &m)
{
    for (int r = m.row0; r < rows; r += m.step) {
        float *srow = s + r * sstride;
        for (int c = m.col; c < w4; c += m.lanes) {
            float4 *q = reinterpret_cast<float4 *>(srow + 4 * c);
            *q = tf32_round4(*q);
        }
    }
}

// In place: row r scaled by w[r], then rounded to TF32.
__device__ __forceinline__ void rows_scale_round(float *s, int sstride, int rows, int w4, const RowMap &m,
                                                 const float *w)
{
    for (int r = m.row0; r < rows; r += m.step) {
        float *srow = s + r * sstride;
        const float f = w[r];
        for (int c = m.col; c < w4; c += m.lanes) {
            float4 *q = reinterpret_cast<float4 *>(srow + 4 * c);
            const float4 v = *q;
            *q = tf32_round4(make_float4(f * v.x, f * v.y, f * v.z, f * v.w));
        }
    }
}

struct ChunkRange {
    int seq, t0, len;     // packed token range [t0, t0 + len)
};

__device__ __forceinline__ bool chunk_of(const ScanArgs &a, const SsdPlan &p, int u, ChunkRange &c)
{
    if (u >= *p.n_units)
        return false;
    const int2 sk = p.units[u];
    const int L = a.seq_lens[sk.x];
    c.seq = sk.x;
    c.t0 = a.seq_starts[sk.x] + sk.y * p.chunk;
    c.len = max(0, min(p.chunk, L - sk.y * p.chunk));
    return true;
}

// One warp: the chunk-local cumulative log decay a_t = sum_{s<=t} dt_s A[h]
// for t = lane*R .. lane*R+R-1 (dt = 0 past the chunk's end, so a_t stays at
// a_last there), with each lane's dt values.
template <int Q>
struct ChunkDecay {
    static constexpr int R = Q / 32;
    float a[R];
    float d[R];
    float last;
};

// This lane's dt values of head h in the chunk (tokens lane*R .. +R-1; 0 past its end).
template <int Q>
__device__ __forceinline__ void chunk_dt(const ScanArgs &a, const ChunkRange &c, int h, int lane,
                                         float (&d)[ChunkDecay<Q>::R])
{
    constexpr int R = ChunkDecay<Q>::R;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int t = lane * R + r;
        d[r] = t < c.len ? a.dt[(size_t)(c.t0 + t) * a.H + h] : 0.f;
    }
}

// chunk_decay from dt values this lane already holds (chunk_dt), A[h] = Ah.
template <int Q>
__device__ __forceinline__ void chunk_decay_from(float Ah, const float (&d)[ChunkDecay<Q>::R], int lane,
                                                 ChunkDecay<Q> &cd)
{
    constexpr int R = ChunkDecay<Q>::R;
    float run = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        cd.d[r] = d[r];
        run += cd.d[r] * Ah;
        cd.a[r] = run;
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float v = __shfl_up_sync(kFullMask, incl, off);
        if (lane >= off)
            incl += v;
    }
    float excl = __shfl_up_sync(kFullMask, incl, 1);
    if (lane == 0)
        excl = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r)
        cd.a[r] += excl;
    cd.last = __shfl_sync(kFullMask, incl, 31);
}

template <int Q>
__device__ __forceinline__ void chunk_decay(const ScanArgs &a, const ChunkRange &c, int h, int lane,
                                            ChunkDecay<Q> &cd)
{
    constexpr int R = ChunkDecay<Q>::R;
    const float Ah = a.A[h];
    float run = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int t = lane * R + r;
        cd.d[r] = t < c.len ? a.dt[(size_t)(c.t0 + t) * a.H + h] : 0.f;
        run += cd.d[r] * Ah;
        cd.a[r] = run;
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float v = __shfl_up_sync(kFullMask, incl, off);
        if (lane >= off)
            incl += v;
    }
    float excl = __shfl_up_sync(kFullMask, incl, 1);
    if (lane == 0)
        excl = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r)
        cd.a[r] += excl;
    cd.last = __shfl_sync(kFullMask, incl, 31);
}

}  // namespace ssd
}  // namespace ssm
