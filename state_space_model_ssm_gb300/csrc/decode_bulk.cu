// Decode as a stream of state tiles through shared memory (sm_103a).
//
// A decode step is almost nothing but state traffic: every state row is read
// from its slot, updated once and written back ("keep the Mamba2 scan state in
// registers", gllm PR 90, "How the layout was chosen").  The warp-per-row
// kernel in decode.cu keeps a few rows in flight per warp and retires its
// blocks in waves, so each wave pays the full memory latency.  Here a
// persistent grid streams the slots instead:
//
//   - the state of all sequences is cut into tiles of kDbRows consecutive rows
//     of one slot (kDbRows * d_state * 4 contiguous bytes: 8 KiB at d_state
//     128); block b takes tiles b, b + gridDim.x, ... (its local tiles 0, 1, ...);
//   - a producer thread moves each local tile into stage (i % kDbStages) of a
//     shared-memory ring with one bulk copy (cp.async.bulk, completion counted
//     on the stage's mbarrier) and writes the tile's sequence data (length,
//     first token, resume flag) beside it, up to kDbStages tiles ahead;
//   - compute warp w takes local tiles w, w + kDbComputeWarps, ...: it holds
//     the tile's rows in registers (lane j holds a row's float4 j), issues a
//     token's loads for the whole tile at once (x and dt by the lane of each
//     row, B and C once for the tile's group) and hands them to the rows by
//     shuffles, steps kDbBatch rows at a time (their sums reduced together by
//     a transposing shuffle reduction), writes y, and writes the tile back to
//     its slot with one bulk store (cp.async.bulk to global); the stage is
//     released once that store has read it.
// The warps work on different tiles at once, so a tile's memory latency
// overlaps the other warps' tiles, and the grid never drains between tiles.
// The arithmetic is the recurrence of "The llama journey", Day 14 (decay
// exp(dt A), input dt x B, y from the updated state) plus the D x skip term,
// the same as decode.cu; every sequence length works (the rows step through
// the sequence's tokens with the state in registers), though the kernel is
// meant for one token per sequence.
//
// Every wait is bounded.  A wait that gives up sets the kernel's status word
// and marks the block failed: its warps then write NaN to the y rows of their
// remaining tiles, store no further tile (those slots keep their contents),
// wait for the copies in flight and return.
#include <algorithm>
#include <climits>

#include "scan_common.cuh"
#include "tc_common.cuh"

namespace ssm {

namespace {

constexpr int kDbRows = 16;                 // state rows per tile
constexpr int kDbStages = 16;               // tiles in flight per block
constexpr int kDbComputeWarps = 8;          // each takes whole tiles
constexpr int kDbThreads = 32 * (kDbComputeWarps + 1);
constexpr int kDbBatch = 4;                 // rows a warp steps together
static_assert(kDbStages % kDbComputeWarps == 0 && kDbStages >= 2 * kDbComputeWarps, "stage ring");

// Set when a bounded wait of decode_bulk_kernel gave up (read back under
// SSM_SCAN_CHECK, cleared by the host before each checked call).
__device__ int g_decode_bulk_status;

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *mbar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
                 ::"r"(tc::smem_u32(dst)), "l"(src), "r"(bytes), "r"(tc::smem_u32(mbar)) : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n"
                 ::"l"(dst), "r"(tc::smem_u32(src)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }

// Every bulk store group of this thread but the newest `N` has read its
// shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;\n" ::"n"(N) : "memory");
}

// Every bulk store group of this thread is complete (its writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

struct Tile {
    int seq, r0, rows;
};

__device__ __forceinline__ Tile tile_of(int tile, int tiles_per_seq, int HP)
{
    Tile t;
    t.seq = tile / tiles_per_seq;
    t.r0 = (tile - t.seq * tiles_per_seq) * kDbRows;
    t.rows = min(kDbRows, HP - t.r0);
    return t;
}

// Sequence data of a staged tile, written by the producer beside the stage.
struct TileMeta {
    int len, tok_start, resume, pad;
};

// A tile's slot is read when its sequence resumes, written unless the sequence
// resumes with no tokens (then the slot keeps its contents).
__global__ void __launch_bounds__(kDbThreads, 1)
decode_bulk_kernel(const ScanArgs a, int n_tiles, int tiles_per_seq, int fail_waits)
{
    griddep_entry();
    extern __shared__ __align__(128) float db_smem[];
    const int N = a.N, N4 = a.N >> 2, P = a.P, H = a.H;
    const int HP = H * P;
    const uint32_t tile_floats = (uint32_t)kDbRows * N;
    TileMeta *meta = reinterpret_cast<TileMeta *>(db_smem + kDbStages * tile_floats);
    uint64_t *full = reinterpret_cast<uint64_t *>(meta + kDbStages);
    uint64_t *empty = full + kDbStages;
    int *failed = reinterpret_cast<int *>(empty + kDbStages);
    const long cap = fail_waits ? 0 : tc::kSpinLimit;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_local = n_tiles > (int)blockIdx.x ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

    if (tid == 0) {
        for (int s = 0; s < kDbStages; ++s) {
            tc::mbar_init(full + s, 1);
            tc::mbar_init(empty + s, 1);
        }
        *failed = 0;
        tc::mbar_init_fence();
    }
    __syncthreads();

    if (warp == kDbComputeWarps) {
        // ---- producer: lane 0 moves the block's tiles into the ring; the
        // warp's 32 lanes fetch the sequence data of 32 tiles at a time, so the
        // issuing lane never waits on one tile's metadata before its copy ----
        int issued = 0;
        bool stop = false;
        for (int base = 0; base < n_local && !stop; base += 32) {
            TileMeta mine{0, 0, 0, 0};
            Tile tl{0, 0, 0};
            if (base + lane < n_local) {
                tl = tile_of((int)blockIdx.x + (base + lane) * (int)gridDim.x, tiles_per_seq, HP);
                mine.len = a.seq_lens[tl.seq];
                mine.tok_start = a.seq_starts[tl.seq];
                mine.resume = a.resume[tl.seq] != 0;
            }
            const int nb = min(32, n_local - base);
            for (int j = 0; j < nb; ++j) {
                TileMeta m;
                m.len = __shfl_sync(kFullMask, mine.len, j);
                m.tok_start = __shfl_sync(kFullMask, mine.tok_start, j);
                m.resume = __shfl_sync(kFullMask, mine.resume, j);
                m.pad = 0;
                const int seq = __shfl_sync(kFullMask, tl.seq, j);
                const int r0 = __shfl_sync(kFullMask, tl.r0, j);
                const int rows = __shfl_sync(kFullMask, tl.rows, j);
                int go = 1;
                if (lane == 0) {
                    const int i = base + j;
                    const int s = i % kDbStages;
                    if (i >= kDbStages && !tc::mbar_wait(empty + s, (uint32_t)((i / kDbStages - 1) & 1), cap)) {
                        atomicExch(&g_decode_bulk_status, 1);
                        atomicExch(failed, 1);
                        go = 0;
                    } else if (*reinterpret_cast<volatile int *>(failed)) {
                        go = 0;
                    } else {
                        meta[s] = m;
                        if (m.resume) {
                            const uint32_t bytes = (uint32_t)rows * N * 4;
                            tc::mbar_expect_tx(full + s, bytes);
                            bulk_load(db_smem + s * tile_floats, a.state + ((long long)seq * HP + r0) * N, bytes,
                                      full + s);
                        } else {
                            tc::mbar_arrive(full + s);   // a fresh sequence starts from zero: nothing to read
                        }
                        issued = i + 1;
                    }
                }
                if (!__shfl_sync(kFullMask, go, 0)) {
                    stop = true;
                    break;
                }
            }
        }
        // no copy may land after the block is gone: wait for the loads of the
        // stages whose tiles were issued but may not have been consumed
        if (lane == 0)
            for (int k = max(0, issued - kDbStages); k < issued; ++k)
                tc::mbar_wait(full + k % kDbStages, (uint32_t)((k / kDbStages) & 1));
        return;
    }

    // ---- compute warps: warp w takes local tiles w, w + kDbComputeWarps, ... ----
    constexpr int R = kDbBatch;
    bool ok = true;
    int prev_stage = -1;                              // stage of this warp's previous tile
    for (int i = warp; i < n_local; i += kDbComputeWarps) {
        const int s = i % kDbStages;
        const Tile t = tile_of((int)blockIdx.x + i * (int)gridDim.x, tiles_per_seq, HP);
        bool got = true;                              // every lane acquires the stage's data itself
        if (ok && !tc::mbar_wait(full + s, (uint32_t)((i / kDbStages) & 1), cap)) {
            atomicExch(&g_decode_bulk_status, 1);
            atomicExch(failed, 1);
            got = false;
        }
        // one decision per warp (its lanes shuffle together), taken by lane 0
        ok = __shfl_sync(kFullMask, ok && got && !*reinterpret_cast<volatile int *>(failed), 0);
        const TileMeta m = meta[s];                   // published before the stage's barrier completed
        const int len = ok ? m.len : a.seq_lens[t.seq];
        const long long tok_start = ok ? m.tok_start : a.seq_starts[t.seq];
        const bool resume = m.resume != 0;
        float *st = db_smem + s * tile_floats;
        if (!ok) {                                    // a failed wait: mark this tile's outputs
            for (int k = 0; k < len; ++k)
                if (lane < t.rows)
                    a.y[(tok_start + k) * HP + t.r0 + lane] = __int_as_float(0x7fc00000);
        } else {
            // lane l < rows carries row l's scalars; each token's loads for the
            // whole tile (x and dt per row, B and C per group) are issued
            // together and reach the rows through shuffles
            const int rl = min(lane, t.rows - 1), r = t.r0 + rl;
            const int hl = r / P, gl = hl / (H / a.G);
            const float Al = __ldg(a.A + hl), Dl = __ldg(a.D + hl);   // lane l: row l's head
            const int g_first = __shfl_sync(kFullMask, gl, 0), g_last = __shfl_sync(kFullMask, gl, t.rows - 1);
            const bool one_group = g_first == g_last;
            float4 v[kDbRows];
#pragma unroll
            for (int q = 0; q < kDbRows; ++q) {
                v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (resume && q < t.rows && lane < N4)
                    v[q] = *reinterpret_cast<const float4 *>(st + q * N + 4 * lane);
            }
            const int qy = reduced_row<32, R>(lane);
            for (int k = 0; k < len; ++k) {
                const long long tok = tok_start + k;
                // row l's scalars, formed once by its lane: decay, input weight, skip term
                const float xl = __ldg(a.x + tok * HP + r);
                const float dtl = __ldg(a.dt + tok * H + hl);
                const float dAl = expf(dtl * Al), xdtl = dtl * xl, dxl = Dl * xl;
                float4 b1 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = b1;
                if (one_group && lane < N4) {
                    b1 = __ldg(reinterpret_cast<const float4 *>(a.B + (tok * a.G + g_first) * N) + lane);
                    c1 = __ldg(reinterpret_cast<const float4 *>(a.C + (tok * a.G + g_first) * N) + lane);
                }
#pragma unroll
                for (int rb = 0; rb < kDbRows; rb += R) {
                    if (rb >= t.rows)
                        break;                        // uniform over the warp
                    float part[R];
#pragma unroll
                    for (int q = 0; q < R; ++q) {
                        const int row = min(rb + q, t.rows - 1);
                        const float dA = __shfl_sync(kFullMask, dAl, row);
                        const float xdt = __shfl_sync(kFullMask, xdtl, row);
                        float4 bq = b1, cq = c1;
                        if (!one_group) {             // a tile across a group boundary
                            const int gq = __shfl_sync(kFullMask, gl, row);
                            if (lane < N4) {
                                bq = __ldg(reinterpret_cast<const float4 *>(a.B + (tok * a.G + gq) * N) + lane);
                                cq = __ldg(reinterpret_cast<const float4 *>(a.C + (tok * a.G + gq) * N) + lane);
                            }
                        }
                        float4 &w = v[rb + q];
                        if (lane < N4) {
                            w.x = fmaf(w.x, dA, xdt * bq.x);
                            w.y = fmaf(w.y, dA, xdt * bq.y);
                            w.z = fmaf(w.z, dA, xdt * bq.z);
                            w.w = fmaf(w.w, dA, xdt * bq.w);
                        }
                        part[q] = fmaf(w.x, cq.x, w.y * cq.y) + fmaf(w.z, cq.z, w.w * cq.w);
                    }
                    const float ysum = reduce_rows<32, R>(part, lane);
                    const float dx = __shfl_sync(kFullMask, dxl, min(rb + qy, t.rows - 1));
                    if (reduced_writer<32, R>(lane) && rb + qy < t.rows)
                        a.y[tok * HP + t.r0 + rb + qy] = dx + ysum;
                }
            }
            if (lane < N4) {
#pragma unroll
                for (int q = 0; q < kDbRows; ++q)
                    if (q < t.rows)
                        *reinterpret_cast<float4 *>(st + q * N + 4 * lane) = v[q];
            }
        }
        // the tile written in shared memory, visible to the bulk copy engine
        tc::fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (ok && (len > 0 || !resume))
                bulk_store(a.state + ((long long)t.seq * HP + t.r0) * N, st, (uint32_t)t.rows * N * 4);
            bulk_commit();                            // one group per tile (possibly empty)
            bulk_wait_read<1>();                      // this warp's previous store has read its stage
            if (prev_stage >= 0)
                tc::mbar_arrive(empty + prev_stage);
        }
        prev_stage = s;
    }
    if (lane == 0) {
        bulk_wait_all();                              // every store performed before the block ends
        if (prev_stage >= 0)
            tc::mbar_arrive(empty + prev_stage);
    }
}

}  // namespace

bool decode_bulk_supported(int N, size_t smem_optin)
{
    return N % 4 == 0 && N <= 128 && decode_bulk_smem_bytes(N) <= smem_optin;
}

size_t decode_bulk_smem_bytes(int N)
{
    return (size_t)kDbStages * kDbRows * N * sizeof(float) + kDbStages * sizeof(TileMeta) +
           2 * kDbStages * sizeof(uint64_t) + 16;
}

cudaError_t launch_decode_bulk(const ScanArgs &a, int sms, int fail_waits, cudaStream_t stream)
{
    const int HP = a.H * a.P;
    const int tiles_per_seq = (HP + kDbRows - 1) / kDbRows;
    const long long n_tiles = (long long)a.n_seqs * tiles_per_seq;
    if (n_tiles <= 0)
        return cudaSuccess;
    if (n_tiles > INT_MAX)
        return cudaErrorInvalidValue;
    const size_t smem = decode_bulk_smem_bytes(a.N);
    const cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(decode_bulk_kernel), smem);
    if (e != cudaSuccess)
        return e;
    // a persistent grid: as many blocks as can be resident at once, no more than tiles
    int per_sm = 0;
    const cudaError_t eo = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_bulk_kernel, kDbThreads, smem);
    if (eo != cudaSuccess)
        return eo;
    const long long grid = std::min<long long>(n_tiles, (long long)std::max(1, per_sm) * sms);
    return launch_pdl(decode_bulk_kernel, dim3((unsigned)grid), dim3(kDbThreads), smem, stream, a, (int)n_tiles,
                      tiles_per_seq, fail_waits);
}

cudaError_t decode_bulk_status(int *status, cudaStream_t stream, bool clear)
{
    if (clear) {
        const int zero = 0;
        return cudaMemcpyToSymbolAsync(g_decode_bulk_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                                       stream);
    }
    cudaError_t e = cudaMemcpyFromSymbolAsync(status, g_decode_bulk_status, sizeof(int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(stream);
    return e;
}

}  // namespace ssm
