// libssmscan C ABI: argument checks, path and launch-shape choice.
//
// Everything here runs on the host and returns before any launch when an
// argument is wrong.  Nothing is allocated and the stream is never
// synchronised (except in the opt-in SSM_SCAN_CHECK=1 debug mode).
#include <climits>
#include <mutex>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <vector>
#include <algorithm>

#include "../../include/ssmscan.h"
#include "scan_common.cuh"

namespace ssm {

cudaError_t set_dynamic_smem(const void *kernel, size_t bytes)
{
    struct Entry {
        int dev;
        const void *kernel;
        size_t bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lock(mu);
    for (Entry &d : done)
        if (d.dev == dev && d.kernel == kernel) {
            if (d.bytes >= bytes)
                return cudaSuccess;
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
            if (e == cudaSuccess)
                d.bytes = bytes;
            return e;
        }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess)
        done.push_back(Entry{dev, kernel, bytes});
    return e;
}

}  // namespace ssm

namespace {

constexpr int kMaxDState = 1024;
constexpr int kMaxConvKernel = 8;
constexpr int kMaxDevices = 64;

int pow2ceil(int v)
{
    int p = 1;
    while (p < v)
        p <<= 1;
    return p;
}

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Smallest compiled float4-per-lane count that covers a row of N4 float4
// chunks with `lanes` lanes, or 0 when no compiled kernel fits.
int pick_vpl(int N4, int lanes, int rpt, bool (*supported)(int, int, int))
{
    const int need = (N4 + lanes - 1) / lanes;
    for (int v = 1; v <= 8; v <<= 1)
        if (v >= need && supported(lanes, v, rpt))
            return v;
    return 0;
}

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;        // largest dynamic shared memory of one block
    int smem_per_sm = 0;       // shared memory of one SM
};

int device_info(DeviceInfo *out)
{
    static DeviceInfo cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return SSM_ERR_CUDA;
    if (cache[dev].sms == 0) {
        DeviceInfo d;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SSM_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return SSM_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
            return SSM_ERR_CUDA;
        cache[dev] = d;
    }
    *out = cache[dev];
    return SSM_OK;
}

bool check_env()
{
    static int v = -1;
    if (v < 0) {
        const char *e = std::getenv("SSM_SCAN_CHECK");
        v = (e && e[0] && std::strcmp(e, "0") != 0) ? 1 : 0;
    }
    return v == 1;
}

// Test hook (SSM_SCAN_TEST_FAIL_WAITS=1, read once): the pipelined tensor-core
// kernels' bounded waits give up at once, so a test sees the timeout path
// (status word, SSM_ERR_TIMEOUT under SSM_SCAN_CHECK) without a stalled GPU.
// Their drain of the copies and products in flight keeps its full bound.
bool fail_waits_env()
{
    static int v = -1;
    if (v < 0) {
        const char *e = std::getenv("SSM_SCAN_TEST_FAIL_WAITS");
        v = (e && e[0] && std::strcmp(e, "0") != 0) ? 1 : 0;
    }
    return v == 1;
}

// Debug mode: SSM_ERR_TIMEOUT when a kernel's bounded wait gave up (the
// device status word is nonzero); synchronises the stream.
int read_status(const int *status, cudaStream_t stream)
{
    int st = 0;
    if (cudaMemcpyAsync(&st, status, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return SSM_ERR_CUDA;
    return st != 0 ? SSM_ERR_TIMEOUT : SSM_OK;
}

// Debug mode: copy the sequence table to the host and check the ranges.
int check_metadata(const ssm::ScanArgs &a, cudaStream_t stream)
{
    const size_t n = (size_t)a.n_seqs;
    std::vector<int32_t> st(n), ln(n);
    if (cudaMemcpyAsync(st.data(), a.seq_starts, n * sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyAsync(ln.data(), a.seq_lens, n * sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return SSM_ERR_CUDA;
    std::vector<std::pair<int32_t, int32_t>> ranges;
    for (size_t i = 0; i < n; ++i) {
        if (st[i] < 0 || ln[i] < 0 || (long long)st[i] + ln[i] > a.n_tokens)
            return SSM_ERR_INVALID_ARG;
        if (ln[i] > 0)
            ranges.emplace_back(st[i], st[i] + ln[i]);
    }
    std::sort(ranges.begin(), ranges.end());
    for (size_t i = 1; i < ranges.size(); ++i)
        if (ranges[i].first < ranges[i - 1].second)
            return SSM_ERR_INVALID_ARG;
    return SSM_OK;
}

// Launch shape and segment plan of the prefill path.
struct PrefillPlan {
    bool scaled = true;
    int lanes = 0, rpt = 0, vpl = 0;
    ssm::PrefillGeom g{};
    size_t smem = 0;
    int seg_len = 0;              // 0: no time segments
    long long max_units = 0;      // upper bound of (sequence, segment) units
    size_t ws_bytes = 0;          // workspace the segment plan needs
    bool tc_state = false;        // state pass on the tensor cores (segment_state_tc.cu)
    // workspace offsets (bytes)
    size_t off_units = 0, off_n_units = 0, off_unit_base = 0, off_status = 0, off_decay = 0, off_state = 0;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Shapes for the prefill kernels; also the time-segment plan when segments
// are allowed.  Returns SSM_OK or an error status (no launch happens here).
int plan_prefill(const ssm_scan_tuning &t, bool scaled, int n_seqs, int n_tokens, int H, int P, int N,
                 int G, const DeviceInfo &dev, bool allow_segments, PrefillPlan *out)
{
    PrefillPlan pl;
    pl.scaled = scaled;
    const int N4 = N / 4;
    auto supported = scaled ? ssm::prefill_scaled_supported : ssm::prefill_supported;
    int lanes, rpt;
    if (scaled) {
        // About 16 state elements of a row per lane and up to 4 rows per lane
        // (at most 64 state registers): each B/C value read from shared memory
        // feeds several rows, and the y reduction spans few lanes.  Where no
        // compiled kernel has that shape, about 8 elements per lane.  The rows
        // of a lane must share a head: RPT | P.
        const int cand[2] = {std::min(32, pow2ceil((N + 15) / 16)), std::min(32, pow2ceil((N + 7) / 8))};
        lanes = rpt = 0;
        for (int ci = 0; ci < 2 && !rpt; ++ci) {
            const int l = t.lanes_per_row ? t.lanes_per_row : cand[ci];
            for (int r = t.rows_per_thread ? t.rows_per_thread : 4; r >= 1 && !rpt; r >>= 1) {
                const int v = pick_vpl(N4, l, r, supported);
                if (P % r == 0 && r <= l && v > 0 && v * 4 * r <= 64) {
                    lanes = l;
                    rpt = r;
                }
                if (t.rows_per_thread)
                    break;
            }
        }
        if (!rpt) {                          // an explicit shape the rules above reject
            lanes = t.lanes_per_row ? t.lanes_per_row : cand[1];
            rpt = t.rows_per_thread ? t.rows_per_thread : 1;
        }
        if (P % rpt != 0)
            return SSM_ERR_INVALID_ARG;
    } else {
        lanes = t.lanes_per_row ? t.lanes_per_row : std::min(32, pow2ceil((N + 31) / 32));
        rpt = t.rows_per_thread ? t.rows_per_thread : 1;
    }
    const int vpl = pick_vpl(N4, lanes, rpt, supported);
    if (rpt > lanes || vpl == 0)
        return SSM_ERR_INVALID_ARG;
    if (scaled && t.chunk_tokens > ssm::kScaledMaxChunk)
        return SSM_ERR_INVALID_ARG;
    auto smem_of = [&](const ssm::PrefillGeom &gg) {
        return scaled ? ssm::prefill_scaled_smem_bytes(gg, N, lanes) : ssm::prefill_smem_bytes(gg, N);
    };
    const int rows_per_warp = (32 / lanes) * rpt;
    ssm::PrefillGeom &g = pl.g;
    g.rows_per_group = (H / G) * P;
    if (t.rows_per_cta) {
        // the rescaled kernel adds one producer warp to the block's 256 threads
        if (t.rows_per_cta % rows_per_warp != 0 || (t.rows_per_cta / rpt) * lanes > (scaled ? 224 : 256))
            return SSM_ERR_INVALID_ARG;
        g.rows_per_cta = t.rows_per_cta;
    } else {
        // Largest block (up to 4 warps) that still gives every SM a block; with
        // time segments the segments supply the blocks.
        int warps = 4;
        while (warps > 1 && !(scaled && allow_segments)) {
            const long long runs = (g.rows_per_group + warps * rows_per_warp - 1) / (warps * rows_per_warp);
            if ((long long)n_seqs * G * runs >= dev.sms)
                break;
            warps >>= 1;
        }
        g.rows_per_cta = warps * rows_per_warp;
    }
    const int threads = (g.rows_per_cta / rpt) * lanes;
    g.runs_per_group = (g.rows_per_group + g.rows_per_cta - 1) / g.rows_per_cta;
    g.heads_cap = (P + g.rows_per_cta - 2) / P + 1;
    // The direct kernel carries one chunk's dt in 4 registers per thread.
    const int dt_cap = scaled ? INT_MAX : 4 * threads;
    // Two blocks per SM fit in the 228 KB of shared memory (1 KB per block is reserved).
    const size_t smem_cap = (size_t)(N > 256 ? dev.smem_optin : std::min(dev.smem_optin, 113 * 1024));
    if (t.chunk_tokens) {
        g.chunk = t.chunk_tokens;
        if ((long long)g.chunk * g.heads_cap > dt_cap || smem_of(g) > (size_t)dev.smem_optin)
            return SSM_ERR_INVALID_ARG;
    } else {
        // 16 tokens for the rescaled kernel: a chunk's running decay seldom
        // crosses a re-anchor point, so its tokens run in straight-line groups
        // of four.  An explicit segment length must be a multiple of the chunk.
        g.chunk = scaled ? 16 : 32;
        while (g.chunk > 1 && ((long long)g.chunk * g.heads_cap > dt_cap || smem_of(g) > smem_cap ||
                               (scaled && t.segment_tokens > 0 && t.segment_tokens % g.chunk != 0)))
            g.chunk >>= 1;
        if (smem_of(g) > (size_t)dev.smem_optin)
            return SSM_ERR_UNSUPPORTED;
    }
    pl.smem = smem_of(g);
    pl.lanes = lanes;
    pl.rpt = rpt;
    pl.vpl = vpl;

    // Time segments: only the rescaled kernel has the state pass.  Automatic
    // choice (the host does not see the lengths): about as many units as
    // sequences, and at least enough for about six consumer warps per SM
    // sub-partition, so that the tokens spread evenly over the units and no
    // long sequence of a ragged batch runs alone; off when no sequence can be
    // long enough to split.
    if (scaled && allow_segments && t.segment_tokens >= 0 && n_tokens > 0) {
        int seg = 0;
        if (t.segment_tokens > 0) {
            if (t.segment_tokens % g.chunk != 0)
                return SSM_ERR_INVALID_ARG;
            seg = t.segment_tokens;
        } else {
            const long long warps_per_unit = (long long)G * g.runs_per_group * (threads / 32);
            const long long target = 6LL * 4 * dev.sms;      // consumer warps to keep resident
            const long long want = std::max<long long>((target + warps_per_unit - 1) / warps_per_unit, n_seqs);
            long long L = ((long long)n_tokens + want - 1) / want;
            L = std::max<long long>(L, 4LL * g.chunk);
            L = ((L + g.chunk - 1) / g.chunk) * g.chunk;
            const long long longest = (long long)n_tokens - std::max(0, n_seqs - 1);   // every other one >= 1
            seg = L < longest ? (int)L : 0;
        }
        if (seg > 0) {
            // The state pass: tensor cores where the shapes fit, unless the
            // caller asks for the sequential kernel's state-only mode.
            if (t.segment_state == SSM_SEGMENT_STATE_FP32) {
                pl.tc_state = false;
            } else {
                pl.tc_state = ssm::segment_state_tc_supported(N, P, (size_t)dev.smem_optin);
                if (!pl.tc_state && t.segment_state == SSM_SEGMENT_STATE_TENSOR)
                    return SSM_ERR_UNSUPPORTED;
            }
            pl.seg_len = seg;
            pl.max_units = (long long)n_seqs + ((long long)n_tokens + seg - 1) / seg;
            const size_t slot = (size_t)H * P * N * sizeof(float);
            size_t off = 0;
            pl.off_units = off;      off = align256(off + (size_t)pl.max_units * sizeof(int2));
            pl.off_n_units = off;    off = align256(off + sizeof(int));
            pl.off_unit_base = off;  off = align256(off + ((size_t)n_seqs + 1) * sizeof(int));
            pl.off_status = off;     off = align256(off + sizeof(int));
            pl.off_decay = off;      off = align256(off + (size_t)pl.max_units * H * sizeof(float));
            pl.off_state = off;      off = align256(off + (size_t)pl.max_units * slot);
            pl.ws_bytes = off;
        }
    }
    *out = pl;
    return SSM_OK;
}

// Workspace bytes the discretised step takes (0 without the dt options).
size_t dt_buffer_bytes(const ssm_scan_options &o, int n_tokens, int H)
{
    if (!o.dt_bias && !o.dt_softplus)
        return 0;
    return align256((size_t)n_tokens * H * sizeof(float));
}

// Copy the caller's options (NULL = all off) and check their pointers.
int read_options(const ssm_scan_options *opts, ssm_scan_options *out)
{
    std::memset(out, 0, sizeof *out);
    if (!opts)
        return SSM_OK;
    *out = *opts;
    if (!aligned(out->dt_bias, 4) || !aligned(out->state_snapshots, 16))
        return SSM_ERR_INVALID_ARG;
    if (out->n_launch_events < 0 || (out->n_launch_events > 0 && !out->launch_events))
        return SSM_ERR_INVALID_ARG;
    if (out->gated_y) {
        if (!out->gate_z || !out->norm_weight || !(out->norm_eps > 0.f))
            return SSM_ERR_INVALID_ARG;
        if (!aligned(out->gated_y, 16) || !aligned(out->gate_z, 16) || !aligned(out->norm_weight, 16))
            return SSM_ERR_INVALID_ARG;
    }
    return SSM_OK;
}

// Launches the scan kernels for a checked call (everything after the argument
// checks); the options' post-scan steps run in scan_impl.
// With `gated` set, the full pass of the rescaled prefill writes the gated
// RMSNorm output itself where its shape allows (*gated_done = true); otherwise
// the caller runs the separate norm kernel after the scan.
int scan_kernels(const ssm::ScanArgs &a, const ssm_scan_tuning &t, const DeviceInfo &dev, void *workspace,
                 size_t workspace_bytes, cudaStream_t stream, ssm::LaunchTimer *tm, const ssm::GatedOut *gated,
                 bool *gated_done);

int scan_impl(float *state, const float *x, const float *dt, const float *A, const float *B,
              const float *C, const float *D, float *y, const int32_t *seq_starts,
              const int32_t *seq_lens, const int32_t *resume, int n_seqs, int n_tokens,
              int H, int P, int N, int G, const ssm_scan_tuning *tun, const ssm_scan_options *opts,
              void *workspace, size_t workspace_bytes, void *stream_v)
{
    // ---- host-checkable arguments ----
    if (n_seqs < 0 || n_tokens < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0)
        return SSM_ERR_INVALID_ARG;
    if (H % G != 0)
        return SSM_ERR_INVALID_ARG;
    if (N % 4 != 0 || N > kMaxDState)
        return SSM_ERR_UNSUPPORTED;
    if ((long long)H * P > INT_MAX / 2)
        return SSM_ERR_UNSUPPORTED;
    if (n_seqs == 0)
        return SSM_OK;
    if (!state || !A || !D || !seq_starts || !seq_lens || !resume)
        return SSM_ERR_INVALID_ARG;
    if (n_tokens > 0 && (!x || !dt || !B || !C || !y))
        return SSM_ERR_INVALID_ARG;
    if (!aligned(state, 16) || !aligned(B, 16) || !aligned(C, 16))
        return SSM_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(dt, 4) || !aligned(A, 4) || !aligned(D, 4) || !aligned(y, 4) ||
        !aligned(seq_starts, 4) || !aligned(seq_lens, 4) || !aligned(resume, 4))
        return SSM_ERR_INVALID_ARG;

    ssm_scan_options o;
    int rc = read_options(opts, &o);
    if (rc != SSM_OK)
        return rc;
    // The discretised step goes to the front of the workspace; the rest is
    // what the segment plan may use.
    const size_t dtb = dt_buffer_bytes(o, n_tokens, H);
    if (dtb > 0 && (!workspace || !aligned(workspace, 256) || workspace_bytes < dtb))
        return SSM_ERR_INVALID_ARG;
    ssm_scan_tuning t;
    std::memset(&t, 0, sizeof t);
    if (tun)
        t = *tun;
    if (t.path < SSM_PATH_AUTO || t.path > SSM_PATH_PREFILL_DIRECT || t.lanes_per_row < 0 ||
        t.rows_per_thread < 0 || t.rows_per_cta < 0 || t.chunk_tokens < 0 || t.chunk_tokens > 256 ||
        t.ctas_per_sm < 0 || t.segment_state < SSM_SEGMENT_STATE_AUTO || t.segment_state > SSM_SEGMENT_STATE_TENSOR)
        return SSM_ERR_INVALID_ARG;
    if (t.lanes_per_row && (!is_pow2(t.lanes_per_row) || t.lanes_per_row > 32))
        return SSM_ERR_INVALID_ARG;
    if (t.rows_per_thread && !is_pow2(t.rows_per_thread))
        return SSM_ERR_INVALID_ARG;

    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != SSM_OK)
        return rc;

    ssm::ScanArgs a;
    a.state = state; a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.y = y;
    a.seq_starts = seq_starts; a.seq_lens = seq_lens; a.resume = resume;
    a.n_seqs = n_seqs; a.n_tokens = n_tokens; a.H = H; a.P = P; a.N = N; a.G = G;
    a.snaps = o.state_snapshots;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
    if (a.snaps) {                          // the decode kernel steps tokens one by one
        if (t.path == SSM_PATH_PREFILL || t.path == SSM_PATH_PREFILL_DIRECT)
            return SSM_ERR_UNSUPPORTED;
        t.path = SSM_PATH_DECODE;
    }

    if (check_env()) {
        rc = check_metadata(a, stream);
        if (rc != SSM_OK)
            return rc;
    }
    ssm::LaunchTimer tm{o.launch_events, o.n_launch_events, 0, stream, false};
    if (dtb > 0) {
        float *step = static_cast<float *>(workspace);
        if (ssm::timed(&tm, [&] { return ssm::launch_dt_prep(a, o.dt_bias, o.dt_softplus, step, stream); }) !=
            cudaSuccess)
            return SSM_ERR_CUDA;
        a.dt = step;
        workspace = static_cast<char *>(workspace) + dtb;
        workspace_bytes -= dtb;
    }
    const ssm::GatedOut gated{o.gate_z, o.norm_weight, o.norm_eps, o.gated_y};
    bool gated_done = false;
    rc = scan_kernels(a, t, dev, workspace, workspace_bytes, stream, &tm, o.gated_y ? &gated : nullptr,
                      &gated_done);
    if (rc != SSM_OK)
        return rc;
    if (o.gated_y && n_tokens > 0 && !gated_done &&
        ssm::timed(&tm, [&] {
            return ssm::launch_gated_norm(a, o.gate_z, o.norm_weight, o.norm_eps, o.gated_y, stream);
        }) != cudaSuccess)
        return SSM_ERR_CUDA;
    return tm.failed ? SSM_ERR_CUDA : SSM_OK;
}

int scan_kernels(const ssm::ScanArgs &a, const ssm_scan_tuning &t, const DeviceInfo &dev, void *workspace,
                 size_t workspace_bytes, cudaStream_t stream, ssm::LaunchTimer *tm, const ssm::GatedOut *gated,
                 bool *gated_done)
{
    *gated_done = false;
    const int n_seqs = a.n_seqs, n_tokens = a.n_tokens, H = a.H, P = a.P, N = a.N, G = a.G;
    int rc = SSM_OK;
    const int N4 = N / 4;
    int path = t.path;
    if (path == SSM_PATH_AUTO)
        path = (n_tokens == n_seqs) ? SSM_PATH_DECODE : SSM_PATH_PREFILL;

    if (path == SSM_PATH_DECODE) {
        const int lanes = t.lanes_per_row ? t.lanes_per_row : std::min(32, pow2ceil(N4));
        int rpt = t.rows_per_thread;
        if (!rpt) {     // up to 4 rows in flight per lane, a divisor of P
            rpt = (lanes == 32 && N4 <= 32) ? 4 : 1;
            while (P % rpt)
                rpt >>= 1;
        }
        const int vpl = pick_vpl(N4, lanes, rpt, ssm::decode_supported);
        if (rpt > lanes || vpl == 0 || P % rpt != 0)
            return SSM_ERR_INVALID_ARG;
        ssm::DecodeGeom g;
        g.rows_per_warp = (32 / lanes) * rpt;
        g.tasks_per_seq = (H * P + g.rows_per_warp - 1) / g.rows_per_warp;
        const long long blocks_per_seq = (g.tasks_per_seq + ssm::kDecodeWarps - 1) / ssm::kDecodeWarps;
        long long grid_seqs = std::min<long long>(n_seqs, 65535);
        if (t.ctas_per_sm > 0)
            grid_seqs = std::max<long long>(1, std::min<long long>(
                grid_seqs, (long long)t.ctas_per_sm * dev.sms / std::max<long long>(1, blocks_per_seq)));
        if (blocks_per_seq > INT_MAX)
            return SSM_ERR_UNSUPPORTED;
        if (ssm::timed(tm, [&] { return ssm::launch_decode(a, g, lanes, vpl, rpt, (int)grid_seqs, stream); }) !=
            cudaSuccess)
            return SSM_ERR_CUDA;
        return SSM_OK;
    }

    // ---- prefill ----
    const bool scaled = (path == SSM_PATH_PREFILL);
    PrefillPlan pl;
    rc = plan_prefill(t, scaled, n_seqs, n_tokens, H, P, N, G, dev, workspace != nullptr, &pl);
    if (rc != SSM_OK)
        return rc;
    if (pl.seg_len > 0 && (workspace_bytes < pl.ws_bytes || !aligned(workspace, 256))) {
        if (t.segment_tokens > 0)
            return SSM_ERR_INVALID_ARG;     // explicit segments need the workspace
        pl.seg_len = 0;                     // automatic: run without segments
    }
    ssm::SegStateMaps maps;                 // TMA descriptors of the tensor-core state pass
    if (pl.seg_len > 0 && pl.tc_state && !(aligned(a.x, 16) && ssm::segment_state_tc_maps(a, &maps))) {
        if (t.segment_state == SSM_SEGMENT_STATE_TENSOR)
            return SSM_ERR_UNSUPPORTED;
        pl.tc_state = false;
    }
    if (pl.max_units * G * pl.g.runs_per_group > INT_MAX || (long long)n_seqs * G * pl.g.runs_per_group > INT_MAX)
        return SSM_ERR_UNSUPPORTED;
    if (!scaled) {
        if (ssm::timed(tm, [&] {
                return ssm::launch_prefill(a, pl.g, pl.lanes, pl.vpl, pl.rpt, pl.smem, dev.sms, stream);
            }) != cudaSuccess)
            return SSM_ERR_CUDA;
        return SSM_OK;
    }
    // Output of the full pass.  Blocks of exactly four consumer warps run
    // self-staged, without a producer warp, three per SM: y through tiles that
    // all warps write out one chunk later (epi 5), and with the gated RMSNorm requested y and
    // z through tiles (epi 4: blocks of exactly one head, x, y, z and the gated
    // output 16-byte aligned).  Other shapes with the
    // output-tile variants keep a producer warp: y goes through a shared-memory
    // tile that it writes out (epi 1; about 1 % faster than the consumers' own
    // stores, which the remaining shapes keep: epi 0), and the gated output is
    // applied by the consumer warps from that tile (epi 2, one head per block,
    // z 16-byte aligned and staged like x).  Each needs its extra tiles to fit
    // the shared memory.
    const ssm::GatedOut *fuse = nullptr;
    int epi = 0;
    size_t smem_full = pl.smem;
    const bool self_ok = n_tokens > 0 && ssm::prefill_scaled_self_supported(pl.lanes, pl.vpl, pl.rpt, pl.g.rows_per_cta);
    auto three_per_sm = [&](int e) {
        return 3 * (ssm::prefill_scaled_smem_bytes(pl.g, N, pl.lanes, e) + 1024) <= (size_t)dev.smem_per_sm;
    };
    if (self_ok && !gated && three_per_sm(5)) {
        epi = 5;                            // self-staged, y through tiles: three blocks per SM
        smem_full = ssm::prefill_scaled_smem_bytes(pl.g, N, pl.lanes, 5);
    } else if (self_ok && gated && pl.g.rows_per_cta == P && P % 4 == 0 && aligned(gated->z, 16) &&
               aligned(gated->out, 16) && aligned(a.y, 16) && aligned(a.x, 16) && three_per_sm(4)) {
        fuse = gated;                       // self-staged with the gated output
        epi = 4;
        smem_full = ssm::prefill_scaled_smem_bytes(pl.g, N, pl.lanes, 4);
    } else if (n_tokens > 0 && ssm::prefill_scaled_tile_supported(pl.lanes, pl.vpl, pl.rpt, pl.g.rows_per_cta)) {
        if (gated && pl.g.rows_per_cta == P && P % 4 == 0 && P <= 256 && aligned(gated->z, 16) &&
            aligned(gated->out, 16) &&
            ssm::prefill_scaled_smem_bytes(pl.g, N, pl.lanes, 2) <= (size_t)dev.smem_optin) {
            fuse = gated;
            epi = 2;
        } else if (ssm::prefill_scaled_smem_bytes(pl.g, N, pl.lanes, 1) <= (size_t)dev.smem_optin) {
            epi = 1;
        }
        smem_full = ssm::prefill_scaled_smem_bytes(pl.g, N, pl.lanes, epi);
    }
    ssm::SegmentPlan plan{};
    if (pl.seg_len == 0) {
        if (ssm::timed(tm, [&] {
                return ssm::launch_prefill_scaled(a, pl.g, pl.lanes, pl.vpl, pl.rpt, plan, ssm::kScanFull, n_seqs,
                                                  smem_full, stream, epi, fuse);
            }) != cudaSuccess)
            return SSM_ERR_CUDA;
        *gated_done = fuse != nullptr;
        return SSM_OK;
    }
    char *ws = static_cast<char *>(workspace);
    plan.units = reinterpret_cast<const int2 *>(ws + pl.off_units);
    plan.n_units = reinterpret_cast<const int *>(ws + pl.off_n_units);
    plan.unit_base = reinterpret_cast<const int *>(ws + pl.off_unit_base);
    plan.seg_len = pl.seg_len;
    plan.seg_decay = reinterpret_cast<float *>(ws + pl.off_decay);
    plan.seg_state = reinterpret_cast<float *>(ws + pl.off_state);
    plan.status = reinterpret_cast<int *>(ws + pl.off_status);
    plan.fail_waits = fail_waits_env() ? 1 : 0;
    const int mu = (int)pl.max_units;
    if (ssm::timed(tm, [&] { return ssm::launch_segment_plan(a, plan, mu, stream); }) != cudaSuccess)
        return SSM_ERR_CUDA;
    const cudaError_t e = ssm::timed(tm, [&] {
        return pl.tc_state ? ssm::launch_segment_state_tc(a, plan, maps, mu, stream)
                           : ssm::launch_prefill_scaled(a, pl.g, pl.lanes, pl.vpl, pl.rpt, plan, ssm::kScanStateOnly,
                                                        mu, pl.smem, stream);
    });
    if (e != cudaSuccess || ssm::timed(tm, [&] { return ssm::launch_segment_combine(a, plan, mu, stream); }) !=
                                cudaSuccess ||
        ssm::timed(tm, [&] {
            return ssm::launch_prefill_scaled(a, pl.g, pl.lanes, pl.vpl, pl.rpt, plan, ssm::kScanFull, mu, smem_full,
                                              stream, epi, fuse);
        }) != cudaSuccess)
        return SSM_ERR_CUDA;
    *gated_done = fuse != nullptr;
    if (pl.tc_state && check_env())         // debug: report a bounded wait that gave up
        return read_status(plan.status, stream);
    return SSM_OK;
}

// Layout of the SSD workspace and launch shape of its kernels.
struct SsdLayout {
    int chunk = 0;
    long long max_units = 0;
    size_t off_step = 0, off_units = 0, off_n_units = 0, off_status = 0, off_unit_base = 0, off_decay = 0,
           off_state = 0;
    size_t bytes = 0;
    ssm::SsdGeom g{};
};

// Shared-memory row stride (floats) of at least `width` that is == `residue`
// (mod 32), so the fragment loads of a warp hit 32 distinct banks.
int bank_stride(int width, int residue) { return width + ((residue - width % 32) + 64) % 32; }

// Arguments the SSD form accepts, its workspace layout and (with dev) its
// launch shape.  Host only; returns SSM_OK or an error status.
int plan_ssd(int n_seqs, int n_tokens, int H, int P, int N, int G, int chunk, const DeviceInfo *dev,
             SsdLayout *out)
{
    SsdLayout L;
    L.chunk = chunk ? chunk : 128;
    if (!ssm::ssd_supported_chunk(L.chunk))
        return SSM_ERR_INVALID_ARG;
    if (P % 16 != 0 || P > ssm::ssd_max_head_dim())
        return SSM_ERR_UNSUPPORTED;
    const int Q = L.chunk;
    ssm::SsdGeom &g = L.g;
    g.n_pad = (N + 7) & ~7;
    g.bs_stride = bank_stride(g.n_pad, 8);
    g.xw_stride = bank_stride(P, 8);
    g.cs_stride = bank_stride(g.n_pad, 4);
    g.xs_stride = bank_stride(P, 4);
    // Shared memory of each kernel with `nb` tiles in flight (see ssd.cu).
    auto smem_state = [&](int nb) {
        return sizeof(float) * ((size_t)Q * g.bs_stride + (size_t)nb * Q * g.xw_stride + 2 * (size_t)Q);
    };
    const size_t out_buf = (size_t)Q * g.xs_stride + (size_t)P * g.cs_stride;
    auto smem_out = [&](int nb) {
        return sizeof(float) * ((size_t)Q * g.cs_stride + std::max((size_t)Q * g.cs_stride, out_buf) +
                                (nb == 2 ? out_buf : 0) + 4 * (size_t)Q);
    };
    g.state_buffers = g.out_buffers = 2;
    g.smem_state = smem_state(2);
    g.smem_out = smem_out(2);
    L.max_units = (long long)n_seqs + ((long long)n_tokens + Q - 1) / Q;
    if (L.max_units > INT_MAX || G > 65535)
        return SSM_ERR_UNSUPPORTED;
    const size_t slot = (size_t)H * P * N * sizeof(float);
    size_t off = 0;
    L.off_step = off;       off = align256(off + (size_t)n_tokens * H * sizeof(float));
    L.off_units = off;      off = align256(off + (size_t)L.max_units * sizeof(int2));
    L.off_n_units = off;    off = align256(off + sizeof(int));
    L.off_status = off;     off = align256(off + sizeof(int));
    L.off_unit_base = off;  off = align256(off + ((size_t)n_seqs + 1) * sizeof(int));
    L.off_decay = off;      off = align256(off + (size_t)L.max_units * H * sizeof(float));
    L.off_state = off;      off = align256(off + (size_t)L.max_units * slot);
    L.bytes = off;
    if (dev) {
        const size_t cap = (size_t)dev->smem_optin;
        // Blocks of `bytes` dynamic shared memory that fit one SM (1 KiB per
        // block is reserved by the runtime).
        auto per_sm = [&](size_t bytes) { return (size_t)dev->smem_per_sm / (bytes + 1024); };
        // One x tile at a time when two tiles do not fit, or when one tile lets
        // more blocks share an SM (their copies then overlap across blocks).
        if (g.smem_state > cap || per_sm(smem_state(1)) > per_sm(smem_state(2))) {
            g.state_buffers = 1;
            g.smem_state = smem_state(1);
        }
        if (g.smem_out > cap) {                 // one (x, S_in) tile pair at a time
            g.out_buffers = 1;
            g.smem_out = smem_out(1);
        }
        // The output kernel on tcgen05 where its tiles fit, else on mma.sync.
        const int tc_buffers = ssm::ssd_tc_buffers(Q, g.n_pad, P, cap);
        g.use_tc = tc_buffers > 0 ? 1 : 0;
        if (g.use_tc) {
            g.out_buffers = tc_buffers;
            g.smem_out = ssm::ssd_tc_smem_bytes(g.n_pad, P, tc_buffers);
            g.tmem_cols = ssm::ssd_tc_tmem_cols(g.n_pad, P);
        }
        if (g.smem_state > cap || g.smem_out > cap)
            return SSM_ERR_UNSUPPORTED;
        // Split a group's heads over blocks until there are about four
        // blocks per SM (C B^T is formed once per block).  The tcgen05 kernel
        // runs one block per SM, so it splits only until every SM has one:
        // each split forms C B^T and reads C and B once more.
        const int hpg = H / G;
        const long long blocks = L.max_units * G;
        const long long want = (g.use_tc ? 1LL : 4LL) * dev->sms;
        const int split = (int)std::min<long long>(hpg, std::max<long long>(1, (want + blocks - 1) / blocks));
        g.heads_per_cta = (hpg + split - 1) / split;
    }
    *out = L;
    return SSM_OK;
}

int ssd_impl(float *state, const float *x, const float *dt, const float *A, const float *B,
             const float *C, const float *D, float *y, const int32_t *seq_starts,
             const int32_t *seq_lens, const int32_t *resume, int n_seqs, int n_tokens, int H, int P,
             int N, int G, int chunk, const ssm_scan_options *opts, void *workspace, size_t workspace_bytes,
             void *stream_v)
{
    if (n_seqs < 0 || n_tokens < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || chunk < 0)
        return SSM_ERR_INVALID_ARG;
    if (H % G != 0)
        return SSM_ERR_INVALID_ARG;
    if (N % 4 != 0 || N > kMaxDState)
        return SSM_ERR_UNSUPPORTED;
    if ((long long)H * P > INT_MAX / 2)
        return SSM_ERR_UNSUPPORTED;
    SsdLayout L;
    int rc = plan_ssd(n_seqs, n_tokens, H, P, N, G, chunk, nullptr, &L);
    if (rc != SSM_OK)
        return rc;
    if (n_seqs == 0)
        return SSM_OK;
    if (!state || !A || !D || !seq_starts || !seq_lens || !resume)
        return SSM_ERR_INVALID_ARG;
    if (n_tokens > 0 && (!x || !dt || !B || !C || !y))
        return SSM_ERR_INVALID_ARG;
    if (!aligned(state, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(x, 16) || !aligned(y, 16))
        return SSM_ERR_INVALID_ARG;
    if (!aligned(dt, 4) || !aligned(A, 4) || !aligned(D, 4) || !aligned(seq_starts, 4) ||
        !aligned(seq_lens, 4) || !aligned(resume, 4))
        return SSM_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.bytes)
        return SSM_ERR_INVALID_ARG;
    ssm_scan_options o;
    rc = read_options(opts, &o);
    if (rc != SSM_OK)
        return rc;
    if (o.state_snapshots)
        return SSM_ERR_UNSUPPORTED;

    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != SSM_OK)
        return rc;
    rc = plan_ssd(n_seqs, n_tokens, H, P, N, G, chunk, &dev, &L);
    if (rc != SSM_OK)
        return rc;

    ssm::ScanArgs a;
    a.state = state; a.x = x; a.dt = dt; a.A = A; a.B = B; a.C = C; a.D = D; a.y = y;
    a.seq_starts = seq_starts; a.seq_lens = seq_lens; a.resume = resume;
    a.n_seqs = n_seqs; a.n_tokens = n_tokens; a.H = H; a.P = P; a.N = N; a.G = G;
    a.snaps = nullptr;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
    if (check_env()) {
        rc = check_metadata(a, stream);
        if (rc != SSM_OK)
            return rc;
    }
    ssm::LaunchTimer tm{o.launch_events, o.n_launch_events, 0, stream, false};
    if (dt_buffer_bytes(o, n_tokens, H) > 0) {
        float *step = reinterpret_cast<float *>(static_cast<char *>(workspace) + L.off_step);
        if (ssm::timed(&tm, [&] { return ssm::launch_dt_prep(a, o.dt_bias, o.dt_softplus, step, stream); }) !=
            cudaSuccess)
            return SSM_ERR_CUDA;
        a.dt = step;
    }

    char *ws = static_cast<char *>(workspace);
    ssm::SegmentPlan seg{};
    seg.units = reinterpret_cast<const int2 *>(ws + L.off_units);
    seg.n_units = reinterpret_cast<const int *>(ws + L.off_n_units);
    seg.unit_base = reinterpret_cast<const int *>(ws + L.off_unit_base);
    seg.seg_len = L.chunk;
    ssm::SsdPlan plan{};
    plan.units = seg.units;
    plan.n_units = seg.n_units;
    plan.unit_base = seg.unit_base;
    plan.chunk = L.chunk;
    plan.chunk_logdecay = reinterpret_cast<float *>(ws + L.off_decay);
    plan.chunk_state = reinterpret_cast<float *>(ws + L.off_state);
    plan.status = reinterpret_cast<int *>(ws + L.off_status);
    plan.fail_waits = fail_waits_env() ? 1 : 0;
    seg.status = plan.status;               // zeroed by the plan kernel
    const int mu = (int)L.max_units;
    // The chunk states on the tensor-core state pass where its shapes fit (TMA
    // descriptors encoded before any launch), else on the mma.sync kernel.
    ssm::SegStateMaps maps;
    const bool tc_states = ssm::segment_state_tc_supported(N, P, (size_t)dev.smem_optin) &&
                           ssm::segment_state_tc_maps(a, &maps);
    if (ssm::timed(&tm, [&] { return ssm::launch_segment_plan(a, seg, mu, stream); }) != cudaSuccess ||
        ssm::launch_ssd(a, plan, L.g, mu, stream, &tm, tc_states ? &maps : nullptr) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (o.gated_y && n_tokens > 0 &&
        ssm::timed(&tm, [&] {
            return ssm::launch_gated_norm(a, o.gate_z, o.norm_weight, o.norm_eps, o.gated_y, stream);
        }) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (tm.failed)
        return SSM_ERR_CUDA;
    if (check_env())                        // debug: report a bounded wait that gave up
        return read_status(plan.status, stream);
    return SSM_OK;
}

}  // namespace

extern "C" {

int ssm_scan(float *state_slots, const float *x, const float *dt, const float *A, const float *B,
             const float *C, const float *D, float *y, const int32_t *seq_starts,
             const int32_t *seq_lens, const int32_t *resume_flags, int n_seqs, int n_tokens,
             int n_heads, int head_dim, int d_state, int n_groups, void *stream)
{
    return scan_impl(state_slots, x, dt, A, B, C, D, y, seq_starts, seq_lens, resume_flags, n_seqs,
                     n_tokens, n_heads, head_dim, d_state, n_groups, nullptr, nullptr, nullptr, 0, stream);
}

int ssm_scan_tuned(float *state_slots, const float *x, const float *dt, const float *A,
                   const float *B, const float *C, const float *D, float *y,
                   const int32_t *seq_starts, const int32_t *seq_lens, const int32_t *resume_flags,
                   int n_seqs, int n_tokens, int n_heads, int head_dim, int d_state, int n_groups,
                   const ssm_scan_tuning *tuning, void *stream)
{
    return scan_impl(state_slots, x, dt, A, B, C, D, y, seq_starts, seq_lens, resume_flags, n_seqs,
                     n_tokens, n_heads, head_dim, d_state, n_groups, tuning, nullptr, nullptr, 0, stream);
}

int ssm_scan_ws(float *state_slots, const float *x, const float *dt, const float *A, const float *B,
                const float *C, const float *D, float *y, const int32_t *seq_starts,
                const int32_t *seq_lens, const int32_t *resume_flags, int n_seqs, int n_tokens,
                int n_heads, int head_dim, int d_state, int n_groups, const ssm_scan_tuning *tuning,
                void *workspace, size_t workspace_bytes, void *stream)
{
    return scan_impl(state_slots, x, dt, A, B, C, D, y, seq_starts, seq_lens, resume_flags, n_seqs,
                     n_tokens, n_heads, head_dim, d_state, n_groups, tuning, nullptr, workspace, workspace_bytes,
                     stream);
}

int ssm_scan_ex(float *state_slots, const float *x, const float *dt, const float *A, const float *B,
                const float *C, const float *D, float *y, const int32_t *seq_starts,
                const int32_t *seq_lens, const int32_t *resume_flags, int n_seqs, int n_tokens,
                int n_heads, int head_dim, int d_state, int n_groups, const ssm_scan_tuning *tuning,
                const ssm_scan_options *options, void *workspace, size_t workspace_bytes, void *stream)
{
    return scan_impl(state_slots, x, dt, A, B, C, D, y, seq_starts, seq_lens, resume_flags, n_seqs,
                     n_tokens, n_heads, head_dim, d_state, n_groups, tuning, options, workspace,
                     workspace_bytes, stream);
}

size_t ssm_scan_workspace_bytes(int n_seqs, int n_tokens, int n_heads, int head_dim, int d_state,
                                int n_groups, const ssm_scan_tuning *tuning)
{
    if (n_seqs <= 0 || n_tokens < 0 || n_heads <= 0 || head_dim <= 0 || d_state <= 0 || n_groups <= 0 ||
        n_heads % n_groups != 0 || d_state % 4 != 0 || d_state > kMaxDState)
        return 0;
    ssm_scan_tuning t;
    std::memset(&t, 0, sizeof t);
    if (tuning)
        t = *tuning;
    int path = t.path;
    if (path == SSM_PATH_AUTO)
        path = (n_tokens == n_seqs) ? SSM_PATH_DECODE : SSM_PATH_PREFILL;
    if (path != SSM_PATH_PREFILL)
        return 0;
    DeviceInfo dev;
    if (device_info(&dev) != SSM_OK)
        return 0;
    PrefillPlan pl;
    if (plan_prefill(t, true, n_seqs, n_tokens, n_heads, head_dim, d_state, n_groups, dev, true, &pl) != SSM_OK)
        return 0;
    return pl.seg_len > 0 ? pl.ws_bytes : 0;
}

int ssm_scan_ssd(float *state_slots, const float *x, const float *dt, const float *A, const float *B,
                 const float *C, const float *D, float *y, const int32_t *seq_starts,
                 const int32_t *seq_lens, const int32_t *resume_flags, int n_seqs, int n_tokens,
                 int n_heads, int head_dim, int d_state, int n_groups, int chunk,
                 const ssm_scan_options *options, void *workspace, size_t workspace_bytes, void *stream)
{
    return ssd_impl(state_slots, x, dt, A, B, C, D, y, seq_starts, seq_lens, resume_flags, n_seqs,
                    n_tokens, n_heads, head_dim, d_state, n_groups, chunk, options, workspace,
                    workspace_bytes, stream);
}

size_t ssm_scan_ssd_workspace_bytes(int n_seqs, int n_tokens, int n_heads, int head_dim, int d_state,
                                    int n_groups, int chunk)
{
    if (n_seqs <= 0 || n_tokens < 0 || n_heads <= 0 || head_dim <= 0 || d_state <= 0 || n_groups <= 0 ||
        chunk < 0 || n_heads % n_groups != 0 || d_state % 4 != 0 || d_state > kMaxDState)
        return 0;
    SsdLayout L;
    if (plan_ssd(n_seqs, n_tokens, n_heads, head_dim, d_state, n_groups, chunk, nullptr, &L) != SSM_OK)
        return 0;
    return L.bytes;
}

int ssm_conv1d(const float *x, const float *weight, const float *bias, float *conv_state, float *out,
               const int32_t *seq_starts, const int32_t *seq_lens, const int32_t *resume_flags, int n_seqs,
               int n_tokens, int channels, int kernel_size, float *snapshots, void *stream)
{
    if (n_seqs < 0 || n_tokens < 0 || channels <= 0 || kernel_size < 1 || kernel_size > kMaxConvKernel)
        return SSM_ERR_INVALID_ARG;
    if ((long long)n_tokens * channels > INT_MAX || (long long)n_seqs * channels > INT_MAX)
        return SSM_ERR_UNSUPPORTED;
    if (n_seqs == 0)
        return SSM_OK;
    if (!weight || !seq_starts || !seq_lens || !resume_flags || (kernel_size > 1 && !conv_state))
        return SSM_ERR_INVALID_ARG;
    if (n_tokens > 0 && (!x || !out))
        return SSM_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(weight, 4) || !aligned(bias, 4) || !aligned(conv_state, 4) ||
        !aligned(out, 4) || !aligned(snapshots, 4) || !aligned(seq_starts, 4) || !aligned(seq_lens, 4) ||
        !aligned(resume_flags, 4))
        return SSM_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (check_env()) {
        ssm::ScanArgs m{};
        m.seq_starts = seq_starts; m.seq_lens = seq_lens; m.n_seqs = n_seqs; m.n_tokens = n_tokens;
        const int rc = check_metadata(m, st);
        if (rc != SSM_OK)
            return rc;
    }
    if (ssm::launch_conv1d(x, weight, bias, conv_state, out, snapshots, seq_starts, seq_lens, resume_flags, n_seqs,
                           n_tokens, channels, kernel_size, st) != cudaSuccess)
        return SSM_ERR_CUDA;
    return SSM_OK;
}

size_t ssm_scan_ex_workspace_bytes(int n_seqs, int n_tokens, int n_heads, int head_dim, int d_state,
                                   int n_groups, const ssm_scan_tuning *tuning, const ssm_scan_options *options)
{
    ssm_scan_options o;
    if (n_tokens < 0 || n_heads <= 0 || read_options(options, &o) != SSM_OK)
        return 0;
    const size_t dtb = dt_buffer_bytes(o, n_tokens, n_heads);
    if (o.state_snapshots)                  // the decode kernel: no time segments
        return dtb;
    return dtb + ssm_scan_workspace_bytes(n_seqs, n_tokens, n_heads, head_dim, d_state, n_groups, tuning);
}

const char *ssm_status_string(int status)
{
    switch (status) {
    case SSM_OK: return "ok";
    case SSM_ERR_INVALID_ARG: return "invalid argument";
    case SSM_ERR_UNSUPPORTED: return "unsupported geometry";
    case SSM_ERR_CUDA: return "CUDA error";
    case SSM_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
    }
}

}  // extern "C"
