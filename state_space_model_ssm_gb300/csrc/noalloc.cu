// ssm_scan_static: the scan for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs
// where cudaMalloc is not allowed or not wanted (an allocator-free embedded
// runtime, a plugin whose host owns every device allocation, a latency path
// that must never enter the allocator).  This entry point gives them the
// time-segmented prefill of ssm_scan_ws with the library's own scratch: a
// fixed array in device global memory that exists from module load until the
// process exits.  A plan whose segment states would not fit it runs with
// longer segments, or none.  Nothing here calls cudaMalloc, cudaFree or any allocating
// library routine.
//
// The scratch is shared by every call in the process on a device and keeps
// whatever the last call left in it.  The segment pass writes every word it
// reads later in the same call (plan, segment states, decays), so nothing has
// to start at zero; calls whose GPU work overlaps (two streams, two threads)
// race on it and must be serialised by the caller.
#include <mutex>

#include "../../include/ssmscan.h"
#include "scan_common.cuh"

namespace {

constexpr int kMaxDevices = 64;

// The scratch itself.  In host code `g_static_scratch` names a host-side
// stand-in, not device memory: only its device address (below) may be passed
// to a kernel.
static __device__ __align__(256) unsigned char g_static_scratch[SSM_SCAN_STATIC_SCRATCH_BYTES];

void *g_scratch_addr[kMaxDevices];
bool g_scratch_ready[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
int static_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return SSM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ready[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
            return SSM_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ready[dev] = true;
    }
    *out = g_scratch_addr[dev];
    return SSM_OK;
}

}  // namespace

extern "C" int ssm_scan_static(float *state_slots, const float *x, const float *dt, const float *A,
                               const float *B, const float *C, const float *D, float *y,
                               const int32_t *seq_starts, const int32_t *seq_lens,
                               const int32_t *resume_flags, int n_seqs, int n_tokens, int n_heads,
                               int head_dim, int d_state, int n_groups, void *stream)
{
    // The automatic plan, or, when its segment states do not fit the scratch,
    // longer segments (fewer states: 1024 tokens, doubled until they fit), or
    // none once a segment would be as long as the longest sequence can be
    // (every other sequence holds at least one token): such a plan splits
    // nothing and would only add the segment passes.  Host arithmetic only;
    // nothing is launched before the plan fits.
    ssm_scan_tuning t = {};
    const size_t cap = (size_t)SSM_SCAN_STATIC_SCRATCH_BYTES;
    if (ssm_scan_workspace_bytes(n_seqs, n_tokens, n_heads, head_dim, d_state, n_groups, &t) > cap) {
        t.segment_tokens = -1;                        // no segments: no scratch
        const long long longest = (long long)n_tokens - (n_seqs > 1 ? n_seqs - 1 : 0);
        for (long long seg = 1024; seg < longest; seg *= 2) {
            ssm_scan_tuning c = {};
            c.segment_tokens = (int)seg;
            const size_t need = ssm_scan_workspace_bytes(n_seqs, n_tokens, n_heads, head_dim, d_state,
                                                         n_groups, &c);
            if (need > 0 && need <= cap) {
                t = c;
                break;
            }
        }
    }
    // The scratch address is the current device's: the stream must belong to it.
    if (stream) {
        int cur = 0, sdev = 0;
        if (cudaGetDevice(&cur) != cudaSuccess ||
            cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &sdev) != cudaSuccess)
            return SSM_ERR_CUDA;
        if (cur != sdev)
            return SSM_ERR_INVALID_ARG;
    }
    void *scratch = nullptr;
    const int rc = static_scratch(&scratch);
    if (rc != SSM_OK)
        return rc;
    return ssm_scan_ws(state_slots, x, dt, A, B, C, D, y, seq_starts, seq_lens, resume_flags, n_seqs,
                       n_tokens, n_heads, head_dim, d_state, n_groups, &t, scratch, cap, stream);
}
