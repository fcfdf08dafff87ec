// Time segments for long sequences (sm_103a).
//
// A single long sequence leaves most of the GPU idle: its state has H*P rows,
// and the scan is serial in time.  The recurrence is linear in the state, so a
// sequence can be cut into time segments k = 0..K-1 of seg_len tokens:
//
//   state pass   segment k < K-1 runs from zero (segment 0 from the slot or
//                zero) and leaves its final state L_k and its decay
//                prod_t exp(dt_t A) = d_k (per head), in parallel over k;
//   combine      the incoming state of segment k+1 is
//                S_in[1] = L_0,  S_in[k+1] = d_k S_in[k] + L_k;
//   full pass    every segment runs the scan with y from S_in[k], in
//                parallel over k; the last one writes the slot.
//
// The combine step is the recurrence itself applied to whole segments (the
// decay of a segment is the product of its tokens' decays), so the result is
// the scan of "The llama journey", Day 14, with float association changed.
//
// This file holds the plan kernel (which (sequence, segment) each work unit
// is) and the combine kernel.  The state and full passes are modes of the
// prefill kernel in prefill_scaled.cu.
#include "scan_common.cuh"

namespace ssm {

namespace {

// One block: segment counts per sequence, their prefix sum (unit_base) and the
// unit list.  Writes stay inside max_units even for inconsistent metadata.
__global__ void __launch_bounds__(1024)
segment_plan_kernel(const int32_t *seq_lens, int n_seqs, int seg_len, int max_units,
                    int2 *units, int *unit_base, int *n_units, int *status)
{
    griddep_entry();
    __shared__ int warp_tot[32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    if (tid == 0)
        carry = 0;
    __syncthreads();
    for (int base = 0; base < n_seqs; base += blockDim.x) {
        const int i = base + tid;
        int cnt = 0;
        if (i < n_seqs) {
            const int L = max(0, seq_lens[i]);
            cnt = max(1, (int)(((long long)L + seg_len - 1) / seg_len));
        }
        int incl = cnt;                               // warp inclusive scan
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(kFullMask, incl, off);
            if (lane >= off)
                incl += v;
        }
        if (lane == 31)
            warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {                              // scan of the warp totals
            int wt = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(kFullMask, wt, off);
                if (lane >= off)
                    wt += v;
            }
            if (lane < nw)
                warp_tot[lane] = wt;                  // inclusive
        }
        __syncthreads();
        const int excl = carry + (warp ? warp_tot[warp - 1] : 0) + incl - cnt;
        if (i < n_seqs)
            unit_base[i] = excl;
        __syncthreads();
        if (tid == blockDim.x - 1)
            carry = excl + cnt;
        __syncthreads();
    }
    if (tid == 0) {
        unit_base[n_seqs] = carry;
        *n_units = min(carry, max_units);
        if (status)
            *status = 0;
    }
    __syncthreads();
    for (int i = tid; i < n_seqs; i += blockDim.x) {
        const int b = unit_base[i], e = unit_base[i + 1];
        for (int k = 0; k < e - b && b + k < max_units; ++k)
            units[b + k] = make_int2(i, k);
    }
}

// S_in[k+1] = d_k S_in[k] + L_k for k >= 1, in place over the units' scratch
// (unit b+k of sequence i ends up holding S_in[k+1]; unit b already holds
// L_0 = S_in[1]).  One thread per float4 of a state slot.  The chain is serial
// in k but its loads are not: each thread reads the L_k and d_k of up to
// kCombineBatch segments before it runs them through the chain, so a
// sequence's segments wait on one memory latency per batch, not one each.
constexpr int kCombineBatch = 8;

__global__ void __launch_bounds__(256)
segment_combine_kernel(const ScanArgs a, const SegmentPlan plan, int max_units)
{
    griddep_entry();
    const int N4 = a.N >> 2;
    const long long slot4 = (long long)a.H * a.P * N4;         // float4 per state slot
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= slot4 || call_failed(plan.status))      // no valid segment states to combine
        return;
    const int head = (int)((e / N4) / a.P);
    float4 *__restrict__ st = reinterpret_cast<float4 *>(plan.seg_state);
    const float *__restrict__ dec = plan.seg_decay;
    for (int seq = blockIdx.y; seq < a.n_seqs; seq += gridDim.y) {
        const int b = plan.unit_base[seq];
        const int nseg = plan.unit_base[seq + 1] - b;
        if (nseg <= 2 || b + nseg > max_units)
            continue;
        float4 S = st[(long long)b * slot4 + e];
        for (int k0 = 1; k0 <= nseg - 2; k0 += kCombineBatch) {
            float4 L[kCombineBatch];
            float d[kCombineBatch];
#pragma unroll
            for (int i = 0; i < kCombineBatch; ++i) {
                const int k = k0 + i;
                if (k <= nseg - 2) {
                    L[i] = st[(long long)(b + k) * slot4 + e];
                    d[i] = dec[(long long)(b + k) * a.H + head];
                }
            }
#pragma unroll
            for (int i = 0; i < kCombineBatch; ++i) {
                const int k = k0 + i;
                if (k <= nseg - 2) {
                    S = make_float4(fmaf(d[i], S.x, L[i].x), fmaf(d[i], S.y, L[i].y), fmaf(d[i], S.z, L[i].z),
                                    fmaf(d[i], S.w, L[i].w));
                    st[(long long)(b + k) * slot4 + e] = S;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_segment_plan(const ScanArgs &a, const SegmentPlan &plan, int max_units, cudaStream_t stream)
{
    return launch_pdl(segment_plan_kernel, dim3(1), dim3(1024), 0, stream, a.seq_lens, a.n_seqs, plan.seg_len,
                      max_units, const_cast<int2 *>(plan.units), const_cast<int *>(plan.unit_base),
                      const_cast<int *>(plan.n_units), plan.status);
}

cudaError_t launch_segment_combine(const ScanArgs &a, const SegmentPlan &plan, int max_units, cudaStream_t stream)
{
    const long long slot4 = (long long)a.H * a.P * (a.N >> 2);
    const dim3 grid((unsigned)((slot4 + 255) / 256), (unsigned)(a.n_seqs < 65535 ? a.n_seqs : 65535));
    return launch_pdl(segment_combine_kernel, grid, dim3(256), 0, stream, a, plan, max_units);
}

}  // namespace ssm
