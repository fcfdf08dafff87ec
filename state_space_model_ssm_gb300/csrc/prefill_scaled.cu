// Prefill kernel of the Mamba2 scan with a decay-rescaled state (sm_103a).
//
// Work mapping and register layout follow prefill.cu (a block owns one
// sequence and a run of rows inside one group; a row's state lives in the
// registers of LANES lanes as interleaved float4 chunks), with two changes.
//
// 1. Rescaled state.  The registers hold U = S / Lambda, where Lambda is the
//    decay accumulated since an anchor token.  Because Lambda_t = dA_t Lambda_{t-1},
//
//        S_t = dA_t S_{t-1} + dt_t x_t B_t  <=>  U_t = U_{t-1} + (dt_t / Lambda_t) x_t B_t
//        y_t = S_t . C_t + D x_t            =    Lambda_t (U_t . C_t) + D x_t
//
//    so a state element costs one multiply-add for the update and one for the
//    readout (the decay multiply of the direct form disappears); both run as
//    packed fp32x2 FMAs.  Lambda must stay inside the fp32 range, so the
//    reference is re-anchored at the first token of every chunk and whenever the
//    chunk's running log-decay sum(dt*A) crosses a multiple of kAnchorSpan: U is
//    multiplied by the decay since the previous anchor and Lambda restarts at 1
//    (between anchors 1/Lambda < e^40).  At the end of each chunk U is scaled
//    back to S, so every chunk's coefficients are independent.
//
// 2. Staging.  Each chunk's B, C and x go into shared-memory slots with
//    cp.async ahead of use, and its coefficients are formed with lane = token
//    (a warp prefix sum places the anchors, a segmented prefix product of
//    dA = exp(dt*A) gives Lambda, ~1 ulp per factor).  Blocks of exactly four
//    consumer warps of the default shapes stage their own chunks
//    ("self-staged", three blocks per SM: three warps on every SM
//    sub-partition): every thread copies its share, the warps take turns
//    forming the next chunk's coefficients, and the block meets at one
//    barrier per chunk.  Other shapes add one producer warp that stages two
//    chunks ahead into three slots and meets the consumers at named barriers
//    (bar.arrive / bar.sync, no spin loop): FULL[s] when slot s holds a staged
//    chunk, EMPTY[s] when the consumers are done with it.  Consumers run the
//    token loop: per token U += alpha B, each lane's part of U . C, a shuffle
//    reduction over the row's lanes and the y store.  A lane holds RPT rows so
//    that each B/C value read from shared memory (128-bit reads cost four
//    wavefronts even when broadcast) feeds RPT rows.
//
// 3. Token runs.  Consumers take a chunk's tokens in runs of eight with no
//    anchor after the run's first token (the rescale of an anchor at the first
//    token happens before the run), compiled as straight-line code so that the
//    next token's shared-memory reads overlap the current token's arithmetic
//    and reduction; tokens outside such runs go one at a time.  The default
//    shape gives a lane 16 elements of each of 4 rows (8 lanes per row at
//    d_state 128): 64 state registers, B/C reads shared by 4 rows and a
//    three-step shuffle reduction.  Where y goes through a tile, the row sums
//    of two tokens are reduced together (8 values over the row's 8 lanes,
//    one (token, row) sum per lane); otherwise every lane ends the reduction
//    holding its row's full sum and all lanes of a row store y (the same
//    value), with no divergent branch.
//
// 4. Output through tiles (EPI 1, 2, 4, 5).  The consumers leave each chunk's
//    y in a shared-memory tile instead of storing it; the producer writes it
//    out once the consumers release the chunk (EPI 1), or, self-staged, all
//    warps write chunk c-1's tile after chunk c's barrier (EPI 5).  With
//    EPI 2 and 4 (a block's rows are exactly one head) the kernel also applies
//    Mamba2's output gate RMSNorm(y) * w * silu(z) per (token, head) row
//    (kernel 3 of "ssm_gated_delta.cu"): z is staged beside the chunk, and the
//    consumer warps share the row norms and the gated values (eight lanes per
//    token), so the gated output needs no second pass over y.  (One producer
//    warp alone would hold up the whole block with that work.)
//
// The rescaling is an algebraic identity of the recurrence defined by "The
// llama journey", Day 14 (decay exp(dt*A), input dt*x*B, y from the updated
// state); only the rounding differs from the direct form.
#include "scan_common.cuh"

namespace ssm {

namespace {

constexpr float kAnchorSpan = 40.f;
constexpr int kSlots = 3;         // staging slots: two chunks in flight while one is consumed
// Self-staged slots: 3 (two chunks ahead) for the plain output; 2 (one chunk
// ahead, which a chunk's work covers many times) for the gated output, whose
// z tiles then fit twice and need no second barrier per chunk.
__host__ __device__ constexpr int self_slots(int epi) { return epi == 4 ? 2 : 3; }
constexpr int kBarFull = 1;       // named barriers kBarFull + s: slot s staged
constexpr int kBarEmpty = 4;      // named barriers kBarEmpty + s: slot s consumed
constexpr int kBarConsumers = 7;  // the consumer warps alone (the gated output)

__device__ __forceinline__ void bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void bar_arrive(int id, int nthreads)
{
    asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

struct ScaledSmem {
    float *base;
    int cb, cx, cc, cm; // floats per buffer: B (= C), x, coefficients (float4 per token and
                        // head), anchor masks (one word per head)
    int cg;             // output through the producer: the y tile (cx floats) and with the
                        // gated output the z tile (cx more), else 0
    // slot s: [B | C | x | coefficients | anchor masks | y | z], each 16-byte aligned
    __device__ __forceinline__ float *slot(int s) const { return base + s * (2 * cb + cx + cc + cm + cg); }
    __device__ __forceinline__ float *B(int s) const { return slot(s); }
    __device__ __forceinline__ float *C(int s) const { return slot(s) + cb; }
    __device__ __forceinline__ float *X(int s) const { return slot(s) + 2 * cb; }
    __device__ __forceinline__ float4 *Coef(int s) const
    {
        return reinterpret_cast<float4 *>(slot(s) + 2 * cb + cx);
    }
    __device__ __forceinline__ unsigned *Mask(int s) const
    {
        return reinterpret_cast<unsigned *>(slot(s) + 2 * cb + cx + cc);
    }
    __device__ __forceinline__ float *Ytile(int s) const { return slot(s) + 2 * cb + cx + cc + cm; }
    __device__ __forceinline__ float *Ztile(int s) const { return slot(s) + 2 * cb + 2 * cx + cc + cm; }
    // after the NS slots (kSlots, or self_slots(EPI) when self-staged)
    template <int NS>
    __device__ __forceinline__ float *Dec() const { return base + NS * (2 * cb + cx + cc + cm + cg); }
    // self-staged output (EPI 5, 4): two y tiles and (EPI 4) two z tiles after the
    // decay area, cx floats each; chunk c in tile c % 2
    template <int NS>
    __device__ __forceinline__ float *SelfY(int i) const { return Dec<NS>() + cm + i * cx; }
    template <int NS>
    __device__ __forceinline__ float *SelfZ(int i) const { return Dec<NS>() + cm + (2 + i) * cx; }
};

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// A shared-memory store the compiler may move other shared-memory reads across
// (no memory clobber): the y tile is written only here and read only by the
// producer after the chunk's EMPTY barrier, which orders it.  A plain store
// would pin every later operand read of the token run behind it.
__device__ __forceinline__ void st_shared_unordered(float *p, float v)
{
    asm volatile("st.shared.f32 [%0], %1;\n" ::"r"(static_cast<unsigned>(__cvta_generic_to_shared(p))), "f"(v));
}

// R consecutive floats from shared memory (16-byte aligned when R = 4, 8 bytes when R = 2).
template <int R>
__device__ __forceinline__ void load_rows(float (&v)[R], const float *p)
{
    if constexpr (R % 4 == 0) {
#pragma unroll
        for (int i = 0; i < R; i += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(p + i);
            v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
        }
    } else if constexpr (R == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        v[0] = t.x; v[1] = t.y;
    } else {
#pragma unroll
        for (int i = 0; i < R; ++i)
            v[i] = p[i];
    }
}

// Coefficients of one head for one chunk of n <= 32 tokens; lane = token.
// out[t * stride] = {dt_t / Lambda_t, Lambda_t, r_t, 0}; *mask = bit t set for
// every anchor token t.
__device__ __forceinline__ float chunk_coefficients(float dt, float A, int n, int lane,
                                                    float4 *out, int stride, unsigned *mask)
{
    const bool live = lane < n;
    const float a = live ? dt * A : 0.f;
    float L = a;                                   // inclusive prefix sum of dt*A
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float v = __shfl_up_sync(kFullMask, L, off);
        if (lane >= off)
            L += v;
    }
    const float bucket = floorf(L * (1.f / kAnchorSpan));
    const float prev_bucket = __shfl_up_sync(kFullMask, bucket, 1);
    const bool anchor = (lane == 0) || (bucket != prev_bucket);
    const float dA = expf(a);
    // segmented inclusive prefix product; an anchor token starts a segment at 1
    float lam = anchor ? 1.f : dA;
    int seg = anchor ? 1 : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float lo = __shfl_up_sync(kFullMask, lam, off);
        const int so = __shfl_up_sync(kFullMask, seg, off);
        if (lane >= off && !seg) {
            lam *= lo;
            seg = so;
        }
    }
    const float lam_prev = __shfl_up_sync(kFullMask, lam, 1);
    const float r = anchor ? (lane == 0 ? dA : lam_prev * dA) : 1.f;
    if (live)
        out[lane * stride] = make_float4(dt / lam, lam, r, 0.f);
    const unsigned m = __ballot_sync(kFullMask, anchor && live);
    if (lane == 0)
        *mask = m;
    // total decay of the chunk, prod dA (lanes past n contribute exp(0) = 1)
    float prod = dA;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        prod *= __shfl_xor_sync(kFullMask, prod, off);
    return prod;
}

}  // namespace

size_t prefill_scaled_smem_bytes(const PrefillGeom &g, int N, int lanes, int epi)
{
    const size_t cx = ((size_t)g.chunk * g.rows_per_cta + 3) & ~(size_t)3;
    const size_t cm = ((size_t)g.heads_cap + 3) & ~(size_t)3;
    const size_t per_slot = (size_t)g.chunk * (2 * (size_t)N + 4 * (size_t)g.heads_cap) + cx + cm +
                            (epi == 1 || epi == 2 ? (size_t)epi * cx : 0);
    (void)lanes;
    // self-staged (epi 4, 5): self_slots(epi) slots, then two y tiles and (epi 4)
    // two z tiles after the decay area
    const bool self = epi == 4 || epi == 5;
    return ((self ? self_slots(epi) : kSlots) * per_slot + cm + (epi == 4 ? 4 * cx : epi == 5 ? 2 * cx : 0)) *
           sizeof(float);
}

// MODE kScanFull: the scan with y.  MODE kScanStateOnly: one time segment's
// state from zero (no C, no y), for the segment pass of long sequences.
// EPI (kScanFull only): 0 the consumers store y; 1 y through a shared-memory
// tile, stored by the producer; 2 as 1 and the gated RMSNorm output (a block's
// rows are exactly one head); without a producer warp (the consumers stage
// the chunks): 5 y through tiles written out by all warps one chunk later, 4
// as 5 with the gated output (z through a tile too).  (3, the self-staged
// form with the consumers' own y stores, measured slower than 5 and is not
// launched.)  The tile variants
// (prefill_scaled_tile_kernel) run blocks of at most kTileThreads (four
// consumer warps and the producer) and keep two blocks per SM; the
// self-staged ones (prefill_scaled_self_kernel) exactly kSelfThreads, three
// per SM.
constexpr int kTileThreads = 160;
constexpr int kSelfThreads = 128;      // self-staged (EPI 4, 5): exactly four consumer warps, no producer

template <int LANES, int VPL, int RPT, bool EXACT, int MODE, int EPI>
__device__ __forceinline__ void prefill_scaled_body(const ScanArgs &a, const PrefillGeom &geo,
                                                    const SegmentPlan &plan, const GatedOut &gt)
{
    constexpr bool kFull = (MODE == kScanFull);
    // EPI 4 and 5 (and 3): self-staged (no producer warp); 4 with the gated
    // output, 5 with y through tiles
    constexpr bool SELF = EPI == 3 || EPI == 4 || EPI == 5;
    constexpr bool TILE = EPI == 1 || EPI == 2 || EPI == 4 || EPI == 5, GATED = EPI == 2 || EPI == 4;
    static_assert(kFull || EPI == 0, "the output tile and the self-staged form need y");
    extern __shared__ __align__(16) float smem[];
    const int N = a.N, N4 = a.N >> 2, P = a.P, H = a.H;
    const long long HP = (long long)H * P;
    ScaledSmem sm;
    sm.base = smem;
    sm.cb = geo.chunk * N;
    sm.cx = (geo.chunk * geo.rows_per_cta + 3) & ~3;     // keeps the float4 coefficients 16-byte aligned
    sm.cc = geo.chunk * geo.heads_cap * 4;
    sm.cm = (geo.heads_cap + 3) & ~3;                    // keeps the next slot 16-byte aligned
    sm.cg = (EPI == 1 || EPI == 2) ? EPI * sm.cx : 0;
    constexpr int NS = SELF ? self_slots(EPI) : kSlots;

    // ---- A1 work mapping: (work unit, group, run of rows) ----
    // A work unit is a whole sequence, or with a segment plan one time segment
    // (seq, seg) of it: tokens [seg * seg_len, (seg + 1) * seg_len).
    const int ctas_per_unit = a.G * geo.runs_per_group;
    const int unit = blockIdx.x / ctas_per_unit;
    const int rem = blockIdx.x - unit * ctas_per_unit;
    const int grp = rem / geo.runs_per_group;
    const int run = rem - grp * geo.runs_per_group;
    const int r0 = grp * geo.rows_per_group + run * geo.rows_per_cta;
    const int nrows = min(geo.rows_per_cta, geo.rows_per_group - run * geo.rows_per_cta);
    const int h0 = r0 / P;
    const int nheads = (r0 + nrows - 1) / P - h0 + 1;

    int seq = unit, seg = 0, nseg = 1;
    if (plan.units) {
        if (unit >= *plan.n_units)
            return;                                      // whole block: beyond the plan
        const int2 us = plan.units[unit];
        seq = us.x;
        seg = us.y;
    }
    const int seq_len = a.seq_lens[seq];
    int seg_off = 0, len = seq_len;
    if (plan.units) {
        nseg = max(1, (seq_len + plan.seg_len - 1) / plan.seg_len);
        seg_off = seg * plan.seg_len;
        len = min(plan.seg_len, seq_len - seg_off);
    }
    if (!kFull && seg == nseg - 1)
        return;                                          // the last segment needs no state pass
    const int tok_start = a.seq_starts[seq] + seg_off;
    const bool resume = a.resume[seq] != 0;
    const bool from_slot = (seg == 0) && resume;                 // initial state from the slot
    const bool from_plan = kFull && seg > 0;                     // incoming state of the segment
    const bool to_slot = kFull && seg == nseg - 1;               // final state to the slot
    const int n_chunks = (len + geo.chunk - 1) / geo.chunk;

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int producer = SELF ? -1 : (nthr >> 5) - 1;   // the last warp (none when self-staged)
    if (kFull && plan.units && call_failed(plan.status)) {
        // The state pass gave up a bounded wait, so the segments' incoming
        // states are not valid: y becomes NaN and the slot keeps its contents.
        poison_y(a.y, HP, tok_start, len, r0, nrows, tid, nthr);
        if (GATED)
            poison_y(gt.out, HP, tok_start, len, r0, nrows, tid, nthr);
        return;
    }

    // Staging of a chunk (A3) and its coefficients (A4): by the producer warp
    // (sid = lane of 32), or by all the block's threads when it has no
    // producer (sid = tid of nthr); the coefficients by one warp either way.
    const int sid = SELF ? tid : lane;
    constexpr int scount = SELF ? kSelfThreads : 32;      // the block size when self-staged
    const float *Bg = a.B + (long long)grp * N;
    const float *Cg = a.C + (long long)grp * N;
    const long long tokN = (long long)a.G * N;
    // A3: stage B, C and x of chunk c0 into slot b (cp.async by the staging
    // threads, one commit group per chunk)
    float *seg_decay = sm.Dec<NS>();     // state pass: running decay of the segment per head
    // Walk over (token, column) items in steps of scount without divisions:
    // start at (sid / width, sid % width), step (scount / width, scount % width).
    const int bt0 = sid / N4, bv0 = sid - bt0 * N4, bdt = scount / N4, bdv = scount - bdt * N4;
    // x moves in 16-byte pieces when the block's rows start on 16 bytes in
    // global and shared memory, else in 4-byte pieces; xw pieces per token.
    const bool x16 = ((r0 | nrows | geo.rows_per_cta) & 3) == 0 && (HP & 3) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.x) & 15) == 0;
    const int xw = x16 ? nrows >> 2 : nrows;
    const int xt0 = sid / xw, xv0 = sid - xt0 * xw, xdt = scount / xw, xdv = scount - xdt * xw;
    auto stage = [&](int c0, int b) {
        const int t0 = c0 * geo.chunk;
        const int cnt = min(geo.chunk, len - t0);
        const long long tok0 = (long long)tok_start + t0;
        float *sB = sm.B(b), *sC = sm.C(b), *sX = sm.X(b);
        if ((EXACT ? LANES * VPL : N4) % 32 == 0) {   // known at compile time for the exact shapes
            // thread sid: float4 columns sid % 32, + 32, ... of tokens sid / 32, + scount / 32, ...
            const int col = sid & 31, tstep = scount >> 5;
            const float *gB = Bg + (tok0 + (sid >> 5)) * tokN + 4 * col;
            const float *gC = Cg + (tok0 + (sid >> 5)) * tokN + 4 * col;
            float *dB = sB + (sid >> 5) * N + 4 * col, *dC = sC + (sid >> 5) * N + 4 * col;
            for (int t = sid >> 5; t < cnt; t += tstep) {
                for (int v = 0; v < N4; v += 32) {
                    cp_async16(dB + 4 * v, gB + 4 * v);
                    if (kFull)
                        cp_async16(dC + 4 * v, gC + 4 * v);
                }
                gB += tstep * tokN;
                gC += tstep * tokN;
                dB += tstep * N;
                dC += tstep * N;
            }
        } else {
            for (int t = bt0, v = bv0; t < cnt;) {
                const long long goff = (tok0 + t) * tokN + 4 * v;
                cp_async16(sB + t * N + 4 * v, Bg + goff);
                if (kFull)
                    cp_async16(sC + t * N + 4 * v, Cg + goff);
                t += bdt;
                v += bdv;
                if (v >= N4) { v -= N4; ++t; }
            }
        }
        const float *gx = a.x + tok0 * HP + r0;
        constexpr bool kZ = EPI == 2;                // z staged with the chunk (self-staged: see stage_z)
        const float *gz = kZ ? gt.z + tok0 * HP + r0 : nullptr;
        float *sZ = kZ ? sm.Ztile(b) : nullptr;
        if (x16) {
            for (int t = xt0, r = xv0; t < cnt;) {
                cp_async16(sX + t * geo.rows_per_cta + 4 * r, gx + t * HP + 4 * r);
                if (kZ)                 // z: the same layout as x (16-byte aligned: checked by the host)
                    cp_async16(sZ + t * geo.rows_per_cta + 4 * r, gz + t * HP + 4 * r);
                t += xdt;
                r += xdv;
                if (r >= xw) { r -= xw; ++t; }
            }
        } else {
            for (int t = xt0, r = xv0; t < cnt;) {
                cp_async4(sX + t * geo.rows_per_cta + r, gx + t * HP + r);
                if (kZ)
                    cp_async4(sZ + t * geo.rows_per_cta + r, gz + t * HP + r);
                t += xdt;
                r += xdv;
                if (r >= xw) { r -= xw; ++t; }
            }
        }
        if (SELF && warp == c0 % (kSelfThreads / 32)) {
            // self-staged: the warp that will form this chunk's coefficients copies
            // its dt (lane = token) into the unused fourth word of each slot
            float4 *cf = sm.Coef(b);
            for (int hh = 0; hh < nheads; ++hh)
                if (lane < cnt)
                    cp_async4(&cf[lane * geo.heads_cap + hh].w, a.dt + (tok0 + lane) * H + h0 + hh);
        }
        cp_async_commit();
    };
    // Self-staged gated output: z of chunk c0 into the z tile (the x layout),
    // one commit group of its own.
    auto stage_z = [&](int c0) {
        const int t0 = c0 * geo.chunk;
        const int cnt = min(geo.chunk, len - t0);
        const float *gz = gt.z + ((long long)tok_start + t0) * HP + r0;
        float *sZ = sm.SelfZ<NS>(c0 & 1);
        for (int t = xt0, r = xv0; t < cnt;) {      // 16-byte pieces (checked by the host)
            cp_async16(sZ + t * geo.rows_per_cta + 4 * r, gz + t * HP + 4 * r);
            t += xdt;
            r += xdv;
            if (r >= xw) { r -= xw; ++t; }
        }
        cp_async_commit();
    };
    // A4: dt of chunk c0 (lane = token) for the first kDtHeads heads, read two
    // chunks before its coefficients are needed.
    constexpr int kDtHeads = 4;
    auto load_dt = [&](int c0, float (&d)[kDtHeads]) {
        const int t0 = c0 * geo.chunk;
        const int cnt = min(geo.chunk, len - t0);
#pragma unroll
        for (int q = 0; q < kDtHeads; ++q)
            d[q] = (q < nheads && lane < cnt) ? a.dt[((long long)tok_start + t0 + lane) * H + h0 + q] : 0.f;
    };
    auto coefficients = [&](int c0, int b, const float (&d)[kDtHeads]) {
        const int t0 = c0 * geo.chunk;
        const int cnt = min(geo.chunk, len - t0);
        for (int hh = 0; hh < nheads; ++hh) {
            float dtv = d[0];
#pragma unroll
            for (int q = 1; q < kDtHeads; ++q)
                if (hh == q) dtv = d[q];
            if (hh >= kDtHeads)
                dtv = lane < cnt ? a.dt[((long long)tok_start + t0 + lane) * H + h0 + hh] : 0.f;
            if (SELF)                                 // staged with the chunk (see stage)
                dtv = lane < cnt ? sm.Coef(b)[lane * geo.heads_cap + hh].w : 0.f;
            const float dec = chunk_coefficients(dtv, a.A[h0 + hh], cnt, lane, sm.Coef(b) + hh,
                                                 geo.heads_cap, sm.Mask(b) + hh);
            if (!kFull && lane == 0)
                seg_decay[hh] = (c0 == 0 ? 1.f : seg_decay[hh]) * dec;
        }
    };
    if (warp == producer) {
        // ================= producer warp =================
        // Output of chunk c0 (slot b), after the consumers are done with it: the
        // y tile to global memory (128-bit stores where the rows allow).
        const bool y16 = ((r0 | nrows | geo.rows_per_cta) & 3) == 0 && (HP & 3) == 0 &&
                         (reinterpret_cast<uintptr_t>(a.y) & 15) == 0;
        // (token, piece) walk of the y write-out: yw pieces (16 or 4 bytes) per token
        const int yw = y16 ? nrows >> 2 : nrows;
        const int yt0 = lane / yw, yv0 = lane - yt0 * yw, ydt = 32 / yw, ydv = 32 - ydt * yw;
        auto epilogue = [&](int c0, int b) {
            const int t0 = c0 * geo.chunk;
            const int cnt = min(geo.chunk, len - t0);
            const float *Y = sm.Ytile(b);
            const int xs = geo.rows_per_cta;
            float *yg = a.y + ((long long)tok_start + t0) * HP + r0;
            if (y16) {
                for (int t = yt0, r = yv0; t < cnt;) {
                    *reinterpret_cast<float4 *>(yg + t * HP + 4 * r) =
                        *reinterpret_cast<const float4 *>(Y + t * xs + 4 * r);
                    t += ydt;
                    r += ydv;
                    if (r >= yw) { r -= yw; ++t; }
                }
            } else {
                for (int t = yt0, r = yv0; t < cnt;) {
                    yg[t * HP + r] = Y[t * xs + r];
                    t += ydt;
                    r += ydv;
                    if (r >= yw) { r -= yw; ++t; }
                }
            }
            __syncwarp();               // every read of the tile done before the slot is restaged
        };
        // Staging runs two chunks ahead: chunks k and k+1 are in flight while the
        // consumers work on chunk k-1.  A slot is refilled only after EMPTY says
        // the consumers are done with the chunk three back.  With the output
        // tile the consumers release every chunk and the producer writes out
        // chunk k-1 before it restages that slot.
        float dt0[kDtHeads], dt1[kDtHeads], dt2[kDtHeads];
        if (n_chunks > 0) {
            stage(0, 0);
            load_dt(0, dt0);
        }
        if (n_chunks > 1) {
            stage(1, 1);
            load_dt(1, dt1);
        }
        for (int k = 0; k < n_chunks; ++k) {
            const int s = k % kSlots;
            if (k + 2 < n_chunks)
                load_dt(k + 2, dt2);
            coefficients(k, s, dt0);
            if (k + 1 < n_chunks)
                cp_async_wait<1>();          // chunk k landed, chunk k+1 may still fly
            else
                cp_async_wait<0>();
            __syncwarp();
            bar_arrive(kBarFull + s, nthr);
            if (TILE && k >= 1) {             // chunk k-1 (slot (k+2) % 3) consumed: its output
                bar_sync(kBarEmpty + (k + 2) % kSlots, nthr);
                epilogue(k - 1, (k + 2) % kSlots);
            }
            if (k + 2 < n_chunks) {
                const int s2 = (k + 2) % kSlots;
                if (!TILE && k >= 1)          // chunk k-1 used slot s2
                    bar_sync(kBarEmpty + s2, nthr);
                stage(k + 2, s2);
            }
#pragma unroll
            for (int q = 0; q < kDtHeads; ++q) {
                dt0[q] = dt1[q];
                dt1[q] = dt2[q];
            }
        }
        if (TILE && n_chunks > 0) {           // the last chunk's output
            bar_sync(kBarEmpty + (n_chunks - 1) % kSlots, nthr);
            epilogue(n_chunks - 1, (n_chunks - 1) % kSlots);
        }
        if (!kFull && lane == 0) {
            // the segment's decay per head, written by the block holding the head's first row
            for (int hh = 0; hh < nheads; ++hh)
                if ((h0 + hh) * P >= r0)
                    plan.seg_decay[(long long)unit * H + h0 + hh] = n_chunks > 0 ? seg_decay[hh] : 1.f;
        }
        return;
    }

    // ================= consumer warps =================
    const int j = lane % LANES;
    // A lane group (LANES lanes) holds RPT consecutive rows.  RPT divides P and
    // the rows per block (checked by the host), so the group's rows are all
    // valid or all padding, and they share one head.
    const int row_raw = (warp * (32 / LANES) + lane / LANES) * RPT;
    const bool rvalid = row_raw < nrows;
    const int rl = rvalid ? row_raw : nrows - RPT;          // first of the RPT rows
    const int hl = (r0 + rl) / P - h0;
    const float Dv = __ldg(a.D + h0 + hl);
    const int yq = reduced_row<LANES, RPT>(j);               // row of this lane's reduced sum
    // Pairwise reduction (two tokens of a run at once) where 2 RPT <= LANES
    // and y goes through a tile (measured slower with the consumers' own
    // global stores): this lane's sum is row q2 of the pair's token t2.
    constexpr bool kPair = kFull && TILE && 2 * RPT <= LANES;
    const int r2 = kPair ? reduced_row<LANES, (kPair ? 2 * RPT : RPT)>(j) : 0;
    const int q2 = r2 % RPT, t2 = r2 / RPT;
    const bool ystore = kFull && rvalid;

    // ---- A2 state load: U = S at the start (slot, segment plan, or zero) ----
    float2 u[RPT][VPL][2];
    {
        const float *src = nullptr;
        if (from_slot)
            src = a.state + (long long)seq * HP * N;
        else if (from_plan)          // the combine pass left S_in[seg] in unit-1's scratch
            src = plan.seg_state + (long long)(unit - 1) * HP * N;
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            const float *row = src + ((long long)r0 + rl + q) * N;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int c = k * LANES + j;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (src && rvalid && (EXACT || c < N4))
                    v = *reinterpret_cast<const float4 *>(row + 4 * c);
                u[q][k][0] = f2(v.x, v.y);
                u[q][k][1] = f2(v.z, v.w);
            }
        }
    }

    // Per-token strides of the staged operands, in floats.  With the exact
    // shapes N is a compile-time constant, so the B and C reads of a group of
    // tokens take immediate offsets from one pointer.
    const int Ns = EXACT ? 4 * LANES * VPL : N;
    const int xs = geo.rows_per_cta, hc = geo.heads_cap;

    // The gated RMSNorm of chunk cc, shared by the consumer warps once all of
    // the chunk's y is in its tile: eight lanes per token (lane group g of
    // warp w takes token 4 w + g, then every 4 * warps tokens), each lane the
    // 128-bit pieces l, l + 8, ... of the row (a quarter warp reads 128
    // contiguous bytes: no bank conflicts); the row's sum of squares by three
    // shuffles, then gated = y / sqrt(mean(y^2) + eps) * w * silu(z), silu from
    // the hardware exponential and an approximate division (about 1e-6
    // relative, far inside the scan's bound).
    auto gate = [&](int cc) {
        const int bb = cc % kSlots;
        const int cnt = min(geo.chunk, len - cc * geo.chunk);
        const int xs = geo.rows_per_cta;
        const int nw = SELF ? kSelfThreads / 32 : (nthr >> 5) - 1, sub = lane >> 3, l8 = lane & 7;
        const float *Y = SELF ? sm.SelfY<NS>(cc & 1) : sm.Ytile(bb);
        const float *Z = SELF ? sm.SelfZ<NS>(cc & 1) : sm.Ztile(bb);
        const float inv_p = 1.f / (float)nrows;
        float *out = gt.out + ((long long)tok_start + cc * geo.chunk) * HP + r0;
        float *yout = a.y + ((long long)tok_start + cc * geo.chunk) * HP + r0;   // self-staged: y too
        for (int tr = warp * 4; tr < cnt; tr += nw * 4) {
            const int t = tr + sub;
            const bool live = t < cnt;
            float ss = 0.f;
            for (int e = 4 * l8; e < nrows; e += 32) {
                if (live) {
                    const float4 v = *reinterpret_cast<const float4 *>(Y + t * xs + e);
                    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
                }
            }
            ss += __shfl_xor_sync(kFullMask, ss, 4);
            ss += __shfl_xor_sync(kFullMask, ss, 2);
            ss += __shfl_xor_sync(kFullMask, ss, 1);
            const float inv = rsqrtf(ss * inv_p + gt.eps);
            if (live) {
                for (int e = 4 * l8; e < nrows; e += 32) {
                    const float4 v = *reinterpret_cast<const float4 *>(Y + t * xs + e);
                    const float4 z = *reinterpret_cast<const float4 *>(Z + t * xs + e);
                    const float4 w = __ldg(reinterpret_cast<const float4 *>(gt.w + e));
                    float4 o;
                    o.x = v.x * inv * w.x * __fdividef(z.x, 1.f + __expf(-z.x));
                    o.y = v.y * inv * w.y * __fdividef(z.y, 1.f + __expf(-z.y));
                    o.z = v.z * inv * w.z * __fdividef(z.z, 1.f + __expf(-z.z));
                    o.w = v.w * inv * w.w * __fdividef(z.w, 1.f + __expf(-z.w));
                    *reinterpret_cast<float4 *>(out + (long long)t * HP + e) = o;
                    if (SELF)                         // no producer writes the y tile out
                        *reinterpret_cast<float4 *>(yout + (long long)t * HP + e) = v;
                }
            }
        }
    };

    // Self-staged y through tiles (EPI 5): chunk cc's y tile to global memory,
    // spread over the whole block; 128-bit stores where the rows allow (then x
    // moves in 16-byte pieces too, and its walk fits y).
    const bool y16 = x16 && (reinterpret_cast<uintptr_t>(a.y) & 15) == 0;
    auto flush_y = [&](int cc) {
        const int cnt = min(geo.chunk, len - cc * geo.chunk);
        const int xs = geo.rows_per_cta;
        const float *Y = sm.SelfY<NS>(cc & 1);
        float *yg = a.y + ((long long)tok_start + cc * geo.chunk) * HP + r0;
        if (y16) {
            for (int t = xt0, r = xv0; t < cnt;) {   // the x walk: xw = nrows / 4 pieces per token
                *reinterpret_cast<float4 *>(yg + t * HP + 4 * r) =
                    *reinterpret_cast<const float4 *>(Y + t * xs + 4 * r);
                t += xdt;
                r += xdv;
                if (r >= xw) { r -= xw; ++t; }
            }
        } else {
            for (int i = tid; i < cnt * nrows; i += kSelfThreads) {
                const int t = i / nrows, r = i - t * nrows;
                yg[t * HP + r] = Y[t * xs + r];
            }
        }
    };

    // Self-staged (no producer warp): every thread copies its share of each
    // chunk NS - 1 chunks ahead (one commit group per chunk, and one for z),
    // and the warps take turns forming the next chunk's coefficients at the end
    // of a chunk; one block barrier per chunk.
    constexpr int ncw = kSelfThreads / 32;
    const float dnone[kDtHeads] = {};                 // self-staged: dt comes through shared memory
    float pend = 1.f;                                 // Lambda_last of the previous chunk, not yet applied to U
    // U <- r U (an anchor's rescale, or Lambda_last back to S)
    auto rescale = [&](float r) {
        const float2 r2 = f2(r, r);
#pragma unroll
        for (int q = 0; q < RPT; ++q)
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                u[q][k][0] = __fmul2_rn(u[q][k][0], r2);
                u[q][k][1] = __fmul2_rn(u[q][k][1], r2);
            }
    };
    if constexpr (SELF) {
        if (n_chunks > 0)
            stage(0, 0);
        else
            cp_async_commit();
        if constexpr (NS == 3) {
            if (n_chunks > 1)
                stage(1, 1);
            else
                cp_async_commit();                    // one commit group per chunk, empty past the end
        }
        if (warp == 0 && n_chunks > 0) {
            cp_async_wait<NS - 2>();                  // this warp's copies of chunk 0 (its dt) landed
            coefficients(0, 0, dnone);
        }
    }
    for (int c = 0; c < n_chunks; ++c) {
        const int b = c % NS;
        bool coef_warp = false;                       // self-staged: this warp forms chunk c+1's coefficients
        if constexpr (SELF) {
            // (bar.sync as inline asm, like the y-tile stores, so the compiler keeps their order)
            cp_async_wait<NS - 2>();                  // this thread's copies of chunk c (and z of c-1) landed
            bar_sync(0, kSelfThreads);                // everyone's, and chunk c's coefficients; chunk c-1 done
            // chunk c-1's y tile (and z) are complete; tile (c - 1) % 2 is rewritten in
            // chunk c+1, after the next barrier
            if constexpr (GATED) {
                if (c >= 1)
                    gate(c - 1);
                stage_z(c);                           // into z tile c % 2 (z of c-2 was gated in chunk c-1)
            } else if constexpr (TILE) {
                if (c >= 1)
                    flush_y(c - 1);
            }
            if (c + NS - 1 < n_chunks)
                stage(c + NS - 1, (c + NS - 1) % NS); // its slot held chunk c-1
            else
                cp_async_commit();
            coef_warp = c + 1 < n_chunks && warp == (c + 1) % ncw;
        } else {
            bar_sync(kBarFull + b, nthr);
        }
        if constexpr (GATED && !SELF) {
            // every consumer warp has arrived here, so all of chunk c-1's y is
            // in its tile: gate it, then release its slot
            if (c >= 1) {
                gate(c - 1);
                __syncwarp();
                bar_arrive(kBarEmpty + (c - 1) % kSlots, nthr);
            }
        }
        const int cnt = min(geo.chunk, len - c * geo.chunk);
        const float *__restrict__ pB = sm.B(b) + 4 * j;      // this lane's first float4 of a token's B
        const float *__restrict__ pC = sm.C(b) + 4 * j;
        const float4 *__restrict__ pCf = sm.Coef(b) + hl;
        const float *__restrict__ pX = sm.X(b) + rl;
        float *yrow = a.y + ((long long)tok_start + c * geo.chunk) * HP + r0 + rl + yq;
        float *pY = !TILE ? nullptr                            // the chunk's y tile (EPI 1, 2, 4)
                          : (SELF ? sm.SelfY<NS>(c & 1) : sm.Ytile(b)) + rl + yq;
        float *yrow2 = yrow - yq + q2, *pY2 = TILE ? pY - yq + q2 : nullptr;   // the pairwise reduction's row

        // Shared-memory operands of one token.
        struct TokenIn {
            float4 cf;          // {dt/Lambda, Lambda, r, -}
            float xv[RPT];
            float4 b[VPL], c[VPL];
        };
        auto load_token = [&](int t, TokenIn &in) {
            in.cf = pCf[t * hc];
            load_rows<RPT>(in.xv, pX + t * xs);
            const float *bt = pB + t * Ns;
            const float *ct = pC + t * Ns;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                if (EXACT || k * LANES + j < N4) {
                    in.b[k] = *reinterpret_cast<const float4 *>(bt + 4 * k * LANES);
                    if constexpr (kFull)
                        in.c[k] = *reinterpret_cast<const float4 *>(ct + 4 * k * LANES);
                }
            }
        };
        // One token: U += (x dt / Lambda) B; with y, this lane's parts of U . C
        // for its RPT rows (before the reduction over the row's lanes).
        auto step_part = [&](const TokenIn &in, float (&part)[RPT]) {
            float2 a2[RPT];
#pragma unroll
            for (int q = 0; q < RPT; ++q) {
                const float alpha = in.xv[q] * in.cf.x;
                a2[q] = f2(alpha, alpha);
            }
            // all state updates first, then the dot products, so no FMA waits
            // on the one issued just before it
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                if (EXACT || k * LANES + j < N4) {
                    const float4 bb = in.b[k];
#pragma unroll
                    for (int q = 0; q < RPT; ++q) {
                        u[q][k][0] = __ffma2_rn(a2[q], f2(bb.x, bb.y), u[q][k][0]);      // A5
                        u[q][k][1] = __ffma2_rn(a2[q], f2(bb.z, bb.w), u[q][k][1]);
                    }
                }
            }
            if constexpr (kFull) {                                                       // A6
                // two accumulator chains per row (one when a lane holds a
                // single float4 of it); the first product starts each chain
                constexpr int NACC = VPL > 1 ? 2 : 1;
                float2 acc[RPT][NACC];
#pragma unroll
                for (int k = 0; k < VPL; ++k) {
                    const bool live = EXACT || k * LANES + j < N4;
                    const float4 cc = in.c[k];
#pragma unroll
                    for (int q = 0; q < RPT; ++q) {
                        float2 &ac = acc[q][k % NACC];
                        if (live) {
                            if (k < NACC)
                                ac = __fmul2_rn(u[q][k][0], f2(cc.x, cc.y));
                            else
                                ac = __ffma2_rn(u[q][k][0], f2(cc.x, cc.y), ac);
                            ac = __ffma2_rn(u[q][k][1], f2(cc.z, cc.w), ac);
                        } else if (k < NACC) {
                            ac = f2(0.f, 0.f);
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < RPT; ++q) {
                    const float2 s2 = NACC > 1 ? __fadd2_rn(acc[q][0], acc[q][NACC - 1]) : acc[q][0];
                    part[q] = s2.x + s2.y;
                }
            }
        };
        // One token with y: the lanes' parts summed by shuffles (transposing
        // over the RPT rows), then y = Lambda (U . C) + D x from the lane that
        // holds the row's sum.  Every lane holds the full sum of its row, so all
        // lanes of a row store the same value (no divergent branch).
        auto step = [&](const TokenIn &in, int t) {
            float part[RPT];
            step_part(in, part);
            if constexpr (kFull) {
                const float ysum = reduce_rows<LANES, RPT>(part, j);
                const float yv = fmaf(in.cf.y, ysum, Dv * pX[t * xs + yq]);
                if (ystore) {
                    if constexpr (TILE)
                        st_shared_unordered(pY + t * xs, yv);
                    else
                        yrow[t * HP] = yv;
                }
            }
        };
        // Two tokens t0, t0 + 1 with y: their 2 RPT row sums in one transposing
        // reduction (twice the independent shuffles per level); every lane ends
        // with the sum of one (token, row) pair (q2, t2 above) and stores it.
        auto step_pair = [&](const TokenIn &i0, const TokenIn &i1, int t0) {
            if constexpr (kPair) {
                float p[2 * RPT];
                step_part(i0, reinterpret_cast<float (&)[RPT]>(p[0]));
                step_part(i1, reinterpret_cast<float (&)[RPT]>(p[RPT]));
                const float ysum = reduce_rows<LANES, 2 * RPT>(p, j);
                const int tt = t0 + t2;
                const float yv = fmaf(t2 ? i1.cf.y : i0.cf.y, ysum, Dv * pX[tt * xs + q2]);
                if (ystore) {
                    if constexpr (TILE)
                        st_shared_unordered(pY2 + tt * xs, yv);
                    else
                        yrow2[tt * HP] = yv;
                }
            }
        };
        // Anchor tokens (any head of the block) rescale U before their update;
        // a head that does not anchor there has r = 1 (exact no-op).  Token 0
        // anchors every head.  Runs of kRun tokens with no anchor after their
        // first go through straight-line code; the rest one token at a time.
        unsigned amask = 0;
        for (int hh = 0; hh < nheads; ++hh)
            amask |= sm.Mask(b)[hh];
        // The compiler schedules a run's tokens as one block of code, so
        // the operands of the next token are read while the current one
        // computes.
        constexpr int kRun = 8;
        constexpr unsigned kRunMask = (1u << kRun) - 2u;    // the run's tokens after its first
        int t = 0;
        while (t < cnt) {
            if ((amask >> t) & 1u)                    // token 0 anchors: also the previous chunk's Lambda_last
                rescale(t == 0 ? pCf[0].z * pend : pCf[t * hc].z);
            if (t + kRun <= cnt && ((amask >> t) & kRunMask) == 0u) {
                if constexpr (kPair) {
#pragma unroll
                    for (int v = 0; v < kRun; v += 2) {
                        TokenIn i0, i1;
                        load_token(t + v, i0);
                        load_token(t + v + 1, i1);
                        step_pair(i0, i1, t + v);
                    }
                } else {
#pragma unroll
                    for (int v = 0; v < kRun; ++v) {
                        TokenIn in;
                        load_token(t + v, in);
                        step(in, t + v);
                    }
                }
                t += kRun;
            } else {
                TokenIn in;
                load_token(t, in);
                step(in, t);
                ++t;
            }
        }
        // back to S at the chunk end (U <- Lambda_last U), folded into the next
        // chunk's first rescale or applied after the last chunk
        pend = pCf[(cnt - 1) * hc].y;
        __syncwarp();
        if constexpr (SELF) {
            if (coef_warp) {                          // into chunk c+1's slot, read after the next barrier
                cp_async_wait<NS - 2>();              // this warp's copies of chunk c+1 (its dt) landed
                coefficients(c + 1, (c + 1) % NS, dnone);
            }
        } else if (!GATED && (TILE || c + kSlots < n_chunks)) {
            // release the slot: the producer refills it with chunk c+3 (with the
            // output tile it first writes the tile out; with the gated output the
            // release comes after the chunk's gating, at the start of chunk c+1)
            bar_arrive(kBarEmpty + b, nthr);
        }
    }
    if constexpr (GATED && SELF) {
        if (n_chunks > 0) {                 // the last chunk: its y tile and z complete
            cp_async_wait<0>();
            bar_sync(0, kSelfThreads);
            gate(n_chunks - 1);
        }
    } else if constexpr (SELF && TILE) {
        if (n_chunks > 0) {                 // the last chunk's y tile
            bar_sync(0, kSelfThreads);
            flush_y(n_chunks - 1);
        }
    } else if constexpr (GATED) {
        if (n_chunks > 0) {                 // the last chunk: every consumer warp done with it
            bar_sync(kBarConsumers, nthr - 32);
            gate(n_chunks - 1);
            __syncwarp();
            bar_arrive(kBarEmpty + (n_chunks - 1) % kSlots, nthr);
        }
    }

    if (n_chunks > 0)
        rescale(pend);                                // U <- Lambda_last U: the state S again

    // ---- A7 state store: slot (last segment) or the unit's scratch (state pass) ----
    float *dst = nullptr;
    if (to_slot)
        dst = a.state + (long long)seq * HP * N;
    else if (!kFull)
        dst = plan.seg_state + (long long)unit * HP * N;
    if (dst && rvalid) {
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
            float *slot = dst + ((long long)r0 + rl + q) * N;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int c = k * LANES + j;
                if (EXACT || c < N4)
                    *reinterpret_cast<float4 *>(slot + 4 * c) =
                        make_float4(u[q][k][0].x, u[q][k][0].y, u[q][k][1].x, u[q][k][1].y);
            }
        }
    }
}

template <int LANES, int VPL, int RPT, bool EXACT, int MODE>
__global__ void __launch_bounds__(256, 1)
prefill_scaled_kernel(const ScanArgs a, const PrefillGeom geo, const SegmentPlan plan, const GatedOut gt)
{
    griddep_entry();
    prefill_scaled_body<LANES, VPL, RPT, EXACT, MODE, 0>(a, geo, plan, gt);
}

// At most 168 registers: two blocks of five warps put three warps on some SM
// sub-partition, whose register file holds 16 K registers.
template <int LANES, int VPL, int RPT, bool EXACT, int EPI>
__global__ void __maxnreg__(168)
prefill_scaled_tile_kernel(const ScanArgs a, const PrefillGeom geo, const SegmentPlan plan, const GatedOut gt)
{
    griddep_entry();
    prefill_scaled_body<LANES, VPL, RPT, EXACT, kScanFull, EPI>(a, geo, plan, gt);
}

// Self-staged full pass (EPI 4, 5): blocks of four consumer warps and no producer,
// three per SM (three warps on every SM sub-partition, at most 168 registers).

template <int LANES, int VPL, int RPT, bool EXACT, int EPI>
__global__ void __launch_bounds__(kSelfThreads, 3)
prefill_scaled_self_kernel(const ScanArgs a, const PrefillGeom geo, const SegmentPlan plan, const GatedOut gt)
{
    griddep_entry();
    prefill_scaled_body<LANES, VPL, RPT, EXACT, kScanFull, EPI>(a, geo, plan, gt);
}

namespace {

// Shapes with the output-tile variants (EPI 1 and 2): the automatic shapes of
// head_dim 64 at d_state 128 and 64.
template <int LANES, int VPL, int RPT>
constexpr bool kHasTile = LANES == 8 && RPT == 4 && (VPL == 4 || VPL == 2);

template <int LANES, int VPL, int RPT>
cudaError_t launch_scaled_one(const ScanArgs &a, const PrefillGeom &g, const SegmentPlan &plan, int mode,
                              long long n_units, size_t smem, int epi, const GatedOut &gt, cudaStream_t stream)
{
    const bool exact = (a.N / 4) == LANES * VPL;
    const int threads = (g.rows_per_cta / RPT) * LANES + (epi >= 3 ? 0 : 32);   // consumers (+ the producer)
    const dim3 grid((unsigned)(n_units * a.G * g.runs_per_group));
    void (*kern)(const ScanArgs, const PrefillGeom, const SegmentPlan, const GatedOut) = nullptr;
    if (mode != kScanFull) {
        if (epi != 0)
            return cudaErrorInvalidValue;
        kern = exact ? prefill_scaled_kernel<LANES, VPL, RPT, true, kScanStateOnly>
                     : prefill_scaled_kernel<LANES, VPL, RPT, false, kScanStateOnly>;
    } else if (epi == 0) {
        kern = exact ? prefill_scaled_kernel<LANES, VPL, RPT, true, kScanFull>
                     : prefill_scaled_kernel<LANES, VPL, RPT, false, kScanFull>;
    } else if (epi == 4 || epi == 5) {
        if (threads != kSelfThreads || (epi == 4 && !gt.out))
            return cudaErrorInvalidValue;
        if constexpr (kHasTile<LANES, VPL, RPT>) {
            if (epi == 4)
                kern = exact ? prefill_scaled_self_kernel<LANES, VPL, RPT, true, 4>
                             : prefill_scaled_self_kernel<LANES, VPL, RPT, false, 4>;
            else
                kern = exact ? prefill_scaled_self_kernel<LANES, VPL, RPT, true, 5>
                             : prefill_scaled_self_kernel<LANES, VPL, RPT, false, 5>;
        }
        if (!kern)
            return cudaErrorInvalidValue;
    } else {
        if (threads > kTileThreads)
            return cudaErrorInvalidValue;
        if constexpr (kHasTile<LANES, VPL, RPT>) {
            if (epi == 1)
                kern = exact ? prefill_scaled_tile_kernel<LANES, VPL, RPT, true, 1>
                             : prefill_scaled_tile_kernel<LANES, VPL, RPT, false, 1>;
            else if (epi == 2 && gt.out)
                kern = exact ? prefill_scaled_tile_kernel<LANES, VPL, RPT, true, 2>
                             : prefill_scaled_tile_kernel<LANES, VPL, RPT, false, 2>;
        }
        if (!kern)
            return cudaErrorInvalidValue;
    }
    if (smem > 48 * 1024) {
        cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(kern), smem);
        if (e != cudaSuccess)
            return e;
    }
    return launch_pdl(kern, grid, dim3(threads), smem, stream, a, g, plan, gt);
}

}  // namespace

// (lanes per row, float4 per lane and row, rows per lane)
#define SSM_SCALED_SHAPES(X) \
    X(16, 2, 8) X(16, 2, 4) X(16, 2, 2) X(16, 2, 1) X(32, 1, 8) X(32, 1, 4) X(8, 4, 4) \
    X(8, 2, 8) X(8, 2, 4) X(8, 2, 2) X(8, 2, 1) X(4, 2, 4) X(4, 2, 2) X(4, 2, 1) \
    X(2, 2, 2) X(2, 2, 1) X(1, 2, 1) X(1, 1, 1) \
    X(32, 2, 8) X(32, 2, 4) X(32, 2, 1) X(32, 4, 4) X(32, 4, 2) X(32, 4, 1) X(32, 8, 2) X(32, 8, 1)

bool prefill_scaled_supported(int lanes, int vpl, int rpt)
{
#define X(L, V, R) if (lanes == L && vpl == V && rpt == R) return true;
    SSM_SCALED_SHAPES(X)
#undef X
    return false;
}

bool prefill_scaled_self_supported(int lanes, int vpl, int rpt, int rows_per_cta)
{
    if ((rows_per_cta / rpt) * lanes != kSelfThreads)     // the staging walk assumes the whole block
        return false;
#define X(L, V, R) if (lanes == L && vpl == V && rpt == R) return kHasTile<L, V, R>;
    SSM_SCALED_SHAPES(X)
#undef X
    return false;
}

bool prefill_scaled_tile_supported(int lanes, int vpl, int rpt, int rows_per_cta)
{
    if ((rows_per_cta / rpt) * lanes + 32 > kTileThreads)
        return false;
#define X(L, V, R) if (lanes == L && vpl == V && rpt == R) return kHasTile<L, V, R>;
    SSM_SCALED_SHAPES(X)
#undef X
    return false;
}

cudaError_t launch_prefill_scaled(const ScanArgs &a, const PrefillGeom &g, int lanes, int vpl, int rpt,
                                  const SegmentPlan &plan, int mode, long long n_units, size_t smem,
                                  cudaStream_t stream, int epi, const GatedOut *gated)
{
    const GatedOut gt = gated ? *gated : GatedOut{};
#define X(L, V, R) \
    if (lanes == L && vpl == V && rpt == R) \
        return launch_scaled_one<L, V, R>(a, g, plan, mode, n_units, smem, epi, gt, stream);
    SSM_SCALED_SHAPES(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace ssm
