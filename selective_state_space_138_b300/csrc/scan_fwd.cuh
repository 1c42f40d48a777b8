// scan_fwd.cuh -- the forward selective scan kernels: the n-split kernel and the time-lane kernel (the host side is in scan_fwd_host.cuh).
//
// Part of the single translation unit ss_scan.cu (included inside its
// anonymous namespace); not compiled on its own.

#pragma once

// ------------------------------------------------------------------ time-lane scan kernel
//
// A CTA owns one batch row b and CH consecutive channels d. Each channel is
// served by W lanes of one warp ("time lanes"); the sequence is walked in
// chunks of LC = W * K steps, lane j of a channel owning steps
// [t0 + j*K, t0 + j*K + K) of every chunk.
//   * B and C of the chunk (shared by every channel of the batch row) are
//     staged once per CTA into shared memory as fp32, layout [t][n], so that
//     all CH channels reuse them.
//   * x, dt, z of a lane's K steps are read with 16-byte loads.
//   * W == 1: the lane walks its K steps with all N states in registers.
//   * W > 1: for each state n the lane forms its K pairs
//     (a_i, b_i) = (exp(delta_i A_n), delta_i x_i B_{i,n}), folds them into one
//     affine map, the W lanes combine their maps with
//     (a1, b1) then (a2, b2) = (a1 a2, a2 b1 + b2) in a shuffle scan
//     ("Mamba, annotated", "The scan, in one equation"), and each lane then
//     re-walks its K pairs (kept in registers) from its incoming state.
//   * The state of each (channel, n) is carried between chunks in registers and
//     written to HBM only once, as final_state.
// Steps past L are given delta = 0, which is the identity map (a = 1, b = 0).

struct ScanParams {
    const void *x, *dt, *B, *C, *z;
    const float *A, *D, *dt_bias;
    void *y;
    float *final_state;
    int64_t batch, d_inner, L, N;
    int softplus;
    int vec;          // 16-byte vector loads/stores allowed
    int nseg;         // segments per channel group (a thread-block cluster when > 1)
    int64_t seg_len;  // steps per segment, a multiple of the chunk length
    const float *h0;        // (batch, d_inner, N) initial state, or NULL for zero
    const uint8_t *reset;   // (batch, L) sequence starts, or NULL (n-split kernel only)
    float4 *ckpt;           // the backward's stored states (its workspace layout), or NULL
    int64_t nsub;           // 16-step sub-chunks of the sequence (when ckpt is set)
    int tma;                // n-split kernel: tiles come in through the tensor maps below
    // 3-d maps over (step, row, batch row): x, dt, z with rows = channels and
    // B, C with rows = states; boxes as the n-split kernel stages them
    CUtensorMap tm_x, tm_dt, tm_z, tm_B, tm_C;
};

// Shared-memory index of (t, n) within a chunk: K-step blocks of NT floats per
// step, each block followed by 4 floats of padding so that the W lanes of a
// channel (which read steps K apart) hit distinct banks.
template <int NT, int K>
__device__ __forceinline__ int sidx(int t, int n)
{
    return (t / K) * (K * NT + 4) + (t % K) * NT + n;
}

template <typename T, int NT, int W, int K>
__global__ void __launch_bounds__(kBlock)
scan_fwd_kernel(const ScanParams p)
{
    constexpr int CH = kBlock / W;      // channels per CTA
    constexpr int LC = W * K;           // steps per chunk
    constexpr int TILE = W * (K * NT + 4);
    extern __shared__ __align__(16) float smem[];
    float *Bs = smem;
    float *Cs = smem + TILE;

    const int tid = threadIdx.x;
    const int c = tid / W;              // channel within CTA
    const int j = tid % W;              // time lane
    const int64_t b = blockIdx.y;
    const int64_t d = static_cast<int64_t>(blockIdx.x) * CH + c;
    const bool active = d < p.d_inner;
    const int64_t dd = active ? d : 0;
    const int64_t N = p.N;
    const int64_t L = p.L;
    const int64_t row = b * p.d_inner + dd;

    const T *xr = static_cast<const T *>(p.x) + row * L;
    const T *dtr = static_cast<const T *>(p.dt) + row * L;
    const T *zr = p.z ? static_cast<const T *>(p.z) + row * L : nullptr;
    T *yr = static_cast<T *>(p.y) + row * L;
    const T *Bb = static_cast<const T *>(p.B) + b * N * L;
    const T *Cb = static_cast<const T *>(p.C) + b * N * L;

    float A2[NT];
    float h[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        A2[n] = (n < N) ? __ldg(p.A + dd * N + n) * kLog2e : 0.0f;
        h[n] = 0.0f;
    }
    const float bias = p.dt_bias ? __ldg(p.dt_bias + dd) : 0.0f;
    const float Dd = p.D ? __ldg(p.D + dd) : 0.0f;
    const bool vec = p.vec != 0;

    const int64_t nchunks = (L + LC - 1) / LC;
    for (int64_t ch = 0; ch < nchunks; ++ch) {
        const int64_t t0 = ch * LC;
        __syncthreads();
        for (int e = tid; e < NT * LC; e += kBlock) {
            const int n = e / LC;
            const int tl = e % LC;
            const int64_t t = t0 + tl;
            float bv = 0.0f, cv = 0.0f;
            if (n < N && t < L) {
                bv = Io<T>::load1(Bb + n * L + t);
                cv = Io<T>::load1(Cb + n * L + t);
            }
            Bs[sidx<NT, K>(tl, n)] = bv;
            Cs[sidx<NT, K>(tl, n)] = cv;
        }
        __syncthreads();

        const int64_t tb = t0 + j * K;  // first step of this lane
        float dl[K], dx[K], yv[K];
        {
            float xv[K], dtv[K];
            load_items<T, K>(xr, tb, L, vec, xv);
            load_items<T, K>(dtr, tb, L, vec, dtv);
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const float v = dtv[i] + bias;
                float s = p.softplus ? softplus_f(v) : v;
                s = (tb + i < L) ? s : 0.0f;
                dl[i] = s;
                dx[i] = s * xv[i];
                yv[i] = Dd * xv[i];
            }
        }

        if constexpr (W == 1) {
#pragma unroll
            for (int i = 0; i < K; ++i) {
                const float *Bi = Bs + sidx<NT, K>(i, 0);
                const float *Ci = Cs + sidx<NT, K>(i, 0);
                float acc = yv[i];
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const float a = ex2_approx(dl[i] * A2[n]);
                    h[n] = fmaf(a, h[n], dx[i] * Bi[n]);
                    acc = fmaf(Ci[n], h[n], acc);
                }
                yv[i] = acc;
            }
        } else {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                float a[K], bb[K];
                float Pa = 1.0f, Pb = 0.0f;
#pragma unroll
                for (int i = 0; i < K; ++i) {
                    a[i] = ex2_approx(dl[i] * A2[n]);
                    bb[i] = dx[i] * Bs[sidx<NT, K>(j * K + i, n)];
                    Pb = fmaf(a[i], Pb, bb[i]);
                    Pa *= a[i];
                }
                // inclusive scan of the lanes' maps, earlier lanes first
#pragma unroll
                for (int off = 1; off < W; off *= 2) {
                    const float pa = __shfl_up_sync(0xffffffffu, Pa, off, W);
                    const float pb = __shfl_up_sync(0xffffffffu, Pb, off, W);
                    if (j >= off) {
                        Pb = fmaf(Pa, pb, Pb);
                        Pa = Pa * pa;
                    }
                }
                float ea = __shfl_up_sync(0xffffffffu, Pa, 1, W);
                float eb = __shfl_up_sync(0xffffffffu, Pb, 1, W);
                if (j == 0) {
                    ea = 1.0f;
                    eb = 0.0f;
                }
                float hh = fmaf(ea, h[n], eb);  // state entering this lane's steps
                const float hend = fmaf(Pa, h[n], Pb);
                h[n] = __shfl_sync(0xffffffffu, hend, W - 1, W);
#pragma unroll
                for (int i = 0; i < K; ++i) {
                    hh = fmaf(a[i], hh, bb[i]);
                    yv[i] = fmaf(Cs[sidx<NT, K>(j * K + i, n)], hh, yv[i]);
                }
            }
        }

        if (zr) {
            float zv[K];
            load_items<T, K>(zr, tb, L, vec, zv);
#pragma unroll
            for (int i = 0; i < K; ++i)
                yv[i] *= silu_f(zv[i]);
        }
        if (active)
            store_items<T, K>(yr, tb, L, vec, yv);
    }

    if (p.final_state && active && j == 0) {
        float *fs = p.final_state + row * N;
#pragma unroll
        for (int n = 0; n < NT; ++n)
            if (n < N)
                fs[n] = h[n];
    }
}

// ------------------------------------------------------------------ n-split scan kernel
//
// A CTA owns batch row b and CH = 32 channels, with S warps, lane c of every
// warp serving channel c. Warp q holds NPL consecutive states (8q.. for NPL =
// 8, 4q.. for NPL = 4) of all 32 channels; N is padded to S*NPL states with
// A = B = C = 0, which leaves the padded states at zero. Every lane walks the
// whole sequence one step after another, so each element-step costs one
// exponential and four fp32 multiply(-add)s, done in pairs with the packed
// f32x2 instructions; time is not split, so no combine work is added.
//
// Shared-memory delivery and issue slots set the pace on this part, so the
// layout keeps both low: B_t and C_t of a warp's states are the same for all
// its lanes (a warp-uniform load), a lane reads the (delta, delta*x) of two
// steps in one 16-byte load, and NPL = 8 states per lane share each of those
// loads and the lane's per-step bookkeeping (N > 8; NPL = 4 for N <= 8 keeps
// more warps per SM).
//
// The sequence is cut into chunks of LC = 32 steps. Per chunk k:
//   scan      lane c of warp q advances its NPL states over the chunk (decays
//             of the next AHEAD steps formed ahead of the state update) and
//             keeps its partial readouts sum over its states of C_t[n] h_t[n]
//             in registers, storing them when the chunk is done;
//   -- barrier --
//   epilogue  thread (c, r) adds the S partials of its RL = LC / S steps,
//             adds D x, applies the silu(z) gate and stores y;
//   prep      the same thread forms delta = softplus(dt + bias) (or dt + bias)
//             and delta*x for its steps of chunk k+1, and B, C of chunk k+1
//             are converted to fp32 [t][n];
//   -- barrier --
// The raw x, dt, z, B, C tiles of every chunk are brought into a ring of
// STAGES chunks (tensor copies, or cp.async pieces for rows that are not
// 16-byte aligned) three chunks ahead of their use, so DRAM latency hides
// behind three iterations. The per-step work (softplus, gate, conversions)
// is done once per (channel, step), two steps at a time with f32x2 arithmetic.

#ifndef SS_NSPLIT_AHEAD
#define SS_NSPLIT_AHEAD 4  // steps whose decays are formed ahead of the state update
#endif
#ifndef SS_NSPLIT_STAGES
#define SS_NSPLIT_STAGES 4  // raw chunks resident in shared memory: k .. k+3 (a power of two)
#endif

// row stride (floats) of the fp32 B, C tiles [t][n]: 16-byte rows, and the
// conversion's 16-byte stores (lanes over 4-state groups, then step pairs)
// spread over all banks
constexpr int nsplit_bc_stride(int ns) { return ns <= 4 ? 8 : (ns == 8 ? 12 : ns + 8); }

template <typename T, int S, int NPL, int ST = SS_NSPLIT_STAGES>
struct NSplitShape {
    static constexpr int CH = 32;                 // channels per CTA
    static constexpr int NT = CH * S;             // threads per CTA
    static constexpr int NS = NPL * S;            // padded states
    static constexpr int NSP = nsplit_bc_stride(NS);
    static constexpr int LC = 32;                 // steps per chunk
    static constexpr int RL = LC / S;             // steps per epilogue/prep thread
    static constexpr int STAGES = ST;
    static constexpr int EPP = 16 / (int)sizeof(T);        // elements per 16-byte piece
    static constexpr int PR = LC / EPP;                    // pieces per raw row
    static constexpr int ROWB = LC * (int)sizeof(T) + 16;  // raw x/dt/z row stride, padded
    static constexpr int RAW_X = CH * ROWB;                // one raw x, dt or z tile
    static constexpr int RAW_BC = NS * LC * (int)sizeof(T);  // one raw B or C tile
    static constexpr int STAGE_BYTES = 3 * RAW_X + 2 * RAW_BC;
    static constexpr int NPIECE = (3 * CH + 2 * NS) * PR;
    static constexpr int PPT = (NPIECE + NT - 1) / NT;    // raw pieces per thread
    static constexpr int YROW = LC + 4;           // floats per partial row (conflict-free)
    static constexpr int YQ = CH * YROW;          // floats per state group
    static constexpr int PD_BYTES = (LC / 2) * CH * 16;   // (delta, delta x) of step pairs, [t/2][c]
    static constexpr int BC_BYTES = LC * NSP * 4;
    static constexpr int Y_BYTES = S * YQ * 4;
    static constexpr int X_BYTES = S * CH * NPL * 4 + S * CH * 4;   // segment end states and step sums
    static constexpr int R_BYTES = LC + 16;                          // sequence starts of a chunk, segment flag
    static constexpr size_t BAR_OFF = ((size_t)STAGES * STAGE_BYTES + PD_BYTES + 2 * BC_BYTES + Y_BYTES + X_BYTES +
                                       R_BYTES + 7) / 8 * 8;
    static constexpr size_t BYTES = BAR_OFF + 8 * STAGES;   // + the stage barriers
    static_assert(STAGE_BYTES % 128 == 0 && RAW_X % 128 == 0 && RAW_BC % 128 == 0, "tensor-copy tiles 128-aligned");
    static_assert(RL % 4 == 0, "epilogue runs are read 4 steps at a time");
    static_assert(NPL == 4 || NPL == 8, "states per lane");
};

// REV: the recurrence runs from t = L-1 down to 0 (h_t = a_t h_{t+1} + delta_t
// B_t x_t); chunks and the steps inside them are walked in that order, the
// tiles themselves are the same. RST: p.reset marks sequence starts; the
// carried state is zeroed before a marked step (forward) or after it
// (reverse), i.e. at the boundary between t-1 and t either way.

// TMA: the chunks arrive by tensor copies (the maps in p are encoded); the
// cp.async form is a separate instantiation, so neither carries the other's
// registers.
// ST: the stages of the ring; 2 stages with 4 states per lane on 4 warps fit four CTAs
// on an SM (the wide form, for grids that three per SM would leave as a partial
// second wave).
template <typename T, int S, int NPL, bool REV, bool RST, bool TMA, int ST = SS_NSPLIT_STAGES>
__global__ void __launch_bounds__(NSplitShape<T, S, NPL, ST>::NT,
                                  NPL == 8 ? (S <= 2 ? 4 : 2)
                                           : (S <= 2 ? 4 : (S == 4 ? (ST == 2 ? 4 : 3) : 1)))
scan_nsplit_kernel(const __grid_constant__ ScanParams p)
{
    using SH = NSplitShape<T, S, NPL, ST>;
    constexpr int NT = SH::NT, CH = SH::CH, NS = SH::NS, NSP = SH::NSP, LC = SH::LC, RL = SH::RL, PR = SH::PR;
    constexpr int STAGES = SH::STAGES, EPP = SH::EPP, PPT = SH::PPT;
    constexpr int D = SS_NSPLIT_AHEAD;
    constexpr int P = NPL / 2;                    // state pairs per lane
    constexpr int G4 = NPL / 4;                   // 4-state groups per lane
    constexpr int RW = RL * (int)sizeof(T) / 4;   // 32-bit words per prep/epilogue run
    static_assert(LC % 4 == 0 && D >= 1 && D <= LC, "chunk shape");

    extern __shared__ __align__(128) unsigned char smem_tiles[];
    unsigned char *smem_raw = smem_tiles;
    unsigned char *raw = smem_raw;                                             // [STAGES][x, dt, z, B, C]
    float4 *Pd = reinterpret_cast<float4 *>(smem_raw + STAGES * SH::STAGE_BYTES);  // [LC/2][CH] step pairs
    float *Bf = reinterpret_cast<float *>(Pd + (LC / 2) * CH);                 // [LC][NSP]
    float *Cf = Bf + LC * NSP;                                                 // [LC][NSP]
    float *Yp = Cf + LC * NSP;                                                 // [S][CH][YROW]
    float4 *Hx = reinterpret_cast<float4 *>(Yp + S * SH::YQ);                  // [S][CH][G4] segment end states
    float *Sx = reinterpret_cast<float *>(Hx + S * CH * G4);                   // [S][CH] step sums
    unsigned char *Rst = reinterpret_cast<unsigned char *>(Sx + S * CH);       // [LC] sequence starts
    int *Rx = reinterpret_cast<int *>(Rst + LC);                               // any start in the segment
    const uint32_t raw_s = static_cast<uint32_t>(__cvta_generic_to_shared(raw));
    const uint32_t bars_s = raw_s + static_cast<uint32_t>(SH::BAR_OFF);   // [STAGES] "stage filled" barriers
    constexpr bool tma = TMA;
    if (TMA && (raw_s & 127u) != 0) {   // tensor copies need 128-byte aligned destinations
        if (threadIdx.x == 0)
            atomicOr(&g_fault_flags, kFaultSmemAlign);
        return;
    }

    const int tid = threadIdx.x;
    const int nseg = p.nseg;
    const int seg = static_cast<int>(blockIdx.x % nseg);
    const int64_t b = blockIdx.y;
    const int64_t d0 = static_cast<int64_t>(blockIdx.x / nseg) * CH;
    const int64_t L = p.L, N = p.N, Dn = p.d_inner;
    const int64_t t_lo = seg * p.seg_len;
    const int64_t t_hi = (t_lo + p.seg_len < L) ? t_lo + p.seg_len : L;
    const bool vec = p.vec != 0;
    const int64_t nchunks = (t_hi - t_lo + LC - 1) / LC;
    // chunk j in walking order sits at chunk phys(j) of the segment
    auto phys = [&](int64_t j) -> int64_t { return REV ? nchunks - 1 - j : j; };

    // scan role: channel cs = lane, states NPL*q .. NPL*q + NPL-1
    const int cs = tid % CH;
    const int q = tid / CH;
    const bool act_s = d0 + cs < Dn;
    const int64_t ds = act_s ? d0 + cs : 0;
    // epilogue/prep role: channel ce, run re (steps re*RL .. re*RL+RL-1 of a chunk)
    const int ce = tid % CH;
    const int re = tid / CH;
    const bool act_e = d0 + ce < Dn;
    const int64_t de = act_e ? d0 + ce : 0;
    T *yr = static_cast<T *>(p.y) + (b * Dn + de) * L;

    const u64 bias2 = splat((p.dt_bias && act_e) ? __ldg(p.dt_bias + de) : 0.0f);
    const u64 D2 = splat((p.D && act_e) ? __ldg(p.D + de) : 0.0f);
    const bool gate = p.z != nullptr;

    u64 A2p[P];   // (A_n, A_n+1) log2(e) of the lane's states
#pragma unroll
    for (int i = 0; i < P; ++i) {
        const int n = NPL * q + 2 * i;
        A2p[i] = pk((n < N) ? __ldg(p.A + ds * N + n) * kLog2e : 0.0f,
                    (n + 1 < N) ? __ldg(p.A + ds * N + n + 1) * kLog2e : 0.0f);
    }
    u64 h[P];
#pragma unroll
    for (int i = 0; i < P; ++i)
        h[i] = 0;   // +0.0f in both halves

    // the raw pieces this thread copies: source row pointer, element offset
    // within the chunk, shared-memory offset within a stage, whether the piece
    // is needed by the readout only (z, C); rows past d_inner or N (and a
    // missing z) copy nothing
    const T *src[PPT];
    uint32_t soff[PPT];
    int poff[PPT];
    bool ro_only[PPT];
#pragma unroll
    for (int u = 0; u < PPT; ++u) {
        const int pi = tid + u * NT;
        int r, pc;
        const T *base;
        uint32_t off;
        bool ok = pi < SH::NPIECE;
        if (pi < 3 * CH * PR) {
            const int tensor = pi / (CH * PR);
            r = (pi % (CH * PR)) / PR;
            pc = pi % PR;
            const T *g = static_cast<const T *>(tensor == 0 ? p.x : (tensor == 1 ? p.dt : p.z));
            ok = ok && d0 + r < Dn && g != nullptr;
            base = ok ? g + (b * Dn + d0 + r) * L : static_cast<const T *>(p.x);
            off = tensor * SH::RAW_X + r * SH::ROWB;
            ro_only[u] = tensor == 2;
        } else {
            const int v = pi - 3 * CH * PR;
            const int m = v / (NS * PR);
            r = (v % (NS * PR)) / PR;
            pc = v % PR;
            ok = ok && r < N;
            base = static_cast<const T *>(m == 0 ? p.B : p.C) + (b * N + (ok ? r : 0)) * L;
            off = 3 * SH::RAW_X + m * SH::RAW_BC + r * LC * (int)sizeof(T);
            ro_only[u] = m == 1;
        }
        src[u] = base;
        soff[u] = off + pc * 16;
        poff[u] = ok ? pc * EPP : (1 << 30);   // a piece that does not exist is always past the end
    }

    // Chunks are numbered across the walks of this CTA: chunk j of the current
    // walk is number g0 + j and sits in stage (g0 + j) % STAGES. With tensor
    // maps, a stage is filled by one thread's tensor copies completing on the
    // stage's barrier (phase parity (g0 + j) / STAGES); g_issued and g_done
    // count the numbers issued and waited for, so that copies still in flight
    // after a wait gave up can be let land before the CTA exits.
    int64_t g0 = 0, g_issued = 0, g_done = 0;
    bool aborted = false;
    static_assert((STAGES & (STAGES - 1)) == 0, "stage of a chunk number by masking");
    auto stage_of = [](int64_t g) { return static_cast<int>(static_cast<uint32_t>(g) & (STAGES - 1)); };
    auto parity_of = [](int64_t g) { return (static_cast<uint32_t>(g) / STAGES) & 1u; };
    if (tma) {
        if (tid == 0) {
            for (int s = 0; s < STAGES; ++s)
                mbar_init(bars_s + 8u * s, 1);
            mbar_fence_init();
        }
        __syncthreads();
    }
    auto wait_chunk = [&](int64_t j) {
        if (tma && !aborted) {
            const int64_t g = g0 + j;
            aborted = !mbar_wait(bars_s + 8u * stage_of(g), parity_of(g));
            if (!aborted)
                g_done = g + 1;
        }
    };

    // bring chunk j of the segment into its stage (with the pieces: steps at
    // or past the segment end and rows that do not exist are zero; with the
    // tensor maps: rows past d_inner or N and steps past L are zero, a raw
    // row holds the 16 bytes that follow the chunk as well)
    auto stage_in = [&](int64_t j, bool readout) {
        const int stage = stage_of(g0 + j);
        const uint32_t st = raw_s + static_cast<uint32_t>(stage * SH::STAGE_BYTES);
        const int64_t t1 = t_lo + phys(j) * LC;
        if (tma) {
            if (tid == 0 && !aborted) {
                const uint32_t bar = bars_s + 8u * stage;
                const bool zz = readout && gate;
                mbar_expect_tx(bar, 2 * SH::RAW_X + SH::RAW_BC + (zz ? SH::RAW_X : 0) + (readout ? SH::RAW_BC : 0));
                const int c0 = static_cast<int>(t1), cd = static_cast<int>(d0), cb = static_cast<int>(b);
                tma_load_3d(st, &p.tm_x, bar, c0, cd, cb);
                tma_load_3d(st + SH::RAW_X, &p.tm_dt, bar, c0, cd, cb);
                if (zz)
                    tma_load_3d(st + 2 * SH::RAW_X, &p.tm_z, bar, c0, cd, cb);
                tma_load_3d(st + 3 * SH::RAW_X, &p.tm_B, bar, c0, 0, cb);
                if (readout)
                    tma_load_3d(st + 3 * SH::RAW_X + SH::RAW_BC, &p.tm_C, bar, c0, 0, cb);
                g_issued = g0 + j + 1;
            }
            return;
        }
        const int rem = static_cast<int>(t_hi - t1 < (1 << 29) ? t_hi - t1 : (1 << 29));   // steps left
#pragma unroll
        for (int u = 0; u < PPT; ++u) {
            if (tid + u * NT >= SH::NPIECE)
                break;
            if (!readout && ro_only[u])
                continue;
            const int left = rem - poff[u];
            const int nb = left >= EPP ? 16 : (left > 0 ? left * (int)sizeof(T) : 0);
            const T *g = src[u] + (nb > 0 ? t1 + poff[u] : 0);
            if (vec) {
                cp_async16(st + soff[u], g, nb);
            } else {
                unsigned char *dst = raw + stage * SH::STAGE_BYTES + soff[u];
                const int ne = nb / (int)sizeof(T);
#pragma unroll
                for (int e = 0; e < EPP; ++e) {
                    if constexpr (sizeof(T) == 4)
                        reinterpret_cast<float *>(dst)[e] = e < ne ? g[e] : 0.0f;
                    else
                        reinterpret_cast<unsigned short *>(dst)[e] =
                            e < ne ? reinterpret_cast<const unsigned short *>(g)[e] : (unsigned short)0;
                }
            }
        }
        cp_async_commit();
    };

    // raw B (and C) of chunk j -> fp32 [t][n]: each item is (tensor, step
    // pair, 4-state group): four 2-step reads of the raw rows, written as two
    // 16-byte words (lanes run over the groups first, then the step pairs, so
    // that the stores of a quarter-warp cover every bank once)
    auto convert_bc = [&](int64_t j, bool readout) {
        const unsigned char *st = raw + stage_of(g0 + j) * SH::STAGE_BYTES + 3 * SH::RAW_X;
        constexpr int GN = NS / 4;
        constexpr int TPN = LC / 2;
        const int items = (readout ? 2 : 1) * TPN * GN;
        for (int w = tid; w < items; w += NT) {
            const int g = w % GN;
            const int tp = (w / GN) % TPN;
            const int m = w / (GN * TPN);
            const unsigned char *srcm = st + m * SH::RAW_BC;
            float lo[4], hi[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = 4 * g + e;
                if constexpr (sizeof(T) == 4) {
                    const float2 v = *reinterpret_cast<const float2 *>(srcm + (n * LC + 2 * tp) * 4);
                    lo[e] = v.x;
                    hi[e] = v.y;
                } else {
                    const uint32_t v = *reinterpret_cast<const uint32_t *>(srcm + (n * LC + 2 * tp) * 2);
                    lo[e] = bf16lo(v);
                    hi[e] = bf16hi(v);
                }
            }
            float *dst = (m == 0 ? Bf : Cf) + (2 * tp) * NSP + 4 * g;
            *reinterpret_cast<float4 *>(dst) = make_float4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<float4 *>(dst + NSP) = make_float4(hi[0], hi[1], hi[2], hi[3]);
        }
    };

    // this thread's sum of the steps it prepares (compensated), for the segment carry
    float ssum = 0.0f, scomp = 0.0f;
    auto kahan = [&](float v) {
        const float yv = v - scomp;
        const float tv = ssum + yv;
        scomp = (tv - ssum) - yv;
        ssum = tv;
    };

    // delta and delta*x of this thread's steps of chunk j, stored by step pair
    auto prep = [&](int64_t j, bool sum_steps) {
        const unsigned char *st = raw + stage_of(g0 + j) * SH::STAGE_BYTES;
        uint32_t xw[RW], dw[RW];
        read_run_raw<T, RL>(st + ce * SH::ROWB, re * RL, xw);
        read_run_raw<T, RL>(st + SH::RAW_X + ce * SH::ROWB, re * RL, dw);
        const int64_t left64 = t_hi - (t_lo + phys(j) * LC + re * RL);
        if (RST && tid < LC) {
            const int64_t tt = t_lo + phys(j) * LC + tid;
            Rst[tid] = (tt < t_hi && p.reset[b * L + tt]) ? 1 : 0;
        }
        const int lim = act_e ? static_cast<int>(left64 < RL ? left64 : RL) : 0;
#pragma unroll
        for (int i = 0; i < RL; i += 2) {
            const u64 xx = word_pair<T>(xw, i);
            const u64 u = add2(word_pair<T>(dw, i), bias2);
            const u64 s2 = p.softplus ? softplus2(u) : u;
            float s0, s1;
            upk(s2, s0, s1);
            s0 = i < lim ? s0 : 0.0f;
            s1 = i + 1 < lim ? s1 : 0.0f;
            if (sum_steps) {
                kahan(s0);
                kahan(s1);
            }
            float sx0, sx1;
            upk(mul2(pk(s0, s1), xx), sx0, sx1);
            Pd[((re * RL + i) >> 1) * CH + ce] = make_float4(s0, sx0, s1, sx1);
        }
    };

    float *yq_s = Yp + q * SH::YQ + cs * SH::YROW;   // this lane's partial readouts
    const float *Bq_s = Bf + NPL * q;                 // this warp's states of B_t, C_t
    const float *Cq_s = Cf + NPL * q;

    // the lane's states as NPL/4 words of 4
    auto store_groups = [&](float4 *dst, int64_t stride) {
#pragma unroll
        for (int gq = 0; gq < G4; ++gq) {
            float hv[4];
            upk(h[2 * gq], hv[0], hv[1]);
            upk(h[2 * gq + 1], hv[2], hv[3]);
            dst[gq * stride] = make_float4(hv[0], hv[1], hv[2], hv[3]);
        }
    };

    // walk the segment [t_lo, t_hi): with the readout (y stored) or without
    // it (state and step sum only)
    auto run = [&](auto ro) {
        constexpr bool RO = decltype(ro)::value;
#pragma unroll
        for (int s = 0; s < STAGES - 1; ++s)
            if (s < nchunks)
                stage_in(s, RO);
            else
                cp_async_commit();
        cp_async_wait<STAGES - 2>();
        if (nchunks > 0)
            wait_chunk(0);
        __syncthreads();
        prep(0, !RO);
        convert_bc(0, RO);
        __syncthreads();

        for (int64_t k = 0; k < nchunks; ++k) {
            const int64_t t0 = t_lo + phys(k) * LC;
            if (k + STAGES - 1 < nchunks)
                stage_in(k + STAGES - 1, RO);
            else
                cp_async_commit();

            // ---- scan: the lane's NPL states of channel cs over the chunk;
            // the decays and writes of step t + D are formed while the state
            // takes step t
            {
                u64 ra[D][P], rb[D][P];
                float yv[LC];
                float4 pdv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                // walking step u is chunk step t = tu(u)
                auto tu = [](int u) { return REV ? LC - 1 - u : u; };
                auto form = [&](int u, int slot) {
                    const int t = tu(u);
                    if ((u & 1) == 0)   // the first step of a pair in walking order loads the pair
                        pdv = Pd[(t >> 1) * CH + cs];
                    const u64 dd = splat((t & 1) ? pdv.z : pdv.x);
                    const u64 xx = splat((t & 1) ? pdv.w : pdv.y);
                    const float *bt = Bq_s + t * NSP;
#pragma unroll
                    for (int i = 0; i < P; i += 2) {
                        const ulonglong2 Bq = *reinterpret_cast<const ulonglong2 *>(bt + 2 * i);
                        ra[slot][i] = ex2_2(mul2(dd, A2p[i]));
                        ra[slot][i + 1] = ex2_2(mul2(dd, A2p[i + 1]));
                        rb[slot][i] = mul2(xx, Bq.x);
                        rb[slot][i + 1] = mul2(xx, Bq.y);
                    }
                };
#pragma unroll
                for (int i = 0; i < D; ++i)
                    form(i, i);
#pragma unroll
                for (int u = 0; u < LC; ++u) {
                    const int t = tu(u);
                    const int slot = u % D;
                    u64 a[P], bb[P];
#pragma unroll
                    for (int i = 0; i < P; ++i) {
                        a[i] = ra[slot][i];
                        bb[i] = rb[slot][i];
                    }
                    if (u + D < LC)
                        form(u + D, slot);
                    if (RST && !REV && Rst[t]) {   // a sequence starts at t: nothing carries in
#pragma unroll
                        for (int i = 0; i < P; ++i)
                            h[i] = 0;
                    }
#pragma unroll
                    for (int i = 0; i < P; ++i)
                        h[i] = fma2(a[i], h[i], bb[i]);
                    if constexpr (RO) {
                        const float *ct = Cq_s + t * NSP;
                        u64 acc = 0;
#pragma unroll
                        for (int i = 0; i < P; i += 2) {
                            const ulonglong2 Cq = *reinterpret_cast<const ulonglong2 *>(ct + 2 * i);
                            acc = (i == 0) ? mul2(Cq.x, h[i]) : fma2(Cq.x, h[i], acc);
                            acc = fma2(Cq.y, h[i + 1], acc);
                        }
                        yv[t] = hsum(acc);
                    }
                    if (RST && REV && Rst[t]) {    // a sequence starts at t: nothing carries to t-1
#pragma unroll
                        for (int i = 0; i < P; ++i)
                            h[i] = 0;
                    }
                    if constexpr (RO && !REV && !RST) {
                        // the state entering each 16-step sub-chunk, for the backward pass
                        if ((u == 15 || u == 31) && p.ckpt && act_s) {
                            const int64_t sc = (t0 + u + 1) / 16;
                            if (sc < p.nsub)
                                store_groups(p.ckpt + ((b * p.nsub + sc) * (NS / 4) + G4 * q) * Dn + ds, Dn);
                        }
                    }
                }
                if constexpr (RO) {
#pragma unroll
                    for (int t = 0; t < LC; t += 4)
                        *reinterpret_cast<float4 *>(yq_s + t) = make_float4(yv[t], yv[t + 1], yv[t + 2], yv[t + 3]);
                }
            }
            cp_async_wait<STAGES - 2>();   // chunk k+1 has landed (this thread's copies)
            if (k + 1 < nchunks)
                wait_chunk(k + 1);          // (the tensor copies of chunk k+1)
            __syncthreads();

            // ---- epilogue of chunk k: sum partials, skip term, gate, store
            if constexpr (RO) {
                const unsigned char *st = raw + stage_of(g0 + k) * SH::STAGE_BYTES;
                uint32_t xw[RW], zw[RW];
                read_run_raw<T, RL>(st + ce * SH::ROWB, re * RL, xw);
                if (gate)
                    read_run_raw<T, RL>(st + 2 * SH::RAW_X + ce * SH::ROWB, re * RL, zw);
                float out[RL];
#pragma unroll
                for (int i = 0; i < RL; i += 4) {
                    const float *yp = Yp + ce * SH::YROW + re * RL + i;
                    ulonglong2 acc = *reinterpret_cast<const ulonglong2 *>(yp);
#pragma unroll
                    for (int qq = 1; qq < S; ++qq) {
                        const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(yp + qq * SH::YQ);
                        acc.x = add2(acc.x, v.x);
                        acc.y = add2(acc.y, v.y);
                    }
                    acc.x = fma2(D2, word_pair<T>(xw, i), acc.x);
                    acc.y = fma2(D2, word_pair<T>(xw, i + 2), acc.y);
                    if (gate) {
                        acc.x = mul2(acc.x, silu2(word_pair<T>(zw, i)));
                        acc.y = mul2(acc.y, silu2(word_pair<T>(zw, i + 2)));
                    }
                    upk(acc.x, out[i], out[i + 1]);
                    upk(acc.y, out[i + 2], out[i + 3]);
                }
                if (act_e)
                    write_run<T, RL>(yr, t0 + re * RL, t_hi, vec, out);
            }

            // ---- prep of chunk k+1
            if (k + 1 < nchunks) {
                prep(k + 1, !RO);
                convert_bc(k + 1, RO);
            }
            __syncthreads();
        }
        cp_async_wait<0>();
        g0 += nchunks;
    };

    // the initial state (zero unless given)
    u64 g0h[P];
#pragma unroll
    for (int i = 0; i < P; ++i)
        g0h[i] = 0;
    if (p.h0 && act_s) {
        const float *hp = p.h0 + (b * Dn + ds) * N;
#pragma unroll
        for (int i = 0; i < P; ++i) {
            const int n = NPL * q + 2 * i;
            g0h[i] = pk(n < N ? hp[n] : 0.0f, n + 1 < N ? hp[n + 1] : 0.0f);
        }
    }
    if (nseg > 1) {
        // Segments of one channel group form a thread-block cluster. Each
        // segment but the one walked last walks its steps from a zero state
        // (no readout) and publishes its end state, its step sum and whether a
        // sequence starts inside it; the state entering segment s is then the
        // initial state and the maps of the segments walked before it, folded
        // in walking order, h <- exp(A * sum of steps) h + end state (the
        // decay is 0 across a sequence start), read through distributed shared
        // memory.
        cg::cluster_group cluster = cg::this_cluster();
        const int last = REV ? 0 : nseg - 1;
        if (seg != last)
            run(Flag<false>{});
        int has_start = 0;
        if (RST)
            for (int64_t t = t_lo + tid; t < t_hi; t += NT)
                has_start |= p.reset[b * L + t] != 0;
        has_start = __syncthreads_or(has_start);
        if (tid == 0)
            *Rx = has_start;
        store_groups(Hx + (q * CH + cs) * G4, 1);
        Sx[re * CH + ce] = ssum;
        cluster.sync();
        u64 f[P];
#pragma unroll
        for (int i = 0; i < P; ++i)
            f[i] = g0h[i];
        const int n_before = REV ? nseg - 1 - seg : seg;
        for (int i = 0; i < n_before; ++i) {
            const int sp = REV ? nseg - 1 - i : i;
            const float4 *ph = cluster.map_shared_rank(Hx, sp);
            const float *psum = cluster.map_shared_rank(Sx, sp);
            float tot = 0.0f;
#pragma unroll
            for (int r = 0; r < S; ++r)
                tot += psum[r * CH + cs];
            const bool cut = RST && *cluster.map_shared_rank(Rx, sp);
#pragma unroll
            for (int gq = 0; gq < G4; ++gq) {
                const float4 he = ph[(q * CH + cs) * G4 + gq];
                u64 a01 = ex2_2(mul2(splat(tot), A2p[2 * gq])), a23 = ex2_2(mul2(splat(tot), A2p[2 * gq + 1]));
                if (cut) {
                    a01 = 0;
                    a23 = 0;
                }
                f[2 * gq] = fma2(a01, f[2 * gq], pk(he.x, he.y));
                f[2 * gq + 1] = fma2(a23, f[2 * gq + 1], pk(he.z, he.w));
            }
        }
        cluster.sync();   // peers have finished reading this CTA's end state
#pragma unroll
        for (int i = 0; i < P; ++i)
            h[i] = f[i];
    } else {
#pragma unroll
        for (int i = 0; i < P; ++i)
            h[i] = g0h[i];
    }
    if (!REV && !RST && p.ckpt && act_s && seg == 0)   // the state entering sub-chunk 0
        store_groups(p.ckpt + ((b * p.nsub) * (NS / 4) + G4 * q) * Dn + ds, Dn);
    run(Flag<true>{});

    if (p.final_state && act_s && seg == (REV ? 0 : nseg - 1)) {
        float *fs = p.final_state + (b * Dn + ds) * N;
#pragma unroll
        for (int i = 0; i < P; ++i) {
            const int n = NPL * q + 2 * i;
            float h0v, h1v;
            upk(h[i], h0v, h1v);
            if (n < N)
                fs[n] = h0v;
            if (n + 1 < N)
                fs[n + 1] = h1v;
        }
    }
    if (tma && tid == 0)   // after a wait gave up: let the copies issued since land (each wait bounded)
        for (int64_t g = g_done; g < g_issued; ++g)
            mbar_wait(bars_s + 8u * stage_of(g), parity_of(g));
}
