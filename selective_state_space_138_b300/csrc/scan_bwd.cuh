// scan_bwd.cuh -- the backward pass of the scan (states recomputed) and its launch logic.
//
// Part of the single translation unit ss_scan.cu (included inside its
// anonymous namespace); not compiled on its own.

#pragma once

// ------------------------------------------------------------------ backward kernel
//
// Gradient of the scan with the states recomputed from the inputs ("Mamba and
// selective state spaces", section "Why the scan must be fused": the backward
// pass reloads x, delta, B, C and recomputes the states instead of storing
// them; the backward of a linear recurrence is a linear recurrence run in
// reverse). With g(z) = z sigmoid(z), per channel d and state n:
//   gy_t      = dout_t g(z_t)
//   lam_t     = a_{t+1} lam_{t+1} + C_t gy_t,   lam_{L-1} = dfinal + C_{L-1} gy_{L-1}
//   dB_t[n]  += lam_t delta_t x_t,  dC_t[n] += gy_t h_t   (summed over channels)
//   dA_n     += lam_t delta_t a_t h_{t-1}
//   dx_t      = D gy_t + delta_t sum_n lam_t B_t
//   ddelta_t  = sum_n lam_t A_n a_t h_{t-1} + x_t sum_n lam_t B_t
//   ddt_t     = ddelta_t sigmoid(dt_t + bias) (softplus) or ddelta_t
//   dz_t      = dout_t y_t g'(z_t),  y_t = sum_n C_t h_t + D x_t
//   dh0       = a_0 lam_0
//
// Layout as in the forward n-split kernel: a CTA owns batch row b and 32
// channels, warp q holds states 4q..4q+3, lane c channel c.
//   phase 1  walks the sequence forward (x, dt, B only) and stores the state
//            at the start of every HC-step sub-chunk in the workspace;
//   phase 2  walks the chunks in reverse. For each sub-chunk it reloads the
//            stored state, recomputes the HC states into registers, then runs
//            the adjoint recurrence backwards over them. Per step, the
//            channel sums of lam * delta x and gy * h (dB, dC) are formed by a
//            transposing butterfly over the 32 lanes; the state sums
//            (lam B, lam A a h, C h) are left per warp in shared memory and
//            added over the warps by the epilogue, which forms dx, ddt, dz.
// dB, dC, dA, dD and ddt_bias are accumulated with atomic adds into buffers the
// host clears first (the order of those fp32 additions is not fixed).
//
// Long rows with few channel groups (forward direction, no sequence starts)
// are cut into segments that form a thread-block cluster, as in the forward
// scan. Phase 1: every segment but the last walks its steps from a zero state
// without storing and publishes its end state and step sum; each segment folds
// the maps of the segments before it, h <- exp(A sum delta) h + h_end, through
// distributed shared memory, and walks again storing its states. Phase 2:
// every segment but the first walks the adjoint alone over its steps from
// zero, in reverse (lam += C gy, lam *= a), and publishes what flows out of
// its first step and its step sum; each segment folds the segments after it
// from the right, X <- X_zero + exp(A sum delta) X (the last from dfinal), and
// runs its reverse walk from that adjoint.

struct BwdParams {
    const void *x, *dt, *B, *C, *z, *dout;
    const float *A, *D, *dt_bias, *h0, *dfinal;
    void *dx, *ddt, *dz;
    float *dA, *dB, *dC, *dD, *ddt_bias, *dh0;
    float4 *ckpt;   // [batch][nsub][S][d_inner] states at sub-chunk starts
    int64_t batch, d_inner, L, N, nsub;
    int softplus;
    int vec;    // io rows 16-byte aligned with L a multiple of the piece
    int vec4;   // dB, dC rows take 16-byte atomic adds (L % 4 == 0, aligned)
    int states_ready;   // the workspace already holds the stored states (written by the forward pass)
    int nseg;           // segments per channel group (a thread-block cluster when > 1; forward direction,
                        // no sequence starts)
    int64_t seg_len;    // steps per segment, a multiple of the chunk length
    const uint8_t *reset;   // (batch, L) sequence starts (RST kernels only)
    int tma;                // the tiles come in through the tensor maps below
    // 3-d maps over (step, row, batch row) as in the forward scan: x, dt, z,
    // dout by channel rows, B, C by state rows
    CUtensorMap tm_x, tm_dt, tm_z, tm_dout, tm_B, tm_C;
};

#define SS_BWD_STAGES 2

template <typename T, int S>
struct BwdShape {
    static constexpr int CH = 32;
    static constexpr int NT = CH * S;
    static constexpr int NS = 4 * S;
    static constexpr int LC = 32;                 // steps per chunk
    static constexpr int HC = 16;                 // steps per recomputed sub-chunk
    static constexpr int NH = LC / HC;
    static constexpr int RL = LC / S;             // prep steps per thread
    static constexpr int RH = HC / S;             // epilogue steps per thread
    static constexpr int STAGES = SS_BWD_STAGES;
    static constexpr int EPP = 16 / (int)sizeof(T);
    static constexpr int PR = LC / EPP;
    static constexpr int ROWB = LC * (int)sizeof(T) + 16;
    static constexpr int RAW_X = CH * ROWB;                     // x, dt, z or dout tile
    static constexpr int RAW_BC = NS * LC * (int)sizeof(T);    // B or C tile
    static constexpr int STAGE_BYTES = 4 * RAW_X + 2 * RAW_BC;
    static constexpr int NPIECE = (4 * CH + 2 * NS) * PR;
    static constexpr int PPT = (NPIECE + NT - 1) / NT;
    static constexpr int PD_BYTES = LC * CH * 8;
    static constexpr int DY_BYTES = LC * CH * 4;
    static constexpr int BC_BYTES = LC * NS * 4;
    static constexpr int PART_BYTES = 3 * S * HC * CH * 4;
    static constexpr int DBC_BYTES = 2 * LC * NS * 4;
    static constexpr int R_BYTES = LC;                          // sequence starts of a chunk
    static constexpr int HX_BYTES = S * CH * 16;                // a segment's end state or adjoint outflow
    static constexpr int SX_BYTES = S * CH * 4;                 // a segment's step sums (per prep thread)
    static constexpr size_t BAR_OFF = (size_t)STAGES * STAGE_BYTES + PD_BYTES + DY_BYTES + 2 * BC_BYTES +
                                      PART_BYTES + DBC_BYTES + R_BYTES + HX_BYTES + SX_BYTES;   // "slot filled" barriers
    static constexpr size_t BYTES = BAR_OFF + 8 * STAGES;
    static_assert(STAGE_BYTES % 128 == 0 && RAW_X % 128 == 0 && RAW_BC % 128 == 0 && BAR_OFF % 8 == 0,
                  "tensor-copy tiles on 128-byte boundaries");
    static_assert(RH >= 2 && RH % 2 == 0, "epilogue runs are processed in pairs");
};

// both halves negated
__device__ __forceinline__ u64 neg2(u64 a) { return a ^ 0x8000000080000000ull; }

// REV: the gradient of the reverse-direction scan (h_t = a_t h_{t+1} + delta_t
// B_t x_t); RST: of the scan with sequence starts (nothing carried across the
// boundary before a marked step). Both are written in walking coordinates: the
// forward walk of phase 1 follows the recurrence (chunk phys1(j), chunk step
// tu(u)), phase 2 walks the other way; the tiles, the stored states (indexed by
// physical 16-step sub-chunk) and every per-step buffer stay in physical order.
// A walking step can be cut before it (RST forward: its start flag) or after
// it (RST reverse: its start flag); a cut zeroes the carried state in the
// walks and the adjoint passed across it.
//
// TMA: the tiles arrive by tensor copies (one thread per chunk, completion on
// the slot's barrier, bounded waits) in an instantiation of their own.
template <typename T, int S, bool REV, bool RST, bool TMA>
__global__ void __launch_bounds__(BwdShape<T, S>::NT, BwdShape<T, S>::NT <= 128 ? 3 : 1)
scan_bwd_kernel(const __grid_constant__ BwdParams p)
{
    using SH = BwdShape<T, S>;
    constexpr int NT = SH::NT, CH = SH::CH, NS = SH::NS, LC = SH::LC, HC = SH::HC, NH = SH::NH;
    constexpr int RL = SH::RL, RH = SH::RH, PR = SH::PR, STAGES = SH::STAGES, EPP = SH::EPP, PPT = SH::PPT;
    constexpr int RW = RL * (int)sizeof(T) / 4;
    constexpr int RHW = RH * (int)sizeof(T) / 4 > 0 ? RH * (int)sizeof(T) / 4 : 1;

    extern __shared__ __align__(128) unsigned char smem_bwd[];
    unsigned char *smem_raw = smem_bwd;
    unsigned char *raw = smem_raw;                                          // [STAGES][x, dt, z, dout, B, C]
    u64 *Pd = reinterpret_cast<u64 *>(smem_raw + STAGES * SH::STAGE_BYTES);  // [LC][CH] (delta, delta x)
    float *DY = reinterpret_cast<float *>(Pd + LC * CH);                    // [LC][CH] gy
    float *Bf = DY + LC * CH;                                               // [LC][NS]
    float *Cf = Bf + LC * NS;                                               // [LC][NS]
    float *Part = Cf + LC * NS;                                             // [3][S][HC/2][CH] step pairs
    float *DBC = Part + 3 * S * HC * CH;                                    // [2][LC][NS]
    unsigned char *Rst = reinterpret_cast<unsigned char *>(DBC + 2 * LC * NS);  // [LC] sequence starts
    float4 *Hx = reinterpret_cast<float4 *>(Rst + SH::R_BYTES);             // [S][CH] published per lane
    float *Sx = reinterpret_cast<float *>(Hx + S * CH);                      // [S][CH] step sums per prep thread
    const uint32_t raw_s = static_cast<uint32_t>(__cvta_generic_to_shared(raw));
    const uint32_t bars_s = raw_s + static_cast<uint32_t>(SH::BAR_OFF);
    if (TMA && (raw_s & 127u) != 0) {   // tensor copies need 128-byte aligned destinations
        if (threadIdx.x == 0)
            atomicOr(&g_fault_flags, kFaultSmemAlign);
        return;
    }

    const int tid = threadIdx.x;
    const int64_t b = blockIdx.y;
    const int nseg = p.nseg;
    const int seg = static_cast<int>(blockIdx.x % static_cast<unsigned>(nseg));
    const int64_t d0 = static_cast<int64_t>(blockIdx.x / static_cast<unsigned>(nseg)) * CH;
    const int64_t L = p.L, N = p.N, Dn = p.d_inner;
    const bool vec = p.vec != 0;
    // this segment's chunks [c_lo, c_hi) (the whole row when nseg = 1)
    const int64_t seg_chunks = p.seg_len / LC;
    const int64_t c_lo = seg * seg_chunks;
    const int64_t c_hi = ((L + LC - 1) / LC < c_lo + seg_chunks) ? (L + LC - 1) / LC : c_lo + seg_chunks;
    const int64_t nchunks = c_hi - c_lo;
    // physical chunk of the j-th chunk of the forward walk (phase 1) and of the
    // reverse walk (phase 2); physical step in a chunk of walking step u
    auto phys1 = [&](int64_t j) -> int64_t { return REV ? c_hi - 1 - j : c_lo + j; };
    auto phys2 = [&](int64_t j) -> int64_t { return REV ? c_lo + j : c_hi - 1 - j; };
    auto tu = [](int u) { return REV ? LC - 1 - u : u; };

    const int cs = tid % CH;     // scan role: lane = channel, warp = state group
    const int q = tid / CH;
    const int lane = tid & 31;
    const bool act_s = d0 + cs < Dn;
    const int64_t ds = act_s ? d0 + cs : 0;
    const int ce = tid % CH;     // prep/epilogue role: channel ce, run re
    const int re = tid / CH;
    const bool act_e = d0 + ce < Dn;
    const int64_t de = act_e ? d0 + ce : 0;

    const float biasv = (p.dt_bias && act_e) ? __ldg(p.dt_bias + de) : 0.0f;
    const u64 bias2 = splat(biasv);
    const float Dv = (p.D && act_e) ? __ldg(p.D + de) : 0.0f;
    const bool gate = p.z != nullptr;

    float A2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int n = 4 * q + e;
        A2[e] = (n < N) ? __ldg(p.A + ds * N + n) * kLog2e : 0.0f;
    }
    const u64 A01 = pk(A2[0], A2[1]);
    const u64 A23 = pk(A2[2], A2[3]);

    // raw pieces this thread copies (x, dt, z, dout rows, then B, C rows)
    const T *src[PPT];
    uint32_t soff[PPT];
    int poff[PPT];
    bool p2_only[PPT];   // needed by phase 2 only (z, dout, C)
#pragma unroll
    for (int u = 0; u < PPT; ++u) {
        const int pi = tid + u * NT;
        int r, pc;
        const T *base;
        uint32_t off;
        bool ok = pi < SH::NPIECE;
        if (pi < 4 * CH * PR) {
            const int tensor = pi / (CH * PR);
            r = (pi % (CH * PR)) / PR;
            pc = pi % PR;
            const void *gv = tensor == 0 ? p.x : (tensor == 1 ? p.dt : (tensor == 2 ? p.z : p.dout));
            const T *g = static_cast<const T *>(gv);
            ok = ok && d0 + r < Dn && g != nullptr;
            base = ok ? g + (b * Dn + d0 + r) * L : static_cast<const T *>(p.x);
            off = tensor * SH::RAW_X + r * SH::ROWB;
            p2_only[u] = tensor >= 2;
        } else {
            const int v = pi - 4 * CH * PR;
            const int m = v / (NS * PR);
            r = (v % (NS * PR)) / PR;
            pc = v % PR;
            ok = ok && r < N;
            base = static_cast<const T *>(m == 0 ? p.B : p.C) + (b * N + (ok ? r : 0)) * L;
            off = 4 * SH::RAW_X + m * SH::RAW_BC + r * LC * (int)sizeof(T);
            p2_only[u] = m == 1;
        }
        src[u] = base;
        soff[u] = off + pc * 16;
        poff[u] = ok ? pc * EPP : (1 << 30);
    }

    // copy the raw pieces of chunk k into ring slot `slot`
    // tensor copies: copies issued into and waits completed on each of the two
    // slots (the n-th completion of a slot's barrier has parity n & 1)
    static_assert(STAGES == 2, "two slots");
    int iss0 = 0, iss1 = 0, wt0 = 0, wt1 = 0;
    bool aborted = false;
    if (TMA) {
        if (tid == 0) {
            for (int s2 = 0; s2 < STAGES; ++s2)
                mbar_init(bars_s + 8u * s2, 1);
            mbar_fence_init();
        }
        __syncthreads();
    }
    auto wait_slot = [&](int slot) {
        if constexpr (TMA) {
            if (!aborted)
                aborted = !mbar_wait(bars_s + 8u * slot, static_cast<uint32_t>((slot ? wt1 : wt0) & 1));
            if (!aborted) {
                if (slot)
                    ++wt1;
                else
                    ++wt0;
            }
        }
    };

    auto stage_in = [&](int64_t k, int slot, bool phase2) {
        const uint32_t st = raw_s + static_cast<uint32_t>(slot * SH::STAGE_BYTES);
        const int64_t t1 = k * LC;
        if constexpr (TMA) {
            if (tid == 0 && !aborted) {
                const uint32_t bar = bars_s + 8u * slot;
                const bool zz = phase2 && gate;
                mbar_expect_tx(bar, 2 * SH::RAW_X + SH::RAW_BC + (zz ? SH::RAW_X : 0) +
                                        (phase2 ? SH::RAW_X + SH::RAW_BC : 0));
                const int c0 = static_cast<int>(t1), cd = static_cast<int>(d0), cb = static_cast<int>(b);
                tma_load_3d(st, &p.tm_x, bar, c0, cd, cb);
                tma_load_3d(st + SH::RAW_X, &p.tm_dt, bar, c0, cd, cb);
                if (zz)
                    tma_load_3d(st + 2 * SH::RAW_X, &p.tm_z, bar, c0, cd, cb);
                if (phase2)
                    tma_load_3d(st + 3 * SH::RAW_X, &p.tm_dout, bar, c0, cd, cb);
                tma_load_3d(st + 4 * SH::RAW_X, &p.tm_B, bar, c0, 0, cb);
                if (phase2)
                    tma_load_3d(st + 4 * SH::RAW_X + SH::RAW_BC, &p.tm_C, bar, c0, 0, cb);
                if (slot)
                    ++iss1;
                else
                    ++iss0;
            }
            return;
        }
        const int rem = static_cast<int>(L - t1 < (1 << 29) ? L - t1 : (1 << 29));
#pragma unroll
        for (int u = 0; u < PPT; ++u) {
            if (tid + u * NT >= SH::NPIECE)
                break;
            if (!phase2 && p2_only[u])
                continue;
            const int left = rem - poff[u];
            const int nb = left >= EPP ? 16 : (left > 0 ? left * (int)sizeof(T) : 0);
            const T *g = src[u] + (nb > 0 ? t1 + poff[u] : 0);
            if (vec) {
                cp_async16(st + soff[u], g, nb);
            } else {
                unsigned char *dst = raw + slot * SH::STAGE_BYTES + soff[u];
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

    // raw B (and C) of the chunk in `slot` -> fp32 [t][n]
    auto convert_bc = [&](int slot, bool phase2) {
        const unsigned char *st = raw + slot * SH::STAGE_BYTES + 4 * SH::RAW_X;
        const int items = (phase2 ? 2 : 1) * LC * S;
        for (int w = tid; w < items; w += NT) {
            const int m = w / (LC * S);
            const int t = (w % (LC * S)) / S;
            const int g = w % S;
            const T *srcm = reinterpret_cast<const T *>(st + m * SH::RAW_BC);
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if constexpr (sizeof(T) == 4)
                    v[e] = srcm[(4 * g + e) * LC + t];
                else
                    v[e] = __uint_as_float(static_cast<uint32_t>(
                                               reinterpret_cast<const unsigned short *>(srcm)[(4 * g + e) * LC + t])
                                           << 16);
            }
            *reinterpret_cast<float4 *>((m == 0 ? Bf : Cf) + t * NS + 4 * g) = make_float4(v[0], v[1], v[2], v[3]);
        }
    };

    // this thread's compensated sum of the steps it prepares while `summing`
    // (the segment folds)
    float ssum = 0.0f, scomp = 0.0f;
    bool summing = false;
    auto kahan = [&](float v) {
        const float yv = v - scomp;
        const float tv = ssum + yv;
        scomp = (tv - ssum) - yv;
        ssum = tv;
    };

    // delta, delta*x (and, in phase 2, gy) of this thread's steps of chunk k
    auto prep = [&](int64_t k, int slot, bool phase2) {
        const unsigned char *st = raw + slot * SH::STAGE_BYTES;
        uint32_t xw[RW], dw[RW], zw[RW], gw[RW];
        read_run_raw<T, RL>(st + ce * SH::ROWB, re * RL, xw);
        read_run_raw<T, RL>(st + SH::RAW_X + ce * SH::ROWB, re * RL, dw);
        if (phase2) {
            read_run_raw<T, RL>(st + 3 * SH::RAW_X + ce * SH::ROWB, re * RL, gw);
            if (gate)
                read_run_raw<T, RL>(st + 2 * SH::RAW_X + ce * SH::ROWB, re * RL, zw);
        }
        const int64_t left64 = L - (k * LC + re * RL);
        const int lim = act_e ? static_cast<int>(left64 < RL ? left64 : RL) : 0;
        if (RST && tid < LC) {
            const int64_t tt = k * LC + tid;
            Rst[tid] = (tt < L && p.reset[b * L + tt]) ? 1 : 0;
        }
#pragma unroll
        for (int i = 0; i < RL; i += 2) {
            const u64 xx = word_pair<T>(xw, i);
            const u64 u = add2(word_pair<T>(dw, i), bias2);
            const u64 s2 = p.softplus ? softplus2(u) : u;
            float s0, s1;
            upk(s2, s0, s1);
            s0 = i < lim ? s0 : 0.0f;
            s1 = i + 1 < lim ? s1 : 0.0f;
            if (summing) {
                kahan(s0);
                kahan(s1);
            }
            float sx0, sx1;
            upk(mul2(pk(s0, s1), xx), sx0, sx1);
            Pd[(re * RL + i) * CH + ce] = pk(s0, sx0);
            Pd[(re * RL + i + 1) * CH + ce] = pk(s1, sx1);
            if (phase2) {
                u64 gy = word_pair<T>(gw, i);
                if (gate)
                    gy = mul2(gy, silu2(word_pair<T>(zw, i)));
                float g0, g1;
                upk(gy, g0, g1);
                DY[(re * RL + i) * CH + ce] = i < lim ? g0 : 0.0f;
                DY[(re * RL + i + 1) * CH + ce] = i + 1 < lim ? g1 : 0.0f;
            }
        }
    };

    const float *Bq_s = Bf + 4 * q;
    const float *Cq_s = Cf + 4 * q;
    float4 *ck = p.ckpt + (b * p.nsub * S + q) * Dn + ds;   // + s * S * Dn for sub-chunk s
    const int64_t ckstride = static_cast<int64_t>(S) * Dn;

    // ---- phase 1: forward, storing the state at every sub-chunk start (skipped
    // when the forward pass has stored them)
    u64 h01 = 0, h23 = 0;
    if (p.h0 && act_s) {
        const float *hp = p.h0 + (b * Dn + ds) * N;
        float hv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            hv[e] = (4 * q + e < N) ? hp[4 * q + e] : 0.0f;
        h01 = pk(hv[0], hv[1]);
        h23 = pk(hv[2], hv[3]);
    }
    // phase 1 over this segment's chunks from the state in (h01, h23); with
    // `store`, the state at every sub-chunk start goes to the workspace
    auto walk1 = [&](bool store) {
#pragma unroll
        for (int s = 0; s < STAGES - 1; ++s)
            if (s < nchunks)
                stage_in(phys1(s), s, false);
            else
                cp_async_commit();
        cp_async_wait<STAGES - 2>();
        wait_slot(0);
        __syncthreads();
        prep(phys1(0), 0, false);
        convert_bc(0, false);
        __syncthreads();
        for (int64_t j = 0; j < nchunks; ++j) {
            const int64_t k = phys1(j);
            if (j + STAGES - 1 < nchunks)
                stage_in(phys1(j + STAGES - 1), static_cast<int>((j + STAGES - 1) % STAGES), false);
            else
                cp_async_commit();
#pragma unroll
            for (int hw = 0; hw < NH; ++hw) {
                const int64_t s = k * NH + (REV ? NH - 1 - hw : hw);   // physical sub-chunk
                if (store && act_s && s < p.nsub) {
                    float a0, a1, a2, a3;
                    upk(h01, a0, a1);
                    upk(h23, a2, a3);
                    ck[s * ckstride] = make_float4(a0, a1, a2, a3);
                }
#pragma unroll 4
                for (int i = 0; i < HC; ++i) {
                    const int t = tu(hw * HC + i);
                    if (RST && !REV && Rst[t]) {   // a sequence starts at t: nothing carries in
                        h01 = 0;
                        h23 = 0;
                    }
                    float dl, dx;
                    upk(Pd[t * CH + cs], dl, dx);
                    const ulonglong2 Bq = *reinterpret_cast<const ulonglong2 *>(Bq_s + t * NS);
                    const u64 dd = splat(dl), xx = splat(dx);
                    h01 = fma2(ex2_2(mul2(dd, A01)), h01, mul2(xx, Bq.x));
                    h23 = fma2(ex2_2(mul2(dd, A23)), h23, mul2(xx, Bq.y));
                    if (RST && REV && Rst[t]) {    // a sequence starts at t: nothing carries to t-1
                        h01 = 0;
                        h23 = 0;
                    }
                }
            }
            cp_async_wait<STAGES - 2>();
            if (j + 1 < nchunks)
                wait_slot(static_cast<int>((j + 1) % STAGES));
            __syncthreads();
            if (j + 1 < nchunks) {
                prep(phys1(j + 1), static_cast<int>((j + 1) % STAGES), false);
                convert_bc(static_cast<int>((j + 1) % STAGES), false);
            }
            __syncthreads();
        }
        cp_async_wait<0>();
        __syncthreads();
    };

    // the lane's four values as one word for the peers of its cluster, and back
    auto publish = [&](u64 v01, u64 v23) {
        float a0, a1, a2, a3;
        upk(v01, a0, a1);
        upk(v23, a2, a3);
        Hx[q * CH + cs] = make_float4(a0, a1, a2, a3);
        Sx[re * CH + ce] = ssum;
    };
    // (segment i's value for this lane, exp(A * segment i's step sum)), read through distributed shared memory
    auto peer = [&](cg::cluster_group &cl, int i, u64 &v01, u64 &v23, u64 &a01, u64 &a23) {
        const float4 *ph = cl.map_shared_rank(Hx, i);
        const float *ps = cl.map_shared_rank(Sx, i);
        float tot = 0.0f;
#pragma unroll
        for (int r = 0; r < S; ++r)
            tot += ps[r * CH + cs];
        const float4 v = ph[q * CH + cs];
        v01 = pk(v.x, v.y);
        v23 = pk(v.z, v.w);
        a01 = ex2_2(mul2(splat(tot), A01));
        a23 = ex2_2(mul2(splat(tot), A23));
    };

    if (!p.states_ready) {
        if (nseg > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            const u64 g01 = h01, g23 = h23;   // the state entering segment 0
            if (seg != nseg - 1) {            // the end state of this segment from a zero start
                h01 = 0;
                h23 = 0;
                ssum = scomp = 0.0f;
                summing = true;
                walk1(false);
                summing = false;
            }
            publish(h01, h23);
            cluster.sync();
            u64 f01 = g01, f23 = g23;
            for (int i = 0; i < seg; ++i) {   // h <- exp(A sum delta) h + h_end over the segments before
                u64 e01, e23, a01, a23;
                peer(cluster, i, e01, e23, a01, a23);
                f01 = fma2(a01, f01, e01);
                f23 = fma2(a23, f23, e23);
            }
            cluster.sync();   // the peers have read this CTA's values
            h01 = f01;
            h23 = f23;
        }
        walk1(true);
    }

    // ---- phase 2: reverse
    u64 lam01 = 0, lam23 = 0, dA01 = 0, dA23 = 0;
    if (p.dfinal && act_s) {
        const float *fp = p.dfinal + (b * Dn + ds) * N;
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            v[e] = (4 * q + e < N) ? fp[4 * q + e] : 0.0f;
        lam01 = pk(v[0], v[1]);
        lam23 = pk(v[2], v[3]);
    }
    float dD_acc = 0.0f, db_acc = 0.0f;
    T *dxr = static_cast<T *>(p.dx) + (b * Dn + de) * L;
    T *ddtr = static_cast<T *>(p.ddt) + (b * Dn + de) * L;
    T *dzr = gate && p.dz ? static_cast<T *>(p.dz) + (b * Dn + de) * L : nullptr;
    const u64 ln2_2 = splat(0.6931471805599453f);

    if (nseg > 1) {
        // the adjoint of this segment alone (zero inflow), walked in reverse over
        // its chunks: lam += C gy, lam *= a; what flows out of its first step
        auto walk2pre = [&]() {
#pragma unroll 1
            for (int s2 = 0; s2 < STAGES - 1; ++s2)
                if (s2 < nchunks)
                    stage_in(phys2(s2), s2, true);
                else
                    cp_async_commit();
            cp_async_wait<STAGES - 2>();
            wait_slot(0);
            __syncthreads();
            prep(phys2(0), 0, true);
            convert_bc(0, true);
            __syncthreads();
#pragma unroll 1
            for (int64_t j = 0; j < nchunks; ++j) {
                if (j + STAGES - 1 < nchunks)
                    stage_in(phys2(j + STAGES - 1), static_cast<int>((j + STAGES - 1) % STAGES), true);
                else
                    cp_async_commit();
#pragma unroll 4
                for (int u = 0; u < LC; ++u) {
                    const int t = LC - 1 - u;
                    float dl, dx;
                    upk(Pd[t * CH + cs], dl, dx);
                    const u64 gy2 = splat(DY[t * CH + cs]);
                    const ulonglong2 Cq = *reinterpret_cast<const ulonglong2 *>(Cq_s + t * NS);
                    const u64 dd = splat(dl);
                    lam01 = fma2(Cq.x, gy2, lam01);
                    lam23 = fma2(Cq.y, gy2, lam23);
                    lam01 = mul2(lam01, ex2_2(mul2(dd, A01)));
                    lam23 = mul2(lam23, ex2_2(mul2(dd, A23)));
                }
                cp_async_wait<STAGES - 2>();
                if (j + 1 < nchunks)
                    wait_slot(static_cast<int>((j + 1) % STAGES));
                __syncthreads();
                if (j + 1 < nchunks) {
                    const int nslot = static_cast<int>((j + 1) % STAGES);
                    prep(phys2(j + 1), nslot, true);
                    convert_bc(nslot, true);
                }
                __syncthreads();
            }
            cp_async_wait<0>();
            __syncthreads();
        };
        cg::cluster_group cluster = cg::this_cluster();
        const u64 l01 = lam01, l23 = lam23;   // dfinal, the inflow of the last segment
        if (seg != 0) {
            lam01 = 0;
            lam23 = 0;
            ssum = scomp = 0.0f;
            summing = true;
            walk2pre();
            summing = false;
        }
        publish(lam01, lam23);
        cluster.sync();
        u64 f01 = l01, f23 = l23;
        for (int i = nseg - 1; i > seg; --i) {   // X <- X_zero + exp(A sum delta) X over the segments after
            u64 x01, x23, a01, a23;
            peer(cluster, i, x01, x23, a01, a23);
            f01 = fma2(a01, f01, x01);
            f23 = fma2(a23, f23, x23);
        }
        cluster.sync();   // the peers have read this CTA's values
        lam01 = f01;
        lam23 = f23;
    }

    float4 ck_cur = make_float4(0.f, 0.f, 0.f, 0.f);   // stored state of the sub-chunk processed next
    if (act_s) {   // the last sub-chunk of the forward walk comes first
        const int64_t s_end = p.nsub < c_hi * NH ? p.nsub : c_hi * NH;   // past this segment's last sub-chunk
        ck_cur = ck[(REV ? c_lo * NH : s_end - 1) * ckstride];
    }

    // chunk j of the reverse walk is physical chunk phys2(j)
#pragma unroll 1
    for (int s = 0; s < STAGES - 1; ++s)
        if (s < nchunks)
            stage_in(phys2(s), s, true);
        else
            cp_async_commit();
    cp_async_wait<STAGES - 2>();
    wait_slot(0);
    __syncthreads();
    prep(phys2(0), 0, true);
    convert_bc(0, true);
    __syncthreads();

#pragma unroll 1
    for (int64_t j = 0; j < nchunks; ++j) {
        const int64_t k = phys2(j);
        const int slot = static_cast<int>(j % STAGES);
        if (j + STAGES - 1 < nchunks)
            stage_in(phys2(j + STAGES - 1), static_cast<int>((j + STAGES - 1) % STAGES), true);
        else
            cp_async_commit();

#pragma unroll 1
        for (int hh = NH - 1; hh >= 0; --hh) {   // walking sub-chunk hh, physical ph
            const int ph = REV ? NH - 1 - hh : hh;
            const int64_t s = k * NH + ph;
            if (s < p.nsub) {
                // the stored state of the sub-chunk walked before this one is fetched while this one runs
                const int64_t s_next = REV ? s + 1 : s - 1;
                float4 ck_next = make_float4(0.f, 0.f, 0.f, 0.f);
                if (act_s && s_next >= 0 && s_next < p.nsub)
                    ck_next = ck[s_next * ckstride];
                // recompute the HC states of this sub-chunk from its stored start
                u64 H01[HC], H23[HC];
                u64 S01, S23;   // the state before the sub-chunk
                {
                    const float4 c4 = ck_cur;
                    ck_cur = ck_next;
                    S01 = pk(c4.x, c4.y);
                    S23 = pk(c4.z, c4.w);
                    u64 g01 = S01, g23 = S23;
#pragma unroll
                    for (int i = 0; i < HC; ++i) {
                        const int t = tu(hh * HC + i);
                        if (RST && !REV && Rst[t]) {
                            g01 = 0;
                            g23 = 0;
                        }
                        float dl, dx;
                        upk(Pd[t * CH + cs], dl, dx);
                        const ulonglong2 Bq = *reinterpret_cast<const ulonglong2 *>(Bq_s + t * NS);
                        const u64 dd = splat(dl), xx = splat(dx);
                        g01 = fma2(ex2_2(mul2(dd, A01)), g01, mul2(xx, Bq.x));
                        g23 = fma2(ex2_2(mul2(dd, A23)), g23, mul2(xx, Bq.y));
                        H01[i] = g01;   // the step's output, before a cut after it
                        H23[i] = g23;
                        if (RST && REV && Rst[t]) {
                            g01 = 0;
                            g23 = 0;
                        }
                    }
                }
                // adjoint recurrence backwards over the sub-chunk, two steps per round
                // step i: lam += C gy; v = (lam dx, gy h) for the channel sums; the
                // state sums for the epilogue; then lam *= a_i for step i-1
                auto step = [&](int i, float *v, float &r_, float &pa, float &yy) {
                    const int t = tu(hh * HC + i);
                    if (RST && REV && Rst[t]) {   // cut after this step: nothing flows back from the later ones
                        lam01 = 0;
                        lam23 = 0;
                    }
                    float dl, dx;
                    upk(Pd[t * CH + cs], dl, dx);
                    const float gy = DY[t * CH + cs];
                    const ulonglong2 Bq = *reinterpret_cast<const ulonglong2 *>(Bq_s + t * NS);
                    const ulonglong2 Cq = *reinterpret_cast<const ulonglong2 *>(Cq_s + t * NS);
                    const u64 gy2 = splat(gy), dx2 = splat(dx), dd = splat(dl);
                    lam01 = fma2(Cq.x, gy2, lam01);
                    lam23 = fma2(Cq.y, gy2, lam23);
                    upk(mul2(lam01, dx2), v[0], v[1]);
                    upk(mul2(lam23, dx2), v[2], v[3]);
                    upk(mul2(gy2, H01[i]), v[4], v[5]);
                    upk(mul2(gy2, H23[i]), v[6], v[7]);
                    const u64 a01 = ex2_2(mul2(dd, A01));
                    const u64 a23 = ex2_2(mul2(dd, A23));
                    // the state entering the step (zero across a cut)
                    const bool cut_in = RST && ((!REV && Rst[t]) || (REV && i > 0 && Rst[tu(hh * HC + (i > 0 ? i - 1 : 0))]));
                    const u64 hin01 = cut_in ? 0 : (i > 0 ? H01[i > 0 ? i - 1 : 0] : S01);
                    const u64 hin23 = cut_in ? 0 : (i > 0 ? H23[i > 0 ? i - 1 : 0] : S23);
                    const u64 p01 = mul2(lam01, mul2(a01, hin01));   // lam a_t h_in
                    const u64 p23 = mul2(lam23, mul2(a23, hin23));
                    dA01 = fma2(p01, dd, dA01);
                    dA23 = fma2(p23, dd, dA23);
                    r_ = hsum(fma2(lam23, Bq.y, mul2(lam01, Bq.x)));
                    pa = hsum(fma2(p23, A23, mul2(p01, A01)));
                    yy = hsum(fma2(Cq.y, H23[i], mul2(Cq.x, H01[i])));
                    lam01 = mul2(lam01, a01);
                    lam23 = mul2(lam23, a23);
                    if (RST && !REV && Rst[t]) {   // cut before this step: nothing flows to the earlier ones
                        lam01 = 0;
                        lam23 = 0;
                    }
                };
                const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
                for (int i = HC - 1; i >= 1; i -= 2) {
                    float val[16];   // [0, 8): step i, [8, 16): step i-1
                    float r1, pa1, y1, r0, pa0, y0;
                    step(i, val, r1, pa1, y1);
                    step(i - 1, val + 8, r0, pa0, y0);
                    // the pair of physical steps (2m, 2m+1) of the sub-chunk: walking (i-1, i), or (i, i-1) when reversed
                    float2 *pp = reinterpret_cast<float2 *>(Part) + (q * (HC / 2) + (REV ? (HC - 1 - i) >> 1 : i >> 1)) * CH + cs;
                    pp[0] = REV ? make_float2(r1, r0) : make_float2(r0, r1);
                    pp[S * (HC / 2) * CH] = REV ? make_float2(pa1, pa0) : make_float2(pa0, pa1);
                    pp[2 * S * (HC / 2) * CH] = REV ? make_float2(y1, y0) : make_float2(y0, y1);
                    // transposing butterfly: value (lane >> 1) & 15 ends summed over the warp
                    float w[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float send = b4 ? val[e] : val[e + 8];
                        const float keep = b4 ? val[e + 8] : val[e];
                        w[e] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                    }
                    float u4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float send = b3 ? w[e] : w[e + 4];
                        const float keep = b3 ? w[e + 4] : w[e];
                        u4[e] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                    }
                    float u2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float send = b2 ? u4[e] : u4[e + 2];
                        const float keep = b2 ? u4[e + 2] : u4[e];
                        u2[e] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                    }
                    const float send = b1 ? u2[0] : u2[1];
                    const float keep = b1 ? u2[1] : u2[0];
                    float sum = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                    if ((lane & 1) == 0) {
                        const int kk = (lane >> 1) & 15;   // < 8: step i, else step i-1
                        const int kv = kk & 7;             // 0..3: dB of state 4q+kv, 4..7: dC of 4q+kv-4
                        const int t = tu(hh * HC + i - (kk >> 3));
                        DBC[((kv >> 2) * LC + t) * NS + 4 * q + (kv & 3)] = sum;
                    }
                }
            }
            __syncthreads();
            // ---- epilogue of the sub-chunk: steps hh*HC + re*RH .. + RH - 1
            if (s < p.nsub) {
                const unsigned char *st = raw + slot * SH::STAGE_BYTES;
                const int off = ph * HC + re * RH;
                uint32_t xw[RHW], dw[RHW], zw[RHW], gw[RHW];
                read_run_raw<T, RH>(st + ce * SH::ROWB, off, xw);
                read_run_raw<T, RH>(st + SH::RAW_X + ce * SH::ROWB, off, dw);
                read_run_raw<T, RH>(st + 3 * SH::RAW_X + ce * SH::ROWB, off, gw);
                if (gate)
                    read_run_raw<T, RH>(st + 2 * SH::RAW_X + ce * SH::ROWB, off, zw);
                float o_dx[RH], o_dt[RH], o_dz[RH];
                const int64_t tg0 = k * LC + off;
                const int lim = act_e ? static_cast<int>(L - tg0 < RH ? L - tg0 : RH) : 0;
#pragma unroll
                for (int i = 0; i < RH; i += 2) {
                    u64 r2 = 0, pa2 = 0, y2 = 0;
                    const u64 *pp = reinterpret_cast<const u64 *>(Part) + ((re * RH + i) >> 1) * CH + ce;
#pragma unroll
                    for (int qq = 0; qq < S; ++qq) {
                        r2 = add2(r2, pp[(0 * S + qq) * (HC / 2) * CH]);
                        pa2 = add2(pa2, pp[(1 * S + qq) * (HC / 2) * CH]);
                        y2 = add2(y2, pp[(2 * S + qq) * (HC / 2) * CH]);
                    }
                    const int tl = off + i;   // step within the chunk
                    float dl0, dx0_, dl1, dx1_;
                    upk(Pd[tl * CH + ce], dl0, dx0_);
                    upk(Pd[(tl + 1) * CH + ce], dl1, dx1_);
                    const u64 dl2 = pk(dl0, dl1);
                    const u64 gy2 = pk(DY[tl * CH + ce], DY[(tl + 1) * CH + ce]);
                    const u64 xx = word_pair<T>(xw, i);
                    const u64 D2 = splat(Dv);
                    // dx = D gy + delta r ; ddelta = ln2 * pa + x r
                    const u64 gdx = fma2(dl2, r2, mul2(D2, gy2));
                    u64 gdl = fma2(xx, r2, mul2(ln2_2, pa2));
                    if (p.softplus) {
                        const u64 v2 = add2(word_pair<T>(dw, i), bias2);
                        // sigmoid(v) = 1 / (1 + 2^(-v log2 e))
                        const u64 sg = rcp_2(add2(splat(1.0f), ex2_2(mul2(v2, splat(-kLog2e)))));
                        gdl = mul2(gdl, sg);
                    }
                    upk(gdx, o_dx[i], o_dx[i + 1]);
                    upk(gdl, o_dt[i], o_dt[i + 1]);
                    if (gate) {
                        const u64 zz = word_pair<T>(zw, i);
                        const u64 go = word_pair<T>(gw, i);
                        const u64 yf = fma2(D2, xx, y2);   // pre-gate output
                        const u64 sz = rcp_2(add2(splat(1.0f), ex2_2(mul2(zz, splat(-kLog2e)))));
                        // g'(z) = s (1 + z (1 - s))
                        const u64 one = splat(1.0f);
                        const u64 gp = mul2(sz, fma2(zz, fma2(neg2(sz), one, one), one));
                        upk(mul2(mul2(go, yf), gp), o_dz[i], o_dz[i + 1]);
                    }
                    float gy0, gy1, x0, x1;
                    upk(gy2, gy0, gy1);
                    upk(xx, x0, x1);
                    if (i < lim) {
                        dD_acc = fmaf(gy0, x0, dD_acc);
                        db_acc += o_dt[i];
                    }
                    if (i + 1 < lim) {
                        dD_acc = fmaf(gy1, x1, dD_acc);
                        db_acc += o_dt[i + 1];
                    }
                }
                if (act_e) {
                    write_run<T, RH>(dxr, tg0, L, vec, o_dx);
                    write_run<T, RH>(ddtr, tg0, L, vec, o_dt);
                    if (dzr)
                        write_run<T, RH>(dzr, tg0, L, vec, o_dz);
                }
            }
            __syncthreads();   // Part is reused by the next sub-chunk
        }

        // ---- dB, dC of chunk k: add the CTA's channel sums into global memory
        {
            const int64_t t0 = k * LC;
            constexpr int ITEMS = 2 * NS * (LC / 4);
            for (int w = tid; w < ITEMS; w += NT) {
                const int m = w / (NS * (LC / 4));
                const int n = (w % (NS * (LC / 4))) / (LC / 4);
                const int t4 = w % (LC / 4);
                if (n >= N)
                    continue;
                const float *sp = DBC + (m * LC + 4 * t4) * NS + n;
                float *g = (m == 0 ? p.dB : p.dC) + (b * N + n) * L + t0 + 4 * t4;
                const int64_t left = L - (t0 + 4 * t4);
                if (p.vec4 && left >= 4) {
                    atomicAdd(reinterpret_cast<float4 *>(g), make_float4(sp[0], sp[NS], sp[2 * NS], sp[3 * NS]));
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (e < left)
                            atomicAdd(g + e, sp[e * NS]);
                }
            }
        }

        cp_async_wait<STAGES - 2>();
        if (j + 1 < nchunks)
            wait_slot(static_cast<int>((j + 1) % STAGES));
        __syncthreads();
        if (j + 1 < nchunks) {
            const int nslot = static_cast<int>((j + 1) % STAGES);
            prep(phys2(j + 1), nslot, true);
            convert_bc(nslot, true);
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // ---- per-channel and per-(channel, state) sums
    if (act_s) {
        float v[4];
        upk(dA01, v[0], v[1]);
        upk(dA23, v[2], v[3]);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (4 * q + e < N)
                atomicAdd(p.dA + ds * N + 4 * q + e, v[e]);
        if (p.dh0 && seg == 0) {
            float l[4];
            upk(lam01, l[0], l[1]);
            upk(lam23, l[2], l[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (4 * q + e < N)
                    p.dh0[(b * Dn + ds) * N + 4 * q + e] = l[e];
        }
    }
    if (act_e) {
        if (p.dD)
            atomicAdd(p.dD + de, dD_acc);
        if (p.ddt_bias)
            atomicAdd(p.ddt_bias + de, db_acc);
    }
    if (TMA && tid == 0) {   // after a wait gave up: let the copies issued since land (each wait bounded)
        for (int n = wt0; n < iss0; ++n)
            mbar_wait(bars_s, static_cast<uint32_t>(n & 1));
        for (int n = wt1; n < iss1; ++n)
            mbar_wait(bars_s + 8u, static_cast<uint32_t>(n & 1));
    }
}

// ------------------------------------------------------------------ backward host side

template <typename T, int S, bool REV, bool RST>
ss_status launch_bwd(const BwdParams &p0, cudaStream_t stream, int sms)
{
    using SH = BwdShape<T, S>;
    auto kernel = p0.tma ? scan_bwd_kernel<T, S, REV, RST, true> : scan_bwd_kernel<T, S, REV, RST, false>;
    const size_t smem = SH::BYTES;
    if (smem > 48u * 1024u) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SS_ERR_LAUNCH, "cudaFuncSetAttribute failed: %s", cudaGetErrorString(e));
        }
    }
    BwdParams p = p0;
    const int64_t gpr = (p.d_inner + SH::CH - 1) / SH::CH;
    const int64_t nchunks = (p.L + SH::LC - 1) / SH::LC;
    // segments (thread-block clusters) for long rows with few channel groups:
    // forward direction without sequence starts only
    int nseg = 1;
    if (!REV && !RST) {
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, SH::NT, smem) != cudaSuccess || occ < 1) {
            cudaGetLastError();
            occ = 1;
        }
        nseg = pick_segments(gpr * p.batch, p.L, SH::LC, static_cast<int64_t>(sms) * occ, "SS_BWD_SEGMENTS");
    }
    int64_t seg_chunks = (nchunks + nseg - 1) / nseg;
    nseg = static_cast<int>((nchunks + seg_chunks - 1) / seg_chunks);
    if (gpr * nseg > 0x7fffffff || p.batch > 65535)
        return fail(SS_ERR_DIM, "grid too large: %lld channel blocks x %lld batch rows", (long long)(gpr * nseg),
                    (long long)p.batch);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(gpr * nseg), static_cast<unsigned>(p.batch));
    cfg.blockDim = dim3(SH::NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    if (nseg > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = nseg;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();   // a cluster of this size cannot be placed: do not split
            nseg = 1;
            seg_chunks = nchunks;
            cfg.gridDim.x = static_cast<unsigned>(gpr);
            cfg.attrs = nullptr;
            cfg.numAttrs = 0;
        }
    }
    p.nseg = nseg;
    p.seg_len = seg_chunks * SH::LC;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e == cudaSuccess)
        e = cudaGetLastError();
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SS_ERR_LAUNCH, "backward kernel launch failed: %s", cudaGetErrorString(e));
    }
    return SS_OK;
}

// The backward's tile maps: the forward scan's boxes, plus dout (SS_SCAN_TMA=0
// keeps the cp.async pieces).
template <typename T>
bool encode_bwd_maps(BwdParams &p)
{
    const char *env = getenv("SS_SCAN_TMA");
    if (env && strcmp(env, "0") == 0)
        return false;
    using SH = BwdShape<T, 1>;   // CH, LC and the raw row do not depend on the state split
    const uint32_t ns = static_cast<uint32_t>(4 * bwd_groups(p.N));
    const uint32_t row_t = SH::ROWB / sizeof(T);
    bool ok = encode_rows_map<T>(&p.tm_x, p.x, p.L, p.d_inner, p.batch, row_t, SH::CH) &&
              encode_rows_map<T>(&p.tm_dt, p.dt, p.L, p.d_inner, p.batch, row_t, SH::CH) &&
              encode_rows_map<T>(&p.tm_dout, p.dout, p.L, p.d_inner, p.batch, row_t, SH::CH) &&
              encode_rows_map<T>(&p.tm_B, p.B, p.L, p.N, p.batch, SH::LC, ns) &&
              encode_rows_map<T>(&p.tm_C, p.C, p.L, p.N, p.batch, SH::LC, ns);
    if (ok && p.z)
        ok = encode_rows_map<T>(&p.tm_z, p.z, p.L, p.d_inner, p.batch, row_t, SH::CH);
    return ok;
}

template <typename T, int S>
ss_status dispatch_bwd(const BwdParams &p, bool reverse, cudaStream_t stream, int sms)
{
    const bool rst = p.reset != nullptr;
    if (!reverse && !rst) return launch_bwd<T, S, false, false>(p, stream, sms);
    if (!reverse) return launch_bwd<T, S, false, true>(p, stream, sms);
    if (!rst) return launch_bwd<T, S, true, false>(p, stream, sms);
    return launch_bwd<T, S, true, true>(p, stream, sms);
}

template <typename T>
ss_status scan_bwd(const void *x, const void *dt, const float *A, const void *B, const void *C, const float *D,
                   const void *z, const float *dt_bias, int softplus, const float *h0, const void *dout,
                   const float *dfinal, void *dx, void *ddt, float *dA, float *dB, float *dC, float *dD, void *dz,
                   float *ddt_bias, float *dh0, void *workspace, size_t workspace_bytes, int64_t batch,
                   int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream, int states_ready = 0,
                   const uint8_t *reset = nullptr, int reverse = 0)
{
    g_err[0] = '\0';
    if (batch <= 0 || d_inner <= 0 || L <= 0)
        return fail(SS_ERR_DIM, "sizes must be positive: batch=%lld d_inner=%lld L=%lld",
                    (long long)batch, (long long)d_inner, (long long)L);
    if (N < 1 || N > 32)
        return fail(SS_ERR_N, "N=%lld outside [1, 32] (the backward pass)", (long long)N);
    if (batch > (int64_t(1) << 40) / d_inner || batch * d_inner > (int64_t(1) << 50) / L)
        return fail(SS_ERR_DIM, "element count overflows");
    const size_t need = bwd_workspace_bytes(batch, d_inner, L, N);
    const PtrCheck list[] = {{x, "x", true},         {dt, "delta", true},   {A, "A", true},
                             {B, "B", true},         {C, "C", true},        {dout, "dout", true},
                             {dx, "dx", true},       {ddt, "ddelta", true}, {dA, "dA", true},
                             {dB, "dB", true},       {dC, "dC", true},      {workspace, "workspace", true},
                             {D, "D", false},        {z, "z", false},       {dt_bias, "dt_bias", false},
                             {h0, "h0", false},      {dfinal, "dfinal_state", false},
                             {dD, "dD", false},      {dz, "dz", false},     {ddt_bias, "ddt_bias", false},
                             {dh0, "dh0", false},    {reset, "seq_start", false}};
    int dev = 0;
    ss_status st = check_ptrs(list, static_cast<int>(sizeof(list) / sizeof(list[0])), &dev);
    if (st != SS_OK)
        return st;
    if (workspace_bytes < need)
        return fail(SS_ERR_DIM, "workspace of %zu bytes is smaller than the %zu bytes required", workspace_bytes,
                    need);
    if (states_ready && (reset || reverse))
        return fail(SS_ERR_DIM, "states stored by the training forward are kept for the forward direction "
                    "without sequence starts only");
    if (!aligned16(workspace))
        return fail(SS_ERR_DIM, "workspace must be 16-byte aligned");

    // accumulated outputs start from zero
    const struct { void *p; size_t n; } zero[] = {
        {dA, static_cast<size_t>(d_inner * N) * 4}, {dB, static_cast<size_t>(batch * N * L) * 4},
        {dC, static_cast<size_t>(batch * N * L) * 4}, {dD, static_cast<size_t>(d_inner) * 4},
        {ddt_bias, static_cast<size_t>(d_inner) * 4}};
    for (const auto &zc : zero) {
        if (!zc.p)
            continue;
        cudaError_t e = cudaMemsetAsync(zc.p, 0, zc.n, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SS_ERR_LAUNCH, "cudaMemsetAsync failed: %s", cudaGetErrorString(e));
        }
    }

    BwdParams p{};
    p.x = x; p.dt = dt; p.B = B; p.C = C; p.z = z; p.dout = dout;
    p.A = A; p.D = D; p.dt_bias = dt_bias; p.h0 = h0; p.dfinal = dfinal;
    p.dx = dx; p.ddt = ddt; p.dz = z ? dz : nullptr;
    p.dA = dA; p.dB = dB; p.dC = dC; p.dD = D ? dD : nullptr; p.ddt_bias = ddt_bias; p.dh0 = dh0;
    p.ckpt = static_cast<float4 *>(workspace);
    p.batch = batch; p.d_inner = d_inner; p.L = L; p.N = N;
    p.nsub = (L + kBwdHC - 1) / kBwdHC;
    p.softplus = softplus ? 1 : 0;
    p.states_ready = states_ready ? 1 : 0;
    p.reset = reset;
    p.vec = (L % 16 == 0) && aligned16(x) && aligned16(dt) && aligned16(dout) && aligned16(dx) &&
            aligned16(ddt) && (!z || aligned16(z)) && (!p.dz || aligned16(p.dz));
    p.vec4 = (L % 4 == 0) && aligned16(dB) && aligned16(dC);
    p.tma = (p.vec && aligned16(B) && aligned16(C) && encode_bwd_maps<T>(p)) ? 1 : 0;
    const int64_t S = bwd_groups(N);
    const bool rev = reverse != 0;
    const int sms = sm_count(dev);
    if (S == 1) return dispatch_bwd<T, 1>(p, rev, stream, sms);
    if (S == 2) return dispatch_bwd<T, 2>(p, rev, stream, sms);
    if (S == 4) return dispatch_bwd<T, 4>(p, rev, stream, sms);
    return dispatch_bwd<T, 8>(p, rev, stream, sms);
}

// ------------------------------------------------------------------ built-in scratch (no caller workspace)
//
// ss_scan_bwd_noalloc_* keeps the stored states in this file-scope device
// array instead of a caller workspace, so a call allocates nothing and needs
// nothing beyond its inputs and outputs. Every CUDA context that loads the
// library's module holds one copy of the array (kBwdScratchBytes of device
// memory), whether or not it ever calls the entry point. The copy is shared by
// every call made in that context: two calls whose work overlaps in time
// (different streams without ordering, or different host threads) race on it,
// so callers order them. Nothing in it has to start at zero: the forward walk
// writes every stored state before the reverse walk reads it.
//
// Host code cannot use the array's name as a device address; the address is
// resolved with cudaGetSymbolAddress. It belongs to the current context, so it
// is cached together with that context's unique id: after cudaDeviceReset (or
// in another context on the same device) the next call resolves it again. The
// first call in a context resolves it (which can load the module), so that
// call should come before any stream capture.
constexpr size_t kBwdScratchBytes = static_cast<size_t>(SS_BWD_NOALLOC_MAX_BYTES);
static __device__ __align__(256) unsigned char g_bwd_scratch[kBwdScratchBytes];

using CtxGetCurrentFn = PFN_cuCtxGetCurrent_v4000;
using CtxGetIdFn = PFN_cuCtxGetId_v12000;

// unique id of the current context (0 if there is none or it cannot be read)
unsigned long long current_context_id()
{
    static const CtxGetCurrentFn get_ctx = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            f = nullptr;
        }
        return reinterpret_cast<CtxGetCurrentFn>(f);
    }();
    static const CtxGetIdFn get_id = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            f = nullptr;
        }
        return reinterpret_cast<CtxGetIdFn>(f);
    }();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_ctx || !get_id || get_ctx(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// device address of g_bwd_scratch in the current context (the runtime's
// context of device dev, made current by the caller), or NULL
void *bwd_scratch(int dev)
{
    struct Entry {
        unsigned long long ctx_id;
        void *addr;
    };
    static std::mutex mu;
    static Entry cache[64] = {};
    const unsigned long long id = current_context_id();
    if (id != 0 && dev >= 0 && dev < 64) {
        std::lock_guard<std::mutex> lock(mu);
        if (cache[dev].ctx_id == id && cache[dev].addr)
            return cache[dev].addr;
    }
    void *q = nullptr;
    if (cudaGetSymbolAddress(&q, g_bwd_scratch) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    // the context id after the call: resolving the address can create the context
    const unsigned long long id2 = current_context_id();
    if (id2 != 0 && dev >= 0 && dev < 64) {
        std::lock_guard<std::mutex> lock(mu);
        cache[dev] = Entry{id2, q};
    }
    return q;
}

template <typename T>
ss_status scan_bwd_noalloc(const void *x, const void *dt, const float *A, const void *B, const void *C,
                           const float *D, const void *z, const float *dt_bias, int softplus, const float *h0,
                           const void *dout, const float *dfinal, void *dx, void *ddt, float *dA, float *dB,
                           float *dC, float *dD, void *dz, float *ddt_bias, float *dh0, int64_t batch,
                           int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream)
{
    g_err[0] = '\0';
    const PtrCheck req[] = {{x, "x", true},   {dt, "delta", true}, {A, "A", true},    {B, "B", true},
                            {C, "C", true},   {dout, "dout", true}, {dx, "dx", true}, {ddt, "ddelta", true},
                            {dA, "dA", true}, {dB, "dB", true},     {dC, "dC", true}};
    for (const auto &r : req)
        if (!r.p)
            return fail(SS_ERR_NULL, "required pointer %s is NULL", r.name);
    // sizes and N are checked before the stored-state bytes are formed
    if (batch <= 0 || d_inner <= 0 || L <= 0)
        return fail(SS_ERR_DIM, "sizes must be positive: batch=%lld d_inner=%lld L=%lld",
                    (long long)batch, (long long)d_inner, (long long)L);
    if (N < 1 || N > 32)
        return fail(SS_ERR_N, "N=%lld outside [1, 32] (the backward pass)", (long long)N);
    if (batch > (int64_t(1) << 40) / d_inner || batch * d_inner > (int64_t(1) << 50) / L)
        return fail(SS_ERR_DIM, "element count overflows");
    const size_t need = bwd_workspace_bytes(batch, d_inner, L, N);
    if (need > kBwdScratchBytes)
        return fail(SS_ERR_DIM, "this problem needs %zu bytes of stored states; the built-in scratch holds %zu "
                    "(use ss_scan_bwd_* with a workspace)", need, kBwdScratchBytes);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SS_ERR_INTERNAL, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    }
    void *ws = bwd_scratch(dev);
    if (!ws)
        return fail(SS_ERR_INTERNAL, "the address of the built-in scratch could not be resolved");
    return scan_bwd<T>(x, dt, A, B, C, D, z, dt_bias, softplus, h0, dout, dfinal, dx, ddt, dA, dB, dC, dD, dz,
                       ddt_bias, dh0, ws, kBwdScratchBytes, batch, d_inner, L, N, stream);
}
