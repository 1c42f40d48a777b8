// ss_scan.cu -- sm_103a kernels and C ABI of the selective scan (S6) library.
//
// What is computed is stated in include/ss_scan.h ("Mamba and selective state
// spaces": box "Selective state-space model (S6)", sections "The
// discretization the code actually uses", "The Mamba block", "Decoding with a
// constant-size cache").
//
// Scan kernel layout
// ------------------
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

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cooperative_groups.h>

#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "ss_scan.h"

namespace cg = cooperative_groups;

namespace {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)

// ------------------------------------------------------------------ device math

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(v) = log(1 + e^v) = max(v, 0) + log1p(w), w = e^{-|v|} in (0, 1],
// finite for every finite v. log1p(w) = w * Q(w) with Q of degree 8, fitted
// to log1p(w)/w on [0, 1] by Lawson-reweighted least squares on Chebyshev
// nodes (csrc/fit_log1p.py); relative error 2.3e-7 in float32 Horner
// evaluation, i.e. at float32 rounding level.
__device__ __forceinline__ float softplus_f(float v)
{
    const float w = ex2_approx(-fabsf(v) * kLog2e);
    float q = 5.232624244e-03f;
    q = fmaf(q, w, -2.950495668e-02f);
    q = fmaf(q, w, 7.822549343e-02f);
    q = fmaf(q, w, -1.366320699e-01f);
    q = fmaf(q, w, 1.910598874e-01f);
    q = fmaf(q, w, -2.484297752e-01f);
    q = fmaf(q, w, 3.331909478e-01f);
    q = fmaf(q, w, -4.999949336e-01f);
    q = fmaf(q, w, 9.999999404e-01f);
    return fmaf(w, q, fmaxf(v, 0.0f));
}

// z * sigmoid(z) = z / (1 + e^{-z}); e^{-z} = inf for very negative z gives 0.
__device__ __forceinline__ float silu_f(float z)
{
    return z * rcp_approx(1.0f + ex2_approx(-z * kLog2e));
}

// ------------------------------------------------------------------ io helpers

template <typename T> struct Io;

template <> struct Io<float> {
    static constexpr int kPerVec = 4;  // elements per 16-byte vector
    __device__ static __forceinline__ float load1(const float *p) { return __ldg(p); }
    __device__ static __forceinline__ void loadvec(const float *p, float *out)
    {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(p));
        out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    }
    __device__ static __forceinline__ void store1(float *p, float v) { *p = v; }
    __device__ static __forceinline__ void storevec(float *p, const float *v)
    {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <> struct Io<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    __device__ static __forceinline__ float load1(const __nv_bfloat16 *p)
    {
        const unsigned short s = __ldg(reinterpret_cast<const unsigned short *>(p));
        return __uint_as_float(static_cast<uint32_t>(s) << 16);
    }
    __device__ static __forceinline__ void loadvec(const __nv_bfloat16 *p, float *out)
    {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
        out[0] = bf16lo(v.x); out[1] = bf16hi(v.x);
        out[2] = bf16lo(v.y); out[3] = bf16hi(v.y);
        out[4] = bf16lo(v.z); out[5] = bf16hi(v.z);
        out[6] = bf16lo(v.w); out[7] = bf16hi(v.w);
    }
    __device__ static __forceinline__ void store1(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
    __device__ static __forceinline__ void storevec(__nv_bfloat16 *p, const float *v)
    {
        uint4 o;
        o.x = pack_bf16x2(v[0], v[1]);
        o.y = pack_bf16x2(v[2], v[3]);
        o.z = pack_bf16x2(v[4], v[5]);
        o.w = pack_bf16x2(v[6], v[7]);
        *reinterpret_cast<uint4 *>(p) = o;
    }
};

// K consecutive elements starting at row[t]; out-of-range steps read as 0.
template <typename T, int K>
__device__ __forceinline__ void load_items(const T *row, int64_t t, int64_t L, bool vec, float *out)
{
    if (vec && t + K <= L) {
#pragma unroll
        for (int v = 0; v < K; v += Io<T>::kPerVec)
            Io<T>::loadvec(row + t + v, out + v);
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i)
            out[i] = (t + i < L) ? Io<T>::load1(row + t + i) : 0.0f;
    }
}

template <typename T, int K>
__device__ __forceinline__ void store_items(T *row, int64_t t, int64_t L, bool vec, const float *v)
{
    if (vec && t + K <= L) {
#pragma unroll
        for (int e = 0; e < K; e += Io<T>::kPerVec)
            Io<T>::storevec(row + t + e, v + e);
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i)
            if (t + i < L)
                Io<T>::store1(row + t + i, v[i]);
    }
}

// ------------------------------------------------------------------ scan kernel

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
};

constexpr int kBlock = 128;

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

// ------------------------------------------------------------------ 16-byte pieces

// kPerVec consecutive elements of `row` starting at step t, as raw 16 bytes;
// steps at or past L read as 0.
template <typename T>
__device__ __forceinline__ uint4 load_piece(const T *row, int64_t t, int64_t L, bool vec)
{
    constexpr int V = Io<T>::kPerVec;
    if (vec && t + V <= L)
        return __ldg(reinterpret_cast<const uint4 *>(row + t));
    float v[V];
#pragma unroll
    for (int i = 0; i < V; ++i)
        v[i] = (t + i < L) ? Io<T>::load1(row + t + i) : 0.0f;
    uint4 o;
    if constexpr (V == 4) {
        o.x = __float_as_uint(v[0]); o.y = __float_as_uint(v[1]);
        o.z = __float_as_uint(v[2]); o.w = __float_as_uint(v[3]);
    } else {
        o.x = pack_bf16x2(v[0], v[1]); o.y = pack_bf16x2(v[2], v[3]);
        o.z = pack_bf16x2(v[4], v[5]); o.w = pack_bf16x2(v[6], v[7]);
    }
    return o;
}

template <typename T>
__device__ __forceinline__ void unpack_piece(const uint4 &w, float *out)
{
    if constexpr (Io<T>::kPerVec == 4) {
        out[0] = __uint_as_float(w.x); out[1] = __uint_as_float(w.y);
        out[2] = __uint_as_float(w.z); out[3] = __uint_as_float(w.w);
    } else {
        out[0] = bf16lo(w.x); out[1] = bf16hi(w.x);
        out[2] = bf16lo(w.y); out[3] = bf16hi(w.y);
        out[4] = bf16lo(w.z); out[5] = bf16hi(w.z);
        out[6] = bf16lo(w.w); out[7] = bf16hi(w.w);
    }
}

// ------------------------------------------------------------------ packed pairs
//
// A pair of fp32 values lives in one 64-bit register (low word first), the
// operand form of the sm_100+ f32x2 instructions.

typedef unsigned long long u64;

__device__ __forceinline__ u64 pk(float a, float b)
{
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void upk(u64 v, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

__device__ __forceinline__ u64 mul2(u64 a, u64 b)
{
    u64 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ u64 add2(u64 a, u64 b)
{
    u64 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c)
{
    u64 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// 2^v elementwise
__device__ __forceinline__ u64 ex2_2(u64 v)
{
    u64 d;
    asm("{ .reg .f32 a, b;\n\t"
        "mov.b64 {a, b}, %1;\n\t"
        "ex2.approx.ftz.f32 a, a;\n\t"
        "ex2.approx.ftz.f32 b, b;\n\t"
        "mov.b64 %0, {a, b}; }"
        : "=l"(d) : "l"(v));
    return d;
}

// 1/v elementwise
__device__ __forceinline__ u64 rcp_2(u64 v)
{
    u64 d;
    asm("{ .reg .f32 a, b;\n\t"
        "mov.b64 {a, b}, %1;\n\t"
        "rcp.approx.ftz.f32 a, a;\n\t"
        "rcp.approx.ftz.f32 b, b;\n\t"
        "mov.b64 %0, {a, b}; }"
        : "=l"(d) : "l"(v));
    return d;
}

__device__ __forceinline__ u64 splat(float a) { return pk(a, a); }

__device__ __forceinline__ float hsum(u64 v)
{
    float a, b;
    upk(v, a, b);
    return a + b;
}

// softplus of a pair: max(v, 0) + w Q(w), w = e^{-|v|} (see softplus_f)
__device__ __forceinline__ u64 softplus2(u64 v)
{
    float v0, v1;
    upk(v, v0, v1);
    const u64 w = ex2_2(pk(-fabsf(v0) * kLog2e, -fabsf(v1) * kLog2e));
    u64 q = splat(5.232624244e-03f);
    q = fma2(q, w, splat(-2.950495668e-02f));
    q = fma2(q, w, splat(7.822549343e-02f));
    q = fma2(q, w, splat(-1.366320699e-01f));
    q = fma2(q, w, splat(1.910598874e-01f));
    q = fma2(q, w, splat(-2.484297752e-01f));
    q = fma2(q, w, splat(3.331909478e-01f));
    q = fma2(q, w, splat(-4.999949336e-01f));
    q = fma2(q, w, splat(9.999999404e-01f));
    return fma2(w, q, pk(fmaxf(v0, 0.0f), fmaxf(v1, 0.0f)));
}

// z sigmoid(z) of a pair
__device__ __forceinline__ u64 silu2(u64 z)
{
    const u64 e = ex2_2(mul2(z, splat(-kLog2e)));
    return mul2(z, rcp_2(add2(e, splat(1.0f))));
}

// ------------------------------------------------------------------ n-split scan kernel
//
// A CTA owns batch row b and CH = 32 channels, with S warps (S = ceil(N/4),
// N padded to 4S with A = B = C = 0, which leaves the padded states at zero):
// warp q holds states 4q..4q+3 of all 32 channels, lane c holding channel c.
// Every lane walks the whole sequence one step after another, so each
// element-step costs one exponential and four fp32 multiply(-add)s, done in
// pairs with the packed f32x2 instructions; time is not split, so no combine
// work is added.
//
// Shared-memory traffic sets the pace on this part (a 16-byte load by 32
// lanes takes four shared-memory cycles), so the layout keeps it low: B_t and
// C_t of a warp's states are the same for all its lanes (a warp-uniform load
// costs half of a scattered one), the per-step pair (delta, delta*x) is 8
// bytes, and the raw tiles are read with conflict-free 16-byte loads.
//
// The sequence is cut into chunks of LC = 32 steps. Per chunk k:
//   scan      lane c of warp q advances its 4 states over the chunk (decays of
//             the next AHEAD steps formed ahead of the state update) and
//             keeps its partial readouts sum over its states of C_t[n] h_t[n]
//             in registers, storing them when the chunk is done;
//   -- barrier --
//   epilogue  thread (c, r) adds the S partials of its RL = LC / S steps,
//             adds D x, applies the silu(z) gate and stores y;
//   prep      the same thread forms delta = softplus(dt + bias) (or dt + bias)
//             and delta*x for its steps of chunk k+1, and B, C of chunk k+1
//             are converted to fp32 [t][n];
//   -- barrier --
// The raw x, dt, z, B, C tiles of every chunk are copied into a ring of
// STAGES chunks with cp.async (16-byte pieces, zero fill past the ends) three
// chunks ahead of their use, so DRAM latency hides behind three iterations.
// The per-step work (softplus, gate, conversions) is done once per (channel,
// step), two steps at a time with f32x2 arithmetic.

#ifndef SS_NSPLIT_AHEAD
#define SS_NSPLIT_AHEAD 4  // steps whose decays are formed ahead of the state update
#endif
#define SS_NSPLIT_STAGES 4  // raw chunks resident in shared memory: k .. k+3

template <typename T, int S>
struct NSplitShape {
    static constexpr int CH = 32;                 // channels per CTA
    static constexpr int NT = CH * S;             // threads per CTA
    static constexpr int NS = 4 * S;              // padded states
    static constexpr int LC = 32;                 // steps per chunk
    static constexpr int RL = LC / S;             // steps per epilogue/prep thread
    static constexpr int STAGES = SS_NSPLIT_STAGES;
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
    static constexpr int PD_BYTES = LC * CH * 8;
    static constexpr int BC_BYTES = LC * NS * 4;
    static constexpr int Y_BYTES = S * YQ * 4;
    static constexpr int X_BYTES = S * CH * 16 + S * CH * 4;   // segment end states and step sums
    static constexpr size_t BYTES = (size_t)STAGES * STAGE_BYTES + PD_BYTES + 2 * BC_BYTES + Y_BYTES + X_BYTES;
    static_assert(RL % 2 == 0, "steps are processed in pairs");
};

__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void *gsrc, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_dst), "l"(gsrc), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int PENDING>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(PENDING) : "memory"); }

// element pair i, i+1 of a raw shared-memory row (i even)
template <typename T>
__device__ __forceinline__ u64 raw_pair(const unsigned char *row, int i)
{
    if constexpr (sizeof(T) == 4) {
        return *reinterpret_cast<const u64 *>(row + 4 * i);
    } else {
        const uint32_t x = *reinterpret_cast<const uint32_t *>(row + 2 * i);
        return pk(bf16lo(x), bf16hi(x));
    }
}

template <typename T, int RL>
__device__ __forceinline__ void write_run(T *row, int64_t t, int64_t L, bool vec, const float *v)
{
    if constexpr ((RL * sizeof(T)) % 16 == 0) {
        if (vec && t + RL <= L) {
#pragma unroll
            for (int e = 0; e < RL; e += Io<T>::kPerVec)
                Io<T>::storevec(row + t + e, v + e);
            return;
        }
    } else if constexpr (RL * sizeof(T) == 8 && sizeof(T) == 2) {
        if (vec && t + RL <= L) {
            *reinterpret_cast<uint2 *>(row + t) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
            return;
        }
    }
#pragma unroll
    for (int i = 0; i < RL; ++i)
        if (t + i < L)
            Io<T>::store1(row + t + i, v[i]);
}

// RL raw elements of a shared-memory row starting at element offset off, as
// 32-bit words, with the widest aligned loads
template <typename T, int RL>
__device__ __forceinline__ void read_run_raw(const unsigned char *row, int off, uint32_t *w)
{
    constexpr int BYTES = RL * (int)sizeof(T);
    const unsigned char *s = row + off * (int)sizeof(T);
    if constexpr (BYTES % 16 == 0) {
#pragma unroll
        for (int v = 0; v < BYTES / 16; ++v) {
            const uint4 x = *reinterpret_cast<const uint4 *>(s + 16 * v);
            w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
        }
    } else if constexpr (BYTES % 8 == 0) {
#pragma unroll
        for (int v = 0; v < BYTES / 8; ++v) {
            const uint2 x = *reinterpret_cast<const uint2 *>(s + 8 * v);
            w[2 * v] = x.x; w[2 * v + 1] = x.y;
        }
    } else {
#pragma unroll
        for (int v = 0; v < BYTES / 4; ++v)
            w[v] = *reinterpret_cast<const uint32_t *>(s + 4 * v);
    }
}

// element pair i, i+1 (i even) of a run read by read_run_raw
template <typename T>
__device__ __forceinline__ u64 word_pair(const uint32_t *w, int i)
{
    if constexpr (sizeof(T) == 4)
        return pk(__uint_as_float(w[i]), __uint_as_float(w[i + 1]));
    else
        return pk(bf16lo(w[i / 2]), bf16hi(w[i / 2]));
}

template <bool V> struct Flag { static constexpr bool value = V; };

template <typename T, int S>
__global__ void __launch_bounds__(NSplitShape<T, S>::NT, NSplitShape<T, S>::NT <= 128 ? 3 : 1)
scan_nsplit_kernel(const ScanParams p)
{
    using SH = NSplitShape<T, S>;
    constexpr int NT = SH::NT, CH = SH::CH, NS = SH::NS, LC = SH::LC, RL = SH::RL, PR = SH::PR;
    constexpr int STAGES = SH::STAGES, EPP = SH::EPP, PPT = SH::PPT;
    constexpr int D = SS_NSPLIT_AHEAD;
    constexpr int RW = RL * (int)sizeof(T) / 4;   // 32-bit words per prep/epilogue run
    static_assert(LC % 4 == 0 && D >= 1 && D <= LC, "chunk shape");

    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *raw = smem_raw;                                          // [STAGES][x, dt, z, B, C]
    u64 *Pd = reinterpret_cast<u64 *>(smem_raw + STAGES * SH::STAGE_BYTES);  // [LC][CH] (delta, delta x)
    float *Bf = reinterpret_cast<float *>(Pd + LC * CH);                    // [LC][NS]
    float *Cf = Bf + LC * NS;                                               // [LC][NS]
    float *Yp = Cf + LC * NS;                                               // [S][CH][YROW]
    float4 *Hx = reinterpret_cast<float4 *>(Yp + S * SH::YQ);               // [S][CH] segment end states
    float *Sx = reinterpret_cast<float *>(Hx + S * CH);                     // [S][CH] step sums
    const uint32_t raw_s = static_cast<uint32_t>(__cvta_generic_to_shared(raw));

    const int tid = threadIdx.x;
    const int nseg = p.nseg;
    const int seg = static_cast<int>(blockIdx.x % nseg);
    const int64_t b = blockIdx.y;
    const int64_t d0 = static_cast<int64_t>(blockIdx.x / nseg) * CH;
    const int64_t L = p.L, N = p.N, Dn = p.d_inner;
    const int64_t t_lo = seg * p.seg_len;
    const int64_t t_hi = (t_lo + p.seg_len < L) ? t_lo + p.seg_len : L;
    const bool vec = p.vec != 0;

    // scan role: channel cs = lane, state group q = warp
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

    float A2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int n = 4 * q + e;
        A2[e] = (n < N) ? __ldg(p.A + ds * N + n) * kLog2e : 0.0f;
    }
    const u64 A01 = pk(A2[0], A2[1]);
    const u64 A23 = pk(A2[2], A2[3]);
    u64 h01 = 0, h23 = 0;   // +0.0f in both halves

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

    // copy the raw pieces of chunk j of the segment into stage j % STAGES
    // (steps at or past the segment end and rows that do not exist are zero)
    auto stage_in = [&](int64_t j, bool readout) {
        const uint32_t st = raw_s + static_cast<uint32_t>((j % STAGES) * SH::STAGE_BYTES);
        const int64_t t1 = t_lo + j * LC;
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
                unsigned char *dst = raw + (j % STAGES) * SH::STAGE_BYTES + soff[u];
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

    // raw B (and C) of chunk j -> fp32 [t][n]: each item is (tensor, step t,
    // states 4g..4g+3), written as one 16-byte word
    auto convert_bc = [&](int64_t j, bool readout) {
        const unsigned char *st = raw + (j % STAGES) * SH::STAGE_BYTES + 3 * SH::RAW_X;
        const int items = (readout ? 2 : 1) * LC * S;
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

    // this thread's sum of the steps it prepares (compensated), for the segment carry
    float ssum = 0.0f, scomp = 0.0f;
    auto kahan = [&](float v) {
        const float yv = v - scomp;
        const float tv = ssum + yv;
        scomp = (tv - ssum) - yv;
        ssum = tv;
    };

    // delta and delta*x of this thread's steps of chunk j
    auto prep = [&](int64_t j, bool sum_steps) {
        const unsigned char *st = raw + (j % STAGES) * SH::STAGE_BYTES;
        uint32_t xw[RW], dw[RW];
        read_run_raw<T, RL>(st + ce * SH::ROWB, re * RL, xw);
        read_run_raw<T, RL>(st + SH::RAW_X + ce * SH::ROWB, re * RL, dw);
        const int64_t left64 = t_hi - (t_lo + j * LC + re * RL);
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
            Pd[(re * RL + i) * CH + ce] = pk(s0, sx0);
            Pd[(re * RL + i + 1) * CH + ce] = pk(s1, sx1);
        }
    };

    float *yq_s = Yp + q * SH::YQ + cs * SH::YROW;   // this lane's partial readouts
    const float *Bq_s = Bf + 4 * q;                   // this warp's states of B_t, C_t
    const float *Cq_s = Cf + 4 * q;

    // walk the segment [t_lo, t_hi): with the readout (y stored) or without
    // it (state and step sum only)
    auto run = [&](auto ro) {
        constexpr bool RO = decltype(ro)::value;
        const int64_t nchunks = (t_hi - t_lo + LC - 1) / LC;
#pragma unroll
        for (int s = 0; s < STAGES - 1; ++s)
            if (s < nchunks)
                stage_in(s, RO);
            else
                cp_async_commit();
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        prep(0, !RO);
        convert_bc(0, RO);
        __syncthreads();

        for (int64_t k = 0; k < nchunks; ++k) {
            const int64_t t0 = t_lo + k * LC;
            if (k + STAGES - 1 < nchunks)
                stage_in(k + STAGES - 1, RO);
            else
                cp_async_commit();

            // ---- scan: 4 states of channel cs over the chunk; the decays and
            // writes of step t + D are formed while the state takes step t
            {
                u64 ra01[D], ra23[D], rb01[D], rb23[D];
                float yv[LC];
                auto form = [&](int t, int slot) {
                    float dl, dx;
                    upk(Pd[t * CH + cs], dl, dx);
                    const ulonglong2 Bq = *reinterpret_cast<const ulonglong2 *>(Bq_s + t * NS);
                    const u64 dd = splat(dl);
                    const u64 xx = splat(dx);
                    ra01[slot] = ex2_2(mul2(dd, A01));
                    ra23[slot] = ex2_2(mul2(dd, A23));
                    rb01[slot] = mul2(xx, Bq.x);
                    rb23[slot] = mul2(xx, Bq.y);
                };
#pragma unroll
                for (int i = 0; i < D; ++i)
                    form(i, i);
#pragma unroll
                for (int t = 0; t < LC; ++t) {
                    const int slot = t % D;
                    const u64 a01 = ra01[slot], a23 = ra23[slot], b01 = rb01[slot], b23 = rb23[slot];
                    if (t + D < LC)
                        form(t + D, slot);
                    h01 = fma2(a01, h01, b01);
                    h23 = fma2(a23, h23, b23);
                    if constexpr (RO) {
                        const ulonglong2 Cq = *reinterpret_cast<const ulonglong2 *>(Cq_s + t * NS);
                        yv[t] = hsum(fma2(Cq.y, h23, mul2(Cq.x, h01)));
                    }
                }
                if constexpr (RO) {
#pragma unroll
                    for (int t = 0; t < LC; t += 4)
                        *reinterpret_cast<float4 *>(yq_s + t) = make_float4(yv[t], yv[t + 1], yv[t + 2], yv[t + 3]);
                }
            }
            cp_async_wait<STAGES - 2>();   // chunk k+1 has landed (this thread's copies)
            __syncthreads();

            // ---- epilogue of chunk k: sum partials, skip term, gate, store
            if constexpr (RO) {
                const unsigned char *st = raw + (k % STAGES) * SH::STAGE_BYTES;
                uint32_t xw[RW], zw[RW];
                read_run_raw<T, RL>(st + ce * SH::ROWB, re * RL, xw);
                if (gate)
                    read_run_raw<T, RL>(st + 2 * SH::RAW_X + ce * SH::ROWB, re * RL, zw);
                float out[RL];
#pragma unroll
                for (int i = 0; i < RL; i += 2) {
                    const float *yp = Yp + ce * SH::YROW + re * RL + i;
                    u64 acc = *reinterpret_cast<const u64 *>(yp);
#pragma unroll
                    for (int qq = 1; qq < S; ++qq)
                        acc = add2(acc, *reinterpret_cast<const u64 *>(yp + qq * SH::YQ));
                    acc = fma2(D2, word_pair<T>(xw, i), acc);
                    if (gate)
                        acc = mul2(acc, silu2(word_pair<T>(zw, i)));
                    upk(acc, out[i], out[i + 1]);
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
    };

    if (nseg > 1) {
        // Segments of one channel group form a thread-block cluster. Each
        // segment but the last walks its steps from a zero state (no readout)
        // and publishes its end state and step sum; the state entering
        // segment s is then the predecessors' maps folded in order,
        // h <- exp(A * sum of steps) h + end state, read through distributed
        // shared memory.
        cg::cluster_group cluster = cg::this_cluster();
        if (seg < nseg - 1)
            run(Flag<false>{});
        float hv[4];
        upk(h01, hv[0], hv[1]);
        upk(h23, hv[2], hv[3]);
        Hx[q * CH + cs] = make_float4(hv[0], hv[1], hv[2], hv[3]);
        Sx[re * CH + ce] = ssum;
        cluster.sync();
        u64 f01 = 0, f23 = 0;
        for (int sp = 0; sp < seg; ++sp) {
            const float4 *ph = cluster.map_shared_rank(Hx, sp);
            const float *psum = cluster.map_shared_rank(Sx, sp);
            float tot = 0.0f;
#pragma unroll
            for (int r = 0; r < S; ++r)
                tot += psum[r * CH + cs];
            const float4 he = ph[q * CH + cs];
            const u64 tt = splat(tot);
            f01 = fma2(ex2_2(mul2(tt, A01)), f01, pk(he.x, he.y));
            f23 = fma2(ex2_2(mul2(tt, A23)), f23, pk(he.z, he.w));
        }
        cluster.sync();   // peers have finished reading this CTA's end state
        h01 = f01;
        h23 = f23;
    }
    run(Flag<true>{});

    if (p.final_state && act_s && seg == nseg - 1) {
        float *fs = p.final_state + (b * Dn + ds) * N;
        float hv[4];
        upk(h01, hv[0], hv[1]);
        upk(h23, hv[2], hv[3]);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (4 * q + e < N)
                fs[4 * q + e] = hv[e];
    }
}

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
    static constexpr size_t BYTES = (size_t)STAGES * STAGE_BYTES + PD_BYTES + DY_BYTES + 2 * BC_BYTES + PART_BYTES +
                                    DBC_BYTES;
    static_assert(RH >= 2 && RH % 2 == 0, "epilogue runs are processed in pairs");
};

// both halves negated
__device__ __forceinline__ u64 neg2(u64 a) { return a ^ 0x8000000080000000ull; }

template <typename T, int S>
__global__ void __launch_bounds__(BwdShape<T, S>::NT, BwdShape<T, S>::NT <= 128 ? 3 : 1)
scan_bwd_kernel(const BwdParams p)
{
    using SH = BwdShape<T, S>;
    constexpr int NT = SH::NT, CH = SH::CH, NS = SH::NS, LC = SH::LC, HC = SH::HC, NH = SH::NH;
    constexpr int RL = SH::RL, RH = SH::RH, PR = SH::PR, STAGES = SH::STAGES, EPP = SH::EPP, PPT = SH::PPT;
    constexpr int RW = RL * (int)sizeof(T) / 4;
    constexpr int RHW = RH * (int)sizeof(T) / 4 > 0 ? RH * (int)sizeof(T) / 4 : 1;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *raw = smem_raw;                                          // [STAGES][x, dt, z, dout, B, C]
    u64 *Pd = reinterpret_cast<u64 *>(smem_raw + STAGES * SH::STAGE_BYTES);  // [LC][CH] (delta, delta x)
    float *DY = reinterpret_cast<float *>(Pd + LC * CH);                    // [LC][CH] gy
    float *Bf = DY + LC * CH;                                               // [LC][NS]
    float *Cf = Bf + LC * NS;                                               // [LC][NS]
    float *Part = Cf + LC * NS;                                             // [3][S][HC/2][CH] step pairs
    float *DBC = Part + 3 * S * HC * CH;                                    // [2][LC][NS]
    const uint32_t raw_s = static_cast<uint32_t>(__cvta_generic_to_shared(raw));

    const int tid = threadIdx.x;
    const int64_t b = blockIdx.y;
    const int64_t d0 = static_cast<int64_t>(blockIdx.x) * CH;
    const int64_t L = p.L, N = p.N, Dn = p.d_inner;
    const bool vec = p.vec != 0;
    const int64_t nchunks = (L + LC - 1) / LC;

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
    auto stage_in = [&](int64_t k, int slot, bool phase2) {
        const uint32_t st = raw_s + static_cast<uint32_t>(slot * SH::STAGE_BYTES);
        const int64_t t1 = k * LC;
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
#pragma unroll
        for (int i = 0; i < RL; i += 2) {
            const u64 xx = word_pair<T>(xw, i);
            const u64 u = add2(word_pair<T>(dw, i), bias2);
            const u64 s2 = p.softplus ? softplus2(u) : u;
            float s0, s1;
            upk(s2, s0, s1);
            s0 = i < lim ? s0 : 0.0f;
            s1 = i + 1 < lim ? s1 : 0.0f;
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

    // ---- phase 1: forward, storing the state at every sub-chunk start
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
    {
#pragma unroll
        for (int s = 0; s < STAGES - 1; ++s)
            if (s < nchunks)
                stage_in(s, s, false);
            else
                cp_async_commit();
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        prep(0, 0, false);
        convert_bc(0, false);
        __syncthreads();
        for (int64_t k = 0; k < nchunks; ++k) {
            if (k + STAGES - 1 < nchunks)
                stage_in(k + STAGES - 1, static_cast<int>((k + STAGES - 1) % STAGES), false);
            else
                cp_async_commit();
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const int64_t s = k * NH + hh;
                if (act_s && s < p.nsub) {
                    float a0, a1, a2, a3;
                    upk(h01, a0, a1);
                    upk(h23, a2, a3);
                    ck[s * ckstride] = make_float4(a0, a1, a2, a3);
                }
#pragma unroll 4
                for (int i = 0; i < HC; ++i) {
                    const int t = hh * HC + i;
                    float dl, dx;
                    upk(Pd[t * CH + cs], dl, dx);
                    const ulonglong2 Bq = *reinterpret_cast<const ulonglong2 *>(Bq_s + t * NS);
                    const u64 dd = splat(dl), xx = splat(dx);
                    h01 = fma2(ex2_2(mul2(dd, A01)), h01, mul2(xx, Bq.x));
                    h23 = fma2(ex2_2(mul2(dd, A23)), h23, mul2(xx, Bq.y));
                }
            }
            cp_async_wait<STAGES - 2>();
            __syncthreads();
            if (k + 1 < nchunks) {
                prep(k + 1, static_cast<int>((k + 1) % STAGES), false);
                convert_bc(static_cast<int>((k + 1) % STAGES), false);
            }
            __syncthreads();
        }
        cp_async_wait<0>();
        __syncthreads();
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

    float4 ck_cur = make_float4(0.f, 0.f, 0.f, 0.f);   // stored state of the sub-chunk processed next
    if (act_s)
        ck_cur = ck[(p.nsub - 1) * ckstride];

    // chunk order j = 0, 1, ... is k = nchunks - 1 - j
#pragma unroll 1
    for (int s = 0; s < STAGES - 1; ++s)
        if (s < nchunks)
            stage_in(nchunks - 1 - s, s, true);
        else
            cp_async_commit();
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    prep(nchunks - 1, 0, true);
    convert_bc(0, true);
    __syncthreads();

#pragma unroll 1
    for (int64_t j = 0; j < nchunks; ++j) {
        const int64_t k = nchunks - 1 - j;
        const int slot = static_cast<int>(j % STAGES);
        if (j + STAGES - 1 < nchunks)
            stage_in(k - (STAGES - 1), static_cast<int>((j + STAGES - 1) % STAGES), true);
        else
            cp_async_commit();

#pragma unroll 1
        for (int hh = NH - 1; hh >= 0; --hh) {
            const int64_t s = k * NH + hh;
            if (s < p.nsub) {
                // the stored state of the next sub-chunk is fetched while this one runs
                float4 ck_next = make_float4(0.f, 0.f, 0.f, 0.f);
                if (act_s && s >= 1)
                    ck_next = ck[(s - 1) * ckstride];
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
                        const int t = hh * HC + i;
                        float dl, dx;
                        upk(Pd[t * CH + cs], dl, dx);
                        const ulonglong2 Bq = *reinterpret_cast<const ulonglong2 *>(Bq_s + t * NS);
                        const u64 dd = splat(dl), xx = splat(dx);
                        g01 = fma2(ex2_2(mul2(dd, A01)), g01, mul2(xx, Bq.x));
                        g23 = fma2(ex2_2(mul2(dd, A23)), g23, mul2(xx, Bq.y));
                        H01[i] = g01;
                        H23[i] = g23;
                    }
                }
                // adjoint recurrence backwards over the sub-chunk, two steps per round
                // step i: lam += C gy; v = (lam dx, gy h) for the channel sums; the
                // state sums for the epilogue; then lam *= a_i for step i-1
                auto step = [&](int i, float *v, float &r_, float &pa, float &yy) {
                    const int t = hh * HC + i;
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
                    const u64 p01 = mul2(lam01, mul2(a01, i > 0 ? H01[i > 0 ? i - 1 : 0] : S01));   // lam a_t h_{t-1}
                    const u64 p23 = mul2(lam23, mul2(a23, i > 0 ? H23[i > 0 ? i - 1 : 0] : S23));
                    dA01 = fma2(p01, dd, dA01);
                    dA23 = fma2(p23, dd, dA23);
                    r_ = hsum(fma2(lam23, Bq.y, mul2(lam01, Bq.x)));
                    pa = hsum(fma2(p23, A23, mul2(p01, A01)));
                    yy = hsum(fma2(Cq.y, H23[i], mul2(Cq.x, H01[i])));
                    lam01 = mul2(lam01, a01);
                    lam23 = mul2(lam23, a23);
                };
                const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
                for (int i = HC - 1; i >= 1; i -= 2) {
                    float val[16];   // [0, 8): step i, [8, 16): step i-1
                    float r1, pa1, y1, r0, pa0, y0;
                    step(i, val, r1, pa1, y1);
                    step(i - 1, val + 8, r0, pa0, y0);
                    float2 *pp = reinterpret_cast<float2 *>(Part) + (q * (HC / 2) + (i >> 1)) * CH + cs;
                    pp[0] = make_float2(r0, r1);
                    pp[S * (HC / 2) * CH] = make_float2(pa0, pa1);
                    pp[2 * S * (HC / 2) * CH] = make_float2(y0, y1);
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
                        const int t = hh * HC + i - (kk >> 3);
                        DBC[((kv >> 2) * LC + t) * NS + 4 * q + (kv & 3)] = sum;
                    }
                }
            }
            __syncthreads();
            // ---- epilogue of the sub-chunk: steps hh*HC + re*RH .. + RH - 1
            if (s < p.nsub) {
                const unsigned char *st = raw + slot * SH::STAGE_BYTES;
                const int off = hh * HC + re * RH;
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
        __syncthreads();
        if (j + 1 < nchunks) {
            const int nslot = static_cast<int>((j + 1) % STAGES);
            prep(k - 1, nslot, true);
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
        if (p.dh0) {
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
}

// ------------------------------------------------------------------ decode kernel

struct UpdateParams {
    float *state;
    const void *x, *delta, *B, *C, *z;
    const float *A, *D;
    void *y;
    int64_t batch, d_inner, N;
    int vec;     // N % 4 == 0 and 16-byte aligned state and A
    int vec_bc;  // B and C rows are whole 16-byte words (16-byte aligned, N * sizeof(T) % 16 == 0)
};

// One thread per (batch row, channel) holding all N = 4 NV states: the state
// and A of the row move as 16-byte words, B and C of the batch row (shared by
// all its channels, so served from L1 after the first warp) as 16-byte words
// where their size allows, and the readout is summed inside the thread.
template <typename T, int NV>
__global__ void __launch_bounds__(kBlock)
state_update_row_kernel(const UpdateParams p)
{
    constexpr int N = 4 * NV;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (row >= p.batch * p.d_inner)
        return;
    const int64_t b = row / p.d_inner;
    const int64_t d = row % p.d_inner;
    float4 *st = reinterpret_cast<float4 *>(p.state + row * N);
    const float4 *Ad = reinterpret_cast<const float4 *>(p.A + d * N);
    const T *Bb = static_cast<const T *>(p.B) + b * N;
    const T *Cb = static_cast<const T *>(p.C) + b * N;

    float4 h[NV], a[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        h[v] = st[v];
        a[v] = __ldg(Ad + v);
    }
    float bv[N], cv[N];
    if (p.vec_bc) {
#pragma unroll
        for (int e = 0; e < N; e += Io<T>::kPerVec) {
            Io<T>::loadvec(Bb + e, bv + e);
            Io<T>::loadvec(Cb + e, cv + e);
        }
    } else {
#pragma unroll
        for (int e = 0; e < N; ++e) {
            bv[e] = Io<T>::load1(Bb + e);
            cv[e] = Io<T>::load1(Cb + e);
        }
    }
    const float xv = Io<T>::load1(static_cast<const T *>(p.x) + row);
    const float dl = Io<T>::load1(static_cast<const T *>(p.delta) + row);
    const float dx = dl * xv;
    const float dl2 = dl * kLog2e;
    float out = 0.0f;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        float *hv = reinterpret_cast<float *>(&h[v]);
        const float *av = reinterpret_cast<const float *>(&a[v]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int n = 4 * v + e;
            hv[e] = fmaf(ex2_approx(dl2 * av[e]), hv[e], dx * bv[n]);
            out = fmaf(cv[n], hv[e], out);
        }
        st[v] = h[v];
    }
    out = fmaf(p.D ? __ldg(p.D + d) : 0.0f, xv, out);
    if (p.z)
        out *= silu_f(Io<T>::load1(static_cast<const T *>(p.z) + row));
    Io<T>::store1(static_cast<T *>(p.y) + row, out);
}

// One thread per (row, group of 4 states); the NQ threads of a row are
// adjacent lanes of one warp and sum their partial readouts by shuffles.
template <typename T, int NQ>
__global__ void __launch_bounds__(kBlock)
state_update_kernel(const UpdateParams p)
{
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    const int q = static_cast<int>(gid % NQ);
    int64_t row = gid / NQ;
    const int64_t rows = p.batch * p.d_inner;
    const bool active = row < rows;
    row = active ? row : 0;
    const int64_t b = row / p.d_inner;
    const int64_t d = row % p.d_inner;
    const int64_t N = p.N;
    const int n0 = 4 * q;

    const float xv = Io<T>::load1(static_cast<const T *>(p.x) + row);
    const float dl = Io<T>::load1(static_cast<const T *>(p.delta) + row);
    const float dx = dl * xv;
    float *st = p.state + row * N;
    const float *Ad = p.A + d * N;
    const T *Bb = static_cast<const T *>(p.B) + b * N;
    const T *Cb = static_cast<const T *>(p.C) + b * N;

    float hv[4] = {0.f, 0.f, 0.f, 0.f}, av[4] = {0.f, 0.f, 0.f, 0.f};
    float bv[4] = {0.f, 0.f, 0.f, 0.f}, cv[4] = {0.f, 0.f, 0.f, 0.f};
    const bool mine = active && n0 < N;
    if (mine) {
        if (p.vec) {
            const float4 h4 = *reinterpret_cast<const float4 *>(st + n0);
            const float4 a4 = __ldg(reinterpret_cast<const float4 *>(Ad + n0));
            hv[0] = h4.x; hv[1] = h4.y; hv[2] = h4.z; hv[3] = h4.w;
            av[0] = a4.x; av[1] = a4.y; av[2] = a4.z; av[3] = a4.w;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                bv[k] = Io<T>::load1(Bb + n0 + k);
                cv[k] = Io<T>::load1(Cb + n0 + k);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (n0 + k < N) {
                    hv[k] = st[n0 + k];
                    av[k] = __ldg(Ad + n0 + k);
                    bv[k] = Io<T>::load1(Bb + n0 + k);
                    cv[k] = Io<T>::load1(Cb + n0 + k);
                }
            }
        }
    }
    float part = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float a = ex2_approx(dl * av[k] * kLog2e);
        hv[k] = fmaf(a, hv[k], dx * bv[k]);
        part = fmaf(cv[k], hv[k], part);
    }
#pragma unroll
    for (int off = NQ / 2; off > 0; off /= 2)
        part += __shfl_xor_sync(0xffffffffu, part, off, NQ);

    if (mine) {
        if (p.vec) {
            *reinterpret_cast<float4 *>(st + n0) = make_float4(hv[0], hv[1], hv[2], hv[3]);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (n0 + k < N)
                    st[n0 + k] = hv[k];
        }
    }
    if (active && q == 0) {
        float out = part + (p.D ? __ldg(p.D + d) : 0.0f) * xv;
        if (p.z)
            out *= silu_f(Io<T>::load1(static_cast<const T *>(p.z) + row));
        Io<T>::store1(static_cast<T *>(p.y) + row, out);
    }
}

// ------------------------------------------------------------------ causal depthwise conv1d
//
// out[b,d,t] = act(sum_{i<k} w[d,i] xin[b,d,t-i] + bias[d]), act = SiLU or
// identity ("The Mamba block"); inputs before t = 0 come from the carried
// history (batch, k-1, d_inner), oldest first, or are zero. One thread per
// EPP-element (16-byte) piece of a row: it reads its piece and the HP pieces
// before it (the halo of k-1 inputs), and writes its outputs as one 16-byte
// word.

struct ConvParams {
    const void *x, *state_in;
    const float *w, *bias;
    void *out, *state_out;
    int64_t batch, d_inner, L;
    int silu;
    int vec;  // 16-byte aligned rows of whole pieces
};

// Input t of row (b, d): x for t >= 0, the carried history for -(K-1) <= t < 0
// (zero when there is none).
template <typename T, int K>
__device__ __forceinline__ float conv_input(const ConvParams &p, const T *xr, int64_t b, int64_t d, int64_t t)
{
    if (t >= 0)
        return Io<T>::load1(xr + t);
    if (p.state_in)
        return Io<T>::load1(static_cast<const T *>(p.state_in) + (b * (K - 1) + (K - 1 + t)) * p.d_inner + d);
    return 0.0f;
}

// grid = (piece blocks of a row, channel groups of R, batch rows); each thread
// owns the 16-byte piece (EPP consecutive steps) at the same position of R
// consecutive channels, whose loads are all issued before any is used. The
// K-1 inputs before a piece come from the lane below by shuffle; the lowest
// lanes of a warp, whose predecessors sit in another warp, load them (or the
// carried history) directly.
template <typename T, int K, int R>
__global__ void __launch_bounds__(kBlock)
causal_conv1d_kernel(const ConvParams p)
{
    constexpr int EPP = 16 / (int)sizeof(T);
    constexpr int H = K - 1;
    constexpr int HW = H > 0 ? H : 1;
    const int lane = threadIdx.x & 31;
    const int64_t npieces = (p.L + EPP - 1) / EPP;
    const int64_t pc = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    const bool inb = pc < npieces;
    const int64_t t0 = pc * EPP;

    for (int64_t b = blockIdx.z; b < p.batch; b += gridDim.z) {
        for (int64_t d0 = static_cast<int64_t>(blockIdx.y) * R; d0 < p.d_inner; d0 += static_cast<int64_t>(gridDim.y) * R) {
            uint4 raw[R];   // kept packed until used
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t d = d0 + r;
                raw[r] = make_uint4(0u, 0u, 0u, 0u);
                if (d < p.d_inner && inb)
                    raw[r] = load_piece<T>(static_cast<const T *>(p.x) + (b * p.d_inner + d) * p.L, t0, p.L,
                                           p.vec);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t d = d0 + r;
                if (d >= p.d_inner)   // uniform over the block
                    break;
                const int64_t row = b * p.d_inner + d;
                const T *xr = static_cast<const T *>(p.x) + row * p.L;
                float own[EPP];
                unpack_piece<T>(raw[r], own);
                // hist[j] = input at t0 - H + j
                float hist[HW];
#pragma unroll
                for (int j = 0; j < H; ++j) {
                    const int back = H - j;
                    const int v = (back + EPP - 1) / EPP;   // source lane offset
                    const int e = v * EPP - back;           // element within that lane's piece
                    float val = __shfl_up_sync(0xffffffffu, own[e], v);
                    if (lane < v && inb)
                        val = conv_input<T, K>(p, xr, b, d, t0 - back);
                    hist[j] = val;
                }
                if (!inb)
                    continue;
                float wd[K];
#pragma unroll
                for (int i = 0; i < K; ++i)
                    wd[i] = __ldg(p.w + d * K + i);
                const float bv = p.bias ? __ldg(p.bias + d) : 0.0f;
                float o[EPP];
#pragma unroll
                for (int e = 0; e < EPP; ++e) {
                    float acc = bv;
#pragma unroll
                    for (int i = 0; i < K; ++i)
                        acc = fmaf(wd[i], (e - i >= 0) ? own[(e - i) >= 0 ? e - i : 0] : hist[H + e - i >= 0 ? H + e - i : 0], acc);
                    o[e] = p.silu ? silu_f(acc) : acc;
                }
                T *orow = static_cast<T *>(p.out) + row * p.L;
                if (p.vec) {
                    Io<T>::storevec(orow + t0, o);
                } else {
#pragma unroll
                    for (int e = 0; e < EPP; ++e)
                        if (t0 + e < p.L)
                            Io<T>::store1(orow + t0 + e, o[e]);
                }
                // the piece holding the last input writes the history for the next call
                if (H > 0 && p.state_out && p.L - 1 < t0 + EPP) {
                    T *so = static_cast<T *>(p.state_out);
#pragma unroll
                    for (int j = 0; j < H; ++j) {
                        const int64_t w = p.L - t0 + j;   // window index of input L-H+j
                        float val = 0.0f;
#pragma unroll
                        for (int u = 0; u < H + EPP; ++u)
                            if (w == u)
                                val = u < H ? hist[u < H ? u : 0] : own[u >= H ? u - H : 0];
                        Io<T>::store1(so + (b * H + j) * p.d_inner + d, val);
                    }
                }
            }
        }
    }
}

// Vector path (16-byte aligned rows, L a multiple of the piece): a CTA stages
// CG channels x LT steps of one batch row, plus the HP pieces before them, into
// shared memory with asynchronous 16-byte copies (no registers held while the
// loads are in flight), then each thread turns pieces of that tile into
// outputs. Inputs before t = 0 come from the carried history (or are zero).
constexpr int kConvTileBytes = 2048;   // one row of a tile
constexpr int kConvRows = 8;           // channels per tile

template <typename T, int K>
__global__ void __launch_bounds__(kBlock)
causal_conv1d_tile_kernel(const ConvParams p)
{
    constexpr int EPP = 16 / (int)sizeof(T);
    constexpr int H = K - 1;
    constexpr int HP = (H + EPP - 1) / EPP;      // halo pieces
    constexpr int PT = kConvTileBytes / 16;      // pieces per tile row
    constexpr int CG = kConvRows;
    __shared__ __align__(16) uint4 tile[CG][PT + HP];

    const int64_t npieces = p.L / EPP;
    const int64_t pc0 = static_cast<int64_t>(blockIdx.x) * PT;
    const int64_t d0 = static_cast<int64_t>(blockIdx.y) * CG;
    const T *x = static_cast<const T *>(p.x);
    for (int64_t b = blockIdx.z; b < p.batch; b += gridDim.z) {
        for (int i = threadIdx.x; i < CG * (PT + HP); i += kBlock) {
            const int r = i / (PT + HP);
            const int j = i % (PT + HP);
            const int64_t d = d0 + r;
            const int64_t pc = pc0 - HP + j;
            const bool ok = d < p.d_inner && pc >= 0 && pc < npieces;
            const T *src = ok ? x + (b * p.d_inner + d) * p.L + pc * EPP : x;
            cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(&tile[r][j])), src, ok ? 16 : 0);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        for (int i = threadIdx.x; i < CG * PT; i += kBlock) {
            const int r = i / PT;
            const int j = i % PT;
            const int64_t d = d0 + r;
            const int64_t pc = pc0 + j;
            if (d >= p.d_inner || pc >= npieces)
                continue;
            float win[(HP + 1) * EPP];   // steps (pc - HP) * EPP ... pc * EPP + EPP - 1
#pragma unroll
            for (int v = 0; v <= HP; ++v)
                unpack_piece<T>(tile[r][j + v], win + v * EPP);
            if (pc < HP && p.state_in) {   // steps before 0 come from the carried history
#pragma unroll
                for (int u = 0; u < HP * EPP; ++u) {
                    const int64_t t = (pc - HP) * EPP + u;
                    if (t < 0 && t >= -H)
                        win[u] = Io<T>::load1(static_cast<const T *>(p.state_in) + (b * H + (H + t)) * p.d_inner + d);
                }
            }
            float wd[K];
#pragma unroll
            for (int k = 0; k < K; ++k)
                wd[k] = __ldg(p.w + d * K + k);
            const float bv = p.bias ? __ldg(p.bias + d) : 0.0f;
            float o[EPP];
#pragma unroll
            for (int e = 0; e < EPP; ++e) {
                float acc = bv;
#pragma unroll
                for (int k = 0; k < K; ++k)
                    acc = fmaf(wd[k], win[HP * EPP + e - k], acc);
                o[e] = p.silu ? silu_f(acc) : acc;
            }
            const int64_t row = b * p.d_inner + d;
            Io<T>::storevec(static_cast<T *>(p.out) + row * p.L + pc * EPP, o);
            if (H > 0 && p.state_out && pc == npieces - 1) {
                // the last H inputs: window index HP * EPP + EPP - H + jj
#pragma unroll
                for (int jj = 0; jj < H; ++jj)
                    Io<T>::store1(static_cast<T *>(p.state_out) + (b * H + jj) * p.d_inner + d,
                                  win[HP * EPP + EPP - H + jj]);
            }
        }
        __syncthreads();   // the tile is reused by the next batch row
    }
}

// One decode step of the convolution: the k-1 cached inputs (oldest first)
// and the new input give the output; the cache then drops its oldest entry
// and takes the new input ("Decoding with a constant-size cache").
struct ConvStepParams {
    void *state;
    const void *x;
    const float *w, *bias;
    void *out;
    int64_t batch, d_inner;
    int silu;
    int vec;  // pairs of channels: d_inner even, rows aligned to a pair
};

// Two adjacent channels of io type T as one 4- or 8-byte word.
template <typename T> struct Pair;
template <> struct Pair<float> {
    __device__ static __forceinline__ void load(const float *p, float &a, float &b)
    {
        const float2 v = __ldg(reinterpret_cast<const float2 *>(p));
        a = v.x; b = v.y;
    }
    __device__ static __forceinline__ void store(float *p, float a, float b)
    {
        *reinterpret_cast<float2 *>(p) = make_float2(a, b);
    }
};
template <> struct Pair<__nv_bfloat16> {
    __device__ static __forceinline__ void load(const __nv_bfloat16 *p, float &a, float &b)
    {
        const uint32_t v = __ldg(reinterpret_cast<const unsigned int *>(p));
        a = bf16lo(v); b = bf16hi(v);
    }
    __device__ static __forceinline__ void store(__nv_bfloat16 *p, float a, float b)
    {
        *reinterpret_cast<uint32_t *>(p) = pack_bf16x2(a, b);
    }
};

// grid = (channel blocks, batch-row groups). On the pair path a thread owns two
// adjacent channels of kStepRows batch rows, and issues all their loads before
// using any; otherwise one channel of one batch row at a time.
constexpr int kStepRows = 4;

template <typename T, int K>
__global__ void __launch_bounds__(kBlock)
conv_state_update_kernel(const ConvStepParams p)
{
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    T *st = static_cast<T *>(p.state);
    const T *xg = static_cast<const T *>(p.x);
    if (p.vec) {
        constexpr int RB = kStepRows;
        const int64_t d0 = tid * 2;
        if (d0 >= p.d_inner)
            return;
        float wd[K][2];
#pragma unroll
        for (int i = 0; i < K; ++i) {
            wd[i][0] = __ldg(p.w + d0 * K + i);
            wd[i][1] = __ldg(p.w + (d0 + 1) * K + i);
        }
        const float b0 = p.bias ? __ldg(p.bias + d0) : 0.0f;
        const float b1 = p.bias ? __ldg(p.bias + d0 + 1) : 0.0f;
        for (int64_t bb = static_cast<int64_t>(blockIdx.y) * RB; bb < p.batch; bb += static_cast<int64_t>(gridDim.y) * RB) {
            float hist[RB][K][2];   // hist[.][i]: inputs i steps back, [0] = the new input
            const T *xs = xg + bb * p.d_inner + d0;
            const T *ss = st + bb * (K - 1) * p.d_inner + d0;
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                if (bb + r < p.batch) {
                    Pair<T>::load(xs, hist[r][0][0], hist[r][0][1]);
#pragma unroll
                    for (int i = 1; i < K; ++i)
                        Pair<T>::load(ss + (K - 1 - i) * p.d_inner, hist[r][i][0], hist[r][i][1]);
                }
                xs += p.d_inner;
                ss += (K - 1) * p.d_inner;
            }
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const int64_t b = bb + r;
                if (b >= p.batch)
                    break;
                float a0 = b0, a1 = b1;
#pragma unroll
                for (int i = 0; i < K; ++i) {
                    a0 = fmaf(wd[i][0], hist[r][i][0], a0);
                    a1 = fmaf(wd[i][1], hist[r][i][1], a1);
                }
                if (p.silu) {
                    a0 = silu_f(a0);
                    a1 = silu_f(a1);
                }
                Pair<T>::store(static_cast<T *>(p.out) + b * p.d_inner + d0, a0, a1);
#pragma unroll
                for (int j = 0; j < K - 1; ++j)   // slot j takes the inputs (K-2-j) steps back
                    Pair<T>::store(st + (b * (K - 1) + j) * p.d_inner + d0, hist[r][K - 2 - j][0],
                                   hist[r][K - 2 - j][1]);
            }
        }
        return;
    }
    const int64_t d = tid;
    if (d >= p.d_inner)
        return;
    float wd[K];
#pragma unroll
    for (int i = 0; i < K; ++i)
        wd[i] = __ldg(p.w + d * K + i);
    const float bv = p.bias ? __ldg(p.bias + d) : 0.0f;
    for (int64_t b = blockIdx.y; b < p.batch; b += gridDim.y) {
        const int64_t row = b * p.d_inner + d;
        float hist[K];   // hist[i]: input i steps back, hist[0] = the new input
        hist[0] = Io<T>::load1(xg + row);
#pragma unroll
        for (int i = 1; i < K; ++i)
            hist[i] = Io<T>::load1(st + (b * (K - 1) + (K - 1 - i)) * p.d_inner + d);
        float acc = bv;
#pragma unroll
        for (int i = 0; i < K; ++i)
            acc = fmaf(wd[i], hist[i], acc);
        Io<T>::store1(static_cast<T *>(p.out) + row, p.silu ? silu_f(acc) : acc);
#pragma unroll
        for (int j = 0; j < K - 1; ++j)   // slot j takes the input (K-2-j) steps back
            Io<T>::store1(st + (b * (K - 1) + j) * p.d_inner + d, hist[K - 2 - j]);
    }
}

// ------------------------------------------------------------------ host side

thread_local char g_err[512] = "";

ss_status fail(ss_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

ss_status check_ptr(const void *ptr, const char *name, int dev)
{
    cudaPointerAttributes at;
    const cudaError_t e = cudaPointerGetAttributes(&at, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SS_ERR_DEVICE_PTR, "%s: cudaPointerGetAttributes failed: %s", name,
                    cudaGetErrorString(e));
    }
    if (at.type == cudaMemoryTypeManaged)
        return SS_OK;
    if (at.type != cudaMemoryTypeDevice)
        return fail(SS_ERR_DEVICE_PTR, "%s is not device memory", name);
    if (at.device != dev)
        return fail(SS_ERR_DEVICE_PTR, "%s lives on device %d, current device is %d", name, at.device, dev);
    return SS_OK;
}

struct PtrCheck {
    const void *p;
    const char *name;
    bool required;
};

ss_status check_ptrs(const PtrCheck *list, int n, int *dev_out)
{
    for (int i = 0; i < n; ++i)
        if (!list[i].p && list[i].required)
            return fail(SS_ERR_NULL, "required pointer %s is NULL", list[i].name);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SS_ERR_INTERNAL, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    }
    for (int i = 0; i < n; ++i) {
        if (!list[i].p)
            continue;
        ss_status s = check_ptr(list[i].p, list[i].name, dev);
        if (s != SS_OK)
            return s;
    }
    *dev_out = dev;
    return SS_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count(int dev)
{
    static std::atomic<int> cache[64];
    if (dev < 0 || dev >= 64)
        return 148;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0)
        return v;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        sms = 148;
    }
    cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

template <typename T, int NT, int W, int K>
ss_status launch_scan(const ScanParams &p, cudaStream_t stream)
{
    constexpr int CH = kBlock / W;
    const size_t smem = 2u * W * (K * NT + 4) * sizeof(float);
    if (smem > 48u * 1024u) {
        cudaError_t e = cudaFuncSetAttribute(scan_fwd_kernel<T, NT, W, K>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SS_ERR_LAUNCH, "cudaFuncSetAttribute failed: %s", cudaGetErrorString(e));
        }
    }
    const int64_t gx = (p.d_inner + CH - 1) / CH;
    if (gx > 0x7fffffff || p.batch > 65535)
        return fail(SS_ERR_DIM, "grid too large: %lld channel blocks x %lld batch rows",
                    (long long)gx, (long long)p.batch);
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(p.batch));
    scan_fwd_kernel<T, NT, W, K><<<grid, kBlock, smem, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SS_ERR_LAUNCH, "scan kernel launch failed: %s", cudaGetErrorString(e));
    return SS_OK;
}

// Time lanes per channel: the fewest that give every SM enough warps.
int pick_lanes(int64_t channels, int64_t L, int sms)
{
    const char *env = getenv("SS_SCAN_LANES");
    if (env) {
        int w = atoi(env);
        if (w == 1 || w == 4 || w == 16)
            return w;
    }
    const int64_t want_threads = static_cast<int64_t>(sms) * 512;
    int w = 1;
    while (w < 16 && channels * w < want_threads && static_cast<int64_t>(w) * 16 * 4 <= L)
        w *= 4;
    return w;
}

template <typename T, int NT>
ss_status dispatch_scan_lanes(const ScanParams &p, int lanes, cudaStream_t s)
{
    switch (lanes) {
    case 1: return launch_scan<T, NT, 1, 16>(p, s);
    case 4: return launch_scan<T, NT, 4, 16>(p, s);
    default: return launch_scan<T, NT, 16, 16>(p, s);
    }
}

// Segments per channel group for the n-split kernel: when the channel groups
// fill less than half of the CTA slots of the GPU, the sequence is cut into
// up to 8 segments (one thread-block cluster per group) so that the grid
// fills one wave, keeping at least 4 chunks per segment.
int pick_segments(int64_t groups, int64_t L, int64_t lc, int64_t slots)
{
    const char *env = getenv("SS_SCAN_SEGMENTS");
    if (env) {
        const int v = atoi(env);
        if (v >= 1 && v <= 8)
            return v;
    }
    if (2 * groups > slots)
        return 1;
    int64_t n = slots / groups;
    n = n < 8 ? n : 8;
    const int64_t by_len = L / (4 * lc);
    n = n < by_len ? n : by_len;
    return n < 1 ? 1 : static_cast<int>(n);
}

template <typename T, int S>
ss_status launch_nsplit(const ScanParams &p0, cudaStream_t stream, int sms)
{
    using SH = NSplitShape<T, S>;
    auto kernel = scan_nsplit_kernel<T, S>;
    const size_t smem = SH::BYTES;
    if (smem > 48u * 1024u) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SS_ERR_LAUNCH, "cudaFuncSetAttribute failed: %s", cudaGetErrorString(e));
        }
    }
    ScanParams p = p0;
    const int64_t gpr = (p.d_inner + SH::CH - 1) / SH::CH;   // channel groups per batch row
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, SH::NT, smem) != cudaSuccess || occ < 1) {
        cudaGetLastError();
        occ = 1;
    }
    int nseg = pick_segments(gpr * p.batch, p.L, SH::LC, static_cast<int64_t>(sms) * occ);
    int64_t seg_len = (p.L + nseg - 1) / nseg;
    seg_len = (seg_len + SH::LC - 1) / SH::LC * SH::LC;
    nseg = static_cast<int>((p.L + seg_len - 1) / seg_len);
    if (gpr * nseg > 0x7fffffff || p.batch > 65535)
        return fail(SS_ERR_DIM, "grid too large: %lld channel blocks x %lld batch rows",
                    (long long)(gpr * nseg), (long long)p.batch);

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
            seg_len = p.L;
            cfg.gridDim.x = static_cast<unsigned>(gpr);
            cfg.attrs = nullptr;
            cfg.numAttrs = 0;
        }
    }
    p.nseg = nseg;
    p.seg_len = seg_len;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e == cudaSuccess)
        e = cudaGetLastError();
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SS_ERR_LAUNCH, "scan kernel launch failed: %s", cudaGetErrorString(e));
    }
    return SS_OK;
}

template <typename T>
ss_status dispatch_nsplit(const ScanParams &p, cudaStream_t s, int sms)
{
    if (p.N <= 4) return launch_nsplit<T, 1>(p, s, sms);
    if (p.N <= 8) return launch_nsplit<T, 2>(p, s, sms);
    if (p.N <= 16) return launch_nsplit<T, 4>(p, s, sms);
    return launch_nsplit<T, 8>(p, s, sms);
}

// The n-split kernel serves N <= 32 (cutting long sequences into segments
// when the channels alone do not fill the GPU); the time-lane kernel serves
// N > 32. SS_SCAN_KERNEL=nsplit|lanes overrides the choice.
bool use_nsplit(int64_t N)
{
    if (N > 32)
        return false;
    const char *env = getenv("SS_SCAN_KERNEL");
    if (env && strcmp(env, "lanes") == 0)
        return false;
    return true;
}

template <typename T>
ss_status scan_fwd(const void *x, const void *dt, const float *A, const void *B, const void *C,
                   const float *D, const void *z, const float *dt_bias, int softplus, void *y,
                   float *final_state, int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                   cudaStream_t stream)
{
    g_err[0] = '\0';
    if (batch <= 0 || d_inner <= 0 || L <= 0)
        return fail(SS_ERR_DIM, "sizes must be positive: batch=%lld d_inner=%lld L=%lld",
                    (long long)batch, (long long)d_inner, (long long)L);
    if (N < 1 || N > SS_MAX_N)
        return fail(SS_ERR_N, "N=%lld outside [1, %d]", (long long)N, SS_MAX_N);
    if (batch > (int64_t(1) << 40) / d_inner || batch * d_inner > (int64_t(1) << 50) / L)
        return fail(SS_ERR_DIM, "element count overflows");
    const PtrCheck list[] = {{x, "x", true},          {dt, "delta", true},  {A, "A", true},
                             {B, "B", true},          {C, "C", true},       {y, "y", true},
                             {D, "D", false},         {z, "z", false},      {dt_bias, "dt_bias", false},
                             {final_state, "final_state", false}};
    int dev = 0;
    ss_status st = check_ptrs(list, static_cast<int>(sizeof(list) / sizeof(list[0])), &dev);
    if (st != SS_OK)
        return st;

    ScanParams p;
    p.x = x; p.dt = dt; p.B = B; p.C = C; p.z = z;
    p.A = A; p.D = D; p.dt_bias = dt_bias;
    p.y = y; p.final_state = final_state;
    p.batch = batch; p.d_inner = d_inner; p.L = L; p.N = N;
    p.softplus = softplus ? 1 : 0;
    p.vec = (L % 16 == 0) && aligned16(x) && aligned16(dt) && aligned16(y) && (!z || aligned16(z));

    p.nseg = 1;
    p.seg_len = L;
    if (use_nsplit(N))
        return dispatch_nsplit<T>(p, stream, sm_count(dev));
    const int lanes = pick_lanes(batch * d_inner, L, sm_count(dev));
    if (N <= 4)
        return dispatch_scan_lanes<T, 4>(p, lanes, stream);
    if (N <= 16)
        return dispatch_scan_lanes<T, 16>(p, lanes, stream);
    return dispatch_scan_lanes<T, 64>(p, lanes, stream);
}

// ------------------------------------------------------------------ backward host side

constexpr int64_t kBwdHC = 16;   // steps per stored state (BwdShape::HC)

int64_t bwd_groups(int64_t N) { return N <= 4 ? 1 : (N <= 8 ? 2 : (N <= 16 ? 4 : 8)); }

size_t bwd_workspace_bytes(int64_t batch, int64_t d_inner, int64_t L, int64_t N)
{
    if (batch <= 0 || d_inner <= 0 || L <= 0 || N < 1 || N > 32)
        return 0;
    const int64_t nsub = (L + kBwdHC - 1) / kBwdHC;
    return static_cast<size_t>(batch) * nsub * bwd_groups(N) * d_inner * 16;
}

template <typename T, int S>
ss_status launch_bwd(const BwdParams &p, cudaStream_t stream)
{
    using SH = BwdShape<T, S>;
    auto kernel = scan_bwd_kernel<T, S>;
    const size_t smem = SH::BYTES;
    if (smem > 48u * 1024u) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SS_ERR_LAUNCH, "cudaFuncSetAttribute failed: %s", cudaGetErrorString(e));
        }
    }
    const int64_t gpr = (p.d_inner + SH::CH - 1) / SH::CH;
    if (gpr > 0x7fffffff || p.batch > 65535)
        return fail(SS_ERR_DIM, "grid too large: %lld channel blocks x %lld batch rows", (long long)gpr,
                    (long long)p.batch);
    kernel<<<dim3(static_cast<unsigned>(gpr), static_cast<unsigned>(p.batch)), SH::NT, smem, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SS_ERR_LAUNCH, "backward kernel launch failed: %s", cudaGetErrorString(e));
    return SS_OK;
}

template <typename T>
ss_status scan_bwd(const void *x, const void *dt, const float *A, const void *B, const void *C, const float *D,
                   const void *z, const float *dt_bias, int softplus, const float *h0, const void *dout,
                   const float *dfinal, void *dx, void *ddt, float *dA, float *dB, float *dC, float *dD, void *dz,
                   float *ddt_bias, float *dh0, void *workspace, size_t workspace_bytes, int64_t batch,
                   int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream)
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
                             {dh0, "dh0", false}};
    int dev = 0;
    ss_status st = check_ptrs(list, static_cast<int>(sizeof(list) / sizeof(list[0])), &dev);
    if (st != SS_OK)
        return st;
    if (workspace_bytes < need)
        return fail(SS_ERR_DIM, "workspace of %zu bytes is smaller than the %zu bytes required", workspace_bytes,
                    need);
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

    BwdParams p;
    p.x = x; p.dt = dt; p.B = B; p.C = C; p.z = z; p.dout = dout;
    p.A = A; p.D = D; p.dt_bias = dt_bias; p.h0 = h0; p.dfinal = dfinal;
    p.dx = dx; p.ddt = ddt; p.dz = z ? dz : nullptr;
    p.dA = dA; p.dB = dB; p.dC = dC; p.dD = D ? dD : nullptr; p.ddt_bias = ddt_bias; p.dh0 = dh0;
    p.ckpt = static_cast<float4 *>(workspace);
    p.batch = batch; p.d_inner = d_inner; p.L = L; p.N = N;
    p.nsub = (L + kBwdHC - 1) / kBwdHC;
    p.softplus = softplus ? 1 : 0;
    p.vec = (L % 16 == 0) && aligned16(x) && aligned16(dt) && aligned16(dout) && aligned16(dx) &&
            aligned16(ddt) && (!z || aligned16(z)) && (!p.dz || aligned16(p.dz));
    p.vec4 = (L % 4 == 0) && aligned16(dB) && aligned16(dC);
    const int64_t S = bwd_groups(N);
    if (S == 1) return launch_bwd<T, 1>(p, stream);
    if (S == 2) return launch_bwd<T, 2>(p, stream);
    if (S == 4) return launch_bwd<T, 4>(p, stream);
    return launch_bwd<T, 8>(p, stream);
}

template <typename T, int NQ>
ss_status launch_update(const UpdateParams &p, cudaStream_t stream)
{
    const int64_t threads = p.batch * p.d_inner * NQ;
    const int64_t blocks = (threads + kBlock - 1) / kBlock;
    if (blocks > 0x7fffffff)
        return fail(SS_ERR_DIM, "grid too large");
    state_update_kernel<T, NQ><<<static_cast<unsigned>(blocks), kBlock, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SS_ERR_LAUNCH, "state update launch failed: %s", cudaGetErrorString(e));
    return SS_OK;
}

template <typename T, int NV>
ss_status launch_update_rows(const UpdateParams &p, cudaStream_t stream)
{
    const int64_t blocks = (p.batch * p.d_inner + kBlock - 1) / kBlock;
    if (blocks > 0x7fffffff)
        return fail(SS_ERR_DIM, "grid too large");
    state_update_row_kernel<T, NV><<<static_cast<unsigned>(blocks), kBlock, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SS_ERR_LAUNCH, "state update launch failed: %s", cudaGetErrorString(e));
    return SS_OK;
}

template <typename T>
ss_status state_update(float *state, const void *x, const void *delta, const float *A, const void *B,
                       const void *C, const float *D, const void *z, void *y, int64_t batch,
                       int64_t d_inner, int64_t N, cudaStream_t stream)
{
    g_err[0] = '\0';
    if (batch <= 0 || d_inner <= 0)
        return fail(SS_ERR_DIM, "sizes must be positive: batch=%lld d_inner=%lld",
                    (long long)batch, (long long)d_inner);
    if (N < 1 || N > SS_MAX_N)
        return fail(SS_ERR_N, "N=%lld outside [1, %d]", (long long)N, SS_MAX_N);
    if (batch > (int64_t(1) << 40) / d_inner)
        return fail(SS_ERR_DIM, "element count overflows");
    const PtrCheck list[] = {{state, "state", true}, {x, "x", true}, {delta, "delta", true},
                             {A, "A", true},         {B, "B", true}, {C, "C", true},
                             {y, "y", true},         {D, "D", false}, {z, "z", false}};
    int dev = 0;
    ss_status st = check_ptrs(list, static_cast<int>(sizeof(list) / sizeof(list[0])), &dev);
    if (st != SS_OK)
        return st;
    UpdateParams p;
    p.state = state; p.x = x; p.delta = delta; p.B = B; p.C = C; p.z = z;
    p.A = A; p.D = D; p.y = y;
    p.batch = batch; p.d_inner = d_inner; p.N = N;
    p.vec = (N % 4 == 0) && aligned16(state) && aligned16(A);
    p.vec_bc = ((N * static_cast<int64_t>(sizeof(T))) % 16 == 0) && aligned16(B) && aligned16(C);
    if (p.vec && N <= 16) {
        switch (N / 4) {
        case 1: return launch_update_rows<T, 1>(p, stream);
        case 2: return launch_update_rows<T, 2>(p, stream);
        case 3: return launch_update_rows<T, 3>(p, stream);
        default: return launch_update_rows<T, 4>(p, stream);
        }
    }
    const int64_t nq = (N + 3) / 4;
    if (nq <= 1) return launch_update<T, 1>(p, stream);
    if (nq <= 2) return launch_update<T, 2>(p, stream);
    if (nq <= 4) return launch_update<T, 4>(p, stream);
    if (nq <= 8) return launch_update<T, 8>(p, stream);
    return launch_update<T, 16>(p, stream);
}

template <typename T, int K>
ss_status launch_conv(const ConvParams &p, cudaStream_t stream)
{
    constexpr int EPP = 16 / (int)sizeof(T);
    const int64_t pblocks = ((p.L + EPP - 1) / EPP + kBlock - 1) / kBlock;
    if (pblocks > 0x7fffffff)
        return fail(SS_ERR_DIM, "grid too large");
    if (p.vec) {
        constexpr int PT = kConvTileBytes / 16;
        const int64_t tblocks = (p.L / EPP + PT - 1) / PT;
        if (tblocks > 0x7fffffff || (p.d_inner + kConvRows - 1) / kConvRows > 65535)
            return fail(SS_ERR_DIM, "grid too large");
        const dim3 g(static_cast<unsigned>(tblocks),
                     static_cast<unsigned>((p.d_inner + kConvRows - 1) / kConvRows),
                     static_cast<unsigned>(std::min<int64_t>(p.batch, 65535)));
        causal_conv1d_tile_kernel<T, K><<<g, kBlock, 0, stream>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return fail(SS_ERR_LAUNCH, "conv launch failed: %s", cudaGetErrorString(e));
        return SS_OK;
    }
    constexpr int R = 2;
    const dim3 grid(static_cast<unsigned>(pblocks),
                    static_cast<unsigned>(std::min<int64_t>((p.d_inner + R - 1) / R, 65535)),
                    static_cast<unsigned>(std::min<int64_t>(p.batch, 65535)));
    causal_conv1d_kernel<T, K, R><<<grid, kBlock, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SS_ERR_LAUNCH, "conv launch failed: %s", cudaGetErrorString(e));
    return SS_OK;
}

template <typename T>
ss_status causal_conv1d(const void *x, const float *w, const float *bias, const void *state_in, int silu, void *out,
                        void *state_out, int64_t batch, int64_t d_inner, int64_t L, int64_t k, cudaStream_t stream)
{
    g_err[0] = '\0';
    if (batch <= 0 || d_inner <= 0 || L <= 0)
        return fail(SS_ERR_DIM, "sizes must be positive: batch=%lld d_inner=%lld L=%lld",
                    (long long)batch, (long long)d_inner, (long long)L);
    if (k < 1 || k > SS_MAX_CONV_K)
        return fail(SS_ERR_DIM, "k=%lld outside [1, %d]", (long long)k, SS_MAX_CONV_K);
    if (batch > (int64_t(1) << 40) / d_inner || batch * d_inner > (int64_t(1) << 50) / L)
        return fail(SS_ERR_DIM, "element count overflows");
    const PtrCheck list[] = {{x, "x", true}, {w, "w", true}, {out, "out", true}, {bias, "bias", false},
                             {state_in, "state_in", false}, {state_out, "state_out", false}};
    int dev = 0;
    ss_status st = check_ptrs(list, static_cast<int>(sizeof(list) / sizeof(list[0])), &dev);
    if (st != SS_OK)
        return st;
    ConvParams p;
    p.x = x; p.state_in = k > 1 ? state_in : nullptr; p.w = w; p.bias = bias;
    p.out = out; p.state_out = k > 1 ? state_out : nullptr;
    p.batch = batch; p.d_inner = d_inner; p.L = L; p.silu = silu ? 1 : 0;
    p.vec = ((L * static_cast<int64_t>(sizeof(T))) % 16 == 0) && aligned16(x) && aligned16(out);
    switch (k) {
    case 1: return launch_conv<T, 1>(p, stream);
    case 2: return launch_conv<T, 2>(p, stream);
    case 3: return launch_conv<T, 3>(p, stream);
    case 4: return launch_conv<T, 4>(p, stream);
    case 5: return launch_conv<T, 5>(p, stream);
    case 6: return launch_conv<T, 6>(p, stream);
    case 7: return launch_conv<T, 7>(p, stream);
    default: return launch_conv<T, 8>(p, stream);
    }
}

template <typename T, int K>
ss_status launch_conv_step(const ConvStepParams &p, cudaStream_t stream)
{
    const int64_t per = p.vec ? 2 : 1;
    const int64_t rows = p.vec ? (p.batch + kStepRows - 1) / kStepRows : p.batch;
    const int64_t dblocks = ((p.d_inner + per - 1) / per + kBlock - 1) / kBlock;
    if (dblocks > 0x7fffffff)
        return fail(SS_ERR_DIM, "grid too large");
    const dim3 grid(static_cast<unsigned>(dblocks), static_cast<unsigned>(std::min<int64_t>(rows, 65535)));
    conv_state_update_kernel<T, K><<<grid, kBlock, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SS_ERR_LAUNCH, "conv step launch failed: %s", cudaGetErrorString(e));
    return SS_OK;
}

template <typename T>
ss_status conv_state_update(void *state, const void *x, const float *w, const float *bias, int silu, void *out,
                            int64_t batch, int64_t d_inner, int64_t k, cudaStream_t stream)
{
    g_err[0] = '\0';
    if (batch <= 0 || d_inner <= 0)
        return fail(SS_ERR_DIM, "sizes must be positive: batch=%lld d_inner=%lld", (long long)batch,
                    (long long)d_inner);
    if (k < 1 || k > SS_MAX_CONV_K)
        return fail(SS_ERR_DIM, "k=%lld outside [1, %d]", (long long)k, SS_MAX_CONV_K);
    if (batch > (int64_t(1) << 40) / d_inner)
        return fail(SS_ERR_DIM, "element count overflows");
    const PtrCheck list[] = {{x, "x", true}, {w, "w", true}, {out, "out", true},
                             {state, "conv_state", k > 1}, {bias, "bias", false}};
    int dev = 0;
    ss_status st = check_ptrs(list, static_cast<int>(sizeof(list) / sizeof(list[0])), &dev);
    if (st != SS_OK)
        return st;
    ConvStepParams p;
    p.state = state; p.x = x; p.w = w; p.bias = bias; p.out = out;
    p.batch = batch; p.d_inner = d_inner; p.silu = silu ? 1 : 0;
    const uintptr_t pair_bytes = 2 * sizeof(T);
    p.vec = (d_inner % 2 == 0) && reinterpret_cast<uintptr_t>(x) % pair_bytes == 0 &&
            reinterpret_cast<uintptr_t>(out) % pair_bytes == 0 &&
            (k == 1 || reinterpret_cast<uintptr_t>(state) % pair_bytes == 0);
    switch (k) {
    case 1: return launch_conv_step<T, 1>(p, stream);
    case 2: return launch_conv_step<T, 2>(p, stream);
    case 3: return launch_conv_step<T, 3>(p, stream);
    case 4: return launch_conv_step<T, 4>(p, stream);
    case 5: return launch_conv_step<T, 5>(p, stream);
    case 6: return launch_conv_step<T, 6>(p, stream);
    case 7: return launch_conv_step<T, 7>(p, stream);
    default: return launch_conv_step<T, 8>(p, stream);
    }
}

}  // namespace

// ------------------------------------------------------------------ C ABI

extern "C" {

ss_status ss_scan_fwd_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A, const ss_bf16 *B,
                           const ss_bf16 *C, const float *D, const ss_bf16 *z, const float *dt_bias,
                           int delta_softplus, ss_bf16 *y, float *final_state, int64_t batch,
                           int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream)
{
    return scan_fwd<__nv_bfloat16>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, y, final_state,
                                   batch, d_inner, L, N, stream);
}

ss_status ss_scan_fwd_f32(const float *x, const float *delta, const float *A, const float *B,
                          const float *C, const float *D, const float *z, const float *dt_bias,
                          int delta_softplus, float *y, float *final_state, int64_t batch,
                          int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream)
{
    return scan_fwd<float>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, y, final_state, batch,
                           d_inner, L, N, stream);
}

ss_status ss_state_update_bf16(float *state, const ss_bf16 *x, const ss_bf16 *delta, const float *A,
                               const ss_bf16 *B, const ss_bf16 *C, const float *D, const ss_bf16 *z,
                               ss_bf16 *y, int64_t batch, int64_t d_inner, int64_t N,
                               cudaStream_t stream)
{
    return state_update<__nv_bfloat16>(state, x, delta, A, B, C, D, z, y, batch, d_inner, N, stream);
}

ss_status ss_state_update_f32(float *state, const float *x, const float *delta, const float *A,
                              const float *B, const float *C, const float *D, const float *z, float *y,
                              int64_t batch, int64_t d_inner, int64_t N, cudaStream_t stream)
{
    return state_update<float>(state, x, delta, A, B, C, D, z, y, batch, d_inner, N, stream);
}

ss_status ss_causal_conv1d_bf16(const ss_bf16 *x, const float *w, const float *bias, const ss_bf16 *state_in,
                                int silu, ss_bf16 *out, ss_bf16 *state_out, int64_t batch, int64_t d_inner,
                                int64_t L, int64_t k, cudaStream_t stream)
{
    return causal_conv1d<__nv_bfloat16>(x, w, bias, state_in, silu, out, state_out, batch, d_inner, L, k, stream);
}

ss_status ss_causal_conv1d_f32(const float *x, const float *w, const float *bias, const float *state_in, int silu,
                               float *out, float *state_out, int64_t batch, int64_t d_inner, int64_t L, int64_t k,
                               cudaStream_t stream)
{
    return causal_conv1d<float>(x, w, bias, state_in, silu, out, state_out, batch, d_inner, L, k, stream);
}

ss_status ss_conv_state_update_bf16(ss_bf16 *conv_state, const ss_bf16 *x, const float *w, const float *bias,
                                    int silu, ss_bf16 *out, int64_t batch, int64_t d_inner, int64_t k,
                                    cudaStream_t stream)
{
    return conv_state_update<__nv_bfloat16>(conv_state, x, w, bias, silu, out, batch, d_inner, k, stream);
}

ss_status ss_conv_state_update_f32(float *conv_state, const float *x, const float *w, const float *bias, int silu,
                                   float *out, int64_t batch, int64_t d_inner, int64_t k, cudaStream_t stream)
{
    return conv_state_update<float>(conv_state, x, w, bias, silu, out, batch, d_inner, k, stream);
}

size_t ss_scan_bwd_workspace_bytes(int64_t batch, int64_t d_inner, int64_t L, int64_t N)
{
    return bwd_workspace_bytes(batch, d_inner, L, N);
}

ss_status ss_scan_bwd_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A, const ss_bf16 *B,
                           const ss_bf16 *C, const float *D, const ss_bf16 *z, const float *dt_bias,
                           int delta_softplus, const float *h0, const ss_bf16 *dout, const float *dfinal_state,
                           ss_bf16 *dx, ss_bf16 *ddelta, float *dA, float *dB, float *dC, float *dD, ss_bf16 *dz,
                           float *ddt_bias, float *dh0, void *workspace, size_t workspace_bytes, int64_t batch,
                           int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream)
{
    return scan_bwd<__nv_bfloat16>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, dout, dfinal_state, dx,
                                   ddelta, dA, dB, dC, dD, dz, ddt_bias, dh0, workspace, workspace_bytes, batch,
                                   d_inner, L, N, stream);
}

ss_status ss_scan_bwd_f32(const float *x, const float *delta, const float *A, const float *B, const float *C,
                          const float *D, const float *z, const float *dt_bias, int delta_softplus, const float *h0,
                          const float *dout, const float *dfinal_state, float *dx, float *ddelta, float *dA,
                          float *dB, float *dC, float *dD, float *dz, float *ddt_bias, float *dh0, void *workspace,
                          size_t workspace_bytes, int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                          cudaStream_t stream)
{
    return scan_bwd<float>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, dout, dfinal_state, dx, ddelta,
                           dA, dB, dC, dD, dz, ddt_bias, dh0, workspace, workspace_bytes, batch, d_inner, L, N,
                           stream);
}

const char *ss_last_error(void) { return g_err; }

int ss_abi_version(void) { return SS_ABI_VERSION; }

}  // extern "C"
