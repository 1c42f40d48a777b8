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

#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "ss_scan.h"

namespace {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr float kLn2 = 0.6931471805599453f;    // ln(2)

// ------------------------------------------------------------------ device math

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2_approx(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(v) = log(1 + e^v) = max(v, 0) + log1p(e), e = e^{-|v|} in (0, 1].
// log1p(e) is taken from its alternating Taylor series when e <= 1/16
// (five terms; the first omitted term e^6/6 is below 2^-24 relative), and
// otherwise as ln2 * log2(u) - r with u = fl(1 + e) and r = (u - 1) - e, the
// exact rounding error of 1 + e (Sterbenz), which removes the cancellation of
// log2(1 + e) to first order. Finite for every finite v.
__device__ __forceinline__ float softplus_f(float v)
{
    const float e = ex2_approx(-fabsf(v) * kLog2e);
    const float series = e * fmaf(e, fmaf(e, fmaf(e, fmaf(e, 0.2f, -0.25f), 1.0f / 3.0f), -0.5f), 1.0f);
    const float u = 1.0f + e;
    const float r = (u - 1.0f) - e;
    const float viaLog = fmaf(lg2_approx(u), kLn2, -r);
    return fmaxf(v, 0.0f) + (e <= 0.0625f ? series : viaLog);
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
    int vec;  // 16-byte vector loads/stores allowed
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

// ------------------------------------------------------------------ decode kernel

struct UpdateParams {
    float *state;
    const void *x, *delta, *B, *C, *z;
    const float *A, *D;
    void *y;
    int64_t batch, d_inner, N;
    int vec;  // N % 4 == 0 and 16-byte aligned state/A, 8-byte aligned B/C
};

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

    const int lanes = pick_lanes(batch * d_inner, L, sm_count(dev));
    if (N <= 4)
        return dispatch_scan_lanes<T, 4>(p, lanes, stream);
    if (N <= 16)
        return dispatch_scan_lanes<T, 16>(p, lanes, stream);
    return dispatch_scan_lanes<T, 64>(p, lanes, stream);
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
    const int64_t nq = (N + 3) / 4;
    if (nq <= 1) return launch_update<T, 1>(p, stream);
    if (nq <= 2) return launch_update<T, 2>(p, stream);
    if (nq <= 4) return launch_update<T, 4>(p, stream);
    if (nq <= 8) return launch_update<T, 8>(p, stream);
    return launch_update<T, 16>(p, stream);
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

const char *ss_last_error(void) { return g_err; }

int ss_abi_version(void) { return SS_ABI_VERSION; }

}  // extern "C"
