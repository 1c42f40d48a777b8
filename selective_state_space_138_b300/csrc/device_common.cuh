// device_common.cuh -- device math, io conversion, packed f32x2 pairs and cp.async helpers shared by every kernel.
//
// Part of the single translation unit ss_scan.cu (included inside its
// anonymous namespace); not compiled on its own.

#pragma once

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


constexpr int kBlock = 128;

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

__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void *gsrc, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_dst), "l"(gsrc), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int PENDING>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(PENDING) : "memory"); }

// ------------------------------------------------------------------ mbarriers and tensor copies
//
// Tiles are brought into shared memory by the tensor-memory accelerator
// (cp.async.bulk.tensor) and signal an mbarrier with the bytes they deliver.
// Every wait on such a barrier is bounded: after kWaitLimitNs it sets
// kFaultWaitTimeout in g_fault_flags (read by the host through
// ss_device_faults) and gives up, so that a copy that never lands cannot hang
// the GPU.

constexpr unsigned int kFaultWaitTimeout = 1u;
// A kernel that stages its tiles by tensor copies found its dynamic shared
// memory off the 128-byte boundary the copies need (SS_FAULT_SMEM_ALIGN).
constexpr unsigned int kFaultSmemAlign = 2u;
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // one second
__device__ unsigned int g_fault_flags;

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// makes initialised barriers visible to the tensor copies (the async proxy)
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// waits until the phase of the barrier with this parity has completed;
// false (and the fault flag set) if it did not within kWaitLimitNs
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_fault_flags, kFaultWaitTimeout);
            return false;
        }
    }
    return true;
}

// tile (c0, c1, c2) of a 3-d tensor map into shared memory at dst, completing
// on the barrier bar
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, uint32_t bar, int c0, int c1, int c2)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

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
