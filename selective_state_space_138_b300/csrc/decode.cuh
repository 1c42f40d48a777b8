// decode.cuh -- the single-token decode state update and its launch logic.
//
// Part of the single translation unit ss_scan.cu (included inside its
// anonymous namespace); not compiled on its own.

#pragma once

// ------------------------------------------------------------------ decode kernel

struct UpdateParams {
    float *state;
    const void *x, *delta, *B, *C, *z;
    const float *A, *D;
    void *y;
    int64_t batch, d_inner, N;
    int vec;     // N % 4 == 0 and 16-byte aligned state and A
    int vec_bc;  // B and C rows are whole 16-byte words (16-byte aligned, N * sizeof(T) % 16 == 0)
    // N = 16 kernel with tensor copies: the state as (16, d_inner, batch) fp32 with a
    // box of 128 channels of one batch row and the 64-byte swizzle; B, C as (16, batch)
    // with a box of kDecRows rows
    CUtensorMap tm_state, tm_B, tm_C;
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

// N = 16 with 16-byte rows (the decode workload): grid = (channel blocks,
// groups of kDecRows batch rows); a thread owns channel d of kDecRows batch
// rows. The fp32 states of all its rows, and B, C of the batch rows, are
// requested at once with cp.async into shared memory (no registers held while
// they are in flight, so ~200 KB per SM is outstanding), the per-row scalars
// are loaded together, A of the channel once for all rows; each row is then
// updated from its staged state and written straight back. State pieces are
// XOR-swizzled so that the row reads are free of bank conflicts.
constexpr int kDecRows = 4;

// TMA: the states and B, C arrive by tensor copies instead: one thread issues
// a box of 128 channels per batch row with the 64-byte swizzle (16-byte piece
// v of a channel's 64 bytes at v ^ ((channel >> 1) & 3), the layout the pieces
// use) and the rows' B and C, completing on one barrier (bounded wait).
template <typename T, bool TMA>
__global__ void __launch_bounds__(kBlock)
state_update_rows16_kernel(const __grid_constant__ UpdateParams p)
{
    constexpr int NV = 4, R = kDecRows;
    constexpr int BCP = 2 * 16 * (int)sizeof(T) / 16;   // 16-byte pieces of one batch row's B and C
    __shared__ __align__(1024) float4 sst[R * kBlock * NV];
    __shared__ __align__(128) T sbc[R * 2 * 16];       // pieces: [row][B, C][16]; copies: [B, C][row][16]
    __shared__ __align__(8) uint64_t dec_bar;
    const uint32_t sst_s = static_cast<uint32_t>(__cvta_generic_to_shared(sst));
    const uint32_t sbc_s = static_cast<uint32_t>(__cvta_generic_to_shared(sbc));
    const uint32_t bar_s = static_cast<uint32_t>(__cvta_generic_to_shared(&dec_bar));
    if (TMA && ((sst_s & 1023u) != 0 || (sbc_s & 127u) != 0)) {   // the swizzle and the copies need these
        if (threadIdx.x == 0)
            atomicOr(&g_fault_flags, kFaultSmemAlign);
        return;
    }
    bool aborted = false;
    int waits = 0;
    if (TMA) {
        if (threadIdx.x == 0) {
            mbar_init(bar_s, 1);
            mbar_fence_init();
        }
        __syncthreads();
    }
    const int r = threadIdx.x;
    const int64_t d = static_cast<int64_t>(blockIdx.x) * kBlock + r;
    const bool act = d < p.d_inner;
    const int64_t dd = act ? d : 0;
    const int sw = (r >> 1) & 3;
    float4 a[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v)
        a[v] = __ldg(reinterpret_cast<const float4 *>(p.A + dd * 16) + v);
    const float Dd = p.D ? __ldg(p.D + dd) : 0.0f;
    for (int64_t b0 = static_cast<int64_t>(blockIdx.y) * R; b0 < p.batch;
         b0 += static_cast<int64_t>(gridDim.y) * R) {
        // the states of this thread's R rows, and B, C of the R batch rows, into shared memory
        if constexpr (TMA) {
            if (r == 0 && !aborted) {
                mbar_expect_tx(bar_s, R * kBlock * 64 + 2 * R * 16 * (int)sizeof(T));
                const int c1 = static_cast<int>(blockIdx.x) * kBlock;
#pragma unroll
                for (int k = 0; k < R; ++k)
                    tma_load_3d(sst_s + k * kBlock * 64, &p.tm_state, bar_s, 0, c1, static_cast<int>(b0 + k));
                tma_load_3d(sbc_s, &p.tm_B, bar_s, 0, static_cast<int>(b0), 0);
                tma_load_3d(sbc_s + R * 16 * (int)sizeof(T), &p.tm_C, bar_s, 0, static_cast<int>(b0), 0);
            }
        } else {
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const int64_t b = b0 + k;
            const bool ok = act && b < p.batch;
            const float4 *st = reinterpret_cast<const float4 *>(p.state + ((ok ? b : 0) * p.d_inner + dd) * 16);
#pragma unroll
            for (int v = 0; v < NV; ++v)
                cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(&sst[(k * kBlock + r) * NV + (v ^ sw)])),
                           st + v, ok ? 16 : 0);
        }
        if (r < R * BCP) {
            const int k = r / BCP, piece = r % BCP;   // pieces of B first, then C
            const int half = piece / (BCP / 2), pp = piece % (BCP / 2);
            const int64_t b = b0 + k;
            const bool ok = b < p.batch;
            const T *src = static_cast<const T *>(half ? p.C : p.B) + (ok ? b : 0) * 16 + pp * (16 / (int)sizeof(T));
            cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(sbc + (k * 2 + half) * 16 +
                                                                       pp * (16 / (int)sizeof(T)))),
                       src, ok ? 16 : 0);
        }
        cp_async_commit();
        }
        float xv[R], dlv[R], zv[R];
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const int64_t b = b0 + k;
            const bool ok = act && b < p.batch;
            const int64_t row = (ok ? b : 0) * p.d_inner + dd;
            xv[k] = ok ? Io<T>::load1(static_cast<const T *>(p.x) + row) : 0.0f;
            dlv[k] = ok ? Io<T>::load1(static_cast<const T *>(p.delta) + row) : 0.0f;
            zv[k] = (ok && p.z) ? Io<T>::load1(static_cast<const T *>(p.z) + row) : 0.0f;
        }
        if constexpr (TMA) {
            if (!aborted)
                aborted = !mbar_wait(bar_s, static_cast<uint32_t>(waits & 1));
            ++waits;
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();   // B and C were staged by a few threads for all
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const int64_t b = b0 + k;
            if (!act || b >= p.batch)
                continue;
            const int64_t row = b * p.d_inner + d;
            float bv[16], cv[16];
            // B then C of row k (pieces: [row][B, C], copies: [B, C][row])
            const uint4 *sb = reinterpret_cast<const uint4 *>(sbc + (TMA ? k : k * 2) * 16);
            const uint4 *sc = reinterpret_cast<const uint4 *>(sbc + (TMA ? R * 16 + k * 16 : k * 2 * 16 + 16));
#pragma unroll
            for (int e = 0; e < 16 / Io<T>::kPerVec; ++e) {   // plain shared loads, one address for all threads
                unpack_piece<T>(sb[e], bv + e * Io<T>::kPerVec);
                unpack_piece<T>(sc[e], cv + e * Io<T>::kPerVec);
            }
            const float dx = dlv[k] * xv[k], dl2 = dlv[k] * kLog2e;
            float out = 0.0f;
            float4 *so = reinterpret_cast<float4 *>(p.state + row * 16);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                float4 h = sst[(k * kBlock + r) * NV + (v ^ sw)];
                float *hv = reinterpret_cast<float *>(&h);
                const float *av = reinterpret_cast<const float *>(&a[v]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int n = 4 * v + e;
                    hv[e] = fmaf(ex2_approx(dl2 * av[e]), hv[e], dx * bv[n]);
                    out = fmaf(cv[n], hv[e], out);
                }
                so[v] = h;
            }
            out = fmaf(Dd, xv[k], out);
            if (p.z)
                out *= silu_f(zv[k]);
            Io<T>::store1(static_cast<T *>(p.y) + row, out);
        }
        __syncthreads();   // the staged B, C (and states) are reused by the next group of rows
    }
    if (TMA && threadIdx.x == 0 && aborted)   // the copies whose wait gave up: let them land (bounded)
        mbar_wait(bar_s, static_cast<uint32_t>((waits - 1) & 1));
}

// 3-d tensor map with box (b0, b1, 1); elements outside the tensor read as zero
bool encode_dec_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, CUtensorMapSwizzle swz)
{
    const EncodeTiledFn fn = encode_tiled_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1, s2};
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The N = 16 kernel's maps (SS_SCAN_TMA=0 keeps the cp.async pieces).
template <typename T>
bool encode_dec_maps(UpdateParams &p)
{
    const char *env = getenv("SS_SCAN_TMA");
    if (env && strcmp(env, "0") == 0)
        return false;
    const uint64_t D = static_cast<uint64_t>(p.d_inner), Bt = static_cast<uint64_t>(p.batch);
    const CUtensorMapDataType io = sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const uint64_t row = 16 * sizeof(T);
    return encode_dec_map(&p.tm_state, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.state, 16, D, Bt, 64, D * 64, 16, kBlock,
                          CU_TENSOR_MAP_SWIZZLE_64B) &&
           encode_dec_map(&p.tm_B, io, p.B, 16, Bt, 1, row, row * Bt, 16, kDecRows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           encode_dec_map(&p.tm_C, io, p.C, 16, Bt, 1, row, row * Bt, 16, kDecRows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <typename T>
ss_status launch_update_rows16(UpdateParams p, cudaStream_t stream)
{
    const int64_t dblocks = (p.d_inner + kBlock - 1) / kBlock;
    const int64_t groups = (p.batch + kDecRows - 1) / kDecRows;
    if (dblocks > 0x7fffffff)
        return fail(SS_ERR_DIM, "grid too large");
    const dim3 grid(static_cast<unsigned>(dblocks), static_cast<unsigned>(std::min<int64_t>(groups, 65535)));
    if (encode_dec_maps<T>(p))
        state_update_rows16_kernel<T, true><<<grid, kBlock, 0, stream>>>(p);
    else
        state_update_rows16_kernel<T, false><<<grid, kBlock, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SS_ERR_LAUNCH, "state update launch failed: %s", cudaGetErrorString(e));
    return SS_OK;
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
    UpdateParams p{};
    p.state = state; p.x = x; p.delta = delta; p.B = B; p.C = C; p.z = z;
    p.A = A; p.D = D; p.y = y;
    p.batch = batch; p.d_inner = d_inner; p.N = N;
    p.vec = (N % 4 == 0) && aligned16(state) && aligned16(A);
    p.vec_bc = ((N * static_cast<int64_t>(sizeof(T))) % 16 == 0) && aligned16(B) && aligned16(C);
    const char *env = getenv("SS_DECODE_KERNEL");
    if (p.vec && p.vec_bc && N == 16 && !(env && strcmp(env, "rows") == 0))
        return launch_update_rows16<T>(p, stream);
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
