// conv.cuh -- the causal depthwise convolution (+ SiLU), its decode step, and their launch logic.
//
// Part of the single translation unit ss_scan.cu (included inside its
// anonymous namespace); not compiled on its own.

#pragma once

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
// CG channels x PT pieces of one batch row, plus the HP pieces before them,
// into shared memory with asynchronous 16-byte copies (no registers held while
// the loads are in flight). Then 16 threads share a row, each turning PPL
// consecutive pieces into outputs: the last K-1 inputs ride along in
// registers from one piece to the next, so each input is unpacked once, and
// the channel's taps and bias are read once. Outputs overwrite their own
// input pieces in shared memory and leave for HBM with consecutive threads on
// consecutive pieces. Pieces are stored XOR-swizzled within groups of 8
// (piece j at column (j & ~7) | ((j ^ (j >> 3)) & 7)), so that the 16 threads
// of a row, reading pieces PPL apart, hit distinct banks. Inputs before t = 0
// come from the carried history (or are zero).
constexpr int kConvTileBytes = 2048;   // one row of a tile
constexpr int kConvRows = 8;           // channels per tile

__device__ __forceinline__ int conv_swz(int j) { return (j & ~7) | ((j ^ (j >> 3)) & 7); }

// 16 bytes of outputs in the io type
template <typename T>
__device__ __forceinline__ uint4 conv_pack(const float *o)
{
    uint4 w;
    if constexpr (sizeof(T) == 4) {
        w = make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]), __float_as_uint(o[3]));
    } else {
        w.x = pack_bf16x2(o[0], o[1]);
        w.y = pack_bf16x2(o[2], o[3]);
        w.z = pack_bf16x2(o[4], o[5]);
        w.w = pack_bf16x2(o[6], o[7]);
    }
    return w;
}

template <typename T, int K>
__global__ void __launch_bounds__(kBlock)
causal_conv1d_tile_kernel(const ConvParams p)
{
    constexpr int EPP = 16 / (int)sizeof(T);
    constexpr int H = K - 1;
    constexpr int HP = (H + EPP - 1) / EPP;      // halo pieces
    constexpr int PT = kConvTileBytes / 16;      // pieces per tile row
    constexpr int CG = kConvRows;
    constexpr int LPR = kBlock / CG;             // threads per row
    constexpr int PPL = PT / LPR;                // consecutive pieces per thread
    static_assert(PT % LPR == 0 && PPL % 8 == 0 && kBlock % CG == 0, "tile shape");
    __shared__ __align__(16) uint4 tile[CG][HP + PT];   // [halo pieces][swizzled pieces]

    const int64_t npieces = p.L / EPP;
    const int64_t pc0 = static_cast<int64_t>(blockIdx.x) * PT;
    const int64_t d0 = static_cast<int64_t>(blockIdx.y) * CG;
    const T *x = static_cast<const T *>(p.x);
    const int r = threadIdx.x / LPR;             // compute role: row r, pieces j0 .. j0 + PPL - 1
    const int j0 = (threadIdx.x % LPR) * PPL;
    const int64_t d = d0 + r;
    const bool act = d < p.d_inner;
    float wd[K];
#pragma unroll
    for (int k = 0; k < K; ++k)
        wd[k] = act ? __ldg(p.w + d * K + k) : 0.0f;
    const float bv = (act && p.bias) ? __ldg(p.bias + d) : 0.0f;

    for (int64_t b = blockIdx.z; b < p.batch; b += gridDim.z) {
#pragma unroll
        for (int rr = 0; rr < CG; ++rr) {
            const int64_t dr = d0 + rr;
            for (int jj = threadIdx.x; jj < HP + PT; jj += kBlock) {
                const int64_t pc = jj < HP ? pc0 - HP + jj : pc0 + (jj - HP);
                const int col = jj < HP ? jj : HP + conv_swz(jj - HP);
                const bool ok = dr < p.d_inner && pc >= 0 && pc < npieces;
                const T *src = ok ? x + (b * p.d_inner + dr) * p.L + pc * EPP : x;
                cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(&tile[rr][col])), src, ok ? 16 : 0);
            }
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        const bool work = act && pc0 + j0 < npieces;
        // the H inputs before piece j0: hist[i] is input (H - i) steps back
        float hist[H > 0 ? H : 1];
        if (work) {
            float pv[HP * EPP > 0 ? HP * EPP : 1];
#pragma unroll
            for (int v = 0; v < HP; ++v) {
                const int jp = j0 - HP + v;   // piece index within the tile, negative in the halo
                const uint4 w = jp < 0 ? tile[r][HP + jp] : tile[r][HP + conv_swz(jp)];
                unpack_piece<T>(w, pv + v * EPP);
            }
#pragma unroll
            for (int i = 0; i < H; ++i)
                hist[i] = pv[HP * EPP - H + i];
            if (pc0 + j0 == 0 && p.state_in) {   // steps before 0 come from the carried history
#pragma unroll
                for (int i = 0; i < H; ++i)
                    hist[i] = Io<T>::load1(static_cast<const T *>(p.state_in) + (b * H + i) * p.d_inner + d);
            }
        }
        __syncthreads();   // every thread has its history: pieces may now be overwritten by outputs
        if (work) {
#pragma unroll 2
            for (int m = 0; m < PPL; ++m) {
                const int j = j0 + m;
                const int64_t pc = pc0 + j;
                if (pc >= npieces)
                    break;
                float v[EPP];
                unpack_piece<T>(tile[r][HP + conv_swz(j)], v);
                float o[EPP];
#pragma unroll
                for (int e = 0; e < EPP; ++e) {
                    float acc = bv;
#pragma unroll
                    for (int k = 0; k < K; ++k)
                        acc = fmaf(wd[k], e - k >= 0 ? v[e - k >= 0 ? e - k : 0] : hist[H + e - k >= 0 ? H + e - k : 0],
                                   acc);
                    o[e] = p.silu ? silu_f(acc) : acc;
                }
                tile[r][HP + conv_swz(j)] = conv_pack<T>(o);   // in place; to HBM below
                // the last H inputs become the history of the next piece
                float nh[H > 0 ? H : 1];
#pragma unroll
                for (int i = 0; i < H; ++i) {
                    const int u = EPP - H + i;   // window index relative to v
                    nh[i] = u >= 0 ? v[u >= 0 ? u : 0] : hist[H + u >= 0 ? H + u : 0];
                }
#pragma unroll
                for (int i = 0; i < H; ++i)
                    hist[i] = nh[i];
                if (H > 0 && p.state_out && pc == npieces - 1) {
#pragma unroll
                    for (int i = 0; i < H; ++i)
                        Io<T>::store1(static_cast<T *>(p.state_out) + (b * H + i) * p.d_inner + d, hist[i]);
                }
            }
        }
        __syncthreads();
        // outputs to HBM, consecutive threads on consecutive pieces of a row
#pragma unroll
        for (int rr = 0; rr < CG; ++rr) {
            const int64_t dr = d0 + rr;
            if (dr >= p.d_inner)
                break;
            T *orow = static_cast<T *>(p.out) + (b * p.d_inner + dr) * p.L;
            for (int jj = threadIdx.x; jj < PT; jj += kBlock) {
                const int64_t pc = pc0 + jj;
                if (pc < npieces)
                    *reinterpret_cast<uint4 *>(orow + pc * EPP) = tile[rr][HP + conv_swz(jj)];
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
