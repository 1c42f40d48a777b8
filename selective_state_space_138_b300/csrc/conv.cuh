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
    CUtensorMap tm_x, tm_out;   // (L, d_inner, batch) boxes of 128 bytes x kConvRows channels, 128-byte swizzle
    const void *x, *state_in;
    const float *w, *bias;
    void *out, *state_out;
    int64_t batch, d_inner, L;
    int silu;
    int vec;  // 16-byte aligned rows of whole pieces
    int tma;  // tm_x and tm_out are encoded: the tile kernel runs
    int ntt, ngr, ntiles;   // tile kernel: tiles of steps per row, channel groups, tiles (below 2^31)
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

// Aligned rows (16-byte aligned x and out, rows a whole number of 16-byte
// pieces): tensor copies and persistent CTAs. A tile is kConvRows channels x
// kConvSegs segments of 128 bytes of one batch row. Each segment arrives as
// one box of 8 channel rows x 128 bytes with the 128-byte swizzle (16-byte
// chunk c of channel row ch at ch * 128 + ((c ^ ch) * 16)), and one more box,
// the segment just before the tile, gives the first segment its k-1 inputs of
// history (inputs before t = 0 come from the carried history or are zero).
// A CTA walks its tiles through a ring of kConvStages stages with two roles:
// four compute warps, in which thread (s, ch) = (tid / 8, tid % 8) turns
// segment s of channel ch into outputs piece by piece (the last k-1 inputs
// ride along in registers; the 8 channels of a quarter-warp sit on different
// chunks, so its 16-byte shared-memory accesses are free of bank conflicts),
// writing them over their inputs; and one copy warp, which sends each
// computed tile out with tensor stores and refills its stage with the tensor
// loads of the tile kConvStages further on.
constexpr int kConvRows = 8;     // channels per tile (rows of a box)
constexpr int kConvSegs = 16;    // 128-byte segments per tile row
constexpr int kConvStages = 3;   // tiles in the ring
constexpr int kConvThreads = kBlock + 32;   // four compute warps and the copy warp

template <typename T>
struct ConvTileShape {
    static constexpr int EPP = 16 / (int)sizeof(T);     // elements per 16-byte piece
    static constexpr int SEGE = 128 / (int)sizeof(T);   // elements per segment
    static constexpr int TT = kConvSegs * SEGE;         // steps per tile
    static constexpr int BOX = kConvRows * 128;         // bytes of one box
    static constexpr int STAGE = (kConvSegs + 1) * BOX; // the halo box, then the tile's boxes
    static constexpr int BYTES = 1024 + kConvStages * STAGE + 2 * kConvStages * 8;   // with the alignment slack
    static_assert(kConvRows * kConvSegs == kBlock, "one thread per (segment, channel)");
};

__device__ __forceinline__ void conv_fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// box (c0, c1, c2) of a 3-d tensor map from shared memory at src to global memory
__device__ __forceinline__ void conv_tma_store_3d(const void *tmap, uint32_t src, int c0, int c1, int c2)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void conv_mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// barrier 1 over the four compute warps (barrier 0 is __syncthreads)
__device__ __forceinline__ void conv_compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kBlock) : "memory"); }

__device__ __forceinline__ void conv_bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// every bulk group but the newest PENDING has finished reading shared memory
template <int PENDING>
__device__ __forceinline__ void conv_bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(PENDING) : "memory");
}

// every bulk group has completed
__device__ __forceinline__ void conv_bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// One piece of outputs from the window win[i] = input (i - H) steps from the
// piece's first element (H = K - 1 history values, then the piece's EPP
// inputs), in packed f32x2 arithmetic on output pairs (e, e + EPP/2):
// a = bias + sum_k w_k (x_{e-k}, x_{e+EPP/2-k}). Without SILU the output is a.
// With SILU the taps and bias come scaled by -log2(e), so a = -log2(e) z, and
// z sigmoid(z) = z / (1 + 2^a) = a / ((1 + 2^a) (-log2(e))).
template <int K, int EPP, bool SILU>
__device__ __forceinline__ void conv_piece_pairs(const float *win, const u64 *w2, u64 bias2, float *o)
{
    constexpr int H = K - 1, HALF = EPP / 2;
#pragma unroll
    for (int e = 0; e < HALF; ++e) {
        u64 acc = bias2;
#pragma unroll
        for (int k = 0; k < K; ++k)
            acc = fma2(w2[k], pk(win[H + e - k], win[H + e + HALF - k]), acc);
        if constexpr (SILU) {
            const u64 c = splat(-kLog2e);
            acc = mul2(acc, rcp_2(fma2(ex2_2(acc), c, c)));
        }
        upk(acc, o[e], o[e + HALF]);
    }
}

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

// piece m of a thread's segment (channel row `row` of a stage, 128-byte
// swizzle, chunk m at (m ^ ch) * 16): outputs replace the inputs, and hist
// (the H inputs before the piece) moves on to the H inputs before the next
template <typename T, int K, bool SILU>
__device__ __forceinline__ void conv_tile_piece(unsigned char *row, int m, int ch, float *hist, const u64 *w2,
                                                u64 bias2)
{
    constexpr int H = K - 1, EPP = 16 / (int)sizeof(T);
    uint4 *piece = reinterpret_cast<uint4 *>(row + ((m ^ ch) << 4));
    float win[H + EPP];   // the window: H history values, then the piece
#pragma unroll
    for (int j = 0; j < H; ++j)
        win[j] = hist[j];
    unpack_piece<T>(*piece, win + H);
    float o[EPP];
    conv_piece_pairs<K, EPP, SILU>(win, w2, bias2, o);
    *piece = conv_pack<T>(o);
#pragma unroll
    for (int j = 0; j < H; ++j)
        hist[j] = win[EPP + j];
}

// (tile of steps, channel group, batch row) of a tile number; a CTA's tiles
// are its first plus multiples of the grid size, reached by adding the
// step's own digits with carries
struct ConvTileIdx {
    int tt, g, b;
};

__device__ __forceinline__ ConvTileIdx conv_tile_digits(int tile, int ntt, int ngr)
{
    const int r = tile / ntt;
    return {tile - r * ntt, r % ngr, r / ngr};
}

__device__ __forceinline__ void conv_tile_advance(ConvTileIdx &t, const ConvTileIdx &step, int ntt, int ngr)
{
    t.tt += step.tt;
    if (t.tt >= ntt) {
        t.tt -= ntt;
        ++t.g;
    }
    t.g += step.g;
    if (t.g >= ngr) {
        t.g -= ngr;
        ++t.b;
    }
    t.b += step.b;
}

template <typename T, int K, bool SILU>
__global__ void __launch_bounds__(kConvThreads, 4)
causal_conv1d_tile_kernel(const __grid_constant__ ConvParams p)
{
    using SH = ConvTileShape<T>;
    constexpr int H = K - 1, EPP = SH::EPP, SEGE = SH::SEGE, TT = SH::TT, BOX = SH::BOX, NS = kConvStages;
    constexpr int HP = (H + EPP - 1) / EPP;   // pieces of the previous segment that hold the history
    constexpr int PPS = 8;                    // pieces per segment
    static_assert(HP <= PPS, "history within one segment");
    extern __shared__ unsigned char conv_smem[];
    const uint32_t raw_s = static_cast<uint32_t>(__cvta_generic_to_shared(conv_smem));
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;   // boxes with the 128-byte swizzle sit on 1024 bytes
    unsigned char *base = conv_smem + (base_s - raw_s);
    const uint32_t full_s = base_s + NS * SH::STAGE;   // [NS] "stage filled" (the tensor loads landed)
    const uint32_t done_s = full_s + 8u * NS;          // [NS] "stage computed" (every compute thread arrived)

    const int tid = threadIdx.x, lane = tid & 31;
    const int L = static_cast<int>(p.L), ntt = p.ntt, ngr = p.ngr;
    const int mine = static_cast<int>(blockIdx.x) < p.ntiles
                         ? (p.ntiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                         : 0;
    const ConvTileIdx step = conv_tile_digits(static_cast<int>(gridDim.x), ntt, ngr);
    const ConvTileIdx first = conv_tile_digits(static_cast<int>(blockIdx.x), ntt, ngr);

    if (tid == 0) {
#pragma unroll
        for (int j = 0; j < NS; ++j) {
            mbar_init(full_s + 8u * j, 1);
            mbar_init(done_s + 8u * j, kBlock);
        }
        mbar_fence_init();
    }
    __syncthreads();

    if (tid >= kBlock) {
        // the copy warp: lane j loads box j of a tile and stores segment j;
        // boxes wholly outside the row are not fetched (the halo before t = 0,
        // segments past L)
        ConvTileIdx ld = first, sv = first;
        auto issue_load = [&](int n) {
            const int st = n % NS;
            const uint32_t bar = full_s + 8u * st;
            const int t0 = ld.tt * TT;
            const int lo = ld.tt == 0 ? 1 : 0;
            const int live = (L - t0 + SEGE - 1) / SEGE;   // segments of the tile that hold inputs
            const int hi = live < kConvSegs ? live : kConvSegs;
            if (lane == 0)
                mbar_expect_tx(bar, static_cast<uint32_t>((hi + 1 - lo) * BOX));
            __syncwarp();
            if (lane >= lo && lane <= hi)
                tma_load_3d(base_s + st * SH::STAGE + lane * BOX, &p.tm_x, bar, t0 + (lane - 1) * SEGE,
                            ld.g * kConvRows, ld.b);
            conv_tile_advance(ld, step, ntt, ngr);
        };
        for (int n = 0; n < NS && n < mine; ++n)
            issue_load(n);
        for (int i = 0; i < mine; ++i, conv_tile_advance(sv, step, ntt, ngr)) {
            const int st = i % NS;
            mbar_wait(done_s + 8u * st, static_cast<uint32_t>((i / NS) & 1));
            const int t0 = sv.tt * TT;
            if (lane < kConvSegs && t0 + lane * SEGE < L)
                conv_tma_store_3d(&p.tm_out, base_s + st * SH::STAGE + (lane + 1) * BOX, t0 + lane * SEGE,
                                  sv.g * kConvRows, sv.b);
            conv_bulk_commit();
            if (i + NS < mine) {
                conv_bulk_wait_read<0>();   // the stores have left the stage: refill it
                __syncwarp();
                issue_load(i + NS);
            }
        }
        conv_bulk_wait_all();
        return;
    }

    // the compute warps
    const int ch = tid & (kConvRows - 1), s = tid / kConvRows;
    const float tscale = SILU ? -kLog2e : 1.0f;
    ConvTileIdx cur = first;
    // the taps of a tile's channel, each in both halves of a pair (scaled for
    // SILU), loaded one tile ahead
    auto load_taps = [&](const ConvTileIdx &t, u64 *w2, u64 &bias2) {
        const int64_t d = static_cast<int64_t>(t.g) * kConvRows + ch;
        const bool act = d < p.d_inner;
#pragma unroll
        for (int k = 0; k < K; ++k)
            w2[k] = splat(act ? __ldg(p.w + d * K + k) * tscale : 0.0f);
        bias2 = splat((act && p.bias) ? __ldg(p.bias + d) * tscale : 0.0f);
    };
    u64 w2n[K], bias2n;
    load_taps(cur, w2n, bias2n);
    for (int i = 0; i < mine; ++i) {
        u64 w2[K], bias2 = bias2n;
#pragma unroll
        for (int k = 0; k < K; ++k)
            w2[k] = w2n[k];
        ConvTileIdx nxt = cur;
        conv_tile_advance(nxt, step, ntt, ngr);
        if (i + 1 < mine)
            load_taps(nxt, w2n, bias2n);
        const int64_t d = static_cast<int64_t>(cur.g) * kConvRows + ch;
        const bool act = d < p.d_inner;
        const int st = i % NS;
        unsigned char *stage = base + st * SH::STAGE;
        const int ts = cur.tt * TT + s * SEGE;   // first step of this thread's segment
        const bool live = ts < L;
        mbar_wait(full_s + 8u * st, static_cast<uint32_t>((i / NS) & 1));

        // hist[j] = input H - j steps before the segment
        float hist[H > 0 ? H : 1];
        if (live && H > 0) {
            if (ts == 0) {
#pragma unroll
                for (int j = 0; j < H; ++j)
                    hist[j] = (act && p.state_in)
                                  ? Io<T>::load1(static_cast<const T *>(p.state_in) +
                                                 (static_cast<int64_t>(cur.b) * H + j) * p.d_inner + d)
                                  : 0.0f;
            } else {
                float pv[HP * EPP > 0 ? HP * EPP : 1];
                const unsigned char *prev = stage + s * BOX + ch * 128;   // the segment before (the halo for s = 0)
#pragma unroll
                for (int v = 0; v < HP; ++v) {
                    const int c = PPS - HP + v;
                    unpack_piece<T>(*reinterpret_cast<const uint4 *>(prev + ((c ^ ch) << 4)), pv + v * EPP);
                }
#pragma unroll
                for (int j = 0; j < H; ++j)
                    hist[j] = pv[HP * EPP - H + j];
            }
        }
        conv_compute_sync();   // every history is read: outputs may now replace their inputs

        unsigned char *row = stage + (s + 1) * BOX + ch * 128;
        if (ts + SEGE <= L) {   // a whole segment: no bound checks, so its pieces overlap
#pragma unroll
            for (int m = 0; m < PPS; ++m)
                conv_tile_piece<T, K, SILU>(row, m, ch, hist, w2, bias2);
        } else if (live) {
#pragma unroll
            for (int m = 0; m < PPS; ++m) {
                if (ts + m * EPP >= L)
                    break;
                conv_tile_piece<T, K, SILU>(row, m, ch, hist, w2, bias2);
            }
        }
        // the segment holding the row's last input leaves the last H inputs as the next call's history
        if (H > 0 && p.state_out && act && live && ts + SEGE >= L) {
#pragma unroll
            for (int j = 0; j < H; ++j)
                Io<T>::store1(static_cast<T *>(p.state_out) + (static_cast<int64_t>(cur.b) * H + j) * p.d_inner + d,
                              hist[j]);
        }
        conv_fence_async_smem();   // the outputs, written by threads, are read by the tensor stores
        conv_mbar_arrive(done_s + 8u * st);
        cur = nxt;
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

// map of a (batch, d_inner, L) tensor of T as (L, d_inner, batch), box
// (128 bytes, kConvRows, 1) with the 128-byte swizzle; reads outside the
// tensor give zero, writes outside it are dropped
template <typename T>
bool conv_encode(CUtensorMap *m, const void *base, int64_t L, int64_t d_inner, int64_t batch)
{
    const EncodeTiledFn fn = encode_tiled_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(d_inner),
                                static_cast<cuuint64_t>(batch)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(L) * sizeof(T),
                                   static_cast<cuuint64_t>(L) * static_cast<cuuint64_t>(d_inner) * sizeof(T)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / sizeof(T)), kConvRows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// resident CTAs of the tile kernel per SM, after raising its shared-memory
// limit on the current device (every call: the limit is a per-device
// attribute); 0 on failure
template <typename T, int K, bool SILU>
int conv_tile_setup()
{
    static std::atomic<int> per_sm{-1};
    auto kernel = causal_conv1d_tile_kernel<T, K, SILU>;
    const int smem = ConvTileShape<T>::BYTES;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    int n = per_sm.load(std::memory_order_relaxed);
    if (n < 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kConvThreads, smem) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        per_sm.store(n, std::memory_order_relaxed);
    }
    return n;
}

template <typename T, int K, bool SILU>
ss_status launch_conv_tile(const ConvParams &p, int dev, cudaStream_t stream)
{
    using SH = ConvTileShape<T>;
    const int per_sm = conv_tile_setup<T, K, SILU>();
    if (per_sm <= 0)
        return fail(SS_ERR_LAUNCH, "conv tile kernel cannot be made resident (%d bytes of shared memory)", SH::BYTES);
    const int64_t grid = std::min<int64_t>(p.ntiles, static_cast<int64_t>(sm_count(dev)) * per_sm);
    causal_conv1d_tile_kernel<T, K, SILU><<<static_cast<unsigned>(grid), kConvThreads, SH::BYTES, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SS_ERR_LAUNCH, "conv launch failed: %s", cudaGetErrorString(e));
    return SS_OK;
}

template <typename T, int K>
ss_status launch_conv(const ConvParams &p, int dev, cudaStream_t stream)
{
    if (p.tma)
        return p.silu ? launch_conv_tile<T, K, true>(p, dev, stream) : launch_conv_tile<T, K, false>(p, dev, stream);
    constexpr int EPP = 16 / (int)sizeof(T);
    const int64_t pblocks = ((p.L + EPP - 1) / EPP + kBlock - 1) / kBlock;
    if (pblocks > 0x7fffffff)
        return fail(SS_ERR_DIM, "grid too large");
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
    // tensor coordinates and tile numbers are 32-bit: the tile kernel takes
    // rows below 2^31 steps (a tile's last step included) and fewer than 2^31 tiles
    {
        const int64_t ntt = (L + ConvTileShape<T>::TT - 1) / ConvTileShape<T>::TT;
        const int64_t ngr = (d_inner + kConvRows - 1) / kConvRows;
        const bool fits = L < (int64_t(1) << 31) - ConvTileShape<T>::TT && ngr < (int64_t(1) << 27) &&
                          ntt * ngr < (int64_t(1) << 31) / batch;
        p.ntt = fits ? static_cast<int>(ntt) : 0;
        p.ngr = fits ? static_cast<int>(ngr) : 0;
        p.ntiles = fits ? static_cast<int>(ntt * ngr * batch) : 0;
        p.tma = p.vec && fits && conv_encode<T>(&p.tm_x, x, L, d_inner, batch) &&
                conv_encode<T>(&p.tm_out, out, L, d_inner, batch);
    }
    switch (k) {
    case 1: return launch_conv<T, 1>(p, dev, stream);
    case 2: return launch_conv<T, 2>(p, dev, stream);
    case 3: return launch_conv<T, 3>(p, dev, stream);
    case 4: return launch_conv<T, 4>(p, dev, stream);
    case 5: return launch_conv<T, 5>(p, dev, stream);
    case 6: return launch_conv<T, 6>(p, dev, stream);
    case 7: return launch_conv<T, 7>(p, dev, stream);
    default: return launch_conv<T, 8>(p, dev, stream);
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
