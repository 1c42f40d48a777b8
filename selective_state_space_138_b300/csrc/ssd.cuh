// ssd.cuh -- Mamba-2's scalar-decay scan (SSD) kernels on the tensor cores (the host side is in ssd_host.cuh).
//
// Part of the single translation unit ss_scan.cu (included inside its
// anonymous namespace); not compiled on its own.
//
// With one decay per head ("Mamba and selective state spaces": each head, a
// group of P channels, gets a single scalar decay, which turns most of the work
// into matrix products; "Mamba in practice": Y = M o (pairwise scores) X with a
// 1-semiseparable mask M), a chunk of Q steps of one head is
//
//   Y_c = diag(e^{cum}) C_c H_{c-1}^T + (CB_c o M_c o delta) X_c + D X_c
//   H_c = e^{cum[Q-1]} H_{c-1} + (w o X_c)^T B_c,   w_s = e^{cum[Q-1] - cum[s]} delta_s
//
// where cum[t] = A_h * (delta_0 + .. + delta_t) within the chunk, CB_c = C_c B_c^T
// (Q x Q, shared by the heads of a group), M_c[t][s] = e^{cum[t] - cum[s]} for
// s <= t and 0 above the diagonal, and H (P x N, fp32) is the state carried
// between chunks. Every product is a bf16 x bf16 -> fp32 tensor-core MMA
// (mma.sync m16n8k16); the decays, masks and the carried state are fp32, and
// the state enters C_c H^T rounded to bf16 straight from the accumulator
// registers that hold it. C B^T is kept in bf16.
//
//   ssd_cb_kernel     CB_c for every (batch, chunk, group) into the workspace (bf16).
//   ssd_chunk_kernel  one CTA per (batch, head), walking its chunks in order;
//                     C and CB of chunk c+1 are fetched as soon as chunk c has
//                     used them, X and B of chunk c+1 while chunk c's outputs
//                     are written.

constexpr int kSsdQ = 64;    // steps per chunk
constexpr int kSsdP = 64;    // channels per head (headdim)

struct SsdParams {
    const __nv_bfloat16 *x, *dt, *B, *C, *z;
    const float *A, *D, *dt_bias, *h0;
    __nv_bfloat16 *y;
    float *final_state;
    __nv_bfloat16 *cb;   // workspace: [batch][nchunks][G][Q][Q] bf16
    // workspace of the tensor-core chunk walk: work[0] counts the work items claimed,
    // work[1 + row] the chunk segments of row (b, h) done; hbuf holds the state one
    // segment hands to the next, laid out as final_state
    unsigned int *work;
    float *hbuf;
    int nseg, cps;   // chunk segments per row and chunks per segment
    int64_t batch, L, H, G, nchunks;
    int softplus;
    int tma;   // the chunk kernel's X, B, C and C B^T tiles come in through the tensor maps below
    // the state dimension as stored (the B, C row length per group, the h0 and final-state
    // stride) and the first state this call handles: N = 256 runs as two passes over the
    // 128-state halves (n_off 0 and 128) of the tensor-core kernels
    int Nt, n_off;
    // 0: the whole state (D skip, gate, y stored); 1: first half (D skip, no gate, the partial y
    // stored in y); 2: second half (no D, the stored partial added, gate, y stored)
    int mode;
    // 3-d maps: x over (H*P channels, L, batch) with a box of one head's P + 8 channels x Q steps;
    // B, C over (G*N, L, batch) with a box of N + 8 x Q; C B^T over (Q, Q, batch*nchunks*G) with
    // a box of Q + 8 x Q. The 8 extra columns fill each shared-memory row's pad (never read).
    CUtensorMap tm_x, tm_B, tm_C, tm_cb;
    // B, C over (G*N, L, batch) with a box of 64 states x 128 steps, 128-byte swizzled (the C B^T product)
    CUtensorMap tm_Bsw, tm_Csw;
    // the tensor-core chunk walk's tiles, 128-byte swizzled: x over (H*P, L, batch) with a box of
    // 64 channels x Q steps; B, C with 64 states x Q steps; C B^T with Q x Q
    CUtensorMap tm_xq, tm_Bq, tm_Cq, tm_cbq;
    CUtensorMap tm_yq;   // y by (channel of the row, step, batch row), box 64 x 64, 128-byte swizzle (stores)
};

// the segment count of a row as published by the CTA that walked the segment before:
// waits (bounded, thread 0) until it reaches v; false (and the fault flag set) if not
__device__ __forceinline__ bool ssd_flag_wait(const unsigned int *f, unsigned int v)
{
    const uint64_t t0 = global_ns();
    for (;;) {
        unsigned int x;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(x) : "l"(f) : "memory");
        if (x >= v)
            return true;
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_fault_flags, kFaultWaitTimeout);
            return false;
        }
        __nanosleep(256);
    }
}

__device__ __forceinline__ void ssd_flag_release(unsigned int *f, unsigned int v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}

// ---- warp-level MMA helpers (PTX mma.sync / ldmatrix; operands in shared memory)

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A (16x16, row) * B (16x8, col), bf16 in, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};\n"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// A fragment (16 rows x 16 k) of a row-major bf16 tile: rows r0.., k0.., row stride `ld` elements
__device__ __forceinline__ void frag_a(const __nv_bfloat16 *base, int ld, int r0, int k0, int lane, uint32_t *a)
{
    const int r = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int k = k0 + (lane >> 4) * 8;
    ldsm_x4(smem_u32(base + r * ld + k), a[0], a[1], a[2], a[3]);
}

// A fragment of the transpose of a row-major tile T (A[m][k] = T[k][m]): m0.., k0..
__device__ __forceinline__ void frag_a_t(const __nv_bfloat16 *base, int ld, int m0, int k0, int lane, uint32_t *a)
{
    const int k = k0 + (lane & 7) + (lane >> 4) * 8;
    const int m = m0 + ((lane >> 3) & 1) * 8;
    ldsm_x4_t(smem_u32(base + k * ld + m), a[0], a[1], a[2], a[3]);
}

// B fragments for two 8-column tiles (n0.. and n0+8..) x 16 k, from a tile stored
// [n][k] (k contiguous): b[0], b[1] for columns n0..n0+7, b[2], b[3] for n0+8..
__device__ __forceinline__ void frag_b_nk(const __nv_bfloat16 *base, int ld, int n0, int k0, int lane, uint32_t *b)
{
    const int n = n0 + (lane & 7) + (lane >> 4) * 8;
    const int k = k0 + ((lane >> 3) & 1) * 8;
    ldsm_x4(smem_u32(base + n * ld + k), b[0], b[1], b[2], b[3]);
}

// the same from a tile stored [k][n] (n contiguous)
__device__ __forceinline__ void frag_b_kn(const __nv_bfloat16 *base, int ld, int n0, int k0, int lane, uint32_t *b)
{
    const int k = k0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int n = n0 + (lane >> 4) * 8;
    ldsm_x4_t(smem_u32(base + k * ld + n), b[0], b[1], b[2], b[3]);
}

// Copy `rows` rows of `row_elems` bf16 (a multiple of 8) from global rows at
// stride `gstride` elements into shared rows at stride `sld`, zero-filling rows
// at or past `valid`, with 16-byte cp.async pieces spread over the CTA.
__device__ __forceinline__ void stage_rows(__nv_bfloat16 *s, int sld, const __nv_bfloat16 *g, int gstride,
                                           int rows, int row_elems, int valid, int tid, int nthreads)
{
    const int ppr = row_elems / 8;
    for (int i = tid; i < rows * ppr; i += nthreads) {
        const int r = i / ppr;
        const int c = (i % ppr) * 8;
        const bool ok = r < valid;
        cp_async16(smem_u32(s + r * sld + c), ok ? g + r * gstride + c : g, ok ? 16 : 0);
    }
}

// ---- CB_c = C_c B_c^T, one CTA (4 warps) per (chunk, batch, group)
template <int N>
__global__ void __launch_bounds__(128)
ssd_cb_kernel(const SsdParams p)
{
    constexpr int Q = kSsdQ, LDN = N + 8;
    __shared__ __align__(16) __nv_bfloat16 Cs[Q * LDN];
    __shared__ __align__(16) __nv_bfloat16 Bs[Q * LDN];
    const int c = blockIdx.x;
    const int64_t b = blockIdx.y;
    const int g = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int64_t t0 = static_cast<int64_t>(c) * Q;
    const int valid = static_cast<int>(p.L - t0 < Q ? p.L - t0 : Q);
    const int rs = static_cast<int>(p.G * N);   // B, C row stride
    stage_rows(Cs, LDN, p.C + ((b * p.L + t0) * p.G + g) * N, rs, Q, N, valid, tid, 128);
    stage_rows(Bs, LDN, p.B + ((b * p.L + t0) * p.G + g) * N, rs, Q, N, valid, tid, 128);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    float acc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < N; kk += 16) {
        uint32_t a[4];
        frag_a(Cs, LDN, 16 * w, kk, lane, a);
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            uint32_t bb[4];
            frag_b_nk(Bs, LDN, 8 * j, kk, lane, bb);   // column s = row of B_c
            mma_bf16(acc[j], a[0], a[1], a[2], a[3], bb[0], bb[1]);
            mma_bf16(acc[j + 1], a[0], a[1], a[2], a[3], bb[2], bb[3]);
        }
    }
    __nv_bfloat16 *out = p.cb + (((b * p.nchunks + c) * p.G + g) * Q) * Q;
    const int gr = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int col = 8 * j + 2 * t4;
        *reinterpret_cast<uint32_t *>(out + (16 * w + gr) * Q + col) = pack_bf16x2(acc[j][0], acc[j][1]);
        *reinterpret_cast<uint32_t *>(out + (16 * w + gr + 8) * Q + col) = pack_bf16x2(acc[j][2], acc[j][3]);
    }
}

// ---- 5th-generation tensor cores (tcgen05): the accumulator lives in tensor
// memory (TMEM, 128 lanes x 512 32-bit columns per SM), operands are read from
// shared memory through 64-bit matrix descriptors, one thread issues the MMA
// and its completion arrives on an mbarrier.

// K-major bf16 operand tile stored as TMA writes it with the 128-byte swizzle:
// rows of 64 elements (128 bytes), 8-row groups of 1024 bytes. Fields: start
// address >> 4 (bits 0-13), leading offset (unused for this layout, 1),
// stride between 8-row groups >> 4 (bits 32-45), descriptor version 1 (bit
// 46), swizzle mode 2 = 128-byte (bits 61-63). The tile must start on a
// 1024-byte boundary; the K slice k (16 elements) of a row starts 32 k bytes
// in, which the swizzle maps through the address bits.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr)
{
    return static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// instruction descriptor of kind::f16 with bf16 A and B, fp32 D, both
// operands K-major: D format (bits 4-5) = 1, A format (7-9) = 1, B format
// (10-12) = 1, N >> 3 (17-22), M >> 4 (24-28)
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// D (tmem) (+)= A (smem desc) * B (smem desc)^T, issued by one thread
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          bool accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0)
                 : "memory");
}

// arrive on the mbarrier once every MMA issued so far by this thread has completed
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// tensor-memory allocation by one whole warp: the base address is written to shared memory at dst
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive 32-bit columns of this thread's lane (warp w reads lanes 32w .. 32w+31)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *v)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                 "%13, %14, %15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                   "=r"(v[15])
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---- CB_c = C_c B_c^T on the tcgen05 tensor cores: one CTA (4 warps) per
// (pair of chunks, batch, group). The 128 steps of two chunks are the M rows
// (C) and the N columns (B) of one 128 x 128 product over K = N states,
// accumulated in tensor memory; the two diagonal 64 x 64 blocks are the
// chunks' C B^T, read back lane by lane and stored in bf16.
template <int N>
struct SsdCbShape {
    static constexpr int ATOMS = N / 64;                 // 64-element (128-byte) K slices
    static constexpr int TILE = 128 * 128;               // one [128 rows][64] bf16 slice, bytes
    static constexpr int A_OFF = 0;                      // C rows, ATOMS slices
    static constexpr int B_OFF = ATOMS * TILE;           // B rows, ATOMS slices
    static constexpr int BAR_OFF = 2 * ATOMS * TILE;     // tile barrier, MMA barrier
    static constexpr int TMEM_OFF = BAR_OFF + 16;        // the allocated tensor-memory address
    static constexpr size_t BYTES = TMEM_OFF + 16 + 1024;   // + room to align the base to 1024 bytes
};

template <int N>
__global__ void __launch_bounds__(128, 1)
ssd_cb_tc_kernel(const __grid_constant__ SsdParams p)
{
    using SH = SsdCbShape<N>;
    constexpr int Q = kSsdQ;
    extern __shared__ __align__(1024) unsigned char smem_cb[];
    const uint32_t raw_s = static_cast<uint32_t>(__cvta_generic_to_shared(smem_cb));
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;   // 128-byte swizzled tiles on 1024-byte boundaries
    unsigned char *base = smem_cb + (base_s - raw_s);
    const uint32_t bar_tile = base_s + SH::BAR_OFF, bar_mma = bar_tile + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + SH::TMEM_OFF);

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int64_t b = blockIdx.y;
    const int g = blockIdx.z;
    const int64_t c0 = 2 * static_cast<int64_t>(blockIdx.x);   // first chunk of the pair
    if (p.work) {   // the chunk walk's counters, fresh for this call (every block a share)
        const int64_t blk = (static_cast<int64_t>(blockIdx.z) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        const int64_t nblk = static_cast<int64_t>(gridDim.x) * gridDim.y * gridDim.z;
        for (int64_t i = blk * 128 + tid; i <= p.batch * p.H; i += nblk * 128)
            p.work[i] = 0u;
    }
    if (w == 0)
        tmem_alloc(base_s + SH::TMEM_OFF, 128);
    if (tid == 0) {
        mbar_init(bar_tile, 1);
        mbar_init(bar_mma, 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    bool ok = true;
    if (tid == 0) {
        mbar_expect_tx(bar_tile, 2 * SH::ATOMS * SH::TILE);
        const int t0 = static_cast<int>(c0 * Q);
#pragma unroll
        for (int a = 0; a < SH::ATOMS; ++a) {
            tma_load_3d(base_s + SH::A_OFF + a * SH::TILE, &p.tm_Csw, bar_tile, g * p.Nt + p.n_off + 64 * a, t0,
                        static_cast<int>(b));
            tma_load_3d(base_s + SH::B_OFF + a * SH::TILE, &p.tm_Bsw, bar_tile, g * p.Nt + p.n_off + 64 * a, t0,
                        static_cast<int>(b));
        }
        ok = mbar_wait(bar_tile, 0);
        if (!ok)   // the wait gave up: let the copies land before the CTA leaves (bounded)
            mbar_wait(bar_tile, 0);
        if (ok) {
            constexpr uint32_t idesc = umma_idesc_bf16(128, 128);
#pragma unroll
            for (int kk = 0; kk < N / 16; ++kk) {
                const uint32_t koff = static_cast<uint32_t>((kk / 4) * SH::TILE + (kk % 4) * 32);
                umma_bf16(tmem, umma_desc_sw128(base_s + SH::A_OFF + koff), umma_desc_sw128(base_s + SH::B_OFF + koff),
                          idesc, kk > 0);
            }
            umma_commit(bar_mma);
        }
    }
    ok = __syncthreads_and(ok ? 1 : 0) != 0;
    if (ok && mbar_wait(bar_mma, 0)) {
        tc_fence_after();
        // lane t of warp w holds row r = 32w + t: the step of chunk c0 + r / 64, whose
        // diagonal block is columns 64 (r / 64) ..
        const int r = 32 * w + lane;
        const int64_t c = c0 + r / 64;
        uint32_t v[64];
        const uint32_t ta = tmem + (static_cast<uint32_t>(32 * w) << 16) + static_cast<uint32_t>((r / 64) * 64);
        tmem_ld16(ta, v);
        tmem_ld16(ta + 16, v + 16);
        tmem_ld16(ta + 32, v + 32);
        tmem_ld16(ta + 48, v + 48);
        tmem_ld_wait();
        if (c < p.nchunks) {
            __nv_bfloat16 *out = p.cb + (((b * p.nchunks + c) * p.G + g) * Q + (r % 64)) * Q;
#pragma unroll
            for (int j = 0; j < 64; j += 8) {
                uint4 o;
                o.x = pack_bf16x2(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
                o.y = pack_bf16x2(__uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
                o.z = pack_bf16x2(__uint_as_float(v[j + 4]), __uint_as_float(v[j + 5]));
                o.w = pack_bf16x2(__uint_as_float(v[j + 6]), __uint_as_float(v[j + 7]));
                *reinterpret_cast<uint4 *>(out + j) = o;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (w == 0)
        tmem_dealloc(tmem, 128);
}

// 16 consecutive 32-bit columns of this thread's lane written to tensor memory
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                 "%13, %14, %15, %16};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
                 "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
}

// M = 64 accumulators sit in lanes 0-15 of each warp's quarter: threads 0-15 read 16
// columns of lanes 0-15 at taddr, threads 16-31 the same lanes at taddr + `half` columns
template <int HALF>
__device__ __forceinline__ void tmem_ld16_split(uint32_t taddr, uint32_t *v)
{
    asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                 "%13, %14, %15}, [%16], %17;"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                   "=r"(v[15])
                 : "r"(taddr), "n"(HALF)
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// shared-memory writes of this thread become visible to the tensor cores (async proxy)
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// box (c0, c1, c2) of a 3-d tensor map from shared memory at src to global memory
__device__ __forceinline__ void ssd_tma_store_3d(const void *tmap, uint32_t src, int c0, int c1, int c2)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void ssd_bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void ssd_bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void ssd_bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// MN-major operand descriptor (128-byte swizzle): atoms of 64 MN elements x 8 K
// rows (8 rows of 128 bytes), `lbo` bytes between MN atoms, 1024 bytes between
// 8-row K groups; a K step of 16 rows advances the start by 2048 bytes
__device__ __forceinline__ uint64_t umma_desc_mn_sw128(uint32_t smem_addr, uint32_t lbo)
{
    return static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// kind::f16 instruction descriptor with the operand majorness: a_mn / b_mn = 1 for MN-major
__host__ __device__ constexpr uint32_t umma_idesc_bf16_mj(int M, int N, int a_mn, int b_mn)
{
    return umma_idesc_bf16(M, N) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16);
}

// a bf16 pair times f (both lanes of f2), rounded back to a bf16 pair
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t w, u64 f2)
{
    float a, b;
    upk(mul2(pk(bf16lo(w), bf16hi(w)), f2), a, b);
    return pack_bf16x2(a, b);
}

// byte offset of element (r, c), c < 64, in a tile of 128-byte rows stored with
// the 128-byte swizzle (16-byte piece c/8 of row r sits at piece (c/8) ^ (r % 8))
__device__ __forceinline__ int sw128_off(int r, int c) { return r * 128 + (((c >> 3) ^ (r & 7)) << 4) + (c & 7) * 2; }

// ---- the chunk walk on the tcgen05 tensor cores: CTAs of 8 warps, at most as
// many as fit on the GPU at once, each claiming work items in order: a (batch,
// head) row's chunks of Q = 64 steps, or one of the 2 or 4 segments of them
// (walked one after another: a segment starts from the state the segment before
// hands over), so that rows x segments spread evenly over the CTAs. Per chunk,
// with T the tensor memory of the CTA:
//   Y[t][p]   = sum_n (e^{cum[t]} C[t][n]) H[p][n] + sum_s (S' + D I)[t][s] X[s][p]   (T cols 64..127;
//               M = 64 rows t; the decay of the carried state is folded into the C rows, the skip
//               term D x into the diagonal of S', so both products accumulate in one place)
//   y[t][p]   = Y[t][p] silu(z[t][p])
//   H^T[n][p] <- e^{cum[Q-1]} H^T[n][p] + sum_s B[s][n] (w o X)[s][p]   (T cols 0..63; M = N rows n)
// H^T stays in tensor memory from chunk to chunk (fp32). Operands: C, B, X and
// C B^T arrive by 128-byte swizzled tensor copies; the threads scale the C rows
// in place, form S' = C B^T o M o delta (+ D on the diagonal) in place over
// C B^T, and write w o X and the bf16 copy of H (the B operand of the first
// product) in the same swizzled layout. Every operand of a product is rounded
// once to bf16. With N = 128 the state product has M = 128 (row n in lane n);
// with N = 64, M = 64 (row n in lane 32 (n / 16) + n % 16), as for Y.
// One warp forms the next chunk's step sizes while the products run, and the
// state copy for the next chunk follows the epilogue.
constexpr int kSsdTcThreads = 256;   // 8 warps: two per lane quarter of tensor memory
constexpr int kSsdStepWarp = 4;      // forms the step sizes (not warp 0, whose thread 0 issues the products)

template <int N>
struct SsdTcShape {
    static constexpr int Q = kSsdQ, P = kSsdP;
    static constexpr int NS = N / 64;                       // 64-state slices of C and B
    static constexpr int XT = Q * 128;                      // X tile [Q][64] bf16
    static constexpr int CT = Q * 128;                      // one 64-state slice of C or B [Q][64]
    static constexpr int X_OFF = 0;                         // X
    static constexpr int C_OFF = X_OFF + XT;                // C slices (scaled in place)
    static constexpr int B_OFF = C_OFF + NS * CT;           // B slices
    static constexpr int S_OFF = B_OFF + NS * CT;           // C B^T, then S' in place [Q][Q]
    static constexpr int XW_OFF = S_OFF + Q * 128;          // w o X [Q][64]
    static constexpr int H_OFF = XW_OFF + XT;               // bf16 H, stored [N][64]
    static constexpr int F_OFF = H_OFF + N * 128;           // fp32 per-step values: cum, e^cum, w, delta
    static constexpr int BAR_OFF = F_OFF + 4 * Q * 4;       // barriers: the chunk's tiles, MMA
    static constexpr int TMEM_OFF = BAR_OFF + 16;
    static constexpr size_t BYTES = TMEM_OFF + 16 + 1024;  // + room to align the base to 1024 bytes
    static constexpr uint32_t TCOLS = 128;
    static_assert(X_OFF % 1024 == 0 && C_OFF % 1024 == 0 && B_OFF % 1024 == 0 && S_OFF % 1024 == 0 &&
                      XW_OFF % 1024 == 0 && H_OFF % 1024 == 0,
                  "swizzled tiles on 1024-byte boundaries");
};

template <int N>
__global__ void __launch_bounds__(kSsdTcThreads, 3)
ssd_chunk_tc_kernel(const __grid_constant__ SsdParams p)
{
    using SH = SsdTcShape<N>;
    constexpr int Q = SH::Q, P = SH::P;
    extern __shared__ __align__(1024) unsigned char smem_tc[];
    const uint32_t raw_s = static_cast<uint32_t>(__cvta_generic_to_shared(smem_tc));
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    unsigned char *base = smem_tc + (base_s - raw_s);
    float *cum = reinterpret_cast<float *>(base + SH::F_OFF);
    float *ecum = cum + Q;
    float *wsx = ecum + Q;   // w_s = e^{cum[Q-1] - cum[s]} delta_s
    float *dl = wsx + Q;     // delta_s
    const uint32_t bar_cb = base_s + SH::BAR_OFF;      // X, C, B, C B^T of a chunk
    const uint32_t bar_mma = bar_cb + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + SH::TMEM_OFF);

    // warp w reads and writes lane quarter q = w % 4 of tensor memory; warps w and w + 4
    // share a quarter and split its columns (hf = w / 4)
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, q = w & 3, hf = w >> 2;
    int64_t b = 0;   // the work item's row (b, h), group g and per-head values
    int h = 0, g = 0;
    float Ah = 0.0f, Dh = 0.0f, bias = 0.0f;
    const bool gate = p.z != nullptr && p.mode != 1;   // the gate once, on the whole state's y
    const bool add_partial = p.mode == 2;
    const int Nt = p.Nt, n_off = p.n_off;
    const int64_t xs = p.H * P;   // x, z, y row stride (one time step)

    if (w == 0)
        tmem_alloc(base_s + SH::TMEM_OFF, SH::TCOLS);
    if (tid == 0) {
        mbar_init(bar_cb, 1);
        mbar_init(bar_mma, 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_h = tmem, t_y = tmem + 64;   // column bases
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;

    // the state row this thread holds in tensor memory (H^T[n][.]), or -1
    const int hrow = (N == 128) ? 32 * q + lane : ((lane < 16) ? 16 * q + lane : -1);

    // tensor copies of a chunk's tiles (X, C, B, C B^T) on one barrier; every wait is
    // bounded, and after one gives up the CTA issues no more and leaves after the
    // copies it issued have landed
    int cb_issued = 0, cb_done = 0;
    bool aborted = false;
    auto issue_cb = [&](int64_t c) {
        if (tid == 0 && !aborted) {
            mbar_expect_tx(bar_cb, SH::XT + 2 * SH::NS * SH::CT + Q * 128);
            tma_load_3d(base_s + SH::X_OFF, &p.tm_xq, bar_cb, h * P, static_cast<int>(c * Q), static_cast<int>(b));
#pragma unroll
            for (int j = 0; j < SH::NS; ++j) {
                tma_load_3d(base_s + SH::C_OFF + j * SH::CT, &p.tm_Cq, bar_cb, g * Nt + n_off + 64 * j, static_cast<int>(c * Q),
                            static_cast<int>(b));
                tma_load_3d(base_s + SH::B_OFF + j * SH::CT, &p.tm_Bq, bar_cb, g * Nt + n_off + 64 * j, static_cast<int>(c * Q),
                            static_cast<int>(b));
            }
            tma_load_3d(base_s + SH::S_OFF, &p.tm_cbq, bar_cb, 0, 0, static_cast<int>((b * p.nchunks + c) * p.G + g));
            ++cb_issued;
        }
    };
    auto wait_cb = [&]() {
        if (!aborted) {
            aborted = !mbar_wait(bar_cb, static_cast<uint32_t>(cb_done & 1));
            if (!aborted)
                ++cb_done;
        }
    };

    // the raw step sizes of steps 2 lane and 2 lane + 1 of chunk c (the step warp; zero past L)
    float dta = 0.0f, dtb = 0.0f;
    auto load_dt = [&](int64_t c) {
        const int64_t ta = c * Q + 2 * lane;
        dta = (c < p.nchunks && ta < p.L) ? __bfloat162float(p.dt[(b * p.L + ta) * p.H + h]) : 0.0f;
        dtb = (c < p.nchunks && ta + 1 < p.L) ? __bfloat162float(p.dt[(b * p.L + ta + 1) * p.H + h]) : 0.0f;
    };
    // the step warp: the step sizes of chunk c from (dta, dtb) and, in shared memory, delta, cum[t] =
    // A delta_0 + .. + A delta_t (log2 e units), e^cum and w_s = e^{cum[Q-1] - cum[s]} delta_s
    auto step_sizes = [&](int64_t c) {
        const int64_t ta = c * Q + 2 * lane;
        float d0 = 0.0f, d1 = 0.0f;
        if (ta < p.L)
            d0 = p.softplus ? softplus_f(dta + bias) : dta + bias;
        if (ta + 1 < p.L)
            d1 = p.softplus ? softplus_f(dtb + bias) : dtb + bias;
        const float a0 = Ah * kLog2e * d0, a1 = Ah * kLog2e * d1;
        float sum = a0 + a1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, sum, o);
            if (lane >= o)
                sum += u;
        }
        const float c0v = sum - a1, c1v = sum;
        const float cq = __shfl_sync(0xffffffffu, c1v, 31);
        *reinterpret_cast<float2 *>(dl + 2 * lane) = make_float2(d0, d1);
        *reinterpret_cast<float2 *>(cum + 2 * lane) = make_float2(c0v, c1v);
        *reinterpret_cast<float2 *>(ecum + 2 * lane) = make_float2(ex2_approx(c0v), ex2_approx(c1v));
        *reinterpret_cast<float2 *>(wsx + 2 * lane) =
            make_float2(ex2_approx(cq - c0v) * d0, ex2_approx(cq - c1v) * d1);
    };
    // the state entering a chunk (this thread's half row of H^T, columns 32 hf .., in hv):
    // its bf16 copy, the B operand of Y = (e^cum C) H^T, and e^{cum[Q-1]} H back into
    // tensor memory
    auto put_h = [&](uint32_t (&hv)[32], float ec) {
        if (hrow >= 0) {
            unsigned char *hr = base + SH::H_OFF;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint4 o;
                o.x = pack_bf16x2(__uint_as_float(hv[8 * j]), __uint_as_float(hv[8 * j + 1]));
                o.y = pack_bf16x2(__uint_as_float(hv[8 * j + 2]), __uint_as_float(hv[8 * j + 3]));
                o.z = pack_bf16x2(__uint_as_float(hv[8 * j + 4]), __uint_as_float(hv[8 * j + 5]));
                o.w = pack_bf16x2(__uint_as_float(hv[8 * j + 6]), __uint_as_float(hv[8 * j + 7]));
                *reinterpret_cast<uint4 *>(hr + sw128_off(hrow, 32 * hf + 8 * j)) = o;
            }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j)
            hv[j] = __float_as_uint(__uint_as_float(hv[j]) * ec);
#pragma unroll
        for (int j = 0; j < 2; ++j)
            tmem_st16(t_h + lane_base + 32 * hf + 16 * j, hv + 16 * j);
    };

    // Work items: row (b, h) = item % rows, chunk segment item / rows (cps chunks). Items
    // are claimed in order from a counter, so a row's segment is claimed only after the
    // one before it, by a CTA that is already running: it starts from the state that
    // segment hands over (the row's flag counts the segments done) and never waits on a
    // CTA that has not started.
    const int64_t rows = p.batch * p.H;
    const int64_t total = rows * p.nseg;
    int64_t *item_slot = reinterpret_cast<int64_t *>(base + SH::TMEM_OFF + 8);
    int mma_phase = 0;
    for (;;) {
        if (tid == 0)
            *item_slot = static_cast<int64_t>(atomicAdd(p.work, 1u));
        __syncthreads();
        const int64_t item = *item_slot;
        if (item >= total)
            break;
        const int seg = static_cast<int>(item / rows);
        const int64_t row = item % rows;
        b = row / p.H;
        h = static_cast<int>(row % p.H);
        g = static_cast<int>(h / (p.H / p.G));
        Ah = __ldg(p.A + h);
        Dh = (p.D && p.mode != 2) ? __ldg(p.D + h) : 0.0f;   // D x once, in the first half's pass
        bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.0f;
        const int64_t c_begin = static_cast<int64_t>(seg) * p.cps;
        const int64_t c_end = c_begin + p.cps < p.nchunks ? c_begin + p.cps : p.nchunks;
        const bool last = c_end >= p.nchunks;
        float *hand = p.hbuf + row * P * Nt + n_off;   // the state handed between the row's segments, [p][n]
        if (seg > 0 && tid == 0)
            aborted = !ssd_flag_wait(p.work + 1 + row, static_cast<unsigned int>(seg));
        aborted = __syncthreads_or(aborted ? 1 : 0) != 0;
        if (aborted)
            break;
        issue_cb(c_begin);
        if (w == kSsdStepWarp) {
            load_dt(c_begin);
            step_sizes(c_begin);
            load_dt(c_begin + 1);
        }
        __syncthreads();   // the segment's first step sizes
        {   // the state entering the segment: h0 (zero without it) or the one handed over
            uint32_t hv[32];
#pragma unroll
            for (int pp = 0; pp < 32; ++pp) {
                const int64_t o = static_cast<int64_t>(32 * hf + pp) * Nt + hrow;
                float v = 0.0f;
                if (hrow >= 0)
                    v = seg > 0 ? __ldcg(hand + o) : (p.h0 ? p.h0[row * P * Nt + n_off + o] : 0.0f);
                hv[pp] = __float_as_uint(v);
            }
            put_h(hv, ex2_approx(cum[Q - 1]));
        }

        for (int64_t c = c_begin; c < c_end; ++c) {
            const int64_t t0 = c * Q;
            const int valid = static_cast<int>(p.L - t0 < Q ? p.L - t0 : Q);
            const uint32_t xs_s = base_s + SH::X_OFF;
            const unsigned char *xt = base + SH::X_OFF;
            uint4 zpre[2], ypre[2];
            wait_cb();
            // ---- S' = C B^T o M o delta in place and w o X; thread (row r, quarter j) does 16
            //      elements of row r: M[t][s] delta_s = e^{cum[t] - cum[s]} delta_s (<= 1) for s <= t
            {
                const int r = tid & (Q - 1), j = tid >> 6;
                unsigned char *srow = base + SH::S_OFF;
                const float ct = cum[r];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int s0 = 16 * j + 8 * k;
                    if ((w & 1) == 0 && s0 >= 32) {   // rows 0-31 of this warp, steps past all of them
                        *reinterpret_cast<uint4 *>(srow + sw128_off(r, s0)) = make_uint4(0, 0, 0, 0);
                        continue;
                    }
                    const uint4 cbw = *reinterpret_cast<const uint4 *>(srow + sw128_off(r, s0));
                    const uint32_t wv[4] = {cbw.x, cbw.y, cbw.z, cbw.w};
                    const ulonglong2 cu0 = *reinterpret_cast<const ulonglong2 *>(cum + s0);   // step pairs
                    const ulonglong2 cu1 = *reinterpret_cast<const ulonglong2 *>(cum + s0 + 4);
                    const ulonglong2 dd0 = *reinterpret_cast<const ulonglong2 *>(dl + s0);
                    const ulonglong2 dd1 = *reinterpret_cast<const ulonglong2 *>(dl + s0 + 4);
                    const u64 cu[4] = {cu0.x, cu0.y, cu1.x, cu1.y};
                    const u64 dd[4] = {dd0.x, dd0.y, dd1.x, dd1.y};
                    const u64 ct2 = splat(ct), m1 = splat(-1.0f);
                    uint32_t ow[4];
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        const int e = 2 * e2;
                        // C B^T e^{cum[t] - cum[s]} delta_s for the pair of steps s, s + 1
                        const u64 g = mul2(mul2(ex2_2(fma2(cu[e2], m1, ct2)), dd[e2]),
                                           pk(bf16lo(wv[e2]), bf16hi(wv[e2])));
                        float v0, v1;
                        upk(g, v0, v1);
                        v0 = (s0 + e <= r) ? v0 : 0.0f;
                        v1 = (s0 + e + 1 <= r) ? v1 : 0.0f;
                        v0 += (s0 + e == r) ? Dh : 0.0f;   // the skip term D x through the diagonal
                        v1 += (s0 + e + 1 == r) ? Dh : 0.0f;
                        ow[e2] = pack_bf16x2(v0, v1);
                    }
                    *reinterpret_cast<uint4 *>(srow + sw128_off(r, s0)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                }
                // the C rows scaled by e^{cum[t]} (the decay of the carried state to step t)
                const u64 er = splat(ecum[r]);
                unsigned char *crow = base + SH::C_OFF;
#pragma unroll
                for (int k2 = 0; k2 < N / 32; ++k2) {
                    const int n0 = 8 * j + 32 * k2;   // pieces j, j + 4, .. of the row
                    unsigned char *cp = crow + (n0 / 64) * SH::CT + sw128_off(r, n0 % 64);
                    const uint4 cv = *reinterpret_cast<const uint4 *>(cp);
                    *reinterpret_cast<uint4 *>(cp) = make_uint4(scale_bf16x2(cv.x, er), scale_bf16x2(cv.y, er),
                                                                scale_bf16x2(cv.z, er), scale_bf16x2(cv.w, er));
                }
                const u64 ws = splat(wsx[r]);
                unsigned char *xw = base + SH::XW_OFF;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int p0 = 8 * j + 32 * k;
                    const uint4 xv = *reinterpret_cast<const uint4 *>(xt + sw128_off(r, p0));
                    *reinterpret_cast<uint4 *>(xw + sw128_off(r, p0)) = make_uint4(
                        scale_bf16x2(xv.x, ws), scale_bf16x2(xv.y, ws), scale_bf16x2(xv.z, ws), scale_bf16x2(xv.w, ws));
                }
            }
            tmem_st_wait();
            fence_proxy_async();
            tc_fence_before();
            const int go = __syncthreads_and(aborted ? 0 : 1);
            tc_fence_after();
            if (!go) {
                aborted = true;
                break;
            }
            if (tid == 0) {
                constexpr uint32_t id_y = umma_idesc_bf16_mj(64, 64, 0, 1);
                constexpr uint32_t id_h = umma_idesc_bf16_mj(N, 64, 1, 1);
                // Y = (e^cum C) H^T: A = scaled C (K-major, 64-state slices), B = H stored [n][p] (MN-major)
#pragma unroll
                for (int kk = 0; kk < N / 16; ++kk)
                    umma_bf16(t_y, umma_desc_sw128(base_s + SH::C_OFF + (kk / 4) * SH::CT + (kk % 4) * 32),
                              umma_desc_mn_sw128(base_s + SH::H_OFF + kk * 2048, 8192), id_y, kk > 0);
                // Y += (S' + D I) X: A = S' (K-major), B = X stored [s][p] (MN-major)
#pragma unroll
                for (int kk = 0; kk < Q / 16; ++kk)
                    umma_bf16(t_y, umma_desc_sw128(base_s + SH::S_OFF + kk * 32),
                              umma_desc_mn_sw128(xs_s + kk * 2048, 8192), id_y, true);
                // H^T += B^T (w o X): A = B stored [s][n] (MN-major, 64-state atoms CT bytes apart),
                // B = w o X stored [s][p] (MN-major)
#pragma unroll
                for (int kk = 0; kk < Q / 16; ++kk)
                    umma_bf16(t_h, umma_desc_mn_sw128(base_s + SH::B_OFF + kk * 2048, SH::CT),
                              umma_desc_mn_sw128(base_s + SH::XW_OFF + kk * 2048, 8192), id_h, true);
                umma_commit(bar_mma);
            }
            {   // the gate inputs of this thread's epilogue piece, fetched while the products run
                const int t = 16 * q + (lane & 15), half = lane >> 4;
                const int64_t ro = (b * p.L + t0 + t) * xs + static_cast<int64_t>(h) * P + 32 * half + 16 * hf;
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    zpre[k] = (gate && t < valid) ? __ldg(reinterpret_cast<const uint4 *>(p.z + ro + 8 * k))
                                                  : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int k = 0; k < 2; ++k)   // the first half's partial y (second-half pass)
                    ypre[k] = (add_partial && t < valid) ? *reinterpret_cast<const uint4 *>(p.y + ro + 8 * k)
                                                         : make_uint4(0, 0, 0, 0);
            }
            if (w == kSsdStepWarp && c + 1 < c_end) {   // the next chunk's step sizes, also while the products run
                step_sizes(c + 1);
                load_dt(c + 2);
            }
            const bool mma_ok = __syncthreads_and(mbar_wait(bar_mma, static_cast<uint32_t>(mma_phase & 1)) ? 1 : 0) != 0;
            ++mma_phase;
            tc_fence_after();
            // X, C, B and C B^T are free: the next chunk's land while this one finishes
            if (c + 1 < c_end && mma_ok)
                issue_cb(c + 1);
            // ---- epilogue: y[t][p] = Y[t][p] silu(z); warp w holds rows t = 16q .. 16q+15,
            //      lane l row 16q + (l % 16), columns 32 (l / 16) + 16 hf .. (16 of them)
            {
                uint32_t yv[16];
                tmem_ld16_split<32>(t_y + lane_base + 16 * hf, yv);
                tmem_ld_wait();
                const int t = 16 * q + (lane & 15), half = lane >> 4;
                unsigned char *yt = base + SH::XW_OFF;   // y of the chunk, [t][p] 128-byte swizzled, for one tensor store
#pragma unroll
                for (int k4 = 0; k4 < 2; ++k4) {
                    const uint32_t zw4[4] = {zpre[k4].x, zpre[k4].y, zpre[k4].z, zpre[k4].w};
                    const uint32_t yw4[4] = {ypre[k4].x, ypre[k4].y, ypre[k4].z, ypre[k4].w};
                    uint32_t ow[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int pp = 8 * k4 + 2 * e;
                        float o0 = __uint_as_float(yv[pp]), o1 = __uint_as_float(yv[pp + 1]);
                        if (add_partial) {
                            o0 += bf16lo(yw4[e]);
                            o1 += bf16hi(yw4[e]);
                        }
                        if (gate) {
                            o0 *= silu_f(bf16lo(zw4[e]));
                            o1 *= silu_f(bf16hi(zw4[e]));
                        }
                        ow[e] = pack_bf16x2(o0, o1);
                    }
                    *reinterpret_cast<uint4 *>(yt + sw128_off(t, 32 * half + 16 * hf + 8 * k4)) =
                        make_uint4(ow[0], ow[1], ow[2], ow[3]);
                }
                fence_proxy_async();
            }
            if (!mma_ok) {
                aborted = true;
                break;
            }
            tc_fence_before();
            __syncthreads();   // every thread is done with this chunk's S', w o X, bf16 H and Y
            tc_fence_after();
            if (tid == 0) {   // y of the chunk (steps past L are dropped by the map)
                ssd_tma_store_3d(&p.tm_yq, base_s + SH::XW_OFF, h * P, static_cast<int>(t0), static_cast<int>(b));
                ssd_bulk_commit();
            }
            if (c + 1 < c_end) {   // the state entering the next chunk, meanwhile
                uint32_t hv[32];
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    tmem_ld16(t_h + lane_base + 32 * hf + 16 * j, hv + 16 * j);
                tmem_ld_wait();
                put_h(hv, ex2_approx(cum[Q - 1]));
            }
            if (tid == 0)
                ssd_bulk_wait_read_all();
            __syncthreads();   // y has left the w o X buffer before the next chunk writes it
        }
        if (aborted)
            break;
        // the state at the end of the segment: handed to the row's next segment, or the final state
        if (!last || p.final_state) {
            uint32_t hv[32];
#pragma unroll
            for (int j = 0; j < 2; ++j)
                tmem_ld16(t_h + lane_base + 32 * hf + 16 * j, hv + 16 * j);
            tmem_ld_wait();
            if (hrow >= 0) {
                float *dst = last ? p.final_state + row * P * Nt + n_off : hand;
#pragma unroll
                for (int pp = 0; pp < 32; ++pp)
                    dst[static_cast<int64_t>(32 * hf + pp) * Nt + hrow] = __uint_as_float(hv[pp]);
            }
            if (!last)
                __threadfence();
        }
        tc_fence_before();
        __syncthreads();   // the end state is out of tensor memory before the next item's enters
        tc_fence_after();
        if (!last && tid == 0)
            ssd_flag_release(p.work + 1 + row, static_cast<unsigned int>(seg + 1));
    }
    if (tid == 0)
        ssd_bulk_wait_all();
    if (tid == 0)   // copies issued and not yet waited for (after an abort) land before the CTA leaves
        for (int i = cb_done; i < cb_issued; ++i)
            mbar_wait(bar_cb, static_cast<uint32_t>(i & 1));
    tc_fence_before();
    __syncthreads();
    if (w == 0)
        tmem_dealloc(tmem, SH::TCOLS);
}

template <int N>
struct SsdShape {
    static constexpr int Q = kSsdQ, P = kSsdP;
    static constexpr int LDP = P + 8, LDN = N + 8, LDQ = Q + 8;
    static constexpr int X_OFF = 0;                                  // X_c   [Q][LDP] bf16
    static constexpr int B_OFF = X_OFF + Q * LDP * 2;                // B_c   [Q][LDN] bf16
    static constexpr int C_OFF = B_OFF + Q * LDN * 2;                // C_c   [Q][LDN] bf16
    static constexpr int CB_OFF = C_OFF + Q * LDN * 2;               // CB_c  [Q][LDQ] bf16
    static constexpr int S_OFF = CB_OFF + Q * LDQ * 2;               // S'_c  [Q][LDQ] bf16
    static constexpr int XW_OFF = S_OFF + Q * LDQ * 2;               // w o X [Q][LDP] bf16
    static constexpr int CUM_OFF = XW_OFF + Q * LDP * 2;             // cum, delta, e^cum, e4, w [Q] fp32
    static constexpr int BAR_OFF = CUM_OFF + 5 * Q * 4;              // "C, CB landed", "X, B landed"
    static constexpr size_t BYTES = BAR_OFF + 16;
    static_assert(B_OFF % 128 == 0 && C_OFF % 128 == 0 && CB_OFF % 128 == 0 && BAR_OFF % 8 == 0,
                  "tensor-copy destinations on 128-byte boundaries");
};

// ---- one CTA (4 warps) per (batch, head); the chunks of the row in order.
// Warp w owns channels p = 16w .. 16w+15: those rows of H and those columns of Y_c.
// TMA: the tiles arrive by tensor copies (the maps in p are encoded); the
// cp.async form is a separate instantiation, so neither carries the other's
// registers.
template <int N, bool TMA>
__global__ void __launch_bounds__(128, 3)
ssd_chunk_kernel(const __grid_constant__ SsdParams p)
{
    using SH = SsdShape<N>;
    constexpr int Q = SH::Q, P = SH::P, LDP = SH::LDP, LDN = SH::LDN, LDQ = SH::LDQ;
    constexpr int NT = N / 8;   // 8-column tiles of the state
    extern __shared__ __align__(128) unsigned char smem_ssd[];
    unsigned char *smem_raw = smem_ssd;
    __nv_bfloat16 *Xs = reinterpret_cast<__nv_bfloat16 *>(smem_raw + SH::X_OFF);
    __nv_bfloat16 *Bs = reinterpret_cast<__nv_bfloat16 *>(smem_raw + SH::B_OFF);
    __nv_bfloat16 *Cs = reinterpret_cast<__nv_bfloat16 *>(smem_raw + SH::C_OFF);
    __nv_bfloat16 *CBs = reinterpret_cast<__nv_bfloat16 *>(smem_raw + SH::CB_OFF);
    __nv_bfloat16 *Sp = reinterpret_cast<__nv_bfloat16 *>(smem_raw + SH::S_OFF);
    __nv_bfloat16 *Xw = reinterpret_cast<__nv_bfloat16 *>(smem_raw + SH::XW_OFF);
    float *cum = reinterpret_cast<float *>(smem_raw + SH::CUM_OFF);
    float *dl = cum + Q;
    float *ecum = dl + Q;
    float *e4 = ecum + Q;    // e^{cum[t] - cum[t-4]} (t >= 4)
    float *wsx = e4 + Q;     // w_s = e^{cum[Q-1] - cum[s]} delta_s

    const int64_t b = blockIdx.y;
    const int h = blockIdx.x;
    const int g = static_cast<int>(h / (p.H / p.G));
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int gr = lane >> 2, t4 = lane & 3;
    const float Ah = __ldg(p.A + h);
    const float Dh = p.D ? __ldg(p.D + h) : 0.0f;
    const float bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.0f;
    const bool gate = p.z != nullptr;
    const int xs = static_cast<int>(p.H * P);   // x, z, y row stride (one time step)
    const int bcs = static_cast<int>(p.G * N);  // B, C row stride
    const int dts = static_cast<int>(p.H);      // dt row stride

    // the carried state H, fp32 fragments: rows p = 16w + gr (+8), columns n = 8j + 2t4 (+1)
    float Hf[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int pr = 16 * w + gr + (e >> 1) * 8;
            const int n = 8 * j + 2 * t4 + (e & 1);
            Hf[j][e] = p.h0 ? p.h0[((b * p.H + h) * P + pr) * N + n] : 0.0f;
        }
    }
    bool have_state = p.h0 != nullptr;

    // Tiles arrive by tensor copies when the maps are given (and shared memory
    // starts on a 128-byte boundary), else by 16-byte cp.async pieces. Each of
    // the two barriers completes once per chunk (phase parity c & 1); waits are
    // bounded, and after one gives up the CTA issues and waits no more and
    // thread 0 lets the copies it issued land before exiting.
    const uint32_t smem_s = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
    constexpr bool tma = TMA;
    if (TMA && (smem_s & 127u) != 0) {   // tensor copies need 128-byte aligned destinations
        if (tid == 0)
            atomicOr(&g_fault_flags, kFaultSmemAlign);
        return;
    }
    const uint32_t bar_cc = smem_s + SH::BAR_OFF, bar_xb = bar_cc + 8;
    int cc_issued = 0, cc_done = 0, xb_issued = 0, xb_done = 0;   // chunk counts (< 2^31)
    bool aborted = false;
    if (tma) {
        if (tid == 0) {
            mbar_init(bar_cc, 1);
            mbar_init(bar_xb, 1);
            mbar_fence_init();
        }
        __syncthreads();
    }

    // C_c and C_c B_c^T of chunk c (issued early: their buffers free up first)
    auto stage_c = [&](int64_t c) {
        const int64_t t0 = c * Q;
        if constexpr (TMA) {
            if (tid == 0 && !aborted) {
                mbar_expect_tx(bar_cc, 2 * Q * LDN + 2 * Q * LDQ);
                tma_load_3d(smem_s + SH::C_OFF, &p.tm_C, bar_cc, g * N, static_cast<int>(t0), static_cast<int>(b));
                tma_load_3d(smem_s + SH::CB_OFF, &p.tm_cb, bar_cc, 0, 0,
                            static_cast<int>((b * p.nchunks + c) * p.G + g));
                cc_issued = static_cast<int>(c) + 1;
            }
        } else {
            const int valid = static_cast<int>(p.L - t0 < Q ? p.L - t0 : Q);
            stage_rows(Cs, LDN, p.C + ((b * p.L + t0) * p.G + g) * N, bcs, Q, N, valid, tid, 128);
            stage_rows(CBs, LDQ, p.cb + (((b * p.nchunks + c) * p.G + g) * Q) * Q, Q, Q, Q, Q, tid, 128);
            cp_async_commit();
        }
    };
    // X_c and B_c
    auto stage_xb = [&](int64_t c) {
        const int64_t t0 = c * Q;
        if constexpr (TMA) {
            if (tid == 0 && !aborted) {
                mbar_expect_tx(bar_xb, 2 * Q * LDP + 2 * Q * LDN);
                tma_load_3d(smem_s + SH::X_OFF, &p.tm_x, bar_xb, h * P, static_cast<int>(t0), static_cast<int>(b));
                tma_load_3d(smem_s + SH::B_OFF, &p.tm_B, bar_xb, g * N, static_cast<int>(t0), static_cast<int>(b));
                xb_issued = static_cast<int>(c) + 1;
            }
        } else {
            const int v = static_cast<int>(p.L - t0 < Q ? p.L - t0 : Q);
            stage_rows(Xs, LDP, p.x + ((b * p.L + t0) * p.H + h) * P, xs, Q, P, v, tid, 128);
            stage_rows(Bs, LDN, p.B + ((b * p.L + t0) * p.G + g) * N, bcs, Q, N, v, tid, 128);
            cp_async_commit();
        }
    };
    auto wait_chunk = [&](int64_t c) {
        if (tma && !aborted) {
            const uint32_t par = static_cast<uint32_t>(c & 1);
            aborted = !mbar_wait(bar_cc, par) || !mbar_wait(bar_xb, par);
            if (!aborted)
                cc_done = xb_done = static_cast<int>(c) + 1;
        }
    };
    stage_c(0);
    stage_xb(0);
    // raw step of this thread's row of the next chunk, fetched a chunk ahead
    auto load_dt = [&](int64_t c) -> float {
        const int64_t t = c * Q + tid;
        return (tid < Q && t < p.L) ? __bfloat162float(p.dt[(b * p.L + t) * dts + h]) : 0.0f;
    };
    float dt_next = load_dt(0);

    for (int64_t c = 0; c < p.nchunks; ++c) {
        const int64_t t0 = c * Q;
        const int valid = static_cast<int>(p.L - t0 < Q ? p.L - t0 : Q);
        // ---- (X_c and B_c were issued at the end of the previous chunk); the step sizes (zero past L)
        if (tid < Q) {
            float d = 0.0f;
            if (tid < valid) {
                const float v = dt_next + bias;
                d = p.softplus ? softplus_f(v) : v;
            }
            dl[tid] = d;
        }
        if (c + 1 < p.nchunks)
            dt_next = load_dt(c + 1);
        cp_async_wait<0>();
        wait_chunk(c);
        __syncthreads();
        // ---- cum[t] = A_h * (delta_0 + .. + delta_t) in units of log2 e, one warp; with
        // it e^{cum}, the 4-step decays e4 and the state-update weights w
        if (w == 0) {
            const float a0 = Ah * kLog2e * dl[2 * lane], a1 = Ah * kLog2e * dl[2 * lane + 1];
            float sum = a0 + a1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, sum, o);
                if (lane >= o)
                    sum += u;
            }
            const float c0 = sum - a1, c1 = sum;
            cum[2 * lane] = c0;
            cum[2 * lane + 1] = c1;
            ecum[2 * lane] = ex2_approx(c0);
            ecum[2 * lane + 1] = ex2_approx(c1);
            const float cq = __shfl_sync(0xffffffffu, c1, 31);
            wsx[2 * lane] = ex2_approx(cq - c0) * dl[2 * lane];
            wsx[2 * lane + 1] = ex2_approx(cq - c1) * dl[2 * lane + 1];
            const float q0 = __shfl_up_sync(0xffffffffu, c0, 2), q1 = __shfl_up_sync(0xffffffffu, c1, 2);
            e4[2 * lane] = ex2_approx(c0 - q0);   // lanes 0, 1 (t < 4): unused
            e4[2 * lane + 1] = ex2_approx(c1 - q1);
        }
        __syncthreads();
        // ---- S' = CB o M o delta and w o X, both bf16. A thread owns columns s2, s2 + 1
        // and the rows t = t0 + 4k: M[t][s] delta_s starts at the first such row on or
        // below the diagonal and is carried down with M[t][s] = M[t-4][s] e4[t].
        {
            const int s2 = 2 * (tid & 31), t0 = tid >> 5;
            const int tf0 = s2 + ((t0 - s2) & 3), tf1 = s2 + 1 + ((t0 - s2 - 1) & 3);
            float m0 = tf0 < Q ? ex2_approx(cum[tf0] - cum[s2]) * dl[s2] : 0.0f;
            float m1 = tf1 < Q ? ex2_approx(cum[tf1] - cum[s2 + 1]) * dl[s2 + 1] : 0.0f;
#pragma unroll 4
            for (int k = 0; k < Q / 4; ++k) {
                const int t = t0 + 4 * k;
                const uint32_t cb2 = *reinterpret_cast<const uint32_t *>(CBs + t * LDQ + s2);
                const float f = e4[t];
                m0 = t > tf0 ? m0 * f : m0;
                m1 = t > tf1 ? m1 * f : m1;
                const float v0 = t >= tf0 ? bf16lo(cb2) * m0 : 0.0f;
                const float v1 = t >= tf1 ? bf16hi(cb2) * m1 : 0.0f;
                *reinterpret_cast<uint32_t *>(Sp + t * LDQ + s2) = pack_bf16x2(v0, v1);
            }
        }
        for (int i = tid; i < Q * P / 8; i += 128) {
            const int s_ = i >> 3, p8 = (i & 7) * 8;   // P / 8 = 8 16-byte pieces per row
            const float ws = wsx[s_];
            const uint4 xw = *reinterpret_cast<const uint4 *>(Xs + s_ * LDP + p8);
            uint4 o;
            o.x = pack_bf16x2(bf16lo(xw.x) * ws, bf16hi(xw.x) * ws);
            o.y = pack_bf16x2(bf16lo(xw.y) * ws, bf16hi(xw.y) * ws);
            o.z = pack_bf16x2(bf16lo(xw.z) * ws, bf16hi(xw.z) * ws);
            o.w = pack_bf16x2(bf16lo(xw.w) * ws, bf16hi(xw.w) * ws);
            *reinterpret_cast<uint4 *>(Xw + s_ * LDP + p8) = o;
        }
        __syncthreads();

        // ---- Y columns p = 16w .. 16w+15, all Q rows: e^{cum[t]} C_c H^T + S' X_c.
        // The warp's own state rows are the B operand of C_c H^T, converted to
        // bf16 from the fp32 accumulator registers that hold them.
        float acc[4][2][4];   // [row tile][column tile][fragment]
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
                acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.0f;
        if (have_state) {
#pragma unroll
            for (int kk = 0; kk < N / 16; ++kk) {
                uint32_t bh[2][2];   // [column tile][b0, b1]
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int half = 0; half < 2; ++half)
                        bh[nt][half] = pack_bf16x2(Hf[2 * kk + half][2 * nt], Hf[2 * kk + half][2 * nt + 1]);
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    uint32_t a[4];
                    frag_a(Cs, LDN, 16 * mt, 16 * kk, lane, a);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        mma_bf16(acc[mt][nt], a[0], a[1], a[2], a[3], bh[nt][0], bh[nt][1]);
                }
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const float e0 = ecum[16 * mt + gr], e1 = ecum[16 * mt + gr + 8];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    acc[mt][nt][0] *= e0;
                    acc[mt][nt][1] *= e0;
                    acc[mt][nt][2] *= e1;
                    acc[mt][nt][3] *= e1;
                }
            }
        }
        __syncthreads();   // Cs and CBs are free: fetch the next chunk's while this one finishes
        if (c + 1 < p.nchunks)
            stage_c(c + 1);
        // the gate's z of this warp's outputs, fetched before the products that precede their use
        uint32_t zv[4][2][2];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int t = 16 * mt + gr + half * 8;
                const __nv_bfloat16 *zr = p.z + ((b * p.L + t0) * p.H + h) * P + t * static_cast<int64_t>(xs);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    zv[mt][half][nt] = (gate && t < valid)
                                           ? __ldg(reinterpret_cast<const unsigned int *>(zr + 16 * w + 8 * nt + 2 * t4))
                                           : 0u;
            }
#pragma unroll
        for (int kk = 0; kk < Q; kk += 16) {
            uint32_t bb[4];
            frag_b_kn(Xs, LDP, 16 * w, kk, lane, bb);    // X stored [s][p]: k = s, columns 16w ..
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                uint32_t a[4];
                frag_a(Sp, LDQ, 16 * mt, kk, lane, a);
                mma_bf16(acc[mt][0], a[0], a[1], a[2], a[3], bb[0], bb[1]);
                mma_bf16(acc[mt][1], a[0], a[1], a[2], a[3], bb[2], bb[3]);
            }
        }
        // x of this warp's outputs (for D x), so that the shared tiles can be refilled
        uint32_t xv[4][2][2];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    xv[mt][half][nt] = *reinterpret_cast<const uint32_t *>(
                        Xs + (16 * mt + gr + half * 8) * LDP + 16 * w + 8 * nt + 2 * t4);

        // ---- H rows p = 16w .. : e^{cum[Q-1]} H + (w o X)^T B_c
        const float ec = ecum[Q - 1];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            Hf[j][0] *= ec;
            Hf[j][1] *= ec;
            Hf[j][2] *= ec;
            Hf[j][3] *= ec;
        }
#pragma unroll
        for (int kk = 0; kk < Q; kk += 16) {
            uint32_t a[4];
            frag_a_t(Xw, LDP, 16 * w, kk, lane, a);          // A[p][s] = Xw[s][p]
#pragma unroll
            for (int j = 0; j < NT; j += 2) {
                uint32_t bb[4];
                frag_b_kn(Bs, LDN, 8 * j, kk, lane, bb);     // B_c stored [s][n]: k = s, column n
                mma_bf16(Hf[j], a[0], a[1], a[2], a[3], bb[0], bb[1]);
                mma_bf16(Hf[j + 1], a[0], a[1], a[2], a[3], bb[2], bb[3]);
            }
        }
        have_state = true;
        __syncthreads();   // every warp is done with Xs, Bs, Sp, Xw and the step sizes of this chunk
        // the next chunk's X and B land while this one's outputs are written
        if (c + 1 < p.nchunks)
            stage_xb(c + 1);
        // ---- epilogue: + D x, gate, store
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int t = 16 * mt + gr + half * 8;
                if (t < valid) {
                    const int64_t ro = t * static_cast<int64_t>(xs);
                    __nv_bfloat16 *yr = p.y + ((b * p.L + t0) * p.H + h) * P + ro;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const int col = 16 * w + 8 * nt + 2 * t4;
                        const uint32_t xw = xv[mt][half][nt];
                        float o0 = fmaf(Dh, bf16lo(xw), acc[mt][nt][2 * half]);
                        float o1 = fmaf(Dh, bf16hi(xw), acc[mt][nt][2 * half + 1]);
                        if (gate) {
                            const uint32_t zw = zv[mt][half][nt];
                            o0 *= silu_f(bf16lo(zw));
                            o1 *= silu_f(bf16hi(zw));
                        }
                        *reinterpret_cast<uint32_t *>(yr + col) = pack_bf16x2(o0, o1);
                    }
                }
            }
        }

    }
    if (p.final_state) {
        float *fs = p.final_state + ((b * p.H + h) * P) * N;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int n = 8 * j + 2 * t4;
            *reinterpret_cast<float2 *>(fs + (16 * w + gr) * N + n) = make_float2(Hf[j][0], Hf[j][1]);
            *reinterpret_cast<float2 *>(fs + (16 * w + gr + 8) * N + n) = make_float2(Hf[j][2], Hf[j][3]);
        }
    }
    if (tma && tid == 0) {   // after a wait gave up: let the copies issued since land (each wait bounded)
        for (int c = cc_done; c < cc_issued; ++c)
            mbar_wait(bar_cc, static_cast<uint32_t>(c & 1));
        for (int c = xb_done; c < xb_issued; ++c)
            mbar_wait(bar_xb, static_cast<uint32_t>(c & 1));
    }
}
