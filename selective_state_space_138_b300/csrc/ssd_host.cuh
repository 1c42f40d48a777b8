// ssd_host.cuh -- the host side of the SSD: workspace layout, tensor maps,
// segment choice and launches of the kernels in ssd.cuh.
//
// Part of the single translation unit ss_scan.cu (included inside its
// anonymous namespace, after ssd.cuh); not compiled on its own.

#pragma once

// ------------------------------------------------------------------ SSD host side

// The workspace: C B^T of every chunk ([batch][nchunks][G][Q][Q] bf16), then the
// chunk walk's counters (1 + batch * nheads words), then the states handed between
// the chunk segments of a row (batch * nheads * P * N fp32); each part starts on a
// 256-byte boundary. Sizes are checked by the caller (ssd_fwd) or give 0 here.
struct SsdWorkspace {
    size_t cb, work, hbuf, total;
};

SsdWorkspace ssd_workspace_layout(int64_t batch, int64_t L, int64_t H, int64_t G, int64_t N)
{
    SsdWorkspace w{0, 0, 0, 0};
    if (batch <= 0 || L <= 0 || H <= 0 || G <= 0 || N <= 0 || G > H || N > 256 || L > (int64_t(1) << 40) ||
        batch > (int64_t(1) << 40) / L || batch > (int64_t(1) << 40) / H)
        return w;
    const int64_t nchunks = (L + kSsdQ - 1) / kSsdQ;
    if (batch * nchunks > (int64_t(1) << 40) / G)
        return w;
    auto up = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
    w.work = up(static_cast<size_t>(batch) * nchunks * G * kSsdQ * kSsdQ * 2);
    w.hbuf = w.work + up((1 + static_cast<size_t>(batch) * H) * 4);
    w.total = w.hbuf + static_cast<size_t>(batch) * H * kSsdP * N * 4;
    return w;
}

size_t ssd_workspace_bytes(int64_t batch, int64_t L, int64_t H, int64_t G, int64_t N)
{
    return ssd_workspace_layout(batch, L, H, G, N).total;
}

// Chunk segments per row for the tensor-core chunk walk: with rows (b, h) walked by
// `slots` resident CTAs that claim work items in order, a CTA walks at most
// ceil(rows * s / slots) items of nchunks / s chunks; s = 2 or 4 when that is shorter
// than s = 1 (SS_SSD_SEGMENTS overrides). A row's segments still run one after another.
int ssd_pick_segments(int64_t rows, int64_t nchunks, int64_t slots)
{
    int s_best = 1;
    if (const char *env = getenv("SS_SSD_SEGMENTS")) {
        const int v = atoi(env);
        if (v >= 1 && v <= 8)
            s_best = v;
    } else if (slots > 0) {
        int64_t num = (rows + slots - 1) / slots, den = 1;   // the cost ceil(rows s / slots) / s
        for (int s = 2; s <= 4; s *= 2) {
            const int64_t k = (rows * s + slots - 1) / slots;
            if (nchunks >= s && (nchunks + s - 1) / s <= 4096 && k * den < num * s) {
                num = k;
                den = s;
                s_best = s;
            }
        }
    }
    return static_cast<int>(std::min<int64_t>(s_best, nchunks));
}

// The grid and segments of ssd_chunk_tc_kernel<N>: one CTA per resident slot at most
template <int N>
ss_status ssd_tc_grid(SsdParams &p, unsigned *grid)
{
    using TS = SsdTcShape<N>;
    static std::atomic<int> per_sm{0};
    static std::atomic<int> sms{0};
    if (per_sm.load() == 0) {
        // CTAs per SM from the kernel's registers and shared memory, the SM's limits and
        // the 512 tensor-memory columns (the runtime's occupancy query answers 1 for this
        // kernel). The work items are claimed dynamically, so the result is a grid size,
        // not a residency the kernel relies on.
        int dev = 0, n_sm = 0, regs_sm = 0, smem_sm = 0, smem_rsv = 0, thr_sm = 0;
        cudaFuncAttributes fa{};
        cudaError_t e = cudaFuncSetAttribute(ssd_chunk_tc_kernel<N>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
        if (e == cudaSuccess)
            e = cudaGetDevice(&dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
        if (e == cudaSuccess)
            e = cudaFuncGetAttributes(&fa, ssd_chunk_tc_kernel<N>);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SS_ERR_LAUNCH, "device or kernel attribute query failed: %s", cudaGetErrorString(e));
        }
        const int warp_regs = (fa.numRegs * 32 + 255) / 256 * 256;   // registers go to warps 256 at a time
        int occ = std::min(thr_sm / kSsdTcThreads, 512 / static_cast<int>(TS::TCOLS));
        occ = std::min(occ, regs_sm / (warp_regs * (kSsdTcThreads / 32)));
        occ = std::min(occ, smem_sm / (static_cast<int>(TS::BYTES + fa.sharedSizeBytes) + smem_rsv));
        sms.store(n_sm > 0 ? n_sm : 1);
        per_sm.store(occ > 0 ? occ : 1);
    }
    const int64_t rows = p.batch * p.H;
    const int64_t slots = static_cast<int64_t>(per_sm.load()) * sms.load();
    p.nseg = ssd_pick_segments(rows, p.nchunks, slots);
    p.cps = static_cast<int>((p.nchunks + p.nseg - 1) / p.nseg);
    p.nseg = static_cast<int>((p.nchunks + p.cps - 1) / p.cps);   // no empty segment
    const int64_t items = rows * p.nseg;
    if (items > 0x7fffffff)
        return fail(SS_ERR_DIM, "too many work items for the chunk walk");
    *grid = static_cast<unsigned>(std::min(items, slots));
    return SS_OK;
}

// 3-d bf16 tensor map (d0 contiguous, then d1, d2; strides in bytes) with box
// (b0, b1, 1); elements outside the tensor read as zero
bool ssd_encode_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                   uint64_t s2, uint32_t b0, uint32_t b1,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE)
{
    const EncodeTiledFn fn = encode_tiled_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1, s2};
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-core kernels' tile maps (128-byte swizzled boxes of 64 states or
// channels): B, C over (G*N, L, batch) with 64 states x 128 steps (C B^T) and
// 64 states x Q steps (the chunk walk); x and y over (H*P, L, batch) with 64
// channels x Q steps; C B^T over (Q, Q, batch*nchunks*G).
bool ssd_encode_tc_maps(SsdParams &p, int64_t N)
{
    constexpr int Q = kSsdQ, P = kSsdP;
    const uint64_t HP = static_cast<uint64_t>(p.H) * P, GN = static_cast<uint64_t>(p.G) * N;
    const uint64_t L = static_cast<uint64_t>(p.L), bt = static_cast<uint64_t>(p.batch);
    return ssd_encode_3d(&p.tm_Bsw, p.B, GN, L, bt, GN * 2, GN * L * 2, 64, 2 * Q, CU_TENSOR_MAP_SWIZZLE_128B) &&
           ssd_encode_3d(&p.tm_Csw, p.C, GN, L, bt, GN * 2, GN * L * 2, 64, 2 * Q, CU_TENSOR_MAP_SWIZZLE_128B) &&
           ssd_encode_3d(&p.tm_xq, p.x, HP, L, bt, HP * 2, HP * L * 2, 64, Q, CU_TENSOR_MAP_SWIZZLE_128B) &&
           ssd_encode_3d(&p.tm_Bq, p.B, GN, L, bt, GN * 2, GN * L * 2, 64, Q, CU_TENSOR_MAP_SWIZZLE_128B) &&
           ssd_encode_3d(&p.tm_Cq, p.C, GN, L, bt, GN * 2, GN * L * 2, 64, Q, CU_TENSOR_MAP_SWIZZLE_128B) &&
           ssd_encode_3d(&p.tm_cbq, p.cb, Q, Q, bt * static_cast<uint64_t>(p.nchunks) * static_cast<uint64_t>(p.G),
                         Q * 2, Q * Q * 2, 64, Q, CU_TENSOR_MAP_SWIZZLE_128B) &&
           ssd_encode_3d(&p.tm_yq, p.y, HP, L, bt, HP * 2, HP * L * 2, 64, Q, CU_TENSOR_MAP_SWIZZLE_128B);
}

// All the chunk kernels' tile maps (SS_SCAN_TMA=0 keeps the cp.async pieces):
// the mma.sync kernels' padded boxes (a whole state row + 8) and the
// tensor-core kernels' swizzled ones.
bool ssd_encode_maps(SsdParams &p, int64_t N)
{
    const char *env = getenv("SS_SCAN_TMA");
    if (env && strcmp(env, "0") == 0)
        return false;
    constexpr int Q = kSsdQ, P = kSsdP;
    const uint64_t HP = static_cast<uint64_t>(p.H) * P, GN = static_cast<uint64_t>(p.G) * N;
    const uint64_t L = static_cast<uint64_t>(p.L), bt = static_cast<uint64_t>(p.batch);
    return ssd_encode_3d(&p.tm_x, p.x, HP, L, bt, HP * 2, HP * L * 2, P + 8, Q) &&
           ssd_encode_3d(&p.tm_B, p.B, GN, L, bt, GN * 2, GN * L * 2, static_cast<uint32_t>(N + 8), Q) &&
           ssd_encode_3d(&p.tm_C, p.C, GN, L, bt, GN * 2, GN * L * 2, static_cast<uint32_t>(N + 8), Q) &&
           ssd_encode_3d(&p.tm_cb, p.cb, Q, Q, bt * static_cast<uint64_t>(p.nchunks) * static_cast<uint64_t>(p.G),
                         Q * 2, Q * Q * 2, Q + 8, Q) &&
           ssd_encode_tc_maps(p, N);
}

// N = 256 on the tensor-core kernels: two passes over the 128-state halves.
// The output is linear in the state (y = C h + D x, before the gate), so the
// first pass stores its partial y without the gate (rounded to bf16 once) and
// the second adds it, then gates; B, C, h0 and the final state are addressed
// with their full 256-state stride and the half's offset.
ss_status launch_ssd_halves(SsdParams p, cudaStream_t stream)
{
    using CS = SsdCbShape<128>;
    using TS = SsdTcShape<128>;
    if (p.nchunks > 0x7fffffff || p.batch > 65535 || p.G > 65535 || p.H > 0x7fffffff)
        return fail(SS_ERR_DIM, "grid too large");
    cudaError_t e = cudaFuncSetAttribute(ssd_cb_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(CS::BYTES));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(ssd_chunk_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(TS::BYTES));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SS_ERR_LAUNCH, "cudaFuncSetAttribute failed: %s", cudaGetErrorString(e));
    }
    unsigned grid = 0;
    const ss_status st = ssd_tc_grid<128>(p, &grid);
    if (st != SS_OK)
        return st;
    for (int half = 0; half < 2; ++half) {
        p.n_off = 128 * half;
        p.mode = 1 + half;
        ssd_cb_tc_kernel<128><<<dim3(static_cast<unsigned>((p.nchunks + 1) / 2), static_cast<unsigned>(p.batch),
                                     static_cast<unsigned>(p.G)), 128, CS::BYTES, stream>>>(p);
        ssd_chunk_tc_kernel<128><<<grid, kSsdTcThreads, TS::BYTES, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess)
            return fail(SS_ERR_LAUNCH, "SSD kernel launch failed: %s", cudaGetErrorString(e));
    }
    return SS_OK;
}

template <int N>
ss_status launch_ssd(SsdParams p, cudaStream_t stream)
{
    using SH = SsdShape<N>;
    if (p.nchunks > 0x7fffffff || p.batch > 65535 || p.G > 65535 || p.H > 0x7fffffff)
        return fail(SS_ERR_DIM, "grid too large");
    cudaError_t e = cudaSuccess;
    if (p.tma) {   // C B^T on the tcgen05 tensor cores (tiles by 128-byte swizzled tensor copies)
        using CS = SsdCbShape<N>;
        e = cudaFuncSetAttribute(ssd_cb_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(CS::BYTES));
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SS_ERR_LAUNCH, "cudaFuncSetAttribute failed: %s", cudaGetErrorString(e));
        }
        ssd_cb_tc_kernel<N><<<dim3(static_cast<unsigned>((p.nchunks + 1) / 2), static_cast<unsigned>(p.batch),
                                   static_cast<unsigned>(p.G)), 128, CS::BYTES, stream>>>(p);
    } else {
        ssd_cb_kernel<N><<<dim3(static_cast<unsigned>(p.nchunks), static_cast<unsigned>(p.batch),
                                static_cast<unsigned>(p.G)), 128, 0, stream>>>(p);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SS_ERR_LAUNCH, "SSD CB kernel launch failed: %s", cudaGetErrorString(e));
    const char *env = getenv("SS_SSD_MMA_SYNC");
    if (p.tma && !(env && strcmp(env, "1") == 0)) {   // the chunk walk on the tcgen05 tensor cores
        using TS = SsdTcShape<N>;
        e = cudaFuncSetAttribute(ssd_chunk_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(TS::BYTES));
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SS_ERR_LAUNCH, "cudaFuncSetAttribute failed: %s", cudaGetErrorString(e));
        }
        unsigned grid = 0;
        const ss_status st = ssd_tc_grid<N>(p, &grid);
        if (st != SS_OK)
            return st;
        ssd_chunk_tc_kernel<N><<<grid, kSsdTcThreads, TS::BYTES, stream>>>(p);
    } else {   // mma.sync (rows that cannot be copied by tensor maps, or SS_SSD_MMA_SYNC=1)
        auto kernel = p.tma ? ssd_chunk_kernel<N, true> : ssd_chunk_kernel<N, false>;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SH::BYTES));
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SS_ERR_LAUNCH, "cudaFuncSetAttribute failed: %s", cudaGetErrorString(e));
        }
        kernel<<<dim3(static_cast<unsigned>(p.H), static_cast<unsigned>(p.batch)), 128, SH::BYTES, stream>>>(p);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SS_ERR_LAUNCH, "SSD chunk kernel launch failed: %s", cudaGetErrorString(e));
    return SS_OK;
}

ss_status ssd_fwd(const void *x, const void *dt, const float *A, const void *B, const void *C, const float *D,
                  const void *z, const float *dt_bias, int softplus, const float *h0, void *y, float *final_state,
                  void *workspace, size_t workspace_bytes, int64_t batch, int64_t L, int64_t nheads,
                  int64_t headdim, int64_t ngroups, int64_t N, cudaStream_t stream)
{
    g_err[0] = '\0';
    if (batch <= 0 || L <= 0 || nheads <= 0 || ngroups <= 0)
        return fail(SS_ERR_DIM, "sizes must be positive: batch=%lld L=%lld nheads=%lld ngroups=%lld",
                    (long long)batch, (long long)L, (long long)nheads, (long long)ngroups);
    if (nheads % ngroups != 0)
        return fail(SS_ERR_DIM, "nheads=%lld is not a multiple of ngroups=%lld", (long long)nheads,
                    (long long)ngroups);
    if (headdim != kSsdP)
        return fail(SS_ERR_DIM, "headdim=%lld: this kernel takes headdim %d", (long long)headdim, kSsdP);
    if (N != 64 && N != 128 && N != 256)
        return fail(SS_ERR_N, "N=%lld: this kernel takes N = 64, 128 or 256", (long long)N);
    if (batch > (int64_t(1) << 40) / L || batch * L > (int64_t(1) << 50) / (nheads * headdim))
        return fail(SS_ERR_DIM, "element count overflows");
    const PtrCheck list[] = {{x, "x", true},       {dt, "dt", true},         {A, "A", true},
                             {B, "B", true},       {C, "C", true},           {y, "y", true},
                             {workspace, "workspace", true}, {D, "D", false}, {z, "z", false},
                             {dt_bias, "dt_bias", false},    {h0, "h0", false},
                             {final_state, "final_state", false}};
    int dev = 0;
    ss_status st = check_ptrs(list, static_cast<int>(sizeof(list) / sizeof(list[0])), &dev);
    if (st != SS_OK)
        return st;
    const SsdWorkspace ws = ssd_workspace_layout(batch, L, nheads, ngroups, N);
    const size_t need = ws.total;
    if (need == 0)
        return fail(SS_ERR_DIM, "sizes too large for the workspace");
    if (workspace_bytes < need)
        return fail(SS_ERR_DIM, "workspace of %zu bytes is smaller than the %zu bytes required", workspace_bytes,
                    need);
    const void *ptrs[] = {x, B, C, y, workspace, z};
    for (const void *q : ptrs)
        if (q && !aligned16(q))
            return fail(SS_ERR_DIM, "x, B, C, y, z and the workspace must be 16-byte aligned");
    if ((ngroups * N * 2) % 16 != 0)
        return fail(SS_ERR_DIM, "B and C rows must be whole 16-byte pieces");
    if (nheads * headdim > 0x7fffffff || ngroups * N > 0x7fffffff)
        return fail(SS_ERR_DIM, "nheads * headdim and ngroups * N must fit in 31 bits");
    if (L > 0x7fffffff)   // step coordinates of the tensor copies are 32-bit
        return fail(SS_ERR_DIM, "L=%lld must fit in 31 bits", (long long)L);
    SsdParams p{};
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.dt = static_cast<const __nv_bfloat16 *>(dt);
    p.B = static_cast<const __nv_bfloat16 *>(B);
    p.C = static_cast<const __nv_bfloat16 *>(C);
    p.z = static_cast<const __nv_bfloat16 *>(z);
    p.A = A; p.D = D; p.dt_bias = dt_bias; p.h0 = h0;
    p.y = static_cast<__nv_bfloat16 *>(y);
    p.final_state = final_state;
    p.cb = static_cast<__nv_bfloat16 *>(workspace);
    p.work = reinterpret_cast<unsigned int *>(static_cast<unsigned char *>(workspace) + ws.work);
    p.hbuf = reinterpret_cast<float *>(static_cast<unsigned char *>(workspace) + ws.hbuf);
    p.nseg = 1;
    p.cps = 1;
    p.batch = batch; p.L = L; p.H = nheads; p.G = ngroups;
    p.nchunks = (L + kSsdQ - 1) / kSsdQ;
    p.softplus = softplus ? 1 : 0;
    p.Nt = static_cast<int>(N);
    p.n_off = 0;
    p.mode = 0;
    if (N == 256) {   // the tensor-core kernels only, in two passes over the state halves
        const char *env = getenv("SS_SCAN_TMA");
        if ((env && strcmp(env, "0") == 0) || !ssd_encode_tc_maps(p, N))
            return fail(SS_ERR_N, "N=256 runs on the tensor-core kernels only, whose tensor maps could not be made");
        p.tma = 1;
        return launch_ssd_halves(p, stream);
    }
    p.tma = ssd_encode_maps(p, N) ? 1 : 0;
    return N == 64 ? launch_ssd<64>(p, stream) : launch_ssd<128>(p, stream);
}
