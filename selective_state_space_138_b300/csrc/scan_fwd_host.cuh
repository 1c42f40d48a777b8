// scan_fwd_host.cuh -- the host side of the forward scan: launches, tensor maps,
// the choice of kernel, form and segments, and the entry point's checks.
//
// Part of the single translation unit ss_scan.cu (included inside its
// anonymous namespace, after scan_fwd.cuh); not compiled on its own.

#pragma once

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

// ------------------------------------------------------------------ tensor maps of the n-split kernel

// The n-split kernel's tiles as tensor maps: x, dt, z by channel rows with a
// box of CH channels x one padded raw row (LC steps + 16 bytes), B and C by
// state rows with a box of NS states x LC steps. Needs 16-byte aligned rows
// (the caller's vec condition); SS_SCAN_TMA=0 keeps the cp.async staging.
template <typename T>
bool encode_scan_maps(ScanParams &p)
{
    const char *env = getenv("SS_SCAN_TMA");
    if (env && strcmp(env, "0") == 0)
        return false;
    using SH = NSplitShape<T, 1, 4>;   // CH, LC and the raw row do not depend on the state split
    const uint32_t ns = p.N <= 4 ? 4u : (p.N <= 8 ? 8u : (p.N <= 16 ? 16u : 32u));
    const uint32_t row_t = SH::ROWB / sizeof(T);
    bool ok = encode_rows_map<T>(&p.tm_x, p.x, p.L, p.d_inner, p.batch, row_t, SH::CH) &&
              encode_rows_map<T>(&p.tm_dt, p.dt, p.L, p.d_inner, p.batch, row_t, SH::CH) &&
              encode_rows_map<T>(&p.tm_B, p.B, p.L, p.N, p.batch, SH::LC, ns) &&
              encode_rows_map<T>(&p.tm_C, p.C, p.L, p.N, p.batch, SH::LC, ns);
    if (ok && p.z)
        ok = encode_rows_map<T>(&p.tm_z, p.z, p.L, p.d_inner, p.batch, row_t, SH::CH);
    return ok;
}

template <typename T, int S, int NPL, bool REV, bool RST, int ST = SS_NSPLIT_STAGES>
ss_status launch_nsplit(const ScanParams &p0, cudaStream_t stream, int sms)
{
    using SH = NSplitShape<T, S, NPL, ST>;
    // the wide form (ST != the default) stages by cp.async pieces: its tensor-copy
    // instantiation does not fit four CTAs' registers without spilling
    auto kernel = scan_nsplit_kernel<T, S, NPL, REV, RST, false, ST>;
    if constexpr (ST == SS_NSPLIT_STAGES) {
        if (p0.tma)
            kernel = scan_nsplit_kernel<T, S, NPL, REV, RST, true, ST>;
    }
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
    int nseg = pick_segments(gpr * p.batch, p.L, SH::LC, static_cast<int64_t>(sms) * occ, "SS_SCAN_SEGMENTS");
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

// (warps, states per lane) by N: 4 states per lane, so that a 32-channel
// group runs on ceil(N/4) warps (more warps per SM measured faster than 8
// states per lane on 2 warps); SS_SCAN_NPL=8 selects 8 states per lane for
// 8 < N <= 32.
// The wide form (2 stages, 4 CTAs per SM) for 8 < N <= 16 in the plain direction when
// the channel groups of all batch rows outnumber the CTAs that fit three per SM but not
// four (a grid that would otherwise run a partial second wave); SS_SCAN_WIDE=0 / 1
// turns it off / on whatever the grid.
template <typename T>
bool use_wide_nsplit(const ScanParams &p, int sms)
{
    const char *env = getenv("SS_SCAN_WIDE");
    if (env && strcmp(env, "0") == 0)
        return false;
    if (env && strcmp(env, "1") == 0)
        return true;
    // CTAs per SM of the default and the wide form, queried once (0: not yet; -1: failed)
    static std::atomic<int> occ3_c{0}, occ4_c{0};
    if (occ3_c.load() == 0) {
        auto k3 = scan_nsplit_kernel<T, 4, 4, false, false, true>;
        auto k4 = scan_nsplit_kernel<T, 4, 4, false, false, false, 2>;
        const int b3 = static_cast<int>(NSplitShape<T, 4, 4>::BYTES), b4 = static_cast<int>(NSplitShape<T, 4, 4, 2>::BYTES);
        int o3 = 0, o4 = 0;   // (the dynamic shared memory each asks for is allowed first)
        if (cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, b3) != cudaSuccess ||
            cudaFuncSetAttribute(k4, cudaFuncAttributeMaxDynamicSharedMemorySize, b4) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o3, k3, 128, b3) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o4, k4, 128, b4) != cudaSuccess) {
            cudaGetLastError();
            o3 = o4 = -1;
        }
        occ4_c.store(o4);
        occ3_c.store(o3);
    }
    const int occ3 = occ3_c.load(), occ4 = occ4_c.load();
    if (occ3 < 1 || occ4 < 1)
        return false;
    const int64_t rows = (p.d_inner + 31) / 32 * p.batch;
    return occ4 > occ3 && rows > static_cast<int64_t>(occ3) * sms && rows <= static_cast<int64_t>(occ4) * sms;
}

template <typename T, bool REV, bool RST>
ss_status dispatch_nsplit_n(const ScanParams &p, cudaStream_t s, int sms)
{
    if (p.N <= 4) return launch_nsplit<T, 1, 4, REV, RST>(p, s, sms);
    if (p.N <= 8) return launch_nsplit<T, 2, 4, REV, RST>(p, s, sms);
    const char *env = getenv("SS_SCAN_NPL");
    const bool npl8 = env && strcmp(env, "8") == 0;
    if constexpr (!REV && !RST) {
        if (p.N <= 16 && !npl8 && use_wide_nsplit<T>(p, sms))
            return launch_nsplit<T, 4, 4, false, false, 2>(p, s, sms);
    }
    if (p.N <= 16) return npl8 ? launch_nsplit<T, 2, 8, REV, RST>(p, s, sms) : launch_nsplit<T, 4, 4, REV, RST>(p, s, sms);
    return npl8 ? launch_nsplit<T, 4, 8, REV, RST>(p, s, sms) : launch_nsplit<T, 8, 4, REV, RST>(p, s, sms);
}

template <typename T>
ss_status dispatch_nsplit(const ScanParams &p, bool reverse, cudaStream_t s, int sms)
{
    const bool rst = p.reset != nullptr;
    if (!reverse && !rst) return dispatch_nsplit_n<T, false, false>(p, s, sms);
    if (!reverse) return dispatch_nsplit_n<T, false, true>(p, s, sms);
    if (!rst) return dispatch_nsplit_n<T, true, false>(p, s, sms);
    return dispatch_nsplit_n<T, true, true>(p, s, sms);
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
                   const float *D, const void *z, const float *dt_bias, int softplus, const float *h0,
                   const uint8_t *reset, int reverse, void *y, float *final_state, int64_t batch,
                   int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream, void *ckpt = nullptr,
                   size_t ckpt_bytes = 0)
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
                             {final_state, "final_state", false}, {h0, "h0", false},
                             {reset, "reset", false}, {ckpt, "workspace", false}};
    const bool extended = h0 || reset || reverse || ckpt;
    if (extended && N > 32)
        return fail(SS_ERR_N, "N=%lld: an initial state, sequence starts, the reverse direction or stored states "
                    "need N <= 32", (long long)N);
    if (ckpt) {
        if (reset || reverse)
            return fail(SS_ERR_DIM, "stored states for the backward pass are kept for the forward direction "
                        "without sequence starts only");
        const size_t need = bwd_workspace_bytes(batch, d_inner, L, N);
        if (ckpt_bytes < need)
            return fail(SS_ERR_DIM, "workspace of %zu bytes is smaller than the %zu bytes required", ckpt_bytes,
                        need);
        if (!aligned16(ckpt))
            return fail(SS_ERR_DIM, "workspace must be 16-byte aligned");
    }
    int dev = 0;
    ss_status st = check_ptrs(list, static_cast<int>(sizeof(list) / sizeof(list[0])), &dev);
    if (st != SS_OK)
        return st;

    ScanParams p{};
    p.h0 = h0;
    p.reset = reset;
    p.ckpt = static_cast<float4 *>(ckpt);
    p.nsub = (L + 15) / 16;
    p.x = x; p.dt = dt; p.B = B; p.C = C; p.z = z;
    p.A = A; p.D = D; p.dt_bias = dt_bias;
    p.y = y; p.final_state = final_state;
    p.batch = batch; p.d_inner = d_inner; p.L = L; p.N = N;
    p.softplus = softplus ? 1 : 0;
    p.vec = (L % 16 == 0) && aligned16(x) && aligned16(dt) && aligned16(y) && (!z || aligned16(z)) &&
            aligned16(B) && aligned16(C);
    p.tma = 0;

    p.nseg = 1;
    p.seg_len = L;
    if (extended || use_nsplit(N)) {
        if (p.vec && encode_scan_maps<T>(p))
            p.tma = 1;
        return dispatch_nsplit<T>(p, reverse != 0, stream, sm_count(dev));
    }
    const int lanes = pick_lanes(batch * d_inner, L, sm_count(dev));
    if (N <= 4)
        return dispatch_scan_lanes<T, 4>(p, lanes, stream);
    if (N <= 16)
        return dispatch_scan_lanes<T, 16>(p, lanes, stream);
    return dispatch_scan_lanes<T, 64>(p, lanes, stream);
}
