// host_common.cuh -- host-side error reporting, pointer validation and device queries shared by every entry point.
//
// Part of the single translation unit ss_scan.cu (included inside its
// anonymous namespace); not compiled on its own.

#pragma once

// ------------------------------------------------------------------ host side

using ssi::g_err;   // one message buffer per host thread, shared by every part of the library

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

// ------------------------------------------------------------------ sequence segments

// Segments per channel group of a scan walk (the forward n-split kernel and
// the backward pass): when the channel groups fill less than half of the CTA
// slots of the GPU, the sequence is cut into up to 8 segments (one
// thread-block cluster per group) so that the grid fills one wave, keeping at
// least 4 chunks per segment. The environment variable env_name, when set to
// 1..8, overrides the choice.
int pick_segments(int64_t groups, int64_t L, int64_t lc, int64_t slots, const char *env_name)
{
    const char *env = getenv(env_name);
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

// ------------------------------------------------------------------ tensor maps (cuTensorMapEncodeTiled)

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

// the driver's tensor-map encoder, looked up once; null when unavailable
EncodeTiledFn encode_tiled_fn()
{
    static const EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            f = nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// map of a (batch, rows, L) tensor of T as three dimensions (L, rows, batch),
// box (box_t, box_rows, 1); elements outside the tensor read as zero
template <typename T>
bool encode_rows_map(CUtensorMap *m, const void *base, int64_t L, int64_t rows, int64_t batch, uint32_t box_t,
                     uint32_t box_rows)
{
    const EncodeTiledFn fn = encode_tiled_fn();
    if (!fn || !base)
        return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(batch)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(L) * sizeof(T),
                                   static_cast<cuuint64_t>(L) * static_cast<cuuint64_t>(rows) * sizeof(T)};
    const cuuint32_t box[3] = {box_t, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ the backward pass's stored states
//
// Shared by the backward pass and the training forward, which fills the same
// workspace layout.

constexpr int64_t kBwdHC = 16;   // steps per stored state (BwdShape::HC)

int64_t bwd_groups(int64_t N) { return N <= 4 ? 1 : (N <= 8 ? 2 : (N <= 16 ? 4 : 8)); }

// 0 for sizes the backward pass rejects: a size <= 0, N outside [1, 32], or an
// element count past the limits of scan_bwd (checked before any product is
// formed, so nothing here can overflow)
size_t bwd_workspace_bytes(int64_t batch, int64_t d_inner, int64_t L, int64_t N)
{
    if (batch <= 0 || d_inner <= 0 || L <= 0 || N < 1 || N > 32)
        return 0;
    if (batch > (int64_t(1) << 40) / d_inner || batch * d_inner > (int64_t(1) << 50) / L)
        return 0;
    const int64_t nsub = (L + kBwdHC - 1) / kBwdHC;
    return static_cast<size_t>(batch) * nsub * bwd_groups(N) * d_inner * 16;
}
