// host_common.cuh -- host-side error reporting, pointer validation and device queries shared by every entry point.
//
// Part of the single translation unit ss_scan.cu (included inside its
// anonymous namespace); not compiled on its own.

#pragma once

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
