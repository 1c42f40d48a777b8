// ss_scan.cu -- sm_103a kernels and C ABI of the selective scan (S6) library.
//
// What is computed is stated in include/ss_scan.h ("Mamba and selective state
// spaces": box "Selective state-space model (S6)", sections "The
// discretization the code actually uses", "The Mamba block", "Decoding with a
// constant-size cache", "Why the scan must be fused").
//
// One source, kept in parts:
//   device_common.cuh  device math, io conversion, f32x2 pairs, cp.async, mbarriers and tensor copies
//   host_common.cuh    error strings, pointer validation, device queries, tensor maps, stored-state layout
//   scan_fwd.cuh       forward scan (n-split and time-lane kernels)
//   scan_bwd.cuh       backward pass (states recomputed)
//   decode.cuh         single-token state update
//   conv.cuh           causal depthwise conv1d + SiLU and its decode step
//   ssd.cuh            Mamba-2's scalar-decay scan on the tensor cores
// followed here by the extern "C" entry points.
//
// The library is compiled as several objects from this one file, one per
// value of SS_PART (1 forward scan, 2 backward pass, 3 decode update and conv,
// 4 SSD, 0 the entry points every part shares), so that the parts build in
// parallel; with SS_PART undefined everything is compiled at once. Each
// object has its own device fault word; ss_device_faults reads them all.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cooperative_groups.h>

#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "ss_scan.h"

#ifndef SS_PART
#define SS_PART_IS(k) 1
#else
#define SS_PART_IS(k) (SS_PART == (k))
#endif

namespace cg = cooperative_groups;

namespace ssi {
// the message of the last non-OK status on this host thread (defined once, in part 0)
extern thread_local char g_err[512];
// each part's device fault word: read (and cleared when `clear`) into *flags
cudaError_t fault_word_fwd(unsigned int *flags, int clear);
cudaError_t fault_word_bwd(unsigned int *flags, int clear);
cudaError_t fault_word_dec(unsigned int *flags, int clear);
cudaError_t fault_word_ssd(unsigned int *flags, int clear);
}  // namespace ssi

namespace {

#include "device_common.cuh"
#include "host_common.cuh"
#if SS_PART_IS(1)
#include "scan_fwd.cuh"
#include "scan_fwd_host.cuh"
#include "fault_probe.cuh"
#endif
#if SS_PART_IS(2)
#include "scan_bwd.cuh"
#endif
#if SS_PART_IS(3)
#include "decode.cuh"
#include "conv.cuh"
#endif
#if SS_PART_IS(4)
#include "ssd.cuh"
#include "ssd_host.cuh"
#endif

// this object's device fault word, read (and cleared) from the host
[[maybe_unused]] cudaError_t read_fault_word(unsigned int *flags, int clear)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fault_flags, sizeof(v));
    if (e == cudaSuccess && clear) {
        const unsigned int none = 0;
        e = cudaMemcpyToSymbol(g_fault_flags, &none, sizeof(none));
    }
    *flags = v;
    return e;
}

}  // namespace

namespace ssi {
#if SS_PART_IS(0)
thread_local char g_err[512] = "";
#endif
#if SS_PART_IS(1)
cudaError_t fault_word_fwd(unsigned int *flags, int clear) { return read_fault_word(flags, clear); }
#endif
#if SS_PART_IS(2)
cudaError_t fault_word_bwd(unsigned int *flags, int clear) { return read_fault_word(flags, clear); }
#endif
#if SS_PART_IS(3)
cudaError_t fault_word_dec(unsigned int *flags, int clear) { return read_fault_word(flags, clear); }
#endif
#if SS_PART_IS(4)
cudaError_t fault_word_ssd(unsigned int *flags, int clear) { return read_fault_word(flags, clear); }
#endif
}  // namespace ssi

// ------------------------------------------------------------------ C ABI

extern "C" {

// ---- forward scan
#if SS_PART_IS(1)

ss_status ss_scan_fwd_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A, const ss_bf16 *B,
                           const ss_bf16 *C, const float *D, const ss_bf16 *z, const float *dt_bias,
                           int delta_softplus, ss_bf16 *y, float *final_state, int64_t batch,
                           int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream)
{
    return scan_fwd<__nv_bfloat16>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, nullptr, nullptr, 0, y,
                                   final_state, batch, d_inner, L, N, stream);
}

ss_status ss_scan_fwd_f32(const float *x, const float *delta, const float *A, const float *B,
                          const float *C, const float *D, const float *z, const float *dt_bias,
                          int delta_softplus, float *y, float *final_state, int64_t batch,
                          int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream)
{
    return scan_fwd<float>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, nullptr, nullptr, 0, y, final_state,
                           batch, d_inner, L, N, stream);
}

ss_status ss_scan_fwd_ex_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A, const ss_bf16 *B,
                              const ss_bf16 *C, const float *D, const ss_bf16 *z, const float *dt_bias,
                              int delta_softplus, const float *h0, const uint8_t *seq_start, int reverse,
                              ss_bf16 *y, float *final_state, int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                              cudaStream_t stream)
{
    return scan_fwd<__nv_bfloat16>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, seq_start, reverse, y,
                                   final_state, batch, d_inner, L, N, stream);
}

ss_status ss_scan_fwd_ex_f32(const float *x, const float *delta, const float *A, const float *B, const float *C,
                             const float *D, const float *z, const float *dt_bias, int delta_softplus,
                             const float *h0, const uint8_t *seq_start, int reverse, float *y, float *final_state,
                             int64_t batch, int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream)
{
    return scan_fwd<float>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, seq_start, reverse, y, final_state,
                           batch, d_inner, L, N, stream);
}

ss_status ss_scan_fwd_train_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A, const ss_bf16 *B,
                                 const ss_bf16 *C, const float *D, const ss_bf16 *z, const float *dt_bias,
                                 int delta_softplus, const float *h0, ss_bf16 *y, float *final_state, void *workspace,
                                 size_t workspace_bytes, int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                                 cudaStream_t stream)
{
    if (!workspace) {
        g_err[0] = '\0';
        return fail(SS_ERR_NULL, "required pointer workspace is NULL");
    }
    return scan_fwd<__nv_bfloat16>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, nullptr, 0, y, final_state,
                                   batch, d_inner, L, N, stream, workspace, workspace_bytes);
}

ss_status ss_scan_fwd_train_f32(const float *x, const float *delta, const float *A, const float *B, const float *C,
                                const float *D, const float *z, const float *dt_bias, int delta_softplus,
                                const float *h0, float *y, float *final_state, void *workspace, size_t workspace_bytes,
                                int64_t batch, int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream)
{
    if (!workspace) {
        g_err[0] = '\0';
        return fail(SS_ERR_NULL, "required pointer workspace is NULL");
    }
    return scan_fwd<float>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, nullptr, 0, y, final_state, batch,
                           d_inner, L, N, stream, workspace, workspace_bytes);
}

ss_status ss_kernel_binary_version(int *binary_version)
{
    g_err[0] = '\0';
    if (!binary_version)
        return fail(SS_ERR_NULL, "binary_version is NULL");
    cudaFuncAttributes a{};
    const cudaError_t e = cudaFuncGetAttributes(&a, scan_nsplit_kernel<__nv_bfloat16, 4, 4, false, false, true>);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SS_ERR_INTERNAL, "cudaFuncGetAttributes failed: %s", cudaGetErrorString(e));
    }
    *binary_version = a.binaryVersion;
    return SS_OK;
}

ss_status ss_fault_probe(cudaStream_t stream)
{
    g_err[0] = '\0';
    fault_probe_kernel<<<1, 32, 0, stream>>>();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SS_ERR_LAUNCH, "fault probe launch failed: %s", cudaGetErrorString(e));
    return SS_OK;
}

#endif

// ---- backward pass
#if SS_PART_IS(2)

size_t ss_scan_bwd_workspace_bytes(int64_t batch, int64_t d_inner, int64_t L, int64_t N)
{
    return bwd_workspace_bytes(batch, d_inner, L, N);
}

ss_status ss_scan_bwd_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A, const ss_bf16 *B,
                           const ss_bf16 *C, const float *D, const ss_bf16 *z, const float *dt_bias,
                           int delta_softplus, const float *h0, const ss_bf16 *dout, const float *dfinal_state,
                           ss_bf16 *dx, ss_bf16 *ddelta, float *dA, float *dB, float *dC, float *dD, ss_bf16 *dz,
                           float *ddt_bias, float *dh0, void *workspace, size_t workspace_bytes,
                           int states_from_forward, int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                           cudaStream_t stream)
{
    return scan_bwd<__nv_bfloat16>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, dout, dfinal_state, dx,
                                   ddelta, dA, dB, dC, dD, dz, ddt_bias, dh0, workspace, workspace_bytes, batch,
                                   d_inner, L, N, stream, states_from_forward);
}

ss_status ss_scan_bwd_f32(const float *x, const float *delta, const float *A, const float *B, const float *C,
                          const float *D, const float *z, const float *dt_bias, int delta_softplus, const float *h0,
                          const float *dout, const float *dfinal_state, float *dx, float *ddelta, float *dA,
                          float *dB, float *dC, float *dD, float *dz, float *ddt_bias, float *dh0, void *workspace,
                          size_t workspace_bytes, int states_from_forward, int64_t batch, int64_t d_inner, int64_t L,
                          int64_t N, cudaStream_t stream)
{
    return scan_bwd<float>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, dout, dfinal_state, dx, ddelta,
                           dA, dB, dC, dD, dz, ddt_bias, dh0, workspace, workspace_bytes, batch, d_inner, L, N,
                           stream, states_from_forward);
}

ss_status ss_scan_bwd_ex_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A, const ss_bf16 *B,
                              const ss_bf16 *C, const float *D, const ss_bf16 *z, const float *dt_bias,
                              int delta_softplus, const float *h0, const uint8_t *seq_start, int reverse,
                              const ss_bf16 *dout, const float *dfinal_state, ss_bf16 *dx, ss_bf16 *ddelta, float *dA,
                              float *dB, float *dC, float *dD, ss_bf16 *dz, float *ddt_bias, float *dh0,
                              void *workspace, size_t workspace_bytes, int64_t batch, int64_t d_inner, int64_t L,
                              int64_t N, cudaStream_t stream)
{
    return scan_bwd<__nv_bfloat16>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, dout, dfinal_state, dx,
                                   ddelta, dA, dB, dC, dD, dz, ddt_bias, dh0, workspace, workspace_bytes, batch,
                                   d_inner, L, N, stream, 0, seq_start, reverse);
}

ss_status ss_scan_bwd_ex_f32(const float *x, const float *delta, const float *A, const float *B, const float *C,
                             const float *D, const float *z, const float *dt_bias, int delta_softplus,
                             const float *h0, const uint8_t *seq_start, int reverse, const float *dout,
                             const float *dfinal_state, float *dx, float *ddelta, float *dA, float *dB, float *dC,
                             float *dD, float *dz, float *ddt_bias, float *dh0, void *workspace,
                             size_t workspace_bytes, int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                             cudaStream_t stream)
{
    return scan_bwd<float>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, dout, dfinal_state, dx, ddelta,
                           dA, dB, dC, dD, dz, ddt_bias, dh0, workspace, workspace_bytes, batch, d_inner, L, N,
                           stream, 0, seq_start, reverse);
}

ss_status ss_scan_bwd_noalloc_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A, const ss_bf16 *B,
                                   const ss_bf16 *C, const float *D, const ss_bf16 *z, const float *dt_bias,
                                   int delta_softplus, const float *h0, const ss_bf16 *dout,
                                   const float *dfinal_state, ss_bf16 *dx, ss_bf16 *ddelta, float *dA, float *dB,
                                   float *dC, float *dD, ss_bf16 *dz, float *ddt_bias, float *dh0, int64_t batch,
                                   int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream)
{
    return scan_bwd_noalloc<__nv_bfloat16>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, dout, dfinal_state,
                                           dx, ddelta, dA, dB, dC, dD, dz, ddt_bias, dh0, batch, d_inner, L, N,
                                           stream);
}

ss_status ss_scan_bwd_noalloc_f32(const float *x, const float *delta, const float *A, const float *B,
                                  const float *C, const float *D, const float *z, const float *dt_bias,
                                  int delta_softplus, const float *h0, const float *dout, const float *dfinal_state,
                                  float *dx, float *ddelta, float *dA, float *dB, float *dC, float *dD, float *dz,
                                  float *ddt_bias, float *dh0, int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                                  cudaStream_t stream)
{
    return scan_bwd_noalloc<float>(x, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, dout, dfinal_state, dx,
                                   ddelta, dA, dB, dC, dD, dz, ddt_bias, dh0, batch, d_inner, L, N, stream);
}

#endif

// ---- decode update and conv
#if SS_PART_IS(3)

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

ss_status ss_causal_conv1d_bf16(const ss_bf16 *x, const float *w, const float *bias, const ss_bf16 *state_in,
                                int silu, ss_bf16 *out, ss_bf16 *state_out, int64_t batch, int64_t d_inner,
                                int64_t L, int64_t k, cudaStream_t stream)
{
    return causal_conv1d<__nv_bfloat16>(x, w, bias, state_in, silu, out, state_out, batch, d_inner, L, k, stream);
}

ss_status ss_causal_conv1d_f32(const float *x, const float *w, const float *bias, const float *state_in, int silu,
                               float *out, float *state_out, int64_t batch, int64_t d_inner, int64_t L, int64_t k,
                               cudaStream_t stream)
{
    return causal_conv1d<float>(x, w, bias, state_in, silu, out, state_out, batch, d_inner, L, k, stream);
}

ss_status ss_conv_state_update_bf16(ss_bf16 *conv_state, const ss_bf16 *x, const float *w, const float *bias,
                                    int silu, ss_bf16 *out, int64_t batch, int64_t d_inner, int64_t k,
                                    cudaStream_t stream)
{
    return conv_state_update<__nv_bfloat16>(conv_state, x, w, bias, silu, out, batch, d_inner, k, stream);
}

ss_status ss_conv_state_update_f32(float *conv_state, const float *x, const float *w, const float *bias, int silu,
                                   float *out, int64_t batch, int64_t d_inner, int64_t k, cudaStream_t stream)
{
    return conv_state_update<float>(conv_state, x, w, bias, silu, out, batch, d_inner, k, stream);
}

#endif

// ---- SSD
#if SS_PART_IS(4)

size_t ss_ssd_workspace_bytes(int64_t batch, int64_t L, int64_t nheads, int64_t ngroups, int64_t N)
{
    return ssd_workspace_bytes(batch, L, nheads, ngroups, N);
}

ss_status ss_ssd_fwd_bf16(const ss_bf16 *x, const ss_bf16 *dt, const float *A, const ss_bf16 *B, const ss_bf16 *C,
                          const float *D, const ss_bf16 *z, const float *dt_bias, int delta_softplus,
                          const float *h0, ss_bf16 *y, float *final_state, void *workspace, size_t workspace_bytes,
                          int64_t batch, int64_t L, int64_t nheads, int64_t headdim, int64_t ngroups, int64_t N,
                          cudaStream_t stream)
{
    return ssd_fwd(x, dt, A, B, C, D, z, dt_bias, delta_softplus, h0, y, final_state, workspace, workspace_bytes,
                   batch, L, nheads, headdim, ngroups, N, stream);
}

#endif

// ---- shared by every part
#if SS_PART_IS(0)

ss_status ss_device_faults(unsigned int *flags, int clear)
{
    g_err[0] = '\0';
    if (!flags)
        return fail(SS_ERR_NULL, "flags is NULL");
    static_assert(SS_FAULT_WAIT_TIMEOUT == kFaultWaitTimeout && SS_FAULT_SMEM_ALIGN == kFaultSmemAlign,
                  "fault bits agree");
    cudaError_t (*const parts[])(unsigned int *, int) = {ssi::fault_word_fwd, ssi::fault_word_bwd,
                                                          ssi::fault_word_dec, ssi::fault_word_ssd};
    unsigned int v = 0;
    for (auto read : parts) {
        unsigned int w = 0;
        const cudaError_t e = read(&w, clear);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SS_ERR_INTERNAL, "reading the device fault word failed: %s", cudaGetErrorString(e));
        }
        v |= w;
    }
    *flags = v;
    return SS_OK;
}

const char *ss_last_error(void) { return g_err; }

int ss_abi_version(void) { return SS_ABI_VERSION; }

#endif

}  // extern "C"
