// fault_probe.cuh -- a kernel whose only job is to let a bounded wait run out.
//
// Part of the single translation unit ss_scan.cu (included inside its
// anonymous namespace, in the forward-scan object); not compiled on its own.

#pragma once

// One thread waits on a barrier that nothing completes (no thread arrives on
// it and no copy is addressed to it): the bounded wait every kernel uses gives
// up after kWaitLimitNs, records kFaultWaitTimeout in this object's fault word
// and returns, leaving the context usable. The test of that mechanism.
__global__ void fault_probe_kernel()
{
    __shared__ __align__(8) unsigned long long probe_bar;
    const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(&probe_bar));
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
        (void)mbar_wait(bar, 0);   // phase 0 needs one arrival, and none comes
    }
}
