// rkv_free_blocks_push: FREE_BLOCKS on the device. The R-KV review page ("How
// R-KV decides what to drop") describes FREE_BLOCKS as handing evicted KV
// blocks back to the allocator instead of leaving them stranded; this kernel
// appends the block ids that one compression call freed (its CSR output) to a
// device-resident stack of free pool blocks, so that a decode loop can recycle
// them without a round trip to the host (and inside a captured CUDA graph).
#pragma once

#include "rkv_device.cuh"

namespace rkv {

constexpr int kPushThreads = 1024;

// One CTA: stack[top .. top + total) <- freed_ids[0 .. total), top += total,
// where total = freed_off[batch]. If the stack would overflow (or top or the
// offsets are invalid, or ids are missing for a non-empty list) nothing is
// written and the device error word is set.
__global__ void __launch_bounds__(kPushThreads)
    rkv_free_push_kernel(const int32_t *freed_off, const int32_t *freed_ids, int batch, int32_t *stack,
                         int32_t *top, int capacity)
{
    __shared__ int s_top, s_total, s_ok;
    pdl_wait();
    if (threadIdx.x == 0) {
        const int t = *top;
        const int total = freed_off[batch];
        const bool ok = t >= 0 && t <= capacity && total >= 0 && total <= capacity - t &&
                        (total == 0 || freed_ids != nullptr);
        s_top = t;
        s_total = total;
        s_ok = ok ? 1 : 0;
        if (!ok)
            record_error(kErrDevice);
    }
    __syncthreads();
    if (!s_ok)
        return;
    for (int i = threadIdx.x; i < s_total; i += kPushThreads)
        stack[s_top + i] = freed_ids[i];
    if (threadIdx.x == 0)
        *top = s_top + s_total;
}

} // namespace rkv
