// Stream-ordered copy between device-reachable buffers by a kernel: device
// memory, and pinned host memory, which GB300's NVLink-C2C lets the SMs read
// and write in place.  Launched like the layer's kernels (programmatic
// dependent launch), so a host -> device copy, the layer and the device ->
// host copy of its output chain without copy-engine round trips between them.
// The pages have no counterpart: this is the plumbing of the end-to-end call.
#include "internal.cuh"

namespace qe {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy_kernel(const uint4 *__restrict__ src,
                                                            uint4 *__restrict__ dst,
                                                            long long n16)
{
    pdl_enter();
    for (long long i = (long long)blockIdx.x * kCopyThreads + threadIdx.x; i < n16;
         i += (long long)gridDim.x * kCopyThreads)
        dst[i] = src[i];
}

cudaError_t launch_copy(void *dst, const void *src, size_t bytes, int num_sms, cudaStream_t st)
{
    const long long n16 = (long long)(bytes / 16);
    long long blocks = (n16 + kCopyThreads - 1) / kCopyThreads;
    if (blocks > 2LL * num_sms)
        blocks = 2LL * num_sms;
    if (blocks < 1)
        blocks = 1;
    return launch_pdl(copy_kernel, dim3((unsigned)blocks), dim3(kCopyThreads), 0, st,
                      static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16);
}

}  // namespace qe
