// kvd_measure.cu — read-only HBM stream, the second denominator of the decode roofline.
//
// The decode kernel only reads HBM (K/V records in, a few KB of results out), so its achieved
// bandwidth is compared with a copy (read + write) and with this pure read: every 16-byte word
// of a caller buffer read once through the L1-bypassing, evict-first load path, folded with
// xor so the loads cannot be dropped, one word per CTA written at the end.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvd.h"

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;   // independent 16-byte loads in flight per thread

__global__ void __launch_bounds__(kThreads) read_stream_kernel(const uint4* __restrict__ buf, uint64_t n16,
                                                               uint32_t* __restrict__ sink) {
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
    uint64_t i = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x;
    uint32_t acc = 0;
    for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
        uint4 v[kUnroll];
        #pragma unroll
        for (int j = 0; j < kUnroll; ++j) v[j] = __ldcs(buf + i + j * stride);
        #pragma unroll
        for (int j = 0; j < kUnroll; ++j) acc ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = __ldcs(buf + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    #pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, off);
    __shared__ uint32_t red[kThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t a = 0;
        for (int w = 0; w < kThreads / 32; ++w) a ^= red[w];
        sink[blockIdx.x] = a;
    }
}

}  // namespace

extern "C" kvd_status kvd_measure_read_stream(const void* buf, size_t bytes, void* sink, size_t sink_bytes,
                                              void* stream) {
    if (!buf || !sink || bytes == 0 || (bytes & 15u) || (reinterpret_cast<uintptr_t>(buf) & 15u) ||
        (reinterpret_cast<uintptr_t>(sink) & 3u))
        return KVD_ERR_INVALID;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, read_stream_kernel, kThreads, 0) != cudaSuccess) {
        cudaGetLastError();
        return KVD_ERR_CUDA;
    }
    const size_t grid = static_cast<size_t>(sms) * (per_sm > 0 ? per_sm : 1);
    if (sink_bytes < grid * sizeof(uint32_t)) return KVD_ERR_NOMEM;
    read_stream_kernel<<<static_cast<unsigned>(grid), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(buf), static_cast<uint64_t>(bytes / 16), static_cast<uint32_t*>(sink));
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}
