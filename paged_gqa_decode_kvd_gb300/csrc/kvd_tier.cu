// kvd_tier.cu — the host tier's per-layer prefetch.
//
// Tier T1 keeps mid-importance tokens at full precision in host memory and brings them to the
// GPU before every attention step (page "기술 요약: 모든 사고가 HBM 을 필요로 하는 것은
// 아님", section "1. 4 단계 분류").  Before a layer's attention, that layer's host records
// are copied into an HBM staging slot, which the decode kernel then reads like any other
// block; the output is the same as with every block in HBM (section "3. 제로-근사오차
// 오프로딩", Prop. 1).
//
// The copy is a plain grid-stride loop of 16-byte loads from the host memory's device
// address and 16-byte stores to HBM, four loads in flight per thread to cover the host link's
// latency.
#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {

__global__ void __launch_bounds__(256) tier_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                       int64_t n16) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = src[i];
}

cudaError_t launch_tier_copy(const uint8_t* src, uint8_t* dst, size_t bytes, int num_sms, cudaStream_t stream) {
    const int64_t n16 = static_cast<int64_t>(bytes / 16);
    if (n16 == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (n16 + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    tier_copy_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(reinterpret_cast<const uint4*>(src),
                                                                           reinterpret_cast<uint4*>(dst), n16);
    return cudaGetLastError();
}

}  // namespace kvd
