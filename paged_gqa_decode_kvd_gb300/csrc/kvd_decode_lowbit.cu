// kvd_decode_lowbit.cu — the decode kernel (kvd_decode_kernel.cuh) for low-bit pools: 4-bit or
// 2-bit codes with a half-precision scale and zero point per group of 32, 64 or 128 values of a
// (token, KV head) row (page "The KV Cache Is the New Memory Wall", §4.2 and Tab. 7: INT4 and
// 2-bit KV; §3.2: 2-bit storage lifts decode to 2g/w_kv = 64 FLOP per byte at g = 8).
#include "kvd_decode_kernel.cuh"

namespace kvd {

// Ring depth: a 4-bit record is 2,176..2,560 bytes and a 2-bit one 1,152..1,536, so a stage of
// either keeps far fewer bytes in flight than an 8 KB BF16 stage; 16 (4-bit) and 24 (2-bit)
// stages give three CTAs an SM about 100 KB in flight, as the BF16 ring does.
template <int KIND>
constexpr int lowbit_stages() { return KIND == kKindInt4 ? 16 : 24; }

template <int KIND>
static size_t smem_bytes_ng(int ng, int batch, int g) {
    constexpr int S = lowbit_stages<KIND>();
    return ng == 4 ? smem_layout<KIND, S, 4>(batch, g).total
           : ng == 2 ? smem_layout<KIND, S, 2>(batch, g).total
                     : smem_layout<KIND, S, 1>(batch, g).total;
}

template <int KIND>
static int ctas_ng(int ng, int batch, int g) {
    constexpr int S = lowbit_stages<KIND>();
    return ng == 4 ? ctas_per_sm_impl<KIND, S, 4>(batch, g)
           : ng == 2 ? ctas_per_sm_impl<KIND, S, 2>(batch, g)
                     : ctas_per_sm_impl<KIND, S, 1>(batch, g);
}

template <int KIND>
static cudaError_t launch_ng(const DecodeParams& p, int carveout, cudaStream_t stream) {
    constexpr int S = lowbit_stages<KIND>();
    return p.ng == 4 ? launch_variant<KIND, S, false, 4>(p, carveout, stream)
           : p.ng == 2 ? launch_variant<KIND, S, false, 2>(p, carveout, stream)
                       : launch_variant<KIND, S, false, 1>(p, carveout, stream);
}

size_t decode_smem_bytes_lowbit(int kind, int ng, int batch, int g) {
    return kind == kKindInt4 ? smem_bytes_ng<kKindInt4>(ng, batch, g) : smem_bytes_ng<kKindInt2>(ng, batch, g);
}

int decode_ctas_per_sm_lowbit(int kind, int ng, int batch, int g) {
    return kind == kKindInt4 ? ctas_ng<kKindInt4>(ng, batch, g) : ctas_ng<kKindInt2>(ng, batch, g);
}

cudaError_t launch_decode_lowbit(const DecodeParams& p, int kind, int carveout, cudaStream_t stream) {
    return kind == kKindInt4 ? launch_ng<kKindInt4>(p, carveout, stream) : launch_ng<kKindInt2>(p, carveout, stream);
}

}  // namespace kvd
