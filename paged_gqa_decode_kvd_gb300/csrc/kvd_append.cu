// kvd_append.cu — decode-step append ("reshape and cache") into the paged pool.
//
// Each decode step writes the new token's K and V at the end of the request's
// cache before attention runs (page "LLM에서 KV 캐시는 얼마나 생길까",
// section "KV 캐시란": prefill stores every prompt token's K·V, decode appends
// one token's K·V per step).  FP8 mode stores x / scale as E4M3 and keeps the
// scale to multiply back on read (same page, section "KV 캐시를 줄이는 기법");
// the scale is one fp32 value per (token, KV head), separately for K and V:
// scale = absmax/448, or 1 for an all-zero row.
//
// One warp per (token, KV head).  Lane l holds dims 4l..4l+3 (an 8-byte
// coalesced load) and scatters them to their fragment-order positions.
#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {

template <bool FP8>
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
    const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t n = warp_global / p.n_kv;
    const int h = static_cast<int>(warp_global % p.n_kv);
    if (n >= p.n_tokens) return;
    const int64_t slot = p.slot_mapping[n];
    if (slot < 0) return;
    const int64_t blk = slot / kBs;
    const int t = static_cast<int>(slot % kBs);
    if (blk >= p.num_blocks) {
        if (lane == 0) report(p.err, KVD_ERR_OOB);
        return;
    }
    const int64_t row = (n * p.n_kv + h) * kDh + lane * 4;
    const uint2 kraw = *reinterpret_cast<const uint2*>(p.k_new + row);
    const uint2 vraw = *reinterpret_cast<const uint2*>(p.v_new + row);
    const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(&kraw);
    const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(&vraw);
    const int64_t rec = (blk * p.n_kv + h);

    if constexpr (!FP8) {
        __nv_bfloat16* ktile = reinterpret_cast<__nv_bfloat16*>(p.kv + rec * kRecordBf16);
        __nv_bfloat16* vtile = ktile + kBs * kDh;
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = lane * 4 + j;
            int fl, fe;
            int i = k_frag_i(t, d, &fl, &fe);
            ktile[bf16_tile_index(i, fl, fe)] = kb[j];
            i = v_frag_i(t, d, &fl, &fe);
            vtile[bf16_tile_index(i, fl, fe)] = vb[j];
        }
    } else {
        float kx[4], vx[4];
        float kmax = 0.f, vmax = 0.f;
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            kx[j] = __bfloat162float(kb[j]);
            vx[j] = __bfloat162float(vb[j]);
            kmax = fmaxf(kmax, fabsf(kx[j]));
            vmax = fmaxf(vmax, fabsf(vx[j]));
        }
        #pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            kmax = fmaxf(kmax, __shfl_xor_sync(kFull, kmax, o));
            vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, o));
        }
        const float ks = (kmax == 0.f) ? 1.f : __fdiv_rn(kmax, 448.f);
        const float vs = (vmax == 0.f) ? 1.f : __fdiv_rn(vmax, 448.f);
        uint8_t* ktile = p.kv + rec * kRecordFp8;
        uint8_t* vtile = ktile + kTileFp8;
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = lane * 4 + j;
            const uint8_t kc = __nv_cvt_float_to_fp8(__fdiv_rn(kx[j], ks), __NV_SATFINITE, __NV_E4M3);
            const uint8_t vc = __nv_cvt_float_to_fp8(__fdiv_rn(vx[j], vs), __NV_SATFINITE, __NV_E4M3);
            int fl, fe;
            int i = k_frag_i(t, d, &fl, &fe);
            ktile[fp8_tile_index(i, fl, fe)] = kc;
            i = v_frag_i(t, d, &fl, &fe);
            vtile[fp8_tile_index(i, fl, fe)] = vc;
        }
        if (lane == 0) {
            float* sc = reinterpret_cast<float*>(ktile + 2 * kTileFp8);
            sc[t] = ks;
            sc[kBs + t] = vs;
        }
    }
}

cudaError_t launch_append(const AppendParams& p, bool fp8, cudaStream_t stream) {
    const int64_t warps = p.n_tokens * p.n_kv;
    const int threads = 256;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    if (fp8)
        append_kernel<true><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(p);
    else
        append_kernel<false><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kvd
