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
// Low-bit pools (4-bit or 2-bit codes) store, per group of 128/ng values of a (token, KV
// head) row, a half-precision scale (span/(2^bits − 1)) and zero point (the group minimum), and
// the code of each value (page "The KV Cache Is the New Memory Wall", §4.2, Tab. 7).
//
// One warp per (token, KV head).  Lane l holds dims 4l..4l+3 (an 8-byte
// coalesced load) and scatters them to their fragment-order positions.  A slot in a
// host-tier block is written to that block's record in host memory.
#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {

// KIND: kKindBf16 / kKindFp8 (every block in the pool's one format), kKindMixed (each
// block's format read from the pool's per-block precision array; such a pool has no host tier
// and every record slot is sized for BF16) or kKindInt4 / kKindInt2 with NG groups per row (no
// host tier).
template <int KIND, int NG = 1>
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
    if (blk >= p.num_blocks + p.host_blocks) {
        if (lane == 0) report(p.err, KVD_ERR_OOB);
        return;
    }
    const int64_t row = (n * p.n_kv + h) * kDh;
    constexpr int kBits = KIND == kKindInt4 ? 4 : 2;
    constexpr int64_t kRec = KIND == kKindFp8 || KIND == kKindAngle ? kRecordFp8
                             : is_lowbit(KIND) ? lowbit_record_bytes(kBits, NG)
                                               : kRecordBf16;
    // a host-tier block (id ≥ num_blocks) keeps its record in host memory
    uint8_t* record = blk < p.num_blocks ? p.kv + (blk * p.n_kv + h) * kRec
                                         : p.host_kv + ((blk - p.num_blocks) * p.n_kv + h) * kRec;
    if constexpr (is_lowbit(KIND)) {
        write_token_lowbit<kBits, NG>(record, t, p.k_new + row, p.v_new + row, lane);
    } else if constexpr (KIND == kKindAngle) {
        write_token<kFmtE4m3, true>(record, t, p.k_new + row, p.v_new + row, lane);
    } else if constexpr (KIND == kKindMixed) {
        const int fmt = block_format(p.block_fmt[blk]);
        if (fmt == kFmtBf16) write_token<kFmtBf16>(record, t, p.k_new + row, p.v_new + row, lane);
        else if (fmt == kFmtE4m3) write_token<kFmtE4m3>(record, t, p.k_new + row, p.v_new + row, lane);
        else if (fmt == kFmtE5m2) write_token<kFmtE5m2>(record, t, p.k_new + row, p.v_new + row, lane);
        else if (lane == 0) report(p.err, KVD_ERR_OOB);   // not a precision code: the token is skipped
    } else {
        write_token<KIND == kKindFp8 ? kFmtE4m3 : kFmtBf16>(record, t, p.k_new + row, p.v_new + row, lane);
    }
}

cudaError_t launch_append(const AppendParams& p, int kind, cudaStream_t stream) {
    const int64_t warps = p.n_tokens * p.n_kv;
    const int threads = 256;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    const unsigned grid = static_cast<unsigned>(blocks);
    if (is_lowbit(kind)) {
        if (kind == kKindInt4) {
            if (p.ng == 4) append_kernel<kKindInt4, 4><<<grid, threads, 0, stream>>>(p);
            else if (p.ng == 2) append_kernel<kKindInt4, 2><<<grid, threads, 0, stream>>>(p);
            else append_kernel<kKindInt4, 1><<<grid, threads, 0, stream>>>(p);
        } else {
            if (p.ng == 4) append_kernel<kKindInt2, 4><<<grid, threads, 0, stream>>>(p);
            else if (p.ng == 2) append_kernel<kKindInt2, 2><<<grid, threads, 0, stream>>>(p);
            else append_kernel<kKindInt2, 1><<<grid, threads, 0, stream>>>(p);
        }
    } else if (kind == kKindAngle)
        append_kernel<kKindAngle><<<grid, threads, 0, stream>>>(p);
    else if (kind == kKindFp8)
        append_kernel<kKindFp8><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(p);
    else if (kind == kKindMixed)
        append_kernel<kKindMixed><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(p);
    else
        append_kernel<kKindBf16><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kvd
