// kvd_tier.cu — the host tier's block plan and block moves.
//
// Tier T1 keeps mid-importance tokens at full precision in host memory and brings them to the
// GPU before every attention step (page "기술 요약: 모든 사고가 HBM 을 필요로 하는 것은
// 아님", section "1. 4 단계 분류").  Before a layer's attention, that layer's host records
// are copied into an HBM staging slot (a copy-engine DMA issued by the C ABI), which the
// decode kernel then reads like any other block; the output is the same as with every block
// in HBM (section "3. 제로-근사오차 오프로딩", Prop. 1).
//
// Every Δ steps the tier plan ranks each request's blocks by importance (section "4. 시스템
// 구현"), and the block move copies records between the tiers once the caller has picked
// new homes for them.
#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {

// ---------------------------------------------------------------- tier plan
// One CTA per request.  Block importances go to shared memory; a block's rank among the
// unprotected blocks is the count of unprotected blocks with a smaller (importance, index),
// and the t1 blocks of rank < t1 go to the host tier.  O(nb²) per request, run once per Δ
// steps.
__device__ __forceinline__ bool plan_protected(int j, int len, int protect_prompt, int protect_recent) {
    const int last = min(kBs * j + kBs - 1, len - 1);   // the block's last position
    return kBs * j < protect_prompt || last >= len - protect_recent;
}

__global__ void __launch_bounds__(256) tier_plan_kernel(const TierPlanParams p) {
    extern __shared__ float imp[];   // [max_blocks]
    const int b = blockIdx.x;
    const int len = p.seq_lens[b];
    int nb = (len + kBs - 1) / kBs;
    if (len < 1 || nb > p.max_blocks) nb = 0;
    const float* srow = p.scores + static_cast<int64_t>(b) * p.scores_stride;
    int8_t* trow = p.tier + static_cast<int64_t>(b) * p.max_blocks;
    for (int j = threadIdx.x; j < p.max_blocks; j += blockDim.x) {
        float s = 0.f;
        if (j < nb) {
            for (int o = 0; o < kBs; ++o) {
                const int64_t pos = static_cast<int64_t>(kBs) * j + o;
                if (pos < len && pos < p.scores_stride) s += srow[pos];
            }
            imp[j] = s;
        } else {
            trow[j] = -1;
        }
        if (p.importance) p.importance[static_cast<int64_t>(b) * p.max_blocks + j] = s;
    }
    __syncthreads();
    for (int j = threadIdx.x; j < nb; j += blockDim.x) {
        if (plan_protected(j, len, p.protect_prompt, p.protect_recent)) {
            trow[j] = 0;
            continue;
        }
        const float x = imp[j];
        int rank = 0;
        for (int i = 0; i < nb && rank < p.t1; ++i)
            if (!plan_protected(i, len, p.protect_prompt, p.protect_recent) && (imp[i] < x || (imp[i] == x && i < j)))
                ++rank;
        trow[j] = rank < p.t1 ? 1 : 0;
    }
}

cudaError_t launch_tier_plan(const TierPlanParams& p, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(p.max_blocks) * sizeof(float);
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(tier_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    tier_plan_kernel<<<p.B, 256, smem, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- block moves
// Grid-stride over 16-byte chunks of every (pair, layer, head) record.
__global__ void __launch_bounds__(256) tier_move_kernel(const TierMoveParams p) {
    const int64_t per_rec = p.record_bytes / 16;
    const int64_t recs = static_cast<int64_t>(p.n) * p.L * p.n_kv;
    const int64_t total = recs * per_rec;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t r = i / per_rec, c = i % per_rec;
        const int pair = static_cast<int>(r / (static_cast<int64_t>(p.L) * p.n_kv));
        const int layer = static_cast<int>((r / p.n_kv) % p.L);
        const int h = static_cast<int>(r % p.n_kv);
        const int64_t from = p.from_ids[pair], to = p.to_ids[pair];
        const int64_t lim = p.num_blocks + p.host_blocks;
        if (from < 0 || from >= lim || to < 0 || to >= lim) {
            if (c == 0 && layer == 0 && h == 0) report(p.err, KVD_ERR_OOB);
            continue;
        }
        auto rec = [&](int64_t id) -> uint8_t* {
            return id < p.num_blocks
                       ? p.kv + ((static_cast<int64_t>(layer) * p.num_blocks + id) * p.n_kv + h) * p.record_bytes
                       : p.host_kv + ((static_cast<int64_t>(layer) * p.host_blocks + (id - p.num_blocks)) * p.n_kv + h) *
                                         p.record_bytes;
        };
        reinterpret_cast<uint4*>(rec(to))[c] = reinterpret_cast<const uint4*>(rec(from))[c];
    }
}

cudaError_t launch_tier_move(const TierMoveParams& p, int num_sms, cudaStream_t stream) {
    const int64_t total = static_cast<int64_t>(p.n) * p.L * p.n_kv * (p.record_bytes / 16);
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    tier_move_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kvd
