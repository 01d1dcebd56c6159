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
// One CTA per request.  Each block's importance becomes an order-preserving 32-bit key; a
// radix select (four 8-bit histogram passes over the unprotected blocks) finds the key T of
// the t1-th smallest.  Blocks with a smaller key go to the host tier, and of those whose key
// equals T the lowest-indexed ones fill the remaining places: the same set as sorting the
// unprotected blocks by (importance, index) and taking the first t1.  O(nb) per pass.
constexpr int kPlanThreads = 256;

__device__ __forceinline__ bool plan_protected(int j, int len, int protect_prompt, int protect_recent) {
    const int last = min(kBs * j + kBs - 1, len - 1);   // the block's last position
    return kBs * j < protect_prompt || last >= len - protect_recent;
}

// Unsigned key with the float order (−0 ranks with +0): flip every bit of a negative value,
// set the sign bit of a non-negative one.
__device__ __forceinline__ uint32_t order_key(float x) {
    const uint32_t u = __float_as_uint(x == 0.f ? 0.f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kPlanThreads) tier_plan_kernel(const TierPlanParams p) {
    extern __shared__ __align__(16) uint32_t key[];   // [max_blocks] keys, then [max_blocks] free flags
    uint8_t* is_free = reinterpret_cast<uint8_t*>(key + p.max_blocks);
    __shared__ uint32_t hist[256];
    __shared__ int scan[kPlanThreads];
    __shared__ uint32_t s_prefix, s_need;
    __shared__ int s_free;
    const int tid = threadIdx.x, lane = tid & 31;
    const int b = blockIdx.x;
    const int len = p.seq_lens[b];
    int nb = (len + kBs - 1) / kBs;
    if (len < 1 || nb > p.max_blocks) nb = 0;
    const float* srow = p.scores + static_cast<int64_t>(b) * p.scores_stride;
    int8_t* trow = p.tier + static_cast<int64_t>(b) * p.max_blocks;
    if (tid == 0) s_free = 0;
    __syncthreads();
    int my_free = 0;
    for (int j = tid; j < p.max_blocks; j += kPlanThreads) {
        float s = 0.f;
        uint8_t f = 0;
        if (j < nb) {
            for (int o = 0; o < kBs; ++o) {
                const int64_t pos = static_cast<int64_t>(kBs) * j + o;
                if (pos < len && pos < p.scores_stride) s += srow[pos];
            }
            f = plan_protected(j, len, p.protect_prompt, p.protect_recent) ? 0 : 1;
            key[j] = order_key(s);
            trow[j] = 0;
        } else {
            trow[j] = -1;
        }
        is_free[j] = f;
        my_free += f;
        if (p.importance) p.importance[static_cast<int64_t>(b) * p.max_blocks + j] = s;
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) my_free += __shfl_xor_sync(kFull, my_free, o);
    if (lane == 0 && my_free) atomicAdd(&s_free, my_free);
    __syncthreads();
    const int n_free = s_free;
    if (p.t1 == 0 || n_free == 0) return;
    if (p.t1 >= n_free) {   // every unprotected block goes
        for (int j = tid; j < nb; j += kPlanThreads)
            if (is_free[j]) trow[j] = 1;
        return;
    }

    // radix select of the t1-th smallest key among the unprotected blocks
    uint32_t prefix = 0, pmask = 0, need = static_cast<uint32_t>(p.t1);
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int d = tid; d < 256; d += kPlanThreads) hist[d] = 0;
        __syncthreads();
        for (int j0 = 0; j0 < nb; j0 += kPlanThreads) {   // same trip count in every lane: the match below
            const int j = j0 + tid;
            int d = 256;   // not a candidate
            if (j < nb && is_free[j] && (key[j] & pmask) == prefix) d = static_cast<int>((key[j] >> shift) & 255u);
            const unsigned peers = __match_any_sync(kFull, d);
            if (d < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[d], static_cast<uint32_t>(__popc(peers)));
        }
        __syncthreads();
        if (tid == 0) {
            uint32_t below = 0;
            int d = 0;
            for (; d < 255; ++d) {
                if (below + hist[d] >= need) break;
                below += hist[d];
            }
            s_prefix = prefix | (static_cast<uint32_t>(d) << shift);
            s_need = need - below;
        }
        __syncthreads();
        prefix = s_prefix;
        need = s_need;
        pmask |= 255u << shift;
    }

    // keys below T all go; of the keys equal to T, the `need` lowest-indexed blocks
    const uint32_t T = prefix;
    const int chunk = (nb + kPlanThreads - 1) / kPlanThreads;
    const int a = min(nb, tid * chunk), e = min(nb, a + chunk);
    int eq = 0;
    for (int j = a; j < e; ++j) eq += (is_free[j] && key[j] == T) ? 1 : 0;
    scan[tid] = eq;
    __syncthreads();
    for (int off = 1; off < kPlanThreads; off <<= 1) {   // inclusive scan over the threads' chunks
        const int v = tid >= off ? scan[tid - off] : 0;
        __syncthreads();
        scan[tid] += v;
        __syncthreads();
    }
    uint32_t before = static_cast<uint32_t>(scan[tid] - eq);
    for (int j = a; j < e; ++j) {
        if (!is_free[j]) continue;
        const uint32_t kj = key[j];
        if (kj < T) {
            trow[j] = 1;
        } else if (kj == T) {
            if (before < need) trow[j] = 1;
            ++before;
        }
    }
}

cudaError_t launch_tier_plan(const TierPlanParams& p, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(p.max_blocks) * (sizeof(uint32_t) + 1);
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(tier_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    tier_plan_kernel<<<p.B, kPlanThreads, smem, stream>>>(p);
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
