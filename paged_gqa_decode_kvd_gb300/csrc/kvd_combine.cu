// kvd_combine.cu — split-KV log-sum-exp merge and the importance-score epilogue.
//
// Combine: a unit's context is cut into pieces, each reduced to (o_s, lse_s)
// with o_s normalised over its own positions.  The exact softmax over the union
// is LSE = log Σ_s exp(lse_s), out = Σ_s exp(lse_s − LSE)·o_s.
//
// Score epilogue: the cumulative importance score adds, per decode step, the
// attention weight of every position averaged over heads and layers,
//   s_i += (1/|L|) Σ_ℓ (1/H) Σ_h α_{ℓ,h}[i]
// (page "기술 요약: 모든 사고가 HBM 을 필요로 하는 것은 아님", section
// "2. 중요도 점수화").  One call adds one layer's term with weight 1/(L·H);
// α_h[i] = exp(l_h[i] − lse_h) from the logits and lse the decode kernel wrote.
#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {

// Merge of one (request, query head) by the nw warps of a CTA.  Warp w folds slots
// s ≡ w (mod nw) in one online pass (running max, rescaled sum and accumulator; lane l owns
// dims 4l..4l+3), then warp 0 merges the warps' states.  A unit whose output the decode
// kernel already wrote (count < 0) is skipped; a unit with no partial (count 0) gets
// out = 0 and lse = −inf.
constexpr int kMaxWarps = 16;

__device__ void combine_bh(const CombineParams& p, int bh, int nw, int warp, int lane) {
    __shared__ float s_m[kMaxWarps];
    __shared__ float s_l[kMaxWarps];
    __shared__ float4 s_acc[kMaxWarps][32];
    const int b = bh / p.n_q;
    const int h = bh % p.n_q;
    const int u = b * p.n_kv + h / p.g;
    const int hg = h % p.g;
    const int cnt = p.unit_count[u];
    if (cnt < 0) return;
    const int first = p.unit_first[u];

    float m = -INFINITY, l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    #pragma unroll 4
    for (int s = warp; s < cnt; s += nw) {
        const int64_t row = static_cast<int64_t>(first + s) * p.g + hg;
        const float ls = p.part_lse[row];
        const float4 v = reinterpret_cast<const float4*>(p.part_o + row * kDh)[lane];
        if (ls == -INFINITY) continue;
        const float mn = fmaxf(m, ls);
        const float a = expf(m - mn);          // 0 while m is -inf
        const float w = expf(ls - mn);
        l = l * a + w;
        acc.x = acc.x * a + w * v.x;
        acc.y = acc.y * a + w * v.y;
        acc.z = acc.z * a + w * v.z;
        acc.w = acc.w * a + w * v.w;
        m = mn;
    }
    s_acc[warp][lane] = acc;
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
    __syncthreads();
    if (warp != 0) return;
    float M = -INFINITY;
    for (int w = 0; w < nw; ++w) M = fmaxf(M, s_m[w]);
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
        for (int w = 0; w < nw; ++w) {
            const float e = expf(s_m[w] - M);  // 0 for a warp that saw nothing
            const float4 v = s_acc[w][lane];
            L += s_l[w] * e;
            t.x += v.x * e;
            t.y += v.y * e;
            t.z += v.z * e;
            t.w += v.w * e;
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    t.x *= inv;
    t.y *= inv;
    t.z *= inv;
    t.w *= inv;
    const int64_t orow = static_cast<int64_t>(b) * p.n_q + h;
    if (p.out_f32) {
        reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * kDh)[lane] = t;
    } else {
        uint2 v;
        v.x = pack_bf16(t.x, t.y);
        v.y = pack_bf16(t.z, t.w);
        reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + orow * kDh)[lane] = v;
    }
    if (p.lse_out && lane == 0) p.lse_out[orow] = L > 0.f ? M + logf(L) : -INFINITY;
}

// One CTA of W warps (W from the expected partials per unit) per (request, query head).
__global__ void __launch_bounds__(kMaxWarps * 32) combine_kernel(const CombineParams p) {
    pdl_wait();
    pdl_trigger();
    combine_bh(p, blockIdx.x, blockDim.x >> 5, threadIdx.x >> 5, threadIdx.x & 31);
}

static int combine_warps(int slots_hint) {
    // about four partials per warp: a unit split 76 ways takes about one memory round trip
    const int expect = slots_hint > 0 ? slots_hint : 1;
    int warps = 1;
    while (warps < kMaxWarps && warps * 4 < expect) warps <<= 1;
    return warps;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    return launch_dependent(combine_kernel, dim3(static_cast<unsigned>(p.B * p.n_q)),
                            dim3(combine_warps(p.slots_hint) * 32), 0, stream, p);
}

// Importance-score update of a tile of kScorePos·blockDim.x positions of request b, each
// thread taking kScorePos positions blockDim.x apart (warp loads stay coalesced):
// scores[b][t] += inv_LH · Σ_h exp(logits[b][h][t] − lse[h]), heads in order h = 0..n_q-1.
// The n_q final LSEs are staged in shared memory in the exp2 domain, so each term is one
// FFMA and one ex2.approx (relative error about 1e-6, well inside the 1e-5 score bound).
constexpr int kScoreThreads = 256;
constexpr int kScorePos = 1;
constexpr int kScoreTile = kScoreThreads * kScorePos;
constexpr int kMaxHeads = 256;

__device__ void scores_tile(const ScoreParams& p, const float* s_lse2, int b, int t0) {
    const int len = p.seq_lens[b];
    int64_t lim = p.logits_stride < p.scores_stride ? p.logits_stride : p.scores_stride;
    if (len < lim) lim = len;
    const float* lrow = p.logits + static_cast<int64_t>(b) * p.n_q * p.logits_stride;
    float acc[kScorePos];
    int tt[kScorePos];
    #pragma unroll
    for (int k = 0; k < kScorePos; ++k) {
        acc[k] = 0.f;
        tt[k] = t0 + threadIdx.x + k * kScoreThreads;
    }
    if (tt[0] >= lim) return;
    #pragma unroll 4
    for (int h = 0; h < p.n_q; ++h) {
        const float m2 = s_lse2[h];
        if (m2 == -INFINITY) continue;                 // head with no retained position
        const float* hrow = lrow + static_cast<int64_t>(h) * p.logits_stride;
        #pragma unroll
        for (int k = 0; k < kScorePos; ++k)
            if (tt[k] < lim) acc[k] += ex2(fmaf(hrow[tt[k]], kLog2e, -m2));
    }
    #pragma unroll
    for (int k = 0; k < kScorePos; ++k)
        if (tt[k] < lim) p.scores[static_cast<int64_t>(b) * p.scores_stride + tt[k]] += acc[k] * p.inv_LH;
}

__global__ void __launch_bounds__(kScoreThreads) scores_kernel(const ScoreParams p) {
    __shared__ float s_lse2[kMaxHeads];
    const int b = blockIdx.y;
    for (int h = threadIdx.x; h < p.n_q; h += blockDim.x) {
        const float m = p.lse[static_cast<int64_t>(b) * p.n_q + h];
        s_lse2[h] = m == -INFINITY ? -INFINITY : m * kLog2e;
    }
    __syncthreads();
    scores_tile(p, s_lse2, b, blockIdx.x * kScoreTile);
}

cudaError_t launch_scores(const ScoreParams& p, cudaStream_t stream) {
    const int64_t extent = p.logits_stride < p.scores_stride ? p.logits_stride : p.scores_stride;
    dim3 grid(static_cast<unsigned>((extent + kScoreTile - 1) / kScoreTile), p.B);
    scores_kernel<<<grid, kScoreThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

// Split merge and score update of one layer in one launch.  CTAs [0, B·n_q) merge one
// (request, head) each; the rest each update a tile of positions of one request.  A score
// CTA derives the final LSE of every head of its request from the split partials itself
// (the merge CTAs of the same launch write lse_out concurrently), or reads lse_out where
// the decode kernel already finished the unit.
__global__ void __launch_bounds__(kScoreThreads) epilogue_kernel(const CombineParams c, const ScoreParams sp,
                                                                  int tiles_per_req) {
    pdl_wait();
    pdl_trigger();
    const int bid = blockIdx.x;
    const int ncomb = c.B * c.n_q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (bid < ncomb) {
        combine_bh(c, bid, blockDim.x >> 5, warp, lane);
        return;
    }
    __shared__ float s_lse[kMaxHeads];
    const int b = (bid - ncomb) / tiles_per_req;
    const int tile = (bid - ncomb) % tiles_per_req;
    for (int h = warp; h < c.n_q; h += blockDim.x >> 5) {
        const int u = b * c.n_kv + h / c.g, hg = h % c.g;
        const int cnt = c.unit_count[u];
        float lse = -INFINITY;
        if (cnt < 0) {
            lse = c.lse_out[static_cast<int64_t>(b) * c.n_q + h];
        } else if (cnt > 0) {
            const int first = c.unit_first[u];
            float M = -INFINITY;
            for (int s = lane; s < cnt; s += 32) M = fmaxf(M, c.part_lse[static_cast<int64_t>(first + s) * c.g + hg]);
            #pragma unroll
            for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
            float L = 0.f;
            if (M != -INFINITY)
                for (int s = lane; s < cnt; s += 32) {
                    const float ls = c.part_lse[static_cast<int64_t>(first + s) * c.g + hg];
                    L += ls == -INFINITY ? 0.f : expf(ls - M);
                }
            #pragma unroll
            for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
            lse = L > 0.f ? M + logf(L) : -INFINITY;
        }
        if (lane == 0) s_lse[h] = lse == -INFINITY ? -INFINITY : lse * kLog2e;
    }
    __syncthreads();
    scores_tile(sp, s_lse, b, tile * kScoreTile);
}

cudaError_t launch_epilogue(const CombineParams& c, const ScoreParams& sp, cudaStream_t stream) {
    const int64_t extent = sp.logits_stride < sp.scores_stride ? sp.logits_stride : sp.scores_stride;
    const int tiles = static_cast<int>((extent + kScoreTile - 1) / kScoreTile);
    const int64_t ctas = static_cast<int64_t>(c.B) * c.n_q + static_cast<int64_t>(c.B) * tiles;
    return launch_dependent(epilogue_kernel, dim3(static_cast<unsigned>(ctas)), dim3(kScoreThreads), 0, stream, c, sp,
                            tiles);
}

}  // namespace kvd
