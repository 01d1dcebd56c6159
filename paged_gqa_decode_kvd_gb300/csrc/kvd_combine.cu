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

// One warp per (request, query head); lane l owns dims 4l..4l+3.  Split weights are
// computed 32 slots at a time, one per lane, and broadcast for the accumulation.
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
    const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= static_cast<int64_t>(p.B) * p.n_q) return;
    const int b = static_cast<int>(wid / p.n_q);
    const int h = static_cast<int>(wid % p.n_q);
    const int u = b * p.n_kv + h / p.g;
    const int hg = h % p.g;
    const int first = p.unit_first[u];
    const int cnt = p.unit_count[u];
    const float* lse_col = p.part_lse + hg;      // slot s: lse_col[s * g]

    float M = -INFINITY;
    for (int s = lane; s < cnt; s += 32) M = fmaxf(M, lse_col[static_cast<int64_t>(first + s) * p.g]);
    #pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse = -INFINITY;
    if (M != -INFINITY) {
        float Ls = 0.f;
        for (int s0 = 0; s0 < cnt; s0 += 32) {
            const int s = s0 + lane;
            float w = 0.f;
            if (s < cnt) {
                const float ls = lse_col[static_cast<int64_t>(first + s) * p.g];
                w = ls == -INFINITY ? 0.f : expf(ls - M);
            }
            Ls += w;
            const int n = min(32, cnt - s0);
            #pragma unroll 4
            for (int j = 0; j < n; ++j) {
                const float wj = __shfl_sync(kFull, w, j);
                const int64_t row = static_cast<int64_t>(first + s0 + j) * p.g + hg;
                const float4 v = reinterpret_cast<const float4*>(p.part_o + row * kDh)[lane];
                acc.x += wj * v.x;
                acc.y += wj * v.y;
                acc.z += wj * v.z;
                acc.w += wj * v.w;
            }
        }
        #pragma unroll
        for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(kFull, Ls, off);
        const float inv = 1.f / Ls;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        lse = M + logf(Ls);
    }
    const int64_t orow = static_cast<int64_t>(b) * p.n_q + h;
    if (p.out_f32) {
        reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * kDh)[lane] = acc;
    } else {
        uint2 v;
        v.x = pack_bf16(acc.x, acc.y);
        v.y = pack_bf16(acc.z, acc.w);
        reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + orow * kDh)[lane] = v;
    }
    if (p.lse_out && lane == 0) p.lse_out[orow] = lse;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    const int64_t threads = static_cast<int64_t>(p.B) * p.n_q * 32;
    const int blk = 256;
    combine_kernel<<<static_cast<unsigned>((threads + blk - 1) / blk), blk, 0, stream>>>(p);
    return cudaGetLastError();
}

// One thread per (request, position); heads are summed in order h = 0 .. n_q-1.
__global__ void __launch_bounds__(256) scores_kernel(const ScoreParams p) {
    const int b = blockIdx.y;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int len = p.seq_lens[b];
    if (t >= len || t >= p.logits_stride || t >= p.scores_stride) return;
    const float* lrow = p.logits + static_cast<int64_t>(b) * p.n_q * p.logits_stride + t;
    const float* lse = p.lse + static_cast<int64_t>(b) * p.n_q;
    float acc = 0.f;
    for (int h = 0; h < p.n_q; ++h) {
        const float m = lse[h];
        if (m == -INFINITY) continue;
        acc += expf(lrow[static_cast<int64_t>(h) * p.logits_stride] - m);
    }
    p.scores[static_cast<int64_t>(b) * p.scores_stride + t] += acc * p.inv_LH;
}

cudaError_t launch_scores(const ScoreParams& p, cudaStream_t stream) {
    const int blk = 256;
    const int64_t extent = p.logits_stride < p.scores_stride ? p.logits_stride : p.scores_stride;
    dim3 grid(static_cast<unsigned>((extent + blk - 1) / blk), p.B);
    scores_kernel<<<grid, blk, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kvd
