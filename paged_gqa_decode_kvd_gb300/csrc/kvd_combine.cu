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

// One CTA of W warps (W = blockDim.x/32 ≤ 16, chosen from the expected partials per unit)
// per (request, query head).  Warp w folds slots s ≡ w (mod W) in one online pass
// (running max, rescaled sum and accumulator; lane l owns dims 4l..4l+3), then warp 0
// merges the warps' states: a unit split 76 ways takes about one memory round trip with
// W = 16, while two or three partials need a single warp.  A unit whose output the decode
// kernel already wrote (count < 0) is skipped; a unit with no partial (count 0) gets
// out = 0 and lse = −inf.
constexpr int kCombineWarps = 16;

__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineParams p) {
    __shared__ float s_m[kCombineWarps];
    __shared__ float s_l[kCombineWarps];
    __shared__ float4 s_acc[kCombineWarps][32];
    const int bh = blockIdx.x;
    const int b = bh / p.n_q;
    const int h = bh % p.n_q;
    const int u = b * p.n_kv + h / p.g;
    const int hg = h % p.g;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
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

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    // about four partials per warp: expected partials per unit ≈ splits / units + 2
    const int expect = (p.slots_hint > 0 ? p.slots_hint : 1);
    int warps = 1;
    while (warps < kCombineWarps && warps * 4 < expect) warps <<= 1;
    combine_kernel<<<static_cast<unsigned>(p.B * p.n_q), warps * 32, 0, stream>>>(p);
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
