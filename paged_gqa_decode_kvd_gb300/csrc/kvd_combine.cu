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
// dims 4l..4l+3); with several warps, warp 0 then merges their states, handed over in `red`
// (red_bytes(nw) of shared memory; a single warp needs none).  A unit whose output the
// decode kernel already wrote (count < 0) is skipped; a unit with no partial (count 0) gets
// out = 0 and lse = −inf.
constexpr int kMaxWarps = 16;

__host__ __device__ constexpr int red_bytes(int nw) {
    return nw > 1 ? nw * 32 * static_cast<int>(sizeof(float4)) + 2 * nw * static_cast<int>(sizeof(float)) : 0;
}

extern __shared__ float4 dyn_smem[];

__device__ void combine_bh(const CombineParams& p, int bh, int nw, int warp, int lane, float4* red) {
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
    float M = m, L = l;
    float4 t = acc;
    if (nw > 1) {
        float* s_m = reinterpret_cast<float*>(red + nw * 32);
        float* s_l = s_m + nw;
        red[warp * 32 + lane] = acc;
        if (lane == 0) {
            s_m[warp] = m;
            s_l[warp] = l;
        }
        __syncthreads();
        if (warp != 0) return;
        M = -INFINITY;
        for (int w = 0; w < nw; ++w) M = fmaxf(M, s_m[w]);
        t = make_float4(0.f, 0.f, 0.f, 0.f);
        L = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < nw; ++w) {
                const float e = expf(s_m[w] - M);  // 0 for a warp that saw nothing
                const float4 v = red[w * 32 + lane];
                L += s_l[w] * e;
                t.x += v.x * e;
                t.y += v.y * e;
                t.z += v.z * e;
                t.w += v.w * e;
            }
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
// It signals its dependents once its own wait has returned: the next decode kernel is then
// scheduled while this merge runs.
__global__ void __launch_bounds__(kMaxWarps * 32) combine_kernel(const CombineParams p) {
    pdl_wait();
    pdl_trigger();
    combine_bh(p, blockIdx.x, blockDim.x >> 5, threadIdx.x >> 5, threadIdx.x & 31, dyn_smem);
}

static int combine_warps(int slots_hint) {
    // about four partials per warp: a unit split 76 ways takes about one memory round trip
    const int expect = slots_hint > 0 ? slots_hint : 1;
    int warps = 1;
    while (warps < kMaxWarps && warps * 4 < expect) warps <<= 1;
    return warps;
}

// Importance-score update of one position t of request b per thread (a CTA covers
// kScoreTile consecutive positions, so warp loads stay coalesced):
// scores[b][t] += inv_LH · Σ_h exp(logits[b][h][t] − lse[h]), heads in order h = 0..n_q-1.
// score_load starts, before the final LSEs are known, asynchronous 4-byte copies of this
// thread's logits of the first kPrefetchHeads heads into its own column of a shared tile
// (no registers held) and loads the running score; score_add waits for its own copies and
// finishes the sum.  The n_q final LSEs are staged in shared memory in the exp2 domain, so
// each term is one FFMA and one ex2.approx (relative error about 1e-6, well inside the
// 1e-5 score bound).
constexpr int kScoreThreads = 256;
constexpr int kScoreTile = kScoreThreads;
constexpr int kMaxHeads = 256;
constexpr int kPrefetchHeads = 32;
constexpr int kLseValues = 1024;   // partial LSEs a score CTA stages in shared memory
constexpr int kOffSlots = kMaxHeads + 4;   // value offsets per unit, padded to keep 16-byte alignment

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(float* dst, const float* src) {   // both 16-byte aligned
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

struct ScoreLane {
    float old;      // scores[b][t] before this update
    int64_t t;
    bool in_rows;   // t lies inside both row strides (every load is in bounds)
};

// xs: shared [kPrefetchHeads][kScoreThreads] floats, column j = position t0 + j (t0 a multiple
// of kScoreTile).  With a logits row stride that is a multiple of 4 floats and a 16-byte
// aligned buffer, the rows are copied in 16-byte chunks (a chunk never crosses the end of a
// row), a quarter of the copy instructions of 4-byte copies.  Every thread must then wait
// for its copies before a CTA barrier that precedes score_add.
__device__ __forceinline__ ScoreLane score_load(const ScoreParams& p, int b, int64_t t0, float* xs) {
    ScoreLane r;
    r.t = t0 + threadIdx.x;
    r.in_rows = r.t < p.logits_stride && r.t < p.scores_stride;
    const float* rows = p.logits + static_cast<int64_t>(b) * p.n_q * p.logits_stride;
    const int nh = p.n_q < kPrefetchHeads ? p.n_q : kPrefetchHeads;
    if ((p.logits_stride & 3) == 0 && (reinterpret_cast<uintptr_t>(p.logits) & 15u) == 0) {
        constexpr int kChunks = kScoreThreads / 4;
        for (int i = threadIdx.x; i < nh * kChunks; i += kScoreThreads) {
            const int h = i / kChunks, c = i % kChunks;
            const int64_t t = t0 + 4 * c;
            if (t < p.logits_stride)
                cp_async16(xs + h * kScoreThreads + 4 * c, rows + static_cast<int64_t>(h) * p.logits_stride + t);
        }
    } else if (r.in_rows) {
        for (int h = 0; h < nh; ++h)
            cp_async4(xs + h * kScoreThreads + threadIdx.x, rows + static_cast<int64_t>(h) * p.logits_stride + r.t);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    r.old = r.in_rows ? p.scores[static_cast<int64_t>(b) * p.scores_stride + r.t] : 0.f;
    return r;
}

__device__ __forceinline__ void score_add(const ScoreParams& p, const float* s_lse2, int b, const ScoreLane& r,
                                          const float* xs) {
    if (!r.in_rows || r.t >= p.seq_lens[b]) return;
    float acc = 0.f;
    const int nh = p.n_q < kPrefetchHeads ? p.n_q : kPrefetchHeads;
    #pragma unroll 4
    for (int h = 0; h < nh; ++h) {
        const float m2 = s_lse2[h];
        if (m2 != -INFINITY) acc += ex2(fmaf(xs[h * kScoreThreads + threadIdx.x], kLog2e, -m2));   // -inf: no retained position
    }
    const float* col = p.logits + static_cast<int64_t>(b) * p.n_q * p.logits_stride + r.t;
    #pragma unroll 4
    for (int h = kPrefetchHeads; h < p.n_q; ++h) {
        const float m2 = s_lse2[h];
        if (m2 != -INFINITY) acc += ex2(fmaf(col[static_cast<int64_t>(h) * p.logits_stride], kLog2e, -m2));
    }
    p.scores[static_cast<int64_t>(b) * p.scores_stride + r.t] = r.old + acc * p.inv_LH;
}

__global__ void __launch_bounds__(kScoreThreads) scores_kernel(const ScoreParams p) {
    __shared__ float s_lse2[kMaxHeads];
    __shared__ __align__(16) float xs[kPrefetchHeads * kScoreThreads];
    const int b = blockIdx.y;
    const ScoreLane r = score_load(p, b, static_cast<int64_t>(blockIdx.x) * kScoreTile, xs);
    for (int h = threadIdx.x; h < p.n_q; h += blockDim.x) {
        const float m = p.lse[static_cast<int64_t>(b) * p.n_q + h];
        s_lse2[h] = m == -INFINITY ? -INFINITY : m * kLog2e;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();   // every thread's copies and LSEs visible to all
    score_add(p, s_lse2, b, r, xs);
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
// Six CTAs an SM (at most 42 registers a thread): as many as the score CTAs' shared memory
// allows with up to 28 heads (about 37 KB each).
__global__ void __launch_bounds__(kScoreThreads, 6) epilogue_kernel(const CombineParams c, const ScoreParams sp,
                                                                  int tiles_per_req) {
    pdl_wait();
    pdl_trigger();
    const int bid = blockIdx.x;
    const int ncomb = c.B * c.n_q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (bid < ncomb) {
        combine_bh(c, bid, blockDim.x >> 5, warp, lane, dyn_smem);
        return;
    }
    // Score CTA.  Shared memory: the heads' final LSEs (exp2 domain), the request's unit
    // tables and value offsets, each head's unit, the values the LSEs need, then the logit
    // prefetch tile.
    const int nw = blockDim.x >> 5;
    const int nkv = c.n_kv, g = c.g;
    float* s_lse = reinterpret_cast<float*>(dyn_smem);          // kMaxHeads
    int* s_cnt = reinterpret_cast<int*>(s_lse + kMaxHeads);     // kMaxHeads
    int* s_first = s_cnt + kMaxHeads;                           // kMaxHeads
    int* s_off = s_first + kMaxHeads;                           // kOffSlots (≥ kMaxHeads + 1)
    float* vals = reinterpret_cast<float*>(s_off + kOffSlots);  // kLseValues (16-byte aligned)
    float* xs = vals + kLseValues;                              // min(n_q, kPrefetchHeads) rows
    uint8_t* s_unit = reinterpret_cast<uint8_t*>(xs + (c.n_q < kPrefetchHeads ? c.n_q : kPrefetchHeads) * kScoreThreads);
                                                                // kMaxHeads bytes: h / g (< 256)
    const int b = (bid - ncomb) / tiles_per_req;
    const int tile = (bid - ncomb) % tiles_per_req;
    // unit tables first: the prefetch below would queue ahead of them
    int cnt0 = 0, first0 = 0;
    if (threadIdx.x < nkv) {
        cnt0 = c.unit_count[b * nkv + threadIdx.x];
        first0 = c.unit_first[b * nkv + threadIdx.x];
    }
    const ScoreLane r = score_load(sp, b, static_cast<int64_t>(tile) * kScoreTile, xs);
    if (threadIdx.x < nkv) {
        s_cnt[threadIdx.x] = cnt0;
        s_first[threadIdx.x] = first0;
    }
    for (int k = kScoreThreads + threadIdx.x; k < nkv; k += kScoreThreads) {
        s_cnt[k] = c.unit_count[b * nkv + k];
        s_first[k] = c.unit_first[b * nkv + k];
    }
    for (int h = threadIdx.x; h < c.n_q; h += kScoreThreads) s_unit[h] = static_cast<uint8_t>(h / g);
    __syncthreads();
    if (threadIdx.x == 0) {   // unit k contributes g·count partial LSEs, or g finished LSEs (count < 0)
        int acc = 0;
        for (int k = 0; k < nkv; ++k) {
            s_off[k] = acc;
            const int cnt = s_cnt[k];
            acc += cnt > 0 ? g * cnt : (cnt < 0 ? g : 0);
        }
        s_off[nkv] = acc;
    }
    __syncthreads();
    const int total = s_off[nkv];
    // Final LSE of each head in the exp2 domain: LSE2 = M2 + log2 Σ_s 2^(lse_s·log2e − M2),
    // M2 = max_s lse_s·log2e (ex2/lg2.approx: about 1e-6, inside the score bound).
    auto head_lse2 = [&](int cnt, auto value) {   // value(s): natural-log LSE of partial s
        float M = -INFINITY;
        for (int s2 = lane; s2 < cnt; s2 += 32) M = fmaxf(M, value(s2));
        #pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
        if (M == -INFINITY) return -INFINITY;
        const float M2 = M * kLog2e;
        float L = 0.f;
        for (int s2 = lane; s2 < cnt; s2 += 32) {
            const float ls = value(s2);
            L += ls == -INFINITY ? 0.f : ex2(fmaf(ls, kLog2e, -M2));
        }
        #pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
        return M2 + lg2(L);
    };
    if (total <= kLseValues) {
        // Every value at once (independent loads, one memory round trip): a unit's partial
        // LSEs are slot-major with its g heads contiguous, so value j of unit k sits at
        // part_lse[first·g + j]; a unit the decode kernel finished reads lse_out.
        float v[kLseValues / kScoreThreads];
        #pragma unroll
        for (int m = 0; m < kLseValues / kScoreThreads; ++m) {
            const int i = threadIdx.x + m * kScoreThreads;
            v[m] = 0.f;
            if (i < total) {
                int lo = 0, hi = nkv - 1;   // the last unit with s_off[k] <= i
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_off[mid] <= i) lo = mid; else hi = mid - 1;
                }
                const int j = i - s_off[lo];
                v[m] = s_cnt[lo] < 0 ? c.lse_out[static_cast<int64_t>(b) * c.n_q + lo * g + j]
                                     : c.part_lse[static_cast<int64_t>(s_first[lo]) * g + j];
            }
        }
        #pragma unroll
        for (int m = 0; m < kLseValues / kScoreThreads; ++m) {
            const int i = threadIdx.x + m * kScoreThreads;
            if (i < total) vals[i] = v[m];
        }
        __syncthreads();
        for (int h = warp; h < c.n_q; h += nw) {
            const int k = s_unit[h], cnt = s_cnt[k];
            const float* hv = vals + s_off[k] + (h - k * g);   // value s of head h at hv[s·g]
            float lse2 = -INFINITY;
            if (cnt < 0) {
                lse2 = hv[0] == -INFINITY ? -INFINITY : hv[0] * kLog2e;
            } else if (cnt > 0) {
                lse2 = head_lse2(cnt, [&](int s2) { return hv[s2 * g]; });
            }
            if (lane == 0) s_lse[h] = lse2;
        }
    } else {
        // more values than the buffer holds: each warp walks its heads' partials in global memory
        for (int h = warp; h < c.n_q; h += nw) {
            const int k = s_unit[h], hg = h - k * g, cnt = s_cnt[k];
            float lse2 = -INFINITY;
            if (cnt < 0) {
                const float l = c.lse_out[static_cast<int64_t>(b) * c.n_q + h];
                lse2 = l == -INFINITY ? -INFINITY : l * kLog2e;
            } else if (cnt > 0) {
                const float* col = c.part_lse + static_cast<int64_t>(s_first[k]) * g + hg;
                lse2 = head_lse2(cnt, [&](int s2) { return col[static_cast<int64_t>(s2) * g]; });
            }
            if (lane == 0) s_lse[h] = lse2;
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();   // every thread's copies and the LSEs visible to all
    score_add(sp, s_lse, b, r, xs);
}

cudaError_t launch_combine(const CombineParams& p, int carveout, cudaStream_t stream) {
    const int w = combine_warps(p.slots_hint);
    return launch_dependent(combine_kernel, dim3(static_cast<unsigned>(p.B * p.n_q)), dim3(w * 32),
                            static_cast<size_t>(red_bytes(w)), carveout, stream, p);
}

cudaError_t launch_epilogue(const CombineParams& c, const ScoreParams& sp, int carveout, cudaStream_t stream) {
    const int64_t extent = sp.logits_stride < sp.scores_stride ? sp.logits_stride : sp.scores_stride;
    const int tiles = static_cast<int>((extent + kScoreTile - 1) / kScoreTile);
    const int64_t ctas = static_cast<int64_t>(c.B) * c.n_q + static_cast<int64_t>(c.B) * tiles;
    const int npre = sp.n_q < kPrefetchHeads ? sp.n_q : kPrefetchHeads;
    const int score_smem = (3 * kMaxHeads + kOffSlots) * 4 + kLseValues * 4 + npre * kScoreThreads * 4 + kMaxHeads;
    const int smem = red_bytes(kScoreThreads / 32) > score_smem ? red_bytes(kScoreThreads / 32) : score_smem;
    return launch_dependent(epilogue_kernel, dim3(static_cast<unsigned>(ctas)), dim3(kScoreThreads),
                            static_cast<size_t>(smem), carveout, stream, c, sp, tiles);
}

}  // namespace kvd
