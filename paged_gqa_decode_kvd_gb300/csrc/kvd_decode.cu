// kvd_decode.cu — paged GQA decode attention for BF16, FP8-E4M3, mixed-precision and
// angle-domain pools:
// launch geometry and dispatch of the decode kernel (kvd_decode_kernel.cuh), and the self-test
// of its bounded waits.
#include "kvd_decode_kernel.cuh"

namespace kvd {


// Mixed pools: 12 stages of 8 KB record slots, two CTAs an SM (the kernel holds a bf16 and an
// f16 copy of q, 168 registers); an 8-bit block fills only half a stage.
constexpr int kMixedStages = 12;

// Ring depth of a call.  BF16: 8 stages (8 KB records).  FP8: 16 stages when three
// such CTAs fit an SM (the per-request arrays are small enough), else 8 stages (4 CTAs/SM).
// With 16 the CTA keeps twice the bytes in flight; measured on GB300 it is 1% faster for one
// or eight long requests and equal for 32 requests of 8,192 tokens.  The 16-stage variant runs
// three CTAs per SM anyway, so its launch bounds let it use 128 registers (the 8-stage one,
// four per SM, gets 96); without spills it is another 1% faster on one long request.  Angle-domain
// pools have FP8 records and follow the same rule.
static int decode_stages(int kind, int batch, int g) {
    if (kind != kKindFp8 && kind != kKindAngle) return 8;
    int per_sm = 0, reserved = 0;
    if (!smem_attrs(&per_sm, &reserved)) return 8;
    const int64_t need = 3 * (static_cast<int64_t>(smem_layout<kKindFp8, 16>(batch, g).total) + reserved);
    return need <= per_sm ? 16 : 8;
}

size_t decode_smem_bytes(int kind, int ng, int batch, int g) {
    if (is_lowbit(kind)) return decode_smem_bytes_lowbit(kind, ng, batch, g);
    if (kind == kKindBf16) return smem_layout<kKindBf16, 8>(batch, g).total;
    if (kind == kKindMixed) return smem_layout<kKindMixed, kMixedStages>(batch, g).total;
    if (kind == kKindAngle)
        return decode_stages(kind, batch, g) == 16 ? smem_layout<kKindAngle, 16>(batch, g).total
                                                   : smem_layout<kKindAngle, 8>(batch, g).total;
    return decode_stages(kind, batch, g) == 16 ? smem_layout<kKindFp8, 16>(batch, g).total
                                               : smem_layout<kKindFp8, 8>(batch, g).total;
}

int decode_ctas_per_sm(int kind, int ng, int batch, int g) {
    if (is_lowbit(kind)) return decode_ctas_per_sm_lowbit(kind, ng, batch, g);
    if (kind == kKindBf16) return ctas_per_sm_impl<kKindBf16, 8>(batch, g);
    if (kind == kKindMixed) return ctas_per_sm_impl<kKindMixed, kMixedStages>(batch, g);
    if (kind == kKindAngle)
        return decode_stages(kind, batch, g) == 16 ? ctas_per_sm_impl<kKindAngle, 16>(batch, g)
                                                   : ctas_per_sm_impl<kKindAngle, 8>(batch, g);
    return decode_stages(kind, batch, g) == 16 ? ctas_per_sm_impl<kKindFp8, 16>(batch, g)
                                               : ctas_per_sm_impl<kKindFp8, 8>(batch, g);
}

// Shared-memory carveout (percent of the SM's shared memory) that holds a full complement
// of decode CTAs, each with the per-block reservation; -1 if the device cannot be queried.
int decode_carveout(int kind, int ng, int batch, int g) {
    int per_sm = 0, reserved = 0;
    if (!smem_attrs(&per_sm, &reserved)) return -1;
    const int64_t need = static_cast<int64_t>(decode_ctas_per_sm(kind, ng, batch, g)) *
                         (static_cast<int64_t>(decode_smem_bytes(kind, ng, batch, g)) + reserved);
    const int64_t pct = (100 * need + per_sm - 1) / per_sm;
    return static_cast<int>(pct > 100 ? 100 : pct);
}

template <bool DIRECT>
static cudaError_t launch_decode_impl(const DecodeParams& p, int kind, int carveout, cudaStream_t stream) {
    if (kind == kKindBf16) return launch_variant<kKindBf16, 8, DIRECT>(p, carveout, stream);
    return decode_stages(kind, p.B, p.g) == 16 ? launch_variant<kKindFp8, 16, DIRECT>(p, carveout, stream)
                                               : launch_variant<kKindFp8, 8, DIRECT>(p, carveout, stream);
}

cudaError_t launch_decode(const DecodeParams& p, int kind, int carveout, cudaStream_t stream) {
    if (is_lowbit(kind)) return launch_decode_lowbit(p, kind, carveout, stream);   // no host tier
    if (kind == kKindAngle)   // no host tier
        return decode_stages(kind, p.B, p.g) == 16 ? launch_variant<kKindAngle, 16, false>(p, carveout, stream)
                                                   : launch_variant<kKindAngle, 8, false>(p, carveout, stream);
    // a mixed pool has no host tier
    if (kind == kKindMixed) return launch_variant<kKindMixed, kMixedStages, false>(p, carveout, stream);
    return p.host_direct && p.host_blocks > 0 ? launch_decode_impl<true>(p, kind, carveout, stream)
                                              : launch_decode_impl<false>(p, kind, carveout, stream);
}

// ---------------------------------------------------------------- step plan
// One warp per decode CTA of the step: the prefix sums of blocks per request exactly as the
// decode kernel forms them, and this CTA's first batch of (physical block, block word) pairs.
// It never signals its dependents early, so a decode launched right after it sees the plan.
__global__ void __launch_bounds__(32) plan_kernel(const DecodeParams p, int32_t* plan) {
    extern __shared__ int plan_pref[];
    const int lane = threadIdx.x;
    const int cta = blockIdx.x;
    for (int b = lane; b < p.B; b += 32) {
        const int len = p.seq_lens[b];
        int n = (len + kBs - 1) / kBs;
        if (len < 1 || n > p.max_blocks) {
            n = 0;
            if (cta == 0) report(p.err, KVD_ERR_OOB);
        }
        plan_pref[b + 1] = n;
        if (cta == 0) plan[p.B + 1 + b] = len;
    }
    if (lane == 0) plan_pref[0] = 0;
    __syncwarp();
    scan_pref(plan_pref, p.B, lane);
    __syncwarp();
    if (cta == 0)
        for (int i = lane; i <= p.B; i += 32) plan[i] = plan_pref[i];
    const int64_t T = static_cast<int64_t>(p.n_kv) * plan_pref[p.B];
    const int64_t chunk = (T + p.nsplit - 1) / p.nsplit;
    const int64_t lo = chunk * cta;
    const int64_t hi = (lo + chunk < T) ? lo + chunk : T;
    int phys = -1;
    uint32_t vm = 0;
    if (lo < hi) {
        const Segment sg = find_segment(plan_pref, p.B, p.n_kv, lo, hi);
        const int j = sg.j0 + lane;
        if (j < sg.j1) {
            phys = p.block_table[static_cast<int64_t>(sg.b) * p.max_blocks + j];
            vm = block_word(phys, j, p.seq_lens[sg.b], p.num_blocks, p.host_blocks, p.retain, p.block_fmt, p.err);
        }
    }
    reinterpret_cast<int2*>(plan + plan_cta_off(p.B) + static_cast<int64_t>(cta) * 2 * kPlanBatch)[lane] =
        make_int2(phys, static_cast<int>(vm));
    if (cta == 0 && lane < 2) plan[plan_dyn_off(p.B, p.nsplit) + lane] = 0;
}

int64_t decode_plan_words(int batch, int nsplit) { return plan_words(batch, nsplit); }
int64_t decode_plan_dyn_off(int batch, int nsplit) { return plan_dyn_off(batch, nsplit); }

cudaError_t launch_plan(const DecodeParams& p, int32_t* plan, cudaStream_t stream) {
    plan_kernel<<<p.nsplit, 32, (p.B + 1) * sizeof(int), stream>>>(p, plan);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- wait self-test
__global__ void wait_timeout_kernel(int32_t* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing arrives on `bar`: the wait must give up and report
        if (!mbar_wait(&bar, 0, nullptr, limit_ns)) report(err, KVD_ERR_TIMEOUT);
    }
}

cudaError_t launch_wait_timeout(int32_t* err, int64_t timeout_ns, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(err, static_cast<uint64_t>(timeout_ns));
    return cudaGetLastError();
}

}  // namespace kvd
