// kvd_decode_kernel.cuh — paged GQA decode attention, split-KV, for sm_103a: the kernel
// template shared by the translation units that instantiate its pool kinds.
//
// What it computes (per request b, query head h, KV head h/g):
//   l_t = softmax_scale · q_h · K_t  for every attended position t (−inf if evicted),
//   out_h = Σ_t softmax(l)_t · V_t,   lse_h = log Σ_t exp(l_t);
// the K/V of position t come from physical block block_table[b][t/16], slot
// t%16 (page "LLM에서 KV 캐시는 얼마나 생길까", section "KV 캐시를 줄이는 기법":
// the kernel follows the block table, so scattered blocks give the same result;
// section "KV 캐시란": scores scaled by 1/√128, softmax, weighted sum of V).
//
// How (GB300 design):
//  * Work = the flattened sequence of (request, KV head, logical block); it is
//    cut into `nsplit` equal contiguous ranges, one CTA each, so every CTA
//    streams the same number of blocks whatever the length mix.  A CTA writes
//    one partial (o, lse) per unit segment it touches into slot u + piece, and
//    the combine kernel merges the partials of each unit by log-sum-exp.
//    With a step plan, BF16 kernels balance the work at run time: the last
//    sixth of every range is cut into pieces that CTAs done with their own part
//    take from a counter (see kPieces).
//  * One producer warp reads the block table (32 entries per coalesced load)
//    and issues 1-D bulk copies (TMA engine) of each (block, KV head) record —
//    K tile + V tile, 8 KiB BF16 or 4 KiB FP8 (+128 B of scales) — into a ring
//    of shared-memory stages guarded by mbarriers.
//  * NCW consumer warps take stages round-robin.  The record is stored in
//    tensor-core fragment order, so each lane's 16-byte shared loads are the
//    A operands of mma.m16n8k16 directly: S^T = K·Q^T (16 tokens × g heads,
//    the g query heads of the group share every K load), online softmax in
//    fp32 (exp2 domain), P^T built with movmatrix, O^T += V^T·P^T.
//  * FP8: codes convert exactly to f16; the K scale multiplies the fp32 logit,
//    the V scale folds into p before it is rounded to f16 for the MMA.
//  * Angle-domain keys: the K codes are each row's direction code and the
//    row's word is its logit factor r̃/||d_k||; the kernel codes q the same way
//    (E4M3 at its absmax scale, per head) and multiplies the logit by the
//    head's ||q||/||d_q||: the logit is ||q||·r̃·cos(d_q, d_k) from the codes.
//  * Low-bit (4-bit / 2-bit codes, a scale and a zero point per group of a
//    row): codes convert exactly to f16 through the E4M3 path; K accumulates
//    one MMA sum per group, combined with the group's scale and zero point in
//    fp32; V folds the group's scale into p, and the zero point's share,
//    Σ_t p_t·zero_t, is summed in fp32 beside the MMAs.
//  * Every mbarrier wait is bounded (%globaltimer); a timeout records
//    KVD_ERR_TIMEOUT and the CTA drains its copies and returns.
#pragma once

#include "kvd_common.cuh"
#include "kvd_internal.h"

namespace kvd {

constexpr int kNcw = 4;                    // consumer warps per CTA
constexpr int kThreads = (kNcw + 1) * 32;  // + 1 producer warp
constexpr int kMergeStride = 132;          // floats per head row in the merge buffer (bank spread)
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s

// Floats of one merge slot: O [g][kMergeStride], then m [kMaxG], then l [kMaxG].  Two
// slots suffice for the register tree merge of the four consumer warps.
__host__ __device__ inline int merge_floats(int g) { return g * kMergeStride + 2 * kMaxG; }

template <int KIND, int STAGES, int NG = 1>
struct Cfg {
    // record slot of one (block, KV head): a mixed pool sizes every slot for BF16 and an 8-bit
    // block fills the first kRecordFp8 bytes of it
    static constexpr int kBits = KIND == kKindInt4 ? 4 : KIND == kKindInt2 ? 2 : 0;
    static constexpr int kRecord = KIND == kKindFp8 || KIND == kKindAngle ? kRecordFp8
                                   : is_lowbit(KIND) ? lowbit_record_bytes(kBits, NG)
                                                     : kRecordBf16;
    static constexpr int kStage = kRecord;
    // Stage k%kStages is consumed by warp (k - segment start) % kNcw.  With kStages a
    // multiple of kNcw every reuse of a stage inside a segment belongs to the same warp,
    // and across segments the merge barrier orders it, so a consumer never waits on a
    // phase whose predecessor is still incomplete (mbarrier parity cannot alias).
    static constexpr int kStages = STAGES;
    static_assert(kStages % kNcw == 0, "stages must be a multiple of the consumer warps");
};

struct Smem {
    int ring_off, full_off, empty_off, meta_off, merge_off, pref_off, lens_off, abort_off, flag_off, total;
};

template <int KIND, int S, int NG = 1>
__host__ __device__ inline Smem smem_layout(int batch, int g) {
    constexpr int kStages = Cfg<KIND, S, NG>::kStages;
    Smem s;
    int o = 0;
    s.ring_off = o;
    o += kStages * Cfg<KIND, S, NG>::kStage;
    s.full_off = o;
    o += kStages * 8;
    s.empty_off = o;
    o += kStages * 8;
    s.meta_off = o;
    o += 2 * kStages * 4;   // per stage: the block word, then the tag of a taken piece
    o = (o + 15) & ~15;
    s.merge_off = o;
    o += 2 * merge_floats(g) * 4;
    s.pref_off = o;
    o += (batch + 1) * 4;
    s.lens_off = o;
    o += batch * 4;
    s.abort_off = o;
    o += 4;
    s.flag_off = o;
    o += 4;
    s.total = (o + 127) & ~127;
    return s;
}

struct Segment {
    int b, kvh;
    int j0, j1;       // logical block range of this CTA's piece of the unit
    int nblk;         // blocks of the whole unit (n_b)
    int64_t end;      // flattened index one past this piece
    int64_t unit_end; // flattened index one past the unit
};

// Record of (physical block ph, KV head h) to read: a pool block, or the staged copy of a
// host-tier block (ids num_blocks and up).
template <int64_t kRec>
__device__ __forceinline__ const uint8_t* record_of(const DecodeParams& p, int ph, int h) {
    return ph < p.num_blocks ? p.kv + (static_cast<int64_t>(ph) * p.n_kv + h) * kRec
                             : p.stage + ((static_cast<int64_t>(ph) - p.num_blocks) * p.n_kv + h) * kRec;
}

// A ring stage filled from a host-tier record in place, by the whole producer warp: 16-byte
// cp.async copies over the host link.  Each lane's copies hold the stage's phase open until
// they land, and lane 0's arrive (after every lane has registered) is the one arrival the
// phase expects.
template <int kRec>
__device__ __forceinline__ void lsu_fill(uint8_t* dst, const uint8_t* rec, uint64_t* full, int lane) {
    for (int c = lane; c < kRec / 16; c += 32) cp_async16_g2s(dst + 16 * c, rec + 16 * c);
    cp_async_mbar_arrive(full);
    __syncwarp();
    if (lane == 0) mbar_arrive(full);
}

struct IssueState {
    uint32_t k;            // copies issued so far (stage k % stages is next)
    uint32_t lsu_filled;   // lane 0: stages whose last fill was cp.async (generic proxy)
    int aborted;
    int piece;             // taken piece the stages belong to (stage tag, see kPieces)
};

// The producer's issue loop for a 32-block batch that holds host-tier blocks read in place:
// pool blocks by one bulk copy from lane 0, host-tier blocks copied by the whole warp
// (lsu_fill).  Out of line so that the plain loop, which every other batch runs, keeps its
// code as it is.
template <int kRec, int kStages>
__device__ __noinline__ IssueState issue_batch_with_hosts(const DecodeParams& p, uint8_t* ring, int stage_bytes,
                                                          uint64_t* full, uint64_t* empty, int* meta,
                                                          volatile int* abort_flag, uint64_t policy, int phys,
                                                          uint32_t vm, unsigned long long raddr, int cnt, int lane,
                                                          IssueState st) {
    for (int i = 0; i < cnt; ++i) {
        const int ph = __shfl_sync(kFull, phys, i);
        const uint32_t m = __shfl_sync(kFull, vm, i);
        const unsigned long long ra = __shfl_sync(kFull, raddr, i);
        const int s = st.k % kStages;
        const uint32_t par = (st.k / kStages) & 1u;
        const bool lsu = ph >= p.num_blocks && (m >> 16);   // warp-uniform
        int ok = 1;
        if (lane == 0) {
            ok = mbar_wait(&empty[s], par ^ 1u, abort_flag, kWaitNs);
            if (ok) {
                meta[s] = static_cast<int>(m);
                meta[kStages + s] = st.piece;
                if (lsu) {
                    st.lsu_filled |= 1u << s;
                } else if (m >> 16) {
                    if (st.lsu_filled >> s & 1u) {   // the stage's last writes were generic
                        fence_proxy_async_shared();
                        st.lsu_filled &= ~(1u << s);
                    }
                    mbar_arrive_expect_tx(&full[s], kRec);
                    bulk_g2s(ring + s * stage_bytes, reinterpret_cast<const uint8_t*>(ra), kRec, &full[s], policy);
                } else {
                    mbar_arrive(&full[s]);
                }
            } else {
                report(p.err, KVD_ERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) {
            st.aborted = 1;
            break;
        }
        if (lsu) lsu_fill<kRec>(ring + s * stage_bytes, reinterpret_cast<const uint8_t*>(ra), &full[s], lane);
        ++st.k;
    }
    return st;
}

// The producer's word for logical block j of a request of length len whose physical block is phys:
// bits 0-15 the slots to attend (valid positions, minus evicted ones), bit 16 set for a block
// inside the pool (else KVD_ERR_OOB is reported and the block is empty), bits 17-18 a mixed pool
// block's format.
__device__ __forceinline__ uint32_t block_word(int phys, int j, int len, int64_t num_blocks, int64_t host_blocks,
                                               const uint16_t* retain, const uint8_t* block_fmt, int32_t* err) {
    if (phys < 0 || phys >= num_blocks + host_blocks) {
        report(err, KVD_ERR_OOB);
        return 0;
    }
    const int valid = len - j * kBs;
    uint32_t vm = valid >= kBs ? 0xFFFFu : ((1u << valid) - 1u);
    if (retain) vm &= retain[phys];
    vm |= 1u << 16;
    if (block_fmt) {   // a mixed pool: the block's precision, bits 17-18
        const int fmt = block_format(block_fmt[phys]);
        if (fmt < 0) {
            report(err, KVD_ERR_OOB);
            return 0;
        }
        vm |= static_cast<uint32_t>(fmt) << 17;
    }
    return vm;
}

// Inclusive scan of pref[1..B] in shared memory by one warp (pref[0] = 0 stays).
__device__ __forceinline__ void scan_pref(int* pref, int B, int lane) {
    const int per = (B + 31) / 32;
    const int a = 1 + lane * per;
    const int e = min(B + 1, a + per);
    int run = 0;
    for (int i = a; i < e; ++i) run += pref[i];
    int incl = run;
    #pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    int acc = incl - run;
    for (int i = a; i < e; ++i) {
        acc += pref[i];
        pref[i] = acc;
    }
}

// A step's plan (kvd_decode_plan) in int32 words: pref [B + 1] (pref[b] = blocks of requests
// before b), lens [B], then, from a 16-byte boundary, per CTA the (physical block, block word)
// pairs of the first kPlanBatch blocks of its first segment, then the two counters of dynamic
// balancing (zeroed by the plan; the last CTA of each launch puts them back to zero).
constexpr int kPlanBatch = 32;
__host__ __device__ inline int64_t plan_cta_off(int B) { return (2 * static_cast<int64_t>(B) + 1 + 3) / 4 * 4; }
__host__ __device__ inline int64_t plan_dyn_off(int B, int nsplit) {
    return plan_cta_off(B) + static_cast<int64_t>(nsplit) * 2 * kPlanBatch;
}
__host__ __device__ inline int64_t plan_words(int B, int nsplit) { return plan_dyn_off(B, nsplit) + 2; }

// Dynamic balancing (with a step plan).  The flattened work is cut into nsplit equal ranges as
// without it, and each range into parts: its own part (the first 5/6), then kDynLevels pieces
// that make up the last sixth, of 1/2, 1/4, 1/8 and the rest of it.  A CTA streams its own part,
// then takes pieces from a counter shared by the grid, every CTA's largest pieces first, until
// none is left; early CTAs so take the work that late or slow ones would have finished last.
// Part i of range c is piece c·kPieces + i; a unit's partial for piece π goes to slot u + π (the
// pieces are in flattened order, so the slot is unique and a unit's slots are contiguous).
// Without dynamic balancing a range is one piece, π = c.
constexpr int kDynLevels = 4;
constexpr int kPieces = kDynLevels + 1;
constexpr int64_t kDynMinChunk = 192;
static_assert(kPieces == kDecodePieces, "pieces per range");

// Start of part i (0 ≤ i ≤ kPieces) inside a range of `chunk` blocks.
__host__ __device__ inline int64_t part_off(int64_t chunk, int i) {
    const int64_t d = chunk / 6;
    const int64_t a = chunk - d;
    switch (i) {
        case 0: return 0;
        case 1: return a;
        case 2: return a + d / 2;
        case 3: return a + d / 2 + d / 4;
        case 4: return a + d / 2 + d / 4 + d / 8;
        default: return chunk;
    }
}

// Piece holding flattened index x.
__device__ __forceinline__ int64_t piece_of(int64_t x, int64_t chunk, bool dyn) {
    const int64_t c = x / chunk;
    if (!dyn) return c;
    const int64_t o = x - c * chunk;
    const int i = (o >= part_off(chunk, 1)) + (o >= part_off(chunk, 2)) + (o >= part_off(chunk, 3)) +
                  (o >= part_off(chunk, 4));
    return c * kPieces + i;
}

// Flattened range [x0, x1) of piece π (empty past the end of the work).
__device__ __forceinline__ void piece_range(int64_t piece, int64_t chunk, int64_t T, bool dyn, int64_t& x0,
                                            int64_t& x1) {
    const int64_t c = dyn ? piece / kPieces : piece;
    const int i = dyn ? static_cast<int>(piece % kPieces) : 0;
    x0 = c * chunk + part_off(chunk, dyn ? i : 0);
    x1 = c * chunk + (dyn ? part_off(chunk, i + 1) : chunk);
    if (x0 > T) x0 = T;
    if (x1 > T) x1 = T;
}

// The piece behind taken number d (0 ≤ d < kDynLevels·nsplit): level d / nsplit of range d % nsplit.
__device__ __forceinline__ int64_t taken_piece(int d, int nsplit) {
    return static_cast<int64_t>(d % nsplit) * kPieces + 1 + d / nsplit;
}

// Unit holding flattened block index x: units are ordered (b, kvh); unit (b, kvh)
// covers [n_kv·pref[b] + kvh·n_b, n_kv·pref[b] + (kvh+1)·n_b).
__device__ __forceinline__ Segment find_segment(const int* pref, int B, int n_kv, int64_t x, int64_t hi) {
    int lo = 0, up = B - 1;
    while (lo < up) {
        const int mid = (lo + up + 1) >> 1;
        if (static_cast<int64_t>(n_kv) * pref[mid] <= x) lo = mid;
        else up = mid - 1;
    }
    Segment s;
    s.b = lo;
    s.nblk = pref[lo + 1] - pref[lo];
    const int64_t base = static_cast<int64_t>(n_kv) * pref[lo];
    s.kvh = static_cast<int>((x - base) / s.nblk);
    const int64_t ustart = base + static_cast<int64_t>(s.kvh) * s.nblk;
    s.unit_end = ustart + s.nblk;
    s.end = s.unit_end < hi ? s.unit_end : hi;
    s.j0 = static_cast<int>(x - ustart);
    s.j1 = static_cast<int>(s.end - ustart);
    return s;
}

__device__ __forceinline__ void store_out(const DecodeParams& p, int64_t idx, float v) {
    if (p.out_f32) {
        static_cast<float*>(p.out)[idx] = v;
    } else {
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        static_cast<__nv_bfloat16*>(p.out)[idx] = h;
    }
}

// One 16-token block of a unit by one consumer warp: S^T = K·Q^T for the g query heads of the
// group, online softmax (fp32, exp2 domain) and O^T += V^T·P^T.  FMT is the block's storage:
// kFmtBf16 (bf16 tiles, bf16 MMAs, qf in bf16) or kFmtE4m3 / kFmtE5m2 (8-bit codes converted
// exactly to f16, f16 MMAs, qf in f16; the K scale multiplies the fp32 logit and the V scale
// folds into p).  m: the block's valid-slot mask (bits 0..15).  lg0 / lg1: logit rows of heads
// h0 / h1 (or null), written at positions tb + slot below lim.  The stage is released (arrive
// on empty_s) as soon as its V tile is in registers.
// HF (angle-domain keys): the row's word is its logit factor, and hf0 / hf1 (softmax scale·log2(e)
// times the head's ||q||/||d_q||) multiply the logits of heads h0 / h1.
template <int FMT, bool HF = false>
__device__ __forceinline__ void consume_block(const uint8_t* st, const uint32_t (&qf)[8][2], float (&o)[8][4],
                                              float& m0, float& m1, float& s0, float& s1, uint32_t m,
                                              float scale_log2, float* lg0, float* lg1, int tb, int64_t lim,
                                              uint64_t* empty_s, int lane, float hf0 = 1.f, float hf1 = 1.f) {
    const int gid = lane >> 2;   // token row (S^T) / dim row (O^T) within an 8-row group
    const int tq = lane & 3;     // head pair 2tq, 2tq+1
    // ---- S^T = K · Q^T  (16 tokens × 8 heads) ----
    float ca[4] = {0.f, 0.f, 0.f, 0.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};
    float fk0, fk1, fv0 = 1.f, fv1 = 1.f;
    if constexpr (FMT == kFmtBf16) {
        const uint4* kt = reinterpret_cast<const uint4*>(st);
        #pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const uint4 a0 = kt[i * 32 + lane];
            const uint4 a1 = kt[(i + 1) * 32 + lane];
            const uint32_t fa[4] = {a0.x, a0.y, a0.z, a0.w};
            const uint32_t fb[4] = {a1.x, a1.y, a1.z, a1.w};
            mma_bf16(ca, fa, qf[i][0], qf[i][1]);
            mma_bf16(cb, fb, qf[i + 1][0], qf[i + 1][1]);
        }
        fk0 = fk1 = scale_log2;
    } else {
        const uint4* kt = reinterpret_cast<const uint4*>(st);
        #pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
            const uint4 w = kt[u4 * 32 + lane];
            uint32_t fa[4], fb[4];
            f8x4_to_f16x2x2<FMT>(w.x, fa[0], fa[1]);
            f8x4_to_f16x2x2<FMT>(w.y, fa[2], fa[3]);
            f8x4_to_f16x2x2<FMT>(w.z, fb[0], fb[1]);
            f8x4_to_f16x2x2<FMT>(w.w, fb[2], fb[3]);
            mma_f16(ca, fa, qf[2 * u4][0], qf[2 * u4][1]);
            mma_f16(cb, fb, qf[2 * u4 + 1][0], qf[2 * u4 + 1][1]);
        }
        const float* sc = reinterpret_cast<const float*>(st + 2 * kTileFp8);
        fk0 = HF ? sc[gid] : sc[gid] * scale_log2;
        fk1 = HF ? sc[gid + 8] : sc[gid + 8] * scale_log2;
        fv0 = sc[kBs + gid];
        fv1 = sc[kBs + gid + 8];
    }
    const bool v0 = (m >> gid) & 1u;        // token gid
    const bool v1 = (m >> (gid + 8)) & 1u;  // token gid + 8
    float l0 = v0 ? (ca[0] + cb[0]) * fk0 : -INFINITY;  // (gid,   h0)
    float l1 = v0 ? (ca[1] + cb[1]) * fk0 : -INFINITY;  // (gid,   h1)
    float l2 = v1 ? (ca[2] + cb[2]) * fk1 : -INFINITY;  // (gid+8, h0)
    float l3 = v1 ? (ca[3] + cb[3]) * fk1 : -INFINITY;  // (gid+8, h1)
    if constexpr (HF) {
        l0 *= hf0;
        l1 *= hf1;
        l2 *= hf0;
        l3 *= hf1;
    }

    {
        const int t0 = tb + gid, t1 = t0 + 8;
        if (lg0) {
            if (t0 < lim) st_logit(lg0 + t0, l0 * kLn2);
            if (t1 < lim) st_logit(lg0 + t1, l2 * kLn2);
        }
        if (lg1) {
            if (t0 < lim) st_logit(lg1 + t0, l1 * kLn2);
            if (t1 < lim) st_logit(lg1 + t1, l3 * kLn2);
        }
    }

    // ---- online softmax (exp2 domain), heads h0 and h1 ----
    float bm0 = fmaxf(l0, l2), bm1 = fmaxf(l1, l3);
    #pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, off));
        bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, off));
    }
    const float n0 = fmaxf(m0, bm0), n1 = fmaxf(m1, bm1);
    const float z0 = n0 == -INFINITY ? 0.f : n0;
    const float z1 = n1 == -INFINITY ? 0.f : n1;
    const float c0 = ex2(m0 - z0), c1 = ex2(m1 - z1);   // 0 when m was −inf
    const float p0 = ex2(l0 - z0), p1 = ex2(l1 - z1), p2 = ex2(l2 - z0), p3 = ex2(l3 - z1);
    s0 = s0 * c0 + (p0 + p2);
    s1 = s1 * c1 + (p1 + p3);
    m0 = n0;
    m1 = n1;
    if (__any_sync(kFull, c0 != 1.f || c1 != 1.f)) {
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            o[i][0] *= c0;
            o[i][1] *= c1;
            o[i][2] *= c0;
            o[i][3] *= c1;
        }
    }

    // ---- P^T fragment: rows = tokens, cols = heads -> transpose ----
    // p goes to the MMA as a 16-bit value plus the 16-bit value of its rounding remainder
    // (two MMAs): about 2^-17 (bf16) or 2^-22 (f16) relative per term.  A single 16-bit
    // p (2^-9 bf16, 2^-11 f16) lets outputs that cancel (few dominant positions, or FP8
    // channels 20x the others) lose more than the output tolerance.  FP8 folds the V
    // scale into p first.
    uint32_t pb0, pb1, pl0, pl1;
    if constexpr (FMT == kFmtBf16) {
        const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
        const float2 r01 = unpack_bf16(h01), r23 = unpack_bf16(h23);
        pb0 = movmatrix_t(h01);
        pb1 = movmatrix_t(h23);
        pl0 = movmatrix_t(pack_bf16(p0 - r01.x, p1 - r01.y));
        pl1 = movmatrix_t(pack_bf16(p2 - r23.x, p3 - r23.y));
    } else {
        const float w0 = v0 ? fv0 : 0.f, w1 = v1 ? fv1 : 0.f;
        const float a0 = p0 * w0, a1 = p1 * w0, a2 = p2 * w1, a3 = p3 * w1;
        const uint32_t h01 = pack_f16(a0, a1), h23 = pack_f16(a2, a3);
        const float2 r01 = unpack_f16(h01), r23 = unpack_f16(h23);
        pb0 = movmatrix_t(h01);
        pb1 = movmatrix_t(h23);
        pl0 = movmatrix_t(pack_f16(a0 - r01.x, a1 - r01.y));
        pl1 = movmatrix_t(pack_f16(a2 - r23.x, a3 - r23.y));
    }

    // ---- O^T += V^T · P^T ----
    // A block with an invalid slot (context tail, evicted) zeroes that slot's V in
    // this lane's fragment, so garbage (NaN) in unused slots cannot reach the output
    // through 0·NaN; full blocks (warp-uniform test) skip the masking.
    const bool partial = (m & 0xFFFFu) != 0xFFFFu;
    const int ta = 2 * tq;
    if constexpr (FMT == kFmtBf16) {
        const uint4* vt = reinterpret_cast<const uint4*>(st + kTileBf16);
        uint4 vv[8];
        #pragma unroll
        for (int i = 0; i < 8; ++i) vv[i] = vt[i * 32 + lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_s);
        if (partial) {   // 16-bit halves: tokens (2tq, 2tq+1) in .x/.y, (2tq+8, 2tq+9) in .z/.w
            const uint32_t zlo = (((m >> ta) & 1u) ? 0x0000FFFFu : 0u) | (((m >> (ta + 1)) & 1u) ? 0xFFFF0000u : 0u);
            const uint32_t zhi =
                (((m >> (ta + 8)) & 1u) ? 0x0000FFFFu : 0u) | (((m >> (ta + 9)) & 1u) ? 0xFFFF0000u : 0u);
            #pragma unroll
            for (int i = 0; i < 8; ++i) {
                vv[i].x &= zlo;
                vv[i].y &= zlo;
                vv[i].z &= zhi;
                vv[i].w &= zhi;
            }
        }
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t fa[4] = {vv[i].x, vv[i].y, vv[i].z, vv[i].w};
            mma_bf16(o[i], fa, pb0, pb1);
            mma_bf16(o[i], fa, pl0, pl1);
        }
    } else {
        const uint4* vt = reinterpret_cast<const uint4*>(st + kTileFp8);
        uint32_t zlo = 0xFFFFFFFFu, zhi = 0xFFFFFFFFu;
        if (partial) {   // bytes: tokens (2tq, 2tq+1) in .x/.z, (2tq+8, 2tq+9) in .y/.w; code 0 = +0
            zlo = (((m >> ta) & 1u) ? 0x00FFu : 0u) | (((m >> (ta + 1)) & 1u) ? 0xFF00u : 0u);
            zhi = (((m >> (ta + 8)) & 1u) ? 0x00FFu : 0u) | (((m >> (ta + 9)) & 1u) ? 0xFF00u : 0u);
            zlo |= zlo << 16;
            zhi |= zhi << 16;
        }
        // two halves of four m-tiles each keep fewer V registers live
        #pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint4 vv[2];
            vv[0] = vt[(2 * half) * 32 + lane];
            vv[1] = vt[(2 * half + 1) * 32 + lane];
            if (half == 1) {
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_s);
            }
            if (partial) {
                #pragma unroll
                for (int i = 0; i < 2; ++i) {
                    vv[i].x &= zlo;
                    vv[i].y &= zhi;
                    vv[i].z &= zlo;
                    vv[i].w &= zhi;
                }
            }
            #pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int u4 = 2 * half + i;
                uint32_t fa[4], fb[4];
                f8x4_to_f16x2x2<FMT>(vv[i].x, fa[0], fa[1]);
                f8x4_to_f16x2x2<FMT>(vv[i].y, fa[2], fa[3]);
                f8x4_to_f16x2x2<FMT>(vv[i].z, fb[0], fb[1]);
                f8x4_to_f16x2x2<FMT>(vv[i].w, fb[2], fb[3]);
                mma_f16(o[2 * u4], fa, pb0, pb1);
                mma_f16(o[2 * u4 + 1], fb, pb0, pb1);
                mma_f16(o[2 * u4], fa, pl0, pl1);
                mma_f16(o[2 * u4 + 1], fb, pl0, pl1);
            }
        }
    }
}

// Per-segment state of a low-bit unit: qz[g][0/1] = scale_log2 · Σ_{dims of group g} q of heads
// h0 / h1 (the f16 q the MMAs use), the zero point's coefficient in the logit; oz[g][0/1] = the
// running Σ_t p_t·zero_V[t][g] of heads h0 / h1 over this lane's tokens (rescaled with o).
template <int NG>
__device__ __forceinline__ void lowbit_q_sums(const uint32_t (&qf)[8][2], float scale_log2, float (&qz)[NG][2],
                                              int lane) {
    constexpr int kStepsPerGroup = 8 / NG;
    float part[NG];
    #pragma unroll
    for (int gi = 0; gi < NG; ++gi) part[gi] = 0.f;
    #pragma unroll
    for (int i = 0; i < 8; ++i) {   // head lane/4, dims 16i + 2(lane%4) + {0, 1, 8, 9}
        const float2 a = unpack_f16(qf[i][0]), b = unpack_f16(qf[i][1]);
        part[i / kStepsPerGroup] += (a.x + a.y) + (b.x + b.y);
    }
    const int tq = lane & 3;
    #pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        part[gi] += __shfl_xor_sync(kFull, part[gi], 1);
        part[gi] += __shfl_xor_sync(kFull, part[gi], 2);
        qz[gi][0] = scale_log2 * __shfl_sync(kFull, part[gi], 4 * (2 * tq));
        qz[gi][1] = scale_log2 * __shfl_sync(kFull, part[gi], 4 * (2 * tq + 1));
    }
}

// Four f16 fragment registers of k-step (K) / m-tile (V) P·kg + h from the two words (th = 0, 1)
// of group kg: field h of each word masked to one code per byte, bytes (0,1) and (2,3) through
// the E4M3 conversion (code c -> c·2^-9, exact).
template <int BITS>
__device__ __forceinline__ void lowbit_regs(uint32_t w0, uint32_t w1, int h, uint32_t& a01, uint32_t& a23,
                                            uint32_t& b01, uint32_t& b23) {
    constexpr uint32_t kMask = BITS == 4 ? 0x0F0F0F0Fu : 0x03030303u;
    const uint32_t m0 = (w0 >> (BITS * h)) & kMask;
    const uint32_t m1 = (w1 >> (BITS * h)) & kMask;
    e4m3x4_to_f16x2x2(m0, a01, a23);
    e4m3x4_to_f16x2x2(m1, b01, b23);
}

// The NG metadata words (scale | zero << 16) of one token, one per group, in one shared-memory load
// (a token's words are contiguous and 4·NG-byte aligned).
template <int NG>
__device__ __forceinline__ void load_meta(const uint32_t* row, uint32_t (&w)[NG]) {
    if constexpr (NG == 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(row);
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
    } else if constexpr (NG == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(row);
        w[0] = v.x;
        w[1] = v.y;
    } else {
        w[0] = row[0];
    }
}

// One 16-token block of a low-bit unit by one consumer warp (see consume_block for the fragment
// roles).  K: S^T accumulates one MMA sum per group (codes·2^-9 against q), and the logit of
// (token t, head h) is Σ_g scale_log2·(512·scale_K[t][g]·acc_g + zero_K[t][g]·Σ_{group} q_h).
// V: for the m-tiles of group g, p·scale_V[t][g] (≤ 65,504, since p ≤ 1) enters the MMA as an f16
// value plus the f16 of its remainder, so o holds Σ p·scale·code·2^-9 and the owner multiplies it
// by 512 at the end of the segment; oz[g] collects p·zero_V[t][g] in fp32.
template <int BITS, int NG>
__device__ __forceinline__ void consume_block_lowbit(const uint8_t* st, const uint32_t (&qf)[8][2],
                                                     const float (&qz)[NG][2], float (&o)[8][4], float (&oz)[NG][2],
                                                     float& m0, float& m1, float& s0, float& s1, uint32_t m,
                                                     float scale_log2, float* lg0, float* lg1, int tb, int64_t lim,
                                                     uint64_t* empty_s, int lane) {
    constexpr int kTile = lowbit_tile_bytes(BITS);
    constexpr int kPer = 8 / BITS;           // k-steps (m-tiles) per word
    constexpr int kGroups = 8 / kPer;        // word groups kg per tile
    constexpr int kChunks = kGroups / 2;     // 16-byte chunks per lane per tile
    constexpr int kStepsPerGroup = 8 / NG;   // k-steps (m-tiles) per scale group
    const int gid = lane >> 2;
    const int tq = lane & 3;
    const uint4* kt = reinterpret_cast<const uint4*>(st);
    const uint32_t* kmeta = reinterpret_cast<const uint32_t*>(st + 2 * kTile);
    const uint32_t* vmeta = kmeta + kBs * NG;

    // ---- S^T = K · Q^T, one accumulator per group ----
    float acc[NG][4];
    #pragma unroll
    for (int gi = 0; gi < NG; ++gi) acc[gi][0] = acc[gi][1] = acc[gi][2] = acc[gi][3] = 0.f;
    #pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        const uint4 w = kt[c * 32 + lane];
        #pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int kg = 2 * c + half;
            const uint32_t w0 = half ? w.z : w.x, w1 = half ? w.w : w.y;
            #pragma unroll
            for (int h = 0; h < kPer; ++h) {
                const int i = kPer * kg + h;
                uint32_t a[4];
                lowbit_regs<BITS>(w0, w1, h, a[0], a[2], a[1], a[3]);
                mma_f16(acc[i / kStepsPerGroup], a, qf[i][0], qf[i][1]);
            }
        }
    }
    const bool v0 = (m >> gid) & 1u;        // token gid
    const bool v1 = (m >> (gid + 8)) & 1u;  // token gid + 8
    float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
    uint32_t ka[NG], kb[NG];
    load_meta<NG>(kmeta + gid * NG, ka);         // token gid
    load_meta<NG>(kmeta + (gid + 8) * NG, kb);   // token gid + 8
    #pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        const float2 a = unpack_f16(ka[gi]);   // (scale, zero) of token gid
        const float2 b = unpack_f16(kb[gi]);
        const float sa = a.x * (512.f * scale_log2), sb = b.x * (512.f * scale_log2);
        l0 = fmaf(sa, acc[gi][0], fmaf(a.y, qz[gi][0], l0));
        l1 = fmaf(sa, acc[gi][1], fmaf(a.y, qz[gi][1], l1));
        l2 = fmaf(sb, acc[gi][2], fmaf(b.y, qz[gi][0], l2));
        l3 = fmaf(sb, acc[gi][3], fmaf(b.y, qz[gi][1], l3));
    }
    if (!v0) l0 = l1 = -INFINITY;
    if (!v1) l2 = l3 = -INFINITY;

    {
        const int t0 = tb + gid, t1 = t0 + 8;
        if (lg0) {
            if (t0 < lim) st_logit(lg0 + t0, l0 * kLn2);
            if (t1 < lim) st_logit(lg0 + t1, l2 * kLn2);
        }
        if (lg1) {
            if (t0 < lim) st_logit(lg1 + t0, l1 * kLn2);
            if (t1 < lim) st_logit(lg1 + t1, l3 * kLn2);
        }
    }

    // ---- online softmax (exp2 domain), heads h0 and h1 ----
    float bm0 = fmaxf(l0, l2), bm1 = fmaxf(l1, l3);
    #pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, off));
        bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, off));
    }
    const float n0 = fmaxf(m0, bm0), n1 = fmaxf(m1, bm1);
    const float z0 = n0 == -INFINITY ? 0.f : n0;
    const float z1 = n1 == -INFINITY ? 0.f : n1;
    const float c0 = ex2(m0 - z0), c1 = ex2(m1 - z1);   // 0 when m was −inf
    const float p0 = ex2(l0 - z0), p1 = ex2(l1 - z1), p2 = ex2(l2 - z0), p3 = ex2(l3 - z1);
    s0 = s0 * c0 + (p0 + p2);
    s1 = s1 * c1 + (p1 + p3);
    m0 = n0;
    m1 = n1;
    if (__any_sync(kFull, c0 != 1.f || c1 != 1.f)) {
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
            o[i][0] *= c0;
            o[i][1] *= c1;
            o[i][2] *= c0;
            o[i][3] *= c1;
        }
        #pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            oz[gi][0] *= c0;
            oz[gi][1] *= c1;
        }
    }

    // ---- V words and scales into registers, then the stage is free ----
    const uint4* vt = reinterpret_cast<const uint4*>(st + kTile);
    uint4 vw[kChunks];
    #pragma unroll
    for (int c = 0; c < kChunks; ++c) vw[c] = vt[c * 32 + lane];
    uint32_t va_w[NG], vb_w[NG];
    load_meta<NG>(vmeta + gid * NG, va_w);
    load_meta<NG>(vmeta + (gid + 8) * NG, vb_w);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_s);
    float2 va[NG], vb[NG];
    #pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        // an invalid slot's scale and zero point may be garbage (NaN): its p is 0, keep it 0
        va[gi] = unpack_f16(v0 ? va_w[gi] : 0u);
        vb[gi] = unpack_f16(v1 ? vb_w[gi] : 0u);
    }

    // ---- O^T += V^T · P'^T per group; zero-point share in fp32 ----
    #pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
        oz[gi][0] = fmaf(p0, va[gi].y, fmaf(p2, vb[gi].y, oz[gi][0]));
        oz[gi][1] = fmaf(p1, va[gi].y, fmaf(p3, vb[gi].y, oz[gi][1]));
        const float wa = va[gi].x, wb = vb[gi].x;
        const float a0 = p0 * wa, a1 = p1 * wa, a2 = p2 * wb, a3 = p3 * wb;
        const uint32_t h01 = pack_f16(a0, a1), h23 = pack_f16(a2, a3);
        const float2 r01 = unpack_f16(h01), r23 = unpack_f16(h23);
        const uint32_t pb0 = movmatrix_t(h01), pb1 = movmatrix_t(h23);
        const uint32_t pl0 = movmatrix_t(pack_f16(a0 - r01.x, a1 - r01.y));
        const uint32_t pl1 = movmatrix_t(pack_f16(a2 - r23.x, a3 - r23.y));
        #pragma unroll
        for (int ii = 0; ii < kStepsPerGroup; ++ii) {
            const int i = gi * kStepsPerGroup + ii;   // m-tile
            const int kg = i / kPer, h = i % kPer;
            const uint4 w = vw[kg >> 1];
            const uint32_t w0 = (kg & 1) ? w.z : w.x, w1 = (kg & 1) ? w.w : w.y;
            uint32_t a[4];
            lowbit_regs<BITS>(w0, w1, h, a[0], a[1], a[2], a[3]);
            mma_f16(o[i], a, pb0, pb1);
            mma_f16(o[i], a, pl0, pl1);
        }
    }
    (void)tq;
}

// DIRECT: the pool's host-tier blocks are read in place from host memory (lsu_fill); only
// pools with such a tier launch this variant, so the others carry none of its code.
template <int KIND, int S, bool DIRECT, int NG = 1>
__global__ void __launch_bounds__(kThreads, ((KIND == kKindFp8 || KIND == kKindAngle) && S == 8) ||
                                                   (is_lowbit(KIND) && NG == 1)
                                               ? 4
                                           : KIND == kKindMixed ? 2
                                                                : 3)
    decode_kernel(const DecodeParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    using C = Cfg<KIND, S, NG>;
    constexpr int kStages = C::kStages;
    const Smem L = smem_layout<KIND, S, NG>(p.B, p.g);
    uint8_t* ring = smem + L.ring_off;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full_off);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty_off);
    int* meta = reinterpret_cast<int*>(smem + L.meta_off);
    float* merge = reinterpret_cast<float*>(smem + L.merge_off);
    int* pref = reinterpret_cast<int*>(smem + L.pref_off);
    int* lens = reinterpret_cast<int*>(smem + L.lens_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_off);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int cta = blockIdx.x;
    // The previous kernel of the stream may write any input.  With p.early the caller has
    // promised that the block table, lengths, retain mask and the pool (except the slot the
    // fused append writes) are not among them: the plan and the K/V copies start at once,
    // and only the reads of q / k_new / v_new and every global write wait below.
    if (!p.early) pdl_wait();
    if (warp == kNcw) {
        // Warm L2 with the block-table row this CTA would start on if every request had
        // max_seq_len tokens (exact for uniform batches, a harmless miss otherwise); the real
        // loads come after the plan below.
        const int64_t nbg = (static_cast<int64_t>(p.max_seq_len) + kBs - 1) / kBs;
        const int64_t tg = nbg * p.n_kv * p.B;
        const int64_t lg = ((tg + p.nsplit - 1) / p.nsplit) * cta;
        if (nbg > 0 && lg < tg && lane < 2) {
            const int64_t ug = lg / nbg;
            const int64_t bg = ug / p.n_kv;
            const int64_t jg = lg % nbg + 32 * lane;
            if (bg < p.B && jg < p.max_blocks) {
                const int32_t* a = p.block_table + bg * p.max_blocks + jg;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
            }
        }
    }

    // ---- plan: blocks per request, prefix sums, this CTA's range -----------------
    // With a step plan (kvd_decode_plan) the prefix sums and lengths are read from it, and the
    // producer takes its first batch of blocks from it below: one round trip instead of three.
    int plan_phys = -1;
    uint32_t plan_vm = 0;
    if (p.plan) {
        if (warp == kNcw) {
            const int32_t* e = p.plan + plan_cta_off(p.B) + static_cast<int64_t>(cta) * 2 * kPlanBatch;
            const int2 pv = reinterpret_cast<const int2*>(e)[lane];
            plan_phys = pv.x;
            plan_vm = static_cast<uint32_t>(pv.y);
        }
        for (int i = tid; i <= p.B; i += kThreads) pref[i] = p.plan[i];
        for (int b = tid; b < p.B; b += kThreads) lens[b] = p.plan[p.B + 1 + b];
    } else {
        for (int b = tid; b < p.B; b += kThreads) {
            const int len = p.seq_lens[b];
            lens[b] = len;
            int n = (len + kBs - 1) / kBs;
            if (len < 1 || n > p.max_blocks) {
                n = 0;
                if (cta == 0) report(p.err, KVD_ERR_OOB);
            }
            pref[b + 1] = n;
        }
    }
    if (tid == 0) {
        if (!p.plan) pref[0] = 0;
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_fence_init();
    }
    __syncthreads();
    if (!p.plan && warp == 0) scan_pref(pref, p.B, lane);
    __syncthreads();

    const int64_t T = static_cast<int64_t>(p.n_kv) * pref[p.B];
    const int64_t chunk = (T + p.nsplit - 1) / p.nsplit;
    // Dynamic balancing needs long ranges: a taken piece costs its CTA a segment switch (q reload,
    // state merge, partial write, about 1.5 µs), which a piece of a few blocks does not repay
    // (measured: 70B FP8 ranges of 144 blocks 24% slower, 8B BF16 ranges of 288 blocks 3% faster).
    // From 48 blocks on no part is empty, so a unit's pieces have consecutive numbers.
    // (BF16 kernels only: the launch sets p.dyn for BF16 pools alone, and the other kinds carry
    // none of its code)
    const bool dyn = KIND == kKindBf16 && p.dyn != nullptr && chunk >= kDynMinChunk;
    const int64_t lo = chunk * cta < T ? chunk * cta : T;
    // the CTA's own part: all of its range, or with dynamic balancing the part before the pieces
    const int64_t own = lo + (dyn ? part_off(chunk, 1) : chunk);
    const int64_t hi = own < T ? own : T;

    // Units with no block: no CTA covers them, so CTA 0's consumer warps mark them empty.
    if (cta == 0 && warp < kNcw) {
        if (p.early) pdl_wait();
        const int U = p.B * p.n_kv;
        for (int u = tid; u < U; u += kNcw * 32) {
            const int b = u / p.n_kv;
            if (pref[b + 1] == pref[b]) {
                p.unit_first[u] = 0;
                p.unit_count[u] = 0;
            }
        }
    }

    if (warp == kNcw) {
        // =========================== producer warp ===========================
        const uint64_t policy = policy_evict_first();
        uint32_t k = 0;
        uint32_t lsu_filled = 0;   // lane 0: stages whose last fill was cp.async (generic proxy)
        bool aborted = false;
        int64_t rx0 = lo, rx1 = hi;   // the range being issued: the own part, then each taken piece
        int tag = -2;                 // stage tag: the taken piece the stages belong to
        while (!aborted) {
            for (int64_t x = rx0; x < rx1 && !aborted;) {
                const Segment sg = find_segment(pref, p.B, p.n_kv, x, rx1);
                const int32_t* bt = p.block_table + static_cast<int64_t>(sg.b) * p.max_blocks;
                const int len = lens[sg.b];
                if (p.k_new && sg.j1 == sg.nblk) {
                    // Fused append: this CTA owns the unit's last block, so it writes the new token
                    // (position len-1) into the pool before it bulk-copies that block.
                    const int pos = len - 1;
                    const int ph = bt[pos / kBs];
                    if (p.early) pdl_wait();   // k_new / v_new come from the previous kernel
                    if (ph >= 0 && ph < p.num_blocks + p.host_blocks) {
                        const int64_t row = (static_cast<int64_t>(sg.b) * p.n_kv + sg.kvh) * kDh;
                        uint8_t* rec = const_cast<uint8_t*>(record_of<C::kRecord>(p, ph, sg.kvh));
                        if constexpr (is_lowbit(KIND)) {      // no host tier
                            write_token_lowbit<C::kBits, NG>(rec, pos % kBs, p.k_new + row, p.v_new + row, lane);
                        } else if constexpr (KIND == kKindAngle) {   // no host tier
                            write_token<kFmtE4m3, true>(rec, pos % kBs, p.k_new + row, p.v_new + row, lane);
                        } else if constexpr (KIND == kKindMixed) {   // the block's own format (no host tier)
                            const int fmt = ph < p.num_blocks ? block_format(p.block_fmt[ph]) : -1;
                            const uint16_t* kn = p.k_new + row;
                            const uint16_t* vn = p.v_new + row;
                            if (fmt == kFmtBf16) write_token<kFmtBf16>(rec, pos % kBs, kn, vn, lane);
                            else if (fmt == kFmtE4m3) write_token<kFmtE4m3>(rec, pos % kBs, kn, vn, lane);
                            else if (fmt == kFmtE5m2) write_token<kFmtE5m2>(rec, pos % kBs, kn, vn, lane);
                        } else {
                            constexpr int kF = KIND == kKindFp8 ? kFmtE4m3 : kFmtBf16;
                            write_token<kF>(rec, pos % kBs, p.k_new + row, p.v_new + row, lane);
                            if (ph >= p.num_blocks && !p.host_direct) {   // a staged host-tier block: its host copy too
                                const int64_t hrec = (static_cast<int64_t>(ph) - p.num_blocks) * p.n_kv + sg.kvh;
                                write_token<kF>(p.host_kv + hrec * C::kRecord, pos % kBs, p.k_new + row, p.v_new + row,
                                                lane);
                            }
                        }
                        fence_proxy_async_global();
                    }
                    __syncwarp();
                }
                for (int jb = sg.j0; jb < sg.j1 && !aborted; jb += 32) {
                    const int j = jb + lane;
                    int phys = -1;
                    uint32_t vm = 0;
                    unsigned long long raddr = 0;
                    if (j < sg.j1) {
                        if (p.plan && k == 0) {   // the CTA's first batch, from the step plan
                            phys = plan_phys;
                            vm = plan_vm;
                        } else {
                            phys = bt[j];
                            vm = block_word(phys, j, len, p.num_blocks, p.host_blocks, p.retain,
                                            KIND == kKindMixed ? p.block_fmt : nullptr, p.err);
                        }
                        // each lane forms its block's record address here, in parallel, so that
                        // lane 0's serial issue loop below only shuffles it in
                        if (vm >> 16)
                            raddr = reinterpret_cast<unsigned long long>(record_of<C::kRecord>(p, phys, sg.kvh));
                    }
                    const int cnt = min(32, sg.j1 - jb);
                    if (DIRECT && __any_sync(kFull, phys >= p.num_blocks)) {
                        // a batch holding host-tier blocks read in place: issued out of line, so the
                        // loop below stays the plain pool-block loop
                        const IssueState st = issue_batch_with_hosts<C::kRecord, kStages>(
                            p, ring, C::kStage, full, empty, meta, abort_flag, policy, phys, vm, raddr, cnt, lane,
                            IssueState{k, lsu_filled, aborted ? 1 : 0, tag});
                        k = st.k;
                        lsu_filled = st.lsu_filled;
                        aborted = st.aborted != 0;
                        continue;
                    }
                    for (int i = 0; i < cnt; ++i) {
                        const uint32_t m = __shfl_sync(kFull, vm, i);
                        const unsigned long long ra = __shfl_sync(kFull, raddr, i);
                        const int s = k % kStages;
                        const uint32_t par = (k / kStages) & 1u;
                        int ok = 1;
                        if (lane == 0) {
                            ok = mbar_wait(&empty[s], par ^ 1u, abort_flag, kWaitNs);
                            if (ok) {
                                meta[s] = static_cast<int>(m);
                                if constexpr (KIND == kKindBf16) meta[kStages + s] = tag;   // run-time balancing
                                if (m >> 16) {
                                    const uint8_t* rec = reinterpret_cast<const uint8_t*>(ra);
                                    uint8_t* dst = ring + s * C::kStage;
                                    if (DIRECT && (lsu_filled >> s & 1u)) {   // the stage's last writes were generic
                                        fence_proxy_async_shared();
                                        lsu_filled &= ~(1u << s);
                                    }
                                    // a mixed pool's 8-bit block fills only the first kRecordFp8 bytes of its slot
                                    const uint32_t bytes =
                                        KIND == kKindMixed && ((m >> 17) & 3u) != kFmtBf16 ? kRecordFp8 : C::kRecord;
                                    mbar_arrive_expect_tx(&full[s], bytes);
                                    bulk_g2s(dst, rec, bytes, &full[s], policy);
                                } else {
                                    mbar_arrive(&full[s]);
                                }
                            } else {
                                report(p.err, KVD_ERR_TIMEOUT);
                                *abort_flag = 1;
                            }
                        }
                        ok = __shfl_sync(kFull, ok, 0);
                        if (!ok) {
                            aborted = true;
                            break;
                        }
                        ++k;
                    }
                }
                x = sg.end;
            }
            if (!dyn || aborted) break;
            // Take the next piece.  A number past the last piece ends the CTA's work: one stage tagged
            // -1 tells the consumer warps, and the last CTA to get here puts the counters back to zero
            // for the next launch that shares the plan.  That launch cannot take a piece earlier: its
            // own part (at least 5/6 of kDynMinChunk blocks) outlasts its ring, so its producer waits
            // for its consumers, and they wait for this launch to complete before their first block.
            int d = 0;
            if (lane == 0) d = atomicAdd(p.dyn, 1);
            d = __shfl_sync(kFull, d, 0);
            if (d >= kDynLevels * p.nsplit) {
                int ok = 1;
                if (lane == 0) {
                    const int s = k % kStages;
                    ok = mbar_wait(&empty[s], ((k / kStages) & 1u) ^ 1u, abort_flag, kWaitNs);
                    if (ok) {
                        meta[s] = 0;
                        meta[kStages + s] = -1;
                        mbar_arrive(&full[s]);
                    } else {
                        report(p.err, KVD_ERR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    if (atomicAdd(p.dyn + 1, 1) == p.nsplit - 1) {
                        p.dyn[0] = 0;
                        p.dyn[1] = 0;
                    }
                }
                if (__shfl_sync(kFull, ok, 0)) ++k;
                break;
            }
            const int64_t pc = taken_piece(d, p.nsplit);
            piece_range(pc, chunk, T, true, rx0, rx1);
            tag = static_cast<int>(pc);
        }
        // Drain: every issued copy must land before the CTA may exit.
        if (lane == 0) {
            const uint32_t first = k > static_cast<uint32_t>(kStages) ? k - kStages : 0u;
            for (uint32_t kk = first; kk < k; ++kk)
                if (!mbar_wait(&full[kk % kStages], (kk / kStages) & 1u, nullptr, kWaitNs))
                    report(p.err, KVD_ERR_TIMEOUT);
        }
        return;
    }

    // ============================ consumer warps ============================
    const int gid = lane >> 2;   // token row (S^T) / dim row (O^T) within an 8-row group
    const int tq = lane & 3;     // head pair 2tq, 2tq+1
    const int h0 = 2 * tq, h1 = 2 * tq + 1;
    const int g = p.g;
    if (p.early) pdl_wait();   // q and every output of this kernel
    uint32_t k = 0;
    int64_t rx0 = lo, rx1 = hi;                                  // the own part, then each taken piece
    int64_t piece = dyn ? static_cast<int64_t>(cta) * kPieces : cta;
    while (true) {
        for (int64_t x = rx0; x < rx1;) {
            const Segment sg = find_segment(pref, p.B, p.n_kv, x, rx1);
            const int nseg = sg.j1 - sg.j0;
            const int len = lens[sg.b];
            const int u = sg.b * p.n_kv + sg.kvh;

            // Q^T fragments (B operand): head gid, dims 16i + 2tq + {0,1,8,9}; in f16 for 8-bit
            // blocks (qf), in bf16 for BF16 blocks (qf of a BF16 pool, qfb of a mixed pool).
            uint32_t qf[8][2];
            uint32_t qfb[8][2];
            {
                const uint16_t* qh = p.q + (static_cast<int64_t>(sg.b) * p.n_q + sg.kvh * g + gid) * kDh;
                #pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint32_t lo2 = 0, hi2 = 0;
                    if (gid < g) {
                        lo2 = *reinterpret_cast<const uint32_t*>(qh + 16 * i + 2 * tq);
                        hi2 = *reinterpret_cast<const uint32_t*>(qh + 16 * i + 2 * tq + 8);
                    }
                    if constexpr (KIND == kKindMixed) {
                        qfb[i][0] = lo2;
                        qfb[i][1] = hi2;
                    }
                    if constexpr (KIND != kKindBf16) {  // bf16 -> f16 (exact inside the f16 range)
                        const __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&lo2);
                        const __nv_bfloat162 c = *reinterpret_cast<__nv_bfloat162*>(&hi2);
                        lo2 = pack_f16(__low2float(a), __high2float(a));
                        hi2 = pack_f16(__low2float(c), __high2float(c));
                    }
                    qf[i][0] = lo2;
                    qf[i][1] = hi2;
                }
            }

            // Angle-domain keys: q of head gid becomes its E4M3 direction code at its absmax scale (the
            // f16 fragments hold the code values, exactly) and hf0 / hf1 carry ||q||/||d_q|| of heads
            // h0 / h1 times the softmax scale.
            float hf0 = 1.f, hf1 = 1.f;
            if constexpr (KIND == kKindAngle) {
                float amax = 0.f;
                #pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 a = unpack_f16(qf[i][0]), b = unpack_f16(qf[i][1]);
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y))));
                }
                amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
                const float qs = amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
                float q2 = 0.f, d2 = 0.f;
                #pragma unroll
                for (int i = 0; i < 8; ++i) {
                    #pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float2 a = unpack_f16(qf[i][r]);
                        const uint32_t c0 = __nv_cvt_float_to_fp8(__fdiv_rn(a.x, qs), __NV_SATFINITE, __NV_E4M3);
                        const uint32_t c1 = __nv_cvt_float_to_fp8(__fdiv_rn(a.y, qs), __NV_SATFINITE, __NV_E4M3);
                        qf[i][r] = e4m3x2_to_f16x2(c0 | (c1 << 8));
                        const float2 dv = unpack_f16(qf[i][r]);
                        q2 = fmaf(a.x, a.x, fmaf(a.y, a.y, q2));
                        d2 = fmaf(dv.x, dv.x, fmaf(dv.y, dv.y, d2));
                    }
                }
                q2 += __shfl_xor_sync(kFull, q2, 1);
                q2 += __shfl_xor_sync(kFull, q2, 2);
                d2 += __shfl_xor_sync(kFull, d2, 1);
                d2 += __shfl_xor_sync(kFull, d2, 2);
                const float f = d2 > 0.f ? sqrtf(q2) / sqrtf(d2) : 0.f;   // head gid
                hf0 = p.scale_log2 * __shfl_sync(kFull, f, 4 * h0);
                hf1 = p.scale_log2 * __shfl_sync(kFull, f, 4 * h1);
            }

            float m0 = -INFINITY, m1 = -INFINITY;   // running max (log2 domain), heads h0, h1
            float s0 = 0.f, s1 = 0.f;               // running sum of p (this lane's tokens)
            float o[8][4];
            #pragma unroll
            for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
            float qz[NG][2], oz[NG][2];             // low-bit pools: zero-point terms
            #pragma unroll
            for (int gi = 0; gi < NG; ++gi) oz[gi][0] = oz[gi][1] = 0.f;
            if constexpr (is_lowbit(KIND)) lowbit_q_sums<NG>(qf, p.scale_log2, qz, lane);

            float* lg0 = nullptr;
            float* lg1 = nullptr;
            if (p.logits) {
                const int64_t rowb = static_cast<int64_t>(sg.b) * p.n_q + sg.kvh * g;
                lg0 = h0 < g ? p.logits + (rowb + h0) * p.logits_stride : nullptr;
                lg1 = h1 < g ? p.logits + (rowb + h1) * p.logits_stride : nullptr;
            }
            const int64_t lim = len < p.logits_stride ? len : p.logits_stride;

            for (int kk = warp; kk < nseg; kk += kNcw) {
                const uint32_t kg = k + kk;
                const int s = kg % kStages;
                // every lane observes the phase (acquire); the outcome is made warp-uniform so a
                // timeout racing with completion cannot split the warp before the MMAs
                const bool got = mbar_wait(&full[s], (kg / kStages) & 1u, abort_flag, kWaitNs);
                if (!__all_sync(kFull, got)) {
                    if (lane == 0) {
                        report(p.err, KVD_ERR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    break;
                }
                const uint32_t m = static_cast<uint32_t>(meta[s]);
                if (!(m >> 16)) {  // bad block id: reported by the producer, treated as empty
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                    continue;
                }
                const uint8_t* st = ring + s * C::kStage;
                const int j = sg.j0 + kk;

                const int tb = j * kBs;
                if constexpr (KIND == kKindMixed) {
                    const uint32_t fmt = (m >> 17) & 3u;
                    if (fmt == kFmtBf16)
                        consume_block<kFmtBf16>(st, qfb, o, m0, m1, s0, s1, m, p.scale_log2, lg0, lg1, tb, lim,
                                                &empty[s], lane);
                    else if (fmt == kFmtE4m3)
                        consume_block<kFmtE4m3>(st, qf, o, m0, m1, s0, s1, m, p.scale_log2, lg0, lg1, tb, lim,
                                                &empty[s], lane);
                    else
                        consume_block<kFmtE5m2>(st, qf, o, m0, m1, s0, s1, m, p.scale_log2, lg0, lg1, tb, lim,
                                                &empty[s], lane);
                } else if constexpr (is_lowbit(KIND)) {
                    consume_block_lowbit<C::kBits, NG>(st, qf, qz, o, oz, m0, m1, s0, s1, m, p.scale_log2, lg0, lg1, tb,
                                                       lim, &empty[s], lane);
                } else if constexpr (KIND == kKindAngle) {
                    consume_block<kFmtE4m3, true>(st, qf, o, m0, m1, s0, s1, m, p.scale_log2, lg0, lg1, tb, lim,
                                                  &empty[s], lane, hf0, hf1);
                } else {
                    constexpr int kF = KIND == kKindFp8 ? kFmtE4m3 : kFmtBf16;
                    consume_block<kF>(st, qf, o, m0, m1, s0, s1, m, p.scale_log2, lg0, lg1, tb, lim, &empty[s], lane);
                }
            }
            k += nseg;
            if constexpr (is_lowbit(KIND)) {
                // o holds Σ p·scale·code·2^-9 per lane's fragment; add the zero-point share, summed
                // over the eight lanes that hold the warp's tokens of heads h0, h1
                constexpr int kStepsPerGroup = 8 / NG;
                #pragma unroll
                for (int gi = 0; gi < NG; ++gi) {
                    #pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        oz[gi][0] += __shfl_xor_sync(kFull, oz[gi][0], off);
                        oz[gi][1] += __shfl_xor_sync(kFull, oz[gi][1], off);
                    }
                }
                #pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int gi = i / kStepsPerGroup;
                    o[i][0] = fmaf(o[i][0], 512.f, oz[gi][0]);
                    o[i][2] = fmaf(o[i][2], 512.f, oz[gi][0]);
                    o[i][1] = fmaf(o[i][1], 512.f, oz[gi][1]);
                    o[i][3] = fmaf(o[i][3], 512.f, oz[gi][1]);
                }
            }
            if (!dyn && sg.end == hi) pdl_trigger();   // this CTA's last piece has been streamed

            // ---- merge the consumer warps' states (register tree: 3+2 -> 1+0, then 1 -> 0) ----
            #pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                s0 += __shfl_xor_sync(kFull, s0, off);
                s1 += __shfl_xor_sync(kFull, s1, off);
            }
            const int MF = merge_floats(g);
            auto publish = [&](float* mb) {
                #pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int d0 = 16 * i + gid, d1 = d0 + 8;
                    if (h0 < g) {
                        mb[h0 * kMergeStride + d0] = o[i][0];
                        mb[h0 * kMergeStride + d1] = o[i][2];
                    }
                    if (h1 < g) {
                        mb[h1 * kMergeStride + d0] = o[i][1];
                        mb[h1 * kMergeStride + d1] = o[i][3];
                    }
                }
                if (gid == 0) {
                    mb[g * kMergeStride + h0] = m0;
                    mb[g * kMergeStride + h1] = m1;
                    mb[g * kMergeStride + kMaxG + h0] = s0;
                    mb[g * kMergeStride + kMaxG + h1] = s1;
                }
            };
            auto fold = [&](const float* mb) {
                const float mo0 = mb[g * kMergeStride + h0], mo1 = mb[g * kMergeStride + h1];
                const float so0 = mb[g * kMergeStride + kMaxG + h0], so1 = mb[g * kMergeStride + kMaxG + h1];
                const float M0 = fmaxf(m0, mo0), M1 = fmaxf(m1, mo1);
                const float z0 = M0 == -INFINITY ? 0.f : M0, z1 = M1 == -INFINITY ? 0.f : M1;
                const float a0 = ex2(m0 - z0), b0 = ex2(mo0 - z0);   // 0 for a -inf side
                const float a1 = ex2(m1 - z1), b1 = ex2(mo1 - z1);
                s0 = s0 * a0 + so0 * b0;
                s1 = s1 * a1 + so1 * b1;
                m0 = M0;
                m1 = M1;
                #pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int d0 = 16 * i + gid, d1 = d0 + 8;
                    const float p00 = h0 < g ? mb[h0 * kMergeStride + d0] : 0.f;
                    const float p02 = h0 < g ? mb[h0 * kMergeStride + d1] : 0.f;
                    const float p11 = h1 < g ? mb[h1 * kMergeStride + d0] : 0.f;
                    const float p13 = h1 < g ? mb[h1 * kMergeStride + d1] : 0.f;
                    o[i][0] = o[i][0] * a0 + p00 * b0;
                    o[i][2] = o[i][2] * a0 + p02 * b0;
                    o[i][1] = o[i][1] * a1 + p11 * b1;
                    o[i][3] = o[i][3] * a1 + p13 * b1;
                }
            };
            if (warp >= 2) publish(merge + (warp - 2) * MF);
            named_barrier(1, kNcw * 32);
            if (warp < 2) fold(merge + warp * MF);
            named_barrier(1, kNcw * 32);
            if (warp == 1) publish(merge);
            named_barrier(1, kNcw * 32);
            // A unit that lies in this CTA alone is final here: write the output straight from
            // registers and mark it done (unit_count = -1) so the combine kernel skips it.
            const bool whole = p.out != nullptr && sg.j0 == 0 && sg.end == sg.unit_end;
            if (warp == 0) {
                fold(merge);
                const float i0 = s0 > 0.f ? 1.f / s0 : 0.f, i1 = s1 > 0.f ? 1.f / s1 : 0.f;
                const float ls0 = s0 > 0.f ? (m0 + log2f(s0)) * kLn2 : -INFINITY;
                const float ls1 = s1 > 0.f ? (m1 + log2f(s1)) * kLn2 : -INFINITY;
                if (whole) {
                    const int64_t orow = static_cast<int64_t>(sg.b) * p.n_q + sg.kvh * g;
                    #pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int d0 = 16 * i + gid, d1 = d0 + 8;
                        if (h0 < g) {
                            store_out(p, (orow + h0) * kDh + d0, o[i][0] * i0);
                            store_out(p, (orow + h0) * kDh + d1, o[i][2] * i0);
                        }
                        if (h1 < g) {
                            store_out(p, (orow + h1) * kDh + d0, o[i][1] * i1);
                            store_out(p, (orow + h1) * kDh + d1, o[i][3] * i1);
                        }
                    }
                    if (p.lse_out && gid == 0) {
                        if (h0 < g) p.lse_out[orow + h0] = ls0;
                        if (h1 < g) p.lse_out[orow + h1] = ls1;
                    }
                    if (lane == 0) {
                        p.unit_first[u] = u + static_cast<int>(piece);
                        p.unit_count[u] = -1;
                    }
                } else {
                    // this unit piece's partial: o normalised over its own positions, and its lse
                    const int slot = u + static_cast<int>(piece);
                    float* po = p.part_o + static_cast<int64_t>(slot) * g * kDh;
                    #pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int d0 = 16 * i + gid, d1 = d0 + 8;
                        if (h0 < g) {
                            po[h0 * kDh + d0] = o[i][0] * i0;
                            po[h0 * kDh + d1] = o[i][2] * i0;
                        }
                        if (h1 < g) {
                            po[h1 * kDh + d0] = o[i][1] * i1;
                            po[h1 * kDh + d1] = o[i][3] * i1;
                        }
                    }
                    if (gid == 0) {
                        float* pl = p.part_lse + static_cast<int64_t>(slot) * g;
                        if (h0 < g) pl[h0] = ls0;
                        if (h1 < g) pl[h1] = ls1;
                    }
                    if (sg.j0 == 0 && lane == 0) {
                        p.unit_first[u] = slot;
                        p.unit_count[u] = static_cast<int>(piece_of(sg.unit_end - 1, chunk, dyn) - piece + 1);
                    }
                }
            }
            named_barrier(1, kNcw * 32);   // the buffer is free again for the next segment
            x = sg.end;
        }
        if (!dyn) break;
        // The next taken piece: its first stage carries the piece's number (-1: none left).
        const int s = k % kStages;
        const bool got = mbar_wait(&full[s], (k / kStages) & 1u, abort_flag, kWaitNs);
        if (!__all_sync(kFull, got)) {
            if (lane == 0) {
                report(p.err, KVD_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            break;
        }
        const int t = meta[kStages + s];
        if (t < 0) break;
        piece = t;
        piece_range(piece, chunk, T, true, rx0, rx1);
    }
    if (dyn) pdl_trigger();   // every piece of this CTA has been streamed
}

// Shared memory per SM and per-block reservation of the current device (cached per device).
static inline bool smem_attrs(int* per_sm, int* reserved) {
    static int cached_dev = -1, c_per_sm = 0, c_reserved = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (dev != cached_dev) {
        int a = 0, r = 0;
        if (cudaDeviceGetAttribute(&a, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) return false;
        if (cudaDeviceGetAttribute(&r, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) return false;
        c_per_sm = a;
        c_reserved = r;
        cached_dev = dev;
    }
    *per_sm = c_per_sm;
    *reserved = c_reserved;
    return c_per_sm > 0;
}

// Raise the kernel's dynamic shared-memory limit once per device to the largest
// layout any batch size can need (batch ≤ kMaxBatch).
template <int KIND, int S, bool DIRECT, int NG = 1>
static cudaError_t ensure_smem_attr() {
    static int done_for_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (done_for_device == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(decode_kernel<KIND, S, DIRECT, NG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_layout<KIND, S, NG>(kMaxBatch, kMaxG).total);
    if (e == cudaSuccess) done_for_device = dev;
    return e;
}

template <int KIND, int S, int NG = 1>
static int ctas_per_sm_impl(int batch, int g) {
    const int smem = smem_layout<KIND, S, NG>(batch, g).total;
    if (ensure_smem_attr<KIND, S, false, NG>() != cudaSuccess) return 1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<KIND, S, false, NG>, kThreads, smem) !=
        cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

template <int KIND, int S, bool DIRECT, int NG = 1>
static cudaError_t launch_variant(const DecodeParams& p, int carveout, cudaStream_t stream) {
    const cudaError_t e = ensure_smem_attr<KIND, S, DIRECT, NG>();
    if (e != cudaSuccess) return e;
    const size_t smem = smem_layout<KIND, S, NG>(p.B, p.g).total;
    return launch_dependent(decode_kernel<KIND, S, DIRECT, NG>, dim3(p.nsplit), dim3(kThreads), smem, carveout,
                            stream, p);
}

}  // namespace kvd
