// kvd_internal.h — kernel parameter blocks and launchers (host <-> device, not exported).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

struct kvd_pool;

namespace kvd {

// Pool kinds: every block BF16, every block FP8-E4M3, mixed (a precision byte per block), or
// low-bit (4-bit or 2-bit codes with a half-precision scale and zero point per group of values).
constexpr int kKindBf16 = 0, kKindFp8 = 1, kKindMixed = 2, kKindInt4 = 3, kKindInt2 = 4;
// Angle-domain keys: FP8 records whose K codes are the direction code of each key row and whose
// K scale word is the row's logit factor w = r̃/||d||; the query is coded the same way in-kernel.
constexpr int kKindAngle = 5;
__host__ __device__ constexpr bool is_lowbit(int kind) { return kind == kKindInt4 || kind == kKindInt2; }

// Device ordinal the pool was created on (its memory and state live there).
int pool_device(const kvd_pool* pool);

struct AppendParams {
    const uint16_t* k_new;       // bf16 bits [n_tokens][n_kv][128]
    const uint16_t* v_new;
    const int64_t* slot_mapping; // [n_tokens]
    uint8_t* kv;                 // this layer's records
    uint8_t* host_kv;            // this layer's host-tier records (device address), or null
    const uint8_t* block_fmt;    // mixed pools: precision code of every physical block
    int32_t* err;
    int ng;                      // low-bit pools: groups per 128-value row (128 / group size)
    int64_t n_tokens;
    int64_t num_blocks;
    int64_t host_blocks;         // host-tier blocks: ids num_blocks .. num_blocks + host_blocks - 1
    int n_kv;
};

struct DecodeParams {
    const uint8_t* kv;           // this layer's records (FP8: scales inline after the tiles)
    const uint8_t* stage;        // where the decode reads this layer's host-tier records: their
                                 // staged copy in HBM, or (host_direct) the host records themselves
    int host_direct;             // 1: host-tier blocks are read from host memory by cp.async
    uint8_t* host_kv;            // this layer's host-tier records (device address), or null
    int64_t host_blocks;         // host-tier blocks: ids num_blocks .. num_blocks + host_blocks - 1
    const uint16_t* q;           // bf16 bits [B][n_q][128]
    const uint16_t* k_new;       // fused append: bf16 [B][n_kv][128] new token, or null
    const uint16_t* v_new;
    void* out;                   // [B][n_q][128] output for units that lie in one CTA, or null
    float* lse_out;              // [B][n_q] or null
    int out_f32;
    const int32_t* block_table;  // [B][max_blocks]
    const int32_t* seq_lens;     // [B]
    const uint16_t* retain;      // [num_blocks] or null
    const uint8_t* block_fmt;    // mixed pools: [num_blocks] precision code (KVD_BF16 / _FP8_E4M3 / _FP8_E5M2)
    float* part_o;               // [S + U][g][128]
    float* part_lse;             // [S + U][g]
    int32_t* unit_first;         // [U]
    int32_t* unit_count;         // [U]
    const int32_t* plan;         // a step plan (kvd_decode_plan) in the workspace, or null
    int32_t* dyn;                // dynamic balancing: the plan's piece counter and finished-CTA count,
                                 // or null (each CTA streams its whole range)
    float* logits;               // [B][n_q][logits_stride] or null
    int64_t logits_stride;
    int32_t* err;
    int64_t num_blocks;
    int max_blocks;
    int B;
    int n_kv;
    int g;
    int n_q;
    int nsplit;
    int ng;                      // low-bit pools: groups per 128-value row (1, 2 or 4)
    int max_seq_len;             // host bound on seq_lens (only used to warm L2)
    int early;                   // KVD_EARLY_START: plan and K/V copies before the grid dependency wait
    float scale_log2;            // softmax_scale * log2(e)
};

struct CombineParams {
    const float* part_o;
    const float* part_lse;
    const int32_t* unit_first;
    const int32_t* unit_count;
    void* out;
    float* lse_out;
    int B;
    int n_q;
    int n_kv;
    int g;
    int out_f32;
    int slots_hint;              // expected partials per unit (sizes the combine CTA), 0 = unknown
};

struct ScoreParams {
    const float* logits;
    int64_t logits_stride;
    const float* lse;
    const int32_t* seq_lens;
    float* scores;
    int64_t scores_stride;
    int B;
    int n_q;
    float inv_LH;
};

// Launch `kernel` as a programmatic dependent of the preceding kernel in the stream, with
// a preferred shared-memory carveout (percent of the SM's shared memory) when carveout ≥ 0.
// The kernels of one decode call share the decode kernel's carveout, so an SM moving from
// one to the next keeps its L1/shared-memory split.
template <typename... P>
inline cudaError_t launch_dependent(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, int carveout,
                                    cudaStream_t stream, const P&... params) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (carveout >= 0) {
        attr[1].id = cudaLaunchAttributePreferredSharedMemoryCarveout;
        attr[1].val.sharedMemCarveout = static_cast<unsigned>(carveout);
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kernel, params...);
}

cudaError_t launch_append(const AppendParams& p, int kind, cudaStream_t stream);
constexpr int kMaxPlanBlocks = 16384;   // the plan keeps a request's importances in shared memory

struct TierPlanParams {
    const float* scores;
    int64_t scores_stride;
    const int32_t* seq_lens;
    float* importance;           // [B][max_blocks] or null
    int8_t* tier;                // [B][max_blocks]
    int B;
    int max_blocks;
    int protect_prompt;
    int protect_recent;
    int t1;
};
cudaError_t launch_tier_plan(const TierPlanParams& p, cudaStream_t stream);

struct TierMoveParams {
    const int32_t* from_ids;
    const int32_t* to_ids;
    uint8_t* kv;                 // the whole pool (every layer)
    uint8_t* host_kv;            // the whole host tier (device address), or null
    int32_t* err;
    int64_t num_blocks;
    int64_t host_blocks;
    int64_t record_bytes;
    int n;
    int L;
    int n_kv;
};
cudaError_t launch_tier_move(const TierMoveParams& p, int num_sms, cudaStream_t stream);
// Decode launch geometry and launch for a pool kind (ng: groups per row of a low-bit pool, else 1).
size_t decode_smem_bytes(int kind, int ng, int batch, int g);
int decode_ctas_per_sm(int kind, int ng, int batch, int g);
int decode_carveout(int kind, int ng, int batch, int g);   // percent, for the decode call's launches
cudaError_t launch_decode(const DecodeParams& p, int kind, int carveout, cudaStream_t stream);
// The low-bit kinds' variants (their own translation unit).
size_t decode_smem_bytes_lowbit(int kind, int ng, int batch, int g);
int decode_ctas_per_sm_lowbit(int kind, int ng, int batch, int g);
cudaError_t launch_decode_lowbit(const DecodeParams& p, int kind, int carveout, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, int carveout, cudaStream_t stream);
// The step plan: prefix sums and lengths, and every decode CTA's first batch of blocks.
int64_t decode_plan_words(int batch, int nsplit);
int64_t decode_plan_dyn_off(int batch, int nsplit);
constexpr int kDecodePieces = 5;   // pieces per CTA range with dynamic balancing
cudaError_t launch_plan(const DecodeParams& p, int32_t* plan, cudaStream_t stream);
cudaError_t launch_scores(const ScoreParams& p, cudaStream_t stream);
cudaError_t launch_epilogue(const CombineParams& c, const ScoreParams& sp, int carveout, cudaStream_t stream);
cudaError_t launch_wait_timeout(int32_t* err, int64_t timeout_ns, cudaStream_t stream);

}  // namespace kvd
