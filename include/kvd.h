/*
 * kvd.h — C ABI of the paged GQA decode-attention library for GB300 (sm_103a).
 *
 * One decode step of grouped-query attention over a paged KV cache: every
 * request holds its keys and values in fixed 16-token blocks reached through
 * a per-request block table, the new token's K/V is appended first, and each
 * query head attends softmax(q·Kᵀ/√d_h)·V over the request's context.  Groups
 * of g = n_q / n_kv query heads share one KV head.
 *   Paged blocks, block table, append-then-attend and FP8 storage: page
 *   "LLM에서 KV 캐시는 얼마나 생길까" (froggydisk.github.io/kv-cache-per-request),
 *   sections "KV 캐시란" (q/k/v heads, √128 scaling, prefill/decode append)
 *   and "KV 캐시를 줄이는 기법" (16-token blocks, block tables, FP8 E4M3).
 *   Bytes per token 2·L·n_kv·d_h·w_kv: page "The KV Cache Is the New Memory
 *   Wall" (jaehun.me/posts/paper-2609-30854v1), background (paper §2.1, Tab. 1).
 *   Importance score s_i: page "기술 요약: 모든 사고가 HBM 을 필요로 하는 것은
 *   아님" (gist.science/ko/paper/2605.09490), section "2. 중요도 점수화".
 *
 * Conventions for every entry point
 *  - Device pointers are caller-owned CUDA device memory; the library never
 *    frees them.  The library itself allocates only the pool handle (host) and a
 *    4-byte device error word inside kvd_pool_create.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Calls are asynchronous: the return status covers argument
 *    validation and kernel launch only.
 *  - Kernels never trap.  A problem found on the device (a block id outside
 *    the pool, a sequence length outside [1, max_blocks_per_seq·16], a bounded
 *    wait that ran out) records the first error code in the pool's error word;
 *    the affected work item is treated as empty.  Read it with
 *    kvd_get_device_error.
 *  - Supported set: d_h = 128, block_size = 16, 1 ≤ g ≤ 8, batch ≤ 2048, at most 64 GiB
 *    of pool (and of host tier) per layer.
 *    Anything else valid returns KVD_ERR_UNSUPPORTED before any launch.
 *
 * Pool layout (per layer ℓ, physical block p, KV head h)
 *  - One record per (ℓ, p, h) at byte offset ((ℓ·num_blocks + p)·n_kv + h)·record_bytes:
 *    the K tile, then the V tile (2·16·128 elements), then for FP8 the 32 fp32
 *    scales [2][16] (index 0 = K, 1 = V; last index = slot offset t).
 *    record_bytes = 8192 (BF16) or 4096 + 128 = 4224 (FP8), so one (block, head)
 *    is a single contiguous, 16-byte aligned copy.  A tile holds token t ∈ [0,16)
 *    (slot offset within the block) × dim d ∈ [0,128), permuted into tensor-core
 *    fragment order:
 *      K tile: i = d/16, c = d%16, lane = 4·(t%8) + (c%8)/2,
 *              e = (c%2) + 2·(t/8) + 4·(c/8)
 *      V tile: i = d/16, r = d%16, lane = 4·(r%8) + (t%8)/2,
 *              e = (t%2) + 2·(r/8) + 4·(t/8)
 *      BF16 element index within the tile: (i·32 + lane)·8 + e
 *      FP8  byte index within the tile:   ((i/2)·32 + lane)·16 + (i%2)·8 + e
 *  - The pool is written only through kvd_append_kv.
 *  - A mixed pool (KVD_MIXED) gives every record the BF16 size, 8192 bytes; a block stored
 *    in E4M3 or E5M2 puts the 4224-byte FP8 record (codes of its own format, then the 32
 *    scales) at the start of its slot and leaves the rest unused.
 *  - A low-bit pool (KVD_INT4, KVD_INT2: bits = 4 or 2, group_size G ∈ {32, 64, 128}, NG =
 *    128/G groups per row) has records of 2·(256·bits) + 2·(64·NG) bytes: the K code tile, the
 *    V code tile (16·128 codes each, bits wide), then for K and then for V the table
 *    [16 tokens][NG groups] of 32-bit entries (scale half-precision bits | zero-point bits << 16).
 *    Value = code·scale + zero.  Codes: with P = 8/bits codes per byte, kg = d/(16·P),
 *    h = (d/16) % P (the code sits in bits h·bits of its byte), c = d % 16:
 *      K code of (t, d): lane = 4·(t%8) + (c%8)/2, th = t/8, j = (c%2) + 2·(c/8)
 *      V code of (t, d): lane = 4·(c%8) + (t%8)/2, th = t/8, j = (t%2) + 2·(c/8)
 *      byte index within the tile: (((kg/2)·32 + lane)·4 + (kg%2)·2 + th)·4 + j
 *    so every byte holds codes of one token only.
 *  - An angle-domain pool (KVD_ANGLE) has FP8 records (4224 bytes, same tile layout): the K
 *    tile holds the E4M3 codes of each key row's direction, the V tile FP8 values; of the 32
 *    fp32 words after the tiles, index 0 holds per token the key's logit factor w (not a scale)
 *    and index 1 the V scale.
 */
#ifndef KVD_H
#define KVD_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVD_API __attribute__((visibility("default")))
#else
#define KVD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVD_OK = 0,
    KVD_ERR_INVALID = 1,      /* bad argument: null pointer, negative size, index out of range */
    KVD_ERR_UNSUPPORTED = 2,  /* valid but outside the supported set (see above) */
    KVD_ERR_NOMEM = 3,        /* a caller buffer is smaller than required */
    KVD_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    KVD_ERR_OOB = 5,          /* device-detected: block id or sequence length out of range */
    KVD_ERR_TIMEOUT = 6       /* device-detected: a bounded wait inside a kernel ran out */
} kvd_status;

typedef enum {
    KVD_BF16 = 0,             /* w_kv = 2 bytes */
    KVD_FP8_E4M3 = 1,         /* w_kv = 1 byte, plus a per-(token, KV head) fp32 scale for K and for V */
    KVD_F32 = 2,              /* output only (full-precision check output) */
    KVD_FP8_E5M2 = 3,         /* block format of a mixed pool: like E4M3, codes 1·5·2 bits, max 57,344 */
    KVD_MIXED = 4,            /* pool of mixed-precision blocks (kvd_pool_set_block_formats) */
    KVD_INT4 = 5,             /* w_kv = 1/2: 4-bit codes, half-precision scale and zero point per group */
    KVD_INT2 = 6,             /* w_kv = 1/4: 2-bit codes, likewise */
    KVD_ANGLE = 7             /* angle-domain keys (E4M3 direction code + radius factor), FP8 values */
} kvd_dtype;

typedef struct {
    int32_t num_layers;       /* L */
    int32_t n_kv;             /* KV heads per layer */
    int32_t d_h;              /* head dimension; 128 */
    int32_t block_size;       /* tokens per block; 16 */
    int64_t num_blocks;       /* physical blocks per layer */
    int32_t kv_dtype;         /* KVD_BF16, KVD_FP8_E4M3, KVD_MIXED, KVD_INT4, KVD_INT2 or KVD_ANGLE */
    int32_t group_size;       /* KVD_INT4 / KVD_INT2: values per scale group, 32, 64 or 128; ignored
                                 for the other types */
} kvd_pool_desc;

typedef struct kvd_pool kvd_pool;  /* opaque */

/* Flags of kvd_decode_attn.
 * KVD_EARLY_START: the caller promises that block_table, seq_lens, retain_mask and the pool
 *   contents (all but the slot the fused append writes) are not written by the kernel that
 *   precedes this call in the stream.  The decode kernel, launched as a programmatic
 *   dependent of that kernel, may then plan its split and start copying K/V while that
 *   kernel is still running; reads of q, k_new, v_new and every write still wait for it to
 *   complete.  Without the flag the kernel waits before touching any global memory. */
#define KVD_EARLY_START 1u
/* KVD_PLANNED: the workspace holds a step plan made by kvd_decode_plan for this call's shape
 * (pool, n_q, batch, max_seq_len, num_splits) and for the block_table, seq_lens and retain_mask
 * the call passes, which have not changed since; the decode kernel reads its split and its first
 * blocks from it instead of deriving them.  With the plan the work of a BF16 pool is also balanced
 * at run time: when each split's range holds 192 blocks or more, every CTA streams the first 5/6
 * of its range, and the last sixth of every range is cut into four pieces (1/2, 1/4, 1/8 and the
 * rest of it) that CTAs take from a counter in the plan once their own part is done, the largest
 * first.  A piece's partial does not depend on the CTA that takes it, so results repeat bit for
 * bit.  Calls that share one workspace's plan must not run concurrently. */
#define KVD_PLANNED 2u

/* Optional score epilogue of kvd_decode_attn: adds this layer's share of the cumulative
 * importance score, scores[b][t] += inv_LH · Σ_h α_h[t], exactly as kvd_accum_scores would
 * from the call's logits and final LSE, but inside the call's merge launch. */
typedef struct {
    float* scores;            /* f32 [batch][scores_stride], device, caller-owned, accumulated */
    int64_t scores_stride;    /* ≥ every seq_lens[b] */
    float inv_LH;             /* 1/(L·H): L layers and H = n_q query heads per step */
} kvd_scores_desc;

/* Readable name of a status code (static string). */
KVD_API const char* kvd_status_string(kvd_status s);

/* Bytes of a pool.  kv_bytes = L·num_blocks·n_kv·2·block_size·d_h·w_kv, the closed form
 * 2·L·n_kv·d_h·w_kv bytes per token times num_blocks·block_size tokens (K and V elements
 * only; w_kv = 2, 1, 1/2 or 1/4 for BF16, FP8, INT4, INT2; a mixed pool counts 2); pool_bytes =
 * kv_bytes plus, for FP8, L·num_blocks·n_kv·2·block_size·4 bytes of scales, for INT4 / INT2
 * L·num_blocks·n_kv·2·block_size·(128/group_size)·4 bytes of group scales and zero points:
 * the size of the buffer kvd_pool_create needs.  A low-bit type with a group_size other than
 * 32, 64 or 128 is KVD_ERR_UNSUPPORTED.  Host only.
 * Low-bit pools: page "The KV Cache Is the New Memory Wall", §4.2, §4.6 and Tab. 7 (INT4 and
 * 2-bit KV with group-wise scales, KVQuant, KIVI), §3.2 (2-bit storage raises decode intensity
 * to 2g/w_kv = 64 FLOP/B at g = 8).  The pages give no group layout; this library quantises
 * each group of group_size consecutive dims of a (token, KV head) row, K and V alike:
 * scale = half(fp32((max − min)/(2^bits − 1))) (1 if that is 0), zero = half(min), code =
 * clamp(rint(fp32(fp32(x − zero)/scale)), 0, 2^bits − 1), half() = nearest half-precision
 * value saturated at ±65,504, rint ties to even.  Low-bit pools take no host tier
 * (kvd_pool_attach_host_tier: KVD_ERR_UNSUPPORTED).
 * Angle-domain pools (KVD_ANGLE): page "기술 요약: Spherical KV", §2.1 (Angle-Domain Attention):
 * a key is a radius r = ||k|| and a direction; the cache keeps a quantised radius r̃ and a code of
 * the direction, and the decode kernel computes the logit ||q||·r̃·f_b(c_q, c_k) from the codes,
 * f_b the cosine of two direction codes, without rebuilding a dense key.  The page defines
 * neither the code nor f_b; this library takes the E4M3 codes of the row at its absmax scale as
 * the direction code (they do not depend on ||k||), r̃ = the nearest half-precision value of
 * ||k|| (saturating), and f_b = <d_q, d_k>/(||d_q||·||d_k||) with d the code values.  Each key row
 * stores w = fp32(r̃/||d_k||) (computed in fp64; 0 for a zero row) where an FP8 record keeps its
 * K scale; values are FP8-E4M3 as in an FP8 pool.  The query of each head is coded the same way
 * inside kvd_decode_attn.  pool_bytes as for FP8.  No host tier. */
KVD_API kvd_status kvd_pool_bytes(const kvd_pool_desc* desc, size_t* pool_bytes, size_t* kv_bytes);

/* Wrap caller memory as a pool.  mem is a device buffer of len ≥ pool_bytes bytes,
 * 16-byte aligned (else KVD_ERR_NOMEM / KVD_ERR_INVALID).  Allocates the handle and a
 * 4-byte device error word on the current device (KVD_ERR_CUDA if that fails).  *out is
 * set on success. */
KVD_API kvd_status kvd_pool_create(const kvd_pool_desc* desc, void* mem, size_t len, kvd_pool** out);

/* Free the handle and its error word (not the caller's pool memory).  NULL is a no-op. */
KVD_API void kvd_pool_destroy(kvd_pool* pool);

/* Mixed-precision pool, tier-homogeneous pages.  Page "The KV Cache Is the New Memory Wall",
 * §5.5 (first open direction): one paged layout that carries a precision per block next to its
 * retention mask; page "기술 요약: Spherical KV", §2.2 (tier-homogeneous pages): every entry of
 * a page shares one precision tier, so the decode kernel reads a page in a single pass guided
 * by its header.  A pool created with kv_dtype = KVD_MIXED stores physical block p in the
 * format block_fmt[p]: KVD_BF16 (values), KVD_FP8_E4M3 or KVD_FP8_E5M2 (codes with a
 * per-(token, KV head) fp32 scale for K and for V; scale = fp32(absmax/top), top = 448 or
 * 57,344, code = round to nearest even, saturating, of the fp32 quotient x/scale).  The
 * decode kernel reads a block's precision byte beside its retain bits and copies 8192 or 4224
 * bytes.  block_fmt: uint8 [count ≥ num_blocks], device, caller-owned, read by every later
 * kvd_append_kv and kvd_decode_attn of the pool (for every layer); change a block's format
 * only while it holds no token.  A byte that is none of the three codes makes the block's
 * tokens skipped (append) or treated as empty (decode) with KVD_ERR_OOB in the error word.
 * KVD_ERR_INVALID for a pool that is not mixed, a NULL array or count < num_blocks.  A mixed
 * pool takes no host tier (kvd_pool_attach_host_tier: KVD_ERR_UNSUPPORTED). */
KVD_API kvd_status kvd_pool_set_block_formats(kvd_pool* pool, const uint8_t* block_fmt, int64_t count);

/* Host tier (T1) of a pool.  Page "기술 요약: 모든 사고가 HBM 을 필요로 하는 것은 아님",
 * section "1. 4 단계 분류": mid-importance tokens (tier T1) live at full precision in host
 * memory and are brought to the GPU before every attention step; section "3. 제로-근사오차
 * 오프로딩", Prop. 1: the attention output does not depend on how tokens are split between
 * HBM (T0) and host memory (T1).
 * A pool with a host tier has host_blocks more physical blocks, ids num_blocks ..
 * num_blocks + host_blocks - 1, whose records (same record layout; per layer ℓ the record of
 * host block i, head h sits at ((ℓ·host_blocks + i)·n_kv + h)·record_bytes) live in pinned
 * host memory.  Two ways to bring them to the GPU:
 *  - direct (attached without staging memory): the decode kernel copies each host-tier
 *    block it attends straight from host memory into shared memory, over the host link,
 *    while it streams the HBM blocks; nothing else is needed per step.
 *  - staged: kvd_tier_prefetch copies one layer's host records into one of two HBM staging
 *    slots (slot layer % 2); kvd_decode_attn reads a host-tier block from that staged copy,
 *    so the staged layer must be the one attended.
 * A retain_mask then has num_blocks + host_blocks entries.  Block tables may mix both kinds
 * of ids freely.  Mixed pools (KVD_MIXED) have no host tier. */

/* host_bytes = L·host_blocks·n_kv·record_bytes (pinned host memory); staging_bytes =
 * 2·host_blocks·n_kv·record_bytes (device).  host_blocks ≥ 0.  Host only. */
KVD_API kvd_status kvd_tier_bytes(const kvd_pool_desc* desc, int64_t host_blocks, size_t* host_bytes,
                                  size_t* staging_bytes);

/* Give the pool a host tier of host_blocks blocks (0 removes it).  host_mem: host memory the
 * device can address — page-locked (cudaHostAlloc or registered), or on systems where the
 * device reads pageable memory any host memory — 16-byte aligned, ≥ host_bytes; its device
 * address is looked up here (KVD_ERR_INVALID if there is none).  staging_mem: device,
 * 16-byte aligned, ≥ staging_bytes; or NULL with staging_len = 0 for direct reads.  Both stay
 * caller-owned; the host records are written by kvd_append_kv (slots in host blocks) and by
 * the fused append of kvd_decode_attn. */
KVD_API kvd_status kvd_pool_attach_host_tier(kvd_pool* pool, void* host_mem, size_t host_len, void* staging_mem,
                                             size_t staging_len, int64_t host_blocks);

/* Copy layer's host-tier records into staging slot layer % 2 (host_blocks·n_kv·record_bytes
 * bytes over the host link, one asynchronous DMA on a copy engine, so that it overlaps a
 * decode kernel running on another stream) on `stream`.  It must complete before a kvd_decode_attn of that
 * layer reads a host-tier block (same stream, or an event), and a slot is refilled two layers
 * later, so the prefetch of layer ℓ+2 must wait for the attention of layer ℓ.  A no-op
 * without a host tier or with direct reads. */
KVD_API kvd_status kvd_tier_prefetch(kvd_pool* pool, int layer, void* stream);

/* Tier plan from the cumulative importance scores (same page, section "4. 시스템 구현":
 * tiers are reassigned every Δ = 64 decode steps; section "1. 4 단계 분류": protected
 * tokens — prompt, attention sinks, recent window — and the most important ones stay in HBM,
 * mid-importance ones go to host memory).  For request b with seq_lens[b] = len and
 * nb = ⌈len/16⌉ logical blocks (nb = 0 for a length outside [1, max_blocks_per_seq·16]):
 *   importance[b][j] = Σ_{o=0..15, 16j+o < len} scores[b][16j+o], added in that order in fp32
 *   (positions at or past scores_stride count 0);
 *   block j is protected if it holds a position < protect_prompt or ≥ len - protect_recent;
 *   tier[b][j] = 1 (host tier) for the t1_blocks unprotected blocks of smallest
 *   (importance, j) — all unprotected blocks if there are fewer — else 0; tier[b][j] = -1
 *   for j ≥ nb.  Evicted slots (tier T3, the retain mask) carry score 0 and are not treated
 *   specially.
 *  scores      f32 [batch][scores_stride], device (as accumulated by kvd_accum_scores)
 *  importance  f32 [batch][max_blocks_per_seq] out (0 for j ≥ nb), or NULL
 *  tier        int8 [batch][max_blocks_per_seq] out, device
 * Moving the blocks (kvd_tier_move) and patching the block tables is the caller's: only
 * blocks whose tier changed need to move.  Needs max_blocks_per_seq ≤ 16384
 * (KVD_ERR_UNSUPPORTED otherwise); one CTA per request, work O(nb).  Scores must be finite
 * (a NaN has no place in the order).  Negative protect_*,
 * t1_blocks or batch, scores_stride < 1 or max_blocks_per_seq < 1: KVD_ERR_INVALID; batch = 0
 * is a no-op. */
KVD_API kvd_status kvd_tier_plan(const float* scores, int64_t scores_stride, const int32_t* seq_lens, int batch,
                                 int max_blocks_per_seq, int protect_prompt, int protect_recent, int t1_blocks,
                                 float* importance, int8_t* tier, void* stream);

/* Copy every layer's and KV head's record of physical block from_ids[i] to physical block
 * to_ids[i], i < n (int32 device arrays; ids of either tier).  No block may be both a source
 * and a destination of the same call.  An id outside the pool and its host tier sets
 * KVD_ERR_OOB on the device and that pair is skipped. */
KVD_API kvd_status kvd_tier_move(kvd_pool* pool, const int32_t* from_ids, const int32_t* to_ids, int n,
                                 void* stream);

/* One tier reassignment, on the host (same page, section "4. 시스템 구현": only blocks whose
 * tier changed move).  For request b and logical block j with tier[b][j] ≥ 0, the block's
 * current id p = block_table[b][j] is a host-tier id when p ≥ num_blocks.  Where that differs
 * from tier[b][j] = 1, the last id of the planned tier's free list becomes its destination d:
 * block_table[b][j] = d, the pair (p, d) is appended to from_ids/to_ids, and, with a retain
 * mask, retain_mask[d] = retain_mask[p].  A block id shared by several table entries moves
 * once and every entry follows it (the first entry's plan decides).  Once all destinations
 * are taken, each source id is appended to its own tier's free list.  Entries with tier < 0
 * are left alone.  num_blocks, host_blocks: the pool's (ids num_blocks .. + host_blocks - 1
 * are host-tier ids).
 *  tier          int8 [batch][max_blocks_per_seq] (kvd_tier_plan's output copied to the host)
 *  block_table   int32 [batch][max_blocks_per_seq], in/out
 *  hbm_free      int32, capacity num_blocks, the first *hbm_free_n entries free pool ids (in/out)
 *  host_free     int32, capacity host_blocks, the first *host_free_n entries free host-tier ids
 *  retain_mask   uint16 [num_blocks + host_blocks] or NULL (in/out)
 *  from_ids, to_ids  int32 [batch·max_blocks_per_seq] out; *n_moves out
 * All host memory.  Afterwards the caller copies block_table (and retain_mask) to the device
 * and runs kvd_tier_move(from_ids, to_ids) on the stream before the next decode.  A block whose
 * planned tier has no free id stays where it is (KVD_ERR_NOMEM once the rest is done); a table
 * id outside the pool and its host tier is skipped (KVD_ERR_OOB likewise); a free list holding
 * an id of the other tier, or more ids than its tier has, is KVD_ERR_INVALID.  Host only, no
 * GPU needed. */
KVD_API kvd_status kvd_tier_reassign(int64_t num_blocks, int64_t host_blocks, const int8_t* tier,
                                     int32_t* block_table, int batch, int max_blocks_per_seq, int32_t* hbm_free,
                                     int32_t* hbm_free_n, int32_t* host_free, int32_t* host_free_n,
                                     uint16_t* retain_mask, int32_t* from_ids, int32_t* to_ids, int32_t* n_moves);

/* Decode-step append ("reshape and cache").  Page "LLM에서 KV 캐시는 얼마나 생길까", section
 * "KV 캐시란": every decode step writes the new token's K and V into the cache before its
 * attention; section "KV 캐시를 줄이는 기법": the cache lives in fixed 16-token blocks, and FP8
 * E4M3 storage divides a value by a scale before rounding and multiplies it back on read.
 * Token n's keys k_new[n][h][:] and values
 * v_new[n][h][:] (bf16, [n_tokens][n_kv][d_h], device) are written for every KV head h of
 * `layer` at slot s = slot_mapping[n] (int64, device) = physical_block·16 + offset;
 * s < 0 skips the token.  FP8 pools store per (token, head) and separately for K and V:
 * scale = fp32(absmax/448) (1 when the row is zero), code = e4m3 round-to-nearest-even,
 * saturating, of the fp32 quotient x/scale.  n_tokens = 0 is a no-op.  A slot in a host-tier
 * block writes that block's host record (with a staged host tier, before that layer's
 * kvd_tier_prefetch: the staged copy is not updated).  A slot beyond the pool (and its host tier) sets
 * KVD_ERR_OOB on the device and that token is skipped. */
KVD_API kvd_status kvd_append_kv(kvd_pool* pool, int layer, const void* k_new, const void* v_new,
                         const int64_t* slot_mapping, int n_tokens, void* stream);

/* The split plan: number of KV splits (CTAs) kvd_decode_attn uses for this shape when
 * num_splits = 0, and the workspace bytes it needs.  Host only (queries the device's SM
 * count and the kernel's occupancy through the pool's device). */
KVD_API kvd_status kvd_decode_workspace_bytes(const kvd_pool* pool, int n_q, int batch, int max_seq_len,
                                      int num_splits, int* splits_out, size_t* bytes_out);

/* Paged GQA decode attention for one layer (the decode kernel, then the split merge).
 * Page "LLM에서 KV 캐시는 얼마나 생길까", section "KV 캐시란": a query head scores every cached
 * key, q·kᵀ/√128, takes the softmax and sums the values, and several query heads share one
 * KV head (GQA); section "KV 캐시를 줄이는 기법": the kernel follows the request's block table
 * to blocks scattered anywhere in the pool.  Page "The KV Cache Is the New Memory Wall", §3.2:
 * at decode this is a stream of the whole cache at about g FLOP per byte, bound by memory
 * bandwidth.  Page "기술 요약: 모든 사고가 HBM 을 필요로 하는 것은 아님", section "3.
 * 제로-근사오차 오프로딩": an evicted token is left out of the softmax (the retain mask).
 *  q            bf16 [batch][n_q][d_h], device
 *  k_new, v_new bf16 [batch][n_kv][d_h] or both NULL: the fused decode-step append.  The
 *               token at position seq_lens[b]-1 of request b — slot
 *               block_table[b][(len-1)/16]·16 + (len-1)%16 — is written into the pool (FP8
 *               quantised as kvd_append_kv does) by the CTA that attends that block, before
 *               it reads it.  That block must not be shared with another request of the call.
 *               A host-tier block gets the token in its host record (and, staged, in its
 *               staged copy).
 *  block_table  int32 [batch][max_blocks_per_seq], device; entry j of request b is the
 *               physical block of its logical block j (entries past the context unread)
 *  seq_lens     int32 [batch], device; positions 0 .. seq_lens[b]-1 are attended (the
 *               append of this step included); must be in [1, max_blocks_per_seq·16]
 *  max_seq_len  host upper bound on seq_lens, used only for the split plan
 *  num_splits   0 = automatic; else the number of KV splits: the flattened sequence of
 *               (request, KV head, block) work is cut into num_splits equal contiguous
 *               ranges, one CTA each (with KVD_PLANNED a BF16 pool's long ranges are also
 *               balanced at run time, see KVD_PLANNED); partial results are merged by
 *               log-sum-exp (a unit that lies inside one piece is finished directly)
 *  retain_mask  uint16 [num_blocks + host_blocks] or NULL; bit o of retain_mask[p] clear =
 *               slot o of physical block p is evicted (logit −inf, weight 0) in every layer
 *  softmax_scale  multiplies q·k (1/√d_h for the plain definition)
 *  workspace    device scratch of workspace_bytes ≥ kvd_decode_workspace_bytes, no
 *               initialisation needed; layout: part_o f32 [U + P·S][g][d_h], part_lse f32
 *               [U + P·S][g], unit_first int32 [U], unit_count int32 [U] (−1 = output already
 *               final; a unit's partials are slots unit_first .. unit_first + count − 1), then,
 *               with KVD_PLANNED, the step plan region (kvd_decode_plan), each region on a
 *               256-byte boundary (U = batch·n_kv, S splits, P = 5 pieces a split with
 *               KVD_PLANNED, else 1; kvd_decode_workspace_bytes reports the planned size)
 *  out          [batch][n_q][d_h] in out_dtype (KVD_BF16 rounds to nearest even, or KVD_F32);
 *               NULL = write only the partials and unit tables into the workspace (merge
 *               them later with kvd_combine_splits; lse_out is then unused)
 *  lse_out      f32 [batch][n_q] natural-log log-sum-exp of the logits, or NULL
 *  logits_out   f32 [batch][n_q][logits_stride] or NULL: the scaled logit q·k·scale of
 *               every attended position (−inf where evicted), input of kvd_accum_scores
 *  scores_epilogue  NULL, or the score update to fuse into the merge launch (needs out,
 *               lse_out and logits_out, else KVD_ERR_INVALID; n_q ≤ 256)
 *  flags        0, KVD_EARLY_START and / or KVD_PLANNED (see above); other bits are KVD_ERR_INVALID
 * Query head h reads KV head h / g.  A head with no retained position gets out = 0 and
 * lse = −inf. */
KVD_API kvd_status kvd_decode_attn(kvd_pool* pool, int layer, const void* q, int n_q,
                           const void* k_new, const void* v_new,
                           const int32_t* block_table, int max_blocks_per_seq,
                           const int32_t* seq_lens, int batch, int max_seq_len, int num_splits,
                           const uint16_t* retain_mask, float softmax_scale,
                           void* workspace, size_t workspace_bytes,
                           void* out, int out_dtype, float* lse_out,
                           float* logits_out, int64_t logits_stride,
                           const kvd_scores_desc* scores_epilogue, unsigned flags, void* stream);

/* Size of the fixed device scratch array used by kvd_decode_attn_noalloc: 16 MiB, held on
 * every GPU that loads the library until the process exits. */
#define KVD_NOALLOC_SCRATCH_BYTES (16u << 20)

/* kvd_decode_attn for callers that may not allocate device memory (for example a host
 * framework whose own allocator owns all device memory, or a latency-critical loop that
 * cannot take cudaMalloc's implicit synchronisation).  The pages describe no such entry
 * point; it has no counterpart in them.
 * Same arguments and results as kvd_decode_attn, minus the workspace: the split partials
 * go to a file-scope device array of KVD_NOALLOC_SCRATCH_BYTES bytes inside the library.
 * It allocates nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *  - A shape whose unplanned workspace (kvd_decode_attn's layout without KVD_PLANNED, at most
 *    kvd_decode_workspace_bytes) exceeds KVD_NOALLOC_SCRATCH_BYTES
 *    is rejected with KVD_ERR_NOMEM before any launch; `out` may not be NULL; KVD_PLANNED is
 *    KVD_ERR_INVALID (no step plan can have been made in the library's array).
 *  - The current device must be the pool's device (else KVD_ERR_INVALID).  The first call on
 *    a device, with that device current, looks up the array's device address
 *    (cudaGetSymbolAddress) once for that device and keeps it for the lifetime of the
 *    device's primary context: make that first call before any stream capture begins, and
 *    do not call this entry point again in a process that has reset the device
 *    (cudaDeviceReset) after its first call there.
 *  - Every call on a device shares the one array, and it keeps the previous call's
 *    contents; every partial and unit-table entry is written before it is read, so nothing
 *    needs clearing.  Calls whose kernels overlap on the GPU (e.g. on two streams at once)
 *    race on the array: serialise them. */
KVD_API kvd_status kvd_decode_attn_noalloc(kvd_pool* pool, int layer, const void* q, int n_q,
                                           const void* k_new, const void* v_new,
                                           const int32_t* block_table, int max_blocks_per_seq,
                                           const int32_t* seq_lens, int batch, int max_seq_len, int num_splits,
                                           const uint16_t* retain_mask, float softmax_scale,
                                           void* out, int out_dtype, float* lse_out,
                                           float* logits_out, int64_t logits_stride,
                                           const kvd_scores_desc* scores_epilogue, unsigned flags,
                                           void* stream);

/* The step plan, for the layers of one decode step that share block tables and lengths.  The
 * pages describe no split plan; this is an entry point of the library's own design.  Writes into
 * the workspace's plan region (same workspace as the step's kvd_decode_attn calls, sized by
 * kvd_decode_workspace_bytes) the per-request block counts' prefix sums and lengths, and, for each
 * of the split count's CTAs, the physical ids and valid-slot masks of the first 32 blocks it will
 * attend; kvd_decode_attn with KVD_PLANNED then starts copying K/V after one read of the plan
 * instead of three dependent reads (lengths, block table, retain mask) per layer.  Arguments as
 * kvd_decode_attn's; the plan stays valid while block_table, seq_lens, retain_mask (and a mixed
 * pool's formats) are unchanged, for any layer of the pool.  Its kernel does not release a
 * following launch before it completes, so the next kvd_decode_attn may pass KVD_EARLY_START.
 * It also zeroes the two counters of the run-time balancing (each planned launch leaves them at
 * zero again).  Bad lengths and block ids are reported on the device as kvd_decode_attn reports
 * them. */
KVD_API kvd_status kvd_decode_plan(kvd_pool* pool, int n_q, const int32_t* block_table, int max_blocks_per_seq,
                                   const int32_t* seq_lens, int batch, int max_seq_len, int num_splits,
                                   const uint16_t* retain_mask, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* Merge split partials by log-sum-exp.  The pages describe no split of a request's context
 * across CTAs; this is the exact identity for the softmax over a union of disjoint position
 * sets, each summarised by its normalised output o_s and its log-sum-exp lse_s.
 * For unit u = b·n_kv + h/g and head h:
 * LSE = log Σ_s exp(lse_s), out = Σ_s exp(lse_s − LSE)·o_s over the unit_count[u] slots
 * starting at unit_first[u] of part_o f32 [slots][g][d_h] and part_lse f32 [slots][g]
 * (device).  Slots with lse = −inf are skipped; a unit with none (or count 0) yields
 * out = 0, lse = −inf; a unit with count < 0 is left untouched (already final).  out in
 * out_dtype (KVD_BF16 or KVD_F32), lse_out may be NULL. */
KVD_API kvd_status kvd_combine_splits(const float* part_o, const float* part_lse,
                              const int32_t* unit_first, const int32_t* unit_count,
                              int batch, int n_q, int n_kv, int d_h,
                              void* out, int out_dtype, float* lse_out, void* stream);

/* Score epilogue.  Page "기술 요약: 모든 사고가 HBM 을 필요로 하는 것은 아님", section
 * "2. 중요도 점수화": a token's importance s_i accumulates, every decode step, its attention
 * weight averaged over the heads H and the layers L.
 * scores[b][t] += inv_LH · Σ_h exp(logits[b][h][t] − lse[b][h]) for
 * t < seq_lens[b], i.e. this layer's share (1/(L·H))·Σ_h α_h[t] of the cumulative
 * importance score update.  logits f32 [batch][n_q][logits_stride], lse f32 [batch][n_q]
 * (both as written by kvd_decode_attn), scores f32 [batch][scores_stride]; all device.
 * Heads with lse = −inf add nothing. */
KVD_API kvd_status kvd_accum_scores(const float* logits, int64_t logits_stride, const float* lse,
                            const int32_t* seq_lens, int batch, int n_q, float inv_LH,
                            float* scores, int64_t scores_stride, void* stream);

/* Synchronise `stream`, return the pool's device error word in *code (KVD_OK if none) and
 * clear it. */
KVD_API kvd_status kvd_get_device_error(kvd_pool* pool, void* stream, int32_t* code);

/* Self-test of the bounded wait: launches one CTA that waits on an mbarrier nothing will
 * complete, with a limit of timeout_ns nanoseconds; the kernel then records
 * KVD_ERR_TIMEOUT in the pool's error word and returns.  Lets a caller check that device
 * waits give up and report instead of hanging. */
KVD_API kvd_status kvd_selftest_wait_timeout(kvd_pool* pool, int64_t timeout_ns, void* stream);

/* Measurement helper, not part of the method (the pages have no counterpart): reads every
 * byte of the device buffer buf (bytes > 0, a multiple of 16, 16-byte aligned) once with
 * 16-byte streaming loads, on `stream`, one CTA per resident slot of every SM, and writes one
 * 32-bit fold per CTA into sink (device, 4-byte aligned).  It gives the read-only HBM
 * bandwidth a decode kernel, which only reads, is compared with.  KVD_ERR_NOMEM if sink_bytes
 * is smaller than 4 bytes per CTA (4·SMs·resident CTAs ≤ 32 KiB on any current GPU). */
KVD_API kvd_status kvd_measure_read_stream(const void* buf, size_t bytes, void* sink, size_t sink_bytes,
                                           void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVD_H */
