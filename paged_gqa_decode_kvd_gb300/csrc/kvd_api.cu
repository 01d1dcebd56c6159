// kvd_api.cu — the exported C ABI: argument checks, split plan, launches, error word.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <new>

#include "../../include/kvd.h"
#include "kvd_common.cuh"
#include "kvd_internal.h"

struct kvd_pool {
    kvd_pool_desc desc;
    uint8_t* mem;
    int32_t* err;       // device error word
    int device;
    int num_sms;
    size_t layer_bytes;
    // host tier (T1): records in pinned host memory (device address) and two HBM staging slots
    uint8_t* host_kv;      // device address of the host records
    uint8_t* host_mem;     // the same records' host address (the prefetch's DMA source)
    uint8_t* staging;
    int64_t host_blocks;
    size_t host_layer_bytes;
    int host_direct;       // no staging: the decode kernel reads host records over the host link
    // mixed pools: precision code of every physical block (device, caller-owned)
    const uint8_t* block_fmt;
    int64_t block_fmt_count;
};

namespace {

constexpr int kMinBlocksPerSplit = 16;  // smallest per-CTA share the planner creates

bool mul_ok(size_t a, size_t b, size_t* out) {
    if (a != 0 && b > SIZE_MAX / a) return false;
    *out = a * b;
    return true;
}

kvd_status check_desc(const kvd_pool_desc* d) {
    if (!d) return KVD_ERR_INVALID;
    if (d->num_layers < 1 || d->n_kv < 1 || d->num_blocks < 1 || d->d_h < 1 || d->block_size < 1)
        return KVD_ERR_INVALID;
    if (d->kv_dtype != KVD_BF16 && d->kv_dtype != KVD_FP8_E4M3 && d->kv_dtype != KVD_MIXED &&
        d->kv_dtype != KVD_INT4 && d->kv_dtype != KVD_INT2 && d->kv_dtype != KVD_ANGLE)
        return KVD_ERR_INVALID;
    if (d->d_h != kvd::kDh || d->block_size != kvd::kBs) return KVD_ERR_UNSUPPORTED;
    if ((d->kv_dtype == KVD_INT4 || d->kv_dtype == KVD_INT2) && d->group_size != 32 && d->group_size != 64 &&
        d->group_size != 128)
        return KVD_ERR_UNSUPPORTED;
    return KVD_OK;
}

bool lowbit_dtype(int32_t t) { return t == KVD_INT4 || t == KVD_INT2; }

// Groups per 128-value row of a low-bit pool (1 otherwise).
int pool_ng(const kvd_pool_desc* d) { return lowbit_dtype(d->kv_dtype) ? kvd::kDh / d->group_size : 1; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
    size_t part_o, part_lse, unit_first, unit_count, plan, total;
};

// The workspace of a call: a partial slot per (unit, piece), a range being one piece, or with a
// step plan (run-time balancing) kDecodePieces; then the unit tables and, for a planned call,
// the plan.  kvd_decode_workspace_bytes reports the planned size, which serves both.
WsLayout ws_layout(int units, int nsplit, int g, int batch, bool planned) {
    WsLayout w;
    const size_t slots = static_cast<size_t>(units) + static_cast<size_t>(nsplit) * (planned ? kvd::kDecodePieces : 1);
    size_t o = 0;
    w.part_o = o;
    o = align256(o + slots * g * kvd::kDh * sizeof(float));
    w.part_lse = o;
    o = align256(o + slots * g * sizeof(float));
    w.unit_first = o;
    o = align256(o + static_cast<size_t>(units) * sizeof(int32_t));
    w.unit_count = o;
    o = align256(o + static_cast<size_t>(units) * sizeof(int32_t));
    w.plan = o;
    if (planned) o = align256(o + static_cast<size_t>(kvd::decode_plan_words(batch, nsplit)) * sizeof(int32_t));
    w.total = o;
    return w;
}

// Split count: enough CTAs to fill every SM at the kernel's occupancy, but no CTA
// with fewer than kMinBlocksPerSplit blocks of the (upper-bound) total work.
int pool_kind(const kvd_pool* pool);

int plan_splits(const kvd_pool* pool, int batch, int max_seq_len, int g) {
    const int64_t nblk = (static_cast<int64_t>(max_seq_len) + kvd::kBs - 1) / kvd::kBs;
    const int64_t total = nblk * batch * pool->desc.n_kv;
    const int64_t by_work = (total + kMinBlocksPerSplit - 1) / kMinBlocksPerSplit;
    const int64_t by_sms =
        static_cast<int64_t>(pool->num_sms) * kvd::decode_ctas_per_sm(pool_kind(pool), pool_ng(&pool->desc), batch, g);
    int64_t s = by_work < by_sms ? by_work : by_sms;
    return static_cast<int>(s < 1 ? 1 : s);
}

kvd_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVD_OK : KVD_ERR_CUDA; }

int pool_kind(const kvd_pool* pool) {
    switch (pool->desc.kv_dtype) {
        case KVD_FP8_E4M3: return kvd::kKindFp8;
        case KVD_MIXED: return kvd::kKindMixed;
        case KVD_INT4: return kvd::kKindInt4;
        case KVD_INT2: return kvd::kKindInt2;
        case KVD_ANGLE: return kvd::kKindAngle;
        default: return kvd::kKindBf16;
    }
}

// Bytes of one (layer, block, KV head) record slot.
size_t record_bytes(const kvd_pool_desc* d) {
    if (d->kv_dtype == KVD_INT4) return kvd::lowbit_record_bytes(4, pool_ng(d));
    if (d->kv_dtype == KVD_INT2) return kvd::lowbit_record_bytes(2, pool_ng(d));
    return d->kv_dtype == KVD_FP8_E4M3 || d->kv_dtype == KVD_ANGLE ? kvd::kRecordFp8 : kvd::kRecordBf16;
}

}  // namespace

int kvd::pool_device(const kvd_pool* pool) { return pool ? pool->device : -1; }

extern "C" {

const char* kvd_status_string(kvd_status s) {
    switch (s) {
        case KVD_OK: return "ok";
        case KVD_ERR_INVALID: return "invalid argument";
        case KVD_ERR_UNSUPPORTED: return "unsupported shape or type";
        case KVD_ERR_NOMEM: return "buffer too small";
        case KVD_ERR_CUDA: return "CUDA error";
        case KVD_ERR_OOB: return "device-detected index out of range";
        case KVD_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

kvd_status kvd_pool_bytes(const kvd_pool_desc* desc, size_t* pool_bytes, size_t* kv_bytes) {
    kvd_status st = check_desc(desc);
    if (st != KVD_OK) return st;
    if (!kv_bytes || !pool_bytes) return KVD_ERR_INVALID;
    // a mixed pool sizes every record slot for BF16 (an 8-bit block uses the first part of it);
    // element bits: 16, 8, 4 or 2
    const bool fp8_records = desc->kv_dtype == KVD_FP8_E4M3 || desc->kv_dtype == KVD_ANGLE;
    const size_t bits = fp8_records ? 8 : desc->kv_dtype == KVD_INT4 ? 4
                        : desc->kv_dtype == KVD_INT2   ? 2 : 16;
    size_t per_block = 0, rows = 0, total = 0;
    // 2 (K and V) · block_size · d_h · w_kv bytes per (layer, block, KV head)
    if (!mul_ok(2 * static_cast<size_t>(desc->block_size) * desc->d_h, bits, &per_block)) return KVD_ERR_INVALID;
    per_block /= 8;
    if (!mul_ok(static_cast<size_t>(desc->num_layers), static_cast<size_t>(desc->num_blocks), &rows)) return KVD_ERR_INVALID;
    if (!mul_ok(rows, static_cast<size_t>(desc->n_kv), &rows)) return KVD_ERR_INVALID;
    if (!mul_ok(rows, per_block, &total)) return KVD_ERR_INVALID;
    *kv_bytes = total;
    *pool_bytes = total;
    if (lowbit_dtype(desc->kv_dtype)) {   // a (scale, zero) word per (token, group) for K and for V
        size_t mb = 0;
        if (!mul_ok(rows, 2 * static_cast<size_t>(desc->block_size) * pool_ng(desc) * 4, &mb)) return KVD_ERR_INVALID;
        if (total > SIZE_MAX - mb) return KVD_ERR_INVALID;
        *pool_bytes = total + mb;
    }
    if (fp8_records) {   // one fp32 word per (token, head) for K and for V
        size_t sb = 0;
        if (!mul_ok(rows, 2 * static_cast<size_t>(desc->block_size) * sizeof(float), &sb)) return KVD_ERR_INVALID;
        if (total > SIZE_MAX - sb) return KVD_ERR_INVALID;
        *pool_bytes = total + sb;
    }
    return KVD_OK;
}

kvd_status kvd_pool_create(const kvd_pool_desc* desc, void* mem, size_t len, kvd_pool** out) {
    if (!out) return KVD_ERR_INVALID;
    *out = nullptr;
    size_t need = 0, kv = 0;
    kvd_status st = kvd_pool_bytes(desc, &need, &kv);
    if (st != KVD_OK) return st;
    if (!mem || !aligned16(mem)) return KVD_ERR_INVALID;
    if (len < need) return KVD_ERR_NOMEM;
    kvd_pool* p = new (std::nothrow) kvd_pool;
    if (!p) return KVD_ERR_NOMEM;
    p->desc = *desc;
    p->mem = static_cast<uint8_t*>(mem);
    p->layer_bytes = need / desc->num_layers;
    p->err = nullptr;
    p->host_kv = nullptr;
    p->host_mem = nullptr;
    p->staging = nullptr;
    p->host_blocks = 0;
    p->host_layer_bytes = 0;
    p->host_direct = 0;
    p->block_fmt = nullptr;
    p->block_fmt_count = 0;
    const size_t state_bytes = sizeof(int32_t);
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess ||
        cudaMalloc(&p->err, state_bytes) != cudaSuccess || cudaMemset(p->err, 0, state_bytes) != cudaSuccess) {
        if (p->err) cudaFree(p->err);
        delete p;
        cudaGetLastError();
        return KVD_ERR_CUDA;
    }
    *out = p;
    return KVD_OK;
}

kvd_status kvd_tier_bytes(const kvd_pool_desc* desc, int64_t host_blocks, size_t* host_bytes, size_t* staging_bytes) {
    kvd_status st = check_desc(desc);
    if (st != KVD_OK) return st;
    if (host_blocks < 0 || !host_bytes || !staging_bytes) return KVD_ERR_INVALID;
    const size_t rec = record_bytes(desc);
    size_t layer = 0, all = 0;
    if (!mul_ok(static_cast<size_t>(host_blocks), static_cast<size_t>(desc->n_kv), &layer)) return KVD_ERR_INVALID;
    if (!mul_ok(layer, rec, &layer)) return KVD_ERR_INVALID;
    if (!mul_ok(layer, static_cast<size_t>(desc->num_layers), &all)) return KVD_ERR_INVALID;
    *host_bytes = all;
    *staging_bytes = 2 * layer;
    return KVD_OK;
}

kvd_status kvd_pool_set_block_formats(kvd_pool* pool, const uint8_t* block_fmt, int64_t count) {
    if (!pool || pool->desc.kv_dtype != KVD_MIXED || !block_fmt || count < pool->desc.num_blocks)
        return KVD_ERR_INVALID;
    pool->block_fmt = block_fmt;
    pool->block_fmt_count = count;
    return KVD_OK;
}

kvd_status kvd_pool_attach_host_tier(kvd_pool* pool, void* host_mem, size_t host_len, void* staging_mem,
                                     size_t staging_len, int64_t host_blocks) {
    if (!pool || host_blocks < 0) return KVD_ERR_INVALID;
    if ((pool->desc.kv_dtype == KVD_MIXED || pool->desc.kv_dtype == KVD_ANGLE || lowbit_dtype(pool->desc.kv_dtype)) &&
        host_blocks > 0)
        return KVD_ERR_UNSUPPORTED;
    if (host_blocks == 0) {
        pool->host_kv = nullptr;
        pool->host_mem = nullptr;
        pool->staging = nullptr;
        pool->host_blocks = 0;
        pool->host_layer_bytes = 0;
        pool->host_direct = 0;
        return KVD_OK;
    }
    size_t need_host = 0, need_stage = 0;
    kvd_status st = kvd_tier_bytes(&pool->desc, host_blocks, &need_host, &need_stage);
    if (st != KVD_OK) return st;
    const bool direct = !staging_mem && staging_len == 0;
    if (!host_mem || !aligned16(host_mem) || (!direct && (!staging_mem || !aligned16(staging_mem))))
        return KVD_ERR_INVALID;
    if (host_len < need_host || (!direct && staging_len < need_stage)) return KVD_ERR_NOMEM;
    void* dev = nullptr;
    if (cudaHostGetDevicePointer(&dev, host_mem, 0) != cudaSuccess || !dev || !aligned16(dev)) {
        cudaGetLastError();
        return KVD_ERR_INVALID;   // host memory this device cannot address
    }
    pool->host_kv = static_cast<uint8_t*>(dev);
    pool->host_mem = static_cast<uint8_t*>(host_mem);
    pool->staging = static_cast<uint8_t*>(staging_mem);
    pool->host_blocks = host_blocks;
    pool->host_layer_bytes = need_stage / 2;
    pool->host_direct = direct ? 1 : 0;
    return KVD_OK;
}

kvd_status kvd_tier_prefetch(kvd_pool* pool, int layer, void* stream) {
    if (!pool || layer < 0 || layer >= pool->desc.num_layers) return KVD_ERR_INVALID;
    if (pool->host_blocks == 0 || pool->host_direct) return KVD_OK;
    // One DMA on a copy engine: the decode kernel holds every SM while it runs, so a copy
    // made by SMs could not overlap it.
    const uint8_t* src = pool->host_mem + static_cast<size_t>(layer) * pool->host_layer_bytes;
    uint8_t* dst = pool->staging + static_cast<size_t>(layer % 2) * pool->host_layer_bytes;
    return cuda_status(cudaMemcpyAsync(dst, src, pool->host_layer_bytes, cudaMemcpyHostToDevice,
                                       static_cast<cudaStream_t>(stream)));
}

kvd_status kvd_tier_plan(const float* scores, int64_t scores_stride, const int32_t* seq_lens, int batch,
                         int max_blocks_per_seq, int protect_prompt, int protect_recent, int t1_blocks,
                         float* importance, int8_t* tier, void* stream) {
    if (batch < 0 || scores_stride < 1 || max_blocks_per_seq < 1 || protect_prompt < 0 || protect_recent < 0 ||
        t1_blocks < 0)
        return KVD_ERR_INVALID;
    if (max_blocks_per_seq > kvd::kMaxPlanBlocks) return KVD_ERR_UNSUPPORTED;
    if (batch == 0) return KVD_OK;
    if (!scores || !seq_lens || !tier) return KVD_ERR_INVALID;
    kvd::TierPlanParams p;
    p.scores = scores;
    p.scores_stride = scores_stride;
    p.seq_lens = seq_lens;
    p.importance = importance;
    p.tier = tier;
    p.B = batch;
    p.max_blocks = max_blocks_per_seq;
    p.protect_prompt = protect_prompt;
    p.protect_recent = protect_recent;
    p.t1 = t1_blocks;
    return cuda_status(kvd::launch_tier_plan(p, static_cast<cudaStream_t>(stream)));
}

kvd_status kvd_tier_move(kvd_pool* pool, const int32_t* from_ids, const int32_t* to_ids, int n, void* stream) {
    if (!pool || n < 0) return KVD_ERR_INVALID;
    if (n == 0) return KVD_OK;
    if (!from_ids || !to_ids) return KVD_ERR_INVALID;
    kvd::TierMoveParams p;
    p.from_ids = from_ids;
    p.to_ids = to_ids;
    p.kv = pool->mem;
    p.host_kv = pool->host_kv;
    p.err = pool->err;
    p.num_blocks = pool->desc.num_blocks;
    p.host_blocks = pool->host_blocks;
    p.record_bytes = static_cast<int64_t>(record_bytes(&pool->desc));
    p.n = n;
    p.L = pool->desc.num_layers;
    p.n_kv = pool->desc.n_kv;
    return cuda_status(kvd::launch_tier_move(p, pool->num_sms, static_cast<cudaStream_t>(stream)));
}

kvd_status kvd_tier_reassign(int64_t num_blocks, int64_t host_blocks, const int8_t* tier, int32_t* block_table,
                             int batch, int max_blocks_per_seq, int32_t* hbm_free, int32_t* hbm_free_n,
                             int32_t* host_free, int32_t* host_free_n, uint16_t* retain_mask, int32_t* from_ids,
                             int32_t* to_ids, int32_t* n_moves) {
    if (num_blocks < 1 || host_blocks < 0 || num_blocks + host_blocks > INT32_MAX || batch < 0 ||
        max_blocks_per_seq < 1 || !n_moves)
        return KVD_ERR_INVALID;
    *n_moves = 0;
    if (batch == 0) return KVD_OK;
    if (!tier || !block_table || !hbm_free || !hbm_free_n || !host_free || !host_free_n || !from_ids || !to_ids)
        return KVD_ERR_INVALID;
    const int64_t nb = num_blocks, ids = num_blocks + host_blocks;
    if (*hbm_free_n < 0 || *hbm_free_n > nb || *host_free_n < 0 || *host_free_n > host_blocks) return KVD_ERR_INVALID;
    // remap[p]: where block p is after this call, decided by its first table entry (-1: not seen)
    int32_t* remap = static_cast<int32_t*>(std::malloc(sizeof(int32_t) * static_cast<size_t>(ids)));
    if (!remap) return KVD_ERR_NOMEM;
    for (int64_t i = 0; i < ids; ++i) remap[i] = -1;
    kvd_status st = KVD_OK;
    int32_t n = 0;
    const int64_t entries = static_cast<int64_t>(batch) * max_blocks_per_seq;
    for (int64_t e = 0; e < entries; ++e) {
        if (tier[e] < 0) continue;
        const int32_t p = block_table[e];
        if (p < 0 || p >= ids) {
            st = KVD_ERR_OOB;
            continue;
        }
        if (remap[p] >= 0) {   // shared with an entry already decided
            block_table[e] = remap[p];
            continue;
        }
        remap[p] = p;
        const bool in_host = p >= nb, want_host = tier[e] == 1;
        if (in_host == want_host) continue;
        int32_t* list = want_host ? host_free : hbm_free;
        int32_t* len = want_host ? host_free_n : hbm_free_n;
        if (*len == 0) {
            if (st == KVD_OK) st = KVD_ERR_NOMEM;
            continue;
        }
        const int32_t d = list[--*len];
        if (d < (want_host ? nb : 0) || d >= (want_host ? ids : nb)) {   // a free list holding a wrong id
            std::free(remap);
            return KVD_ERR_INVALID;
        }
        remap[p] = d;
        block_table[e] = d;
        if (retain_mask) retain_mask[d] = retain_mask[p];
        from_ids[n] = p;
        to_ids[n] = d;
        ++n;
    }
    for (int32_t i = 0; i < n; ++i) {   // the sources are free once their copies have run
        const int32_t p = from_ids[i];
        int32_t* list = p >= nb ? host_free : hbm_free;
        int32_t* len = p >= nb ? host_free_n : hbm_free_n;
        if (*len >= (p >= nb ? host_blocks : nb)) {   // more free ids than the tier has: inconsistent input
            st = KVD_ERR_INVALID;
            continue;
        }
        list[(*len)++] = p;
    }
    std::free(remap);
    *n_moves = n;
    return st;
}

void kvd_pool_destroy(kvd_pool* pool) {
    if (!pool) return;
    if (pool->err) cudaFree(pool->err);
    delete pool;
}

kvd_status kvd_append_kv(kvd_pool* pool, int layer, const void* k_new, const void* v_new,
                         const int64_t* slot_mapping, int n_tokens, void* stream) {
    if (!pool || layer < 0 || layer >= pool->desc.num_layers || n_tokens < 0) return KVD_ERR_INVALID;
    if (n_tokens == 0) return KVD_OK;
    if (!k_new || !v_new || !slot_mapping) return KVD_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(k_new) & 7u) || (reinterpret_cast<uintptr_t>(v_new) & 7u)) return KVD_ERR_INVALID;
    if (pool->desc.kv_dtype == KVD_MIXED && !pool->block_fmt) return KVD_ERR_INVALID;
    kvd::AppendParams p;
    p.k_new = static_cast<const uint16_t*>(k_new);
    p.v_new = static_cast<const uint16_t*>(v_new);
    p.slot_mapping = slot_mapping;
    p.kv = pool->mem + static_cast<size_t>(layer) * pool->layer_bytes;
    p.host_kv = pool->host_kv ? pool->host_kv + static_cast<size_t>(layer) * pool->host_layer_bytes : nullptr;
    p.block_fmt = pool->block_fmt;
    p.err = pool->err;
    p.ng = pool_ng(&pool->desc);
    p.n_tokens = n_tokens;
    p.num_blocks = pool->desc.num_blocks;
    p.host_blocks = pool->host_blocks;
    p.n_kv = pool->desc.n_kv;
    return cuda_status(kvd::launch_append(p, pool_kind(pool), static_cast<cudaStream_t>(stream)));
}

static kvd_status check_decode_shape(const kvd_pool* pool, int n_q, int batch, int max_seq_len) {
    if (!pool || n_q < 1 || batch < 0 || max_seq_len < 1) return KVD_ERR_INVALID;
    if (n_q % pool->desc.n_kv != 0) return KVD_ERR_INVALID;
    const int g = n_q / pool->desc.n_kv;
    if (g > kvd::kMaxG || batch > kvd::kMaxBatch) return KVD_ERR_UNSUPPORTED;
    // the decode kernel addresses a record by its offset in 16-byte units, 32 bits wide
    if (pool->layer_bytes / 16 > UINT32_MAX || pool->host_layer_bytes / 16 > UINT32_MAX) return KVD_ERR_UNSUPPORTED;
    return KVD_OK;
}

}  // extern "C"

namespace kvd {
// Workspace bytes of a planned call (which also serve an unplanned one), or of an unplanned call
// alone (the no-alloc entry point, which takes no plan).
kvd_status decode_workspace_bytes(const kvd_pool* pool, int n_q, int batch, int max_seq_len, int num_splits,
                                  bool planned, int* splits_out, size_t* bytes_out) {
    kvd_status st = check_decode_shape(pool, n_q, batch, max_seq_len);
    if (st != KVD_OK) return st;
    if (num_splits < 0 || !bytes_out) return KVD_ERR_INVALID;
    const int S = num_splits > 0 ? num_splits : plan_splits(pool, batch, max_seq_len, n_q / pool->desc.n_kv);
    const WsLayout w = ws_layout(batch * pool->desc.n_kv, S, n_q / pool->desc.n_kv, batch, planned);
    if (splits_out) *splits_out = S;
    *bytes_out = w.total;
    return KVD_OK;
}
}  // namespace kvd

extern "C" {

kvd_status kvd_decode_workspace_bytes(const kvd_pool* pool, int n_q, int batch, int max_seq_len, int num_splits,
                                      int* splits_out, size_t* bytes_out) {
    return kvd::decode_workspace_bytes(pool, n_q, batch, max_seq_len, num_splits, true, splits_out, bytes_out);
}

kvd_status kvd_decode_attn(kvd_pool* pool, int layer, const void* q, int n_q, const void* k_new, const void* v_new,
                           const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                           int max_seq_len,
                           int num_splits, const uint16_t* retain_mask, float softmax_scale, void* workspace,
                           size_t workspace_bytes, void* out, int out_dtype, float* lse_out, float* logits_out,
                           int64_t logits_stride, const kvd_scores_desc* scores_epilogue, unsigned flags,
                           void* stream) {
    kvd_status st = check_decode_shape(pool, n_q, batch, max_seq_len);
    if (st != KVD_OK) return st;
    if (layer < 0 || layer >= pool->desc.num_layers || num_splits < 0 || max_blocks_per_seq < 1) return KVD_ERR_INVALID;
    if (out_dtype != KVD_BF16 && out_dtype != KVD_F32) return KVD_ERR_INVALID;
    if (flags & ~static_cast<unsigned>(KVD_EARLY_START | KVD_PLANNED)) return KVD_ERR_INVALID;
    if (batch == 0) return KVD_OK;
    if (!q || !block_table || !seq_lens || !workspace) return KVD_ERR_INVALID;
    if ((k_new == nullptr) != (v_new == nullptr)) return KVD_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(k_new) & 7u) || (reinterpret_cast<uintptr_t>(v_new) & 7u)) return KVD_ERR_INVALID;
    if (logits_out && logits_stride < 1) return KVD_ERR_INVALID;
    if (scores_epilogue) {
        // the score update reads every head's final LSE: lse_out is required
        if (!out || !lse_out || !logits_out || !scores_epilogue->scores || scores_epilogue->scores_stride < 1)
            return KVD_ERR_INVALID;
        if (n_q > 256 || batch > 65535) return KVD_ERR_UNSUPPORTED;
    }
    if ((reinterpret_cast<uintptr_t>(q) & 3u) || (reinterpret_cast<uintptr_t>(out) & 15u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KVD_ERR_INVALID;
    const int g = n_q / pool->desc.n_kv;
    const int U = batch * pool->desc.n_kv;
    const int S = num_splits > 0 ? num_splits : plan_splits(pool, batch, max_seq_len, g);
    const WsLayout w = ws_layout(U, S, g, batch, (flags & KVD_PLANNED) != 0);
    if (workspace_bytes < w.total) return KVD_ERR_NOMEM;
    if (pool->desc.kv_dtype == KVD_MIXED && !pool->block_fmt) return KVD_ERR_INVALID;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int kind = pool_kind(pool);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    kvd::DecodeParams p;
    p.kv = pool->mem + static_cast<size_t>(layer) * pool->layer_bytes;
    p.host_blocks = pool->host_blocks;
    p.host_kv = pool->host_blocks ? pool->host_kv + static_cast<size_t>(layer) * pool->host_layer_bytes : nullptr;
    p.host_direct = pool->host_direct;
    p.stage = !pool->host_blocks ? nullptr
              : pool->host_direct ? p.host_kv
                                  : pool->staging + static_cast<size_t>(layer % 2) * pool->host_layer_bytes;
    p.q = static_cast<const uint16_t*>(q);
    p.k_new = static_cast<const uint16_t*>(k_new);
    p.v_new = static_cast<const uint16_t*>(v_new);
    p.out = out;
    p.lse_out = out ? lse_out : nullptr;
    p.out_f32 = out_dtype == KVD_F32;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.retain = retain_mask;
    p.block_fmt = pool->block_fmt;
    p.part_o = reinterpret_cast<float*>(ws + w.part_o);
    p.part_lse = reinterpret_cast<float*>(ws + w.part_lse);
    p.unit_first = reinterpret_cast<int32_t*>(ws + w.unit_first);
    p.unit_count = reinterpret_cast<int32_t*>(ws + w.unit_count);
    p.plan = (flags & KVD_PLANNED) ? reinterpret_cast<const int32_t*>(ws + w.plan) : nullptr;
    // Run-time balancing with a step plan (its counters live in the plan), for BF16 pools: there
    // the decode kernel is bound by HBM and its consumer warps have time for the segment switch
    // a taken piece costs; the 8-bit and low-bit kernels are bound by their consumers' instructions
    // (measured: mixed pool 7.6% slower with it, 8B BF16 2.1% and ragged BF16 4.7% faster).
    p.dyn = (flags & KVD_PLANNED) && kind == kvd::kKindBf16
                ? reinterpret_cast<int32_t*>(ws + w.plan) + kvd::decode_plan_dyn_off(batch, S)
                : nullptr;
    p.logits = logits_out;
    p.logits_stride = logits_stride;
    p.err = pool->err;
    p.num_blocks = pool->desc.num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.B = batch;
    p.n_kv = pool->desc.n_kv;
    p.g = g;
    p.n_q = n_q;
    p.nsplit = S;
    p.ng = pool_ng(&pool->desc);
    p.max_seq_len = max_seq_len;
    p.early = (flags & KVD_EARLY_START) ? 1 : 0;
    p.scale_log2 = softmax_scale * kvd::kLog2e;
    const int carveout = kvd::decode_carveout(kind, p.ng, batch, g);
    cudaError_t e = kvd::launch_decode(p, kind, carveout, s);
    if (e != cudaSuccess) return KVD_ERR_CUDA;
    if (!out) return KVD_OK;  // partials only: the caller merges them with kvd_combine_splits

    kvd::CombineParams c;
    c.part_o = p.part_o;
    c.part_lse = p.part_lse;
    c.unit_first = p.unit_first;
    c.unit_count = p.unit_count;
    c.out = out;
    c.lse_out = lse_out;
    c.B = batch;
    c.n_q = n_q;
    c.n_kv = pool->desc.n_kv;
    c.g = g;
    c.out_f32 = out_dtype == KVD_F32;
    c.slots_hint = (p.dyn ? S * kvd::kDecodePieces : S) / U + 2;
    if (!scores_epilogue) return cuda_status(kvd::launch_combine(c, carveout, s));
    kvd::ScoreParams sp;
    sp.logits = logits_out;
    sp.logits_stride = logits_stride;
    sp.lse = nullptr;
    sp.seq_lens = seq_lens;
    sp.scores = scores_epilogue->scores;
    sp.scores_stride = scores_epilogue->scores_stride;
    sp.B = batch;
    sp.n_q = n_q;
    sp.inv_LH = scores_epilogue->inv_LH;
    return cuda_status(kvd::launch_epilogue(c, sp, carveout, s));
}

kvd_status kvd_decode_plan(kvd_pool* pool, int n_q, const int32_t* block_table, int max_blocks_per_seq,
                           const int32_t* seq_lens, int batch, int max_seq_len, int num_splits,
                           const uint16_t* retain_mask, void* workspace, size_t workspace_bytes, void* stream) {
    kvd_status st = check_decode_shape(pool, n_q, batch, max_seq_len);
    if (st != KVD_OK) return st;
    if (num_splits < 0 || max_blocks_per_seq < 1) return KVD_ERR_INVALID;
    if (batch == 0) return KVD_OK;
    if (!block_table || !seq_lens || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KVD_ERR_INVALID;
    if (pool->desc.kv_dtype == KVD_MIXED && !pool->block_fmt) return KVD_ERR_INVALID;
    const int g = n_q / pool->desc.n_kv;
    const int S = num_splits > 0 ? num_splits : plan_splits(pool, batch, max_seq_len, g);
    const WsLayout w = ws_layout(batch * pool->desc.n_kv, S, g, batch, true);
    if (workspace_bytes < w.total) return KVD_ERR_NOMEM;
    kvd::DecodeParams p = {};
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.retain = retain_mask;
    p.block_fmt = pool->block_fmt;
    p.err = pool->err;
    p.num_blocks = pool->desc.num_blocks;
    p.host_blocks = pool->host_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.B = batch;
    p.n_kv = pool->desc.n_kv;
    p.g = g;
    p.n_q = n_q;
    p.nsplit = S;
    int32_t* plan = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + w.plan);
    return cuda_status(kvd::launch_plan(p, plan, static_cast<cudaStream_t>(stream)));
}

kvd_status kvd_combine_splits(const float* part_o, const float* part_lse, const int32_t* unit_first,
                              const int32_t* unit_count, int batch, int n_q, int n_kv, int d_h, void* out,
                              int out_dtype, float* lse_out, void* stream) {
    if (batch < 0 || n_q < 1 || n_kv < 1 || n_q % n_kv != 0) return KVD_ERR_INVALID;
    if (out_dtype != KVD_BF16 && out_dtype != KVD_F32) return KVD_ERR_INVALID;
    if (d_h != kvd::kDh || n_q / n_kv > kvd::kMaxG) return KVD_ERR_UNSUPPORTED;
    if (batch == 0) return KVD_OK;
    if (!part_o || !part_lse || !unit_first || !unit_count || !out) return KVD_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(part_o) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u)) return KVD_ERR_INVALID;
    kvd::CombineParams c;
    c.part_o = part_o;
    c.part_lse = part_lse;
    c.unit_first = unit_first;
    c.unit_count = unit_count;
    c.out = out;
    c.lse_out = lse_out;
    c.B = batch;
    c.n_q = n_q;
    c.n_kv = n_kv;
    c.g = n_q / n_kv;
    c.out_f32 = out_dtype == KVD_F32;
    c.slots_hint = 64;   // counts unknown on the host: assume many partials per unit
    return cuda_status(kvd::launch_combine(c, -1, static_cast<cudaStream_t>(stream)));
}

kvd_status kvd_accum_scores(const float* logits, int64_t logits_stride, const float* lse, const int32_t* seq_lens,
                            int batch, int n_q, float inv_LH, float* scores, int64_t scores_stride, void* stream) {
    if (batch < 0 || n_q < 1 || logits_stride < 1 || scores_stride < 1) return KVD_ERR_INVALID;
    if (batch == 0) return KVD_OK;
    if (!logits || !lse || !seq_lens || !scores) return KVD_ERR_INVALID;
    if (batch > 65535 || n_q > 256) return KVD_ERR_UNSUPPORTED;
    kvd::ScoreParams p;
    p.logits = logits;
    p.logits_stride = logits_stride;
    p.lse = lse;
    p.seq_lens = seq_lens;
    p.scores = scores;
    p.scores_stride = scores_stride;
    p.B = batch;
    p.n_q = n_q;
    p.inv_LH = inv_LH;
    return cuda_status(kvd::launch_scores(p, static_cast<cudaStream_t>(stream)));
}

kvd_status kvd_get_device_error(kvd_pool* pool, void* stream, int32_t* code) {
    if (!pool || !code) return KVD_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t h = 0;
    if (cudaMemcpyAsync(&h, pool->err, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KVD_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVD_ERR_CUDA;
    if (cudaMemsetAsync(pool->err, 0, sizeof(int32_t), s) != cudaSuccess) return KVD_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVD_ERR_CUDA;
    *code = h;
    return KVD_OK;
}

kvd_status kvd_selftest_wait_timeout(kvd_pool* pool, int64_t timeout_ns, void* stream) {
    if (!pool || timeout_ns < 1 || timeout_ns > 10000000000ll) return KVD_ERR_INVALID;
    return cuda_status(kvd::launch_wait_timeout(pool->err, timeout_ns, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
