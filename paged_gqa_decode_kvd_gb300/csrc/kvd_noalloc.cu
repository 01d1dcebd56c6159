// kvd_noalloc.cu — decode attention that allocates nothing: its split scratch lives in a
// fixed-size array in the library's own device image.
//
// Some callers may not allocate device memory themselves: a host framework that owns
// every byte of device memory through its own arena and forbids raw allocations by
// plugins, or a latency-critical serving loop that cannot afford cudaMalloc's implicit
// device synchronisation.  kvd_decode_attn_noalloc lets them run decode attention with
// only their inputs and outputs.  The scratch array below is created when the library's
// device code is loaded on a GPU and stays resident on every GPU that loads the library
// until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kvd.h"
#include "kvd_internal.h"

namespace {

// Split partials and unit tables of one kvd_decode_attn call (its "workspace").
__device__ __align__(256) unsigned char g_noalloc_scratch[KVD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on device `dev` (the current device), looked up once
// per device and kept for the lifetime of that device's primary context.
kvd_status scratch_for_device(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return KVD_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return KVD_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KVD_OK;
}

}  // namespace

namespace kvd {
kvd_status decode_workspace_bytes(const kvd_pool* pool, int n_q, int batch, int max_seq_len, int num_splits,
                                  bool planned, int* splits_out, size_t* bytes_out);   // kvd_api.cu
}

extern "C" kvd_status kvd_decode_attn_noalloc(kvd_pool* pool, int layer, const void* q, int n_q,
                                              const void* k_new, const void* v_new,
                                              const int32_t* block_table, int max_blocks_per_seq,
                                              const int32_t* seq_lens, int batch, int max_seq_len, int num_splits,
                                              const uint16_t* retain_mask, float softmax_scale, void* out,
                                              int out_dtype, float* lse_out, float* logits_out,
                                              int64_t logits_stride, const kvd_scores_desc* scores_epilogue,
                                              unsigned flags, void* stream) {
    if (!pool) return KVD_ERR_INVALID;
    if (!out && batch > 0) return KVD_ERR_INVALID;  // the partials would be unreachable
    if (flags & KVD_PLANNED) return KVD_ERR_INVALID;  // no step plan can be in the shared array
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVD_ERR_CUDA;
    // the scratch address below is the current device's: it must be the pool's device
    if (dev != kvd::pool_device(pool)) return KVD_ERR_INVALID;
    int splits = 0;
    size_t need = 0;
    kvd_status st = kvd::decode_workspace_bytes(pool, n_q, batch, max_seq_len, num_splits, false, &splits, &need);
    if (st != KVD_OK) return st;
    if (need > static_cast<size_t>(KVD_NOALLOC_SCRATCH_BYTES)) return KVD_ERR_NOMEM;
    void* scratch = nullptr;
    st = scratch_for_device(dev, &scratch);
    if (st != KVD_OK) return st;
    return kvd_decode_attn(pool, layer, q, n_q, k_new, v_new, block_table, max_blocks_per_seq, seq_lens, batch,
                           max_seq_len,
                           splits, retain_mask, softmax_scale, scratch, static_cast<size_t>(KVD_NOALLOC_SCRATCH_BYTES),
                           out, out_dtype, lse_out, logits_out, logits_stride, scores_epilogue, flags, stream);
}
