// Internal host-side definitions shared by the library's translation units.
#pragma once
#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "paged_kv.h"

struct kv_pool {
    int num_blocks = 0;
    int block_size = 0;
    int num_kv_heads = 0;
    int head_dim = 0;
    kv_dtype dtype = KV_BF16;
    int device = 0;
    void *k = nullptr;  // [num_blocks][num_kv_heads][block_size][head_dim]
    void *v = nullptr;
    int *err = nullptr;  // device error word
    // arrival counters of the fused split merge, one per (sequence, kv head),
    // zero between calls (each merging CTA resets its own)
    static constexpr int kCounterSlots = 65536;
    int *counters = nullptr;
    kv_allocator_t alloc = nullptr;
    // tiled-TMA descriptors of the K and V pools (built on first prefill)
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    bool tmaps_ready = false;
    // decode launches may overlap the previous kernel in the stream
    // (kv_pool_set_launch_overlap)
    bool launch_overlap = false;
};

namespace pkv {

inline int dtype_bytes(kv_dtype t) { return t == KV_F32 ? 4 : 2; }

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Remembers the text of the last CUDA error seen by this thread.
void note_cuda_error(cudaError_t e);

// A pool or contiguous context keeps its memory on the device that was
// current when it was created, and its kernels must run there.  Returns
// KV_OK when that device is current, KV_ERR_ARG when another one is (the
// call then launches nothing), KV_ERR_CUDA when the current device cannot be
// read.
kv_status require_device(int device);

// Set the pipeline-wait limit of the kernels of one source file (each has
// its own copy of the device variable) on the current device.
cudaError_t set_wait_limit_decode(unsigned long long ns);
cudaError_t set_wait_limit_prefill(unsigned long long ns);
cudaError_t set_wait_limit_cascade(unsigned long long ns);

// True once a test has set a pipeline-wait limit other than the default
// (kv_debug_set_wait_limit_ns): launches then take the kernels' test
// instantiations, which read the limit at run time.
bool test_waits_enabled();

// Test hook of the contiguous path: page creations left before one fails
// (-1: none fails).  Read and decremented by the page-taking code.
extern std::atomic<int> g_fail_page_create_after;

// Maps a CUDA runtime error to a status.
inline kv_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return KV_OK;
    note_cuda_error(e);
    if (e == cudaErrorMemoryAllocation) return KV_ERR_OOM;
    return KV_ERR_CUDA;
}

inline kv_status device_error_status(int code) {
    if (code == 0) return KV_OK;
    if (code & KV_DEVERR_TIMEOUT) return KV_ERR_TIMEOUT;
    if (code == KV_DEVERR_VALUE_RANGE) return KV_ERR_UNSUPPORTED;
    return KV_ERR_DEVICE_BOUNDS;
}

int sm_count();

// tiled-TMA maps (tmap.cu): bf16 rows of 128 values, boxes 16 x 64, 128B swizzle
bool encode_rows_map(CUtensorMap *m, void *base, long long rows);
bool encode_q_map(CUtensorMap *m, const void *q, int rows, int hq);
kv_status pool_tensor_maps(kv_pool *p);

// ---- decode (shared by the paged and contiguous paths) ----
struct DecodeArgs {
    const void *q;
    // paged addressing
    const void *k_pool;
    const void *v_pool;
    const int32_t *block_tables;
    int max_blocks;
    int num_blocks;
    // contiguous addressing
    const unsigned long long *k_bases;  // per request
    const unsigned long long *v_bases;
    const int32_t *req_ids;
    const long long *mapped_tokens;  // per request
    const CUtensorMap *req_maps;     // per request: K map, V map (contiguous, bf16 d128)
    long long head_stride;           // tokens per head region
    int max_requests;
    // paged: tiled-TMA maps of the pools (bf16 d128 only; else null)
    const CUtensorMap *pool_map_k;
    const CUtensorMap *pool_map_v;
    // common
    const int32_t *seq_lens;
    int batch;
    int num_q_heads;
    int num_kv_heads;
    int head_dim;
    kv_dtype dtype;
    float scale;
    void *out;
    kv_dtype out_dtype;
    float *lse;
    int num_splits;
    // cascade: the first start_tokens[b] tokens of sequence b (whole blocks)
    // were attended elsewhere and left part_base partial results in slots
    // [0, part_base) of the workspace; null / 0 otherwise
    const int32_t *start_tokens;
    int part_base;
    // fused append of one new token per sequence (tensor-core decode only):
    // device [batch][num_kv_heads][head_dim] K and V rows and, on the paged
    // path, int64 slots (the contiguous path writes row seq_lens[b] - 1), or null
    const void *new_k;
    const void *new_v;
    const int64_t *new_slots;
    const int32_t *seq_order;  // device permutation of the batch: grid order, or null
    // balanced schedule (kv_decode_schedule): its device copy, or null, and
    // the header values read from the host copy
    const int32_t *sched;
    int sched_ctas, sched_pieces, sched_max_splits, sched_part_blocks, sched_deep;
    // cascade suffix: the tensor-core decode may start while the prefix kernel
    // (the previous launch in the stream) still runs; only its merges wait
    // for that kernel (griddepcontrol.wait), and every merge must then be
    // inside the decode kernel
    bool overlap_previous;
    // any decode: launched to overlap the previous kernel in the stream, the
    // kernel waits for it (griddepcontrol.wait) before touching memory
    bool chain;
    int *counters;
    long long counter_slots;
    void *workspace;
    size_t workspace_bytes;
    int *err;
    cudaStream_t stream;
};

// Splits per (sequence, kv head) merged inside the decode kernel by the last
// CTA of that pair; longer plans leave the merge to merge_kernel.
constexpr int kFuseMaxSplits = 32;

void split_plan(int batch, int num_kv_heads, int max_blocks, int num_splits, int *part_blocks,
                int *max_splits);
size_t decode_workspace_bytes(int batch, int num_q_heads, int head_dim, int max_splits);
kv_status launch_decode(const DecodeArgs &a, bool linear);

}  // namespace pkv
