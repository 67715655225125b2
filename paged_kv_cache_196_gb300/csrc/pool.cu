// Device pool, KV append (slot-mapping write) and copy-on-write block copy.
//
// KV append: "Makale Bulteni -- PagedAttention ve vLLM", "Iddia ve Gerceklik"
// (a new token goes into the current block; a free block is taken when it is
// full) and "PagedAttention Nedir?", "Nasil Calisir?" steps 1-3.  The host
// decides the slots (kv_prepare_append); the kernel is an exact scatter.
//
// Copy-on-write: same page, "Iddia ve Gerceklik" (blocks shared by pointer
// between parallel samples and branches, copied when written).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <new>

#include "common.cuh"
#include "internal.h"

namespace pkv {

static thread_local char g_last_error[256] = "no CUDA error recorded";

void note_cuda_error(cudaError_t e) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
             cudaGetErrorString(e));
}

static std::atomic<bool> g_test_waits{false};

bool test_waits_enabled() { return g_test_waits.load(std::memory_order_relaxed); }

kv_status require_device(int device) {
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return KV_ERR_CUDA;
    }
    return cur == device ? KV_OK : KV_ERR_ARG;
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

// Append.  Work item i is 16-byte chunk c of kv head h of token t:
// i = (t * hkv + h) * row_chunks + c, with k_new / v_new laid out
// [T][Hkv][row_chunks] and the pools [NB][Hkv][16][row_chunks].  Each thread
// takes kAppendUnroll items a grid apart and issues all their loads before
// its stores (more bytes in flight per thread).  Idx is 32-bit when the item
// count allows it (the host decides): the token index costs a 32-bit division
// instead of a 64-bit one.  row_chunks is a power of two and the block size
// is 16, so the rest is shifts and masks.
constexpr int kAppendUnroll = 2;
constexpr int kAppendThreads = 256;

template <typename Idx>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(uint4 *__restrict__ k_pool,
                                                                uint4 *__restrict__ v_pool,
                                                                const uint4 *__restrict__ k_new,
                                                                const uint4 *__restrict__ v_new,
                                                                const int64_t *__restrict__ slots,
                                                                Idx total, int hkv, int rc_log2,
                                                                long long num_slots, int *err) {
    const Idx per_token = (Idx)hkv << rc_log2;
    const Idx stride = (Idx)gridDim.x * kAppendThreads;
    const int rc_mask = (1 << rc_log2) - 1;
    for (Idx base = (Idx)blockIdx.x * kAppendThreads + threadIdx.x; base < total;
         base += stride * kAppendUnroll) {
        uint4 kv[kAppendUnroll], vv[kAppendUnroll];
        long long dst[kAppendUnroll];
#pragma unroll
        for (int u = 0; u < kAppendUnroll; ++u) {
            const Idx i = base + (Idx)u * stride;
            dst[u] = -1;
            if (i < total) {
                const Idx t = i / per_token;
                const int rem = (int)(i - t * per_token);
                const int64_t slot = __ldg(slots + t);
                if (slot >= num_slots) {
                    if (rem == 0) atomicOr(err, KV_DEVERR_SLOT_RANGE);
                } else if (slot >= 0) {
                    const long long row = ((slot >> 4) * hkv + (rem >> rc_log2)) * 16 + (slot & 15);
                    dst[u] = (row << rc_log2) + (rem & rc_mask);
                    kv[u] = __ldg(k_new + i);
                    vv[u] = __ldg(v_new + i);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kAppendUnroll; ++u)
            if (dst[u] >= 0) {
                k_pool[dst[u]] = kv[u];
                v_pool[dst[u]] = vv[u];
            }
    }
}

// Copies whole blocks (all heads and slots) of K and V: pair p moves block
// src[p] to block dst[p].  block_chunks = 16-byte chunks per block per pool.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4 *__restrict__ k_pool,
                                                          uint4 *__restrict__ v_pool,
                                                          const int32_t *__restrict__ src,
                                                          const int32_t *__restrict__ dst,
                                                          int n, int block_chunks, int num_blocks,
                                                          int *err) {
    const long long total = (long long)n * block_chunks;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int p = (int)(i / block_chunks);
        const int c = (int)(i - (long long)p * block_chunks);
        const int s = __ldg(src + p), d = __ldg(dst + p);
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
            if (c == 0) atomicOr(err, KV_DEVERR_BLOCK_RANGE);
            continue;
        }
        k_pool[(long long)d * block_chunks + c] = k_pool[(long long)s * block_chunks + c];
        v_pool[(long long)d * block_chunks + c] = v_pool[(long long)s * block_chunks + c];
    }
}

// Copies one whole block (all heads and slots of K and V), src -> dst; the
// host checked both ids.
__global__ void __launch_bounds__(256) copy_block_kernel(uint4 *__restrict__ k_pool,
                                                         uint4 *__restrict__ v_pool, int src,
                                                         int dst, int block_chunks) {
    for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < block_chunks; c += gridDim.x * blockDim.x) {
        k_pool[(long long)dst * block_chunks + c] = k_pool[(long long)src * block_chunks + c];
        v_pool[(long long)dst * block_chunks + c] = v_pool[(long long)src * block_chunks + c];
    }
}

// Swap: whole blocks (K and V, all heads) between the pool and a buffer the
// GPU can address directly (pinned host memory on this system: the stores /
// loads cross NVLink-C2C or PCIe).  Host layout: [n][K|V][block chunks].
// dir = 0: pool -> host (swap out); dir = 1: host -> pool (swap in).
__global__ void __launch_bounds__(256) swap_blocks_kernel(uint4 *__restrict__ k_pool,
                                                          uint4 *__restrict__ v_pool,
                                                          uint4 *__restrict__ host,
                                                          const int32_t *__restrict__ ids, int n,
                                                          int block_chunks, int num_blocks, int dir,
                                                          int *err) {
    const long long total = (long long)n * block_chunks;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int p = (int)(i / block_chunks);
        const int c = (int)(i - (long long)p * block_chunks);
        const int id = __ldg(ids + p);
        if (id < 0 || id >= num_blocks) {
            if (c == 0) atomicOr(err, KV_DEVERR_BLOCK_RANGE);
            continue;
        }
        uint4 *hk = host + (2LL * p) * block_chunks + c;
        uint4 *hv = hk + block_chunks;
        const long long pc = (long long)id * block_chunks + c;
        if (dir == 0) {
            *hk = k_pool[pc];
            *hv = v_pool[pc];
        } else {
            k_pool[pc] = *hk;
            v_pool[pc] = *hv;
        }
    }
}

static int grid_for(long long work, int threads) {
    long long blocks = (work + threads - 1) / threads;
    long long cap = (long long)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : (int)blocks;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char *kv_last_cuda_error(void) { return g_last_error; }

kv_status kv_pool_create(int num_blocks, int block_size, int num_kv_heads, int head_dim,
                         kv_dtype dtype, kv_pool_t *out) {
    if (!out || num_blocks <= 0 || num_kv_heads <= 0) return KV_ERR_ARG;
    if (block_size != 16 || (head_dim != 64 && head_dim != 128) ||
        (dtype != KV_F32 && dtype != KV_BF16 && dtype != KV_F16))
        return KV_ERR_UNSUPPORTED;
    kv_pool *p = new (std::nothrow) kv_pool();
    if (!p) return KV_ERR_OOM;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->num_kv_heads = num_kv_heads;
    p->head_dim = head_dim;
    p->dtype = dtype;
    cudaGetDevice(&p->device);
    const size_t bytes = (size_t)num_blocks * num_kv_heads * block_size * head_dim * dtype_bytes(dtype);
    kv_status st = KV_OK;
    if (cudaMalloc(&p->k, bytes) != cudaSuccess || cudaMalloc(&p->v, bytes) != cudaSuccess ||
        cudaMalloc(&p->err, sizeof(int)) != cudaSuccess ||
        cudaMalloc(&p->counters, sizeof(int) * kv_pool::kCounterSlots) != cudaSuccess) {
        cudaGetLastError();
        st = KV_ERR_OOM;
    } else if (cudaMemset(p->err, 0, sizeof(int)) != cudaSuccess ||
               cudaMemset(p->counters, 0, sizeof(int) * kv_pool::kCounterSlots) != cudaSuccess) {
        st = KV_ERR_CUDA;
    } else {
        st = kv_allocator_create(num_blocks, &p->alloc);
    }
    if (st != KV_OK) {
        kv_pool_destroy(p);
        return st;
    }
    *out = p;
    return KV_OK;
}

kv_status kv_pool_destroy(kv_pool_t p) {
    if (!p) return KV_ERR_ARG;
    // free on the pool's own device, then give the caller its device back
    int cur = -1;
    const bool switched = cudaGetDevice(&cur) == cudaSuccess && cur != p->device &&
                          cudaSetDevice(p->device) == cudaSuccess;
    if (p->k) cudaFree(p->k);
    if (p->v) cudaFree(p->v);
    if (p->err) cudaFree(p->err);
    if (p->counters) cudaFree(p->counters);
    if (switched) cudaSetDevice(cur);
    if (p->alloc) kv_allocator_destroy(p->alloc);
    delete p;
    return KV_OK;
}

kv_status kv_pool_ptrs(kv_pool_t p, void **k_pool, void **v_pool) {
    if (!p) return KV_ERR_ARG;
    if (k_pool) *k_pool = p->k;
    if (v_pool) *v_pool = p->v;
    return KV_OK;
}

kv_status kv_pool_set_launch_overlap(kv_pool_t p, int enable) {
    if (!p || (enable != 0 && enable != 1)) return KV_ERR_ARG;
    p->launch_overlap = enable != 0;
    return KV_OK;
}

kv_status kv_pool_allocator(kv_pool_t p, kv_allocator_t *out) {
    if (!p || !out) return KV_ERR_ARG;
    *out = p->alloc;
    return KV_OK;
}

kv_status kv_alloc_blocks(kv_pool_t p, int n, int32_t *ids_out) {
    if (!p) return KV_ERR_ARG;
    return kv_allocator_alloc(p->alloc, n, ids_out);
}

kv_status kv_share_blocks(kv_pool_t p, int n, const int32_t *ids) {
    if (!p) return KV_ERR_ARG;
    return kv_allocator_share(p->alloc, n, ids);
}

kv_status kv_free_blocks(kv_pool_t p, int n, const int32_t *ids) {
    if (!p) return KV_ERR_ARG;
    return kv_allocator_free(p->alloc, n, ids);
}

kv_status kv_cow_if_shared(kv_pool_t p, int32_t *block_id_inout, int *copied, void *stream) {
    if (!p || !block_id_inout || !copied) return KV_ERR_ARG;
    if (kv_status st = require_device(p->device)) return st;
    *copied = 0;
    const int32_t old = *block_id_inout;
    int rc = 0;
    if (kv_allocator_refcount(p->alloc, old, &rc) != KV_OK || rc <= 0) return KV_ERR_ARG;
    if (rc == 1) return KV_OK;  // private already: write in place
    int32_t fresh = -1;
    if (kv_status st = kv_allocator_alloc(p->alloc, 1, &fresh)) return st;
    const int block_chunks = p->num_kv_heads * p->block_size * p->head_dim * dtype_bytes(p->dtype) / 16;
    copy_block_kernel<<<grid_for(block_chunks, 256), 256, 0, as_stream(stream)>>>(
        (uint4 *)p->k, (uint4 *)p->v, old, fresh, block_chunks);
    if (kv_status st = cuda_status(cudaGetLastError())) {
        kv_allocator_free(p->alloc, 1, &fresh);
        return st;
    }
    kv_allocator_free(p->alloc, 1, &old);  // the other holders keep it (rc > 1)
    *block_id_inout = fresh;
    *copied = 1;
    return KV_OK;
}

kv_status kv_append(kv_pool_t p, const void *k_new, const void *v_new,
                    const int64_t *slot_mapping, int num_tokens, void *stream) {
    if (!p || num_tokens < 0) return KV_ERR_ARG;
    if (kv_status st = require_device(p->device)) return st;
    if (num_tokens == 0) return KV_OK;
    if (!k_new || !v_new || !slot_mapping) return KV_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
        return KV_ERR_ARG;  // rows are moved as 16-byte chunks
    const int row_chunks = p->head_dim * dtype_bytes(p->dtype) / 16;  // 8, 16 or 32
    const int rc_log2 = row_chunks == 8 ? 3 : row_chunks == 16 ? 4 : 5;
    const long long total = (long long)num_tokens * p->num_kv_heads * row_chunks;
    // eight CTAs per SM at most (full occupancy); fewer for small appends
    long long blocks = (total + (long long)kAppendThreads * kAppendUnroll - 1) /
                       ((long long)kAppendThreads * kAppendUnroll);
    const long long cap = 8LL * sm_count();
    if (blocks > cap) blocks = cap;
    // a whole number of CTAs per SM
    if (blocks > sm_count()) blocks = (blocks + sm_count() - 1) / sm_count() * sm_count();
    const long long span = blocks * kAppendThreads * kAppendUnroll;  // one loop step of the grid
    const long long num_slots = (long long)p->num_blocks * p->block_size;
    if (total + span < (1LL << 31))
        append_kernel<uint32_t><<<(int)blocks, kAppendThreads, 0, as_stream(stream)>>>(
            (uint4 *)p->k, (uint4 *)p->v, (const uint4 *)k_new, (const uint4 *)v_new,
            slot_mapping, (uint32_t)total, p->num_kv_heads, rc_log2, num_slots, p->err);
    else
        append_kernel<unsigned long long><<<(int)blocks, kAppendThreads, 0, as_stream(stream)>>>(
            (uint4 *)p->k, (uint4 *)p->v, (const uint4 *)k_new, (const uint4 *)v_new,
            slot_mapping, (unsigned long long)total, p->num_kv_heads, rc_log2, num_slots, p->err);
    return cuda_status(cudaGetLastError());
}

kv_status kv_copy_blocks(kv_pool_t p, const int32_t *src, const int32_t *dst, int n,
                         void *stream) {
    if (!p || n < 0) return KV_ERR_ARG;
    if (kv_status st = require_device(p->device)) return st;
    if (n == 0) return KV_OK;
    if (!src || !dst) return KV_ERR_ARG;
    const int block_chunks = p->num_kv_heads * p->block_size * p->head_dim * dtype_bytes(p->dtype) / 16;
    copy_blocks_kernel<<<grid_for((long long)n * block_chunks, 256), 256, 0, as_stream(stream)>>>(
        (uint4 *)p->k, (uint4 *)p->v, src, dst, n, block_chunks, p->num_blocks, p->err);
    return cuda_status(cudaGetLastError());
}

static kv_status swap(kv_pool_t p, const int32_t *ids, int n, void *host, int dir, void *stream) {
    if (!p || n < 0) return KV_ERR_ARG;
    if (kv_status st = require_device(p->device)) return st;
    if (n == 0) return KV_OK;
    if (!ids || !host || (reinterpret_cast<uintptr_t>(host) & 15)) return KV_ERR_ARG;
    const int block_chunks = p->num_kv_heads * p->block_size * p->head_dim * dtype_bytes(p->dtype) / 16;
    const long long total = (long long)n * block_chunks;
    swap_blocks_kernel<<<grid_for(total, 256), 256, 0, as_stream(stream)>>>(
        (uint4 *)p->k, (uint4 *)p->v, (uint4 *)host, ids, n, block_chunks, p->num_blocks, dir,
        p->err);
    return cuda_status(cudaGetLastError());
}

kv_status kv_swap_out(kv_pool_t p, const int32_t *block_ids, int n, void *host_buf, void *stream) {
    return swap(p, block_ids, n, host_buf, 0, stream);
}

kv_status kv_swap_in(kv_pool_t p, const int32_t *block_ids, int n, const void *host_buf,
                     void *stream) {
    return swap(p, block_ids, n, const_cast<void *>(host_buf), 1, stream);
}

kv_status kv_swap_bytes(kv_pool_t p, int n, size_t *bytes) {
    if (!p || n < 0 || !bytes) return KV_ERR_ARG;
    *bytes = (size_t)n * 2 * p->num_kv_heads * p->block_size * p->head_dim * dtype_bytes(p->dtype);
    return KV_OK;
}

kv_status kv_debug_set_wait_limit_ns(uint64_t ns) {
    cudaError_t e = set_wait_limit_decode(ns);
    if (e == cudaSuccess) e = set_wait_limit_prefill(ns);
    if (e == cudaSuccess) e = set_wait_limit_cascade(ns);
    if (e == cudaSuccess) g_test_waits.store(ns != KV_WAIT_LIMIT_DEFAULT_NS);
    return cuda_status(e);
}

kv_status kv_get_device_error(kv_pool_t p, int *code, void *stream) {
    if (!p || !code) return KV_ERR_ARG;
    if (kv_status st = require_device(p->device)) return st;
    int h = 0;
    cudaStream_t s = as_stream(stream);
    if (cudaMemcpyAsync(&h, p->err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return KV_ERR_CUDA;
    // After a device error a merge may have been left half counted: clear the
    // arrival counters along with the error word.
    if (h != 0 && (cudaMemsetAsync(p->err, 0, sizeof(int), s) != cudaSuccess ||
                   cudaMemsetAsync(p->counters, 0, sizeof(int) * kv_pool::kCounterSlots, s) !=
                       cudaSuccess))
        return KV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KV_ERR_CUDA;
    *code = h;
    return device_error_status(h);
}

}  // extern "C"
