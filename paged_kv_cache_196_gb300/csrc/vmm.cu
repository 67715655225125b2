// Contiguous (vAttention-style) KV path.
//
// "Makale Bulteni -- vAttention", section "Iddia ve Gerceklik: vAttention":
// at request start a contiguous virtual buffer large enough for the maximum
// context is reserved (cuMemAddressRangeReserve) and uses no physical memory;
// physical pages are created and mapped (cuMemCreate, cuMemMap) only as the
// request grows; the attention kernel then sees one contiguous tensor and the
// GPU's MMU/TLB does the translation.  The stock driver's smallest page for
// this is its allocation granularity (2 MiB), which is what is used here.
//
// Per request: one reservation holding the K region [Hkv][head_stride][D]
// followed by the V region of the same shape.  head_stride is max_tokens
// rounded up to whole pages so every head's region starts on a page and
// grows page by page.  Each page is its own physical allocation.
//
// Driver entry points are fetched through the runtime at first use, so the
// library loads on machines without a GPU driver.
#include <cuda.h>
#include <cuda_runtime.h>

#include <chrono>
#include <condition_variable>
#include <cstdint>
#include <deque>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace pkv {

struct DriverVmm {
    CUresult (*getGranularity)(size_t *, const CUmemAllocationProp *, CUmemAllocationGranularity_flags) = nullptr;
    CUresult (*addressReserve)(CUdeviceptr *, size_t, size_t, CUdeviceptr, unsigned long long) = nullptr;
    CUresult (*addressFree)(CUdeviceptr, size_t) = nullptr;
    CUresult (*create)(CUmemGenericAllocationHandle *, size_t, const CUmemAllocationProp *, unsigned long long) = nullptr;
    CUresult (*release)(CUmemGenericAllocationHandle) = nullptr;
    CUresult (*map)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle, unsigned long long) = nullptr;
    CUresult (*unmap)(CUdeviceptr, size_t) = nullptr;
    CUresult (*setAccess)(CUdeviceptr, size_t, const CUmemAccessDesc *, size_t) = nullptr;
    bool ok = false;
};

static DriverVmm &driver() {
    static DriverVmm d;
    static std::once_flag once;
    std::call_once(once, [] {
        auto get = [](const char *name, void **fn) {
            cudaDriverEntryPointQueryResult q;
            return cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q) ==
                       cudaSuccess &&
                   q == cudaDriverEntryPointSuccess && *fn != nullptr;
        };
        bool ok = true;
        ok &= get("cuMemGetAllocationGranularity", (void **)&d.getGranularity);
        ok &= get("cuMemAddressReserve", (void **)&d.addressReserve);
        ok &= get("cuMemAddressFree", (void **)&d.addressFree);
        ok &= get("cuMemCreate", (void **)&d.create);
        ok &= get("cuMemRelease", (void **)&d.release);
        ok &= get("cuMemMap", (void **)&d.map);
        ok &= get("cuMemUnmap", (void **)&d.unmap);
        ok &= get("cuMemSetAccess", (void **)&d.setAccess);
        d.ok = ok;
    });
    return d;
}

// Writes new tokens at (request, position) of the contiguous layout.
__global__ void __launch_bounds__(256) contig_append_kernel(
    const unsigned long long *__restrict__ k_bases, const unsigned long long *__restrict__ v_bases,
    const long long *__restrict__ mapped, const uint4 *__restrict__ k_new,
    const uint4 *__restrict__ v_new, const int32_t *__restrict__ req_ids,
    const int32_t *__restrict__ positions, const int32_t *__restrict__ lens, long long total_chunks,
    int hkv, int row_chunks, long long head_stride, int max_requests, int *err, int chain) {
    if (chain) {  // an overlapping launch: let the next one begin, wait for the previous
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    const int per_token = hkv * row_chunks;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total_chunks;
         i += (long long)gridDim.x * blockDim.x) {
        const long long t = i / per_token;
        const int rem = (int)(i - t * per_token);
        const int h = rem / row_chunks, c = rem - h * row_chunks;
        const int req = __ldg(req_ids + t);
        // the token's position, or the last position of a sequence of lens[t]
        // tokens (an empty sequence has no new token)
        const int pos = positions ? __ldg(positions + t) : __ldg(lens + t) - 1;
        if (!positions && pos < 0) continue;
        if (req < 0 || req >= max_requests || pos < 0 || (long long)pos >= mapped[req] ||
            k_bases[req] == 0) {
            if (rem == 0) atomicOr(err, KV_DEVERR_UNMAPPED);
            continue;
        }
        const long long dst = ((long long)h * head_stride + pos) * row_chunks + c;
        reinterpret_cast<uint4 *>(k_bases[req])[dst] = __ldg(k_new + i);
        reinterpret_cast<uint4 *>(v_bases[req])[dst] = __ldg(v_new + i);
    }
}

}  // namespace pkv

using namespace pkv;

struct kv_contig {
    int max_requests = 0, max_tokens = 0, hkv = 0, head_dim = 0;
    kv_dtype dtype = KV_BF16;
    int device = 0;
    size_t page = 0;            // bytes per physical page
    long long head_stride = 0;  // tokens per head region
    size_t head_bytes = 0;      // bytes per head region (a whole number of pages)
    size_t region_bytes = 0;    // K (or V) region = hkv * head_bytes
    size_t reserve_bytes = 0;   // 2 * region_bytes
    long long tokens_per_page = 0;
    struct Req {
        CUdeviceptr base = 0;
        std::vector<CUmemGenericAllocationHandle> pages;  // [2][hkv][pages_per_head], 0 = unmapped
        long long pages_mapped = 0;                       // per head region
    };
    std::vector<Req> reqs;
    long long pages_per_head = 0;
    long long mapped_bytes = 0;
    unsigned long long *d_kbase = nullptr;
    unsigned long long *d_vbase = nullptr;
    long long *d_mapped = nullptr;
    int *err = nullptr;
    int *counters = nullptr;  // fused split-merge arrival counters (see kv_pool)
    // tiled-TMA maps of each request's K and V region (bf16, head_dim 128 only)
    CUtensorMap *d_maps = nullptr;  // [max_requests][2]
    bool maps = false;
    // Physical pages kept ready off the request path ("Makale Bulteni --
    // vAttention", "Iddia ve Gerceklik": background pre-allocation threads and
    // deferred reclamation hide the latency of the VMM calls).  A worker
    // thread creates pages while fewer than `low` are spare; released
    // requests hand their pages back instead of releasing them, up to `high`.
    struct PagePool {
        std::mutex mu;
        std::condition_variable cv;
        std::deque<CUmemGenericAllocationHandle> spare;
        std::thread worker;
        bool running = false, stop = false;
        int low = 0, high = 0;
        long long created = 0, reused = 0;
        double map_ns = 0, unmap_ns = 0;
        long long maps = 0, unmaps = 0;
    } pp;
    // appends and decodes may overlap the previous kernel in the stream
    // (kv_contig_set_launch_overlap)
    bool launch_overlap = false;
};

static CUmemAllocationProp page_prop(int device) {
    CUmemAllocationProp prop{};
    prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
    prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    prop.location.id = device;
    return prop;
}

std::atomic<int> pkv::g_fail_page_create_after{-1};

// A physical page for a mapping: a spare one if the pool has it, else a new one.
static bool take_page(kv_contig *c, CUmemGenericAllocationHandle *h) {
    {
        std::lock_guard<std::mutex> lk(c->pp.mu);
        if (!c->pp.spare.empty()) {
            *h = c->pp.spare.front();
            c->pp.spare.pop_front();
            c->pp.reused += 1;
            if (c->pp.running && (int)c->pp.spare.size() < c->pp.low) c->pp.cv.notify_one();
            return true;
        }
        c->pp.created += 1;
    }
    // test hook: the creation after `after` more successful ones fails, once
    int after = g_fail_page_create_after.load();
    while (after >= 0 && !g_fail_page_create_after.compare_exchange_weak(after, after - 1)) {
    }
    if (after == 0) return false;
    const CUmemAllocationProp prop = page_prop(c->device);
    return driver().create(h, c->page, &prop, 0) == CUDA_SUCCESS;
}

// An unmapped page: kept for reuse while the pool wants it, else released.
static void give_page(kv_contig *c, CUmemGenericAllocationHandle h) {
    {
        std::lock_guard<std::mutex> lk(c->pp.mu);
        if ((int)c->pp.spare.size() < c->pp.high) {
            c->pp.spare.push_back(h);
            return;
        }
    }
    driver().release(h);
}

static void page_worker(kv_contig *c) {
    cudaSetDevice(c->device);
    const CUmemAllocationProp prop = page_prop(c->device);
    std::unique_lock<std::mutex> lk(c->pp.mu);
    while (true) {
        c->pp.cv.wait(lk, [&] { return c->pp.stop || (int)c->pp.spare.size() < c->pp.low; });
        if (c->pp.stop) break;
        const int want = c->pp.high - (int)c->pp.spare.size();
        lk.unlock();
        std::vector<CUmemGenericAllocationHandle> made;
        for (int i = 0; i < want; ++i) {
            CUmemGenericAllocationHandle h = 0;
            if (driver().create(&h, c->page, &prop, 0) != CUDA_SUCCESS) break;
            made.push_back(h);
        }
        lk.lock();
        for (auto h : made) c->pp.spare.push_back(h);
        c->pp.created += (long long)made.size();
        if (made.empty()) c->pp.cv.wait_for(lk, std::chrono::milliseconds(50));  // out of memory: back off
    }
}

static void stop_page_worker(kv_contig *c) {
    {
        std::lock_guard<std::mutex> lk(c->pp.mu);
        c->pp.stop = true;
    }
    c->pp.cv.notify_all();
    if (c->pp.worker.joinable()) c->pp.worker.join();
    c->pp.running = false;
    c->pp.stop = false;
}

static kv_status sync_request(kv_contig *c, int req) {
    const kv_contig::Req &r = c->reqs[req];
    const unsigned long long kb = r.base, vb = r.base ? r.base + c->region_bytes : 0;
    const long long mt = r.pages_mapped * c->tokens_per_page;
    if (cudaMemcpy(c->d_kbase + req, &kb, sizeof(kb), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(c->d_vbase + req, &vb, sizeof(vb), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(c->d_mapped + req, &mt, sizeof(mt), cudaMemcpyHostToDevice) != cudaSuccess)
        return KV_ERR_CUDA;
    if (c->maps && r.base) {
        // The maps describe the whole reserved region; kernels only read rows
        // below the mapped length.
        CUtensorMap m[2];
        const long long rows = (long long)c->hkv * c->head_stride;
        if (!encode_rows_map(&m[0], reinterpret_cast<void *>(kb), rows) ||
            !encode_rows_map(&m[1], reinterpret_cast<void *>(vb), rows) ||
            cudaMemcpy(c->d_maps + 2 * req, m, sizeof(m), cudaMemcpyHostToDevice) != cudaSuccess)
            return KV_ERR_CUDA;
    }
    return KV_OK;
}

extern "C" {

kv_status kv_contig_create(int max_requests, int max_tokens, int num_kv_heads, int head_dim,
                           kv_dtype dtype, kv_contig_t *out) {
    if (!out || max_requests <= 0 || max_tokens <= 0 || num_kv_heads <= 0) return KV_ERR_ARG;
    if ((head_dim != 64 && head_dim != 128) || (dtype != KV_F32 && dtype != KV_BF16 && dtype != KV_F16))
        return KV_ERR_UNSUPPORTED;
    DriverVmm &d = driver();
    if (!d.ok) return KV_ERR_CUDA;
    if (cudaFree(nullptr) != cudaSuccess) return KV_ERR_CUDA;  // make the primary context current
    kv_contig *c = new (std::nothrow) kv_contig();
    if (!c) return KV_ERR_OOM;
    cudaGetDevice(&c->device);
    c->max_requests = max_requests;
    c->max_tokens = max_tokens;
    c->hkv = num_kv_heads;
    c->head_dim = head_dim;
    c->dtype = dtype;
    CUmemAllocationProp prop{};
    prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
    prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    prop.location.id = c->device;
    if (d.getGranularity(&c->page, &prop, CU_MEM_ALLOC_GRANULARITY_MINIMUM) != CUDA_SUCCESS ||
        c->page == 0) {
        delete c;
        return KV_ERR_CUDA;
    }
    const size_t tok_bytes = (size_t)head_dim * dtype_bytes(dtype);
    if (c->page % (16 * tok_bytes) != 0) {
        delete c;
        return KV_ERR_UNSUPPORTED;
    }
    c->tokens_per_page = (long long)(c->page / tok_bytes);
    c->pages_per_head = ((long long)max_tokens + c->tokens_per_page - 1) / c->tokens_per_page;
    c->head_stride = c->pages_per_head * c->tokens_per_page;
    c->head_bytes = (size_t)c->pages_per_head * c->page;
    c->region_bytes = c->head_bytes * num_kv_heads;
    c->reserve_bytes = 2 * c->region_bytes;
    try {
        c->reqs.resize(max_requests);
    } catch (...) {
        delete c;
        return KV_ERR_OOM;
    }
    if (cudaMalloc(&c->d_kbase, sizeof(unsigned long long) * max_requests) != cudaSuccess ||
        cudaMalloc(&c->d_vbase, sizeof(unsigned long long) * max_requests) != cudaSuccess ||
        cudaMalloc(&c->d_mapped, sizeof(long long) * max_requests) != cudaSuccess ||
        cudaMalloc(&c->err, sizeof(int)) != cudaSuccess ||
        cudaMalloc(&c->counters, sizeof(int) * kv_pool::kCounterSlots) != cudaSuccess ||
        cudaMemset(c->counters, 0, sizeof(int) * kv_pool::kCounterSlots) != cudaSuccess ||
        cudaMemset(c->d_kbase, 0, sizeof(unsigned long long) * max_requests) != cudaSuccess ||
        cudaMemset(c->d_vbase, 0, sizeof(unsigned long long) * max_requests) != cudaSuccess ||
        cudaMemset(c->d_mapped, 0, sizeof(long long) * max_requests) != cudaSuccess ||
        cudaMemset(c->err, 0, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        kv_contig_destroy(c);
        return KV_ERR_OOM;
    }
    if (dtype != KV_F32 && head_dim == 128 && (long long)num_kv_heads * c->head_stride <= INT32_MAX) {
        if (cudaMalloc(&c->d_maps, sizeof(CUtensorMap) * 2 * max_requests) != cudaSuccess) {
            cudaGetLastError();
            kv_contig_destroy(c);
            return KV_ERR_OOM;
        }
        c->maps = true;
    }
    *out = c;
    return KV_OK;
}

kv_status kv_contig_layout(kv_contig_t c, int64_t *head_stride, int64_t *page_bytes,
                           int64_t *reserved_bytes_per_request) {
    if (!c) return KV_ERR_ARG;
    if (head_stride) *head_stride = c->head_stride;
    if (page_bytes) *page_bytes = (int64_t)c->page;
    if (reserved_bytes_per_request) *reserved_bytes_per_request = (int64_t)c->reserve_bytes;
    return KV_OK;
}

kv_status kv_contig_reserve(kv_contig_t c, int req) {
    if (!c || req < 0 || req >= c->max_requests) return KV_ERR_ARG;
    if (kv_status st = require_device(c->device)) return st;
    kv_contig::Req &r = c->reqs[req];
    if (r.base) return KV_ERR_STATE;
    DriverVmm &d = driver();
    CUdeviceptr base = 0;
    if (d.addressReserve(&base, c->reserve_bytes, c->page, 0, 0) != CUDA_SUCCESS) return KV_ERR_OOM;
    try {
        r.pages.assign((size_t)2 * c->hkv * c->pages_per_head, 0);
    } catch (...) {
        d.addressFree(base, c->reserve_bytes);
        return KV_ERR_OOM;
    }
    r.base = base;
    r.pages_mapped = 0;
    return sync_request(c, req);
}

kv_status kv_contig_ensure(kv_contig_t c, int req, int64_t n_tokens) {
    if (!c || req < 0 || req >= c->max_requests || n_tokens < 0 || n_tokens > c->max_tokens)
        return KV_ERR_ARG;
    if (kv_status st = require_device(c->device)) return st;
    kv_contig::Req &r = c->reqs[req];
    if (!r.base) return KV_ERR_STATE;
    const long long need = (n_tokens + c->tokens_per_page - 1) / c->tokens_per_page;
    if (need <= r.pages_mapped) return KV_OK;
    DriverVmm &d = driver();
    CUmemAllocationProp prop{};
    prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
    prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    prop.location.id = c->device;
    CUmemAccessDesc access{};
    access.location = prop.location;
    access.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    std::vector<size_t> made;  // page slots filled by this call (for undo)
    kv_status st = KV_OK;
    for (int kv = 0; kv < 2 && st == KV_OK; ++kv)
        for (int h = 0; h < c->hkv && st == KV_OK; ++h)
            for (long long k = r.pages_mapped; k < need; ++k) {
                const size_t slot = ((size_t)kv * c->hkv + h) * c->pages_per_head + k;
                const CUdeviceptr va = r.base + kv * c->region_bytes + h * c->head_bytes + k * c->page;
                CUmemGenericAllocationHandle hdl = 0;
                const auto t0 = std::chrono::steady_clock::now();
                if (!take_page(c, &hdl)) {
                    st = KV_ERR_OOM;
                    break;
                }
                if (d.map(va, c->page, 0, hdl, 0) != CUDA_SUCCESS) {
                    give_page(c, hdl);
                    st = KV_ERR_CUDA;
                    break;
                }
                r.pages[slot] = hdl;
                made.push_back(slot);
                if (d.setAccess(va, c->page, &access, 1) != CUDA_SUCCESS) {
                    st = KV_ERR_CUDA;
                    break;
                }
                c->pp.map_ns += std::chrono::duration<double, std::nano>(std::chrono::steady_clock::now() - t0).count();
                c->pp.maps += 1;
            }
    if (st != KV_OK) {
        for (size_t slot : made) {
            const size_t kv = slot / ((size_t)c->hkv * c->pages_per_head);
            const size_t rem = slot % ((size_t)c->hkv * c->pages_per_head);
            const size_t h = rem / c->pages_per_head, k = rem % c->pages_per_head;
            d.unmap(r.base + kv * c->region_bytes + h * c->head_bytes + k * c->page, c->page);
            give_page(c, r.pages[slot]);
            r.pages[slot] = 0;
        }
        return st;
    }
    c->mapped_bytes += (long long)made.size() * (long long)c->page;
    r.pages_mapped = need;
    return sync_request(c, req);
}

kv_status kv_contig_release(kv_contig_t c, int req) {
    if (!c || req < 0 || req >= c->max_requests) return KV_ERR_ARG;
    if (kv_status st = require_device(c->device)) return st;
    kv_contig::Req &r = c->reqs[req];
    if (!r.base) return KV_OK;
    DriverVmm &d = driver();
    kv_status st = KV_OK;
    for (size_t slot = 0; slot < r.pages.size(); ++slot) {
        if (!r.pages[slot]) continue;
        const size_t kv = slot / ((size_t)c->hkv * c->pages_per_head);
        const size_t rem = slot % ((size_t)c->hkv * c->pages_per_head);
        const size_t h = rem / c->pages_per_head, k = rem % c->pages_per_head;
        const auto t0 = std::chrono::steady_clock::now();
        if (d.unmap(r.base + kv * c->region_bytes + h * c->head_bytes + k * c->page, c->page) !=
            CUDA_SUCCESS)
            st = KV_ERR_CUDA;
        else
            give_page(c, r.pages[slot]);  // deferred reclamation: kept for reuse while wanted
        c->pp.unmap_ns += std::chrono::duration<double, std::nano>(std::chrono::steady_clock::now() - t0).count();
        c->pp.unmaps += 1;
        r.pages[slot] = 0;
        c->mapped_bytes -= (long long)c->page;
    }
    if (d.addressFree(r.base, c->reserve_bytes) != CUDA_SUCCESS) st = KV_ERR_CUDA;
    r.base = 0;
    r.pages_mapped = 0;
    r.pages.clear();
    kv_status s2 = sync_request(c, req);
    return st != KV_OK ? st : s2;
}

kv_status kv_contig_destroy(kv_contig_t c) {
    if (!c) return KV_ERR_ARG;
    // unmap and free on the context's own device, then give the caller its
    // device back
    int cur = -1;
    const bool switched = cudaGetDevice(&cur) == cudaSuccess && cur != c->device &&
                          cudaSetDevice(c->device) == cudaSuccess;
    stop_page_worker(c);
    c->pp.high = 0;  // released pages are not kept any more
    for (int r = 0; r < c->max_requests; ++r)
        if (c->reqs[r].base && c->d_kbase) kv_contig_release(c, r);
    for (auto h : c->pp.spare) driver().release(h);
    c->pp.spare.clear();
    if (c->d_kbase) cudaFree(c->d_kbase);
    if (c->d_vbase) cudaFree(c->d_vbase);
    if (c->d_mapped) cudaFree(c->d_mapped);
    if (c->err) cudaFree(c->err);
    if (c->counters) cudaFree(c->counters);
    if (c->d_maps) cudaFree(c->d_maps);
    if (switched) cudaSetDevice(cur);
    delete c;
    return KV_OK;
}

kv_status kv_contig_page_pool(kv_contig_t c, int low, int high) {
    if (!c || low < 0 || high < low) return KV_ERR_ARG;
    stop_page_worker(c);
    std::vector<CUmemGenericAllocationHandle> drop;
    {
        std::lock_guard<std::mutex> lk(c->pp.mu);
        c->pp.low = low;
        c->pp.high = high;
        while ((int)c->pp.spare.size() > high) {
            drop.push_back(c->pp.spare.back());
            c->pp.spare.pop_back();
        }
    }
    for (auto h : drop) driver().release(h);
    if (low > 0) {
        try {
            c->pp.worker = std::thread(page_worker, c);
        } catch (...) {
            return KV_ERR_OOM;
        }
        c->pp.running = true;
    }
    return KV_OK;
}

kv_status kv_contig_page_stats(kv_contig_t c, int *spare_pages, int64_t *created, int64_t *reused,
                               double *map_us_per_page, double *unmap_us_per_page) {
    if (!c) return KV_ERR_ARG;
    std::lock_guard<std::mutex> lk(c->pp.mu);
    if (spare_pages) *spare_pages = (int)c->pp.spare.size();
    if (created) *created = c->pp.created;
    if (reused) *reused = c->pp.reused;
    if (map_us_per_page) *map_us_per_page = c->pp.maps ? c->pp.map_ns / c->pp.maps / 1e3 : 0.0;
    if (unmap_us_per_page) *unmap_us_per_page = c->pp.unmaps ? c->pp.unmap_ns / c->pp.unmaps / 1e3 : 0.0;
    return KV_OK;
}

kv_status kv_contig_ptrs(kv_contig_t c, int req, void **k_base, void **v_base) {
    if (!c || req < 0 || req >= c->max_requests) return KV_ERR_ARG;
    const kv_contig::Req &r = c->reqs[req];
    if (!r.base) return KV_ERR_STATE;
    if (k_base) *k_base = reinterpret_cast<void *>(r.base);
    if (v_base) *v_base = reinterpret_cast<void *>(r.base + c->region_bytes);
    return KV_OK;
}

kv_status kv_contig_stats(kv_contig_t c, int req, int64_t *mapped_tokens,
                          int64_t *mapped_bytes_total) {
    if (!c || req < 0 || req >= c->max_requests) return KV_ERR_ARG;
    if (mapped_tokens) *mapped_tokens = c->reqs[req].pages_mapped * c->tokens_per_page;
    if (mapped_bytes_total) *mapped_bytes_total = c->mapped_bytes;
    return KV_OK;
}

// Writes num_tokens K/V rows into their requests' head regions: token t at
// positions[t], or (positions null) at lens[t] - 1.
static kv_status contig_append_rows(kv_contig_t c, const void *k_new, const void *v_new,
                                    const int32_t *req_ids, const int32_t *positions,
                                    const int32_t *lens, int num_tokens, void *stream) {
    const int row_chunks = c->head_dim * dtype_bytes(c->dtype) / 16;
    const long long total = (long long)num_tokens * c->hkv * row_chunks;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (c->launch_overlap) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(256);
        cfg.stream = as_stream(stream);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cuda_status(cudaLaunchKernelEx(
            &cfg, contig_append_kernel, (const unsigned long long *)c->d_kbase,
            (const unsigned long long *)c->d_vbase, (const long long *)c->d_mapped,
            (const uint4 *)k_new, (const uint4 *)v_new, req_ids, positions, lens, total, c->hkv,
            row_chunks, c->head_stride, c->max_requests, c->err, 1));
    }
    contig_append_kernel<<<(int)blocks, 256, 0, as_stream(stream)>>>(
        c->d_kbase, c->d_vbase, c->d_mapped, (const uint4 *)k_new, (const uint4 *)v_new, req_ids,
        positions, lens, total, c->hkv, row_chunks, c->head_stride, c->max_requests, c->err, 0);
    return cuda_status(cudaGetLastError());
}

kv_status kv_contig_append(kv_contig_t c, const void *k_new, const void *v_new,
                           const int32_t *req_ids, const int32_t *positions, int num_tokens,
                           void *stream) {
    if (!c || num_tokens < 0) return KV_ERR_ARG;
    if (kv_status st = require_device(c->device)) return st;
    if (num_tokens == 0) return KV_OK;
    if (!k_new || !v_new || !req_ids || !positions) return KV_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
        return KV_ERR_ARG;
    return contig_append_rows(c, k_new, v_new, req_ids, positions, nullptr, num_tokens, stream);
}

static DecodeArgs contig_decode_args(kv_contig_t c, const void *q, const int32_t *req_ids,
                                     const int32_t *seq_lens, int batch, int num_q_heads,
                                     float scale, void *out, kv_dtype out_dtype, float *lse_out,
                                     int num_splits, void *workspace, size_t workspace_bytes,
                                     void *stream) {
    DecodeArgs a{};
    a.q = q;
    a.max_blocks = (c->max_tokens + 15) / 16;  // the split plan of an equal-width block table
    a.k_bases = c->d_kbase;
    a.v_bases = c->d_vbase;
    a.req_ids = req_ids;
    a.mapped_tokens = c->d_mapped;
    a.req_maps = c->maps ? c->d_maps : nullptr;
    a.head_stride = c->head_stride;
    a.max_requests = c->max_requests;
    a.seq_lens = seq_lens;
    a.batch = batch;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = c->hkv;
    a.head_dim = c->head_dim;
    a.dtype = c->dtype;
    a.scale = scale;
    a.out = out;
    a.out_dtype = out_dtype;
    a.lse = lse_out;
    a.num_splits = num_splits;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.err = c->err;
    a.counters = c->counters;
    a.counter_slots = kv_pool::kCounterSlots;
    a.stream = as_stream(stream);
    a.chain = c->launch_overlap;
    return a;
}

kv_status contig_decode_attention(kv_contig_t c, const void *q, const int32_t *req_ids,
                                  const int32_t *seq_lens, int batch, int num_q_heads,
                                  float scale, void *out, kv_dtype out_dtype, float *lse_out,
                                  int num_splits, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    if (!c || (batch > 0 && !req_ids)) return KV_ERR_ARG;
    if (kv_status st = require_device(c->device)) return st;
    const DecodeArgs a = contig_decode_args(c, q, req_ids, seq_lens, batch, num_q_heads, scale, out,
                                            out_dtype, lse_out, num_splits, workspace,
                                            workspace_bytes, stream);
    return launch_decode(a, true);
}

kv_status contig_append_and_decode(kv_contig_t c, const void *q, const void *k_new,
                                   const void *v_new, const int32_t *req_ids,
                                   const int32_t *seq_lens, int batch, int num_q_heads,
                                   float scale, void *out, kv_dtype out_dtype, float *lse_out,
                                   int num_splits, void *workspace, size_t workspace_bytes,
                                   void *stream) {
    if (!c || batch < 0) return KV_ERR_ARG;
    if (batch == 0) return KV_OK;
    if (!req_ids || !seq_lens || !k_new || !v_new) return KV_ERR_ARG;
    if (kv_status st = require_device(c->device)) return st;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
        return KV_ERR_ARG;
    DecodeArgs a = contig_decode_args(c, q, req_ids, seq_lens, batch, num_q_heads, scale, out,
                                      out_dtype, lse_out, num_splits, workspace, workspace_bytes,
                                      stream);
    a.new_k = k_new;
    a.new_v = v_new;
    const kv_status st = launch_decode(a, true);
    if (st != KV_ERR_UNSUPPORTED) return st;
    // shapes the fused kernel does not cover: the append, then the decode
    if (kv_status st1 = contig_append_rows(c, k_new, v_new, req_ids, nullptr, seq_lens, batch, stream))
        return st1;
    a.new_k = a.new_v = nullptr;
    return launch_decode(a, true);
}

kv_status kv_contig_set_launch_overlap(kv_contig_t c, int enable) {
    if (!c || (enable != 0 && enable != 1)) return KV_ERR_ARG;
    c->launch_overlap = enable != 0;
    return KV_OK;
}

kv_status kv_debug_fail_page_create(int after) {
    g_fail_page_create_after.store(after < 0 ? -1 : after);
    return KV_OK;
}

kv_status kv_contig_get_device_error(kv_contig_t c, int *code, void *stream) {
    if (!c || !code) return KV_ERR_ARG;
    if (kv_status st = require_device(c->device)) return st;
    int h = 0;
    cudaStream_t s = as_stream(stream);
    if (cudaMemcpyAsync(&h, c->err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return KV_ERR_CUDA;
    if (h != 0 && (cudaMemsetAsync(c->err, 0, sizeof(int), s) != cudaSuccess ||
                   cudaMemsetAsync(c->counters, 0, sizeof(int) * kv_pool::kCounterSlots, s) !=
                       cudaSuccess))
        return KV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KV_ERR_CUDA;
    *code = h;
    return device_error_status(h);
}

}  // extern "C"
