// Chunked causal paged prefill on the tcgen05 tensor cores.
//
// "Makale Bulteni -- vAttention", section "Iddia ve Gerceklik": paged prefill
// kernels (FlashAttention-2, FlashInfer) are the ones that lose most to
// block-table indirection.  Here the indirection is paid once per 16-token
// block: the producer turns each block-table entry into two tiled TMA copies
// (one per 64-dimension half of the head) that land in the same swizzled
// shared-memory tile a contiguous kernel would build, so the tensor-core
// part does not know the keys were paged.
//
// Maths: sequence b holds L = seq_lens[b] tokens; its last T tokens are the
// new chunk, already written to the pool.  Query i of the chunk sits at
// position c + i (c = L - T) and attends keys 0..c+i: o = softmax(scale q K^T) V.
// The score matrix is never written to memory ("PagedAttention Nedir?",
// "FlashAttention ile Ayni mi?").
//
// One CTA = one 128-query tile of one query head of one sequence, 192 threads:
//   warps 0-3  softmax: thread r owns query row r (tensor-memory lane r);
//   warp 4     TMA producer: Q once, then K and V tiles of 128 keys (8 blocks)
//              into a 2-deep ring per operand;
//   warp 5     MMA issuer: S = Q K^T and O += P V with tcgen05.mma
//              (M=128, N=128, K=16 steps), fp32 accumulators in tensor memory.
// Tensor memory (512 columns): S ping-pong [0,128) and [128,256), O
// [256,384), P ping-pong (bf16 pairs) [384,448) and [448,512).  While the
// softmax warps turn S_j into P_j the tensor core already computes S_{j+1}.
//
// Online softmax keeps a per-row reference maximum m and rescales O and the
// row sum only when the running maximum exceeds m by more than 2^8, so the
// unnormalised weights stay <= 256 (exact maths: O and the sum share m).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace pkv {

constexpr int kPfBM = 128;           // queries per CTA
constexpr int kPfBN = 128;           // keys per tile
constexpr int kPfD = 128;            // head dim (only size supported)
constexpr int kPfThreads = 192;
constexpr int kPfHalfBytes = 128 * 128;         // 128 rows x 64 bf16 (one half of D)
constexpr int kPfTileBytes = 2 * kPfHalfBytes;  // 128 rows x 128 bf16
constexpr int kPfQOff = 0;
constexpr int kPfKOff = kPfTileBytes;                 // 2 stages
constexpr int kPfVOff = kPfKOff + 2 * kPfTileBytes;   // 2 stages
constexpr int kPfBarOff = kPfVOff + 2 * kPfTileBytes; // 160 KiB
constexpr int kPfSmemBytes = kPfBarOff + 256 + 1024;  // barriers, slot, alignment slack
constexpr float kRescaleThreshold = 8.0f;             // log2 units

// 2^x with the hardware approximation (relative error ~2^-22, far below the
// bf16 rounding the weights get next); -inf gives 0.
KV_DEVICE float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// TMEM column map
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP0 = 384, kColP1 = 448;

struct PrefillParams {
    const int32_t *cu_q;
    int total_q;
    const int32_t *tables;
    const int32_t *seq_lens;
    int max_blocks;
    int num_blocks;
    int num_q_heads;
    int num_kv_heads;
    int g;
    float scale_log2;
    void *out;
    int out_bf16;
    float *lse;
    int *err;
};

struct PfBars {
    uint64_t qfull;
    uint64_t kfull[2], vfull[2], kempty[2], vempty[2];
    uint64_t sfull[2], pfull[2], pfree[2];
    uint32_t tmem_slot;
    int abort;
};

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    const int hq = blockIdx.x, qt = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q_begin = p.cu_q[b];
    const int T = p.cu_q[b + 1] - q_begin;
    const int q0 = qt * kPfBM;
    if (q0 >= T) return;  // uniform: this sequence's chunk has no tile here
    long long L = p.seq_lens[b];
    const long long c = L - T;
    if (c < 0 || L > (long long)p.max_blocks * 16 || q_begin < 0 || q_begin + T > p.total_q) {
        if (tid == 0) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
        return;
    }
    const int h = hq / p.g;
    const long long kv_end = c + min(q0 + kPfBM, T);  // keys any row of this tile can see
    const int n = (int)((kv_end + kPfBN - 1) / kPfBN);
    const int nblk = (int)((L + 15) / 16);

    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    char *sQ = smem + kPfQOff;
    char *sK = smem + kPfKOff;
    char *sV = smem + kPfVOff;
    PfBars *bars = reinterpret_cast<PfBars *>(smem + kPfBarOff);

    if (warp == 5) {
        tc::tmem_alloc(&bars->tmem_slot, 512);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bars->qfull, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->kfull[s], 1);
            mbar_init(&bars->vfull[s], 1);
            mbar_init(&bars->kempty[s], 1);
            mbar_init(&bars->vempty[s], 1);
            mbar_init(&bars->sfull[s], 1);
            mbar_init(&bars->pfull[s], 128);
            mbar_init(&bars->pfree[s], 1);
        }
        bars->abort = 0;
        mbar_init_fence();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars->tmem_slot;
    volatile int *abort_flag = &bars->abort;

    if (warp == 4) {
        // ================================================== TMA producer
        if (lane == 0) {
            tc::prefetch_tensormap(&tm_q);
            tc::prefetch_tensormap(&tm_k);
            tc::prefetch_tensormap(&tm_v);
            mbar_arrive_expect_tx(&bars->qfull, kPfTileBytes);
            tc::tma_load_3d(sQ, &tm_q, 0, hq, q_begin + q0, &bars->qfull);
            tc::tma_load_3d(sQ + kPfHalfBytes, &tm_q, 64, hq, q_begin + q0, &bars->qfull);
            const int32_t *row = p.tables + (size_t)b * p.max_blocks;
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < n && !*abort_flag; ++j) {
                const int s = j & 1;
                int ys[8];
#pragma unroll
                for (int bi = 0; bi < 8; ++bi) {
                    const int ib = j * 8 + bi;
                    int y = -16;  // rows -16..-1: outside the tensor, read as zeros
                    if (ib < nblk) {
                        const int id = __ldg(row + ib);
                        if (id >= 0 && id < p.num_blocks)
                            y = (id * p.num_kv_heads + h) * 16;
                        else
                            atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
                    }
                    ys[bi] = y;
                }
                if (j >= 2 && !mbar_wait(&bars->kempty[s], ((j - 2) >> 1) & 1, p.err)) {
                    *abort_flag = 1;
                    break;
                }
                char *dk = sK + s * kPfTileBytes;
                mbar_arrive_expect_tx(&bars->kfull[s], kPfTileBytes);
#pragma unroll
                for (int bi = 0; bi < 8; ++bi) {
                    tc::tma_load_2d(dk + bi * 2048, &tm_k, 0, ys[bi], &bars->kfull[s]);
                    tc::tma_load_2d(dk + kPfHalfBytes + bi * 2048, &tm_k, 64, ys[bi], &bars->kfull[s]);
                }
                k_issued = j + 1;
                if (j >= 2 && !mbar_wait(&bars->vempty[s], ((j - 2) >> 1) & 1, p.err)) {
                    *abort_flag = 1;
                    break;
                }
                char *dv = sV + s * kPfTileBytes;
                mbar_arrive_expect_tx(&bars->vfull[s], kPfTileBytes);
#pragma unroll
                for (int bi = 0; bi < 8; ++bi) {
                    tc::tma_load_2d(dv + bi * 2048, &tm_v, 0, ys[bi], &bars->vfull[s]);
                    tc::tma_load_2d(dv + kPfHalfBytes + bi * 2048, &tm_v, 64, ys[bi], &bars->vfull[s]);
                }
                v_issued = j + 1;
            }
            // Never leave copies in flight into this CTA's shared memory.
            mbar_wait(&bars->qfull, 0, p.err);
            for (int j = (k_issued > 2 ? k_issued - 2 : 0); j < k_issued; ++j)
                mbar_wait(&bars->kfull[j & 1], (j >> 1) & 1, p.err);
            for (int j = (v_issued > 2 ? v_issued - 2 : 0); j < v_issued; ++j)
                mbar_wait(&bars->vfull[j & 1], (j >> 1) & 1, p.err);
        }
    } else if (warp == 5) {
        // ================================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(128, 128, false, true);
            const uint32_t q_addr = smem_addr(sQ), k_addr = smem_addr(sK), v_addr = smem_addr(sV);
            auto issue_s = [&](int j) {
                const int s = j & 1;
                const uint32_t d = tmem + (s ? kColS1 : kColS0);
                const uint32_t kb = k_addr + s * kPfTileBytes;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t da = tc::smem_desc_sw128(q_addr + hh * kPfHalfBytes + kk * 32, 16, 1024);
                        const uint64_t db = tc::smem_desc_sw128(kb + hh * kPfHalfBytes + kk * 32, 16, 1024);
                        tc::mma_ss(d, da, db, idesc_qk, (hh | kk) != 0);
                    }
                tc::mma_commit(&bars->sfull[s]);
                tc::mma_commit(&bars->kempty[s]);
            };
            bool ok = mbar_wait(&bars->qfull, 0, p.err);
            for (int j = 0; ok && j < 2 && j < n; ++j) {
                ok = mbar_wait(&bars->kfull[j], 0, p.err);
                if (ok) {
                    tc::fence_after_sync();
                    issue_s(j);
                }
            }
            for (int j = 0; ok && j < n; ++j) {
                const int s = j & 1;
                if (!mbar_wait(&bars->pfull[s], (j >> 1) & 1, p.err) ||
                    !mbar_wait(&bars->vfull[s], (j >> 1) & 1, p.err)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t pcol = tmem + (s ? kColP1 : kColP0);
                const uint32_t vb = v_addr + s * kPfTileBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    // B = V tile, keys 16kk..16kk+15 x all 128 dims (MN-major):
                    // the two 64-dim halves are 16 KiB apart, 8-key groups 1 KiB apart.
                    const uint64_t db = tc::smem_desc_sw128(vb + kk * 2048, kPfHalfBytes, 1024);
                    tc::mma_ts(tmem + kColO, pcol + kk * 8, db, idesc_pv, (j | kk) != 0);
                }
                tc::mma_commit(&bars->pfree[s]);
                tc::mma_commit(&bars->vempty[s]);
                if (j + 2 < n) {
                    if (!mbar_wait(&bars->kfull[s], ((j + 2) >> 1) & 1, p.err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    issue_s(j + 2);
                }
            }
            if (!ok) *abort_flag = 1;
        }
    } else {
        // ================================================== softmax warps
        const int r = tid;  // query row = TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const bool row_valid = q0 + r < T;
        // Invalid rows (past the chunk) see every key; they are never stored.
        const long long qpos = row_valid ? c + q0 + r : L - 1;
        float m_used = -INFINITY, l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            if (*abort_flag) { ok = false; break; }
            const int s = j & 1;
            if (!mbar_wait(&bars->sfull[s], (j >> 1) & 1, p.err)) { ok = false; break; }
            tc::fence_after_sync();
            // S row: four 32-column loads in flight, one wait.
            uint32_t sv[128];
            {
                uint32_t (&a)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sv[0]);
                uint32_t (&b2)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sv[32]);
                uint32_t (&c2)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sv[64]);
                uint32_t (&d2)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sv[96]);
                const uint32_t sc = tmem + lane_base + (s ? kColS1 : kColS0);
                tc::tmem_ld32(sc, a);
                tc::tmem_ld32(sc + 32, b2);
                tc::tmem_ld32(sc + 64, c2);
                tc::tmem_ld32(sc + 96, d2);
                tc::tmem_wait_ld();
            }
            const long long key0 = (long long)j * kPfBN;
            if (key0 + kPfBN - 1 > qpos) {
                // diagonal tile: keys past this row's position get -inf
#pragma unroll
                for (int k = 0; k < 128; ++k)
                    if (key0 + k > qpos) sv[k] = __float_as_uint(-INFINITY);
            }
            // raw row maximum with eight independent chains (scale > 0, so
            // max(scale * s) = scale * max(s))
            float mx[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mx[k] = __uint_as_float(sv[k]);
#pragma unroll
            for (int k = 8; k < 128; ++k) mx[k & 7] = fmaxf(mx[k & 7], __uint_as_float(sv[k]));
            const float mrow = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
                               p.scale_log2;
            float alpha = 1.f;
            bool rescale = false;
            if (j == 0) {
                m_used = mrow;
            } else if (mrow > m_used + kRescaleThreshold) {
                alpha = ex2_approx(m_used - mrow);
                m_used = mrow;
                l_sum *= alpha;
                rescale = true;
            }
            // P_j goes into buffer s: PV_{j-2} must have consumed it.
            if (j >= 2 && !mbar_wait(&bars->pfree[s], ((j - 2) >> 1) & 1, p.err)) { ok = false; break; }
            if (__any_sync(0xffffffffu, rescale)) {
                // O must hold PV_{j-1} before it is rescaled.
                const int sp = (j - 1) & 1;
                if (!mbar_wait(&bars->pfree[sp], ((j - 1) >> 1) & 1, p.err)) { ok = false; break; }
                tc::fence_after_sync();
                uint32_t v[32];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    tc::tmem_ld32(tmem + lane_base + kColO + 32 * i, v);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
                    tc::tmem_st32(tmem + lane_base + kColO + 32 * i, v);
                }
                tc::tmem_wait_st();
            }
            // p = 2^(scale*s - m): packed fma, hardware exp2, bf16 pairs
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
            const float2 nm2 = make_float2(-m_used, -m_used);
            float2 acc2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                              make_float2(0.f, 0.f)};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t w[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[64 * half + 2 * k]),
                                                            __uint_as_float(sv[64 * half + 2 * k + 1])),
                                                sc2, nm2);
                    const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    acc2[k & 3] = __fadd2_rn(acc2[k & 3], e);
                    w[k] = tc::pack_bf16x2(e.x, e.y);
                }
                tc::tmem_st32(tmem + lane_base + (s ? kColP1 : kColP0) + 32 * half, w);
            }
            l_sum += (acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y) + (acc2[2].x + acc2[2].y) +
                     (acc2[3].x + acc2[3].y);
            tc::tmem_wait_st();
            if (key0 + kPfBN > L) {
                // Keys at or past L: the V rows there may hold anything; zero
                // them so the zero weights cannot meet a NaN in the tensor core.
                if (!mbar_wait(&bars->vfull[s], (j >> 1) & 1, p.err)) { ok = false; break; }
                const int first = (int)(L - key0);
                char *vt = sV + s * kPfTileBytes;
                for (int idx = r; idx < (kPfBN - first) * 16; idx += 128) {
                    const int row = first + idx / 16, chunk = idx % 16;
                    *reinterpret_cast<uint4 *>(vt + (chunk >> 3) * kPfHalfBytes + row * 128 +
                                               (chunk & 7) * 16) = make_uint4(0, 0, 0, 0);
                }
                tc::fence_proxy_async_smem();
            }
            tc::fence_before_sync();
            mbar_arrive(&bars->pfull[s]);
        }
        // ---- epilogue: O / l for this row
        if (ok && n > 0) {
            const int sl = (n - 1) & 1;
            ok = mbar_wait(&bars->pfree[sl], ((n - 1) >> 1) & 1, p.err);
        }
        if (!ok) *abort_flag = 1;
        tc::fence_after_sync();
        const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
        const size_t orow = ((size_t)(q_begin + q0 + r) * p.num_q_heads + hq) * kPfD;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t v[32];
            tc::tmem_ld32(tmem + lane_base + kColO + 32 * i, v);
            tc::tmem_wait_ld();
            if (row_valid && ok) {
                if (p.out_bf16) {
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.out) + orow + 32 * i);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint4 u;
                        u.x = tc::pack_bf16x2(__uint_as_float(v[8 * k + 0]) * inv, __uint_as_float(v[8 * k + 1]) * inv);
                        u.y = tc::pack_bf16x2(__uint_as_float(v[8 * k + 2]) * inv, __uint_as_float(v[8 * k + 3]) * inv);
                        u.z = tc::pack_bf16x2(__uint_as_float(v[8 * k + 4]) * inv, __uint_as_float(v[8 * k + 5]) * inv);
                        u.w = tc::pack_bf16x2(__uint_as_float(v[8 * k + 6]) * inv, __uint_as_float(v[8 * k + 7]) * inv);
                        dst[k] = u;
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + orow + 32 * i);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(v[4 * k]) * inv, __uint_as_float(v[4 * k + 1]) * inv,
                                             __uint_as_float(v[4 * k + 2]) * inv, __uint_as_float(v[4 * k + 3]) * inv);
                }
            }
        }
        if (row_valid && ok && p.lse)
            p.lse[(size_t)(q_begin + q0 + r) * p.num_q_heads + hq] =
                l_sum > 0.f ? (m_used + log2f(l_sum)) * 0.6931471805599453f : -INFINITY;
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace pkv

using namespace pkv;

extern "C" kv_status paged_prefill_attention(kv_pool_t p, const void *q, const int32_t *cu_q,
                                             int total_q, int max_q_len, const int32_t *block_tables,
                                             int max_blocks, const int32_t *seq_lens, int batch,
                                             int num_q_heads, float scale, void *out,
                                             kv_dtype out_dtype, float *lse_out, void *stream) {
    if (!p || batch < 0 || total_q < 0 || max_q_len < 0 || max_blocks < 0 || num_q_heads <= 0)
        return KV_ERR_ARG;
    if (p->dtype != KV_BF16 || p->head_dim != kPfD) return KV_ERR_UNSUPPORTED;
    if (num_q_heads % p->num_kv_heads) return KV_ERR_ARG;
    if (out_dtype != KV_F32 && out_dtype != KV_BF16) return KV_ERR_UNSUPPORTED;
    if (batch == 0 || max_q_len == 0 || total_q == 0) return KV_OK;
    if (!q || !cu_q || !block_tables || !seq_lens || !out) return KV_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(q) & 15) return KV_ERR_ARG;
    const long long pool_rows = (long long)p->num_blocks * p->num_kv_heads * 16;
    if (pool_rows > INT32_MAX || batch > 65535) return KV_ERR_UNSUPPORTED;
    if (pool_tensor_maps(p) != KV_OK) return KV_ERR_CUDA;
    // The q map covers exactly total_q rows: a tile reaching past them reads
    // zeros, and rows past a chunk or past total_q are never stored.
    CUtensorMap tm_q;
    if (!encode_q_map(&tm_q, q, total_q, num_q_heads)) return KV_ERR_CUDA;
    PrefillParams pp{};
    pp.cu_q = cu_q;
    pp.total_q = total_q;
    pp.tables = block_tables;
    pp.seq_lens = seq_lens;
    pp.max_blocks = max_blocks;
    pp.num_blocks = p->num_blocks;
    pp.num_q_heads = num_q_heads;
    pp.num_kv_heads = p->num_kv_heads;
    pp.g = num_q_heads / p->num_kv_heads;
    pp.scale_log2 = scale * 1.4426950408889634f;
    pp.out = out;
    pp.out_bf16 = out_dtype == KV_BF16;
    pp.lse = lse_out;
    pp.err = p->err;
    if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPfSmemBytes) != cudaSuccess)
        return KV_ERR_CUDA;
    const dim3 grid(num_q_heads, (max_q_len + kPfBM - 1) / kPfBM, batch);
    prefill_kernel<<<grid, kPfThreads, kPfSmemBytes, as_stream(stream)>>>(tm_q, p->tmap_k,
                                                                         p->tmap_v, pp);
    return cuda_status(cudaGetLastError());
}
