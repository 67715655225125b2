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
// One CTA = two 128-query tiles (A: rows 0-127, B: rows 128-255 of a 256-query
// slice) of one query head of one sequence; every K/V tile of 128 keys (8
// blocks) is loaded once and used by both.  384 threads:
//   warps 0-3  softmax of tile A (thread = query row = tensor-memory lane)
//   warps 4-7  softmax of tile B
//   warp 8     TMA producer: Q once, K into a 2-deep ring
//   warp 9     MMA issuer (tcgen05.mma, M=128, N=128, K=16 steps, fp32 in TMEM)
//   warp 10    TMA producer: V into a 3-deep ring
// Each softmax warp also rewrites an eighth of every landed V tile in place
// as fp16 (tile 0 first, tile j+1 right after handing P(j) to the tensor
// core, while it waits for S(j+1)); the MMA issuer reads a V tile only once
// all eight parts are done.
// QK^T multiplies bf16 operands (exact products, fp32 sums).  PV multiplies
// fp16 weights by fp16 V: one MMA takes one operand type, and bf16 weights
// (8 significant bits) would leave an error of about 2e-3 of the output
// scale, the whole tolerance; fp16 (11 bits) leaves about 3e-4.  bf16 V
// converts to fp16 exactly for magnitudes in [2^-14, 65280]; larger attended
// values saturate to +-65504 and set KV_DEVERR_VALUE_RANGE.
// Tensor memory (512 columns): S_A [0,128), S_B [128,256), O_A [256,384),
// O_B [384,512); each tile's fp16 weights P overwrite the first 64 columns of
// its S once read.  MMA issue order per key tile j:
//   ... PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) ...
// so while one softmax group turns S into P the tensor core works for the
// other.  tcgen05.mma operations of one thread run in issue order, which
// orders PV_X(j)'s read of P before S_X(j+1) overwrites it, and makes the
// completion of S_X(j+1) imply that of PV_X(j) (so O_X is stable when the
// softmax warps see S_X(j+1)).
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

constexpr int kPfBM = 256;           // queries per CTA (two tensor-core tiles)
constexpr int kPfBN = 128;           // keys per tile
constexpr int kPfD = 128;            // head dim (only size supported)
constexpr int kPfThreads = 352;  // 8 softmax warps, MMA issuer, K and V producers
constexpr int kPfProducerWarp = 8, kPfMmaWarp = 9, kPfVProducerWarp = 10;
constexpr int kPfHalfBytes = 128 * 128;         // 128 rows x 64 bf16 (one half of D)
constexpr int kPfTileBytes = 2 * kPfHalfBytes;  // 128 rows x 128 bf16
constexpr int kPfVStages = 3;                          // V ring depth (K: 2)
constexpr int kPfQOff = 0;                             // Q_A, Q_B
constexpr int kPfKOff = 2 * kPfTileBytes;              // 2 stages
constexpr int kPfVOff = kPfKOff + 2 * kPfTileBytes;    // kPfVStages stages
constexpr int kPfBarOff = kPfVOff + kPfVStages * kPfTileBytes;  // 224 KiB
constexpr int kPfSmemBytes = kPfBarOff + 256 + 1024;   // barriers, slot, alignment slack
static_assert(kPfSmemBytes <= 227 * 1024, "prefill shared memory exceeds the per-CTA limit");
constexpr float kRescaleThreshold = 8.0f;              // log2 units

// 2^x with the hardware approximation (relative error ~2^-22, far below the
// fp16 rounding the weights get next); -inf gives 0.
KV_DEVICE float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction
KV_DEVICE float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// TMEM column map: S of tile x at colS(x), O of tile x at colO(x)
KV_DEVICE constexpr uint32_t colS(int x) { return x ? 128u : 0u; }
KV_DEVICE constexpr uint32_t colO(int x) { return x ? 384u : 256u; }

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
    int out_type;  // kv_dtype of out: KV_F32 or the pool's type
    float *lse;
    int *err;
};

struct PfBars {
    uint64_t qfull;
    uint64_t kfull[2], kempty[2];
    uint64_t vland[kPfVStages], vfull[kPfVStages], vempty[kPfVStages];  // vland: V copy landed
    uint64_t sfull[2], pfull[2];  // per query tile
    uint64_t done;                // all MMAs complete
    uint32_t tmem_slot;
    int abort;
};

template <bool TW, bool F16>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    // A sequence's query tiles are launched last-first: a later tile of a
    // chunk sees more keys, so the grid's last wave holds light CTAs.  The
    // sequences stay in order, so the CTAs running at one time share one
    // sequence's K/V in L2.
    const int hq = blockIdx.x, qt = gridDim.y - 1 - blockIdx.y, b = blockIdx.z;
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
    const long long kv_end = c + min(q0 + kPfBM, T);  // keys any row of this CTA can see
    const int n = (int)((kv_end + kPfBN - 1) / kPfBN);
    const int nblk = (int)((L + 15) / 16);

    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    char *sQ = smem + kPfQOff;
    char *sK = smem + kPfKOff;
    char *sV = smem + kPfVOff;
    PfBars *bars = reinterpret_cast<PfBars *>(smem + kPfBarOff);

    if (warp == kPfMmaWarp) {
        tc::tmem_alloc(&bars->tmem_slot, 512);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bars->qfull, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->kfull[s], 1);
            mbar_init(&bars->kempty[s], 1);
            mbar_init(&bars->sfull[s], 1);
            mbar_init(&bars->pfull[s], 4);
        }
        for (int s = 0; s < kPfVStages; ++s) {
            mbar_init(&bars->vland[s], 1);
            mbar_init(&bars->vfull[s], 8);  // one arrival per softmax warp
            mbar_init(&bars->vempty[s], 1);
        }
        mbar_init(&bars->done, 1);
        bars->abort = 0;
        mbar_init_fence();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars->tmem_slot;
    volatile int *abort_flag = &bars->abort;

    const int32_t *table_row = p.tables + (size_t)b * p.max_blocks;
    // Tensor row of block (8*jj + lane) of this sequence and head for lanes
    // 0-7; rows -16..-1 lie outside the tensor and read as zeros.
    auto fetch = [&](int jj, bool flag_bad) {
        int y = -16;
        const int ib = jj * 8 + lane;
        if (lane < 8 && jj < n && ib < nblk) {
            const int id = __ldg(table_row + ib);
            if (id >= 0 && id < p.num_blocks)
                y = (id * p.num_kv_heads + h) * 16;
            else if (flag_bad)
                atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
        }
        return y;
    };
    float big = 0.f;  // largest |v| this warp converted (NaN not counted)
    // Softmax warp `part` (0-7) rewrites its eighth of V tile t (landed in
    // stage t % kPfVStages) as fp16, zeroing the rows of keys at or past L,
    // and arrives on the tile's vfull; false if the copy never landed.
    auto convert = [&](int t, int part) {
        const int s = t % kPfVStages;
        bool stop = false;
        if (lane == 0) stop = *abort_flag || !mbar_wait<TW>(&bars->vland[s], (t / kPfVStages) & 1, p.err);
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
        // Lane l of part x rewrites 16-byte chunks 32x + l + 256k: chunk i holds
        // dims 8(i % 8).. of key row (i % 1024) / 8 of half i / 1024 (the
        // swizzle permutes chunks within a 128-byte row, never across rows).
        uint4 *vt = reinterpret_cast<uint4 *>(sV + s * kPfTileBytes);
        const long long valid = L - (long long)t * kPfBN;  // rows below this hold keys < L
        if constexpr (F16) {
            // an fp16 pool: V is already in the MMA's type; only the rows of
            // keys at or past L are zeroed
            if (valid < kPfBN)
                for (int i = 32 * part + lane; i < 2048; i += 256)
                    if (((i & 1023) >> 3) >= valid) vt[i] = make_uint4(0u, 0u, 0u, 0u);
        } else if (valid >= kPfBN) {
#pragma unroll 8
            for (int i = 32 * part + lane; i < 2048; i += 256) {
                uint4 u = vt[i];
                u.x = tc::bf16x2_to_f16x2(u.x, &big);
                u.y = tc::bf16x2_to_f16x2(u.y, &big);
                u.z = tc::bf16x2_to_f16x2(u.z, &big);
                u.w = tc::bf16x2_to_f16x2(u.w, &big);
                vt[i] = u;
            }
        } else {
            for (int i = 32 * part + lane; i < 2048; i += 256) {
                uint4 u = make_uint4(0u, 0u, 0u, 0u);
                if (((i & 1023) >> 3) < valid) {
                    u = vt[i];
                    u.x = tc::bf16x2_to_f16x2(u.x, &big);
                    u.y = tc::bf16x2_to_f16x2(u.y, &big);
                    u.z = tc::bf16x2_to_f16x2(u.z, &big);
                    u.w = tc::bf16x2_to_f16x2(u.w, &big);
                }
                vt[i] = u;
            }
        }
        tc::fence_proxy_async_smem();  // these writes before the tensor core's reads
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->vfull[s]);
        return true;
    };
    // bf16 magnitudes of 65536 and up (the largest finite fp16 is 65504)
    // and infinities were saturated: report them
    auto report_range = [&]() {
        if (__any_sync(0xffffffffu, big > 65504.f) && lane == 0) atomicOr(p.err, KV_DEVERR_VALUE_RANGE);
    };
    if (warp == kPfProducerWarp) {
        // ================================================== K producer
        // Fills the K ring (and loads Q).  Lanes 0-7 hold the block-table
        // entries (as tensor rows) of the next two key tiles, loaded two tiles
        // ahead so their latency never stalls a copy; lane 0 waits on the ring
        // barriers.
        if (lane == 0) {
            tc::prefetch_tensormap(&tm_q);
            tc::prefetch_tensormap(&tm_k);
            mbar_arrive_expect_tx(&bars->qfull, 2 * kPfTileBytes);
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                tc::tma_load_3d(sQ + x * kPfTileBytes, &tm_q, 0, hq, q_begin + q0 + 128 * x, &bars->qfull);
                tc::tma_load_3d(sQ + x * kPfTileBytes + kPfHalfBytes, &tm_q, 64, hq,
                                q_begin + q0 + 128 * x, &bars->qfull);
            }
        }
        int issued = 0;
        int y_cur = fetch(0, true), y_nxt = fetch(1, true);  // entries of tiles t and t+1
        for (int t = 0; t < n; ++t) {
            const int y_later = fetch(t + 2, true);  // in flight during this iteration
            const int s = t & 1;
            bool stop = false;
            if (lane == 0)
                stop = *abort_flag || (t >= 2 && !mbar_wait<TW>(&bars->kempty[s], ((t - 2) >> 1) & 1, p.err));
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
            char *dst = sK + s * kPfTileBytes;
            if (lane == 0) mbar_arrive_expect_tx(&bars->kfull[s], kPfTileBytes);
            __syncwarp();
            // lane b < 8 issues the two boxes of block b (its own table entry):
            // one thread issuing all 16 boxes of a tile is the slower path
            if (lane < 8) {
                tc::tma_load_2d(dst + lane * 2048, &tm_k, 0, y_cur, &bars->kfull[s]);
                tc::tma_load_2d(dst + kPfHalfBytes + lane * 2048, &tm_k, 64, y_cur, &bars->kfull[s]);
            }
            issued = t + 1;
            y_cur = y_nxt;
            y_nxt = y_later;
        }
        if (lane == 0) {
            if (issued < n) *abort_flag = 1;
            // Never leave copies in flight into this CTA's shared memory.
            mbar_wait_drain(&bars->qfull, 0, p.err);
            for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
                mbar_wait_drain(&bars->kfull[j & 1], (j >> 1) & 1, p.err);
        }
    } else if (warp == kPfVProducerWarp) {
        // ================================================== V producer
        // Fills the V ring (kPfVStages deep) as soon as a stage is free: tile
        // t + kPfVStages reuses tile t's stage once PV(t) has completed.  It
        // never waits for a copy to land (the converter does), so the copies
        // are issued at the rate the tensor core frees the stages.
        if (lane == 0) tc::prefetch_tensormap(&tm_v);
        int issued = 0;
        int y_cur = fetch(0, false), y_nxt = fetch(1, false);
        for (int t = 0; t < n; ++t) {
            const int y_later = fetch(t + 2, false);
            const int s = t % kPfVStages;
            bool stop = false;
            if (lane == 0)
                stop = *abort_flag ||
                       (t >= kPfVStages &&
                        !mbar_wait<TW>(&bars->vempty[s], ((t - kPfVStages) / kPfVStages) & 1, p.err));
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
            char *dst = sV + s * kPfTileBytes;
            if (lane == 0) mbar_arrive_expect_tx(&bars->vland[s], kPfTileBytes);
            __syncwarp();
            if (lane < 8) {
                tc::tma_load_2d(dst + lane * 2048, &tm_v, 0, y_cur, &bars->vland[s]);
                tc::tma_load_2d(dst + kPfHalfBytes + lane * 2048, &tm_v, 64, y_cur, &bars->vland[s]);
            }
            issued = t + 1;
            y_cur = y_nxt;
            y_nxt = y_later;
        }
        if (lane == 0) {
            if (issued < n) *abort_flag = 1;
            // Never leave copies in flight into this CTA's shared memory.
            for (int j = (issued > kPfVStages ? issued - kPfVStages : 0); j < issued; ++j)
                mbar_wait_drain(&bars->vland[j % kPfVStages], (j / kPfVStages) & 1, p.err);
        }
    } else if (warp == kPfMmaWarp) {
        // ================================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = F16 ? tc::idesc_f16_f32(128, 128, false, false)
                                              : tc::idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t idesc_pv = tc::idesc_f16_f32(128, 128, false, true);
            // One thread issues every MMA while two softmax warps share its
            // SM sub-partition, so each 128-deep product is one block of PTX
            // whose MMAs cost two 32-bit adds each: the descriptors' low words
            // (start address, leading offset) are formed once and offset in
            // 16-byte units (shared-memory addresses stay below 2^18, so the
            // 14-bit address field never carries); the high word (stride
            // offset 1 KiB, format version, 128-byte swizzle) is the same for
            // Q, K and V.
            const uint32_t d_hi = tc::smem_desc_sw128_hi(1024);
            const uint32_t q_lo = tc::smem_desc_sw128_lo(smem_addr(sQ), 16);
            const uint32_t k_lo = tc::smem_desc_sw128_lo(smem_addr(sK), 16);
            const uint32_t v_lo = tc::smem_desc_sw128_lo(smem_addr(sV), kPfHalfBytes);
            auto issue_s = [&](int x, int j) {  // S_x = Q_x K_j^T
                tc::mma_ss_k128(tmem + colS(x), q_lo + ((x * kPfTileBytes) >> 4),
                                k_lo + (((j & 1) * kPfTileBytes) >> 4), d_hi, idesc_qk, 0);
                tc::mma_commit(&bars->sfull[x]);
            };
            auto issue_pv = [&](int x, int j) {  // O_x += P_x V_j
                // B = V tile, 16 keys x all 128 dims per step (MN-major): the two
                // 64-dim halves are 16 KiB apart, 8-key groups 1 KiB apart.
                tc::mma_ts_k128(tmem + colO(x), tmem + colS(x), v_lo + (((j % kPfVStages) * kPfTileBytes) >> 4),
                                d_hi, idesc_pv, j != 0);
            };
            bool ok = mbar_wait<TW>(&bars->qfull, 0, p.err) && mbar_wait<TW>(&bars->kfull[0], 0, p.err);
            if (ok) {
                tc::fence_after_sync();
                issue_s(0, 0);
                issue_s(1, 0);
                tc::mma_commit(&bars->kempty[0]);
            }
            for (int j = 0; ok && j < n; ++j) {
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    if (!mbar_wait<TW>(&bars->pfull[x], j & 1, p.err) ||
                        (x == 0 && !mbar_wait<TW>(&bars->vfull[j % kPfVStages], (j / kPfVStages) & 1,
                                              p.err))) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    issue_pv(x, j);
                    if (x == 1) tc::mma_commit(&bars->vempty[j % kPfVStages]);
                    if (j + 1 < n) {
                        if (x == 0 && !mbar_wait<TW>(&bars->kfull[(j + 1) & 1], ((j + 1) >> 1) & 1, p.err)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        issue_s(x, j + 1);
                        if (x == 1) tc::mma_commit(&bars->kempty[(j + 1) & 1]);
                    }
                }
            }
            tc::mma_commit(&bars->done);
            if (!ok) *abort_flag = 1;
            // No MMA may still write tensor memory when it is freed.  In the
            // ordinary instantiations the softmax warps' wait for `done` has
            // the full limit and guarantees it already.
            if constexpr (TW) mbar_wait_drain(&bars->done, 0, p.err);
        }
    } else {
        // ================================================== softmax warps
        const int x = warp >> 2;       // query tile
        const int r = tid & 127;       // query row within the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int qrow = q0 + 128 * x + r;
        const bool row_valid = qrow < T;
        // Invalid rows (past the chunk) see every key; they are never stored.
        const long long qpos = row_valid ? c + qrow : L - 1;
        float m_used = -INFINITY, l_sum = 0.f;
        bool ok = convert(0, warp);
        if (!ok) *abort_flag = 1;
        for (int j = 0; ok && j < n; ++j) {
            // Exits are warp-uniform: the warp arrives on pfull as one.
            bool bad = *abort_flag != 0;
            if (!bad) bad = !mbar_wait<TW>(&bars->sfull[x], j & 1, p.err);
            if (__any_sync(0xffffffffu, bad)) { ok = false; break; }
            tc::fence_after_sync();
            const long long key0 = (long long)j * kPfBN;
            // The row's 128 scores are read from tensor memory once and kept
            // in registers for both the maximum and the exponentials.
            uint32_t sv[4][32];
            const uint32_t scol = tmem + lane_base + colS(x);
#pragma unroll
            for (int i = 0; i < 4; ++i) tc::tmem_ld32(scol + 32 * i, sv[i]);
            tc::tmem_wait_ld();
            // Keys past this row's position are masked: column k is kept iff
            // k <= lim.  Only tiles on the diagonal need it; the branch is
            // warp-uniform so interior tiles pay nothing.
            const int lim = (int)max(-1LL, min(127LL, qpos - key0));
            if (__any_sync(0xffffffffu, lim < 127)) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        if (32 * i + k > lim) sv[i][k] = __float_as_uint(-INFINITY);
            }
            // raw row maximum (scale > 0, so max(scale*s) = scale*max(s)),
            // eight independent chains of three-input maxima
            float mx[8];
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const uint32_t *v = &sv[c8 >> 1][16 * (c8 & 1)];
                float m = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
                for (int k = 3; k < 15; k += 2)
                    m = fmax3(m, __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
                mx[c8] = fmaxf(m, __uint_as_float(v[15]));
            }
            const float mrow = fmaxf(fmax3(mx[0], mx[1], mx[2]),
                                     fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7])) *
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
            // p = 2^(scale*s - m) with a packed fma and the hardware exp2; fp16
            // pairs (p <= 2^8) written over the first 64 columns of this S, 32
            // keys at a time.  fp16 keeps 11 significant bits: bf16's 8 would put
            // the weights' rounding error at about 2e-3 of the output scale.
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
            const float2 nm2 = make_float2(-m_used, -m_used);
            float2 acc2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                              make_float2(0.f, 0.f)};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t w[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float2 xx = __ffma2_rn(make_float2(__uint_as_float(sv[i][2 * k]),
                                                             __uint_as_float(sv[i][2 * k + 1])),
                                                 sc2, nm2);
                    const float2 e = make_float2(ex2_approx(xx.x), ex2_approx(xx.y));
                    acc2[k & 3] = __fadd2_rn(acc2[k & 3], e);
                    w[k] = tc::pack_f16x2(e.x, e.y);
                }
                tc::tmem_st16(scol + 16 * i, w);
            }
            l_sum += (acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y) + (acc2[2].x + acc2[2].y) +
                     (acc2[3].x + acc2[3].y);
            if (__any_sync(0xffffffffu, rescale)) {
                // O_x holds PV_x(j-1): its completion precedes S_x(j)'s.  Done after
                // the exponentials, when the scores no longer occupy registers.
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint32_t v[16];
                    const uint32_t oc = tmem + lane_base + colO(x) + 16 * i;
                    tc::tmem_ld16(oc, v);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
                    tc::tmem_st16(oc, v);
                }
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->pfull[x]);  // one arrival per warp
            // the next V tile, while the tensor core computes PV(j) and S(j+1)
            if (j + 1 < n && !convert(j + 1, warp)) {
                ok = false;
                *abort_flag = 1;
                break;
            }
        }
        report_range();
        // ---- epilogue: O / l for this row
        if (ok) ok = mbar_wait<TW>(&bars->done, 0, p.err);
        if (!ok) *abort_flag = 1;
        tc::fence_after_sync();
        const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
        const size_t orow = ((size_t)(q_begin + qrow) * p.num_q_heads + hq) * kPfD;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t v[32];
            tc::tmem_ld32(tmem + lane_base + colO(x) + 32 * i, v);
            tc::tmem_wait_ld();
            if (row_valid && ok) {
                if (p.out_type != KV_F32) {  // the pool's 16-bit type
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.out) + orow + 32 * i);
                    auto pack = [&](int k2) {
                        const float lo = __uint_as_float(v[k2]) * inv, hi = __uint_as_float(v[k2 + 1]) * inv;
                        return F16 ? tc::pack_f16x2(lo, hi) : tc::pack_bf16x2(lo, hi);
                    };
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_uint4(pack(8 * k), pack(8 * k + 2), pack(8 * k + 4), pack(8 * k + 6));
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
            p.lse[(size_t)(q_begin + qrow) * p.num_q_heads + hq] =
                l_sum > 0.f ? (m_used + log2f(l_sum)) * 0.6931471805599453f : -INFINITY;
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kPfMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

cudaError_t set_wait_limit_prefill(unsigned long long ns) { return set_wait_limit_here(ns); }

}  // namespace pkv

using namespace pkv;

extern "C" kv_status paged_prefill_attention(kv_pool_t p, const void *q, const int32_t *cu_q,
                                             int total_q, int max_q_len, const int32_t *block_tables,
                                             int max_blocks, const int32_t *seq_lens, int batch,
                                             int num_q_heads, float scale, void *out,
                                             kv_dtype out_dtype, float *lse_out, void *stream) {
    if (!p || batch < 0 || total_q < 0 || max_q_len < 0 || max_blocks < 0 || num_q_heads <= 0)
        return KV_ERR_ARG;
    if (kv_status st = require_device(p->device)) return st;
    if (p->dtype == KV_F32 || p->head_dim != kPfD) return KV_ERR_UNSUPPORTED;
    if (num_q_heads % p->num_kv_heads) return KV_ERR_ARG;
    if (out_dtype != KV_F32 && out_dtype != p->dtype) return KV_ERR_UNSUPPORTED;
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
    pp.out_type = out_dtype;
    pp.lse = lse_out;
    pp.err = p->err;
    const bool f16 = p->dtype == KV_F16;
    auto fn = test_waits_enabled() ? (f16 ? prefill_kernel<true, true> : prefill_kernel<true, false>)
                                   : (f16 ? prefill_kernel<false, true> : prefill_kernel<false, false>);
    if (kv_status st0 = cuda_status(cudaFuncSetAttribute(
            fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmemBytes)))
        return st0;
    const int q_tiles = (max_q_len + kPfBM - 1) / kPfBM;
    if (q_tiles > 65535) return KV_ERR_UNSUPPORTED;
    const dim3 grid(num_q_heads, q_tiles, batch);
    fn<<<grid, kPfThreads, kPfSmemBytes, as_stream(stream)>>>(tm_q, p->tmap_k,
                                                                         p->tmap_v, pp);
    return cuda_status(cudaGetLastError());
}
