// Cascade decode over shared prefixes on the tcgen05 tensor cores.
//
// "PagedAttention Nedir?", section "Prefix Sharing Nasil Calisir?", and
// "Makale Bulteni -- PagedAttention ve vLLM", section "Ticari Etki": requests
// that start with the same tokens keep that part of the KV cache once, as the
// same physical blocks.  A plain paged decode still reads those blocks once
// per sequence.  Here the decode of a group of sequences that share blocks is
// cut in two, with the same result (exact maths, up to rounding):
//   1. prefix: one CTA per (prefix split, kv head, group) reads the group's
//      shared blocks once and attends them with the query rows of every
//      sequence of the group and every query head of the kv head - a real
//      matrix product (rows = sequences x heads, up to 128) on the tensor core;
//   2. suffix: the ordinary decode kernels attend each sequence's own blocks
//      after its shared part (start_tokens);
// and the split-KV merge combines the partial results of both by their
// log-sum-exp: o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M).
//
// Sequence b of a group uses the first shared_tokens[b] tokens of the
// group's prefix (rounded down to whole blocks, clamped to seq_lens[b]).  The
// prefix blocks are read from the block table of the member with the longest
// shared part; every member's table holds the same ids for its shared blocks.
//
// Prefix kernel, per key tile of 128 keys (8 blocks of 16):
//   S(j) = Q K_j^T   (tcgen05, M = 128 query rows, N = 128 keys, K = 128 dims)
//   softmax warps: S -> P, per-row key limit; P is written over S as two
//                    parts of the pool's 16-bit type t, P_hi = t(P) in
//                    columns 0-63 and P_lo = t(P - P_hi) in columns 64-127,
//                    so the weights keep about 16 significant bits with bf16
//                    (a bf16 P alone, 8 bits, is off by up to 2^-9 of the
//                    largest V on short rows) and about 22 with fp16
//   O += P_hi V_j + P_lo V_j   (tcgen05, P from tensor memory)
// Tensor memory: S double-buffered at columns [0,128) and [128,256), O at
// [256,384).  MMA issue order: S(0), S(1), PV(0), S(2), PV(1), S(3), ...  so
// the tensor core computes S(j+1) while the softmax warps work on S(j).
// Because S(j+1) is issued before PV(j), a softmax warp that must rescale O
// at tile j+1 first waits for PV(j) (barrier odone); the rescale happens only
// when a row's running maximum rises by more than 2^8.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace pkv {
namespace {

constexpr int kCsRows = 128;                  // query rows per CTA (tensor-core M)
constexpr int kCsBN = 128;                    // keys per tile
constexpr int kCsD = 128;                     // head dim (only size supported)
constexpr int kCsThreads = 224;               // 4 softmax warps, MMA issuer, K and V producers
constexpr int kCsMmaWarp = 4, kCsKWarp = 5, kCsVWarp = 6;
constexpr int kCsHalfBytes = 128 * 128;       // 128 rows x 64 bf16 (one half of D)
constexpr int kCsTileBytes = 2 * kCsHalfBytes;
constexpr int kCsQOff = 0;
constexpr int kCsKOff = kCsTileBytes;                   // 2 stages
constexpr int kCsVOff = kCsKOff + 2 * kCsTileBytes;     // 2 stages
constexpr int kCsBarOff = kCsVOff + 2 * kCsTileBytes;   // 160 KiB
constexpr int kCsSmemBytes = kCsBarOff + 2048 + 1024;   // barriers and exchange, alignment slack
constexpr float kCsRescaleThreshold = 8.0f;             // log2 units
constexpr uint32_t kColO = 256;
constexpr int kCsBlockTokens = 16;                       // tokens per KV block

KV_DEVICE float cs_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

KV_DEVICE float cs_max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

struct CascadeParams {
    const uint16_t *q;  // [batch][num_q_heads][128], the pool's 16-bit type
    const int32_t *tables;
    int max_blocks;
    int num_blocks;
    const int32_t *seq_lens;
    int batch;
    const int32_t *group_seqs;  // [num_groups][group_size], -1 = empty
    int group_size;
    const int32_t *shared_tokens;
    int num_q_heads;
    int num_kv_heads;
    int g;
    float scale_log2;
    int tiles_per_split;
    float *ws_o;  // [batch][num_q_heads][max_splits][128]
    float *ws_lse;
    int max_splits;
    int *err;
};

struct CsBars {
    uint64_t qfull;
    uint64_t kfull[2], vfull[2], kempty[2], vempty[2];
    uint64_t sfull[2], pfull[2];  // per S buffer
    uint64_t odone;               // one phase per PV
    uint64_t done;                // all MMAs complete
    uint32_t tmem_slot;
    int abort;
    int n_pre;   // prefix tokens of the group (longest member)
    int leader;  // sequence whose table lists the prefix blocks
    // duplicated rows (groups of at most 64 rows): the two threads of a row
    // exchange half-row maxima (by tile parity) and, at the end, row sums
    float xmax[2][64][2];
    float xsum[64][2];
};
static_assert(sizeof(CsBars) <= 2048, "barrier block too large");

// Tokens of sequence b attended by the prefix kernel: shared_tokens[b]
// clamped to [0, min(L, max_blocks * 16)], rounded down to whole blocks.
// (The decode kernels clamp to L and round down the same way.)
KV_DEVICE int prefix_limit(const CascadeParams &p, int b) {
    if (b < 0 || b >= p.batch) return 0;
    long long L = p.seq_lens[b];
    L = L < 0 ? 0 : L;
    const long long cap = (long long)p.max_blocks * 16;
    long long st = p.shared_tokens[b];
    st = st < 0 ? 0 : (st > L ? L : st);
    st = st > cap ? cap : st;
    return (int)(st / 16) * 16;
}

// DUP: the group has at most 64 query rows.  Q rows 64..127 repeat rows
// 0..63, so the tensor core produces every score row twice, in TMEM lanes r
// and r + 64, at no extra cost; thread r then takes keys 0..63 of the row and
// thread r + 64 keys 64..127 (the two warps sit on different SM sub-partitions,
// which a TMEM lane quadrant would not allow otherwise).  Each writes its P
// into its own key half of the row and zeros into the other half, so the one
// PV product yields two partial O rows, added in the epilogue.
// Two weights (x, y) as the packed 16-bit pair hi = t(x), t(y) of the pool's
// type t and the packed remainders lo = t(x - hi.x), t(y - hi.y); hi + lo
// carries about twice t's significant bits.  Widening t to fp32 is exact.
template <bool F16>
KV_DEVICE void split_weights(float x, float y, uint32_t &hi, uint32_t &lo) {
    if constexpr (F16) {
        hi = tc::pack_f16x2(x, y);
        float hx, hy;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\t"
            "cvt.f32.f16 %1, h;\n\t}"
            : "=f"(hx), "=f"(hy)
            : "r"(hi));
        lo = tc::pack_f16x2(x - hx, y - hy);
    } else {
        hi = tc::pack_bf16x2(x, y);
        // the high halves of the packed word, widened
        const float hx = __uint_as_float(hi << 16), hy = __uint_as_float(hi & 0xffff0000u);
        lo = tc::pack_bf16x2(x - hx, y - hy);
    }
}

template <bool DUP, bool TW, bool F16>
__global__ void __launch_bounds__(kCsThreads, 1)
    cascade_prefix_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const CascadeParams p) {
    const int ps = blockIdx.x, h = blockIdx.y, grp = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the suffix decode, launched after this kernel, may start on the SM room
    // this grid leaves (it waits for this grid only where it merges)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    char *sQ = smem + kCsQOff;
    char *sK = smem + kCsKOff;
    char *sV = smem + kCsVOff;
    CsBars *bars = reinterpret_cast<CsBars *>(smem + kCsBarOff);

    // ---- the group's prefix length and the member whose table lists it
    if (warp == 0) {
        int best = 0, best_s = -1;
        for (int s = lane; s < p.group_size; s += 32) {
            const int lim = prefix_limit(p, p.group_seqs[(size_t)grp * p.group_size + s]);
            if (lim > best) {
                best = lim;
                best_s = s;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const int ob = __shfl_xor_sync(0xffffffffu, best, off);
            const int os = __shfl_xor_sync(0xffffffffu, best_s, off);
            if (ob > best || (ob == best && os >= 0 && (best_s < 0 || os < best_s))) {
                best = ob;
                best_s = os;
            }
        }
        if (lane == 0) {
            bars->n_pre = best;
            bars->leader = best_s >= 0 ? p.group_seqs[(size_t)grp * p.group_size + best_s] : -1;
        }
    }
    __syncthreads();
    const int n_pre = bars->n_pre;
    const int leader = bars->leader;
    const int tiles_all = (n_pre + kCsBN - 1) / kCsBN;
    const int t0 = ps * p.tiles_per_split;
    const int n = max(0, min(p.tiles_per_split, tiles_all - t0));  // key tiles of this CTA
    if (ps == gridDim.x - 1 && tid == 0 && tiles_all > t0 + p.tiles_per_split)
        atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);  // prefix longer than the planned splits

    // ---- this thread's query row (softmax warps): member slot s, head i
    const int r = tid;               // TMEM lane, valid for tid < 128
    const int qr = DUP ? r & 63 : r;  // query row of the group
    const int half = DUP ? r >> 6 : 0;  // DUP: which 64 keys of each tile
    int member = -1, lim = 0;
    if (tid < kCsRows && qr < p.group_size * p.g) {
        member = p.group_seqs[(size_t)grp * p.group_size + qr / p.g];
        if (member >= p.batch) member = -1;
        lim = prefix_limit(p, member);
    }
    const size_t orow = member >= 0 ? (size_t)member * p.num_q_heads + h * p.g + qr % p.g : 0;

    if (n == 0) {  // no keys of the prefix here: empty partial results
        if (tid < kCsRows && half == 0 && member >= 0 && lim > 0) {
            float4 *dst = reinterpret_cast<float4 *>(p.ws_o + (orow * p.max_splits + ps) * kCsD);
            for (int k = 0; k < kCsD / 4; ++k) dst[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            p.ws_lse[orow * p.max_splits + ps] = -INFINITY;
        }
        return;
    }

    if (warp == kCsMmaWarp) {
        tc::tmem_alloc(&bars->tmem_slot, 512);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bars->qfull, kCsRows);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->kfull[s], 1);
            mbar_init(&bars->vfull[s], 1);
            mbar_init(&bars->kempty[s], 1);
            mbar_init(&bars->vempty[s], 1);
            mbar_init(&bars->sfull[s], 1);
            mbar_init(&bars->pfull[s], 4);
        }
        mbar_init(&bars->odone, 1);
        mbar_init(&bars->done, 1);
        bars->abort = 0;
        mbar_init_fence();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars->tmem_slot;
    volatile int *abort_flag = &bars->abort;

    if (warp == kCsKWarp || warp == kCsVWarp) {
        // ================================================== TMA producers
        // K ring and V ring, one warp each; lanes 0-7 hold the tensor rows of
        // the next two key tiles' blocks (leader's table), loaded two tiles ahead.
        const bool is_v = warp == kCsVWarp;
        if (lane == 0) tc::prefetch_tensormap(is_v ? &tm_v : &tm_k);
        const CUtensorMap *map = is_v ? &tm_v : &tm_k;
        char *ring = is_v ? sV : sK;
        uint64_t *full = is_v ? bars->vfull : bars->kfull;
        uint64_t *empty = is_v ? bars->vempty : bars->kempty;
        const int32_t *row = p.tables + (size_t)(leader < 0 ? 0 : leader) * p.max_blocks;
        const int nblk_pre = n_pre / 16;
        auto fetch = [&](int jj) {
            int y = -16;  // rows -16..-1 lie outside the tensor and read as zeros
            const int ib = (t0 + jj) * 8 + lane;
            if (lane < 8 && jj < n && ib < nblk_pre && leader >= 0) {
                const int id = __ldg(row + ib);
                if (id >= 0 && id < p.num_blocks)
                    y = (id * p.num_kv_heads + h) * 16;
                else if (!is_v)
                    atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
            }
            return y;
        };
        int issued = 0;
        int y_cur = fetch(0), y_nxt = fetch(1);
        for (int t = 0; t < n; ++t) {
            const int y_later = fetch(t + 2);
            const int s = t & 1;
            bool stop = false;
            if (lane == 0)
                stop = *abort_flag || (t >= 2 && !mbar_wait<TW>(&empty[s], ((t - 2) >> 1) & 1, p.err));
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
            char *dst = ring + s * kCsTileBytes;
            if (lane == 0) mbar_arrive_expect_tx(&full[s], kCsTileBytes);
            __syncwarp();
            // lane b < 8 issues the two boxes of block b (its own table entry):
            // one thread issuing all 16 boxes of a tile is the slower path
            if (lane < 8) {
                tc::tma_load_2d(dst + lane * 2048, map, 0, y_cur, &full[s]);
                tc::tma_load_2d(dst + kCsHalfBytes + lane * 2048, map, 64, y_cur, &full[s]);
            }
            issued = t + 1;
            y_cur = y_nxt;
            y_nxt = y_later;
        }
        if (lane == 0) {
            if (issued < n) *abort_flag = 1;
            // Never leave copies in flight into this CTA's shared memory.
            for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
                mbar_wait_drain(&full[j & 1], (j >> 1) & 1, p.err);
        }
    } else if (warp == kCsMmaWarp) {
        // ================================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = F16 ? tc::idesc_f16_f32(128, 128, false, false)
                                              : tc::idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t idesc_pv = F16 ? tc::idesc_f16_f32(128, 128, false, true)
                                              : tc::idesc_bf16_f32(128, 128, false, true);
            // Each 128-deep product is one block of PTX (two 32-bit adds per
            // MMA): descriptor low words formed once, offset in 16-byte units;
            // one high word (stride 1 KiB, 128-byte swizzle) for Q, K and V.
            const uint32_t d_hi = tc::smem_desc_sw128_hi(1024);
            const uint32_t q_lo = tc::smem_desc_sw128_lo(smem_addr(sQ), 16);
            const uint32_t k_lo = tc::smem_desc_sw128_lo(smem_addr(sK), 16);
            const uint32_t v_lo = tc::smem_desc_sw128_lo(smem_addr(sV), kCsHalfBytes);
            auto issue_s = [&](int j) {  // S(j) = Q K_j^T into S buffer j & 1
                tc::mma_ss_k128(tmem + (j & 1) * 128, q_lo, k_lo + (((j & 1) * kCsTileBytes) >> 4), d_hi,
                                idesc_qk, 0);
                tc::mma_commit(&bars->sfull[j & 1]);
                tc::mma_commit(&bars->kempty[j & 1]);
            };
            auto issue_pv = [&](int j) {  // O += P(j) V_j, P = P_hi + P_lo
                // B = V tile, 16 keys x 128 dims per step (MN-major): the two
                // 64-dim halves are 16 KiB apart, 8-key groups 1 KiB apart.
                const uint32_t vb = v_lo + (((j & 1) * kCsTileBytes) >> 4);
                const uint32_t pcol = tmem + (j & 1) * 128;
                tc::mma_ts_k128(tmem + kColO, pcol, vb, d_hi, idesc_pv, j != 0);  // P_hi
                tc::mma_ts_k128(tmem + kColO, pcol + 64, vb, d_hi, idesc_pv, 1);  // P_lo
                tc::mma_commit(&bars->vempty[j & 1]);
                tc::mma_commit(&bars->odone);
            };
            bool ok = mbar_wait<TW>(&bars->qfull, 0, p.err) && mbar_wait<TW>(&bars->kfull[0], 0, p.err);
            if (ok) {
                tc::fence_after_sync();
                issue_s(0);
                if (n > 1) {
                    ok = mbar_wait<TW>(&bars->kfull[1], 0, p.err);
                    tc::fence_after_sync();
                    if (ok) issue_s(1);
                }
            }
            for (int j = 0; ok && j < n; ++j) {
                const int s = j & 1;
                if (!mbar_wait<TW>(&bars->pfull[s], (j >> 1) & 1, p.err) ||
                    !mbar_wait<TW>(&bars->vfull[s], (j >> 1) & 1, p.err)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                issue_pv(j);
                if (j + 2 < n) {
                    if (!mbar_wait<TW>(&bars->kfull[s], ((j + 2) >> 1) & 1, p.err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    issue_s(j + 2);
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
        // Thread = query row = TMEM lane.  Q rows are gathered here (the
        // rows of one group are not contiguous in q) and stored in the
        // 128-byte-swizzled K-major layout the MMA descriptor expects.
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(p.q + orow * kCsD);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint4 v = member >= 0 ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                const int hh = c >> 3, cc = c & 7;
                *reinterpret_cast<uint4 *>(sQ + hh * kCsHalfBytes + r * 128 + ((cc ^ (r & 7)) << 4)) = v;
            }
            tc::fence_proxy_async_smem();
            mbar_arrive(&bars->qfull);
        }
        if constexpr (DUP) {
            // pair barrier of the two warps holding the same rows (warps w, w + 2)
            const int pair_bar = 1 + (warp & 1);
            float m_used = -INFINITY, l_sum = 0.f;
            bool ok = true, bad_next = false;
            const uint32_t zero16[16] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
            for (int j = 0; j < n; ++j) {
                const int sb = j & 1;
                bool bad = bad_next || *abort_flag != 0;
                if (!bad) bad = !mbar_wait<TW>(&bars->sfull[sb], (j >> 1) & 1, p.err);
                tc::fence_after_sync();
                const uint32_t scol = tmem + lane_base + sb * 128;
                uint32_t sv[2][32];
                float mhalf = -INFINITY;
                const int klim = max(0, min(64, lim - (t0 + j) * kCsBN - 64 * half));  // keys kept in my half
                if (!bad) {
                    tc::tmem_ld32(scol + 64 * half, sv[0]);
                    tc::tmem_ld32(scol + 64 * half + 32, sv[1]);
                    tc::tmem_wait_ld();
                    if (__any_sync(0xffffffffu, klim < 64)) {
#pragma unroll
                        for (int i = 0; i < 2; ++i)
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                if (32 * i + k >= klim) sv[i][k] = __float_as_uint(-INFINITY);
                    }
                    float mx[4];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const uint32_t *v = &sv[c4 >> 1][16 * (c4 & 1)];
                        float m = cs_max3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
                        for (int k = 3; k < 15; k += 2)
                            m = cs_max3(m, __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
                        mx[c4] = fmaxf(m, __uint_as_float(v[15]));
                    }
                    mhalf = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                }
                bars->xmax[j & 1][qr][half] = mhalf;
                // both halves decide together whether to go on (the barrier has no timeout)
                if (named_bar_or(pair_bar, 64, bad)) {
                    ok = false;
                    *abort_flag = 1;
                    break;
                }
                const float mrow = fmaxf(bars->xmax[j & 1][qr][0], bars->xmax[j & 1][qr][1]) *
                                   p.scale_log2;  // scale > 0
                float alpha = 1.f;
                bool rescale = false;
                if (m_used == -INFINITY) {
                    m_used = mrow;
                } else if (mrow > m_used + kCsRescaleThreshold) {
                    alpha = cs_ex2(m_used - mrow);
                    m_used = mrow;
                    l_sum *= alpha;
                    rescale = true;
                }
                const float mref = m_used == -INFINITY ? 0.f : m_used;
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                const float2 nm2 = make_float2(-mref, -mref);
                float2 acc2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                  make_float2(0.f, 0.f)};
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    uint32_t whi[16], wlo[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float2 xx = __ffma2_rn(make_float2(__uint_as_float(sv[i][2 * k]),
                                                                 __uint_as_float(sv[i][2 * k + 1])),
                                                     sc2, nm2);
                        const float2 e = make_float2(cs_ex2(xx.x), cs_ex2(xx.y));
                        acc2[k & 3] = __fadd2_rn(acc2[k & 3], e);
                        split_weights<F16>(e.x, e.y, whi[k], wlo[k]);
                    }
                    // my keys: P columns 32*half + 16i (hi) and 64 + 32*half + 16i (lo)
                    tc::tmem_st16(scol + 32 * half + 16 * i, whi);
                    tc::tmem_st16(scol + 64 + 32 * half + 16 * i, wlo);
                    // the other half's keys are not in this lane's row
                    tc::tmem_st16(scol + 32 * (1 - half) + 16 * i, zero16);
                    tc::tmem_st16(scol + 64 + 32 * (1 - half) + 16 * i, zero16);
                }
                l_sum += (acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y) + (acc2[2].x + acc2[2].y) +
                         (acc2[3].x + acc2[3].y);
                if (__any_sync(0xffffffffu, rescale)) {
                    // this lane's partial O holds PV(j-1) once that completes
                    if (__any_sync(0xffffffffu, !mbar_wait<TW>(&bars->odone, (j - 1) & 1, p.err))) {
                        bad_next = true;  // leave together at the next exchange
                    } else {
                        tc::fence_after_sync();
#pragma unroll 1
                        for (int i = 0; i < 8; ++i) {
                            uint32_t v[16];
                            const uint32_t oc = tmem + lane_base + kColO + 16 * i;
                            tc::tmem_ld16(oc, v);
                            tc::tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
                            tc::tmem_st16(oc, v);
                        }
                    }
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->pfull[sb]);  // one arrival per warp
            }
            // ---- epilogue: the two partial O rows of a query row are added
            // (lane r + 64's through shared memory: the K ring is idle once
            // every MMA has completed)
            if (ok) ok = mbar_wait<TW>(&bars->done, 0, p.err);
            tc::fence_after_sync();
            float *xo = reinterpret_cast<float *>(sK);  // [64][128]
            bars->xsum[qr][half] = l_sum;
            if (half == 1) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint32_t v[16];
                    tc::tmem_ld16(tmem + lane_base + kColO + 16 * i, v);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) xo[qr * kCsD + 16 * i + k] = __uint_as_float(v[k]);
                }
            }
            const bool okay = !named_bar_or(pair_bar, 64, !ok);
            if (!okay) *abort_flag = 1;
            if (half == 0) {
                const float lrow = bars->xsum[qr][0] + bars->xsum[qr][1];
                const bool write = okay && member >= 0 && lim > 0;
                const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
                float4 *dst = reinterpret_cast<float4 *>(p.ws_o + (orow * p.max_splits + ps) * kCsD);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint32_t v[16];
                    tc::tmem_ld16(tmem + lane_base + kColO + 16 * i, v);
                    tc::tmem_wait_ld();
                    if (write) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float *o2 = xo + qr * kCsD + 16 * i + 4 * k;
                            dst[4 * i + k] = make_float4((__uint_as_float(v[4 * k]) + o2[0]) * inv,
                                                         (__uint_as_float(v[4 * k + 1]) + o2[1]) * inv,
                                                         (__uint_as_float(v[4 * k + 2]) + o2[2]) * inv,
                                                         (__uint_as_float(v[4 * k + 3]) + o2[3]) * inv);
                        }
                    }
                }
                if (write) p.ws_lse[orow * p.max_splits + ps] = lrow > 0.f ? m_used + log2f(lrow) : -INFINITY;
            }
        } else {
        const bool warp_idle = __all_sync(0xffffffffu, lim == 0);  // padding rows only
        float m_used = -INFINITY, l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int sb = j & 1;
            bool bad = *abort_flag != 0;
            if (!bad) bad = !mbar_wait<TW>(&bars->sfull[sb], (j >> 1) & 1, p.err);
            if (__any_sync(0xffffffffu, bad)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            if (!warp_idle) {
                const uint32_t scol = tmem + lane_base + sb * 128;
                uint32_t sv[4][32];
#pragma unroll
                for (int i = 0; i < 4; ++i) tc::tmem_ld32(scol + 32 * i, sv[i]);
                tc::tmem_wait_ld();
                // keys k of this tile are kept iff key0 + k < lim
                const int klim = max(0, min(kCsBN, lim - (t0 + j) * kCsBN));
                if (__any_sync(0xffffffffu, klim < kCsBN)) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            if (32 * i + k >= klim) sv[i][k] = __float_as_uint(-INFINITY);
                }
                float mx[8];
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint32_t *v = &sv[c8 >> 1][16 * (c8 & 1)];
                    float m = cs_max3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
                    for (int k = 3; k < 15; k += 2)
                        m = cs_max3(m, __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
                    mx[c8] = fmaxf(m, __uint_as_float(v[15]));
                }
                const float mrow = fmaxf(cs_max3(mx[0], mx[1], mx[2]),
                                         cs_max3(cs_max3(mx[3], mx[4], mx[5]), mx[6], mx[7])) *
                                   p.scale_log2;  // scale > 0
                float alpha = 1.f;
                bool rescale = false;
                if (m_used == -INFINITY) {
                    m_used = mrow;  // first kept keys of the row (O is still zero)
                } else if (mrow > m_used + kCsRescaleThreshold) {
                    alpha = cs_ex2(m_used - mrow);
                    m_used = mrow;
                    l_sum *= alpha;
                    rescale = true;
                }
                const float mref = m_used == -INFINITY ? 0.f : m_used;  // no kept key yet: all weights 0
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                const float2 nm2 = make_float2(-mref, -mref);
                float2 acc2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                  make_float2(0.f, 0.f)};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t whi[16], wlo[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float2 xx = __ffma2_rn(make_float2(__uint_as_float(sv[i][2 * k]),
                                                                 __uint_as_float(sv[i][2 * k + 1])),
                                                     sc2, nm2);
                        const float2 e = make_float2(cs_ex2(xx.x), cs_ex2(xx.y));
                        acc2[k & 3] = __fadd2_rn(acc2[k & 3], e);
                        split_weights<F16>(e.x, e.y, whi[k], wlo[k]);
                    }
                    tc::tmem_st16(scol + 16 * i, whi);
                    tc::tmem_st16(scol + 64 + 16 * i, wlo);
                }
                l_sum += (acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y) + (acc2[2].x + acc2[2].y) +
                         (acc2[3].x + acc2[3].y);
                if (__any_sync(0xffffffffu, rescale)) {
                    // O holds PV(j-1) once that completes (S(j) was issued before it)
                    if (__any_sync(0xffffffffu, !mbar_wait<TW>(&bars->odone, (j - 1) & 1, p.err))) {
                        ok = false;
                        *abort_flag = 1;
                        break;
                    }
                    tc::fence_after_sync();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint32_t v[16];
                        const uint32_t oc = tmem + lane_base + kColO + 16 * i;
                        tc::tmem_ld16(oc, v);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
                        tc::tmem_st16(oc, v);
                    }
                }
                tc::tmem_wait_st();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->pfull[sb]);  // one arrival per warp
        }
        // ---- epilogue: this row's partial result (normalised o, lse in log2 units)
        if (ok) ok = mbar_wait<TW>(&bars->done, 0, p.err);
        if (!ok) *abort_flag = 1;
        tc::fence_after_sync();
        const bool write = ok && member >= 0 && lim > 0;
        const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
        float4 *dst = reinterpret_cast<float4 *>(p.ws_o + (orow * p.max_splits + ps) * kCsD);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t v[16];
            tc::tmem_ld16(tmem + lane_base + kColO + 16 * i, v);
            tc::tmem_wait_ld();
            if (write) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    dst[4 * i + k] = make_float4(__uint_as_float(v[4 * k]) * inv, __uint_as_float(v[4 * k + 1]) * inv,
                                                 __uint_as_float(v[4 * k + 2]) * inv, __uint_as_float(v[4 * k + 3]) * inv);
            }
        }
        if (write) p.ws_lse[orow * p.max_splits + ps] = l_sum > 0.f ? m_used + log2f(l_sum) : -INFINITY;
    }
        }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kCsMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

// Prefix splits: enough CTAs to cover the SMs once, at most one per key tile.
static int cascade_splits(int num_groups, int num_kv_heads, int max_prefix_blocks, int requested) {
    const int tiles = (max_prefix_blocks + 7) / 8;
    if (tiles <= 0) return 1;
    int ps = requested > 0 ? requested : sm_count() / (num_groups * num_kv_heads > 0 ? num_groups * num_kv_heads : 1);
    if (ps < 1) ps = 1;
    if (ps > tiles) ps = tiles;
    return ps;
}

cudaError_t set_wait_limit_cascade(unsigned long long ns) { return set_wait_limit_here(ns); }

}  // namespace pkv

using namespace pkv;

extern "C" {

kv_status kv_cascade_plan(int num_groups, int num_kv_heads, int max_prefix_blocks, int requested,
                          int *prefix_splits) {
    if (!prefix_splits || num_groups < 0 || num_kv_heads <= 0 || max_prefix_blocks < 0 || requested < 0)
        return KV_ERR_ARG;
    *prefix_splits = cascade_splits(num_groups, num_kv_heads, max_prefix_blocks, requested);
    return KV_OK;
}

// The suffix grid order of a cascade decode.  A sequence whose own part is at
// most one block attends its partial last block only: its CTA's time is
// start-up and the merge with the prefix's result, latency rather than
// bandwidth.  Run at the end of a longest-first grid, 880 such CTAs (the
// shared-prefix step: 110 of 256 sequences x 8 kv heads) formed a tail in
// which HBM idled; at the start they held the SMs the longest sequences need
// first.  Placed as one run after the first 40% of the others, they overlap
// the long CTAs' streaming: the step's decode went from 0.0844-0.0848 ms to
// 0.0771-0.0772 ms on GB300 (after the first 20% / 25% / 33% / 36% / 38% /
// 42% / 44% / 50%: 0.0809, 0.0804, 0.0785, 0.0776, 0.0777-0.0779, 0.0773,
// 0.0782, 0.0798 ms).
kv_status kv_cascade_order(const int32_t *host_suffix_lens, int batch, int32_t *order_out) {
    if (batch < 0 || (batch > 0 && (!host_suffix_lens || !order_out))) return KV_ERR_ARG;
    std::vector<int32_t> idx(batch), longs, shorts;
    for (int b = 0; b < batch; ++b) idx[b] = b;
    std::stable_sort(idx.begin(), idx.end(),
                     [&](int32_t x, int32_t y) { return host_suffix_lens[x] > host_suffix_lens[y]; });
    for (int32_t b : idx) (host_suffix_lens[b] > kCsBlockTokens ? longs : shorts).push_back(b);
    const size_t head = (2 * longs.size() + 2) / 5;  // the first 40%, rounded
    size_t o = 0;
    for (size_t i = 0; i < head; ++i) order_out[o++] = longs[i];
    for (int32_t b : shorts) order_out[o++] = b;
    for (size_t i = head; i < longs.size(); ++i) order_out[o++] = longs[i];
    return KV_OK;
}

kv_status kv_cascade_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                    int max_blocks, int num_splits, int prefix_splits,
                                    size_t *bytes) {
    if (!bytes || batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks < 0 ||
        num_splits < 0 || prefix_splits < 1)
        return KV_ERR_ARG;
    int pb = 0, ms = 0;
    split_plan(batch, num_kv_heads, max_blocks, num_splits, &pb, &ms);
    *bytes = decode_workspace_bytes(batch, num_q_heads, head_dim, prefix_splits + ms);
    return KV_OK;
}

kv_status paged_decode_attention_cascade(
    kv_pool_t p, const void *q, const int32_t *block_tables, int max_blocks, const int32_t *seq_lens,
    int batch, int num_q_heads, float scale, const int32_t *group_seqs, int num_groups,
    int group_size, const int32_t *shared_tokens, int max_prefix_blocks, int prefix_splits,
    void *out, kv_dtype out_dtype, float *lse_out, int num_splits, const int32_t *seq_order,
    void *workspace, size_t workspace_bytes, void *stream) {
    if (!p || batch < 0 || max_blocks < 0 || num_q_heads <= 0 || num_groups < 0 || group_size < 0 ||
        max_prefix_blocks < 0 || prefix_splits < 0 || num_splits < 0)
        return KV_ERR_ARG;
    if (kv_status st = require_device(p->device)) return st;
    if ((p->dtype != KV_BF16 && p->dtype != KV_F16) || p->head_dim != kCsD) return KV_ERR_UNSUPPORTED;
    if (num_q_heads % p->num_kv_heads) return KV_ERR_ARG;
    const int g = num_q_heads / p->num_kv_heads;
    if ((long long)group_size * g > kCsRows) return KV_ERR_UNSUPPORTED;
    if (max_prefix_blocks > max_blocks) return KV_ERR_ARG;
    if (batch == 0) return KV_OK;
    if (!q || !block_tables || !seq_lens || !out || !shared_tokens ||
        (num_groups > 0 && group_size > 0 && !group_seqs))
        return KV_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(q) & 15) return KV_ERR_ARG;
    if (num_groups > 65535 || p->num_kv_heads > 65535) return KV_ERR_UNSUPPORTED;
    const int ps = cascade_splits(num_groups, p->num_kv_heads, max_prefix_blocks, prefix_splits);
    const int tiles = (max_prefix_blocks + 7) / 8;
    if (pool_tensor_maps(p) != KV_OK) return KV_ERR_CUDA;
    cudaStream_t s = as_stream(stream);

    // suffix: the ordinary decode, after each sequence's shared part
    DecodeArgs a{};
    a.q = q;
    a.k_pool = p->k;
    a.v_pool = p->v;
    a.block_tables = block_tables;
    a.max_blocks = max_blocks;
    a.num_blocks = p->num_blocks;
    a.seq_lens = seq_lens;
    a.batch = batch;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = p->num_kv_heads;
    a.head_dim = p->head_dim;
    a.dtype = p->dtype;
    a.scale = scale;
    a.out = out;
    a.out_dtype = out_dtype;
    a.lse = lse_out;
    a.num_splits = num_splits;
    a.start_tokens = shared_tokens;
    a.part_base = ps;
    a.seq_order = seq_order;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.err = p->err;
    a.counters = p->counters;
    a.counter_slots = kv_pool::kCounterSlots;
    a.stream = s;
    a.pool_map_k = &p->tmap_k;
    a.pool_map_v = &p->tmap_v;
    int pb = 0, ms = 0;
    split_plan(batch, p->num_kv_heads, max_blocks, num_splits, &pb, &ms);
    const size_t need = decode_workspace_bytes(batch, num_q_heads, kCsD, ps + ms);
    if (!workspace || workspace_bytes < need) return KV_ERR_ARG;
    if (out_dtype != KV_F32 && out_dtype != p->dtype) return KV_ERR_UNSUPPORTED;

    // prefix first: its partial results must be in place before the suffix's
    // merge reads them.  The suffix decode may overlap it (a programmatic
    // dependent launch): its CTAs attend their own blocks meanwhile, and a
    // merging CTA waits for the prefix grid before it reads the prefix slots.
    // That needs every merge inside the decode kernel (fused merge).
    const bool fused_merges = ps + ms <= kFuseMaxSplits &&
                              (long long)batch * p->num_kv_heads <= kv_pool::kCounterSlots;
    if (num_groups > 0 && group_size > 0 && tiles > 0) {
        CascadeParams cp{};
        cp.q = static_cast<const uint16_t *>(q);
        cp.tables = block_tables;
        cp.max_blocks = max_blocks;
        cp.num_blocks = p->num_blocks;
        cp.seq_lens = seq_lens;
        cp.batch = batch;
        cp.group_seqs = group_seqs;
        cp.group_size = group_size;
        cp.shared_tokens = shared_tokens;
        cp.num_q_heads = num_q_heads;
        cp.num_kv_heads = p->num_kv_heads;
        cp.g = g;
        cp.scale_log2 = scale * 1.4426950408889634f;
        cp.tiles_per_split = (tiles + ps - 1) / ps;
        cp.ws_o = static_cast<float *>(workspace);
        cp.max_splits = ps + ms;
        cp.ws_lse = cp.ws_o + (size_t)batch * num_q_heads * cp.max_splits * kCsD;
        cp.err = p->err;
        // groups of at most 64 rows: duplicated rows, keys split over two threads
        const bool dup = (long long)group_size * g <= 64;
        const bool tw = test_waits_enabled(), f16 = p->dtype == KV_F16;
        auto fn = f16 ? (tw ? (dup ? cascade_prefix_kernel<true, true, true> : cascade_prefix_kernel<false, true, true>)
                            : (dup ? cascade_prefix_kernel<true, false, true> : cascade_prefix_kernel<false, false, true>))
                      : (tw ? (dup ? cascade_prefix_kernel<true, true, false> : cascade_prefix_kernel<false, true, false>)
                            : (dup ? cascade_prefix_kernel<true, false, false> : cascade_prefix_kernel<false, false, false>));
        if (kv_status st0 = cuda_status(
                cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kCsSmemBytes)))
            return st0;
        // The whole shared memory as carveout: an SM holding a prefix CTA
        // (about 164 KiB) then keeps room for a suffix decode CTA beside it
        // (without, the SM was sized for the prefix CTA alone and the suffix
        // ran on the 24 other SMs only until the prefix grid ended).
        if (kv_status st0 = cuda_status(cudaFuncSetAttribute(
                fn, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared)))
            return st0;
        const dim3 grid(ps, p->num_kv_heads, num_groups);
        fn<<<grid, kCsThreads, kCsSmemBytes, s>>>(p->tmap_k, p->tmap_v, cp);
        if (kv_status st1 = cuda_status(cudaGetLastError())) return st1;
        a.overlap_previous = fused_merges;
    }
    return launch_decode(a, false);
}

}  // extern "C"
