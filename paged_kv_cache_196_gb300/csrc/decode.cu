// Paged decode attention, its contiguous (vAttention-style) twin, and the
// split-KV log-sum-exp merge.
//
// Maths: o = softmax(scale * q K^T) V over the sequence's logical keys, read
// through the block table ("PagedAttention Nedir?", "Nasil Calisir?" step 4)
// or from one contiguous per-request range ("Makale Bulteni -- vAttention",
// "Iddia ve Gerceklik: vAttention").  The score matrix is never written out:
// keys are visited block by block with a running max and sum ("PagedAttention
// Nedir?", "FlashAttention ile Ayni mi?": the large intermediate attention
// matrix is not materialised).
//
// Work decomposition.  One CTA handles (split s, kv head h, sequence b): the
// blocks [s*PB, min((s+1)*PB, ceil(L/16))) of that sequence for all g query
// heads that read kv head h, so every K/V byte is fetched once per kv head.
// Warp kNW (the producer) copies the CTA's block-table slice into shared
// memory once, then streams each (block, head) tile -- 16 tokens x head_dim,
// contiguous in the pool -- with one-dimensional bulk (TMA) copies into an
// NSTAGE-deep ring of shared-memory stages guarded by mbarriers.  Consumer
// warp w owns the blocks i = w (mod kNW); it keeps its own running max, sum
// and output accumulators, so no CTA-wide barrier is taken per block.  The kNW
// partial states are merged once at the end; with several splits per
// sequence a second kernel merges the splits through their log-sum-exp.
//
// Inside a consumer warp, half-warp hf takes token 2p+hf of pass p and lane
// c = lane % 16 owns head_dim/16 consecutive dimensions.  Partial dot products
// for the g heads are reduced across the 16 lanes with a reduce-scatter
// (each exchange step halves the number of values carried), ending with lane c
// holding the score of head c / (16/G).  Products use packed fp32x2 FMAs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace pkv {

constexpr int kNW = 4;                   // consumer warps per CTA
constexpr int kDecodeThreads = (kNW + 1) * 32;
constexpr int kBS = 16;                  // tokens per block
constexpr int kMaxPartBlocks = 1024;     // blocks per split (bounds the table slice in smem)
constexpr int kNStage = 8;               // pipeline depth (a multiple of kNW)
constexpr int kDecodeMinBlocks = 3;      // CTAs per SM the CUDA-core decode is built for
constexpr int kTcMinGroup = 3;           // smallest head group routed to the tensor-core decode
constexpr int kTcDeepBlocks = 256;       // partitions this long use the deep-ring tensor-core decode
// Balanced schedules (kv_decode_schedule), int32 words:
//   [0] CTAs C, [1] pieces P, [2] most pieces of one (sequence, kv head),
//   [3] most blocks of one CTA, [4] deep ring (1) or wide (0), [5] batch,
//   [6] kv heads, [7] partial results per (sequence, query head) in the
//   workspace;
//   [8, 8 + C] the first piece of each CTA, then P;
//   from sched_piece_off(C) (a multiple of 4 words): P pieces of 4 words
//   {b, h | split << 16, first block, blocks | pieces of the pair << 16}.
constexpr int kSchedHeader = 8;
inline size_t sched_piece_off(int ctas) { return ((size_t)kSchedHeader + ctas + 1 + 3) & ~size_t(3); }
static_assert(kNStage % kNW == 0, "each stage must belong to one consumer warp");

struct DecodeKParams {
    const void *q;
    const char *k_pool;
    const char *v_pool;
    const int32_t *tables;
    int max_blocks;
    int num_blocks;
    const unsigned long long *k_bases;
    const unsigned long long *v_bases;
    const int32_t *req_ids;
    const long long *mapped_tokens;
    const CUtensorMap *req_maps;
    long long head_stride;
    int max_requests;
    const int32_t *seq_lens;
    int num_q_heads;
    int num_kv_heads;
    int g;
    float scale_log2;  // scale * log2(e): scores are kept in the log2 domain
    int part_blocks;
    int max_splits;
    const int32_t *start_tokens;  // cascade: tokens of each sequence attended elsewhere, or null
    int part_base;                // cascade: workspace slots [0, part_base) hold those results
    // fused append (tensor-core decode only): each sequence's new token
    // ([batch][num_kv_heads][128], 16-bit) and its pool slot (paged path; the
    // contiguous path writes row seq_lens[b] - 1), or null
    const uint4 *new_k;
    const uint4 *new_v;
    const int64_t *new_slots;
    // order in which the grid takes the sequences (a permutation of the
    // batch, e.g. longest first so a single wave loads the SMs evenly), or null
    const int32_t *seq_order;
    // balanced schedule (tensor-core decode): CTA c runs pieces
    // [sched_cta[c], sched_cta[c + 1]) of sched_pieces, each a run of blocks
    // of one (sequence, kv head): {b, h | split << 16, first block,
    // blocks | pieces of the pair << 16}; null for the grid-indexed plan
    const int32_t *sched_cta;
    const int4 *sched_pieces;
    int sched_npieces;
    int batch;
    // launched to overlap the previous kernel in the stream (the cascade's
    // prefix kernel): no CTA exits before that kernel has completed, so
    // nothing after this grid can start before it either
    int overlap;
    // launched to overlap the previous kernel in the stream: every CTA waits
    // for it before touching memory, and lets the next launch begin at once
    int chain;
    void *out;
    int out_type;  // kv_dtype of out
    float *lse;
    float *ws_o;
    float *ws_lse;
    int *counters;  // per (sequence, kv head) arrival counters for the fused merge, or null
    int *err;
};

// Element types of the pool (the kv_dtype values): ET = KV_F32, KV_BF16 or KV_F16.
template <int D, int ET>
struct TileShape {
    static constexpr int kElem = ET == KV_F32 ? 4 : 2;
    static constexpr int kBytes = kBS * D * kElem;  // one (block, kv head) tile
    static constexpr int kDPL = D / 16;             // dimensions per lane
    static constexpr int kPairs = kDPL / 2;
};

// Two 16-bit elements of type ET as fp32 (exact).
template <int ET>
KV_DEVICE float2 half2_to_float2(uint32_t w) {
    if constexpr (ET == KV_BF16)
        return bf16x2_to_float2(w);
    else
        return f16x2_to_float2(w);
}

// Loads this lane's kDPL dimensions of row t of a tile as fp32 pairs.
template <int D, int ET>
KV_DEVICE void load_row(const char *tile, int t, int c, float2 (&x)[TileShape<D, ET>::kPairs]) {
    using S = TileShape<D, ET>;
    const char *row = tile + (size_t)t * D * S::kElem + (size_t)c * S::kDPL * S::kElem;
    if constexpr (ET != KV_F32) {
        if constexpr (S::kDPL == 8) {
            const uint4 w = *reinterpret_cast<const uint4 *>(row);
            x[0] = half2_to_float2<ET>(w.x);
            x[1] = half2_to_float2<ET>(w.y);
            x[2] = half2_to_float2<ET>(w.z);
            x[3] = half2_to_float2<ET>(w.w);
        } else {
            const uint2 w = *reinterpret_cast<const uint2 *>(row);
            x[0] = half2_to_float2<ET>(w.x);
            x[1] = half2_to_float2<ET>(w.y);
        }
    } else {
#pragma unroll
        for (int i = 0; i < S::kDPL / 4; ++i) {
            const float4 f = reinterpret_cast<const float4 *>(row)[i];
            x[2 * i] = make_float2(f.x, f.y);
            x[2 * i + 1] = make_float2(f.z, f.w);
        }
    }
}

// Sum of v[0..N) over the 16 lanes of a half-warp, scattered: on return v[0]
// of lane c holds the total of entry c / (16/N_initial).  DIST walks 8,4,2,1.
template <int N, int DIST>
KV_DEVICE void reduce_scatter16(float *v, int lane) {
    if constexpr (DIST > 0) {
        if constexpr (N > 1) {
            constexpr int H = N / 2;
            const bool up = (lane & DIST) != 0;
#pragma unroll
            for (int k = 0; k < H; ++k) {
                const float send = up ? v[k] : v[k + H];
                const float keep = up ? v[k + H] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, send, DIST);
            }
            reduce_scatter16<H, DIST / 2>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], DIST);
            reduce_scatter16<1, DIST / 2>(v, lane);
        }
    }
}

// Bytes of the stage ring; the final cross-warp merge reuses it.
template <int D, int G, int ET>
constexpr size_t decode_ring_bytes(int nstage = kNStage) {
    const size_t ring = (size_t)nstage * 2 * TileShape<D, ET>::kBytes;
    constexpr size_t merge =
        (size_t)kNW * (G * D + 2 * G) * sizeof(float) + (G * kFuseMaxSplits + 4) * sizeof(float);
    return ((ring > merge ? ring : merge) + 127) / 128 * 128;
}

// Blocks of sequence b before this call's part of it: its first
// start_tokens[b] tokens (clamped to [0, L], whole blocks) were attended by
// the cascade's prefix kernel.
// With p.chain: lets the next launch in the stream begin, then waits for the
// previous kernel to complete (its writes visible) before anything else.
KV_DEVICE void chain_entry(const DecodeKParams &p) {
    if (p.chain) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
}

// With p.overlap, holds the CTA (its thread 0) until the previous kernel in
// the stream has completed.
KV_DEVICE void overlap_exit(const DecodeKParams &p) {
    if (p.overlap && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

KV_DEVICE int start_block(const DecodeKParams &p, int b, long long L) {
    if (!p.start_tokens) return 0;
    long long st = p.start_tokens[b];
    st = st < 0 ? 0 : (st > L ? L : st);
    return (int)(st / kBS);
}

// End of a partition: combine the kNW warp states (running max m, sum l,
// unnormalised output o, all in the log2 domain) into this partition's
// result.  With one partition the result is final.  Otherwise it is written
// to the workspace; the CTA that finishes last for its (sequence, kv head)
// -- found with an arrival counter that it resets afterwards -- merges all
// partitions: o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M).
template <int G, int D>
//
// Cascade: a sequence whose prefix was attended by the prefix kernel (pre > 0)
// has pre more partial results in workspace slots [0, pre); this call's
// partitions use slots part_base + split, and the merge takes both.
//
// w ([G][kFuseMaxSplits] floats) and flag hold the merge's weights and
// decision.  With release set, the consumer warps meet the producer warp on
// named barrier 2 as soon as sm_o / sm_m / sm_l have been read, so that the
// producer may refill the ring they live in while the merge runs.
KV_DEVICE void finish_partition(const DecodeKParams &p, const float *sm_o, const float *sm_m,
                                const float *sm_l, int b, int h, int split, int nsplit, int pre,
                                int tid, float *w, int *flag, bool release) {
    const int ntot = pre + nsplit;
    constexpr float kLn2 = 0.6931471805599453f;
    // Cascade, one partition after the prefix: this CTA is the only one left
    // to contribute once the prefix grid is complete, so it merges its result
    // with the prefix's partial results itself (no workspace write of its
    // own, no arrival counter).  Only with fused merges: then no merge kernel
    // runs afterwards over these rows.
    const bool direct = pre > 0 && nsplit == 1 && p.counters && ntot <= kFuseMaxSplits;
    if (direct) asm volatile("griddepcontrol.wait;" ::: "memory");  // the prefix's results are complete
    for (int idx = tid; idx < p.g * D; idx += kNW * 32) {
        const int j = idx / D, d = idx - j * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kNW; ++w) M = fmaxf(M, sm_m[w * G + j]);
        float num = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kNW; ++w) {
                const float f = exp2f(sm_m[w * G + j] - M);
                num += f * sm_o[(w * G + j) * D + d];
                den += f * sm_l[w * G + j];
            }
        }
        const float o = den > 0.f ? num / den : 0.f;
        const float lse2 = den > 0.f ? M + log2f(den) : -INFINITY;
        const size_t row = (size_t)b * p.num_q_heads + h * p.g + j;
        if (ntot == 1) {
            store_out(p.out, row * D + d, o, p.out_type);
            if (p.lse && d == 0) p.lse[row] = lse2 * kLn2;
        } else if (direct) {
            // o = (2^(lse2 - Mx) o + sum_s 2^(lse_s - Mx) o_s) / (the same weights' sum)
            const float *ls = p.ws_lse + row * p.max_splits;
            const float *os = p.ws_o + row * p.max_splits * D + d;
            float Mx = lse2;
            for (int s2 = 0; s2 < pre; ++s2) Mx = fmaxf(Mx, __ldcg(ls + s2));
            float acc = 0.f, wsum = 0.f;
            if (Mx != -INFINITY) {
                wsum = exp2f(lse2 - Mx);
                acc = wsum * o;
                for (int s2 = 0; s2 < pre; ++s2) {
                    const float e = exp2f(__ldcg(ls + s2) - Mx);
                    acc += e * __ldcg(os + (size_t)s2 * D);
                    wsum += e;
                }
            }
            store_out(p.out, row * D + d, wsum > 0.f ? acc / wsum : 0.f, p.out_type);
            if (p.lse && d == 0) p.lse[row] = wsum > 0.f ? (Mx + log2f(wsum)) * kLn2 : -INFINITY;
        } else {
            p.ws_o[(row * p.max_splits + p.part_base + split) * D + d] = o;
            if (d == 0) p.ws_lse[row * p.max_splits + p.part_base + split] = lse2;
        }
    }
    if (release) named_bar_sync(2, kDecodeThreads);
    if (ntot == 1 || direct || !p.counters || ntot > kFuseMaxSplits) return;

    // ---- fused merge by the last-arriving CTA of this (sequence, kv head)
    __threadfence();  // partial results visible device-wide before the arrival
    named_bar_sync(1, kNW * 32);
    if (tid == 0) {
        const int old = atomicAdd(p.counters + (size_t)b * p.num_kv_heads + h, 1);
        *flag = old == nsplit - 1;
    }
    named_bar_sync(1, kNW * 32);
    if (!*flag) return;
    __threadfence();
    // The cascade's prefix kernel may still be running when this grid was
    // launched to overlap it: its partial results are complete once it is.
    if (pre > 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    // split weights per head: 2^(lse_s - M) / sum
    for (int j = tid; j < p.g; j += kNW * 32) {
        const size_t row = (size_t)b * p.num_q_heads + h * p.g + j;
        const float *ls = p.ws_lse + row * p.max_splits;
        float M = -INFINITY;
        for (int s2 = 0; s2 < ntot; ++s2) M = fmaxf(M, __ldcg(ls + (s2 < pre ? s2 : p.part_base + s2 - pre)));
        float den = 0.f;
        for (int s2 = 0; s2 < ntot; ++s2) {
            const float e =
                M == -INFINITY ? 0.f : exp2f(__ldcg(ls + (s2 < pre ? s2 : p.part_base + s2 - pre)) - M);
            w[j * kFuseMaxSplits + s2] = e;
            den += e;
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        for (int s2 = 0; s2 < ntot; ++s2) w[j * kFuseMaxSplits + s2] *= inv;
        if (p.lse) p.lse[row] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
    }
    named_bar_sync(1, kNW * 32);
    for (int idx = tid; idx < p.g * (D / 4); idx += kNW * 32) {
        const int j = idx / (D / 4), d4 = idx - j * (D / 4);
        const size_t row = (size_t)b * p.num_q_heads + h * p.g + j;
        const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + row * p.max_splits * D) + d4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s2 = 0; s2 < ntot; ++s2) {
            const float ws = w[j * kFuseMaxSplits + s2];
            const float4 v = __ldcg(src + (size_t)(s2 < pre ? s2 : p.part_base + s2 - pre) * (D / 4));
            acc.x += ws * v.x;
            acc.y += ws * v.y;
            acc.z += ws * v.z;
            acc.w += ws * v.w;
        }
        if (p.out_type != KV_F32) {
            const size_t o0 = row * D + 4 * d4;
            store_out(p.out, o0, acc.x, p.out_type);
            store_out(p.out, o0 + 1, acc.y, p.out_type);
            store_out(p.out, o0 + 2, acc.z, p.out_type);
            store_out(p.out, o0 + 3, acc.w, p.out_type);
        } else {
            reinterpret_cast<float4 *>(p.out)[(row * D) / 4 + d4] = acc;
        }
    }
    if (tid == 0) p.counters[(size_t)b * p.num_kv_heads + h] = 0;  // ready for the next call
}

// HS = 1: the two half-warps take different tokens (2 per pass) and every
// lane carries all G heads.  HS = 2: both halves take the same token and each
// carries G/2 heads (half the q and accumulator registers, for large G).
template <int D, int G, int HS, int ET, bool LINEAR>
__global__ void __launch_bounds__(kDecodeThreads, kDecodeMinBlocks) decode_kernel(const DecodeKParams p) {
    using S = TileShape<D, ET>;
    constexpr int kTile = S::kBytes;
    constexpr int kPairs = S::kPairs;
    constexpr int GH = G / HS;                 // heads per lane
    constexpr int kLanesPerHead = 16 / GH;
    constexpr int kPasses = 8 * HS;            // passes over a 16-token block
    static_assert(GH >= 1 && (HS == 1 || HS == 2), "bad head split");

    const int split = blockIdx.x, h = blockIdx.y;
    const int b = p.seq_order ? __ldg(p.seq_order + blockIdx.z) : (int)blockIdx.z;
    if (b < 0 || b >= (int)gridDim.z) {  // not a permutation of the batch
        if (threadIdx.x == 0 && split == 0 && h == 0) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- the slice of keys this CTA owns
    long long L = p.seq_lens[b];
    const char *k_lin = nullptr, *v_lin = nullptr;
    if constexpr (LINEAR) {
        const int req = p.req_ids[b];
        if (req < 0 || req >= p.max_requests || p.k_bases[req] == 0) {
            if (tid == 0 && split == 0 && h == 0) atomicOr(p.err, KV_DEVERR_UNMAPPED);
            L = 0;
        } else {
            const long long mapped = p.mapped_tokens[req];
            if (L > mapped) {
                if (tid == 0 && split == 0 && h == 0) atomicOr(p.err, KV_DEVERR_UNMAPPED);
                L = mapped;
            }
            k_lin = reinterpret_cast<const char *>(p.k_bases[req]);
            v_lin = reinterpret_cast<const char *>(p.v_bases[req]);
        }
    }
    // The split plan covers max_blocks blocks (the table width, or the
    // contiguous path's max_tokens); longer lengths are clamped and flagged.
    if (L > (long long)p.max_blocks * kBS) {
        if (tid == 0 && split == 0 && h == 0)
            atomicOr(p.err, LINEAR ? KV_DEVERR_UNMAPPED : KV_DEVERR_BLOCK_RANGE);
        L = (long long)p.max_blocks * kBS;
    }
    if (L < 0) L = 0;
    const int nblk = (int)((L + kBS - 1) / kBS);
    const int sblk = start_block(p, b, L);
    const int pre = sblk > 0 ? p.part_base : 0;  // partial results of the cascade's prefix
    const int blk0 = sblk + split * p.part_blocks;
    if (blk0 >= nblk && split > 0) return;  // nothing for this split (uniform across the CTA)
    const int nloc = max(0, min(p.part_blocks, nblk - blk0));
    const int nsplit = max(1, (nblk - sblk + p.part_blocks - 1) / p.part_blocks);

    // ---- shared memory
    extern __shared__ __align__(128) char smem[];
    char *stages = smem;                                                   // kNStage x (K, V)
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + decode_ring_bytes<D, G, ET>());
    uint64_t *empty = full + kNStage;
    int *stage_valid = reinterpret_cast<int *>(empty + kNStage);
    float2 *pscr = reinterpret_cast<float2 *>(stage_valid + kNStage);      // [kNW][16][G]
    float *ascr = reinterpret_cast<float *>(pscr + kNW * kBS * G);         // [kNW][G]
    int32_t *tbl = reinterpret_cast<int32_t *>(ascr + kNW * G);            // [part_blocks]

    if (warp == kNW) {
        if constexpr (!LINEAR) {
            const int32_t *row = p.tables + (size_t)b * p.max_blocks + blk0;
            for (int i = lane; i < nloc; i += 32) tbl[i] = __ldg(row + i);
        }
        if (lane == 0) {
            for (int s = 0; s < kNStage; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], 32);
            }
            mbar_init_fence();
        }
    }
    __syncthreads();

    // ======================================================== producer warp
    if (warp == kNW) {
        if (lane == 0) {
            const uint64_t policy = l2_evict_first_policy();
            int issued = 0;
            for (int i = 0; i < nloc; ++i) {
                const int st = i % kNStage, r = i / kNStage;
                if (r > 0 && !mbar_wait(&empty[st], (r - 1) & 1, p.err)) break;
                const char *ks;
                const char *vs;
                bool valid = true;
                if constexpr (LINEAR) {
                    const size_t off =
                        ((size_t)h * p.head_stride + (size_t)(blk0 + i) * kBS) * D * S::kElem;
                    ks = k_lin + off;
                    vs = v_lin + off;
                } else {
                    const int id = tbl[i];
                    valid = id >= 0 && id < p.num_blocks;
                    if (!valid) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
                    const size_t off = ((size_t)(valid ? id : 0) * p.num_kv_heads + h) * kTile;
                    ks = p.k_pool + off;
                    vs = p.v_pool + off;
                }
                stage_valid[st] = valid ? 1 : 0;
                char *dst = stages + st * 2 * kTile;
                if (valid) {
                    mbar_arrive_expect_tx(&full[st], 2 * kTile);
                    bulk_g2s(dst, ks, kTile, &full[st], policy);
                    bulk_g2s(dst + kTile, vs, kTile, &full[st], policy);
                } else {
                    mbar_arrive(&full[st]);
                }
                issued = i + 1;
            }
            // Do not leave while a copy into this CTA's shared memory may be in flight.
            for (int st = 0; st < kNStage && st < issued; ++st) {
                const int r_last = (issued - 1 - st) / kNStage;
                mbar_wait_drain(&full[st], r_last & 1, p.err);
            }
        }
        return;
    }

    // ======================================================== consumer warps
    const int hf = lane >> 4, c = lane & 15;
    const int hoff = HS == 2 ? hf * GH : 0;             // first head this lane carries
    const int my_head = hoff + c / kLanesPerHead;       // head whose score this lane ends with
    const bool rep = (c % kLanesPerHead) == 0;          // one writer per (half, head)
    const bool rep_once = rep && (HS == 2 || hf == 0);  // one writer per head

    // q for this lane's heads and dimensions, pre-scaled into the log2 domain.
    float2 qv[GH][kPairs];
#pragma unroll
    for (int j = 0; j < GH; ++j) {
        const int jj = hoff + j;
        if (jj < p.g) {
            const size_t base = ((size_t)b * p.num_q_heads + h * p.g + jj) * D + c * S::kDPL;
            float2 x[kPairs];
            load_row<D, ET>(reinterpret_cast<const char *>(p.q) + base * S::kElem, 0, 0, x);
#pragma unroll
            for (int m = 0; m < kPairs; ++m)
                qv[j][m] = make_float2(x[m].x * p.scale_log2, x[m].y * p.scale_log2);
        } else {
#pragma unroll
            for (int m = 0; m < kPairs; ++m) qv[j][m] = make_float2(0.f, 0.f);
        }
    }

    float m_run = -INFINITY, l_run = 0.f;
    float2 acc[GH][kPairs];
#pragma unroll
    for (int j = 0; j < GH; ++j)
#pragma unroll
        for (int m = 0; m < kPairs; ++m) acc[j][m] = make_float2(0.f, 0.f);

    float2 *pw = pscr + warp * kBS * G;
    float *aw = ascr + warp * G;

    for (int i = warp; i < nloc; i += kNW) {
        const int st = i % kNStage, r = i / kNStage;
        if (!mbar_wait(&full[st], r & 1, p.err)) break;
        const char *kt = stages + st * 2 * kTile;
        const char *vt = kt + kTile;
        int ntok = (int)min((long long)kBS, L - (long long)(blk0 + i) * kBS);
        if (!stage_valid[st]) ntok = 0;

        const bool full_block = ntok == kBS;  // uniform across the warp

        // ---- scores for this lane's head
        float s[kPasses];
#pragma unroll
        for (int pass = 0; pass < kPasses; ++pass) {
            const int t = HS == 1 ? 2 * pass + hf : pass;
            float2 kx[kPairs];
            load_row<D, ET>(kt, t, c, kx);
            float part[GH];
#pragma unroll
            for (int j = 0; j < GH; ++j) {
                float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int m = 0; m < kPairs; ++m) a2 = ffma2(qv[j][m], kx[m], a2);
                part[j] = a2.x + a2.y;
            }
            reduce_scatter16<GH, 8>(part, c);
            s[pass] = (full_block || t < ntok) ? part[0] : -INFINITY;
        }

        // ---- online softmax update for this lane's head
        float mb = s[0];
#pragma unroll
        for (int pass = 1; pass < kPasses; ++pass) mb = fmaxf(mb, s[pass]);
        if (HS == 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
        const float m_new = fmaxf(m_run, mb);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = exp2f(m_run - m_use);
        float psum = 0.f;
#pragma unroll
        for (int pass = 0; pass < kPasses; ++pass) {
            const float pr = exp2f(s[pass] - m_use);
            psum += pr;
            const int t = HS == 1 ? 2 * pass + hf : pass;
            if (rep) pw[t * G + my_head] = make_float2(pr, pr);
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        if (rep_once) aw[my_head] = alpha;
        __syncwarp();

        // ---- rescale and accumulate P V
#pragma unroll
        for (int j = 0; j < GH; ++j) {
            const float a = aw[hoff + j];
            const float2 a2 = make_float2(a, a);
#pragma unroll
            for (int m = 0; m < kPairs; ++m) acc[j][m] = __fmul2_rn(acc[j][m], a2);
        }
        if (full_block) {
#pragma unroll
            for (int pass = 0; pass < kPasses; ++pass) {
                const int t = HS == 1 ? 2 * pass + hf : pass;
                float2 vx[kPairs];
                load_row<D, ET>(vt, t, c, vx);
                const float2 *prow = pw + t * G + hoff;
#pragma unroll
                for (int j = 0; j < GH; ++j) {
                    const float2 pj = prow[j];
#pragma unroll
                    for (int m = 0; m < kPairs; ++m) acc[j][m] = ffma2(pj, vx[m], acc[j][m]);
                }
            }
        } else {
            // Partial or invalid block: tokens at or past ntok are skipped, never
            // multiplied by a zero weight -- the unused slots may hold anything.
#pragma unroll
            for (int pass = 0; pass < kPasses; ++pass) {
                const int t = HS == 1 ? 2 * pass + hf : pass;
                if (t < ntok) {
                    float2 vx[kPairs];
                    load_row<D, ET>(vt, t, c, vx);
                    const float2 *prow = pw + t * G + hoff;
#pragma unroll
                    for (int j = 0; j < GH; ++j) {
                        const float2 pj = prow[j];
#pragma unroll
                        for (int m = 0; m < kPairs; ++m) acc[j][m] = ffma2(pj, vx[m], acc[j][m]);
                    }
                }
            }
        }
        __syncwarp();
        mbar_arrive(&empty[st]);
    }

    if constexpr (HS == 1) {
        // merge the two half-warps (same heads and dims, disjoint tokens)
#pragma unroll
        for (int j = 0; j < GH; ++j)
#pragma unroll
            for (int m = 0; m < kPairs; ++m) {
                acc[j][m].x += __shfl_xor_sync(0xffffffffu, acc[j][m].x, 16);
                acc[j][m].y += __shfl_xor_sync(0xffffffffu, acc[j][m].y, 16);
            }
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
    }

    // ---- merge the kNW warps through shared memory (reusing the stage ring)
    named_bar_sync(1, kNW * 32);  // every consumer is done reading stages
    float *sm_o = reinterpret_cast<float *>(stages);   // [kNW][G][D]
    float *sm_m = sm_o + kNW * G * D;                  // [kNW][G]
    float *sm_l = sm_m + kNW * G;                      // [kNW][G]
    if (HS == 2 || hf == 0) {
#pragma unroll
        for (int j = 0; j < GH; ++j)
#pragma unroll
            for (int m = 0; m < kPairs; ++m)
                *reinterpret_cast<float2 *>(sm_o + (warp * G + hoff + j) * D + c * S::kDPL +
                                            2 * m) = acc[j][m];
        if (rep_once) {
            sm_m[warp * G + my_head] = m_run;
            sm_l[warp * G + my_head] = l_run;
        }
    }
    named_bar_sync(1, kNW * 32);

    float *mw = sm_l + kNW * G;  // merge weights, then a flag (still in the ring)
    finish_partition<G, D>(p, sm_o, sm_m, sm_l, b, h, split, nsplit, pre, tid, mw,
                           reinterpret_cast<int *>(mw + G * kFuseMaxSplits), false);
}

// ---------------------------------------------------------------------------
// Tensor-core decode for GQA groups of 3..8 query heads per kv head (bf16,
// head_dim 128).  With g heads sharing every K/V element the CUDA-core kernel
// above is issue-bound (ncu: ~55% issue-active at g = 4, about half the HBM
// rate at g = 8, where it needs ~2x the instructions per byte); here the two
// small contractions of each
// 16-token block run as warp-level mma.sync (the 16 tokens are M, the eight
// heads N):
//   S^T[16 tok][8 heads] = K[16][128] . Q^T        (8 k-steps of 16 dims)
//   O^T[128][8] += V^T[128][16 tok] . P^T[16][8]    (8 m-tiles of 16 dims)
// K/V tiles arrive by tiled TMA with 128-byte swizzle (two 16 x 64 boxes per
// tile) so ldmatrix reads are bank-conflict-free.  P^T is formed from the S
// fragment with movmatrix.trans and fed as bf16 hi + lo parts (two MMAs), so
// the weights keep ~16 bits of precision.  Same CTA decomposition, pipeline,
// split plan, masking and final merge as decode_kernel.
// ---------------------------------------------------------------------------
namespace mma {

KV_DEVICE void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
KV_DEVICE void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
KV_DEVICE uint32_t movm_t(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}
// d += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate
KV_DEVICE void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// d += A(16x16 fp16, row) * B(16x8 fp16, col), fp32 accumulate
KV_DEVICE void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                       uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
KV_DEVICE uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
KV_DEVICE uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
KV_DEVICE float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
KV_DEVICE float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

KV_DEVICE void tma2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                     uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

}  // namespace mma

constexpr int kTcTile = 16 * 128 * 2;  // one (block, head) tile: 4 KiB, two 2 KiB swizzled halves

// The Q^T fragment of k-step kk for this lane: held in registers, or staged
// in shared memory as [kk][lane] pairs of words (one copy for all warps).
KV_DEVICE void q_fragment(const uint32_t (&qf)[8][2], int kk, int, uint32_t &q0, uint32_t &q1) {
    q0 = qf[kk][0];
    q1 = qf[kk][1];
}
KV_DEVICE void q_fragment(const uint2 *qs, int kk, int lane, uint32_t &q0, uint32_t &q1) {
    const uint2 v = qs[kk * 32 + lane];
    q0 = v.x;
    q1 = v.y;
}

// One 16-token block for the 8 (padded) query heads of a warp: S^T = K Q^T
// on mma.sync, online softmax in the log2 domain, O^T += V^T P^T with P split
// into bf16 hi + lo parts.  kt / vt: shared addresses of the block's swizzled
// K and V tiles; ntok: valid tokens in the block (the rest are masked, their V
// lanes zeroed).  State (m_run, l_run, o) is this lane's share.
// F16: the pool, q and the weights are IEEE half precision (one PV MMA with
// fp16 weights, 11 significant bits); otherwise bf16, the weights split into
// bf16 hi + lo parts (two PV MMAs).
template <bool F16, typename QF>
KV_DEVICE void tc_attend_block(const QF &qf, uint32_t kt, uint32_t vt, int ntok,
                               float scale_log2, int lane, float (&m_run)[2], float (&l_run)[2],
                               float (&o)[8][4]) {
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3;
    const int rowA = (lane & 7) + (mi & 1) * 8;   // K: token row (non-transposed A)
    const int tokV = (lane & 7) + (mi >> 1) * 8;  // V: token row (transposed A)
    // ---- S^T = K Q^T
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const int chunk = 2 * (kk & 3) + (mi >> 1);
        const uint32_t addr = kt + (kk >> 2) * (kTcTile / 2) + rowA * 128 + ((chunk ^ (rowA & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        mma::ldsm_x4(addr, a0, a1, a2, a3);
        uint32_t q0, q1;
        q_fragment(qf, kk, lane, q0, q1);
        if constexpr (F16)
            mma::mma_f16(c, a0, a1, a2, a3, q0, q1);
        else
            mma::mma_bf16(c, a0, a1, a2, a3, q0, q1);
    }
    // c0,c1: token g, heads 2t,2t+1; c2,c3: token g+8
    const bool v0 = g < ntok, v1 = g + 8 < ntok;
    float s0 = v0 ? c[0] * scale_log2 : -INFINITY;
    float s1 = v0 ? c[1] * scale_log2 : -INFINITY;
    float s2 = v1 ? c[2] * scale_log2 : -INFINITY;
    float s3 = v1 ? c[3] * scale_log2 : -INFINITY;
    float mh0 = fmaxf(s0, s2), mh1 = fmaxf(s1, s3);
#pragma unroll
    for (int x = 4; x <= 16; x <<= 1) {
        mh0 = fmaxf(mh0, __shfl_xor_sync(0xffffffffu, mh0, x));
        mh1 = fmaxf(mh1, __shfl_xor_sync(0xffffffffu, mh1, x));
    }
    const float mn0 = fmaxf(m_run[0], mh0), mn1 = fmaxf(m_run[1], mh1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = exp2f(m_run[0] - mu0), al1 = exp2f(m_run[1] - mu1);
    m_run[0] = mn0;
    m_run[1] = mn1;
    const float p0 = exp2f(s0 - mu0), p1 = exp2f(s1 - mu1);
    const float p2 = exp2f(s2 - mu0), p3 = exp2f(s3 - mu1);
    l_run[0] = l_run[0] * al0 + (p0 + p2);
    l_run[1] = l_run[1] * al1 + (p1 + p3);
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
        }
    }
    // ---- P^T fragments (fp16, or bf16 hi + lo), via transpose of the S layout
    uint32_t bh0, bh1, bl0 = 0, bl1 = 0;
    if constexpr (F16) {
        bh0 = mma::movm_t(mma::pack_f16(p0, p1));
        bh1 = mma::movm_t(mma::pack_f16(p2, p3));
    } else {
        const uint32_t h01 = mma::pack_bf16(p0, p1), h23 = mma::pack_bf16(p2, p3);
        const uint32_t l01 = mma::pack_bf16(p0 - mma::bf16_lo_f(h01), p1 - mma::bf16_hi_f(h01));
        const uint32_t l23 = mma::pack_bf16(p2 - mma::bf16_lo_f(h23), p3 - mma::bf16_hi_f(h23));
        bh0 = mma::movm_t(h01);
        bh1 = mma::movm_t(h23);
        bl0 = mma::movm_t(l01);
        bl1 = mma::movm_t(l23);
    }
    // token masks for the V fragments (pairs 2t,2t+1 and 2t+8,2t+9)
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (ntok < kBS) {
        mlo = (2 * t < ntok ? 0xffffu : 0u) | (2 * t + 1 < ntok ? 0xffff0000u : 0u);
        mhi = (2 * t + 8 < ntok ? 0xffffu : 0u) | (2 * t + 9 < ntok ? 0xffff0000u : 0u);
    }
    // ---- O^T += V^T P^T
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int cidx = 2 * mt + (mi & 1);
        const uint32_t addr = vt + (cidx >> 3) * (kTcTile / 2) + tokV * 128 +
                              (((cidx & 7) ^ (tokV & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        mma::ldsm_x4_t(addr, a0, a1, a2, a3);
        // a0/a1: tokens 2t,2t+1; a2/a3: tokens 2t+8,2t+9.  Unused slots may
        // hold anything: their lanes are zeroed, never multiplied by 0.
        a0 &= mlo;
        a1 &= mlo;
        a2 &= mhi;
        a3 &= mhi;
        if constexpr (F16) {
            mma::mma_f16(o[mt], a0, a1, a2, a3, bh0, bh1);
        } else {
            mma::mma_bf16(o[mt], a0, a1, a2, a3, bh0, bh1);
            mma::mma_bf16(o[mt], a0, a1, a2, a3, bl0, bl1);
        }
    }
}


// NST ring stages (a multiple of kNW: stage st belongs to warp st % kNW),
// compiled for MINB resident CTAs per SM.
template <bool LINEAR, int NST, int MINB, bool TW, bool F16>
__global__ void __launch_bounds__(kDecodeThreads, MINB)
    decode_tc_kernel(const __grid_constant__ CUtensorMap pool_k_map,
                     const __grid_constant__ CUtensorMap pool_v_map, const DecodeKParams p) {
    constexpr int G = 8, D = 128;
    // With launch overlap the paged decode reads the inputs a decode step
    // never writes (block tables, lengths, order, q) before it waits for the
    // previous kernel, and everything else after: the table slice and q are
    // on chip when that kernel ends.  The contiguous path waits first (its
    // request maps and mapped lengths change between calls).
    if constexpr (LINEAR) {
        chain_entry(p);
    } else if (p.chain) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    const int split = blockIdx.x, h = blockIdx.y;
    const int b = p.seq_order ? __ldg(p.seq_order + blockIdx.z) : (int)blockIdx.z;
    if (b < 0 || b >= (int)gridDim.z) {  // not a permutation of the batch
        if (threadIdx.x == 0 && split == 0 && h == 0) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
        overlap_exit(p);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    long long L = p.seq_lens[b];
    const CUtensorMap *map_k = &pool_k_map, *map_v = &pool_v_map;
    int req = -1;             // contiguous path: the sequence's request
    bool len_ok = true;       // L is the sequence's length, not clamped after an error
    if constexpr (LINEAR) {
        req = p.req_ids[b];
        if (req < 0 || req >= p.max_requests || p.k_bases[req] == 0) {
            if (tid == 0 && split == 0 && h == 0) atomicOr(p.err, KV_DEVERR_UNMAPPED);
            L = 0;
            len_ok = false;
        } else {
            const long long mapped = p.mapped_tokens[req];
            if (L > mapped) {
                if (tid == 0 && split == 0 && h == 0) atomicOr(p.err, KV_DEVERR_UNMAPPED);
                L = mapped;
                len_ok = false;
            }
            map_k = p.req_maps + 2 * req;
            map_v = p.req_maps + 2 * req + 1;
        }
    }
    if (L > (long long)p.max_blocks * kBS) {
        if (tid == 0 && split == 0 && h == 0)
            atomicOr(p.err, LINEAR ? KV_DEVERR_UNMAPPED : KV_DEVERR_BLOCK_RANGE);
        L = (long long)p.max_blocks * kBS;
        len_ok = false;
    }
    if (L < 0) L = 0;
    const int nblk = (int)((L + kBS - 1) / kBS);
    const int sblk = start_block(p, b, L);
    const int pre = sblk > 0 ? p.part_base : 0;  // partial results of the cascade's prefix
    const int blk0 = sblk + split * p.part_blocks;
    if (blk0 >= nblk && split > 0) {  // nothing for this split (uniform across the CTA)
        overlap_exit(p);
        return;
    }
    const int nloc = max(0, min(p.part_blocks, nblk - blk0));
    const int nsplit = max(1, (nblk - sblk + p.part_blocks - 1) / p.part_blocks);

    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    char *stages = smem;  // NST x (K tile, V tile), swizzled
    constexpr size_t kRing = decode_ring_bytes<D, G, KV_BF16>(NST);
    static_assert(NST % kNW == 0, "each stage must belong to one consumer warp");
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kRing);
    uint64_t *empty = full + NST;
    int *stage_valid = reinterpret_cast<int *>(empty + NST);
    uint4 *newrow = reinterpret_cast<uint4 *>(stage_valid + NST);  // [32]: fused append's K, V rows
    int32_t *tbl = reinterpret_cast<int32_t *>(newrow + 32);       // [part_blocks]

    if (warp == kNW) {
        if constexpr (!LINEAR) {
            const int32_t *row = p.tables + (size_t)b * p.max_blocks + blk0;
            for (int i = lane; i < nloc; i += 32) tbl[i] = __ldg(row + i);
        }
        if (lane == 0) {
            for (int st = 0; st < NST; ++st) {
                mbar_init(&full[st], 1);
                mbar_init(&empty[st], 32);
            }
            mbar_init_fence();
        }
    }
    __syncthreads();

    if (warp == kNW) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(map_k) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(map_v) : "memory");
        }
        if (!LINEAR && p.chain) asm volatile("griddepcontrol.wait;" ::: "memory");  // before the pool reads
        const uint64_t policy = l2_evict_first_policy();
        int issued = 0;
        for (int i = 0; i < nloc; ++i) {
            const int st = i % NST, r = i / NST;
            bool bad = false;
            if (lane == 0) bad = r > 0 && !mbar_wait<TW>(&empty[st], (r - 1) & 1, p.err);
            if (__shfl_sync(0xffffffffu, bad, 0)) break;
            int y;
            bool valid = true;
            if constexpr (LINEAR) {
                y = (int)((long long)h * p.head_stride + (long long)(blk0 + i) * kBS);
            } else {
                const int id = tbl[i];
                valid = id >= 0 && id < p.num_blocks;
                y = ((valid ? id : 0) * p.num_kv_heads + h) * kBS;
            }
            char *dst = stages + st * 2 * kTcTile;
            if (lane == 0) {
                if (!valid) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
                stage_valid[st] = valid ? 1 : 0;
                if (valid)
                    mbar_arrive_expect_tx(&full[st], 2 * kTcTile);
                else
                    mbar_arrive(&full[st]);
            }
            if (valid) {
                // lane x issues box x: K half 0, K half 1, V half 0, V half 1
                if (lane < 4)
                    mma::tma2d(dst + (lane >> 1) * kTcTile + (lane & 1) * (kTcTile / 2),
                               lane < 2 ? map_k : map_v, (lane & 1) * 64, y, &full[st], policy);
            }
            issued = i + 1;
        }
        if (lane == 0)
            for (int st = 0; st < NST && st < issued; ++st)
                mbar_wait_drain(&full[st], ((issued - 1 - st) / NST) & 1, p.err);
        return;
    }

    // ---- consumer warps: lane = (g = lane / 4, t = lane % 4)
    const int g = lane >> 2, t = lane & 3;
    // Fused append: the last split of (b, h) writes the new token's K/V row
    // (head h) to its pool slot (contiguous path: row L - 1 of the request's
    // head region) and, since the block holding it may have been copied
    // before that write lands, patches the row into its own copy of the
    // sequence's last block.  Lane x < 16 carries 16-byte chunk x of the K
    // row, lane 16 + x chunk x of the V row.
    const bool fuse = p.new_k != nullptr && split == nsplit - 1;
    const bool patch = fuse && nloc > 0 && blk0 + nloc == nblk && (!LINEAR || len_ok);
    // Q^T fragments for the 8 k-steps (head g, dims 16kk + 2t (+1) and +8
    // (+9)), staged once in shared memory by warp 0 and read per block: held
    // in registers they cost the 4-stage instantiation spills at its
    // 72-register budget.
    __shared__ uint2 s_q[8 * 32];
    if (warp == 0) {
        const bool live = g < p.g;
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
            reinterpret_cast<const uint16_t *>(p.q) + ((size_t)b * p.num_q_heads + h * p.g + (live ? g : 0)) * D);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            s_q[kk * 32 + lane] = make_uint2(live ? __ldg(qrow + 8 * kk + t) : 0u,
                                             live ? __ldg(qrow + 8 * kk + 4 + t) : 0u);
    }
    if (!LINEAR && p.chain) asm volatile("griddepcontrol.wait;" ::: "memory");  // before the pool access
    if (fuse && warp == (patch ? (nloc - 1) % kNW : 0)) {
        const size_t src = ((size_t)b * p.num_kv_heads + h) * (D * 2 / 16) + (lane & 15);
        const uint4 v = lane < 16 ? __ldg(p.new_k + src) : __ldg(p.new_v + src);
        newrow[lane] = v;  // kept in shared memory until the last block arrives
        if constexpr (LINEAR) {
            // row L - 1 is mapped (L never exceeds the mapped tokens); after a
            // clamped length nothing is written
            if (len_ok && L > 0) {
                const unsigned long long base = lane < 16 ? p.k_bases[req] : p.v_bases[req];
                reinterpret_cast<uint4 *>(base)[((long long)h * p.head_stride + (L - 1)) * (D * 2 / 16) +
                                                (lane & 15)] = v;
            }
        } else {
            const long long slot = p.new_slots[b];
            if (slot >= 0 && slot < (long long)p.num_blocks * kBS) {
                const long long row = ((slot / kBS) * p.num_kv_heads + h) * kBS + slot % kBS;
                uint4 *dst = reinterpret_cast<uint4 *>(const_cast<char *>(lane < 16 ? p.k_pool : p.v_pool)) +
                             row * (D * 2 / 16) + (lane & 15);
                *dst = v;
            } else if (slot >= 0 && lane == 0) {
                atomicOr(p.err, KV_DEVERR_SLOT_RANGE);
            }
        }
    }
    named_bar_sync(1, kNW * 32);
    // running state for heads 2t, 2t+1 (replicated over g)
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    const uint32_t stage_base = smem_addr(stages);

    for (int i = warp; i < nloc; i += kNW) {
        const int st = i % NST, r = i / NST;
        if (!mbar_wait<TW>(&full[st], r & 1, p.err)) break;
        int ntok = (int)min((long long)kBS, L - (long long)(blk0 + i) * kBS);
        if (!stage_valid[st]) ntok = 0;
        const uint32_t kt = stage_base + st * 2 * kTcTile;
        const uint32_t vt = kt + kTcTile;
        if (patch && i == nloc - 1 && ntok > 0) {
            // the new token is row (L - 1) % 16 of the sequence's last block
            const int orow = (int)((L - 1) % kBS), c = lane & 15;
            char *tile = stages + st * 2 * kTcTile + (lane < 16 ? 0 : kTcTile);
            *reinterpret_cast<uint4 *>(tile + (c >> 3) * (kTcTile / 2) + orow * 128 +
                                       (((c & 7) ^ (orow & 7)) << 4)) = newrow[lane];
            __syncwarp();
        }

        tc_attend_block<F16>(s_q, kt, vt, ntok, p.scale_log2, lane, m_run, l_run, o);
        __syncwarp();
        mbar_arrive(&empty[st]);
    }

    // ---- per-warp totals over the 8 token lanes (g)
#pragma unroll
    for (int x = 4; x <= 16; x <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], x);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], x);
    }
    named_bar_sync(1, kNW * 32);
    float *sm_o = reinterpret_cast<float *>(stages);  // [kNW][G][D]
    float *sm_m = sm_o + kNW * G * D;
    float *sm_l = sm_m + kNW * G;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        sm_o[(warp * G + 2 * t) * D + 16 * mt + g] = o[mt][0];
        sm_o[(warp * G + 2 * t + 1) * D + 16 * mt + g] = o[mt][1];
        sm_o[(warp * G + 2 * t) * D + 16 * mt + g + 8] = o[mt][2];
        sm_o[(warp * G + 2 * t + 1) * D + 16 * mt + g + 8] = o[mt][3];
    }
    if (g == 0) {
        sm_m[warp * G + 2 * t] = m_run[0];
        sm_m[warp * G + 2 * t + 1] = m_run[1];
        sm_l[warp * G + 2 * t] = l_run[0];
        sm_l[warp * G + 2 * t + 1] = l_run[1];
    }
    named_bar_sync(1, kNW * 32);

    float *mw = sm_l + kNW * G;  // merge weights, then a flag (still in the ring)
    finish_partition<G, D>(p, sm_o, sm_m, sm_l, b, h, split, nsplit, pre, tid, mw,
                           reinterpret_cast<int *>(mw + G * kFuseMaxSplits), false);
    overlap_exit(p);
}

// One piece of a balanced schedule: blocks [blk0, blk0 + nloc) of kv head h
// of sequence b, partial result `split` of the pair's nsplit.  run == 0:
// nothing to attend or write (the same for every thread of the CTA).
struct TcPiece {
    long long L;  // tokens of sequence b (clamped to what may be read)
    int b, h, split, nsplit, blk0, nloc, nblk;
    int run;
};

// Reads and checks piece pc of the schedule against the device lengths.  Only
// the thread with report set records device errors.
KV_DEVICE TcPiece tc_piece(const DecodeKParams &p, int pc, bool report) {
    TcPiece w{};
    const int4 d = __ldg(p.sched_pieces + pc);
    w.b = d.x;
    w.h = d.y & 0xffff;
    w.split = (int)((unsigned)d.y >> 16);
    w.blk0 = d.z;
    w.nloc = d.w & 0xffff;
    w.nsplit = (int)((unsigned)d.w >> 16);
    if (w.b < 0 || w.b >= p.batch || w.h >= p.num_kv_heads || w.nsplit < 1 ||
        w.split >= w.nsplit || w.nsplit > p.max_splits || w.blk0 < 0 || w.nloc > p.part_blocks) {
        if (report) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
        return w;
    }
    long long L = p.seq_lens[w.b];
    if (L > (long long)p.max_blocks * kBS) {
        if (report && w.split == 0 && w.h == 0) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
        L = (long long)p.max_blocks * kBS;
    }
    if (L < 0) L = 0;
    w.nblk = (int)((L + kBS - 1) / kBS);
    // The schedule was made from host copies of the lengths: a piece past the
    // end, or a last piece that stops short of it, means they differ.
    const long long end = (long long)w.blk0 + w.nloc;
    if (end > w.nblk || (w.split == w.nsplit - 1 && end != w.nblk)) {
        if (report) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
        w.nloc = (int)max(0LL, min((long long)w.nloc, (long long)w.nblk - w.blk0));
    }
    w.L = L;
    w.run = 1;
    return w;
}

// decode_tc_kernel's attention on a balanced schedule (kv_decode_schedule):
// CTA c runs the pieces [sched_cta[c], sched_cta[c + 1]), runs of blocks of
// several (sequence, kv head) pairs, one after the other through the same
// ring (ring position and barrier phases continue across pieces).  While the
// consumers finish a piece, the producer reads the next piece and its table
// slice; it refills the ring as soon as the consumers have read their merge
// scratch out of it (named barrier 2), so the split merge of one piece
// overlaps the first copies of the next.  NST ring stages, MINB CTAs per SM.
template <int NST, int MINB, bool TW, bool F16>
__global__ void __launch_bounds__(kDecodeThreads, MINB)
    decode_tc_sched_kernel(const __grid_constant__ CUtensorMap pool_k_map,
                           const __grid_constant__ CUtensorMap pool_v_map, const DecodeKParams p) {
    constexpr int G = 8, D = 128;
    chain_entry(p);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pc0 = __ldg(p.sched_cta + blockIdx.x);
    const int pc1 = __ldg(p.sched_cta + blockIdx.x + 1);
    if (pc0 < 0 || pc1 < pc0 || pc1 > p.sched_npieces) {
        if (tid == 0) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
        return;
    }
    if (pc0 == pc1) return;

    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    char *stages = smem;  // NST x (K tile, V tile), swizzled
    constexpr size_t kRing = decode_ring_bytes<D, G, KV_BF16>(NST);
    static_assert(NST % kNW == 0, "each stage must belong to one consumer warp");
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kRing);
    uint64_t *empty = full + NST;
    int *stage_valid = reinterpret_cast<int *>(empty + NST);
    uint4 *newrow = reinterpret_cast<uint4 *>(stage_valid + NST);  // [32]: fused append's K, V rows
    int32_t *tbl_buf = reinterpret_cast<int32_t *>(newrow + 32);   // [2][part_blocks]
    __shared__ TcPiece s_work[2];                     // this piece and the next one
    __shared__ float s_mw[G * kFuseMaxSplits];        // split-merge weights
    __shared__ int s_flag, s_abort;

    if (warp == kNW) {
        const TcPiece w0 = tc_piece(p, pc0, lane == 0);
        if (lane == 0) {
            s_work[0] = w0;
            s_abort = 0;
            for (int st = 0; st < NST; ++st) {
                mbar_init(&full[st], 1);
                mbar_init(&empty[st], 32);
            }
            mbar_init_fence();
        }
        if (w0.run) {
            const int32_t *row = p.tables + (size_t)w0.b * p.max_blocks + w0.blk0;
            for (int i = lane; i < w0.nloc; i += 32) tbl_buf[i] = __ldg(row + i);
        }
    }
    __syncthreads();

    if (warp == kNW) {
        const CUtensorMap *map_k = &pool_k_map, *map_v = &pool_v_map;
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(map_k) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(map_v) : "memory");
        }
        const uint64_t policy = l2_evict_first_policy();
        int gi = 0;  // tiles issued so far: ring position across pieces
        bool stop = false;
        for (int pc = pc0; pc < pc1; ++pc) {
            const int k = pc - pc0;
            const TcPiece w = s_work[k & 1];
            const int32_t *tbl = tbl_buf + (k & 1) * p.part_blocks;
            if (w.run && !stop) {
                for (int i = 0; i < w.nloc; ++i) {
                    const int st = gi % NST, r = gi / NST;
                    bool bad = false;
                    if (lane == 0) bad = r > 0 && !mbar_wait<TW>(&empty[st], (r - 1) & 1, p.err);
                    if (__shfl_sync(0xffffffffu, bad, 0)) {
                        stop = true;
                        break;
                    }
                    const int id = tbl[i];
                    const bool valid = id >= 0 && id < p.num_blocks;
                    const int y = ((valid ? id : 0) * p.num_kv_heads + w.h) * kBS;
                    char *dst = stages + st * 2 * kTcTile;
                    if (lane == 0) {
                        if (!valid) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
                        stage_valid[st] = valid ? 1 : 0;
                        if (valid)
                            mbar_arrive_expect_tx(&full[st], 2 * kTcTile);
                        else
                            mbar_arrive(&full[st]);
                    }
                    // lane x issues box x: K half 0, K half 1, V half 0, V half 1
                    if (valid && lane < 4)
                        mma::tma2d(dst + (lane >> 1) * kTcTile + (lane & 1) * (kTcTile / 2),
                                   lane < 2 ? map_k : map_v, (lane & 1) * 64, y, &full[st], policy);
                    ++gi;
                }
            }
            if (pc + 1 < pc1) {
                // the next piece and its table slice, read while the consumers
                // finish this one
                const TcPiece nx = tc_piece(p, pc + 1, lane == 0);
                if (lane == 0) {
                    s_work[(k + 1) & 1] = nx;
                    if (stop) s_abort = 1;
                }
                if (nx.run && !stop) {
                    int32_t *t2 = tbl_buf + ((k + 1) & 1) * p.part_blocks;
                    const int32_t *row = p.tables + (size_t)nx.b * p.max_blocks + nx.blk0;
                    for (int i = lane; i < nx.nloc; i += 32) t2[i] = __ldg(row + i);
                }
                named_bar_sync(2, kDecodeThreads);  // the consumers are out of the ring
            }
        }
        if (lane == 0)  // no copy may land after the CTA has exited
            for (int st = 0; st < NST && st < gi; ++st)
                mbar_wait_drain(&full[st], ((gi - 1 - st) / NST) & 1, p.err);
        return;
    }

    // ---- consumer warps: lane = (g = lane / 4, t = lane % 4)
    const int g = lane >> 2, t = lane & 3;
    const uint32_t stage_base = smem_addr(stages);
    int gbase = 0;  // ring position of this piece's first tile
    for (int pc = pc0; pc < pc1; ++pc) {
        const int k = pc - pc0;
        const bool more = pc + 1 < pc1;
        if (!s_work[k & 1].run) {
            if (more) named_bar_sync(2, kDecodeThreads);  // in step with the producer
            continue;
        }
        const int b = s_work[k & 1].b, h = s_work[k & 1].h, nloc = s_work[k & 1].nloc;
        const int blk0 = s_work[k & 1].blk0;
        // tokens from this piece's first block on (at most nloc * 16), and the
        // new token's row in the sequence's last block
        const int rem = (int)(s_work[k & 1].L - (long long)blk0 * kBS);
        const int orow = (int)((s_work[k & 1].L - 1) & (kBS - 1));
        // Fused append: the last piece of (b, h) writes the new token's K/V
        // row (head h) to its pool slot and, since the block holding it may
        // have been copied before that write lands, patches the row into its
        // own copy of the sequence's last block.  Lane x < 16 carries 16-byte
        // chunk x of the K row, lane 16 + x chunk x of the V row.
        const bool fuse = p.new_k != nullptr && s_work[k & 1].split == s_work[k & 1].nsplit - 1;
        const bool patch = fuse && nloc > 0 && blk0 + nloc == s_work[k & 1].nblk;
        if (fuse && warp == (patch ? (gbase + nloc - 1) % kNW : 0)) {
            const size_t src = ((size_t)b * p.num_kv_heads + h) * (D * 2 / 16) + (lane & 15);
            const uint4 v = lane < 16 ? __ldg(p.new_k + src) : __ldg(p.new_v + src);
            newrow[lane] = v;  // kept in shared memory until the last block arrives
            const long long slot = p.new_slots[b];
            if (slot >= 0 && slot < (long long)p.num_blocks * kBS) {
                const long long row = ((slot / kBS) * p.num_kv_heads + h) * kBS + slot % kBS;
                uint4 *dst = reinterpret_cast<uint4 *>(const_cast<char *>(lane < 16 ? p.k_pool : p.v_pool)) +
                             row * (D * 2 / 16) + (lane & 15);
                *dst = v;
            } else if (slot >= 0 && lane == 0) {
                atomicOr(p.err, KV_DEVERR_SLOT_RANGE);
            }
        }
        // Q^T fragments for the 8 k-steps: head g, dims 16kk + 2t (+1) and +8 (+9).
        uint32_t qf[8][2];
        {
            const bool live = g < p.g;
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                reinterpret_cast<const uint16_t *>(p.q) + ((size_t)b * p.num_q_heads + h * p.g + (live ? g : 0)) * D);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                qf[kk][0] = live ? __ldg(qrow + 8 * kk + t) : 0u;
                qf[kk][1] = live ? __ldg(qrow + 8 * kk + 4 + t) : 0u;
            }
        }
        // running state for heads 2t, 2t+1 (replicated over g)
        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
        float o[8][4];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

        if (!s_abort) {
            for (int i = ((warp - gbase) % kNW + kNW) % kNW; i < nloc; i += kNW) {
                const int gi = gbase + i, st = gi % NST, r = gi / NST;
                if (!mbar_wait<TW>(&full[st], r & 1, p.err)) {
                    s_abort = 1;
                    break;
                }
                int ntok = min(kBS, rem - i * kBS);
                if (!stage_valid[st]) ntok = 0;
                const uint32_t kt = stage_base + st * 2 * kTcTile;
                const uint32_t vt = kt + kTcTile;
                if (patch && i == nloc - 1 && ntok > 0) {
                    // the new token is row orow of the sequence's last block
                    const int c = lane & 15;
                    char *tile = stages + st * 2 * kTcTile + (lane < 16 ? 0 : kTcTile);
                    *reinterpret_cast<uint4 *>(tile + (c >> 3) * (kTcTile / 2) + orow * 128 +
                                               (((c & 7) ^ (orow & 7)) << 4)) = newrow[lane];
                    __syncwarp();
                }

                tc_attend_block<F16>(qf, kt, vt, ntok, p.scale_log2, lane, m_run, l_run, o);
                __syncwarp();
                mbar_arrive(&empty[st]);
            }
        }
        gbase += nloc;

        // ---- per-warp totals over the 8 token lanes (g)
#pragma unroll
        for (int x = 4; x <= 16; x <<= 1) {
            l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], x);
            l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], x);
        }
        named_bar_sync(1, kNW * 32);
        float *sm_o = reinterpret_cast<float *>(stages);  // [kNW][G][D]
        float *sm_m = sm_o + kNW * G * D;
        float *sm_l = sm_m + kNW * G;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            sm_o[(warp * G + 2 * t) * D + 16 * mt + g] = o[mt][0];
            sm_o[(warp * G + 2 * t + 1) * D + 16 * mt + g] = o[mt][1];
            sm_o[(warp * G + 2 * t) * D + 16 * mt + g + 8] = o[mt][2];
            sm_o[(warp * G + 2 * t + 1) * D + 16 * mt + g + 8] = o[mt][3];
        }
        if (g == 0) {
            sm_m[warp * G + 2 * t] = m_run[0];
            sm_m[warp * G + 2 * t + 1] = m_run[1];
            sm_l[warp * G + 2 * t] = l_run[0];
            sm_l[warp * G + 2 * t + 1] = l_run[1];
        }
        named_bar_sync(1, kNW * 32);

        // the piece is re-read here: the producer overwrites its slot only
        // after barrier 2, inside finish_partition
        finish_partition<G, D>(p, sm_o, sm_m, sm_l, s_work[k & 1].b, s_work[k & 1].h,
                               s_work[k & 1].split, s_work[k & 1].nsplit, 0, tid, s_mw, &s_flag,
                               more);
    }
}

// The tensor-core decode kernel for a schedule or a grid plan, ring depth
// and addressing; TW: the test instantiation (run-time wait limit); F16:
// half-precision pool.
template <bool TW, bool F16>
static auto tc_decode_fn(bool sched, bool deep, bool linear) {
    return sched ? (deep ? decode_tc_sched_kernel<8, 3, TW, F16> : decode_tc_sched_kernel<4, 5, TW, F16>)
           : deep ? (linear ? decode_tc_kernel<true, 8, 3, TW, F16> : decode_tc_kernel<false, 8, 3, TW, F16>)
                  : (linear ? decode_tc_kernel<true, 4, 5, TW, F16> : decode_tc_kernel<false, 4, 5, TW, F16>);
}

static size_t decode_tc_smem_bytes(bool linear, int part_blocks, int nst, int tables) {
    return 1024 + decode_ring_bytes<128, 8, KV_BF16>(nst) + 2 * nst * sizeof(uint64_t) +
           nst * sizeof(int) + 32 * sizeof(uint4) +
           (size_t)(linear ? 0 : tables * part_blocks) * sizeof(int32_t);
}

// Merges the per-split results of sequences cut into more than one split:
// o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M), lse in the log2 domain.
// One warp per (sequence, query head); lanes cover head_dim.
__global__ void __launch_bounds__(128) merge_kernel(const float *__restrict__ ws_o,
                                                    const float *__restrict__ ws_lse,
                                                    const int32_t *__restrict__ seq_lens,
                                                    const long long *mapped_tokens,
                                                    const int32_t *req_ids, int max_requests,
                                                    int max_len_tokens, int batch,
                                                    int num_q_heads, int head_dim,
                                                    int part_blocks, int max_splits, void *out,
                                                    int out_type, float *lse, int min_splits,
                                                    const int32_t *start_tokens, int part_base) {
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= batch * num_q_heads) return;
    const int b = row / num_q_heads;
    long long L = seq_lens[b];
    if (mapped_tokens) {  // contiguous path: clamp exactly as the decode kernel did
        const int req = req_ids[b];
        L = (req < 0 || req >= max_requests) ? 0 : min(L, mapped_tokens[req]);
    }
    if (L > max_len_tokens) L = max_len_tokens;
    if (L < 0) L = 0;
    const int nblk = (int)((L + kBS - 1) / kBS);
    int sblk = 0;  // as start_block() in the decode kernels
    if (start_tokens) {
        long long st = start_tokens[b];
        st = st < 0 ? 0 : (st > L ? L : st);
        sblk = (int)(st / kBS);
    }
    const int pre = sblk > 0 ? part_base : 0;
    const int nsplit = max(1, (nblk - sblk + part_blocks - 1) / part_blocks);
    const int ntot = pre + nsplit;
    if (ntot < min_splits) return;  // the decode kernel wrote the final result
    auto slot = [&](int s) { return s < pre ? s : part_base + s - pre; };
    const float *ls = ws_lse + (size_t)row * max_splits;
    float M = -INFINITY;
    for (int s = 0; s < ntot; ++s) M = fmaxf(M, ls[slot(s)]);
    float den = 0.f;
    for (int s = 0; s < ntot; ++s) den += M == -INFINITY ? 0.f : exp2f(ls[slot(s)] - M);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int d = lane; d < head_dim; d += 32) {
        float num = 0.f;
        if (M != -INFINITY)
            for (int s = 0; s < ntot; ++s)
                num += exp2f(ls[slot(s)] - M) * ws_o[((size_t)row * max_splits + slot(s)) * head_dim + d];
        const float o = num * inv;
        store_out(out, (size_t)row * head_dim + d, o, out_type);
    }
    if (lse && lane == 0) lse[row] = den > 0.f ? (M + log2f(den)) * 0.6931471805599453f : -INFINITY;
}

void split_plan(int batch, int num_kv_heads, int max_blocks, int num_splits, int *part_blocks,
                int *max_splits) {
    int pb;
    if (max_blocks <= 0) {
        pb = kNW;
    } else if (num_splits > 0) {
        pb = (max_blocks + num_splits - 1) / num_splits;
    } else {
        // Partitions sized so the widest possible tables would give about 12
        // CTAs per SM: real lengths are shorter, and small partitions keep
        // the last wave short.  At least 32 blocks (512 tokens) each.
        const long long work = (long long)batch * num_kv_heads * max_blocks;
        const long long target = 12LL * sm_count();
        pb = (int)((work + target - 1) / target);
        if (pb < 32) pb = 32;
    }
    pb = (pb + kNW - 1) / kNW * kNW;
    if (pb > kMaxPartBlocks) pb = kMaxPartBlocks;
    if (pb < kNW) pb = kNW;
    *part_blocks = pb;
    *max_splits = max_blocks <= 0 ? 1 : (max_blocks + pb - 1) / pb;
}

size_t decode_workspace_bytes(int batch, int num_q_heads, int head_dim, int max_splits) {
    if (max_splits <= 1) return 0;
    return (size_t)batch * num_q_heads * max_splits * (head_dim + 1) * sizeof(float);
}

template <int D, int G, int ET, bool LINEAR>
static size_t decode_smem_bytes(int part_blocks) {
    return decode_ring_bytes<D, G, ET>() + 2 * kNStage * sizeof(uint64_t) + kNStage * sizeof(int) +
           (size_t)kNW * kBS * G * sizeof(float2) + (size_t)kNW * G * sizeof(float) +
           (size_t)(LINEAR ? 0 : part_blocks) * sizeof(int32_t);
}

template <int D, int G, int ET, bool LINEAR>
static kv_status launch_t(const DecodeKParams &kp, dim3 grid, cudaStream_t s) {
    const size_t smem = decode_smem_bytes<D, G, ET, LINEAR>(kp.part_blocks);
    // Large head groups split their heads across the two half-warps (register pressure).
    constexpr int HS = (G >= 8 && D == 128) ? 2 : 1;
    auto fn = decode_kernel<D, G, HS, ET, LINEAR>;
    if (kv_status st0 = cuda_status(
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
        return st0;
    fn<<<grid, kDecodeThreads, smem, s>>>(kp);
    return cuda_status(cudaGetLastError());
}

template <int D, int ET, bool LINEAR>
static kv_status launch_g(int G, const DecodeKParams &kp, dim3 grid, cudaStream_t s) {
    switch (G) {
        case 1: return launch_t<D, 1, ET, LINEAR>(kp, grid, s);
        case 2: return launch_t<D, 2, ET, LINEAR>(kp, grid, s);
        case 4: return launch_t<D, 4, ET, LINEAR>(kp, grid, s);
        case 8: return launch_t<D, 8, ET, LINEAR>(kp, grid, s);
    }
    return KV_ERR_UNSUPPORTED;
}

// The CUDA-core decode for this element type and addressing.
template <int D>
static kv_status launch_cc(kv_dtype dt, bool linear, int G, const DecodeKParams &kp, dim3 grid,
                           cudaStream_t s) {
    if (dt == KV_BF16)
        return linear ? launch_g<D, KV_BF16, true>(G, kp, grid, s) : launch_g<D, KV_BF16, false>(G, kp, grid, s);
    if (dt == KV_F16)
        return linear ? launch_g<D, KV_F16, true>(G, kp, grid, s) : launch_g<D, KV_F16, false>(G, kp, grid, s);
    return linear ? launch_g<D, KV_F32, true>(G, kp, grid, s) : launch_g<D, KV_F32, false>(G, kp, grid, s);
}

kv_status launch_decode(const DecodeArgs &a, bool linear) {
    if (a.batch < 0 || a.num_q_heads <= 0 || a.num_kv_heads <= 0) return KV_ERR_ARG;
    if (a.num_q_heads % a.num_kv_heads) return KV_ERR_ARG;
    const int g = a.num_q_heads / a.num_kv_heads;
    if (g > 8) return KV_ERR_UNSUPPORTED;
    if (a.head_dim != 64 && a.head_dim != 128) return KV_ERR_UNSUPPORTED;
    if (a.out_dtype != KV_F32 && a.out_dtype != a.dtype) return KV_ERR_UNSUPPORTED;
    if (a.batch == 0) return KV_OK;
    if (!a.q || !a.seq_lens || !a.out) return KV_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(a.q) & 15) return KV_ERR_ARG;
    const int G = g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8;
    int pb = 0, ms = 0;
    if (a.sched) {
        pb = a.sched_part_blocks;
        ms = a.sched_max_splits;
        if (a.part_base != 0 || a.start_tokens || a.seq_order) return KV_ERR_ARG;
    } else {
        split_plan(a.batch, a.num_kv_heads, a.max_blocks, a.num_splits, &pb, &ms);
    }
    if (a.part_base < 0 || (a.part_base > 0 && !a.start_tokens)) return KV_ERR_ARG;
    const int slots = a.part_base + ms;  // workspace partial results per (sequence, query head)
    const size_t need = decode_workspace_bytes(a.batch, a.num_q_heads, a.head_dim, slots);
    if (need > 0 && (!a.workspace || a.workspace_bytes < need)) return KV_ERR_ARG;
    if (ms > 65535 || a.batch > 65535 || a.num_kv_heads > 65535) return KV_ERR_UNSUPPORTED;

    DecodeKParams kp{};
    kp.q = a.q;
    kp.k_pool = static_cast<const char *>(a.k_pool);
    kp.v_pool = static_cast<const char *>(a.v_pool);
    kp.tables = a.block_tables;
    kp.max_blocks = a.max_blocks;
    kp.num_blocks = a.num_blocks;
    kp.k_bases = a.k_bases;
    kp.v_bases = a.v_bases;
    kp.req_ids = a.req_ids;
    kp.mapped_tokens = a.mapped_tokens;
    kp.head_stride = a.head_stride;
    kp.max_requests = a.max_requests;
    kp.seq_lens = a.seq_lens;
    kp.num_q_heads = a.num_q_heads;
    kp.num_kv_heads = a.num_kv_heads;
    kp.g = g;
    kp.scale_log2 = a.scale * 1.4426950408889634f;
    kp.part_blocks = pb;
    kp.max_splits = slots;
    kp.start_tokens = a.start_tokens;
    kp.part_base = a.part_base;
    kp.new_k = static_cast<const uint4 *>(a.new_k);
    kp.new_v = static_cast<const uint4 *>(a.new_v);
    kp.new_slots = a.new_slots;
    kp.seq_order = a.seq_order;
    kp.batch = a.batch;
    kp.overlap = a.overlap_previous ? 1 : 0;
    kp.chain = a.chain && !a.overlap_previous ? 1 : 0;
    if (a.sched) {
        kp.sched_cta = a.sched + kSchedHeader;
        kp.sched_pieces = reinterpret_cast<const int4 *>(a.sched + sched_piece_off(a.sched_ctas));
        kp.sched_npieces = a.sched_pieces;
    }
    kp.out = a.out;
    kp.out_type = a.out_dtype;
    kp.lse = a.lse;
    kp.ws_o = static_cast<float *>(a.workspace);
    kp.ws_lse = need > 0 ? kp.ws_o + (size_t)a.batch * a.num_q_heads * slots * a.head_dim : nullptr;
    kp.err = a.err;

    kp.req_maps = a.req_maps;
    kp.counters = (a.counters && (long long)a.batch * a.num_kv_heads <= a.counter_slots) ? a.counters
                                                                                       : nullptr;
    const dim3 grid = a.sched ? dim3(a.sched_ctas, 1, 1) : dim3(ms, a.num_kv_heads, a.batch);
    kv_status st;
    // Large head groups on 16-bit storage (bf16 or fp16) with d128 go to the
    // tensor-core variant when the tiled-TMA maps of the K/V storage are
    // available.
    const bool use_tc = a.dtype != KV_F32 && a.head_dim == 128 && g >= kTcMinGroup &&
                        (linear ? a.req_maps != nullptr : a.pool_map_k != nullptr);
    if (a.new_k && !use_tc) return KV_ERR_UNSUPPORTED;  // fused append: tensor-core kernels only
    // a schedule: paged tensor-core path, every merge inside the kernel
    if (a.sched && (!use_tc || linear || (slots > 1 && !kp.counters))) return KV_ERR_UNSUPPORTED;
    // an overlapping launch: the grid-indexed tensor-core kernel, merges inside it
    if (a.overlap_previous && (!use_tc || a.sched || (slots > kFuseMaxSplits) ||
                               (slots > 1 && !kp.counters))) {
        kp.overlap = 0;
        DecodeArgs b2 = a;
        b2.overlap_previous = false;
        return launch_decode(b2, linear);
    }
    if (use_tc) {
        // Long partitions: a deep ring (8 stages) and 3 CTAs per SM; short
        // ones: more CTAs at once (5 per SM) with 4 stages each.  Sweeps on
        // GB300 (Llama-3-8B shape, 129-block partitions: 5959 vs 5502 GB/s;
        // Yi-6B shape, 384-512-block partitions: 6288 vs 5965 GB/s).
        const bool deep = a.sched ? a.sched_deep != 0 : pb >= kTcDeepBlocks;
        const int nst = deep ? 8 : 4;
        const size_t smem = decode_tc_smem_bytes(linear, pb, nst, a.sched ? 2 : 1);
        CUtensorMap dummy{};
        const CUtensorMap &mk = linear ? dummy : *a.pool_map_k;
        const CUtensorMap &mv = linear ? dummy : *a.pool_map_v;
        const bool sched = a.sched != nullptr, f16 = a.dtype == KV_F16;
        auto fn = test_waits_enabled()
                      ? (f16 ? tc_decode_fn<true, true>(sched, deep, linear)
                             : tc_decode_fn<true, false>(sched, deep, linear))
                      : (f16 ? tc_decode_fn<false, true>(sched, deep, linear)
                             : tc_decode_fn<false, false>(sched, deep, linear));
        if (kv_status st0 = cuda_status(
                cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
            return st0;
        if (a.overlap_previous || kp.chain) {
            // may start while the previous kernel in the stream still runs
            cudaLaunchConfig_t cfg{};
            cfg.gridDim = grid;
            cfg.blockDim = dim3(kDecodeThreads);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = a.stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            st = cuda_status(cudaLaunchKernelEx(&cfg, fn, mk, mv, kp));
        } else {
            fn<<<grid, kDecodeThreads, smem, a.stream>>>(mk, mv, kp);
            st = cuda_status(cudaGetLastError());
        }
    } else if (a.head_dim == 128) {
        st = launch_cc<128>(a.dtype, linear, G, kp, grid, a.stream);
    } else {
        st = launch_cc<64>(a.dtype, linear, G, kp, grid, a.stream);
    }
    if (st != KV_OK || slots <= 1 || a.sched) return st;  // schedules merge inside the kernel
    const int min_splits = kp.counters ? kFuseMaxSplits + 1 : 2;
    if (slots < min_splits) return st;  // every merge happens inside the decode kernel
    const int rows = a.batch * a.num_q_heads;
    merge_kernel<<<(rows + 3) / 4, 128, 0, a.stream>>>(
        kp.ws_o, kp.ws_lse, a.seq_lens, linear ? a.mapped_tokens : nullptr, a.req_ids,
        a.max_requests, a.max_blocks * kBS, a.batch, a.num_q_heads, a.head_dim, pb, slots, a.out,
        kp.out_type, a.lse, min_splits, a.start_tokens, a.part_base);
    return cuda_status(cudaGetLastError());
}

}  // namespace pkv

using namespace pkv;

extern "C" {

kv_status kv_decode_split_plan(int batch, int num_kv_heads, int max_blocks, int num_splits,
                               int *part_blocks, int *max_splits) {
    if (!part_blocks || !max_splits || batch < 0 || num_kv_heads <= 0 || max_blocks < 0)
        return KV_ERR_ARG;
    split_plan(batch, num_kv_heads, max_blocks, num_splits, part_blocks, max_splits);
    return KV_OK;
}

kv_status kv_decode_order(const int32_t *host_seq_lens, int batch, int32_t *order_out) {
    if (batch < 0 || (batch > 0 && (!host_seq_lens || !order_out))) return KV_ERR_ARG;
    std::vector<int32_t> idx(batch);
    for (int b = 0; b < batch; ++b) idx[b] = b;
    std::stable_sort(idx.begin(), idx.end(),
                     [&](int32_t x, int32_t y) { return host_seq_lens[x] > host_seq_lens[y]; });
    for (int b = 0; b < batch; ++b) order_out[b] = idx[b];
    return KV_OK;
}

kv_status kv_decode_plan(const int32_t *host_seq_lens, int batch, int num_kv_heads,
                         int max_blocks, int *num_splits) {
    if (!num_splits || batch < 0 || num_kv_heads <= 0 || max_blocks < 0 ||
        (batch > 0 && !host_seq_lens))
        return KV_ERR_ARG;
    if (batch == 0 || max_blocks == 0) {
        *num_splits = 1;
        return KV_OK;
    }
    // The tensor-core decode runs long partitions (>= kTcDeepBlocks blocks)
    // with a deep ring at three CTAs per SM and shorter ones at five CTAs per
    // SM.  A deep-ring wave streams fastest at about two to two and a half
    // CTAs per SM (sweeps of the Yi-6B-shaped workload on GB300: 2.0-2.3 per
    // SM reach ~0.95 of the copy bandwidth, 2.7-3.0 per SM drop to ~0.65); the
    // five-per-SM kernel is best with a full single wave (Llama-3-8B shape:
    // 760 CTAs on 152 SMs, 0.89).  The CUDA-core decode keeps three per SM.
    const int sm = sm_count();
    auto deep = [&](int pb) { return pb >= kTcDeepBlocks; };
    auto one_wave = [&](int pb) { return deep(pb) ? (long long)(2.4 * sm) : 5LL * sm; };
    auto resident = [&](int pb) { return deep(pb) ? 3LL * sm : 5LL * sm; };
    std::vector<int> nblk(batch);
    int longest = 1;
    for (int b = 0; b < batch; ++b) {
        long long L = host_seq_lens[b];
        if (L < 0) L = 0;
        if (L > (long long)max_blocks * kBS) L = (long long)max_blocks * kBS;
        nblk[b] = (int)((L + kBS - 1) / kBS);
        if (nblk[b] > longest) longest = nblk[b];
    }
    auto ctas = [&](int pb) {
        long long n = 0;
        for (int b = 0; b < batch; ++b) n += nblk[b] > pb ? (nblk[b] + pb - 1) / pb : 1;
        return n * num_kv_heads;
    };
    // The partition size a given split count turns into inside the kernel.
    auto plan_pb = [&](int splits) {
        int pb, ms;
        split_plan(batch, num_kv_heads, max_blocks, splits, &pb, &ms);
        return pb;
    };
    // 1) One wave if it fits (every CTA streams at the same time, none waits
    //    for a slot): the smallest deep-ring partitions that fit, else the
    //    smallest short partitions that fit.
    // 2) Otherwise the largest partitions that still give several full waves
    //    (three deep, two short), so the last, partly filled wave is a small
    //    share of the time.
    int best_deep = 0, best_wide = 0;
    for (int s = 1; s <= 4096; ++s) {
        const int pb = plan_pb(s);
        if (ctas(pb) <= one_wave(pb)) (deep(pb) ? best_deep : best_wide) = s;
        if (pb <= kNW) break;
    }
    int best = best_deep ? best_deep : best_wide;
    if (best == 0) {
        best = 1;
        for (int s = 1; s <= 4096; ++s) {
            const int pb = plan_pb(s);
            best = s;
            if (ctas(pb) >= (deep(pb) ? 3 : 2) * resident(pb) || pb <= 32) break;
        }
    }
    *num_splits = best;
    return KV_OK;
}

// ---- balanced schedule ------------------------------------------------------
// One wave of CTAs that all stream the same number of blocks.  The blocks of
// every (sequence, kv head) pair are laid end to end (sequence-major, heads
// inside) and cut into C equal runs; a run that crosses pairs becomes several
// pieces.  A pair's pieces are its split-KV partitions, merged by the last CTA
// to finish one of them.
static int sched_sms(int num_sms) { return num_sms > 0 ? num_sms : sm_count(); }

kv_status kv_decode_schedule_capacity(int batch, int num_kv_heads, int max_blocks, int num_sms,
                                      size_t *ints) {
    if (!ints || batch < 0 || num_kv_heads <= 0 || max_blocks < 0 || num_sms < 0)
        return KV_ERR_ARG;
    const long long total = (long long)batch * num_kv_heads * max_blocks;
    long long c = 5LL * sched_sms(num_sms);
    const long long c_long = (total + kMaxPartBlocks - 1) / kMaxPartBlocks;
    if (c_long > c) c = c_long;
    c += (long long)batch * num_kv_heads;  // whole pieces: up to one more CTA per pair
    if (c > (1LL << 30)) return KV_ERR_UNSUPPORTED;
    *ints = sched_piece_off((int)c) + 4 * (size_t)(c + (long long)batch * num_kv_heads);
    return KV_OK;
}

kv_status kv_decode_schedule(const int32_t *host_seq_lens, int batch, int num_kv_heads,
                             int max_blocks, int num_sms, int num_ctas, int ring_stages, int flags,
                             int32_t *schedule_out, size_t capacity_ints, size_t *used_ints) {
    if (!schedule_out || batch < 0 || num_kv_heads <= 0 || max_blocks < 0 || num_sms < 0 ||
        num_ctas < 0 || (ring_stages != 0 && ring_stages != 4 && ring_stages != 8) ||
        (flags & ~KV_SCHED_WHOLE_PIECES) || (batch > 0 && !host_seq_lens))
        return KV_ERR_ARG;
    if (num_kv_heads > 0xffff) return KV_ERR_UNSUPPORTED;
    const int sms = sched_sms(num_sms);
    std::vector<int> nb(batch);
    long long T = 0;
    int nbmax = 0;
    for (int b = 0; b < batch; ++b) {
        long long L = host_seq_lens[b];
        if (L < 0) L = 0;
        if (L > (long long)max_blocks * kBS) L = (long long)max_blocks * kBS;
        nb[b] = (int)((L + kBS - 1) / kBS);
        T += (long long)nb[b] * num_kv_heads;
        if (nb[b] > nbmax) nbmax = nb[b];
    }
    // One wave: the deep ring (at most 2.4 CTAs per SM, the rate the
    // grid-indexed plan found best) when every CTA gets at least
    // kTcDeepBlocks blocks, else the wide kernel at five CTAs per SM.
    const long long c_deep = (12LL * sms) / 5, c_wide = 5LL * sms;
    long long W;
    if (num_ctas > 0) {  // the caller's CTA count
        if (num_ctas > (ring_stages == 8 ? 3 : 5) * sms) return KV_ERR_ARG;  // one wave
        W = (T + num_ctas - 1) / num_ctas;
    } else if (ring_stages == 8) {
        W = (T + c_deep - 1) / c_deep;
    } else if (ring_stages == 4) {
        W = (T + c_wide - 1) / c_wide;
    } else {
        W = (T + c_deep - 1) / c_deep;
        if (W < kTcDeepBlocks) W = (T + c_wide - 1) / c_wide;
    }
    // A pair of n blocks spans at most ceil(n / W) + 1 runs; keep that within
    // the merge done inside the kernel.
    const long long w_pairs = (nbmax + kFuseMaxSplits - 2) / (kFuseMaxSplits - 1);
    if (W < w_pairs) W = w_pairs;
    if (W < 1) W = 1;
    if (W > kMaxPartBlocks) W = kMaxPartBlocks;
    if ((nbmax + W - 1) / W + 1 > kFuseMaxSplits) return KV_ERR_UNSUPPORTED;
    const long long C = T > 0 ? (T + W - 1) / W : 1;
    if (C > (1LL << 30)) return KV_ERR_UNSUPPORTED;
    const size_t need = sched_piece_off((int)C) + 4 * (size_t)(C + (long long)batch * num_kv_heads);
    if (used_ints) *used_ints = need;
    if (capacity_ints < need) return KV_ERR_ARG;

    if (flags & KV_SCHED_WHOLE_PIECES) {
        // Each pair cut into ceil(n / W) pieces of near-equal length, one CTA
        // per piece, CTAs ordered longest piece first: the in-order dispatch
        // of the grid then does longest-first list scheduling over slightly
        // more than one wave, and no CTA streams more than one piece.
        struct Pc { int b, h, split, ns, blk0, n; };
        std::vector<Pc> all;
        int most_w = 1, longest = 1;
        for (int b = 0; b < batch; ++b) {
            const int n = nb[b];
            const int ns = n == 0 ? 1 : (int)((n + W - 1) / W);
            if (ns > most_w) most_w = ns;
            for (int h = 0; h < num_kv_heads; ++h) {
                int blk0 = 0;
                for (int sp = 0; sp < ns; ++sp) {
                    const int len = n / ns + (sp < n % ns ? 1 : 0);
                    all.push_back({b, h, sp, ns, blk0, len});
                    if (len > longest) longest = len;
                    blk0 += len;
                }
            }
        }
        if (most_w > kFuseMaxSplits) return KV_ERR_UNSUPPORTED;
        std::stable_sort(all.begin(), all.end(), [](const Pc &x, const Pc &y) { return x.n > y.n; });
        const long long Cw = std::max<long long>(1, (long long)all.size());
        const size_t need_w = sched_piece_off((int)Cw) + 4 * (size_t)all.size();
        if (used_ints) *used_ints = need_w;
        if (capacity_ints < need_w) return KV_ERR_ARG;
        int32_t *cta_w = schedule_out + kSchedHeader;
        int32_t *pcs_w = schedule_out + sched_piece_off((int)Cw);
        for (long long c = 0; c <= Cw; ++c) cta_w[c] = (int32_t)std::min<long long>(c, all.size());
        for (size_t i = 0; i < all.size(); ++i) {
            int32_t *q = pcs_w + 4 * i;
            q[0] = all[i].b;
            q[1] = all[i].h | (all[i].split << 16);
            q[2] = all[i].blk0;
            q[3] = all[i].n | (all[i].ns << 16);
        }
        const int deep_w = ring_stages ? (ring_stages == 8 ? 1 : 0) : (W >= kTcDeepBlocks ? 1 : 0);
        schedule_out[0] = (int32_t)Cw;
        schedule_out[1] = (int32_t)all.size();
        schedule_out[2] = most_w;
        schedule_out[3] = longest;
        schedule_out[4] = deep_w;
        schedule_out[5] = batch;
        schedule_out[6] = num_kv_heads;
        schedule_out[7] = most_w;
        return KV_OK;
    }
    int32_t *cta = schedule_out + kSchedHeader;
    int32_t *pcs = schedule_out + sched_piece_off((int)C);
    long long pos = 0, next_cta = 0;
    int np = 0, most = 1;
    auto open_to = [&](long long c) {  // CTAs up to c start at the next piece
        while (next_cta <= c) cta[next_cta++] = np;
    };
    auto emit = [&](int b, int h, long long blk0, long long n, long long split, long long ns) {
        int32_t *q = pcs + 4 * (size_t)np++;
        q[0] = b;
        q[1] = h | (int32_t)(split << 16);
        q[2] = (int32_t)blk0;
        q[3] = (int32_t)n | (int32_t)(ns << 16);
    };
    for (int b = 0; b < batch; ++b) {
        for (int h = 0; h < num_kv_heads; ++h) {
            const long long n = nb[b];
            if (n == 0) {  // an empty pair still writes out = 0, lse = -inf
                open_to(std::min(pos / W, C - 1));
                emit(b, h, 0, 0, 0, 1);
                continue;
            }
            const long long s0 = pos / W, s1 = (pos + n - 1) / W, ns = s1 - s0 + 1;
            if (ns > most) most = (int)ns;
            for (long long c = s0; c <= s1; ++c) {
                const long long lo = std::max(pos, c * W), hi = std::min(pos + n, (c + 1) * W);
                open_to(c);
                emit(b, h, lo - pos, hi - lo, c - s0, ns);
            }
            pos += n;
        }
    }
    open_to(C);  // CTAs without pieces of their own, then the end marker
    schedule_out[0] = (int32_t)C;
    schedule_out[1] = np;
    schedule_out[2] = most;
    schedule_out[3] = (int32_t)W;
    const int deep = ring_stages ? (ring_stages == 8 ? 1 : 0) : (W >= kTcDeepBlocks ? 1 : 0);
    schedule_out[4] = deep;
    schedule_out[5] = batch;
    schedule_out[6] = num_kv_heads;
    schedule_out[7] = most;  // partial results per (sequence, query head)
    if (used_ints) *used_ints = sched_piece_off((int)C) + 4 * (size_t)np;
    return KV_OK;
}

kv_status kv_decode_schedule_workspace_size(const int32_t *host_schedule, int num_q_heads,
                                            int head_dim, size_t *bytes) {
    if (!host_schedule || !bytes || num_q_heads <= 0 || head_dim <= 0 || host_schedule[5] < 0 ||
        host_schedule[7] < 1)
        return KV_ERR_ARG;
    *bytes = decode_workspace_bytes(host_schedule[5], num_q_heads, head_dim, host_schedule[7]);
    return KV_OK;
}

kv_status kv_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                   int max_blocks, int num_splits, size_t *bytes) {
    if (!bytes || batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks < 0)
        return KV_ERR_ARG;
    int pb, ms;
    split_plan(batch, num_kv_heads, max_blocks, num_splits, &pb, &ms);
    *bytes = decode_workspace_bytes(batch, num_q_heads, head_dim, ms);
    return KV_OK;
}

kv_status paged_decode_attention(kv_pool_t p, const void *q, const int32_t *block_tables,
                                 int max_blocks, const int32_t *seq_lens, int batch,
                                 int num_q_heads, float scale, void *out, kv_dtype out_dtype,
                                 float *lse_out, int num_splits, void *workspace,
                                 size_t workspace_bytes, void *stream) {
    if (!p || max_blocks < 0 || (batch > 0 && max_blocks > 0 && !block_tables)) return KV_ERR_ARG;
    DecodeArgs a{};
    if (kv_status st = require_device(p->device)) return st;
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
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.err = p->err;
    a.chain = p->launch_overlap;
    a.counters = p->counters;
    a.counter_slots = kv_pool::kCounterSlots;
    a.stream = as_stream(stream);
    if (p->dtype != KV_F32 && p->head_dim == 128 && pool_tensor_maps(p) == KV_OK) {
        a.pool_map_k = &p->tmap_k;
        a.pool_map_v = &p->tmap_v;
    }
    return launch_decode(a, false);
}

kv_status paged_append_and_decode(kv_pool_t p, const void *q, const void *k_new,
                                  const void *v_new, const int64_t *slot_mapping,
                                  const int32_t *block_tables, int max_blocks,
                                  const int32_t *seq_lens, const int32_t *seq_order, int batch,
                                  int num_q_heads, float scale,
                                  void *out, kv_dtype out_dtype, float *lse_out, int num_splits,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    if (!p || batch < 0 || max_blocks < 0 || (batch > 0 && max_blocks > 0 && !block_tables))
        return KV_ERR_ARG;
    if (batch == 0) return KV_OK;
    if (!k_new || !v_new || !slot_mapping) return KV_ERR_ARG;
    if (kv_status st = require_device(p->device)) return st;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15) return KV_ERR_ARG;
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
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.err = p->err;
    a.chain = p->launch_overlap;
    a.counters = p->counters;
    a.counter_slots = kv_pool::kCounterSlots;
    a.stream = as_stream(stream);
    if (p->dtype != KV_F32 && p->head_dim == 128 && pool_tensor_maps(p) == KV_OK) {
        a.pool_map_k = &p->tmap_k;
        a.pool_map_v = &p->tmap_v;
    }
    a.new_k = k_new;
    a.new_v = v_new;
    a.new_slots = slot_mapping;
    a.seq_order = seq_order;
    const kv_status st = launch_decode(a, false);
    if (st != KV_ERR_UNSUPPORTED) return st;
    // shapes the fused kernel does not cover: the append, then the decode
    if (kv_status st1 = kv_append(p, k_new, v_new, slot_mapping, batch, stream)) return st1;
    a.new_k = a.new_v = nullptr;
    a.new_slots = nullptr;
    return launch_decode(a, false);
}

kv_status paged_decode_attention_scheduled(kv_pool_t p, const void *q, const void *k_new,
                                           const void *v_new, const int64_t *slot_mapping,
                                           const int32_t *block_tables, int max_blocks,
                                           const int32_t *seq_lens, int batch, int num_q_heads,
                                           float scale, const int32_t *host_schedule,
                                           const int32_t *schedule, void *out, kv_dtype out_dtype,
                                           float *lse_out, void *workspace,
                                           size_t workspace_bytes, void *stream) {
    if (!p || batch < 0 || max_blocks < 0 || !host_schedule || !schedule ||
        (batch > 0 && max_blocks > 0 && !block_tables))
        return KV_ERR_ARG;
    if (kv_status st = require_device(p->device)) return st;
    if (batch == 0) return KV_OK;
    const int32_t *hs = host_schedule;
    if (hs[0] < 1 || hs[1] < 0 || hs[2] < 1 || hs[2] > kFuseMaxSplits || hs[3] < 1 ||
        hs[3] > kMaxPartBlocks || (hs[4] != 0 && hs[4] != 1) || hs[5] != batch ||
        hs[6] != p->num_kv_heads || hs[7] != hs[2])
        return KV_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(schedule) & 15) return KV_ERR_ARG;
    if (k_new && (!v_new || !slot_mapping)) return KV_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
        return KV_ERR_ARG;
    if (p->dtype == KV_F32 || p->head_dim != 128) return KV_ERR_UNSUPPORTED;
    if (kv_status st = pool_tensor_maps(p)) return st;
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
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.err = p->err;
    a.chain = p->launch_overlap;
    a.counters = p->counters;
    a.counter_slots = kv_pool::kCounterSlots;
    a.stream = as_stream(stream);
    a.pool_map_k = &p->tmap_k;
    a.pool_map_v = &p->tmap_v;
    a.new_k = k_new;
    a.new_v = v_new;
    a.new_slots = k_new ? slot_mapping : nullptr;
    a.sched = schedule;
    a.sched_ctas = hs[0];
    a.sched_pieces = hs[1];
    a.sched_max_splits = hs[7];
    a.sched_part_blocks = hs[3];
    a.sched_deep = hs[4];
    return launch_decode(a, false);
}

}  // extern "C"

namespace pkv {
cudaError_t set_wait_limit_decode(unsigned long long ns) { return set_wait_limit_here(ns); }
}  // namespace pkv

// ---------------------------------------------------------------------------
// Decode without caller-provided scratch.
//
// Some callers cannot allocate device memory at the point where they run
// decode: a plugin inside a host framework that owns all device memory, or a
// serving loop that must not call cudaMalloc after start-up (it can
// synchronise the device and stall other streams).  For them the split-KV
// partial results go to one fixed array that lives in the library's device
// image instead of a caller-supplied workspace.
//
// The array is kStaticScratchBytes (8 MiB) per device and stays resident on
// every GPU that loads the library until the process exits.  In host code
// the array's name is only a host-side stand-in; its device address is looked
// up once per device with cudaGetSymbolAddress (with that device current) on
// the first call, so that first call should come before any stream capture.
// Every call shares the array: calls that overlap on the GPU (different
// streams without ordering) race on it.  Nothing in it needs to start at zero:
// each split writes its partial result before the merge reads it.
// ---------------------------------------------------------------------------
namespace pkv {
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
constexpr int kStaticMaxDevices = 64;
static __device__ __align__(256) float g_decode_scratch[kStaticScratchBytes / sizeof(float)];

// The scratch address on `dev`, which must be the current device (the
// caller checks that it is the pool's).
static kv_status static_scratch(int dev, void **ptr) {
    static std::mutex mu;
    static void *addr[kStaticMaxDevices] = {};
    if (dev < 0 || dev >= kStaticMaxDevices) return KV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return KV_ERR_CUDA;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return KV_OK;
}
}  // namespace pkv

extern "C" {

kv_status paged_decode_attention_noalloc(kv_pool_t p, const void *q, const int32_t *block_tables,
                                         int max_blocks, const int32_t *seq_lens, int batch,
                                         int num_q_heads, float scale, void *out,
                                         kv_dtype out_dtype, float *lse_out, int num_splits,
                                         void *stream) {
    if (!p || batch < 0 || num_q_heads <= 0 || max_blocks < 0) return KV_ERR_ARG;
    if (kv_status st = require_device(p->device)) return st;
    int pb = 0, ms = 0;
    split_plan(batch, p->num_kv_heads, max_blocks, num_splits, &pb, &ms);
    const size_t need = decode_workspace_bytes(batch, num_q_heads, p->head_dim, ms);
    if (need > kStaticScratchBytes) return KV_ERR_UNSUPPORTED;  // beyond the fixed scratch array
    void *ws = nullptr;
    if (need > 0) {
        const kv_status st = static_scratch(p->device, &ws);
        if (st != KV_OK) return st;
    }
    return paged_decode_attention(p, q, block_tables, max_blocks, seq_lens, batch, num_q_heads,
                                  scale, out, out_dtype, lse_out, num_splits, ws,
                                  need > 0 ? kStaticScratchBytes : 0, stream);
}

}  // extern "C"
