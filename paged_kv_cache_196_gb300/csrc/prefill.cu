// Chunked causal paged prefill (tcgen05 tensor cores).  Placeholder entry
// point until the kernel lands.
#include "internal.h"

extern "C" kv_status paged_prefill_attention(kv_pool_t p, const void *q, const int32_t *cu_q,
                                             int max_q_len, const int32_t *block_tables,
                                             int max_blocks, const int32_t *seq_lens, int batch,
                                             int num_q_heads, float scale, void *out,
                                             kv_dtype out_dtype, float *lse_out, void *stream) {
    (void)p; (void)q; (void)cu_q; (void)max_q_len; (void)block_tables; (void)max_blocks;
    (void)seq_lens; (void)batch; (void)num_q_heads; (void)scale; (void)out; (void)out_dtype;
    (void)lse_out; (void)stream;
    return KV_ERR_UNSUPPORTED;
}
