// A8 kv_b_proj expansion and A9 prefill attention (chunked-prefill context
// step).  Source: "DeepSeek MLA 在 DCP 分布式环境中的 Prefill 阶段解析",
// §MLA Prefill vs Decode and §Chunked Prefill 与 LSE Merge.
#include "common.cuh"

extern "C" int mla_expand_kv(const void *kv_rows, const void *w_kvb, int N,
                             int H, void *k_out, void *v_out,
                             mla_stream_t stream) {
  (void)kv_rows; (void)w_kvb; (void)N; (void)H; (void)k_out; (void)v_out;
  (void)stream;
  return MLA_ERR_UNSUPPORTED;
}

extern "C" int mla_prefill_attn(const void *q, const void *k, const void *v,
                                const int32_t *cu_q, const int32_t *cu_k,
                                int B, int Tq, int Nk, int H, int max_q_len,
                                int causal, float sm_scale, void *out,
                                float *lse, mla_stream_t stream) {
  (void)q; (void)k; (void)v; (void)cu_q; (void)cu_k; (void)B; (void)Tq;
  (void)Nk; (void)H; (void)max_q_len; (void)causal; (void)sm_scale;
  (void)out; (void)lse; (void)stream;
  return MLA_ERR_UNSUPPORTED;
}
