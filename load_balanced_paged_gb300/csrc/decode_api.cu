// The C entry points of the decode kernels (include/dsa.h): argument checks, the kernel
// parameters of each call, and the choice of kernel -- the one-token persistent kernel (also
// with the early KV gather, or with the combine folded in), the static split-KV grid, the
// mma.sync E4M3 multi-token kernel (attention.cu) or the tensor-memory multi-token kernel
// (attention_tc.cu).  Host code only.
#include "engine.cuh"

using namespace dsa;

extern "C" int32_t dsa_multi_slots_per_desc(int32_t q_len, int32_t group) {
    if (q_len < 1 || group < 1) return -1;
    return q_len > 1 ? 2 : 1;
}

namespace {

// dsa_decode_ex, and dsa_decode_chained when new_tokens >= 0 (early KV gather, one query token).
dsa_status decode_impl(int32_t q_len, int32_t kv_layout, const void *q, dsa_dtype q_dtype, const float *q_scale,
                       const void *k_pages, const void *v_pages, dsa_dtype kv_dtype, const float *k_scale,
                       const float *v_scale, const int32_t *block_table, int32_t max_pages_per_req,
                       int32_t num_pages, const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, int32_t page_size, float sm_scale,
                       const dsa_task_map *map, float *partial_o, float *partial_lse, uint64_t *cta_times,
                       int32_t new_tokens, dsa_stream stream) {
    const AttnArgs a{q, q_dtype, q_scale, k_pages, v_pages, kv_dtype, k_scale, v_scale, block_table,
                     max_pages_per_req, num_pages, seq_lens, batch, num_q_heads, num_kv_heads, head_dim,
                     page_size, sm_scale, kv_layout};
    dsa_status s = validate_attn(a);
    if (s != DSA_OK) return s;
    if (q_len < 1) return DSA_ERR_INVALID_ARG;
    const int R = q_len * (num_q_heads / num_kv_heads);
    if (q_len > 1 && R > kMaxRows) return DSA_ERR_UNSUPPORTED;
    if (!map || !map->cta_desc_begin || !map->descs || !map->meta || !partial_o || !partial_lse)
        return DSA_ERR_INVALID_ARG;
    if (map->num_units != batch * num_kv_heads || map->num_ctas < 1) return DSA_ERR_INVALID_ARG;
    if (!aligned16(partial_o) || !aligned16(map->descs)) return DSA_ERR_INVALID_ARG;
    if (batch == 0) return DSA_OK;
    KernelParams kp = base_params(a, partial_o, partial_lse, map->meta + 3);
    kp.max_slots = map->max_descs;
    kp.cta_desc_begin = map->cta_desc_begin;
    kp.descs = reinterpret_cast<const int4 *>(map->descs);
    kp.cta_times = cta_times;
    if (new_tokens >= 0) {
        kp.early = 1;
        kp.new_tokens = new_tokens;
    }
    if (q_len == 1) {
        return launch_decode(a, kp, map->num_ctas, false, to_cuda(stream));
    }
    kp.q_len = q_len;
    kp.slots_per_desc = dsa_multi_slots_per_desc(q_len, num_q_heads / num_kv_heads);
    // E4M3 K/V: up to 16 rows mma.sync warps (the groups take alternate tiles, 16 tokens x all
    // rows per warp), more rows the tensor-memory kernel
    if (kv_dtype == DSA_FP8_E4M3) {
        if (R <= 16) return launch_multi_mma(a, kp, map->num_ctas, to_cuda(stream));
        return launch_tc(a, kp, map->num_ctas, to_cuda(stream));
    }
    // bf16 K/V: the tensor-memory kernel, for any number of query rows up to 64
    return launch_tc(a, kp, map->num_ctas, to_cuda(stream));
}

}  // namespace

extern "C" dsa_status dsa_decode_ex(int32_t q_len, int32_t kv_layout, const void *q, dsa_dtype q_dtype,
                                    const float *q_scale, const void *k_pages, const void *v_pages,
                                    dsa_dtype kv_dtype, const float *k_scale, const float *v_scale,
                                    const int32_t *block_table, int32_t max_pages_per_req, int32_t num_pages,
                                    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t page_size, float sm_scale,
                                    const dsa_task_map *map, float *partial_o, float *partial_lse,
                                    uint64_t *cta_times, dsa_stream stream) {
    return decode_impl(q_len, kv_layout, q, q_dtype, q_scale, k_pages, v_pages, kv_dtype, k_scale, v_scale,
                       block_table, max_pages_per_req, num_pages, seq_lens, batch, num_q_heads, num_kv_heads,
                       head_dim, page_size, sm_scale, map, partial_o, partial_lse, cta_times, -1, stream);
}

extern "C" dsa_status dsa_decode_chained(int32_t new_tokens, const void *q, dsa_dtype q_dtype, const float *q_scale,
                                         const void *k_pages, const void *v_pages, dsa_dtype kv_dtype,
                                         const float *k_scale, const float *v_scale, const int32_t *block_table,
                                         int32_t max_pages_per_req, int32_t num_pages, const int32_t *seq_lens,
                                         int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t page_size, float sm_scale,
                                         const dsa_task_map *map, float *partial_o, float *partial_lse,
                                         dsa_stream stream) {
    if (new_tokens < 0) return DSA_ERR_INVALID_ARG;
    return decode_impl(1, DSA_HND, q, q_dtype, q_scale, k_pages, v_pages, kv_dtype, k_scale, v_scale, block_table,
                       max_pages_per_req, num_pages, seq_lens, batch, num_q_heads, num_kv_heads, head_dim,
                       page_size, sm_scale, map, partial_o, partial_lse, nullptr, new_tokens, stream);
}

extern "C" dsa_status dsa_decode(const void *q, dsa_dtype q_dtype, const float *q_scale, const void *k_pages,
                                 const void *v_pages, dsa_dtype kv_dtype, const float *k_scale,
                                 const float *v_scale, const int32_t *block_table, int32_t max_pages_per_req,
                                 int32_t num_pages, const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t page_size, float sm_scale,
                                 const dsa_task_map *map, float *partial_o, float *partial_lse,
                                 dsa_stream stream) {
    return dsa_decode_ex(1, DSA_HND, q, q_dtype, q_scale, k_pages, v_pages, kv_dtype, k_scale, v_scale,
                         block_table, max_pages_per_req, num_pages, seq_lens, batch, num_q_heads, num_kv_heads,
                         head_dim, page_size, sm_scale, map, partial_o, partial_lse, nullptr, stream);
}

extern "C" dsa_status dsa_decode_multi(int32_t q_len, const void *q, dsa_dtype q_dtype, const float *q_scale,
                                       const void *k_pages, const void *v_pages, dsa_dtype kv_dtype,
                                       const float *k_scale, const float *v_scale, const int32_t *block_table,
                                       int32_t max_pages_per_req, int32_t num_pages, const int32_t *seq_lens,
                                       int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                       int32_t page_size, float sm_scale, const dsa_task_map *map, float *partial_o,
                                       float *partial_lse, dsa_stream stream) {
    return dsa_decode_ex(q_len, DSA_HND, q, q_dtype, q_scale, k_pages, v_pages, kv_dtype, k_scale, v_scale,
                         block_table, max_pages_per_req, num_pages, seq_lens, batch, num_q_heads, num_kv_heads,
                         head_dim, page_size, sm_scale, map, partial_o, partial_lse, nullptr, stream);
}

extern "C" dsa_status dsa_decode_fused(const void *q, dsa_dtype q_dtype, const float *q_scale, const void *k_pages,
                                       const void *v_pages, dsa_dtype kv_dtype, const float *k_scale,
                                       const float *v_scale, const int32_t *block_table,
                                       int32_t max_pages_per_req, int32_t num_pages, const int32_t *seq_lens,
                                       int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                       int32_t page_size, float sm_scale, const dsa_task_map *map, float *partial_o,
                                       float *partial_lse, int32_t *unit_counters, void *out, dsa_dtype out_dtype,
                                       float *out_lse, dsa_stream stream) {
    const AttnArgs a{q, q_dtype, q_scale, k_pages, v_pages, kv_dtype, k_scale, v_scale, block_table,
                     max_pages_per_req, num_pages, seq_lens, batch, num_q_heads, num_kv_heads, head_dim,
                     page_size, sm_scale};
    dsa_status s = validate_attn(a);
    if (s != DSA_OK) return s;
    if (out_dtype != DSA_BF16 && out_dtype != DSA_FP32) return DSA_ERR_UNSUPPORTED;
    if (!map || !map->cta_desc_begin || !map->descs || !map->meta || !partial_o || !partial_lse) return DSA_ERR_INVALID_ARG;
    if (map->num_units != batch * num_kv_heads || map->num_ctas < 1) return DSA_ERR_INVALID_ARG;
    if (batch > 0 && (!map->unit_partial_begin || !map->unit_num_partials || !unit_counters || !out))
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(partial_o) || !aligned16(map->descs) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
    if (batch == 0) return DSA_OK;
    KernelParams kp = base_params(a, partial_o, partial_lse, map->meta + 3);
    kp.max_slots = map->max_descs;
    kp.cta_desc_begin = map->cta_desc_begin;
    kp.descs = reinterpret_cast<const int4 *>(map->descs);
    kp.unit_partial_begin = map->unit_partial_begin;
    kp.unit_num_partials = map->unit_num_partials;
    kp.unit_counters = unit_counters;
    kp.out = out;
    kp.out_bf16 = out_dtype == DSA_BF16;
    kp.out_lse = out_lse;
    return launch_decode(a, kp, map->num_ctas, true, to_cuda(stream));
}

extern "C" dsa_status dsa_selftest_wait_timeout(int32_t *status, int64_t limit_ns, dsa_stream stream) {
    if (!status || limit_ns <= 0 || limit_ns > static_cast<int64_t>(kWaitLimitNs)) return DSA_ERR_INVALID_ARG;
    return launch_wait_selftest(status, static_cast<uint64_t>(limit_ns), to_cuda(stream));
}

extern "C" int32_t dsa_static_num_splits(int32_t mode, int32_t param, int32_t max_seq_len) {
    if (mode == 0) return param >= 1 ? param : -1;
    if (mode != 1 || param < kTile || param % kTile != 0 || max_seq_len < 0) return -1;
    const int64_t s = (static_cast<int64_t>(max_seq_len) + param - 1) / param;
    return s < 1 ? 1 : (s > 65535 ? -1 : static_cast<int32_t>(s));
}

extern "C" dsa_status dsa_static_splitkv(int32_t mode, int32_t param, int32_t max_seq_len, const void *q,
                                         dsa_dtype q_dtype, const float *q_scale, const void *k_pages,
                                         const void *v_pages, dsa_dtype kv_dtype, const float *k_scale,
                                         const float *v_scale, const int32_t *block_table,
                                         int32_t max_pages_per_req, int32_t num_pages, const int32_t *seq_lens,
                                         int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t page_size, float sm_scale, float *partial_o,
                                         float *partial_lse, int32_t *status, uint64_t *cta_times,
                                         dsa_stream stream) {
    const AttnArgs a{q, q_dtype, q_scale, k_pages, v_pages, kv_dtype, k_scale, v_scale, block_table,
                     max_pages_per_req, num_pages, seq_lens, batch, num_q_heads, num_kv_heads, head_dim,
                     page_size, sm_scale};
    dsa_status s = validate_attn(a);
    if (s != DSA_OK) return s;
    const int32_t S = dsa_static_num_splits(mode, param, max_seq_len);
    if (S < 1 || S > 65535) return DSA_ERR_INVALID_ARG;
    if (!partial_o || !partial_lse || !status || !aligned16(partial_o)) return DSA_ERR_INVALID_ARG;
    if (num_kv_heads > 65535 || batch > 65535) return DSA_ERR_UNSUPPORTED;
    if (batch == 0) return DSA_OK;
    KernelParams kp = base_params(a, partial_o, partial_lse, status);
    kp.static_mode = mode;
    kp.static_tiles = mode == 1 ? param / kTile : 0;
    kp.num_splits = S;
    kp.max_slots = batch * num_kv_heads * S;
    kp.cta_times = cta_times;
    const dim3 grid(S, num_kv_heads, batch);
    return launch_static(a, kp, grid, to_cuda(stream));
}
