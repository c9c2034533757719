// A whole decode step (plan -> persistent decode -> combine) that allocates nothing.
//
// Some callers cannot call cudaMalloc: code that runs where the allocator must not be
// touched (inside another framework's memory pool, a custom allocator's hooks, a
// real-time loop that forbids allocation after start-up), or a plain C program that
// owns only its inputs and outputs.  dsa_decode needs two scratch buffers between its
// kernels -- the task map and the fp32 partial outputs -- so this entry point keeps
// them in one fixed file-scope device array instead of asking the caller for them.
//
// The array lives in every GPU that loads this library, for as long as the process
// runs.  All calls share it, and each call overwrites it: two calls whose kernels
// overlap on the GPU (different streams, or different host threads) race on it.
// Nothing in it has to start at zero: the plan kernel writes every task-map field
// that decode and combine read (status word included), and decode writes every
// partial slot that combine reads.
#include <mutex>

#include "common.h"

namespace dsa {
namespace {

constexpr size_t kScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_step_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_step_scratch on the current device (looked up once per device).
dsa_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_step_scratch) != cudaSuccess || !p) return DSA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return DSA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_decode_step_noalloc(
    const void *q, dsa_dtype q_dtype, const float *q_scale, const void *k_pages, const void *v_pages,
    dsa_dtype kv_dtype, const float *k_scale, const float *v_scale, const int32_t *block_table,
    int32_t max_pages_per_req, int32_t num_pages, const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t page_size, float sm_scale, int32_t num_persistent_ctas,
    int32_t min_tiles_per_split, void *out, dsa_dtype out_dtype, float *out_lse, int32_t *status,
    dsa_stream stream) {
    const AttnArgs a{q, q_dtype, q_scale, k_pages, v_pages, kv_dtype, k_scale, v_scale, block_table,
                     max_pages_per_req, num_pages, seq_lens, batch, num_q_heads, num_kv_heads, head_dim,
                     page_size, sm_scale};
    dsa_status s = validate_attn(a);
    if (s != DSA_OK) return s;
    // every check that dsa_plan, dsa_decode and dsa_combine make on these arguments is made
    // here, before anything is launched: a step is either refused whole or enqueued whole
    if (num_persistent_ctas < 1 || min_tiles_per_split < 1) return DSA_ERR_INVALID_ARG;
    if (out_dtype != DSA_BF16 && out_dtype != DSA_FP32) return DSA_ERR_UNSUPPORTED;
    if (batch > 0 && !out) return DSA_ERR_INVALID_ARG;
    if (!aligned16(out)) return DSA_ERR_INVALID_ARG;
    const int64_t units = static_cast<int64_t>(batch) * num_kv_heads;
    if (units > kPlanMaxUnits || num_persistent_ctas > kPlanMaxCtas) return DSA_ERR_UNSUPPORTED;
    const int32_t md = dsa_max_descs(batch, num_kv_heads, num_persistent_ctas);
    if (md < 0) return DSA_ERR_INVALID_ARG;
    const int64_t G = num_q_heads / num_kv_heads;
    // carve the array: task map, then partial outputs and their LSEs
    const size_t off_begin = 0;
    const size_t off_descs = align256(off_begin + sizeof(int32_t) * (static_cast<size_t>(num_persistent_ctas) + 1));
    const size_t off_upb = align256(off_descs + sizeof(int32_t) * 4 * static_cast<size_t>(md > 0 ? md : 1));
    const size_t off_unp = align256(off_upb + sizeof(int32_t) * static_cast<size_t>(units > 0 ? units : 1));
    const size_t off_meta = align256(off_unp + sizeof(int32_t) * static_cast<size_t>(units > 0 ? units : 1));
    const size_t off_po = align256(off_meta + sizeof(int32_t) * 4);
    const size_t off_pl = align256(off_po + sizeof(float) * static_cast<size_t>(md > 0 ? md : 1) * G * kHeadDim);
    const size_t need = off_pl + sizeof(float) * static_cast<size_t>(md > 0 ? md : 1) * G;
    if (need > kScratchBytes) return DSA_ERR_BUFFER_TOO_SMALL;

    void *base = nullptr;
    s = scratch_address(&base);
    if (s != DSA_OK) return s;
    unsigned char *b = static_cast<unsigned char *>(base);
    dsa_task_map map;
    map.cta_desc_begin = reinterpret_cast<int32_t *>(b + off_begin);
    map.descs = reinterpret_cast<int32_t *>(b + off_descs);
    map.unit_partial_begin = reinterpret_cast<int32_t *>(b + off_upb);
    map.unit_num_partials = reinterpret_cast<int32_t *>(b + off_unp);
    map.meta = reinterpret_cast<int32_t *>(b + off_meta);
    map.max_descs = md;
    map.num_ctas = num_persistent_ctas;
    map.num_units = static_cast<int32_t>(units);
    float *partial_o = reinterpret_cast<float *>(b + off_po);
    float *partial_lse = reinterpret_cast<float *>(b + off_pl);

    s = dsa_plan(seq_lens, batch, num_kv_heads, num_persistent_ctas, kTile, min_tiles_per_split, &map, stream);
    if (s != DSA_OK) return s;
    s = dsa_decode(q, q_dtype, q_scale, k_pages, v_pages, kv_dtype, k_scale, v_scale, block_table,
                   max_pages_per_req, num_pages, seq_lens, batch, num_q_heads, num_kv_heads, head_dim, page_size,
                   sm_scale, &map, partial_o, partial_lse, stream);
    if (s != DSA_OK) return s;
    s = dsa_combine(&map, partial_o, partial_lse, batch, num_q_heads, num_kv_heads, head_dim, out, out_dtype,
                    out_lse, stream);
    if (s != DSA_OK) return s;
    if (status &&
        cudaMemcpyAsync(status, map.meta + 3, sizeof(int32_t), cudaMemcpyDeviceToDevice, to_cuda(stream)) !=
            cudaSuccess)
        return DSA_ERR_CUDA;
    return DSA_OK;
}
