// Argument validation shared by the attention entry points, status readback and
// status strings.
#include "common.h"

namespace dsa {

int sm_count() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!cached[dev]) cudaDeviceGetAttribute(&cached[dev], cudaDevAttrMultiProcessorCount, dev);
    return cached[dev];
}

dsa_status validate_attn(const AttnArgs &a) {
    if (a.batch < 0 || a.num_q_heads < 1 || a.num_kv_heads < 1 || a.num_q_heads % a.num_kv_heads != 0 ||
        a.max_pages_per_req < 0 || a.num_pages < 0)
        return DSA_ERR_INVALID_ARG;
    if (a.head_dim != kHeadDim || !(a.page_size == 16 || a.page_size == 32 || a.page_size == kTile))
        return DSA_ERR_UNSUPPORTED;
    if (a.kv_layout != DSA_HND && a.kv_layout != DSA_NHD) return DSA_ERR_INVALID_ARG;
    if (a.num_q_heads / a.num_kv_heads > kMaxGroup) return DSA_ERR_UNSUPPORTED;
    const bool fp8 = a.kv_dtype == DSA_FP8_E4M3;
    if (!((a.q_dtype == DSA_BF16 && a.kv_dtype == DSA_BF16) || (a.q_dtype == DSA_FP8_E4M3 && fp8)))
        return DSA_ERR_UNSUPPORTED;
    if (!(a.sm_scale == a.sm_scale) || a.sm_scale == INFINITY || a.sm_scale == -INFINITY)
        return DSA_ERR_INVALID_ARG;
    if (a.batch == 0) return DSA_OK;
    if (!a.q || !a.block_table || !a.seq_lens) return DSA_ERR_INVALID_ARG;
    if (a.num_pages > 0 && (!a.k_pages || !a.v_pages)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(a.q) || !aligned16(a.k_pages) || !aligned16(a.v_pages)) return DSA_ERR_INVALID_ARG;
    if (fp8) {
        if (!a.q_scale || (a.num_pages > 0 && (!a.k_scale || !a.v_scale))) return DSA_ERR_INVALID_ARG;
        if (!aligned16(a.k_scale) || !aligned16(a.v_scale)) return DSA_ERR_INVALID_ARG;
    }
    if (static_cast<int64_t>(a.batch) * a.max_pages_per_req > INT32_MAX / 2 ||
        static_cast<int64_t>(a.max_pages_per_req) * a.page_size > INT32_MAX / 2)
        return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_read_status(const int32_t *device_status, int32_t *host_status) {
    if (!device_status || !host_status) return DSA_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return DSA_ERR_CUDA;
    if (cudaMemcpy(host_status, device_status, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return DSA_ERR_CUDA;
    return *host_status == 0 ? DSA_OK : DSA_ERR_DEVICE_INPUT;
}

extern "C" dsa_status dsa_get_status(const dsa_task_map *map, int32_t *host_status) {
    if (!map || !map->meta) return DSA_ERR_INVALID_ARG;
    return dsa_read_status(map->meta + 3, host_status);
}

extern "C" const char *dsa_status_string(dsa_status s) {
    switch (s) {
        case DSA_OK: return "DSA_OK";
        case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG: invalid argument";
        case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: configuration not supported";
        case DSA_ERR_BUFFER_TOO_SMALL: return "DSA_ERR_BUFFER_TOO_SMALL: caller buffer too small";
        case DSA_ERR_CUDA: return "DSA_ERR_CUDA: CUDA call or launch failed";
        case DSA_ERR_DEVICE_INPUT: return "DSA_ERR_DEVICE_INPUT: kernels flagged bad device input";
    }
    return "unknown dsa_status";
}
