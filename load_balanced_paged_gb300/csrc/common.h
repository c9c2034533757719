// Library-internal constants and helpers shared by the kernels and their host launchers.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kHeadDim = 128;  // d
constexpr int kTile = 64;      // tokens per tile = tokens per page
constexpr int kMaxGroup = 8;   // query heads per KV head handled in one MMA column block
constexpr int kPlanMaxUnits = 16384;
constexpr int kPlanMaxCtas = 16384;

inline cudaStream_t to_cuda(dsa_stream s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline dsa_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// Launch with programmatic stream serialization: the kernel may begin while the previous
// kernel in the stream finishes; every kernel of this library calls griddepcontrol.wait
// before it reads global memory, so it never sees unfinished writes.
template <typename... KArgs, typename... Args>
dsa_status launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// Problem description shared by the persistent and the static attention paths.
struct AttnArgs {
    const void *q;
    dsa_dtype q_dtype;
    const float *q_scale;
    const void *k_pages;
    const void *v_pages;
    dsa_dtype kv_dtype;
    const float *k_scale;
    const float *v_scale;
    const int32_t *block_table;
    int32_t max_pages_per_req;
    int32_t num_pages;
    const int32_t *seq_lens;
    int32_t batch;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t page_size;
    float sm_scale;
    int32_t kv_layout = DSA_HND;  // dsa_kv_layout
};

dsa_status validate_attn(const AttnArgs &a);

// Multiprocessor count of the current device (cached per device; 0 if unknown).
int sm_count();

}  // namespace dsa
