// Combine: merges the partial outputs of each (request, KV head) unit under the
// global softmax normalisation (HPC-Ops × SGLang blog, section "围绕活跃 KV 工作进行
// 调度": the combine kernel reads the actual number of partials per request and
// head; Hy3 preview write-up 2.1.1 "Combine Kernel"):
//   L = ln sum_k exp(lse_k),   out = sum_k exp(lse_k - L) * o_k.
// One CTA per unit and block of 8 query rows, one warp per query row of the unit (query
// token i, head g: row i*G + g; one query token in a plain decode step), each lane owning
// 4 of the 128 output dims (float4 loads of the fp32 partials, coalesced per row).
#include <cuda_bf16.h>

#include "common.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <typename OutT>
__device__ __forceinline__ void store4(OutT *dst, float4 v);

template <>
__device__ __forceinline__ void store4<float>(float *dst, float4 v) {
    *reinterpret_cast<float4 *>(dst) = v;
}

template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *dst, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t *>(&a);
    packed.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(dst) = packed;
}

// STATIC: unit u owns slots [u*S, u*S + S); otherwise the task map's slots.
template <bool STATIC, typename OutT>
__global__ void __launch_bounds__(kMaxGroup * 32)
    combine_kernel(const int32_t *__restrict__ unit_begin, const int32_t *__restrict__ unit_count, int32_t S,
                   const float *__restrict__ partial_o, const float *__restrict__ partial_lse, int32_t hq,
                   int32_t hkv, int32_t G, int32_t q_len, int32_t spd, OutT *__restrict__ out,
                   float *__restrict__ out_lse) {
    const int u = blockIdx.x;
    const int row = blockIdx.y * kMaxGroup + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    // spd partial slots per descriptor: the unit's slots are [spd * begin, spd * (begin + count)).
    // The task map is read before the wait: the decode before this kernel releases it only after
    // its own wait, when the plan that wrote the map has completed.
    const int64_t beg = STATIC ? static_cast<int64_t>(u) * S : static_cast<int64_t>(unit_begin[u]) * spd;
    const int n = STATIC ? S : unit_count[u] * spd;
    grid_launch_dependents();
    grid_dependency_wait();  // partials from the decode kernel
    const int R = q_len * G;  // partial rows per slot
    if (row >= R) return;
    const int b = u / hkv, h = u - b * hkv;

    // the first kPre partials' rows are loaded together with the LSEs, so the merge of a unit
    // with few partials waits for one round trip to memory after the lengths, not two
    constexpr int kPre = 8;
    float4 pre[kPre];
#pragma unroll
    for (int j = 0; j < kPre; ++j)
        if (j < n) pre[j] = *reinterpret_cast<const float4 *>(partial_o + ((beg + j) * R + row) * kHeadDim + lane * 4);
    const float lse0 = lane < n ? partial_lse[(beg + lane) * R + row] : -INFINITY;
    float M = lse0;
    for (int k = lane + 32; k < n; k += 32) M = fmaxf(M, partial_lse[(beg + k) * R + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = -INFINITY;
    if (M != -INFINITY) {
        float sum = lane < n ? exp2f((lse0 - M) * kLog2e) : 0.f;
        for (int k = lane + 32; k < n; k += 32) sum += exp2f((partial_lse[(beg + k) * R + row] - M) * kLog2e);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        L = M + logf(sum);
        // 32 partials at a time: lane k holds the weight of partial k0 + k
        for (int k0 = 0; k0 < n; k0 += 32) {
            const int kn = min(32, n - k0);
            const float lk = k0 == 0 ? lse0 : (lane < kn ? partial_lse[(beg + k0 + lane) * R + row] : -INFINITY);
            const float w = lane < kn ? exp2f((lk - L) * kLog2e) : 0.f;
            if (k0 == 0) {
#pragma unroll
                for (int j = 0; j < kPre; ++j) {
                    if (j >= kn) break;
                    const float wj = __shfl_sync(0xffffffffu, w, j);
                    acc.x += wj * pre[j].x;
                    acc.y += wj * pre[j].y;
                    acc.z += wj * pre[j].z;
                    acc.w += wj * pre[j].w;
                }
            }
#pragma unroll 8
            for (int j = k0 == 0 ? kPre : 0; j < kn; ++j) {
                const float4 v =
                    *reinterpret_cast<const float4 *>(partial_o + ((beg + k0 + j) * R + row) * kHeadDim + lane * 4);
                const float wj = __shfl_sync(0xffffffffu, w, j);
                acc.x += wj * v.x;
                acc.y += wj * v.y;
                acc.z += wj * v.z;
                acc.w += wj * v.w;
            }
        }
    }
    const int qi = row / G, g = row - qi * G;
    const int64_t orow = (static_cast<int64_t>(b) * q_len + qi) * hq + h * G + g;
    store4<OutT>(out + orow * kHeadDim + lane * 4, acc);
    if (out_lse && lane == 0) out_lse[orow] = L;
}

dsa_status validate_combine(int32_t batch, int32_t hq, int32_t hkv, int32_t head_dim, const float *po,
                            const float *plse, void *out, dsa_dtype out_dtype) {
    if (batch < 0 || hq < 1 || hkv < 1 || hq % hkv != 0) return DSA_ERR_INVALID_ARG;
    if (head_dim != kHeadDim) return DSA_ERR_UNSUPPORTED;
    if (hq / hkv > kMaxGroup) return DSA_ERR_UNSUPPORTED;
    if (out_dtype != DSA_BF16 && out_dtype != DSA_FP32) return DSA_ERR_UNSUPPORTED;
    if (batch > 0 && (!po || !plse || !out)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(po) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

template <bool STATIC>
dsa_status launch_combine(const int32_t *ub, const int32_t *uc, int32_t S, const float *po, const float *plse,
                          int32_t batch, int32_t hq, int32_t hkv, void *out, dsa_dtype out_dtype, float *out_lse,
                          cudaStream_t st, int32_t q_len = 1, int32_t spd = 1) {
    const int units = batch * hkv;
    if (units == 0) return DSA_OK;
    const int G = hq / hkv;
    const dim3 grid(units, (q_len * G + kMaxGroup - 1) / kMaxGroup);
    if (out_dtype == DSA_BF16)
        return launch_pdl(combine_kernel<STATIC, __nv_bfloat16>, grid, dim3(kMaxGroup * 32), 0, st, ub, uc, S, po,
                          plse, hq, hkv, G, q_len, spd, static_cast<__nv_bfloat16 *>(out), out_lse);
    return launch_pdl(combine_kernel<STATIC, float>, grid, dim3(kMaxGroup * 32), 0, st, ub, uc, S, po, plse, hq,
                      hkv, G, q_len, spd, static_cast<float *>(out), out_lse);
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_combine(const dsa_task_map *map, const float *partial_o, const float *partial_lse,
                                  int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  void *out, dsa_dtype out_dtype, float *out_lse, dsa_stream stream) {
    dsa_status s = validate_combine(batch, num_q_heads, num_kv_heads, head_dim, partial_o, partial_lse, out, out_dtype);
    if (s != DSA_OK) return s;
    if (!map || map->num_units != batch * num_kv_heads) return DSA_ERR_INVALID_ARG;
    if (batch > 0 && (!map->unit_partial_begin || !map->unit_num_partials)) return DSA_ERR_INVALID_ARG;
    return launch_combine<false>(map->unit_partial_begin, map->unit_num_partials, 0, partial_o, partial_lse, batch,
                                 num_q_heads, num_kv_heads, out, out_dtype, out_lse, to_cuda(stream));
}

extern "C" dsa_status dsa_combine_multi(int32_t q_len, const dsa_task_map *map, const float *partial_o,
                                        const float *partial_lse, int32_t batch, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_dim, void *out, dsa_dtype out_dtype,
                                        float *out_lse, dsa_stream stream) {
    dsa_status s = validate_combine(batch, num_q_heads, num_kv_heads, head_dim, partial_o, partial_lse, out, out_dtype);
    if (s != DSA_OK) return s;
    if (q_len < 1) return DSA_ERR_INVALID_ARG;
    if (q_len * (num_q_heads / num_kv_heads) > 64) return DSA_ERR_UNSUPPORTED;
    if (!map || map->num_units != batch * num_kv_heads) return DSA_ERR_INVALID_ARG;
    if (batch > 0 && (!map->unit_partial_begin || !map->unit_num_partials)) return DSA_ERR_INVALID_ARG;
    return launch_combine<false>(map->unit_partial_begin, map->unit_num_partials, 0, partial_o, partial_lse, batch,
                                 num_q_heads, num_kv_heads, out, out_dtype, out_lse, to_cuda(stream), q_len,
                                 dsa_multi_slots_per_desc(q_len, num_q_heads / num_kv_heads));
}

extern "C" dsa_status dsa_static_combine(int32_t num_splits, const float *partial_o, const float *partial_lse,
                                         int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, void *out, dsa_dtype out_dtype, float *out_lse,
                                         dsa_stream stream) {
    dsa_status s = validate_combine(batch, num_q_heads, num_kv_heads, head_dim, partial_o, partial_lse, out, out_dtype);
    if (s != DSA_OK) return s;
    if (num_splits < 1) return DSA_ERR_INVALID_ARG;
    return launch_combine<true>(nullptr, nullptr, num_splits, partial_o, partial_lse, batch, num_q_heads,
                                num_kv_heads, out, out_dtype, out_lse, to_cuda(stream));
}
