// Fused attention prologue: QK-Norm -> RoPE -> optional Hadamard rotation -> encoding,
// with Q written for the attention kernel and K/V written straight into the paged cache.
//
// HPC-Ops × SGLang blog, "融合式 attention 前导": QK-Norm before RoPE, FP8 Q with one
// scale per (token, head) handed to the attention kernel as is, K and V written directly
// into the paged FP8 cache, so no intermediate tensor makes an HBM round trip.  Hy3
// preview write-up §2.2.1 "Fused Rope+Norm+[Hadamard]+Quant+Store KV" (the same chain
// with an optional Hadamard product, kept in registers, written once) and §2.6.1
// "Hadamard在线旋转变换" (an orthogonal rotation of Q and K before quantisation).
//
// Work layout: four lanes hold one (token, head) row of 128 values, 32 each, as four
// chunks of 8 consecutive dims, dims(c, e) = 32 c + 8 l + e for lane l of the four and
// chunk c.  So the RoPE pairs of the full-width neox form (i, i + 64) and of the half-width
// form (i, i + 32) and all interleaved pairs (2i, 2i + 1) sit inside one lane, five of the
// seven Hadamard butterfly stages are in-lane additions, and a row reduction takes two
// shuffles.  A warp takes 8 tokens (one per 4-lane group) and a block of consecutive heads
// of each; the head index is the same for the whole warp at every step, so Q / K / V
// handling is uniform, and the token's position, cache slot and cos/sin values are loaded
// once for the block.  The next head's row is loaded while the current one is computed.
#include "common.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kProTokens = 8;     // tokens per warp (one per 4-lane group)
// CTA shapes: warps per CTA and resident CTAs per SM.  Up to kProSmallTokens tokens, CTAs of
// 4 warps, 3 per SM (up to 170 registers a thread, no spill); beyond, CTAs of 8 warps, 2 per
// SM (128 registers, 16 warps per SM).  Measured on the 64 / 8-head chain: the small shape is
// 0.3-2.5 us faster from 32 to 4096 tokens, the large one 3-5 us faster from 8192 on.
constexpr int kProSmallTokens = 4096;
constexpr float kE4m3Max = 448.0f;
constexpr float kInvSqrtHeadDim = 0.08838834764831845f;  // 1 / sqrt(128)

enum RopeMode { kRopeNone = 0, kRopeNeox128, kRopeNeox64, kRopeNeoxNarrow, kRopeInterleaved };

struct ProParams {
    const uint16_t *qkv;
    int32_t n_tokens, hq, hkv;
    int32_t heads_per_item;  // heads a warp takes per token group
    int32_t items;           // token groups x head blocks
    const int32_t *positions;
    const float *cos_sin;
    int32_t max_position, rot, rope_mode;
    const float *q_norm_w, *k_norm_w;
    float eps;
    int32_t hadamard;
    const int32_t *slots;
    int64_t num_slots;  // num_pages * page_size
    int32_t page_shift; // log2(page_size): page size 16, 32 or 64
    int32_t nhd;        // pages [num_pages][P][Hkv][128] instead of [num_pages][Hkv][P][128]
    void *q_out;
    float *q_scale;
    int32_t q_fp8;
    void *k_pages, *v_pages;
    float *k_scale, *v_scale;
    int32_t kv_fp8;
    int32_t *status;
};

struct Row {
    uint4 c[4];  // 4 chunks x 8 bf16
};

__device__ __forceinline__ Row load_row(const uint16_t *row, int l) {
    Row r;
#pragma unroll
    for (int c = 0; c < 4; ++c) r.c[c] = __ldg(reinterpret_cast<const uint4 *>(row + 32 * c + 8 * l));
    return r;
}

__device__ __forceinline__ void unpack_row(const Row &r, float (&y)[4][8]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t w[4] = {r.c[c].x, r.c[c].y, r.c[c].z, r.c[c].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            y[c][2 * k] = bf16lo_to_f32(w[k]);
            y[c][2 * k + 1] = bf16hi_to_f32(w[k]);
        }
    }
}

// Sum / maximum over the 4 lanes of a row.
__device__ __forceinline__ float row_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

__device__ __forceinline__ float row_max(float v) {
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}

// Angle index of rotation pair p held by lane l, and whether the lane holds that pair.
// neox128: pairs (chunk c, chunk c + 2), p = 8 c + e, c < 2 -> angle 32 c + 8 l + e.
// neox64:  pairs (chunk 0, chunk 1), p = e -> angle 8 l + e.
// narrow neox (rot 16 / 32): chunk 0 only, partner in another lane, p = e
//          -> angle (8 l + e) mod (rot / 2), for lanes with 8 l < rot.
// interleaved: pairs (2k, 2k + 1) of chunk c, p = 4 c + k -> angle 16 c + 4 l + k, for
//          chunks with 32 c + 8 l < rot.
__device__ __forceinline__ void load_angles(const ProParams &p, int l, int pos, float (&cs)[16], float (&sn)[16]) {
    const float *row = p.cos_sin + static_cast<int64_t>(pos) * p.rot;
    const int half = p.rot >> 1;
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // 4 groups of 4 pairs
        int i = -1;
        if (p.rope_mode == kRopeNeox128) i = 32 * (q >> 1) + 8 * l + 4 * (q & 1);
        else if (p.rope_mode == kRopeNeox64) i = q < 2 ? 8 * l + 4 * q : -1;
        else if (p.rope_mode == kRopeNeoxNarrow) i = (q < 2 && 8 * l < p.rot) ? ((8 * l + 4 * q) & (half - 1)) : -1;
        else if (p.rope_mode == kRopeInterleaved) i = (32 * q + 8 * l < p.rot) ? 16 * q + 4 * l : -1;
        float4 c = make_float4(1.f, 1.f, 1.f, 1.f), s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i >= 0) {
            c = __ldg(reinterpret_cast<const float4 *>(row + i));
            s = __ldg(reinterpret_cast<const float4 *>(row + half + i));
        }
        cs[4 * q] = c.x, cs[4 * q + 1] = c.y, cs[4 * q + 2] = c.z, cs[4 * q + 3] = c.w;
        sn[4 * q] = s.x, sn[4 * q + 1] = s.y, sn[4 * q + 2] = s.z, sn[4 * q + 3] = s.w;
    }
}

__device__ __forceinline__ void rotate(float &a, float &b, float c, float s) {
    const float x = a, y = b;
    a = x * c - y * s;
    b = y * c + x * s;
}

// RoPE on the lane's 32 values; uniform control flow (the narrow form shuffles).
__device__ __forceinline__ void rope(const ProParams &p, int l, const float (&cs)[16], const float (&sn)[16],
                                     float (&y)[4][8]) {
    if (p.rope_mode == kRopeNeox128) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) rotate(y[c][e], y[c + 2][e], cs[8 * c + e], sn[8 * c + e]);
    } else if (p.rope_mode == kRopeNeox64) {
#pragma unroll
        for (int e = 0; e < 8; ++e) rotate(y[0][e], y[1][e], cs[e], sn[e]);
    } else if (p.rope_mode == kRopeInterleaved) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k) rotate(y[c][2 * k], y[c][2 * k + 1], cs[4 * c + k], sn[4 * c + k]);
    } else if (p.rope_mode == kRopeNeoxNarrow) {
        // pairs (i, i + rot/2) inside chunk 0: the partner of lane l is lane l xor (rot / 16)
        const int m = p.rot >> 4;
        const bool mine = 8 * l < p.rot, lower = 8 * l < (p.rot >> 1);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, y[0][e], m);
            if (mine) y[0][e] = lower ? y[0][e] * cs[e] - o * sn[e] : y[0][e] * cs[e] + o * sn[e];
        }
    }
}

// y <- H_128 y (Sylvester order; the 1/sqrt(128) is left to the caller).  Dim bits 0-2
// (e) and 5-6 (c) are in-lane butterflies; bits 3-4 (l) pair lanes l and l xor 1, l xor 2
// of the same row.
__device__ __forceinline__ void hadamard(int l, float (&y)[4][8]) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int h = 1; h < 8; h <<= 1)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (!(e & h)) {
                    const float a = y[c][e], b = y[c][e + h];
                    y[c][e] = a + b;
                    y[c][e + h] = a - b;
                }
#pragma unroll
    for (int h = 1; h < 4; h <<= 1)
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (!(c & h))
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float a = y[c][e], b = y[c + h][e];
                    y[c][e] = a + b;
                    y[c + h][e] = a - b;
                }
#pragma unroll
    for (int m = 1; m < 4; m <<= 1) {
        const float sgn = (l & m) ? -1.f : 1.f;  // lower lane: a + b; upper lane: a - b
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float o = __shfl_xor_sync(0xffffffffu, y[c][e], m);
                y[c][e] = fmaf(sgn, y[c][e], o);
            }
    }
}

// RMSNorm with weight w over the row, split into its per-element part y <- y * w and its
// row-wide factor 1 / sqrt(mean(y^2) + eps), which is returned for the caller to apply
// once, together with the other row-wide factor of the chain.  Both shuffles are taken by
// every lane.
__device__ __forceinline__ float rms_norm_weight(const float *w, float eps, int l, float (&y)[4][8]) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(y[c][e], y[c][e], ss);
    const float inv = 1.f / sqrtf(row_sum(ss) * (1.f / kHeadDim) + eps);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float4 w0 = __ldg(reinterpret_cast<const float4 *>(w + 32 * c + 8 * l));
        const float4 w1 = __ldg(reinterpret_cast<const float4 *>(w + 32 * c + 8 * l + 4));
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) y[c][e] *= wv[e];
    }
    return inv;
}

// Encode the row z * f and store it (if `store`); f > 0 is the row-wide factor the chain
// left unapplied (RMSNorm's 1/rms and the Hadamard's 1/sqrt(128)).  E4M3: scale = amax /
// 448 (1 for a zero row) with values z * (448 / amax(z)), which f does not change, and
// the stored scale amax(z) * f / 448.  bf16: z * f rounded.  The amax shuffles are taken
// by every lane.
// row: the 128-element row written in base; srow: the scale's index (FP8)
__device__ __forceinline__ void encode_store(int l, float (&y)[4][8], float f, bool fp8, bool store, void *base,
                                             int64_t row, int64_t srow, float *scale_out) {
    if (fp8) {
        float m = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(y[c][e]));
        const float amax = row_max(m);
        const float inv = amax > 0.f ? kE4m3Max / amax : 1.f;
        if (!store) return;
        uint8_t *dst = static_cast<uint8_t *>(base) + row * kHeadDim + 8 * l;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint2 v;
            v.x = f32x2_to_e4m3x2(y[c][0] * inv, y[c][1] * inv) | (uint32_t(f32x2_to_e4m3x2(y[c][2] * inv, y[c][3] * inv)) << 16);
            v.y = f32x2_to_e4m3x2(y[c][4] * inv, y[c][5] * inv) | (uint32_t(f32x2_to_e4m3x2(y[c][6] * inv, y[c][7] * inv)) << 16);
            *reinterpret_cast<uint2 *>(dst + 32 * c) = v;
        }
        if (l == 0) scale_out[srow] = amax > 0.f ? amax * f / kE4m3Max : 1.f;
    } else {
        if (!store) return;
        uint16_t *dst = static_cast<uint16_t *>(base) + row * kHeadDim + 8 * l;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint4 v;
            v.x = pack_bf16x2(y[c][0] * f, y[c][1] * f);
            v.y = pack_bf16x2(y[c][2] * f, y[c][3] * f);
            v.z = pack_bf16x2(y[c][4] * f, y[c][5] * f);
            v.w = pack_bf16x2(y[c][6] * f, y[c][7] * f);
            *reinterpret_cast<uint4 *>(dst + 32 * c) = v;
        }
    }
}

template <int W, int CPS>
__global__ void __launch_bounds__(W * 32, CPS) prologue_kernel(ProParams p) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int lane = threadIdx.x & 31, grp = lane >> 2, l = lane & 3;
    const int H = p.hq + 2 * p.hkv;
    const int head_blocks = (H + p.heads_per_item - 1) / p.heads_per_item;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * W;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * W + (threadIdx.x >> 5); it < p.items; it += warps) {
        const int item = static_cast<int>(it);
        const int tg = item / head_blocks, hb = item - tg * head_blocks;
        const int n_raw = tg * kProTokens + grp;
        const bool valid = n_raw < p.n_tokens;
        const int n = valid ? n_raw : p.n_tokens - 1;  // idle groups recompute a real row, store nothing
        int pos = 0;
        bool pos_ok = true;
        if (p.rope_mode != kRopeNone) {
            pos = p.positions[n];
            pos_ok = pos >= 0 && pos < p.max_position;
            if (!pos_ok) pos = 0;
        }
        const int64_t slot = p.slots[n];
        const bool slot_ok = slot >= 0 && slot < p.num_slots;
        // cache row of KV head h: HND (page * Hkv + h) * P + offset, NHD slot * Hkv + h; the
        // FP8 scales are [num_pages][Hkv][P] in both
        const int64_t page = slot >> p.page_shift, off = slot - (page << p.page_shift);
        auto kv_row = [&](int h) { return p.nhd ? slot * p.hkv + h : ((page * p.hkv + h) << p.page_shift) + off; };
        auto kv_srow = [&](int h) { return ((page * p.hkv + h) << p.page_shift) + off; };
        if (valid && l == 0 && hb == 0 && p.status) {
            if (!pos_ok) atomicOr(p.status, DSA_DEV_BAD_POSITION);
            if (slot < -1 || slot >= p.num_slots) atomicOr(p.status, DSA_DEV_BAD_PAGE);
        }
        float cs[16], sn[16];
        if (p.rope_mode != kRopeNone) load_angles(p, l, pos, cs, sn);
        const int j0 = hb * p.heads_per_item;
        const int j1 = min(H, j0 + p.heads_per_item);
        const uint16_t *tok = p.qkv + static_cast<int64_t>(n) * H * kHeadDim;
        Row next = load_row(tok + static_cast<int64_t>(j0) * kHeadDim, l);
        for (int j = j0; j < j1; ++j) {
            const Row cur = next;
            if (j + 1 < j1) next = load_row(tok + static_cast<int64_t>(j + 1) * kHeadDim, l);
            float y[4][8];
            unpack_row(cur, y);
            if (j < p.hq + p.hkv) {  // Q or K head (uniform over the warp)
                // RoPE and the Hadamard rotation are linear, so RMSNorm's row factor and the
                // rotation's 1/sqrt(128) are applied once, at the encoding
                const bool is_q = j < p.hq;
                const float *w = is_q ? p.q_norm_w : p.k_norm_w;
                float f = w ? rms_norm_weight(w, p.eps, l, y) : 1.f;
                if (p.rope_mode != kRopeNone) rope(p, l, cs, sn, y);
                if (p.hadamard) {
                    hadamard(l, y);
                    f *= kInvSqrtHeadDim;
                }
                if (is_q) {
                    const int64_t row = static_cast<int64_t>(n) * p.hq + j;
                    encode_store(l, y, f, p.q_fp8, valid && pos_ok, p.q_out, row, row, p.q_scale);
                } else {
                    const int h = j - p.hq;
                    encode_store(l, y, f, p.kv_fp8, valid && pos_ok && slot_ok, p.k_pages, kv_row(h), kv_srow(h),
                                 p.k_scale);
                }
            } else {
                const int h = j - p.hq - p.hkv;
                encode_store(l, y, 1.f, p.kv_fp8, valid && slot_ok, p.v_pages, kv_row(h), kv_srow(h), p.v_scale);
            }
        }
    }
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_prologue(const void *qkv, int32_t n_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, const int32_t *positions, const float *cos_sin,
                                   int32_t max_position, int32_t rotary_dim, int32_t rope_style,
                                   const float *q_norm_weight, const float *k_norm_weight, float norm_eps,
                                   int32_t hadamard, const int32_t *slot_mapping, void *q_out, dsa_dtype q_dtype,
                                   float *q_scale, void *k_pages, void *v_pages, dsa_dtype kv_dtype,
                                   float *k_scale, float *v_scale, int32_t num_pages, int32_t page_size,
                                   int32_t kv_layout, int32_t *status, dsa_stream stream) {
    if (n_tokens < 0 || num_q_heads < 1 || num_kv_heads < 1 || num_pages < 0) return DSA_ERR_INVALID_ARG;
    if (head_dim != kHeadDim || !(page_size == 16 || page_size == 32 || page_size == kTile))
        return DSA_ERR_UNSUPPORTED;
    if (kv_layout != DSA_HND && kv_layout != DSA_NHD) return DSA_ERR_INVALID_ARG;
    if (!(rotary_dim == 0 || rotary_dim == 16 || rotary_dim == 32 || rotary_dim == 64 || rotary_dim == 128))
        return DSA_ERR_UNSUPPORTED;
    if (rope_style != DSA_ROPE_NEOX && rope_style != DSA_ROPE_INTERLEAVED) return DSA_ERR_INVALID_ARG;
    if ((q_dtype != DSA_BF16 && q_dtype != DSA_FP8_E4M3) || (kv_dtype != DSA_BF16 && kv_dtype != DSA_FP8_E4M3))
        return DSA_ERR_UNSUPPORTED;
    if (!(norm_eps >= 0.f) || norm_eps == INFINITY) return DSA_ERR_INVALID_ARG;
    if (n_tokens == 0) return DSA_OK;
    if (!qkv || !q_out || !slot_mapping || !k_pages || !v_pages) return DSA_ERR_INVALID_ARG;
    if (rotary_dim && (!positions || !cos_sin || max_position < 1)) return DSA_ERR_INVALID_ARG;
    if (q_dtype == DSA_FP8_E4M3 && !q_scale) return DSA_ERR_INVALID_ARG;
    if (kv_dtype == DSA_FP8_E4M3 && (!k_scale || !v_scale)) return DSA_ERR_INVALID_ARG;
    for (const void *ptr : {qkv, static_cast<const void *>(q_out), static_cast<const void *>(k_pages),
                            static_cast<const void *>(v_pages), static_cast<const void *>(cos_sin),
                            static_cast<const void *>(q_norm_weight), static_cast<const void *>(k_norm_weight)})
        if (!aligned16(ptr)) return DSA_ERR_INVALID_ARG;

    const int64_t H = static_cast<int64_t>(num_q_heads) + 2 * num_kv_heads;
    const int64_t groups = (static_cast<int64_t>(n_tokens) + kProTokens - 1) / kProTokens;
    if (H * kHeadDim > INT32_MAX || groups * H > INT32_MAX) return DSA_ERR_UNSUPPORTED;
    const bool small = n_tokens <= kProSmallTokens;
    const int W = small ? 4 : 8, CPS = small ? 3 : 2;
    const int sms = sm_count();
    const int64_t warps_resident = static_cast<int64_t>(sms > 0 ? sms : 148) * CPS * W;
    // Heads per work item: blocks of 8 consecutive heads amortise the per-token loads; fewer
    // when that would leave the GPU's warps short of work (small decode batches).
    int hpi = 8;
    while (hpi > 1 && groups * ((H + hpi - 1) / hpi) < warps_resident) hpi >>= 1;

    ProParams p = {};
    p.qkv = static_cast<const uint16_t *>(qkv);
    p.n_tokens = n_tokens;
    p.hq = num_q_heads;
    p.hkv = num_kv_heads;
    p.heads_per_item = hpi;
    p.items = static_cast<int32_t>(groups * ((H + hpi - 1) / hpi));
    p.positions = positions;
    p.cos_sin = cos_sin;
    p.max_position = max_position;
    p.rot = rotary_dim;
    p.rope_mode = rotary_dim == 0                        ? kRopeNone
                  : rope_style == DSA_ROPE_INTERLEAVED   ? kRopeInterleaved
                  : rotary_dim == 128                    ? kRopeNeox128
                  : rotary_dim == 64                     ? kRopeNeox64
                                                         : kRopeNeoxNarrow;
    p.q_norm_w = q_norm_weight;
    p.k_norm_w = k_norm_weight;
    p.eps = norm_eps;
    p.hadamard = hadamard != 0;
    p.slots = slot_mapping;
    p.num_slots = static_cast<int64_t>(num_pages) * page_size;
    p.page_shift = page_size == 16 ? 4 : page_size == 32 ? 5 : 6;
    p.nhd = kv_layout == DSA_NHD;
    p.q_out = q_out;
    p.q_scale = q_scale;
    p.q_fp8 = q_dtype == DSA_FP8_E4M3;
    p.k_pages = k_pages;
    p.v_pages = v_pages;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.kv_fp8 = kv_dtype == DSA_FP8_E4M3;
    p.status = status;

    const int64_t want = (p.items + W - 1) / W;
    const int64_t cap = warps_resident / W;
    const int grid = static_cast<int>(want < cap ? want : cap);
    return small ? launch_pdl(prologue_kernel<4, 3>, dim3(grid), dim3(4 * 32), 0, to_cuda(stream), p)
                 : launch_pdl(prologue_kernel<8, 2>, dim3(grid), dim3(8 * 32), 0, to_cuda(stream), p);
}
