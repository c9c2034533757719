// Paged-KV GQA decode attention over 64-token tiles, in two schedules:
//   - persistent (dsa_decode): one CTA per task-map bin drains its descriptors
//     (HPC-Ops × SGLang blog, section "围绕活跃 KV 工作进行调度");
//   - static split-KV (dsa_static_splitkv): one CTA per (split, KV head, request)
//     on a fixed grid (same blog, section "Attention：变长 decode 的负载均衡").
// Both run the same per-tile engine.
//
// Engine (per CTA):
//   * one producer warp walks the descriptors, reads the page ids of the tiles
//     from the block table (32 at a time, one per lane) and streams each
//     (page, KV head) K and V block -- contiguous 16 KB (bf16) / 8 KB (E4M3) --
//     into a ring of shared-memory stages with TMA (cp.async.bulk.tensor, 128-byte
//     swizzle), completion counted on mbarriers; E4M3 scales and Q come by bulk copy;
//   * GROUPS groups of 4 consumer warps take alternate tiles; warp w of a group
//     owns tokens [16w, 16w+16) of its tile.  One KV tile feeds all G <= 8 query
//     heads of its KV head (GQA: the KV stream is read once):
//       S^T[16 tok x 8 heads] = K[16 x 128] . Q^T   (mma.sync m16n8k16 bf16 or
//                                                    m16n8k32 e4m3, fp32 accumulate)
//       online softmax in base 2, fp32, per warp and head
//       O^T[128 x 8] += V^T[128 x 16] . P^T         (P transposed in registers
//                                                    with movmatrix)
//     bf16: P is split into a bf16 high part and a bf16 residual, two MMAs, so the
//     probabilities carry ~16 bits; E4M3: V is converted exactly to f16 in registers
//     and P (times the per-token V scale) is f16;
//   * at the end of a descriptor the warps' (m, l, O) are merged in shared memory
//     and written as a normalised fp32 partial with its natural-log LSE.
// Every wait is bounded (a few seconds of %globaltimer); on expiry the CTA sets
// DSA_DEV_TIMEOUT, stops, lets its in-flight copies land and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct KernelParams {
    const uint8_t *q;
    const float *q_scale;
    const float *k_scale;
    const float *v_scale;
    const int32_t *block_table;
    const int32_t *seq_lens;
    int32_t max_pages, num_pages, hq, hkv, G, num_units, max_slots;
    int32_t q_len;      // query tokens per request (1: plain decode; > 1: multi-token verify)
    int32_t slots_per_desc;  // partial slots per descriptor (2 for the tensor-core multi-token path)
    int32_t page_size;       // tokens per page P (16, 32 or 64); a 64-token tile spans 64 / P pages
    int32_t nhd;             // pages laid out [num_pages][P][Hkv][d] instead of [num_pages][Hkv][P][d]
    float score_scale;  // sm_scale * log2(e)
    // persistent schedule
    const int32_t *cta_desc_begin;
    const int4 *descs;
    // static schedule
    int32_t static_mode, static_tiles, num_splits;
    float *partial_o;
    float *partial_lse;
    int32_t *status;
    // fused combine (dsa_decode_fused)
    const int32_t *unit_partial_begin;
    const int32_t *unit_num_partials;
    int32_t *unit_counters;  // [B * Hkv]: partials of the unit published so far; 0 between steps
    void *out;               // [B, Hq, 128] bf16 or fp32
    int32_t out_bf16;
    float *out_lse;          // [B, Hq] or null
    uint64_t *cta_times;     // null, or [CTAs][2]: %globaltimer ns when a CTA starts work and ends
};

// Stamps the end of a CTA's work: every warp raises the CTA's end time as it leaves.
struct EndStamp {
    uint64_t *at;
    __device__ ~EndStamp() {
        if (at && (threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned long long *>(at), globaltimer_ns());
    }
};

template <int KV>
struct Cfg;
template <>
struct Cfg<0> {  // bf16 K/V and Q
    static constexpr int kTileBytes = kTile * kHeadDim * 2;
    static constexpr int kScaleBytes = 0;
    static constexpr int kQHeadBytes = kHeadDim * 2;
};
template <>
struct Cfg<1> {  // E4M3 K/V and Q, fp32 scales
    static constexpr int kTileBytes = kTile * kHeadDim;
    static constexpr int kScaleBytes = kTile * 4;
    static constexpr int kQHeadBytes = kHeadDim;
};

constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

constexpr int kEpiRing = 8;  // merged descriptors the epilogue warp may lag behind (fused combine)
constexpr int kMaxRows = 64; // query rows (query tokens x G) of one unit in a multi-token step
constexpr int kDescInfoBytes = 80;
constexpr int kMaxPagesPerTile = kTile / 16;  // pages of 16 tokens: four per tile

// QW = 0: one query token per request; the consumer groups take alternate tiles and all
// warps of the CTA merge at each descriptor end.  QW = 3: multi-token queries on the
// 5th-generation tensor cores: S = Q K^T and O = P V accumulate in tensor memory, two
// teams of four softmax warps, a warp issuing S (and laying Q out as its operand), a warp
// issuing P.V.  (An mma.sync kernel for up to 16 query rows per unit of bf16 K/V measured
// 214-221 us on the mixed lengths against 191-195 us for the tensor-memory kernel at 2-16
// rows: bf16 K/V always takes the tensor-memory kernel.)  E4M3 K/V above 16 rows takes it
// too (S with E4M3 products, V widened to f16 in shared memory).  QW = 4: E4M3 K/V with up
// to 16 rows on mma.sync, the one-token shape (groups on alternate tiles, 16 tokens per
// warp) over two 8-row blocks; each group merges its warps into its own partial slot.
// (There the tensor-memory kernel, bound by its per-tile chain, measured twice the time; an
// mma.sync kernel giving each warp a 32-token half of every tile measured 1.1-1.6x the
// tensor-memory kernel's time at 24-64 rows.)
template <int KV, int STAGES, int GROUPS, int MSLOTS = 2, int QW = 0>
struct Layout {
    // descriptors handed ahead to the consumers (Q + info): with one query token a slot is
    // small, and more of them let the producer run ahead through runs of short descriptors
    static constexpr int kQSlots = (QW == 0 || QW == 4) ? 4 : 2;
    static constexpr bool kTc = QW == 3;
    static constexpr int kNcw = GROUPS * 4;  // consumer warps (softmax warps for QW = 3)
    static constexpr int kThreads = (kNcw + (kTc ? 3 : 1)) * 32;  // consumers + producer (+ MMA, Q warps)
    static constexpr int kThreadsFused = (kNcw + 2) * 32;  // + epilogue warp (fused combine)
    static constexpr int kStageTx = 2 * Cfg<KV>::kTileBytes + 2 * Cfg<KV>::kScaleBytes;
    // QW = 3 with E4M3: each stage also holds its V widened to f16 ([half][64 rows][128 B],
    // 128-byte swizzle: the P.V operand layout of a bf16 V tile)
    static constexpr int kVcOff = round_up(kStageTx, 1024);
    static constexpr int kStageBytes = kVcOff + (kTc && KV == 1 ? kTile * kHeadDim * 2 : 0);
    static constexpr int kQRows = QW == 0 ? kMaxGroup : (QW == 4 ? 16 : kMaxRows);
    static constexpr int kQSlot = kQRows * Cfg<KV>::kQHeadBytes;
    static constexpr int kQOff = STAGES * kStageBytes;
    static constexpr int kOStride = 132;  // floats per head row of a warp's O (padding avoids bank conflicts)
    static constexpr int kWarpRows = QW == 4 ? 16 : kMaxGroup;  // rows of a warp's merge deposit
    static constexpr int kWarpFloats = kWarpRows * kOStride + 2 * kWarpRows;
    // QW = 3: Q as the MMA's A operand (64 rows x 128, K-major with the 128-byte swizzle, two
    // 64-column halves of 8 KB, as the TMA lays out a K tile), two buffers.
    static constexpr int kQcOff = kQOff + kQSlots * kQSlot;
    static constexpr int kQcBytes = kTc ? 2 * kMaxRows * Cfg<KV>::kQHeadBytes : 0;
    static constexpr int kMergeOff = kQcOff + kQcBytes;
    static constexpr bool kMerge = QW == 0 || QW == 4;  // warps merge their states in shared memory
    static constexpr int kMergeSlot = kMerge ? kNcw * kWarpFloats : 0;  // floats per merge slot
    static constexpr int kMergeBars = kMerge ? 2 : 0;  // merge_full / merge_done barriers each (QW = 4: per group)
    static constexpr int kTcBars = kTc ? 22 : 0;  // s_full, s_free, p_full x4; o_done, o_free, qc_full, qc_free, qd_full x2
    static constexpr int kBarOff = kMergeOff + MSLOTS * kMergeSlot * 4;
    // full, empty, qfull, qempty, merge_full, merge_done, epi_ready, epi_free, tensor-core barriers
    static constexpr int kNumBars = 2 * STAGES + 2 * kQSlots + 2 * kMergeBars + 2 * kEpiRing + kTcBars;
    static constexpr int kNValidOff = kBarOff + kNumBars * 8;
    static constexpr int kAbortOff = kNValidOff + STAGES * 4;  // abort flag, then the TMEM base address
    static constexpr int kInfoOff = round_up(kAbortOff + 16, 64);  // one DescInfo per Q slot
    static constexpr int kEpiOff = kInfoOff + kQSlots * kDescInfoBytes;  // kEpiRing EpiRecords + descriptor total
    static constexpr int kBytes = kEpiOff + kEpiRing * 16 + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024
    static_assert(MSLOTS == 1 || MSLOTS == 2, "merge slots");
    static_assert(QW == 0 || (MSLOTS == 1 && GROUPS == 2), "multi-token shapes");
    static_assert(!kTc || kQcOff % 1024 == 0, "tensor-core operand buffers");
    // Each stage must be consumed by one group only: a group then meets the phases of its
    // stages' full barriers in order.  With stages shared by two groups, one group could wait
    // for phase k+1 while phase k is still pending, pass the parity test early and arrive on
    // the stage's empty barrier out of turn (an undefined mbarrier use that faults the GPU).
    static_assert(!(QW == 0 || QW == 4) || STAGES % GROUPS == 0, "each stage must belong to one consumer group");
    static_assert(kStageBytes % 1024 == 0 && kQOff % 1024 == 0, "swizzled TMA boxes need 1024-byte alignment");
    static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

struct Desc {
    int u, t0, t1, slot;
    bool ok;
};

// What the producer hands the consumers with each descriptor's Q (shared memory).
struct DescInfo {
    int end;      // 1: no more descriptors in this CTA
    int b, h;     // request, KV head
    int n;        // tiles
    int slot;     // partial-output slot
    int c_start;  // ring position of the descriptor's first tile
    int np;       // partials of the descriptor's unit (fused combine)
    int pbeg;     // first partial slot of the unit (fused combine)
    int t0;       // first tile of the descriptor within its unit
    int len;      // the request's KV length
    int pad[2];
    float qscale[kMaxGroup];  // E4M3: q_scale of the G query heads
};
static_assert(sizeof(DescInfo) == kDescInfoBytes, "DescInfo slot size");

// What the consumers hand the epilogue warp with each merged descriptor (fused combine).
struct EpiRecord {
    int b, h, np, pbeg;
};

template <bool PERSIST>
__device__ __forceinline__ Desc get_desc(const KernelParams &p, int d_begin, int i, int t0s, int t1s) {
    Desc x;
    if (PERSIST) {
        const int4 v = p.descs[d_begin + i];
        x.u = v.x;
        x.t0 = v.y;
        x.t1 = v.z;
        x.slot = d_begin + i;
        x.ok = v.x >= 0 && v.x < p.num_units && v.y >= 0 && v.y <= v.z && x.slot < p.max_slots;
    } else {
        x.u = blockIdx.z * p.hkv + blockIdx.y;
        x.t0 = t0s;
        x.t1 = t1s;
        x.slot = x.u * p.num_splits + blockIdx.x;
        x.ok = true;
    }
    return x;
}

// Bounded wait on an mbarrier phase; gives up (false) when the CTA aborted or the
// time limit passed (then it records the timeout and raises the abort flag).
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             int32_t *status, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                atomicOr(status, DSA_DEV_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// The same with the common case inline: a phase that has already completed costs one
// non-blocking test, not a call (measured: 11% off the tensor-core multi-token kernel,
// whose warps meet many completed barriers per tile).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           int32_t *status, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_test_wait(bar, parity)) return true;
    return wait_phase_slow(bar, parity, abort_flag, status, limit_ns);
}

// Wait used while draining after an abort: ignores the abort flag; gives up at `deadline`
// (%globaltimer ns), shared by all the drain's waits.
__device__ __noinline__ void drain_phase(uint32_t bar, uint32_t parity, uint64_t deadline) {
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() > deadline) return;
    }
}

// E4M3 bytes {V[t][2g], V[t][2g+1], V[t+1][2g], V[t+1][2g+1]} -> f16x2 pairs over tokens
// (t, t+1) for dims 2g (lo) and 2g+1 (hi).
__device__ __forceinline__ void cvt_pair(uint32_t x, uint32_t &lo, uint32_t &hi) {
    const uint32_t y = prmt(x, 0, 0x3120);
    lo = e4m3x2_to_f16x2(static_cast<uint16_t>(y & 0xFFFF));
    hi = e4m3x2_to_f16x2(static_cast<uint16_t>(y >> 16));
}

// Byte offset of tile row r (a token) in a bf16 stage laid out [page][half][P rows][128 B]
// (P = 64: [half][64 rows][128 B]); the second 128-B half of the row is P * 128 bytes on.
// Pages are 1024-byte aligned in the stage, so the 128-byte swizzle phase is still r & 7.
__device__ __forceinline__ uint32_t kv_row_off(int r, int P) {
    return static_cast<uint32_t>(r + (r & -P)) * 128u;
}

__device__ __forceinline__ uint32_t tok_mask(int t, int nv) {
    return (t < nv ? 0x0000FFFFu : 0u) | (t + 1 < nv ? 0xFFFF0000u : 0u);
}

template <typename T>
__device__ __forceinline__ void store_out4(void *out, int64_t row, int lane, float4 v, int bf16) {
    if (bf16) {
        const uint32_t lo = pack_bf16x2(v.x, v.y), hi = pack_bf16x2(v.z, v.w);
        reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + row * kHeadDim)[lane] = make_uint2(lo, hi);
    } else {
        reinterpret_cast<float4 *>(static_cast<float *>(out) + row * kHeadDim)[lane] = v;
    }
}

// Last-arriver merge of a unit's partials by one warp (fused combine): per query head the
// global softmax over the partials' LSEs; lane = 4 output dims.  The LSEs of up to 32
// partials are held one per lane, so the per-head maxima and sums are warp reductions, and
// the G rows of each partial are loaded together.
__device__ __noinline__ void combine_unit(const KernelParams &p, int lane, int ub, int uh, int unp, int upbeg) {
    const int G = p.G;
    float4 acc[kMaxGroup];
    float Lh[kMaxGroup];
#pragma unroll
    for (int hd = 0; hd < kMaxGroup; ++hd) {
        acc[hd] = make_float4(0.f, 0.f, 0.f, 0.f);
        Lh[hd] = -INFINITY;
    }
    for (int k0 = 0; k0 < unp; k0 += 32) {
        const int kn = min(32, unp - k0);
        // this chunk's LSEs: lane k holds partial k0 + k
        float lk[kMaxGroup];
#pragma unroll
        for (int hd = 0; hd < kMaxGroup; ++hd)
            lk[hd] = (lane < kn && hd < G) ? __ldcg(p.partial_lse + static_cast<int64_t>(upbeg + k0 + lane) * G + hd)
                                           : -INFINITY;
        // fold the chunk into the running (L, acc) per head: L' = log(e^L + sum e^lk)
        float scale[kMaxGroup], wk[kMaxGroup];
#pragma unroll
        for (int hd = 0; hd < kMaxGroup; ++hd) {
            float m = lk[hd];
#pragma unroll
            for (int o_ = 1; o_ < 32; o_ <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o_));
            m = fmaxf(m, Lh[hd]);
            float e = (lk[hd] == -INFINITY) ? 0.f : exp2f((lk[hd] - m) * kLog2e);
            float sum = e;
#pragma unroll
            for (int o_ = 1; o_ < 32; o_ <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o_);
            const float eprev = (Lh[hd] == -INFINITY) ? 0.f : exp2f((Lh[hd] - m) * kLog2e);
            const float tot = sum + eprev;
            const float Lnew = tot > 0.f ? m + logf(tot) : -INFINITY;
            scale[hd] = tot > 0.f ? eprev / tot : 0.f;   // weight of what acc already holds
            wk[hd] = tot > 0.f ? e / tot : 0.f;          // weight of this lane's partial
            Lh[hd] = Lnew;
        }
#pragma unroll
        for (int hd = 0; hd < kMaxGroup; ++hd) {
            acc[hd].x *= scale[hd];
            acc[hd].y *= scale[hd];
            acc[hd].z *= scale[hd];
            acc[hd].w *= scale[hd];
        }
        for (int k = 0; k < kn; ++k) {
            const float4 *row = reinterpret_cast<const float4 *>(p.partial_o + static_cast<int64_t>(upbeg + k0 + k) * G * kHeadDim);
            float4 v[kMaxGroup];
#pragma unroll
            for (int hd = 0; hd < kMaxGroup; ++hd)
                if (hd < G) v[hd] = __ldcg(row + hd * (kHeadDim / 4) + lane);
#pragma unroll
            for (int hd = 0; hd < kMaxGroup; ++hd) {
                if (hd >= G) continue;
                const float w = __shfl_sync(0xffffffffu, wk[hd], k);
                acc[hd].x += w * v[hd].x;
                acc[hd].y += w * v[hd].y;
                acc[hd].z += w * v[hd].z;
                acc[hd].w += w * v[hd].w;
            }
        }
    }
#pragma unroll
    for (int hd = 0; hd < kMaxGroup; ++hd) {
        if (hd >= G) continue;
        const int64_t orow = static_cast<int64_t>(ub) * p.hq + uh * G + hd;
        store_out4<float>(p.out, orow, lane, acc[hd], p.out_bf16);
        if (lane == 0 && p.out_lse) p.out_lse[orow] = Lh[hd];
    }
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

template <int KV, int STAGES, int GROUPS, bool PERSIST, bool FUSE, int MSLOTS, int QW>
__global__ void __launch_bounds__(FUSE ? Layout<KV, STAGES, GROUPS, MSLOTS, QW>::kThreadsFused
                                       : Layout<KV, STAGES, GROUPS, MSLOTS, QW>::kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                const KernelParams p) {
    using L = Layout<KV, STAGES, GROUPS, MSLOTS, QW>;
    using C = Cfg<KV>;
    constexpr int NCW = L::kNcw;
    constexpr int kQSlots = L::kQSlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::kBarOff;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto qfull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
    auto qempty_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + kQSlots + s); };
    constexpr int MB = L::kMergeBars;
    auto merge_full = [&](int s) { return bar0 + 8u * (2 * STAGES + 2 * kQSlots + s); };
    auto merge_done = [&](int s) { return bar0 + 8u * (2 * STAGES + 2 * kQSlots + MB + s); };
    auto epi_ready = [&](int s) { return bar0 + 8u * (2 * STAGES + 2 * kQSlots + 2 * MB + s); };
    auto epi_free = [&](int s) { return bar0 + 8u * (2 * STAGES + 2 * kQSlots + 2 * MB + kEpiRing + s); };
    const uint32_t tc_bar0 = bar0 + 8u * (2 * STAGES + 2 * kQSlots + 2 * MB + 2 * kEpiRing);
    auto s_full = [&](int b) { return tc_bar0 + 8u * b; };         // 4 S/P buffers
    auto s_free = [&](int b) { return tc_bar0 + 8u * (4 + b); };
    auto p_full = [&](int b) { return tc_bar0 + 8u * (8 + b); };
    auto o_done = [&](int t) { return tc_bar0 + 8u * (12 + t); };  // 2 softmax teams
    auto o_free = [&](int t) { return tc_bar0 + 8u * (14 + t); };
    auto qc_full = [&](int b) { return tc_bar0 + 8u * (16 + b); };
    auto qc_free = [&](int b) { return tc_bar0 + 8u * (18 + b); };
    auto qd_full = [&](int b) { return tc_bar0 + 8u * (20 + b); };  // plain Q rows landed
    EpiRecord *epi_rec = reinterpret_cast<EpiRecord *>(smem + L::kEpiOff);
    volatile int *epi_total = reinterpret_cast<volatile int *>(smem + L::kEpiOff + kEpiRing * sizeof(EpiRecord));
    int *nvalid = reinterpret_cast<int *>(smem + L::kNValidOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kAbortOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            // one consumer group releases a stage; QW = 3: the S and PV warps
            mbar_init(empty_bar(s), QW == 3 ? 2 : 4);
        }
        for (int s = 0; s < kQSlots; ++s) {
            mbar_init(qfull_bar(s), 1);
            mbar_init(qempty_bar(s), QW == 3 ? NCW + 2 : NCW);  // every warp that reads the hand-off
        }
        if (QW == 3) {
            for (int b = 0; b < 4; ++b) {
                mbar_init(s_full(b), 1);  // S warp
                mbar_init(s_free(b), 1);  // PV warp: the buffer's P has been read
                mbar_init(p_full(b), 4);  // the owning softmax team
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(o_done(b), 1);
                mbar_init(o_free(b), 4);
                mbar_init(qc_full(b), 1);
                mbar_init(qc_free(b), 1);
                mbar_init(qd_full(b), 1);
            }
        } else if (QW == 4) {
            for (int s = 0; s < 2; ++s) {  // one pair per consumer group
                mbar_init(merge_full(s), 4);
                mbar_init(merge_done(s), 4);
            }
        } else if (QW == 0) {
            for (int s = 0; s < MSLOTS; ++s) {
                mbar_init(merge_full(s), NCW);
                mbar_init(merge_done(s), NCW);
            }
        }
        for (int s = 0; s < kEpiRing; ++s) {
            mbar_init(epi_ready(s), NCW);
            mbar_init(epi_free(s), 1);
        }
        *epi_total = -1;
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    grid_launch_dependents();
    grid_dependency_wait();  // task map, lengths, pages and Q from earlier kernels
    EndStamp end_stamp{nullptr};
    if (p.cta_times) {  // uniform over the CTA
        uint64_t *t = p.cta_times + 2 * (blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
        if (threadIdx.x == 0) t[0] = t[1] = globaltimer_ns();
        __syncthreads();
        end_stamp.at = t + 1;
    }

    // ---- this CTA's work
    int d_begin = 0, d_count = 1, st0 = 0, st1 = 0;
    if (PERSIST) {
        d_begin = p.cta_desc_begin[blockIdx.x];
        d_count = p.cta_desc_begin[blockIdx.x + 1] - d_begin;
        if (FUSE && warp == NCW + 1) {
            // units with no tiles have no descriptor: their output is 0 and their LSE -inf
            for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
                if (p.unit_num_partials[u] != 0) continue;
                const int b = u / p.hkv, h = u - b * p.hkv;
                for (int i = lane; i < G * (kHeadDim / 4); i += 32) {
                    const int64_t orow = static_cast<int64_t>(b) * p.hq + h * G + i / (kHeadDim / 4);
                    store_out4<float>(p.out, orow, i % (kHeadDim / 4), make_float4(0.f, 0.f, 0.f, 0.f), p.out_bf16);
                    if (i % (kHeadDim / 4) == 0 && p.out_lse) p.out_lse[orow] = -INFINITY;
                }
            }
        }
        if (d_count <= 0) return;
    } else {
        const int b = blockIdx.z;
        int len = p.seq_lens[b];
        if (len < 0) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(p.status, DSA_DEV_BAD_SEQLEN);
            len = 0;
        }
        const int n = len / kTile + (len % kTile != 0);
        const int c = p.static_mode == 0 ? (n + p.num_splits - 1) / p.num_splits : p.static_tiles;
        st0 = min(static_cast<int>(blockIdx.x) * c, n);
        st1 = min(st0 + c, n);
        if (p.static_mode == 1 && blockIdx.x == p.num_splits - 1 && n > st1 && threadIdx.x == 0)
            atomicOr(p.status, DSA_DEV_BAD_SEQLEN);  // grid too small for this request
        if (st0 >= st1) {  // empty split: o = 0, lse = -inf
            const int slot = (b * p.hkv + blockIdx.y) * p.num_splits + blockIdx.x;
            for (int i = threadIdx.x; i < G * kHeadDim; i += blockDim.x)
                p.partial_o[static_cast<int64_t>(slot) * G * kHeadDim + i] = 0.f;
            if (threadIdx.x < G) p.partial_lse[static_cast<int64_t>(slot) * G + threadIdx.x] = -INFINITY;
            return;
        }
    }

    if (warp == NCW) {
        // =========================== producer warp ===========================
        // The CTA's descriptors are read 32 at a time (one per lane, with their
        // lengths and Q scales); their tiles form one stream, mapped 32 at a time
        // onto lanes, whose page ids are fetched one chunk ahead of the chunk whose
        // TMA copies are being issued.  Lane 0 issues; the warp stays converged.
        if (lane == 0) {
            prefetch_tmap(&kmap);
            prefetch_tmap(&vmap);
        }
        const uint64_t policy = policy_evict_first();
        int c = 0;          // tiles issued so far (ring position)
        int qi = 0;         // descriptors handed to the consumers
        int q_issued = -1;  // hand-off index of the last Q copy issued
        bool aborted = false;
        for (int wbase = 0; wbase < d_count && !aborted; wbase += 32) {
            // ---- window: descriptor wbase + lane
            int wb = 0, wh = 0, wt0 = 0, wn = 0, wslot = 0, wlen = 0, wnp = 1, wpbeg = 0;
            float wqs[kMaxGroup];
#pragma unroll
            for (int g = 0; g < kMaxGroup; ++g) wqs[g] = 0.f;
            if (wbase + lane < d_count) {
                const Desc x = get_desc<PERSIST>(p, d_begin, wbase + lane, st0, st1);
                if (x.ok) {
                    wb = x.u / p.hkv;
                    wh = x.u - wb * p.hkv;
                    wt0 = x.t0;
                    wn = x.t1 - x.t0;
                    wslot = x.slot;
                    wlen = p.seq_lens[wb];
                    if (FUSE) {
                        wnp = p.unit_num_partials[x.u];
                        wpbeg = p.unit_partial_begin[x.u];
                    }
                    if (wlen < 0 || wlen > p.max_pages * p.page_size) atomicOr(p.status, DSA_DEV_BAD_SEQLEN);
                    if (KV == 1) {
                        const float *qs = p.q_scale + static_cast<int64_t>(wb) * p.hq + wh * G;
#pragma unroll
                        for (int g = 0; g < kMaxGroup; ++g)
                            if (g < G) wqs[g] = qs[g];
                    }
                    if (wn == 0) {  // no tiles: its partials are empty, the consumers never see it
                        const int R = p.q_len * G;
                        const int64_t s0 = static_cast<int64_t>(wslot) * p.slots_per_desc;
                        for (int i = 0; i < p.slots_per_desc * R * kHeadDim; ++i)
                            p.partial_o[s0 * R * kHeadDim + i] = 0.f;
                        for (int g = 0; g < p.slots_per_desc * R; ++g) p.partial_lse[s0 * R + g] = -INFINITY;
                    }
                } else {
                    atomicOr(p.status, DSA_DEV_BAD_MAP);
                }
            }
            // stream offset of each descriptor in the window (exclusive scan of tile counts)
            int incl = wn;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int wstart = incl - wn;
            const int wtotal = __shfl_sync(0xffffffffu, incl, 31);

            // lane -> (descriptor, tile, page) for stream tile s0 + lane
            // a 64-token tile spans ppt pages of P tokens: pages t * ppt .. t * ppt + ppt - 1
            const int P = p.page_size, ppt = kTile / P;
            auto map_chunk = [&](int s0, int &j, int &t, int (&pg)[kMaxPagesPerTile]) {
                const int s = s0 + lane;
                j = 0;
#pragma unroll
                for (int step = 16; step > 0; step >>= 1) {
                    const int v = __shfl_sync(0xffffffffu, wstart, j + step);
                    if (v <= s) j += step;
                }
                t = __shfl_sync(0xffffffffu, wt0, j) + (s - __shfl_sync(0xffffffffu, wstart, j));
                const int bj = __shfl_sync(0xffffffffu, wb, j);
#pragma unroll
                for (int k = 0; k < kMaxPagesPerTile; ++k) {
                    const int idx = t * ppt + k;
                    pg[k] = -1;
                    if (k < ppt && s < wtotal && idx < p.max_pages)
                        pg[k] = p.block_table[static_cast<int64_t>(bj) * p.max_pages + idx];
                }
            };

            int cj = 0, ct = 0, cpg[kMaxPagesPerTile];
#pragma unroll
            for (int k = 0; k < kMaxPagesPerTile; ++k) cpg[k] = -1;
            if (wtotal > 0) map_chunk(0, cj, ct, cpg);
            for (int s0 = 0; s0 < wtotal && !aborted; s0 += 32) {
                int nj = 0, nt = 0, npg[kMaxPagesPerTile];
#pragma unroll
                for (int k = 0; k < kMaxPagesPerTile; ++k) npg[k] = -1;
                if (s0 + 32 < wtotal) map_chunk(s0 + 32, nj, nt, npg);  // next chunk's page ids in flight
                const int cnt = min(32, wtotal - s0);
                // ---- per-lane view of this lane's own tile (stream tile s0 + lane)
                const int h_l = __shfl_sync(0xffffffffu, wh, cj);
                const int len_l = __shfl_sync(0xffffffffu, wlen, cj);
                const int t0_l = __shfl_sync(0xffffffffu, wt0, cj);
                const bool first_l = lane < cnt && ct == t0_l;
                int nv_l = 0;
                if (lane < cnt) {
                    const bool len_ok = len_l >= 0 && len_l <= p.max_pages * P;
                    nv_l = len_ok ? min(kTile, len_l - ct * kTile) : 0;
                    if (nv_l < 0 || ct * ppt >= p.max_pages) nv_l = 0;
                    // the pages holding the tile's valid tokens must be inside the pool
                    bool bad = false;
#pragma unroll
                    for (int k = 0; k < kMaxPagesPerTile; ++k)
                        if (k * P < nv_l && (cpg[k] < 0 || cpg[k] >= p.num_pages)) bad = true;
                    if (nv_l > 0 && bad) {
                        atomicOr(p.status, DSA_DEV_BAD_PAGE);
                        nv_l = 0;
                    }
                }
                const uint32_t starts = __ballot_sync(0xffffffffu, first_l);
                // ---- one converged loop over the chunk.  Lane l issues its tile the moment
                //      its ring stage is free, once the tile STAGES positions earlier has been
                //      issued (so the parity it tests names exactly the release it needs);
                //      descriptors starting in the chunk are handed to the consumers in order,
                //      each as soon as a hand-off slot is free.  Nothing waits in a divergent
                //      loop: lanes spinning on their own barriers starved one another.
                bool pend = lane < cnt;
                uint32_t todo = starts;  // descriptor starts not yet handed off
                const int cl = c + lane;
                const int stage = cl % STAGES;
                const uint32_t epar = ((cl / STAGES) & 1) ^ 1;
                uint64_t idle_t0 = globaltimer_ns();  // last progress
                for (uint32_t it = 1;; ++it) {
                    const uint32_t done = __ballot_sync(0xffffffffu, !pend);
                    if (done == 0xffffffffu && todo == 0) break;
                    bool progress = false;
                    int hand = 0;  // a hand-off slot is free for the next descriptor
                    if (todo && lane == 0) hand = mbar_test_wait(qempty_bar(qi % kQSlots), ((qi / kQSlots) & 1) ^ 1);
                    if (__shfl_sync(0xffffffffu, hand, 0)) {
                        // next descriptor to hand off starts at chunk lane k
                        const int k = __ffs(todo) - 1;
                        const int j = __shfl_sync(0xffffffffu, cj, k);
                        float qs[kMaxGroup];
#pragma unroll
                        for (int g = 0; g < kMaxGroup; ++g) qs[g] = __shfl_sync(0xffffffffu, wqs[g], j);
                        const int b = __shfl_sync(0xffffffffu, wb, j);
                        const int h = __shfl_sync(0xffffffffu, wh, j);
                        const int n = __shfl_sync(0xffffffffu, wn, j);
                        const int slot = __shfl_sync(0xffffffffu, wslot, j);
                        const int np = __shfl_sync(0xffffffffu, wnp, j);
                        const int pbeg = __shfl_sync(0xffffffffu, wpbeg, j);
                        const int dt0 = __shfl_sync(0xffffffffu, wt0, j);
                        const int dlen = __shfl_sync(0xffffffffu, wlen, j);
                        const int qs_ = qi % kQSlots;
                        if (lane == 0) {
                            const int c_desc = c + k;  // ring position of the descriptor's first tile
                            DescInfo *inf = reinterpret_cast<DescInfo *>(smem + L::kInfoOff) + qs_;
                            inf->end = 0;
                            inf->b = b;
                            inf->h = h;
                            inf->n = n;
                            inf->slot = slot;
                            inf->c_start = c_desc;
                            inf->np = np;
                            inf->pbeg = pbeg;
                            inf->t0 = dt0;
                            inf->len = dlen;
#pragma unroll
                            for (int g = 0; g < kMaxGroup; ++g) inf->qscale[g] = qs[g];
                            // the G query rows of each of the request's q_len query tokens,
                            // one after the other (row i*G + g)
                            if (QW == 3) {  // the S warp fetches Q itself, a descriptor ahead
                                mbar_arrive(qfull_bar(qs_));
                            } else {
                                const uint32_t bytes = G * C::kQHeadBytes;
                                mbar_arrive_expect_tx(qfull_bar(qs_), bytes * p.q_len);
                                for (int i = 0; i < p.q_len; ++i) {
                                    const uint8_t *src = p.q + ((static_cast<int64_t>(b) * p.q_len + i) * p.hq + h * G) *
                                                                   C::kQHeadBytes;
                                    bulk_load(sbase + L::kQOff + qs_ * L::kQSlot + i * bytes, src, bytes,
                                              qfull_bar(qs_));
                                }
                                q_issued = qi;
                            }
                        }
                        ++qi;
                        todo &= todo - 1;
                        progress = true;
                    }
                    // a lane may test its stage once the tile STAGES positions earlier is issued
                    const bool ready = pend && (lane < STAGES || ((done >> (lane - STAGES)) & 1u));
                    if (ready && mbar_test_wait(empty_bar(stage), epar)) {
                        pend = false;
                        nvalid[stage] = nv_l;
                        const uint32_t fb = full_bar(stage);
                        if (nv_l > 0) {
                            const uint32_t kdst = sbase + stage * L::kStageBytes;
                            const uint32_t vdst = kdst + C::kTileBytes;
                            // the pages holding valid tokens, one box of P rows each (both 128-B
                            // halves of a bf16 row: the stage is [page][half][P rows][128 B]);
                            // the tensor-core kernel's operands want [half][64 rows][128 B],
                            // so there each half of a page smaller than the tile is its own box
                            if (P == kTile) {  // one page per tile: the common case, no loop
                                mbar_arrive_expect_tx(fb, L::kStageTx);
                                tma_load_5d(kdst, &kmap, fb, 0, 0, 0, h_l, cpg[0], policy);
                                tma_load_5d(vdst, &vmap, fb, 0, 0, 0, h_l, cpg[0], policy);
                                if (KV == 1) {
                                    const int64_t srow = (static_cast<int64_t>(cpg[0]) * p.hkv + h_l) * kTile;
                                    bulk_load(vdst + C::kTileBytes, p.k_scale + srow, C::kScaleBytes, fb);
                                    bulk_load(vdst + C::kTileBytes + C::kScaleBytes, p.v_scale + srow, C::kScaleBytes, fb);
                                }
                            } else {
                                const int nsub = (nv_l + P - 1) / P;
                                mbar_arrive_expect_tx(fb, nsub * (L::kStageTx / ppt));
#pragma unroll
                                for (int k = 0; k < kMaxPagesPerTile; ++k) {
                                    if (k >= nsub) break;
                                    const int pg = cpg[k];
                                    if (QW == 3 && KV == 0 && P < kTile) {
                                        const uint32_t ro = static_cast<uint32_t>(k * P) * 128u;
                                        tma_load_5d(kdst + ro, &kmap, fb, 0, 0, 0, h_l, pg, policy);
                                        tma_load_5d(kdst + C::kTileBytes / 2 + ro, &kmap, fb, 0, 0, 1, h_l, pg, policy);
                                        tma_load_5d(vdst + ro, &vmap, fb, 0, 0, 0, h_l, pg, policy);
                                        tma_load_5d(vdst + C::kTileBytes / 2 + ro, &vmap, fb, 0, 0, 1, h_l, pg, policy);
                                    } else {
                                        const uint32_t ro = static_cast<uint32_t>(k * P) * (C::kTileBytes / kTile);
                                        tma_load_5d(kdst + ro, &kmap, fb, 0, 0, 0, h_l, pg, policy);
                                        tma_load_5d(vdst + ro, &vmap, fb, 0, 0, 0, h_l, pg, policy);
                                    }
                                    if (KV == 1) {
                                        const int64_t srow = (static_cast<int64_t>(pg) * p.hkv + h_l) * P;
                                        bulk_load(vdst + C::kTileBytes + 4 * k * P, p.k_scale + srow, 4 * P, fb);
                                        bulk_load(vdst + C::kTileBytes + C::kScaleBytes + 4 * k * P, p.v_scale + srow,
                                                  4 * P, fb);
                                    }
                                }
                            }
                        } else {
                            mbar_arrive(fb);
                        }
                    }
                    if (__any_sync(0xffffffffu, ready && !pend)) progress = true;
                    if (progress) {
                        idle_t0 = globaltimer_ns();
                    } else if ((it & 31u) == 0) {  // bounded wait
                        int ab = 0;
                        if (lane == 0) {
                            if (*abort_flag) {
                                ab = 1;
                            } else if (globaltimer_ns() - idle_t0 > kWaitLimitNs) {
                                atomicOr(p.status, DSA_DEV_TIMEOUT);
                                *abort_flag = 1;
                                ab = 1;
                            }
                        }
                        if (__shfl_sync(0xffffffffu, ab, 0)) {
                            aborted = true;
                            break;
                        }
                    }
                }
                if (aborted) {
                    // tiles up to the last one issued are counted for the drain below
                    const uint32_t done = __ballot_sync(0xffffffffu, !pend && lane < cnt);
                    c += done ? 32 - __clz(done) : 0;
                    break;
                }
                c += cnt;
                cj = nj;
                ct = nt;
#pragma unroll
                for (int k = 0; k < kMaxPagesPerTile; ++k) cpg[k] = npg[k];
            }
        }
        if (FUSE && lane == 0) *epi_total = qi;  // descriptors handed off (the epilogue's count)
        if (!aborted && lane == 0) {
            // end marker for the consumers
            if (wait_phase(qempty_bar(qi % kQSlots), ((qi / kQSlots) & 1) ^ 1, abort_flag, p.status)) {
                reinterpret_cast<DescInfo *>(smem + L::kInfoOff)[qi % kQSlots].end = 1;
                mbar_arrive(qfull_bar(qi % kQSlots));
            } else {
                aborted = true;
            }
        }
        if (aborted && lane == 0) {
            // let every copy this CTA started land before the CTA exits
            const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
            for (int cc = max(0, c - STAGES); cc < c; ++cc)
                drain_phase(full_bar(cc % STAGES), (cc / STAGES) & 1, deadline);
            if (q_issued >= 0) drain_phase(qfull_bar(q_issued % kQSlots), (q_issued / kQSlots) & 1, deadline);
        }
        return;
    }

    if (FUSE && warp == NCW + 1) {
        // =========================== epilogue warp (fused combine) ===========================
        // Follows the consumers' merges in order.  For a unit with several partials it
        // publishes the merged partial at gpu scope (the consumers' writes, ordered by the
        // epi_ready barrier, are covered by this warp's release) and counts it; the warp that
        // completes the unit's count merges all its partials.  epi_free bounds its lag to
        // kEpiRing descriptors.
        for (int d = 0;; ++d) {
            const int er = d % kEpiRing;
            bool have = false;
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t it = 0;; ++it) {
                if (mbar_try_wait(epi_ready(er), (d / kEpiRing) & 1)) {
                    have = true;
                    break;
                }
                const int tot = *epi_total;
                if ((tot >= 0 && d >= tot) || *abort_flag) break;
                if ((it & 31u) == 31u && globaltimer_ns() - t0 > kWaitLimitNs) {
                    if (lane == 0) atomicOr(p.status, DSA_DEV_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
            }
            if (!have) return;
            const EpiRecord r = epi_rec[er];
            if (r.np > 1) {
                const int u = r.b * p.hkv + r.h;
                int prev = 0;
                if (lane == 0) {
                    fence_acq_rel_gpu();
                    prev = atomicAdd(p.unit_counters + u, 1);
                }
                prev = __shfl_sync(0xffffffffu, prev, 0);
                if (prev == r.np - 1) {  // every partial of the unit is published
                    fence_acq_rel_gpu();
                    combine_unit(p, lane, r.b, r.h, r.np, r.pbeg);
                    if (lane == 0) p.unit_counters[u] = 0;  // ready for the next step
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(epi_free(er));
        }
    }

    if constexpr (QW == 3) {
        // ============ multi-token queries on the 5th-generation tensor cores ============
        // Rows r = i * G + g (query token i, head g), r < R = q_len * G <= 64.  Per tile:
        //   S[64 x 64] = Qc . K^T in one of two 64-column TMEM buffers (M = 64: row r sits in
        //   lane 32 (r / 16) + r % 16, i.e. lanes 0-15 of each warp's 32-lane quarter);
        //   the softmax thread of row r (lane r % 16 of warp r / 16) masks it (causal within
        //   the draft, past the length), keeps the running max m, raised lazily (O is
        //   rescaled only when the max grows by more than 8 in base 2), and writes P =
        //   2^(s - m) as bf16 high and low parts;
        //   O[64 x 128] += P_hi . V + P_lo . V in TMEM columns 128-255.
        // Two warps issue the products: the S warp runs ahead (two S buffers) as stages land,
        // the PV warp follows the softmax; each releases its half of a ring stage (K, V) when
        // its products have read it, so the softmax of tile g overlaps the products of its
        // neighbours and no product waits for an unrelated load.
        const int R = p.q_len * G;
        uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kAbortOff + 4);
        constexpr int kTcThreads = (NCW + 2) * 32;  // softmax warps, S warp, PV warp
        constexpr uint32_t kQcBuf = kMaxRows * C::kQHeadBytes;
        if (warp == NCW + 1) tmem_alloc(smem_u32(tmem_slot), 512);
        tc_fence_before();
        named_bar_sync(1, kTcThreads);
        tc_fence_after();
        const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
        // Q K-major, K K-major (bf16, or E4M3 with kind::f8f6f4); P K-major, V M/N-major
        // (bf16, or f16 for E4M3 K/V: V widened exactly, P carrying the V scale)
        constexpr uint32_t kIdS = KV == 0 ? umma_idesc_bf16(64, 64, 0, 0) : umma_idesc_fmt0(64, 64, 0, 0);
        constexpr uint32_t kIdO = KV == 0 ? umma_idesc_bf16(64, 128, 0, 1) : umma_idesc_fmt0(64, 128, 0, 1);
        bool failed = false;

        if (warp == NCW + 1) {
            // ---- S warp: fetches each descriptor's Q rows one descriptor ahead (plain rows
            //      into one of two buffers), lays them out as the A operand (zero past R), then
            //      issues S = Q K^T for its tiles as soon as a stage and an S buffer are ready
            //      (lane 0 issues, the warp waits together); its commit on the stage's empty
            //      barrier says the K half is no longer read
            // descriptors of this CTA, 32 at a time: lane j holds the unit of descriptor wbase + j
            // if the producer hands it over (valid, with tiles), else -1
            int wbase = 0, wu = -1;
            auto load_window = [&](int base) {
                wbase = base;
                wu = -1;
                if (base + lane < d_count) {
                    const int4 v = p.descs[d_begin + base + lane];
                    if (v.x >= 0 && v.x < p.num_units && v.y >= 0 && v.y < v.z && d_begin + base + lane < p.max_slots)
                        wu = v.x;
                }
            };
            load_window(0);
            auto next_desc = [&](int after) {  // the next handed-over descriptor (raw slot) after `after`
                for (int rel = after - d_begin + 1; rel < d_count;) {
                    if (rel < wbase || rel >= wbase + 32) load_window(rel & ~31);
                    const uint32_t m = __ballot_sync(0xffffffffu, wu >= 0) & (~0u << (rel - wbase));
                    if (m) return d_begin + wbase + __ffs(m) - 1;
                    rel = wbase + 32;
                }
                return -1;
            };
            int fetched[2] = {0, 0};  // Q copies issued into each plain buffer (each one waited for)
            auto fetch_q = [&](int x, int j) {  // x in the current window
                const int u = __shfl_sync(0xffffffffu, wu, x - d_begin - wbase);
                if (lane == 0) {
                    const int b = u / p.hkv, h = u - b * p.hkv;
                    const uint32_t bytes = G * C::kQHeadBytes;
                    mbar_arrive_expect_tx(qd_full(j), bytes * p.q_len);
                    for (int i = 0; i < p.q_len; ++i)
                        bulk_load(sbase + L::kQOff + j * L::kQSlot + i * bytes,
                                  p.q + ((static_cast<int64_t>(b) * p.q_len + i) * p.hq + h * G) * C::kQHeadBytes, bytes,
                                  qd_full(j));
                }
                ++fetched[j];
            };
            auto land_q = [&](int j) { return wait_phase(qd_full(j), (fetched[j] - 1) & 1, abort_flag, p.status); };
            int pf_slot = next_desc(d_begin - 1), pf_buf = 0;  // the descriptor whose Q is in flight
            if (pf_slot >= 0) fetch_q(pf_slot, 0);
            int g = 0, last_d = -1;
            for (int d = 0;; ++d) {
                const int qslot = d % kQSlots;
                if (!wait_phase(qfull_bar(qslot), (d / kQSlots) & 1, abort_flag, p.status)) {
                    failed = true;
                    break;
                }
                const DescInfo *inf = reinterpret_cast<const DescInfo *>(smem + L::kInfoOff) + qslot;
                const int end = inf->end, n = inf->n, c_start = inf->c_start, xs = inf->slot;
                if (!end) {
                    // this descriptor's Q: normally the prefetched one; otherwise fetched now
                    const int qb = pf_buf;
                    if (pf_slot != xs) {
                        if (pf_slot >= 0 && !land_q(qb)) {
                            failed = true;
                            break;
                        }
                        if (xs < d_begin + wbase || xs >= d_begin + wbase + 32) load_window((xs - d_begin) & ~31);
                        fetch_q(xs, qb);
                    }
                    if (!land_q(qb) || !wait_phase(qc_free(d & 1), ((d >> 1) & 1) ^ 1, abort_flag, p.status)) {
                        pf_slot = -1;  // consumed (or abandoned with the CTA)
                        failed = true;
                        break;
                    }
                    const uint8_t *src = smem + L::kQOff + qb * L::kQSlot;
                    uint8_t *dst = smem + L::kQcOff + (d & 1) * kQcBuf;
                    if constexpr (KV == 0) {
                    // 128-byte-swizzled K-major operand (as the TMA lays out K): dims 64 b .. 64 b + 63
                    // of row r at b * 8 KB + r * 128 B, 16-byte chunk c at (c ^ (r % 8)) * 16.  Each
                    // quarter-warp writes one 128-byte row: no bank conflicts either way.
#pragma unroll
                    for (int rd = 0; rd < 4; ++rd) {
                        uint4 v[8];
#pragma unroll
                        for (int it = 0; it < 8; ++it) {  // chunk kc of row r
                            const int i = lane + 32 * (8 * rd + it), r = i >> 4, kc = i & 15;
                            v[it] = r < R ? *reinterpret_cast<const uint4 *>(src + r * (kHeadDim * 2) + kc * 16)
                                          : make_uint4(0u, 0u, 0u, 0u);
                        }
#pragma unroll
                        for (int it = 0; it < 8; ++it) {
                            const int i = lane + 32 * (8 * rd + it), r = i >> 4, kc = i & 15;
                            *reinterpret_cast<uint4 *>(dst + (kc >> 3) * 8192 + r * 128 + (((kc & 7) ^ (r & 7)) << 4)) = v[it];
                        }
                    }
                    } else {
                    // E4M3: a row is one 128-byte swizzle row (r * 128 B, chunk c at (c ^ (r % 8)) * 16)
#pragma unroll
                    for (int rd = 0; rd < 2; ++rd) {
                        uint4 v[8];
#pragma unroll
                        for (int it = 0; it < 8; ++it) {  // chunk kc of row r
                            const int i = lane + 32 * (8 * rd + it), r = i >> 3, kc = i & 7;
                            v[it] = r < R ? *reinterpret_cast<const uint4 *>(src + r * kHeadDim + kc * 16)
                                          : make_uint4(0u, 0u, 0u, 0u);
                        }
#pragma unroll
                        for (int it = 0; it < 8; ++it) {
                            const int i = lane + 32 * (8 * rd + it), r = i >> 3, kc = i & 7;
                            *reinterpret_cast<uint4 *>(dst + r * 128 + ((kc ^ (r & 7)) << 4)) = v[it];
                        }
                    }
                    }
                    fence_proxy_async_smem();
                    // the next descriptor's Q lands while this one's tiles are worked on
                    pf_slot = next_desc(xs);
                    if (pf_slot >= 0) {
                        pf_buf = qb ^ 1;
                        fetch_q(pf_slot, pf_buf);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty_bar(qslot));
                if (end) break;
                const uint32_t qa = sbase + L::kQcOff + (d & 1) * kQcBuf;
                for (int li = 0; li < n; ++li, ++g) {
                    const int c = c_start + li, stage = c % STAGES, buf = g & 3;
                    if (!wait_phase(full_bar(stage), (c / STAGES) & 1, abort_flag, p.status) ||
                        !wait_phase(s_free(buf), ((g >> 2) & 1) ^ 1, abort_flag, p.status)) {
                        failed = true;
                        break;
                    }
                    const int nv = nvalid[stage];
                    if (lane == 0) {
                        if (nv > 0) {
                            tc_fence_after();
                            const uint32_t kb = sbase + stage * L::kStageBytes;
                            if constexpr (KV == 0) {
#pragma unroll
                                for (int ks = 0; ks < 8; ++ks)
                                    umma_bf16(tmem + 64 * buf, umma_desc(qa + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, 2),
                                              umma_desc(kb + (ks >> 2) * (C::kTileBytes / 2) + (ks & 3) * 32, 16, 1024, 2),
                                              kIdS, ks > 0);
                            } else {  // E4M3: 32 dims (32 bytes) per product
#pragma unroll
                                for (int ks = 0; ks < 4; ++ks)
                                    umma_e4m3(tmem + 64 * buf, umma_desc(qa + ks * 32, 16, 1024, 2),
                                              umma_desc(kb + ks * 32, 16, 1024, 2), kIdS, ks > 0);
                            }
                            umma_commit(s_full(buf));
                            umma_commit(empty_bar(stage));
                        } else {
                            mbar_arrive(s_full(buf));
                            mbar_arrive(empty_bar(stage));
                        }
                    }
                    __syncwarp();
                }
                if (failed) break;
                if (lane == 0) umma_commit(qc_free(d & 1));  // the descriptor's S products have read Qc
                __syncwarp();
                last_d = d;
            }
            // the last commit lands once every product this warp issued has completed; a Q copy
            // still in flight lands before the CTA leaves
            if (!failed && last_d >= 0) wait_phase(qc_free(last_d & 1), (last_d >> 1) & 1, abort_flag, p.status);
            if (pf_slot >= 0) {
                const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
                drain_phase(qd_full(pf_buf), (fetched[pf_buf] - 1) & 1, deadline);
            }
        } else if (warp == NCW + 2) {
            // ---- PV warp: O += P_hi . V + P_lo . V as soon as the softmax warps hand P over;
            //      its commit on the stage's empty barrier says the V half is no longer read
            int g = 0;
            for (int d = 0;; ++d) {
                const int qslot = d % kQSlots;
                if (!wait_phase(qfull_bar(qslot), (d / kQSlots) & 1, abort_flag, p.status)) {
                    failed = true;
                    break;
                }
                const DescInfo *inf = reinterpret_cast<const DescInfo *>(smem + L::kInfoOff) + qslot;
                const int end = inf->end, n = inf->n, c_start = inf->c_start;
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty_bar(qslot));
                if (end) break;
                bool first_pv[2] = {true, true};  // per softmax team (tile parity): O_t not yet written
                for (int li = 0; li < n; ++li, ++g) {
                    const int c = c_start + li, stage = c % STAGES, buf = g & 3, t = g & 1;
                    if (!wait_phase(full_bar(stage), (c / STAGES) & 1, abort_flag, p.status) ||
                        !wait_phase(p_full(buf), (g >> 2) & 1, abort_flag, p.status)) {
                        failed = true;
                        break;
                    }
                    const int nv = nvalid[stage];
                    if (nv > 0) {
                        // O_t is free once team t has read out the previous descriptor's
                        if (first_pv[t] && !wait_phase(o_free(t), (d & 1) ^ 1, abort_flag, p.status)) {
                            failed = true;
                            break;
                        }
                        if (lane == 0) {
                            tc_fence_after();
                            // bf16: V as loaded, P high part in columns 0-31, low part in 32-63;
                            // E4M3: V widened to f16 by the softmax team, P (f16) in columns 0-31
                            const uint32_t vb = sbase + stage * L::kStageBytes + (KV == 0 ? C::kTileBytes : L::kVcOff);
                            const uint32_t pt = tmem + 64 * buf;
                            const uint32_t od = tmem + 256 + 128 * t;
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks) {
                                const uint64_t bd = umma_desc(vb + ks * 2048, 8192, 1024, 2);
                                umma_bf16_ta(od, pt + 8 * ks, bd, kIdO, !(first_pv[t] && ks == 0));
                                if (KV == 0) umma_bf16_ta(od, pt + 32 + 8 * ks, bd, kIdO, true);
                            }
                        }
                        first_pv[t] = false;
                    }
                    // commits, not arrives: a phase also means every earlier product is done
                    if (lane == 0) {
                        umma_commit(o_done(t));
                        umma_commit(s_free(buf));
                        umma_commit(empty_bar(stage));
                    }
                    __syncwarp();
                }
                if (failed) break;
            }
        } else {
            // ---- softmax warps: two teams of four (team t = warps 4t .. 4t + 3) take the tiles
            //      of parity t (S/P buffers t and t + 2 in turn, O_t).  Warp w reads the 16 rows
            //      16 (w & 3) .. + 15
            //      (M = 64 accumulators: lanes 0-15 of each sub-partition) as m16n8 fragments:
            //      thread (gid = lane / 4, tig = lane % 4) holds rows ra = 16 (w & 3) + gid and
            //      rb = ra + 8, columns 8 k + 2 tig, + 1; a row's max and sum combine over the
            //      four threads of its quad.  At each descriptor end each team writes its own
            //      partial (slot 2 x descriptor + team); the combine merges them with the others.
            const int team = warp >> 2, sp = warp & 3;
            const int gid = lane >> 2, tig = lane & 3;
            const int ra = 16 * sp + gid, rb = ra + 8;
            const uint32_t lane_base = static_cast<uint32_t>(32 * sp) << 16;
            const uint32_t o_col = 256 + 128 * team;
            const int tid = sp * 32 + lane;  // within the team
            // The descriptor end of a team (its partial, slot 2 x descriptor + team), deferred
            // until the team has handed over the P of its first tile of the next descriptor: a
            // descriptor's first tile never rescales O, so it need not wait for the previous
            // descriptor's last P.V, and the team computes it while that P.V completes.
            float ep_vref = 1.f;  // E4M3: the V scale reference of the deferred descriptor end
            auto team_epilogue = [&](int slot, float (&m)[2], float (&l)[2], int pv_desc, int last_g) -> bool {
                // ---- this team's products of the descriptor are done once its last tile's buffer
                //      phase is (that commit covers every earlier product)
                if (last_g >= 0) {
                    if (!wait_phase(o_done(team), (last_g >> 1) & 1, abort_flag, p.status)) return false;
                    tc_fence_after();
                }
                // ---- this team's partial (slot 2 x descriptor + team): O_t / l, lse = ln(2) (m + log2 l)
                float inv[2], lse[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
                    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
                    if constexpr (KV == 0)
                        inv[h] = l[h] > 0.f ? 1.f / l[h] : 0.f;
                    else
                        inv[h] = l[h] > 0.f ? ep_vref / l[h] : 0.f;
                    lse[h] = l[h] > 0.f ? (m[h] + lg2(l[h])) * kLn2 : -INFINITY;
                }
                const int64_t slot_row = (2 * static_cast<int64_t>(slot) + team) * R;
                float *dst_a = p.partial_o + (slot_row + ra) * kHeadDim + 2 * tig;
                float *dst_b = p.partial_o + (slot_row + rb) * kHeadDim + 2 * tig;
                // O_t into registers first, then release it for the next descriptor's products
                float o[16][4];
                if (pv_desc > 0) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) tmem_ld16x8(tmem + lane_base + o_col + 8 * k, o[k]);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int k = 0; k < 16; ++k) o[k][0] = o[k][1] = o[k][2] = o[k][3] = 0.f;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free(team));
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    if (ra < R) *reinterpret_cast<float2 *>(dst_a + 8 * k) = make_float2(o[k][0] * inv[0], o[k][1] * inv[0]);
                    if (rb < R) *reinterpret_cast<float2 *>(dst_b + 8 * k) = make_float2(o[k][2] * inv[1], o[k][3] * inv[1]);
                }
                if (tig == 0) {
                    if (ra < R) p.partial_lse[slot_row + ra] = lse[0];
                    if (rb < R) p.partial_lse[slot_row + rb] = lse[1];
                }
                return true;
            };
            bool ep_pending = false;
            int ep_slot = 0, ep_pv = 0, ep_last_g = -1;
            float ep_m[2] = {0.f, 0.f}, ep_l[2] = {0.f, 0.f};
            auto flush_epilogue = [&]() -> bool {
                if (!ep_pending) return true;
                ep_pending = false;
                return team_epilogue(ep_slot, ep_m, ep_l, ep_pv, ep_last_g);
            };
            int g = 0;
            for (int d = 0;; ++d) {
                const int qslot = d % kQSlots;
                if (!wait_phase(qfull_bar(qslot), (d / kQSlots) & 1, abort_flag, p.status)) {
                    failed = true;
                    break;
                }
                const DescInfo *inf = reinterpret_cast<const DescInfo *>(smem + L::kInfoOff) + qslot;
                const int end = inf->end, n = inf->n, slot = inf->slot, c_start = inf->c_start;
                const int dt0 = inf->t0, len = inf->len;
                int d_b = 0, d_h = 0;
                if constexpr (KV == 1) d_b = inf->b, d_h = inf->h;
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty_bar(qslot));
                if (end) {
                    if (!flush_epilogue()) failed = true;
                    break;
                }
                // visible tokens of each row: t < lim (-1: a row past R)
                const int lim[2] = {ra < R ? len - p.q_len + ra / G + 1 : -1, rb < R ? len - p.q_len + rb / G + 1 : -1};
                float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
                // E4M3: score factor per row (softmax scale x the row's q_scale), the V scale
                // reference (the largest V scale seen, O holds the output divided by it) and its inverse
                float qsc[2] = {p.score_scale, p.score_scale}, vref = 1.f, vinv = 1.f;
                if constexpr (KV == 1) {
                    const int rr[2] = {ra, rb};
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (rr[h] < R) {
                            const int i = rr[h] / G;
                            qsc[h] *= p.q_scale[(static_cast<int64_t>(d_b) * p.q_len + i) * p.hq + d_h * G + rr[h] - i * G];
                        }
                    vref = vinv = 0.f;
                }
                int pv_desc = 0, last_g = -1;
                for (int li = 0; li < n; ++li, ++g) {
                    if ((g & 1) != team) continue;
                    const int c = c_start + li, stage = c % STAGES, buf = g & 3;
                    if (!wait_phase(full_bar(stage), (c / STAGES) & 1, abort_flag, p.status) ||
                        !wait_phase(s_full(buf), (g >> 2) & 1, abort_flag, p.status)) {
                        failed = true;
                        break;
                    }
                    const int nv = nvalid[stage];
                    tc_fence_after();
                    float sv[8][4];  // [column block k][(ra, 2tig), (ra, 2tig+1), (rb, 2tig), (rb, 2tig+1)]
                    if (nv > 0) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) tmem_ld16x8(tmem + lane_base + 64 * buf + 8 * k, sv[k]);
                        tmem_wait_ld();
                    }
                    // this team's previous tile of the descriptor (-1: none; the first tile starts
                    // from m = -inf and never rescales O).  Its P.V is waited for before this tile's
                    // P is handed over (so the team stays within one phase of o_done, which the
                    // descriptor end's wait needs), and before a rescale of O, which reads O.  (S of
                    // this tile was issued after the P.V two team tiles back had released its
                    // buffer, so until this tile's P is handed over the barrier is at most one
                    // phase behind the one waited for.)
                    const int prev_g = last_g;
                    last_g = g;
                    auto wait_prev_pv = [&]() {
                        return prev_g < 0 || wait_phase(o_done(team), ((g >> 1) & 1) ^ 1, abort_flag, p.status);
                    };
                    if (nv == 0) {  // no data in this stage: the PV warp skips its P.V
                        if (!wait_prev_pv()) {
                            failed = true;
                            break;
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(p_full(buf));
                        if (!flush_epilogue()) {
                            failed = true;
                            break;
                        }
                        continue;
                    }
                    // ---- E4M3: S times the K scale of its column; P's factor per column, the V
                    //      scale over the reference, which moves only when a larger scale appears
                    //      (O is then rescaled with the maxima below); columns past nv get 0
                    float vw[8][2];
                    float vf = 1.f;
                    if constexpr (KV == 1) {
                        const float *ksm = reinterpret_cast<const float *>(smem + stage * L::kStageBytes + 2 * C::kTileBytes);
                        const float *vsm = ksm + kTile;
                        float vmax = 0.f;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int j = 8 * k + 2 * tig;
                            const float2 kk = *reinterpret_cast<const float2 *>(ksm + j);
                            const float2 vv = *reinterpret_cast<const float2 *>(vsm + j);
                            sv[k][0] *= kk.x;
                            sv[k][1] *= kk.y;
                            sv[k][2] *= kk.x;
                            sv[k][3] *= kk.y;
                            vw[k][0] = j < nv ? vv.x : 0.f;
                            vw[k][1] = j + 1 < nv ? vv.y : 0.f;
                            vmax = fmaxf(vmax, fmaxf(vw[k][0], vw[k][1]));
                        }
                        if (__any_sync(0xffffffffu, vmax > vref)) {  // the quad's four lanes cover the 64 columns
                            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 1));
                            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));
                            if (vmax > vref) {
                                if (vref > 0.f) vf = vref / vmax;  // from 0: nothing accumulated yet
                                vref = vmax;
                                vinv = 1.f / vmax;
                            }
                        }
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            vw[k][0] *= vinv;
                            vw[k][1] *= vinv;
                        }
                    }
                    // ---- running maximum over each row's visible tokens (t < lim, slot < nv)
                    const int tt = (dt0 + li) * kTile;
                    const int vis[2] = {max(0, min(nv, lim[0] - tt)), max(0, min(nv, lim[1] - tt))};
                    const bool full = vis[0] == kTile && vis[1] == kTile;
                    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                    for (int k = 0; k < 8; ++k)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int h = e >> 1, j = 8 * k + 2 * tig + (e & 1);
                            mx[h] = fmaxf(mx[h], (full || j < vis[h]) ? sv[k][e] : -INFINITY);
                        }
                    bool grow[2];
                    float alpha[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
                        const float mnew = fmaxf(m[h], mx[h] * (KV == 0 ? p.score_scale : qsc[h]));
                        grow[h] = m[h] != -INFINITY && mnew > m[h] + 8.f;
                        alpha[h] = grow[h] ? ex2(m[h] - mnew) : 1.f;
                        if (grow[h] || m[h] == -INFINITY) m[h] = mnew;
                    }
                    if (__any_sync(0xffffffffu, grow[0] || grow[1] || (KV == 1 && vf != 1.f))) {
                        // rows whose maximum grew: O_team *= 2^(m_old - m_new); E4M3: all rows also
                        // by the V scale reference's change (after the previous P.V into O_team)
                        if (!wait_prev_pv()) {
                            failed = true;
                            break;
                        }
                        tc_fence_after();
#pragma unroll 1  // rare: kept small for the instruction cache
                        for (int half = 0; half < 2; ++half) {
                            float o[8][4];
#pragma unroll
                            for (int k = 0; k < 8; ++k) tmem_ld16x8(tmem + lane_base + o_col + 64 * half + 8 * k, o[k]);
                            tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                if constexpr (KV == 0) {
                                    o[k][0] *= alpha[0];
                                    o[k][1] *= alpha[0];
                                    o[k][2] *= alpha[1];
                                    o[k][3] *= alpha[1];
                                } else {
                                    o[k][0] *= alpha[0] * vf;
                                    o[k][1] *= alpha[0] * vf;
                                    o[k][2] *= alpha[1] * vf;
                                    o[k][3] *= alpha[1] * vf;
                                }
                                tmem_st16x8(tmem + lane_base + o_col + 64 * half + 8 * k, o[k]);
                            }
                            tmem_wait_st();
                        }
                        l[0] *= alpha[0];
                        l[1] *= alpha[1];
                    }
                    // ---- P = 2^(s * scale - m) (0 where not visible) as bf16 high part (the top 16
                    //      bits) and low part (the rest, rounded), written over S in the buffer: the
                    //      P.V's A operand, tokens (2c, 2c + 1) packed in column c (high part:
                    //      columns 0-31, low part: 32-63)
                    const float nm0 = -m[0], nm1 = -m[1];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        float pv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int h = e >> 1, j = 8 * k + 2 * tig + (e & 1);
                            const float q = ex2(fmaf(sv[k][e], KV == 0 ? p.score_scale : qsc[h], h ? nm1 : nm0));
                            pv[e] = (full || j < vis[h]) ? q : 0.f;
                        }
                        l[0] += pv[0] + pv[1];
                        l[1] += pv[2] + pv[3];
                        if constexpr (KV == 0) {
                            const uint32_t h0 = __float_as_uint(pv[0]) & 0xFFFF0000u, h1 = __float_as_uint(pv[1]) & 0xFFFF0000u;
                            const uint32_t h2 = __float_as_uint(pv[2]) & 0xFFFF0000u, h3 = __float_as_uint(pv[3]) & 0xFFFF0000u;
                            tmem_st16x4(tmem + lane_base + 64 * buf + 4 * k, prmt(h0, h1, 0x7632u), prmt(h2, h3, 0x7632u));
                            tmem_st16x4(tmem + lane_base + 64 * buf + 32 + 4 * k,
                                        pack_bf16x2(pv[0] - __uint_as_float(h0), pv[1] - __uint_as_float(h1)),
                                        pack_bf16x2(pv[2] - __uint_as_float(h2), pv[3] - __uint_as_float(h3)));
                        } else {  // E4M3: P x vs / vref <= 2^8 in f16, one product
                            tmem_st16x4(tmem + lane_base + 64 * buf + 4 * k, pack_f16x2(pv[0] * vw[k][0], pv[1] * vw[k][1]),
                                        pack_f16x2(pv[2] * vw[k][0], pv[3] * vw[k][1]));
                        }
                    }
                    tmem_wait_st();
                    if constexpr (KV == 0) {
                        // ---- V rows past the request's length are zeroed (stale or NaN slots of the page)
                        if (nv < kTile) {
                            uint8_t *vt = smem + stage * L::kStageBytes + C::kTileBytes;
                            for (int i = tid; i < (kTile - nv) * 16; i += 128) {
                                const int row = nv + (i >> 4), ch = i & 15;
                                *reinterpret_cast<uint4 *>(vt + (ch >> 3) * (C::kTileBytes / 2) + row * 128 + (ch & 7) * 16) =
                                    make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                    } else {
                        // ---- E4M3: V widened exactly to f16 into the stage's operand area, in the
                        //      layout of a bf16 V tile ([half][64 rows][128 B], 128-byte swizzle);
                        //      rows past nv are zero (their slots may hold NaN codes).  Thread work:
                        //      16-byte chunk c (dims 16 c .. 16 c + 15) of row t in, two chunks out
                        const uint8_t *vr = smem + stage * L::kStageBytes + C::kTileBytes;
                        uint8_t *vc = smem + stage * L::kStageBytes + L::kVcOff;
#pragma unroll
                        for (int it = 0; it < 4; ++it) {
                            const int i = tid + 128 * it, t = i >> 3, c = i & 7;
                            uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
                            if (t < nv) {
                                const uint4 x = *reinterpret_cast<const uint4 *>(vr + t * 128 + ((c ^ (t & 7)) << 4));
                                lo = make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(x.x & 0xFFFFu)),
                                                e4m3x2_to_f16x2(static_cast<uint16_t>(x.x >> 16)),
                                                e4m3x2_to_f16x2(static_cast<uint16_t>(x.y & 0xFFFFu)),
                                                e4m3x2_to_f16x2(static_cast<uint16_t>(x.y >> 16)));
                                hi = make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(x.z & 0xFFFFu)),
                                                e4m3x2_to_f16x2(static_cast<uint16_t>(x.z >> 16)),
                                                e4m3x2_to_f16x2(static_cast<uint16_t>(x.w & 0xFFFFu)),
                                                e4m3x2_to_f16x2(static_cast<uint16_t>(x.w >> 16)));
                            }
                            uint8_t *row = vc + (c >> 2) * 8192 + t * 128;  // half c / 4, chunks 2 (c % 4), + 1
                            const int cc = 2 * (c & 3);
                            *reinterpret_cast<uint4 *>(row + ((cc ^ (t & 7)) << 4)) = lo;
                            *reinterpret_cast<uint4 *>(row + (((cc + 1) ^ (t & 7)) << 4)) = hi;
                        }
                    }
                    if (!wait_prev_pv()) {
                        failed = true;
                        break;
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_full(buf));
                    ++pv_desc;
                    // the previous descriptor's end, now that this tile's P is handed over
                    if (!flush_epilogue()) {
                        failed = true;
                        break;
                    }
                }
                if (failed) break;
                // ---- a team without tiles here still owes the previous descriptor's end; this
                //      descriptor's end waits for the next descriptor's first tile
                if (!flush_epilogue()) {
                    failed = true;
                    break;
                }
                ep_pending = true;
                ep_slot = slot;
                ep_pv = pv_desc;
                ep_last_g = last_g;
                ep_m[0] = m[0], ep_m[1] = m[1], ep_l[0] = l[0], ep_l[1] = l[1];
                if constexpr (KV == 1) ep_vref = vref;
            }
        }
        (void)failed;
        // ---- every tensor-core role is done: release the tensor memory
        tc_fence_before();
        named_bar_sync(1, kTcThreads);
        if (warp == NCW + 1) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
        return;
    } else if constexpr (QW == 4) {
        // ======= multi-token queries over E4M3 K/V, up to 16 rows per unit (mma.sync) =======
        // The one-token kernel's shape with two 8-row column blocks: the two consumer groups
        // take alternate tiles (a stage belongs to one group), warp wig of a group takes the
        // tokens [16 wig, +16) of its tiles for all rows r = i * G + g < R = q_len * G <= 16
        // (row r of a request of length len sees the tokens t < len - q_len + i + 1).  At a
        // descriptor end the four warps of a group merge their (m, l, O) in shared memory into
        // the group's partial, slot 2 x descriptor + group.
        constexpr int NBW = 2;
        const int grp = warp / 4, wig = warp & 3;
        const int gid = lane >> 2, tig = lane & 3;
        const int tok_base = wig * 16;
        const int R = p.q_len * G;
        const int xr = lane & 7;
        const int k_row = tok_base + xr + ((lane >> 3) & 1) * 8;  // matrices (tokens 0-7 | 8-15) x (chunk 2s | 2s + 1)
        const int k_chunk = lane >> 4;
        float *W = reinterpret_cast<float *>(smem + L::kMergeOff) + warp * L::kWarpFloats;
        const float *WG = reinterpret_cast<const float *>(smem + L::kMergeOff) + 4 * grp * L::kWarpFloats;
        constexpr int kMl = 16 * L::kOStride;  // m of the 16 rows, then l

        for (int qi = 0;; ++qi) {
            const int qslot = qi % kQSlots;
            if (!wait_phase(qfull_bar(qslot), (qi / kQSlots) & 1, abort_flag, p.status)) return;
            const DescInfo *inf = reinterpret_cast<const DescInfo *>(smem + L::kInfoOff) + qslot;
            if (inf->end) break;
            const int n = inf->n, slot = inf->slot, c_start = inf->c_start, dt0 = inf->t0, len = inf->len;
            const int d_b = inf->b, d_h = inf->h;

            // Q fragments (B operand, n = row 8 nb + gid), zero past R
            uint32_t qf[NBW][4][2];
#pragma unroll
            for (int nb = 0; nb < NBW; ++nb) {
                const int r = 8 * nb + gid;
                const uint8_t *qs = smem + L::kQOff + qslot * L::kQSlot + r * C::kQHeadBytes;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    qf[nb][ks][0] = r < R ? *reinterpret_cast<const uint32_t *>(qs + 32 * ks + 4 * tig) : 0u;
                    qf[nb][ks][1] = r < R ? *reinterpret_cast<const uint32_t *>(qs + 32 * ks + 4 * tig + 16) : 0u;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(qempty_bar(qslot));

            // this lane's rows 8 nb + 2 tig + e: score factor (softmax scale x q_scale) and
            // causal limit; rows past R get 0 and are never stored
            float qsc[NBW][2];
            int lim[NBW][2];
#pragma unroll
            for (int nb = 0; nb < NBW; ++nb)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = 8 * nb + 2 * tig + e;
                    const int i = r < R ? r / G : 0;
                    qsc[nb][e] = r < R ? p.score_scale *
                                             p.q_scale[(static_cast<int64_t>(d_b) * p.q_len + i) * p.hq + d_h * G + (r - i * G)]
                                       : 0.f;
                    lim[nb][e] = len - p.q_len + i + 1;
                }
            const int lim_min = len - p.q_len + 1;  // every row sees the tokens below this

            float m[NBW][2], l[NBW][2], o[NBW][8][4];
#pragma unroll
            for (int nb = 0; nb < NBW; ++nb) {
                m[nb][0] = m[nb][1] = -INFINITY;
                l[nb][0] = l[nb][1] = 0.f;
#pragma unroll
                for (int mb = 0; mb < 8; ++mb) o[nb][mb][0] = o[nb][mb][1] = o[nb][mb][2] = o[nb][mb][3] = 0.f;
            }
            float vsc = 0.f, vinv = 0.f;  // O holds the true output divided by vsc; vinv = 1 / vsc

            bool aborted = false;
            for (int li = ((grp - c_start) % GROUPS + GROUPS) % GROUPS; li < n; li += GROUPS) {
                const int c = c_start + li;
                const int stage = c % STAGES;
                if (!wait_phase(full_bar(stage), (c / STAGES) & 1, abort_flag, p.status)) {
                    aborted = true;
                    break;
                }
                const int nv = nvalid[stage];
                if (nv > tok_base) {
                    const uint32_t kbase = sbase + stage * L::kStageBytes;
                    const uint32_t vbase = kbase + C::kTileBytes;
                    const float *ksm = reinterpret_cast<const float *>(smem + stage * L::kStageBytes + 2 * C::kTileBytes);
                    const float *vsm = ksm + kTile;
                    // ---- S^T = K . Q^T  (rows: tokens tok_base + gid / + 8; columns: rows 8 nb + 2 tig, + 1)
                    float sc[NBW][4];
#pragma unroll
                    for (int nb = 0; nb < NBW; ++nb) sc[nb][0] = sc[nb][1] = sc[nb][2] = sc[nb][3] = 0.f;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const int ch = 2 * ks + k_chunk;
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(kbase + k_row * 128 + ((ch ^ xr) << 4), a0, a1, a2, a3);
#pragma unroll
                        for (int nb = 0; nb < NBW; ++nb) mma_e4m3(sc[nb], a0, a1, a2, a3, qf[nb][ks][0], qf[nb][ks][1]);
                    }
                    // per-token scales; tokens past the tile's valid rows get none (their shared
                    // memory may hold anything) and are masked below
                    const int ta = tok_base + gid, tb = ta + 8;
                    const float ksa = ta < nv ? ksm[ta] : 0.f, ksb = tb < nv ? ksm[tb] : 0.f;
                    const float vsa = ta < nv ? vsm[ta] : 0.f, vsb = tb < nv ? vsm[tb] : 0.f;
                    const int T0 = (dt0 + li) * kTile + tok_base;  // token of this warp's first row
                    const bool mask = T0 + 16 > lim_min;  // some row of the warp's tokens is past a limit
#pragma unroll
                    for (int nb = 0; nb < NBW; ++nb) {
                        sc[nb][0] *= qsc[nb][0] * ksa;
                        sc[nb][1] *= qsc[nb][1] * ksa;
                        sc[nb][2] *= qsc[nb][0] * ksb;
                        sc[nb][3] *= qsc[nb][1] * ksb;
                        if (mask) {
                            if (T0 + gid >= lim[nb][0]) sc[nb][0] = -INFINITY;
                            if (T0 + gid >= lim[nb][1]) sc[nb][1] = -INFINITY;
                            if (T0 + gid + 8 >= lim[nb][0]) sc[nb][2] = -INFINITY;
                            if (T0 + gid + 8 >= lim[nb][1]) sc[nb][3] = -INFINITY;
                        }
                    }
                    // ---- lazy references, so that rescaling O is rare: the V scale reference vsc is
                    //      the largest V scale seen (P carries vs / vsc <= 1), and a row's reference
                    //      m moves only when the row's maximum passes it by more than 8 (P <= 2^8,
                    //      well inside f16); the warp reduces maxima only when some lane sees growth
                    bool grow = fmaxf(vsa, vsb) > vsc;
#pragma unroll
                    for (int nb = 0; nb < NBW; ++nb)
                        grow |= fmaxf(sc[nb][0], sc[nb][2]) > m[nb][0] + 8.f || fmaxf(sc[nb][1], sc[nb][3]) > m[nb][1] + 8.f;
                    if (__any_sync(0xffffffffu, grow)) {
                        float vm = fmaxf(vsa, vsb);
#pragma unroll
                        for (int o_ = 4; o_ < 32; o_ <<= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o_));
                        float vf = 1.f;
                        if (vm > vsc) {
                            if (vsc > 0.f) vf = vsc / vm;
                            vsc = vm;
                            vinv = 1.f / vm;
                        }
#pragma unroll
                        for (int nb = 0; nb < NBW; ++nb) {
                            float mx[2] = {fmaxf(sc[nb][0], sc[nb][2]), fmaxf(sc[nb][1], sc[nb][3])};
                            float f[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
#pragma unroll
                                for (int o_ = 4; o_ < 32; o_ <<= 1) mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], o_));
                                float alpha = 1.f;
                                if (mx[e] > m[nb][e] + 8.f) {  // from m = -inf: alpha = 0 (nothing accumulated yet)
                                    alpha = ex2(m[nb][e] - mx[e]);
                                    m[nb][e] = mx[e];
                                }
                                l[nb][e] *= alpha;
                                f[e] = alpha * vf;
                            }
#pragma unroll
                            for (int mb = 0; mb < 8; ++mb) {
                                o[nb][mb][0] *= f[0];
                                o[nb][mb][1] *= f[1];
                                o[nb][mb][2] *= f[0];
                                o[nb][mb][3] *= f[1];
                            }
                        }
                    }
                    // ---- P = 2^(s - m) (a row still at m = -inf has seen no visible token: P = 0)
                    const float wa = vsa * vinv, wb = vsb * vinv;
                    uint32_t bh[NBW][2];
#pragma unroll
                    for (int nb = 0; nb < NBW; ++nb) {
                        const float r0 = m[nb][0] == -INFINITY ? 0.f : m[nb][0], r1 = m[nb][1] == -INFINITY ? 0.f : m[nb][1];
                        const float p0 = ex2(sc[nb][0] - r0), p1 = ex2(sc[nb][1] - r1);
                        const float p2 = ex2(sc[nb][2] - r0), p3 = ex2(sc[nb][3] - r1);
                        l[nb][0] += p0 + p2;
                        l[nb][1] += p1 + p3;
                        bh[nb][0] = movmatrix_trans(pack_f16x2(p0 * wa, p1 * wa));
                        bh[nb][1] = movmatrix_trans(pack_f16x2(p2 * wb, p3 * wb));
                    }
                    // ---- O^T += V^T . P^T (V widened to f16); V rows past the valid tokens are zeroed
                    const bool partial = nv < tok_base + 16;
                    const uint32_t mlo = partial ? tok_mask(tok_base + 2 * tig, nv) : 0xFFFFFFFFu;
                    const uint32_t mhi = partial ? tok_mask(tok_base + 8 + 2 * tig, nv) : 0xFFFFFFFFu;
#pragma unroll
                    for (int mp = 0; mp < 4; ++mp) {
                        const int ch = 2 * mp + k_chunk;
                        uint32_t x0, x1, x2, x3;
                        ldsm_x4_trans(vbase + k_row * 128 + ((ch ^ xr) << 4), x0, x1, x2, x3);
                        // x0 / x1: tokens 0-7 / 8-15 of chunk 2 mp; x2 / x3: of chunk 2 mp + 1;
                        // each holds, for dims (2 gid, 2 gid + 1) of its chunk, tokens (2 tig, 2 tig + 1)
                        uint32_t a0, a1, a2, a3;
                        cvt_pair(x0, a0, a1);
                        cvt_pair(x1, a2, a3);
                        if (partial) {
                            a0 &= mlo;
                            a1 &= mlo;
                            a2 &= mhi;
                            a3 &= mhi;
                        }
#pragma unroll
                        for (int nb = 0; nb < NBW; ++nb) mma_f16(o[nb][2 * mp], a0, a1, a2, a3, bh[nb][0], bh[nb][1]);
                        cvt_pair(x2, a0, a1);
                        cvt_pair(x3, a2, a3);
                        if (partial) {
                            a0 &= mlo;
                            a1 &= mlo;
                            a2 &= mhi;
                            a3 &= mhi;
                        }
#pragma unroll
                        for (int nb = 0; nb < NBW; ++nb) mma_f16(o[nb][2 * mp + 1], a0, a1, a2, a3, bh[nb][0], bh[nb][1]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(stage));
            }
            if (aborted) return;

            // ---- deposit this warp's (m, l, O x vsc) for the group's merge
#pragma unroll
            for (int nb = 0; nb < NBW; ++nb)
#pragma unroll
                for (int e = 0; e < 2; ++e)
#pragma unroll
                    for (int o_ = 4; o_ < 32; o_ <<= 1) l[nb][e] += __shfl_xor_sync(0xffffffffu, l[nb][e], o_);
            if (!wait_phase(merge_done(grp), (qi & 1) ^ 1, abort_flag, p.status)) return;
#pragma unroll
            for (int nb = 0; nb < NBW; ++nb) {
                const int r0 = 8 * nb + 2 * tig;
                if (gid == 0) {
                    W[kMl + r0] = m[nb][0];
                    W[kMl + r0 + 1] = m[nb][1];
                    W[kMl + 16 + r0] = l[nb][0];
                    W[kMl + 16 + r0 + 1] = l[nb][1];
                }
#pragma unroll
                for (int mb = 0; mb < 8; ++mb) {
                    const int d0 = 16 * mb + 2 * gid;
                    *reinterpret_cast<float2 *>(W + r0 * L::kOStride + d0) = make_float2(o[nb][mb][0] * vsc, o[nb][mb][2] * vsc);
                    *reinterpret_cast<float2 *>(W + (r0 + 1) * L::kOStride + d0) =
                        make_float2(o[nb][mb][1] * vsc, o[nb][mb][3] * vsc);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(merge_full(grp));
            if (!wait_phase(merge_full(grp), qi & 1, abort_flag, p.status)) return;
            // ---- merge of the group's four warps: the partial of rows below R, slot 2 x descriptor + group
            const int64_t slot_row = (2 * static_cast<int64_t>(slot) + grp) * R;
            for (int idx = wig * 32 + lane; idx < R * 32; idx += 128) {
                const int hd = idx >> 5, d4 = (idx & 31) * 4;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < 4; ++w) M = fmaxf(M, WG[w * L::kWarpFloats + kMl + hd]);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                float lse = -INFINITY;
                if (M != -INFINITY) {
                    float Lsum = 0.f;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float *Ww = WG + w * L::kWarpFloats;
                        const float e = ex2(Ww[kMl + hd] - M);
                        Lsum += e * Ww[kMl + 16 + hd];
                        const float4 v = *reinterpret_cast<const float4 *>(Ww + hd * L::kOStride + d4);
                        acc.x += e * v.x;
                        acc.y += e * v.y;
                        acc.z += e * v.z;
                        acc.w += e * v.w;
                    }
                    const float inv = 1.f / Lsum;
                    acc.x *= inv;
                    acc.y *= inv;
                    acc.z *= inv;
                    acc.w *= inv;
                    lse = (M + lg2(Lsum)) * kLn2;
                }
                *reinterpret_cast<float4 *>(p.partial_o + (slot_row + hd) * kHeadDim + d4) = acc;
                if ((idx & 31) == 0) p.partial_lse[slot_row + hd] = lse;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(merge_done(grp));
        }
        return;
    } else {
    // =========================== consumer warps ===========================
    const int grp = warp / 4, wig = warp & 3;
    const int gid = lane >> 2, tig = lane & 3;
    const int tok_base = wig * 16;
    // per-lane ldmatrix row offsets (row & 7 == lane & 7 for every 8-row block)
    const int xr = lane & 7;
    const int k_row = tok_base + xr + ((lane >> 3) & 1) * 8;  // K: matrices (rows 0-7|8-15) x (chunk 0|1)
    const int k_chunk = lane >> 4;
    const int v_row = (KV == 0) ? tok_base + xr + (lane >> 4) * 8 : k_row;
    const int v_chunk = (KV == 0) ? ((lane >> 3) & 1) : (lane >> 4);
    // bf16 stage [page][half][P rows][128 B]: byte offsets of this lane's rows and of the second half
    const uint32_t half_off = static_cast<uint32_t>(p.page_size) * 128u;
    const uint32_t k_off = kv_row_off(k_row, p.page_size), v_off = kv_row_off(v_row, p.page_size);

    // Merge of descriptor d (states deposited in merge slot d & 1 by all consumer warps):
    // the warps' (m, l, O) combined under one softmax, written as a normalised partial.
    auto merge_and_write = [&](int d, int pslot, int ub, int uh, int unp, int upbeg) -> bool {
        const int ms = d % MSLOTS;
        if (!wait_phase(merge_full(ms), (d / MSLOTS) & 1, abort_flag, p.status)) return false;
        const float *M0 = reinterpret_cast<const float *>(smem + L::kMergeOff) + ms * L::kMergeSlot;
        for (int idx = warp * 32 + lane; idx < G * 32; idx += NCW * 32) {
            const int hd = idx >> 5, d4 = (idx & 31) * 4;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NCW; ++w) M = fmaxf(M, M0[w * L::kWarpFloats + kMaxGroup * L::kOStride + hd]);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            float lse = -INFINITY;
            if (M != -INFINITY) {
                float Lsum = 0.f;
#pragma unroll
                for (int w = 0; w < NCW; ++w) {
                    const float *Ww = M0 + w * L::kWarpFloats;
                    const float e = ex2(Ww[kMaxGroup * L::kOStride + hd] - M);
                    Lsum += e * Ww[kMaxGroup * L::kOStride + kMaxGroup + hd];
                    const float4 v = *reinterpret_cast<const float4 *>(Ww + hd * L::kOStride + d4);
                    acc.x += e * v.x;
                    acc.y += e * v.y;
                    acc.z += e * v.z;
                    acc.w += e * v.w;
                }
                const float inv = 1.f / Lsum;
                acc.x *= inv;
                acc.y *= inv;
                acc.z *= inv;
                acc.w *= inv;
                lse = (M + lg2(Lsum)) * kLn2;
            }
            if (FUSE && unp == 1) {  // the descriptor is the whole unit: final output
                const int64_t orow = static_cast<int64_t>(ub) * p.hq + uh * G + hd;
                store_out4<float>(p.out, orow, idx & 31, acc, p.out_bf16);
                if ((idx & 31) == 0 && p.out_lse) p.out_lse[orow] = lse;
                continue;
            }
            const int64_t row = static_cast<int64_t>(pslot) * G + hd;
            *reinterpret_cast<float4 *>(p.partial_o + row * kHeadDim + d4) = acc;
            if ((idx & 31) == 0) p.partial_lse[row] = lse;
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(merge_done(ms));
            if (FUSE) mbar_arrive(epi_ready(d % kEpiRing));
        }
        return true;
    };

    // The merge of a descriptor runs after the NEXT descriptor's tiles, when every warp
    // deposited its state long ago: no warp waits for the slowest at each boundary.
    int pend_d = -1, pend_slot = 0, pend_b = 0, pend_h = 0, pend_np = 1, pend_pbeg = 0;
    for (int qi = 0;; ++qi) {
        // ---- next descriptor from the producer (info + Q in shared memory)
        const int qslot = qi % kQSlots;
        if (!wait_phase(qfull_bar(qslot), (qi / kQSlots) & 1, abort_flag, p.status)) return;
        const DescInfo *inf = reinterpret_cast<const DescInfo *>(smem + L::kInfoOff) + qslot;
        if (inf->end) break;
        const int n = inf->n, slot = inf->slot, c_start = inf->c_start;
        const int d_b = inf->b, d_h = inf->h, d_np = inf->np, d_pbeg = inf->pbeg;
        float qsc0 = p.score_scale, qsc1 = p.score_scale;
        if (KV == 1) {
            qsc0 *= inf->qscale[2 * tig];
            qsc1 *= inf->qscale[2 * tig + 1];
        }

        // ---- Q fragments (B operand, n = query head gid), zero past G
        constexpr int KSTEPS = (KV == 0) ? 8 : 4;
        uint32_t qf[KSTEPS][2];
        {
            const uint8_t *qs = smem + L::kQOff + qslot * L::kQSlot + gid * C::kQHeadBytes;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                const int off = 32 * ks + 4 * tig;
                qf[ks][0] = gid < G ? *reinterpret_cast<const uint32_t *>(qs + off) : 0u;
                qf[ks][1] = gid < G ? *reinterpret_cast<const uint32_t *>(qs + off + 16) : 0u;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(qempty_bar(qslot));

        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        // E4M3: O holds the true output divided by vsc (set by the first scaled tile); bf16: 1
        float vsc = (KV == 1) ? 0.f : 1.f, vinv = 0.f;  // vinv = 1 / vsc (E4M3)
        float o[8][4];
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) o[mb][0] = o[mb][1] = o[mb][2] = o[mb][3] = 0.f;

        bool aborted = false;
        for (int li = ((grp - c_start) % GROUPS + GROUPS) % GROUPS; li < n; li += GROUPS) {
            const int c = c_start + li;
            const int stage = c % STAGES;
            // the merge still owed for the previous descriptor is done while this tile's data
            // is in flight (and every warp has deposited), so it never delays a landed tile
            if (MSLOTS == 2 && pend_d >= 0 && !mbar_test_wait(full_bar(stage), (c / STAGES) & 1) &&
                mbar_test_wait(merge_full(pend_d % MSLOTS), (pend_d / MSLOTS) & 1)) {
                if (!merge_and_write(pend_d, pend_slot, pend_b, pend_h, pend_np, pend_pbeg)) return;
                pend_d = -1;
            }
            if (!wait_phase(full_bar(stage), (c / STAGES) & 1, abort_flag, p.status)) {
                aborted = true;
                break;
            }
            const int nv = nvalid[stage];
            if (nv > tok_base) {
                const uint32_t kbase = sbase + stage * L::kStageBytes;
                const uint32_t vbase = kbase + C::kTileBytes;
                // ---- S^T = K . Q^T  (rows: tokens tok_base + gid / + 8; cols: heads 2tig, 2tig+1)
                // two independent accumulation chains (even / odd k-steps) halve the MMA latency
                float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks) {
                    const int ch = 2 * ks + k_chunk;
                    uint32_t addr;
                    if (KV == 0)
                        addr = kbase + (ch >> 3) * half_off + k_off + (((ch & 7) ^ xr) << 4);
                    else
                        addr = kbase + k_row * 128 + ((ch ^ xr) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(addr, a0, a1, a2, a3);
                    float(&acc)[4] = (ks & 1) ? s2 : s;
                    if (KV == 0) mma_bf16(acc, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
                    else mma_e4m3(acc, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) s[i] += s2[i];
                const int ta = tok_base + gid, tb = ta + 8;
                float ksa = 1.f, ksb = 1.f, vsa = 0.f, vsb = 0.f;
                if (KV == 1) {
                    const float *ksm = reinterpret_cast<const float *>(smem + stage * L::kStageBytes + 2 * C::kTileBytes);
                    const float *vsm = ksm + kTile;
                    ksa = ksm[ta];
                    ksb = ksm[tb];
                    vsa = ta < nv ? vsm[ta] : 0.f;
                    vsb = tb < nv ? vsm[tb] : 0.f;
                }
                s[0] *= qsc0 * ksa;
                s[1] *= qsc1 * ksa;
                s[2] *= qsc0 * ksb;
                s[3] *= qsc1 * ksb;
                const bool partial = nv < tok_base + 16;
                if (partial) {
                    if (ta >= nv) s[0] = s[1] = -INFINITY;
                    if (tb >= nv) s[2] = s[3] = -INFINITY;
                }
                uint32_t b0h, b1h, b0l = 0, b1l = 0;
                if constexpr (KV == 1) {
                    // ---- lazy references, so that rescaling O is rare: the V scale reference vsc
                    //      is the largest V scale seen (P carries vs / vsc <= 1), and a head's
                    //      reference m moves only when its maximum passes it by more than 8 (P <=
                    //      2^8, well inside f16); the warp reduces maxima only when a lane sees growth
                    const bool grow = fmaxf(vsa, vsb) > vsc || fmaxf(s[0], s[2]) > m0 + 8.f || fmaxf(s[1], s[3]) > m1 + 8.f;
                    if (__any_sync(0xffffffffu, grow)) {
                        float vm = fmaxf(vsa, vsb), mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
                        for (int o_ = 4; o_ < 32; o_ <<= 1) {
                            vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o_));
                            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o_));
                            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o_));
                        }
                        float vf = 1.f;
                        if (vm > vsc) {
                            if (vsc > 0.f) vf = vsc / vm;
                            vsc = vm;
                            vinv = 1.f / vm;
                        }
                        float al0 = 1.f, al1 = 1.f;  // from m = -inf: 0 (nothing accumulated yet)
                        if (mx0 > m0 + 8.f) {
                            al0 = ex2(m0 - mx0);
                            m0 = mx0;
                        }
                        if (mx1 > m1 + 8.f) {
                            al1 = ex2(m1 - mx1);
                            m1 = mx1;
                        }
                        l0 *= al0;
                        l1 *= al1;
                        al0 *= vf;
                        al1 *= vf;
#pragma unroll
                        for (int mb = 0; mb < 8; ++mb) {
                            o[mb][0] *= al0;
                            o[mb][1] *= al1;
                            o[mb][2] *= al0;
                            o[mb][3] *= al1;
                        }
                    }
                    // P = 2^(s - m) (a head still at m = -inf has seen no valid token: P = 0)
                    const float r0 = m0 == -INFINITY ? 0.f : m0, r1 = m1 == -INFINITY ? 0.f : m1;
                    const float p0 = ex2(s[0] - r0), p1 = ex2(s[1] - r1), p2 = ex2(s[2] - r0), p3 = ex2(s[3] - r1);
                    l0 += p0 + p2;
                    l1 += p1 + p3;
                    const float wa = vsa * vinv, wb = vsb * vinv;
                    b0h = movmatrix_trans(pack_f16x2(p0 * wa, p1 * wa));
                    b1h = movmatrix_trans(pack_f16x2(p2 * wb, p3 * wb));
                } else {
                    // ---- online softmax (base 2), per head, over this warp's tokens
                    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
                    for (int o_ = 4; o_ < 32; o_ <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o_));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o_));
                    }
                    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                    const float r0 = mn0 == -INFINITY ? 0.f : mn0, r1 = mn1 == -INFINITY ? 0.f : mn1;
                    const float al0 = ex2(m0 - r0), al1 = ex2(m1 - r1);
                    const float p0 = ex2(s[0] - r0), p1 = ex2(s[1] - r1), p2 = ex2(s[2] - r0), p3 = ex2(s[3] - r1);
                    l0 = l0 * al0 + p0 + p2;
                    l1 = l1 * al1 + p1 + p3;
                    m0 = mn0;
                    m1 = mn1;
                    const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
                    const uint32_t l01 = pack_bf16x2(p0 - bf16lo_to_f32(h01), p1 - bf16hi_to_f32(h01));
                    const uint32_t l23 = pack_bf16x2(p2 - bf16lo_to_f32(h23), p3 - bf16hi_to_f32(h23));
                    b0h = movmatrix_trans(h01);
                    b1h = movmatrix_trans(h23);
                    b0l = movmatrix_trans(l01);
                    b1l = movmatrix_trans(l23);
#pragma unroll
                    for (int mb = 0; mb < 8; ++mb) {
                        o[mb][0] *= al0;
                        o[mb][1] *= al1;
                        o[mb][2] *= al0;
                        o[mb][3] *= al1;
                    }
                }
                // masks for the A (V^T) fragments: tokens (2tig, 2tig+1) and (8+2tig, 9+2tig)
                const uint32_t mlo = partial ? tok_mask(tok_base + 2 * tig, nv) : 0xFFFFFFFFu;
                const uint32_t mhi = partial ? tok_mask(tok_base + 8 + 2 * tig, nv) : 0xFFFFFFFFu;
                // ---- O^T += V^T . P^T
                if (KV == 0) {
#pragma unroll
                    for (int mb = 0; mb < 8; ++mb) {
                        const int ch = 2 * mb + v_chunk;
                        const uint32_t addr = vbase + (ch >> 3) * half_off + v_off + (((ch & 7) ^ xr) << 4);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_trans(addr, a0, a1, a2, a3);
                        if (partial) {
                            a0 &= mlo;
                            a1 &= mlo;
                            a2 &= mhi;
                            a3 &= mhi;
                        }
                        mma_bf16(o[mb], a0, a1, a2, a3, b0h, b1h);
                        mma_bf16(o[mb], a0, a1, a2, a3, b0l, b1l);
                    }
                } else {
#pragma unroll
                    for (int mp = 0; mp < 4; ++mp) {
                        const int ch = 2 * mp + v_chunk;
                        const uint32_t addr = vbase + v_row * 128 + ((ch ^ xr) << 4);
                        uint32_t x0, x1, x2, x3;
                        ldsm_x4_trans(addr, x0, x1, x2, x3);
                        // x0/x1: tokens 0-7 / 8-15 of chunk 2mp; x2/x3: of chunk 2mp+1.
                        // Each holds, for dims (2gid, 2gid+1) of the chunk, tokens (2tig, 2tig+1).
                        uint32_t a0, a1, a2, a3;
                        cvt_pair(x0, a0, a1);
                        cvt_pair(x1, a2, a3);
                        if (partial) {
                            a0 &= mlo;
                            a1 &= mlo;
                            a2 &= mhi;
                            a3 &= mhi;
                        }
                        mma_f16(o[2 * mp], a0, a1, a2, a3, b0h, b1h);
                        cvt_pair(x2, a0, a1);
                        cvt_pair(x3, a2, a3);
                        if (partial) {
                            a0 &= mlo;
                            a1 &= mlo;
                            a2 &= mhi;
                            a3 &= mhi;
                        }
                        mma_f16(o[2 * mp + 1], a0, a1, a2, a3, b0h, b1h);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(stage));
        }
        if (aborted) return;

        // ---- deposit this warp's (m, l, O) in merge slot qi & 1, then merge the previous descriptor
#pragma unroll
        for (int o_ = 4; o_ < 32; o_ <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o_);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o_);
        }
        const int ms = qi % MSLOTS;
        if (!wait_phase(merge_done(ms), ((qi / MSLOTS) & 1) ^ 1, abort_flag, p.status)) return;
        if (FUSE) {
            const int er = qi % kEpiRing;
            if (!wait_phase(epi_free(er), ((qi / kEpiRing) & 1) ^ 1, abort_flag, p.status)) return;
            if (warp == 0 && lane == 0) epi_rec[er] = EpiRecord{d_b, d_h, d_np, d_pbeg};
        }
        float *W = reinterpret_cast<float *>(smem + L::kMergeOff) + ms * L::kMergeSlot + warp * L::kWarpFloats;
        if (gid == 0) {
            W[kMaxGroup * L::kOStride + 2 * tig] = m0;
            W[kMaxGroup * L::kOStride + 2 * tig + 1] = m1;
            W[kMaxGroup * L::kOStride + kMaxGroup + 2 * tig] = l0;
            W[kMaxGroup * L::kOStride + kMaxGroup + 2 * tig + 1] = l1;
        }
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
            const int d0 = (KV == 0) ? 16 * mb + gid : 16 * mb + 2 * gid;
            const int d1 = (KV == 0) ? d0 + 8 : d0 + 1;
            W[(2 * tig) * L::kOStride + d0] = o[mb][0] * vsc;
            W[(2 * tig + 1) * L::kOStride + d0] = o[mb][1] * vsc;
            W[(2 * tig) * L::kOStride + d1] = o[mb][2] * vsc;
            W[(2 * tig + 1) * L::kOStride + d1] = o[mb][3] * vsc;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(merge_full(ms));
        if (MSLOTS == 1) {  // one merge slot: merge this descriptor at once
            if (!merge_and_write(qi, slot, d_b, d_h, d_np, d_pbeg)) return;
            continue;
        }
        if (pend_d >= 0 && !merge_and_write(pend_d, pend_slot, pend_b, pend_h, pend_np, pend_pbeg)) return;
        pend_d = qi;
        pend_slot = slot;
        pend_b = d_b;
        pend_h = d_h;
        pend_np = d_np;
        pend_pbeg = d_pbeg;
    }
    if (pend_d >= 0) merge_and_write(pend_d, pend_slot, pend_b, pend_h, pend_np, pend_pbeg);
    }  // QW == 0
}

// Self-test of the bounded wait: warp 0 waits on an mbarrier that nothing ever arrives at;
// when its limit passes it records DSA_DEV_TIMEOUT and raises the CTA's abort flag; warp 1
// waits on a second such barrier and must leave on the abort flag.  *status also gets bit
// 16 when warp 1 observed the abort.
__global__ void __launch_bounds__(64, 1) wait_selftest_kernel(int32_t *status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (lane != 0) return;
    volatile int *ab = &abort_flag;
    if (warp == 0) {
        wait_phase(smem_u32(&bars[0]), 0, ab, status, limit_ns);
    } else {
        // a limit far beyond warp 0's: this wait can only end through the abort flag
        if (!wait_phase(smem_u32(&bars[1]), 0, ab, status, 8 * limit_ns) && *ab) atomicOr(status, 1 << 16);
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 5-D view (128-byte piece of a row, token in page, piece, KV head, page) of a page pool,
// 128-byte swizzle.  A bf16 row is two 128-B pieces, an E4M3 row one.  HND pages
// [num_pages][Hkv][P][128] and NHD pages [num_pages][P][Hkv][128] differ only in the strides.
// The box is the P tokens of one (page, head): both pieces (lands as [piece][P rows][128 B]),
// or one piece when `split` (the tensor-core kernel's per-half operand layout).
bool make_pool_map(CUtensorMap *m, const void *pool, int kv, int num_pages, int hkv, int page, bool nhd,
                   bool split) {
    std::memset(m, 0, sizeof(*m));
    if (num_pages == 0) return true;  // nothing can be loaded
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t es = kv == 0 ? 2 : 1, pieces = kv == 0 ? 2 : 1;
    const cuuint64_t row = kHeadDim * es, P = static_cast<cuuint64_t>(page), H = static_cast<cuuint64_t>(hkv);
    const cuuint64_t dims[5] = {128 / es, P, pieces, H, static_cast<cuuint64_t>(num_pages)};
    const cuuint64_t strides[4] = {nhd ? H * row : row, 128, nhd ? row : P * row, P * H * row};
    const cuuint32_t box[5] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(page),
                               split ? 1u : static_cast<cuuint32_t>(pieces), 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, kv == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 5,
                    const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int KV, int STAGES, int GROUPS, bool PERSIST, bool FUSE = false, int MSLOTS = 2, int QW = 0>
dsa_status launch(const AttnArgs &a, const KernelParams &kp, dim3 grid, cudaStream_t st) {
    using L = Layout<KV, STAGES, GROUPS, MSLOTS, QW>;
    CUtensorMap km, vm;
    const bool nhd = a.kv_layout == DSA_NHD, split = QW == 3 && KV == 0 && a.page_size < kTile;
    if (!make_pool_map(&km, a.k_pages, KV, a.num_pages, a.num_kv_heads, a.page_size, nhd, split) ||
        !make_pool_map(&vm, a.v_pages, KV, a.num_pages, a.num_kv_heads, a.page_size, nhd, split))
        return DSA_ERR_CUDA;
    auto kern = attn_kernel<KV, STAGES, GROUPS, PERSIST, FUSE, MSLOTS, QW>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) != cudaSuccess)
        return DSA_ERR_CUDA;
    return launch_pdl(kern, grid, dim3(FUSE ? L::kThreadsFused : L::kThreads), L::kAlloc, st, km, vm, kp);
}

KernelParams base_params(const AttnArgs &a, float *partial_o, float *partial_lse, int32_t *status) {
    KernelParams kp{};
    kp.q = static_cast<const uint8_t *>(a.q);
    kp.q_scale = a.q_scale;
    kp.k_scale = a.k_scale;
    kp.v_scale = a.v_scale;
    kp.block_table = a.block_table;
    kp.seq_lens = a.seq_lens;
    kp.max_pages = a.max_pages_per_req;
    kp.num_pages = a.num_pages;
    kp.hq = a.num_q_heads;
    kp.hkv = a.num_kv_heads;
    kp.G = a.num_q_heads / a.num_kv_heads;
    kp.num_units = a.batch * a.num_kv_heads;
    kp.q_len = 1;
    kp.slots_per_desc = 1;
    kp.page_size = a.page_size;
    kp.nhd = a.kv_layout == DSA_NHD;
    kp.score_scale = a.sm_scale * kLog2e;
    kp.partial_o = partial_o;
    kp.partial_lse = partial_lse;
    kp.status = status;
    return kp;
}

// CTA shapes.  One persistent CTA per SM: two consumer groups and a deep ring.  Two CTAs per
// SM (used by the static grid, and by the persistent kernel when the task map has at least
// two bins per SM): one consumer group and a shallow ring each, so both fit in shared memory.
// (A sweep on the GB300 found the lagged two-slot merge with 4 / 8 stages faster than one
// merge slot with the same or deeper rings.)
constexpr int kPersistStagesBf16 = 4, kPersistStagesFp8 = 8, kPersistGroups = 2, kPersistMergeSlots = 2;
constexpr int kPairStagesBf16 = 2, kPairStagesFp8 = 4, kPairGroups = 1;
// The multi-token tensor-memory kernel keeps P in tensor memory, so its shared memory holds a
// fifth stage (tiles stay in the ring from their load until their P.V, several microseconds).
constexpr int kTcStages = 5;
// The E4M3 multi-token kernel: every warp reads every stage, 8 stages of 17 KB.
constexpr int kMultiStagesFp8 = 8;

// Persistent launch: the CTA shape that keeps all of the map's bins resident at once.
template <int KV, bool FUSE>
dsa_status launch_persistent(const AttnArgs &a, const KernelParams &kp, int num_ctas, cudaStream_t st) {
    const int sms = sm_count();
    const dim3 grid(num_ctas);
    if (sms > 0 && num_ctas >= 2 * sms)
        return launch<KV, KV == 0 ? kPairStagesBf16 : kPairStagesFp8, kPairGroups, true, FUSE>(a, kp, grid, st);
    return launch<KV, KV == 0 ? kPersistStagesBf16 : kPersistStagesFp8, kPersistGroups, true, FUSE, kPersistMergeSlots>(
        a, kp, grid, st);
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int32_t dsa_multi_slots_per_desc(int32_t q_len, int32_t group) {
    if (q_len < 1 || group < 1) return -1;
    return q_len > 1 ? 2 : 1;
}

extern "C" dsa_status dsa_decode_ex(int32_t q_len, int32_t kv_layout, const void *q, dsa_dtype q_dtype,
                                    const float *q_scale, const void *k_pages, const void *v_pages,
                                    dsa_dtype kv_dtype, const float *k_scale, const float *v_scale,
                                    const int32_t *block_table, int32_t max_pages_per_req, int32_t num_pages,
                                    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t page_size, float sm_scale,
                                    const dsa_task_map *map, float *partial_o, float *partial_lse,
                                    uint64_t *cta_times, dsa_stream stream) {
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
    if (q_len == 1) {
        if (kv_dtype == DSA_BF16) return launch_persistent<0, false>(a, kp, map->num_ctas, to_cuda(stream));
        return launch_persistent<1, false>(a, kp, map->num_ctas, to_cuda(stream));
    }
    kp.q_len = q_len;
    kp.slots_per_desc = dsa_multi_slots_per_desc(q_len, num_q_heads / num_kv_heads);
    const dim3 grid(map->num_ctas);
    // E4M3 K/V: up to 16 rows mma.sync warps (the groups take alternate tiles, 16 tokens x all
    // rows per warp), more rows the tensor-memory kernel
    if (kv_dtype == DSA_FP8_E4M3) {
        if (R <= 16) return launch<1, kMultiStagesFp8, 2, true, false, 1, 4>(a, kp, grid, to_cuda(stream));
        return launch<1, kTcStages, 2, true, false, 1, 3>(a, kp, grid, to_cuda(stream));
    }
    // bf16 K/V: the tensor-memory kernel, for any number of query rows up to 64
    return launch<0, kTcStages, 2, true, false, 1, 3>(a, kp, grid, to_cuda(stream));
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
    if (kv_dtype == DSA_BF16) return launch_persistent<0, true>(a, kp, map->num_ctas, to_cuda(stream));
    return launch_persistent<1, true>(a, kp, map->num_ctas, to_cuda(stream));
}

extern "C" dsa_status dsa_selftest_wait_timeout(int32_t *status, int64_t limit_ns, dsa_stream stream) {
    if (!status || limit_ns <= 0 || limit_ns > static_cast<int64_t>(kWaitLimitNs)) return DSA_ERR_INVALID_ARG;
    wait_selftest_kernel<<<1, 64, 0, to_cuda(stream)>>>(status, static_cast<uint64_t>(limit_ns));
    return launch_status();
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
    if (kv_dtype == DSA_BF16) return launch<0, kPairStagesBf16, kPairGroups, false>(a, kp, grid, to_cuda(stream));
    return launch<1, kPairStagesFp8, kPairGroups, false>(a, kp, grid, to_cuda(stream));
}
