// Paged-KV GQA decode attention over 64-token tiles, in two schedules:
//   - persistent (dsa_decode): one CTA per task-map bin drains its descriptors
//     (HPC-Ops × SGLang blog, section "围绕活跃 KV 工作进行调度");
//   - static split-KV (dsa_static_splitkv): one CTA per (split, KV head, request)
//     on a fixed grid (same blog, section "Attention：变长 decode 的负载均衡").
// Both run the same per-tile engine.
//
// Engine (per CTA):
//   * one producer warp (engine.cuh, shared with the tensor-memory multi-token kernel in
//     attention_tc.cu) walks the descriptors, reads the page ids of the tiles
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
#include "engine.cuh"

namespace dsa {
namespace {

constexpr int kEpiRing = 8;  // merged descriptors the epilogue warp may lag behind (fused combine)

// QW = 0: one query token per request; the consumer groups take alternate tiles and all
// warps of the CTA merge at each descriptor end.  QW = 4: multi-token queries over E4M3 K/V
// with up to 16 query rows per unit on mma.sync, the one-token shape (groups on alternate
// tiles, 16 tokens per warp) over two 8-row blocks; each group merges its warps into its own
// partial slot.  (Other multi-token steps run on the tensor-memory kernel, attention_tc.cu:
// for E4M3 K/V at up to 16 rows it measured twice the time of this one, bound by its per-tile
// chain; an mma.sync kernel giving each warp a 32-token half of every tile measured 1.1-1.6x
// the tensor-memory kernel's time at 24-64 rows.)
template <int KV, int STAGES, int GROUPS, int MSLOTS = 2, int QW = 0>
struct Layout {
    // descriptors handed ahead to the consumers (Q + info): with one query token a slot is
    // small, and more of them let the producer run ahead through runs of short descriptors
    static constexpr int kQSlots = 4;
    static constexpr int kNcw = GROUPS * 4;  // consumer warps
    static constexpr int kThreads = (kNcw + 1) * 32;  // consumers + producer
    static constexpr int kThreadsFused = (kNcw + 2) * 32;  // + epilogue warp (fused combine)
    static constexpr int kStageTx = 2 * Cfg<KV>::kTileBytes + 2 * Cfg<KV>::kScaleBytes;
    static constexpr int kStageBytes = round_up(kStageTx, 1024);
    static constexpr int kQRows = QW == 0 ? kMaxGroup : 16;
    static constexpr int kQSlot = kQRows * Cfg<KV>::kQHeadBytes;
    static constexpr int kQOff = STAGES * kStageBytes;
    static constexpr int kOStride = 132;  // floats per head row of a warp's O (padding avoids bank conflicts)
    static constexpr int kWarpRows = QW == 4 ? 16 : kMaxGroup;  // rows of a warp's merge deposit
    static constexpr int kWarpFloats = kWarpRows * kOStride + 2 * kWarpRows;
    static constexpr int kMergeOff = kQOff + kQSlots * kQSlot;
    static constexpr int kMergeSlot = kNcw * kWarpFloats;  // floats per merge slot
    static constexpr int kMergeBars = 2;  // merge_full / merge_done barriers each (QW = 4: per group)
    static constexpr int kBarOff = kMergeOff + MSLOTS * kMergeSlot * 4;
    // full, empty, qfull, qempty, merge_full, merge_done, epi_ready, epi_free
    static constexpr int kNumBars = 2 * STAGES + 2 * kQSlots + 2 * kMergeBars + 2 * kEpiRing;
    static constexpr int kNValidOff = kBarOff + kNumBars * 8;
    static constexpr int kAbortOff = kNValidOff + STAGES * 4;  // abort flag
    static constexpr int kInfoOff = round_up(kAbortOff + 16, 64);  // one DescInfo per Q slot
    static constexpr int kEpiOff = kInfoOff + kQSlots * kDescInfoBytes;  // kEpiRing EpiRecords + descriptor total
    static constexpr int kBytes = kEpiOff + kEpiRing * 16 + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024
    static_assert(MSLOTS == 1 || MSLOTS == 2, "merge slots");
    static_assert(QW == 0 || QW == 4, "kernel shapes");
    static_assert(QW == 0 || (MSLOTS == 1 && GROUPS == 2), "multi-token shapes");
    // Each stage must be consumed by one group only: a group then meets the phases of its
    // stages' full barriers in order.  With stages shared by two groups, one group could wait
    // for phase k+1 while phase k is still pending, pass the parity test early and arrive on
    // the stage's empty barrier out of turn (an undefined mbarrier use that faults the GPU).
    static_assert(STAGES % GROUPS == 0, "each stage must belong to one consumer group");
    static_assert(kStageBytes % 1024 == 0 && kQOff % 1024 == 0, "swizzled TMA boxes need 1024-byte alignment");
    static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

// What the consumers hand the epilogue warp with each merged descriptor (fused combine).
struct EpiRecord {
    int b, h, np, pbeg;
};


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
    EpiRecord *epi_rec = reinterpret_cast<EpiRecord *>(smem + L::kEpiOff);
    volatile int *epi_total = reinterpret_cast<volatile int *>(smem + L::kEpiOff + kEpiRing * sizeof(EpiRecord));
    int *nvalid = reinterpret_cast<int *>(smem + L::kNValidOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kAbortOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 4);  // one consumer group releases a stage
        }
        for (int s = 0; s < kQSlots; ++s) {
            mbar_init(qfull_bar(s), 1);
            mbar_init(qempty_bar(s), NCW);  // every warp that reads the hand-off
        }
        if (QW == 4) {
            for (int s = 0; s < 2; ++s) {  // one pair per consumer group
                mbar_init(merge_full(s), 4);
                mbar_init(merge_done(s), 4);
            }
        } else {
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

    // The next kernel may start only once this one has waited for its predecessor, so that
    // whatever it reads before its own wait (the combine: the task map's unit arrays) comes from
    // kernels that have completed.  Early KV gather (dsa_decode_chained): the producer warp
    // waits later, after issuing the tiles it may load before the preceding kernel completes.
    if (p.early == 0 || warp != NCW) {
        grid_dependency_wait();  // task map, lengths, pages and Q from earlier kernels
        grid_launch_dependents();
    }
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
        // (the producer of dsa_decode_chained reads these before its wait)
        d_begin = early_load<!FUSE && QW == 0>(p.cta_desc_begin + blockIdx.x);
        d_count = early_load<!FUSE && QW == 0>(p.cta_desc_begin + blockIdx.x + 1) - d_begin;
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
        producer_warp<KV, STAGES, PERSIST, FUSE, false, L, PERSIST && !FUSE && QW == 0>(
            &kmap, &vmap, p, smem, sbase, bar0, nvalid, abort_flag, epi_total, d_begin, d_count, st0, st1, lane);
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

    if constexpr (QW == 4) {
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

}  // namespace

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

namespace {

template <int KV, int STAGES, int GROUPS, bool PERSIST, bool FUSE = false, int MSLOTS = 2, int QW = 0>
dsa_status launch(const AttnArgs &a, const KernelParams &kp, dim3 grid, cudaStream_t st) {
    using L = Layout<KV, STAGES, GROUPS, MSLOTS, QW>;
    CUtensorMap km, vm;
    const bool nhd = a.kv_layout == DSA_NHD;
    if (!make_pool_map(&km, a.k_pages, KV, a.num_pages, a.num_kv_heads, a.page_size, nhd, false) ||
        !make_pool_map(&vm, a.v_pages, KV, a.num_pages, a.num_kv_heads, a.page_size, nhd, false))
        return DSA_ERR_CUDA;
    auto kern = attn_kernel<KV, STAGES, GROUPS, PERSIST, FUSE, MSLOTS, QW>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) != cudaSuccess)
        return DSA_ERR_CUDA;
    return launch_pdl(kern, grid, dim3(FUSE ? L::kThreadsFused : L::kThreads), L::kAlloc, st, km, vm, kp);
}


// CTA shapes.  One persistent CTA per SM: two consumer groups and a deep ring.  Two CTAs per
// SM (used by the static grid, and by the persistent kernel when the task map has at least
// two bins per SM): one consumer group and a shallow ring each, so both fit in shared memory.
// (A sweep on the GB300 found the lagged two-slot merge with 4 / 8 stages faster than one
// merge slot with the same or deeper rings.)
constexpr int kPersistStagesBf16 = 4, kPersistStagesFp8 = 8, kPersistGroups = 2, kPersistMergeSlots = 2;
constexpr int kPairStagesBf16 = 2, kPairStagesFp8 = 4, kPairGroups = 1;
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

dsa_status launch_decode(const AttnArgs &a, const KernelParams &kp, int num_ctas, bool fused, cudaStream_t st) {
    if (a.kv_dtype == DSA_BF16)
        return fused ? launch_persistent<0, true>(a, kp, num_ctas, st) : launch_persistent<0, false>(a, kp, num_ctas, st);
    return fused ? launch_persistent<1, true>(a, kp, num_ctas, st) : launch_persistent<1, false>(a, kp, num_ctas, st);
}

dsa_status launch_multi_mma(const AttnArgs &a, const KernelParams &kp, int num_ctas, cudaStream_t st) {
    return launch<1, kMultiStagesFp8, 2, true, false, 1, 4>(a, kp, dim3(num_ctas), st);
}

dsa_status launch_static(const AttnArgs &a, const KernelParams &kp, dim3 grid, cudaStream_t st) {
    if (a.kv_dtype == DSA_BF16) return launch<0, kPairStagesBf16, kPairGroups, false>(a, kp, grid, st);
    return launch<1, kPairStagesFp8, kPairGroups, false>(a, kp, grid, st);
}

dsa_status launch_wait_selftest(int32_t *status, uint64_t limit_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 64, 0, st>>>(status, limit_ns);
    return launch_status();
}

}  // namespace dsa
