// Multi-token decode (q_len query tokens per request: a verify step of a draft; Hy3 preview
// write-up 2.5 "MTP与异步调度优化"; SGLang Low-Latency Mode: Kernels and Runtime, section 1) on
// the 5th-generation tensor cores.  The scheduler, the task map and the producer warp are
// those of the one-token kernel (engine.cuh: each resident CTA drains its bin of descriptors,
// HPC-Ops × SGLang blog, "围绕活跃 KV 工作进行调度"); every KV tile serves all q_len x G query
// rows of its unit.  Only the consumers differ: S = Q K^T and O = P V accumulate in tensor
// memory (tcgen05.mma, M = 64), two teams of four softmax warps take alternate tiles, one
// warp issues S (and lays Q out as its operand; bf16 with at most 48 query rows: the fourth
// warp of each team, whose rows are all padding, does that instead), one issues P.V.  Each team writes its own
// partial at a descriptor end (two slots per descriptor).
#include "engine.cuh"

namespace dsa {
namespace {

// Shared memory of the tensor-memory kernel.  From the base: STAGES ring stages (K tile, V
// tile, E4M3 scales; E4M3 also a V tile widened to f16), the plain Q rows of kQSlots
// descriptors, two Q operand buffers, the barriers, the stages' valid-token counts, the abort
// flag and tensor-memory address, the descriptor hand-off records.
template <int KV, int STAGES>
struct TcLayout {
    static constexpr int kQSlots = 2;  // descriptors handed ahead to the consumers
    static constexpr int kNcw = 8;     // softmax warps (two teams of four)
    static constexpr int kThreads = (kNcw + 3) * 32;  // + producer, S and PV warps
    static constexpr int kStageTx = 2 * Cfg<KV>::kTileBytes + 2 * Cfg<KV>::kScaleBytes;
    // E4M3: each stage also holds its V widened to f16 ([half][64 rows][128 B], 128-byte
    // swizzle: the P.V operand layout of a bf16 V tile)
    static constexpr int kVcOff = round_up(kStageTx, 1024);
    static constexpr int kStageBytes = kVcOff + (KV == 1 ? kTile * kHeadDim * 2 : 0);
    static constexpr int kQSlot = kMaxRows * Cfg<KV>::kQHeadBytes;
    static constexpr int kQOff = STAGES * kStageBytes;
    // Q as the MMA's A operand (64 rows x 128, K-major with the 128-byte swizzle, two 64-column
    // halves of 8 KB for bf16, as the TMA lays out a K tile), two buffers
    static constexpr int kQcOff = kQOff + kQSlots * kQSlot;
    static constexpr int kQcBytes = 2 * kMaxRows * Cfg<KV>::kQHeadBytes;
    static constexpr int kBarOff = kQcOff + kQcBytes;
    // full, empty, qfull, qempty; s_full, s_free, p_full x4; o_done, o_free, qc_full, qc_free, qd_full x2
    static constexpr int kTcBars = 22;
    static constexpr int kNumBars = 2 * STAGES + 2 * kQSlots + kTcBars;
    static constexpr int kNValidOff = kBarOff + kNumBars * 8;
    // abort flag, the TMEM base address, the slots of the descriptors in the two Q operand
    // buffers (written by the Q helpers)
    static constexpr int kAbortOff = kNValidOff + STAGES * 4;
    static constexpr int kInfoOff = round_up(kAbortOff + 16, 64);  // one DescInfo per Q slot
    static constexpr int kBytes = kInfoOff + kQSlots * kDescInfoBytes;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024
    static_assert(kQcOff % 1024 == 0, "tensor-core operand buffers");
    static_assert(kStageBytes % 1024 == 0 && kQOff % 1024 == 0, "swizzled TMA boxes need 1024-byte alignment");
    static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

// 16 TMEM lanes x 64 columns over the warp in one load: v[k] holds columns 8 k .. 8 k + 7
// as an m16n8 accumulator fragment (the layout of tmem_ld16x8, eight times side by side).
__device__ __forceinline__ void tmem_ld16x64(uint32_t taddr, float (&v)[8][4]) {
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                 "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i >> 2][i & 3] = __uint_as_float(r[i]);
}

// 16 TMEM lanes x 32 columns over the warp in one store: w[2 k] and w[2 k + 1] go where
// tmem_st16x4 at column 4 k puts its two words (eight of those side by side).
__device__ __forceinline__ void tmem_st16x32(uint32_t taddr, const uint32_t (&w)[16]) {
    asm volatile("tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                 "%13, %14, %15, %16};" ::"r"(taddr),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]),
                 "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
                 : "memory");
}

// Four E4M3 bytes (byte k -> element k) to two f16x2 words, exactly.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t x, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}

// The descriptor end of one softmax team.  It waits until the team's products of the
// descriptor are done (its last tile's phase of o_done; that commit covers every earlier
// product), reads O_team (o_tmem: the warp's lane quarter, O's first column) into registers,
// releases it (o_free) and writes the team's partial for rows ra, rb (< R): O / l (E4M3: times
// the V scale reference vref, by which O was divided) and lse = ln 2 (m + log2 l), slot
// 2 x descriptor + team.
template <int KV>
static __device__ __forceinline__ bool tc_team_epilogue(float *partial_o, float *partial_lse, int32_t *status,
                                                        volatile int *abort_flag, uint32_t o_done_bar,
                                                        uint32_t o_free_bar, uint32_t o_tmem, int R, int ra, int rb,
                                                        int tig, int lane, int team, int slot, float m0, float m1,
                                                        float l0, float l1, int pv_desc, int last_g, float vref) {
    if (last_g >= 0) {
        if (!wait_phase(o_done_bar, (last_g >> 1) & 1, abort_flag, status)) return false;
        tc_fence_after();
    }
    const float m[2] = {m0, m1};
    float l[2] = {l0, l1}, inv[2], lse[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
        inv[h] = l[h] > 0.f ? (KV == 0 ? 1.f : vref) / l[h] : 0.f;
        lse[h] = l[h] > 0.f ? (m[h] + lg2(l[h])) * kLn2 : -INFINITY;
    }
    const int64_t slot_row = (2 * static_cast<int64_t>(slot) + team) * R;
    float *dst_a = partial_o + (slot_row + ra) * kHeadDim + 2 * tig;
    float *dst_b = partial_o + (slot_row + rb) * kHeadDim + 2 * tig;
    // O_t into registers first, then release it for the next descriptor's products
    float o[16][4];
    if (pv_desc > 0) {
#pragma unroll
        for (int k = 0; k < 16; ++k) tmem_ld16x8(o_tmem + 8 * k, o[k]);
        tmem_wait_ld();
    } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) o[k][0] = o[k][1] = o[k][2] = o[k][3] = 0.f;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(o_free_bar);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        if (ra < R) *reinterpret_cast<float2 *>(dst_a + 8 * k) = make_float2(o[k][0] * inv[0], o[k][1] * inv[0]);
        if (rb < R) *reinterpret_cast<float2 *>(dst_b + 8 * k) = make_float2(o[k][2] * inv[1], o[k][3] * inv[1]);
    }
    if (tig == 0) {
        if (ra < R) partial_lse[slot_row + ra] = lse[0];
        if (rb < R) partial_lse[slot_row + rb] = lse[1];
    }
    return true;
}

// The same kept out of line: one copy of its code for the kernel's four call sites, which
// the E4M3 kernel's instruction cache needs (measured 7% faster at q_len 6 there; the bf16
// kernel, with more descriptor ends per tile, is faster with it inline).
template <int KV>
static __device__ __noinline__ bool tc_team_epilogue_call(float *partial_o, float *partial_lse, int32_t *status,
                                                          volatile int *abort_flag, uint32_t o_done_bar,
                                                          uint32_t o_free_bar, uint32_t o_tmem, int R, int ra, int rb,
                                                          int tig, int lane, int team, int slot, float m0, float m1,
                                                          float l0, float l1, int pv_desc, int last_g, float vref) {
    return tc_team_epilogue<KV>(partial_o, partial_lse, status, abort_flag, o_done_bar, o_free_bar, o_tmem, R, ra, rb,
                                tig, lane, team, slot, m0, m1, l0, l1, pv_desc, last_g, vref);
}

template <int KV, int STAGES>
__global__ void __launch_bounds__(TcLayout<KV, STAGES>::kThreads, 1)
    tc_attn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const KernelParams p) {
    using L = TcLayout<KV, STAGES>;
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
    const uint32_t tc_bar0 = bar0 + 8u * (2 * STAGES + 2 * kQSlots);
    auto s_full = [&](int b) { return tc_bar0 + 8u * b; };         // 4 S/P buffers
    auto s_free = [&](int b) { return tc_bar0 + 8u * (4 + b); };
    auto p_full = [&](int b) { return tc_bar0 + 8u * (8 + b); };
    auto o_done = [&](int t) { return tc_bar0 + 8u * (12 + t); };  // 2 softmax teams
    auto o_free = [&](int t) { return tc_bar0 + 8u * (14 + t); };
    auto qc_full = [&](int b) { return tc_bar0 + 8u * (16 + b); };
    auto qc_free = [&](int b) { return tc_bar0 + 8u * (18 + b); };
    auto qd_full = [&](int b) { return tc_bar0 + 8u * (20 + b); };  // plain Q rows landed
    int *nvalid = reinterpret_cast<int *>(smem + L::kNValidOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kAbortOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G;
    // bf16 with at most 48 query rows per unit: the fourth warp of each team holds only
    // padding rows, and lays out Q for the S warp instead of joining the team's softmax
    const bool helpers = KV == 0 && p.q_len * G <= 48;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 2);  // the S and PV warps each release their half of a stage
        }
        for (int s = 0; s < kQSlots; ++s) {
            mbar_init(qfull_bar(s), 1);
            mbar_init(qempty_bar(s), helpers ? NCW : NCW + 2);  // every warp that reads the hand-off (not the Q helpers)
        }
        for (int b = 0; b < 4; ++b) {
            mbar_init(s_full(b), 1);  // S warp
            mbar_init(s_free(b), 1);  // PV warp: the buffer's P has been read
            mbar_init(p_full(b), helpers ? 3 : 4);  // the owning softmax team
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(o_done(b), 1);
            mbar_init(o_free(b), helpers ? 3 : 4);
            mbar_init(qc_full(b), 1);
            mbar_init(qc_free(b), 1);
            mbar_init(qd_full(b), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // released after the wait: the combine reads the task map before its own wait
    grid_dependency_wait();  // task map, lengths, pages and Q from earlier kernels
    grid_launch_dependents();
    EndStamp end_stamp{nullptr};
    if (p.cta_times) {  // uniform over the CTA
        uint64_t *t = p.cta_times + 2 * blockIdx.x;
        if (threadIdx.x == 0) t[0] = t[1] = globaltimer_ns();
        __syncthreads();
        end_stamp.at = t + 1;
    }
    const int d_begin = p.cta_desc_begin[blockIdx.x];
    const int d_count = p.cta_desc_begin[blockIdx.x + 1] - d_begin;
    if (d_count <= 0) return;

    if (warp == NCW) {
        producer_warp<KV, STAGES, true, false, true, L>(&kmap, &vmap, p, smem, sbase, bar0, nvalid, abort_flag,
                                                        nullptr, d_begin, d_count, 0, 0, lane);
        return;
    }

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
        //      into one of two buffers), lays them out as the A operand (zero past R; bf16 with
        //      at most 48 rows: waits for the Q helpers, which do both, instead), then
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
        // bf16: rows R .. 63 of both Q operand buffers are zero for the whole launch (R is fixed);
        // the per-descriptor layout writes rows 0 .. R - 1 only
        if constexpr (KV == 0) {
            for (int i = lane; i < 2 * (kMaxRows - R) * 16; i += 32) {
                const int b = i / ((kMaxRows - R) * 16), rem = i - b * ((kMaxRows - R) * 16);
                const int r = R + (rem >> 4), kc = rem & 15;
                *reinterpret_cast<uint4 *>(smem + L::kQcOff + b * kQcBuf + (kc >> 3) * 8192 + r * 128 +
                                           (((kc & 7) ^ (r & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
        }
        // the descriptor whose Q is in flight (none with helpers: they fetch it)
        int pf_slot = helpers ? -1 : next_desc(d_begin - 1), pf_buf = 0;
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
            if (!end && helpers) {
                // laid out by the helper of team d % 2 in operand buffer d % 2, which follows the
                // same descriptor sequence (a mismatch would be a map the two read differently)
                if (!wait_phase(qc_full(d & 1), (d >> 1) & 1, abort_flag, p.status)) {
                    failed = true;
                    break;
                }
                if (lane == 0 && *reinterpret_cast<volatile int *>(smem + L::kAbortOff + 8 + 4 * (d & 1)) != xs)
                    atomicOr(p.status, DSA_DEV_BAD_MAP);
            } else if (!end) {
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
                // quarter-warp writes one 128-byte row: no bank conflicts either way.  Rows R .. 63
                // stay as zeroed at the start.  A negative softmax scale is moved onto Q (its sign
                // bits flipped, exact), so that the softmax sees S x |scale| and may take the
                // maximum of the raw scores.
                const uint32_t qneg = p.score_scale < 0.f ? 0x80008000u : 0u;
#pragma unroll
                for (int rd = 0; rd < 4; ++rd) {
                    if (16 * rd >= R) break;  // rows 16 rd .. are padding
                    uint4 v[8];
#pragma unroll
                    for (int it = 0; it < 8; ++it) {  // chunk kc of row r
                        const int i = lane + 32 * (8 * rd + it), r = i >> 4, kc = i & 15;
                        if (r < R) {
                            v[it] = *reinterpret_cast<const uint4 *>(src + r * (kHeadDim * 2) + kc * 16);
                            v[it].x ^= qneg, v[it].y ^= qneg, v[it].z ^= qneg, v[it].w ^= qneg;
                        }
                    }
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int i = lane + 32 * (8 * rd + it), r = i >> 4, kc = i & 15;
                        if (r < R)
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
    } else if (helpers && (warp & 3) == 3) {
        // ---- Q helper (bf16, at most 48 rows: the fourth warp of team t, whose 16 rows are
        //      all padding).  The descriptors the producer hands over (valid, with tiles) come
        //      in the order of the task map, the d-th of them being the S warp's descriptor d;
        //      the helper walks the map itself (so it never holds up the hand-off ring) and
        //      takes those with d % 2 == t: it fetches the descriptor's Q rows into plain
        //      buffer t, lays them out as the A operand (rows 0 .. R - 1; the S warp zeroed the
        //      rest) in operand buffer t once the S products of descriptor d - 2 have read it,
        //      notes the descriptor's slot for the S warp to check, and signals it
        const int team = warp >> 2;
        const uint32_t qneg = p.score_scale < 0.f ? 0x80008000u : 0u;  // a negative scale moves onto Q
        const uint8_t *src = smem + L::kQOff + team * L::kQSlot;
        uint8_t *dst = smem + L::kQcOff + team * kQcBuf;
        volatile int *laid_slot = reinterpret_cast<volatile int *>(smem + L::kAbortOff + 8) + team;
        int fetched = 0;  // Q copies into plain buffer t, each one waited for
        bool in_flight = false;
        int d = -1;
        for (int base = 0; base < d_count && !failed; base += 32) {
            int wu = -1;  // lane j: the unit of descriptor base + j if it is handed over
            if (base + lane < d_count) {
                const int4 v = p.descs[d_begin + base + lane];
                if (v.x >= 0 && v.x < p.num_units && v.y >= 0 && v.y < v.z && d_begin + base + lane < p.max_slots)
                    wu = v.x;
            }
            for (uint32_t valid = __ballot_sync(0xffffffffu, wu >= 0); valid; valid &= valid - 1) {
                const int j = __ffs(valid) - 1;
                if (((++d) & 1) != team) continue;
                const int u = __shfl_sync(0xffffffffu, wu, j), b = u / p.hkv, h = u - b * p.hkv;
                if (lane == 0) {
                    const uint32_t bytes = G * C::kQHeadBytes;
                    mbar_arrive_expect_tx(qd_full(team), bytes * p.q_len);
                    for (int i = 0; i < p.q_len; ++i)
                        bulk_load(sbase + L::kQOff + team * L::kQSlot + i * bytes,
                                  p.q + ((static_cast<int64_t>(b) * p.q_len + i) * p.hq + h * G) * C::kQHeadBytes,
                                  bytes, qd_full(team));
                }
                ++fetched;
                in_flight = true;
                if (!wait_phase(qd_full(team), (fetched - 1) & 1, abort_flag, p.status)) {
                    failed = true;
                    break;
                }
                in_flight = false;
                if (!wait_phase(qc_free(team), ((d >> 1) & 1) ^ 1, abort_flag, p.status)) {
                    failed = true;
                    break;
                }
                if (lane == 0) *laid_slot = d_begin + base + j;
                // the S warp's layout (128-byte swizzle, K-major), rows 0 .. R - 1
#pragma unroll
                for (int rd = 0; rd < 3; ++rd) {
                    if (16 * rd >= R) break;
                    uint4 v[8];
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int i = lane + 32 * (8 * rd + it), r = i >> 4, kc = i & 15;
                        if (r < R) {
                            v[it] = *reinterpret_cast<const uint4 *>(src + r * (kHeadDim * 2) + kc * 16);
                            v[it].x ^= qneg, v[it].y ^= qneg, v[it].z ^= qneg, v[it].w ^= qneg;
                        }
                    }
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int i = lane + 32 * (8 * rd + it), r = i >> 4, kc = i & 15;
                        if (r < R)
                            *reinterpret_cast<uint4 *>(dst + (kc >> 3) * 8192 + r * 128 + (((kc & 7) ^ (r & 7)) << 4)) =
                                v[it];
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(qc_full(team));
            }
        }
        if (in_flight) {  // a Q copy still in flight lands before the CTA leaves
            const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
            drain_phase(qd_full(team), (fetched - 1) & 1, deadline);
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
        const bool rows = 16 * sp < R;  // the warp holds at least one query row (warp-uniform)
        const uint32_t lane_base = static_cast<uint32_t>(32 * sp) << 16;
        const uint32_t o_col = 256 + 128 * team;
        const int tid = sp * 32 + lane;  // within the team
        // The descriptor end of a team (its partial, slot 2 x descriptor + team), deferred
        // until the team has handed over the P of its first tile of the next descriptor: a
        // descriptor's first tile never rescales O, so it need not wait for the previous
        // descriptor's last P.V, and the team computes it while that P.V completes.
        float ep_vref = 1.f;  // E4M3: the V scale reference of the deferred descriptor end
        auto team_epilogue = [&](int slot, float (&m)[2], float (&l)[2], int pv_desc, int last_g) -> bool {
            if constexpr (KV == 1)
                return tc_team_epilogue_call<KV>(p.partial_o, p.partial_lse, p.status, abort_flag, o_done(team),
                                                 o_free(team), tmem + lane_base + o_col, R, ra, rb, tig, lane, team,
                                                 slot, m[0], m[1], l[0], l[1], pv_desc, last_g, ep_vref);
            else
                return tc_team_epilogue<KV>(p.partial_o, p.partial_lse, p.status, abort_flag, o_done(team),
                                            o_free(team), tmem + lane_base + o_col, R, ra, rb, tig, lane, team, slot,
                                            m[0], m[1], l[0], l[1], pv_desc, last_g, ep_vref);
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
            // the team's tiles of this descriptor: every other one, from the first of parity team
            const int g_first = g;
            g += n;
            for (int li = (team - g_first) & 1; li < n; li += 2) {
                const int g = g_first + li;  // the tile's position in the CTA's stream
                const int c = c_start + li, stage = c % STAGES, buf = g & 3;
                if (!wait_phase(full_bar(stage), (c / STAGES) & 1, abort_flag, p.status) ||
                    !wait_phase(s_full(buf), (g >> 2) & 1, abort_flag, p.status)) {
                    failed = true;
                    break;
                }
                const int nv = nvalid[stage];
                tc_fence_after();
                float sv[8][4];  // [column block k][(ra, 2tig), (ra, 2tig+1), (rb, 2tig), (rb, 2tig+1)]
                if (nv > 0 && rows) {
                    if constexpr (KV == 1) {
                        tmem_ld16x64(tmem + lane_base + 64 * buf, sv);
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k) tmem_ld16x8(tmem + lane_base + 64 * buf + 8 * k, sv[k]);
                    }
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
                // O_team rows ra, rb *= fa, fb, after the team's previous P.V into it
                auto rescale_o = [&](float fa, float fb) -> bool {
                    if (!wait_prev_pv()) return false;
                    tc_fence_after();
#pragma unroll 1  // rare: kept small for the instruction cache
                    for (int half = 0; half < 2; ++half) {
                        float o[8][4];
#pragma unroll
                        for (int k = 0; k < 8; ++k) tmem_ld16x8(tmem + lane_base + o_col + 64 * half + 8 * k, o[k]);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            o[k][0] *= fa;
                            o[k][1] *= fa;
                            o[k][2] *= fb;
                            o[k][3] *= fb;
                            tmem_st16x8(tmem + lane_base + o_col + 64 * half + 8 * k, o[k]);
                        }
                        tmem_wait_st();
                    }
                    return true;
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
                // A warp whose 16 rows all lie past R (rows 48-63 at q_len 6 and G = 8) has no
                // softmax to do: its rows of S are zero (Q is zero there), their P lanes keep
                // those zeros, and its rows of O are never read out.  It still takes its share
                // of the stage's V work below and hands the buffer over with the team.
                if constexpr (KV == 0) {
                    if (rows) {
                        // ---- running maximum over each row's visible tokens (t < lim, slot < nv)
                        //      of the raw scores, scaled once: the scale is positive here (the S
                        //      warp negated Q for a negative one; a zero scale is raised to the
                        //      smallest normal float, which gives every visible token weight 1 as 0
                        //      does).  Columns a row may not see are set to -inf first (a branch
                        //      taken only by tiles with such a column), so P = 2^-inf = 0 there.
                        const float sc = fmaxf(fabsf(p.score_scale), 1.17549435e-38f);
                        const int tt = (dt0 + li) * kTile;
                        const int vis0 = max(0, min(nv, lim[0] - tt)), vis1 = max(0, min(nv, lim[1] - tt));
                        if (vis0 < kTile || vis1 < kTile) {
#pragma unroll
                            for (int k = 0; k < 8; ++k)
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int j = 8 * k + 2 * tig + (e & 1);
                                    if (j >= ((e >> 1) ? vis1 : vis0)) sv[k][e] = -INFINITY;
                                }
                        }
                        float mx[2] = {fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[0][2], sv[0][3])};
#pragma unroll
                        for (int k = 1; k < 8; ++k) {
                            mx[0] = max3f(mx[0], sv[k][0], sv[k][1]);
                            mx[1] = max3f(mx[1], sv[k][2], sv[k][3]);
                        }
                        bool grow[2];
                        float alpha[2];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
                            const float mnew = fmaxf(m[h], mx[h] * sc);
                            grow[h] = m[h] != -INFINITY && mnew > m[h] + 8.f;
                            alpha[h] = grow[h] ? ex2(m[h] - mnew) : 1.f;
                            if (grow[h] || m[h] == -INFINITY) m[h] = mnew;
                        }
                        if (__any_sync(0xffffffffu, grow[0] || grow[1])) {
                            if (!rescale_o(alpha[0], alpha[1])) {
                                failed = true;
                                break;
                            }
                            l[0] *= alpha[0];
                            l[1] *= alpha[1];
                        }
                        // ---- P = 2^(s * scale - m) as bf16 high part (the top 16 bits) and low part
                        //      (the rest, rounded), written over S in the buffer: the P.V's A
                        //      operand, tokens (2c, 2c + 1) packed in column c (high part: columns
                        //      0-31, low part: 32-63).  A row that has seen nothing yet has m = -inf
                        //      and only -inf scores: P = 0.
                        const float nm0 = m[0] == -INFINITY ? 0.f : -m[0], nm1 = m[1] == -INFINITY ? 0.f : -m[1];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            float pv[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) pv[e] = ex2(fmaf(sv[k][e], sc, (e >> 1) ? nm1 : nm0));
                            l[0] += pv[0] + pv[1];
                            l[1] += pv[2] + pv[3];
                            const uint32_t h0 = __float_as_uint(pv[0]) & 0xFFFF0000u, h1 = __float_as_uint(pv[1]) & 0xFFFF0000u;
                            const uint32_t h2 = __float_as_uint(pv[2]) & 0xFFFF0000u, h3 = __float_as_uint(pv[3]) & 0xFFFF0000u;
                            tmem_st16x4(tmem + lane_base + 64 * buf + 4 * k, prmt(h0, h1, 0x7632u), prmt(h2, h3, 0x7632u));
                            tmem_st16x4(tmem + lane_base + 64 * buf + 32 + 4 * k,
                                        pack_bf16x2(pv[0] - __uint_as_float(h0), pv[1] - __uint_as_float(h1)),
                                        pack_bf16x2(pv[2] - __uint_as_float(h2), pv[3] - __uint_as_float(h3)));
                        }
                        tmem_wait_st();
                    }
                } else if (rows) {
                    // ---- E4M3: base-2 scores t = s x score scale x the row's Q scale x the
                    //      column's K scale, two columns per instruction, scaled before the maximum
                    //      (any sign of the scales is handled).  P's factor per column: the V scale
                    //      over the reference, which moves only when a larger scale appears (O is
                    //      then rescaled with the maxima below); columns past nv get 0
                    float2 vw[8];
                    float vf = 1.f;
                    const float *ksm = reinterpret_cast<const float *>(smem + stage * L::kStageBytes + 2 * C::kTileBytes);
                    const float *vsm = ksm + kTile;
                    const float2 qa = make_float2(qsc[0], qsc[0]), qb = make_float2(qsc[1], qsc[1]);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int j = 8 * k + 2 * tig;
                        const float2 kk = *reinterpret_cast<const float2 *>(ksm + j);
                        vw[k] = *reinterpret_cast<const float2 *>(vsm + j);
                        const float2 a = mul2(make_float2(sv[k][0], sv[k][1]), mul2(kk, qa));
                        const float2 b = mul2(make_float2(sv[k][2], sv[k][3]), mul2(kk, qb));
                        sv[k][0] = a.x, sv[k][1] = a.y, sv[k][2] = b.x, sv[k][3] = b.y;
                    }
                    if (nv < kTile) {  // uniform over the CTA: the stage's valid-token count
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int j = 8 * k + 2 * tig;
                            if (j >= nv) vw[k].x = 0.f;
                            if (j + 1 >= nv) vw[k].y = 0.f;
                        }
                    }
                    float vmax = fmaxf(vw[0].x, vw[0].y);
#pragma unroll
                    for (int k = 1; k < 8; ++k) vmax = max3f(vmax, vw[k].x, vw[k].y);
                    if (__any_sync(0xffffffffu, vmax > vref)) {  // the quad's four lanes cover the 64 columns
                        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 1));
                        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));
                        if (vmax > vref) {
                            if (vref > 0.f) vf = vref / vmax;  // from 0: nothing accumulated yet
                            vref = vmax;
                            vinv = 1.f / vmax;
                        }
                    }
                    const float2 vi = make_float2(vinv, vinv);
#pragma unroll
                    for (int k = 0; k < 8; ++k) vw[k] = mul2(vw[k], vi);
                    // ---- columns a row may not see (slot >= nv, past its draft token's causal
                    //      limit, or a row past R) are -inf: P = 2^-inf = 0 there, whatever the
                    //      slot held
                    const int tt = (dt0 + li) * kTile;
                    const int vis0 = max(0, min(nv, lim[0] - tt)), vis1 = max(0, min(nv, lim[1] - tt));
                    if (vis0 < kTile || vis1 < kTile) {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int j = 8 * k + 2 * tig + (e & 1);
                                if (j >= ((e >> 1) ? vis1 : vis0)) sv[k][e] = -INFINITY;
                            }
                    }
                    // ---- running maximum of each row (three-input maxima, then the quad)
                    float mx[2] = {fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[0][2], sv[0][3])};
#pragma unroll
                    for (int k = 1; k < 8; ++k) {
                        mx[0] = max3f(mx[0], sv[k][0], sv[k][1]);
                        mx[1] = max3f(mx[1], sv[k][2], sv[k][3]);
                    }
                    bool grow[2];
                    float alpha[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
                        const float mnew = fmaxf(m[h], mx[h]);
                        grow[h] = m[h] != -INFINITY && mnew > m[h] + 8.f;
                        alpha[h] = grow[h] ? ex2(m[h] - mnew) : 1.f;
                        if (grow[h] || m[h] == -INFINITY) m[h] = mnew;
                    }
                    // rows whose maximum grew, and all rows by the V reference's change
                    if (__any_sync(0xffffffffu, grow[0] || grow[1] || vf != 1.f)) {
                        if (!rescale_o(alpha[0] * vf, alpha[1] * vf)) {
                            failed = true;
                            break;
                        }
                        l[0] *= alpha[0];
                        l[1] *= alpha[1];
                    }
                    // ---- P = 2^(t - m) x the column's V factor (<= 2^8) as f16, written over S
                    //      in the buffer, tokens (2c, 2c + 1) packed in column c: the P.V's A
                    //      operand.  A row that has seen nothing yet has m = -inf and only -inf
                    //      scores: P = 0.
                    const float n0 = m[0] == -INFINITY ? 0.f : -m[0], n1 = m[1] == -INFINITY ? 0.f : -m[1];
                    const float2 nm0 = make_float2(n0, n0), nm1 = make_float2(n1, n1);
                    float2 la = make_float2(0.f, 0.f), lb = la;
                    uint32_t pw[16];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        float2 a = add2(make_float2(sv[k][0], sv[k][1]), nm0);
                        float2 b = add2(make_float2(sv[k][2], sv[k][3]), nm1);
                        a = make_float2(ex2(a.x), ex2(a.y));
                        b = make_float2(ex2(b.x), ex2(b.y));
                        la = add2(la, a);
                        lb = add2(lb, b);
                        a = mul2(a, vw[k]);
                        b = mul2(b, vw[k]);
                        pw[2 * k] = pack_f16x2(a.x, a.y), pw[2 * k + 1] = pack_f16x2(b.x, b.y);
                    }
                    tmem_st16x32(tmem + lane_base + 64 * buf, pw);
                    l[0] += la.x + la.y;
                    l[1] += lb.x + lb.y;
                    tmem_wait_st();
                }
                if constexpr (KV == 0) {
                    // ---- V rows past the request's length are zeroed (stale or NaN slots of the page)
                    if (nv < kTile) {
                        uint8_t *vt = smem + stage * L::kStageBytes + C::kTileBytes;
                        for (int i = tid; i < (kTile - nv) * 16; i += helpers ? 96 : 128) {
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
                    auto widen = [&](int t, int c, uint4 x) {
                        uint4 lo, hi;
                        e4m3x4_to_f16x4(x.x, lo.x, lo.y);
                        e4m3x4_to_f16x4(x.y, lo.z, lo.w);
                        e4m3x4_to_f16x4(x.z, hi.x, hi.y);
                        e4m3x4_to_f16x4(x.w, hi.z, hi.w);
                        uint8_t *row = vc + (c >> 2) * 8192 + t * 128;  // half c / 4, chunks 2 (c % 4), + 1
                        const int cc = 2 * (c & 3);
                        *reinterpret_cast<uint4 *>(row + ((cc ^ (t & 7)) << 4)) = lo;
                        *reinterpret_cast<uint4 *>(row + (((cc + 1) ^ (t & 7)) << 4)) = hi;
                    };
                    if (nv == kTile) {  // uniform over the CTA: a full tile, no row to zero
#pragma unroll
                        for (int it = 0; it < 4; ++it) {
                            const int i = tid + 128 * it, t = i >> 3, c = i & 7;
                            widen(t, c, *reinterpret_cast<const uint4 *>(vr + t * 128 + ((c ^ (t & 7)) << 4)));
                        }
                    } else {
#pragma unroll 1
                        for (int it = 0; it < 4; ++it) {
                            const int i = tid + 128 * it, t = i >> 3, c = i & 7;
                            widen(t, c, t < nv ? *reinterpret_cast<const uint4 *>(vr + t * 128 + ((c ^ (t & 7)) << 4))
                                               : make_uint4(0u, 0u, 0u, 0u));
                        }
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
}

}  // namespace

// The tensor-memory kernel needs its stages from the load of a tile until its P.V, several
// microseconds; P lives in tensor memory, so shared memory holds five stages.
constexpr int kTcStages = 5;

dsa_status launch_tc(const AttnArgs &a, const KernelParams &kp, int num_ctas, cudaStream_t st) {
    const bool nhd = a.kv_layout == DSA_NHD;
    const int kv = a.kv_dtype == DSA_BF16 ? 0 : 1;
    // bf16 pages smaller than the tile: each 128-byte half of a page is its own box, so that a
    // stage lands as [half][64 rows][128 B], the operand layout
    const bool split = kv == 0 && a.page_size < kTile;
    CUtensorMap km, vm;
    if (!make_pool_map(&km, a.k_pages, kv, a.num_pages, a.num_kv_heads, a.page_size, nhd, split) ||
        !make_pool_map(&vm, a.v_pages, kv, a.num_pages, a.num_kv_heads, a.page_size, nhd, split))
        return DSA_ERR_CUDA;
    auto go = [&](auto kern, int smem, int threads) -> dsa_status {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return DSA_ERR_CUDA;
        return launch_pdl(kern, dim3(num_ctas), dim3(threads), smem, st, km, vm, kp);
    };
    if (kv == 0)
        return go(tc_attn_kernel<0, kTcStages>, TcLayout<0, kTcStages>::kAlloc, TcLayout<0, kTcStages>::kThreads);
    return go(tc_attn_kernel<1, kTcStages>, TcLayout<1, kTcStages>::kAlloc, TcLayout<1, kTcStages>::kThreads);
}

}  // namespace dsa
