// The engine shared by the decode kernels: launch parameters, the descriptor hand-off, the
// bounded waits and the producer warp that streams the paged K/V tiles into a ring of
// shared-memory stages (HPC-Ops × SGLang blog, "围绕活跃 KV 工作进行调度": each resident CTA
// drains its bin of descriptors, one or more contiguous 64-token tiles of one (request, KV
// head) each).  Both the mma.sync kernels (attention.cu) and the tensor-memory multi-token
// kernel (attention_tc.cu) run this producer; only their consumers differ.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.h"
#include "ptx.cuh"

namespace dsa {

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
    // early KV gather (dsa_decode_chained): the producer loads the first ring pass of tiles that
    // hold none of the newest new_tokens tokens of their request before waiting for the
    // preceding kernel (which writes those tokens and Q)
    int32_t early, new_tokens;
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

// Loads that a producer with the early KV gather may issue before its grid dependency wait go
// to L2 (ld.global.cg), past any line this SM cached before the data's writer completed.
template <bool EARLY, typename T>
__device__ __forceinline__ T early_load(const T *ptr) {
    if constexpr (EARLY)
        return __ldcg(ptr);
    else
        return *ptr;
}

template <bool PERSIST, bool EARLY = false>
__device__ __forceinline__ Desc get_desc(const KernelParams &p, int d_begin, int i, int t0s, int t1s) {
    Desc x;
    if (PERSIST) {
        const int4 v = early_load<EARLY>(p.descs + d_begin + i);
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
static __device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
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
static __device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           int32_t *status, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_test_wait(bar, parity)) return true;
    return wait_phase_slow(bar, parity, abort_flag, status, limit_ns);
}

// Wait used while draining after an abort: ignores the abort flag; gives up at `deadline`
// (%globaltimer ns), shared by all the drain's waits.
static __device__ __noinline__ void drain_phase(uint32_t bar, uint32_t parity, uint64_t deadline) {
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() > deadline) return;
    }
}

// 5-D TMA view of a page pool (attention.cu).
bool make_pool_map(CUtensorMap *m, const void *pool, int kv, int num_pages, int hkv, int page, bool nhd, bool split);

// The tensor-memory multi-token kernel over a task map's num_ctas bins (attention_tc.cu).
dsa_status launch_tc(const AttnArgs &a, const KernelParams &kp, int num_ctas, cudaStream_t st);

// attention.cu: the launch parameters every decode call starts from, and its kernels' launchers
// (the CTA shape is chosen from the bin count and the SM count).
KernelParams base_params(const AttnArgs &a, float *partial_o, float *partial_lse, int32_t *status);
dsa_status launch_decode(const AttnArgs &a, const KernelParams &kp, int num_ctas, bool fused, cudaStream_t st);
dsa_status launch_multi_mma(const AttnArgs &a, const KernelParams &kp, int num_ctas, cudaStream_t st);
dsa_status launch_static(const AttnArgs &a, const KernelParams &kp, dim3 grid, cudaStream_t st);
dsa_status launch_wait_selftest(int32_t *status, uint64_t limit_ns, cudaStream_t st);

// ---------------------------------------------------------------------------------------
// Producer warp.  L supplies the shared-memory layout (kInfoOff, kQOff, kQSlot, kStageBytes,
// kStageTx, kQSlots); from bar0 the barriers are full[STAGES], empty[STAGES], qfull[kQSlots],
// qempty[kQSlots].  TC: the tensor-memory kernel, whose S warp fetches each descriptor's Q
// itself and whose operands want each 128-byte half of a page smaller than the tile as its
// own box.  EARLY: the early KV gather is built in (it runs when p.early is set).  The whole
// warp calls this; it returns when the CTA's tiles are all issued (or the CTA aborted and its
// copies have landed).
template <int KV, int STAGES, bool PERSIST, bool FUSE, bool TC, class L, bool EARLY = false>
__device__ __forceinline__ void producer_warp(const CUtensorMap *kmap, const CUtensorMap *vmap, const KernelParams &p,
                                              uint8_t *smem, uint32_t sbase, uint32_t bar0, int *nvalid,
                                              volatile int *abort_flag, volatile int *epi_total, int d_begin,
                                              int d_count, int st0, int st1, int lane) {
    using C = Cfg<KV>;
    constexpr int kQSlots = L::kQSlots;
    const int G = p.G;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto qfull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
    auto qempty_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + kQSlots + s); };
    // =========================== producer warp ===========================
    // The CTA's descriptors are read 32 at a time (one per lane, with their
    // lengths and Q scales); their tiles form one stream, mapped 32 at a time
    // onto lanes, whose page ids are fetched one chunk ahead of the chunk whose
    // TMA copies are being issued.  Lane 0 issues; the warp stays converged.
    if (lane == 0) {
        prefetch_tmap(kmap);
        prefetch_tmap(vmap);
    }
    const uint64_t policy = policy_evict_first();
    int c = 0;          // tiles issued so far (ring position)
    int qi = 0;         // descriptors handed to the consumers
    int q_issued = -1;  // hand-off index of the last Q copy issued
    bool aborted = false;
    // early KV gather: the kernel's other warps wait for the preceding kernel at once; this warp
    // first issues the tiles it may (see below), then waits
    bool waited = !EARLY || p.early == 0;
    for (int wbase = 0; wbase < d_count && !aborted; wbase += 32) {
        // ---- window: descriptor wbase + lane
        int wb = 0, wh = 0, wt0 = 0, wn = 0, wslot = 0, wlen = 0, wnp = 1, wpbeg = 0;
        bool wok = false;
        float wqs[kMaxGroup];
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g) wqs[g] = 0.f;
        if (wbase + lane < d_count) {
            const Desc x = get_desc<PERSIST, EARLY>(p, d_begin, wbase + lane, st0, st1);
            if (x.ok) {
                wok = true;
                wb = x.u / p.hkv;
                wh = x.u - wb * p.hkv;
                wt0 = x.t0;
                wn = x.t1 - x.t0;
                wslot = x.slot;
                wlen = early_load<EARLY>(p.seq_lens + wb);
                if (FUSE) {
                    wnp = p.unit_num_partials[x.u];
                    wpbeg = p.unit_partial_begin[x.u];
                }
                if (wlen < 0 || wlen > p.max_pages * p.page_size) atomicOr(p.status, DSA_DEV_BAD_SEQLEN);
            } else {
                atomicOr(p.status, DSA_DEV_BAD_MAP);
            }
        }
        // what depends on the preceding kernel (Q scales) or may race with its reads (partial
        // outputs): after the grid dependency wait
        auto finish_window = [&]() {
            if (wbase + lane >= d_count) return;
            if (KV == 1) {
                const float *qs = p.q_scale + static_cast<int64_t>(wb) * p.hq + wh * G;
#pragma unroll
                for (int g = 0; g < kMaxGroup; ++g)
                    if (g < G) wqs[g] = qs[g];
            }
            if (wok && wn == 0) {  // no tiles: its partials are empty, the consumers never see it
                const int R = p.q_len * G;
                const int64_t s0 = static_cast<int64_t>(wslot) * p.slots_per_desc;
                for (int i = 0; i < p.slots_per_desc * R * kHeadDim; ++i)
                    p.partial_o[s0 * R * kHeadDim + i] = 0.f;
                for (int g = 0; g < p.slots_per_desc * R; ++g) p.partial_lse[s0 * R + g] = -INFINITY;
            }
        };
        if (waited) finish_window();
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
                    pg[k] = early_load<EARLY>(p.block_table + static_cast<int64_t>(bj) * p.max_pages + idx);
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
            const int cl = c + lane;
            const int stage = cl % STAGES;
            const uint32_t epar = ((cl / STAGES) & 1) ^ 1;
            // Early KV gather (first chunk only): pass 0 issues the first ring pass of the tiles
            // that hold none of the request's newest new_tokens tokens, with no hand-offs (Q is
            // the preceding kernel's output); then the warp waits for that kernel.  Pass 1 is
            // the loop over everything else.
            const bool early_l = EARLY && !waited && lane < cnt && lane < STAGES && nv_l > 0 &&
                                 ct * kTile + kTile <= len_l - p.new_tokens;
            uint32_t todo = 0;  // descriptor starts not yet handed off
            bool pend = false;
            for (int pass = (!EARLY || waited) ? 1 : 0; pass < 2; ++pass) {
            pend = pass == 0 ? early_l : (lane < cnt && !early_l);
            todo = pass == 0 ? 0u : starts;
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
                        if (TC) {  // the S warp fetches Q itself, a descriptor ahead
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
                            tma_load_5d(kdst, kmap, fb, 0, 0, 0, h_l, cpg[0], policy);
                            tma_load_5d(vdst, vmap, fb, 0, 0, 0, h_l, cpg[0], policy);
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
                                if (TC && KV == 0 && P < kTile) {
                                    const uint32_t ro = static_cast<uint32_t>(k * P) * 128u;
                                    tma_load_5d(kdst + ro, kmap, fb, 0, 0, 0, h_l, pg, policy);
                                    tma_load_5d(kdst + C::kTileBytes / 2 + ro, kmap, fb, 0, 0, 1, h_l, pg, policy);
                                    tma_load_5d(vdst + ro, vmap, fb, 0, 0, 0, h_l, pg, policy);
                                    tma_load_5d(vdst + C::kTileBytes / 2 + ro, vmap, fb, 0, 0, 1, h_l, pg, policy);
                                } else {
                                    const uint32_t ro = static_cast<uint32_t>(k * P) * (C::kTileBytes / kTile);
                                    tma_load_5d(kdst + ro, kmap, fb, 0, 0, 0, h_l, pg, policy);
                                    tma_load_5d(vdst + ro, vmap, fb, 0, 0, 0, h_l, pg, policy);
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
            if (aborted) break;
            if (EARLY && pass == 0) {
                grid_dependency_wait();  // Q, its scales and the newest tokens are in memory now
                grid_launch_dependents();
                waited = true;
                finish_window();
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
}

}  // namespace dsa
