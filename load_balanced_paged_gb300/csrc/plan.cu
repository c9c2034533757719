// The assign step: builds the per-step task map on the device from device-resident
// KV lengths (HPC-Ops × SGLang blog, section "围绕活跃 KV 工作进行调度"; Hy3 preview
// write-up, section 2.1.1 "Attention动态调度", "贪心装桶").
//
// One CTA.  Instead of walking tiles one by one, it uses the
// closed form of the greedy fill: with a real-valued budget T / C_eff, bin i holds the
// global tiles [floor(i*T/C_eff), floor((i+1)*T/C_eff)); these starts go to a shared
// table, and the bin holding a tile is found from an fp32 estimate corrected against it.
// Every unit and
// every descriptor is then placed independently:
//   1. n_u = ceil(len_b / 64), exclusive scan -> P_u, total T;
//   2. per unit, the number of bins it touches -> exclusive scan -> first slot;
//   3. per bin, its first descriptor = first slot of the unit holding its first tile
//      plus the number of that unit's bins before it;
//   4. per unit, its descriptors: one per bin it touches, tile ranges clipped to the unit.
#include "common.h"
#include "ptx.cuh"

namespace dsa {
namespace {

// First index in a[0, n) with a[i] > x (a nondecreasing).
__device__ __forceinline__ int upper_bound(const int32_t *a, int n, int64_t x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (a[mid] <= x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// In-place exclusive scan of a[0, n) by the whole block; returns the total.
__device__ int64_t block_exclusive_scan(int32_t *a, int n, int64_t *warp_tot) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, w = tid >> 5, nw = nt >> 5;
    const int per = (n + nt - 1) / nt;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int64_t s = 0;
    for (int i = lo; i < hi; ++i) s += a[i];
    int64_t x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[w] = x;
    __syncthreads();
    if (w == 0) {
        int64_t t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < nw) warp_tot[lane] = t;
    }
    __syncthreads();
    int64_t run = x - s + (w > 0 ? warp_tot[w - 1] : 0);
    const int64_t total = warp_tot[nw - 1];
    for (int i = lo; i < hi; ++i) {
        int32_t v = a[i];
        a[i] = static_cast<int32_t>(run);
        run += v;
    }
    __syncthreads();
    return total;
}

template <int NT>
__global__ void __launch_bounds__(NT, 1)
plan_kernel(const int32_t *__restrict__ seq_lens, int32_t batch, int32_t num_kv_heads, int32_t num_ctas,
            int32_t min_tiles, dsa_task_map map) {
    extern __shared__ int32_t smem[];
    __shared__ int64_t warp_tot[32];
    __shared__ int s_status;
    const int U = batch * num_kv_heads;
    int32_t *sP = smem;                 // [U + 1] first global tile of each unit, then T
    int32_t *sBeg = smem + U + 1;       // [U + 1] first descriptor of each unit, then num_descs
    int32_t *sBin = smem + 2 * (U + 1);  // [num_ctas + 1] first global tile of each bin, then T
    const int tid = threadIdx.x, nt = blockDim.x;

    if (tid == 0) s_status = 0;
    grid_launch_dependents();
    grid_dependency_wait();  // lengths (and the map's previous readers) from earlier kernels
    __syncthreads();

    // 1. tiles per unit (u = b * Hkv + h)
    for (int u = tid; u < U; u += nt) {
        int32_t len = seq_lens[u / num_kv_heads];
        if (len < 0) {
            atomicOr(&s_status, DSA_DEV_BAD_SEQLEN);
            len = 0;
        }
        sP[u] = len / kTile + (len % kTile != 0);
    }
    __syncthreads();
    int64_t T = block_exclusive_scan(sP, U, warp_tot);
    bool overflow = T > INT32_MAX;  // cannot index the tiles: schedule nothing
    if (overflow) T = 0;
    int64_t C_eff = T / min_tiles;
    if (C_eff < 1) C_eff = 1;
    if (C_eff > num_ctas) C_eff = num_ctas;
    if (T == 0) C_eff = 0;
    if (tid == 0) {
        sP[U] = static_cast<int32_t>(T);
        if (overflow) s_status |= DSA_DEV_BAD_SEQLEN;
    }
    // bin i starts at global tile floor(i * T / C_eff): the cumulative budget, rounded down.
    // With T = q * C_eff + r this is i * q + floor(i * r / C_eff), all in 32 bits.
    const int32_t Ti = static_cast<int32_t>(T), Ci = static_cast<int32_t>(C_eff);
    const int32_t q_ = Ci > 0 ? Ti / Ci : 0, r_ = Ci > 0 ? Ti % Ci : 0;
    for (int i = tid; Ci > 0 && i <= Ci; i += nt) sBin[i] = i * q_ + (i * r_) / Ci;
    __syncthreads();
    // bin holding global tile x: an fp32 estimate of x * C_eff / T, corrected against the table
    const float ratio = Ci > 0 ? static_cast<float>(Ci) / static_cast<float>(Ti) : 0.f;
    auto bin_of = [&](int64_t x) -> int64_t {
        int i = min(Ci - 1, max(0, static_cast<int>((static_cast<float>(x) + 0.5f) * ratio)));
        while (i > 0 && sBin[i] > x) --i;
        while (i + 1 < Ci && sBin[i + 1] <= x) ++i;
        return i;
    };

    // 2. bins touched by each unit
    for (int u = tid; u < U; u += nt) {
        const int64_t p = sP[u], n = overflow ? 0 : sP[u + 1] - p;
        sBeg[u] = n > 0 ? static_cast<int32_t>(bin_of(p + n - 1) - bin_of(p) + 1) : 0;
    }
    __syncthreads();
    int64_t nd = block_exclusive_scan(sBeg, U, warp_tot);
    if (nd > map.max_descs) {  // cannot happen with a map sized by dsa_max_descs
        if (tid == 0) s_status |= DSA_DEV_BAD_MAP;
        nd = 0;
    }
    if (tid == 0) sBeg[U] = static_cast<int32_t>(nd);
    __syncthreads();
    const bool empty_map = nd == 0;

    for (int u = tid; u < U; u += nt) {
        map.unit_partial_begin[u] = empty_map ? 0 : sBeg[u];
        map.unit_num_partials[u] = empty_map ? 0 : sBeg[u + 1] - sBeg[u];
    }

    // 3. first descriptor of every bin
    for (int i = tid; i <= num_ctas; i += nt) {
        int32_t b;
        if (empty_map || i >= C_eff) {
            b = static_cast<int32_t>(nd);
        } else {
            const int v = upper_bound(sP, U, sBin[i]) - 1;
            b = static_cast<int32_t>(sBeg[v] + (i - bin_of(sP[v])));
        }
        map.cta_desc_begin[i] = b;
    }

    // 4. descriptors: each unit walks the bins it touches, in order
    for (int u = tid; u < U && !empty_map; u += nt) {
        const int32_t first = sBeg[u], np = sBeg[u + 1] - first;
        if (np == 0) continue;
        const int64_t p = sP[u], n = sP[u + 1] - p;
        const int64_t b0 = bin_of(p);
        for (int k = 0; k < np; ++k) {
            const int64_t i = b0 + k;
            const int64_t g0 = max(static_cast<int64_t>(sBin[i]), p);
            const int64_t g1 = min(static_cast<int64_t>(sBin[i + 1]), p + n);
            reinterpret_cast<int4 *>(map.descs)[first + k] =
                make_int4(u, static_cast<int32_t>(g0 - p), static_cast<int32_t>(g1 - p), k);
        }
    }

    __syncthreads();
    if (tid == 0) {
        map.meta[0] = static_cast<int32_t>(T);
        map.meta[1] = static_cast<int32_t>(C_eff);
        map.meta[2] = static_cast<int32_t>(nd);
        map.meta[3] = s_status;
    }
}

// Small maps (B*Hkv <= NW * 32 * K units): the same map with fewer dependent steps.
// Each thread owns K consecutive units in registers; each of the two scans is a
// warp shuffle scan plus one barrier; the bins a unit touches come from the fp32 estimate
// corrected against the table of bin starts; and the first descriptor of each bin is written
// by the unit holding the bin's first tile (exactly one unit does: bins are never empty), so
// nothing has to search.
template <int NW>
__device__ __forceinline__ void small_barrier() {
    if constexpr (NW == 1)
        __syncwarp();
    else
        __syncthreads();
}

// Exclusive prefix over the block of one value per thread (threads in order), and the total.
template <int NW>
__device__ __forceinline__ int64_t small_scan(int64_t v, int64_t *s_wsum, int64_t &total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int64_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[w] = incl;
    small_barrier<NW>();
    int64_t off = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
        const int64_t x = s_wsum[i];
        off += i < w ? x : 0;
        tot += x;
    }
    total = tot;
    small_barrier<NW>();  // s_wsum is reused by the next scan
    return off + incl - v;
}

template <int NW, int K>
__global__ void __launch_bounds__(NW * 32, 1)
plan_small_kernel(const int32_t *__restrict__ seq_lens, int32_t batch, int32_t num_kv_heads, int32_t num_ctas,
                  int32_t min_tiles, dsa_task_map map) {
    extern __shared__ int32_t sBin[];  // [num_ctas + 1] first global tile of each bin, then T
    __shared__ int64_t s_wsum[NW];
    __shared__ int s_status;
    const int U = batch * num_kv_heads;
    const int tid = threadIdx.x;
    const int base = tid * K;  // this thread's first unit

    if (tid == 0) s_status = 0;
    grid_launch_dependents();
    grid_dependency_wait();  // lengths (and the map's previous readers) from earlier kernels

    // 1. tiles of this thread's units (u = b * Hkv + h, walked without a division per unit)
    int n[K];
    bool bad = false;
    {
        int b = base / num_kv_heads, h = base - b * num_kv_heads;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            int t = 0;
            if (base + j < U) {
                int len = seq_lens[b];
                if (len < 0) {
                    bad = true;
                    len = 0;
                }
                t = len / kTile + (len % kTile != 0);
            }
            n[j] = t;
            if (++h == num_kv_heads) {
                h = 0;
                ++b;
            }
        }
    }
    // 2. first global tile of each unit, total T
    int64_t sum = 0;
#pragma unroll
    for (int j = 0; j < K; ++j) sum += n[j];
    int64_t T = 0;
    const int64_t first = small_scan<NW>(sum, s_wsum, T);
    const bool overflow = T > INT32_MAX;  // cannot index the tiles: schedule nothing
    if (overflow) T = 0;
    int P[K];
    {
        int run = overflow ? 0 : static_cast<int32_t>(first);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (overflow) n[j] = 0;
            P[j] = run;
            run += n[j];
        }
    }
    int64_t C_eff = T / min_tiles;
    if (C_eff < 1) C_eff = 1;
    if (C_eff > num_ctas) C_eff = num_ctas;
    if (T == 0) C_eff = 0;
    // bin i starts at global tile floor(i * T / C_eff) = i * q + floor(i * r / C_eff), T = q * C_eff + r
    const int32_t Ti = static_cast<int32_t>(T), Ci = static_cast<int32_t>(C_eff);
    const int32_t q_ = Ci > 0 ? Ti / Ci : 0, r_ = Ci > 0 ? Ti % Ci : 0;
    for (int i = tid; Ci > 0 && i <= Ci; i += NW * 32) sBin[i] = i * q_ + (i * r_) / Ci;
    small_barrier<NW>();
    const float ratio = Ci > 0 ? static_cast<float>(Ci) / static_cast<float>(Ti) : 0.f;
    auto bin_of = [&](int x) -> int {
        int i = min(Ci - 1, max(0, static_cast<int>((static_cast<float>(x) + 0.5f) * ratio)));
        while (i > 0 && sBin[i] > x) --i;
        while (i + 1 < Ci && sBin[i + 1] <= x) ++i;
        return i;
    };
    // 3. bins touched by each unit, and its first descriptor
    int b0[K], cnt[K];
    int64_t csum = 0;
#pragma unroll
    for (int j = 0; j < K; ++j) {
        b0[j] = 0;
        cnt[j] = 0;
        if (n[j] > 0) {
            b0[j] = bin_of(P[j]);
            cnt[j] = bin_of(P[j] + n[j] - 1) - b0[j] + 1;
        }
        csum += cnt[j];
    }
    int64_t nd = 0;
    const int64_t dfirst = small_scan<NW>(csum, s_wsum, nd);
    if (nd > map.max_descs) {  // cannot happen with a map sized by dsa_max_descs
        if (tid == 0) atomicOr(&s_status, DSA_DEV_BAD_MAP);
        nd = 0;
    }
    const bool empty_map = nd == 0;
    // 4. per unit: its partial slots, its descriptors (one per bin it touches) and the first
    //    descriptor of every bin whose first tile it holds
    int beg = static_cast<int32_t>(dfirst);
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const int u = base + j;
        if (u < U) {
            map.unit_partial_begin[u] = empty_map ? 0 : beg;
            map.unit_num_partials[u] = empty_map ? 0 : cnt[j];
        }
        if (!empty_map) {
            for (int k = 0; k < cnt[j]; ++k) {
                const int i = b0[j] + k;
                const int g0 = max(sBin[i], P[j]), g1 = min(sBin[i + 1], P[j] + n[j]);
                reinterpret_cast<int4 *>(map.descs)[beg + k] = make_int4(u, g0 - P[j], g1 - P[j], k);
                if (k > 0 || sBin[i] >= P[j]) map.cta_desc_begin[i] = beg + k;
            }
        }
        beg += cnt[j];
    }
    // bins past C_eff (and every bin of an empty map) start at the end
    for (int i = empty_map ? tid : Ci + tid; i <= num_ctas; i += NW * 32) map.cta_desc_begin[i] = static_cast<int32_t>(nd);

    if (bad || overflow) atomicOr(&s_status, DSA_DEV_BAD_SEQLEN);
    small_barrier<NW>();
    if (tid == 0) {
        map.meta[0] = static_cast<int32_t>(T);
        map.meta[1] = static_cast<int32_t>(C_eff);
        map.meta[2] = static_cast<int32_t>(nd);
        map.meta[3] = s_status;
    }
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int32_t dsa_max_descs(int32_t batch, int32_t num_kv_heads, int32_t num_ctas) {
    if (batch < 0 || num_kv_heads < 1 || num_ctas < 1) return -1;
    int64_t v = static_cast<int64_t>(batch) * num_kv_heads + num_ctas - 1;
    return v > INT32_MAX ? -1 : static_cast<int32_t>(v);
}

extern "C" dsa_status dsa_plan(const int32_t *seq_lens, int32_t batch, int32_t num_kv_heads,
                               int32_t num_persistent_ctas, int32_t tile, int32_t min_tiles_per_split,
                               const dsa_task_map *map, dsa_stream stream) {
    if (!map || batch < 0 || num_kv_heads < 1 || num_persistent_ctas < 1 || min_tiles_per_split < 1)
        return DSA_ERR_INVALID_ARG;
    if (batch > 0 && !seq_lens) return DSA_ERR_INVALID_ARG;
    if (!map->cta_desc_begin || !map->descs || !map->meta ||
        (batch > 0 && (!map->unit_partial_begin || !map->unit_num_partials)))
        return DSA_ERR_INVALID_ARG;
    if (tile != kTile) return DSA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(map->descs) & 15u) != 0) return DSA_ERR_INVALID_ARG;
    const int64_t U = static_cast<int64_t>(batch) * num_kv_heads;
    if (U > kPlanMaxUnits || num_persistent_ctas > kPlanMaxCtas) return DSA_ERR_UNSUPPORTED;
    if (map->num_ctas != num_persistent_ctas || map->num_units != U) return DSA_ERR_INVALID_ARG;
    const int32_t need = dsa_max_descs(batch, num_kv_heads, num_persistent_ctas);
    if (need < 0) return DSA_ERR_INVALID_ARG;
    if (map->max_descs < need) return DSA_ERR_BUFFER_TOO_SMALL;

    // small maps: units in registers, one barrier per scan, no searches (the bin table, up to
    // 8192 entries, stays within the default shared-memory size with the kernel's own)
    const size_t bins = sizeof(int32_t) * (static_cast<size_t>(num_persistent_ctas) + 1);
    if (bins <= 32 * 1024) {
        if (U <= 256)
            return launch_pdl(plan_small_kernel<8, 1>, dim3(1), dim3(256), bins, to_cuda(stream), seq_lens, batch,
                              num_kv_heads, num_persistent_ctas, min_tiles_per_split, *map);
        if (U <= 1024)
            return launch_pdl(plan_small_kernel<8, 4>, dim3(1), dim3(256), bins, to_cuda(stream), seq_lens, batch,
                              num_kv_heads, num_persistent_ctas, min_tiles_per_split, *map);
        if (U <= 2048)
            return launch_pdl(plan_small_kernel<8, 8>, dim3(1), dim3(256), bins, to_cuda(stream), seq_lens, batch,
                              num_kv_heads, num_persistent_ctas, min_tiles_per_split, *map);
    }
    const size_t smem = sizeof(int32_t) * (2 * static_cast<size_t>(U + 1) + num_persistent_ctas + 1);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(plan_kernel<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return DSA_ERR_CUDA;
    return launch_pdl(plan_kernel<1024>, dim3(1), dim3(1024), smem, to_cuda(stream), seq_lens, batch,
                      num_kv_heads, num_persistent_ctas, min_tiles_per_split, *map);
}
