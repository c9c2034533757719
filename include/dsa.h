/*
 * dsa.h -- C ABI of libdsa: load-balanced, variable-length, paged-KV GQA decode
 * attention for GB300 (sm_103a), scheduled by a per-step task map.
 *
 * The operation (sources are web pages; section names as printed on them):
 *   HPC-Ops × SGLang blog, "Attention：变长 decode 的负载均衡":
 *     decode attention work grows with each request's live KV length; a static
 *     split-KV grid over (KV head, request, chunk) either uses a fixed split
 *     count (long requests make heavy chunks and a tail) or a fixed chunk size
 *     (the grid reserves splits for the longest request, short ones leave empty
 *     chunks).
 *   Same page, "围绕活跃 KV 工作进行调度": an assign kernel builds a global task
 *     map from the live device-side KV lengths once per decode step (reused by
 *     every layer): 64-token tiles, total over heads and requests, per-CTA budget
 *     = total / persistent CTAs, bins filled up to the budget then spilled, with
 *     a minimum-work floor.  Each resident CTA drains its bin; each descriptor
 *     covers one or more contiguous KV tiles of one (request, head) and yields a
 *     partial output with its log-sum-exp; a combine kernel merges the actual
 *     number of partials per (request, head) under the global softmax.
 *   Hy3 preview write-up, 2.1.1 "Attention动态调度": the same
 *     scheme as uniform tiles, greedy bin packing, a task map generated before
 *     each step, and a combine kernel.
 *
 * Conventions for every call:
 *   - All array arguments are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or synchronises (dsa_get_status and
 *     dsa_read_status excepted).  Work is enqueued on `stream` (a cudaStream_t;
 *     NULL = the legacy default stream) and returns before it runs.  Kernels are
 *     launched with programmatic stream serialization: each may start while the
 *     previous kernel in the stream finishes, and waits for it (griddepcontrol)
 *     before reading any global memory.
 *   - Shapes: B = batch, Hq = query heads, Hkv = KV heads, G = Hq / Hkv query
 *     heads per KV head (query head j reads KV head j / G), d = head_dim = 128,
 *     P = page_size tokens per page: 64 (the tile) everywhere, also 16 or 32
 *     for the decode and split-KV calls (a 64-token tile then spans 64 / P
 *     consecutive block-table entries).  Unit u = (request b, KV head h),
 *     u = b * Hkv + h.
 *   - Layouts (row-major, innermost last):
 *       q            [B, Hq, d]              bf16, or E4M3 bytes
 *       q_scale      [B, Hq] fp32            E4M3 Q only: real = e4m3 * scale
 *       k/v_pages    [num_pages, Hkv, P, d]  bf16, or E4M3 bytes; one
 *                                            (page, KV head) block is contiguous
 *                                            ("HND"; dsa_decode_ex also reads
 *                                            "NHD" pages [num_pages, P, Hkv, d])
 *       k/v_scale    [num_pages, Hkv, P] fp32  E4M3 K/V only, per token and head
 *       block_table  [B, max_pages_per_req] int32; token t of request b is slot
 *                    t % P of page block_table[b][t / P]; entries at or past
 *                    ceil(seq_lens[b] / P) are never read
 *       seq_lens     [B] int32, live KV length of each request (0 allowed)
 *       out          [B, Hq, d] bf16 or fp32;  out_lse [B, Hq] fp32
 *   - Log-sum-exp values are natural logarithms of sum_t exp(s_t), with
 *     s_t = sm_scale * q . k_t already scaled; an empty request has lse = -inf
 *     and output 0.
 *   - Pointers to q, k/v pages, scales and partials must be 16-byte aligned.
 *   - Host-side checks fail with DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED /
 *     DSA_ERR_BUFFER_TOO_SMALL before anything is launched; a failed launch
 *     returns DSA_ERR_CUDA.  Bad device-resident input (a negative length, a
 *     length beyond max_pages_per_req * P, a page id outside [0, num_pages))
 *     cannot be seen from the host: the kernels set a bit in a device status
 *     word (DSA_DEV_* below), skip the affected work and never trap.
 */
#ifndef DSA_H
#define DSA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *dsa_stream; /* same type as cudaStream_t */

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,      /* null pointer, bad size, inconsistent shapes */
    DSA_ERR_UNSUPPORTED = 2,      /* valid but not built: head_dim != 128, P != 64, G > 8, ... */
    DSA_ERR_BUFFER_TOO_SMALL = 3, /* a caller buffer is smaller than the call needs */
    DSA_ERR_CUDA = 4,             /* a CUDA runtime/driver call or a launch failed */
    DSA_ERR_DEVICE_INPUT = 5      /* returned by dsa_get_status when a DSA_DEV_* bit is set */
} dsa_status;

/* Bits of the device status word (task map meta[3], or the static path's word). */
#define DSA_DEV_BAD_SEQLEN 1   /* seq_len < 0, > max_pages_per_req * P, or not covered by the grid */
#define DSA_DEV_BAD_PAGE 2     /* block_table entry outside [0, num_pages); dsa_prologue: a
                                  cache slot outside [-1, num_pages * P) */
#define DSA_DEV_TIMEOUT 4      /* an in-kernel pipeline wait passed its time limit; work abandoned */
#define DSA_DEV_BAD_MAP 8      /* task map inconsistent with the decode arguments */
#define DSA_DEV_BAD_POSITION 32 /* dsa_prologue: a position outside [0, max_position) */

typedef enum { DSA_BF16 = 0, DSA_FP8_E4M3 = 1, DSA_FP32 = 2 } dsa_dtype;

/* Order of a K/V page's dimensions: HND = [num_pages, Hkv, P, d] (one (page, head)
 * block contiguous), NHD = [num_pages, P, Hkv, d] (one token's heads contiguous).
 * FP8 scales are [num_pages, Hkv, P] in both. */
typedef enum { DSA_HND = 0, DSA_NHD = 1 } dsa_kv_layout;

/*
 * Task map: the per-step schedule ("全局任务映射" in the blog's "围绕活跃 KV
 * 工作进行调度").  Caller-allocated device buffers; dsa_plan fills them.
 *   cta_desc_begin [num_ctas + 1]: the descriptors of bin (CTA) i are
 *       [cta_desc_begin[i], cta_desc_begin[i+1]).
 *   descs [max_descs * 4]: {u, t0, t1, k}: tiles [t0, t1) (64-token tiles,
 *       local to unit u), k = index of the descriptor among u's descriptors.
 *       Descriptor index = partial-output slot.
 *   unit_partial_begin [num_units], unit_num_partials [num_units]: the slots
 *       of unit u are [begin, begin + count); count = 0 for an empty unit.
 *   meta [4]: {T = total tiles, C_eff = bins in use, num_descs, status}.
 */
typedef struct {
    int32_t *cta_desc_begin;
    int32_t *descs;
    int32_t *unit_partial_begin;
    int32_t *unit_num_partials;
    int32_t *meta;
    int32_t max_descs; /* capacity of descs, in descriptors */
    int32_t num_ctas;  /* persistent CTAs = bins */
    int32_t num_units; /* B * Hkv the map is sized for */
} dsa_task_map;

/*
 * Capacity bound for the task map: every bin boundary cuts at most one unit,
 * so a map never holds more than B*Hkv + num_ctas - 1 descriptors.  Size
 * descs, partial_o ([max_descs, G, d] fp32) and partial_lse ([max_descs, G]
 * fp32) from it.  Returns -1 on a non-positive or overflowing argument.
 */
int32_t dsa_max_descs(int32_t batch, int32_t num_kv_heads, int32_t num_ctas);

/*
 * dsa_plan -- the assign step (blog, "围绕活跃 KV 工作进行调度"; Hy3 write-up
 * 2.1.1 "贪心装桶"), run on the device from device-resident lengths so that it
 * needs no host synchronisation and can be captured in a CUDA graph.
 *   n_u = ceil(len_b / tile) for u = b*Hkv + h; T = sum n_u (walked b-major,
 *   then h, then tile); C_eff = min(num_persistent_ctas, max(1, T /
 *   min_tiles_per_split)) (0 when T = 0); bin i gets the global tiles
 *   [floor(i*T/C_eff), floor((i+1)*T/C_eff)), i.e. bins filled up to the
 *   real-valued budget T/C_eff then spilled; each bin is cut at unit boundaries
 *   into descriptors.  One CTA; the result is unique and bit-exact.
 * Arguments: seq_lens [batch] device int32; tile must be 64; min_tiles_per_split
 * >= 1; map->num_ctas must equal num_persistent_ctas, map->num_units must equal
 * batch*num_kv_heads, map->max_descs >= dsa_max_descs(...).  B*Hkv <= 16384 and
 * num_persistent_ctas <= 16384 (else DSA_ERR_UNSUPPORTED).
 * A negative length counts as zero tiles and sets DSA_DEV_BAD_SEQLEN in meta[3];
 * dsa_plan resets meta[3] for the step.
 */
dsa_status dsa_plan(const int32_t *seq_lens, int32_t batch, int32_t num_kv_heads,
                    int32_t num_persistent_ctas, int32_t tile, int32_t min_tiles_per_split,
                    const dsa_task_map *map, dsa_stream stream);

/*
 * dsa_decode -- the persistent attention kernel (blog, "围绕活跃 KV 工作进行调度":
 * each resident CTA drains its bin; for each descriptor it computes attention
 * over the descriptor's contiguous tiles and writes a partial output with its
 * log-sum-exp).  Grid = map->num_ctas CTAs, one per bin.  Each KV tile is read
 * once and serves all G query heads of its KV head (GQA).
 *   For descriptor x = {u, t0, t1, k} (b = u / Hkv, h = u % Hkv) and each of the
 *   G query heads j = h*G + g, over the tokens t in [64*t0, min(64*t1, len_b)):
 *     s_t = sm_scale * q_j . k_t    (FP8: * q_scale[b][j] * k_scale[t])
 *     partial_lse[x][g] = ln sum_t exp(s_t)
 *     partial_o[x][g][:] = sum_t exp(s_t - partial_lse) * v_t  (FP8: * v_scale[t])
 * Supported: (q_dtype, kv_dtype) = (BF16, BF16) or (FP8_E4M3, FP8_E4M3);
 * head_dim 128; page_size 16, 32 or 64; 1 <= G <= 8.  q_scale is required for FP8 Q,
 * k_scale/v_scale for FP8 K/V, otherwise ignored.  partial_o holds
 * [map->max_descs, G, 128] fp32, partial_lse [map->max_descs, G] fp32.
 * Device input errors set bits in map->meta[3] (see above).
 */
dsa_status dsa_decode(const void *q, dsa_dtype q_dtype, const float *q_scale,
                      const void *k_pages, const void *v_pages, dsa_dtype kv_dtype,
                      const float *k_scale, const float *v_scale,
                      const int32_t *block_table, int32_t max_pages_per_req, int32_t num_pages,
                      const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                      int32_t num_kv_heads, int32_t head_dim, int32_t page_size, float sm_scale,
                      const dsa_task_map *map, float *partial_o, float *partial_lse,
                      dsa_stream stream);

/*
 * dsa_decode_fused -- dsa_decode with the combine step done inside the persistent
 * kernel: the blog's persistent kernel and combine kernel as one launch, with the
 * same results as dsa_decode followed by dsa_combine up to rounding order.
 *   - A unit covered by a single descriptor writes its final output directly.
 *   - For a unit with several partials, each descriptor's partial is published at
 *     GPU scope and counted in unit_counters[u]; the CTA whose count completes the
 *     unit merges all its partials (same formula as dsa_combine) and resets the
 *     counter to 0.  No CTA waits for another.  A dedicated epilogue warp does this
 *     off the consumers' path.
 *   - Units with no tiles get output 0 and LSE -inf.
 * Extra arguments:
 *   - unit_counters [B*Hkv] int32: all 0 before the first call.  The kernel leaves
 *     them 0 after every completed step; after a step that reported
 *     DSA_DEV_TIMEOUT the caller must zero them again.
 *   - out [B, Hq, 128] in out_dtype (DSA_BF16 or DSA_FP32), 16-byte aligned.
 *   - out_lse [B, Hq] fp32, or NULL.
 * The map's unit_partial_begin and unit_num_partials must be present.  Other
 * arguments and errors are as for dsa_decode.
 */
dsa_status dsa_decode_fused(const void *q, dsa_dtype q_dtype, const float *q_scale,
                            const void *k_pages, const void *v_pages, dsa_dtype kv_dtype,
                            const float *k_scale, const float *v_scale,
                            const int32_t *block_table, int32_t max_pages_per_req, int32_t num_pages,
                            const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t page_size, float sm_scale,
                            const dsa_task_map *map, float *partial_o, float *partial_lse,
                            int32_t *unit_counters, void *out, dsa_dtype out_dtype, float *out_lse,
                            dsa_stream stream);

/*
 * dsa_decode_multi -- dsa_decode for q_len query tokens per request (a multi-token
 * verify step: Hy3 preview write-up 2.5 "MTP与异步调度优化"; SGLang Low-Latency Mode:
 * Kernels and Runtime, section 1, a verify of 1 + 5 draft tokens
 * in one pass).  The task map, the scheduler and the KV
 * stream are those of dsa_decode: each KV tile is read once and serves all q_len * G
 * query rows of its unit.  Query token i of request b stands at position
 * seq_lens[b] - q_len + i and sees the tokens t <= that position (causal within the
 * draft; rows with no visible token in a descriptor get o = 0, lse = -inf there).
 *   q        [B, q_len, Hq, 128] bf16 or E4M3 (row i*G + g of unit (b, h) is
 *            q[b][i][h*G + g]); E4M3: q_scale [B, q_len, Hq] fp32, K/V and their
 *            scales as for dsa_decode.
 *   partial_o [S * map->max_descs, q_len*G, 128] fp32, partial_lse [S * map->max_descs,
 *            q_len*G] with S = dsa_multi_slots_per_desc(q_len, G): 2 for q_len > 1
 *            (slots 2x and 2x + 1, each the attention over part of the descriptor's
 *            tiles: the two softmax teams of the tensor-memory kernel, or, for E4M3 K/V
 *            with q_len * G <= 16, the two consumer groups that take alternate tiles),
 *            1 for q_len = 1;
 *            merging a descriptor's slots gives its attention, and dsa_combine_multi
 *            does so.
 * Supported: the dtypes of dsa_decode (BF16, or E4M3 Q and K/V), q_len * G <= 64;
 * q_len = 1 is exactly dsa_decode.  Other arguments and errors are as for dsa_decode.
 */
int32_t dsa_multi_slots_per_desc(int32_t q_len, int32_t group);
dsa_status dsa_decode_multi(int32_t q_len, const void *q, dsa_dtype q_dtype, const float *q_scale,
                            const void *k_pages, const void *v_pages, dsa_dtype kv_dtype,
                            const float *k_scale, const float *v_scale,
                            const int32_t *block_table, int32_t max_pages_per_req, int32_t num_pages,
                            const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t page_size, float sm_scale,
                            const dsa_task_map *map, float *partial_o, float *partial_lse,
                            dsa_stream stream);

/*
 * dsa_decode_ex -- dsa_decode / dsa_decode_multi with the page layout as an argument
 * (HPC-Ops × SGLang blog, "从 HPC-Ops kernel 到 SGLang": the attention kernel reads
 * the serving runtime's own paged KV store, with no layout conversion first).
 * kv_layout is DSA_HND or DSA_NHD (k/v_pages shaped [num_pages, Hkv, P, d] or
 * [num_pages, P, Hkv, d]); page_size is 16, 32 or 64 for either.  q_len = 1 is
 * dsa_decode, q_len > 1 dsa_decode_multi; the results do not depend on the layout
 * or the page size (the same tokens in another arrangement give the same bits).
 * A 64-token tile reads 64 / P pages, each with its own block-table entry; only
 * pages holding a token below the request's length are read.
 * cta_times: NULL, or device uint64 [map->num_ctas][2]: CTA i writes the global
 * timer (%globaltimer, ns) when it starts work (after the previous kernel in the
 * stream has finished) to [i][0], and the time its last warp finished to [i][1]
 * (a diagnostic of how evenly the bins finish; costs one barrier per CTA).  Errors: a
 * kv_layout outside dsa_kv_layout gives DSA_ERR_INVALID_ARG, other page sizes
 * DSA_ERR_UNSUPPORTED; the rest as for dsa_decode.
 */
dsa_status dsa_decode_ex(int32_t q_len, int32_t kv_layout, const void *q, dsa_dtype q_dtype,
                         const float *q_scale, const void *k_pages, const void *v_pages,
                         dsa_dtype kv_dtype, const float *k_scale, const float *v_scale,
                         const int32_t *block_table, int32_t max_pages_per_req, int32_t num_pages,
                         const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t page_size, float sm_scale,
                         const dsa_task_map *map, float *partial_o, float *partial_lse,
                         uint64_t *cta_times, dsa_stream stream);

/*
 * dsa_decode_chained -- dsa_decode for one layer of a chain of layers that share one task
 * map, starting the KV gather before the layer's Q is ready (SGLang Low-Latency Mode: Kernels
 * and Runtime, section 2, item 1: the next kernel launches early and the attention kernel
 * begins gathering KV before it waits for the query).  The kernel immediately before this call
 * in the stream (normally the layer's prologue, dsa_prologue) writes Q (and its scales) and the
 * newest new_tokens K/V tokens of every request; while it runs, the decode loads the first
 * ring stages' tiles that hold none of those tokens, and waits for it before anything else.
 * Caller's guarantee: the task map, seq_lens, block_table and every other K/V token of this
 * layer were written by kernels that completed before that preceding kernel started -- e.g.
 * the map was built before the previous layer's decode (every layer of a step but the first),
 * the cache's older tokens by earlier steps.  Under that guarantee the results are those of
 * dsa_decode, bit for bit.  The next kernel in the stream is released only after this one has
 * waited for its predecessor, so the guarantee carries from layer to layer.
 * One query token per request, pages of 64 tokens in HND layout; new_tokens >= 0 (0: every
 * tile may be loaded early).  Other arguments and errors are as for dsa_decode.
 */
dsa_status dsa_decode_chained(int32_t new_tokens, const void *q, dsa_dtype q_dtype, const float *q_scale,
                              const void *k_pages, const void *v_pages, dsa_dtype kv_dtype,
                              const float *k_scale, const float *v_scale,
                              const int32_t *block_table, int32_t max_pages_per_req, int32_t num_pages,
                              const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t page_size, float sm_scale,
                              const dsa_task_map *map, float *partial_o, float *partial_lse,
                              dsa_stream stream);

/*
 * dsa_combine_multi -- dsa_combine over the q_len * G partial rows of each unit:
 * out [B, q_len, Hq, 128] (out_dtype DSA_BF16 or DSA_FP32), out_lse [B, q_len, Hq] or
 * NULL.  q_len * G <= 64.  q_len = 1 is dsa_combine.
 */
dsa_status dsa_combine_multi(int32_t q_len, const dsa_task_map *map, const float *partial_o,
                             const float *partial_lse, int32_t batch, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, void *out, dsa_dtype out_dtype,
                             float *out_lse, dsa_stream stream);

/*
 * dsa_combine -- the combine kernel (blog, "围绕活跃 KV 工作进行调度": reads the
 * actual number of partials of each (request, head) and merges them under the
 * global softmax normalisation; Hy3 write-up 2.1.1 "Combine Kernel"):
 *   L = ln sum_k exp(lse_k),  out = sum_k exp(lse_k - L) * o_k
 * over unit u's slots [unit_partial_begin[u], + unit_num_partials[u]).
 * out: [B, Hq, 128] in out_dtype (DSA_BF16, round to nearest even, or DSA_FP32);
 * out_lse: [B, Hq] fp32, may be NULL.  A unit with no partials gives out = 0,
 * lse = -inf.  The kernel reads the map's unit arrays before it waits for the preceding
 * kernel in the stream (programmatic dependent launch).  That is safe after this library's
 * decode calls (dsa_decode, dsa_decode_multi, dsa_decode_ex, dsa_decode_chained), which
 * release the next kernel only after their own wait, when the plan that wrote the map has
 * completed.  After any other kernel, the map must have been written by a kernel that
 * completed before that one started.
 */
dsa_status dsa_combine(const dsa_task_map *map, const float *partial_o, const float *partial_lse,
                       int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                       void *out, dsa_dtype out_dtype, float *out_lse, dsa_stream stream);

/*
 * Static split-KV, the in-run comparison (blog, "Attention：变长 decode 的负载
 * 均衡", its two forms).  Grid (S, Hkv, B), one CTA per (split, unit), the same
 * per-tile engine as dsa_decode.  Unit u with n_u tiles:
 *   mode 0 (fixed split count, param = S): c = ceil(n_u / S) tiles per split;
 *   mode 1 (fixed chunk, param = chunk tokens, a multiple of 64):
 *           c = param / 64, S = ceil(max_seq_len / param), max_seq_len given by
 *           the host (the static grid must be sized for the longest request).
 *   split s covers tiles [s*c, min((s+1)*c, n_u)); an empty split writes
 *   o = 0, lse = -inf.  Slot of (u, s) = u*S + s.
 * dsa_static_num_splits returns S (or -1 on bad arguments).
 * partial_o: [B*Hkv*S, G, 128] fp32, partial_lse: [B*Hkv*S, G] fp32.
 * status: device int32 word for DSA_DEV_* bits (required); a request longer
 * than S*param in mode 1 is not covered and sets DSA_DEV_BAD_SEQLEN.
 * cta_times: NULL, or device uint64 [S*Hkv*B][2] that receives each CTA's start
 * and end of work (%globaltimer ns; CTA (s, h, b) at index s + S*(h + Hkv*b)),
 * as for dsa_decode_ex.
 */
int32_t dsa_static_num_splits(int32_t mode, int32_t param, int32_t max_seq_len);
dsa_status dsa_static_splitkv(int32_t mode, int32_t param, int32_t max_seq_len,
                              const void *q, dsa_dtype q_dtype, const float *q_scale,
                              const void *k_pages, const void *v_pages, dsa_dtype kv_dtype,
                              const float *k_scale, const float *v_scale,
                              const int32_t *block_table, int32_t max_pages_per_req,
                              int32_t num_pages, const int32_t *seq_lens, int32_t batch,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t page_size, float sm_scale, float *partial_o,
                              float *partial_lse, int32_t *status, uint64_t *cta_times,
                              dsa_stream stream);

/*
 * Combine for the static grid: merges all S slots of each unit, empty ones
 * included (they carry lse = -inf).  Same formula and outputs as dsa_combine.
 */
dsa_status dsa_static_combine(int32_t num_splits, const float *partial_o, const float *partial_lse,
                              int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, void *out, dsa_dtype out_dtype, float *out_lse,
                              dsa_stream stream);

/*
 * Status readback.  dsa_read_status copies one device status word to
 * *host_status after synchronising the device; dsa_get_status does the same
 * for map->meta[3].  Both return DSA_OK when the word is 0,
 * DSA_ERR_DEVICE_INPUT when any DSA_DEV_* bit is set, DSA_ERR_CUDA if the copy
 * fails, DSA_ERR_INVALID_ARG for NULL pointers.
 */
dsa_status dsa_read_status(const int32_t *device_status, int32_t *host_status);
dsa_status dsa_get_status(const dsa_task_map *map, int32_t *host_status);

/*
 * dsa_prologue -- the fused attention prologue that produces this library's inputs
 * (HPC-Ops × SGLang blog, "融合式 attention 前导": QK-Norm before RoPE, Q in FP8 with
 * one scale per (token, head) passed to the attention kernel without requantising, K
 * and V written directly into the paged FP8 cache; Hy3 preview write-up 2.2.1 "Fused
 * Rope+Norm+[Hadamard]+Quant+Store KV", one kernel, intermediates kept in registers,
 * quantised online before the cache write; 2.6.1 "Hadamard在线旋转变换", an orthogonal
 * rotation of Q and K before quantisation).  For every token n and head:
 *   Q and K heads:  y = RMSNorm(x) = x / sqrt(mean(x^2) + norm_eps) * w   (if w given)
 *                   y = RoPE(y, positions[n])                           (if rotary_dim)
 *                   y = H_128 y / sqrt(128)                              (if hadamard)
 *   V heads:        y = x
 *   encoding:       FP8: scale = amax(|y|) / 448 (1 if y = 0), byte = E4M3(y / scale),
 *                   round to nearest even, saturating; BF16: round to nearest even.
 * Q goes to q_out [n_tokens, Hq, 128] (q_scale [n_tokens, Hq] for FP8); K and V go
 * to slot s = slot_mapping[n] of the cache, i.e. page s / P, offset s % P of
 * k_pages / v_pages, [num_pages, Hkv, P, 128] for kv_layout DSA_HND or
 * [num_pages, P, Hkv, 128] for DSA_NHD (k/v_scale [num_pages, Hkv, P] for FP8 in
 * both), the layouts dsa_decode_ex reads.  s = -1 writes nothing for that token.
 * Arguments:
 *   qkv            [n_tokens, (Hq + 2 Hkv) * 128] bf16: the QKV projection output,
 *                  heads in the order Q, K, V.
 *   positions      [n_tokens] int32, row of cos_sin (needed when rotary_dim > 0).
 *   cos_sin        [max_position, rotary_dim] fp32: cos(angle i) in column i and
 *                  sin(angle i) in column rotary_dim/2 + i, i < rotary_dim/2.
 *   rotary_dim     0 (no RoPE), 16, 32, 64 or 128: dims >= rotary_dim pass through.
 *   rope_style     DSA_ROPE_NEOX rotates the pairs (i, i + rotary_dim/2);
 *                  DSA_ROPE_INTERLEAVED the pairs (2i, 2i + 1); pair i uses angle i.
 *   q_norm_weight, k_norm_weight  [128] fp32, or NULL for no normalisation of that
 *                  input; norm_eps >= 0.
 *   hadamard       nonzero: apply the Hadamard rotation to Q and K.
 *   q_dtype, kv_dtype  DSA_BF16 or DSA_FP8_E4M3 (scales required for FP8).
 *   status         device int32 or NULL: DSA_DEV_BAD_POSITION for a position outside
 *                  [0, max_position) (that token's Q and K rows are not written),
 *                  DSA_DEV_BAD_PAGE for a slot outside [-1, num_pages * P) (that
 *                  token's K and V are not written).
 * head_dim must be 128 and page_size P 16, 32 or 64 (else DSA_ERR_UNSUPPORTED);
 * kv_layout DSA_HND or DSA_NHD (else DSA_ERR_INVALID_ARG).  qkv, q_out, the pages, cos_sin and the
 * weights must be 16-byte aligned.  Several tokens must not share a slot.
 */
typedef enum { DSA_ROPE_NEOX = 0, DSA_ROPE_INTERLEAVED = 1 } dsa_rope_style;
dsa_status dsa_prologue(const void *qkv, int32_t n_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, const int32_t *positions, const float *cos_sin,
                        int32_t max_position, int32_t rotary_dim, int32_t rope_style,
                        const float *q_norm_weight, const float *k_norm_weight, float norm_eps,
                        int32_t hadamard, const int32_t *slot_mapping, void *q_out, dsa_dtype q_dtype,
                        float *q_scale, void *k_pages, void *v_pages, dsa_dtype kv_dtype,
                        float *k_scale, float *v_scale, int32_t num_pages, int32_t page_size,
                        int32_t kv_layout, int32_t *status, dsa_stream stream);

/*
 * dsa_decode_step_noalloc -- one whole decode step (dsa_plan, dsa_decode,
 * dsa_combine with the same arguments and results) that allocates nothing.  The
 * pages have no counterpart of this call: it exists for callers that cannot
 * call cudaMalloc -- code running under another framework's memory pool or
 * allocator hooks, loops that forbid allocation once started, C programs that
 * own only their inputs and outputs -- and so cannot provide the task map and
 * partial-output buffers dsa_decode needs between its kernels.
 *
 * Scratch: a fixed device array of DSA_NOALLOC_SCRATCH_BYTES inside the
 * library, present on every GPU that loads it until the process exits.  The
 * step needs about 16*(B*Hkv + C) + 4*C + 8*B*Hkv bytes of task map plus
 * (B*Hkv + C - 1) * G * 129 * 4 bytes of partials (C = num_persistent_ctas);
 * larger steps are rejected with DSA_ERR_BUFFER_TOO_SMALL before anything is
 * launched, as are all arguments dsa_plan, dsa_decode or dsa_combine would refuse
 * (out must be 16-byte aligned; B*Hkv and num_persistent_ctas at most 16384): a
 * step is either refused before any launch or enqueued whole.  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current and keeps it for the life of the process; make that first call
 * before any stream capture, and do not call this entry point on a device after
 * cudaDeviceReset (the kept address then names freed memory).  Every call reuses
 * the same array, so calls whose work overlaps on the GPU (other streams, other
 * threads) race on it; calls in one stream are safe.  Nothing in the array needs
 * clearing between calls.
 * status: device int32, may be NULL; receives the step's DSA_DEV_* bits.  When it
 * is nonzero, out and out_lse are undefined (the kernels skipped the bad work).
 * No cudaMalloc, cudaFree or allocating library routine is called.
 */
#define DSA_NOALLOC_SCRATCH_BYTES (8u << 20)
dsa_status dsa_decode_step_noalloc(const void *q, dsa_dtype q_dtype, const float *q_scale,
                                   const void *k_pages, const void *v_pages, dsa_dtype kv_dtype,
                                   const float *k_scale, const float *v_scale,
                                   const int32_t *block_table, int32_t max_pages_per_req,
                                   int32_t num_pages, const int32_t *seq_lens, int32_t batch,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t page_size, float sm_scale, int32_t num_persistent_ctas,
                                   int32_t min_tiles_per_split, void *out, dsa_dtype out_dtype,
                                   float *out_lse, int32_t *status, dsa_stream stream);

/*
 * dsa_selftest_wait_timeout -- exercises the bounded wait every kernel of this
 * library uses (no counterpart on the pages).  One CTA waits on an mbarrier that
 * nothing ever arrives at; after limit_ns (0 < limit_ns <= 2 s) it sets
 * DSA_DEV_TIMEOUT in *status and raises the CTA's abort flag, on which a second
 * waiting warp must leave (it then also sets bit 16).  The kernel returns, and the
 * context stays usable.  status: device int32, which the caller zeroes first.
 */
dsa_status dsa_selftest_wait_timeout(int32_t *status, int64_t limit_ns, dsa_stream stream);

/* Static string naming a dsa_status value. */
const char *dsa_status_string(dsa_status s);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
