/*
 * split_switched_decode.h -- C ABI of the small-batch decode hot path for one NVIDIA
 * GB300 (sm_103a): the decode projection with a batch-size kernel switch, the MoE
 * front end (router scores + latent projection as one product, then softmax/top-k),
 * the routed-expert grouped GEMV with the shared expert overlapping it (inside the same
 * launch, or on a side stream), and an L2 prefetch kernel.
 *
 * The method is the one described in "Hyper Optimizing Kimi K3 in vLLM: Moving Fast
 * and Responsibly" (vLLM blog), Part 1, sections 1-4. Each entry point below cites
 * the section that describes the operation.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Types. dec_bf16 is the raw 16-bit pattern of an IEEE bfloat16. Matrices are
 *    row-major with the last dimension contiguous. Weights W[N,K] use the nn.Linear
 *    layout, so Y = X . W^T -- except for the *_packed entry points, which read the
 *    tile-packed copy made once by dec_pack_weight / dec_pack_expert_weights.
 *  - Memory. Every pointer is DEVICE memory owned by the caller. The library never
 *    allocates or frees memory. Where a call needs scratch memory it takes a caller
 *    workspace whose size comes from the matching *_workspace_bytes() query; the
 *    workspace must be zero-filled once before its first use (cudaMemset), every
 *    completed call leaves it ready for the next (a call whose kernels timed out, see
 *    Errors, does not: zero-fill it again), and one workspace must not be used by two
 *    calls that can run at the same time.
 *  - Alignment. X, W, Wcat, Wgu, Wd and every workspace must be 16-byte aligned; K and
 *    every other reduction length must be a multiple of 8 (rows are then 16-byte
 *    multiples). Other pointers need their natural alignment.
 *  - Streams. Every call is asynchronous on the stream(s) it is given (NULL = legacy
 *    default stream) and never synchronises the host.
 *  - Errors. Arguments are checked on the host before anything is launched; a failed
 *    check returns a status and launches nothing. DEC_ERR_UNSUPPORTED_SHAPE means
 *    "outside the validated envelope: use your standard path". A failed launch returns
 *    DEC_ERR_CUDA. Every wait inside a kernel is bounded in time; a wait that runs out
 *    makes the kernel stop early and sets a device status word that dec_sync_status()
 *    reports (DEC_ERR_TIMEOUT). No kernel traps.
 *  - Batch. Decode batch B is 1..64. The tensor-core projections (dec_splitk_gemm with
 *    use_tc = 1, dec_linear) also take B = 65..512 rows: speculative-decoding
 *    verification scores B sequences x (draft length + 1) tokens in one projection
 *    ("Part 3: Performance Deep Dive", decode with DSpark, seven draft tokens: 8 rows
 *    per sequence, so up to 64 sequences). From 129 rows (split_k = 0), and from 65
 *    rows where W has enough 256-row slices to cover 80 % of the SMs, a call is one
 *    launch on CTA-pair tensor-core tiles (two SMs share each MMA of 256 weight rows,
 *    each SM staging half of the activation rows), reading W once; other calls run on
 *    one-CTA tiles, at most 256 rows per launch.
 */
#ifndef SPLIT_SWITCHED_DECODE_H
#define SPLIT_SWITCHED_DECODE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DEC_API __attribute__((visibility("default")))
#else
#define DEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t dec_bf16;
/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *dec_stream_t;

typedef enum {
    DEC_OK = 0,
    DEC_ERR_INVALID_ARG = 1,         /* null pointer, non-positive size, bad option   */
    DEC_ERR_UNSUPPORTED_SHAPE = 2,   /* outside the envelope: use the standard path   */
    DEC_ERR_MISALIGNED = 3,          /* pointer or length breaks the alignment rules  */
    DEC_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes below the *_workspace_bytes() value  */
    DEC_ERR_CUDA = 5,                /* a CUDA runtime call or launch failed          */
    DEC_ERR_TIMEOUT = 6              /* a bounded device wait ran out (see above)     */
} dec_status;

/* Kernel variants that dec_linear can pick ("different batch sizes need different
 * kernel choices", Part 1 / 1. Tune shapes for the workload). */
typedef enum {
    DEC_VARIANT_NONE = -1,
    DEC_VARIANT_TINY = 0,        /* tiny-matrix GEMV, B <= 2, CUDA cores              */
    DEC_VARIANT_SPLITK = 1,      /* split-K, TMA-staged weight tiles, CUDA cores     */
    DEC_VARIANT_SPLITK_TC = 2,   /* split-K, TMA-staged tiles, tcgen05 tensor cores  */
    DEC_VARIANT_FRONT_ONE_LAUNCH = 3, /* moe_front as one launch: tensor-core product,
                                         on-chip split-K reduction, routing, route map */
    DEC_VARIANT_SPLITK_TC_PAIR = 4   /* 65..512 rows: CTA-pair tensor-core tiles (M = 256
                                        weight rows per MMA over two SMs), one launch */
} dec_variant;

/* ------------------------------------------------------------ diagnostics ---- */

/* Static English text for a status code (never NULL). */
DEC_API const char *dec_status_string(int status);
/* Static name of a variant ("tiny", "splitk", "splitk_tc", "front_one_launch",
 * "splitk_tc_pair", "none"). */
DEC_API const char *dec_variant_name(int variant);
/* Variant launched by the most recent successful projection call on this host
 * thread (dec_gemv, dec_splitk_gemm, dec_linear, moe_front), or DEC_VARIANT_NONE. */
DEC_API int dec_last_variant(void);
/* Library ABI version: 100 * major + minor. */
DEC_API int dec_version(void);

/* Force the variant dec_linear picks on this process: DEC_VARIANT_NONE restores the
 * batch-size switch. A forced variant that cannot run the shape makes dec_linear
 * return DEC_ERR_UNSUPPORTED_SHAPE. Used to test every variant at every batch size.
 * The environment variable DEC_FORCE_VARIANT (tiny|splitk|splitk_tc) sets the
 * initial value. Returns DEC_ERR_INVALID_ARG for an unknown value. */
DEC_API dec_status dec_set_force_variant(int variant);

/* Host-side fault injection for tests: the next `count` launches of this process
 * fail before reaching the GPU and return DEC_ERR_CUDA. 0 disables. */
DEC_API dec_status dec_set_fault_inject(int count);

/* Time limit of every bounded device wait, in nanoseconds (default 2e9).
 * Values below 1e6 are rejected with DEC_ERR_INVALID_ARG. */
DEC_API dec_status dec_set_wait_limit_ns(uint64_t ns);

/* Synchronise `s`, then read and clear the current device's status word.
 * Returns DEC_ERR_TIMEOUT if any kernel since the last read gave up on a wait,
 * DEC_ERR_INVALID_ARG if moe_experts found an expert index out of range or repeated
 * within a token (its output is then undefined), DEC_ERR_CUDA if the stream reports
 * an error, DEC_OK otherwise. */
DEC_API dec_status dec_sync_status(dec_stream_t s);

/* Self-test of the bounded-wait path: launches one kernel on `s` that waits on an
 * mbarrier nothing ever arrives at, with a limit of `limit_ns` nanoseconds
 * (1e6 .. 1e10). The kernel gives up, records the timeout and returns; the caller
 * then sees DEC_ERR_TIMEOUT from dec_sync_status(). Nothing faults or traps. */
DEC_API dec_status dec_debug_wait_timeout(uint64_t limit_ns, dec_stream_t s);

/* ------------------------------------------------------ decode projection ---- */

/*
 * Tiny-matrix projection for decode batches of 1 to 4
 * ("Part 1 / 1. Tune shapes for the workload": specialised small-matrix kernels at
 * batch sizes 1-2), with the optional residual add of the output projection
 * ("Part 1 / 2. Overlap computation and communication", single-GPU part):
 *
 *     Y[b,n] = bf16( sum_k X[b,k] * W[n,k]  (+ R[b,n]) ),  fp32 accumulation,
 *                                                           one round to nearest even
 *
 * X [B,K], W [N,K], R [B,N] or NULL, Y [B,N]. B in 1..4 (dec_linear uses it for 1..2:
 * with 3-4 rows the kernel runs out of instruction issue before HBM bandwidth, measured
 * 25.9 / 30.3 us on the 7168 -> 8192 projection against 21.7 us on tensor cores);
 * N >= 1; K >= 8, K % 8 == 0; B > 4 -> DEC_ERR_UNSUPPORTED_SHAPE. Streams W once with
 * 128-bit loads; no workspace. Y may not alias X, W or R.
 */
DEC_API dec_status dec_gemv(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R, dec_bf16 *Y,
                    int B, int N, int K, dec_stream_t s);

/*
 * Split-K projection for larger decode batches ("Part 1 / 1. Tune shapes for the
 * workload": split-K kernels that divide the matrix multiplication across more GPU
 * workers), same result as dec_gemv for any B in 1..64.
 *
 * W is cut into 128-row tiles and 64-wide k-blocks. The (tile, k-block) sequence is
 * divided into contiguous ranges, one per CTA ("worker"); partial sums of a tile
 * produced by several workers go to the workspace and are added in worker order
 * (fixed order: bit-identical results for a fixed split), R is added and the sum is
 * rounded once. The adding is done by the last worker to finish the tile or, for
 * B >= 32 with K >= 12288 (DEC_DEFER_MIN_B sets the batch), by a second kernel
 * launched behind the first on the same stream. When twice the tile count still
 * occupies at least 80 % of the SMs (and B >= 2, B <= 64), every tile is split into
 * exactly two k-halves instead; with use_tc = 1 and an even k-block count the two
 * halves run as a 2-CTA thread-block cluster and are added on chip through
 * distributed shared memory (same order, same bits).
 *
 *   split_k == 0 : one worker per SM, ranges of equal length (stream-K style).
 *   split_k == S : every tile split into S equal k-ranges (S <= k-blocks per tile).
 * use_tc: 0 = CUDA-core tiles (B <= 64), 1 = tcgen05 tensor-core tiles (W rows are
 * the MMA M dimension, the batch is the MMA N dimension, accumulator in tensor
 * memory). With use_tc = 1, B may be 65..512 (speculative verification rows): groups
 * of 64 batch columns share every weight tile, each group reduced separately, at most
 * 256 rows per launch; use_tc = 0 then returns DEC_ERR_UNSUPPORTED_SHAPE. With
 * use_tc = 1, split_k = 0, at least two k-blocks and 129 <= B <= 512 (or 65 <= B <= 128
 * with 4 x ceil(ceil(N / 128) / 2) >= 80 % of the SMs), the call is
 * instead one launch of 4-CTA clusters, one per 256 rows of W: two CTA pairs (tcgen05
 * .cta_group::2, M = 256) hold the two k-halves, the batch taken as B rounded up to a
 * multiple of 64 columns (at least 128; one MMA of that width up to 256, else two of
 * half of it), the halves added inside the cluster through
 * distributed shared memory in a fixed order (deterministic; the summation order
 * differs from the one-CTA tiles, so bits may differ from them within the tolerance);
 * DEC_WIDE_PAIR_MMA=0 turns it off, DEC_WIDE_PAIR_MIN_B moves its lower bound.
 * dec_splitk_workspace_bytes() covers every launch of the call (they reuse it in turn;
 * the CTA-pair launch checks the same size and uses none of it).
 */
DEC_API size_t dec_splitk_workspace_bytes(int B, int N, int K, int split_k);
DEC_API dec_status dec_splitk_gemm(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R,
                           dec_bf16 *Y, int B, int N, int K, int split_k, int use_tc,
                           void *ws, size_t ws_bytes, dec_stream_t s);

/*
 * dec_splitk_gemm without a workspace, for callers that cannot allocate device memory
 * (for example a plugin running inside another runtime that owns the GPU memory pool,
 * or a serving loop whose memory is frozen after warm-up). The blog post has no
 * counterpart: it is an addition of this library. Same arguments as dec_splitk_gemm
 * with split_k = 0, and the same kernels, schedule and bits; the scratch lives in a
 * fixed 16 MiB device array inside the library (held on every GPU that loads it until
 * the process exits), so a shape whose split-K scratch would exceed 16 MiB is rejected
 * with DEC_ERR_WORKSPACE_TOO_SMALL, more than 256 rows (or more than 64 with use_tc = 0)
 * with DEC_ERR_UNSUPPORTED_SHAPE. The first call on a device looks up the array's
 * address (a failed lookup is retried on the next call): make it before any stream
 * capture. Every call on a device shares the one array, and each call first clears its
 * arrival counters with an asynchronous memset on s (so a call after one that gave up
 * on a bounded wait still starts from zero): two calls that can overlap on that GPU
 * race, so issue them on one stream or otherwise serialise them. No cudaMalloc,
 * cudaFree or allocating library routine is called.
 */
DEC_API dec_status dec_splitk_gemm_noalloc(const dec_bf16 *X, const dec_bf16 *W,
                                           const dec_bf16 *R, dec_bf16 *Y, int B, int N, int K,
                                           int use_tc, dec_stream_t s);

/*
 * The batch-size switch: picks dec_gemv for B <= 2 (B = 1 only for shapes whose tiles,
 * split into two k-halves, still occupy >= 80 % of the SMs: there the tensor-core
 * two-halves schedule is measured faster from B = 2), the split-K tiles on CUDA cores
 * for small B and on tensor cores from a threshold batch upward (always for
 * B = 65..512), then runs it.
 * dec_linear_workspace_bytes() covers whichever variant the switch can pick.
 */
DEC_API size_t dec_linear_workspace_bytes(int B, int N, int K);
DEC_API dec_status dec_linear(const dec_bf16 *X, const dec_bf16 *W, const dec_bf16 *R, dec_bf16 *Y,
                      int B, int N, int K, void *ws, size_t ws_bytes, dec_stream_t s);

/*
 * Tile-packed weights: the same W stored for the split-K tiles instead of row-major. Wp
 * is N*K bf16 values in 16 KB blocks of 128 rows x 64 k (each row of a block is 64
 * consecutive k, 128 bytes); block (n/128, k/64) starts at element
 * ((n/128)*(K/64) + k/64) * 8192, and W[n,k] is at that block's start + (n%128)*64 + k%64.
 * A split-K worker then streams whole contiguous 16 KB blocks instead of 128 separate
 * 128-byte row pieces (measured on the Kimi projections: 3 % faster for 7168 -> 8192,
 * 5-6 % for 16384 -> 7168). Requires N % 128 == 0 and K % 64 == 0
 * (DEC_ERR_UNSUPPORTED_SHAPE otherwise).
 *
 * dec_pack_weight: Wp = packed(W), one launch on s (a copy: pack once when the weights
 * are loaded). W and Wp must not overlap (DEC_ERR_INVALID_ARG) and are 16-byte aligned.
 * dec_gemv_packed, dec_splitk_gemm_packed, dec_linear_packed: dec_gemv, dec_splitk_gemm
 * and dec_linear with a packed weight, same arguments. The split-K tiles run the same
 * schedule and give the same bits as on the unpacked W. The tiny kernel reads the packed
 * blocks with its own lane mapping (a warp load covers 4 adjacent rows x 128 bytes of
 * one block) and adds in its own fixed order: the same result up to fp32 rounding order
 * (repeatable bit for bit). dec_linear_packed picks the tiny kernel only for K < 12288;
 * from there the split-K tiles are faster on packed weights at every batch.
 */
DEC_API dec_status dec_pack_weight(const dec_bf16 *W, int N, int K, dec_bf16 *Wp,
                                   dec_stream_t s);
DEC_API dec_status dec_gemv_packed(const dec_bf16 *X, const dec_bf16 *Wp, const dec_bf16 *R,
                                   dec_bf16 *Y, int B, int N, int K, dec_stream_t s);
DEC_API dec_status dec_splitk_gemm_packed(const dec_bf16 *X, const dec_bf16 *Wp,
                                          const dec_bf16 *R, dec_bf16 *Y, int B, int N, int K,
                                          int split_k, int use_tc, void *ws, size_t ws_bytes,
                                          dec_stream_t s);
DEC_API dec_status dec_linear_packed(const dec_bf16 *X, const dec_bf16 *Wp, const dec_bf16 *R,
                                     dec_bf16 *Y, int B, int N, int K, void *ws,
                                     size_t ws_bytes, dec_stream_t s);

/* ------------------------------------------------------------ MoE front ------- */

/*
 * Route-map layout (int32), written by moe_front when route_map is given and read by
 * moe_experts. With P = B*topk:
 *   [0, E)              counts[e]   tokens routed to expert e
 *   [E, 2E+1)           offsets[e]  exclusive prefix sum of counts; offsets[E] = P
 *   [2E+1, 2E+1+P)      pairs[i]    entries b*topk+j sorted by (expert, b)
 *   [2E+1+P, 2E+1+2P)   pos[b*topk+j] position of that entry in pairs
 *   [2E+1+2P]           num_used    number of experts with counts > 0
 *   [2E+2+2P, 3E+2+2P)  used[u]     those experts, ascending
 */
DEC_API size_t moe_route_map_ints(int B, int E, int topk);

/*
 * MoE front end ("Part 1 / 3. Improve MoE scheduling and overlap": the router scores
 * and the latent input projection combined into one matrix multiplication), followed
 * by the routing the pages leave implicit, read as: softmax over the E raw router
 * logits; the topk experts with the largest logits (fp32), ties to the lower expert
 * index, listed by descending logit; weights renormalised over the chosen experts.
 *
 *     Z = X . Wcat^T          Wcat [E+L, K]: router rows first, then latent rows
 *     latent[b,:] = bf16(Z[b, E:E+L])
 *     topk_idx[b,:], topk_w[b,:]  as above;  probs[b,e] = softmax(Z[b,0:E])_e
 *
 * X [B,K]; latent [B,L] (NULL allowed when L == 0); topk_idx int32 [B,topk];
 * topk_w fp32 [B,topk]; probs_opt fp32 [B,E] or NULL; route_map_opt int32
 * [moe_route_map_ints(B,E,topk)] or NULL. E in 1..512, topk in 1..min(E,16), L >= 0.
 * One launch on `s` where the device can hold its thread-block clusters (the default):
 * each 128-row tile of Wcat is one cluster of up to 16 CTAs that split K and add their
 * partials through distributed shared memory; router CTAs publish the logits (fp32, in
 * the workspace) and arrival counters elect the CTAs that route (a warp per token) and
 * build the route map. Otherwise, or with the environment switch DEC_FRONT_FUSED=0, two
 * launches: the product, then a finishing kernel that starts as the product's CTAs
 * retire (programmatic dependent launch). Every way gives the same top-k ids, weights
 * and route map. The workspace must be zeroed once before its first use (its arrival
 * counters return to zero at the end of every call).
 */
DEC_API size_t moe_front_workspace_bytes(int B, int E, int L, int K);
DEC_API dec_status moe_front(const dec_bf16 *X, const dec_bf16 *Wcat, int B, int K, int E, int L,
                     int topk, dec_bf16 *latent, int32_t *topk_idx, float *topk_w,
                     float *probs_opt, int32_t *route_map_opt, void *ws, size_t ws_bytes,
                     dec_stream_t s);

/* --------------------------------------------------------------- experts ------ */

/*
 * Routed experts as a grouped GEMV plus the shared expert on a side stream
 * ("Part 1 / 3. Improve MoE scheduling and overlap": the shared expert runs on a
 * separate stream and overlaps the routed-expert computation; the schedule limits
 * the GPU resources each operation uses):
 *
 *     for each token b and rank j, e = topk_idx[b,j]:
 *        g = X[b] . Wgu[e, 0:I]^T,   u = X[b] . Wgu[e, I:2I]^T
 *        A = bf16(silu(g) * u),      silu(t) = t / (1 + exp(-t))
 *        Yp[b,j] = A . Wd[e]^T       (fp32)
 *     S[b] = the same MLP with Wgu_shared / Wd_shared (when given)
 *     Y[b] = bf16( sum_j topk_w[b,j] * Yp[b,j]  +  S[b] )   (j ascending, fp32)
 *
 * X [B,H]; topk_idx int32 [B,topk]; topk_w fp32 [B,topk]; route_map from moe_front or
 * NULL (then rebuilt on `main`); Wgu [E,2I,H]; Wd [E,H,I]; Wgu_shared [2I,H] and
 * Wd_shared [H,I], both NULL for no shared expert; Y [B,H].
 * Each used expert's weights are read once for all of its tokens.
 * On tensor cores (the default from B = 1) the routed experts' gate/up and down run as
 * one launch on `main`, and the shared expert's tiles join it as one more group, claimed
 * by every SM like the routed ones (the pages' overlap of the shared and routed experts,
 * inside one launch; `side` is then unused). With side_max_ctas > 0, the environment
 * switch DEC_SHARED_IN_ROUTED=0 or the fused combine, the shared expert runs instead on
 * `side` with at most side_max_ctas CTAs (0 = chosen from the expected weight bytes)
 * while the routed experts use the remaining SMs on `main`; `side` may equal `main`
 * (then no overlap), and the call records events so that `main` waits for `side` before
 * the combine. On return all work is ordered after `main`.
 * The combine is its own launch; with a route map and the environment switch
 * DEC_FUSED_COMBINE=1 it runs instead inside the down launches (the tile that completes
 * a token's 128-row block adds it up, in the same order: the same bits).
 * Schedule: in the one launch, whole tiles claimed one by one from a counter in the
 * workspace (cleared by the call's gather launch), each accumulated over all of its
 * k-blocks by one CTA, down tiles after their expert's gate/up tiles; so the bits do not
 * depend on which CTA computes a tile. With DEC_EXPERT_ONE_LAUNCH=0, gate/up and down
 * are two launches: whole tiles (a static share per CTA, the rest claimed) from about
 * 6.5 expected tiles per CTA, equal stream-K ranges of (expert, tile, k-block) with a
 * fixed-order reduction of split tiles below. All are deterministic; the whole-tile
 * schedules give the same bits as each other, the stream-K ranges differ from them by
 * fp32 summation order.
 * H % 128 == 0, I % 64 == 0, topk <= 16, E <= 512.
 */
DEC_API size_t moe_experts_workspace_bytes(int B, int E, int topk, int H, int I);
DEC_API dec_status moe_experts(const dec_bf16 *X, const int32_t *topk_idx, const float *topk_w,
                       const int32_t *route_map, const dec_bf16 *Wgu, const dec_bf16 *Wd,
                       int E, const dec_bf16 *Wgu_shared, const dec_bf16 *Wd_shared, int B,
                       int H, int I, int topk, dec_bf16 *Y, void *ws, size_t ws_bytes,
                       dec_stream_t main_stream, dec_stream_t side_stream, int side_max_ctas);

/*
 * The MoE layer in one call: moe_front followed by moe_experts, with the shared expert
 * overlapping the routing ("Part 1 / 3. Improve MoE scheduling and overlap": the shared
 * expert runs on a separate stream overlapping routing or routed-expert work). The
 * shared expert's launches go on `side_stream` first; the front end then runs on
 * `main_stream` on the remaining SMs while the shared expert streams its weights, and
 * the routed experts and the combine follow on `main_stream`, which waits for
 * `side_stream` before the combine. Outputs: latent [B,L] (when L > 0), topk_idx and
 * topk_w [B,topk], route_map_opt (optional, as moe_front), Y [B,H] as moe_experts.
 * Same shapes, alignment and errors as moe_front (K = H) and moe_experts;
 * ws = moe_layer_workspace_bytes(B, E, L, H, I, topk) bytes.
 */
DEC_API size_t moe_layer_workspace_bytes(int B, int E, int L, int H, int I, int topk);
DEC_API dec_status moe_layer(const dec_bf16 *X, const dec_bf16 *Wcat, int E, int L, int topk,
                             const dec_bf16 *Wgu, const dec_bf16 *Wd, const dec_bf16 *Wgu_shared,
                             const dec_bf16 *Wd_shared, int B, int H, int I, dec_bf16 *latent,
                             int32_t *topk_idx, float *topk_w, int32_t *route_map_opt,
                             dec_bf16 *Y, void *ws, size_t ws_bytes, dec_stream_t main_stream,
                             dec_stream_t side_stream, int side_max_ctas);

/*
 * Tile-packed expert banks (the layout of dec_pack_weight, for the expert GEMV tiles):
 *   Wgu_p: E * (I/64) * (H/64) blocks of 16 KB, block ((e*(I/64) + t)*(H/64) + kb) holding
 *          the 64 gate rows t*64.. and then the 64 matching up rows I + t*64.. of expert e,
 *          each row the 64 values k = 64 kb .. 64 kb + 63 (128 bytes);
 *   Wd_p:  dec_pack_weight of Wd viewed as [E*H, I] (H % 128 == 0: a block never spans
 *          two experts).
 * A grouped launch then streams whole contiguous 16 KB blocks (measured at the Kimi
 * shape: the expert layer 2.8 % faster at B = 64, 4-6 % at B = 1-8).
 * dec_pack_expert_weights: packs a bank (E experts; E = 1 for the shared expert), two
 * launches on s; H % 128 == 0 and I % 64 == 0 (DEC_ERR_UNSUPPORTED_SHAPE otherwise); the
 * four buffers must not overlap (DEC_ERR_INVALID_ARG). A copy: pack once at load time.
 * moe_experts_packed / moe_layer_packed: moe_experts / moe_layer with packed routed and
 * shared banks (Wcat stays row-major); same arguments, same schedule, same bits.
 */
DEC_API dec_status dec_pack_expert_weights(const dec_bf16 *Wgu, const dec_bf16 *Wd, int E, int H,
                                           int I, dec_bf16 *Wgu_p, dec_bf16 *Wd_p,
                                           dec_stream_t s);
DEC_API dec_status moe_experts_packed(const dec_bf16 *X, const int32_t *topk_idx,
                                      const float *topk_w, const int32_t *route_map,
                                      const dec_bf16 *Wgu_p, const dec_bf16 *Wd_p, int E,
                                      const dec_bf16 *Wgu_shared_p, const dec_bf16 *Wd_shared_p,
                                      int B, int H, int I, int topk, dec_bf16 *Y, void *ws,
                                      size_t ws_bytes, dec_stream_t main_stream,
                                      dec_stream_t side_stream, int side_max_ctas);
DEC_API dec_status moe_layer_packed(const dec_bf16 *X, const dec_bf16 *Wcat, int E, int L,
                                    int topk, const dec_bf16 *Wgu_p, const dec_bf16 *Wd_p,
                                    const dec_bf16 *Wgu_shared_p, const dec_bf16 *Wd_shared_p,
                                    int B, int H, int I, dec_bf16 *latent, int32_t *topk_idx,
                                    float *topk_w, int32_t *route_map_opt, dec_bf16 *Y,
                                    void *ws, size_t ws_bytes, dec_stream_t main_stream,
                                    dec_stream_t side_stream, int side_max_ctas);

/* ------------------------------------------------------------ read stream ----- */

/*
 * A measurement helper, not part of the decode path (like dec_sim_comm_wait): reads
 * dec_read_stream_bytes(bytes) bytes (whole 256 KB chunks) from the start of p into
 * shared memory and writes nothing. One CTA per SM claims chunks from a counter until
 * none is left and streams each with 1-D bulk copies of 16 KB, 8 in flight, the way the
 * expert tiles stream packed weights; the rate it reaches is the read-only HBM ceiling
 * the weight streams are measured against (a copy benchmark counts read and written
 * bytes). The counter is a library variable zeroed on `s` before each launch: calls on
 * one device must not overlap. p: device memory, 16-byte aligned (DEC_ERR_MISALIGNED),
 * not NULL (DEC_ERR_INVALID_ARG). Less than one chunk reads nothing (DEC_OK, no launch).
 * Bounded waits as everywhere (DEC_ERR_TIMEOUT through dec_sync_status).
 */
DEC_API size_t dec_read_stream_bytes(size_t bytes);
DEC_API dec_status dec_read_stream(const void *p, size_t bytes, dec_stream_t s);

/* ------------------------------------------------------------ L2 prefetch ----- */

/*
 * Pull the byte range [p, p+bytes) toward L2 on stream `s` with at most max_ctas
 * CTAs (0 = 8) and write nothing ("Part 1 / 4. Prefetching upcoming weights into
 * cache": a dedicated side-stream kernel raises the cache hit rate of the next
 * operation's weights during phases that cannot use the full memory bandwidth).
 * p must be 16-byte aligned; bytes is rounded down to a multiple of 16.
 * Results of other calls never depend on it.
 */
DEC_API dec_status l2_prefetch(const void *p, size_t bytes, int max_ctas, dec_stream_t s);

/*
 * Stand-in for a communication phase, for measuring the prefetch of "Part 1 / 4.
 * Prefetching upcoming weights into cache" on one GPU (the all-reduce that precedes
 * the output projection in "Part 1 / 2. Overlap computation and communication" is
 * multi-GPU): one CTA on `s` that keeps the stream busy for `ns` nanoseconds
 * (1e3 .. 1e9, else DEC_ERR_INVALID_ARG, nothing launched) by the GPU's global timer
 * and touches no memory, so HBM is idle meanwhile. It always ends on time.
 */
DEC_API dec_status dec_sim_comm_wait(uint64_t ns, dec_stream_t s);

#ifdef __cplusplus
}
#endif

#endif /* SPLIT_SWITCHED_DECODE_H */
