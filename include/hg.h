/*
 * hg.h -- C ABI of libhg: grouped-contiguous FP8 x MXFP4 (W4A8) MoE expert
 * GEMM and its routing plan, for NVIDIA GB300 (sm_103a).
 *
 * Every entry point takes plain pointers and sizes.  All array pointers are
 * DEVICE pointers owned by the caller unless stated otherwise; the library
 * never allocates or frees caller memory and never synchronises inside the
 * compute calls, so they can be enqueued on any stream.  The plan
 * (hg_plan_expert_offsets), the GEMM (both scale layouts) and the
 * host-buffer call can also be captured into a CUDA graph and replayed (each
 * is tested that way).  Errors are returned as hg_status codes; nothing is
 * thrown across this interface.  Argument checks happen before any CUDA call,
 * so a bad argument is reported even on a machine without a GPU.
 *
 * Sources the operations follow (web pages, cited by title and section):
 *  [H129] humming PR #129 "perf(sm90): size grouped W4A8 tiles per expert" --
 *         benchmark command (operand formats, group sizes 128 and 32,
 *         grouped_contiguous layout) and first section (rows of one expert
 *         are one contiguous range; tile size per expert, not from total
 *         rows).
 *  [M38]  MoonEP PR #38 "fit planning block size to device SMEM limit" --
 *         the planning kernel (per-expert histogram, per-warp scratch of
 *         (E+1) x (warps+1) counts, per-expert placement), the block size
 *         chosen by dropping one warp at a time until the shared memory fits,
 *         and a resource error when even one warp does not fit.
 */
#ifndef HG_H_
#define HG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t.  NULL means the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* hg_stream_t;

typedef enum {
    HG_OK = 0,
    HG_ERR_INVALID_ARG = 1,       /* null pointer, negative size, misaligned pointer      */
    HG_ERR_UNSUPPORTED_SHAPE = 2, /* K % 128 != 0, N % 128 != 0, or a size beyond limits  */
    HG_ERR_RESOURCE = 3,          /* shared memory does not fit even the smallest block   */
    HG_ERR_CUDA = 4,              /* a CUDA runtime / driver call failed                  */
    HG_ERR_TIMEOUT = 5,           /* device: a bounded wait inside a kernel gave up        */
    HG_ERR_BAD_OFFSETS = 6,       /* device: expert_offsets not monotone or beyond rows    */
    HG_ERR_BAD_IDS = 7            /* device: an expert id outside [0, E) was dropped       */
} hg_status;

/* Static description of a status code.  Never NULL. */
const char* hg_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int hg_version(void);

/*
 * Drop the library's per-device state: the cached device properties, the
 * device addresses of its status word and of the no-allocation plan's
 * scratch array, the kernels' shared-memory settings, the
 * cluster-residency answers and the cache of encoded TMA tensor maps (keyed
 * by base address and shape).  The next call on a device queries them again.
 * Call it before using the library in a new context on a device whose
 * context was destroyed (cudaDeviceReset): the cached addresses and settings
 * belong to the old context.  Frees nothing: the status word and the scratch
 * array are module variables that live and die with their context, and the
 * library makes no device allocation of its own.  Must not run concurrently
 * with other calls of the library.  Host-only; returns HG_OK.
 */
hg_status hg_shutdown(void);

/* ---------------------------------------------------------------- plan -- */

/*
 * Bytes of device workspace hg_plan_expert_offsets needs for M tokens with
 * top_k experts each and E experts.  Pure function of its arguments (no
 * device query).  Returns 0 for invalid arguments.
 */
size_t hg_plan_workspace_bytes(int32_t M, int32_t top_k, int32_t E);

/*
 * Threads per block the plan kernels use for E experts when a block may
 * hold at most smem_limit_bytes of dynamic shared memory: the largest
 * multiple of 32 not above 512 whose per-warp count table fits [M38,
 * "修改方案"].  Returns 0 when not even 32 threads fit (the caller sees
 * HG_ERR_RESOURCE from hg_plan_expert_offsets).  Host-only.
 */
int32_t hg_plan_block_threads(int32_t E, int32_t smem_limit_bytes);

/*
 * Routing plan [M38 background; H129 first section]: turn top-k expert ids
 * into the grouped-contiguous row layout.
 *
 *   topk_ids        int32 [M, top_k], row-major; flat source index s = t*top_k + j.
 *   expert_offsets  int32 [E+1] out: exclusive prefix sum of per-expert counts;
 *                   expert e owns sorted rows [off[e], off[e+1]); off[E] = number
 *                   of in-range ids (= M*top_k when all ids are in [0, E)).
 *   sorted_to_src   int32 [M*top_k] out: source index s placed at each sorted
 *                   row, ascending s inside an expert (stable); entries at and
 *                   beyond off[E] are -1.
 *   src_to_sorted   int32 [M*top_k] out: inverse permutation; -1 for an id
 *                   outside [0, E).
 *   workspace       device scratch of at least hg_plan_workspace_bytes(M, top_k, E)
 *                   bytes (contents on entry ignored).
 *
 * Ids outside [0, E) are dropped from the layout and counted; the count is
 * reported by hg_get_device_status as HG_ERR_BAD_IDS.  M = 0 writes zero
 * offsets.  Results are bit-exact and deterministic.  Up to 32768 routed
 * rows (and E small enough for the count tables of one CTA) the plan is one
 * launch of one thread-block cluster; beyond that, two kernels
 * (hg_plan_launches tells which).  Launches on `stream`; no host
 * synchronisation.
 */
hg_status hg_plan_expert_offsets(const int32_t* topk_ids, int32_t M, int32_t top_k, int32_t E,
                                 int32_t* expert_offsets, int32_t* sorted_to_src,
                                 int32_t* src_to_sorted, void* workspace, size_t workspace_bytes,
                                 hg_stream_t stream);

/*
 * Kernel launches hg_plan_expert_offsets makes for these sizes on the
 * current device: 1 (the whole plan in one thread-block cluster, up to 32768
 * routed rows when the count tables fit) or 2 (histogram, then scatter);
 * 0 when M*top_k == 0 (the offsets are cleared with one memset); -1 for
 * arguments the plan rejects or when the device cannot be queried.
 * Host-only: launches nothing.
 */
int32_t hg_plan_launches(int32_t M, int32_t top_k, int32_t E);

/*
 * The routing plan without a workspace argument, for callers that cannot
 * call cudaMalloc where they plan: a host framework that owns every device
 * allocation through its own memory pool and does not let a library allocate
 * behind its back, or a latency-critical loop that cannot take the
 * device-wide synchronisation cudaMalloc and cudaFree may imply.  The pages
 * this library follows have no counterpart to this entry point.
 *
 * Arguments and results are those of hg_plan_expert_offsets without the
 * workspace.  The workspace is instead a fixed 256 KiB array in this
 * library's device memory; every GPU that loads the library holds it until
 * the process exits.  Shapes whose workspace (hg_plan_workspace_bytes)
 * exceeds 256 KiB are rejected with HG_ERR_RESOURCE before anything is
 * launched.  The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *
 * Every call on a device shares the one array, which keeps the last call's
 * contents; each call overwrites every entry it later reads, so nothing has
 * to be cleared between calls.  Calls whose executions overlap on the GPU
 * (different streams, or several host threads) race on the array: put them
 * on one stream or synchronise between them.  The first call on a device
 * looks up the array's device address, with that device current; make that
 * first call before any stream capture.
 */
hg_status hg_plan_expert_offsets_noalloc(const int32_t* topk_ids, int32_t M, int32_t top_k,
                                         int32_t E, int32_t* expert_offsets,
                                         int32_t* sorted_to_src, int32_t* src_to_sorted,
                                         hg_stream_t stream);

/* ---------------------------------------------------------------- GEMM -- */

/*
 * Grouped-contiguous W4A8 GEMM [H129 benchmark command and first section]:
 *
 *   out[r, n] = bf16_rne( sum_k  A(r,k) * W(e(r), n, k) ),  e(r): off[e] <= r < off[e+1]
 *   A(r,k)    = e4m3(a_fp8[r,k]) * 2^(a_scale[r, k/128] - 127)
 *   W(e,n,k)  = e2m1(w_fp4[e,n,k]) * 2^(w_scale[e, n, k/32] - 127)
 *
 *   a_fp8      uint8 [rows, K]     E4M3 codes, row-major, rows sorted by expert;
 *                                  16-byte aligned.
 *   a_scale    uint8 [rows, K/128] E8M0 codes, one per row per 128-K group, row-major.
 *   w_fp4      uint8 [E, N, K/2]   E2M1 codes, two per byte, element 2j in the low
 *                                  nibble of byte j; 32-byte aligned.
 *   w_scale    uint8 [E, N, K/32]  E8M0 codes, one per output column per 32-K group;
 *                                  4-byte aligned.
 *   expert_offsets int32 [E+1]     device array, e.g. from hg_plan_expert_offsets.
 *   rows       number of rows of a_fp8 / a_scale / out (>= off[E]).
 *   out_bf16   uint16 [rows, N]    bfloat16 bit patterns, row-major.  Rows at and
 *                                  beyond off[E] are not written.
 *
 * Accumulation is FP32 inside the tensor cores; the scales are applied per
 * 32-K block by the block-scaled MMA.  Supported: E in [1, 512],
 * N % 128 == 0, K % 128 == 0, rows in [0, 2^31).  Offsets that are not
 * monotone or exceed rows are detected on the device: the affected experts
 * are skipped and HG_ERR_BAD_OFFSETS is recorded for hg_get_device_status.
 * E2M1/E4M3 NaN codes and E8M0 code 255 are not supported inputs.
 * One persistent kernel launch on `stream`; no host synchronisation.  The
 * pipeline shape (largest token tile, CTAs per SM, split-K) is chosen from
 * the mean rows per expert, rows / E, and for launches with few weight tiles
 * per CTA from the device's resident CTA count.  Shapes differ only in FP32
 * rounding (the split-K shape sums the partial products of K ranges in K
 * order); for given arguments on a given device the result is the same on
 * every run.  The kernel is launched with programmatic dependent launch:
 * its set-up (barriers, TMEM allocation, tensor-map prefetch) may start
 * while the kernel before it on `stream` is still running, once that kernel
 * allows it (hg_plan_expert_offsets' last kernel does); it reads and writes
 * no global memory until that kernel has completed, so stream order holds
 * for every argument as with a plain launch.
 */
hg_status hg_grouped_w4a8_gemm(const uint8_t* a_fp8, const uint8_t* a_scale,
                               const uint8_t* w_fp4, const uint8_t* w_scale,
                               const int32_t* expert_offsets, int32_t E, int32_t N, int32_t K,
                               int32_t rows, uint16_t* out_bf16, hg_stream_t stream);

/*
 * The same GEMM with the activation scales in M-major order [H129 benchmark
 * command, option --use_m_major_input_scale]: a_scale_mmajor is uint8
 * [K/128, rows], the scale of row r for 128-K group g at g * rows + r.  All
 * other arguments, results and errors as hg_grouped_w4a8_gemm.
 */
hg_status hg_grouped_w4a8_gemm_mmajor(const uint8_t* a_fp8, const uint8_t* a_scale_mmajor,
                                      const uint8_t* w_fp4, const uint8_t* w_scale,
                                      const int32_t* expert_offsets, int32_t E, int32_t N,
                                      int32_t K, int32_t rows, uint16_t* out_bf16,
                                      hg_stream_t stream);

/*
 * Largest token tile (MMA N) hg_grouped_w4a8_gemm uses for these arguments:
 * an expert with r rows is cut into ceil(r / T) tiles of equal size rounded
 * up to 16 rows (32 on CTA pairs).  The choice can depend on the current
 * device's SM count and cluster occupancy, which this asks for when a
 * device is present (without one, the split-K variant is never chosen, and
 * the 224-row tiles are used above 100 rows per expert when N % 256 == 0 and
 * exactly above 256 rows per expert otherwise).  Launches nothing; 0 for
 * invalid arguments.
 */
int32_t hg_gemm_token_tile(int32_t E, int32_t N, int32_t K, int32_t rows);

/*
 * Number of CTAs hg_grouped_w4a8_gemm launches on the current device for
 * these arguments (its grids are persistent: at most one wave, fewer when
 * there are fewer work units than resident CTAs).  Queries the device (SM
 * count, cluster occupancy); -1 when that fails, 0 for unsupported
 * arguments.  Host-only; launches nothing.
 */
int32_t hg_gemm_ctas(int32_t E, int32_t N, int32_t K, int32_t rows);

/*
 * Force the GEMM pipeline variant for later calls in this process: 0 = choose
 * automatically (default), 1 = 64-row token tiles with two CTAs per SM,
 * 2 = 112-row tiles with two CTAs per SM, 4 = 224-row tiles on CTA pairs
 * (tcgen05 cta_group::2: 256 weight rows per MMA; stages of 256 K when
 * K % 256 == 0, else 128 K; used only when N % 256 == 0, else variant 8),
 * 6 = 32-row tiles with two CTAs per SM in
 * clusters of four that split the K loop of each tile over 1, 2 or 4 CTAs
 * (chosen on the device to even out the work when there are few tiles per
 * CTA; the partial sums are added in a fixed order, so results do not vary
 * from run to run), 8 = 224-row tiles with two CTAs per SM and one TMEM
 * accumulator each.  (The numbers 3, 5 and 7 belonged to shapes that were
 * never the fastest and are rejected.)  Meant for tests and tuning.
 * Returns the previous setting, or -1 for an invalid value (setting
 * unchanged).  Host-only.
 */
int32_t hg_set_gemm_variant(int32_t variant);

/* ------------------------------------------------ around the GEMM (MoE) -- */

/*
 * Quantise BF16 token activations to the GEMM's input format and gather them
 * into the plan's sorted order in one pass.  Row r of the output takes token
 * t = sorted_to_src[r] / top_k; rows with sorted_to_src[r] < 0 are not
 * written.  Per 128-element group of a row: e = the smallest integer with
 * amax <= 448 * 2^e (amax = 0 gives e = 0), clamped to [-127, 127];
 * a_scale = 127 + e (E8M0); a_fp8 = E4M3 round-to-nearest-even of x / 2^e.
 * A group holding an Inf or NaN gets scale code 0xFF and element codes 0x7F
 * (the NaN codes of both formats).  The cast is the 128-group counterpart of
 * the rowwise MXFP8 cast of TransformerEngine PR #3459 ("non-TMA MXFP8
 * cast-only kernels", description).
 *
 *   x_bf16         uint16 [M, K] BF16 bit patterns, 16-byte aligned.
 *   sorted_to_src  int32 [M*top_k] from hg_plan_expert_offsets.
 *   a_fp8          uint8 [M*top_k, K] out, 16-byte aligned; a_scale uint8 [M*top_k, K/128] out.
 * K % 128 == 0.  One kernel on `stream`; no host synchronisation.
 *
 * This is the slow form: organised per sorted row, it reads and quantises
 * every token top_k times, and the quantisation arithmetic, not memory,
 * bounds it (about 0.24 of HBM bandwidth at top_k = 8, M = 2048, K = 6144,
 * against about 0.70 for hg_quantize_scatter_acts, which writes the same
 * bytes).  Prefer hg_quantize_scatter_acts; this form serves callers that
 * hold only sorted_to_src.
 */
hg_status hg_quantize_gather_acts(const uint16_t* x_bf16, int32_t M, int32_t K, int32_t top_k,
                                  const int32_t* sorted_to_src, uint8_t* a_fp8,
                                  uint8_t* a_scale, hg_stream_t stream);

/*
 * The same quantisation as hg_quantize_gather_acts, organised per token:
 * token t is read and quantised once, and its codes and scales are stored
 * to the sorted rows src_to_sorted[t*top_k + j], j = 0 .. top_k-1 (the
 * inverse permutation hg_plan_expert_offsets returns).  Entries outside
 * [0, M*top_k) are skipped (ids the plan dropped are -1); rows no entry
 * names are not written.  For a plan's pair of permutations the result is
 * identical to hg_quantize_gather_acts, with each token read once instead
 * of top_k times.
 *
 *   x_bf16         uint16 [M, K] BF16 bit patterns, 16-byte aligned.
 *   src_to_sorted  int32 [M*top_k] from hg_plan_expert_offsets.
 *   a_fp8          uint8 [M*top_k, K] out, 16-byte aligned; a_scale uint8 [M*top_k, K/128] out.
 * K % 128 == 0; top_k <= 64 (else HG_ERR_UNSUPPORTED_SHAPE).  One kernel on
 * `stream`; no host synchronisation.  The pages have no counterpart to the
 * per-token organisation; it moves the same bytes as the gather with each
 * token read once.
 */
hg_status hg_quantize_scatter_acts(const uint16_t* x_bf16, int32_t M, int32_t K, int32_t top_k,
                                   const int32_t* src_to_sorted, uint8_t* a_fp8,
                                   uint8_t* a_scale, hg_stream_t stream);

/*
 * Combine the experts' outputs back into token order with the router's top-k
 * weights: out[t, :] = bf16_rne( sum_j w[t, j] * y[src_to_sorted[t*top_k + j], :] ),
 * the sum in FP32 over j ascending; terms with src_to_sorted < 0 (ids the
 * plan dropped) are skipped.
 *
 *   y_bf16         uint16 [M*top_k, N] BF16 (the GEMM output), 16-byte aligned.
 *   src_to_sorted  int32 [M*top_k] from hg_plan_expert_offsets.
 *   topk_weights   float32 [M, top_k].
 *   out_bf16       uint16 [M, N] out, 16-byte aligned.
 * N % 8 == 0.  One kernel on `stream`; no host synchronisation.
 */
hg_status hg_combine_topk(const uint16_t* y_bf16, const int32_t* src_to_sorted,
                          const float* topk_weights, int32_t M, int32_t top_k, int32_t N,
                          uint16_t* out_bf16, hg_stream_t stream);

/* ------------------------------------------------- from host buffers -- */

/*
 * Device workspace bytes of hg_grouped_w4a8_gemm_host for these sizes (the
 * device copies of the ids, activations, scales and output, the plan's
 * results and the plan's own workspace, each region 256-byte aligned); 0 for
 * M < 0, top_k < 1, E < 1, N < 1, K < 128 or M*top_k >= 2^31.
 */
size_t hg_gemm_host_workspace_bytes(int32_t M, int32_t top_k, int32_t E, int32_t N, int32_t K);

/*
 * The routing plan and the grouped GEMM on inputs and outputs in host
 * memory: the same computation as hg_plan_expert_offsets followed by
 * hg_grouped_w4a8_gemm with rows = M*top_k, with the host<->device copies
 * made by the library.  On `stream`, in order: copies of topk_ids, a_fp8 and
 * a_scale to the workspace; the plan; the GEMM; copies of the output (and of
 * the offsets and sorted_to_src when those pointers are non-null) back to
 * host memory.  The host buffers must stay valid and unchanged until the
 * stream reaches the end of the call; they should be page-locked
 * (cudaHostAlloc or cudaHostRegister), else the copies do not overlap other
 * work and may block the calling thread.
 *
 *   topk_ids_host        int32 [M, top_k] host.
 *   a_fp8_host           uint8 [M*top_k, K] host, E4M3 rows in the plan's order
 *                        (sorted by expert, stable), as hg_grouped_w4a8_gemm takes.
 *   a_scale_host         uint8 [M*top_k, K/128] host, E8M0.
 *   w_fp4, w_scale       device, as for hg_grouped_w4a8_gemm (weights stay
 *                        resident across calls).
 *   out_bf16_host        uint16 [M*top_k, N] host out; rows at and beyond off[E]
 *                        (dropped ids) are written with the workspace's
 *                        contents and carry no result.
 *   expert_offsets_host  int32 [E+1] host out, or NULL.
 *   sorted_to_src_host   int32 [M*top_k] host out, or NULL.
 *   workspace            device, at least hg_gemm_host_workspace_bytes bytes,
 *                        256-byte aligned; one call at a time may use it.
 *
 * Argument errors, shapes and device-detected problems as the two calls it
 * makes; a workspace that is missing, too small or misaligned is
 * HG_ERR_INVALID_ARG.  Nothing is launched or copied when an argument is
 * rejected.  No host synchronisation.
 */
hg_status hg_grouped_w4a8_gemm_host(const int32_t* topk_ids_host, const uint8_t* a_fp8_host,
                                    const uint8_t* a_scale_host, const uint8_t* w_fp4,
                                    const uint8_t* w_scale, int32_t M, int32_t top_k, int32_t E,
                                    int32_t N, int32_t K, uint16_t* out_bf16_host,
                                    int32_t* expert_offsets_host, int32_t* sorted_to_src_host,
                                    void* workspace, size_t workspace_bytes, hg_stream_t stream);

/* ------------------------------------------------------------- status -- */

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device: HG_OK, or the first device-side error recorded
 * since the last call (HG_ERR_TIMEOUT, HG_ERR_BAD_OFFSETS, HG_ERR_BAD_IDS).
 * If `detail` is not NULL it receives an error-specific value (for
 * HG_ERR_BAD_IDS the number of dropped ids; for HG_ERR_TIMEOUT the role and
 * stage of the wait that gave up).  Returns HG_ERR_CUDA if the stream or the
 * context reports an error.
 */
hg_status hg_get_device_status(hg_stream_t stream, uint32_t* detail);

/*
 * Wait-timeout self test: launches one block that waits on a barrier nobody
 * arrives at, through the same bounded wait the GEMM uses, with a limit of
 * timeout_us microseconds.  The wait gives up, records HG_ERR_TIMEOUT in the
 * status word and the kernel returns normally; the context stays usable.
 */
hg_status hg_selftest_wait_timeout(uint32_t timeout_us, hg_stream_t stream);

/*
 * Per-wait limit of the GEMM's barrier waits in microseconds (default
 * 1000000).  Host-side setting, applied to later launches.  0 restores the
 * default.
 */
void hg_set_wait_timeout_us(uint32_t timeout_us);

#ifdef __cplusplus
}
#endif

#endif /* HG_H_ */
