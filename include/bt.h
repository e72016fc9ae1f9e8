/*
 * bt.h -- C ABI of libbt: matrix products over affine group-quantized weights
 * with the dequantization done inside the compute loop (B300, sm_103a).
 *
 * What is computed.  The BaseRT pages store model weights as affine codes of
 * 2 to 8 bits (thakicloud.com, "Apple Silicon 로컬 LLM 추론의 새 기준 BaseRT",
 * section "BaseRT는 무엇인가").  Their matmul kernels are split by M: a GEMV
 * for single-token decode, a GEMM for prefill.  Both expand the codes to
 * weights inside the inner loop, so full-precision weights never go to
 * memory and the bytes read shrink with the bit width (thetesserapress.com,
 * "BaseRT claims fastest Apple Silicon inference", section "What BaseRT does
 * differently").  Every product here is
 *
 *     y[m, n] = sum_k x[m, k] * (s[n, k/g] * q[n, k] + b[n, k/g])
 *
 * with q an unsigned b-bit code.  No dequantized weight is ever written to
 * global memory.
 *
 * Packed-weight layout (all row-major, bases 16-byte aligned):
 *   codes   uint32 [N][K*bits/32]  each group of g codes is a group-local
 *           LSB-first bitstream of g*bits bits in g*bits/32 words: code j of a
 *           group is stream bits [j*bits, j*bits+bits), stream bit t is bit
 *           t%32 of the group's word t/32.  bits = 4 gives "8 codes per
 *           uint32", code j in bits [4*(j%8), +4) of word j/8.
 *   scales  fp16 bit patterns (uint16) [N][K/g]
 *   biases  fp16 bit patterns (uint16) [N][K/g]
 * Supported: bits in {2,3,4,5,6,8}; g in {32, 64, 128}; K a multiple of g.
 * Because g*bits is a multiple of 32, every 32-code slice of a row starts on a
 * word, so a row is one contiguous stream whatever g is.
 *
 * fp16 weights ("bits = 16", the FP16 end of the pages' Q2..FP16 range,
 * gist.science summary, "Metodologia"): codes holds the weights' fp16 bit
 * patterns, weight k of a row in bits [16*(k%2), +16) of word k/2 ([N][K/2]
 * words); scales and biases are not read and may be NULL.
 *
 * Conventions for every entry point:
 *   - All pointers are device memory owned by the caller; the library keeps no
 *     pointer after the call returns and allocates no device memory.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and never
 *     synchronize.  Argument errors return before any launch and leave the
 *     outputs untouched.  A failed launch returns BT_ERR_CUDA.
 *   - Results are deterministic: the same inputs give bitwise-identical
 *     outputs (no atomics in any reduction).
 *   - Device-side bounded waits that expire set a device error word, which
 *     bt_last_device_error() reports as BT_ERR_TIMEOUT.
 */
#ifndef BT_H_
#define BT_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define BT_API __attribute__((visibility("default")))
#else
#define BT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BT_OK = 0,
  BT_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, K % g != 0, bad dtype */
  BT_ERR_UNSUPPORTED = 2,  /* bits or group size not supported, size beyond a kernel limit */
  BT_ERR_MISALIGNED = 3,   /* a base pointer is not 16-byte aligned */
  BT_ERR_CUDA = 4,         /* a CUDA runtime call or a launch failed */
  BT_ERR_TIMEOUT = 5       /* a device-side bounded wait expired (see bt_last_device_error) */
} bt_status;

typedef enum { BT_F16 = 0, BT_BF16 = 1, BT_F32 = 2 } bt_dtype;

/*
 * Dequant-GEMV, M = 1 (decode): y[n] = sum_k x[k] * w_deq[n, k], n < N.
 * BaseRT pages, thetesserapress.com "What BaseRT does differently": the
 * dedicated decode GEMV with inline dequantization.
 *   codes/scales/biases  packed weight [N, K] (layout above)
 *   x        [K] of x_dtype (BT_F16 or BT_BF16)
 *   y        [N] of y_dtype (BT_F32, BT_BF16 or BT_F16); accumulation is fp32
 * Limits: N >= 1, 64 <= K <= 32768.
 */
BT_API bt_status bt_qgemv(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                   int bits, int group_size, int N, int K,
                   const void* x, bt_dtype x_dtype,
                   void* y, bt_dtype y_dtype, cudaStream_t stream);

/*
 * Batched dequant-GEMV: `count` independent M = 1 products in one launch, all
 * with the same bits, group size and dtypes, each with its own weight, x, y,
 * row count and (when K = 0) its own K.  Persistent CTAs stream the problems'
 * rows back to back, so a decode step's many small GEMVs cost one launch
 * instead of one each (BaseRT pages, thetesserapress.com "Where the wins
 * land": launch overhead dominates small models; gist.science "Contribuições":
 * cheap dispatch).
 *   problems  HOST array of `count` descriptors (read during the call only;
 *             the pointers in it are device memory, 16-byte aligned)
 *   K         > 0: every problem has this K (the descriptors' k is ignored);
 *             0: each problem uses its descriptor's k (a mixed-K batch, e.g. a
 *             whole decode step in one launch)
 * Limits: 1 <= count <= 256; each problem's K (the call's, or its own k) as
 * for bt_qgemv.  A batch that one launch cannot hold (in a mixed-K batch, a k
 * above 8192) runs as one bt_qgemv launch per problem, in order, on `stream`:
 * the results are the same, only the launch count differs.
 */
typedef struct {
  const uint32_t* codes;     /* [n, k*bits/32] */
  const uint16_t* scales;    /* [n, k/g] fp16 */
  const uint16_t* biases;    /* [n, k/g] fp16 */
  const void* x;             /* [k] of x_dtype */
  void* y;                   /* [n] of y_dtype */
  int32_t n;                 /* rows, >= 1 */
  int32_t k;                 /* this problem's K when the call's K is 0 */
} bt_gemv_problem;
BT_API bt_status bt_qgemv_batched(const bt_gemv_problem* problems, int count, int bits, int group_size,
                                  int K, bt_dtype x_dtype, bt_dtype y_dtype, cudaStream_t stream);

/*
 * Batched dequant-GEMM for a few tokens: `count` dense products that share M
 * (the tokens of one decode step), bits, group size and dtypes, each with its
 * own weight, X [M, k] and Y [M, n], in one launch.  BaseRT pages,
 * thetesserapress.com "What BaseRT does differently" (more than one token runs
 * a GEMM) and "Where the wins land, and where they don't" (launch overhead
 * dominates small models), the M > 1 counterpart of bt_qgemv_batched.
 *   problems  HOST array of `count` descriptors (read during the call only;
 *             the pointers in it are device memory: codes and X 16-byte
 *             aligned, scales and biases 8-byte aligned for the one-launch path)
 *   M         rows of every X and Y (tokens)
 * M = 2..8 with fp16 x, bits = 4, group_size = 64 and every K a multiple of
 * 256 runs as one launch of the batched GEMV's four-column consumer, the
 * tokens sharing the MMA's columns with the groups (each weight read and
 * unpacked once for all tokens; up to 256 problems per launch).  Otherwise one launch of the
 * small-token tensor-pipe kernel (path 4 of bt_plan_gemm)
 * takes the whole table when M <= 16, bits = 4, group_size = 64 and every
 * problem has K a multiple of 256 and n a multiple of 8, and the x of the
 * largest K fits the kernel's staging (up to 120 problems per launch; longer
 * tables take several).  M = 1 runs as one bt_qgemv_batched
 * launch.  Anything else runs one bt_qgemm per problem, in order, on `stream`:
 * the results are the same, only the launch count differs.
 * Errors: as for bt_qgemm, for the first problem that fails a check (nothing
 * is launched then); BT_ERR_INVALID_ARG for count < 1 or M < 1.
 */
typedef struct {
  const uint32_t* codes;     /* [n, k*bits/32] */
  const uint16_t* scales;    /* [n, k/g] fp16 */
  const uint16_t* biases;    /* [n, k/g] fp16 */
  const void* x;             /* [M, k] of x_dtype */
  void* y;                   /* [M, n] of y_dtype */
  int32_t n;
  int32_t k;
} bt_gemm_problem;
BT_API bt_status bt_qgemm_batched(const bt_gemm_problem* problems, int count, int bits, int group_size, int M,
                                  bt_dtype x_dtype, bt_dtype y_dtype, cudaStream_t stream);

/*
 * Decode pass: an ordered list of stages of products over buffers the caller
 * sized once, planned once and then replayed as one CUDA graph per call.
 * BaseRT pages, gist.science "Metodologia" (the decode loop allocates nothing:
 * every buffer is sized at load and a step is only GPU dispatch plus light
 * host-side patching) and thetesserapress.com "What BaseRT does differently"
 * (residuals, scratch and intermediates pre-sized and reused).
 *
 * A stage is a set of independent products with the same M, bits, group size
 * and dtypes, as for bt_qgemm_batched; stage s + 1 may read what stage s
 * writes (its x may be an earlier stage's y), and stages run in order.
 *   stages      HOST array of `num_stages` stage descriptors; each stage's
 *               `problems` is a HOST array of `count` bt_gemm_problem.  Both
 *               are read during bt_pass_create only: the pass keeps its own
 *               copy of every pointer and size.
 *   pass        receives the new pass; the caller owns it and frees it with
 *               bt_pass_destroy.
 * The device pointers inside the problems (weights, x, y) stay the caller's:
 * they must stay valid, and keep their sizes, for the life of the pass.  The
 * caller changes a run's inputs by writing new values into the same x
 * buffers (on the stream it runs the pass on, or before).
 *
 * bt_pass_create validates and plans every stage (the checks of
 * bt_qgemm_batched, the launch tables, the tensor maps) on the host; it
 * launches nothing.  It binds the pass to the current device.
 * bt_pass_run launches the pass on `stream`.  The first run launches every
 * stage directly (this loads the kernels and makes the per-device settings)
 * and then records the same launches into a CUDA graph on a stream the pass
 * owns; every later run is one cudaGraphLaunch of that graph, with no host
 * allocation, no validation and no planning.  The options in force at the
 * first run (PDL, the constant-weights hint, the wait bound) are the ones the
 * graph keeps.  Call the first run outside any stream capture; later runs
 * may themselves be captured.  Runs of one pass on two streams at once race
 * on the pass's y buffers.
 * Errors: bt_pass_create returns the first check that fails (as for
 * bt_qgemm_batched) and sets *pass to NULL; BT_ERR_INVALID_ARG for a NULL
 * `pass` or `stages` or num_stages < 1.  bt_pass_run returns
 * BT_ERR_INVALID_ARG for a NULL pass or a current device other than the
 * pass's, BT_ERR_CUDA when a launch, the recording or the graph launch
 * fails.  bt_pass_destroy accepts NULL; call it only once no run of the
 * pass is in flight (after the run's stream has been synchronised).
 */
typedef struct bt_pass bt_pass;
typedef struct {
  const bt_gemm_problem* problems;
  int count;
} bt_pass_stage;
BT_API bt_status bt_pass_create(const bt_pass_stage* stages, int num_stages, int bits, int group_size, int M,
                                bt_dtype x_dtype, bt_dtype y_dtype, bt_pass** pass);
BT_API bt_status bt_pass_run(bt_pass* pass, cudaStream_t stream);
BT_API void bt_pass_destroy(bt_pass* pass);

/*
 * Dequant-GEMM, M > 1 (prefill): Y[m, n] = sum_k X[m, k] * w_deq[n, k].
 * BaseRT pages, thetesserapress.com "What BaseRT does differently" (prefill,
 * with several tokens, runs a GEMM) and gist.science "Metodologia" (tiled
 * prefill GEMM on the matrix units).  Weights are dequantized in registers and fed to the
 * tensor cores (M >= 64) or to a CUDA-core tile (small M); fp32 accumulation.
 *   X  [M, K] row-major, x_dtype BT_BF16 or BT_F16
 *   Y  [M, N] row-major, y_dtype BT_BF16, BT_F16 or BT_F32
 * M = 1 is accepted and runs the GEMV.  Limits: 1 <= M, 64 <= K <= 32768.
 */
BT_API bt_status bt_qgemm(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                   int bits, int group_size, int M, int N, int K,
                   const void* x, bt_dtype x_dtype,
                   void* y, bt_dtype y_dtype, cudaStream_t stream);

/*
 * Grouped expert GEMM: for each expert e, rows r in [off[e], off[e+1]) of the
 * grouped activation matrix use expert e's weight:
 *     Y[r, n] = sum_k Xg[r, k] * w_deq_e[n, k].
 * BaseRT pages, thetesserapress.com "Where the wins land, and where they
 * don't" (the MoE prefill lead, credited to code that does not fork on the
 * experts a token picked).
 *   codes/scales/biases  experts stacked: [E][N][K*bits/32], [E][N][K/g]
 *   expert_offsets  device int32 [E+1], non-decreasing, off[0] = 0,
 *                   off[E] = total_rows; experts may be empty
 *   x_row_index     device int32 [total_rows] or NULL.  When given, grouped
 *                   row r reads X row x_row_index[r] (a gather); when NULL,
 *                   X is already in grouped order, [total_rows, K]
 *   x     X of x_dtype (BT_F16 or BT_BF16), rows of K elements
 *   y     [total_rows, N] of y_dtype, grouped order
 * Offsets are read on the device; rows outside [0, total_rows) are never
 * touched.  Limits: E >= 1, total_rows >= 0, 64 <= K <= 32768.
 */
BT_API bt_status bt_moe_qgemm(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                       int bits, int group_size, int num_experts, int N, int K,
                       const int32_t* expert_offsets, int total_rows,
                       const int32_t* x_row_index,
                       const void* x, bt_dtype x_dtype,
                       void* y, bt_dtype y_dtype, cudaStream_t stream);

/*
 * Grouped expert product with the SwiGLU epilogue fused into its store: the
 * gate and up products of an expert layer in one launch whose output is
 * already the activation h = silu(gate . x) * (up . x).  BaseRT pages,
 * gist.science "Metodologia" (fusing two kernels saves a dispatch and a trip
 * through memory); thetesserapress.com "Where the wins land, and where they
 * don't" (the expert layers).
 *   codes/scales/biases  experts stacked [E][N][...] with N = 2*I rows in
 *                        interleaved order: row 2i is gate row i, row 2i+1 is
 *                        up row i (so every gate/up pair is produced together)
 *   expert_offsets, total_rows, x_row_index, x   as bt_moe_qgemm
 *   h     [total_rows, I] of h_dtype (BT_F32, BT_BF16 or BT_F16), grouped order
 * Runs on the GEMV (at most one row per expert), the tensor cores or the
 * CUDA-core tile like bt_moe_qgemm; silu is evaluated in fp32 on the fp32
 * accumulators.  Errors: BT_ERR_INVALID_ARG for an odd N, otherwise as
 * bt_moe_qgemm.
 */
BT_API bt_status bt_moe_qgemm_swiglu(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                                     int bits, int group_size, int num_experts, int N, int K,
                                     const int32_t* expert_offsets, int total_rows, const int32_t* x_row_index,
                                     const void* x, bt_dtype x_dtype, void* h, bt_dtype h_dtype,
                                     cudaStream_t stream);

/*
 * Expert products of routed (token, slot) pairs at decode, without a sort: pair
 * r = t*top_k + s uses expert topk_ids[r] and x row t, and writes output row r
 * (pair order).  The experts a token picked are data read on the device, so no
 * host code forks on them (thetesserapress.com "Where the wins land, and where
 * they don't"; gist.science "Contribuições").  With swiglu != 0 the weight rows
 * are gate/up interleaved as in bt_moe_qgemm_swiglu and the output rows hold
 * N/2 activations.
 *   topk_ids  device int32 [tokens, top_k], each in [0, E); an id out of range
 *             sets the device error word (BT_ERR_INVALID_ARG from
 *             bt_last_device_error) and its pair's output is not written
 *   x         [tokens, K] of x_dtype;  y [tokens*top_k, N or N/2] of y_dtype
 * Runs on the GEMV kernel only: BT_ERR_UNSUPPORTED when no GEMV plan fits
 * (K above the GEMV's limit for the width).  Limits: 1 <= top_k <= 32.
 */
BT_API bt_status bt_moe_qgemv_pairs(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, int bits,
                                    int group_size, int num_experts, int N, int K, const int32_t* topk_ids,
                                    int tokens, int top_k, const void* x, bt_dtype x_dtype, void* y,
                                    bt_dtype y_dtype, int swiglu, cudaStream_t stream);

/*
 * Down products of a token's routed experts with the gate-weighted combine
 * fused into the store (decode):
 *     out[t, n] = sum_{s < top_k} gates[t, s] * sum_k w_deq_{e(t,s)}[n, k] * h[t*top_k + s, k]
 * with e(t, s) = topk_ids[t, s].  Each token is one product over top_k K
 * segments, one per expert, summed inside the kernel in slot order (no
 * atomics, deterministic).  BaseRT pages, gist.science "Metodologia" (fusing
 * two kernels saves a dispatch and a trip through memory); thetesserapress.com
 * "Where the wins land, and where they don't" (the expert layers).
 *   codes/scales/biases  down weights stacked [E][N][K*bits/32], [E][N][K/g]
 *   topk_ids  device int32 [tokens, top_k]; gates device float32 [tokens, top_k]
 *   h         [tokens*top_k, K] of h_dtype (BT_F16 or BT_BF16), pair order (the
 *             output of bt_moe_qgemv_pairs with the SwiGLU epilogue)
 *   out       [tokens, N] of out_dtype
 * Each x segment is gates[t, s] * h[t*top_k + s] (rounded once to fp16 on the
 * fp16 path).  Every expert's weight rows are read once per token, so this is
 * for decode; at prefill sizes run the grouped down product and
 * bt_moe_combine.  Errors: BT_ERR_UNSUPPORTED when top_k*K exceeds the GEMV's
 * K or an expert plane is not 16-byte sized (N*K*bits/8 or N*(K/g)*2 not a
 * multiple of 16); ids out of range set the device error word and their
 * token's output is not written.
 */
BT_API bt_status bt_moe_down_combine(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                                     int bits, int group_size, int num_experts, int N, int K,
                                     const int32_t* topk_ids, const float* gates, int tokens, int top_k,
                                     const void* h, bt_dtype h_dtype, void* out, bt_dtype out_dtype,
                                     cudaStream_t stream);

/*
 * Expert routing step of a mixture-of-experts layer: groups the T*top_k
 * (token, slot) pairs by expert id with a stable counting sort, so that within
 * an expert the pairs keep (token, slot) order.
 *   topk_ids        device int32 [T, top_k], each in [0, E)
 *   expert_offsets  device int32 [E+1] (out)
 *   pair_index      device int32 [T*top_k] (out): grouped row r holds pair
 *                   pair_index[r] = t*top_k + slot
 *   pair_row        device int32 [T*top_k] (out): inverse of pair_index
 *   pair_token      device int32 [T*top_k] (out, may be NULL): token of grouped
 *                   row r, pair_index[r] / top_k -- the x_row_index that
 *                   gathers the layer input for the grouped product
 * Ids outside [0, E) set the device error word and are placed in no group
 * (bt_last_device_error then returns BT_ERR_INVALID_ARG).
 * Limits: T >= 0, 1 <= top_k <= 32, 1 <= E <= 4096.
 */
BT_API bt_status bt_moe_route(const int32_t* topk_ids, int tokens, int top_k, int num_experts,
                       int32_t* expert_offsets, int32_t* pair_index, int32_t* pair_row,
                       int32_t* pair_token, cudaStream_t stream);

/*
 * SwiGLU between the gate/up and down products: h[r, i] = silu(a[r, i]) * a[r, I + i]
 * for a = [gate | up] of shape [rows, 2*I] (dtype BT_F32, BT_BF16 or BT_F16);
 * h is [rows, I] of h_dtype.  Computed in fp32.
 */
BT_API bt_status bt_swiglu(const void* gate_up, bt_dtype in_dtype, int rows, int inter,
                    void* h, bt_dtype h_dtype, cudaStream_t stream);

/*
 * Weighted combine of expert outputs: out[t, :] = sum_{s < top_k} gates[t, s] *
 * Yg[pair_row[t*top_k + s], :], summed in slot order in fp32.
 *   y_grouped  [T*top_k, H] of y_dtype (grouped order)
 *   gates      device float32 [T, top_k]
 *   pair_row   device int32 [T*top_k] from bt_moe_route
 *   out        [T, H] of out_dtype
 */
BT_API bt_status bt_moe_combine(const void* y_grouped, bt_dtype y_dtype, const float* gates,
                         const int32_t* pair_row, int tokens, int top_k, int hidden,
                         void* out, bt_dtype out_dtype, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
BT_API const char* bt_status_string(bt_status status);

/*
 * Synchronizes `stream`, then reads and clears the device error word.
 * Returns BT_OK, BT_ERR_TIMEOUT (a bounded wait expired), BT_ERR_INVALID_ARG
 * (a device-side argument check failed, e.g. a routing id out of range) or
 * BT_ERR_CUDA (the synchronization itself failed).
 */
BT_API bt_status bt_last_device_error(cudaStream_t stream);

/*
 * Launch options.  They are process-wide: one value per option for every
 * thread, stream and device of the process, read when a call plans its launch.
 * Setting an option while another thread is inside a call is safe (each value
 * is a relaxed atomic), but which value that call sees is not defined; set
 * options before launching work that depends on them.
 *   BT_OPT_PDL          1: launch with programmatic dependent launch so a call's
 *                       prologue overlaps the previous kernel on the stream.
 *   BT_OPT_CONST_WEIGHTS 1 (with PDL): the caller promises that the packed
 *                       weights are not written by the kernel launched just
 *                       before on the same stream, so weight loads may start
 *                       before that kernel finishes.  Activations are always
 *                       read after it finishes.
 *   BT_OPT_WAIT_TIMEOUT_US  bound of every device-side wait, microseconds
 *                       (default 4,000,000).
 *   BT_OPT_TEST_DROP_STAGE  test hook, 1: the next GEMV launch leaves its first
 *                       pipeline stage unfilled in CTA 0, so that CTA's waits
 *                       expire after BT_OPT_WAIT_TIMEOUT_US and the call reports
 *                       BT_ERR_TIMEOUT through bt_last_device_error().  Resets
 *                       itself after one launch.
 *   BT_OPT_GEMV_GENERIC  tuning, 1: GEMV uses the generic unpack path for all bits.
 *   BT_OPT_GEMV_STAGES   tuning: GEMV pipeline depth (0 = heuristic, else 2..8).
 *   BT_OPT_GEMM_PATH     tuning: 0 = heuristic, 1 = CUDA-core tile,
 *                       2 = tensor-core tile where supported, 3 = small-token
 *                       tensor-pipe kernel where supported (bt_qgemm at M = 1
 *                       included, which otherwise takes the GEMV).
 *   BT_OPT_GEMM_SPLITS   tuning: tensor-core GEMM K split across a cluster (0 = heuristic, 1..8).
 *   BT_OPT_GEMV_MAX_CPL  tuning: GEMV chunks of 32 codes per lane before K is split
 *                       over more warps (0 = heuristic, else 1..4).
 *   BT_OPT_GEMV_STAGE_KB tuning: GEMV pipeline stage size in KiB (0 = heuristic, else 4..96).
 *   BT_OPT_GEMV_RI       tuning: GEMV rows in flight per warp (0 = heuristic, else 1, 2, 4 or 8).
 *   BT_OPT_GEMV_CUDA_CORE tuning, 1: GEMV on the CUDA-core kernel even where the
 *                       tensor-pipe one applies (4-bit codes, fp16 x, K <= 8192).
 *   BT_OPT_GEMM_DEQ_WARPS tuning: tensor-core GEMM dequantizing warps per CTA,
 *                       8 (one set) or 16 (two sets on alternating K blocks);
 *                       0 = default: 16 for bt_qgemm, 8 for the grouped expert
 *                       launches (two CTAs per SM there).
 *   BT_OPT_GEMM_SMALL_WARPS tuning: consumer warps per CTA of the small-token
 *                       kernel (path 4 of bt_plan_gemm), 8 or 16; 0 = 16 where
 *                       that layout fits shared memory and at most 16 tokens
 *                       share a staging of x, else 8.
 *   BT_OPT_GEMV_TENSOR_PIPE tuning: 0 = by launch (default): the tensor-pipe
 *                       GEMV's diagonal consumer for launches of at most one
 *                       16-row tile per SM, its four-column consumer for
 *                       launches of at least eight tiles per SM whose every K
 *                       is a multiple of 256 and at most 4096, else the
 *                       CUDA-core kernel;
 *                       1 = the tensor pipe wherever it
 *                       applies; 2 = never.
 *   BT_OPT_GEMV_MMA_STAGE_KB tuning: tensor-pipe GEMV stage size in KiB (0 = heuristic, else 8..112).
 *   BT_OPT_GEMV_MMA_SHAPE tuning: tensor-pipe GEMV kernel shape, 0 = default,
 *                       1: 8 consumer warps, 1 CTA per SM, two steps per loop
 *                       iteration; 2: the same, one step; 3: 16 consumer warps,
 *                       1 CTA per SM; 4: 8 consumer warps, 2 CTAs per SM;
 *                       5, 6, 7: the four-column consumer (each MMA covers four
 *                       quantization groups of 16 rows) with 8 warps and 1 CTA,
 *                       8 warps and 2 CTAs, 16 warps and 1 CTA per SM.  A launch
 *                       with some K not a multiple of 256 takes shape 0 instead.
 *   BT_OPT_GEMV_MMA_GROUPS tuning: most quantization groups of K one warp of the
 *                       tensor-pipe GEMV takes before K is split over more warps
 *                       (0 = heuristic).
 */
typedef enum {
  BT_OPT_PDL = 0,
  BT_OPT_CONST_WEIGHTS = 1,
  BT_OPT_WAIT_TIMEOUT_US = 2,
  BT_OPT_TEST_DROP_STAGE = 3,
  BT_OPT_GEMV_GENERIC = 4,
  BT_OPT_GEMV_STAGES = 5,
  BT_OPT_GEMM_PATH = 6,
  BT_OPT_GEMM_SPLITS = 7,
  BT_OPT_GEMV_MAX_CPL = 8,
  BT_OPT_GEMV_STAGE_KB = 9,
  BT_OPT_GEMV_RI = 10,
  BT_OPT_GEMV_CUDA_CORE = 11,
  BT_OPT_GEMV_MMA_STAGE_KB = 12,
  BT_OPT_GEMV_MMA_SHAPE = 13,
  BT_OPT_GEMV_MMA_GROUPS = 14,
  BT_OPT_GEMV_TENSOR_PIPE = 15,
  BT_OPT_GEMM_DEQ_WARPS = 16,
  BT_OPT_GEMM_SMALL_WARPS = 17
} bt_option;
/* Returns BT_ERR_INVALID_ARG for an unknown option or a negative value. */
BT_API bt_status bt_set_option(bt_option option, long long value);

/*
 * GEMV launch plan (host only, no CUDA call): what bt_qgemv / bt_qgemv_batched
 * would launch on a device with `sms` multiprocessors, under the current
 * options.  The per-shape launch heuristics (BaseRT pages, gist.science
 * "Metodologia": kernel choice and threadgroup sizes per chip) in inspectable
 * form, for tests and tuning.
 *   feasible      0: no GEMV kernel fits (the library runs the CUDA-core tile)
 *   tensor_pipe   0: the CUDA-core kernel; the tensor-pipe kernel (dot
 *                 products on mma.sync) with 1: the diagonal consumer (one
 *                 group per lane group and MMA), 2: the four-column consumer
 *                 (four groups of 16 rows per MMA)
 *   kw            warps sharing one row (K split); cpl: 32-code chunks per lane
 *   ri            rows in flight per warp (16 on the tensor pipe: one MMA tile);
 *                 rows_per_unit: rows per pipeline stage
 *   stage_bytes, stages, smem_bytes   shared-memory ring of one CTA
 *   ctas_per_sm   CTAs per SM the kernel is built for; grid: CTAs launched
 */
typedef struct {
  int32_t feasible, kw, cpl, ri, rows_per_unit, stage_bytes, stages, ctas_per_sm, grid;
  int64_t num_units, smem_bytes;
  int32_t tensor_pipe;
} bt_gemv_plan;
/* One problem shape repeated `problems` times (bt_qgemv: problems = 1). */
BT_API bt_status bt_plan_gemv(int bits, bt_dtype x_dtype, int N, int K, int problems, int sms,
                              bt_gemv_plan* plan);
/* A mixed-K batch: n[i], k[i] per problem; kw[i] and rows_per_unit[i] receive
 * each problem's geometry (host arrays of `count`). */
BT_API bt_status bt_plan_gemv_batch(int bits, bt_dtype x_dtype, const int32_t* n, const int32_t* k, int count,
                                    int sms, bt_gemv_plan* plan, int32_t* kw, int32_t* rows_per_unit);

/*
 * Launch plan of a dense (num_experts = 0) or grouped (num_experts > 0, M rows
 * in total) product (host only, no CUDA call): what bt_qgemm / bt_moe_qgemm
 * would launch for these sizes on `sms` multiprocessors under the current
 * options, assuming 16-byte aligned pointers.  The per-shape kernel choice
 * and tiling (BaseRT pages, gist.science "Metodologia") in inspectable form.
 *   path       0 no launch (grouped, M = 0); 1 GEMV; 2 CUDA-core tile;
 *              3 tensor cores (tcgen05); 4 small-token tensor-pipe kernel
 *              (mma.sync, tokens as the MMA's N: dense M <= 8, or grouped
 *              with at most 16 rows per expert on average; 4-bit codes,
 *              groups of 64, K a multiple of 256, N a multiple of 8)
 *   feasible   0: these sizes exceed the chosen kernel's limits (the call
 *              would return BT_ERR_CUDA)
 *   bn         token-tile width (the MMA's N on path 3; 32 on path 2; on
 *              path 4 the tokens that share one staging of x)
 *   splits     K split: CTAs per cluster on path 3; on path 4 the warps that
 *              split one 16-row tile's K range
 *   stages     ring depth (paths 1, 3 and 4); k_blocks: most 64-wide K blocks
 *              one split walks (path 3)
 *   grid_*     launch grid; smem_bytes: dynamic shared memory per CTA
 *   rows_per_unit  weight rows per ring stage (path 4)
 * Errors: BT_ERR_INVALID_ARG for a null plan, M < 0 (or 0 when dense),
 * N <= 0, K not a positive multiple of 64, num_experts outside [0, 4096],
 * sms <= 0 or a bad x_dtype; BT_ERR_UNSUPPORTED for bits or K beyond limits.
 */
typedef struct {
  int32_t path, feasible, bn, splits, stages, k_blocks, grid_x, grid_y, grid_z;
  int64_t smem_bytes;
  int32_t rows_per_unit;
} bt_gemm_plan;
BT_API bt_status bt_plan_gemm(int bits, bt_dtype x_dtype, int M, int N, int K, int num_experts, int sms,
                              bt_gemm_plan* plan);

#ifdef __cplusplus
}
#endif
#endif /* BT_H_ */
