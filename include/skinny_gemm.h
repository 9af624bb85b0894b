/*
 * skinny_gemm.h — C ABI of the GB300 (sm_103a) skinny BF16 decode projection.
 *
 *   out[M, N] = x[M, K] @ W[N, K]^T,   1 <= M <= 256 tokens (decode: 1..64),
 *   x and W bf16, accumulation fp32, out bf16 (round to nearest even) or fp32.
 *
 * Operation: page "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.
 * gemm.warp_splitk", class PreparedWarpSplitK docstring (out[M, N] = x[M, K]
 * @ weight[N, K]^T, x and out packed row-major, 32 B aligned); page
 * "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.gemm.projection",
 * class PreparedProjection (prepare once, then run(x, out) into a
 * caller-owned out; BF16 or FP32 output).  FP16 operands are also accepted
 * (same projection page: "BF16/FP16 [N, K]" weights), with FP16 or FP32 output.
 *
 * Conventions for every entry point:
 *   - Pointers named W, x, out, fa, out_* are DEVICE pointers on the current
 *     CUDA device; pointers named *_host are HOST pointers.  Sizes are in
 *     elements unless the name ends in _bytes.  Matrices are row-major with a
 *     unit inner stride; ld* is the row pitch in elements.
 *   - A stream argument is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream).  Events are cudaEvent_t passed as void*.
 *   - Functions returning int return SKG_OK (0) or one of the codes below;
 *     skinny_gemm_last_error() then describes the failure (thread-local
 *     string, valid until the next call on the same thread).
 *   - Nothing here allocates, synchronizes or copies between host and device
 *     except where a function says so.
 */
#ifndef SKINNY_GEMM_H_
#define SKINNY_GEMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SKINNY_GEMM_ABI_VERSION 1
#define SKINNY_GEMM_MAX_M 256

typedef struct skinny_gemm_plan* skinny_gemm_t; /* opaque prepared projection */

/* Element types.  W and x: SKG_BF16 or SKG_FP16 (both operands the same type).
 * out: SKG_FP32 or the operands' own type (projection page, PreparedProjection:
 * "BF16/FP16 [N, K]" weights, output dtype BF16 or FP32). */
enum skinny_gemm_dtype { SKG_BF16 = 0, SKG_FP16 = 1, SKG_FP32 = 2 };

/* Return codes.  The pages raise ValueError for the EINVAL/EALIGN cases
 * (warp_splitk page, PreparedWarpSplitK.__init__; projection page,
 * PreparedProjection.__init__ and .run) and fall back (None) where a token
 * count has no kernel (low_latency_gemm page, select_kimi_k3_backend). */
enum skinny_gemm_status {
  SKG_OK = 0,
  SKG_EINVAL = 1,          /* bad handle, shape, pitch or dtype */
  SKG_EALIGN = 2,          /* pointer or row pitch not 16-byte aligned */
  SKG_EUNSUPPORTED_M = 3,  /* M outside 1..256: caller falls back */
  SKG_EDEVICE = 4,         /* current device is not sm_103 */
  SKG_ECUDA = 5,           /* a CUDA runtime/driver call failed */
  SKG_ECAPTURING = 6,      /* prepare/autotune called while the stream captures */
  SKG_ETIMEOUT = 7,        /* a device-side bounded wait expired (watchdog) */
  SKG_ECHECK = 8           /* checked build only: a device-side bounds check failed */
};

/* Flags for skinny_gemm_prepare_ex. */
#define SKG_PREPARE_NO_TUNE_CACHE 0x1u /* ignore SKINNY_GEMM_TACTIC_FILE */
/* Launch without programmatic dependent launch: each projection then starts
 * only after the previous kernel on the stream has finished, so its weight
 * prologue no longer overlaps that kernel (for measuring what the overlap
 * hides, or for streams mixing kernels that must not overlap at all). */
#define SKG_PREPARE_NO_PDL 0x2u
/* Keep every output bit-reproducible run to run: the autotuners then leave
 * out tactics with run-time K sharing (":w", see skinny_gemm_set_tactic),
 * whose fp32 summation order depends on which CTA of a cluster took which
 * K box.  Without this flag a tuned plan may use them (each result is still
 * within the acceptance bound; only its last bits may vary).  The default,
 * untuned plan always has a fixed order. */
#define SKG_PREPARE_DETERMINISTIC 0x4u

/*
 * Prepare a projection for weight W[N, K] (packed, row pitch K).
 * Validates W, encodes its TMA maps (box {64, rows}, 128-byte swizzle,
 * 256-byte L2 promotion, out-of-bounds zero fill; projection page,
 * weight_map) and builds the {M: tactic} plan for M = 1..256 (low_latency_gemm
 * page, module docstring: the static part of the choice is resolved once, the
 * per-call path is one lookup).  A tactic for M is the one of the smallest
 * token tile >= M (glm5next gemm page, Projection.__init__).
 *
 * W is BORROWED: the handle stores its address; W must stay allocated and
 * must not move while the handle lives (its contents may change between
 * runs).  Requirements: N >= 1, K >= 8, K % 8 == 0, W 16-byte aligned;
 * dtype SKG_BF16 or SKG_FP16; out_dtype SKG_FP32 or equal to dtype.
 * Allocates a small device status word (the watchdog) and clears it with a
 * synchronous memset, so it must be called before CUDA graph capture
 * (low_latency_gemm page, autotune_kda_qkvg: compiled/tuned before capture).
 * Refused with NULL / ECAPTURING, before any device work, when a capture is
 * visible from the calling thread: the per-thread default stream capturing,
 * or the legacy stream capturing or tied to a capturing blocking stream.  (A
 * capture on a non-blocking stream in another thread is not visible; the
 * allocation then fails with ECAPTURING and the driver may invalidate that
 * capture.)
 *
 * Plan sources, by the environment variable SKINNY_GEMM_TUNE read here:
 *   "off"    the built-in default tactic for every M (tactic file ignored);
 *   "cache"  (default) the default plan, with the entries of the file named
 *            by SKINNY_GEMM_TACTIC_FILE for this device/N/K/dtypes applied;
 *   "full"   as "cache", then M = 1, 2, 4, 8, 16, 32, 48, 64 not found in the
 *            file are autotuned here (skinny_gemm_autotune on the legacy
 *            stream: synchronizes, allocates scratch) and appended to it.
 * Any other value: NULL / EINVAL.  SKG_PREPARE_NO_TUNE_CACHE means "off".
 * Returns NULL on error (see skinny_gemm_last_error / skinny_gemm_last_status).
 */
skinny_gemm_t skinny_gemm_prepare(const void* W, int64_t N, int64_t K, int dtype, int out_dtype);

/* As skinny_gemm_prepare with an explicit row pitch ldw >= K (ldw % 8 == 0),
 * so a row slice or column slice of a larger weight can be prepared in place
 * (projection page, weight_map: "row pitch kept").  flags: SKG_PREPARE_*. */
skinny_gemm_t skinny_gemm_prepare_ex(const void* W, int64_t N, int64_t K, int64_t ldw,
                                     int dtype, int out_dtype, unsigned flags);

/*
 * out[M, N] = x[M, K] @ W^T on `stream`: one kernel launch, no allocation,
 * no synchronization, no host<->device copy, so it can be captured in a CUDA
 * graph.  x: device [M, K] packed (pitch K), 16-byte aligned.  out: device
 * [M, N] packed (pitch N), 16-byte aligned base, in the prepared output dtype,
 * caller-owned (projection page, PreparedProjection.run writes into out and
 * returns it).  Rows >= M of x are never read and rows >= M of out are never
 * written.  The launch carries programmatic dependent launch: the weight's
 * first tiles are fetched before the kernel waits for the previous kernel on
 * the stream (warp_splitk page, module docstring).
 * Errors: EINVAL (bad handle/pointers), EUNSUPPORTED_M, EALIGN, ECUDA.
 */
int skinny_gemm_run(skinny_gemm_t h, const void* x, int64_t M, void* out, void* stream);

/* As skinny_gemm_run with row pitches: x rows ldx >= K apart (ldx % 8 == 0,
 * since x is read by TMA), out rows ldo >= N apart (any pitch; out is written
 * with plain stores).  Used to feed a column slice of one output to the next
 * projection. */
int skinny_gemm_run_strided(skinny_gemm_t h, const void* x, int64_t ldx, int64_t M,
                            void* out, int64_t ldo, void* stream);

/*
 * out[M, N] = x[M, K] @ W^T + residual[M, N], fused: the residual (in the
 * prepared output type, row pitch ldr >= N, aligned to its element size) is
 * added to the fp32 sum before the one rounding to the output type (page
 * "vllm.models.kimi_k3.nvidia.low_latency_gemm", try_low_latency_gemm(x,
 * weight, residual) and select_kimi_k3_backend(..., has_residual)).
 * residual may be out itself (same pointer and pitch: in place); any other
 * overlap with out is rejected (EINVAL).  Otherwise as skinny_gemm_run_strided.
 */
int skinny_gemm_run_residual(skinny_gemm_t h, const void* x, int64_t ldx, int64_t M,
                             const void* residual, int64_t ldr, void* out, int64_t ldo,
                             void* stream);

/*
 * End-to-end call with HOST buffers: copies x_host [M, K] (pinned host memory
 * gives an asynchronous copy) into a device staging buffer owned by the
 * handle, runs the projection, copies the result into out_host [M, N] and
 * synchronizes `stream` before returning.  The staging buffers are allocated
 * on the first call (not capturable).  Calls on one handle must not overlap.
 */
int skinny_gemm_run_host(skinny_gemm_t h, const void* x_host, int64_t M, void* out_host,
                         void* stream);

/* The same three steps as skinny_gemm_run_host (H2D of x into the handle's
 * staging buffer, the projection, D2H of out), enqueued on `stream` without
 * waiting: the caller synchronizes the stream before reading out_host, and
 * keeps both host buffers alive until then.  Pinned host memory makes the
 * copies asynchronous (pageable memory works but the copies then block).  Two
 * calls on one handle must be on the same stream (they share the staging
 * buffers).  The first call per handle allocates the staging buffers. */
int skinny_gemm_run_host_async(skinny_gemm_t h, const void* x_host, int64_t M, void* out_host,
                               void* stream);

/*
 * The two-stream decode step (low_latency_gemm page, run_kda_projection_overlap:
 * hidden [M, 7168], packed Q/K/V/G/F_A/beta weight [6288, 7168], F_B weight
 * [1536, 128], an aux stream running "F_A/beta then F_B", start and
 * completion events for the fork and the join).
 *   main:  out_main[M, N_main] = x @ W_main^T                  (h_main)
 *   aux:   fa[M, N_fa]         = x @ W_fa^T                    (h_fa, bf16 out)
 *          out_fb[0][M, N_fb]  = fa @ W_fb^T                   (h_fb)
 *          out_fb[i][M, N_fb]  = out_fb[i-1][:, :K_fb] @ W_fb^T, i = 1..chain-1
 * out_fb holds `chain` consecutive [M, N_fb] blocks.  h_fb's K must equal
 * h_fa's N; h_fa must have bf16 output; for chain > 1, h_fb must have bf16
 * output and N_fb >= K_fb.  Records fork_event on main, makes aux wait on it,
 * records join_event on aux after the chain and makes main wait on it.  No
 * synchronization: the whole step can be captured from `main`.
 * Every launch's arguments are checked before the fork is recorded: x, fa and
 * out_fb must be 16-byte aligned device pointers (out_main too), and for
 * chain > 1 the F_B rows must be 16-byte multiples (N_fb % 8 == 0), since each
 * link reads the previous block by TMA.  A refused step enqueues nothing
 * (EINVAL / EALIGN / EUNSUPPORTED_M); if a launch itself fails after the
 * fork, the join is still recorded so aux is always joined back into main.
 */
int skinny_gemm_run_overlap(skinny_gemm_t h_main, skinny_gemm_t h_fa, skinny_gemm_t h_fb,
                            int chain, const void* x, int64_t M, void* out_main, void* fa,
                            void* out_fb, void* main_stream, void* aux_stream,
                            void* fork_event, void* join_event);

/*
 * Time the candidate tactics for each M in Ms[0..nM) on this GPU and install
 * the fastest in the plan; M values not listed take the tuned tactic of the
 * smallest listed M' >= M, else keep the default (low_latency_gemm page,
 * autotune_kda_qkvg: autotune before CUDA graph capture).  Each candidate is
 * timed as a CUDA graph of back-to-back launches that rotate over scratch
 * copies of the weight's layout (>= 4.5x the L2 size, so reads come from HBM),
 * i.e. in the steady state of a decode step; the fastest six are timed again
 * with every combination of a later PDL trigger (:d1-:d4) and an L2 prefetch
 * depth (:p1, :p2, :p4), tcgen05 cluster tactics at >= 64 tokens also with
 * per-thread reduction stores (:s), and, unless the handle was prepared with
 * SKG_PREPARE_DETERMINISTIC, with run-time K sharing (:w); the fastest six of
 * all are then timed with twice the launches and five repetitions to decide.  Listed M values with the same candidate list (the
 * same token tiles, e.g. M = 1..8) are tuned together and get one tactic.
 * Synchronizes `stream`;
 * allocates and frees those copies; may grow the handle's workspace; writes
 * nothing the caller owns.  Must not be called while capturing (ECAPTURING).
 * When SKINNY_GEMM_TACTIC_FILE names a file, results are appended there and
 * reused by later prepares.
 */
int skinny_gemm_autotune(skinny_gemm_t h, const int64_t* Ms, int nM, void* stream);

/*
 * Tune the two-stream step for concurrency: for each M in Ms, the candidate
 * tactics of F_A, then of the main projection, then of F_A again are each
 * timed inside the whole step (main projection rotating over scratch copies of
 * its weight, F_A -> F_B chain on a high-priority aux stream, fork/join by
 * events), as a CUDA graph of back-to-back steps; the four fastest of each
 * pass are timed again with twice the steps and five replays, and the
 * fastest of those is installed in h_fa's / h_main's plan.  A last pass times
 * the main pick with every later PDL trigger (:d1-:d4) and L2 prefetch depth
 * (:p1, :p2) inside the step and keeps the fastest of the three best timed
 * the longer way.  (A tactic that is
 * fastest alone can be slow next to a grid that fills the GPU; the main
 * projection's step-tuned plan may be slower when it runs alone.)  F_B keeps
 * its plan.  Same rules as skinny_gemm_autotune: synchronizes `stream`,
 * allocates and frees scratch, not while capturing.
 */
int skinny_gemm_autotune_overlap(skinny_gemm_t h_main, skinny_gemm_t h_fa, skinny_gemm_t h_fb,
                                 int chain, const int64_t* Ms, int nM, void* stream);

/* Force the tactic used for token count M (1..256), given as the string
 * skinny_gemm_plan_query prints:
 *   "tc:r<64|128>:t<tok>:b<boxes>:s<stages>:c<cluster>[:d<k>][:p<k>][:a][:s][:w]"  tcgen05
 *   "mma:r<64|128>:t<tok>:b<boxes>:s<stages>:c<cluster>[:d<k>][:p<k>][:w]"  mma.sync
 *   "sk:r128:t<tok>:b<boxes>:s<stages>:<g|p><n>"             stream-K kernel
 * (t = token tile, b = 64-wide K boxes per pipeline stage, c = split-K cluster
 * size, g = CTAs per SM / p = parts per row tile for stream-K; d<k> launches
 * the next kernel on the stream (PDL) only once all but k-1 of a CTA's weight
 * stages are issued; p<k> (not with :w) also brings the weight boxes of the
 * k stages after the first ones into L2 before the PDL wait, so they are
 * fetched while the previous kernel finishes; :a places a cluster's receive
 * buffer in the pipeline
 * stages, which frees shared memory for more CTAs per SM at the price of a
 * cluster barrier after the MMAs; :s (tcgen05 clusters at >= 64 tokens) sends the
 * partial sums with per-thread stores instead of one bulk copy per peer; :w, with c > 1 and not with :a, shares a
 * cluster's K boxes out at run time: after its first `s` stages, whose boxes
 * are fixed, each CTA takes the next boxes from a counter in the cluster's
 * first CTA, so the CTAs of a cluster end their K work together; the fp32
 * summation order then varies from run to run).  tcgen05 tactics with tok < M run
 * ceil(M / tok) token tiles; the other kernels need tok >= M.  EINVAL if the string does not
 * parse or the tactic does not fit this weight and M. */
int skinny_gemm_set_tactic(skinny_gemm_t h, int64_t M, const char* tactic);

/* Parse a tactic string (grammar at skinny_gemm_set_tactic) and write its
 * canonical spelling into buf (NUL-terminated, truncated to len): suffixes in
 * the order ":d<k>", ":p<k>", ":a", ":s", ":w".  No handle and no device needed.  EINVAL if it does
 * not parse. */
int skinny_gemm_tactic_normalize(const char* tactic, char* buf, size_t len);

/* Write the tactic the plan uses for M into buf (NUL-terminated, truncated to
 * len).  Returns SKG_OK, or EINVAL/EUNSUPPORTED_M. */
int skinny_gemm_plan_query(skinny_gemm_t h, int64_t M, char* buf, size_t len);

/* Write the candidate tactics valid for this weight at M into buf, separated
 * by ';'.  Returns the number of candidates (>= 0) or a negated error code. */
int skinny_gemm_list_tactics(skinny_gemm_t h, int64_t M, char* buf, size_t len);

/* Synchronize `stream`, then read and clear the handle's device status word.
 * Returns SKG_OK, SKG_ETIMEOUT if a kernel's bounded wait expired since the
 * last check, SKG_ECHECK if (in the checked build, libskinny_gemm_checked.so,
 * compiled with SKG_DEVICE_CHECKS) an access failed its bounds test and was
 * skipped (the message names the access), or ECUDA.  Not capturable. */
int skinny_gemm_check_status(skinny_gemm_t h, void* stream);

/* Debug aid for the watchdog: the next `count` launches on this handle
 * return early after waiting timeout_ns on a barrier that nothing signals,
 * setting the status word (no output is written).  count 0 clears it. */
int skinny_gemm_debug_inject_timeout(skinny_gemm_t h, int count, uint64_t timeout_ns);

/* Self-test of the checked build (libskinny_gemm_checked.so): the next `count`
 * launches on this handle record one failed device check (access code 11) in
 * the status word and return at once, without touching x or out, so that
 * skinny_gemm_check_status reports SKG_ECHECK.  count 0 clears it.  EINVAL in
 * the normal library, which has no device checks. */
int skinny_gemm_debug_inject_check(skinny_gemm_t h, int count);

/* Release the handle (its status word and staging buffers).  The caller must
 * make sure no launch using it is still pending.  NULL, an already destroyed
 * handle and a pointer that never was a handle are ignored.  Every entry point
 * refuses a destroyed or unknown handle with SKG_EINVAL (the library keeps a
 * set of live handles; an address reused by a later prepare counts as that
 * new handle). */
void skinny_gemm_destroy(skinny_gemm_t h);

/*
 * One projection with NO allocation and no handle: out[M, N] = x[M, K] @ W^T.
 * (The pages have no counterpart; this entry point is this library's own.)
 *
 * For callers that cannot allocate device memory: code that runs while a
 * stream is being captured in global mode (where cudaMalloc is refused and
 * spoils the capture), serving engines that hand all of HBM to their own
 * pool allocator up front, and code that must not risk the device-wide
 * synchronization cudaMalloc/cudaFree may imply.  skinny_gemm_prepare
 * allocates a device status word, so such callers use this function instead.
 *
 * Arguments: W [N, K] with row pitch ldw, x [M, K] with pitch ldx, out [M, N]
 * with pitch ldo, all DEVICE pointers on the current device (same alignment
 * rules as skinny_gemm_prepare_ex / skinny_gemm_run_strided); out_dtype
 * SKG_BF16 or SKG_FP32; weights and inputs bf16.  Uses the untuned default
 * tactic for (N, K, M).
 *
 * Scratch: the kernels' one piece of scratch, the 4-byte watchdog status word,
 * lives in a static 256-byte device array inside the library (held on every
 * GPU that loads the library until the process exits).  A request needing more
 * scratch than 256 bytes is rejected with SKG_EINVAL and a message.  The array
 * keeps the last call's contents; it is zeroed once, at set-up.  The word only
 * goes from zero to a code (the first expired wait wins) and is not read back
 * (use the handle API for watchdog reports), so no call needs it cleared and
 * consecutive calls on one stream still overlap under programmatic dependent
 * launch.  All calls share the array, so calls that overlap on the GPU
 * (different streams, or different host threads) race on it; serialize them
 * on one stream.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current), zeroes the array with a
 * synchronous cudaMemset and caches the address; make that first call before
 * any stream capture.  Calls no cudaMalloc, cudaFree or other allocating
 * routine.  Asynchronous: returns after the launch.
 * Errors: EINVAL, EALIGN, EUNSUPPORTED_M, EDEVICE, ECUDA.
 */
int skinny_gemm_run_noalloc(const void* W, int64_t N, int64_t K, int64_t ldw, int out_dtype,
                            const void* x, int64_t ldx, int64_t M, void* out, int64_t ldo,
                            void* stream);

/* Thread-local description of the last failure on this thread ("" if none). */
const char* skinny_gemm_last_error(void);

/* Thread-local status code of the last failing call on this thread (0 if none);
 * lets callers of the NULL-returning prepare functions read the reason. */
int skinny_gemm_last_status(void);

/* SKINNY_GEMM_ABI_VERSION of the loaded library. */
int skinny_gemm_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SKINNY_GEMM_H_ */
