/*
 * fa.h -- C ABI of the GB300 (sm_103a) tiled online-softmax attention forward pass.
 *
 * The operation (aiml.sh "Speed up long contexts with FlashAttention", lab.py:
 * `standard_attention` defines the result, `tiled_flash_attention` the blocked
 * online-softmax method that reaches it without holding the N x N matrix):
 *
 *     for every head h of every batch b and every query row i < N
 *       s_j   = scale * <q[b,h,i,:], k[b,h,j,:]>      j in J_i
 *       J_i   = {0..i} when causal (query i sees keys j <= i), else {0..N-1}
 *       o[b,h,i,:] = sum_j softmax(s)_j * v[b,h,j,:]
 *       lse[b,h,i] = ln( sum_j exp(s_j) )             (natural-log logsumexp)
 *
 * computed tile by tile: a running row maximum, a running sum and an accumulator
 * rescaled when the maximum grows, so the score matrix never reaches device memory.
 * The logsumexp output is not on the pages; it is the plain definition above.
 *
 * All functions are plain C and take raw pointers and sizes.  Compute is asynchronous
 * on the caller's stream.  None allocates device memory, and the library links no BLAS:
 * the materialised baseline (cuBLAS GEMMs, N x N matrices in device memory) is a
 * separate library, declared in fa_baseline.h.
 *
 * CUDA graphs: fa_fwd, fa_fwd_opts, fa_fwd_splitkv and fa_fwd_splitkv_noalloc may be
 * captured into a graph on the caller's stream and replayed (the launch is planned at
 * capture time from the sizes).  Make one call per device, head dim and entry point
 * before the capture: the first call sets the kernels' shared-memory attribute and
 * probes the device, which a capture should not see.  fa_get_device_status copies
 * from the device and must not be called while capturing.
 */
#ifndef FA_SM103_H
#define FA_SM103_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,    /* null pointer, negative size, non-finite or negative scale, aliasing */
    FA_ERR_UNSUPPORTED = 2,    /* head dim not in {16, 32, 64, 128, 256}, a kernel pinned for a head dim it does not serve, or a size beyond the kernel's range */
    FA_ERR_MISALIGNED = 3,     /* a tensor base address not 16-byte aligned (lse: 4-byte) */
    FA_ERR_ARCH = 4,           /* current device is not compute capability 10.3 (sm_103) */
    FA_ERR_CUDA = 5,           /* a CUDA runtime / driver call failed; see fa_last_error() */
    FA_ERR_DEVICE_TIMEOUT = 6  /* a kernel's bounded wait ran out (reported by fa_get_device_status) */
} fa_status;

/*
 * fa_fwd -- attention forward pass.
 *
 *   q, k, v  device pointers, bf16, shape [B, H, N, d], contiguous row-major
 *            (d fastest), 16-byte aligned.  Read only.  q, k and v may alias.
 *   o        device pointer, bf16, [B, H, N, d] contiguous, 16-byte aligned.
 *            Written: o = softmax(scale q k^T + mask) v, rounded to bf16 (nearest even).
 *   lse      device pointer, fp32, [B, H, N] contiguous, or NULL to skip it.
 *   B, H, N  batch, heads, sequence length (queries = keys = N).  B*H*N == 0 is a no-op.
 *   d        head dimension, one of 16, 32, 64, 128, 256.  (256 runs a kernel with one
 *            128-row query tile per work unit: 2 x 128 score columns + 256 output
 *            columns fill the 512 tensor-memory columns of an SM.  At 32, 64 and 128
 *            the library picks that kernel or the two-tile one per call; see
 *            fa_fwd_plan.)
 *   causal   nonzero: query i attends keys j <= i (top-left aligned square mask).
 *   scale    finite, >= 0 (usually 1/sqrt(d)); applied to q.k before the softmax.
 *   stream   cudaStream_t to launch on (NULL = the legacy default stream).
 *
 * Ownership: the caller owns every buffer and keeps it alive until the stream's
 * work completes; the library keeps no pointer after returning.  o and lse must
 * not overlap q, k, v or each other.  Every argument is checked before any launch;
 * on an error nothing is launched and nothing is written.  The call itself does not
 * synchronise; a device-side wait that ran out is reported later by
 * fa_get_device_status().
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
           void* stream);

/*
 * Options for fa_fwd_opts (zero-initialise, then set what you need).
 *   wait_budget_cycles  cap, in SM clock cycles, on any single wait inside the kernel
 *                       (0 = default, about one second).  A wait that runs out ends
 *                       the kernel's work early and raises FA_ERR_DEVICE_TIMEOUT.
 *   inject_skip_kv_load test hook: when > 0, work unit 0 never issues its
 *                       (inject_skip_kv_load)-th K/V tile load, so the consumer's
 *                       bounded wait must run out (host-side fault injection; no
 *                       GPU fault is involved).  0 = off.
 *   max_ctas            cap on the persistent grid (0 = one CTA per SM).
 *   kernel              FA_KERNEL_AUTO (0): the library's choice (fa_fwd_plan);
 *                       FA_KERNEL_TWO_TILE or FA_KERNEL_ONE_TILE pins that kernel
 *                       (FA_ERR_UNSUPPORTED for a head dim it does not serve).
 *   order               FA_ORDER_AUTO (0): the library's choice; FA_ORDER_ONE_SNAKE or
 *                       FA_ORDER_GROUP_SNAKES pins how work units are handed to the
 *                       CTAs (see fa_order).  Results are identical either way.
 *   block_kv            keys per K/V tile, the pages' `block_kv` (aiml.sh "Speed up long
 *                       contexts with FlashAttention", lab.py `tiled_flash_attention`):
 *                       0 = automatic (128), 128, or 64.  64 runs the two-tile kernel
 *                       (head dims 16-128; FA_ERR_UNSUPPORTED at 256 or with the one-tile
 *                       kernel pinned) with 64-key score tiles: half the keys per online-
 *                       softmax step and per MMA pair.  Any other value: FA_ERR_INVALID_ARG.
 *                       With 64 and splits = 0 the split count is the heuristic's
 *                       (fa_splitkv_auto_splits).
 * Zero-initialise the whole struct: fields are appended as the library grows (version
 * 0.3.0 appended block_kv).
 */
typedef struct {
    int64_t wait_budget_cycles;
    int32_t inject_skip_kv_load;
    int32_t max_ctas;
    int32_t kernel;
    int32_t order;
    int32_t block_kv;
} fa_fwd_options;

/*
 * The forward kernels.  Both compute the same result with the same arithmetic; they
 * differ in the query rows of one work unit (one unit per CTA at a time, units handed
 * out in a fixed longest-first order over a persistent grid of one CTA per SM).
 */
typedef enum {
    FA_KERNEL_AUTO = 0,
    FA_KERNEL_TWO_TILE = 1,  /* 256 query rows per unit (two 128-row Q tiles sharing each
                                K/V tile); head dims 16-128 */
    FA_KERNEL_ONE_TILE = 2   /* 128 query rows per unit; head dims 32 to 256 */
} fa_kernel;

/*
 * How a persistent launch hands its work units to the CTAs.  Units are numbered in
 * groups of heads whose K and V fit in part of L2 together, longest unit first inside
 * a group.  Round k gives each CTA one unit, in a snake (CTA c takes position c on even
 * rounds, G-1-c on odd ones, G = CTAs).
 */
typedef enum {
    FA_ORDER_AUTO = 0,
    FA_ORDER_ONE_SNAKE = 1,     /* one snake over all units */
    FA_ORDER_GROUP_SNAKES = 2,  /* a snake restarted in each head group, CTA order mirrored
                                   in odd groups: balances launches whose groups end in
                                   part-filled rounds (e.g. one batch of 32 heads at 8192) */
    FA_ORDER_SHIFTED_SNAKES = 3 /* a snake restarted in each head group, each group starting
                                   at the CTAs its predecessor's part-filled last round
                                   left out: balances launches of many groups */
} fa_order;

/* fa_fwd with options; opts may be NULL (same as fa_fwd). */
int fa_fwd_opts(const void* q, const void* k, const void* v, void* o, float* lse,
                int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                void* stream, const fa_fwd_options* opts);

/*
 * Split-KV forward (the same result as fa_fwd, more parallelism for small B*H*N).
 *
 * Each work unit's key range (256 query rows on the two-tile kernel, 128 on the one-tile
 * kernel) is cut into `splits` pieces processed by
 * different CTAs; every piece writes its normalised partial output O_s and the
 * logsumexp lse_s of its scores to `workspace`, and a second kernel merges them:
 *     lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s.
 * The pages do not describe this; it follows from the definition above (the
 * logsumexp of a union of key ranges), and it is what the lse output enables.
 *
 *   splits     1..64, or 0 to let the library choose the launch (fa_fwd_plan with
 *              allow_split) among the split counts whose partial results fit the
 *              workspace given (none: unsplit); 1 runs fa_fwd and needs no workspace.
 *              An explicit count > 1 runs the two-tile kernel (the one-tile kernel at
 *              head dim 256); fa_fwd_splitkv_opts can pin either.
 *   workspace  device memory, 16-byte aligned, caller-owned, at least
 *              fa_splitkv_workspace_bytes(B, H, N, d, splits) bytes for splits > 1 (for
 *              splits = 0, size it with the count fa_fwd_plan reports to get the plan's
 *              own launch; a smaller workspace limits the choice); must not overlap any
 *              tensor.
 *              Its contents on entry do not matter; they are scratch after the call.
 * Other arguments, ownership and errors as fa_fwd.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                   int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                   int splits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_fwd_splitkv with options (opts may be NULL): opts->kernel pins the kernel, which
 * then needs an explicit splits >= 1 (FA_ERR_INVALID_ARG for splits = 0);
 * opts->order pins the unit order; the other fields as fa_fwd_opts.
 */
int fa_fwd_splitkv_opts(const void* q, const void* k, const void* v, void* o, float* lse,
                        int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                        int splits, void* workspace, size_t workspace_bytes, void* stream,
                        const fa_fwd_options* opts);

/* Workspace bytes fa_fwd_splitkv needs for these sizes and `splits` (>= 1), for either
   kernel (a one-tile item holds 128 rows, a two-tile one 256); -1 on bad arguments. */
int64_t fa_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d, int splits);

/*
 * The split heuristic's count for these sizes on the current device (1 on error): more
 * than one only when the longest query block's key range would be the critical path
 * (few, long blocks for the number of SMs, e.g. one head at N = 32768).  It is one of
 * the candidates fa_fwd_plan models; the plan may take another count or kernel, so size
 * a splits = 0 workspace with fa_fwd_plan.
 */
int fa_splitkv_auto_splits(int64_t B, int64_t H, int64_t N, int causal);

/*
 * fa_fwd_plan -- the launch the library picks for these sizes: which kernel
 * (FA_KERNEL_TWO_TILE or FA_KERNEL_ONE_TILE, written to *kernel) and how many key-range
 * pieces (*splits; 1 = unsplit).  allow_split = 0 gives fa_fwd's choice, nonzero the
 * choice of fa_fwd_splitkv / fa_fwd_splitkv_noalloc with splits = 0.  num_sms = 0 asks
 * the current device for its SM count (a CUDA call); > 0 plans for that many SMs
 * without touching CUDA.
 *
 * Head dim 16 always takes the two-tile kernel and 256 the one-tile kernel.  At 32, 64
 * and 128 (and at 256 for the one-tile kernel's splits), when there are at most four
 * 256-row units per SM, the library models the run time of each candidate -- the
 * two-tile kernel unsplit, split as fa_splitkv_auto_splits says or (with no more units
 * than SMs) 2, 3, 4, 5, 6 or 8 ways, and the one-tile kernel unsplit or (with at most
 * two 128-row units per SM) split 2-8 ways -- by replaying the kernels' static schedule (unit
 * lengths in key tiles, a one-tile step costing 1.14-1.18 two-tile steps, fixed costs
 * per unit, per split piece and for the merge, all fitted per head dim to GB300 timings)
 * and takes the shortest.  Few long units (one head at N = 8192) go to the one-tile
 * kernel, whose half-size units spread the causal triangle more evenly, split when a
 * workspace allows.  Decisions are cached per shape (the first call of a shape replays
 * the schedules: up to ~0.4 ms of host time).
 *
 * *order (may be NULL) receives the unit order the launch takes (FA_ORDER_ONE_SNAKE or
 * FA_ORDER_GROUP_SNAKES): the one whose modelled busiest CTA finishes first, on a grid of
 * min(SMs, units) CTAs.
 *
 * Returns FA_OK, FA_ERR_INVALID_ARG (negative size, null kernel or splits pointer),
 * FA_ERR_UNSUPPORTED (head dim, sizes) or, with num_sms = 0, the error of the device
 * query; an empty problem plans (FA_KERNEL_TWO_TILE, 1), or (FA_KERNEL_ONE_TILE, 1) at
 * head dim 256, with FA_ORDER_ONE_SNAKE.
 */
int fa_fwd_plan(int64_t B, int64_t H, int64_t N, int64_t d, int causal, int allow_split,
                int num_sms, int* kernel, int* splits, int* order);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv for callers that may not allocate device
 * memory.  The source pages have no counterpart; this is a deployment convenience.
 *
 * Some callers cannot call cudaMalloc (or any allocator) while they run: plug-ins
 * whose host framework owns every device buffer, and latency-critical loops that
 * forbid allocator calls after start-up.  This entry point takes the same inputs and
 * outputs as fa_fwd_splitkv but no workspace: the partial results live in a fixed
 * 64 MiB array inside the library (fa_noalloc_scratch_bytes()), which every GPU that
 * loads the library holds until the process exits.
 *
 *   splits  as fa_fwd_splitkv (0 = automatic); when the split count needs more than
 *           the built-in scratch, the call returns FA_ERR_UNSUPPORTED with a message
 *           naming the limit, and launches nothing.
 *
 * The first call on a device (that needs more than one split) looks up the device
 * address of the scratch array, once per device; make that first call before any
 * stream capture.  The call allocates nothing.  All calls share the one array and it
 * keeps the last call's contents; nothing in it needs to start at zero (every value
 * the merge reads is written earlier in the same call).  Calls whose work overlaps on
 * the GPU (for example on two streams at once) race on the array: serialise them.
 */
int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int64_t B, int64_t H, int64_t N, int64_t d, int causal, float scale,
                           int splits, void* stream);

/* Size in bytes of the built-in scratch used by fa_fwd_splitkv_noalloc. */
int64_t fa_noalloc_scratch_bytes(void);

/* Static description of a status code. Never NULL. */
const char* fa_strerror(int status);

/* Detail of the last error on this host thread ("" if the last call succeeded). */
const char* fa_last_error(void);

/*
 * Synchronise `stream`, then read and clear the current device's status word.
 * Returns FA_OK, FA_ERR_DEVICE_TIMEOUT if a kernel on this device gave up a wait
 * since the last call, or FA_ERR_CUDA if the synchronisation itself failed.
 */
int fa_get_device_status(void* stream);

/* Library version, as major*10000 + minor*100 + patch. */
int fa_version(void);

/*
 * fa_row_kernel_register_check -- the check every first launch of the two-tile kernel
 * (fa_fwd_row_kernel, head dims 16-128) makes on its compiled register allocation, as a
 * pure function (no CUDA call).  That kernel moves registers between its warpgroups with
 * setmaxnreg: the softmax warpgroups raise their share while the epilogue and control
 * warpgroups lower theirs, and the shares add up to exactly 512 threads x 128 registers.
 * setmaxnreg waits, without any bound, until the block's pool can satisfy it, so a build
 * compiled to another allocation (a different compiler release, -G, -maxrregcount) would
 * hang the GPU.  The library therefore launches that kernel only when
 * cudaFuncGetAttributes reports num_regs == 128 and max_threads_per_block >= 512.
 * Returns FA_OK, or FA_ERR_UNSUPPORTED with the reason in fa_last_error().
 */
int fa_row_kernel_register_check(int num_regs, int max_threads_per_block);

/*
 * Test hook: while num_regs > 0, every launch of the two-tile kernel runs the check above
 * with num_regs in place of the compiled count (and is refused when that fails, before
 * anything is launched); 0 restores normal operation.  Process-wide; for tests only.
 */
void fa_test_override_kernel_registers(int num_regs);

#ifdef __cplusplus
}
#endif

#endif /* FA_SM103_H */
