/*
 * fa.h -- C interface of libfa, the sm_103a attention forward pass.
 *
 * The operation (sources named by page title and section):
 *   O = softmax(scale * Q K^T) V, row by row, computed as a tiled online softmax: a tile of
 *   128 query rows stays on chip while tiles of 128 keys stream past it, each row carrying a
 *   running maximum m, denominator l and unnormalised accumulator o that are rescaled by
 *   exp(m_old - m_new) when the maximum moves; o is divided by l once, at write-back.
 *   - definition of S, P, O: "11. Fusion, recompute, and flash attention", section 11.2;
 *   - the running (m, l, o) recurrence: same chapter, section 11.6 "Online softmax", and
 *     "Flash Attention 2" (linearalgebraforprogrammers.com), "Overview of the algorithm";
 *   - one tile of queries per thread block, keys streamed, division at write-back:
 *     same chapter, section 11.9 "How FlashAttention tiles on a GPU";
 *   - a masked, partial last key block: "Attention" (phobos stdlib docs), `attention`;
 *   - causal masking that stops the key loop at the tile's last query: same page,
 *     "Causal attention".
 *
 * Layout: Q and O are contiguous [B, H, Nq, D]; K and V are contiguous [B, H, Nk, D]; D is the
 * innermost (fastest) index and rows of one (b, h) slice are adjacent. All four tensors have
 * the same 16-bit element type `dtype`; accumulation is fp32 inside the kernel. O is written
 * by rounding the fp32 result to nearest (ties to even).
 *
 * Causal masking (causal = 1): query i sees key j iff j <= i, counting both from 0 within
 * their slice (top-left alignment, also when Nq != Nk). Key 0 is always visible, so no row
 * is ever empty.
 *
 * Ownership: every pointer is owned by the caller. libfa keeps no reference to them after a
 * call returns (for fa_fwd: after the launched work has finished on `stream`).
 *
 * Errors: every entry point returns a fa_status. Argument checks happen before any CUDA call;
 * a rejected call has no side effect. fa_last_error_message() gives a one-line reason for the
 * last non-FA_OK status returned on the calling host thread.
 *
 * Stream order: libfa's kernels are launched as programmatic dependents of the kernel before
 * them in the stream (their start-up overlaps its last blocks), but each waits for that kernel
 * to complete before touching global memory, and each call's results are complete for any work
 * queued after it on the stream. Stream semantics are therefore those of ordinary launches,
 * also under CUDA graph capture.
 */
#ifndef TILED_ONLINE_SOFTMAX_FA_H
#define TILED_ONLINE_SOFTMAX_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_dtype {
    FA_F16 = 0,  /* IEEE binary16 */
    FA_BF16 = 1  /* bfloat16 */
} fa_dtype;

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARGUMENT = 1, /* null pointer, size < 1, non-finite scale, causal not 0/1,
                                    overlapping output, unknown dtype */
    FA_ERR_UNSUPPORTED = 2,      /* a valid request this build has no kernel for (D not 64/128,
                                    no sm_103a device) */
    FA_ERR_MISALIGNED = 3,       /* a tensor pointer not 16-byte aligned */
    FA_ERR_CUDA = 4,             /* a CUDA runtime or driver call failed */
    FA_ERR_TIMEOUT = 5           /* a kernel's bounded wait ran out (see fa_last_device_error) */
} fa_status;

/*
 * fa_fwd -- attention forward on device memory, asynchronous on `stream`.
 *
 *   Q  device pointer, [B, H, Nq, D] of `dtype`, read only.
 *   K  device pointer, [B, H, Nk, D] of `dtype`, read only.
 *   V  device pointer, [B, H, Nk, D] of `dtype`, read only.
 *   O  device pointer, [B, H, Nq, D] of `dtype`, written; must not overlap Q, K or V.
 *   B, H, Nq, Nk >= 1; B*H*max(Nq, Nk)*D must fit the tensor-map limits (2^31 rows per slice).
 *   D      head dimension: 64 or 128 (others return FA_ERR_UNSUPPORTED).
 *   scale  finite softmax temperature multiplying Q K^T (usually 1/sqrt(D)).
 *   causal 0 = every key visible, 1 = causal mask as above.
 *   stream a cudaStream_t (NULL = the legacy default stream).
 *
 * All four pointers must be 16-byte aligned (the tensor-memory-access unit requires it).
 * FA_OK means validated and launched; the result is ready once `stream` reaches this point.
 * The first call on a device allocates one 16-byte device word for kernel error reports
 * (kept until process exit); make that first call outside any stream capture.
 *
 * Work balancing (non-causal), by splitting 256-row work units over keys and merging them as in
 * fa_fwd_splitkv (two launches), on a device with S streaming multiprocessors (read from the
 * device: 152 on a GB300):
 *   - at most S/2 units: each unit is split into floor(S / units) key ranges of at least 2 key
 *     tiles (256 keys), so that one wave covers nearly all SMs;
 *   - more than S units whose last wave fills at most half of the SMs: the units of that wave
 *     are split into 2-4 ranges.
 * Shapes with fewer than 4 key tiles (Nk <= 384), and causal launches, always run as one
 * launch; fa_fwd_plan reports what a shape gets. The split units times their ranges never exceed
 * S CTAs, so their partial states fit a fixed-size workspace. libfa keeps a pool of 4 such
 * workspaces per device (about 20 MB each on 152 SMs), allocated together by the first call that
 * splits and kept until process exit; no call allocates, grows or frees it afterwards. A call
 * uses the workspace its stream used last, else one whose previous user has finished on the GPU,
 * and records an event on `stream` after its merge: calls on different streams never share
 * partial states, with no ordering required between them. A call runs as one unsplit launch
 * instead (no workspace; rows differ only by rounding) when its stream is being captured into a
 * CUDA graph, or when all 4 workspaces are still in use by other streams' unfinished calls, or
 * while the pool cannot be allocated (out of device memory: from then on; another host thread
 * capturing a graph in global mode, which forbids allocation: until a later call succeeds).
 * fa_set_tail_split(0) turns the balancing off (always one launch).
 */
fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, int64_t B, int64_t H,
                 int64_t Nq, int64_t Nk, int64_t D, float scale, int causal, fa_dtype dtype,
                 void* stream);

/*
 * fa_fwd_lse -- fa_fwd that also writes each query row's log-sum-exp
 *   LSE[b, h, i] = log sum_j exp(scale * Q[b,h,i,:] . K[b,h,j,:])   over the visible keys j,
 * the per-row statistic a backward pass recomputes P from ("Flash Attention 2", "Write the
 * data back to HBM": L = m + log l). LSE is a device pointer to fp32 [B, H, Nq], 4-byte
 * aligned, written, not overlapping any other tensor. Everything else is as in fa_fwd.
 */
fa_status fa_fwd_lse(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t B,
                     int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale, int causal,
                     fa_dtype dtype, void* stream);

/*
 * fa_fwd_f32out -- fa_fwd_lse with O written in fp32, unrounded: O32 [B, H, Nq, D] float,
 * device pointer, 16-byte aligned, not overlapping any input (LSE optional, as in fa_fwd_lse).
 * A checking aid: it separates the kernel's arithmetic error from the rounding of O to 16 bits,
 * which alone costs up to half an ulp of |O| (0.0156 for bf16 at |O| >= 4). Always one
 * launch (no key split); the arithmetic up to the output is that of fa_fwd's single launch.
 */
fa_status fa_fwd_f32out(const void* Q, const void* K, const void* V, float* O32, float* LSE,
                        int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale,
                        int causal, fa_dtype dtype, void* stream);

/*
 * fa_fwd_plan -- how fa_fwd and fa_fwd_lse divide a shape into launches (host only, no GPU work).
 *   num_sms  the SM count to plan for; 0 = the current device's (FA_ERR_UNSUPPORTED without an
 *            sm_103 device).
 * Sizes, D and causal are checked as in fa_fwd (no pointers). The plan follows the balancing rules
 * above and the fa_set_tail_split setting; it does not model the run-time fall-backs to one launch
 * (stream capture, every workspace busy).
 */
typedef struct fa_plan {
    int64_t units;           /* 256-row work units: B * H * ceil(Nq / 256) */
    int64_t split_begin;     /* first unit split over keys (== units when none is) */
    int64_t split_units;     /* units split over keys (0: one launch) */
    int num_splits;          /* key ranges of each split unit (1 when none) */
    int tiles_per_split;     /* 128-key tiles per range (all key tiles when none) */
    int64_t ctas;            /* thread blocks of the attention launch */
    int launches;            /* 1: attention only; 2: attention, then the merge */
    size_t workspace_bytes;  /* partial state the split writes (0 when none) */
} fa_plan;
fa_status fa_fwd_plan(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal,
                      int num_sms, fa_plan* out);

/*
 * Split over keys (flash-decoding), non-causal only.
 *
 * With few query rows (decoding, short chunks against a long context) one CTA per 256 query
 * rows leaves most SMs idle. fa_fwd_splitkv also splits each slice's keys into ranges: every
 * (query block, key range) pair runs on its own CTA and leaves its partial online-softmax state
 * (m, l and the unnormalised o, fp32) in `workspace`; a second kernel merges the states of each
 * row with the state-merge rule (m = max m_s, l = sum l_s e^(m_s - m), o = sum o_s e^(m_s - m);
 * "11. Fusion, recompute, and flash attention", section 11.6, last paragraph, and exercise
 * "Flash-decoding") and writes O = o / l (and LSE when non-null).
 *
 *   num_splits  requested number of key ranges per slice; 0 picks one that covers the current
 *               device's SMs (152 when there is no sm_103 device, for a size query).
 *               The effective count is at most ceil(Nk / 128), every range holds whole tiles
 *               of 128 keys, and 1 runs fa_fwd itself (no workspace needed).
 *   workspace   caller-owned device memory, 256-byte aligned, at least
 *               fa_splitkv_workspace_bytes(B, H, Nq, Nk, D, num_splits) bytes; its contents on
 *               entry do not matter and are overwritten. Calls sharing one workspace must be
 *               ordered on the GPU.
 *   LSE         optional fp32 [B, H, Nq] log-sum-exp output (NULL: not written).
 * Other arguments as in fa_fwd. Asynchronous on `stream`; two launches.
 */
size_t fa_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D,
                                  int num_splits);
fa_status fa_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE,
                         int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale,
                         int num_splits, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Rotary position embedding ("Attention", phobos stdlib docs, "Rotary position embeddings").
 *
 * fa_rope rotates every row of X [B, H, N, D] (16-bit `dtype`) pairwise and writes Y:
 *   form 0, rotate-half: pair i of a row is (x_i, x_{i+D/2});
 *   form 1, interleaved: pair i is (x_{2i}, x_{2i+1});
 *   x0' = x0 cos - x1 sin,  x1' = x1 cos + x0 sin,
 * with cos/sin of row n's pair i from the fp32 tables cos_t, sin_t [N][D/2] (shared by every
 * batch and head: row n holds the angles of the position that row sits at). fp32 arithmetic,
 * one rounding to `dtype`. Y may equal X (in place); otherwise they must not overlap. All
 * pointers are device pointers, 16-byte aligned; D a multiple of 16 (at most 512).
 *
 * fa_fwd_rope runs attention on the rotated Q and K (tables cos_q/sin_q [Nq][D/2] for Q and
 * cos_k/sin_k [Nk][D/2] for K, 16-byte aligned) and writes O (and LSE when non-null, as in
 * fa_fwd_lse); Q and K themselves are left unchanged. K is rotated first, by the fa_rope pass,
 * into `workspace` (caller-owned device memory, 256-byte aligned, at least
 * fa_rope_workspace_bytes(B, H, Nq, Nk, D) bytes = the size of K): every query block of a slice
 * reads all of K, so rotating it once is cheaper than rotating it in each thread block. Q is
 * rotated inside the attention kernel: each 128-row tile right after its load into shared
 * memory, before its first product, by the same fp32 arithmetic as fa_rope (so the result equals
 * fa_rope on Q and K followed by fa_fwd_lse, bit for bit, whenever both run the same launches).
 * Two launches (three when the attention's work balancing splits the shape over keys).
 */
fa_status fa_rope(const void* X, void* Y, const float* cos_t, const float* sin_t, int64_t B,
                  int64_t H, int64_t N, int64_t D, int form, fa_dtype dtype, void* stream);
size_t fa_rope_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D);
fa_status fa_fwd_rope(const void* Q, const void* K, const void* V, void* O, float* LSE,
                      const float* cos_q, const float* sin_q, const float* cos_k,
                      const float* sin_k, int rope_form, int64_t B, int64_t H, int64_t Nq,
                      int64_t Nk, int64_t D, float scale, int causal, fa_dtype dtype,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd -- gradients of the forward pass, by recompute ("11. Fusion, recompute, and flash
 * attention", section 11.9 "Backward" and the exercise "Backward with recompute"): the forward
 * keeps only O and the per-row log-sum-exp; P is recomputed tile by tile from Q, K and LSE.
 * With P = exp(scale Q K^T - LSE) and D_i = sum_d dO_i O_i:
 *   dV = P^T dO,  dS = P * (dO V^T - D),  dQ = scale dS K,  dK = scale dS^T Q.
 *
 *   Q, K, V    the forward's inputs ([B,H,Nq,D], [B,H,Nk,D], [B,H,Nk,D], 16-bit `dtype`)
 *   O, LSE     the forward's outputs (fa_fwd_lse): [B,H,Nq,D] and fp32 [B,H,Nq]
 *   dO         gradient of the loss with respect to O, [B,H,Nq,D]
 *   dQ, dK, dV written, shaped like Q, K, V; they must not overlap any input or each other
 *   scale, causal, dtype as in the forward call that produced O and LSE
 *   workspace  caller-owned device memory, 256-byte aligned, at least
 *              fa_bwd_workspace_bytes(B, H, Nq) bytes (per-row D_i and base-2 LSE)
 * Device pointers, 16-byte aligned (LSE 4-byte). Three launches on `stream`: a per-row
 * preprocessing kernel, a key-block-outer kernel for dK and dV, a query-block-outer kernel
 * for dQ (no atomics: results do not depend on scheduling). Accumulation is fp32; P and dS
 * are rounded to `dtype` as MMA operands; outputs are rounded once.
 */
size_t fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t Nq);
fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, int64_t B, int64_t H, int64_t Nq,
                 int64_t Nk, int64_t D, float scale, int causal, fa_dtype dtype, void* workspace,
                 size_t workspace_bytes, void* stream);

/*
 * fa_fwd_host -- the same operation on HOST buffers, synchronous.
 *
 * Q, K, V, O are host pointers with the layout above (pinned memory gives full copy speed and
 * lets copies overlap the computation). The call copies Q, K, V to device memory owned by
 * libfa, computes, copies O back and returns when O is complete. The (batch, head) slices are
 * processed in up to 6 chunks on libfa-owned streams, ordered after the work already on
 * `stream`: one stream copies the chunks' inputs in back to back, two run each chunk's attention
 * once its inputs are there, one copies each chunk's output back once it is complete. Each
 * chunk is one attention launch (no key split). The device staging buffers grow to the
 * largest request seen and are kept until process exit (or fa_release_host_buffers); the
 * streams live until process exit. Calls from several host threads on one device run one after
 * another (a per-device lock held for the whole call, which is synchronous anyway). On an error
 * the contents of O are undefined.
 */
fa_status fa_fwd_host(const void* Q, const void* K, const void* V, void* O, int64_t B,
                      int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale, int causal,
                      fa_dtype dtype, void* stream);

/* Free the staging buffers of fa_fwd_host on the current device. */
fa_status fa_release_host_buffers(void);

/*
 * fa_fwd_noalloc -- fa_fwd for callers that must not allocate device memory.
 * (The attention pages have no counterpart to this entry point: it only changes where the
 * kernel's scratch lives.)
 *
 * Who needs it: code that runs where cudaMalloc is off limits -- inside a custom allocator or
 * memory-pool callback, in a process whose device memory was reserved up front by a framework
 * pool, or in code that must not allocate after start-up (fixed-footprint serving, real-time
 * paths). fa_fwd allocates a small device error record on its first call on each device; this
 * entry point never calls cudaMalloc, cudaFree or any allocating routine.
 *
 * Scratch: the kernel's only scratch is its error record (one int, site code of a timed-out
 * wait). Here it lives in a file-scope device array of FA_NOALLOC_SCRATCH_BYTES bytes, which
 * every GPU that loads libfa holds until process exit. A request whose scratch would exceed
 * that array is rejected with FA_ERR_UNSUPPORTED (the record does not grow with B, H, Nq, Nk or
 * D, so no valid problem reaches that limit today).
 *
 * Arguments, layouts, ownership and validation are those of fa_fwd (device pointers, async
 * on `stream`), except that the whole computation is always one launch (no key split, which
 * would need a workspace). Each call clears the record with cudaMemsetAsync on `stream` before
 * its launch. All calls share the one array and it keeps the last call's contents, so calls that
 * overlap on the GPU (different streams with no ordering between them) race on it.
 * fa_last_device_error also reads and clears this record: after a call, it returns
 * FA_ERR_TIMEOUT if one of that call's bounded waits ran out (the output is then incomplete).
 * fa_wait_selftest_noalloc makes a wait run out on purpose with this record as its target.
 *
 * The first call on each device, with that device current, looks up the array's device address
 * (cudaGetSymbolAddress) and sets the kernel's shared-memory limit; make that first call before
 * any stream capture.
 */
#define FA_NOALLOC_SCRATCH_BYTES 256
fa_status fa_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, int64_t B,
                         int64_t H, int64_t Nq, int64_t Nk, int64_t D, float scale, int causal,
                         fa_dtype dtype, void* stream);
/* fa_wait_selftest (below) aimed at fa_fwd_noalloc's static record; allocates nothing. */
fa_status fa_wait_selftest_noalloc(unsigned long long timeout_ns, void* stream);

/*
 * fa_last_device_error -- synchronise `stream`, then read and clear the current device's
 * kernel error words: the one every entry point but fa_fwd_noalloc reports into, and
 * fa_fwd_noalloc's static record. Returns FA_ERR_TIMEOUT if a kernel launched by libfa on this
 * device gave up a bounded wait since the last check (its output is then incomplete), FA_ERR_CUDA
 * if the synchronisation failed, FA_OK otherwise. `site` (may be NULL) receives the wait site
 * code. Allocates nothing.
 */
fa_status fa_last_device_error(void* stream, int* site);

/*
 * fa_wait_selftest -- check the bounded-wait machinery on the device, asynchronous on `stream`.
 * Launches one warp that waits, through the same routine every libfa kernel waits with, on a
 * barrier that nothing ever arrives on. After `timeout_ns` (0 < timeout_ns <= 1e9) the wait
 * gives up and records site code 30 in the error word, so the next fa_last_device_error on
 * `stream` returns FA_ERR_TIMEOUT with *site == 30; the CUDA context stays usable. Nothing is
 * read or written besides the error word. FA_ERR_INVALID_ARGUMENT for a timeout out of range.
 * The pages have no counterpart; it exists so that the failure path can be tested.
 */
fa_status fa_wait_selftest(unsigned long long timeout_ns, void* stream);

/*
 * Lazy (conditional) rescaling threshold, process-wide, in log2 units of the scaled scores.
 * A row keeps its reference maximum, and so skips rescaling its accumulator, while the new
 * maximum exceeds the reference by at most this much (the conditional rescaling paragraph of
 * ithelp article 10405336, "FlashAttention 保留三個狀態"). O / l is unchanged by the choice;
 * the 16-bit weights P stay <= 2^threshold. 0 rescales on every rise of the maximum. Range
 * [0, 64]; default 32. fp16 launches use min(threshold, 15), so that their weights stay below
 * the fp16 maximum; bf16 weights have fp32's exponent range and keep their relative precision
 * at any size, and O and l accumulate in fp32. Affects launches made after the call.
 */
fa_status fa_set_rescale_threshold(float log2_threshold);
float fa_get_rescale_threshold(void);

/* Turn fa_fwd's work balancing (key splits, see fa_fwd) on (1, the default) or off (0).
 * Process-wide. */
fa_status fa_set_tail_split(int enable);

/*
 * Kernel timer, a measurement aid (no counterpart in the pages). Between fa_timer_start and
 * fa_timer_stop, every kernel launch libfa makes, on any stream, is bracketed by two CUDA events
 * recorded on that stream; fa_timer_stop waits for the events and sums each launch's device
 * time by kernel kind; fa_timer_read returns the sum (milliseconds) and the launch count of one
 * kind. The events come from a pool of 8192 pairs created by the first fa_timer_start on the
 * current device (kept until process exit); launches past that are not timed and
 * fa_timer_stop returns FA_ERR_UNSUPPORTED. Use one device while the timer runs. Off, the timer
 * costs one flag test per launch.
 */
typedef enum {
    FA_KERNEL_FWD = 0,        /* the attention forward kernel (all fa_fwd* entry points) */
    FA_KERNEL_MERGE = 1,      /* merge of split-over-keys partial states */
    FA_KERNEL_ROPE = 2,       /* rotary embedding */
    FA_KERNEL_BWD_PREP = 3,   /* backward: D = rowsum(dO * O) and scaled LSE */
    FA_KERNEL_BWD_DKDV = 4,   /* backward: dK and dV */
    FA_KERNEL_BWD_DQ = 5,     /* backward: dQ */
    FA_KERNEL_KINDS = 6
} fa_kernel_kind;
fa_status fa_timer_start(void);
fa_status fa_timer_stop(void);
fa_status fa_timer_read(fa_kernel_kind kind, double* total_ms, int* launches);

/*
 * Checked build. libfa_debug.so is libfa built with FA_DEBUG_BOUNDS: every kernel checks the
 * index of each global store against the extent of the tensor it writes, and a store that would
 * leave it is skipped and recorded (site code 40-47 by kernel, and the offending element or row
 * index) instead of being made. It exports the same functions and gives the same results; the
 * release build compiles the checks away.
 *
 * fa_debug_bounds_enabled   1 in the checked build, 0 in the release build.
 * fa_debug_bounds_report    read and clear the first violation recorded since the last report
 *                           (*site 0: none). Call once the work has finished (after synchronising
 *                           the streams that ran it). The release build always reports none.
 * fa_debug_bounds_selftest  checked build only (else FA_ERR_UNSUPPORTED): two stores into `buf`
 *                           (device memory of at least 64 ints, 4-byte aligned), at indices 8 and
 *                           40, both checked against a stated bound of 32. The first is made; the
 *                           second is recorded (site 49, index 40) and skipped. Asynchronous on
 *                           `stream`. The pages have no counterpart: this tests the checks.
 */
int fa_debug_bounds_enabled(void);
fa_status fa_debug_bounds_report(int* site, long long* index);
fa_status fa_debug_bounds_selftest(int* buf, void* stream);

/* A static, human-readable name for a status code. */
const char* fa_status_string(fa_status status);

/* One line on why the last non-FA_OK status on this host thread was returned. */
const char* fa_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* TILED_ONLINE_SOFTMAX_FA_H */
