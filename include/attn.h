/*
 * attn.h — C ABI of the exact attention-forward library (libattn.so, sm_103a).
 *
 * Operation. Exact scaled-dot-product attention forward, the standard attention of
 * the "Flash Attention optimization" skill page (hermes-agent, mlops-flash-attention),
 * workflow 1 step 2: out = softmax(q kᵀ · scale) · v, with the options of workflow 2
 * steps 2-3: layout [batch, seq, heads, dim], causal masking, fewer K/V heads than
 * query heads (MQA/GQA), and a left sliding window. It is computed the IO-aware way
 * described in "What is memory-efficient attention for long context on 8x H100?"
 * (aivaro.ru, answers 650), section 2: Q/K/V are processed in blocks held on chip
 * with an online softmax, so the L x L score matrix never reaches HBM and the extra
 * memory is O(L·d) (inputs, outputs and a workspace: a fixed 256 bytes for fp16
 * inputs, a copy of V for bfloat16 inputs).
 *
 * For batch b, query head h, row i, with g = h / (Hq / Hkv) and the visible keys
 *   J_i = { j < L : (causal => j <= i) and (window_left >= 0 => j >= i - window_left) }:
 *   O[b, i, h, :] = sum_{j in J_i} softmax_j(scale · q[b,i,h,:]·k[b,j,g,:]) · v[b, j, g, :]
 *   LSE[b, h, i]  = ln sum_{j in J_i} exp(scale · q[b,i,h,:]·k[b,j,g,:])
 *
 * Layouts (all contiguous, row-major, element strides implied by the sizes):
 *   q, o : [B, L, Hq, d]      k, v : [B, L, Hkv, d]      lse : [B, Hq, L] float32
 *
 * Ownership. The caller owns every buffer. The library never allocates device
 * memory; it keeps only host-side caches (device properties, driver entry point).
 * All pointers passed to attn_fwd are DEVICE pointers of the current CUDA device.
 *
 * Asynchrony. attn_fwd enqueues one kernel on `stream` (a cudaStream_t; NULL = the
 * legacy default stream; with bfloat16 inputs and the full workspace, first a memset
 * and two kernels that write the fp16 copy of V) and returns without synchronising. Argument errors are
 * returned before anything is enqueued. Errors detected on the device (a bounded
 * wait that ran out) are recorded in the workspace status word and reported by
 * attn_fwd_sync_status.
 *
 * Launch order. Every call launches its attention kernels as programmatic
 * dependents (programmatic stream serialization): a kernel may begin
 * its prologue (barrier setup, tensor-map prefetch) while the previous kernel on the
 * stream finishes, and waits for that kernel's completion and memory
 * (griddepcontrol.wait) before it allocates tensor memory or touches global memory.
 * Stream order is kept for every buffer. The kernels of attn_fwd_kv on a dense cache,
 * and attn_fwd's kernel when it deals its units statically (small problems), also
 * ask for their first tiles in L2 before that wait: a prefetch hint, so what they
 * compute with is still the memory as the earlier kernels left it. Once a kernel has
 * issued its last loads it lets the next kernel on the stream start its prologue
 * (except when a merge kernel of the same call follows).
 *
 * Graphs. Every entry point may be captured into a CUDA graph (stream capture): the
 * capture records the kernels with the call's pointers and sizes, so a replay
 * recomputes the result from whatever the same buffers hold, without the host-side
 * preparation of a call (checks, tensor-map encoding). Make one call of the entry
 * point on the device before the capture starts (one-time function setup).
 *
 * Threading. Calls are thread-safe; concurrent calls must use distinct workspaces.
 */
#ifndef EXACT_ATTN_H
#define EXACT_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_ABI_VERSION 5

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* a size, pointer, alignment or option is invalid          */
    ATTN_ERR_UNSUPPORTED = 2, /* valid request this build does not implement (d, arch ...) */
    ATTN_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or smaller than required        */
    ATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (detail string kept)     */
    ATTN_ERR_TIMEOUT = 5      /* a device-side bounded wait ran out; the kernel stopped     */
} attn_status_t;

typedef enum {
    ATTN_FP16 = 0, /* IEEE binary16 inputs (and outputs with ATTN_OUT_SAME) */
    ATTN_BF16 = 1  /* bfloat16 inputs (and outputs with ATTN_OUT_SAME)      */
} attn_dtype_t;

typedef enum {
    ATTN_OUT_SAME = 0, /* O in the input dtype, rounded to nearest even */
    ATTN_OUT_FP32 = 1  /* O in float32 (no final rounding to 16 bits)   */
} attn_out_t;

/*
 * Bytes of device workspace attn_fwd needs for this problem. fp16: 256 (a status
 * word and, from byte 64, the persistent kernel's unit counter, cleared by each call
 * that uses it). bfloat16: 256 + (4·B·Hkv rounded up to 256) + 2·B·L·Hkv·d, the status word,
 * then per (batch, K/V head) the largest finite |v| and an fp16 copy of V scaled by
 * a power of two per (batch, K/V head), so that the attention weights enter the P·V
 * product as fp16 (11 significant bits) in one product per key block; the scale is
 * undone on the output. Every bfloat16 value of V whose scaled magnitude is at least
 * 2^-17 is copied exactly (the largest scaled |v| is in [2^14, 2^15)); smaller ones,
 * below 2^-31 of their head's largest |v|, round to the nearest multiple of 2^-24.
 * attn_fwd also accepts a bfloat16 call with a workspace of at least 256 bytes but
 * less than this: it then splits the weights into two bfloat16 parts (hi + lo) and
 * runs two P·V products per key block instead, with the same accuracy bound and
 * about 1.4x the time at d = 128 (this is what attn_fwd_noalloc runs).
 * Returns 0 for sizes or a dtype attn_fwd would reject.
 */
size_t attn_fwd_workspace_size(int B, int L, int Hq, int Hkv, int d, int causal,
                               int window_left, attn_dtype_t dtype);

/*
 * Attention forward (see the header comment for the definition).
 *   q, k, v     device pointers, 16-byte aligned, layouts above, dtype `dtype`
 *   o           device pointer, 16-byte aligned, [B, L, Hq, d] of `dtype` or float32
 *   lse         device pointer to [B, Hq, L] float32, 4-byte aligned, or NULL to skip
 *   B, L        batch and sequence length, both >= 1; B*Hq*L < 2^31
 *   Hq, Hkv     query / key-value heads, Hkv >= 1, Hq % Hkv == 0
 *   d           head dimension: 64 or 128
 *   causal      0 or 1 (causal: key j visible from query i only when j <= i)
 *   window_left -1 for none, or w >= 0 (keys i-w .. i); requires causal = 1
 *   scale       finite multiplier of q·k (1/sqrt(d) is the usual choice)
 *   workspace   device pointer, 16-byte aligned, >= attn_fwd_workspace_size bytes
 *               (bfloat16: >= 256 bytes, see attn_fwd_workspace_size); must not be used
 *               by another call that is still running
 *   stream      cudaStream_t to enqueue on
 * Returns ATTN_OK when the kernel was enqueued; otherwise nothing was enqueued and
 * the outputs are untouched. Requires a device of compute capability 10.3.
 */
attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                       int B, int L, int Hq, int Hkv, int d, int causal, int window_left,
                       float scale, attn_dtype_t dtype, attn_out_t out_dtype,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * Attention forward on float8 e4m3 inputs: the FP8 path of the "Flash Attention
 * optimization" skill page (workflow 3: q, k, v cast to float8_e4m3fn, no scale
 * factors) and of "What is memory-efficient attention for long context on 8x
 * H100?" section 2. Same definition, masks, layouts and LSE as attn_fwd, with
 *   q, k, v   device, [B, L, H, 64] bytes of float8 e4m3 (1 sign, 4 exponent bits,
 *             bias 7, 3 fraction bits), 16-byte aligned; d must be 64
 *   o         [B, L, Hq, 64] bfloat16 (ATTN_OUT_SAME) or float32 (ATTN_OUT_FP32)
 *   workspace >= attn_fwd_fp8_workspace_size(...) bytes: the status word and a
 *             transposed copy of v ([B, Hkv, 64, L rounded up to 16])
 * The attention weights enter the P·V product as e4m3 values (3 fraction bits), so
 * the result differs from the exact one by up to about 2^-3 of the weighted mean of
 * |v| per element, and the LSE by up to ln(1/(1 - 2^-4)); see the tests for the
 * bound. Enqueues a transpose kernel and the attention kernel on `stream`.
 */
size_t attn_fwd_fp8_workspace_size(int B, int L, int Hq, int Hkv, int d, int causal,
                                   int window_left);
attn_status_t attn_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int L, int Hq, int Hkv, int d, int causal, int window_left,
                           float scale, attn_out_t out_dtype, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * Backward pass: the gradients dq, dk, dv of the square problem (attn_fwd's
 * definition, causal and left-window masks, GQA) for an upstream gradient dout of O:
 *   P = softmax rows of scale·q kᵀ on the visible keys, D_i = Σ_c dout_ic o_ic,
 *   dV = Pᵀ dout, dS = P ∘ (dout vᵀ − D), dQ = scale · dS k, dK = scale · dSᵀ q,
 * with dk and dv summed over the query heads that share a K/V head. The spec page
 * ("compare Hyena vs FlashAttention at 128k", stage 5) lists the backward pass as
 * not measured. Inputs: q, k, v, dtype and sizes as for attn_fwd; o [B, L, Hq, d]
 * and lse [B, Hq, L] are attn_fwd's outputs for these inputs (o in the input dtype);
 * dout [B, L, Hq, d] in the input dtype. Outputs dq [B, L, Hq, d], dk, dv [B, L,
 * Hkv, d] in the input dtype (ATTN_OUT_SAME) or float32. workspace >=
 * attn_bwd_workspace_size(...) bytes (the status word and per-row D and LSE). At
 * most 128 query heads per K/V head. Enqueues three kernels on `stream`; nothing of
 * size L x L is stored.
 */
size_t attn_bwd_workspace_size(int B, int L, int Hq, int Hkv, int d, int causal,
                               int window_left);
attn_status_t attn_bwd(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                       int L, int Hq, int Hkv, int d, int causal, int window_left, float scale,
                       attn_dtype_t dtype, attn_out_t out_dtype, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * attn_fwd with a window on both sides, the window_size = (left, right) option of
 * the "Flash Attention optimization" skill page (workflow 2 step 3; its symmetric
 * example is (256, 256)). Row i sees keys
 *   J_i = { j < L : (window_left >= 0 => j >= i - window_left) and
 *                   (window_right >= 0 => j <= i + window_right) },
 * each bound -1 for none: (-1, 0) is causal attention, (-1, -1) full attention.
 * Other arguments, layouts and errors as for attn_fwd; the workspace is at least 256
 * bytes (the status word; bfloat16 inputs run the split-weight path, without a copy
 * of V); at most 128 query heads per K/V head. It runs on the one-tile kernel
 * (ATTN_PATH_TILES below): a band of a few hundred keys per row is little work per
 * query tile, which that kernel spreads over one CTA per 128-row tile.
 */
attn_status_t attn_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int L, int Hq, int Hkv, int d, int window_left,
                              int window_right, float scale, attn_dtype_t dtype,
                              attn_out_t out_dtype, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * attn_fwd without a caller-provided workspace, for callers that cannot allocate
 * device memory: code running where cudaMalloc is forbidden or unsafe (inside an
 * allocator or memory-pool callback, under another framework's allocator that owns
 * all device memory, or on a path that must never enter the allocator). The pages
 * have no counterpart; this is an interface addition of this library.
 *
 * The call allocates nothing. Its scratch (the kernel's 16-byte status word) lives
 * in a fixed 256-byte device array inside the library that every GPU loading the
 * library keeps until the process exits. Arguments and results are those of
 * attn_fwd. Rules:
 *   - Problems needing more scratch than 256 bytes return ATTN_ERR_WORKSPACE (none
 *     do: bfloat16 inputs run the split-weight path of attn_fwd, which makes no copy
 *     of V; see attn_fwd_workspace_size).
 *   - All calls on a device share the array, and each call clears its status word
 *     (after its arguments are validated: a rejected call enqueues nothing): calls
 *     that overlap on the GPU (other streams, other threads) race.
 *   - The first call on a device looks up the array's address (and may load the
 *     library's device code); make it before any stream capture starts. A device
 *     reset (cudaDeviceReset) invalidates that address: the first call in the new
 *     context looks it up again, and the same rule applies to it.
 *   - On a device other than compute capability 10.3 the call returns
 *     ATTN_ERR_UNSUPPORTED, as attn_fwd does.
 *   - A device-side timeout is recorded only in that shared word, which no entry
 *     point reads; use attn_fwd with a workspace when that report is needed.
 */
attn_status_t attn_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                               int B, int L, int Hq, int Hkv, int d, int causal,
                               int window_left, float scale, attn_dtype_t dtype,
                               attn_out_t out_dtype, void *stream);

/*
 * Decode-shaped forward: Lq query rows that are the LAST Lq positions of an
 * Lk-long sequence whose keys and values are all given, as in a generation step
 * that reads the whole KV cache ("What is memory-efficient attention for long
 * context on 8x H100?", section 1, key limitations: each step reads O(n) cached
 * data, so the step is bound by HBM bandwidth). Query row i sits at position
 * p_i = Lk - Lq + i, and its visible keys are
 *   J_i = { j < Lk : (causal => j <= p_i) and (window_left >= 0 => j >= p_i - window_left) },
 * with O and LSE defined over J_i exactly as for attn_fwd (Lq = Lk gives attn_fwd's
 * result). The keys of each row tile may be cut into `num_splits` consecutive
 * ranges that run in parallel; their partial results are combined by their
 * log-sum-exp (LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s; the same
 * page, section 4, computes attention in parts this way), which gives the same O
 * and LSE up to rounding.
 *
 * Layouts: q, o : [B, Lq, Hq, d]   k, v : [B, Lk, Hkv, d]   lse : [B, Hq, Lq] float32.
 * Arguments as for attn_fwd, plus
 *   Lq, Lk      1 <= Lq <= Lk; B*Hq*Lq < 2^31 and B*Hkv*Lk < 2^31
 *   Hq / Hkv    at most 128 (the query heads of one K/V head share a 128-row tile)
 *   num_splits  0 = the library's choice (attn_fwd_kv_num_splits), else 1..256
 *   workspace   >= attn_fwd_kv_workspace_size(..., num_splits) bytes: a status word
 *               and, when splits > 1, the float32 partial results and an 8-byte
 *               merge ticket per work item. The tickets need no initialisation:
 *               each call tags them with a value of its own (a fresh workspace is
 *               fine, and so is one used before by any call of this library). A
 *               ticket found carrying another call's tag at the merge (two calls
 *               running at once on one workspace) is recorded in the status word as
 *               ATTN_ERR_WORKSPACE.
 * Enqueues one kernel on `stream` when a work item has at most 8 query rows
 * (Lq * Hq / Hkv <= 8, a decode step): with splits > 1 the last CTA of each work
 * item to finish combines the splits' partial results itself. Larger items add a
 * merge kernel when splits > 1.
 *
 * attn_fwd_kv_num_splits returns the split count attn_fwd_kv uses for num_splits
 * = 0 on the current device (0 for rejected sizes or no device);
 * attn_fwd_kv_workspace_size returns the workspace bytes of attn_fwd_kv for a split
 * count (0 = the library's choice), or 0 for rejected sizes.
 */
int attn_fwd_kv_num_splits(int B, int Lq, int Lk, int Hq, int Hkv, int d, int causal,
                           int window_left);
size_t attn_fwd_kv_workspace_size(int B, int Lq, int Lk, int Hq, int Hkv, int d, int causal,
                                  int window_left, int num_splits);
attn_status_t attn_fwd_kv(const void *q, const void *k, const void *v, void *o, float *lse,
                          int B, int Lq, int Lk, int Hq, int Hkv, int d, int causal,
                          int window_left, float scale, attn_dtype_t dtype,
                          attn_out_t out_dtype, int num_splits, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * Synchronises `stream`, reads the workspace status word written by earlier
 * attn_fwd calls on it, clears it, and returns it (ATTN_OK when no device-side
 * error was recorded). A CUDA error while synchronising returns ATTN_ERR_CUDA.
 */
attn_status_t attn_fwd_sync_status(void *workspace, void *stream);

/*
 * attn_fwd_kv over a paged K/V cache ("What is memory-efficient attention for long
 * context on 8x H100?", section 3: the cache is cut into fixed-size blocks of
 * tokens stored anywhere in memory, and a page table maps each sequence's logical
 * blocks to physical pages). Sequence b has seq_lens[b] keys; its key t is row
 * t % page_size of page block_table[b * max_pages_per_seq + t / page_size] of the
 * caches, and its Lq queries are its last Lq positions (as in attn_fwd_kv, with
 * Lk = seq_lens[b]).
 *   k_cache, v_cache  device, [num_pages, page_size, Hkv, d] of `dtype`, 16-byte aligned
 *   block_table       device int32 [B, max_pages_per_seq]; entries past a sequence's
 *                     last page are never read, entries outside [0, num_pages) read
 *                     as pages of zeros
 *   seq_lens          device int32 [B], each in [Lq, max_seq_len]; a length outside
 *                     that range records ATTN_ERR_INVALID_ARG in the workspace status
 *                     word and leaves that sequence's outputs unspecified
 *   page_size         8, 16, 32, 64 or 128; num_pages * page_size < 2^31
 *   max_pages_per_seq >= ceil(max_seq_len / page_size)
 *   max_seq_len       host-side bound of seq_lens; sizes the grid and the workspace:
 *                     use attn_fwd_kv_workspace_size / attn_fwd_kv_num_splits with
 *                     Lk = max_seq_len
 * Other arguments and the result as for attn_fwd_kv.
 */
attn_status_t attn_fwd_kv_paged(const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *block_table, const int32_t *seq_lens, void *o,
                                float *lse, int B, int Lq, int Hq, int Hkv, int d, int page_size,
                                int num_pages, int max_pages_per_seq, int max_seq_len,
                                int causal, int window_left, float scale, attn_dtype_t dtype,
                                attn_out_t out_dtype, int num_splits, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * Which kernel attn_fwd (and attn_fwd_noalloc) uses, process-wide. All compute the
 * same result (up to rounding order); they differ in how the work is cut:
 *   ATTN_PATH_AUTO       fp16, d = 64, no window, L >= 512: the alternating mode below
 *                        when its units (B * Hq * ceil(L / 128)) number at most 8 per
 *                        SM (causal) or one per SM (non-causal). Otherwise the
 *                        persistent two-tile kernel (256 query rows per work unit),
 *                        unless the problem has at most half as many such units as the
 *                        device has SMs (causal: at most as many); then the one-tile
 *                        kernel (128 rows per CTA, the longest tiles first). bfloat16
 *                        inputs with a workspace too small for the copy of V (see
 *                        attn_fwd_workspace_size) also take the one-tile kernel under a
 *                        left window whose K/V rows (B * Hkv * (window_left + 128))
 *                        take at most 192 MiB.
 *   ATTN_PATH_SQUARE     always the persistent two-tile kernel.
 *   ATTN_PATH_TILES      always the one-tile kernel (attn_fwd_kv's with Lq = Lk and one
 *                        key split).
 *   ATTN_PATH_ALTERNATE  the persistent kernel with one 128-row tile per work unit,
 *                        its two pipelines taking alternate key blocks of that tile
 *                        (each with its own running max, sum and O, combined at the
 *                        end): the longest tile's chain of blocks is half as long.
 *                        fp16 inputs with d = 64; other calls fall back to AUTO.
 * Any other value selects ATTN_PATH_AUTO. attn_get_path_policy returns the setting.
 */
enum { ATTN_PATH_AUTO = 0, ATTN_PATH_SQUARE = 1, ATTN_PATH_TILES = 2, ATTN_PATH_ALTERNATE = 3 };
void attn_set_path_policy(int policy);
int attn_get_path_policy(void);

/*
 * Sets the limit, in nanoseconds, of every device-side wait in kernels launched
 * afterwards by this process (default 4e9 = 4 s; 0 restores the default). A wait
 * that runs out records ATTN_ERR_TIMEOUT in the workspace and makes every role of
 * the kernel stop, let the copies and MMAs it already issued complete (these drain
 * waits run for at least 1 s whatever the limit), free its tensor memory and exit.
 * Limits below 1 ms make every wait poll without sleeping in hardware, so that a
 * wait runs out as soon as it has lasted longer than the limit: a limit of a few
 * nanoseconds makes a kernel time out at its first wait that has to wait at all
 * (used by the tests of the timeout path; no fault is involved).
 */
void attn_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Launches a one-warp kernel that waits, with the same bounded wait the attention
 * kernel uses, on a barrier that nothing completes, for `limit_ns` nanoseconds, and
 * records ATTN_ERR_TIMEOUT in `workspace`. It exists so the timeout path can be
 * tested without stalling the real kernel. Same argument rules as attn_fwd.
 */
attn_status_t attn_debug_wait_probe(void *workspace, size_t workspace_bytes,
                                    uint64_t limit_ns, void *stream);

/*
 * Evaluates 2^x[i] for i < n with the exp2 paths of the attention kernels: the
 * fp32 MUFU instruction (y_mufu) and, when y_f16 is not NULL, the packed fp16 MUFU
 * instruction on arguments rounded to fp16 (y_f16, widened back to float). Device
 * float32 arrays; used by the accuracy tests.
 */
attn_status_t attn_debug_exp2(const float *x, float *y_mufu, float *y_f16, int n, void *stream);

/*
 * The power-of-two exponent e of the fp16 copy of a bfloat16 V (see
 * attn_fwd_workspace_size) for a head whose largest finite |v| has the bfloat16 bit
 * pattern `absmax_bits` (sign clear): the kernels scale that head's V by 2^e and its
 * output by 2^-e. Host arithmetic only (the device runs the same function); used by
 * the tests.
 */
int attn_debug_v16_exponent(uint32_t absmax_bits);

/* Static description of a status code. */
const char *attn_status_string(attn_status_t s);

/* Detail of the last non-OK status returned to the calling thread ("" if none). */
const char *attn_last_error_detail(void);

/* ATTN_ABI_VERSION of the loaded library. */
int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTN_H */
