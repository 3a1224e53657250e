/*
 * fa.h — C ABI of the GB300 (sm_103a) FlashAttention forward library.
 *
 * The library computes exact softmax attention
 *
 *     O = softmax(scale * Q K^T + M) V,     LSE = logsumexp(scale * Q K^T + M)
 *
 * row by row, tile by tile with online softmax, so the Sq x Sk score and
 * probability matrices never reach device memory. Sources:
 *   - "MiniPaged-Qwen: Qwen3 Prefill FlashAttention" (blog.zsmgc.love),
 *     section 1 (the operation and the causal mask M), sections 3.1 and 4
 *     (tiling and the online-softmax recurrence), section 6 (GQA head map
 *     kv_head = q_head / (Hq / Hkv)), section 13 (bottom-right causal limit
 *     causal_limit = kv_len - q_len + qi + 1);
 *   - "NVIDIA闪存注意力实操：极速提升4倍性能" (nmedialink.com), sections
 *     "在线Softmax算法" and "因果注意力与分组查询注意力";
 *   - "FlashAttention 个人实现思路" (blueriverlhr.github.io), introduction
 *     (the (batch, seq_len, n_heads, d_head) layout) and the kernel argument
 *     struct (contiguous strided tensors).
 * LSE is not defined on any page; here it is the natural-log log-sum-exp of
 * the scaled, masked scores of each query row.
 *
 * Every function is thread-safe and returns an fa_status_t code. Nothing
 * here allocates or frees caller memory.
 */
#ifndef FA_GB300_H_
#define FA_GB300_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle; the same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* fa_stream_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* a pointer, size, alignment or flag is invalid */
  FA_ERR_UNSUPPORTED = 2,  /* valid request outside what the kernel covers */
  FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  FA_ERR_TIMEOUT = 4       /* a device-side bounded wait ran out (see fa_status) */
} fa_status_t;

typedef enum { FA_DTYPE_FP16 = 0, FA_DTYPE_BF16 = 1 } fa_dtype_t;

/*
 * fa_fwd — attention forward on one GPU, enqueued on `stream`.
 *
 * q    device pointer, (B, Sq, Hq, D) contiguous, element type `dtype`
 * k, v device pointers, (B, Sk, Hkv, D) contiguous, element type `dtype`
 * o    device pointer, (B, Sq, Hq, D) contiguous, written (fully overwritten)
 * lse  device pointer, (B, Hq, Sq) contiguous float32 (natural log), or NULL
 *      to skip it. Rows that see no key get O = 0 and LSE = -inf.
 * B, Sq, Sk, Hq, Hkv, D   sizes; Hq must be a multiple of Hkv (query head h
 *      reads key/value head h / (Hq / Hkv)); D must be a multiple of 16 from
 *      16 to 256. The kernels work on D = 64, 128 or 256: a smaller D runs
 *      on the next one with the head dimension zero padded on load (no
 *      effect on the result, extra arithmetic). D > 128 runs the one-tile
 *      kernel of fa_fwd_decode with a single key range (no workspace) and
 *      needs Hq / Hkv <= 128.
 * scale  softmax scale (1/sqrt(D) in the usual case): any finite value,
 *      zero and negative ones included (the pages leave it a free
 *      argument of softmax(scale * Q K^T + M)); |scale| * log2(e) must be
 *      a finite float (|scale| < 2.36e38).
 * causal 0: every key is visible; 1: bottom-right causal mask, query i sees
 *      key j iff j <= i + Sk - Sq (top-left when Sq == Sk).
 * dtype  FA_DTYPE_FP16 or FA_DTYPE_BF16 (inputs and O share it; P is rounded
 *      to it before the P V product; accumulation is fp32).
 * stream CUDA stream of the current device (NULL = legacy default stream).
 *
 * Ownership: the caller allocates and owns every buffer; q, k and v are only
 * read. The library keeps a per-device status word and no other state.
 * Alignment: q, k, v, o must be 16-byte aligned; lse 4-byte aligned.
 * Errors: arguments are checked before anything is enqueued. Negative sizes,
 * NULL pointers, Hkv == 0 or Hq % Hkv != 0, a non-finite scale, causal not
 * in {0,1}, dtype not in {0,1} or a misaligned pointer give
 * FA_ERR_INVALID_ARG; D outside 16..256 or not a multiple of 16, a scale
 * whose |scale| * log2(e) overflows a float, or sizes whose element offsets
 * do not fit the kernel's 32-bit tile coordinates give FA_ERR_UNSUPPORTED. With
 * B, Sq or Hq equal to 0 nothing is written and FA_OK is returned. Sk == 0 is
 * valid: O = 0 and LSE = -inf. A failed launch returns FA_ERR_CUDA. The call
 * is asynchronous; a device-side timeout is reported later by fa_status().
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Sk, int Hq,
           int Hkv, int D, float scale, int causal, int dtype, fa_stream_t stream);

/*
 * fa_fwd_strided — fa_fwd on strided tensors (e.g. the (B, H, S, D) layout of
 * "NVIDIA闪存注意力实操" or views into a packed QKV buffer). Each tensor keeps
 * its logical (batch, seq, head, d) indexing; `*_strides` point to three
 * int64 element strides for (batch, seq, head), the head dimension d being
 * contiguous. Strides of dimensions of size > 1 must be positive multiples
 * of 8 elements (16 bytes) and below 2^39 elements; strides of size-1
 * dimensions are ignored. lse stays (B, Hq, Sq) contiguous. Arguments and
 * errors are otherwise those of fa_fwd; NULL stride pointers or invalid
 * strides give FA_ERR_INVALID_ARG. Overlapping o with q, k or v is undefined.
 */
int fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Sk,
                   int Hq, int Hkv, int D, const long long* q_strides, const long long* k_strides,
                   const long long* v_strides, const long long* o_strides, float scale, int causal, int dtype,
                   fa_stream_t stream);

/*
 * fa_merge — combine attention outputs computed over disjoint key sets (for
 * example key shards of a context-parallel run, each produced by fa_fwd):
 *     LSE = ln sum_r exp(LSE_r),   O = sum_r exp(LSE_r - LSE) O_r,
 * the online-softmax rescale of "MiniPaged-Qwen: Qwen3 Prefill
 * FlashAttention" section 4 applied to whole partial states.
 * o_parts   device, (n_parts, B, Sq, Hq, D) contiguous, element type `dtype`
 * lse_parts device, (n_parts, B, Hq, Sq) contiguous float32 (natural log);
 *           a part with LSE_r = -inf holds no key for that row and is skipped
 * o         device, (B, Sq, Hq, D) contiguous `dtype`, fully overwritten
 * lse       device, (B, Hq, Sq) float32, or NULL. Rows where every part is
 *           -inf get O = 0 and LSE = -inf.
 * n_parts >= 1; D a multiple of 16, at most 1024. o_parts and o 16-byte
 * aligned, lse arrays 4-byte aligned. Errors as for fa_fwd (FA_ERR_INVALID_ARG
 * for bad sizes, pointers or dtype, FA_ERR_UNSUPPORTED for D). Asynchronous on
 * `stream`; allocates nothing.
 */
int fa_merge(const void* o_parts, const float* lse_parts, int n_parts, void* o, float* lse, int B, int Sq, int Hq,
             int D, int dtype, fa_stream_t stream);

/*
 * fa_fwd_decode — attention split over the keys: decode, short chunks and
 * small prefill problems (too few (batch, head, row tile) units to fill the
 * GPU with fa_fwd). The Hq/Hkv query heads of a KV group times
 * floor(128 / (Hq/Hkv)) query positions form one row tile, so Hq/Hkv <= 128
 * is required (else FA_ERR_UNSUPPORTED). The keys are cut into `num_splits`
 * ranges of whole 128-key tiles (num_splits <= 0 picks the most splits
 * that keep all CTAs in one wave on the current device's SMs, at least one;
 * the count is clamped to the number of key tiles), each range gives a
 * normalised partial (O_s, LSE_s), and fa_merge's
 * rule combines them into O and LSE. Layouts, dtypes, mask and errors as for
 * fa_fwd (contiguous tensors).
 * workspace        device scratch of at least the size returned by
 *                  fa_decode_workspace_size for the same arguments and
 *                  current device, 16-byte aligned, owned by the caller and
 *                  used only until the call's work on `stream` completes; it
 *                  may be NULL when that size is 0 (one split). A smaller or
 *                  NULL workspace when one is needed gives FA_ERR_INVALID_ARG.
 * Two calls that share a workspace must not overlap on the device.
 */
int fa_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Sk, int Hq,
                  int Hkv, int D, float scale, int causal, int dtype, int num_splits, void* workspace,
                  unsigned long long workspace_bytes, fa_stream_t stream);

/*
 * fa_decode_workspace_size — bytes of workspace fa_fwd_decode needs for
 * these sizes and `num_splits` (written to *bytes; 0 when one split
 * suffices). Errors as for fa_fwd_decode's size checks.
 */
int fa_decode_workspace_size(int B, int Sq, int Sk, int Hq, int Hkv, int D, int num_splits,
                             unsigned long long* bytes);

/*
 * fa_decode_splits — the number of key ranges fa_fwd_decode would use for
 * these sizes and `num_splits` on a GPU with `num_sms` SMs, without touching
 * any GPU (host arithmetic only). FA_ERR_INVALID_ARG for a null `n_splits`,
 * num_sms <= 0, or sizes with nothing to split (B, Sq, Hq or Sk zero); other
 * argument errors as fa_fwd_decode.
 */
int fa_decode_splits(int B, int Sq, int Sk, int Hq, int Hkv, int D, int num_splits, int num_sms, int* n_splits);

/*
 * fa_fwd_decode_noalloc — fa_fwd_decode without a caller-provided workspace,
 * for callers that cannot allocate device memory when they call: code under
 * a memory manager that owns the whole device heap (for example a serving
 * process whose memory plan is fixed at start-up), or code that must not
 * allocate on its hot path because an allocation can block on the device or
 * fail once memory is fragmented. No page describes this call; it exists
 * for those callers only.
 * The split workspace is a fixed 16 MiB array in the library's own device
 * memory, which every GPU that loads the library holds until the process
 * exits. A call whose workspace (fa_decode_workspace_size for the same
 * arguments) exceeds 16 MiB returns FA_ERR_UNSUPPORTED; a smaller num_splits
 * or fa_fwd_decode with a workspace serves those sizes. The call allocates
 * nothing (no cudaMalloc/cudaFree). The first call on a device looks up the
 * array's device address on that device (once per device, with the device
 * current). The array sits in a device-code module of its own (the library
 * has no relocatable device code), and under CUDA's default lazy module
 * loading that first lookup is what loads the module and reserves its
 * 16 MiB. A caller whose device heap is later handed to another memory
 * manager, or who captures streams, should therefore make one call on each
 * device at start-up, before either; setting CUDA_MODULE_LOADING=EAGER
 * instead loads the module, array included, when the library loads. If that
 * first lookup fails (for example no memory left for the module) the call
 * returns FA_ERR_CUDA and the next call tries again. Every call on a
 * device shares the one array, so calls that overlap on the GPU (different
 * streams, or host threads without ordering) race on it; order them on one
 * stream. Arguments, results and errors are otherwise those of fa_fwd_decode.
 */
int fa_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Sk,
                          int Hq, int Hkv, int D, float scale, int causal, int dtype, int num_splits,
                          fa_stream_t stream);

/*
 * fa_fwd_host_workspace_size — device bytes fa_fwd_host needs for these
 * sizes: room for a device copy of Q, K, V, O and LSE (each 256-byte
 * aligned). FA_ERR_INVALID_ARG for a null `bytes` or a negative size.
 */
int fa_fwd_host_workspace_size(int B, int Sq, int Sk, int Hq, int Hkv, int D, unsigned long long* bytes);

/*
 * fa_fwd_host — fa_fwd for tensors in HOST memory. The operation, layouts
 * (contiguous (B, S, H, D) q, k, v, o; contiguous (B, Hq, Sq) fp32 lse, which
 * may be NULL), dtypes, masks and results are those of fa_fwd; only the
 * placement differs: q, k, v, o, lse are host pointers (page-locked memory
 * lets the copies run asynchronously and overlap; pageable memory works but
 * serialises them). `workspace` is a device buffer of at least
 * fa_fwd_host_workspace_size(...) bytes, 256-byte aligned, owned by the
 * caller and not read before being written.
 *
 * The call splits the problem into up to eight chunks (ranges of batches,
 * times two ranges of KV heads when eight chunks fit, when B >= 4; else up
 * to four ranges of KV heads times up to two ranges of
 * query rows; at most one chunk per 32 MiB of copies, so small problems run
 * as one) and pipelines, per chunk, the host-to-device copy of its Q and of
 * the K/V rows it newly needs (with a causal mask early rows need only the
 * first keys), the attention kernel and the device-to-host copy of its O and
 * LSE: copies run on two streams of the library (one per direction), kernels
 * alternately on `stream` and a third library stream (streams created once
 * per device), ordered by events. It returns after enqueueing; o and lse are complete
 * once `stream` has completed (the call makes `stream` wait for the last
 * copy). Overlapping calls on one device share the library's copy streams
 * and so run one after another; they must not share a workspace.
 *
 * Errors: those of fa_fwd for the arguments it shares, FA_ERR_INVALID_ARG for
 * a null, misaligned or too small workspace, FA_ERR_CUDA when a copy, event
 * or stream call fails. "NVIDIA闪存注意力实操" and the other pages describe
 * the kernel only; this call is the data movement around it.
 */
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Sk, int Hq,
                int Hkv, int D, float scale, int causal, int dtype, void* workspace,
                unsigned long long workspace_bytes, fa_stream_t stream);

/*
 * fa_fwd_host_plan — the chunks fa_fwd_host cuts these sizes into, without
 * touching any GPU (host arithmetic only). For chunk i < min(*n_chunks, cap)
 * it writes nine ints at chunks[9 i]: batches [b0, b1), KV heads [h0, h1)
 * (query heads [h0 G, h1 G), G = Hq / Hkv), query rows [r0, r1), the keys
 * [k0, k1) the chunk copies in (those its rows need that no earlier chunk of
 * the same heads copied), and lim: its kernel runs on keys [0, lim) with the
 * bottom-right mask, which for rows [r0, r1) is the mask of the whole
 * problem. *n_chunks is the chunk count (1 to 8). `chunks` is caller memory
 * of at least 9 * cap ints (may be NULL when cap is 0). FA_ERR_INVALID_ARG
 * for a null `n_chunks`, non-positive B, Sq, Hq, Hkv or D, a negative Sk, Hq
 * not a multiple of Hkv, or causal outside {0, 1}.
 */
int fa_fwd_host_plan(int B, int Sq, int Sk, int Hq, int Hkv, int D, int causal, int* chunks, int cap, int* n_chunks);

/*
 * fa_status — synchronise `stream`, then read and clear the device status
 * word of the current device: FA_OK, or FA_ERR_TIMEOUT if a kernel's bounded
 * wait on an mbarrier ran out (the kernel then released its tensor memory
 * and returned; the CUDA context stays usable). FA_ERR_CUDA if the
 * synchronisation itself failed.
 */
int fa_status(fa_stream_t stream);

/* fa_status_string — static, human-readable name of a status code. */
const char* fa_status_string(int code);

/* fa_version — library version as major * 10000 + minor * 100 + patch. */
int fa_version(void);

/*
 * fa_debug_set_fault — test hook for failure detection. With `skip_load`
 * >= 0 every later fa_fwd launch on this process drops its K/V load number
 * `skip_load` (counted per CTA), so the consumer's bounded wait runs out after
 * `timeout_ms` milliseconds (<= 0 keeps the default of 2000 ms) and the kernel
 * records FA_ERR_TIMEOUT. -1 restores normal operation. The default timeout
 * is also overridable with the environment variable FA_WAIT_TIMEOUT_MS.
 */
int fa_debug_set_fault(int skip_load, int timeout_ms);

/*
 * fa_fwd_schedule — the work decomposition fa_fwd would use for these sizes
 * (head dimension <= 128) on a GPU with `num_sms` SMs, without touching any
 * GPU: *key_split = 0 for row-tile pairs, 1 for key-split items (see
 * fa_debug_set_schedule, whose override it reports too). Host arithmetic
 * only: a static cost model of the persistent schedule, in key-tile steps.
 * FA_ERR_INVALID_ARG for a null `key_split`, non-positive sizes, Hq not a
 * multiple of Hkv or causal not 0/1.
 */
int fa_fwd_schedule(int B, int Sq, int Sk, int Hq, int Hkv, int causal, int num_sms, int* key_split);

/*
 * fa_fwd_work_items — the work items of fa_fwd's persistent kernel for these
 * sizes (head dimension <= 128) under one decomposition (key_split 0:
 * row-tile pairs, 1: key-split items), from the functions the kernel itself
 * runs, without touching any GPU. Items are numbered longest first (row
 * tiles from the last down, then batch, then head unit) and run by CTA
 * r * grid + c on even rounds r and r * grid + (grid - 1 - c) on odd ones
 * ("NVIDIA闪存注意力实操" section "ProgramId重映射": longest work first).
 * For item n < min(*n_items, cap) it writes eight ints at items[8 n]:
 *   b, hq0, hq1  batch and the query heads of its two 128-row tiles,
 *   kvh          their key/value head (hq / (Hq / Hkv), "MiniPaged-Qwen"
 *                section 6),
 *   r0, r1       first rows of the two tiles (a key-split item has one tile:
 *                hq1 = hq0, r1 = r0; a tile with r >= Sq is empty),
 *   n_kv         key tiles [0, n_kv) the item visits (the causal limit of
 *                its last row, "MiniPaged-Qwen" section 13; 0: no key),
 *   cta          the CTA that runs it.
 * *n_items is the full item count and *grid the CTA count (at most
 * num_sms). `items` is caller memory of at least 8 * cap ints (may be NULL
 * when cap is 0). FA_ERR_INVALID_ARG for null outputs, non-positive sizes,
 * Hq not a multiple of Hkv, or causal / key_split outside {0, 1}.
 */
int fa_fwd_work_items(int B, int Sq, int Sk, int Hq, int Hkv, int causal, int key_split, int num_sms, int* items,
                      int cap, int* n_items, int* grid);

/*
 * fa_debug_set_schedule — test hook that fixes the work decomposition of
 * every later fa_fwd / fa_fwd_strided call in this process (D <= 128):
 *   -1  (default) a host cost model picks per call;
 *    0  row-tile pairs: each CTA work item is two 128-row query tiles that
 *       share every K/V tile (two heads of a GQA group, or two row tiles);
 *    1  key-split: each item is one 128-row query tile whose even and odd key
 *       tiles run side by side and are combined before the store (more,
 *       shorter items: the short-sequence case of "NVIDIA闪存注意力实操"
 *       section "自动调优").
 * The result is the same attention either way, up to rounding. Returns
 * FA_ERR_INVALID_ARG for any other mode.
 */
int fa_debug_set_schedule(int mode);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H_ */
