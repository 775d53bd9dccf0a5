/*
 * attn.h — C ABI of the GB300 (sm_103a) fused attention library
 * (libattn_gb300.so).
 *
 * Operation.  Scaled-dot-product attention per (sequence, head):
 *     S = s * Q K^T,  P = softmax(S) row by row,  O = P V,
 * and its backward for the scalar loss whose gradient with respect to O is dO:
 *     dV = P^T dO,  dP = dO V^T,  dS = P ⊙ (dP - D),  D_i = sum_k dO_ik O_ik,
 *     dQ = s * dS K,  dK = s * dS^T Q.
 * Defined in "ops(8)：self-attention 的 CUDA 实现及优化 (下) - 深度分析",
 * §2.1 (forward, and the five backward steps with the softmax derivative) and
 * Appendix A; D is the row sum of dP ⊙ P that the softmax backward subtracts
 * (§2.1 step 3), computed from dO and O because the two are equal.  The
 * forward also returns the softmax statistic the backward needs (§1.3 of the
 * same page: "stats", only in training mode); here that is the natural-log
 * log-sum-exp of the scaled scores, LSE_i = ln sum_j exp(S_ij).
 * Causal masking: key j is visible to query i iff j <= i + (Tk - Tq): with
 * Tq == Tk that is the §2.2 CPU loop's t2 <= t; with fewer queries than keys
 * (separate query and key lengths, as the cuDNN graph of "ops(8)..." §1.3
 * allows) the queries are the last Tq positions of the key sequence
 * (bottom-right alignment).  Causal (or windowed) attention with more queries
 * than keys is not supported: Tq > Tk at fixed length, or a sequence with
 * Lq > Lk in a variable-length batch with separate offsets (attn_fwd_ex).
 *
 * Precision.  Inputs and outputs are bf16; products accumulate in fp32; the
 * softmax runs in fp32; P and dS are rounded to bf16 before they enter the
 * tensor-core products; dQ is accumulated across key tiles in fp32.
 *
 * Memory.  Every pointer is a DEVICE pointer except the offset tables
 * `cu_seqlens`, `cu_seqlens_q`, `cu_seqlens_k` (host) and the tensors of
 * attn_step_host (host).
 * The library allocates no device memory: the caller owns all buffers,
 * including the backward workspace, sized with attn_bwd_workspace_size().
 * Every tensor pointer must be 16-byte aligned.
 *
 * Layouts (`layout` argument):
 *   ATTN_LAYOUT_BTHD (0): q (B,Tq,H,dqk), k (B,Tk,H,dqk), v (B,Tk,H,dv),
 *       o and dO (B,Tq,H,dv); dq, dk, dv like q, k, v.
 *   ATTN_LAYOUT_PACKED_QKV (1): q, k, v point at slots 0, 1, 2 of one
 *       (B,T,3,H,d) buffer (k = q + H*d, v = q + 2*H*d elements), the format
 *       of "ops(8)..." §1.3 (QKV as (B, T, 3, NH, HS), no permute); o and dO
 *       are (B,T,H,d); dq, dk, dv likewise point at slots of a packed
 *       (B,T,3,H,d) gradient buffer.  Needs dqk == dv and Tq == Tk.
 *   Variable length: when `cu_seqlens` is non-NULL, B is the number of
 *       sequences, Tq == Tk is the TOTAL number of token rows, tensors are
 *       (Tq, H, d) (or (Tq, 3, H, d) packed), sequence b occupies rows
 *       cu_seqlens[b] .. cu_seqlens[b+1]-1 (int32, host memory, B+1 entries,
 *       cu_seqlens[0] == 0, nondecreasing, cu_seqlens[B] == Tq), and LSE is
 *       (H, Tq).  At most ATTN_MAX_VARLEN_SEQS sequences.  attn_fwd_ex /
 *       attn_bwd_ex also take separate key offsets (keys (Tk, H, d), Tk the
 *       total key count).
 *   Fixed length: LSE is (B, H, Tq) fp32.
 *
 * Supported head sizes: (dqk, dv) in {(64, 64), (128, 128), (192, 128)}.
 *
 * Errors.  Functions return ATTN_OK (0) or a negative ATTN_ERR_* code.
 * Argument errors are detected on the host before anything is launched.
 * Launches are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 * default stream); a device-side failure (a bounded wait inside a kernel that
 * gave up) is reported later through attn_fwd_status() / attn_bwd_status().
 *
 * Threading.  Calls on different streams with different workspaces may run
 * concurrently.  Calls that share a workspace must be ordered on the GPU.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_OK 0
#define ATTN_ERR_INVALID_ARG (-1)         /* NULL / misaligned pointer, bad size */
#define ATTN_ERR_UNSUPPORTED (-2)         /* head sizes, causal with Tq > Tk, ... */
#define ATTN_ERR_WORKSPACE_TOO_SMALL (-3) /* workspace_bytes below the query */
#define ATTN_ERR_CUDA (-4)                /* a CUDA runtime call or launch failed */
#define ATTN_ERR_TIMEOUT (-5)             /* a kernel's bounded wait gave up */
#define ATTN_ERR_INTERNAL (-6)            /* a kernel found its launch set-up unusable */
#define ATTN_ERR_SCRATCH_TOO_SMALL (-7)   /* attn_bwd_noalloc: problem exceeds its scratch */

#define ATTN_LAYOUT_BTHD 0
#define ATTN_LAYOUT_PACKED_QKV 1
#define ATTN_MAX_VARLEN_SEQS 1024
#define ATTN_BLOCK 128 /* rows per block of a block-sparse mask (the kernels' tile) */

/*
 * Forward: O and (unless lse == NULL, inference mode) LSE.
 * q, k, v: inputs (bf16); o: output (bf16); lse: output (fp32) or NULL.
 * B, H, Tq, Tk, dqk, dv: sizes (see Layouts); causal: 0/1; scale: the s in
 * S = s Q K^T, finite and > 0 (the pages use 1/sqrt(dqk)); cu_seqlens: NULL or
 * host offsets.
 * "ops(8)..." §1.2-1.3 (sdpa returns [O, stats]; stats only when training),
 * §2.1 forward formulas.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int Tq, int Tk, int dqk, int dv, int causal, float scale, const int* cu_seqlens,
             int layout, void* stream);

/*
 * Local (sliding-window) attention: as attn_fwd, with key j visible to query i
 * iff  i + (Tk - Tq) - window_left <= j <= i + (Tk - Tq) + window_right
 * (each bound >= 0, or -1 for no bound on that side; variable-length batches
 * use Tk - Tq = 0 within each sequence), intersected with the causal bound
 * when causal = 1.  (-1, -1) is attn_fwd; (-1, 0) is causal.  A window needs
 * Tq <= Tk.  A mask mode in the sense of "深度学习反向传播优化：2-CTA MMA模式与
 * 内存访问优化" §5.1-5.2 (FlexAttention-style variants as independent mask
 * modules): the kernels visit only the tiles the band touches and mask the
 * band's edge tiles per element.  Returns ATTN_ERR_INVALID_ARG for bounds
 * below -1.
 */
int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H, int Tq, int Tk, int dqk, int dv, int causal, int window_left,
                    int window_right, float scale, const int* cu_seqlens, int layout,
                    void* stream);

/*
 * Bytes of device workspace attn_bwd needs for these sizes (varlen: 1 when
 * cu_seqlens will be given; Tq is then the total token count).  The
 * workspace holds the fp32 dQ accumulator, D and LSE*log2(e) per query row,
 * one semaphore per (query tile, head), a work counter and a status word.
 * Returns 0 for invalid sizes.  "ops(8)..." §1.3: the caller-provided
 * workspace sized by a query, as the cuDNN graph does.
 */
size_t attn_bwd_workspace_size(int B, int H, int Tq, int Tk, int dqk, int dv, int varlen,
                               int deterministic);

/*
 * Backward: dq, dk, dv (bf16) from q, k, v, o, dO (bf16) and the forward's
 * lse (fp32, required).  deterministic = 1 adds each key tile's dQ
 * contribution in a fixed order (descending key tile, "深度学习反向传播优化：
 * 2-CTA MMA模式与内存访问优化" §3.2), so results are bit-identical run to run;
 * 0 uses unordered fp32 atomics (§3.1).  workspace: device memory of at least
 * attn_bwd_workspace_size() bytes, 256-byte aligned; its contents need no
 * initialisation.  "ops(8)..." §2.1 backward steps 1-5.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
             const float* lse, void* dq, void* dk, void* dv_out, int B, int H, int Tq, int Tk,
             int dqk, int dv, int causal, float scale, const int* cu_seqlens, int layout,
             int deterministic, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward of attn_fwd_window (same window arguments; lse from that forward).
 * Keys that no query sees get dK = dV = 0.
 */
int attn_bwd_window(const void* q, const void* k, const void* v, const void* o, const void* dO,
                    const float* lse, void* dq, void* dk, void* dv_out, int B, int H, int Tq,
                    int Tk, int dqk, int dv, int causal, int window_left, int window_right,
                    float scale, const int* cu_seqlens, int layout, int deterministic,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * The general forward: every option of the calls above in one entry point.
 *
 * Local window: as attn_fwd_window (window_left / window_right, -1 = open).
 *
 * Block-sparse attention: key j is visible to query i only where the block
 * mask marks the pair of blocks (i / ATTN_BLOCK, j / ATTN_BLOCK) with a
 * non-zero byte.  The block-sparse mask module of "深度学习反向传播优化：2-CTA
 * MMA模式与内存访问优化" §5.1-5.2 (FlexAttention and block-sparse variants built
 * from the same kernels by a mask module alone): the kernels skip every tile
 * pair the mask drops.
 *   block_mask: DEVICE pointer to uint8 [mask_batches][mask_heads][NQ][NK],
 *     C order, read only, owned by the caller, unchanged until the call's work
 *     on `stream` is done.  NQ = ceil(Tq / ATTN_BLOCK), NK = ceil(Tk /
 *     ATTN_BLOCK); for variable-length batches NQ = ceil(longest query
 *     sequence / ATTN_BLOCK), NK likewise for the keys, and sequence b uses its
 *     own block coordinates (entries past its ends are not read).
 *     mask_batches is 1 (one mask for every sequence) or B; mask_heads is 1 or
 *     H.  NULL: no block mask.
 * A query row that sees no key gets O = 0 and LSE = -inf (and, in attn_bwd_ex,
 * dQ = 0; it adds nothing to dK or dV).
 *
 * Variable-length batches with separate query and key lengths ("ops(8)..."
 * §1.3: seq_len_q and seq_len_kv given apart): cu_seqlens_q (host, B + 1
 * offsets into the (sum Tq, H, d) queries) and cu_seqlens_k (host, B + 1
 * offsets into the (sum Tk, H, d) keys and values); Tq and Tk are the totals.
 * cu_seqlens_k = NULL: the keys use cu_seqlens_q (Tq == Tk); both NULL: fixed
 * length.  Within sequence b the queries are the last Lq = cu_seqlens_q[b+1] -
 * cu_seqlens_q[b] of its Lk key positions (causal and windows align
 * bottom-right, as for fixed length); a causal or windowed sequence needs
 * Lq <= Lk (ATTN_ERR_UNSUPPORTED otherwise), and a sequence with queries needs
 * keys (ATTN_ERR_INVALID_ARG).  LSE is (H, sum Tq).  Packed QKV needs shared
 * offsets.
 *
 * Returns ATTN_ERR_INVALID_ARG for other mask_batches / mask_heads values or
 * offsets that do not start at 0, decrease, or do not end at the totals.
 */
int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Tq, int Tk, int dqk, int dv, int causal, int window_left, int window_right,
                const unsigned char* block_mask, int mask_batches, int mask_heads, float scale,
                const int* cu_seqlens_q, const int* cu_seqlens_k, int layout, void* stream);

/*
 * Backward of attn_fwd_ex (same options; lse from that forward).  Workspace as
 * for attn_bwd (its size query takes Tq = the total query count and varlen =
 * 1).  Deterministic mode adds the dQ contributions of the kept key tiles in
 * descending key-tile order.
 */
int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dO,
                const float* lse, void* dq, void* dk, void* dv_out, int B, int H, int Tq, int Tk,
                int dqk, int dv, int causal, int window_left, int window_right,
                const unsigned char* block_mask, int mask_batches, int mask_heads, float scale,
                const int* cu_seqlens_q, const int* cu_seqlens_k, int layout, int deterministic,
                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward for callers that cannot allocate device memory (a plugin whose host
 * framework owns all device memory, or a loop where a device-synchronising
 * cudaMalloc is not allowed).  Same arguments and results as attn_bwd, minus
 * the workspace: the library's own 32 MiB device array stands in for it, so
 * it needs attn_bwd_workspace_size() <= 32 MiB (larger problems return
 * ATTN_ERR_SCRATCH_TOO_SMALL; e.g. B=8, H=12, T=1024, d=64 fits).  The first
 * call in each CUDA context looks up the array's address (make it before any
 * stream capture); a call after the device's context was reset and
 * re-created looks it up again.  Every device that loads this code holds the
 * array until exit.  All calls share the array: calls that overlap on the GPU
 * race, so order them on one stream.  A device-side timeout of the last call
 * is read with attn_bwd_noalloc_status().  No counterpart on the pages.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv_out, int B, int H, int Tq,
                     int Tk, int dqk, int dv, int causal, float scale, const int* cu_seqlens,
                     int layout, int deterministic, void* stream);

/*
 * Synchronises `stream` and returns the device status of the last
 * attn_bwd_noalloc call on the current device (ATTN_OK or ATTN_ERR_TIMEOUT),
 * read from the library's scratch array; allocates nothing.  No counterpart
 * on the pages.
 */
int attn_bwd_noalloc_status(void* stream);

/*
 * Synchronises `stream` and returns the device status of the last backward
 * that used `workspace` (ATTN_OK or ATTN_ERR_TIMEOUT).
 */
int attn_bwd_status(const void* workspace, void* stream);

/*
 * Synchronises `stream`, returns the sticky device status of the forward
 * kernels on the current device (ATTN_OK or ATTN_ERR_TIMEOUT) and clears it.
 */
int attn_fwd_status(void* stream);

/*
 * Instrumentation: when both are non-NULL (cudaEvent_t handles), every later
 * attn_bwd call records event_start on its stream just before the backward
 * main kernel and event_stop just after it, so the caller can time that
 * kernel alone.  Pass two NULLs to turn it off.  Returns ATTN_OK, or
 * ATTN_ERR_INVALID_ARG when only one is NULL.  Benchmark support; no
 * counterpart on the pages.
 */
int attn_profile_main_kernel(void* event_start, void* event_stop);

/*
 * Instrumentation, like attn_profile_main_kernel: when all four are non-NULL
 * (cudaEvent_t handles), every later attn_bwd call records pre_start and
 * pre_stop around its preprocess kernel (D and the per-row statistics) and
 * convert_start and convert_stop around its dQ conversion kernel.  Four NULLs
 * turn it off; a mix returns ATTN_ERR_INVALID_ARG.  Benchmark support (the
 * HBM rates of the two memory-bound kernels); no counterpart on the pages.
 */
int attn_profile_aux_kernels(void* pre_start, void* pre_stop, void* convert_start,
                             void* convert_stop);

/*
 * Which backward main kernel later calls use where both apply (dqk = dv = 128,
 * no block mask, no left window edge): 0 = the library's choice, 1 = one CTA
 * per key tile, 2 = CTA pairs (two key tiles per cluster of two CTAs, tcgen05
 * pair MMAs, dQ contracted over both tiles before its atomics; "深度学习反向传播
 * 优化：2-CTA MMA模式与内存访问优化" §2.1-2.2 and §3.1).  Both give results within
 * the same tolerance; deterministic mode is bit-identical run to run with
 * either, though not between them (the pair kernel adds dQ per pair of key
 * tiles).  Returns ATTN_ERR_INVALID_ARG for other values.  Tests and
 * benchmarks use it to run both kernels.
 */
int attn_debug_set_bwd_variant(int variant);

/*
 * Counters of the library's host-side cache (TMA tensor maps and the
 * schedule tables of variable-length batches, reused across calls with the
 * same pointers, shapes and options): out4[0] tensor maps encoded, out4[1]
 * tensor maps reused, out4[2] tables built, out4[3] tables reused, since the
 * library was loaded.  Returns ATTN_ERR_INVALID_ARG for NULL.  Test and
 * diagnostics support; the cache itself follows the build-once, run-many
 * graphs of "ops(8)..." §1.3.
 */
int attn_debug_cache_stats(long long* out4);

/*
 * Test hook (host-side fault injection; 0 = normal operation): every ordered
 * dQ wait of later deterministic attn_bwd calls in this process waits for a
 * semaphore value `bias` higher than the one that will come (a bias above the
 * number of key tiles can never be met), so the bounded wait gives up and
 * attn_bwd_status() reports ATTN_ERR_TIMEOUT.  The kernels
 * stop, free their tensor memory and leave the CUDA context usable.  No
 * counterpart on the pages (whose printed spin-wait, §3.2 of "深度学习反向传播
 * 优化：2-CTA MMA模式与内存访问优化", has no bound).
 */
int attn_debug_set_wait_bias(int bias);

/*
 * Forward + backward for tensors in HOST memory, with the copies overlapped
 * with the kernels (the step a caller makes when its data starts and ends on
 * the host).  q, k, v, dO: host (B,T,H,d) bf16 inputs (layout 0, fixed
 * length, Tq == Tk == T); dq, dk, dv_out: host (B,T,H,d) bf16 outputs; o: host
 * (B,T,H,dv) bf16 output or NULL (O stays on the device).  Host memory should
 * be page-locked (cudaHostAlloc / cudaHostRegister): pageable memory works but
 * its copies do not overlap.  The heads are split into groups of at most
 * heads_per_group (0 = half the heads, rounded up); the first and the last
 * group are about half that size, to shorten the pipeline's fill and drain
 * (H = 16 with the default gives groups of 4, 8, 4).  Each group's slices are copied
 * in on h2d_stream, computed with attn_fwd + attn_bwd on `stream`, and copied
 * back on d2h_stream, two groups in flight.  With stream2 != NULL the two
 * alternating device sets compute on `stream` and stream2, so one group's
 * kernels can start on SMs that the previous group's last work items leave
 * idle.  NULL streams mean `stream` (no overlap).  scratch: device memory of at least
 * attn_step_host_scratch_size() bytes, 256-byte aligned, used only by this
 * call until `stream` passes its end.  Asynchronous: `stream` waits for every
 * copy, so synchronising `stream` makes the host outputs valid.  Results are
 * those of attn_fwd / attn_bwd on the whole tensors (bit-identical with
 * deterministic = 1).  No counterpart on the pages; it moves the data of the
 * step that "ops(8)..." §2.1 defines.
 */
size_t attn_step_host_scratch_size(int B, int H, int T, int dqk, int dv, int heads_per_group,
                                   int deterministic);
int attn_step_host(const void* q, const void* k, const void* v, const void* dO, void* o,
                   void* dq, void* dk, void* dv_out, int B, int H, int T, int dqk, int dv,
                   int causal, float scale, int deterministic, int heads_per_group,
                   void* scratch, size_t scratch_bytes, void* stream, void* stream2,
                   void* h2d_stream, void* d2h_stream);

/*
 * Synchronises `stream` and returns the device status of the last
 * attn_step_host call that used `scratch` with these sizes: ATTN_OK, or the
 * first group's ATTN_ERR_TIMEOUT (forward or backward).
 */
int attn_step_host_status(const void* scratch, int B, int H, int T, int dqk, int dv,
                          int heads_per_group, int deterministic, void* stream);

/* Static text for an ATTN_* code. */
const char* attn_strerror(int code);

/*
 * Host helper (no GPU needed): the order in which the kernels take the
 * sequences of a variable-length batch — longest first, ties by index
 * ("深度学习反向传播优化..." §3.2, batches sorted by expected time).
 * Writes `nseq` sequence indices to order_out.  Returns ATTN_OK or
 * ATTN_ERR_INVALID_ARG.
 */
int attn_varlen_order(const int* cu_seqlens, int nseq, int* order_out);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
