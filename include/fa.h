/*
 * fa.h -- C ABI of the exact tiled attention library for GB300 (sm_103a).
 *
 * The library computes exact scaled-dot-product attention
 *
 *     O = softmax(scale * Q K^T) V
 *
 * tile by tile with the streaming (online) softmax rescale, so the N x N score
 * matrix never reaches device memory, and the backward pass that recomputes the
 * probabilities on chip from Q, K and the saved per-row log-sum-exp.
 *
 * Sources (page title and section):
 *   "Flash Attention" chapter (mlx.void.app), sections "地基：流式 softmax",
 *     "FlashAttention——把整件事分块塞进 SRAM" and "FlashAttention-2——让每个核心都忙起来";
 *   review of "FlashAttention: Fast and Memory-Efficient Exact Attention with
 *     IO-Awareness" (trdm.cn), section "方法细节";
 *   FlashAttention practitioner article (cf-1.com/news/4497868), sections 1.1, 2.2, 3.1;
 *   "大模型数学速成（17）：Flash Attention——不物化注意力矩阵", sections 一 to 三.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors q, k, v, o, dO, dq, dk, dv are DEVICE pointers to contiguous
 *    (batch, heads, seq, head_dim) arrays -- the layout of the practitioner
 *    article's section 1.1 -- with element (b, h, n, c) at offset
 *    ((b*H + h)*N + n)*d + c.  All of them share one 16-bit element type `dtype`.
 *    Each base address must be 16-byte aligned (the tiles are moved by TMA).
 *  - lse is a DEVICE pointer to a float32 (batch, heads, seq) array holding the
 *    natural-log log-sum-exp of each row of scaled scores: lse = m + ln(l), where m
 *    is the row maximum of scale*q.k and l = sum_j exp(scale*q.k_j - m).  It carries
 *    the pair (m, l) that the pages' forward keeps for the backward.
 *  - Causal masking: key j is visible to query i iff j <= i (lower triangle).
 *  - Supported: d in {64, 128}; N >= 1; B >= 1; H >= 1; B*H <= 2^30 and
 *    B*H*N < 2^31 rows per tensor (so row indices fit in 32 bits); scale finite and
 *    > 0; dtype FA_BF16 or FA_FP16.  The row limit never binds a call whose tensors
 *    fit in one GPU: 2^31 rows of q and of o alone take 512 GiB at d = 64.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and runs on the calling thread's current CUDA device.
 *  - Ownership: the caller owns every buffer.  fa_fwd and fa_bwd allocate no
 *    device memory; the backward's scratch is the caller's `workspace`.
 *  - Errors: arguments are validated before any launch; on a validation error
 *    the call returns the code and writes nothing.  FA_ERR_LAUNCH means a launch
 *    was rejected by the runtime (cudaGetLastError != success).  Device-side
 *    pipeline timeouts are reported by fa_get_last_kernel_status.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_BF16 = 0, FA_FP16 = 1 } fa_dtype;

typedef enum {
  FA_OK = 0,
  FA_ERR_NULL = 1,            /* a required pointer is NULL                        */
  FA_ERR_SHAPE = 2,           /* B, H or N < 1, or B*H*N too large                 */
  FA_ERR_UNSUPPORTED_D = 3,   /* head_dim not in {64, 128}                         */
  FA_ERR_DTYPE = 4,           /* dtype not FA_BF16 / FA_FP16                       */
  FA_ERR_ALIGN = 5,           /* a tensor base address is not 16-byte aligned      */
  FA_ERR_WORKSPACE = 6,       /* workspace NULL or smaller than fa_bwd_workspace_size */
  FA_ERR_LAUNCH = 7,          /* the CUDA runtime rejected a launch                */
  FA_ERR_DEVICE_TIMEOUT = 8,  /* a kernel's bounded pipeline wait gave up          */
  FA_ERR_NO_DEVICE = 9,       /* no usable sm_100-family device is current         */
  FA_ERR_SCALE = 10,          /* scale not finite or not > 0                       */
  FA_ERR_SCRATCH_LIMIT = 11,  /* fa_bwd_noalloc: the problem needs more scratch than
                                 the library's built-in array holds                 */
  FA_ERR_PATTERN = 12         /* fa_fwd_sparse / fa_bwd_sparse: unknown block pattern */
} fa_status;

/* Block patterns of fa_fwd_sparse / fa_bwd_sparse. */
typedef enum { FA_PATTERN_BUTTERFLY = 1 } fa_pattern;

/*
 * Forward: O and lse from Q, K, V.
 *
 * Computes, for every (b, h), S = scale * Q K^T (masked when `causal` != 0),
 * O = softmax(S) V and lse = row log-sum-exp of S, tile by tile: each block of
 * 128 query rows streams the key/value blocks through shared memory, keeps the
 * running maximum m, running sum l and an unnormalised output in on-chip memory,
 * rescales them by 2^(m_old - m_new) when the maximum moves, and divides by l once
 * at the end ("Flash Attention" chapter, sections "地基：流式 softmax" and
 * "FlashAttention-2"; practitioner article section 2.2).  Blocks wholly above the
 * causal diagonal are skipped.
 *
 *   q, k, v : in,  (B, H, N, d) `dtype`
 *   o       : out, (B, H, N, d) `dtype`, overwritten
 *   lse     : out, (B, H, N) float32, overwritten
 *   Returns FA_OK or an fa_status error code.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, float scale, int causal, int dtype, void* stream);

/*
 * Forward with different query and key lengths and with grouped key/value heads.
 *   q, o  : [B, H, Nq, d];   k, v : [B, Hkv, Nk, d];   lse : [B, H, Nq] float32.
 *   Query head h reads key/value head h / (H / Hkv) (Hkv must divide H; Hkv = H is
 *   ordinary multi-head attention, Hkv = 1 multi-query attention).
 *   causal : the mask is aligned bottom-right: query row i sees key j iff
 *            j <= i + (Nk - Nq), so the last query row is the newest token and
 *            Nq = Nk gives fa_fwd's mask.  When Nk < Nq the first Nq - Nk rows see no
 *            key; their O rows are 0 and their lse is -inf.
 * Everything else (layout, alignment, dtype, scale, stream, errors; FA_ERR_SHAPE
 * also when Hkv does not divide H) is as for fa_fwd, which is this call with
 * Hkv = H and Nq = Nk = N.  The pages define attention for one sequence length; the
 * cross lengths, the bottom-right alignment and the head grouping are this
 * library's reading (the practitioner article, section 3.1, decodes new tokens
 * against a key/value cache; "大模型数学速成（17）", section 五, names grouped-query
 * attention as orthogonal to the tiling).
 */
int fa_fwd_cross(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                 int dtype, void* stream);

/*
 * Bytes of device scratch that fa_bwd needs for these sizes: per 128-row query
 * block a 4 KB tile holding -lse/scale and -D = -rowsum(dO o O) of its rows (the
 * operand of the rank-one products that subtract them on the tensor core), plus a
 * float32 dQ accumulator of B*H*N*d elements.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward: dq, dk, dv from Q, K, V, O, dO and lse (as written by fa_fwd).
 *
 * Recomputes P = exp(scale*Q K^T - lse) tile by tile on chip instead of reading a
 * stored probability matrix (review of the FlashAttention paper, "方法细节";
 * "Flash Attention" chapter, end of the section "FlashAttention——把整件事分块塞进
 * SRAM").  With D_i = sum_c dO_ic O_ic it forms dV = P^T dO, dP = dO V^T,
 * dS = P o (dP - D), dQ = scale dS K and dK = scale dS^T Q.  The loop runs over
 * key/value blocks on the outside and query blocks inside; dQ partial products
 * are summed in float32 in the workspace and converted at the end, so dq may
 * differ in the last bits from run to run.
 *
 *   q, k, v, o, dO : in,  (B, H, N, d) `dtype`
 *   lse            : in,  (B, H, N) float32
 *   dq, dk, dv     : out, (B, H, N, d) `dtype`, overwritten (not accumulated)
 *   workspace      : scratch, >= fa_bwd_workspace_size(B,H,N,d) bytes, 256-byte
 *                    aligned; contents on entry are ignored and on exit undefined.
 *                    Two calls in flight at once must not share it.
 *   Returns FA_OK or an fa_status error code.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
           const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
           int B, int H, int N, int d, float scale, int causal, int dtype, void* stream);

/*
 * Backward with grouped key/value heads (square N): the gradients of fa_fwd_cross
 * with Nq = Nk = N.
 *   q, o, dO, dq : [B, H, N, d];   k, v, dk, dv : [B, Hkv, N, d];   lse : [B, H, N].
 *   Query head h reads key/value head h / (H / Hkv); dk and dv of a key/value head
 *   are the sums of the per-query-head gradients over the H / Hkv query heads that
 *   read it (accumulated on chip, written once).  The workspace is
 *   fa_bwd_workspace_size(B, H, N, d).  Everything else, including the errors
 *   (FA_ERR_SHAPE also when Hkv does not divide H), is as for fa_bwd, which is this
 *   call with Hkv = H.
 */
int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO,
               const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
               int B, int H, int Hkv, int N, int d, float scale, int causal, int dtype,
               void* stream);

/*
 * Split-key decode: attention for a few query rows per key/value head, e.g. new
 * tokens against a key/value cache.  Shapes, head grouping, the bottom-right causal
 * mask and the O = 0 / lse = -inf convention are those of fa_fwd_cross; the result
 * is the same attention (within the usual rounding).  Requires (H / Hkv) * Nq <= 8
 * (FA_ERR_SHAPE otherwise; use fa_fwd_cross for more rows) and B * Hkv <= 65535
 * (FA_ERR_SHAPE otherwise).
 *
 * The keys of each head are cut into ranges processed by separate CTAs on the CUDA
 * cores (the pass reads K and V once and is bound by memory bandwidth); the
 * per-range results are combined with lse = ln sum_s e^{lse_s},
 * O = sum_s e^{lse_s - lse} O_s.
 *   workspace : device scratch for the per-range results, 256-byte aligned, at least
 *               fa_decode_workspace_size(B, H, Hkv, Nq, Nk, d) bytes (may be NULL when
 *               that is 0); FA_ERR_WORKSPACE otherwise.  Overwritten.
 * fa_decode_workspace_size returns 0 for invalid sizes as well.
 */
size_t fa_decode_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d);
int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
              size_t ws_bytes, int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
              int dtype, void* stream);

/*
 * Block-sparse attention with a fixed butterfly pattern (FlashAttention review,
 * "方法细节": block-sparse FlashAttention with a fixed butterfly mask).  The pattern's
 * blocks are 256 rows and 256 keys (two 128-row tiles): query block p sees key block q
 * iff p == q or the binary block indices differ in exactly one bit.  With `causal` the
 * element mask key <= query applies on top.  Blocks outside the pattern are never
 * loaded or computed (as the causal skip), so the work grows as N log N.
 *   pattern : FA_PATTERN_BUTTERFLY (FA_ERR_PATTERN otherwise).
 * Shapes, layout, dtypes, lse, workspace and errors are those of fa_fwd / fa_bwd
 * (square N, one key/value head per query head).
 */
int fa_fwd_sparse(const void* q, const void* k, const void* v, void* o, float* lse,
                  int B, int H, int N, int d, float scale, int causal, int pattern, int dtype,
                  void* stream);
int fa_bwd_sparse(const void* q, const void* k, const void* v, const void* o, const void* dO,
                  const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                  int B, int H, int N, int d, float scale, int causal, int pattern, int dtype,
                  void* stream);

/*
 * Host utility: the 128-row key blocks that the query blocks of butterfly pair `pair`
 * (query blocks 2*pair and 2*pair+1) visit, in order, for `nblocks` 128-row blocks.
 * causal_dir: 0 all linked pairs, -1 only pairs <= `pair` (the causal forward), +1 only
 * pairs >= `pair`.  Writes up to `cap` block indices to `out` and returns their number
 * (-1 for invalid arguments).  Runs on the host; needs no device.
 */
int fa_butterfly_blocks(int nblocks, int pair, int causal_dir, int* out, int cap);

/*
 * FP8 forward ("Flash Attention" chapter, mlx.void.app, section "FlashAttention-3——重叠
 * 与低精度": E4M3 numbers, block quantization, and a fixed random rotation of Q and K
 * applied before rounding).
 *
 * fa_quantize_fp8: E4M3 codes and per-block scales of a 16-bit (B, H, N, d) tensor.
 *   x          : in,  (B, H, N, d) `dtype`, 16-byte aligned
 *   x8         : out, E4M3 codes, 16-byte aligned: (B, H, N, d) bytes, or with
 *                `transpose` (B, H, d, Nt) bytes with Nt = fa_fp8_vt_cols(N) -- the V^T
 *                layout fa_fwd_fp8 reads (keys N .. Nt-1 are written as +0)
 *   scales     : out, (B, H, ceil(N/128)) float32: block j of a head holds rows
 *                128j .. 128j+127 and represents code * scales[j]
 *   signs      : NULL, or d floats of +-1 (device memory): rows are first multiplied by
 *                the rotation diag(signs) H / sqrt(d) (H the Sylvester-Hadamard matrix);
 *                give the same signs for Q and K, none for V
 *   per_tensor : 0: scale = amax(block) / 448 per block; 1: the head's amax for every
 *                block (one scale per (b, h) -- the failure mode block scales avoid)
 *   Blocks whose values are all 0 get scale 1.  Codes round to nearest even and
 *   saturate at +-448.  Three launches on `stream`; errors as fa_fwd.
 *
 * fa_fwd_fp8: O and lse from E4M3 codes, Nq = Nk = N, one key/value head per query head.
 *   q8, k8     : in, (B, H, N, d) E4M3 codes; vt8 : in, (B, H, d, Nt) codes of V^T
 *   q_scale, k_scale, v_scale : in, (B, H, ceil(N/128)) float32 block scales (> 0)
 *   o, lse     : out as fa_fwd, o in `dtype` (bf16 or fp16)
 *   The products run on the 8-bit tensor-core path with fp32 accumulation; P is rounded
 *   to E4M3 (relative error up to 2^-4 per entry) before P.V, so O carries that error on
 *   top of the inputs' quantization; lse uses the unrounded P.
 * Both return FA_OK or an fa_status error code, validated before any launch.
 */
int fa_fp8_vt_cols(int N);
int fa_quantize_fp8(const void* x, void* x8, float* scales, int B, int H, int N, int d, int dtype,
                    const float* signs, int per_tensor, int transpose, void* stream);
int fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale,
               const float* k_scale, const float* v_scale, void* o, float* lse, int B, int H,
               int N, int d, float scale, int causal, int dtype, void* stream);

/*
 * The three stages fa_bwd runs, one launch each, for callers that want to time or
 * schedule them separately.  Arguments, validation and errors are exactly fa_bwd's;
 * calling the three in this order on one stream with one workspace is fa_bwd.
 *   fa_bwd_preprocess : -D_i = -sum_c dO_ic O_ic and -lse*log2(e) into the workspace
 *                       (padding rows of the last block get 0 and -inf, so their
 *                       probabilities are exactly 0), and zeroes the workspace's
 *                       float32 dQ accumulator and its tile counter.
 *   fa_bwd_dkdv       : the key/value-outer kernel: writes dk and dv, adds the dQ
 *                       partial products into the accumulator.  Its CTAs take work
 *                       tiles from the workspace's tile counter, so each fa_bwd_dkdv
 *                       needs a fa_bwd_preprocess on the same workspace before it.
 *   fa_bwd_dq_convert : dq = scale * accumulator, rounded to `dtype`.
 */
int fa_bwd_preprocess(const void* q, const void* k, const void* v, const void* o, const void* dO,
                      const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                      int B, int H, int N, int d, float scale, int causal, int dtype, void* stream);
int fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* o, const void* dO,
                const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                int B, int H, int N, int d, float scale, int causal, int dtype, void* stream);
int fa_bwd_dq_convert(const void* q, const void* k, const void* v, const void* o, const void* dO,
                      const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                      int B, int H, int N, int d, float scale, int causal, int dtype, void* stream);

/*
 * Backward without any device allocation (no counterpart in the paper: this entry
 * point exists for callers, not for the method).
 *
 * Same computation, arguments and validation as fa_bwd, minus the workspace.  It is
 * for callers that cannot allocate device memory when they run the backward -- for
 * example, code running under a framework whose caching allocator already holds the
 * device's memory, a plugin host that passes a kernel library nothing but the tensors
 * it works on, or a latency-critical path that cannot afford cudaMalloc's possible
 * device synchronisation or failure.  Its scratch is a fixed array of
 * fa_bwd_noalloc_max_scratch() bytes (32 MiB) that the library keeps in device memory
 * on every GPU where it is loaded, until the process exits.
 *
 *   - Sizes whose fa_bwd_workspace_size exceeds that limit are rejected with
 *     FA_ERR_SCRATCH_LIMIT before anything is launched (at d = 64 the limit is
 *     about 7.4 million elements of B*H*N*d).
 *   - No cudaMalloc, cudaFree or other allocating call is made.
 *   - The first call on each device looks up the array's device address (with that
 *     device current); make that first call before any stream capture.  The lookup
 *     is repeated when the device's current context has changed since (a device
 *     reset replaces the context and the address).
 *   - Every call on a device shares the one array and it keeps the last call's
 *     contents (each call re-zeroes what must start at zero).  Calls whose work
 *     overlaps on the GPU -- two streams, or two host threads -- race on it.
 */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, void* dq, void* dk, void* dv,
                   int B, int H, int N, int d, float scale, int causal, int dtype, void* stream);

/* Size in bytes of fa_bwd_noalloc's built-in scratch array. */
size_t fa_bwd_noalloc_max_scratch(void);

/* Static, human-readable text for a status code; never NULL. */
const char* fa_strerror(int status);

/*
 * Synchronises `stream`, then reads and clears the current device's kernel error
 * word.  Returns FA_OK, FA_ERR_DEVICE_TIMEOUT when a kernel's bounded mbarrier
 * wait gave up (the kernel then skipped its remaining work, released its tensor
 * memory and returned), or FA_ERR_LAUNCH if the stream reported a CUDA error.
 */
int fa_get_last_kernel_status(void* stream);

/* Number of streaming multiprocessors the persistent kernels size their grids to
 * on the current device, or a negative fa_status on error. */
int fa_device_sm_count(void);

/*
 * Test hook for the bounded-wait path: launches one block that waits on an
 * mbarrier nobody arrives on, with a wait limit of `limit_us` microseconds
 * (clamped to [1, 2000000]).  The kernel gives up, records FA_ERR_DEVICE_TIMEOUT in
 * the error word and returns; fa_get_last_kernel_status then reports it.  No trap,
 * no fault.
 */
int fa_debug_wait_timeout(unsigned limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
