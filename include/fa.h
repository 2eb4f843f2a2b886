/*
 * fa.h - C ABI of the GB300 (sm_103a) exact-attention library, libfa.so.
 *
 * The library computes exact scaled-dot-product attention
 *
 *     O = softmax(scale * Q K^T [+ causal mask]) V
 *
 * tile by tile with the online softmax (running row maximum and row sum, partial
 * outputs rescaled as the maximum grows), so the N x N score and probability
 * matrices never reach device memory; and its backward pass.  The method is the one
 * described in "FlashAttention-2: atención eficiente en GPU para contextos largos"
 * (sections "El coste de mover datos en secuencias largas", "Bloques pequeños,
 * normalización global" and "Tres mejoras en la utilización de la GPU"): exact
 * attention, results equal to the plain definition up to floating-point rounding
 * order, forward and backward, with and without a causal mask.  Grouped-query
 * attention follows "FlashAttention-T: Optimización GPU para LLMs Escalables"
 * (section "Innovaciones técnicas frente a FlashAttention original").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All pointers are DEVICE pointers on the current CUDA device, owned and
 *    allocated by the caller; the library never allocates or frees device memory
 *    during a call.  Every pointer must be 16-byte aligned (tensor-memory-access
 *    copies require it).
 *  - Layouts (row-major, last index fastest, all contiguous):
 *        q, o, dq, dout : [B, N, Hq,  d]     16-bit (see fa_dtype)
 *        k, v, dk, dv   : [B, N, Hkv, d]     16-bit
 *        lse            : [B, Hq, N]         fp32, natural-log log-sum-exp of the
 *                                            SCALED scores of each query row
 *  - Query head h reads key/value head h / (Hq / Hkv) (contiguous groups).
 *  - Causal: key j is visible to query i iff j <= i (queries and keys share N, the
 *    mask is aligned at the top-left corner).
 *  - Supported: d in {64, 128}; 1 <= N <= 2^20; B, Hq, Hkv >= 1; Hq % Hkv == 0;
 *    scale finite and > 0.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Argument errors are reported synchronously, before any
 *    work is enqueued.  Errors inside a kernel (a bounded wait that ran out) are
 *    recorded in a per-device error word that fa_check_device_error() reads.  That
 *    word is shared by every stream and host thread using the device: a check on one
 *    stream reports, and clears, an error raised by a kernel on any stream of the
 *    device, including one that has not finished when the check reads the word.
 *  - Calls on different streams may overlap; the library keeps no per-call state,
 *    except fa_bwd_noalloc, whose calls all share one scratch array and must be
 *    serialised (see there), the persistent kernels of fa_fwd and of the backward
 *    passes for short sequences, whose launches each take a counter pair from a ring of
 *    256 (see fa_fwd), and fa_bwd_deterministic, whose calls each take an event pair
 *    from a ring of 64 for its side stream (see there).
 *  - Per device the library remembers a few addresses and settings (the error word's,
 *    the counter ring's and fa_bwd_noalloc's scratch addresses, each kernel's
 *    shared-memory limit, the deterministic backward's side stream and events), taken on
 *    the first call that needs them.  cudaDeviceReset() discards them on the device
 *    side, so the library must not be used on a device after cudaDeviceReset() in the
 *    same process.
 *  - The compute entry points may be captured into a CUDA graph and replayed (their
 *    host-side work, tensor-map encoding and launch attributes, happens at capture and
 *    is baked into the graph's kernel parameters; the buffers must then stay at the
 *    captured addresses).  Make one call on the device before capturing: the first
 *    call looks up the device's error word and counter ring.  fa_check_device_error synchronises and
 *    cannot be captured.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle (binary-compatible with cudaStream_t / CUstream). */
typedef struct CUstream_st* fa_stream_t;

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID = 1,     /* bad argument: null/misaligned pointer, bad size, Hq % Hkv != 0 */
  FA_ERR_UNSUPPORTED = 2, /* valid but not implemented: d not in {64,128}, N too large */
  FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call or kernel launch failed */
  FA_ERR_TIMEOUT = 4      /* a kernel's bounded wait ran out (reported by fa_check_device_error) */
} fa_status;

typedef enum fa_dtype { FA_BF16 = 0, FA_FP16 = 1 } fa_dtype;

/*
 * Forward pass.
 *   q [B,N,Hq,d], k/v [B,N,Hkv,d] (inputs, dtype), o [B,N,Hq,d] (output, dtype),
 *   lse [B,Hq,N] (output, fp32; needed by fa_bwd).
 *   scale multiplies the scores before the softmax (1/sqrt(d) for standard attention).
 * O is rounded to nearest into `dtype` from an fp32 accumulator.  The kernel is
 * exact attention: it differs from the plain definition only by rounding
 * ("Bloques pequeños, normalización global").
 * Short sequences (N <= 512, or N <= 1024 with the mask) run a persistent kernel: one
 * CTA per SM takes (batch, head, 256-query) units from a counter pair in device memory,
 * one pair per launch from a ring of 256 per device, put back to zero by the launch's
 * last CTA.  Launches that overlap in time get different pairs unless 256 launches
 * separate them; a CUDA graph keeps the pair it was captured with.  Longer sequences
 * run one CTA per unit.  Both kernels round the same operations in the same order.
 * Returns FA_OK once the work is enqueued.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                 int N, int d, int causal, float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd needs for these sizes: an fp32 dQ accumulator of
 * B*Hq*Npad*d elements ([B*Hq, Npad, d] at d=128, [B*Hq, d, Npad] at d=64), then
 * -D = -rowsum(dO * O) and -lse * log2(e), each [B*Hq, Npad] fp32, with Npad = N rounded
 * up to a multiple of 64; each part rounded up to 256 bytes.
 * Returns 0 for invalid or unsupported sizes.
 */
size_t fa_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d);

/*
 * Backward pass: gradients of L = sum(dout * o) with respect to q, k and v.
 *   q, k, v, o, lse : the forward's inputs and outputs (o and lse from fa_fwd with
 *                     the same q, k, v, causal and scale)
 *   dout            : [B,N,Hq,d] upstream gradient dO (dtype)
 *   dq [B,N,Hq,d], dk/dv [B,N,Hkv,d] : outputs (dtype), fully overwritten; dk and
 *                     dv of a key/value head sum over the query heads of its group
 *   workspace       : device scratch of at least fa_bwd_workspace_size() bytes,
 *                     256-byte aligned; its contents on entry do not matter and
 *                     it must not be shared by calls that may overlap.
 * The pass runs D = rowsum(dO * O), then a kernel over key blocks that recomputes
 * P from lse, accumulates dV and dK in tensor memory and adds dS K into the fp32
 * dQ accumulator, then converts dQ to dtype.  Short sequences (N <= 512) run the key
 * blocks in a persistent kernel: one CTA per SM takes (batch, key/value head, 128-key
 * block) units from a counter pair of the ring fa_fwd's persistent kernel uses (same
 * rules).  Longer sequences run one CTA per key block.  For a key block both kernels
 * issue the same products in the same order, so dk and dv agree bit for bit.  Without
 * the mask, when the one-CTA-per-block grid's last wave would occupy at most half of the
 * SMs, its key blocks run as two CTAs each (one per half of the query walk) whose fp32 dK
 * and dV partials are summed before rounding; the partials are kept in dq's memory, which
 * the pass writes last (not when dq overlaps one of the pass's inputs: then the grid is
 * not split).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                 int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                 fa_stream_t stream);

/*
 * Variable-length batches and unequal query / key lengths
 * ------------------------------------------------------
 * Several sequences packed along the token axis, each with its own query length
 * len_q(b) and key length len_k(b).  The pages name boundary handling as a cost of the
 * method ("FlashAttention-2: atención eficiente en GPU para contextos largos", section
 * "Tres mejoras en la utilización de la GPU") and distinguish prefill from decode
 * (section "Cómo documentar una diferencia técnica"); they give no interface, so this
 * one is a reading:
 *  - Layouts (packed, contiguous): q, o, dq, dout [total_q, Hq, d]; k, v, dk, dv
 *    [total_k, Hkv, d] (dtype); lse [Hq, total_q] fp32.
 *  - cu_seqlens_q / cu_seqlens_k: DEVICE int32 arrays of B+1 offsets.  Sequence b owns
 *    rows [cu[b], cu[b+1]).  seqused_q / seqused_k: optional DEVICE int32 arrays of B
 *    lengths (NULL = none).  When given, only the first seqused[b] rows of the segment
 *    are real.  This serves padded batches: cu[b] = b * Nmax with the true lengths in
 *    seqused.
 *  - len(b) = seqused[b] if given, else cu[b+1] - cu[b]; every len(b) must be <= the
 *    max_seqlen_* given (which sizes the grid).  Length 0 is allowed.
 *  - Causal mask aligned at the BOTTOM-RIGHT corner: query i of sequence b sees key j
 *    iff j <= i + len_k(b) - len_q(b), so the last query sees every key (with equal
 *    lengths this is the usual j <= i).  A query that sees no key (len_k = 0, or
 *    i < len_q - len_k under the mask) gets o = 0, lse = -inf, and zero gradients.
 *  - Rows that belong to no sequence (the padding past seqused, gaps between
 *    segments) are not written by any call.  They are read, though (a tile may run past
 *    its sequence), and must hold finite values: masked products multiply them by 0,
 *    and 0 * NaN is NaN.
 *  - The offsets and lengths are read by the kernels, not on the host.  A sequence
 *    whose values contradict total_* / max_seqlen_* (negative length, segment past the
 *    end, length above the maximum, decreasing offsets) is skipped, and the next
 *    fa_check_device_error() returns FA_ERR_INVALID.
 *  - Pointers: 16-byte aligned as above, except that the tensors of a side whose
 *    total is 0 are not read or written and may be NULL; offset arrays 4-byte aligned.
 */

/*
 * Forward pass over a variable-length batch (see above).  total_q / total_k: rows of
 * the packed tensors; max_seqlen_q / max_seqlen_k: bounds on the lengths.  Other
 * arguments as fa_fwd.  total_q == 0 enqueues nothing.
 */
fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                        const int* cu_seqlens_k, const int* seqused_q, const int* seqused_k, int B, int Hq,
                        int Hkv, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d, int causal,
                        float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * Workspace bytes for fa_bwd_varlen: the fa_bwd layout with N replaced by
 * max_seqlen_q (Npad = max_seqlen_q rounded up to 64, at least 64), i.e. an fp32 dQ
 * accumulator of B*Hq*Npad*d elements plus two [B*Hq, Npad] fp32 vectors.  0 for
 * invalid sizes.
 */
size_t fa_bwd_varlen_workspace_size(int B, int Hq, int max_seqlen_q, int d);

/*
 * Backward pass over a variable-length batch: gradients of L = sum(dout * o) for the
 * rows of every sequence; o and lse from fa_fwd_varlen with the same inputs.  dq, dk
 * and dv rows of each sequence are overwritten; other rows are left as they are.
 * workspace as for fa_bwd, sized by fa_bwd_varlen_workspace_size().
 */
fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                        const int* cu_seqlens_k, const int* seqused_q, const int* seqused_k, int B, int Hq, int Hkv,
                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d, int causal, float scale,
                        fa_dtype dtype, void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Decode: a few new queries per sequence against a key/value cache
 * ----------------------------------------------------------------
 * The pages separate decode from prefill ("FlashAttention-2: atención eficiente en GPU
 * para contextos largos", section "Cómo documentar una diferencia técnica") and split
 * work along the sequence when batch and heads leave the GPU idle (section "Tres
 * mejoras en la utilización de la GPU").  The interface is a reading:
 *   q          : [B, Nq, Hq, d]     the new queries (dtype)
 *   k_cache,
 *   v_cache    : [B, Nmax, Hkv, d]  caches (dtype); sequence b uses rows [0, len_b)
 *   cache_seqlens : DEVICE int32 [B], len_b in [0, Nmax] (the new tokens' keys are
 *                   already in the cache: they are its last Nq rows)
 *   o          : [B, Nq, Hq, d] output (dtype);  lse : [B, Hq, Nq] fp32
 * Causal: query i sees key j iff j <= i + len_b - Nq (bottom-right alignment, as for
 * the variable-length calls); a query that sees no key gets o = 0, lse = -inf.
 * The key range of each (batch, key/value head) is split into num_splits parts
 * processed in parallel and merged by their log-sum-exp (num_splits = 0 picks a count
 * from the sizes).  Requires d in {64, 128} and (Hq / Hkv) * Nq <= 128 (the group's
 * queries share one 128-row tile).  Cache rows at or past len_b must hold finite
 * values (they are read and masked, and 0 * NaN would still be NaN); a zero-filled
 * cache satisfies this.  A len_b outside [0, Nmax] is reported as FA_ERR_INVALID by
 * the next fa_check_device_error(), and that sequence is not written.
 */

/* Split count fa_fwd_decode will use for these sizes (0 for invalid sizes). */
int fa_decode_num_splits(int B, int Hq, int Hkv, int Nq, int Nmax, int d, int num_splits);

/*
 * Workspace bytes for fa_fwd_decode: 0 with one split, else fp32 partial outputs
 * [B*Hkv*S, (Hq/Hkv)*Nq, d] and partial log-sum-exps [B*Hkv*S, (Hq/Hkv)*Nq], each
 * rounded up to 256 bytes.  0 also for invalid sizes.
 */
size_t fa_decode_workspace_size(int B, int Hq, int Hkv, int Nq, int Nmax, int d, int num_splits);

/* Decode forward (see above).  workspace: 256-byte aligned, at least
 * fa_decode_workspace_size() bytes (may be NULL when that is 0). */
fa_status fa_fwd_decode(const void* q, const void* k_cache, const void* v_cache, const int* cache_seqlens, void* o,
                        float* lse, int B, int Hq, int Hkv, int Nq, int Nmax, int d, int causal, float scale,
                        int num_splits, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                        fa_stream_t stream);

/*
 * fa_fwd_decode over a paged cache: the keys and values of all sequences live in pages
 * of 128 rows, k_pages / v_pages [num_pages, 128, Hkv, d], and block_table (DEVICE int32
 * [B, max_pages]) gives the page holding keys [128 j, 128 j + 128) of sequence b at
 * block_table[b * max_pages + j].  Entries past a sequence's last block are not read.
 * cache_seqlens[b] <= max_pages * 128.  Other arguments, results and workspace as
 * fa_fwd_decode with Nmax = max_pages * 128 (use fa_decode_workspace_size with that
 * Nmax).  A page index outside [0, num_pages) reads zeros and is reported as
 * FA_ERR_INVALID by the next fa_check_device_error().  Serving engines keep caches this
 * way so that sequences grow without moving memory; the pages describe no paging.
 */
fa_status fa_fwd_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                              const int* cache_seqlens, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                              int num_pages, int max_pages, int d, int causal, float scale, int num_splits,
                              fa_dtype dtype, void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_bwd with a fixed summation order: the same arguments, results within the same
 * tolerance, and dq, dk, dv identical bit for bit from run to run (fa_bwd's dq depends
 * on the order in which key blocks land their fp32 additions).  The dK/dV kernel runs
 * without its dQ path, and a second kernel over 128-query tiles recomputes S and dP and
 * accumulates dQ = scale * sum_j dS_j K_j over the key blocks in ascending order in
 * tensor memory: seven GEMM-shaped products per (query, key) block instead of five.
 * The pages mention no deterministic mode; this is the plain way to get one without
 * atomics or cross-block waits.  workspace as for fa_bwd (only its D and lse parts are
 * used).  The dQ kernel needs only D and lse, so it runs on a non-blocking stream of the
 * library's (one per device) while the dK/dV kernel runs on `stream`; `stream` waits for
 * it before anything enqueued after the call (event fork and join, which CUDA graph
 * capture records as graph edges).
 */
fa_status fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                               int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                               fa_stream_t stream);

/*
 * FP8 (E4M3) forward
 * ------------------
 * The pages report an 8-bit forward ("FlashAttention-T: Optimización GPU para LLMs
 * Escalables", section "Innovaciones técnicas frente a FlashAttention original"); the
 * interface and scaling are a reading:
 *   q [B,N,Hq,128], k/v [B,N,Hkv,128]: E4M3 bytes (the OCP FP8 format with 4 exponent
 *   and 3 mantissa bits, NaN only at 0x7F/0xFF), real value = stored value x the
 *   tensor's descale (q_descale, k_descale, v_descale: finite, > 0).
 *   o [B,N,Hq,128]: bf16.  lse [B,Hq,N]: fp32, natural log of the scaled scores.
 * Scores and their softmax are computed in fp32 from the 8-bit products; P is rounded to
 * E4M3 (as P * 2^7) for the P V product, so O carries up to 2^-4 relative error per term
 * of its sum over keys.  Head dimension 128 only (FA_ERR_UNSUPPORTED otherwise).
 * workspace: at least fa_fwd_fp8_workspace_size() bytes, 256-byte aligned; it receives a
 * transposed copy of V (the 8-bit P V product reads V with keys contiguous).
 * Other conventions as fa_fwd.
 */
size_t fa_fwd_fp8_workspace_size(int B, int Hkv, int N, int d);
fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
                     int d, int causal, float scale, float q_descale, float k_descale, float v_descale,
                     void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * FP8 (E4M3) forward with one descale per 128-row block of each head instead of one per
 * tensor (a reading of the same page: block scaling keeps a block of large values from
 * costing the rest of the tensor its precision).
 *   q_descale: DEVICE fp32 [B, Hq, nb], k_descale and v_descale: DEVICE fp32 [B, Hkv, nb],
 *   nb = ceil(N / 128); rows [128 i, 128 i + 128) of head h of batch b have real value =
 *   stored E4M3 value x descale[b, h, i].  Every entry must be finite and > 0 (not
 *   checked; a value outside that range gives undefined results, not an error).
 * The scores take the query block's and the key block's descales; P is rounded to E4M3
 * as P * 2^7 * v_j / v_max (v_j the key block's V descale, v_max the largest among the
 * blocks a query tile visits), and the row sum and O / l undo that factor, so a key block
 * whose V descale is far below the largest loses P's low values to the subnormal range
 * first.  Other arguments, workspace and conventions as fa_fwd_fp8.
 */
fa_status fa_fwd_fp8_blockscaled(const void* q, const void* k, const void* v, const float* q_descale,
                                 const float* k_descale, const float* v_descale, void* o, float* lse, int B, int Hq,
                                 int Hkv, int N, int d, int causal, float scale, void* workspace,
                                 size_t workspace_bytes, fa_stream_t stream);

/*
 * Size of the scratch array inside the library that fa_bwd_noalloc uses (32 MiB).
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * fa_bwd for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point; it exists for callers such as plugins or engines
 * that are handed only their input and output buffers, programs whose allocator is
 * frozen after start-up, and real-time paths where an allocation's latency or failure
 * is not acceptable.  They cannot provide fa_bwd's workspace.
 *
 * Arguments, layouts and results are those of fa_bwd, without the workspace: the
 * call uses a FA_NOALLOC_SCRATCH_BYTES array that lives in the library.  That array is
 * reserved on every GPU that loads the library's device code and is held until the
 * process exits.  The call itself allocates nothing (no cudaMalloc, no allocating
 * library routine).
 *  - Sizes whose fa_bwd_workspace_size() exceeds FA_NOALLOC_SCRATCH_BYTES return
 *    FA_ERR_UNSUPPORTED before any CUDA call (for example B=1, Hq=16, d=128 fits up
 *    to N of about 4000); other argument errors are fa_bwd's.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call outside
 *    any stream capture.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents; each call re-initialises what it reads (the dQ accumulator is zeroed,
 *    D and lse are rewritten).  Calls that may overlap on the GPU (other streams,
 *    other host threads) race on the array and give wrong results: serialise them.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                         int causal, float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error word.
 * Returns FA_OK, FA_ERR_TIMEOUT (a kernel gave up waiting and wound down without
 * finishing its work; its outputs are undefined), FA_ERR_INVALID (a variable-length
 * call found inconsistent sequence offsets or lengths) or FA_ERR_CUDA (a CUDA call failed,
 * or a kernel found its launch unusable, e.g. a misaligned shared-memory base, and did
 * no work).
 */
fa_status fa_check_device_error(fa_stream_t stream);

/*
 * Self-test of failure detection: launches one small kernel that waits, through the
 * same bounded wait the attention kernels use, on a barrier nothing ever arrives on,
 * with a limit of `limit_us` microseconds (1 .. 1000000).  The wait gives up, the kernel
 * records the timeout in the device error word and exits normally, so the context stays
 * usable.  Returns FA_OK once enqueued (FA_ERR_INVALID for a limit out of range); the
 * next fa_check_device_error() on the stream reports FA_ERR_TIMEOUT.
 */
fa_status fa_selftest_wait_timeout(int limit_us, fa_stream_t stream);

/*
 * Self-test of the exponentials the softmax kernels use: for each of the n fp32 inputs
 * x[i] (DEVICE pointers, 4-byte aligned, n >= 0), y_poly[i] receives 2^x[i] from the
 * polynomial form evaluated on the FMA pipe (round-to-nearest range reduction
 * x = n + f, f in [-1/2, 1/2], and a degree-3 polynomial for 2^f exact at f = 0; relative
 * error below 1.1e-4 for -125 <= x <= 8, exact at integers, exactly 0 below -125) and y_mufu[i] receives
 * the special-function unit's ex2.approx.ftz result, which the attention kernels use.  The
 * polynomial form is an alternative for kernels whose special-function unit is the bound;
 * in this library's forward it measured slower, so no kernel uses it.  The library's own
 * tests compare both forms with the exact value.  Returns FA_OK once
 * enqueued, FA_ERR_INVALID for a negative n or a misaligned pointer.
 */
fa_status fa_selftest_exp2(const float* x, float* y_poly, float* y_mufu, int n, fa_stream_t stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
