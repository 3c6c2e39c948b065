/*
 * Fused multi-head scaled-dot-product attention forward for GB300 (sm_103a).
 *
 *   O = softmax(scale * Q K^T + mask) V,   LSE_i = ln sum_j exp(scale * q_i . k_j)
 *
 * Definition: page "Multi-Head Attention的计算本质与性能瓶颈" (mlqm.cn), §1 and
 * §2.1 (Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V); causal rule from §3.1 of
 * the same page (score kept when key index j <= query index i, else -inf).
 * Packed variable-length batches follow the varlen call of page
 * "长文本处理性能断层真相" (lnrk.cn), §1 (int32 cu_seqlens prefix offsets).
 * The kernel tiles over key blocks with the online softmax of page
 * "深度学习算子优化：从TFLOPS幻觉到FlashAttention实战" (jianying88.com), §3, so
 * the Sq x Sk score matrix never reaches global memory.
 *
 * All functions are plain C.  Device pointers are owned by the caller; the
 * library never frees or keeps them past the call.  Every launch is
 * asynchronous on the caller's stream.  There is no CPU fallback: on anything
 * other than an sm_103 device the call returns ATTN_ERR_UNSUPPORTED.
 */
#ifndef ATTN_TCGEN05_H
#define ATTN_TCGEN05_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  Zero is success; every failure is negative. */
typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1,    /* null pointer, negative size, non-finite scale, ... */
  ATTN_ERR_UNSUPPORTED = -2,    /* head dim, dtype or device not supported */
  ATTN_ERR_MISALIGNED = -3,     /* q/k/v/o not 16-byte aligned, lse/cu_seqlens not 4-byte */
  ATTN_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed */
  ATTN_ERR_DEVICE_TIMEOUT = -5, /* a kernel pipeline wait ran past its limit (reported by attn_check) */
  ATTN_ERR_BAD_SEQLENS = -6     /* cu_seqlens not non-decreasing within [0, total] (attn_check) */
} attn_status;

typedef enum { ATTN_DTYPE_FP16 = 0, ATTN_DTYPE_BF16 = 1 } attn_dtype;

/*
 * attn_fwd -- fused attention forward (O and LSE) in one persistent kernel.
 *
 * Layouts (all row-major, contiguous, head dim innermost):
 *   dense  (cu_seqlens_q == cu_seqlens_k == NULL):
 *     q, o : [B, Sq, H, D]   k, v : [B, Sk, H, D]   lse : float [B, H, Sq]
 *   varlen (both cu_seqlens non-NULL, int32 device arrays of B+1 entries):
 *     q, o : [Sq, H, D]      k, v : [Sk, H, D]      lse : float [H, Sq]
 *     Sq / Sk are the TOTAL packed rows (the allocation lengths).  Sequence b
 *     owns query rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key rows
 *     [cu_seqlens_k[b], cu_seqlens_k[b+1]); it never attends to another one.
 *     Rows that belong to no sequence are still read as padding of a
 *     neighbour's tiles (with weight zero) and must hold finite values.
 *
 * Arguments:
 *   q, k, v   fp16 or bf16 (per dtype), 16-byte aligned device pointers.
 *   o         output, same dtype, 16-byte aligned; written for valid rows only.
 *   lse       output, fp32, natural-log logsumexp of the scaled, masked scores;
 *             -inf for a row that sees no key (an empty key sequence).
 *   B, H      batch (dense) or number of sequences (varlen); heads.  B >= 0, H >= 1.
 *   Sq, Sk    see above.  Sk >= 1.  B == 0 or Sq == 0 is a no-op.
 *   D         head dim, 64 or 128 (else ATTN_ERR_UNSUPPORTED).
 *   scale     finite score scale (1/sqrt(D) is the usual choice; 0 allowed).
 *   causal    non-zero: key j visible to query i (indices within the
 *             sequence) only when j <= i (top-left aligned; Sq != Sk allowed).
 *   dtype     attn_dtype.
 *   stream    cudaStream_t (passed as void*), NULL = legacy default stream.
 *
 * Errors: argument, alignment, dtype and device errors are returned before
 * anything is launched and leave o/lse untouched.  Each pointer is checked to
 * be device (or managed) memory of the current device; a pointer that passed
 * the check is remembered per thread (the last 16), so the check tests where a
 * buffer lives, not whether it is still allocated.  Launch failures return
 * ATTN_ERR_CUDA.  Problems found on the device (a bad cu_seqlens array, a
 * pipeline wait past its limit) set a per-device error word that attn_check
 * reports; outputs of that call are then undefined.
 * Thread-safe; per-device state is created on first use.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int Sq, int Sk, int D, float scale, int causal,
             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
             int dtype, void* stream);

/*
 * attn_fwd_window -- attn_fwd with a sliding-window mask and global query rows.
 *
 * The mask follows the "sliding window + global tokens" scheme of page
 * "长文本处理性能断层真相" (lnrk.cn), §2.5, for 128K-token contexts: every
 * query attends to a band of nearby keys, and the first global_q queries of
 * each sequence attend to all keys.  With indices i (query) and j (key) inside
 * one sequence, key j is visible to query i when
 *   i >= global_q:  i - window_left <= j <= i + window_right   (and j <= i if causal)
 *   i <  global_q:  always                                      (j <= i if causal)
 * window_left / window_right = -1 leave that side unbounded, so
 * attn_fwd_window(..., -1, -1, 0, ...) computes exactly attn_fwd.  A causal
 * sliding window of W keys (the query itself and the W-1 before it) is
 * window_left = W - 1, window_right = 0 (or -1), causal = 1.
 *
 * Arguments, layouts, ownership, stream semantics and errors as attn_fwd, and:
 *   window_left, window_right  >= -1, else ATTN_ERR_INVALID_ARG; with causal
 *                              set, window_right > 0 is ATTN_ERR_INVALID_ARG.
 *   global_q                   >= 0, else ATTN_ERR_INVALID_ARG.
 * A row that sees no key gets O = 0 and LSE = -inf.  K/V tiles that no row of
 * a query tile can see are skipped, so the work grows with the band width, not
 * with Sk.
 */
int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int Sq, int Sk, int D, float scale, int causal,
                    int window_left, int window_right, int global_q,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                    int dtype, void* stream);

/*
 * attn_fwd_decode -- attention of a few new queries against a KV cache.
 *
 * Decode step of page "长文本处理性能断层真相" (lnrk.cn), §2.2: the cache holds
 * the keys/values of every earlier token and grows with the sequence; the Sq
 * new queries of sequence b are the last Sq positions, L_b - Sq .. L_b - 1, of
 * a sequence whose cache holds L_b rows.  Key j of the cache is visible to new
 * query t when j < L_b and, if causal, j <= L_b - Sq + t (queries at negative
 * positions see nothing: O = 0, LSE = -inf).  The keys are split into chunks
 * processed in parallel and the partial results are combined with the
 * log-sum-exp merge of attn_merge (the ring-attention combine step of the same
 * page, §1), so one sequence can use the whole GPU.
 *
 * Layouts (row-major, contiguous, head dim innermost):
 *   q, o              [B, Sq, H, D]       fp16/bf16 (per dtype)
 *   k_cache, v_cache  [B, Sk, H, D]       Sk = cache capacity (rows per sequence)
 *   lse               float [B, H, Sq]    natural log, like attn_fwd
 *   seqlens_k         int32 [B] on the device: valid rows L_b (0 <= L_b <= Sk),
 *                     or NULL for L_b = Sk.  A value outside [0, Sk] sets the
 *                     device error word (ATTN_ERR_BAD_SEQLENS via attn_check).
 * Arguments: 1 <= Sq <= 16 (else ATTN_ERR_UNSUPPORTED), D 64 or 128, finite
 * scale; q, k_cache, v_cache, o 16-byte aligned, lse and seqlens_k 4-byte.
 * workspace: device scratch of at least the size attn_decode_workspace reports
 * for the same B, H, Sq, Sk, D on the current device (256-byte aligned; may be
 * NULL when that size is 0).  The caller owns it and must not use it for
 * anything else until the call's work on `stream` has finished.
 * Errors and ownership as attn_fwd; asynchronous on `stream`.
 */
int attn_fwd_decode(const void* q, const void* k_cache, const void* v_cache, void* o,
                    float* lse, int B, int H, int Sq, int Sk, int D, float scale, int causal,
                    const int32_t* seqlens_k, void* workspace, size_t workspace_bytes,
                    int dtype, void* stream);

/*
 * attn_decode_workspace -- bytes of workspace attn_fwd_decode needs for these
 * sizes on the current device (0 when the keys are not split).  Same argument
 * rules as attn_fwd_decode; the value depends on the device's SM count.
 */
int attn_decode_workspace(int B, int H, int Sq, int Sk, int D, size_t* bytes);

/*
 * attn_merge -- combine attention results computed over disjoint key sets.
 *
 * For n_parts results of the same queries over disjoint key sets (for example
 * the shards of a ring attention, page "长文本处理性能断层真相", §1, or the
 * key chunks of a long sequence), returns attention over the union:
 *   w_p = exp(LSE_p - max_p LSE_p),  O = sum_p w_p O_p / sum_p w_p,
 *   LSE = max_p LSE_p + ln sum_p w_p;   rows where every LSE_p is -inf get
 *   O = 0 and LSE = -inf.
 * Layouts: o_parts [n_parts, B, S, H, D] (dtype), lse_parts float
 * [n_parts, B, H, S] -- the outputs of n_parts attn_fwd calls stacked (a varlen
 * result is B = 1, S = total rows); o [B, S, H, D] (dtype), lse float [B, H, S].
 * n_parts >= 1; 1 <= D <= 1024 (else ATTN_ERR_UNSUPPORTED); B * S * H < 2^31;
 * 2-byte (o) and 4-byte (lse) alignment.
 * Errors and ownership as attn_fwd; asynchronous on `stream`.
 */
int attn_merge(const void* o_parts, const float* lse_parts, int n_parts, int B, int S, int H,
               int D, void* o, float* lse, int dtype, void* stream);

/*
 * attn_bwd -- gradients of attn_fwd: dQ, dK, dV from dO.
 *
 * Page "Multi-Head Attention的计算本质与性能瓶颈" (mlqm.cn), §3.3 reserves a
 * backward for every operator and states that masked connections carry no
 * gradient; the formulas are the chain rule through the forward definition,
 * with P recomputed from the forward's LSE (P = exp(scale q.k - LSE)):
 *   dV = P^T dO,  dS = P * (dO V^T - D),  D = rowsum(dO * O),
 *   dQ = scale dS K,  dK = scale dS^T Q.
 * Layouts as attn_fwd:
 *   dense (cu_seqlens_q = cu_seqlens_k = NULL):
 *     q, o, dout, dq   [B, Sq, H, D]     k, v, dk, dv  [B, Sk, H, D]   (dtype)
 *     lse              float [B, H, Sq]
 *   packed sequences (both cu_seqlens given, device int32 [B + 1], as attn_fwd):
 *     q, o, dout, dq   [Sq, H, D]        k, v, dk, dv  [Sk, H, D]      (Sq, Sk: total rows)
 *     lse              float [H, Sq]
 * lse is the LSE attn_fwd returned for q, k, v.  causal as attn_fwd
 * (top-left, within each sequence).  D 64 or 128.  scale must be finite and
 * non-zero (ATTN_ERR_UNSUPPORTED for 0: the LSE term is carried as -LSE/scale).
 * All 16-bit pointers 16-byte aligned, lse and cu_seqlens 4-byte.  workspace:
 * device scratch of at least attn_bwd_workspace(B, H, Sq, D, packed) bytes
 * (packed = 1 when cu_seqlens are given), 256-byte aligned; the call
 * initialises what it needs.  As in attn_fwd, rows of q, k, v and dout that
 * belong to no sequence must be finite (o and lse there are not read).  dq
 * rows that belong to no sequence come out zero; dk/dv rows of keys that
 * belong to no sequence are not written (with no query rows at all, Sq = 0,
 * the whole of dk and dv is zeroed).  Malformed sequence bounds (cu_seqlens
 * not non-decreasing within [0, Sq] / [0, Sk]) make the call do nothing
 * further and attn_check report ATTN_ERR_BAD_SEQLENS.  dQ is accumulated with
 * fp32 reduce-adds, so its last bits may differ between runs; dK and dV are
 * deterministic.  Errors and ownership as attn_fwd; asynchronous on `stream`.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk,
             int D, float scale, int causal, const int32_t* cu_seqlens_q,
             const int32_t* cu_seqlens_k, void* workspace, size_t workspace_bytes, int dtype,
             void* stream);

/*
 * attn_bwd_workspace -- bytes of workspace attn_bwd needs: an fp32 dQ
 * accumulator (query rows * H * D * 4, rounded up to 256) and 8 KiB per
 * 128-query tile per (sequence, head) for the per-query terms -LSE/scale and
 * -D.  Dense (packed = 0): B * ceil(Sq / 128) tiles per head.  Packed
 * (packed = 1; B sequences, Sq total query rows): at most
 * floor((Sq + 127 B) / 128) tiles per head, plus 4 * (B + 2) bytes (rounded up
 * to 256) for the per-sequence tile offsets.
 */
int attn_bwd_workspace(int B, int H, int Sq, int D, int packed, size_t* bytes);

/*
 * attn_fwd_fp8 -- attn_fwd for 8-bit (e4m3) Q, K, V with per-tensor scales.
 *
 * Low-precision operands as a memory and throughput lever of the fused kernel
 * (page "深度学习算子优化：从TFLOPS幻觉到FlashAttention实战", §3).  The inputs are
 * e4m3 codes (OCP FP8, 1-4-3, no infinities) and the real values are
 * q = q_code * q_scale, k = k_code * k_scale, v = v_code * v_scale; O and LSE
 * are those of attn_fwd on these real values, O in out_dtype (fp16/bf16).
 * The probabilities are rounded to e4m3 for the P V product (the rounding
 * largely cancels against the row sum, which adds the same rounded values).
 * Dense layouts only: q [B, Sq, H, 128], k, v [B, Sk, H, 128] (1 byte each),
 * o [B, Sq, H, 128] (out_dtype), lse float [B, H, Sq]; D must be 128
 * (ATTN_ERR_UNSUPPORTED otherwise); causal as attn_fwd; all scales finite.
 * workspace: device scratch of at least attn_fwd_fp8_workspace(B, H, Sk, 128)
 * bytes (V transposed to [H, 128, keys], keys padded to a multiple of 16),
 * 256-byte aligned.  Errors and ownership as attn_fwd; asynchronous on `stream`.
 */
int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                 int H, int Sq, int Sk, int D, float scale, float q_scale, float k_scale,
                 float v_scale, int causal, void* workspace, size_t workspace_bytes,
                 int out_dtype, void* stream);

/* attn_fwd_fp8_workspace -- bytes of workspace attn_fwd_fp8 needs: H * 128 * B * round16(Sk). */
int attn_fwd_fp8_workspace(int B, int H, int Sk, int D, size_t* bytes);

/*
 * attn_check -- synchronise `stream`, then report and clear the device error
 * word of the current device: ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT,
 * ATTN_ERR_BAD_SEQLENS, or ATTN_ERR_CUDA if the stream itself failed.
 * The error word is one per device, not per stream: every call of the
 * allocating entry points on that device reports into it, so an error raised
 * by a kernel on another stream (that has finished by then) is reported too,
 * to whichever caller checks first, and is cleared by that check.
 *
 * Debug environment (read at every call): ATTN_WAIT_TIMEOUT_MS bounds every
 * device-side wait (default 5000); when one runs out the kernel sets the
 * error word, its roles drain and it exits, leaving the context usable.
 * ATTN_INJECT_FAULT (tests only): 1 = block 0 of the forward kernels
 * (attn_fwd, attn_fwd_window) skips its first K tile, block 0 of the decode
 * kernel its first tile fill, so that a wait runs out (ATTN_ERR_DEVICE_TIMEOUT
 * from attn_check); 2 = attn_fwd_decode launches its kernel with an empty
 * grid, which the launch rejects (the call returns ATTN_ERR_CUDA).
 */
int attn_check(void* stream);

/* attn_status_string -- static, human-readable name of a status code. */
const char* attn_status_string(int status);

/*
 * attn_num_sms -- SM count the persistent grid is sized from on the current
 * device (>0), or a negative status.
 */
int attn_num_sms(void);

/*
 * attn_last_launch -- grid size (CTAs) and dynamic shared memory bytes of the
 * main kernel of the most recent launch by attn_fwd, attn_fwd_window,
 * attn_fwd_decode, attn_bwd or attn_fwd_fp8 on this thread; either pointer may
 * be NULL.  Returns ATTN_OK, or ATTN_ERR_INVALID_ARG if nothing was launched
 * yet.  With ATTN_DEBUG=1 in the environment each such launch also prints one
 * line ("attn: <entry point> grid=<CTAs> smem=<bytes>") to stderr; the library
 * prints nothing otherwise.
 */
int attn_last_launch(int* grid_ctas, int* smem_bytes);

/*
 * attn_fwd_noalloc -- attn_fwd for callers that must not allocate device memory.
 * (The pages have no counterpart; this is an integration entry point.)
 *
 * Same arguments, layouts and argument errors as attn_fwd, plus device_status.
 * attn_fwd cudaMalloc's a 4-byte device error word on its first call on a
 * device; a caller whose framework owns all device memory through its own
 * allocator, or that cannot accept cudaMalloc's implicit synchronisation,
 * cannot allow that.  This call runs the same kernel with its scratch in a
 * fixed 256-byte static device array (held by every GPU that loads the library
 * until exit) and calls no cudaMalloc, cudaFree or other allocating routine.
 *   device_status  optional host pointer.  NULL: the call stays asynchronous
 *                  and device-side errors are not reported.  Non-NULL: the call
 *                  waits for `stream` and stores ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT
 *                  or ATTN_ERR_BAD_SEQLENS there.
 * Device-side waits are bounded as in attn_fwd (ATTN_WAIT_TIMEOUT_MS, read at
 * every call; see attn_check).
 * The scratch needed by a call (one error word, any problem size) is checked
 * against the array's 256 bytes; a call needing more returns
 * ATTN_ERR_INVALID_ARG.  All calls on a device share the array and it keeps the
 * last call's contents: each call clears its error word on `stream` first, and
 * calls whose kernels overlap on the GPU race on it.  The first call on a
 * device looks up the array's address with that device current; make it before
 * any stream capture on that device.
 */
int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int Sq, int Sk, int D, float scale, int causal,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                     int dtype, void* stream, int* device_status);

/*
 * attn_release -- free the library-owned per-device state of every device it
 * was created on: the device error word that attn_fwd, attn_fwd_window,
 * attn_fwd_decode, attn_merge, attn_bwd and attn_fwd_fp8 report into (see
 * attn_check), and the record of device pointers already checked.  Call only
 * when none of their launches is in flight.  Later calls recreate the state.
 */
int attn_release(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_TCGEN05_H */
