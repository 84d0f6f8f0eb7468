/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact attention forward and backward
 * passes.
 *
 * The operation is exact scaled-dot-product attention with the per-row
 * log-sum-exp, computed FlashAttention-style: tiles of Q stay on chip, K and
 * V stream through in tiles, and an online softmax keeps a running row max
 * and row sum so the L x L score matrix never reaches global memory.
 *
 *   Definition -- "FlashAttention 深度解析" (171host.com), first part,
 *     section 2.3: S = Q K^T, P = softmax(S), O = P V; scores are scaled
 *     before the softmax ("FlashAttention: как реально считается attention
 *     на GPU", section "Формулы online softmax").
 *   Algorithm -- "04 Transformers, Attention, and FlashAttention", Algorithm 1
 *     (FlashAttention-2 forward): Q split into row blocks, K/V into column
 *     blocks; per block the running max m, running sum l and unnormalised O
 *     are updated; O / l and L = m + log l are written at the end (steps
 *     12-15).  Causal masking keeps key <= query and skips blocks wholly
 *     above the diagonal ("FlashAttention 深度解析", second part, section 2.3).
 *
 * All entry points are plain C, take raw pointers and sizes, and never
 * allocate memory.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA runtime stream (same type as cudaStream_t); NULL = legacy default. */
typedef struct CUstream_st *fa_stream_t;

/* Status codes returned by every entry point. */
enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,   /* null pointer, B/H/L < 1, causal not 0/1,
                               non-finite scale, or sizes beyond int32 grid /
                               tensor-map limits                          */
  FA_ERR_UNSUPPORTED_D = 2, /* head dimension d other than 64 or 128      */
  FA_ERR_MISALIGNED = 3,    /* q, k, v or o not 16-byte aligned, or lse
                               not 4-byte aligned                         */
  FA_ERR_DEVICE = 4,        /* no usable CUDA device, or the current device
                               is not compute capability 10.3 (sm_103a)   */
  FA_ERR_LAUNCH = 5,        /* a CUDA runtime call or the launch failed   */
  FA_ERR_TIMEOUT = 6        /* a kernel's bounded wait gave up (reported by
                               fa_device_status, never by fa_fwd itself)  */
};

/*
 * fa_fwd -- exact attention forward on the current CUDA device.
 *
 *   q, k, v : device pointers, bf16, shape [B, H, L, d], row-major and
 *             contiguous (element (b,h,i,t) at ((b*H + h)*L + i)*d + t);
 *             16-byte aligned.  Read only.
 *   o       : device pointer, bf16 [B, H, L, d], same layout; 16-byte
 *             aligned.  Fully overwritten with
 *               o[b,h,i,:] = sum_j softmax_j(scale * q_i . k_j) v_j
 *             over the allowed keys j (all j < L; j <= i when causal),
 *             rounded to bf16 (nearest even).
 *   lse     : device pointer, fp32 [B, H, L]; 4-byte aligned.  Fully
 *             overwritten with log(sum_j exp(scale * q_i . k_j)) over the
 *             allowed keys (natural log of the scaled scores).
 *   B, H, L : batch, heads, sequence length (>= 1; queries and keys share L).
 *   d       : head dimension, 64 or 128.
 *   scale   : multiplier of q.k before the softmax (finite; 0 and negative
 *             values are allowed).
 *   causal  : 0 = every key; 1 = key index <= query index.
 *   stream  : stream the kernel is launched on.
 *
 * The caller owns every buffer; o and lse must not overlap q, k or v.  The
 * call is asynchronous on `stream`.  On any validation error it returns the
 * status without launching and without touching o or lse.  Arithmetic: bf16
 * operands, fp32 accumulation of both products, fp32 softmax statistics.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
           int L, int d, float scale, int causal, fa_stream_t stream);

/*
 * fa_fwd_splitkv -- the same result as fa_fwd, computed in key splits and
 * merged (Flash-Decoding: "04 Transformers, Attention, and FlashAttention",
 * section on Flash-Decoding -- split K/V into chunks, attend to each chunk
 * in parallel, combine the chunk results).  Worth it when B * H * ceil(L/256)
 * is small next to the number of SMs (few heads, long sequences).
 *
 *   q..causal : as for fa_fwd.
 *   n_splits  : requested number of key splits, 1..64.  The kernel uses
 *               min(n_splits, ceil(L/128)) splits of whole 128-key blocks.
 *   workspace : device scratch owned by the caller, 256-byte aligned, at
 *               least fa_splitkv_workspace_bytes(B, H, L, d, n_splits)
 *               bytes.  It receives the per-split fp32 partial O and LSE;
 *               its contents on entry do not matter and are undefined after.
 *   workspace_bytes : size of that buffer.
 *
 * Split s of row i holds O_s, normalised over the split's keys, and LSE_s;
 * the merge writes LSE = log sum_s exp(LSE_s) and O = sum_s exp(LSE_s - LSE)
 * O_s (bf16, round to nearest even).  Two kernels are launched on `stream`:
 * the split pass and the merge; calls that share a workspace on concurrent
 * streams race.  Errors: those of fa_fwd, plus FA_ERR_INVALID_ARG for
 * n_splits outside 1..64, a null workspace or one smaller than required,
 * and FA_ERR_MISALIGNED for a workspace not 256-byte aligned.
 */
int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                   int H, int L, int d, float scale, int causal, int n_splits, void *workspace,
                   size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_splitkv_workspace_bytes -- bytes of workspace fa_fwd_splitkv needs for
 * these sizes: 256-byte-aligned room for fp32 partial O [S, B, H, L, d]
 * followed by fp32 partial LSE [S, B, H, L], where S is the split count the
 * call actually uses: n_splits capped at the number of 128-key blocks
 * ceil(L / 128), then reduced so that no split is left without a block.
 * Returns 0 for invalid sizes (B/H/L < 1, d not 64/128, n_splits outside
 * 1..64).  Host only; no CUDA call.
 */
size_t fa_splitkv_workspace_bytes(int B, int H, int L, int d, int n_splits);

/*
 * fa_splitkv_splits -- the split count this library recommends for
 * fa_fwd_splitkv on these sizes: as many splits as fit the single-pass
 * CTAs (one per 256 query rows of a head) into one wave over `num_sms`
 * SMs, two waves when causal (the causal CTAs of a head differ in cost, so
 * splitting the longest shortens the launch even past one wave), and at
 * least 1, at most min(64, ceil(L / 128)).  A result of 1 means the
 * single pass (fa_fwd) fills the GPU by itself.  Measured on GB300 (152
 * SMs), one split more than this puts a few CTAs in an extra wave and
 * costs 20-35%.
 *
 *   num_sms : SMs of the target GPU; <= 0 queries the current device (the
 *             only case that makes a CUDA call).
 *
 * Returns 0 for invalid sizes (B/H/L < 1, d not 64/128, causal not 0/1) or
 * when the device query fails.
 */
int fa_splitkv_splits(int B, int H, int L, int d, int causal, int num_sms);

/*
 * FA_STATIC_WORKSPACE_BYTES -- size of the split-KV scratch array the library
 * keeps in device memory for fa_fwd_splitkv_static (64 MiB, held on every
 * GPU that loads the library until the process exits).
 */
#define FA_STATIC_WORKSPACE_BYTES ((size_t)64 << 20)

/*
 * fa_fwd_splitkv_static -- fa_fwd_splitkv for callers that cannot allocate
 * device memory (an engine or plugin host that owns the whole memory budget
 * and gives out no scratch): it takes no workspace and calls no allocation
 * routine; its scratch is the library's own FA_STATIC_WORKSPACE_BYTES array.
 * The paper has no counterpart to this entry point: it exists only for
 * callers that cannot hand the library scratch memory.
 *
 *   q..n_splits, stream : as for fa_fwd_splitkv.
 *
 * Returns FA_ERR_INVALID_ARG, launching nothing, when
 * fa_splitkv_workspace_bytes(B, H, L, d, n_splits) exceeds
 * FA_STATIC_WORKSPACE_BYTES (fewer splits, or fa_fwd, then apply), and
 * otherwise the statuses of fa_fwd_splitkv.  The first call on a device looks
 * up the array's address on that device (with it current) and keeps it for
 * the life of the process; make that first call before any stream capture.
 * The address belongs to the device's current context: after the context is
 * destroyed (cudaDeviceReset) the kept address is stale, so do not call this
 * entry point again in that process.  Every call uses the same array and
 * finds it as the previous call left it (nothing in it needs to start at
 * zero), so calls that overlap on the GPU -- on different streams, or from
 * different host threads -- race.
 */
int fa_fwd_splitkv_static(const void *q, const void *k, const void *v, void *o, float *lse,
                          int B, int H, int L, int d, float scale, int causal, int n_splits,
                          fa_stream_t stream);

/*
 * fa_fwd_host_workspace_bytes -- device workspace fa_fwd_host needs: room for
 * device copies of Q, K, V and O (bf16, back to back) and LSE (fp32),
 * 256-byte aligned.  Returns 0 for invalid sizes.  Host only.
 */
size_t fa_fwd_host_workspace_bytes(int B, int H, int L, int d);

/*
 * fa_fwd_host -- fa_fwd on HOST buffers: copies q, k, v to the device,
 * runs the forward, copies o and lse back, all asynchronous on `stream`.
 *
 *   q, k, v : host bf16 [B, H, L, d] (layout as for fa_fwd).  Inputs that lie
 *             back to back in host memory (k == q + size, v == k + size)
 *             travel in one copy.
 *   o, lse  : host outputs; o and lse back to back travel in one copy.
 *   workspace : device scratch of fa_fwd_host_workspace_bytes(B, H, L, d)
 *             bytes or more, 256-byte aligned; its contents on entry do not
 *             matter.
 *   other arguments as for fa_fwd.
 *
 * For the copies to be asynchronous (and to overlap with other work) the
 * host buffers must be page-locked; pageable buffers work but the copies
 * then block the calling thread.  The outputs are valid once `stream` has
 * reached the end of the call.  Calls on different streams with different
 * workspaces may overlap (one call's copies with another's kernel); calls
 * sharing a workspace on concurrent streams race.  Errors: those of fa_fwd,
 * plus FA_ERR_INVALID_ARG for a null or too-small workspace and
 * FA_ERR_MISALIGNED for a workspace not 256-byte aligned; nothing is copied
 * or launched on a validation error.
 */
int fa_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                int L, int d, float scale, int causal, void *workspace, size_t workspace_bytes,
                fa_stream_t stream);

/*
 * fa_quantize_fp8 -- FP8 (E4M3) block quantisation of Q or K for
 * fa_fwd_fp8 ("FlashAttention 深度解析", third part, section 2.3: each block
 * gets s = max|block| / FP8_MAX and is stored as Quantize(block / s)).
 *
 *   x      : device bf16 [B, H, L, d], layout as for fa_fwd; 16-byte aligned.
 *   codes  : device output, one byte per element [B, H, L, d] (E4M3: sign,
 *            4 exponent bits with bias 7, 3 mantissa bits); 16-byte aligned.
 *   scales : device output fp32 [B, H, ceil(L / 128)]: the scale of each
 *            block of 128 consecutive rows of a head, amax / 448 (correctly
 *            rounded fp32 division), or 1 for a block of zeros.
 *
 * codes = x / s (correctly rounded fp32 division), rounded to the nearest
 * E4M3 value (ties to even) and saturated to +-448.  Asynchronous on
 * `stream`; errors as for fa_fwd (d = 64 or 128); nothing is launched on an
 * error.
 */
int fa_quantize_fp8(const void *x, void *codes, float *scales, int B, int H, int L, int d,
                    fa_stream_t stream);

/*
 * fa_fwd_fp8 -- fa_fwd with Q and K in FP8: S = (Q_FP8 K_FP8^T) * s_q * s_k
 * * scale (the same page and section), P and V in bf16 as in fa_fwd.
 *
 *   q8, k8          : E4M3 codes and their block scales from fa_quantize_fp8
 *   q_scale, k_scale  (codes 16-byte aligned, scales 4-byte aligned).
 *   v, o, lse, B..causal, stream : as for fa_fwd.
 *
 * The S product runs on the 8-bit tensor-core path (tcgen05 kind::f8f6f4,
 * fp32 accumulation); s_q * s_k join the softmax's scale per block.  The
 * result is exact attention of the de-quantised Q and K (codes times their
 * block scale) with V, within the tolerances of fa_fwd.  Errors: those of
 * fa_fwd, plus FA_ERR_INVALID_ARG / FA_ERR_MISALIGNED for the scale arrays.
 */
int fa_fwd_fp8(const void *q8, const void *k8, const void *v, const float *q_scale,
               const float *k_scale, void *o, float *lse, int B, int H, int L, int d,
               float scale, int causal, fa_stream_t stream);

/*
 * fa_bwd_workspace_bytes -- bytes of workspace fa_bwd needs for these sizes:
 * 256-byte-aligned room for an fp32 dQ accumulator [B, H, L, d], two fp32
 * per-query arrays [B, H, Lp] (Lp = L rounded up to a multiple of 128) and
 * 256 bytes for the gradient kernel's work counter.  Returns 0 for invalid
 * sizes (B/H/L < 1, d not 64/128).  Host only.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int L, int d);

/*
 * fa_bwd -- gradients of exact attention (the backward pass by
 * recomputation): given the forward's inputs, its outputs o and lse, and the
 * gradient dout of a loss with respect to o, write the gradients with
 * respect to q, k and v.
 *
 *   The formulas are those of "FlashAttention 深度解析", first part, section
 *   4.1 (dV = P^T dO; dP = dO V^T; dS = P (.) (dP - rowsum(dP (.) P))) with
 *   the chain rule through the scaled scores (dQ = scale dS K, dK = scale
 *   dS^T Q).  P is recomputed block by block from q, k and lse, never stored
 *   (section 4.2, 重计算策略); rowsum(dP (.) P) is computed as <dO_i, O_i>,
 *   equal to it because O = P V.
 *
 *   q, k, v, o, dout : device bf16 [B, H, L, d], layout as for fa_fwd,
 *               16-byte aligned; o is fa_fwd's output for q, k, v, scale,
 *               causal.  Read only.
 *   lse       : device fp32 [B, H, L], fa_fwd's log-sum-exp for the same
 *               call; 4-byte aligned.  Read only.
 *   dq, dk, dv: device bf16 [B, H, L, d], 16-byte aligned, fully overwritten
 *               (round to nearest even from fp32 accumulators).
 *   B..causal : as for fa_fwd (d = 64 or 128).
 *   workspace : device scratch owned by the caller, 256-byte aligned, at
 *               least fa_bwd_workspace_bytes(B, H, L, d) bytes; contents on
 *               entry do not matter and are undefined after.
 *
 * The caller owns every buffer; dq, dk, dv and workspace must not overlap
 * each other or the inputs.  Three kernels are launched on `stream` (a
 * per-row pre-pass, the gradient kernel, a dQ conversion pass); calls that
 * share a workspace on concurrent streams race.  Arithmetic: bf16 operands
 * (P and dS rounded to bf16 before their products), fp32 accumulation, dQ
 * summed over key blocks with fp32 atomic adds, so its last bits may differ
 * from run to run.  Errors: those of fa_fwd, plus FA_ERR_INVALID_ARG for a
 * null or too-small workspace and FA_ERR_MISALIGNED for a workspace that is
 * not 256-byte aligned; nothing is launched on an error.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
           const float *lse, void *dq, void *dk, void *dv, int B, int H, int L, int d,
           float scale, int causal, void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_device_status -- synchronise `stream` and report whether any kernel of
 * this library on the current device gave up a bounded wait since the status
 * was last cleared (FA_ERR_TIMEOUT) or FA_OK.  A nonzero `clear` resets the
 * status afterwards.  Returns FA_ERR_LAUNCH if the synchronisation fails.
 */
int fa_device_status(fa_stream_t stream, int clear);

/*
 * fa_set_wait_timeout_ns -- time limit of every wait inside the kernels
 * (default 1e9 ns).  A wait that exceeds it makes the kernel record
 * FA_ERR_TIMEOUT, drain its own copies, free its tensor memory and return.
 * Values below 1000 ns are raised to 1000 ns.  Process-wide; not thread-safe
 * against concurrent fa_fwd calls.
 */
void fa_set_wait_timeout_ns(uint64_t ns);

/*
 * fa_test_withhold_q_load -- test hook for the timeout path.  While enabled
 * (nonzero), the forward kernels launched afterwards skip their Q copy and
 * the backward kernel its K/V copy, so the first wait on that copy never
 * completes: it gives up after the wait limit, every role stops and drains,
 * the tensor memory is freed and fa_device_status reports FA_ERR_TIMEOUT.
 * Outputs of such launches are undefined.  Process-wide; leave at 0 outside
 * such tests.
 */
void fa_test_withhold_q_load(int enable);

/* Human-readable text for a status code (static storage, never NULL). */
const char *fa_status_string(int status);

/* ABI version of this library (major * 10000 + minor * 100 + patch). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
