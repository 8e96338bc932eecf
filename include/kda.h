/*
 * kda.h -- C ABI of libkda, the GB300 (sm_103a) Kimi / Kernel Delta Attention forward.
 *
 * KDA keeps, per (sequence, head), an fp32 memory S of shape [dk, dv] (rows = key
 * channels, columns = value channels).  For each token, with
 *     k^    = k / sqrt(|k|^2 + 1e-6)                  (L2 norm over dk)
 *     q^    = scale * q / sqrt(|q|^2 + 1e-6)
 *     gamma = lower_bound * sigmoid(exp(a_log[h]) * (g + dt_bias[:, h]))   (per channel, <= 0)
 *     beta  = sigmoid(beta_logit)
 * the memory is first decayed, S' = diag(exp(gamma)) S, then receives the delta-rule
 * write S = S' + k^ (beta (v - S'^T k^))^T, and the token emits o = S^T q^.
 *   - recurrence: ejkernel "kernel_delta_attention" module page, "The core recurrence"
 *     (the error term is taken against the decayed memory: decay first, then write);
 *   - gate / beta / scale / in-place state: NKI "KDA TKG Kernel API Reference", kda_tkg
 *     parameters q, k, v, g, beta, a_log, dt_bias, out, S, scale, lower_bound;
 *   - chunked / state passthrough: kernel_delta_attention page, "Algorithm modes" and the
 *     chunk_size / initial_state / return_state parameters;
 *   - packed sequences: ejkernel "recurrent" module page, cu_seqlens parameter.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers of the current CUDA device, dense (row-major,
 *     no padding) and 16-byte aligned.  The caller allocates every buffer, outputs
 *     included; the library allocates nothing and keeps no state between calls (the one
 *     exception is the fixed scratch array behind kda_chunk_fwd_noalloc).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and
 *     the call returns without synchronising.  Inputs must stay valid until the stream
 *     reaches the launch.
 *   - Head dimensions dk, dv must each be 32, 64 or 128 (kda_tkg: dk <= 128).
 *   - lower_bound must lie in [-5, 0] (kda_tkg lower_bound): then exp(gamma) is in (0, 1]
 *     and the kernels' factorised gate exponentials stay inside the fp32 range.
 *   - scale <= 0 selects the default dk^-0.5 (kernel_delta_attention: softmax_scale None).
 *   - Return value: KDA_OK (0) or a negative kda_status.  Argument errors are detected on
 *     the host before anything is enqueued; KDA_ERR_LAUNCH reports cudaGetLastError()
 *     after the launch.  Errors never abort the process.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t (struct CUstream_st*); NULL is the legacy default stream. */
typedef struct CUstream_st* kda_stream_t;

/* Element type of q, k, v and out in the chunked entry points. */
enum kda_dtype {
  KDA_F32 = 0,  /* fp32 q/k/v/out */
  KDA_BF16 = 1  /* bf16 q/k/v/out (fp32 accumulation, fp32 state) */
};

enum kda_status {
  KDA_OK = 0,
  KDA_ERR_NULL_POINTER = -1,    /* a required pointer is NULL */
  KDA_ERR_BAD_SHAPE = -2,       /* a size is negative / zero where it must be positive */
  KDA_ERR_HEAD_DIM = -3,        /* dk or dv not in {32, 64, 128} */
  KDA_ERR_CHUNK = -4,           /* chunk not in {16, 64} */
  KDA_ERR_LOWER_BOUND = -5,     /* lower_bound outside [-5, 0] or not finite */
  KDA_ERR_MISALIGNED = -6,      /* a pointer is not 16-byte aligned */
  KDA_ERR_DTYPE = -7,           /* dtype not a kda_dtype */
  KDA_ERR_LAUNCH = -8,          /* the CUDA launch failed (cudaGetLastError) */
  KDA_ERR_DEVICE = -9,          /* no usable device / not a compute capability 10.3 GPU */
  KDA_ERR_SCALE = -10,          /* scale is NaN or infinite */
  KDA_ERR_TOO_LARGE = -11,      /* an index would overflow the kernels' 64-bit limits */
  KDA_ERR_WORKSPACE = -12,      /* workspace NULL, too small or not 256-byte aligned */
  KDA_ERR_FLAGS = -13           /* unknown bits in a flags argument */
};

/*
 * kda_chunk_fwd -- whole-sequence chunked forward for B equal-length sequences.
 *   kernel_delta_attention.run / kda_attention (query, key, value, beta, decay,
 *   initial_state, softmax_scale, chunk_size, return_state), with the per-channel raw gate
 *   and beta logits of kda_tkg in place of the pre-activated per-head decay and beta.
 *
 *   q, k        [B, T, H, dk]   dtype (fp32 or bf16), raw (normalised inside)
 *   v           [B, T, H, dv]   dtype
 *   g           [B, T, H, dk]   fp32, raw per-channel gate
 *   beta_logits [B, T, H]       fp32
 *   a_log       [H]             fp32 (kda_tkg's [1, H])
 *   dt_bias     [dk, H]         fp32 (kda_tkg layout)
 *   initial_state [B, H, dk, dv] fp32, or NULL for zeros
 *   out         [B, T, H, dv]   dtype, written
 *   final_state [B, H, dk, dv]  fp32, written; NULL if not wanted.  May alias initial_state
 *                               (the state is then advanced in place).
 *   chunk       16 or 64: tokens per chunk of the chunked algorithm ("chunk_size").  The
 *               result does not depend on it beyond rounding.
 *   T == 0 is allowed: out is untouched and final_state receives initial_state (or zeros).
 */
int kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                  const float* beta_logits, const float* a_log, const float* dt_bias,
                  float scale, float lower_bound, const float* initial_state, void* out,
                  float* final_state, int B, int T, int H, int dk, int dv, int chunk,
                  int dtype, kda_stream_t stream);

/*
 * kda_chunk_fwd_varlen -- the same forward over N sequences packed along the token axis
 *   (recurrent page, cu_seqlens: cumulative sequence lengths, [N + 1]).
 *
 *   q, k, g     [total_T, H, dk]; v, out [total_T, H, dv]; beta_logits [total_T, H]
 *   cu_seqlens  [N + 1] int32 DEVICE array: cu_seqlens[0] = 0, non-decreasing,
 *               cu_seqlens[N] = total_T.  Sequence n owns tokens
 *               [cu_seqlens[n], cu_seqlens[n + 1]) and starts from initial_state[n].
 *               The kernels clamp every entry into [0, total_T], so a malformed array
 *               gives wrong numbers but no out-of-bounds access.
 *   initial_state, final_state [N, H, dk, dv] fp32 (same NULL / aliasing rules as above).
 *   Empty sequences are allowed (their final state is their initial state).
 */
int kda_chunk_fwd_varlen(const void* q, const void* k, const void* v, const float* g,
                         const float* beta_logits, const float* a_log, const float* dt_bias,
                         float scale, float lower_bound, const int32_t* cu_seqlens, int N,
                         int total_T, const float* initial_state, void* out,
                         float* final_state, int H, int dk, int dv, int chunk, int dtype,
                         kda_stream_t stream);

/*
 * Workspace variants of the two chunked entry points.  For bf16 q/k/v with dk = dv = 128
 * and chunk = 64 they run the forward in two launches: every chunk's state-independent
 * part (gates, norms, the gate-scaled products, the UT solve and transform; the
 * kernel_delta_attention page's "parallel within chunks") for all chunks of all sequences
 * at once, then the sequential pass over the state, which reads one workspace record per
 * (chunk, head).  The results equal those of kda_chunk_fwd / kda_chunk_fwd_varlen up to
 * rounding.  For every other configuration the workspace is not used and the call runs the
 * same kernels as the entry point without it.
 *
 *   kda_chunk_fwd_workspace_size / kda_chunk_fwd_varlen_workspace_size
 *       bytes of device workspace the matching call needs (0: none).  About 74 KB per
 *       (64-token chunk, head): 612 MB for B = 4, T = 4096, H = 32.  The varlen size is an
 *       upper bound from total_T and N (every sequence may end in a partial chunk), plus
 *       the room to split the scans of up to 8 long sequences: a sequence's chunks form a
 *       chain of affine state maps (S' = A S + B per chunk), and a long chain is cut in two
 *       whose second half runs from zero beside a third chain from the identity, then
 *       corrected by the first half's end state (three fp32 [128 x 128] states per split
 *       sequence and head, and a bf16 [total_T, H, 128] buffer).
 *   workspace       DEVICE buffer of at least that many bytes, 256-byte aligned, owned by
 *                   the caller; its contents on entry are irrelevant and on return are
 *                   unspecified.  It must not be used by anything else until the stream
 *                   has passed the call.  May be NULL when the size is 0.
 *   workspace_bytes its size; a smaller or misaligned buffer gives KDA_ERR_WORKSPACE.
 * All other arguments, layouts and errors are those of kda_chunk_fwd / _varlen.
 */
size_t kda_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, int chunk, int dtype);
size_t kda_chunk_fwd_varlen_workspace_size(int N, int total_T, int H, int dk, int dv,
                                           int chunk, int dtype);
int kda_chunk_fwd_ws(const void* q, const void* k, const void* v, const float* g,
                     const float* beta_logits, const float* a_log, const float* dt_bias,
                     float scale, float lower_bound, const float* initial_state, void* out,
                     float* final_state, int B, int T, int H, int dk, int dv, int chunk,
                     int dtype, void* workspace, size_t workspace_bytes, kda_stream_t stream);
int kda_chunk_fwd_varlen_ws(const void* q, const void* k, const void* v, const float* g,
                            const float* beta_logits, const float* a_log,
                            const float* dt_bias, float scale, float lower_bound,
                            const int32_t* cu_seqlens, int N, int total_T,
                            const float* initial_state, void* out, float* final_state, int H,
                            int dk, int dv, int chunk, int dtype, void* workspace,
                            size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_fwd_noalloc -- kda_chunk_fwd_ws with the workspace taken from a scratch array
 *   that the library keeps in device memory (KDA_NOALLOC_SCRATCH_BYTES per device), so the
 *   caller passes none.  It is meant for callers that cannot call cudaMalloc themselves
 *   (an allocator that owns all device memory, code running inside a captured or
 *   pre-planned execution that forbids allocation).  It has no counterpart on the source
 *   pages: an interface convenience over the workspace entry point.
 *   Arguments, layouts and results are those of kda_chunk_fwd.  Errors are those of
 *   kda_chunk_fwd, checked in the same order; a configuration whose arguments are valid but
 *   whose workspace (kda_chunk_fwd_workspace_size) exceeds the array is then rejected with
 *   KDA_ERR_WORKSPACE, before anything is enqueued.  The array is shared by every call on
 *   a device and keeps the last call's contents: calls must not overlap in time (issue them
 *   on one stream, or synchronise between streams); overlapping calls race.
 *   Set-up: the array's device address is looked up once per CUDA context, by the first
 *   call made with that context current (a context that replaces one destroyed by
 *   cudaDeviceReset gets its own lookup); make that first call before any stream capture.
 *   Under lazy module loading (the CUDA default) the array's device memory is reserved by
 *   that first call; with CUDA_MODULE_LOADING=EAGER every context that loads the library
 *   reserves it at start-up.  Either way it is held until the process exits.
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)256 << 20)
int kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                          const float* beta_logits, const float* a_log, const float* dt_bias,
                          float scale, float lower_bound, const float* initial_state, void* out,
                          float* final_state, int B, int T, int H, int dk, int dv, int chunk,
                          int dtype, kda_stream_t stream);

/*
 * kda_chunk_bwd -- gradients of the kda_chunk_fwd forward (fixed-length sequences, decay
 *   first) for L = <d_out, out> + <d_final_state, final_state>.  The pages give no backward
 *   pass (the kernel_delta_attention page presents the chunked mode as the training path):
 *   this is reverse-mode differentiation of the recurrence.  For bf16 with dk = dv = 128 it
 *   runs on the chunk form (64-token chunks, tensor cores): the forward's chunk records
 *   and per-chunk states, a reverse scan over chunks carrying the state's adjoint, and one
 *   pass over all (chunk, head) pairs for the remaining products and the norm, sigmoid and
 *   gate chain rules.  Other shapes and fp32 differentiate token by token: a forward scan
 *   that checkpoints the state every 64 tokens, a reverse scan that recomputes each
 *   chunk's states from its checkpoint, and an elementwise pass for the chain rules.
 *
 *   Inputs: those of kda_chunk_fwd (q, k, v, g, beta_logits, a_log, dt_bias, scale,
 *   lower_bound, initial_state; same layouts, dtype for q/k/v) and
 *     d_out          [B, T, H, dv]   dtype, the output cotangent
 *     d_final_state  [B, H, dk, dv]  fp32 or NULL (zero)
 *   Outputs (caller-allocated, fully written):
 *     dq, dk         [B, T, H, dk]   dtype          dv  [B, T, H, dv] dtype
 *     dg             [B, T, H, dk]   fp32           dbeta_logits [B, T, H] fp32
 *     da_log         [H] fp32        ddt_bias       [dk, H] fp32   (sums over B and T)
 *     d_initial_state [B, H, dk, dv] fp32 or NULL (not wanted)
 *   dim_k, dim_v   the head dimensions dk, dv (named apart from the dk / dv gradients)
 *   workspace / workspace_bytes: device scratch of at least
 *   kda_chunk_bwd_workspace_size(B, T, H, dk, dv, dtype) bytes, 256-byte aligned (chunk
 *   records and bf16 states and adjoints per (chunk, head) on the tensor-core path;
 *   checkpoints, one chunk of states per (sequence, head) and per-token fp32 intermediates
 *   otherwise).  0 is returned for unsupported arguments.
 */
size_t kda_chunk_bwd_workspace_size(int B, int T, int H, int dk, int dv, int dtype);
int kda_chunk_bwd(const void* q, const void* k, const void* v, const float* g,
                  const float* beta_logits, const float* a_log, const float* dt_bias,
                  float scale, float lower_bound, const float* initial_state, const void* d_out,
                  const float* d_final_state, void* dq, void* dk, void* dv, float* dg,
                  float* dbeta_logits, float* da_log, float* ddt_bias, float* d_initial_state,
                  int B, int T, int H, int dim_k, int dim_v, int dtype, void* workspace,
                  size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_bwd_varlen -- kda_chunk_bwd for packed sequences (the cu_seqlens convention of
 *   kda_chunk_fwd_varlen): q, k, g, d_out, dq, dk, dg [total_T, H, dk], v, dv [total_T, H, dv],
 *   beta_logits, dbeta_logits [total_T, H]; initial_state, d_final_state, d_initial_state
 *   [N, H, dk, dv] (each nullable as in kda_chunk_bwd); da_log [H] and ddt_bias [dk, H] sum
 *   over every sequence.  Each sequence is differentiated on its own (its own initial state
 *   and final-state cotangent).  Served on the tensor-core path only: bf16 q/k/v/d_out with
 *   dk = dv = 128 (others give KDA_ERR_DTYPE / KDA_ERR_HEAD_DIM).  workspace: at least
 *   kda_chunk_bwd_varlen_workspace_size(N, total_T, H, dk, dv, dtype) bytes (0 for an
 *   unsupported configuration), 256-byte aligned.
 */
size_t kda_chunk_bwd_varlen_workspace_size(int N, int total_T, int H, int dk, int dv,
                                          int dtype);
int kda_chunk_bwd_varlen(const void* q, const void* k, const void* v, const float* g,
                         const float* beta_logits, const float* a_log, const float* dt_bias,
                         float scale, float lower_bound, const int32_t* cu_seqlens, int N,
                         int total_T, const float* initial_state, const void* d_out,
                         const float* d_final_state, void* dq, void* dk, void* dv, float* dg,
                         float* dbeta_logits, float* da_log, float* ddt_bias,
                         float* d_initial_state, int H, int dim_k, int dim_v, int dtype,
                         void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_fwd_train_varlen / kda_chunk_bwd_saved_varlen -- the training pair below
 *   (kda_chunk_fwd_train, kda_chunk_bwd_saved) for packed sequences: the arguments of
 *   kda_chunk_fwd_varlen_ws and of kda_chunk_bwd_varlen, the workspace of
 *   kda_chunk_bwd_varlen_workspace_size(N, total_T, H, 128, 128, KDA_BF16).
 */
int kda_chunk_fwd_train_varlen(const void* q, const void* k, const void* v, const float* g,
                               const float* beta_logits, const float* a_log,
                               const float* dt_bias, float scale, float lower_bound,
                               const int32_t* cu_seqlens, int N, int total_T,
                               const float* initial_state, void* out, float* final_state, int H,
                               int dk, int dv, int chunk, int dtype, void* workspace,
                               size_t workspace_bytes, kda_stream_t stream);
int kda_chunk_bwd_saved_varlen(const void* q, const void* k, const void* v, const float* g,
                               const float* beta_logits, const float* a_log,
                               const float* dt_bias, float scale, float lower_bound,
                               const int32_t* cu_seqlens, int N, int total_T,
                               const float* initial_state, const void* d_out,
                               const float* d_final_state, void* dq, void* dk, void* dv,
                               float* dg, float* dbeta_logits, float* da_log, float* ddt_bias,
                               float* d_initial_state, int H, int dim_k, int dim_v, int dtype,
                               void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_fwd_train -- the forward of kda_chunk_fwd_ws (same inputs, outputs, layouts and
 *   error codes) for training: besides out and final_state it leaves in `workspace` the
 *   chunk records and per-chunk states that kda_chunk_bwd_saved reads, so that the backward
 *   does not recompute them.  No paper counterpart: the pages present the chunked mode as
 *   the training path and give no backward.  Serves bf16 q/k/v with dk = dv = 128 and
 *   chunk = 64 (fixed-length sequences); other dtypes, head dims or chunk sizes give
 *   KDA_ERR_DTYPE / KDA_ERR_HEAD_DIM / KDA_ERR_CHUNK (no tokens at all: the plain forward).
 *   workspace / workspace_bytes: at least kda_chunk_bwd_workspace_size(B, T, H, 128, 128,
 *   KDA_BF16) bytes, 256-byte aligned, caller-owned; what it holds stays valid for
 *   kda_chunk_bwd_saved until the caller reuses the buffer.  The output can differ from
 *   kda_chunk_fwd_ws's in the last bf16 bit (the query scale rides in the operands instead
 *   of the output).
 */
int kda_chunk_fwd_train(const void* q, const void* k, const void* v, const float* g,
                        const float* beta_logits, const float* a_log, const float* dt_bias,
                        float scale, float lower_bound, const float* initial_state, void* out,
                        float* final_state, int B, int T, int H, int dk, int dv, int chunk,
                        int dtype, void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_bwd_saved -- kda_chunk_bwd (same arguments, outputs and error codes) that reads
 *   the records and per-chunk states kda_chunk_fwd_train left in `workspace` for the same
 *   inputs instead of recomputing them (the workspace is also its scratch).  Only the
 *   configurations of kda_chunk_fwd_train (others give KDA_ERR_DTYPE / KDA_ERR_HEAD_DIM).
 *   On a workspace that kda_chunk_fwd_train did not fill for these inputs the gradients are
 *   wrong, though every access stays inside the workspace.
 */
int kda_chunk_bwd_saved(const void* q, const void* k, const void* v, const float* g,
                        const float* beta_logits, const float* a_log, const float* dt_bias,
                        float scale, float lower_bound, const float* initial_state,
                        const void* d_out, const float* d_final_state, void* dq, void* dk,
                        void* dv, float* dg, float* dbeta_logits, float* da_log, float* ddt_bias,
                        float* d_initial_state, int B, int T, int H, int dim_k, int dim_v,
                        int dtype, void* workspace, size_t workspace_bytes, kda_stream_t stream);

/* Options of kda_attention_fwd (bitwise OR). */
enum kda_attention_flags {
  KDA_ATTN_NO_QK_L2NORM = 1,  /* use_qk_l2norm=False: q and k are used as given */
  KDA_ATTN_RECURRENT = 2,     /* use_chunked=False: the token-by-token scan */
  KDA_ATTN_ORDER_LITERAL = 4  /* the error term reads the memory before the token's decay,
                                 as the printed recurrence has it (default: after) */
};

/*
 * kda_attention_fwd -- the kernel_delta_attention / kda_attention call of the ejkernel
 *   kernel_delta_attention page (parameters query, key, value, beta, decay, initial_state,
 *   softmax_scale, chunk_size, use_qk_l2norm, use_chunked, return_state), for B equal-length
 *   sequences:
 *
 *   query, key  [B, T, H, dk]   dtype (fp32 or bf16)
 *   value, out  [B, T, H, dv]   dtype
 *   beta        [B, T, H]       fp32: the per-token rate itself (not a logit)
 *   decay       [B, T, H]       fp32 per-head log-decay, the same for every key channel
 *                               (the page asks for values <= 0); NULL = no decay.  Values
 *                               must lie in [-5, 5] for the chunked algorithm's factorised
 *                               exponentials to stay in range.
 *   initial_state / final_state [B, H, dk, dv] fp32, as for kda_chunk_fwd
 *   softmax_scale  multiplies q (after its L2 norm when that is on); <= 0 selects dk^-0.5
 *   chunk       16 or 64 (chunked mode; results do not depend on it beyond rounding)
 *   flags       kda_attention_flags; unknown bits give KDA_ERR_FLAGS
 *   The recurrence is kda_chunk_fwd's with gamma = decay[t, h] on every channel and beta
 *   taken as given.  Runs on the fp32 SIMT kernels (chunked, 16-token chunks, or the
 *   sequential scan); kda_attention_fwd_ws below runs the bf16 dk = dv = 128 chunked call on
 *   the tensor cores.
 */
int kda_attention_fwd(const void* query, const void* key, const void* value, const float* beta,
                      const float* decay, const float* initial_state, void* out,
                      float* final_state, float softmax_scale, int B, int T, int H, int dk,
                      int dv, int chunk, int flags, int dtype, kda_stream_t stream);

/*
 * kda_attention_fwd_workspace_size / kda_attention_fwd_ws -- kda_attention_fwd through a
 *   caller workspace (same arguments, layouts, results and errors, plus the workspace).  For
 *   bf16 with dk = dv = 128, chunk = 64 and the chunked mode (no KDA_ATTN_RECURRENT) it runs
 *   on the two-launch tensor-core path of kda_chunk_fwd_ws -- every chunk's
 *   state-independent part for all chunks at once, then the sequential pass over the state
 *   (kernel_delta_attention page, "Algorithm modes": chunked, parallel within chunks) --
 *   with the call's own variants: the per-head log-decay on every channel, beta as given,
 *   use_qk_l2norm and the literal order.  On that path the decay must lie in [-5, 1] (the
 *   page asks for decays <= 0): 64-token chunks keep their factorised exponentials inside
 *   the fp32 range only there; outside it the results are unspecified (no fault), and
 *   decays far enough outside to overflow a sub-chunk's factors set bit 5 of
 *   kda_device_error.  Every
 *   other configuration ignores the workspace and runs kda_attention_fwd's kernels.
 *   workspace: at least kda_attention_fwd_workspace_size(B, T, H, dk, dv, chunk, flags,
 *   dtype) bytes (0: none needed), 256-byte aligned, caller-owned, contents unspecified on
 *   return; a smaller or misaligned buffer gives KDA_ERR_WORKSPACE.
 */
size_t kda_attention_fwd_workspace_size(int B, int T, int H, int dk, int dv, int chunk,
                                        int flags, int dtype);
int kda_attention_fwd_ws(const void* query, const void* key, const void* value,
                         const float* beta, const float* decay, const float* initial_state,
                         void* out, float* final_state, float softmax_scale, int B, int T, int H,
                         int dk, int dv, int chunk, int flags, int dtype, void* workspace,
                         size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_recurrent_attention_fwd -- the recurrent_attention call of the ejkernel "recurrent"
 *   page: a gated linear recurrence per (sequence, query head), token by token.  The page
 *   names the gates but prints no formula; the reading implemented is (all gates are
 *   log-space decays, each term only when its pointer is non-NULL)
 *       a_t = g_t + gk_t + g_gamma           (per key channel)
 *       h_t = diag(exp(a_t)) h_{t-1} diag(exp(gv_t)) + k_t v_t^T,   o_t = h_t^T (scale q_t)
 *
 *   query, out   [B, T, Hq, D]    dtype (fp32 or bf16)
 *   key, value   [B, T, Hkv, D]   dtype; query head h reads kv head h / (Hq / Hkv)
 *   g, gk, gv    [B, T, Hq, D]    fp32 or NULL
 *   g_gamma      [B, Hq]          fp32 or NULL
 *   initial_state / final_state [nseq, Hq, D, D] fp32 (NULL: zeros / not wanted)
 *   softmax_scale  multiplies q; <= 0 selects D^-0.5
 *   cu_seqlens   NULL for B sequences of T tokens (nseq = B); otherwise [N + 1] int32
 *                DEVICE offsets of N packed sequences, B must be 1 and T is the packed
 *                token count (nseq = N); entries are clamped into [0, T]
 *   reverse      non-zero: each sequence is processed from its last token to its first
 *   D in {32, 64, 128}; Hq a multiple of Hkv.
 */
int kda_recurrent_attention_fwd(const void* query, const void* key, const void* value,
                                const float* g, const float* g_gamma, const float* gk,
                                const float* gv, float softmax_scale, const float* initial_state,
                                void* out, float* final_state, const int32_t* cu_seqlens, int N,
                                int B, int T, int Hq, int Hkv, int D, int reverse, int dtype,
                                kda_stream_t stream);

/* Shape options of kda_recurrent_attention_fwd_workspace_size (bitwise OR). */
enum kda_recurrent_flags {
  KDA_REC_PACKED = 1,      /* cu_seqlens given: N packed sequences, B = 1, T = packed tokens */
  KDA_REC_VALUE_GATE = 2,  /* gv given */
  KDA_REC_REVERSE = 4      /* reverse != 0 */
};

/*
 * kda_recurrent_attention_fwd_workspace_size / kda_recurrent_attention_fwd_ws --
 *   kda_recurrent_attention_fwd through a caller workspace (same arguments, layouts, results
 *   and errors, plus the workspace).  For bf16 with D = 128 it runs the recurrence in its
 *   chunked form on the tensor cores (64-token chunks: every chunk's gate-scaled product
 *   q k^T and its records at once, then the sequential pass over the state; the recurrent
 *   page's run parameters g, gk, g_gamma, gv, cu_seqlens, reverse).  On that path the summed
 *   key-axis gate g + gk + g_gamma and the value-axis gate gv must each lie in [-5, 1] at
 *   every token and channel, where the chunks' factorised exponentials stay inside the fp32
 *   range; outside it the results are unspecified (no fault), and gates far enough outside
 *   to overflow a sub-chunk's factors set bit 5 of kda_device_error.  Every other configuration
 *   (fp32, other head dims) ignores the workspace and runs the token-serial kernel.
 *   workspace: at least kda_recurrent_attention_fwd_workspace_size(N, B, T, Hq, Hkv, D,
 *   flags, dtype) bytes (flags: kda_recurrent_flags describing the call; 0: none needed),
 *   256-byte aligned, caller-owned, contents unspecified on return; a smaller or misaligned
 *   buffer gives KDA_ERR_WORKSPACE.  About 41 KB per (64-token chunk, query head), 91 KB
 *   with a value-axis gate or in reverse order.
 */
size_t kda_recurrent_attention_fwd_workspace_size(int N, int B, int T, int Hq, int Hkv, int D,
                                                  int flags, int dtype);
int kda_recurrent_attention_fwd_ws(const void* query, const void* key, const void* value,
                                   const float* g, const float* g_gamma, const float* gk,
                                   const float* gv, float softmax_scale,
                                   const float* initial_state, void* out, float* final_state,
                                   const int32_t* cu_seqlens, int N, int B, int T, int Hq,
                                   int Hkv, int D, int reverse, int dtype, void* workspace,
                                   size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_decode_step -- advance the recurrence by exactly one token for B requests, in the
 *   kda_tkg layouts (NKI "KDA TKG Kernel API Reference", kda_tkg), all fp32:
 *
 *   q, k, g     [B, dk, H]   (head innermost; raw, pre-norm / pre-activation)
 *   v           [B, H, dv]
 *   beta_logits [B, 1, H]
 *   a_log       [H]          (the page's [1, H])
 *   dt_bias     [dk, H]
 *   out         [B, H, dv]   written
 *   S           [B, H, dk, dv] IN/OUT: read, then overwritten with the advanced state.
 *   scale, lower_bound: host floats (the page passes [1, 1] device tensors; host values
 *   keep the call free of device reads and capturable in a CUDA graph).
 */
int kda_decode_step(const float* q, const float* k, const float* v, const float* g,
                    const float* beta_logits, const float* a_log, const float* dt_bias,
                    float scale, float lower_bound, float* out, float* S, int B, int H,
                    int dk, int dv, kda_stream_t stream);

/* Static, human-readable text for a kda_status value (never NULL). */
const char* kda_status_string(int status);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int kda_version(void);

/*
 * kda_device_error -- bitmask of errors that kernels recorded on the current device since
 *   the last reset (no paper counterpart: it reports the kernels' own safeguards).
 *   Bit 0: a bounded wait inside the single-pass tensor-core chunk kernel gave up; bit 1:
 *   one inside the two-launch (workspace) chunk kernels did; bit 2: one inside the
 *   chunked backward's kernels did (the outputs of that launch are incomplete); bit 3: the
 *   wait of kda_selftest_bounded_wait gave up (which is what it is for); bit 4: one inside
 *   the chunked recurrent-attention kernels did; bit 5: a tensor-core kernel of
 *   kda_recurrent_attention_fwd_ws or kda_attention_fwd_ws met gates outside its range,
 *   detected per 16-token sub-chunk (a summed key-axis gate or decay totalling outside
 *   [-80, 16] over a sub-chunk, or a value-axis gate outside [-40, 8] over half of one,
 *   which gates in [-5, 1] rule out; that call's results are unspecified).  Synchronises
 *   the device.  reset != 0
 *   clears the mask.
 *   Returns the mask (>= 0) or KDA_ERR_DEVICE.
 */
int kda_device_error(int reset);

/*
 * kda_selftest_bounded_wait -- launches one kernel whose single wait, on an mbarrier that
 *   nothing arrives on, runs out after limit_ns nanoseconds (1 .. 1e9) and records bit 3 of
 *   kda_device_error: the give-up path every tensor-core kernel takes instead of hanging
 *   the device.  No paper counterpart.  Returns KDA_OK once enqueued; limit_ns outside
 *   (0, 1e9] gives KDA_ERR_BAD_SHAPE.
 */
int kda_selftest_bounded_wait(unsigned long long limit_ns, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
