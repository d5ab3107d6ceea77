/*
 * gdp.h - C ABI of the Gated Delta Product (GDP) forward-pass library for
 * NVIDIA GB300 (sm_103a).
 *
 * The operations follow three Megatron-core API pages:
 *   "core.ssm.ops.gdp.prepare"  (gdp_prepare_kernel, gdp_decode_prepare,
 *                                gdp_prefill_prepare, softplus)
 *   "core.ssm.ops.gdp.wy_fast"  (recompute_w_u_fwd: WY factors w, u from the
 *                                inverted transition block of solve_tril)
 *   "core.ssm.ops.gdp.chunk_o"  (chunk_gated_delta_product_fwd_o: output from
 *                                the chunk-boundary state of chunk_h plus the
 *                                causal within-chunk attention over the copies)
 *
 * Conventions shared by every call:
 *   - Every pointer is a DEVICE pointer owned by the caller, unless a comment
 *     says otherwise. The library allocates no device memory: scratch comes
 *     from a caller-provided workspace whose size a query function returns.
 *   - Every call is asynchronous on `stream`, performs no host
 *     synchronisation (except gdp_read_status, which is for debugging) and
 *     validates all scalar arguments before launching anything. On a
 *     validation error nothing is launched. Work is ordered on `stream` as
 *     usual: the prepare and chunk kernels are launched with programmatic
 *     dependent launch, so each may be scheduled while the work before it is
 *     finishing, but none touches global memory before everything earlier on
 *     the stream has completed and its writes are visible.
 *   - Tensors are row-major with the shapes given; strides, where a call takes
 *     them, are in elements. Only x and ba may be strided (rows), and their
 *     last dimension must be contiguous.
 *   - Returns GDP_OK, or an error code; gdp_status_string() describes it.
 *     GDP_ERR_CUDA means a CUDA runtime call failed (the CUDA error is left
 *     for the caller to read with cudaGetLastError()).
 */
#ifndef GDP_H_
#define GDP_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdp_status {
  GDP_OK = 0,
  GDP_ERR_INVALID_ARG = 1,     /* a pointer, size or stride is invalid */
  GDP_ERR_UNSUPPORTED = 2,     /* valid, but this combination is not built */
  GDP_ERR_CUDA = 3,            /* a CUDA runtime call or launch failed */
  GDP_ERR_DEVICE_TIMEOUT = 4,  /* a bounded device-side wait gave up */
  GDP_ERR_WORKSPACE = 5        /* workspace too small or misaligned (256 B) */
} gdp_status;

typedef enum gdp_dtype { GDP_BF16 = 0, GDP_F16 = 1, GDP_F32 = 2 } gdp_dtype;

/* Human-readable text for a status code (static storage, never NULL). */
const char* gdp_status_string(gdp_status s);

/* Library ABI version (major * 100 + minor). */
int gdp_version(void);

/*
 * gdp_prefill_prepare - split, reshape and gate one prefill step's post-conv
 * activations in one launch (prepare page, module overview and
 * gdp_prefill_prepare).
 *
 *   x       [n, T, M*H*P + M*G*N + G*N] value | key | query, dtype `dt`;
 *           element strides x_sn (per request) and x_st (per token); the last
 *           dimension is contiguous.
 *   ba      [n, T, M*H + H]: M*H beta logits b (copy-major), then H decay
 *           inputs a; strides ba_sn, ba_st; last dimension contiguous.
 *   A_log   [H] fp32 log decay rates.   dt_bias [H] fp32 softplus bias.
 * Outputs (contiguous, caller-allocated):
 *   q [n, T, H, N] (dt), k [n, T*M, H, N] (dt), v [n, T*M, H, P] (dt),
 *   beta [n, T*M, H] fp32 = sigmoid(b), g [n, T, H] fp32 =
 *   -exp(A_log) * softplus(a + dt_bias), softplus(x) = x > 20 ? x : log1p(exp(x)).
 * Copy j of token t sits at expanded position t*M + j. Key/query group
 * grp = h / (H/G) feeds head h. Requires H % G == 0. q/k/v are bit copies;
 * beta and g use the CUDA math library's expf/log1pf with IEEE division,
 * operation by operation in fp32.
 * Errors: GDP_ERR_INVALID_ARG (null pointer, non-positive size, H % G != 0,
 * row strides shorter than a row), GDP_ERR_UNSUPPORTED (dtype), GDP_ERR_CUDA.
 */
gdp_status gdp_prefill_prepare(const void* x, int64_t x_sn, int64_t x_st, const void* ba,
                               int64_t ba_sn, int64_t ba_st, const float* A_log,
                               const float* dt_bias, int n, int T, int M, int H, int G, int P,
                               int N, gdp_dtype dt, void* q, void* k, void* v, float* beta,
                               float* g, cudaStream_t stream);

/*
 * gdp_decode_prepare - the same map for one decode step of S = 1 + drafts
 * tokens per request (prepare page, gdp_decode_prepare), with query and
 * decay placed on the copies: the query on the last copy, g on the first,
 * +0.0 on the others.
 * Inputs as gdp_prefill_prepare with T replaced by S (S in 1..16).
 * Outputs: q [n, S*M, H, N], k [n, S*M, H, N], v [n, S*M, H, P] (dt),
 *          beta [n, S*M, H], g [n, S*M, H] fp32.
 */
gdp_status gdp_decode_prepare(const void* x, int64_t x_sn, int64_t x_st, const void* ba,
                              int64_t ba_sn, int64_t ba_st, const float* A_log,
                              const float* dt_bias, int n, int S, int M, int H, int G, int P,
                              int N, gdp_dtype dt, void* q, void* k, void* v, float* beta,
                              float* g, cudaStream_t stream);

/*
 * gdp_prefill_conv_prepare - the short causal conv that precedes prepare in
 * the layer, fused with gdp_prefill_prepare (prepare page, module overview:
 * prepare consumes the conv's output, and padding is handled by that conv).
 * The pages name the conv but not its form; this call takes the usual
 * depthwise causal short conv with SiLU:
 *   z[t, c] = conv_b[c] + sum_{i<W} conv_w[c, i] * xin[t - (W-1) + i, c]
 *   x[t, c] = z / (1 + exp(-z)), rounded to dtype `dt`,
 * in fp32, one operation at a time (no fused multiply-add), and then applies
 * exactly the map of gdp_prefill_prepare to x. The conv output never reaches
 * memory.
 *   xp        [n, T, C] pre-conv activations, C = M*H*P + M*G*N + G*N (the
 *             channel layout of prepare's x), strides xp_sn, xp_st.
 *   conv_w    [C, W] fp32, tap i multiplies input t - (W-1) + i; W in 1..4.
 *   conv_b    [C] fp32 or NULL (no bias).
 *   conv_state_in  [N_seq, C, W-1] (dtype dt) or NULL (zeros): per sequence,
 *             the W-1 inputs before its first token, oldest first.
 *   conv_state_out [N_seq, C, W-1] (dtype dt) or NULL: per sequence, the last
 *             W-1 inputs of (conv_state_in ++ its tokens), for the next call.
 *             Must not alias conv_state_in.
 *   cu_seqlens [N_seq + 1] int32 token offsets (device) with n == 1, or NULL
 *             (then N_seq == n and each batch row is one sequence); the conv
 *             does not cross a sequence start. Rows past cu_seqlens[N_seq]
 *             are not written.
 * ba, A_log, dt_bias, the sizes and the outputs q, k, v, beta, g are those of
 * gdp_prefill_prepare. Requires 16-byte channel vectors: P and N times the
 * element size multiples of 16 bytes, 16-byte aligned xp, q, k, v, conv
 * states and row strides (else GDP_ERR_UNSUPPORTED).
 */
gdp_status gdp_prefill_conv_prepare(const void* xp, int64_t xp_sn, int64_t xp_st,
                                    const float* conv_w, const float* conv_b, int W,
                                    const void* conv_state_in, void* conv_state_out,
                                    const int32_t* cu_seqlens, int N_seq, const void* ba,
                                    int64_t ba_sn, int64_t ba_st, const float* A_log,
                                    const float* dt_bias, int n, int T, int M, int H, int G,
                                    int P, int N, gdp_dtype dt, void* q, void* k, void* v,
                                    float* beta, float* g, cudaStream_t stream);

/*
 * gdp_decode_conv_prepare - the conv of gdp_prefill_conv_prepare fused with
 * gdp_decode_prepare for one decode step of S tokens per request, with the
 * conv states in a pool indexed by request (prepare page, module overview: "a
 * -1 slot zeroes its conv output, which propagates here"):
 *   conv_state_pool [n_slots, C, W-1] (dtype dt), read and updated in place
 *             at the entries the slots name (the new state is the last W-1
 *             inputs of entry ++ the request's S tokens);
 *   conv_slot [n] int32 (device): the request's pool entry, or -1 for a
 *             padding request, whose q, k and v are written as zeros and which
 *             touches no state (beta and g still come from ba);
 *   status    (device, nullable) int32 set to 1 when a slot is outside
 *             [-1, n_slots) or named by two requests; those requests are
 *             treated as padding. The call never clears it.
 * Other arguments and outputs as gdp_decode_prepare (S in 1..16) and
 * gdp_prefill_conv_prepare. No host synchronisation; graph-capturable.
 */
gdp_status gdp_decode_conv_prepare(const void* xp, int64_t xp_sn, int64_t xp_st,
                                   const float* conv_w, const float* conv_b, int W,
                                   void* conv_state_pool, const int32_t* conv_slot, int n_slots,
                                   const void* ba, int64_t ba_sn, int64_t ba_st,
                                   const float* A_log, const float* dt_bias, int n, int S, int M,
                                   int H, int G, int P, int N, gdp_dtype dt, void* q, void* k,
                                   void* v, float* beta, float* g, int32_t* status,
                                   cudaStream_t stream);

/*
 * gdp_chunk_fwd_workspace_size - bytes of device workspace gdp_chunk_fwd
 * needs for these sizes (pure host arithmetic; 0 if the sizes are invalid).
 * N_seq is the number of packed sequences when cu_seqlens is used, else B.
 */
size_t gdp_chunk_fwd_workspace_size(int B, int T, int N_seq, int H, int HV, int K, int V, int M,
                                    int chunk_size, gdp_dtype dt);

/*
 * gdp_chunk_fwd - chunked Gated Delta Product forward (wy_fast page:
 * recompute_w_u_fwd; chunk_o page: chunk_gated_delta_product_fwd_o), from
 * the prepared tensors to the outputs and the final state:
 *   per (sequence, value head hv), with key/query head kh = hv / (HV/H), the
 *   state S (V x K) walks the expanded stream, copy j of token t at t*M + j:
 *     S <- exp(g_e) S (I - beta_e k_e k_e^T) + beta_e v_e k_e^T,
 *   g_e = g_t on a token's first copy and 0 on the others, and
 *   o_t = scale * S q_t after the token's last copy.
 * computed chunk-wise: transition block and its inverse (solve_tril), WY
 * factors w and u, chunk-boundary state recurrence with corrected values
 * v_new = u - w h, then output = q h + causal within-chunk attention summed
 * over the M copies.
 *
 *   q [B, T, H, K], k [B, T*M, H, K], v [B, T*M, HV, V]   dtype dt
 *   beta [B, T*M, HV] fp32; g [B, T, HV] fp32 natural-log decay per token, or
 *   NULL (ungated: g = 0)
 *   initial_state [N_seq, HV, K, V] fp32 or NULL (zeros)
 *   cu_seqlens [N_seq + 1] int32 token offsets on the unexpanded stream, or
 *   NULL (then N_seq must equal B). With cu_seqlens, B must be 1, offsets must
 *   be non-decreasing with cu_seqlens[0] = 0 and cu_seqlens[N_seq] <= T; they
 *   are read on the device only (no host synchronisation). A list that breaks
 *   these rules sets the workspace status word (gdp_read_status then returns
 *   GDP_ERR_INVALID_ARG); o is left untouched and final_state receives each
 *   sequence's initial state (zeros without one).
 *   chunk_size: 16, 32 or 64. scale: score scale (the pages' default is
 *   K^-0.5; the caller passes it). use_qk_l2norm: 1 to L2-normalise q and k
 *   per (position, head) as x / sqrt(sum x^2 + 1e-6) before use.
 * Outputs: o [B, T, HV, V] fp32; final_state [N_seq, HV, K, V] fp32 or NULL.
 * workspace: device scratch of at least gdp_chunk_fwd_workspace_size() bytes,
 * 256-byte aligned; its first 256 bytes hold the device status word that
 * gdp_read_status() reads back. Calls that share a workspace must not overlap
 * on the GPU.
 * Requires HV % H == 0, K <= 256, V <= 1024, M in 1..8; GDP_ERR_UNSUPPORTED
 * when B*T*M*HV, the expanded chunks times chunk_size, or the token chunks
 * times HV*K reach 2^31 (the kernels' 32-bit row coordinates; such tensors
 * exceed one GPU's memory).
 * Path: bf16 inputs with K = 128, chunk_size 64, V in {64, 128, 256} and
 * M <= 3 run on the tensor cores (bf16 hi/lo operand splits, fp32
 * accumulation; for M = 2 the output is formed inside the state-scan kernel);
 * every other shape runs an fp32 CUDA-core path of the same algebra.
 * gdp_chunk_fwd_stage_offsets reports which path a shape takes.
 */
gdp_status gdp_chunk_fwd(const void* q, const void* k, const void* v, const float* beta,
                         const float* g, const float* initial_state, const int32_t* cu_seqlens,
                         int N_seq, int B, int T, int H, int HV, int K, int V, int M,
                         int chunk_size, float scale, int use_qk_l2norm, gdp_dtype dt, float* o,
                         float* final_state, void* workspace, size_t ws_bytes,
                         cudaStream_t stream);

/*
 * gdp_recurrent_update - fused recurrent update for decode (prepare page,
 * decode bullet: the copies are walked as a sequence). For each request r
 * and value head hv the fp32 state h = S^T [K, V] is updated in place over
 * L = S*M steps, each step e using its own inputs:
 *   S <- exp(g_e) S (I - beta_e k_e k_e^T) + beta_e v_e k_e^T;
 *   o_e = scale * S q_e.
 *   q [n, L, H, K], k [n, L, H, K], v [n, L, HV, V] dtype dt (q is zero on all
 *   but a token's last copy when it comes from gdp_decode_prepare);
 *   beta [n, L, HV], g [n, L, HV] fp32 (natural log);
 *   state [n, HV, K, V] fp32, read and written in place;
 *   o [n, L, HV, V] fp32.
 * Requires HV % H == 0, K in {32, 64, 128, 256}, V % 8 == 0, V <= 1024.
 * No scratch, no host synchronisation, fixed launch shape for fixed sizes.
 */
gdp_status gdp_recurrent_update(const void* q, const void* k, const void* v, const float* beta,
                                const float* g, float* state, int n, int L, int H, int HV, int K,
                                int V, float scale, int use_qk_l2norm, gdp_dtype dt, float* o,
                                cudaStream_t stream);

/*
 * gdp_recurrent_update_slots - gdp_recurrent_update for a decode batch whose
 * requests keep their states in a shared pool (the serving side of the
 * prepare page's decode bullet: padding requests carry slot -1 upstream,
 * where the conv zeroes their output, and the recurrent update must leave
 * them out). Request r updates pool entry state_slot[r]:
 *   state_pool [n_slots, HV, K, V] fp32, read and written in place at the
 *              entries the slots name; other entries are not touched;
 *   state_slot [n] int32 (device): entry of request r, or -1 for a padding
 *              request, whose o rows are written as zeros and which reads and
 *              writes no state;
 *   status     (device, nullable) int32 set to 1 (GDP_ERR_INVALID_ARG) when a
 *              slot is outside [-1, n_slots) or is named by two requests; such
 *              requests are skipped like padding. The call never clears it.
 * Other arguments and o as gdp_recurrent_update. Slots are read on the device
 * only: no host synchronisation, static launch shape for fixed sizes, so the
 * call can be captured in a CUDA graph with the slot table updated in place
 * between replays.
 */
gdp_status gdp_recurrent_update_slots(const void* q, const void* k, const void* v,
                                      const float* beta, const float* g, float* state_pool,
                                      const int32_t* state_slot, int n_slots, int n, int L,
                                      int H, int HV, int K, int V, float scale,
                                      int use_qk_l2norm, gdp_dtype dt, float* o,
                                      int32_t* status, cudaStream_t stream);

/*
 * gdp_read_status - synchronise `stream` and return the device status word
 * in the first bytes of a gdp_chunk_fwd workspace: GDP_OK, or
 * GDP_ERR_DEVICE_TIMEOUT if a bounded wait inside a kernel gave up.
 * Debugging aid; it does synchronise.
 */
gdp_status gdp_read_status(const void* workspace, cudaStream_t stream);

/*
 * gdp_chunk_fwd_stage_offsets - byte offsets, inside a gdp_chunk_fwd
 * workspace for these sizes, of the intermediate stages the last call left
 * there (for stage-by-stage checks), or SIZE_MAX for a stage the selected
 * path does not materialise. `out` (HOST pointer, 8 entries) receives:
 *   [0] A      fp32 [B*T*M, HV, BT]  inverted transition blocks (row p = its
 *                                    chunk row, zero-padded)
 *   [1] w      fp32 [B*T*M, HV, K]
 *   [2] u      fp32 [B*T*M, HV, V]
 *   [3] v_new  fp32 [B*T*M, HV, V]   corrected values
 *   [4] h      fp32 [n_tok_chunks, HV, K, V] state at each token-chunk start,
 *                                    sequences in order
 *   [5] path   not an offset: 0 = generic fp32 path, 1 = tensor-core path
 *   [6] wy_len not an offset: positions per WY block (the A/w/u stages); the
 *              tensor-core path uses 128-position blocks (two chunks) for even M
 *   [7] fused  not an offset: 1 when the chunk output is computed inside the
 *              state-scan kernel (the tensor-core path for M = 2: no separate
 *              output launch, v_new and h are not stored), else 0
 * Returns GDP_ERR_INVALID_ARG on invalid sizes.
 */
gdp_status gdp_chunk_fwd_stage_offsets(int B, int T, int N_seq, int H, int HV, int K, int V,
                                       int M, int chunk_size, gdp_dtype dt, size_t* out);

/*
 * gdp_chunk_fwd_noalloc - gdp_chunk_fwd for callers that cannot allocate
 * device memory. The pages have no counterpart to this call; it exists for
 * callers that run under a memory budget fixed in advance, from inside
 * another allocator's callbacks, or in loops that must never reach
 * cudaMalloc/cudaFree (which can synchronise the device), and so cannot
 * provide a workspace.
 * Arguments and outputs are those of gdp_chunk_fwd without the workspace.
 * Scratch: a 32 MiB array in device memory that the library holds on every
 * GPU that loads it, until the process exits. Problems whose workspace
 * (gdp_chunk_fwd_workspace_size) exceeds 32 MiB are rejected with
 * GDP_ERR_WORKSPACE before anything is launched. The call allocates nothing.
 * All calls share the array and it keeps the previous call's contents; each
 * call clears what must start at zero. Calls that overlap on the GPU (other
 * streams or host threads) race on the array: serialise them.
 * The first call on a device looks up the array's device address with that
 * device current and keeps it for the life of the process; make that first
 * call before any stream capture, and do not reset the device
 * (cudaDeviceReset) between calls, which would leave the kept address stale.
 * cu_seqlens is validated on the device as in gdp_chunk_fwd; a bad list
 * leaves o untouched and passes the initial states to final_state, but this
 * call has no workspace whose status word the caller could read.
 */
gdp_status gdp_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* beta,
                                 const float* g, const float* initial_state,
                                 const int32_t* cu_seqlens, int N_seq, int B, int T, int H,
                                 int HV, int K, int V, int M, int chunk_size, float scale,
                                 int use_qk_l2norm, gdp_dtype dt, float* o, float* final_state,
                                 cudaStream_t stream);

/*
 * gdp_debug_wait_fault - TEST HOOK for the device-side failure path; off by
 * default and never needed in normal use. Every mbarrier wait inside the
 * tensor-core kernels is bounded (2 s of wall time); a wait that runs out
 * records GDP_ERR_DEVICE_TIMEOUT in the workspace status word, and the kernel
 * leaves cleanly (it waits, bounded, for its own copies in flight and frees
 * its tensor memory) instead of hanging the GPU.
 *   arm = 1: the next gdp_chunk_fwd that runs the 128-position WY kernel
 *            (tensor-core path, even M) leaves out one tensor-core commit in
 *            its first CTA, so that CTA's wait for it runs out; the hook then
 *            disarms itself. arm = 0: disarm.
 *   budget_seconds: new wait budget (0 < budget <= 10), or <= 0 for the
 *            default 2 s. The budget applies to every later launch until
 *            changed.
 * Synchronous (it writes a device variable on the current device). Results of
 * the faulted call are undefined; later calls are unaffected.
 * Errors: GDP_ERR_INVALID_ARG (budget above 10 s), GDP_ERR_CUDA.
 */
gdp_status gdp_debug_wait_fault(int arm, double budget_seconds);

/* Number of stage-boundary events gdp_set_stage_events takes. */
#define GDP_STAGE_EVENTS 5

/*
 * gdp_set_stage_events - profiling hook. When `events` (HOST array of n >=
 * GDP_STAGE_EVENTS caller-created cudaEvent_t) is non-NULL, every later
 * gdp_chunk_fwd call records events[i] on its stream at its stage
 * boundaries: [0] entry, [1] after the chunk tables, [2] after the WY stage
 * (transition block, solve_tril, w and u), [3] after the chunk-boundary state
 * recurrence, [4] after the output stage. A path that fuses stages records
 * the fused boundaries back to back. NULL switches the hook off. The hook is
 * process-wide and not thread-safe; the events stay owned by the caller.
 */
gdp_status gdp_set_stage_events(cudaEvent_t* events, int n);

#ifdef __cplusplus
}
#endif

#endif /* GDP_H_ */
