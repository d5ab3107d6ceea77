// C ABI entry points of libgdp: argument validation, workspace layout and
// dispatch to the kernels. Every validation runs before anything is launched;
// nothing here allocates device memory or synchronises (gdp_read_status
// excepted).
#include <mutex>
#include <vector>

#include "gdp_internal.cuh"

namespace gdp {

int sm_count() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// Profiling hook (gdp_set_stage_events): caller-created events recorded at the
// stage boundaries of every gdp_chunk_fwd call.
static cudaEvent_t g_stage_events[GDP_STAGE_EVENTS];
static bool g_stage_on = false;

void record_stage(int i, cudaStream_t s) {
  if (g_stage_on && i >= 0 && i < GDP_STAGE_EVENTS) cudaEventRecord(g_stage_events[i], s);
}

}  // namespace gdp

using namespace gdp;

namespace {

bool dtype_ok(gdp_dtype dt) { return dt == GDP_BF16 || dt == GDP_F16 || dt == GDP_F32; }

gdp_status check_prepare(const void* x, int64_t x_sn, int64_t x_st, const void* ba, int64_t ba_sn,
                         int64_t ba_st, const float* A_log, const float* dt_bias, int n, int T,
                         int M, int H, int G, int P, int N, gdp_dtype dt, const void* q,
                         const void* k, const void* v, const float* beta, const float* g) {
  if (!dtype_ok(dt)) return GDP_ERR_UNSUPPORTED;
  if (n < 0 || T < 0 || M <= 0 || H <= 0 || G <= 0 || P <= 0 || N <= 0) return GDP_ERR_INVALID_ARG;
  if (H % G != 0) return GDP_ERR_INVALID_ARG;
  if ((int64_t)n * T == 0) return GDP_OK;
  if (!x || !ba || !A_log || !dt_bias || !q || !k || !v || !beta || !g) return GDP_ERR_INVALID_ARG;
  const int64_t D = (int64_t)M * H * P + (int64_t)M * G * N + (int64_t)G * N;
  const int64_t Dba = (int64_t)M * H + H;
  if (x_st < D || ba_st < Dba) return GDP_ERR_INVALID_ARG;
  if (n > 1 && (x_sn < (int64_t)T * x_st || ba_sn < (int64_t)T * ba_st)) return GDP_ERR_INVALID_ARG;
  return GDP_OK;
}

gdp_status check_chunk(const void* q, const void* k, const void* v, const float* beta,
                       const int32_t* cu_seqlens, int N_seq, int B, int T, int H, int HV, int K,
                       int V, int M, int BT, gdp_dtype dt, const float* o, const void* ws,
                       size_t ws_bytes, size_t need) {
  if (!dtype_ok(dt)) return GDP_ERR_UNSUPPORTED;
  if (B <= 0 || T < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || M <= 0 || N_seq < 0)
    return GDP_ERR_INVALID_ARG;
  if (HV % H != 0) return GDP_ERR_INVALID_ARG;
  if (cu_seqlens ? (B != 1) : (N_seq != B)) return GDP_ERR_INVALID_ARG;
  if (!(BT == 16 || BT == 32 || BT == 64)) return GDP_ERR_UNSUPPORTED;
  if (K > 256 || V > 1024 || M > 8) return GDP_ERR_UNSUPPORTED;
  // The kernels address positions, decay-record rows and state rows with 32-bit
  // tensor-map coordinates and table entries; every one of them stays below
  // 2^31 for problems whose tensors fit in a GPU's memory, and larger ones are
  // refused here.
  {
    int64_t NE, NT;
    chunk_bounds(B, T, N_seq, M, BT, &NE, &NT);
    if ((int64_t)B * T * M * HV > INT32_MAX || NE * BT > INT32_MAX || NT * HV * K > INT32_MAX)
      return GDP_ERR_UNSUPPORTED;
  }
  if ((int64_t)B * T > 0 && (!q || !k || !v || !beta || !o)) return GDP_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < need)
    return GDP_ERR_WORKSPACE;
  return GDP_OK;
}

WsLayout layout_for(int B, int T, int N_seq, int H, int HV, int K, int V, int M, int BT,
                    gdp_dtype dt) {
  if (tc_supported(H, HV, K, V, M, BT, dt)) return tc_layout(B, T, N_seq, H, HV, K, V, M, BT);
  return generic_layout(B, T, N_seq, H, HV, K, V, M, BT);
}

bool sizes_valid(int B, int T, int N_seq, int H, int HV, int K, int V, int M, int BT) {
  return B > 0 && T >= 0 && N_seq >= 0 && H > 0 && HV > 0 && K > 0 && V > 0 && M > 0 &&
         HV % H == 0 && (BT == 16 || BT == 32 || BT == 64) && K <= 256 && V <= 1024 && M <= 8;
}

}  // namespace

extern "C" {

const char* gdp_status_string(gdp_status s) {
  switch (s) {
    case GDP_OK: return "ok";
    case GDP_ERR_INVALID_ARG: return "invalid argument";
    case GDP_ERR_UNSUPPORTED: return "unsupported combination";
    case GDP_ERR_CUDA: return "CUDA runtime error";
    case GDP_ERR_DEVICE_TIMEOUT: return "device-side bounded wait timed out";
    case GDP_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
  }
  return "unknown status";
}

int gdp_version(void) { return 100; }

gdp_status gdp_prefill_prepare(const void* x, int64_t x_sn, int64_t x_st, const void* ba,
                               int64_t ba_sn, int64_t ba_st, const float* A_log,
                               const float* dt_bias, int n, int T, int M, int H, int G, int P,
                               int N, gdp_dtype dt, void* q, void* k, void* v, float* beta,
                               float* g, cudaStream_t stream) {
  gdp_status s = check_prepare(x, x_sn, x_st, ba, ba_sn, ba_st, A_log, dt_bias, n, T, M, H, G,
                               P, N, dt, q, k, v, beta, g);
  if (s != GDP_OK || (int64_t)n * T == 0) return s;
  cudaError_t e = launch_prepare(x, x_sn, x_st, ba, ba_sn, ba_st, A_log, dt_bias, n, T, M, H, G,
                                 P, N, dt, false, q, k, v, beta, g, stream);
  return e == cudaSuccess ? GDP_OK : GDP_ERR_CUDA;
}

gdp_status gdp_decode_prepare(const void* x, int64_t x_sn, int64_t x_st, const void* ba,
                              int64_t ba_sn, int64_t ba_st, const float* A_log,
                              const float* dt_bias, int n, int S, int M, int H, int G, int P,
                              int N, gdp_dtype dt, void* q, void* k, void* v, float* beta,
                              float* g, cudaStream_t stream) {
  if (S < 1 || S > 16) return GDP_ERR_INVALID_ARG;
  gdp_status s = check_prepare(x, x_sn, x_st, ba, ba_sn, ba_st, A_log, dt_bias, n, S, M, H, G,
                               P, N, dt, q, k, v, beta, g);
  if (s != GDP_OK || n == 0) return s;
  cudaError_t e = launch_prepare(x, x_sn, x_st, ba, ba_sn, ba_st, A_log, dt_bias, n, S, M, H, G,
                                 P, N, dt, true, q, k, v, beta, g, stream);
  return e == cudaSuccess ? GDP_OK : GDP_ERR_CUDA;
}

}  // extern "C"

namespace {

// The fused conv + prepare calls need 16-byte channel vectors: every head
// size a multiple of 16 bytes, 16-byte aligned bases and row strides.
gdp_status check_conv(const void* xp, int64_t xp_sn, int64_t xp_st, const float* w, int W, int P,
                      int N, gdp_dtype dt, const void* q, const void* k, const void* v) {
  if (W < 1 || W > 4 || !w) return W < 1 || !w ? GDP_ERR_INVALID_ARG : GDP_ERR_UNSUPPORTED;
  const int64_t es = dt == GDP_F32 ? 4 : 2;
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if ((P * es) % 16 || (N * es) % 16 || (xp_sn * es) % 16 || (xp_st * es) % 16 || !al(xp) ||
      !al(q) || !al(k) || !al(v))
    return GDP_ERR_UNSUPPORTED;
  return GDP_OK;
}

}  // namespace

extern "C" {

gdp_status gdp_prefill_conv_prepare(const void* xp, int64_t xp_sn, int64_t xp_st,
                                    const float* conv_w, const float* conv_b, int W,
                                    const void* conv_state_in, void* conv_state_out,
                                    const int32_t* cu_seqlens, int N_seq, const void* ba,
                                    int64_t ba_sn, int64_t ba_st, const float* A_log,
                                    const float* dt_bias, int n, int T, int M, int H, int G,
                                    int P, int N, gdp_dtype dt, void* q, void* k, void* v,
                                    float* beta, float* g, cudaStream_t stream) {
  gdp_status s = check_prepare(xp, xp_sn, xp_st, ba, ba_sn, ba_st, A_log, dt_bias, n, T, M, H,
                               G, P, N, dt, q, k, v, beta, g);
  if (s != GDP_OK) return s;
  if (cu_seqlens ? (n != 1 || N_seq < 0) : (N_seq != n)) return GDP_ERR_INVALID_ARG;
  if (conv_state_in && conv_state_in == conv_state_out) return GDP_ERR_INVALID_ARG;
  if (W < 1 || !conv_w) return GDP_ERR_INVALID_ARG;
  if ((int64_t)n * T == 0) {  // no tokens: every sequence keeps its initial state
    if (!conv_state_out || W == 1 || N_seq == 0) return GDP_OK;
    const size_t bytes = (size_t)N_seq * ((size_t)M * H * P + (size_t)M * G * N + (size_t)G * N) *
                         (size_t)(W - 1) * (dt == GDP_F32 ? 4 : 2);
    const cudaError_t e = conv_state_in ? cudaMemcpyAsync(conv_state_out, conv_state_in, bytes,
                                                          cudaMemcpyDeviceToDevice, stream)
                                        : cudaMemsetAsync(conv_state_out, 0, bytes, stream);
    return e == cudaSuccess ? GDP_OK : GDP_ERR_CUDA;
  }
  if ((s = check_conv(xp, xp_sn, xp_st, conv_w, W, P, N, dt, q, k, v)) != GDP_OK) return s;
  if ((reinterpret_cast<uintptr_t>(conv_state_in) | reinterpret_cast<uintptr_t>(conv_state_out)) % 16)
    return GDP_ERR_UNSUPPORTED;
  const cudaError_t e = launch_conv_prepare(
      xp, xp_sn, xp_st, conv_w, conv_b, W, conv_state_in, conv_state_out, cu_seqlens, N_seq,
      nullptr, 0, nullptr, ba, ba_sn, ba_st, A_log, dt_bias, n, T, M, H, G, P, N, dt, false, q,
      k, v, beta, g, stream);
  return e == cudaSuccess ? GDP_OK : GDP_ERR_CUDA;
}

gdp_status gdp_decode_conv_prepare(const void* xp, int64_t xp_sn, int64_t xp_st,
                                   const float* conv_w, const float* conv_b, int W,
                                   void* conv_state_pool, const int32_t* conv_slot, int n_slots,
                                   const void* ba, int64_t ba_sn, int64_t ba_st,
                                   const float* A_log, const float* dt_bias, int n, int S, int M,
                                   int H, int G, int P, int N, gdp_dtype dt, void* q, void* k,
                                   void* v, float* beta, float* g, int32_t* status,
                                   cudaStream_t stream) {
  if (S < 1 || S > 16 || n_slots < 0) return GDP_ERR_INVALID_ARG;
  gdp_status s = check_prepare(xp, xp_sn, xp_st, ba, ba_sn, ba_st, A_log, dt_bias, n, S, M, H,
                               G, P, N, dt, q, k, v, beta, g);
  if (s != GDP_OK || n == 0) return s;
  if (!conv_slot || (W > 1 && n_slots > 0 && !conv_state_pool)) return GDP_ERR_INVALID_ARG;
  if ((s = check_conv(xp, xp_sn, xp_st, conv_w, W, P, N, dt, q, k, v)) != GDP_OK) return s;
  if (reinterpret_cast<uintptr_t>(conv_state_pool) % 16) return GDP_ERR_UNSUPPORTED;
  const cudaError_t e = launch_conv_prepare(
      xp, xp_sn, xp_st, conv_w, conv_b, W, conv_state_pool, conv_state_pool, nullptr, n,
      conv_slot, n_slots, status, ba, ba_sn, ba_st, A_log, dt_bias, n, S, M, H, G, P, N, dt,
      true, q, k, v, beta, g, stream);
  return e == cudaSuccess ? GDP_OK : GDP_ERR_CUDA;
}

size_t gdp_chunk_fwd_workspace_size(int B, int T, int N_seq, int H, int HV, int K, int V, int M,
                                    int chunk_size, gdp_dtype dt) {
  if (!sizes_valid(B, T, N_seq, H, HV, K, V, M, chunk_size) || !dtype_ok(dt)) return 0;
  return layout_for(B, T, N_seq, H, HV, K, V, M, chunk_size, dt).total;
}

gdp_status gdp_chunk_fwd_stage_offsets(int B, int T, int N_seq, int H, int HV, int K, int V,
                                       int M, int chunk_size, gdp_dtype dt, size_t* out) {
  if (!out || !sizes_valid(B, T, N_seq, H, HV, K, V, M, chunk_size) || !dtype_ok(dt))
    return GDP_ERR_INVALID_ARG;
  const WsLayout L = layout_for(B, T, N_seq, H, HV, K, V, M, chunk_size, dt);
  out[0] = L.A;
  out[1] = L.w;
  out[2] = L.u;
  out[3] = L.v_new;
  out[4] = L.h;
  out[5] = (size_t)L.path;
  out[6] = (size_t)((L.path == 1 && M % 2 == 0) ? 128 : chunk_size);
  out[7] = (L.path == 1 && M == 2) ? 1 : 0;
  return GDP_OK;
}

gdp_status gdp_chunk_fwd(const void* q, const void* k, const void* v, const float* beta,
                         const float* g, const float* initial_state, const int32_t* cu_seqlens,
                         int N_seq, int B, int T, int H, int HV, int K, int V, int M,
                         int chunk_size, float scale, int use_qk_l2norm, gdp_dtype dt, float* o,
                         float* final_state, void* workspace, size_t ws_bytes,
                         cudaStream_t stream) {
  if (!sizes_valid(B, T, N_seq, H, HV, K, V, M, chunk_size)) {
    if (!dtype_ok(dt)) return GDP_ERR_UNSUPPORTED;
    if (chunk_size != 16 && chunk_size != 32 && chunk_size != 64) return GDP_ERR_UNSUPPORTED;
    if (K > 256 || V > 1024 || M > 8) return GDP_ERR_UNSUPPORTED;
    return GDP_ERR_INVALID_ARG;
  }
  const WsLayout L = layout_for(B, T, N_seq, H, HV, K, V, M, chunk_size, dt);
  gdp_status s = check_chunk(q, k, v, beta, cu_seqlens, N_seq, B, T, H, HV, K, V, M, chunk_size,
                             dt, o, workspace, ws_bytes, L.total);
  if (s != GDP_OK) return s;
  ChunkProblem p;
  p.q = q; p.k = k; p.v = v; p.beta = beta; p.g = g; p.h0 = initial_state;
  p.cu_seqlens = cu_seqlens;
  p.N_seq = N_seq; p.B = B; p.T = T; p.H = H; p.HV = HV; p.K = K; p.V = V; p.M = M;
  p.BT = chunk_size; p.scale = scale; p.l2norm = use_qk_l2norm ? 1 : 0; p.dt = dt;
  p.o = o; p.hT = final_state; p.stream = stream;
  chunk_bounds(B, T, N_seq, M, chunk_size, &p.NE_max, &p.NT_max);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  record_stage(0, stream);
  if (N_seq == 0) {
    if (cudaMemsetAsync(ws + L.status, 0, sizeof(int32_t), stream) != cudaSuccess)
      return GDP_ERR_CUDA;
    for (int i = 1; i < GDP_STAGE_EVENTS; ++i) record_stage(i, stream);
    return GDP_OK;
  }
  // the chunk-table kernel, first of the call, writes the status word (0 or the
  // bad-offsets code); later kernels only ever record errors in it
  if (launch_tables(p, L, ws) != cudaSuccess) return GDP_ERR_CUDA;
  record_stage(1, stream);
  const cudaError_t e = L.path == 1 ? launch_chunk_tc(p, L, ws) : launch_chunk_generic(p, L, ws);
  return e == cudaSuccess ? GDP_OK : GDP_ERR_CUDA;
}

gdp_status gdp_recurrent_update(const void* q, const void* k, const void* v, const float* beta,
                                const float* g, float* state, int n, int L, int H, int HV, int K,
                                int V, float scale, int use_qk_l2norm, gdp_dtype dt, float* o,
                                cudaStream_t stream) {
  if (!dtype_ok(dt)) return GDP_ERR_UNSUPPORTED;
  if (n < 0 || L < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || HV % H != 0)
    return GDP_ERR_INVALID_ARG;
  if (!(K == 32 || K == 64 || K == 128 || K == 256) || V % 8 != 0 || V > 1024)
    return GDP_ERR_UNSUPPORTED;
  if ((int64_t)n * L == 0) return GDP_OK;
  if (!q || !k || !v || !beta || !g || !state || !o) return GDP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(state) | reinterpret_cast<uintptr_t>(o)) % 16 != 0)
    return GDP_ERR_INVALID_ARG;
  const cudaError_t e = launch_recurrent(q, k, v, beta, g, state, n, L, H, HV, K, V, scale,
                                         use_qk_l2norm ? 1 : 0, dt, o, nullptr, 0, nullptr,
                                         stream);
  return e == cudaSuccess ? GDP_OK : GDP_ERR_CUDA;
}

gdp_status gdp_recurrent_update_slots(const void* q, const void* k, const void* v,
                                      const float* beta, const float* g, float* state_pool,
                                      const int32_t* state_slot, int n_slots, int n, int L,
                                      int H, int HV, int K, int V, float scale,
                                      int use_qk_l2norm, gdp_dtype dt, float* o,
                                      int32_t* status, cudaStream_t stream) {
  if (!dtype_ok(dt)) return GDP_ERR_UNSUPPORTED;
  if (n < 0 || L < 0 || n_slots < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || HV % H != 0)
    return GDP_ERR_INVALID_ARG;
  if (!(K == 32 || K == 64 || K == 128 || K == 256) || V % 8 != 0 || V > 1024)
    return GDP_ERR_UNSUPPORTED;
  if ((int64_t)n * L == 0) return GDP_OK;
  if (!q || !k || !v || !beta || !g || !state_slot || !o || (n_slots > 0 && !state_pool))
    return GDP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(state_pool) | reinterpret_cast<uintptr_t>(o)) % 16 != 0)
    return GDP_ERR_INVALID_ARG;
  const cudaError_t e = launch_recurrent(q, k, v, beta, g, state_pool, n, L, H, HV, K, V, scale,
                                         use_qk_l2norm ? 1 : 0, dt, o, state_slot, n_slots,
                                         status, stream);
  return e == cudaSuccess ? GDP_OK : GDP_ERR_CUDA;
}

gdp_status gdp_set_stage_events(cudaEvent_t* events, int n) {
  if (!events) {
    g_stage_on = false;
    return GDP_OK;
  }
  if (n < GDP_STAGE_EVENTS) return GDP_ERR_INVALID_ARG;
  for (int i = 0; i < GDP_STAGE_EVENTS; ++i) {
    if (!events[i]) return GDP_ERR_INVALID_ARG;
    g_stage_events[i] = events[i];
  }
  g_stage_on = true;
  return GDP_OK;
}

gdp_status gdp_read_status(const void* workspace, cudaStream_t stream) {
  if (!workspace) return GDP_ERR_INVALID_ARG;
  int word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return GDP_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GDP_ERR_CUDA;
  if (word == kDevOk) return GDP_OK;
  if (word == kDevBadSeqlens) return GDP_ERR_INVALID_ARG;
  return GDP_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
