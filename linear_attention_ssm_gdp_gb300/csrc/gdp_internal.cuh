// Internal declarations shared by the CUDA translation units of libgdp.
// Nothing here is part of the C ABI (include/gdp.h is).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "gdp.h"

namespace gdp {

constexpr size_t kAlign = 256;
__host__ __device__ inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }
__host__ __device__ inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Device status word codes (first int32 of a chunk_fwd workspace).
enum DeviceStatus : int { kDevOk = 0, kDevBadSeqlens = 1, kDevTimeout = 2 };

// Per-sequence descriptor built on the device from cu_seqlens (or from B, T):
// x = first token in the flattened [B*T] token stream, y = length in tokens,
// z = index of its first expanded chunk, w = index of its first token chunk.
// Chunk tables map a global chunk index to (sequence, chunk-in-sequence);
// entries past the real total hold sequence -1 and their CTAs exit.

// One chunked-forward problem, as validated by the API layer.
struct ChunkProblem {
  const void* q;
  const void* k;
  const void* v;
  const float* beta;
  const float* g;  // may be null (ungated)
  const float* h0; // may be null
  const int32_t* cu_seqlens;  // may be null
  int N_seq, B, T, H, HV, K, V, M, BT;
  float scale;
  int l2norm;
  gdp_dtype dt;
  float* o;
  float* hT;  // may be null
  cudaStream_t stream;
  int64_t NE_max;  // upper bound on expanded chunks over all sequences
  int64_t NT_max;  // upper bound on token chunks over all sequences
};

// Byte offsets inside a chunk_fwd workspace.
struct WsLayout {
  size_t status = 0, seq_info = 0, exp_tab = 0, tok_tab = 0;
  // tensor-core path: launch order of the state-scan chains (sequences by length)
  size_t seq_order = SIZE_MAX;
  // tensor-core path, even M: list of 128-position blocks (sequence, first 64-chunk)
  size_t blk_tab = SIZE_MAX;
  size_t A = SIZE_MAX, w = SIZE_MAX, u = SIZE_MAX, gexp = SIZE_MAX, v_new = SIZE_MAX,
         h = SIZE_MAX;
  // tensor-core path buffers: w and v_new as bf16 hi/lo pairs, per-position
  // (Gam hi, Gam lo, 1/|k|) records, chunk-start states as bf16 hi/lo [.., V, K]
  size_t w_hi = SIZE_MAX, w_lo = SIZE_MAX, gam = SIZE_MAX, vn_hi = SIZE_MAX, vn_lo = SIZE_MAX,
         h_hi = SIZE_MAX, h_lo = SIZE_MAX;
  size_t total = 0;
  int path = 0;  // 0 generic, 1 tensor core
};

// Upper bound on 128-position blocks over all sequences.
inline int64_t block128_bound(int B, int T, int N_seq, int M) {
  return ((int64_t)B * T * M + 127) / 128 + N_seq;
}

// Sizes derived from (B, T, N_seq, M, BT): upper bounds on chunk counts.
inline void chunk_bounds(int B, int T, int N_seq, int M, int BT, int64_t* NE, int64_t* NT) {
  const int64_t Ttot = (int64_t)B * T;
  *NE = cdiv(Ttot * M, BT) + N_seq;
  *NT = cdiv(Ttot, BT) + N_seq;
}

WsLayout generic_layout(int B, int T, int N_seq, int H, int HV, int K, int V, int M, int BT);
WsLayout tc_layout(int B, int T, int N_seq, int H, int HV, int K, int V, int M, int BT);
bool tc_supported(int H, int HV, int K, int V, int M, int BT, gdp_dtype dt);

// Launchers (return cudaSuccess or the launch error).
cudaError_t launch_prepare(const void* x, int64_t x_sn, int64_t x_st, const void* ba,
                           int64_t ba_sn, int64_t ba_st, const float* A_log,
                           const float* dt_bias, int n, int T, int M, int H, int G, int P,
                           int N, gdp_dtype dt, bool decode, void* q, void* k, void* v,
                           float* beta, float* g, cudaStream_t stream);

// Short causal conv fused with prepare (prepare.cu). Prefill: st_in/st_out are
// per-sequence conv states (nullable), cu the varlen offsets (nullable). Decode:
// st_in == st_out is the state pool, slot the per-request pool entries.
cudaError_t launch_conv_prepare(const void* xp, int64_t xp_sn, int64_t xp_st, const float* w,
                                const float* bias, int W, const void* st_in, void* st_out,
                                const int32_t* cu, int N_seq, const int32_t* slot, int n_slots,
                                int32_t* status, const void* ba, int64_t ba_sn, int64_t ba_st,
                                const float* A_log, const float* dt_bias, int n, int T, int M,
                                int H, int G, int P, int N, gdp_dtype dt, bool decode, void* q,
                                void* k, void* v, float* beta, float* g, cudaStream_t stream);

cudaError_t launch_tables(const ChunkProblem& p, const WsLayout& L, uint8_t* ws);
cudaError_t launch_chunk_generic(const ChunkProblem& p, const WsLayout& L, uint8_t* ws);
cudaError_t launch_chunk_tc(const ChunkProblem& p, const WsLayout& L, uint8_t* ws);

// slot: null (request r updates state entry r) or int32 [n] entries of a pool of
// n_slots states (-1: padding request); status (nullable) is set to 1 when a slot
// is out of range or shared by two requests.
cudaError_t launch_recurrent(const void* q, const void* k, const void* v, const float* beta,
                             const float* g, float* state, int n, int L, int H, int HV, int K,
                             int V, float scale, int l2norm, gdp_dtype dt, float* o,
                             const int32_t* slot, int n_slots, int32_t* status,
                             cudaStream_t stream);

int sm_count();  // multiprocessors on the current device (cached per device)

// Programmatic dependent launch. A kernel launched with launch_pdl is launched
// as soon as the kernel before it in the stream completes, while that kernel's
// writes are still being made visible, so the launch overlaps the flush; it
// calls pdl_wait() before its first global-memory access, which returns once
// every earlier kernel of the stream has completed and its writes are visible.
// No kernel triggers its dependents early: with an early trigger the fused scan's
// CTAs were placed on SMs as WY-128's CTAs drained and the prefill step took
// 0.541 ms instead of 0.482 ms.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Records stage-boundary event i (gdp_set_stage_events) on `s`; no-op when off.
// Slots: 0 entry, 1 after the chunk tables, 2 after the WY stage (transition
// block, solve_tril, w/u), 3 after the state recurrence, 4 after the output.
void record_stage(int i, cudaStream_t s);

}  // namespace gdp
