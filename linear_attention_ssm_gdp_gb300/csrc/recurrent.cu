// Fused recurrent update for one decode step of the Gated Delta Product.
//
// The prepare page ("core.ssm.ops.gdp.prepare", decode bullet) feeds a fused
// recurrent gated-delta update that walks the Householder copies as a
// sequence: per request r and value head hv (key/query head hv / (HV/H)) the
// fp32 state h = S^T [K, V] takes L = S*M steps, each with its own inputs,
//     h <- e^{g} h ;  delta = beta (v - h^T k) ;  h <- h + k delta^T ;
//     o = scale h^T q,
// which is S <- e^g S (I - beta k k^T) + beta v k^T followed by o = scale S q.
//
// GB300 design: the work is the fp32 state read + write (8 bytes per state
// element per call), so the kernel is an HBM stream: one CTA per (request,
// value head, 128-column slice), 16 warps, each warp owning 8 columns and
// every lane K/32 rows, so a lane holds its K/32 x 8 state block in registers
// for all L steps. The column reductions h^T k and h^T q are warp shuffles;
// each state element is read once and written once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gdp_internal.cuh"

namespace gdp {
namespace {

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float ldf(const __half* p) { return __half2float(*p); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

constexpr int kCols = 8;      // columns per warp
constexpr int kWarps = 16;    // warps per CTA -> 128 columns per CTA

template <typename Tin, int KR>
__global__ void __launch_bounds__(kWarps * 32)
recurrent_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                 const float* __restrict__ beta, const float* __restrict__ g,
                 float* __restrict__ state, int L, int H, int HV, int V, float scale,
                 int l2norm, float* __restrict__ o) {
  constexpr int K = KR * 32;
  const int rh = blockIdx.x;  // request * HV + hv
  const int r = rh / HV, hv = rh - r * HV, kh = hv / (HV / H);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.y * (kWarps * kCols) + warp * kCols;
  if (c0 >= V) return;  // V % 8 == 0: a warp is either fully in or fully out
  float* st = state + (int64_t)rh * K * V;
  float h[KR][kCols];
#pragma unroll
  for (int i = 0; i < KR; ++i) {
    const float4* p = reinterpret_cast<const float4*>(st + (int64_t)(lane + 32 * i) * V + c0);
    const float4 a = p[0], b = p[1];
    h[i][0] = a.x; h[i][1] = a.y; h[i][2] = a.z; h[i][3] = a.w;
    h[i][4] = b.x; h[i][5] = b.y; h[i][6] = b.z; h[i][7] = b.w;
  }
  for (int e = 0; e < L; ++e) {
    const int64_t re = (int64_t)r * L + e;
    float kv[KR], qv[KR];
    float skk = 0.f, sqq = 0.f;
#pragma unroll
    for (int i = 0; i < KR; ++i) {
      kv[i] = ldf(k + (re * H + kh) * K + lane + 32 * i);
      qv[i] = ldf(q + (re * H + kh) * K + lane + 32 * i);
      skk += kv[i] * kv[i];
      sqq += qv[i] * qv[i];
    }
    if (l2norm) {
      const float rk = 1.0f / sqrtf(warp_sum(skk) + 1e-6f);
      const float rq = 1.0f / sqrtf(warp_sum(sqq) + 1e-6f);
#pragma unroll
      for (int i = 0; i < KR; ++i) { kv[i] *= rk; qv[i] *= rq; }
    }
    float vv[kCols];
    {
      const Tin* vp = v + (re * HV + hv) * V + c0;
#pragma unroll
      for (int c = 0; c < kCols; ++c) vv[c] = ldf(vp + c);
    }
    const float bt = beta[re * HV + hv];
    const float eg = expf(g[re * HV + hv]);
    float out[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c) {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < KR; ++i) {
        h[i][c] *= eg;
        part += h[i][c] * kv[i];
      }
      const float delta = bt * (vv[c] - warp_sum(part));
      float po = 0.f;
#pragma unroll
      for (int i = 0; i < KR; ++i) {
        h[i][c] += kv[i] * delta;
        po += h[i][c] * qv[i];
      }
      out[c] = scale * warp_sum(po);
    }
    if (lane == 0) {
      float4* op = reinterpret_cast<float4*>(o + (re * HV + hv) * V + c0);
      op[0] = make_float4(out[0], out[1], out[2], out[3]);
      op[1] = make_float4(out[4], out[5], out[6], out[7]);
    }
  }
#pragma unroll
  for (int i = 0; i < KR; ++i) {
    float4* p = reinterpret_cast<float4*>(st + (int64_t)(lane + 32 * i) * V + c0);
    p[0] = make_float4(h[i][0], h[i][1], h[i][2], h[i][3]);
    p[1] = make_float4(h[i][4], h[i][5], h[i][6], h[i][7]);
  }
}

template <typename Tin>
cudaError_t run(const void* q, const void* k, const void* v, const float* beta, const float* g,
                float* state, int n, int L, int H, int HV, int K, int V, float scale, int l2norm,
                float* o, cudaStream_t s) {
  const dim3 grid((unsigned)((int64_t)n * HV), (unsigned)cdiv(V, kWarps * kCols));
  const dim3 block(kWarps * 32);
  auto qq = static_cast<const Tin*>(q);
  auto kk = static_cast<const Tin*>(k);
  auto vv = static_cast<const Tin*>(v);
  switch (K) {
    case 32: recurrent_kernel<Tin, 1><<<grid, block, 0, s>>>(qq, kk, vv, beta, g, state, L, H, HV, V, scale, l2norm, o); break;
    case 64: recurrent_kernel<Tin, 2><<<grid, block, 0, s>>>(qq, kk, vv, beta, g, state, L, H, HV, V, scale, l2norm, o); break;
    case 128: recurrent_kernel<Tin, 4><<<grid, block, 0, s>>>(qq, kk, vv, beta, g, state, L, H, HV, V, scale, l2norm, o); break;
    default: recurrent_kernel<Tin, 8><<<grid, block, 0, s>>>(qq, kk, vv, beta, g, state, L, H, HV, V, scale, l2norm, o); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(const void* q, const void* k, const void* v, const float* beta,
                             const float* g, float* state, int n, int L, int H, int HV, int K,
                             int V, float scale, int l2norm, gdp_dtype dt, float* o,
                             cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  switch (dt) {
    case GDP_BF16:
      return run<__nv_bfloat16>(q, k, v, beta, g, state, n, L, H, HV, K, V, scale, l2norm, o, stream);
    case GDP_F16:
      return run<__half>(q, k, v, beta, g, state, n, L, H, HV, K, V, scale, l2norm, o, stream);
    default:
      return run<float>(q, k, v, beta, g, state, n, L, H, HV, K, V, scale, l2norm, o, stream);
  }
}

}  // namespace gdp
