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
// value head, 32-column slice) with K/32 warps; warp w holds state rows
// [32w, 32w + 32) of all 32 columns (lane = column), so every warp reads and
// writes whole 128-byte rows, each element once (streaming cache hints). A
// step's inputs (k, q, v, beta, e^g) are staged in shared memory for up to 16
// steps with one batched load and k, q are normalised there once per step;
// in the step loop the key/query rows are warp-broadcast 16-byte loads, the
// per-element arithmetic runs on packed pairs of rows (f32x2 multiply and
// fused multiply-add: half the instructions, the same per-element rounding),
// and the column sums over K combine per-thread partials across the K/32 warps
// through shared memory (two barriers per step).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gdp_internal.cuh"

namespace gdp {
namespace {

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float ldf(const __half* p) { return __half2float(*p); }

// Packed pairs of fp32 (Blackwell f32x2 arithmetic: each lane of the pair is
// rounded exactly like the scalar fp32 operation).
typedef unsigned long long f2;
__device__ __forceinline__ f2 pk2(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 upk2(f2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

constexpr int kCtaCols = 32;  // value columns per CTA (one per lane)
constexpr int kLC = 16;       // steps staged in shared memory at a time

// Shared memory per CTA: normalised k and q rows [kLC][K] fp32, the CTA's value
// columns [kLC][32], beta and e^g per step, and two double-buffered
// [K/32][32] tables of per-warp partial column sums.
template <int K>
constexpr int rec_smem() {
  return (2 * kLC * K + kLC * kCtaCols + 2 * kLC + 4 * (K / 32) * 32) * 4;
}

// Thread layout: K/32 warps; warp w owns state rows [32 w, 32 w + 32), lane l
// owns value column cbase + l, so a warp touches full 128-byte rows of the
// state. Column sums over K are in-thread over 32 rows, then across the K/32
// warps through shared memory.
template <typename Tin, int KW>
__global__ void __launch_bounds__(KW * 32, KW >= 4 ? 24 / KW : 8)
recurrent_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
                 const float* __restrict__ beta, const float* __restrict__ g,
                 float* __restrict__ state, int L, int H, int HV, int V, float scale,
                 int l2norm, float* __restrict__ o) {
  constexpr int K = KW * 32;
  extern __shared__ __align__(16) float smr[];
  float* kn = smr;                      // [kLC][K]
  float* qn = kn + kLC * K;             // [kLC][K]
  float* vs = qn + kLC * K;             // [kLC][32]
  float* bt = vs + kLC * kCtaCols;      // [kLC]
  float* eg = bt + kLC;                 // [kLC]
  float* part = eg + kLC;               // [2][KW][32]  h^T k partials
  float* parto = part + 2 * KW * 32;    // [2][KW][32]  h^T q partials
  const int rh = blockIdx.x;  // request * HV + hv
  const int r = rh / HV, hv = rh - r * HV, kh = hv / (HV / H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cbase = blockIdx.y * kCtaCols;
  const int c = cbase + lane;
  const bool active = c < V;
  const int nth = KW * 32;
  float* st = state + (int64_t)rh * K * V + (int64_t)(warp * 32) * V + c;
  f2 h[16];  // rows (2i, 2i + 1) of this thread's 32, packed
#pragma unroll
  for (int i = 0; i < 16; ++i)
    h[i] = active ? pk2(__ldcs(st + (int64_t)(2 * i) * V), __ldcs(st + (int64_t)(2 * i + 1) * V))
                  : pk2(0.f, 0.f);
  int buf = 0;
  for (int e0 = 0; e0 < L; e0 += kLC) {
    const int lc = min(kLC, L - e0);
    const int64_t re0 = (int64_t)r * L + e0;
    __syncthreads();  // the previous batch has been consumed
    for (int idx = tid; idx < lc * K; idx += nth) {
      const int e = idx / K, cc = idx - e * K;
      kn[idx] = ldf(k + ((re0 + e) * H + kh) * K + cc);
      qn[idx] = ldf(q + ((re0 + e) * H + kh) * K + cc);
    }
    for (int idx = tid; idx < lc * kCtaCols; idx += nth) {
      const int e = idx / kCtaCols, cc = idx - e * kCtaCols;
      vs[idx] = (cbase + cc < V) ? ldf(v + ((re0 + e) * HV + hv) * V + cbase + cc) : 0.f;
    }
    if (tid < lc) {
      bt[tid] = beta[(re0 + tid) * HV + hv];
      eg[tid] = expf(g[(re0 + tid) * HV + hv]);
    }
    __syncthreads();
    if (l2norm) {  // one warp per row, each row normalised once for the whole CTA
      for (int rr = warp; rr < 2 * lc; rr += KW) {
        float* x = rr < lc ? kn + rr * K : qn + (rr - lc) * K;
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < KW; ++i) ss += x[lane + 32 * i] * x[lane + 32 * i];
        const float rn = 1.0f / sqrtf(warp_sum(ss) + 1e-6f);
#pragma unroll
        for (int i = 0; i < KW; ++i) x[lane + 32 * i] *= rn;
      }
      __syncthreads();
    }
    for (int e = 0; e < lc; ++e) {
      const ulonglong2* kr = reinterpret_cast<const ulonglong2*>(kn + e * K + warp * 32);
      const ulonglong2* qr = reinterpret_cast<const ulonglong2*>(qn + e * K + warp * 32);
      const f2 d2 = pk2(eg[e], eg[e]);
      f2 pa = pk2(0.f, 0.f), pb2 = pa;
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4) {  // broadcast 16-byte loads of this warp's 32 key rows
        const ulonglong2 kk = kr[i4];
        h[2 * i4] = mul2(h[2 * i4], d2);
        h[2 * i4 + 1] = mul2(h[2 * i4 + 1], d2);
        pa = fma2(h[2 * i4], kk.x, pa);
        pb2 = fma2(h[2 * i4 + 1], kk.y, pb2);
      }
      const float2 pav = upk2(pa), pbv = upk2(pb2);
      const float p = (pav.x + pav.y) + (pbv.x + pbv.y);
      float* pb = part + buf * KW * 32;
      pb[warp * 32 + lane] = p;
      __syncthreads();
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < KW; ++w) s += pb[w * 32 + lane];
      const float delta = bt[e] * (vs[e * kCtaCols + lane] - s);
      const f2 dl2 = pk2(delta, delta);
      f2 oa = pk2(0.f, 0.f), ob2 = oa;
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4) {
        const ulonglong2 kk = kr[i4], qq = qr[i4];
        h[2 * i4] = fma2(kk.x, dl2, h[2 * i4]);
        h[2 * i4 + 1] = fma2(kk.y, dl2, h[2 * i4 + 1]);
        oa = fma2(h[2 * i4], qq.x, oa);
        ob2 = fma2(h[2 * i4 + 1], qq.y, ob2);
      }
      const float2 oav = upk2(oa), obv = upk2(ob2);
      const float po = (oav.x + oav.y) + (obv.x + obv.y);
      float* ob = parto + buf * KW * 32;
      ob[warp * 32 + lane] = po;
      __syncthreads();
      if (warp == 0 && active) {
        float so = 0.f;
#pragma unroll
        for (int w = 0; w < KW; ++w) so += ob[w * 32 + lane];
        o[((re0 + e) * HV + hv) * V + c] = scale * so;
      }
      buf ^= 1;  // the next step writes the other buffers; reuse is two barriers away
    }
  }
  if (active) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 hv2 = upk2(h[i]);
      __stcs(st + (int64_t)(2 * i) * V, hv2.x);
      __stcs(st + (int64_t)(2 * i + 1) * V, hv2.y);
    }
  }
}

template <typename Tin, int KW>
cudaError_t launch_k(const dim3& grid, const void* q, const void* k, const void* v,
                     const float* beta, const float* g, float* state, int L, int H, int HV,
                     int V, float scale, int l2norm, float* o, cudaStream_t s) {
  constexpr int smem = rec_smem<KW * 32>();
  cudaError_t e = cudaFuncSetAttribute(recurrent_kernel<Tin, KW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  recurrent_kernel<Tin, KW><<<grid, KW * 32, smem, s>>>(
      static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v), beta,
      g, state, L, H, HV, V, scale, l2norm, o);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t run(const void* q, const void* k, const void* v, const float* beta, const float* g,
                float* state, int n, int L, int H, int HV, int K, int V, float scale, int l2norm,
                float* o, cudaStream_t s) {
  const dim3 grid((unsigned)((int64_t)n * HV), (unsigned)cdiv(V, kCtaCols));
  switch (K) {
    case 32: return launch_k<Tin, 1>(grid, q, k, v, beta, g, state, L, H, HV, V, scale, l2norm, o, s);
    case 64: return launch_k<Tin, 2>(grid, q, k, v, beta, g, state, L, H, HV, V, scale, l2norm, o, s);
    case 128: return launch_k<Tin, 4>(grid, q, k, v, beta, g, state, L, H, HV, V, scale, l2norm, o, s);
    default: return launch_k<Tin, 8>(grid, q, k, v, beta, g, state, L, H, HV, V, scale, l2norm, o, s);
  }
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
