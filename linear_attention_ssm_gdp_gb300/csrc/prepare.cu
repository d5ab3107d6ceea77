// Fused prepare step for the Gated Delta Product: split, GQA-expand, fold the
// Householder copies into the sequence, and gate, in one launch.
//
// Follows the Megatron-core API page "core.ssm.ops.gdp.prepare" (module
// overview; softplus; gdp_prepare_kernel; gdp_decode_prepare;
// gdp_prefill_prepare):
//   x[n,t,:] = [ value: M*H*P (copy-major) | key: M*G*N | query: G*N ]
//   v[n, t*M+j, h, :] = value block of copy j, head h      (a contiguous copy)
//   k[n, t*M+j, h, :] = key block of copy j, group h/(H/G)
//   q: prefill one row per token; decode one row per copy, the query on the
//      last copy and +0 elsewhere
//   beta = sigmoid(b) per (copy, head); g = -exp(A_log) * softplus(a + dt_bias)
//      per head, on the token (prefill) or on the first copy (decode).
//
// GB300 design: a persistent grid (a multiple of the SM count) walks token
// rows with 16-byte vector loads/stores (the row's value block maps onto the
// output contiguously, key/query heads are 16-byte-aligned runs), so the
// kernel is a pure HBM stream. When a row fits one pass of the block
// (prepare_rows_kernel, the prefill rows of the usual head sizes) each CTA
// already has the next row's loads in flight while it stores the current one;
// longer rows go through prepare_kernel, a row at a time. The gates use
// the CUDA math library's expf/log1pf and IEEE division, one fp32 operation at
// a time; this translation unit is compiled with --fmad=false so no
// multiply-add is contracted, which keeps beta and g bitwise equal to the
// eager PyTorch composition of the same fp32 operations.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gdp_internal.cuh"

namespace gdp {
namespace {

__device__ __forceinline__ float to_f32(const void* base, int64_t idx, int dt) {
  if (dt == GDP_F32) return static_cast<const float*>(base)[idx];
  const unsigned short bits = static_cast<const unsigned short*>(base)[idx];
  if (dt == GDP_BF16) return __uint_as_float(static_cast<unsigned>(bits) << 16);
  return __half2float(__ushort_as_half(bits));
}

__device__ __forceinline__ float softplus_page(float x) {
  // identity strictly above 20, else log1p(exp(x)), in fp32
  return x > 20.0f ? x : log1pf(expf(x));
}

struct PrepArgs {
  const uint8_t* x;
  int64_t x_sn_b, x_st_b;  // byte strides
  const void* ba;
  int64_t ba_sn, ba_st;    // element strides
  const float* A_log;
  const float* dt_bias;
  int n, T, M, H, G, P, N, dt, es;
  uint8_t* q;
  uint8_t* k;
  uint8_t* v;
  float* beta;
  float* g;
};

// VB: bytes moved per vector access (16, or the element size when the
// alignment of some pointer/stride/head size forbids 16-byte vectors).
template <int VB, bool DECODE>
__global__ void __launch_bounds__(256) prepare_kernel(PrepArgs a) {
  using VT = typename std::conditional<VB == 16, uint4,
             typename std::conditional<VB == 4, uint32_t, uint16_t>::type>::type;
  constexpr int U = 8;  // vectors in flight per thread
  const int64_t rows = (int64_t)a.n * a.T;
  const int hpg = a.H / a.G;
  const int64_t vrow_b = (int64_t)a.M * a.H * a.P * a.es;   // value bytes per token
  const int64_t krow_b = (int64_t)a.M * a.H * a.N * a.es;   // key bytes per token (out)
  const int64_t head_kb = (int64_t)a.N * a.es;              // bytes per key/query head
  const int64_t kbase_b = vrow_b;                            // key block offset in x row
  const int64_t qbase_b = kbase_b + (int64_t)a.M * a.G * head_kb;
  const int64_t qrow_b = (DECODE ? (int64_t)a.M : 1) * a.H * head_kb;
  const int nv = (int)(vrow_b / VB), nk = (int)(krow_b / VB), nq = (int)(qrow_b / VB);
  const int head_v = (int)(head_kb / VB);  // vectors per head row

  const int ntot = nv + nk + nq;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const int64_t in = r / a.T, t = r - in * a.T;
    const uint8_t* xr = a.x + in * a.x_sn_b + t * a.x_st_b;
    VT* vdst = reinterpret_cast<VT*>(a.v + r * vrow_b);
    VT* kdst = reinterpret_cast<VT*>(a.k + r * krow_b);
    VT* qdst = reinterpret_cast<VT*>(a.q + r * qrow_b);
    // one index space over the row's value, key and query outputs, so that a
    // thread has all of its loads for the row in flight before it stores
    for (int c0 = threadIdx.x; c0 < ntot; c0 += blockDim.x * U) {
      VT buf[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * blockDim.x;
        if (c < nv) {  // value: contiguous copy of the row's value block
          buf[u] = __ldcs(reinterpret_cast<const VT*>(xr) + c);
        } else if (c < nv + nk) {  // key: output head (j, h) reads group (j, h / hpg)
          const int ck = c - nv;
          const int jh = ck / head_v, w = ck - jh * head_v;
          const int j = jh / a.H, h = jh - j * a.H;
          buf[u] = __ldcs(reinterpret_cast<const VT*>(
                              xr + kbase_b + ((int64_t)j * a.G + h / hpg) * head_kb) + w);
        } else if (c < ntot) {  // query: prefill one row per token; decode the last copy
          const int cq = c - nv - nk;
          const int jh = cq / head_v, w = cq - jh * head_v;
          const int j = DECODE ? jh / a.H : a.M - 1;
          const int h = DECODE ? jh - j * a.H : jh;
          if (j == a.M - 1)
            buf[u] = __ldcs(reinterpret_cast<const VT*>(xr + qbase_b +
                                                        (int64_t)(h / hpg) * head_kb) + w);
          else
            buf[u] = VT{};  // +0.0 in every dtype
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * blockDim.x;
        if (c < nv) __stcs(vdst + c, buf[u]);
        else if (c < nv + nk) __stcs(kdst + (c - nv), buf[u]);
        else if (c < ntot) __stcs(qdst + (c - nv - nk), buf[u]);
      }
    }
    // gates
    const int64_t bar = in * a.ba_sn + t * a.ba_st;
    const int MH = a.M * a.H;
    for (int i = threadIdx.x; i < MH; i += blockDim.x) {
      const float b = to_f32(a.ba, bar + i, a.dt);
      a.beta[r * MH + i] = 1.0f / (1.0f + expf(-b));
    }
    const int ng = DECODE ? MH : a.H;
    for (int i = threadIdx.x; i < ng; i += blockDim.x) {
      const int j = DECODE ? i / a.H : 0;
      const int h = DECODE ? i - j * a.H : i;
      float gv = 0.0f;
      if (j == 0) {
        const float av = to_f32(a.ba, bar + MH + h, a.dt);
        const float sp = softplus_page(av + a.dt_bias[h]);
        gv = -(expf(a.A_log[h]) * sp);
      }
      a.g[r * ng + i] = gv;
    }
  }
}

// Rows that fit one pass of the block (at most 256 x kPU 16-byte vectors, at
// most 256 gate columns): each CTA loads row r + gridDim.x, gate inputs
// included, before it stores row r, so every thread keeps a row of loads in
// flight while it stores and gates the previous one. Loaded values stay raw
// until they are stored (a conversion on arrival would stall the warp on its
// own prefetch). Same copies and the same fp32 gate operations as
// prepare_kernel.
constexpr int kPU = 5;

struct RowGeo {
  int64_t vrow_b, krow_b, head_kb, kbase_b, qbase_b, qrow_b;
  int nv, nk, nq, head_v, hpg, MH;
};

__device__ __forceinline__ RowGeo row_geo(const PrepArgs& a, bool decode) {
  RowGeo g;
  g.hpg = a.H / a.G;
  g.vrow_b = (int64_t)a.M * a.H * a.P * a.es;
  g.krow_b = (int64_t)a.M * a.H * a.N * a.es;
  g.head_kb = (int64_t)a.N * a.es;
  g.kbase_b = g.vrow_b;
  g.qbase_b = g.kbase_b + (int64_t)a.M * a.G * g.head_kb;
  g.qrow_b = (decode ? (int64_t)a.M : 1) * a.H * g.head_kb;
  g.nv = (int)(g.vrow_b / 16);
  g.nk = (int)(g.krow_b / 16);
  g.nq = (int)(g.qrow_b / 16);
  g.head_v = (int)(g.head_kb / 16);
  g.MH = a.M * a.H;
  return g;
}

struct RowBuf {
  uint4 x[kPU];
  uint32_t b, av;  // raw gate inputs: b for column tid < M*H, a for head tid < H
};

__device__ __forceinline__ uint32_t raw_ld(const void* base, int64_t idx, int dt) {
  return dt == GDP_F32 ? static_cast<const uint32_t*>(base)[idx]
                       : static_cast<const unsigned short*>(base)[idx];
}
__device__ __forceinline__ float raw_f32(uint32_t r, int dt) {
  if (dt == GDP_F32) return __uint_as_float(r);
  if (dt == GDP_BF16) return __uint_as_float(r << 16);
  return __half2float(__ushort_as_half((unsigned short)r));
}

template <bool DECODE>
__device__ __forceinline__ void load_row(const PrepArgs& a, const RowGeo& g, int64_t r,
                                         RowBuf& rb) {
  const int64_t in = r / a.T, t = r - in * a.T;
  const uint8_t* xr = a.x + in * a.x_sn_b + t * a.x_st_b;
  const int tid = threadIdx.x;
#pragma unroll
  for (int u = 0; u < kPU; ++u) {
    const int c = tid + u * 256;
    if (c < g.nv) {
      rb.x[u] = __ldcs(reinterpret_cast<const uint4*>(xr) + c);
    } else if (c < g.nv + g.nk) {
      const int ck = c - g.nv;
      const int jh = ck / g.head_v, w = ck - jh * g.head_v;
      const int j = jh / a.H, h = jh - j * a.H;
      rb.x[u] = __ldcs(reinterpret_cast<const uint4*>(
                           xr + g.kbase_b + ((int64_t)j * a.G + h / g.hpg) * g.head_kb) + w);
    } else if (c < g.nv + g.nk + g.nq) {
      const int cq = c - g.nv - g.nk;
      const int jh = cq / g.head_v, w = cq - jh * g.head_v;
      const int j = DECODE ? jh / a.H : a.M - 1;
      const int h = DECODE ? jh - j * a.H : jh;
      rb.x[u] = make_uint4(0u, 0u, 0u, 0u);  // +0.0 in every dtype
      if (j == a.M - 1)
        rb.x[u] = __ldcs(reinterpret_cast<const uint4*>(xr + g.qbase_b +
                                                        (int64_t)(h / g.hpg) * g.head_kb) + w);
    }
  }
  const int64_t bar = in * a.ba_sn + t * a.ba_st;
  if (tid < g.MH) rb.b = raw_ld(a.ba, bar + tid, a.dt);
  if (tid < a.H) rb.av = raw_ld(a.ba, bar + g.MH + tid, a.dt);
}

template <bool DECODE>
__device__ __forceinline__ void store_row(const PrepArgs& a, const RowGeo& g, int64_t r,
                                          const RowBuf& rb) {
  const int tid = threadIdx.x;
  uint4* vdst = reinterpret_cast<uint4*>(a.v + r * g.vrow_b);
  uint4* kdst = reinterpret_cast<uint4*>(a.k + r * g.krow_b);
  uint4* qdst = reinterpret_cast<uint4*>(a.q + r * g.qrow_b);
#pragma unroll
  for (int u = 0; u < kPU; ++u) {
    const int c = tid + u * 256;
    if (c < g.nv) __stcs(vdst + c, rb.x[u]);
    else if (c < g.nv + g.nk) __stcs(kdst + (c - g.nv), rb.x[u]);
    else if (c < g.nv + g.nk + g.nq) __stcs(qdst + (c - g.nv - g.nk), rb.x[u]);
  }
  if (tid < g.MH) a.beta[r * g.MH + tid] = 1.0f / (1.0f + expf(-raw_f32(rb.b, a.dt)));
  const int ng = DECODE ? g.MH : a.H;
  if (tid < ng) {
    const int j = DECODE ? tid / a.H : 0;
    const int h = DECODE ? tid - j * a.H : tid;
    float gv = 0.0f;
    if (j == 0) {
      const float sp = softplus_page(raw_f32(rb.av, a.dt) + a.dt_bias[h]);
      gv = -(expf(a.A_log[h]) * sp);
    }
    a.g[r * ng + tid] = gv;
  }
}

template <bool DECODE>
__global__ void __launch_bounds__(256, 4) prepare_rows_kernel(PrepArgs a) {
  const int64_t rows = (int64_t)a.n * a.T;
  const RowGeo g = row_geo(a, DECODE);
  int64_t r = blockIdx.x;
  if (r >= rows) return;
  RowBuf cur;
  load_row<DECODE>(a, g, r, cur);
  for (; r < rows; r += gridDim.x) {
    RowBuf nxt;
    const int64_t rn = r + gridDim.x;
    if (rn < rows) load_row<DECODE>(a, g, rn, nxt);
    store_row<DECODE>(a, g, r, cur);
    cur = nxt;
  }
}

template <int VB>
cudaError_t launch_vb(const PrepArgs& a, bool decode, cudaStream_t s) {
  const int64_t rows = (int64_t)a.n * a.T;
  const int64_t cap = (int64_t)sm_count() * 8;  // 8 resident 256-thread CTAs per SM
  const int grid = (int)(rows < cap ? rows : cap);
  if (decode)
    prepare_kernel<VB, true><<<grid, 256, 0, s>>>(a);
  else
    prepare_kernel<VB, false><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prepare(const void* x, int64_t x_sn, int64_t x_st, const void* ba,
                           int64_t ba_sn, int64_t ba_st, const float* A_log,
                           const float* dt_bias, int n, int T, int M, int H, int G, int P,
                           int N, gdp_dtype dt, bool decode, void* q, void* k, void* v,
                           float* beta, float* g, cudaStream_t stream) {
  if ((int64_t)n * T == 0) return cudaSuccess;
  PrepArgs a;
  a.es = dt == GDP_F32 ? 4 : 2;
  a.x = static_cast<const uint8_t*>(x);
  a.x_sn_b = x_sn * a.es;
  a.x_st_b = x_st * a.es;
  a.ba = ba;
  a.ba_sn = ba_sn;
  a.ba_st = ba_st;
  a.A_log = A_log;
  a.dt_bias = dt_bias;
  a.n = n; a.T = T; a.M = M; a.H = H; a.G = G; a.P = P; a.N = N; a.dt = (int)dt;
  a.q = static_cast<uint8_t*>(q);
  a.k = static_cast<uint8_t*>(k);
  a.v = static_cast<uint8_t*>(v);
  a.beta = beta;
  a.g = g;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool vec16 = al16(x) && al16(q) && al16(k) && al16(v) && (a.x_sn_b % 16 == 0) &&
                     (a.x_st_b % 16 == 0) && ((int64_t)P * a.es % 16 == 0) &&
                     ((int64_t)N * a.es % 16 == 0);
  if (vec16) {
    const int64_t ntot = ((int64_t)M * H * P + (int64_t)(decode ? 2 * M : M + 1) * H * N) *
                         a.es / 16;
    if (ntot <= 256 * kPU && M * H <= 256) {
      const int64_t rows = (int64_t)n * T;
      int per_sm = 0;
      cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, decode ? prepare_rows_kernel<true> : prepare_rows_kernel<false>, 256, 0);
      if (e != cudaSuccess) return e;
      const int64_t cap = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
      const int grid = (int)(rows < cap ? rows : cap);
      if (decode)
        prepare_rows_kernel<true><<<grid, 256, 0, stream>>>(a);
      else
        prepare_rows_kernel<false><<<grid, 256, 0, stream>>>(a);
      return cudaGetLastError();
    }
    return launch_vb<16>(a, decode, stream);
  }
  if (a.es == 4) return launch_vb<4>(a, decode, stream);
  return launch_vb<2>(a, decode, stream);
}

}  // namespace gdp
