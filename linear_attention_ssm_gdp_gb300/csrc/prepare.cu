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
// kernel is a pure HBM stream. Prefill rows, and decode rows longer than one
// pass of a 256-thread block, stream through a shared-memory ring of raw rows
// filled by cp.async (prepare_ring_kernel: each CTA has its next two rows in
// flight without holding registers while it stores the current one); shorter
// decode rows take prepare_rows_kernel, which keeps the next row's loads in
// registers; rows too long for the ring, or not 16-byte aligned, go through
// prepare_kernel, a row at a time. The gates use
// the CUDA math library's expf/log1pf and IEEE division, one fp32 operation at
// a time; this translation unit is compiled with --fmad=false so no
// multiply-add is contracted, which keeps beta and g bitwise equal to the
// eager PyTorch composition of the same fp32 operations.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

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

// Division of non-negative ints below 2^31 by a divisor fixed for the launch,
// as a multiply-high, an add and a shift (Granlund and Montgomery, "Division by
// invariant integers using multiplication", 1994: with s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1, n / d = (umulhi(m, n) + n) >> s). The
// prepare kernels' index arithmetic (vectors per head, heads, heads per
// group) would otherwise be a chain of 32-bit divisions per 16-byte vector.
struct FastDiv {
  uint32_t d, m, s;
  __host__ __device__ FastDiv() : d(1), m(1), s(0) {}
  __host__ explicit FastDiv(uint32_t div) : d(div) {
    s = 0;
    while ((1ull << s) < div) ++s;
    m = (uint32_t)(((1ull << 32) * ((1ull << s) - div)) / div + 1);
  }
  __device__ __forceinline__ int div(int n) const {
    const uint32_t un = (uint32_t)n;
    return (int)((__umulhi(m, un) + un) >> s);
  }
};

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
  FastDiv fd_H, fd_hpg, fd_hv;  // by H, H / G, and the vectors per key/query head
};

// VB: bytes moved per vector access (16, or the element size when the
// alignment of some pointer/stride/head size forbids 16-byte vectors).
template <int VB, bool DECODE>
__global__ void __launch_bounds__(256) prepare_kernel(PrepArgs a) {
  pdl_wait();
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
          const int jh = a.fd_hv.div(ck), w = ck - jh * head_v;
          const int j = a.fd_H.div(jh), h = jh - j * a.H;
          buf[u] = __ldcs(reinterpret_cast<const VT*>(
                              xr + kbase_b + ((int64_t)j * a.G + a.fd_hpg.div(h)) * head_kb) + w);
        } else if (c < ntot) {  // query: prefill one row per token; decode the last copy
          const int cq = c - nv - nk;
          const int jh = a.fd_hv.div(cq), w = cq - jh * head_v;
          const int j = DECODE ? a.fd_H.div(jh) : a.M - 1;
          const int h = DECODE ? jh - j * a.H : jh;
          if (j == a.M - 1)
            buf[u] = __ldcs(reinterpret_cast<const VT*>(xr + qbase_b +
                                                        (int64_t)a.fd_hpg.div(h) * head_kb) + w);
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

// Asynchronous 16-byte global -> shared copy (zero-filled when bytes is 0).
__device__ __forceinline__ void cp16(void* dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   (unsigned)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(bytes)
               : "memory");
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
  pdl_wait();
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

// Long rows (beyond one pass of prepare_rows_kernel: the decode rows, where q
// has a row per copy, and prefill rows with many heads). Each CTA walks rows
// blockIdx.x + i * gridDim.x; the raw x row streams into a ring of kRing
// row buffers in shared memory with cp.async (one commit group per row), so
// the next kRing - 1 rows are in flight without holding registers while the
// threads store the current one: v as a contiguous copy, k and q as one
// 16-byte shared-memory read per output vector (group expansion and decode
// copy placement as prepare_kernel). Same fp32 gate operations.
constexpr int kRing = 3;

// Output stores of the ring kernel: streaming (evict-first) for prefill, whose
// outputs exceed L2; plain for decode, whose outputs stay in L2 for the update.
template <bool DECODE>
__device__ __forceinline__ void st_row(uint4* p, uint4 v) {
  if (DECODE)
    *p = v;
  else
    __stcs(p, v);
}

template <bool DECODE, int NT>
__global__ void __launch_bounds__(NT, 3) prepare_ring_kernel(PrepArgs a, int xrow_v) {
  pdl_wait();
  extern __shared__ uint4 ring[];  // [kRing][xrow_v]
  const int64_t rows = (int64_t)a.n * a.T;
  const RowGeo g = row_geo(a, DECODE);
  const int tid = threadIdx.x;
  const int mine = (int)((rows - blockIdx.x + gridDim.x - 1) / gridDim.x);
  const int ntot = g.nv + g.nk + g.nq;
  const int kb_v = (int)(g.kbase_b / 16), qb_v = (int)(g.qbase_b / 16);
  auto fetch = [&](int i) {  // row i of this CTA into slot i % kRing (always one group)
    if (i < mine) {
      const int64_t r = blockIdx.x + (int64_t)i * gridDim.x;
      const int64_t in = r / a.T, t = r - in * a.T;
      const uint4* src = reinterpret_cast<const uint4*>(a.x + in * a.x_sn_b + t * a.x_st_b);
      uint4* dst = ring + (i % kRing) * xrow_v;
      for (int c = tid; c < xrow_v; c += NT) cp16(dst + c, src + c, 16);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
#pragma unroll
  for (int i = 0; i < kRing - 1; ++i) fetch(i);
  for (int i = 0; i < mine; ++i) {
    fetch(i + kRing - 1);  // into the slot row i - 1 used (freed by the barrier below)
    const int64_t r = blockIdx.x + (int64_t)i * gridDim.x;
    const int64_t in = r / a.T, t = r - in * a.T;
    const int64_t bar = in * a.ba_sn + t * a.ba_st;
    uint32_t b = 0, av = 0;
    if (tid < g.MH) b = raw_ld(a.ba, bar + tid, a.dt);
    if (tid < a.H) av = raw_ld(a.ba, bar + g.MH + tid, a.dt);
    asm volatile("cp.async.wait_group %0;" ::"n"(kRing - 1) : "memory");
    __syncthreads();  // row i is in its slot
    const uint4* s = ring + (i % kRing) * xrow_v;
    uint4* vdst = reinterpret_cast<uint4*>(a.v + r * g.vrow_b);
    uint4* kdst = reinterpret_cast<uint4*>(a.k + r * g.krow_b);
    uint4* qdst = reinterpret_cast<uint4*>(a.q + r * g.qrow_b);
    for (int c = tid; c < ntot; c += NT) {
      if (c < g.nv) {  // value: contiguous copy of the row's value block
        st_row<DECODE>(vdst + c, s[c]);
      } else if (c < g.nv + g.nk) {  // key: output head (j, h) reads group (j, h / hpg)
        const int ck = c - g.nv;
        const int jh = a.fd_hv.div(ck), w = ck - jh * g.head_v;
        const int j = a.fd_H.div(jh), h = jh - j * a.H;
        st_row<DECODE>(kdst + ck, s[kb_v + (j * a.G + a.fd_hpg.div(h)) * g.head_v + w]);
      } else {  // query: prefill one row per token; decode the last copy, +0 elsewhere
        const int cq = c - g.nv - g.nk;
        const int jh = a.fd_hv.div(cq), w = cq - jh * g.head_v;
        const int j = DECODE ? a.fd_H.div(jh) : a.M - 1;
        const int h = DECODE ? jh - j * a.H : jh;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (j == a.M - 1) val = s[qb_v + a.fd_hpg.div(h) * g.head_v + w];
        st_row<DECODE>(qdst + cq, val);
      }
    }
    if (tid < g.MH) a.beta[r * g.MH + tid] = 1.0f / (1.0f + expf(-raw_f32(b, a.dt)));
    const int ng = DECODE ? g.MH : a.H;
    if (tid < ng) {
      const int j = DECODE ? tid / a.H : 0;
      const int h = DECODE ? tid - j * a.H : tid;
      float gv = 0.0f;
      if (j == 0) {
        const float sp = softplus_page(raw_f32(av, a.dt) + a.dt_bias[h]);
        gv = -(expf(a.A_log[h]) * sp);
      }
      a.g[r * ng + tid] = gv;
    }
    __syncthreads();  // slot i % kRing is read: row i + kRing may land there
  }
}

// ---------------------------------------------------------------------------
// Short causal conv fused with prepare. The step before prepare in the layer
// (the prepare page's module overview: "padding handled by the conv kernel
// upstream (a -1 slot zeroes its conv output, which propagates here)") is a
// depthwise causal conv of width W over the pre-conv activations xp [n, T, C]
// (C = M*H*P + M*G*N + G*N, the channel layout prepare splits), followed by
// SiLU:  z = bias[c] + sum_i w[c][i] xin[t - (W-1) + i][c],  y = z / (1 + e^-z),
// rounded to the activation dtype. Each sequence continues from its conv state
// (the last W-1 inputs before it, oldest first, [.., C, W-1] in the activation
// dtype; zeros without one). Here the conv output never reaches HBM: each
// thread keeps a sliding window of W-1 inputs for 16 bytes of channels, walks a
// tile of consecutive tokens, and writes the SiLU outputs straight to their
// q/k/v destinations (group expansion and copy placement as prepare_kernel).
// CTAs of channel segment 0 also compute the gates of their rows.
struct ConvArgs {
  PrepArgs pa;               // x = xp (pre-conv), strides in bytes
  const float* w;            // [C][W]
  const float* bias;         // [C] or null
  int W, C, RT;              // taps, channels, token rows per tile (prefill)
  const uint8_t* st_in;      // prefill: [N_seq][C][W-1] or null; decode: the pool
  uint8_t* st_out;           // prefill: [N_seq][C][W-1] or null; decode: the pool
  const int* cu;             // prefill varlen offsets [N_seq + 1] (n == 1) or null
  int N_seq;
  const int* slot;           // decode: [n] pool entries (-1 padding)
  int n_slots;
  int* status;               // decode: set to 1 for an out-of-range or repeated slot
};

template <typename T>
__device__ __forceinline__ float cv_ld(const uint8_t* p) {
  return to_f32(p, 0, sizeof(T) == 4 ? GDP_F32 : (std::is_same<T, __half>::value ? GDP_F16 : GDP_BF16));
}

template <typename T, int VE>
__device__ __forceinline__ void cv_unpack(uint4 u, float* f) {
  if constexpr (VE == 4) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  } else {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (std::is_same<T, __half>::value) {
        f[2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xffffu)));
        f[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
      } else {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    }
  }
}

template <typename T, int VE>
__device__ __forceinline__ uint4 cv_pack(const float* f) {
  if constexpr (VE == 4) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      unsigned short a, b;
      if constexpr (std::is_same<T, __half>::value) {
        a = __half_as_ushort(__float2half_rn(f[2 * i]));
        b = __half_as_ushort(__float2half_rn(f[2 * i + 1]));
      } else {
        a = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * i]));
        b = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * i + 1]));
      }
      w[i] = (uint32_t)a | ((uint32_t)b << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Where one 16-byte vector of post-conv channels c0.. (within one head) goes,
// worked out once per thread: element offset of its first destination inside
// a token row's block of the output, the row stride of that output, and the
// number of destinations (the heads of a key/query group) spaced N apart.
struct CvDst {
  uint8_t* base;   // v, k or q
  int64_t off;     // elements, first destination in row 0
  int64_t rstride; // elements per token row
  int count;       // destinations (1 for values, H/G for keys and queries)
  int zcopies;     // decode queries: copies j < M-1 per destination get zeros
};

template <bool DECODE>
__device__ __forceinline__ CvDst cv_plan(const PrepArgs& a, int c0) {
  const int hpg = a.H / a.G;
  const int KB = a.M * a.H * a.P, QB = KB + a.M * a.G * a.N;
  CvDst d;
  d.zcopies = 0;
  if (c0 < KB) {
    const int j = c0 / (a.H * a.P), rem = c0 - j * a.H * a.P, h = rem / a.P, p = rem - h * a.P;
    d.base = a.v;
    d.off = ((int64_t)j * a.H + h) * a.P + p;
    d.rstride = (int64_t)a.M * a.H * a.P;
    d.count = 1;
  } else if (c0 < QB) {
    const int c1 = c0 - KB, j = c1 / (a.G * a.N), rem = c1 - j * a.G * a.N;
    const int gi = rem / a.N, nn = rem - gi * a.N;
    d.base = a.k;
    d.off = ((int64_t)j * a.H + gi * hpg) * a.N + nn;
    d.rstride = (int64_t)a.M * a.H * a.N;
    d.count = hpg;
  } else {
    const int c2 = c0 - QB, gi = c2 / a.N, nn = c2 - gi * a.N;
    d.base = a.q;
    d.count = hpg;
    if (DECODE) {  // the last copy carries the query
      d.off = ((int64_t)(a.M - 1) * a.H + gi * hpg) * a.N + nn;
      d.rstride = (int64_t)a.M * a.H * a.N;
      d.zcopies = a.M - 1;
    } else {
      d.off = (int64_t)gi * hpg * a.N + nn;
      d.rstride = (int64_t)a.H * a.N;
    }
  }
  return d;
}

__device__ __forceinline__ void cv_scatter(const PrepArgs& a, const CvDst& d, int64_t row,
                                           uint4 val) {
  const int es = a.es;
  const int64_t hstride = (int64_t)a.N * es;
  uint8_t* p = d.base + (row * d.rstride + d.off) * es;
  for (int i = 0; i < d.count; ++i) __stcs(reinterpret_cast<uint4*>(p + i * hstride), val);
  if (d.zcopies) {  // decode queries: +0 on the other copies of this token
    const int64_t cstride = (int64_t)a.H * a.N * es;
    for (int j = 1; j <= d.zcopies; ++j)
      for (int i = 0; i < d.count; ++i)
        __stcs(reinterpret_cast<uint4*>(p - j * cstride + i * hstride), make_uint4(0u, 0u, 0u, 0u));
  }
}

// The gates of one token row (prepare's fp32 operations).
template <bool DECODE>
__device__ __forceinline__ void cv_gates(const PrepArgs& a, int64_t r, int i) {
  const int64_t in = r / a.T, t = r - in * a.T;
  const int64_t bar = in * a.ba_sn + t * a.ba_st;
  const int MH = a.M * a.H;
  if (i < MH) a.beta[r * MH + i] = 1.0f / (1.0f + expf(-to_f32(a.ba, bar + i, a.dt)));
  const int ng = DECODE ? MH : a.H;
  if (i < ng) {
    const int j = DECODE ? i / a.H : 0;
    const int h = DECODE ? i - j * a.H : i;
    float gv = 0.0f;
    if (j == 0) {
      const float sp = softplus_page(to_f32(a.ba, bar + MH + h, a.dt) + a.dt_bias[h]);
      gv = -(expf(a.A_log[h]) * sp);
    }
    a.g[r * ng + i] = gv;
  }
}

// Grid: x = token tile (prefill: RT rows of one batch row; decode: the S rows of
// one request), y = segment of 256 channel vectors. 256 threads, one 16-byte
// channel vector each; its conv taps (loaded as contiguous 16-byte vectors)
// stay in registers for the tile. The thread streams its column of the tile's
// input rows (and the W-1 rows before it) through a private ring of kConvD
// slots in shared memory with cp.async, one commit group per row, so kConvD
// loads are in flight without holding registers; it reads back only its own
// slots (no block barrier). The last W-1 raw rows stay in registers; for a row
// near the start of its sequence the entries before the start are taken from
// the sequence's conv state instead. Conv states move as whole 16-byte vectors:
// a thread's VE channels x (W-1) entries are contiguous in [.., C, W-1].
constexpr int kConvRT = 64;  // prefill token rows per tile
constexpr int kConvD = 8;    // rows in flight per thread

template <typename T, int W, bool DECODE>
__global__ void __launch_bounds__(256, 2) conv_prepare_kernel(ConvArgs ca) {
  constexpr int VE = 16 / sizeof(T);  // channels per vector
  constexpr int WS = W > 1 ? W - 1 : 1;
  __shared__ uint4 ring[kConvD][256];
  const PrepArgs& a = ca.pa;
  const int es = a.es;
  const int nvec = ca.C / VE;
  const int tiles_per_row = DECODE ? 1 : (a.T + ca.RT - 1) / ca.RT;
  const int in = blockIdx.x / tiles_per_row;
  const int t0 = DECODE ? 0 : (blockIdx.x - in * tiles_per_row) * ca.RT;
  const int t1 = DECODE ? a.T : min(a.T, t0 + ca.RT);
  const int cv = blockIdx.y * 256 + threadIdx.x;
  const int c0 = cv * VE;
  const bool has = cv < nvec;
  const uint8_t* xrow0 = a.x + (int64_t)in * a.x_sn_b;
  const int nrows = t1 - t0 + W - 1;  // rows streamed: t0-(W-1) .. t1-1
  auto issue = [&](int rr) {          // row t0-(W-1)+rr into its ring slot (before row 0: zeros)
    const int row = t0 - (W - 1) + rr;
    if (rr < nrows)
      cp16(&ring[rr % kConvD][threadIdx.x],
           xrow0 + (int64_t)(row >= 0 ? row : 0) * a.x_st_b + (int64_t)c0 * es, row >= 0 ? 16 : 0);
    asm volatile("cp.async.commit_group;" ::: "memory");  // one group per row (possibly empty)
  };
  if (has)
    for (int rr = 0; rr < kConvD; ++rr) issue(rr);
  // decode: this request's pool entry (-1: padding or rejected)
  int sl = 0;
  if (DECODE) {
    sl = ca.slot[in];
    if (sl != -1) {
      int bad = sl < -1 || sl >= ca.n_slots;
      if (!bad) {
        int dup = 0;
        for (int i = threadIdx.x; i < a.n; i += blockDim.x) dup |= (i != in) & (ca.slot[i] == sl);
        bad = __syncthreads_or(dup);
      }
      if (bad) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && ca.status) atomicExch(ca.status, 1);
        sl = -1;
      }
    }
  }
  if (blockIdx.y == 0) {  // gates of this tile's rows
    const int ng = a.M * a.H;
    for (int idx = threadIdx.x; idx < (t1 - t0) * ng; idx += blockDim.x) {
      const int tt = idx / ng;
      cv_gates<DECODE>(a, (int64_t)in * a.T + t0 + tt, idx - tt * ng);
    }
  }
  if (!has) return;
  float wv[W][VE], bv[VE];
  {
    float wr[W * VE];  // channel-major taps: wr[e * W + i] = w[c0 + e][i]
    const float4* wp = reinterpret_cast<const float4*>(ca.w + (int64_t)c0 * W);
#pragma unroll
    for (int i = 0; i < W * VE / 4; ++i) {
      const float4 f = __ldg(wp + i);
      wr[4 * i] = f.x; wr[4 * i + 1] = f.y; wr[4 * i + 2] = f.z; wr[4 * i + 3] = f.w;
    }
#pragma unroll
    for (int e = 0; e < VE; ++e)
#pragma unroll
      for (int i = 0; i < W; ++i) wv[i][e] = wr[e * W + i];
    if (ca.bias) {
      const float4* bp = reinterpret_cast<const float4*>(ca.bias + c0);
#pragma unroll
      for (int i = 0; i < VE / 4; ++i) {
        const float4 f = __ldg(bp + i);
        bv[4 * i] = f.x; bv[4 * i + 1] = f.y; bv[4 * i + 2] = f.z; bv[4 * i + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e) bv[e] = 0.f;
    }
  }
  const CvDst dst = cv_plan<DECODE>(a, c0);
  if (DECODE && sl < 0) {  // padding request: zero conv output, no state access
    asm volatile("cp.async.wait_all;" ::: "memory");
    for (int t = t0; t < t1; ++t) cv_scatter(a, dst, (int64_t)in * a.T + t, make_uint4(0u, 0u, 0u, 0u));
    return;
  }
  const int64_t sC = (int64_t)ca.C * (W - 1);  // state entries per sequence
  auto st_ptr = [&](const uint8_t* base, int64_t sq) {
    return base + (sq * sC + (int64_t)c0 * (W - 1)) * es;
  };
  float sw[WS][VE];  // the current sequence's state, [entry][channel]
  auto load_state = [&](const uint8_t* base, int64_t sq) {
#pragma unroll
    for (int i = 0; i < WS; ++i)
#pragma unroll
      for (int e = 0; e < VE; ++e) sw[i][e] = 0.f;
    if (!base || W == 1) return;
    float raw[WS * VE];
    const uint4* p = reinterpret_cast<const uint4*>(st_ptr(base, sq));
#pragma unroll
    for (int i = 0; i < WS; ++i) cv_unpack<T, VE>(p[i], raw + i * VE);
#pragma unroll
    for (int e = 0; e < VE; ++e)
#pragma unroll
      for (int i = 0; i < WS; ++i) sw[i][e] = raw[e * (W - 1) + i];
  };
  // sw[si][e] for a runtime si (0 .. W-2, else 0) by unrolled selects, so the
  // state stays in registers
  auto sw_at = [&](int si, int e) {
    float r = 0.f;
#pragma unroll
    for (int j = 0; j < WS; ++j) r = (si == j) ? sw[j][e] : r;
    return r;
  };
  float win[WS][VE];  // raw inputs of rows t-(W-1) .. t-1
  auto store_state = [&](uint8_t* base, int64_t sq, int t_last, int s0) {
    // the last W-1 inputs of (state ++ sequence rows up to t_last), oldest first
    if (W == 1) return;
    float raw[WS * VE];
#pragma unroll
    for (int i = 0; i < WS; ++i) {
      const int src = t_last - (W - 2) + i;  // entry i of the new state
      const int si = (W - 1) - (s0 - src);   // its place in the old state, if before s0
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        // rows t_last-(W-2) .. t_last: win holds t_last-(W-2) .. t_last after the shift
        raw[e * (W - 1) + i] = src >= s0 ? win[i][e] : sw_at(si, e);
      }
    }
    uint4* p = reinterpret_cast<uint4*>(const_cast<uint8_t*>(st_ptr(base, sq)));
#pragma unroll
    for (int i = 0; i < WS; ++i) p[i] = cv_pack<T, VE>(raw + i * VE);
  };
  // the sequence of row t0 (varlen) and its bounds; offsets are clamped to
  // [0, T] so that no list, however malformed, moves a read outside the rows
  int seq = in, s_start = 0, s_end = a.T;
  auto bounds = [&](int sq) {
    s_start = sq < ca.N_seq ? min(max(ca.cu[sq], 0), a.T) : a.T;
    s_end = sq < ca.N_seq ? min(max(ca.cu[sq + 1], s_start), a.T) : a.T;
  };
  if (!DECODE && ca.cu) {
    int lo = 0, hi = ca.N_seq;  // largest s < N_seq with cu[s] <= t0
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ca.cu[mid] <= t0) lo = mid; else hi = mid;
    }
    seq = lo;
    bounds(seq);
    while (seq < ca.N_seq && s_end <= t0) bounds(++seq);  // skip sequences ending before t0
    if (t0 == 0 && ca.st_out && W > 1) {  // empty sequences keep their initial state
      for (int sq = 0; sq < ca.N_seq; ++sq) {
        const int b0 = min(max(ca.cu[sq], 0), a.T), b1 = min(max(ca.cu[sq + 1], b0), a.T);
        if (b1 > b0) continue;
        const uint4* src = ca.st_in ? reinterpret_cast<const uint4*>(st_ptr(ca.st_in, sq)) : nullptr;
        uint4* d = reinterpret_cast<uint4*>(const_cast<uint8_t*>(st_ptr(ca.st_out, sq)));
        for (int i = 0; i < W - 1; ++i) d[i] = src ? src[i] : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  load_state(ca.st_in, DECODE ? (int64_t)sl : (int64_t)seq);
#pragma unroll(DECODE ? 1 : (W > 1 ? W - 1 : 1))
  for (int rr = 0; rr < nrows; ++rr) {
    asm volatile("cp.async.wait_group %0;" ::"n"(kConvD - 1) : "memory");
    float x[VE];
    cv_unpack<T, VE>(ring[rr % kConvD][threadIdx.x], x);
    issue(rr + kConvD);  // the slot is free again: the row kConvD ahead goes in
    const int t = t0 - (W - 1) + rr;
    if (rr >= W - 1) {
      if (!DECODE && ca.cu && t >= s_end) {
        while (t >= s_end && seq < ca.N_seq) bounds(++seq);  // crossed into the next sequence
        if (seq >= ca.N_seq) break;  // rows past the last sequence are not outputs
        load_state(ca.st_in, seq);
      }
      float y[VE];
      if (t - s_start < W - 1) {  // some window entries precede the sequence: take the state's
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          float z = bv[e];
#pragma unroll
          for (int i = 0; i < W - 1; ++i) {
            const int src = t - (W - 1) + i, si = (W - 1) - (s_start - src);
            z = z + wv[i][e] * (src < s_start ? sw_at(si, e) : win[i][e]);
          }
          z = z + wv[W - 1][e] * x[e];
          y[e] = z / (1.0f + expf(-z));
        }
      } else {  // the whole window is inside the sequence
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          float z = bv[e];
#pragma unroll
          for (int i = 0; i < W - 1; ++i) z = z + wv[i][e] * win[i][e];
          z = z + wv[W - 1][e] * x[e];
          y[e] = z / (1.0f + expf(-z));
        }
      }
      cv_scatter(a, dst, (int64_t)in * a.T + t, cv_pack<T, VE>(y));
    }
#pragma unroll
    for (int i = 0; i + 1 < W - 1; ++i)
#pragma unroll
      for (int e = 0; e < VE; ++e) win[i][e] = win[i + 1][e];
    if (W > 1) {
#pragma unroll
      for (int e = 0; e < VE; ++e) win[WS - 1][e] = x[e];
    }
    if (rr >= W - 1 && ca.st_out && W > 1 && (DECODE ? t == t1 - 1 : t == s_end - 1))
      store_state(ca.st_out, DECODE ? (int64_t)sl : (int64_t)(ca.cu ? seq : in), t, s_start);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

template <typename T, int W>
cudaError_t launch_conv_w(const ConvArgs& ca, bool decode, cudaStream_t s) {
  const int nvec = ca.C / (16 / (int)sizeof(T));
  const int64_t gx = decode ? ca.pa.n : (int64_t)ca.pa.n * ((ca.pa.T + ca.RT - 1) / ca.RT);
  const dim3 grid((unsigned)gx, (unsigned)((nvec + 255) / 256));
  auto kern = decode ? conv_prepare_kernel<T, W, true> : conv_prepare_kernel<T, W, false>;
  kern<<<grid, 256, 0, s>>>(ca);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_conv_t(const ConvArgs& ca, bool decode, cudaStream_t s) {
  switch (ca.W) {
    case 1: return launch_conv_w<T, 1>(ca, decode, s);
    case 2: return launch_conv_w<T, 2>(ca, decode, s);
    case 3: return launch_conv_w<T, 3>(ca, decode, s);
    default: return launch_conv_w<T, 4>(ca, decode, s);
  }
}

template <int VB>
cudaError_t launch_vb(PrepArgs a, bool decode, cudaStream_t s) {
  a.fd_hv = FastDiv((uint32_t)((int64_t)a.N * a.es / VB));
  const int64_t rows = (int64_t)a.n * a.T;
  const int64_t cap = (int64_t)sm_count() * 8;  // 8 resident 256-thread CTAs per SM
  const int grid = (int)(rows < cap ? rows : cap);
  return launch_pdl(decode ? prepare_kernel<VB, true> : prepare_kernel<VB, false>, dim3(grid),
                    dim3(256), 0, s, a);
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
  a.fd_H = FastDiv((uint32_t)H);
  a.fd_hpg = FastDiv((uint32_t)(H / G));
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool vec16 = al16(x) && al16(q) && al16(k) && al16(v) && (a.x_sn_b % 16 == 0) &&
                     (a.x_st_b % 16 == 0) && ((int64_t)P * a.es % 16 == 0) &&
                     ((int64_t)N * a.es % 16 == 0);
  if (vec16) {
    const int64_t ntot = ((int64_t)M * H * P + (int64_t)(decode ? 2 * M : M + 1) * H * N) *
                         a.es / 16;
    const int64_t xrow_b = (int64_t)(M * H * P + M * G * N + G * N) * a.es;
    const int64_t ring_b = kRing * xrow_b;
    // Prefill rows go through the ring with 256-thread CTAs (measured: 51 us on
    // the B2 T4096 H16 workload against 55 us for the register-prefetch row
    // kernel); decode rows that fit one pass of the row kernel stay there, longer
    // decode rows take the ring with 512-thread CTAs (14.3 against 16.3 us).
    const int nt = decode ? 512 : 256;
    const bool ring = ring_b <= 200 * 1024 && M * H <= nt && (!decode || ntot > 256 * kPU);
    if (!ring && ntot <= 256 * kPU && M * H <= 256) {
      const int64_t rows = (int64_t)n * T;
      int per_sm = 0;
      cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, decode ? prepare_rows_kernel<true> : prepare_rows_kernel<false>, 256, 0);
      if (e != cudaSuccess) return e;
      const int64_t cap = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
      const int grid = (int)(rows < cap ? rows : cap);
      return launch_pdl(decode ? prepare_rows_kernel<true> : prepare_rows_kernel<false>,
                        dim3(grid), dim3(256), 0, stream, a);
    }
    if (ring) {
      a.fd_hv = FastDiv((uint32_t)((int64_t)N * a.es / 16));
      auto kern = decode ? prepare_ring_kernel<true, 512> : prepare_ring_kernel<false, 256>;
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)ring_b);
      if (e != cudaSuccess) return e;
      int per_sm = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nt, (size_t)ring_b);
      if (e != cudaSuccess) return e;
      const int64_t rows = (int64_t)n * T;
      const int64_t cap = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
      const int grid = (int)(rows < cap ? rows : cap);
      return launch_pdl(kern, dim3(grid), dim3(nt), (size_t)ring_b, stream, a,
                        (int)(xrow_b / 16));
    }
    return launch_vb<16>(a, decode, stream);
  }
  if (a.es == 4) return launch_vb<4>(a, decode, stream);
  return launch_vb<2>(a, decode, stream);
}

cudaError_t launch_conv_prepare(const void* xp, int64_t xp_sn, int64_t xp_st, const float* w,
                                const float* bias, int W, const void* st_in, void* st_out,
                                const int32_t* cu, int N_seq, const int32_t* slot, int n_slots,
                                int32_t* status, const void* ba, int64_t ba_sn, int64_t ba_st,
                                const float* A_log, const float* dt_bias, int n, int T, int M,
                                int H, int G, int P, int N, gdp_dtype dt, bool decode, void* q,
                                void* k, void* v, float* beta, float* g, cudaStream_t stream) {
  if ((int64_t)n * T == 0) return cudaSuccess;
  ConvArgs ca;
  PrepArgs& a = ca.pa;
  a.es = dt == GDP_F32 ? 4 : 2;
  a.x = static_cast<const uint8_t*>(xp);
  a.x_sn_b = xp_sn * a.es;
  a.x_st_b = xp_st * a.es;
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
  ca.w = w;
  ca.bias = bias;
  ca.W = W;
  ca.C = M * H * P + M * G * N + G * N;
  ca.RT = kConvRT;
  ca.st_in = static_cast<const uint8_t*>(st_in);
  ca.st_out = static_cast<uint8_t*>(st_out);
  ca.cu = cu;
  ca.N_seq = N_seq;
  ca.slot = slot;
  ca.n_slots = n_slots;
  ca.status = status;
  switch (dt) {
    case GDP_BF16: return launch_conv_t<__nv_bfloat16>(ca, decode, stream);
    case GDP_F16: return launch_conv_t<__half>(ca, decode, stream);
    default: return launch_conv_t<float>(ca, decode, stream);
  }
}

}  // namespace gdp
