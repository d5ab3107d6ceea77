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
// element per call), so the kernels are HBM streams that touch each state
// element once (streaming cache hints on the global side).
//
// K = 128 (recurrent128_kernel): persistent CTAs, two per SM, walk work items
// (request, value head, 64-column slice). Inside an item every warp runs the
// steps on its own columns with no block barrier (the sums over K fold four
// per-thread row groups with warp shuffles); meanwhile the next item's state
// slice streams into shared memory with cp.async and the next batch of step
// inputs into registers, so the state traffic overlaps the arithmetic.
//
// Other K (recurrent_kernel): one CTA per (request, value head, 32-column
// slice) with K/32 warps; warp w holds state rows [32w, 32w + 32) of all 32
// columns (lane = column), so every warp reads and writes whole 128-byte rows.
// A step's inputs are staged in shared memory for up to 16 steps with one
// batched load, and the column sums over K combine per-thread partials across
// the K/32 warps through shared memory (two barriers per step).
//
// Both kernels normalise k and q once per staged step, read the key/query
// rows as 16-byte broadcast loads, and run the per-element arithmetic on
// packed pairs of rows (f32x2 multiply and fused multiply-add: half the
// instructions, the same per-element rounding).
#include <algorithm>

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

// State slots (decode serving): request r updates state row block slot[r] of a
// state pool of n_slots entries, or nothing when slot[r] is -1 (a padding
// request: its o rows are written as zeros). Without a slot table request r
// uses entry r. A slot outside [-1, n_slots) or shared by two requests would
// make the update ill-defined (two requests racing on one state), so such a
// request is skipped like padding and *status (if given) is set to 1. Every
// thread of the block calls this with the same r; each warp scans the table
// for repeats on its own (no block barrier) and all reach the same answer.
__device__ __forceinline__ int resolve_slot(const int* __restrict__ slot, int n, int n_slots,
                                            int r, int* status) {
  if (!slot) return r;
  const int s = slot[r];
  if (s == -1) return -1;
  int bad = s < -1 || s >= n_slots;
  if (!bad) {
    int dup = 0;
    for (int i = threadIdx.x & 31; i < n; i += 32) dup |= (i != r) & (slot[i] == s);
    bad = __any_sync(0xffffffffu, dup);
  }
  if (bad) {
    if (threadIdx.x == 0 && status) atomicExch(status, 1);
    return -1;
  }
  return s;
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
                 int l2norm, float* __restrict__ o, const int* __restrict__ slot, int n,
                 int n_slots, int* status) {
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
  const int sl = resolve_slot(slot, n, n_slots, r, status);
  const bool active = c < V;
  const bool live = sl >= 0;  // false: padding or rejected slot (no state, zero o rows)
  const int nth = KW * 32;
  float* st = state + ((int64_t)(live ? sl : 0) * HV + hv) * K * V + (int64_t)(warp * 32) * V + c;
  f2 h[16];  // rows (2i, 2i + 1) of this thread's 32, packed
#pragma unroll
  for (int i = 0; i < 16; ++i)
    h[i] = (active && live)
               ? pk2(__ldcs(st + (int64_t)(2 * i) * V), __ldcs(st + (int64_t)(2 * i + 1) * V))
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
        o[((re0 + e) * HV + hv) * V + c] = live ? scale * so : 0.f;
      }
      buf ^= 1;  // the next step writes the other buffers; reuse is two barriers away
    }
  }
  if (active && live) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 hv2 = upk2(h[i]);
      __stcs(st + (int64_t)(2 * i) * V, hv2.x);
      __stcs(st + (int64_t)(2 * i + 1) * V, hv2.y);
    }
  }
}

struct SlotArgs {
  const int* slot;  // null: request r uses state entry r
  int n, n_slots;
  int* status;
};

template <typename Tin, int KW>
cudaError_t launch_k(const dim3& grid, const void* q, const void* k, const void* v,
                     const float* beta, const float* g, float* state, int L, int H, int HV,
                     int V, float scale, int l2norm, float* o, const SlotArgs& sa,
                     cudaStream_t s) {
  constexpr int smem = rec_smem<KW * 32>();
  cudaError_t e = cudaFuncSetAttribute(recurrent_kernel<Tin, KW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  recurrent_kernel<Tin, KW><<<grid, KW * 32, smem, s>>>(
      static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v), beta,
      g, state, L, H, HV, V, scale, l2norm, o, sa.slot, sa.n, sa.n_slots, sa.status);
  return cudaGetLastError();
}

// K = 128: persistent CTAs with warp-independent steps and prefetch.
//
// A work item is (request, value head, 64-column slice). A 256-thread CTA
// holds one item at a time: warp w owns columns [8w, 8w + 8) of the slice and
// lane (grp = lane / 8, col = lane % 8) holds state rows [32 grp, 32 grp + 32)
// of its column, so the sums over K are per-thread partials folded by two
// warp shuffles: a step has no block barrier. Each global state read covers
// four full 32-byte sectors. While a CTA runs the steps of one item, the next
// item's state and the next batch of step inputs are already loading into
// registers, so the state stream overlaps the arithmetic instead of
// alternating with it. k and q rows sit in shared memory with the four row
// groups 36 floats apart, so a warp's four 16-byte broadcast reads hit
// distinct banks.
constexpr int kB = 8;                // steps staged per batch
constexpr int kSliceCols = 64;       // value columns per work item
constexpr int kGrpPad = 36;          // floats between row groups of a staged k / q row
constexpr int kRowPad = 4 * kGrpPad; // floats per staged k / q row

// One thread's share of a batch of step inputs, held as loaded: converting on
// arrival would make the warp wait for the loads before its steps, so the
// conversion happens when the batch is staged.
template <typename Tin>
struct Batch {
  Tin q[4], k[4], v[2];
  float b, g;
};

template <typename Tin>
__device__ __forceinline__ void load_batch(Batch<Tin>& p, const Tin* __restrict__ q,
                                           const Tin* __restrict__ k, const Tin* __restrict__ v,
                                           const float* __restrict__ beta,
                                           const float* __restrict__ g, int it, int e0, int L,
                                           int H, int HV, int V, int ncs) {
  const int rh = it / ncs, cs = it - rh * ncs;
  const int r = rh / HV, hv = rh - r * HV, kh = hv / (HV / H);
  const int lc = min(kB, L - e0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t re0 = (int64_t)r * L + e0;
  if (warp < lc) {  // warp w loads step row w of k and q, four elements per lane
    const int64_t base = ((re0 + warp) * H + kh) * 128 + 4 * lane;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      p.q[i] = q[base + i];
      p.k[i] = k[base + i];
    }
  }
  const int e = tid >> 5, cc = cs * kSliceCols + 2 * lane;  // v: row tid / 32, two columns
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    p.v[i] = Tin(0.f);
    if (e < lc && cc + i < V) p.v[i] = v[((re0 + e) * HV + hv) * V + cc + i];
  }
  if (tid < lc) {
    p.b = beta[(re0 + tid) * HV + hv];
    p.g = g[(re0 + tid) * HV + hv];
  }
}

// Asynchronous 16-byte global -> shared copy (zero-filled when src_bytes is 0).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   (unsigned)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Start the copy of one item's state slice, [128][64] fp32, into shared
// memory. Row R's 16-byte chunk c lands at chunk c ^ (2 (R / 32)): the four
// row groups a warp reads at once then fall on distinct banks. Columns past V
// are zero-filled.
// srh: the item's state-row block (slot * HV + hv); SLOTS: srh < 0 means the
// item has no state, every chunk is zero-filled and nothing is read.
template <bool SLOTS>
__device__ __forceinline__ void prefetch_state(float* sst, const float* state, int it, int ncs,
                                               int V, int64_t srh) {
  const int cs = it % ncs;
  const int tid = threadIdx.x, c16 = tid & 15;
  const bool has = !SLOTS || srh >= 0;
  const int valid = (has && cs * kSliceCols + 4 * c16 < V) ? 16 : 0;
  const float* src = state + (has ? srh : 0) * 128 * V + cs * kSliceCols + (valid ? 4 * c16 : 0);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = (tid >> 4) + 16 * i;
    cp_async16(sst + row * kSliceCols + 4 * (c16 ^ (2 * (row >> 5))), src + (int64_t)row * V,
               valid);
  }
  cp_async_commit();
}

__device__ __forceinline__ float* state_ptr(float* state, int it, int ncs, int V, int64_t srh) {
  const int cs = it % ncs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  return state + srh * 128 * V + (int64_t)(32 * (lane >> 3)) * V + cs * kSliceCols +
         8 * warp + (lane & 7);
}

// State-row block (slot * HV + hv) of item `it`, or -1 when the item's request
// has no state (padding or a rejected slot). Without slots it is request * HV + hv.
template <bool SLOTS>
__device__ __forceinline__ int64_t item_srh(int it, int ncs, int HV, const int* slot, int n,
                                            int n_slots, int* status) {
  const int rh = it / ncs;
  if (!SLOTS) return rh;
  const int r = rh / HV, hv = rh - r * HV;
  const int sl = resolve_slot(slot, n, n_slots, r, status);
  return sl < 0 ? -1 : (int64_t)sl * HV + hv;
}

template <typename Tin, bool SLOTS>
__global__ void __launch_bounds__(256, 2)
recurrent128_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                    const Tin* __restrict__ v, const float* __restrict__ beta,
                    const float* __restrict__ g, float* __restrict__ state, int n_items, int L,
                    int H, int HV, int V, int ncs, float scale, int l2norm,
                    float* __restrict__ o, const int* __restrict__ slot, int n, int n_slots,
                    int* status) {
  __shared__ __align__(16) float kn[kB * kRowPad];
  __shared__ __align__(16) float qn[kB * kRowPad];
  __shared__ __align__(16) float vs[kB * kSliceCols];
  __shared__ float bt[kB], eg[kB];
  extern __shared__ __align__(16) float sst[];  // [128][64] next item's state, swizzled
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = lane >> 3, cw = 8 * warp + (lane & 7);  // row group, column in the slice
  // where this thread's column sits in each of its rows of the swizzled buffer
  const int scol = 4 * ((2 * warp + ((lane >> 2) & 1)) ^ (2 * grp)) + (lane & 3);
  int it = blockIdx.x;
  if (it >= n_items) return;
  Batch<Tin> pf;
  int64_t srh = item_srh<SLOTS>(it, ncs, HV, slot, n, n_slots, status);
  prefetch_state<SLOTS>(sst, state, it, ncs, V, srh);
  load_batch(pf, q, k, v, beta, g, it, 0, L, H, HV, V, ncs);
  for (; it < n_items; it += gridDim.x) {
    const int rh = it / ncs, cs = it - rh * ncs;
    const int r = rh / HV, hv = rh - r * HV;
    const int col = cs * kSliceCols + cw;
    const bool active = col < V;
    const bool live = !SLOTS || srh >= 0;  // false: padding or rejected slot (zero o rows)
    const int nx = it + gridDim.x;
    int64_t srh_nx = SLOTS ? -1 : (int64_t)(nx / ncs);
    cp_async_wait_all();
    __syncthreads();  // this item's state is in shared memory
    f2 h[16];  // rows (2i, 2i + 1) of this thread's 32, packed
#pragma unroll
    for (int i = 0; i < 16; ++i)
      h[i] = pk2(sst[(32 * grp + 2 * i) * kSliceCols + scol],
                 sst[(32 * grp + 2 * i + 1) * kSliceCols + scol]);
    for (int e0 = 0; e0 < L; e0 += kB) {
      const int lc = min(kB, L - e0);
      const int64_t re0 = (int64_t)r * L + e0;
      __syncthreads();  // every warp has finished the previous batch
      if (warp < lc) {  // normalise k and q rows in registers, one row per warp
        float kf[4], qf[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          kf[i] = ldf(&pf.k[i]);
          qf[i] = ldf(&pf.q[i]);
        }
        float rk = 1.f, rq = 1.f;
        if (l2norm) {
          float sk = 0.f, sq = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            sk += kf[i] * kf[i];
            sq += qf[i] * qf[i];
          }
          rk = 1.0f / sqrtf(warp_sum(sk) + 1e-6f);
          rq = 1.0f / sqrtf(warp_sum(sq) + 1e-6f);
        }
        const int off = warp * kRowPad + (lane >> 3) * kGrpPad + 4 * (lane & 7);
        *reinterpret_cast<float4*>(kn + off) =
            make_float4(kf[0] * rk, kf[1] * rk, kf[2] * rk, kf[3] * rk);
        *reinterpret_cast<float4*>(qn + off) =
            make_float4(qf[0] * rq, qf[1] * rq, qf[2] * rq, qf[3] * rq);
      }
      *reinterpret_cast<float2*>(vs + (tid >> 5) * kSliceCols + 2 * lane) =
          make_float2(ldf(&pf.v[0]), ldf(&pf.v[1]));
      if (tid < lc) {
        bt[tid] = pf.b;
        eg[tid] = expf(pf.g);
      }
      __syncthreads();
      // the state buffer has been read (barrier above): the next item's state
      // streams in behind this item's steps
      if (e0 == 0 && nx < n_items) {
        srh_nx = item_srh<SLOTS>(nx, ncs, HV, slot, n, n_slots, status);
        prefetch_state<SLOTS>(sst, state, nx, ncs, V, srh_nx);
      }
      if (e0 + kB < L)
        load_batch(pf, q, k, v, beta, g, it, e0 + kB, L, H, HV, V, ncs);
      else if (nx < n_items)
        load_batch(pf, q, k, v, beta, g, nx, 0, L, H, HV, V, ncs);
      // one step: decay, k^T h, the rank-1 update and o = scale h^T q
      float* ob = o + (re0 * HV + hv) * V + col;  // this thread's o entry of step e0
      const float* kg = kn + grp * kGrpPad;
      const float* qg = qn + grp * kGrpPad;
      auto step = [&](int e) {
        const ulonglong2* kr = reinterpret_cast<const ulonglong2*>(kg + e * kRowPad);
        const ulonglong2* qr = reinterpret_cast<const ulonglong2*>(qg + e * kRowPad);
        const f2 d2 = pk2(eg[e], eg[e]);
        f2 pa = pk2(0.f, 0.f), pb = pa;
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const ulonglong2 kk = kr[i4];
          h[2 * i4] = mul2(h[2 * i4], d2);
          h[2 * i4 + 1] = mul2(h[2 * i4 + 1], d2);
          pa = fma2(h[2 * i4], kk.x, pa);
          pb = fma2(h[2 * i4 + 1], kk.y, pb);
        }
        const float2 pav = upk2(pa), pbv = upk2(pb);
        float p = (pav.x + pav.y) + (pbv.x + pbv.y);
        p += __shfl_xor_sync(0xffffffffu, p, 8);
        p += __shfl_xor_sync(0xffffffffu, p, 16);
        const float delta = bt[e] * (vs[e * kSliceCols + cw] - p);
        const f2 dl2 = pk2(delta, delta);
        f2 oa = pk2(0.f, 0.f), obb = oa;
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const ulonglong2 kk = kr[i4], qq = qr[i4];
          h[2 * i4] = fma2(kk.x, dl2, h[2 * i4]);
          h[2 * i4 + 1] = fma2(kk.y, dl2, h[2 * i4 + 1]);
          oa = fma2(h[2 * i4], qq.x, oa);
          obb = fma2(h[2 * i4 + 1], qq.y, obb);
        }
        const float2 oav = upk2(oa), obv = upk2(obb);
        float po = (oav.x + oav.y) + (obv.x + obv.y);
        po += __shfl_xor_sync(0xffffffffu, po, 8);
        po += __shfl_xor_sync(0xffffffffu, po, 16);
        if (grp == 0 && active) ob[(int64_t)e * HV * V] = live ? scale * po : 0.f;
      };
      if (lc == kB) {  // a full batch: straight-line steps
#pragma unroll
        for (int e = 0; e < kB; ++e) step(e);
      } else {
        for (int e = 0; e < lc; ++e) step(e);
      }
    }
    if (active && live) {
      float* sp = state_ptr(state, it, ncs, V, srh);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 hv2 = upk2(h[i]);
        __stcs(sp + (int64_t)(2 * i) * V, hv2.x);
        __stcs(sp + (int64_t)(2 * i + 1) * V, hv2.y);
      }
    }
    srh = srh_nx;
  }
}

template <typename Tin>
cudaError_t launch_k128(const void* q, const void* k, const void* v, const float* beta,
                        const float* g, float* state, int n, int L, int H, int HV, int V,
                        float scale, int l2norm, float* o, const SlotArgs& sa, cudaStream_t s) {
  const int ncs = (int)cdiv(V, kSliceCols);
  const int64_t items = (int64_t)n * HV * ncs;
  if (items > INT32_MAX) return cudaErrorInvalidValue;
  const int grid = (int)std::min<int64_t>(items, (int64_t)sm_count() * 2);  // 2 resident CTAs / SM
  constexpr int smem = 128 * kSliceCols * 4;
  auto kern = sa.slot ? recurrent128_kernel<Tin, true> : recurrent128_kernel<Tin, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, 256, smem, s>>>(
      static_cast<const Tin*>(q), static_cast<const Tin*>(k), static_cast<const Tin*>(v), beta,
      g, state, (int)items, L, H, HV, V, ncs, scale, l2norm, o, sa.slot, sa.n, sa.n_slots,
      sa.status);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t run(const void* q, const void* k, const void* v, const float* beta, const float* g,
                float* state, int n, int L, int H, int HV, int K, int V, float scale, int l2norm,
                float* o, const SlotArgs& sa, cudaStream_t s) {
  const dim3 grid((unsigned)((int64_t)n * HV), (unsigned)cdiv(V, kCtaCols));
  switch (K) {
    case 32: return launch_k<Tin, 1>(grid, q, k, v, beta, g, state, L, H, HV, V, scale, l2norm, o, sa, s);
    case 64: return launch_k<Tin, 2>(grid, q, k, v, beta, g, state, L, H, HV, V, scale, l2norm, o, sa, s);
    case 128:  // the entry point guarantees V % 8 == 0 and a 16-byte aligned state
      return launch_k128<Tin>(q, k, v, beta, g, state, n, L, H, HV, V, scale, l2norm, o, sa, s);
    default: return launch_k<Tin, 8>(grid, q, k, v, beta, g, state, L, H, HV, V, scale, l2norm, o, sa, s);
  }
}

}  // namespace

cudaError_t launch_recurrent(const void* q, const void* k, const void* v, const float* beta,
                             const float* g, float* state, int n, int L, int H, int HV, int K,
                             int V, float scale, int l2norm, gdp_dtype dt, float* o,
                             const int32_t* slot, int n_slots, int32_t* status,
                             cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const SlotArgs sa{slot, n, n_slots, status};
  switch (dt) {
    case GDP_BF16:
      return run<__nv_bfloat16>(q, k, v, beta, g, state, n, L, H, HV, K, V, scale, l2norm, o, sa, stream);
    case GDP_F16:
      return run<__half>(q, k, v, beta, g, state, n, L, H, HV, K, V, scale, l2norm, o, sa, stream);
    default:
      return run<float>(q, k, v, beta, g, state, n, L, H, HV, K, V, scale, l2norm, o, sa, stream);
  }
}

}  // namespace gdp
