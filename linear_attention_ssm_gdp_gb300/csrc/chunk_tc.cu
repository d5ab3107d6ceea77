// Tensor-core chunked Gated Delta Product forward for GB300 (sm_103a):
// bf16 inputs, K = 128, chunk 64, V in {64, 128, 256}, M <= 3.
//
// Same stages and algebra as the generic path (Megatron-core API pages
// "core.ssm.ops.gdp.wy_fast" and "core.ssm.ops.gdp.chunk_o"; the WY form of
// the gated delta rule over the Householder-expanded stream), with every
// dense contraction on the 5th-generation tensor core: operands staged in
// shared memory by TMA (128-byte swizzle), tcgen05.mma issued from one or a
// few threads, fp32 accumulators in TMEM read back with tcgen05.ld.
//
// Precision. Raw q, k, v are bf16 and enter the MMAs exactly; the L2 norms,
// gates and decays are applied as fp32 row/column scales outside the MMAs.
// Every operand computed on chip (A, h, v_new, the score matrix P) is split
// into bf16 hi + lo (x = hi + lo to ~2^-16 relative) and a product of two
// such operands takes three MMAs (hi*hi + hi*lo + lo*hi), a product with an
// exact operand two. One bf16 rounding of any of them would by itself cost
// about 2^-9 of the output RMS per element.
//
// Kernels (one launch each):
//   wy128  persistent, one CTA per SM over (128-position block, HV) items: Gram
//       matrix k k^T (MMA), transition block L and its inverse A = (I+L)^-1
//       (blocked: forward substitution and 32 merges in fp32 on CUDA cores, the
//       top merge on the tensor cores), then w = (A diag(beta e^Gam/|k|)) k and
//       u = (A diag(beta)) v (MMAs) -> w as bf16 hi/lo, u fp32 (whole blocks
//       leave through TMA bulk stores while the next item's k and v load). For
//       odd M an item is two 64-position chunks with their own inverses and
//       decay prefixes (no top merge), the factors the 64-position state
//       recurrence steps with.
//   ho128 (M = 2) grid (sequence, HV, 32-column slice of V): the sequential
//       state recurrence and the chunk output in one kernel (a 128-position
//       block is one 64-token output chunk); a chain warp group and an output
//       warp group meeting at mbarriers; states and v_new never reach HBM.
//   h   (odd M) grid (sequence, HV, 32-column slice of V), ragged sequences
//       longest first: the sequential chunk-state recurrence on 64-position
//       steps, fp32 state in registers (thread = state row), per step
//       v_new = u - w h and h <- e^Gam_last h + k^T (e^(Gam_last - Gam)/|k| v_new);
//       writes v_new (hi/lo) and the state at every token-chunk start (hi/lo).
//   o   (odd M) persistent, one CTA per SM over (token chunk, HV, 64-column
//       slice) items: scores k q^T and q h (MMA), P^T = masked decayed scores
//       (fp32 -> hi/lo), P v_new, o = scale |q|^-1 (e^Gt q h + P v_new); two
//       TMEM column sets, so one item's products and norms overlap the previous
//       item's O product and stores.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "gdp_internal.cuh"
#include "ptx.cuh"

namespace gdp {
namespace {

using bf16 = __nv_bfloat16;
using namespace ptx;

constexpr int kBT = 64;    // chunk length (positions for wy/h, tokens for o)
constexpr int kK = 128;    // key/query head dimension
constexpr int kHBV = 32;   // value columns per chunk_h CTA
constexpr int kOBV = 64;   // value columns per chunk_o CTA

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ float gam_diff4(const float* hi, const float* lo, int p, int i) {
  return (hi[p] - hi[i]) + (lo[p] - lo[i]);
}

// Error-free sum (Knuth's TwoSum): a + b = s + e exactly.
__device__ __forceinline__ float two_sum(float a, float b, float& e) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return s;
}

// Compensated inclusive prefix sum of 128 values by one warp: lane l owns
// positions 4l .. 4l + 3 (hi[] holds the summands on entry). Each lane sums its
// four values with running TwoSum corrections, the lane totals are scanned
// across the warp as (sum, correction) pairs combined by TwoSum, and each
// lane re-adds its exclusive prefix. hi[p] + lo[p] carries the prefix to about
// twice fp32 precision, like the serial Neumaier form, in 4 + 5 + 4 steps
// instead of 128. SPLIT: two independent prefixes, positions 0..63 and
// 64..127 (lanes 0-15 and 16-31), for two 64-position chunks.
template <bool SPLIT>
__device__ __forceinline__ void comp_prefix128_warp(float* hi, float* lo, int lane) {
  float s[4], c[4];
  const float4 x = *reinterpret_cast<const float4*>(hi + 4 * lane);
  const float xs[4] = {x.x, x.y, x.z, x.w};
  s[0] = xs[0];
  c[0] = 0.f;
#pragma unroll
  for (int i = 1; i < 4; ++i) {
    float e;
    s[i] = two_sum(s[i - 1], xs[i], e);
    c[i] = __fadd_rn(c[i - 1], e);
  }
  float S = s[3], C = c[3];  // inclusive scan of the lane totals
  const int sl = SPLIT ? (lane & 15) : lane;  // lane within its scan
#pragma unroll
  for (int off = 1; off < (SPLIT ? 16 : 32); off <<= 1) {
    const float S2 = __shfl_up_sync(0xffffffffu, S, off);
    const float C2 = __shfl_up_sync(0xffffffffu, C, off);
    if (sl >= off) {
      float e;
      const float t = two_sum(S2, S, e);
      C = __fadd_rn(__fadd_rn(C2, C), e);
      S = t;
    }
  }
  float ES = __shfl_up_sync(0xffffffffu, S, 1), EC = __shfl_up_sync(0xffffffffu, C, 1);
  if (sl == 0) ES = EC = 0.f;
  float oh[4], ol[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float e;
    oh[i] = two_sum(ES, s[i], e);
    ol[i] = __fadd_rn(__fadd_rn(EC, c[i]), e);
  }
  *reinterpret_cast<float4*>(hi + 4 * lane) = make_float4(oh[0], oh[1], oh[2], oh[3]);
  *reinterpret_cast<float4*>(lo + 4 * lane) = make_float4(ol[0], ol[1], ol[2], ol[3]);
}

__device__ __forceinline__ void split_bf16(float x, bf16& hi, bf16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

// split_bf16 of n (even) values, two per conversion instruction (same rounding).
template <int n>
__device__ __forceinline__ void split_bf16_n(const float* x, bf16* hi, bf16* lo) {
#pragma unroll
  for (int i = 0; i < n; i += 2) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x[i], x[i + 1]);
    const float2 hf = __bfloat1622float2(h);
    *reinterpret_cast<__nv_bfloat162*>(hi + i) = h;
    *reinterpret_cast<__nv_bfloat162*>(lo + i) = __floats2bfloat162_rn(x[i] - hf.x, x[i + 1] - hf.y);
  }
}

// Sum of squares of row p (128 bytes of bf16) of a tile stored with the
// 128-byte swizzle. The chunks are visited in the order j ^ (p & 7), which is
// the physical order 0..7, so the lanes of a warp (consecutive rows) read
// distinct banks; four partial sums keep the additions independent.
// Packed pairs of fp32 (Blackwell f32x2 arithmetic, each lane rounded like the
// scalar operation).
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
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
  f2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// 2^x by the hardware approximation (relative error ~2^-22; subnormal results
// flush to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// A natural-log two-float value hi + lo in base-2 units as a two-float pair:
// p = fl(hi log2e) and its exact product error plus lo log2e. Differences of
// such pairs keep the cancellation of the hi parts exact, as for the natural
// values, so 2^(difference) carries the precision of e^(difference).
__device__ __forceinline__ float2 log2e_pair(float hi, float lo) {
  constexpr float kLog2e = 1.44269504088896341f;
  const float p = hi * kLog2e;
  return make_float2(p, fmaf(lo, kLog2e, fmaf(hi, kLog2e, -p)));
}

__device__ __forceinline__ float row_sumsq(const uint8_t* row, int p) {
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 u = reinterpret_cast<const uint4*>(row)[j ^ (p & 7)];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float a = __uint_as_float(w[t] << 16), b = __uint_as_float(w[t] & 0xffff0000u);
      s[t] = fmaf(a, a, fmaf(b, b, s[t]));
    }
  }
  return (s[0] + s[1]) + (s[2] + s[3]);
}

__device__ __forceinline__ void store_bf16x32(bf16* dst, const bf16* src) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    reinterpret_cast<uint4*>(dst)[j] = reinterpret_cast<const uint4*>(src)[j];
}

// Ends the CTA's tensor-core use: make every thread's TMEM traffic complete,
// then free the columns (warp 0).
__device__ __forceinline__ void tmem_release(uint32_t tmem, uint32_t ncols) {
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tmem_dealloc(tmem, ncols);
}

// ============================================================================ wy
struct WyArgs {
  int H, HV, V, M, l2norm;
  int64_t Te;
  const float* beta;
  const float* g;
  const int4* seq_info;
  const int4* blk_tab;  // 128-position blocks: sequence, first 64-chunk, the
                        // sequence's first token, its length; sequence -1 past the end
  bf16* w_hi;
  bf16* w_lo;
  float* u;
  float4* gk;  // [HV][Te]: (Gam hi, Gam lo, 1/|k|, 0)
  int* status;
  int fault;   // test hook (gdp_debug_wait_fault): CTA 0 skips its first Gram product
};

// ============================================================================ chunk_h
struct HArgs {
  int HV, V, M;
  int64_t Te;
  const int4* seq_info;
  const float* u;
  const float4* gk;
  const float* h0;
  float* hT;
  bf16* vn_hi;
  bf16* vn_lo;
  bf16* h_hi;   // [n_tok_chunks][HV][K][V]
  bf16* h_lo;
  int* status;
};

// The (sequence, value head, value slice) of a state-scan CTA. The value slices
// of one (sequence, head), which read the same w, k and q tiles, are always
// neighbours in launch order. Without an order table the grid is
// (sequence x slice, head); with one (ragged sequences) the launch order walks
// the sequences longest first, every head of one sequence before the next, so
// that the chains that start last are the shortest and the grid ends evenly.
struct ChainPos {
  int seq, hv, slice;
};
__device__ __forceinline__ ChainPos chain_pos(const int* order, int nsl, int HV) {
  if (!order) return {(int)blockIdx.x / nsl, (int)blockIdx.y, (int)(blockIdx.x % nsl)};
  const int lin = (int)(blockIdx.y * gridDim.x + blockIdx.x), per = HV * nsl;
  const int r = lin / per, rem = lin - r * per;
  return {order[r], rem / nsl, rem % nsl};
}

// Shared memory: w_hi (16 KB) | w_lo (16 KB) | k (16 KB) | u fp32 64x32 (8 KB) | gk
// 64x16 B (1 KB) | h^T hi | lo (16 KB) | v'^T hi | lo (8 KB) | barriers: 82 KB, so two
// CTAs share an SM. Each operand has one buffer and its own barrier; the next
// chunk's tile is requested as soon as this chunk's last reader of that buffer
// is done (w after product 1, u and the records after the value phase, k after
// product 2), so each load streams in behind the rest of the step.
constexpr int H_W = 0;
constexpr int H_K = 32768;
constexpr int H_U = 49152;
constexpr int H_G = 57344;
constexpr int H_HT = 58368;                               // 1024-aligned
constexpr int H_VP = H_HT + 16384;
constexpr int H_BAR = H_VP + 8192;
constexpr int H_SMEM = H_BAR + 64 + 1024;

// 256 threads: thread (warp w, lane l) owns state row kf = 32 (w % 4) + l (the
// TMEM lane quarter its warp may access) and the 16 value columns
// [16 (w / 4), 16 (w / 4) + 16) of the CTA's 32; in the value phase the warps
// of lane quarters 0 and 1 own position p = 32 (w % 4) + l and the same 16
// columns. Splitting the columns over two warps per lane quarter halves the
// per-thread work on the sequential critical path.
constexpr int kHCols = kHBV / 2;

__global__ void __launch_bounds__(256, 2) h_tc_kernel(
    const __grid_constant__ CUtensorMap map_whi, const __grid_constant__ CUtensorMap map_wlo,
    const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_u,
    const __grid_constant__ CUtensorMap map_gk, HArgs a, int H, const int* seq_order) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, chalf = warp >> 2;
  const int row = quarter * 32 + lane;          // state row kf / position p
  const int cb = chalf * kHCols;                // first of this thread's 16 columns
  const int nsl = a.V / kHBV;
  const ChainPos cp = chain_pos(seq_order, nsl, a.HV);
  const int seq = cp.seq, hv = cp.hv, kh = hv / (a.HV / H);
  const int v0 = cp.slice * kHBV;
  const int V = a.V, M = a.M;
  const int4 si = a.seq_info[seq];
  const int ne = (int)cdiv((int64_t)si.y * M, kBT);
  uint8_t* ht = sm + H_HT;
  uint8_t* vp = sm + H_VP;
  // [0] w full, [1] k full, [2] u and records full, [3] product 1, [4] product 2
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + H_BAR);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 5);
  const int64_t hoff = ((int64_t)seq * a.HV + hv) * kK * V;
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;

  // TMEM columns: D1 = w_hi [h_hi | h_lo] [0, 64), D1B = w_lo h_hi [64, 96),
  // D2 = k^T [v'_hi | v'_lo] [128, 192); a product is the sum of its halves
  constexpr uint32_t TD1 = 0, TD1B = 64, TD2 = 128;
  if (warp == 0) {
    tmem_alloc(s_tmem, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bars[i], i == 3 ? 2 : 1);  // product 1: two issuers
    fence_mbar_init();
  }
  // The B operands h (rows kf) and v' (rows p) are MN-major tiles with 64-byte
  // rows (32 value columns, 64-byte swizzle): a thread stores its 16 columns
  // of its own row as two 16-byte chunks.
  const uint32_t off_r0 = sw64_chunk(row, 2 * chalf), off_r1 = sw64_chunk(row, 2 * chalf + 1);
  float h[kHCols];
  {
    const float* src = a.h0 ? a.h0 + hoff + (int64_t)row * V + v0 + cb : nullptr;
#pragma unroll
    for (int c = 0; c < kHCols; ++c) h[c] = src ? src[c] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int64_t Rseq = (int64_t)si.x * M;
  const int64_t gk0 = (int64_t)hv * a.Te + Rseq;
  auto load_w = [&](int64_t R) {
    mbar_expect_tx(&bars[0], 32768);
    tma_load_3d(sm + H_W, &map_whi, 0, hv, (int)R, &bars[0]);
    tma_load_3d(sm + H_W + 8192, &map_whi, 64, hv, (int)R, &bars[0]);
    tma_load_3d(sm + H_W + 16384, &map_wlo, 0, hv, (int)R, &bars[0]);
    tma_load_3d(sm + H_W + 24576, &map_wlo, 64, hv, (int)R, &bars[0]);
  };
  auto load_k = [&](int64_t R) {
    mbar_expect_tx(&bars[1], 16384);
    tma_load_3d(sm + H_K, &map_k, 0, kh, (int)R, &bars[1]);
    tma_load_3d(sm + H_K + 8192, &map_k, 64, kh, (int)R, &bars[1]);
  };
  auto load_ug = [&](int64_t R, int64_t G) {
    mbar_expect_tx(&bars[2], 8192 + 1024);
    tma_load_3d(sm + H_U, &map_u, v0, hv, (int)R, &bars[2]);
    tma_load_2d(sm + H_G, &map_gk, 0, (int)G, &bars[2]);
  };
  if (tid == 0 && ne > 0) {
    load_w(Rseq);
    load_k(Rseq);
    load_ug(Rseq, gk0);
  }
  const uint32_t id1 = idesc_bf16(128, kHBV, false, true);
  const uint32_t id1w = idesc_bf16(128, 2 * kHBV, false, true);
  const uint32_t id2w = idesc_bf16(128, 2 * kHBV, true, true);
  const float4* gk = reinterpret_cast<const float4*>(sm + H_G);
  for (int j = 0; j <= ne; ++j) {
    // publish the state at the start of chunk j (operand h^T, and for chunk_o at token-chunk starts)
    {
      __align__(16) bf16 hi[kHCols];
      __align__(16) bf16 lo[kHCols];
#pragma unroll
      for (int c = 0; c < kHCols; ++c) split_bf16(h[c], hi[c], lo[c]);
      const uint4* h4 = reinterpret_cast<const uint4*>(hi);
      const uint4* l4 = reinterpret_cast<const uint4*>(lo);
      *reinterpret_cast<uint4*>(ht + off_r0) = h4[0];
      *reinterpret_cast<uint4*>(ht + off_r1) = h4[1];
      *reinterpret_cast<uint4*>(ht + 8192 + off_r0) = l4[0];
      *reinterpret_cast<uint4*>(ht + 8192 + off_r1) = l4[1];
      if (j < ne && j % M == 0) {  // state at a token-chunk start, [chunk][HV][K][V]
        const int64_t base = ((((int64_t)si.w + j / M) * a.HV + hv) * kK + row) * V + v0 + cb;
        uint4* dh = reinterpret_cast<uint4*>(a.h_hi + base);
        uint4* dl = reinterpret_cast<uint4*>(a.h_lo + base);
        dh[0] = h4[0];
        dh[1] = h4[1];
        dl[0] = l4[0];
        dl[1] = l4[1];
      }
    }
    if (j == ne) break;
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t ph = j & 1;
    const int n = min(kBT, si.y * M - j * kBT);
    const int64_t R = Rseq + (int64_t)j * kBT;
    bool ok = true;
    if (tid == 0 || tid == 32) {  // product 1: D1 = w h (rows = positions), two issuers
      ok = mbar_wait(&bars[0], ph, a.status, kDevTimeout);
      if (ok) {
        const uint32_t whi = smem_u32(sm + H_W), wlo = smem_u32(sm + H_W + 16384), hb = smem_u32(ht);
        if (tid == 0)  // w_hi [h_hi | h_lo]: the lo tile is the next 32-column group (LBO)
          mma_run<8, false, 8192, 32, 4096, 1024>(tmem + TD1, sdesc_sw128(whi, 16, 1024),
                                                  sdesc_sw64(hb, 8192, 512), id1w);
        else  // w_lo h_hi
          mma_run<8, false, 8192, 32, 4096, 1024>(tmem + TD1B, sdesc_sw128(wlo, 16, 1024),
                                                  sdesc_sw64(hb, 8192, 512), id1);
        mma_commit(&bars[3]);
      }
    }
    // every thread reads the chunk's last decay record (the state update needs it)
    ok = mbar_wait(&bars[2], ph, a.status, kDevTimeout) && ok;
    const float4 glast = gk[n - 1];
    if (quarter < 2) {  // positions p = row, columns cb .. cb + 15
      const int p = row;
      ok = mbar_wait(&bars[3], ph, a.status, kDevTimeout) && ok;
      tc_fence_after();
      // product 1 has read w: the next chunk's w streams in behind this step
      if (tid == 0 && ok && j + 1 < ne) load_w(R + kBT);
      uint32_t r[16], r1[16], r2[16];
      GDP_TMEM_LD16(tmem + lane_base + TD1 + cb, r);
      GDP_TMEM_LD16(tmem + lane_base + TD1 + 32 + cb, r1);
      GDP_TMEM_LD16(tmem + lane_base + TD1B + cb, r2);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < kHCols; ++c)
        r[c] = __float_as_uint((__uint_as_float(r[c]) + __uint_as_float(r2[c])) + __uint_as_float(r1[c]));
      const uint8_t* urow = sm + H_U + p * 128;  // u row p, 128B-swizzled 16-byte chunks
      float us[kHCols];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v4 = *reinterpret_cast<const float4*>(urow + ((((cb >> 2) + q) ^ (p & 7)) << 4));
        us[4 * q] = v4.x; us[4 * q + 1] = v4.y; us[4 * q + 2] = v4.z; us[4 * q + 3] = v4.w;
      }
      const float4 gp = gk[p];
      const float sc = (p < n) ? expf((glast.x - gp.x) + (glast.y - gp.y)) * gp.z : 0.f;
      __align__(16) bf16 vh[kHCols];
      __align__(16) bf16 vl[kHCols];
      __align__(16) bf16 pvh[kHCols];
      __align__(16) bf16 pvl[kHCols];
#pragma unroll
      for (int c = 0; c < kHCols; ++c) {
        const float vn = us[c] - __uint_as_float(r[c]);
        split_bf16(vn, vh[c], vl[c]);
        split_bf16(p < n ? vn * sc : 0.f, pvh[c], pvl[c]);
      }
      if (p < n) {
        const int64_t rowg = (R + p) * a.HV * V + (int64_t)hv * V + v0 + cb;
        uint4* dh = reinterpret_cast<uint4*>(a.vn_hi + rowg);
        uint4* dl = reinterpret_cast<uint4*>(a.vn_lo + rowg);
        dh[0] = reinterpret_cast<const uint4*>(vh)[0];
        dh[1] = reinterpret_cast<const uint4*>(vh)[1];
        dl[0] = reinterpret_cast<const uint4*>(vl)[0];
        dl[1] = reinterpret_cast<const uint4*>(vl)[1];
      }
      *reinterpret_cast<uint4*>(vp + off_r0) = reinterpret_cast<const uint4*>(pvh)[0];
      *reinterpret_cast<uint4*>(vp + off_r1) = reinterpret_cast<const uint4*>(pvh)[1];
      *reinterpret_cast<uint4*>(vp + 4096 + off_r0) = reinterpret_cast<const uint4*>(pvl)[0];
      *reinterpret_cast<uint4*>(vp + 4096 + off_r1) = reinterpret_cast<const uint4*>(pvl)[1];
      fence_async_smem();
      tc_fence_before();
    } else {
      fence_async_smem();  // the record reads end before the next records load
    }
    ok = __syncthreads_and(ok);
    if (!ok) break;
    tc_fence_after();
    if (tid == 0) {
      // u and the records have been read: the next chunk's stream in
      if (j + 1 < ne) load_ug(R + kBT, gk0 + (int64_t)(j + 1) * kBT);
      ok = mbar_wait(&bars[1], ph, a.status, kDevTimeout);
      if (ok) {  // product 2: D2 = k^T v'  (rows = state rows kf)
        const uint32_t kb = smem_u32(sm + H_K), vb = smem_u32(vp);
        const uint64_t kd = sdesc_sw128(kb, 8192, 1024);
        // k^T [v'_hi | v'_lo]: the lo tile is the next 32-column group (LBO)
        mma_run<4, false, 0, 2048, 0, 1024>(tmem + TD2, kd, sdesc_sw64(vb, 4096, 512), id2w);
        mma_commit(&bars[4]);
      }
    }
    ok = mbar_wait(&bars[4], ph, a.status, kDevTimeout) && ok;
    tc_fence_after();
    // product 2 has read k: the next chunk's k streams in
    if (tid == 0 && ok && j + 1 < ne) load_k(R + kBT);
    {
      uint32_t r[16], r1[16];
      GDP_TMEM_LD16(tmem + lane_base + TD2 + cb, r);
      GDP_TMEM_LD16(tmem + lane_base + TD2 + 32 + cb, r1);
      tmem_wait_ld();
      const float dl = expf(glast.x + glast.y);
#pragma unroll
      for (int c = 0; c < kHCols; ++c)
        h[c] = dl * h[c] + (__uint_as_float(r[c]) + __uint_as_float(r1[c]));
    }
    tc_fence_before();
    if (!__syncthreads_and(ok)) break;
  }
  if (a.hT) {
    float* dst = a.hT + hoff + (int64_t)row * V + v0 + cb;
#pragma unroll
    for (int c = 0; c < kHCols; c += 4)
      *reinterpret_cast<float4*>(dst + c) = make_float4(h[c], h[c + 1], h[c + 2], h[c + 3]);
  }
  tmem_release(tmem, 256);
}

// ============================================================================ wy, 128-position blocks
// For even M the WY factors are built for blocks of 128 expanded positions (two
// of the pages' 64-position chunks): the 128x128 inverse
// A = (I + L)^-1 = [[A0, 0], [-A1 (L10 A0), A1]] is formed in place in fp32,
// so the state recurrence can advance 128 positions per step. v_new does not
// depend on where the blocks fall, so the results are those of the 64-chunk
// algebra up to rounding.
//
// Shared memory: k (2 K-halves of 128 rows, 32 KB) | v (two 64-column chunks of
// 128 rows, 32 KB; V = 256 loads it in two rounds) | operand tiles (2 x 32 KB;
// the solve scratch lives here before the tiles are built) | L/A fp32 [128][129]
// | small arrays (two sets, by item parity) | barriers
constexpr int W8_K = 0;
constexpr int W8_V = 32768;
constexpr int W8_T = 65536;
constexpr int W8_LA = W8_T + 65536;
constexpr int W8_S = W8_LA + 128 * 129 * 4;
// aligned copy of L's four 32x32 diagonal blocks ([4][32][32], 16-byte chunks
// swizzled by row), read by the diagonal-block forward substitution
constexpr int W8_LD = 204800;
static_assert(W8_LD >= W8_S + 2 * 7 * 128 * 4 + 64, "diagonal-block copy overlaps");
constexpr int W8_SMEM = W8_LD + 4 * 32 * 32 * 4 + 1024;

// Top merge of the 128x128 inverse on the tensor cores: X = L10 A00, then
// A10 = -A11 X, each as x_hi [y_hi | y_lo] (one N = 128 MMA per k-step) plus
// x_lo y_hi (N = 64), fp32 accumulation; the two 64-column halves of an
// accumulator are summed when read. A operands are 128 rows of LA (the upper
// 64 rows only produce accumulator rows that are not read): rows of
// LA[:, 0:64] for the first product, of LA[:, 64:128] (A11 below zeros) for
// the second; K-major, 128-byte swizzle. B operands (A00, then X) are MN-major
// 128-byte-swizzle tiles with the lo tile one 64-column atom (8 KB) after the
// hi tile. Operand tiles live in `tiles` (48 KB used), accumulators in TMEM
// columns [0, 256). `bar` is an unused mbarrier whose phases 0 and 1 are taken.
// Relative error of the products ~2^-16 of sum |x||y|, the precision the
// inverse is later used at (its hi/lo operand tiles).
__device__ bool merge64_tc(float* LA, uint8_t* tiles, uint32_t tmem, uint64_t* bar, int* status) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, cq = warp >> 2;
  const int p = quarter * 32 + lane;  // row of LA / TMEM lane
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  uint8_t* a_hi = tiles;              // [128 rows][64 K] bf16, swizzled
  uint8_t* a_lo = tiles + 16384;
  uint8_t* b_hi = tiles + 32768;      // [64 K rows][64 N] bf16, swizzled (MN-major)
  uint8_t* b_lo = tiles + 40960;
  // 16 consecutive values of row r into a 128-byte swizzled row at column 16 cq
  auto put16 = [&](uint8_t* hi_base, uint8_t* lo_base, int r, const float* x) {
    __align__(16) bf16 h[16];
    __align__(16) bf16 l[16];
    split_bf16_n<16>(x, h, l);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t off = r * 128 + (((2 * cq + q) ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(hi_base + off) = reinterpret_cast<const uint4*>(h)[q];
      *reinterpret_cast<uint4*>(lo_base + off) = reinterpret_cast<const uint4*>(l)[q];
    }
  };
  auto issue = [&](uint32_t dcol) {  // D[dcol..] = A B over K = 64
    const uint32_t ah = smem_u32(a_hi), al = smem_u32(a_lo), bh = smem_u32(b_hi);
    const uint32_t idw = idesc_bf16(128, 128, false, true), idn = idesc_bf16(128, 64, false, true);
    const uint64_t bd = sdesc_sw128(bh, 8192, 1024);
    mma_run<4, false, 0, 32, 0, 2048>(tmem + dcol, sdesc_sw128(ah, 16, 1024), bd, idw);
    mma_run<4, true, 0, 32, 0, 2048>(tmem + dcol, sdesc_sw128(al, 16, 1024), bd, idn);
    mma_commit(bar);
  };
  float x[16];
  // operands of X = L10 A00
#pragma unroll
  for (int e = 0; e < 16; ++e) x[e] = LA[p * 129 + 16 * cq + e];
  put16(a_hi, a_lo, p, x);
  if (p < 64) put16(b_hi, b_lo, p, x);  // A00 rows (zero above the diagonal)
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) issue(0);
  bool ok = mbar_wait(bar, 0, status, kDevTimeout);
  tc_fence_after();
  // operands of A10 = -A11 X: A11 rows from LA, X from TMEM (lanes 64..127)
#pragma unroll
  for (int e = 0; e < 16; ++e) x[e] = LA[p * 129 + 64 + 16 * cq + e];
  if (quarter >= 2) {
    uint32_t r0[16], r1[16];
    GDP_TMEM_LD16(tmem + lane_base + 16 * cq, r0);
    GDP_TMEM_LD16(tmem + lane_base + 64 + 16 * cq, r1);
    tmem_wait_ld();
    float xs[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) xs[e] = __uint_as_float(r0[e]) + __uint_as_float(r1[e]);
    put16(b_hi, b_lo, p - 64, xs);
  }
  __syncthreads();  // every read of the first operands is done (MMA 1 waited)
  put16(a_hi, a_lo, p, x);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) issue(128);
  ok = mbar_wait(bar, 1, status, kDevTimeout) && ok;
  tc_fence_after();
  if (quarter >= 2) {
    uint32_t r0[16], r1[16];
    GDP_TMEM_LD16(tmem + lane_base + 128 + 16 * cq, r0);
    GDP_TMEM_LD16(tmem + lane_base + 192 + 16 * cq, r1);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e)
      LA[p * 129 + 16 * cq + e] = -(__uint_as_float(r0[e]) + __uint_as_float(r1[e]));
  }
  tc_fence_before();
  return __syncthreads_and(ok);
}

// In-place inverse of the unit lower-triangular 128x128 matrix I + L held
// strictly lower in LA (row stride 129, zeros on and above the diagonal):
//  * the four 32x32 diagonal blocks by forward substitution, warp b (0..3) on
//    block b, lane c on its column c, the column in registers; L's diagonal
//    blocks come from Ld (an aligned copy, [4][32][32] with row r's 16-byte
//    chunk q at chunk q ^ (r & 7), so a row is eight broadcast vector loads);
//    the inverse blocks go to LA and to an aligned copy Ad [4][32][36];
//  * the 32 merges A10 = -A11 (L10 A00) of the two 64 blocks on the CUDA cores,
//    their A00 / A11 / X operands read as vectors from Ad and the scratch Xs;
//  * the 64 merge on the tensor cores (merge64_tc).
// Both CUDA-core stages are bound by shared-memory load issue (one load a clock
// for the whole SM), which the vector loads cut. scratch: the 64 KB operand-tile
// region; TMEM columns [0, 256) and `bar` (phases 0, 1) are used. 512 threads.
// Returns false if a bounded wait gave up.
template <bool C64>
__device__ bool solve_tril128(float* LA, const float* Ld, float* scratch, uint32_t tmem,
                              uint64_t* bar, int* status) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* Ad = scratch;            // [4][32][36]
  float* Xs = scratch + 4 * 1152; // [2][32][36]
  if (warp < 4) {
    const float* Lb = Ld + warp * 1024;
    float col[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) col[i] = (i == lane) ? 1.f : 0.f;
#pragma unroll
    for (int r = 1; r < 32; ++r) {
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < (r + 3) / 4; ++q) {
        const float4 l = *reinterpret_cast<const float4*>(Lb + r * 32 + ((q ^ (r & 7)) << 2));
        const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (4 * q + e < r) s4[e] = fmaf(lv[e], col[4 * q + e], s4[e]);  // col[i] = 0 for i < lane
      }
      if (r > lane) col[r] = -((s4[0] + s4[1]) + (s4[2] + s4[3]));
    }
    float* la = LA + (warp * 32) * 129 + warp * 32 + lane;
    float* ad = Ad + warp * 1152 + lane;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      la[i * 129] = col[i];
      ad[i * 36] = col[i];
    }
  }
  __syncthreads();
  {  // 32 merges of the two 64 blocks, 4 outputs a thread
    const int pair = tid >> 8, rem = tid & 255;
    const int base = pair * 64;
    const float* A00 = Ad + (2 * pair) * 1152;
    const float* A11 = Ad + (2 * pair + 1) * 1152;
    float* X = Xs + pair * 1152;
    // warps of a pair take their column (row) blocks in the order 0 1 2 3 7 6 5 4, so
    // that warps sharing an SM sub-partition get a heavy and a light block
    const int wip = rem >> 5, li = rem & 31;
    const int mw = ((wip >> 2) & 1) ? (wip | 3) - (wip & 3) : wip;
    float acc[4];
    {  // X = L10 A00, A00 lower triangular: i >= c0
      const int r = li, c0 = mw * 4;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) acc[cc] = 0.f;
      const float* lrow = LA + (base + 32 + r) * 129 + base;
#pragma unroll 4
      for (int i = c0; i < 32; ++i) {
        const float av = lrow[i];
        const float4 b = *reinterpret_cast<const float4*>(A00 + i * 36 + c0);
        acc[0] = fmaf(av, b.x, acc[0]);
        acc[1] = fmaf(av, b.y, acc[1]);
        acc[2] = fmaf(av, b.z, acc[2]);
        acc[3] = fmaf(av, b.w, acc[3]);
      }
      *reinterpret_cast<float4*>(X + r * 36 + c0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    }
    __syncthreads();
    {  // A10 = -A11 X, A11 lower triangular: i <= r0
      const int r0 = mw * 4 + (li >> 3), c0 = (li & 7) * 4;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) acc[cc] = 0.f;
      const float* arow = A11 + r0 * 36;
#pragma unroll 4
      for (int i = 0; i <= r0; ++i) {
        const float av = arow[i];
        const float4 b = *reinterpret_cast<const float4*>(X + i * 36 + c0);
        acc[0] = fmaf(av, b.x, acc[0]);
        acc[1] = fmaf(av, b.y, acc[1]);
        acc[2] = fmaf(av, b.z, acc[2]);
        acc[3] = fmaf(av, b.w, acc[3]);
      }
      float* dst = LA + (base + 32 + r0) * 129 + base + c0;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) dst[cc] = -acc[cc];
    }
    __syncthreads();
  }
  // C64: two 64-position chunks, L10 = 0 and so A10 = 0: no top merge
  return C64 ? true : merge64_tc(LA, reinterpret_cast<uint8_t*>(scratch), tmem, bar, status);
}

// Persistent: one CTA per SM walks (128-position block, value head) items,
// item = head * NB + block, skipping the block list's unused tail entries.
// TMEM, barriers and tensor maps are set up once per CTA. The items are
// pipelined: w (hi, lo) is staged in LA and u in the operand tiles (V = 256:
// and in LA), so the k and v buffers are free as soon as the products have
// read them. For V <= 128 the next item's k and v stream in behind this item's
// epilogues; for V = 256 the second round of value columns streams into the k
// buffer once the W product has read it, the next item's first round into the
// v buffer after the first U product and its k after the second. The bulk
// stores only have to have read their staging before the next item writes LA
// (or, for the operand tiles, before its solve). Warp 15, idle in the second
// tile build, stages the next item's beta and decay and takes their
// compensated prefix there.
// G = false is the ungated form (no decay, g = None on the pages): the decay
// prefixes stay zero and no exponential is taken.
// C64: the item is two of the pages' 64-position chunks, each with its own
// transition block, inverse and decay prefix (odd M, whose state recurrence
// steps 64 positions): the L block coupling the two is zero, the prefix
// restarts at position 64, and the inverse skips its top merge (A10 = 0), so
// w, u and the decay records are those of the 64-position chunks.
template <int V, bool G, bool C64>
__global__ void __launch_bounds__(512, 1) wy128_tc_kernel(
    const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
    const __grid_constant__ CUtensorMap map_whs, const __grid_constant__ CUtensorMap map_wls,
    const __grid_constant__ CUtensorMap map_us, WyArgs a, int NB) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  constexpr bool kPipe = V <= 128;
  constexpr int VR = V < 128 ? V : 128;          // value columns per round
  constexpr int NR = V / VR;                     // rounds
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, cq = warp >> 2;  // TMEM lane quarter, column quarter
  const int M = a.M;
  const int n_items = NB * a.HV;
  // a block's record (one 16-byte load); items past the end read as invalid
  auto tab_of = [&](int i) { return i < n_items ? a.blk_tab[i % NB] : make_int4(-1, 0, 0, 0); };
  int it = blockIdx.x;
  int4 tab = tab_of(it);
  while (it < n_items && tab.x < 0) tab = tab_of(it += gridDim.x);  // only the padded tail
  if (it >= n_items) return;
  struct Item {
    int hv, kh, n, b_start, t0;
    int64_t R0;
  };
  auto item = [&](int i, int4 tb) {
    Item x;
    x.hv = i / NB;
    x.kh = x.hv / (a.HV / a.H);
    x.b_start = tb.y * kBT;
    x.n = min(128, tb.w * M - x.b_start);
    x.t0 = tb.z;
    x.R0 = (int64_t)tb.z * M + x.b_start;
    return x;
  };
  // the next item's record is loaded one item ahead, so no item waits on it
  int nx = it + gridDim.x;
  int4 ntab = tab_of(nx);
  // beta and the decay (on a token's first copy) of position p of item x
  auto gates = [&](const Item& x, int p, float& b, float& gl) {
    b = 0.f;
    gl = 0.f;
    if (p < x.n) {
      const int e = x.b_start + p, t = e / M;
      b = a.beta[(x.R0 + p) * a.HV + x.hv];
      if (a.g && e - t * M == 0) gl = a.g[((int64_t)x.t0 + t) * a.HV + x.hv];
    }
  };
  uint8_t* kbuf = sm + W8_K;
  uint8_t* vbuf = sm + W8_V;
  uint8_t* tiles = sm + W8_T;
  float* LA = reinterpret_cast<float*>(sm + W8_LA);
  float* Ld = reinterpret_cast<float*>(sm + W8_LD);
  float* scratch = reinterpret_cast<float*>(tiles);
  // [2][7][128] by item parity: beta, Gam hi, Gam lo, 1/|k|, column scale,
  // Gam hi and lo in base 2
  float* sarr = reinterpret_cast<float*>(sm + W8_S);
  // [0] k, [1] mma, [2] v round, [3] solve MMAs, [4] v, [5] the next item's Gram
  uint64_t* bars = reinterpret_cast<uint64_t*>(sarr + 2 * 7 * 128);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 6);
  // TMEM: Gram, solve scratch, W [0, 128), U [128, 128 + V); with V <= 128 (and
  // 128-position items) the next item's Gram product is issued early, into
  // [TGE, TGE + 128)
  constexpr uint32_t kCols = 512;
  constexpr uint32_t TGE = 384;
  auto issue_k = [&](const Item& x) {
    mbar_expect_tx(&bars[0], 32768);
    tma_load_3d(kbuf, &map_k, 0, x.kh, (int)x.R0, &bars[0]);
    tma_load_3d(kbuf + 16384, &map_k, 64, x.kh, (int)x.R0, &bars[0]);
  };
  auto issue_v = [&](const Item& x) {
    mbar_expect_tx(&bars[4], (VR / 64) * 16384);
#pragma unroll
    for (int c = 0; c < VR / 64; ++c) tma_load_3d(vbuf + c * 16384, &map_v, 64 * c, x.hv, (int)x.R0, &bars[4]);
  };
  if (warp == 0) {
    tmem_alloc(s_tmem, kCols);
    tmem_relinquish();
  }
  Item x = item(it, tab);
  if (tid == 0) {
    for (int i = 0; i < 6; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    issue_k(x);
    issue_v(x);
  }
  if (tid < 128) gates(x, tid, sarr[tid], sarr[128 + tid]);
  if (!G) {  // both parities' decay prefixes (hi, lo; base e and base 2) stay zero
    for (int i = tid; i < 2 * 128; i += 512) {
      const int par = i >> 7, j = i & 127;
      float* sp = sarr + par * 896;
      sp[128 + j] = sp[256 + j] = sp[640 + j] = sp[768 + j] = 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (G && warp == 0) comp_prefix128_warp<C64>(sarr + 128, sarr + 256, lane);
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  uint32_t mma_phase = 0;
  // k / v loads issued and consumed so far: load i completes phase i of bars[0] / bars[4]
  int k_iss = 1, k_got = 0, v_iss = 1, v_got = 0;
  int r_iss = 0, r_got = 0;  // V = 256: loads of the second value round (bars[2])
  bool gram_early = false;   // this item's Gram product was issued during the previous item
  uint32_t ge_phase = 0;     // bars[5] phase
  bool ok = true;
  for (int c = 0;; ++c) {
    const int par = c & 1;
    float* sb = sarr + par * 896;
    float* sgh = sb + 128;
    float* sgl = sgh + 128;
    float* srk = sgl + 128;
    float* sco = srk + 128;
    float* s2h = sco + 128;
    float* s2l = s2h + 128;
    float* nsb = sarr + (par ^ 1) * 896;  // the next item's beta and decay
    while (nx < n_items && ntab.x < 0) ntab = tab_of(nx += gridDim.x);  // only the padded tail
    const bool has_next = nx < n_items;
    const Item y = has_next ? item(nx, ntab) : x;
    const int nnx = nx + gridDim.x;
    const int4 nntab = tab_of(nnx);  // used by the next iteration
    float pb[4], pg[4];  // warp 15: the next item's gate inputs (positions 4 lane + i)
    if (warp == 15 && has_next) {
#pragma unroll
      for (int i = 0; i < 4; ++i) gates(y, 4 * lane + i, pb[i], pg[i]);
    }
    const int n = x.n, hv = x.hv;
    const int64_t R0 = x.R0;
    ok = mbar_wait(&bars[0], k_got & 1, a.status, kDevTimeout);
    if (ok) ++k_got;
    if (!__syncthreads_and(ok)) break;
    // (the test hook leaves CTA 0's first Gram product, and so its commit, out:
    // every thread's bounded wait below then runs out and the CTA leaves cleanly)
    // Gram k k^T, 128 x 128: issued beside the row norms of tid < 128, unless the
    // previous item already issued it into [TGE, TGE + 128)
    if (!gram_early && tid == 128 && !(a.fault && blockIdx.x == 0 && c == 0)) {
      const uint32_t kb = smem_u32(kbuf);
      const uint32_t id = idesc_bf16(128, 128, false, false);
      const uint64_t d0 = sdesc_sw128(kb, 16, 1024);
      mma_run<8, false, 16384, 32, 16384, 32>(tmem, d0, d0, id);
      mma_commit(&bars[1]);
    }
    const uint32_t tg = gram_early ? TGE : 0u;  // this item's Gram columns
    if (tid < 128) {
      const float ss = row_sumsq(kbuf + tid * 128, tid) + row_sumsq(kbuf + 16384 + tid * 128, tid);
      const float r = a.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
      srk[tid] = r;
      if (G) {
        sco[tid] = sb[tid] * expf(sgh[tid] + sgl[tid]) * r;
        const float2 g2 = log2e_pair(sgh[tid], sgl[tid]);
        s2h[tid] = g2.x;
        s2l[tid] = g2.y;
      } else {
        sco[tid] = sb[tid] * r;
      }
    }
    fence_async_smem();  // the k buffer's generic reads end before the next k load
    // The previous item's w stores (staged in LA, which the L build overwrites)
    // must have read shared memory; its u stores (staged in the operand tiles,
    // the solve's scratch, and for V = 256 also in LA) may go on reading until
    // just before the solve (V = 256: the L build).
    if (tid == 0) {
      if (kPipe)
        tma_store_wait_read_but_last();
      else
        tma_store_wait_read();
    }
    if (gram_early) {
      ok = mbar_wait(&bars[5], ge_phase, a.status, kDevTimeout);
      ge_phase ^= 1;
    } else {
      ok = mbar_wait(&bars[1], mma_phase, a.status, kDevTimeout);
      mma_phase ^= 1;
    }
    tc_fence_after();
    if (!__syncthreads_and(ok)) break;
    {  // L[p][i] = beta_p e^(Gam_p - Gam_i) k_p.k_i / (|k_p||k_i|) for i < p
      const int p = quarter * 32 + lane;
      const float bp = sb[p] * srk[p];
      const int c0 = cq * 32;
      // blocks on or above the diagonal, and for C64 the block coupling the two chunks: zeros
      if (cq > quarter || (C64 && quarter >= 2 && cq < 2)) {
#pragma unroll
        for (int j = 0; j < 32; ++j) LA[p * 129 + c0 + j] = 0.f;
      } else {
        uint32_t r[32];
        GDP_TMEM_LD32(tmem + lane_base + tg + c0, r);
        tmem_wait_ld();
        const f2 ph2 = pk2(s2h[p], s2h[p]), pl2 = pk2(s2l[p], s2l[p]), bp2 = pk2(bp, bp);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {  // column pairs, branch-free so that they interleave
          const int i = c0 + j;
          const f2 ih = *reinterpret_cast<const f2*>(s2h + i);
          const f2 il = *reinterpret_cast<const f2*>(s2l + i);
          const f2 rk = *reinterpret_cast<const f2*>(srk + i);
          const f2 kk = mul2(rk, pk2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])));
          float2 v;
          if (G) {
            const float2 d = upk2(add2(sub2(ph2, ih), sub2(pl2, il)));  // Gam_p - Gam_i, base 2
            v = upk2(mul2(mul2(bp2, pk2(ex2_approx(d.x), ex2_approx(d.y))), kk));
          } else {
            v = upk2(mul2(bp2, kk));
          }
          // (the register array r now carries this row's L values)
          r[j] = __float_as_uint((i < p) ? v.x : 0.f);
          r[j + 1] = __float_as_uint((i + 1 < p) ? v.y : 0.f);
          LA[p * 129 + i] = __uint_as_float(r[j]);
          LA[p * 129 + i + 1] = __uint_as_float(r[j + 1]);
        }
        if (cq == quarter) {  // a diagonal block: also its aligned, swizzled copy
          float* ld = Ld + quarter * 1024 + lane * 32;
#pragma unroll
          for (int qq = 0; qq < 8; ++qq)
            *reinterpret_cast<uint4*>(ld + ((qq ^ (lane & 7)) << 2)) =
                make_uint4(r[4 * qq], r[4 * qq + 1], r[4 * qq + 2], r[4 * qq + 3]);
        }
      }
    }
    if (tid == 0) tma_store_wait_read();  // the u stores have read the operand tiles
    tc_fence_before();
    __syncthreads();
    ok = solve_tril128<C64>(LA, Ld, scratch, tmem, &bars[3], a.status);
    if (!ok) break;
    // operand tiles for pass `which`: 0 -> A diag(beta e^Gam/|k|) (for w), 1 -> A diag(beta) (for u).
    // Warp w builds one 32 x 32 chunk (row block R, column block C) of A, lane =
    // row 32 R + lane: LA rows (stride 129) are read without bank conflicts,
    // the column scales are broadcasts, and each 8-column group is one 16-byte
    // swizzled store per half. Warps 0-9 take the ten chunks on or below the
    // diagonal, ordered so that each SM sub-partition (warps s, s + 4, ...) gets
    // two or three of them; warps 10-15 write the six zero chunks above the
    // diagonal in the first build (the second leaves them in place: the w MMAs
    // only read them), and in the second build warp 15 stages the next item's
    // gates and takes their prefix.
    auto build_tiles = [&](int which) {
      // (R, C) by warp, one hex digit per warp (warp 0 lowest): lower chunks
      // (0,0) (1,0) (2,0) (3,0) (1,1) (2,1) (3,1) (2,2) (3,2) (3,3), then the
      // zero chunks (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
      const float* sc = which == 0 ? sco : sb;
      const int R = (int)((0x2110003323213210ull >> (4 * warp)) & 15), C = (int)((0x3323213221110000ull >> (4 * warp)) & 15);
      const int p = R * 32 + lane, c0 = C * 32;
      uint8_t* trow = tiles + (c0 >> 6) * 16384 + p * 128;
      const int ch0 = (c0 & 63) >> 3;
      if (warp < 10) {
        const float* lrow = LA + p * 129 + c0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          __align__(16) bf16 hi[8];
          __align__(16) bf16 lo[8];
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = lrow[8 * q + e] * sc[c0 + 8 * q + e];
          split_bf16_n<8>(v, hi, lo);
          const uint32_t off = ((ch0 + q) ^ (p & 7)) << 4;
          *reinterpret_cast<uint4*>(trow + off) = *reinterpret_cast<const uint4*>(hi);
          *reinterpret_cast<uint4*>(trow + 32768 + off) = *reinterpret_cast<const uint4*>(lo);
        }
      } else if (which == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t off = ((ch0 + q) ^ (p & 7)) << 4;
          *reinterpret_cast<uint4*>(trow + off) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(trow + 32768 + off) = make_uint4(0, 0, 0, 0);
        }
      } else if (warp == 15 && has_next) {
        *reinterpret_cast<float4*>(nsb + 4 * lane) = make_float4(pb[0], pb[1], pb[2], pb[3]);
        if (G) {
          *reinterpret_cast<float4*>(nsb + 128 + 4 * lane) = make_float4(pg[0], pg[1], pg[2], pg[3]);
          __syncwarp();
          comp_prefix128_warp<C64>(nsb + 128, nsb + 256, lane);
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    };
    build_tiles(0);
    if (tid == 0) {  // w = A' k: M = 128 positions, N = 128, K = 128 positions
      const uint32_t tb = smem_u32(tiles), kb = smem_u32(kbuf);
      const uint32_t idw = idesc_bf16(128, 128, false, true);
      const uint64_t kd = sdesc_sw128(kb, 16384, 1024);
      mma_run<8, false, 16384, 32, 8192, 2048>(tmem, sdesc_sw128(tb, 16, 1024), kd, idw);
      mma_run<8, true, 16384, 32, 8192, 2048>(tmem, sdesc_sw128(tb + 32768, 16, 1024), kd, idw);
      mma_commit(&bars[1]);
    }
    ok = mbar_wait(&bars[1], mma_phase, a.status, kDevTimeout);
    mma_phase ^= 1;
    tc_fence_after();
    if (!__syncthreads_and(ok)) break;
    if (kPipe && has_next) {  // the W product was the k buffer's last reader
      if (tid == 0) issue_k(y);
      ++k_iss;
    }
    if (!kPipe && tid == 0) {  // V = 256: the value columns of round 1 go to the k buffer
      mbar_expect_tx(&bars[2], (VR / 64) * 16384);
#pragma unroll
      for (int c2 = 0; c2 < VR / 64; ++c2)
        tma_load_3d(kbuf + c2 * 16384, &map_v, VR + 64 * c2, x.hv, (int)x.R0, &bars[2]);
    }
    if (!kPipe) ++r_iss;
    build_tiles(1);
    ok = mbar_wait(&bars[4], v_got & 1, a.status, kDevTimeout);
    if (ok) ++v_got;
    if (!__syncthreads_and(ok)) break;
    auto issue_u = [&](int round) {
      const uint32_t tb = smem_u32(tiles), vb = smem_u32(round == 0 ? vbuf : kbuf);
      const uint32_t idu = idesc_bf16(128, VR, false, true);
      const uint64_t vd = sdesc_sw128(vb, 16384, 1024);
      mma_run<8, false, 16384, 32, 8192, 2048>(tmem + 128 + round * VR, sdesc_sw128(tb, 16, 1024), vd, idu);
      mma_run<8, true, 16384, 32, 8192, 2048>(tmem + 128 + round * VR, sdesc_sw128(tb + 32768, 16, 1024), vd, idu);
      mma_commit(&bars[1]);
    };
    if (tid == 0) issue_u(0);
    // Epilogues. A whole block is staged in shared memory that its last reader
    // has released and written with bulk tensor stores; a sequence's last,
    // partial block is written row by row, so that no store reaches the rows of
    // the next sequence.
    const bool full = n == 128;
    // w staging, two 64-column boxes per array, w_hi and w_lo in LA
    uint8_t* whs = reinterpret_cast<uint8_t*>(LA);
    uint8_t* wls = reinterpret_cast<uint8_t*>(LA) + 32768;
    {  // w epilogue (overlaps the u MMAs): row p, 32 of the 128 columns per thread
      const int p = quarter * 32 + lane;
      const int c0 = cq * 32;
      uint32_t r[32];
      GDP_TMEM_LD32(tmem + lane_base + c0, r);
      tmem_wait_ld();
      __align__(16) bf16 hi[32];
      __align__(16) bf16 lo[32];
      split_bf16_n<32>(reinterpret_cast<const float*>(r), hi, lo);
      if (full) {
        const uint32_t base = (c0 >> 6) * 16384 + p * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t off = base + (((((c0 & 63) >> 3) + i) ^ (p & 7)) << 4);
          *reinterpret_cast<uint4*>(whs + off) = reinterpret_cast<const uint4*>(hi)[i];
          *reinterpret_cast<uint4*>(wls + off) = reinterpret_cast<const uint4*>(lo)[i];
        }
      } else if (p < n) {
        const int64_t row = ((R0 + p) * a.HV + hv) * kK + c0;
        store_bf16x32(a.w_hi + row, hi);
        store_bf16x32(a.w_lo + row, lo);
      }
    }
    if (full) {
      fence_async_smem();
      __syncthreads();
      if (tid == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tma_store_3d(&map_whs, whs + h * 16384, 64 * h, hv, (int)R0);
          tma_store_3d(&map_wls, wls + h * 16384, 64 * h, hv, (int)R0);
        }
        tma_store_commit();
      }
    }
#pragma unroll 1
    for (int round = 1; round < NR; ++round) {  // V = 256: second half of the value columns
      ok = mbar_wait(&bars[1], mma_phase, a.status, kDevTimeout);
      mma_phase ^= 1;
      if (!__syncthreads_and(ok)) break;
      if (has_next) {  // U round 0 was the v buffer's last reader
        if (tid == 0) issue_v(y);
        ++v_iss;
      }
      // round 1's columns were requested into the k buffer after the W product
      ok = mbar_wait(&bars[2], (c * (NR - 1) + round - 1) & 1, a.status, kDevTimeout);
      if (ok) ++r_got;
      if (!__syncthreads_and(ok)) break;
      if (tid == 0) issue_u(round);
    }
    if (!ok) break;
    ok = mbar_wait(&bars[1], mma_phase, a.status, kDevTimeout);
    mma_phase ^= 1;
    tc_fence_after();
    // V = 256: u boxes 4-7 go to LA, which the w stores must have read
    if (!kPipe && tid == 0) tma_store_wait_read();
    if (!__syncthreads_and(ok)) break;
    // V <= 128: the next item's k was requested after the W product; its Gram
    // product goes to the spare columns now, behind this item's u epilogue (not
    // for C64, whose shorter items reach this point before that k has landed:
    // measured slower)
    const bool early_next = kPipe && !C64 && has_next;
    if (early_next && tid == 128) {
      if (mbar_wait(&bars[0], k_got & 1, a.status, kDevTimeout)) {
        tc_fence_after();
        const uint32_t kb = smem_u32(kbuf);
        const uint32_t id = idesc_bf16(128, 128, false, false);
        const uint64_t d0 = sdesc_sw128(kb, 16, 1024);
        mma_run<8, false, 16384, 32, 16384, 32>(tmem + TGE, d0, d0, id);
        mma_commit(&bars[5]);
      }
    }
    if (has_next) {
      if (kPipe) {  // the U product was the v buffer's last reader
        if (tid == 0) issue_v(y);
        ++v_iss;
      } else {  // U round 1 was the k buffer's last reader
        if (tid == 0) issue_k(y);
        ++k_iss;
      }
    }
    // u staging: 32-column boxes, 0-3 in the operand tiles, 4-7 (V = 256) in LA;
    // the loads of the next item use neither
    auto ustage = [&](int cc) -> uint8_t* {
      return cc < 4 ? tiles + cc * 16384 : reinterpret_cast<uint8_t*>(LA) + (cc - 4) * 16384;
    };
    {  // u epilogue: row p, V / 4 columns per thread
      const int p = quarter * 32 + lane;
#pragma unroll 1
      for (int c0 = cq * (V / 4); c0 < (cq + 1) * (V / 4); c0 += 16) {
        uint32_t r[16];
        GDP_TMEM_LD16(tmem + lane_base + 128 + c0, r);
        tmem_wait_ld();
        if (full) {
          uint8_t* st = ustage(c0 >> 5) + p * 128;
          const int u0 = (c0 & 31) >> 2;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<float4*>(st + (((u0 + j) ^ (p & 7)) << 4)) =
                make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                            __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        } else if (p < n) {
          float4* dst = reinterpret_cast<float4*>(a.u + ((R0 + p) * a.HV + hv) * V + c0);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
      }
      if (tid < n) a.gk[(int64_t)hv * a.Te + R0 + tid] = make_float4(sgh[tid], sgl[tid], srk[tid], 0.f);
    }
    if (full) fence_async_smem();
    tc_fence_before();
    __syncthreads();  // TMEM reads and the staging are done
    tc_fence_after();
    if (tid == 0) {
      if (full) {
#pragma unroll
        for (int cc = 0; cc < V / 32; ++cc) tma_store_3d(&map_us, ustage(cc), 32 * cc, hv, (int)R0);
        tma_store_commit();
      }
    }
    if (!has_next) break;
    gram_early = early_next;
    it = nx;
    x = y;
    nx = nnx;
    ntab = nntab;
  }
  if (tid == 0) {  // nothing may still write or read shared memory when the CTA leaves
    bool w = true;
    for (; w && k_got < k_iss; ++k_got) w = mbar_wait(&bars[0], k_got & 1, nullptr, 0);
    for (; w && v_got < v_iss; ++v_got) w = mbar_wait(&bars[4], v_got & 1, nullptr, 0);
    for (; w && r_got < r_iss; ++r_got) w = mbar_wait(&bars[2], r_got & 1, nullptr, 0);
    tma_store_wait_read();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  tmem_release(tmem, kCols);
}

// ============================================================================ chunk_h, 128-position steps
// Shared memory of the state chain on 128-position blocks (the chain warps of
// ho128_tc_kernel below). Operand buffers are single: each group is refilled
// for the next block as soon as its last consumer of this block is done (w
// after product 1, u and the per-position records after the value phase, k
// after product 2).
constexpr int S8_WHI = 0;                   // w hi: 2 K-halves x 128 rows x 128 B
constexpr int S8_WLO = 32768;               // w lo
constexpr int S8_K = 65536;                 // k: 2 K-halves x 128 rows x 128 B
constexpr int S8_U = 98304;                 // u fp32 128 x 32
constexpr int S8_G = 114688;                // (Gam hi, Gam lo, 1/|k|, 0) x 128

// ============================================================================ chunk_h + chunk_o, M = 2
// For M = 2 a 128-position block is exactly one 64-token output chunk, so the
// output of a block can be formed from what the scan CTA already holds on
// chip: the state at the start of the block (product 1's h tile), the block's
// keys (product 2's k tile) and v_new. Neither states nor v_new go to HBM.
//
// Warp roles (512 threads):
//  * warps 0-7, the chain: the state recurrence of h_tc_kernel, one
//    128-position block per step (WY factors from wy128_tc_kernel, every
//    accumulator row in use). Thread
//    (warp w, lane l) owns state row / position 32 (w % 4) + l and value
//    columns [16 (w / 4), +16) of the CTA's 32. Besides the v' operand it
//    writes v_new / |k_p| as the output's operand tile.
//  * warps 8-15, the output: per block, from S^T = k q^T (positions x tokens)
//    and Qh = q h (tokens x columns), the masked decayed scores
//      P^T[e][t] = S^T[e][t] e^(Gam_t - Gam_e),  e <= 2t + 1,
//    as hi/lo operand tiles (thread = position e, 32 tokens), then
//    O = P (v_new / |k|) and o_t = scale |q_t|^-1 (e^Gam_t Qh_t + O_t), Gam_t
//    being the cumulative log decay at the token's last copy. Warps idle in
//    the epilogue compute the next block's token records (Gam_t, 1/|q_t|).
// A single thread issuing a whole product was a bottleneck, so products are
// issued from several threads into their own accumulators (summed when read):
// product 1 by chain threads 0 and 32, product 2 by thread 0 with Qh and S
// beside it from threads 32 and 64, O by output threads 0 and 32. S and Qh go
// to one of two TMEM column sets by block parity. The groups meet only at
// mbarriers (P1, O: two commits each; QH[b]: Qh done, the h tile may be
// re-written, q may be re-loaded; S[b] and P2: k may be re-loaded; VN: v_new
// written; O: O done, v_new may be re-written; E[b]: the output of a block is
// finished, its column set may be re-used). Each group syncs internally with
// its own named barrier.
struct HOArgs {
  HArgs h;
  int H, l2norm;
  float scale;
  float* o;
};

constexpr int F_OG = 116736;                // output group's records: 2 buffers x 128 x 16 B
constexpr int F_HT = F_OG + 4096;           // h operand hi | lo
constexpr int F_VP = F_HT + 16384;          // v' operand hi | lo
constexpr int F_Q = F_VP + 16384;           // q: 2 K-halves x 64 rows x 128 B
constexpr int F_VN = F_Q + 16384;           // v_new operand hi | lo: 128 rows x 64 B each
constexpr int F_P = F_VN + 16384;           // P^T operand hi | lo: 128 rows (e) x 128 B (64 t)
constexpr int F_SM = F_P + 32768;           // token records x 2, barriers, TMEM address
constexpr int F_SMEM = F_SM + 2048 + 16 * 8 + 16 + 1024;
enum { FB_W, FB_UG, FB_K, FB_Q, FB_OG0, FB_OG1, FB_P1, FB_P2, FB_QH0, FB_QH1, FB_S0, FB_S1,
       FB_O, FB_E0, FB_E1, FB_VN, FB_N };

// AND of pred over the count threads of named barrier id (warp-uniform use)
__device__ __forceinline__ bool group_and(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(count) : "memory");
  return r != 0;
}

template <bool G, bool ORD>
__global__ void __launch_bounds__(512, 1) ho128_tc_kernel(
    const __grid_constant__ CUtensorMap map_whi, const __grid_constant__ CUtensorMap map_wlo,
    const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_u,
    const __grid_constant__ CUtensorMap map_gk, const __grid_constant__ CUtensorMap map_q,
    HOArgs f, const int* seq_order) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, cgrp = (warp >> 2) & 1;
  const int row = quarter * 32 + lane;
  constexpr int NC = 16;
  const int cb = cgrp * NC;
  const int HVn = f.h.HV, V = f.h.V;
  const int nsl = V / kHBV;
  // ORD: ragged sequences, launched longest first; dense batches: blockIdx.x =
  // sequence * (V / 32) + value slice (slices of one head side by side)
  int seq, hv, v0;
  if (ORD) {
    const ChainPos cp = chain_pos(seq_order, nsl, HVn);
    seq = cp.seq;
    hv = cp.hv;
    v0 = cp.slice * kHBV;
  } else {
    seq = blockIdx.x / nsl;
    hv = blockIdx.y;
    v0 = (blockIdx.x - seq * nsl) * kHBV;
  }
  const int kh = hv / (HVn / f.H);
  const int4 si = f.h.seq_info[seq];
  const int nb = (int)cdiv((int64_t)si.y * 2, 128);
  int* status = f.h.status;
  uint8_t* ht = sm + F_HT;
  uint8_t* vp = sm + F_VP;
  uint8_t* vnt = sm + F_VN;
  uint8_t* pt = sm + F_P;
  // per token, by block parity: [64] Gam hi, [64] Gam lo (base 2), [64] 1/|q|
  float* stok2 = reinterpret_cast<float*>(sm + F_SM);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + F_SM + 2048);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 16);
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const int64_t Rseq = (int64_t)si.x * 2;
  const int64_t gk_base = (int64_t)hv * f.h.Te + Rseq;
  // TMEM columns: D1 [0,64) D2 [64,128) O [128,192) S^T[b] [192 + 64b, +64)
  // Qh[b] [320 + 64b, +64). The hi and lo halves of an operand tile sit 8 KB
  // apart, the leading-byte offset of a 64-column MN-major operand, so
  // x_hi [y_hi | y_lo] is one N = 64 MMA per k-step (columns [0,32) take
  // x_hi y_hi, [32,64) x_hi y_lo) and the lo-hi term accumulates into [0,32):
  // a product is the sum of its two 32-column halves.
  constexpr uint32_t TD1 = 0, TD2 = 64, TO = 128, TS = 192, TQH = 320, TD1B = 448, TOB = 480;

  if (warp == 0) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < FB_N; ++i) mbar_init(&bars[i], (i == FB_P1 || i == FB_O) ? 2 : 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t off_r0 = sw64_chunk(row, 2 * cgrp), off_r1 = sw64_chunk(row, 2 * cgrp + 1);

  if (warp < 8) {  // ------------------------------------------------ chain
    const int64_t hoff = ((int64_t)seq * HVn + hv) * kK * V;
    float h[NC];
    {
      const float* src = f.h.h0 ? f.h.h0 + hoff + (int64_t)row * V + v0 + cb : nullptr;
#pragma unroll
      for (int c = 0; c < NC; ++c) h[c] = src ? src[c] : 0.f;
    }
    auto load_w = [&](int64_t R) {
      mbar_expect_tx(&bars[FB_W], 65536);
      tma_load_3d(sm + S8_WHI, &map_whi, 0, hv, (int)R, &bars[FB_W]);
      tma_load_3d(sm + S8_WHI + 16384, &map_whi, 64, hv, (int)R, &bars[FB_W]);
      tma_load_3d(sm + S8_WLO, &map_wlo, 0, hv, (int)R, &bars[FB_W]);
      tma_load_3d(sm + S8_WLO + 16384, &map_wlo, 64, hv, (int)R, &bars[FB_W]);
    };
    auto load_ug = [&](int64_t R, int64_t grow) {
      mbar_expect_tx(&bars[FB_UG], 16384 + 2048);
      tma_load_3d(sm + S8_U, &map_u, v0, hv, (int)R, &bars[FB_UG]);
      tma_load_2d(sm + S8_G, &map_gk, 0, (int)grow, &bars[FB_UG]);
    };
    if (tid == 0 && nb > 0) {
      load_w(Rseq);
      load_ug(Rseq, gk_base);
    }
    const uint32_t id1w = idesc_bf16(128, 2 * kHBV, false, true);
    const uint32_t id1 = idesc_bf16(128, kHBV, false, true);
    const uint32_t id2w = idesc_bf16(128, 2 * kHBV, true, true);
    const uint32_t ids = idesc_bf16(128, 64, false, false);
    bool ok = true;
    for (int j = 0; j <= nb; ++j) {
      // the h tile is re-written once Qh of the previous block has read it
      if (j > 0)
        ok = mbar_wait(&bars[FB_QH0 + ((j - 1) & 1)], ((j - 1) >> 1) & 1, status, kDevTimeout) && ok;
      {
        __align__(16) bf16 hi[NC];
        __align__(16) bf16 lo[NC];
        split_bf16_n<NC>(h, hi, lo);
        const uint4* h4 = reinterpret_cast<const uint4*>(hi);
        const uint4* l4 = reinterpret_cast<const uint4*>(lo);
        *reinterpret_cast<uint4*>(ht + off_r0) = h4[0];
        *reinterpret_cast<uint4*>(ht + off_r1) = h4[1];
        *reinterpret_cast<uint4*>(ht + 8192 + off_r0) = l4[0];
        *reinterpret_cast<uint4*>(ht + 8192 + off_r1) = l4[1];
      }
      if (j == nb) break;
      fence_async_smem();
      tc_fence_before();
      ok = group_and(1, 256, ok);
      if (!ok) break;
      tc_fence_after();
      const int n = min(128, si.y * 2 - j * 128);
      const int64_t R = Rseq + (int64_t)j * 128;
      const uint32_t ph = j & 1;
      if (tid == 0 || tid == 32) {  // product 1: D1 = w h, issued from two warps
        ok = mbar_wait(&bars[FB_W], ph, status, kDevTimeout);
        if (ok) {
          const uint32_t whi = smem_u32(sm + S8_WHI), wlo = smem_u32(sm + S8_WLO);
          const uint32_t hb = smem_u32(ht);
          if (tid == 0)  // w_hi [h_hi | h_lo]
            mma_run<8, false, 16384, 32, 4096, 1024>(tmem + TD1, sdesc_sw128(whi, 16, 1024),
                                                     sdesc_sw64(hb, 8192, 512), id1w);
          else  // w_lo h_hi, its own accumulator
            mma_run<8, false, 16384, 32, 4096, 1024>(tmem + TD1B, sdesc_sw128(wlo, 16, 1024),
                                                     sdesc_sw64(hb, 8192, 512), id1);
          mma_commit(&bars[FB_P1]);
        }
      }
      ok = mbar_wait(&bars[FB_UG], ph, status, kDevTimeout) && ok;
      const float4* gk = reinterpret_cast<const float4*>(sm + S8_G);
      const float4 glast = gk[n - 1];
      {  // value phase: position p = row, columns cb .. cb + 15
        const int p = row;
        const float4 gp = gk[p];
        const float sc = (p < n) ? (G ? expf((glast.x - gp.x) + (glast.y - gp.y)) : 1.f) * gp.z : 0.f;
        ok = mbar_wait(&bars[FB_P1], ph, status, kDevTimeout) && ok;
        tc_fence_after();
        if (tid == 0 && ok && j + 1 < nb) load_w(R + 128);
        float d1[NC];
        {
          uint32_t r0[NC], r1[NC], r2[NC];
          GDP_TMEM_LD16(tmem + lane_base + TD1 + cb, r0);
          GDP_TMEM_LD16(tmem + lane_base + TD1 + 32 + cb, r1);
          GDP_TMEM_LD16(tmem + lane_base + TD1B + cb, r2);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < NC; ++c)
            d1[c] = (__uint_as_float(r0[c]) + __uint_as_float(r2[c])) + __uint_as_float(r1[c]);
        }
        const uint8_t* urow = sm + S8_U + p * 128;
        __align__(16) bf16 vh[NC];
        __align__(16) bf16 vl[NC];
        __align__(16) bf16 pvh[NC];
        __align__(16) bf16 pvl[NC];
        float vn[NC], pv[NC];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const float4 u4 =
              *reinterpret_cast<const float4*>(urow + ((((cb >> 2) + jj) ^ (p & 7)) << 4));
          const float us[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = 4 * jj + q;
            const float vv = (p < n) ? us[q] - d1[c] : 0.f;
            pv[c] = vv * sc;
            vn[c] = vv * gp.z;  // the output's operand carries the key norm 1/|k_p|
          }
        }
        split_bf16_n<NC>(vn, vh, vl);
        split_bf16_n<NC>(pv, pvh, pvl);
        *reinterpret_cast<uint4*>(vp + off_r0) = reinterpret_cast<const uint4*>(pvh)[0];
        *reinterpret_cast<uint4*>(vp + off_r1) = reinterpret_cast<const uint4*>(pvh)[1];
        *reinterpret_cast<uint4*>(vp + 8192 + off_r0) = reinterpret_cast<const uint4*>(pvl)[0];
        *reinterpret_cast<uint4*>(vp + 8192 + off_r1) = reinterpret_cast<const uint4*>(pvl)[1];
        // the v_new tile is re-written once O of the previous block has read it
        if (j > 0) ok = mbar_wait(&bars[FB_O], (j - 1) & 1, status, kDevTimeout) && ok;
        *reinterpret_cast<uint4*>(vnt + off_r0) = reinterpret_cast<const uint4*>(vh)[0];
        *reinterpret_cast<uint4*>(vnt + off_r1) = reinterpret_cast<const uint4*>(vh)[1];
        *reinterpret_cast<uint4*>(vnt + 8192 + off_r0) = reinterpret_cast<const uint4*>(vl)[0];
        *reinterpret_cast<uint4*>(vnt + 8192 + off_r1) = reinterpret_cast<const uint4*>(vl)[1];
        fence_async_smem();
        tc_fence_before();
      }
      ok = group_and(1, 256, ok);
      if (!ok) break;
      tc_fence_after();
      if (tid == 0) {
        mbar_arrive(&bars[FB_VN]);
        if (j + 1 < nb) load_ug(R + 128, gk_base + (int64_t)(j + 1) * 128);
        ok = mbar_wait(&bars[FB_K], ph, status, kDevTimeout);
        if (ok) {  // product 2: D2 = k^T v', K = 128 positions
          const uint32_t kb = smem_u32(sm + S8_K), vb = smem_u32(vp);
          // k^T [v'_hi | v'_lo]
          mma_run<8, false, 8192, 2048, 4096, 1024>(tmem + TD2, sdesc_sw128(kb, 16384, 1024),
                                                    sdesc_sw64(vb, 8192, 512), id2w);
          mma_commit(&bars[FB_P2]);
        }
      } else if (tid == 32 || tid == 64) {  // Qh (tid 32) and S (tid 64) beside product 2
        // column set cs is re-used once the output has finished block j - 2
        const int cs = j & 1;
        if (j > 1) ok = mbar_wait(&bars[FB_E0 + cs], ((j - 2) >> 1) & 1, status, kDevTimeout) && ok;
        ok = mbar_wait(&bars[FB_Q], ph, status, kDevTimeout) && ok;
        if (tid == 64) ok = mbar_wait(&bars[FB_K], ph, status, kDevTimeout) && ok;
        if (ok) {
          const uint32_t qb = smem_u32(sm + F_Q), kb = smem_u32(sm + S8_K), hb = smem_u32(ht);
          if (tid == 32) {  // Qh = q [h_hi | h_lo]: rows = tokens (64.. unused)
            mma_run<8, false, 8192, 32, 4096, 1024>(tmem + TQH + 64 * cs, sdesc_sw128(qb, 16, 1024),
                                                    sdesc_sw64(hb, 8192, 512), id1w);
            mma_commit(&bars[FB_QH0 + cs]);
          } else {  // S^T = k q^T: rows = the block's 128 positions, columns = 64 tokens
            mma_run<8, false, 16384, 32, 8192, 32>(tmem + TS + 64 * cs, sdesc_sw128(kb, 16, 1024),
                                                   sdesc_sw128(qb, 16, 1024), ids);
            mma_commit(&bars[FB_S0 + cs]);
          }
        }
      }
      ok = mbar_wait(&bars[FB_P2], ph, status, kDevTimeout) && ok;
      tc_fence_after();
      {
        uint32_t r0[NC], r1[NC];
        GDP_TMEM_LD16(tmem + lane_base + TD2 + cb, r0);
        GDP_TMEM_LD16(tmem + lane_base + TD2 + 32 + cb, r1);
        tmem_wait_ld();
        const float dl = G ? expf(glast.x + glast.y) : 1.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) h[c] = dl * h[c] + (__uint_as_float(r0[c]) + __uint_as_float(r1[c]));
      }
      tc_fence_before();
    }
    if (f.h.hT) {
      float* dst = f.h.hT + hoff + (int64_t)row * V + v0 + cb;
#pragma unroll
      for (int c = 0; c < NC; c += 4)
        *reinterpret_cast<float4*>(dst + c) = make_float4(h[c], h[c + 1], h[c + 2], h[c + 3]);
    }
  } else {  // ------------------------------------------------------ output
    const int otid = tid - 256;
    auto load_q = [&](int64_t T0) {
      mbar_expect_tx(&bars[FB_Q], 16384);
      tma_load_3d(sm + F_Q, &map_q, 0, kh, (int)T0, &bars[FB_Q]);
      tma_load_3d(sm + F_Q + 8192, &map_q, 64, kh, (int)T0, &bars[FB_Q]);
    };
    auto load_k = [&](int64_t R) {
      mbar_expect_tx(&bars[FB_K], 32768);
      tma_load_3d(sm + S8_K, &map_k, 0, kh, (int)R, &bars[FB_K]);
      tma_load_3d(sm + S8_K + 16384, &map_k, 64, kh, (int)R, &bars[FB_K]);
    };
    auto load_og = [&](int b, int64_t grow) {
      mbar_expect_tx(&bars[FB_OG0 + b], 2048);
      tma_load_2d(sm + F_OG + b * 2048, &map_gk, 0, (int)grow, &bars[FB_OG0 + b]);
    };
    if (otid == 0 && nb > 0) {
      load_k(Rseq);
      load_q(si.x);
      load_og(0, gk_base);
      if (nb > 1) load_og(1, gk_base + 128);
    }
    // token t of block jb: Gam at its last copy, query norm from the staged q
    // tile (waits for that block's q tile and records)
    auto tok_records = [&](int jb, int t, float* dst) -> bool {
      bool okr = mbar_wait(&bars[FB_Q], jb & 1, status, kDevTimeout);
      okr = mbar_wait(&bars[FB_OG0 + (jb & 1)], (jb >> 1) & 1, status, kDevTimeout) && okr;
      const uint8_t* qt = sm + F_Q;
      const float ss = row_sumsq(qt + t * 128, t) + row_sumsq(qt + 8192 + t * 128, t);
      const float4 rt = reinterpret_cast<const float4*>(sm + F_OG + (jb & 1) * 2048)[2 * t + 1];
      const float2 g2 = G ? log2e_pair(rt.x, rt.y) : make_float2(0.f, 0.f);
      dst[t] = g2.x;
      dst[64 + t] = g2.y;
      dst[128 + t] = f.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
      return okr;
    };
    const uint32_t idow = idesc_bf16(128, 2 * kHBV, true, true);
    const uint32_t ido = idesc_bf16(128, kHBV, true, true);
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      const int n = min(128, si.y * 2 - j * 128);
      const int nt = n >> 1;
      const int64_t T0 = (int64_t)si.x + (int64_t)j * 64;
      const uint32_t ph = j & 1;
      const float4* og = reinterpret_cast<const float4*>(sm + F_OG + (j & 1) * 2048);
      float* stok = stok2 + 256 * (j & 1);
      ok = mbar_wait(&bars[FB_OG0 + (j & 1)], (j >> 1) & 1, status, kDevTimeout) && ok;
      if (j == 0 && otid < 64) ok = tok_records(0, otid, stok) && ok;  // later blocks: see the end
      ok = group_and(2, 256, ok);
      if (!ok) break;
      // S done; k is free once product 2 is done too, q once Qh is
      const int cs = j & 1;
      ok = mbar_wait(&bars[FB_S0 + cs], (j >> 1) & 1, status, kDevTimeout);
      tc_fence_after();
      if (otid == 0 && ok && j + 1 < nb) {
        ok = mbar_wait(&bars[FB_P2], ph, status, kDevTimeout);
        ok = mbar_wait(&bars[FB_QH0 + cs], (j >> 1) & 1, status, kDevTimeout) && ok;
        if (ok) {
          load_k(Rseq + (int64_t)(j + 1) * 128);
          load_q(T0 + 64);
        }
      }
      {  // P^T row e = row, tokens [32 cgrp, 32 cgrp + 32)
        const int e = row, s = e >> 1;
        const float4 re = og[e];
        const float2 re2 = log2e_pair(re.x, re.y);
        const f2 rh = pk2(re2.x, re2.x), rl = pk2(re2.y, re2.y);
        uint32_t r[32];
        GDP_TMEM_LD32(tmem + lane_base + TS + 64 * cs + 32 * cgrp, r);
        tmem_wait_ld();
        __align__(16) bf16 ph_[32];
        __align__(16) bf16 pl_[32];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {  // token pairs, branch-free so that they interleave
          const int t = 32 * cgrp + i;
          const f2 th = *reinterpret_cast<const f2*>(stok + t);
          const f2 tl = *reinterpret_cast<const f2*>(stok + 64 + t);
          float2 x;
          if (G) {
            const float2 d = upk2(add2(sub2(th, rh), sub2(tl, rl)));  // Gam_t - Gam_e, base 2
            x = upk2(mul2(pk2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                          pk2(ex2_approx(d.x), ex2_approx(d.y))));
          } else {
            x = make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1]));
          }
          r[i] = __float_as_uint((e < n && s <= t && t < nt) ? x.x : 0.f);
          r[i + 1] = __float_as_uint((e < n && s <= t + 1 && t + 1 < nt) ? x.y : 0.f);
        }
        split_bf16_n<32>(reinterpret_cast<const float*>(r), ph_, pl_);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t off = e * 128 + ((((uint32_t)(4 * cgrp + q)) ^ (e & 7)) << 4);
          *reinterpret_cast<uint4*>(pt + off) = reinterpret_cast<const uint4*>(ph_)[q];
          *reinterpret_cast<uint4*>(pt + 16384 + off) = reinterpret_cast<const uint4*>(pl_)[q];
        }
        fence_async_smem();
        tc_fence_before();
      }
      ok = group_and(2, 256, ok);
      if (!ok) break;
      tc_fence_after();
      if (otid == 0 || otid == 32) {  // O = P v_new from two warps; A = P^T MN-major (LBO = 0)
        ok = mbar_wait(&bars[FB_VN], ph, status, kDevTimeout);
        if (ok) {
          const uint32_t pb = smem_u32(pt), vv = smem_u32(vnt);
          if (otid == 0)  // P_hi [vn_hi | vn_lo]
            mma_run<8, false, 8192, 2048, 4096, 1024>(tmem + TO, sdesc_sw128(pb, 0, 1024),
                                                      sdesc_sw64(vv, 8192, 512), idow);
          else  // P_lo vn_hi, its own accumulator
            mma_run<8, false, 8192, 2048, 4096, 1024>(tmem + TOB, sdesc_sw128(pb + 16384, 0, 1024),
                                                      sdesc_sw64(vv, 8192, 512), ido);
          mma_commit(&bars[FB_O]);
        }
      }
      if (quarter < 2) {  // output rows t = row, columns cb .. cb + 15
        const int t = row;
        ok = mbar_wait(&bars[FB_O], ph, status, kDevTimeout) && ok;
        tc_fence_after();
        ok = mbar_wait(&bars[FB_QH0 + cs], (j >> 1) & 1, status, kDevTimeout) && ok;
        uint32_t ro[16], ro2[16], ro3[16], rq[16], rq2[16];
        GDP_TMEM_LD16(tmem + lane_base + TO + cb, ro);
        GDP_TMEM_LD16(tmem + lane_base + TO + 32 + cb, ro2);
        GDP_TMEM_LD16(tmem + lane_base + TOB + cb, ro3);
        GDP_TMEM_LD16(tmem + lane_base + TQH + 64 * cs + cb, rq);
        GDP_TMEM_LD16(tmem + lane_base + TQH + 64 * cs + 32 + cb, rq2);
        tmem_wait_ld();
        if (t < nt && ok) {
          const float qs = G ? ex2_approx(stok[t] + stok[64 + t]) : 1.f, rqn = stok[128 + t];  // o = scale |q|^-1 (e^Gam Qh + O)
          float4* dst = reinterpret_cast<float4*>(f.o + ((T0 + t) * HVn + hv) * V + v0 + cb);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            float x[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              x[q] = f.scale * rqn *
                     (qs * (__uint_as_float(rq[4 * jj + q]) + __uint_as_float(rq2[4 * jj + q])) +
                      ((__uint_as_float(ro[4 * jj + q]) + __uint_as_float(ro3[4 * jj + q])) +
                       __uint_as_float(ro2[4 * jj + q])));
            dst[jj] = make_float4(x[0], x[1], x[2], x[3]);
          }
        }
      }
      if (quarter >= 2 && cgrp == 0 && j + 1 < nb)  // idle in the epilogue: next block's records
        ok = tok_records(j + 1, otid - 64, stok2 + 256 * ((j + 1) & 1)) && ok;
      tc_fence_before();
      ok = group_and(2, 256, ok);
      if (!ok) break;
      tc_fence_after();
      if (otid == 0) {
        mbar_arrive(&bars[FB_E0 + cs]);
        if (j + 2 < nb) load_og(j & 1, gk_base + (int64_t)(j + 2) * 128);
      }
    }
  }
  tmem_release(tmem, 512);
}

// ============================================================================ chunk_o
struct OArgs {
  int H, HV, V, M, l2norm;
  float scale;
  const float* g;
  const int4* seq_info;
  const int2* tok_tab;
  float* o;
  int* status;
};

// q (24 KB incl. view) | k (2 halves of 64M rows, 16M KB) | h hi, lo (16 KB each) |
// v_new hi, lo (8M KB each) | P hi, lo (MN-major: 64M rows e x 64 tokens t, 8M KB each) |
// gate prefixes [2][hi 128 | lo 128] | 1/|q| [2][64] | 1/|k| [64M] | barriers
constexpr int o_k_off() { return 24576; }
constexpr int o_h_off(int M) { return o_k_off() + 16384 * M; }
constexpr int o_v_off(int M) { return o_h_off(M) + 32768; }
constexpr int o_p_off(int M) { return o_v_off(M) + 16384 * M; }
constexpr int o_s_off(int M) { return o_p_off(M) + 2 * M * 8192; }
constexpr int o_smem(int M) { return o_s_off(M) + (2 * 256 + 2 * 64 + 64 * M) * 4 + 64 + 1024; }

template <int M>
__global__ void __launch_bounds__(512, 1) o_tc_kernel(
    const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
    const __grid_constant__ CUtensorMap map_hhi, const __grid_constant__ CUtensorMap map_hlo,
    const __grid_constant__ CUtensorMap map_vhi, const __grid_constant__ CUtensorMap map_vlo,
    OArgs a, int n_items) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  // Persistent: item = hv * (NT_max * nsl) + token chunk * nsl + value slice, so
  // the value slices of one chunk, which read the same q and k tiles, are
  // processed side by side by neighbouring CTAs. Two items overlap: TMEM holds
  // two column sets, one per item parity, and while the output warps wait for
  // item j's O product and store its output, the other warps wait for item
  // j + 1's q, k and h, issue its score and q h products and compute its row
  // norms. Each tile buffer is reloaded as soon as its last reader is done: q, k
  // and h once item j's score and q h products have completed, v once its O
  // product has.
  const int nsl = a.V / kOBV;
  const int per_hv = n_items / a.HV;  // NT_max * nsl
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, cq = warp >> 2;  // TMEM lane quarter, column quarter
  constexpr int NE = 64 * M;  // expanded positions in a full token chunk
  constexpr int NMMA = (NE + 127) / 128;  // score MMAs of 128 positions
  // TMEM columns of the set at base (0 or 256, by item parity): S^T [base, base +
  // 64 NMMA), then O = P_hi [v_hi | v_lo] [base, base + 128); q h = q h_hi + q h_lo
  // [base + 128, +64); P_lo v_hi [base + 192, +64). O is the sum of its three
  // 64-column parts.
  constexpr uint32_t TQH = 128, TOB = 192;
  uint8_t* qb = sm;
  uint8_t* kb = sm + o_k_off();
  uint8_t* hb = sm + o_h_off(M);
  uint8_t* vb = sm + o_v_off(M);
  uint8_t* pb = sm + o_p_off(M);
  // token gate prefixes, one buffer per item parity: hi [0, 64) and lo [128, 192)
  // (the second 64 of each half take comp_prefix128_warp's unused second scan)
  float* sgb = reinterpret_cast<float*>(sm + o_s_off(M));
  float* srq = sgb + 2 * 256;  // [2][64], by item parity
  float* srk = srq + 2 * 64;   // [64 M]
  // [0] q, k, h loaded, [1] v loaded, [2 + b] score and q h products of parity b,
  // [4 + b] O product of parity b (two issuers)
  uint64_t* bars = reinterpret_cast<uint64_t*>(srk + NE);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 6);
  constexpr uint32_t kCols = 512;

  // an item's geometry; tab.x < 0 marks a padding token chunk (no work)
  struct Item {
    int2 tab;
    int hv, kh, v0, nt, ne;
    int64_t T0, E0, hrow;
  };
  auto item = [&](int i) {
    Item x;
    x.hv = i / per_hv;
    const int rem = i - x.hv * per_hv, tc = rem / nsl;
    x.v0 = (rem - tc * nsl) * kOBV;
    x.kh = x.hv / (a.HV / a.H);
    x.tab = a.tok_tab[tc];
    x.nt = x.ne = 0;
    x.T0 = x.E0 = x.hrow = 0;
    if (x.tab.x >= 0) {
      const int4 si = a.seq_info[x.tab.x];
      const int t_start = x.tab.y * kBT;
      x.nt = min(kBT, si.y - t_start);
      x.ne = x.nt * M;
      x.T0 = (int64_t)si.x + t_start;
      x.E0 = x.T0 * M;
      x.hrow = (((int64_t)si.w + x.tab.y) * a.HV + x.hv) * kK;  // first of K rows
    }
    return x;
  };
  // the next item with work at or after i (n_items when none)
  auto next_live = [&](int i) {
    for (; i < n_items; i += gridDim.x)
      if (a.tok_tab[(i - (i / per_hv) * per_hv) / nsl].x >= 0) break;
    return i;
  };
  auto load_qkh = [&](const Item& x) {
    mbar_expect_tx(&bars[0], 2 * 8192 + 2 * NE * 128 + 4 * 8192);
    tma_load_3d(qb, &map_q, 0, x.kh, (int)x.T0, &bars[0]);
    tma_load_3d(qb + 8192, &map_q, 64, x.kh, (int)x.T0, &bars[0]);
    tma_load_3d(kb, &map_k, 0, x.kh, (int)x.E0, &bars[0]);
    tma_load_3d(kb + NE * 128, &map_k, 64, x.kh, (int)x.E0, &bars[0]);
    tma_load_2d(hb, &map_hhi, x.v0, (int)x.hrow, &bars[0]);
    tma_load_2d(hb + 16384, &map_hlo, x.v0, (int)x.hrow, &bars[0]);
  };
  auto load_v = [&](const Item& x) {
    mbar_expect_tx(&bars[1], 2 * NE * 128);
    tma_load_3d(vb, &map_vhi, x.v0, x.hv, (int)x.E0, &bars[1]);
    tma_load_3d(vb + NE * 128, &map_vlo, x.v0, x.hv, (int)x.E0, &bars[1]);
  };
  // An item's gates: warp 2 loads them (lanes 0-15, four tokens each) as soon
  // as the item is known and builds their compensated prefix while the output
  // warps run the previous item's epilogue.
  float gv[4];
  auto gate_load = [&](const Item& z) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * lane + i;
      gv[i] = (lane < 16 && t < z.nt && a.g) ? a.g[(z.T0 + t) * a.HV + z.hv] : 0.f;
    }
  };
  auto gate_prefix = [&](float* buf) {
    *reinterpret_cast<float4*>(buf + 4 * lane) = make_float4(gv[0], gv[1], gv[2], gv[3]);
    comp_prefix128_warp<true>(buf, buf + 128, lane);
  };
  // Score and q h products of the item in q, k, h into the column set at base:
  // S^T = k q^T, rows = positions, N = 64 tokens, one MMA per 128 positions into
  // columns [64 m, 64 m + 64) (rows past the chunk's 64 M positions read the
  // buffers behind k and feed accumulator rows that are never read); q h as
  // q h_hi then q h_lo into one accumulator (N = 64 each).
  auto issue_sq = [&](uint32_t tm, uint32_t base) {
    const uint32_t q0 = smem_u32(qb), k0 = smem_u32(kb), h0 = smem_u32(hb);
    const uint32_t ids = idesc_bf16(128, 64, false, false);
    const uint32_t idh = idesc_bf16(128, kOBV, false, true);
    const uint64_t qd = sdesc_sw128(q0, 16, 1024);
#pragma unroll
    for (int m = 0; m < NMMA; ++m)
      mma_run<8, false, NE * 128, 32, 8192, 32>(tm + base + 64 * m,
                                                sdesc_sw128(k0 + 16384 * m, 16, 1024), qd, ids);
    mma_run<8, false, 8192, 32, 8192, 2048>(tm + base + TQH, qd, sdesc_sw128(h0, 16384, 1024), idh);
    mma_run<8, true, 8192, 32, 8192, 2048>(tm + base + TQH, qd,
                                           sdesc_sw128(h0 + 16384, 16384, 1024), idh);
  };
  // Row norms of the staged q and k tiles (swizzle only permutes 16-byte
  // chunks), one row per thread of the 256 threads of lane quarters 2 and 3.
  auto norms = [&](float* rq) {
    const int gi = (warp >> 2) * 64 + (quarter - 2) * 32 + lane;
    if (gi < kBT) {
      const float ss = row_sumsq(qb + gi * 128, gi) + row_sumsq(qb + 8192 + gi * 128, gi);
      rq[gi] = a.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
    } else if (gi < kBT + NE) {
      const int e = gi - kBT;
      const float ss = row_sumsq(kb + e * 128, e) + row_sumsq(kb + NE * 128 + e * 128, e);
      srk[e] = a.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
    }
    fence_async_smem();  // the reads of q and k end before the next item's loads
  };
  static_assert(kBT + NE <= 256, "one norm row per thread of lane quarters 2 and 3");

  int it = next_live(blockIdx.x);
  if (it >= n_items) return;
  if (warp == 0) {
    tmem_alloc(s_tmem, kCols);
    tmem_relinquish();
  }
  Item x = item(it);
  if (warp == 2) {
    gate_load(x);
    gate_prefix(sgb);
  }
  if (tid == 0) {
    for (int i = 0; i < 6; ++i) mbar_init(&bars[i], i >= 4 ? 2 : 1);
    fence_mbar_init();
    load_qkh(x);
    load_v(x);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  int qkh_iss = 1, qkh_got = 0, v_iss = 1, v_got = 0;  // loads issued / consumed (thread 0's count)
  // the first item's products and norms
  bool ok = mbar_wait(&bars[0], 0, a.status, kDevTimeout);
  if (ok) {
    qkh_got = 1;
    if (tid == 64) {
      issue_sq(tmem, 0);
      mma_commit(&bars[2]);
    }
    if (quarter >= 2) norms(srq);
  }
  ok = __syncthreads_and(ok);
  for (int j = 0; ok; ++j) {
    const uint32_t b = j & 1, base = 256 * b, ph = (j >> 1) & 1;
    const int nx = next_live(it + gridDim.x);
    const bool has_next = nx < n_items;
    const Item y = has_next ? item(nx) : x;
    const float* sgh = sgb + b * 256;
    const float* sgl = sgh + 128;
    if (warp == 2 && has_next) gate_load(y);
    ok = mbar_wait(&bars[2 + b], ph, a.status, kDevTimeout);
    tc_fence_after();
    if (!__syncthreads_and(ok)) break;
    // the score and q h products and the norms have read q, k and h
    if (has_next && tid == 0) {
      load_qkh(y);
      ++qkh_iss;
    }
    {  // P^T rows e (positions), this warp's 16 of the 64 tokens: every warp builds rows
#pragma unroll
      for (int m = 0; m < NMMA; ++m) {
        if (128 * m + quarter * 32 < NE) {  // warp-uniform
          const int e = 128 * m + quarter * 32 + lane, s = e / M;
          uint32_t r[16];
          GDP_TMEM_LD16(tmem + ((uint32_t)(quarter * 32) << 16) + base + 64 * m + 16 * cq, r);
          tmem_wait_ld();
          const float rk = srk[e];
          __align__(16) bf16 ph_[16];
          __align__(16) bf16 pl_[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {  // branch-free, so that the iterations interleave
            const int t = 16 * cq + jj;
            const float v = __uint_as_float(r[jj]) * rk * __expf(gam_diff4(sgh, sgl, t, s));
            split_bf16((e < x.ne && s <= t && t < x.nt) ? v : 0.f, ph_[jj], pl_[jj]);
          }
          // MN-major operand: row e (K), 64 tokens (M) of 128 bytes; two 16-byte chunks
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint32_t off = (uint32_t)e * 128u + ((((uint32_t)(2 * cq + c)) ^ (e & 7u)) << 4);
            *reinterpret_cast<uint4*>(pb + off) = reinterpret_cast<const uint4*>(ph_)[c];
            *reinterpret_cast<uint4*>(pb + M * 8192 + off) = reinterpret_cast<const uint4*>(pl_)[c];
          }
        }
      }
    }
    ok = mbar_wait(&bars[1], v_got & 1, a.status, kDevTimeout);
    if (ok) ++v_got;
    // value rows past the chunk's end may hold anything: zero them (their P is 0)
    for (int idx = tid; idx < 2 * NE * 8; idx += 512) {
      const int row = idx >> 3, ch = idx & 7;
      const int e = row % NE;
      if (e >= x.ne) reinterpret_cast<uint4*>(vb + row * 128)[ch] = make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    tc_fence_before();
    if (!__syncthreads_and(ok)) break;
    tc_fence_after();
    if (tid == 0 || tid == 32) {  // O = P v_new, into the score columns (consumed)
      const uint32_t p0 = smem_u32(pb), vv = smem_u32(vb);
      // A = P, MN-major with M = 128: the second 64-token atom is never written and
      // LBO = 0 re-reads the first, which only feeds the unused accumulator rows
      if (tid == 0)  // P_hi [v_hi | v_lo], N = 128: the lo tile is the next 64-column group
        mma_run<4 * M, false, 8192, 2048, 8192, 2048>(tmem + base, sdesc_sw128(p0, 0, 1024),
                                                      sdesc_sw128(vv, NE * 128, 1024),
                                                      idesc_bf16(128, 2 * kOBV, true, true));
      else  // P_lo v_hi
        mma_run<4 * M, false, 8192, 2048, 8192, 2048>(tmem + base + TOB,
                                                      sdesc_sw128(p0 + M * 8192, 0, 1024),
                                                      sdesc_sw128(vv, NE * 128, 1024),
                                                      idesc_bf16(128, kOBV, true, true));
      mma_commit(&bars[4 + b]);
    }
    if (quarter < 2) {  // the output: wait for O, store o rows
      ok = mbar_wait(&bars[4 + b], ph, a.status, kDevTimeout);
      tc_fence_after();
      // the O product has read v (and P): the next item's v streams in
      if (ok && has_next && tid == 0) {
        load_v(y);
        ++v_iss;
      }
      const int t = quarter * 32 + lane;
      const float rq = srq[64 * b + t];
      const float qs = expf(sgh[t] + sgl[t]) * rq;  // o = scale |q|^-1 (e^Gam Qh + O)
      const uint32_t la = tmem + ((uint32_t)(quarter * 32) << 16) + base;
      const int c0 = cq * 16;
      uint32_t ro[16], rh[16], t16[16];
      GDP_TMEM_LD16(la + c0, ro);
      GDP_TMEM_LD16(la + TQH + c0, rh);
      tmem_wait_ld();
      GDP_TMEM_LD16(la + 64 + c0, t16);
      tmem_wait_ld();
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) ro[jj] = __float_as_uint(__uint_as_float(ro[jj]) + __uint_as_float(t16[jj]));
      GDP_TMEM_LD16(la + TOB + c0, t16);
      tmem_wait_ld();
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) ro[jj] = __float_as_uint(__uint_as_float(ro[jj]) + __uint_as_float(t16[jj]));
      if (t < x.nt && ok) {
        float4* dst = reinterpret_cast<float4*>(a.o + ((x.T0 + t) * a.HV + x.hv) * a.V + x.v0 + c0);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          float o4[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            o4[q] = a.scale * (qs * __uint_as_float(rh[4 * jj + q]) + rq * __uint_as_float(ro[4 * jj + q]));
          dst[jj] = make_float4(o4[0], o4[1], o4[2], o4[3]);
        }
      }
    } else if (has_next) {  // the next item: its products into the other column set, its norms
      ok = mbar_wait(&bars[0], qkh_got & 1, a.status, kDevTimeout);
      if (ok) {
        if (tid == 64) {
          tc_fence_after();
          issue_sq(tmem, 256 * (b ^ 1));
          mma_commit(&bars[2 + (b ^ 1)]);
        }
        norms(srq + 64 * (b ^ 1));
      }
      if (warp == 2) gate_prefix(sgb + (b ^ 1) * 256);
    }
    tc_fence_before();
    // TMEM set b, P, the gates and norms of parity b are free for item j + 2
    if (!__syncthreads_and(ok)) break;
    tc_fence_after();
    if (!has_next) break;
    ++qkh_got;
    it = nx;
    x = y;
  }
  if (tid == 0) {  // nothing may still write shared memory when the CTA leaves
    bool w = true;
    for (; w && qkh_got < qkh_iss; ++qkh_got) w = mbar_wait(&bars[0], qkh_got & 1, nullptr, 0);
    for (; w && v_got < v_iss; ++v_got) w = mbar_wait(&bars[1], v_got & 1, nullptr, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  tmem_release(tmem, kCols);
}

// ============================================================================ host
// Test hook state (gdp_debug_wait_fault): armed for the next WY-128 launch only.
std::atomic<int> g_wy_fault{0};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Row-major [rows][heads][width] tensor; box = box_w elements x 1 head x box_rows rows.
bool map3(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint32_t esz, uint64_t width,
          uint64_t heads, uint64_t rows, uint32_t box_w, uint32_t box_rows, bool swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {width, heads, rows};
  const cuuint64_t strides[2] = {width * esz, heads * width * esz};
  const cuuint32_t box[3] = {box_w, 1, box_rows};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major [rows][width]; box = box_w x box_rows.
bool map2(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint32_t esz, uint64_t width,
          uint64_t rows, uint32_t box_w, uint32_t box_rows, bool swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {width, rows};
  const cuuint64_t strides[1] = {width * esz};
  const cuuint32_t box[2] = {box_w, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
constexpr CUtensorMapDataType F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;


template <int V, bool G, bool C64>
cudaError_t run_wy128(const ChunkProblem& p, const WyArgs& a) {
  const int64_t Te = (int64_t)p.B * p.T * p.M;
  CUtensorMap mk, mv, mwh, mwl, mu;
  if (!map3(&mk, p.k, BF, 2, kK, p.H, Te, 64, 128, true)) return cudaErrorInvalidValue;
  if (!map3(&mv, p.v, BF, 2, V, p.HV, Te, 64, 128, true)) return cudaErrorInvalidValue;
  if (!map3(&mwh, a.w_hi, BF, 2, kK, p.HV, Te, 64, 128, true) ||
      !map3(&mwl, a.w_lo, BF, 2, kK, p.HV, Te, 64, 128, true) ||
      !map3(&mu, a.u, F32, 4, V, p.HV, Te, 32, 128, true))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(wy128_tc_kernel<V, G, C64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, W8_SMEM);
  if (e != cudaSuccess) return e;
  const int64_t NB = block128_bound(p.B, p.T, p.N_seq, p.M);
  const int64_t items = NB * p.HV;
  if (items > INT32_MAX) return cudaErrorInvalidValue;
  const int grid = (int)std::min<int64_t>(items, sm_count());  // persistent, one CTA per SM
  return launch_pdl(wy128_tc_kernel<V, G, C64>, dim3(grid), dim3(512), W8_SMEM, p.stream, mk, mv, mwh,
                    mwl, mu, a, (int)NB);
}

template <int M>
cudaError_t run_o(const ChunkProblem& p, const OArgs& a, const CUtensorMap& mhhi,
                  const CUtensorMap& mhlo, const CUtensorMap& mvhi, const CUtensorMap& mvlo) {
  const int64_t Tt = (int64_t)p.B * p.T, Te = Tt * M;
  CUtensorMap mq, mk;
  if (!map3(&mq, p.q, BF, 2, kK, p.H, Tt, 64, 64, true)) return cudaErrorInvalidValue;
  if (!map3(&mk, p.k, BF, 2, kK, p.H, Te, 64, 64 * M, true)) return cudaErrorInvalidValue;
  const int smem = o_smem(M);
  cudaError_t e = cudaFuncSetAttribute(o_tc_kernel<M>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t items = p.NT_max * (p.V / kOBV) * p.HV;
  if (items > INT32_MAX) return cudaErrorInvalidValue;
  const int grid = (int)std::min<int64_t>(items, sm_count());  // persistent, one CTA per SM
  return launch_pdl(o_tc_kernel<M>, dim3(grid), dim3(512), smem, p.stream, mq, mk, mhhi, mhlo, mvhi,
                    mvlo, a, (int)items);
}

}  // namespace

bool tc_supported(int H, int HV, int K, int V, int M, int BT, gdp_dtype dt) {
  (void)H;
  (void)HV;
  return dt == GDP_BF16 && K == kK && BT == kBT && (V == 64 || V == 128 || V == 256) && M >= 1 &&
         M <= 3;
}

WsLayout tc_layout(int B, int T, int N_seq, int H, int HV, int K, int V, int M, int BT) {
  (void)H;
  WsLayout L;
  int64_t NE, NT;
  chunk_bounds(B, T, N_seq, M, BT, &NE, &NT);
  const size_t Te = (size_t)B * T * M;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t at = off; off = align_up(off + bytes); return at; };
  L.status = take(kAlign);
  L.seq_info = take(sizeof(int4) * (size_t)(N_seq > 0 ? N_seq : 1));
  L.exp_tab = take(sizeof(int2) * (size_t)NE);
  L.tok_tab = take(sizeof(int2) * (size_t)NT);
  // 128-position blocks: WY-128 for every M (odd M in its two-chunk form)
  L.blk_tab = take(sizeof(int4) * (size_t)block128_bound(B, T, N_seq, M));
  L.w_hi = take(2 * Te * HV * K);
  L.w_lo = take(2 * Te * HV * K);
  L.u = take(4 * Te * HV * V);
  L.gam = take(16 * Te * HV);
  // v_new and the chunk states go through HBM only when the output is a
  // separate kernel (M != 2)
  const size_t keep = M == 2 ? 0 : 1;
  L.vn_hi = take(keep * 2 * Te * HV * V);
  L.vn_lo = take(keep * 2 * Te * HV * V);
  L.h_hi = take(keep * 2 * (size_t)NT * HV * V * K);
  L.h_lo = take(keep * 2 * (size_t)NT * HV * V * K);
  L.seq_order = take(sizeof(int32_t) * (size_t)(N_seq > 0 ? N_seq : 1));
  L.total = off;
  L.path = 1;
  return L;
}

cudaError_t launch_chunk_tc(const ChunkProblem& p, const WsLayout& L, uint8_t* ws) {
  const int64_t Te = (int64_t)p.B * p.T * p.M;
  int* status = reinterpret_cast<int*>(ws + L.status);
  const int4* seq_info = reinterpret_cast<const int4*>(ws + L.seq_info);
  bf16* w_hi = reinterpret_cast<bf16*>(ws + L.w_hi);
  bf16* w_lo = reinterpret_cast<bf16*>(ws + L.w_lo);
  float* u = reinterpret_cast<float*>(ws + L.u);
  float4* gk = reinterpret_cast<float4*>(ws + L.gam);
  bf16* vn_hi = reinterpret_cast<bf16*>(ws + L.vn_hi);
  bf16* vn_lo = reinterpret_cast<bf16*>(ws + L.vn_lo);
  bf16* h_hi = reinterpret_cast<bf16*>(ws + L.h_hi);
  bf16* h_lo = reinterpret_cast<bf16*>(ws + L.h_lo);
  cudaError_t e;
  // WY stage
  if (p.NE_max > 0 && Te > 0) {
    WyArgs a{p.H, p.HV, p.V, p.M, p.l2norm, Te, p.beta, p.g, seq_info,
             reinterpret_cast<const int4*>(ws + L.blk_tab), w_hi, w_lo, u, gk, status, 0};
    if ((p.M % 2) == 0) a.fault = g_wy_fault.exchange(0);  // one-shot test hook
    // even M: 128-position blocks; odd M: the same kernel on pairs of 64-position
    // chunks (the state recurrence steps 64 positions)
    const bool c64 = (p.M % 2) != 0;
    const bool G = p.g != nullptr;
    switch (p.V) {
      case 64:
        e = c64 ? (G ? run_wy128<64, true, true>(p, a) : run_wy128<64, false, true>(p, a))
                : (G ? run_wy128<64, true, false>(p, a) : run_wy128<64, false, false>(p, a));
        break;
      case 128:
        e = c64 ? (G ? run_wy128<128, true, true>(p, a) : run_wy128<128, false, true>(p, a))
                : (G ? run_wy128<128, true, false>(p, a) : run_wy128<128, false, false>(p, a));
        break;
      default:
        e = c64 ? (G ? run_wy128<256, true, true>(p, a) : run_wy128<256, false, true>(p, a))
                : (G ? run_wy128<256, true, false>(p, a) : run_wy128<256, false, false>(p, a));
        break;
    }
    if (e != cudaSuccess) return e;
  }
  record_stage(2, p.stream);
  // state recurrence: 128-position steps for even M, 64-position steps otherwise
  {
    const uint32_t rows = p.M == 2 ? 128 : 64;  // M = 2: 128-position steps
    CUtensorMap mwh, mwl, mk, mu, mg;
    const int64_t Tr = Te > 0 ? Te : 1;
    if (!map3(&mwh, w_hi, BF, 2, kK, p.HV, Tr, 64, rows, true) ||
        !map3(&mwl, w_lo, BF, 2, kK, p.HV, Tr, 64, rows, true) ||
        !map3(&mk, p.k ? p.k : w_hi, BF, 2, kK, p.H, Tr, 64, rows, true) ||
        !map3(&mu, u, F32, 4, p.V, p.HV, Tr, kHBV, rows, true) ||
        !map2(&mg, gk, F32, 4, 4, (uint64_t)p.HV * Tr, 4, rows, false))
      return cudaErrorInvalidValue;
    // ragged sequences: chains in the tables kernel's longest-first order
    const int* order = p.cu_seqlens ? reinterpret_cast<const int*>(ws + L.seq_order) : nullptr;
    HArgs a{p.HV, p.V, p.M, Te, seq_info, u, gk, p.h0, p.hT, vn_hi, vn_lo, h_hi, h_lo, status};
    const dim3 grid((unsigned)((int64_t)p.N_seq * (p.V / kHBV)), p.HV);
    if (p.M == 2) {  // state recurrence and output fused
      CUtensorMap mq;
      const int64_t Tt = (int64_t)p.B * p.T;
      if (!map3(&mq, p.q ? p.q : w_hi, BF, 2, kK, p.H, Tt > 0 ? Tt : 1, 64, 64, true))
        return cudaErrorInvalidValue;
      HOArgs fa{a, p.H, p.l2norm, p.scale, p.o};
      auto kern = p.g ? (order ? ho128_tc_kernel<true, true> : ho128_tc_kernel<true, false>)
                      : (order ? ho128_tc_kernel<false, true> : ho128_tc_kernel<false, false>);
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F_SMEM);
      if (e != cudaSuccess) return e;
      if ((e = launch_pdl(kern, grid, dim3(512), F_SMEM, p.stream, mwh, mwl, mk, mu, mg, mq, fa,
                          order)) !=
          cudaSuccess)
        return e;
      record_stage(3, p.stream);
      record_stage(4, p.stream);
      return cudaSuccess;
    }
    // odd M: 64-position steps (the WY factors are the 64-position chunks')
    e = cudaFuncSetAttribute(h_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, H_SMEM);
    if (e != cudaSuccess) return e;
    e = launch_pdl(h_tc_kernel, grid, dim3(256), H_SMEM, p.stream, mwh, mwl, mk, mu, mg, a, p.H,
                   order);
    if (e != cudaSuccess) return e;
  }
  record_stage(3, p.stream);
  // output
  if (p.NT_max > 0 && Te > 0) {
    CUtensorMap mhh, mhl, mvh, mvl;
    const uint64_t hrows = (uint64_t)p.NT_max * p.HV * kK;
    if (!map2(&mhh, h_hi, BF, 2, p.V, hrows, kOBV, kK, true) ||
        !map2(&mhl, h_lo, BF, 2, p.V, hrows, kOBV, kK, true) ||
        !map3(&mvh, vn_hi, BF, 2, p.V, p.HV, Te, 64, 64 * p.M, true) ||
        !map3(&mvl, vn_lo, BF, 2, p.V, p.HV, Te, 64, 64 * p.M, true))
      return cudaErrorInvalidValue;
    OArgs a{p.H, p.HV, p.V, p.M, p.l2norm, p.scale, p.g, seq_info,
            reinterpret_cast<const int2*>(ws + L.tok_tab), p.o, status};
    switch (p.M) {
      case 1: e = run_o<1>(p, a, mhh, mhl, mvh, mvl); break;
      case 2: e = run_o<2>(p, a, mhh, mhl, mvh, mvl); break;
      default: e = run_o<3>(p, a, mhh, mhl, mvh, mvl); break;
    }
    if (e != cudaSuccess) return e;
  }
  record_stage(4, p.stream);
  return cudaSuccess;
}

}  // namespace gdp

extern "C" gdp_status gdp_debug_wait_fault(int arm, double budget_seconds) {
  unsigned long long ns = gdp::ptx::kWaitBudgetNs;
  if (budget_seconds > 0.0) {
    if (budget_seconds > 10.0) return GDP_ERR_INVALID_ARG;
    ns = (unsigned long long)(budget_seconds * 1e9);
    if (ns == 0) ns = 1;
  }
  if (cudaMemcpyToSymbol(gdp::ptx::g_wait_budget_ns, &ns, sizeof(ns)) != cudaSuccess)
    return GDP_ERR_CUDA;
  gdp::g_wy_fault.store(arm ? 1 : 0);
  return GDP_OK;
}
