// Generic chunked Gated Delta Product forward: fp32 arithmetic on CUDA cores,
// any input dtype (bf16/fp16/fp32), any K <= 256, V <= 1024, chunk 16/32/64.
// Used for fp32/fp16 inputs and for shapes outside the tensor-core path, and
// keeps every intermediate stage in the workspace for stage-by-stage checks.
//
// Stages (Megatron-core API pages "core.ssm.ops.gdp.wy_fast" and
// "core.ssm.ops.gdp.chunk_o"; the chunk algebra is the WY form of the gated
// delta rule over the Householder-expanded stream, copy j of token t at t*M+j):
//   tables   device-built chunk descriptors from cu_seqlens (no host sync)
//   wy       per expanded chunk of BT positions: Gam = inclusive cumsum of the
//            per-position log decay (g_t on a token's first copy, 0 on the
//            others), kept as a compensated two-float sum,
//            L[p,i] = beta_p e^(Gam_p-Gam_i) k_p.k_i (i<p), A = (I+L)^-1
//            (solve_tril, forward substitution), w = A(beta e^Gam k),
//            u = A(beta v)  (recompute_w_u)
//   chunk_h  per (sequence, value head, value slice), sequential over chunks:
//            v_new = u - w h ; h <- e^Gam_last h + (k e^(Gam_last-Gam))^T v_new;
//            the state at each token-chunk start is stored for chunk_o
//   chunk_o  per token chunk of BT tokens: o_t = scale (e^Gt_t q_t.h_c +
//            sum_{s<=t} sum_j e^(Gt_t-Gt_s) (q_t.k_{s,j}) v_new_{s,j}), the
//            token chunk c starting at expanded chunk c*M.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gdp_internal.cuh"

namespace gdp {
namespace {

// Inclusive prefix sum of the per-position log decays, compensated (Neumaier):
// hi[p] + lo[p] carries the sum to about twice fp32 precision, so that the
// difference of two prefixes, (hi[p]-hi[i]) + (lo[p]-lo[i]), stays accurate
// even when the prefixes themselves are large (strong decay over a chunk).
__device__ __forceinline__ void comp_prefix(float* hi, float* lo, int n) {
  float s = 0.f, c = 0.f;
  for (int p = 0; p < n; ++p) {
    const float x = hi[p];
    const float t = s + x;
    c += (fabsf(s) >= fabsf(x)) ? ((s - t) + x) : ((x - t) + s);
    s = t;
    hi[p] = s;
    lo[p] = c;
  }
}
__device__ __forceinline__ float gam_diff(const float* hi, const float* lo, int p, int i) {
  return (hi[p] - hi[i]) + (lo[p] - lo[i]);
}

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float ldf(const __half* p) { return __half2float(*p); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ------------------------------------------------------------------------------------
// chunk tables
// ------------------------------------------------------------------------------------
// One CTA of kTabThreads threads. A dense batch (no offsets) has every entry in
// closed form and fills the tables directly. With offsets, the sequences are
// taken kTabThreads at a time:
// each thread loads its sequence's offsets, checks them and counts its chunks,
// and a block-wide scan turns the counts into the sequence's first chunk
// indices (no thread walks the list alone). Records and chunk counts of the
// first kTabSmem sequences stay in shared memory for the table fill, so the
// fill takes no division (chunk sizes are powers of two: counts are shifts).
constexpr int kTabThreads = 512;
constexpr int kTabSmem = 1024;

// Exclusive block-wide scan of three counts (all threads of the block call it);
// returns the block's totals in tot.
__device__ __forceinline__ void scan3(int64_t (&x)[3], int64_t (&tot)[3], int64_t* sw) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = kTabThreads / 32;
  int64_t inc[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    inc[j] = x[j];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, inc[j], o);
      if (lane >= o) inc[j] += y;
    }
  }
  if (lane == 31)
#pragma unroll
    for (int j = 0; j < 3; ++j) sw[warp * 3 + j] = inc[j];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      int64_t w = lane < NW ? sw[lane * 3 + j] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < NW) sw[lane * 3 + j] = w;  // inclusive warp prefix
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int64_t before = warp > 0 ? sw[(warp - 1) * 3 + j] : 0;
    x[j] = before + inc[j] - x[j];
    tot[j] = sw[(NW - 1) * 3 + j];
  }
  __syncthreads();  // sw is reused by the next call
}

__global__ void __launch_bounds__(kTabThreads) tables_kernel(
    const int32_t* cu, int N_seq, int B, int T, int M, int BT, int64_t NE_max, int64_t NT_max,
    int4* seq_info, int2* exp_tab, int2* tok_tab, int4* blk_tab, int64_t NB_max, int* status,
    int* seq_order) {
  pdl_wait();
  const int sh = __ffs(BT) - 1;  // BT = 2^sh
  if (!cu) {  // dense batch: B sequences of T tokens, every table entry in closed form
    const int tid = threadIdx.x;
    const int ne = (int)((((int64_t)T * M) + BT - 1) >> sh), nt = (T + BT - 1) >> sh;
    const int nb = (int)((((int64_t)T * M) + 127) >> 7);
    if (tid == 0) *status = kDevOk;
    for (int i = tid; i < B; i += kTabThreads) seq_info[i] = make_int4(i * T, T, i * ne, i * nt);
    for (int64_t c = tid; c < NE_max; c += kTabThreads)
      exp_tab[c] = c < (int64_t)B * ne ? make_int2((int)(c / ne), (int)(c % ne)) : make_int2(-1, 0);
    for (int64_t c = tid; c < NT_max; c += kTabThreads)
      tok_tab[c] = c < (int64_t)B * nt ? make_int2((int)(c / nt), (int)(c % nt)) : make_int2(-1, 0);
    if (blk_tab)
      for (int64_t c = tid; c < NB_max; c += kTabThreads) {
        const int i = nb > 0 ? (int)(c / nb) : 0;
        blk_tab[c] = c < (int64_t)B * nb ? make_int4(i, (int)(2 * (c - (int64_t)i * nb)), i * T, T)
                                         : make_int4(-1, 0, 0, 0);
      }
    if (seq_order)
      for (int i = tid; i < B; i += kTabThreads) seq_order[i] = i;
    return;
  }
  __shared__ int4 s_info[kTabSmem];     // (first token, length, first exp chunk, first token chunk)
  __shared__ int4 s_cnt[kTabSmem];      // (exp chunks, token chunks, 128-position blocks, first block)
  __shared__ int64_t s_scan[3 * (kTabThreads / 32)];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  int64_t carry[3] = {0, 0, 0};  // expanded chunks, token chunks, 128-position blocks so far
  for (int base = 0; base < N_seq; base += kTabThreads) {
    const int i = base + tid;
    int t0 = 0, len = 0;
    bool bad = false;
    if (i < N_seq) {
      t0 = cu[i];
      const int t1 = cu[i + 1];
      // cu[0] = 0, non-decreasing, within B*T: each sequence checks its own pair
      bad = (i == 0 && t0 != 0) || t1 < t0 || (int64_t)t1 > (int64_t)B * T;
      len = t1 - t0;
    }
    if (bad) s_bad = 1;
    int64_t cnt[3] = {0, 0, 0}, tot[3];
    int c3[3] = {0, 0, 0};
    if (i < N_seq && !bad) {
      c3[0] = (int)((((int64_t)len * M) + BT - 1) >> sh);
      c3[1] = (int)((((int64_t)len) + BT - 1) >> sh);
      c3[2] = (int)((((int64_t)len * M) + 127) >> 7);
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) cnt[j] = c3[j];
    scan3(cnt, tot, s_scan);
    if (i < N_seq) {
      const int4 rec = make_int4(t0, len, (int)(carry[0] + cnt[0]), (int)(carry[1] + cnt[1]));
      seq_info[i] = rec;
      if (i < kTabSmem) {
        s_info[i] = rec;
        s_cnt[i] = make_int4(c3[0], c3[1], c3[2], (int)(carry[2] + cnt[2]));
      }
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) carry[j] += tot[j];
  }
  __syncthreads();
  const bool bad = s_bad || carry[0] > NE_max || carry[1] > NT_max;
  if (tid == 0) *status = bad ? kDevBadSeqlens : kDevOk;  // the call's status word starts here
  // A bad list leaves every sequence with a zero-length record: the state
  // kernels, which launch one CTA row per sequence, then read no input rows,
  // write no output rows and only pass the initial state through.
  if (bad)
    for (int i = tid; i < N_seq; i += kTabThreads) seq_info[i] = make_int4(0, 0, 0, 0);
  if (seq_order) {
    // Launch order of the state-scan chains: sequences by length, longest first
    // (equal lengths by index), so that the CTAs that start last run the shortest
    // chains; the identity when the records do not all fit in shared memory
    const bool sort = !bad && N_seq <= kTabSmem;
    for (int i = tid; i < N_seq; i += kTabThreads) {
      int r = i;
      if (sort) {
        const int li = s_info[i].y;
        r = 0;
        for (int j = 0; j < N_seq; ++j) {
          const int lj = s_info[j].y;
          r += (lj > li) | (lj == li & j < i);
        }
      }
      seq_order[r] = i;
    }
  }
  const int64_t ne = bad ? 0 : carry[0], nt = bad ? 0 : carry[1], nb = bad ? 0 : carry[2];
  if (!bad) {
    // one warp per sequence over the shared records, lanes over its chunks
    const int warp = tid >> 5, lane = tid & 31;
    const int ns = N_seq < kTabSmem ? N_seq : kTabSmem;
    for (int i = warp; i < ns; i += kTabThreads / 32) {
      const int4 si = s_info[i], cn = s_cnt[i];
      for (int c = lane; c < cn.x; c += 32) exp_tab[si.z + c] = make_int2(i, c);
      for (int c = lane; c < cn.y; c += 32) tok_tab[si.w + c] = make_int2(i, c);
      if (blk_tab)
        // 128-position blocks: (sequence, index of the block's first 64-chunk, the
        // sequence's first token, its length), so that a block's reader needs one load
        for (int c = lane; c < cn.z; c += 32) blk_tab[cn.w + c] = make_int4(i, 2 * c, si.x, si.y);
    }
    // sequences past the shared records: all threads, one sequence at a time
    int64_t b_run = ns > 0 ? (int64_t)s_cnt[ns - 1].w + s_cnt[ns - 1].z : 0;
    for (int i = kTabSmem; i < N_seq; ++i) {
      const int4 si = seq_info[i];
      const int nei = (int)((((int64_t)si.y * M) + BT - 1) >> sh);
      const int nti = (int)((((int64_t)si.y) + BT - 1) >> sh);
      const int nbi = (int)((((int64_t)si.y * M) + 127) >> 7);
      for (int c = tid; c < nei; c += kTabThreads) exp_tab[si.z + c] = make_int2(i, c);
      for (int c = tid; c < nti; c += kTabThreads) tok_tab[si.w + c] = make_int2(i, c);
      if (blk_tab)
        for (int c = tid; c < nbi; c += kTabThreads)
          blk_tab[b_run + c] = make_int4(i, 2 * c, si.x, si.y);
      b_run += nbi;
    }
  }
  for (int64_t c = ne + tid; c < NE_max; c += kTabThreads) exp_tab[c] = make_int2(-1, 0);
  for (int64_t c = nt + tid; c < NT_max; c += kTabThreads) tok_tab[c] = make_int2(-1, 0);
  if (blk_tab)
    for (int64_t c = nb + tid; c < NB_max; c += kTabThreads) blk_tab[c] = make_int4(-1, 0, 0, 0);
}

// ------------------------------------------------------------------------------------
// wy: transition block, solve_tril, w and u for one expanded chunk and value head
// ------------------------------------------------------------------------------------
struct GenArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* beta;
  const float* g;
  const float* h0;
  float* o;
  float* hT;
  int N_seq, H, HV, K, V, M, BT, l2norm;
  float scale;
  const int4* seq_info;
  const int2* exp_tab;
  const int2* tok_tab;
  float* A;
  float* w;
  float* u;
  float* gexp;
  float* v_new;
  float* h;
};

template <typename Tin>
__global__ void __launch_bounds__(256) wy_generic_kernel(GenArgs a) {
  extern __shared__ float sm[];
  const int2 tab = a.exp_tab[blockIdx.x];
  if (tab.x < 0) return;
  const int hv = blockIdx.y, kh = hv / (a.HV / a.H);
  const int4 si = a.seq_info[tab.x];
  const int BT = a.BT, K = a.K, V = a.V, M = a.M;
  const int e_start = tab.y * BT;
  const int n = min(BT, si.y * M - e_start);
  const int64_t R0 = (int64_t)si.x * M + e_start;  // first global expanded row
  const int KP = K + 1, BP = BT + 1;
  float* ks = sm;                 // [BT][KP]
  float* Ls = ks + BT * KP;       // [BT][BP]
  float* As = Ls + BT * BP;       // [BT][BP]
  float* sb = As + BT * BP;       // beta
  float* sG = sb + BT;            // Gam, compensated prefix: high part
  float* sGl = sG + BT;           //                            low part
  float* srk = sGl + BT;          // 1/|k| or 1
  const Tin* kin = static_cast<const Tin*>(a.k);
  const Tin* vin = static_cast<const Tin*>(a.v);
  const int tid = threadIdx.x, nth = blockDim.x;

  for (int p = tid; p < BT; p += nth) {
    float b = 0.f, gl = 0.f;
    if (p < n) {
      const int e = e_start + p, t = e / M, jj = e - t * M;
      b = a.beta[(R0 + p) * a.HV + hv];
      if (a.g && jj == 0) gl = a.g[((int64_t)si.x + t) * a.HV + hv];
    }
    sb[p] = b;
    sG[p] = gl;
  }
  for (int i = tid; i < BT * K; i += nth) {
    const int p = i / K, c = i - p * K;
    ks[p * KP + c] = p < n ? ldf(kin + ((R0 + p) * a.H + kh) * K + c) : 0.f;
  }
  __syncthreads();
  if (tid == 0) comp_prefix(sG, sGl, BT);
  {
    const int wid = tid >> 5, lane = tid & 31, nw = nth >> 5;
    for (int p = wid; p < BT; p += nw) {
      float ss = 0.f;
      for (int c = lane; c < K; c += 32) ss += ks[p * KP + c] * ks[p * KP + c];
      ss = warp_sum(ss);
      if (lane == 0) srk[p] = a.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
    }
  }
  __syncthreads();
  // strictly-lower transition block
  for (int i2 = tid; i2 < BT * BT; i2 += nth) {
    const int p = i2 / BT, i = i2 - p * BT;
    float val = 0.f;
    if (i < p && p < n) {
      float d = 0.f;
      for (int c = 0; c < K; ++c) d += ks[p * KP + c] * ks[i * KP + c];
      val = sb[p] * expf(gam_diff(sG, sGl, p, i)) * srk[p] * srk[i] * d;
    }
    Ls[p * BP + i] = val;
    As[p * BP + i] = (p == i) ? 1.f : 0.f;
  }
  __syncthreads();
  // solve_tril: rows of A = (I + L)^-1 by forward substitution
  for (int p = 1; p < n; ++p) {
    for (int c = tid; c < p; c += nth) {
      float s = 0.f;
      for (int i = c; i < p; ++i) s += Ls[p * BP + i] * As[i * BP + c];
      As[p * BP + c] = -s;
    }
    __syncthreads();
  }
  for (int i2 = tid; i2 < n * BT; i2 += nth) {
    const int p = i2 / BT, c = i2 - p * BT;
    a.A[((R0 + p) * a.HV + hv) * BT + c] = As[p * BP + c];
  }
  // w = A (beta 2^Gam k / |k|)
  for (int i2 = tid; i2 < n * K; i2 += nth) {
    const int p = i2 / K, c = i2 - p * K;
    float s = 0.f;
    for (int i = 0; i <= p; ++i)
      s += As[p * BP + i] * (sb[i] * expf(sG[i] + sGl[i]) * srk[i]) * ks[i * KP + c];
    a.w[((R0 + p) * a.HV + hv) * K + c] = s;
  }
  // u = A (beta v)
  for (int i2 = tid; i2 < n * V; i2 += nth) {
    const int p = i2 / V, c = i2 - p * V;
    float s = 0.f;
    for (int i = 0; i <= p; ++i)
      s += As[p * BP + i] * sb[i] * ldf(vin + ((R0 + i) * a.HV + hv) * V + c);
    a.u[((R0 + p) * a.HV + hv) * V + c] = s;
  }
  for (int p = tid; p < n; p += nth) {
    a.gexp[2 * ((R0 + p) * a.HV + hv)] = sG[p];
    a.gexp[2 * ((R0 + p) * a.HV + hv) + 1] = sGl[p];
  }
}

// ------------------------------------------------------------------------------------
// chunk_h: sequential state recurrence over the expanded chunks of one sequence
// ------------------------------------------------------------------------------------
constexpr int kBVH = 32;

template <typename Tin>
__global__ void __launch_bounds__(256) h_generic_kernel(GenArgs a) {
  extern __shared__ float sm[];
  const int seq = blockIdx.x, hv = blockIdx.y, kh = hv / (a.HV / a.H);
  const int v0 = blockIdx.z * kBVH;
  const int nv = min(kBVH, a.V - v0);
  const int4 si = a.seq_info[seq];
  const int BT = a.BT, K = a.K, V = a.V, M = a.M;
  const int KP = K + 1;
  float* hs = sm;                 // [K][kBVH]
  float* ws = hs + K * kBVH;      // [BT][KP]
  float* ks = ws + BT * KP;       // [BT][KP]
  float* us = ks + BT * KP;       // [BT][kBVH]
  float* vn = us + BT * kBVH;     // [BT][kBVH]
  float* sG = vn + BT * kBVH;     // [BT] Gam high part
  float* sGl = sG + BT;           // [BT] Gam low part
  float* srk = sGl + BT;          // [BT]
  const Tin* kin = static_cast<const Tin*>(a.k);
  const int tid = threadIdx.x, nth = blockDim.x;
  const int64_t hoff = ((int64_t)seq * a.HV + hv) * K * V;

  for (int i = tid; i < K * kBVH; i += nth) {
    const int r = i / kBVH, c = i - r * kBVH;
    hs[i] = (a.h0 && c < nv) ? a.h0[hoff + (int64_t)r * V + v0 + c] : 0.f;
  }
  const int ne = (int)cdiv((int64_t)si.y * M, BT);
  for (int jc = 0; jc < ne; ++jc) {
    __syncthreads();
    if (jc % M == 0) {
      float* hb = a.h + (((int64_t)si.w + jc / M) * a.HV + hv) * K * V;
      for (int i = tid; i < K * nv; i += nth) {
        const int r = i / nv, c = i - r * nv;
        hb[(int64_t)r * V + v0 + c] = hs[r * kBVH + c];
      }
    }
    const int e_start = jc * BT;
    const int n = min(BT, si.y * M - e_start);
    const int64_t R0 = (int64_t)si.x * M + e_start;
    for (int i = tid; i < BT * K; i += nth) {
      const int p = i / K, c = i - p * K;
      const bool ok = p < n;
      ws[p * KP + c] = ok ? a.w[((R0 + p) * a.HV + hv) * K + c] : 0.f;
      ks[p * KP + c] = ok ? ldf(kin + ((R0 + p) * a.H + kh) * K + c) : 0.f;
    }
    for (int i = tid; i < BT * kBVH; i += nth) {
      const int p = i / kBVH, c = i - p * kBVH;
      us[i] = (p < n && c < nv) ? a.u[((R0 + p) * a.HV + hv) * V + v0 + c] : 0.f;
    }
    for (int p = tid; p < BT; p += nth) {
      sG[p] = p < n ? a.gexp[2 * ((R0 + p) * a.HV + hv)] : 0.f;
      sGl[p] = p < n ? a.gexp[2 * ((R0 + p) * a.HV + hv) + 1] : 0.f;
    }
    __syncthreads();
    {
      const int wid = tid >> 5, lane = tid & 31, nw = nth >> 5;
      for (int p = wid; p < BT; p += nw) {
        float ss = 0.f;
        for (int c = lane; c < K; c += 32) ss += ks[p * KP + c] * ks[p * KP + c];
        ss = warp_sum(ss);
        if (lane == 0) srk[p] = a.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
      }
    }
    // v_new = u - w h
    for (int i = tid; i < BT * kBVH; i += nth) {
      const int p = i / kBVH, c = i - p * kBVH;
      float s = 0.f;
      for (int r = 0; r < K; ++r) s += ws[p * KP + r] * hs[r * kBVH + c];
      const float val = (p < n) ? us[i] - s : 0.f;
      vn[i] = val;
      if (p < n && c < nv) a.v_new[((R0 + p) * a.HV + hv) * V + v0 + c] = val;
    }
    __syncthreads();
    const float dlast = expf(sG[n - 1] + sGl[n - 1]);
    // h <- e^Gam_last h + (k e^(Gam_last - Gam) / |k|)^T v_new
    for (int i = tid; i < K * kBVH; i += nth) {
      const int r = i / kBVH, c = i - r * kBVH;
      float s = 0.f;
      for (int p = 0; p < n; ++p)
        s += ks[p * KP + r] * srk[p] * expf(gam_diff(sG, sGl, n - 1, p)) * vn[p * kBVH + c];
      hs[i] = dlast * hs[i] + s;
    }
  }
  __syncthreads();
  if (a.hT) {
    for (int i = tid; i < K * nv; i += nth) {
      const int r = i / nv, c = i - r * nv;
      a.hT[hoff + (int64_t)r * V + v0 + c] = hs[r * kBVH + c];
    }
  }
}

// ------------------------------------------------------------------------------------
// chunk_o: output of one token chunk, one value head, one value slice
// ------------------------------------------------------------------------------------
constexpr int kBVO = 64, kKT = 32, kEB = 64;

template <typename Tin>
__global__ void __launch_bounds__(256) o_generic_kernel(GenArgs a) {
  extern __shared__ float sm[];
  const int2 tab = a.tok_tab[blockIdx.x];
  if (tab.x < 0) return;
  const int hv = blockIdx.y, kh = hv / (a.HV / a.H);
  const int v0 = blockIdx.z * kBVO;
  const int nv = min(kBVO, a.V - v0);
  const int4 si = a.seq_info[tab.x];
  const int BT = a.BT, K = a.K, V = a.V, M = a.M;
  const int t_start = tab.y * BT;
  const int nt = min(BT, si.y - t_start);
  const int ne = nt * M;
  const int64_t T0 = (int64_t)si.x + t_start;  // first global token
  const int64_t E0 = T0 * M;                   // first global expanded row
  float* sGt = sm;                   // [BT] token-chunk Gam, high part
  float* sGtl = sGt + BT;            // [BT] low part
  float* srq = sGtl + BT;            // [BT]
  float* srk = srq + BT;             // [BT*M]
  float* qt = srk + BT * M;          // [BT][kKT+1]
  float* kt = qt + BT * (kKT + 1);   // [kEB][kKT+1]
  float* Ps = kt + kEB * (kKT + 1);  // [BT][kEB+1]
  float* ht = Ps + BT * (kEB + 1);   // [kKT][kBVO]
  float* vt = ht + kKT * kBVO;       // [kEB][kBVO]
  const Tin* qin = static_cast<const Tin*>(a.q);
  const Tin* kin = static_cast<const Tin*>(a.k);
  const int tid = threadIdx.x, nth = blockDim.x;
  const int wid = tid >> 5, lane = tid & 31, nw = nth >> 5;
  const float* hc = a.h + (((int64_t)si.w + tab.y) * a.HV + hv) * K * V;

  for (int p = tid; p < BT; p += nth)
    sGt[p] = (p < nt && a.g) ? a.g[(T0 + p) * a.HV + hv] : 0.f;
  for (int t = wid; t < BT; t += nw) {
    float ss = 0.f;
    if (t < nt)
      for (int c = lane; c < K; c += 32) {
        const float x = ldf(qin + ((T0 + t) * a.H + kh) * K + c);
        ss += x * x;
      }
    ss = warp_sum(ss);
    if (lane == 0) srq[t] = a.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
  }
  for (int e = wid; e < BT * M; e += nw) {
    float ss = 0.f;
    if (e < ne)
      for (int c = lane; c < K; c += 32) {
        const float x = ldf(kin + ((E0 + e) * a.H + kh) * K + c);
        ss += x * x;
      }
    ss = warp_sum(ss);
    if (lane == 0) srk[e] = a.l2norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
  }
  __syncthreads();
  if (tid == 0) comp_prefix(sGt, sGtl, BT);
  // thread owns column c of rows tg, tg+4, ...
  const int c = tid % kBVO, tg = tid / kBVO;
  constexpr int RPT = 64 / 4;  // rows per thread for BT <= 64 with 256 threads
  float acc[RPT];
#pragma unroll
  for (int r = 0; r < RPT; ++r) acc[r] = 0.f;
  // inter-chunk term q.h over K tiles
  for (int k0 = 0; k0 < K; k0 += kKT) {
    __syncthreads();
    for (int i = tid; i < BT * kKT; i += nth) {
      const int t = i / kKT, cc = i - t * kKT;
      qt[t * (kKT + 1) + cc] =
          (t < nt && k0 + cc < K) ? ldf(qin + ((T0 + t) * a.H + kh) * K + k0 + cc) : 0.f;
    }
    for (int i = tid; i < kKT * kBVO; i += nth) {
      const int r = i / kBVO, cc = i - r * kBVO;
      ht[i] = (k0 + r < K && cc < nv) ? hc[(int64_t)(k0 + r) * V + v0 + cc] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const int t = tg + 4 * r;
      if (t < BT) {
        float s = 0.f;
        for (int kk = 0; kk < kKT; ++kk) s += qt[t * (kKT + 1) + kk] * ht[kk * kBVO + c];
        acc[r] += s;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RPT; ++r) {
    const int t = tg + 4 * r;
    if (t < BT) acc[r] *= expf(sGt[t] + sGtl[t]) * srq[t];
  }
  // intra-chunk term, expanded positions in tiles of kEB
  for (int e0 = 0; e0 < ne; e0 += kEB) {
    __syncthreads();
    for (int i = tid; i < BT * kEB; i += nth) Ps[(i / kEB) * (kEB + 1) + i % kEB] = 0.f;
    for (int k0 = 0; k0 < K; k0 += kKT) {
      __syncthreads();
      for (int i = tid; i < BT * kKT; i += nth) {
        const int t = i / kKT, cc = i - t * kKT;
        qt[t * (kKT + 1) + cc] =
            (t < nt && k0 + cc < K) ? ldf(qin + ((T0 + t) * a.H + kh) * K + k0 + cc) : 0.f;
      }
      for (int i = tid; i < kEB * kKT; i += nth) {
        const int e = i / kKT, cc = i - e * kKT;
        kt[e * (kKT + 1) + cc] = (e0 + e < ne && k0 + cc < K)
                                     ? ldf(kin + ((E0 + e0 + e) * a.H + kh) * K + k0 + cc)
                                     : 0.f;
      }
      __syncthreads();
      for (int i = tid; i < BT * kEB; i += nth) {
        const int t = i / kEB, e = i - t * kEB;
        float s = 0.f;
        for (int kk = 0; kk < kKT; ++kk) s += qt[t * (kKT + 1) + kk] * kt[e * (kKT + 1) + kk];
        Ps[t * (kEB + 1) + e] += s;
      }
    }
    __syncthreads();
    for (int i = tid; i < BT * kEB; i += nth) {
      const int t = i / kEB, e = i - t * kEB;
      const int eg = e0 + e, s = eg / M;
      float val = 0.f;
      if (t < nt && eg < ne && s <= t)
        val = Ps[t * (kEB + 1) + e] * srq[t] * srk[eg] * expf(gam_diff(sGt, sGtl, t, s));
      Ps[t * (kEB + 1) + e] = val;
    }
    for (int i = tid; i < kEB * kBVO; i += nth) {
      const int e = i / kBVO, cc = i - e * kBVO;
      vt[i] = (e0 + e < ne && cc < nv) ? a.v_new[((E0 + e0 + e) * a.HV + hv) * V + v0 + cc]
                                       : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const int t = tg + 4 * r;
      if (t < BT) {
        float s = 0.f;
        for (int e = 0; e < kEB; ++e) s += Ps[t * (kEB + 1) + e] * vt[e * kBVO + c];
        acc[r] += s;
      }
    }
  }
  if (c < nv) {
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const int t = tg + 4 * r;
      if (t < nt) a.o[((T0 + t) * a.HV + hv) * V + v0 + c] = a.scale * acc[r];
    }
  }
}

template <typename Tin>
cudaError_t run_generic(const ChunkProblem& p, const GenArgs& a) {
  const int BT = p.BT, K = p.K;
  const size_t smem_wy = sizeof(float) * ((size_t)BT * (K + 1) + 2 * (size_t)BT * (BT + 1) + 4 * BT);
  const size_t smem_h = sizeof(float) * ((size_t)K * kBVH + 2 * (size_t)BT * (K + 1) +
                                         2 * (size_t)BT * kBVH + 3 * BT);
  const size_t smem_o = sizeof(float) * (3 * (size_t)BT + (size_t)BT * p.M + BT * (kKT + 1) +
                                         kEB * (kKT + 1) + BT * (kEB + 1) + kKT * kBVO +
                                         kEB * kBVO);
  cudaError_t e;
  e = cudaFuncSetAttribute(wy_generic_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_wy);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(h_generic_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_h);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(o_generic_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_o);
  if (e != cudaSuccess) return e;
  if (p.NE_max > 0) {
    wy_generic_kernel<Tin><<<dim3((unsigned)p.NE_max, p.HV), 256, smem_wy, p.stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  record_stage(2, p.stream);
  if (p.N_seq > 0) {
    h_generic_kernel<Tin><<<dim3(p.N_seq, p.HV, (unsigned)cdiv(p.V, kBVH)), 256, smem_h,
                            p.stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  record_stage(3, p.stream);
  if (p.NT_max > 0) {
    o_generic_kernel<Tin><<<dim3((unsigned)p.NT_max, p.HV, (unsigned)cdiv(p.V, kBVO)), 256,
                            smem_o, p.stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  record_stage(4, p.stream);
  return cudaSuccess;
}

}  // namespace

WsLayout generic_layout(int B, int T, int N_seq, int H, int HV, int K, int V, int M, int BT) {
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
  L.A = take(sizeof(float) * Te * HV * BT);
  L.w = take(sizeof(float) * Te * HV * K);
  L.u = take(sizeof(float) * Te * HV * V);
  L.gexp = take(sizeof(float) * Te * HV * 2);
  L.v_new = take(sizeof(float) * Te * HV * V);
  L.h = take(sizeof(float) * (size_t)NT * HV * K * V);
  L.total = off;
  L.path = 0;
  return L;
}

cudaError_t launch_tables(const ChunkProblem& p, const WsLayout& L, uint8_t* ws) {
  return launch_pdl(
      tables_kernel, dim3(1), dim3(kTabThreads), 0, p.stream, p.cu_seqlens, p.N_seq, p.B, p.T, p.M, p.BT,
      p.NE_max, p.NT_max, reinterpret_cast<int4*>(ws + L.seq_info),
      reinterpret_cast<int2*>(ws + L.exp_tab), reinterpret_cast<int2*>(ws + L.tok_tab),
      L.blk_tab == SIZE_MAX ? nullptr : reinterpret_cast<int4*>(ws + L.blk_tab),
      block128_bound(p.B, p.T, p.N_seq, p.M), reinterpret_cast<int*>(ws + L.status),
      // the chain order only matters for ragged sequences
      (L.seq_order == SIZE_MAX || !p.cu_seqlens) ? nullptr : reinterpret_cast<int*>(ws + L.seq_order));
}

cudaError_t launch_chunk_generic(const ChunkProblem& p, const WsLayout& L, uint8_t* ws) {
  GenArgs a;
  a.q = p.q; a.k = p.k; a.v = p.v; a.beta = p.beta; a.g = p.g; a.h0 = p.h0; a.o = p.o;
  a.hT = p.hT;
  a.N_seq = p.N_seq; a.H = p.H; a.HV = p.HV; a.K = p.K; a.V = p.V; a.M = p.M; a.BT = p.BT;
  a.l2norm = p.l2norm; a.scale = p.scale;
  a.seq_info = reinterpret_cast<const int4*>(ws + L.seq_info);
  a.exp_tab = reinterpret_cast<const int2*>(ws + L.exp_tab);
  a.tok_tab = reinterpret_cast<const int2*>(ws + L.tok_tab);
  a.A = reinterpret_cast<float*>(ws + L.A);
  a.w = reinterpret_cast<float*>(ws + L.w);
  a.u = reinterpret_cast<float*>(ws + L.u);
  a.gexp = reinterpret_cast<float*>(ws + L.gexp);
  a.v_new = reinterpret_cast<float*>(ws + L.v_new);
  a.h = reinterpret_cast<float*>(ws + L.h);
  switch (p.dt) {
    case GDP_BF16: return run_generic<__nv_bfloat16>(p, a);
    case GDP_F16: return run_generic<__half>(p, a);
    default: return run_generic<float>(p, a);
  }
}

}  // namespace gdp
