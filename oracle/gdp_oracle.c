/*
 * Gated Delta Product (GDP) oracle: plain, slow, obviously-correct CPU code.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call this file;
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes (sources are the three Megatron-core API pages
 * "core.ssm.ops.gdp.prepare", "core.ssm.ops.gdp.chunk_o",
 * "core.ssm.ops.gdp.wy_fast"):
 *
 *   oracle_gate_map / oracle_prepare
 *       The prepare page, module overview and gdp_prepare_kernel /
 *       gdp_{decode,prefill}_prepare sections: split the post-conv row
 *       x[n,t,:] = [ value (M*H*P) | key (M*G*N) | query (G*N) ], expand the
 *       G key/query groups to H heads, fold the M Householder copies into the
 *       sequence (expanded position t*M + j), beta = sigmoid(b),
 *       g = -exp(A_log) * softplus(a + dt_bias), softplus as on the page's
 *       softplus section (identity above 20, else log1p(exp(x))). Decode puts
 *       the query on the last copy and g on the first copy, zeros elsewhere.
 *       Evaluated in fp32, operation by operation, with the host libm.
 *       Parity with the GPU: copies are bit moves (bit-exact); the gates use
 *       the host libm's expf/log1pf, so they agree with CUDA's to a few ulp.
 *
 *   oracle_gdp_walk / oracle_gdp_recurrent
 *       The gated delta rule applied over the Householder-expanded stream,
 *       token by token and copy by copy, in fp64:
 *           S <- exp(g_e) * S * (I - beta_e k_e k_e^T) + beta_e v_e k_e^T
 *       with S the V x K state of one (sequence, value head); g_e = g_t on the
 *       first copy of token t and 0 on the others; the output for token t is
 *       o_t = scale * S q_t read after its last copy (prepare page, decode
 *       bullet: query on the last copy, decay on the first). The chunk_o page
 *       states the same placement for the chunked form (queries on the
 *       unexpanded stream, keys/values on the expanded one).
 *       GVA (wy_fast page, recompute_w_u_fwd parameters): value head hv reads
 *       key/query head hv / (HV/H).
 *       Varlen (cu_seqlens on the unexpanded stream, chunk_o page): each
 *       sequence starts from its own initial state.
 *       Optional L2 norm of q and k per (position, head): x / sqrt(sum x^2 + 1e-6)
 *       (prepare page, gdp_prefill_prepare returns: the norm is left to the
 *       chunked consumer).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off (no FMA contraction, so the fp32
 * map is the literal sequence of IEEE operations).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype codes used by this file (the Python wrapper passes them). */
#define OR_BF16 0
#define OR_F16 1
#define OR_F32 2

static float or_bf16_to_f32(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* IEEE binary16 -> binary32, exact (every half is representable). */
static float or_f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h >> 15) & 1u;
  uint32_t ex = (uint32_t)(h >> 10) & 0x1fu;
  uint32_t man = (uint32_t)h & 0x3ffu;
  float mag;
  if (ex == 0) {
    mag = ldexpf((float)man, -24); /* subnormal (or zero) */
  } else if (ex == 31) {
    mag = man ? NAN : INFINITY;
  } else {
    mag = ldexpf((float)(man | 0x400u), (int)ex - 25);
  }
  return sign ? -mag : mag;
}

static size_t or_esize(int dtype) { return dtype == OR_F32 ? 4u : 2u; }

static float or_load(const void* base, int64_t idx, int dtype) {
  if (dtype == OR_F32) return ((const float*)base)[idx];
  uint16_t h = ((const uint16_t*)base)[idx];
  return dtype == OR_BF16 ? or_bf16_to_f32(h) : or_f16_to_f32(h);
}

/* softplus as the prepare page defines it: identity strictly above 20,
 * otherwise log1p(exp(x)) in fp32. */
static float or_softplus(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

static float or_sigmoid(float b) { return 1.0f / (1.0f + expf(-b)); }

static float or_decay(float a, float A_log, float dt_bias) {
  float sp = or_softplus(a + dt_bias);
  return -(expf(A_log) * sp);
}

/* The two gates alone, for callers that already hold b and a as fp32.
 * b: [nb_rows, H] beta logits, a: [na_rows, H] decay inputs (row-major). */
int oracle_gate_map(const float* b, int64_t nb_rows, const float* a, int64_t na_rows, int H,
                    const float* A_log, const float* dt_bias, float* beta, float* g) {
  if (H <= 0) return 1;
  for (int64_t r = 0; r < nb_rows; ++r)
    for (int h = 0; h < H; ++h) beta[r * H + h] = or_sigmoid(b[r * H + h]);
  for (int64_t r = 0; r < na_rows; ++r)
    for (int h = 0; h < H; ++h) g[r * H + h] = or_decay(a[r * H + h], A_log[h], dt_bias[h]);
  return 0;
}

/*
 * The prepare map for one call.
 *   x  : [n, T, M*H*P + M*G*N + G*N] in `dtype`, element strides x_sn, x_st
 *        (last dim contiguous)
 *   ba : [n, T, M*H + H] in `dtype`, strides ba_sn, ba_st
 *   interleave == 1 (decode):  q [n,T*M,H,N]  g [n,T*M,H]
 *   interleave == 0 (prefill): q [n,T,H,N]    g [n,T,H]
 *   always: k [n,T*M,H,N], v [n,T*M,H,P] (dtype), beta [n,T*M,H] fp32
 * Returns 0 on success, 1 on a bad argument.
 */
int oracle_prepare(const void* x, int64_t x_sn, int64_t x_st, const void* ba, int64_t ba_sn,
                   int64_t ba_st, const float* A_log, const float* dt_bias, int n, int T, int M,
                   int H, int G, int P, int N, int dtype, int interleave, void* q, void* k,
                   void* v, float* beta, float* g) {
  if (n < 0 || T < 0 || M <= 0 || H <= 0 || G <= 0 || P <= 0 || N <= 0) return 1;
  if (H % G != 0) return 1;
  const size_t es = or_esize(dtype);
  const int hpg = H / G;
  const int64_t k_base = (int64_t)M * H * P;
  const int64_t q_base = k_base + (int64_t)M * G * N;
  const uint8_t* xb = (const uint8_t*)x;
  uint8_t* qb = (uint8_t*)q;
  uint8_t* kb = (uint8_t*)k;
  uint8_t* vb = (uint8_t*)v;
  for (int in = 0; in < n; ++in) {
    for (int t = 0; t < T; ++t) {
      const int64_t xrow = (int64_t)in * x_sn + (int64_t)t * x_st;
      const int64_t barow = (int64_t)in * ba_sn + (int64_t)t * ba_st;
      float gt[1024];
      if (H > 1024) return 1;
      for (int h = 0; h < H; ++h) {
        float a = or_load(ba, barow + (int64_t)M * H + h, dtype);
        gt[h] = or_decay(a, A_log[h], dt_bias[h]);
      }
      for (int j = 0; j < M; ++j) {
        const int64_t e = (int64_t)in * T * M + (int64_t)t * M + j; /* expanded row */
        for (int h = 0; h < H; ++h) {
          const int grp = h / hpg;
          /* value: copy-major [M][H][P] block */
          memcpy(vb + ((e * H + h) * (int64_t)P) * es,
                 xb + (xrow + (int64_t)j * H * P + (int64_t)h * P) * es, (size_t)P * es);
          /* key: copy-major [M][G][N] block, group grp expanded to head h */
          memcpy(kb + ((e * H + h) * (int64_t)N) * es,
                 xb + (xrow + k_base + (int64_t)j * G * N + (int64_t)grp * N) * es,
                 (size_t)N * es);
          float b = or_load(ba, barow + (int64_t)j * H + h, dtype);
          beta[e * H + h] = or_sigmoid(b);
          if (interleave) {
            uint8_t* qdst = qb + ((e * H + h) * (int64_t)N) * es;
            if (j == M - 1)
              memcpy(qdst, xb + (xrow + q_base + (int64_t)grp * N) * es, (size_t)N * es);
            else
              memset(qdst, 0, (size_t)N * es); /* +0.0 in every supported dtype */
            g[e * H + h] = (j == 0) ? gt[h] : 0.0f;
          }
        }
      }
      if (!interleave) {
        const int64_t r = (int64_t)in * T + t;
        for (int h = 0; h < H; ++h) {
          const int grp = h / hpg;
          memcpy(qb + ((r * H + h) * (int64_t)N) * es,
                 xb + (xrow + q_base + (int64_t)grp * N) * es, (size_t)N * es);
          g[r * H + h] = gt[h];
        }
      }
    }
  }
  return 0;
}

/* fp32 -> bf16, round to nearest even (NaN kept quiet). */
static uint16_t or_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static void or_store(void* base, int64_t idx, int dtype, float v) {
  if (dtype == OR_F32)
    ((float*)base)[idx] = v;
  else
    ((uint16_t*)base)[idx] = or_f32_to_bf16(v);
}

/*
 * The short causal conv that precedes prepare (prepare page, module overview:
 * prepare reads the conv's output; "a -1 slot zeroes its conv output"). The
 * pages do not spell the conv out; this is the depthwise causal short conv
 * with SiLU, written from its definition, per channel c of a sequence:
 *     xin(t) = the sequence's input at t, or for t < 0 its state entry
 *              W-1+t (the W-1 inputs before the sequence, oldest first), or 0
 *              without a state;
 *     z = b[c];  z = z + w[c][i] * xin(t - (W-1) + i)   for i = 0 .. W-1;
 *     y = z / (1 + exp(-z)),  stored in `dtype` (bf16 rounds to nearest even).
 * Evaluated in fp32 one operation at a time (no contraction) with host libm.
 *   xp     [n, T, C] dtype, strides xp_sn, xp_st (elements)
 *   w      [C, W] fp32; b [C] fp32 or NULL
 *   decode = 0: sequences are the batch rows, or (n == 1) the cu [N_seq + 1]
 *            ranges; st_in [N_seq, C, W-1] or NULL, st_out [N_seq, C, W-1]
 *            or NULL receives the last W-1 inputs of state ++ tokens. Rows
 *            outside every sequence are left as they are in x_out.
 *   decode = 1: request r's S = T tokens continue from pool entry slot[r]
 *            (st_in == st_out, [n_slots, C, W-1], updated in place); slot -1,
 *            a slot outside [-1, n_slots) or one named twice makes the request
 *            padding: zero output rows, no state touched.
 *   x_out  [n, T, C] dtype (contiguous).
 * dtype: OR_BF16 or OR_F32. Returns 0, or 1 on a bad argument.
 */
int oracle_conv(const void* xp, int64_t xp_sn, int64_t xp_st, const float* w, const float* b,
                int W, const void* st_in, void* st_out, const int32_t* cu, int N_seq,
                const int32_t* slot, int n_slots, int n, int T, int C, int dtype, int decode,
                void* x_out) {
  if (n < 0 || T < 0 || C <= 0 || W < 1 || W > 64 || (dtype != OR_BF16 && dtype != OR_F32))
    return 1;
  const int nseq = decode ? n : (cu ? N_seq : n);
  float* win = (float*)malloc(sizeof(float) * (size_t)(W + T));
  if (!win) return 1;
  for (int s = 0; s < nseq; ++s) {
    int in = s, t0 = 0, t1 = T;
    const void* sin = st_in;
    void* sout = st_out;
    int64_t sidx = s;
    if (!decode && cu) {
      in = 0;
      t0 = cu[s];
      t1 = cu[s + 1];
      if (t0 < 0 || t1 < t0 || t1 > T) { free(win); return 1; }
    }
    if (decode) {
      int sl = slot[s];
      int pad = sl < 0 || sl >= n_slots;
      for (int r = 0; r < n && !pad; ++r)
        if (r != s && slot[r] == sl) pad = 1;
      if (pad) {
        for (int t = 0; t < T; ++t)
          for (int c = 0; c < C; ++c) or_store(x_out, ((int64_t)s * T + t) * C + c, dtype, 0.0f);
        continue;
      }
      sidx = sl;
    }
    const int len = t1 - t0;
    for (int c = 0; c < C; ++c) {
      /* win[0 .. W-2]: the state; win[W-1 + j]: token t0 + j */
      for (int i = 0; i < W - 1; ++i)
        win[i] = sin ? or_load(sin, (sidx * C + c) * (int64_t)(W - 1) + i, dtype) : 0.0f;
      for (int j = 0; j < len; ++j)
        win[W - 1 + j] = or_load(xp, (int64_t)in * xp_sn + (int64_t)(t0 + j) * xp_st + c, dtype);
      for (int j = 0; j < len; ++j) {
        float z = b ? b[c] : 0.0f;
        for (int i = 0; i < W; ++i) z = z + w[(int64_t)c * W + i] * win[j + i];
        const float y = z / (1.0f + expf(-z));
        or_store(x_out, ((int64_t)in * T + t0 + j) * C + c, dtype, y);
      }
      if (sout)
        for (int i = 0; i < W - 1; ++i) {
          const float v = win[len + i]; /* the last W-1 entries of state ++ tokens */
          if (dtype == OR_F32)
            ((float*)sout)[(sidx * C + c) * (int64_t)(W - 1) + i] = v;
          else
            ((uint16_t*)sout)[(sidx * C + c) * (int64_t)(W - 1) + i] = or_f32_to_bf16(v);
        }
    }
  }
  free(win);
  return 0;
}

/* One gated-delta step on the V x K state S (row-major, S[i*K + c]):
 *   S <- eg * S * (I - b kk kk^T) + b vv kk^T.   sk: V-sized scratch for S kk. */
static void or_step(double* S, int K, int V, const double* kk, const double* vv, double b,
                    double eg, double* sk) {
  for (int i = 0; i < V; ++i) {
    double acc = 0.0;
    for (int c = 0; c < K; ++c) acc += S[(int64_t)i * K + c] * kk[c];
    sk[i] = acc; /* (S k)_i */
  }
  for (int i = 0; i < V; ++i)
    for (int c = 0; c < K; ++c) {
      double proj = S[(int64_t)i * K + c] - b * sk[i] * kk[c]; /* S (I - b k k^T) */
      S[(int64_t)i * K + c] = eg * proj + b * vv[i] * kk[c];
    }
}

static void or_read(const double* S, int K, int V, const double* qq, double scale, double* out) {
  for (int i = 0; i < V; ++i) {
    double acc = 0.0;
    for (int c = 0; c < K; ++c) acc += S[(int64_t)i * K + c] * qq[c];
    out[i] = scale * acc;
  }
}

static void or_vec(const double* src, int n, int l2norm, double* dst) {
  if (!l2norm) {
    memcpy(dst, src, sizeof(double) * (size_t)n);
    return;
  }
  double ss = 0.0;
  for (int c = 0; c < n; ++c) ss += src[c] * src[c];
  double r = 1.0 / sqrt(ss + 1e-6);
  for (int c = 0; c < n; ++c) dst[c] = src[c] * r;
}

/*
 * Token walk for the chunked prefill problem (all inputs fp64, row-major):
 *   q [B,T,H,K]   k [B,T*M,H,K]   v [B,T*M,HV,V]   beta [B,T*M,HV]
 *   g [B,T,HV] natural-log decay per token (NULL = ungated, g = 0)
 *   h0 [S_count,HV,K,V] initial state per sequence (NULL = zeros)
 *   cu_seqlens [nseq+1] token offsets into row 0 (NULL = B sequences of T)
 * Outputs: o [B,T,HV,V], hT [S_count,HV,K,V] (may be NULL), with
 * S_count = nseq when cu_seqlens is given (then B must be 1), else B.
 */
int oracle_gdp_walk(const double* q, const double* k, const double* v, const double* beta,
                    const double* g, const double* h0, const int32_t* cu_seqlens, int nseq, int B,
                    int T, int H, int HV, int K, int V, int M, double scale, int l2norm,
                    int nthreads, double* o, double* hT) {
  if (B <= 0 || T < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || M <= 0) return 1;
  if (HV % H != 0) return 1;
  if (cu_seqlens && B != 1) return 1;
  const int S_count = cu_seqlens ? nseq : B;
  const int grp = HV / H;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
  int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int s = 0; s < S_count; ++s) {
    for (int hv = 0; hv < HV; ++hv) {
      const int b = cu_seqlens ? 0 : s;
      const int t0 = cu_seqlens ? cu_seqlens[s] : 0;
      const int t1 = cu_seqlens ? cu_seqlens[s + 1] : T;
      const int kh = hv / grp;
      double* S = (double*)calloc((size_t)V * K, sizeof(double));
      double* sk = (double*)malloc(sizeof(double) * (size_t)V);
      double* kk = (double*)malloc(sizeof(double) * (size_t)K);
      double* qq = (double*)malloc(sizeof(double) * (size_t)K);
      if (!S || !sk || !kk || !qq || t0 < 0 || t1 > T || t1 < t0) {
#pragma omp atomic write
        bad = 1;
        free(S); free(sk); free(kk); free(qq);
        continue;
      }
      if (h0) { /* h0 is stored [K][V]; S is its transpose */
        const double* H0 = h0 + ((int64_t)s * HV + hv) * (int64_t)K * V;
        for (int i = 0; i < V; ++i)
          for (int c = 0; c < K; ++c) S[(int64_t)i * K + c] = H0[(int64_t)c * V + i];
      }
      for (int t = t0; t < t1; ++t) {
        for (int j = 0; j < M; ++j) {
          const int64_t e = ((int64_t)b * T + t) * M + j;
          or_vec(k + (e * H + kh) * (int64_t)K, K, l2norm, kk);
          const double be = beta[e * HV + hv];
          const double ge = (j == 0 && g) ? g[((int64_t)b * T + t) * HV + hv] : 0.0;
          or_step(S, K, V, kk, v + (e * HV + hv) * (int64_t)V, be, exp(ge), sk);
        }
        const int64_t r = (int64_t)b * T + t;
        or_vec(q + (r * H + kh) * (int64_t)K, K, l2norm, qq);
        or_read(S, K, V, qq, scale, o + (r * HV + hv) * (int64_t)V);
      }
      if (hT) {
        double* HT = hT + ((int64_t)s * HV + hv) * (int64_t)K * V;
        for (int i = 0; i < V; ++i)
          for (int c = 0; c < K; ++c) HT[(int64_t)c * V + i] = S[(int64_t)i * K + c];
      }
      free(S); free(sk); free(kk); free(qq);
    }
  }
  return bad;
}

/*
 * Recurrent (decode) walk: every request runs L = S*M steps, each step
 * consuming its own q/k/v/beta/g (the decode prepare layout, where q and g
 * have already been placed on the copies), and emitting o after every step.
 *   q [n,L,H,K] k [n,L,H,K] v [n,L,HV,V] beta [n,L,HV] g [n,L,HV] (natural log)
 *   state [n,HV,K,V] in/out, o [n,L,HV,V]
 */
int oracle_gdp_recurrent(const double* q, const double* k, const double* v, const double* beta,
                         const double* g, double* state, int n, int L, int H, int HV, int K, int V,
                         double scale, int l2norm, int nthreads, double* o) {
  if (n < 0 || L < 0 || H <= 0 || HV <= 0 || K <= 0 || V <= 0 || HV % H != 0) return 1;
  const int grp = HV / H;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
  int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int r = 0; r < n; ++r) {
    for (int hv = 0; hv < HV; ++hv) {
      const int kh = hv / grp;
      double* S = (double*)malloc(sizeof(double) * (size_t)V * K);
      double* sk = (double*)malloc(sizeof(double) * (size_t)V);
      double* kk = (double*)malloc(sizeof(double) * (size_t)K);
      double* qq = (double*)malloc(sizeof(double) * (size_t)K);
      if (!S || !sk || !kk || !qq) {
#pragma omp atomic write
        bad = 1;
        free(S); free(sk); free(kk); free(qq);
        continue;
      }
      double* st = state + ((int64_t)r * HV + hv) * (int64_t)K * V;
      for (int i = 0; i < V; ++i)
        for (int c = 0; c < K; ++c) S[(int64_t)i * K + c] = st[(int64_t)c * V + i];
      for (int e = 0; e < L; ++e) {
        const int64_t re = (int64_t)r * L + e;
        or_vec(k + (re * H + kh) * (int64_t)K, K, l2norm, kk);
        or_step(S, K, V, kk, v + (re * HV + hv) * (int64_t)V, beta[re * HV + hv],
                exp(g[re * HV + hv]), sk);
        or_vec(q + (re * H + kh) * (int64_t)K, K, l2norm, qq);
        or_read(S, K, V, qq, scale, o + (re * HV + hv) * (int64_t)V);
      }
      for (int i = 0; i < V; ++i)
        for (int c = 0; c < K; ++c) st[(int64_t)c * V + i] = S[(int64_t)i * K + c];
      free(S); free(sk); free(kk); free(qq);
    }
  }
  return bad;
}

/* Threads the OpenMP runtime will use for the walks (for reporting). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
