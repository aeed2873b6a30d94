// Log-linear Gated DeltaNet forward: Gated DeltaNet's transition kept, its attention mask
// combined with the hierarchical mask (write-up https://www.yoousoft.com/industry/3746.html,
// section 对Mamba-2和门控的对数线性推广).
//
// The gated delta rule S_t = a_t S_{t-1} (I - beta_t k_t k_tᵀ) + beta_t v_t k_tᵀ is the
// same recurrence as S_t = a_t S_{t-1} + u_t k_tᵀ with u_t = beta_t (v_t - a_t S_{t-1} k_t),
// so the model's output is the masked form over the transformed values u; the log-linear
// model weights the same terms by lambda_t^{l(t,s)}.  This file computes u; the level-fused
// forward then runs on (q, k, u, a, lambda).
//
// Chunked as in the delta rule's WY/UT form.  Within a chunk (C <= 32 tokens, g the
// chunk-local log2 decay cumsum, S the d_k x d_v state at the chunk's start):
//   u = T diag(beta) (V - diag(2^g) K S) = U_loc - W S,
//   T = (I + diag(beta) A)^-1,  A = (K Kᵀ) ⊙ 2^(g_t - g_s) strictly lower,
//   U_loc = T diag(beta) V,  W = T diag(beta 2^g) K.
//   gdn_local (every chunk at once): T by blocks, then [W | U_loc] by one triangular
//              product, written to the workspace as W, U_loc and g, chunk by chunk;
//   gdn_pass   (per (b, h) and block of value columns, chunks in order; the columns of S
//              are independent): u = U_loc - W S, written in the input dtype, then
//              S <- 2^(g_end) S + Kᵀ diag(2^(g_end - g)) u.  The next chunk's W, g, U_loc and
//              keys are copied in behind the two products.
#include <cuda_runtime.h>

#include "ll_internal.cuh"
#include "ptx.cuh"

namespace ll {

namespace {

constexpr int kG = 256;  // threads per CTA

// Chunk-local log2 decay cumsum and beta of one chunk, by warp 0.
__device__ __forceinline__ void chunk_decay(int tid, int C, const float* a, const float* beta, size_t base,
                                            size_t stride, float* gs, float* bs) {
  if (tid >= 32) return;
  float carry = 0.f;
  for (int s0 = 0; s0 < C; s0 += 32) {
    const int s = s0 + tid;
    float x = s < C ? log2f(a[base + (size_t)s * stride]) : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, off);
      if (tid >= off) x += y;
    }
    if (s < C) {
      gs[s] = x + carry;
      if (bs) bs[s] = beta[base + (size_t)s * stride];
    }
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
}

__device__ __forceinline__ void load4(const float* p, float (&x)[4]) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  x[0] = v.x;
  x[1] = v.y;
  x[2] = v.z;
  x[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&x)[4]) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  x[0] = __uint_as_float(v.x << 16);
  x[1] = __uint_as_float(v.x & 0xffff0000u);
  x[2] = __uint_as_float(v.y << 16);
  x[3] = __uint_as_float(v.y & 0xffff0000u);
}

// 16 bytes of a row of TIn (4 fp32 or 8 bf16 values), as fp32.
__device__ __forceinline__ void load16(const float* p, float* x) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  x[0] = v.x;
  x[1] = v.y;
  x[2] = v.z;
  x[3] = v.w;
}
__device__ __forceinline__ void load16(const __nv_bfloat16* p, float* x) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// One chunk of one (b, h): A, then T = (I + diag(beta) A)^-1 by 16-row blocks (the
// diagonal blocks by substitution in registers, one column per thread; the blocks below
// them as T_ij = -T_ii sum_{j <= k < i} A_ik T_kj, one block distance at a time), then
// [W | U_loc] = T [diag(beta 2^g) K | diag(beta) V] as a triangular product whose tiles go
// straight to the workspace (W, U_loc, then g).
template <typename TIn>
__global__ void __launch_bounds__(kG) gdn_local(int T, int H, int hpg, int dk, int dv, int C,
                                                const TIn* __restrict__ k, const TIn* __restrict__ v,
                                                const float* __restrict__ a, const float* __restrict__ beta,
                                                float* __restrict__ xg) {
  extern __shared__ __align__(16) float sm[];
  const int c = blockIdx.x, bh = blockIdx.y, b = bh / H, h = bh % H, G = H / hpg, grp = h / hpg;
  const int tid = threadIdx.x;
  const long long t0 = (long long)c * C;
  const int KP = dk + 4, CP = C + 4, nb = C >> 4;
  float* Kr = sm;             // C x KP: keys (rows padded), then scaled by beta 2^g
  float* Vs = Kr + C * KP;    // C x dv: values, then scaled by beta
  float* Am = Vs + C * dv;    // C x CP: diag(beta) A below the diagonal
  float* Tm = Am + C * CP;    // C x CP: T, zero above the diagonal
  float* Ym = Tm + C * CP;    // C x CP: block sums of the off-diagonal step
  float* gs = Ym + C * CP;    // C
  float* bs = gs + C;         // C
  chunk_decay(tid, C, a, beta, ((size_t)b * T + t0) * H + h, H, gs, bs);
  constexpr int per = 16 / sizeof(TIn);
  {
    const int qk = dk / per;
    const TIn* ks = k + ((size_t)b * T + t0) * G * dk + (size_t)grp * dk;
    for (int e = tid; e < C * qk; e += kG) {
      const int s = e / qk, q = e % qk;
      float x[per];
      load16(ks + (size_t)s * G * dk + q * per, x);
#pragma unroll
      for (int j = 0; j < per; j += 4)
        *reinterpret_cast<float4*>(Kr + s * KP + q * per + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
    }
    const int qv = dv / per;
    const TIn* vsrc = v + (((size_t)b * T + t0) * H + h) * dv;
    for (int e = tid; e < C * qv; e += kG) {
      const int s = e / qv, q = e % qv;
      float x[per];
      load16(vsrc + (size_t)s * H * dv + q * per, x);
#pragma unroll
      for (int j = 0; j < per; j += 4)
        *reinterpret_cast<float4*>(Vs + s * dv + q * per + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
    }
    for (int e = tid; e < C * CP; e += kG) Tm[e] = 0.f;
  }
  __syncthreads();
  // A_ts = beta_t 2^(g_t - g_s) k_t . k_s for s < t, by 2 x 2 tiles of the lower triangle
  const int ht = C >> 1, ntri = ht * (ht + 1) / 2;
  for (int tile = tid; tile < ntri; tile += kG) {
    int ta = (int)((sqrtf(8.f * tile + 1.f) - 1.f) * 0.5f);
    while ((ta + 1) * (ta + 2) / 2 <= tile) ++ta;
    while (ta * (ta + 1) / 2 > tile) --ta;
    const int tr = 2 * ta, sr = 2 * (tile - ta * (ta + 1) / 2);
    const float* x0 = Kr + tr * KP;
    const float* y0 = Kr + sr * KP;
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll 2
    for (int i = 0; i < dk; i += 4) {
      float xa[4], xb[4], ya[4], yb[4];
      load4(x0 + i, xa);
      load4(x0 + KP + i, xb);
      load4(y0 + i, ya);
      load4(y0 + KP + i, yb);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[0][0] += xa[q] * ya[q];
        acc[0][1] += xa[q] * yb[q];
        acc[1][0] += xb[q] * ya[q];
        acc[1][1] += xb[q] * yb[q];
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int t = tr + r, s2 = sr + q;
        if (s2 < t) Am[t * CP + s2] = bs[t] * exp2f(gs[t] - gs[s2]) * acc[r][q];
      }
  }
  __syncthreads();
  // right-hand sides of the product (K no longer read unscaled)
  for (int e = tid; e < C * dv; e += kG) Vs[e] *= bs[e / dv];
  for (int e = tid; e < C * dk; e += kG) {
    const int s = e / dk;
    Kr[s * KP + e % dk] *= bs[s] * exp2f(gs[s]);
  }
  if (tid < C) {  // diagonal blocks: column j of block r0 / 16
    const int r0 = tid & ~15, j = tid & 15;
    float x[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < t; ++s) acc += Am[(r0 + t) * CP + r0 + s] * x[s];
      x[t] = t < j ? 0.f : (t == j ? 1.f : -acc);
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) Tm[(r0 + t) * CP + r0 + j] = x[t];
  }
  __syncthreads();
  for (int d = 1; d < nb; ++d) {  // blocks (jb + d, jb)
    const int nel = (nb - d) * 256;
    for (int e = tid; e < nel; e += kG) {
      const int jb = e >> 8, r = (e >> 4) & 15, cc = e & 15, ib = jb + d;
      const float* arow = Am + (16 * ib + r) * CP;
      float acc = 0.f;
      for (int s = 16 * jb; s < 16 * ib; ++s) acc += arow[s] * Tm[s * CP + 16 * jb + cc];
      Ym[(16 * ib + r) * CP + 16 * jb + cc] = acc;
    }
    __syncthreads();
    for (int e = tid; e < nel; e += kG) {
      const int jb = e >> 8, r = (e >> 4) & 15, cc = e & 15, ib = jb + d;
      const float* trow = Tm + (16 * ib + r) * CP + 16 * ib;
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < 16; ++s) acc += trow[s] * Ym[(16 * ib + s) * CP + 16 * jb + cc];
      Tm[(16 * ib + r) * CP + 16 * jb + cc] = -acc;
    }
    __syncthreads();
  }
  float* dst = xg + ((size_t)bh * (T / C) + c) * (size_t)C * (dk + dv + 1);
  // out rows m0..m0+3 = T rows m0..m0+3 times B; T is zero right of the diagonal
  auto tri_mm = [&](int N, const float* B, int ldb, float* out) {
    const int tn = N >> 2, tiles = (C >> 2) * tn;
    for (int tile = tid; tile < tiles; tile += kG) {
      const int m0 = (tile / tn) * 4, n0 = (tile % tn) * 4;
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
      for (int s = 0; s < m0 + 4; ++s) {
        float bv[4];
        load4(B + s * ldb + n0, bv);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float av = Tm[(m0 + i) * CP + s];
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] += av * bv[j];
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(out + (size_t)(m0 + i) * N + n0) =
            make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
  };
  tri_mm(dk, Kr, KP, dst);
  tri_mm(dv, Vs, dv, dst + (size_t)C * dk);
  for (int e = tid; e < C; e += kG) dst[(size_t)C * (dk + dv) + e] = gs[e];
}

// Value columns j0 .. j0 + JW - 1 of one (b, h).  Each thread owns fixed output tiles: a
// 2 x 4 tile (tokens x columns) of u = U_loc - W S and a 4 x 4 tile (key rows x columns) of
// the state, kept in registers across chunks; shared memory holds S only as the operand
// of u.  Copies run in two groups per chunk: W and g (needed first; two buffers) are
// fetched a chunk and a half ahead, U_loc and the keys behind the product W S.
template <typename TIn>
__global__ void __launch_bounds__(kG, 3) gdn_pass(int T, int H, int hpg, int dk, int dv, int C, int JW,
                                                  const TIn* __restrict__ k, const float* __restrict__ xg,
                                                  TIn* __restrict__ u) {
  extern __shared__ __align__(16) float sm[];
  const int nj = dv / JW;
  const int j0 = (blockIdx.x % nj) * JW, bh = blockIdx.x / nj;
  const int b = bh / H, h = bh % H, G = H / hpg, grp = h / hpg;
  const int tid = threadIdx.x, n = T / C, WP = dk + 4;
  const size_t cst = (size_t)C * (dk + dv + 1);   // workspace floats per chunk: W, U_loc, g
  float* Wm = sm;                                   // 2 x C x WP: W (rows padded), by chunk parity
  float* gm = Wm + 2 * C * WP;                      // 2 x C: g, by chunk parity
  float* Um = gm + 2 * C;                           // C x JW: U_loc, then 2^(g_end - g) u
  float* Sm = Um + C * JW;                          // dk x JW: S
  TIn* Km = reinterpret_cast<TIn*>(Sm + dk * JW);   // C x dk: keys
  const float* xb = xg + (size_t)bh * n * cst;
  auto load_wg = [&](int c) {
    if (c < n) {
      const float* src = xb + c * cst;
      float* wd = Wm + (c & 1) * C * WP;
      float* gd = gm + (c & 1) * C;
      const int q4 = dk >> 2;
      for (int e = tid; e < C * q4; e += kG) ptx::cp_async16(wd + (e / q4) * WP + 4 * (e % q4), src + 4 * e);
      for (int e = tid; e < (C >> 2); e += kG) ptx::cp_async16(gd + 4 * e, src + (size_t)C * (dk + dv) + 4 * e);
    }
    ptx::cp_async_commit();
  };
  auto load_uk = [&](int c) {
    if (c < n) {
      const float* src = xb + c * cst + (size_t)C * dk + j0;
      const int q4 = JW >> 2;
      for (int e = tid; e < C * q4; e += kG)
        ptx::cp_async16(Um + 4 * e, src + (size_t)(e / q4) * dv + 4 * (e % q4));
      constexpr int per = 16 / sizeof(TIn);
      const int qk = dk / per;
      const TIn* ks = k + ((size_t)b * T + (size_t)c * C) * G * dk + (size_t)grp * dk;
      for (int e = tid; e < C * qk; e += kG)
        ptx::cp_async16(Km + e * per, ks + (size_t)(e / qk) * G * dk + (e % qk) * per);
    }
    ptx::cp_async_commit();
  };
  const int tn = JW >> 2;
  const bool own1 = tid < (C >> 1) * tn, own2 = tid < (dk >> 2) * tn;
  const int m1 = (tid / tn) * 2, m2 = (tid / tn) * 4, n0 = (tid % tn) * 4;
  float st[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) st[i][j] = 0.f;
  for (int e = tid; e < dk * JW; e += kG) Sm[e] = 0.f;
  load_wg(0);
  load_uk(0);
  load_wg(1);
  for (int c = 0; c < n; ++c) {
    const float* Wc = Wm + (c & 1) * C * WP;
    const float* gc = gm + (c & 1) * C;
    ptx::cp_async_wait_group<2>();  // W and g of chunk c (only chunk 0 can still be waiting)
    __syncthreads();                // ... and S of the previous chunk
    float acc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    if (own1) {
      const float* w0 = Wc + m1 * WP;
      const float* w1 = w0 + WP;
#pragma unroll 2
      for (int i = 0; i < dk; i += 4) {
        float a0[4], a1[4];
        load4(w0 + i, a0);
        load4(w1 + i, a1);
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
          float sv[4];
          load4(Sm + (i + ii) * JW + n0, sv);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[0][j] += a0[ii] * sv[j];
            acc[1][j] += a1[ii] * sv[j];
          }
        }
      }
    }
    const float gend = gc[C - 1];
    ptx::cp_async_wait_group<0>();
    __syncthreads();  // U_loc and keys of chunk c (and W and g of chunk c + 1)
    if (own1) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int s = m1 + r;
        const float f = exp2f(gend - gc[s]);
        float* ur = Um + s * JW + n0;
        TIn* out = u + (((size_t)b * T + (size_t)c * C + s) * H + h) * dv + j0 + n0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float val = ur[j] - acc[r][j];
          ll_store(out, j, val);
          ur[j] = f * val;
        }
      }
    }
    __syncthreads();  // decayed u complete; W and g of chunk c no longer read
    load_wg(c + 2);
    if (own2) {
      float a2[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) a2[i][j] = 0.f;
#pragma unroll 4
      for (int s = 0; s < C; ++s) {
        float kv[4], uv[4];
        load4(Km + s * dk + m2, kv);
        load4(Um + s * JW + n0, uv);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) a2[i][j] += kv[i] * uv[j];
      }
      const float dS = exp2f(gend);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 4; ++j) st[i][j] = dS * st[i][j] + a2[i][j];
        *reinterpret_cast<float4*>(Sm + (m2 + i) * JW + n0) = make_float4(st[i][0], st[i][1], st[i][2], st[i][3]);
      }
    }
    __syncthreads();  // keys and u read; S complete
    load_uk(c + 1);
  }
  ptx::cp_async_wait_all();
}

}  // namespace

size_t gdn_values_bytes(const ll_shape& s) {
  const size_t e = s.dtype == LL_BF16 ? 2 : 4;
  const size_t ub = (((size_t)s.batch * s.T * s.heads * s.d_v * e) + 255) & ~size_t(255);
  if (tc_supported(s)) return ub + tc_gdn_bytes(s);  // the tensor-core chunks (128 tokens)
  const size_t xb = (size_t)s.batch * s.T * s.heads * (s.d_v + s.d_k + 1) * sizeof(float);
  return ub + ((xb + 255) & ~size_t(255));
}

namespace {
template <typename TIn>
cudaError_t run_gdn(const ll_shape& s, const void* k, const void* v, const float* a, const float* beta,
                    void* u, cudaStream_t st) {
  const int C = s.chunk < 32 ? s.chunk : 32;  // divides T, since chunk does
  const size_t ub = (((size_t)s.batch * s.T * s.heads * s.d_v * (s.dtype == LL_BF16 ? 2 : 4)) + 255) &
                    ~size_t(255);
  float* xg = reinterpret_cast<float*>(static_cast<char*>(u) + ub);
  const int dk = s.d_k, dv = s.d_v, BH = s.batch * s.heads;
  const size_t sm1 = sizeof(float) * ((size_t)C * (dk + 4) + (size_t)C * dv + 3 * (size_t)C * (C + 4) + 2 * C);
  cudaError_t e = cudaFuncSetAttribute(gdn_local<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
  if (e != cudaSuccess) return e;
  gdn_local<TIn><<<dim3(s.T / C, BH), kG, sm1, st>>>(s.T, s.heads, s.heads_per_group, dk, dv, C,
                                                      static_cast<const TIn*>(k), static_cast<const TIn*>(v), a,
                                                      beta, xg);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  const int JW = dv > 32 ? 32 : dv;
  const size_t sm2 = sizeof(float) * (2 * (size_t)C * (dk + 4) + 2 * (size_t)C + (size_t)C * JW + (size_t)dk * JW) +
                     sizeof(TIn) * (size_t)C * dk;
  if ((e = cudaFuncSetAttribute(gdn_pass<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)) !=
      cudaSuccess)
    return e;
  gdn_pass<TIn><<<BH * (dv / JW), kG, sm2, st>>>(s.T, s.heads, s.heads_per_group, dk, dv, C, JW,
                                                 static_cast<const TIn*>(k), xg, static_cast<TIn*>(u));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_gdn_values(const ll_shape& s, const void* k, const void* v, const float* a,
                              const float* beta, void* u, unsigned* status, cudaStream_t st) {
  if (tc_supported(s)) {
    const size_t ub = (((size_t)s.batch * s.T * s.heads * s.d_v * 2) + 255) & ~size_t(255);
    return launch_tc_gdn(s, k, v, a, beta, u, static_cast<char*>(u) + ub, status, st);
  }
  return s.dtype == LL_BF16 ? run_gdn<__nv_bfloat16>(s, k, v, a, beta, u, st)
                            : run_gdn<float>(s, k, v, a, beta, u, st);
}

}  // namespace ll
