// Backward of the log-linear Mamba-2 forward on the CUDA cores (fp32 arithmetic), for
// the loss sum(dO * o): dq, dk (per Q/K group), dv, d(log a) and dlambda.
//
// The write-up gives no backward; this is the chain rule on the masked form
// o_t = sum_{s<=t} lambda_t^{l(t,s)} M^S(t,s) (q_t . k_s) v_s (write-up
// https://www.yoousoft.com/industry/3746.html, sections 特殊结构：树划分 and
// 对Mamba-2和门控的对数线性推广), organised by the same chunks and Fenwick blocks as the
// forward's chunkwise algorithm (section 高效训练算法, Algorithm 1).  With
// w_ts = lambda_t^{l(t,s)} 2^(G_t - G_s):
//   dq_t  = sum_s w_ts (dO_t . v_s) k_s
//   dk_s  = sum_t w_ts (dO_t . v_s) q_t
//   dv_s  = sum_t w_ts (q_t . k_s) dO_t
//   dlambda_t^l = sum over s at level l of 2^(G_t - G_s) (q_t . k_s)(dO_t . v_s)
//   d(log a_r) = sum over u >= r of (R_u - C_u), with R_u = dO_u . o_u =
//     sum_l lambda_u^l dlambda_u^l (o is linear in lambda_u) and C_u = v_u . dv_u;
//     this is the sum of the terms A_ts over t >= r > s, in which log a_r appears.
// Kernels (chunk C <= 64 tokens; the forward's chunk states and Fenwick blocks first):
//   bwd_intra     per chunk: the in-chunk pairs (levels 0 .. log2 C) of every output;
//   bwd_inter_q   per query chunk, per set bit m of its index: dq and dlambda from the
//                 block it reads, and that block's "dual" Σ w_t q_t dO_tᵀ (added up over
//                 the query chunks that read the block, with atomics);
//   bwd_inter_kv  per key chunk, per level whose block holds it and has readers: dk and
//                 dv from the dual, decayed from each key to the end of the block;
//   bwd_final     group sums of dq and dk, casts;
//   bwd_dloga     d(log a) as a reverse running sum per (b, h), kept in fp64.
// The gradient is returned with respect to log a, the form a enters the forward in: for
// a close to 0 the one with respect to a, d(log a)/a, would turn the fp32 rounding of
// the running sum into arbitrarily large errors.
#include <cuda_runtime.h>

#include "ll_internal.cuh"

namespace ll {

namespace {

constexpr int kT = 256;  // threads per CTA

struct BwdPlan {
  GenPlan g;       // the forward's chunk states and blocks, at chunk C <= 64
  size_t off_dual; // BH * nblk * dk * dv fp32, zeroed per call
  size_t off_dq;   // (B, T, H, dk) fp32 per-head dq
  size_t off_dk;   // (B, T, H, dk) fp32 per-head dk
  size_t off_dv;   // (B, T, H, dv) fp32
  size_t bytes;
};

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* a;
  const float* lam;
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  float* dloga;
  float* dlam;
  char* ws;
};

// ---- in-chunk pairs -----------------------------------------------------------------
template <typename TIn>
__global__ void __launch_bounds__(kT) bwd_intra(GenPlan p, BwdArgs x, size_t off_dq, size_t off_dk,
                                               size_t off_dv) {
  extern __shared__ float sm[];
  const int C = p.C, dk = p.dk, dv = p.dv, L = p.L, nl = p.clog + 1;
  const int j = blockIdx.x, bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H, grp = h / p.hpg;
  const long long t0 = (long long)j * C;
  float* qs = sm;               // C * dk
  float* ks = qs + C * dk;      // C * dk
  float* vs = ks + C * dk;      // C * dv
  float* ds = vs + C * dv;      // C * dv  (dO)
  float* gs = ds + C * dv;      // C
  float* ls = gs + C;           // C * nl  (lambda of the in-chunk levels)
  float* dS = ls + C * nl;      // C * C: w (dO . v)
  float* P = dS + C * C;        // C * C: w (q . k)
  float* X = P + C * C;         // C * C: 2^(g_t - g_s) (q . k)(dO . v)
  const TIn* q = static_cast<const TIn*>(x.q);
  const TIn* k = static_cast<const TIn*>(x.k);
  const TIn* v = static_cast<const TIn*>(x.v);
  const TIn* dO = static_cast<const TIn*>(x.dO);
  for (int e = threadIdx.x; e < C * dk; e += kT) {
    const int s = e / dk, i = e % dk;
    const size_t gi = (((size_t)b * p.T + t0 + s) * p.G + grp) * dk + i;
    qs[e] = ll_load(q, gi);
    ks[e] = ll_load(k, gi);
  }
  for (int e = threadIdx.x; e < C * dv; e += kT) {
    const int s = e / dv, jv = e % dv;
    const size_t gi = (((size_t)b * p.T + t0 + s) * p.H + h) * dv + jv;
    vs[e] = ll_load(v, gi);
    ds[e] = ll_load(dO, gi);
  }
  const float* g = reinterpret_cast<const float*>(x.ws + p.off_g) + (size_t)bh * p.T + t0;
  for (int s = threadIdx.x; s < C; s += kT) gs[s] = g[s];
  for (int e = threadIdx.x; e < C * nl; e += kT) {
    const int t = e / nl, l = e % nl;
    ls[e] = x.lam[(((size_t)b * p.T + t0 + t) * p.H + h) * L + l];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < C * C; e += kT) {
    const int t = e / C, s = e % C;
    float a1 = 0.f, a2 = 0.f, a3 = 0.f;
    if (s <= t) {
      float qk = 0.f, dov = 0.f;
      for (int i = 0; i < dk; ++i) qk += qs[t * dk + i] * ks[s * dk + i];
      for (int jv = 0; jv < dv; ++jv) dov += ds[t * dv + jv] * vs[s * dv + jv];
      const float ed = exp2f(gs[t] - gs[s]);
      const float w = ls[t * nl + bit_length(t ^ s)] * ed;
      a1 = w * dov;
      a2 = w * qk;
      a3 = ed * qk * dov;
    }
    dS[e] = a1;
    P[e] = a2;
    X[e] = a3;
  }
  __syncthreads();
  float* dq32 = reinterpret_cast<float*>(x.ws + off_dq);
  float* dk32 = reinterpret_cast<float*>(x.ws + off_dk);
  float* dv32 = reinterpret_cast<float*>(x.ws + off_dv);
  for (int e = threadIdx.x; e < C * dk; e += kT) {
    const int r = e / dk, i = e % dk;
    float aq = 0.f, ak = 0.f;
    for (int s = 0; s <= r; ++s) aq += dS[r * C + s] * ks[s * dk + i];  // r as query
    for (int t = r; t < C; ++t) ak += dS[t * C + r] * qs[t * dk + i];   // r as key
    const size_t o = (((size_t)b * p.T + t0 + r) * p.H + h) * dk + i;
    dq32[o] = aq;
    dk32[o] = ak;
  }
  for (int e = threadIdx.x; e < C * dv; e += kT) {
    const int r = e / dv, jv = e % dv;
    float av = 0.f;
    for (int t = r; t < C; ++t) av += P[t * C + r] * ds[t * dv + jv];
    dv32[(((size_t)b * p.T + t0 + r) * p.H + h) * dv + jv] = av;
  }
  for (int e = threadIdx.x; e < C * L; e += kT) {
    const int t = e / L, l = e % L;
    float acc = 0.f;
    if (l < nl)
      for (int s = 0; s <= t; ++s)
        if (bit_length(t ^ s) == l) acc += X[t * C + s];
    x.dlam[(((size_t)b * p.T + t0 + t) * p.H + h) * L + l] = acc;  // inter levels: next kernel
  }
}

// ---- query side of the inter-chunk levels ---------------------------------------------
template <typename TIn>
__global__ void __launch_bounds__(kT) bwd_inter_q(GenPlan p, BwdArgs x, size_t off_dq, size_t off_dual) {
  extern __shared__ float sm[];
  const int C = p.C, dk = p.dk, dv = p.dv, L = p.L;
  const int j = blockIdx.x, bh = blockIdx.y;
  if (j == 0) return;  // the first chunk reads no block
  const int b = bh / p.H, h = bh % p.H, grp = h / p.hpg;
  const long long t0 = (long long)j * C;
  const int S = dk * dv;
  float* qs = sm;            // C * dk
  float* ds = qs + C * dk;   // C * dv
  float* Bm = ds + C * dv;   // dk * dv: the block
  float* ws_ = Bm + S;       // C: 2^(g_t + D) of this level
  float* wl = ws_ + C;       // C: lambda_t^l 2^(g_t + D)
  const TIn* q = static_cast<const TIn*>(x.q);
  const TIn* dO = static_cast<const TIn*>(x.dO);
  for (int e = threadIdx.x; e < C * dk; e += kT) {
    const int s = e / dk, i = e % dk;
    qs[e] = ll_load(q, (((size_t)b * p.T + t0 + s) * p.G + grp) * dk + i);
  }
  for (int e = threadIdx.x; e < C * dv; e += kT) {
    const int s = e / dv, jv = e % dv;
    ds[e] = ll_load(dO, (((size_t)b * p.T + t0 + s) * p.H + h) * dv + jv);
  }
  const float* g = reinterpret_cast<const float*>(x.ws + p.off_g) + (size_t)bh * p.T + t0;
  const float* blk = reinterpret_cast<const float*>(x.ws + p.off_blk);
  const float* blkG = reinterpret_cast<const float*>(x.ws + p.off_blkG) + (size_t)bh * p.nblk;
  float* dq32 = reinterpret_cast<float*>(x.ws + off_dq);
  float* dual = reinterpret_cast<float*>(x.ws + off_dual);
  float D = 0.f;
  for (int m = 0; (j >> m) > 0; ++m) {
    if (!((j >> m) & 1)) continue;
    const int bidx = p.blk_off[m] + (((j >> m) - 1) >> 1);
    const int lvl = p.clog + 1 + m;
    __syncthreads();  // previous level done with Bm, ws_, wl
    const float* Bsrc = blk + ((size_t)bh * p.nblk + bidx) * S;
    for (int e = threadIdx.x; e < S; e += kT) Bm[e] = Bsrc[e];
    for (int t = threadIdx.x; t < C; t += kT) {
      const float e2 = exp2f(g[t] + D);
      ws_[t] = e2;
      wl[t] = x.lam[(((size_t)b * p.T + t0 + t) * p.H + h) * L + lvl] * e2;
    }
    __syncthreads();
    // dq_t += w_t Bm dO_t
    for (int e = threadIdx.x; e < C * dk; e += kT) {
      const int t = e / dk, i = e % dk;
      float acc = 0.f;
      for (int jv = 0; jv < dv; ++jv) acc += Bm[i * dv + jv] * ds[t * dv + jv];
      dq32[(((size_t)b * p.T + t0 + t) * p.H + h) * dk + i] += wl[t] * acc;
    }
    // dlambda_t^lvl = 2^(g_t + D) q_tᵀ Bm dO_t
    for (int t = threadIdx.x; t < C; t += kT) {
      float acc = 0.f;
      for (int jv = 0; jv < dv; ++jv) {
        float u = 0.f;
        for (int i = 0; i < dk; ++i) u += qs[t * dk + i] * Bm[i * dv + jv];
        acc += u * ds[t * dv + jv];
      }
      x.dlam[(((size_t)b * p.T + t0 + t) * p.H + h) * L + lvl] = ws_[t] * acc;
    }
    // dual of the block: sum_t w_t q_t dO_tᵀ
    float* dst = dual + ((size_t)bh * p.nblk + bidx) * S;
    for (int e = threadIdx.x; e < S; e += kT) {
      const int i = e / dv, jv = e % dv;
      float acc = 0.f;
      for (int t = 0; t < C; ++t) acc += wl[t] * qs[t * dk + i] * ds[t * dv + jv];
      atomicAdd(dst + e, acc);
    }
    D += blkG[bidx];
  }
}

// ---- key side of the inter-chunk levels -----------------------------------------------
template <typename TIn>
__global__ void __launch_bounds__(kT) bwd_inter_kv(GenPlan p, BwdArgs x, size_t off_dk, size_t off_dv,
                                                  size_t off_dual) {
  extern __shared__ float sm[];
  const int C = p.C, dk = p.dk, dv = p.dv;
  const int u = blockIdx.x, bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H, grp = h / p.hpg;
  const long long t0 = (long long)u * C;
  const int S = dk * dv;
  float* ks = sm;            // C * dk
  float* vs = ks + C * dk;   // C * dv
  float* Dm = vs + C * dv;   // dk * dv: the dual
  float* ts = Dm + S;        // C: 2^(decay from key s to the end of the block)
  const TIn* k = static_cast<const TIn*>(x.k);
  const TIn* v = static_cast<const TIn*>(x.v);
  for (int e = threadIdx.x; e < C * dk; e += kT) {
    const int s = e / dk, i = e % dk;
    ks[e] = ll_load(k, (((size_t)b * p.T + t0 + s) * p.G + grp) * dk + i);
  }
  for (int e = threadIdx.x; e < C * dv; e += kT) {
    const int s = e / dv, jv = e % dv;
    vs[e] = ll_load(v, (((size_t)b * p.T + t0 + s) * p.H + h) * dv + jv);
  }
  const float* g = reinterpret_cast<const float*>(x.ws + p.off_g) + (size_t)bh * p.T + t0;
  const float* gamma = reinterpret_cast<const float*>(x.ws + p.off_gamma) + (size_t)bh * p.N;
  const float* dual = reinterpret_cast<const float*>(x.ws + off_dual);
  float* dk32 = reinterpret_cast<float*>(x.ws + off_dk);
  float* dv32 = reinterpret_cast<float*>(x.ws + off_dv);
  const float gend = g[C - 1];
  for (int m = 0; m < p.M; ++m) {
    const int i = u >> m;
    // node (m, i) is read at level log2 C + 1 + m by the chunks of node (m, i + 1) when
    // i is even and that node starts inside the sequence
    if ((i & 1) || ((long long)(i + 1) << m) >= p.N) continue;
    const int bidx = p.blk_off[m] + (i >> 1);
    float tail = 0.f;  // decay of the chunks after u up to the end of node (m, i)
    for (int c = u + 1; c < ((i + 1) << m); ++c) tail += gamma[c];
    __syncthreads();  // previous level done with Dm, ts
    const float* src = dual + ((size_t)bh * p.nblk + bidx) * S;
    for (int e = threadIdx.x; e < S; e += kT) Dm[e] = src[e];
    for (int s = threadIdx.x; s < C; s += kT) ts[s] = exp2f(gend - g[s] + tail);
    __syncthreads();
    for (int e = threadIdx.x; e < C * dk; e += kT) {
      const int s = e / dk, ii = e % dk;
      float acc = 0.f;
      for (int jv = 0; jv < dv; ++jv) acc += Dm[ii * dv + jv] * vs[s * dv + jv];
      dk32[(((size_t)b * p.T + t0 + s) * p.H + h) * dk + ii] += ts[s] * acc;
    }
    for (int e = threadIdx.x; e < C * dv; e += kT) {
      const int s = e / dv, jv = e % dv;
      float acc = 0.f;
      for (int ii = 0; ii < dk; ++ii) acc += Dm[ii * dv + jv] * ks[s * dk + ii];
      dv32[(((size_t)b * p.T + t0 + s) * p.H + h) * dv + jv] += ts[s] * acc;
    }
  }
}

// ---- group sums and casts -----------------------------------------------------------------
template <typename TIn>
__global__ void __launch_bounds__(kT) bwd_final(GenPlan p, BwdArgs x, size_t off_dq, size_t off_dk,
                                               size_t off_dv) {
  const float* dq32 = reinterpret_cast<const float*>(x.ws + off_dq);
  const float* dk32 = reinterpret_cast<const float*>(x.ws + off_dk);
  const float* dv32 = reinterpret_cast<const float*>(x.ws + off_dv);
  const size_t nqk = (size_t)p.B * p.T * p.G * p.dk;
  const size_t nv = (size_t)p.B * p.T * p.H * p.dv;
  for (size_t e = blockIdx.x * (size_t)kT + threadIdx.x; e < nqk + nv; e += (size_t)gridDim.x * kT) {
    if (e < nqk) {
      const size_t i = e % p.dk, bt_g = e / p.dk, grp = bt_g % p.G, bt = bt_g / p.G;
      float sq = 0.f, sk = 0.f;
      for (int hh = 0; hh < p.hpg; ++hh) {
        const size_t o = (bt * p.H + grp * p.hpg + hh) * p.dk + i;
        sq += dq32[o];
        sk += dk32[o];
      }
      ll_store(static_cast<TIn*>(x.dq), e, sq);
      ll_store(static_cast<TIn*>(x.dk), e, sk);
    } else {
      ll_store(static_cast<TIn*>(x.dv), e - nqk, dv32[e - nqk]);
    }
  }
}

// ---- d(log a) as a reverse running sum of R_u - C_u ----------------------------------------
template <typename TIn>
__global__ void __launch_bounds__(kT) bwd_dloga(GenPlan p, BwdArgs x, size_t off_dv) {
  __shared__ double s_part[kT / 32];
  __shared__ double s_carry;
  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
  const int L = p.L, dv = p.dv;
  const float* dv32 = reinterpret_cast<const float*>(x.ws + off_dv);
  const TIn* v = static_cast<const TIn*>(x.v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_carry = 0.0;
  __syncthreads();
  // segments of kT tokens from the end; inside a segment thread i holds token end - i
  for (long long end = (long long)p.T - 1; end >= 0; end -= kT) {
    const long long t = end - threadIdx.x;
    double val = 0.0;
    if (t >= 0) {
      const size_t row = ((size_t)b * p.T + t) * p.H + h;
      float R = 0.f, Cv = 0.f;
      for (int l = 0; l < L; ++l) R += x.lam[row * L + l] * x.dlam[row * L + l];
      for (int jv = 0; jv < dv; ++jv) Cv += ll_load(v, row * dv + jv) * dv32[row * dv + jv];
      val = (double)R - (double)Cv;
    }
    // inclusive scan over the segment in thread order (= decreasing token index)
    double inc = val;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += y;
    }
    if (lane == 31) s_part[warp] = inc;
    __syncthreads();
    double add = s_carry;
    for (int w = 0; w < warp; ++w) add += s_part[w];
    inc += add;
    if (t >= 0) {
      const size_t row = ((size_t)b * p.T + t) * p.H + h;
      // position 0 of the sequence: no key precedes it, so its log-decay has no effect
      x.dloga[row] = t == 0 ? 0.f : (float)inc;
    }
    __syncthreads();
    if (threadIdx.x == kT - 1) s_carry = inc;
    __syncthreads();
  }
}

bool make_bwd_plan(const ll_shape& s, BwdPlan* bp) {
  ll_shape c = s;
  c.chunk = s.chunk < 64 ? s.chunk : 64;  // the result does not depend on the chunk
  if (!make_gen_plan(c, &bp->g)) return false;
  const size_t BH = (size_t)s.batch * s.heads, S = (size_t)s.d_k * s.d_v;
  size_t o = al(bp->g.bytes);
  bp->off_dual = o;
  o = al(o + sizeof(float) * BH * bp->g.nblk * S);
  bp->off_dq = o;
  o = al(o + sizeof(float) * (size_t)s.batch * s.T * s.heads * s.d_k);
  bp->off_dk = o;
  o = al(o + sizeof(float) * (size_t)s.batch * s.T * s.heads * s.d_k);
  bp->off_dv = o;
  o = al(o + sizeof(float) * (size_t)s.batch * s.T * s.heads * s.d_v);
  bp->bytes = o;
  return true;
}

template <typename TIn>
cudaError_t run_bwd(const BwdPlan& bp, const BwdArgs& x, const FwdArgs& fa, cudaStream_t st) {
  const GenPlan& p = bp.g;
  const int BH = p.B * p.H;
  const int C = p.C, dk = p.dk, dv = p.dv;
  // the forward's chunk states and Fenwick blocks (same kernels as the generic forward)
  cudaError_t e = launch_generic_states(p, sizeof(TIn) == 2, fa, st);
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(x.ws + bp.off_dual, 0, sizeof(float) * (size_t)BH * p.nblk * dk * dv, st)) !=
      cudaSuccess)
    return e;
  const size_t sm1 = sizeof(float) * ((size_t)2 * C * dk + 2 * C * dv + C + C * (p.clog + 1) + 3 * C * C);
  if ((e = cudaFuncSetAttribute(bwd_intra<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) !=
      cudaSuccess)
    return e;
  bwd_intra<TIn><<<dim3(p.N, BH), kT, sm1, st>>>(p, x, bp.off_dq, bp.off_dk, bp.off_dv);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  const size_t sm2 = sizeof(float) * ((size_t)C * dk + C * dv + dk * dv + 2 * C);
  if ((e = cudaFuncSetAttribute(bwd_inter_q<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)) !=
      cudaSuccess)
    return e;
  bwd_inter_q<TIn><<<dim3(p.N, BH), kT, sm2, st>>>(p, x, bp.off_dq, bp.off_dual);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  const size_t sm3 = sizeof(float) * ((size_t)C * dk + C * dv + dk * dv + C);
  if ((e = cudaFuncSetAttribute(bwd_inter_kv<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)) !=
      cudaSuccess)
    return e;
  bwd_inter_kv<TIn><<<dim3(p.N, BH), kT, sm3, st>>>(p, x, bp.off_dk, bp.off_dv, bp.off_dual);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  const size_t n = (size_t)p.B * p.T * (p.G * dk + p.H * dv);
  const unsigned gf = (unsigned)((n + kT - 1) / kT < 4096 ? (n + kT - 1) / kT : 4096);
  bwd_final<TIn><<<gf, kT, 0, st>>>(p, x, bp.off_dq, bp.off_dk, bp.off_dv);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  bwd_dloga<TIn><<<BH, kT, 0, st>>>(p, x, bp.off_dv);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

}  // namespace

size_t bwd_workspace_bytes(const ll_shape& s) {
  BwdPlan bp;
  return make_bwd_plan(s, &bp) ? bp.bytes : 0;
}

cudaError_t launch_bwd(const ll_shape& s, const void* q, const void* k, const void* v, const float* a,
                       const float* lam, const void* dO, void* dq, void* dk, void* dv, float* dloga,
                       float* dlam, char* ws, unsigned* status, cudaStream_t st) {
  BwdPlan bp;
  if (!make_bwd_plan(s, &bp)) return cudaErrorInvalidValue;
  BwdArgs x{q, k, v, a, lam, dO, dq, dk, dv, dloga, dlam, ws};
  FwdArgs fa{q, k, v, a, lam, nullptr, ws, nullptr, nullptr, 0, status, nullptr, 0};
  return s.dtype == LL_BF16 ? run_bwd<__nv_bfloat16>(bp, x, fa, st) : run_bwd<float>(bp, x, fa, st);
}

}  // namespace ll
