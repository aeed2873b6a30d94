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
//   bwd_intra     per chunk: the in-chunk pairs (levels 0 .. log2 C) of every output; for
//                 bf16, d_k = 128, d_v = 64 and T % 128 == 0 the tensor-core kernel
//                 tc_bwd_intra does the pairs inside 128-token tiles instead (chunk level
//                 0 included), and the two inter kernels start at chunk level 1;
//   bwd_inter_q   per query chunk, per set bit m of its index: dq and dlambda from the
//                 block it reads (both from the one product Bm dO_t), and that block's
//                 "dual" Σ w_t q_t dO_tᵀ (added up over the query chunks that read the
//                 block, with atomics);
//   bwd_inter_kv  per key chunk, per level whose block holds it and has readers: dk and
//                 dv from the dual, decayed from each key to the end of the block;
//   bwd_final     group sums of dq and dk, casts;
//   bwd_dloga_*   d(log a) as a reverse running sum per (b, h), kept in fp64 (per 128-token
//                 chunk, across chunks, then both added).  R_u and C_u nearly cancel (their
//                 totals are equal), so on the tensor-core path C_u is the fp32 sum of the
//                 pair terms from the exact products S and E (in-tile) plus v_u . (the
//                 inter-tile part of dv_u), not v_u . dv_u with dv from fp16 operands.
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
  bool tc;         // 128-token tiles on the tensor cores (in-tile pairs, query side)
  TcPlan tp;       // the forward's tree over tiles, at off_tc, when tc
  size_t off_dual; // BH * nblk * dk * dv fp32, zeroed per call
  size_t off_dq;   // (B, T, H, dk) fp32 per-head dq
  size_t off_dk;   // (B, T, H, dk) fp32 per-head dk
  size_t off_dv;   // (B, T, H, dv) fp32
  size_t off_tc;   // tc: the tree over tiles (TcPlan layout)
  size_t off_dimg; // tc: the duals as fp16 images, 16 KB per slot
  size_t off_dmeta;// tc: their scalars, 4 u32 per slot
  size_t off_P;    // tc: running sums of the tile decays, (B*H, NT + 1) fp64
  size_t off_cu;   // tc: C_u = v_u . dv_u summed from the pair terms, (B, T, H) fp32
  size_t off_loc;  // d(log a): per-token reverse running sums inside 128-token chunks, fp64
  size_t off_tot;  // chunk totals, then (off_carry) their reverse running sums, fp64
  size_t off_carry;
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
  extern __shared__ __align__(16) float sm[];
  const int C = p.C, dk = p.dk, dv = p.dv, L = p.L, nl = p.clog + 1;
  const int j = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int b = bh / p.H, h = bh % p.H, grp = h / p.hpg;
  const long long t0 = (long long)j * C;
  float* qs = sm;               // C x dk
  float* ks = qs + C * dk;      // C x dk
  const int CP = C + 4;         // padded row of a transposed tile (16-byte rows, 4-way banks)
  float* kTr = ks + C * dk;     // dk x C (row stride CP)
  float* vTr = kTr + CP * dk;   // dv x C (row stride CP)
  float* ds = vTr + CP * dv;    // C x dv  (dO)
  float* gs = ds + C * dv;      // C
  float* ls = gs + C;           // C x nl  (lambda of the in-chunk levels)
  float* dS = ls + C * nl;      // C x C: dO.v, then w (dO . v)
  float* P = dS + C * C;        // C x C: q.k, then w (q . k)
  float* X = P + C * C;         // C x C: 2^(g_t - g_s) (q . k)(dO . v)
  const TIn* q = static_cast<const TIn*>(x.q);
  const TIn* k = static_cast<const TIn*>(x.k);
  const TIn* v = static_cast<const TIn*>(x.v);
  const TIn* dO = static_cast<const TIn*>(x.dO);
  for (int e = tid; e < C * dk; e += kT) {
    const int s = e / dk, i = e % dk;
    const size_t gi = (((size_t)b * p.T + t0 + s) * p.G + grp) * dk + i;
    qs[e] = ll_load(q, gi);
    const float kv = ll_load(k, gi);
    ks[e] = kv;
    kTr[i * CP + s] = kv;
  }
  for (int e = tid; e < C * dv; e += kT) {
    const int s = e / dv, jv = e % dv;
    const size_t gi = (((size_t)b * p.T + t0 + s) * p.H + h) * dv + jv;
    vTr[jv * CP + s] = ll_load(v, gi);
    ds[e] = ll_load(dO, gi);
  }
  const float* g = reinterpret_cast<const float*>(x.ws + p.off_g) + (size_t)bh * p.T + t0;
  for (int s = tid; s < C; s += kT) gs[s] = g[s];
  for (int e = tid; e < C * nl; e += kT) {
    const int t = e / nl, l = e % nl;
    ls[e] = x.lam[(((size_t)b * p.T + t0 + t) * p.H + h) * L + l];
  }
  __syncthreads();
  // causal ranges: tiles of (t, s) above the diagonal are zero; in dS K (rows t) only keys
  // s < m0 + 4 contribute, in dSᵀ Q and Pᵀ dO (rows s) only queries t >= m0
  auto lower = [](int m0, int n0, int& kb, int& ke) {
    if (n0 > m0) kb = ke = 0;
  };
  auto upto = [](int m0, int, int& kb, int& ke) { ke = m0 + 4; };
  auto from = [](int m0, int, int& kb, int& ke) { kb = m0; };
  smem_mm_r(C, C, dk, qs, dk, 1, kTr, CP, tid, kT, lower, [&](int m0, int n0, float (&acc)[4][4]) {
    for (int i = 0; i < 4; ++i)
      for (int jj = 0; jj < 4; ++jj) P[(m0 + i) * C + n0 + jj] = acc[i][jj];
  });
  smem_mm_r(C, C, dv, ds, dv, 1, vTr, CP, tid, kT, lower, [&](int m0, int n0, float (&acc)[4][4]) {
    for (int i = 0; i < 4; ++i)
      for (int jj = 0; jj < 4; ++jj) dS[(m0 + i) * C + n0 + jj] = acc[i][jj];
  });
  __syncthreads();
  for (int e = tid; e < C * C; e += kT) {
    const int t = e / C, s = e % C;
    float a1 = 0.f, a2 = 0.f, a3 = 0.f;
    if (s <= t) {
      const float qk = P[e], dov = dS[e];
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
  auto row = [&](int r) { return ((size_t)b * p.T + t0 + r) * p.H + h; };
  // dq = dS K (rows: queries); dk = dSᵀ Q and dv = Pᵀ dO (rows: keys)
  smem_mm_r(C, dk, C, dS, C, 1, ks, dk, tid, kT, upto, [&](int m0, int n0, float (&acc)[4][4]) {
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(dq32 + row(m0 + i) * dk + n0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  });
  smem_mm_r(C, dk, C, dS, 1, C, qs, dk, tid, kT, from, [&](int m0, int n0, float (&acc)[4][4]) {
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(dk32 + row(m0 + i) * dk + n0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  });
  smem_mm_r(C, dv, C, P, 1, C, ds, dv, tid, kT, from, [&](int m0, int n0, float (&acc)[4][4]) {
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(dv32 + row(m0 + i) * dv + n0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  });
  for (int e = tid; e < C * L; e += kT) {
    const int t = e / L, l = e % L;
    float acc = 0.f;
    if (l < nl)
      for (int s = 0; s <= t; ++s)
        if (bit_length(t ^ s) == l) acc += X[t * C + s];
    x.dlam[row(t) * L + l] = acc;  // inter levels: next kernel
  }
}

// ---- query side of the inter-chunk levels ---------------------------------------------
template <typename TIn>
__global__ void __launch_bounds__(kT) bwd_inter_q(GenPlan p, BwdArgs x, size_t off_dq, size_t off_dual,
                                                 int m_start) {
  extern __shared__ __align__(16) float sm[];
  const int C = p.C, dk = p.dk, dv = p.dv, L = p.L;
  const int j = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  if (j == 0) return;  // the first chunk reads no block
  const int b = bh / p.H, h = bh % p.H, grp = h / p.hpg;
  const long long t0 = (long long)j * C;
  const int S = dk * dv;
  const int CP = C;            // row stride of the transposed tile (unpadded: two CTAs per SM)
  float* qs = sm;              // C x dk
  float* ds = qs + C * dk;     // C x dv   (dO)
  float* dT = ds + C * dv;     // dv x C   (dOᵀ)
  float* dw = dT + CP * dv;    // C x dv   (w_t dO_t)
  float* Bm = dw + C * dv;     // dk x dv: the block
  float* ws_ = Bm + S;         // C: 2^(g_t + D) of this level
  float* wl = ws_ + C;         // C: lambda_t^l 2^(g_t + D)
  float* dl = wl + C;          // C: q_tᵀ Bm dO_t
  const TIn* q = static_cast<const TIn*>(x.q);
  const TIn* dO = static_cast<const TIn*>(x.dO);
  for (int e = tid; e < C * dk; e += kT) {
    const int s = e / dk, i = e % dk;
    qs[e] = ll_load(q, (((size_t)b * p.T + t0 + s) * p.G + grp) * dk + i);
  }
  for (int e = tid; e < C * dv; e += kT) {
    const int s = e / dv, jv = e % dv;
    const float d = ll_load(dO, (((size_t)b * p.T + t0 + s) * p.H + h) * dv + jv);
    ds[e] = d;
    dT[jv * CP + s] = d;
  }
  const float* g = reinterpret_cast<const float*>(x.ws + p.off_g) + (size_t)bh * p.T + t0;
  const float* blk = reinterpret_cast<const float*>(x.ws + p.off_blk);
  const float* blkG = reinterpret_cast<const float*>(x.ws + p.off_blkG) + (size_t)bh * p.nblk;
  float* dq32 = reinterpret_cast<float*>(x.ws + off_dq);
  float* dual = reinterpret_cast<float*>(x.ws + off_dual);
  auto row = [&](int r) { return ((size_t)b * p.T + t0 + r) * p.H + h; };
  float D = 0.f;
  for (int m = 0; (j >> m) > 0; ++m) {
    if (!((j >> m) & 1)) continue;
    const int bidx = p.blk_off[m] + (((j >> m) - 1) >> 1);
    if (m < m_start) {  // done by the in-tile kernel; its decay still separates the levels above
      D += blkG[bidx];
      continue;
    }
    const int lvl = p.clog + 1 + m;
    __syncthreads();  // the previous level is done with the buffers
    const float* Bsrc = blk + ((size_t)bh * p.nblk + bidx) * S;
    for (int e = tid; e < S; e += kT) Bm[e] = Bsrc[e];
    for (int t = tid; t < C; t += kT) {
      const float e2 = exp2f(g[t] + D);
      ws_[t] = e2;
      wl[t] = x.lam[row(t) * L + lvl] * e2;
      dl[t] = 0.f;
    }
    __syncthreads();
    for (int e = tid; e < C * dv; e += kT) dw[e] = wl[e / dv] * ds[e];
    // (Bm dO_t) for every t, as dqᵀ = Bm dOᵀ (rows i of d_k, columns t): dq_t += w_t (Bm dO_t),
    // and dl_t = q_tᵀ (Bm dO_t) from the same tiles
    smem_mm(dk, C, dv, Bm, dv, 1, dT, CP, tid, kT, [&](int m0, int n0, float (&acc)[4][4]) {
      for (int jj = 0; jj < 4; ++jj) {
        const int t = n0 + jj;
        float4* d4 = reinterpret_cast<float4*>(dq32 + row(t) * dk + m0);
        float4 o4 = *d4;
        const float w = wl[t];
        o4.x += w * acc[0][jj];
        o4.y += w * acc[1][jj];
        o4.z += w * acc[2][jj];
        o4.w += w * acc[3][jj];
        *d4 = o4;
        const float4 q4 = *reinterpret_cast<const float4*>(qs + t * dk + m0);
        atomicAdd(dl + t, q4.x * acc[0][jj] + q4.y * acc[1][jj] + q4.z * acc[2][jj] + q4.w * acc[3][jj]);
      }
    });
    __syncthreads();  // dw and dl complete
    // dual of the block: sum_t q_t (w_t dO_t)ᵀ, added to the sums of the other readers
    float* dst = dual + ((size_t)bh * p.nblk + bidx) * S;
    smem_mm(dk, dv, C, qs, 1, dk, dw, dv, tid, kT, [&](int m0, int n0, float (&acc)[4][4]) {
      for (int i = 0; i < 4; ++i)
        atomicAdd(reinterpret_cast<float4*>(dst + (m0 + i) * dv + n0),
                  make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
    });
    for (int t = tid; t < C; t += kT) x.dlam[row(t) * L + lvl] = ws_[t] * dl[t];
    D += blkG[bidx];
  }
}

// ---- key side of the inter-chunk levels -----------------------------------------------
template <typename TIn>
__global__ void __launch_bounds__(kT) bwd_inter_kv(GenPlan p, BwdArgs x, size_t off_dk, size_t off_dv,
                                                  size_t off_dual, int m_start) {
  extern __shared__ __align__(16) float sm[];
  const int C = p.C, dk = p.dk, dv = p.dv;
  const int u = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int b = bh / p.H, h = bh % p.H, grp = h / p.hpg;
  const long long t0 = (long long)u * C;
  const int S = dk * dv;
  const int CP = C + 4;      // padded row of a transposed tile
  float* ks = sm;            // C x dk
  float* vT = ks + C * dk;   // dv x C  (Vᵀ, row stride CP)
  float* Dm = vT + CP * dv;  // dk x dv: the dual
  float* ts = Dm + S;        // C: 2^(decay from key s to the end of the block)
  const TIn* k = static_cast<const TIn*>(x.k);
  const TIn* v = static_cast<const TIn*>(x.v);
  for (int e = tid; e < C * dk; e += kT) {
    const int s = e / dk, i = e % dk;
    ks[e] = ll_load(k, (((size_t)b * p.T + t0 + s) * p.G + grp) * dk + i);
  }
  for (int e = tid; e < C * dv; e += kT) {
    const int s = e / dv, jv = e % dv;
    vT[jv * CP + s] = ll_load(v, (((size_t)b * p.T + t0 + s) * p.H + h) * dv + jv);
  }
  const float* g = reinterpret_cast<const float*>(x.ws + p.off_g) + (size_t)bh * p.T + t0;
  const float* gamma = reinterpret_cast<const float*>(x.ws + p.off_gamma) + (size_t)bh * p.N;
  const float* dual = reinterpret_cast<const float*>(x.ws + off_dual);
  float* dk32 = reinterpret_cast<float*>(x.ws + off_dk);
  float* dv32 = reinterpret_cast<float*>(x.ws + off_dv);
  auto row = [&](int r) { return ((size_t)b * p.T + t0 + r) * p.H + h; };
  const float gend = g[C - 1];
  for (int m = m_start; m < p.M; ++m) {
    const int i = u >> m;
    // node (m, i) is read at level log2 C + 1 + m by the chunks of node (m, i + 1) when
    // i is even and that node starts inside the sequence
    if ((i & 1) || ((long long)(i + 1) << m) >= p.N) continue;
    const int bidx = p.blk_off[m] + (i >> 1);
    float tail = 0.f;  // decay of the chunks after u up to the end of node (m, i)
    for (int c = u + 1; c < ((i + 1) << m); ++c) tail += gamma[c];
    __syncthreads();  // the previous level is done with the buffers
    const float* src = dual + ((size_t)bh * p.nblk + bidx) * S;
    for (int e = tid; e < S; e += kT) Dm[e] = src[e];
    for (int s = tid; s < C; s += kT) ts[s] = exp2f(gend - g[s] + tail);
    __syncthreads();
    // dkᵀ = Dual Vᵀ (rows i of d_k, columns s): dk_s += t_s (Dual v_s)
    smem_mm(dk, C, dv, Dm, dv, 1, vT, CP, tid, kT, [&](int m0, int n0, float (&acc)[4][4]) {
      for (int jj = 0; jj < 4; ++jj) {
        const int s = n0 + jj;
        float4* d4 = reinterpret_cast<float4*>(dk32 + row(s) * dk + m0);
        float4 o4 = *d4;
        const float w = ts[s];
        o4.x += w * acc[0][jj];
        o4.y += w * acc[1][jj];
        o4.z += w * acc[2][jj];
        o4.w += w * acc[3][jj];
        *d4 = o4;
      }
    });
    // dv_s += t_s (Dualᵀ k_s)
    smem_mm(C, dv, dk, ks, dk, 1, Dm, dv, tid, kT, [&](int m0, int n0, float (&acc)[4][4]) {
      for (int r = 0; r < 4; ++r) {
        float4* d4 = reinterpret_cast<float4*>(dv32 + row(m0 + r) * dv + n0);
        float4 o4 = *d4;
        const float w = ts[m0 + r];
        o4.x += w * acc[r][0];
        o4.y += w * acc[r][1];
        o4.z += w * acc[r][2];
        o4.w += w * acc[r][3];
        *d4 = o4;
      }
    });
  }
}

// ---- group sums and casts -----------------------------------------------------------------
__device__ __forceinline__ void store4(float* p, size_t i, float4 v) { *reinterpret_cast<float4*>(p + i) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, size_t i, float4 v) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  *reinterpret_cast<uint2*>(p + i) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

// Four consecutive elements per thread (d_k and d_v are multiples of 4).
template <typename TIn>
__global__ void __launch_bounds__(kT) bwd_final(GenPlan p, BwdArgs x, size_t off_dq, size_t off_dk,
                                               size_t off_dv, bool with_dv) {
  const float* dq32 = reinterpret_cast<const float*>(x.ws + off_dq);
  const float* dk32 = reinterpret_cast<const float*>(x.ws + off_dk);
  const float* dv32 = reinterpret_cast<const float*>(x.ws + off_dv);
  const size_t nqk = (size_t)p.B * p.T * p.G * p.dk;
  const size_t nv = with_dv ? (size_t)p.B * p.T * p.H * p.dv : 0;  // (tensor cores: written by tc_bwd_kv)
  for (size_t e4 = blockIdx.x * (size_t)kT + threadIdx.x; 4 * e4 < nqk + nv; e4 += (size_t)gridDim.x * kT) {
    const size_t e = 4 * e4;
    if (e < nqk) {
      const size_t i = e % p.dk, bt_g = e / p.dk, grp = bt_g % p.G, bt = bt_g / p.G;
      float4 sq = make_float4(0.f, 0.f, 0.f, 0.f), sk = sq;
      for (int hh = 0; hh < p.hpg; ++hh) {
        const size_t o = (bt * p.H + grp * p.hpg + hh) * p.dk + i;
        const float4 a = *reinterpret_cast<const float4*>(dq32 + o), c = *reinterpret_cast<const float4*>(dk32 + o);
        sq.x += a.x; sq.y += a.y; sq.z += a.z; sq.w += a.w;
        sk.x += c.x; sk.y += c.y; sk.z += c.z; sk.w += c.w;
      }
      store4(static_cast<TIn*>(x.dq), e, sq);
      store4(static_cast<TIn*>(x.dk), e, sk);
    } else {
      store4(static_cast<TIn*>(x.dv), e - nqk, *reinterpret_cast<const float4*>(dv32 + (e - nqk)));
    }
  }
}

// ---- d(log a) as a reverse running sum of R_u - C_u ----------------------------------------
// Three passes over chunks of 128 tokens, every sum in fp64: per chunk the values and their
// reverse running sums (thread i holds token 128 c + 127 - i) and the chunk's total; per
// (b, h) the reverse running sums of the chunk totals after each chunk; then both added.
constexpr int kDlChunk = 128;

__device__ __forceinline__ void load4v(const float* p, float (&x)[4]) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  x[0] = v.x;
  x[1] = v.y;
  x[2] = v.z;
  x[3] = v.w;
}
__device__ __forceinline__ void load4v(const __nv_bfloat16* p, float (&x)[4]) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  x[0] = __uint_as_float(v.x << 16);
  x[1] = __uint_as_float(v.x & 0xffff0000u);
  x[2] = __uint_as_float(v.y << 16);
  x[3] = __uint_as_float(v.y & 0xffff0000u);
}

// cu: C_u from the pair terms and R_u where the tensor-core kernels summed them (else
// v_u . dv_u and sum_l lambda_u^l dlambda_u^l here).
template <typename TIn>
__global__ void __launch_bounds__(kDlChunk) bwd_dloga_local(GenPlan p, BwdArgs x, size_t off_dv, const float* cu,
                                                           double* loc, double* tot) {
  __shared__ double s_part[kDlChunk / 32];
  const int c = blockIdx.x, bh = blockIdx.y, b = bh / p.H, h = bh % p.H, nch = gridDim.x;
  const int L = p.L, dv = p.dv, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* dv32 = reinterpret_cast<const float*>(x.ws + off_dv);
  const TIn* v = static_cast<const TIn*>(x.v);
  const long long t = (long long)c * kDlChunk + (kDlChunk - 1 - threadIdx.x);
  double val = 0.0;
  if (t < p.T) {
    const size_t row = ((size_t)b * p.T + t) * p.H + h;
    float R = 0.f, Cv = 0.f;
    if (cu) {  // both summed by the tensor-core kernels: C_u, then R_u after B T H values
      Cv = cu[row];
      R = cu[(size_t)p.B * p.T * p.H + row];
    } else {
      if ((L & 1) == 0) {  // rows of an even level count are 8-byte aligned: pairs
        const float2* l2 = reinterpret_cast<const float2*>(x.lam + row * L);
        const float2* d2 = reinterpret_cast<const float2*>(x.dlam + row * L);
#pragma unroll 4
        for (int l = 0; l < L / 2; ++l) {
          const float2 a2 = l2[l], b2 = d2[l];
          R += a2.x * b2.x + a2.y * b2.y;
        }
      } else {
#pragma unroll 4
        for (int l = 0; l < L; ++l) R += x.lam[row * L + l] * x.dlam[row * L + l];
      }
      const float* dr = dv32 + row * dv;
      const TIn* vr = v + row * dv;
      for (int jv = 0; jv < dv; jv += 4) {  // rows 16-byte aligned (d_v a multiple of 16)
        const float4 d4 = *reinterpret_cast<const float4*>(dr + jv);
        float v4[4];
        load4v(vr + jv, v4);
        Cv += v4[0] * d4.x + v4[1] * d4.y + v4[2] * d4.z + v4[3] * d4.w;
      }
    }
    val = (double)R - (double)Cv;
  }
  double inc = val;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  if (lane == 31) s_part[warp] = inc;
  __syncthreads();
  for (int w = 0; w < warp; ++w) inc += s_part[w];
  if (t < p.T) loc[(size_t)bh * p.T + t] = inc;
  if (threadIdx.x == kDlChunk - 1) tot[(size_t)bh * nch + c] = inc;
}

// carry[c] = sum of the totals of the chunks after c, per (b, h)
__global__ void __launch_bounds__(kT) bwd_dloga_carry(int nch, const double* tot, double* carry) {
  __shared__ double s_part[kT / 32];
  __shared__ double s_carry;
  const int bh = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_carry = 0.0;
  __syncthreads();
  for (int end = nch - 1; end >= 0; end -= kT) {  // thread i holds chunk end - i
    const int c = end - (int)threadIdx.x;
    const double val = c >= 0 ? tot[(size_t)bh * nch + c] : 0.0;
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
    if (c >= 0) carry[(size_t)bh * nch + c] = inc - val;  // exclusive: the chunks after c
    __syncthreads();
    if (threadIdx.x == kT - 1) s_carry = inc;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kDlChunk) bwd_dloga_apply(GenPlan p, BwdArgs x, const double* loc,
                                                           const double* carry) {
  const int c = blockIdx.x, bh = blockIdx.y, b = bh / p.H, h = bh % p.H, nch = gridDim.x;
  const long long t = (long long)c * kDlChunk + threadIdx.x;
  if (t >= p.T) return;
  // position 0 of the sequence: no key precedes it, so its log-decay has no effect
  x.dloga[((size_t)b * p.T + t) * p.H + h] =
      t == 0 ? 0.f : (float)(loc[(size_t)bh * p.T + t] + carry[(size_t)bh * nch + c]);
}

bool make_bwd_plan(const ll_shape& s, BwdPlan* bp) {
  ll_shape c = s;
  c.chunk = s.chunk < 64 ? s.chunk : 64;  // the result does not depend on the chunk
  if (!make_gen_plan(c, &bp->g)) return false;
  const size_t BH = (size_t)s.batch * s.heads, S = (size_t)s.d_k * s.d_v;
  bp->tc = s.dtype == LL_BF16 && bp->g.C == 64 && make_tc_plan(s, &bp->tp);
  // the generic chunk states and blocks only off the tensor-core path (which uses the
  // plan for the dual slots alone)
  size_t o = bp->tc ? 0 : al(bp->g.bytes);
  // dual slots per (b, h): every block, or on the tensor-core path those from chunk level 1
  const size_t nsl = bp->tc ? (size_t)(bp->g.nblk - (bp->g.M > 1 ? bp->g.blk_off[1] : 0)) : (size_t)bp->g.nblk;
  bp->off_dual = o;
  o = al(o + sizeof(float) * BH * nsl * S);
  bp->off_dq = o;
  o = al(o + sizeof(float) * (size_t)s.batch * s.T * s.heads * s.d_k);
  bp->off_dk = o;
  o = al(o + sizeof(float) * (size_t)s.batch * s.T * s.heads * s.d_k);
  bp->off_dv = o;
  o = al(o + sizeof(float) * (size_t)s.batch * s.T * s.heads * s.d_v);
  bp->off_tc = bp->off_dimg = bp->off_dmeta = bp->off_P = bp->off_cu = o;
  if (bp->tc) {
    o = al(o + bp->tp.bytes);
    bp->off_dimg = o;
    o = al(o + BH * nsl * S * 2);
    bp->off_dmeta = o;
    o = al(o + BH * nsl * 4 * sizeof(unsigned));
    bp->off_P = o;
    o = al(o + BH * (bp->tp.NT + 1) * sizeof(double));
    bp->off_cu = o;  // C_u, then R_u
    o = al(o + 2 * (size_t)s.batch * s.T * s.heads * sizeof(float));
  }
  const size_t nch = ((size_t)s.T + kDlChunk - 1) / kDlChunk;
  bp->off_loc = o;
  o = al(o + BH * (size_t)s.T * sizeof(double));
  bp->off_tot = o;
  o = al(o + BH * nch * sizeof(double));
  bp->off_carry = o;
  o = al(o + BH * nch * sizeof(double));
  bp->bytes = o;
  return true;
}

template <typename TIn>
cudaError_t run_bwd(const ll_shape& s, const BwdPlan& bp, const BwdArgs& x, const FwdArgs& fa, cudaStream_t st) {
  const GenPlan& p = bp.g;
  const int BH = p.B * p.H;
  const int C = p.C, dk = p.dk, dv = p.dv;
  // the forward's chunk states and Fenwick blocks (same kernels as the generic forward),
  // off the tensor-core path
  cudaError_t e = cudaSuccess;
  if (!bp.tc && (e = launch_generic_states(p, sizeof(TIn) == 2, fa, st)) != cudaSuccess) return e;
  // The tensor-core kernels use the blocks from chunk level 1 up only, so their duals take
  // a compact slot range per (b, h): slot = blk_off[m + 1] - blk_off[1] + index, of
  // tc_slots per (b, h); the CUDA-core kernels use every block.
  const int tc_base = p.M > 1 ? p.blk_off[1] : 0, tc_slots = p.nblk - tc_base;
  int tc_dual_off[32];
  for (int m = 0; m < 32; ++m) tc_dual_off[m] = m + 1 < p.M ? p.blk_off[m + 1] - tc_base : 0;  // chunk level m + 1
  // The duals start at zero, except, on the tensor-core path with an even tile count, those
  // of the tile nodes (tile level 0, the first n0 slots of each (b, h)): each has one reader
  // tile, whose tc_bwd_q CTA publishes it as an fp16 image straight away.
  const size_t S = (size_t)dk * dv * sizeof(float);
  const size_t n0 = bp.tc && bp.tp.NT % 2 == 0 && bp.tp.MT > 1 ? (size_t)tc_dual_off[1] : 0;
  if (n0 > 0) {
    if ((e = cudaMemset2DAsync(x.ws + bp.off_dual + n0 * S, tc_slots * S, 0, (tc_slots - n0) * S, BH, st)) !=
        cudaSuccess)
      return e;
  } else {
    const size_t nslot_zero = (size_t)BH * (bp.tc ? tc_slots : p.nblk);
    if ((e = cudaMemsetAsync(x.ws + bp.off_dual, 0, nslot_zero * S, st)) != cudaSuccess) return e;
  }
  // the pairs inside 128-token tiles (two 64-token chunks) on the tensor cores where the
  // shape allows; the inter-chunk kernels then start at chunk level 1, and the query side
  // of those levels runs on the tensor cores over the forward's tree of tile nodes
  const bool tc = bp.tc;
  const int m_start = tc ? 1 : 0;
  if (tc) {
    FwdArgs ta = fa;
    ta.ws = x.ws + bp.off_tc;
    if ((e = launch_tc_nodes(bp.tp, ta, st)) != cudaSuccess) return e;
    if ((e = launch_tc_bwd_intra(s, x.q, x.k, x.v, x.dO, x.a, x.lam, reinterpret_cast<float*>(x.ws + bp.off_dq),
                                 reinterpret_cast<float*>(x.ws + bp.off_dk),
                                 reinterpret_cast<float*>(x.ws + bp.off_dv), x.dlam,
                                 reinterpret_cast<float*>(x.ws + bp.off_cu), fa.status, st)) != cudaSuccess)
      return e;
  } else {
    const size_t sm1 = sizeof(float) * ((size_t)2 * C * dk + (size_t)(C + 4) * (dk + dv) + C * dv + C +
                                        C * (p.clog + 1) + 3 * C * C);
    if ((e = cudaFuncSetAttribute(bwd_intra<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) !=
        cudaSuccess)
      return e;
    bwd_intra<TIn><<<dim3(p.N, BH), kT, sm1, st>>>(p, x, bp.off_dq, bp.off_dk, bp.off_dv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launch();
  }
  const size_t sm2 = sizeof(float) * ((size_t)C * dk + 3 * C * dv + dk * dv + 3 * C);
  if ((e = cudaFuncSetAttribute(bwd_inter_q<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)) !=
      cudaSuccess)
    return e;
  if (tc) {
    if ((e = launch_tc_bwd_q(bp.tp, x.q, x.dO, x.a, x.lam, x.ws + bp.off_tc, reinterpret_cast<float*>(x.ws + bp.off_dq),
                             x.dlam, reinterpret_cast<float*>(x.ws + bp.off_dual), tc_dual_off, tc_slots,
                             reinterpret_cast<float*>(x.ws + bp.off_cu) + (size_t)p.B * p.T * p.H,
                             n0 > 0 ? reinterpret_cast<uint8_t*>(x.ws + bp.off_dimg) : nullptr,
                             n0 > 0 ? reinterpret_cast<unsigned*>(x.ws + bp.off_dmeta) : nullptr, fa.status,
                             st)) != cudaSuccess)
      return e;
  } else {
    bwd_inter_q<TIn><<<dim3(p.N, BH), kT, sm2, st>>>(p, x, bp.off_dq, bp.off_dual, m_start);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launch();
  }
  if (tc) {
    if ((e = launch_tc_bwd_kv(bp.tp, x.k, x.v, x.a, x.ws + bp.off_tc, reinterpret_cast<const float*>(x.ws + bp.off_dual),
                              reinterpret_cast<uint8_t*>(x.ws + bp.off_dimg),
                              reinterpret_cast<unsigned*>(x.ws + bp.off_dmeta),
                              reinterpret_cast<double*>(x.ws + bp.off_P), tc_dual_off, tc_slots, (int)n0,
                              reinterpret_cast<float*>(x.ws + bp.off_dk), reinterpret_cast<float*>(x.ws + bp.off_dv), x.dv,
                              reinterpret_cast<float*>(x.ws + bp.off_cu), fa.status, st)) != cudaSuccess)
      return e;
  } else {
    const size_t sm3 = sizeof(float) * ((size_t)C * dk + (size_t)(C + 4) * dv + dk * dv + C);
    if ((e = cudaFuncSetAttribute(bwd_inter_kv<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)) !=
        cudaSuccess)
      return e;
    bwd_inter_kv<TIn><<<dim3(p.N, BH), kT, sm3, st>>>(p, x, bp.off_dk, bp.off_dv, bp.off_dual, m_start);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launch();
  }
  const size_t n4 = (size_t)p.B * p.T * (p.G * dk + p.H * dv) / 4;
  const unsigned gf = (unsigned)((n4 + kT - 1) / kT < 8192 ? (n4 + kT - 1) / kT : 8192);
  bwd_final<TIn><<<gf, kT, 0, st>>>(p, x, bp.off_dq, bp.off_dk, bp.off_dv, !bp.tc);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  const int nch = (p.T + kDlChunk - 1) / kDlChunk;
  double* loc = reinterpret_cast<double*>(x.ws + bp.off_loc);
  double* tot = reinterpret_cast<double*>(x.ws + bp.off_tot);
  double* carry = reinterpret_cast<double*>(x.ws + bp.off_carry);
  const float* cu = tc ? reinterpret_cast<const float*>(x.ws + bp.off_cu) : nullptr;
  bwd_dloga_local<TIn><<<dim3(nch, BH), kDlChunk, 0, st>>>(p, x, bp.off_dv, cu, loc, tot);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  bwd_dloga_carry<<<BH, kT, 0, st>>>(nch, tot, carry);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  bwd_dloga_apply<<<dim3(nch, BH), kDlChunk, 0, st>>>(p, x, loc, carry);
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
  return s.dtype == LL_BF16 ? run_bwd<__nv_bfloat16>(s, bp, x, fa, st) : run_bwd<float>(s, bp, x, fa, st);
}

}  // namespace ll
