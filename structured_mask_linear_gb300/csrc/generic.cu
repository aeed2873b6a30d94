// Generic CUDA-core path of the log-linear Mamba-2 forward: every supported shape
// (d_k 16..128, d_v 16..64, chunk 16..128, fp32 or bf16), fp32 arithmetic.
//
// Follows the chunkwise algorithm of the log-linear attention write-up
// (https://www.yoousoft.com/industry/3746.html, section 高效训练算法, Algorithm 1):
//   1. per chunk: chunk-local log2 decay cumsum g, chunk decay gamma and the chunk
//      state H_j = sum_s 2^(gamma_j - g_s) k_s v_sᵀ (the state-passing primitive);
//   2. per (b, h): the Fenwick block states of the chunk-level hierarchy
//      Block_m[i] = decayed sum of the 2^m chunk states i*2^m .. (i+1)*2^m - 1, kept
//      for even i only (those are the buckets later chunks read);
//   3. per chunk: the intra-chunk masked product (levels 0 .. log2 C) plus, for every
//      set bit m of the chunk index j, lambda_t^{log2 C + 1 + m} times the decayed
//      q_tᵀ Block_m[(j >> m) - 1] (levels above log2 C);
//   4. optional export of the bucket states at position T.
// Decays are exponentials of differences of non-positive log sums, never ratios.
#include <cuda_runtime.h>

#include "ll_internal.cuh"

namespace ll {

namespace {

constexpr int kThreads = 256;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

template <typename TIn>
__global__ void __launch_bounds__(kThreads) gen_chunk_state(GenPlan p, const TIn* __restrict__ k,
                                                            const TIn* __restrict__ v,
                                                            const float* __restrict__ a, char* ws) {
  extern __shared__ __align__(16) float sm[];
  const int C = p.C, dk = p.dk, dv = p.dv;
  float* ks = sm;
  float* vs = ks + C * dk;
  float* gs = vs + C * dv;
  const int j = blockIdx.x, bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H, grp = h / p.hpg;
  const long long t0 = (long long)j * C;
  for (int e = threadIdx.x; e < C * dk; e += kThreads) {
    int s = e / dk, i = e % dk;
    ks[e] = ll_load(k, (((size_t)b * p.T + t0 + s) * p.G + grp) * dk + i);
  }
  for (int e = threadIdx.x; e < C * dv; e += kThreads) {
    int s = e / dv, jv = e % dv;
    vs[e] = ll_load(v, (((size_t)b * p.T + t0 + s) * p.H + h) * dv + jv);
  }
  if (threadIdx.x == 0) {
    float acc = 0.f;
    for (int s = 0; s < C; ++s) {
      acc += log2f(a[((size_t)b * p.T + t0 + s) * p.H + h]);
      gs[s] = acc;
    }
  }
  __syncthreads();
  float* g = reinterpret_cast<float*>(ws + p.off_g);
  float* gamma = reinterpret_cast<float*>(ws + p.off_gamma);
  float* Hst = reinterpret_cast<float*>(ws + p.off_H);
  for (int s = threadIdx.x; s < C; s += kThreads) g[(size_t)bh * p.T + t0 + s] = gs[s];
  if (threadIdx.x == 0) gamma[(size_t)bh * p.N + j] = gs[C - 1];
  const float gend = gs[C - 1];
  const int S = dk * dv;
  // H_j = Kᵀ diag(2^(gend - g)) V: scale the keys once, then a tiled product
  for (int e = threadIdx.x; e < C * dk; e += kThreads) ks[e] *= exp2f(gend - gs[e / dk]);
  __syncthreads();
  float* dst = Hst + ((size_t)bh * p.N + j) * S;
  smem_mm(dk, dv, C, ks, 1, dk, vs, dv, threadIdx.x, kThreads, [&](int m0, int n0, float (&acc)[4][4]) {
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(dst + (m0 + i) * dv + n0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  });
}

__global__ void __launch_bounds__(kThreads) gen_blocks(GenPlan p, char* ws) {
  const int idx = blockIdx.x, bh = blockIdx.y;
  int m = 0;
  while (m + 1 < p.M && p.blk_off[m + 1] <= idx) ++m;
  const int i = 2 * (idx - p.blk_off[m]);
  const int u0 = i << m, u1 = u0 + (1 << m);
  const float* gamma = reinterpret_cast<const float*>(ws + p.off_gamma) + (size_t)bh * p.N;
  const float* Hst = reinterpret_cast<const float*>(ws + p.off_H);
  float* blk = reinterpret_cast<float*>(ws + p.off_blk);
  float* blkG = reinterpret_cast<float*>(ws + p.off_blkG);
  const int S = p.dk * p.dv;
  for (int e = threadIdx.x; e < S; e += kThreads) {
    float acc = 0.f, dec = 0.f;
    for (int u = u1 - 1; u >= u0; --u) {
      acc += exp2f(dec) * Hst[((size_t)bh * p.N + u) * S + e];
      dec += gamma[u];
    }
    blk[((size_t)bh * p.nblk + idx) * S + e] = acc;
  }
  if (threadIdx.x == 0) {
    float dec = 0.f;
    for (int u = u0; u < u1; ++u) dec += gamma[u];
    blkG[(size_t)bh * p.nblk + idx] = dec;
  }
}

// One CTA per (query sub-tile of QT rows of chunk j, b*h).
template <typename TIn>
__global__ void __launch_bounds__(kThreads) gen_output(GenPlan p, int QT, const TIn* __restrict__ q,
                                                       const TIn* __restrict__ k,
                                                       const TIn* __restrict__ v,
                                                       const float* __restrict__ lam, TIn* o,
                                                       const char* ws) {
  extern __shared__ float sm[];
  const int C = p.C, dk = p.dk, dv = p.dv, L = p.L;
  const int sub_per_chunk = C / QT;
  const int j = blockIdx.x / sub_per_chunk, r0 = (blockIdx.x % sub_per_chunk) * QT;
  const int bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H, grp = h / p.hpg;
  const long long t0 = (long long)j * C;
  const int ns = r0 + QT;  // keys 0 .. ns-1 of the chunk can be seen by these queries
  float* qs = sm;                // QT * dk
  float* ks = qs + QT * dk;      // ns * dk
  float* vs = ks + C * dk;       // ns * dv
  float* gs = vs + C * dv;       // C
  float* P = gs + C;             // QT * C
  float* ls = P + QT * C;        // QT * L
  const float* g = reinterpret_cast<const float*>(ws + p.off_g) + (size_t)bh * p.T + t0;
  for (int e = threadIdx.x; e < QT * dk; e += kThreads) {
    int r = e / dk, i = e % dk;
    qs[e] = ll_load(q, (((size_t)b * p.T + t0 + r0 + r) * p.G + grp) * dk + i);
  }
  for (int e = threadIdx.x; e < ns * dk; e += kThreads) {
    int s = e / dk, i = e % dk;
    ks[e] = ll_load(k, (((size_t)b * p.T + t0 + s) * p.G + grp) * dk + i);
  }
  for (int e = threadIdx.x; e < ns * dv; e += kThreads) {
    int s = e / dv, jv = e % dv;
    vs[e] = ll_load(v, (((size_t)b * p.T + t0 + s) * p.H + h) * dv + jv);
  }
  for (int s = threadIdx.x; s < C; s += kThreads) gs[s] = g[s];
  for (int e = threadIdx.x; e < QT * L; e += kThreads) {
    int r = e / L, l = e % L;
    ls[e] = lam[(((size_t)b * p.T + t0 + r0 + r) * p.H + h) * L + l];
  }
  __syncthreads();
  // intra-chunk scores: levels 0 .. log2 C (t xor s < C inside an aligned chunk)
  for (int e = threadIdx.x; e < QT * C; e += kThreads) {
    int r = e / C, s = e % C, t = r0 + r;
    float val = 0.f;
    if (s <= t) {
      float dot = 0.f;
      for (int i = 0; i < dk; ++i) dot += qs[r * dk + i] * ks[s * dk + i];
      int lvl = bit_length(t ^ s);
      val = ls[r * L + lvl] * exp2f(gs[t] - gs[s]) * dot;
    }
    P[e] = val;
  }
  __syncthreads();
  const float* blk = reinterpret_cast<const float*>(ws + p.off_blk);
  const float* blkG = reinterpret_cast<const float*>(ws + p.off_blkG) + (size_t)bh * p.nblk;
  const int S = dk * dv;
  for (int e = threadIdx.x; e < QT * dv; e += kThreads) {
    int r = e / dv, jv = e % dv, t = r0 + r;
    float acc = 0.f;
    for (int s = 0; s <= t; ++s) acc += P[r * C + s] * vs[s * dv + jv];
    // inter-chunk levels: one Fenwick block per set bit of j, nearest first
    float D = 0.f;
    for (int m = 0; (j >> m) > 0; ++m) {
      if (!((j >> m) & 1)) continue;
      int bidx = p.blk_off[m] + (((j >> m) - 1) >> 1);
      const float* B = blk + ((size_t)bh * p.nblk + bidx) * S;
      float w = ls[r * L + p.clog + 1 + m] * exp2f(gs[t] + D);
      float dot = 0.f;
      for (int i = 0; i < dk; ++i) dot += qs[r * dk + i] * B[i * dv + jv];
      acc += w * dot;
      D += blkG[bidx];
    }
    // continuation: the live levels of the start position, whose memories lie before every
    // chunk of the segment (D now spans the chunks 0 .. j-1) and carry their own log-scale
    for (int ip = 0; ip < p.npre; ++ip) {
      const int lv = p.prelev[ip];
      const float* Sp = p.pre_st + ((size_t)bh * p.Lp + lv) * S;
      const float w = ls[r * L + lv] * exp2f(gs[t] + D + p.pre_lsc[(size_t)bh * p.Lp + lv] * 1.4426950408889634f);
      float dot = 0.f;
      for (int i = 0; i < dk; ++i) dot += qs[r * dk + i] * Sp[i * dv + jv];
      acc += w * dot;
    }
    ll_store(o, (((size_t)b * p.T + t0 + t) * p.H + h) * dv + jv, acc);
  }
}

// Bucket states at position T: level l >= 1 is live when bit l-1 of T is set; since
// T % C == 0 these are chunk levels m = l - 1 - log2 C of the chunk count N.
__global__ void __launch_bounds__(kThreads) gen_export(GenPlan p, int SL, const char* ws, float* st,
                                                       float* lsc) {
  const int lvl = blockIdx.x, bh = blockIdx.y;
  const int S = p.dk * p.dv;
  float* dst = st + ((size_t)bh * SL + lvl) * S;
  bool live = lvl >= 1 && ((((long long)p.T) >> (lvl - 1)) & 1);
  float scale = 0.f;
  const float* src = nullptr;
  if (live) {
    const int m = lvl - 1 - p.clog;
    const float* blkG = reinterpret_cast<const float*>(ws + p.off_blkG) + (size_t)bh * p.nblk;
    float D = 0.f;
    for (int mm = 0; mm < m; ++mm)
      if ((p.N >> mm) & 1) D += blkG[p.blk_off[mm] + (((p.N >> mm) - 1) >> 1)];
    scale = exp2f(D);
    int bidx = p.blk_off[m] + (((p.N >> m) - 1) >> 1);
    src = reinterpret_cast<const float*>(ws + p.off_blk) + ((size_t)bh * p.nblk + bidx) * S;
  }
  for (int e = threadIdx.x; e < S; e += kThreads) dst[e] = live ? scale * src[e] : 0.f;
  if (lsc && threadIdx.x == 0) lsc[(size_t)bh * SL + lvl] = 0.f;
}

template <typename TIn>
cudaError_t run(const GenPlan& p0, const FwdArgs& a, cudaStream_t st, bool states_only = false,
                bool export_only = false) {
  GenPlan p = p0;
  p.npre = 0;
  if (a.T0 > 0) {  // continuation: the live levels of the start position
    for (int l = 1; l <= 62 && p.npre < 32; ++l)
      if ((a.T0 >> (l - 1)) & 1) p.prelev[p.npre++] = l;
    p.Lp = a.pre_levels;
    p.pre_st = a.pre_st;
    p.pre_lsc = a.pre_lsc;
  }
  const int BH = p.B * p.H;
  size_t sm1 = sizeof(float) * ((size_t)p.C * p.dk + (size_t)p.C * p.dv + p.C);
  cudaError_t e = cudaFuncSetAttribute(gen_chunk_state<TIn>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
  if (e != cudaSuccess) return e;
  gen_chunk_state<TIn><<<dim3(p.N, BH), kThreads, sm1, st>>>(
      p, static_cast<const TIn*>(a.k), static_cast<const TIn*>(a.v), a.a, a.ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch(a, 0, st);
  gen_blocks<<<dim3(p.nblk, BH), kThreads, 0, st>>>(p, a.ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch(a, 1, st);
  if (states_only) return cudaSuccess;
  if (export_only) {
    if (!a.states_out) return cudaErrorInvalidValue;
    gen_export<<<dim3(a.state_levels, BH), kThreads, 0, st>>>(p, a.state_levels, a.ws, a.states_out,
                                                             a.logscale_out);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launch();
    return cudaSuccess;
  }
  const int QT = p.C < 32 ? p.C : 32;
  size_t sm3 = sizeof(float) * ((size_t)QT * p.dk + (size_t)p.C * p.dk + (size_t)p.C * p.dv + p.C +
                                (size_t)QT * p.C + (size_t)QT * p.L);
  e = cudaFuncSetAttribute(gen_output<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3);
  if (e != cudaSuccess) return e;
  gen_output<TIn><<<dim3(p.N * (p.C / QT), BH), kThreads, sm3, st>>>(
      p, QT, static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k),
      static_cast<const TIn*>(a.v), a.lam, static_cast<TIn*>(a.o), a.ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch(a, 2, st);
  if (a.states_out) {
    gen_export<<<dim3(a.state_levels, BH), kThreads, 0, st>>>(p, a.state_levels, a.ws, a.states_out,
                                                             a.logscale_out);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launch(a, 3, st);
  }
  return cudaSuccess;
}

}  // namespace

bool make_gen_plan(const ll_shape& s, GenPlan* p) {
  p->B = s.batch;
  p->T = s.T;
  p->H = s.heads;
  p->hpg = s.heads_per_group;
  p->G = s.heads / s.heads_per_group;
  p->dk = s.d_k;
  p->dv = s.d_v;
  p->C = s.chunk;
  p->clog = bit_length(s.chunk) - 1;
  p->L = s.levels;
  p->N = s.T / s.chunk;
  p->M = bit_length(p->N);
  if (p->M > 31) return false;
  int off = 0;
  for (int m = 0; m < p->M; ++m) {
    p->blk_off[m] = off;
    off += ((p->N >> m) + 1) / 2;
  }
  p->nblk = off;
  const size_t BH = (size_t)p->B * p->H;
  const size_t S = (size_t)p->dk * p->dv;
  size_t o = 0;
  p->off_g = o;
  o = align256(o + sizeof(float) * BH * p->T);
  p->off_gamma = o;
  o = align256(o + sizeof(float) * BH * p->N);
  p->off_H = o;
  o = align256(o + sizeof(float) * BH * p->N * S);
  p->off_blk = o;
  o = align256(o + sizeof(float) * BH * p->nblk * S);
  p->off_blkG = o;
  o = align256(o + sizeof(float) * BH * p->nblk);
  p->bytes = o;
  p->npre = 0;
  p->Lp = 0;
  p->pre_st = nullptr;
  p->pre_lsc = nullptr;
  return true;
}

cudaError_t launch_generic_fwd(const GenPlan& p, bool bf16, const FwdArgs& a, cudaStream_t st) {
  return bf16 ? run<__nv_bfloat16>(p, a, st) : run<float>(p, a, st);
}

cudaError_t launch_generic_states(const GenPlan& p, bool bf16, const FwdArgs& a, cudaStream_t st) {
  return bf16 ? run<__nv_bfloat16>(p, a, st, true) : run<float>(p, a, st, true);
}

cudaError_t launch_generic_export_only(const GenPlan& p, bool bf16, const FwdArgs& a, cudaStream_t st) {
  return bf16 ? run<__nv_bfloat16>(p, a, st, false, true) : run<float>(p, a, st, false, true);
}

}  // namespace ll
