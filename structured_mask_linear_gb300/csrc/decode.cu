// Decode step of log-linear Mamba-2 over the Fenwick bucket states.
//
// Log-linear attention write-up (https://www.yoousoft.com/industry/3746.html),
// section 特殊结构：树划分: a query keeps one d_k x d_v memory per bucket, O(log T)
// of them, combined with data-dependent per-level weights; decoding costs O(log T)
// time and memory per token.  Per (b, h) and token position t:
//   1. the live buckets (bit l-1 of t set) decay by a_t: only their log-scale changes;
//   2. o_t = lambda^0 (q.k) v + sum_live lambda^l exp(sigma_l) qᵀ X_l;
//   3. the token and the buckets 1..m (m = trailing ones of t) merge into bucket m+1
//      of position t+1: X_{m+1} = k vᵀ + sum_{l<=m} exp(sigma_l) X_l, sigma_{m+1} = 0.
// Everything is one pass over the live states: each thread owns a fixed set of
// float4 columns of the states, reads every live level once (128-bit, coalesced),
// accumulates its output partial and its merge sum, and writes the merged level.
#include <cuda_runtime.h>

#include "ll_internal.cuh"

namespace ll {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxLevels = 64;

template <typename TIn, int DK, int DV>
__global__ void __launch_bounds__(kThreads) decode_step_kernel(DecodeArgs d) {
  constexpr int V4 = DV / 4;                       // float4 columns per state row
  constexpr int N4 = DK * V4;                      // float4 per state
  constexpr int NPT = (N4 + kThreads - 1) / kThreads;
  static_assert(kThreads % V4 == 0, "column group must be fixed per thread");
  __shared__ float qs[DK], ks[DK], vs[DV];
  __shared__ float wout[kMaxLevels], wmerge[kMaxLevels];
  __shared__ float4 red[kThreads];
  __shared__ float dots[kThreads / 32];

  const int bh = blockIdx.x;
  const int b = bh / d.H, h = bh % d.H, grp = h / d.hpg;
  const long long t = d.pos;
  const int L = d.L;
  const int tid = threadIdx.x;
  for (int i = tid; i < DK; i += kThreads) {
    qs[i] = ll_load(static_cast<const TIn*>(d.q), ((size_t)b * d.G + grp) * DK + i);
    ks[i] = ll_load(static_cast<const TIn*>(d.k), ((size_t)b * d.G + grp) * DK + i);
  }
  for (int j = tid; j < DV; j += kThreads)
    vs[j] = ll_load(static_cast<const TIn*>(d.v), ((size_t)b * d.H + h) * DV + j);
  int m = 0;
  while ((t >> m) & 1) ++m;  // trailing ones of t
  const float la = logf(d.a[(size_t)b * d.H + h]);
  float* lsc = d.logscale + (size_t)bh * L;
  const float* lam = d.lam + (size_t)bh * L;
  if (tid < L) {
    const int l = tid;
    const bool live = l >= 1 && ((t >> (l - 1)) & 1);
    const float sig = live ? lsc[l] + la : 0.f;
    const float e = live ? expf(sig) : 0.f;
    wout[l] = live ? lam[l] * e : 0.f;
    wmerge[l] = (live && l <= m) ? e : 0.f;
  }
  __syncthreads();
  // q.k for the diagonal term
  float part = 0.f;
  for (int i = tid; i < DK; i += kThreads) part += qs[i] * ks[i];
  for (int off = 16; off; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
  if ((tid & 31) == 0) dots[tid >> 5] = part;

  const int c4 = tid % V4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 mg[NPT];
#pragma unroll
  for (int r = 0; r < NPT; ++r) {
    const int e4 = tid + r * kThreads;
    const int i = e4 / V4;
    if (e4 < N4) {
      const float ki = ks[i];
      mg[r] = make_float4(ki * vs[4 * c4], ki * vs[4 * c4 + 1], ki * vs[4 * c4 + 2],
                          ki * vs[4 * c4 + 3]);
    }
  }
  float4* S4 = reinterpret_cast<float4*>(d.states) + (size_t)bh * L * N4;
  for (int l = 1; l < L; ++l) {
    if (!((t >> (l - 1)) & 1)) continue;
    const float wo = wout[l], wm = wmerge[l];
    const float4* X = S4 + (size_t)l * N4;
#pragma unroll
    for (int r = 0; r < NPT; ++r) {
      const int e4 = tid + r * kThreads;
      if (e4 < N4) {
        const float4 x = __ldcs(X + e4);
        const float qi = wo * qs[e4 / V4];
        acc.x += qi * x.x;
        acc.y += qi * x.y;
        acc.z += qi * x.z;
        acc.w += qi * x.w;
        mg[r].x += wm * x.x;
        mg[r].y += wm * x.y;
        mg[r].z += wm * x.z;
        mg[r].w += wm * x.w;
      }
    }
  }
  float4* Xn = S4 + (size_t)(m + 1) * N4;
#pragma unroll
  for (int r = 0; r < NPT; ++r) {
    const int e4 = tid + r * kThreads;
    if (e4 < N4) __stcs(Xn + e4, mg[r]);
  }
  red[tid] = acc;
  __syncthreads();
  if (tid < V4) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int u = tid; u < kThreads; u += V4) {
      s.x += red[u].x;
      s.y += red[u].y;
      s.z += red[u].z;
      s.w += red[u].w;
    }
    float dot = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) dot += dots[w];
    const float w0 = lam[0] * dot;
    TIn* o = static_cast<TIn*>(d.o) + ((size_t)b * d.H + h) * DV + 4 * tid;
    ll_store(o, 0, s.x + w0 * vs[4 * tid]);
    ll_store(o, 1, s.y + w0 * vs[4 * tid + 1]);
    ll_store(o, 2, s.z + w0 * vs[4 * tid + 2]);
    ll_store(o, 3, s.w + w0 * vs[4 * tid + 3]);
  }
  // log-scales of position t+1: decayed live levels above m+1 keep theirs, the merged
  // level starts at 0, the merged-away levels are no longer live.
  if (tid < L) {
    const int l = tid;
    const bool live = l >= 1 && ((t >> (l - 1)) & 1);
    if (l == m + 1)
      lsc[l] = 0.f;
    else if (live && l > m + 1)
      lsc[l] = lsc[l] + la;
    else if (live)
      lsc[l] = 0.f;
  }
}

template <typename TIn, int DK>
cudaError_t dispatch_dv(const DecodeArgs& d, cudaStream_t st) {
  dim3 grid(d.B * d.H);
  switch (d.dv) {
    case 16: decode_step_kernel<TIn, DK, 16><<<grid, kThreads, 0, st>>>(d); break;
    case 32: decode_step_kernel<TIn, DK, 32><<<grid, kThreads, 0, st>>>(d); break;
    case 64: decode_step_kernel<TIn, DK, 64><<<grid, kThreads, 0, st>>>(d); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

template <typename TIn>
cudaError_t dispatch_dk(const DecodeArgs& d, cudaStream_t st) {
  switch (d.dk) {
    case 16: return dispatch_dv<TIn, 16>(d, st);
    case 32: return dispatch_dv<TIn, 32>(d, st);
    case 64: return dispatch_dv<TIn, 64>(d, st);
    case 128: return dispatch_dv<TIn, 128>(d, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& d, bool bf16, cudaStream_t st) {
  if (d.L > kMaxLevels) return cudaErrorInvalidValue;
  return bf16 ? dispatch_dk<__nv_bfloat16>(d, st) : dispatch_dk<float>(d, st);
}

}  // namespace ll
