// Sequence segments: the pieces that let a forward start at a position T0 > 0 from the
// bucket memories there, and that build those memories from the memories of whole
// earlier segments (one exchange between ranks that each hold one segment).
//
// Log-linear attention write-up (https://www.yoousoft.com/industry/3746.html): each
// position keeps one memory per bucket of the Fenwick partition of its prefix (section
// 特殊结构：树划分, Fig. 2), and the memories of larger buckets are decayed sums of the
// memories of the pieces inside them (section 高效训练算法, Algorithm 1).  With T0 a
// multiple of a power of two P >= T, the buckets of every position T0 + t (t < T) are
// the buckets of T0 plus the segment's own buckets, so the forward over the segment is
// the ordinary forward plus one term per live level of T0.
//
// Memories are fp32 (d_k, d_v) blocks; a memory with log-scale c stands for
// exp(c) * block, as in the decode step.  All kernels here are bandwidth-bound and
// stream float4s; one CTA covers a whole memory where it writes a log-scale, so that a
// log-scale slot is read and written by the same CTA.
#include <cuda_runtime.h>

#include "ll_internal.cuh"

namespace ll {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int nth_bit(unsigned long long x, int i) {
  for (int j = 0; j < i; ++j) x &= x - 1;
  return __ffsll((long long)x) - 1;
}

// out[b, h] = sum over t of ln a[b, t, h], accumulated in fp64.  One CTA per (b, block of
// 32 heads): lane = head, warp w takes the tokens t = w, w + 8, ... (coalesced rows).
__global__ void __launch_bounds__(kThreads) seg_logdecay_kernel(const float* __restrict__ a, int T, int H,
                                                                float* __restrict__ out) {
  __shared__ double part[kThreads / 32][32];
  const int b = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.y * 32 + lane;
  double acc = 0.0;
  if (h < H)
    for (int t = warp; t < T; t += kThreads / 32) acc += (double)logf(a[((size_t)b * T + t) * H + h]);
  part[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && h < H) {
    double s = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) s += part[w][lane];
    out[(size_t)b * H + h] = (float)s;
  }
}

// total[bh] = sum of the memories of the levels live at position T (bit l-1 of T set)
// in st (BH, SL, S); the memories there carry no log-scale.
__global__ void __launch_bounds__(kThreads) sum_live_levels_kernel(const float* __restrict__ st, int SL,
                                                                   long long T, int S4,
                                                                   float* __restrict__ total) {
  const int bh = blockIdx.x;
  const float4* src = reinterpret_cast<const float4*>(st) + (size_t)bh * SL * S4;
  float4* dst = reinterpret_cast<float4*>(total) + (size_t)bh * S4;
  for (int e = blockIdx.y * kThreads + threadIdx.x; e < S4; e += gridDim.y * kThreads) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int l = 1; l < SL; ++l) {
      if (!((T >> (l - 1)) & 1)) continue;
      const float4 x = src[(size_t)l * S4 + e];
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
    dst[e] = acc;
  }
}

// The bucket memories at T0 = r * 2^seg_log from the memories of the r segments before
// it (seg_st (r, BH, S), seg_g (r, BH) their summed ln-decays).  The bucket of set bit j
// of r is made of the segments [(r >> (j+1)) << (j+1), that + 2^j), it has level
// j + 1 + seg_log, and each of its segments counts decayed by the segments after it
// and before T0.  One CTA per (bh, live level); the log-scale of a written level is 0.
__global__ void __launch_bounds__(kThreads) prefix_from_segments_kernel(
    int r, int seg_log, int BH, const float* __restrict__ seg_st, const float* __restrict__ seg_g, int S4,
    float* __restrict__ st, float* __restrict__ lsc, int SL) {
  constexpr int kMaxSeg = 64;
  __shared__ float w[kMaxSeg];
  const int bh = blockIdx.x;
  const int j = nth_bit((unsigned long long)r, blockIdx.y);
  const int s0 = (r >> (j + 1)) << (j + 1), s1 = s0 + (1 << j);
  const int level = j + 1 + seg_log;
  if (threadIdx.x == 0) {
    double g = 0.0;
    for (int s = r - 1; s >= s0; --s) {  // g = summed ln-decay of the segments after s
      if (s < s1) w[s - s0] = (float)exp(g);
      g += (double)seg_g[(size_t)s * BH + bh];
    }
  }
  __syncthreads();
  float4* dst = reinterpret_cast<float4*>(st) + ((size_t)bh * SL + level) * S4;
  for (int e = threadIdx.x; e < S4; e += kThreads) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = s0; s < s1; ++s) {
      const float4 x = reinterpret_cast<const float4*>(seg_st)[((size_t)s * BH + bh) * S4 + e];
      const float ws = w[s - s0];
      acc.x += ws * x.x;
      acc.y += ws * x.y;
      acc.z += ws * x.z;
      acc.w += ws * x.w;
    }
    dst[e] = acc;
  }
  if (lsc && threadIdx.x == 0) lsc[(size_t)bh * SL + level] = 0.f;
}

// Bucket memories at E = T0 + T: every bucket of E is made of whole buckets of T0
// (memories pst with log-scales plsc, decayed to T0 - 1, so they take the segment's
// decay segg on top) and whole buckets of the segment (its own export at local
// position T, loc (BH, SLloc, S), already decayed to E - 1).  One CTA per (bh, level
// live at E); the CTA reads every input element before it writes that element, and the
// prefix levels it reads belong to no other CTA, so st may be pst (and lsc plsc).
__global__ void __launch_bounds__(kThreads) continue_export_kernel(
    long long T0, long long T, const float* pst, const float* plsc, int Lp, const float* __restrict__ loc,
    int SLloc, const float* __restrict__ segg, int S4, float* st, float* lsc, int SL) {
  __shared__ float wp[64];
  __shared__ unsigned long long use_loc;
  const int bh = blockIdx.x;
  const long long E = T0 + T;
  const int l = nth_bit((unsigned long long)E, blockIdx.y) + 1;
  const long long lo = (E >> l) << l, hi = lo + (1LL << (l - 1));
  if (threadIdx.x < 64) {
    const int i = threadIdx.x;
    float wi = 0.f;
    if (i >= 1 && i < Lp && ((T0 >> (i - 1)) & 1)) {
      const long long plo = (T0 >> i) << i, phi = plo + (1LL << (i - 1));
      if (plo >= lo && phi <= hi) wi = expf(plsc[(size_t)bh * Lp + i] + segg[bh]);
    }
    wp[i] = wi;
  }
  if (threadIdx.x == 0) {
    unsigned long long m = 0;
    for (int k = 1; k < SLloc && k < 64; ++k) {
      if (!((T >> (k - 1)) & 1)) continue;
      const long long klo = T0 + ((T >> k) << k), khi = klo + (1LL << (k - 1));
      if (klo >= lo && khi <= hi) m |= 1ull << k;
    }
    use_loc = m;
  }
  __syncthreads();
  const unsigned long long mloc = use_loc;
  const float4* p4 = reinterpret_cast<const float4*>(pst) + (size_t)bh * Lp * S4;
  const float4* l4 = reinterpret_cast<const float4*>(loc) + (size_t)bh * SLloc * S4;
  float4* dst = reinterpret_cast<float4*>(st) + ((size_t)bh * SL + l) * S4;
  for (int e = threadIdx.x; e < S4; e += kThreads) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 1; i < Lp && i < 64; ++i) {
      const float wi = wp[i];
      if (wi == 0.f) continue;
      const float4 x = p4[(size_t)i * S4 + e];
      acc.x += wi * x.x;
      acc.y += wi * x.y;
      acc.z += wi * x.z;
      acc.w += wi * x.w;
    }
    for (unsigned long long m = mloc; m; m &= m - 1) {
      const int k = __ffsll((long long)m) - 1;
      const float4 x = l4[(size_t)k * S4 + e];
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
    dst[e] = acc;
  }
  __syncthreads();  // every read of plsc in this CTA came before the write below
  if (lsc && threadIdx.x == 0) lsc[(size_t)bh * SL + l] = 0.f;
}

int popcount64(unsigned long long x) { return __builtin_popcountll(x); }

}  // namespace

cudaError_t launch_seg_logdecay(const float* a, int B, int T, int H, float* out, cudaStream_t st) {
  seg_logdecay_kernel<<<dim3(B, (H + 31) / 32), kThreads, 0, st>>>(a, T, H, out);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

cudaError_t launch_sum_live_levels(const float* stl, int BH, int SL, long long T, int S, float* total,
                                   cudaStream_t st) {
  const int S4 = S / 4;
  sum_live_levels_kernel<<<dim3(BH, (S4 + kThreads - 1) / kThreads), kThreads, 0, st>>>(stl, SL, T, S4, total);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

cudaError_t launch_prefix_from_segments(int r, int seg_log, int BH, const float* seg_st, const float* seg_g,
                                        int S, float* stl, float* lsc, int SL, cudaStream_t st) {
  if (r <= 0) return cudaSuccess;
  if (r > 64) return cudaErrorInvalidValue;
  prefix_from_segments_kernel<<<dim3(BH, popcount64((unsigned long long)r)), kThreads, 0, st>>>(
      r, seg_log, BH, seg_st, seg_g, S / 4, stl, lsc, SL);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

cudaError_t launch_continue_export(long long T0, long long T, int BH, const float* pst, const float* plsc, int Lp,
                                   const float* loc, int SLloc, const float* segg, int S, float* stl, float* lsc,
                                   int SL, cudaStream_t st) {
  if (Lp > 64 || SLloc > 64) return cudaErrorInvalidValue;
  continue_export_kernel<<<dim3(BH, popcount64((unsigned long long)(T0 + T))), kThreads, 0, st>>>(
      T0, T, pst, plsc, Lp, loc, SLloc, segg, S / 4, stl, lsc, SL);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace ll
