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
// gdn_values: one CTA per (b, h) walks the chunks (C <= 64 tokens) in order, holding the
// d_k x d_v state in shared memory.  Per chunk, with g the chunk-local log2 decay cumsum:
//   R   = V - diag(2^g) K S            (the start state's part of a_t S_{t-1} k_t)
//   A   = (K Kᵀ) ⊙ 2^(g_t - g_s) for s < t
//   u_t = beta_t (R_t - sum_{s<t} A_ts u_s)   (forward substitution, in token order)
//   S  <- 2^(g_end) S + sum_s 2^(g_end - g_s) k_s u_sᵀ
#include <cuda_runtime.h>

#include "ll_internal.cuh"

namespace ll {

namespace {

constexpr int kG = 256;  // threads per CTA

template <typename TIn>
__global__ void __launch_bounds__(kG) gdn_values(int B, int T, int H, int hpg, int dk, int dv, int C,
                                                 const TIn* __restrict__ k, const TIn* __restrict__ v,
                                                 const float* __restrict__ a,
                                                 const float* __restrict__ beta, TIn* __restrict__ u) {
  extern __shared__ __align__(16) float sm[];
  const int bh = blockIdx.x, b = bh / H, h = bh % H, G = H / hpg, grp = h / hpg;
  const int tid = threadIdx.x;
  float* KT = sm;              // dk x C   (Kᵀ of the chunk; scaled in place for the update)
  float* R = KT + dk * C;      // C x dv   (R, then read by the substitution)
  float* U = R + C * dv;       // C x dv   (u of the chunk)
  float* Sm = U + C * dv;      // dk x dv  (the state)
  float* A = Sm + dk * dv;     // C x C
  float* gs = A + C * C;       // C: chunk-local log2 decay cumsum
  float* bs = gs + C;          // C: beta
  for (int e = tid; e < dk * dv; e += kG) Sm[e] = 0.f;
  const int n = T / C;
  for (int c = 0; c < n; ++c) {
    const long long t0 = (long long)c * C;
    __syncthreads();  // the previous chunk is done with every buffer
    for (int e = tid; e < C * dk; e += kG) {
      const int s = e / dk, i = e % dk;
      KT[i * C + s] = ll_load(k, (((size_t)b * T + t0 + s) * G + grp) * dk + i);
    }
    for (int e = tid; e < C * dv; e += kG) {
      const int s = e / dv, j = e % dv;
      R[e] = ll_load(v, (((size_t)b * T + t0 + s) * H + h) * dv + j);
    }
    if (tid < 32) {  // one warp: inclusive log2 cumsum over the chunk, beta
      float carry = 0.f;
      for (int s0 = 0; s0 < C; s0 += 32) {
        const int s = s0 + tid;
        float x = s < C ? log2f(a[((size_t)b * T + t0 + s) * H + h]) : 0.f;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, x, off);
          if (tid >= off) x += y;
        }
        if (s < C) {
          gs[s] = x + carry;
          bs[s] = beta[((size_t)b * T + t0 + s) * H + h];
        }
        carry += __shfl_sync(0xffffffffu, x, 31);
      }
    }
    __syncthreads();
    // R = V - diag(2^g) K S ;  A = (K Kᵀ) ⊙ 2^(g_t - g_s), strictly lower
    smem_mm(C, dv, dk, KT, 1, C, Sm, dv, tid, kG, [&](int m0, int n0, float (&acc)[4][4]) {
      for (int i = 0; i < 4; ++i) {
        const float w = exp2f(gs[m0 + i]);
        for (int j = 0; j < 4; ++j) R[(m0 + i) * dv + n0 + j] -= w * acc[i][j];
      }
    });
    smem_mm(C, C, dk, KT, 1, C, KT, C, tid, kG, [&](int m0, int n0, float (&acc)[4][4]) {
      for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 4; ++j) {
          const int t = m0 + i, s = n0 + j;
          A[t * C + s] = s < t ? exp2f(gs[t] - gs[s]) * acc[i][j] : 0.f;
        }
    });
    __syncthreads();
    // forward substitution: thread (j, part) sums every 4th earlier token for column j
    for (int t = 0; t < C; ++t) {
      const int j = tid >> 2, part = tid & 3;
      float acc = 0.f;
      if (j < dv)
        for (int s = part; s < t; s += 4) acc += A[t * C + s] * U[s * dv + j];
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (j < dv && part == 0) U[t * dv + j] = bs[t] * (R[t * dv + j] - acc);  // d_v <= 64
      __syncthreads();
    }
    // u out; state update S <- 2^(g_end) S + sum_s 2^(g_end - g_s) k_s u_sᵀ
    for (int e = tid; e < C * dv; e += kG) {
      const int s = e / dv, j = e % dv;
      ll_store(u, (((size_t)b * T + t0 + s) * H + h) * dv + j, U[e]);
    }
    const float gend = gs[C - 1];
    for (int e = tid; e < dk * C; e += kG) KT[e] *= exp2f(gend - gs[e % C]);
    __syncthreads();
    const float dS = exp2f(gend);
    smem_mm(dk, dv, C, KT, C, 1, U, dv, tid, kG, [&](int m0, int n0, float (&acc)[4][4]) {
      for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 4; ++j) {
          float* s = Sm + (m0 + i) * dv + n0 + j;
          *s = dS * *s + acc[i][j];
        }
    });
  }
}

}  // namespace

size_t gdn_values_bytes(const ll_shape& s) {
  const size_t e = s.dtype == LL_BF16 ? 2 : 4;
  return (((size_t)s.batch * s.T * s.heads * s.d_v * e) + 255) & ~size_t(255);
}

cudaError_t launch_gdn_values(const ll_shape& s, const void* k, const void* v, const float* a,
                              const float* beta, void* u, cudaStream_t st) {
  const int C = s.chunk < 64 ? s.chunk : 64;  // divides T, since chunk does
  const size_t smem = sizeof(float) * ((size_t)s.d_k * C + 2 * (size_t)C * s.d_v +
                                       (size_t)s.d_k * s.d_v + (size_t)C * C + 2 * C);
  cudaError_t e;
  if (s.dtype == LL_BF16) {
    if ((e = cudaFuncSetAttribute(gdn_values<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
      return e;
    gdn_values<__nv_bfloat16><<<s.batch * s.heads, kG, smem, st>>>(
        s.batch, s.T, s.heads, s.heads_per_group, s.d_k, s.d_v, C,
        static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), a, beta,
        static_cast<__nv_bfloat16*>(u));
  } else {
    if ((e = cudaFuncSetAttribute(gdn_values<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    gdn_values<float><<<s.batch * s.heads, kG, smem, st>>>(s.batch, s.T, s.heads, s.heads_per_group, s.d_k,
                                                          s.d_v, C, static_cast<const float*>(k),
                                                          static_cast<const float*>(v), a, beta,
                                                          static_cast<float*>(u));
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

}  // namespace ll
