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
// Chunked as in the delta rule's WY/UT form.  Within a chunk (C <= 64 tokens, g the
// chunk-local log2 decay cumsum, S the d_k x d_v state at the chunk's start):
//   u = T diag(beta) (V - diag(2^g) K S) = U_loc - W S,
//   T = (I + diag(beta) A)^-1,  A = (K Kᵀ) ⊙ 2^(g_t - g_s) strictly lower,
//   U_loc = T diag(beta) V,  W = T diag(beta 2^g) K.
//   gdn_local (every chunk at once): X = [U_loc | W] by forward substitution, each thread
//              owning one column (no barrier inside the solve);
//   gdn_pass   (one CTA per (b, h), chunks in order): u = U_loc - W S, written in the
//              input dtype, then S <- 2^(g_end) S + (2^(g_end - g) K)ᵀ u.
#include <cuda_runtime.h>

#include "ll_internal.cuh"
#include "ptx.cuh"

namespace ll {

namespace {

constexpr int kG = 256;  // threads per CTA

// Bounded wait for a bulk copy (2 s of %globaltimer), false when it ran out.
__device__ __forceinline__ bool bulk_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer_ns() - t0 > 2000000000ull) return false;
  return true;
}

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

template <typename TIn>
__global__ void __launch_bounds__(kG) gdn_local(int T, int H, int hpg, int dk, int dv, int C,
                                                const TIn* __restrict__ k, const TIn* __restrict__ v,
                                                const float* __restrict__ a, const float* __restrict__ beta,
                                                float* __restrict__ xg) {
  extern __shared__ __align__(16) float sm[];
  const int c = blockIdx.x, bh = blockIdx.y, b = bh / H, h = bh % H, G = H / hpg, grp = h / hpg;
  const int tid = threadIdx.x, nc = dv + dk;
  const long long t0 = (long long)c * C;
  const int CP = C + 4;        // padded row of a transposed tile (16-byte rows, 4-way banks)
  float* KT = sm;              // dk x C (row stride CP)
  float* A = KT + dk * CP;     // C x C
  float* X = A + C * C;        // C x (dv + dk)
  float* gs = X + C * nc;      // C
  float* bs = gs + C;          // C
  chunk_decay(tid, C, a, beta, ((size_t)b * T + t0) * H + h, H, gs, bs);
  for (int e = tid; e < C * dk; e += kG) {
    const int s = e / dk, i = e % dk;
    KT[i * CP + s] = ll_load(k, (((size_t)b * T + t0 + s) * G + grp) * dk + i);
  }
  __syncthreads();
  for (int e = tid; e < C * dv; e += kG) {
    const int s = e / dv, j = e % dv;
    X[s * nc + j] = bs[s] * ll_load(v, (((size_t)b * T + t0 + s) * H + h) * dv + j);
  }
  for (int e = tid; e < C * dk; e += kG) {
    const int s = e / dk, i = e % dk;
    X[s * nc + dv + i] = bs[s] * exp2f(gs[s]) * KT[i * CP + s];
  }
  smem_mm(C, C, dk, KT, 1, CP, KT, CP, tid, kG, [&](int m0, int n0, float (&acc)[4][4]) {
    for (int i = 0; i < 4; ++i)
      for (int j = 0; j < 4; ++j) {
        const int t = m0 + i, s = n0 + j;
        A[t * C + s] = s < t ? bs[t] * exp2f(gs[t] - gs[s]) * acc[i][j] : 0.f;  // diag(beta) A
      }
  });
  __syncthreads();
  // (I + diag(beta) A) X = X0 by blocks of 16 rows: the rows before a block enter by one
  // tiled product, X_blk -= L_blk,<blk X_<blk; then inside the block each thread owns a
  // column and substitutes over the block's earlier rows (at most 15).
  for (int r0 = 0; r0 < C; r0 += 16) {
    const int nb = C - r0 < 16 ? C - r0 : 16;
    if (r0 > 0)
      smem_mm(nb, nc, r0, A + r0 * C, C, 1, X, nc, tid, kG, [&](int m0, int n0, float (&acc)[4][4]) {
        for (int i = 0; i < 4; ++i)
          for (int j = 0; j < 4; ++j) X[(r0 + m0 + i) * nc + n0 + j] -= acc[i][j];
      });
    __syncthreads();
    for (int col = tid; col < nc; col += kG)
      for (int t = r0 + 1; t < r0 + nb; ++t) {
        float acc = 0.f;
        for (int s = r0; s < t; ++s) acc += A[t * C + s] * X[s * nc + col];
        X[t * nc + col] -= acc;
      }
    __syncthreads();
  }
  float* dst = xg + ((size_t)bh * (T / C) + c) * (size_t)C * nc;
  for (int e = tid; e < C * nc; e += kG) dst[e] = X[e];
}

template <typename TIn>
__global__ void __launch_bounds__(kG) gdn_pass(int T, int H, int hpg, int dk, int dv, int C,
                                               const TIn* __restrict__ k, const float* __restrict__ a,
                                               const float* __restrict__ xg, TIn* __restrict__ u,
                                               unsigned* status) {
  extern __shared__ __align__(16) float sm[];
  const int bh = blockIdx.x, b = bh / H, h = bh % H, G = H / hpg, grp = h / hpg;
  const int tid = threadIdx.x, nc = dv + dk;
  const int CP = C;            // row stride of the transposed tile (unpadded: two CTAs per SM)
  float* X = sm;               // C x (dv + dk): [U_loc | W] of the chunk, U_loc then u in place
  float* KT = X + C * nc;      // dk x C, scaled by 2^(g_end - g_s)
  float* Sm = KT + dk * CP;    // dk x dv: the state
  float* gs = Sm + dk * dv;    // C
  __shared__ __align__(8) uint64_t bar;
  if (tid == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  for (int e = tid; e < dk * dv; e += kG) Sm[e] = 0.f;
  const int n = T / C;
  const uint32_t xbytes = (uint32_t)(C * nc * sizeof(float));
  bool ok = true;
  for (int c = 0; c < n && ok; ++c) {
    const long long t0 = (long long)c * C;
    __syncthreads();  // the previous chunk is done with every buffer
    if (tid == 0) {   // the chunk's [U_loc | W] in one bulk copy
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive_expect_tx(&bar, xbytes);
      ptx::bulk_load(X, xg + ((size_t)bh * n + c) * (size_t)C * nc, xbytes, &bar);
    }
    chunk_decay(tid, C, a, nullptr, ((size_t)b * T + t0) * H + h, H, gs, nullptr);
    for (int e = tid; e < C * dk; e += kG) {
      const int s = e / dk, i = e % dk;
      KT[i * CP + s] = ll_load(k, (((size_t)b * T + t0 + s) * G + grp) * dk + i);
    }
    ok = bulk_wait(&bar, c & 1);
    if (!ok && tid == 0) atomicExch(status, kStatusTimeout);
    ok = __syncthreads_and(ok);
    if (!ok) break;
    // u = U_loc - W S, written out
    smem_mm(C, dv, dk, X + dv, nc, 1, Sm, dv, tid, kG, [&](int m0, int n0, float (&acc)[4][4]) {
      for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 4; ++j) {
          const int s = m0 + i, jj = n0 + j;
          const float val = X[s * nc + jj] - acc[i][j];
          X[s * nc + jj] = val;
          ll_store(u, (((size_t)b * T + t0 + s) * H + h) * dv + jj, val);
        }
    });
    const float gend = gs[C - 1];
    for (int e = tid; e < dk * C; e += kG) KT[(e / C) * CP + e % C] *= exp2f(gend - gs[e % C]);
    __syncthreads();
    // S <- 2^(g_end) S + (2^(g_end - g) K)ᵀ u
    const float dS = exp2f(gend);
    smem_mm(dk, dv, C, KT, CP, 1, X, nc, tid, kG, [&](int m0, int n0, float (&acc)[4][4]) {
      for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 4; ++j) {
          float* sp = Sm + (m0 + i) * dv + n0 + j;
          *sp = dS * *sp + acc[i][j];
        }
    });
  }
  if (!ok && tid == 0) bulk_wait(&bar, 0) || bulk_wait(&bar, 1);  // bounded: let the copy land
}

}  // namespace

size_t gdn_values_bytes(const ll_shape& s) {
  const size_t e = s.dtype == LL_BF16 ? 2 : 4;
  const size_t ub = (((size_t)s.batch * s.T * s.heads * s.d_v * e) + 255) & ~size_t(255);
  const size_t xb = (size_t)s.batch * s.T * s.heads * (s.d_v + s.d_k) * sizeof(float);
  return ub + ((xb + 255) & ~size_t(255));
}

namespace {
template <typename TIn>
cudaError_t run_gdn(const ll_shape& s, const void* k, const void* v, const float* a, const float* beta,
                    void* u, unsigned* status, cudaStream_t st) {
  const int C = s.chunk < 64 ? s.chunk : 64;  // divides T, since chunk does
  const size_t ub = (((size_t)s.batch * s.T * s.heads * s.d_v * (s.dtype == LL_BF16 ? 2 : 4)) + 255) &
                    ~size_t(255);
  float* xg = reinterpret_cast<float*>(static_cast<char*>(u) + ub);
  const int dk = s.d_k, dv = s.d_v, BH = s.batch * s.heads;
  const size_t sm1 = sizeof(float) * ((size_t)dk * (C + 4) + (size_t)C * C + (size_t)C * (dv + dk) + 2 * C);
  cudaError_t e = cudaFuncSetAttribute(gdn_local<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
  if (e != cudaSuccess) return e;
  gdn_local<TIn><<<dim3(s.T / C, BH), kG, sm1, st>>>(s.T, s.heads, s.heads_per_group, dk, dv, C,
                                                      static_cast<const TIn*>(k), static_cast<const TIn*>(v), a,
                                                      beta, xg);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  const size_t sm2 = sizeof(float) * ((size_t)C * (dv + dk) + (size_t)dk * C + (size_t)dk * dv + C);
  if ((e = cudaFuncSetAttribute(gdn_pass<TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)) !=
      cudaSuccess)
    return e;
  gdn_pass<TIn><<<BH, kG, sm2, st>>>(s.T, s.heads, s.heads_per_group, dk, dv, C, static_cast<const TIn*>(k), a,
                                     xg, static_cast<TIn*>(u), status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_gdn_values(const ll_shape& s, const void* k, const void* v, const float* a,
                              const float* beta, void* u, unsigned* status, cudaStream_t st) {
  return s.dtype == LL_BF16 ? run_gdn<__nv_bfloat16>(s, k, v, a, beta, u, status, st)
                            : run_gdn<float>(s, k, v, a, beta, u, status, st);
}

}  // namespace ll
