// Tensor-core (tcgen05 / TMEM / TMA) path of the log-linear Mamba-2 forward for
// bf16 q/k/v/o, d_k = 128, d_v = 64, T % 128 == 0.
//
// Chunkwise algorithm of the log-linear attention write-up
// (https://www.yoousoft.com/industry/3746.html, section 高效训练算法, Algorithm 1 / Fig. 3),
// with 128-token tiles (two 64-token chunks; the result does not depend on the chunk
// length, so the tile only decides which levels are dense inside a tile: 0..7):
//
//  tc_state   one CTA per (b, h, tile u): chunk-local log2 decay cumsum g, tile decay
//             gamma_u, tile state H_u = K_uᵀ diag(2^(gamma_u - g)) V_u on the tensor
//             cores (M = d_k, N = d_v, K = tokens).  Then the Fenwick tree over tiles is
//             built without any waiting: the CTA stores its node and climbs while it is
//             the second of two siblings to arrive (atomic counter per parent), merging
//             Node_{m+1}[i] = 2^(Gamma(right)) Node_m[2i] + Node_m[2i+1].  Even nodes also
//             get a bf16 hi/lo image in the UMMA operand layout for tc_output.
//  tc_output  one CTA per (b, h, tile u): S = Q Kᵀ on the tensor cores; for every set
//             bit m of u one MMA Y = Q · Node_m[(u >> m) - 1] whose rows are added with
//             weight lambda_t^(8+m) 2^(g_t + D_m), D_m the decay of the nearer buckets
//             (write-up section 特殊结构：树划分: one memory per bucket level); then
//             P = S ⊙ lambda^l ⊙ 2^(g_t - g_s) ⊙ [s <= t] written to shared memory and
//             O = P V.
//
// Operands the kernels form themselves (decayed V, P, node images) are stored as a bf16
// hi part plus a bf16 lo part (the rounding remainder) and multiplied by both, so the
// products keep about 16 significant bits while q, k, v enter exactly.
//  tc_export  bucket states at position T from the fp32 nodes (decode hand-off).
//
// Every mbarrier wait is bounded; a wait that runs out records LL_ERR_TIMEOUT in the
// status word and the CTA skips the rest of its work.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ll_internal.cuh"
#include "ptx.cuh"

namespace ll {

namespace {

constexpr int kTile = 128;         // tokens per tile
constexpr int kDk = 128, kDv = 64;  // supported head dims
constexpr int kLevIntra = 8;        // levels 0..7 live inside a 128-token tile
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait before giving up
constexpr int kNodeF = kDk * kDv;   // floats per fp32 node
constexpr int kImgHalf = kDk * kDv * 2;    // bytes of one bf16 d_k x d_v image
constexpr int kImgBytes = 2 * kImgHalf;    // node image: hi part then lo part

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (ptx::globaltimer_ns() - t0 > kWaitNs) return false;
  }
}

struct TcParams {
  int B, T, H, hpg, G, L, NT, nnodes, MT;
  int node_off[32];
  const float* a;
  const float* lam;
  __nv_bfloat16* o;
  float* node32;  // (B*H, nnodes, d_k, d_v)
  float* nodeG;   // (B*H, nnodes) total log2 decay of each node
  unsigned* cnt;  // (B*H, nnodes) arrival counters (zeroed before tc_state)
  uint8_t* img;   // (B*H, nnodes, 32 KB) bf16 hi/lo images of even nodes
  unsigned* status;
};

// Block-wide inclusive prefix sum over 128 threads (one value each).
__device__ __forceinline__ float block_scan128(float x, float* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    float y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  float add = 0.f;
  for (int w = 0; w < warp; ++w) add += s_warp[w];
  __syncthreads();
  return x + add;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// (a, b) -> bf16 pair hi = round(a, b) and lo = round((a, b) - hi): hi + lo carries about
// 16 significant bits, which a pair of MMAs accumulating in fp32 preserves.
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  float2 r = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(a - r.x, b - r.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

// ---------------------------------------------------------------------------------
// tc_state: tile states and the Fenwick tree over tiles.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) tc_state_kernel(const __grid_constant__ CUtensorMap mapK,
                                                       const __grid_constant__ CUtensorMap mapV,
                                                       TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;            // 32 KB: two 64-wide d_k boxes of 128 tokens (SW128)
  uint8_t* sV = smem + 32768;    // 32 KB: Ṽ hi part (the TMA box) then Ṽ lo part
  __shared__ __align__(8) uint64_t bar_ld, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ float s_warp[4];
  __shared__ float s_gamma;
  __shared__ unsigned s_flag;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int lin = blockIdx.x;
  const int h = lin % p.H;
  const int u = (lin / p.H) % p.NT;
  const int b = lin / (p.H * p.NT);
  const int g = h / p.hpg;
  const int bh = b * p.H + h;
  const long long t0 = (long long)u * kTile;

  if (tid == 0) {
    ptx::mbar_init(&bar_ld, 1);
    ptx::mbar_init(&bar_mma, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 128);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = tmem_base;

  if (tid == 0) {
    ptx::mbar_arrive_expect_tx(&bar_ld, 32768 + 16384);
    ptx::tma_load_4d(sK, &mapK, &bar_ld, 0, g, (int)t0, b);
    ptx::tma_load_4d(sK + 16384, &mapK, &bar_ld, 64, g, (int)t0, b);
    ptx::tma_load_4d(sV, &mapV, &bar_ld, 0, h, (int)t0, b);
  }
  // decay of token t0 + tid: chunk-local log2 cumsum
  const float la = log2f(p.a[((size_t)b * p.T + t0 + tid) * p.H + h]);
  const float gi = block_scan128(la, s_warp);
  if (tid == kTile - 1) s_gamma = gi;
  bool ok = wait_bar(&bar_ld, 0);
  if (!ok) atomicExch(p.status, kStatusTimeout);
  ok = __syncthreads_and(ok);
  const float gamma = s_gamma;
  if (ok) {
    // Ṽ row tid = 2^(gamma - g_tid) v_tid, split into a bf16 hi part (in place) and a
    // bf16 lo part (the rounding remainder) so that Kᵀ(Ṽhi + Ṽlo) keeps ~16 bits.  The
    // 128-byte swizzle permutes 16-byte chunks inside a row only, so rows map in place.
    const float w = exp2f(gamma - gi);
    uint4* vrow = reinterpret_cast<uint4*>(sV + tid * 128);
    uint4* vlo = reinterpret_cast<uint4*>(sV + 16384 + tid * 128);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 x = vrow[c], y;
      __nv_bfloat162* hx = reinterpret_cast<__nv_bfloat162*>(&x);
      __nv_bfloat162* hy = reinterpret_cast<__nv_bfloat162*>(&y);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 f = __bfloat1622float2(hx[e]);
        f.x *= w;
        f.y *= w;
        hx[e] = __floats2bfloat162_rn(f.x, f.y);
        float2 r = __bfloat1622float2(hx[e]);
        hy[e] = __floats2bfloat162_rn(f.x - r.x, f.y - r.y);
      }
      vrow[c] = x;
      vlo[c] = y;
    }
    ptx::fence_proxy_async_smem();
  }
  __syncthreads();
  if (ok && tid == 0) {
    ptx::tc_fence_after();
    // [Hhi | Hlo] (M = d_k 128, N = 2 x d_v, K = 128 tokens): A = Kᵀ and B = [Ṽhi | Ṽlo],
    // both MN-major; the two 64-wide N atoms of B sit 16 KB apart.
    const uint32_t idesc = ptx::idesc_bf16_f32(128, 128, 1, 1);
    const uint32_t a0 = ptx::smem_u32(sK), b0 = ptx::smem_u32(sV);
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk) {
      uint64_t da = ptx::smem_desc_sw128(a0 + kk * 2048, 16384, 1024);
      uint64_t db = ptx::smem_desc_sw128(b0 + kk * 2048, 16384, 1024);
      ptx::umma_f16(tbase, da, db, idesc, kk > 0);
    }
    ptx::umma_commit(&bar_mma);
  }
  if (ok) {
    ok = wait_bar(&bar_mma, 0);
    if (!ok) atomicExch(p.status, kStatusTimeout);
  }
  ok = __syncthreads_and(ok);
  float cur[kDv];
#pragma unroll
  for (int j = 0; j < kDv; ++j) cur[j] = 0.f;
  if (ok) {
    ptx::tc_fence_after();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float hi[32], lo[32];
      ptx::tmem_ld32(tbase + ((uint32_t)(warp * 32) << 16) + half * 32, hi);
      ptx::tmem_ld32(tbase + ((uint32_t)(warp * 32) << 16) + 64 + half * 32, lo);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) cur[half * 32 + j] = hi[j] + lo[j];
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tbase, 128);
  if (!ok) return;

  // Fenwick tree climb.  Row `tid` of every node is owned by thread tid.
  float Gcur = gamma;
  int k = 0, idx = u;
  const size_t nbase = (size_t)bh * p.nnodes;
  while (true) {
    const size_t node = nbase + p.node_off[k] + idx;
    float4* dst = reinterpret_cast<float4*>(p.node32 + node * kNodeF + tid * kDv);
#pragma unroll
    for (int c = 0; c < kDv / 4; ++c)
      dst[c] = make_float4(cur[4 * c], cur[4 * c + 1], cur[4 * c + 2], cur[4 * c + 3]);
    if ((idx & 1) == 0) {
      // bf16 image, hi part then lo part (rounding remainder): row tid (d_k index) holds
      // 64 d_v values; 16-byte chunk c sits at c ^ (tid & 7) (128-byte swizzle).
      uint8_t* img = p.img + node * kImgBytes + tid * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_bf16(cur[8 * c + 2 * e], cur[8 * c + 2 * e + 1], hw[e], lw[e]);
        *reinterpret_cast<uint4*>(img + ((c ^ (tid & 7)) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(img + kImgHalf + ((c ^ (tid & 7)) << 4)) =
            make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
    if (tid == 0) p.nodeG[node] = Gcur;
    // parent exists only if both children are complete nodes
    if ((idx >> 1) >= (p.NT >> (k + 1))) break;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_flag = atomicAdd(p.cnt + nbase + p.node_off[k + 1] + (idx >> 1), 1u);
    __syncthreads();
    const unsigned first = (s_flag == 0u);
    if (first) break;  // first of the two siblings: the other one merges
    __threadfence();
    const size_t sib = nbase + p.node_off[k] + (idx ^ 1);
    const float Gs = __ldcg(p.nodeG + sib);
    const float4* src = reinterpret_cast<const float4*>(p.node32 + sib * kNodeF + tid * kDv);
    if (idx & 1) {  // sibling is the left (earlier) block: decay it across ours
      const float d = exp2f(Gcur);
#pragma unroll
      for (int c = 0; c < kDv / 4; ++c) {
        float4 s4 = __ldcg(src + c);
        cur[4 * c] += d * s4.x;
        cur[4 * c + 1] += d * s4.y;
        cur[4 * c + 2] += d * s4.z;
        cur[4 * c + 3] += d * s4.w;
      }
    } else {  // sibling is the right block: decay ours across it
      const float d = exp2f(Gs);
#pragma unroll
      for (int c = 0; c < kDv / 4; ++c) {
        float4 s4 = __ldcg(src + c);
        cur[4 * c] = d * cur[4 * c] + s4.x;
        cur[4 * c + 1] = d * cur[4 * c + 1] + s4.y;
        cur[4 * c + 2] = d * cur[4 * c + 2] + s4.z;
        cur[4 * c + 3] = d * cur[4 * c + 3] + s4.w;
      }
    }
    Gcur += Gs;
    ++k;
    idx >>= 1;
    __syncthreads();  // s_flag is rewritten next round
  }
}

// ---------------------------------------------------------------------------------
// tc_output: level-fused inter-tile buckets, then intra-tile masked attention.
//
// Shared memory (2 CTAs per SM): R1 = Q, later the lo part of P; R2 = K, later the hi
// part of P; R3 = the current node image [hi | lo], later V.  TMEM (256 columns):
// S = Q Kᵀ in columns 0..127; Y = Q [Ehi | Elo] in 128..255, later O = P V in 128..191.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) tc_output_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                        const __grid_constant__ CUtensorMap mapK,
                                                        const __grid_constant__ CUtensorMap mapV,
                                                        TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* R1 = smem;             // 32 KB
  uint8_t* R2 = smem + 32768;     // 32 KB
  uint8_t* R3 = smem + 65536;     // 32 KB
  float* sG = reinterpret_cast<float*>(smem + 98304);    // 128 floats: g
  float* sLam = reinterpret_cast<float*>(smem + 98816);  // 128 x 9 floats: lambda^0..7
  __shared__ __align__(8) uint64_t bar_qk, bar_s, bar_e, bar_y, bar_v, bar_o;
  __shared__ uint32_t tmem_base;
  __shared__ float s_warp[4];
  __shared__ int s_ok;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int lin = blockIdx.x;
  const int h = lin % p.H;
  const int u = (lin / p.H) % p.NT;
  const int b = lin / (p.H * p.NT);
  const int g = h / p.hpg;
  const int bh = b * p.H + h;
  const long long t0 = (long long)u * kTile;
  const size_t nbase = (size_t)bh * p.nnodes;

  if (tid == 0) {
    ptx::mbar_init(&bar_qk, 1);
    ptx::mbar_init(&bar_s, 1);
    ptx::mbar_init(&bar_e, 1);
    ptx::mbar_init(&bar_y, 1);
    ptx::mbar_init(&bar_v, 1);
    ptx::mbar_init(&bar_o, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 256);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t tS = tbase, tY = tbase + 128, tO = tbase + 128;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

  const int mlow = (u == 0) ? -1 : __ffs(u) - 1;  // nearest inter-tile level, if any
  if (tid == 0) {
    ptx::mbar_arrive_expect_tx(&bar_qk, 32768 * 2);
    ptx::tma_load_4d(R1, &mapQ, &bar_qk, 0, g, (int)t0, b);
    ptx::tma_load_4d(R1 + 16384, &mapQ, &bar_qk, 64, g, (int)t0, b);
    ptx::tma_load_4d(R2, &mapK, &bar_qk, 0, g, (int)t0, b);
    ptx::tma_load_4d(R2 + 16384, &mapK, &bar_qk, 64, g, (int)t0, b);
    if (mlow >= 0) {
      const size_t node = nbase + p.node_off[mlow] + ((u >> mlow) - 1);
      ptx::mbar_arrive_expect_tx(&bar_e, kImgBytes);
      ptx::bulk_load(R3, p.img + node * kImgBytes, kImgBytes, &bar_e);
    }
  }
  const size_t row = (size_t)b * p.T + t0 + tid;  // token of this thread's query row
  const float la = log2f(p.a[row * p.H + h]);
  const float gt = block_scan128(la, s_warp);
  sG[tid] = gt;
  const float* lrow = p.lam + (row * p.H + h) * p.L;
#pragma unroll
  for (int l = 0; l < kLevIntra; ++l) sLam[tid * 9 + l] = lrow[l];
  bool ok = wait_bar(&bar_qk, 0);
  if (!ok) atomicExch(p.status, kStatusTimeout);
  ok = __syncthreads_and(ok);

  // S = Q Kᵀ (M = 128 queries, N = 128 keys, K = 128 d_k), both K-major.
  if (ok && tid == 0) {
    ptx::tc_fence_after();
    const uint32_t idesc = ptx::idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t q0 = ptx::smem_u32(R1), k0 = ptx::smem_u32(R2);
#pragma unroll
    for (int kk = 0; kk < kDk / 16; ++kk) {
      const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
      ptx::umma_f16(tS, ptx::smem_desc_sw128(q0 + off, 16, 1024),
                    ptx::smem_desc_sw128(k0 + off, 16, 1024), idesc, kk > 0);
    }
    ptx::umma_commit(&bar_s);
  }

  // inter-tile levels, nearest first: Y = Q [Ehi | Elo] (N = 128: two 64-wide MN atoms of
  // the node image, 16 KB apart), rows weighted by lambda_t^(8+m) 2^(g_t + D).
  float acc[kDv];
#pragma unroll
  for (int j = 0; j < kDv; ++j) acc[j] = 0.f;
  float D = 0.f;
  int it = 0;
  for (int m = mlow; ok && m >= 0 && m < 31 && (u >> m) > 0; ++m) {
    if (!((u >> m) & 1)) continue;
    const size_t node = nbase + p.node_off[m] + ((u >> m) - 1);
    if (tid == 0) {
      bool okw = wait_bar(&bar_e, it & 1);
      if (okw) {
        ptx::tc_fence_after();
        const uint32_t idesc = ptx::idesc_bf16_f32(128, 128, 0, 1);
        const uint32_t q0 = ptx::smem_u32(R1), e0 = ptx::smem_u32(R3);
#pragma unroll
        for (int kk = 0; kk < kDk / 16; ++kk) {
          const uint32_t offq = (kk >> 2) * 16384 + (kk & 3) * 32;
          ptx::umma_f16(tY, ptx::smem_desc_sw128(q0 + offq, 16, 1024),
                        ptx::smem_desc_sw128(e0 + kk * 2048, kImgHalf, 1024), idesc, kk > 0);
        }
        ptx::umma_commit(&bar_y);
        okw = wait_bar(&bar_y, it & 1);
      }
      if (!okw) atomicExch(p.status, kStatusTimeout);
      // next level's image (the MMA reading R3 has completed)
      int mn = m + 1;
      while (mn < 31 && (u >> mn) > 0 && !((u >> mn) & 1)) ++mn;
      if (okw && mn < 31 && (u >> mn) > 0) {
        const size_t nn = nbase + p.node_off[mn] + ((u >> mn) - 1);
        ptx::mbar_arrive_expect_tx(&bar_e, kImgBytes);
        ptx::bulk_load(R3, p.img + nn * kImgBytes, kImgBytes, &bar_e);
      }
      s_ok = okw ? 1 : 0;
    }
    __syncthreads();
    ok = s_ok != 0;
    if (!ok) break;
    ptx::tc_fence_after();
    const float w = lrow[kLevIntra + m] * exp2f(gt + D);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float yh[32], yl[32];
      ptx::tmem_ld32(tY + lane_off + half * 32, yh);
      ptx::tmem_ld32(tY + lane_off + 64 + half * 32, yl);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[half * 32 + j] += w * (yh[j] + yl[j]);
    }
    D += __ldcg(p.nodeG + node);
    ++it;
    ptx::tc_fence_before();
    __syncthreads();  // Y is rewritten by the next level's MMA
  }
  // every MMA reading Q or the node image has completed: R3 takes V
  if (ok && tid == 0) {
    ptx::mbar_arrive_expect_tx(&bar_v, 16384);
    ptx::tma_load_4d(R3, &mapV, &bar_v, 0, h, (int)t0, b);
  }
  if (ok) {
    ok = wait_bar(&bar_s, 0);
    if (!ok) atomicExch(p.status, kStatusTimeout);
  }
  ok = __syncthreads_and(ok);
  if (ok) {
    ptx::tc_fence_after();
    // P row t = tid, keys in 32-column groups; groups above the diagonal are zero.
    // hi part -> R2 (K is consumed), lo part -> R1 (Q is consumed).
    const int t = tid;
#pragma unroll 1
    for (int cg = 0; cg < 4; ++cg) {
      float sv[32];
      // tcgen05.ld is warp-collective: the whole warp loads when any lane needs it
      const bool warp_any = cg <= warp;
      if (warp_any) {
        ptx::tmem_ld32(tS + lane_off + cg * 32, sv);
        ptx::tmem_ld_wait();
      }
      uint32_t ph[16], pl[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        float v0 = 0.f, v1 = 0.f;
        const int s0 = cg * 32 + j, s1 = s0 + 1;
        if (warp_any && s0 <= t) {
          const int l0 = (s0 == t) ? 0 : 32 - __clz(t ^ s0);
          v0 = sv[j] * sLam[t * 9 + l0] * exp2f(gt - sG[s0]);
        }
        if (warp_any && s1 <= t) {
          const int l1 = (s1 == t) ? 0 : 32 - __clz(t ^ s1);
          v1 = sv[j + 1] * sLam[t * 9 + l1] * exp2f(gt - sG[s1]);
        }
        split_bf16(v0, v1, ph[j >> 1], pl[j >> 1]);
      }
      // 4 chunks of 8 keys: key block kb = cg / 2, chunk index c = (cg % 2) * 4 + qd
      const int off = (cg >> 1) * 16384 + t * 128;
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        const int c = (cg & 1) * 4 + qd;
        const int o16 = off + ((c ^ (t & 7)) << 4);
        *reinterpret_cast<uint4*>(R2 + o16) =
            make_uint4(ph[4 * qd], ph[4 * qd + 1], ph[4 * qd + 2], ph[4 * qd + 3]);
        *reinterpret_cast<uint4*>(R1 + o16) =
            make_uint4(pl[4 * qd], pl[4 * qd + 1], pl[4 * qd + 2], pl[4 * qd + 3]);
      }
    }
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  // O = (Phi + Plo) V (M = 128, N = 64, K = 128 keys): P K-major, V MN-major.
  if (ok && tid == 0) {
    bool okv = wait_bar(&bar_v, 0);
    if (okv) {
      ptx::tc_fence_after();
      const uint32_t idesc = ptx::idesc_bf16_f32(128, 64, 0, 1);
      const uint32_t ph0 = ptx::smem_u32(R2), pl0 = ptx::smem_u32(R1), v0 = ptx::smem_u32(R3);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        const uint32_t offp = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint64_t dv = ptx::smem_desc_sw128(v0 + kk * 2048, 1024, 1024);
        ptx::umma_f16(tO, ptx::smem_desc_sw128(ph0 + offp, 16, 1024), dv, idesc, kk > 0);
        ptx::umma_f16(tO, ptx::smem_desc_sw128(pl0 + offp, 16, 1024), dv, idesc, 1);
      }
      ptx::umma_commit(&bar_o);
    } else {
      atomicExch(p.status, kStatusTimeout);
    }
    s_ok = okv ? 1 : 0;
  }
  __syncthreads();
  if (ok) ok = s_ok != 0;
  if (ok) {
    ok = wait_bar(&bar_o, 0);
    if (!ok) atomicExch(p.status, kStatusTimeout);
  }
  ok = __syncthreads_and(ok);
  if (ok) {
    ptx::tc_fence_after();
    __nv_bfloat16* orow = p.o + (row * p.H + h) * kDv;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float y[32];
      ptx::tmem_ld32(tO + lane_off + half * 32, y);
      ptx::tmem_ld_wait();
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2)
        pk[j >> 1] = pack_bf16(y[j] + acc[half * 32 + j], y[j + 1] + acc[half * 32 + j + 1]);
      uint4* dst = reinterpret_cast<uint4*>(orow + half * 32);
#pragma unroll
      for (int c = 0; c < 4; ++c) dst[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tbase, 256);
}

// ---------------------------------------------------------------------------------
// tc_export: bucket states at position T (T % 128 == 0, so live levels are >= 8).
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tc_export_kernel(TcParams p, int SL, float* st, float* lsc) {
  const int lvl = blockIdx.x, bh = blockIdx.y;
  float* dst = st + ((size_t)bh * SL + lvl) * kNodeF;
  const bool live = lvl >= 1 && ((((long long)p.T) >> (lvl - 1)) & 1);
  float scale = 0.f;
  const float* src = nullptr;
  if (live) {
    const int m = lvl - kLevIntra;
    const size_t nbase = (size_t)bh * p.nnodes;
    float D = 0.f;
    for (int mm = 0; mm < m; ++mm)
      if ((p.NT >> mm) & 1) D += p.nodeG[nbase + p.node_off[mm] + ((p.NT >> mm) - 1)];
    scale = exp2f(D);
    src = p.node32 + (nbase + p.node_off[m] + ((p.NT >> m) - 1)) * kNodeF;
  }
  for (int e = threadIdx.x; e < kNodeF; e += 256) dst[e] = live ? scale * src[e] : 0.f;
  if (lsc && threadIdx.x == 0) lsc[(size_t)bh * SL + lvl] = 0.f;
}

// ---------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 4-D bf16 map over (inner, count, T, B) with a (64, 1, 128, 1) box, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int inner, int count, int T, int B) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)count, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * 2 * count,
                           (cuuint64_t)inner * 2 * count * T};
  cuuint32_t box[4] = {64, 1, kTile, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int kSmemState = 32768 + 32768 + 1024;
constexpr int kSmemOutput = 98816 + 128 * 9 * 4 + 1024;

__global__ void wait_selftest_kernel(unsigned* status, long long spins) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!ptx::mbar_wait(&bar, 0, spins)) atomicExch(status, kStatusTimeout);
  }
}

}  // namespace

bool tc_supported(const ll_shape& s) {
  return s.dtype == LL_BF16 && s.d_k == kDk && s.d_v == kDv && s.T % kTile == 0 &&
         s.levels <= 32 && encode_fn() != nullptr;
}

const char* tc_kernel_names(bool with_export) {
  return with_export ? "tc_state,tc_output,tc_export" : "tc_state,tc_output";
}

bool make_tc_plan(const ll_shape& s, TcPlan* p) {
  if (!tc_supported(s)) return false;
  p->B = s.batch;
  p->T = s.T;
  p->H = s.heads;
  p->hpg = s.heads_per_group;
  p->G = s.heads / s.heads_per_group;
  p->L = s.levels;
  p->NT = s.T / kTile;
  p->MT = bit_length(p->NT);
  int off = 0;
  for (int m = 0; m < p->MT; ++m) {
    p->node_off[m] = off;
    off += p->NT >> m;
  }
  p->nnodes = off;
  const size_t BH = (size_t)p->B * p->H;
  size_t o = 0;
  p->off_node32 = o;
  o = a256(o + sizeof(float) * BH * p->nnodes * kNodeF);
  p->off_node16 = o;
  o = a256(o + BH * p->nnodes * (size_t)kImgBytes);
  p->off_nodeG = o;
  o = a256(o + sizeof(float) * BH * p->nnodes);
  p->off_cnt = o;
  p->cnt_bytes = sizeof(unsigned) * BH * p->nnodes;
  o = a256(o + p->cnt_bytes);
  p->off_gam = 0;
  p->bytes = o;
  return true;
}

cudaError_t launch_tc_fwd(const TcPlan& tp, const FwdArgs& a, cudaStream_t st) {
  CUtensorMap mQ, mK, mV;
  if (!make_map(&mQ, a.q, kDk, tp.G, tp.T, tp.B) || !make_map(&mK, a.k, kDk, tp.G, tp.T, tp.B) ||
      !make_map(&mV, a.v, kDv, tp.H, tp.T, tp.B))
    return cudaErrorInvalidValue;
  TcParams p;
  p.B = tp.B;
  p.T = tp.T;
  p.H = tp.H;
  p.hpg = tp.hpg;
  p.G = tp.G;
  p.L = tp.L;
  p.NT = tp.NT;
  p.nnodes = tp.nnodes;
  p.MT = tp.MT;
  for (int m = 0; m < 32; ++m) p.node_off[m] = m < tp.MT ? tp.node_off[m] : 0;
  p.a = a.a;
  p.lam = a.lam;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.node32 = reinterpret_cast<float*>(a.ws + tp.off_node32);
  p.img = reinterpret_cast<uint8_t*>(a.ws + tp.off_node16);
  p.nodeG = reinterpret_cast<float*>(a.ws + tp.off_nodeG);
  p.cnt = reinterpret_cast<unsigned*>(a.ws + tp.off_cnt);
  p.status = a.status;
  cudaError_t e = cudaMemsetAsync(p.cnt, 0, tp.cnt_bytes, st);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((size_t)tp.B * tp.NT * tp.H);
  e = cudaFuncSetAttribute(tc_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemState);
  if (e != cudaSuccess) return e;
  tc_state_kernel<<<grid, 128, kSmemState, st>>>(mK, mV, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch(a, 0, st);
  e = cudaFuncSetAttribute(tc_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOutput);
  if (e != cudaSuccess) return e;
  tc_output_kernel<<<grid, 128, kSmemOutput, st>>>(mQ, mK, mV, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch(a, 1, st);
  if (a.states_out) {
    tc_export_kernel<<<dim3(a.state_levels, tp.B * tp.H), 256, 0, st>>>(p, a.state_levels, a.states_out,
                                                                        a.logscale_out);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launch(a, 2, st);
  }
  return cudaSuccess;
}

cudaError_t launch_wait_selftest(unsigned* status, long long spins, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, spins);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace ll
