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
//             cores (M = d_k, N = d_v, K = tokens), published as node (0, u) of the
//             Fenwick tree over tiles.  Nodes are fp16 images in the UMMA operand layout
//             with a power-of-two scale and their total log2 decay.
//  tc_tree    two tree levels per launch, Node_{m+1}[i] = 2^(Gamma(right)) Node_m[2i] +
//             Node_m[2i+1], from the images of the level below (no CTA waits for another).
//  tc_output  one CTA per (b, h, tile u): S = Q Kᵀ on the tensor cores; P = S ⊙ lambda^l
//             ⊙ 2^(g_t - g_s) ⊙ [s <= t] (levels 0..7) written to tensor memory as fp16
//             with a power-of-two row scale; O = P V with P as the tensor-memory operand;
//             then for every set bit m of u one more MMA
//             Y = Q · Node_m[(u >> m) - 1], its rows added with weight
//             lambda_t^(8+m) 2^(g_t + D_m), D_m the decay of the nearer buckets (write-up
//             section 特殊结构：树划分: one memory per bucket level); one write of o.
//  tc_export  bucket states at position T from the published nodes (decode hand-off).
//
// Operands formed inside the kernels are fp16 with exact power-of-two scales chosen from
// their maxima (fp16 keeps 11 significant bits, bf16 only 8); the decayed V of the state
// product is split into a bf16 hi part and a bf16 lo part.  q, k, v enter exactly.
//
// Every mbarrier wait is bounded by 2 s of %globaltimer; a wait that runs out records
// LL_ERR_TIMEOUT in the status word and the CTA skips the rest of its work.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <utility>

#include "ll_internal.cuh"
#include "ptx.cuh"

namespace ll {

namespace {

constexpr int kTile = 128;                   // tokens per tile
constexpr int kDk = 128, kDv = 64;            // supported head dims
constexpr int kLevIntra = 8;                  // levels 0..7 live inside a 128-token tile
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s per wait before giving up
constexpr int kImgBytes = kDk * kDv * 2;      // fp16 node image, 128 rows x 128 bytes
constexpr int kMeta = 4;  // u32 per node: spare, scale exponent, log2 decay (f32 bits), spare

struct TcParams {
  int B, T, H, hpg, G, L, NT, nnodes, MT;
  int node_off[32];
  const float* a;
  const float* lam;
  __nv_bfloat16* o;
  uint8_t* img;    // (B*H, nnodes, 16 KB) fp16 node images
  unsigned* meta;  // (B*H, nnodes, 4)
  unsigned* status;
  // comparators only (single-level and SSD output modes)
  float* o32;      // (B, T, H, d_v) fp32 running sum of the single-level passes
  int lsel;        // the one level of a single-level pass
  int lflags;      // bit 0: first pass (store), bit 1: last pass (write o)
  uint8_t* pimg;   // (B*H, NT, 16 KB) SSD prefix-state images
  unsigned* pmeta; // (B*H, NT, 4)
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (ptx::globaltimer_ns() - t0 > kWaitNs) return false;
  }
}

// 2^e as an exact float, e in [-126, 127].
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }
// 2^e for a sum of two exponents (|e| <= 252): product of two exact powers of two.
__device__ __forceinline__ float pow2s(int e) {
  const int h = e / 2;
  return pow2i(h) * pow2i(e - h);
}

// Exponent e with m * 2^-e in [2^14, 2^15): scaling by 2^-e keeps fp16 away from
// overflow (max 65504) and keeps 29 binades below the maximum in fp16's normal range.
__device__ __forceinline__ int f16_exp(float m) {
  if (!(m > 0.f)) return 0;
  int eb = ((__float_as_int(m) >> 23) & 0xff) - 127;
  if (eb < -126) eb = -126;
  int e = eb - 14;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}

// Block-wide inclusive prefix sum over 128 threads (one value each).
__device__ __forceinline__ float block_scan128(float x, float* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    float y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_red[warp] = x;
  __syncthreads();
  float add = 0.f;
  for (int w = 0; w < warp; ++w) add += s_red[w];
  __syncthreads();
  return x + add;
}

// Block-wide max of two values (128 threads).
__device__ __forceinline__ float2 block_max2(float2 v, float2* s_red2) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    v.x = fmaxf(v.x, __shfl_xor_sync(0xffffffffu, v.x, off));
    v.y = fmaxf(v.y, __shfl_xor_sync(0xffffffffu, v.y, off));
  }
  if (lane == 0) s_red2[warp] = v;
  __syncthreads();
  float2 r = s_red2[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
    r.x = fmaxf(r.x, s_red2[w].x);
    r.y = fmaxf(r.y, s_red2[w].y);
  }
  __syncthreads();
  return r;
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Publishes one tree node from 128 threads, thread tid holding row tid (d_k index) of the
// d_k x d_v fp32 state in cur: an fp16 image with a power-of-two scale 2^e (maximum in
// [2^14, 2^15)), row tid at chunk slots c ^ (tid & 7), staged through `stage` (16 KB of
// shared memory whose row tid only this thread uses before the call) so that the global
// stores coalesce; then the scale exponent and the node's log2 decay G into meta.
__device__ __forceinline__ void publish_node(const float (&cur)[kDv], uint8_t* stage, size_t node,
                                             float G, float2* s_red2, uint8_t* img, unsigned* meta) {
  const int tid = threadIdx.x, rot = tid & 7;
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < kDv; ++j) m = fmaxf(m, fabsf(cur[j]));
  const int e = f16_exp(block_max2(make_float2(m, 0.f), s_red2).x);
  const float s = pow2i(-e);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int cc = c ^ rot;
    *reinterpret_cast<uint4*>(stage + tid * 128 + (cc << 4)) =
        make_uint4(pack_h2(cur[8 * c] * s, cur[8 * c + 1] * s), pack_h2(cur[8 * c + 2] * s, cur[8 * c + 3] * s),
                   pack_h2(cur[8 * c + 4] * s, cur[8 * c + 5] * s), pack_h2(cur[8 * c + 6] * s, cur[8 * c + 7] * s));
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(img + node * kImgBytes);
#pragma unroll
  for (int r = 0; r < kImgBytes / 16 / 128; ++r)
    dst[r * 128 + tid] = reinterpret_cast<const uint4*>(stage)[r * 128 + tid];
  if (tid == 0) {
    meta[node * kMeta + 1] = (unsigned)e;
    meta[node * kMeta + 2] = __float_as_uint(G);
  }
}

// ---------------------------------------------------------------------------------
// tc_state: tile states (level 0 of the Fenwick tree over tiles).
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) tc_state_kernel(const __grid_constant__ CUtensorMap mapK,
                                                       const __grid_constant__ CUtensorMap mapV,
                                                       TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;          // 32 KB: K (bf16, two 64-wide d_k boxes); later node staging
  uint8_t* sV = smem + 32768;  // 32 KB: Ṽ hi part (the TMA box) then Ṽ lo part
  __shared__ __align__(8) uint64_t bar_ld, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ float s_red[4];
  __shared__ float2 s_red2[4];
  __shared__ float s_gamma;

  const int tid = threadIdx.x, warp = tid >> 5, rot = tid & 7;
  const int lin = blockIdx.x;
  const int h = lin % p.H;
  const int u = (lin / p.H) % p.NT;
  const int b = lin / (p.H * p.NT);
  const int g = h / p.hpg;
  const int bh = b * p.H + h;
  const long long t0 = (long long)u * kTile;
  const float la = log2f(p.a[((size_t)b * p.T + t0 + tid) * p.H + h]);
  ptx::griddep_launch_dependents();

  if (tid == 0) {
    ptx::mbar_init(&bar_ld, 1);
    ptx::mbar_init(&bar_mma, 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(&bar_ld, 32768 + 16384);
    ptx::tma_load_4d(sK, &mapK, &bar_ld, 0, g, (int)t0, b);
    ptx::tma_load_4d(sK + 16384, &mapK, &bar_ld, 64, g, (int)t0, b);
    ptx::tma_load_4d(sV, &mapV, &bar_ld, 0, h, (int)t0, b);
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 128);
    ptx::tmem_relinquish();
  }
  // decay of token t0 + tid: chunk-local log2 cumsum (the scan also publishes tmem_base)
  ptx::tc_fence_before();
  const float gi = block_scan128(la, s_red);
  ptx::tc_fence_after();
  const uint32_t tbase = tmem_base;
  if (tid == kTile - 1) s_gamma = gi;
  bool ok = wait_bar(&bar_ld, 0);
  if (!ok) atomicExch(p.status, kStatusTimeout);
  ok = __syncthreads_and(ok);
  const float gamma = s_gamma;
  if (ok) {
    // Ṽ row tid = 2^(gamma - g_tid) v_tid as a bf16 hi part (in place) plus a bf16 lo
    // part (the rounding remainder), so that Kᵀ(Ṽhi + Ṽlo) keeps ~16 bits.  The 128-byte
    // swizzle permutes 16-byte chunks inside a row only, so rows map in place.
    const float w = exp2f(gamma - gi);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int off = tid * 128 + ((c ^ rot) << 4);
      uint4 x = *reinterpret_cast<uint4*>(sV + off), y;
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
      *reinterpret_cast<uint4*>(sV + off) = x;
      *reinterpret_cast<uint4*>(sV + 16384 + off) = y;
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

  // the tile's node (level 0; node_off[0] == 0), staged in sK (free now)
  publish_node(cur, sK, (size_t)bh * p.nnodes + u, gamma, s_red2, p.img, p.meta);
}

// ---------------------------------------------------------------------------------
// tc_tree: levels m0 and m0 + 1 of the Fenwick tree over tiles, from the published
// images of level m0 - 1.  Node_{m+1}[i] = 2^(Gamma(Node_m[2i+1])) Node_m[2i] +
// Node_m[2i+1].  One CTA per pair of level-m0 nodes (2i, 2i+1): it loads their four
// children with bulk copies, merges each pair in fp32 (thread tid owns row tid),
// publishes the even one, and the parent Node_{m0+1}[i] from the fp32 sums when it exists.  No
// CTA waits for another: the launches before it on the stream produced its inputs.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 3) tc_tree_kernel(TcParams p, int m0) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar_ld;
  __shared__ float2 s_red2[4];
  const int tid = threadIdx.x, rot = tid & 7;
  const int n0 = p.NT >> m0;         // nodes at level m0
  const int ni = (n0 + 1) >> 1;      // CTAs per (b, h)
  const int bh = blockIdx.x / ni, i = blockIdx.x % ni;
  const int nj = (2 * i + 1 < n0) ? 2 : 1;  // level-m0 nodes built here
  const size_t nbase = (size_t)bh * p.nnodes;
  const size_t child0 = nbase + p.node_off[m0 - 1] + 4 * i;
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();  // the level below is the previous launch's output
  if (tid == 0) {
    ptx::mbar_init(&bar_ld, 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(&bar_ld, 2 * nj * kImgBytes);
    for (int c = 0; c < 2 * nj; ++c)
      ptx::bulk_load(smem + c * kImgBytes, p.img + (child0 + c) * kImgBytes, kImgBytes, &bar_ld);
  }
  float sc[4], gm[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    sc[c] = c < 2 * nj ? pow2i((int)p.meta[(child0 + c) * kMeta + 1]) : 0.f;
    gm[c] = c < 2 * nj ? __uint_as_float(p.meta[(child0 + c) * kMeta + 2]) : 0.f;
  }
  __syncthreads();  // barrier initialised
  bool ok = wait_bar(&bar_ld, 0);
  if (!ok) atomicExch(p.status, kStatusTimeout);
  ok = __syncthreads_and(ok);
  if (!ok) {
    if (tid == 0) wait_bar(&bar_ld, 0);  // bounded: let the copies land before exit
    return;
  }
  float par[kDv], cur[kDv];
  float G0 = 0.f;
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    if (jj >= nj) break;
    const uint8_t* L = smem + (2 * jj) * kImgBytes + tid * 128;
    const uint8_t* R = L + kImgBytes;
    const float wl = exp2f(gm[2 * jj + 1]) * sc[2 * jj], wr = sc[2 * jj + 1];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 l4 = *reinterpret_cast<const uint4*>(L + ((c ^ rot) << 4));
      const uint4 r4 = *reinterpret_cast<const uint4*>(R + ((c ^ rot) << 4));
      const __half2* hl = reinterpret_cast<const __half2*>(&l4);
      const __half2* hr = reinterpret_cast<const __half2*>(&r4);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fl = __half22float2(hl[e]), fr = __half22float2(hr[e]);
        cur[8 * c + 2 * e] = wl * fl.x + wr * fr.x;
        cur[8 * c + 2 * e + 1] = wl * fl.y + wr * fr.y;
      }
    }
    const float G = gm[2 * jj] + gm[2 * jj + 1];
    // staged over the left child, whose row tid only this thread has read.  An odd node
    // is read by nothing but its parent (tile u reads Node_m[(u >> m) - 1] with u >> m
    // odd; the export reads Node_m[(NT >> m) - 1] with NT >> m odd; the next launch reads
    // the parents), so it stays in registers.
    if (jj == 0)
      publish_node(cur, smem, nbase + p.node_off[m0] + 2 * i, G, s_red2, p.img, p.meta);
    if (jj == 0) {
      G0 = G;
#pragma unroll
      for (int j = 0; j < kDv; ++j) par[j] = cur[j];
    } else {
      const float d = exp2f(G);
#pragma unroll
      for (int j = 0; j < kDv; ++j) par[j] = d * par[j] + cur[j];
    }
  }
  if (nj == 2)  // then i < NT >> (m0 + 1): the parent exists
    publish_node(par, smem + kImgBytes, nbase + p.node_off[m0 + 1] + i, G0 + gm[2] + gm[3], s_red2, p.img,
                 p.meta);
}

// ---------------------------------------------------------------------------------
// tc_output: intra-tile masked attention + level-fused inter-tile buckets.
//
// 256 threads in two roles after a common prologue (loads, decay cumsum):
//  role a (warps 0-3): once S has landed, P row t = thread, written as fp16 into tensor
//          memory over the columns of S it has consumed; then the V tile scale and V ->
//          fp16 in place; O = P V with P as the tensor-memory A operand.
//  role b (warps 4-7): issues S = Q Kᵀ; waits for the tree's launches and fetches the
//          node scalars and the first node image; Q row t -> fp16 with a power-of-two
//          scale of its own (undone in the row weight) in place once S has read Q; the
//          inter-tile levels, nearest first and two per MMA (N = 128 over two node
//          images), with up to three node images in flight; then the write of o.
// Both roles see every TMEM lane through warp % 4.
// Shared memory (2 CTAs per SM): RQ = Q (bf16, then fp16 in place); RK = K (bf16) until
// S completes, then node image buffers 1 and 2; RV = V (bf16, then fp16 in place);
// RE = node image buffer 0.  The image of level index i (i-th set bit of u from the
// bottom) goes to buffer i % 3, completing phase (i / 3) & 1 of bar_e[i % 3].
// lambda rows and the node scalars are copied into shared memory at the start
// (asynchronously), so that no global load sits on the path of P or of a level.
// TMEM (256 columns): S in 0..127; once role a has consumed S, P in 0..63 and O in
// 64..127; Y of a pair of levels in 128..255 (free from the start).
//
// kMode selects what one launch computes (1 and 2 exist only as comparators):
//  0  the level-fused forward above;
//  1  the lambda-constant special case (Mamba-2 SSD): lambda = 1 at every level and one
//     inter-tile term per tile, from the prefix state of all earlier tiles (pimg);
//  2  one level lsel only, accumulated in fp32 across launches (no level fusion): an
//     intra level masks P to that level; an inter level skips S, P and O.
// ---------------------------------------------------------------------------------
constexpr int kOutFixed = 104704;  // shared bytes in front of the inter-level lambda table
constexpr int kMaxInter = 19;      // inter-tile levels per tile supported (NT <= 2^19)
__host__ __device__ constexpr int out_smem_bytes(int ninter) {
  return kOutFixed + 512 * (ninter > 0 ? ninter : 1) + 1024;
}

__device__ __forceinline__ int nth_set_bit(unsigned x, int i) {
  for (int j = 0; j < i; ++j) x &= x - 1;
  return __ffs(x) - 1;
}
// |.|-max of two bf16 pairs, halfwise (the sign of the result is meaningless)
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t acc, uint32_t w) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(acc), "r"(w));
  return d;
}
__device__ __forceinline__ float bf16x2_maxhalf(uint32_t w) {
  return fmaxf(fabsf(__uint_as_float(w << 16)), fabsf(__uint_as_float(w & 0xffff0000u)));
}
__device__ __forceinline__ uint32_t absmax_u4(uint32_t acc, const uint4& x) {
  return bf16x2_absmax(bf16x2_absmax(acc, x.x), bf16x2_absmax(x.y, bf16x2_absmax(x.z, x.w)));
}
// bf16 pair -> fp16 pair, both times s2 (an exact power of two, so the bf16 product is exact)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, __nv_bfloat162 s2) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&w);
  x = __hmul2(x, s2);
  const uint32_t y = *reinterpret_cast<uint32_t*>(&x);
  return pack_h2(__uint_as_float(y << 16), __uint_as_float(y & 0xffff0000u));
}
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4& x, __nv_bfloat162 s2) {
  return make_uint4(bf16x2_to_f16x2(x.x, s2), bf16x2_to_f16x2(x.y, s2), bf16x2_to_f16x2(x.z, s2),
                    bf16x2_to_f16x2(x.w, s2));
}

template <int kMode>
__global__ void __launch_bounds__(256, 2) tc_output_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                           const __grid_constant__ CUtensorMap mapK,
                                                           const __grid_constant__ CUtensorMap mapV,
                                                           TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* RQ = smem;           // 32 KB (two d_k blocks of 64)
  uint8_t* RK = smem + 32768;   // 32 KB
  uint8_t* RV = smem + 65536;   // 16 KB
  uint8_t* RE = smem + 81920;   // 16 KB
  float* sG = reinterpret_cast<float*>(smem + 98304);      // 128: g
  float* sB8 = reinterpret_cast<float*>(smem + 98816);     // 128: 2^(g_end8(s) - g_s)
  int* sEp = reinterpret_cast<int*>(smem + 99328);         // 128: P row + V scale exponents
  float* sLam8 = reinterpret_cast<float*>(smem + 99840);   // 128 x 9: lambda levels 0..7 of row r
  float* sNode = reinterpret_cast<float*>(smem + 104448);  // 32 x 2: node scale exp. (bits), log2 decay
  float* sLamI = reinterpret_cast<float*>(smem + kOutFixed);  // [level index][row]: lambda_t^(8+m)
  __shared__ __align__(8) uint64_t bar_ld, bar_s, bar_o, bar_e[3], bar_y[2], bar_yf[2];
  __shared__ uint32_t tmem_base;
  __shared__ float s_red[8];
  __shared__ int s_oi;  // role a -> all: the O MMA was issued

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127;             // query row (tile-local token)
  const int quad = warp & 3;           // TMEM lane quadrant of this warp
  const bool role_b = warp >= 4;       // S, inter-tile levels and the final write
  const bool driver = tid == 128;      // role b's MMA and image-load issuer
  const int rot = r & 7;
  const int lin = blockIdx.x;
  const int h = lin % p.H;
  const int u = (lin / p.H) % p.NT;
  const int b = lin / (p.H * p.NT);
  const int g = h / p.hpg;
  const int bh = b * p.H + h;
  const long long t0 = (long long)u * kTile;
  const size_t nbase = (size_t)bh * p.nnodes;
  const size_t row = (size_t)b * p.T + t0 + r;  // token of this thread's query row
  const float* lrow = p.lam + (row * p.H + h) * p.L;
  // inter-tile levels of this tile, and whether the intra-tile part runs
  ptx::griddep_launch_dependents();  // the next launch may start once all CTAs are resident
  const int nlev = kMode == 0 ? __popc((unsigned)u)
                 : kMode == 1 ? (u > 0 ? 1 : 0)
                              : (p.lsel >= kLevIntra && ((u >> (p.lsel - kLevIntra)) & 1) ? 1 : 0);
  const bool intra_on = kMode != 2 || p.lsel < kLevIntra;
  auto ebuf = [&](int k) { return k == 0 ? RE : RK + (k - 1) * 16384; };  // image buffer k
  auto lev_of = [&](int i) {  // tile level m of level index i
    return kMode == 2 ? p.lsel - kLevIntra : nth_set_bit((unsigned)u, i);
  };
  auto img_of = [&](int i) -> const uint8_t* {  // image read by level index i
    if (kMode == 1) return p.pimg + ((size_t)bh * p.NT + u) * kImgBytes;
    const int m = lev_of(i);
    return p.img + (nbase + p.node_off[m] + ((u >> m) - 1)) * kImgBytes;
  };
  auto meta_of = [&](int i) -> const unsigned* {
    if (kMode == 1) return p.pmeta + ((size_t)bh * p.NT + u) * kMeta;
    const int m = lev_of(i);
    return p.meta + (nbase + p.node_off[m] + ((u >> m) - 1)) * kMeta;
  };

  if (tid == 0) {
    s_oi = 0;
    ptx::mbar_init(&bar_ld, 1);
    ptx::mbar_init(&bar_s, 1);
    ptx::mbar_init(&bar_o, 1);
    for (int i = 0; i < 3; ++i) ptx::mbar_init(&bar_e[i], 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bar_y[i], 1);
      ptx::mbar_init(&bar_yf[i], 128);
    }
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(&bar_ld, intra_on ? 32768 * 2 + 16384 : 32768);
    ptx::tma_load_4d(RQ, &mapQ, &bar_ld, 0, g, (int)t0, b);
    ptx::tma_load_4d(RQ + 16384, &mapQ, &bar_ld, 64, g, (int)t0, b);
    if (intra_on) {
      ptx::tma_load_4d(RK, &mapK, &bar_ld, 0, g, (int)t0, b);
      ptx::tma_load_4d(RK + 16384, &mapK, &bar_ld, 64, g, (int)t0, b);
      ptx::tma_load_4d(RV, &mapV, &bar_ld, 0, h, (int)t0, b);
    }
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 256);
    ptx::tmem_relinquish();
  }
  // lambda of this row (levels 0..7 for role a, the tile's inter levels for role b) and
  // the node scalars of the tile's levels, copied asynchronously
  if (!role_b) {
#pragma unroll
    for (int l = 0; l < kLevIntra; ++l) {
      if (kMode == 0 || (kMode == 2 && l == p.lsel)) ptx::cp_async4(sLam8 + r * 9 + l, lrow + l);
      else sLam8[r * 9 + l] = kMode == 1 ? 1.f : 0.f;  // SSD: lambda = 1; single level: others off
    }
  } else {
    if (kMode == 1) {
      if (nlev > 0) sLamI[r] = 1.f;
    } else {
      for (int i = 0; i < nlev; ++i) ptx::cp_async4(sLamI + i * 128 + r, lrow + kLevIntra + lev_of(i));
    }
  }
  // chunk-local log2 decay cumsum over the 128 rows (both roles compute it)
  float gt = log2f(p.a[row * p.H + h]);
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, gt, off);
    if (lane >= off) gt += y;
  }
  if (lane == 31) s_red[warp] = gt;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  for (int w = 0; w < quad; ++w) gt += s_red[w];
  const uint32_t tbase = tmem_base;
  const uint32_t tS = tbase, tO = tbase + 64;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  if (!role_b) sG[r] = gt;
  __syncthreads();  // sG complete; s_red free again
  if (!role_b) sB8[r] = exp2f(sG[r | 7] - gt);  // decay from key r to the end of its 8-block
  bool ok = wait_bar(&bar_ld, 0);
  if (!ok) atomicExch(p.status, kStatusTimeout);
  ok = __syncthreads_and(ok);

  // S = Q Kᵀ (M = 128 queries, N = 128 keys, K = 128 d_k), bf16, both K-major.
  if (ok && driver && intra_on) {
    ptx::tc_fence_after();
    const uint32_t idesc = ptx::idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t q0 = ptx::smem_u32(RQ), k0 = ptx::smem_u32(RK);
#pragma unroll
    for (int kk = 0; kk < kDk / 16; ++kk) {
      const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
      ptx::umma_f16(tS, ptx::smem_desc_sw128(q0 + off, 16, 1024),
                    ptx::smem_desc_sw128(k0 + off, 16, 1024), idesc, kk > 0);
    }
    ptx::umma_commit(&bar_s);
  }
  const bool s_issued = ok && intra_on;

  if (!role_b && !intra_on) {
    __syncthreads();  // join: nothing to do without the intra-tile part
  } else if (!role_b) {
    // ---- role a -----------------------------------------------------------------------
    // P as soon as S has landed; then the V tile scale and V -> fp16 in place (V is an
    // operand of O only, and P does not depend on V's scale).
    if (ok) {
      ok = wait_bar(&bar_s, 0);
      if (!ok) atomicExch(p.status, kStatusTimeout);
    }
    ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld / st below are warp-collective
    int ep = 0;
    // P row t = r in fp16 with row scale 2^-ep, into TMEM columns 0..63 over S.
    if (ok) {
      ptx::tc_fence_after();
      ptx::cp_async_wait_all();
      const float* lamr = sLam8 + r * 9;
      const int t = r, tl = t & 31;
      float lmax = 0.f;
#pragma unroll
      for (int l = 0; l < kLevIntra; ++l) lmax = fmaxf(lmax, fabsf(lamr[l]));
      float smax = 0.f;
#pragma unroll 1
      for (int cg = 0; cg < quad; ++cg) {  // warp-uniform bound
        float sv[32];
        ptx::tmem_ld32(tS + lane_off + cg * 32, sv);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) smax = fmaxf(smax, fabsf(sv[j]));
      }
      {
        float sv[32];
        ptx::tmem_ld32(tS + lane_off + quad * 32, sv);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j <= tl) smax = fmaxf(smax, fabsf(sv[j]));
      }
      ep = f16_exp(smax * lmax);  // |P| <= max|S| * max lambda (decays are <= 1)
      const float coef = pow2i(-ep);
      // Decay 2^(g_t - g_s) = A_kb B8[s], with A_kb = 2^(g_t - g_end8(kb)) per row and
      // 8-key block kb and B8[s] = 2^(g_end8(s) - g_s) per key; both are <= 1 for keys of
      // blocks before t's.  In t's own block A_kb >= 1, bounded by 2^(block span): when no
      // block of the diagonal group spans more than 60 the factored form stays inside
      // fp32's range; otherwise each key of that group takes its own exp2 (warp-uniform).
      const float* gq = sG + quad * 32;
      const float span8 = fmaxf(fmaxf(gq[0] - gq[7], gq[8] - gq[15]), fmaxf(gq[16] - gq[23], gq[24] - gq[31]));
      const bool fastd = span8 <= 60.f;
      // Keys cg*32 .. cg*32+31 become packed columns cg*16 .. cg*16+15: those columns held
      // S of keys below cg*32, all read before (the loop runs upward).
#pragma unroll 1
      for (int cg = 0; cg < 4; ++cg) {
        uint32_t pk[16];
        if (cg < quad) {
          // keys of an earlier 32-group: one level (6 or 7) and the factored decay
          float sv[32];
          ptx::tmem_ld32(tS + lane_off + cg * 32, sv);
          ptx::tmem_ld_wait();
          const float cl = coef * lamr[(quad ^ cg) >= 2 ? 7 : 6];
          float ak[4];
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) ak[kb] = cl * exp2f(gt - sG[cg * 32 + kb * 8 + 7]);
          const float4* b4 = reinterpret_cast<const float4*>(sB8 + cg * 32);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 bb = b4[j4];
            const float a = ak[j4 >> 1];
            pk[2 * j4] = pack_h2(sv[4 * j4] * a * bb.x, sv[4 * j4 + 1] * a * bb.y);
            pk[2 * j4 + 1] = pack_h2(sv[4 * j4 + 2] * a * bb.z, sv[4 * j4 + 3] * a * bb.w);
          }
        } else if (cg == quad) {
          // the diagonal 32-group: levels 0..5 (level of key j: bit length of tl ^ j)
          float sv[32];
          ptx::tmem_ld32(tS + lane_off + cg * 32, sv);
          ptx::tmem_ld_wait();
          float v[32];
          if (fastd) {
            // blocks after t's may give A = inf; their keys are masked by the select
            float ak[4];
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) ak[kb] = exp2f(gt - gq[kb * 8 + 7]);
            const float4* b4 = reinterpret_cast<const float4*>(sB8 + cg * 32);
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 bb = b4[j4];
              const float bj[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int j = 4 * j4 + e;
                const float x = (sv[j] * coef) * lamr[32 - __clz(tl ^ j)] * (ak[j >> 3] * bj[e]);
                v[j] = j <= tl ? x : 0.f;
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float x = sv[j] * coef * lamr[32 - __clz(tl ^ j)] * exp2f(gt - gq[j]);
              v[j] = j <= tl ? x : 0.f;
            }
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = pack_h2(v[2 * j], v[2 * j + 1]);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = 0u;
        }
        ptx::tmem_st16(tS + lane_off + cg * 16, pk);
      }
      ptx::tmem_st_wait();
    }
    uint8_t* vrow = RV + r * 128;
    uint4 vv[8];
    if (ok) {
      uint32_t mx = 0u;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        vv[c] = *reinterpret_cast<const uint4*>(vrow + ((c ^ rot) << 4));
        mx = absmax_u4(mx, vv[c]);
      }
      float mv = bf16x2_maxhalf(mx);
#pragma unroll
      for (int off = 16; off; off >>= 1) mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
      if (lane == 0) s_red[warp] = mv;
    }
    ptx::named_bar_sync(1, 128);
    if (ok) {
      const int ev = f16_exp(fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3])));
      const float sv_ = pow2i(-ev);
      const __nv_bfloat162 s2 = __floats2bfloat162_rn(sv_, sv_);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(vrow + ((c ^ rot) << 4)) = bf16x8_to_f16x8(vv[c], s2);
      ptx::fence_proxy_async_smem();
      sEp[r] = ep + ev;
    }
    ptx::tc_fence_before();
    const bool ok_a = ptx::named_bar_and(1, 128, ok);
    // O = P V (M = 128, N = 64, K = 128 keys): P from TMEM, V fp16 MN-major, into the
    // S columns 64..127 that every role-a thread has finished reading.
    if (tid == 0 && ok_a) {
      ptx::tc_fence_after();
      const uint32_t idesc = ptx::idesc_f16_f32(128, 64, 0, 1);
      const uint32_t v0 = ptx::smem_u32(RV);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        ptx::umma_f16_tmem_a(tO, tS + kk * 8, ptx::smem_desc_sw128(v0 + kk * 2048, 1024, 1024),
                             idesc, kk > 0);
      ptx::umma_commit(&bar_o);
      s_oi = 1;
    }
    __syncthreads();  // join (role b waits here after its levels)
  } else {
    // ---- role b -----------------------------------------------------------------------
    // The tree that the previous launches built is read from here on: wait for them (at
    // once unless this grid was launched before they finished), then fetch the node
    // scalars and the first image (into RE, free from the start) behind the Q work.
    // Q row r -> fp16 with scale 2^-eq of its own: read and converted while S runs,
    // stored back once S has completed.  Then images 1 and 2 go into RK.
    uint8_t* qrow0 = RQ + r * 128;
    uint8_t* qrow1 = RQ + 16384 + r * 128;
    int eq = 0;
    int issued = 0;                 // image loads issued
    int consumed = 0;               // image loads waited for by the driver
    int y_issued = 0, y_seen = 0;   // Y MMAs issued / seen complete by the driver
    ptx::griddep_wait();
    if (r < nlev) {
      const unsigned* mt = meta_of(r);
      ptx::cp_async4(sNode + 2 * r, mt + 1);
      ptx::cp_async4(sNode + 2 * r + 1, mt + 2);
    }
    if (ok && driver && nlev > 0) {
      ptx::mbar_arrive_expect_tx(&bar_e[0], kImgBytes);
      ptx::bulk_load(ebuf(0), img_of(0), kImgBytes, &bar_e[0]);
      ++issued;
    }
    if (ok) {
      uint4 qv[16];
      uint32_t mx = 0u;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        qv[c] = *reinterpret_cast<const uint4*>(qrow0 + ((c ^ rot) << 4));
        qv[8 + c] = *reinterpret_cast<const uint4*>(qrow1 + ((c ^ rot) << 4));
        mx = absmax_u4(absmax_u4(mx, qv[c]), qv[8 + c]);
      }
      eq = f16_exp(bf16x2_maxhalf(mx));
      const float sq = pow2i(-eq);
      const __nv_bfloat162 s2 = __floats2bfloat162_rn(sq, sq);
#pragma unroll
      for (int c = 0; c < 16; ++c) qv[c] = bf16x8_to_f16x8(qv[c], s2);
      if (intra_on) {
        ok = wait_bar(&bar_s, 0);
        if (!ok) atomicExch(p.status, kStatusTimeout);
      }
      if (ok) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(qrow0 + ((c ^ rot) << 4)) = qv[c];
          *reinterpret_cast<uint4*>(qrow1 + ((c ^ rot) << 4)) = qv[8 + c];
        }
        ptx::fence_proxy_async_smem();
      }
    }
    if (ok && driver) {
      for (int i = 1; i < 3 && i < nlev; ++i) {  // K has been read by S: RK is free
        ptx::mbar_arrive_expect_tx(&bar_e[i], kImgBytes);
        ptx::bulk_load(ebuf(i), img_of(i), kImgBytes, &bar_e[i]);
        ++issued;
      }
    }
    ptx::cp_async_wait_all();
    ok = ptx::named_bar_and(2, 128, ok);  // Q fp16 in place; sLamI, sNode complete

    // Levels in pairs, nearest first.  One MMA with N = 128 covers levels i and i + 1:
    // B is the two node images as two 64-wide MN atoms, the one at the lower shared
    // address first and the other LBO bytes above it; Y lands in TMEM columns 128..255.
    // A last level without a partner takes N = 64 (columns 128..191).  Rows are added
    // with weight lambda_t^(8+m) 2^(g_t + D) and the two scales.
    auto pair_cols = [&](int i, bool two) {  // TMEM column offset of level i within the pair
      return (two && ebuf(i % 3) > ebuf((i + 1) % 3)) ? 64 : 0;
    };
    auto issue_pair = [&](int i) -> bool {
      const bool two = i + 1 < nlev;
      if (i >= 2 && !wait_bar(&bar_yf[0], ((i >> 1) - 1) & 1)) return false;  // Y read by all
      if (!wait_bar(&bar_e[i % 3], (i / 3) & 1)) return false;                 // images landed
      ++consumed;
      if (two) {
        if (!wait_bar(&bar_e[(i + 1) % 3], ((i + 1) / 3) & 1)) return false;
        ++consumed;
      }
      ptx::tc_fence_after();
      const uint32_t ea = ptx::smem_u32(ebuf(i % 3));
      const uint32_t eb = two ? ptx::smem_u32(ebuf((i + 1) % 3)) : ea;
      const uint32_t e0 = ea < eb ? ea : eb;
      const uint32_t lbo = two ? (ea < eb ? eb - ea : ea - eb) : 1024;
      const uint32_t idesc = ptx::idesc_f16_f32(128, two ? 128 : 64, 0, 1);
      const uint32_t q0 = ptx::smem_u32(RQ);
#pragma unroll
      for (int kk = 0; kk < kDk / 16; ++kk) {
        const uint32_t offq = (kk >> 2) * 16384 + (kk & 3) * 32;
        ptx::umma_f16(tbase + 128, ptx::smem_desc_sw128(q0 + offq, 16, 1024),
                      ptx::smem_desc_sw128(e0 + kk * 2048, lbo, 1024), idesc, kk > 0);
      }
      ptx::umma_commit(&bar_y[0]);
      ++y_issued;
      return true;
    };
    float acc[kDv];
#pragma unroll
    for (int j = 0; j < kDv; ++j) acc[j] = 0.f;
    float D = 0.f;
    if (kMode == 2 && nlev > 0) {  // one level: the nearer buckets' decay still applies
      const int m = p.lsel - kLevIntra;
      for (unsigned rest = (unsigned)u & ((1u << m) - 1u); rest; rest &= rest - 1) {
        const int mm = __ffs(rest) - 1;
        D += __uint_as_float(p.meta[(nbase + p.node_off[mm] + ((u >> mm) - 1)) * kMeta + 2]);
      }
    }
    bool okd = true;
    for (int i = 0; ok && i < nlev; i += 2) {
      const bool two = i + 1 < nlev;
      if (driver) {
        okd = okd && issue_pair(i);
        if (!okd) atomicExch(p.status, kStatusTimeout);
      }
      bool okw = wait_bar(&bar_y[0], (i >> 1) & 1);
      if (!okw) atomicExch(p.status, kStatusTimeout);
      okw = __all_sync(0xffffffffu, okw);
      if (!okw) {
        ok = false;
        break;
      }
      if (driver) {
        ++y_seen;
        for (int l = i; l < i + (two ? 2 : 1); ++l)
          if (l + 3 < nlev) {  // the image buffer of level l is free again
            ptx::mbar_arrive_expect_tx(&bar_e[l % 3], kImgBytes);
            ptx::bulk_load(ebuf(l % 3), img_of(l + 3), kImgBytes, &bar_e[l % 3]);
            ++issued;
          }
      }
      ptx::tc_fence_after();
      const int ci = pair_cols(i, two);
#pragma unroll 1
      for (int l = 0; l < (two ? 2 : 1); ++l) {
        const int lv = i + l;
        const uint32_t ty = tbase + 128 + (l == 0 ? ci : 64 - ci) + lane_off;
        const float wy = sLamI[lv * 128 + r] * exp2f(gt + D) * pow2s(eq + __float_as_int(sNode[2 * lv]));
        float y[32];
        ptx::tmem_ld32(ty, y);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] += wy * y[j];
        ptx::tmem_ld32(ty + 32, y);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[32 + j] += wy * y[j];
        D += sNode[2 * lv + 1];
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bar_yf[0]);
    }
    if (driver) {
      // after a failed wait: let this CTA's own copies and MMAs land (bounded) before exit
      for (int j = consumed; j < issued; ++j) wait_bar(&bar_e[j % 3], (j / 3) & 1);
      for (int j = y_seen; j < y_issued; ++j) wait_bar(&bar_y[0], j & 1);
      if (s_issued) wait_bar(&bar_s, 0);
    }
    __syncthreads();  // join: P, its row scales and the O MMA have been issued
    const bool o_issued = s_oi != 0;
    if (intra_on) {
      ok = ok && o_issued && wait_bar(&bar_o, 0);
      if (!ok && o_issued) atomicExch(p.status, kStatusTimeout);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      ptx::tc_fence_after();
      const float so = pow2s(sEp[r]);
      __nv_bfloat16* orow = p.o + (row * p.H + h) * kDv;
      float* o32row = kMode == 2 ? p.o32 + (row * p.H + h) * kDv : nullptr;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float y[32];
        if (intra_on) {
          ptx::tmem_ld32(tO + lane_off + half * 32, y);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) y[j] = y[j] * so + acc[half * 32 + j];
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) y[j] = acc[half * 32 + j];
        }
        if (kMode == 2 && !(p.lflags & 2)) {  // store or add the running fp32 sum
          float4* d4 = reinterpret_cast<float4*>(o32row + half * 32);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float4 x = make_float4(y[4 * c], y[4 * c + 1], y[4 * c + 2], y[4 * c + 3]);
            if (!(p.lflags & 1)) {
              const float4 o4 = d4[c];
              x.x += o4.x; x.y += o4.y; x.z += o4.z; x.w += o4.w;
            }
            d4[c] = x;
          }
          continue;
        }
        if (kMode == 2) {  // last pass: add the running sum, then write o
          const float4* s4 = reinterpret_cast<const float4*>(o32row + half * 32);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 o4 = s4[c];
            y[4 * c] += o4.x; y[4 * c + 1] += o4.y; y[4 * c + 2] += o4.z; y[4 * c + 3] += o4.w;
          }
        }
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) pk[j >> 1] = pack_bf16(y[j], y[j + 1]);
        uint4* dst = reinterpret_cast<uint4*>(orow + half * 32);
#pragma unroll
        for (int c = 0; c < 4; ++c) dst[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
    }
  }
  if (tid == 0) {
    // bounded: return at once when complete; otherwise let them land before TMEM goes
    wait_bar(&bar_ld, 0);
    if (s_oi) wait_bar(&bar_o, 0);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tbase, 256);
}

// ---------------------------------------------------------------------------------
// ssd_scan: state passing over tiles for the lambda-constant special case (Mamba-2
// SSD): prefix_0 = 0, prefix_{u+1} = 2^(gamma_u) prefix_u + H_u, from the tile states
// (level-0 node images) that tc_state published.  One CTA per (b, h) walks the tiles in
// order, thread tid owning row tid; four tiles' images and scalars are in flight ahead
// of it.  prefix_u is published for u >= 1 as an fp16 image (pimg, pmeta).
// ---------------------------------------------------------------------------------
constexpr int kScanRing = 4;
constexpr int kSmemScan = kScanRing * (kImgBytes + 16) + 1024;

__global__ void __launch_bounds__(128) ssd_scan_kernel(TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned* smeta = reinterpret_cast<unsigned*>(smem + kScanRing * kImgBytes);  // 4 u32 per slot
  __shared__ __align__(8) uint64_t bar[kScanRing];
  __shared__ float2 s_red2[4];
  const int tid = threadIdx.x, rot = tid & 7;
  const int bh = blockIdx.x;
  const size_t nbase = (size_t)bh * p.nnodes;  // level-0 node of tile u: nbase + u
  const int nsteps = p.NT - 1;                 // prefixes 1 .. NT-1
  auto issue = [&](int u) {                    // tile u's image and scalars into slot u % 4
    const int k = u % kScanRing;
    ptx::mbar_arrive_expect_tx(&bar[k], kImgBytes + 16);
    ptx::bulk_load(smem + k * kImgBytes, p.img + (nbase + u) * kImgBytes, kImgBytes, &bar[k]);
    ptx::bulk_load(smeta + 4 * k, p.meta + (nbase + u) * kMeta, 16, &bar[k]);
  };
  int issued = 0;
  if (tid == 0) {
    for (int k = 0; k < kScanRing; ++k) ptx::mbar_init(&bar[k], 1);
    ptx::fence_mbar_init();
    for (; issued < kScanRing && issued < nsteps; ++issued) issue(issued);
  }
  __syncthreads();
  float acc[kDv];
#pragma unroll
  for (int j = 0; j < kDv; ++j) acc[j] = 0.f;
  int u = 0;
  bool ok = true;
  for (; u < nsteps; ++u) {
    const int k = u % kScanRing;
    ok = wait_bar(&bar[k], (u / kScanRing) & 1);
    if (!ok) atomicExch(p.status, kStatusTimeout);
    ok = __syncthreads_and(ok);
    if (!ok) break;
    const float sc = pow2i((int)smeta[4 * k + 1]);
    const float dg = exp2f(__uint_as_float(smeta[4 * k + 2]));
    const uint8_t* row = smem + k * kImgBytes + tid * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 x4 = *reinterpret_cast<const uint4*>(row + ((c ^ rot) << 4));
      const __half2* hx = reinterpret_cast<const __half2*>(&x4);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(hx[e]);
        acc[8 * c + 2 * e] = dg * acc[8 * c + 2 * e] + sc * f.x;
        acc[8 * c + 2 * e + 1] = dg * acc[8 * c + 2 * e + 1] + sc * f.y;
      }
    }
    // prefix_{u+1}, staged over slot k (row tid was read by this thread only)
    publish_node(acc, smem + k * kImgBytes, (size_t)bh * p.NT + u + 1, 0.f, s_red2, p.pimg, p.pmeta);
    __syncthreads();  // every thread has stored its part of the staged image
    if (tid == 0 && issued < nsteps) {
      ptx::fence_proxy_async_smem();
      issue(issued++);
    }
  }
  if (!ok && tid == 0)  // let this CTA's own copies land (bounded) before exit
    for (int v = u; v < issued; ++v) wait_bar(&bar[v % kScanRing], (v / kScanRing) & 1);
}

// ---------------------------------------------------------------------------------
// tc_export: bucket states at position T (T % 128 == 0, so live levels are >= 8).
// ---------------------------------------------------------------------------------
// One CTA per live level of T (level l >= 1 with bit l-1 of T set) and (b, h); CTA 0 of
// each (b, h) also writes the zero log-scales of all SL slots.  Slots of levels that are
// not live at T are left as they are.
__global__ void __launch_bounds__(256) tc_export_kernel(TcParams p, int SL, float* st, float* lsc) {
  ptx::griddep_wait();  // reads the tree
  const int bh = blockIdx.y;
  if (lsc && blockIdx.x == 0)
    for (int l = threadIdx.x; l < SL; l += 256) lsc[(size_t)bh * SL + l] = 0.f;
  const int lvl = nth_set_bit((unsigned)p.T, blockIdx.x) + 1;
  float* dst = st + ((size_t)bh * SL + lvl) * (kDk * kDv);
  const int m = lvl - kLevIntra;
  const size_t nbase = (size_t)bh * p.nnodes;
  float D = 0.f;
  for (int mm = 0; mm < m; ++mm)
    if ((p.NT >> mm) & 1)
      D += __uint_as_float(p.meta[(nbase + p.node_off[mm] + ((p.NT >> mm) - 1)) * kMeta + 2]);
  const size_t node = nbase + p.node_off[m] + ((p.NT >> m) - 1);
  const float scale = exp2f(D) * pow2i((int)p.meta[node * kMeta + 1]);
  const uint8_t* img = p.img + node * kImgBytes;
  for (int e = threadIdx.x; e < kDk * 8; e += 256) {  // 16-byte chunk c of image row i
    const int i = e >> 3, c = e & 7;
    const uint4 x = *reinterpret_cast<const uint4*>(img + i * 128 + ((c ^ (i & 7)) << 4));
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    float f[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 h2 = __half22float2(*reinterpret_cast<const __half2*>(&w[q]));
      f[2 * q] = scale * h2.x;
      f[2 * q + 1] = scale * h2.y;
    }
    float4* d4 = reinterpret_cast<float4*>(dst + i * kDv + c * 8);
    d4[0] = make_float4(f[0], f[1], f[2], f[3]);
    d4[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
}

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

// ---------------------------------------------------------------------------------
// tc_bwd_intra: the in-tile pairs (levels 0..7) of the backward on the tensor cores.
//
// Chain rule on o_t = sum_{s<=t} lambda_t^{l(t,s)} 2^(g_t - g_s) (q_t . k_s) v_s for the
// loss sum(dO . o), restricted to pairs inside one 128-token tile (u): with S = Q Kᵀ,
// E = dO Vᵀ and w_ts = lambda_t^{l(t,s)} 2^(g_t - g_s) [s <= t],
//   dq = (w ⊙ E) K,  dk = (w ⊙ E)ᵀ Q,  dv = (w ⊙ S)ᵀ dO,
//   dlambda_t^l = sum over s at level l of 2^(g_t - g_s) S_ts E_ts   (l = 0..7),
//   C_s = sum_t w_ts S_ts E_ts (the column sums of the pair terms; with the row sums
//   R_t = sum_l lambda_t^l dlambda_t^l they give d(log a) without the rounding of dv).
// One CTA (256 threads, one per SM: 512 TMEM columns, 175 KB shared memory) per
// (b, h, tile):
//   S and E on the tensor cores from the bf16 inputs (TMEM columns 0..127, 128..255);
//   role a (warps 0-3, thread = query row): dS = w ⊙ E and P = w ⊙ S as fp16 with
//     power-of-two tile scales into shared memory (in the layout a TMA box of 64 columns
//     has), dlambda from S ⊙ E in fp32;
//   role b (warps 4-7): Q, K and dO to fp16 in place with power-of-two tile scales;
//   dq = dS K (columns 256..383), dk = dSᵀ Q (384..511) and dv = Pᵀ dO (0..63) on the
//   tensor cores; dq rows are read by role a, dk and dv rows (keys) by role b, and all
//   three are written to the fp32 per-head gradient buffers (assigned, not added).
// The pairs across tiles are the inter-tile part of the backward.
// ---------------------------------------------------------------------------------
struct TcBwdParams {
  int B, T, H, hpg, G, L, NT;
  const float* a;
  const float* lam;
  float* dq32;   // (B, T, H, d_k) fp32, per head
  float* dk32;   // (B, T, H, d_k)
  float* dv32;   // (B, T, H, d_v)
  float* dlam;   // (B, T, H, L): levels 0..7 written, the rest zeroed
  float* cu;     // (B, T, H): C_s = sum_t A_ts over the in-tile pairs (fp32, from S and E)
  unsigned* status;
};

// Warp reduce-scatter of 32 columns: on return lane j holds the sum over the warp's lanes
// of v[j] (31 shuffles).
__device__ __forceinline__ float warp_colsum32(float (&v)[32], int lane) {
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) {
    const bool up = (lane & k) != 0;
#pragma unroll
    for (int i = 0; i < k; ++i) {
      const float send = up ? v[i] : v[i + k];
      const float keep = up ? v[i + k] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, k);
    }
  }
  return v[0];
}

constexpr int kBwdFixed = 163840;  // Q, K, V, dO, dS, P in front of the small tables
constexpr int kSmemBwd = kBwdFixed + 3 * 128 * 4 + 2 * 128 * 9 * 4 + 1024;

// Shared-memory address of the 16-byte chunk holding keys 8c..8c+7 (c = 0..15) of row r of
// a 128 x 128 fp16 tile stored as two 64-column boxes with the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_chunk(int r, int c) {
  return (uint32_t)((c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(256, 1) tc_bwd_intra_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                              const __grid_constant__ CUtensorMap mapK,
                                                              const __grid_constant__ CUtensorMap mapV,
                                                              const __grid_constant__ CUtensorMap mapD,
                                                              TcBwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* RQ = smem;            // 32 KB: Q (bf16, then fp16)
  uint8_t* RK = smem + 32768;    // 32 KB: K (bf16, then fp16)
  uint8_t* RV = smem + 65536;    // 16 KB: V (bf16)
  uint8_t* RD = smem + 81920;    // 16 KB: dO (bf16, then fp16)
  uint8_t* RS = smem + 98304;    // 32 KB: dS (fp16)
  uint8_t* RP = smem + 131072;   // 32 KB: P (fp16)
  float* sG = reinterpret_cast<float*>(smem + kBwdFixed);  // 128: g
  float* sB8 = sG + 128;                                    // 128: 2^(g_end8(s) - g_s)
  float* sLam8 = sB8 + 128;                                 // 128 x 9: lambda levels 0..7 of row r
  float* sAcc = sLam8 + 128 * 9;                            // 128 x 9: dlambda of the diagonal group
  float* sCol = sAcc + 128 * 9;                             // 128: column sums C_s
  __shared__ __align__(8) uint64_t bar_ld, bar_se, bar_mm;
  __shared__ uint32_t tmem_base;
  __shared__ float s_red[8];
  __shared__ float s_mx[8][3];
  __shared__ int s_sc[6];  // tile scale exponents: dS, P (role a); Q, K, dO (role b)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127, quad = warp & 3, rot = r & 7;
  const bool role_b = warp >= 4;
  const int lin = blockIdx.x;
  const int h = lin % p.H;
  const int u = (lin / p.H) % p.NT;
  const int b = lin / (p.H * p.NT);
  const int g = h / p.hpg;
  const long long t0 = (long long)u * kTile;
  const size_t row = (size_t)b * p.T + t0 + r;  // token of this thread's row
  const float* lrow = p.lam + (row * p.H + h) * p.L;

  if (tid == 0) {
    ptx::mbar_init(&bar_ld, 1);
    ptx::mbar_init(&bar_se, 1);
    ptx::mbar_init(&bar_mm, 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(&bar_ld, 32768 * 2 + 16384 * 2);
    ptx::tma_load_4d(RQ, &mapQ, &bar_ld, 0, g, (int)t0, b);
    ptx::tma_load_4d(RQ + 16384, &mapQ, &bar_ld, 64, g, (int)t0, b);
    ptx::tma_load_4d(RK, &mapK, &bar_ld, 0, g, (int)t0, b);
    ptx::tma_load_4d(RK + 16384, &mapK, &bar_ld, 64, g, (int)t0, b);
    ptx::tma_load_4d(RV, &mapV, &bar_ld, 0, h, (int)t0, b);
    ptx::tma_load_4d(RD, &mapD, &bar_ld, 0, h, (int)t0, b);
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 512);
    ptx::tmem_relinquish();
  }
  if (!role_b) {
#pragma unroll
    for (int l = 0; l < kLevIntra; ++l) ptx::cp_async4(sLam8 + r * 9 + l, lrow + l);
#pragma unroll
    for (int l = 0; l < 9; ++l) sAcc[r * 9 + l] = 0.f;
    sCol[r] = 0.f;
  }
  // chunk-local log2 decay cumsum over the 128 rows (both roles compute it)
  float gt = log2f(p.a[row * p.H + h]);
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, gt, off);
    if (lane >= off) gt += y;
  }
  if (lane == 31) s_red[warp] = gt;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  for (int w = 0; w < quad; ++w) gt += s_red[w];
  const uint32_t tbase = tmem_base;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t tS = tbase, tE = tbase + 128, tDQ = tbase + 256, tDK = tbase + 384, tDV = tbase;
  if (!role_b) sG[r] = gt;
  __syncthreads();
  if (!role_b) sB8[r] = exp2f(sG[r | 7] - gt);
  bool ok = wait_bar(&bar_ld, 0);
  if (!ok) atomicExch(p.status, kStatusTimeout);
  ok = __syncthreads_and(ok);

  // S = Q Kᵀ (K = 128 d_k) and E = dO Vᵀ (K = 64 d_v), bf16, all K-major
  if (ok && tid == 128) {
    ptx::tc_fence_after();
    const uint32_t idesc = ptx::idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t q0 = ptx::smem_u32(RQ), k0 = ptx::smem_u32(RK);
    const uint32_t d0 = ptx::smem_u32(RD), v0 = ptx::smem_u32(RV);
#pragma unroll
    for (int kk = 0; kk < kDk / 16; ++kk) {
      const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
      ptx::umma_f16(tS, ptx::smem_desc_sw128(q0 + off, 16, 1024), ptx::smem_desc_sw128(k0 + off, 16, 1024),
                    idesc, kk > 0);
    }
#pragma unroll
    for (int kk = 0; kk < kDv / 16; ++kk)
      ptx::umma_f16(tE, ptx::smem_desc_sw128(d0 + kk * 32, 16, 1024), ptx::smem_desc_sw128(v0 + kk * 32, 16, 1024),
                    idesc, kk > 0);
    ptx::umma_commit(&bar_se);
  }
  const bool se_issued = ok;
  if (ok) {
    ok = wait_bar(&bar_se, 0);
    if (!ok) atomicExch(p.status, kStatusTimeout);
  }
  ok = __syncthreads_and(ok);  // also: S and E no longer read Q, K, V, dO

  if (!role_b) {
    // ---- role a: dS and P into shared memory, dlambda ------------------------------
    const int t = r, tl = t & 31;
    const float* lamr = sLam8 + r * 9;
    float lmax = 0.f, smax = 0.f, emax = 0.f;
    ptx::cp_async_wait_all();  // lambda of this row (issued by this thread)
    if (ok) {
      ptx::tc_fence_after();
#pragma unroll
      for (int l = 0; l < kLevIntra; ++l) lmax = fmaxf(lmax, fabsf(lamr[l]));
#pragma unroll 1
      for (int cg = 0; cg <= quad; ++cg) {
        float sv[32], ev[32];
        ptx::tmem_ld32(tS + lane_off + cg * 32, sv);
        ptx::tmem_ld32(tE + lane_off + cg * 32, ev);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (cg < quad || j <= tl) {
            smax = fmaxf(smax, fabsf(sv[j]));
            emax = fmaxf(emax, fabsf(ev[j]));
          }
      }
    }
    // tile maxima of |P| <= max|S| max lambda and |dS| <= max|E| max lambda (decays <= 1)
    float mp = smax * lmax, ms = emax * lmax;
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, off));
      ms = fmaxf(ms, __shfl_xor_sync(0xffffffffu, ms, off));
    }
    if (lane == 0) {
      s_mx[warp][0] = ms;
      s_mx[warp][1] = mp;
    }
    ptx::named_bar_sync(1, 128);
    const int es = f16_exp(fmaxf(fmaxf(s_mx[0][0], s_mx[1][0]), fmaxf(s_mx[2][0], s_mx[3][0])));
    const int ep = f16_exp(fmaxf(fmaxf(s_mx[0][1], s_mx[1][1]), fmaxf(s_mx[2][1], s_mx[3][1])));
    if (tid == 0) {
      s_sc[0] = es;
      s_sc[1] = ep;
    }
    const float cs = pow2i(-es), cp = pow2i(-ep);
    float acc6 = 0.f, acc7 = 0.f;
    const float* gq = sG + quad * 32;
    const float span8 = fmaxf(fmaxf(gq[0] - gq[7], gq[8] - gq[15]), fmaxf(gq[16] - gq[23], gq[24] - gq[31]));
    const bool fastd = span8 <= 60.f;
#pragma unroll 1
    for (int cg = 0; cg < 4; ++cg) {
      uint32_t pd[16], pp[16];
      if (ok && cg < quad) {
        // keys of an earlier 32-group: one level (6 or 7) and the factored decay
        float sv[32], ev[32];
        ptx::tmem_ld32(tS + lane_off + cg * 32, sv);
        ptx::tmem_ld32(tE + lane_off + cg * 32, ev);
        ptx::tmem_ld_wait();
        const bool l7 = (quad ^ cg) >= 2;
        const float lv = lamr[l7 ? 7 : 6];
        float ak[4];
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) ak[kb] = exp2f(gt - sG[cg * 32 + kb * 8 + 7]);
        const float4* b4 = reinterpret_cast<const float4*>(sB8 + cg * 32);
        float xs = 0.f;
        float colv[32];
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 bb = b4[j4];
          const float bj[4] = {bb.x, bb.y, bb.z, bb.w};
          float vs[4], vp[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            const float dd = ak[j4 >> 1] * bj[e];
            const float xj = dd * (sv[j] * ev[j]);
            xs += xj;
            colv[j] = lv * xj;
            const float w = lv * dd;
            vs[e] = (w * cs) * ev[j];
            vp[e] = (w * cp) * sv[j];
          }
          pd[2 * j4] = pack_h2(vs[0], vs[1]);
          pd[2 * j4 + 1] = pack_h2(vs[2], vs[3]);
          pp[2 * j4] = pack_h2(vp[0], vp[1]);
          pp[2 * j4 + 1] = pack_h2(vp[2], vp[3]);
        }
        if (l7) acc7 += xs;
        else acc6 += xs;
        atomicAdd(sCol + cg * 32 + lane, warp_colsum32(colv, lane));
      } else if (ok && cg == quad) {
        // the diagonal 32-group: levels 0..5 (level of key j: bit length of tl ^ j)
        float sv[32], ev[32];
        ptx::tmem_ld32(tS + lane_off + cg * 32, sv);
        ptx::tmem_ld32(tE + lane_off + cg * 32, ev);
        ptx::tmem_ld_wait();
        float ak[4];
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) ak[kb] = exp2f(gt - gq[kb * 8 + 7]);
        const float4* b4 = reinterpret_cast<const float4*>(sB8 + cg * 32);
        float* accr = sAcc + r * 9;
        float colv[32];
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 bb = b4[j4];
          const float bj[4] = {bb.x, bb.y, bb.z, bb.w};
          float vs[4], vp[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            // blocks after t's may give ak = inf; their keys are masked by the select
            const float dd = fastd ? ak[j >> 3] * bj[e] : exp2f(gt - gq[j]);
            const int lvj = 32 - __clz(tl ^ j);
            const bool on = j <= tl;
            const float w = on ? lamr[lvj] * dd : 0.f;
            vs[e] = (w * cs) * ev[j];
            vp[e] = (w * cp) * sv[j];
            const float xj = on ? dd * (sv[j] * ev[j]) : 0.f;
            if (on) accr[lvj] += xj;
            colv[j] = on ? lamr[lvj] * xj : 0.f;
          }
          pd[2 * j4] = pack_h2(vs[0], vs[1]);
          pd[2 * j4 + 1] = pack_h2(vs[2], vs[3]);
          pp[2 * j4] = pack_h2(vp[0], vp[1]);
          pp[2 * j4 + 1] = pack_h2(vp[2], vp[3]);
        }
        atomicAdd(sCol + cg * 32 + lane, warp_colsum32(colv, lane));
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) pd[j] = pp[j] = 0u;
      }
      // keys cg*32 .. cg*32+31 are chunks 4cg .. 4cg+3 of row r
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t off = tile_chunk(r, 4 * cg + q4);
        *reinterpret_cast<uint4*>(RS + off) = make_uint4(pd[4 * q4], pd[4 * q4 + 1], pd[4 * q4 + 2], pd[4 * q4 + 3]);
        *reinterpret_cast<uint4*>(RP + off) = make_uint4(pp[4 * q4], pp[4 * q4 + 1], pp[4 * q4 + 2], pp[4 * q4 + 3]);
      }
    }
    ptx::fence_proxy_async_smem();
    ptx::named_bar_sync(1, 128);  // column sums complete
    if (ok) {
      p.cu[row * p.H + h] = sCol[r];
      float* dl = p.dlam + (row * p.H + h) * p.L;
      const float* accr = sAcc + r * 9;
#pragma unroll
      for (int l = 0; l < 6; ++l) dl[l] = accr[l];
      dl[6] = acc6 + accr[6];
      dl[7] = acc7 + accr[7];
      for (int l = kLevIntra; l < p.L; ++l) dl[l] = 0.f;  // inter-tile levels: added later
    }
  } else {
    // ---- role b: Q, K, dO -> fp16 in place with tile scales ---------------------------
    uint32_t mq = 0u, mk = 0u, md = 0u;
    uint8_t* qr0 = RQ + r * 128;
    uint8_t* kr0 = RK + r * 128;
    uint8_t* dr0 = RD + r * 128;
    if (ok) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int cc = (c ^ rot) << 4;
        mq = absmax_u4(absmax_u4(mq, *reinterpret_cast<const uint4*>(qr0 + cc)),
                       *reinterpret_cast<const uint4*>(qr0 + 16384 + cc));
        mk = absmax_u4(absmax_u4(mk, *reinterpret_cast<const uint4*>(kr0 + cc)),
                       *reinterpret_cast<const uint4*>(kr0 + 16384 + cc));
        md = absmax_u4(md, *reinterpret_cast<const uint4*>(dr0 + cc));
      }
    }
    float fq = bf16x2_maxhalf(mq), fk = bf16x2_maxhalf(mk), fd = bf16x2_maxhalf(md);
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      fq = fmaxf(fq, __shfl_xor_sync(0xffffffffu, fq, off));
      fk = fmaxf(fk, __shfl_xor_sync(0xffffffffu, fk, off));
      fd = fmaxf(fd, __shfl_xor_sync(0xffffffffu, fd, off));
    }
    if (lane == 0) {
      s_mx[warp][0] = fq;
      s_mx[warp][1] = fk;
      s_mx[warp][2] = fd;
    }
    ptx::named_bar_sync(2, 128);
    int ex[3];
#pragma unroll
    for (int i = 0; i < 3; ++i)
      ex[i] = f16_exp(fmaxf(fmaxf(s_mx[4][i], s_mx[5][i]), fmaxf(s_mx[6][i], s_mx[7][i])));
    if (tid == 128) {
      s_sc[2] = ex[0];
      s_sc[3] = ex[1];
      s_sc[4] = ex[2];
    }
    if (ok) {
      const float sq = pow2i(-ex[0]), sk = pow2i(-ex[1]), sd = pow2i(-ex[2]);
      const __nv_bfloat162 q2 = __floats2bfloat162_rn(sq, sq), k2 = __floats2bfloat162_rn(sk, sk),
                           d2 = __floats2bfloat162_rn(sd, sd);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int cc = (c ^ rot) << 4;
        uint4* a0 = reinterpret_cast<uint4*>(qr0 + cc);
        uint4* a1 = reinterpret_cast<uint4*>(qr0 + 16384 + cc);
        uint4* b0 = reinterpret_cast<uint4*>(kr0 + cc);
        uint4* b1 = reinterpret_cast<uint4*>(kr0 + 16384 + cc);
        uint4* d0 = reinterpret_cast<uint4*>(dr0 + cc);
        *a0 = bf16x8_to_f16x8(*a0, q2);
        *a1 = bf16x8_to_f16x8(*a1, q2);
        *b0 = bf16x8_to_f16x8(*b0, k2);
        *b1 = bf16x8_to_f16x8(*b1, k2);
        *d0 = bf16x8_to_f16x8(*d0, d2);
      }
      ptx::fence_proxy_async_smem();
    }
  }
  ptx::tc_fence_before();
  ok = __syncthreads_and(ok);  // dS, P, fp16 Q, K, dO and the scales complete; S, E read

  // dq = dS K (keys), dk = dSᵀ Q and dv = Pᵀ dO (queries); fp16
  if (ok && tid == 128) {
    ptx::tc_fence_after();
    const uint32_t s0 = ptx::smem_u32(RS), p0 = ptx::smem_u32(RP), q0 = ptx::smem_u32(RQ),
                   k0 = ptx::smem_u32(RK), d0 = ptx::smem_u32(RD);
    const uint32_t id_q = ptx::idesc_f16_f32(128, 128, 0, 1);
    const uint32_t id_k = ptx::idesc_f16_f32(128, 128, 1, 1);
    const uint32_t id_v = ptx::idesc_f16_f32(128, 64, 1, 1);
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk) {
      const uint32_t offk = (kk >> 2) * 16384 + (kk & 3) * 32;  // K-major step over keys
      ptx::umma_f16(tDQ, ptx::smem_desc_sw128(s0 + offk, 16, 1024), ptx::smem_desc_sw128(k0 + kk * 2048, 16384, 1024),
                    id_q, kk > 0);
      ptx::umma_f16(tDK, ptx::smem_desc_sw128(s0 + kk * 2048, 16384, 1024),
                    ptx::smem_desc_sw128(q0 + kk * 2048, 16384, 1024), id_k, kk > 0);
      ptx::umma_f16(tDV, ptx::smem_desc_sw128(p0 + kk * 2048, 16384, 1024),
                    ptx::smem_desc_sw128(d0 + kk * 2048, 1024, 1024), id_v, kk > 0);
    }
    ptx::umma_commit(&bar_mm);
  }
  const bool mm_issued = ok;
  if (ok) {
    ok = wait_bar(&bar_mm, 0);
    if (!ok) atomicExch(p.status, kStatusTimeout);
  }
  ok = __all_sync(0xffffffffu, ok);
  if (ok) {
    ptx::tc_fence_after();
    if (!role_b) {
      const float sc = pow2s(s_sc[0] + s_sc[3]);  // dS and K
      float* dst = p.dq32 + (row * p.H + h) * kDk;
#pragma unroll 1
      for (int c0 = 0; c0 < kDk; c0 += 32) {
        float y[32];
        ptx::tmem_ld32(tDQ + lane_off + c0, y);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(sc * y[j], sc * y[j + 1], sc * y[j + 2], sc * y[j + 3]);
      }
    } else {
      const float sk = pow2s(s_sc[0] + s_sc[2]);  // dS and Q
      const float sv = pow2s(s_sc[1] + s_sc[4]);  // P and dO
      float* dk = p.dk32 + (row * p.H + h) * kDk;
      float* dv = p.dv32 + (row * p.H + h) * kDv;
#pragma unroll 1
      for (int c0 = 0; c0 < kDk + kDv; c0 += 32) {
        const bool isk = c0 < kDk;
        float y[32];
        ptx::tmem_ld32((isk ? tDK + c0 : tDV + (c0 - kDk)) + lane_off, y);
        ptx::tmem_ld_wait();
        const float s = isk ? sk : sv;
        float* d = isk ? dk + c0 : dv + (c0 - kDk);
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(d + j) = make_float4(s * y[j], s * y[j + 1], s * y[j + 2], s * y[j + 3]);
      }
    }
  }
  if (tid == 128) {  // bounded: let this CTA's copies and MMAs land before TMEM goes
    wait_bar(&bar_ld, 0);
    if (se_issued) wait_bar(&bar_se, 0);
    if (mm_issued) wait_bar(&bar_mm, 0);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------------------------
// tc_bwd_q: the query side of the inter-tile levels of the backward on the tensor cores.
//
// With the forward's tree over tiles (node images and scalars), tile u reads for every set
// bit m of u the node N = Node_m[(u >> m) - 1] with weight w_t = lambda_t^(8+m) 2^(g_t + D_m)
// (o_t += w_t q_tᵀ N).  Its backward, per level:
//   dq_t += w_t N dO_t                   Z = dO Nᵀ, added into registers with w_t;
//   dlambda_t^(8+m) = 2^(g_t + D_m) q_tᵀ N dO_t    Y = Q N, dotted with dO_t;
//   dual(N) += sum_t w_t q_t dO_tᵀ       Qᵀ diag(w) dO, added into the node's fp32 dual
//                                        with vector atomics (the readers of a node are
//                                        the 2^m tiles of the node after it).
// One CTA (256 threads, two per SM) per (b, h, tile) with u > 0; levels nearest first,
// node images two deep.  Q, dO fp16 with power-of-two tile scales, diag(w) dO fp16 with
// a power-of-two scale per level.  Thread (row t, half hf) keeps d_k columns 64 hf ..
// 64 hf + 63 of dq_t; half 0 does the dlambda dot; the dual rows (d_k index = TMEM lane)
// are split by d_v halves.  dq is added to the per-head fp32 buffer (the in-tile part
// wrote it); dlambda levels >= 8 are assigned (the in-tile kernel zeroed them).
// ---------------------------------------------------------------------------------
struct TcBwdQParams {
  int B, T, H, hpg, G, L, NT, nnodes;
  int node_off[32];
  int dual_off[32];   // first dual slot of the even nodes of tile level m
  int nslots;         // dual slots per (b, h)
  const float* a;
  const float* lam;
  const uint8_t* img;
  const unsigned* meta;
  float* dq32;
  float* dlam;
  float* dual;        // (B*H, nslots, d_k, d_v) fp32, zero on entry
  unsigned* status;
};

constexpr int kBwdQFixed = 98304;  // Q, dO, two node images, diag(w) dO
__host__ __device__ constexpr int bwdq_smem_bytes(int ninter) {
  return kBwdQFixed + 512 * (ninter > 0 ? ninter : 1) + 1024;
}

__global__ void __launch_bounds__(256, 2) tc_bwd_q_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                          const __grid_constant__ CUtensorMap mapD,
                                                          TcBwdQParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* RQ = smem;             // 32 KB: Q (bf16, then fp16)
  uint8_t* RD = smem + 32768;     // 16 KB: dO (bf16, then fp16)
  uint8_t* RI = smem + 49152;     // 2 x 16 KB: node images
  uint8_t* RB = smem + 81920;     // 16 KB: diag(w) dO of the current level (fp16)
  float* sLamI = reinterpret_cast<float*>(smem + kBwdQFixed);  // [level index][row]
  __shared__ __align__(8) uint64_t bar_ld, bar_y, bar_e[2], bar_yf;
  __shared__ uint32_t tmem_base;
  __shared__ float s_red[8];
  __shared__ float s_mx[8][2];
  __shared__ unsigned s_lmax[32];
  __shared__ float sNode[32][2];  // per level index: scale exponent (bits), log2 decay

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127, hf = tid >> 7, quad = warp & 3, rot = r & 7;
  const int lin = blockIdx.x;
  const int h = lin % p.H;
  const int u = (lin / p.H) % p.NT;
  const int b = lin / (p.H * p.NT);
  const int nlev = __popc((unsigned)u);
  if (nlev == 0) return;  // the first tile reads no node
  const int g = h / p.hpg;
  const int bh = b * p.H + h;
  const long long t0 = (long long)u * kTile;
  const size_t nbase = (size_t)bh * p.nnodes;
  const size_t row = (size_t)b * p.T + t0 + r;
  const float* lrow = p.lam + (row * p.H + h) * p.L;
  auto node_of = [&](int i) {
    const int m = nth_set_bit((unsigned)u, i);
    return nbase + p.node_off[m] + ((u >> m) - 1);
  };

  if (tid == 0) {
    ptx::mbar_init(&bar_ld, 1);
    ptx::mbar_init(&bar_y, 1);
    ptx::mbar_init(&bar_e[0], 1);
    ptx::mbar_init(&bar_e[1], 1);
    ptx::mbar_init(&bar_yf, 256);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(&bar_ld, 32768 + 16384);
    ptx::tma_load_4d(RQ, &mapQ, &bar_ld, 0, g, (int)t0, b);
    ptx::tma_load_4d(RQ + 16384, &mapQ, &bar_ld, 64, g, (int)t0, b);
    ptx::tma_load_4d(RD, &mapD, &bar_ld, 0, h, (int)t0, b);
    for (int i = 0; i < 2 && i < nlev; ++i) {
      ptx::mbar_arrive_expect_tx(&bar_e[i], kImgBytes);
      ptx::bulk_load(RI + i * kImgBytes, p.img + node_of(i) * kImgBytes, kImgBytes, &bar_e[i]);
    }
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 256);
    ptx::tmem_relinquish();
  }
  if (tid < 32) s_lmax[tid] = 0u;
  if (hf == 0)
    for (int i = 0; i < nlev; ++i) ptx::cp_async4(sLamI + i * 128 + r, lrow + kLevIntra + nth_set_bit((unsigned)u, i));
  if (tid < nlev) {
    const unsigned* mt = p.meta + node_of(tid) * kMeta;
    sNode[tid][0] = __uint_as_float(mt[1]);
    sNode[tid][1] = __uint_as_float(mt[2]);
  }
  // chunk-local log2 decay cumsum over the 128 rows (both halves compute it)
  float gt = log2f(p.a[row * p.H + h]);
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, gt, off);
    if (lane >= off) gt += y;
  }
  if (lane == 31) s_red[warp] = gt;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  for (int w = 0; w < quad; ++w) gt += s_red[w];
  const uint32_t tbase = tmem_base;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t tZ = tbase, tY = tbase + 128, tU = tbase + 192;
  bool ok = wait_bar(&bar_ld, 0);
  if (!ok) atomicExch(p.status, kStatusTimeout);
  ok = __syncthreads_and(ok);

  // Q (half hf converts box hf of row r) and dO (half 0) -> fp16 with tile scales
  uint8_t* qrow = RQ + hf * 16384 + r * 128;
  uint8_t* drow = RD + r * 128;
  {
    uint32_t mq = 0u, md = 0u;
    if (ok) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        mq = absmax_u4(mq, *reinterpret_cast<const uint4*>(qrow + ((c ^ rot) << 4)));
        if (hf == 0) md = absmax_u4(md, *reinterpret_cast<const uint4*>(drow + ((c ^ rot) << 4)));
      }
    }
    float fq = bf16x2_maxhalf(mq), fd = bf16x2_maxhalf(md);
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      fq = fmaxf(fq, __shfl_xor_sync(0xffffffffu, fq, off));
      fd = fmaxf(fd, __shfl_xor_sync(0xffffffffu, fd, off));
    }
    if (lane == 0) {
      s_mx[warp][0] = fq;
      s_mx[warp][1] = fd;
    }
  }
  ptx::cp_async_wait_all();
  __syncthreads();  // maxima; lambda rows
  float maxq = 0.f, maxd = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    maxq = fmaxf(maxq, s_mx[w][0]);
    maxd = fmaxf(maxd, s_mx[w][1]);
  }
  const int eq = f16_exp(maxq), ed = f16_exp(maxd);
  if (ok) {
    const float sq = pow2i(-eq), sd = pow2i(-ed);
    const __nv_bfloat162 q2 = __floats2bfloat162_rn(sq, sq), d2 = __floats2bfloat162_rn(sd, sd);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4* x = reinterpret_cast<uint4*>(qrow + ((c ^ rot) << 4));
      *x = bf16x8_to_f16x8(*x, q2);
      if (hf == 0) {
        uint4* y = reinterpret_cast<uint4*>(drow + ((c ^ rot) << 4));
        *y = bf16x8_to_f16x8(*y, d2);
      }
    }
    if (hf == 0)
      for (int i = 0; i < nlev; ++i) atomicMax(&s_lmax[i], __float_as_uint(fabsf(sLamI[i * 128 + r])));
  }
  __syncthreads();  // fp16 Q, dO; lambda maxima
  // level weights: w_t = lambda_t^(8+m) 2^(g_t + D) (D: the nearer levels' decay)
  auto weight = [&](int i, float D) { return sLamI[i * 128 + r] * exp2f(gt + D); };
  // diag(w) dO 2^-tau for level i: row r, d_v columns 32 hf .. 32 hf + 31 (chunks 4 hf ..)
  auto write_b = [&](int i, float D, int tau) {
    const float f = weight(i, D) * pow2s(ed - tau);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int cc = ((4 * hf + c) ^ rot) << 4;
      const uint4 x = *reinterpret_cast<const uint4*>(drow + cc);
      const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
      uint32_t o4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
        o4[e] = pack_h2(f * v.x, f * v.y);
      }
      *reinterpret_cast<uint4*>(RB + r * 128 + cc) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
  };
  auto tau_of = [&](int i) { return f16_exp(__uint_as_float(s_lmax[i]) * maxd); };
  float D = 0.f;
  if (ok) write_b(0, 0.f, tau_of(0));
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  ok = __syncthreads_and(ok);

  float acc[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) acc[j] = 0.f;
  int issued = nlev < 2 ? nlev : 2, consumed = 0, y_issued = 0;
  const uint32_t id_z = ptx::idesc_f16_f32(128, 128, 0, 0);
  const uint32_t id_y = ptx::idesc_f16_f32(128, 64, 0, 1);
  const uint32_t id_u = ptx::idesc_f16_f32(128, 64, 1, 1);
  for (int i = 0; ok && i < nlev; ++i) {
    const int m = nth_set_bit((unsigned)u, i);
    if (tid == 0) {
      bool okd = i == 0 || wait_bar(&bar_yf, (i - 1) & 1);   // TMEM read, next diag(w) dO written
      okd = okd && wait_bar(&bar_e[i & 1], (i >> 1) & 1);    // image landed
      if (okd) {
        ++consumed;
        ptx::tc_fence_after();
        const uint32_t im = ptx::smem_u32(RI + (i & 1) * kImgBytes);
        const uint32_t q0 = ptx::smem_u32(RQ), d0 = ptx::smem_u32(RD), b0 = ptx::smem_u32(RB);
#pragma unroll
        for (int kk = 0; kk < kDv / 16; ++kk)  // Z = dO Nᵀ: K = d_v, B = image rows (d_k) K-major
          ptx::umma_f16(tZ, ptx::smem_desc_sw128(d0 + kk * 32, 16, 1024), ptx::smem_desc_sw128(im + kk * 32, 16, 1024),
                        id_z, kk > 0);
#pragma unroll
        for (int kk = 0; kk < kDk / 16; ++kk) {
          const uint32_t offq = (kk >> 2) * 16384 + (kk & 3) * 32;
          ptx::umma_f16(tY, ptx::smem_desc_sw128(q0 + offq, 16, 1024), ptx::smem_desc_sw128(im + kk * 2048, 1024, 1024),
                        id_y, kk > 0);  // Y = Q N
        }
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)  // Qᵀ diag(w) dO: M = d_k, K = tokens
          ptx::umma_f16(tU, ptx::smem_desc_sw128(q0 + kk * 2048, 16384, 1024),
                        ptx::smem_desc_sw128(b0 + kk * 2048, 1024, 1024), id_u, kk > 0);
        ptx::umma_commit(&bar_y);
        ++y_issued;
      } else {
        atomicExch(p.status, kStatusTimeout);
      }
    }
    bool okw = wait_bar(&bar_y, i & 1);
    if (!okw) atomicExch(p.status, kStatusTimeout);
    okw = __syncthreads_and(okw);
    if (!okw) {
      ok = false;
      break;
    }
    if (tid == 0 && i + 2 < nlev) {  // the image buffer of level i is free again
      ptx::mbar_arrive_expect_tx(&bar_e[i & 1], kImgBytes);
      ptx::bulk_load(RI + (i & 1) * kImgBytes, p.img + node_of(i + 2) * kImgBytes, kImgBytes, &bar_e[i & 1]);
      ++issued;
    }
    ptx::tc_fence_after();
    const int en = __float_as_int(sNode[i][0]);
    const float wt = weight(i, D);
    {  // dq: columns 64 hf .. 64 hf + 63 of Z, weighted
      const float wz = wt * pow2s(ed + en);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float y[32];
        ptx::tmem_ld32(tZ + lane_off + hf * 64 + half * 32, y);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[half * 32 + j] += wz * y[j];
      }
    }
    if (hf == 0) {  // dlambda_t^(8+m) = 2^(g_t + D + eq + en + ed) sum_j Y_tj dO^_tj
      float dot = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float y[32];
        ptx::tmem_ld32(tY + lane_off + half * 32, y);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 x = *reinterpret_cast<const uint4*>(drow + (((4 * half + c) ^ rot) << 4));
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
            dot += y[c * 8 + 2 * e] * v.x + y[c * 8 + 2 * e + 1] * v.y;
          }
        }
      }
      p.dlam[(row * p.H + h) * p.L + kLevIntra + m] = exp2f(gt + D) * pow2s(eq + en + ed) * dot;
    }
    {  // dual rows (TMEM lane = d_k index r), d_v columns 32 hf .. 32 hf + 31
      const int tau = tau_of(i);
      const float su = pow2s(eq + tau);
      float y[32];
      ptx::tmem_ld32(tU + lane_off + hf * 32, y);
      ptx::tmem_ld_wait();
      const int nd = (u >> m) - 1;  // even
      float* dst = p.dual + (((size_t)bh * p.nslots + p.dual_off[m] + (nd >> 1)) * kDk + r) * kDv + hf * 32;
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        atomicAdd(reinterpret_cast<float4*>(dst + j), make_float4(su * y[j], su * y[j + 1], su * y[j + 2], su * y[j + 3]));
    }
    D += sNode[i][1];
    if (i + 1 < nlev) {  // diag(w) dO of the next level (its MMA has read this one)
      write_b(i + 1, D, tau_of(i + 1));
      ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(&bar_yf);
  }
  if (ok) {
    float* dst = p.dq32 + (row * p.H + h) * kDk + hf * 64;
#pragma unroll
    for (int j = 0; j < 64; j += 4) {
      float4 o = *reinterpret_cast<float4*>(dst + j);
      o.x += acc[j];
      o.y += acc[j + 1];
      o.z += acc[j + 2];
      o.w += acc[j + 3];
      *reinterpret_cast<float4*>(dst + j) = o;
    }
  }
  if (tid == 0) {  // bounded: let this CTA's copies and MMAs land before TMEM goes
    wait_bar(&bar_ld, 0);
    for (int j = consumed; j < issued; ++j) wait_bar(&bar_e[j & 1], (j >> 1) & 1);
    if (y_issued > 0) wait_bar(&bar_y, (y_issued - 1) & 1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tbase, 256);
}

// ---------------------------------------------------------------------------------
// Key side of the inter-tile levels of the backward.
//
// tc_tile_prefix: per (b, h) the running sum P[c] of the tile decays gamma_0 .. gamma_{c-1}
//   (the log2 decays of the level-0 nodes), in fp64, c = 0 .. NT.
// tc_dual_publish: every dual slot as an fp16 image with a power-of-two scale (the node
//   publication of the tree), for use as an MMA operand.
// tc_bwd_kv: per key tile u and every tile level m whose node (m, i = u >> m) is read
//   (i even, node (m, i + 1) inside the sequence), with c_m = 2^(P[(i+1) 2^m] - P[u+1])
//   the decay of the tiles after u inside the node and r_s = 2^(gamma_u - g_s):
//     dk_s += r_s sum_m c_m Dual_m v_s,   dv_s += r_s sum_m c_m Dual_mᵀ k_s,
//   as Zk = V Dualᵀ and Zv = K Dual on the tensor cores (V, K fp16 with tile scales),
//   added into registers per level (512 threads: four per key row, 32 d_k and 16 d_v
//   columns each), then added to the per-head fp32 buffers.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tc_tile_prefix_kernel(const unsigned* meta, int nnodes, int NT,
                                                             double* P) {
  __shared__ double s_part[8];
  __shared__ double s_carry;
  const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_carry = 0.0;
  double* out = P + (size_t)bh * (NT + 1);
  if (tid == 0) out[0] = 0.0;
  __syncthreads();
  for (int c0 = 0; c0 < NT; c0 += 256) {
    const int c = c0 + tid;
    double x = c < NT ? (double)__uint_as_float(meta[((size_t)bh * nnodes + c) * kMeta + 2]) : 0.0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_part[warp] = x;
    __syncthreads();
    double add = s_carry;
    for (int w = 0; w < warp; ++w) add += s_part[w];
    x += add;
    if (c < NT) out[c + 1] = x;
    __syncthreads();
    if (tid == 255) s_carry = x;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(128) tc_dual_publish_kernel(const float* dual, uint8_t* img, unsigned* meta) {
  __shared__ __align__(1024) uint8_t stage[kImgBytes];
  __shared__ float2 s_red2[4];
  const size_t slot = blockIdx.x;
  const float* src = dual + (slot * kDk + threadIdx.x) * kDv;
  float cur[kDv];
#pragma unroll
  for (int j = 0; j < kDv; j += 4) {
    const float4 v = *reinterpret_cast<const float4*>(src + j);
    cur[j] = v.x;
    cur[j + 1] = v.y;
    cur[j + 2] = v.z;
    cur[j + 3] = v.w;
  }
  publish_node(cur, stage, slot, 0.f, s_red2, img, meta);
}

struct TcBwdKVParams {
  int B, T, H, hpg, G, NT, MT;
  int dual_off[32];
  int nslots;
  const float* a;
  const uint8_t* dimg;    // dual images (B*H, nslots, 16 KB)
  const unsigned* dmeta;  // (B*H, nslots, 4): scale exponent in [1]
  const double* P;        // (B*H, NT + 1)
  float* dk32;
  float* dv32;
  float* cu;    // (B, T, H): adds v_s . (the inter-tile part of dv_s)
  unsigned* status;
};

constexpr int kSmemBwdKV = 32768 + 16384 + 2 * kImgBytes + 1024;

__global__ void __launch_bounds__(512, 1) tc_bwd_kv_kernel(const __grid_constant__ CUtensorMap mapK,
                                                           const __grid_constant__ CUtensorMap mapV,
                                                           TcBwdKVParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* RK = smem;           // 32 KB: K (bf16, then fp16)
  uint8_t* RV = smem + 32768;   // 16 KB: V (bf16, then fp16)
  uint8_t* RI = smem + 49152;   // 2 x 16 KB: dual images
  __shared__ __align__(8) uint64_t bar_ld, bar_z, bar_e[2], bar_zf;
  __shared__ uint32_t tmem_base;
  __shared__ float s_red[16];
  __shared__ float s_mx[16][2];
  __shared__ int s_lv[32];
  __shared__ int s_nl;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127, qq = tid >> 7, quad = warp & 3, rot = r & 7;
  const int lin = blockIdx.x;
  const int h = lin % p.H;
  const int u = (lin / p.H) % p.NT;
  const int b = lin / (p.H * p.NT);
  const int g = h / p.hpg;
  const int bh = b * p.H + h;
  const long long t0 = (long long)u * kTile;
  const size_t row = (size_t)b * p.T + t0 + r;
  if (tid == 0) {  // tile levels whose node holding u is read by a later node
    int n = 0;
    for (int m = 0; m < p.MT; ++m) {
      const int i = u >> m;
      if (!(i & 1) && ((long long)(i + 1) << m) < p.NT) s_lv[n++] = m;
    }
    s_nl = n;
  }
  __syncthreads();
  const int nl = s_nl;
  if (nl == 0) return;  // no level reads this tile's nodes
  auto slot_of = [&](int j) {
    const int m = s_lv[j];
    return (size_t)bh * p.nslots + p.dual_off[m] + ((u >> m) >> 1);
  };
  if (tid == 0) {
    ptx::mbar_init(&bar_ld, 1);
    ptx::mbar_init(&bar_z, 1);
    ptx::mbar_init(&bar_e[0], 1);
    ptx::mbar_init(&bar_e[1], 1);
    ptx::mbar_init(&bar_zf, 512);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(&bar_ld, 32768 + 16384);
    ptx::tma_load_4d(RK, &mapK, &bar_ld, 0, g, (int)t0, b);
    ptx::tma_load_4d(RK + 16384, &mapK, &bar_ld, 64, g, (int)t0, b);
    ptx::tma_load_4d(RV, &mapV, &bar_ld, 0, h, (int)t0, b);
    for (int j = 0; j < 2 && j < nl; ++j) {
      ptx::mbar_arrive_expect_tx(&bar_e[j], kImgBytes);
      ptx::bulk_load(RI + j * kImgBytes, p.dimg + slot_of(j) * kImgBytes, kImgBytes, &bar_e[j]);
    }
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 256);
    ptx::tmem_relinquish();
  }
  // tile-local log2 decay cumsum (every quarter computes it for its rows)
  float gt = log2f(p.a[row * p.H + h]);
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, gt, off);
    if (lane >= off) gt += y;
  }
  if (lane == 31) s_red[warp] = gt;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  for (int w = 0; w < quad; ++w) gt += s_red[w];
  const float gam = s_red[0] + s_red[1] + s_red[2] + s_red[3];  // gamma_u
  const uint32_t tbase = tmem_base;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t tZk = tbase, tZv = tbase + 128;
  bool ok = wait_bar(&bar_ld, 0);
  if (!ok) atomicExch(p.status, kStatusTimeout);
  ok = __syncthreads_and(ok);
  // K (quarters 0, 1: boxes 0, 1 of row r) and V (quarter 2) -> fp16 with tile scales
  uint8_t* crow = qq < 2 ? RK + qq * 16384 + r * 128 : RV + r * 128;
  {
    uint32_t mx = 0u;
    if (ok && qq < 3) {
#pragma unroll
      for (int c = 0; c < 8; ++c) mx = absmax_u4(mx, *reinterpret_cast<const uint4*>(crow + ((c ^ rot) << 4)));
    }
    float f = bf16x2_maxhalf(mx);
#pragma unroll
    for (int off = 16; off; off >>= 1) f = fmaxf(f, __shfl_xor_sync(0xffffffffu, f, off));
    if (lane == 0) s_mx[warp][0] = f;
  }
  __syncthreads();
  float mk = 0.f, mv = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) mk = fmaxf(mk, s_mx[w][0]);
#pragma unroll
  for (int w = 8; w < 12; ++w) mv = fmaxf(mv, s_mx[w][0]);
  const int ek = f16_exp(mk), ev = f16_exp(mv);
  if (ok && qq < 3) {
    const float sc = pow2i(qq < 2 ? -ek : -ev);
    const __nv_bfloat162 s2 = __floats2bfloat162_rn(sc, sc);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4* x = reinterpret_cast<uint4*>(crow + ((c ^ rot) << 4));
      *x = bf16x8_to_f16x8(*x, s2);
    }
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  ok = __syncthreads_and(ok);

  float ak[32], av[16];
#pragma unroll
  for (int j = 0; j < 32; ++j) ak[j] = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) av[j] = 0.f;
  const double* P = p.P + (size_t)bh * (p.NT + 1);
  const uint32_t id_k = ptx::idesc_f16_f32(128, 128, 0, 0);
  const uint32_t id_v = ptx::idesc_f16_f32(128, 64, 0, 1);
  int issued = nl < 2 ? nl : 2, consumed = 0, z_issued = 0;
  for (int j = 0; ok && j < nl; ++j) {
    if (tid == 0) {
      bool okd = j == 0 || wait_bar(&bar_zf, (j - 1) & 1);  // Z of the level before read
      okd = okd && wait_bar(&bar_e[j & 1], (j >> 1) & 1);
      if (okd) {
        ++consumed;
        ptx::tc_fence_after();
        const uint32_t im = ptx::smem_u32(RI + (j & 1) * kImgBytes);
        const uint32_t k0 = ptx::smem_u32(RK), v0 = ptx::smem_u32(RV);
#pragma unroll
        for (int kk = 0; kk < kDv / 16; ++kk)  // Zk = V Dualᵀ: K = d_v; the image rows (d_k) K-major
          ptx::umma_f16(tZk, ptx::smem_desc_sw128(v0 + kk * 32, 16, 1024), ptx::smem_desc_sw128(im + kk * 32, 16, 1024),
                        id_k, kk > 0);
#pragma unroll
        for (int kk = 0; kk < kDk / 16; ++kk) {  // Zv = K Dual: K = d_k; the image MN-major
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          ptx::umma_f16(tZv, ptx::smem_desc_sw128(k0 + off, 16, 1024), ptx::smem_desc_sw128(im + kk * 2048, 1024, 1024),
                        id_v, kk > 0);
        }
        ptx::umma_commit(&bar_z);
        ++z_issued;
      } else {
        atomicExch(p.status, kStatusTimeout);
      }
    }
    bool okw = wait_bar(&bar_z, j & 1);
    if (!okw) atomicExch(p.status, kStatusTimeout);
    okw = __syncthreads_and(okw);
    if (!okw) {
      ok = false;
      break;
    }
    if (tid == 0 && j + 2 < nl) {
      ptx::mbar_arrive_expect_tx(&bar_e[j & 1], kImgBytes);
      ptx::bulk_load(RI + (j & 1) * kImgBytes, p.dimg + slot_of(j + 2) * kImgBytes, kImgBytes, &bar_e[j & 1]);
      ++issued;
    }
    ptx::tc_fence_after();
    const int m = s_lv[j];
    const int end = ((u >> m) + 1) << m;
    const float cm = exp2f((float)(P[end] - P[u + 1]));
    const int ed = (int)p.dmeta[slot_of(j) * kMeta + 1];
    {
      float y[32];
      ptx::tmem_ld32(tZk + lane_off + qq * 32, y);
      ptx::tmem_ld_wait();
      const float w = cm * pow2s(ed + ev);
#pragma unroll
      for (int c = 0; c < 32; ++c) ak[c] += w * y[c];
    }
    {
      float y[16];
      ptx::tmem_ld16(tZv + lane_off + qq * 16, y);
      ptx::tmem_ld_wait();
      const float w = cm * pow2s(ed + ek);
#pragma unroll
      for (int c = 0; c < 16; ++c) av[c] += w * y[c];
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(&bar_zf);
  }
  if (ok) {
    const float rs = exp2f(gam - gt);
    float* dk = p.dk32 + (row * p.H + h) * kDk + qq * 32;
    float* dv = p.dv32 + (row * p.H + h) * kDv + qq * 16;
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
      float4 o = *reinterpret_cast<float4*>(dk + c);
      o.x += rs * ak[c];
      o.y += rs * ak[c + 1];
      o.z += rs * ak[c + 2];
      o.w += rs * ak[c + 3];
      *reinterpret_cast<float4*>(dk + c) = o;
    }
#pragma unroll
    for (int c = 0; c < 16; c += 4) {
      float4 o = *reinterpret_cast<float4*>(dv + c);
      o.x += rs * av[c];
      o.y += rs * av[c + 1];
      o.z += rs * av[c + 2];
      o.w += rs * av[c + 3];
      *reinterpret_cast<float4*>(dv + c) = o;
    }
    // v_s . (these d_v columns): V is fp16 in shared memory, 2^ev times the input
    float cdot = 0.f;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 x = *reinterpret_cast<const uint4*>(RV + r * 128 + (((2 * qq + c) ^ rot) << 4));
      const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 vv = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
        cdot += vv.x * av[8 * c + 2 * e] + vv.y * av[8 * c + 2 * e + 1];
      }
    }
    atomicAdd(p.cu + row * p.H + h, rs * pow2i(ev) * cdot);
  }
  if (tid == 0) {  // bounded: let this CTA's copies and MMAs land before TMEM goes
    wait_bar(&bar_ld, 0);
    for (int j = consumed; j < issued; ++j) wait_bar(&bar_e[j & 1], (j >> 1) & 1);
    if (z_issued > 0) wait_bar(&bar_z, (z_issued - 1) & 1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tbase, 256);
}

// ---------------------------------------------------------------------------------
// Gated DeltaNet values on the tensor cores, 128-token chunks (the delta rule's WY form,
// as in gdn.cu: u = U_loc - W S per chunk, T = (I + diag(beta) A)^-1, A = (K Kᵀ) ⊙
// 2^(g_t - g_s) strictly lower, U_loc = T diag(beta) V, W = T diag(beta 2^g) K).
//
// tc_gdn_local, one CTA per (b, h, chunk), 256 threads, one CTA per SM:
//   K Kᵀ on tcgen05 from the bf16 keys (exact products, fp32 sums); A in fp32 in shared
//   memory; T by 16-row blocks on the CUDA cores (diagonal blocks by substitution in
//   registers, then T_ij = -T_ii sum_{j <= k < i} A_ik T_kj column block by column block);
//   then [W | U_loc] = T [diag(beta 2^g) K | diag(beta) V] on tcgen05 with every operand
//   split into an fp16 high part and the fp16 rounding remainder (hi hi + lo hi + hi lo,
//   about 22 significant bits), each with a power-of-two tile scale.  Per chunk the
//   workspace gets W split the same way (hi and lo fp16 in the MMA operand layout, with
//   its scale exponent), U_loc (fp32) and g, for tc_gdn_pass.
// ---------------------------------------------------------------------------------
// Workspace per (b, h, chunk): W hi, W lo (fp16, 16 KB boxes of 64 d_k columns with the
// 128-byte swizzle), U_loc (128 x d_v fp32), g (128 fp32), W's scale exponent.
constexpr int kGdnOffU = 65536, kGdnOffG = 65536 + 32768, kGdnOffE = kGdnOffG + 512;
constexpr size_t kGdnChunkBytes = 99328;

struct TcGdnParams {
  int B, T, H, hpg, G;
  const float* a;
  const float* beta;
  uint8_t* xw;  // (B*H, T/128, kGdnChunkBytes)
  void* u;      // (B, T, H, d_v) bf16: the transformed values (tc_gdn_pass)
  unsigned* status;
};

constexpr int kGP = 132;  // padded fp32 row of the 128 x 128 matrices
constexpr int kSmemGdnL = 32768 + 16384 + 2 * 128 * kGP * 4 + 8 * 256 * 4 + 4 * 128 * 4 + 1024;

// fp32 value -> fp16 high part and fp16 remainder, both of x * 2^-e
__device__ __forceinline__ void split_h(float x, float sc, __half& hi, __half& lo) {
  const float y = x * sc;
  hi = __float2half_rn(y);
  lo = __float2half_rn(y - __half2float(hi));
}

__global__ void __launch_bounds__(256, 1) tc_gdn_local_kernel(const __grid_constant__ CUtensorMap mapK,
                                                              const __grid_constant__ CUtensorMap mapV,
                                                              TcGdnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* RK = smem;                                          // 32 KB: K (bf16); later V hi, lo (fp16)
  uint8_t* RV = smem + 32768;                                  // 16 KB: V (bf16)
  float* Am = reinterpret_cast<float*>(smem + 49152);          // 128 x kGP: A; later T hi, lo (fp16)
  float* Tm = Am + 128 * kGP;                                  // 128 x kGP: T; later Kd hi, lo (fp16)
  float* Ym = Tm + 128 * kGP;                                  // 8 x (16 x 16): one per warp
  float* gs = Ym + 8 * 256;                                    // 128: g
  float* bs = gs + 128;                                        // 128: beta
  float* fk = bs + 128;                                        // 128: beta 2^g
  __shared__ __align__(8) uint64_t bar_ld, bar_a, bar_w;
  __shared__ uint32_t tmem_base;
  __shared__ float s_red[8];
  __shared__ float s_mx[8][3];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3;
  const int r = tid & 127, rot = r & 7;
  const int nch = p.T >> 7;
  const int lin = blockIdx.x;
  const int h = lin % p.H;
  const int c = (lin / p.H) % nch;
  const int b = lin / (p.H * nch);
  const int g = h / p.hpg;
  const long long t0 = (long long)c * kTile;
  const size_t row = (size_t)b * p.T + t0 + r;
  if (tid == 0) {
    ptx::mbar_init(&bar_ld, 1);
    ptx::mbar_init(&bar_a, 1);
    ptx::mbar_init(&bar_w, 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(&bar_ld, 32768 + 16384);
    ptx::tma_load_4d(RK, &mapK, &bar_ld, 0, g, (int)t0, b);
    ptx::tma_load_4d(RK + 16384, &mapK, &bar_ld, 64, g, (int)t0, b);
    ptx::tma_load_4d(RV, &mapV, &bar_ld, 0, h, (int)t0, b);
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 256);
    ptx::tmem_relinquish();
  }
  // chunk-local log2 decay cumsum (both halves of the block compute it)
  float gt = log2f(p.a[row * p.H + h]);
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, gt, off);
    if (lane >= off) gt += y;
  }
  if (lane == 31) s_red[warp] = gt;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  for (int w = 0; w < quad; ++w) gt += s_red[w];
  const uint32_t tbase = tmem_base;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t tA = tbase, tW = tbase + 128, tU = tbase;
  if (tid < 128) {
    const float bt = p.beta[row * p.H + h];
    gs[r] = gt;
    bs[r] = bt;
    fk[r] = bt * exp2f(gt);
  }
  bool ok = wait_bar(&bar_ld, 0);
  if (!ok) atomicExch(p.status, kStatusTimeout);
  ok = __syncthreads_and(ok);
  if (ok && tid == 0) {  // K Kᵀ: M = N = 128 tokens, K = 128 d_k, bf16, both K-major
    ptx::tc_fence_after();
    const uint32_t idesc = ptx::idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t k0 = ptx::smem_u32(RK);
#pragma unroll
    for (int kk = 0; kk < kDk / 16; ++kk) {
      const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
      ptx::umma_f16(tA, ptx::smem_desc_sw128(k0 + off, 16, 1024), ptx::smem_desc_sw128(k0 + off, 16, 1024), idesc,
                    kk > 0);
    }
    ptx::umma_commit(&bar_a);
  }
  const bool a_issued = ok;
  if (ok) {
    ok = wait_bar(&bar_a, 0);
    if (!ok) atomicExch(p.status, kStatusTimeout);
  }
  ok = __syncthreads_and(ok);
  // A_ts = beta_t 2^(g_t - g_s) (k_t . k_s), s < t (threads 0..127: row t); T zeroed above
  if (ok) {
    ptx::tc_fence_after();
    if (tid < 128) {
      const int t = r;
      const float bt = bs[t];
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        float y[32];
        ptx::tmem_ld32(tA + lane_off + c0, y);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 v;
          float* vv = reinterpret_cast<float*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s2 = c0 + j + e;
            vv[e] = s2 < t ? bt * exp2f(gt - gs[s2]) * y[j + e] : 0.f;
          }
          *reinterpret_cast<float4*>(Am + t * kGP + c0 + j) = v;
        }
      }
    } else {
      for (int e = r; e < 128 * kGP; e += 128) Tm[e] = 0.f;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // diagonal 16 x 16 blocks of T: thread (block, column j), substitution in registers
  if (ok && tid < 128) {
    const int r0 = tid & ~15, j = tid & 15;
    float x[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      float acc = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < t; ++s2) acc += Am[(r0 + t) * kGP + r0 + s2] * x[s2];
      x[t] = t < j ? 0.f : (t == j ? 1.f : -acc);
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) Tm[(r0 + t) * kGP + r0 + j] = x[t];
  }
  __syncthreads();
  // blocks below the diagonal, column block by column block (each needs only the diagonal
  // blocks and its own earlier ones):
  //   Y = sum_{jb <= k < ib} A_{ib,k} T_{k,jb},  T_{ib,jb} = -T_{ib,ib} Y,  ib = jb+1 .. 7.
  // The work of column block jb falls with jb: blocks 0, 1, 2 go to warp pairs (rows
  // split, a 64-thread barrier per step), blocks 3 + 6 and 4 + 5 to single warps.
  if (ok) {
    const bool pair = warp < 6;
    const int njb = pair ? 1 : 2;
    const int jb0 = pair ? (warp >> 1) : (warp == 6 ? 3 : 4);
    float* Yw = Ym + (pair ? (warp >> 1) : warp - 3) * 256;
    for (int q = 0; q < njb; ++q) {
      const int jb = q == 0 ? jb0 : 9 - jb0;  // 3 then 6, 4 then 5
      for (int ib = jb + 1; ib < 8; ++ib) {
        if (pair) {  // rows 8 (warp & 1) + lane / 4, columns 4 (lane % 4) .. + 3
          const int rr = (warp & 1) * 8 + (lane >> 2), c0 = (lane & 3) * 4;
          float y0 = 0.f, y1 = 0.f, y2 = 0.f, y3 = 0.f;
          const float* arow = Am + (16 * ib + rr) * kGP;
#pragma unroll 4
          for (int s2 = 16 * jb; s2 < 16 * ib; ++s2) {
            const float av = arow[s2];
            const float4 tv = *reinterpret_cast<const float4*>(Tm + s2 * kGP + 16 * jb + c0);
            y0 += av * tv.x; y1 += av * tv.y; y2 += av * tv.z; y3 += av * tv.w;
          }
          *reinterpret_cast<float4*>(Yw + rr * 16 + c0) = make_float4(y0, y1, y2, y3);
          ptx::named_bar_sync(1 + (warp >> 1), 64);
          float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
          const float* trow = Tm + (16 * ib + rr) * kGP + 16 * ib;
#pragma unroll 4
          for (int s2 = 0; s2 < 16; ++s2) {
            const float tv = trow[s2];
            const float4 yv = *reinterpret_cast<const float4*>(Yw + s2 * 16 + c0);
            x0 += tv * yv.x; x1 += tv * yv.y; x2 += tv * yv.z; x3 += tv * yv.w;
          }
          *reinterpret_cast<float4*>(Tm + (16 * ib + rr) * kGP + 16 * jb + c0) = make_float4(-x0, -x1, -x2, -x3);
          ptx::named_bar_sync(1 + (warp >> 1), 64);
        } else {  // row lane / 2, columns 8 (lane % 2) .. + 7
          const int rr = lane >> 1, c0 = (lane & 1) * 8;
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = 0.f;
          const float* arow = Am + (16 * ib + rr) * kGP;
#pragma unroll 4
          for (int s2 = 16 * jb; s2 < 16 * ib; ++s2) {
            const float av = arow[s2];
            const float4 t0v = *reinterpret_cast<const float4*>(Tm + s2 * kGP + 16 * jb + c0);
            const float4 t1v = *reinterpret_cast<const float4*>(Tm + s2 * kGP + 16 * jb + c0 + 4);
            y[0] += av * t0v.x; y[1] += av * t0v.y; y[2] += av * t0v.z; y[3] += av * t0v.w;
            y[4] += av * t1v.x; y[5] += av * t1v.y; y[6] += av * t1v.z; y[7] += av * t1v.w;
          }
          *reinterpret_cast<float4*>(Yw + rr * 16 + c0) = make_float4(y[0], y[1], y[2], y[3]);
          *reinterpret_cast<float4*>(Yw + rr * 16 + c0 + 4) = make_float4(y[4], y[5], y[6], y[7]);
          __syncwarp();
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.f;
          const float* trow = Tm + (16 * ib + rr) * kGP + 16 * ib;
#pragma unroll 4
          for (int s2 = 0; s2 < 16; ++s2) {
            const float tv = trow[s2];
            const float4 y0 = *reinterpret_cast<const float4*>(Yw + s2 * 16 + c0);
            const float4 y1 = *reinterpret_cast<const float4*>(Yw + s2 * 16 + c0 + 4);
            x[0] += tv * y0.x; x[1] += tv * y0.y; x[2] += tv * y0.z; x[3] += tv * y0.w;
            x[4] += tv * y1.x; x[5] += tv * y1.y; x[6] += tv * y1.z; x[7] += tv * y1.w;
          }
          float* dst = Tm + (16 * ib + rr) * kGP + 16 * jb + c0;
          *reinterpret_cast<float4*>(dst) = make_float4(-x[0], -x[1], -x[2], -x[3]);
          *reinterpret_cast<float4*>(dst + 4) = make_float4(-x[4], -x[5], -x[6], -x[7]);
          __syncwarp();
        }
      }
    }
  }
  __syncthreads();
  // tile scales of T, diag(beta 2^g) K, diag(beta) V (maxima over their elements)
  {
    float mt = 0.f, mk = 0.f, mv = 0.f;
    if (ok) {
      // thread: T row r, half (tid >> 7) of its columns; K and V rows r (tid < 128)
      const float* trow = Tm + r * kGP + (tid >> 7) * 64;
      for (int j = 0; j < 64; ++j) mt = fmaxf(mt, fabsf(trow[j]));
      if (tid < 128) {
        uint32_t m0 = 0u, m1 = 0u;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const int off = r * 128 + ((cc ^ rot) << 4);
          m0 = absmax_u4(absmax_u4(m0, *reinterpret_cast<const uint4*>(RK + off)),
                         *reinterpret_cast<const uint4*>(RK + 16384 + off));
          m1 = absmax_u4(m1, *reinterpret_cast<const uint4*>(RV + off));
        }
        mk = bf16x2_maxhalf(m0) * fabsf(fk[r]);
        mv = bf16x2_maxhalf(m1) * fabsf(bs[r]);
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, off));
      mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
    }
    if (lane == 0) {
      s_mx[warp][0] = mt;
      s_mx[warp][1] = mk;
      s_mx[warp][2] = mv;
    }
  }
  __syncthreads();
  float mxs[3] = {0.f, 0.f, 0.f};
#pragma unroll
  for (int w = 0; w < 8; ++w)
#pragma unroll
    for (int i = 0; i < 3; ++i) mxs[i] = fmaxf(mxs[i], s_mx[w][i]);
  const int et = f16_exp(mxs[0]), ek = f16_exp(mxs[1]), ev = f16_exp(mxs[2]);
  // T -> fp16 hi, lo (A operands, K-major: row t, columns s in two 64-wide boxes) over A
  uint8_t* THI = reinterpret_cast<uint8_t*>(Am);
  uint8_t* TLO = THI + 32768;
  if (ok) {
    const float sc = pow2i(-et);
    const int hf = tid >> 7;  // this thread's box (columns 64 hf .. 64 hf + 63) of row r
#pragma unroll 1
    for (int cc = 0; cc < 8; ++cc) {
      const float* src = Tm + r * kGP + hf * 64 + cc * 8;
      __half hi[8], lo[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) split_h(src[e], sc, hi[e], lo[e]);
      const uint32_t off = hf * 16384 + r * 128 + ((cc ^ rot) << 4);
      *reinterpret_cast<uint4*>(THI + off) = *reinterpret_cast<const uint4*>(hi);
      *reinterpret_cast<uint4*>(TLO + off) = *reinterpret_cast<const uint4*>(lo);
    }
  }
  __syncthreads();  // T read: its space takes diag(beta 2^g) K
  // diag(beta 2^g) K -> fp16 hi, lo (B operands, MN-major: row s, d_k in two 64-wide boxes)
  uint8_t* KHI = reinterpret_cast<uint8_t*>(Tm);
  uint8_t* KLO = KHI + 32768;
  if (ok) {
    const float sc = fk[r] * pow2i(-ek);
    const int hf = tid >> 7;
#pragma unroll 1
    for (int cc = 0; cc < 8; ++cc) {
      const uint32_t off = hf * 16384 + r * 128 + ((cc ^ rot) << 4);
      const uint4 x = *reinterpret_cast<const uint4*>(RK + off);
      const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
      __half hi[8], lo[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        split_h(__uint_as_float(w4[e] << 16), sc, hi[2 * e], lo[2 * e]);
        split_h(__uint_as_float(w4[e] & 0xffff0000u), sc, hi[2 * e + 1], lo[2 * e + 1]);
      }
      *reinterpret_cast<uint4*>(KHI + off) = *reinterpret_cast<const uint4*>(hi);
      *reinterpret_cast<uint4*>(KLO + off) = *reinterpret_cast<const uint4*>(lo);
    }
  }
  __syncthreads();  // K read: its space takes diag(beta) V
  uint8_t* VHI = RK;
  uint8_t* VLO = RK + 16384;
  if (ok && tid < 128) {
    const float sc = bs[r] * pow2i(-ev);
#pragma unroll 1
    for (int cc = 0; cc < 8; ++cc) {
      const uint32_t off = r * 128 + ((cc ^ rot) << 4);
      const uint4 x = *reinterpret_cast<const uint4*>(RV + off);
      const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
      __half hi[8], lo[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        split_h(__uint_as_float(w4[e] << 16), sc, hi[2 * e], lo[2 * e]);
        split_h(__uint_as_float(w4[e] & 0xffff0000u), sc, hi[2 * e + 1], lo[2 * e + 1]);
      }
      *reinterpret_cast<uint4*>(VHI + off) = *reinterpret_cast<const uint4*>(hi);
      *reinterpret_cast<uint4*>(VLO + off) = *reinterpret_cast<const uint4*>(lo);
    }
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  ok = __syncthreads_and(ok);
  // W = T Kd and U = T Vd, each as hi hi + lo hi + hi lo (fp16, fp32 accumulation)
  if (ok && tid == 0) {
    ptx::tc_fence_after();
    const uint32_t id_w = ptx::idesc_f16_f32(128, 128, 0, 1);
    const uint32_t id_u = ptx::idesc_f16_f32(128, 64, 0, 1);
    const uint32_t ta[3] = {ptx::smem_u32(THI), ptx::smem_u32(TLO), ptx::smem_u32(THI)};
    const uint32_t kb[3] = {ptx::smem_u32(KHI), ptx::smem_u32(KHI), ptx::smem_u32(KLO)};
    const uint32_t vb[3] = {ptx::smem_u32(VHI), ptx::smem_u32(VHI), ptx::smem_u32(VLO)};
#pragma unroll
    for (int pass = 0; pass < 3; ++pass)
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        const uint64_t da = ptx::smem_desc_sw128(ta[pass] + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        ptx::umma_f16(tW, da, ptx::smem_desc_sw128(kb[pass] + kk * 2048, 16384, 1024), id_w, pass > 0 || kk > 0);
        ptx::umma_f16(tU, da, ptx::smem_desc_sw128(vb[pass] + kk * 2048, 1024, 1024), id_u, pass > 0 || kk > 0);
      }
    ptx::umma_commit(&bar_w);
  }
  const bool w_issued = ok;
  if (ok) {
    ok = wait_bar(&bar_w, 0);
    if (!ok) atomicExch(p.status, kStatusTimeout);
  }
  ok = __all_sync(0xffffffffu, ok);
  // W: its tile maximum, then hi and lo fp16 of W 2^-ew in the operand layout; U_loc, g
  uint8_t* dst = p.xw + ((size_t)(b * p.H + h) * nch + c) * kGdnChunkBytes;
  const float sw = pow2s(et + ek), su = pow2s(et + ev);
  float mw = 0.f;
  if (ok && tid < 128) {
    ptx::tc_fence_after();
#pragma unroll 1
    for (int c0 = 0; c0 < kDk; c0 += 32) {
      float y[32];
      ptx::tmem_ld32(tW + lane_off + c0, y);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) mw = fmaxf(mw, fabsf(y[j]));
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, off));
  if (lane == 0) s_red[warp] = mw;
  __syncthreads();
  const int ew = f16_exp(sw * fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3])));
  if (ok && tid < 128) {
    const float sc = sw * pow2i(-ew);
#pragma unroll 1
    for (int c0 = 0; c0 < kDk; c0 += 32) {
      float y[32];
      ptx::tmem_ld32(tW + lane_off + c0, y);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {  // d_k columns c0 + 8 q4 .. + 7: one 16-byte chunk
        const int col = c0 + 8 * q4, bx = col >> 6, cc = (col & 63) >> 3;
        __half hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) split_h(y[8 * q4 + e], sc, hi[e], lo[e]);
        const size_t off = (size_t)bx * 16384 + r * 128 + ((cc ^ rot) << 4);
        *reinterpret_cast<uint4*>(dst + off) = *reinterpret_cast<const uint4*>(hi);
        *reinterpret_cast<uint4*>(dst + 32768 + off) = *reinterpret_cast<const uint4*>(lo);
      }
    }
    float* du = reinterpret_cast<float*>(dst + kGdnOffU);
#pragma unroll 1
    for (int c0 = 0; c0 < kDv; c0 += 32) {
      float y[32];
      ptx::tmem_ld32(tU + lane_off + c0, y);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(du + r * kDv + c0 + j) = make_float4(su * y[j], su * y[j + 1], su * y[j + 2], su * y[j + 3]);
    }
    reinterpret_cast<float*>(dst + kGdnOffG)[r] = gt;
    if (r == 0) *reinterpret_cast<int*>(dst + kGdnOffE) = ew;
  }
  if (tid == 0) {  // bounded: let this CTA's copies and MMAs land before TMEM goes
    wait_bar(&bar_ld, 0);
    if (a_issued) wait_bar(&bar_a, 0);
    if (w_issued) wait_bar(&bar_w, 0);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tbase, 256);
}

// tc_gdn_pass, one CTA per (b, h), chunks in order, 256 threads, one CTA per SM.  The
// state is kept in TMEM as Ŝ = S 2^-sigma (d_k rows as lanes, d_v columns).  Per chunk:
//   Ŝ -> fp16 hi, lo with a tile scale (the B operand); Z = W S as hi hi + lo hi + hi lo;
//   u = U_loc - Z, written in bf16; ũ = 2^(g_end - g) u -> fp16 hi, lo; K -> fp16;
//   Ŝ <- Ŝ 2^(g_end + sigma - sigma') in TMEM, then Ŝ += Kᵀ (ũ hi + ũ lo) with
//   sigma' = the scales of K and ũ.  W (hi and lo) is copied one chunk ahead, K by TMA
//   behind the product W S.
constexpr int kSmemGdnP = 2 * 65536 + 3 * 32768 + 1024;

__global__ void __launch_bounds__(256, 1) tc_gdn_pass_kernel(const __grid_constant__ CUtensorMap mapK,
                                                             TcGdnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* RWb = smem;           // 2 x 64 KB: W hi | W lo of a chunk
  uint8_t* RS = smem + 131072;   // 32 KB: Ŝ hi | lo (B of W S: rows d_k, 64 d_v)
  uint8_t* RU = smem + 163840;   // 32 KB: ũ hi | lo (B of Kᵀ ũ: rows tokens, 64 d_v)
  uint8_t* RK = smem + 196608;   // 32 KB: K (bf16, then fp16; MN-major A of Kᵀ ũ)
  __shared__ __align__(8) uint64_t bar_w[2], bar_k, bar_z, bar_su;
  __shared__ uint32_t tmem_base;
  __shared__ float s_mx[8][2];
  __shared__ float sg[128];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3;
  const int r = tid & 127, hf = tid >> 7, rot = r & 7;
  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H, g = h / p.hpg;
  const int nch = p.T >> 7;
  const uint8_t* xw = p.xw + (size_t)bh * nch * kGdnChunkBytes;
  __nv_bfloat16* uo = static_cast<__nv_bfloat16*>(p.u);
  if (tid == 0) {
    ptx::mbar_init(&bar_w[0], 1);
    ptx::mbar_init(&bar_w[1], 1);
    ptx::mbar_init(&bar_k, 1);
    ptx::mbar_init(&bar_z, 1);
    ptx::mbar_init(&bar_su, 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(&bar_w[0], 65536);
    ptx::bulk_load(RWb, xw, 65536, &bar_w[0]);
    ptx::mbar_arrive_expect_tx(&bar_k, 32768);
    ptx::tma_load_4d(RK, &mapK, &bar_k, 0, g, 0, b);
    ptx::tma_load_4d(RK + 16384, &mapK, &bar_k, 64, g, 0, b);
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 128);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t tS = tbase + hf * 32, tZ = tbase + 64 + hf * 32;  // this thread's 32 columns
  {
    uint32_t z[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) z[j] = 0u;
    ptx::tmem_st16(tS + lane_off, z);
    ptx::tmem_st16(tS + lane_off + 16, z);
    ptx::tmem_st_wait();
  }
  int sigma = 0;
  bool ok = true;
  int w_issued = 1, w_done = 0, k_issued = 1, k_done = 0, mma_z = 0, z_done = 0, mma_s = 0, s_done = 0;
  const uint32_t id_z = ptx::idesc_f16_f32(128, 64, 0, 1);
  const uint32_t id_s = ptx::idesc_f16_f32(128, 64, 1, 1);
  for (int c = 0; ok && c < nch; ++c) {
    const uint8_t* xc = xw + (size_t)c * kGdnChunkBytes;
    if (tid == 0 && c + 1 < nch) {  // W of the next chunk (its buffer's W S has completed)
      ptx::mbar_arrive_expect_tx(&bar_w[(c + 1) & 1], 65536);
      ptx::bulk_load(RWb + ((c + 1) & 1) * 65536, xc + kGdnChunkBytes, 65536, &bar_w[(c + 1) & 1]);
      ++w_issued;
    }
    const int tokr = c * kTile + r;  // this thread's token (rows of u, Z)
    // this thread's half of U_loc row r, and g
    float uu[32];
    {
      const float4* us = reinterpret_cast<const float4*>(xc + kGdnOffU) + (r * kDv + hf * 32) / 4;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 v = us[j];
        uu[4 * j] = v.x;
        uu[4 * j + 1] = v.y;
        uu[4 * j + 2] = v.z;
        uu[4 * j + 3] = v.w;
      }
      if (tid < 128) sg[r] = reinterpret_cast<const float*>(xc + kGdnOffG)[r];
    }
    const int ew = *reinterpret_cast<const int*>(xc + kGdnOffE);
    // Ŝ (lane r = d_k row) -> tile maximum
    float sv[32];
    ptx::tc_fence_after();
    ptx::tmem_ld32(tS + lane_off, sv);
    ptx::tmem_ld_wait();
    float ms = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) ms = fmaxf(ms, fabsf(sv[j]));
#pragma unroll
    for (int off = 16; off; off >>= 1) ms = fmaxf(ms, __shfl_xor_sync(0xffffffffu, ms, off));
    if (lane == 0) s_mx[warp][0] = ms;
    __syncthreads();
    float mxs = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) mxs = fmaxf(mxs, s_mx[w][0]);
    const int es = f16_exp(mxs);
    {  // Ŝ 2^-es -> hi, lo: row r, d_v columns 32 hf .. (chunks 4 hf ..)
      const float sc = pow2i(-es);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        __half hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) split_h(sv[8 * q4 + e], sc, hi[e], lo[e]);
        const int off = r * 128 + (((4 * hf + q4) ^ rot) << 4);
        *reinterpret_cast<uint4*>(RS + off) = *reinterpret_cast<const uint4*>(hi);
        *reinterpret_cast<uint4*>(RS + 16384 + off) = *reinterpret_cast<const uint4*>(lo);
      }
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // Z = W S (M = 128 tokens, N = 64, K = 128 d_k)
      bool okw = wait_bar(&bar_w[c & 1], (c >> 1) & 1);
      if (okw) {
        ++w_done;
        ptx::tc_fence_after();
        const uint32_t w0 = ptx::smem_u32(RWb + (c & 1) * 65536), s0 = ptx::smem_u32(RS);
        const uint32_t wa[3] = {w0, w0 + 32768, w0};
        const uint32_t sb[3] = {s0, s0, s0 + 16384};
#pragma unroll
        for (int pass = 0; pass < 3; ++pass)
#pragma unroll
          for (int kk = 0; kk < kDk / 16; ++kk)
            ptx::umma_f16(tbase + 64, ptx::smem_desc_sw128(wa[pass] + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                          ptx::smem_desc_sw128(sb[pass] + kk * 2048, 1024, 1024), id_z, pass > 0 || kk > 0);
        ptx::umma_commit(&bar_z);
        ++mma_z;
      } else {
        atomicExch(p.status, kStatusTimeout);
      }
    }
    bool okz = wait_bar(&bar_z, c & 1);
    if (!okz) atomicExch(p.status, kStatusTimeout);
    okz = __syncthreads_and(okz);
    if (okz) ++z_done;
    if (!okz) {
      ok = false;
      break;
    }
    ptx::tc_fence_after();
    // u = U_loc - Z (row r = token), written in bf16; ũ = 2^(g_end - g_r) u
    const float gend = sg[127];
    const float zs = pow2s(ew + sigma + es);
    float z[32];
    ptx::tmem_ld32(tZ + lane_off, z);
    ptx::tmem_ld_wait();
    const float fu = exp2f(gend - sg[r]);
    float mu = 0.f;
    {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        z[j] = uu[j] - zs * z[j];  // u
        uu[j] = fu * z[j];         // ũ
        mu = fmaxf(mu, fabsf(uu[j]));
      }
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[j] = pack_bf16(z[2 * j], z[2 * j + 1]);
      uint4* dst = reinterpret_cast<uint4*>(uo + (((size_t)b * p.T + tokr) * p.H + h) * kDv + hf * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
    // K of this chunk (by TMA, behind W S): tile maximum
    bool okk = true;
    if (tid == 0) {
      okk = wait_bar(&bar_k, c & 1);
      if (okk) ++k_done;
      else atomicExch(p.status, kStatusTimeout);
    }
    okk = __syncthreads_and(okk);
    if (!okk) {
      ok = false;
      break;
    }
    uint8_t* krow = RK + hf * 16384 + r * 128;  // this thread's box of key row r
    uint32_t mk = 0u;
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) mk = absmax_u4(mk, *reinterpret_cast<const uint4*>(krow + ((cc ^ rot) << 4)));
    float fk = bf16x2_maxhalf(mk);
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, off));
      fk = fmaxf(fk, __shfl_xor_sync(0xffffffffu, fk, off));
    }
    if (lane == 0) {
      s_mx[warp][0] = mu;
      s_mx[warp][1] = fk;
    }
    __syncthreads();
    float mxu = 0.f, mxk = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      mxu = fmaxf(mxu, s_mx[w][0]);
      mxk = fmaxf(mxk, s_mx[w][1]);
    }
    const int eu = f16_exp(mxu), ek = f16_exp(mxk);
    {  // ũ 2^-eu -> hi, lo (row r = token, d_v columns 32 hf ..); K -> fp16 2^-ek in place
      const float sc = pow2i(-eu);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        __half hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) split_h(uu[8 * q4 + e], sc, hi[e], lo[e]);
        const int off = r * 128 + (((4 * hf + q4) ^ rot) << 4);
        *reinterpret_cast<uint4*>(RU + off) = *reinterpret_cast<const uint4*>(hi);
        *reinterpret_cast<uint4*>(RU + 16384 + off) = *reinterpret_cast<const uint4*>(lo);
      }
      const float sk = pow2i(-ek);
      const __nv_bfloat162 k2 = __floats2bfloat162_rn(sk, sk);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint4* x = reinterpret_cast<uint4*>(krow + ((cc ^ rot) << 4));
        *x = bf16x8_to_f16x8(*x, k2);
      }
    }
    // Ŝ <- Ŝ 2^(g_end + sigma - (ek + eu)) (the new scale of the state)
    {
      const float f = exp2f(gend + (float)(sigma - (ek + eu)));
      uint32_t o[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(f * sv[j]);
      ptx::tmem_st16(tS + lane_off, o);
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(f * sv[16 + j]);
      ptx::tmem_st16(tS + lane_off + 16, o);
      ptx::tmem_st_wait();
    }
    sigma = ek + eu;
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // Ŝ += Kᵀ (ũ hi + ũ lo): M = 128 d_k, N = 64, K = 128 tokens
      ptx::tc_fence_after();
      const uint32_t k0 = ptx::smem_u32(RK), u0 = ptx::smem_u32(RU);
#pragma unroll
      for (int pass = 0; pass < 2; ++pass)
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          ptx::umma_f16(tbase, ptx::smem_desc_sw128(k0 + kk * 2048, 16384, 1024),
                        ptx::smem_desc_sw128(u0 + pass * 16384 + kk * 2048, 1024, 1024), id_s, 1);
      ptx::umma_commit(&bar_su);
      ++mma_s;
    }
    bool oks = wait_bar(&bar_su, c & 1);
    if (!oks) atomicExch(p.status, kStatusTimeout);
    oks = __syncthreads_and(oks);
    if (oks) ++s_done;
    if (!oks) {
      ok = false;
      break;
    }
    if (tid == 0 && c + 1 < nch) {  // K of the next chunk (Kᵀ ũ has read this one)
      ptx::mbar_arrive_expect_tx(&bar_k, 32768);
      ptx::tma_load_4d(RK, &mapK, &bar_k, 0, g, (c + 1) * kTile, b);
      ptx::tma_load_4d(RK + 16384, &mapK, &bar_k, 64, g, (c + 1) * kTile, b);
      ++k_issued;
    }
  }
  if (tid == 0) {  // bounded: let this CTA's outstanding copies and MMAs land before TMEM goes
    for (int j = w_done; j < w_issued; ++j) wait_bar(&bar_w[j & 1], (j >> 1) & 1);
    for (int j = k_done; j < k_issued; ++j) wait_bar(&bar_k, j & 1);
    if (z_done < mma_z) wait_bar(&bar_z, (mma_z - 1) & 1);
    if (s_done < mma_s) wait_bar(&bar_su, (mma_s - 1) & 1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tbase, 128);
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
constexpr int kSmemTree = 4 * kImgBytes + 1024;

}  // namespace

bool tc_supported(const ll_shape& s) {
  return s.dtype == LL_BF16 && s.d_k == kDk && s.d_v == kDv && s.T % kTile == 0 &&
         s.levels <= 32 && bit_length(s.T / kTile - 1) <= kMaxInter && encode_fn() != nullptr;
}

const char* tc_kernel_names(bool with_export) {
  return with_export ? "tc_state,tc_tree,tc_output,tc_export" : "tc_state,tc_tree,tc_output";
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
  p->off_img = o;
  o = a256(o + BH * p->nnodes * (size_t)kImgBytes);
  p->off_meta = o;
  p->meta_bytes = sizeof(unsigned) * BH * p->nnodes * kMeta;
  o = a256(o + p->meta_bytes);
  p->bytes = o;
  return true;
}

namespace {

// Launch that may begin while the previous launch on the stream is finishing
// (programmatic stream serialisation); the kernel waits (griddep_wait) before it reads
// anything that launch wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

bool tc_setup(const TcPlan& tp, const FwdArgs& a, CUtensorMap* mQ, CUtensorMap* mK, CUtensorMap* mV,
              TcParams* pp) {
  if (!make_map(mQ, a.q, kDk, tp.G, tp.T, tp.B) || !make_map(mK, a.k, kDk, tp.G, tp.T, tp.B) ||
      !make_map(mV, a.v, kDv, tp.H, tp.T, tp.B))
    return false;
  TcParams& p = *pp;
  p = TcParams{};
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
  p.img = reinterpret_cast<uint8_t*>(a.ws + tp.off_img);
  p.meta = reinterpret_cast<unsigned*>(a.ws + tp.off_meta);
  p.status = a.status;
  return true;
}

cudaError_t launch_state(const TcPlan& tp, const FwdArgs& a, const CUtensorMap& mK, const CUtensorMap& mV,
                         const TcParams& p, cudaStream_t st) {
  const unsigned grid = (unsigned)((size_t)tp.B * tp.NT * tp.H);
  cudaError_t e = cudaFuncSetAttribute(tc_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemState);
  if (e != cudaSuccess) return e;
  tc_state_kernel<<<grid, 128, kSmemState, st>>>(mK, mV, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch(a, 0, st);
  return cudaSuccess;
}

cudaError_t launch_tree(const TcPlan& tp, const FwdArgs& a, const TcParams& p, cudaStream_t st) {
  // tree levels 1.. two per launch; the profiling event of slot 1 follows the last one
  cudaError_t e = cudaFuncSetAttribute(tc_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTree);
  if (e != cudaSuccess) return e;
  for (int m0 = 1; m0 < tp.MT; m0 += 2) {
    const unsigned gt = (unsigned)((size_t)tp.B * tp.H * (((tp.NT >> m0) + 1) >> 1));
    if ((e = launch_overlapped(tc_tree_kernel, dim3(gt), dim3(128), kSmemTree, st, p, m0)) != cudaSuccess)
      return e;
    if (m0 + 2 < tp.MT) note_launch();
    else note_launch(a, 1, st);
  }
  if (tp.MT <= 1 && a.events && 2 < a.n_events && a.events[2])  // no tree level above tiles
    cudaEventRecord(static_cast<cudaEvent_t>(a.events[2]), st);
  return cudaSuccess;
}

template <int kMode>
cudaError_t launch_output(const TcPlan& tp, const CUtensorMap& mQ, const CUtensorMap& mK,
                          const CUtensorMap& mV, const TcParams& p, int ninter, cudaStream_t st) {
  const unsigned grid = (unsigned)((size_t)tp.B * tp.NT * tp.H);
  const int smem_out = out_smem_bytes(ninter);
  cudaError_t e = cudaFuncSetAttribute(tc_output_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_out);
  if (e != cudaSuccess) return e;
  if (kMode == 0)  // the comparators' passes read each other's output: plain stream order
    return launch_overlapped(tc_output_kernel<kMode>, dim3(grid), dim3(256), smem_out, st, mQ, mK, mV, p);
  tc_output_kernel<kMode><<<grid, 256, smem_out, st>>>(mQ, mK, mV, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_fwd(const TcPlan& tp, const FwdArgs& a, cudaStream_t st) {
  CUtensorMap mQ, mK, mV;
  TcParams p;
  if (!tc_setup(tp, a, &mQ, &mK, &mV, &p)) return cudaErrorInvalidValue;
  cudaError_t e = launch_state(tp, a, mK, mV, p, st);
  if (e == cudaSuccess) e = launch_tree(tp, a, p, st);
  if (e != cudaSuccess) return e;
  if ((e = launch_output<0>(tp, mQ, mK, mV, p, bit_length(tp.NT - 1), st)) != cudaSuccess) return e;
  note_launch(a, 2, st);
  if (a.states_out) {
    if ((e = launch_overlapped(tc_export_kernel, dim3(__builtin_popcount((unsigned)tp.T), tp.B * tp.H), dim3(256), 0, st, p,
                               a.state_levels, a.states_out, a.logscale_out)) != cudaSuccess)
      return e;
    note_launch(a, 3, st);
  }
  return cudaSuccess;
}

size_t tc_naive_bytes(const TcPlan& tp) {
  return ((tp.bytes + 255) & ~size_t(255)) + (size_t)tp.B * tp.T * tp.H * kDv * sizeof(float);
}

cudaError_t launch_tc_naive(const TcPlan& tp, const FwdArgs& a, cudaStream_t st) {
  CUtensorMap mQ, mK, mV;
  TcParams p;
  if (!tc_setup(tp, a, &mQ, &mK, &mV, &p)) return cudaErrorInvalidValue;
  p.o32 = reinterpret_cast<float*>(a.ws + ((tp.bytes + 255) & ~size_t(255)));
  cudaError_t e = launch_state(tp, a, mK, mV, p, st);
  if (e == cudaSuccess) e = launch_tree(tp, a, p, st);
  if (e != cudaSuccess) return e;
  const int last = kLevIntra + tp.MT - 1;  // highest level with buckets in [0, T)
  for (int l = 0; l <= last; ++l) {  // one pass per level, no fusion
    p.lsel = l;
    p.lflags = (l == 0 ? 1 : 0) | (l == last ? 2 : 0);
    if ((e = launch_output<2>(tp, mQ, mK, mV, p, 1, st)) != cudaSuccess) return e;
    note_launch();
  }
  return cudaSuccess;
}

size_t tc_ssd_bytes(const TcPlan& tp) {
  const size_t n = (size_t)tp.B * tp.H * tp.NT;
  return ((tp.bytes + 255) & ~size_t(255)) + n * kImgBytes + n * kMeta * sizeof(unsigned);
}

cudaError_t launch_tc_ssd(const TcPlan& tp, const FwdArgs& a, cudaStream_t st) {
  CUtensorMap mQ, mK, mV;
  TcParams p;
  if (!tc_setup(tp, a, &mQ, &mK, &mV, &p)) return cudaErrorInvalidValue;
  const size_t base = (tp.bytes + 255) & ~size_t(255);
  p.pimg = reinterpret_cast<uint8_t*>(a.ws + base);
  p.pmeta = reinterpret_cast<unsigned*>(a.ws + base + (size_t)tp.B * tp.H * tp.NT * kImgBytes);
  cudaError_t e = launch_state(tp, a, mK, mV, p, st);
  if (e != cudaSuccess) return e;
  if (tp.NT > 1) {
    if ((e = cudaFuncSetAttribute(ssd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemScan)) !=
        cudaSuccess)
      return e;
    ssd_scan_kernel<<<tp.B * tp.H, 128, kSmemScan, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launch();
  }
  if ((e = launch_output<1>(tp, mQ, mK, mV, p, 1, st)) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

// The forward's tree only (tile states and the levels above), into a.ws per tp's layout.
cudaError_t launch_tc_nodes(const TcPlan& tp, const FwdArgs& a, cudaStream_t st) {
  CUtensorMap mQ, mK, mV;
  TcParams p;
  if (!tc_setup(tp, a, &mQ, &mK, &mV, &p)) return cudaErrorInvalidValue;
  cudaError_t e = launch_state(tp, a, mK, mV, p, st);
  if (e == cudaSuccess) e = launch_tree(tp, a, p, st);
  return e;
}

cudaError_t launch_tc_bwd_q(const TcPlan& tp, const void* q, const void* dO, const float* a, const float* lam,
                            const char* tree_ws, float* dq32, float* dlam, float* dual, const int* dual_off,
                            int nslots, unsigned* status, cudaStream_t st) {
  CUtensorMap mQ, mD;
  if (!make_map(&mQ, q, kDk, tp.G, tp.T, tp.B) || !make_map(&mD, dO, kDv, tp.H, tp.T, tp.B))
    return cudaErrorInvalidValue;
  TcBwdQParams p{};
  p.B = tp.B;
  p.T = tp.T;
  p.H = tp.H;
  p.hpg = tp.hpg;
  p.G = tp.G;
  p.L = tp.L;
  p.NT = tp.NT;
  p.nnodes = tp.nnodes;
  for (int m = 0; m < 32; ++m) {
    p.node_off[m] = m < tp.MT ? tp.node_off[m] : 0;
    p.dual_off[m] = m < tp.MT ? dual_off[m] : 0;
  }
  p.nslots = nslots;
  p.a = a;
  p.lam = lam;
  p.img = reinterpret_cast<const uint8_t*>(tree_ws + tp.off_img);
  p.meta = reinterpret_cast<const unsigned*>(tree_ws + tp.off_meta);
  p.dq32 = dq32;
  p.dlam = dlam;
  p.dual = dual;
  p.status = status;
  const int smem = bwdq_smem_bytes(bit_length(tp.NT - 1));
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  tc_bwd_q_kernel<<<(unsigned)((size_t)tp.B * tp.NT * tp.H), 256, smem, st>>>(mQ, mD, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

cudaError_t launch_tc_bwd_kv(const TcPlan& tp, const void* k, const void* v, const float* a, const char* tree_ws,
                             const float* dual, uint8_t* dimg, unsigned* dmeta, double* P, const int* dual_off,
                             int nslots, float* dk32, float* dv32, float* cu, unsigned* status, cudaStream_t st) {
  const unsigned BH = (unsigned)(tp.B * tp.H);
  tc_tile_prefix_kernel<<<BH, 256, 0, st>>>(reinterpret_cast<const unsigned*>(tree_ws + tp.off_meta), tp.nnodes,
                                            tp.NT, P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  note_launch();
  tc_dual_publish_kernel<<<(unsigned)((size_t)BH * nslots), 128, 0, st>>>(dual, dimg, dmeta);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  CUtensorMap mK, mV;
  if (!make_map(&mK, k, kDk, tp.G, tp.T, tp.B) || !make_map(&mV, v, kDv, tp.H, tp.T, tp.B))
    return cudaErrorInvalidValue;
  TcBwdKVParams p{};
  p.B = tp.B;
  p.T = tp.T;
  p.H = tp.H;
  p.hpg = tp.hpg;
  p.G = tp.G;
  p.NT = tp.NT;
  p.MT = tp.MT;
  for (int m = 0; m < 32; ++m) p.dual_off[m] = m < tp.MT ? dual_off[m] : 0;
  p.nslots = nslots;
  p.a = a;
  p.dimg = dimg;
  p.dmeta = dmeta;
  p.P = P;
  p.dk32 = dk32;
  p.dv32 = dv32;
  p.cu = cu;
  p.status = status;
  if ((e = cudaFuncSetAttribute(tc_bwd_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBwdKV)) !=
      cudaSuccess)
    return e;
  tc_bwd_kv_kernel<<<(unsigned)((size_t)tp.B * tp.NT * tp.H), 512, kSmemBwdKV, st>>>(mK, mV, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

size_t tc_gdn_bytes(const ll_shape& s) {
  return (size_t)s.batch * s.heads * (s.T / kTile) * kGdnChunkBytes;
}

cudaError_t launch_tc_gdn(const ll_shape& s, const void* k, const void* v, const float* a, const float* beta,
                          void* u, char* ws, unsigned* status, cudaStream_t st) {
  if (!tc_supported(s)) return cudaErrorInvalidValue;
  const int G = s.heads / s.heads_per_group, nch = s.T / kTile;
  CUtensorMap mK, mV;
  if (!make_map(&mK, k, kDk, G, s.T, s.batch) || !make_map(&mV, v, kDv, s.heads, s.T, s.batch))
    return cudaErrorInvalidValue;
  TcGdnParams p{s.batch, s.T, s.heads, s.heads_per_group, G, a, beta, reinterpret_cast<uint8_t*>(ws), u, status};
  cudaError_t e = cudaFuncSetAttribute(tc_gdn_local_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemGdnL);
  if (e != cudaSuccess) return e;
  tc_gdn_local_kernel<<<(unsigned)((size_t)s.batch * s.heads * nch), 256, kSmemGdnL, st>>>(mK, mV, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  if ((e = cudaFuncSetAttribute(tc_gdn_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemGdnP)) !=
      cudaSuccess)
    return e;
  tc_gdn_pass_kernel<<<(unsigned)(s.batch * s.heads), 256, kSmemGdnP, st>>>(mK, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

cudaError_t launch_tc_bwd_intra(const ll_shape& s, const void* q, const void* k, const void* v, const void* dO,
                                const float* a, const float* lam, float* dq32, float* dk32, float* dv32,
                                float* dlam, float* cu, unsigned* status, cudaStream_t st) {
  if (!tc_supported(s)) return cudaErrorInvalidValue;
  const int G = s.heads / s.heads_per_group, NT = s.T / kTile;
  CUtensorMap mQ, mK, mV, mD;
  if (!make_map(&mQ, q, kDk, G, s.T, s.batch) || !make_map(&mK, k, kDk, G, s.T, s.batch) ||
      !make_map(&mV, v, kDv, s.heads, s.T, s.batch) || !make_map(&mD, dO, kDv, s.heads, s.T, s.batch))
    return cudaErrorInvalidValue;
  const TcBwdParams p{s.batch, s.T, s.heads, s.heads_per_group, G, s.levels, NT, a, lam,
                      dq32, dk32, dv32, dlam, cu, status};
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBwd);
  if (e != cudaSuccess) return e;
  tc_bwd_intra_kernel<<<(unsigned)((size_t)s.batch * NT * s.heads), 256, kSmemBwd, st>>>(mQ, mK, mV, mD, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

cudaError_t launch_wait_selftest(unsigned* status, long long spins, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, spins);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace ll
