// Tensor-core (tcgen05 / TMEM / TMA) path of the log-linear Mamba-2 forward for
// bf16 q/k/v/o, d_k = 128, d_v = 64, T % 64 == 0.  When T % 128 == 64 the last tile holds
// 64 tokens: TMA fills the rows past T with zeros (k = v = q = 0), their a is 1 and their
// lambda 0, and the store of o leaves them out.
//
// Chunkwise algorithm of the log-linear attention write-up
// (https://www.yoousoft.com/industry/3746.html, section 高效训练算法, Algorithm 1 / Fig. 3),
// with 128-token tiles (two 64-token chunks; the result does not depend on the chunk
// length, so the tile only decides which levels are dense inside a tile: 0..7):
//
//  tc_state   one CTA per (b, h, four tiles): per tile u the chunk-local log2 decay
//             cumsum g, the tile decay gamma_u and the tile state H_u = K_uᵀ
//             diag(2^(gamma_u - g)) V_u on the tensor cores (M = d_k, N = d_v, K = tokens),
//             node (0, u) of the Fenwick tree over tiles; nodes (1, 2i) and (2, i) are summed
//             in fp32 registers on the way.  Nodes are fp16 images in the UMMA operand
//             layout with a power-of-two scale and their total log2 decay.
//  tc_tree    two tree levels per launch from level 3 up, Node_{m+1}[i] =
//             2^(Gamma(right)) Node_m[2i] + Node_m[2i+1], from the images of the level below
//             (no CTA waits for another).
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
#include <utility>

#include "tc_common.cuh"

namespace ll {

namespace {
// ---------------------------------------------------------------------------------
// tc_state: tile states and the first two tree levels above them.  One CTA per (b, h,
// group of four tiles 4i .. 4i+3); tile by tile (thread tid owns row tid of a state):
// g and the tile decay gamma, H_u = K_uᵀ diag(2^(gamma_u - g)) V_u on the tensor cores,
// published as node (0, u); a running fp32 sum L = 2^(gamma_u) L + H_u gives node (1, 2i)
// after the second tile and node (2, i) after the fourth.  The odd node (1, 2i + 1) is read
// by nothing but its parent, so it is never published; nor is the image of an odd tile
// (its decay is), except a last, partial tile or when all_tiles asks for every image.
// The next tile's K and V are requested as soon as the MMA has read the current ones, so
// that the copy overlaps the read-out and the stores.  No CTA waits for another.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 3) tc_state_kernel(const __grid_constant__ CUtensorMap mapK,
                                                       const __grid_constant__ CUtensorMap mapV,
                                                       TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;          // 32 KB: K (bf16, two 64-wide d_k boxes)
  uint8_t* sV = smem + 32768;  // 32 KB: Ṽ hi part (the TMA box) then Ṽ lo part
  // a node's fp16 image on its way out: Ṽ's lo part, free once the MMA has read it (the
  // next tile's copy fills K and Ṽ's hi part only)
  uint8_t* stage = sV + 16384;
  __shared__ __align__(8) uint64_t bar_ld, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ float s_scan[4][4];
  __shared__ float2 s_red2[4];
  __shared__ float s_gamma4[4];

  const int tid = threadIdx.x, warp = tid >> 5, rot = tid & 7;
  const int ng4 = (p.NT + 3) >> 2;  // groups of four tiles per (b, h)
  const int lin = blockIdx.x;
  const int h = lin % p.H;
  const int i4 = (lin / p.H) % ng4;
  const int b = lin / (p.H * ng4);
  const int g = h / p.hpg;
  const size_t nbase = (size_t)(b * p.H + h) * p.nnodes;
  const int nt4 = min(4, p.NT - 4 * i4);  // tiles of this group (fewer at the end)
  // a of token tid of each tile (rows past T in a last, partial tile: a = 1, and TMA
  // fills their k and v with zeros)
  float a4[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const long long t = (long long)(4 * i4 + k) * kTile + tid;
    a4[k] = (k < nt4 && t < p.T) ? p.a[((size_t)b * p.T + t) * p.H + h] : 1.f;
  }
  ptx::griddep_launch_dependents();

  auto load_tile = [&](int u) {
    ptx::mbar_arrive_expect_tx(&bar_ld, 32768 + 16384);
    ptx::tma_load_4d(sK, &mapK, &bar_ld, 0, g, u * kTile, b);
    ptx::tma_load_4d(sK + 16384, &mapK, &bar_ld, 64, g, u * kTile, b);
    ptx::tma_load_4d(sV, &mapV, &bar_ld, 0, h, u * kTile, b);
  };
  if (tid == 0) {
    ptx::mbar_init(&bar_ld, 1);
    ptx::mbar_init(&bar_mma, 1);
    ptx::fence_mbar_init();
    load_tile(4 * i4);
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 128);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = tmem_base;
  // decay of token u * 128 + tid for the group's four tiles u at once (while the first
  // tile loads): chunk-local log2 cumsums, and each tile's total gamma_u
  float gi4[4];
  {
    const int lane = tid & 31;
#pragma unroll
    for (int j = 0; j < 4; ++j) gi4[j] = log2f(a4[j]);
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float y = __shfl_up_sync(0xffffffffu, gi4[j], off);
        if (lane >= off) gi4[j] += y;
      }
    if (lane == 31)
#pragma unroll
      for (int j = 0; j < 4; ++j) s_scan[warp][j] = gi4[j];
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float add = 0.f;
      for (int w = 0; w < warp; ++w) add += s_scan[w][j];
      gi4[j] += add;
    }
    if (tid == kTile - 1)
#pragma unroll
      for (int j = 0; j < 4; ++j) s_gamma4[j] = gi4[j];  // read after the barrier below
  }
  float L[kDv];  // running sum of the group's tile states, decayed to the latest tile's end
  float GL = 0.f;
  int k = 0, fail = 0;  // fail: 1 = tile k's copy timed out, 2 = its MMA did
  for (; k < nt4; ++k) {
    const int u = 4 * i4 + k;
    const float gi = k == 0 ? gi4[0] : k == 1 ? gi4[1] : k == 2 ? gi4[2] : gi4[3];
    bool ok = wait_bar(&bar_ld, k & 1);
    if (!ok) atomicExch(p.status, kStatusTimeout);
    if (!__syncthreads_and(ok)) {
      fail = 1;
      break;
    }
    const float gamma = s_gamma4[k];
    {
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
          float2 rr = __bfloat1622float2(hx[e]);
          hy[e] = __floats2bfloat162_rn(f.x - rr.x, f.y - rr.y);
        }
        *reinterpret_cast<uint4*>(sV + off) = x;
        *reinterpret_cast<uint4*>(sV + 16384 + off) = y;
      }
      ptx::fence_proxy_async_smem();
    }
    __syncthreads();  // also: every read-out of the previous tile's accumulator is done
    if (tid == 0) {
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
    ok = wait_bar(&bar_mma, k & 1);
    if (!ok) atomicExch(p.status, kStatusTimeout);
    if (!__syncthreads_and(ok)) {
      fail = 2;
      break;
    }
    if (tid == 0 && k + 1 < nt4) load_tile(u + 1);  // the MMA has read sK and sV
    ptx::tc_fence_after();
    // H_u row tid = Hhi + Hlo, 16 columns at a time: folded into L and its maximum taken;
    // the tile's node (level 0; node_off[0] == 0) is staged from a second read of the
    // accumulator.  Readers of the tree take even nodes only, and a last, partial tile's
    // node (the state export's nearest bucket); another odd tile's state goes into node
    // (1, 2i) here, so only its decay is stored.
    const uint32_t trow = tbase + ((uint32_t)(warp * 32) << 16);
    const float d = exp2f(gamma);
    float m = 0.f;
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2) {  // 32 columns per wait
      float hi[32], lo[32];
      ptx::tmem_ld16(trow + q2 * 32, hi);
      ptx::tmem_ld16(trow + q2 * 32 + 16, hi + 16);
      ptx::tmem_ld16(trow + 64 + q2 * 32, lo);
      ptx::tmem_ld16(trow + 64 + q2 * 32 + 16, lo + 16);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float c = hi[j] + lo[j];
        m = fmaxf(m, fabsf(c));
        L[q2 * 32 + j] = k == 0 ? c : d * L[q2 * 32 + j] + c;
      }
    }
    const size_t node0 = nbase + u;
    if ((k & 1) == 0 || p.all_tiles || (u == p.NT - 1 && p.T % kTile != 0)) {
      const int e = f16_exp(block_max2(make_float2(m, 0.f), s_red2).x);
      const float sc = pow2i(-e);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float hi[16], lo[16];
        ptx::tmem_ld16(trow + q4 * 16, hi);
        ptx::tmem_ld16(trow + 64 + q4 * 16, lo);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {  // 16-byte chunk 2 q4 + c2 of the row
          const float* x = hi + 8 * c2;
          const float* y = lo + 8 * c2;
          *reinterpret_cast<uint4*>(stage + tid * 128 + (((2 * q4 + c2) ^ rot) << 4)) =
              make_uint4(pack_h2((x[0] + y[0]) * sc, (x[1] + y[1]) * sc), pack_h2((x[2] + y[2]) * sc, (x[3] + y[3]) * sc),
                         pack_h2((x[4] + y[4]) * sc, (x[5] + y[5]) * sc), pack_h2((x[6] + y[6]) * sc, (x[7] + y[7]) * sc));
        }
      }
      __syncthreads();
      uint4* dst = reinterpret_cast<uint4*>(p.img + node0 * kImgBytes);
#pragma unroll
      for (int rr = 0; rr < kImgBytes / 16 / 128; ++rr)
        dst[rr * 128 + tid] = reinterpret_cast<const uint4*>(stage)[rr * 128 + tid];
      if (tid == 0) p.meta[node0 * kMeta + 1] = (unsigned)e;
    }
    if (tid == 0) p.meta[node0 * kMeta + 2] = __float_as_uint(gamma);
    ptx::tc_fence_before();
    GL += gamma;
    if (k == 1 || k == 3) {
      __syncthreads();  // every row of the staged tile node is stored
      publish_node(L, stage, nbase + p.node_off[k == 1 ? 1 : 2] + (k == 1 ? 2 * i4 : i4), GL, s_red2, p.img,
                   p.meta);
    }
    __syncthreads();  // the staging area is free again
  }
  if (fail && tid == 0) {  // tile k gave up: let what it started end (bounded waits)
    wait_bar(&bar_ld, k & 1);
    if (fail == 2) wait_bar(&bar_mma, k & 1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tbase, 128);
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
// 256 threads in two roles after a common prologue (warp 1 issues the tile loads; both
// roles copy their lambda rows and compute the decay cumsum; warp 0 allocates TMEM):
//  role a (warps 0-3): issues S = Q Kᵀ; once S has landed, P row t = thread, written as
//          fp16 into tensor memory over the columns of S it has consumed; then the V tile
//          scale and V -> fp16 in place; O = P V with P as the tensor-memory A operand.
//  role b (warps 4-7): waits for the tree's launches and fetches the node scalars and
//          the first node image, all in the prologue; Q row t -> fp16 with a power-of-two
//          scale of its own (undone in the row weight) in place once S has read Q; the
//          inter-tile levels, nearest first and two per MMA (N = 128 over two node
//          images), with up to three node images in flight; then the write of o, staged
//          in RV and stored with one TMA store.
// Both roles see every TMEM lane through warp % 4.
// Shared memory (2 CTAs per SM): RQ = Q (bf16, then fp16 in place); RK = K (bf16) until
// S completes, then node image buffers 1 and 2; RV = V (bf16, then fp16 in place), then
// the staging of o; RE = node image buffer 0.  The image of level index i (i-th set bit of u from the
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

template <int kMode>
__global__ void __launch_bounds__(256, 2) tc_output_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                           const __grid_constant__ CUtensorMap mapK,
                                                           const __grid_constant__ CUtensorMap mapV,
                                                           const __grid_constant__ CUtensorMap mapO,
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
  __shared__ __align__(8) uint64_t bar_ld, bar_s, bar_o, bar_e[3], bar_y, bar_yf;
  __shared__ uint32_t tmem_base;
  __shared__ float s_red[8];
  __shared__ int s_oi;  // role a -> all: the O MMA was issued
  __shared__ int s_e12; // node images 1 and 2 issued by thread 0 once S has read K

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127;             // query row (tile-local token)
  const int quad = warp & 3;           // TMEM lane quadrant of this warp
  const bool role_b = warp >= 4;       // S, inter-tile levels and the final write
  const bool driver = tid == 128;      // role b's MMA, image-load and o-store issuer
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
  const bool in_t = t0 + r < p.T;  // false for the rows past T of a last, partial tile
  const float* lrow = p.lam + (row * p.H + h) * p.L;
  // inter-tile levels of this tile, and whether the intra-tile part runs
  ptx::griddep_launch_dependents();  // the next launch may start once all CTAs are resident
  // Level indices 0 .. nloc-1 are the set bits of u (nearest first); in the level-fused
  // mode the live levels of a start position T0 > 0 follow them (a forward that continues
  // from the bucket memories at T0: those buckets lie before every bucket of the segment).
  const int nloc = kMode == 0 ? __popc((unsigned)u)
                 : kMode == 1 ? (u > 0 ? 1 : 0)
                              : (p.lsel >= kLevIntra && ((u >> (p.lsel - kLevIntra)) & 1) ? 1 : 0);
  const int nlev = nloc + (kMode == 0 ? p.npre : 0);
  const bool intra_on = kMode != 2 || p.lsel < kLevIntra;
  auto ebuf = [&](int k) { return k == 0 ? RE : RK + (k - 1) * 16384; };  // image buffer k
  auto lev_of = [&](int i) {  // tile level m of level index i < nloc
    return kMode == 2 ? p.lsel - kLevIntra : nth_set_bit((unsigned)u, i);
  };
  auto lam_col = [&](int i) {  // lambda column (token level) of level index i
    return (kMode == 0 && i >= nloc) ? p.prelev[i - nloc] : kLevIntra + lev_of(i);
  };
  auto img_of = [&](int i) -> const uint8_t* {  // image read by level index i
    if (kMode == 1) return p.pimg + ((size_t)bh * p.NT + u) * kImgBytes;
    if (kMode == 0 && i >= nloc) return p.preimg + ((size_t)bh * p.npre + (i - nloc)) * kImgBytes;
    const int m = lev_of(i);
    return p.img + (nbase + p.node_off[m] + ((u >> m) - 1)) * kImgBytes;
  };
  auto meta_of = [&](int i) -> const unsigned* {
    if (kMode == 1) return p.pmeta + ((size_t)bh * p.NT + u) * kMeta;
    if (kMode == 0 && i >= nloc) return p.premeta + ((size_t)bh * p.npre + (i - nloc)) * kMeta;
    const int m = lev_of(i);
    return p.meta + (nbase + p.node_off[m] + ((u >> m) - 1)) * kMeta;
  };

  // Warp 0's prologue path held the tile's loads back: tcgen05.alloc takes about 1 us, and
  // the load of a behind it another 1 us.  So a is loaded first, warp 1 initialises the
  // barriers and issues the tile loads, and warp 0 allocates after the lambda copies.
  const float a_row = in_t ? p.a[row * p.H + h] : 1.f;
  if (tid == 32) {
    s_oi = 0;
    s_e12 = 0;
    ptx::mbar_init(&bar_ld, 1);
    ptx::mbar_init(&bar_s, 1);
    ptx::mbar_init(&bar_o, 1);
    for (int i = 0; i < 3; ++i) ptx::mbar_init(&bar_e[i], 1);
    ptx::mbar_init(&bar_y, 1);
    ptx::mbar_init(&bar_yf, 128);
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
  // lambda of this row (levels 0..7 for role a, the tile's inter levels for role b) and
  // the node scalars of the tile's levels, copied asynchronously
  if (!role_b) {
#pragma unroll
    for (int l = 0; l < kLevIntra; ++l) {
      if (in_t && (kMode == 0 || (kMode == 2 && l == p.lsel))) ptx::cp_async4(sLam8 + r * 9 + l, lrow + l);
      else sLam8[r * 9 + l] = (kMode == 1 && in_t) ? 1.f : 0.f;  // SSD: lambda = 1; single level: others off
    }
  } else {
    if (kMode == 1) {
      if (nlev > 0) sLamI[r] = 1.f;
    } else {
      for (int i = 0; i < nlev; ++i) {
        if (in_t) ptx::cp_async4(sLamI + i * 128 + r, lrow + lam_col(i));
        else sLamI[i * 128 + r] = 0.f;
      }
    }
    // The tree that the previous launches built is read from here on.  The wait (at once
    // unless this grid was launched before they finished) and the node scalars' fetch
    // overlap the tile's loads.
    ptx::griddep_wait();
    if (r < nlev) {
      const unsigned* mt = meta_of(r);
      ptx::cp_async4(sNode + 2 * r, mt + 1);
      ptx::cp_async4(sNode + 2 * r + 1, mt + 2);
    }
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 256);
    ptx::tmem_relinquish();
  }
  // chunk-local log2 decay cumsum over the 128 rows (both roles compute it)
  float gt = log2f(a_row);
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
  // role b's driver: the first node image into RE (free from the start), also while the
  // tile loads; the barriers were initialised before the first __syncthreads
  if (driver && nlev > 0) {
    ptx::mbar_arrive_expect_tx(&bar_e[0], kImgBytes);
    ptx::bulk_load(ebuf(0), img_of(0), kImgBytes, &bar_e[0]);
  }
  bool ok = wait_bar(&bar_ld, 0);
  if (!ok) atomicExch(p.status, kStatusTimeout);
  ok = __syncthreads_and(ok);

  // S = Q Kᵀ (M = 128 queries, N = 128 keys, K = 128 d_k), bf16, both K-major; issued by
  // role a, which waits for it first, so that role b goes straight to its Q work.
  if (ok && tid == 0 && intra_on) {
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
    if (ok && tid == 0 && nlev > 1) {  // K has been read by S: node images 1 and 2 into RK
      ptx::mbar_arrive_expect_tx(&bar_e[1], kImgBytes);
      ptx::bulk_load(RK, img_of(1), kImgBytes, &bar_e[1]);
      if (nlev > 2) {
        ptx::mbar_arrive_expect_tx(&bar_e[2], kImgBytes);
        ptx::bulk_load(RK + 16384, img_of(2), kImgBytes, &bar_e[2]);
      }
      s_e12 = nlev > 2 ? 2 : 1;
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
            // 8-key blocks before t's: one level each, bit length of (tb ^ kb) plus 3, and
            // the factored decay.  t's own block: level of key e is the bit length of
            // te ^ e (0..3), zero above t.  Blocks after t's are zero (a select: A may be
            // inf there).
            const int tb = tl >> 3, te = tl & 7;
            float ak[4];
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
              const float lv = kb == tb ? 1.f : lamr[35 - __clz(tb ^ kb)];
              const float x = coef * lv * exp2f(gt - gq[kb * 8 + 7]);
              ak[kb] = kb > tb ? 0.f : x;
            }
            float fo[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) fo[e] = e <= te ? lamr[32 - __clz(te ^ e)] : 0.f;
            const float4* b4 = reinterpret_cast<const float4*>(sB8 + cg * 32);
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 bb = b4[j4];
              const float bj[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int j = 4 * j4 + e, kb = j >> 3;
                const float f = kb == tb ? fo[j & 7] : 1.f;
                v[j] = sv[j] * (ak[kb] * bj[e]) * f;
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
    // The tree wait, the node scalars and the first image were issued in the prologue.
    // Q row r -> fp16 with scale 2^-eq of its own: read and converted while S runs,
    // stored back once S has completed.  Then images 1 and 2 go into RK.
    uint8_t* qrow0 = RQ + r * 128;
    uint8_t* qrow1 = RQ + 16384 + r * 128;
    int eq = 0;
    // image loads issued by the driver: image 0 in the prologue, images from 3 on in the
    // level loop (thread 0 issues images 1 and 2, or the driver does without the S part)
    int issued = nlev > 0 ? 1 : 0;
    int consumed = 0;               // image loads waited for by the driver
    int y_issued = 0, y_seen = 0;   // Y MMAs issued / seen complete by the driver
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
    if (ok && driver && !intra_on) {
      for (int i = 1; i < 3 && i < nlev; ++i) {  // K was never loaded: RK is free
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
      if (i >= 2 && !wait_bar(&bar_yf, ((i >> 1) - 1) & 1)) return false;  // Y read by all
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
      ptx::umma_commit(&bar_y);
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
      bool okw = wait_bar(&bar_y, (i >> 1) & 1);
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
      ptx::mbar_arrive(&bar_yf);
    }
    __syncthreads();  // join: P, its row scales and the O MMA have been issued
    if (driver) {
      // after a failed wait: let this CTA's own copies and MMAs land (bounded) before exit
      // (image loads are issued in level order, so the unconsumed ones are the last)
      if (intra_on) issued += s_e12;
      for (int j = consumed; j < issued; ++j) wait_bar(&bar_e[j % 3], (j / 3) & 1);
      for (int j = y_seen; j < y_issued; ++j) wait_bar(&bar_y, j & 1);
      if (s_issued) wait_bar(&bar_s, 0);
    }
    const bool o_issued = s_oi != 0;
    if (intra_on) {
      ok = ok && o_issued && wait_bar(&bar_o, 0);
      if (!ok && o_issued) atomicExch(p.status, kStatusTimeout);
    }
    ok = __all_sync(0xffffffffu, ok);
    // o row r is staged in RV (V's buffer: free once O has completed, and never loaded
    // when the intra-tile part is off) in the 128-byte-swizzled layout of o's tensor map,
    // then the tile goes out in one TMA store.
    const bool write_o = kMode != 2 || (p.lflags & 2);
    uint8_t* orow_s = RV + r * 128;
    if (ok) {
      ptx::tc_fence_after();
      const float so = pow2s(sEp[r]);
      float* o32row = (kMode == 2 && in_t) ? p.o32 + (row * p.H + h) * kDv : nullptr;
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
        if (kMode == 2 && !in_t) continue;  // rows past T: nothing to keep (the store clips them)
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
#pragma unroll
        for (int c = 0; c < 4; ++c)  // 16-byte chunk half * 4 + c of the row
          *reinterpret_cast<uint4*>(orow_s + (((half * 4 + c) ^ rot) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
    }
    if (write_o) {
      ptx::fence_proxy_async_smem();
      const bool ok_o = ptx::named_bar_and(2, 128, ok);  // every row staged
      if (driver && ok_o) {
        ptx::tma_store_4d(&mapO, RV, 0, h, (int)t0, b);
        ptx::bulk_commit_group();
        ptx::bulk_wait_read_all();  // RV is read before the CTA ends
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
// tc_export: bucket states at position T (T % 64 == 0, so live levels are >= 7).
// ---------------------------------------------------------------------------------
// One CTA per live level of T (level l >= 1 with bit l-1 of T set) and (b, h); CTA 0 of
// each (b, h) also writes the zero log-scales of all SL slots.  Slots of levels that are
// not live at T are left as they are.  With nf = T / 128 full tiles, level 8 + m is the
// node (m, (nf >> m) - 1) for each set bit m of nf; when T % 128 == 64, level 7 is the
// last, partial tile's node (0, nf), the nearest bucket of all.
__global__ void __launch_bounds__(256) tc_export_kernel(TcParams p, int SL, float* st, float* lsc) {
  ptx::griddep_wait();  // reads the tree
  const int bh = blockIdx.y;
  if (lsc && blockIdx.x == 0)
    for (int l = threadIdx.x; l < SL; l += 256) lsc[(size_t)bh * SL + l] = 0.f;
  const int lvl = nth_set_bit((unsigned)p.T, blockIdx.x) + 1;
  float* dst = st + ((size_t)bh * SL + lvl) * (kDk * kDv);
  const int nf = p.T / kTile;
  const bool part = (p.T % kTile) != 0;
  const size_t nbase = (size_t)bh * p.nnodes;
  size_t node;
  float D = 0.f;
  if (lvl < kLevIntra) {
    node = nbase + nf;  // node (0, nf): the partial tile
  } else {
    const int m = lvl - kLevIntra;
    if (part) D += __uint_as_float(p.meta[(nbase + nf) * kMeta + 2]);
    for (int mm = 0; mm < m; ++mm)
      if ((nf >> mm) & 1) D += __uint_as_float(p.meta[(nbase + p.node_off[mm] + ((nf >> mm) - 1)) * kMeta + 2]);
    node = nbase + p.node_off[m] + ((nf >> m) - 1);
  }
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

// ---------------------------------------------------------------------------------
// tc_prefix_publish: the bucket memories at a start position T0 (continuation) as node
// images for tc_output: exp(log-scale) * memory, published like a tree node with log2
// decay 0.  One CTA per (b, h, live level of T0); thread tid owns row tid.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) tc_prefix_publish_kernel(TcParams p, const float* pst, const float* plsc,
                                                                int Lp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ float2 s_red2[4];
  const int tid = threadIdx.x;
  const int bh = blockIdx.x / p.npre, j = blockIdx.x % p.npre;
  const int lvl = p.prelev[j];
  const float sc = expf(plsc[(size_t)bh * Lp + lvl]);
  const float4* src = reinterpret_cast<const float4*>(pst + ((size_t)bh * Lp + lvl) * (kDk * kDv) + tid * kDv);
  float cur[kDv];
#pragma unroll
  for (int c = 0; c < kDv / 4; ++c) {
    const float4 x = src[c];
    cur[4 * c] = sc * x.x;
    cur[4 * c + 1] = sc * x.y;
    cur[4 * c + 2] = sc * x.z;
    cur[4 * c + 3] = sc * x.w;
  }
  publish_node(cur, stage, (size_t)bh * p.npre + j, 0.f, s_red2, p.preimg, p.premeta);
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
// host side
// ---------------------------------------------------------------------------------

constexpr int kSmemState = 32768 + 32768 + 1024;
constexpr int kSmemTree = 4 * kImgBytes + 1024;
constexpr int kSmemPublish = kImgBytes + 1024;

}  // namespace

bool tc_supported(const ll_shape& s) {
  return s.dtype == LL_BF16 && s.d_k == kDk && s.d_v == kDv && s.T % kTile == 0 &&
         s.levels <= 32 && bit_length(s.T / kTile - 1) <= kMaxInter && encode_fn() != nullptr;
}

bool tc_fwd_supported(const ll_shape& s) {
  const int nt = (s.T + kTile - 1) / kTile;
  return s.dtype == LL_BF16 && s.d_k == kDk && s.d_v == kDv && s.T % (kTile / 2) == 0 && s.T > 0 &&
         s.levels <= 32 && bit_length(nt - 1) <= kMaxInter && encode_fn() != nullptr;
}

const char* tc_kernel_names(bool with_export) {
  return with_export ? "tc_state,tc_tree,tc_output,tc_export" : "tc_state,tc_tree,tc_output";
}

bool make_tc_plan(const ll_shape& s, TcPlan* p) { return tc_supported(s) && make_tc_fwd_plan(s, p); }

bool make_tc_fwd_plan(const ll_shape& s, TcPlan* p) {
  if (!tc_fwd_supported(s)) return false;
  p->B = s.batch;
  p->T = s.T;
  p->H = s.heads;
  p->hpg = s.heads_per_group;
  p->G = s.heads / s.heads_per_group;
  p->L = s.levels;
  p->NT = (s.T + kTile - 1) / kTile;  // a last tile of 64 tokens when T % 128 == 64
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

// Tensor maps of q, k, v (loads) and, when mO is given, of o (the output tile's store,
// with v's geometry; a.o must then be set).
bool tc_setup(const TcPlan& tp, const FwdArgs& a, CUtensorMap* mQ, CUtensorMap* mK, CUtensorMap* mV,
              CUtensorMap* mO, TcParams* pp) {
  if (!make_map(mQ, a.q, kDk, tp.G, tp.T, tp.B) || !make_map(mK, a.k, kDk, tp.G, tp.T, tp.B) ||
      !make_map(mV, a.v, kDv, tp.H, tp.T, tp.B))
    return false;
  if (mO && (!a.o || !make_map(mO, a.o, kDv, tp.H, tp.T, tp.B))) return false;
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
  p.img = reinterpret_cast<uint8_t*>(a.ws + tp.off_img);
  p.meta = reinterpret_cast<unsigned*>(a.ws + tp.off_meta);
  p.status = a.status;
  return true;
}

cudaError_t launch_state(const TcPlan& tp, const FwdArgs& a, const CUtensorMap& mK, const CUtensorMap& mV,
                         const TcParams& p, cudaStream_t st) {
  const unsigned grid = (unsigned)((size_t)tp.B * ((tp.NT + 3) / 4) * tp.H);
  cudaError_t e = cudaFuncSetAttribute(tc_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemState);
  if (e != cudaSuccess) return e;
  tc_state_kernel<<<grid, 128, kSmemState, st>>>(mK, mV, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch(a, 0, st);
  return cudaSuccess;
}

cudaError_t launch_tree(const TcPlan& tp, const FwdArgs& a, const TcParams& p, cudaStream_t st) {
  // tree levels 3.. two per launch (tc_state built levels 0..2); the profiling event of
  // slot 1 follows the last one
  cudaError_t e = cudaFuncSetAttribute(tc_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTree);
  if (e != cudaSuccess) return e;
  for (int m0 = 3; m0 < tp.MT; m0 += 2) {
    const unsigned gt = (unsigned)((size_t)tp.B * tp.H * (((tp.NT >> m0) + 1) >> 1));
    if ((e = launch_overlapped(tc_tree_kernel, dim3(gt), dim3(128), kSmemTree, st, p, m0)) != cudaSuccess)
      return e;
    if (m0 + 2 < tp.MT) note_launch();
    else note_launch(a, 1, st);
  }
  if (tp.MT <= 3 && a.events && 2 < a.n_events && a.events[2])  // no tree level above level 2
    cudaEventRecord(static_cast<cudaEvent_t>(a.events[2]), st);
  return cudaSuccess;
}

template <int kMode>
cudaError_t launch_output(const TcPlan& tp, const CUtensorMap& mQ, const CUtensorMap& mK,
                          const CUtensorMap& mV, const CUtensorMap& mO, const TcParams& p, int ninter,
                          cudaStream_t st) {
  const unsigned grid = (unsigned)((size_t)tp.B * tp.NT * tp.H);
  const int smem_out = out_smem_bytes(ninter);
  cudaError_t e = cudaFuncSetAttribute(tc_output_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_out);
  if (e != cudaSuccess) return e;
  if (kMode == 0)  // the comparators' passes read each other's output: plain stream order
    return launch_overlapped(tc_output_kernel<kMode>, dim3(grid), dim3(256), smem_out, st, mQ, mK, mV, mO, p);
  tc_output_kernel<kMode><<<grid, 256, smem_out, st>>>(mQ, mK, mV, mO, p);
  return cudaGetLastError();
}

}  // namespace

size_t tc_prefix_bytes(const TcPlan& tp, int npre) {
  const size_t n = (size_t)tp.B * tp.H * (npre > 0 ? npre : 0);
  return a256(n * kImgBytes) + a256(n * kMeta * sizeof(unsigned));
}

cudaError_t launch_tc_fwd(const TcPlan& tp, const FwdArgs& a, cudaStream_t st) {
  CUtensorMap mQ, mK, mV, mO;
  TcParams p;
  if (!tc_setup(tp, a, &mQ, &mK, &mV, &mO, &p)) return cudaErrorInvalidValue;
  cudaError_t e;
  if (a.T0 > 0) {
    // continuation: the live levels of T0, nearest first, as images for tc_output.  Plain
    // stream order: the dependent launches after it wait for it transitively.
    p.npre = 0;
    for (int l = 1; l <= 62 && p.npre < 32; ++l)
      if ((a.T0 >> (l - 1)) & 1) p.prelev[p.npre++] = l;
    const size_t n = (size_t)tp.B * tp.H * p.npre;
    p.preimg = reinterpret_cast<uint8_t*>(a.pre_ws);
    p.premeta = reinterpret_cast<unsigned*>(a.pre_ws + a256(n * kImgBytes));
    if ((e = cudaFuncSetAttribute(tc_prefix_publish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kSmemPublish)) != cudaSuccess)
      return e;
    tc_prefix_publish_kernel<<<(unsigned)n, 128, kSmemPublish, st>>>(p, a.pre_st, a.pre_lsc, a.pre_levels);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launch();
  }
  e = launch_state(tp, a, mK, mV, p, st);
  if (e == cudaSuccess) e = launch_tree(tp, a, p, st);
  if (e != cudaSuccess) return e;
  if ((e = launch_output<0>(tp, mQ, mK, mV, mO, p, bit_length(tp.NT - 1) + p.npre, st)) != cudaSuccess) return e;
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
  CUtensorMap mQ, mK, mV, mO;
  TcParams p;
  if (!tc_setup(tp, a, &mQ, &mK, &mV, &mO, &p)) return cudaErrorInvalidValue;
  p.o32 = reinterpret_cast<float*>(a.ws + ((tp.bytes + 255) & ~size_t(255)));
  cudaError_t e = launch_state(tp, a, mK, mV, p, st);
  if (e == cudaSuccess) e = launch_tree(tp, a, p, st);
  if (e != cudaSuccess) return e;
  const int last = kLevIntra + tp.MT - 1;  // highest level with buckets in [0, T)
  for (int l = 0; l <= last; ++l) {  // one pass per level, no fusion
    p.lsel = l;
    p.lflags = (l == 0 ? 1 : 0) | (l == last ? 2 : 0);
    if ((e = launch_output<2>(tp, mQ, mK, mV, mO, p, 1, st)) != cudaSuccess) return e;
    note_launch();
  }
  return cudaSuccess;
}

size_t tc_ssd_bytes(const TcPlan& tp) {
  const size_t n = (size_t)tp.B * tp.H * tp.NT;
  return ((tp.bytes + 255) & ~size_t(255)) + n * kImgBytes + n * kMeta * sizeof(unsigned);
}

cudaError_t launch_tc_ssd(const TcPlan& tp, const FwdArgs& a, cudaStream_t st) {
  CUtensorMap mQ, mK, mV, mO;
  TcParams p;
  if (!tc_setup(tp, a, &mQ, &mK, &mV, &mO, &p)) return cudaErrorInvalidValue;
  const size_t base = (tp.bytes + 255) & ~size_t(255);
  p.pimg = reinterpret_cast<uint8_t*>(a.ws + base);
  p.pmeta = reinterpret_cast<unsigned*>(a.ws + base + (size_t)tp.B * tp.H * tp.NT * kImgBytes);
  p.all_tiles = 1;
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
  if ((e = launch_output<1>(tp, mQ, mK, mV, mO, p, 1, st)) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

// The forward's tree only (tile states and the levels above), into a.ws per tp's layout.
cudaError_t launch_tc_nodes(const TcPlan& tp, const FwdArgs& a, cudaStream_t st) {
  CUtensorMap mQ, mK, mV;
  TcParams p;
  if (!tc_setup(tp, a, &mQ, &mK, &mV, nullptr, &p)) return cudaErrorInvalidValue;
  cudaError_t e = launch_state(tp, a, mK, mV, p, st);
  if (e == cudaSuccess) e = launch_tree(tp, a, p, st);
  return e;
}

// The tree and the export of the memories at position T into a.states_out.
cudaError_t launch_tc_export_only(const TcPlan& tp, const FwdArgs& a, cudaStream_t st) {
  CUtensorMap mQ, mK, mV;
  TcParams p;
  if (!a.states_out || !tc_setup(tp, a, &mQ, &mK, &mV, nullptr, &p)) return cudaErrorInvalidValue;
  cudaError_t e = launch_state(tp, a, mK, mV, p, st);
  if (e == cudaSuccess) e = launch_tree(tp, a, p, st);
  if (e != cudaSuccess) return e;
  if ((e = launch_overlapped(tc_export_kernel, dim3(__builtin_popcount((unsigned)tp.T), tp.B * tp.H), dim3(256), 0,
                             st, p, a.state_levels, a.states_out, a.logscale_out)) != cudaSuccess)
    return e;
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
