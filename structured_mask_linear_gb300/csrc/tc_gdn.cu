// Tensor-core kernels of the log-linear Gated DeltaNet values (for bf16, d_k = 128,
// d_v = 64, T % 128 == 0), in 128-token chunks: tc_gdn_local and tc_gdn_pass.  The
// delta rule's WY form they follow is set out in gdn.cu.
#include "tc_common.cuh"

namespace ll {

namespace {

// ---------------------------------------------------------------------------------
// Gated DeltaNet values on the tensor cores, 128-token chunks (the delta rule's WY form,
// as in gdn.cu: u = U_loc - W S per chunk, T = (I + diag(beta) A)^-1, A = (K Kᵀ) ⊙
// 2^(g_t - g_s) strictly lower, U_loc = T diag(beta) V, W = T diag(beta 2^g) K).
//
// tc_gdn_local, 256 threads, one persistent CTA per SM walking the (b, h, chunk) items
// (the next chunk's K and V copied in while this one finishes); per chunk:
//   K Kᵀ on tcgen05 from the bf16 keys (exact products, fp32 sums); A in fp32 in shared
//   memory (meanwhile the other four warps take the K and V tile maxima and split
//   diag(beta) V); T's 16 x 16 diagonal blocks by substitution in registers, then the
//   blocks below them by doubling, T21 = -T22 A21 T11, for blocks of 16 and 32 on the
//   CUDA cores and of 64 on tcgen05; then [W | U_loc] = T [diag(beta 2^g) K | diag(beta) V] on tcgen05 with every operand
//   split into an fp16 high part and the fp16 rounding remainder (hi hi + lo hi + hi lo,
//   about 22 significant bits), each with a power-of-two tile scale.  Per chunk the
//   workspace gets W split the same way (hi and lo fp16 in the MMA operand layout, with
//   its scale exponent), U_loc (fp32) and g, for tc_gdn_pass.
// ---------------------------------------------------------------------------------
// Workspace per (b, h, chunk): W hi, W lo (fp16, 16 KB boxes of 64 d_k columns with the
// 128-byte swizzle), U_loc (128 x d_v fp32; in each half row of 32 values, 16-byte chunk j
// stored at j ^ (row & 7)), g (128 fp32), W's scale exponent, then the fp16 scale exponent
// of the chunk's keys (from their maximum |k|; tc_gdn_pass converts K with it).
constexpr int kGdnOffU = 65536, kGdnOffG = 65536 + 32768, kGdnOffE = kGdnOffG + 512;
constexpr size_t kGdnChunkBytes = 99328;

struct TcGdnParams {
  int B, T, H, hpg, G;
  const float* a;
  const float* beta;
  uint8_t* xw;  // (B*H, T/128, kGdnChunkBytes)
  int pf_stride;  // the SM count (tc_gdn_local: its grid, one persistent CTA per SM; 0: unknown)
  int b0;         // tc_gdn_pass: first batch element of this launch (CTA x: (b0 + x / H, x % H))
  void* u;        // (B, T, H, d_v) bf16: the transformed values (tc_gdn_pass)
  unsigned* status;
};

constexpr int kGP = 132;  // padded fp32 row of the 128 x 128 matrices
constexpr int kSmemGdnL = 32768 + 16384 + 2 * 128 * kGP * 4 + 4 * 128 * 4 + 32768 + 1024;

// L2 prefetch of one tile through a 4-D tensor map (no shared memory, no completion)
__device__ __forceinline__ void tma_prefetch_4d(const void* tmap, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(tmap), "r"(c0),
               "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// L2 prefetch of a contiguous range (16-byte aligned address, size a multiple of 16)
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// component i (0..3, known at compile time after unrolling) of a float4
__device__ __forceinline__ float f4_at(const float4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Eight fp32 values x * sc -> their fp16 high parts and the fp16 rounding remainders,
// packed two per 32-bit word (element 2j in the low half), with paired conversions.
__device__ __forceinline__ void split8(const float (&x)[8], float sc, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float a = x[2 * j] * sc, b = x[2 * j + 1] * sc;
    const __half2 hh = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(hh);
    const __half2 ll = __floats2half2_rn(a - hf.x, b - hf.y);
    h[j] = *reinterpret_cast<const uint32_t*>(&hh);
    l[j] = *reinterpret_cast<const uint32_t*>(&ll);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}
// ... of eight bf16 values (a 16-byte chunk)
__device__ __forceinline__ void split8_bf16(const uint4& v, float sc, uint4& hi, uint4& lo) {
  const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
  float x[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = __uint_as_float(w4[e] << 16);
    x[2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
  }
  split8(x, sc, hi, lo);
}

// One level of T's doubling for diagonal blocks of size n (every pair at once; see the
// comment at the call): X = A21 T11 into A's upper triangle, then T21 = -T22 X.  Each of
// the 256 threads takes one output tile of RT rows x 4 columns (RT = n / 16), the column
// tiles fastest across a warp, and reads the rows of A21 and T22 four k at a time.  T22
// is lower triangular, so its sum stops at the tile's last row (rounded up to 4).
template <int RT>
__device__ __forceinline__ void gdn_double_level(float* Am, float* Tm, int n, int tid, bool ok) {
  const int nt = n / 4, per = (n / RT) * nt;  // column tiles; tiles per pair (128 / (2 n) pairs)
  const int i0 = (tid / per) * 2 * n, tj = (tid % nt) * 4, ti = ((tid % per) / nt) * RT;
  if (ok) {  // X = A21 T11
    float acc[RT][4] = {};
    const float* arow = Am + (i0 + n + ti) * kGP + i0;
#pragma unroll 1
    for (int k = 0; k < n; k += 4) {
      float4 av[RT];
#pragma unroll
      for (int ii = 0; ii < RT; ++ii) av[ii] = *reinterpret_cast<const float4*>(arow + ii * kGP + k);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float4 tv = *reinterpret_cast<const float4*>(Tm + (i0 + k + kk) * kGP + i0 + tj);
#pragma unroll
        for (int ii = 0; ii < RT; ++ii) {
          const float a = f4_at(av[ii], kk);
          acc[ii][0] += a * tv.x; acc[ii][1] += a * tv.y; acc[ii][2] += a * tv.z; acc[ii][3] += a * tv.w;
        }
      }
    }
#pragma unroll
    for (int ii = 0; ii < RT; ++ii)
      *reinterpret_cast<float4*>(Am + (i0 + ti + ii) * kGP + i0 + n + tj) =
          make_float4(acc[ii][0], acc[ii][1], acc[ii][2], acc[ii][3]);
  }
  __syncthreads();
  if (ok) {  // T21 = -T22 X
    // T22 is lower triangular, so a tile's sum runs over (ti + RT + 3) / 4 steps.  Warps w
    // and w + 4 share a sub-partition: warps 4..7 take their row tiles in reverse order
    // (within their pair, or within the upper half when one pair spans all warps), so that
    // each sub-partition gets a short and a long share while every warp keeps adjacent
    // rows (a uniform trip count).
    const int q = (tid % per) / nt;  // 16 row tiles per pair
    const int qr = tid < 128 ? q : (n == 64 ? 23 - q : 15 - q);
    const int ti = qr * RT;
    float acc[RT][4] = {};
    const float* trow = Tm + (i0 + n + ti) * kGP + i0 + n;
    const int kend = (ti + RT + 3) & ~3;
#pragma unroll 1
    for (int k = 0; k < kend; k += 4) {
      float4 tv[RT];
#pragma unroll
      for (int ii = 0; ii < RT; ++ii) tv[ii] = *reinterpret_cast<const float4*>(trow + ii * kGP + k);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float4 xv = *reinterpret_cast<const float4*>(Am + (i0 + k + kk) * kGP + i0 + n + tj);
#pragma unroll
        for (int ii = 0; ii < RT; ++ii) {
          const float t = f4_at(tv[ii], kk);
          acc[ii][0] += t * xv.x; acc[ii][1] += t * xv.y; acc[ii][2] += t * xv.z; acc[ii][3] += t * xv.w;
        }
      }
    }
#pragma unroll
    for (int ii = 0; ii < RT; ++ii)
      *reinterpret_cast<float4*>(Tm + (i0 + n + ti + ii) * kGP + i0 + tj) =
          make_float4(-acc[ii][0], -acc[ii][1], -acc[ii][2], -acc[ii][3]);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(256, 1) tc_gdn_local_kernel(const __grid_constant__ CUtensorMap mapK,
                                                              const __grid_constant__ CUtensorMap mapV,
                                                              TcGdnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* RK = smem;                                          // 32 KB: K (bf16)
  uint8_t* RV = smem + 32768;                                  // 16 KB: V (bf16)
  float* Am = reinterpret_cast<float*>(smem + 49152);          // 128 x kGP: A; later Kd hi, lo (fp16)
  float* Tm = Am + 128 * kGP;                                  // 128 x kGP: T; later T hi, lo (fp16)
  // (once the products have read them, the first 97 KB take the chunk's workspace record)
  float* gs = Tm + 128 * kGP;                                  // 128: g
  float* bs = gs + 128;                                        // 128: beta
  float* fk = bs + 128;                                        // 128: beta 2^g
  float* b8 = fk + 128;                                        // 128: 2^(g_end8(s) - g_s)
  uint8_t* VHI = reinterpret_cast<uint8_t*>(b8 + 128);         // 16 KB: diag(beta) V hi (fp16)
  uint8_t* VLO = VHI + 16384;                                  // 16 KB: ... lo
  __shared__ __align__(8) uint64_t bar_ld, bar_a, bar_w, bar_d;
  __shared__ uint32_t tmem_base;
  __shared__ float s_red[8];
  __shared__ float s_mx[8];
  __shared__ float s_kv[4][3];
  __shared__ float s_m3[8][3];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3;
  const int r = tid & 127, rot = r & 7;
  const int nch = p.T >> 7;
  const int total = p.B * p.H * nch;  // chunks: lin = (b nch + c) H + h
  // K and V of chunk lin into RK, RV (bar_ld)
  auto load_kv = [&](int lin) {
    const int h = lin % p.H, c = (lin / p.H) % nch, b = lin / (p.H * nch), g = h / p.hpg;
    ptx::mbar_arrive_expect_tx(&bar_ld, 32768 + 16384);
    ptx::tma_load_4d(RK, &mapK, &bar_ld, 0, g, c * kTile, b);
    ptx::tma_load_4d(RK + 16384, &mapK, &bar_ld, 64, g, c * kTile, b);
    ptx::tma_load_4d(RV, &mapV, &bar_ld, 0, h, c * kTile, b);
  };
  // a and beta of row r of chunk lin
  auto row_of = [&](int lin) {
    const int h = lin % p.H, c = (lin / p.H) % nch, b = lin / (p.H * nch);
    return ((size_t)b * p.T + (size_t)c * kTile + r) * p.H + h;
  };
  if (tid == 0) {
    ptx::mbar_init(&bar_ld, 1);
    ptx::mbar_init(&bar_a, 1);
    ptx::mbar_init(&bar_w, 1);
    ptx::mbar_init(&bar_d, 1);
    ptx::fence_mbar_init();
    load_kv(blockIdx.x);
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base, 256);
    ptx::tmem_relinquish();
  }
  float a_nx = p.a[row_of(blockIdx.x)], b_nx = tid < 128 ? p.beta[row_of(blockIdx.x)] : 0.f;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  // A persistent CTA per SM walks chunks lin = blockIdx.x, + gridDim.x, ...; the next
  // chunk's K and V are copied into RK and RV as soon as this chunk has read them (after
  // K's split), and its a and beta are loaded then too.  Barrier phases: bar_ld, bar_a and
  // bar_w complete once per chunk (parity it & 1), bar_d twice (parities 0, 1).
  bool ok = true;
  int ld_issued = 1;                 // K/V copies issued (tid 0); copy j completes phase j & 1
  // MMAs of the chunk in progress (cleared once a chunk has completed), for the final waits
  bool a_issued = false, w_issued = false;
  int d_issued = 0;
  int it = 0, ph = 0;
  for (int lin = blockIdx.x; ok && lin < total; lin += gridDim.x, ++it) {
  const int h = lin % p.H;
  const int c = (lin / p.H) % nch;
  const int b = lin / (p.H * nch);
  ph = it & 1;
  // chunk-local log2 decay cumsum (both halves of the block compute it)
  float gt = log2f(a_nx);
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
  const uint32_t tA = tbase, tW = tbase + 128, tU = tbase;
  if (tid < 128) {
    const float bt = b_nx;
    gs[r] = gt;
    bs[r] = bt;
    fk[r] = bt * exp2f(gt);
  }
  ok = wait_bar(&bar_ld, ph);
  if (!ok) atomicExch(p.status, kStatusTimeout);
  ok = __syncthreads_and(ok);
  if (!ok) break;
  if (tid == 0) {  // K Kᵀ: M = N = 128 tokens, K = 128 d_k, bf16, both K-major
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
  a_issued = true;
  if (tid < 128) b8[r] = exp2f(gs[r | 7] - gt);  // decay from key r to the end of its 8-block
  if (ok) {
    ok = wait_bar(&bar_a, ph);
    if (!ok) atomicExch(p.status, kStatusTimeout);
  }
  ok = __syncthreads_and(ok);
  // A_ts = beta_t 2^(g_t - g_s) (k_t . k_s), s < t (threads 0..127: row t); T zeroed by
  // the others.  Only the lower triangle of A is read later, so a warp stops at the 32-key
  // group of its own rows.  In an earlier group, 2^(g_t - g_s) is 2^(g_t - g_end8) b8[s]
  // (both factors <= 1) with one exp2 per 8-key block; the rows' own group takes one exp2
  // per key.
  if (ok) {
    ptx::tc_fence_after();
    if (tid < 128) {
      const int t = r;
      const float bt = bs[t];
#pragma unroll 1
      for (int c0 = 0; c0 <= quad * 32; c0 += 32) {  // warp-uniform
        float y[32];
        ptx::tmem_ld32(tA + lane_off + c0, y);
        ptx::tmem_ld_wait();
        if (c0 < quad * 32) {  // an earlier group: every block before t's (warp-uniform)
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            const int blk = (c0 >> 3) + kb;
            const float fb = bt * exp2f(gt - gs[8 * blk + 7]);
            const float4 b0 = *reinterpret_cast<const float4*>(b8 + 8 * blk);
            const float4 b1 = *reinterpret_cast<const float4*>(b8 + 8 * blk + 4);
            const float* yy = y + 8 * kb;
            *reinterpret_cast<float4*>(Am + t * kGP + 8 * blk) =
                make_float4(fb * b0.x * yy[0], fb * b0.y * yy[1], fb * b0.z * yy[2], fb * b0.w * yy[3]);
            *reinterpret_cast<float4*>(Am + t * kGP + 8 * blk + 4) =
                make_float4(fb * b1.x * yy[4], fb * b1.y * yy[5], fb * b1.z * yy[6], fb * b1.w * yy[7]);
          }
        } else {  // the rows' own group: one exp2 per key
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int s2 = c0 + j + e;
              v[e] = s2 < t ? bt * exp2f(gt - gs[s2]) * y[j + e] : 0.f;
            }
            *reinterpret_cast<float4*>(Am + t * kGP + c0 + j) = make_float4(v[0], v[1], v[2], v[3]);
          }
        }
      }
    } else {
      for (int e = 4 * r; e < 128 * kGP; e += 512) *reinterpret_cast<float4*>(Tm + e) = make_float4(0.f, 0.f, 0.f, 0.f);
      // the tile maxima of diag(beta 2^g) K and diag(beta) V (row r each), then V's fp16 hi
      // and lo parts (B operand, MN-major: row s, 64 d_v), by these otherwise idle warps
      uint32_t m0 = 0u, m1 = 0u;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const int off = r * 128 + ((cc ^ rot) << 4);
        m0 = absmax_u4(absmax_u4(m0, *reinterpret_cast<const uint4*>(RK + off)),
                       *reinterpret_cast<const uint4*>(RK + 16384 + off));
        m1 = absmax_u4(m1, *reinterpret_cast<const uint4*>(RV + off));
      }
      float kr = bf16x2_maxhalf(m0);
      float mk = kr * fabsf(fk[r]), mv = bf16x2_maxhalf(m1) * fabsf(bs[r]);
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, off));
        mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
        kr = fmaxf(kr, __shfl_xor_sync(0xffffffffu, kr, off));
      }
      if (lane == 0) {
        s_kv[warp - 4][0] = mk;
        s_kv[warp - 4][1] = mv;
        s_kv[warp - 4][2] = kr;
      }
      ptx::named_bar_sync(1, 128);
      const int ev = f16_exp(fmaxf(fmaxf(s_kv[0][1], s_kv[1][1]), fmaxf(s_kv[2][1], s_kv[3][1])));
      const float sc = bs[r] * pow2i(-ev);
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        const uint32_t off = r * 128 + ((cc ^ rot) << 4);
        uint4 hi, lo;
        split8_bf16(*reinterpret_cast<const uint4*>(RV + off), sc, hi, lo);
        *reinterpret_cast<uint4*>(VHI + off) = hi;
        *reinterpret_cast<uint4*>(VLO + off) = lo;
      }
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
  // Blocks below the diagonal by doubling: once the inverses T11 and T22 of two adjacent
  // diagonal blocks of size n are known, the block below them is T21 = -T22 A21 T11, A21
  // the block of A between them (the inverse of a 2 x 2 block lower triangle).  For n =
  // 16 and 32 every pair is done at once: X = A21 T11 into A's upper triangle (zero and
  // not read again) at rows i0.., columns i0 + n.., then T21 = -T22 X.  Each thread takes
  // n / 16 x 4 outputs (so all threads work at every level), the column tiles fastest
  // across a warp: the rows it reads of A21 and T22 are the same for many threads
  // (broadcasts), the rows of T11 and X are read along (conflict-free).
  gdn_double_level<1>(Am, Tm, 16, tid, ok);
  gdn_double_level<2>(Am, Tm, 32, tid, ok);
  // The n = 64 level on the tensor cores: T21 = -T22 X with X = A21 T11 (64 x 64 blocks),
  // as two M = 128 products with the A operand in tensor memory (free since the A phase)
  // and B in RV (free since V's split): X' = A[:, 0:64] T11, whose rows 64..127 are X,
  // then T21' = T[:, 64:128] X, whose rows 64..127 are T22 X (T's rows 0..63 are zero
  // there).  Every operand is split into fp16 high and low parts with a power-of-two tile
  // scale (hi hi + lo hi + hi lo, about 22 significant bits).  Thread (r, hf) holds row r,
  // K columns 32 hf .. 32 hf + 31 of the A operands; B rows are 64 d_k-wide, 128-byte
  // swizzled.
  {
    const int hf = tid >> 7;
    uint8_t* BHI = RV;           // B operand, hi (64 rows x 128 B)
    uint8_t* BLO = RV + 8192;    // ... lo
    const int kb = tid >> 2, qb = tid & 3;  // T11 row and 16-column quarter of this thread
    float mA = 0.f, m1 = 0.f, m2 = 0.f;
    if (ok) {
      const float* ar = Am + r * kGP + 32 * hf;
      const float* t2 = Tm + r * kGP + 64 + 32 * hf;
      const float* t1 = Tm + kb * kGP + 16 * qb;
      if (r >= 64)  // rows 0..63 of A's first 64 columns hold the smaller levels' X blocks
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float4 x = *reinterpret_cast<const float4*>(ar + j), y = *reinterpret_cast<const float4*>(t2 + j);
          mA = fmaxf(mA, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
          m2 = fmaxf(m2, fmaxf(fmaxf(fabsf(y.x), fabsf(y.y)), fmaxf(fabsf(y.z), fabsf(y.w))));
        }
#pragma unroll
      for (int j = 0; j < 16; j += 4) {
        const float4 x = *reinterpret_cast<const float4*>(t1 + j);
        m1 = fmaxf(m1, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, off));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, off));
      m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, off));
    }
    if (lane == 0) {
      s_m3[warp][0] = mA;
      s_m3[warp][1] = m1;
      s_m3[warp][2] = m2;
    }
    __syncthreads();
    float xA = 0.f, x1 = 0.f, x2 = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      xA = fmaxf(xA, s_m3[w][0]);
      x1 = fmaxf(x1, s_m3[w][1]);
      x2 = fmaxf(x2, s_m3[w][2]);
    }
    const int eA = f16_exp(xA), e1 = f16_exp(x1), e2 = f16_exp(x2);
    // A[r, 32 hf ..] (which 0) or T[r, 64 + 32 hf ..] (which 1) -> fp16 hi, lo in TMEM
    // columns 16 hf .. of tA (hi: + 0..31, lo: + 32..63) or of tW
    auto a_operand = [&](int which) {
      {
        const float* src = which == 0 ? Am + r * kGP + 32 * hf : Tm + r * kGP + 64 + 32 * hf;
        const float sc = pow2i(-(which == 0 ? eA : e2));
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          // rows 0..63 take zeros (their products are not read; T is zero there anyway)
          const float4 x0 = r >= 64 ? *reinterpret_cast<const float4*>(src + 8 * q8) : make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 x1v =
              r >= 64 ? *reinterpret_cast<const float4*>(src + 8 * q8 + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
          const float v8[8] = {x0.x, x0.y, x0.z, x0.w, x1v.x, x1v.y, x1v.z, x1v.w};
          uint4 h4, l4;
          split8(v8, sc, h4, l4);
          hi[4 * q8] = h4.x; hi[4 * q8 + 1] = h4.y; hi[4 * q8 + 2] = h4.z; hi[4 * q8 + 3] = h4.w;
          lo[4 * q8] = l4.x; lo[4 * q8 + 1] = l4.y; lo[4 * q8 + 2] = l4.z; lo[4 * q8 + 3] = l4.w;
        }
        const uint32_t tb = (which == 0 ? tA : tW) + lane_off;
        ptx::tmem_st16(tb + 16 * hf, hi);
        ptx::tmem_st16(tb + 32 + 16 * hf, lo);
      }
    };
    if (ok) {
      a_operand(0);
      // T11 row kb, columns 16 qb .. 16 qb + 15 (chunks 2 qb, 2 qb + 1) -> B hi, lo
      const float sc1 = pow2i(-e1);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const float* src = Tm + kb * kGP + 16 * qb + 8 * h2;
        const float4 x0 = *reinterpret_cast<const float4*>(src);
        const float4 x1v = *reinterpret_cast<const float4*>(src + 4);
        const float v8[8] = {x0.x, x0.y, x0.z, x0.w, x1v.x, x1v.y, x1v.z, x1v.w};
        uint4 h4, l4;
        split8(v8, sc1, h4, l4);
        const int off = kb * 128 + (((2 * qb + h2) ^ (kb & 7)) << 4);
        *reinterpret_cast<uint4*>(BHI + off) = h4;
        *reinterpret_cast<uint4*>(BLO + off) = l4;
      }
      ptx::tmem_st_wait();
      ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    ok = __syncthreads_and(ok);
    const uint32_t id64 = ptx::idesc_f16_f32(128, 64, 0, 1);
    const uint32_t b0 = ptx::smem_u32(RV);
    auto issue = [&](uint32_t dcol, uint32_t acol) {  // D (+)= A (TMEM hi/lo) B (smem hi/lo)
      ptx::tc_fence_after();
      const uint32_t ao[3] = {0, 32, 0}, bo[3] = {0, 0, 8192};
#pragma unroll
      for (int pass = 0; pass < 3; ++pass)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::umma_f16_tmem_a(dcol, acol + ao[pass] + kk * 8, ptx::smem_desc_sw128(b0 + bo[pass] + kk * 2048, 1024, 1024),
                               id64, pass > 0 || kk > 0);
      ptx::umma_commit(&bar_d);
    };
    if (ok && tid == 0) {
      issue(tA + 64, tA);  // X' = A[:, 0:64] T11
      ++d_issued;
    }
    if (ok) {  // T22's operand while the product runs (tW is not touched by it)
      a_operand(1);
      ptx::tmem_st_wait();
      ok = wait_bar(&bar_d, 0);
      if (!ok) atomicExch(p.status, kStatusTimeout);
    }
    ptx::tc_fence_before();
    ok = __syncthreads_and(ok);
    // X (rows 64..127 of X', lanes 64..127) -> hi, lo as B (row r - 64), with the scale of
    // a bound: |X'| <= 64 max|A op| max|T11 op| (a few binades above the maximum at most;
    // fp16 keeps 29 binades below 2^15 in its normal range)
    const int eX = f16_exp(64.f * (xA * pow2i(-eA)) * (x1 * pow2i(-e1)));
    if (ok && r >= 64) {
      float xv[32];
      ptx::tc_fence_after();
      ptx::tmem_ld32(tA + 64 + lane_off + 32 * hf, xv);
      ptx::tmem_ld_wait();
      const float scx = pow2i(-eX);
      const int k = r - 64;
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        const float v8[8] = {xv[8 * q8], xv[8 * q8 + 1], xv[8 * q8 + 2], xv[8 * q8 + 3],
                             xv[8 * q8 + 4], xv[8 * q8 + 5], xv[8 * q8 + 6], xv[8 * q8 + 7]};
        uint4 h4, l4;
        split8(v8, scx, h4, l4);
        const int off = k * 128 + (((4 * hf + q8) ^ (k & 7)) << 4);
        *reinterpret_cast<uint4*>(BHI + off) = h4;
        *reinterpret_cast<uint4*>(BLO + off) = l4;
      }
      ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    ok = __syncthreads_and(ok);
    if (ok && tid == 0) {
      issue(tW + 64, tW);  // T21' = T[:, 64:128] X
      ++d_issued;
    }
    if (ok) {
      ok = wait_bar(&bar_d, 1);
      if (!ok) atomicExch(p.status, kStatusTimeout);
    }
    ok = __syncthreads_and(ok);
    // T21 = -T21' 2^(e2 + eX + eA + e1): rows 64..127, columns 0..63 of T
    if (ok && r >= 64) {
      ptx::tc_fence_after();
      float y[32];
      ptx::tmem_ld32(tW + 64 + lane_off + 32 * hf, y);
      ptx::tmem_ld_wait();
      const float sc = -pow2s(e2 + eX) * pow2s(eA + e1);
      float* dst = Tm + r * kGP + 32 * hf;
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(dst + j) = make_float4(sc * y[j], sc * y[j + 1], sc * y[j + 2], sc * y[j + 3]);
    }
    ptx::tc_fence_before();
    __syncthreads();
  }
  // T's tile scale (the maximum over its elements; those of K and V came with the A
  // phase): every thread keeps half of its row r (columns 64 hf ..) in registers, so that
  // T's hi and lo parts can go over T itself.  Meanwhile diag(beta 2^g) K -> fp16 hi, lo
  // (B operands, MN-major: row s, d_k in two 64-wide boxes) into A's space, free since
  // the doubling.
  const int hf = tid >> 7;
  float4 tr[16];
  float mt = 0.f;
  uint8_t* KHI = reinterpret_cast<uint8_t*>(Am);
  uint8_t* KLO = KHI + 32768;
  if (ok) {
    const float4* trow = reinterpret_cast<const float4*>(Tm + r * kGP + hf * 64);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      tr[j] = trow[j];
      mt = fmaxf(mt, fmaxf(fmaxf(fabsf(tr[j].x), fabsf(tr[j].y)), fmaxf(fabsf(tr[j].z), fabsf(tr[j].w))));
    }
    const int ek = f16_exp(fmaxf(fmaxf(s_kv[0][0], s_kv[1][0]), fmaxf(s_kv[2][0], s_kv[3][0])));
    const float sc = fk[r] * pow2i(-ek);
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const uint32_t off = hf * 16384 + r * 128 + ((cc ^ rot) << 4);
      uint4 hi, lo;
      split8_bf16(*reinterpret_cast<const uint4*>(RK + off), sc, hi, lo);
      *reinterpret_cast<uint4*>(KHI + off) = hi;
      *reinterpret_cast<uint4*>(KLO + off) = lo;
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
  if (lane == 0) s_mx[warp] = mt;
  __syncthreads();  // also: every thread has read its part of T, and RK, RV are free
  const int nx = lin + gridDim.x;
  if (nx < total) {  // the next chunk's K, V (into the buffers read for the last time above), a, beta
    if (ok && tid == 0) {
      ptx::fence_proxy_async_smem();
      load_kv(nx);
      ++ld_issued;
    }
    a_nx = p.a[row_of(nx)];
    if (tid < 128) b_nx = p.beta[row_of(nx)];
  }
  float mxt = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) mxt = fmaxf(mxt, s_mx[w]);
  const int et = f16_exp(mxt);
  const int ek = f16_exp(fmaxf(fmaxf(s_kv[0][0], s_kv[1][0]), fmaxf(s_kv[2][0], s_kv[3][0])));
  const int ev = f16_exp(fmaxf(fmaxf(s_kv[0][1], s_kv[1][1]), fmaxf(s_kv[2][1], s_kv[3][1])));
  // T -> fp16 hi, lo (A operands, K-major: row t, columns s in two 64-wide boxes) over T
  uint8_t* THI = reinterpret_cast<uint8_t*>(Tm);
  uint8_t* TLO = THI + 32768;
  if (ok) {
    const float sc = pow2i(-et);
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const float4 x0 = tr[2 * cc], x1 = tr[2 * cc + 1];
      const float src[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      uint4 hi, lo;
      split8(src, sc, hi, lo);
      const uint32_t off = hf * 16384 + r * 128 + ((cc ^ rot) << 4);
      *reinterpret_cast<uint4*>(THI + off) = hi;
      *reinterpret_cast<uint4*>(TLO + off) = lo;
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
  w_issued = ok;
  if (ok) {
    ok = wait_bar(&bar_w, ph);
    if (!ok) atomicExch(p.status, kStatusTimeout);
  }
  ok = __all_sync(0xffffffffu, ok);
  // W: its tile maximum, then hi and lo fp16 of W 2^-ew in the operand layout; U_loc, g.
  // The chunk's workspace record is put together in shared memory from T's space on (T's
  // and V's parts and the small tables, all read for the last time by the products; RK and
  // RV hold the next chunk's K and V by now), in its global layout, then copied out by all
  // threads with consecutive 16-byte stores.
  uint8_t* dst = reinterpret_cast<uint8_t*>(Tm);
  const float sw = pow2s(et + ek), su = pow2s(et + ev);
  // Every thread takes half of its row r: W's d_k columns 64 hf .. 64 hf + 63 (the box hf of
  // the operand layout) and U_loc's d_v columns 32 hf .. 32 hf + 31.
  // W's scale from a bound, with no pass over W: |W| <= 128 max|T| max|diag(beta 2^g) K|
  // (at most a few binades above W's maximum; fp16 keeps 29 below 2^15 in its normal range)
  const float xk = fmaxf(fmaxf(s_kv[0][0], s_kv[1][0]), fmaxf(s_kv[2][0], s_kv[3][0]));
  const int ew = f16_exp(128.f * mxt * xk);
  if (ok) {
    ptx::tc_fence_after();
    const float sc = sw * pow2i(-ew);
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 32) {
      float y[32];
      ptx::tmem_ld32(tW + lane_off + hf * 64 + c0, y);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {  // d_k columns 64 hf + c0 + 8 q4 .. + 7: one 16-byte chunk
        const int cc = (c0 >> 3) + q4;
        const float src[8] = {y[8 * q4], y[8 * q4 + 1], y[8 * q4 + 2], y[8 * q4 + 3],
                              y[8 * q4 + 4], y[8 * q4 + 5], y[8 * q4 + 6], y[8 * q4 + 7]};
        uint4 hi, lo;
        split8(src, sc, hi, lo);
        const size_t off = (size_t)hf * 16384 + r * 128 + ((cc ^ rot) << 4);
        *reinterpret_cast<uint4*>(dst + off) = hi;
        *reinterpret_cast<uint4*>(dst + 32768 + off) = lo;
      }
    }
    // U_loc row r: 16-byte chunk j of its half goes to chunk j ^ (r & 7) of that half
    float* du = reinterpret_cast<float*>(dst + kGdnOffU) + r * kDv + hf * 32;
    {
      float y[32];
      ptx::tmem_ld32(tU + lane_off + hf * 32, y);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(du + 4 * (j ^ rot)) =
            make_float4(su * y[4 * j], su * y[4 * j + 1], su * y[4 * j + 2], su * y[4 * j + 3]);
    }
    if (hf == 0) reinterpret_cast<float*>(dst + kGdnOffG)[r] = gt;
    if (tid == 0) {
      *reinterpret_cast<int*>(dst + kGdnOffE) = ew;
      *reinterpret_cast<int*>(dst + kGdnOffE + 4) =
          f16_exp(fmaxf(fmaxf(s_kv[0][2], s_kv[1][2]), fmaxf(s_kv[2][2], s_kv[3][2])));
    }
  }
  ok = __syncthreads_and(ok);  // the record is complete
  if (ok) {
    uint4* gdst = reinterpret_cast<uint4*>(p.xw + ((size_t)(b * p.H + h) * nch + c) * kGdnChunkBytes);
    const uint4* ssrc = reinterpret_cast<const uint4*>(dst);
    for (int i = tid; i < (int)(kGdnChunkBytes / 16); i += 256) gdst[i] = ssrc[i];
  }
  ptx::tc_fence_before();
  __syncthreads();  // the record and TMEM are read before the next chunk writes them
  if (ok) {
    a_issued = w_issued = false;
    d_issued = 0;
  }
  }
  if (tid == 0) {  // bounded: let this CTA's copies and MMAs land before TMEM goes
    wait_bar(&bar_ld, (ld_issued - 1) & 1);
    if (a_issued) wait_bar(&bar_a, ph);
    if (d_issued) wait_bar(&bar_d, (d_issued - 1) & 1);
    if (w_issued) wait_bar(&bar_w, ph);
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
//   behind the product W S; K's fp16 scale comes with the chunk's record, so each thread
//   converts its row of K while W S runs.
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
  const int bh = p.b0 * p.H + blockIdx.x, b = bh / p.H, h = bh % p.H, g = h / p.hpg;
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
  // |Ŝ| <= sb: Ŝ starts at zero; each chunk scales it by f and adds Kᵀ ũ of fp16 operands
  // below 2^15 over 128 tokens, at most 2^37 (a few binades above Ŝ's maximum at most;
  // fp16 keeps 29 below 2^15 in its normal range)
  float sb = 0.f;
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
      // the next chunk's U_loc, g and scale word, and its K tile, into L2: their loads come
      // one chunk later, on this CTA's serial path
      bulk_prefetch_l2(xc + kGdnChunkBytes + kGdnOffU, 32768 + 512 + 16);
      tma_prefetch_4d(&mapK, 0, g, (c + 1) * kTile, b);
      tma_prefetch_4d(&mapK, 64, g, (c + 1) * kTile, b);
    }
    const int tokr = c * kTile + r;  // this thread's token (rows of u, Z)
    // this thread's half of U_loc row r, and g
    float uu[32];
    {
      const float4* us = reinterpret_cast<const float4*>(xc + kGdnOffU) + (r * kDv + hf * 32) / 4;
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // chunk j of the half row sits at j ^ (r & 7)
        const float4 v = us[j ^ rot];
        uu[4 * j] = v.x;
        uu[4 * j + 1] = v.y;
        uu[4 * j + 2] = v.z;
        uu[4 * j + 3] = v.w;
      }
      if (tid < 128) sg[r] = reinterpret_cast<const float*>(xc + kGdnOffG)[r];
    }
    const int ew = *reinterpret_cast<const int*>(xc + kGdnOffE);
    const int ek = *reinterpret_cast<const int*>(xc + kGdnOffE + 4);
    // Ŝ (lane r = d_k row), with the fp16 scale of its running bound (no block maximum)
    float sv[32];
    ptx::tc_fence_after();
    ptx::tmem_ld32(tS + lane_off, sv);
    ptx::tmem_ld_wait();
    const int es = f16_exp(sb);
    {  // Ŝ 2^-es -> hi, lo: row r, d_v columns 32 hf .. (chunks 4 hf ..)
      const float sc = pow2i(-es);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float src[8] = {sv[8 * q4], sv[8 * q4 + 1], sv[8 * q4 + 2], sv[8 * q4 + 3],
                              sv[8 * q4 + 4], sv[8 * q4 + 5], sv[8 * q4 + 6], sv[8 * q4 + 7]};
        uint4 hi, lo;
        split8(src, sc, hi, lo);
        const int off = r * 128 + (((4 * hf + q4) ^ rot) << 4);
        *reinterpret_cast<uint4*>(RS + off) = hi;
        *reinterpret_cast<uint4*>(RS + 16384 + off) = lo;
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
    // K of this chunk (by TMA, issued after the last chunk's Kᵀ ũ): this thread's half row
    // to fp16 2^-ek in place, while W S runs
    uint8_t* krow = RK + hf * 16384 + r * 128;
    const bool okk = wait_bar(&bar_k, c & 1);
    if (okk) {
      if (tid == 0) ++k_done;
      const float sk = pow2i(-ek);
      const __nv_bfloat162 k2 = __floats2bfloat162_rn(sk, sk);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint4* x = reinterpret_cast<uint4*>(krow + ((cc ^ rot) << 4));
        *x = bf16x8_to_f16x8(*x, k2);
      }
    } else {
      atomicExch(p.status, kStatusTimeout);
    }
    bool okz = wait_bar(&bar_z, c & 1);
    if (!okz) atomicExch(p.status, kStatusTimeout);
    okz = __syncthreads_and(okz && okk);
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
    // ũ's tile maximum
#pragma unroll
    for (int off = 16; off; off >>= 1) mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, off));
    if (lane == 0) s_mx[warp][0] = mu;
    __syncthreads();
    float mxu = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) mxu = fmaxf(mxu, s_mx[w][0]);
    const int eu = f16_exp(mxu);
    {  // ũ 2^-eu -> hi, lo (row r = token, d_v columns 32 hf ..)
      const float sc = pow2i(-eu);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float src[8] = {uu[8 * q4], uu[8 * q4 + 1], uu[8 * q4 + 2], uu[8 * q4 + 3],
                              uu[8 * q4 + 4], uu[8 * q4 + 5], uu[8 * q4 + 6], uu[8 * q4 + 7]};
        uint4 hi, lo;
        split8(src, sc, hi, lo);
        const int off = r * 128 + (((4 * hf + q4) ^ rot) << 4);
        *reinterpret_cast<uint4*>(RU + off) = hi;
        *reinterpret_cast<uint4*>(RU + 16384 + off) = lo;
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
      sb = f * sb + 137438953472.f;  // 2^37
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

}  // namespace

size_t tc_gdn_bytes(const ll_shape& s) {
  return (size_t)s.batch * s.heads * (s.T / kTile) * kGdnChunkBytes;
}

namespace {
bool tc_gdn_params(const ll_shape& s, const void* k, const void* v, const float* a, const float* beta, void* u,
                   char* ws, unsigned* status, CUtensorMap* mK, CUtensorMap* mV, TcGdnParams* p) {
  if (!tc_supported(s)) return false;
  const int G = s.heads / s.heads_per_group;
  if (!make_map(mK, k, kDk, G, s.T, s.batch) || !make_map(mV, v, kDv, s.heads, s.T, s.batch)) return false;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    nsm = 0;  // no prefetch
  *p = TcGdnParams{s.batch, s.T, s.heads, s.heads_per_group, G, a, beta, reinterpret_cast<uint8_t*>(ws), nsm, 0, u,
                   status};
  return true;
}
}  // namespace

cudaError_t launch_tc_gdn_local(const ll_shape& s, const void* k, const void* v, const float* a, const float* beta,
                                void* u, char* ws, unsigned* status, cudaStream_t st) {
  CUtensorMap mK, mV;
  TcGdnParams p;
  if (!tc_gdn_params(s, k, v, a, beta, u, ws, status, &mK, &mV, &p)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_gdn_local_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemGdnL);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (its shared memory allows no more), chunks in turn
  const size_t total = (size_t)s.batch * s.heads * (s.T / kTile);
  const unsigned grid = (unsigned)(p.pf_stride > 0 && (size_t)p.pf_stride < total ? p.pf_stride : total);
  tc_gdn_local_kernel<<<grid, 256, kSmemGdnL, st>>>(mK, mV, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

cudaError_t launch_tc_gdn_pass(const ll_shape& s, int b0, int nb, const void* k, const void* v, const float* a,
                               const float* beta, void* u, char* ws, unsigned* status, cudaStream_t st) {
  CUtensorMap mK, mV;
  TcGdnParams p;
  if (b0 < 0 || nb < 1 || b0 + nb > s.batch) return cudaErrorInvalidValue;
  if (!tc_gdn_params(s, k, v, a, beta, u, ws, status, &mK, &mV, &p)) return cudaErrorInvalidValue;
  p.b0 = b0;
  cudaError_t e = cudaFuncSetAttribute(tc_gdn_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemGdnP);
  if (e != cudaSuccess) return e;
  tc_gdn_pass_kernel<<<(unsigned)(nb * s.heads), 256, kSmemGdnP, st>>>(mK, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

cudaError_t launch_tc_gdn(const ll_shape& s, const void* k, const void* v, const float* a, const float* beta,
                          void* u, char* ws, unsigned* status, cudaStream_t st) {
  cudaError_t e = launch_tc_gdn_local(s, k, v, a, beta, u, ws, status, st);
  if (e != cudaSuccess) return e;
  return launch_tc_gdn_pass(s, 0, s.batch, k, v, a, beta, u, ws, status, st);
}

}  // namespace ll
