// Tensor-core kernels of the backward (for bf16, d_k = 128, d_v = 64, T % 128 == 0): the
// in-tile pairs (tc_bwd_intra), the query side of the inter-tile levels (tc_bwd_q) and
// their key side (tc_tile_prefix, tc_dual_publish, tc_bwd_kv), over the forward's tree of
// tile nodes (tc_fwd.cu).  The chain rule they follow is set out in backward.cu.
#include "tc_common.cuh"

namespace ll {

namespace {

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
  float* cu;     // (B, T, H): C_s = sum_t A_ts over the in-tile pairs (fp32, from S and E);
                 // followed by R_t = sum_l lambda_t^l dlambda_t^l over levels 0..7 (B, T, H)
  unsigned* status;
  int pf_stride;  // the CTA this far ahead (the SM count) gets its tiles prefetched into L2
};

// L2 prefetch of one tile through a 4-D tensor map (no shared memory, no completion)
__device__ __forceinline__ void tma_prefetch_4d(const void* tmap, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(tmap), "r"(c0),
               "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

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
                                                              const __grid_constant__ CUtensorMap mapDQ,
                                                              const __grid_constant__ CUtensorMap mapDK,
                                                              const __grid_constant__ CUtensorMap mapDV,
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
    // One CTA per SM: the CTA that will most likely run next on this SM (one SM count
    // ahead) finds its tiles in L2.
    const int l2 = lin + p.pf_stride;
    if (p.pf_stride > 0 && l2 < (int)gridDim.x) {
      const int h2 = l2 % p.H, u2 = (l2 / p.H) % p.NT, b2 = l2 / (p.H * p.NT), g2 = h2 / p.hpg;
      tma_prefetch_4d(&mapQ, 0, g2, u2 * kTile, b2);
      tma_prefetch_4d(&mapQ, 64, g2, u2 * kTile, b2);
      tma_prefetch_4d(&mapK, 0, g2, u2 * kTile, b2);
      tma_prefetch_4d(&mapK, 64, g2, u2 * kTile, b2);
      tma_prefetch_4d(&mapV, 0, h2, u2 * kTile, b2);
      tma_prefetch_4d(&mapD, 0, h2, u2 * kTile, b2);
    }
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
      const float* lamr = sLam8 + r * 9;
      float dv8[kLevIntra];
#pragma unroll
      for (int l = 0; l < 6; ++l) dv8[l] = accr[l];
      dv8[6] = acc6 + accr[6];
      dv8[7] = acc7 + accr[7];
      float R = 0.f;  // this row's part of R_t (d(log a) reads it instead of lambda and dlambda)
#pragma unroll
      for (int l = 0; l < kLevIntra; ++l) {
        dl[l] = dv8[l];
        R += lamr[l] * dv8[l];
      }
      p.cu[(size_t)p.B * p.T * p.H + row * p.H + h] = R;
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
  // The fp32 rows of dq and dv's columns 0..31 (role a), dk and dv's columns 32..63 (role
  // b) are staged in the tile buffers, free now (every MMA has read them), as
  // 128-byte-swizzled boxes of 32 columns (dq: 4 boxes from 0, dk: 4 from 64 KB, dv: 2
  // from 128 KB), and each role writes its boxes with TMA stores as soon as they are
  // staged, while the other role may still be staging.  Thread r writes row r of a box as
  // eight 16-byte chunks, chunk c at c ^ (r & 7).
  auto stage_row = [&](uint8_t* box, const float (&y)[32], float sc) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<float4*>(box + r * 128 + ((c ^ rot) << 4)) =
          make_float4(sc * y[4 * c], sc * y[4 * c + 1], sc * y[4 * c + 2], sc * y[4 * c + 3]);
  };
  const float sv = pow2s(s_sc[1] + s_sc[4]);  // P and dO
  if (ok) {
    ptx::tc_fence_after();
    const float sx = role_b ? pow2s(s_sc[0] + s_sc[2]) : pow2s(s_sc[0] + s_sc[3]);  // dS and Q / dS and K
    const uint32_t tX = role_b ? tDK : tDQ;
    uint8_t* bx = smem + (role_b ? 65536 : 0);
#pragma unroll 1
    for (int c0 = 0; c0 < kDk; c0 += 32) {
      float y[32];
      ptx::tmem_ld32(tX + lane_off + c0, y);
      ptx::tmem_ld_wait();
      stage_row(bx + (c0 >> 5) * 16384, y, sx);
    }
    {
      const int hv = role_b ? 1 : 0;
      float y[32];
      ptx::tmem_ld32(tDV + lane_off + 32 * hv, y);
      ptx::tmem_ld_wait();
      stage_row(smem + 131072 + hv * 16384, y, sv);
    }
    ptx::fence_proxy_async_smem();
  }
  if (role_b) ok = ptx::named_bar_and(4, 128, ok);  // this role's rows staged
  else ok = ptx::named_bar_and(3, 128, ok);
  if (ok && (tid & 127) == 0) {
    const CUtensorMap* mX = role_b ? &mapDK : &mapDQ;
    uint8_t* bx = smem + (role_b ? 65536 : 0);
    const int hv = role_b ? 1 : 0;
    for (int j = 0; j < 4; ++j) ptx::tma_store_4d(mX, bx + j * 16384, 32 * j, h, (int)t0, b);
    ptx::tma_store_4d(&mapDV, smem + 131072 + hv * 16384, 32 * hv, h, (int)t0, b);
    ptx::bulk_commit_group();
    ptx::bulk_wait_read_all();  // the staging is read before the CTA ends
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
  float* ru;          // (B, T, H): R_t, to which the inter-tile levels' lambda dlambda is added
  // non-null: a tile node's dual (one reader tile, this one) goes straight to its fp16
  // image (dimg: 16 KB per slot) and scale exponent (dmeta[slot * kMeta + 1]), not to dual
  uint8_t* dimg;
  unsigned* dmeta;
  unsigned* status;
};

constexpr int kBwdQFixed = 98304;  // Q, dO, two node images, diag(w) dO
__host__ __device__ constexpr int bwdq_smem_bytes(int ninter) {
  return kBwdQFixed + 512 * (ninter > 0 ? ninter : 1) + 1024;
}

__global__ void __launch_bounds__(256, 2) tc_bwd_q_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                          const __grid_constant__ CUtensorMap mapD,
                                                          const __grid_constant__ CUtensorMap mapDQ,
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
  __shared__ float s_dmx[8];

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
  float Rq = 0.f;  // sum over this tile's inter levels of lambda_t^(8+m) dlambda_t^(8+m)
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
      for (int q = 0; q < 4; ++q) {  // 16 columns at a time (fewer live registers)
        float y[16];
        ptx::tmem_ld16(tY + lane_off + q * 16, y);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4 x = *reinterpret_cast<const uint4*>(drow + (((2 * q + c) ^ rot) << 4));
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
            dot += y[c * 8 + 2 * e] * v.x + y[c * 8 + 2 * e + 1] * v.y;
          }
        }
      }
      const float dlm = exp2f(gt + D) * pow2s(eq + en + ed) * dot;
      p.dlam[(row * p.H + h) * p.L + kLevIntra + m] = dlm;
      Rq += sLamI[i * 128 + r] * dlm;
    }
    {  // dual rows (TMEM lane = d_k index r), d_v columns 32 hf .. 32 hf + 31
      const int tau = tau_of(i);
      const float su = pow2s(eq + tau);
      float y[32];
      ptx::tmem_ld32(tU + lane_off + hf * 32, y);
      ptx::tmem_ld_wait();
      const int nd = (u >> m) - 1;  // even
      const size_t slot = (size_t)bh * p.nslots + p.dual_off[m] + (nd >> 1);
      float* dst = p.dual + (slot * kDk + r) * kDv + hf * 32;
      if (m == 0 && p.dimg) {  // a tile node's dual, complete here: its fp16 image and scale
        float mx = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          y[j] *= su;
          mx = fmaxf(mx, fabsf(y[j]));
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) s_dmx[warp] = mx;
        __syncthreads();
        float bm = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) bm = fmaxf(bm, s_dmx[w]);
        const int e = f16_exp(bm);
        const float sc = pow2i(-e);
        uint8_t* im = p.dimg + slot * kImgBytes + r * 128;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {  // columns 32 hf + 8 q4 ..: the row's 16-byte chunk 4 hf + q4
          const float* x = y + 8 * q4;
          *reinterpret_cast<uint4*>(im + (((4 * hf + q4) ^ rot) << 4)) =
              make_uint4(pack_h2(x[0] * sc, x[1] * sc), pack_h2(x[2] * sc, x[3] * sc), pack_h2(x[4] * sc, x[5] * sc),
                         pack_h2(x[6] * sc, x[7] * sc));
        }
        if (tid == 0) {
          p.dmeta[slot * kMeta + 1] = (unsigned)e;
          p.dmeta[slot * kMeta + 2] = __float_as_uint(0.f);
        }
      } else if (m == 0) {  // a tile node's dual has one reader tile, this one: stored, not added
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(dst + j) = make_float4(su * y[j], su * y[j + 1], su * y[j + 2], su * y[j + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          atomicAdd(reinterpret_cast<float4*>(dst + j),
                    make_float4(su * y[j], su * y[j + 1], su * y[j + 2], su * y[j + 3]));
      }
    }
    D += sNode[i][1];
    if (i + 1 < nlev) {  // diag(w) dO of the next level (its MMA has read this one)
      write_b(i + 1, D, tau_of(i + 1));
      ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(&bar_yf);
  }
  // the in-tile kernel wrote its part; a reduction (not a load and a store) keeps the
  // read off this CTA's path, and this is the only addition to the value
  if (ok && hf == 0) atomicAdd(p.ru + row * p.H + h, Rq);
  // dq rows (columns 64 hf .. 64 hf + 63: boxes 2 hf, 2 hf + 1) are staged over Q, dO and
  // the images, free once every level is read, and added into the per-head buffer (which
  // the in-tile kernel wrote) with TMA reductions.
  __syncthreads();
  if (ok) {
#pragma unroll
    for (int j2 = 0; j2 < 2; ++j2) {
      uint8_t* box = smem + (2 * hf + j2) * 16384 + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(box + ((c ^ rot) << 4)) =
            make_float4(acc[32 * j2 + 4 * c], acc[32 * j2 + 4 * c + 1], acc[32 * j2 + 4 * c + 2],
                        acc[32 * j2 + 4 * c + 3]);
    }
    ptx::fence_proxy_async_smem();
  }
  ok = __syncthreads_and(ok);
  if (ok && tid == 0) {
    for (int j = 0; j < 4; ++j) ptx::tma_reduce_add_4d(&mapDQ, smem + j * 16384, 32 * j, h, (int)t0, b);
    ptx::bulk_commit_group();
    ptx::bulk_wait_read_all();  // the staging is read before the CTA ends
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

// One CTA per dual slot: the fp32 dual (d_k x d_v) -> its fp16 image with a power-of-two
// scale, as a node is published.  The threads read the slot in consecutive 16-byte pieces
// (thread i: pieces i, i + 128, ...), not a row each, so that every warp load is four whole
// 128-byte lines; each piece is half of a 16-byte chunk of the image.
__global__ void __launch_bounds__(128) tc_dual_publish_kernel(const float* dual, uint8_t* img, unsigned* meta,
                                                              int nslots, int n0) {
  __shared__ __align__(1024) uint8_t stage[kImgBytes];
  __shared__ float2 s_red2[4];
  const int tid = threadIdx.x;
  // slots n0 .. nslots - 1 of each (b, h) (those below n0 were published by tc_bwd_q)
  const size_t slot = (size_t)(blockIdx.x / (nslots - n0)) * nslots + n0 + blockIdx.x % (nslots - n0);
  const float4* src = reinterpret_cast<const float4*>(dual + slot * kDk * kDv);
  constexpr int kPieces = kDk * kDv / 4 / 128;  // 16 per thread
  float4 v[kPieces];
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < kPieces; ++i) {
    v[i] = src[tid + 128 * i];
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
  }
  const int e = f16_exp(block_max2(make_float2(m, 0.f), s_red2).x);
  const float sc = pow2i(-e);
#pragma unroll
  for (int i = 0; i < kPieces; ++i) {
    const int idx = tid + 128 * i;           // piece: elements 4 idx .. 4 idx + 3
    const int row = idx >> 4, c = (idx & 15) >> 1, half = idx & 1;  // d_k row, 8-column chunk
    *reinterpret_cast<uint2*>(stage + row * 128 + ((c ^ (row & 7)) << 4) + half * 8) =
        make_uint2(pack_h2(v[i].x * sc, v[i].y * sc), pack_h2(v[i].z * sc, v[i].w * sc));
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(img + slot * kImgBytes);
#pragma unroll
  for (int r = 0; r < kImgBytes / 16 / 128; ++r) dst[r * 128 + tid] = reinterpret_cast<const uint4*>(stage)[r * 128 + tid];
  if (tid == 0) {
    meta[slot * kMeta + 1] = (unsigned)e;
    meta[slot * kMeta + 2] = __float_as_uint(0.f);
  }
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
  int pf_stride;  // the CTA this far ahead (the SM count) gets its K and V tiles prefetched into L2
};

// K, V, two dual images (then the dk staging and dv's bf16 staging), the in-tile part of dv
constexpr int kSmemBwdKV = 98304 + 32768 + 1024;

// dv of row r, columns 16 qq .. 16 qq + 15: the in-tile part (fp32 boxes of 32 columns with
// the 128-byte swizzle, as loaded) plus add[] (already weighted), as bf16 into the 64-wide
// output box (the same swizzle) of the staging area.
__device__ __forceinline__ void kv_stage_dv(const uint8_t* rdv, uint8_t* ob, int r, int qq, const float (&add)[16]) {
  const int rot = r & 7;
  const uint8_t* src = rdv + (qq >> 1) * 16384 + r * 128;
  float d[16];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float4 x = *reinterpret_cast<const float4*>(src + (((4 * (qq & 1) + c) ^ rot) << 4));
    d[4 * c] = x.x + add[4 * c];
    d[4 * c + 1] = x.y + add[4 * c + 1];
    d[4 * c + 2] = x.z + add[4 * c + 2];
    d[4 * c + 3] = x.w + add[4 * c + 3];
  }
#pragma unroll
  for (int j = 0; j < 2; ++j)
    *reinterpret_cast<uint4*>(ob + r * 128 + (((2 * qq + j) ^ rot) << 4)) =
        make_uint4(pack_bf16(d[8 * j], d[8 * j + 1]), pack_bf16(d[8 * j + 2], d[8 * j + 3]),
                   pack_bf16(d[8 * j + 4], d[8 * j + 5]), pack_bf16(d[8 * j + 6], d[8 * j + 7]));
}

__global__ void __launch_bounds__(512, 1) tc_bwd_kv_kernel(const __grid_constant__ CUtensorMap mapK,
                                                           const __grid_constant__ CUtensorMap mapV,
                                                           const __grid_constant__ CUtensorMap mapDK,
                                                           const __grid_constant__ CUtensorMap mapDV,
                                                           const __grid_constant__ CUtensorMap mapDVO,
                                                           TcBwdKVParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* RK = smem;            // 32 KB: K (bf16, then fp16)
  uint8_t* RV = smem + 32768;    // 16 KB: V (bf16, then fp16)
  uint8_t* RI = smem + 49152;    // 2 x 16 KB: dual images
  uint8_t* RDV = smem + 98304;   // 32 KB: the in-tile part of dv (fp32, two 32-column boxes)
  uint8_t* ROV = smem + 65536;   // 16 KB at the end: dv in bf16 (over the second image)
  __shared__ __align__(8) uint64_t bar_ld, bar_z, bar_e[2], bar_zf, bar_dv;
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
  if (nl == 0) {  // no level reads this tile's nodes: dv is the in-tile part, cast to bf16
    if (tid == 0) {
      ptx::mbar_init(&bar_dv, 1);
      ptx::fence_mbar_init();
      ptx::mbar_arrive_expect_tx(&bar_dv, 32768);
      ptx::tma_load_4d(RDV, &mapDV, &bar_dv, 0, h, (int)t0, b);
      ptx::tma_load_4d(RDV + 16384, &mapDV, &bar_dv, 32, h, (int)t0, b);
    }
    __syncthreads();
    bool ok = wait_bar(&bar_dv, 0);
    if (!ok) atomicExch(p.status, kStatusTimeout);
    if (ok) {
      float zero[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) zero[c] = 0.f;
      kv_stage_dv(RDV, ROV, r, qq, zero);
      ptx::fence_proxy_async_smem();
    }
    ok = __syncthreads_and(ok);
    if (ok && tid == 0) {
      ptx::tma_store_4d(&mapDVO, ROV, 0, h, (int)t0, b);
      ptx::bulk_commit_group();
      ptx::bulk_wait_read_all();  // the staging is read before the CTA ends
    }
    if (!ok && tid == 0) wait_bar(&bar_dv, 0);  // bounded: let the copy land before the CTA ends
    __syncthreads();
    return;
  }
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
    ptx::mbar_init(&bar_dv, 1);
    ptx::fence_mbar_init();
    // the in-tile part of dv (the in-tile kernel's store), read at the end
    ptx::mbar_arrive_expect_tx(&bar_dv, 32768);
    ptx::tma_load_4d(RDV, &mapDV, &bar_dv, 0, h, (int)t0, b);
    ptx::tma_load_4d(RDV + 16384, &mapDV, &bar_dv, 32, h, (int)t0, b);
    ptx::mbar_arrive_expect_tx(&bar_ld, 32768 + 16384);
    ptx::tma_load_4d(RK, &mapK, &bar_ld, 0, g, (int)t0, b);
    ptx::tma_load_4d(RK + 16384, &mapK, &bar_ld, 64, g, (int)t0, b);
    ptx::tma_load_4d(RV, &mapV, &bar_ld, 0, h, (int)t0, b);
    const int l2 = lin + p.pf_stride;  // one CTA per SM: the one most likely next on this SM
    if (p.pf_stride > 0 && l2 < (int)gridDim.x) {
      const int h2 = l2 % p.H, u2 = (l2 / p.H) % p.NT, b2 = l2 / (p.H * p.NT), g2 = h2 / p.hpg;
      tma_prefetch_4d(&mapK, 0, g2, u2 * kTile, b2);
      tma_prefetch_4d(&mapK, 64, g2, u2 * kTile, b2);
      tma_prefetch_4d(&mapV, 0, h2, u2 * kTile, b2);
    }
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
  const float rs = exp2f(gam - gt);
  if (ok) {
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
  // dk (columns 32 qq .. 32 qq + 31: box qq, from 0) is staged over K, V and the first
  // image, free once every level is read and V's dot is taken, and added into the per-head
  // buffer with TMA reductions.  dv (columns 16 qq .. 16 qq + 15) is final here: the
  // in-tile part plus this kernel's, in bf16, staged over the second image and stored
  // into the output.
  __syncthreads();
  bool okv = ok && wait_bar(&bar_dv, 0);
  if (ok && !okv) atomicExch(p.status, kStatusTimeout);
  ok = ok && okv;
  if (ok) {
    uint8_t* kb = smem + qq * 16384 + r * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<float4*>(kb + ((c ^ rot) << 4)) =
          make_float4(rs * ak[4 * c], rs * ak[4 * c + 1], rs * ak[4 * c + 2], rs * ak[4 * c + 3]);
    float add[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) add[c] = rs * av[c];
    kv_stage_dv(RDV, ROV, r, qq, add);
    ptx::fence_proxy_async_smem();
  }
  ok = __syncthreads_and(ok);
  if (ok && tid == 0) {
    for (int j = 0; j < 4; ++j) ptx::tma_reduce_add_4d(&mapDK, smem + j * 16384, 32 * j, h, (int)t0, b);
    ptx::tma_store_4d(&mapDVO, ROV, 0, h, (int)t0, b);
    ptx::bulk_commit_group();
    ptx::bulk_wait_read_all();  // the staging is read before the CTA ends
  }
  if (tid == 0) {  // bounded: let this CTA's copies and MMAs land before TMEM goes
    wait_bar(&bar_ld, 0);
    wait_bar(&bar_dv, 0);
    for (int j = consumed; j < issued; ++j) wait_bar(&bar_e[j & 1], (j >> 1) & 1);
    if (z_issued > 0) wait_bar(&bar_z, (z_issued - 1) & 1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tbase, 256);
}

}  // namespace

cudaError_t launch_tc_bwd_intra(const ll_shape& s, const void* q, const void* k, const void* v, const void* dO,
                                const float* a, const float* lam, float* dq32, float* dk32, float* dv32,
                                float* dlam, float* cu, unsigned* status, cudaStream_t st) {
  if (!tc_supported(s)) return cudaErrorInvalidValue;
  const int G = s.heads / s.heads_per_group, NT = s.T / kTile;
  CUtensorMap mQ, mK, mV, mD, mDQ, mDK, mDV;
  if (!make_map(&mQ, q, kDk, G, s.T, s.batch) || !make_map(&mK, k, kDk, G, s.T, s.batch) ||
      !make_map(&mV, v, kDv, s.heads, s.T, s.batch) || !make_map(&mD, dO, kDv, s.heads, s.T, s.batch) ||
      !make_map_f32(&mDQ, dq32, kDk, s.heads, s.T, s.batch) || !make_map_f32(&mDK, dk32, kDk, s.heads, s.T, s.batch) ||
      !make_map_f32(&mDV, dv32, kDv, s.heads, s.T, s.batch))
    return cudaErrorInvalidValue;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    nsm = 0;  // no prefetch
  const TcBwdParams p{s.batch, s.T, s.heads, s.heads_per_group, G, s.levels, NT, a, lam,
                      dq32, dk32, dv32, dlam, cu, status, nsm};
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBwd);
  if (e != cudaSuccess) return e;
  tc_bwd_intra_kernel<<<(unsigned)((size_t)s.batch * NT * s.heads), 256, kSmemBwd, st>>>(mQ, mK, mV, mD, mDQ, mDK,
                                                                                   mDV, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

cudaError_t launch_tc_bwd_q(const TcPlan& tp, const void* q, const void* dO, const float* a, const float* lam,
                            const char* tree_ws, float* dq32, float* dlam, float* dual, const int* dual_off,
                            int nslots, float* ru, uint8_t* dimg0, unsigned* dmeta0, unsigned* status,
                            cudaStream_t st) {
  CUtensorMap mQ, mD, mDQ;
  if (!make_map(&mQ, q, kDk, tp.G, tp.T, tp.B) || !make_map(&mD, dO, kDv, tp.H, tp.T, tp.B) ||
      !make_map_f32(&mDQ, dq32, kDk, tp.H, tp.T, tp.B))
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
  p.ru = ru;
  p.dimg = dimg0;
  p.dmeta = dmeta0;
  p.status = status;
  const int smem = bwdq_smem_bytes(bit_length(tp.NT - 1));
  cudaError_t e = cudaFuncSetAttribute(tc_bwd_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  tc_bwd_q_kernel<<<(unsigned)((size_t)tp.B * tp.NT * tp.H), 256, smem, st>>>(mQ, mD, mDQ, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

cudaError_t launch_tc_bwd_kv(const TcPlan& tp, const void* k, const void* v, const float* a, const char* tree_ws,
                             const float* dual, uint8_t* dimg, unsigned* dmeta, double* P, const int* dual_off,
                             int nslots, int n0, float* dk32, float* dv32, void* dv_out, float* cu,
                             unsigned* status, cudaStream_t st) {
  const unsigned BH = (unsigned)(tp.B * tp.H);
  tc_tile_prefix_kernel<<<BH, 256, 0, st>>>(reinterpret_cast<const unsigned*>(tree_ws + tp.off_meta), tp.nnodes,
                                            tp.NT, P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  note_launch();
  if (n0 < 0 || n0 >= nslots) return cudaErrorInvalidValue;
  tc_dual_publish_kernel<<<(unsigned)((size_t)BH * (nslots - n0)), 128, 0, st>>>(dual, dimg, dmeta, nslots, n0);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  CUtensorMap mK, mV, mDK, mDV, mDVO;
  if (!make_map(&mK, k, kDk, tp.G, tp.T, tp.B) || !make_map(&mV, v, kDv, tp.H, tp.T, tp.B) ||
      !make_map_f32(&mDK, dk32, kDk, tp.H, tp.T, tp.B) || !make_map_f32(&mDV, dv32, kDv, tp.H, tp.T, tp.B) ||
      !make_map(&mDVO, dv_out, kDv, tp.H, tp.T, tp.B))
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
  {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      p.pf_stride = nsm;  // otherwise 0: no prefetch
  }
  if ((e = cudaFuncSetAttribute(tc_bwd_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBwdKV)) !=
      cudaSuccess)
    return e;
  tc_bwd_kv_kernel<<<(unsigned)((size_t)tp.B * tp.NT * tp.H), 512, kSmemBwdKV, st>>>(mK, mV, mDK, mDV, mDVO, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

}  // namespace ll
