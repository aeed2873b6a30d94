// Shared pieces of the tensor-core (tcgen05 / TMEM / TMA) kernels: tile constants, the
// forward's node layout and parameters, bounded mbarrier waits, power-of-two scales,
// fp16 / bf16 packing, node publication, and the host's TMA tensor maps.  Included by
// tc_fwd.cu, tc_bwd.cu and tc_gdn.cu (each gets its own copy: internal linkage).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

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
  uint8_t* img;    // (B*H, nnodes, 16 KB) fp16 node images
  unsigned* meta;  // (B*H, nnodes, 4)
  unsigned* status;
  // comparators only (single-level and SSD output modes)
  float* o32;      // (B, T, H, d_v) fp32 running sum of the single-level passes
  int lsel;        // the one level of a single-level pass
  int lflags;      // bit 0: first pass (store), bit 1: last pass (write o)
  int all_tiles;   // tc_state stores every tile state's image (the SSD scan reads them all)
  uint8_t* pimg;   // (B*H, NT, 16 KB) SSD prefix-state images
  unsigned* pmeta; // (B*H, NT, 4)
  // continuation from the bucket memories at a start position T0 (level-fused mode only):
  // npre live levels of T0, their levels (lambda columns) and their fp16 images, whose
  // log2 decay is 0 (the memories are already decayed to T0 - 1)
  int npre;
  int prelev[32];
  uint8_t* preimg;   // (B*H, npre, 16 KB)
  unsigned* premeta; // (B*H, npre, 4)
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

// ---- host: TMA tensor maps ------------------------------------------------------
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

// 4-D fp32 map over (inner, count, T, B) with a (32, 1, 128, 1) box (128-byte rows),
// 128-byte swizzle: the per-head fp32 gradient rows of a 128-token tile, 32 columns a box.
bool make_map_f32(CUtensorMap* m, void* base, int inner, int count, int T, int B) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)count, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)inner * 4, (cuuint64_t)inner * 4 * count,
                           (cuuint64_t)inner * 4 * count * T};
  cuuint32_t box[4] = {32, 1, kTile, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

}  // namespace ll
