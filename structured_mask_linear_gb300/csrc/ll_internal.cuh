// Internal declarations shared by the CUDA translation units of the library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/loglinear.h"

namespace ll {

// Device status word values (mirror ll_status).
constexpr unsigned kStatusTimeout = LL_ERR_TIMEOUT;

// Chunk / block bookkeeping for the generic path.
struct GenPlan {
  int B, T, H, hpg, G, dk, dv, C, clog, L, N;  // N = T / C chunks
  int M;                                       // chunk levels: bit_length(N)
  int nblk;                                    // Fenwick block states per (b, h)
  int blk_off[32];                             // first block of chunk level m
  size_t off_g, off_gamma, off_H, off_blk, off_blkG, bytes;
  // continuation from the bucket memories at a start position (0 prefix levels otherwise):
  // level prelev[i] of pre_st (B*H, Lp, dk, dv) with log-scale pre_lsc (B*H, Lp)
  int npre;
  int prelev[32];
  int Lp;
  const float* pre_st;
  const float* pre_lsc;
};

bool make_gen_plan(const ll_shape& s, GenPlan* p);

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* a;
  const float* lam;
  void* o;
  char* ws;
  float* states_out;
  float* logscale_out;
  int state_levels;
  unsigned* status;
  void** events;  // optional: events[0] before the first kernel, events[i+1] after kernel i
  int n_events;
  // continuation (loglinear_fwd_continue): the tokens are the positions T0 .. T0+T-1 and
  // the terms of the bucket memories at T0 are added: pre_st (B*H, pre_levels, dk, dv)
  // fp32 with log-scales pre_lsc (B*H, pre_levels); pre_ws holds the tensor-core path's
  // fp16 images of them (tc_prefix_bytes).
  long long T0;
  const float* pre_st;
  const float* pre_lsc;
  int pre_levels;
  char* pre_ws;
};

// Counts a kernel launch and records the profiling event that follows kernel `i`.
void note_launch(const FwdArgs& a, int i, cudaStream_t st);
void note_launch();


cudaError_t launch_generic_fwd(const GenPlan& p, bool bf16, const FwdArgs& a, cudaStream_t st);
// Only the chunk states and Fenwick blocks of the generic forward (for the backward).
cudaError_t launch_generic_states(const GenPlan& p, bool bf16, const FwdArgs& a, cudaStream_t st);

// Gated DeltaNet's transformed values on the tensor cores (128-token chunks) for
// tc_supported shapes: workspace bytes and the launch (u: (B, T, H, d_v) bf16).
size_t tc_gdn_bytes(const ll_shape& s);
cudaError_t launch_tc_gdn(const ll_shape& s, const void* k, const void* v, const float* a, const float* beta,
                          void* u, char* ws, unsigned* status, cudaStream_t st);
// Gated DeltaNet's transformed values (csrc/gdn.cu): buffer bytes and the launch.
size_t gdn_values_bytes(const ll_shape& s);
cudaError_t launch_gdn_values(const ll_shape& s, const void* k, const void* v, const float* a,
                              const float* beta, void* u, unsigned* status, cudaStream_t st);

// Backward (csrc/backward.cu): workspace bytes (0: unsupported) and the launches.
size_t bwd_workspace_bytes(const ll_shape& s);
cudaError_t launch_bwd(const ll_shape& s, const void* q, const void* k, const void* v, const float* a,
                       const float* lam, const void* dO, void* dq, void* dk, void* dv, float* dloga,
                       float* dlam, char* ws, unsigned* status, cudaStream_t st);

struct DecodeArgs {
  int B, H, hpg, G, dk, dv, L;
  long long pos;
  const void* q;
  const void* k;
  const void* v;
  const float* a;
  const float* lam;
  void* o;
  float* states;
  float* logscale;
};

cudaError_t launch_decode(const DecodeArgs& d, bool bf16, cudaStream_t st);

cudaError_t launch_wait_selftest(unsigned* status, long long spins, cudaStream_t st);

// Sequence segments (csrc/segments.cu).
cudaError_t launch_seg_logdecay(const float* a, int B, int T, int H, float* out, cudaStream_t st);
cudaError_t launch_sum_live_levels(const float* stl, int BH, int SL, long long T, int S, float* total,
                                   cudaStream_t st);
cudaError_t launch_prefix_from_segments(int r, int seg_log, int BH, const float* seg_st, const float* seg_g,
                                        int S, float* stl, float* lsc, int SL, cudaStream_t st);
cudaError_t launch_continue_export(long long T0, long long T, int BH, const float* pst, const float* plsc, int Lp,
                                   const float* loc, int SLloc, const float* segg, int S, float* stl, float* lsc,
                                   int SL, cudaStream_t st);
// Generic path: chunk states, Fenwick blocks and the export at position T only.
cudaError_t launch_generic_export_only(const GenPlan& p, bool bf16, const FwdArgs& a, cudaStream_t st);

// ---- tensor-core path (tcgen05) --------------------------------------------
struct TcPlan {
  int B, T, H, hpg, G, L;
  int NT;           // 128-token tiles
  int nnodes;       // Fenwick tree nodes per (b, h)
  int node_off[32]; // first node of tile level m
  int MT;           // tile levels (bit_length(NT))
  size_t off_img;   // fp16 node images, 16 KB each
  size_t off_meta;  // per node: spare, scale exponent, log2 decay, spare
  size_t meta_bytes, bytes;
};

// bf16, d_k = 128, d_v = 64, T % 128 == 0: every tensor-core kernel (backward, Gated
// DeltaNet, comparators); the forward also takes T % 128 == 64 (a last tile of 64 tokens).
bool tc_supported(const ll_shape& s);
bool tc_fwd_supported(const ll_shape& s);
bool make_tc_plan(const ll_shape& s, TcPlan* p);
bool make_tc_fwd_plan(const ll_shape& s, TcPlan* p);
cudaError_t launch_tc_fwd(const TcPlan& p, const FwdArgs& a, cudaStream_t st);
// Comparators on the tensor-core shape (not the product path): the forward with one
// output pass per level (no level fusion), and the lambda-constant special case (SSD).
size_t tc_naive_bytes(const TcPlan& p);
cudaError_t launch_tc_naive(const TcPlan& p, const FwdArgs& a, cudaStream_t st);
size_t tc_ssd_bytes(const TcPlan& p);
cudaError_t launch_tc_ssd(const TcPlan& p, const FwdArgs& a, cudaStream_t st);
const char* tc_kernel_names(bool with_export);
// The forward's tree only (tile states, levels above), into a.ws laid out per p.
cudaError_t launch_tc_nodes(const TcPlan& p, const FwdArgs& a, cudaStream_t st);
// The tree and the export of the memories at position T into a.states_out (no output).
cudaError_t launch_tc_export_only(const TcPlan& p, const FwdArgs& a, cudaStream_t st);
// Bytes of the fp16 images of npre prefix memories per (b, h) (continuation).
size_t tc_prefix_bytes(const TcPlan& p, int npre);
// Backward, query side of the inter-tile levels on the tensor cores: adds into dq32,
// assigns dlambda levels >= 8 of the set bits, adds the nodes' duals (dual slot of the
// even node (m, i): dual_off[m] + i / 2, nslots per (b, h); dual zero before the first call,
// except the tile nodes' (m = 0), which their one reader tile stores), and adds
// sum_m lambda_t^(8+m) dlambda_t^(8+m) into ru (B, T, H) of the tiles it runs.  With dimg0
// and dmeta0 given, the tile nodes' duals go straight to their fp16 images and scale
// exponents there (the layout tc_dual_publish writes) instead of to dual.
cudaError_t launch_tc_bwd_q(const TcPlan& p, const void* q, const void* dO, const float* a, const float* lam,
                            const char* tree_ws, float* dq32, float* dlam, float* dual, const int* dual_off,
                            int nslots, float* ru, uint8_t* dimg0, unsigned* dmeta0, unsigned* status,
                            cudaStream_t st);
// Backward, key side of the inter-tile levels on the tensor cores: the tile-decay running
// sums (fp64, (B*H, NT+1) in P), the duals of slots n0.. of each (b, h) as fp16 images
// (dimg: 16 KB per slot, dmeta: 4 u32 per slot; slots below n0 are published by
// launch_tc_bwd_q), then adds into dk32, writes dv_out (bf16, (B, T, H, d_v)) as dv32 (the
// in-tile part) plus its own part, and adds v_s . (its part of dv_s) into cu.
cudaError_t launch_tc_bwd_kv(const TcPlan& p, const void* k, const void* v, const float* a, const char* tree_ws,
                             const float* dual, uint8_t* dimg, unsigned* dmeta, double* P, const int* dual_off,
                             int nslots, int n0, float* dk32, float* dv32, void* dv_out, float* cu,
                             unsigned* status, cudaStream_t st);
// Backward: the in-tile pairs (levels 0..7) on the tensor cores, for tc_supported shapes;
// assigns the fp32 per-head dq, dk, dv buffers, dlambda (levels >= 8 zeroed) and cu, the
// column sums C_s of the in-tile pair terms, followed in the same buffer by R_t = sum over
// levels 0..7 of lambda_t^l dlambda_t^l (both (B, T, H) fp32).
cudaError_t launch_tc_bwd_intra(const ll_shape& s, const void* q, const void* k, const void* v, const void* dO,
                                const float* a, const float* lam, float* dq32, float* dk32, float* dv32,
                                float* dlam, float* cu, unsigned* status, cudaStream_t st);

__host__ __device__ inline int bit_length(long long x) {
  int l = 0;
  while (x > 0) {
    l++;
    x >>= 1;
  }
  return l;
}

}  // namespace ll

// ---- small device helpers -----------------------------------------------------
// Shared-memory product on the CUDA cores, one 4 x 4 output tile per thread and step:
// for every tile (m0, n0) of an M x N output (M, N multiples of 4) handed out to the
// nthr threads in turn, acc[i][j] = sum_{k < K} A(m0+i, k) B(k, n0+j) with
// A(m, k) = a[m*sam + k*sak] and B(k, n) = b[k*sbk + n] (b rows 16-byte aligned), then
// epi(m0, n0, acc).  Threads of a warp share m0 where N/4 >= 32 (A is a broadcast) and
// read consecutive float4s of B.  Where A's k (sak == 1) or m (sam == 1) index is
// contiguous and 16-byte aligned, A is read four values per load.  smem_mm_r takes the
// k range of each tile from range(m0, n0, kb, ke) (multiples of 4; outside it the
// products are known to be zero, e.g. above a causal diagonal).
template <typename Range, typename Epi>
__device__ __forceinline__ void smem_mm_r(int M, int N, int K, const float* a, int sam, int sak,
                                          const float* b, int sbk, int tid, int nthr, Range range, Epi epi) {
  const int tn_count = N >> 2;
  const int tiles = (M >> 2) * tn_count;
  const bool a16 = (reinterpret_cast<uintptr_t>(a) & 15u) == 0;
  const bool krow = a16 && sak == 1 && (sam & 3) == 0 && (K & 3) == 0;  // A rows along k
  const bool mcol = a16 && !krow && sam == 1 && (sak & 3) == 0;         // A columns along m
  for (int tile = tid; tile < tiles; tile += nthr) {
    const int m0 = (tile / tn_count) << 2, n0 = (tile % tn_count) << 2;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    const float* ap = a + (size_t)m0 * sam;
    const float* bp = b + n0;
    int kb = 0, ke = K;
    range(m0, n0, kb, ke);
    if (krow) {
#pragma unroll 2
      for (int k = kb; k < ke; k += 4) {
        float ar[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 x = *reinterpret_cast<const float4*>(ap + i * sam + k);
          ar[i][0] = x.x;
          ar[i][1] = x.y;
          ar[i][2] = x.z;
          ar[i][3] = x.w;
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float4 bv = *reinterpret_cast<const float4*>(bp + (size_t)(k + kk) * sbk);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[i][0] += ar[i][kk] * bv.x;
            acc[i][1] += ar[i][kk] * bv.y;
            acc[i][2] += ar[i][kk] * bv.z;
            acc[i][3] += ar[i][kk] * bv.w;
          }
        }
      }
    } else if (mcol) {
#pragma unroll 4
      for (int k = kb; k < ke; ++k) {
        const float4 x = *reinterpret_cast<const float4*>(ap + (size_t)k * sak);
        const float4 bv = *reinterpret_cast<const float4*>(bp + (size_t)k * sbk);
        const float av[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i][0] += av[i] * bv.x;
          acc[i][1] += av[i] * bv.y;
          acc[i][2] += av[i] * bv.z;
          acc[i][3] += av[i] * bv.w;
        }
      }
    } else {
#pragma unroll 4
      for (int k = kb; k < ke; ++k) {
        const float4 bv = *reinterpret_cast<const float4*>(bp + (size_t)k * sbk);
        float av[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = ap[i * sam + k * sak];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i][0] += av[i] * bv.x;
          acc[i][1] += av[i] * bv.y;
          acc[i][2] += av[i] * bv.z;
          acc[i][3] += av[i] * bv.w;
        }
      }
    }
    epi(m0, n0, acc);
  }
}
template <typename Epi>
__device__ __forceinline__ void smem_mm(int M, int N, int K, const float* a, int sam, int sak,
                                        const float* b, int sbk, int tid, int nthr, Epi epi) {
  smem_mm_r(M, N, K, a, sam, sak, b, sbk, tid, nthr, [](int, int, int&, int&) {}, epi);
}

__device__ __forceinline__ float ll_load(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ll_load(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void ll_store(float* p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void ll_store(__nv_bfloat16* p, size_t i, float x) {
  p[i] = __float2bfloat16_rn(x);
}
