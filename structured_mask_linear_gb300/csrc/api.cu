// C ABI of the log-linear Mamba-2 library: argument validation, workspace sizing,
// dispatch to the kernels, device status word.  Declarations and contracts are in
// include/loglinear.h.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "ll_internal.cuh"

namespace {

std::atomic<unsigned long long> g_launches{0};

__device__ unsigned g_ll_status;  // device-side error word (0 = ok)

std::mutex g_mu;
unsigned* g_status_addr[128];  // per-device address of g_ll_status

unsigned* status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ll_status) != cudaSuccess) return nullptr;
    g_status_addr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

ll_status check_common(const ll_shape* s) {
  if (!s) return LL_ERR_NULL;
  if (s->dtype != LL_F32 && s->dtype != LL_BF16) return LL_ERR_DTYPE;
  if (s->batch < 1 || s->heads < 1 || s->heads_per_group < 1) return LL_ERR_SHAPE;
  if (s->heads % s->heads_per_group) return LL_ERR_SHAPE;
  if (!pow2_in(s->d_k, 16, 128) || !pow2_in(s->d_v, 16, 64)) return LL_ERR_SHAPE;
  if ((long long)s->batch * s->heads > 65535) return LL_ERR_SHAPE;
  return LL_OK;
}

ll_status check_fwd_shape(const ll_shape* s) {
  ll_status st = check_common(s);
  if (st != LL_OK) return st;
  if (s->T < 1 || !pow2_in(s->chunk, 16, 128) || s->T % s->chunk) return LL_ERR_SHAPE;
  if (s->levels < ll::bit_length(s->T - 1) + 1 || s->levels > 32) return LL_ERR_SHAPE;
  return LL_OK;
}

size_t esize(const ll_shape* s) { return s->dtype == LL_BF16 ? 2 : 4; }

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

// The SSD comparator takes no lambda; its plan uses the smallest valid level count.
bool ssd_shape(const ll_shape* s, ll_shape* out) {
  if (!s) return false;
  *out = *s;
  if (out->T >= 1) out->levels = ll::bit_length(out->T - 1) + 1;
  return true;
}

ll_status fwd_impl(const ll_shape* s, const void* q, const void* k, const void* v, const float* a,
                   const float* lambda, void* o, void* workspace, size_t workspace_bytes,
                   float* states_out, float* state_logscale_out, int state_levels, void* stream,
                   void** events, int n_events);

}  // namespace

namespace ll {
// tc_gdn.cu: the Gated DeltaNet values' chunk solves and the state pass over batch
// elements b0 .. b0 + nb - 1
cudaError_t launch_tc_gdn_local(const ll_shape& s, const void* k, const void* v, const float* a, const float* beta,
                                void* u, char* ws, unsigned* status, cudaStream_t st);
cudaError_t launch_tc_gdn_pass(const ll_shape& s, int b0, int nb, const void* k, const void* v, const float* a,
                               const float* beta, void* u, char* ws, unsigned* status, cudaStream_t st);
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
void note_launch(const FwdArgs& a, int i, cudaStream_t st) {
  note_launch();
  if (a.events && i + 1 < a.n_events && a.events[i + 1])
    cudaEventRecord(static_cast<cudaEvent_t>(a.events[i + 1]), st);
}
}  // namespace ll

extern "C" {

const char* loglinear_status_string(ll_status s) {
  switch (s) {
    case LL_OK: return "ok";
    case LL_ERR_NULL: return "required pointer is NULL";
    case LL_ERR_SHAPE: return "unsupported or inconsistent shape";
    case LL_ERR_DTYPE: return "unsupported dtype";
    case LL_ERR_ALIGN: return "pointer not 16-byte aligned";
    case LL_ERR_WORKSPACE: return "workspace missing or too small";
    case LL_ERR_CUDA: return "CUDA runtime error";
    case LL_ERR_TIMEOUT: return "bounded device wait ran out";
    case LL_ERR_UNIMPLEMENTED: return "not implemented for this shape";
  }
  return "unknown status";
}

int loglinear_fwd_path(const ll_shape* s) {
  if (check_fwd_shape(s) != LL_OK) return 0;
  return ll::tc_fwd_supported(*s) ? 2 : 1;
}

size_t loglinear_fwd_workspace_bytes(const ll_shape* s) {
  if (check_fwd_shape(s) != LL_OK) return 0;
  if (ll::tc_fwd_supported(*s)) {
    ll::TcPlan tp;
    return ll::make_tc_fwd_plan(*s, &tp) ? tp.bytes : 0;
  }
  ll::GenPlan p;
  if (!ll::make_gen_plan(*s, &p)) return 0;
  return p.bytes;
}

ll_status loglinear_fwd(const ll_shape* s, const void* q, const void* k, const void* v,
                        const float* a, const float* lambda, void* o, void* workspace,
                        size_t workspace_bytes, float* states_out, float* state_logscale_out,
                        int state_levels, void* stream) {
  return fwd_impl(s, q, k, v, a, lambda, o, workspace, workspace_bytes, states_out,
                  state_logscale_out, state_levels, stream, nullptr, 0);
}

ll_status loglinear_fwd_profiled(const ll_shape* s, const void* q, const void* k, const void* v,
                                 const float* a, const float* lambda, void* o, void* workspace,
                                 size_t workspace_bytes, float* states_out,
                                 float* state_logscale_out, int state_levels, void* stream,
                                 void** events, int n_events) {
  return fwd_impl(s, q, k, v, a, lambda, o, workspace, workspace_bytes, states_out,
                  state_logscale_out, state_levels, stream, events, n_events);
}

const char* loglinear_fwd_kernel_names(const ll_shape* s, int with_export) {
  if (check_fwd_shape(s) != LL_OK) return "";
  if (ll::tc_fwd_supported(*s)) return ll::tc_kernel_names(with_export != 0);
  return with_export ? "gen_chunk_state,gen_blocks,gen_output,gen_export"
                     : "gen_chunk_state,gen_blocks,gen_output";
}

unsigned long long loglinear_launch_count(void) {
  return g_launches.load(std::memory_order_relaxed);
}

ll_status loglinear_decode_step(const ll_shape* s, long long pos, const void* q_t, const void* k_t,
                                const void* v_t, const float* a_t, const float* lambda_t,
                                void* o_t, float* states, float* state_logscale, void* stream) {
  ll_status st = check_common(s);
  if (st != LL_OK) return st;
  if (pos < 0 || pos >= (1LL << 62)) return LL_ERR_SHAPE;
  if (s->levels < ll::bit_length(pos + 1) + 1 || s->levels > 64) return LL_ERR_SHAPE;
  if (!q_t || !k_t || !v_t || !a_t || !lambda_t || !o_t || !states || !state_logscale)
    return LL_ERR_NULL;
  if (!aligned16(q_t) || !aligned16(k_t) || !aligned16(v_t) || !aligned16(o_t) ||
      !aligned16(states))
    return LL_ERR_ALIGN;
  ll::DecodeArgs d{s->batch, s->heads, s->heads_per_group, s->heads / s->heads_per_group,
                   s->d_k, s->d_v, s->levels, pos, q_t, k_t, v_t, a_t, lambda_t, o_t,
                   states, state_logscale};
  cudaError_t e = ll::launch_decode(d, s->dtype == LL_BF16, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

size_t loglinear_fwd_host_arena_bytes(const ll_shape* s) {
  if (check_fwd_shape(s) != LL_OK) return 0;
  const size_t B = s->batch, T = s->T, H = s->heads, G = s->heads / s->heads_per_group;
  const size_t es = esize(s);
  size_t n = 0;
  n += 2 * a256(B * T * G * s->d_k * es);   // q, k
  n += 2 * a256(B * T * H * s->d_v * es);   // v, o
  n += a256(B * T * H * 4);                 // a
  n += a256(B * T * H * s->levels * 4);     // lambda
  n += a256(loglinear_fwd_workspace_bytes(s));
  return n;
}

}  // extern "C"

namespace {

// Streams and events of the pipelined host forward, created once per device.
constexpr int kHostPieces = 8;
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t ein[kHostPieces] = {}, eout[kHostPieces] = {};
  bool ready = false;
  // Held for the whole enqueue of one call: the events are re-recorded by every call, so
  // a second thread must not record them between this call's record and its wait.
  std::mutex call_mu;
};
std::mutex g_pipe_mu;
HostPipe g_pipe[128];

HostPipe* host_pipe() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.start, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.done, ef) != cudaSuccess)
      return nullptr;
    for (int i = 0; i < kHostPieces; ++i)
      if (cudaEventCreateWithFlags(&hp.ein[i], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&hp.eout[i], ef) != cudaSuccess)
        return nullptr;
    hp.ready = true;
  }
  return &hp;
}

// Streams and events of the Gated DeltaNet forward's split (created once per device): two
// streams of the highest priority, so that the passes and the last element's forward take
// SMs ahead of the other elements' forward on the caller's stream.
struct GdnPipe {
  cudaStream_t first = nullptr, last = nullptr;
  cudaEvent_t local = nullptr, first_done = nullptr, last_done = nullptr;
  bool ready = false;
  std::mutex call_mu;  // the events are re-recorded by every call
};
GdnPipe g_gdn_pipe[128];

GdnPipe* gdn_pipe() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  GdnPipe& gp = g_gdn_pipe[dev];
  if (!gp.ready) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithPriority(&gp.first, cudaStreamNonBlocking, greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&gp.last, cudaStreamNonBlocking, greatest) != cudaSuccess ||
        cudaEventCreateWithFlags(&gp.local, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&gp.first_done, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&gp.last_done, ef) != cudaSuccess)
      return nullptr;
    gp.ready = true;
  }
  return &gp;
}

}  // namespace

extern "C" {

ll_status loglinear_fwd_host(const ll_shape* s, const void* q_host, const void* k_host,
                             const void* v_host, const float* a_host, const float* lambda_host,
                             void* o_host, void* device_arena, size_t arena_bytes, void* stream) {
  ll_status st = check_fwd_shape(s);
  if (st != LL_OK) return st;
  if (!q_host || !k_host || !v_host || !a_host || !lambda_host || !o_host) return LL_ERR_NULL;
  const size_t need = loglinear_fwd_host_arena_bytes(s);
  if (!device_arena || arena_bytes < need) return LL_ERR_WORKSPACE;
  if (!aligned16(device_arena)) return LL_ERR_ALIGN;
  const size_t B = s->batch, T = s->T, H = s->heads, G = s->heads / s->heads_per_group;
  const size_t es = esize(s);
  const size_t bq = B * T * G * s->d_k * es, bv = B * T * H * s->d_v * es, ba = B * T * H * 4,
               bl = B * T * H * s->levels * 4;
  char* p = static_cast<char*>(device_arena);
  char* dq = p; p += a256(bq);
  char* dk = p; p += a256(bq);
  char* dv = p; p += a256(bv);
  char* dout = p; p += a256(bv);
  char* da = p; p += a256(ba);
  char* dl = p; p += a256(bl);
  char* dws = p;
  const size_t wsb = loglinear_fwd_workspace_bytes(s);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  HostPipe* hp = host_pipe();
  if (!hp) return LL_ERR_CUDA;
  std::lock_guard<std::mutex> call_lock(hp->call_mu);
  // Pipeline over pieces of the batch (consecutive batch elements; every tensor is
  // batch-major, so a piece is one contiguous slice of each): the input copies of piece
  // i + 1 run on hp->in while piece i computes on `stream` and piece i - 1's output
  // copies back on hp->out.  `stream` waits for the last output copy at the end.
  const int np = (int)(B < (size_t)kHostPieces ? B : (size_t)kHostPieces);
  const size_t pq = bq / B, pv = bv / B, pa = ba / B, pl = bl / B;  // bytes per batch element
  if (cudaEventRecord(hp->start, cs) != cudaSuccess || cudaStreamWaitEvent(hp->in, hp->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->out, hp->start, 0) != cudaSuccess)
    return LL_ERR_CUDA;
  for (int i = 0; i < np; ++i) {
    const size_t b0 = B * i / np, nb = B * (i + 1) / np - b0;
    const char* qh = static_cast<const char*>(q_host);
    const char* kh = static_cast<const char*>(k_host);
    const char* vh = static_cast<const char*>(v_host);
    const char* ah = reinterpret_cast<const char*>(a_host);
    const char* lh = reinterpret_cast<const char*>(lambda_host);
    if (cudaMemcpyAsync(dq + b0 * pq, qh + b0 * pq, nb * pq, cudaMemcpyHostToDevice, hp->in) != cudaSuccess ||
        cudaMemcpyAsync(dk + b0 * pq, kh + b0 * pq, nb * pq, cudaMemcpyHostToDevice, hp->in) != cudaSuccess ||
        cudaMemcpyAsync(dv + b0 * pv, vh + b0 * pv, nb * pv, cudaMemcpyHostToDevice, hp->in) != cudaSuccess ||
        cudaMemcpyAsync(da + b0 * pa, ah + b0 * pa, nb * pa, cudaMemcpyHostToDevice, hp->in) != cudaSuccess ||
        cudaMemcpyAsync(dl + b0 * pl, lh + b0 * pl, nb * pl, cudaMemcpyHostToDevice, hp->in) != cudaSuccess ||
        cudaEventRecord(hp->ein[i], hp->in) != cudaSuccess || cudaStreamWaitEvent(cs, hp->ein[i], 0) != cudaSuccess)
      return LL_ERR_CUDA;
    ll_shape sp = *s;
    sp.batch = (int)nb;
    st = loglinear_fwd(&sp, dq + b0 * pq, dk + b0 * pq, dv + b0 * pv, reinterpret_cast<float*>(da + b0 * pa),
                       reinterpret_cast<float*>(dl + b0 * pl), dout + b0 * pv, dws, wsb, nullptr, nullptr, 0,
                       stream);
    if (st != LL_OK) return st;
    if (cudaEventRecord(hp->eout[i], cs) != cudaSuccess || cudaStreamWaitEvent(hp->out, hp->eout[i], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<char*>(o_host) + b0 * pv, dout + b0 * pv, nb * pv, cudaMemcpyDeviceToHost,
                        hp->out) != cudaSuccess)
      return LL_ERR_CUDA;
  }
  if (cudaEventRecord(hp->done, hp->out) != cudaSuccess || cudaStreamWaitEvent(cs, hp->done, 0) != cudaSuccess)
    return LL_ERR_CUDA;
  return LL_OK;
}

size_t loglinear_fwd_naive_workspace_bytes(const ll_shape* s) {
  if (check_fwd_shape(s) != LL_OK || !ll::tc_supported(*s)) return 0;
  ll::TcPlan tp;
  return ll::make_tc_plan(*s, &tp) ? ll::tc_naive_bytes(tp) : 0;
}

ll_status loglinear_fwd_naive(const ll_shape* s, const void* q, const void* k, const void* v,
                              const float* a, const float* lambda, void* o, void* workspace,
                              size_t workspace_bytes, void* stream) {
  ll_status st = check_fwd_shape(s);
  if (st != LL_OK) return st;
  if (!ll::tc_supported(*s)) return LL_ERR_UNIMPLEMENTED;
  if (!q || !k || !v || !a || !lambda || !o) return LL_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(a) || !aligned16(lambda) ||
      !aligned16(o) || !aligned16(workspace))
    return LL_ERR_ALIGN;
  ll::TcPlan tp;
  if (!ll::make_tc_plan(*s, &tp)) return LL_ERR_SHAPE;
  if (!workspace || workspace_bytes < ll::tc_naive_bytes(tp)) return LL_ERR_WORKSPACE;
  unsigned* sw = status_word();
  if (!sw) return LL_ERR_CUDA;
  ll::FwdArgs fa{q, k, v, a, lambda, o, static_cast<char*>(workspace), nullptr, nullptr, 0, sw,
                 nullptr, 0};
  return ll::launch_tc_naive(tp, fa, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LL_OK
                                                                                       : LL_ERR_CUDA;
}

size_t ssd_fwd_workspace_bytes(const ll_shape* s) {
  ll_shape t;
  if (!ssd_shape(s, &t) || check_fwd_shape(&t) != LL_OK || !ll::tc_supported(t)) return 0;
  ll::TcPlan tp;
  return ll::make_tc_plan(t, &tp) ? ll::tc_ssd_bytes(tp) : 0;
}

ll_status ssd_fwd(const ll_shape* s, const void* q, const void* k, const void* v, const float* a,
                  void* o, void* workspace, size_t workspace_bytes, void* stream) {
  ll_shape t;
  if (!ssd_shape(s, &t)) return LL_ERR_NULL;
  ll_status st = check_fwd_shape(&t);
  if (st != LL_OK) return st;
  if (!ll::tc_supported(t)) return LL_ERR_UNIMPLEMENTED;
  if (!q || !k || !v || !a || !o) return LL_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(a) || !aligned16(o) ||
      !aligned16(workspace))
    return LL_ERR_ALIGN;
  ll::TcPlan tp;
  if (!ll::make_tc_plan(t, &tp)) return LL_ERR_SHAPE;
  if (!workspace || workspace_bytes < ll::tc_ssd_bytes(tp)) return LL_ERR_WORKSPACE;
  unsigned* sw = status_word();
  if (!sw) return LL_ERR_CUDA;
  ll::FwdArgs fa{q, k, v, a, nullptr, o, static_cast<char*>(workspace), nullptr, nullptr, 0, sw,
                 nullptr, 0};
  return ll::launch_tc_ssd(tp, fa, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

// Gated DeltaNet on the tensor-core shape with more than one batch element: the state pass
// of the last element and its forward run on a second stream, so that the forward of the
// others starts as soon as their passes end (the pass takes one CTA per (b, h) for all
// its chunks; at B * H above the SM count the last element's CTAs would otherwise run as a
// second wave alone).  Its forward has a workspace of its own.
bool gdn_split(const ll_shape* s) { return s->batch >= 2 && ll::tc_supported(*s); }
size_t gdn_fwd_ws_last(const ll_shape* s) {
  ll_shape s1 = *s;
  s1.batch = 1;
  return a256(loglinear_fwd_workspace_bytes(&s1));
}

size_t loglinear_gdn_fwd_workspace_bytes(const ll_shape* s) {
  const size_t f = loglinear_fwd_workspace_bytes(s);
  if (!f) return 0;
  return a256(f) + (gdn_split(s) ? gdn_fwd_ws_last(s) : 0) + ll::gdn_values_bytes(*s);
}

ll_status loglinear_gdn_fwd(const ll_shape* s, const void* q, const void* k, const void* v,
                            const float* a, const float* beta, const float* lambda, void* o,
                            void* workspace, size_t workspace_bytes, void* stream) {
  ll_status st = check_fwd_shape(s);
  if (st != LL_OK) return st;
  if (!beta) return LL_ERR_NULL;
  if (!aligned16(beta)) return LL_ERR_ALIGN;
  const size_t need = loglinear_gdn_fwd_workspace_bytes(s);
  if (!workspace || workspace_bytes < need) return LL_ERR_WORKSPACE;
  if (!q || !k || !v || !a || !lambda || !o) return LL_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(a) || !aligned16(lambda) ||
      !aligned16(o) || !aligned16(workspace))
    return LL_ERR_ALIGN;
  // u (the transformed values) after the forward's own workspace(s)
  const size_t fws = a256(loglinear_fwd_workspace_bytes(s));
  const bool split = gdn_split(s);
  const size_t fws1 = split ? gdn_fwd_ws_last(s) : 0;
  char* u = static_cast<char*>(workspace) + fws + fws1;
  unsigned* sw = status_word();
  if (!sw) return LL_ERR_CUDA;
  if (!split) {
    if (ll::launch_gdn_values(*s, k, v, a, beta, u, sw, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return LL_ERR_CUDA;
    return fwd_impl(s, q, k, u, a, lambda, o, workspace, fws, nullptr, nullptr, 0, stream, nullptr, 0);
  }
  const int B = s->batch;
  const size_t ub = ((size_t)s->batch * s->T * s->heads * s->d_v * 2 + 255) & ~size_t(255);  // bf16 u
  char* rec = u + ub;  // the chunk records (tc_gdn.cu)
  GdnPipe* gp = gdn_pipe();
  if (!gp) return LL_ERR_CUDA;
  std::lock_guard<std::mutex> call_lock(gp->call_mu);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (ll::launch_tc_gdn_local(*s, k, v, a, beta, u, rec, sw, cs) != cudaSuccess) return LL_ERR_CUDA;
  if (cudaEventRecord(gp->local, cs) != cudaSuccess || cudaStreamWaitEvent(gp->first, gp->local, 0) != cudaSuccess ||
      cudaStreamWaitEvent(gp->last, gp->local, 0) != cudaSuccess)
    return LL_ERR_CUDA;
  // the passes of elements 0 .. B-2 are issued first, so that their CTAs start first
  if (ll::launch_tc_gdn_pass(*s, 0, B - 1, k, v, a, beta, u, rec, sw, gp->first) != cudaSuccess ||
      cudaEventRecord(gp->first_done, gp->first) != cudaSuccess ||
      ll::launch_tc_gdn_pass(*s, B - 1, 1, k, v, a, beta, u, rec, sw, gp->last) != cudaSuccess)
    return LL_ERR_CUDA;
  // the forward of the last element on its stream (pointers of element B - 1)
  const size_t G = (size_t)(s->heads / s->heads_per_group), es = 2;
  const size_t pq = (size_t)s->T * G * s->d_k * es, pv = (size_t)s->T * s->heads * s->d_v * es,
               pa = (size_t)s->T * s->heads, pl = (size_t)s->T * s->heads * s->levels;
  ll_shape s1 = *s;
  s1.batch = 1;
  const size_t bl = (size_t)(B - 1);
  ll_status st1 = fwd_impl(&s1, static_cast<const char*>(q) + bl * pq, static_cast<const char*>(k) + bl * pq,
                           u + bl * pv, a + bl * pa, lambda + bl * pl, static_cast<char*>(o) + bl * pv,
                           static_cast<char*>(workspace) + fws, fws1, nullptr, nullptr, 0, gp->last, nullptr, 0);
  if (st1 != LL_OK) return st1;
  if (cudaEventRecord(gp->last_done, gp->last) != cudaSuccess) return LL_ERR_CUDA;
  // the forward of elements 0 .. B-2 on the caller's stream, once their passes are done
  if (cudaStreamWaitEvent(cs, gp->first_done, 0) != cudaSuccess) return LL_ERR_CUDA;
  ll_shape s0 = *s;
  s0.batch = B - 1;
  ll_status st0 = fwd_impl(&s0, q, k, u, a, lambda, o, workspace, fws, nullptr, nullptr, 0, stream, nullptr, 0);
  if (st0 != LL_OK) return st0;
  return cudaStreamWaitEvent(cs, gp->last_done, 0) == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

size_t loglinear_bwd_workspace_bytes(const ll_shape* s) {
  if (check_fwd_shape(s) != LL_OK) return 0;
  return ll::bwd_workspace_bytes(*s);
}

ll_status loglinear_bwd(const ll_shape* s, const void* q, const void* k, const void* v,
                        const float* a, const float* lambda, const void* dO, void* dq, void* dk,
                        void* dv, float* dlog_a, float* dlambda, void* workspace,
                        size_t workspace_bytes, void* stream) {
  ll_status st = check_fwd_shape(s);
  if (st != LL_OK) return st;
  if (!q || !k || !v || !a || !lambda || !dO || !dq || !dk || !dv || !dlog_a || !dlambda)
    return LL_ERR_NULL;
  const void* ptrs[] = {q, k, v, a, lambda, dO, dq, dk, dv, dlog_a, dlambda, workspace};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return LL_ERR_ALIGN;
  const size_t need = ll::bwd_workspace_bytes(*s);
  if (need == 0) return LL_ERR_SHAPE;
  if (!workspace || workspace_bytes < need) return LL_ERR_WORKSPACE;
  unsigned* sw = status_word();
  if (!sw) return LL_ERR_CUDA;
  cudaError_t e = ll::launch_bwd(*s, q, k, v, a, lambda, dO, dq, dk, dv, dlog_a, dlambda,
                                 static_cast<char*>(workspace), sw, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // extern "C"

// ---- sequence segments -----------------------------------------------------------------

namespace {

// Layout of a continuation's workspace after the forward's own: the tensor-core path's
// images of the prefix memories, the segment's export at its end, its summed ln-decay.
struct ContLayout {
  size_t fwd, pre, loc, segg, bytes;
  int npre, SLloc;
};

bool cont_layout(const ll_shape* s, long long T0, ContLayout* c) {
  const size_t f = loglinear_fwd_workspace_bytes(s);
  if (!f) return false;
  const size_t BH = (size_t)s->batch * s->heads, S = (size_t)s->d_k * s->d_v;
  c->npre = __builtin_popcountll((unsigned long long)(T0 > 0 ? T0 : 0));
  c->SLloc = ll::bit_length(s->T) + 1;
  size_t o = a256(f);
  c->fwd = 0;
  c->pre = o;
  if (ll::tc_fwd_supported(*s)) {
    ll::TcPlan tp;
    if (!ll::make_tc_fwd_plan(*s, &tp)) return false;
    o += a256(ll::tc_prefix_bytes(tp, c->npre));
  }
  c->loc = o;
  o += a256(BH * c->SLloc * S * sizeof(float));
  c->segg = o;
  o += a256(BH * sizeof(float));
  c->bytes = o;
  return true;
}

// T0 is a multiple of the smallest power of two >= T: then every bucket of a position
// in [T0, T0 + T) lies either before T0 (a bucket of T0) or inside the segment.
bool aligned_start(long long T0, int T) {
  const long long p2 = 1LL << ll::bit_length((long long)T - 1);
  return T0 >= 0 && T0 % p2 == 0;
}

ll_status check_continue(const ll_shape* s, long long T0) {
  ll_status st = check_fwd_shape(s);
  if (st != LL_OK) return st;
  if (T0 < 0 || T0 > (1LL << 40) || !aligned_start(T0, s->T)) return LL_ERR_SHAPE;
  if (s->levels < ll::bit_length(T0 + s->T - 1) + 1) return LL_ERR_SHAPE;
  return LL_OK;
}

// A shape for the kernels that read no lambda: the smallest valid level count.
ll_shape no_lambda(const ll_shape* s) {
  ll_shape t = *s;
  if (t.T >= 1) t.levels = ll::bit_length(t.T - 1) + 1;
  return t;
}

}  // namespace

extern "C" {

size_t loglinear_fwd_continue_workspace_bytes(const ll_shape* s, long long T0) {
  ContLayout c;
  if (check_continue(s, T0) != LL_OK || !cont_layout(s, T0, &c)) return 0;
  return c.bytes;
}

ll_status loglinear_fwd_continue(const ll_shape* s, long long T0, const void* q, const void* k,
                                 const void* v, const float* a, const float* lambda,
                                 const float* prefix_states, const float* prefix_logscale,
                                 int prefix_levels, void* o, void* workspace, size_t workspace_bytes,
                                 float* states_out, float* state_logscale_out, int state_levels,
                                 void* stream) {
  ll_status st = check_continue(s, T0);
  if (st != LL_OK) return st;
  if (!q || !k || !v || !a || !lambda || !o) return LL_ERR_NULL;
  if (T0 > 0) {
    if (!prefix_states || !prefix_logscale) return LL_ERR_NULL;
    if (prefix_levels < ll::bit_length(T0) + 1 || prefix_levels > 64) return LL_ERR_SHAPE;
    if (!aligned16(prefix_states)) return LL_ERR_ALIGN;
  }
  if (states_out) {
    if (state_levels < ll::bit_length(T0 + s->T) + 1 || state_levels > 64) return LL_ERR_SHAPE;
    if (!aligned16(states_out)) return LL_ERR_ALIGN;
    if (T0 > 0 && (const void*)states_out == (const void*)prefix_states && state_levels != prefix_levels)
      return LL_ERR_SHAPE;  // in place only with one layout
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(a) || !aligned16(lambda) ||
      !aligned16(o))
    return LL_ERR_ALIGN;
  ContLayout c;
  if (!cont_layout(s, T0, &c)) return LL_ERR_SHAPE;
  if (!workspace || workspace_bytes < c.bytes) return LL_ERR_WORKSPACE;
  if (!aligned16(workspace)) return LL_ERR_ALIGN;
  if (T0 == 0)
    return fwd_impl(s, q, k, v, a, lambda, o, workspace, workspace_bytes, states_out, state_logscale_out,
                    state_levels, stream, nullptr, 0);
  unsigned* sw = status_word();
  if (!sw) return LL_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  float* loc = reinterpret_cast<float*>(ws + c.loc);
  float* segg = reinterpret_cast<float*>(ws + c.segg);
  ll::FwdArgs fa{q, k, v, a, lambda, o, ws, states_out ? loc : nullptr, nullptr, c.SLloc, sw, nullptr, 0};
  fa.T0 = T0;
  fa.pre_st = prefix_states;
  fa.pre_lsc = prefix_logscale;
  fa.pre_levels = prefix_levels;
  fa.pre_ws = ws + c.pre;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (ll::tc_fwd_supported(*s)) {
    ll::TcPlan tp;
    if (!ll::make_tc_fwd_plan(*s, &tp)) return LL_ERR_SHAPE;
    e = ll::launch_tc_fwd(tp, fa, cs);
  } else {
    ll::GenPlan p;
    if (!ll::make_gen_plan(*s, &p)) return LL_ERR_SHAPE;
    e = ll::launch_generic_fwd(p, s->dtype == LL_BF16, fa, cs);
  }
  if (e != cudaSuccess) return LL_ERR_CUDA;
  if (states_out) {
    const int BH = s->batch * s->heads, S = s->d_k * s->d_v;
    if (ll::launch_seg_logdecay(a, s->batch, s->T, s->heads, segg, cs) != cudaSuccess ||
        ll::launch_continue_export(T0, s->T, BH, prefix_states, prefix_logscale, prefix_levels, loc, c.SLloc,
                                   segg, S, states_out, state_logscale_out, state_levels, cs) != cudaSuccess)
      return LL_ERR_CUDA;
  }
  return LL_OK;
}

size_t loglinear_segment_total_workspace_bytes(const ll_shape* s) {
  if (!s) return 0;
  const ll_shape t = no_lambda(s);
  ContLayout c;
  if (check_fwd_shape(&t) != LL_OK || !cont_layout(&t, 0, &c)) return 0;
  return c.bytes;
}

ll_status loglinear_segment_total(const ll_shape* s, const void* k, const void* v, const float* a,
                                  void* workspace, size_t workspace_bytes, float* total_state,
                                  float* total_logdecay, void* stream) {
  if (!s) return LL_ERR_NULL;
  const ll_shape t = no_lambda(s);
  ll_status st = check_fwd_shape(&t);
  if (st != LL_OK) return st;
  if (!k || !v || !a || !total_state || !total_logdecay) return LL_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(a) || !aligned16(total_state)) return LL_ERR_ALIGN;
  ContLayout c;
  if (!cont_layout(&t, 0, &c)) return LL_ERR_SHAPE;
  if (!workspace || workspace_bytes < c.bytes) return LL_ERR_WORKSPACE;
  if (!aligned16(workspace)) return LL_ERR_ALIGN;
  unsigned* sw = status_word();
  if (!sw) return LL_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  float* loc = reinterpret_cast<float*>(ws + c.loc);
  // the export needs no q, lambda or o; k stands in for q where a tensor map is built
  ll::FwdArgs fa{k, k, v, a, nullptr, nullptr, ws, loc, nullptr, c.SLloc, sw, nullptr, 0};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (ll::tc_fwd_supported(t)) {
    ll::TcPlan tp;
    if (!ll::make_tc_fwd_plan(t, &tp)) return LL_ERR_SHAPE;
    e = ll::launch_tc_export_only(tp, fa, cs);
  } else {
    ll::GenPlan p;
    if (!ll::make_gen_plan(t, &p)) return LL_ERR_SHAPE;
    e = ll::launch_generic_export_only(p, t.dtype == LL_BF16, fa, cs);
  }
  const int BH = t.batch * t.heads, S = t.d_k * t.d_v;
  if (e != cudaSuccess || ll::launch_sum_live_levels(loc, BH, c.SLloc, t.T, S, total_state, cs) != cudaSuccess ||
      ll::launch_seg_logdecay(a, t.batch, t.T, t.heads, total_logdecay, cs) != cudaSuccess)
    return LL_ERR_CUDA;
  return LL_OK;
}

ll_status loglinear_prefix_states(const ll_shape* s, int n_segments, const float* seg_states,
                                  const float* seg_logdecay, float* states_out,
                                  float* state_logscale_out, int state_levels, void* stream) {
  if (!s) return LL_ERR_NULL;
  ll_status st = check_common(s);
  if (st != LL_OK) return st;
  if (s->T < 1 || (s->T & (s->T - 1)) || n_segments < 0 || n_segments > 64) return LL_ERR_SHAPE;
  const long long T0 = (long long)n_segments * s->T;
  if (state_levels < ll::bit_length(T0) + 1 || state_levels > 64) return LL_ERR_SHAPE;
  if (n_segments == 0) return LL_OK;
  if (!seg_states || !seg_logdecay || !states_out) return LL_ERR_NULL;
  if (!aligned16(seg_states) || !aligned16(states_out)) return LL_ERR_ALIGN;
  const int BH = s->batch * s->heads, S = s->d_k * s->d_v;
  const int seg_log = ll::bit_length(s->T) - 1;
  return ll::launch_prefix_from_segments(n_segments, seg_log, BH, seg_states, seg_logdecay, S, states_out,
                                         state_logscale_out, state_levels,
                                         static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? LL_OK
             : LL_ERR_CUDA;
}

ll_status loglinear_check_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LL_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_ll_status, sizeof(v)) != cudaSuccess) return LL_ERR_CUDA;
  if (v != 0 && cudaMemcpyToSymbol(g_ll_status, &zero, sizeof(zero)) != cudaSuccess)
    return LL_ERR_CUDA;
  if (v == 0) return LL_OK;
  return v == LL_ERR_TIMEOUT ? LL_ERR_TIMEOUT : LL_ERR_CUDA;
}

ll_status loglinear_selftest_wait_timeout(long long spins, void* stream) {
  if (spins < 0) return LL_ERR_SHAPE;
  unsigned* sw = status_word();
  if (!sw) return LL_ERR_CUDA;
  cudaError_t e = ll::launch_wait_selftest(sw, spins, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // extern "C"

namespace {

ll_status fwd_impl(const ll_shape* s, const void* q, const void* k, const void* v, const float* a,
                   const float* lambda, void* o, void* workspace, size_t workspace_bytes,
                   float* states_out, float* state_logscale_out, int state_levels, void* stream,
                   void** events, int n_events) {
  ll_status st = check_fwd_shape(s);
  if (st != LL_OK) return st;
  if (!q || !k || !v || !a || !lambda || !o) return LL_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(a) || !aligned16(lambda) ||
      !aligned16(o))
    return LL_ERR_ALIGN;
  if (states_out) {
    if (state_levels < ll::bit_length(s->T) + 1 || state_levels > 64) return LL_ERR_SHAPE;
    if (!aligned16(states_out)) return LL_ERR_ALIGN;
  }
  const size_t need = loglinear_fwd_workspace_bytes(s);
  if (!workspace || workspace_bytes < need) return LL_ERR_WORKSPACE;
  if (!aligned16(workspace)) return LL_ERR_ALIGN;
  unsigned* sw = status_word();
  if (!sw) return LL_ERR_CUDA;
  ll::FwdArgs fa{q, k, v, a, lambda, o, static_cast<char*>(workspace), states_out,
                 state_logscale_out, state_levels, sw, events, n_events};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (events && n_events > 0 && events[0])
    cudaEventRecord(static_cast<cudaEvent_t>(events[0]), cs);
  cudaError_t e;
  if (ll::tc_fwd_supported(*s)) {
    ll::TcPlan tp;
    if (!ll::make_tc_fwd_plan(*s, &tp)) return LL_ERR_SHAPE;
    e = ll::launch_tc_fwd(tp, fa, cs);
  } else {
    ll::GenPlan p;
    if (!ll::make_gen_plan(*s, &p)) return LL_ERR_SHAPE;
    e = ll::launch_generic_fwd(p, s->dtype == LL_BF16, fa, cs);
  }
  return e == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // namespace
