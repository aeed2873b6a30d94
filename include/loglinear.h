/*
 * loglinear.h — C ABI of the log-linear Mamba-2 forward and decode step
 * (sm_103a, one GPU).
 *
 * What is computed.  For every batch b, head h and query position t
 * (0-indexed), with group g = h / heads_per_group:
 *
 *     o[b,t,h,:] = sum_{s <= t} lambda[b,t,h, l(t,s)] * M^S(t,s) * (q[b,t,g,:] . k[b,s,g,:]) * v[b,s,h,:]
 *
 *   M^S(t,s) = a[b,s+1,h] * ... * a[b,t,h]   (Mamba-2 scalar-decay, 1-semiseparable mask;
 *              state-space-duality article http://biyoush.com/article/202409/463109.htm,
 *              section 狀態空間對偶性)
 *   l(t,s)   = 0 if s == t, else the bit length of (t xor s): the level of the Fenwick-tree
 *              bucket of t that holds s; buckets have power-of-two sizes and are finer near t
 *              (log-linear attention write-up https://www.yoousoft.com/industry/3746.html,
 *              section 特殊结构：树划分; the mask M^H(t,s) = lambda_t^{l(t,s)} and its
 *              composition with M^S, section 对Mamba-2和门控的对数线性推广).
 *
 * The forward uses the chunkwise algorithm of the write-up (section 高效训练算法):
 * dense masked products inside aligned chunks and a hierarchical state pass
 * across chunks.  The result does not depend on the chunk length; it is an exact
 * re-association of the sum above.
 *
 * Conventions shared by all entry points.
 *  - Every tensor is row-major and contiguous, and is owned by the caller.  Device
 *    pointers must be 16-byte aligned (LL_ERR_ALIGN otherwise).
 *  - q, k, v, o share ll_shape.dtype (fp32 or bf16); a, lambda and the states are fp32.
 *  - All work is enqueued on the caller's CUDA stream (`stream`, a cudaStream_t, may be
 *    NULL for the legacy default stream).  The library allocates no device memory, frees
 *    nothing and does not synchronise, except where a function says so.
 *  - Arguments are validated on the host before any launch; a failed check returns its
 *    code and enqueues nothing.  A launch error returns LL_ERR_CUDA.  Errors detected on
 *    the device (a bounded wait that ran out) are recorded in a device status word and
 *    reported by loglinear_check_status().  No C++ exception crosses this boundary.
 */
#ifndef LOGLINEAR_H
#define LOGLINEAR_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LL_OK = 0,
  LL_ERR_NULL = 1,          /* a required pointer is NULL */
  LL_ERR_SHAPE = 2,         /* sizes out of the supported range or inconsistent */
  LL_ERR_DTYPE = 3,         /* unsupported dtype */
  LL_ERR_ALIGN = 4,         /* a pointer is not 16-byte aligned */
  LL_ERR_WORKSPACE = 5,     /* workspace NULL or smaller than the query says */
  LL_ERR_CUDA = 6,          /* a CUDA runtime call or launch failed */
  LL_ERR_TIMEOUT = 7,       /* a bounded device-side wait ran out (see check_status) */
  LL_ERR_UNIMPLEMENTED = 8  /* valid request that this library does not implement */
} ll_status;

typedef enum { LL_F32 = 0, LL_BF16 = 1 } ll_dtype;

/*
 * Problem shape.
 *   batch            B >= 1
 *   T                sequence length, T >= 1 and T % chunk == 0 (forward); unused by decode
 *   heads            H >= 1, H % heads_per_group == 0
 *   heads_per_group  heads sharing one q/k group (MVA); G = H / heads_per_group groups
 *   d_k              16, 32, 64 or 128 (q/k width, the state's row count)
 *   d_v              16, 32 or 64 (v/o width, the state's column count)
 *   chunk            C in {16, 32, 64, 128}
 *   levels           L: lambda holds L weights per (b, t, h); forward needs
 *                    L >= bit_length(T-1) + 1 (every level a query below T can see);
 *                    decode uses L as the number of state slots too
 *   dtype            dtype of q, k, v and o
 */
typedef struct {
  int batch;
  int T;
  int heads;
  int heads_per_group;
  int d_k;
  int d_v;
  int chunk;
  int levels;
  ll_dtype dtype;
} ll_shape;

/* Bytes of device workspace loglinear_fwd needs for this shape (0 if the shape is
 * invalid).  The workspace holds per-chunk decays, chunk states and the Fenwick block
 * states of the inter-chunk pass (write-up section 高效训练算法). */
size_t loglinear_fwd_workspace_bytes(const ll_shape* shape);

/*
 * Forward over the whole sequence (write-up sections 高效训练算法 and
 * 对Mamba-2和门控的对数线性推广, Algorithm 1 / Fig. 3).
 *   q, k      (B, T, G, d_k)     dtype
 *   v         (B, T, H, d_v)     dtype
 *   a         (B, T, H)          fp32, each in (0, 1]; a <= 0 gives undefined results
 *   lambda    (B, T, H, L)       fp32
 *   o         (B, T, H, d_v)     dtype, written
 *   workspace device buffer of at least loglinear_fwd_workspace_bytes(shape) bytes,
 *             16-byte aligned; its contents on entry do not matter
 *   states_out        NULL, or (B, H, state_levels, d_k, d_v) fp32: the Fenwick bucket
 *                     states at position T, i.e. the memory a decode step at position T
 *                     starts from.  Level l holds sum over the level-l bucket of T of
 *                     M^S(T-1, s) k_s v_sᵀ.  Only the levels live at T (level l >= 1
 *                     with bit l-1 of T set) are written; the other slots hold
 *                     unspecified values, as the decode step allows.
 *   state_logscale_out NULL, or (B, H, state_levels) fp32, written as zeros (the decay
 *                     is folded into states_out).
 *   state_levels      slots in states_out; must be >= bit_length(T) + 1 when states_out
 *                     is given, ignored otherwise.
 * Which kernels run (loglinear_fwd_path reports it): bf16 with d_k = 128, d_v = 64 and
 * T % 64 == 0 takes the tensor-core path (tcgen05 products over 128-token tiles; when
 * T % 128 == 64 the last tile holds 64 tokens).  Every other accepted shape runs the fp32
 * CUDA-core path, which computes the same result several times more slowly.
 */
ll_status loglinear_fwd(const ll_shape* shape, const void* q, const void* k, const void* v,
                        const float* a, const float* lambda, void* o, void* workspace,
                        size_t workspace_bytes, float* states_out, float* state_logscale_out,
                        int state_levels, void* stream);

/*
 * One decode step at position `pos` for every (b, h) (write-up section 特殊结构：树划分:
 * O(log T) time and memory per decoded token).  shape->T is ignored;
 * shape->levels = L is the number of state slots and of lambda weights.
 *   q_t, k_t   (B, G, d_k)   dtype
 *   v_t        (B, H, d_v)   dtype
 *   a_t        (B, H)        fp32 in (0, 1]
 *   lambda_t   (B, H, L)     fp32
 *   o_t        (B, H, d_v)   dtype, written
 *   states     (B, H, L, d_k, d_v) fp32, read and updated in place
 *   state_logscale (B, H, L) fp32, read and updated in place
 * The bucket memory of level l is exp(state_logscale[l]) * states[l]; level l >= 1 is
 * live at position pos when bit l-1 of pos is set; slots of levels that are not live
 * hold unspecified values.  The step decays the live levels by a_t (in the log-scale),
 * forms o_t = lambda^0 (q.k) v + sum over live l of lambda^l q^T S^l, then merges the
 * token and the levels 1..m (m = trailing ones of pos) into level m+1 of pos+1.
 * Requires pos >= 0 and L >= bit_length(pos + 1) + 1.  A state exported by
 * loglinear_fwd at T continues with pos = T.
 */
ll_status loglinear_decode_step(const ll_shape* shape, long long pos, const void* q_t,
                                const void* k_t, const void* v_t, const float* a_t,
                                const float* lambda_t, void* o_t, float* states,
                                float* state_logscale, void* stream);

/*
 * End-to-end forward from HOST buffers: copies q, k, v, a, lambda (host, same layouts
 * as loglinear_fwd; pinned memory lets the copies run asynchronously) into
 * `device_arena`, runs loglinear_fwd and copies o back to the host buffer o_host.  The
 * batch is cut into up to 8 pieces of consecutive batch elements whose copies and
 * forwards overlap: inputs go in on a library stream, each piece's forward runs on
 * `stream`, outputs come back on a second library stream, and `stream` waits for the
 * last copy, so the call is complete once `stream` reaches that point.  The first call
 * on a device creates the two streams and their events (kept until exit).  The host
 * buffers must stay valid until then; the caller synchronises.  `device_arena` must hold
 * at least loglinear_fwd_host_arena_bytes(shape) bytes (16-byte aligned).
 * Calls from several host threads are safe: the library holds a per-device lock while a
 * call enqueues its work.  Their copies share the two library streams, so concurrent
 * calls' copies run one after another; each call needs its own arena and host buffers.
 */
size_t loglinear_fwd_host_arena_bytes(const ll_shape* shape);
ll_status loglinear_fwd_host(const ll_shape* shape, const void* q_host, const void* k_host,
                             const void* v_host, const float* a_host, const float* lambda_host,
                             void* o_host, void* device_arena, size_t arena_bytes, void* stream);

/*
 * Forward for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point; it exists for code that is not allowed to call
 * cudaMalloc or any other allocator while it runs (for example a plugin whose host owns
 * every device allocation, or code sharing the context with an allocator it must not
 * disturb), and for callers that cannot size or keep a workspace between calls.
 *
 * Same arguments and results as loglinear_fwd, without the workspace: the library uses
 * a fixed device array of LOGLINEAR_STATIC_WORKSPACE_BYTES (32 MiB) that each GPU loading
 * the library holds until the process exits.  The call allocates nothing and frees
 * nothing.
 *   - Shapes whose loglinear_fwd_workspace_bytes() exceeds LOGLINEAR_STATIC_WORKSPACE_BYTES
 *     are rejected with LL_ERR_WORKSPACE before anything is enqueued (for example
 *     B*H = 16 heads of T = 2048 at d_k = 128, d_v = 64 fit; the pages workload does not).
 *   - The first call on each device looks up the array's device address (with that
 *     device current); make that first call before any stream capture begins.
 *   - Every call on a device shares the one array and leaves its contents behind;
 *     nothing in it needs to start at zero, since every call writes each word before
 *     reading it.  Calls whose work
 *     overlaps on the GPU (other streams, other threads) race on the array: serialise
 *     them, e.g. on one stream.
 */
#define LOGLINEAR_STATIC_WORKSPACE_BYTES (32u << 20)
ll_status loglinear_fwd_static_workspace(const ll_shape* shape, const void* q, const void* k,
                                         const void* v, const float* a, const float* lambda,
                                         void* o, float* states_out, float* state_logscale_out,
                                         int state_levels, void* stream);

/* ---- sequence segments -------------------------------------------------------------------
 * A forward can start at a position T0 > 0 from the bucket memories there, and those
 * memories can be built from the memories of whole earlier segments.  This is what a
 * sequence split over several devices needs (each holds one segment of 2^p tokens; one
 * all-gather of the segments' memories and summed log-decays lets every segment form the
 * buckets of its start), and what a prefill in pieces needs.  Sources: the per-bucket
 * memories of the write-up (section 特殊结构：树划分, Fig. 2) and the combination of the
 * memories of pieces level by level (section 高效训练算法, Algorithm 1).
 *
 * Bucket memories use the decode step's format: (B, H, levels, d_k, d_v) fp32 blocks with
 * (B, H, levels) fp32 log-scales; the memory of level l is exp(logscale[l]) * block[l];
 * level l >= 1 is live at a position p when bit l-1 of p is set, and the block holds
 * sum over the bucket of M^S(p-1, s) k_s v_sᵀ.  Slots of levels that are not live hold
 * unspecified values and are neither read nor written.
 */

/* Bytes of workspace loglinear_fwd_continue needs (0: invalid shape or start). */
size_t loglinear_fwd_continue_workspace_bytes(const ll_shape* shape, long long T0);

/*
 * Forward over the tokens at positions T0 .. T0+T-1 (T = shape->T), given the bucket
 * memories at T0.  q, k, v, a, lambda and o hold the segment's T tokens, laid out as for
 * loglinear_fwd; lambda's levels are absolute (level l of every bucket, near or far), so
 * shape->levels must be >= bit_length(T0 + T - 1) + 1.
 *   T0               >= 0 and a multiple of the smallest power of two >= T (then every
 *                    bucket of a position in the segment lies either inside the segment
 *                    or before T0, where it is a bucket of T0); else LL_ERR_SHAPE
 *   prefix_states    (B, H, prefix_levels, d_k, d_v) fp32, the memories at T0 (read);
 *   prefix_logscale  (B, H, prefix_levels) fp32; both may be NULL when T0 == 0
 *   prefix_levels    >= bit_length(T0) + 1, <= 64
 *   states_out       NULL, or (B, H, state_levels, d_k, d_v): the memories at T0 + T
 *                    (written with zero log-scales into state_logscale_out if given), the
 *                    live levels only; may be the same buffer as prefix_states (then with
 *                    state_levels == prefix_levels, and state_logscale_out may be
 *                    prefix_logscale): a decode or a further continuation goes on from it
 *   state_levels     >= bit_length(T0 + T) + 1 when states_out is given
 *   workspace        >= loglinear_fwd_continue_workspace_bytes(shape, T0) bytes
 * With T0 == 0 this is loglinear_fwd.  The shapes of loglinear_fwd run on the same paths
 * (tensor cores for bf16, d_k = 128, d_v = 64, T % 64 == 0; the CUDA cores otherwise).
 */
ll_status loglinear_fwd_continue(const ll_shape* shape, long long T0, const void* q, const void* k,
                                 const void* v, const float* a, const float* lambda,
                                 const float* prefix_states, const float* prefix_logscale,
                                 int prefix_levels, void* o, void* workspace, size_t workspace_bytes,
                                 float* states_out, float* state_logscale_out, int state_levels,
                                 void* stream);

/* Bytes of workspace loglinear_segment_total needs (0: invalid shape; shape->levels is
 * ignored). */
size_t loglinear_segment_total_workspace_bytes(const ll_shape* shape);

/*
 * The memory of a whole segment of T tokens and the decay it applies to everything
 * before it:
 *   total_state     (B, H, d_k, d_v) fp32: sum over s < T of M^S(T-1, s) k_s v_sᵀ
 *   total_logdecay  (B, H) fp32: sum over t < T of ln a_t
 * k, v, a as for loglinear_fwd (no q or lambda).  shape->levels is ignored.
 */
ll_status loglinear_segment_total(const ll_shape* shape, const void* k, const void* v, const float* a,
                                  void* workspace, size_t workspace_bytes, float* total_state,
                                  float* total_logdecay, void* stream);

/*
 * The bucket memories at T0 = n_segments * T (T = shape->T, a power of two: every bucket
 * of T0 is then made of whole segments) from the memories of the n_segments segments
 * before it, as loglinear_segment_total returns them:
 *   seg_states     (n_segments, B, H, d_k, d_v) fp32, segment 0 first
 *   seg_logdecay   (n_segments, B, H) fp32
 *   states_out     (B, H, state_levels, d_k, d_v): the levels live at T0 are written;
 *   state_logscale_out NULL or (B, H, state_levels): zeros at those levels
 *   state_levels   >= bit_length(T0) + 1, <= 64
 * n_segments <= 64.  Uses shape->batch, heads, d_k, d_v and T.  Nothing is enqueued for
 * n_segments == 0 (position 0 has no buckets).
 */
ll_status loglinear_prefix_states(const ll_shape* shape, int n_segments, const float* seg_states,
                                  const float* seg_logdecay, float* states_out,
                                  float* state_logscale_out, int state_levels, void* stream);

/* ---- log-linear Gated DeltaNet -----------------------------------------------------------
 * The write-up extends Gated DeltaNet the same way (section 对Mamba-2和门控的对数线性推广):
 * the model's own transition, the gated delta rule
 *   S_t = a_t S_{t-1} (I - beta_t k_t k_tᵀ) + beta_t v_t k_tᵀ,
 * is kept and its attention mask is combined with the hierarchical one.  The delta rule
 * equals S_t = a_t S_{t-1} + u_t k_tᵀ with u_t = beta_t (v_t - a_t S_{t-1} k_t), so the
 * output is the masked form over u:
 *   o_t = sum_{s<=t} lambda_t^{l(t,s)} M^S(t,s) (q_t . k_s) u_s.
 */

/* Bytes of device workspace loglinear_gdn_fwd needs (0: invalid shape). */
size_t loglinear_gdn_fwd_workspace_bytes(const ll_shape* shape);

/*
 * Log-linear Gated DeltaNet forward.  Arguments as for loglinear_fwd, plus
 *   beta  (B, T, H)  fp32, the delta-rule write strength (in [0, 1] for a stable rule)
 * Keys are used as given; the model normalises them (the delta rule is stable for
 * beta |k|^2 <= 2).  u is computed chunk by chunk in the delta rule's WY form: the
 * chunks' local solves run in parallel, then one CTA per (b, h) carries the state across
 * the chunks in order.  For bf16 with d_k = 128, d_v = 64 and T % 128 == 0 the chunks
 * are 128 tokens and the products run on the tensor cores (fp16 high and low parts,
 * fp32 accumulation); otherwise 32-token chunks run in fp32 on the CUDA cores.  u is
 * stored in the input dtype in the workspace, then the level-fused forward runs on
 * (q, k, u, a, lambda).  On the tensor-core path with batch >= 2 the last batch element's
 * state pass and forward run on a second, high-priority stream that the library creates
 * on a device's first such call, forked from and joined back into `stream` with events,
 * so that the other elements' forward starts as soon as their passes end; every launch
 * is still ordered after the work already on `stream`, and later work on `stream` waits
 * for all of it.  Concurrent calls on one device are serialised inside the library.
 */
ll_status loglinear_gdn_fwd(const ll_shape* shape, const void* q, const void* k, const void* v,
                            const float* a, const float* beta, const float* lambda, void* o,
                            void* workspace, size_t workspace_bytes, void* stream);

/* ---- backward -------------------------------------------------------------------------
 * The pages give no backward; this is the chain rule on the forward's masked form
 * o_t = sum_{s<=t} lambda_t^{l(t,s)} M^S(t,s) (q_t . k_s) v_s (write-up sections
 * 特殊结构：树划分 and 对Mamba-2和门控的对数线性推广), laid out by the same chunks and
 * Fenwick blocks as the forward (section 高效训练算法, Algorithm 1).
 */

/* Bytes of device workspace loglinear_bwd needs for this shape (0: invalid shape). */
size_t loglinear_bwd_workspace_bytes(const ll_shape* shape);

/*
 * Gradients of the scalar sum(dO * o) where o = loglinear_fwd(q, k, v, a, lambda), for
 * every shape loglinear_fwd accepts.  Inputs as for loglinear_fwd, plus
 *   dO       (B, T, H, d_v)  dtype
 * and the outputs, all written (no accumulation into them):
 *   dq, dk   (B, T, G, d_k)  dtype; the heads of a group add up
 *   dv       (B, T, H, d_v)  dtype
 *   dlog_a   (B, T, H)       fp32, the gradient with respect to log a, the form in which
 *                            a enters the forward; the gradient with respect to a is
 *                            dlog_a / a (badly conditioned for a near 0, hence not
 *                            returned); 0 at t = 0, whose decay multiplies nothing
 *   dlambda  (B, T, H, L)    fp32; levels with no bucket get 0
 *   workspace >= loglinear_bwd_workspace_bytes(shape) bytes, 16-byte aligned, contents on
 *            entry do not matter
 * For bf16 with d_k = 128, d_v = 64, T % 128 == 0 and chunk >= 64 the products run on the
 * tensor cores (fp16 operands with power-of-two scales, fp32 accumulation); other shapes
 * run fp32 on the CUDA cores.  The terms of the levels above a tile (or chunk) are summed
 * through each node's dual with fp32 atomics, so results can differ between calls by
 * rounding.
 */
ll_status loglinear_bwd(const ll_shape* shape, const void* q, const void* k, const void* v,
                        const float* a, const float* lambda, const void* dO, void* dq, void* dk,
                        void* dv, float* dlog_a, float* dlambda, void* workspace,
                        size_t workspace_bytes, void* stream);

/* ---- comparators ---------------------------------------------------------------------
 * Two other ways to compute on the tensor-core shape (bf16, d_k = 128, d_v = 64,
 * T % 128 == 0), kept to measure the level-fused forward against.  Any other shape
 * returns LL_ERR_UNIMPLEMENTED.  Same layouts, alignment and stream rules as
 * loglinear_fwd; outputs written, workspace contents on entry do not matter.
 */

/* Bytes of workspace loglinear_fwd_naive needs (0: invalid or unsupported shape). */
size_t loglinear_fwd_naive_workspace_bytes(const ll_shape* shape);

/*
 * The same output as loglinear_fwd, computed without level fusion: after the tile
 * states and the Fenwick tree, one output pass per level (the intra-tile levels 0..7,
 * then each inter-tile level), each re-reading its inputs and adding its level's term
 * to an fp32 sum in the workspace.  This mirrors the write-up's naive variant, which
 * re-runs an existing Mamba-2 computation once per level (section
 * 对Mamba-2和门控的对数线性推广, Fig. 4).
 */
ll_status loglinear_fwd_naive(const ll_shape* shape, const void* q, const void* k, const void* v,
                              const float* a, const float* lambda, void* o, void* workspace,
                              size_t workspace_bytes, void* stream);

/* Bytes of workspace ssd_fwd needs (0: invalid or unsupported shape). */
size_t ssd_fwd_workspace_bytes(const ll_shape* shape);

/*
 * The lambda-constant special case, i.e. Mamba-2's SSD (state-space-duality article,
 * section 狀態空間對偶性): o_t = sum over s <= t of M^S(t, s) (q_t . k_s) v_s.  It runs
 * the Mamba-2 structure: chunk states, a sequential state pass over tiles, then one
 * chunk output pass with a single prefix state per tile.  Same as loglinear_fwd with
 * lambda = 1 everywhere, up to rounding.  shape->levels is ignored.
 */
ll_status ssd_fwd(const ll_shape* shape, const void* q, const void* k, const void* v,
                  const float* a, void* o, void* workspace, size_t workspace_bytes, void* stream);

/* ---- diagnostics -------------------------------------------------------------------- */

/* Same as loglinear_fwd, and records CUDA events on `stream` around its kernels:
 * events[0] before the first kernel and events[i + 1] right after kernel i, for as many
 * as n_events allows (events are cudaEvent_t handles created by the caller).  The kernel
 * order is the one loglinear_fwd_kernel_names() lists. */
ll_status loglinear_fwd_profiled(const ll_shape* shape, const void* q, const void* k,
                                 const void* v, const float* a, const float* lambda, void* o,
                                 void* workspace, size_t workspace_bytes, float* states_out,
                                 float* state_logscale_out, int state_levels, void* stream,
                                 void** events, int n_events);

/* Comma-separated names of the kernels loglinear_fwd launches for this shape, in launch
 * order (with_export != 0: states_out is given).  Empty string for an invalid shape. */
const char* loglinear_fwd_kernel_names(const ll_shape* shape, int with_export);

/* Number of kernels this library has launched in this process so far (all devices). */
unsigned long long loglinear_launch_count(void);

/* Synchronises `stream`, then reads and clears the device status word of the current
 * device.  Returns LL_OK, LL_ERR_TIMEOUT when a bounded device-side wait ran out since
 * the last check (the launch returned early; its outputs are undefined), or
 * LL_ERR_CUDA when the synchronisation itself failed. */
ll_status loglinear_check_status(void* stream);

/* Self-test of the bounded-wait path: launches one block that waits on a barrier that
 * nothing completes, giving up after about `spins` polls, which records LL_ERR_TIMEOUT
 * in the status word.  Faults nothing; the context stays usable. */
ll_status loglinear_selftest_wait_timeout(long long spins, void* stream);

/* Static description of a status code. */
const char* loglinear_status_string(ll_status status);

/* Which kernels loglinear_fwd would launch for this shape: 0 = invalid shape,
 * 1 = generic CUDA-core path, 2 = tensor-core (tcgen05) path. */
int loglinear_fwd_path(const ll_shape* shape);

#ifdef __cplusplus
}
#endif

#endif /* LOGLINEAR_H */
