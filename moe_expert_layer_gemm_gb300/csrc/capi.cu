// C ABI of the MoE layer library: argument checks, workspace carving, the order of the
// stages, launch accounting, tracing and the device error word.  The arithmetic of every stage
// runs in the kernels of route.cu, rowops.cu, gemm_tc.cu (bf16) and gemm_simt.cu (fp32).
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "moe_gb300.h"

namespace moe {

// ------------------------------------------------------------------ error text
static thread_local char g_errbuf[512];

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_errbuf, sizeof(g_errbuf), fmt, ap);
  va_end(ap);
}

static int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_errbuf, sizeof(g_errbuf), fmt, ap);
  va_end(ap);
  return code;
}

// ------------------------------------------------------------------ device error word
__device__ int g_device_error;

static std::mutex g_dev_mu;
static int g_sms[64];

static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  return dev;
}

// Unique id of the calling thread's current context, 0 if there is none (or it was destroyed).
// The driver's cuCtxGetCurrent / cuCtxGetId are reached through the runtime's entry-point query,
// as the tensor-map encoder is: the library does not link libcuda.
static unsigned long long current_ctx_id() {
  typedef int (*GetCurrentFn)(void**);
  typedef int (*GetIdFn)(void*, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 0;
  return id;
}

int symbol_address(const void* symbol, SymbolCache* cache, void** out, const char* what) {
  const int dev = current_device();
  if (dev < 0) {
    set_error("%s: no usable current device", what);
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  const unsigned long long id = current_ctx_id();
  if (!cache->ptr[dev] || id == 0 || cache->ctx[dev] != id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, symbol);
    if (e != cudaSuccess || !p) {
      set_error("%s: cudaGetSymbolAddress failed on device %d: %s", what, dev,
                cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
    cache->ptr[dev] = p;
    cache->ctx[dev] = current_ctx_id();   // the lookup made the primary context current
  }
  *out = cache->ptr[dev];
  return MOE_OK;
}

static SymbolCache g_err_sym;

int* device_error_word() {
  void* p = nullptr;
  if (symbol_address(&g_device_error, &g_err_sym, &p, "device error word") != MOE_OK) return nullptr;
  return static_cast<int*>(p);
}

int num_sms() {
  const int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return g_sms[dev];
}

// ------------------------------------------------------------------ side stream
// "Megatron-Bridge 深度剖析", §Shared Expert Overlap: the shared expert's computation overlaps
// the routed path instead of following it.  The second stream and its fork/join events are the
// caller's (moe_side_stream); the library holds no stream, event or switch of its own.
struct SideStream {
  cudaStream_t s;
  cudaEvent_t fork, join;
};

static int check_side(const moe_side_stream* side, void* stream) {
  if (!side) return MOE_OK;
  if (!side->stream || !side->fork || !side->join)
    return fail(MOE_ERR_INVALID_ARG, "side: stream, fork and join must all be given");
  if (side->stream == stream)
    return fail(MOE_ERR_INVALID_ARG, "side.stream must differ from the call's stream");
  if (side->fork == side->join)
    return fail(MOE_ERR_INVALID_ARG, "side.fork and side.join must be different events");
  return MOE_OK;
}

static SideStream side_of(const moe_side_stream* side) {
  SideStream ss;
  ss.s = static_cast<cudaStream_t>(side->stream);
  ss.fork = static_cast<cudaEvent_t>(side->fork);
  ss.join = static_cast<cudaEvent_t>(side->join);
  return ss;
}

// ------------------------------------------------------------------ launch accounting, tracing
static std::atomic<uint64_t> g_launches{0};
static std::atomic<int> g_trace_on{0};

struct TraceRec {
  const char* name;
  cudaEvent_t start, stop;
};
static std::mutex g_trace_mu;
static std::vector<TraceRec> g_trace;
static std::vector<cudaEvent_t> g_event_pool;
static thread_local cudaEvent_t t_pending_start = nullptr;

static cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void trace_before(const char*, cudaStream_t s) {
  if (!g_trace_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  t_pending_start = take_event();
  if (t_pending_start) cudaEventRecord(t_pending_start, s);
}

void trace_after(const char* name, cudaStream_t s) {
  if (!g_trace_on.load(std::memory_order_relaxed) || !t_pending_start) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  cudaEvent_t stop = take_event();
  if (stop) {
    cudaEventRecord(stop, s);
    g_trace.push_back({name, t_pending_start, stop});
  }
  t_pending_start = nullptr;
}

// ------------------------------------------------------------------ workspace carving
struct Carve {
  uint8_t* base;
  size_t off = 0;
  explicit Carve(void* b) : base(static_cast<uint8_t*>(b)) {}
  void* take(size_t bytes) {
    off = (off + 255) & ~static_cast<size_t>(255);
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

static size_t esize(const moe_cfg* c) { return c->dtype == MOE_DTYPE_BF16 ? 2 : 4; }
static int64_t Nrows(const moe_cfg* c) { return static_cast<int64_t>(c->T) * c->k; }
static int ext_cols(const moe_cfg* c) { return ((c->E + (c->shared_gate ? 1 : 0)) + 63) / 64 * 64; }

static int router_splits(const moe_cfg* c) {
  const int mr = c->E + (c->shared_gate ? 1 : 0);
  const int tiles = ((mr + 127) / 128) * ((c->d + 255) / 256);
  int s = (num_sms() + tiles - 1) / tiles;
  const int cap_t = c->T / 256 > 1 ? c->T / 256 : 1;
  if (s > cap_t) s = cap_t;
  if (s > 64) s = 64;
  if (s < 1) s = 1;
  return s;
}

struct RouteWs {
  uint8_t* hist;     // expert histogram [route_rows(T)][route_ldh(E)] bytes
  int32_t* rowpre;   // its per-row prefixes [E][route_rows(T)]: large histograms only, else null
  float* logits;
  float* aux;        // balancing-loss partial sums [route_blocks(T)][E]
};
static RouteWs carve_route(Carve& cv, const moe_cfg* c) {
  RouteWs w;
  w.hist = static_cast<uint8_t*>(cv.take(static_cast<size_t>(route_hist_bytes(c->T, c->E))));
  w.rowpre = nullptr;
  if (!route_hist_direct(c->T, c->E))
    w.rowpre = static_cast<int32_t*>(cv.take(static_cast<size_t>(route_rows(c->T)) * c->E * 4));
  w.logits = static_cast<float*>(cv.take(static_cast<size_t>(c->T) * c->E * 4));
  w.aux = static_cast<float*>(cv.take(static_cast<size_t>(route_blocks(c->T)) * c->E * 4));
  return w;
}

// Scratch of the MXFP8 weight gradients: the four operands quantised along the tokens (codes in
// their [N, C] layouts, scales in the token-chunk layout) and the chunk bases of the experts.
struct WgMxWs {
  int32_t* cbase;
  uint8_t *x_q, *dy_q, *h_q, *dH1_q;
  uint8_t *x_s, *dy_s, *h_s, *dH1_s;
  int* sched;   // two 16-byte tile counters
};
static WgMxWs carve_wgmx(Carve& cv, const moe_cfg* c) {
  WgMxWs w;
  const int64_t N = static_cast<int64_t>(c->T) * c->k;
  const int E = c->E, d = c->d, f = c->f;
  w.cbase = static_cast<int32_t*>(cv.take((E + 1) * sizeof(int32_t)));
  w.x_q = static_cast<uint8_t*>(cv.take(static_cast<size_t>(N) * d));
  w.dy_q = static_cast<uint8_t*>(cv.take(static_cast<size_t>(N) * d));
  w.h_q = static_cast<uint8_t*>(cv.take(static_cast<size_t>(N) * f));
  w.dH1_q = static_cast<uint8_t*>(cv.take(static_cast<size_t>(N) * 2 * f));
  w.x_s = static_cast<uint8_t*>(cv.take(static_cast<size_t>(mx_tok_scale_bytes(N, E, d))));
  w.dy_s = static_cast<uint8_t*>(cv.take(static_cast<size_t>(mx_tok_scale_bytes(N, E, d))));
  w.h_s = static_cast<uint8_t*>(cv.take(static_cast<size_t>(mx_tok_scale_bytes(N, E, f))));
  w.dH1_s = static_cast<uint8_t*>(cv.take(static_cast<size_t>(mx_tok_scale_bytes(N, E, 2 * f))));
  w.sched = static_cast<int*>(cv.take(2 * 16));
  return w;
}

// Counters of the weight-gradient GEMMs' run-time tile scheduling, one 16-byte slot per launch
// (routed fc2, routed fc1, shared fc2, shared fc1, router).
constexpr int SCHED_SLOTS = 5;

struct BwdWs {
  void* dy_perm;
  float* dgate;
  void* dH1;
  void* s_dH1;   // the shared expert's [da | du] (its own buffer: it may run concurrently)
  void* dshared;
  float* dcoef;
  void* dx_shared;
  void* dl_ext;
  float* dz;
  void* dx_router;
  float* part;
  int* sched;   // tile counters of the weight-gradient GEMMs (SCHED_SLOTS slots of 4 ints)
};
static BwdWs carve_bwd(Carve& cv, const moe_cfg* c) {
  BwdWs w;
  const size_t es = esize(c);
  const size_t N = static_cast<size_t>(Nrows(c));
  const size_t T = static_cast<size_t>(c->T);
  const bool sh = c->f_shared > 0, gt = c->shared_gate != 0;
  w.dy_perm = cv.take(N * c->d * es);
  w.dgate = static_cast<float*>(cv.take(N * 4));
  w.dH1 = cv.take(N * 2 * c->f * es);
  w.s_dH1 = sh ? cv.take(T * 2 * c->f_shared * es) : nullptr;
  w.dshared = sh ? cv.take(T * c->d * es) : nullptr;
  w.dcoef = gt ? static_cast<float*>(cv.take(T * 4)) : nullptr;
  w.dx_shared = sh ? cv.take(T * c->d * es) : nullptr;
  w.dl_ext = cv.take(T * ext_cols(c) * es);
  w.dz = static_cast<float*>(cv.take(T * 4));
  w.dx_router = cv.take(T * c->d * es);
  const size_t mr = c->E + (gt ? 1 : 0);
  w.part = static_cast<float*>(cv.take(static_cast<size_t>(router_splits(c)) * mr * c->d * 4));
  w.sched = static_cast<int*>(cv.take(SCHED_SLOTS * 4 * sizeof(int)));
  return w;
}

// ------------------------------------------------------------------ checks
static int check_cfg(const moe_cfg* c) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "cfg is NULL");
  if (c->T < 0 || c->d <= 0 || c->E <= 0 || c->k <= 0 || c->f <= 0 || c->f_shared < 0)
    return fail(MOE_ERR_INVALID_ARG, "sizes must be positive (T >= 0): T=%d d=%d E=%d k=%d f=%d f_shared=%d",
                c->T, c->d, c->E, c->k, c->f, c->f_shared);
  if (c->E > MOE_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "E=%d exceeds %d", c->E, MOE_MAX_EXPERTS);
  if (c->k > MOE_MAX_TOPK) return fail(MOE_ERR_UNSUPPORTED, "k=%d exceeds %d", c->k, MOE_MAX_TOPK);
  if (c->k > c->E) return fail(MOE_ERR_INVALID_ARG, "k=%d exceeds E=%d", c->k, c->E);
  if (c->score_fn != MOE_SCORE_SOFTMAX && c->score_fn != MOE_SCORE_SIGMOID)
    return fail(MOE_ERR_INVALID_ARG, "score_fn=%d", c->score_fn);
  if ((c->renorm != 0 && c->renorm != 1) || (c->shared_gate != 0 && c->shared_gate != 1))
    return fail(MOE_ERR_INVALID_ARG, "renorm and shared_gate must be 0 or 1");
  if (c->shared_gate && c->f_shared == 0)
    return fail(MOE_ERR_INVALID_ARG, "shared_gate needs a shared expert (f_shared > 0)");
  if (c->dtype != MOE_DTYPE_BF16 && c->dtype != MOE_DTYPE_F32)
    return fail(MOE_ERR_INVALID_ARG, "dtype=%d", c->dtype);
  if (c->bias_mode != MOE_BIAS_LOGIT && c->bias_mode != MOE_BIAS_SELECT)
    return fail(MOE_ERR_INVALID_ARG, "bias_mode=%d", c->bias_mode);
  if (!(c->aux_coeff >= 0.0f) || c->aux_coeff > 3.0e38f)
    return fail(MOE_ERR_INVALID_ARG, "aux_coeff must be finite and >= 0");
  const int mult = c->dtype == MOE_DTYPE_BF16 ? 8 : 4;
  if (c->d % mult || c->f % mult || c->f_shared % mult)
    return fail(MOE_ERR_UNSUPPORTED, "d, f and f_shared must be multiples of %d (16-byte rows)", mult);
  if (Nrows(c) > 0x7fffffffLL) return fail(MOE_ERR_UNSUPPORTED, "T*k exceeds 2^31-1");
  return MOE_OK;
}

static int check_ptr(const void* p, const char* name, bool required) {
  if (!p) return required ? fail(MOE_ERR_INVALID_ARG, "%s is NULL", name) : MOE_OK;
  if (reinterpret_cast<uintptr_t>(p) & 15u)
    return fail(MOE_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
  return MOE_OK;
}

static int check_ws(const moe_cfg* c, int which, void* ws, size_t ws_bytes) {
  const size_t need = moe_workspace_bytes(c, which);
  if (need == 0) return MOE_OK;
  if (!ws || ws_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                ws ? ws_bytes : static_cast<size_t>(0));
  return check_ptr(ws, "ws", true);
}

static cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }

// Build option: the bf16 layer folds the permutation into its GEMMs' operand loads (fc1 and
// its weight gradient gather x rows by token_of_slot with tile::gather4; no x_perm).  Parity-
// tested, but slower on GB300: one gather4 copy moves 512 bytes, and the TMA unit's copy rate
// (about 6 bytes per clock per SM) is well short of the 27 bytes per clock the MMAs consume
// (fc1 + SwiGLU 1.47 -> 4.5 ms, fc1 weight gradient 1.85 -> 9.8 ms on the 128-expert layer),
// while the explicit permute kernel moves its bytes at ~90% of HBM bandwidth.  Off by default;
// the fp32 CUDA-core path always permutes explicitly.
#ifndef MOE_FUSE_PERMUTE
#define MOE_FUSE_PERMUTE 0
#endif
static bool permute_fused(const moe_cfg* c) {
  return MOE_FUSE_PERMUTE && c->dtype == MOE_DTYPE_BF16;
}

// ------------------------------------------------------------------ stages
static int gemm(const moe_cfg* c, const GemmDesc& g, cudaStream_t st) {
  return c->dtype == MOE_DTYPE_BF16 ? gemm_tc(g, st) : gemm_simt(g, st);
}

static GemmDesc desc0() {
  GemmDesc g;
  memset(&g, 0, sizeof(g));
  return g;
}

static Operand opnd(const void* base, int64_t rows, int64_t cols, bool mn) {
  Operand o;
  o.base = base;
  o.rows = rows;
  o.cols = cols;
  o.ld = cols;
  o.mn_major = mn;
  return o;
}

static int route_impl(const moe_cfg* c, const void* x, const void* W_r, const float* b_r,
                      const float* logits_in, float* logits_out, int32_t* idx, float* gate,
                      int32_t* counts, int32_t* offsets, int32_t* sop, int32_t* tos,
                      const RouteWs& w, cudaStream_t st) {
  // MOE_BIAS_LOGIT: b_r enters the logits (router GEMM epilogue); MOE_BIAS_SELECT: it is the
  // selection-only expert bias of the top-k.
  const bool select_bias = c->bias_mode == MOE_BIAS_SELECT;
  const float* logits = logits_in;
  bool selected = false;   // idx, gate and the histogram rows already written
  if (!logits) {
    float* dst = logits_out ? logits_out : w.logits;
    GemmDesc g = desc0();
    g.name = "gemm_router";
    g.sched = RAGGED_M;
    g.epi = EPI_F32;
    g.G = 1;
    g.M = c->T;
    g.N = c->E;
    g.K = c->d;
    g.A = opnd(x, c->T, c->d, false);
    g.B = opnd(W_r, c->E, c->d, false);
    g.out = dst;
    g.ldo = c->E;
    g.bias = select_bias ? nullptr : b_r;
    if (c->dtype == MOE_DTYPE_BF16) {
      // tensor-core router: each epilogue thread holds one token's E logits in tensor memory
      // and routes the token there (selection, gates, its tile's histogram row)
      g.rt.idx = idx;
      g.rt.gate = gate;
      g.rt.hist = w.hist;
      g.rt.sel_bias = select_bias ? b_r : nullptr;
      g.rt.k = c->k;
      g.rt.score_fn = c->score_fn;
      g.rt.renorm = c->renorm;
      g.rt.ldh = route_ldh(c->E);
      selected = true;
    }
    MOE_TRY(gemm(c, g, st));
    logits = dst;
  }
  if (!selected)
    MOE_TRY(launch_topk(logits, c->T, c->E, c->k, c->score_fn, c->renorm,
                        select_bias ? b_r : nullptr, idx, gate, w.hist, st));
  return launch_slots(idx, c->T, c->k, c->E, w.hist, w.rowpre, counts, offsets, sop, tos, st);
}

// fc1 + SwiGLU and fc2 for G groups whose rows are given by offsets (null: one group of `rows`).
// gather (bf16): fc1 reads row s of its A operand from row gather[s] of x_perm, which is then
// the unpermuted x with src_rows rows (the permutation folded into the operand load).
static int ffn_fwd_impl(const moe_cfg* c, int G, const int32_t* offsets, int64_t rows, int f,
                        const void* x_perm, const void* W1, const void* W2, void* h, void* act,
                        void* y_perm, cudaStream_t st, const int32_t* gather = nullptr,
                        int64_t src_rows = 0) {
  const int d = c->d;
  const bool shared = offsets == nullptr;
  GemmDesc g1 = desc0();
  g1.name = shared ? "gemm_shared_fc1_swiglu" : "gemm_fc1_swiglu";
  g1.sched = RAGGED_M;
  g1.epi = EPI_SWIGLU_FWD;
  g1.G = G;
  g1.offsets = offsets;
  g1.M = static_cast<int>(rows);
  g1.N = 2 * f;
  g1.K = d;
  g1.A = opnd(x_perm, gather ? src_rows : rows, d, false);
  g1.gather = gather;
  g1.B = opnd(W1, static_cast<int64_t>(G) * 2 * f, d, false);
  g1.b_group_rows = 2 * f;
  g1.b_up_rows = f;
  g1.f = f;
  g1.out = h;
  g1.ldo = f;
  g1.out2 = act;
  g1.ldo2 = 2 * f;
  MOE_TRY(gemm(c, g1, st));
  GemmDesc g2 = desc0();
  g2.name = shared ? "gemm_shared_fc2" : "gemm_fc2";
  g2.sched = RAGGED_M;
  g2.epi = EPI_STORE;
  g2.G = G;
  g2.offsets = offsets;
  g2.M = static_cast<int>(rows);
  g2.N = d;
  g2.K = f;
  g2.A = opnd(h, rows, f, false);
  g2.B = opnd(W2, static_cast<int64_t>(G) * d, f, false);
  g2.b_group_rows = d;
  g2.out = y_perm;
  g2.ldo = d;
  return gemm(c, g2, st);
}

// Backward of ffn_fwd_impl.  Order matters when dx_perm aliases dy_perm: dy_perm is last read
// by the fc2 weight gradient, which runs before the fc1 data gradient writes dx_perm.
static int ffn_bwd_impl(const moe_cfg* c, int G, const int32_t* offsets, int64_t rows, int f,
                        const void* x_perm, const void* W1, const void* W2, const void* act,
                        const void* h, const void* dy_perm, void* dH1, void* dx_perm, float* dW1,
                        float* dW2, int* sched, cudaStream_t st, const int32_t* gather = nullptr,
                        int64_t src_rows = 0) {
  const int d = c->d;
  const bool shared = offsets == nullptr;
  // dh = dy_perm . W2_g  (+ SwiGLU backward -> dH1 = [da | du])
  GemmDesc a = desc0();
  a.name = shared ? "gemm_shared_fc2_dgrad" : "gemm_fc2_dgrad";
  a.sched = RAGGED_M;
  a.epi = EPI_SWIGLU_BWD;
  a.G = G;
  a.offsets = offsets;
  a.M = static_cast<int>(rows);
  a.N = f;
  a.K = d;
  a.A = opnd(dy_perm, rows, d, false);
  a.B = opnd(W2, static_cast<int64_t>(G) * d, f, true);
  a.b_group_rows = d;
  a.f = f;
  a.out = dH1;
  a.ldo = 2 * f;
  a.aux = act;
  a.ld_aux = 2 * f;
  MOE_TRY(gemm(c, a, st));
  // dW2_g = dy_perm_g^T . h_g
  GemmDesc b = desc0();
  b.name = shared ? "gemm_shared_fc2_wgrad" : "gemm_fc2_wgrad";
  b.sched = RAGGED_K;
  b.epi = EPI_F32;
  b.G = G;
  b.offsets = offsets;
  b.M = d;
  b.N = f;
  b.K = static_cast<int>(rows);
  b.A = opnd(dy_perm, rows, d, true);
  b.B = opnd(h, rows, f, true);
  b.out = dW2;
  b.ldo = f;
  b.out_group_stride = static_cast<int64_t>(d) * f;
  b.tile_ctr = sched;
  MOE_TRY(gemm(c, b, st));
  // dx_perm = dH1 . W1_g
  GemmDesc e = desc0();
  e.name = shared ? "gemm_shared_fc1_dgrad" : "gemm_fc1_dgrad";
  e.sched = RAGGED_M;
  e.epi = EPI_STORE;
  e.G = G;
  e.offsets = offsets;
  e.M = static_cast<int>(rows);
  e.N = d;
  e.K = 2 * f;
  e.A = opnd(dH1, rows, 2 * f, false);
  e.B = opnd(W1, static_cast<int64_t>(G) * 2 * f, d, true);
  e.b_group_rows = 2 * f;
  e.out = dx_perm;
  e.ldo = d;
  MOE_TRY(gemm(c, e, st));
  // dW1_g = dH1_g^T . x_perm_g
  GemmDesc w = desc0();
  w.name = shared ? "gemm_shared_fc1_wgrad" : "gemm_fc1_wgrad";
  w.sched = RAGGED_K;
  w.epi = EPI_F32;
  w.G = G;
  w.offsets = offsets;
  w.M = 2 * f;
  w.N = d;
  w.K = static_cast<int>(rows);
  w.A = opnd(dH1, rows, 2 * f, true);
  w.B = opnd(x_perm, gather ? src_rows : rows, d, true);
  w.gather = gather;
  w.out = dW1;
  w.ldo = d;
  w.out_group_stride = static_cast<int64_t>(2) * f * d;
  w.tile_ctr = sched + 4;
  return gemm(c, w, st);
}

// The routed experts' forward on E4M3 operands (fc1 + SwiGLU with h's amax, h quantised, fc2).
// G groups of rows (offsets NULL: one group of all rows -- the shared expert), ffn width f.
static int ffn_fwd_fp8_impl(const moe_cfg* c, int G, const int32_t* offsets, int64_t rows, int f,
                            const uint8_t* x_perm_q,
                            const float* x_scale, const uint8_t* W1_q, const float* W1_scale,
                            const uint8_t* W2_q, const float* W2_scale, void* h, void* act,
                            uint8_t* h_q, float* h_scale, float* h_amax, void* y_perm,
                            cudaStream_t st) {
  const int64_t N = rows;
  const int d = c->d, E = G;
  const bool shared = offsets == nullptr;
  // fc1 + SwiGLU on E4M3 operands -> h, [a | u] (bf16)
  GemmDesc g1 = desc0();
  g1.name = shared ? "gemm_shared_fc1_swiglu_fp8" : "gemm_fc1_swiglu_fp8";
  g1.sched = RAGGED_M;
  g1.epi = EPI_SWIGLU_FWD;
  g1.G = E;
  g1.offsets = offsets;
  g1.M = static_cast<int>(N);
  g1.N = 2 * f;
  g1.K = d;
  g1.A = opnd(x_perm_q, N, d, false);
  g1.B = opnd(W1_q, static_cast<int64_t>(E) * 2 * f, d, false);
  g1.b_group_rows = 2 * f;
  g1.b_up_rows = f;
  g1.f = f;
  g1.out = h;
  g1.ldo = f;
  g1.out2 = act;
  g1.ldo2 = 2 * f;
  g1.fp8 = true;
  g1.a_scale = x_scale;
  g1.b_scale = W1_scale;
  g1.amax_out = h_amax;   // max |h| taken in fc1's epilogue
  if (cudaMemsetAsync(h_amax, 0, sizeof(float), st) != cudaSuccess)
    return fail(MOE_ERR_CUDA, "clearing h_amax failed");
  MOE_TRY(gemm_tc(g1, st));
  // h -> E4M3 (one tensor) with that amax
  MOE_TRY(launch_quant_e4m3_given_amax(h, N * f, 1, h_q, h_scale, h_amax, st));
  // fc2 on E4M3 operands -> y_perm (bf16)
  GemmDesc g2 = desc0();
  g2.name = shared ? "gemm_shared_fc2_fp8" : "gemm_fc2_fp8";
  g2.sched = RAGGED_M;
  g2.epi = EPI_STORE;
  g2.G = E;
  g2.offsets = offsets;
  g2.M = static_cast<int>(N);
  g2.N = d;
  g2.K = f;
  g2.A = opnd(h_q, N, f, false);
  g2.B = opnd(W2_q, static_cast<int64_t>(E) * d, f, false);
  g2.b_group_rows = d;
  g2.out = y_perm;
  g2.ldo = d;
  g2.fp8 = true;
  g2.a_scale = h_scale;
  g2.b_scale = W2_scale;
  return gemm_tc(g2, st);
}

// The routed experts' backward on E4M3 operands: dy quantised, fc2 dgrad + SwiGLU backward
// (with [da | du]'s amax), [da | du] quantised, fc2 wgrad, fc1 dgrad, fc1 wgrad.  dx_perm may
// alias dy_perm (dy_perm is read only by the first quantisation).
static int ffn_bwd_fp8_impl(const moe_cfg* c, int G, const int32_t* offsets, int64_t rows, int f,
                            const uint8_t* x_perm_q,
                            const float* x_scale, const uint8_t* W1_q, const float* W1_scale,
                            const uint8_t* W2_q, const float* W2_scale, const void* act,
                            const uint8_t* h_q, const float* h_scale, const void* dy_perm,
                            uint8_t* dy_q, float* dy_scale, float* dy_amax, void* dH1,
                            uint8_t* dH1_q, float* dH1_scale, float* dH1_amax, void* dx_perm,
                            float* dW1, float* dW2, int* sched, cudaStream_t st,
                            bool dy_amax_ready = false) {
  const int64_t N = rows;
  const int d = c->d, E = G;
  const bool shared = offsets == nullptr;
  // dy_perm -> E4M3 (one tensor; its amax already reduced by the producer of dy_perm, or here)
  if (dy_amax_ready)
    MOE_TRY(launch_quant_e4m3_given_amax(dy_perm, N * d, 1, dy_q, dy_scale, dy_amax, st));
  else
    MOE_TRY(launch_quantize_e4m3(dy_perm, N * d, 1, dy_q, dy_scale, dy_amax, st));
  // dh = dy . W2_e on E4M3 operands (W2_q read MN-major: no transposed copy), SwiGLU backward
  // -> dH1 = [da | du] (bf16) with its amax
  GemmDesc a = desc0();
  a.name = shared ? "gemm_shared_fc2_dgrad_fp8" : "gemm_fc2_dgrad_fp8";
  a.sched = RAGGED_M;
  a.epi = EPI_SWIGLU_BWD;
  a.G = E;
  a.offsets = offsets;
  a.M = static_cast<int>(N);
  a.N = f;
  a.K = d;
  a.A = opnd(dy_q, N, d, false);
  a.B = opnd(W2_q, static_cast<int64_t>(E) * d, f, true);
  a.b_group_rows = d;
  a.f = f;
  a.out = dH1;
  a.ldo = 2 * f;
  a.aux = act;
  a.ld_aux = 2 * f;
  a.fp8 = true;
  a.a_scale = dy_scale;
  a.b_scale = W2_scale;
  a.amax_out = dH1_amax;
  if (cudaMemsetAsync(dH1_amax, 0, sizeof(float), st) != cudaSuccess)
    return fail(MOE_ERR_CUDA, "clearing dH1_amax failed");
  MOE_TRY(gemm_tc(a, st));
  // dH1 -> E4M3 (one tensor) with that amax
  MOE_TRY(launch_quant_e4m3_given_amax(dH1, N * 2 * f, 1, dH1_q, dH1_scale, dH1_amax, st));
  // dW2_e = dy_e^T . h_e (both MN-major over the expert's rows)
  GemmDesc b = desc0();
  b.name = shared ? "gemm_shared_fc2_wgrad_fp8" : "gemm_fc2_wgrad_fp8";
  b.sched = RAGGED_K;
  b.epi = EPI_F32;
  b.G = E;
  b.offsets = offsets;
  b.M = d;
  b.N = f;
  b.K = static_cast<int>(N);
  b.A = opnd(dy_q, N, d, true);
  b.B = opnd(h_q, N, f, true);
  b.out = dW2;
  b.ldo = f;
  b.out_group_stride = static_cast<int64_t>(d) * f;
  b.tile_ctr = sched;
  b.fp8 = true;
  b.a_scale = dy_scale;
  b.b_scale = h_scale;
  b.b_scale_scalar = true;
  MOE_TRY(gemm_tc(b, st));
  // dx_perm = dH1 . W1_e
  GemmDesc e = desc0();
  e.name = shared ? "gemm_shared_fc1_dgrad_fp8" : "gemm_fc1_dgrad_fp8";
  e.sched = RAGGED_M;
  e.epi = EPI_STORE;
  e.G = E;
  e.offsets = offsets;
  e.M = static_cast<int>(N);
  e.N = d;
  e.K = 2 * f;
  e.A = opnd(dH1_q, N, 2 * f, false);
  e.B = opnd(W1_q, static_cast<int64_t>(E) * 2 * f, d, true);
  e.b_group_rows = 2 * f;
  e.out = dx_perm;
  e.ldo = d;
  e.fp8 = true;
  e.a_scale = dH1_scale;
  e.b_scale = W1_scale;
  MOE_TRY(gemm_tc(e, st));
  // dW1_e = dH1_e^T . x_perm_e
  GemmDesc w = desc0();
  w.name = shared ? "gemm_shared_fc1_wgrad_fp8" : "gemm_fc1_wgrad_fp8";
  w.sched = RAGGED_K;
  w.epi = EPI_F32;
  w.G = E;
  w.offsets = offsets;
  w.M = 2 * f;
  w.N = d;
  w.K = static_cast<int>(N);
  w.A = opnd(dH1_q, N, 2 * f, true);
  w.B = opnd(x_perm_q, N, d, true);
  w.out = dW1;
  w.ldo = d;
  w.out_group_stride = static_cast<int64_t>(2) * f * d;
  w.tile_ctr = sched + 4;
  w.fp8 = true;
  w.a_scale = dH1_scale;
  w.b_scale = x_scale;
  w.b_scale_scalar = true;
  return gemm_tc(w, st);
}

}  // namespace moe

using namespace moe;

// ====================================================================== C ABI
extern "C" {

int moe_version(void) { return 202; }

const char* moe_last_error(void) { return g_errbuf; }

uint64_t moe_launch_count(void) { return g_launches.load(); }

int moe_trace_enable(int on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on.store(on ? 1 : 0);
  return MOE_OK;
}

int moe_trace_read(char* names, int name_stride, int* launches, double* total_ms, int cap) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  std::vector<std::string> kinds;
  std::vector<int> cnt;
  std::vector<double> ms;
  for (auto& r : g_trace) {
    if (cudaEventSynchronize(r.stop) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "cudaEventSynchronize failed in trace read");
    float t = 0.f;
    cudaEventElapsedTime(&t, r.start, r.stop);
    size_t i = 0;
    for (; i < kinds.size(); ++i)
      if (kinds[i] == r.name) break;
    if (i == kinds.size()) {
      kinds.emplace_back(r.name);
      cnt.push_back(0);
      ms.push_back(0.0);
    }
    cnt[i] += 1;
    ms[i] += t;
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  g_trace.clear();
  const int n = static_cast<int>(kinds.size());
  for (int i = 0; i < n && i < cap; ++i) {
    if (names && name_stride > 0) {
      strncpy(names + static_cast<size_t>(i) * name_stride, kinds[i].c_str(), name_stride - 1);
      names[static_cast<size_t>(i) * name_stride + name_stride - 1] = 0;
    }
    if (launches) launches[i] = cnt[i];
    if (total_ms) total_ms[i] = ms[i];
  }
  return n;
}

int moe_check_device_error(void* stream, int32_t* code) {
  if (cudaStreamSynchronize(S(stream)) != cudaSuccess)
    return fail(MOE_ERR_CUDA, "stream synchronisation failed: %s", cudaGetErrorString(cudaGetLastError()));
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess)
    return fail(MOE_ERR_CUDA, "reading the device error word failed");
  if (code) *code = v;
  if (v) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    return fail(MOE_ERR_DEVICE_CHECK, "a kernel reported device error code %d", v);
  }
  return MOE_OK;
}

size_t moe_workspace_bytes(const moe_cfg* c, int which) {
  if (check_cfg(c) != MOE_OK) return 0;
  Carve cv(nullptr);
  switch (which) {
    case MOE_WS_ROUTE:
    case MOE_WS_LAYER_FWD:
      carve_route(cv, c);
      break;
    case MOE_WS_FFN_FWD:
      return 0;
    case MOE_WS_FFN_BWD:
      cv.take(static_cast<size_t>(Nrows(c)) * 2 * c->f * esize(c));
      cv.take(2 * 4 * sizeof(int));
      break;
    case MOE_WS_LAYER_BWD:
      carve_bwd(cv, c);
      break;
    case MOE_WS_FFN_BWD_FP8:
      cv.take(2 * 4 * sizeof(int));
      break;
    case MOE_WS_WGRAD_MXFP8:
      carve_wgmx(cv, c);
      break;
    case MOE_WS_LAYER_BWD_FP8:
      carve_bwd(cv, c);
      cv.take(static_cast<size_t>(Nrows(c)) * c->d);
      cv.take(static_cast<size_t>(Nrows(c)) * 2 * c->f);
      if (c->f_shared > 0) {   // room for an FP8 shared expert's gradient codes
        cv.take(static_cast<size_t>(c->T) * c->d);
        cv.take(static_cast<size_t>(c->T) * 2 * c->f_shared);
      }
      break;
    default:
      return 0;
  }
  return cv.off + 256;
}

int moe_route_topk(const moe_cfg* c, const void* x, const void* W_r, const float* b_r,
                   const float* logits_in, float* logits_out, int32_t* idx, float* gate,
                   int32_t* counts, int32_t* offsets, int32_t* slot_of_pair,
                   int32_t* token_of_slot, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(c));
  MOE_TRY(check_ptr(x, "x", !logits_in));
  MOE_TRY(check_ptr(W_r, "W_r", !logits_in));
  MOE_TRY(check_ptr(b_r, "b_r", false));
  MOE_TRY(check_ptr(logits_in, "logits_in", false));
  MOE_TRY(check_ptr(logits_out, "logits_out", false));
  MOE_TRY(check_ptr(idx, "idx", true));
  MOE_TRY(check_ptr(gate, "gate", true));
  MOE_TRY(check_ptr(counts, "counts", true));
  MOE_TRY(check_ptr(offsets, "offsets", true));
  MOE_TRY(check_ptr(slot_of_pair, "slot_of_pair", true));
  MOE_TRY(check_ptr(token_of_slot, "token_of_slot", true));
  MOE_TRY(check_ws(c, MOE_WS_ROUTE, ws, ws_bytes));
  cudaStream_t st = S(stream);
  if (c->T == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * c->E, st) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c->E + 1), st) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "cudaMemsetAsync failed");
    return MOE_OK;
  }
  Carve cv(ws);
  RouteWs w = carve_route(cv, c);
  return route_impl(c, x, W_r, b_r, logits_in, logits_out, idx, gate, counts, offsets,
                    slot_of_pair, token_of_slot, w, st);
}

int moe_permute(const moe_cfg* c, const void* x, const int32_t* slot_of_pair, void* x_perm,
                void* stream) {
  MOE_TRY(check_cfg(c));
  MOE_TRY(check_ptr(x, "x", true));
  MOE_TRY(check_ptr(slot_of_pair, "slot_of_pair", true));
  MOE_TRY(check_ptr(x_perm, "x_perm", true));
  return launch_permute(c->dtype, x, slot_of_pair, x_perm, c->T, c->d, c->k, S(stream));
}

int moe_grouped_swiglu_fwd(const moe_cfg* c, const void* x_perm, const int32_t* offsets,
                           const void* W1, const void* W2, void* h, void* act, void* y_perm,
                           void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(c));
  MOE_TRY(check_ptr(x_perm, "x_perm", true));
  MOE_TRY(check_ptr(offsets, "offsets", true));
  MOE_TRY(check_ptr(W1, "W1", true));
  MOE_TRY(check_ptr(W2, "W2", true));
  MOE_TRY(check_ptr(h, "h", true));
  MOE_TRY(check_ptr(act, "act", false));
  MOE_TRY(check_ptr(y_perm, "y_perm", true));
  MOE_TRY(check_ws(c, MOE_WS_FFN_FWD, ws, ws_bytes));
  if (Nrows(c) == 0) return MOE_OK;
  return ffn_fwd_impl(c, c->E, offsets, Nrows(c), c->f, x_perm, W1, W2, h, act, y_perm, S(stream));
}

int moe_grouped_swiglu_bwd(const moe_cfg* c, const void* x_perm, const int32_t* offsets,
                           const void* W1, const void* W2, const void* act, const void* h,
                           const void* dy_perm, void* dx_perm, float* dW1, float* dW2, void* ws,
                           size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(c));
  MOE_TRY(check_ptr(x_perm, "x_perm", true));
  MOE_TRY(check_ptr(offsets, "offsets", true));
  MOE_TRY(check_ptr(W1, "W1", true));
  MOE_TRY(check_ptr(W2, "W2", true));
  MOE_TRY(check_ptr(act, "act", true));
  MOE_TRY(check_ptr(h, "h", true));
  MOE_TRY(check_ptr(dy_perm, "dy_perm", true));
  MOE_TRY(check_ptr(dx_perm, "dx_perm", true));
  MOE_TRY(check_ptr(dW1, "dW1", true));
  MOE_TRY(check_ptr(dW2, "dW2", true));
  MOE_TRY(check_ws(c, MOE_WS_FFN_BWD, ws, ws_bytes));
  cudaStream_t st = S(stream);
  if (Nrows(c) == 0) {
    if (cudaMemsetAsync(dW1, 0, sizeof(float) * c->E * 2 * c->f * c->d, st) != cudaSuccess ||
        cudaMemsetAsync(dW2, 0, sizeof(float) * c->E * c->d * c->f, st) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "cudaMemsetAsync failed");
    return MOE_OK;
  }
  Carve cv(ws);
  void* dH1 = cv.take(static_cast<size_t>(Nrows(c)) * 2 * c->f * esize(c));
  int* sched = static_cast<int*>(cv.take(2 * 4 * sizeof(int)));
  return ffn_bwd_impl(c, c->E, offsets, Nrows(c), c->f, x_perm, W1, W2, act, h, dy_perm, dH1,
                      dx_perm, dW1, dW2, sched, st);
}

int moe_grouped_swiglu_fwd_gathered(const moe_cfg* c, const void* x,
                                    const int32_t* token_of_slot, const int32_t* offsets,
                                    const void* W1, const void* W2, void* h, void* act,
                                    void* y_perm, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(c));
  if (c->dtype != MOE_DTYPE_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "gathered operands need the bf16 tensor-core path");
  MOE_TRY(check_ptr(x, "x", true));
  MOE_TRY(check_ptr(token_of_slot, "token_of_slot", true));
  MOE_TRY(check_ptr(offsets, "offsets", true));
  MOE_TRY(check_ptr(W1, "W1", true));
  MOE_TRY(check_ptr(W2, "W2", true));
  MOE_TRY(check_ptr(h, "h", true));
  MOE_TRY(check_ptr(act, "act", false));
  MOE_TRY(check_ptr(y_perm, "y_perm", true));
  MOE_TRY(check_ws(c, MOE_WS_FFN_FWD, ws, ws_bytes));
  if (Nrows(c) == 0) return MOE_OK;
  return ffn_fwd_impl(c, c->E, offsets, Nrows(c), c->f, x, W1, W2, h, act, y_perm, S(stream),
                      token_of_slot, c->T);
}

int moe_grouped_swiglu_bwd_gathered(const moe_cfg* c, const void* x,
                                    const int32_t* token_of_slot, const int32_t* offsets,
                                    const void* W1, const void* W2, const void* act,
                                    const void* h, const void* dy_perm, void* dx_perm,
                                    float* dW1, float* dW2, void* ws, size_t ws_bytes,
                                    void* stream) {
  MOE_TRY(check_cfg(c));
  if (c->dtype != MOE_DTYPE_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "gathered operands need the bf16 tensor-core path");
  MOE_TRY(check_ptr(x, "x", true));
  MOE_TRY(check_ptr(token_of_slot, "token_of_slot", true));
  MOE_TRY(check_ptr(offsets, "offsets", true));
  MOE_TRY(check_ptr(W1, "W1", true));
  MOE_TRY(check_ptr(W2, "W2", true));
  MOE_TRY(check_ptr(act, "act", true));
  MOE_TRY(check_ptr(h, "h", true));
  MOE_TRY(check_ptr(dy_perm, "dy_perm", true));
  MOE_TRY(check_ptr(dx_perm, "dx_perm", true));
  MOE_TRY(check_ptr(dW1, "dW1", true));
  MOE_TRY(check_ptr(dW2, "dW2", true));
  MOE_TRY(check_ws(c, MOE_WS_FFN_BWD, ws, ws_bytes));
  cudaStream_t st = S(stream);
  if (Nrows(c) == 0) {
    if (cudaMemsetAsync(dW1, 0, sizeof(float) * c->E * 2 * c->f * c->d, st) != cudaSuccess ||
        cudaMemsetAsync(dW2, 0, sizeof(float) * c->E * c->d * c->f, st) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "cudaMemsetAsync failed");
    return MOE_OK;
  }
  Carve cv(ws);
  void* dH1 = cv.take(static_cast<size_t>(Nrows(c)) * 2 * c->f * esize(c));
  int* sched = static_cast<int*>(cv.take(2 * 4 * sizeof(int)));
  return ffn_bwd_impl(c, c->E, offsets, Nrows(c), c->f, x, W1, W2, act, h, dy_perm, dH1, dx_perm,
                      dW1, dW2, sched, st, token_of_slot, c->T);
}

int moe_quantize_e4m3(const void* x, int64_t elems_per_group, int32_t groups, uint8_t* q,
                      float* scale, float* amax, void* stream) {
  if (groups < 1 || elems_per_group < 0)
    return fail(MOE_ERR_INVALID_ARG, "groups=%d elems_per_group=%lld", groups,
                static_cast<long long>(elems_per_group));
  if (elems_per_group % 16)
    return fail(MOE_ERR_UNSUPPORTED, "elems_per_group must be a multiple of 16");
  MOE_TRY(check_ptr(x, "x", true));
  MOE_TRY(check_ptr(q, "q", true));
  MOE_TRY(check_ptr(scale, "scale", true));
  MOE_TRY(check_ptr(amax, "amax", true));
  return launch_quantize_e4m3(x, elems_per_group, groups, q, scale, amax, S(stream));
}

int moe_permute_quantize_e4m3(const moe_cfg* c, const void* x, const int32_t* slot_of_pair,
                              uint8_t* x_perm_q, float* x_scale, float* x_amax, void* stream) {
  MOE_TRY(check_cfg(c));
  if (c->dtype != MOE_DTYPE_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "E4M3 quantisation reads bf16 activations");
  if (c->d % 16) return fail(MOE_ERR_UNSUPPORTED, "d must be a multiple of 16 (16-byte rows)");
  MOE_TRY(check_ptr(x, "x", true));
  MOE_TRY(check_ptr(slot_of_pair, "slot_of_pair", true));
  MOE_TRY(check_ptr(x_perm_q, "x_perm_q", true));
  MOE_TRY(check_ptr(x_scale, "x_scale", true));
  MOE_TRY(check_ptr(x_amax, "x_amax", true));
  if (c->T == 0) return MOE_OK;
  return launch_permute_quant_e4m3(x, slot_of_pair, x_perm_q, nullptr, x_scale, x_amax, c->T, c->d,
                                   c->k, S(stream));
}

int moe_grouped_swiglu_fwd_fp8(const moe_cfg* c, const uint8_t* x_perm_q, const float* x_scale,
                               const int32_t* offsets, const uint8_t* W1_q, const float* W1_scale,
                               const uint8_t* W2_q, const float* W2_scale, void* h, void* act,
                               uint8_t* h_q, float* h_scale, float* h_amax, void* y_perm,
                               void* stream) {
  MOE_TRY(check_cfg(c));
  if (c->dtype != MOE_DTYPE_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "the FP8 path writes bf16 activations (dtype bf16)");
  if (c->d % 16 || c->f % 16)
    return fail(MOE_ERR_UNSUPPORTED, "FP8 rows need d and f multiples of 16 (16-byte rows)");
  MOE_TRY(check_ptr(x_perm_q, "x_perm_q", true));
  MOE_TRY(check_ptr(x_scale, "x_scale", true));
  MOE_TRY(check_ptr(offsets, "offsets", true));
  MOE_TRY(check_ptr(W1_q, "W1_q", true));
  MOE_TRY(check_ptr(W1_scale, "W1_scale", true));
  MOE_TRY(check_ptr(W2_q, "W2_q", true));
  MOE_TRY(check_ptr(W2_scale, "W2_scale", true));
  MOE_TRY(check_ptr(h, "h", true));
  MOE_TRY(check_ptr(act, "act", false));
  MOE_TRY(check_ptr(h_q, "h_q", true));
  MOE_TRY(check_ptr(h_scale, "h_scale", true));
  MOE_TRY(check_ptr(h_amax, "h_amax", true));
  MOE_TRY(check_ptr(y_perm, "y_perm", true));
  cudaStream_t st = S(stream);
  const int64_t N = Nrows(c);
  if (N == 0) return MOE_OK;
  return ffn_fwd_fp8_impl(c, c->E, offsets, Nrows(c), c->f, x_perm_q, x_scale, W1_q, W1_scale, W2_q, W2_scale, h, act,
                          h_q, h_scale, h_amax, y_perm, st);
}

// ------------------------------------------------------------------ MXFP8
static int check_mx_cfg(const moe_cfg* c) {
  MOE_TRY(check_cfg(c));
  if (c->dtype != MOE_DTYPE_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "the MXFP8 path reads and writes bf16 activations (dtype bf16)");
  if (c->d % 32 || c->f % 32)
    return fail(MOE_ERR_UNSUPPORTED, "MXFP8 blocks need d and f multiples of 32");
  return MOE_OK;
}

// The routed experts' forward on MXFP8 operands: fc1 + SwiGLU with h quantised to MXFP8 in its
// epilogue, then fc2 (N rows; bf16 h and [a | u] written only where given).
static int ffn_fwd_mx_impl(const moe_cfg* c, const int32_t* offsets, int64_t N,
                           const uint8_t* x_perm_q, const uint8_t* x_perm_s, const uint8_t* W1_q,
                           const uint8_t* W1_sp, const uint8_t* W2_q, const uint8_t* W2_sp, void* h,
                           void* act, uint8_t* h_q, uint8_t* h_s, void* y_perm, cudaStream_t st) {
  const int d = c->d, f = c->f, E = c->E;
  // fc1 + SwiGLU on MXFP8 operands -> h codes and block scales (and bf16 h, [a | u] if asked)
  GemmDesc g1 = desc0();
  g1.name = "gemm_fc1_swiglu_mxfp8";
  g1.sched = RAGGED_M;
  g1.epi = EPI_SWIGLU_FWD;
  g1.G = E;
  g1.offsets = offsets;
  g1.M = static_cast<int>(N);
  g1.N = 2 * f;
  g1.K = d;
  g1.A = opnd(x_perm_q, N, d, false);
  g1.B = opnd(W1_q, static_cast<int64_t>(E) * 2 * f, d, false);
  g1.b_group_rows = 2 * f;
  g1.b_up_rows = f;
  g1.f = f;
  g1.out = h;
  g1.ldo = f;
  g1.out2 = act;
  g1.ldo2 = 2 * f;
  g1.fp8 = true;
  g1.mx = true;
  g1.sfa = x_perm_s;
  g1.sfb = W1_sp;
  g1.q_out = h_q;
  g1.q_sf = h_s;
  MOE_TRY(gemm_tc(g1, st));
  // fc2 on MXFP8 operands -> y_perm (bf16)
  GemmDesc g2 = desc0();
  g2.name = "gemm_fc2_mxfp8";
  g2.sched = RAGGED_M;
  g2.epi = EPI_STORE;
  g2.G = E;
  g2.offsets = offsets;
  g2.M = static_cast<int>(N);
  g2.N = d;
  g2.K = f;
  g2.A = opnd(h_q, N, f, false);
  g2.B = opnd(W2_q, static_cast<int64_t>(E) * d, f, false);
  g2.b_group_rows = d;
  g2.out = y_perm;
  g2.ldo = d;
  g2.fp8 = true;
  g2.mx = true;
  g2.sfa = h_s;
  g2.sfb = W2_sp;
  return gemm_tc(g2, st);
}

size_t moe_mxfp8_scale_bytes(const moe_cfg* c, int which) {
  if (validate_cfg(c) != MOE_OK) return 0;
  const int64_t N = Nrows(c);
  switch (which) {
    case MOE_MX_SCALES_X: return static_cast<size_t>(mx_act_scale_bytes(N, c->E, c->d));
    case MOE_MX_SCALES_H: return static_cast<size_t>(mx_act_scale_bytes(N, c->E, c->f));
    case MOE_MX_SCALES_W1:
      return static_cast<size_t>(c->E) * mx_fc1_tiles(c->f) * mx_kch(c->d) * MX_SFB_BYTES;
    case MOE_MX_SCALES_W2:
      return static_cast<size_t>(c->E) * mx_fc2_tiles(c->d) * mx_kch(c->f) * MX_SFB_BYTES;
    case MOE_MX_SCALES_DH1: return static_cast<size_t>(mx_act_scale_bytes(N, c->E, 2 * c->f));
    case MOE_MX_SCALES_W1C:   // W1 read as [2f (K), d (N)]: tiles of MX_BN_DGRAD1 columns of d
      return static_cast<size_t>(c->E) * ((c->d + MX_BN_DGRAD1 - 1) / MX_BN_DGRAD1) *
             mx_kch(2 * c->f) * ((MX_BN_DGRAD1 + 127) / 128) * MX_CHUNK;
    case MOE_MX_SCALES_W2C:   // W2 read as [d (K), f (N)]: tiles of MX_BN_DGRAD2 columns of f
      return static_cast<size_t>(c->E) * ((c->f + MX_BN_DGRAD2 - 1) / MX_BN_DGRAD2) *
             mx_kch(c->d) * ((MX_BN_DGRAD2 + 127) / 128) * MX_CHUNK;
    case MOE_MX_SCALES_TOK_D: return static_cast<size_t>(mx_tok_scale_bytes(N, c->E, c->d));
    case MOE_MX_SCALES_TOK_F: return static_cast<size_t>(mx_tok_scale_bytes(N, c->E, c->f));
    case MOE_MX_SCALES_TOK_2F: return static_cast<size_t>(mx_tok_scale_bytes(N, c->E, 2 * c->f));
    default: return 0;
  }
}

int moe_quantize_mxfp8(const void* x, int64_t rows, int32_t cols, uint8_t* q, uint8_t* scales,
                       void* stream) {
  if (rows < 0 || cols < 0)
    return fail(MOE_ERR_INVALID_ARG, "rows=%lld cols=%d", static_cast<long long>(rows), cols);
  if (cols % 32) return fail(MOE_ERR_UNSUPPORTED, "cols must be a multiple of 32 (MXFP8 blocks)");
  MOE_TRY(check_ptr(x, "x", true));
  MOE_TRY(check_ptr(q, "q", true));
  MOE_TRY(validate_ptr(scales, "scales", true));
  return launch_mx_quantize(x, rows, cols, q, scales, S(stream));
}

int moe_mxfp8_pack_expert_scales(const moe_cfg* c, const uint8_t* W1_s, const uint8_t* W2_s,
                                 uint8_t* W1_sp, uint8_t* W2_sp, void* stream) {
  MOE_TRY(check_mx_cfg(c));
  MOE_TRY(validate_ptr(W1_s, "W1_s", true));
  MOE_TRY(validate_ptr(W2_s, "W2_s", true));
  MOE_TRY(check_ptr(W1_sp, "W1_sp", true));
  MOE_TRY(check_ptr(W2_sp, "W2_sp", true));
  cudaStream_t st = S(stream);
  MOE_TRY(launch_mx_pack_weight_scales(W1_s, c->E, 2 * c->f, c->d, c->f, W1_sp, st));
  return launch_mx_pack_weight_scales(W2_s, c->E, c->d, c->f, 0, W2_sp, st);
}

int moe_permute_quantize_mxfp8(const moe_cfg* c, const void* x, const int32_t* slot_of_pair,
                               const int32_t* offsets, uint8_t* x_perm_q, uint8_t* x_perm_s,
                               void* stream) {
  MOE_TRY(check_mx_cfg(c));
  MOE_TRY(check_ptr(x, "x", true));
  MOE_TRY(check_ptr(slot_of_pair, "slot_of_pair", true));
  MOE_TRY(check_ptr(offsets, "offsets", true));
  MOE_TRY(check_ptr(x_perm_q, "x_perm_q", true));
  MOE_TRY(check_ptr(x_perm_s, "x_perm_s", true));
  if (c->T == 0) return MOE_OK;
  return launch_permute_quant_mx(x, slot_of_pair, offsets, x_perm_q, x_perm_s, c->T, c->d, c->k,
                                 c->E, S(stream));
}

int moe_grouped_swiglu_fwd_mxfp8(const moe_cfg* c, const uint8_t* x_perm_q,
                                 const uint8_t* x_perm_s, const int32_t* offsets,
                                 const uint8_t* W1_q, const uint8_t* W1_sp, const uint8_t* W2_q,
                                 const uint8_t* W2_sp, void* h, void* act, uint8_t* h_q,
                                 uint8_t* h_s, void* y_perm, void* stream) {
  MOE_TRY(check_mx_cfg(c));
  const struct { const void* p; const char* n; } req[] = {
      {x_perm_q, "x_perm_q"}, {x_perm_s, "x_perm_s"}, {offsets, "offsets"}, {W1_q, "W1_q"},
      {W1_sp, "W1_sp"},       {W2_q, "W2_q"},         {W2_sp, "W2_sp"},     {h_q, "h_q"},
      {h_s, "h_s"},           {y_perm, "y_perm"}};
  for (const auto& r : req) MOE_TRY(check_ptr(r.p, r.n, true));
  MOE_TRY(check_ptr(h, "h", false));
  MOE_TRY(check_ptr(act, "act", false));
  const int64_t N = Nrows(c);
  if (N == 0) return MOE_OK;
  return ffn_fwd_mx_impl(c, offsets, N, x_perm_q, x_perm_s, W1_q, W1_sp, W2_q, W2_sp, h, act, h_q,
                         h_s, y_perm, S(stream));
}

// MXFP8 data gradients of the routed experts: dy_perm quantised along d (rows in expert order),
// fc2's data gradient with the SwiGLU backward ([da | du] in bf16 when dH1 is given, and as
// MXFP8 codes along 2f), fc1's data gradient.  The weights are the column-blocked copies, read in
// their stored layouts (MN-major).
static int dgrad_mx_impl(const moe_cfg* c, const int32_t* offsets, int64_t N, const void* dy_perm,
                         const void* act, const uint8_t* W1c_q, const uint8_t* W1c_sp,
                         const uint8_t* W2c_q, const uint8_t* W2c_sp, uint8_t* dy_q,
                         uint8_t* dy_s, void* dH1, uint8_t* dH1_q, uint8_t* dH1_s, void* dx_perm,
                         cudaStream_t st) {
  const int d = c->d, f = c->f, E = c->E;
  MOE_TRY(launch_permute_quant_mx(dy_perm, nullptr, offsets, dy_q, dy_s, static_cast<int>(N), d, 1,
                                  E, st));
  GemmDesc a = desc0();
  a.name = "gemm_fc2_dgrad_mxfp8";
  a.sched = RAGGED_M;
  a.epi = EPI_SWIGLU_BWD;
  a.G = E;
  a.offsets = offsets;
  a.M = static_cast<int>(N);
  a.N = f;
  a.K = d;
  a.A = opnd(dy_q, N, d, false);
  a.B = opnd(W2c_q, static_cast<int64_t>(E) * d, f, true);
  a.b_group_rows = d;
  a.f = f;
  a.out = dH1;
  a.ldo = 2 * f;
  a.aux = act;
  a.ld_aux = 2 * f;
  a.fp8 = true;
  a.mx = true;
  a.sfa = dy_s;
  a.sfb = W2c_sp;
  a.q_out = dH1_q;
  a.q_sf = dH1_s;
  MOE_TRY(gemm_tc(a, st));
  GemmDesc b = desc0();
  b.name = "gemm_fc1_dgrad_mxfp8";
  b.sched = RAGGED_M;
  b.epi = EPI_STORE;
  b.G = E;
  b.offsets = offsets;
  b.M = static_cast<int>(N);
  b.N = d;
  b.K = 2 * f;
  b.A = opnd(dH1_q, N, 2 * f, false);
  b.B = opnd(W1c_q, static_cast<int64_t>(E) * 2 * f, d, true);
  b.b_group_rows = 2 * f;
  b.out = dx_perm;
  b.ldo = d;
  b.fp8 = true;
  b.mx = true;
  b.sfa = dH1_s;
  b.sfb = W1c_sp;
  return gemm_tc(b, st);
}

// The routed experts' backward with MXFP8 data gradients and bf16 weight gradients: dy quantised;
// fc2's data gradient + SwiGLU backward (dH1 in bf16 and MXFP8); fc2's weight gradient from the
// bf16 dy_perm and h; fc1's data gradient on the MXFP8 dH1 (dx_perm may alias dy_perm: it is
// written after fc2's weight gradient has read it); fc1's weight gradient from the bf16 dH1 and
// x_perm.
// One expert weight gradient on token-blocked MXFP8 operands: out[e] = dec(A_e)^T . dec(B_e),
// A [N, M] and B [N, C] codes (MN-major: the tokens are the reduction dimension).
static int wgrad_mx_gemm(const moe_cfg* c, const int32_t* offsets, int64_t N, const uint8_t* aq,
                         const uint8_t* as, int M, const uint8_t* bq, const uint8_t* bs, int C,
                         const int32_t* cbase, float* out, int* ctr, const char* name,
                         cudaStream_t st) {
  GemmDesc w = desc0();
  w.name = name;
  w.sched = RAGGED_K;
  w.epi = EPI_F32;
  w.G = c->E;
  w.offsets = offsets;
  w.M = M;
  w.N = C;
  w.K = static_cast<int>(N);
  w.A = opnd(aq, N, M, true);
  w.B = opnd(bq, N, C, true);
  w.out = out;
  w.ldo = C;
  w.out_group_stride = static_cast<int64_t>(M) * C;
  w.tile_ctr = ctr;
  w.fp8 = true;
  w.mx = true;
  w.sfa = as;
  w.sfb = bs;
  w.mx_cbase = cbase;
  return gemm_tc(w, st);
}

// fc2's (dW2 = dy^T h) or fc1's (dW1 = [da | du]^T x_perm) weight gradient in MXFP8: both operands
// quantised along the tokens inside the expert segments, then the block-scaled product.
static int wgrad2_mx(const moe_cfg* c, const int32_t* offsets, int64_t N, const void* dy_perm,
                     const void* h, float* dW2, const WgMxWs& w, int* ctr, cudaStream_t st) {
  const int E = c->E, d = c->d, f = c->f;
  MOE_TRY(launch_mx_quantize_tokens(dy_perm, N, d, offsets, E, w.dy_q, w.dy_s, w.cbase, st));
  MOE_TRY(launch_mx_quantize_tokens(h, N, f, offsets, E, w.h_q, w.h_s, w.cbase, st));
  return wgrad_mx_gemm(c, offsets, N, w.dy_q, w.dy_s, d, w.h_q, w.h_s, f, w.cbase, dW2, ctr,
                       "gemm_fc2_wgrad_mxfp8", st);
}
static int wgrad1_mx(const moe_cfg* c, const int32_t* offsets, int64_t N, const void* dH1,
                     const void* x_perm, float* dW1, const WgMxWs& w, int* ctr, cudaStream_t st) {
  const int E = c->E, d = c->d, f = c->f;
  MOE_TRY(launch_mx_quantize_tokens(dH1, N, 2 * f, offsets, E, w.dH1_q, w.dH1_s, w.cbase, st));
  MOE_TRY(launch_mx_quantize_tokens(x_perm, N, d, offsets, E, w.x_q, w.x_s, w.cbase, st));
  return wgrad_mx_gemm(c, offsets, N, w.dH1_q, w.dH1_s, 2 * f, w.x_q, w.x_s, d, w.cbase, dW1, ctr,
                       "gemm_fc1_wgrad_mxfp8", st);
}

static int ffn_bwd_mx_impl(const moe_cfg* c, const int32_t* offsets, int64_t N, const void* x_perm,
                           const void* act, const void* h, const void* dy_perm, void* dH1,
                           void* dx_perm, float* dW1, float* dW2, int* sched, cudaStream_t st,
                           const moe_mxfp8_dgrad* m, bool dy_quantised = false) {
  const int d = c->d, f = c->f, E = c->E;
  if (!dy_quantised)   // else the layer's combine backward wrote dy_perm's codes and scales
    MOE_TRY(launch_permute_quant_mx(dy_perm, nullptr, offsets, m->dy_q, m->dy_s,
                                    static_cast<int>(N), d, 1, E, st));
  GemmDesc a = desc0();
  a.name = "gemm_fc2_dgrad_mxfp8";
  a.sched = RAGGED_M;
  a.epi = EPI_SWIGLU_BWD;
  a.G = E;
  a.offsets = offsets;
  a.M = static_cast<int>(N);
  a.N = f;
  a.K = d;
  a.A = opnd(m->dy_q, N, d, false);
  a.B = opnd(m->W2c_q, static_cast<int64_t>(E) * d, f, true);
  a.b_group_rows = d;
  a.f = f;
  a.out = dH1;
  a.ldo = 2 * f;
  a.aux = act;
  a.ld_aux = 2 * f;
  a.fp8 = true;
  a.mx = true;
  a.sfa = m->dy_s;
  a.sfb = m->W2c_sp;
  a.q_out = m->dH1_q;
  a.q_sf = m->dH1_s;
  MOE_TRY(gemm_tc(a, st));
  // MXFP8 weight gradients when the caller lends their scratch, else bf16 ones
  WgMxWs wm;
  if (m->wgrad_ws) {
    Carve cv(m->wgrad_ws);
    wm = carve_wgmx(cv, c);
    MOE_TRY(wgrad2_mx(c, offsets, N, dy_perm, h, dW2, wm, sched, st));
  } else {
    GemmDesc b = desc0();
    b.name = "gemm_fc2_wgrad";
    b.sched = RAGGED_K;
    b.epi = EPI_F32;
    b.G = E;
    b.offsets = offsets;
    b.M = d;
    b.N = f;
    b.K = static_cast<int>(N);
    b.A = opnd(dy_perm, N, d, true);
    b.B = opnd(h, N, f, true);
    b.out = dW2;
    b.ldo = f;
    b.out_group_stride = static_cast<int64_t>(d) * f;
    b.tile_ctr = sched;
    MOE_TRY(gemm_tc(b, st));
  }
  GemmDesc e = desc0();
  e.name = "gemm_fc1_dgrad_mxfp8";
  e.sched = RAGGED_M;
  e.epi = EPI_STORE;
  e.G = E;
  e.offsets = offsets;
  e.M = static_cast<int>(N);
  e.N = d;
  e.K = 2 * f;
  e.A = opnd(m->dH1_q, N, 2 * f, false);
  e.B = opnd(m->W1c_q, static_cast<int64_t>(E) * 2 * f, d, true);
  e.b_group_rows = 2 * f;
  e.out = dx_perm;
  e.ldo = d;
  e.fp8 = true;
  e.mx = true;
  e.sfa = m->dH1_s;
  e.sfb = m->W1c_sp;
  MOE_TRY(gemm_tc(e, st));
  if (m->wgrad_ws) return wgrad1_mx(c, offsets, N, dH1, x_perm, dW1, wm, sched + 4, st);
  GemmDesc w = desc0();
  w.name = "gemm_fc1_wgrad";
  w.sched = RAGGED_K;
  w.epi = EPI_F32;
  w.G = E;
  w.offsets = offsets;
  w.M = 2 * f;
  w.N = d;
  w.K = static_cast<int>(N);
  w.A = opnd(dH1, N, 2 * f, true);
  w.B = opnd(x_perm, N, d, true);
  w.out = dW1;
  w.ldo = d;
  w.out_group_stride = static_cast<int64_t>(2) * f * d;
  w.tile_ctr = sched + 4;
  return gemm_tc(w, st);
}

int moe_mxfp8_prepare_dgrad_weights(const moe_cfg* c, const void* W1, const void* W2,
                                    uint8_t* W1c_q, uint8_t* W1c_s, uint8_t* W1c_sp,
                                    uint8_t* W2c_q, uint8_t* W2c_s, uint8_t* W2c_sp, void* stream) {
  MOE_TRY(check_mx_cfg(c));
  const struct { const void* p; const char* n; } req[] = {
      {W1, "W1"},       {W2, "W2"},         {W1c_q, "W1c_q"}, {W1c_s, "W1c_s"},
      {W1c_sp, "W1c_sp"}, {W2c_q, "W2c_q"}, {W2c_s, "W2c_s"}, {W2c_sp, "W2c_sp"}};
  for (const auto& r : req) MOE_TRY(check_ptr(r.p, r.n, true));
  cudaStream_t st = S(stream);
  const int E = c->E, d = c->d, f = c->f;
  // W1 [E, 2f, d] in 32-row blocks along 2f; its columns (d) are the B-rows of fc1's data gradient
  MOE_TRY(launch_mx_quantize_cols(W1, E, 2 * f, d, W1c_q, W1c_s, st));
  MOE_TRY(launch_mx_pack_weight_scales(W1c_s, E, d, 2 * f, 0, W1c_sp, st, MX_BN_DGRAD1, 1));
  // W2 [E, d, f] in 32-row blocks along d; its columns (f) are the B-rows of fc2's data gradient
  MOE_TRY(launch_mx_quantize_cols(W2, E, d, f, W2c_q, W2c_s, st));
  return launch_mx_pack_weight_scales(W2c_s, E, f, d, 0, W2c_sp, st, MX_BN_DGRAD2, 1);
}

int moe_mxfp8_quantize_tokens(const moe_cfg* c, const void* x, int32_t cols,
                              const int32_t* offsets, uint8_t* q, uint8_t* s, int32_t* cbase,
                              void* stream) {
  MOE_TRY(check_mx_cfg(c));
  if (cols <= 0 || cols % 32)
    return fail(MOE_ERR_UNSUPPORTED, "cols=%d: a positive multiple of 32 is needed", cols);
  const struct { const void* p; const char* n; } req[] = {
      {x, "x"}, {offsets, "offsets"}, {q, "q"}, {s, "s"}, {cbase, "cbase"}};
  for (const auto& r : req) MOE_TRY(check_ptr(r.p, r.n, true));
  return launch_mx_quantize_tokens(x, Nrows(c), cols, offsets, c->E, q, s, cbase, S(stream));
}

int moe_grouped_swiglu_wgrad_mxfp8(const moe_cfg* c, const int32_t* offsets, const void* x_perm,
                                   const void* h, const void* dy_perm, const void* dH1,
                                   float* dW1, float* dW2, void* ws, size_t ws_bytes,
                                   void* stream) {
  MOE_TRY(check_mx_cfg(c));
  const struct { const void* p; const char* n; } req[] = {
      {offsets, "offsets"}, {x_perm, "x_perm"}, {h, "h"}, {dy_perm, "dy_perm"},
      {dH1, "dH1"},         {dW1, "dW1"},       {dW2, "dW2"}};
  for (const auto& r : req) MOE_TRY(check_ptr(r.p, r.n, true));
  MOE_TRY(check_ws(c, MOE_WS_WGRAD_MXFP8, ws, ws_bytes));
  Carve cv(ws);
  const WgMxWs w = carve_wgmx(cv, c);
  cudaStream_t st = S(stream);
  const int64_t N = Nrows(c);
  if (N == 0) {   // no rows: every expert's weight gradients are zero blocks
    if (cudaMemsetAsync(dW1, 0, sizeof(float) * c->E * 2 * c->f * c->d, st) != cudaSuccess ||
        cudaMemsetAsync(dW2, 0, sizeof(float) * c->E * c->d * c->f, st) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "cudaMemsetAsync failed");
    return MOE_OK;
  }
  MOE_TRY(wgrad2_mx(c, offsets, N, dy_perm, h, dW2, w, w.sched, st));
  return wgrad1_mx(c, offsets, N, dH1, x_perm, dW1, w, w.sched + 4, st);
}

int moe_grouped_swiglu_dgrad_mxfp8(const moe_cfg* c, const void* dy_perm, const int32_t* offsets,
                                   const void* act, const uint8_t* W1c_q, const uint8_t* W1c_sp,
                                   const uint8_t* W2c_q, const uint8_t* W2c_sp, uint8_t* dy_q,
                                   uint8_t* dy_s, void* dH1, uint8_t* dH1_q, uint8_t* dH1_s,
                                   void* dx_perm, void* stream) {
  MOE_TRY(check_mx_cfg(c));
  const struct { const void* p; const char* n; } req[] = {
      {dy_perm, "dy_perm"}, {offsets, "offsets"}, {act, "act"},     {W1c_q, "W1c_q"},
      {W1c_sp, "W1c_sp"},   {W2c_q, "W2c_q"},     {W2c_sp, "W2c_sp"}, {dy_q, "dy_q"},
      {dy_s, "dy_s"},       {dH1_q, "dH1_q"},     {dH1_s, "dH1_s"},  {dx_perm, "dx_perm"}};
  for (const auto& r : req) MOE_TRY(check_ptr(r.p, r.n, true));
  MOE_TRY(check_ptr(dH1, "dH1", false));
  const int64_t N = Nrows(c);
  if (N == 0) return MOE_OK;
  return dgrad_mx_impl(c, offsets, N, dy_perm, act, W1c_q, W1c_sp, W2c_q, W2c_sp, dy_q, dy_s, dH1,
                       dH1_q, dH1_s, dx_perm, S(stream));
}

int moe_grouped_swiglu_bwd_fp8(const moe_cfg* c, const uint8_t* x_perm_q, const float* x_scale,
                               const int32_t* offsets, const uint8_t* W1_q, const float* W1_scale,
                               const uint8_t* W2_q, const float* W2_scale, const void* act,
                               const uint8_t* h_q, const float* h_scale, const void* dy_perm,
                               uint8_t* dy_q, float* dy_scale, float* dy_amax, void* dH1,
                               uint8_t* dH1_q, float* dH1_scale, float* dH1_amax, void* dx_perm,
                               float* dW1, float* dW2, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(c));
  if (c->dtype != MOE_DTYPE_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "the FP8 path reads and writes bf16 activations (dtype bf16)");
  if (c->d % 16 || c->f % 16)
    return fail(MOE_ERR_UNSUPPORTED, "FP8 rows need d and f multiples of 16 (16-byte rows)");
  const struct { const void* p; const char* n; } req[] = {
      {x_perm_q, "x_perm_q"}, {x_scale, "x_scale"}, {offsets, "offsets"}, {W1_q, "W1_q"},
      {W1_scale, "W1_scale"}, {W2_q, "W2_q"}, {W2_scale, "W2_scale"}, {act, "act"},
      {h_q, "h_q"}, {h_scale, "h_scale"}, {dy_perm, "dy_perm"}, {dy_q, "dy_q"},
      {dy_scale, "dy_scale"}, {dy_amax, "dy_amax"}, {dH1, "dH1"}, {dH1_q, "dH1_q"},
      {dH1_scale, "dH1_scale"}, {dH1_amax, "dH1_amax"}, {dx_perm, "dx_perm"}, {dW1, "dW1"},
      {dW2, "dW2"}};
  for (const auto& r : req) MOE_TRY(check_ptr(r.p, r.n, true));
  MOE_TRY(check_ws(c, MOE_WS_FFN_BWD_FP8, ws, ws_bytes));
  cudaStream_t st = S(stream);
  const int64_t N = Nrows(c);
  const int d = c->d, f = c->f, E = c->E;
  if (N == 0) {
    if (cudaMemsetAsync(dW1, 0, sizeof(float) * E * 2 * f * d, st) != cudaSuccess ||
        cudaMemsetAsync(dW2, 0, sizeof(float) * E * d * f, st) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "cudaMemsetAsync failed");
    return MOE_OK;
  }
  Carve cv(ws);
  int* sched = static_cast<int*>(cv.take(2 * 4 * sizeof(int)));
  return ffn_bwd_fp8_impl(c, c->E, offsets, Nrows(c), c->f, x_perm_q, x_scale, W1_q, W1_scale, W2_q, W2_scale, act, h_q,
                          h_scale, dy_perm, dy_q, dy_scale, dy_amax, dH1, dH1_q, dH1_scale,
                          dH1_amax, dx_perm, dW1, dW2, sched, st);
}

int moe_unpermute_combine(const moe_cfg* c, const void* y_perm, const float* gate,
                          const int32_t* slot_of_pair, const void* shared_out,
                          const float* shared_coef, void* y, void* stream) {
  MOE_TRY(check_cfg(c));
  MOE_TRY(check_ptr(y_perm, "y_perm", true));
  MOE_TRY(check_ptr(gate, "gate", true));
  MOE_TRY(check_ptr(slot_of_pair, "slot_of_pair", true));
  MOE_TRY(check_ptr(shared_out, "shared_out", false));
  MOE_TRY(check_ptr(shared_coef, "shared_coef", false));
  MOE_TRY(check_ptr(y, "y", true));
  return launch_combine(c->dtype, y_perm, gate, slot_of_pair, shared_out, shared_coef, y, c->T,
                        c->d, c->k, S(stream));
}

int moe_unpermute_combine_bwd(const moe_cfg* c, const void* dy, const void* y_perm,
                              const float* gate, const int32_t* slot_of_pair,
                              const void* shared_out, const float* shared_coef, void* dy_perm,
                              float* dgate, void* dshared, float* dcoef, void* stream) {
  MOE_TRY(check_cfg(c));
  MOE_TRY(check_ptr(dy, "dy", true));
  MOE_TRY(check_ptr(y_perm, "y_perm", true));
  MOE_TRY(check_ptr(gate, "gate", true));
  MOE_TRY(check_ptr(slot_of_pair, "slot_of_pair", true));
  MOE_TRY(check_ptr(shared_out, "shared_out", false));
  MOE_TRY(check_ptr(shared_coef, "shared_coef", false));
  MOE_TRY(check_ptr(dy_perm, "dy_perm", true));
  MOE_TRY(check_ptr(dgate, "dgate", true));
  MOE_TRY(check_ptr(dshared, "dshared", false));
  MOE_TRY(check_ptr(dcoef, "dcoef", false));
  return launch_combine_bwd(c->dtype, dy, y_perm, gate, slot_of_pair, shared_out, shared_coef,
                            dy_perm, dgate, dshared, shared_coef ? dcoef : nullptr, c->T, c->d,
                            c->k, S(stream));
}

int moe_router_aux_loss(const moe_cfg* c, const float* logits, const int32_t* counts,
                        float* aux_loss, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_cfg(c));
  if (!(c->aux_coeff > 0.0f)) return fail(MOE_ERR_INVALID_ARG, "aux_coeff is 0: no loss to compute");
  MOE_TRY(check_ptr(logits, "logits", true));
  MOE_TRY(check_ptr(counts, "counts", true));
  MOE_TRY(check_ptr(aux_loss, "aux_loss", true));
  MOE_TRY(check_ws(c, MOE_WS_ROUTE, ws, ws_bytes));
  cudaStream_t st = S(stream);
  if (c->T == 0)
    return cudaMemsetAsync(aux_loss, 0, sizeof(float), st) == cudaSuccess
               ? MOE_OK : fail(MOE_ERR_CUDA, "cudaMemsetAsync failed");
  Carve cv(ws);
  RouteWs w = carve_route(cv, c);
  return launch_aux_loss(logits, counts, c->T, c->E, c->k, c->score_fn, c->aux_coeff, w.aux,
                         aux_loss, st);
}

int moe_expert_bias_update(const moe_cfg* c, const int32_t* counts, float* e_bias, float rate,
                           void* stream) {
  MOE_TRY(check_cfg(c));
  MOE_TRY(check_ptr(counts, "counts", true));
  MOE_TRY(check_ptr(e_bias, "e_bias", true));
  if (!(rate == rate) || rate > 3.0e38f || rate < -3.0e38f)
    return fail(MOE_ERR_INVALID_ARG, "rate must be finite");
  if (c->T == 0) return MOE_OK;   // no batch: no load to correct
  return launch_bias_update(counts, e_bias, c->T, c->k, c->E, rate, S(stream));
}

static int check_fp8_experts(const moe_cfg* c, const moe_fp8_experts* q) {
  if (c->dtype != MOE_DTYPE_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "the FP8 experts read and write bf16 activations (dtype bf16)");
  if (c->d % 16 || c->f % 16)
    return fail(MOE_ERR_UNSUPPORTED, "FP8 rows need d and f multiples of 16 (16-byte rows)");
  MOE_TRY(check_ptr(q->W1_q, "fp8.W1_q", true));
  MOE_TRY(check_ptr(q->W1_scale, "fp8.W1_scale", true));
  MOE_TRY(check_ptr(q->W2_q, "fp8.W2_q", true));
  MOE_TRY(check_ptr(q->W2_scale, "fp8.W2_scale", true));
  MOE_TRY(check_ptr(q->x_perm_q, "fp8.x_perm_q", true));
  MOE_TRY(check_ptr(q->h_q, "fp8.h_q", true));
  MOE_TRY(check_ptr(q->scales, "fp8.scales", true));
  const bool sq = c->f_shared > 0 && q->Ws1_q;   // the shared expert in FP8 too
  if (sq && c->f_shared % 16)
    return fail(MOE_ERR_UNSUPPORTED, "an FP8 shared expert needs f_shared a multiple of 16");
  MOE_TRY(check_ptr(q->Ws1_scale, "fp8.Ws1_scale", sq));
  MOE_TRY(check_ptr(q->Ws2_q, "fp8.Ws2_q", sq));
  MOE_TRY(check_ptr(q->Ws2_scale, "fp8.Ws2_scale", sq));
  MOE_TRY(check_ptr(q->x_q, "fp8.x_q", sq));
  MOE_TRY(check_ptr(q->s_h_q, "fp8.s_h_q", sq));
  return MOE_OK;
}

static bool shared_fp8(const moe_cfg* c, const moe_fp8_experts* q) {
  return q && c->f_shared > 0 && q->Ws1_q;
}

static int check_saved(const moe_cfg* c, const moe_saved* s, bool fp8 = false,
                       bool need_act = true) {
  if (!s) return fail(MOE_ERR_INVALID_ARG, "saved is NULL");
  MOE_TRY(check_ptr(s->logits, "saved.logits", true));
  MOE_TRY(check_ptr(s->idx, "saved.idx", true));
  MOE_TRY(check_ptr(s->gate, "saved.gate", true));
  MOE_TRY(check_ptr(s->counts, "saved.counts", true));
  MOE_TRY(check_ptr(s->offsets, "saved.offsets", true));
  MOE_TRY(check_ptr(s->slot_of_pair, "saved.slot_of_pair", true));
  MOE_TRY(check_ptr(s->token_of_slot, "saved.token_of_slot", true));
  MOE_TRY(check_ptr(s->x_perm, "saved.x_perm", !fp8 && !permute_fused(c)));
  MOE_TRY(check_ptr(s->act, "saved.act", need_act));
  MOE_TRY(check_ptr(s->h, "saved.h", need_act));
  MOE_TRY(check_ptr(s->y_perm, "saved.y_perm", true));
  const bool sh = c->f_shared > 0;
  MOE_TRY(check_ptr(s->s_act, "saved.s_act", sh));
  MOE_TRY(check_ptr(s->s_h, "saved.s_h", sh));
  MOE_TRY(check_ptr(s->s_out, "saved.s_out", sh));
  MOE_TRY(check_ptr(s->s_coef, "saved.s_coef", c->shared_gate != 0));
  MOE_TRY(check_ptr(s->aux_loss, "saved.aux_loss", c->aux_coeff > 0.0f));
  return MOE_OK;
}

static int check_mx_experts(const moe_cfg* c, const moe_mxfp8_experts* m) {
  MOE_TRY(check_mx_cfg(c));
  const struct { const void* p; const char* n; } req[] = {
      {m->W1_q, "mx.W1_q"},         {m->W1_sp, "mx.W1_sp"}, {m->W2_q, "mx.W2_q"},
      {m->W2_sp, "mx.W2_sp"},       {m->x_perm_q, "mx.x_perm_q"},
      {m->x_perm_s, "mx.x_perm_s"}, {m->h_q, "mx.h_q"},     {m->h_s, "mx.h_s"}};
  for (const auto& r : req) MOE_TRY(check_ptr(r.p, r.n, true));
  return MOE_OK;
}

// The layer forward; with q the routed experts run on E4M3 operands (q's weights and buffers),
// with mx on MXFP8 operands.
static int layer_fwd_impl(const moe_cfg* c, const void* x, const void* W_r, const float* b_r,
                          const void* W1, const void* W2, const moe_fp8_experts* q,
                          const void* Ws1, const void* Ws2, const void* w_sg, void* y,
                          const moe_saved* s, void* ws, size_t ws_bytes, void* stream,
                          const moe_side_stream* side_in, const moe_mxfp8_experts* mx = nullptr) {
  MOE_TRY(check_cfg(c));
  MOE_TRY(check_side(side_in, stream));
  MOE_TRY(check_ptr(x, "x", true));
  MOE_TRY(check_ptr(W_r, "W_r", true));
  MOE_TRY(check_ptr(b_r, "b_r", false));
  MOE_TRY(check_ptr(W1, "W1", !q && !mx));
  MOE_TRY(check_ptr(W2, "W2", !q && !mx));
  if (q) MOE_TRY(check_fp8_experts(c, q));
  if (mx) MOE_TRY(check_mx_experts(c, mx));
  const bool sh = c->f_shared > 0, gt = c->shared_gate != 0;
  const bool sq = shared_fp8(c, q);
  MOE_TRY(check_ptr(Ws1, "Ws1", sh && !sq));
  MOE_TRY(check_ptr(Ws2, "Ws2", sh && !sq));
  MOE_TRY(check_ptr(w_sg, "w_sg", gt));
  MOE_TRY(check_ptr(y, "y", true));
  MOE_TRY(check_saved(c, s, q != nullptr || mx != nullptr, mx == nullptr));
  MOE_TRY(check_ws(c, MOE_WS_LAYER_FWD, ws, ws_bytes));
  cudaStream_t st = S(stream);
  if (c->T == 0) {
    if (cudaMemsetAsync(s->counts, 0, sizeof(int32_t) * c->E, st) != cudaSuccess ||
        cudaMemsetAsync(s->offsets, 0, sizeof(int32_t) * (c->E + 1), st) != cudaSuccess ||
        (c->aux_coeff > 0.0f && cudaMemsetAsync(s->aux_loss, 0, sizeof(float), st) != cudaSuccess))
      return fail(MOE_ERR_CUDA, "cudaMemsetAsync failed");
    return MOE_OK;
  }
  Carve cv(ws);
  RouteWs w = carve_route(cv, c);
  // The shared expert (and its gate) needs only x: with a side stream it runs there while the
  // routed path (routing, permute, grouped SwiGLU) runs on `st`; the combine waits for both.
  SideStream side_ss;
  SideStream* side = nullptr;
  if (sh && side_in) {
    side_ss = side_of(side_in);
    side = &side_ss;
  }
  auto shared_fwd = [&](cudaStream_t ss) -> int {
    if (gt) MOE_TRY(launch_shared_gate(c->dtype, x, w_sg, s->s_coef, c->T, c->d, ss));
    if (sq)
      return ffn_fwd_fp8_impl(c, 1, nullptr, c->T, c->f_shared, q->x_q, q->scales + 0, q->Ws1_q,
                              q->Ws1_scale, q->Ws2_q, q->Ws2_scale, s->s_h, s->s_act, q->s_h_q,
                              q->scales + 8, q->scales + 9, s->s_out, ss);
    return ffn_fwd_impl(c, 1, nullptr, c->T, c->f_shared, x, Ws1, Ws2, s->s_h, s->s_act,
                        s->s_out, ss);
  };
  MOE_TRY(route_impl(c, x, W_r, b_r, nullptr, s->logits, s->idx, s->gate, s->counts, s->offsets,
                     s->slot_of_pair, s->token_of_slot, w, st));
  // FP8: x permuted and quantised in one pass ("Megatron-Bridge 深度剖析", §FP8 训练), also in
  // token order for an FP8 shared expert -- before the side stream forks, which reads those codes
  if (q)
    MOE_TRY(launch_permute_quant_e4m3(x, s->slot_of_pair, q->x_perm_q, sq ? q->x_q : nullptr,
                                      q->scales + 0, q->scales + 1, c->T, c->d, c->k, st));
  // MXFP8: x permuted and block-quantised in one pass, its scales in the row tiles of the routing
  // (and the permuted bf16 rows into saved.x_perm when given, for a bf16 backward)
  if (mx)
    MOE_TRY(launch_permute_quant_mx(x, s->slot_of_pair, s->offsets, mx->x_perm_q, mx->x_perm_s,
                                    c->T, c->d, c->k, c->E, st, s->x_perm));
  if (side) {
    if (cudaEventRecord(side->fork, st) != cudaSuccess ||
        cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "forking the shared expert onto the side stream failed");
    MOE_TRY(shared_fwd(side->s));
    if (cudaEventRecord(side->join, side->s) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "recording the shared expert's completion failed");
  }
  if (c->aux_coeff > 0.0f)
    MOE_TRY(launch_aux_loss(s->logits, s->counts, c->T, c->E, c->k, c->score_fn, c->aux_coeff,
                            w.aux, s->aux_loss, st));
  if (q) {
    // E4M3 experts on the codes made above
    MOE_TRY(ffn_fwd_fp8_impl(c, c->E, s->offsets, Nrows(c), c->f, q->x_perm_q, q->scales + 0, q->W1_q, q->W1_scale,
                             q->W2_q, q->W2_scale, s->h, s->act, q->h_q, q->scales + 2,
                             q->scales + 3, s->y_perm, st));
  } else if (mx) {
    // MXFP8 experts; bf16 h and [a | u] written only into the saved buffers given (what the bf16
    // backward reads)
    MOE_TRY(ffn_fwd_mx_impl(c, s->offsets, Nrows(c), mx->x_perm_q, mx->x_perm_s, mx->W1_q,
                            mx->W1_sp, mx->W2_q, mx->W2_sp, s->h, s->act, mx->h_q, mx->h_s,
                            s->y_perm, st));
  } else if (permute_fused(c)) {
    // "Megatron-Bridge 深度剖析", §Permute Fusion: fc1 gathers its rows from x by token_of_slot
    MOE_TRY(ffn_fwd_impl(c, c->E, s->offsets, Nrows(c), c->f, x, W1, W2, s->h, s->act,
                         s->y_perm, st, s->token_of_slot, c->T));
  } else {
    MOE_TRY(launch_permute(c->dtype, x, s->slot_of_pair, s->x_perm, c->T, c->d, c->k, st));
    MOE_TRY(ffn_fwd_impl(c, c->E, s->offsets, Nrows(c), c->f, s->x_perm, W1, W2, s->h, s->act,
                         s->y_perm, st));
  }
  if (side) {
    if (cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "joining the side stream failed");
  } else if (sh) {
    MOE_TRY(shared_fwd(st));
  }
  return launch_combine(c->dtype, s->y_perm, s->gate, s->slot_of_pair, sh ? s->s_out : nullptr,
                        gt ? s->s_coef : nullptr, y, c->T, c->d, c->k, st);
}

// The layer backward; with q the routed experts' backward runs on E4M3 operands.
static int layer_bwd_impl(const moe_cfg* c, const void* dy, const void* x, const void* W_r,
                          const void* W1, const void* W2, const moe_fp8_experts* q,
                          const void* Ws1, const void* Ws2, const void* w_sg, const moe_saved* s,
                          void* dx, float* dW_r, float* dW1, float* dW2, float* dWs1,
                          float* dWs2, float* dw_sg, void* ws, size_t ws_bytes, void* stream,
                          const moe_side_stream* side_in, const moe_mxfp8_dgrad* mxd = nullptr) {
  MOE_TRY(check_cfg(c));
  MOE_TRY(check_side(side_in, stream));
  const bool sh = c->f_shared > 0, gt = c->shared_gate != 0;
  MOE_TRY(check_ptr(dy, "dy", true));
  MOE_TRY(check_ptr(x, "x", true));
  MOE_TRY(check_ptr(W_r, "W_r", true));
  MOE_TRY(check_ptr(W1, "W1", !q && !mxd));
  MOE_TRY(check_ptr(W2, "W2", !q && !mxd));
  if (q) MOE_TRY(check_fp8_experts(c, q));
  if (mxd) {
    MOE_TRY(check_mx_cfg(c));
    if (permute_fused(c))
      return fail(MOE_ERR_UNSUPPORTED, "the MXFP8 backward reads saved.x_perm (no fused permute)");
    const struct { const void* p; const char* n; } req[] = {
        {mxd->W1c_q, "mxd.W1c_q"}, {mxd->W1c_sp, "mxd.W1c_sp"}, {mxd->W2c_q, "mxd.W2c_q"},
        {mxd->W2c_sp, "mxd.W2c_sp"}, {mxd->dy_q, "mxd.dy_q"},  {mxd->dy_s, "mxd.dy_s"},
        {mxd->dH1_q, "mxd.dH1_q"}, {mxd->dH1_s, "mxd.dH1_s"}};
    for (const auto& r : req) MOE_TRY(check_ptr(r.p, r.n, true));
    if (mxd->wgrad_ws) MOE_TRY(check_ws(c, MOE_WS_WGRAD_MXFP8, mxd->wgrad_ws, mxd->wgrad_ws_bytes));
  }
  const bool sq = shared_fp8(c, q);
  MOE_TRY(check_ptr(Ws1, "Ws1", sh && !sq));
  MOE_TRY(check_ptr(Ws2, "Ws2", sh && !sq));
  MOE_TRY(check_ptr(w_sg, "w_sg", gt));
  MOE_TRY(check_saved(c, s, q != nullptr));
  MOE_TRY(check_ptr(dx, "dx", true));
  MOE_TRY(check_ptr(dW_r, "dW_r", true));
  MOE_TRY(check_ptr(dW1, "dW1", true));
  MOE_TRY(check_ptr(dW2, "dW2", true));
  MOE_TRY(check_ptr(dWs1, "dWs1", sh));
  MOE_TRY(check_ptr(dWs2, "dWs2", sh));
  MOE_TRY(check_ptr(dw_sg, "dw_sg", gt));
  MOE_TRY(check_ws(c, q ? MOE_WS_LAYER_BWD_FP8 : MOE_WS_LAYER_BWD, ws, ws_bytes));
  cudaStream_t st = S(stream);
  const int T = c->T, d = c->d, E = c->E, k = c->k;
  if (T == 0) {
    bool ok = cudaMemsetAsync(dW_r, 0, sizeof(float) * E * d, st) == cudaSuccess &&
              cudaMemsetAsync(dW1, 0, sizeof(float) * E * 2 * c->f * d, st) == cudaSuccess &&
              cudaMemsetAsync(dW2, 0, sizeof(float) * E * d * c->f, st) == cudaSuccess;
    if (sh)
      ok = ok && cudaMemsetAsync(dWs1, 0, sizeof(float) * 2 * c->f_shared * d, st) == cudaSuccess &&
           cudaMemsetAsync(dWs2, 0, sizeof(float) * d * c->f_shared, st) == cudaSuccess;
    if (gt) ok = ok && cudaMemsetAsync(dw_sg, 0, sizeof(float) * d, st) == cudaSuccess;
    return ok ? MOE_OK : fail(MOE_ERR_CUDA, "cudaMemsetAsync failed");
  }
  Carve cv(ws);
  BwdWs w = carve_bwd(cv, c);
  uint8_t* dy_q = q ? static_cast<uint8_t*>(cv.take(static_cast<size_t>(Nrows(c)) * d)) : nullptr;
  uint8_t* dH1_q =
      q ? static_cast<uint8_t*>(cv.take(static_cast<size_t>(Nrows(c)) * 2 * c->f)) : nullptr;
  uint8_t* ds_q = sq ? static_cast<uint8_t*>(cv.take(static_cast<size_t>(T) * d)) : nullptr;
  uint8_t* s_dH1_q =
      sq ? static_cast<uint8_t*>(cv.take(static_cast<size_t>(T) * 2 * c->f_shared)) : nullptr;
  // 1. combine backward (FP8: it also reduces the amax of dy_perm, and of the shared expert's
  // upstream gradient, as it stores them)
  if (q && (cudaMemsetAsync(q->scales + 5, 0, sizeof(float), st) != cudaSuccess ||
            (sq && cudaMemsetAsync(q->scales + 11, 0, sizeof(float), st) != cudaSuccess)))
    return fail(MOE_ERR_CUDA, "clearing the gradient amaxes failed");
  if (mxd)   // MXFP8 data gradients: dy_perm's codes come out of the same pass
    MOE_TRY(launch_combine_bwd_mx(dy, s->y_perm, s->gate, s->slot_of_pair, sh ? s->s_out : nullptr,
                                  gt ? s->s_coef : nullptr, w.dy_perm, w.dgate, w.dshared, w.dcoef,
                                  T, d, k, s->offsets, E, mxd->dy_q, mxd->dy_s, st));
  else
    MOE_TRY(launch_combine_bwd(c->dtype, dy, s->y_perm, s->gate, s->slot_of_pair,
                               sh ? s->s_out : nullptr, gt ? s->s_coef : nullptr, w.dy_perm,
                               w.dgate, w.dshared, w.dcoef, T, d, k, st,
                               q ? q->scales + 5 : nullptr, sq ? q->scales + 11 : nullptr));
  // 2.-6. The routed experts run on `st`; the shared expert and the router's backward (which
  // need only combine-backward outputs) run on the side stream, when given, concurrently; dx
  // waits for both.
  SideStream side_ss;
  SideStream* side = nullptr;
  if (side_in) {
    side_ss = side_of(side_in);
    side = &side_ss;
  }
  auto side_work = [&](cudaStream_t ss) -> int {
    // shared expert (one group of all T tokens)
    if (sq)
      MOE_TRY(ffn_bwd_fp8_impl(c, 1, nullptr, T, c->f_shared, q->x_q, q->scales + 0, q->Ws1_q,
                               q->Ws1_scale, q->Ws2_q, q->Ws2_scale, s->s_act, q->s_h_q,
                               q->scales + 8, w.dshared, ds_q, q->scales + 10, q->scales + 11,
                               w.s_dH1, s_dH1_q, q->scales + 12, q->scales + 13, w.dx_shared,
                               dWs1, dWs2, w.sched + 8, ss, true));
    else if (sh)
      MOE_TRY(ffn_bwd_impl(c, 1, nullptr, T, c->f_shared, x, Ws1, Ws2, s->s_act, s->s_h,
                           w.dshared, w.s_dH1, w.dx_shared, dWs1, dWs2, w.sched + 8, ss));
    // router: dlogits (+ shared gate dz in column E), with the balancing loss's gradient
    const int ldx = ext_cols(c);
    const bool aux = c->aux_coeff > 0.0f;
    const float aux_w = aux ? static_cast<float>(static_cast<double>(c->aux_coeff) * E /
                                                 (static_cast<double>(k) * T * T))
                            : 0.0f;
    MOE_TRY(launch_router_bwd(c->dtype, s->logits, s->idx, s->gate, w.dgate,
                              gt ? w.dcoef : nullptr, gt ? s->s_coef : nullptr, w.dl_ext, w.dz, T,
                              E, k, ldx, c->score_fn, c->renorm, aux ? s->counts : nullptr, aux_w,
                              ss));
    // dx_router = dlogits . W_r
    GemmDesc rd = desc0();
    rd.name = "gemm_router_dgrad";
    rd.sched = RAGGED_M;
    rd.epi = EPI_STORE;
    rd.G = 1;
    rd.M = T;
    rd.N = d;
    rd.K = E;
    rd.A = opnd(w.dl_ext, T, ldx, false);
    rd.B = opnd(W_r, E, d, true);
    rd.out = w.dx_router;
    rd.ldo = d;
    MOE_TRY(gemm(c, rd, ss));
    // [dW_r; dw_sg] = [dlogits | dz]^T . x, split over tokens, then a fixed-order sum
    const int mr = E + (gt ? 1 : 0);
    const int S_ = router_splits(c);
    GemmDesc rw = desc0();
    rw.name = "gemm_router_wgrad";
    rw.sched = RAGGED_K;
    rw.epi = EPI_F32;
    rw.G = S_;
    rw.M = mr;
    rw.N = d;
    rw.K = T;
    rw.A = opnd(w.dl_ext, T, ldx, true);
    rw.B = opnd(x, T, d, true);
    rw.out = w.part;
    rw.ldo = d;
    rw.out_group_stride = static_cast<int64_t>(mr) * d;
    rw.tile_ctr = w.sched + 16;
    MOE_TRY(gemm(c, rw, ss));
    return launch_split_reduce(w.part, S_, mr, d, dW_r, E, gt ? dw_sg : nullptr, ss);
  };
  if (side) {
    if (cudaEventRecord(side->fork, st) != cudaSuccess ||
        cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "forking onto the side stream failed");
    MOE_TRY(side_work(side->s));
    if (cudaEventRecord(side->join, side->s) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "recording the side stream's completion failed");
  }
  // routed experts (dx_perm overwrites dy_perm once it is no longer read)
  if (mxd)
    MOE_TRY(ffn_bwd_mx_impl(c, s->offsets, Nrows(c), s->x_perm, s->act, s->h, w.dy_perm, w.dH1,
                            w.dy_perm, dW1, dW2, w.sched, st, mxd, true));
  else if (q)
    MOE_TRY(ffn_bwd_fp8_impl(c, c->E, s->offsets, Nrows(c), c->f, q->x_perm_q, q->scales + 0, q->W1_q, q->W1_scale,
                             q->W2_q, q->W2_scale, s->act, q->h_q, q->scales + 2, w.dy_perm, dy_q,
                             q->scales + 4, q->scales + 5, w.dH1, dH1_q, q->scales + 6,
                             q->scales + 7, w.dy_perm, dW1, dW2, w.sched, st, true));
  else if (permute_fused(c))
    MOE_TRY(ffn_bwd_impl(c, E, s->offsets, Nrows(c), c->f, x, W1, W2, s->act, s->h, w.dy_perm,
                         w.dH1, w.dy_perm, dW1, dW2, w.sched, st, s->token_of_slot, T));
  else
    MOE_TRY(ffn_bwd_impl(c, E, s->offsets, Nrows(c), c->f, s->x_perm, W1, W2, s->act, s->h,
                         w.dy_perm, w.dH1, w.dy_perm, dW1, dW2, w.sched, st));
  if (side) {
    if (cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess)
      return fail(MOE_ERR_CUDA, "joining the side stream failed");
  } else {
    MOE_TRY(side_work(st));
  }
  // 7. dx = sum_j dx_perm[slot(t,j)] + dx_shared + dx_router + dz * w_sg
  return launch_gather_sum(c->dtype, w.dy_perm, s->slot_of_pair, sh ? w.dx_shared : nullptr,
                           w.dx_router, gt ? w.dz : nullptr, gt ? w_sg : nullptr, dx, T, d, k, st);
}

int moe_layer_fwd(const moe_cfg* c, const void* x, const void* W_r, const float* b_r,
                  const void* W1, const void* W2, const void* Ws1, const void* Ws2,
                  const void* w_sg, void* y, const moe_saved* s, void* ws, size_t ws_bytes,
                  void* stream, const moe_side_stream* side) {
  return layer_fwd_impl(c, x, W_r, b_r, W1, W2, nullptr, Ws1, Ws2, w_sg, y, s, ws, ws_bytes,
                        stream, side);
}

int moe_layer_fwd_mxfp8(const moe_cfg* c, const void* x, const void* W_r, const float* b_r,
                        const moe_mxfp8_experts* mx, const void* Ws1, const void* Ws2,
                        const void* w_sg, void* y, const moe_saved* saved, void* ws,
                        size_t ws_bytes, void* stream, const moe_side_stream* side) {
  if (!mx) return fail(MOE_ERR_INVALID_ARG, "mx is NULL");
  return layer_fwd_impl(c, x, W_r, b_r, nullptr, nullptr, nullptr, Ws1, Ws2, w_sg, y, saved, ws,
                        ws_bytes, stream, side, mx);
}

int moe_layer_fwd_fp8(const moe_cfg* c, const void* x, const void* W_r, const float* b_r,
                      const moe_fp8_experts* q, const void* Ws1, const void* Ws2,
                      const void* w_sg, void* y, const moe_saved* s, void* ws, size_t ws_bytes,
                      void* stream, const moe_side_stream* side) {
  if (!q) return fail(MOE_ERR_INVALID_ARG, "fp8 is NULL");
  return layer_fwd_impl(c, x, W_r, b_r, nullptr, nullptr, q, Ws1, Ws2, w_sg, y, s, ws, ws_bytes,
                        stream, side);
}

int moe_layer_bwd(const moe_cfg* c, const void* dy, const void* x, const void* W_r,
                  const void* W1, const void* W2, const void* Ws1, const void* Ws2,
                  const void* w_sg, const moe_saved* s, void* dx, float* dW_r, float* dW1,
                  float* dW2, float* dWs1, float* dWs2, float* dw_sg, void* ws, size_t ws_bytes,
                  void* stream, const moe_side_stream* side) {
  return layer_bwd_impl(c, dy, x, W_r, W1, W2, nullptr, Ws1, Ws2, w_sg, s, dx, dW_r, dW1, dW2,
                        dWs1, dWs2, dw_sg, ws, ws_bytes, stream, side);
}

int moe_layer_bwd_mxfp8(const moe_cfg* c, const void* dy, const void* x, const void* W_r,
                        const moe_mxfp8_dgrad* mxd, const void* Ws1, const void* Ws2,
                        const void* w_sg, const moe_saved* s, void* dx, float* dW_r, float* dW1,
                        float* dW2, float* dWs1, float* dWs2, float* dw_sg, void* ws,
                        size_t ws_bytes, void* stream, const moe_side_stream* side) {
  if (!mxd) return fail(MOE_ERR_INVALID_ARG, "mxd is NULL");
  return layer_bwd_impl(c, dy, x, W_r, nullptr, nullptr, nullptr, Ws1, Ws2, w_sg, s, dx, dW_r, dW1,
                        dW2, dWs1, dWs2, dw_sg, ws, ws_bytes, stream, side, mxd);
}

int moe_layer_bwd_fp8(const moe_cfg* c, const void* dy, const void* x, const void* W_r,
                      const moe_fp8_experts* q, const void* Ws1, const void* Ws2,
                      const void* w_sg, const moe_saved* s, void* dx, float* dW_r, float* dW1,
                      float* dW2, float* dWs1, float* dWs2, float* dw_sg, void* ws,
                      size_t ws_bytes, void* stream, const moe_side_stream* side) {
  if (!q) return fail(MOE_ERR_INVALID_ARG, "fp8 is NULL");
  return layer_bwd_impl(c, dy, x, W_r, nullptr, nullptr, q, Ws1, Ws2, w_sg, s, dx, dW_r, dW1, dW2,
                        dWs1, dWs2, dw_sg, ws, ws_bytes, stream, side);
}

}  // extern "C"

namespace moe {

// Entry points into the checks and the routing stages for other translation units.
int validate_cfg(const moe_cfg* c) { return check_cfg(c); }

int validate_ptr(const void* p, const char* name, bool required) {
  return check_ptr(p, name, required);
}

int route_stages(const moe_cfg* c, const void* x, const void* W_r, const float* b_r,
                 const float* logits_in, float* logits_out, int32_t* idx, float* gate,
                 int32_t* counts, int32_t* offsets, int32_t* slot_of_pair, int32_t* token_of_slot,
                 uint8_t* hist, int32_t* rowpre, cudaStream_t st) {
  RouteWs w;
  w.hist = hist;
  w.rowpre = rowpre;
  w.logits = nullptr;
  w.aux = nullptr;
  return route_impl(c, x, W_r, b_r, logits_in, logits_out, idx, gate, counts, offsets,
                    slot_of_pair, token_of_slot, w, st);
}

}  // namespace moe
