// The step plan: descriptor validation, parameter layout, workspace, and the
// fixed kernel schedule of one training step (forward, loss, backward,
// optimizer), behind the C ABI declared in include/mg.h.
//
// This is the GPU-side counterpart of the Meganeura pages' build_session
// (README Example section: autodiff + compile + GPU init happen once) and of
// its memory planner (abstract): here every value and every gradient gets its
// own region of one workspace allocated at creation, and the backward pass is
// derived by hand per fused node:
//   Linear (+ bias, + ReLU/GELU, + residual add) -> one GEMM with a fused epilogue
//   RMSNorm, causal attention                    -> their own kernels
//   cross-entropy / MSE                           -> a loss+gradient kernel
//   SGD / Adam                                    -> one multi-tensor kernel
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/mg.h"
#include "kernels.h"

using namespace mg;

namespace {

std::mutex g_err_mu;
std::string g_err = "";

constexpr size_t kAlignElems = 64;      // parameter offsets (256 B in fp32)
constexpr size_t kWsAlign = 1024;       // workspace region alignment
// Optimizer chunk (elements; one block of the update kernels per chunk).
// Short-lived blocks: the updates run beside the backward GEMMs on a second
// stream, and an SM holding several long update blocks when a persistent GEMM
// launches keeps that GEMM's CTA waiting for them (measured on GB300: C5 2913
// -> 3083 steps/s going from 16384 to 2048; C3 and C4 unchanged).
constexpr int kChunk = 2048;
constexpr int kNormChunks = 8 * 152;    // RMSNorm backward blocks (dgamma partial rows)
constexpr int kMsePartials = 1024;
constexpr size_t kColsumFloats = (size_t)kColsumBlocks * 2048;   // column-sum partials capacity

enum NodeKind { NK_LINEAR, NK_RMSNORM, NK_ATTN };

struct Value {
  int width = 0;
  size_t off = 0;        // workspace offset (value 0 = caller's x)
  size_t goff = 0;       // workspace offset of its gradient
  bool has_grad = false;
  bool need_grad = false;
  int producer = -1;     // node index
  int producer_act = 0;  // activation fused into the producing Linear
  int z_value = -1;      // saved pre-activation (GELU) of the producer
  int pending_add = -1;  // value whose gradient also flows into this one (skip)
  int consumers = 0;
};

struct Node {
  NodeKind kind;
  int layer = 0;
  int in = -1, out = -1;
  // linear
  int d_in = 0, d_out = 0, has_bias = 0, act = 0, skip = -1, z = -1;
  size_t w_off = 0, b_off = 0;
  // bf16 linear with a bias whose output feeds a linear: workspace offset of
  // the [ceil(batch / 32), d_out] column partials of its output gradient,
  // written by the consumer's input-gradient GEMM (0: none)
  size_t cp_off = 0;
  // bf16 linear under Adam whose weight gradient runs on the tensor cores
  // without a split over K: the weight's update is fused into that GEMM's
  // epilogue, so its input gradient (the last reader of the bf16 weight copy)
  // is formed first
  bool fuse_upd = false;
  // rmsnorm
  int d = 0;
  float eps = 0.f;
  size_t g_off = 0, rstd_off = 0;
  // attention
  int nh = 0, dh = 0, S = 0;
  size_t lse_off = 0, dsum_off = 0;
  // parameter tensors of this node: t0 .. t0+nt-1
  int t0 = 0, nt = 0;
};

struct Site {
  std::string name;
  double flops = 0, bytes = 0;
  int kernels = 1;
  int launches = 0;
  double total_ms = 0;
};

}  // namespace

struct mg_plan {
  int device = 0;
  int batch = 0;
  int loss = 0, precision = 0, optimizer = 0;
  float beta1 = 0.9f, beta2 = 0.999f, adam_eps = 1e-8f;
  DType dt = DT_F32;
  std::vector<mg_layer> layers;
  std::vector<Value> values;
  std::vector<Node> nodes;
  int final_value = 0;
  // parameters
  std::vector<size_t> p_off;
  std::vector<int> p_rows, p_cols;
  std::vector<int> p_is_weight;
  size_t n_params = 0;
  // workspace
  size_t ws_bytes = 0;
  char* ws = nullptr;
  size_t shadow_off = 0, chunks_off = 0, loss_off = 0, rowloss_off = 0, partial_off = 0,
         colsum_off = 0, flag_off = 0, lse_part_off = 0;
  size_t split_off = 0, split_floats = 0;   // strict weight gradients split over K
  size_t scal_off = 0;       // Adam's step scalars for fused updates (2 floats)
  // MG_FUSED_UPDATE=1: Adam's weight updates in the weight-gradient GEMMs'
  // epilogues where they can be (measured slower on GB300 for the large
  // MLPs: the epilogue's extra 26 bytes per weight outlast the next tile's
  // main loop and stall the tensor pipe), else all in the optimizer kernels
  bool fuse_update = false;
  bool any_fused = false;    // some node's update is fused into its weight-gradient GEMM
  int lse_parts = 0;         // 128-column softmax partials per logits row (0: not planned)
  int n_chunks = 0;
  const float* last_params = nullptr;
  bool use_tc = true;        // tcgen05 GEMMs in bf16 mode (MG_GEMM=simt turns them off)
  bool use_pair = true;      // SM-pair GEMMs for large shapes (MG_GEMM=tc1 turns them off)
  bool alias = true;         // gradient buffers share storage by lifetime (MG_NO_ALIAS=1: not)
  // GELU pre-activations recomputed in the backward instead of saved
  // (MG_RECOMPUTE_GELU=1): the forward does not store Z; one Z-sized buffer,
  // shared by every GELU layer, receives Z = X W + b again just before the
  // input-gradient GEMM that needs GELU'(Z)
  bool recompute_gelu = false;
  // A linear node whose weight gradient (and update) is moved to the end of
  // the backward: the smallest one, when it is smaller than the node the
  // backward ends with.  The last node's update has nothing left to overlap,
  // so the step ends with the smallest update instead of the last layer's.
  int defer_dw = -1;
  // CUDA-graph replay of the training step (MG_GRAPH=0: every kernel launched
  // directly): a step is captured on the second call with the same buffers
  // and relaunched with the optimizer nodes' step scalars updated; graphs for
  // the two most recent buffer sets are kept (double-buffered inputs)
  bool use_graph = true;
  struct OptNode {
    cudaGraphNode_t node;
    cudaKernelNodeParams kp;
    OptKernelInfo info;
    uint64_t arg[12];
    void* argv[12];
  };
  struct StepGraph {
    const void* key[6] = {};
    int calls = 0, launches = 0;
    long long last_use = 0;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t gexec = nullptr;
    std::vector<OptNode> opt_nodes;
  };
  std::vector<StepGraph> graphs;
  long long graph_clock = 0, graph_replays = 0;
  cudaStream_t cap = nullptr;   // private stream the step is captured on
  size_t grad_bytes_unaliased = 0, grad_bytes = 0;   // gradient storage without / with sharing
  // schedule bookkeeping
  std::vector<Site> sites;
  // update of each node's parameters on a second stream, overlapping the rest
  // of the backward pass (the optimizer is bandwidth-bound, the GEMMs are not)
  cudaStream_t aux = nullptr;
  std::vector<cudaEvent_t> node_ev;
  cudaEvent_t join_ev = nullptr;
  std::vector<int> tensor_chunk;     // first chunk of tensor t; [n_tensors] = n_chunks
  int last_launches = 0;
  bool profiling = false;
  int prof_max = 0, prof_calls = 0;
  std::vector<cudaEvent_t> events;
  std::string err;
  std::string dump;
};

namespace {

mg_status fail(mg_plan* p, mg_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (p) p->err = buf;
  std::lock_guard<std::mutex> lk(g_err_mu);
  g_err = buf;
  return st;
}

mg_status cuda_fail(mg_plan* p, cudaError_t e, const char* what) {
  return fail(p, MG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Bump {
  size_t top = 0;
  size_t take(size_t bytes) {
    size_t o = round_up(top, kWsAlign);
    top = o + round_up(bytes, 16);
    return o;
  }
};

// ---- execution context ---------------------------------------------------
struct Exec {
  mg_plan* p;
  cudaStream_t s;
  bool dry;          // only register sites
  bool profile;      // record events around each site
  int cursor = 0;
  int launches = 0;
  cudaError_t err = cudaSuccess;
  // optimizer arguments of a training step
  float* params = nullptr;
  float* grads = nullptr;
  float* m = nullptr;
  float* v = nullptr;
  float lr = 0.f;
  int step = 1;
  bool ce_parts = false;   // the head GEMM wrote the logits' softmax partials
  // per node: its output gradient's column partials were written by the
  // consumer's input-gradient GEMM in this backward (bias gradient = their sum)
  std::vector<unsigned char> db_parts;
};

template <class F>
void site_on(Exec& e, cudaStream_t st, const std::string& name, double flops, double bytes,
             int kernels, F&& f);

template <class F>
void site(Exec& e, const std::string& name, double flops, double bytes, int kernels, F&& f) {
  site_on(e, e.s, name, flops, bytes, kernels, static_cast<F&&>(f));
}

template <class F>
void site_on(Exec& e, cudaStream_t st, const std::string& name, double flops, double bytes,
             int kernels, F&& f) {
  mg_plan* p = e.p;
  int id = e.cursor++;
  if (e.dry) {
    Site st;
    st.name = name;
    st.flops = flops;
    st.bytes = bytes;
    st.kernels = kernels;
    p->sites.push_back(st);
    return;
  }
  if (e.err != cudaSuccess) return;
  const int ns = (int)p->sites.size();
  const bool rec = e.profile && p->profiling && p->prof_calls < p->prof_max && id < ns;
  if (rec) cudaEventRecord(p->events[((size_t)p->prof_calls * ns + id) * 2], st);
  cudaError_t r = f();
  if (r != cudaSuccess) e.err = r;
  if (rec) cudaEventRecord(p->events[((size_t)p->prof_calls * ns + id) * 2 + 1], st);
  e.launches += kernels;
}

template <class T>
T* wsp(mg_plan* p, size_t off) {
  return reinterpret_cast<T*>(p->ws + off);
}

const void* val_ptr(mg_plan* p, int v, const void* x) {
  return v == 0 ? x : (const void*)(p->ws + p->values[v].off);
}

void* grad_ptr(mg_plan* p, int v) { return p->ws + p->values[v].goff; }

double gemm_bytes(const GemmArgs& g) {
  double in = (double)dtype_size(g.in_type), aux = (double)dtype_size(g.aux_type);
  double b = ((double)g.M * g.K + (double)g.K * g.N) * in + (double)g.M * g.N * dtype_size(g.out_type);
  if (g.bias) b += 4.0 * g.N;
  if (g.out_z) b += aux * g.M * g.N;
  if (g.dact) b += aux * g.M * g.N;
  if (g.resid) b += aux * g.M * g.N;
  if (g.col_part) b += 4.0 * ((g.M + 31) / 32) * g.N;
  return b;
}

int norm_chunks(const mg_plan* p) { return p->batch < kNormChunks ? p->batch : kNormChunks; }

bool tc_path(const mg_plan* p, const GemmArgs& g) { return p->use_tc && gemm_tc_eligible(g); }

// error word of the tensor-core pipeline: 4 bytes after the loss scalar
int* err_word(mg_plan* p) { return reinterpret_cast<int*>(p->ws + p->loss_off + 4); }

bool pair_path(const mg_plan* p, const GemmArgs& g) {
  return p->use_pair && tc_path(p, g) && gemm_pair_eligible(g);
}

cudaError_t run_gemm(mg_plan* p, const GemmArgs& g, cudaStream_t s) {
  if (pair_path(p, g)) return gemm_pair(g, err_word(p), s);
  if (tc_path(p, g)) return gemm_tc(g, err_word(p), s);
  return gemm_simt(g, s);
}

std::string gemm_name(const mg_plan* p, const char* what, int layer, const GemmArgs& g) {
  char b[160];
  const char* kind = g.in_type != DT_BF16 ? "f32-ffma"
                     : pair_path(p, g)    ? "bf16-tcgen05x2"
                     : tc_path(p, g)      ? "bf16-tcgen05"
                     : gemm_simt_skinny(g) ? "bf16-skinny"
                                          : "bf16-simt";
  snprintf(b, sizeof b, "%s[l%d] %dx%dx%d %s", what, layer, g.M, g.N, g.K, kind);
  return b;
}

// ---- the schedule ----------------------------------------------------------
void forward_pass(Exec& e, const float* params, const void* x) {
  mg_plan* p = e.p;
  const DType dt = p->dt;
  const void* wbase = dt == DT_BF16 ? (const void*)(p->ws + p->shadow_off) : (const void*)params;
  for (size_t ni = 0; ni < p->nodes.size(); ++ni) {
    const Node& n = p->nodes[ni];
    if (n.kind == NK_LINEAR) {
      GemmArgs g;
      g.M = p->batch; g.N = n.d_out; g.K = n.d_in;
      g.A = val_ptr(p, n.in, x); g.lda = n.d_in; g.a_mn = 0;
      g.B = (const char*)wbase + n.w_off * dtype_size(dt); g.ldb = n.d_out; g.b_k = 0;
      g.in_type = dt;
      g.bias = n.has_bias ? params + n.b_off : nullptr;
      g.act = n.act;
      if (n.z >= 0 && !p->recompute_gelu) { g.out_z = p->ws + p->values[n.z].off; g.ldz = n.d_out; }
      if (n.skip >= 0) { g.resid = val_ptr(p, n.skip, x); g.ldr = n.d_out; }
      g.aux_type = dt;
      g.out = p->ws + p->values[n.out].off; g.ldo = n.d_out; g.out_type = dt;
      // the logits' softmax partials come out of the head GEMM's epilogue
      // (tensor-core path only), so the loss reads the logits once
      if (n.out == p->final_value && p->lse_parts && n.act == 0 && n.skip < 0 && n.in != 0 &&
          tc_path(p, g)) {
        g.lse_part = wsp<float2>(p, p->lse_part_off);
        g.lse_ld = p->lse_parts;
        e.ce_parts = true;
      }
      site(e, gemm_name(p, "fwd", n.layer, g), 2.0 * g.M * g.N * g.K, gemm_bytes(g), 1,
           [&] { return run_gemm(p, g, e.s); });
    } else if (n.kind == NK_RMSNORM) {
      double bytes = 2.0 * dtype_size(dt) * p->batch * n.d + 4.0 * n.d + 4.0 * p->batch;
      char nm[96];
      snprintf(nm, sizeof nm, "rmsnorm_fwd[l%d] %dx%d", n.layer, p->batch, n.d);
      site(e, nm, 0, bytes, 1, [&] {
        return rmsnorm_fwd(dt, val_ptr(p, n.in, x), params + n.g_off, p->ws + p->values[n.out].off,
                           wsp<float>(p, n.rstd_off), p->batch, n.d, n.eps, e.s);
      });
    } else {
      int nb = p->batch / n.S;
      double pairs = (double)n.S * (n.S + 1) / 2.0;
      double flops = 4.0 * nb * n.nh * pairs * n.dh;
      double bytes = 2.0 * p->batch * 4.0 * n.nh * n.dh + 4.0 * nb * n.nh * n.S;
      char nm[96];
      const void* qkv = val_ptr(p, n.in, x);
      const bool tc = p->use_tc && attn_tc_eligible(n.S, n.nh, n.dh, qkv);
      snprintf(nm, sizeof nm, "attn_fwd[l%d] b%d s%d h%d d%d %s", n.layer, nb, n.S, n.nh, n.dh,
               tc ? "tcgen05" : "simt");
      site(e, nm, flops, bytes, 1, [&] {
        if (tc)
          return attn_fwd_tc_launch(qkv, p->ws + p->values[n.out].off, wsp<float>(p, n.lse_off),
                                    nb, n.S, n.nh, err_word(p), e.s);
        return attn_fwd(qkv, p->ws + p->values[n.out].off, wsp<float>(p, n.lse_off), nb, n.S,
                        n.nh, n.dh, e.s);
      });
    }
  }
}

void loss_pass(Exec& e, const void* labels) {
  mg_plan* p = e.p;
  const DType dt = p->dt;
  const Value& f = p->values[p->final_value];
  const int C = f.width, B = p->batch;
  const void* logits = p->ws + f.off;
  void* dlogits = p->ws + f.goff;
  if (p->loss == MG_LOSS_MSE) {
    size_t n = (size_t)B * C;
    site(e, "mse_loss", 0, 3.0 * dtype_size(dt) * n, 2, [&] {
      return mse_loss(dt, logits, labels, n, dlogits, wsp<float>(p, p->partial_off), kMsePartials,
                      wsp<float>(p, p->loss_off), e.s);
    });
  } else {
    int kind = p->loss == MG_LOSS_CE_DENSE ? 0 : 1;
    double bytes = 2.0 * dtype_size(dt) * B * C + (kind == 0 ? 4.0 * B * C : 4.0 * B);
    char nm[96];
    if (e.ce_parts) {
      snprintf(nm, sizeof nm, "softmax_ce_%s %dx%d (GEMM partials)", kind == 0 ? "dense" : "index", B, C);
      site(e, nm, 0, bytes + 8.0 * B * p->lse_parts, 2, [&] {
        return ce_loss_from_partials(logits, B, C, C, wsp<float2>(p, p->lse_part_off), p->lse_parts,
                                     kind, labels, dlogits, wsp<float>(p, p->rowloss_off),
                                     wsp<float>(p, p->loss_off), e.s);
      });
    } else {
      snprintf(nm, sizeof nm, "softmax_ce_%s %dx%d", kind == 0 ? "dense" : "index", B, C);
      site(e, nm, 0, bytes, 2, [&] {
        return ce_loss(dt, logits, B, C, C, kind, labels, dlogits, wsp<float>(p, p->rowloss_off),
                       wsp<float>(p, p->loss_off), e.s);
      });
    }
  }
}

// Adam's and LaProp's step scalars: lr / (1 - b1^t) and 1 / sqrt(1 - b2^t).
void step_scalars(const mg_plan* p, float lr, int step, float* lr_bc1, float* inv_sqrt_bc2) {
  double bc1 = 1.0 - std::pow((double)p->beta1, (double)step);
  double bc2 = 1.0 - std::pow((double)p->beta2, (double)step);
  *lr_bc1 = (float)(lr / bc1);
  *inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
}

// Optimizer update of node ni's parameters, on the auxiliary stream once the
// node's backward kernels (the last readers of its weights) have run; with
// skip_weight, only its tensors after the weight (the weight's update was
// fused into its gradient GEMM).
void node_update(Exec& e, int ni, bool skip_weight = false) {
  mg_plan* p = e.p;
  const Node& n = p->nodes[ni];
  const int t_lo = n.t0 + (skip_weight ? 1 : 0), t_hi = n.t0 + n.nt;
  if (t_lo >= t_hi) return;
  const int c0 = p->tensor_chunk[t_lo], c1 = p->tensor_chunk[t_hi];
  double np = 0;
  for (int t = t_lo; t < t_hi; ++t) np += (double)p->p_rows[t] * p->p_cols[t];
  const Chunk* chunks = wsp<Chunk>(p, p->chunks_off) + c0;
  void* shadow = p->dt == DT_BF16 ? p->ws + p->shadow_off : nullptr;
  if (!e.dry && e.err == cudaSuccess) {
    cudaError_t r = cudaEventRecord(p->node_ev[2 * ni], e.s);
    if (r == cudaSuccess) r = cudaStreamWaitEvent(p->aux, p->node_ev[2 * ni], 0);
    if (r != cudaSuccess) e.err = r;
  }
  char nm[96];
  if (p->optimizer == MG_OPT_ADAM || p->optimizer == MG_OPT_LAPROP) {
    float lr_bc1, inv_sqrt_bc2;
    step_scalars(p, e.lr, e.step, &lr_bc1, &inv_sqrt_bc2);
    const bool lap = p->optimizer == MG_OPT_LAPROP;
    snprintf(nm, sizeof nm, "%s[l%d] %.0f params", lap ? "laprop" : "adam", n.layer, np);
    site_on(e, p->aux, nm, 0, np * (28.0 + (shadow ? 2.0 : 0.0)), 1, [&] {
      return (lap ? laprop_update : adam_update)(chunks, c1 - c0, e.params, e.grads, e.m, e.v,
                                                 shadow, lr_bc1, inv_sqrt_bc2, p->beta1,
                                                 p->beta2, p->adam_eps, p->aux);
    });
  } else if (p->optimizer == MG_OPT_SGD_MOMENTUM) {
    snprintf(nm, sizeof nm, "momentum[l%d] %.0f params", n.layer, np);
    site_on(e, p->aux, nm, 0, np * (20.0 + (shadow ? 2.0 : 0.0)), 1, [&] {
      return momentum_update(chunks, c1 - c0, e.params, e.grads, e.m, shadow, e.lr, p->beta1,
                             p->aux);
    });
  } else {
    snprintf(nm, sizeof nm, "sgd[l%d] %.0f params", n.layer, np);
    site_on(e, p->aux, nm, 0, np * (12.0 + (shadow ? 2.0 : 0.0)), 1, [&] {
      return sgd_update(chunks, c1 - c0, e.params, e.grads, shadow, e.lr, p->aux);
    });
  }
}

// dW = X^T dZ of linear node n   (M = d_in, N = d_out, K = batch)
GemmArgs dw_args(mg_plan* p, const Node& n, float* grads, const void* x) {
  GemmArgs g;
  g.M = n.d_in; g.N = n.d_out; g.K = p->batch;
  g.A = val_ptr(p, n.in, x); g.lda = n.d_in; g.a_mn = 1;
  g.B = grad_ptr(p, n.out); g.ldb = n.d_out; g.b_k = 0;
  g.in_type = p->dt; g.aux_type = p->dt;
  g.out = grads + n.w_off; g.ldo = n.d_out; g.out_type = DT_F32;
  if (p->split_floats) {
    g.split_ws = wsp<float>(p, p->split_off);
    g.split_ws_floats = p->split_floats;
  }
  return g;
}

// Whether the weight update of a node with these weight-gradient arguments
// can run in the GEMM's epilogue: Adam, bf16, a tensor-core kernel and no
// split over K (a split's partial tiles are not the gradient).
bool update_fusable(mg_plan* p, const GemmArgs& g) {
  if (!p->fuse_update || p->dt != DT_BF16 || p->optimizer != MG_OPT_ADAM || !tc_path(p, g))
    return false;
  return (pair_path(p, g) ? gemm_pair_split_count(g) : gemm_tc_splits(g, nullptr)) == 1;
}

// Plan-time choice of the fused updates (the input pointer is taken as
// aligned; a step whose input is not falls back to the optimizer kernel).
void plan_fused_updates(mg_plan* p) {
  p->any_fused = false;
  for (Node& n : p->nodes) {
    n.fuse_upd = false;
    if (n.kind != NK_LINEAR || !p->values[n.out].need_grad) continue;
    n.fuse_upd = update_fusable(p, dw_args(p, n, nullptr, nullptr));
    p->any_fused = p->any_fused || n.fuse_upd;
  }
}

void backward_pass(Exec& e, const float* params, float* grads, const void* x) {
  mg_plan* p = e.p;
  e.db_parts.assign(p->nodes.size(), 0);
  const DType dt = p->dt;
  const void* wbase = dt == DT_BF16 ? (const void*)(p->ws + p->shadow_off) : (const void*)params;
  GemmArgs deferred;   // the deferred node's weight gradient
  bool deferred_fused = false;
  for (int ni = (int)p->nodes.size() - 1; ni >= 0; --ni) {
    const Node& n = p->nodes[ni];
    if (!p->values[n.out].need_grad) continue;
    const void* gy = grad_ptr(p, n.out);
    const Value& vin = p->values[n.in];
    const void* dadd = vin.pending_add >= 0 ? grad_ptr(p, vin.pending_add) : nullptr;
    if (n.kind == NK_LINEAR) {
      GemmArgs g = dw_args(p, n, grads, x);
      // the weight's Adam step in the dW epilogue (Adam's state as the
      // optimizer kernel would leave it)
      const bool fused = n.fuse_upd && update_fusable(p, g);
      if (fused && !e.dry) {
        g.upd_p = e.params + n.w_off;
        g.upd_m = e.m + n.w_off;
        g.upd_v = e.v + n.w_off;
        g.upd_shadow = p->ws + p->shadow_off + n.w_off * 2;
        g.upd_scal = wsp<float>(p, p->scal_off);
        g.upd_b1 = p->beta1;
        g.upd_b2 = p->beta2;
        g.upd_eps = p->adam_eps;
      }
      if (n.has_bias) {
        // db = column sums of dZ, on the auxiliary stream (only the optimizer
        // reads it), overlapping this node's dW and dX products: the sum of
        // the column partials the consumer's input-gradient GEMM wrote, else
        // a pass over dZ
        if (!e.dry && e.err == cudaSuccess) {
          cudaError_t r = cudaEventRecord(p->node_ev[2 * ni + 1], e.s);
          if (r == cudaSuccess) r = cudaStreamWaitEvent(p->aux, p->node_ev[2 * ni + 1], 0);
          if (r != cudaSuccess) e.err = r;
        }
        char nm[96];
        if (e.db_parts[ni]) {
          const int chunks = (p->batch + 31) / 32;
          snprintf(nm, sizeof nm, "db_parts[l%d] %dx%d", n.layer, chunks, n.d_out);
          site_on(e, p->aux, nm, 0, 4.0 * chunks * n.d_out + 4.0 * n.d_out, 1, [&] {
            return colsum_partials(wsp<float>(p, n.cp_off), chunks, n.d_out, grads + n.b_off,
                                   p->aux);
          });
        } else {
          snprintf(nm, sizeof nm, "db_colsum[l%d] %dx%d", n.layer, p->batch, n.d_out);
          site_on(e, p->aux, nm, 0, (double)dtype_size(dt) * p->batch * n.d_out + 4.0 * n.d_out,
                  2, [&] {
                    return colsum(dt, gy, p->batch, n.d_out, n.d_out,
                                  wsp<float>(p, p->colsum_off), kColsumFloats, grads + n.b_off,
                                  p->aux);
                  });
        }
      }
      auto weight_grad = [&] {
        if (ni == p->defer_dw) {
          deferred = g;
          deferred_fused = fused;
        } else {
          // a fused update reads p, m, v and writes them and the bf16 copy
          site(e, gemm_name(p, fused ? "dW+adam" : "dW", n.layer, g), 2.0 * g.M * g.N * g.K,
               gemm_bytes(g) + (fused ? 26.0 * g.M * g.N : 0.0), 1,
               [&] { return run_gemm(p, g, e.s); });
        }
      };
      if (!n.fuse_upd) weight_grad();
      if (vin.need_grad) {
        // dX = dZ W^T, times act'(saved) of the producer of X, plus the skip gradient
        GemmArgs h;
        h.M = p->batch; h.N = n.d_in; h.K = n.d_out;
        h.A = gy; h.lda = n.d_out; h.a_mn = 0;
        h.B = (const char*)wbase + n.w_off * dtype_size(dt); h.ldb = n.d_out; h.b_k = 1;
        h.in_type = dt; h.aux_type = dt;
        if (vin.producer_act) {
          h.dact = vin.producer_act;
          int sv = vin.producer_act == ACT_GELU ? vin.z_value : n.in;
          h.saved = p->ws + p->values[sv].off;
          h.lds = n.d_in;
          if (vin.producer_act == ACT_GELU && p->recompute_gelu) {
            // Z of the producing Linear again, exactly as its forward GEMM
            // formed it (same kernel, inputs and weights: the optimizer has
            // not yet updated that node), into the shared Z buffer
            const Node& pn = p->nodes[vin.producer];
            GemmArgs r;
            r.M = p->batch; r.N = pn.d_out; r.K = pn.d_in;
            r.A = val_ptr(p, pn.in, x); r.lda = pn.d_in; r.a_mn = 0;
            r.B = (const char*)wbase + pn.w_off * dtype_size(dt); r.ldb = pn.d_out; r.b_k = 0;
            r.in_type = dt;
            r.bias = pn.has_bias ? params + pn.b_off : nullptr;
            r.aux_type = dt;
            r.out = p->ws + p->values[pn.z].off; r.ldo = pn.d_out; r.out_type = dt;
            site(e, gemm_name(p, "recompute_z", pn.layer, r), 2.0 * r.M * r.N * r.K, gemm_bytes(r),
                 1, [&] { return run_gemm(p, r, e.s); });
          }
        }
        if (dadd) { h.resid = dadd; h.ldr = n.d_in; }
        h.out = grad_ptr(p, n.in); h.ldo = n.d_in; h.out_type = dt;
        if (vin.producer >= 0 && p->nodes[vin.producer].cp_off && tc_path(p, h)) {
          // this GEMM writes the producer's whole output gradient: its
          // epilogue also leaves the column partials of the producer's db
          h.col_part = wsp<float>(p, p->nodes[vin.producer].cp_off);
          e.db_parts[vin.producer] = 1;
        }
        site(e, gemm_name(p, "dX", n.layer, h), 2.0 * h.M * h.N * h.K, gemm_bytes(h), 1,
             [&] { return run_gemm(p, h, e.s); });
      }
      if (n.fuse_upd) weight_grad();   // after dX, the last reader of the bf16 weights
      if (ni != p->defer_dw) node_update(e, ni, fused);
    } else if (n.kind == NK_RMSNORM) {
      void* dx = vin.need_grad ? grad_ptr(p, n.in) : nullptr;
      double bytes = (double)dtype_size(dt) * p->batch * n.d * (dx ? (dadd ? 4 : 3) : 2);
      char nm[96];
      snprintf(nm, sizeof nm, "rmsnorm_bwd[l%d] %dx%d", n.layer, p->batch, n.d);
      site(e, nm, 0, bytes, 2, [&] {
        return rmsnorm_bwd(dt, gy, val_ptr(p, n.in, x), wsp<float>(p, n.rstd_off),
                           params + n.g_off, dx ? dadd : nullptr, dx,
                           wsp<float>(p, p->partial_off), norm_chunks(p), grads + n.g_off,
                           p->batch, n.d, e.s);
      });
      node_update(e, ni);
    } else {
      if (!vin.need_grad) continue;
      int nb = p->batch / n.S;
      double pairs = (double)n.S * (n.S + 1) / 2.0;
      double flops = 10.0 * nb * n.nh * pairs * n.dh;
      double bytes = 2.0 * p->batch * n.nh * n.dh * (3 + 2 + 3);
      char nm[96];
      const void* qkv = val_ptr(p, n.in, x);
      const bool tc = p->use_tc && attn_tc_eligible(n.S, n.nh, n.dh, qkv);
      snprintf(nm, sizeof nm, "attn_bwd[l%d] b%d s%d h%d d%d %s", n.layer, nb, n.S, n.nh, n.dh,
               tc ? "tcgen05" : "simt");
      site(e, nm, flops, bytes, attn_bwd_launches(), [&] {
        if (tc) {
          cudaError_t r = attn_bwd_pre(p->ws + p->values[n.out].off, gy, wsp<float>(p, n.dsum_off),
                                       nb, n.S, n.nh, e.s);
          if (r != cudaSuccess) return r;
          return attn_bwd_tc_launch(qkv, gy, wsp<float>(p, n.lse_off), wsp<float>(p, n.dsum_off),
                                    grad_ptr(p, n.in), nb, n.S, n.nh, err_word(p), e.s);
        }
        return attn_bwd(qkv, p->ws + p->values[n.out].off, gy, wsp<float>(p, n.lse_off),
                        wsp<float>(p, n.dsum_off), grad_ptr(p, n.in), nb, n.S, n.nh, n.dh, e.s);
      });
    }
  }
  if (p->defer_dw >= 0) {
    const Node& n = p->nodes[p->defer_dw];
    site(e, gemm_name(p, deferred_fused ? "dW+adam" : "dW", n.layer, deferred),
         2.0 * deferred.M * deferred.N * deferred.K,
         gemm_bytes(deferred) + (deferred_fused ? 26.0 * deferred.M * deferred.N : 0.0), 1,
         [&] { return run_gemm(p, deferred, e.s); });
    node_update(e, p->defer_dw, deferred_fused);
  }
}

// The step ends when the auxiliary stream's updates have: the caller's stream
// waits for them.
void join_updates(Exec& e) {
  mg_plan* p = e.p;
  if (e.dry || e.err != cudaSuccess) return;
  cudaError_t r = cudaEventRecord(p->join_ev, p->aux);
  if (r == cudaSuccess) r = cudaStreamWaitEvent(e.s, p->join_ev, 0);
  if (r != cudaSuccess) e.err = r;
}

void train_schedule(Exec& e, float* params, float* grads, float* m, float* v, const void* x,
                    const void* labels, float lr, int step) {
  e.params = params;
  e.grads = grads;
  e.m = m;
  e.v = v;
  e.lr = lr;
  e.step = step;
  mg_plan* p = e.p;
  if (p->any_fused) {
    // Adam's step scalars in device memory for the fused updates (a kernel
    // node, so that a replayed graph carries each step's values)
    float lr_bc1, inv;
    step_scalars(p, lr, step, &lr_bc1, &inv);
    site(e, "step_scalars", 0, 8, 1,
         [&] { return write_step_scalars(wsp<float>(p, p->scal_off), lr_bc1, inv, e.s); });
  }
  forward_pass(e, params, x);
  loss_pass(e, labels);
  backward_pass(e, params, grads, x);
  join_updates(e);
}

// ---- descriptor compile ------------------------------------------------------
mg_status compile(mg_plan* p, const mg_graph_desc* d) {
  if (d->batch <= 0) return fail(p, MG_ERR_SHAPE, "batch must be positive (got %d)", d->batch);
  if (d->n_layers <= 0 || !d->layers) return fail(p, MG_ERR_INVALID_ARG, "graph has no layers");
  if (d->loss < 0 || d->loss > 2) return fail(p, MG_ERR_INVALID_ARG, "bad loss kind %d", d->loss);
  if (d->precision < 0 || d->precision > 1)
    return fail(p, MG_ERR_INVALID_ARG, "bad precision %d", d->precision);
  if (d->optimizer < MG_OPT_SGD || d->optimizer > MG_OPT_SGD_MOMENTUM)
    return fail(p, MG_ERR_INVALID_ARG, "bad optimizer %d", d->optimizer);
  if ((d->optimizer == MG_OPT_ADAM || d->optimizer == MG_OPT_LAPROP) &&
      !(d->beta1 >= 0 && d->beta1 < 1 && d->beta2 >= 0 && d->beta2 < 1 && d->adam_eps > 0))
    return fail(p, MG_ERR_INVALID_ARG, "Adam and LaProp need 0 <= beta < 1 and eps > 0");
  if (d->optimizer == MG_OPT_SGD_MOMENTUM && !(d->beta1 >= 0 && d->beta1 < 1))
    return fail(p, MG_ERR_INVALID_ARG, "momentum (beta1) must be in [0, 1)");
  p->batch = d->batch;
  p->loss = d->loss;
  p->precision = d->precision;
  p->optimizer = d->optimizer;
  p->beta1 = d->beta1;
  p->beta2 = d->beta2;
  p->adam_eps = d->adam_eps;
  p->dt = d->precision == MG_PREC_BF16 ? DT_BF16 : DT_F32;
  p->layers.assign(d->layers, d->layers + d->n_layers);

  // input width
  int w0 = -1;
  for (auto& l : p->layers) {
    if (l.op == MG_OP_LINEAR) { w0 = l.d_in; break; }
    if (l.op == MG_OP_RMSNORM) { w0 = l.d_in; break; }
    if (l.op == MG_OP_CAUSAL_ATTENTION) { w0 = 3 * l.n_heads * l.head_dim; break; }
  }
  if (w0 <= 0) return fail(p, MG_ERR_SHAPE, "cannot infer the input width");
  p->values.clear();
  p->nodes.clear();
  Value vx;
  vx.width = w0;
  p->values.push_back(vx);
  int cur = 0;
  std::vector<int> skips;
  size_t poff = 0;
  auto add_param = [&](int rows, int cols, int is_w) {
    poff = round_up(poff, kAlignElems);
    p->p_off.push_back(poff);
    p->p_rows.push_back(rows);
    p->p_cols.push_back(cols);
    p->p_is_weight.push_back(is_w);
    size_t o = poff;
    poff += (size_t)rows * cols;
    return o;
  };
  auto new_value = [&](int width, int producer) {
    Value v;
    v.width = width;
    v.producer = producer;
    p->values.push_back(v);
    return (int)p->values.size() - 1;
  };
  const int nl = (int)p->layers.size();
  for (int i = 0; i < nl; ++i) {
    const mg_layer& l = p->layers[i];
    Value& vc = p->values[cur];
    switch (l.op) {
      case MG_OP_LINEAR: {
        if (l.d_in <= 0 || l.d_out <= 0) return fail(p, MG_ERR_SHAPE, "layer %d: bad Linear widths", i);
        if (l.d_in != vc.width)
          return fail(p, MG_ERR_SHAPE, "layer %d: Linear d_in %d != incoming width %d", i, l.d_in, vc.width);
        Node n;
        n.kind = NK_LINEAR;
        n.layer = i;
        n.in = cur;
        n.d_in = l.d_in;
        n.d_out = l.d_out;
        n.has_bias = l.has_bias ? 1 : 0;
        n.t0 = (int)p->p_off.size();
        n.w_off = add_param(l.d_in, l.d_out, 1);
        if (n.has_bias) n.b_off = add_param(1, l.d_out, 0);
        n.nt = (int)p->p_off.size() - n.t0;
        if (i + 1 < nl && (p->layers[i + 1].op == MG_OP_RELU || p->layers[i + 1].op == MG_OP_GELU_TANH)) {
          n.act = p->layers[i + 1].op == MG_OP_RELU ? ACT_RELU : ACT_GELU;
          ++i;
          if (i + 1 < nl && p->layers[i + 1].op == MG_OP_RESIDUAL_END)
            return fail(p, MG_ERR_UNSUPPORTED, "layer %d: an activation directly before a residual end", i);
        }
        if (i + 1 < nl && p->layers[i + 1].op == MG_OP_RESIDUAL_END) {
          if (skips.empty()) return fail(p, MG_ERR_INVALID_ARG, "layer %d: residual end without begin", i + 1);
          n.skip = skips.back();
          skips.pop_back();
          if (p->values[n.skip].width != l.d_out)
            return fail(p, MG_ERR_SHAPE, "layer %d: residual widths differ (%d vs %d)", i + 1,
                        p->values[n.skip].width, l.d_out);
          ++i;
        }
        int ni = (int)p->nodes.size();
        if (n.act == ACT_GELU) n.z = new_value(l.d_out, ni);
        n.out = new_value(l.d_out, ni);
        p->values[n.out].producer_act = n.act;
        p->values[n.out].z_value = n.z;
        p->values[n.in].consumers++;
        p->nodes.push_back(n);
        cur = n.out;
        break;
      }
      case MG_OP_RMSNORM: {
        if (l.d_in != vc.width)
          return fail(p, MG_ERR_SHAPE, "layer %d: RMSNorm width %d != incoming width %d", i, l.d_in, vc.width);
        if (l.d_in > 4096) return fail(p, MG_ERR_UNSUPPORTED, "layer %d: RMSNorm width above 4096", i);
        if (!(l.eps >= 0)) return fail(p, MG_ERR_INVALID_ARG, "layer %d: RMSNorm eps < 0", i);
        if (vc.producer_act) return fail(p, MG_ERR_UNSUPPORTED, "layer %d: RMSNorm after an activation", i);
        Node n;
        n.kind = NK_RMSNORM;
        n.layer = i;
        n.in = cur;
        n.d = l.d_in;
        n.eps = l.eps;
        n.t0 = (int)p->p_off.size();
        n.g_off = add_param(1, l.d_in, 0);
        n.nt = 1;
        int ni = (int)p->nodes.size();
        n.out = new_value(l.d_in, ni);
        p->values[n.in].consumers++;
        p->nodes.push_back(n);
        cur = n.out;
        break;
      }
      case MG_OP_RESIDUAL_BEGIN:
        if (vc.producer_act) return fail(p, MG_ERR_UNSUPPORTED, "layer %d: residual source is an activation output", i);
        skips.push_back(cur);
        break;
      case MG_OP_RESIDUAL_END:
        return fail(p, MG_ERR_UNSUPPORTED, "layer %d: residual end must directly follow a Linear", i);
      case MG_OP_RELU:
      case MG_OP_GELU_TANH:
        return fail(p, MG_ERR_UNSUPPORTED, "layer %d: activation must directly follow a Linear", i);
      case MG_OP_CAUSAL_ATTENTION: {
        if (p->dt != DT_BF16) return fail(p, MG_ERR_UNSUPPORTED, "layer %d: attention needs bf16 precision", i);
        if (l.n_heads <= 0 || l.head_dim != 64)
          return fail(p, MG_ERR_UNSUPPORTED, "layer %d: attention supports head_dim 64 only", i);
        if (l.seq_len <= 0 || l.seq_len % 64)
          return fail(p, MG_ERR_UNSUPPORTED, "layer %d: seq_len must be a positive multiple of 64", i);
        if (d->batch % l.seq_len) return fail(p, MG_ERR_SHAPE, "layer %d: batch not a multiple of seq_len", i);
        if (vc.width != 3 * l.n_heads * l.head_dim)
          return fail(p, MG_ERR_SHAPE, "layer %d: attention input width %d != 3*%d*%d", i, vc.width,
                      l.n_heads, l.head_dim);
        if (vc.producer_act) return fail(p, MG_ERR_UNSUPPORTED, "layer %d: attention after an activation", i);
        Node n;
        n.kind = NK_ATTN;
        n.layer = i;
        n.in = cur;
        n.nh = l.n_heads;
        n.dh = l.head_dim;
        n.S = l.seq_len;
        int ni = (int)p->nodes.size();
        n.out = new_value(l.n_heads * l.head_dim, ni);
        p->values[n.in].consumers++;
        p->nodes.push_back(n);
        cur = n.out;
        break;
      }
      default:
        return fail(p, MG_ERR_INVALID_ARG, "layer %d: unknown op %d", i, l.op);
    }
  }
  if (!skips.empty()) return fail(p, MG_ERR_INVALID_ARG, "residual begin without end");
  if (p->nodes.empty()) return fail(p, MG_ERR_INVALID_ARG, "graph has no computing layer");
  if (p->values[cur].producer_act)
    return fail(p, MG_ERR_UNSUPPORTED, "an activation directly before the loss is not supported");
  for (auto& v : p->values)
    if (v.consumers > 1) return fail(p, MG_ERR_UNSUPPORTED, "a value feeds two layers");
  p->final_value = cur;
  p->n_params = round_up(poff, kAlignElems);
  if (p->p_off.empty()) return fail(p, MG_ERR_INVALID_ARG, "graph has no parameters");
  if (p->dt == DT_BF16 && p->values[0].width % 8)
    return fail(p, MG_ERR_ALIGN, "bf16 input rows must be a multiple of 16 bytes");

  // which values need a gradient: anything downstream of a parameter
  for (size_t ni = 0; ni < p->nodes.size(); ++ni) {
    const Node& n = p->nodes[ni];
    bool need = n.kind != NK_ATTN || p->values[n.in].need_grad;
    if (n.skip >= 0 && p->values[n.skip].need_grad) need = true;
    p->values[n.out].need_grad = need;
    if (n.skip >= 0) p->values[n.skip].pending_add = n.out;
  }
  return MG_OK;
}

// Gradient buffers share storage when their lifetimes do not overlap (the
// README's buffer-lifetime aliasing).  Positions along the step: the loss is
// 0, the backward of node ni is 1 + (N - 1 - ni).  The gradient of value v is
// written by the loss (the final value) or by the backward of v's consumer;
// it is read by the backward of v's producer, and by the backward that forms
// the gradient of the value whose skip connection ends at v (its dadd term).
// A bias-gradient column sum reads it on the optimizer stream, after the
// fact, so such a buffer is never shared.  Two buffers share a slot only if
// one's last read comes strictly before the other's first write.
void plan_gradients(mg_plan* p, Bump& b) {
  const size_t es = dtype_size(p->dt);
  const size_t B = (size_t)p->batch;
  const int N = (int)p->nodes.size();
  constexpr int kForever = 1 << 30;
  auto pos = [&](int ni) { return 1 + (N - 1 - ni); };
  struct Buf {
    int v, start, end;
    size_t bytes;
  };
  std::vector<Buf> bufs;
  for (size_t vi = 1; vi < p->values.size(); ++vi) {
    Value& v = p->values[vi];
    if (!v.need_grad) continue;
    v.has_grad = true;
    Buf f{(int)vi, 0, 0, B * v.width * es};
    if ((int)vi != p->final_value) {
      f.start = kForever;
      for (int ni = 0; ni < N; ++ni)
        if (p->nodes[ni].in == (int)vi) f.start = std::min(f.start, pos(ni));
    }
    f.end = f.start;
    if (v.producer >= 0) {
      const Node& pr = p->nodes[v.producer];
      f.end = std::max(f.end, pos(v.producer));
      if (pr.kind == NK_LINEAR && pr.has_bias) f.end = kForever;
      if (v.producer == p->defer_dw) f.end = kForever;   // read by the deferred weight gradient
    }
    for (int ni = 0; ni < N; ++ni)
      if (p->values[p->nodes[ni].in].pending_add == (int)vi) f.end = std::max(f.end, pos(ni));
    bufs.push_back(f);
    p->grad_bytes_unaliased += f.bytes;
  }
  std::stable_sort(bufs.begin(), bufs.end(), [](const Buf& a, const Buf& c) { return a.start < c.start; });
  struct Slot {
    size_t bytes;
    int busy_until;
    std::vector<int> members;
  };
  std::vector<Slot> slots;
  for (const Buf& f : bufs) {
    int pick = -1;
    if (p->alias) {
      // the smallest free slot that holds it, else the largest free slot (grown)
      for (size_t k = 0; k < slots.size(); ++k) {
        if (slots[k].busy_until >= f.start) continue;
        if (slots[k].bytes >= f.bytes) {
          if (pick < 0 || slots[pick].bytes < f.bytes || slots[k].bytes < slots[pick].bytes) pick = (int)k;
        } else if (pick < 0 || (slots[pick].bytes < f.bytes && slots[k].bytes > slots[pick].bytes)) {
          pick = (int)k;
        }
      }
    }
    if (pick < 0) {
      slots.push_back(Slot{f.bytes, f.end, {f.v}});
      continue;
    }
    slots[pick].bytes = std::max(slots[pick].bytes, f.bytes);
    slots[pick].busy_until = f.end;
    slots[pick].members.push_back(f.v);
  }
  for (const Slot& sl : slots) {
    const size_t off = b.take(sl.bytes);
    for (int vi : sl.members) p->values[vi].goff = off;
    p->grad_bytes += sl.bytes;
  }
}

// The weight gradient moved to the end of the backward (see mg_plan::defer_dw).
int choose_deferred_dw(const mg_plan* p) {
  int last = -1, smallest = -1;
  auto wcount = [&](int ni) { return (double)p->nodes[ni].d_in * p->nodes[ni].d_out; };
  for (int ni = 0; ni < (int)p->nodes.size(); ++ni) {
    const Node& n = p->nodes[ni];
    if (n.kind != NK_LINEAR || !p->values[n.out].need_grad) continue;
    if (last < 0) last = ni;                    // the backward processes it last
    if (smallest < 0 || wcount(ni) < wcount(smallest)) smallest = ni;
  }
  if (smallest < 0 || smallest == last || wcount(smallest) >= wcount(last)) return -1;
  return smallest;
}

void layout_workspace(mg_plan* p) {
  p->defer_dw = choose_deferred_dw(p);
  Bump b;
  const size_t es = dtype_size(p->dt);
  const size_t B = (size_t)p->batch;
  // saved GELU pre-activations: their own buffers, or one shared buffer that
  // the backward refills (MG_RECOMPUTE_GELU=1)
  std::vector<char> is_z(p->values.size(), 0);
  size_t zmax = 0;
  for (const Node& n : p->nodes)
    if (n.z >= 0) {
      is_z[n.z] = 1;
      zmax = std::max(zmax, (size_t)p->values[n.z].width);
    }
  size_t zshared = 0;
  if (p->recompute_gelu && zmax) zshared = b.take(B * zmax * es);
  for (size_t i = 1; i < p->values.size(); ++i) {
    Value& v = p->values[i];
    v.off = (p->recompute_gelu && is_z[i]) ? zshared : b.take(B * v.width * es);
  }
  plan_gradients(p, b);
  // x's gradient is never formed; a value's need_grad is false for x
  for (Node& n : p->nodes) {
    if (n.kind == NK_RMSNORM) n.rstd_off = b.take(B * 4);
    if (n.kind == NK_ATTN) {
      n.lse_off = b.take(B * n.nh * 4);
      n.dsum_off = b.take(B * n.nh * 4);
    }
  }
  // bias-gradient column partials, one buffer per layer: the optimizer
  // stream sums a layer's partials while the main stream goes on to write the
  // next layer's
  if (p->dt == DT_BF16 && p->use_tc) {
    for (Node& n : p->nodes) {
      if (n.kind != NK_LINEAR || !n.has_bias || !p->values[n.out].need_grad) continue;
      for (const Node& c : p->nodes)
        if (c.in == n.out && c.kind == NK_LINEAR) n.cp_off = b.take((B + 31) / 32 * n.d_out * 4);
    }
  }
  if (p->dt == DT_BF16) p->shadow_off = b.take(p->n_params * 2);
  // chunks
  p->n_chunks = 0;
  for (size_t t = 0; t < p->p_off.size(); ++t) {
    size_t len = (size_t)p->p_rows[t] * p->p_cols[t];
    p->n_chunks += (int)((len + kChunk - 1) / kChunk);
  }
  p->chunks_off = b.take(sizeof(Chunk) * (size_t)p->n_chunks);
  p->loss_off = b.take(16);
  p->scal_off = b.take(16);
  p->flag_off = b.take(16);
  p->rowloss_off = b.take(B * 4);
  size_t part = 0;
  for (auto& n : p->nodes)
    if (n.kind == NK_RMSNORM && (size_t)kNormChunks * n.d * 4 > part) part = (size_t)kNormChunks * n.d * 4;
  if (part < (size_t)kMsePartials * 4) part = (size_t)kMsePartials * 4;
  p->partial_off = b.take(part);
  p->colsum_off = b.take(kColsumFloats * 4);   // the bias-gradient sums' own partials (aux stream)
  // partial tiles of strict weight gradients split over K (main stream only,
  // one at a time): the largest any linear node needs
  p->split_floats = 0;
  if (p->dt == DT_F32) {
    for (const Node& n : p->nodes) {
      if (n.kind != NK_LINEAR) continue;
      GemmArgs g;
      g.M = n.d_in; g.N = n.d_out; g.K = p->batch;
      g.a_mn = 1; g.b_k = 0; g.in_type = DT_F32; g.out_type = DT_F32;
      p->split_floats = std::max(p->split_floats, gemm_simt_split_floats(g));
    }
  }
  p->split_off = b.take(p->split_floats * 4);
  // softmax partials of a cross-entropy head computed by a tensor-core GEMM
  const Value& fv = p->values[p->final_value];
  if (p->dt == DT_BF16 && p->loss != MG_LOSS_MSE && fv.width % 8 == 0 && fv.producer >= 0 &&
      p->nodes[fv.producer].kind == NK_LINEAR) {
    p->lse_parts = (fv.width + 127) / 128;
    p->lse_part_off = b.take(B * (size_t)p->lse_parts * sizeof(float2));
  }
  p->ws_bytes = round_up(b.top, kWsAlign);
}

std::vector<Chunk> chunk_table(mg_plan* p) {
  std::vector<Chunk> t;
  p->tensor_chunk.assign(p->p_off.size() + 1, 0);
  for (size_t i = 0; i < p->p_off.size(); ++i) {
    p->tensor_chunk[i] = (int)t.size();
    size_t len = (size_t)p->p_rows[i] * p->p_cols[i];
    for (size_t s = 0; s < len; s += kChunk) {
      Chunk c;
      c.start = (long long)(p->p_off[i] + s);
      c.len = (int)(len - s < (size_t)kChunk ? len - s : kChunk);
      c.shadow = p->p_is_weight[i];
      t.push_back(c);
    }
  }
  p->tensor_chunk[p->p_off.size()] = (int)t.size();
  return t;
}

void build_dump(mg_plan* p) {
  std::string s;
  char b[256];
  snprintf(b, sizeof b, "plan: batch %d, %s, %s, loss %d, %zu params, workspace %zu bytes\n",
           p->batch, p->dt == DT_BF16 ? "bf16" : "strict-f32",
           p->optimizer == MG_OPT_ADAM     ? "adam"
           : p->optimizer == MG_OPT_LAPROP ? "laprop"
           : p->optimizer == MG_OPT_SGD    ? "sgd"
                                           : "sgd_momentum",
           p->loss, p->n_params, p->ws_bytes);
  s += b;
  snprintf(b, sizeof b, "  gradient storage: %zu bytes (%zu without lifetime sharing%s)\n",
           p->grad_bytes, p->grad_bytes_unaliased, p->alias ? "" : "; MG_NO_ALIAS set");
  s += b;
  if (p->recompute_gelu) s += "  GELU pre-activations: recomputed in the backward (MG_RECOMPUTE_GELU set)\n";
  for (const Node& n : p->nodes)
    if (n.fuse_upd) {
      snprintf(b, sizeof b, "  layer %d: Adam update of the weight fused into its gradient GEMM\n", n.layer);
      s += b;
    }
  if (p->fuse_update && !p->any_fused) s += "  MG_FUSED_UPDATE set: no weight update qualifies\n";
  for (size_t i = 0; i < p->p_off.size(); ++i) {
    snprintf(b, sizeof b, "  param %zu: offset %zu [%d x %d]\n", i, p->p_off[i], p->p_rows[i],
             p->p_cols[i]);
    s += b;
  }
  for (size_t i = 0; i < p->values.size(); ++i) {
    const Value& v = p->values[i];
    snprintf(b, sizeof b, "  value %zu: width %d at ws+%zu%s grad %s\n", i, v.width,
             i == 0 ? (size_t)0 : v.off, i == 0 ? " (caller's x)" : "",
             v.has_grad ? std::to_string(v.goff).c_str() : "-");
    s += b;
  }
  for (size_t i = 0; i < p->sites.size(); ++i) {
    snprintf(b, sizeof b, "  kernel %zu: %s  (%.3g flop, %.3g B)\n", i, p->sites[i].name.c_str(),
             p->sites[i].flops, p->sites[i].bytes);
    s += b;
  }
  p->dump = s;
}

mg_status check_device(mg_plan* p) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(p, e, "cudaGetDevice");
  if (dev != p->device)
    return fail(p, MG_ERR_INVALID_ARG, "plan belongs to device %d but device %d is current", p->device, dev);
  return MG_OK;
}

}  // namespace

void mg::set_global_error(const char* msg) {
  std::lock_guard<std::mutex> lk(g_err_mu);
  g_err = msg;
}

// ============================================================================
namespace {

void drop_graph(mg_plan::StepGraph& g) {
  if (g.gexec) cudaGraphExecDestroy(g.gexec);
  if (g.graph) cudaGraphDestroy(g.graph);
  g.gexec = nullptr;
  g.graph = nullptr;
  g.opt_nodes.clear();
}

// The graph entry for this buffer set (created, evicting the least recently
// used of two, when new).
mg_plan::StepGraph& graph_entry(mg_plan* p, const void* const (&key)[6]) {
  ++p->graph_clock;
  for (auto& g : p->graphs)
    if (memcmp(g.key, key, sizeof g.key) == 0) {
      g.last_use = p->graph_clock;
      return g;
    }
  if (p->graphs.size() >= 2) {
    size_t old = p->graphs[0].last_use <= p->graphs[1].last_use ? 0 : 1;
    drop_graph(p->graphs[old]);
    p->graphs.erase(p->graphs.begin() + old);
  }
  p->graphs.emplace_back();
  mg_plan::StepGraph& g = p->graphs.back();
  memcpy(g.key, key, sizeof g.key);
  g.last_use = p->graph_clock;
  return g;
}

// Capture one step into a graph; false (and nothing kept) if any part of the
// capture fails.
bool capture_step(mg_plan* p, mg_plan::StepGraph& sg, float* params, float* grads,
                  float* m, float* v, const void* x, const void* labels, float lr, int step) {
  // captured on a private stream (the caller's may be the legacy default
  // stream, which cannot be captured); nothing runs during the capture
  if (!p->cap && cudaStreamCreateWithFlags(&p->cap, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (cudaStreamBeginCapture(p->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  Exec ex{p, p->cap, false, false};
  train_schedule(ex, params, grads, m, v, x, labels, lr, step);
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamEndCapture(p->cap, &g);
  if (ex.err != cudaSuccess || e != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return false;
  }
  cudaGraphExec_t ge = nullptr;
  if (cudaGraphInstantiate(&ge, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return false;
  }
  // the optimizer kernel nodes, with a copy of their arguments
  size_t n = 0;
  cudaGraphGetNodes(g, nullptr, &n);
  std::vector<cudaGraphNode_t> nodes(n);
  if (n) cudaGraphGetNodes(g, nodes.data(), &n);
  sg.opt_nodes.clear();
  for (cudaGraphNode_t nd : nodes) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(nd, &t) != cudaSuccess || t != cudaGraphNodeTypeKernel) continue;
    cudaKernelNodeParams kp;
    if (cudaGraphKernelNodeGetParams(nd, &kp) != cudaSuccess) continue;
    mg_plan::OptNode o;
    if (!optimizer_kernel_info(kp.func, &o.info)) continue;
    o.node = nd;
    o.kp = kp;
    for (int i = 0; i < o.info.nargs; ++i) {
      o.arg[i] = 0;
      memcpy(&o.arg[i], kp.kernelParams[i], o.info.size[i]);
    }
    sg.opt_nodes.push_back(o);
  }
  for (auto& o : sg.opt_nodes) {
    for (int i = 0; i < o.info.nargs; ++i) o.argv[i] = &o.arg[i];
    o.kp.kernelParams = o.argv;
    o.kp.extra = nullptr;
  }
  sg.graph = g;
  sg.gexec = ge;
  sg.launches = ex.launches;
  return true;
}

// Relaunch a captured step with this step's optimizer scalars.
cudaError_t replay_step(mg_plan* p, mg_plan::StepGraph& sg, cudaStream_t s, float lr, int step) {
  float lr_bc1 = lr, inv = 1.0f;
  if (p->optimizer == MG_OPT_ADAM || p->optimizer == MG_OPT_LAPROP)
    step_scalars(p, lr, step, &lr_bc1, &inv);
  for (auto& o : sg.opt_nodes) {
    if (o.info.i_lr_bc1 >= 0) memcpy(&o.arg[o.info.i_lr_bc1], &lr_bc1, 4);
    if (o.info.i_inv_sqrt_bc2 >= 0) memcpy(&o.arg[o.info.i_inv_sqrt_bc2], &inv, 4);
    if (o.info.i_lr >= 0) memcpy(&o.arg[o.info.i_lr], &lr, 4);
    cudaError_t e = cudaGraphExecKernelNodeSetParams(sg.gexec, o.node, &o.kp);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaGraphLaunch(sg.gexec, s);
  if (e == cudaSuccess) ++p->graph_replays;
  return e;
}

}  // namespace

extern "C" {

mg_status mg_step_plan_create(const mg_graph_desc* desc, mg_plan** out) {
  if (!out) return fail(nullptr, MG_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!desc) return fail(nullptr, MG_ERR_INVALID_ARG, "desc is NULL");
  mg_plan* p = new (std::nothrow) mg_plan();
  if (!p) return fail(nullptr, MG_ERR_OOM, "host allocation failed");
  mg_status st = compile(p, desc);
  if (st != MG_OK) {
    fail(nullptr, st, "%s", p->err.c_str());
    delete p;
    return st;
  }
  cudaError_t e = cudaGetDevice(&p->device);
  if (e != cudaSuccess) {
    mg_status r = cuda_fail(nullptr, e, "cudaGetDevice");
    delete p;
    return r;
  }
  if (const char* ev = getenv("MG_GEMM")) {
    p->use_tc = strcmp(ev, "simt") != 0;
    p->use_pair = p->use_tc && strcmp(ev, "tc1") != 0;
  }
  if (const char* ev = getenv("MG_NO_ALIAS")) p->alias = !(ev[0] == '1' && ev[1] == 0);
  if (const char* ev = getenv("MG_RECOMPUTE_GELU")) p->recompute_gelu = ev[0] == '1' && ev[1] == 0;
  if (const char* ev = getenv("MG_GRAPH")) p->use_graph = !(ev[0] == '0' && ev[1] == 0);
  if (const char* ev = getenv("MG_FUSED_UPDATE")) p->fuse_update = ev[0] == '1' && ev[1] == 0;
  layout_workspace(p);
  e = cudaMalloc((void**)&p->ws, p->ws_bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    mg_status r = fail(nullptr, MG_ERR_OOM, "workspace of %zu bytes: %s", p->ws_bytes, cudaGetErrorString(e));
    p->ws = nullptr;
    delete p;
    return r;
  }
  std::vector<Chunk> ch = chunk_table(p);
  e = cudaMemcpy(p->ws + p->chunks_off, ch.data(), ch.size() * sizeof(Chunk), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(p->ws + p->loss_off, 0, 16);
  // the optimizer stream gets the lowest priority: when a backward GEMM and
  // optimizer blocks wait for SMs together, the GEMM's CTAs go first
  int prio_lo = 0, prio_hi = 0;
  if (e == cudaSuccess) e = cudaDeviceGetStreamPriorityRange(&prio_lo, &prio_hi);
  if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&p->aux, cudaStreamNonBlocking, prio_lo);
  p->node_ev.assign(2 * p->nodes.size(), nullptr);   // per node: updates, bias-gradient sum
  for (auto& ev : p->node_ev)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->join_ev, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    mg_status r = cuda_fail(nullptr, e, "workspace init");
    for (auto ev : p->node_ev)
      if (ev) cudaEventDestroy(ev);
    if (p->join_ev) cudaEventDestroy(p->join_ev);
    if (p->aux) cudaStreamDestroy(p->aux);
    cudaFree(p->ws);
    delete p;
    return r;
  }
  plan_fused_updates(p);
  // register the schedule's kernels (dry run: no launches)
  Exec ex{p, nullptr, true, false};
  train_schedule(ex, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0.f, 1);
  build_dump(p);
  *out = p;
  return MG_OK;
}

void mg_step_plan_destroy(mg_plan* p) {
  if (!p) return;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(p->device);
  cudaDeviceSynchronize();
  for (auto& g : p->graphs) drop_graph(g);
  if (p->cap) cudaStreamDestroy(p->cap);
  for (auto ev : p->events) cudaEventDestroy(ev);
  for (auto ev : p->node_ev)
    if (ev) cudaEventDestroy(ev);
  if (p->join_ev) cudaEventDestroy(p->join_ev);
  if (p->aux) cudaStreamDestroy(p->aux);
  if (p->ws) cudaFree(p->ws);
  if (prev >= 0) cudaSetDevice(prev);
  delete p;
}

size_t mg_param_count(const mg_plan* p) { return p ? p->n_params : 0; }

int mg_param_tensor_count(const mg_plan* p) { return p ? (int)p->p_off.size() : 0; }

mg_status mg_param_info(const mg_plan* p, int i, size_t* offset, int* rows, int* cols) {
  if (!p) return fail(nullptr, MG_ERR_INVALID_ARG, "plan is NULL");
  if (i < 0 || i >= (int)p->p_off.size())
    return fail(const_cast<mg_plan*>(p), MG_ERR_INVALID_ARG, "tensor index %d out of range", i);
  if (offset) *offset = p->p_off[i];
  if (rows) *rows = p->p_rows[i];
  if (cols) *cols = p->p_cols[i];
  return MG_OK;
}

size_t mg_workspace_bytes(const mg_plan* p) { return p ? p->ws_bytes : 0; }

mg_status mg_forward(mg_plan* p, const float* params, const void* x, float* out, mg_stream_t stream) {
  if (!p) return fail(nullptr, MG_ERR_INVALID_ARG, "plan is NULL");
  if (!params || !x || !out) return fail(p, MG_ERR_INVALID_ARG, "params, x and out must be non-NULL");
  if (!aligned16(params) || !aligned16(x) || !aligned16(out))
    return fail(p, MG_ERR_ALIGN, "params, x and out must be 16-byte aligned");
  mg_status st = check_device(p);
  if (st != MG_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(p, e, "earlier CUDA error");
  Exec ex{p, s, false, false};
  if (p->dt == DT_BF16) {
    site(ex, "cast_bf16_weights", 0, p->n_params * 6.0, 1, [&] {
      return cast_shadow(wsp<Chunk>(p, p->chunks_off), p->n_chunks, params, p->ws + p->shadow_off, s);
    });
    p->last_params = params;
  }
  forward_pass(ex, params, x);
  const Value& f = p->values[p->final_value];
  site(ex, "output_to_f32", 0, 0, 1, [&] {
    return cast_to_f32(p->dt, p->ws + f.off, out, (size_t)p->batch * f.width, s);
  });
  p->last_launches = ex.launches;
  if (ex.err != cudaSuccess) return cuda_fail(p, ex.err, "mg_forward launch");
  return MG_OK;
}

mg_status mg_train_step(mg_plan* p, float* params, float* grads, float* adam_m, float* adam_v,
                        const void* x, const void* labels, float lr, int step, mg_stream_t stream) {
  if (!p) return fail(nullptr, MG_ERR_INVALID_ARG, "plan is NULL");
  if (!params || !grads || !x || !labels)
    return fail(p, MG_ERR_INVALID_ARG, "params, grads, x and labels must be non-NULL");
  const bool two_moments = p->optimizer == MG_OPT_ADAM || p->optimizer == MG_OPT_LAPROP;
  if (two_moments && (!adam_m || !adam_v))
    return fail(p, MG_ERR_INVALID_ARG, "Adam and LaProp need adam_m and adam_v");
  if (p->optimizer == MG_OPT_SGD_MOMENTUM && !adam_m)
    return fail(p, MG_ERR_INVALID_ARG, "SGD with momentum keeps its velocity in adam_m");
  if (two_moments && step < 1) return fail(p, MG_ERR_INVALID_ARG, "step must be >= 1");
  if (!aligned16(params) || !aligned16(grads) || !aligned16(x) || !aligned16(labels) ||
      (adam_m && !aligned16(adam_m)) || (adam_v && !aligned16(adam_v)))
    return fail(p, MG_ERR_ALIGN, "buffers must be 16-byte aligned");
  const size_t nb = p->n_params * sizeof(float);
  const char *pa = (const char*)params, *ga = (const char*)grads;
  if (pa < ga + nb && ga < pa + nb) return fail(p, MG_ERR_INVALID_ARG, "grads must not alias params");
  if (!(std::isfinite(lr))) return fail(p, MG_ERR_INVALID_ARG, "lr is not finite");
  mg_status st = check_device(p);
  if (st != MG_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(p, e, "earlier CUDA error");
  int extra = 0;
  if (p->dt == DT_BF16 && (step == 1 || params != p->last_params)) {
    e = cast_shadow(wsp<Chunk>(p, p->chunks_off), p->n_chunks, params, p->ws + p->shadow_off, s);
    if (e != cudaSuccess) return cuda_fail(p, e, "weight cast");
    extra = 1;
  }
  p->last_params = params;
  // graph replay: the buffers of a captured step, no profiling, and the
  // caller's stream not itself being captured
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  if (p->use_graph && !p->profiling && cs == cudaStreamCaptureStatusNone) {
    const void* key[6] = {params, grads, adam_m, adam_v, x, labels};
    mg_plan::StepGraph& sg = graph_entry(p, key);
    ++sg.calls;
    if (!sg.gexec && sg.calls >= 2 &&
        !capture_step(p, sg, params, grads, adam_m, adam_v, x, labels, lr, step))
      p->use_graph = false;   // capture unavailable here: launch directly from now on
    if (sg.gexec) {
      e = replay_step(p, sg, s, lr, step);
      if (e != cudaSuccess) return cuda_fail(p, e, "mg_train_step graph launch");
      p->last_launches = extra + sg.launches;
      return MG_OK;
    }
  }
  Exec ex{p, s, false, true};
  ex.launches = extra;
  train_schedule(ex, params, grads, adam_m, adam_v, x, labels, lr, step);
  if (p->profiling && p->prof_calls < p->prof_max) p->prof_calls++;
  p->last_launches = ex.launches;
  if (ex.err != cudaSuccess) return cuda_fail(p, ex.err, "mg_train_step launch");
  return MG_OK;
}

mg_status mg_loss(mg_plan* p, float* host_loss, mg_stream_t stream) {
  if (!p || !host_loss) return fail(p, MG_ERR_INVALID_ARG, "plan and host_loss must be non-NULL");
  struct { float loss; int err; } h = {0.f, 0};
  cudaError_t e = cudaMemcpyAsync(&h, p->ws + p->loss_off, sizeof h, cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(p, e, "mg_loss");
  *host_loss = h.loss;
  if (h.err) {
    cudaMemsetAsync(err_word(p), 0, sizeof(int), (cudaStream_t)stream);
    return fail(p, MG_ERR_TIMEOUT, "a tensor-core pipeline wait timed out; results are invalid");
  }
  return MG_OK;
}

mg_status mg_loss_async(mg_plan* p, void* host_dst, mg_stream_t stream) {
  if (!p || !host_dst) return fail(p, MG_ERR_INVALID_ARG, "plan and host_dst must be non-NULL");
  cudaError_t e = cudaMemcpyAsync(host_dst, p->ws + p->loss_off, 8, cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(p, e, "mg_loss_async");
  return MG_OK;
}

const float* mg_loss_device_ptr(const mg_plan* p) {
  return p ? reinterpret_cast<const float*>(p->ws + p->loss_off) : nullptr;
}

mg_status mg_refresh_params(mg_plan* p, const float* params, mg_stream_t stream) {
  if (!p || !params) return fail(p, MG_ERR_INVALID_ARG, "plan and params must be non-NULL");
  if (!aligned16(params)) return fail(p, MG_ERR_ALIGN, "params must be 16-byte aligned");
  if (p->dt != DT_BF16) return MG_OK;
  cudaError_t e = cast_shadow(wsp<Chunk>(p, p->chunks_off), p->n_chunks, params, p->ws + p->shadow_off,
                              (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(p, e, "mg_refresh_params");
  p->last_params = params;
  return MG_OK;
}

// ---- checkpoints -------------------------------------------------------------
// The paper's checkpoint notes: logical tensors without device padding, and a
// restore that is checked before anything is changed.  Layout (little-endian):
// a 64-byte header (magic, version, tensor count, section flags, precision,
// floats per section, checksum), the tensors' (rows, cols), then the sections
// params, first moment, second moment, each the tensors' values back to back.
namespace {

constexpr char kCkptMagic[8] = {'M', 'G', 'C', 'K', 'P', 'T', 0, 1};
constexpr uint32_t kCkptVersion = 1;
constexpr size_t kCkptHeader = 64;

struct CkptHeader {
  char magic[8];
  uint32_t version, n_tensors, flags, precision;
  uint64_t floats, checksum;
  uint8_t reserved[24];
};
static_assert(sizeof(CkptHeader) == kCkptHeader, "checkpoint header is 64 bytes");

size_t logical_floats(const mg_plan* p) {
  size_t n = 0;
  for (size_t t = 0; t < p->p_off.size(); ++t) n += (size_t)p->p_rows[t] * p->p_cols[t];
  return n;
}

size_t ckpt_bytes(const mg_plan* p, int sections) {
  return kCkptHeader + 8 * p->p_off.size() + 4 * logical_floats(p) * sections;
}

// 64-bit multiply-xorshift hash of the data sections, eight bytes at a time.
uint64_t ckpt_hash(const uint8_t* d, size_t n) {
  uint64_t h = 0x9E3779B97F4A7C15ull ^ n;
  size_t i = 0;
  for (; i + 8 <= n; i += 8) {
    uint64_t w;
    memcpy(&w, d + i, 8);
    h = (h ^ w) * 0xBF58476D1CE4E5B9ull;
    h ^= h >> 31;
  }
  for (; i < n; ++i) h = (h ^ d[i]) * 0x100000001B3ull;
  return h ^ (h >> 29);
}

}  // namespace

size_t mg_checkpoint_bytes(const mg_plan* p, int with_m, int with_v) {
  if (!p) return 0;
  return ckpt_bytes(p, 1 + (with_m ? 1 : 0) + (with_v ? 1 : 0));
}

mg_status mg_checkpoint_save(mg_plan* p, const float* params, const float* m, const float* v,
                             void* host_buf, size_t cap, size_t* written, mg_stream_t stream) {
  if (!p || !params || !host_buf) return fail(p, MG_ERR_INVALID_ARG, "plan, params and buffer must be non-NULL");
  if (!m && v) return fail(p, MG_ERR_INVALID_ARG, "a second moment without a first one");
  const int sections = 1 + (m ? 1 : 0) + (v ? 1 : 0);
  const size_t need = ckpt_bytes(p, sections);
  if (written) *written = 0;
  if (cap < need) return fail(p, MG_ERR_INVALID_ARG, "checkpoint needs %zu bytes, buffer has %zu", need, cap);
  cudaSetDevice(p->device);
  uint8_t* out = static_cast<uint8_t*>(host_buf);
  const size_t nt = p->p_off.size(), lf = logical_floats(p);
  uint8_t* data = out + kCkptHeader + 8 * nt;
  const float* src[3] = {params, m, v};
  for (int sct = 0; sct < sections; ++sct) {
    float* dst = reinterpret_cast<float*>(data + 4 * lf * sct);
    for (size_t t = 0; t < nt; ++t) {
      const size_t len = (size_t)p->p_rows[t] * p->p_cols[t];
      cudaError_t e = cudaMemcpyAsync(dst, src[sct] + p->p_off[t], len * 4, cudaMemcpyDeviceToHost,
                                      (cudaStream_t)stream);
      if (e != cudaSuccess) return cuda_fail(p, e, "checkpoint save copy");
      dst += len;
    }
  }
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(p, e, "checkpoint save");
  CkptHeader h;
  memset(&h, 0, sizeof h);
  memcpy(h.magic, kCkptMagic, 8);
  h.version = kCkptVersion;
  h.n_tensors = (uint32_t)nt;
  h.flags = (m ? 1u : 0u) | (v ? 2u : 0u);
  h.precision = (uint32_t)p->precision;
  h.floats = lf;
  h.checksum = ckpt_hash(data, 4 * lf * sections);
  memcpy(out, &h, sizeof h);
  for (size_t t = 0; t < nt; ++t) {
    const uint32_t rc[2] = {(uint32_t)p->p_rows[t], (uint32_t)p->p_cols[t]};
    memcpy(out + kCkptHeader + 8 * t, rc, 8);
  }
  if (written) *written = need;
  return MG_OK;
}

mg_status mg_checkpoint_load(mg_plan* p, const void* host_buf, size_t len, float* params,
                             float* m, float* v, mg_stream_t stream) {
  if (!p || !host_buf || !params) return fail(p, MG_ERR_INVALID_ARG, "plan, buffer and params must be non-NULL");
  // ---- preflight: every check before the first write
  if (!aligned16(params) || (m && !aligned16(m)) || (v && !aligned16(v)))
    return fail(p, MG_ERR_ALIGN, "params and moments must be 16-byte aligned");
  const uint8_t* in = static_cast<const uint8_t*>(host_buf);
  if (len < kCkptHeader) return fail(p, MG_ERR_INVALID_ARG, "checkpoint: %zu bytes is shorter than the header", len);
  CkptHeader h;
  memcpy(&h, in, sizeof h);
  if (memcmp(h.magic, kCkptMagic, 8) != 0) return fail(p, MG_ERR_INVALID_ARG, "checkpoint: bad magic");
  if (h.version != kCkptVersion) return fail(p, MG_ERR_UNSUPPORTED, "checkpoint: version %u", h.version);
  const size_t nt = p->p_off.size(), lf = logical_floats(p);
  if (h.n_tensors != nt)
    return fail(p, MG_ERR_SHAPE, "checkpoint holds %u tensors, the plan has %zu", h.n_tensors, nt);
  if (h.floats != lf) return fail(p, MG_ERR_SHAPE, "checkpoint holds %llu values per section, the plan %zu",
                                  (unsigned long long)h.floats, lf);
  if (h.flags & ~3u || ((h.flags & 2u) && !(h.flags & 1u)))
    return fail(p, MG_ERR_INVALID_ARG, "checkpoint: bad section flags %u", h.flags);
  const int sections = 1 + ((h.flags & 1u) ? 1 : 0) + ((h.flags & 2u) ? 1 : 0);
  if (len != ckpt_bytes(p, sections))
    return fail(p, MG_ERR_SHAPE, "checkpoint is %zu bytes, its header describes %zu", len, ckpt_bytes(p, sections));
  for (size_t t = 0; t < nt; ++t) {
    uint32_t rc[2];
    memcpy(rc, in + kCkptHeader + 8 * t, 8);
    if ((int)rc[0] != p->p_rows[t] || (int)rc[1] != p->p_cols[t])
      return fail(p, MG_ERR_SHAPE, "checkpoint tensor %zu is %ux%u, the plan's is %dx%d", t, rc[0], rc[1],
                  p->p_rows[t], p->p_cols[t]);
  }
  if (m && !(h.flags & 1u)) return fail(p, MG_ERR_INVALID_ARG, "checkpoint has no first moment");
  if (v && !(h.flags & 2u)) return fail(p, MG_ERR_INVALID_ARG, "checkpoint has no second moment");
  const uint8_t* data = in + kCkptHeader + 8 * nt;
  if (ckpt_hash(data, 4 * lf * sections) != h.checksum)
    return fail(p, MG_ERR_INVALID_ARG, "checkpoint: checksum mismatch (corrupted data)");
  // ---- restore
  cudaSetDevice(p->device);
  float* dst[3] = {params, m, v};
  for (int sct = 0; sct < 3; ++sct) {
    if (!dst[sct]) continue;
    const float* src = reinterpret_cast<const float*>(data + 4 * lf * sct);
    for (size_t t = 0; t < nt; ++t) {
      const size_t n = (size_t)p->p_rows[t] * p->p_cols[t];
      cudaError_t e = cudaMemcpyAsync(dst[sct] + p->p_off[t], src, n * 4, cudaMemcpyHostToDevice,
                                      (cudaStream_t)stream);
      if (e != cudaSuccess) return cuda_fail(p, e, "checkpoint restore copy");
      src += n;
    }
  }
  mg_status st = mg_refresh_params(p, params, stream);
  if (st != MG_OK) return st;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(p, e, "checkpoint restore");
  return MG_OK;
}

size_t mg_plan_dump(const mg_plan* p, char* buf, size_t cap) {
  if (!p) return 0;
  if (buf && cap) {
    size_t n = p->dump.size() < cap - 1 ? p->dump.size() : cap - 1;
    memcpy(buf, p->dump.data(), n);
    buf[n] = 0;
  }
  return p->dump.size();
}

const char* mg_last_error(const mg_plan* p) {
  if (p) return p->err.c_str();
  std::lock_guard<std::mutex> lk(g_err_mu);
  return g_err.c_str();
}

mg_status mg_debug_check_finite(mg_plan* p, const float* data, size_t n, long long* first_bad,
                                mg_stream_t stream) {
  if (!p || !data) return fail(p, MG_ERR_INVALID_ARG, "plan and data must be non-NULL");
  cudaStream_t s = (cudaStream_t)stream;
  unsigned long long* flag = wsp<unsigned long long>(p, p->flag_off);
  unsigned long long h = ~0ull;
  cudaError_t e = cudaMemcpyAsync(flag, &h, sizeof h, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = find_nonfinite(data, n, flag, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h, flag, sizeof h, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(p, e, "mg_debug_check_finite");
  if (first_bad) *first_bad = h == ~0ull ? -1 : (long long)h;
  if (h != ~0ull) return fail(p, MG_ERR_NONFINITE, "non-finite value at index %llu", h);
  return MG_OK;
}

int mg_last_launch_count(const mg_plan* p) { return p ? p->last_launches : 0; }

long long mg_graph_replays(const mg_plan* p) { return p ? p->graph_replays : 0; }

mg_status mg_profile_begin(mg_plan* p, int max_calls) {
  if (!p || max_calls <= 0) return fail(p, MG_ERR_INVALID_ARG, "bad profile request");
  for (auto ev : p->events) cudaEventDestroy(ev);
  p->events.assign((size_t)max_calls * p->sites.size() * 2, nullptr);
  for (auto& ev : p->events) {
    cudaError_t e = cudaEventCreate(&ev);
    if (e != cudaSuccess) return cuda_fail(p, e, "cudaEventCreate");
  }
  for (auto& s : p->sites) {
    s.launches = 0;
    s.total_ms = 0;
  }
  p->profiling = true;
  p->prof_max = max_calls;
  p->prof_calls = 0;
  return MG_OK;
}

mg_status mg_profile_end(mg_plan* p) {
  if (!p || !p->profiling) return fail(p, MG_ERR_INVALID_ARG, "profiling not active");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(p, e, "mg_profile_end");
  const size_t ns = p->sites.size();
  for (int c = 0; c < p->prof_calls; ++c)
    for (size_t i = 0; i < ns; ++i) {
      float ms = 0;
      if (cudaEventElapsedTime(&ms, p->events[(c * ns + i) * 2], p->events[(c * ns + i) * 2 + 1]) ==
          cudaSuccess) {
        p->sites[i].launches++;
        p->sites[i].total_ms += ms;
      } else {
        cudaGetLastError();
      }
    }
  p->profiling = false;
  return MG_OK;
}

int mg_profile_entries(const mg_plan* p) { return p ? (int)p->sites.size() : 0; }

mg_status mg_profile_entry(const mg_plan* p, int i, char* name, size_t name_cap, int* launches,
                           double* total_ms, double* flops, double* bytes) {
  if (!p || i < 0 || i >= (int)p->sites.size()) return fail(const_cast<mg_plan*>(p), MG_ERR_INVALID_ARG, "bad entry");
  const Site& s = p->sites[i];
  if (name && name_cap) {
    size_t n = s.name.size() < name_cap - 1 ? s.name.size() : name_cap - 1;
    memcpy(name, s.name.data(), n);
    name[n] = 0;
  }
  if (launches) *launches = s.launches;
  if (total_ms) *total_ms = s.total_ms;
  if (flops) *flops = s.flops;
  if (bytes) *bytes = s.bytes;
  return MG_OK;
}

}  // extern "C"
