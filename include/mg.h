/*
 * mg.h -- C ABI of the GB300 training-step library (libmg.so).
 *
 * One training step of a typed static graph -- forward pass, hand-derived
 * backward pass and optimizer update -- on one GPU, behind a fixed-shape plan.
 * The operation follows the Meganeura pages: "Meganeura" README, Example
 * section (a graph of input / parameter / matmul / relu / cross_entropy_loss
 * nodes, built once with build_session and stepped by a Trainer), Contents
 * section (SGD, Adam), Environment variables section (strict f32 scalar matmul
 * versus validated reduced-precision tiles); and the abstract of "Meganeura:
 * Portable GPU Training and Inference through Vulkan and Metal" (typed static
 * graph, automatic differentiation, optimizer, memory planner, runtime; strict
 * f32 kept apart from validated fast paths).
 *
 * Conventions for every call:
 *  - Pointers named params/grads/adam_m/adam_v/x/labels/out are DEVICE
 *    pointers owned by the caller (e.g. from torch tensors) and must be
 *    16-byte aligned.  The plan never frees them.
 *  - Everything is asynchronous on `stream` (a cudaStream_t; 0 = legacy
 *    default stream) except mg_loss, which synchronises it.
 *  - Every call returns an mg_status; nothing aborts, throws across the ABI or
 *    traps on the device.  mg_last_error() returns the message of the last
 *    failure (per plan, or process-wide for a NULL plan).
 *  - A plan is bound to the CUDA device that was current at creation and is not
 *    thread-safe: drive it from one host thread and one stream at a time.
 */
#ifndef MG_H
#define MG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mg_plan mg_plan;          /* opaque; owns the workspace */
typedef struct CUstream_st* mg_stream_t; /* same type as cudaStream_t */

typedef enum {
  MG_OK = 0,
  MG_ERR_INVALID_ARG = -1, /* NULL where a pointer is required, bad enum, bad value */
  MG_ERR_UNSUPPORTED = -2, /* a valid graph this library has no kernels for */
  MG_ERR_SHAPE = -3,       /* widths that do not chain, batch not a multiple of seq_len */
  MG_ERR_ALIGN = -4,       /* a pointer that is not 16-byte aligned */
  MG_ERR_OOM = -5,         /* workspace allocation failed (nothing leaked) */
  MG_ERR_CUDA = -6,        /* a CUDA runtime/driver error (launch or earlier async fault) */
  MG_ERR_NONFINITE = -7,   /* mg_debug_check_finite found a NaN or Inf */
  MG_ERR_TIMEOUT = -8,     /* a bounded device-side wait gave up */
  MG_ERR_INTERNAL = -9
} mg_status;

typedef enum {
  MG_OP_LINEAR = 0,           /* Y = X W (+ b), W[d_in, d_out] row-major, b[d_out] */
  MG_OP_RELU = 1,             /* max(z, 0); derivative 0 at z = 0 */
  MG_OP_GELU_TANH = 2,        /* 0.5 z (1 + tanh(sqrt(2/pi)(z + 0.044715 z^3))) */
  MG_OP_RMSNORM = 3,          /* y = x / sqrt(mean(x^2) + eps) * gamma, gamma[d] */
  MG_OP_RESIDUAL_BEGIN = 4,   /* remember the current value as the skip input */
  MG_OP_RESIDUAL_END = 5,     /* value = skip + value */
  MG_OP_CAUSAL_ATTENTION = 6  /* input [rows, 3d] = [Q|K|V], output [rows, d], d = n_heads*head_dim */
} mg_op;

typedef enum { MG_LOSS_CE_DENSE = 0, MG_LOSS_CE_INDEX = 1, MG_LOSS_MSE = 2 } mg_loss_kind;
typedef enum { MG_PREC_STRICT_F32 = 0, MG_PREC_BF16 = 1 } mg_precision;
/* SGD: p -= lr g.  ADAM: bias-corrected moments, eps after the root.  LAPROP
 * (named beside Adam in the paper's checkpoint notes; the update is the
 * published LaProp algorithm): v = b2 v + (1-b2) g^2, m = b1 m + (1-b1) g /
 * (sqrt(v / (1 - b2^t)) + eps), p -= lr m / (1 - b1^t).  SGD_MOMENTUM:
 * heavy ball, b = beta1 b + g, p -= lr b (beta1 is the momentum). */
typedef enum {
  MG_OPT_SGD = 0,
  MG_OPT_ADAM = 1,
  MG_OPT_LAPROP = 2,
  MG_OPT_SGD_MOMENTUM = 3
} mg_optimizer;

typedef struct {
  int op;        /* mg_op */
  int d_in;      /* LINEAR: input width; RMSNORM: width */
  int d_out;     /* LINEAR: output width */
  int has_bias;  /* LINEAR: 1 if a bias vector follows W in the parameters */
  float eps;     /* RMSNORM: epsilon inside the square root */
  int n_heads;   /* CAUSAL_ATTENTION */
  int head_dim;  /* CAUSAL_ATTENTION (64 supported) */
  int seq_len;   /* CAUSAL_ATTENTION: rows are [batch, seq_len] flattened */
} mg_layer;

typedef struct {
  int batch;               /* rows of x (tokens) */
  int n_layers;
  const mg_layer* layers;  /* copied at creation */
  int loss;                /* mg_loss_kind, applied to the last layer's output */
  int precision;           /* mg_precision */
  int optimizer;           /* mg_optimizer */
  float beta1, beta2, adam_eps;
} mg_graph_desc;

/* Build a plan for the current CUDA device: validate the descriptor, assign
 * parameter offsets, choose a kernel per GEMM, allocate the workspace once.
 * On failure *out is set to NULL and nothing is leaked.  The descriptor is the
 * typed static graph of the README's Example section, with its shapes fixed. */
mg_status mg_step_plan_create(const mg_graph_desc* desc, mg_plan** out);

/* Free the workspace.  NULL is a no-op.  Synchronises the device first.
 * (The session that build_session returns owns its device buffers for its
 * lifetime: "Meganeura" README, Example section.) */
void mg_step_plan_destroy(mg_plan* plan);

/* Floats in each of the flat parameter / gradient / moment buffers (the
 * parameter nodes of the README's Example section, packed). */
size_t mg_param_count(const mg_plan* plan);

/* Number of parameter tensors (W, b, gamma in declaration order): the graph's
 * parameter nodes ("Meganeura" README, Example section). */
int mg_param_tensor_count(const mg_plan* plan);

/* Tensor i of the flat buffers: element offset, logical rows and cols (a
 * vector has rows = 1).  Offsets are multiples of 64 elements; the gaps
 * between tensors are never read or written.  The logical shape is the one a
 * checkpoint stores, without device padding ("Meganeura" README, Contents
 * section, checkpoint notes). */
mg_status mg_param_info(const mg_plan* plan, int i, size_t* offset, int* rows, int* cols);

/* Bytes of device workspace the plan owns, after the memory planner's
 * lifetime sharing of gradient buffers (abstract of "Meganeura: Portable GPU
 * Training and Inference through Vulkan and Metal": memory planner; README,
 * Environment variables section: buffer lifetime aliasing, off with
 * MG_NO_ALIAS=1 here).  With MG_RECOMPUTE_GELU=1 at plan creation the GELU
 * pre-activations are not kept: the backward recomputes each one (the
 * forward's GEMM again, same inputs and weights, same result) into a single
 * shared buffer just before the input-gradient GEMM that needs it. */
size_t mg_workspace_bytes(const mg_plan* plan);

/* Forward pass only: the inference side of the train-to-deploy stack (README,
 * Contents section: a trained model reloaded into a fresh inference session;
 * abstract: one graph and runtime for training and deployed inference).
 * params: flat fp32 [mg_param_count]; x: [batch, d_in], fp32 in strict mode,
 * bf16 in bf16 mode; out: fp32 [batch, d_out] (logits or the model output),
 * written row-major; in bf16 mode each output value is the bf16 value the
 * graph stores, widened. */
mg_status mg_forward(mg_plan* plan, const float* params, const void* x, float* out,
                     mg_stream_t stream);

/* One full training step: forward, loss, backward, optimizer update (README,
 * Example section: the Trainer's step over the session; Contents section: SGD
 * and Adam; abstract: automatic differentiation and optimizer).
 *  params  fp32 [P]  updated in place (fp32 master weights)
 *  grads   fp32 [P]  overwritten with dLoss/dparams of this step (before the update)
 *  adam_m, adam_v fp32 [P]  optimizer state, updated in place: Adam and LaProp
 *          use both (first and second moment); SGD_MOMENTUM keeps its velocity
 *          in adam_m (adam_v may be NULL); plain SGD needs neither
 *  x       [batch, d_in], fp32 (strict) or bf16 (bf16)
 *  labels  CE_DENSE: fp32 [batch, C]; CE_INDEX: int32 [batch], values in [0, C);
 *          MSE: target [batch, d_out] in the activation dtype (fp32 / bf16)
 *  lr      learning rate; step: Adam's / LaProp's t, 1-based (ignored by SGD)
 * The loss of the step is kept on the device (mg_loss, mg_loss_device_ptr).
 * grads must not alias params.  The bf16 weight copy used by the bf16 path is
 * refreshed from params automatically when step == 1 or params differs from the
 * previous call; otherwise the previous update has kept it current.
 * Graph replay: the second call with the same six buffer addresses captures
 * the step's launches (both streams) into a CUDA graph, and that call and
 * later ones with those addresses launch the graph on `stream`, with lr and
 * the bias corrections of `step` written into its optimizer nodes.  Graphs
 * are kept for the two most recently used address sets (double-buffered
 * inputs).  Results are the same as launching each kernel.  Not used while
 * profiling or when `stream` is itself being captured; the environment
 * variable MG_GRAPH=0, read at plan creation, turns it off.  If a capture
 * fails the plan launches directly from then on.
 * With MG_FUSED_UPDATE=1 at plan creation (Adam, bf16) a weight whose
 * gradient GEMM runs on the tensor cores without a split over K is updated in
 * that GEMM's epilogue instead of the optimizer kernel: same results, one
 * launch fewer per such layer. */
mg_status mg_train_step(mg_plan* plan, float* params, float* grads, float* adam_m,
                        float* adam_v, const void* x, const void* labels, float lr, int step,
                        mg_stream_t stream);

/* Copy the last step's loss (the batch mean the README's Example section
 * prints per step) to the host; synchronises `stream`. */
mg_status mg_loss(mg_plan* plan, float* host_loss, mg_stream_t stream);

/* Enqueue, without waiting, a copy of the last step's loss and the plan's
 * pipeline error word to host memory: host_dst receives { float loss; int
 * timed_out; } (8 bytes; pinned memory keeps the copy asynchronous).  The
 * values are valid once `stream` has passed this point (an event, a later
 * synchronisation).  A nonzero timed_out means that step's results are
 * invalid; mg_loss reports it as MG_ERR_TIMEOUT and clears it.  For training
 * loops that enqueue the next step before reading this one's loss. */
mg_status mg_loss_async(mg_plan* plan, void* host_dst, mg_stream_t stream);

/* Device address of the last step's loss (one fp32, the batch mean of the
 * README's Example section), valid until destroy. */
const float* mg_loss_device_ptr(const mg_plan* plan);

/* Re-derive the bf16 weight copy from params (after the caller changed them,
 * e.g. a checkpoint restore).  A no-op in strict mode.  The copy is the
 * reduced-precision operand of the validated fast path, kept apart from the
 * strict f32 path (abstract; README, Environment variables section). */
mg_status mg_refresh_params(mg_plan* plan, const float* params, mg_stream_t stream);

/* ---- checkpoints --------------------------------------------------------
 * The paper's checkpoint notes: a checkpoint stores the logical tensors (no
 * device padding) and a restore is checked in full before it changes
 * anything.  Host-memory image, little-endian:
 *   64-byte header: magic "MGCKPT\0\1", u32 version (1), u32 tensor count,
 *     u32 flags (bit 0: first moment stored, bit 1: second moment stored),
 *     u32 precision of the saving plan, u64 values per section, u64 checksum
 *     of the sections, 24 reserved bytes;
 *   per tensor (mg_param_info order): u32 rows, u32 cols;
 *   sections, fp32: params, then the first moment, then the second moment,
 *     each the tensors' values back to back.
 * mg_checkpoint_bytes: the image size with the given sections.
 * mg_checkpoint_save: params (and m, v when non-NULL; v needs m) from the
 *   device into host_buf (cap bytes); *written gets the size; synchronises
 *   stream.  MG_ERR_INVALID_ARG when cap is too small.
 * mg_checkpoint_load: checks magic, version, tensor count and every shape
 *   against this plan, the size, the requested sections' presence and the
 *   checksum -- any failure returns an error with no device memory changed --
 *   then copies params (and m, v when non-NULL; moments stored but not asked
 *   for are skipped, e.g. when a forward-only or SGD plan takes a trained
 *   model) and refreshes the bf16 weight copy; synchronises stream.  The
 *   plan may differ from the saving one in everything but the tensors'
 *   shapes (precision, optimizer, batch). */
size_t mg_checkpoint_bytes(const mg_plan* plan, int with_m, int with_v);
mg_status mg_checkpoint_save(mg_plan* plan, const float* params, const float* m, const float* v,
                             void* host_buf, size_t cap, size_t* written, mg_stream_t stream);
mg_status mg_checkpoint_load(mg_plan* plan, const void* host_buf, size_t len, float* params,
                             float* m, float* v, mg_stream_t stream);

/* Human-readable schedule: one line per kernel with its shapes and the
 * workspace offsets: the dispatch order and alias map that the README's plan
 * dump switch prints at build (Environment variables section).  Writes at
 * most cap bytes including the terminating NUL; returns the full length. */
size_t mg_plan_dump(const mg_plan* plan, char* buf, size_t cap);

/* Message of the last failure; NULL plan gives the process-wide message.
 * (The pages have no counterpart: this is the ABI's error convention, in
 * place of the Rust API's panics and structured errors.) */
const char* mg_last_error(const mg_plan* plan);

/* Scan n floats (device) for NaN/Inf; synchronises stream.  Returns
 * MG_ERR_NONFINITE and the first bad index in *first_bad (may be NULL).  The
 * debug session's scan for the first NaN/Inf after a step ("Meganeura"
 * README, Debugging section). */
mg_status mg_debug_check_finite(mg_plan* plan, const float* data, size_t n, long long* first_bad,
                                mg_stream_t stream);

/* Kernels launched by the last mg_train_step / mg_forward call (a replayed
 * step counts the kernels its graph holds): the dispatch count of the
 * README's per-dispatch profile (Profiling section). */
int mg_last_launch_count(const mg_plan* plan);

/* mg_train_step calls served by a graph replay since the plan was created.
 * The step is compiled once and its fixed command list submitted every step
 * (README, Example section: build_session compiles once); here that list is
 * a CUDA graph. */
long long mg_graph_replays(const mg_plan* plan);

/* ---- per-kernel timing (CUDA events around each launch) ----------------
 * The per-dispatch timing profile of the README's Profiling section, with
 * CUDA events in place of hardware timestamp queries.
 * mg_profile_begin(plan, max_calls): from now on, each mg_train_step records
 * a start/stop event pair around every kernel, for up to max_calls calls.
 * mg_profile_end: synchronises, sums the elapsed time per schedule entry and
 * stops recording.  mg_profile_entry reads entry i (a kernel of the step):
 * its name, launches recorded, total milliseconds, and the algorithmic flops
 * and DRAM bytes of one launch. */
mg_status mg_profile_begin(mg_plan* plan, int max_calls);
mg_status mg_profile_end(mg_plan* plan);
int mg_profile_entries(const mg_plan* plan);
mg_status mg_profile_entry(const mg_plan* plan, int i, char* name, size_t name_cap,
                           int* launches, double* total_ms, double* flops, double* bytes);

/* ---- measurement ---------------------------------------------------------
 * The pages have no counterpart to this call: it measures the roofline
 * denominator of the strict-f32 path, whose matrix products run on the FP32
 * FFMA units only (the strict scalar matmul of the "Meganeura" README,
 * Environment variables section).  Runs a fused multiply-add kernel on every
 * SM of the current device for a few milliseconds, synchronises `stream`,
 * and writes the achieved FP32 TFLOP/s (2 flop per FFMA) to *tflops and the
 * same rate in flop per SM per clock of the device's maximum SM clock to
 * *flop_per_clk_per_sm (may be NULL; 0 if the clock rate is not reported).
 * It allocates and frees a few bytes of device memory. */
mg_status mg_ffma_peak(double* tflops, double* flop_per_clk_per_sm, mg_stream_t stream);

/* ---- softmax cross-entropy without device allocation -----------------
 * The Meganeura pages have no counterpart to this call.  It is for callers
 * that may not allocate device memory -- for example code running inside
 * another framework's plugin or kernel-enqueue hook, or a process whose device
 * memory is already reserved by its own caching allocator -- and therefore
 * cannot create a plan, whose workspace mg_step_plan_create allocates.
 *
 * Computes the same softmax cross-entropy loss and gradient as the training
 * step's loss kernel: for logits [rows, cols] row-major (dtype 0 = fp32,
 * 1 = bf16), labels dense fp32 [rows, cols] (label_kind 0) or int32 class ids
 * [rows] (label_kind 1), it writes dlogits (same dtype and layout as logits)
 * = (softmax * sum(y) - y) / rows and *loss (one fp32, device memory) = the
 * mean over rows of -sum_c y_c log softmax_c.  All pointers are caller-owned
 * device memory; nothing is allocated, and no cudaMalloc, cudaFree or
 * allocating library routine is called.
 *
 * Scratch: the per-row losses go to a fixed array in the library's device
 * memory of 65536 floats (256 KB), held by every GPU that loads the library
 * until the process exits.  rows above 65536 return MG_ERR_INVALID_ARG.  The
 * first call in each device context (the first call on a device, and the
 * first after a cudaDeviceReset re-creates the context) looks up that array's
 * device address with that device current; make that first call before any
 * stream capture.  All calls share the array: calls that overlap on the GPU
 * (different streams, or different host threads) race and give wrong results.
 * Each call overwrites the slots it reads, so nothing needs clearing between
 * calls.  A CUDA error already pending on the calling thread is returned as
 * MG_ERR_CUDA (the message says it came before the call) and nothing is
 * launched; launch failures carry the CUDA error string in the message. */
mg_status mg_softmax_ce_noalloc(int dtype, const void* logits, int rows, int cols, int label_kind,
                                const void* labels, void* dlogits, float* loss, mg_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MG_H */
