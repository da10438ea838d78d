// Internal (host-side) launchers of the training-step kernels.  Not part of
// the C ABI; the plan in plan.cu calls these.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mg {

enum DType { DT_F32 = 0, DT_BF16 = 1 };
enum Act { ACT_NONE = 0, ACT_RELU = 1, ACT_GELU = 2 };

inline size_t dtype_size(DType t) { return t == DT_F32 ? 4 : 2; }

// C[M,N] = A[M,K] * B[K,N] with fp32 accumulation and a fused epilogue:
//   v = acc (+ bias[n]);  out_z = v;  v = act(v);  v *= act'(saved);  v += resid;  out = v
// A(m,k) = a_mn ? A[k*lda + m] : A[m*lda + k]       (M-major or K-major storage)
// B(k,n) = b_k  ? B[n*ldb + k] : B[k*ldb + n]       (K-major or N-major storage)
struct GemmArgs {
  int M = 0, N = 0, K = 0;
  const void* A = nullptr; long long lda = 0; int a_mn = 0;
  const void* B = nullptr; long long ldb = 0; int b_k = 0;
  DType in_type = DT_F32;
  const float* bias = nullptr;
  int act = 0;
  void* out_z = nullptr; long long ldz = 0;
  const void* saved = nullptr; long long lds = 0; int dact = 0;
  const void* resid = nullptr; long long ldr = 0;
  DType aux_type = DT_F32;   // dtype of out_z, saved, resid
  void* out = nullptr; long long ldo = 0;
  DType out_type = DT_F32;
  // Softmax partials of the stored outputs (tcgen05 kernels; outputs with no
  // activation, residual or saved value): for row m and 128-column chunk k,
  // lse_part[m * lse_ld + k] = (max of y, sum of 2^(y - max)) over the chunk's
  // columns below N, y = x log2(e), x the value as stored (bias added, rounded
  // to out_type).
  float2* lse_part = nullptr; int lse_ld = 0;
  // Scratch for the strict weight-gradient GEMM's split over K (floats), or
  // null: each split writes its partial tile there and one pass adds the
  // splits in order (deterministic, unlike atomics).
  float* split_ws = nullptr; size_t split_ws_floats = 0;
  // Column partial sums of the stored output (tcgen05 kernels, bf16 outputs,
  // no split over K), or null: col_part[(m / 32) * N + n] = sum of the stored
  // out[m', n] over the rows m' of the 32-row group of m, fixed order.  The
  // bias gradient of the layer whose output gradient this GEMM writes is then
  // the sum of ceil(M / 32) partial rows instead of a pass over out.
  float* col_part = nullptr;
  // Adam update of the weight fused into a weight-gradient epilogue
  // (tcgen05 kernels, fp32 output, no split over K), or upd_p null: the
  // parameters, moments and bf16 copy have out's layout; upd_scal points to
  // {lr / (1 - b1^t), 1 / sqrt(1 - b2^t)} in device memory.
  float* upd_p = nullptr;
  float* upd_m = nullptr;
  float* upd_v = nullptr;
  void* upd_shadow = nullptr;      // bf16
  const float* upd_scal = nullptr;
  float upd_b1 = 0.f, upd_b2 = 0.f, upd_eps = 0.f;
};

cudaError_t gemm_simt(const GemmArgs& g, cudaStream_t s);
// Floats of split_ws gemm_simt uses for g (0: g is not split).
size_t gemm_simt_split_floats(const GemmArgs& g);
// Whether gemm_simt runs g on its narrow-side bf16 kernels (N <= 32 forward
// or weight gradient, K <= 32 input gradient).
bool gemm_simt_skinny(const GemmArgs& g);
// tcgen05/TMA version for bf16 operands whose rows are 16-byte aligned.
// *err is set to 1 if a bounded pipeline wait expires.
bool gemm_tc_eligible(const GemmArgs& g);
cudaError_t gemm_tc(const GemmArgs& g, int* err, cudaStream_t s);
// Split count of the single-SM tensor-core GEMM for g and, in *steps (may be
// NULL), its estimated duration in K-block steps of one SM.
int gemm_tc_splits(const GemmArgs& g, double* steps);
// Same on a pair of SMs (tcgen05 cta_group::2, 256x256 tiles), used where it
// is estimated faster than the single-SM kernel; requires gemm_tc_eligible(g)
// as well.
bool gemm_pair_eligible(const GemmArgs& g);
cudaError_t gemm_pair(const GemmArgs& g, int* err, cudaStream_t s);
// Split count over K the SM-pair kernel picks for g.
int gemm_pair_split_count(const GemmArgs& g);

// ---- loss ------------------------------------------------------------------
// Softmax cross-entropy from logits whose per-row softmax partials the head
// GEMM already wrote (GemmArgs::lse_part, nparts = ceil(C / 128) per row):
// combines them into log-sum-exp, then one pass writes dlogits and the row
// losses exactly as ce_loss does.  bf16 logits, C % 8 == 0.
cudaError_t ce_loss_from_partials(const void* logits, int B, int C, long long ld,
                                  const float2* parts, int nparts, int label_kind,
                                  const void* labels, void* dlogits, float* row_loss,
                                  float* loss, cudaStream_t s);
// Softmax cross-entropy over rows of logits[B, C] (stride ld).  label_kind 0:
// dense fp32 labels [B, C]; 1: int32 class ids [B].  Writes dlogits (same
// dtype and layout as logits) = (p * sum(y) - y) / B, and row_loss[B] =
// -sum_c y_c log p_c.  Then loss = sum(row_loss) / B.
cudaError_t ce_loss(DType t, const void* logits, int B, int C, long long ld, int label_kind,
                    const void* labels, void* dlogits, float* row_loss, float* loss,
                    cudaStream_t s);
// Mean squared error over n elements: dout = 2 (o - t) / n; loss = mean((o - t)^2).
cudaError_t mse_loss(DType t, const void* o, const void* target, size_t n, void* dout,
                     float* partials, int n_partials, float* loss, cudaStream_t s);

// ---- reductions / norms ----------------------------------------------------
// out[n] = sum over rows of src[r, n]  (fp32 result), deterministic two passes.
cudaError_t colsum(DType t, const void* src, int rows, int cols, long long ld, float* partials,
                   size_t partial_floats, float* out, cudaStream_t s);
// out[n] = sum over r < chunks of partials[r * cols + n] (fixed order).
cudaError_t colsum_partials(const float* partials, int chunks, int cols, float* out,
                            cudaStream_t s);
// Target block count of colsum's first pass (about two per SM); a partials
// buffer of kColsumBlocks * 2048 floats lets it reach that for any width.
constexpr int kColsumBlocks = 2 * 152;
cudaError_t rmsnorm_fwd(DType t, const void* x, const float* gamma, void* y, float* rstd, int rows,
                        int d, float eps, cudaStream_t s);
// dx = r (g - x r^2 mean(g x)) + dadd, g = dy * gamma;  dgamma partial sums of dy * x * r.
cudaError_t rmsnorm_bwd(DType t, const void* dy, const void* x, const float* rstd,
                        const float* gamma, const void* dadd, void* dx, float* dgamma_partials,
                        int row_chunks, float* dgamma, int rows, int d, cudaStream_t s);

// ---- attention (bf16 storage, fp32 softmax) ----------------------------------
// qkv [nb*S, 3*H*Dh], o [nb*S, H*Dh], lse [nb, H, S].
cudaError_t attn_fwd(const void* qkv, void* o, float* lse, int nb, int S, int H, int Dh,
                     cudaStream_t s);
cudaError_t attn_bwd(const void* qkv, const void* o, const void* dout, const float* lse,
                     float* dsum, void* dqkv, int nb, int S, int H, int Dh, cudaStream_t s);
int attn_bwd_launches();
// D_i = sum_c dO_ic O_ic into dsum [nb, H, S].
cudaError_t attn_bwd_pre(const void* o, const void* dout, float* dsum, int nb, int S, int H,
                         cudaStream_t s);
// tcgen05 versions (head_dim 64, S a multiple of 128, 16-byte aligned rows).
// *err is set to 1 if a bounded pipeline wait expires.
bool attn_tc_eligible(int S, int H, int Dh, const void* qkv);
cudaError_t attn_fwd_tc_launch(const void* qkv, void* o, float* lse, int nb, int S, int H,
                               int* err, cudaStream_t s);
cudaError_t attn_bwd_tc_launch(const void* qkv, const void* dout, const float* lse,
                               const float* dsum, void* dqkv, int nb, int S, int H, int* err,
                               cudaStream_t s);

// ---- optimizer (multi-tensor over chunk tables) -----------------------------
struct Chunk {  // a run of one tensor's elements in the flat buffers
  long long start;
  int len;
  int shadow;   // 1: write the bf16 copy of the updated value
};
cudaError_t adam_update(const Chunk* chunks, int n_chunks, float* p, const float* g, float* m,
                        float* v, void* shadow, float lr_over_bc1, float inv_sqrt_bc2,
                        float beta1, float beta2, float eps, cudaStream_t s);
// The optimizer update kernels' (and write_step_scalars') argument layout, for replaying a captured
// step with new step scalars: argument count and sizes, and the indices of
// lr / (1 - b1^t), 1 / sqrt(1 - b2^t) (Adam, LaProp) or lr (SGD, momentum).
struct OptKernelInfo {
  int nargs;
  int size[12];
  int i_lr_bc1, i_inv_sqrt_bc2, i_lr;
};
bool optimizer_kernel_info(const void* func, OptKernelInfo* info);
cudaError_t laprop_update(const Chunk* chunks, int n_chunks, float* p, const float* g, float* m,
                          float* v, void* shadow, float lr_over_bc1, float inv_sqrt_bc2,
                          float beta1, float beta2, float eps, cudaStream_t s);
cudaError_t momentum_update(const Chunk* chunks, int n_chunks, float* p, const float* g, float* b,
                            void* shadow, float lr, float mu, cudaStream_t s);
cudaError_t sgd_update(const Chunk* chunks, int n_chunks, float* p, const float* g, void* shadow,
                       float lr, cudaStream_t s);
// dst[0] = lr_bc1, dst[1] = inv_sqrt_bc2 (the step scalars a fused update
// reads; a one-thread kernel, so that a replayed step graph can patch them).
cudaError_t write_step_scalars(float* dst, float lr_bc1, float inv_sqrt_bc2, cudaStream_t s);
cudaError_t cast_shadow(const Chunk* chunks, int n_chunks, const float* p, void* shadow,
                        cudaStream_t s);

// ---- misc --------------------------------------------------------------------
cudaError_t cast_to_f32(DType t, const void* src, float* dst, size_t n, cudaStream_t s);
cudaError_t find_nonfinite(const float* data, size_t n, unsigned long long* first_bad,
                           cudaStream_t s);

// Sets the process-wide message returned by mg_last_error(NULL).
void set_global_error(const char* msg);

}  // namespace mg
