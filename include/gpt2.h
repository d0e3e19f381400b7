/*
 * gpt2.h -- C ABI of the B300 (sm_103a) GPT-2 training-step library.
 *
 * The library runs the training step that the llm.c pages describe, on one GPU:
 *   ujoy.net llm.c article, section "用C语言实现LLM" (implementing an LLM in C):
 *     memory is allocated once, as one 1-D block, and every tensor points into it;
 *     nothing is created or freed while training; each layer (encoder, layernorm,
 *     matmul, self-attention, GELU, residual, softmax, cross-entropy) has a forward
 *     and a backward pass written by hand, and the layers are chained together.
 *   same article, section "训练过程" (training run): forward, backward and an Adam
 *     update chained into one loop ("Adam lr 1e-4").
 *   yinghuohong.cn llm.c article, section "脚动完成每一个层前向/反向流传": all memory
 *     allocated at the start, constant footprint, weights and activations both point
 *     into flat arrays.
 *
 * Conventions for every entry point
 *   - Device pointers are plain CUDA device addresses on the current device; host
 *     pointers are plain host addresses.  No PyTorch types cross this boundary.
 *   - The caller owns every byte of device memory.  gpt2_build carves the one
 *     workspace the caller passes; the library allocates no device memory at all
 *     (it keeps a small host struct and, in bf16 mode, TMA descriptors).
 *   - All work is enqueued on the handle's CUDA stream (set at build, changeable with
 *     gpt2_set_stream) and is asynchronous unless stated otherwise.
 *   - Every call returns a status code (GPT2_OK = 0).  Device-side faults the kernels
 *     detect themselves (an out-of-range token id, a bounded wait that ran out, a
 *     non-finite loss) are latched in a device error word and reported by the next
 *     synchronising call (gpt2_forward with loss_out, gpt2_check).
 *   - Matrices are row-major.  A linear layer's weight is stored (out, in) and computes
 *     y = x W^T + b.  Activations are (B, T, C) row-major, token-major.
 *
 * Model (readings of the pages, pinned by the printed num_parameters 124439808 and
 * num_activations 73323776): GPT-2 pre-LN blocks, learned position table, biases on
 * every linear layer, LM head tied to the token table, layernorm eps 1e-5 (biased
 * variance), tanh-form GELU, causal attention scaled by 1/sqrt(C/NH), mean
 * cross-entropy over the V real vocabulary columns (padded columns are excluded and
 * get zero gradient), AdamW with bias correction and decoupled weight decay on every
 * parameter.
 */
#ifndef GPT2_B300_H
#define GPT2_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int max_seq_len;        /* rows of the position table (maxT) */
    int vocab_size;         /* V: real vocabulary */
    int padded_vocab_size;  /* Vp >= V: rows of the token table; rows >= V stay zero */
    int num_layers;         /* L */
    int num_heads;          /* NH; channels % num_heads == 0 */
    int channels;           /* C; a multiple of 64 */
} GPT2Config;

/* Arithmetic of the step.
 * GPT2_FP32: fp32 activations and weights; every product and sum in fp32 (SIMT FMA).
 * GPT2_BF16: bf16 weights (a shadow of the fp32 master copy), bf16 activations and
 *            activation grads; matmuls and attention on the tcgen05 tensor cores with
 *            fp32 accumulation; fp32 master weights, parameter grads, AdamW state,
 *            layernorm statistics, softmax/loss arithmetic. */
/* GPT2_FP8:  as GPT2_BF16, except that the two products whose input is a layernorm
 *            output (the qkv and MLP-fc forward products) take e4m3 operands on the
 *            tensor cores (tcgen05 kind::f8f6f4, fp32 accumulation): the layernorm writes
 *            its output also as e4m3 codes with one power-of-two scale per row (that row's
 *            largest magnitude maps into the top binade, <= 448), the qkv and fc weights
 *            have e4m3 shadows with one power-of-two scale per (tensor, layer), refreshed
 *            from the fp32 master weights after every update.  The backward pass, the
 *            other products and the LM head stay bf16 (the quantization passes gradients
 *            straight through).  yinghuohong.cn llm.c article, section
 *            "脚动完成每一个层前向/反向流传": precision taken from fp32 down to fp16 or lower. */
enum { GPT2_FP32 = 0, GPT2_BF16 = 1, GPT2_FP8 = 2 };

enum {
    GPT2_OK = 0,
    GPT2_EINVAL = 1,       /* bad argument: null pointer, size out of range, misalignment */
    GPT2_ESTATE = 2,       /* call out of order, e.g. backward without a forward with targets */
    GPT2_ECUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    GPT2_ETOKEN = 4,       /* a token or target id outside [0, V) (its rows were zeroed) */
    GPT2_ENONFINITE = 5,   /* the mean loss was NaN or Inf */
    GPT2_ETIMEOUT = 6,     /* a bounded device-side wait ran out; the kernel gave up */
    GPT2_ENOMEM = 7,       /* the workspace passed to gpt2_build is too small */
    GPT2_EUNSUPPORTED = 8, /* shape or precision this build does not implement */
    GPT2_EIO = 9           /* a parameter file could not be read or written, or its header
                              does not describe this model */
};

/* Names of the 16 parameter tensors, in the order of the flat buffer:
 *  0 wte (Vp,C)   1 wpe (maxT,C)
 *  2 ln1w (L,C)   3 ln1b (L,C)   4 qkvw (L,3C,C)    5 qkvb (L,3C)
 *  6 attprojw (L,C,C)   7 attprojb (L,C)   8 ln2w (L,C)   9 ln2b (L,C)
 * 10 fcw (L,4C,C)  11 fcb (L,4C)  12 fcprojw (L,C,4C)  13 fcprojb (L,C)
 * 14 lnfw (C)  15 lnfb (C)
 * Each tensor starts on a 64-element boundary of the flat buffer; the gap elements are
 * zero and stay zero. */
#define GPT2_NUM_PARAM_TENSORS 16

typedef struct GPT2 GPT2;

/* Bytes of device workspace gpt2_build needs for this model, batch limits and
 * precision.  Returns GPT2_EINVAL for an unsupported shape. */
int gpt2_workspace_bytes(const GPT2Config* cfg, int max_B, int max_T, int precision,
                         size_t* bytes);

/* Carve `workspace` (device, >= gpt2_workspace_bytes, 1024-byte aligned) into the flat
 * parameter, gradient, AdamW-moment and activation buffers and return a handle in *out.
 * The parameters are zeroed; upload the initial weights into gpt2_params() and call
 * gpt2_sync_params().  `stream` is a cudaStream_t (NULL = legacy default stream).
 * Synchronises the stream once.  The workspace must outlive the handle. */
int gpt2_build(const GPT2Config* cfg, int max_B, int max_T, int precision,
               void* workspace, size_t workspace_bytes, void* stream, GPT2** out);

/* Release the host-side handle (the workspace stays the caller's). */
void gpt2_free(GPT2* model);
/* The same, under the name of the boundary sketch (allocate once, then forward,
 * zero_grad, backward, update, destroy). */
void gpt2_destroy(GPT2* model);

int gpt2_set_stream(GPT2* model, void* stream);

/* Parameter counts: n_real counts the tensors with V token rows (the pages' count);
 * n_flat is the length of the flat buffers (padded vocabulary and alignment gaps). */
int gpt2_num_parameters(const GPT2* model, size_t* n_real, size_t* n_flat);

/* Real parameter count (the pages' num_parameters) into *n; GPT2_EINVAL for NULL. */
int gpt2_num_params(const GPT2* model, size_t* n);

/* Element offset of tensor `index` (0..15, order above) in the flat buffers, and its
 * element count. */
int gpt2_param_tensor(const GPT2* model, int index, size_t* offset, size_t* numel);

/* Device pointers to the flat fp32 buffers (n_flat elements each). */
float* gpt2_params(GPT2* model);     /* master weights; write the initial values here */
float* gpt2_grads(GPT2* model);      /* parameter gradients */
float* gpt2_adam_m(GPT2* model);
float* gpt2_adam_v(GPT2* model);
/* The master-weight and gradient pointers with a status (GPT2_EINVAL for NULL arguments). */
int gpt2_param_ptr(GPT2* model, float** master);
int gpt2_grad_ptr(GPT2* model, float** grads);

/* After writing gpt2_params(): refresh the bf16 shadow weights (bf16 mode; a no-op in
 * fp32 mode) and clear the AdamW moments. */
int gpt2_sync_params(GPT2* model);

/* Forward pass of every layer (ujoy.net llm.c article, section "用C语言实现LLM": encoder,
 * then per block layernorm, matmul, self-attention, matmul + residual, layernorm, matmul,
 * GELU, matmul + residual; final layernorm, tied LM head, softmax, cross-entropy) over
 * tokens (device int32, (B,T) row-major, ids in
 * [0,V)).  With targets (device int32, (B,T)) it also computes the per-position
 * cross-entropy, the mean loss, and -- fused with the softmax -- the gradient of the
 * mean loss with respect to the logits, which backward consumes.  With
 * targets == NULL only the logits are produced (gpt2_logits) and backward is refused.
 * B <= max_B, 1 <= T <= min(max_T, max_seq_len).  The token ids are copied into the
 * workspace, so the caller's buffers may be reused once the call returns.
 * loss_out (host, nullable): if given, the call synchronises the stream and stores
 * the mean loss (or -1 without targets); it then also returns any latched device
 * error.  Without it, no synchronisation happens (the loss stays in gpt2_loss()). */
int gpt2_forward(GPT2* model, const int32_t* tokens, const int32_t* targets, int B, int T,
                 float* loss_out);

/* Set every parameter gradient to zero (same article, section "训练过程": the training
 * loop zeroes the gradients before each backward pass). */
int gpt2_zero_grad(GPT2* model);

/* Backward pass of every layer in reverse order (same article, section "用C语言实现LLM":
 * each layer's hand-written backward, chained from the loss back to the encoder); adds d(mean loss)/d(param) into the
 * gradient buffer.  Needs a preceding gpt2_forward with targets (else GPT2_ESTATE). */
int gpt2_backward(GPT2* model);

/* One AdamW step over the whole flat buffer (same article, section "训练过程": the Adam
 * update after each backward pass, here with decoupled weight decay):
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;  mhat = m/(1-b1^t);  vhat = v/(1-b2^t)
 *   p -= lr (mhat / (sqrt(vhat) + eps) + weight_decay p)
 * then (bf16 mode) refresh the bf16 shadow.  t >= 1 is the 1-based step count. */
int gpt2_update(GPT2* model, float lr, float beta1, float beta2, float eps,
                float weight_decay, int t);

/* The Muon optimizer (pimou.com article, sections "优化器的优势" and "相关技术的追溯":
 * Muon orthogonalizes the update with Newton-Schulz iterations, after Bernstein &
 * Newhouse 2024), for the bf16 and fp8 modes (GPT2_EUNSUPPORTED in fp32).  On each
 * block matrix (qkvw, attprojw, fcw, fcprojw of every layer, one matrix per layer):
 *   mom = momentum mom + g  (mom kept in the AdamW first-moment buffer of that matrix)
 *   X = mom / ||mom||_F, then ns_iters times X <- 1.5 X - 0.5 X X^T X (in bf16 on the tensor
 *   cores, fp32 accumulation; on the smaller Gram side)
 *   p -= lr_muon (X + weight_decay p)
 * and AdamW (lr, beta1, beta2, eps, weight_decay, t as gpt2_update) on every other
 * parameter.  Then the bf16 (and fp8) weight shadows are refreshed. */
int gpt2_update_muon(GPT2* model, float lr_muon, float momentum, int ns_iters, float lr, float beta1,
                     float beta2, float eps, float weight_decay, int t);

/* The Newton-Schulz iteration of gpt2_update_muon alone: out (r x c, bf16, device) =
 * iters steps from G (r x c, fp32, device) / ||G||_F.  r, c multiples of 8; out, G and
 * scratch 256-byte aligned; scratch >= gpt2_newton_schulz_scratch_bytes(r, c). */
size_t gpt2_newton_schulz_scratch_bytes(int r, int c);
int gpt2_newton_schulz(void* out, const float* G, int r, int c, int iters, void* scratch,
                       size_t scratch_bytes, void* stream);

/* One whole training step from HOST token buffers: copies tokens/targets (pinned host
 * memory recommended) to the device, runs forward, zero_grad, backward and update (as
 * one CUDA graph once the shape has been seen, see gpt2_step), and copies the mean loss
 * back into *loss_out (host).  Synchronises the stream. */
int gpt2_step_host(GPT2* model, const int32_t* tokens_host, const int32_t* targets_host,
                   int B, int T, float lr, float beta1, float beta2, float eps,
                   float weight_decay, int t, float* loss_out);

/* The same step from DEVICE token buffers (B*T int32 each, read before the call
 * returns control of the stream).  loss_out (host) may be NULL: the call then does not
 * synchronise.  With graphs enabled (the default) and the tracer off, the first step of
 * a (B, T) shape runs kernel by kernel, the second is captured into one CUDA graph, and
 * later steps of that shape replay it with the step's AdamW scalars (same kernels, same
 * results bit for bit).  Other steps of the model (gpt2_forward, ...) are unaffected. */
int gpt2_step(GPT2* model, const int32_t* tokens, const int32_t* targets, int B, int T,
              float lr, float beta1, float beta2, float eps, float weight_decay, int t,
              float* loss_out);

/* The step of gpt2_step with the update of gpt2_update_muon (same arguments; bf16 and fp8
 * models, GPT2_EUNSUPPORTED in fp32): forward, backward and the Muon + AdamW update, as
 * one CUDA graph once the shape has been seen.  A graph serves one (B, T) and one set of
 * Muon constants (ns_iters, lr_muon, momentum, weight_decay): a step with other values
 * runs kernel by kernel and the next one is captured anew; lr, beta1, beta2, eps and t
 * are set on the graph's AdamW nodes before each launch. */
int gpt2_step_muon(GPT2* model, const int32_t* tokens, const int32_t* targets, int B, int T,
                   float lr_muon, float momentum, int ns_iters, float lr, float beta1, float beta2,
                   float eps, float weight_decay, int t, float* loss_out);

/* Enable (1, the default) or disable (0) the step graph of gpt2_step / gpt2_step_host /
 * gpt2_step_muon; disabling frees a captured graph.  GPT2_EINVAL for a NULL model. */
int gpt2_set_graphs(GPT2* model, int enable);

/* Next-token sampling (the llm.c article's training run: after training, the program
 * generates samples from the model).  Needs a preceding gpt2_forward WITHOUT targets
 * (the logits are kept; GPT2_ESTATE otherwise).  For each sequence b of that forward,
 * draws a token from p_j = softmax(z[b, pos, j] / temperature) over the V real columns
 * by inverse CDF: u_b = (top 53 bits of output b+1 of SplitMix64 started at `seed`) /
 * 2^53, and the token is the first j whose running sum of exp((z_j - max) / temperature)
 * exceeds u_b times the total (sums in a fixed order, so a seed always gives the same
 * tokens).  out_tokens: B int32, device, caller-owned; written on the model's stream
 * (no synchronisation).  GPT2_EINVAL for pos outside [0, T) of that forward, a
 * temperature that is not > 0, or a NULL pointer. */
int gpt2_sample(GPT2* model, int pos, float temperature, unsigned long long seed, int32_t* out_tokens);

/* Parameter files.  The llm.c article ("用C语言实现LLM" / the training run) saves the
 * model's weights to a checkpoint that the C program loads into its one parameter
 * buffer before training.  Layout (little-endian): 256 int32 header words -- [0] magic
 * 20240326, [1] version 3, [2] max_seq_len, [3] vocab_size, [4] num_layers, [5] num_heads,
 * [6] channels, [7] padded_vocab_size, the rest 0 -- then every parameter tensor in the
 * order of gpt2_param_tensor (wte with all padded_vocab_size rows, wpe, ln1w, ..., lnfb),
 * fp32, back to back.  gpt2_save_params synchronises the model's stream and writes the
 * fp32 master weights.  gpt2_load_params requires the header to match the model's
 * configuration exactly (else GPT2_EIO, parameters untouched), copies the tensors into
 * the master weights, refreshes the bf16 shadow and zeroes the AdamW moments (a fresh
 * optimiser state for the loaded weights), and synchronises.  GPT2_EIO also for a file
 * that cannot be opened or is shorter than the header says. */
int gpt2_save_params(GPT2* model, const char* path);
int gpt2_load_params(GPT2* model, const char* path);

/* Device pointers into the last forward's outputs: the mean loss (1 float), the
 * per-position losses (B*T floats) and the logits (B*T rows of Vp entries, fp32 or bf16
 * by precision; overwritten by d loss/d logits when targets were given). */
float* gpt2_loss(GPT2* model);
float* gpt2_losses(GPT2* model);
void* gpt2_logits(GPT2* model);

/* Synchronise the stream and return (then clear) the latched device error, if any. */
int gpt2_check(GPT2* model);

const char* gpt2_strerror(int status);

/* The cudaError_t of the most recent failed CUDA call on this thread (0 if none). */
int gpt2_last_cuda_error(void);

/* ---------------------------------------------------------------------------------
 * Single-layer entry points (same kernels as the model; used for per-layer tests and
 * by callers that chain layers themselves).  All pointers are device pointers;
 * `stream` is a cudaStream_t.  The calls are asynchronous.  A bounded device-side wait
 * that runs out in one of their kernels (the kernel then gives up and returns) is
 * latched in a per-device error word of the library, which gpt2_layer_check reads.
 * ------------------------------------------------------------------------------- */

/* Synchronise `stream` and return (then clear) the error latched by the single-layer
 * entry points on the current device: GPT2_ETIMEOUT if a bounded wait ran out since the
 * last check (that call's outputs are then incomplete), else GPT2_OK. */
int gpt2_layer_check(void* stream);

/* Layernorm forward over N rows of C (C % 8 == 0, C <= 2048), fp32; N == 0 is a no-op:
 *   mean = sum(x)/C; rstd = 1/sqrt(sum((x-mean)^2)/C + 1e-5); out = (x-mean) rstd w + b.
 * out (N,C), mean (N), rstd (N) are written. */
int gpt2_layernorm_forward(float* out, float* mean, float* rstd, const float* inp,
                           const float* weight, const float* bias, int N, int C,
                           void* stream);

/* Scratch bytes gpt2_layernorm_backward needs for N rows of C. */
size_t gpt2_layernorm_backward_scratch_bytes(int N, int C);

/* The layernorm forward of the fp8 mode (fp32 tensors here): out, mean, rstd as
 * gpt2_layernorm_forward, and out also as e4m3 codes (N, C bytes, 8-byte aligned) with
 * row_deq[r] = 2^-k, k the largest integer with max_c |out[r, c]| * 2^k <= 448 (0 for an
 * all-zero row, clamped to [-126, 126]); code = e4m3(out * 2^k), round to nearest even,
 * saturating.  The codes are taken of the fp32 values. */
int gpt2_layernorm_forward_fp8(float* out, uint8_t* codes, float* row_deq, float* mean, float* rstd,
                               const float* inp, const float* weight, const float* bias, int N, int C,
                               void* stream);

/* Per-tensor e4m3 quantization of x (n fp32 values, n % 4 == 0, 16-byte aligned):
 * codes (n bytes, 16-byte aligned) = e4m3(x * 2^k) and deq[0] = 2^-k with k as above for
 * the tensor's largest |x| -- the fp8 mode's weight shadows.  amax_scratch: one device
 * word, overwritten. */
int gpt2_quantize_e4m3(uint8_t* codes, float* deq, unsigned* amax_scratch, const float* x, size_t n,
                       void* stream);

/* The fp8 mode's forward product: out (M,N) bf16 = epilogue((inp * inp_deq per row)
 * (weight * weight_deq[0])^T + bias), inp (M,K) and weight (N,K) e4m3 codes, inp_deq (M)
 * and weight_deq (1) fp32 device arrays, bias bf16 (nullable), epilogue and aux as
 * gpt2_matmul_forward_fused.  K a multiple of 16, N of 8, 16-byte aligned operands. */
int gpt2_matmul_forward_fp8(void* out, void* aux, const uint8_t* inp, const float* inp_deq,
                            const uint8_t* weight, const float* weight_deq, const void* bias, int M, int N,
                            int K, int epilogue, void* stream);

/* fp8 mode: the model's e4m3 weight shadows.  which 0: qkvw (L, 3C, C bytes), 1: fcw
 * (L, 4C, C); *deq points at L per-layer unscaling factors.  GPT2_ESTATE for another
 * precision. */
int gpt2_fp8_weights(GPT2* model, int which, uint8_t** codes, float** deq);

/* Layernorm backward, fp32.  dinp += dx (accumulates); dweight += sum_rows dout*xhat;
 * dbias += sum_rows dout.  The column sums are deterministic (fixed-order two-stage
 * reduction through `scratch`, device, >= gpt2_layernorm_backward_scratch_bytes). */
int gpt2_layernorm_backward(float* dinp, float* dweight, float* dbias, const float* dout,
                            const float* inp, const float* weight, const float* mean,
                            const float* rstd, int N, int C, void* scratch,
                            size_t scratch_bytes, void* stream);

/* Layernorm backward that allocates nothing and takes no scratch argument.  The pages
 * have no counterpart; this exists for callers that cannot obtain device memory at
 * all, such as a host program that passes this library only its input and output
 * buffers, or one that commits all device memory at start-up and must not call
 * cudaMalloc mid-step.  Same arguments and results as gpt2_layernorm_backward, whose
 * kernels it runs, with the scratch taken from an array of GPT2_NOALLOC_SCRATCH_BYTES
 * compiled into the library (held on every GPU that loads it, until the process
 * exits).  Returns GPT2_EINVAL when gpt2_layernorm_backward_scratch_bytes(N, C) exceeds
 * that size: any N for C <= 1768, N <= 4096 rows for C = 2048 (the partial sums take
 * min(ceil(N/16), 296) blocks x 2C floats).  Every call looks up the array's address on
 * the current device, so `stream` must belong to the current device.  With lazy module
 * loading the first call on a device also loads the module that holds the array: make it
 * at start-up, before any stream capture.  All calls share the one array, so calls that
 * overlap on the GPU race: serialise them.  Nothing is carried over between calls (every
 * partial sum read is rewritten first).  Timeouts are reported by gpt2_layer_check.
 * Calls no cudaMalloc, cudaFree or allocating routine. */
#define GPT2_NOALLOC_SCRATCH_BYTES (4u << 20)
int gpt2_layernorm_backward_noalloc(float* dinp, float* dweight, float* dbias, const float* dout,
                                    const float* inp, const float* weight, const float* mean,
                                    const float* rstd, int N, int C, void* stream);

/* Causal self-attention forward (ujoy.net llm.c article, section "用C语言实现LLM": the
 * self-attention layer) over qkv (B,T,3C) (q, k, v thirds; head h uses columns
 * [h*hs, (h+1)*hs) of each, hs = C/NH): out (B,T,C) = softmax(q k^T / sqrt(hs) over keys
 * j <= t) v, heads concatenated.  precision GPT2_BF16: bf16 tensors, lse (B,NH,T) fp32
 * receives each score row's log-sum-exp (natural log) for the backward; GPT2_FP32: fp32
 * tensors, and `lse` must hold the probabilities instead: (B,NH,T,T) fp32.
 * bf16: head size C/NH = 64 (the tensor-core kernels; other sizes GPT2_EUNSUPPORTED);
 * fp32: head size <= 128, a multiple of 8. */
int gpt2_attention_forward(void* out, float* lse, const void* qkv, int B, int T, int C, int NH,
                           int precision, void* stream);

/* Backward: dqkv (B,T,3C) [overwritten] from dout (B,T,C) and the forward's qkv, out
 * and lse (fp32 path: probabilities).  dbias (device fp32 (3C), nullable) += the column
 * sums of dqkv over the B*T rows: the qkv bias gradient (bf16: summed from the stored
 * bf16 dqkv in the kernels' output stage, 32 rows at a time, then in a fixed order).
 * scratch (device, 16-byte aligned, gpt2_attention_backward_scratch_bytes): bf16 path the
 * fp32 row sums D = rowsum(dout * out) and, for T not a multiple of 4, a copy of the
 * LSE, each (B,NH,T rounded up to a multiple of 4); fp32 path (B,NH,T,T) fp32; then the
 * bias gradient's partial sums. */
size_t gpt2_attention_backward_scratch_bytes(int B, int T, int C, int NH, int precision);
int gpt2_attention_backward(void* dqkv, float* dbias, const void* dout, const void* qkv, const void* out,
                            const float* lse, int B, int T, int C, int NH, int precision,
                            void* scratch, size_t scratch_bytes, void* stream);

/* Matmul forward: out (M,N) = inp (M,K) * weight(N,K)^T + bias (N, nullable).
 * precision GPT2_FP32: all float*; GPT2_BF16: out, inp, weight, bias are bf16 (bias
 * nullable), fp32 accumulation, on the tensor cores only: N and K multiples of 8 and
 * 16-byte aligned pointers, else GPT2_EUNSUPPORTED. */
int gpt2_matmul_forward(void* out, const void* inp, const void* weight, const void* bias,
                        int M, int N, int K, int precision, void* stream);

/* The matmul forward with the epilogue the model fuses into it (ujoy.net llm.c article,
 * section "用C语言实现LLM": the matmul, GELU and residual layers), with h = inp weight^T
 * + bias (bias nullable):
 *   GPT2_EPI_BIAS      out = h                                  (aux unused)
 *   GPT2_EPI_GELU      aux = h (written); out = gelu(aux as stored), tanh form
 *   GPT2_EPI_RESIDUAL  out = aux + h (aux (M,N) read: the residual stream)
 * Same types and limits as gpt2_matmul_forward; aux has out's type and shape. */
enum { GPT2_EPI_BIAS = 0, GPT2_EPI_GELU = 1, GPT2_EPI_RESIDUAL = 2 };
int gpt2_matmul_forward_fused(void* out, void* aux, const void* inp, const void* weight,
                              const void* bias, int M, int N, int K, int epilogue, int precision,
                              void* stream);

/* Input gradient of a matmul whose input was a GELU output, with the GELU backward fused:
 * dinp (M,K) = (dout (M,N) weight (N,K)) * gelu'(pre), pre (M,K) the GELU's stored input
 * (the model's MLP projection backward).  dbias (device fp32 (K), nullable) += the column
 * sums of dinp: the bias gradient of the layer that produced `pre` (bf16: summed from the
 * stored bf16 dinp in the product's output stage, 32 rows at a time, then in a fixed
 * order); it needs `scratch` (device, 16-byte aligned,
 * gpt2_matmul_backward_input_gelu_scratch_bytes), which is unused otherwise (nullable).
 * Types and limits as gpt2_matmul_forward. */
size_t gpt2_matmul_backward_input_gelu_scratch_bytes(int M, int K);
int gpt2_matmul_backward_input_gelu(void* dinp, float* dbias, const void* dout, const void* weight,
                                    const void* pre, int M, int N, int K, int precision, void* scratch,
                                    size_t scratch_bytes, void* stream);

/* Matmul backward: dinp (M,K) = dout (M,N) * weight (N,K)  [overwrites];
 * dweight (N,K, fp32) += dout^T * inp;  dbias (N, fp32, nullable) += column sums of
 * dout.  dout/inp/weight/dinp are float or bf16 by precision.  `scratch` (device,
 * >= gpt2_matmul_backward_scratch_bytes) holds the deterministic column-sum partials and,
 * in bf16, the partial tiles of a weight gradient whose contraction is split (added in a
 * fixed order). */
size_t gpt2_matmul_backward_scratch_bytes(int M, int N);
int gpt2_matmul_backward(void* dinp, float* dweight, float* dbias, const void* dout,
                         const void* inp, const void* weight, int M, int N, int K,
                         int precision, void* scratch, size_t scratch_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * Observability: kernel-launch counter and per-kernel-class tracing.
 * Tracing brackets every layer launch with two CUDA events on the stream the kernels go
 * to and attributes the elapsed device time and the launch's algorithmic work (flops of
 * a contraction, bytes of a memory-bound layer) to one of gpt2_profile_num_classes()
 * classes (names from gpt2_profile_class_name).  The event pool is created by the first
 * gpt2_profile_enable(1); no device memory is used.
 * ------------------------------------------------------------------------------- */

/* Kernels this library has launched in this process so far. */
long long gpt2_kernel_launches(void);

/* Trace the classes whose bit is set in class_mask (bit i = class i); 0 switches off. */
int gpt2_profile_enable(unsigned class_mask);
/* Wait for the recorded events and fold their times into the per-class totals. */
int gpt2_profile_collect(void);
/* Collect, then zero the totals. */
int gpt2_profile_reset(void);
/* Totals of class `cls` since the last reset: device ms, bracketed launches, flops, bytes. */
int gpt2_profile_read(int cls, double* ms, long long* scopes, double* flops, double* bytes);
/* Brackets skipped because the event pool was exhausted (collect more often). */
long long gpt2_profile_dropped(void);
int gpt2_profile_num_classes(void);
const char* gpt2_profile_class_name(int cls);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_B300_H */
