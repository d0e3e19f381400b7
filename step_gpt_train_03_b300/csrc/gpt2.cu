// GPT-2 training step on one B300: the C ABI of include/gpt2.h.
//
// Structure (ujoy.net llm.c article, section "用C语言实现LLM"; yinghuohong.cn llm.c
// article, section "脚动完成每一个层前向/反向流传"): one block of memory, passed in by
// the caller, carved once into the flat parameter / gradient / AdamW buffers and the
// activation buffers; nothing is allocated afterwards.  Each layer has a hand-written
// forward and backward kernel; gpt2_forward / gpt2_backward chain them, gpt2_update
// runs AdamW over the flat buffer (same article, section "训练过程": forward, backward
// and update chained into one loop).
#include <cuda_runtime.h>
#include <vector>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <algorithm>

#include "../../include/gpt2.h"
#include "common.cuh"
#include "kernels_mem.cuh"
#include "gemm_simt.cuh"
#include "attention_simt.cuh"
#include "gemm_tc.h"
#include "attention_tc.h"
#include "runtime.h"

#define CK(x)                                                   \
    do {                                                        \
        cudaError_t e_ = (x);                                   \
        if (e_ != cudaSuccess) { g_last_cuda_error = e_; return GPT2_ECUDA; } \
    } while (0)

static thread_local cudaError_t g_last_cuda_error = cudaSuccess;

#define RC(x)                          \
    do {                               \
        int rc_ = (x);                 \
        if (rc_ != GPT2_OK) return rc_; \
    } while (0)

// ------------------------------------------------------------------ handle
enum { P_WTE = 0, P_WPE, P_LN1W, P_LN1B, P_QKVW, P_QKVB, P_ATTPROJW, P_ATTPROJB, P_LN2W, P_LN2B,
       P_FCW, P_FCB, P_FCPROJW, P_FCPROJB, P_LNFW, P_LNFB };

struct GPT2 {
    GPT2Config cfg;
    int maxB, maxT, prec;
    int overwrite;                     // the next backward's first write to each gradient stores (no clear before)
    int L, C, NH, V, Vp;
    size_t poff[GPT2_NUM_PARAM_TENSORS], pnum[GPT2_NUM_PARAM_TENSORS];
    size_t n_flat, n_real;
    char* ws;
    size_t ws_bytes;
    cudaStream_t stream;
    // flat parameter buffers
    float *params, *grads, *m, *v;
    bf16* wbf;                         // bf16 shadow of params (bf16 mode)
    // activations; element type is float (fp32 mode) or bf16 (bf16 mode)
    void *encoded, *ln1, *qkv, *atty, *res2, *ln2, *fch, *fchg, *res3, *lnf, *logits;
    float *ln1_mean, *ln1_rstd, *ln2_mean, *ln2_rstd, *lnf_mean, *lnf_rstd;
    float *att;                        // fp32 path: (L, B, NH, T, T) probabilities
    float *lse;                        // bf16 path: (L, B, NH, T) log-sum-exp of each row
    float *losses, *loss;
    // backward scratch
    void *dresid, *dbufC, *dqkv, *dfch;
    float *datt;                       // fp32 path: (B, NH, T, T) dS
    float *attn_scratch;               // bf16 path: (B, NH, T) rowsum(dO * O)
    float *partials;                   // column-sum / layernorm partials
    size_t partials_floats;
    float *enc_partial;                // (BT, C) encoder-backward partial sums
    unsigned* sorted_keys;             // (BT)
    unsigned* sort_tmp;                // (BT) keys between radix passes
    unsigned* sort_hist;               // (256 x ceil(BT / 1024)) digit counts, then offsets
    float* red_arena;                  // per-reduction partials of one backward pass (deferred sums)
    size_t red_arena_floats;
    int *tokens, *targets;             // staging copies of the last batch
    unsigned* err;
    // fp8 mode: e4m3 copy of the layernorm output feeding the qkv / fc products (one
    // layer at a time) with its per-row unscaling factors; e4m3 shadows of qkvw and fcw
    // with per-(tensor, layer) factors and the amax words they are computed from
    uint8_t* lnq;
    float* lnq_deq;
    uint8_t *wq_qkv, *wq_fc;
    float* wq_deq;                     // [0, L): qkvw of layer l; [L, 2L): fcw of layer l
    unsigned* wq_amax;
    // Muon (bf16 / fp8 modes): the normalized momentum of one tensor's L matrices (bf16),
    // a ping-pong matrix, the Gram matrix S and T = 1.5 I - 0.5 S, sum-of-squares partials
    bf16 *mu_x, *mu_xb, *mu_s, *mu_t;
    float* mu_part;
    // state
    int B, T;
    int have_fwd, have_targets;
    // the whole step as one CUDA graph, captured for (gB, gT) and the optimizer (g_opt:
    // 0 AdamW, 1 Muon with its constants) on the second step of that shape; the scalars
    // of its AdamW nodes (one per flat range they update) are set before each launch
    int use_graph, g_seen;
    int gB, gT;
    int g_opt, g_ns;
    float g_lrmu, g_mu, g_wdmu;
    cudaStream_t cap_stream;           // private stream the step is captured on
    cudaGraph_t graph;
    cudaGraphExec_t gexec;
    int g_nadam;
    cudaGraphNode_t g_adam[8];
    float* ga_p[8];                    // each AdamW node's range: pointers, float4 count, grid
    const float* ga_g[8];
    float *ga_m[8], *ga_v[8];
    bf16* ga_sh[8];
    size_t ga_n4[8];
    unsigned ga_grid[8];
    long long g_kernels;
};

static int quantize_model_weights(GPT2* m);
static int layer_err_word(unsigned** out);

static const size_t kAlign = 1024;
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static size_t act_elt(int prec) { return prec == GPT2_FP32 ? 4 : 2; }   // bf16 and fp8 modes: bf16 activations

// Walk the workspace layout: with base == nullptr only sizes are computed.
static size_t plan(GPT2* m, char* base) {
    size_t off = 0;
    auto take = [&](size_t bytes) -> char* {
        off = align_up(off, kAlign);
        char* p = base ? base + off : nullptr;
        off += bytes;
        return p;
    };
    const size_t BT = (size_t)m->maxB * m->maxT;
    const size_t C = m->C, L = m->L, NH = m->NH, Vp = m->Vp;
    const size_t es = act_elt(m->prec);
    const size_t nf = m->n_flat;
    m->params = (float*)take(nf * 4);
    m->grads = (float*)take(nf * 4);
    m->m = (float*)take(nf * 4);
    m->v = (float*)take(nf * 4);
    m->wbf = m->prec != GPT2_FP32 ? (bf16*)take(nf * 2) : nullptr;
    m->encoded = take(BT * C * es);
    m->ln1 = take(L * BT * C * es);
    m->qkv = take(L * BT * 3 * C * es);
    m->atty = take(L * BT * C * es);
    m->res2 = take(L * BT * C * es);
    m->ln2 = take(L * BT * C * es);
    m->fch = take(L * BT * 4 * C * es);
    m->fchg = take(L * BT * 4 * C * es);
    m->res3 = take(L * BT * C * es);
    m->lnf = take(BT * C * es);
    m->logits = take(BT * Vp * es);
    m->ln1_mean = (float*)take(L * BT * 4);
    m->ln1_rstd = (float*)take(L * BT * 4);
    m->ln2_mean = (float*)take(L * BT * 4);
    m->ln2_rstd = (float*)take(L * BT * 4);
    m->lnf_mean = (float*)take(BT * 4);
    m->lnf_rstd = (float*)take(BT * 4);
    const size_t attT = (size_t)m->maxB * NH * m->maxT;
    if (m->prec == GPT2_FP32) {
        m->att = (float*)take(L * attT * m->maxT * 4);
        m->lse = nullptr;
        m->datt = (float*)take(attT * m->maxT * 4);
        m->attn_scratch = nullptr;
    } else {
        m->att = nullptr;
        m->lse = (float*)take(L * attT * 4);
        m->datt = nullptr;
        m->attn_scratch = (float*)take(attention_tc_backward_scratch_floats(m->maxB, m->maxT, m->NH) * 4);
    }
    m->losses = (float*)take(BT * 4);
    m->loss = (float*)take(4);
    m->dresid = take(BT * C * es);
    m->dbufC = take(BT * C * es);
    m->dqkv = take(BT * 3 * C * es);
    m->dfch = take(BT * 4 * C * es);
    // partials: layernorm backward (<= 1024 blocks x 2C) and column sums (<= 256 x 4C);
    // the matmul backward on tensor cores may also use it for split-K partial tiles.
    size_t pf = 1024 * 4 * C;          // >= 296 x 3C (layernorm) and 1024 x 4C (column sums)
    size_t tc_pf = gemm_tc_scratch_floats(BT, C);
    if (tc_pf > pf) pf = tc_pf;
    m->partials_floats = pf;
    m->partials = (float*)take(pf * 4);
    // deferred column sums: (2L+1) layernorm backwards of up to 3C-wide partials over at
    // most 296 blocks, L fc bias gradients of 4C-wide partials over 128-row chunks (or
    // 32-row blocks from the bf16 GELU-backward output stage), and L qkv bias gradients of
    // 3C-wide partials over 128-row chunks (or the 32-row blocks of the bf16 attention
    // backward's output stage)
    {
        const size_t R = std::max<size_t>(1, std::min<size_t>(1024, (BT + 127) / 128));
        const size_t Ra = std::max<size_t>(R, (size_t)attention_tc_bias_partial_rows(m->maxB, m->maxT));
        const size_t Rf = std::max<size_t>(R, (BT + 31) / 32);
        m->red_arena_floats = (2 * L + 1) * 296 * 3 * C + L * Rf * 4 * C + L * Ra * 3 * C;
        m->red_arena = (float*)take(m->red_arena_floats * 4);
    }
    m->enc_partial = (float*)take(BT * C * 4);
    m->sorted_keys = (unsigned*)take(BT * 4);
    m->sort_tmp = (unsigned*)take(BT * 4);
    m->sort_hist = (unsigned*)take(256 * ((BT + RADIX_BLOCK - 1) / RADIX_BLOCK) * 4);
    m->tokens = (int*)take(BT * 4);
    m->targets = (int*)take(BT * 4);
    m->err = (unsigned*)take(16);
    if (m->prec != GPT2_FP32) {
        m->mu_x = (bf16*)take(L * 4 * C * C * 2);
        m->mu_xb = (bf16*)take(L * 4 * C * C * 2);         // the iterates and Gram matrices of
        m->mu_s = (bf16*)take(L * C * C * 2);              // all L layers of a tensor at once
        m->mu_t = (bf16*)take(L * C * C * 2);
        m->mu_part = (float*)take(L * MUON_NB * 4);
    } else {
        m->mu_x = m->mu_xb = m->mu_s = m->mu_t = nullptr;
        m->mu_part = nullptr;
    }
    if (m->prec == GPT2_FP8) {
        m->lnq = (uint8_t*)take(BT * C);
        m->lnq_deq = (float*)take(BT * 4);
        m->wq_qkv = (uint8_t*)take(L * 3 * C * C);
        m->wq_fc = (uint8_t*)take(L * 4 * C * C);
        m->wq_deq = (float*)take(2 * L * 4);
        m->wq_amax = (unsigned*)take(align_up(2 * L * 4, 16));
    } else {
        m->lnq = nullptr;
        m->lnq_deq = nullptr;
        m->wq_qkv = m->wq_fc = nullptr;
        m->wq_deq = nullptr;
        m->wq_amax = nullptr;
    }
    return align_up(off, kAlign);
}

static int validate_cfg(const GPT2Config* c, int maxB, int maxT, int prec) {
    if (!c) return GPT2_EINVAL;
    if (prec != GPT2_FP32 && prec != GPT2_BF16 && prec != GPT2_FP8) return GPT2_EINVAL;
    if (c->num_layers < 1 || c->num_heads < 1 || c->channels < 64) return GPT2_EINVAL;
    if (c->channels % 64 != 0 || c->channels % c->num_heads != 0) return GPT2_EINVAL;
    if (c->channels > 2048) return GPT2_EUNSUPPORTED;
    if (c->channels / c->num_heads > ATT_MAX_HS || (c->channels / c->num_heads) % 8) return GPT2_EUNSUPPORTED;
    // bf16 runs every product on the tensor cores: attention there takes head size 64
    if (prec != GPT2_FP32 && c->channels / c->num_heads != 64) return GPT2_EUNSUPPORTED;
    if (c->vocab_size < 1 || c->padded_vocab_size < c->vocab_size) return GPT2_EINVAL;
    if (c->padded_vocab_size % 64 != 0) return GPT2_EINVAL;
    if (c->max_seq_len < 1 || maxB < 1 || maxT < 1 || maxT > c->max_seq_len) return GPT2_EINVAL;
    const long long BT = (long long)maxB * maxT;
    if (BT > 32768) return GPT2_EUNSUPPORTED;                       // index arithmetic checked up to here
    if ((long long)(c->padded_vocab_size + 1) * BT > 0xffffffffLL) return GPT2_EUNSUPPORTED;
    return GPT2_OK;
}

static void fill_param_table(GPT2* m) {
    const size_t C = m->C, L = m->L;
    size_t num[GPT2_NUM_PARAM_TENSORS] = {
        (size_t)m->Vp * C, (size_t)m->cfg.max_seq_len * C,
        L * C, L * C, L * 3 * C * C, L * 3 * C, L * C * C, L * C,
        L * C, L * C, L * 4 * C * C, L * 4 * C, L * C * 4 * C, L * C,
        C, C};
    size_t off = 0, real = 0;
    for (int i = 0; i < GPT2_NUM_PARAM_TENSORS; i++) {
        off = align_up(off, 64);
        m->poff[i] = off;
        m->pnum[i] = num[i];
        off += num[i];
        real += num[i];
    }
    m->n_flat = align_up(off, 64);
    m->n_real = real - (size_t)(m->Vp - m->V) * C;
}

static void init_dims(GPT2* m, const GPT2Config* cfg, int maxB, int maxT, int prec) {
    memset(m, 0, sizeof(*m));
    m->cfg = *cfg;
    m->maxB = maxB;
    m->maxT = maxT;
    m->prec = prec;
    m->L = cfg->num_layers;
    m->C = cfg->channels;
    m->NH = cfg->num_heads;
    m->V = cfg->vocab_size;
    m->Vp = cfg->padded_vocab_size;
    fill_param_table(m);
}

extern "C" int gpt2_workspace_bytes(const GPT2Config* cfg, int max_B, int max_T, int precision,
                                    size_t* bytes) {
    int st = validate_cfg(cfg, max_B, max_T, precision);
    if (st) return st;
    if (!bytes) return GPT2_EINVAL;
    GPT2 tmp;
    init_dims(&tmp, cfg, max_B, max_T, precision);
    *bytes = plan(&tmp, nullptr);
    return GPT2_OK;
}

static int launch_zero_floats(cudaStream_t s, float* p, size_t n);
static int launch_zero(cudaStream_t s, void* p, size_t bytes) {
    // bytes is a multiple of 16 for every region this is used on
    size_t n4 = bytes / 16;
    if (n4 == 0) return GPT2_OK;
    int grid = (int)std::min<size_t>(ceil_div_sz(n4, 256), 148 * 8);
    ProfScope ps(s, PC_MISC, 0, (double)bytes);
    launch_pdl(zero_kernel, grid, 256, 0, s, (float4*)p, n4);
    rt_note_launches(1);
    CK(cudaGetLastError());
    return GPT2_OK;
}
// any float count and alignment (the short alignment gaps of the flat buffer)
static int launch_zero_floats(cudaStream_t s, float* p, size_t n) {
    CK(cudaMemsetAsync(p, 0, n * sizeof(float), s));
    return GPT2_OK;
}

extern "C" int gpt2_build(const GPT2Config* cfg, int max_B, int max_T, int precision,
                          void* workspace, size_t workspace_bytes, void* stream, GPT2** out) {
    int st = validate_cfg(cfg, max_B, max_T, precision);
    if (st) return st;
    if (!workspace || !out) return GPT2_EINVAL;
    if (((uintptr_t)workspace) % kAlign != 0) return GPT2_EINVAL;
    GPT2* m = (GPT2*)malloc(sizeof(GPT2));
    if (!m) return GPT2_ENOMEM;
    init_dims(m, cfg, max_B, max_T, precision);
    size_t need = plan(m, nullptr);
    if (workspace_bytes < need) { free(m); return GPT2_ENOMEM; }
    plan(m, (char*)workspace);
    m->ws = (char*)workspace;
    m->ws_bytes = workspace_bytes;
    m->stream = (cudaStream_t)stream;
    // bf16 runs only on the tensor-core kernels; no other path is built for it
    if (precision != GPT2_FP32 && (!gemm_tc_available() || !attention_tc_available())) {
        free(m);
        return GPT2_EUNSUPPORTED;
    }
    m->use_graph = 1;
    m->g_seen = 0;
    m->gB = m->gT = 0;
    m->cap_stream = nullptr;
    m->graph = nullptr;
    m->gexec = nullptr;
    m->g_nadam = 0;
    m->g_kernels = 0;
    int rc = launch_zero(m->stream, m->params, (size_t)m->n_flat * 4 * 4);   // params, grads, m, v
    if (rc == GPT2_OK) rc = launch_zero(m->stream, m->err, 16);
    if (rc == GPT2_OK && m->wbf) rc = launch_zero(m->stream, m->wbf, m->n_flat * 2);
    if (rc == GPT2_OK && cudaStreamSynchronize(m->stream) != cudaSuccess) rc = GPT2_ECUDA;
    if (rc != GPT2_OK) { free(m); return rc; }
    *out = m;
    return GPT2_OK;
}

static void drop_graph(GPT2* m) {
    if (m->gexec) cudaGraphExecDestroy(m->gexec);
    if (m->graph) cudaGraphDestroy(m->graph);
    m->gexec = nullptr;
    m->graph = nullptr;
    m->g_nadam = 0;
    m->g_seen = 0;
}

extern "C" void gpt2_free(GPT2* m) {
    if (!m) return;
    drop_graph(m);
    if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
    free(m);
}

extern "C" void gpt2_destroy(GPT2* m) { gpt2_free(m); }

extern "C" int gpt2_set_stream(GPT2* m, void* stream) {
    if (!m) return GPT2_EINVAL;
    m->stream = (cudaStream_t)stream;
    return GPT2_OK;
}

extern "C" int gpt2_num_parameters(const GPT2* m, size_t* n_real, size_t* n_flat) {
    if (!m) return GPT2_EINVAL;
    if (n_real) *n_real = m->n_real;
    if (n_flat) *n_flat = m->n_flat;
    return GPT2_OK;
}

extern "C" int gpt2_num_params(const GPT2* m, size_t* n) {
    if (!m || !n) return GPT2_EINVAL;
    *n = m->n_real;
    return GPT2_OK;
}

extern "C" int gpt2_param_tensor(const GPT2* m, int index, size_t* offset, size_t* numel) {
    if (!m || index < 0 || index >= GPT2_NUM_PARAM_TENSORS) return GPT2_EINVAL;
    if (offset) *offset = m->poff[index];
    if (numel) *numel = m->pnum[index];
    return GPT2_OK;
}

extern "C" float* gpt2_params(GPT2* m) { return m ? m->params : nullptr; }
extern "C" float* gpt2_grads(GPT2* m) { return m ? m->grads : nullptr; }
extern "C" float* gpt2_adam_m(GPT2* m) { return m ? m->m : nullptr; }
extern "C" float* gpt2_adam_v(GPT2* m) { return m ? m->v : nullptr; }
extern "C" int gpt2_param_ptr(GPT2* m, float** master) {
    if (!m || !master) return GPT2_EINVAL;
    *master = m->params;
    return GPT2_OK;
}
extern "C" int gpt2_grad_ptr(GPT2* m, float** grads) {
    if (!m || !grads) return GPT2_EINVAL;
    *grads = m->grads;
    return GPT2_OK;
}
extern "C" float* gpt2_loss(GPT2* m) { return m ? m->loss : nullptr; }
extern "C" float* gpt2_losses(GPT2* m) { return m ? m->losses : nullptr; }
extern "C" void* gpt2_logits(GPT2* m) { return m ? m->logits : nullptr; }

extern "C" int gpt2_sync_params(GPT2* m) {
    if (!m) return GPT2_EINVAL;
    if (m->wbf) {
        launch_pdl(f32_to_bf16_kernel, 148 * 8, 256, 0, m->stream, m->wbf, m->params, m->n_flat);
        rt_note_launches(1);
        CK(cudaGetLastError());
    }
    RC(quantize_model_weights(m));
    int rc = launch_zero(m->stream, m->m, m->n_flat * 4 * 2);   // m and v are adjacent
    return rc;
}

// ------------------------------------------------------------------ sampling
extern "C" int gpt2_sample(GPT2* m, int pos, float temperature, unsigned long long seed, int32_t* out) {
    if (!m || !out || !(temperature > 0.f)) return GPT2_EINVAL;
    if (!m->have_fwd || m->have_targets) return GPT2_ESTATE;
    if (pos < 0 || pos >= m->T) return GPT2_EINVAL;
    const float inv = 1.0f / temperature;
    if (m->prec != GPT2_FP32)
        launch_pdl(sample_kernel<bf16>, m->B, SAMPLE_THREADS, 0, m->stream, out, (const bf16*)m->logits, m->T, pos, m->V,
                                                                   m->Vp, inv, seed);
    else
        launch_pdl(sample_kernel<float>, m->B, SAMPLE_THREADS, 0, m->stream, out, (const float*)m->logits, m->T, pos, m->V,
                                                                    m->Vp, inv, seed);
    rt_note_launches(1);
    CK(cudaGetLastError());
    return GPT2_OK;
}

// ------------------------------------------------------------------ parameter files
#define GPT2_FILE_MAGIC 20240326
#define GPT2_FILE_VERSION 3

static void file_header(const GPT2* m, int32_t (&h)[256]) {
    memset(h, 0, sizeof(h));
    h[0] = GPT2_FILE_MAGIC;
    h[1] = GPT2_FILE_VERSION;
    h[2] = m->cfg.max_seq_len;
    h[3] = m->cfg.vocab_size;
    h[4] = m->cfg.num_layers;
    h[5] = m->cfg.num_heads;
    h[6] = m->cfg.channels;
    h[7] = m->cfg.padded_vocab_size;
}

extern "C" int gpt2_save_params(GPT2* m, const char* path) {
    if (!m || !path) return GPT2_EINVAL;
    CK(cudaStreamSynchronize(m->stream));
    int32_t h[256];
    file_header(m, h);
    FILE* f = fopen(path, "wb");
    if (!f) return GPT2_EIO;
    bool ok = fwrite(h, sizeof(h), 1, f) == 1;
    std::vector<float> buf;
    for (int i = 0; i < GPT2_NUM_PARAM_TENSORS && ok; i++) {
        buf.resize(m->pnum[i]);
        if (cudaMemcpy(buf.data(), m->params + m->poff[i], m->pnum[i] * 4, cudaMemcpyDeviceToHost) != cudaSuccess) {
            fclose(f);
            return GPT2_ECUDA;
        }
        ok = fwrite(buf.data(), 4, m->pnum[i], f) == m->pnum[i];
    }
    if (fclose(f) != 0) ok = false;
    return ok ? GPT2_OK : GPT2_EIO;
}

extern "C" int gpt2_load_params(GPT2* m, const char* path) {
    if (!m || !path) return GPT2_EINVAL;
    int32_t want[256], h[256];
    file_header(m, want);
    FILE* f = fopen(path, "rb");
    if (!f) return GPT2_EIO;
    if (fread(h, sizeof(h), 1, f) != 1 || memcmp(h, want, sizeof(h)) != 0) { fclose(f); return GPT2_EIO; }
    // read everything first, so a short file leaves the parameters untouched
    std::vector<std::vector<float>> t(GPT2_NUM_PARAM_TENSORS);
    for (int i = 0; i < GPT2_NUM_PARAM_TENSORS; i++) {
        t[i].resize(m->pnum[i]);
        if (fread(t[i].data(), 4, m->pnum[i], f) != m->pnum[i]) { fclose(f); return GPT2_EIO; }
    }
    fclose(f);
    CK(cudaStreamSynchronize(m->stream));
    for (int i = 0; i < GPT2_NUM_PARAM_TENSORS; i++)
        CK(cudaMemcpy(m->params + m->poff[i], t[i].data(), m->pnum[i] * 4, cudaMemcpyHostToDevice));
    const int rc = gpt2_sync_params(m);
    if (rc != GPT2_OK) return rc;
    CK(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

// ------------------------------------------------------------------ layer launchers
template <typename T>
static int ln_forward(cudaStream_t s, T* out, float* mean, float* rstd, const T* inp, const T* w,
                      const T* b, int N, int C) {
    constexpr int EPV = Vec<T>::N;
    const int nv = ceil_div(C / EPV, 32);
    dim3 grid(ceil_div(N, LN_WARPS));
    ProfScope ps(s, PC_LAYERNORM_FWD, 0, 2.0 * N * C * sizeof(T) + 8.0 * N + 2.0 * C * sizeof(T));
    rt_note_launches(1);
    switch (nv) {
#define LNF_CASE(k) case k: launch_pdl(layernorm_forward_kernel<T, k>, grid, LN_WARPS * 32, 0, s, out, mean, rstd, inp, w, b, N, C, (uint8_t*)nullptr, (float*)nullptr); break;
        LNF_CASE(1) LNF_CASE(2) LNF_CASE(3) LNF_CASE(4) LNF_CASE(5) LNF_CASE(6) LNF_CASE(7) LNF_CASE(8)
        LNF_CASE(9) LNF_CASE(10) LNF_CASE(11) LNF_CASE(12) LNF_CASE(13) LNF_CASE(14) LNF_CASE(15) LNF_CASE(16)
#undef LNF_CASE
        default: return GPT2_EUNSUPPORTED;
    }
    CK(cudaGetLastError());
    return GPT2_OK;
}

// Layernorm forward that also writes the e4m3 copy of its output (fp8 mode)
template <typename T>
static int ln_forward_q8(cudaStream_t s, T* out, float* mean, float* rstd, const T* inp, const T* w, const T* b,
                         int N, int C, uint8_t* q, float* qdeq) {
    constexpr int EPV = Vec<T>::N;
    const int nv = ceil_div(C / EPV, 32);
    dim3 grid(ceil_div(N, LN_WARPS));
    ProfScope ps(s, PC_LAYERNORM_FWD, 0, 2.0 * N * C * sizeof(T) + 1.0 * N * C + 12.0 * N + 2.0 * C * sizeof(T));
    rt_note_launches(1);
    switch (nv) {
#define LNQ_CASE(k) case k: launch_pdl(layernorm_forward_kernel<T, k, true>, grid, LN_WARPS * 32, 0, s, out, mean, rstd, inp, w, b, N, C, q, qdeq); break;
        LNQ_CASE(1) LNQ_CASE(2) LNQ_CASE(3) LNQ_CASE(4) LNQ_CASE(5) LNQ_CASE(6) LNQ_CASE(7) LNQ_CASE(8)
        LNQ_CASE(9) LNQ_CASE(10) LNQ_CASE(11) LNQ_CASE(12) LNQ_CASE(13) LNQ_CASE(14) LNQ_CASE(15) LNQ_CASE(16)
#undef LNQ_CASE
        default: return GPT2_EUNSUPPORTED;
    }
    CK(cudaGetLastError());
    return GPT2_OK;
}

// Per-tensor e4m3 copies of `ntens` fp32 tensors of `len` elements each (len % 4 == 0),
// back to back from w: codes into q, unscaling factors 2^-k into deq[0..ntens)
static int quantize_tensors(cudaStream_t s, uint8_t* q, float* deq, unsigned* amax_bits, const float* w,
                            size_t len, int ntens) {
    ProfScope ps(s, PC_MISC, 0, 2.0 * 4.0 * len * ntens + 1.0 * len * ntens);
    CK(cudaMemsetAsync(amax_bits, 0, sizeof(unsigned) * ntens, s));
    const int gx = (int)std::min<size_t>(ceil_div_sz(len / 4, 256), 148 * 4 / std::max(1, ntens) + 1);
    rt_note_launches(2);
    launch_pdl(absmax_tensors_kernel, dim3(gx, ntens), 256, 0, s, amax_bits, w, len);
    CK(cudaGetLastError());
    launch_pdl(quantize_tensors_kernel, dim3(gx, ntens), 256, 0, s, q, deq, amax_bits, w, len);
    CK(cudaGetLastError());
    return GPT2_OK;
}

// fp8 mode: refresh the e4m3 shadows of qkvw and fcw from the fp32 master weights
static int quantize_model_weights(GPT2* m) {
    if (m->prec != GPT2_FP8) return GPT2_OK;
    const size_t C = m->C;
    int rc = quantize_tensors(m->stream, m->wq_qkv, m->wq_deq, m->wq_amax, m->params + m->poff[P_QKVW], 3 * C * C, m->L);
    if (rc != GPT2_OK) return rc;
    return quantize_tensors(m->stream, m->wq_fc, m->wq_deq + m->L, m->wq_amax + m->L, m->params + m->poff[P_FCW],
                            4 * C * C, m->L);
}

// two resident blocks per SM on a 148-SM part; each warp then walks ~7 rows at N = 16384
// Column sums deferred to the end of a backward pass: each reduction gets its own
// partial region from the arena and a segment in the batch; flush() reduces them all in
// one launch (the per-segment arithmetic is column_reduce4's, so the sums are the same).
struct RedQueue {
    float* arena;
    size_t cap, used;
    RedBatch batch;
    int n;
    int max_w;
    // a partial region of `floats` (16-byte aligned), or nullptr when the arena is full
    float* take(size_t floats) {
        const size_t need = (floats + 3) & ~(size_t)3;
        if (!arena || used + need > cap || n >= RED_MAX_SEGS) return nullptr;
        float* p = arena + used;
        used += need;
        return p;
    }
    void push(const float* partial, float* out0, float* out1, float* out2, int split, int G, int W, bool assign = false) {
        batch.seg[n++] = RedSeg{partial, out0, out1, out2, split, G, W, assign ? 1 : 0};
        max_w = std::max(max_w, W);
    }
};
static int red_flush(cudaStream_t s, RedQueue& q) {
    if (q.n == 0) return GPT2_OK;
    ProfScope ps(s, PC_MISC, 0, 0);
    rt_note_launches(1);
    launch_pdl(column_reduce_batch_kernel, dim3(ceil_div(q.max_w, 32), q.n), 256, 0, s, q.batch);
    CK(cudaGetLastError());
    q.n = 0;
    q.used = 0;
    q.max_w = 0;
    return GPT2_OK;
}

// column sums of a (G x W) fp32 partial matrix into out0/out1/out2 (see column_reduce_kernel)
static void column_reduce_any(cudaStream_t s, float* out0, float* out1, int split, const float* partial, int G,
                              int W, float* out2) {
    if (W % 4 == 0 && ((uintptr_t)partial & 15) == 0)
        launch_pdl(column_reduce4_kernel, ceil_div(W, 32), 256, 0, s, out0, out1, split, partial, G, W, out2);
    else
        launch_pdl(column_reduce_kernel, ceil_div(W, CR_COLS), CR_COLS * CR_GROUPS, 0, s, out0, out1, split, partial, G, W, out2);
}

static int ln_backward_grid(int N) { return std::max(1, std::min(ceil_div(N, LN_WARPS * 2), 296)); }

// dsum (nullable): also add the column sums of the updated dinp (bias gradient of the
// layer whose output is this residual stream).  The shared-memory pipelined kernel runs
// whenever its stages fit and the rows are 16-byte aligned; otherwise the register one.
template <typename T, int NV, bool SUM>
static int ln_backward_launch(cudaStream_t s, int& G, T* dinp, float* partial, const T* dout, const T* inp, const T* w,
                              const float* mean, const float* rstd, int N, int C, unsigned* err) {
    constexpr int W = SUM ? 3 : 2;
    const size_t pipe_smem = (size_t)(W * C + (SUM ? LN_WARPS * C : 0)) * sizeof(float) +
                             (size_t)LN_WARPS * 2 * 3 * C * sizeof(T) + 2 * LN_WARPS * sizeof(uint64_t);
    const bool aligned = ((((uintptr_t)dinp | (uintptr_t)dout | (uintptr_t)inp) & 15) == 0) &&
                         ((size_t)C * sizeof(T)) % 16 == 0;
    if (aligned && pipe_smem <= 227 * 1024) {
        if (pipe_smem > 48 * 1024 &&
            cudaFuncSetAttribute(layernorm_backward_pipe_kernel<T, NV, SUM>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pipe_smem) != cudaSuccess)
            return GPT2_ECUDA;
        if (pipe_smem > 113 * 1024) G = std::min(G, 148);     // one block per SM: a single wave
        launch_pdl(layernorm_backward_pipe_kernel<T, NV, SUM>, G, LN_WARPS * 32, pipe_smem, s, dinp, partial, dout, inp, w,
                                                                                     mean, rstd, N, C, err);
    } else {
        const size_t smem = (SUM ? (3 + LN_WARPS) : 2) * C * sizeof(float);
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(layernorm_backward_kernel<T, NV, SUM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        launch_pdl(layernorm_backward_kernel<T, NV, SUM>, G, LN_WARPS * 32, smem, s, dinp, partial, dout, inp, w, mean, rstd,
                                                                            N, C);
    }
    CK(cudaGetLastError());
    return GPT2_OK;
}

template <typename T>
static int ln_backward(cudaStream_t s, T* dinp, float* dw, float* db, const T* dout, const T* inp,
                       const T* w, const float* mean, const float* rstd, int N, int C,
                       float* partial, size_t partial_floats, float* dsum = nullptr, unsigned* err = nullptr,
                       RedQueue* q = nullptr, bool assign = false) {
    constexpr int EPV = Vec<T>::N;
    const int nv = ceil_div(C / EPV, 32);
    int G = ln_backward_grid(N);
    const int W = dsum ? 3 : 2;
    // with a queue the partials get their own region and the sums are deferred
    float* qpart = (q && (W * C) % 4 == 0) ? q->take((size_t)G * W * C) : nullptr;
    if (qpart) partial = qpart;
    else if ((size_t)G * W * C > partial_floats) return GPT2_EINVAL;
    ProfScope ps(s, PC_LAYERNORM_BWD, 0, 4.0 * N * C * sizeof(T) + 8.0 * N + 3.0 * C * sizeof(T) + 8.0 * C);
    rt_note_launches(qpart ? 1 : 2);
    int rc = GPT2_EUNSUPPORTED;
    switch (nv) {
#define LNB_CASE(k)                                                                                            \
    case k:                                                                                                    \
        rc = dsum ? ln_backward_launch<T, k, true>(s, G, dinp, partial, dout, inp, w, mean, rstd, N, C, err)   \
                  : ln_backward_launch<T, k, false>(s, G, dinp, partial, dout, inp, w, mean, rstd, N, C, err); \
        break;
        LNB_CASE(1) LNB_CASE(2) LNB_CASE(3) LNB_CASE(4) LNB_CASE(5) LNB_CASE(6) LNB_CASE(7) LNB_CASE(8)
        LNB_CASE(9) LNB_CASE(10) LNB_CASE(11) LNB_CASE(12) LNB_CASE(13) LNB_CASE(14) LNB_CASE(15) LNB_CASE(16)
#undef LNB_CASE
        default: break;
    }
    if (rc != GPT2_OK) return rc;
    if (qpart) {
        q->push(partial, dw, db, dsum, C, G, W * C, assign);         // G may have shrunk in the launcher
        return GPT2_OK;
    }
    // assign without a queue: the outputs are cleared, then the sums added
    if (assign) {
        RC(launch_zero(s, dw, (size_t)C * sizeof(float)));
        RC(launch_zero(s, db, (size_t)C * sizeof(float)));
        if (dsum) RC(launch_zero(s, dsum, (size_t)C * sizeof(float)));
    }
    column_reduce_any(s, dw, db, C, partial, G, W * C, dsum);
    CK(cudaGetLastError());
    return GPT2_OK;
}

static void colsum_shape(int M, int N, int* R, int* rows) {
    (void)N;
    int r = std::max(1, std::min(1024, ceil_div(M, 128)));
    *rows = ceil_div(M, r);
    *R = ceil_div(M, *rows);
}

template <typename T>
static int colsum(cudaStream_t s, float* out, const T* x, int M, int N, float* partial,
                  size_t partial_floats, RedQueue* q = nullptr, bool assign = false) {
    int R, rows;
    colsum_shape(M, N, &R, &rows);
    float* qpart = (q && N % 4 == 0) ? q->take((size_t)R * N) : nullptr;
    if (qpart) partial = qpart;
    else if ((size_t)R * N > partial_floats) return GPT2_EINVAL;
    ProfScope ps(s, PC_BIAS_GRAD, 0, (double)M * N * sizeof(T) + 8.0 * N);
    rt_note_launches(qpart ? 1 : 2);
    constexpr int EPV = Vec<T>::N;
    if (N % EPV) launch_pdl(colsum_partial_scalar_kernel<T>, dim3(ceil_div(N, 128), R), 128, 0, s, partial, x, M, N, rows);
    else launch_pdl(colsum_partial_kernel<T>, dim3(ceil_div(N / EPV, 32), R), CS_WARPS * 32, 0, s, partial, x, M, N, rows);
    CK(cudaGetLastError());
    if (qpart) {
        q->push(partial, out, out, nullptr, N, R, N, assign);
        return GPT2_OK;
    }
    if (assign) RC(launch_zero(s, out, (size_t)N * sizeof(float)));   // cleared, then added
    column_reduce_any(s, out, out, N, partial, R, N, nullptr);
    CK(cudaGetLastError());
    return GPT2_OK;
}

// Linear-layer products.  W is (N, K) row-major for the forward (y = x W^T).  bf16 runs
// on the tcgen05 kernels only (a shape they do not take is GPT2_EUNSUPPORTED); fp32 on
// the FMA kernel.  `err` (device, nullable) is the error word of bounded waits.
template <typename T>
static int mm_forward(cudaStream_t s, T* out, const T* inp, const T* W, const T* bias, int M, int N, int K,
                      int epi, void* aux, unsigned* err, bool gelu_deriv = false, float* scratch = nullptr,
                      size_t scratch_floats = 0) {
    ProfScope ps(s, PC_MATMUL_FWD, 2.0 * M * N * K, 0);
    if constexpr (sizeof(T) == 2) {
        return gemm_tc_forward(s, (bf16*)out, (const bf16*)inp, (const bf16*)W, (const bf16*)bias, M, N, K, epi,
                               (bf16*)aux, err, gelu_deriv);
    } else {
        (void)err;
        EpiArgs ep{out, bias, aux, (long)N};
        cudaError_t e;
        rt_note_launches(1);
        switch (epi) {
            case EPI_STORE:
                e = launch_gemm_simt<T, true, true, EPI_STORE>(s, inp, K, W, K, M, N, K, ep, scratch, scratch_floats);
                break;
            case EPI_GELU:
                e = launch_gemm_simt<T, true, true, EPI_GELU>(s, inp, K, W, K, M, N, K, ep, scratch, scratch_floats);
                break;
            case EPI_RESID:
                e = launch_gemm_simt<T, true, true, EPI_RESID>(s, inp, K, W, K, M, N, K, ep, scratch, scratch_floats);
                break;
            default: return GPT2_EINVAL;
        }
        CK(e);
        return GPT2_OK;
    }
}

// The forward product with e4m3 operands (fp8 mode): A row-scaled codes, W tensor-scaled
static int mm_forward_fp8(cudaStream_t s, bf16* out, const uint8_t* inp, const float* inp_deq, const uint8_t* W,
                          const float* w_deq, const bf16* bias, int M, int N, int K, int epi, bf16* aux,
                          unsigned* err, bool gelu_deriv = false) {
    ProfScope ps(s, PC_MATMUL_FWD, 2.0 * M * N * K, 0);
    return gemm_tc_forward_fp8(s, out, inp, inp_deq, W, w_deq, bias, M, N, K, epi, aux, err, gelu_deriv);
}

// dinp (M,K) = dout (M,N) W (N,K); epi EPI_STORE or EPI_GELU_BWD (aux = pre-activation of dinp's layer)
// csum (bf16 only, nullable): see gemm_tc_backward_dx
template <typename T>
static int mm_backward_dx(cudaStream_t s, T* dinp, const T* dout, const T* W, int M, int N, int K, int epi,
                          const T* aux, unsigned* err, float* csum = nullptr, bool gelu_deriv = false,
                          float* scratch = nullptr, size_t scratch_floats = 0) {
    ProfScope ps(s, PC_MATMUL_BWD_DX, 2.0 * M * N * K, 0);
    if constexpr (sizeof(T) == 2) {
        return gemm_tc_backward_dx(s, (bf16*)dinp, (const bf16*)dout, (const bf16*)W, M, N, K, epi,
                                   (const bf16*)aux, csum, err, gelu_deriv);
    } else {
        (void)err;
        if (csum) return GPT2_EINVAL;
        EpiArgs ep{dinp, nullptr, (void*)aux, (long)K};
        cudaError_t e;
        rt_note_launches(1);
        // C(m, k) = sum_n dout[m][n] W[n][k]: A K-contig over n (lda = N), B(k, n) = W[n*K + k]
        if (epi == EPI_GELU_BWD)
            e = launch_gemm_simt<T, true, false, EPI_GELU_BWD>(s, dout, N, W, K, M, K, N, ep, scratch, scratch_floats);
        else if (epi == EPI_STORE)
            e = launch_gemm_simt<T, true, false, EPI_STORE>(s, dout, N, W, K, M, K, N, ep, scratch, scratch_floats);
        else return GPT2_EINVAL;
        CK(e);
        return GPT2_OK;
    }
}

// dW (N,K) += dout^T (N,M) inp (M,K); `partials` (device fp32, nullable) lets the
// tensor-core product split its contraction when the weight has few tiles
template <typename T>
static int mm_backward_dw(cudaStream_t s, float* dW, const T* dout, const T* inp, int M, int N, int K,
                          float* partials, size_t partials_floats, unsigned* err, bool assign = false) {
    ProfScope ps(s, PC_MATMUL_BWD_DW, 2.0 * M * N * K, 0);
    if constexpr (sizeof(T) == 2) {
        return gemm_tc_backward_dw(s, dW, (const bf16*)dout, (const bf16*)inp, M, N, K, partials, partials_floats,
                                   err, assign);
    } else {
        (void)err;
        if (assign) RC(launch_zero(s, dW, (size_t)N * K * sizeof(float)));
        EpiArgs ep{dW, nullptr, nullptr, (long)K};
        // C(n, k) = sum_m dout[m][n] inp[m][k]: A(n, m) = dout[m*N + n], B(k, m) = inp[m*K + k]
        rt_note_launches(1);
        CK((launch_gemm_simt<T, false, false, EPI_ACC_F32>(s, dout, N, inp, K, N, K, M, ep, partials, partials_floats)));
        return GPT2_OK;
    }
}

static double attn_fwd_flops(int B, int Tn, int C) {
    // q k^T and P v over the causal half (keys j <= t): 2 products x 2 flops per MAC
    return 4.0 * B * C * (double)Tn * (Tn + 1) / 2.0;
}

template <typename T>
static int attn_forward(GPT2* m, cudaStream_t s, T* out, const T* qkv, int l, int B, int Tn) {
    const int C = m->C, NH = m->NH;
    ProfScope ps(s, PC_ATTENTION_FWD, attn_fwd_flops(B, Tn, C), 0);
    if constexpr (sizeof(T) == 2) {
        float* lse = m->lse + (size_t)l * m->maxB * NH * m->maxT;
        return attention_tc_forward(s, (bf16*)out, lse, (const bf16*)qkv, B, Tn, C, NH, m->err);
    } else {
        float* att = m->att + (size_t)l * m->maxB * NH * m->maxT * m->maxT;
        launch_pdl(attention_forward_simt<T>, att_simt_grid(B, NH, Tn), ATT_WARPS * 32, 0, s, out, att, qkv, B, Tn, C, NH);
        rt_note_launches(1);
        CK(cudaGetLastError());
        return GPT2_OK;
    }
}

template <typename T>
static int attn_backward(GPT2* m, cudaStream_t s, T* dqkv, const T* dout, const T* qkv, const T* out,
                         int l, int B, int Tn, float* bias_partial) {
    const int C = m->C, NH = m->NH;
    // dV, dP, dQ, dK: four causal-half products (the recomputed S is not counted)
    ProfScope ps(s, PC_ATTENTION_BWD, 2.0 * attn_fwd_flops(B, Tn, C), 0);
    if constexpr (sizeof(T) == 2) {
        const float* lse = m->lse + (size_t)l * m->maxB * NH * m->maxT;
        return attention_tc_backward(s, (bf16*)dqkv, (const bf16*)dout, (const bf16*)qkv, (const bf16*)out, lse,
                                     m->attn_scratch, bias_partial, B, Tn, C, NH, m->err);
    } else {
        (void)out;
        (void)bias_partial;
        const float* att = m->att + (size_t)l * m->maxB * NH * m->maxT * m->maxT;
        const int grid = att_simt_grid(B, NH, Tn);
        rt_note_launches(3);
        launch_pdl(attention_backward_ds<T>, grid, ATT_WARPS * 32, 0, s, m->datt, att, dout, qkv, B, Tn, C, NH);
        CK(cudaGetLastError());
        launch_pdl(attention_backward_dq<T>, grid, ATT_WARPS * 32, 0, s, dqkv, m->datt, qkv, B, Tn, C, NH);
        CK(cudaGetLastError());
        launch_pdl(attention_backward_dkv<T>, grid, ATT_WARPS * 32, 0, s, dqkv, m->datt, att, qkv, dout, B, Tn, C, NH);
        CK(cudaGetLastError());
        return GPT2_OK;
    }
}


// ------------------------------------------------------------------ forward
template <typename T>
static int forward_impl(GPT2* m, int B, int Tn, bool with_targets) {
    cudaStream_t s = m->stream;
    const int C = m->C, L = m->L, BT = B * Tn;
    const size_t BTmax = (size_t)m->maxB * m->maxT;
    const T* W = (sizeof(T) == 2) ? (const T*)m->wbf : (const T*)m->params;
    auto P = [&](int i) { return W + m->poff[i]; };
    const bool fp8 = m->prec == GPT2_FP8;
    T* encoded = (T*)m->encoded;
    {
        constexpr int EPV = Vec<T>::N;
        size_t n = (size_t)BT * (C / EPV);
        ProfScope ps(s, PC_ENCODER_FWD, 0, 3.0 * BT * C * sizeof(T) + 4.0 * BT);
        rt_note_launches(1);
        launch_pdl(encoder_forward_kernel<T>, (unsigned)ceil_div_sz(n, 256), 256, 0, s, encoded, m->tokens, P(P_WTE), P(P_WPE), BT, Tn, C, m->V, m->err);
        CK(cudaGetLastError());
    }
    const T* x = encoded;
    for (int l = 0; l < L; l++) {
        T* ln1 = (T*)m->ln1 + l * BTmax * C;
        T* qkv = (T*)m->qkv + l * BTmax * 3 * C;
        T* atty = (T*)m->atty + l * BTmax * C;
        T* res2 = (T*)m->res2 + l * BTmax * C;
        T* ln2 = (T*)m->ln2 + l * BTmax * C;
        T* fch = (T*)m->fch + l * BTmax * 4 * C;
        T* fchg = (T*)m->fchg + l * BTmax * 4 * C;
        T* res3 = (T*)m->res3 + l * BTmax * C;
        float* m1 = m->ln1_mean + l * BTmax; float* r1 = m->ln1_rstd + l * BTmax;
        float* m2 = m->ln2_mean + l * BTmax; float* r2 = m->ln2_rstd + l * BTmax;
        if (fp8) {
            // fp8 mode: the layernorm also writes its output as row-scaled e4m3 codes, the
            // qkv product reads them and the e4m3 weight shadow
            RC(ln_forward_q8<T>(s, ln1, m1, r1, x, P(P_LN1W) + l * C, P(P_LN1B) + l * C, BT, C, m->lnq, m->lnq_deq));
            RC(mm_forward_fp8(s, (bf16*)qkv, m->lnq, m->lnq_deq, m->wq_qkv + (size_t)l * 3 * C * C, m->wq_deq + l,
                              (const bf16*)(P(P_QKVB) + l * 3 * C), BT, 3 * C, C, EPI_STORE, nullptr, m->err));
        } else {
            RC(ln_forward<T>(s, ln1, m1, r1, x, P(P_LN1W) + l * C, P(P_LN1B) + l * C, BT, C));
            // fp32: m->partials doubles as the split-contraction scratch of the FMA products
            // (every other user of it consumes its partials before the next kernel)
            RC(mm_forward<T>(s, qkv, ln1, P(P_QKVW) + (size_t)l * 3 * C * C, P(P_QKVB) + l * 3 * C, BT, 3 * C, C, EPI_STORE, nullptr, m->err,
                             false, m->partials, m->partials_floats));
        }
        RC(attn_forward<T>(m, s, atty, qkv, l, B, Tn));
        RC(mm_forward<T>(s, res2, atty, P(P_ATTPROJW) + (size_t)l * C * C, P(P_ATTPROJB) + l * C, BT, C, C, EPI_RESID, (void*)x, m->err,
                         false, m->partials, m->partials_floats));
        if (fp8) {
            RC(ln_forward_q8<T>(s, ln2, m2, r2, res2, P(P_LN2W) + l * C, P(P_LN2B) + l * C, BT, C, m->lnq, m->lnq_deq));
            RC(mm_forward_fp8(s, (bf16*)fchg, m->lnq, m->lnq_deq, m->wq_fc + (size_t)l * 4 * C * C, m->wq_deq + m->L + l,
                              (const bf16*)(P(P_FCB) + l * 4 * C), BT, 4 * C, C, EPI_GELU, (bf16*)fch, m->err, true));
        } else {
            RC(ln_forward<T>(s, ln2, m2, r2, res2, P(P_LN2W) + l * C, P(P_LN2B) + l * C, BT, C));
            // bf16: fch keeps gelu'(h) (what the backward needs) instead of h
            RC(mm_forward<T>(s, fchg, ln2, P(P_FCW) + (size_t)l * 4 * C * C, P(P_FCB) + l * 4 * C, BT, 4 * C, C, EPI_GELU, fch, m->err,
                             sizeof(T) == 2, m->partials, m->partials_floats));
        }
        RC(mm_forward<T>(s, res3, fchg, P(P_FCPROJW) + (size_t)l * 4 * C * C, P(P_FCPROJB) + l * C, BT, C, 4 * C, EPI_RESID, res2, m->err,
                         false, m->partials, m->partials_floats));
        x = res3;
    }
    RC(ln_forward<T>(s, (T*)m->lnf, m->lnf_mean, m->lnf_rstd, x, P(P_LNFW), P(P_LNFB), BT, C));
    RC(mm_forward<T>(s, (T*)m->logits, (const T*)m->lnf, P(P_WTE), (const T*)nullptr, BT, m->Vp, C, EPI_STORE, nullptr, m->err,
                     false, m->partials, m->partials_floats));
    if (with_targets) {
        {
            ProfScope ps(s, PC_SOFTMAX_XENT, 0, 2.0 * BT * m->Vp * sizeof(T) + 12.0 * BT);
            rt_note_launches(2);
            launch_pdl(softmax_xent_kernel<T>, BT, XENT_THREADS, 0, s, (T*)m->logits, m->losses, m->targets, m->V, m->Vp,
                                                               1.0f / (float)BT, m->err);
            CK(cudaGetLastError());
            launch_pdl(mean_loss_kernel, 1, 1024, 0, s, m->loss, m->losses, BT, m->err);
            CK(cudaGetLastError());
        }
        // order the token positions by id now; the encoder backward consumes it.  One
        // 8-bit radix pass per byte of the largest id (V stands for invalid ids); the
        // passes alternate buffers so that the last one writes sorted_keys.
        int npass = 0;
        while (npass < 4 && (m->V >> (8 * npass)) > 0) npass++;
        const int nblk = ceil_div(BT, RADIX_BLOCK);
        ProfScope ps2(s, PC_ENCODER_BWD, 0, 8.0 * BT * npass);
        const unsigned* src = nullptr;
        for (int p = 0; p < npass; p++) {
            unsigned* dst = ((npass - 1 - p) & 1) ? m->sort_tmp : m->sorted_keys;
            rt_note_launches(3);
            launch_pdl(radix_hist_kernel, nblk, RADIX_BLOCK, 0, s, m->sort_hist, src, m->tokens, BT, m->V, 8 * p, nblk);
            CK(cudaGetLastError());
            launch_pdl(radix_scan_kernel, 1, RADIX_BLOCK, 0, s, m->sort_hist, 256 * nblk);
            CK(cudaGetLastError());
            launch_pdl(radix_scatter_kernel, nblk, RADIX_BLOCK, 0, s, dst, src, m->tokens, m->sort_hist, BT, m->V, 8 * p, nblk);
            CK(cudaGetLastError());
            src = dst;
        }
    }
    return GPT2_OK;
}

// ------------------------------------------------------------------ backward
template <typename T>
static int backward_impl(GPT2* m) {
    cudaStream_t s = m->stream;
    const int B = m->B, Tn = m->T, C = m->C, L = m->L, BT = B * Tn;
    const size_t BTmax = (size_t)m->maxB * m->maxT;
    const T* W = (sizeof(T) == 2) ? (const T*)m->wbf : (const T*)m->params;
    auto P = [&](int i) { return W + m->poff[i]; };
    auto G = [&](int i) { return m->grads + m->poff[i]; };
    T* dresid = (T*)m->dresid;
    T* dbufC = (T*)m->dbufC;
    T* dqkv = (T*)m->dqkv;
    T* dfch = (T*)m->dfch;
    const T* dlogits = (const T*)m->logits;
    // overwrite: the gradients were not cleared for this backward; each one's first writer
    // stores (the same values as adding into zeros) and what no writer covers is cleared
    const bool ow = m->overwrite != 0;
    float* part = m->partials;
    const size_t pf = m->partials_floats;
    RedQueue rq;
    rq.arena = m->red_arena;
    rq.cap = m->red_arena_floats;
    rq.used = 0;
    rq.n = 0;
    rq.max_w = 0;
    // LM head (tied): dlnf = dlogits wte; dwte += dlogits^T lnf
    RC(mm_backward_dx<T>(s, dbufC, dlogits, P(P_WTE), BT, m->Vp, C, EPI_STORE, nullptr, m->err, nullptr, false,
                         m->partials, m->partials_floats));
    RC(mm_backward_dw<T>(s, G(P_WTE), dlogits, (const T*)m->lnf, BT, m->Vp, C, m->partials, m->partials_floats, m->err,
                         ow));
    RC(launch_zero(s, dresid, (size_t)BT * C * sizeof(T)));
    const T* xlast = (const T*)m->res3 + (L - 1) * BTmax * C;
    // the updated residual gradient is d(res3) of the last layer: its column sums are
    // that layer's MLP-projection bias gradient
    RC(ln_backward<T>(s, dresid, G(P_LNFW), G(P_LNFB), dbufC, xlast, P(P_LNFW), m->lnf_mean, m->lnf_rstd, BT, C, part, pf,
                      G(P_FCPROJB) + (L - 1) * C, m->err, &rq, ow));
    for (int l = L - 1; l >= 0; l--) {
        const T* x_in = (l == 0) ? (const T*)m->encoded : (const T*)m->res3 + (l - 1) * BTmax * C;
        const T* ln1 = (const T*)m->ln1 + l * BTmax * C;
        const T* qkv = (const T*)m->qkv + l * BTmax * 3 * C;
        const T* atty = (const T*)m->atty + l * BTmax * C;
        const T* res2 = (const T*)m->res2 + l * BTmax * C;
        const T* ln2 = (const T*)m->ln2 + l * BTmax * C;
        const T* fch = (const T*)m->fch + l * BTmax * 4 * C;
        const T* fchg = (const T*)m->fchg + l * BTmax * 4 * C;
        const float* m1 = m->ln1_mean + l * BTmax; const float* r1 = m->ln1_rstd + l * BTmax;
        const float* m2 = m->ln2_mean + l * BTmax; const float* r2 = m->ln2_rstd + l * BTmax;
        // MLP output projection (dresid = d res3); in bf16 its GELU-backward output stage
        // also sums the columns of dfch for the fc bias gradient (a deferred sum)
        const int frows = (int)ceil_div_sz(BT, 32);
        float* fcb_part = sizeof(T) == 2 ? rq.take((size_t)frows * 4 * C) : nullptr;
        RC(mm_backward_dx<T>(s, dfch, dresid, P(P_FCPROJW) + (size_t)l * 4 * C * C, BT, C, 4 * C, EPI_GELU_BWD, fch, m->err,
                             fcb_part, sizeof(T) == 2, m->partials, m->partials_floats));
        if (fcb_part) rq.push(fcb_part, G(P_FCB) + l * 4 * C, G(P_FCB) + l * 4 * C, nullptr, 4 * C, frows, 4 * C, ow);
        RC(mm_backward_dw<T>(s, G(P_FCPROJW) + (size_t)l * 4 * C * C, dresid, fchg, BT, C, 4 * C, m->partials, m->partials_floats, m->err, ow));
        // MLP input projection
        RC(mm_backward_dx<T>(s, dbufC, dfch, P(P_FCW) + (size_t)l * 4 * C * C, BT, 4 * C, C, EPI_STORE, nullptr, m->err,
                             nullptr, false, m->partials, m->partials_floats));
        RC(mm_backward_dw<T>(s, G(P_FCW) + (size_t)l * 4 * C * C, dfch, ln2, BT, 4 * C, C, m->partials, m->partials_floats, m->err, ow));
        if (!fcb_part) RC(colsum<T>(s, G(P_FCB) + l * 4 * C, dfch, BT, 4 * C, part, pf, &rq, ow));
        // ln2 (adds into dresid: d res2 = d res3 + LN2 backward)
        RC(ln_backward<T>(s, dresid, G(P_LN2W) + l * C, G(P_LN2B) + l * C, dbufC, res2, P(P_LN2W) + l * C, m2, r2, BT, C, part, pf,
                          G(P_ATTPROJB) + l * C, m->err, &rq, ow));      // d(res2) column sums: attention-projection bias
        // attention output projection (dresid = d res2)
        RC(mm_backward_dx<T>(s, dbufC, dresid, P(P_ATTPROJW) + (size_t)l * C * C, BT, C, C, EPI_STORE, nullptr, m->err,
                             nullptr, false, m->partials, m->partials_floats));
        RC(mm_backward_dw<T>(s, G(P_ATTPROJW) + (size_t)l * C * C, dresid, atty, BT, C, C, m->partials, m->partials_floats, m->err, ow));
        // attention; in bf16 its output stage also sums the columns of dqkv for the qkv
        // bias gradient (reduced with the other deferred sums)
        const int qrows = attention_tc_bias_partial_rows(B, Tn);
        float* qkvb_part = sizeof(T) == 2 ? rq.take((size_t)qrows * 3 * C) : nullptr;
        RC(attn_backward<T>(m, s, dqkv, dbufC, qkv, atty, l, B, Tn, qkvb_part));
        if (qkvb_part) rq.push(qkvb_part, G(P_QKVB) + l * 3 * C, G(P_QKVB) + l * 3 * C, nullptr, 3 * C, qrows, 3 * C, ow);
        // qkv projection
        RC(mm_backward_dx<T>(s, dbufC, dqkv, P(P_QKVW) + (size_t)l * 3 * C * C, BT, 3 * C, C, EPI_STORE, nullptr, m->err,
                             nullptr, false, m->partials, m->partials_floats));
        RC(mm_backward_dw<T>(s, G(P_QKVW) + (size_t)l * 3 * C * C, dqkv, ln1, BT, 3 * C, C, m->partials, m->partials_floats, m->err, ow));
        if (!qkvb_part) RC(colsum<T>(s, G(P_QKVB) + l * 3 * C, dqkv, BT, 3 * C, part, pf, &rq, ow));
        // ln1 (dresid becomes d x_l)
        RC(ln_backward<T>(s, dresid, G(P_LN1W) + l * C, G(P_LN1B) + l * C, dbufC, x_in, P(P_LN1W) + l * C, m1, r1, BT, C, part, pf,
                          l > 0 ? G(P_FCPROJB) + (l - 1) * C : nullptr, m->err, &rq, ow));   // d(res3) of layer l-1
        if (rq.n + 4 > RED_MAX_SEGS) RC(red_flush(s, rq));
    }
    // the deferred column sums (layernorm weight and bias gradients, linear biases)
    RC(red_flush(s, rq));
    // encoder: deterministic scatter-add into dwte (ids sorted in the forward), dwpe
    ProfScope ps(s, PC_ENCODER_BWD, 0, (double)BT * C * sizeof(T) + 8.0 * BT * C + 8.0 * Tn * C);
    rt_note_launches(3);
    const int enc_threads = std::min(256, ceil_div(C / Vec<T>::N, 32) * 32);
    launch_pdl(encoder_backward_wte_partial<T>, ceil_div(BT, ENC_CHUNK), enc_threads, 0, s, G(P_WTE), m->enc_partial, m->sorted_keys, dresid, BT, C, m->V);
    CK(cudaGetLastError());
    launch_pdl(encoder_backward_wte_final, ceil_div(BT, ENC_CHUNK), 256, 0, s, G(P_WTE), m->enc_partial, m->sorted_keys, BT, C, m->V);
    CK(cudaGetLastError());
    launch_pdl(encoder_backward_wpe<T>, ceil_div(Tn * C / Vec<T>::N, 256), 256, 0, s, G(P_WPE), dresid, B, Tn, C,
               ow ? 1 : 0);
    CK(cudaGetLastError());
    if (ow) {
        // what no writer covers: position rows past this T, and the alignment gaps of the
        // flat buffer
        const int Tw = m->cfg.max_seq_len;                 // rows of the position table
        if (Tn < Tw) RC(launch_zero(s, G(P_WPE) + (size_t)Tn * C, (size_t)(Tw - Tn) * C * sizeof(float)));
        for (int i = 0; i < GPT2_NUM_PARAM_TENSORS; i++) {
            const size_t end = m->poff[i] + m->pnum[i];
            const size_t next = i + 1 < GPT2_NUM_PARAM_TENSORS ? m->poff[i + 1] : m->n_flat;
            if (next > end) RC(launch_zero_floats(s, m->grads + end, next - end));
        }
    }
    return GPT2_OK;
}

static int read_error(GPT2* m) {
    unsigned e = 0;
    CK(cudaMemcpyAsync(&e, m->err, sizeof(unsigned), cudaMemcpyDeviceToHost, m->stream));
    CK(cudaStreamSynchronize(m->stream));
    if (e) {
        CK(cudaMemsetAsync(m->err, 0, sizeof(unsigned), m->stream));
        if (e & ERRBIT_TIMEOUT) return GPT2_ETIMEOUT;
        if (e & ERRBIT_TOKEN) return GPT2_ETOKEN;
        if (e & ERRBIT_NONFINITE) return GPT2_ENONFINITE;
        return GPT2_ECUDA;
    }
    return GPT2_OK;
}

static int check_bt(GPT2* m, int B, int Tn) {
    if (B < 1 || B > m->maxB || Tn < 1 || Tn > m->maxT || Tn > m->cfg.max_seq_len) return GPT2_EINVAL;
    return GPT2_OK;
}

static int forward_dispatch(GPT2* m, int B, int Tn, bool with_targets) {
    m->have_fwd = 0;
    m->have_targets = 0;
    int rc = (m->prec != GPT2_FP32) ? forward_impl<bf16>(m, B, Tn, with_targets)
                                    : forward_impl<float>(m, B, Tn, with_targets);
    if (rc != GPT2_OK) return rc;
    m->B = B;
    m->T = Tn;
    m->have_fwd = 1;
    m->have_targets = with_targets ? 1 : 0;
    return GPT2_OK;
}

extern "C" int gpt2_forward(GPT2* m, const int32_t* tokens, const int32_t* targets, int B, int Tn,
                            float* loss_out) {
    if (!m || !tokens) return GPT2_EINVAL;
    RC(check_bt(m, B, Tn));
    const size_t BT = (size_t)B * Tn;
    CK(cudaMemcpyAsync(m->tokens, tokens, BT * 4, cudaMemcpyDeviceToDevice, m->stream));
    if (targets) CK(cudaMemcpyAsync(m->targets, targets, BT * 4, cudaMemcpyDeviceToDevice, m->stream));
    RC(forward_dispatch(m, B, Tn, targets != nullptr));
    if (loss_out) {
        float l = -1.f;
        if (targets) CK(cudaMemcpyAsync(&l, m->loss, 4, cudaMemcpyDeviceToHost, m->stream));
        int rc = read_error(m);
        *loss_out = l;
        return rc;
    }
    return GPT2_OK;
}

extern "C" int gpt2_zero_grad(GPT2* m) {
    if (!m) return GPT2_EINVAL;
    return launch_zero(m->stream, m->grads, m->n_flat * 4);
}

extern "C" int gpt2_backward(GPT2* m) {
    if (!m) return GPT2_EINVAL;
    if (!m->have_fwd || !m->have_targets) return GPT2_ESTATE;
    int rc = (m->prec != GPT2_FP32) ? backward_impl<bf16>(m) : backward_impl<float>(m);
    // the logits buffer now holds d loss/d logits and has been consumed
    m->have_fwd = 0;
    return rc;
}

// AdamW's launch shape and arguments for step t (bias corrections computed in double)
struct AdamArgs {
    float* p; const float* g; float* mm; float* vv; bf16* shadow; size_t n4;
    float lr, b1, b2, eps, wd, bc1, bc2;
    int grid;
    void* kp[13];
};
static void adam_args(GPT2* m, AdamArgs& a, float lr, float beta1, float beta2, float eps, float wd, int t) {
    a.p = m->params; a.g = m->grads; a.mm = m->m; a.vv = m->v; a.shadow = m->wbf;
    a.n4 = m->n_flat / 4;
    a.lr = lr; a.b1 = beta1; a.b2 = beta2; a.eps = eps; a.wd = wd;
    a.bc1 = (float)(1.0 - pow((double)beta1, (double)t));
    a.bc2 = (float)(1.0 - pow((double)beta2, (double)t));
    a.grid = (int)std::min<size_t>(ceil_div_sz(a.n4, 256), 148 * 16);
    void* kp[13] = {&a.p, &a.g, &a.mm, &a.vv, &a.shadow, &a.n4, &a.lr, &a.b1, &a.b2, &a.eps, &a.wd, &a.bc1, &a.bc2};
    for (int i = 0; i < 13; i++) a.kp[i] = kp[i];
}

extern "C" int gpt2_update(GPT2* m, float lr, float beta1, float beta2, float eps, float wd, int t) {
    if (!m || t < 1) return GPT2_EINVAL;
    AdamArgs a;
    adam_args(m, a, lr, beta1, beta2, eps, wd, t);
    ProfScope ps(m->stream, PC_ADAMW, 0, (double)m->n_flat * (m->wbf ? 30.0 : 28.0));
    rt_note_launches(1);
    launch_pdl(adamw_kernel, a.grid, 256, 0, m->stream, a.p, a.g, a.mm, a.vv, a.shadow, a.n4, a.lr, a.b1, a.b2, a.eps,
                                                a.wd, a.bc1, a.bc2);
    CK(cudaGetLastError());
    return quantize_model_weights(m);        // fp8 mode: the e4m3 weight shadows follow
}

// ------------------------------------------------------------------ Muon
// pimou.com article, sections "优化器的优势" and "相关技术的追溯": the Muon optimizer,
// orthogonalizing with Newton-Schulz iterations (after Bernstein & Newhouse, 2024).
// X (r x c, bf16) <- `iters` cubic Newton-Schulz steps X <- X (1.5 I - 0.5 X^T X) (tall or
// square) or (1.5 I - 0.5 X X^T) X (wide), on the tensor cores; X and xb ping-pong, the
// result's buffer is returned in *res.
// `iters` cubic Newton-Schulz steps on nb r x c bf16 matrices at once (X, xb: nb x r x c;
// S, T: nb x n x n, n = min(r, c)); the products are batched over the nb matrices.
static int newton_schulz_bf16(cudaStream_t s, bf16* X, bf16* xb, bf16* S, bf16* T, int r, int c, int nb, int iters,
                              bf16** res, unsigned* err) {
    const bool tall = r >= c;
    const int n = tall ? c : r;
    for (int k = 0; k < iters; k++) {
        {
            ProfScope ps(s, PC_MATMUL_FWD, 2.0 * nb * n * n * (tall ? r : c), 0);
            // S = X^T X (A(i,k) = X[k][i] and B(j,k) = X[k][j], both MN-major) or X X^T
            RC(tall ? gemm_tc_bf16_batched(s, S, X, true, X, true, c, c, r, nb, err)
                    : gemm_tc_bf16_batched(s, S, X, false, X, false, r, r, c, nb, err));
        }
        rt_note_launches(1);
        launch_pdl(ns_affine_kernel, (unsigned)std::min<size_t>(ceil_div_sz((size_t)nb * n * n, 256), 592), 256, 0, s, T, S,
                   n, nb);
        CK(cudaGetLastError());
        {
            ProfScope ps(s, PC_MATMUL_FWD, 2.0 * nb * r * c * n, 0);
            // xb = X T (B(j,k) = T[k][j], MN-major) or T X (B(j,k) = X[k][j], MN-major)
            RC(tall ? gemm_tc_bf16_batched(s, xb, X, false, T, true, r, c, c, nb, err)
                    : gemm_tc_bf16_batched(s, xb, T, false, X, true, r, c, r, nb, err));
        }
        std::swap(X, xb);
    }
    *res = X;
    return GPT2_OK;
}

extern "C" int gpt2_update_muon(GPT2* m, float lr_muon, float momentum, int ns_iters, float lr, float beta1,
                                float beta2, float eps, float wd, int t) {
    if (!m || t < 1 || ns_iters < 0) return GPT2_EINVAL;
    if (m->prec == GPT2_FP32) return GPT2_EUNSUPPORTED;
    cudaStream_t s = m->stream;
    const int L = m->L, C = m->C;
    const int mu_idx[4] = {P_QKVW, P_ATTPROJW, P_FCW, P_FCPROJW};
    const int mu_r[4] = {3 * C, C, 4 * C, C}, mu_c[4] = {C, C, C, 4 * C};
    // AdamW over the flat ranges between the Muon tensors (gaps are zero and stay zero)
    AdamArgs a;
    adam_args(m, a, lr, beta1, beta2, eps, wd, t);
    size_t start = 0;
    for (int q = 0; q <= 4; q++) {
        const size_t end = q < 4 ? m->poff[mu_idx[q]] : m->n_flat;
        if (end > start) {
            const size_t n4 = (end - start) / 4;
            ProfScope ps(s, PC_ADAMW, 0, (double)(end - start) * 30.0);
            rt_note_launches(1);
            launch_pdl(adamw_kernel, (unsigned)std::min<size_t>(ceil_div_sz(n4, 256), 148 * 16), 256, 0, s, 
                m->params + start, m->grads + start, m->m + start, m->v + start, m->wbf + start, n4, a.lr, a.b1, a.b2,
                a.eps, a.wd, a.bc1, a.bc2);
            CK(cudaGetLastError());
        }
        if (q < 4) start = m->poff[mu_idx[q]] + m->pnum[mu_idx[q]];
    }
    for (int q = 0; q < 4; q++) {
        const size_t off = m->poff[mu_idx[q]], len = (size_t)mu_r[q] * mu_c[q];
        float* mom = m->m + off;
        {
            ProfScope ps(s, PC_MISC, 0, 12.0 * L * len + 2.0 * L * len);
            rt_note_launches(3);
            const size_t n4 = L * len / 4;
            launch_pdl(muon_momentum_kernel, (unsigned)std::min<size_t>(ceil_div_sz(n4, 256), 148 * 8), 256, 0, s, 
                (float4*)mom, (const float4*)(m->grads + off), n4, momentum);
            CK(cudaGetLastError());
            launch_pdl(sumsq_partial_kernel, dim3(MUON_NB, L), 256, 0, s, m->mu_part, mom, len);
            CK(cudaGetLastError());
            launch_pdl(scale_frobenius_bf16_kernel, dim3(std::max(1, 148 * 4 / L), L), 256, 0, s, m->mu_x, mom, m->mu_part, len);
            CK(cudaGetLastError());
        }
        // all L layers' iterations batched in each product when no tile would straddle two
        // layers' matrices (dimensions multiples of 256), else layer by layer
        const bool batched = mu_r[q] % 256 == 0 && mu_c[q] % 256 == 0;
        const int nl = batched ? L : 1;
        for (int l0 = 0; l0 < L; l0 += nl) {
            bf16* res = nullptr;
            RC(newton_schulz_bf16(s, m->mu_x + l0 * len, m->mu_xb + l0 * len, m->mu_s, m->mu_t, mu_r[q], mu_c[q], nl,
                                  ns_iters, &res, m->err));
            ProfScope ps(s, PC_MISC, 0, 14.0 * nl * len);
            rt_note_launches(1);
            launch_pdl(muon_apply_kernel, (unsigned)std::min<size_t>(ceil_div_sz(nl * len / 4, 256), 148 * 4), 256, 0, s,
                       (float4*)(m->params + off + l0 * len), res, m->wbf + off + l0 * len, nl * len / 4, lr_muon, wd);
            CK(cudaGetLastError());
        }
    }
    return quantize_model_weights(m);
}

// The Newton-Schulz iteration alone (single layer): out (r x c, bf16) = `iters` cubic
// steps from G (r x c, fp32) / ||G||_F.  scratch: gpt2_newton_schulz_scratch_bytes.
extern "C" size_t gpt2_newton_schulz_scratch_bytes(int r, int c) {
    if (r <= 0 || c <= 0) return 0;
    const size_t n = (size_t)std::min(r, c);
    return align_up((size_t)r * c * 2, 256) + 2 * align_up(n * n * 2, 256) + align_up(MUON_NB * 4, 256);
}

extern "C" int gpt2_newton_schulz(void* out, const float* G, int r, int c, int iters, void* scratch,
                                  size_t scratch_bytes, void* stream) {
    if (!out || !G || !scratch || r <= 0 || c <= 0 || iters < 0 || r % 8 || c % 8) return GPT2_EINVAL;
    if (scratch_bytes < gpt2_newton_schulz_scratch_bytes(r, c)) return GPT2_EINVAL;
    if ((((uintptr_t)out | (uintptr_t)G | (uintptr_t)scratch) & 255)) return GPT2_EINVAL;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t len = (size_t)r * c, n = (size_t)std::min(r, c);
    char* sc = (char*)scratch;
    bf16* xb = (bf16*)sc;
    bf16* S = (bf16*)(sc + align_up(len * 2, 256));
    bf16* T = (bf16*)((char*)S + align_up(n * n * 2, 256));
    float* part = (float*)((char*)T + align_up(n * n * 2, 256));
    unsigned* err = nullptr;
    RC(layer_err_word(&err));
    rt_note_launches(2);
    launch_pdl(sumsq_partial_kernel, dim3(MUON_NB, 1), 256, 0, s, part, G, len);
    CK(cudaGetLastError());
    launch_pdl(scale_frobenius_bf16_kernel, dim3(148, 1), 256, 0, s, (bf16*)out, G, part, len);
    CK(cudaGetLastError());
    bf16* res = nullptr;
    RC(newton_schulz_bf16(s, (bf16*)out, xb, S, T, r, c, 1, iters, &res, err));
    if (res != (bf16*)out) CK(cudaMemcpyAsync(out, res, len * 2, cudaMemcpyDeviceToDevice, s));
    return GPT2_OK;
}

// forward (with targets), zero_grad, backward and AdamW on the model's stream, as
// launched one by one
// the optimizer of a fused step: AdamW, or Muon on the block matrices with AdamW on the rest
struct StepHp {
    int opt;                           // 0 AdamW, 1 Muon
    float lr, b1, b2, eps, wd;
    int t;
    float lr_mu, mu;                   // Muon
    int ns;
};

static int step_eager(GPT2* m, int B, int Tn, const StepHp& hp) {
    RC(forward_dispatch(m, B, Tn, true));
    // bf16 / fp8: no clear of the gradients; the backward's first write to each stores
    // instead of adding (the same values), and it clears what no writer covers
    if (m->prec == GPT2_FP32) RC(gpt2_zero_grad(m));
    else m->overwrite = 1;
    const int rc = gpt2_backward(m);
    m->overwrite = 0;
    RC(rc);
    if (hp.opt == 1) return gpt2_update_muon(m, hp.lr_mu, hp.mu, hp.ns, hp.lr, hp.b1, hp.b2, hp.eps, hp.wd, hp.t);
    return gpt2_update(m, hp.lr, hp.b1, hp.b2, hp.eps, hp.wd, hp.t);
}

// Capture the step for (B, Tn) into a graph and find its AdamW node.  Lazy set-up
// (function attributes, occupancy queries) has already run in an earlier eager step.
// The capture runs on a private stream (the caller's may be the legacy default stream,
// which cannot be captured); the graph is then launched into the caller's stream.
static int capture_step(GPT2* m, int B, int Tn, StepHp hp) {
    drop_graph(m);
    if (!m->cap_stream) CK(cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking));
    const long long n0 = rt_launches();
    cudaStream_t user = m->stream;
    m->stream = m->cap_stream;
    cudaError_t cb = cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeRelaxed);
    if (cb != cudaSuccess) {
        m->stream = user;
        g_last_cuda_error = cb;
        return GPT2_ECUDA;
    }
    // the AdamW scalars captured here are replaced before every launch
    hp.lr = 0.f;
    hp.t = 1;
    int rc = step_eager(m, B, Tn, hp);
    cudaGraph_t g = nullptr;
    cudaError_t ce = cudaStreamEndCapture(m->cap_stream, &g);
    m->stream = user;
    const long long captured = rt_launches() - n0;
    rt_note_launches(-captured);                // recorded, not run
    if (rc != GPT2_OK || ce != cudaSuccess || !g) {
        if (g) cudaGraphDestroy(g);
        return rc != GPT2_OK ? rc : GPT2_ECUDA;
    }
    size_t nn = 0;
    cudaGraphGetNodes(g, nullptr, &nn);
    std::vector<cudaGraphNode_t> nodes(nn);
    cudaGraphGetNodes(g, nodes.data(), &nn);
    // the AdamW nodes, each with the pointers and float4 count of its range
    int na = 0;
    bool too_many = false;
    for (cudaGraphNode_t nd : nodes) {
        cudaGraphNodeType ty;
        if (cudaGraphNodeGetType(nd, &ty) != cudaSuccess || ty != cudaGraphNodeTypeKernel) continue;
        cudaKernelNodeParams kp;
        if (cudaGraphKernelNodeGetParams(nd, &kp) != cudaSuccess || kp.func != (void*)adamw_kernel) continue;
        if (na == 8) { too_many = true; break; }
        m->g_adam[na] = nd;
        m->ga_p[na] = *(float**)kp.kernelParams[0];
        m->ga_g[na] = *(const float**)kp.kernelParams[1];
        m->ga_m[na] = *(float**)kp.kernelParams[2];
        m->ga_v[na] = *(float**)kp.kernelParams[3];
        m->ga_sh[na] = *(bf16**)kp.kernelParams[4];
        m->ga_n4[na] = *(size_t*)kp.kernelParams[5];
        m->ga_grid[na] = kp.gridDim.x;
        na++;
    }
    cudaGraphExec_t ex = nullptr;
    if (na == 0 || too_many || cudaGraphInstantiate(&ex, g, 0) != cudaSuccess) {
        cudaGraphDestroy(g);
        return GPT2_ECUDA;
    }
    m->graph = g;
    m->gexec = ex;
    m->g_nadam = na;
    m->g_kernels = captured;
    m->gB = B;
    m->gT = Tn;
    return GPT2_OK;
}

// One training step on the batch already in m->tokens / m->targets.  With graphs on and
// the tracer off: the first step of a shape runs eagerly, the second captures the step,
// and from then on each step is one graph launch with this step's AdamW scalars.
static int run_step(GPT2* m, int B, int Tn, const StepHp& hp) {
    if (!m->use_graph || rt_tracing_on()) return step_eager(m, B, Tn, hp);
    // a graph serves one shape and one optimizer (Muon: with its constants)
    const bool same = m->gB == B && m->gT == Tn && m->g_opt == hp.opt &&
                      (hp.opt == 0 || (m->g_ns == hp.ns && m->g_lrmu == hp.lr_mu && m->g_mu == hp.mu &&
                                       m->g_wdmu == hp.wd));
    if (m->gexec && !same) drop_graph(m);
    if (!m->gexec) {
        if (!m->g_seen || !same) {
            m->g_seen = 1;
            m->gB = B;
            m->gT = Tn;
            m->g_opt = hp.opt;
            m->g_ns = hp.ns;
            m->g_lrmu = hp.lr_mu;
            m->g_mu = hp.mu;
            m->g_wdmu = hp.wd;
            return step_eager(m, B, Tn, hp);
        }
        int rc = capture_step(m, B, Tn, hp);
        if (rc != GPT2_OK) {                    // no graph for this model: stay eager
            m->use_graph = 0;
            return step_eager(m, B, Tn, hp);
        }
    }
    for (int i = 0; i < m->g_nadam; i++) {
        AdamArgs a;
        adam_args(m, a, hp.lr, hp.b1, hp.b2, hp.eps, hp.wd, hp.t);
        a.p = m->ga_p[i];
        a.g = m->ga_g[i];
        a.mm = m->ga_m[i];
        a.vv = m->ga_v[i];
        a.shadow = m->ga_sh[i];
        a.n4 = m->ga_n4[i];
        cudaKernelNodeParams kp = {};
        kp.func = (void*)adamw_kernel;
        kp.gridDim = dim3(m->ga_grid[i]);
        kp.blockDim = dim3(256);
        kp.sharedMemBytes = 0;
        kp.kernelParams = a.kp;
        kp.extra = nullptr;
        CK(cudaGraphExecKernelNodeSetParams(m->gexec, m->g_adam[i], &kp));
    }
    CK(cudaGraphLaunch(m->gexec, m->stream));
    rt_note_launches(m->g_kernels);
    m->B = B;
    m->T = Tn;
    m->have_fwd = 0;                            // the logits now hold d loss / d logits
    m->have_targets = 1;
    return GPT2_OK;
}

extern "C" int gpt2_set_graphs(GPT2* m, int enable) {
    if (!m) return GPT2_EINVAL;
    m->use_graph = enable ? 1 : 0;
    if (!enable) drop_graph(m);
    return GPT2_OK;
}

extern "C" int gpt2_step(GPT2* m, const int32_t* tokens, const int32_t* targets, int B, int Tn, float lr,
                         float beta1, float beta2, float eps, float wd, int t, float* loss_out) {
    if (!m || !tokens || !targets || t < 1) return GPT2_EINVAL;
    RC(check_bt(m, B, Tn));
    const size_t BT = (size_t)B * Tn;
    CK(cudaMemcpyAsync(m->tokens, tokens, BT * 4, cudaMemcpyDeviceToDevice, m->stream));
    CK(cudaMemcpyAsync(m->targets, targets, BT * 4, cudaMemcpyDeviceToDevice, m->stream));
    RC(run_step(m, B, Tn, StepHp{0, lr, beta1, beta2, eps, wd, t, 0.f, 0.f, 0}));
    if (!loss_out) return GPT2_OK;
    float l = -1.f;
    CK(cudaMemcpyAsync(&l, m->loss, 4, cudaMemcpyDeviceToHost, m->stream));
    int rc = read_error(m);
    *loss_out = l;
    return rc;
}

extern "C" int gpt2_step_host(GPT2* m, const int32_t* tokens_host, const int32_t* targets_host, int B,
                              int Tn, float lr, float beta1, float beta2, float eps, float wd, int t,
                              float* loss_out) {
    if (!m || !tokens_host || !targets_host || !loss_out) return GPT2_EINVAL;
    RC(check_bt(m, B, Tn));
    const size_t BT = (size_t)B * Tn;
    CK(cudaMemcpyAsync(m->tokens, tokens_host, BT * 4, cudaMemcpyHostToDevice, m->stream));
    CK(cudaMemcpyAsync(m->targets, targets_host, BT * 4, cudaMemcpyHostToDevice, m->stream));
    RC(run_step(m, B, Tn, StepHp{0, lr, beta1, beta2, eps, wd, t, 0.f, 0.f, 0}));
    float l = -1.f;
    CK(cudaMemcpyAsync(&l, m->loss, 4, cudaMemcpyDeviceToHost, m->stream));
    int rc = read_error(m);
    *loss_out = l;
    return rc;
}

extern "C" int gpt2_step_muon(GPT2* m, const int32_t* tokens, const int32_t* targets, int B, int Tn, float lr_muon,
                              float momentum, int ns_iters, float lr, float beta1, float beta2, float eps, float wd,
                              int t, float* loss_out) {
    if (!m || !tokens || !targets || t < 1 || ns_iters < 0) return GPT2_EINVAL;
    if (m->prec == GPT2_FP32) return GPT2_EUNSUPPORTED;
    RC(check_bt(m, B, Tn));
    const size_t BT = (size_t)B * Tn;
    CK(cudaMemcpyAsync(m->tokens, tokens, BT * 4, cudaMemcpyDeviceToDevice, m->stream));
    CK(cudaMemcpyAsync(m->targets, targets, BT * 4, cudaMemcpyDeviceToDevice, m->stream));
    RC(run_step(m, B, Tn, StepHp{1, lr, beta1, beta2, eps, wd, t, lr_muon, momentum, ns_iters}));
    if (!loss_out) return GPT2_OK;
    float l = -1.f;
    CK(cudaMemcpyAsync(&l, m->loss, 4, cudaMemcpyDeviceToHost, m->stream));
    int rc = read_error(m);
    *loss_out = l;
    return rc;
}

extern "C" int gpt2_check(GPT2* m) {
    if (!m) return GPT2_EINVAL;
    return read_error(m);
}

extern "C" int gpt2_last_cuda_error(void) { return (int)g_last_cuda_error; }

extern "C" const char* gpt2_strerror(int st) {
    switch (st) {
        case GPT2_OK: return "ok";
        case GPT2_EINVAL: return "invalid argument";
        case GPT2_ESTATE: return "call out of order (backward needs a forward with targets)";
        case GPT2_ECUDA: return "CUDA error";
        case GPT2_ETOKEN: return "token or target id out of range";
        case GPT2_ENONFINITE: return "non-finite loss";
        case GPT2_ETIMEOUT: return "bounded device wait ran out";
        case GPT2_ENOMEM: return "workspace too small";
        case GPT2_EUNSUPPORTED: return "unsupported shape or precision";
        case GPT2_EIO: return "parameter file unreadable, unwritable or for another model";
        default: return "unknown status";
    }
}

// ------------------------------------------------------------------ single-layer API
// The single-layer entry points have no model, so no workspace error word: their kernels'
// bounded waits report into this word of the library's own device memory (one per
// device), read and cleared by gpt2_layer_check.  Its address is looked up on every call,
// with the caller's device current (a lookup, not an allocation).
static __device__ unsigned g_layer_err;

static int layer_err_word(unsigned** out) {
    void* p = nullptr;
    CK(cudaGetSymbolAddress(&p, g_layer_err));
    *out = (unsigned*)p;
    return GPT2_OK;
}

extern "C" int gpt2_layer_check(void* stream) {
    unsigned* err = nullptr;
    RC(layer_err_word(&err));
    cudaStream_t s = (cudaStream_t)stream;
    unsigned e = 0;
    CK(cudaMemcpyAsync(&e, err, sizeof(unsigned), cudaMemcpyDeviceToHost, s));
    CK(cudaStreamSynchronize(s));
    if (!e) return GPT2_OK;
    CK(cudaMemsetAsync(err, 0, sizeof(unsigned), s));
    CK(cudaStreamSynchronize(s));
    if (e & ERRBIT_TIMEOUT) return GPT2_ETIMEOUT;
    if (e & ERRBIT_TOKEN) return GPT2_ETOKEN;
    if (e & ERRBIT_NONFINITE) return GPT2_ENONFINITE;
    return GPT2_ECUDA;
}

extern "C" int gpt2_layernorm_forward(float* out, float* mean, float* rstd, const float* inp,
                                      const float* weight, const float* bias, int N, int C, void* stream) {
    if (N < 0 || C < 8 || C % 8 || C > 2048) return GPT2_EINVAL;
    if (N == 0) return GPT2_OK;
    if (!out || !mean || !rstd || !inp || !weight || !bias) return GPT2_EINVAL;
    return ln_forward<float>((cudaStream_t)stream, out, mean, rstd, inp, weight, bias, N, C);
}

extern "C" size_t gpt2_layernorm_backward_scratch_bytes(int N, int C) {
    if (N <= 0 || C <= 0) return 0;
    return (size_t)ln_backward_grid(N) * 2 * C * sizeof(float);
}

extern "C" int gpt2_layernorm_backward(float* dinp, float* dweight, float* dbias, const float* dout,
                                       const float* inp, const float* weight, const float* mean,
                                       const float* rstd, int N, int C, void* scratch,
                                       size_t scratch_bytes, void* stream) {
    if (N < 0 || C < 8 || C % 8 || C > 2048) return GPT2_EINVAL;
    if (N == 0) return GPT2_OK;
    if (!dinp || !dweight || !dbias || !dout || !inp || !weight || !mean || !rstd) return GPT2_EINVAL;
    if (!scratch || scratch_bytes < gpt2_layernorm_backward_scratch_bytes(N, C)) return GPT2_EINVAL;
    unsigned* err = nullptr;
    RC(layer_err_word(&err));
    return ln_backward<float>((cudaStream_t)stream, dinp, dweight, dbias, dout, inp, weight, mean, rstd,
                              N, C, (float*)scratch, scratch_bytes / sizeof(float), nullptr, err);
}

static int epi_of(int epilogue) {
    switch (epilogue) {
        case GPT2_EPI_BIAS: return EPI_STORE;
        case GPT2_EPI_GELU: return EPI_GELU;
        case GPT2_EPI_RESIDUAL: return EPI_RESID;
        default: return -1;
    }
}

// ------------------------------------------------------------------ fp8 (single layer)
extern "C" int gpt2_layernorm_forward_fp8(float* out, uint8_t* codes, float* row_deq, float* mean, float* rstd,
                                          const float* inp, const float* weight, const float* bias, int N, int C,
                                          void* stream) {
    if (N < 0 || C < 8 || C % 8 || C > 2048) return GPT2_EINVAL;
    if (N == 0) return GPT2_OK;
    if (!out || !codes || !row_deq || !mean || !rstd || !inp || !weight || !bias) return GPT2_EINVAL;
    if (((uintptr_t)codes & 7)) return GPT2_EINVAL;
    return ln_forward_q8<float>((cudaStream_t)stream, out, mean, rstd, inp, weight, bias, N, C, codes, row_deq);
}

extern "C" int gpt2_quantize_e4m3(uint8_t* codes, float* deq, unsigned* amax_scratch, const float* x, size_t n,
                                  void* stream) {
    if (!codes || !deq || !amax_scratch || !x || n == 0 || n % 4) return GPT2_EINVAL;
    if ((((uintptr_t)codes | (uintptr_t)x) & 15)) return GPT2_EINVAL;
    return quantize_tensors((cudaStream_t)stream, codes, deq, amax_scratch, x, n, 1);
}

extern "C" int gpt2_matmul_forward_fp8(void* out, void* aux, const uint8_t* inp, const float* inp_deq,
                                       const uint8_t* weight, const float* weight_deq, const void* bias, int M, int N,
                                       int K, int epilogue, void* stream) {
    const int epi = epi_of(epilogue);
    if (!out || !inp || !inp_deq || !weight || !weight_deq || M < 0 || N <= 0 || K <= 0 || epi < 0) return GPT2_EINVAL;
    if (epi != EPI_STORE && !aux) return GPT2_EINVAL;
    if (M == 0) return GPT2_OK;
    unsigned* err = nullptr;
    RC(layer_err_word(&err));
    return mm_forward_fp8((cudaStream_t)stream, (bf16*)out, inp, inp_deq, weight, weight_deq, (const bf16*)bias, M, N,
                          K, epi, (bf16*)aux, err);
}

extern "C" int gpt2_fp8_weights(GPT2* m, int which, uint8_t** codes, float** deq) {
    if (!m || !codes || !deq || (which != 0 && which != 1)) return GPT2_EINVAL;
    if (m->prec != GPT2_FP8) return GPT2_ESTATE;
    *codes = which == 0 ? m->wq_qkv : m->wq_fc;
    *deq = m->wq_deq + (which == 0 ? 0 : m->L);
    return GPT2_OK;
}

extern "C" int gpt2_matmul_forward_fused(void* out, void* aux, const void* inp, const void* weight,
                                         const void* bias, int M, int N, int K, int epilogue, int precision,
                                         void* stream) {
    const int epi = epi_of(epilogue);
    if (!out || !inp || !weight || M < 0 || N <= 0 || K <= 0 || epi < 0) return GPT2_EINVAL;
    if (epi != EPI_STORE && !aux) return GPT2_EINVAL;
    if (M == 0) return GPT2_OK;
    cudaStream_t s = (cudaStream_t)stream;
    if (precision == GPT2_FP32)
        return mm_forward<float>(s, (float*)out, (const float*)inp, (const float*)weight, (const float*)bias, M, N,
                                 K, epi, aux, nullptr);
    if (precision == GPT2_BF16) {
        unsigned* err = nullptr;
        RC(layer_err_word(&err));
        return mm_forward<bf16>(s, (bf16*)out, (const bf16*)inp, (const bf16*)weight, (const bf16*)bias, M, N, K,
                                epi, aux, err);
    }
    return GPT2_EINVAL;
}

extern "C" int gpt2_matmul_forward(void* out, const void* inp, const void* weight, const void* bias,
                                   int M, int N, int K, int precision, void* stream) {
    return gpt2_matmul_forward_fused(out, nullptr, inp, weight, bias, M, N, K, GPT2_EPI_BIAS, precision, stream);
}

extern "C" size_t gpt2_matmul_backward_input_gelu_scratch_bytes(int M, int K) {
    if (M <= 0 || K <= 0) return 0;
    int R, rows;
    colsum_shape(M, K, &R, &rows);
    const size_t a = (size_t)R * K, b = (size_t)ceil_div(M, 32) * K;
    return (a > b ? a : b) * sizeof(float);
}

extern "C" int gpt2_matmul_backward_input_gelu(void* dinp, float* dbias, const void* dout, const void* weight,
                                               const void* pre, int M, int N, int K, int precision, void* scratch,
                                               size_t scratch_bytes, void* stream) {
    if (!dinp || !dout || !weight || !pre || M < 0 || N <= 0 || K <= 0) return GPT2_EINVAL;
    if (M == 0) return GPT2_OK;
    if (dbias && (!scratch || ((uintptr_t)scratch & 15) ||
                  scratch_bytes < gpt2_matmul_backward_input_gelu_scratch_bytes(M, K)))
        return GPT2_EINVAL;
    cudaStream_t s = (cudaStream_t)stream;
    float* part = dbias ? (float*)scratch : nullptr;
    if (precision == GPT2_FP32) {
        RC(mm_backward_dx<float>(s, (float*)dinp, (const float*)dout, (const float*)weight, M, N, K, EPI_GELU_BWD,
                                 (const float*)pre, nullptr, nullptr, false, (float*)scratch,
                                 scratch ? scratch_bytes / sizeof(float) : 0));
        if (dbias) RC(colsum<float>(s, dbias, (const float*)dinp, M, K, part, scratch_bytes / sizeof(float)));
        return GPT2_OK;
    }
    if (precision == GPT2_BF16) {
        unsigned* err = nullptr;
        RC(layer_err_word(&err));
        // the column sums come from the product's output stage, 32 rows at a time
        RC(mm_backward_dx<bf16>(s, (bf16*)dinp, (const bf16*)dout, (const bf16*)weight, M, N, K, EPI_GELU_BWD,
                                (const bf16*)pre, err, part));
        if (dbias) {
            column_reduce_any(s, dbias, dbias, K, part, ceil_div(M, 32), K, nullptr);
            CK(cudaGetLastError());
        }
        return GPT2_OK;
    }
    return GPT2_EINVAL;
}

extern "C" size_t gpt2_matmul_backward_scratch_bytes(int M, int N) {
    int R, rows;
    if (M <= 0 || N <= 0) return 0;
    colsum_shape(M, N, &R, &rows);
    size_t a = (size_t)R * N * sizeof(float);
    size_t b = gemm_tc_scratch_floats(M, N) * sizeof(float);
    return a > b ? a : b;
}

extern "C" int gpt2_matmul_backward(void* dinp, float* dweight, float* dbias, const void* dout,
                                    const void* inp, const void* weight, int M, int N, int K,
                                    int precision, void* scratch, size_t scratch_bytes, void* stream) {
    if (!dinp || !dweight || !dout || !inp || !weight || M <= 0 || N <= 0 || K <= 0) return GPT2_EINVAL;
    if (!scratch || scratch_bytes < gpt2_matmul_backward_scratch_bytes(M, N)) return GPT2_EINVAL;
    cudaStream_t s = (cudaStream_t)stream;
    float* part = (float*)scratch;
    size_t pf = scratch_bytes / sizeof(float);
    if (precision == GPT2_FP32) {
        RC(mm_backward_dx<float>(s, (float*)dinp, (const float*)dout, (const float*)weight, M, N, K, EPI_STORE,
                                 nullptr, nullptr, nullptr, false, part, pf));
        RC(mm_backward_dw<float>(s, dweight, (const float*)dout, (const float*)inp, M, N, K, part, pf, nullptr));
        if (dbias) RC(colsum<float>(s, dbias, (const float*)dout, M, N, part, pf));
        return GPT2_OK;
    }
    if (precision == GPT2_BF16) {
        unsigned* err = nullptr;
        RC(layer_err_word(&err));
        RC(mm_backward_dx<bf16>(s, (bf16*)dinp, (const bf16*)dout, (const bf16*)weight, M, N, K, EPI_STORE, nullptr,
                                err));
        RC(mm_backward_dw<bf16>(s, dweight, (const bf16*)dout, (const bf16*)inp, M, N, K, part, pf, err));
        if (dbias) RC(colsum<bf16>(s, dbias, (const bf16*)dout, M, N, part, pf));
        return GPT2_OK;
    }
    return GPT2_EINVAL;
}

// ------------------------------------------------------------------ attention (single layer)
static int attn_args_ok(int B, int Tn, int C, int NH, int precision) {
    if (B < 1 || Tn < 1 || NH < 1 || C < NH || C % NH || C / NH > ATT_MAX_HS || (C / NH) % 8) return 0;
    if (precision == GPT2_BF16 && C / NH != 64) return 0;      // the tensor-core kernels' head size
    return 1;
}

extern "C" int gpt2_attention_forward(void* out, float* lse, const void* qkv, int B, int Tn, int C, int NH,
                                      int precision, void* stream) {
    if (!out || !lse || !qkv) return GPT2_EINVAL;
    if (!attn_args_ok(B, Tn, C, NH, GPT2_FP32)) return GPT2_EINVAL;
    if (!attn_args_ok(B, Tn, C, NH, precision)) return GPT2_EUNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    if (precision == GPT2_BF16) {
        unsigned* err = nullptr;
        RC(layer_err_word(&err));
        return attention_tc_forward(s, (bf16*)out, lse, (const bf16*)qkv, B, Tn, C, NH, err);
    }
    if (precision == GPT2_FP32) {
        launch_pdl(attention_forward_simt<float>, att_simt_grid(B, NH, Tn), ATT_WARPS * 32, 0, s,
            (float*)out, lse, (const float*)qkv, B, Tn, C, NH);
        rt_note_launches(1);
        CK(cudaGetLastError());
        return GPT2_OK;
    }
    return GPT2_EINVAL;
}

// scratch of the attention backward: the kernels' own part (16-byte multiple), then the
// partial column sums of dqkv for the bias gradient
static size_t attn_bwd_own_floats(int B, int Tn, int NH, int precision) {
    const size_t own = precision == GPT2_FP32 ? (size_t)B * NH * Tn * Tn : attention_tc_backward_scratch_floats(B, Tn, NH);
    return (own + 3) / 4 * 4;
}
static size_t attn_bwd_bias_rows(int B, int Tn, int precision) {
    if (precision == GPT2_FP32) {
        int R, rows;
        colsum_shape(B * Tn, 1, &R, &rows);
        return (size_t)R;
    }
    return (size_t)attention_tc_bias_partial_rows(B, Tn);
}

extern "C" size_t gpt2_attention_backward_scratch_bytes(int B, int Tn, int C, int NH, int precision) {
    if (B < 1 || Tn < 1 || C < 1 || NH < 1) return 0;
    return (attn_bwd_own_floats(B, Tn, NH, precision) + attn_bwd_bias_rows(B, Tn, precision) * 3 * C) * sizeof(float);
}

extern "C" int gpt2_attention_backward(void* dqkv, float* dbias, const void* dout, const void* qkv, const void* out,
                                       const float* lse, int B, int Tn, int C, int NH, int precision,
                                       void* scratch, size_t scratch_bytes, void* stream) {
    if (!dqkv || !dout || !qkv || !out || !lse || !scratch) return GPT2_EINVAL;
    if (!attn_args_ok(B, Tn, C, NH, GPT2_FP32)) return GPT2_EINVAL;
    if (!attn_args_ok(B, Tn, C, NH, precision)) return GPT2_EUNSUPPORTED;
    if (scratch_bytes < gpt2_attention_backward_scratch_bytes(B, Tn, C, NH, precision)) return GPT2_EINVAL;
    cudaStream_t s = (cudaStream_t)stream;
    float* part = (float*)scratch + attn_bwd_own_floats(B, Tn, NH, precision);
    const int prow = (int)attn_bwd_bias_rows(B, Tn, precision);
    if (precision == GPT2_BF16) {
        unsigned* err = nullptr;
        RC(layer_err_word(&err));
        RC(attention_tc_backward(s, (bf16*)dqkv, (const bf16*)dout, (const bf16*)qkv, (const bf16*)out, lse,
                                 (float*)scratch, dbias ? part : nullptr, B, Tn, C, NH, err));
        if (dbias) {
            column_reduce_any(s, dbias, dbias, 3 * C, part, prow, 3 * C, nullptr);
            CK(cudaGetLastError());
        }
        return GPT2_OK;
    }
    if (precision == GPT2_FP32) {
        const int grid = att_simt_grid(B, NH, Tn);
        float* ds = (float*)scratch;
        rt_note_launches(3);
        launch_pdl(attention_backward_ds<float>, grid, ATT_WARPS * 32, 0, s, ds, lse, (const float*)dout, (const float*)qkv, B, Tn, C, NH);
        launch_pdl(attention_backward_dq<float>, grid, ATT_WARPS * 32, 0, s, (float*)dqkv, ds, (const float*)qkv, B, Tn, C, NH);
        launch_pdl(attention_backward_dkv<float>, grid, ATT_WARPS * 32, 0, s, (float*)dqkv, ds, lse, (const float*)qkv,
                                                                   (const float*)dout, B, Tn, C, NH);
        CK(cudaGetLastError());
        if (dbias) RC(colsum<float>(s, dbias, (const float*)dqkv, B * Tn, 3 * C, part, (size_t)prow * 3 * C));
        return GPT2_OK;
    }
    return GPT2_EINVAL;
}
