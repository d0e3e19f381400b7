// bf16 causal self-attention, flash-style: the forward keeps only the output and the
// log-sum-exp of each score row; the backward recomputes the probabilities.
//
// ujoy.net llm.c article, section "用C语言实现LLM": self-attention forward and backward
// written by hand.  Head h of position t reads q, k, v from columns [h*hs, (h+1)*hs) of
// the three C-wide thirds of qkv[b, t]; S = q k^T / sqrt(hs) over keys j <= t;
// P = softmax(S); out = P v.  Backward: dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
// dS = P (dP - D), dQ = dS K / sqrt(hs), dK = dS^T Q / sqrt(hs).
//
// This file holds the FMA (SIMT) formulation: one warp per query row (forward, dQ) or
// per key row (dK, dV), 32 keys at a time with an online softmax.
#include "common.cuh"
#include "attention_flash.h"
#include "../../include/gpt2.h"
#include "runtime.h"
#include "attention_mma.cuh"
#include "attention_tc.h"

#define FA_WARPS 8
#define FA_MAX_HS 128

template <int NDV>
__global__ void __launch_bounds__(FA_WARPS * 32)
fa_forward_simt(bf16* __restrict__ out, float* __restrict__ lse, const bf16* __restrict__ qkv,
                int B, int Tn, int C, int NH) {
    __shared__ float qs[FA_WARPS][FA_MAX_HS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * FA_WARPS + warp;
    if (gw >= B * NH * Tn) return;
    // heavy rows (large t) first: reverse the row order inside each (b, h)
    const int t = Tn - 1 - gw % Tn, h = (gw / Tn) % NH, b = gw / (Tn * NH);
    const int hs = C / NH, C3 = 3 * C;
    const float scale = 1.0f / sqrtf((float)hs);
    const bf16* base = qkv + (size_t)b * Tn * C3;
    for (int d = lane; d < hs; d += 32) qs[warp][d] = __bfloat162float(base[(size_t)t * C3 + h * hs + d]);
    __syncwarp();
    float o[NDV];
#pragma unroll
    for (int i = 0; i < NDV; i++) o[i] = 0.f;
    float mx = -INFINITY, sum = 0.f;
    for (int j0 = 0; j0 <= t; j0 += 32) {
        const int j = j0 + lane;
        float s = -INFINITY;
        if (j <= t) {
            const bf16* kj = base + (size_t)j * C3 + C + h * hs;
            float a = 0.f;
            for (int d = 0; d < hs; d++) a += qs[warp][d] * __bfloat162float(kj[d]);
            s = a * scale;
        }
        const float cm = warp_max(s);
        const float nm = fmaxf(mx, cm);
        const float corr = expf(mx - nm);      // mx = -inf on the first chunk gives 0
        const float p = (j <= t) ? expf(s - nm) : 0.f;
        sum = sum * corr + warp_sum(p);
#pragma unroll
        for (int i = 0; i < NDV; i++) o[i] *= corr;
        const int nk = min(32, t - j0 + 1);
        for (int jj = 0; jj < nk; jj++) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            const bf16* vj = base + (size_t)(j0 + jj) * C3 + 2 * C + h * hs;
#pragma unroll
            for (int i = 0; i < NDV; i++) {
                int d = lane + 32 * i;
                if (d < hs) o[i] += pj * __bfloat162float(vj[d]);
            }
        }
        mx = nm;
    }
    const float inv = 1.0f / sum;
#pragma unroll
    for (int i = 0; i < NDV; i++) {
        int d = lane + 32 * i;
        if (d < hs) out[((size_t)b * Tn + t) * C + h * hs + d] = __float2bfloat16_rn(o[i] * inv);
    }
    if (lane == 0) lse[((size_t)b * NH + h) * Tn + t] = mx + logf(sum);
}

// D[b,h,t] = sum_d dO[b,t,h,d] * O[b,t,h,d]; one thread per (b, t, h), 16-byte loads
// (hs a multiple of 8)
__global__ void fa_backward_D(float* __restrict__ D, const bf16* __restrict__ dout,
                              const bf16* __restrict__ out, int B, int Tn, int C, int NH) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= B * Tn * NH) return;
    const int h = idx % NH, bt = idx / NH, b = bt / Tn, t = bt % Tn;
    const int hs = C / NH;
    const size_t o = (size_t)bt * C + h * hs;
    float s = 0.f;
    for (int d = 0; d < hs; d += 8) {
        Vec<bf16> a = load_vec(dout + o + d), c = load_vec(out + o + d);
#pragma unroll
        for (int e = 0; e < 8; e++) s += a.get(e) * c.get(e);
    }
    D[((size_t)b * NH + h) * Tn + t] = s;
}

// The same row sums for hs == 64: eight lanes per (b, h, t) row, one 16-byte packet of
// dO and of O each, added across the eight lanes by shuffles (a warp reads four rows of
// one head at consecutive t: four whole 128-byte segments per load).
__global__ void fa_backward_D64(float* __restrict__ D, const bf16* __restrict__ dout,
                                const bf16* __restrict__ out, int B, int Tn, int C, int NH) {
    // rows in D's own order, so a warp's four results are consecutive floats
    // (B*NH*T < 2^31: 32-bit indices)
    const int row = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 3);
    const int sub = threadIdx.x & 7;
    const bool valid = row < B * NH * Tn;
    float s = 0.f;
    if (valid) {
        const int t = row % Tn, bh = row / Tn;
        const int b = bh / NH, h = bh % NH;
        const size_t o = ((size_t)b * Tn + t) * C + h * 64 + sub * 8;
        Vec<bf16> a = load_vec(dout + o), c = load_vec(out + o);
#pragma unroll
        for (int e = 0; e < 8; e++) s += a.get(e) * c.get(e);
    }
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    if (valid && sub == 0) D[row] = s;
}

// dQ, one warp per query row t: dq = scale * sum_{j<=t} P_tj (dP_tj - D_t) k_j
template <int NDV>
__global__ void __launch_bounds__(FA_WARPS * 32)
fa_backward_dq_simt(bf16* __restrict__ dqkv, const bf16* __restrict__ dout, const bf16* __restrict__ qkv,
                    const float* __restrict__ lse, const float* __restrict__ D, int B, int Tn, int C, int NH) {
    __shared__ float qs[FA_WARPS][FA_MAX_HS], dos[FA_WARPS][FA_MAX_HS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * FA_WARPS + warp;
    if (gw >= B * NH * Tn) return;
    const int t = Tn - 1 - gw % Tn, h = (gw / Tn) % NH, b = gw / (Tn * NH);
    const int hs = C / NH, C3 = 3 * C;
    const float scale = 1.0f / sqrtf((float)hs);
    const bf16* base = qkv + (size_t)b * Tn * C3;
    for (int d = lane; d < hs; d += 32) {
        qs[warp][d] = __bfloat162float(base[(size_t)t * C3 + h * hs + d]);
        dos[warp][d] = __bfloat162float(dout[((size_t)b * Tn + t) * C + h * hs + d]);
    }
    __syncwarp();
    const size_t row = ((size_t)b * NH + h) * Tn + t;
    const float L_t = lse[row], D_t = D[row];
    float acc[NDV];
#pragma unroll
    for (int i = 0; i < NDV; i++) acc[i] = 0.f;
    for (int j0 = 0; j0 <= t; j0 += 32) {
        const int j = j0 + lane;
        float ds = 0.f;
        if (j <= t) {
            const bf16* kj = base + (size_t)j * C3 + C + h * hs;
            const bf16* vj = base + (size_t)j * C3 + 2 * C + h * hs;
            float s = 0.f, dp = 0.f;
            for (int d = 0; d < hs; d++) {
                s += qs[warp][d] * __bfloat162float(kj[d]);
                dp += dos[warp][d] * __bfloat162float(vj[d]);
            }
            const float p = expf(s * scale - L_t);
            ds = p * (dp - D_t);
        }
        const int nk = min(32, t - j0 + 1);
        for (int jj = 0; jj < nk; jj++) {
            const float dsj = __shfl_sync(0xffffffffu, ds, jj);
            const bf16* kj = base + (size_t)(j0 + jj) * C3 + C + h * hs;
#pragma unroll
            for (int i = 0; i < NDV; i++) {
                int d = lane + 32 * i;
                if (d < hs) acc[i] += dsj * __bfloat162float(kj[d]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NDV; i++) {
        int d = lane + 32 * i;
        if (d < hs) dqkv[((size_t)b * Tn + t) * C3 + h * hs + d] = __float2bfloat16_rn(acc[i] * scale);
    }
}

// dK, dV, one warp per key row j: dk = scale * sum_{t>=j} dS_tj q_t, dv = sum_{t>=j} P_tj dO_t
template <int NDV>
__global__ void __launch_bounds__(FA_WARPS * 32)
fa_backward_dkv_simt(bf16* __restrict__ dqkv, const bf16* __restrict__ dout, const bf16* __restrict__ qkv,
                     const float* __restrict__ lse, const float* __restrict__ D, int B, int Tn, int C, int NH) {
    __shared__ float ks[FA_WARPS][FA_MAX_HS], vs[FA_WARPS][FA_MAX_HS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * FA_WARPS + warp;
    if (gw >= B * NH * Tn) return;
    const int j = gw % Tn, h = (gw / Tn) % NH, b = gw / (Tn * NH);   // small j = most work, first
    const int hs = C / NH, C3 = 3 * C;
    const float scale = 1.0f / sqrtf((float)hs);
    const bf16* base = qkv + (size_t)b * Tn * C3;
    for (int d = lane; d < hs; d += 32) {
        ks[warp][d] = __bfloat162float(base[(size_t)j * C3 + C + h * hs + d]);
        vs[warp][d] = __bfloat162float(base[(size_t)j * C3 + 2 * C + h * hs + d]);
    }
    __syncwarp();
    const size_t hrow = ((size_t)b * NH + h) * Tn;
    float ak[NDV], av[NDV];
#pragma unroll
    for (int i = 0; i < NDV; i++) { ak[i] = 0.f; av[i] = 0.f; }
    for (int t0 = j; t0 < Tn; t0 += 32) {
        const int t = t0 + lane;
        float p = 0.f, ds = 0.f;
        if (t < Tn) {
            const bf16* qt = base + (size_t)t * C3 + h * hs;
            const bf16* dot = dout + ((size_t)b * Tn + t) * C + h * hs;
            float s = 0.f, dp = 0.f;
            for (int d = 0; d < hs; d++) {
                s += __bfloat162float(qt[d]) * ks[warp][d];
                dp += __bfloat162float(dot[d]) * vs[warp][d];
            }
            p = expf(s * scale - lse[hrow + t]);
            ds = p * (dp - D[hrow + t]);
        }
        const int nq = min(32, Tn - t0);
        for (int tt = 0; tt < nq; tt++) {
            const float pt = __shfl_sync(0xffffffffu, p, tt);
            const float dst = __shfl_sync(0xffffffffu, ds, tt);
            const bf16* qt = base + (size_t)(t0 + tt) * C3 + h * hs;
            const bf16* dot = dout + ((size_t)b * Tn + t0 + tt) * C + h * hs;
#pragma unroll
            for (int i = 0; i < NDV; i++) {
                int d = lane + 32 * i;
                if (d < hs) {
                    ak[i] += dst * __bfloat162float(qt[d]);
                    av[i] += pt * __bfloat162float(dot[d]);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NDV; i++) {
        int d = lane + 32 * i;
        if (d < hs) {
            dqkv[((size_t)b * Tn + j) * C3 + C + h * hs + d] = __float2bfloat16_rn(ak[i] * scale);
            dqkv[((size_t)b * Tn + j) * C3 + 2 * C + h * hs + d] = __float2bfloat16_rn(av[i]);
        }
    }
}

int attention_flash_forward(cudaStream_t s, bf16* out, float* lse, const bf16* qkv, int B, int Tn, int C,
                            int NH, unsigned* err) {
    const int hs = C / NH;
    if (hs > FA_MAX_HS) return GPT2_EUNSUPPORTED;
    if (hs == AM_HS) {
        int rc = attention_tc_forward(s, out, lse, qkv, B, Tn, C, NH, err);
        if (rc != GPT2_EUNSUPPORTED) return rc;
        dim3 grid((Tn + AMF_Q - 1) / AMF_Q, B * NH);
        attention_forward_mma<<<grid, AMF_THREADS, 0, s>>>(out, lse, qkv, B, Tn, C, NH);
        rt_note_launches(1);
        return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ECUDA;
    }
    const int rows = B * NH * Tn;
    const int grid = ceil_div(rows, FA_WARPS);
    rt_note_launches(1);
    switch (ceil_div(hs, 32)) {
        case 1: fa_forward_simt<1><<<grid, FA_WARPS * 32, 0, s>>>(out, lse, qkv, B, Tn, C, NH); break;
        case 2: fa_forward_simt<2><<<grid, FA_WARPS * 32, 0, s>>>(out, lse, qkv, B, Tn, C, NH); break;
        case 3: fa_forward_simt<3><<<grid, FA_WARPS * 32, 0, s>>>(out, lse, qkv, B, Tn, C, NH); break;
        case 4: fa_forward_simt<4><<<grid, FA_WARPS * 32, 0, s>>>(out, lse, qkv, B, Tn, C, NH); break;
        default: return GPT2_EUNSUPPORTED;
    }
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ECUDA;
}

int attention_flash_backward(cudaStream_t s, bf16* dqkv, const bf16* dout, const bf16* qkv, const bf16* out,
                             const float* lse, float* scratch, int B, int Tn, int C, int NH, unsigned* err) {
    const int hs = C / NH;
    if (hs > FA_MAX_HS) return GPT2_EUNSUPPORTED;
    const int rows = B * NH * Tn;
    const int grid = ceil_div(rows, FA_WARPS);
    rt_note_launches(3);
    if (hs == 64) fa_backward_D64<<<(int)(((long long)rows * 8 + 255) / 256), 256, 0, s>>>(scratch, dout, out, B, Tn, C, NH);
    else fa_backward_D<<<ceil_div(rows, 256), 256, 0, s>>>(scratch, dout, out, B, Tn, C, NH);
    if (hs == AM_HS) {
        int rc = attention_tc_backward(s, dqkv, dout, qkv, lse, scratch, B, Tn, C, NH, err);
        if (rc != GPT2_EUNSUPPORTED) return rc;
        dim3 g2((Tn + AMB_ROWS - 1) / AMB_ROWS, B * NH);
        attention_backward_dkv_mma<<<g2, AMB_THREADS, 0, s>>>(dqkv, dout, qkv, lse, scratch, B, Tn, C, NH);
        attention_backward_dq_mma<<<g2, AMB_THREADS, 0, s>>>(dqkv, dout, qkv, lse, scratch, B, Tn, C, NH);
        return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ECUDA;
    }
    switch (ceil_div(hs, 32)) {
#define FA_BWD_CASE(k)                                                                                 \
    case k:                                                                                            \
        fa_backward_dq_simt<k><<<grid, FA_WARPS * 32, 0, s>>>(dqkv, dout, qkv, lse, scratch, B, Tn, C, NH); \
        fa_backward_dkv_simt<k><<<grid, FA_WARPS * 32, 0, s>>>(dqkv, dout, qkv, lse, scratch, B, Tn, C, NH); \
        break;
        FA_BWD_CASE(1) FA_BWD_CASE(2) FA_BWD_CASE(3) FA_BWD_CASE(4)
#undef FA_BWD_CASE
        default: return GPT2_EUNSUPPORTED;
    }
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ECUDA;
}
