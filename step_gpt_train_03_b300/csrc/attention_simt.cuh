// Causal multi-head self-attention with the probabilities kept in memory (fp32 path).
//
// ujoy.net llm.c article, section "用C语言实现LLM": self-attention forward and backward
// by hand.  Head h of position t reads q, k, v from columns [h*hs, (h+1)*hs) of the
// three C-wide thirds of qkv[b, t]; scores are q.k/sqrt(hs) over keys j <= t; att is
// their row softmax; out = att v.  att (B, NH, T, T) fp32 is kept for the backward.
#pragma once
#include "common.cuh"

#define ATT_WARPS 8
#define ATT_MAX_HS 128

// One warp per query row (b, h, t).
template <typename T>
__global__ void __launch_bounds__(ATT_WARPS * 32)
attention_forward_simt(T* __restrict__ out, float* __restrict__ att, const T* __restrict__ qkv,
                       int B, int Tn, int C, int NH) {
    pdl_wait();
    __shared__ float qs[ATT_WARPS][ATT_MAX_HS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * ATT_WARPS + warp;
    if (gw >= B * NH * Tn) return;
    const int t = gw % Tn, h = (gw / Tn) % NH, b = gw / (Tn * NH);
    const int hs = C / NH, C3 = 3 * C;
    const float scale = 1.0f / sqrtf((float)hs);
    const T* base = qkv + (size_t)b * Tn * C3;
    for (int d = lane; d < hs; d += 32) qs[warp][d] = to_f32(base[(size_t)t * C3 + h * hs + d]);
    __syncwarp();
    float* arow = att + (((size_t)b * NH + h) * Tn + t) * Tn;
    float mx = -INFINITY;
    for (int j = lane; j <= t; j += 32) {
        const T* kj = base + (size_t)j * C3 + C + h * hs;
        float s = 0.f;
        for (int d = 0; d < hs; d++) s += qs[warp][d] * to_f32(kj[d]);
        s *= scale;
        arow[j] = s;
        mx = fmaxf(mx, s);
    }
    mx = warp_max(mx);
    float sum = 0.f;
    for (int j = lane; j <= t; j += 32) {
        float e = expf(arow[j] - mx);
        arow[j] = e;
        sum += e;
    }
    sum = warp_sum(sum);
    const float inv = 1.0f / sum;
    for (int j = lane; j < Tn; j += 32) arow[j] = (j <= t) ? arow[j] * inv : 0.f;
    __syncwarp();
    for (int d = lane; d < hs; d += 32) {
        float o = 0.f;
        for (int j = 0; j <= t; j++) o += arow[j] * to_f32(base[(size_t)j * C3 + 2 * C + h * hs + d]);
        out[((size_t)b * Tn + t) * C + h * hs + d] = from_f32<T>(o);
    }
}

// Backward step 1, one warp per query row: datt_j = dO_t . v_j;
// dS_j = att_j (datt_j - sum_i att_i datt_i); dS (B, NH, T, T) fp32.
template <typename T>
__global__ void __launch_bounds__(ATT_WARPS * 32)
attention_backward_ds(float* __restrict__ ds, const float* __restrict__ att,
                      const T* __restrict__ dout, const T* __restrict__ qkv,
                      int B, int Tn, int C, int NH) {
    pdl_wait();
    __shared__ float dos[ATT_WARPS][ATT_MAX_HS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * ATT_WARPS + warp;
    if (gw >= B * NH * Tn) return;
    const int t = gw % Tn, h = (gw / Tn) % NH, b = gw / (Tn * NH);
    const int hs = C / NH, C3 = 3 * C;
    const T* base = qkv + (size_t)b * Tn * C3;
    for (int d = lane; d < hs; d += 32) dos[warp][d] = to_f32(dout[((size_t)b * Tn + t) * C + h * hs + d]);
    __syncwarp();
    const size_t roff = (((size_t)b * NH + h) * Tn + t) * Tn;
    const float* arow = att + roff;
    float* drow = ds + roff;
    float acc = 0.f;
    for (int j = lane; j <= t; j += 32) {
        const T* vj = base + (size_t)j * C3 + 2 * C + h * hs;
        float dp = 0.f;
        for (int d = 0; d < hs; d++) dp += dos[warp][d] * to_f32(vj[d]);
        drow[j] = dp;
        acc += arow[j] * dp;
    }
    acc = warp_sum(acc);
    __syncwarp();
    for (int j = lane; j < Tn; j += 32) drow[j] = (j <= t) ? arow[j] * (drow[j] - acc) : 0.f;
}

// Backward step 2, one warp per query row: dq = scale * sum_{j<=t} dS[t][j] k_j.
template <typename T>
__global__ void __launch_bounds__(ATT_WARPS * 32)
attention_backward_dq(T* __restrict__ dqkv, const float* __restrict__ ds, const T* __restrict__ qkv,
                      int B, int Tn, int C, int NH) {
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * ATT_WARPS + warp;
    if (gw >= B * NH * Tn) return;
    const int t = gw % Tn, h = (gw / Tn) % NH, b = gw / (Tn * NH);
    const int hs = C / NH, C3 = 3 * C;
    const float scale = 1.0f / sqrtf((float)hs);
    const T* base = qkv + (size_t)b * Tn * C3;
    const float* drow = ds + (((size_t)b * NH + h) * Tn + t) * Tn;
    for (int d = lane; d < hs; d += 32) {
        float s = 0.f;
        for (int j = 0; j <= t; j++) s += drow[j] * to_f32(base[(size_t)j * C3 + C + h * hs + d]);
        dqkv[((size_t)b * Tn + t) * C3 + h * hs + d] = from_f32<T>(s * scale);
    }
}

// Backward step 3, one warp per key row j: dk = scale * sum_{t>=j} dS[t][j] q_t,
// dv = sum_{t>=j} att[t][j] dO_t.
template <typename T>
__global__ void __launch_bounds__(ATT_WARPS * 32)
attention_backward_dkv(T* __restrict__ dqkv, const float* __restrict__ ds,
                       const float* __restrict__ att, const T* __restrict__ qkv,
                       const T* __restrict__ dout, int B, int Tn, int C, int NH) {
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * ATT_WARPS + warp;
    if (gw >= B * NH * Tn) return;
    const int j = gw % Tn, h = (gw / Tn) % NH, b = gw / (Tn * NH);
    const int hs = C / NH, C3 = 3 * C;
    const float scale = 1.0f / sqrtf((float)hs);
    const T* base = qkv + (size_t)b * Tn * C3;
    const size_t hoff = ((size_t)b * NH + h) * Tn * Tn;
    for (int d = lane; d < hs; d += 32) {
        float sk = 0.f, sv = 0.f;
        for (int t = j; t < Tn; t++) {
            size_t o = hoff + (size_t)t * Tn + j;
            sk += ds[o] * to_f32(base[(size_t)t * C3 + h * hs + d]);
            sv += att[o] * to_f32(dout[((size_t)b * Tn + t) * C + h * hs + d]);
        }
        dqkv[((size_t)b * Tn + j) * C3 + C + h * hs + d] = from_f32<T>(sk * scale);
        dqkv[((size_t)b * Tn + j) * C3 + 2 * C + h * hs + d] = from_f32<T>(sv);
    }
}
