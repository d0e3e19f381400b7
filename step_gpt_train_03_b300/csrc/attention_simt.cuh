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
#define ATT_KCH 32                 // rows of a shared-memory chunk: one per lane

// Blocks: one per (b, h, ATT_WARPS consecutive rows); warp w takes row r0 + w.  The
// other operand's rows are staged in chunks of 32 (row pitch hs + 1: lane j reading row
// j, column d hits bank (j + d) mod 32), so each lane's dot product reads shared memory
// without conflicts and the global loads are coalesced.  Sums run in the same order as
// a plain loop over keys (or queries) and over d.
static inline int att_simt_grid(int B, int NH, int Tn) { return B * NH * ((Tn + ATT_WARPS - 1) / ATT_WARPS); }

__device__ __forceinline__ void att_block(int Tn, int NH, int& b, int& h, int& r0) {
    const int nt = (Tn + ATT_WARPS - 1) / ATT_WARPS;
    const int bh = blockIdx.x / nt;
    r0 = (blockIdx.x % nt) * ATT_WARPS;
    b = bh / NH;
    h = bh % NH;
}

// rows [c0, c0 + 32) (zero past Tn), columns [col, col + hs) of a (Tn, pitch) matrix
template <typename T>
__device__ __forceinline__ void att_stage(float (*S)[ATT_MAX_HS + 1], const T* __restrict__ base, int pitch,
                                          int col, int c0, int Tn, int hs) {
    for (int e = threadIdx.x; e < ATT_KCH * hs; e += blockDim.x) {
        const int j = e / hs, d = e % hs;
        S[j][d] = (c0 + j < Tn) ? to_f32(base[(size_t)(c0 + j) * pitch + col + d]) : 0.f;
    }
}

// Forward: scores q_t . k_j for j <= t, row softmax into att, out = att v.
template <typename T>
__global__ void __launch_bounds__(ATT_WARPS * 32)
attention_forward_simt(T* __restrict__ out, float* __restrict__ att, const T* __restrict__ qkv,
                       int B, int Tn, int C, int NH) {
    pdl_wait();
    __shared__ float qs[ATT_WARPS][ATT_MAX_HS];
    __shared__ float ks[ATT_KCH][ATT_MAX_HS + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int b, h, r0;
    att_block(Tn, NH, b, h, r0);
    const int t = r0 + warp, tlast = min(r0 + ATT_WARPS, Tn) - 1;
    const bool active = t < Tn;                      // warp-uniform
    const int hs = C / NH, C3 = 3 * C;
    const float scale = 1.0f / sqrtf((float)hs);
    const T* base = qkv + (size_t)b * Tn * C3;
    if (active)
        for (int d = lane; d < hs; d += 32) qs[warp][d] = to_f32(base[(size_t)t * C3 + h * hs + d]);
    float* arow = att + (((size_t)b * NH + h) * Tn + (active ? t : 0)) * Tn;
    float mx = -INFINITY;
    for (int c0 = 0; c0 <= tlast; c0 += ATT_KCH) {
        __syncthreads();
        att_stage(ks, base, C3, C + h * hs, c0, Tn, hs);
        __syncthreads();
        const int j = c0 + lane;
        if (active && j <= t) {
            float sc = 0.f;
            for (int d = 0; d < hs; d++) sc += qs[warp][d] * ks[lane][d];
            sc *= scale;
            arow[j] = sc;
            mx = fmaxf(mx, sc);
        }
    }
    if (active) {
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
    }
    // out[d] = sum_{j <= t} att_j v_j[d]; lane j's probability reaches the warp by shuffle
    float o[ATT_MAX_HS / 32] = {};
    for (int c0 = 0; c0 <= tlast; c0 += ATT_KCH) {
        __syncthreads();
        att_stage(ks, base, C3, 2 * C + h * hs, c0, Tn, hs);
        __syncthreads();
        if (active && c0 <= t) {
            const float p = (c0 + lane <= t) ? arow[c0 + lane] : 0.f;
            const int jn = min(ATT_KCH, t - c0 + 1);
            for (int jj = 0; jj < jn; jj++) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
                for (int i = 0; i < ATT_MAX_HS / 32; i++)
                    if (lane + 32 * i < hs) o[i] += pj * ks[jj][lane + 32 * i];
            }
        }
    }
    if (active) {
#pragma unroll
        for (int i = 0; i < ATT_MAX_HS / 32; i++)
            if (lane + 32 * i < hs) out[((size_t)b * Tn + t) * C + h * hs + lane + 32 * i] = from_f32<T>(o[i]);
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
    __shared__ float vs[ATT_KCH][ATT_MAX_HS + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int b, h, r0;
    att_block(Tn, NH, b, h, r0);
    const int t = r0 + warp, tlast = min(r0 + ATT_WARPS, Tn) - 1;
    const bool active = t < Tn;
    const int hs = C / NH, C3 = 3 * C;
    const T* base = qkv + (size_t)b * Tn * C3;
    if (active)
        for (int d = lane; d < hs; d += 32) dos[warp][d] = to_f32(dout[((size_t)b * Tn + t) * C + h * hs + d]);
    const size_t roff = (((size_t)b * NH + h) * Tn + (active ? t : 0)) * Tn;
    const float* arow = att + roff;
    float* drow = ds + roff;
    float acc = 0.f;
    for (int c0 = 0; c0 <= tlast; c0 += ATT_KCH) {
        __syncthreads();
        att_stage(vs, base, C3, 2 * C + h * hs, c0, Tn, hs);
        __syncthreads();
        const int j = c0 + lane;
        if (active && j <= t) {
            float dp = 0.f;
            for (int d = 0; d < hs; d++) dp += dos[warp][d] * vs[lane][d];
            drow[j] = dp;
            acc += arow[j] * dp;
        }
    }
    if (!active) return;                             // no barrier follows
    acc = warp_sum(acc);
    for (int j = lane; j < Tn; j += 32) drow[j] = (j <= t) ? arow[j] * (drow[j] - acc) : 0.f;
}

// Backward step 2, one warp per query row: dq = scale * sum_{j<=t} dS[t][j] k_j.
template <typename T>
__global__ void __launch_bounds__(ATT_WARPS * 32)
attention_backward_dq(T* __restrict__ dqkv, const float* __restrict__ ds, const T* __restrict__ qkv,
                      int B, int Tn, int C, int NH) {
    pdl_wait();
    __shared__ float ks[ATT_KCH][ATT_MAX_HS + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int b, h, r0;
    att_block(Tn, NH, b, h, r0);
    const int t = r0 + warp, tlast = min(r0 + ATT_WARPS, Tn) - 1;
    const bool active = t < Tn;
    const int hs = C / NH, C3 = 3 * C;
    const float scale = 1.0f / sqrtf((float)hs);
    const T* base = qkv + (size_t)b * Tn * C3;
    const float* drow = ds + (((size_t)b * NH + h) * Tn + (active ? t : 0)) * Tn;
    float o[ATT_MAX_HS / 32] = {};
    for (int c0 = 0; c0 <= tlast; c0 += ATT_KCH) {
        __syncthreads();
        att_stage(ks, base, C3, C + h * hs, c0, Tn, hs);
        __syncthreads();
        if (active && c0 <= t) {
            const float p = (c0 + lane <= t) ? drow[c0 + lane] : 0.f;
            const int jn = min(ATT_KCH, t - c0 + 1);
            for (int jj = 0; jj < jn; jj++) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
                for (int i = 0; i < ATT_MAX_HS / 32; i++)
                    if (lane + 32 * i < hs) o[i] += pj * ks[jj][lane + 32 * i];
            }
        }
    }
    if (active) {
#pragma unroll
        for (int i = 0; i < ATT_MAX_HS / 32; i++)
            if (lane + 32 * i < hs)
                dqkv[((size_t)b * Tn + t) * C3 + h * hs + lane + 32 * i] = from_f32<T>(o[i] * scale);
    }
}

// Backward step 3, one warp per key row j: dk = scale * sum_{t>=j} dS[t][j] q_t,
// dv = sum_{t>=j} att[t][j] dO_t (queries staged in chunks, dS and att by shuffle).
template <typename T>
__global__ void __launch_bounds__(ATT_WARPS * 32)
attention_backward_dkv(T* __restrict__ dqkv, const float* __restrict__ ds,
                       const float* __restrict__ att, const T* __restrict__ qkv,
                       const T* __restrict__ dout, int B, int Tn, int C, int NH) {
    pdl_wait();
    __shared__ float qs[ATT_KCH][ATT_MAX_HS + 1];
    __shared__ float gs[ATT_KCH][ATT_MAX_HS + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int b, h, r0;
    att_block(Tn, NH, b, h, r0);
    const int j = r0 + warp;
    const bool active = j < Tn;
    const int hs = C / NH, C3 = 3 * C;
    const float scale = 1.0f / sqrtf((float)hs);
    const T* base = qkv + (size_t)b * Tn * C3;
    const T* dbase = dout + (size_t)b * Tn * C;
    const size_t hoff = ((size_t)b * NH + h) * Tn * Tn;
    float sk[ATT_MAX_HS / 32] = {}, sv[ATT_MAX_HS / 32] = {};
    for (int c0 = r0; c0 < Tn; c0 += ATT_KCH) {      // queries t >= the block's first key
        __syncthreads();
        att_stage(qs, base, C3, h * hs, c0, Tn, hs);
        att_stage(gs, dbase, C, h * hs, c0, Tn, hs);
        __syncthreads();
        if (active && c0 + ATT_KCH > j) {
            const int tq = c0 + lane;
            const bool in = tq >= j && tq < Tn;
            const float pd = in ? ds[hoff + (size_t)tq * Tn + j] : 0.f;
            const float pa = in ? att[hoff + (size_t)tq * Tn + j] : 0.f;
            const int tt0 = max(j - c0, 0), tt1 = min(ATT_KCH, Tn - c0);
            for (int tt = tt0; tt < tt1; tt++) {
                const float d1 = __shfl_sync(0xffffffffu, pd, tt), a1 = __shfl_sync(0xffffffffu, pa, tt);
#pragma unroll
                for (int i = 0; i < ATT_MAX_HS / 32; i++)
                    if (lane + 32 * i < hs) {
                        sk[i] += d1 * qs[tt][lane + 32 * i];
                        sv[i] += a1 * gs[tt][lane + 32 * i];
                    }
            }
        }
    }
    if (active) {
#pragma unroll
        for (int i = 0; i < ATT_MAX_HS / 32; i++)
            if (lane + 32 * i < hs) {
                const size_t o = ((size_t)b * Tn + j) * C3 + h * hs + lane + 32 * i;
                dqkv[o + C] = from_f32<T>(sk[i] * scale);
                dqkv[o + 2 * C] = from_f32<T>(sv[i]);
            }
    }
}
