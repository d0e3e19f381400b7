// Memory-bound layers of the training step: encoder, layernorm, fused softmax +
// cross-entropy, AdamW, zeroing and the deterministic column reductions.
//
// Layer list: ujoy.net llm.c article, section "用C语言实现LLM" (encoder, layernorm,
// matmul, self-attention, GELU, residual, softmax, cross-entropy, each with a
// hand-written forward and backward).  Every reduction here runs in a fixed order, so
// results are bitwise reproducible run to run (no floating-point atomics).
#pragma once
#include <cuda_fp8.h>

#include "common.cuh"
#include "tc_ptx.cuh"

// ============================================================== encoder
// out[bt, :] = wte[tok[bt], :] + wpe[bt % T, :].  One thread per 16-byte packet.
// An id outside [0, V) raises ERRBIT_TOKEN and yields a zero row.
template <typename T>
__global__ void encoder_forward_kernel(T* __restrict__ out, const int* __restrict__ tok,
                                       const T* __restrict__ wte, const T* __restrict__ wpe,
                                       int BT, int Tn, int C, int V, unsigned* err) {
    pdl_wait();
    constexpr int EPV = Vec<T>::N;
    const int vpr = C / EPV;
    size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)BT * vpr) return;
    int bt = (int)(idx / vpr), cv = (int)(idx % vpr);
    int t = bt % Tn;
    int id = tok[bt];
    Vec<T> o;
    if (id < 0 || id >= V) {
        if (cv == 0) raise_error(err, ERRBIT_TOKEN);
#pragma unroll
        for (int i = 0; i < EPV; i++) o.set(i, 0.f);
    } else {
        Vec<T> a = load_vec(wte + (size_t)id * C + cv * EPV);
        Vec<T> b = load_vec(wpe + (size_t)t * C + cv * EPV);
#pragma unroll
        for (int i = 0; i < EPV; i++) o.set(i, a.get(i) + b.get(i));
    }
    store_vec(out + (size_t)bt * C + cv * EPV, o);
}

// Sort keys (id * BT + position) ascending; invalid ids count as V, so they sort after
// every valid one.  Equal ids thus become contiguous runs ordered by position, which
// fixes the order of the scatter-add sums below.  The sort is a stable LSD radix sort
// on the id alone (the input is already in position order), 8 bits per pass, 1024 keys
// per block:
// per-block digit counts (digit-major), one exclusive scan, then a stable scatter --
// a key's rank among equal digits is its rank in its warp (matching lanes) plus the
// counts of that digit in the block's earlier warps plus the scanned offset.  Pass 0
// reads the tokens (key = id * BT + position, invalid ids as V); later passes read
// the previous pass's keys.
#define RADIX_BLOCK 1024
__device__ __forceinline__ unsigned radix_key(const unsigned* keys_in, const int* tok, int e, int BT, int V) {
    if (keys_in) return keys_in[e];
    int id = tok[e];
    if (id < 0 || id >= V) id = V;
    return (unsigned)id * (unsigned)BT + (unsigned)e;
}
__global__ void __launch_bounds__(RADIX_BLOCK)
radix_hist_kernel(unsigned* __restrict__ hist, const unsigned* __restrict__ keys_in, const int* __restrict__ tok,
                  int BT, int V, int shift, int nblk) {
    pdl_wait();
    __shared__ unsigned cnt[256];
    if (threadIdx.x < 256) cnt[threadIdx.x] = 0;
    __syncthreads();
    const int e = blockIdx.x * RADIX_BLOCK + threadIdx.x;
    if (e < BT) atomicAdd(&cnt[((radix_key(keys_in, tok, e, BT, V) / (unsigned)BT) >> shift) & 255u], 1u);
    __syncthreads();
    if (threadIdx.x < 256) hist[threadIdx.x * nblk + blockIdx.x] = cnt[threadIdx.x];
}
// exclusive scan of n counts, in place (one block, fixed order)
__global__ void __launch_bounds__(RADIX_BLOCK) radix_scan_kernel(unsigned* __restrict__ hist, int n) {
    pdl_wait();
    __shared__ unsigned wsum[32];
    const int per = (n + RADIX_BLOCK - 1) / RADIX_BLOCK;
    const int b0 = threadIdx.x * per, b1 = min(n, b0 + per);
    unsigned local = 0;
    for (int i = b0; i < b1; i++) local += hist[i];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned inc = local;
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        unsigned w = wsum[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned v = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += v;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    unsigned run = (warp > 0 ? wsum[warp - 1] : 0u) + inc - local;
    for (int i = b0; i < b1; i++) {
        const unsigned c = hist[i];
        hist[i] = run;
        run += c;
    }
}
__global__ void __launch_bounds__(RADIX_BLOCK)
radix_scatter_kernel(unsigned* __restrict__ keys_out, const unsigned* __restrict__ keys_in, const int* __restrict__ tok,
                     const unsigned* __restrict__ hist, int BT, int V, int shift, int nblk) {
    pdl_wait();
    __shared__ unsigned wcnt[RADIX_BLOCK / 32][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < (RADIX_BLOCK / 32) * 256; i += RADIX_BLOCK) (&wcnt[0][0])[i] = 0;
    __syncthreads();
    const int e = blockIdx.x * RADIX_BLOCK + threadIdx.x;
    const bool valid = e < BT;
    const unsigned key = valid ? radix_key(keys_in, tok, e, BT, V) : 0u;
    const unsigned d = valid ? (((key / (unsigned)BT) >> shift) & 255u) : 256u + lane;   // unique for padding lanes
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    const unsigned rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) wcnt[warp][d] = __popc(peers);
    __syncthreads();
    // counts of each digit in the earlier warps of the block (thread t: digit t)
    if (threadIdx.x < 256) {
        unsigned run = 0;
        for (int w = 0; w < RADIX_BLOCK / 32; w++) {
            const unsigned c = wcnt[w][threadIdx.x];
            wcnt[w][threadIdx.x] = run;
            run += c;
        }
    }
    __syncthreads();
    if (valid) keys_out[hist[d * nblk + blockIdx.x] + wcnt[warp][d] + rank] = key;
}

#define ENC_CHUNK 32
// dwte[id, :] += sum of dout rows with that id, in position order.  Pass 1: each chunk
// of ENC_CHUNK sorted positions walks its runs of equal id; a run whose id occurs
// only inside this chunk is added straight into dwte (no other chunk touches that
// row), a run of an id that spans chunks leaves its partial sum at the run's first
// sorted index.  A thread owns one 16-byte packet of columns and has eight rows in
// flight.  C must be a multiple of the packet.
template <typename T>
__global__ void encoder_backward_wte_partial(float* __restrict__ dwte, float* __restrict__ partial,
                                             const unsigned* __restrict__ sorted,
                                             const T* __restrict__ dout, int BT, int C, int V) {
    pdl_wait();
    constexpr int EPV = Vec<T>::N;
    constexpr int U = 8;
    __shared__ unsigned sk[ENC_CHUNK + 2];
    const int c0 = blockIdx.x * ENC_CHUNK;
    const int n = min(ENC_CHUNK, BT - c0);
    for (int i = threadIdx.x; i < n + 2; i += blockDim.x) {
        int gi = c0 - 1 + i;
        sk[i] = (gi >= 0 && gi < BT) ? sorted[gi] : 0xffffffffu;
    }
    __syncthreads();
    const unsigned ubt = (unsigned)BT;
    const int nvec = C / EPV;
    for (int cv = threadIdx.x; cv < nvec; cv += blockDim.x) {
        float acc[EPV];
#pragma unroll
        for (int e = 0; e < EPV; e++) acc[e] = 0.f;
        int run_start = 0;
        for (int i0 = 0; i0 < n; i0 += U) {
            Vec<T> a[U];
#pragma unroll
            for (int k = 0; k < U; k++)
                if (i0 + k < n) a[k] = load_vec(dout + (size_t)(sk[i0 + k + 1] % ubt) * C + cv * EPV);
#pragma unroll
            for (int k = 0; k < U; k++) {
                const int i = i0 + k;
                if (i >= n) break;
                const unsigned id = sk[i + 1] / ubt;
#pragma unroll
                for (int e = 0; e < EPV; e++) acc[e] += a[k].get(e);
                const unsigned nxt = sk[i + 2];
                const bool last = (i == n - 1) || (nxt / ubt != id);
                if (last) {
                    const bool from_prev = (run_start == 0) && (c0 > 0) && (sk[0] / ubt == id);
                    const bool into_next = (i == n - 1) && (c0 + n < BT) && (nxt / ubt == id);
                    if ((int)id < V) {
                        float* dst = (!from_prev && !into_next) ? dwte + (size_t)id * C + cv * EPV
                                                                 : partial + (size_t)(c0 + run_start) * C + cv * EPV;
                        const bool add = !from_prev && !into_next;
#pragma unroll
                        for (int q = 0; q < EPV / 4; q++) {
                            float4* d4 = reinterpret_cast<float4*>(dst) + q;
                            float4 o = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
                            if (add) { const float4 c = *d4; o.x += c.x; o.y += c.y; o.z += c.z; o.w += c.w; }
                            *d4 = o;
                        }
                    }
#pragma unroll
                    for (int e = 0; e < EPV; e++) acc[e] = 0.f;
                    run_start = i + 1;
                }
            }
        }
    }
}

// Pass 2: a run that spans chunks is the last run of the chunk it starts in; that
// chunk's block adds the run's partials (at the run start and at every later chunk
// start inside the run) in order.
__global__ void encoder_backward_wte_final(float* __restrict__ dwte, const float* __restrict__ partial,
                                           const unsigned* __restrict__ sorted, int BT, int C, int V) {
    pdl_wait();
    const int c0 = blockIdx.x * ENC_CHUNK;
    const int last = min(BT, c0 + ENC_CHUNK) - 1;
    if (last + 1 >= BT) return;                            // no later chunk
    const unsigned ubt = (unsigned)BT;
    const unsigned id = sorted[last] / ubt;
    if ((int)id >= V) return;
    if (sorted[last + 1] / ubt != id) return;              // the chunk's last run ends inside it
    // first index of the run: first key >= id * BT
    const unsigned lo_key = id * ubt;
    int lo = 0, hi = last;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (sorted[mid] < lo_key) lo = mid + 1; else hi = mid;
    }
    const int i = lo;
    if (i < c0) return;                                     // started in an earlier chunk
    // end of the run: first index whose key reaches (id+1)*BT
    const unsigned lim = (id + 1) * ubt;
    lo = last + 1; hi = BT;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (sorted[mid] < lim) lo = mid + 1; else hi = mid;
    }
    const int e = lo;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        float s = partial[(size_t)i * C + c];
        int b = c0 + ENC_CHUNK;
        // eight partials in flight, added in chunk order
        for (; b + 7 * ENC_CHUNK < e; b += 8 * ENC_CHUNK) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; k++) v[k] = partial[(size_t)(b + k * ENC_CHUNK) * C + c];
#pragma unroll
            for (int k = 0; k < 8; k++) s += v[k];
        }
        for (; b < e; b += ENC_CHUNK) s += partial[(size_t)b * C + c];
        dwte[(size_t)id * C + c] += s;
    }
}

// dwpe[t, :] += sum over b of dout[b, t, :], b in order.
// One thread per 16-byte packet of a row (C a multiple of the packet): the B loads of a
// packet are issued four at a time, then added in b order.
template <typename T>
__global__ void encoder_backward_wpe(float* __restrict__ dwpe, const T* __restrict__ dout,
                                     int B, int Tn, int C, int assign) {
    pdl_wait();
    constexpr int EPV = Vec<T>::N;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;     // packet index over (t, c)
    if (idx >= (size_t)Tn * C / EPV) return;
    const size_t off = idx * EPV;                                         // = t * C + c
    float s[EPV];
#pragma unroll
    for (int e = 0; e < EPV; e++) s[e] = 0.f;
    const size_t bstride = (size_t)Tn * C;
    int b = 0;
    for (; b + 3 < B; b += 4) {
        Vec<T> a[4];
#pragma unroll
        for (int k = 0; k < 4; k++) a[k] = load_vec(dout + (size_t)(b + k) * bstride + off);
#pragma unroll
        for (int k = 0; k < 4; k++)
#pragma unroll
            for (int e = 0; e < EPV; e++) s[e] += a[k].get(e);
    }
    for (; b < B; b++) {
        Vec<T> a = load_vec(dout + (size_t)b * bstride + off);
#pragma unroll
        for (int e = 0; e < EPV; e++) s[e] += a.get(e);
    }
#pragma unroll
    for (int q = 0; q < EPV / 4; q++) {
        float4* d = reinterpret_cast<float4*>(dwpe + off) + q;
        float4 v = assign ? make_float4(0.f, 0.f, 0.f, 0.f) : *d;
        v.x += s[4 * q]; v.y += s[4 * q + 1]; v.z += s[4 * q + 2]; v.w += s[4 * q + 3];
        *d = v;
    }
}

// ============================================================== e4m3 quantization
// Power-of-two scales (so scaling and unscaling are exact): the largest k with
// amax * 2^k <= 448, the largest e4m3 value.  With amax = f 2^e, f in [0.5, 1):
// k = 9 - e if f <= 0.875 (448 = 0.875 2^9), else 8 - e; 0 for amax == 0; clamped to
// [-126, 126] so that 2^k and 2^-k are normal floats.
__device__ __forceinline__ int e4m3_scale_exp(float amax) {
    if (!(amax > 0.f)) return 0;
    int e;
    const float f = frexpf(amax, &e);
    const int k = (f <= 0.875f) ? 9 - e : 8 - e;
    return max(-126, min(126, k));
}
__device__ __forceinline__ float pow2f(int k) { return __int_as_float((127 + k) << 23); }
// two values to e4m3 (round to nearest even, saturating at +-448): lo in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// ============================================================== layernorm
#define LN_EPS 1e-5f
#define LN_WARPS 8
// One warp per row; the row lives in registers (NV 16-byte packets per lane).
// mean = sum(x)/C; var = sum((x-mean)^2)/C (two passes over registers); rstd =
// 1/sqrt(var + eps); out = (x-mean)*rstd*w + b.
// Q8: also the row as e4m3 codes q (C bytes) of out * 2^k, k the power-of-two scale of
// the row's largest |out| (taken before out is rounded to T), and qdeq[row] = 2^-k.
template <typename T, int NV, bool Q8 = false>
__global__ void __launch_bounds__(LN_WARPS * 32)
layernorm_forward_kernel(T* __restrict__ out, float* __restrict__ mean, float* __restrict__ rstd,
                         const T* __restrict__ inp, const T* __restrict__ w,
                         const T* __restrict__ b, int N, int C, uint8_t* __restrict__ q,
                         float* __restrict__ qdeq) {
    pdl_wait();
    constexpr int EPV = Vec<T>::N;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * LN_WARPS + (threadIdx.x >> 5);
    if (row >= N) return;
    const int nvec = C / EPV;
    const T* x = inp + (size_t)row * C;
    float v[NV][EPV];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) {
        int vi = lane + 32 * i;
        if (vi < nvec) {
            Vec<T> p = load_vec(x + vi * EPV);
#pragma unroll
            for (int e = 0; e < EPV; e++) { v[i][e] = p.get(e); s += v[i][e]; }
        } else {
#pragma unroll
            for (int e = 0; e < EPV; e++) v[i][e] = 0.f;
        }
    }
    const float m = warp_sum(s) / (float)C;
    float qs = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) {
        if (lane + 32 * i < nvec) {
#pragma unroll
            for (int e = 0; e < EPV; e++) { float d = v[i][e] - m; qs += d * d; }
        }
    }
    const float var = warp_sum(qs) / (float)C;
    const float r = 1.0f / sqrtf(var + LN_EPS);
    T* o = out + (size_t)row * C;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) {
        int vi = lane + 32 * i;
        if (vi < nvec) {
            Vec<T> wv = load_vec(w + vi * EPV), bv = load_vec(b + vi * EPV), ov;
#pragma unroll
            for (int e = 0; e < EPV; e++) {
                v[i][e] = (v[i][e] - m) * r * wv.get(e) + bv.get(e);
                ov.set(e, v[i][e]);
                if (Q8) amax = fmaxf(amax, fabsf(v[i][e]));
            }
            store_vec(o + vi * EPV, ov);
        }
    }
    if constexpr (Q8) {
        const int k = e4m3_scale_exp(warp_max(amax));
        const float sc = pow2f(k);
        uint8_t* qr = q + (size_t)row * C;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            int vi = lane + 32 * i;
            if (vi < nvec) {
                uint32_t c[EPV / 4];
#pragma unroll
                for (int e = 0; e < EPV; e += 4)
                    c[e / 4] = e4m3x2(v[i][e] * sc, v[i][e + 1] * sc) |
                               (e4m3x2(v[i][e + 2] * sc, v[i][e + 3] * sc) << 16);
                if constexpr (EPV == 8) *reinterpret_cast<uint2*>(qr + vi * EPV) = make_uint2(c[0], c[1]);
                else *reinterpret_cast<uint32_t*>(qr + vi * EPV) = c[0];
            }
        }
        if (lane == 0) qdeq[row] = pow2f(-k);
    }
    if (lane == 0) { mean[row] = m; rstd[row] = r; }
}

// Per-tensor e4m3 quantization of fp32 weights: tensor t (blockIdx.y) is
// [t * len, (t + 1) * len) of w.  First the largest |w| of each tensor (each block's
// maximum folded in with an integer atomicMax on the float's bits: order-free, so
// deterministic; amax_bits zeroed beforehand), then codes of w * 2^k and deq[t] = 2^-k.
__global__ void absmax_tensors_kernel(unsigned* __restrict__ amax_bits, const float* __restrict__ w, size_t len) {
    pdl_wait();
    const float4* p = reinterpret_cast<const float4*>(w + (size_t)blockIdx.y * len);
    const size_t n4 = len / 4;
    float mx = 0.f;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 a = p[i];
        mx = fmaxf(mx, fmax3(fabsf(a.x), fabsf(a.y), fmaxf(fabsf(a.z), fabsf(a.w))));
    }
    mx = warp_max(mx);
    __shared__ float wm[32];
    if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < blockDim.x / 32 ? wm[threadIdx.x] : 0.f;
        v = warp_max(v);
        if (threadIdx.x == 0) atomicMax(amax_bits + blockIdx.y, __float_as_uint(v));
    }
}
__global__ void quantize_tensors_kernel(uint8_t* __restrict__ q, float* __restrict__ deq,
                                        const unsigned* __restrict__ amax_bits, const float* __restrict__ w,
                                        size_t len) {
    pdl_wait();
    const int k = e4m3_scale_exp(__uint_as_float(amax_bits[blockIdx.y]));
    const float sc = pow2f(k);
    const float4* p = reinterpret_cast<const float4*>(w + (size_t)blockIdx.y * len);
    uint32_t* qo = reinterpret_cast<uint32_t*>(q + (size_t)blockIdx.y * len);
    const size_t n4 = len / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 a = p[i];
        qo[i] = e4m3x2(a.x * sc, a.y * sc) | (e4m3x2(a.z * sc, a.w * sc) << 16);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) deq[blockIdx.y] = pow2f(-k);
}

// Backward.  With xhat = (x-mean)*rstd, g = dy*w:
//   dinp += rstd * (g - mean(g) - xhat * mean(g*xhat))
//   dw partial += dy*xhat, db partial += dy, per block over a fixed set of rows
// Block j handles rows j*LN_WARPS + warp + k*gridDim.x*LN_WARPS; warps then combine in
// warp order through shared memory and the block writes partial[j][0:2C].  The row's
// x and dy stay packed (16-byte packets) in registers and xhat is recomputed in the
// second pass, which keeps two blocks resident per SM.
// With SUM the block also sums the updated dinp rows (partial[j][2C:3C]): in the model
// that is the bias gradient of the linear layer whose output is the residual stream.
// Each warp keeps that sum in its own shared-memory row (its lanes own distinct
// columns), which leaves the register budget of two blocks per SM untouched.
// Per-warp running column sums of the layernorm backward, laid out as EPV/4 planes of
// float4 (plane p holds elements 4p..4p+3 of every vector), so that the 32 lanes of a warp
// touch 32 consecutive 16-byte words: no shared-memory bank conflicts.
template <int EPV>
__device__ __forceinline__ void wsum_zero(float* ws, int nvec, int vi) {
#pragma unroll
    for (int p = 0; p < EPV / 4; p++)
        *reinterpret_cast<float4*>(ws + (size_t)p * nvec * 4 + vi * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
}
template <int EPV, typename V>
__device__ __forceinline__ void wsum_add(float* ws, int nvec, int vi, const V& v) {
#pragma unroll
    for (int p = 0; p < EPV / 4; p++) {
        float4* q = reinterpret_cast<float4*>(ws + (size_t)p * nvec * 4 + vi * 4);
        float4 a = *q;
        a.x += v.get(4 * p); a.y += v.get(4 * p + 1); a.z += v.get(4 * p + 2); a.w += v.get(4 * p + 3);
        *q = a;
    }
}
__device__ __forceinline__ float wsum_get(const float* ws, int nvec, int vi, int e) {
    return ws[(size_t)(e >> 2) * nvec * 4 + vi * 4 + (e & 3)];
}

// The block's column sums: every warp's dw, db (and column sums of the new dinp) are
// added into `red`, warps in order, in the float4 plane layout of the per-warp sums (32
// consecutive 16-byte words per warp access: no bank conflicts); the block's partial
// row is then written in column order.
template <int EPV, int NV, bool SUM>
__device__ __forceinline__ void ln_combine(float* red, const float* wsum, const float (&dwa)[NV][EPV],
                                           const float (&dba)[NV][EPV], int warp, int lane, int nvec, int C,
                                           float* __restrict__ pj) {
    constexpr int W = SUM ? 3 : 2;
    for (int wi = 0; wi < LN_WARPS; wi++) {
        if (warp == wi) {
#pragma unroll
            for (int i = 0; i < NV; i++) {
                const int vi = lane + 32 * i;
                if (vi < nvec) {
#pragma unroll
                    for (int p = 0; p < EPV / 4; p++) {
                        const int o = p * nvec * 4 + vi * 4;
                        const float4 a = make_float4(dwa[i][4 * p], dwa[i][4 * p + 1], dwa[i][4 * p + 2], dwa[i][4 * p + 3]);
                        const float4 b = make_float4(dba[i][4 * p], dba[i][4 * p + 1], dba[i][4 * p + 2], dba[i][4 * p + 3]);
                        float4* r0 = reinterpret_cast<float4*>(red + o);
                        float4* r1 = reinterpret_cast<float4*>(red + C + o);
                        if (wi == 0) {
                            *r0 = a;
                            *r1 = b;
                            if (SUM) *reinterpret_cast<float4*>(red + 2 * C + o) = *reinterpret_cast<const float4*>(wsum + o);
                        } else {
                            float4 x = *r0, y = *r1;
                            x.x += a.x; x.y += a.y; x.z += a.z; x.w += a.w;
                            y.x += b.x; y.y += b.y; y.z += b.z; y.w += b.w;
                            *r0 = x;
                            *r1 = y;
                            if (SUM) {
                                float4* r2 = reinterpret_cast<float4*>(red + 2 * C + o);
                                const float4 z = *reinterpret_cast<const float4*>(wsum + o);
                                float4 t = *r2;
                                t.x += z.x; t.y += z.y; t.z += z.z; t.w += z.w;
                                *r2 = t;
                            }
                        }
                    }
                }
            }
        }
        __syncthreads();
    }
    for (int c = threadIdx.x; c < W * C; c += blockDim.x) {
        const int arr = c / C, cc = c - arr * C, vi = cc / EPV, e = cc - vi * EPV;
        pj[c] = red[arr * C + (e >> 2) * nvec * 4 + vi * 4 + (e & 3)];
    }
}


template <typename T, int NV, bool SUM>
__global__ void __launch_bounds__(LN_WARPS * 32, (NV * Vec<T>::N <= 24) ? 2 : 1)
layernorm_backward_kernel(T* __restrict__ dinp, float* __restrict__ partial,
                          const T* __restrict__ dout, const T* __restrict__ inp,
                          const T* __restrict__ w, const float* __restrict__ mean,
                          const float* __restrict__ rstd, int N, int C) {
    pdl_wait();
    constexpr int EPV = Vec<T>::N;
    extern __shared__ float red[];   // 2C floats (SUM: 3C, then LN_WARPS rows of C)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nvec = C / EPV;
    constexpr int W = SUM ? 3 : 2;
    float* wsum = red + 3 * C + warp * C;           // this warp's running column sums (SUM)
    Vec<T> wv[NV];
    float dwa[NV][EPV], dba[NV][EPV];
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int vi = lane + 32 * i;
        if (vi < nvec) wv[i] = load_vec(w + vi * EPV);
#pragma unroll
        for (int e = 0; e < EPV; e++) { dwa[i][e] = 0.f; dba[i][e] = 0.f; }
        if (SUM && vi < nvec) wsum_zero<EPV>(wsum, nvec, vi);
    }
    for (int row = blockIdx.x * LN_WARPS + warp; row < N; row += gridDim.x * LN_WARPS) {
        const T* x = inp + (size_t)row * C;
        const T* dy = dout + (size_t)row * C;
        T* dx = dinp + (size_t)row * C;
        const float m = mean[row], r = rstd[row];
        Vec<T> xp[NV], dp[NV], cur[NV];
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int vi = lane + 32 * i;
            if (vi < nvec) {
                xp[i] = load_vec(x + vi * EPV);
                dp[i] = load_vec(dy + vi * EPV);
                cur[i] = load_vec(dx + vi * EPV);
            }
        }
        float sg = 0.f, sgx = 0.f;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            if (lane + 32 * i < nvec) {
#pragma unroll
                for (int e = 0; e < EPV; e++) {
                    const float xh = (xp[i].get(e) - m) * r;
                    const float d = dp[i].get(e);
                    const float g = d * wv[i].get(e);
                    sg += g;
                    sgx += g * xh;
                    dwa[i][e] += d * xh;
                    dba[i][e] += d;
                }
            }
        }
        const float mg = warp_sum(sg) / (float)C;
        const float mgx = warp_sum(sgx) / (float)C;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int vi = lane + 32 * i;
            if (vi < nvec) {
                Vec<T> nv;
#pragma unroll
                for (int e = 0; e < EPV; e++) {
                    const float xh = (xp[i].get(e) - m) * r;
                    const float g = dp[i].get(e) * wv[i].get(e);
                    nv.set(e, cur[i].get(e) + r * (g - mg - xh * mgx));
                }
                store_vec(dx + vi * EPV, nv);
                if (SUM) wsum_add<EPV>(wsum, nvec, vi, nv);          // the stored (rounded) value
            }
        }
    }
    // combine the warps in order 0..LN_WARPS-1
    ln_combine<EPV, NV, SUM>(red, wsum, dwa, dba, warp, lane, nvec, C, partial + (size_t)blockIdx.x * W * C);
}

// Same computation, with each warp's rows streamed through shared memory: lane 0 of the
// warp fetches row k+1's x, dy and dinp with 1-D bulk copies (two stages, one mbarrier
// each) while the warp works on row k from shared memory, so loads stay in flight the
// whole time and the row no longer occupies registers.  Shared memory: partial sums
// (W*C floats), the SUM rows (LN_WARPS*C floats), then LN_WARPS x 2 stages x 3 rows of C
// elements, then 2*LN_WARPS mbarriers.  Bounded waits: on a timeout the warp stops,
// sets the error bit, and lets its copies land before the block finishes.
template <typename T, int NV, bool SUM>
__global__ void __launch_bounds__(LN_WARPS * 32, (NV * Vec<T>::N <= 24) ? 2 : 1)
layernorm_backward_pipe_kernel(T* __restrict__ dinp, float* __restrict__ partial,
                               const T* __restrict__ dout, const T* __restrict__ inp,
                               const T* __restrict__ w, const float* __restrict__ mean,
                               const float* __restrict__ rstd, int N, int C, unsigned* err) {
    pdl_wait();
    constexpr int EPV = Vec<T>::N;
    constexpr int W = SUM ? 3 : 2;
    extern __shared__ __align__(16) float red[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nvec = C / EPV;
    const size_t row_bytes = (size_t)C * sizeof(T);
    float* wsum = red + W * C + warp * C;
    T* stage_base = reinterpret_cast<T*>(red + W * C + (SUM ? LN_WARPS * C : 0));
    T* st = stage_base + (size_t)warp * 2 * 3 * C;          // this warp's two stages
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage_base + (size_t)LN_WARPS * 2 * 3 * C) + 2 * warp;
    if (lane == 0) { mbar_init(&bars[0], 1); mbar_init(&bars[1], 1); }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();
    float wf[NV][EPV];                                  // the weight, converted once
    float dwa[NV][EPV], dba[NV][EPV];
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int vi = lane + 32 * i;
        Vec<T> wv;
        if (vi < nvec) wv = load_vec(w + vi * EPV);
#pragma unroll
        for (int e = 0; e < EPV; e++) { wf[i][e] = vi < nvec ? wv.get(e) : 0.f; dwa[i][e] = 0.f; dba[i][e] = 0.f; }
        if (SUM && vi < nvec) wsum_zero<EPV>(wsum, nvec, vi);
    }
    const int step = gridDim.x * LN_WARPS;
    const int row0 = blockIdx.x * LN_WARPS + warp;
    const int nrows = row0 < N ? (N - row0 + step - 1) / step : 0;
    auto fetch = [&](int k) {
        const int row = row0 + k * step;
        T* d = st + (size_t)(k & 1) * 3 * C;
        fence_async_smem();
        mbar_expect_tx(&bars[k & 1], (uint32_t)(3 * row_bytes));
        bulk_load(d, inp + (size_t)row * C, (uint32_t)row_bytes, &bars[k & 1]);
        bulk_load(d + C, dout + (size_t)row * C, (uint32_t)row_bytes, &bars[k & 1]);
        bulk_load(d + 2 * C, dinp + (size_t)row * C, (uint32_t)row_bytes, &bars[k & 1]);
    };
    if (lane == 0 && nrows > 0) fetch(0);
    // the statistics of this warp's rows, fetched together up front: lane k holds row k's
    // (rows past the 32nd load their own when reached)
    float mk = 0.f, rk = 0.f;
    if (lane < nrows) { mk = mean[row0 + lane * step]; rk = rstd[row0 + lane * step]; }
    int issued = nrows > 0 ? 1 : 0, waited = 0;
    for (int k = 0; k < nrows; k++) {
        const int row = row0 + k * step;
        float m = __shfl_sync(0xffffffffu, mk, k & 31), r = __shfl_sync(0xffffffffu, rk, k & 31);
        if (k >= 32) { m = mean[row]; r = rstd[row]; }
        __syncwarp();                                  // every lane is done with row k-1's stage
        if (lane == 0 && k + 1 < nrows) { fetch(k + 1); issued++; }
        // wait for row k (bounded)
        bool ok = mbar_try_wait(&bars[k & 1], (k >> 1) & 1);
        if (!ok) {
            const long long t0 = clock64();
            while (!(ok = mbar_try_wait(&bars[k & 1], (k >> 1) & 1)))
                if (clock64() - t0 > TC_WAIT_LIMIT) break;
        }
        if (!__all_sync(0xffffffffu, ok)) { if (lane == 0) raise_error(err, ERRBIT_TIMEOUT); break; }
        waited++;
        const T* xs = st + (size_t)(k & 1) * 3 * C;
        const T* dys = xs + C;
        const T* cs = xs + 2 * C;
        float sg = 0.f, sgx = 0.f;
        const float2 m2 = make_float2(-m, -m), r2 = make_float2(r, r);
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int vi = lane + 32 * i;
            if (vi < nvec) {
                Vec<T> xp = load_vec(xs + vi * EPV), dp = load_vec(dys + vi * EPV);
                // element pairs in packed f32x2 arithmetic; the row sums keep their order
#pragma unroll
                for (int e = 0; e < EPV; e += 2) {
                    const float2 xh = __fmul2_rn(__fadd2_rn(xp.get2(e), m2), r2);
                    const float2 d = dp.get2(e);
                    const float2 g = __fmul2_rn(d, make_float2(wf[i][e], wf[i][e + 1]));
                    sg += g.x;
                    sg += g.y;
                    sgx = fmaf(g.x, xh.x, sgx);
                    sgx = fmaf(g.y, xh.y, sgx);
                    const float2 dw = __ffma2_rn(d, xh, make_float2(dwa[i][e], dwa[i][e + 1]));
                    const float2 db = __fadd2_rn(make_float2(dba[i][e], dba[i][e + 1]), d);
                    dwa[i][e] = dw.x; dwa[i][e + 1] = dw.y;
                    dba[i][e] = db.x; dba[i][e + 1] = db.y;
                }
            }
        }
        const float mg = warp_sum(sg) / (float)C;
        const float mgx = warp_sum(sgx) / (float)C;
        T* dx = dinp + (size_t)row * C;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int vi = lane + 32 * i;
            if (vi < nvec) {
                Vec<T> xp = load_vec(xs + vi * EPV), dp = load_vec(dys + vi * EPV), cur = load_vec(cs + vi * EPV), nv;
#pragma unroll
                for (int e = 0; e < EPV; e += 2) {
                    const float2 xh = __fmul2_rn(__fadd2_rn(xp.get2(e), m2), r2);
                    const float2 g = __fmul2_rn(dp.get2(e), make_float2(wf[i][e], wf[i][e + 1]));
                    // cur + r (g - mg - xh mgx)
                    const float2 t = __ffma2_rn(make_float2(-xh.x, -xh.y), make_float2(mgx, mgx), __fadd2_rn(g, make_float2(-mg, -mg)));
                    const float2 o = __ffma2_rn(r2, t, cur.get2(e));
                    nv.set2(e, o.x, o.y);
                }
                store_vec(dx + vi * EPV, nv);
                if (SUM) wsum_add<EPV>(wsum, nvec, vi, nv);
            }
        }
    }
    // copies issued but not waited for (only after a timeout) land before the block ends
    if (lane == 0) {
        for (int k = waited; k < issued; k++) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&bars[k & 1], (k >> 1) & 1))
                if (clock64() - t0 > TC_WAIT_LIMIT) break;
        }
    }
    __syncwarp();
    ln_combine<EPV, NV, SUM>(red, wsum, dwa, dba, warp, lane, nvec, C, partial + (size_t)blockIdx.x * W * C);
}

// Column sums of a (G x W) fp32 partial matrix, in a fixed order: a 256-thread block
// takes 32 columns; thread (c, g) sums rows g, g+8, g+16, ... of column c, then the
// eight group sums are added in group order.  Column w < split goes to out0[w], the
// rest to out1[w - split], or with out2, columns [2*split, 3*split) to out2 (all
// accumulate).
#define CR_COLS 32
#define CR_GROUPS 8
__global__ void __launch_bounds__(CR_COLS * CR_GROUPS)
column_reduce_kernel(float* __restrict__ out0, float* __restrict__ out1, int split,
                     const float* __restrict__ partial, int G, int W, float* __restrict__ out2 = nullptr) {
    pdl_wait();
    __shared__ float sm[CR_GROUPS][CR_COLS];
    const int c = threadIdx.x % CR_COLS, g = threadIdx.x / CR_COLS;
    const int w = blockIdx.x * CR_COLS + c;
    float s0 = 0.f, s1 = 0.f;
    if (w < W) {
        int j = g;
        for (; j + CR_GROUPS < G; j += 2 * CR_GROUPS) {
            s0 += partial[(size_t)j * W + w];
            s1 += partial[(size_t)(j + CR_GROUPS) * W + w];
        }
        if (j < G) s0 += partial[(size_t)j * W + w];
    }
    sm[g][c] = s0 + s1;
    __syncthreads();
    if (g == 0 && w < W) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < CR_GROUPS; k++) s += sm[k][c];
        if (w < split) out0[w] += s;
        else if (!out2 || w < 2 * split) out1[w - split] += s;
        else out2[w - 2 * split] += s;
    }
}

// The same sums for W a multiple of 4 (16-byte aligned rows): a 256-thread block takes
// 32 columns as 8 float4 packets; thread (p, g) adds rows g, g+32, g+64, ... of packet p
// (four loads in flight), then the 32 group sums of each column are added in group order.
__device__ __forceinline__ void column_reduce4_block(float* __restrict__ out0, float* __restrict__ out1, int split,
                                                     const float* __restrict__ partial, int G, int W,
                                                     float* __restrict__ out2, int bx, bool assign = false) {
    __shared__ float sm[32][33];
    const int p = threadIdx.x & 7, g = threadIdx.x >> 3;
    const int w = bx * 32 + p * 4;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (w < W) {
        const float* col = partial + w;
        int j = g;
        for (; j + 96 < G; j += 128) {
            float4 a[4];
#pragma unroll
            for (int k = 0; k < 4; k++) a[k] = *reinterpret_cast<const float4*>(col + (size_t)(j + 32 * k) * W);
#pragma unroll
            for (int k = 0; k < 4; k++) { s.x += a[k].x; s.y += a[k].y; s.z += a[k].z; s.w += a[k].w; }
        }
        for (; j < G; j += 32) {
            const float4 a = *reinterpret_cast<const float4*>(col + (size_t)j * W);
            s.x += a.x; s.y += a.y; s.z += a.z; s.w += a.w;
        }
    }
    sm[g][p * 4 + 0] = s.x; sm[g][p * 4 + 1] = s.y; sm[g][p * 4 + 2] = s.z; sm[g][p * 4 + 3] = s.w;
    __syncthreads();
    const int t = threadIdx.x, wc = bx * 32 + t;
    if (t < 32 && wc < W) {
        float acc = 0.f;
#pragma unroll 8
        for (int k = 0; k < 32; k++) acc += sm[k][t];
        // assign: the output's first write of the step (the same value as 0 + acc)
        float* o = wc < split ? out0 + wc : (!out2 || wc < 2 * split) ? out1 + (wc - split) : out2 + (wc - 2 * split);
        *o = assign ? acc : *o + acc;
    }
}
__global__ void __launch_bounds__(256)
column_reduce4_kernel(float* __restrict__ out0, float* __restrict__ out1, int split,
                      const float* __restrict__ partial, int G, int W, float* __restrict__ out2 = nullptr) {
    pdl_wait();
    column_reduce4_block(out0, out1, split, partial, G, W, out2, blockIdx.x);
}

// The same reduction for many (G x W) partial matrices in one launch: blockIdx.y picks
// the segment (the step's layernorm and bias-gradient reductions, all deferred to the
// end of the backward pass, since only the optimiser reads those gradients).
struct RedSeg {
    const float* partial;
    float *out0, *out1, *out2;
    int split, G, W, assign;   // assign: store the sums instead of adding them
};
#define RED_MAX_SEGS 128
struct RedBatch {
    RedSeg seg[RED_MAX_SEGS];
};
__global__ void __launch_bounds__(256) column_reduce_batch_kernel(const __grid_constant__ RedBatch b) {
    pdl_wait();
    const RedSeg& sg = b.seg[blockIdx.y];
    if ((int)blockIdx.x * 32 >= sg.W) return;
    column_reduce4_block(sg.out0, sg.out1, sg.split, sg.partial, sg.G, sg.W, sg.out2, blockIdx.x, sg.assign != 0);
}

// ============================================================== column sums (bias grads)
// partial[r][n] = sum of x[m][n] over the rows m of chunk r.  A 256-thread block takes
// 32 16-byte packets of columns of one chunk; warp w adds rows w, w+8, w+16, ... (four
// loads in flight per lane), then the eight warp sums are added in warp order.
#define CS_WARPS 8
template <typename T>
__global__ void __launch_bounds__(CS_WARPS * 32)
colsum_partial_kernel(float* __restrict__ partial, const T* __restrict__ x, int M, int N, int rows_per_chunk) {
    pdl_wait();
    constexpr int EPV = Vec<T>::N;
    constexpr int U = 4;
    __shared__ float sm[CS_WARPS][EPV * 32];          // [warp][element][lane]: conflict-free
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cv = blockIdx.x * 32 + lane;
    const int r = blockIdx.y;
    const int m0 = r * rows_per_chunk, m1 = min(M, m0 + rows_per_chunk);
    float s[EPV];
#pragma unroll
    for (int e = 0; e < EPV; e++) s[e] = 0.f;
    if (cv * EPV < N) {
        const T* xc = x + cv * EPV;
        int m = m0 + warp;
        for (; m + (U - 1) * CS_WARPS < m1; m += U * CS_WARPS) {
            Vec<T> a[U];
#pragma unroll
            for (int k = 0; k < U; k++) a[k] = load_vec(xc + (size_t)(m + k * CS_WARPS) * N);
#pragma unroll
            for (int k = 0; k < U; k++)
#pragma unroll
                for (int e = 0; e < EPV; e++) s[e] += a[k].get(e);
        }
        for (; m < m1; m += CS_WARPS) {
            Vec<T> a = load_vec(xc + (size_t)m * N);
#pragma unroll
            for (int e = 0; e < EPV; e++) s[e] += a.get(e);
        }
    }
#pragma unroll
    for (int e = 0; e < EPV; e++) sm[warp][e * 32 + lane] = s[e];
    __syncthreads();
    for (int t = threadIdx.x; t < 32 * EPV; t += blockDim.x) {
        const int l = t / EPV, e = t % EPV;
        const int n = (blockIdx.x * 32 + l) * EPV + e;
        if (n < N) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < CS_WARPS; w++) acc += sm[w][e * 32 + l];
            partial[(size_t)r * N + n] = acc;
        }
    }
}
// one column per thread, for widths that are not a multiple of the packet
template <typename T>
__global__ void colsum_partial_scalar_kernel(float* __restrict__ partial, const T* __restrict__ x,
                                             int M, int N, int rows_per_chunk) {
    pdl_wait();
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    const int r = blockIdx.y;
    if (n >= N) return;
    const int m0 = r * rows_per_chunk, m1 = min(M, m0 + rows_per_chunk);
    float s = 0.f;
    for (int m = m0; m < m1; m++) s += to_f32(x[(size_t)m * N + n]);
    partial[(size_t)r * N + n] = s;
}

// ============================================================== softmax + cross-entropy
// One 256-thread block per row of logits (Vp entries); eight rows in flight per SM.
// Pass 1: online max / sum of exp over the V real columns, four 16-byte packets per
// step (one rescale per step); lse = max + log(sum); loss = lse - z[target].  Pass 2
// (the row is still in L2) overwrites it with d(mean loss)/dz = (exp(z - lse) -
// [j == target]) * dloss for j < V and 0 for the padded columns.  exp(a) is computed as
// exp2(a * log2 e).
#define XENT_THREADS 256
#define XENT_U 4
#define XENT_LOG2E 1.4426950408889634f
// 2^x by the hardware approximation (relative error ~2^-22); 2^-inf = 0
__device__ __forceinline__ float xent_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// (m, s) pairs in the log2 domain: the combined pair of two partial sums
__device__ __forceinline__ void xent_merge(float& m, float& s, float om, float os) {
    const float nm = fmaxf(m, om);
    const float a = (m == -INFINITY) ? 0.f : s * exp2f(m - nm);
    const float b = (om == -INFINITY) ? 0.f : os * exp2f(om - nm);
    m = nm;
    s = a + b;
}
template <typename T>
__global__ void __launch_bounds__(XENT_THREADS)
softmax_xent_kernel(T* __restrict__ logits, float* __restrict__ losses,
                    const int* __restrict__ targets, int V, int Vp, float dloss, unsigned* err) {
    pdl_wait();
    constexpr int EPV = Vec<T>::N;
    constexpr int NW = XENT_THREADS / 32;
    __shared__ float sm_m[NW], sm_s[NW];
    __shared__ float sm_lse;
    const int row = blockIdx.x;
    T* z = logits + (size_t)row * Vp;
    const int tgt_raw = targets[row];
    const bool tgt_ok = tgt_raw >= 0 && tgt_raw < V;
    const int tgt = tgt_ok ? tgt_raw : -1;
    const int nfull = V / EPV;              // packets whose columns are all real
    const int nvec = Vp / EPV;
    // pass 1, in the log2 domain: mx2 = max(z) log2e, sum = sum 2^(z log2e - mx2)
    float mx2 = -INFINITY, sum = 0.f;
    for (int v0 = threadIdx.x; v0 < nvec; v0 += XENT_U * XENT_THREADS) {
        Vec<T> p[XENT_U];
#pragma unroll
        for (int u = 0; u < XENT_U; u++) {
            const int vi = v0 + u * XENT_THREADS;
            if (vi < nvec) p[u] = load_vec(z + (size_t)vi * EPV);
        }
        float y[XENT_U][EPV];
        float vmax = -INFINITY;
#pragma unroll
        for (int u = 0; u < XENT_U; u++) {
            const int vi = v0 + u * XENT_THREADS;
            if (vi < nfull) {
                // all columns real: packed pairs, three-input maxima
#pragma unroll
                for (int e = 0; e < EPV; e += 2) {
                    const float2 f = __fmul2_rn(p[u].get2(e), make_float2(XENT_LOG2E, XENT_LOG2E));
                    y[u][e] = f.x;
                    y[u][e + 1] = f.y;
                    vmax = fmax3(vmax, f.x, f.y);
                }
            } else {
#pragma unroll
                for (int e = 0; e < EPV; e++) {
                    y[u][e] = (vi < nvec && vi * EPV + e < V) ? p[u].get(e) * XENT_LOG2E : -INFINITY;
                    vmax = fmaxf(vmax, y[u][e]);
                }
            }
        }
        if (vmax == -INFINITY) continue;
        const float nm = fmaxf(mx2, vmax);
        float acc = sum * xent_ex2(mx2 - nm);
#pragma unroll
        for (int u = 0; u < XENT_U; u++)
#pragma unroll
            for (int e = 0; e < EPV; e += 2) {
                const float2 a = __fadd2_rn(make_float2(y[u][e], y[u][e + 1]), make_float2(-nm, -nm));
                acc += xent_ex2(a.x);
                acc += xent_ex2(a.y);
            }
        mx2 = nm;
        sum = acc;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        xent_merge(mx2, sum, __shfl_xor_sync(0xffffffffu, mx2, o), __shfl_xor_sync(0xffffffffu, sum, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) { sm_m[warp] = mx2; sm_s[warp] = sum; }
    __syncthreads();
    if (warp == 0) {
        float M = lane < NW ? sm_m[lane] : -INFINITY, S = lane < NW ? sm_s[lane] : 0.f;
#pragma unroll
        for (int o = NW / 2; o > 0; o >>= 1)
            xent_merge(M, S, __shfl_xor_sync(0xffffffffu, M, o), __shfl_xor_sync(0xffffffffu, S, o));
        if (lane == 0) {
            const float lse2 = M + log2f(S);            // log2 of sum exp(z)
            sm_lse = lse2;
            if (!tgt_ok) raise_error(err, ERRBIT_TOKEN);
            losses[row] = tgt_ok ? (lse2 / XENT_LOG2E - to_f32(z[tgt])) : 0.f;
        }
    }
    __syncthreads();
    const float lse2 = sm_lse;
    for (int v0 = threadIdx.x; v0 < nvec; v0 += XENT_U * XENT_THREADS) {
        Vec<T> p[XENT_U];
#pragma unroll
        for (int u = 0; u < XENT_U; u++) {
            const int vi = v0 + u * XENT_THREADS;
            if (vi < nvec) p[u] = load_vec(z + (size_t)vi * EPV);
        }
#pragma unroll
        for (int u = 0; u < XENT_U; u++) {
            const int vi = v0 + u * XENT_THREADS;
            if (vi >= nvec) break;
            Vec<T> o;
            if (vi < nfull) {
                // all columns real: (2^(z log2e - lse2) - [j == target]) * dloss in packed
                // pairs, the target column (at most one packet of the row) redone apart
#pragma unroll
                for (int e = 0; e < EPV; e += 2) {
                    const float2 a = __ffma2_rn(p[u].get2(e), make_float2(XENT_LOG2E, XENT_LOG2E), make_float2(-lse2, -lse2));
                    const float2 d = __fmul2_rn(make_float2(xent_ex2(a.x), xent_ex2(a.y)), make_float2(dloss, dloss));
                    o.set2(e, d.x, d.y);
                }
                if ((unsigned)(tgt - vi * EPV) < (unsigned)EPV) {
#pragma unroll
                    for (int e = 0; e < EPV; e++)
                        if (vi * EPV + e == tgt) o.set(e, (xent_ex2(fmaf(p[u].get(e), XENT_LOG2E, -lse2)) - 1.f) * dloss);
                }
            } else {
#pragma unroll
                for (int e = 0; e < EPV; e++) {
                    const int j = vi * EPV + e;
                    float d = 0.f;
                    if (j < V) d = (xent_ex2(fmaf(p[u].get(e), XENT_LOG2E, -lse2)) - (j == tgt ? 1.f : 0.f)) * dloss;
                    o.set(e, d);
                }
            }
            store_vec(z + (size_t)vi * EPV, o);
        }
    }
}

// Mean of n per-position losses, fixed order: thread i sums i, i+1024, ...; then a tree.
__global__ void __launch_bounds__(1024)
mean_loss_kernel(float* __restrict__ loss, const float* __restrict__ losses, int n, unsigned* err) {
    pdl_wait();
    __shared__ float sm[32];
    float s = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s += losses[i];
    s = warp_sum(s);
    if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = (threadIdx.x < (blockDim.x >> 5)) ? sm[threadIdx.x] : 0.f;
        v = warp_sum(v);
        if (threadIdx.x == 0) {
            float mval = v / (float)n;
            if (!isfinite(mval)) raise_error(err, ERRBIT_NONFINITE);
            *loss = mval;
        }
    }
}

// ============================================================== next-token sampling
// SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
// OOPSLA 2014): output i of the generator started at `seed` mixes seed + i * gamma
// (gamma = the 64-bit golden-ratio constant) with two multiply-xorshift rounds.
__device__ __forceinline__ unsigned long long splitmix64_at(unsigned long long seed, unsigned long long i) {
    unsigned long long z = seed + i * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// One 1024-thread block per sequence b: e_j = exp((z_j - max) / temperature) over the V
// real columns of row (b, pos); thread t sums its contiguous chunk of e in order, the
// chunk sums are scanned in a fixed order (warp shuffles, then warp totals), u_b = the
// top 53 bits of SplitMix64 output b+1 scaled to [0, 1), and the token is the first
// index whose running sum exceeds u_b * total: the last chunk whose prefix is <= that
// threshold is scanned by its thread.
#define SAMPLE_THREADS 1024
template <typename T>
__global__ void __launch_bounds__(SAMPLE_THREADS)
sample_kernel(int* __restrict__ out, const T* __restrict__ logits, int Tn, int pos, int V, int Vp,
              float inv_temp, unsigned long long seed) {
    pdl_wait();
    __shared__ float s_red[32];
    __shared__ float s_pre[SAMPLE_THREADS];
    __shared__ int s_pick;
    const int b = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const T* z = logits + ((size_t)b * Tn + pos) * Vp;
    float mx = -INFINITY;
    for (int j = t; j < V; j += SAMPLE_THREADS) mx = fmaxf(mx, to_f32(z[j]));
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_red[warp] = mx;
    __syncthreads();
    mx = s_red[0];
    for (int w = 1; w < SAMPLE_THREADS / 32; w++) mx = fmaxf(mx, s_red[w]);
    __syncthreads();
    const int chunk = (V + SAMPLE_THREADS - 1) / SAMPLE_THREADS;
    const int j0 = min(V, t * chunk), j1 = min(V, j0 + chunk);
    float cs = 0.f;
    for (int j = j0; j < j1; j++) cs += expf((to_f32(z[j]) - mx) * inv_temp);
    // exclusive prefix of the chunk sums, in a fixed order
    float inc = cs;
    for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) s_red[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        float w = s_red[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += v;
        }
        s_red[lane] = w;                                   // inclusive warp totals
    }
    __syncthreads();
    const float pre = (warp > 0 ? s_red[warp - 1] : 0.f) + (inc - cs);
    const float total = s_red[SAMPLE_THREADS / 32 - 1];
    s_pre[t] = pre;
    if (t == 0) s_pick = 0;
    __syncthreads();
    const unsigned long long r = splitmix64_at(seed, (unsigned long long)b + 1ull);
    const float thr = (float)((double)(r >> 11) * (1.0 / 9007199254740992.0)) * total;
    // the last chunk (highest t with a non-empty chunk) whose prefix is <= thr
    if (j0 < j1 && pre <= thr) atomicMax(&s_pick, t);
    __syncthreads();
    if (t == s_pick) {
        int k = j1 - 1;
        float acc = pre;
        for (int j = j0; j < j1; j++) {
            const float e = expf((to_f32(z[j]) - mx) * inv_temp);
            acc += e;
            if (acc > thr && e > 0.f) { k = j; break; }
        }
        out[b] = k;
    }
}

// ============================================================== AdamW
// One pass over the flat buffer (n a multiple of 4).  bc1 = 1 - b1^t, bc2 = 1 - b2^t.
__global__ void adamw_kernel(float* __restrict__ p, const float* __restrict__ g,
                             float* __restrict__ m, float* __restrict__ v, bf16* __restrict__ shadow,
                             size_t n4, float lr, float b1, float b2, float eps, float wd,
                             float bc1, float bc2) {
    pdl_wait();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        float4 pp = reinterpret_cast<float4*>(p)[i];
        float4 gg = __ldcs(reinterpret_cast<const float4*>(g) + i);
        float4 mm = reinterpret_cast<float4*>(m)[i];
        float4 vv = reinterpret_cast<float4*>(v)[i];
        float* P = &pp.x; const float* G = &gg.x; float* Mm = &mm.x; float* Vv = &vv.x;
#pragma unroll
        for (int e = 0; e < 4; e++) {
            Mm[e] = b1 * Mm[e] + (1.f - b1) * G[e];
            Vv[e] = b2 * Vv[e] + (1.f - b2) * G[e] * G[e];
            float mhat = Mm[e] / bc1;
            float vhat = Vv[e] / bc2;
            P[e] -= lr * (mhat / (sqrtf(vhat) + eps) + wd * P[e]);
        }
        reinterpret_cast<float4*>(p)[i] = pp;
        reinterpret_cast<float4*>(m)[i] = mm;
        reinterpret_cast<float4*>(v)[i] = vv;
        if (shadow) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(pp.x, pp.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(pp.z, pp.w);
            uint2 pk;
            pk.x = *reinterpret_cast<unsigned*>(&lo);
            pk.y = *reinterpret_cast<unsigned*>(&hi);
            reinterpret_cast<uint2*>(shadow)[i] = pk;
        }
    }
}

// ============================================================== small utilities
__global__ void zero_kernel(float4* __restrict__ p, size_t n4) {
    pdl_wait();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void f32_to_bf16_kernel(bf16* __restrict__ out, const float* __restrict__ in, size_t n) {
    pdl_wait();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        out[i] = __float2bfloat16_rn(in[i]);
}

// ============================================================== Muon
// pimou.com article, sections "优化器的优势" and "相关技术的追溯": the Muon optimizer
// orthogonalizes each block matrix's momentum with Newton-Schulz iterations.
// mom = mu mom + g over the matrices' flat range (fp32)
__global__ void muon_momentum_kernel(float4* __restrict__ mom, const float4* __restrict__ g, size_t n4, float mu) {
    pdl_wait();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        float4 a = mom[i];
        const float4 b = g[i];
        a.x = fmaf(mu, a.x, b.x); a.y = fmaf(mu, a.y, b.y); a.z = fmaf(mu, a.z, b.z); a.w = fmaf(mu, a.w, b.w);
        mom[i] = a;
    }
}
#define MUON_NB 64          // blocks per matrix of the sum-of-squares partials
// partial[mat * MUON_NB + block] = sum of squares of the block's grid-stride slice of
// matrix `mat` (blockIdx.y; matrices of `len` elements back to back), tree-added in a
// fixed order
__global__ void __launch_bounds__(256) sumsq_partial_kernel(float* __restrict__ partial, const float* __restrict__ x,
                                                            size_t len) {
    pdl_wait();
    const float4* p = reinterpret_cast<const float4*>(x + (size_t)blockIdx.y * len);
    float acc = 0.f;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < len / 4; i += (size_t)MUON_NB * blockDim.x) {
        const float4 a = p[i];
        acc = fmaf(a.x, a.x, acc); acc = fmaf(a.y, a.y, acc); acc = fmaf(a.z, a.z, acc); acc = fmaf(a.w, a.w, acc);
    }
    acc = warp_sum(acc);
    __shared__ float ws[8];
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; w++) t += ws[w];
        partial[(size_t)blockIdx.y * MUON_NB + blockIdx.x] = t;
    }
}
// out = bf16(x / ||x||_F) for matrix blockIdx.y (0 where the norm is 0); every block sums
// the matrix's MUON_NB partials in the same order, so all agree on the norm
__global__ void __launch_bounds__(256) scale_frobenius_bf16_kernel(bf16* __restrict__ out, const float* __restrict__ x,
                                                                   const float* __restrict__ partial, size_t len) {
    pdl_wait();
    float ss = 0.f;
    for (int b = 0; b < MUON_NB; b++) ss += partial[(size_t)blockIdx.y * MUON_NB + b];
    const float inv = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
    const float4* p = reinterpret_cast<const float4*>(x + (size_t)blockIdx.y * len);
    __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(out + (size_t)blockIdx.y * len);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < len / 4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 a = p[i];
        o[2 * i] = __floats2bfloat162_rn(a.x * inv, a.y * inv);
        o[2 * i + 1] = __floats2bfloat162_rn(a.z * inv, a.w * inv);
    }
}
// T = 1.5 I - 0.5 S (n x n, bf16): the Newton-Schulz step X <- 1.5 X - 0.5 X S = X T
__global__ void ns_affine_kernel(bf16* __restrict__ T, const bf16* __restrict__ S, int n, int nb) {
    pdl_wait();
    const size_t nn = (size_t)n * n;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nn * nb; i += (size_t)gridDim.x * blockDim.x) {
        const size_t j = i % nn;                       // element of matrix i / nn
        const int r = (int)(j / n), c = (int)(j % n);
        T[i] = __float2bfloat16_rn((r == c ? 1.5f : 0.f) - 0.5f * __bfloat162float(S[i]));
    }
}
// p -= lr (X + wd p); shadow (nullable) = bf16(p)
__global__ void muon_apply_kernel(float4* __restrict__ p, const bf16* __restrict__ X, bf16* __restrict__ shadow,
                                  size_t n4, float lr, float wd) {
    pdl_wait();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        float4 a = p[i];
        const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(X) + 2 * i;
        const float2 x0 = __bfloat1622float2(xp[0]), x1 = __bfloat1622float2(xp[1]);
        a.x -= lr * (x0.x + wd * a.x); a.y -= lr * (x0.y + wd * a.y);
        a.z -= lr * (x1.x + wd * a.z); a.w -= lr * (x1.y + wd * a.w);
        p[i] = a;
        if (shadow) {
            __nv_bfloat162* sp = reinterpret_cast<__nv_bfloat162*>(shadow) + 2 * i;
            sp[0] = __floats2bfloat162_rn(a.x, a.y);
            sp[1] = __floats2bfloat162_rn(a.z, a.w);
        }
    }
}
