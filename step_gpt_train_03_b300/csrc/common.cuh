// Shared device helpers: element types, vector access, warp reductions, error word.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

typedef __nv_bfloat16 bf16;

// Bits of the device error word (bit index = status code).
#define ERRBIT_TOKEN (1u << 4)
#define ERRBIT_NONFINITE (1u << 5)
#define ERRBIT_TIMEOUT (1u << 6)

__device__ __forceinline__ void raise_error(unsigned int* err, unsigned int bit) {
    if (err) atomicOr(err, bit);
}

// ------------------------------------------------------------------ scalar conversion
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// ------------------------------------------------------------------ 16-byte vectors
// Vec<T> is one 16-byte packet: 4 floats or 8 bf16.
template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int N = 4;
    float4 v;
    __device__ __forceinline__ float get(int i) const { return (&v.x)[i]; }
    __device__ __forceinline__ void set(int i, float x) { (&v.x)[i] = x; }
    __device__ __forceinline__ float2 get2(int i) const { return i == 0 ? make_float2(v.x, v.y) : make_float2(v.z, v.w); }
    __device__ __forceinline__ void set2(int i, float x, float y) {
        if (i == 0) { v.x = x; v.y = y; } else { v.z = x; v.w = y; }
    }
};
template <> struct Vec<bf16> {
    static constexpr int N = 8;
    uint4 v;
    __device__ __forceinline__ float get(int i) const {
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
        float2 f = __bfloat1622float2(p[i >> 1]);
        return (i & 1) ? f.y : f.x;
    }
    __device__ __forceinline__ void set(int i, float x) {
        bf16* p = reinterpret_cast<bf16*>(&v);
        p[i] = __float2bfloat16_rn(x);
    }
    // elements i, i+1 (i even): one packed conversion each way
    __device__ __forceinline__ float2 get2(int i) const {
        return __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(&v)[i >> 1]);
    }
    __device__ __forceinline__ void set2(int i, float x, float y) {
        reinterpret_cast<__nv_bfloat162*>(&v)[i >> 1] = __floats2bfloat162_rn(x, y);
    }
};

template <typename T> __device__ __forceinline__ Vec<T> load_vec(const T* p) {
    Vec<T> r;
    if constexpr (sizeof(T) == 4) r.v = *reinterpret_cast<const float4*>(p);
    else r.v = *reinterpret_cast<const uint4*>(p);
    return r;
}
template <typename T> __device__ __forceinline__ Vec<T> load_vec_stream(const T* p) {
    Vec<T> r;
    if constexpr (sizeof(T) == 4) r.v = __ldcs(reinterpret_cast<const float4*>(p));
    else r.v = __ldcs(reinterpret_cast<const uint4*>(p));
    return r;
}
template <typename T> __device__ __forceinline__ void store_vec(T* p, const Vec<T>& x) {
    if constexpr (sizeof(T) == 4) *reinterpret_cast<float4*>(p) = x.v;
    else *reinterpret_cast<uint4*>(p) = x.v;
}

// ------------------------------------------------------------------ reductions
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// ------------------------------------------------------------------ GELU (tanh form)
#define GELU_K0 0.7978845608028654f   /* sqrt(2/pi) */
#define GELU_K1 0.044715f
__device__ __forceinline__ float gelu_f(float x) {
    float u = GELU_K0 * (x + GELU_K1 * x * x * x);
    return 0.5f * x * (1.0f + tanhf(u));
}
__device__ __forceinline__ float gelu_grad_f(float x) {
    float u = GELU_K0 * (x + GELU_K1 * x * x * x);
    float th = tanhf(u);
    float sech2 = 1.0f - th * th;
    return 0.5f * (1.0f + th) + 0.5f * x * sech2 * GELU_K0 * (1.0f + 3.0f * GELU_K1 * x * x);
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ size_t ceil_div_sz(size_t a, size_t b) { return (a + b - 1) / b; }

// Column sums of a warp's 32 x 32 block, v[i] being column i of this lane's row: a
// halving exchange (at width w, a lane keeps the half of its w pending columns that its
// bit w selects and adds its partner's copy of that half), 31 shuffles per lane.  Returns
// the sum over the 32 lanes of column `lane`; the order of the additions is fixed.
__device__ __forceinline__ float warp_colsum32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int i = 0; i < w; i++) {
            const float send = up ? v[i] : v[i + w];
            const float keep = up ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return v[0];
}

// ------------------------------------------------------------------ dependent launches
// Every kernel of the library starts with pdl_wait(): launched with programmatic stream
// serialization, a kernel may begin before its predecessor in the stream has finished,
// and this waits until the predecessor has completed and its memory writes are visible
// (launched normally, it returns at once).  Kernels whose CTAs are all resident from
// their launch (the persistent tensor-core kernels) also call pdl_trigger() after their
// set-up, letting the next kernel's CTAs launch onto SMs as they free up and do their
// own set-up before they, in turn, wait.  Kernels with more CTAs than resident slots do
// not trigger, so a waiting successor can never hold a slot one of their CTAs needs.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

#include <utility>
// Launch `kern` with programmatic stream serialization allowed (see pdl_wait).
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
