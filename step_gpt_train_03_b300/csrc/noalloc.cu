// Layernorm backward for callers that cannot allocate device memory.
//
// gpt2_layernorm_backward needs a scratch buffer for its deterministic two-stage column
// sums, and expects the caller to provide it.  Some callers have no way to get one: a
// host program that hands this library only its input and output buffers (a plugin
// inside another framework's step, say), or a program that commits all of its device
// memory at start-up and must not call cudaMalloc later, because the call would fail or
// would synchronise the whole device in the middle of the step.  For them,
// gpt2_layernorm_backward_noalloc takes its scratch from a fixed array compiled into
// this library.
//
// The array is a file-scope __device__ variable of GPT2_NOALLOC_SCRATCH_BYTES.  Every
// GPU that loads the library holds it until the process exits.  Every call shares it,
// so calls that overlap on the GPU (on two streams, or from two threads) race on it and
// must be serialised by the caller.  Each call rewrites every partial sum it later
// reads, so nothing is carried over from the previous call and nothing needs clearing.
#include <cuda_runtime.h>

#include "../../include/gpt2.h"

static __device__ __align__(256) float g_layernorm_scratch[GPT2_NOALLOC_SCRATCH_BYTES / sizeof(float)];

// Host code cannot pass the array's name to a kernel: on the host that name is a
// stand-in object, not a device address.  The device address is looked up on every
// call, with the caller's device current, so it always belongs to the current device
// and its current context (a cached address would go stale after cudaDeviceReset).  The
// lookup is cheap and allocates nothing; with lazy module loading the first lookup on a
// device is what loads the module holding the array, which is why the first call belongs
// in the caller's start-up.
static int scratch_address(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_layernorm_scratch) != cudaSuccess || !p) return GPT2_ECUDA;
    *out = p;
    return GPT2_OK;
}

extern "C" int gpt2_layernorm_backward_noalloc(float* dinp, float* dweight, float* dbias, const float* dout,
                                               const float* inp, const float* weight, const float* mean,
                                               const float* rstd, int N, int C, void* stream) {
    if (N < 0 || C < 8 || C % 8 || C > 2048) return GPT2_EINVAL;
    if (N == 0) return GPT2_OK;
    if (gpt2_layernorm_backward_scratch_bytes(N, C) > (size_t)GPT2_NOALLOC_SCRATCH_BYTES) return GPT2_EINVAL;
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != GPT2_OK) return rc;
    return gpt2_layernorm_backward(dinp, dweight, dbias, dout, inp, weight, mean, rstd, N, C, scratch,
                                   (size_t)GPT2_NOALLOC_SCRATCH_BYTES, stream);
}
