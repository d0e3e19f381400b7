// Host-side runtime shared by the library's translation units: the kernel-launch
// counter and the per-kernel-class tracer (CUDA events on the launching stream).
#pragma once
#include <cuda_runtime.h>

enum ProfClass {
    PC_ENCODER_FWD = 0, PC_ENCODER_BWD, PC_LAYERNORM_FWD, PC_LAYERNORM_BWD, PC_MATMUL_FWD,
    PC_MATMUL_BWD_DX, PC_MATMUL_BWD_DW, PC_BIAS_GRAD, PC_ATTENTION_FWD, PC_ATTENTION_BWD,
    PC_SOFTMAX_XENT, PC_ADAMW, PC_MISC, PC_NUM_CLASSES
};

// Count `n` kernel launches made by this library (process-wide).
void rt_note_launches(long long n);
// The launch count so far, and whether the tracer is recording (the step graph is then
// not used: its launches carry no events).
long long rt_launches();
bool rt_tracing_on();

// RAII scope: when tracing is on, records a CUDA event on `s` at construction and at
// destruction, attributing the interval and the given algorithmic work to `cls`.
struct ProfScope {
    ProfScope(cudaStream_t s, int cls, double flops, double bytes);
    ~ProfScope();
    cudaStream_t s_;
    int slot_;
};
