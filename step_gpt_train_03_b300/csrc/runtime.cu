// Launch counter and per-kernel-class tracer of the library (exports in include/gpt2.h).
//
// The tracer brackets every layer launch with two CUDA events recorded on the stream
// the kernels go to, and attributes the elapsed device time and the launch's algorithmic
// work (flops for contractions, bytes for memory-bound layers) to a kernel class.  The
// events come from a pool created when tracing is switched on; nothing is allocated on
// the device.
#include <atomic>
#include <vector>

#include "runtime.h"
#include "../../include/gpt2.h"

static std::atomic<long long> g_launches{0};

void rt_note_launches(long long n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {
struct Rec {
    int cls, e0, e1;
    double flops, bytes;
};
struct Tracer {
    bool on = false;
    unsigned mask = 0;
    std::vector<cudaEvent_t> ev;
    int next = 0;
    std::vector<Rec> recs;
    double ms[PC_NUM_CLASSES] = {};
    long long cnt[PC_NUM_CLASSES] = {};
    double fl[PC_NUM_CLASSES] = {}, by[PC_NUM_CLASSES] = {};
    long long dropped = 0;
};
Tracer T;
const int kPoolEvents = 1 << 17;
const char* kNames[PC_NUM_CLASSES] = {
    "encoder_forward", "encoder_backward", "layernorm_forward", "layernorm_backward", "matmul_forward",
    "matmul_backward_dx", "matmul_backward_dw", "bias_grad", "attention_forward", "attention_backward",
    "softmax_xent", "adamw", "misc"};
}  // namespace

ProfScope::ProfScope(cudaStream_t s, int cls, double flops, double bytes) : s_(s), slot_(-1) {
    if (!T.on || !((T.mask >> cls) & 1u)) return;
    if (T.next + 2 > (int)T.ev.size()) { T.dropped++; return; }
    Rec r{cls, T.next, T.next + 1, flops, bytes};
    T.next += 2;
    if (cudaEventRecord(T.ev[r.e0], s) != cudaSuccess) return;
    T.recs.push_back(r);
    slot_ = (int)T.recs.size() - 1;
}

ProfScope::~ProfScope() {
    if (slot_ >= 0) cudaEventRecord(T.ev[T.recs[slot_].e1], s_);
}

extern "C" long long gpt2_kernel_launches(void) { return g_launches.load(); }
long long rt_launches() { return g_launches.load(); }
bool rt_tracing_on() { return T.on; }

extern "C" int gpt2_profile_enable(unsigned class_mask) {
    const bool on = class_mask != 0;
    if (on && T.ev.empty()) {
        T.ev.resize(kPoolEvents);
        for (auto& e : T.ev)
            if (cudaEventCreate(&e) != cudaSuccess) return GPT2_ECUDA;
    }
    T.on = on;
    T.mask = class_mask;
    return GPT2_OK;
}

extern "C" int gpt2_profile_collect(void) {
    for (const Rec& r : T.recs) {
        if (cudaEventSynchronize(T.ev[r.e1]) != cudaSuccess) return GPT2_ECUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, T.ev[r.e0], T.ev[r.e1]) != cudaSuccess) return GPT2_ECUDA;
        T.ms[r.cls] += ms;
        T.cnt[r.cls] += 1;
        T.fl[r.cls] += r.flops;
        T.by[r.cls] += r.bytes;
    }
    T.recs.clear();
    T.next = 0;
    return GPT2_OK;
}

extern "C" int gpt2_profile_reset(void) {
    int rc = gpt2_profile_collect();
    for (int i = 0; i < PC_NUM_CLASSES; i++) { T.ms[i] = 0; T.cnt[i] = 0; T.fl[i] = 0; T.by[i] = 0; }
    T.dropped = 0;
    return rc;
}

extern "C" int gpt2_profile_read(int cls, double* ms, long long* scopes, double* flops, double* bytes) {
    if (cls < 0 || cls >= PC_NUM_CLASSES) return GPT2_EINVAL;
    if (ms) *ms = T.ms[cls];
    if (scopes) *scopes = T.cnt[cls];
    if (flops) *flops = T.fl[cls];
    if (bytes) *bytes = T.by[cls];
    return GPT2_OK;
}

extern "C" long long gpt2_profile_dropped(void) { return T.dropped; }

extern "C" int gpt2_profile_num_classes(void) { return PC_NUM_CLASSES; }

extern "C" const char* gpt2_profile_class_name(int cls) {
    return (cls >= 0 && cls < PC_NUM_CLASSES) ? kNames[cls] : "";
}
