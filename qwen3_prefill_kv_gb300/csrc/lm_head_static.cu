// qdec_op_lm_head_argmax_static: the tied lm_head + argmax without any allocation.
//
// Some callers cannot let a library allocate device memory: hosts that own every byte of
// the GPU through their own pooling allocator (a framework's caching allocator that has
// reserved the device), or real-time audio threads where cudaMalloc's implicit
// device-wide synchronisation and unbounded latency are not acceptable.  For them the
// per-block partial maxima and the ticket counter that qdec_op_lm_head_argmax keeps in
// caller-provided scratch live here in one file-scope device array instead.
//
// In host code the array's name is only a host-side stand-in, never a device address:
// its device address is looked up once per device with cudaGetSymbolAddress (with that
// device current) and passed to the kernel.  Every GPU that loads the library holds the
// array until the process exits.
#include <mutex>

#include "../../include/qdec.h"
#include "../../include/qdec_ops.h"
#include "common.cuh"

using namespace qdec;

namespace {

constexpr size_t kStaticScratchBytes = 65792;   // >= lm_head_scratch_bytes(QDEC_LM_HEAD_STATIC_MAX_VOCAB)
static __device__ __align__(256) unsigned char g_lm_head_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_dev_addr[kMaxDevices] = {};

// Device address of g_lm_head_scratch on the current device (looked up on first use).
int scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(QDEC_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return set_error(QDEC_E_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_dev_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_lm_head_scratch);
        if (e != cudaSuccess || !p)
            return set_error(QDEC_E_CUDA, "cudaGetSymbolAddress(lm_head scratch): %s", cudaGetErrorString(e));
        g_dev_addr[dev] = p;
    }
    *out = g_dev_addr[dev];
    return QDEC_OK;
}

}  // namespace

extern "C" int qdec_op_lm_head_argmax_static(const void* E, int32_t V, int32_t H, const float* x, const void* g_final,
                                             float eps, float* logits, int32_t* argmax, void* stream) {
    if (!E || !x || !g_final || !logits || !argmax || V <= 0 || H <= 0 || H % 8 != 0)
        return set_error(QDEC_E_INVALID_ARG, "qdec_op_lm_head_argmax_static: null pointer or bad size");
    if (V > QDEC_LM_HEAD_STATIC_MAX_VOCAB)
        return set_error(QDEC_E_INVALID_ARG, "qdec_op_lm_head_argmax_static: vocab %d exceeds the static maximum %d",
                         V, QDEC_LM_HEAD_STATIC_MAX_VOCAB);
    static_assert(kStaticScratchBytes >= 16 + ((QDEC_LM_HEAD_STATIC_MAX_VOCAB + 31) / 32) * 8,
                  "static scratch too small for the maximum vocabulary");
    if (lm_head_scratch_bytes(V) > kStaticScratchBytes)
        return set_error(QDEC_E_INVALID_ARG, "qdec_op_lm_head_argmax_static: scratch layout exceeds the static array");
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != QDEC_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps whatever the last call left; the ticket counter must start at zero.
    cudaError_t e = cudaMemsetAsync(scratch, 0, 16, s);
    if (e != cudaSuccess) return set_error(QDEC_E_CUDA, "clearing the static scratch: %s", cudaGetErrorString(e));
    e = launch_lm_head_argmax(static_cast<const bf16_t*>(E), V, H, x, static_cast<const bf16_t*>(g_final), eps,
                              logits, argmax, scratch, s);
    if (e != cudaSuccess) return set_error(QDEC_E_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    return QDEC_OK;
}
