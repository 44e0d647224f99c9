// cq_gemm_q4_noalloc: the Q4 GEMM for callers that cannot allocate device
// memory.  cq_gemm_q4 needs a scratch buffer (the fp16 copy of X behind its
// power-of-two guard, plus one inverse scale per row) and asks the caller
// for it.  Some callers have no way to provide one: a plugin that runs inside
// a host framework which owns every device allocation, a runtime whose
// memory budget is fixed up front, or a latency-critical loop where a
// cudaMalloc / cudaFree (which can synchronise the whole device) is not
// acceptable.  This entry point keeps that scratch in a fixed array of this
// library instead, and otherwise runs exactly the kernels cq_gemm_q4 runs.
#include <mutex>

#include "cq_internal.h"

namespace cq {
namespace {

// Scratch for one call: [T][K] fp16 activations, then [T] f32 inverse
// scales, each section 256-byte aligned.  Every GPU that loads the library
// holds this array until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[CQ_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_scratch_ptr[MAX_DEVICES] = {};

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// The array's device address on the current device.  In host code the
// symbol's name is only a stand-in; the address must come from the runtime,
// once per device, with that device current.
cq_status scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= MAX_DEVICES) return fail(CQ_ERR_ARG, "cq_gemm_q4_noalloc: device index %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress (noalloc scratch)");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return CQ_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace cq

using namespace cq;

extern "C" cq_status cq_gemm_q4_noalloc(const void* X, int xt, int64_t T, int64_t K, const uint8_t* Wq,
                                         const uint16_t* Ws, int64_t N, void* Y, int yt, void* stream) {
    clear_last_error();
    if (!X || !Wq || !Ws || !Y) return fail(CQ_ERR_NULL, "cq_gemm_q4_noalloc: null pointer");
    if (xt != CQ_F16 && xt != CQ_BF16) return fail(CQ_ERR_DTYPE, "cq_gemm_q4_noalloc: activations must be fp16 or bf16");
    if (yt != CQ_F32 && yt != CQ_BF16) return fail(CQ_ERR_DTYPE, "cq_gemm_q4_noalloc: output must be f32 or bf16");
    if (T < 1 || N < 1 || K < 256 || K % 256 || T > (1LL << 31) - 1 || N > (1LL << 31) - 1)
        return fail(CQ_ERR_SHAPE, "cq_gemm_q4_noalloc: need T>=1, N>=1, K%%256==0 (T=%lld K=%lld N=%lld)",
                    (long long)T, (long long)K, (long long)N);
    const size_t xh_bytes = up256((size_t)T * (size_t)K * 2);
    const size_t need = xh_bytes + up256((size_t)T * 4);
    if (need > (size_t)CQ_NOALLOC_SCRATCH_BYTES)
        return fail(CQ_ERR_SHAPE,
                    "cq_gemm_q4_noalloc: T*K*2 (+ row scales) = %zu bytes exceeds the fixed %d-byte scratch; "
                    "use cq_gemm_q4 with a workspace",
                    need, (int)CQ_NOALLOC_SCRATCH_BYTES);
    if (!al16(X) || !al16(Wq) || !al16(Ws) || !al16(Y)) return fail(CQ_ERR_ALIGN, "cq_gemm_q4_noalloc: pointers must be 16-byte aligned");
    int dev = 0, major = 0, minor = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return fail(CQ_ERR_ARCH, "device %d is sm_%d%d, this library is built for sm_103a", dev, major, minor);
    void* scratch = nullptr;
    cq_status st = scratch_for_current_device(&scratch);
    if (st != CQ_OK) return st;
    // Nothing in the scratch has to start at zero: the guard pass writes every
    // element the GEMM reads for this call's T rows.
    uint16_t* xh = static_cast<uint16_t*>(scratch);
    float* rsx = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + xh_bytes);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = stream_error_word(s);
    if (!err) return CQ_ERR_CUDA;
    const Options& o = options();
    const bool skinny = o.force_path == 1 || (o.force_path == 0 && T <= o.small_t_max);
    if (skinny && T > 32) return fail(CQ_ERR_ARG, "cq_gemm_q4_noalloc: the weight-streaming path serves T <= 32");
    if (skinny) {   // the activations as given: no guard pass
        SkinnyDense a = {X, xt == CQ_BF16 ? 1 : 0, nullptr, nullptr, Wq, Ws, T, K, N, Y, yt, err};
        e = launch_skinny_q4(a, s);
        return e == cudaSuccess ? CQ_OK : cuda_fail(e, "weight-streaming Q4 GEMM");
    }
    e = launch_x_half(X, xt, T, K, xh, rsx, s);
    if (e != cudaSuccess) return cuda_fail(e, "activation guard pass");
    TcArgs a = {xh, 0, rsx, nullptr, Wq, Ws, T, K, N, Y, yt, err};
    e = launch_tc_q4(a, s);
    return e == cudaSuccess ? CQ_OK : cuda_fail(e, "tcgen05 Q4 GEMM");
}
