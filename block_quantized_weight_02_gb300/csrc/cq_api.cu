// The C ABI: argument checks, workspace carve-up, path choice and launch
// order.  Every step of the computation runs in the kernels of k_aux.cu,
// k_skinny.cu and k_tc.cu; nothing here touches the data.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "cq_internal.h"

namespace cq {

Options& options() {
    static Options o;
    return o;
}

static thread_local char g_msg[512] = "";

cq_status fail(cq_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    int n = snprintf(g_msg, sizeof g_msg, "decline: ");
    vsnprintf(g_msg + n, sizeof g_msg - n, fmt, ap);
    va_end(ap);
    return st;
}

static thread_local int g_launches = 0;   // kernel launches of the thread's current entry-point call

void clear_last_error() {
    g_msg[0] = 0;
    g_launches = 0;
}
cudaError_t counted(cudaError_t e) {
    if (e == cudaSuccess) ++g_launches;
    return e;
}
int launches_so_far() { return g_launches; }

cq_status cuda_fail(cudaError_t e, const char* what) {
    return fail(CQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    if (!fn) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, dt, (cuuint32_t)rank, const_cast<void*>(base), reinterpret_cast<const cuuint64_t*>(dims),
                    reinterpret_cast<const cuuint64_t*>(strides_bytes), reinterpret_cast<const cuuint32_t*>(box),
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ---- per-stream device error words ----------------------------------------
// A fixed table in device memory (every GPU that loads the library holds it):
// slot 0 is shared by the streams beyond the first CQ_ERR_SLOTS - 1 of a device,
// every other slot belongs to one (device, stream) pair from its first call on.
constexpr int CQ_ERR_SLOTS = 1024;
static __device__ int g_err_slots[CQ_ERR_SLOTS];

namespace {
constexpr int MAX_DEVICES = 64;
std::mutex g_slot_mu;
int* g_slot_base[MAX_DEVICES] = {};
int g_slot_next[MAX_DEVICES] = {};
std::map<std::pair<int, uintptr_t>, int>& slot_map() {
    static std::map<std::pair<int, uintptr_t>, int> m;
    return m;
}
}  // namespace

int* stream_error_word(cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cuda_fail(e, "cudaGetDevice");
        return nullptr;
    }
    if (dev < 0 || dev >= MAX_DEVICES) {
        fail(CQ_ERR_ARG, "device index %d out of range", dev);
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_slot_mu);
    if (!g_slot_base[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_err_slots);   // the array's address on this device
        if (e != cudaSuccess || !p) {
            cuda_fail(e, "cudaGetSymbolAddress (device error words)");
            return nullptr;
        }
        g_slot_base[dev] = static_cast<int*>(p);
        g_slot_next[dev] = 1;
    }
    auto& m = slot_map();
    const auto key = std::make_pair(dev, reinterpret_cast<uintptr_t>(s));
    auto it = m.find(key);
    int slot = 0;
    if (it != m.end()) {
        slot = it->second;
    } else if (g_slot_next[dev] < CQ_ERR_SLOTS) {
        slot = g_slot_next[dev]++;
        m.emplace(key, slot);
    }
    return g_slot_base[dev] + slot;
}

int num_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

namespace {

constexpr size_t ALIGN = 256;
size_t up(size_t v) { return (v + ALIGN - 1) / ALIGN * ALIGN; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

cq_status check_arch() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return fail(CQ_ERR_ARCH, "device %d is sm_%d%d, this library is built for sm_103a", dev, major, minor);
    return CQ_OK;
}

cq_status check_x(int xt) {
    if (xt != CQ_F16 && xt != CQ_BF16) return fail(CQ_ERR_DTYPE, "activations must be fp16 or bf16 (got %d)", xt);
    return CQ_OK;
}
cq_status check_y(int yt) {
    if (yt != CQ_F32 && yt != CQ_BF16) return fail(CQ_ERR_DTYPE, "output must be f32 or bf16 (got %d)", yt);
    return CQ_OK;
}

// Workspace of the Q4 GEMM: guarded fp16 activations, then inverse scales.
struct Q4Ws {
    uint16_t* xh;
    float* rsx;
};
size_t q4_ws_bytes(int64_t T, int64_t K) { return up((size_t)T * K * 2) + up((size_t)T * 4); }
Q4Ws q4_ws(void* ws, int64_t T, int64_t K) {
    uint8_t* b = static_cast<uint8_t*>(ws);
    return {reinterpret_cast<uint16_t*>(b), reinterpret_cast<float*>(b + up((size_t)T * K * 2))};
}

struct MoeLayout {
    size_t status, seg, perm, inv, act, cnt, xh, rsx, a, ah, rsa, eo, total;
};
MoeLayout moe_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk) {
    const size_t P = (size_t)(T * topk);
    MoeLayout l;
    size_t o = 0;
    l.status = o; o += up(4);
    l.seg = o; o += up((size_t)(E + 1) * 4);
    l.perm = o; o += up(P * 4);
    l.inv = o; o += up(P * 4);
    l.act = o; o += up((size_t)(E + 1) * 4);   // active experts, then their count
    l.cnt = o; o += up((size_t)(H / 128) * 4);  // down items finished per 128-row block
    l.xh = o; o += up(P * H * 2);
    l.rsx = o; o += up(P * 4);
    l.a = o; o += up(P * I * 4);
    l.ah = o; o += up(P * I * 2);
    l.rsa = o; o += up(P * 4);
    l.eo = o; o += up(P * H * 4);
    l.total = o;
    return l;
}

// Workspace of the dense FFN chain: guarded fp16 X and its scales, the f32
// SwiGLU activations a, their guarded fp16 copy and its scales.
struct FfnLayout {
    size_t xh, rsx, a, ah, rsa, total;
};
FfnLayout ffn_layout(int64_t T, int64_t H, int64_t I) {
    FfnLayout l;
    size_t o = 0;
    l.xh = o; o += up((size_t)T * H * 2);
    l.rsx = o; o += up((size_t)T * 4);
    l.a = o; o += up((size_t)T * I * 4);
    l.ah = o; o += up((size_t)T * I * 2);
    l.rsa = o; o += up((size_t)T * 4);
    l.total = o;
    return l;
}

bool use_skinny(int64_t T) {
    const Options& o = options();
    if (o.force_path == 1) return true;
    if (o.force_path == 2) return false;
    return T <= o.small_t_max;
}

cq_status launched(cudaError_t e, const char* what) {
    if (e != cudaSuccess) return cuda_fail(e, what);
    return CQ_OK;
}

}  // namespace
}  // namespace cq

using namespace cq;

extern "C" {

int cq_version(void) { return 100; }

const char* cq_last_error(void) { return g_msg; }
int cq_last_launches(void) { return launches_so_far(); }

cq_status cq_set_option(int option, int64_t value) {
    Options& o = options();
    switch (option) {
        case CQ_OPT_SMALL_T_MAX:
            if (value < 0 || value > 32) return fail(CQ_ERR_ARG, "small-T limit must be in [0, 32]");
            o.small_t_max = value;
            return CQ_OK;
        case CQ_OPT_FORCE_PATH:
            if (value < 0 || value > 2) return fail(CQ_ERR_ARG, "path must be 0, 1 or 2");
            o.force_path = value;
            return CQ_OK;
        case CQ_OPT_WAIT_NS:
            if (value < 1000000 || value > 60000000000LL) return fail(CQ_ERR_ARG, "wait limit must be in [1 ms, 60 s]");
            o.wait_ns = value;
            return CQ_OK;
        case CQ_OPT_TEST_STALL:
            if (value != 0 && value != 1) return fail(CQ_ERR_ARG, "stall must be 0 or 1");
            o.test_stall = value;
            return CQ_OK;
        case CQ_OPT_TRACE:
            o.trace = value != 0;
            return CQ_OK;
        case CQ_OPT_TC_BN:
            if (value != 0 && value != 32 && value != 64 && value != 128 && value != 192 && value != 256) return fail(CQ_ERR_ARG, "token tile must be 0, 32, 64, 128, 192 or 256");
            o.tc_bn = value;
            return CQ_OK;
        case CQ_OPT_TC_KSPLIT:
            if (value != 0 && value != 1 && value != 2) return fail(CQ_ERR_ARG, "K split must be 0, 1 or 2");
            o.tc_ksplit = value;
            return CQ_OK;
        case CQ_OPT_TC_AMODE:
            if (value < 0 || value > 2) return fail(CQ_ERR_ARG, "operand mode must be 0, 1 or 2");
            o.tc_amode = value;
            return CQ_OK;
        case CQ_OPT_TC_PAIR:
            if (value < 0 || value > 2) return fail(CQ_ERR_ARG, "CTA pair mode must be 0, 1 or 2");
            o.tc_pair = value;
            return CQ_OK;
        case CQ_OPT_STREAM_KERNEL:
            if (value < 0 || value > 2) return fail(CQ_ERR_ARG, "weight-streaming kernel must be 0, 1 or 2");
            o.stream_kernel = value;
            return CQ_OK;
        default:
            return fail(CQ_ERR_ARG, "unknown option %d", option);
    }
}

int64_t cq_get_option(int option) {
    const Options& o = options();
    switch (option) {
        case CQ_OPT_SMALL_T_MAX: return o.small_t_max;
        case CQ_OPT_FORCE_PATH: return o.force_path;
        case CQ_OPT_WAIT_NS: return o.wait_ns;
        case CQ_OPT_TEST_STALL: return o.test_stall;
        case CQ_OPT_TRACE: return o.trace;
        case CQ_OPT_TC_BN: return o.tc_bn;
        case CQ_OPT_TC_KSPLIT: return o.tc_ksplit;
        case CQ_OPT_TC_AMODE: return o.tc_amode;
        case CQ_OPT_TC_PAIR: return o.tc_pair;
        case CQ_OPT_STREAM_KERNEL: return o.stream_kernel;
        default: return -1;
    }
}

size_t cq_gemm_q4_workspace_bytes(int64_t T, int64_t K) {
    if (T < 1 || K < 1) return 0;
    return q4_ws_bytes(T, K);
}

cq_status cq_gemm_q4(const void* X, int xt, int64_t T, int64_t K, const uint8_t* Wq, const uint16_t* Ws, int64_t N,
                     void* Y, int yt, void* ws, size_t ws_bytes, void* stream) {
    clear_last_error();
    if (!X || !Wq || !Ws || !Y || !ws) return fail(CQ_ERR_NULL, "cq_gemm_q4: null pointer");
    cq_status st;
    if ((st = check_x(xt)) || (st = check_y(yt))) return st;
    if (T < 1 || N < 1 || K < 256 || K % 256) return fail(CQ_ERR_SHAPE, "cq_gemm_q4: need T>=1, N>=1, K%%256==0 (T=%lld K=%lld N=%lld)", (long long)T, (long long)K, (long long)N);
    if (T > (1LL << 31) - 1 || N > (1LL << 31) - 1) return fail(CQ_ERR_SHAPE, "cq_gemm_q4: T and N must fit in int32");
    if (!aligned16(X) || !aligned16(Wq) || !aligned16(Ws) || !aligned16(Y)) return fail(CQ_ERR_ALIGN, "cq_gemm_q4: pointers must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(ws) & (ALIGN - 1)) || ws_bytes < q4_ws_bytes(T, K)) return fail(CQ_ERR_WORKSPACE, "cq_gemm_q4: workspace needs %zu bytes, 256-aligned", q4_ws_bytes(T, K));
    if ((st = check_arch())) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = stream_error_word(s);
    if (!err) return CQ_ERR_CUDA;
    const Q4Ws w = q4_ws(ws, T, K);
    const bool skinny = use_skinny(T);
    if (skinny && T > 32) return fail(CQ_ERR_ARG, "cq_gemm_q4: the weight-streaming path serves T <= 32");
    if (skinny) {   // the activations as given: no guard pass
        SkinnyDense a = {X, xt == CQ_BF16 ? 1 : 0, nullptr, nullptr, Wq, Ws, T, K, N, Y, yt, err};
        return launched(launch_skinny_q4(a, s), "weight-streaming Q4 GEMM");
    }
    if ((st = launched(launch_x_half(X, xt, T, K, w.xh, w.rsx, s), "activation guard pass"))) return st;
    TcArgs a = {w.xh, 0, w.rsx, nullptr, Wq, Ws, T, K, N, Y, yt, err};
    return launched(launch_tc_q4(a, s), "tcgen05 Q4 GEMM");
}

cq_status cq_gemm_q8row(const void* X, int xt, int64_t T, int64_t K, const int8_t* Wq, const float* rs, int64_t N,
                        void* Y, int yt, void* stream) {
    clear_last_error();
    if (!X || !Wq || !rs || !Y) return fail(CQ_ERR_NULL, "cq_gemm_q8row: null pointer");
    cq_status st;
    if ((st = check_x(xt)) || (st = check_y(yt))) return st;
    if (T < 1 || N < 1 || K < 128 || K % 128) return fail(CQ_ERR_SHAPE, "cq_gemm_q8row: need T>=1, N>=1, K%%128==0 (T=%lld K=%lld N=%lld)", (long long)T, (long long)K, (long long)N);
    if (T > (1LL << 31) - 1 || N > (1LL << 31) - 1) return fail(CQ_ERR_SHAPE, "cq_gemm_q8row: T and N must fit in int32");
    if (!aligned16(X) || !aligned16(Wq) || !aligned16(rs) || !aligned16(Y)) return fail(CQ_ERR_ALIGN, "cq_gemm_q8row: pointers must be 16-byte aligned");
    if ((st = check_arch())) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = stream_error_word(s);
    if (!err) return CQ_ERR_CUDA;
    if (use_skinny(T)) {
        if (T > 32) return fail(CQ_ERR_ARG, "cq_gemm_q8row: the weight-streaming path serves T <= 32");
        SkinnyDense a = {X, xt == CQ_BF16, nullptr, rs, reinterpret_cast<const uint8_t*>(Wq), nullptr, T, K, N, Y, yt, err};
        return launched(launch_skinny_q8(a, s), "weight-streaming Q8-row GEMM");
    }
    TcArgs a = {X, xt == CQ_BF16, nullptr, rs, reinterpret_cast<const uint8_t*>(Wq), nullptr, T, K, N, Y, yt, err};
    return launched(launch_tc_q8(a, s), "tcgen05 Q8-row GEMM");
}

size_t cq_moe_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk) {
    if (T < 1 || H < 1 || I < 1 || E < 1 || topk < 1) return 0;
    return moe_layout(T, H, I, E, topk).total;
}

cq_status cq_moe_panels(const void* X, int xt, int64_t T, int64_t H, int64_t E, int64_t I, int64_t topk,
                        const int32_t* idx, const float* w, const uint8_t* Wgu_q, const uint16_t* Wgu_s,
                        const uint8_t* Wd_q, const uint16_t* Wd_s, void* Y, int yt, void* ws, size_t ws_bytes,
                        void* stream) {
    clear_last_error();
    if (!X || !idx || !w || !Wgu_q || !Wgu_s || !Wd_q || !Wd_s || !Y || !ws) return fail(CQ_ERR_NULL, "cq_moe_panels: null pointer");
    cq_status st;
    if ((st = check_x(xt)) || (st = check_y(yt))) return st;
    if (T < 1 || topk < 1 || topk > 64 || E < 1 || E > 1024 || T * topk > 65536 || H < 256 || H % 256 || I < 256 ||
        I % 256 || H > 16384)
        return fail(CQ_ERR_SHAPE, "cq_moe_panels: shape rules broken (T=%lld H=%lld I=%lld E=%lld topk=%lld)",
                    (long long)T, (long long)H, (long long)I, (long long)E, (long long)topk);
    if (!aligned16(X) || !aligned16(idx) || !aligned16(w) || !aligned16(Wgu_q) || !aligned16(Wgu_s) ||
        !aligned16(Wd_q) || !aligned16(Wd_s) || !aligned16(Y))
        return fail(CQ_ERR_ALIGN, "cq_moe_panels: pointers must be 16-byte aligned");
    const MoeLayout l = moe_layout(T, H, I, E, topk);
    if ((reinterpret_cast<uintptr_t>(ws) & (ALIGN - 1)) || ws_bytes < l.total) return fail(CQ_ERR_WORKSPACE, "cq_moe_panels: workspace needs %zu bytes, 256-aligned", l.total);
    if ((st = check_arch())) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = stream_error_word(s);
    if (!err) return CQ_ERR_CUDA;
    uint8_t* b = static_cast<uint8_t*>(ws);
    int32_t* status = reinterpret_cast<int32_t*>(b + l.status);
    SkinnyMoe m = {};
    m.err = err;
    m.xh = reinterpret_cast<uint16_t*>(b + l.xh);
    m.rsx = reinterpret_cast<float*>(b + l.rsx);
    m.ah = reinterpret_cast<uint16_t*>(b + l.ah);
    m.rsa = reinterpret_cast<float*>(b + l.rsa);
    m.w = w;
    m.seg = reinterpret_cast<int32_t*>(b + l.seg);
    m.perm = reinterpret_cast<int32_t*>(b + l.perm);
    m.status = status;
    m.gu_q = Wgu_q;
    m.gu_s = Wgu_s;
    m.d_q = Wd_q;
    m.d_s = Wd_s;
    m.a = reinterpret_cast<float*>(b + l.a);
    m.eo = reinterpret_cast<float*>(b + l.eo);
    m.T = T;
    m.H = H;
    m.I = I;
    m.E = E;
    m.topk = topk;
    int32_t* inv = reinterpret_cast<int32_t*>(b + l.inv);
    int32_t* act = reinterpret_cast<int32_t*>(b + l.act);
    m.act = act;
    m.n_act = act + E;
    m.inv = inv;
    m.cnt = reinterpret_cast<int32_t*>(b + l.cnt);
    m.y = Y;
    m.yt = yt;
    if ((st = launched(launch_moe_route_gather(idx, T, topk, E, const_cast<int32_t*>(m.seg), const_cast<int32_t*>(m.perm),
                                               inv, act, act + E, status, m.cnt, (int)(H / 128), err, X, xt, H,
                                               const_cast<uint16_t*>(m.xh), const_cast<float*>(m.rsx), s),
                       "MoE routing layout + gathered guard pass")))
        return st;
    if ((st = launched(launch_moe_gateup(m, s), "MoE gate/up panels"))) return st;
    if ((st = launched(launch_a_half(m.a, T * topk, I, const_cast<uint16_t*>(m.ah), const_cast<float*>(m.rsa), status, s), "MoE SwiGLU guard pass"))) return st;
    return launched(launch_moe_down(m, s), "MoE down panels + combine");
}

size_t cq_gemm_q4_batched_workspace_bytes(int64_t T, int64_t K, int z) {
    if (T < 1 || K < 1 || z < 1 || z > ZMAX) return 0;
    return (size_t)z * q4_ws_bytes(T, K);
}

cq_status cq_gemm_q4_batched(const void* X, int xt, int64_t T, int64_t K, int64_t ldx, const cq_q4_job* jobs, int z,
                             int64_t N, void* Y, int yt, int64_t ldy, void* ws, size_t ws_bytes, void* stream) {
    clear_last_error();
    if (!X || !jobs || !Y || !ws) return fail(CQ_ERR_NULL, "cq_gemm_q4_batched: null pointer");
    if (z < 1 || z > ZMAX) return fail(CQ_ERR_ARG, "cq_gemm_q4_batched: z must be in [1, %d] (got %d)", ZMAX, z);
    cq_status st;
    if ((st = check_x(xt)) || (st = check_y(yt))) return st;
    if (T < 1 || N < 1 || K < 256 || K % 256 || T > (1LL << 31) - 1 || N > (1LL << 31) - 1)
        return fail(CQ_ERR_SHAPE, "cq_gemm_q4_batched: need T>=1, N>=1, K%%256==0 (T=%lld K=%lld N=%lld)", (long long)T,
                    (long long)K, (long long)N);
    if (ldx < K || ldx % 8 || ldy < N)
        return fail(CQ_ERR_SHAPE, "cq_gemm_q4_batched: need ldx >= K, ldx %% 8 == 0, ldy >= N (ldx=%lld ldy=%lld)",
                    (long long)ldx, (long long)ldy);
    for (int j = 0; j < z; ++j) {
        const cq_q4_job& jb = jobs[j];
        if (!jb.Wq || !jb.Ws) return fail(CQ_ERR_NULL, "cq_gemm_q4_batched: job %d: null weight pointer", j);
        if (!aligned16(jb.Wq) || !aligned16(jb.Ws)) return fail(CQ_ERR_ALIGN, "cq_gemm_q4_batched: job %d: weights must be 16-byte aligned", j);
        if (jb.x_off < 0 || jb.x_off % 8 || jb.x_off + K > ldx || jb.y_off < 0 || jb.y_off + N > ldy)
            return fail(CQ_ERR_SHAPE, "cq_gemm_q4_batched: job %d: need x_off %% 8 == 0, x_off + K <= ldx, y_off + N <= ldy", j);
    }
    if (!aligned16(X) || !aligned16(Y)) return fail(CQ_ERR_ALIGN, "cq_gemm_q4_batched: X and Y must be 16-byte aligned");
    const size_t need = (size_t)z * q4_ws_bytes(T, K);
    if ((reinterpret_cast<uintptr_t>(ws) & (ALIGN - 1)) || ws_bytes < need)
        return fail(CQ_ERR_WORKSPACE, "cq_gemm_q4_batched: workspace needs %zu bytes, 256-aligned", need);
    if ((st = check_arch())) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = stream_error_word(s);
    if (!err) return CQ_ERR_CUDA;
    const size_t esz = yt == CQ_F32 ? 4 : 2;
    const uint16_t* x16 = static_cast<const uint16_t*>(X);
    uint8_t* y8 = static_cast<uint8_t*>(Y);
    if (use_skinny(T)) {   // the activations as given: no guard pass
        if (T > 32) return fail(CQ_ERR_ARG, "cq_gemm_q4_batched: the weight-streaming path serves T <= 32");
        SkinnyDense a = {};
        a.x_bf16 = xt == CQ_BF16;
        a.T = T;
        a.K = K;
        a.N = N;
        a.yt = yt;
        a.err = err;
        a.nz = z;
        a.ldx = ldx;
        a.ldy = ldy;
        for (int j = 0; j < z; ++j)
            a.more[j] = {x16 + jobs[j].x_off, nullptr, jobs[j].Wq, jobs[j].Ws, y8 + jobs[j].y_off * esz};
        a.x = a.more[0].x;
        a.wq = a.more[0].wq;
        a.ws = a.more[0].ws;
        a.y = a.more[0].y;
        return launched(launch_skinny_q4(a, s), "z-batched weight-streaming Q4 GEMM");
    }
    // one guard pass per distinct activation slice (jobs that share X share it)
    TcArgs a = {};
    a.T = T;
    a.K = K;
    a.N = N;
    a.yt = yt;
    a.err = err;
    a.nz = z;
    a.ldy = ldy;
    int slot_of[ZMAX];
    int64_t slot_off[ZMAX];
    int nslots = 0;
    for (int j = 0; j < z; ++j) {
        int c = 0;
        while (c < nslots && slot_off[c] != jobs[j].x_off) ++c;
        if (c == nslots) {
            slot_off[nslots++] = jobs[j].x_off;
            const Q4Ws w = q4_ws(static_cast<uint8_t*>(ws) + (size_t)c * q4_ws_bytes(T, K), T, K);
            if ((st = launched(launch_x_half(x16 + jobs[j].x_off, xt, T, K, w.xh, w.rsx, s, ldx), "activation guard pass")))
                return st;
        }
        slot_of[j] = c;
    }
    for (int j = 0; j < z; ++j) {
        const Q4Ws w = q4_ws(static_cast<uint8_t*>(ws) + (size_t)slot_of[j] * q4_ws_bytes(T, K), T, K);
        a.more[j] = {w.xh, w.rsx, nullptr, jobs[j].Wq, jobs[j].Ws, y8 + jobs[j].y_off * esz};
    }
    a.x = a.more[0].x;
    a.rsx = a.more[0].rsx;
    a.wq = a.more[0].wq;
    a.ws = a.more[0].ws;
    a.y = a.more[0].y;
    return launched(launch_tc_q4(a, s), "z-batched tcgen05 Q4 GEMM");
}

// ---- format variants --------------------------------------------------------

size_t cq_gemm_q8_2f_workspace_bytes(int64_t T, int64_t K) { return (T < 1 || K < 1) ? 0 : q4_ws_bytes(T, K); }
size_t cq_gemm_q8b_workspace_bytes(int64_t T, int64_t K) { return (T < 1 || K < 1) ? 0 : q4_ws_bytes(T, K); }
size_t cq_gemm_q4a_workspace_bytes(int64_t T, int64_t K, int64_t N, int64_t gk) {
    if (T < 1 || K < 32 || N < 1 || gk < 1) return 0;
    return q4_ws_bytes(T, K) + up((size_t)T * (size_t)(K / 32 / gk) * 4) + up((size_t)T * N * 4);
}

cq_status cq_gemm_q8_2f(const void* X, int xt, int64_t T, int64_t K, const int8_t* Wq, const float* rs, const float* col,
                        int64_t N, void* Y, int yt, void* ws, size_t ws_bytes, void* stream) {
    clear_last_error();
    if (!X || !Wq || !rs || !col || !Y || !ws) return fail(CQ_ERR_NULL, "cq_gemm_q8_2f: null pointer");
    cq_status st;
    if ((st = check_x(xt)) || (st = check_y(yt))) return st;
    if (T < 1 || N < 1 || K < 128 || K % 128 || T > (1LL << 31) - 1 || N > (1LL << 31) - 1)
        return fail(CQ_ERR_SHAPE, "cq_gemm_q8_2f: need T>=1, N>=1, K%%128==0 (T=%lld K=%lld N=%lld)", (long long)T,
                    (long long)K, (long long)N);
    if (!aligned16(X) || !aligned16(Wq) || !aligned16(rs) || !aligned16(col) || !aligned16(Y))
        return fail(CQ_ERR_ALIGN, "cq_gemm_q8_2f: pointers must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(ws) & (ALIGN - 1)) || ws_bytes < q4_ws_bytes(T, K))
        return fail(CQ_ERR_WORKSPACE, "cq_gemm_q8_2f: workspace needs %zu bytes, 256-aligned", q4_ws_bytes(T, K));
    if ((st = check_arch())) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = stream_error_word(s);
    if (!err) return CQ_ERR_CUDA;
    const Q4Ws w = q4_ws(ws, T, K);
    // X times the column field, to fp16 behind the guard (k order); the Q8-row kernels then apply
    // the row scale and the guard's inverse per token
    if ((st = launched(launch_x_col_half(X, xt, col, T, K, w.xh, w.rsx, s), "q8_2f column-field guard pass"))) return st;
    const uint8_t* q = reinterpret_cast<const uint8_t*>(Wq);
    if (use_skinny(T)) {
        if (T > 32) return fail(CQ_ERR_ARG, "cq_gemm_q8_2f: the weight-streaming path serves T <= 32");
        SkinnyDense a = {w.xh, 0, w.rsx, rs, q, nullptr, T, K, N, Y, yt, err};
        return launched(launch_skinny_q8(a, s), "weight-streaming q8_2f GEMM");
    }
    TcArgs a = {w.xh, 0, w.rsx, rs, q, nullptr, T, K, N, Y, yt, err};
    return launched(launch_tc_q8(a, s), "tcgen05 q8_2f GEMM");
}

cq_status cq_gemm_q8b(const void* X, int xt, int64_t T, int64_t K, const int8_t* Wq, const float* Ws, int64_t N,
                      void* Y, int yt, void* ws, size_t ws_bytes, void* stream) {
    clear_last_error();
    if (!X || !Wq || !Ws || !Y || !ws) return fail(CQ_ERR_NULL, "cq_gemm_q8b: null pointer");
    cq_status st;
    if ((st = check_x(xt)) || (st = check_y(yt))) return st;
    if (T < 1 || N < 1 || K < 128 || K % 128 || T > (1LL << 31) - 1 || N > (1LL << 31) - 1)
        return fail(CQ_ERR_SHAPE, "cq_gemm_q8b: need T>=1, N>=1, K%%128==0 (T=%lld K=%lld N=%lld)", (long long)T,
                    (long long)K, (long long)N);
    if (!aligned16(X) || !aligned16(Wq) || !aligned16(Ws) || !aligned16(Y))
        return fail(CQ_ERR_ALIGN, "cq_gemm_q8b: pointers must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(ws) & (ALIGN - 1)) || ws_bytes < q4_ws_bytes(T, K))
        return fail(CQ_ERR_WORKSPACE, "cq_gemm_q8b: workspace needs %zu bytes, 256-aligned", q4_ws_bytes(T, K));
    if ((st = check_arch())) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = stream_error_word(s);
    if (!err) return CQ_ERR_CUDA;
    const uint8_t* q = reinterpret_cast<const uint8_t*>(Wq);
    if (use_skinny(T)) {   // the activations as given
        if (T > 32) return fail(CQ_ERR_ARG, "cq_gemm_q8b: the weight-streaming path serves T <= 32");
        SkinnyDense a = {X, xt == CQ_BF16 ? 1 : 0, nullptr, nullptr, q, nullptr, T, K, N, Y, yt, err};
        a.wsf = Ws;
        return launched(launch_skinny_q8b(a, s), "weight-streaming Q8/32 GEMM");
    }
    const Q4Ws w = q4_ws(ws, T, K);
    if ((st = launched(launch_x_col_half(X, xt, nullptr, T, K, w.xh, w.rsx, s), "Q8/32 activation guard pass"))) return st;
    TcArgs a = {w.xh, 0, w.rsx, nullptr, q, nullptr, T, K, N, Y, yt, err};
    a.wsf = Ws;
    return launched(launch_tc_q8b(a, s), "tcgen05 Q8/32 GEMM");
}

cq_status cq_gemm_q4a(const void* X, int xt, int64_t T, int64_t K, const uint8_t* Wq, const uint16_t* Ws,
                      const uint16_t* Wo, int64_t gk, int64_t N, void* Y, int yt, void* ws, size_t ws_bytes,
                      void* stream) {
    clear_last_error();
    if (!X || !Wq || !Ws || !Wo || !Y || !ws) return fail(CQ_ERR_NULL, "cq_gemm_q4a: null pointer");
    cq_status st;
    if ((st = check_x(xt)) || (st = check_y(yt))) return st;
    if (T < 1 || N < 1 || K < 256 || K % 256 || T > (1LL << 31) - 1 || N > (1LL << 31) - 1 || gk < 1 ||
        (K / 32) % gk || K / 32 / gk > 512)
        return fail(CQ_ERR_SHAPE, "cq_gemm_q4a: need T>=1, N>=1, K%%256==0, gk dividing K/32, K/32/gk <= 512 "
                    "(T=%lld K=%lld N=%lld gk=%lld)", (long long)T, (long long)K, (long long)N, (long long)gk);
    if (!aligned16(X) || !aligned16(Wq) || !aligned16(Ws) || !aligned16(Y) || (reinterpret_cast<uintptr_t>(Wo) & 1))
        return fail(CQ_ERR_ALIGN, "cq_gemm_q4a: X, Wq, Ws, Y must be 16-byte aligned, Wo 2-byte aligned");
    const size_t need = cq_gemm_q4a_workspace_bytes(T, K, N, gk);
    if ((reinterpret_cast<uintptr_t>(ws) & (ALIGN - 1)) || ws_bytes < need)
        return fail(CQ_ERR_WORKSPACE, "cq_gemm_q4a: workspace needs %zu bytes, 256-aligned", need);
    if ((st = check_arch())) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = stream_error_word(s);
    if (!err) return CQ_ERR_CUDA;
    uint8_t* b = static_cast<uint8_t*>(ws);
    const Q4Ws w = q4_ws(ws, T, K);
    float* xs = reinterpret_cast<float*>(b + q4_ws_bytes(T, K));
    float* add = reinterpret_cast<float*>(b + q4_ws_bytes(T, K) + up((size_t)T * (size_t)(K / 32 / gk) * 4));
    if (use_skinny(T)) {
        if (T > 32) return fail(CQ_ERR_ARG, "cq_gemm_q4a: the weight-streaming path serves T <= 32");
        // the offsets' term sum_g off[n][g] * (sum of X over group g), added by the GEMM's epilogue
        if ((st = launched(launch_offset_term(X, xt, T, K, Wo, (int)gk, N, xs, add, s), "affine Q4 offset term")))
            return st;
        SkinnyDense a = {X, xt == CQ_BF16 ? 1 : 0, nullptr, nullptr, Wq, Ws, T, K, N, Y, yt, err};
        a.add = add;
        return launched(launch_skinny_q4(a, s), "weight-streaming affine Q4 GEMM");
    }
    // tcgen05: the offsets join the weight decode, fp16((nibble - 8) * scale + offset) in one rounding
    if ((st = launched(launch_x_half(X, xt, T, K, w.xh, w.rsx, s), "activation guard pass"))) return st;
    TcArgs a = {w.xh, 0, w.rsx, nullptr, Wq, Ws, T, K, N, Y, yt, err};
    a.off = Wo;
    a.gk = (int)gk;
    return launched(launch_tc_q4a(a, s), "tcgen05 affine Q4 GEMM");
}

size_t cq_ffn_q4_workspace_bytes(int64_t T, int64_t H, int64_t I) {
    if (T < 1 || H < 1 || I < 1) return 0;
    return ffn_layout(T, H, I).total;
}

cq_status cq_ffn_q4(const void* X, int xt, int64_t T, int64_t H, int64_t I, const uint8_t* Wgu_q,
                    const uint16_t* Wgu_s, const uint8_t* Wd_q, const uint16_t* Wd_s, void* Y, int yt, void* ws,
                    size_t ws_bytes, void* stream) {
    clear_last_error();
    if (!X || !Wgu_q || !Wgu_s || !Wd_q || !Wd_s || !Y || !ws) return fail(CQ_ERR_NULL, "cq_ffn_q4: null pointer");
    cq_status st;
    if ((st = check_x(xt)) || (st = check_y(yt))) return st;
    if (T < 1 || H < 256 || H % 256 || I < 256 || I % 256 || T > (1LL << 31) - 1 || H > (1LL << 30) ||
        I > (1LL << 30))
        return fail(CQ_ERR_SHAPE, "cq_ffn_q4: need T>=1, H%%256==0, I%%256==0 (T=%lld H=%lld I=%lld)", (long long)T,
                    (long long)H, (long long)I);
    if (!aligned16(X) || !aligned16(Wgu_q) || !aligned16(Wgu_s) || !aligned16(Wd_q) || !aligned16(Wd_s) ||
        !aligned16(Y))
        return fail(CQ_ERR_ALIGN, "cq_ffn_q4: pointers must be 16-byte aligned");
    const FfnLayout l = ffn_layout(T, H, I);
    if ((reinterpret_cast<uintptr_t>(ws) & (ALIGN - 1)) || ws_bytes < l.total)
        return fail(CQ_ERR_WORKSPACE, "cq_ffn_q4: workspace needs %zu bytes, 256-aligned", l.total);
    if ((st = check_arch())) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = stream_error_word(s);
    if (!err) return CQ_ERR_CUDA;
    uint8_t* b = static_cast<uint8_t*>(ws);
    uint16_t* xh = reinterpret_cast<uint16_t*>(b + l.xh);
    float* rsx = reinterpret_cast<float*>(b + l.rsx);
    float* a = reinterpret_cast<float*>(b + l.a);
    uint16_t* ah = reinterpret_cast<uint16_t*>(b + l.ah);
    float* rsa = reinterpret_cast<float*>(b + l.rsa);
    if ((st = launched(launch_x_half(X, xt, T, H, xh, rsx, s), "FFN activation guard pass"))) return st;
    TcArgs g = {xh, 0, rsx, nullptr, Wgu_q, Wgu_s, T, H, I, a, CQ_F32, err};
    if ((st = launched(launch_tc_q4_gateup(g, s), "FFN gate/up GEMM + SwiGLU"))) return st;
    if ((st = launched(launch_a_half(a, T, I, ah, rsa, nullptr, s), "FFN SwiGLU guard pass"))) return st;
    TcArgs d = {ah, 0, rsa, nullptr, Wd_q, Wd_s, T, I, H, Y, yt, err};
    return launched(launch_tc_q4(d, s), "FFN down GEMM");
}

cq_status cq_moe_route(const float* logits, int64_t T, int64_t E, int64_t topk, int shared, int32_t* idx, float* w,
                       void* stream) {
    clear_last_error();
    if (!logits || !idx || !w) return fail(CQ_ERR_NULL, "cq_moe_route: null pointer");
    if (T < 1 || T > (1LL << 31) - 1 || E < 1 || E > 1024 || topk < 1 || topk > 64 || topk > E ||
        (shared != 0 && shared != 1))
        return fail(CQ_ERR_SHAPE, "cq_moe_route: need T>=1, 1<=E<=1024, 1<=topk<=min(E,64), shared 0 or 1 "
                    "(T=%lld E=%lld topk=%lld shared=%d)", (long long)T, (long long)E, (long long)topk, shared);
    if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(idx) | reinterpret_cast<uintptr_t>(w)) & 3)
        return fail(CQ_ERR_ALIGN, "cq_moe_route: pointers must be 4-byte aligned");
    cq_status st;
    if ((st = check_arch())) return st;
    return launched(launch_route_logits(logits, T, E, topk, shared, idx, w, static_cast<cudaStream_t>(stream)),
                    "MoE routing from logits");
}

cq_status cq_moe_layout(const void* ws, int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk, int32_t* perm_out,
                        int32_t* seg_out, void* stream) {
    clear_last_error();
    if (!ws || !perm_out || !seg_out) return fail(CQ_ERR_NULL, "cq_moe_layout: null pointer");
    if (T < 1 || topk < 1 || E < 1) return fail(CQ_ERR_SHAPE, "cq_moe_layout: bad shape");
    const MoeLayout l = moe_layout(T, H, I, E, topk);
    const uint8_t* b = static_cast<const uint8_t*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(perm_out, b + l.perm, (size_t)(T * topk) * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(seg_out, b + l.seg, (size_t)(E + 1) * 4, cudaMemcpyDeviceToDevice, s);
    return launched(e, "cq_moe_layout copy");
}

cq_status cq_dequant_q4(const uint8_t* Wq, const uint16_t* Ws, int64_t N, int64_t K, float* W, void* stream) {
    clear_last_error();
    if (!Wq || !Ws || !W) return fail(CQ_ERR_NULL, "cq_dequant_q4: null pointer");
    if (N < 1 || K < 32 || K % 32) return fail(CQ_ERR_SHAPE, "cq_dequant_q4: need N>=1, K%%32==0");
    if (!aligned16(Wq) || !aligned16(W)) return fail(CQ_ERR_ALIGN, "cq_dequant_q4: Wq and W must be 16-byte aligned");
    cq_status st;
    if ((st = check_arch())) return st;
    return launched(launch_dequant_q4(Wq, Ws, N, K, W, static_cast<cudaStream_t>(stream)), "dequant Q4");
}

cq_status cq_dequant_q8row(const int8_t* Wq, const float* rs, int64_t N, int64_t K, float* W, void* stream) {
    clear_last_error();
    if (!Wq || !rs || !W) return fail(CQ_ERR_NULL, "cq_dequant_q8row: null pointer");
    if (N < 1 || K < 1) return fail(CQ_ERR_SHAPE, "cq_dequant_q8row: need N>=1, K>=1");
    cq_status st;
    if ((st = check_arch())) return st;
    return launched(launch_dequant_q8row(Wq, rs, N, K, W, static_cast<cudaStream_t>(stream)), "dequant Q8-row");
}

cq_status cq_get_device_error(void* stream) {
    clear_last_error();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* word = stream_error_word(s);
    if (!word) return CQ_ERR_CUDA;
    // read, then clear, with copies ordered on this stream only
    int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, word, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(word, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the stream's device error word");
    if (v == DEV_INDEX) return fail(CQ_ERR_INDEX, "a routing index is outside [0, E)");
    if (v == DEV_TIMEOUT) return fail(CQ_ERR_TIMEOUT, "a device pipeline wait ran past its limit");
    return CQ_OK;
}

}  // extern "C"
