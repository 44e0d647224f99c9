// Host-side declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>
#include <cstddef>
#include <cstdio>

#include "../../include/cq.h"

namespace cq {

// Device error word values (shared by all kernels; first writer wins).
enum DevErr : int { DEV_OK = 0, DEV_INDEX = 1, DEV_TIMEOUT = 2 };

// Process-wide options (every thread and stream sees the same values); each
// field is read and written atomically.
struct Options {
    std::atomic<int64_t> small_t_max{32};
    std::atomic<int64_t> force_path{0};
    std::atomic<int64_t> wait_ns{1000000000LL};
    std::atomic<int64_t> test_stall{0};
    std::atomic<int64_t> trace{0};
    std::atomic<int64_t> tc_bn{0};
    std::atomic<int64_t> tc_ksplit{0};
    std::atomic<int64_t> tc_amode{0};
    std::atomic<int64_t> tc_pair{0};
    std::atomic<int64_t> stream_kernel{0};
};
Options& options();

// The device error word of a stream: one slot of a fixed table in device
// memory, assigned to the (device, stream) pair on first use.  Kernels set it
// (first writer wins) and cq_get_device_error(stream) reads and clears it with
// copies ordered on that stream only.  Returns nullptr (and sets the message)
// if the runtime fails.
int* stream_error_word(cudaStream_t s);

// Host error reporting (a thread-local "decline: ..." message).
cq_status fail(cq_status st, const char* fmt, ...);
void clear_last_error();   // start of an entry-point call: no message, no launches yet
// Counts a successful kernel launch of the current entry-point call (returns e).
cudaError_t counted(cudaError_t e);
int launches_so_far();
cq_status cuda_fail(cudaError_t e, const char* what);

// Tensor map encoding (driver entry point fetched through the runtime, so
// the library has no link-time dependency on libcuda).
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes /* rank-1 entries */, const uint32_t* box,
                  CUtensorMapSwizzle swz);

int num_sms();

// ---- launchers (one translation unit each) ------------------------------

// aux kernels
cudaError_t launch_dequant_q4(const uint8_t* wq, const uint16_t* ws, int64_t N, int64_t K, float* w, cudaStream_t s);
cudaError_t launch_dequant_q8row(const int8_t* wq, const float* rs, int64_t N, int64_t K, float* w, cudaStream_t s);
// X rows -> fp16 with a per-row power-of-two guard; rsx = inverse scales.
// Inside each 32-k block the output is in the Q4 streaming order (position
// 8 wi + t <- k = 4 wi + {0,2,16,18,1,3,17,19}[t]) that both Q4 GEMMs read.
// x rows of pitch ldx elements (0: K), 16-byte aligned.
cudaError_t launch_x_half(const void* x, int xt, int64_t T, int64_t K, uint16_t* xh, float* rsx, cudaStream_t s,
                          int64_t ldx = 0);
// MoE routing layout and gathered guard pass in one launch: the layout (counts,
// segment starts, stable grouping by expert, inverse map, active experts and
// their number, status) and, for every pair in grouped order, its token's row
// of x guarded into xh / rsx; also zeroes the down panels' per-row-block
// counters cnt[ncnt].  An index outside [0, E) sets status = 1 and the device
// error, and no row is written.
cudaError_t launch_moe_route_gather(const int32_t* idx, int64_t T, int64_t topk, int64_t E, int32_t* seg,
                                    int32_t* perm, int32_t* inv, int32_t* act, int32_t* n_act, int32_t* status,
                                    int32_t* cnt, int ncnt, int* err, const void* x, int xt, int64_t H, uint16_t* xh,
                                    float* rsx, cudaStream_t s);
// Activations times the column field col[K] (nullable: none) -> fp16 behind the
// per-row guard, in k order (q8_2f and the Q8 per-32-block tcgen05 path).
cudaError_t launch_x_col_half(const void* x, int xt, const float* col, int64_t T, int64_t K, uint16_t* xh, float* rsx,
                              cudaStream_t s);
// Affine Q4 offset term: xs[T][G] group sums of X, add[T][N] = off . xs^T (G = K/32/gk <= 512).
cudaError_t launch_offset_term(const void* x, int xt, int64_t T, int64_t K, const uint16_t* off, int gk, int64_t N,
                               float* xs, float* add, cudaStream_t s);
// Routing from router logits [T][E (+1 with shared)] -> idx, w [T][topk (+1)].
cudaError_t launch_route_logits(const float* logits, int64_t T, int64_t E, int64_t topk, int shared, int32_t* idx,
                                float* w, cudaStream_t s);
// f32 rows -> fp16 behind a per-row power-of-two guard, in the Q4 streaming
// order (the down panels and the tcgen05 Q4 GEMM read it); status nullable.
cudaError_t launch_a_half(const float* a, int64_t P, int64_t I, uint16_t* ah, float* rsa, const int32_t* status,
                          cudaStream_t s);

// Up to ZMAX weights of one shape in one launch (z-batched GEMM).
constexpr int ZMAX = 4;

// Weight-streaming (small-T) GEMM.  One job: the fields below; z-batched
// (nz > 1): job j takes its activations, weights, scales and output from
// more[j].  Activation rows have pitch ldx (0: K), output rows pitch ldy (0: N).
struct SkJob {
    const void* x;
    const float* rs;
    const uint8_t* wq;
    const uint16_t* ws;
    void* y;
};
struct SkinnyDense {
    const void* x;       // fp16/bf16 [T][K] as given (k order)
    int x_bf16;
    const float* rsx;    // unused (no guard on this path)
    const float* rs;     // Q8: row scales [N]
    const uint8_t* wq;   // Q4 nibbles / Q8 int8 bytes
    const uint16_t* ws;  // Q4 scales
    int64_t T, K, N;
    void* y;
    int yt;
    int* err;            // the stream's device error word
    int nz;
    SkJob more[ZMAX];
    int64_t ldx, ldy;
    const float* wsf;    // Q8 per 32-k block: f32 block scales [N][K/32] (single job)
    const float* add;    // nullable f32 [T][N] added before the output rounding (single job)
    SkJob job(int j) const { return nz > 1 ? more[j] : SkJob{x, rs, wq, ws, y}; }
    int jobs() const { return nz > 1 ? nz : 1; }
};
cudaError_t launch_skinny_q4(const SkinnyDense& a, cudaStream_t s);
cudaError_t launch_skinny_q8(const SkinnyDense& a, cudaStream_t s);    // rsx nullable: per-token scales (q8_2f)
cudaError_t launch_skinny_q8b(const SkinnyDense& a, cudaStream_t s);   // Q8 per 32-k block, activations as given
// Row-partitioned weight streaming (k_rows.cu) for T <= 32 (Q8/32: T <= 16), one job, K a
// multiple of the 512-k stage; fmt 0 Q4, 1 Q8-row, 2 Q8/32.
bool rows_path_serves(int fmt, int64_t T, int64_t K, int nz);
bool rows_path_preferred(int fmt, int64_t T, int64_t K, int64_t N, int nz);   // the default's choice
cudaError_t launch_rows(int fmt, const SkinnyDense& a, cudaStream_t s);

struct SkinnyMoe {
    const uint16_t* xh;     // [P][H] fp16 (guarded, streaming order), rows gathered into grouped order
    const float* rsx;       // [P]
    const uint16_t* ah;     // [P][I] fp16 (guarded, streaming order), grouped order
    const float* rsa;       // [P]
    const float* w;         // routing weights [T*topk] (pair id order)
    const int32_t* seg;     // [E+1]
    const int32_t* perm;    // [P] pair ids in grouped order
    const int32_t* status;  // non-zero: skip
    const int32_t* act;     // [E] active experts, ascending
    const int32_t* n_act;   // number of active experts
    const uint8_t *gu_q, *d_q;
    const uint16_t *gu_s, *d_s;
    float* a;               // [P][I] f32 SwiGLU output, grouped order
    float* eo;              // [P][H] f32 weighted expert outputs, grouped order
    int64_t T, H, I, E, topk;
    int* err;               // the stream's device error word
    const int32_t* inv;     // [P] grouped position of each pair id
    int32_t* cnt;           // [H / 128] down items finished per row block
    void* y;                // Y [T][H], f32 or bf16 (yt): written by the down panels' folded combine
    int yt;
};
cudaError_t launch_moe_gateup(const SkinnyMoe& m, cudaStream_t s);
cudaError_t launch_moe_down(const SkinnyMoe& m, cudaStream_t s);

// tcgen05 (large-T) GEMM.  One job: the fields below; z-batched (nz > 1):
// job j takes its activations, scales, weights and output from more[j].
struct TcJob {
    const void* x;
    const float* rsx;
    const float* rs;
    const uint8_t* wq;
    const uint16_t* ws;
    void* y;
    const float* wsf;    // Q8 per 32-k block: f32 block scales [N][K/32]
    const float* add;    // nullable f32 [T][N] added before the output rounding
};
struct TcArgs {
    const void* x;       // [T][K] fp16/bf16 (Q4: guarded fp16 in the streaming order)
    int x_bf16;
    const float* rsx;    // Q4
    const float* rs;     // Q8
    const uint8_t* wq;
    const uint16_t* ws;
    int64_t T, K, N;
    void* y;
    int yt;
    int* err;            // the stream's device error word
    int nz;              // z-batched: number of jobs in more[] (0 or 1: the single job above)
    TcJob more[ZMAX];
    int64_t ldy;         // output row pitch in elements (0: N)
    const float* wsf;    // single job: Q8/32 block scales
    const float* add;    // single job: addend
    const uint16_t* off; // affine Q4 (single job): offsets bf16 [N][K/32/gk], joined to the decode
    int gk;              // blocks per offset group
    TcJob job(int j) const { return nz > 1 ? more[j] : TcJob{x, rsx, rs, wq, ws, y, wsf, add}; }
    int jobs() const { return nz > 1 ? nz : 1; }
};
cudaError_t launch_tc_q4(const TcArgs& a, cudaStream_t s);
cudaError_t launch_tc_q4a(const TcArgs& a, cudaStream_t s);   // affine Q4: off, gk set, one job
cudaError_t launch_tc_q8(const TcArgs& a, cudaStream_t s);   // x fp16 or bf16; rsx nullable (q8_2f: the guard)
// Q8 per 32-k block: x guarded fp16 in k order, rsx its scales, wsf the f32 block scales.
cudaError_t launch_tc_q8b(const TcArgs& a, cudaStream_t s);
// Gate/up mode: wq is the Q4 [2I][K] gate|up matrix, N = I; y = a[T][I] f32,
// a = silu(gate) * up (x: guarded fp16 in the streaming order, rsx its scales).
cudaError_t launch_tc_q4_gateup(const TcArgs& a, cudaStream_t s);

}  // namespace cq
