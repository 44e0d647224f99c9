/*
 * cq — matmul against block-quantized weights, dequantized on the fly, on
 * one GB300 (sm_103a).  C ABI of libcq.so.
 *
 * Weight formats
 *  - Q4 split plane.  Wq[N][K/2] bytes plus Ws[N][K/32] fp16 block scales.
 *    Block b of row n is the 16 bytes at n*K/2 + 16*b; byte i holds element
 *    32b+i in its low nibble and element 32b+16+i in its high nibble; an
 *    element decodes as (nibble - 8) * Ws[n][b].  ("oxinfer 0.0.5
 *    src/metal.rs", shader section "Dequantizers", struct Q4W and
 *    load(Q4W ...); restated by load(Q4_0W ...) on the same page.)
 *  - Q8-row.  Wq[N][K] int8 plus rs[N] f32; the row scale multiplies the
 *    f32 accumulator of each output row.  ("cortiq-engine 0.8.3
 *    src/gpu_metal/qi21.rs", module header on q8_row weights: integer
 *    weights exact in half precision, row scale in the epilogue.)
 *
 * Common conventions
 *  - Every pointer argument is a DEVICE pointer unless it says otherwise;
 *    `stream` is a cudaStream_t (NULL = the legacy default stream).
 *  - The caller owns every buffer.  No entry point allocates device memory
 *    or synchronises the stream (cq_get_device_error excepted); all work is
 *    enqueued on `stream`.  Scratch memory comes from the caller's
 *    workspace `ws` of `ws_bytes` bytes (size it with the *_workspace_bytes
 *    query; 256-byte aligned).
 *  - Row-major, densely packed tensors.  All pointers 16-byte aligned.
 *  - Errors found on the host (bad pointer, dtype, shape, alignment, short
 *    workspace) return a status before anything is enqueued and set a
 *    thread-local message (cq_last_error), in the style of the pages'
 *    "decline: <reason>" (cortiq-engine src/gpu_metal/qi21.rs, decline()).
 *    A failed launch returns CQ_ERR_CUDA.  Problems only the device can see
 *    (a routing index out of range, a pipeline wait that exceeded its time
 *    limit) set the device error word of the stream the call was enqueued
 *    on, which cq_get_device_error(stream) reports; the remaining kernels of
 *    that call do no work.  Each (device, stream) pair gets its own word on
 *    first use, from a fixed table of 1023 per device (further streams share
 *    one more word); a word is cleared when it is read.
 *  - Outputs are overwritten, never accumulated into.
 */
#ifndef CQ_H
#define CQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CQ_OK = 0,
    CQ_ERR_NULL = 1,        /* a required pointer is NULL */
    CQ_ERR_DTYPE = 2,       /* unsupported activation or output type */
    CQ_ERR_SHAPE = 3,       /* a size breaks the shape rules */
    CQ_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned */
    CQ_ERR_INDEX = 5,       /* a routing index outside [0, E) (device-detected) */
    CQ_ERR_WORKSPACE = 6,   /* workspace missing, short or misaligned */
    CQ_ERR_CUDA = 7,        /* a CUDA runtime call or launch failed */
    CQ_ERR_TIMEOUT = 8,     /* a device pipeline wait ran past its limit */
    CQ_ERR_ARCH = 9,        /* the current device is not sm_103 */
    CQ_ERR_ARG = 10         /* any other invalid argument */
} cq_status;

typedef enum { CQ_F16 = 0, CQ_BF16 = 1, CQ_F32 = 2 } cq_dtype;

/* ---------------------------------------------------------------------------
 * Q4 GEMM:  Y[T][N] = X[T][K] . dequant(Wq, Ws)[N][K]^T
 *
 * X: fp16 or bf16 (xt), [T][K].  Wq: [N][K/2] bytes.  Ws: fp16 bits
 * [N][K/32].  Y: f32 or bf16 (yt), [T][N], overwritten.
 * Shape rules: T >= 1, N >= 1, K >= 256 and K % 256 == 0.
 * Arithmetic, T > 32 (tcgen05 path): each activation row is scaled by a
 * power of two that puts its largest magnitude in [2^13, 2^14) and rounded
 * to fp16; each weight is (nibble - 8) * scale rounded once to fp16;
 * products accumulate in f32; the output is scaled back by the inverse
 * power of two and rounded once to yt.  (The guard follows "oxinfer 0.0.5
 * src/metal.rs", MMA_SHADER_SRC header and the x_half shader; the scale
 * folded into the half operand follows mma_tile on the same page.)
 * Arithmetic, T <= 32 (weight-streaming path): the activations as given
 * (fp16 or bf16, no guard); nibble - 8 is exact in either type, so every
 * product is exact in f32; the products of one 32-k block accumulate in f32
 * and are multiplied by the block scale into an f32 sum, rounded once to yt.
 * This path uses no workspace (the argument is still checked).
 * Workspace: cq_gemm_q4_workspace_bytes(T, K) bytes.
 * ------------------------------------------------------------------------- */
size_t cq_gemm_q4_workspace_bytes(int64_t T, int64_t K);
cq_status cq_gemm_q4(const void* X, int xt, int64_t T, int64_t K,
                     const uint8_t* Wq, const uint16_t* Ws, int64_t N,
                     void* Y, int yt, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Q4 GEMM without caller scratch:  the same result as cq_gemm_q4 (same
 * kernels, same arithmetic), for callers that cannot allocate device memory
 * or hand out a workspace -- for example a plugin inside a host framework
 * that owns every device allocation, a runtime whose memory budget is fixed
 * in advance, or a latency-critical loop that must not call cudaMalloc /
 * cudaFree (which can synchronise the device).  The pages have no
 * counterpart of this entry point.
 *
 * The guarded fp16 copy of X and its per-row scales live in one fixed array
 * of CQ_NOALLOC_SCRATCH_BYTES inside the library; every GPU that loads the
 * library holds it until the process exits.  Limit: round256(T*K*2) +
 * round256(T*4) <= CQ_NOALLOC_SCRATCH_BYTES, else CQ_ERR_SHAPE (use
 * cq_gemm_q4 with a workspace).  The entry point allocates nothing.
 * The first call on a device looks up the array's device address for that
 * device (with it current); make that first call before any stream capture.
 * Nothing in the array needs to start at zero.  All calls share the array
 * and it keeps the last call's contents, so calls that can overlap on the
 * GPU (different streams, different host threads on one device) race: order
 * them on one stream or serialise them.
 * Same arguments, shape rules and errors as cq_gemm_q4, without ws/ws_bytes.
 * ------------------------------------------------------------------------- */
#define CQ_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)
cq_status cq_gemm_q4_noalloc(const void* X, int xt, int64_t T, int64_t K,
                             const uint8_t* Wq, const uint16_t* Ws, int64_t N,
                             void* Y, int yt, void* stream);

/* ---------------------------------------------------------------------------
 * z-batched Q4 GEMM: up to four weights of one shape in one launch.
 *   for each job j < z:
 *     Y[t][y_off_j + n] = sum_k X[t][x_off_j + k] * dequant(Wq_j, Ws_j)[n][k]
 * The pages dispatch the tensors of one shape and codec that read one
 * activation buffer as one z-batched launch (the qkv GEMM with z = 3, the
 * gate/up GEMM with z = 2), each with its own activation and output offset:
 * "cortiq-engine 0.8.3 src/gpu_metal/qi21.rs", struct PMm (x_off[4],
 * y_off[4]) and Enc::gemm; "oxinfer 0.0.5 src/metal.rs", fn matmul_mma (jobs
 * sharing one guarded X).
 *
 * X: fp16/bf16 rows of pitch ldx elements ([T][ldx]).  jobs: HOST array of
 * z descriptors (the library reads it during the call only).  Each job's
 * Wq [N][K/2], Ws fp16 [N][K/32] as for cq_gemm_q4.  Y: f32 or bf16 rows of
 * pitch ldy ([T][ldy]); job j overwrites columns y_off_j .. y_off_j + N - 1
 * of every row and nothing else (the jobs' column ranges must not overlap).
 * Shape rules: 1 <= z <= 4, T >= 1, N >= 1, K % 256 == 0, ldx % 8 == 0,
 * x_off_j % 8 == 0, x_off_j + K <= ldx, y_off_j + N <= ldy; X, Y and every
 * weight pointer 16-byte aligned.  Arithmetic: as cq_gemm_q4 on each job
 * (T <= 32 the weight-streaming path, else tcgen05 behind one guard pass per
 * distinct x_off).
 * Workspace: cq_gemm_q4_batched_workspace_bytes(T, K, z) bytes.
 * ------------------------------------------------------------------------- */
typedef struct {
    const uint8_t* Wq;     /* [N][K/2] packed nibbles (device) */
    const uint16_t* Ws;    /* [N][K/32] fp16 block scales (device) */
    int64_t x_off;         /* first activation column of this job */
    int64_t y_off;         /* first output column of this job */
} cq_q4_job;
size_t cq_gemm_q4_batched_workspace_bytes(int64_t T, int64_t K, int z);
cq_status cq_gemm_q4_batched(const void* X, int xt, int64_t T, int64_t K, int64_t ldx,
                             const cq_q4_job* jobs, int z, int64_t N,
                             void* Y, int yt, int64_t ldy, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Format variants
 *
 * Q8 per 32-k block ("oxinfer 0.0.5 src/metal.rs", Dequantizers, struct Q8W
 * and load(Q8W ...)): Wq int8 [N][K], Ws f32 [N][K/32];
 *   W[n][k] = q[n][k] * Ws[n][k/32].
 *   T <= 32: the activations as given, int8 -> the activation type exactly,
 *   the block scale on the f32 result of its block; T > 32 (tcgen05): X to
 *   fp16 behind the per-row power-of-two guard, each weight q * fp16(scale)
 *   rounded once to fp16, f32 accumulation, the guard's inverse per token.
 *   Shape rules: T >= 1, N >= 1, K >= 128, K % 128 == 0.
 *
 * Affine Q4 ("oxinfer 0.0.5 src/metal.rs", Dequantizers, struct Q4A and
 * load(Q4A ...)): the Q4 split plane Wq, Ws plus Wo bf16 [N][K/32/gk], one
 * offset per group of gk blocks of 32;  W[n][k] = (nibble - 8) * scale +
 * Wo[n][(k/32)/gk].  Weight streaming (T <= 32): the Q4 GEMM plus the
 * offsets' term sum_g Wo[n][g] * (sum of X[t] over group g) (f32), added
 * before the output's rounding.  tcgen05 (T > 32): the offset joins the
 * decode, each weight fp16((nibble - 8) * scale + fp16(Wo)) with one
 * rounding (the bf16 offset reaches fp16 exactly in fp16's normal range), so
 * the decoded weights must lie in fp16's range, as for cq_gemm_q4.
 * Shape rules: as cq_gemm_q4, gk >= 1 dividing K/32, K/32/gk <= 512.
 *
 * q8_2f ("cortiq-engine 0.8.3 src/gpu_metal/qi21.rs", module header: int8
 * weights staged times the column field, the row scale in the epilogue; the
 * blob q[rows][cols], f16 rs[rows], f16 col[cols] of fn build_block):
 *   Y[t][n] = rs[n] * sum_k q[n][k] * col[k] * X[t][k]
 * rs f32 [N] and col f32 [K] (the stored f16 values widened exactly).  X
 * times the column field goes to fp16 behind the per-row guard; the Q8-row
 * kernels take it from there with the row scale and the guard's inverse.
 * Shape rules: as cq_gemm_q8row.
 *
 * Each takes a workspace of the size its *_workspace_bytes query returns.
 * ------------------------------------------------------------------------- */
size_t cq_gemm_q8b_workspace_bytes(int64_t T, int64_t K);
cq_status cq_gemm_q8b(const void* X, int xt, int64_t T, int64_t K, const int8_t* Wq, const float* Ws,
                      int64_t N, void* Y, int yt, void* ws, size_t ws_bytes, void* stream);
size_t cq_gemm_q4a_workspace_bytes(int64_t T, int64_t K, int64_t N, int64_t gk);
cq_status cq_gemm_q4a(const void* X, int xt, int64_t T, int64_t K, const uint8_t* Wq, const uint16_t* Ws,
                      const uint16_t* Wo, int64_t gk, int64_t N, void* Y, int yt, void* ws, size_t ws_bytes,
                      void* stream);
size_t cq_gemm_q8_2f_workspace_bytes(int64_t T, int64_t K);
cq_status cq_gemm_q8_2f(const void* X, int xt, int64_t T, int64_t K, const int8_t* Wq, const float* rs,
                        const float* col, int64_t N, void* Y, int yt, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Q8-row GEMM:  Y[T][N] = (X[T][K] . Wq[N][K]^T) * rs[N]
 *
 * X: fp16 or bf16 [T][K]; the int8 weights are converted exactly to the
 * same type, products accumulate in f32, rs[n] multiplies the accumulator
 * of output row n, one rounding to yt (f32 or bf16).
 * Shape rules: T >= 1, N >= 1, K >= 128 and K % 128 == 0.  No workspace.
 * ------------------------------------------------------------------------- */
cq_status cq_gemm_q8row(const void* X, int xt, int64_t T, int64_t K,
                        const int8_t* Wq, const float* rs, int64_t N,
                        void* Y, int yt, void* stream);

/* ---------------------------------------------------------------------------
 * Dense FFN chain (Q4):  Y[t] = Wd . (silu(Wg . x_t) * (Wu . x_t))
 *
 * The denoiser block's gate/up GEMM, SwiGLU and down GEMM as one call
 * ("cortiq-engine 0.8.3 src/gpu_metal/qi21.rs", fn blocks: gemm(TG, TU) ->
 * swiglu -> gemm(TD); gate and up fused into one [2I][H] weight as its
 * module header describes).  SwiGLU runs in the gate/up GEMM's epilogue.
 *
 * X: fp16/bf16 [T][H].  Wgu_q: [2I][H/2], Wgu_s: fp16 [2I][H/32] (rows
 * 0..I-1 gate, I..2I-1 up).  Wd_q: [H][I/2], Wd_s: fp16 [H][I/32].
 * Y: f32 or bf16 [T][H], overwritten.
 * Arithmetic: both GEMMs as the tcgen05 path of cq_gemm_q4 (guarded fp16
 * operands, f32 accumulation); a = g / (1 + exp(-g)) * u in f32, then a
 * guarded fp16 copy of a feeds the down GEMM.  Every T takes this path.
 * Shape rules: T >= 1, H >= 256, H % 256 == 0, I >= 256, I % 256 == 0.
 * Workspace: cq_ffn_q4_workspace_bytes(T, H, I) bytes (256-byte aligned).
 * ------------------------------------------------------------------------- */
size_t cq_ffn_q4_workspace_bytes(int64_t T, int64_t H, int64_t I);
cq_status cq_ffn_q4(const void* X, int xt, int64_t T, int64_t H, int64_t I,
                    const uint8_t* Wgu_q, const uint16_t* Wgu_s,
                    const uint8_t* Wd_q, const uint16_t* Wd_s,
                    void* Y, int yt, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Routed MoE expert panels (all experts Q4):
 *   for each token t and slot j < topk, e = idx[t][j]:
 *     g = Wgate[e] . x_t,  u = Wup[e] . x_t          (Wgu rows 0..I-1, I..2I-1)
 *     a = g / (1 + exp(-g)) * u                       (SwiGLU)
 *     Y[t] += w[t][j] * (Wd[e] . a)                   (Y starts at zero)
 * ("oxinfer 0.0.5 src/metal.rs": Backend::moe and the silu_half /
 *  moe_combine shaders; its tests module, mma_moe_matches_cpu, states the
 *  same chain in f64.)
 *
 * X: fp16/bf16 [T][H].  idx: int32 [T][topk].  w: f32 [T][topk].
 * Wgu_q: [E][2I][H/2], Wgu_s: fp16 [E][2I][H/32].
 * Wd_q:  [E][H][I/2],  Wd_s:  fp16 [E][H][I/32].
 * Y: f32 or bf16 [T][H], overwritten.
 * Routed pairs are grouped by expert (ascending), token order inside an
 * expert; each (t, j) is its own entry, so repeated experts in a row are
 * counted twice.  The j-sum per token runs in slot order (deterministic).
 * Shape rules: T >= 1, 1 <= topk <= 64, 1 <= E <= 1024, T*topk <= 65536,
 * H % 256 == 0, I % 256 == 0, 256 <= H <= 16384, I >= 256.
 * Workspace: cq_moe_workspace_bytes(T, H, I, E, topk) bytes.  After the
 * call completes, cq_moe_layout reads the routing layout kept there.
 * An index outside [0, E) sets CQ_ERR_INDEX on the device and leaves Y
 * untouched.
 * ------------------------------------------------------------------------- */
size_t cq_moe_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk);
cq_status cq_moe_panels(const void* X, int xt, int64_t T, int64_t H, int64_t E,
                        int64_t I, int64_t topk,
                        const int32_t* idx, const float* w,
                        const uint8_t* Wgu_q, const uint16_t* Wgu_s,
                        const uint8_t* Wd_q, const uint16_t* Wd_s,
                        void* Y, int yt, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Routing on the device, from the router logits, and the shared expert:
 *   idx[t][0..topk) = the topk experts with the largest logits, descending,
 *                     the lower index first on ties;
 *   w[t][j]         = p_e / sum of p over the picked experts, where
 *                     p = softmax of the row's E logits (computed in f32 as
 *                     exp(l - max) / its sum over the picked experts: the
 *                     softmax denominator cancels);
 *   shared = 1:       logits rows hold E + 1 values, the last one the shared
 *                     expert's gate g; slot topk is expert E with weight
 *                     1 / (1 + exp(-g)).
 * ("cortiq-engine 0.8.44 src/clover.rs": the coreset's top-k rule and the
 * route closure, p[e] / wsum; "cortiq-engine 0.8.41 src/gpu_metal/clover.rs",
 * fn run_on: the shared expert appended as one more slot of every row with
 * its sigmoid gate weight.)
 * logits: f32 [T][E + shared].  idx: int32 [T][topk + shared], w: f32
 * [T][topk + shared], written on `stream`; cq_moe_panels then takes them as
 * its idx and w with topk + shared slots, the shared expert stacked as
 * expert E of its weight arrays (E + 1 experts; every expert of one shape).
 * Shape rules: T >= 1, 1 <= E <= 1024, 1 <= topk <= min(E, 64), shared 0/1;
 * pointers 4-byte aligned.
 * ------------------------------------------------------------------------- */
cq_status cq_moe_route(const float* logits, int64_t T, int64_t E, int64_t topk, int shared,
                       int32_t* idx, float* w, void* stream);

/* Copies the routing layout of the last cq_moe_panels call on `ws` into
 * perm_out[T*topk] (pair ids t*topk + j in grouped order) and
 * seg_out[E+1] (exclusive prefix of per-expert pair counts), both device
 * int32 arrays, enqueued on `stream`. */
cq_status cq_moe_layout(const void* ws, int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk,
                        int32_t* perm_out, int32_t* seg_out, void* stream);

/* ---------------------------------------------------------------------------
 * Test hooks: the dequantized weights in f32 (bit-exact definitions).
 *  cq_dequant_q4:    W[n][k] = (nibble - 8) * f32(scale)   (exact)
 *  cq_dequant_q8row: W[n][k] = f32(q) * rs[n]              (one rounding)
 * Shape rules: N >= 1, K >= 32, K % 32 == 0 (Q4); K >= 1 (Q8).
 * ------------------------------------------------------------------------- */
cq_status cq_dequant_q4(const uint8_t* Wq, const uint16_t* Ws, int64_t N, int64_t K,
                        float* W, void* stream);
cq_status cq_dequant_q8row(const int8_t* Wq, const float* rs, int64_t N, int64_t K,
                           float* W, void* stream);

/* ---------------------------------------------------------------------------
 * Errors and options
 * ------------------------------------------------------------------------- */
/* Reads and clears the device error word of `stream` (on the current
 * device) with copies ordered on that stream, and synchronises that stream
 * only; returns CQ_OK, CQ_ERR_INDEX or CQ_ERR_TIMEOUT, or CQ_ERR_CUDA if a
 * copy or the synchronisation failed.  Errors of other streams stay where
 * they are. */
cq_status cq_get_device_error(void* stream);
/* The calling thread's last host-side error message ("" if none). */
const char* cq_last_error(void);
/* Kernel launches the calling thread's most recent library call issued
 * (0 if it declined before launching; a host-only call resets it to 0): the
 * number of kernel nodes such a call adds to a captured CUDA graph.  The
 * pages have no counterpart; it exists for callers that size graphs or
 * count launches. */
int cq_last_launches(void);

typedef enum {
    CQ_OPT_SMALL_T_MAX = 0,  /* largest T served by the weight-streaming path (default 32, max 32) */
    CQ_OPT_FORCE_PATH = 1,   /* 0 auto, 1 weight-streaming, 2 tensor-memory (tcgen05) path */
    CQ_OPT_WAIT_NS = 2,      /* time limit of every device pipeline wait, ns (default 1e9) */
    CQ_OPT_TEST_STALL = 3,   /* test only: 1 makes the next tcgen05 launch's loader issue nothing */
    CQ_OPT_TRACE = 4,        /* 1 prints the chosen path and grid of each call to stderr */
    CQ_OPT_TC_BN = 5,        /* tcgen05 token tile: 0 auto (default), or 32, 64, 128, 192 (CTA pairs only, no K split), 256 */
    CQ_OPT_TC_KSPLIT = 6,    /* tcgen05 K split over a 2-CTA cluster (partials exchanged in shared memory): 0 auto, 1, 2 */
    CQ_OPT_TC_AMODE = 7,     /* decoded weight operand of the tcgen05 MMA: 0 auto (tensor memory), 1 shared, 2 tensor memory
                                (affine Q4 and the gate/up GEMM: tensor memory always) */
    CQ_OPT_TC_PAIR = 8,      /* tcgen05 CTA pairs (neighbouring weight-row tiles share one 256-row MMA, each
                                CTA loading half of the activation tile; decoded weights in tensor memory, an
                                even number of row tiles): 2 on, 1 off, 0 auto (on wherever the row tiles
                                pair up) */
    CQ_OPT_STREAM_KERNEL = 9 /* weight-streaming kernel: 2 the row-partitioned kernel (one CTA per SM, each
                                streaming the whole K of an equal share of the weight rows) wherever it serves
                                (one job, K % 512 == 0, T <= 32; Q8/32: T <= 16), 1 the K-split cluster
                                kernel, 0 (default) the
                                row-partitioned kernel where it serves and every CTA holds 6 to 8 units of 8 rows
                                (on 152 SMs: 6081 <= N <= 9728; Q8 formats: T <= 16) or
                                N * K <= 2^19, else the K-split kernel */
} cq_option;
/* Process-wide: one value for every thread, stream and device (set before
 * the calls it should affect); reads and writes are atomic, so concurrent
 * callers see either the old or the new value.  Returns CQ_ERR_ARG for an
 * unknown option or value. */
cq_status cq_set_option(int option, int64_t value);
int64_t cq_get_option(int option);

/* Library version (major * 10000 + minor * 100 + patch). */
int cq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CQ_H */
