// Small kernels around the GEMMs: the dequantization test hooks, the
// activation guard pass (rows -> fp16 behind a power-of-two scale), the
// MoE routing layout and the SwiGLU-activation guard pass.  (The MoE
// combine runs inside the down panels, k_skinny.cu.)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cq_internal.h"
#include "cq_ptx.cuh"

namespace cq {

// Launch with a programmatic dependency on the previous kernel in the
// stream: the kernel may be scheduled while that one finishes, and waits for
// it (griddepcontrol.wait) before touching anything.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return counted(cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...));
}

// First writer wins: a later error of the same call does not replace the first.
__device__ __forceinline__ void set_err(int* err, int code) { atomicCAS(err, 0, code); }

// ---- dequantization hooks ---------------------------------------------
// Q4 ("oxinfer 0.0.5 src/metal.rs", Dequantizers / load(Q4W ...)): one
// thread per 32-element block; W = f32(nibble - 8) * f32(scale), one exact
// f32 product per element.
__global__ void k_dequant_q4(const uint8_t* __restrict__ wq, const uint16_t* __restrict__ ws, int64_t nblocks,
                             int64_t bpr, float* __restrict__ w) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nblocks) return;
    const int64_t n = i / bpr, b = i % bpr;
    const float d = __half2float(__ushort_as_half(ws[i]));
    const uint4 v = *reinterpret_cast<const uint4*>(wq + 16 * i);
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
    float* out = w + n * (bpr * 32) + b * 32;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t byte = (words[j >> 2] >> (8 * (j & 3))) & 0xFF;
        out[j] = __fmul_rn((float)((int)(byte & 15) - 8), d);
        out[16 + j] = __fmul_rn((float)((int)(byte >> 4) - 8), d);
    }
}

__global__ void k_dequant_q8row(const int8_t* __restrict__ wq, const float* __restrict__ rs, int64_t N, int64_t K,
                                float* __restrict__ w) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N * K) return;
    w[i] = __fmul_rn((float)wq[i], rs[i / K]);
}

cudaError_t launch_dequant_q4(const uint8_t* wq, const uint16_t* ws, int64_t N, int64_t K, float* w, cudaStream_t s) {
    const int64_t nb = N * (K / 32);
    k_dequant_q4<<<(unsigned)((nb + 255) / 256), 256, 0, s>>>(wq, ws, nb, K / 32, w);
    return counted(cudaGetLastError());
}

cudaError_t launch_dequant_q8row(const int8_t* wq, const float* rs, int64_t N, int64_t K, float* w, cudaStream_t s) {
    const int64_t n = N * K;
    k_dequant_q8row<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(wq, rs, N, K, w);
    return counted(cudaGetLastError());
}

// ---- power-of-two guard -------------------------------------------------
// A row whose largest magnitude is m is multiplied by 2^(14 - e), where
// m = f * 2^e with f in [0.5, 1), so that m lands in [2^13, 2^14) before
// the fp16 rounding; the inverse factor goes to the epilogue.  ("oxinfer
// 0.0.5 src/metal.rs", MMA_SHADER_SRC header, row_scale / x_half.)
__device__ __forceinline__ int guard_shift(float m) {
    if (!(m > 0.f) || !isfinite(m)) return 0;
    int e;
    frexpf(m, &e);
    int sh = 14 - e;
    return sh < -120 ? -120 : (sh > 120 ? 120 : sh);
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

__device__ __forceinline__ float block_max_256(float m, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) r = fmaxf(r, red[i]);
    return r;
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Order of the 16-bit activations inside each 32-k block for the Q4 GEMMs
// (both paths): position 8 wi + t holds k = 4 wi + TAU[t], TAU =
// {0, 2, 16, 18, 1, 3, 17, 19}.  Byte 4 wi + b of a packed Q4 block carries
// elements 4 wi + b (low nibble) and 16 + 4 wi + b (high nibble); masking a
// 32-bit word of four such bytes yields the pairs (b0, b2) and (b1, b3) of
// each nibble plane, and this order puts the matching activations of one
// word side by side (one 16-byte shared-memory load feeds two MMAs of the
// weight-streaming path; the tcgen05 path stores its decoded weights in the
// same order).  The contraction is the same sum in another order.
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// v: 32 scaled values of one block in k order -> four 16-byte chunks in stream order.
__device__ __forceinline__ void store_block_stream_order(const float* v, uint4* dst) {
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        const int b = 4 * wi;
        dst[wi] = make_uint4(pack_h2(v[b], v[b + 2]), pack_h2(v[16 + b], v[18 + b]), pack_h2(v[b + 1], v[b + 3]),
                             pack_h2(v[17 + b], v[19 + b]));
    }
}

// One row by one CTA of 256 threads; K % 32 == 0; the output is in the
// streaming order above, its inverse guard scale in *rs_out.
template <typename T>
__device__ __forceinline__ void guard_row(const T* __restrict__ xrow, int64_t K, __half* __restrict__ dst_row,
                                          float* __restrict__ rs_out, float* red) {
    const uint4* src = reinterpret_cast<const uint4*>(xrow);
    uint4* dst = reinterpret_cast<uint4*>(dst_row);
    const int64_t nblk = K / 32;
    const int tid = threadIdx.x;
    int sh;
    if (nblk <= 2 * 256) {
        // up to two 32-element blocks per thread: read once, kept in registers
        uint4 c[2][4];
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int64_t blk = tid + 256 * i;
            if (blk < nblk) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    c[i][q] = src[4 * blk + q];
                    const T* e = reinterpret_cast<const T*>(&c[i][q]);
#pragma unroll
                    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(to_f32<T>(e[j])));
                }
            }
        }
        m = block_max_256(m, red);
        sh = guard_shift(m);
        const float sc = pow2f(sh);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int64_t blk = tid + 256 * i;
            if (blk < nblk) {
                float v[32];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const T* e = reinterpret_cast<const T*>(&c[i][q]);
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[8 * q + j] = to_f32<T>(e[j]) * sc;
                }
                store_block_stream_order(v, dst + 4 * blk);
            }
        }
    } else {
        // longer rows: one pass for the maximum, one for the conversion
        const int64_t n8 = K / 8;
        float m = 0.f;
        for (int64_t i = tid; i < n8; i += 256) {
            uint4 v = src[i];
            const T* e = reinterpret_cast<const T*>(&v);
#pragma unroll
            for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(to_f32<T>(e[j])));
        }
        m = block_max_256(m, red);
        sh = guard_shift(m);
        const float sc = pow2f(sh);
        for (int64_t blk = tid; blk < nblk; blk += 256) {
            float v[32];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 u = src[4 * blk + q];
                const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
                for (int j = 0; j < 8; ++j) v[8 * q + j] = to_f32<T>(e[j]) * sc;
            }
            store_block_stream_order(v, dst + 4 * blk);
        }
    }
    if (threadIdx.x == 0) *rs_out = pow2f(-sh);
}

// One CTA of 256 threads per activation row.
template <typename T>
__global__ void __launch_bounds__(256) k_x_half(const T* __restrict__ x, int64_t K, int64_t ldx, __half* __restrict__ xh,
                                                float* __restrict__ rsx) {
    pdl_launch_dependents();   // the GEMM after this pass may start streaming its weights now
    pdl_wait();                // inputs ready and the previous readers of xh done
    __shared__ float red[8];
    const int64_t row = blockIdx.x;
    guard_row<T>(x + row * ldx, K, xh + row * K, rsx + row, red);
}

cudaError_t launch_x_half(const void* x, int xt, int64_t T, int64_t K, uint16_t* xh, float* rsx, cudaStream_t s,
                          int64_t ldx) {
    if (ldx <= 0) ldx = K;
    if (xt == CQ_BF16)
        return launch_pdl(k_x_half<__nv_bfloat16>, dim3((unsigned)T), dim3(256), 0, s,
                          reinterpret_cast<const __nv_bfloat16*>(x), K, ldx, reinterpret_cast<__half*>(xh), rsx);
    return launch_pdl(k_x_half<__half>, dim3((unsigned)T), dim3(256), 0, s, reinterpret_cast<const __half*>(x), K, ldx,
                      reinterpret_cast<__half*>(xh), rsx);
}

// ---- MoE routing layout -------------------------------------------------
// Routed (t, j) pairs grouped by expert, token order kept inside an expert
// ("oxinfer 0.0.5 src/metal.rs", Backend::moe: per-expert counts, segment
// starts, gathered sources filled in token order).  One CTA: shared-memory
// counts, a block scan for the segment starts and the active experts, and a
// stable rank inside each expert from a warp match on the expert index.
//   seg[e]   = number of pairs routed to experts below e  (seg[E] = P)
//   perm[q]  = pair id (t*topk + j) at grouped position q
//   inv[p]   = grouped position of pair p
//   status   = 0, or 1 if an index is outside [0, E) (nothing else written)
__device__ __forceinline__ void route_layout(const int32_t* __restrict__ idx, int P, int E, int32_t* __restrict__ seg,
                                             int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                             int32_t* __restrict__ act, int32_t* __restrict__ n_act,
                                             int32_t* __restrict__ status, int32_t* __restrict__ rb_cnt, int ncnt,
                                             int* __restrict__ err) {
    extern __shared__ int sh[];
    int* cnt = sh;            // [E] pairs per expert
    int* fill = sh + E;       // [E] next free grouped position of each expert
    __shared__ int bad;
    __shared__ int wsum[2][8];  // per-warp totals of the block scan (counts, active flags)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) bad = 0;
    for (int i = tid; i < ncnt; i += 256) rb_cnt[i] = 0;   // the down panels' row-block counters
    for (int e = tid; e < E; e += 256) cnt[e] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += 256) {
        const int e = idx[p];
        if (e < 0 || e >= E)
            bad = 1;
        else
            atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) {
            *status = 1;
            set_err(err, DEV_INDEX);
        }
        return;
    }
    // exclusive scans of cnt[e] and of [cnt[e] > 0] over the experts: thread tid owns the
    // contiguous experts [tid * per, (tid + 1) * per)
    const int per = (E + 255) / 256;
    const int e0 = tid * per;
    int lc = 0, la = 0;
    for (int i = 0; i < per; ++i) {
        const int e = e0 + i;
        if (e < E) {
            lc += cnt[e];
            la += cnt[e] > 0;
        }
    }
    int xc = lc, xa = la;      // inclusive warp scans
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yc = __shfl_up_sync(0xffffffffu, xc, o), ya = __shfl_up_sync(0xffffffffu, xa, o);
        if (lane >= o) {
            xc += yc;
            xa += ya;
        }
    }
    if (lane == 31) {
        wsum[0][warp] = xc;
        wsum[1][warp] = xa;
    }
    __syncthreads();
    int bc = 0, ba = 0;
    for (int w = 0; w < warp; ++w) {
        bc += wsum[0][w];
        ba += wsum[1][w];
    }
    int c = bc + xc - lc, na = ba + xa - la;   // exclusive prefixes at e0
    for (int i = 0; i < per; ++i) {
        const int e = e0 + i;
        if (e < E) {
            seg[e] = c;
            fill[e] = c;
            if (cnt[e] > 0) act[na++] = e;
            c += cnt[e];
        }
    }
    if (tid == 255) {
        seg[E] = c;      // = P
        *n_act = na;
    }
    __syncthreads();
    // stable positions: pairs in id order (t ascending, then j), 256 per chunk; inside a
    // chunk the warps take turns, and a warp ranks its lanes with a match on the expert
    for (int base = 0; base < P; base += 256) {
        const int p = base + tid;
        const int e = p < P ? idx[p] : -1;
        for (int w = 0; w < 8; ++w) {
            if (warp == w) {
                const unsigned peers = __match_any_sync(0xffffffffu, e);
                if (e >= 0) {
                    const int rank = __popc(peers & ((1u << lane) - 1u));
                    const int pos = fill[e] + rank;
                    perm[pos] = p;
                    inv[p] = pos;
                }
                __syncwarp();
                if (e >= 0 && (peers & ((1u << lane) - 1u)) == 0u) fill[e] += __popc(peers);
            }
            __syncthreads();
        }
    }
    if (tid == 0) *status = 0;
}

// Routing layout and gathered guard pass in one launch of P + 1 CTAs.  CTA P
// writes the layout (route_layout above).  CTA p < P guards the activation row
// of pair p = t * topk + j into its grouped position, which it finds from the
// indices alone: the pairs routed to lower experts plus the earlier pairs of
// its own expert (the same stable order as the layout).  With an index out of
// range anywhere, no CTA writes a row and the layout CTA reports it.
template <typename T>
__global__ void __launch_bounds__(256) k_moe_route_gather(const int32_t* __restrict__ idx, int P, int E, int topk,
                                                          int32_t* __restrict__ seg, int32_t* __restrict__ perm,
                                                          int32_t* __restrict__ inv, int32_t* __restrict__ act,
                                                          int32_t* __restrict__ n_act, int32_t* __restrict__ status,
                                                          int32_t* __restrict__ rb_cnt, int ncnt, int* __restrict__ err,
                                                          const T* __restrict__ x, int64_t H, __half* __restrict__ xh,
                                                          float* __restrict__ rsx) {
    pdl_launch_dependents();  // the gate/up panels may be scheduled (and stream weights) now
    pdl_wait();               // idx and x may come from the previous kernel; the previous call's readers are done
    if ((int)blockIdx.x == P) {
        route_layout(idx, P, E, seg, perm, inv, act, n_act, status, rb_cnt, ncnt, err);
        return;
    }
    __shared__ int s_below, s_before, s_bad;
    __shared__ float red[8];
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) {
        s_below = 0;
        s_before = 0;
        s_bad = 0;
    }
    __syncthreads();
    const int p = blockIdx.x;
    const int e = idx[p];
    int below = 0, before = 0, bad = 0;
    for (int q = tid; q < P; q += 256) {
        const int f = idx[q];
        bad |= (f < 0 || f >= E) ? 1 : 0;
        below += f < e ? 1 : 0;
        before += (f == e && q < p) ? 1 : 0;
    }
    below = __reduce_add_sync(0xffffffffu, below);
    before = __reduce_add_sync(0xffffffffu, before);
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) {
        atomicAdd(&s_below, below);
        atomicAdd(&s_before, before);
        atomicOr(&s_bad, bad);
    }
    __syncthreads();
    if (s_bad) return;
    const int pos = s_below + s_before;
    guard_row<T>(x + (int64_t)(p / topk) * H, H, xh + (int64_t)pos * H, rsx + pos, red);
}

cudaError_t launch_moe_route_gather(const int32_t* idx, int64_t T, int64_t topk, int64_t E, int32_t* seg,
                                    int32_t* perm, int32_t* inv, int32_t* act, int32_t* n_act, int32_t* status,
                                    int32_t* cnt, int ncnt, int* err, const void* x, int xt, int64_t H, uint16_t* xh,
                                    float* rsx, cudaStream_t s) {
    const size_t smem = (size_t)(2 * E) * sizeof(int);
    const int P = (int)(T * topk);
    if (xt == CQ_BF16)
        return launch_pdl(k_moe_route_gather<__nv_bfloat16>, dim3((unsigned)P + 1), dim3(256), smem, s, idx, P, (int)E,
                          (int)topk, seg, perm, inv, act, n_act, status, cnt, ncnt, err,
                          reinterpret_cast<const __nv_bfloat16*>(x), H, reinterpret_cast<__half*>(xh), rsx);
    return launch_pdl(k_moe_route_gather<__half>, dim3((unsigned)P + 1), dim3(256), smem, s, idx, P, (int)E, (int)topk,
                      seg, perm, inv, act, n_act, status, cnt, ncnt, err, reinterpret_cast<const __half*>(x), H,
                      reinterpret_cast<__half*>(xh), rsx);
}

// ---- format variants: activation pre-passes --------------------------------
// Activations times an optional column field (q8_2f: "cortiq-engine 0.8.3
// src/gpu_metal/qi21.rs", module header: int8 staged times the column field),
// to fp16 behind the same per-row power-of-two guard, in k order (the int8
// decoders produce k order).  One CTA of 256 threads per row, K % 8 == 0.
template <typename T>
__global__ void __launch_bounds__(256) k_x_col_half(const T* __restrict__ x, const float* __restrict__ col, int64_t K,
                                                    __half* __restrict__ xh, float* __restrict__ rsx) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float red[8];
    const int64_t row = blockIdx.x;
    const uint4* src = reinterpret_cast<const uint4*>(x + row * K);
    const int64_t n8 = K / 8;
    float m = 0.f;
    for (int64_t i = threadIdx.x; i < n8; i += 256) {
        const uint4 u = src[i];
        const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(to_f32<T>(e[j]) * (col ? col[8 * i + j] : 1.f)));
    }
    m = block_max_256(m, red);
    const int sh = guard_shift(m);
    const float sc = pow2f(sh);
    uint4* dst = reinterpret_cast<uint4*>(xh + row * K);
    for (int64_t i = threadIdx.x; i < n8; i += 256) {
        const uint4 u = src[i];
        const T* e = reinterpret_cast<const T*>(&u);
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = to_f32<T>(e[j]) * (col ? col[8 * i + j] : 1.f) * sc;
        dst[i] = make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]), pack_h2(v[6], v[7]));
    }
    if (threadIdx.x == 0) rsx[row] = pow2f(-sh);
}

cudaError_t launch_x_col_half(const void* x, int xt, const float* col, int64_t T, int64_t K, uint16_t* xh, float* rsx,
                              cudaStream_t s) {
    if (xt == CQ_BF16)
        return launch_pdl(k_x_col_half<__nv_bfloat16>, dim3((unsigned)T), dim3(256), 0, s,
                          reinterpret_cast<const __nv_bfloat16*>(x), col, K, reinterpret_cast<__half*>(xh), rsx);
    return launch_pdl(k_x_col_half<__half>, dim3((unsigned)T), dim3(256), 0, s, reinterpret_cast<const __half*>(x), col,
                      K, reinterpret_cast<__half*>(xh), rsx);
}

// Affine Q4 ("oxinfer 0.0.5 src/metal.rs", Dequantizers, load(Q4A ...)): every
// element of group g (gk blocks of 32) of row n carries the offset m[n][g], so
// the product with X has the term sum_g m[n][g] * xs[t][g], xs[t][g] the sum of
// X[t] over the group.  These two kernels form that term in f32; the Q4 GEMM's
// epilogue adds it before its final rounding.
// xs[t][g]: one warp per (t, g), f32 sum of the group's 32 gk activations.
template <typename T>
__global__ void __launch_bounds__(256) k_group_sums(const T* __restrict__ x, int64_t Tn, int64_t K, int gk,
                                                    float* __restrict__ xs) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t G = K / 32 / gk;
    const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (wid >= Tn * G) return;
    const int64_t t = wid / G, g = wid % G;
    const T* src = x + t * K + g * 32 * gk;
    float s = 0.f;
    for (int i = lane; i < 32 * gk; i += 32) s += to_f32<T>(src[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) xs[wid] = s;
}

// add[t][n] = sum_g m[n][g] * xs[t][g] (g in order, one fused multiply-add each): a
// CTA of 256 threads takes 32 RI rows n and 32 tokens t, the offsets and group sums
// staged through shared memory 32 groups at a time with coalesced loads; thread
// (tx, ty) computes rows tx + 32 i (i < RI) and tokens ty + 8 j (j < 4).  RI = 1
// where there are few tokens, so that the rows alone spread over enough CTAs.
template <int RI>
__global__ void __launch_bounds__(256) k_offset_term(const uint16_t* __restrict__ off, const float* __restrict__ xs,
                                                     int64_t Tn, int64_t N, int G, float* __restrict__ add) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float sm[32][129];   // [g][row]
    __shared__ float sx[32][33];    // [token][g]
    const int64_t n0 = (int64_t)blockIdx.x * (32 * RI), t0 = (int64_t)blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    float acc[RI][4];
#pragma unroll
    for (int i = 0; i < RI; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int g0 = 0; g0 < G; g0 += 32) {
        const int ng = G - g0 < 32 ? G - g0 : 32;
        // offsets: row r = e / 32, group e % 32 (a warp reads 32 consecutive groups of one row)
        for (int e = threadIdx.x; e < 32 * RI * 32; e += 256) {
            const int r = e >> 5, gg = e & 31;
            const int64_t n = n0 + r;
            sm[gg][r] = (gg < ng && n < N) ? __uint_as_float((uint32_t)off[n * G + g0 + gg] << 16) : 0.f;
        }
        for (int e = threadIdx.x; e < 32 * 32; e += 256) {
            const int t = e >> 5, gg = e & 31;
            sx[t][gg] = (gg < ng && t0 + t < Tn) ? xs[(t0 + t) * G + g0 + gg] : 0.f;
        }
        __syncthreads();
        for (int gg = 0; gg < ng; ++gg) {
            float m[RI], x[4];
#pragma unroll
            for (int i = 0; i < RI; ++i) m[i] = sm[gg][tx + 32 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] = sx[ty + 8 * j][gg];
#pragma unroll
            for (int i = 0; i < RI; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(m[i], x[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t t = t0 + ty + 8 * j;
        if (t >= Tn) continue;
#pragma unroll
        for (int i = 0; i < RI; ++i) {
            const int64_t n = n0 + tx + 32 * i;
            if (n < N) add[t * N + n] = acc[i][j];
        }
    }
}

cudaError_t launch_offset_term(const void* x, int xt, int64_t T, int64_t K, const uint16_t* off, int gk, int64_t N,
                               float* xs, float* add, cudaStream_t s) {
    const int64_t G = K / 32 / gk;
    const unsigned gs = (unsigned)((T * G + 7) / 8);
    cudaError_t e = xt == CQ_BF16
        ? launch_pdl(k_group_sums<__nv_bfloat16>, dim3(gs), dim3(256), 0, s, reinterpret_cast<const __nv_bfloat16*>(x),
                     T, K, gk, xs)
        : launch_pdl(k_group_sums<__half>, dim3(gs), dim3(256), 0, s, reinterpret_cast<const __half*>(x), T, K, gk, xs);
    if (e != cudaSuccess) return e;
    if (T <= 32)
        return launch_pdl(k_offset_term<1>, dim3((unsigned)((N + 31) / 32), 1u), dim3(256), 0, s, off, (const float*)xs, T,
                          N, (int)G, add);
    return launch_pdl(k_offset_term<4>, dim3((unsigned)((N + 127) / 128), (unsigned)((T + 31) / 32)), dim3(256), 0, s, off,
                      (const float*)xs, T, N, (int)G, add);
}

// ---- MoE routing from router logits ---------------------------------------
// One warp per token ("cortiq-engine 0.8.44 src/clover.rs": moe_route and the
// route closure; the shared expert's slot from "cortiq-engine 0.8.41
// src/gpu_metal/clover.rs", fn run_on).  The top-k experts are picked one at a
// time by a warp-wide argmax over the f32 logits not yet taken (ties: the lower
// index), which is the top-k by softmax probability because exp is increasing;
// lane l holds the logits l, l + 32, ... and a bit per held logit marks it
// taken.  Weights: w_j = exp(l_j - max) / sum over the picked experts of
// exp(l - max), in f32: the softmax's own denominator cancels in the
// renormalisation (p_e = exp(l_e - max) / sum_e' ..., w_j = p_j / sum p), so it
// is not formed.  With `shared`, slot topk is expert E with weight
// 1 / (1 + exp(-l[E])).
__global__ void __launch_bounds__(256) k_route_logits(const float* __restrict__ logits, int T, int E, int topk,
                                                      int shared, int32_t* __restrict__ idx, float* __restrict__ w) {
    pdl_launch_dependents();
    pdl_wait();
    const int t = (int)blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= T) return;
    const int ld = E + (shared ? 1 : 0), slots = topk + (shared ? 1 : 0);
    const float* l = logits + (int64_t)t * ld;
    const int per = (E + 31) / 32;
    uint32_t taken = 0;
    float mx = 0.f, wsum = 0.f, e0 = 0.f, e1 = 0.f;   // lane j keeps exp(l - max) of slots j and 32 + j
    for (int j = 0; j < topk; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = 0; i < per; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u)) {
                const float v = l[e];
                if (v > bv || (v == bv && e < bi)) {
                    bv = v;
                    bi = e;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (j == 0) mx = bv;                 // the first pick is the row's largest logit
        const float ev = expf(bv - mx);
        wsum += ev;
        if (lane == (j & 31)) {
            if (j < 32) e0 = ev;
            else e1 = ev;
        }
        if (lane == 0) idx[(int64_t)t * slots + j] = bi;
    }
    if (lane < topk) w[(int64_t)t * slots + lane] = e0 / wsum;
    if (lane + 32 < topk) w[(int64_t)t * slots + lane + 32] = e1 / wsum;
    if (shared && lane == 0) {
        idx[(int64_t)t * slots + topk] = E;
        w[(int64_t)t * slots + topk] = 1.0f / (1.0f + expf(-l[E]));
    }
}

cudaError_t launch_route_logits(const float* logits, int64_t T, int64_t E, int64_t topk, int shared, int32_t* idx,
                                float* w, cudaStream_t s) {
    return launch_pdl(k_route_logits, dim3((unsigned)((T + 7) / 8)), dim3(256), 0, s, logits, (int)T, (int)E,
                      (int)topk, shared, idx, w);
}

// SwiGLU activations (f32, grouped order) -> fp16 behind the same
// power-of-two guard as the inputs, in the weight-streaming order ("oxinfer 0.0.5 src/metal.rs",
// silu_half: scaled half rows and an inverse scale per row).
__global__ void __launch_bounds__(256) k_a_half(const float* __restrict__ a, int64_t I, __half* __restrict__ ah,
                                                float* __restrict__ rsa, const int32_t* __restrict__ status) {
    pdl_launch_dependents();
    pdl_wait();
    if (status && *status != 0) return;
    __shared__ float red[8];
    const int64_t row = blockIdx.x;
    const float4* src = reinterpret_cast<const float4*>(a + row * I);
    const int64_t n4 = I / 4;
    float m = 0.f;
    for (int64_t i = threadIdx.x; i < n4; i += 256) {
        float4 v = src[i];
        m = fmaxf(fmaxf(fmaxf(m, fabsf(v.x)), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    }
    m = block_max_256(m, red);
    const int sh = guard_shift(m);
    const float sc = pow2f(sh);
    // written in the weight-streaming GEMM's order inside each 32-k block (I % 32 == 0)
    uint4* dst = reinterpret_cast<uint4*>(ah + row * I);
    for (int64_t blk = threadIdx.x; blk < I / 32; blk += 256) {
        float v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 u = src[8 * blk + q];
            v[4 * q] = u.x * sc;
            v[4 * q + 1] = u.y * sc;
            v[4 * q + 2] = u.z * sc;
            v[4 * q + 3] = u.w * sc;
        }
        store_block_stream_order(v, dst + 4 * blk);
    }
    if (threadIdx.x == 0) rsa[row] = pow2f(-sh);
}

cudaError_t launch_a_half(const float* a, int64_t P, int64_t I, uint16_t* ah, float* rsa, const int32_t* status,
                          cudaStream_t s) {
    return launch_pdl(k_a_half, dim3((unsigned)P), dim3(256), 0, s, a, I, reinterpret_cast<__half*>(ah), rsa, status);
}

}  // namespace cq
