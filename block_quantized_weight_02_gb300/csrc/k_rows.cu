// Weight-streaming GEMM for up to 16 activation rows, partitioned by weight
// rows so that every SM streams the same number of weight bytes.
//
// The weight rows are cut into units of 8 (the N = 8 side of mma.sync
// m16n8k16: weights are the MMA's B operand, the activation rows its A
// operand, padded to 16), and the units are spread over one CTA per SM as
// evenly as integers allow (for N = 8192 on 148 SMs: 7 or 6 units, within
// 1.2 % of the mean).  Each CTA streams the whole K range of its rows, so no
// partial sums cross CTAs and nothing is reduced afterwards.  Inside a CTA,
// consumer warp w owns unit w of the current pass (eight units per pass) for
// every k-block, so no partial sums cross warps either.
//
// Stages of 512 k (Q4) or 256 k (Q8): for every unit of the pass two 8-row
// x 128-byte weight boxes (128-byte swizzle: 16-byte chunk j of row r at
// j ^ r) and, for the block-scaled formats, one 8-row box of scales; one box of
// the activations {64 k, 8 or 16 rows, stage / 64 slabs}.  Producer lane s
// issues every copy of the stages that land in ring slot s.
//
// Decode (lane c of a quad, row g of its warp's unit): Q4 word c of a 32-k
// block holds k = 4c .. 4c + 3 (low nibbles) and 16 + 4c .. (high nibbles);
// adjacent nibbles are paired, so the MMA's virtual k = 2c, 2c + 1, 2c + 8,
// 2c + 9 are the physical k = 4c .. 4c + 3 (first MMA) and 16 + 4c .. (second),
// and the activation operand of each MMA is one 8-byte run of a row.  Q8:
// words c and c + 4 of the block's 32 bytes give the same k.  Every product
// of the Q4 and Q8 decodes is exact (q - 8, or q, in the activation type); the
// block scale multiplies the f32 result of the block's two MMAs (Q4, Q8 per
// 32-k block), the Q8-row scale multiplies the finished sum.
//
// The CTA is small (288 threads, at most about 105 KB of shared memory) so
// that the next call's CTA can be resident beside it: launched with
// programmatic dependent launch, it requests the weights of its first ring
// fill before it waits for this kernel, and the activations after.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>

#include "cq_internal.h"
#include "cq_ptx.cuh"

namespace cq {
namespace {

constexpr int RW_CONS = 8;                    // consumer warps: one unit each per pass
constexpr int RW_PROD = RW_CONS;              // the producer warp
constexpr int RW_THREADS = (RW_CONS + 1) * 32;
constexpr int UNIT = 8;                       // weight rows per unit

struct RParams {
    int64_t N, K, T;
    int units;           // ceil(N / 8)
    int nst;             // stages over K
    const float* rs;     // Q8-row: row scales
    const float* add;    // nullable f32 [T][N] added before the rounding
    void* y;
    int yt;
    uint64_t wait_ns;
    int* err;
};

struct RMaps {
    CUtensorMap w;       // weights {K bytes, N}, box {128 B, 8 rows}
    CUtensorMap s;       // Q4: fp16 scales {K/32, N} box {16, 8}; Q8/32: f32 {K/32, N} box {8, 8}
    CUtensorMap x;       // activations {64, T, K/64}, box {64, TP, stage/64}
};

__device__ __forceinline__ uint32_t r_lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 r_lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 r_lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// Q4 word -> four adjacent-k pairs holding nibble - 8 exactly:
// d[0] = k (4c, 4c + 1), d[1] = (4c + 2, 4c + 3) from the low nibbles,
// d[2], d[3] the same from the high nibbles (k + 16).  bf16: 0x4300 | n is
// 128 + n, minus 136 gives n - 8; fp16: 0x6400 | n is 1024 + n, minus 1032, and
// 0x6400 | 16 n is 1024 + 16 n, times 1/16 minus 72.
template <int XBF>
__device__ __forceinline__ void q4_adjacent(uint32_t w, uint32_t d[4]) {
    if (XBF) {
        const uint32_t c43 = 0x43434343u, k136 = 0x43084308u;
        const uint32_t lo = and_mask<0x0F0F0F0Fu>(w), hi = and_mask<0x0F0F0F0Fu>(w >> 4);
        d[0] = sub_bf16x2(prmt(lo, c43, 0x4140u), k136);
        d[1] = sub_bf16x2(prmt(lo, c43, 0x4342u), k136);
        d[2] = sub_bf16x2(prmt(hi, c43, 0x4140u), k136);
        d[3] = sub_bf16x2(prmt(hi, c43, 0x4342u), k136);
    } else {
        const uint32_t c64 = 0x64646464u, k1032 = 0x64086408u, k16th = 0x2C002C00u, km72 = 0xD480D480u;
        const uint32_t lo = and_mask<0x0F0F0F0Fu>(w), hi = and_mask<0xF0F0F0F0u>(w);
        d[0] = sub_f16x2(prmt(lo, c64, 0x4140u), k1032);
        d[1] = sub_f16x2(prmt(lo, c64, 0x4342u), k1032);
        d[2] = fma_f16x2(prmt(hi, c64, 0x4140u), k16th, km72);
        d[3] = fma_f16x2(prmt(hi, c64, 0x4342u), k16th, km72);
    }
}
// int8 pair (bytes sel of w) -> exactly in the activation type.  fp16: (v ^ 0x80) | 0x6400 is
// 1024 + v + 128, minus 1152 is v.  bf16: with 0x43 as the high byte the low seven bits give
// 128 + (v & 127) and the sign bit 128 or 256; their difference is v.
template <int XBF>
__device__ __forceinline__ uint32_t i8_pair(uint32_t w, uint32_t sel) {
    if (XBF) {
        const uint32_t t = prmt(w, 0x43434343u, sel);
        return sub_bf16x2(and_mask<0xFF7FFF7Fu>(t), and_mask<0xFF80FF80u>(t));
    }
    return sub_f16x2(prmt(w ^ 0x80808080u, 0x64646464u, sel), 0x64806480u);
}
template <int XBF>
__device__ __forceinline__ void mma_f(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if (XBF) mma_16816_bf16(d, a, b0, b1);
    else mma_16816_f16(d, a, b0, b1);
}

template <int FMT>
struct RGeo {
    static constexpr int KSTAGE = FMT == 0 ? 512 : 256;       // k per stage
    static constexpr int BPS = KSTAGE / 32;                   // 32-k blocks per stage
    static constexpr int ROWB = FMT == 0 ? KSTAGE / 2 : KSTAGE;   // weight bytes per row and stage
    static constexpr int NBOX = ROWB / 128;                   // 128-byte boxes per unit and stage (2)
    static constexpr int W_BYTES = NBOX * RW_CONS * UNIT * 128;
    static constexpr int S_UNIT = FMT == 1 ? 0 : 256;         // scale box per unit (8 rows x 32 B)
    static constexpr int S_BYTES = RW_CONS * S_UNIT;
    static constexpr int XSL = KSTAGE / 64;                   // 64-k slabs per stage
};

template <int FMT, int TP>
struct RLayout {
    using G = RGeo<FMT>;
    static constexpr int X_BYTES = G::XSL * TP * 128;
    static constexpr int X_OFF = G::W_BYTES + G::S_BYTES;     // 1024-aligned
    static constexpr int SLOT = X_OFF + X_BYTES;
    static_assert(G::W_BYTES % 1024 == 0 && X_OFF % 1024 == 0 && SLOT % 1024 == 0, "1024-byte aligned boxes");
};

// FMT 0: Q4 (fp16 block scales), 1: Q8-row, 2: Q8 per 32-k block (f32 block scales).
// TP: activation rows of the MMA tile (8: rows g + 8 are zero; 16).  XBF: bf16 activations.
template <int FMT, int TP, int XBF, int NSLOT>
__global__ void __maxnreg__(112)
k_rows(const __grid_constant__ RMaps maps, const RParams p) {
    using G = RGeo<FMT>;
    using L = RLayout<FMT, TP>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NSLOT * L::SLOT);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(NSLOT + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * NSLOT);
    volatile int* never_flag = abort_flag + 1;   // stays 0: waits that must not be cut short

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    // this CTA's units (as even a split as integers allow) and its passes of eight
    const int u0 = (int)((int64_t)blockIdx.x * p.units / gridDim.x);
    const int u1 = (int)((int64_t)(blockIdx.x + 1) * p.units / gridDim.x);
    const int npass = (u1 - u0 + RW_CONS - 1) / RW_CONS;
    const int nst = p.nst;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), RW_CONS);
        }
        *abort_flag = 0;
        *never_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();   // the next kernel in the stream may be scheduled now

    if (warp == RW_PROD) {
        // ================= producer =================
        // Lane s owns ring slot s and issues every copy of the stages that land in it.
        if (lane < NSLOT) {
            const int s = lane;
            if (lane == 0) {
                tma_prefetch_desc(&maps.w);
                if (FMT != 1) tma_prefetch_desc(&maps.s);
                tma_prefetch_desc(&maps.x);
            }
            const uint32_t base = sb + (uint32_t)(s * L::SLOT);
            auto issue_w = [&](int pass, int i) {   // weights (and scales) of every unit of the pass
                const int ub = u0 + pass * RW_CONS, nu = min(RW_CONS, u1 - ub);
#pragma unroll 1
                for (int u = 0; u < nu; ++u) {
                    const int row = (ub + u) * UNIT;
#pragma unroll
                    for (int q = 0; q < G::NBOX; ++q)
                        tma_load_2d(base + (uint32_t)((q * RW_CONS + u) * UNIT * 128), &maps.w, full_bar(s),
                                    i * G::ROWB + q * 128, row);
                    if (FMT != 1)
                        tma_load_2d(base + (uint32_t)(G::W_BYTES + u * G::S_UNIT), &maps.s, full_bar(s),
                                    i * G::BPS, row);
                }
            };
            auto bytes_of = [&](int pass) {
                const int nu = min(RW_CONS, u1 - (u0 + pass * RW_CONS));
                return (uint32_t)(nu * (G::NBOX * UNIT * 128 + G::S_UNIT) + L::X_BYTES);
            };
            int gi_last = -1;
            bool ok = true;
            int gi = 0;
            for (int pass = 0; pass < npass && ok; ++pass) {
                for (int i = 0; i < nst; ++i, ++gi) {
                    if (gi % NSLOT != s) continue;
                    const int round = gi / NSLOT;
                    if (round > 0 && !mbar_wait(empty_bar(s), (uint32_t)((round - 1) & 1), p.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), bytes_of(pass));
                    issue_w(pass, i);
                    // weights are never written by this library: the first ring fill is requested
                    // before waiting for the previous kernel; the activations only after
                    if (gi < NSLOT) pdl_wait();
                    tma_load_3d(base + (uint32_t)L::X_OFF, &maps.x, full_bar(s), 0, 0, i * G::XSL);
                    gi_last = gi;
                }
            }
            if (gi_last < 0) pdl_wait();   // every path waits once, so later kernels stay ordered
            if (!ok) {
                *abort_flag = 1;
                atomicCAS(p.err, 0, DEV_TIMEOUT);
            }
            if (*abort_flag && gi_last >= 0)   // this lane's last copies land before the CTA may exit
                mbar_wait(full_bar(s), (uint32_t)((gi_last / NSLOT) & 1), p.wait_ns, never_flag);
        } else {
            pdl_wait();
        }
        __syncwarp();
        return;
    }

    // ================= consumers =================
    pdl_wait();   // outputs (and the previous kernel's readers of them) only after the previous kernel
    int gi = 0;
    for (int pass = 0; pass < npass; ++pass) {
        const int unit = u0 + pass * RW_CONS + warp;
        const bool active = unit < u1;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        bool ok = !*abort_flag;
        for (int i = 0; i < nst; ++i, ++gi) {
            const int slot = gi % NSLOT;
            if (ok && !mbar_wait(full_bar(slot), (uint32_t)((gi / NSLOT) & 1), p.wait_ns, abort_flag)) {
                ok = false;
                *abort_flag = 1;
                atomicCAS(p.err, 0, DEV_TIMEOUT);
            }
            if (ok && active) {
                const uint32_t sW = sb + (uint32_t)(slot * L::SLOT);
                const uint32_t sX = sW + (uint32_t)L::X_OFF;
                // this lane's weight rows g of the unit: 128-byte rows, chunk j at j ^ g
                const uint32_t wrow = sW + (uint32_t)((warp * UNIT + g) * 128 + 4 * c);
                // scales of rows 2c and 2c + 1 of the unit (C-fragment columns): 32 bytes per row,
                // loaded 16 bytes of each row at a time (8 Q4 blocks, or 4 Q8/32 blocks)
                const uint32_t srow = sW + (uint32_t)(G::W_BYTES + warp * G::S_UNIT + 2 * c * 32);
                uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
#pragma unroll
                for (int jb = 0; jb < G::BPS; ++jb) {
                    // activations: rows g (and g + 8), slab jb / 2, the 8-byte runs at k 4c (lo) and 16 + 4c (hi)
                    const uint32_t slab = (uint32_t)(jb >> 1);
                    const uint32_t clo = (uint32_t)(4 * (jb & 1) + (c >> 1)), off8 = 8u * (uint32_t)(c & 1);
                    const uint32_t xr = sX + (slab * TP + (uint32_t)g) * 128u + off8;
                    const uint2 lo = r_lds64(xr + ((clo ^ (uint32_t)g) << 4));
                    const uint2 hi = r_lds64(xr + (((clo + 2u) ^ (uint32_t)g) << 4));
                    uint2 lo8 = make_uint2(0u, 0u), hi8 = make_uint2(0u, 0u);
                    if (TP == 16) {
                        lo8 = r_lds64(xr + 8u * 128u + ((clo ^ (uint32_t)g) << 4));
                        hi8 = r_lds64(xr + 8u * 128u + (((clo + 2u) ^ (uint32_t)g) << 4));
                    }
                    const uint32_t a1[4] = {lo.x, lo8.x, lo.y, lo8.y};
                    const uint32_t a2[4] = {hi.x, hi8.x, hi.y, hi8.y};
                    uint32_t b[4];
                    if (FMT == 0) {
                        q4_adjacent<XBF>(r_lds32(wrow + (((uint32_t)((jb >> 3) * RW_CONS * UNIT * 128)) |
                                                        ((((uint32_t)(jb & 7) ^ (uint32_t)g)) << 4))), b);
                    } else {
                        const uint32_t rb = wrow + (uint32_t)((jb >> 2) * RW_CONS * UNIT * 128);
                        const uint32_t w0 = r_lds32(rb + ((((uint32_t)(2 * (jb & 3))) ^ (uint32_t)g) << 4));
                        const uint32_t w1 = r_lds32(rb + ((((uint32_t)(2 * (jb & 3) + 1)) ^ (uint32_t)g) << 4));
                        b[0] = i8_pair<XBF>(w0, 0x4140u);
                        b[1] = i8_pair<XBF>(w0, 0x4342u);
                        b[2] = i8_pair<XBF>(w1, 0x4140u);
                        b[3] = i8_pair<XBF>(w1, 0x4342u);
                    }
                    if (FMT == 1) {
                        mma_f<XBF>(acc, a1, b[0], b[1]);
                        mma_f<XBF>(acc, a2, b[2], b[3]);
                    } else {
                        float pb[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_f<XBF>(pb, a1, b[0], b[1]);
                        mma_f<XBF>(pb, a2, b[2], b[3]);
                        float sa, sbv;   // block jb's scales of rows 2c, 2c + 1
                        constexpr int PER16 = FMT == 0 ? 8 : 4;   // blocks per 16 bytes of scales
                        if (jb % PER16 == 0) {
                            v0 = r_lds128(srow + 16u * (uint32_t)(jb / PER16));
                            v1 = r_lds128(srow + 32u + 16u * (uint32_t)(jb / PER16));
                        }
                        if (FMT == 0) {
                            const int k = jb & 7;
                            const uint32_t x0 = (k >> 1) == 0 ? v0.x : (k >> 1) == 1 ? v0.y : (k >> 1) == 2 ? v0.z : v0.w;
                            const uint32_t x1 = (k >> 1) == 0 ? v1.x : (k >> 1) == 1 ? v1.y : (k >> 1) == 2 ? v1.z : v1.w;
                            sa = __half2float(__ushort_as_half((unsigned short)((k & 1) ? (x0 >> 16) : (x0 & 0xFFFFu))));
                            sbv = __half2float(__ushort_as_half((unsigned short)((k & 1) ? (x1 >> 16) : (x1 & 0xFFFFu))));
                        } else {
                            const int k = jb & 3;
                            sa = __uint_as_float(k == 0 ? v0.x : k == 1 ? v0.y : k == 2 ? v0.z : v0.w);
                            sbv = __uint_as_float(k == 0 ? v1.x : k == 1 ? v1.y : k == 2 ? v1.z : v1.w);
                        }
                        acc[0] = fmaf(sa, pb[0], acc[0]);
                        acc[1] = fmaf(sbv, pb[1], acc[1]);
                        if (TP == 16) {
                            acc[2] = fmaf(sa, pb[2], acc[2]);
                            acc[3] = fmaf(sbv, pb[3], acc[3]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(slot));
        }
        // ---- epilogue of this unit: (token g or g + 8, rows 2c and 2c + 1) ----
        if (ok && active && !*abort_flag) {
            const int64_t n = (int64_t)unit * UNIT + 2 * c;
            float sc0 = 1.f, sc1 = 1.f;
            if (FMT == 1) {
                if (n < p.N) sc0 = p.rs[n];
                if (n + 1 < p.N) sc1 = p.rs[n + 1];
            }
#pragma unroll
            for (int h = 0; h < (TP == 16 ? 2 : 1); ++h) {
                const int64_t t = g + 8 * h;
                if (t >= p.T) continue;
                float v0 = acc[2 * h] * sc0, v1 = acc[2 * h + 1] * sc1;
                if (p.add) {
                    if (n < p.N) v0 += p.add[t * p.N + n];
                    if (n + 1 < p.N) v1 += p.add[t * p.N + n + 1];
                }
                if (p.yt == CQ_F32) {
                    float* yr = reinterpret_cast<float*>(p.y) + t * p.N;
                    if (n + 1 < p.N && (p.N & 1) == 0) {
                        *reinterpret_cast<float2*>(yr + n) = make_float2(v0, v1);
                    } else {
                        if (n < p.N) yr[n] = v0;
                        if (n + 1 < p.N) yr[n + 1] = v1;
                    }
                } else {
                    __nv_bfloat16* yr = reinterpret_cast<__nv_bfloat16*>(p.y) + t * p.N;
                    if (n + 1 < p.N && (p.N & 1) == 0) {
                        *reinterpret_cast<__nv_bfloat162*>(yr + n) = __floats2bfloat162_rn(v0, v1);
                    } else {
                        if (n < p.N) yr[n] = __float2bfloat16_rn(v0);
                        if (n + 1 < p.N) yr[n + 1] = __float2bfloat16_rn(v1);
                    }
                }
            }
        }
    }
}

template <int FMT, int TP, int XBF, int NSLOT>
cudaError_t launch_rows_t(const RMaps& maps, const RParams& p, int grid, cudaStream_t s) {
    using L = RLayout<FMT, TP>;
    constexpr size_t smem = (size_t)NSLOT * L::SLOT + 2 * NSLOT * 8 + 16 + 1024;
    static_assert(smem <= 113 * 1024, "two CTAs per SM: the next call's CTA fits beside this one");
    auto kern = k_rows<FMT, TP, XBF, NSLOT>;
    static int configured_device = -1;   // attributes are per device; set once per instantiation
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(RW_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, maps, p);
}

template <int FMT, int XBF>
cudaError_t launch_rows_x(const RMaps& maps, const RParams& p, int grid, int64_t T, cudaStream_t s) {
    // ring depth: as many stages as fit beside the next call's CTA
    if (T <= 8) return launch_rows_t<FMT, 8, XBF, FMT == 0 ? 4 : 4>(maps, p, grid, s);
    return launch_rows_t<FMT, 16, XBF, FMT == 0 ? 3 : 4>(maps, p, grid, s);
}

}  // namespace

bool rows_path_serves(int fmt, int64_t T, int64_t K, int nz) {
    return nz <= 1 && T >= 1 && T <= 16 && K % (fmt == 0 ? 512 : 256) == 0;
}

cudaError_t launch_rows(int fmt, const SkinnyDense& a, cudaStream_t s) {
    constexpr int TPX = 16;   // the activation box spans the padded rows; TMA fills the ones past T with zeros
    const int64_t kstage = fmt == 0 ? 512 : 256;
    RParams p = {};
    p.N = a.N;
    p.K = a.K;
    p.T = a.T;
    p.units = (int)((a.N + UNIT - 1) / UNIT);
    p.nst = (int)(a.K / kstage);
    p.rs = a.rs;
    p.add = a.add;
    p.y = a.y;
    p.yt = a.yt;
    p.wait_ns = (uint64_t)options().wait_ns;
    p.err = a.err;
    RMaps maps;
    memset(&maps, 0, sizeof maps);
    const uint64_t kbytes = fmt == 0 ? (uint64_t)a.K / 2 : (uint64_t)a.K;
    {
        uint64_t d[2] = {kbytes, (uint64_t)a.N};
        uint64_t st[1] = {kbytes};
        uint32_t box[2] = {128, UNIT};
        if (!encode_tiled(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.wq, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (fmt == 0) {
        uint64_t d[2] = {(uint64_t)a.K / 32, (uint64_t)a.N};
        uint64_t st[1] = {(uint64_t)a.K / 32 * 2};
        uint32_t box[2] = {16, UNIT};
        if (!encode_tiled(&maps.s, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, a.ws, d, st, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else if (fmt == 2) {
        uint64_t d[2] = {(uint64_t)a.K / 32, (uint64_t)a.N};
        uint64_t st[1] = {(uint64_t)a.K / 32 * 4};
        uint32_t box[2] = {8, UNIT};
        if (!encode_tiled(&maps.s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.wsf, d, st, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    {
        // {64 elements, T rows, K/64 slabs} (strides K*2 B, 128 B): a box of TP rows x stage/64 slabs
        // lands as [slab][row][128 B], 128-byte swizzled
        const int tp = a.T <= 8 ? 8 : TPX;
        uint64_t d[3] = {64, (uint64_t)a.T, (uint64_t)a.K / 64};
        uint64_t st[2] = {(uint64_t)a.K * 2, 128};
        uint32_t box[3] = {64, (uint32_t)tp, (uint32_t)(kstage / 64)};
        if (!encode_tiled(&maps.x, a.x_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.x,
                          d, st, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    const int grid = (int)std::min<int64_t>((int64_t)num_sms(), p.units);
    if (options().trace)
        fprintf(stderr, "cq: rows fmt=%d T=%lld N=%lld K=%lld units=%d grid=%d\n", fmt, (long long)a.T,
                (long long)a.N, (long long)a.K, p.units, grid);
    if (fmt == 0) return a.x_bf16 ? launch_rows_x<0, 1>(maps, p, grid, a.T, s) : launch_rows_x<0, 0>(maps, p, grid, a.T, s);
    if (fmt == 1) return a.x_bf16 ? launch_rows_x<1, 1>(maps, p, grid, a.T, s) : launch_rows_x<1, 0>(maps, p, grid, a.T, s);
    return a.x_bf16 ? launch_rows_x<2, 1>(maps, p, grid, a.T, s) : launch_rows_x<2, 0>(maps, p, grid, a.T, s);
}

}  // namespace cq
