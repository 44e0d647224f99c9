// Weight-streaming GEMM for few activation rows (T <= 32) and the routed
// MoE expert panels.
//
// Y^T = W . X^T with the weight rows in the MMA's M dimension and the
// activation rows (tokens or routed pairs) in N, so a small T only narrows
// N.  One CTA owns 64 weight rows and a contiguous range of K:
//  - a producer warp streams the packed weights (and, for Q4, the fp16
//    block scales) into a shared-memory ring with TMA, one stage per
//    256 k (Q4) or 128 k (Q8), each stage tracked by full/empty mbarriers;
//  - eight consumer warps take the stages round-robin, decode the weights
//    from shared memory straight into mma.sync A fragments (Q4:
//    (nibble - 8) * scale rounded once to fp16; Q8: int8 converted exactly
//    to the activation type) and multiply with activation fragments read
//    from global memory (L1/L2 resident);
//  - the eight partial tiles are summed in a fixed order in shared memory,
//    and, when K is split across a thread-block cluster, the CTAs' partial
//    tiles are summed in rank order through distributed shared memory, so
//    results are deterministic.
// Inside a 128-k chunk the contraction order is permuted (the same way for
// weights and activations): each thread of a quad owns one 32-k block (Q4)
// or two 16-k runs (Q8), which makes every shared-memory read a
// conflict-free 16-byte load.  The sum is unchanged.
//
// Prior art on the pages: the 8-row expert panels ("cortiq-engine 0.8.41
// src/gpu_metal/clover.rs", q4tp_mul_mm_n8) and the 32-token MMA tiles for
// short inputs ("oxinfer 0.0.5 src/metal.rs", mma_tile with TM = 32).
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cq_internal.h"
#include "cq_ptx.cuh"

namespace cg = cooperative_groups;

namespace cq {

__device__ int g_err_skinny = 0;

int take_error_skinny() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_err_skinny, sizeof(int));
    cudaMemcpyToSymbol(g_err_skinny, &z, sizeof(int));
    return v;
}

namespace {

constexpr int RB = 64;           // weight rows per CTA (two TMA row boxes of 32)
constexpr int MT = 4;            // m16 tiles per consumer warp
constexpr int CONSUMERS = 8;     // consumer warps
constexpr int THREADS = (CONSUMERS + 1) * 32;
constexpr int BOX_BYTES = 32 * 64;  // one TMA box: 32 rows x 64 bytes

enum Mode { DENSE = 0, GATEUP = 1, DOWN = 2 };

struct Params {
    // weights: tensor maps over [E][R][Kbytes] (bytes) and [E][R][K/32] (fp16)
    int64_t K;
    int nst_total;        // stages over the whole K
    int ks;               // K split (cluster size)
    int64_t N;            // DENSE: output rows; MoE: rows of one expert matrix
    // activations
    const uint16_t* x;    // 16-bit activations, row stride K
    int64_t T;            // DENSE: activation rows
    const float* rsx;     // Q4 guard inverse scales per activation row (DENSE / GATEUP)
    const float* rs;      // Q8 row scales
    void* y;
    int yt;
    // MoE
    const int32_t* seg;
    const int32_t* perm;
    const int32_t* status;
    const float* w;       // routing weights by pair id
    const float* rsa;     // DOWN: guard inverse scale per grouped pair
    float* out;           // GATEUP: a [P][I]; DOWN: eo [P][H]
    int topk;
    int64_t I, H;
    uint64_t wait_ns;
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Two nibbles at bits 0-3 and 16-19 -> half2 (nibble - 8), exact:
// 0x6400 | n is the fp16 value 1024 + n; subtracting 1032 leaves n - 8.
__device__ __forceinline__ uint32_t nib2_to_h2(uint32_t v) {
    const uint32_t h = (v & 0x000F000Fu) | 0x64006400u;
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408)));
    return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, __half2 s) {
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), s);
    return *reinterpret_cast<const uint32_t*>(&r);
}

// int8 pair (bytes sel0, sel1 of w) -> half2 exactly: (v ^ 0x80) | 0x6400
// is 1024 + v + 128; subtracting 1152 leaves v.
__device__ __forceinline__ uint32_t i8x2_to_h2(uint32_t w, uint32_t sel) {
    const uint32_t h = prmt(w ^ 0x80808080u, 0x64646464u, sel);
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t i8x2_to_bf2(uint32_t w, int lo_byte) {
    const float a = (float)(int)(int8_t)((w >> (8 * lo_byte)) & 0xFF);
    const float b = (float)(int)(int8_t)((w >> (8 * (lo_byte + 1))) & 0xFF);
    const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&r);
}

template <int FMT>
struct StageGeo;
template <>
struct StageGeo<0> {                       // Q4: 256 k per stage
    static constexpr int KSTAGE = 256;
    static constexpr int W_BYTES = 4 * BOX_BYTES;     // [kh 2][rbox 2][32][64 B]
    static constexpr int S_BYTES = 2 * 32 * 16;       // [rbox 2][32][8 fp16]
    static constexpr int BYTES = W_BYTES + S_BYTES;
};
template <>
struct StageGeo<1> {                       // Q8: 128 k per stage
    static constexpr int KSTAGE = 128;
    static constexpr int W_BYTES = 4 * BOX_BYTES;     // [kh 2][rbox 2][32][64 B]
    static constexpr int S_BYTES = 0;
    static constexpr int BYTES = W_BYTES;
};

template <int FMT, int NT, int XBF, int MODE, int NSLOT>
__global__ void __launch_bounds__(THREADS, 1)
k_skinny(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS, const Params p) {
    using G = StageGeo<FMT>;
    constexpr int NCOL = 8 * NT;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int rb = blockIdx.y;
    const int expert = blockIdx.z;

    // ---- which columns (activation rows) this CTA serves ----
    int64_t ncols_total;
    int64_t col0 = 0;  // grouped-position base (MoE)
    if (MODE == DENSE) {
        ncols_total = p.T;
    } else {
        if (*p.status != 0) return;
        col0 = p.seg[expert];
        ncols_total = p.seg[expert + 1] - col0;
        if (ncols_total == 0) return;
    }
    const int ngroups = (int)((ncols_total + NCOL - 1) / NCOL);

    // ---- k range ----
    const int ks = MODE == DENSE ? (int)blockIdx.x : 0;
    const int st0 = (int)((int64_t)p.nst_total * ks / p.ks);
    const int st1 = (int)((int64_t)p.nst_total * (ks + 1) / p.ks);
    const int nst = st1 - st0;

    // ---- shared memory carve-up ----
    constexpr int RING = NSLOT * G::BYTES;
    constexpr int RED = CONSUMERS * RB * NCOL * 4;
    constexpr int RED_OFF = (MODE == DENSE) ? 0 : RING;
    constexpr int PART_OFF = (MODE == DENSE) ? (RING > RED ? RING : RED) : RING + RED;
    constexpr int BAR_OFF = PART_OFF + RB * NCOL * 4;
    float* red = reinterpret_cast<float*>(smem + RED_OFF);
    float* part = reinterpret_cast<float*>(smem + PART_OFF);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);  // full[NSLOT], empty[NSLOT]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * NSLOT);
    volatile int* never_flag = abort_flag + 1;  // stays 0: waits that must not be cut short

    const uint32_t smem_base = smem_u32(smem);
    const uint32_t bar_base = smem_u32(bars);
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (NSLOT + s); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        *abort_flag = 0;
        *never_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // rows of the two 32-row boxes
    int row_box[2];
    if (MODE == GATEUP) {
        row_box[0] = rb * 32;
        row_box[1] = (int)p.I + rb * 32;
    } else {
        row_box[0] = rb * RB;
        row_box[1] = rb * RB + 32;
    }

    if (warp == CONSUMERS) {
        // ================= producer =================
        if (lane == 0) {
            tma_prefetch_desc(&tmW);
            if (FMT == 0) tma_prefetch_desc(&tmS);
            int64_t issued = 0;
            bool ok = true;
            for (int grp = 0; grp < ngroups && ok; ++grp) {
                for (int i = 0; i < nst; ++i) {
                    const int64_t gi = (int64_t)grp * nst + i;
                    const int slot = (int)(gi % NSLOT);
                    const uint32_t par = (uint32_t)((gi / NSLOT) & 1);
                    if (!mbar_wait(empty_bar(slot), par ^ 1u, p.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sbase = smem_base + (uint32_t)(slot * G::BYTES);
                    mbar_arrive_expect_tx(full_bar(slot), (uint32_t)G::BYTES);
                    const int st = st0 + i;
                    for (int kh = 0; kh < 2; ++kh)
                        for (int bx = 0; bx < 2; ++bx)
                            tma_load_3d(sbase + (uint32_t)((kh * 2 + bx) * BOX_BYTES), &tmW, full_bar(slot),
                                        st * 128 + kh * 64, row_box[bx], expert);
                    if (FMT == 0)
                        for (int bx = 0; bx < 2; ++bx)
                            tma_load_3d(sbase + (uint32_t)(G::W_BYTES + bx * 512), &tmS, full_bar(slot), st * 8,
                                        row_box[bx], expert);
                    ++issued;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicCAS(&g_err_skinny, 0, DEV_TIMEOUT);
                // let copies already in flight land before the CTA can exit
                const int64_t first = issued > NSLOT ? issued - NSLOT : 0;
                for (int64_t gi = first; gi < issued; ++gi)
                    mbar_wait(full_bar((int)(gi % NSLOT)), (uint32_t)((gi / NSLOT) & 1), p.wait_ns, never_flag);
            }
        }
        __syncwarp();
    } else {
        // ================= consumers =================
        for (int grp = 0; grp < ngroups; ++grp) {
            const int64_t cbase = (int64_t)grp * NCOL;
            // activation row pointers for this thread's columns (col = 8*nt + g)
            const uint16_t* xrow[NT];
            bool xval[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int64_t col = cbase + 8 * nt + g;
                xval[nt] = col < ncols_total;
                int64_t r = 0;
                if (xval[nt]) {
                    if (MODE == DENSE) r = col;
                    else if (MODE == GATEUP) r = p.perm[col0 + col] / p.topk;
                    else r = col0 + col;
                }
                xrow[nt] = p.x + r * p.K;
            }
            float acc[MT][NT][4];
#pragma unroll
            for (int a = 0; a < MT; ++a)
#pragma unroll
                for (int b = 0; b < NT; ++b)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[a][b][q] = 0.f;

            bool ok = !*abort_flag;
            for (int i = warp; i < nst && ok; i += CONSUMERS) {
                const int64_t gi = (int64_t)grp * nst + i;
                const int slot = (int)(gi % NSLOT);
                if (!mbar_wait(full_bar(slot), (uint32_t)((gi / NSLOT) & 1), p.wait_ns, abort_flag)) {
                    ok = false;
                    *abort_flag = 1;
                    atomicCAS(&g_err_skinny, 0, DEV_TIMEOUT);
                    break;
                }
                const uint8_t* sW = smem + slot * G::BYTES;
                const int64_t kst = (int64_t)(st0 + i) * G::KSTAGE;
                if (FMT == 0) {
                    const __half* sS = reinterpret_cast<const __half*>(sW + G::W_BYTES);
#pragma unroll
                    for (int kh = 0; kh < 2; ++kh) {
                        const int64_t kc = kst + kh * 128;
                        uint32_t bw[NT][16];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            if (xval[nt]) {
                                const uint16_t* src = xrow[nt] + kc + 32 * c;
#pragma unroll
                                for (int v = 0; v < 4; ++v) {
                                    const uint4 q = ld_nc_v4(src + 8 * v);
                                    bw[nt][4 * v] = q.x; bw[nt][4 * v + 1] = q.y; bw[nt][4 * v + 2] = q.z; bw[nt][4 * v + 3] = q.w;
                                }
                            } else {
#pragma unroll
                                for (int v = 0; v < 16; ++v) bw[nt][v] = 0u;
                            }
                        }
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            const int bx = mt >> 1, lr = 16 * (mt & 1) + g;
                            const uint8_t* box = sW + (kh * 2 + bx) * BOX_BYTES;
                            const uint4 w0 = *reinterpret_cast<const uint4*>(box + lr * 64 + 16 * c);
                            const uint4 w1 = *reinterpret_cast<const uint4*>(box + (lr + 8) * 64 + 16 * c);
                            const __half s0 = sS[(bx * 32 + lr) * 8 + kh * 4 + c];
                            const __half s1 = sS[(bx * 32 + lr + 8) * 8 + kh * 4 + c];
                            const __half2 s0h = __halves2half2(s0, s0), s1h = __halves2half2(s1, s1);
                            const uint32_t r0[4] = {w0.x, w0.y, w0.z, w0.w};
                            const uint32_t r1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                            for (int s = 0; s < 4; ++s) {
                                const uint32_t p0 = prmt(r0[s], 0u, 0x3120u), p1 = prmt(r1[s], 0u, 0x3120u);
                                uint32_t alo[4], ahi[4];
                                alo[0] = hmul2_u32(nib2_to_h2(p0), s0h);
                                alo[1] = hmul2_u32(nib2_to_h2(p1), s1h);
                                alo[2] = hmul2_u32(nib2_to_h2(p0 >> 8), s0h);
                                alo[3] = hmul2_u32(nib2_to_h2(p1 >> 8), s1h);
                                ahi[0] = hmul2_u32(nib2_to_h2(p0 >> 4), s0h);
                                ahi[1] = hmul2_u32(nib2_to_h2(p1 >> 4), s1h);
                                ahi[2] = hmul2_u32(nib2_to_h2(p0 >> 12), s0h);
                                ahi[3] = hmul2_u32(nib2_to_h2(p1 >> 12), s1h);
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    mma_16816_f16(acc[mt][nt], alo, bw[nt][2 * s], bw[nt][2 * s + 1]);
                                    mma_16816_f16(acc[mt][nt], ahi, bw[nt][2 * s + 8], bw[nt][2 * s + 9]);
                                }
                            }
                        }
                    }
                } else {
                    const int64_t kc = kst;
                    uint32_t bw[NT][16];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (xval[nt]) {
                            const uint16_t* src = xrow[nt] + kc + 16 * c;
                            const uint4 q0 = ld_nc_v4(src), q1 = ld_nc_v4(src + 8);
                            const uint4 q2 = ld_nc_v4(src + 64), q3 = ld_nc_v4(src + 72);
                            bw[nt][0] = q0.x; bw[nt][1] = q0.y; bw[nt][2] = q0.z; bw[nt][3] = q0.w;
                            bw[nt][4] = q1.x; bw[nt][5] = q1.y; bw[nt][6] = q1.z; bw[nt][7] = q1.w;
                            bw[nt][8] = q2.x; bw[nt][9] = q2.y; bw[nt][10] = q2.z; bw[nt][11] = q2.w;
                            bw[nt][12] = q3.x; bw[nt][13] = q3.y; bw[nt][14] = q3.z; bw[nt][15] = q3.w;
                        } else {
#pragma unroll
                            for (int v = 0; v < 16; ++v) bw[nt][v] = 0u;
                        }
                    }
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        const int bx = mt >> 1, lr = 16 * (mt & 1) + g;
#pragma unroll
                        for (int kh = 0; kh < 2; ++kh) {
                            const uint8_t* box = sW + (kh * 2 + bx) * BOX_BYTES;
                            const uint4 w0 = *reinterpret_cast<const uint4*>(box + lr * 64 + 16 * c);
                            const uint4 w1 = *reinterpret_cast<const uint4*>(box + (lr + 8) * 64 + 16 * c);
                            const uint32_t r0[4] = {w0.x, w0.y, w0.z, w0.w};
                            const uint32_t r1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                            for (int s4 = 0; s4 < 4; ++s4) {
                                const int s = kh * 4 + s4;
                                uint32_t a[4];
                                if (XBF) {
                                    a[0] = i8x2_to_bf2(r0[s4], 0);
                                    a[1] = i8x2_to_bf2(r1[s4], 0);
                                    a[2] = i8x2_to_bf2(r0[s4], 2);
                                    a[3] = i8x2_to_bf2(r1[s4], 2);
                                } else {
                                    a[0] = i8x2_to_h2(r0[s4], 0x4140u);
                                    a[1] = i8x2_to_h2(r1[s4], 0x4140u);
                                    a[2] = i8x2_to_h2(r0[s4], 0x4342u);
                                    a[3] = i8x2_to_h2(r1[s4], 0x4342u);
                                }
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    if (XBF) mma_16816_bf16(acc[mt][nt], a, bw[nt][2 * s], bw[nt][2 * s + 1]);
                                    else mma_16816_f16(acc[mt][nt], a, bw[nt][2 * s], bw[nt][2 * s + 1]);
                                }
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(slot));
            }

            // ---- deterministic reduction over the consumer warps ----
            // (dense: red aliases the ring, so every warp must be done with it)
            if (MODE == DENSE) asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS * 32) : "memory");
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int r = 16 * mt + g, col = 8 * nt + 2 * c;
                    float* base = red + ((size_t)warp * RB) * NCOL;
                    base[r * NCOL + col] = acc[mt][nt][0];
                    base[r * NCOL + col + 1] = acc[mt][nt][1];
                    base[(r + 8) * NCOL + col] = acc[mt][nt][2];
                    base[(r + 8) * NCOL + col + 1] = acc[mt][nt][3];
                }
            asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS * 32) : "memory");
            for (int e = threadIdx.x; e < RB * NCOL; e += CONSUMERS * 32) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < CONSUMERS; ++w) s += red[(size_t)w * RB * NCOL + e];
                part[e] = s;
            }
            asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS * 32) : "memory");

            if (MODE != DENSE && !*abort_flag) {
                // MoE epilogues (single CTA per k range)
                if (MODE == GATEUP) {
                    // element (i, col): gate at local row i, up at local row 32 + i
                    for (int e = threadIdx.x; e < 32 * NCOL; e += CONSUMERS * 32) {
                        const int i = e & 31, col = e >> 5;
                        const int64_t q = cbase + col;
                        if (q >= ncols_total) continue;
                        const int64_t pos = col0 + q;
                        const int tok = p.perm[pos] / p.topk;
                        const float sc = p.rsx[tok];
                        const float gv = part[i * NCOL + col] * sc;
                        const float uv = part[(32 + i) * NCOL + col] * sc;
                        p.out[pos * p.I + (int64_t)rb * 32 + i] = gv / (1.0f + expf(-gv)) * uv;
                    }
                } else {
                    for (int e = threadIdx.x; e < RB * NCOL; e += CONSUMERS * 32) {
                        const int r = e & (RB - 1), col = e / RB;
                        const int64_t q = cbase + col;
                        if (q >= ncols_total) continue;
                        const int64_t pos = col0 + q;
                        const float v = part[r * NCOL + col] * p.rsa[pos] * p.w[p.perm[pos]];
                        p.out[pos * p.H + (int64_t)rb * RB + r] = v;
                    }
                }
                asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS * 32) : "memory");
            }
        }
    }

    if (MODE == DENSE) {
        // ---- sum the cluster's partial tiles in rank order, epilogue ----
        if (p.ks > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();
            const int rank = (int)cluster.block_rank();
            if (warp < CONSUMERS && !*abort_flag) {
                const int per = (RB * NCOL + p.ks - 1) / p.ks;
                const int lo = rank * per, hi = min(RB * NCOL, lo + per);
                for (int e = lo + threadIdx.x; e < hi; e += CONSUMERS * 32) {
                    const int r = e & (RB - 1), col = e / RB;
                    float s = 0.f;
                    for (int q = 0; q < p.ks; ++q) s += cluster.map_shared_rank(part, q)[r * NCOL + col];
                    const int64_t n = (int64_t)rb * RB + r, t = col;
                    if (n < p.N && t < p.T) {
                        const float v = s * (FMT == 0 ? p.rsx[t] : p.rs[n]);
                        if (p.yt == CQ_F32) reinterpret_cast<float*>(p.y)[t * p.N + n] = v;
                        else reinterpret_cast<__nv_bfloat16*>(p.y)[t * p.N + n] = __float2bfloat16_rn(v);
                    }
                }
            }
            cluster.sync();
        } else if (warp < CONSUMERS && !*abort_flag) {
            for (int e = threadIdx.x; e < RB * NCOL; e += CONSUMERS * 32) {
                const int r = e & (RB - 1), col = e / RB;
                const int64_t n = (int64_t)rb * RB + r, t = col;
                if (n < p.N && t < p.T) {
                    const float v = part[r * NCOL + col] * (FMT == 0 ? p.rsx[t] : p.rs[n]);
                    if (p.yt == CQ_F32) reinterpret_cast<float*>(p.y)[t * p.N + n] = v;
                    else reinterpret_cast<__nv_bfloat16*>(p.y)[t * p.N + n] = __float2bfloat16_rn(v);
                }
            }
        }
    }
}

template <int FMT, int NT, int XBF, int MODE, int NSLOT>
size_t smem_bytes() {
    using G = StageGeo<FMT>;
    constexpr int NCOL = 8 * NT;
    constexpr int RING = NSLOT * G::BYTES;
    constexpr int RED = CONSUMERS * RB * NCOL * 4;
    constexpr int PART_OFF = (MODE == DENSE) ? (RING > RED ? RING : RED) : RING + RED;
    return (size_t)PART_OFF + RB * NCOL * 4 + 2 * NSLOT * 8 + 16 + 1024;
}

bool make_maps(CUtensorMap* mw, CUtensorMap* ms, int fmt, const uint8_t* wq, const uint16_t* ws, int64_t R,
               int64_t K, int64_t E) {
    const uint64_t kbytes = fmt == 0 ? (uint64_t)K / 2 : (uint64_t)K;
    uint64_t dw[3] = {kbytes, (uint64_t)R, (uint64_t)E};
    uint64_t sw[2] = {kbytes, kbytes * (uint64_t)R};
    uint32_t bw[3] = {64, 32, 1};
    if (!encode_tiled(mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, wq, dw, sw, bw, CU_TENSOR_MAP_SWIZZLE_NONE)) return false;
    if (fmt == 0) {
        uint64_t ds[3] = {(uint64_t)K / 32, (uint64_t)R, (uint64_t)E};
        uint64_t ss[2] = {(uint64_t)K / 32 * 2, (uint64_t)K / 32 * 2 * (uint64_t)R};
        uint32_t bs[3] = {8, 32, 1};
        if (!encode_tiled(ms, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, ws, ds, ss, bs, CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
    } else {
        *ms = *mw;
    }
    return true;
}

template <int FMT, int NT, int XBF, int MODE, int NSLOT>
cudaError_t launch_t(const CUtensorMap& mw, const CUtensorMap& ms, const Params& p, dim3 grid, int cluster,
                     cudaStream_t s) {
    auto kern = k_skinny<FMT, NT, XBF, MODE, NSLOT>;
    const size_t smem = smem_bytes<FMT, NT, XBF, MODE, NSLOT>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mw, ms, p);
}

template <int FMT, int XBF>
cudaError_t launch_dense_nt(const CUtensorMap& mw, const CUtensorMap& ms, const Params& p, dim3 grid, int cluster,
                            int64_t T, cudaStream_t s) {
    if (T <= 8) return launch_t<FMT, 1, XBF, DENSE, 8>(mw, ms, p, grid, cluster, s);
    if (T <= 16) return launch_t<FMT, 2, XBF, DENSE, 8>(mw, ms, p, grid, cluster, s);
    return launch_t<FMT, 4, XBF, DENSE, 8>(mw, ms, p, grid, cluster, s);
}

cudaError_t launch_dense(int fmt, const SkinnyDense& a, cudaStream_t s) {
    CUtensorMap mw, ms;
    if (!make_maps(&mw, &ms, fmt, a.wq, a.ws, a.N, a.K, 1)) return cudaErrorInvalidValue;
    Params p = {};
    p.K = a.K;
    p.nst_total = (int)(a.K / (fmt == 0 ? 256 : 128));
    p.N = a.N;
    p.x = reinterpret_cast<const uint16_t*>(a.x);
    p.T = a.T;
    p.rsx = a.rsx;
    p.rs = a.rs;
    p.y = a.y;
    p.yt = a.yt;
    p.wait_ns = (uint64_t)options().wait_ns;
    const int64_t rbs = (a.N + RB - 1) / RB;
    int ks = 1;
    const int64_t cap = 2 * (int64_t)num_sms();
    for (int cand : {2, 4, 8})
        if (rbs * cand <= cap && p.nst_total / cand >= 2) ks = cand;
    p.ks = ks;
    dim3 grid((unsigned)ks, (unsigned)rbs, 1);
    if (options().trace)
        fprintf(stderr, "cq: skinny fmt=%d T=%lld N=%lld K=%lld grid=(%d,%lld) cluster=%d\n", fmt, (long long)a.T,
                (long long)a.N, (long long)a.K, ks, (long long)rbs, ks);
    if (fmt == 0) return launch_dense_nt<0, 0>(mw, ms, p, grid, ks, a.T, s);
    if (a.x_bf16) return launch_dense_nt<1, 1>(mw, ms, p, grid, ks, a.T, s);
    return launch_dense_nt<1, 0>(mw, ms, p, grid, ks, a.T, s);
}

}  // namespace

cudaError_t launch_skinny_q4(const SkinnyDense& a, cudaStream_t s) { return launch_dense(0, a, s); }
cudaError_t launch_skinny_q8(const SkinnyDense& a, cudaStream_t s) { return launch_dense(1, a, s); }

cudaError_t launch_moe_gateup(const SkinnyMoe& m, cudaStream_t s) {
    CUtensorMap mw, ms;
    if (!make_maps(&mw, &ms, 0, m.gu_q, m.gu_s, 2 * m.I, m.H, m.E)) return cudaErrorInvalidValue;
    Params p = {};
    p.K = m.H;
    p.nst_total = (int)(m.H / 256);
    p.ks = 1;
    p.N = 2 * m.I;
    p.x = m.xh;
    p.rsx = m.rsx;
    p.seg = m.seg;
    p.perm = m.perm;
    p.status = m.status;
    p.w = m.w;
    p.out = m.a;
    p.topk = (int)m.topk;
    p.I = m.I;
    p.H = m.H;
    p.wait_ns = (uint64_t)options().wait_ns;
    dim3 grid(1, (unsigned)(m.I / 32), (unsigned)m.E);
    return launch_t<0, 1, 0, GATEUP, 8>(mw, ms, p, grid, 1, s);
}

cudaError_t launch_moe_down(const SkinnyMoe& m, cudaStream_t s) {
    CUtensorMap mw, ms;
    if (!make_maps(&mw, &ms, 0, m.d_q, m.d_s, m.H, m.I, m.E)) return cudaErrorInvalidValue;
    Params p = {};
    p.K = m.I;
    p.nst_total = (int)(m.I / 256);
    p.ks = 1;
    p.N = m.H;
    p.x = m.ah;
    p.rsa = m.rsa;
    p.seg = m.seg;
    p.perm = m.perm;
    p.status = m.status;
    p.w = m.w;
    p.out = m.eo;
    p.topk = (int)m.topk;
    p.I = m.I;
    p.H = m.H;
    p.wait_ns = (uint64_t)options().wait_ns;
    dim3 grid(1, (unsigned)(m.H / RB), (unsigned)m.E);
    return launch_t<0, 1, 0, DOWN, 8>(mw, ms, p, grid, 1, s);
}

}  // namespace cq
