// Weight-streaming GEMM for few activation rows (T <= 32) and the routed
// MoE expert panels.
//
// Y^T = W . X^T with the weight rows in the MMA's M dimension and the
// activation rows (tokens or routed pairs) in N, so a small T only narrows
// N.  One CTA owns 64 weight rows and a contiguous range of K:
//  - a producer warp streams the packed weights (and, for Q4, the fp16
//    block scales) and the matching slice of the activations (fp16/bf16,
//    128-byte swizzled) into a shared-memory ring with TMA, one stage per
//    256 k (Q4) or 128 k (Q8), each stage tracked by full/empty mbarriers;
//  - four consumer warps take the stages round-robin, decode the weights
//    from shared memory straight into mma.sync A fragments (Q4:
//    (nibble - 8) * scale rounded once to fp16; Q8: int8 converted exactly
//    to the activation type) and multiply with activation fragments read
//    from the same stage;
//  - the four partial tiles are summed in a fixed order in shared memory,
//    and, when K is split across a thread-block cluster, the CTAs' partial
//    tiles are summed in rank order through distributed shared memory, so
//    results are deterministic.
// Inside a stage the contraction order is permuted (the same way for weights
// and activations): thread c of a quad owns 32-k blocks 2c and 2c+1 (Q4) or
// 16-k runs 2c and 2c+1 (Q8), which with the 128-byte swizzles makes every
// shared-memory read a conflict-free 16-byte load.  The sum is unchanged.
//
// Prior art on the pages: the 8-row expert panels ("cortiq-engine 0.8.41
// src/gpu_metal/clover.rs", q4tp_mul_mm_n8) and the 32-token MMA tiles for
// short inputs ("oxinfer 0.0.5 src/metal.rs", mma_tile with TM = 32).
#include <algorithm>
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
constexpr int CONSUMERS = 4;     // consumer warps (two CTAs share an SM)
constexpr int THREADS = (CONSUMERS + 1) * 32;

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
    int pdl;              // launched with a programmatic dependency on the previous kernel
    const int32_t* act;   // MoE: active experts, ascending
    const int32_t* n_act; // MoE: number of active experts
    int rbs;              // MoE: row blocks per expert matrix
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
// int8 pair (bytes lo_byte, lo_byte+1 of w) -> bf16x2 exactly: 0x4B0000uu is
// the f32 2^23 + u with u = v + 128; subtracting 2^23 + 128 leaves v.
__device__ __forceinline__ uint32_t i8x2_to_bf2(uint32_t w, int lo_byte) {
    const uint32_t wx = w ^ 0x80808080u;
    const float a = __uint_as_float(prmt(wx, 0x4B000000u, 0x7440u + (uint32_t)lo_byte)) - 8388736.0f;
    const float b = __uint_as_float(prmt(wx, 0x4B000000u, 0x7441u + (uint32_t)lo_byte)) - 8388736.0f;
    const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&r);
}

// One stage in shared memory, filled by three TMA copies (five for gate/up):
//  W  [64 rows][128 B], 128-byte swizzle: 16-byte chunk j of row r at j ^ (r % 8)
//     (Q4: 256 k = eight 32-k blocks; Q8: 128 k = eight 16-k runs)
//  S  [64 rows][8 fp16] block scales (Q4 only)
//  X  [NCOL rows][XSL slabs of 64 k][128 B], 128-byte swizzle over the 3-D
//     view {64 elements, K/64 slabs, rows} of the activations.
template <int FMT, int NCOL>
struct StageGeo {
    static constexpr int KSTAGE = FMT == 0 ? 256 : 128;
    static constexpr int W_BYTES = RB * 128;
    static constexpr int S_BYTES = FMT == 0 ? RB * 16 : 0;
    static constexpr int XSL = KSTAGE / 64;            // 64-k slabs per stage
    static constexpr int X_OFF = W_BYTES + S_BYTES;    // 1024-aligned
    static constexpr int X_BYTES = NCOL * XSL * 128;
    static constexpr int BYTES = X_OFF + X_BYTES;
};

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

template <int FMT, int NT, int XBF, int MODE, int NSLOT>
__global__ void __launch_bounds__(THREADS, 2)
k_skinny(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
         const __grid_constant__ CUtensorMap tmX, const Params p) {
    constexpr int NCOL = 8 * NT;
    using G = StageGeo<FMT, NCOL>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    // ---- work items: (expert, row block) pairs; each may hold several column groups ----
    // dense: one item per CTA (row block blockIdx.y, k range blockIdx.x of the cluster);
    // MoE: a static round-robin share of (active expert x row block), so the
    // weight stream of one CTA continues across items without refilling.
    int nitems = 1, first = 0, stride = 1;
    if (MODE != DENSE) {
        pdl_wait();   // the routing layout and gathered rows come from the previous kernels
        if (*p.status != 0) return;
        nitems = *p.n_act * p.rbs;
        first = blockIdx.x;
        stride = gridDim.x;
        if (first >= nitems) return;
    }
    struct Item {
        int expert, rb;
        int64_t col0, ncols;
        int ngroups;
        int row_box[2];
    };
    auto get_item = [&](int idx) {
        Item it;
        if (MODE == DENSE) {
            it.expert = 0;
            it.rb = blockIdx.y;
            it.col0 = 0;
            it.ncols = p.T;
        } else {
            it.expert = p.act[idx / p.rbs];
            it.rb = idx % p.rbs;
            it.col0 = p.seg[it.expert];
            it.ncols = p.seg[it.expert + 1] - it.col0;
        }
        it.ngroups = (int)((it.ncols + NCOL - 1) / NCOL);
        if (MODE == GATEUP) {
            it.row_box[0] = it.rb * 32;
            it.row_box[1] = (int)p.I + it.rb * 32;
        } else {
            it.row_box[0] = it.rb * RB;
            it.row_box[1] = it.rb * RB + 32;
        }
        return it;
    };

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

    if (warp == CONSUMERS) {
        // ================= producers =================
        // Lane s owns ring slot s and issues every copy of the stages that land in it
        // (stage gi goes to slot gi % NSLOT): one thread keeps only a few bulk copies
        // outstanding, so the ring is filled from NSLOT threads.
        if (lane < NSLOT) {
            const int s = lane;
            if (lane == 0) {
                tma_prefetch_desc(&tmW);
                if (FMT == 0) tma_prefetch_desc(&tmS);
                tma_prefetch_desc(&tmX);
            }
            int64_t last_gi = -1;     // the last stage this lane issued
            bool ok = true;
            auto load_w = [&](const Item& it, int i) {
                const uint32_t sbase = smem_base + (uint32_t)(s * G::BYTES);
                const int st = st0 + i;
                if (MODE == GATEUP) {      // gate rows and up rows are 32-row boxes apart in the matrix
                    for (int bx = 0; bx < 2; ++bx) {
                        tma_load_3d(sbase + (uint32_t)(bx * 32 * 128), &tmW, full_bar(s), st * 128, it.row_box[bx],
                                    it.expert);
                        tma_load_3d(sbase + (uint32_t)(G::W_BYTES + bx * 32 * 16), &tmS, full_bar(s), st * 8,
                                    it.row_box[bx], it.expert);
                    }
                } else {
                    tma_load_3d(sbase, &tmW, full_bar(s), st * 128, it.row_box[0], it.expert);
                    if (FMT == 0) tma_load_3d(sbase + (uint32_t)G::W_BYTES, &tmS, full_bar(s), st * 8, it.row_box[0], it.expert);
                }
            };
            auto load_x = [&](const Item& it, int i, int grp) {
                const uint32_t sbase = smem_base + (uint32_t)(s * G::BYTES);
                const int st = st0 + i;
                // activation rows of this column group (dense: tokens; MoE: grouped pairs)
                const int xrow0 = (int)(it.col0 + (int64_t)grp * NCOL);
                tma_load_3d(sbase + (uint32_t)G::X_OFF, &tmX, full_bar(s), 0, st * G::XSL, xrow0);
            };
            // With a programmatic dependency (dense Q4: the activation guard pass runs just
            // before), the weights of the first ring fill are requested before waiting for
            // the activations; everything else follows the wait.
            const bool pre = MODE == DENSE && p.pdl && s < nst;
            if (MODE == DENSE) {
                if (pre) {                                   // fresh slot: no empty wait needed
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)G::BYTES);
                    load_w(get_item(0), s);
                }
                pdl_wait();
                if (pre) {
                    load_x(get_item(0), s, 0);
                    last_gi = s;
                }
            }
            int64_t gi = 0;
            for (int idx = first; idx < nitems && ok; idx += stride) {
                const Item it = get_item(idx);
                for (int grp = 0; grp < it.ngroups && ok; ++grp) {
                    for (int i = 0; i < nst; ++i, ++gi) {
                        if (gi % NSLOT != s || (pre && gi == s)) continue;
                        const uint32_t par = (uint32_t)((gi / NSLOT) & 1);
                        if (!mbar_wait(empty_bar(s), par ^ 1u, p.wait_ns, abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full_bar(s), (uint32_t)G::BYTES);
                        load_w(it, i);
                        load_x(it, i, grp);
                        last_gi = gi;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicCAS(&g_err_skinny, 0, DEV_TIMEOUT);
            }
            if (*abort_flag && last_gi >= 0)   // this lane's last copy must land before the CTA can exit
                mbar_wait(full_bar(s), (uint32_t)((last_gi / NSLOT) & 1), p.wait_ns, never_flag);
        }
        __syncwarp();
    } else {
        // ================= consumers =================
        int64_t gbase = 0;   // global index of the first stage of the current column group
        for (int idx = first; idx < nitems; idx += stride) {
          const Item it = get_item(idx);
          const int64_t col0 = it.col0, ncols_total = it.ncols;
          const int rb = it.rb;
          for (int grp = 0; grp < it.ngroups; ++grp, gbase += nst) {
            const int64_t cbase = (int64_t)grp * NCOL;
            float acc[MT][NT][4];
#pragma unroll
            for (int a = 0; a < MT; ++a)
#pragma unroll
                for (int b = 0; b < NT; ++b)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[a][b][q] = 0.f;

            bool ok = !*abort_flag;
            // Stage gi goes to warp gi % CONSUMERS and slot gi % NSLOT; NSLOT is a multiple of
            // CONSUMERS, so each slot always belongs to one warp, which then waits for the
            // slot's rounds in order (a parity wait cannot tell round r+1 from round r-1).
            for (int i = (int)((warp - gbase % CONSUMERS + CONSUMERS) % CONSUMERS); i < nst && ok; i += CONSUMERS) {
                const int64_t gi = gbase + i;
                const int slot = (int)(gi % NSLOT);
                if (!mbar_wait(full_bar(slot), (uint32_t)((gi / NSLOT) & 1), p.wait_ns, abort_flag)) {
                    ok = false;
                    *abort_flag = 1;
                    atomicCAS(&g_err_skinny, 0, DEV_TIMEOUT);
                    break;
                }
                const uint8_t* sW = smem + slot * G::BYTES;
                const uint8_t* sX = sW + G::X_OFF;
                if (FMT == 0) {
                    const __half* sS = reinterpret_cast<const __half*>(sW + G::W_BYTES);
#pragma unroll
                    for (int kh = 0; kh < 2; ++kh) {
                        // this thread's 32-k block j = 2c + kh: weight chunk j of each row, and
                        // activations k = 32 j .. 32 j + 31 = slab c, bytes 64 kh .. 64 kh + 63
                        const int j = 2 * c + kh;
#pragma unroll
                        for (int sp = 0; sp < 2; ++sp) {
                            // words 4sp..4sp+3 (low-nibble steps 2sp, 2sp+1) and 8+4sp.. (high-nibble steps)
                            uint4 blo[NT], bhi[NT];
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const int row = 8 * nt + g;
                                const uint8_t* xr = sX + row * (G::XSL * 128) + c * 128;
                                const int sw = (G::XSL * row + c) & 7;
                                blo[nt] = lds128(xr + (((4 * kh + sp) ^ sw) << 4));
                                bhi[nt] = lds128(xr + (((4 * kh + 2 + sp) ^ sw) << 4));
                            }
#pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                const int lr = 16 * mt + g;
                                const uint4 wa = lds128(sW + lr * 128 + ((j ^ (lr & 7)) << 4));
                                const uint4 wb = lds128(sW + (lr + 8) * 128 + ((j ^ ((lr + 8) & 7)) << 4));
                                const __half s0 = sS[lr * 8 + j];
                                const __half s1 = sS[(lr + 8) * 8 + j];
                                const __half2 sa = __halves2half2(s0, s0), sb2 = __halves2half2(s1, s1);
                                const uint32_t r0[4] = {wa.x, wa.y, wa.z, wa.w};
                                const uint32_t r1[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                                for (int u = 0; u < 2; ++u) {
                                    const int st4 = 2 * sp + u;
                                    const uint32_t p0 = prmt(r0[st4], 0u, 0x3120u), p1 = prmt(r1[st4], 0u, 0x3120u);
                                    uint32_t alo[4], ahi[4];
                                    alo[0] = hmul2_u32(nib2_to_h2(p0), sa);
                                    alo[1] = hmul2_u32(nib2_to_h2(p1), sb2);
                                    alo[2] = hmul2_u32(nib2_to_h2(p0 >> 8), sa);
                                    alo[3] = hmul2_u32(nib2_to_h2(p1 >> 8), sb2);
                                    ahi[0] = hmul2_u32(nib2_to_h2(p0 >> 4), sa);
                                    ahi[1] = hmul2_u32(nib2_to_h2(p1 >> 4), sb2);
                                    ahi[2] = hmul2_u32(nib2_to_h2(p0 >> 12), sa);
                                    ahi[3] = hmul2_u32(nib2_to_h2(p1 >> 12), sb2);
#pragma unroll
                                    for (int nt = 0; nt < NT; ++nt) {
                                        const uint32_t l0 = u ? blo[nt].z : blo[nt].x, l1 = u ? blo[nt].w : blo[nt].y;
                                        const uint32_t h0 = u ? bhi[nt].z : bhi[nt].x, h1 = u ? bhi[nt].w : bhi[nt].y;
                                        mma_16816_f16(acc[mt][nt], alo, l0, l1);
                                        mma_16816_f16(acc[mt][nt], ahi, h0, h1);
                                    }
                                }
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int kh = 0; kh < 2; ++kh) {
                        // this thread's 16-k run j = 2c + kh: weight chunk j of each row, and
                        // activations k = 16 j .. 16 j + 15 = slab j / 4, 32 bytes at 32 (j % 4)
                        const int j = 2 * c + kh;
                        const int slab = j >> 2;
                        uint4 b0[NT], b1[NT];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const int row = 8 * nt + g;
                            const uint8_t* xr = sX + row * (G::XSL * 128) + slab * 128;
                            const int sw = (G::XSL * row + slab) & 7;
                            b0[nt] = lds128(xr + (((2 * (j & 3)) ^ sw) << 4));
                            b1[nt] = lds128(xr + (((2 * (j & 3) + 1) ^ sw) << 4));
                        }
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            const int lr = 16 * mt + g;
                            const uint4 w0 = lds128(sW + lr * 128 + ((j ^ (lr & 7)) << 4));
                            const uint4 w1 = lds128(sW + (lr + 8) * 128 + ((j ^ ((lr + 8) & 7)) << 4));
                            const uint32_t r0[4] = {w0.x, w0.y, w0.z, w0.w};
                            const uint32_t r1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                            for (int s4 = 0; s4 < 4; ++s4) {
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
                                    // words 2 s4, 2 s4 + 1 of the 16-k run
                                    const uint4& bb = s4 < 2 ? b0[nt] : b1[nt];
                                    const uint32_t x0 = (s4 & 1) ? bb.z : bb.x, x1 = (s4 & 1) ? bb.w : bb.y;
                                    if (XBF) mma_16816_bf16(acc[mt][nt], a, x0, x1);
                                    else mma_16816_f16(acc[mt][nt], a, x0, x1);
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
                        const float sc = p.rsx[pos];
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
    }

    if (MODE == DENSE) {
        const int rb = blockIdx.y;
        pdl_wait();   // outputs and guard scales only after the previous kernel has finished
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
constexpr size_t smem_bytes() {
    constexpr int NCOL = 8 * NT;
    using G = StageGeo<FMT, NCOL>;
    constexpr int RING = NSLOT * G::BYTES;
    constexpr int RED = CONSUMERS * RB * NCOL * 4;
    constexpr int PART_OFF = (MODE == DENSE) ? (RING > RED ? RING : RED) : RING + RED;
    return (size_t)PART_OFF + RB * NCOL * 4 + 2 * NSLOT * 8 + 16 + 1024;
}

// Weights [E][R][K bytes] and scales [E][R][K/32], boxes of rows_box rows.
bool make_maps(CUtensorMap* mw, CUtensorMap* ms, int fmt, const uint8_t* wq, const uint16_t* ws, int64_t R,
               int64_t K, int64_t E, int rows_box) {
    const uint64_t kbytes = fmt == 0 ? (uint64_t)K / 2 : (uint64_t)K;
    uint64_t dw[3] = {kbytes, (uint64_t)R, (uint64_t)E};
    uint64_t sw[2] = {kbytes, kbytes * (uint64_t)R};
    uint32_t bw[3] = {128, (uint32_t)rows_box, 1};
    if (!encode_tiled(mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, wq, dw, sw, bw, CU_TENSOR_MAP_SWIZZLE_128B)) return false;
    if (fmt == 0) {
        uint64_t ds[3] = {(uint64_t)K / 32, (uint64_t)R, (uint64_t)E};
        uint64_t ss[2] = {(uint64_t)K / 32 * 2, (uint64_t)K / 32 * 2 * (uint64_t)R};
        uint32_t bs[3] = {8, (uint32_t)rows_box, 1};
        if (!encode_tiled(ms, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, ws, ds, ss, bs, CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
    } else {
        *ms = *mw;
    }
    return true;
}

// Activations [rows][K] 16-bit seen as {64 elements, K/64 slabs, rows}; one box
// is xsl slabs of ncol rows, stored [row][slab][128 B] with the 128-byte swizzle.
bool make_xmap(CUtensorMap* mx, const void* x, int64_t rows, int64_t K, int bf16, int ncol, int xsl) {
    uint64_t d[3] = {64, (uint64_t)K / 64, (uint64_t)rows};
    uint64_t st[2] = {128, (uint64_t)K * 2};
    uint32_t box[3] = {64, (uint32_t)xsl, (uint32_t)ncol};
    return encode_tiled(mx, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, x, d, st,
                        box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int FMT, int NT, int XBF, int MODE, int NSLOT>
cudaError_t launch_t(const CUtensorMap& mw, const CUtensorMap& ms, const void* x, int64_t xrows, const Params& p,
                     dim3 grid, int cluster, cudaStream_t s) {
    CUtensorMap mx;
    if (!make_xmap(&mx, x, xrows, p.K, XBF, 8 * NT, StageGeo<FMT, 8 * NT>::XSL)) return cudaErrorInvalidValue;
    auto kern = k_skinny<FMT, NT, XBF, MODE, NSLOT>;
    constexpr size_t smem = smem_bytes<FMT, NT, XBF, MODE, NSLOT>();
    static_assert(smem <= 113 * 1024, "two CTAs per SM");
    static_assert(NSLOT % CONSUMERS == 0, "each ring slot is consumed by one warp");
    static int configured_device = -1;       // attributes are per device; set once per instantiation
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
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, mw, ms, mx, p);
}

template <int FMT, int XBF>
cudaError_t launch_dense_nt(const CUtensorMap& mw, const CUtensorMap& ms, const void* x, const Params& p, dim3 grid,
                            int cluster, int64_t T, cudaStream_t s) {
    constexpr int S1 = 8, S2 = FMT == 0 ? 4 : 8, S4 = 4;
    if (T <= 8) return launch_t<FMT, 1, XBF, DENSE, S1>(mw, ms, x, T, p, grid, cluster, s);
    if (T <= 16) return launch_t<FMT, 2, XBF, DENSE, S2>(mw, ms, x, T, p, grid, cluster, s);
    return launch_t<FMT, 4, XBF, DENSE, S4>(mw, ms, x, T, p, grid, cluster, s);
}

cudaError_t launch_dense(int fmt, const SkinnyDense& a, cudaStream_t s) {
    CUtensorMap mw, ms;
    if (!make_maps(&mw, &ms, fmt, a.wq, a.ws, a.N, a.K, 1, RB)) return cudaErrorInvalidValue;
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
    p.pdl = fmt == 0 ? 1 : 0;     // Q4: the guard pass just before touches neither weights nor Y
    const int64_t rbs = (a.N + RB - 1) / RB;
    int ks = 1;
    const int64_t cap = 2 * (int64_t)num_sms();      // two CTAs fit per SM
    for (int cand : {2, 4, 8})
        if (rbs * cand <= cap && p.nst_total / cand >= 2) ks = cand;
    p.ks = ks;
    dim3 grid((unsigned)ks, (unsigned)rbs, 1);
    if (options().trace)
        fprintf(stderr, "cq: skinny fmt=%d T=%lld N=%lld K=%lld grid=(%d,%lld) cluster=%d\n", fmt, (long long)a.T,
                (long long)a.N, (long long)a.K, ks, (long long)rbs, ks);
    if (fmt == 0) return launch_dense_nt<0, 0>(mw, ms, a.x, p, grid, ks, a.T, s);
    if (a.x_bf16) return launch_dense_nt<1, 1>(mw, ms, a.x, p, grid, ks, a.T, s);
    return launch_dense_nt<1, 0>(mw, ms, a.x, p, grid, ks, a.T, s);
}

}  // namespace

cudaError_t launch_skinny_q4(const SkinnyDense& a, cudaStream_t s) { return launch_dense(0, a, s); }
cudaError_t launch_skinny_q8(const SkinnyDense& a, cudaStream_t s) { return launch_dense(1, a, s); }

// Gate/up panels: activations are the guarded rows already gathered into
// grouped order ([P][H] fp16, inverse scales [P]).
cudaError_t launch_moe_gateup(const SkinnyMoe& m, cudaStream_t s) {
    CUtensorMap mw, ms;
    if (!make_maps(&mw, &ms, 0, m.gu_q, m.gu_s, 2 * m.I, m.H, m.E, 32)) return cudaErrorInvalidValue;
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
    p.act = m.act;
    p.n_act = m.n_act;
    p.rbs = (int)(m.I / 32);
    // persistent: two CTAs per SM share the (active expert x row block) items
    const int64_t items_max = m.E * p.rbs;
    dim3 grid((unsigned)std::min<int64_t>(2 * (int64_t)num_sms(), items_max), 1, 1);
    return launch_t<0, 1, 0, GATEUP, 4>(mw, ms, m.xh, m.T * m.topk, p, grid, 1, s);
}

cudaError_t launch_moe_down(const SkinnyMoe& m, cudaStream_t s) {
    CUtensorMap mw, ms;
    if (!make_maps(&mw, &ms, 0, m.d_q, m.d_s, m.H, m.I, m.E, RB)) return cudaErrorInvalidValue;
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
    p.act = m.act;
    p.n_act = m.n_act;
    p.rbs = (int)(m.H / RB);
    const int64_t items_max = m.E * p.rbs;
    dim3 grid((unsigned)std::min<int64_t>(2 * (int64_t)num_sms(), items_max), 1, 1);
    return launch_t<0, 1, 0, DOWN, 4>(mw, ms, m.ah, m.T * m.topk, p, grid, 1, s);
}

}  // namespace cq
