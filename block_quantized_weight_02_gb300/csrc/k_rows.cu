// Weight-streaming GEMM for up to 32 activation rows, partitioned by weight
// rows so that every SM streams the same number of weight bytes.
//
// The weight rows are cut into units of 8 and the units are spread over one
// CTA per SM as evenly as integers allow (for N = 8192 on 152 SMs: 7 or 6
// units, within 4 % of the mean).  Each CTA streams the whole K range of its
// rows, so no partial sums cross CTAs.  Inside a CTA the units come in passes
// of up to eight (as many passes as needed, units split evenly over them);
// a pass is four m16 tiles of two units each (the weights are the A operand
// of mma.sync m16n8k16, the activation rows its n8 B operand in one to four
// n8 tiles), and consumer
// warp w takes tile w % 4 and the quarter w / 4 of every stage's 32-k blocks.
// The four quarters' sums of a tile are added in a fixed order at the end of
// the pass.  A tile whose second unit lies past the CTA's units multiplies
// whatever its rows 8..15 hold; an MMA's output row depends only on its own A
// row, and those outputs are not stored.
//
// Stages of 512 k: weight boxes {128 bytes, the pass's rows} (two for Q4, four
// for Q8; 128-byte swizzle: 16-byte chunk j of row r at j ^ (r % 8)), for the
// block-scaled formats one box of scales over the same rows, and one box of
// the activations {64 k, 8, 16 or 32 rows, 8 slabs} -- at most six boxes per
// stage, since a TMA box costs about the same however few bytes it holds.
// Producer lane s issues every copy of the stages that land in ring slot s.
//
// Decode (lane c of a quad, rows g and g + 8 of its warp's tile): Q4 word c
// of a 32-k block holds k = 4c .. 4c + 3 (low nibbles) and 16 + 4c ..
// (high nibbles); adjacent nibbles are paired, so the MMA's virtual k = 2c,
// 2c + 1, 2c + 8, 2c + 9 are the physical k = 4c .. 4c + 3 (first MMA) and
// 16 + 4c .. (second), and the activation operand of each MMA is one 8-byte
// run of a token's row.  Q8: words c of the block's two 16-byte chunks give
// the same k.  Every product of the Q4 and Q8 decodes is exact (q - 8, or q,
// in the activation type); the block scale multiplies the f32 result of the
// block's two MMAs (Q4, Q8 per 32-k block), the Q8-row scale multiplies the
// finished sum.
//
// Launched with programmatic dependent launch: the producer requests the
// weights of its first ring fill before it waits for the previous kernel, and
// the activations after.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>

#include "cq_internal.h"
#include "cq_ptx.cuh"

namespace cq {
namespace {

constexpr int UPASS = 8;                      // units per pass at most
constexpr int TILES = UPASS / 2;              // m16 tiles per pass
constexpr int PARTS = 4;                      // warps along the k-blocks of a stage
constexpr int RW_CONS = TILES * PARTS;        // consumer warps
constexpr int RW_PROD = RW_CONS;              // the producer warp
constexpr int RW_THREADS = (RW_CONS + 1) * 32;
constexpr int UNIT = 8;                       // weight rows per unit
constexpr int KSTAGE = 512;                   // k per stage

struct RParams {
    int64_t N, K, T;
    int units;           // ceil(N / 8)
    int upp;             // units per pass (the boxes span 8 upp rows)
    int nst;             // stages over K
    const float* rs;     // Q8-row: row scales
    const float* rsx;    // nullable: per-token scale of the activations (q8_2f: the guard's inverse)
    const float* add;    // nullable f32 [T][N] added before the rounding
    void* y;
    int yt;
    uint64_t wait_ns;
    int* err;
};

struct RMaps {
    CUtensorMap w;       // weights {K bytes, N}, box {128 B, 8 upp rows}
    CUtensorMap s;       // Q4: fp16 scales {K/32, N} box {16, 8 upp}; Q8/32: f32 {K/32, N} box {8, 8 upp}
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
    static constexpr int BPS = KSTAGE / 32;                   // 32-k blocks per stage
    static constexpr int BPW = BPS / PARTS;                   // ... per warp and stage
    static constexpr int ROWB = FMT == 0 ? KSTAGE / 2 : KSTAGE;   // weight bytes per row and stage
    static constexpr int NBOX = ROWB / 128;                   // 128-byte weight boxes per stage
    static constexpr int WBOX = UPASS * UNIT * 128;           // room of one weight box (64 rows)
    static constexpr int W_BYTES = NBOX * WBOX;
    static constexpr int S_ROW = FMT == 0 ? 32 : FMT == 2 ? 64 : 0;   // scale bytes per row and stage
    static constexpr int S_BYTES = UPASS * UNIT * S_ROW;
    static constexpr int XSL = KSTAGE / 64;                   // 64-k slabs per stage
};

template <int FMT, int TP>
struct RLayout {
    using G = RGeo<FMT>;
    static constexpr int X_BYTES = G::XSL * TP * 128;
    static constexpr int X_OFF = G::W_BYTES + G::S_BYTES;     // 1024-aligned
    static constexpr int SLOT = X_OFF + X_BYTES;
    static constexpr int RED_BYTES = TILES * (PARTS - 1) * 32 * TP / 2 * 4;   // quarters 1..3 of each tile
    static_assert(G::W_BYTES % 1024 == 0 && X_OFF % 1024 == 0 && SLOT % 1024 == 0, "1024-byte aligned boxes");
};

// FMT 0: Q4 (fp16 block scales), 1: Q8-row, 2: Q8 per 32-k block (f32 block scales).
// TP: activation rows, 8, 16 or 32 (one, two or four n8 tiles).  XBF: bf16 activations.
template <int FMT, int TP, int XBF, int NSLOT>
__global__ void __launch_bounds__(RW_THREADS, 1)
k_rows(const __grid_constant__ RMaps maps, const RParams p) {
    using G = RGeo<FMT>;
    using L = RLayout<FMT, TP>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    float* red = reinterpret_cast<float*>(smem + NSLOT * L::SLOT);   // [TILES][PARTS - 1][32 lanes][4 NT]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NSLOT * L::SLOT + L::RED_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(NSLOT + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * NSLOT);
    volatile int* never_flag = abort_flag + 1;   // stays 0: waits that must not be cut short

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    // this CTA's units (as even a split as integers allow) and its passes of upp units
    const int u0 = (int)((int64_t)blockIdx.x * p.units / gridDim.x);
    const int u1 = (int)((int64_t)(blockIdx.x + 1) * p.units / gridDim.x);
    const int upp = p.upp;
    const int npass = (u1 - u0 + upp - 1) / upp;
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
            // weights (and scales) of the pass: one box per 128-byte column of the stage, over
            // the pass's 8 upp rows (rows of other CTAs, or past N, in a short pass are loaded
            // and not used)
            auto issue_w = [&](int pass, int i) {
                const int row = (u0 + pass * upp) * UNIT;
#pragma unroll
                for (int q = 0; q < G::NBOX; ++q)
                    tma_load_2d(base + (uint32_t)(q * G::WBOX), &maps.w, full_bar(s), i * G::ROWB + q * 128, row);
                if (FMT != 1) tma_load_2d(base + (uint32_t)G::W_BYTES, &maps.s, full_bar(s), i * G::BPS, row);
            };
            const uint32_t stage_bytes = (uint32_t)(upp * UNIT * (G::NBOX * 128 + G::S_ROW) + L::X_BYTES);
            auto bytes_of = [&](int) { return stage_bytes; };
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
    constexpr int NT = TP / 8;                             // n8 tiles of activation rows
    const int tile = warp % TILES, part = warp / TILES;    // m16 tile of the pass, quarter of the blocks
    // This thread's offsets from a ring slot's base, the same in every stage (Q4): the weight word
    // of each of its blocks (row g; row g + 8 is 1024 bytes on) and the two 8-byte activation runs
    // of token g of the first n8 tile (the others 1024 bytes apart)
    uint32_t woff[G::BPW], xoff[G::BPW][2];
#pragma unroll
    for (int jh = 0; jh < G::BPW; ++jh) {
        const int jb = part * G::BPW + jh;
        woff[jh] = (uint32_t)((16 * tile + g) * 128 + 4 * c + (jb >> 3) * G::WBOX) + ((((uint32_t)(jb & 7)) ^ (uint32_t)g) << 4);
        const uint32_t clo = (uint32_t)(4 * (jb & 1) + (c >> 1));
        const uint32_t xr = (uint32_t)L::X_OFF + ((uint32_t)(jb >> 1) * TP + (uint32_t)g) * 128u + 8u * (uint32_t)(c & 1);
        xoff[jh][0] = xr + ((clo ^ (uint32_t)g) << 4);
        xoff[jh][1] = xr + (((clo + 2u) ^ (uint32_t)g) << 4);
    }
    int gi = 0;
    for (int pass = 0; pass < npass; ++pass) {
        const int ub = u0 + pass * upp, nu = min(upp, u1 - ub);
        const bool lo_ok = 2 * tile < nu, hi_ok = 2 * tile + 1 < nu;
        // Q8-row: the epilogue's row scales (rows g, g + 8 of the tile), loaded before the stages
        float rsc[2] = {1.f, 1.f};
        if (FMT == 1 && part == 0 && lo_ok) {
            const int64_t n0 = (int64_t)(ub + 2 * tile) * UNIT + g;
            if (n0 < p.N) rsc[0] = p.rs[n0];
            if (hi_ok && n0 + 8 < p.N) rsc[1] = p.rs[n0 + 8];
        }
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        bool ok = !*abort_flag;
        for (int i = 0; i < nst; ++i, ++gi) {
            const int slot = gi % NSLOT;
            if (ok && !mbar_wait_spin(full_bar(slot), (uint32_t)((gi / NSLOT) & 1), p.wait_ns, abort_flag)) {
                ok = false;
                *abort_flag = 1;
                atomicCAS(p.err, 0, DEV_TIMEOUT);
            }
            if (ok && lo_ok) {
                const uint32_t sW = sb + (uint32_t)(slot * L::SLOT);
                const uint32_t sX = sW + (uint32_t)L::X_OFF;
                // rows g (and g + 8, 1024 bytes on) of the tile: 128-byte rows, chunk j at j ^ g
                const uint32_t wrow = sW + (uint32_t)((16 * tile + g) * 128 + 4 * c);
                // block scales of this warp's quarter for rows g and g + 8
                const uint32_t srow = sW + (uint32_t)(G::W_BYTES + (16 * tile + g) * G::S_ROW);
                float slo[G::BPW], shi[G::BPW];
                if (FMT == 0) {
                    const uint2 a = r_lds64(srow + 8u * (uint32_t)part);
                    const uint2 b = r_lds64(srow + 8u * G::S_ROW + 8u * (uint32_t)part);
                    const uint32_t av[2] = {a.x, a.y}, bv[2] = {b.x, b.y};
#pragma unroll
                    for (int j = 0; j < G::BPW; ++j) {
                        slo[j] = __half2float(__ushort_as_half((unsigned short)(j & 1 ? av[j >> 1] >> 16 : av[j >> 1] & 0xFFFFu)));
                        shi[j] = __half2float(__ushort_as_half((unsigned short)(j & 1 ? bv[j >> 1] >> 16 : bv[j >> 1] & 0xFFFFu)));
                    }
                } else if (FMT == 2) {
                    const uint4 a = r_lds128(srow + 16u * (uint32_t)part);
                    const uint4 b = r_lds128(srow + 8u * G::S_ROW + 16u * (uint32_t)part);
                    slo[0] = __uint_as_float(a.x), slo[1] = __uint_as_float(a.y);
                    slo[2] = __uint_as_float(a.z), slo[3] = __uint_as_float(a.w);
                    shi[0] = __uint_as_float(b.x), shi[1] = __uint_as_float(b.y);
                    shi[2] = __uint_as_float(b.z), shi[3] = __uint_as_float(b.w);
                }
#pragma unroll
                for (int jh = 0; jh < G::BPW; ++jh) {
                    const int jb = part * G::BPW + jh;   // block of the stage
                    // activations: token g (and g + 8), slab jb / 2, the 8-byte runs at k 4c (lo) and 16 + 4c (hi)
                    const uint32_t slab = (uint32_t)(jb >> 1);
                    const uint32_t clo = (uint32_t)(4 * (jb & 1) + (c >> 1)), off8 = 8u * (uint32_t)(c & 1);
                    const uint32_t xr = sX + (slab * TP + (uint32_t)g) * 128u + off8;
                    uint32_t a1[4], a2[4];
                    if (FMT == 0) {
                        const uint32_t wa = sW + woff[jh];
                        uint32_t dl[4], dh[4];
                        q4_adjacent<XBF>(r_lds32(wa), dl);
                        q4_adjacent<XBF>(r_lds32(wa + 1024u), dh);
                        a1[0] = dl[0], a1[1] = dh[0], a1[2] = dl[1], a1[3] = dh[1];
                        a2[0] = dl[2], a2[1] = dh[2], a2[2] = dl[3], a2[3] = dh[3];
                    } else {
                        const uint32_t rb = wrow + (uint32_t)((jb >> 2) * G::WBOX);
                        const uint32_t o0 = (((uint32_t)(2 * (jb & 3))) ^ (uint32_t)g) << 4;
                        const uint32_t o1 = (((uint32_t)(2 * (jb & 3) + 1)) ^ (uint32_t)g) << 4;
                        const uint32_t l0 = r_lds32(rb + o0), l1 = r_lds32(rb + o1);
                        const uint32_t h0 = r_lds32(rb + 1024u + o0), h1 = r_lds32(rb + 1024u + o1);
                        a1[0] = i8_pair<XBF>(l0, 0x4140u), a1[1] = i8_pair<XBF>(h0, 0x4140u);
                        a1[2] = i8_pair<XBF>(l0, 0x4342u), a1[3] = i8_pair<XBF>(h0, 0x4342u);
                        a2[0] = i8_pair<XBF>(l1, 0x4140u), a2[1] = i8_pair<XBF>(h1, 0x4140u);
                        a2[2] = i8_pair<XBF>(l1, 0x4342u), a2[3] = i8_pair<XBF>(h1, 0x4342u);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {   // tokens 8 nt + g
                        const uint2 xlo = r_lds64(FMT == 0 ? sW + xoff[jh][0] + 1024u * nt : xr + 1024u * nt + ((clo ^ (uint32_t)g) << 4));
                        const uint2 xhi = r_lds64(FMT == 0 ? sW + xoff[jh][1] + 1024u * nt : xr + 1024u * nt + (((clo + 2u) ^ (uint32_t)g) << 4));
                        if (FMT == 1) {
                            mma_f<XBF>(acc[nt], a1, xlo.x, xlo.y);
                            mma_f<XBF>(acc[nt], a2, xhi.x, xhi.y);
                        } else {
                            float pb[4] = {0.f, 0.f, 0.f, 0.f};
                            mma_f<XBF>(pb, a1, xlo.x, xlo.y);
                            mma_f<XBF>(pb, a2, xhi.x, xhi.y);
                            acc[nt][0] = fmaf(slo[jh], pb[0], acc[nt][0]);
                            acc[nt][1] = fmaf(slo[jh], pb[1], acc[nt][1]);
                            acc[nt][2] = fmaf(shi[jh], pb[2], acc[nt][2]);
                            acc[nt][3] = fmaf(shi[jh], pb[3], acc[nt][3]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(slot));
        }
        // ---- the quarters' sums (quarters 1..3 handed over in shared memory, added in
        // quarter order), then the epilogue of the tile by its first quarter: lane (g, c)
        // holds rows g, g + 8 of the tile and tokens 2c, 2c + 1 of each n8 tile ----
        float* rd = red + ((tile * (PARTS - 1)) * 32 + lane) * (4 * NT);
        if (part > 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                *reinterpret_cast<float4*>(rd + (part - 1) * 32 * 4 * NT + 4 * nt) =
                    make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(RW_CONS * 32) : "memory");
        if (part == 0) {
#pragma unroll
            for (int q = 0; q < PARTS - 1; ++q) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float4 o = *reinterpret_cast<const float4*>(rd + q * 32 * 4 * NT + 4 * nt);
                    acc[nt][0] += o.x;
                    acc[nt][1] += o.y;
                    acc[nt][2] += o.z;
                    acc[nt][3] += o.w;
                }
            }
        }
        if (part == 0 && ok && lo_ok && !*abort_flag) {
            const int64_t n0 = (int64_t)(ub + 2 * tile) * UNIT + g;   // row g; row g + 8 is n0 + 8
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int64_t n = n0 + 8 * hr;
                if ((hr == 1 && !hi_ok) || n >= p.N) continue;
                const float sc = rsc[hr];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int64_t t = 8 * nt + 2 * c + e;
                        if (t >= p.T) continue;
                        float v = acc[nt][2 * hr + e] * sc;
                        if (p.rsx) v *= p.rsx[t];
                        if (p.add) v += p.add[t * p.N + n];
                        if (p.yt == CQ_F32) reinterpret_cast<float*>(p.y)[t * p.N + n] = v;
                        else reinterpret_cast<__nv_bfloat16*>(p.y)[t * p.N + n] = __float2bfloat16_rn(v);
                    }
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(RW_CONS * 32) : "memory");   // the hand-over memory is free again
    }
}

template <int FMT, int TP, int XBF, int NSLOT>
cudaError_t launch_rows_t(const RMaps& maps, const RParams& p, int grid, cudaStream_t s) {
    using L = RLayout<FMT, TP>;
    constexpr size_t smem = (size_t)NSLOT * L::SLOT + L::RED_BYTES + 2 * NSLOT * 8 + 16 + 1024;
    static_assert(smem <= 227 * 1024, "shared memory budget");
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
    return counted(cudaLaunchKernelEx(&cfg, kern, maps, p));
}

template <int FMT, int XBF>
cudaError_t launch_rows_x(const RMaps& maps, const RParams& p, int grid, int64_t T, cudaStream_t s) {
    // ring depth: as many 512-k stages as fit (Q4 26 / 34 / 50 KB, Q8-row 40 / 48 / 64 KB,
    // Q8/32 44 / 52 KB for 8 / 16 / 32 activation rows)
    if (T <= 8) return launch_rows_t<FMT, 8, XBF, FMT == 0 ? 8 : FMT == 1 ? 5 : 4>(maps, p, grid, s);
    if (T <= 16) return launch_rows_t<FMT, 16, XBF, FMT == 0 ? 6 : 4>(maps, p, grid, s);
    if constexpr (FMT != 2) return launch_rows_t<FMT, 32, XBF, FMT == 0 ? 4 : 3>(maps, p, grid, s);
    return cudaErrorInvalidValue;   // Q8/32 serves T <= 16 (rows_path_serves)
}

}  // namespace

bool rows_path_serves(int fmt, int64_t T, int64_t K, int nz) {
    return nz <= 1 && T >= 1 && T <= (fmt == 2 ? 16 : 32) && K % KSTAGE == 0;
}

bool rows_path_preferred(int fmt, int64_t T, int64_t K, int64_t N, int nz) {
    if (!rows_path_serves(fmt, T, K, nz)) return false;
    // measured on GB300 (T = 1-32; Q4 and Q8-row): faster than the K-split kernel, or level
    // with it, when every CTA holds 6 to 8 units in one pass (at least three full tiles) -- for
    // Q8 only up to T = 16 -- and for very small weights (K = 512, N = 256: one launch without a
    // cluster); with fewer units (idle warps) or two passes the K-split kernel was faster
    if (N * K <= (int64_t)1 << 19) return true;
    if (fmt != 0 && T > 16) return false;
    const int64_t units = (N + UNIT - 1) / UNIT, grid = std::min<int64_t>((int64_t)num_sms(), units);
    const int64_t maxu = (units + grid - 1) / grid;
    return maxu >= 6 && maxu <= UPASS;
}

cudaError_t launch_rows(int fmt, const SkinnyDense& a, cudaStream_t s) {
    const int64_t kstage = KSTAGE;
    RParams p = {};
    p.N = a.N;
    p.K = a.K;
    p.T = a.T;
    p.units = (int)((a.N + UNIT - 1) / UNIT);
    p.nst = (int)(a.K / kstage);
    p.rs = a.rs;
    p.rsx = a.rsx;
    p.add = a.add;
    p.y = a.y;
    p.yt = a.yt;
    p.wait_ns = (uint64_t)options().wait_ns;
    p.err = a.err;
    const int grid = (int)std::min<int64_t>((int64_t)num_sms(), p.units);
    // units per pass: the most units a CTA holds, split evenly over as few passes of <= 8 as needed
    const int maxu = (p.units + grid - 1) / grid, np = (maxu + UPASS - 1) / UPASS;
    p.upp = (maxu + np - 1) / np;
    RMaps maps;
    memset(&maps, 0, sizeof maps);
    const uint64_t kbytes = fmt == 0 ? (uint64_t)a.K / 2 : (uint64_t)a.K;
    {
        uint64_t d[2] = {kbytes, (uint64_t)a.N};
        uint64_t st[1] = {kbytes};
        uint32_t box[2] = {128, (uint32_t)(UNIT * p.upp)};
        if (!encode_tiled(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.wq, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (fmt == 0) {
        uint64_t d[2] = {(uint64_t)a.K / 32, (uint64_t)a.N};
        uint64_t st[1] = {(uint64_t)a.K / 32 * 2};
        uint32_t box[2] = {16, (uint32_t)(UNIT * p.upp)};
        if (!encode_tiled(&maps.s, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, a.ws, d, st, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else if (fmt == 2) {
        uint64_t d[2] = {(uint64_t)a.K / 32, (uint64_t)a.N};
        uint64_t st[1] = {(uint64_t)a.K / 32 * 4};
        uint32_t box[2] = {16, (uint32_t)(UNIT * p.upp)};
        if (!encode_tiled(&maps.s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.wsf, d, st, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    {
        // {64 elements, T rows, K/64 slabs} (strides K*2 B, 128 B): a box of TP rows x stage/64 slabs
        // lands as [slab][row][128 B], 128-byte swizzled
        const int tp = a.T <= 8 ? 8 : a.T <= 16 ? 16 : 32;
        uint64_t d[3] = {64, (uint64_t)a.T, (uint64_t)a.K / 64};
        uint64_t st[2] = {(uint64_t)a.K * 2, 128};
        uint32_t box[3] = {64, (uint32_t)tp, (uint32_t)(kstage / 64)};
        if (!encode_tiled(&maps.x, a.x_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.x,
                          d, st, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (options().trace)
        fprintf(stderr, "cq: rows fmt=%d T=%lld N=%lld K=%lld units=%d per pass=%d grid=%d\n", fmt, (long long)a.T,
                (long long)a.N, (long long)a.K, p.units, p.upp, grid);
    if (fmt == 0) return a.x_bf16 ? launch_rows_x<0, 1>(maps, p, grid, a.T, s) : launch_rows_x<0, 0>(maps, p, grid, a.T, s);
    if (fmt == 1) return a.x_bf16 ? launch_rows_x<1, 1>(maps, p, grid, a.T, s) : launch_rows_x<1, 0>(maps, p, grid, a.T, s);
    return a.x_bf16 ? launch_rows_x<2, 1>(maps, p, grid, a.T, s) : launch_rows_x<2, 0>(maps, p, grid, a.T, s);
}

}  // namespace cq
