// Large-T GEMM on the 5th-generation tensor cores (tcgen05, accumulator in
// tensor memory), weights dequantized on the fly in shared memory.
//
// Y^T tile = W tile (128 weight rows, M) x X tile^T (BN activation rows, N),
// K in stages of 64, loaded in super-stages of G stages (one weight box of
// G * 32 or G * 64 bytes per row and one activation box of G 64-k chunks:
// a TMA box costs nearly the same whatever its size, so fewer, larger boxes
// keep the copies ahead of the tensor core).  Warp roles in a CTA of 576
// threads:
//   warp 16     TMA producers: lane s issues the weight box of super-slot s,
//               lane LSS + s its activation box;
//   warps 0-15  decoders: group w / 4 takes every fourth stage, warp w
//               rows 32 (w % 4) .. +31 of it (one 64-k row per thread),
//               decoded into the A operand (tensor memory by default, else
//               the 128-byte swizzled K-major tile in shared memory); four
//               stages are in decode at once.  Then the epilogue;
//   warp 17     allocates the tensor memory and issues tcgen05.mma
//               (M = 128, N = BN, K = 16) from one thread, a round of 2 or 4
//               stages at a time, committing each round's decoded slots and
//               each super-stage's load slot back, and the last round to the
//               epilogue.
// CTA pairs (cta_group::2): two neighbouring weight-row tiles share one MMA
// of M = 256; each CTA decodes its own rows into its own tensor memory and
// loads half of the activation rows; the even CTA issues.  K split: two CTAs
// of a cluster take the two halves of K and exchange half of their f32
// accumulators through distributed shared memory.  Epilogue: scaled,
// staged in shared memory and stored with TMA per decoder group and chunk.
// Q4 decode: (nibble - 8) * fp16 block scale, rounded once to fp16 (the
// scale folded into the half operand, as in mma_tile of "oxinfer 0.0.5
// src/metal.rs"); the activations arrive as fp16 behind a per-row
// power-of-two guard whose inverse the epilogue applies, stored by the
// guard pass in the streaming order inside each 32-k block, the order in
// which two masks per word yield the nibble pairs; the decoded weights are
// written in that same order, so the contraction is unchanged.  Q8-row decode:
// int8 -> the activation type exactly; the row scale is applied to the f32
// accumulator in the epilogue ("cortiq-engine 0.8.3 src/gpu_metal/qi21.rs",
// module header on q8_row).
// Affine mode (GU = 2, Q4): a bf16 offset per group of gk blocks joins the
// decode, fp16((n - 8) * scale + fp16(offset)) in one rounding ("oxinfer 0.0.5
// src/metal.rs", Dequantizers, struct Q4A).
// Gate/up mode (GU = 1): the CTA's 128 weight rows are 64 gate rows i0 .. i0 + 63
// and the matching 64 up rows I + i0 .. (one 3-D TMA box over the two
// halves of the [2I][K] matrix), and the epilogue applies SwiGLU,
// a = g / (1 + exp(-g)) * u, writing a[T][I] in f32: the gate/up GEMM of the
// denoiser block's chain gemm(TG, TU) -> swiglu ("cortiq-engine 0.8.3
// src/gpu_metal/qi21.rs", fn blocks) with the SwiGLU moved into the epilogue.
// Every wait is time-bounded; on a timeout the CTA stops, lets copies in
// flight land, frees its tensor memory and reports CQ_ERR_TIMEOUT in the
// calling stream's device error word.
//
// Included by k_tc.cu (dense GEMMs), k_tc_ffn.cu (gate/up mode), k_tc_q4a.cu
// (affine mode) and k_tc_q8b.cu (Q8/32), so that the sets of instantiations
// compile in parallel.
#pragma once
#include <algorithm>
#include <cstring>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cq_internal.h"
#include "cq_ptx.cuh"

namespace cq {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB

// Per-job pointers of a z-batched launch (job = blockIdx.y / tiles_y).
struct Job {
    const float* rsx;     // guard inverse scale per activation row (Q4, Q8/32; Q8-row: nullable)
    const float* rs;      // Q8-row: row scales
    const uint16_t* ws;   // Q4 block scales [N][K/32] fp16
    const float* wsf;     // Q8/32 block scales [N][K/32] f32
    const float* add;     // nullable: f32 [T][N] added to the scaled accumulator before the rounding
    void* y;              // output rows of pitch ldy
};
// Tensor maps of every job: weights, activations, outputs.
struct Maps {
    CUtensorMap w[ZMAX];
    CUtensorMap x[ZMAX];
    CUtensorMap y[ZMAX];
};

struct Params {
    Job job[ZMAX];
    const uint16_t* off;  // affine mode (single job): offsets bf16 [N][K/32/gk]
    int gk;               // blocks per offset group
    int mt0;              // first weight-row tile of this launch (a call may split its tiles over two)
    int tiles_y;          // token tiles per job
    int64_t ldy;          // output row pitch (elements)
    int yt;
    int64_t T, N, K;
    uint64_t wait_ns;
    int stall;
    int pdl;   // launched with a programmatic dependency on the guard pass
    int y_tma; // Y row pitch is a multiple of 16 bytes: tiles leave through a TMA store
    int* err;  // the calling stream's device error word
};

__device__ __forceinline__ uint32_t i8x2_to_h2(uint32_t w, uint32_t sel) {
    return sub_f16x2(prmt(w ^ 0x80808080u, 0x64646464u, sel), 0x64806480u);
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Eight nibbles (bytes b0..b3 of w) -> four fp16 pairs (n - 8) * scale, each
// rounded once, in the activations' streaming order: (low b0, low b2),
// (high b0, high b2), (low b1, low b3), (high b1, high b3).  0x6400 | n is
// 1024 + n and 0x6400 | (n << 4) is 1024 + 16 n; 1024 + n - 1032 and
// (1024 + 16 n) / 16 - 72 are n - 8 exactly.
__device__ __forceinline__ void decode_q4_word_scaled(uint32_t w, uint32_t sc, uint32_t* o) {
    const uint32_t c6400 = 0x64006400u, k1032 = 0x64086408u, k16th = 0x2C002C00u, km72 = 0xD480D480u;
    const uint32_t w8 = w >> 8;
    o[0] = mul_f16x2(sub_f16x2(and_or<0x000F000Fu>(w, c6400), k1032), sc);
    o[1] = mul_f16x2(fma_f16x2(and_or<0x00F000F0u>(w, c6400), k16th, km72), sc);
    o[2] = mul_f16x2(sub_f16x2(and_or<0x000F000Fu>(w8, c6400), k1032), sc);
    o[3] = mul_f16x2(fma_f16x2(and_or<0x00F000F0u>(w8, c6400), k16th, km72), sc);
}
// The same with an affine offset m in both halves: (n - 8) * scale + m, rounded once.
__device__ __forceinline__ void decode_q4_word_scaled_off(uint32_t w, uint32_t sc, uint32_t m, uint32_t* o) {
    const uint32_t c6400 = 0x64006400u, k1032 = 0x64086408u, k16th = 0x2C002C00u, km72 = 0xD480D480u;
    const uint32_t w8 = w >> 8;
    o[0] = fma_f16x2(sub_f16x2(and_or<0x000F000Fu>(w, c6400), k1032), sc, m);
    o[1] = fma_f16x2(fma_f16x2(and_or<0x00F000F0u>(w, c6400), k16th, km72), sc, m);
    o[2] = fma_f16x2(sub_f16x2(and_or<0x000F000Fu>(w8, c6400), k1032), sc, m);
    o[3] = fma_f16x2(fma_f16x2(and_or<0x00F000F0u>(w8, c6400), k16th, km72), sc, m);
}

template <int FMT>
struct Raw;
template <>
struct Raw<0> { static constexpr int ROW = 32; };   // Q4: 64 k = 32 bytes per row and stage
template <>
struct Raw<1> { static constexpr int ROW = 64; };   // Q8: 64 bytes per row and stage
template <>
struct Raw<2> { static constexpr int ROW = 64; };   // Q8 per 32-k block: 64 bytes per row and stage

// Loads come in super-stages of G stages (G x 64 k), two TMA boxes each: a TMA
// box costs about the same however few bytes it holds, so the weight rows are
// fetched G stages at a time (G * ROW bytes per row) and the activation tile as
// one 3-D box of G 64-k chunks.
// Shared memory per super-slot: X [G][BN rows][128 B] (each chunk one
// 128-byte-swizzled K-major operand tile), then W [128 rows][G * ROW B]
// (128- or 64-byte swizzle).  AM 0 adds AS decoded tiles [128][128 B] in
// front; AM 1 keeps the decoded tiles in tensor memory.  With CTA pairs (CG 2)
// each CTA holds half of the activation rows (its half of the MMA's B operand).
template <int FMT, int BN, int G, int LSS, int AS, int AM, int CG = 1>
struct Layout {
    static constexpr int WROW = G * Raw<FMT>::ROW;            // 64 or 128 bytes
    static constexpr int X_CHUNK = (BN / CG) * 128;
    static constexpr int X_BYTES = G * X_CHUNK;
    static constexpr int W_BYTES = BM * WROW;
    static constexpr int SLOT = X_BYTES + W_BYTES;             // multiple of 1024
    static constexpr int A_OFF = 0;
    static constexpr int S_OFF = AM == 0 ? AS * A_BYTES : 0;
    static constexpr int BAR_OFF = S_OFF + LSS * SLOT;
    // Decoded slots are handed over in rounds of RS stages, NRB rounds in flight: four stages
    // when the ring holds many stages (tensor-memory slots with BN <= 128), else two, so that
    // a round never waits for ring slots its own MMAs free; and four for Q4 in CTA pairs,
    // whose MMA thread then waits for a decoded round half as often (about 300 cycles a
    // wait; measured on GB300: Q4 192-token pairs 12 % faster, Q8-row pairs slower).
    static constexpr int RS = (AM == 1 && (BN <= 128 || (CG > 1 && FMT == 0))) ? 4 : 2;
    static constexpr int NRB = AS / RS;
    // When a round is one super-stage, the super-slot's release (committed after the
    // round's MMAs) also frees the round's decoded slots: the decoders wait on it and no
    // separate release is committed.  With LSS >= NRB no wait can fall two phases behind.
    static constexpr bool MERGE = RS == G && LSS >= NRB;
    // full[LSS], empty[LSS], afull[NRB], aempty[NRB] (one per round in flight), accf,
    // xchg[4] (split K: one per decoder group); then tmem slot, abort, never
    static constexpr int NBAR = 2 * LSS + 2 * NRB + 5;
    static constexpr int MISC = NBAR * 8 + 16;
    static constexpr int TOTAL = BAR_OFF + MISC + 1024;  // + alignment slack
    // tensor memory: accumulator in columns [0, BN); AM 1 adds AS decoded A tiles of 32 columns
    static constexpr int A_COL = BN;
    static constexpr int NEED = AM == 0 ? BN : BN + AS * 32;
    static constexpr int TMEM_COLS = NEED <= 32 ? 32 : NEED <= 64 ? 64 : NEED <= 128 ? 128 : NEED <= 256 ? 256 : 512;
    static_assert(NEED <= 512, "tensor memory budget");
    static_assert(SLOT % 1024 == 0 && X_CHUNK % 1024 == 0, "1024-byte aligned swizzled tiles");
    static_assert(WROW == 32 || WROW == 64 || WROW == 128, "weight rows of 32, 64 or 128 bytes");
};

// Epilogue geometry: a CTA finishes NC columns of its tile (all BN, or its half under a
// K split); each of the first NG decoder groups (all four from 64 columns, else group 0)
// owns NC / NG of them and handles them CH at a time (one tensor-memory load, one
// output box, one exchange copy per chunk).
constexpr int ep_cols(int BN, int KS) { return KS > 1 ? BN / 2 : BN; }
constexpr int ep_groups(int BN, int KS) { return ep_cols(BN, KS) >= 64 ? 4 : 1; }
constexpr int ep_chunk(int BN, int KS) {
    return (ep_cols(BN, KS) / ep_groups(BN, KS)) % 32 == 0 ? 32 : 16;
}

template <int CH>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[CH]) {
    static_assert(CH == 16 || CH == 32, "16 or 32 columns per load");
    if constexpr (CH == 32) tmem_ld_32x32b_x32(taddr, v);
    else tmem_ld_32x32b_x16(taddr, v);
}

constexpr int DEC_WARPS = 16;                // 4 groups (stages kb % 4) x 4 row quarters
constexpr int THREADS = (DEC_WARPS + 2) * 32;
constexpr int PRODUCER_WARP = DEC_WARPS;
constexpr int MMA_WARP = DEC_WARPS + 1;

// int8 pair (bytes sel of w) -> bf16x2 exactly: with 0x43 as the high byte, the
// low seven bits of v give 128 + (v & 127) and the sign bit gives 128 or 256
// (0x4300 / 0x4380); their difference is v, an integer bf16 holds exactly.
__device__ __forceinline__ uint32_t i8x2_to_bf2(uint32_t w, uint32_t sel) {
    const uint32_t t = prmt(w, 0x43434343u, sel);
    return sub_bf16x2(and_mask<0xFF7FFF7Fu>(t), and_mask<0xFF80FF80u>(t));
}

// KS: K split over a cluster of KS CTAs along z (1 or 2); the two partial
// accumulators are exchanged through distributed shared memory and each CTA
// finishes half of the tile's columns.
// CG: CTA pairs along x (1 or 2).  With 2, two neighbouring weight-row tiles share
// one 256-row MMA (cta_group::2): each CTA decodes its 128 rows into its own tensor
// memory and loads half of the activation rows; the even CTA's MMA thread issues
// for both once both CTAs' decoders have arrived on its barrier (the odd CTA's
// decoder warps arrive there directly, each after its tensor-memory stores have
// completed), and every release it commits reaches both CTAs.  Each CTA's accumulator holds its rows x all BN
// columns, so the epilogue is unchanged.  Cluster ranks run x fastest: the pair
// peer is rank ^ 1, the K-split partner rank ^ CG.
template <int FMT, int BN, int XBF, int G, int LSS, int AS, int AM, int KS, int CG, int GU>
__global__ void __launch_bounds__(THREADS, 1)
k_tc(const __grid_constant__ Maps maps, const Params p) {
    using L = Layout<FMT, BN, G, LSS, AS, AM, CG>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // first weight row (gate/up mode: first gate row i0; the tile is i0 .. i0 + 63 and I + i0 ..)
    const int m0 = (p.mt0 + (int)blockIdx.x) * (GU == 1 ? BM / 2 : BM);
    const int jz = (int)blockIdx.y / p.tiles_y;                 // job of a z-batched launch
    const int t0 = ((int)blockIdx.y - jz * p.tiles_y) * BN;    // first activation row
    const Job J = jz == 0 ? p.job[0] : jz == 1 ? p.job[1] : jz == 2 ? p.job[2] : p.job[3];
    const CUtensorMap* tmW = &maps.w[jz];
    const CUtensorMap* tmX = &maps.x[jz];
    const CUtensorMap* tmY = &maps.y[jz];
    const int kz = KS > 1 ? (int)blockIdx.z : 0;
    const uint32_t crank = (KS > 1 || CG > 1) ? cluster_ctarank() : 0u;   // rank in the cluster
    const int cx = CG > 1 ? (int)(crank & 1u) : 0;                // position in the CTA pair
    const bool leader = cx == 0;                                   // issues the pair's MMAs
    const uint16_t pair_mask = (uint16_t)(3u << (crank - (uint32_t)cx));
    const int nk = (int)(p.K / BK) / KS;     // stages of this CTA's k range
    const int k0 = kz * nk;                  // its first stage
    const int ns = nk / G;                   // super-stages
    const int j0 = k0 / G;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (LSS + s); };
    // Decoded slots come in rounds of RS stages (stages r RS .. r RS + RS - 1 in slots
    // (r % NRB) RS ..): per round in flight one barrier says the round is decoded, one
    // that its MMAs are done.
    constexpr int RS = L::RS, NRB = L::NRB;
    constexpr bool MERGE = L::MERGE;
    auto afull_bar = [&](int rb) { return bar0 + 8u * (2 * LSS + rb); };
    auto aempty_bar = [&](int rb) { return bar0 + 8u * (2 * LSS + NRB + rb); };
    const uint32_t accf_bar = bar0 + 8u * (2 * LSS + 2 * NRB);
    // split K: the partner's columns of decoder group g have arrived
    auto xchg_bar = [&](int g) { return accf_bar + 8u + 8u * (uint32_t)g; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never_flag = abort_flag + 1;
    auto slot_base = [&](int s) { return sb + (uint32_t)(L::S_OFF + s * L::SLOT); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < LSS; ++s) {
            mbar_init(full_bar(s), 1);   // the weight lane's arrival + both boxes' bytes
            mbar_init(empty_bar(s), 1);  // the MMA's commit after the super-stage's last stage
        }
        for (int rb = 0; rb < NRB; ++rb) {
            // one arrival per warp of each of the round's RS stages; in a pair the even CTA's
            // barrier takes both CTAs' (the odd CTA's barriers stay unused)
            mbar_init(afull_bar(rb), (CG > 1 && leader ? 8 : 4) * RS);
            mbar_init(aempty_bar(rb), 1);       // the MMA's commit of the round
        }
        mbar_init(accf_bar, 1);
        for (int g = 0; g < 4; ++g) mbar_init(xchg_bar(g), 1);
        *abort_flag = 0;
        *never_flag = 0;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        if (CG > 1) {
            tmem_alloc_pair(smem_u32(tmem_slot), L::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    // the peer's barriers and tensor memory exist before any use (the barriers' initialisation
    // was released at cluster scope by its own fence, so the arrival itself need not release)
    if (CG > 1) {
        cluster_arrive_relaxed();
        cluster_wait_acquire();
    }
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto give_up = [&]() {
        *abort_flag = 1;
        atomicCAS(p.err, 0, DEV_TIMEOUT);
    };
    // The next kernel in the stream may be scheduled on idle SMs now; it waits for this
    // grid to finish before it touches memory.
    pdl_launch_dependents();

    constexpr int NC = ep_cols(BN, KS);      // epilogue: columns this CTA finishes
    constexpr int NG = ep_groups(BN, KS);    //           decoder groups that take part
    constexpr int CW = NC / NG;              //           columns per such group
    constexpr int CH = ep_chunk(BN, KS);     //           columns per chunk
    static_assert(CW % 16 == 0 && CW % CH == 0 && CW <= 64, "epilogue chunks");
    const int cbase = kz * NC;               // first column finished here
    // epilogue scales, loaded before the last MMAs end: per token (guard inverse; lane l of a
    // group holds columns l and 32 + l) and, for Q8-row, per weight row
    float etk0 = 1.f, etk1 = 1.f, erow = 1.f;

    if (warp == PRODUCER_WARP) {
        // ================= TMA producers =================
        // Lane s < LSS issues the weight box of super-slot s (and posts the bytes of
        // both boxes), lane LSS + s its activation box: a thread keeps only a few bulk
        // copies in flight, so the boxes come from 2 LSS threads.
        const int s = lane % LSS;
        const bool wl = lane < LSS, xl = lane >= LSS && lane < 2 * LSS;
        if (wl || xl) {
            if (lane == 0) {
                tma_prefetch_desc(tmW);
                tma_prefetch_desc(tmX);
            }
            const uint32_t base = slot_base(s);
            int issued = 0;        // super-stages issued by this lane
            auto issue = [&](int j) {
                if (wl) {
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)(L::X_BYTES + L::W_BYTES));
                    if (GU == 1) tma_load_3d(base + L::X_BYTES, tmW, full_bar(s), (j0 + j) * L::WROW, m0, 0);
                    else tma_load_2d(base + L::X_BYTES, tmW, full_bar(s), (j0 + j) * L::WROW, m0);
                } else {
                    tma_load_3d(base, tmX, full_bar(s), 0, t0 + cx * (BN / CG), (j0 + j) * G);
                }
            };
            if (!p.stall) {
                // With a programmatic dependency the weights of the first ring fill are
                // requested before waiting for the previous kernel (the guard pass);
                // the activations only after it.
                const bool pre = s < ns;
                if (pre && wl) issue(s);
                pdl_wait();
                if (pre) {
                    if (xl) issue(s);
                    ++issued;
                }
                uint32_t ph = pre ? 1u : 0u;     // phase of this slot's round for super-stage j
                for (int j = s + (pre ? LSS : 0); j < ns; j += LSS, ph ^= 1u) {
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, p.wait_ns, abort_flag)) {
                        give_up();
                        break;
                    }
                    issue(j);
                    ++issued;
                }
            } else {
                pdl_wait();   // every path waits once, so kernels later in the stream stay ordered
            }
            if (*abort_flag && issued > 0) {
                // this lane's last copy must land before the CTA can exit (round issued - 1)
                mbar_wait(full_bar(s), (uint32_t)((issued - 1) & 1), p.wait_ns, never_flag);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ================= MMA issuer =================
        // One thread issues the tensor-core work, two stages per round: wait for both
        // decoded slots (their groups had waited for the super-slot, so the activations are
        // in too), eight MMAs, one commit that frees the pair of decoded slots and, at the end
        // of a super-stage, one that frees the super-slot.  Descriptors advance by adding.
        // A super-slot's (decoded round's) release is committed only when a later load
        // (decode) waits for it.  In a CTA pair only the even CTA's thread issues.
        if (lane == 0 && (CG == 1 || leader)) {
            constexpr uint32_t idesc = idesc_f16(BM * CG, BN, XBF);
            // One thread's serial address arithmetic sits between MMAs, so the operand
            // addresses advance by adding constants: the descriptors' address field is the
            // shared-memory address in 16-byte units (no carry: addresses stay below 256 KB).
            const uint64_t bd0 = smem_desc_sw128(slot_base(0));
            const uint64_t ad0 = AM == 0 ? smem_desc_sw128(sb + L::A_OFF) : 0;
            const uint32_t at0 = tmem + (uint32_t)L::A_COL;
            constexpr uint32_t X_STEP = (uint32_t)(L::X_CHUNK >> 4);                      // next chunk
            constexpr uint32_t S_STEP = (uint32_t)((L::SLOT - (G - 1) * L::X_CHUNK) >> 4); // next super-slot
            const int nr = (nk + RS - 1) / RS;     // rounds (the last one may be short)
            int s = 0, u = 0, js = 0;             // super-slot, chunk and super-stage of the next stage
            uint32_t boff = 0;                    // its activation tile, 16-byte units from super-slot 0
            for (int r = 0; r < nr; ++r) {
                const int rb = r % NRB;
                const bool got = CG > 1 ? mbar_wait_cluster_spin(afull_bar(rb), (uint32_t)((r / NRB) & 1), p.wait_ns, abort_flag)
                                        : mbar_wait_spin(afull_bar(rb), (uint32_t)((r / NRB) & 1), p.wait_ns, abort_flag);
                if (!got) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t a_r = (uint32_t)(rb * RS);   // the round's first decoded slot
#pragma unroll
                for (int i = 0; i < RS; ++i) {
                    const int kb = r * RS + i;
                    if (kb < nk) {
                        const uint64_t bd = bd0 + boff;
                        const uint64_t ad = AM == 0 ? ad0 + (uint64_t)((a_r + (uint32_t)i) * (uint32_t)(A_BYTES >> 4)) : 0;
                        const uint32_t at = at0 + (a_r + (uint32_t)i) * 32u;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint32_t acc = (kb + kk) != 0 ? 1u : 0u;
                            // +32 bytes of K = +2 in the descriptor's 16-byte address units
                            if (AM == 0) tc_mma_f16(tmem, ad + 2u * kk, bd + 2u * kk, idesc, acc);
                            else if (CG > 1) tc_mma_f16_ts_pair(tmem, at + 8u * kk, bd + 2u * kk, idesc, acc);
                            else tc_mma_f16_ts(tmem, at + 8u * kk, bd + 2u * kk, idesc, acc);
                        }
                        if (++u == G) {
                            u = 0;
                            // super-slot free (and, merged, the round's decoded slots)
                            if (js + (MERGE && NRB < LSS ? NRB : LSS) < ns) {
                                if (CG > 1) tc_commit_pair_mc(empty_bar(s), pair_mask);
                                else tc_commit(empty_bar(s));
                            }
                            ++js;
                            if (++s == LSS) {
                                s = 0;
                                boff = 0;
                            } else {
                                boff += S_STEP;
                            }
                        } else {
                            boff += X_STEP;
                        }
                    }
                }
                if (!MERGE && r + NRB < nr) {                   // the round's decoded slots free
                    if (CG > 1) tc_commit_pair_mc(aempty_bar(rb), pair_mask);
                    else tc_commit(aempty_bar(rb));
                }
            }
            // also lets teardown know every MMA has finished
            if (CG > 1) tc_commit_pair_mc(accf_bar, pair_mask);
            else tc_commit(accf_bar);
        }
        __syncwarp();
    } else {
        // ================= decoders, then epilogue =================
        // Four groups of four warps; group g = w / 4 decodes stages g, g + 4, g + 8, ...
        // and in each of them warp w covers rows 32 (w % 4) .. +31 (its tensor-memory lane
        // quarter), one whole 64-k row per thread.  Four stages are decoded at once, so the
        // per-stage chain (wait, load, decode, store, hand-off) of one warp overlaps the
        // others' instead of setting the pace.
        const int q4w = warp & 3, grp = warp >> 2;
        const int r = 32 * q4w + lane;             // weight row within the tile
        // its row of the weight matrix (gate/up mode: gate row m0 + r, or up row I + m0 + r - 64)
        const int64_t n = GU == 1 ? (r < BM / 2 ? (int64_t)m0 + r : p.N + m0 + (r - BM / 2)) : (int64_t)m0 + r;
        const bool row_ok = GU == 1 ? (int64_t)m0 + (r & (BM / 2 - 1)) < p.N : n < p.N;
        const uint32_t xr = (uint32_t)(r & 7);
        const uint32_t t_lane = (uint32_t)(32 * q4w) << 16;
        // a decoded round is announced on the pair's even CTA (its own barrier there)
        const uint32_t afull0 = (CG > 1 && !leader) ? mapa_shared(afull_bar(0), crank ^ 1u) : afull_bar(0);
        auto announce = [&](int rb) {
            if (CG > 1 && !leader) mbar_arrive_remote(afull0 + 8u * (uint32_t)rb);
            else mbar_arrive(afull0 + 8u * (uint32_t)rb);
        };
        // weight rows of G * ROW bytes: 128-byte swizzle (chunk c at c ^ (r % 8)), 64-byte
        // swizzle (chunk c at c ^ ((r / 2) % 4)) or 32-byte swizzle (chunk c at c ^ ((r / 4) % 2))
        const uint32_t wsw = L::WROW == 128 ? (uint32_t)(r & 7)
                           : L::WROW == 64  ? (uint32_t)((r >> 1) & 3)
                                            : (uint32_t)((r >> 2) & 1);
        // Block scales of this row: the two of stage kb (blocks 2 kb, 2 kb + 1) as an fp16 pair
        // (Q4: stored so; Q8/32: f32, rounded to fp16), loaded two of this group's stages ahead
        const uint32_t* srow = reinterpret_cast<const uint32_t*>(J.ws + n * (p.K / 32)) + k0;
        const float2* srowf = reinterpret_cast<const float2*>(J.wsf + n * (p.K / 32)) + k0;
        auto scale_pair = [&](int kbi) -> uint32_t {
            if (FMT == 0) return __ldg(srow + kbi);
            const float2 f = __ldg(srowf + kbi);
            const __half2 h = __floats2half2_rn(f.x, f.y);
            return *reinterpret_cast<const uint32_t*>(&h);
        };
        uint32_t sc0 = 0, sc1 = 0;
        if (FMT != 1 && row_ok) {
            if (grp < nk) sc0 = scale_pair(grp);
            if (grp + 4 < nk) sc1 = scale_pair(grp + 4);
        }
        // Affine Q4: the offsets of stage kb's two blocks (2 kb, 2 kb + 1: groups of gk blocks,
        // a shift where gk is a power of two) as an fp16 pair, prefetched like the scales
        constexpr bool aff = GU == 2;
        const uint16_t* orow = aff ? p.off + n * (p.K / 32 / p.gk) : nullptr;
        const uint32_t gsh = (p.gk & (p.gk - 1)) == 0 ? (uint32_t)(__ffs(p.gk) - 1) : 32u;
        auto offset_pair = [&](int kbi) -> uint32_t {
            const uint32_t b0 = 2u * (uint32_t)(k0 + kbi);
            const uint32_t g0 = gsh < 32u ? b0 >> gsh : b0 / (uint32_t)p.gk;
            const uint32_t g1 = gsh < 32u ? (b0 + 1u) >> gsh : (b0 + 1u) / (uint32_t)p.gk;
            const uint32_t ua = __ldg(orow + g0);
            const uint32_t ub = g1 == g0 ? ua : (uint32_t)__ldg(orow + g1);
            const __half2 h = __floats2half2_rn(__uint_as_float(ua << 16), __uint_as_float(ub << 16));
            return *reinterpret_cast<const uint32_t*>(&h);
        };
        uint32_t mo0 = 0, mo1 = 0;
        if (aff && row_ok) {
            if (grp < nk) mo0 = offset_pair(grp);
            if (grp + 4 < nk) mo1 = offset_pair(grp + 4);
        }
        // Every group waits for every super-stage in order (decoding only its own stages
        // in it), so each round of each super-slot is waited for in order and a parity
        // wait never mistakes round r for round r - 2, whatever LSS is.
        int s = 0;
        uint32_t ph = 0;
        bool stop = false;
        for (int j = 0; j < ns && !stop; ++j) {
          if (!mbar_wait_spin(full_bar(s), ph, p.wait_ns, abort_flag)) {
              give_up();
              break;
          }
#pragma unroll
          for (int u = 0; u < G; ++u) {
            const int kb = j * G + u;
            if ((kb & 3) != grp) continue;
            const int a = kb % AS;                             // decoded slot
            const int rb = (kb / RS) % NRB;                    // its round's barriers
            const uint32_t rph = (uint32_t)((kb / AS) & 1);    // and their phase
            uint32_t sc_next = 0, mo_next = 0;
            if (FMT != 1 && row_ok && kb + 8 < nk) sc_next = scale_pair(kb + 8);
            if (aff && row_ok && kb + 8 < nk) mo_next = offset_pair(kb + 8);
            const uint32_t wrow = slot_base(s) + (uint32_t)(L::X_BYTES + r * L::WROW);
            // this thread's 64 decoded values (the whole stage for row r), two per word
            uint32_t o[32];
            if (FMT == 0) {
                // stage u = chunks 2u, 2u + 1 (one 32-k block each) of the row.  Each block is
                // decoded in the activations' streaming order (the guard pass wrote them in
                // that order): columns 16 b .. 16 b + 15 for block b.
                const uint4 v0 = ld_shared_v4(wrow + (((uint32_t)(2 * u) ^ wsw) << 4));
                const uint4 v1 = ld_shared_v4(wrow + (((uint32_t)(2 * u + 1) ^ wsw) << 4));
                // the block scales, each in both halves of a register
                const uint32_t s0 = prmt(sc0, sc0, 0x1010u), s1 = prmt(sc0, sc0, 0x3232u);
                if (aff) {   // and the two offsets
                    const uint32_t ma = prmt(mo0, mo0, 0x1010u), mb = prmt(mo0, mo0, 0x3232u);
                    decode_q4_word_scaled_off(v0.x, s0, ma, o);
                    decode_q4_word_scaled_off(v0.y, s0, ma, o + 4);
                    decode_q4_word_scaled_off(v0.z, s0, ma, o + 8);
                    decode_q4_word_scaled_off(v0.w, s0, ma, o + 12);
                    decode_q4_word_scaled_off(v1.x, s1, mb, o + 16);
                    decode_q4_word_scaled_off(v1.y, s1, mb, o + 20);
                    decode_q4_word_scaled_off(v1.z, s1, mb, o + 24);
                    decode_q4_word_scaled_off(v1.w, s1, mb, o + 28);
                } else {
                    decode_q4_word_scaled(v0.x, s0, o);
                    decode_q4_word_scaled(v0.y, s0, o + 4);
                    decode_q4_word_scaled(v0.z, s0, o + 8);
                    decode_q4_word_scaled(v0.w, s0, o + 12);
                    decode_q4_word_scaled(v1.x, s1, o + 16);
                    decode_q4_word_scaled(v1.y, s1, o + 20);
                    decode_q4_word_scaled(v1.z, s1, o + 24);
                    decode_q4_word_scaled(v1.w, s1, o + 28);
                }
            } else {
                // stage u = chunks 4u .. 4u + 3 of the row, in k order; Q8/32: chunks 0, 1 are
                // block 2 kb, chunks 2, 3 block 2 kb + 1, each pair times its fp16 block scale
                // (one rounding of q * fp16(scale))
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = ld_shared_v4(wrow + (((uint32_t)(4 * u + c) ^ wsw) << 4));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                    const uint32_t sh2 = FMT == 2 ? prmt(sc0, sc0, c < 2 ? 0x1010u : 0x3232u) : 0u;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (XBF) {
                            o[8 * c + 2 * i] = i8x2_to_bf2(wv[i], 0x4140u);
                            o[8 * c + 2 * i + 1] = i8x2_to_bf2(wv[i], 0x4342u);
                        } else if (FMT == 2) {
                            o[8 * c + 2 * i] = mul_f16x2(i8x2_to_h2(wv[i], 0x4140u), sh2);
                            o[8 * c + 2 * i + 1] = mul_f16x2(i8x2_to_h2(wv[i], 0x4342u), sh2);
                        } else {
                            o[8 * c + 2 * i] = i8x2_to_h2(wv[i], 0x4140u);
                            o[8 * c + 2 * i + 1] = i8x2_to_h2(wv[i], 0x4342u);
                        }
                    }
                }
            }
            // Only the store waits for the decoded slot: the slot's previous round (NRB back)
            // must have been consumed.  The loads and the decode above read the super-slot,
            // which stays full until this stage's MMAs are done, so they run ahead of it.
            const int rp = kb / RS - NRB;
            const bool freed = MERGE ? (rp < 0 || mbar_wait_spin(empty_bar(rp % LSS), (uint32_t)((rp / LSS) & 1), p.wait_ns, abort_flag))
                                     : mbar_wait_spin(aempty_bar(rb), rph ^ 1u, p.wait_ns, abort_flag);
            if (!freed) {
                give_up();
                stop = true;
                break;
            }
            tc_fence_after();   // the slot's earlier MMAs (committed by this or the pair's CTA) are done
            if (AM == 0) {
                // shared-memory A tile, 128-byte swizzled K-major: the 8 chunks of row r
                const uint32_t adst = sb + L::A_OFF + a * A_BYTES + (uint32_t)(r * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(adst + ((((uint32_t)c) ^ xr) << 4), o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                fence_proxy_async_smem();
            } else {
                // tensor-memory A tile: lane r, columns A_COL + 32 a .. +31
                tmem_st_32x32b_x32(tmem + t_lane + (uint32_t)(L::A_COL + a * 32), o);
                tmem_st_wait();
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) announce(rb);
            sc0 = sc1;
            sc1 = sc_next;
            mo0 = mo1;
            mo1 = mo_next;
          }
          if (++s == LSS) {
              s = 0;
              ph ^= 1u;
          }
        }
        // A short last round: the groups without a stage in it still arrive (after the
        // round NRB back has freed the barrier), so the MMA thread's wait completes.
        for (int kb = nk; kb < (nk + RS - 1) / RS * RS && !stop && !*abort_flag; ++kb) {
            if ((kb & 3) != grp) continue;
            const int rb = (kb / RS) % NRB;
            const int rp = kb / RS - NRB;
            const bool freed = MERGE ? (rp < 0 || mbar_wait(empty_bar(rp % LSS), (uint32_t)((rp / LSS) & 1), p.wait_ns, abort_flag))
                                     : mbar_wait(aempty_bar(rb), (uint32_t)(((kb / AS) & 1) ^ 1), p.wait_ns, abort_flag);
            if (!freed) {
                give_up();
                break;
            }
            __syncwarp();
            if (lane == 0) announce(rb);
        }

        // Output scales of the epilogue (Q4: the guard inverse of each token this thread's
        // group finishes, lane l holding columns l and 32 + l; Q8: the row scale), read
        // while the last MMAs run.  Outputs and guard scales only after the previous
        // kernel has finished.
        pdl_wait();
        if (FMT != 1 || J.rsx) {
            const int64_t tb = (int64_t)t0 + cbase + grp * CW;
            if (grp < NG && lane < CW && tb + lane < p.T) etk0 = J.rsx[tb + lane];
            if (grp < NG && CW > 32 && tb + 32 + lane < p.T) etk1 = J.rsx[tb + 32 + lane];
        }
        if (FMT == 1 && row_ok) erow = J.rs[n];
        // the accumulator is complete once the MMA thread's last commit arrives
        if (!*abort_flag && !mbar_wait(accf_bar, 0, p.wait_ns, abort_flag)) give_up();
        tc_fence_after();
    }

    // ================= epilogue (every thread reaches it) =================
    // The decoder warps read the accumulator (warp w: TMEM lanes 32 (w % 4).., the CW
    // columns of its group g = w / 4, CH at a time), scale it and stage each chunk in the
    // idle ring memory as [token][128 rows] in the output type; after a barrier of the
    // group's four warps its first thread stores the chunk with TMA (rows and tokens
    // outside Y are clipped), so the stores overlap the staging of later chunks.  When
    // Y's row pitch is not a multiple of 16 bytes the decoders store element by element.
    // Split K: after a first cluster barrier both CTAs' MMAs are done and their rings
    // idle; the CTA of k half z finishes columns [z BN/2, (z + 1) BN/2).  Each stages the other half of
    // its accumulator ([column][128 rows] f32) chunk by chunk, and the group's first
    // thread copies each chunk in bulk into the partner, completing on the partner's
    // exchange barrier of the same group, so each group finishes as soon as its own
    // columns are in.  The sum is own + partner (a + b, the same in both orders).  A
    // thread arrives on a second cluster barrier once its group's columns are in and
    // waits on it before exiting, so no copy still reads the memory of a CTA that has left.
    // Barriers are taken by every decoder warp whatever the abort flag; only the copies
    // and stores are skipped after a timeout.
    {
        constexpr int HALF = BN / 2;
        constexpr uint32_t SEND_OFF = 0;              // split K: outgoing half
        constexpr uint32_t RECV_OFF = HALF * 128 * 4; //          incoming half
        constexpr uint32_t YST_OFF = KS > 1 ? 2 * HALF * 128 * 4 : 0;   // staged output tile
        const bool dec = warp < DEC_WARPS;
        const int q4w = warp & 3, grp = warp >> 2;
        const int r = 32 * q4w + lane;
        const uint32_t t_lane = (uint32_t)(32 * q4w) << 16;
        const bool lead = q4w == 0 && lane == 0;     // issues the group's copies and stores
        const int gbar = 2 + grp;                    // the group's named barrier (1 is all decoders)
        if (KS > 1) {
            const uint32_t partner = crank ^ (uint32_t)CG;
            // both CTAs past their last MMAs (each waited for its accumulator barrier), so their
            // rings are idle: arrivals without release, the exchange itself completes on mbarriers
            cluster_arrive_relaxed();
            cluster_wait_acquire();
            // each group receives the partner's values of its own CW columns
            if (dec && grp < NG && lead) mbar_arrive_expect_tx(xchg_bar(grp), (uint32_t)(CW * 128 * 4));
            if (dec && grp < NG) {
                const int hb = (kz ^ 1) * HALF;         // the columns the partner finishes
                uint32_t* st = reinterpret_cast<uint32_t*>(smem + SEND_OFF);
#pragma unroll 1
                for (int cc = grp * CW; cc < (grp + 1) * CW; cc += CH) {
                    uint32_t v[CH];
                    tmem_ld_cols<CH>(tmem + t_lane + (uint32_t)(hb + cc), v);
                    tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < CH; ++jj) st[(cc + jj) * 128 + r] = v[jj];
                    fence_proxy_async_smem();
                    named_bar_sync(gbar, 128);
                    if (lead && !*abort_flag)
                        bulk_copy_to_cluster(mapa_shared(sb + RECV_OFF + (uint32_t)(cc * 512), partner),
                                             sb + SEND_OFF + (uint32_t)(cc * 512), (uint32_t)(CH * 512),
                                             mapa_shared(xchg_bar(grp), partner));
                }
                if (!*abort_flag && !mbar_wait(xchg_bar(grp), 0, p.wait_ns, abort_flag)) give_up();
            }
            cluster_arrive_relaxed();
        } else if (CG > 1) {
            // neither CTA of a pair leaves before the other is done; every MMA of the pair has
            // finished (the accumulator barrier), so nothing of one is read by the other any more
            cluster_arrive_relaxed();
        }
        if (dec && grp < NG) {
            const int64_t n = (int64_t)m0 + r;
            const bool row_ok = n < p.N;
            const float* recv = reinterpret_cast<const float*>(smem + RECV_OFF);
            const bool f32 = p.yt == CQ_F32;
            const int esz = f32 ? 4 : 2;
            // the addend (affine offset term) only where a format uses it: its loads stay out of
            // the loop that stages the outputs
            const float* addp = (FMT != 1 && GU != 1 && row_ok) ? J.add : nullptr;
            // every column of the group out of tensor memory at once, one wait
            uint32_t vall[CW];
#pragma unroll
            for (int ci = 0; ci < CW / CH; ++ci)
                tmem_ld_cols<CH>(tmem + t_lane + (uint32_t)(cbase + grp * CW + ci * CH),
                                 *reinterpret_cast<uint32_t(*)[CH]>(&vall[ci * CH]));
            tmem_ld_wait();
#pragma unroll
            for (int ci = 0; ci < CW / CH; ++ci) {
                const int cc = grp * CW + ci * CH;
                const uint32_t* v = &vall[ci * CH];
                const int64_t tb = (int64_t)t0 + cbase + cc;
                const bool skip = *abort_flag != 0;
                float vals[CH];
#pragma unroll
                for (int jj = 0; jj < CH; ++jj) {
                    // column ci CH + jj of the group: its token scale sits in lane (column % 32) of
                    // etk0 (columns 0..31) or etk1 (32..63)
                    const int gc = ci * CH + jj;
                    const float tsc = __shfl_sync(0xffffffffu, gc < 32 ? etk0 : etk1, gc & 31);
                    float acc = __uint_as_float(v[jj]);
                    if (KS > 1) acc += recv[(cc + jj) * 128 + r];
                    vals[jj] = acc * tsc;
                    if (FMT == 1) vals[jj] *= erow;
                }
                if (addp) {
#pragma unroll
                    for (int jj = 0; jj < CH; ++jj)
                        if (tb + jj < p.T) vals[jj] += addp[(tb + jj) * p.N + n];
                }
#pragma unroll
                for (int jj = 0; jj < CH; ++jj) {
                    const int64_t t = tb + jj;
                    const float val = vals[jj];
                    if (GU == 1) {
                        reinterpret_cast<float*>(smem + YST_OFF)[(cc + jj) * 128 + r] = val;
                    } else if (p.y_tma) {
                        if (f32) reinterpret_cast<float*>(smem + YST_OFF)[(cc + jj) * 128 + r] = val;
                        else reinterpret_cast<__nv_bfloat16*>(smem + YST_OFF)[(cc + jj) * 128 + r] = __float2bfloat16_rn(val);
                    } else if (!skip && row_ok && t < p.T) {
                        if (f32) reinterpret_cast<float*>(J.y)[t * p.ldy + n] = val;
                        else reinterpret_cast<__nv_bfloat16*>(J.y)[t * p.ldy + n] = __float2bfloat16_rn(val);
                    }
                }
                if (GU == 1) {
                    // SwiGLU over the staged chunk: gate rows in staged rows 0..63, up rows in
                    // 64..127; thread (q4w, lane) takes gate row i = lane + 32 (q4w % 2) and the
                    // chunk's columns q4w / 2, q4w / 2 + 2, ...  a[t][m0 + i] in f32, coalesced
                    // along i.  (Each chunk has its own staging columns: no reuse hazard.)
                    named_bar_sync(gbar, 128);
                    const int i = lane + 32 * (q4w & 1);
                    const int64_t gi = (int64_t)m0 + i;
                    const float* stg = reinterpret_cast<const float*>(smem + YST_OFF);
#pragma unroll
                    for (int m = 0; m < CH / 2; ++m) {
                        const int jj = (q4w >> 1) + 2 * m;
                        const int64_t t = tb + jj;
                        const float g = stg[(cc + jj) * 128 + i], u = stg[(cc + jj) * 128 + BM / 2 + i];
                        if (!skip && gi < p.N && t < p.T)
                            reinterpret_cast<float*>(J.y)[t * p.ldy + gi] = g / (1.0f + expf(-g)) * u;
                    }
                } else if (p.y_tma) {
                    fence_proxy_async_smem();
                    named_bar_sync(gbar, 128);
                    if (lead && !*abort_flag) {
                        tma_store_2d(tmY, sb + YST_OFF + (uint32_t)(cc * 128 * esz), m0, (int)tb);
                        bulk_commit();
                    }
                }
            }
            if (lead) bulk_wait_read0();   // the staging memory must stay valid until TMA has read it
        }
        if (KS > 1 || CG > 1) cluster_wait_acquire();
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        if (*abort_flag && lane == 0) mbar_wait(accf_bar, 0, p.wait_ns, never_flag);  // MMAs done
        __syncwarp();
        tc_fence_after();
        if (CG > 1) tmem_dealloc_pair(tmem, L::TMEM_COLS);
        else tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

template <int FMT, int BN, int XBF, int G, int LSS, int AS, int AM, int KS = 1, int CG = 1, int GU = 0>
cudaError_t launch_bn(const TcArgs& a, const Params& p, dim3 grid, cudaStream_t s) {
    using L = Layout<FMT, BN, G, LSS, AS, AM, CG>;
    static_assert(CG == 1 || (CG == 2 && AM == 1 && BN >= 32), "CTA pairs: decoded weights in tensor memory");
    static_assert(L::TOTAL <= 232448, "shared memory budget");
    // epilogue staging (f32 at most) below the barriers: split K needs the outgoing and the
    // incoming half and the staged output half; otherwise the staged output tile
    static_assert(L::S_OFF + LSS * L::SLOT >= (KS > 1 ? 3 * (BN / 2) * 128 * 4 : BN * 128 * 4),
                  "epilogue staging fits in the ring memory");
    static_assert(2 * LSS <= 32, "two producer lanes per super-slot");
    // Group g decodes the stages kb % 4 == g, in rounds of RS = 2 or 4 stages, NRB = AS / RS
    // rounds in flight: with RS = 4 every group is in every round; with RS = 2 groups 0, 1
    // take the even rounds and 2, 3 the odd ones, so NRB must be even.  Either way each
    // round barrier is waited for by fixed groups, every one of its rounds in order.
    static_assert(AS % L::RS == 0 && (L::RS == 4 || L::NRB % 2 == 0) && (G == 1 || G == 2 || G == 4),
                  "decoded slots owned by fixed decoder groups");
    static_assert(GU == 0 || FMT == 0, "gate/up and affine modes: Q4 weights");
    // weights: rows of G stages (G * ROW bytes) per box
    // one set of tensor maps per job (a z-batched launch holds up to ZMAX jobs of one shape)
    Maps maps;
    memset(&maps, 0, sizeof maps);
    const uint64_t kbytes = FMT == 0 ? (uint64_t)a.K / 2 : (uint64_t)a.K;
    const CUtensorMapSwizzle swz = L::WROW == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : L::WROW == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    const int64_t ldy = a.ldy > 0 ? a.ldy : a.N;
    for (int j = 0; j < a.jobs(); ++j) {
        const TcJob jb = a.job(j);
        if (GU == 1) {
            // [2][I][K bytes]: gate half, up half; one box = 64 gate rows then the 64 matching up rows
            uint64_t d[3] = {kbytes, (uint64_t)a.N, 2};
            uint64_t st[2] = {kbytes, kbytes * (uint64_t)a.N};
            uint32_t box[3] = {(uint32_t)L::WROW, (uint32_t)(BM / 2), 2};
            if (!encode_tiled(&maps.w[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, jb.wq, d, st, box, swz))
                return cudaErrorInvalidValue;
        } else {
            uint64_t d[2] = {kbytes, (uint64_t)a.N};
            uint64_t st[1] = {kbytes};
            uint32_t box[2] = {(uint32_t)L::WROW, (uint32_t)BM};
            if (!encode_tiled(&maps.w[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, jb.wq, d, st, box, swz))
                return cudaErrorInvalidValue;
        }
        // activations seen as {64 elements, T rows, K/64 chunks} (strides K*2 B, 128 B): one
        // box of G chunks of BN / CG rows lands as [chunk][row][128 B], G operand tiles
        {
            uint64_t d[3] = {64, (uint64_t)a.T, (uint64_t)a.K / 64};
            uint64_t st[2] = {(uint64_t)a.K * 2, 128};
            uint32_t box[3] = {64, (uint32_t)(BN / CG), (uint32_t)G};
            if (!encode_tiled(&maps.x[j], XBF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                              jb.x, d, st, box, CU_TENSOR_MAP_SWIZZLE_128B))
                return cudaErrorInvalidValue;
        }
        // output tiles: Y [T][N] (pitch ldy) seen as {N, T}; a box is 128 rows x one epilogue chunk
        if (p.y_tma) {
            const uint64_t es = a.yt == CQ_F32 ? 4 : 2;
            uint64_t d[2] = {(uint64_t)a.N, (uint64_t)a.T};
            uint64_t st[1] = {(uint64_t)ldy * es};
            uint32_t box[2] = {(uint32_t)BM, (uint32_t)ep_chunk(BN, KS)};
            if (!encode_tiled(&maps.y[j], a.yt == CQ_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              2, jb.y, d, st, box, CU_TENSOR_MAP_SWIZZLE_NONE))
                return cudaErrorInvalidValue;
        }
    }
    auto kern = k_tc<FMT, BN, XBF, G, LSS, AS, AM, KS, CG, GU>;
    static int configured_device = -1;       // attributes are per device; set once per instantiation
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = L::TOTAL;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (KS > 1 || CG > 1) {
        if (grid.x % CG != 0) return cudaErrorInvalidValue;
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = CG;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = KS;
        ++na;
    }
    if (p.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return counted(cudaLaunchKernelEx(&cfg, kern, maps, p));
}

// Tile plan: token tile BN and K split.  One CTA per SM.  Time of a CTA ~ its
// stages x the measured cost of a 64-k stage (clock stamps in the kernel: about
// 520 cycles at BN = 64, 570 at 128 and 800 at 256, 515, 680 and 690 in CTA pairs
// at 128, 192 and 256; 192-column pairs fill the SMs where 256-column tiles leave a
// third idle), plus about 6000 cycles for the exchange when K is split over two
// CTAs; times the waves.  Tiles at least twice as wide as the tokens are not
// considered.  The cheapest candidate wins (ties: the earlier, wider one).
// mt: weight-row tiles (128 rows; in gate/up mode 64 gate + 64 up rows).
struct Plan {
    int bn, ks;
    bool pair_ok;
};
Plan plan_tiles(const TcArgs& a, int64_t mt, bool tmem_only) {
    const int64_t nk = a.K / BK;
    const int amode = tmem_only ? 0 : (int)options().tc_amode;
    int bn = (int)options().tc_bn;
    int ks = (int)options().tc_ksplit;
    if (bn == 32 && amode == 1) bn = 64;   // 32-column tiles keep decoded weights in tensor memory
    if (bn == 192 && !(mt % 2 == 0 && amode != 1 && options().tc_pair != 1)) bn = 256;   // pairs only
    if (bn == 192 && options().tc_ksplit == 2) ks = 1;                                    // no K split
    const bool ks2_ok = nk % 8 == 0;
    // 256-column tiles in CTA pairs (one 256-row MMA over two neighbouring row tiles):
    // an even number of row tiles and decoded weights in tensor memory
    const bool pair_ok = mt % 2 == 0 && amode != 1 && options().tc_pair != 1;
    struct Cand { int bn, ks; };
    const Cand cands[] = {{256, 1}, {256, 2}, {192, 1}, {128, 1}, {128, 2}, {64, 1}, {32, 1}, {32, 2}};
    double best = -1.0;
    int bbn = 128, bks = 1;
    for (const Cand& c : cands) {
        if (bn != 0 && c.bn != bn) continue;
        if (ks != 0 && c.ks != ks) continue;
        // at least half of every tile's columns unused: skipped for the wide tiles, whose stages cost
        // more; narrow tiles cost about the same per stage whatever their width (measured), so the
        // cost model decides among them
        if (bn == 0 && 2 * a.T <= c.bn && c.bn >= 192) continue;
        if (c.bn == 32 && amode == 1) continue;
        // split only to fill the GPU: when the unsplit tiles leave a quarter of the SMs idle
        if (c.ks == 2 && (!ks2_ok || (ks == 0 && mt * ((a.T + c.bn - 1) / c.bn) * a.jobs() * 4 > 3 * num_sms()))) continue;
        if (c.bn == 192 && c.ks != 1) continue;
        if (c.bn == 192 && !pair_ok) continue;   // 192-column tiles only in CTA pairs
        // measured cycles per 64-k stage (N = K = 8192; 32-column pairs about 550, T = 32-64)
        const double stage = c.bn == 256 ? (pair_ok ? 690.0 : 800.0) : c.bn == 192 ? 680.0
                           : c.bn == 128 ? (pair_ok ? 515.0 : 570.0) : c.bn == 64 ? 520.0 : (pair_ok ? 560.0 : 530.0);
        const int64_t ctas = mt * ((a.T + c.bn - 1) / c.bn) * c.ks * a.jobs();
        const int64_t waves = (ctas + num_sms() - 1) / num_sms();
        const double cost = (double)waves * ((double)(nk / c.ks) * stage + (c.ks > 1 ? 6000.0 : 0.0));
        if (best < 0.0 || cost < best - 1e-9) {
            best = cost;
            bbn = c.bn;
            bks = c.ks;
        }
    }
    if (best < 0.0) {   // a forced combination that cannot run: fall back to no split
        bbn = bn != 0 ? bn : 128;
        bks = 1;
    }
    return {bbn, bks, pair_ok};
}

// Weight-row tiles to move into a second launch that splits K over a cluster, so
// that the first launch fills whole waves of the GPU: a last wave that would hold
// only a few tiles (each as long as a full one) becomes a launch of those row
// tiles at half their length, in the narrowest token tiles that still fit in one
// wave (narrow tiles cost less per stage).  r = 0 when there is nothing to gain or
// the tile shape has no K-split form.
struct Tail {
    int64_t r;   // row tiles of the tail launch (the last r)
    int bn;      // its token-tile width
};
Tail tail_plan(const Plan& pl, bool pair, int64_t mt, int64_t T, int64_t jobs, int64_t K) {
    const int64_t nk = K / BK;
    if (pl.ks != 1 || !(pl.bn == 256 || pl.bn == 128 || pl.bn == 32) || nk % 8 != 0 || nk < 24) return {0, 0};
    const int64_t sms = num_sms(), cols = (T + pl.bn - 1) / pl.bn * jobs, ctas = mt * cols;
    if (ctas <= sms || ctas % sms == 0) return {0, 0};
    int64_t r = (ctas % sms + cols - 1) / cols;   // row tiles of the partial last wave
    if (pair) r = (r + 1) & ~(int64_t)1;          // CTA pairs take neighbouring row tiles
    if (r >= mt) return {0, 0};
    for (int bn : {32, 128, 256}) {
        if (bn > pl.bn) break;
        if (2 * r * ((T + bn - 1) / bn) * jobs <= sms) return {r, bn};
    }
    return {0, 0};
}

Params make_params(const TcArgs& a) {
    Params p = {};
    for (int j = 0; j < a.jobs(); ++j) {
        const TcJob jb = a.job(j);
        p.job[j] = {jb.rsx, jb.rs, jb.ws, jb.wsf, jb.add, jb.y};
    }
    p.off = a.jobs() == 1 ? a.off : nullptr;
    p.gk = a.gk > 0 ? a.gk : 1;
    p.mt0 = 0;
    p.tiles_y = 1;
    p.ldy = a.ldy > 0 ? a.ldy : a.N;
    p.yt = a.yt;
    p.T = a.T;
    p.N = a.N;
    p.K = a.K;
    p.wait_ns = (uint64_t)options().wait_ns;
    p.stall = (int)options().test_stall.exchange(0);
    p.pdl = 1;   // the guard pass (Q4) or the previous kernel touches neither the weights nor anything before the wait
    // every job's output tiles leave through TMA stores when every row pitch and base is 16-byte aligned
    p.y_tma = (p.ldy * (a.yt == CQ_F32 ? 4 : 2)) % 16 == 0 ? 1 : 0;
    for (int j = 0; j < a.jobs(); ++j)
        if (reinterpret_cast<uintptr_t>(a.job(j).y) & 15) p.y_tma = 0;
    p.err = a.err;
    return p;
}

void trace_plan(const char* what, int fmt, const TcArgs& a, const Plan& pl, bool pair, dim3 grid) {
    if (options().trace)
        fprintf(stderr, "cq: tcgen05 %s fmt=%d T=%lld N=%lld K=%lld BN=%d ksplit=%d pair=%d grid=(%u,%u,%u)\n", what,
                fmt, (long long)a.T, (long long)a.N, (long long)a.K, pl.bn, pl.ks, (int)pair, grid.x, grid.y, grid.z);
}

// Q4 with the decoded weights in tensor memory, every tile shape; GU selects the
// gate/up (SwiGLU, 1) or the affine (2) mode.  <FMT, BN, XBF, G, LSS, AS, AM, KS, CG, GU>: super-stages
// of G stages, as many super-slots as fit next to the decoded slots.
template <int GU>
cudaError_t launch_q4_tmem_one(const TcArgs& a, const Params& p, const Plan& pl, dim3 grid, cudaStream_t s) {
    const int bn = pl.bn, ks = pl.ks;
    const bool pair = (bn >= 128 || bn == 32) && pl.pair_ok;
    if (bn == 192) return launch_bn<0, 192, 0, 4, 3, 8, 1, 1, 2, GU>(a, p, grid, s);
    if (bn == 32) {
        if (pair) return ks == 2 ? launch_bn<0, 32, 0, 4, 8, 12, 1, 2, 2, GU>(a, p, grid, s) : launch_bn<0, 32, 0, 4, 8, 12, 1, 1, 2, GU>(a, p, grid, s);
        return ks == 2 ? launch_bn<0, 32, 0, 4, 6, 12, 1, 2, 1, GU>(a, p, grid, s) : launch_bn<0, 32, 0, 4, 6, 12, 1, 1, 1, GU>(a, p, grid, s);
    }
    if (pair && bn == 128) return ks == 2 ? launch_bn<0, 128, 0, 4, 4, 12, 1, 2, 2, GU>(a, p, grid, s) : launch_bn<0, 128, 0, 4, 4, 12, 1, 1, 2, GU>(a, p, grid, s);
    if (pair) return ks == 2 ? launch_bn<0, 256, 0, 2, 5, 8, 1, 2, 2, GU>(a, p, grid, s) : launch_bn<0, 256, 0, 2, 5, 8, 1, 1, 2, GU>(a, p, grid, s);
    if (bn == 256) return ks == 2 ? launch_bn<0, 256, 0, 2, 3, 8, 1, 2, 1, GU>(a, p, grid, s) : launch_bn<0, 256, 0, 2, 3, 8, 1, 1, 1, GU>(a, p, grid, s);
    if (bn == 128) return ks == 2 ? launch_bn<0, 128, 0, 2, 5, 12, 1, 2, 1, GU>(a, p, grid, s) : launch_bn<0, 128, 0, 2, 5, 12, 1, 1, 1, GU>(a, p, grid, s);
    return launch_bn<0, 64, 0, 4, 4, 12, 1, 1, 1, GU>(a, p, grid, s);
}

// grid = (row tiles, token tiles x jobs, K split); the last row tiles may go to a second,
// K-split launch (tail_row_tiles)
template <int GU>
cudaError_t launch_q4_tmem(const TcArgs& a, const Params& p, const Plan& pl, dim3 grid, cudaStream_t s) {
    const bool pair = (pl.bn >= 128 || pl.bn == 32) && pl.pair_ok;
    const Tail tl = tail_plan(pl, pair, grid.x, a.T, a.jobs(), a.K);
    if (tl.r == 0) return launch_q4_tmem_one<GU>(a, p, pl, grid, s);
    cudaError_t e = launch_q4_tmem_one<GU>(a, p, pl, dim3(grid.x - (unsigned)tl.r, grid.y, 1), s);
    if (e != cudaSuccess) return e;
    Params pt = p;
    pt.mt0 = (int)(grid.x - tl.r);
    pt.tiles_y = (int)((a.T + tl.bn - 1) / tl.bn);
    const Plan plt = {tl.bn, 2, pl.pair_ok};
    const dim3 gt((unsigned)tl.r, (unsigned)(pt.tiles_y * a.jobs()), 2);
    trace_plan("tail", 0, a, plt, pair, gt);
    return launch_q4_tmem_one<GU>(a, pt, plt, gt, s);
}

}  // namespace
}  // namespace cq
