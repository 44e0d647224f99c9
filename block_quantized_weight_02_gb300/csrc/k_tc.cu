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
//               (M = 128, N = BN, K = 16) from one thread, committing each
//               stage's decoded slot and each super-stage's load slot back,
//               and the last stage to the epilogue.
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
// Every wait is time-bounded; on a timeout the CTA stops, lets copies in
// flight land, frees its tensor memory and reports CQ_ERR_TIMEOUT.
#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cq_internal.h"
#include "cq_ptx.cuh"

namespace cq {

__device__ int g_err_tc = 0;

int take_error_tc() {
    int v = 0, z = 0;
    cudaMemcpyFromSymbol(&v, g_err_tc, sizeof(int));
    cudaMemcpyToSymbol(g_err_tc, &z, sizeof(int));
    return v;
}

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB

struct Params {
    const float* rsx;
    const float* rs;
    const uint16_t* ws;   // Q4 block scales [N][K/32]
    void* y;
    int yt;
    int64_t T, N, K;
    uint64_t wait_ns;
    int stall;
    int pdl;   // launched with a programmatic dependency on the guard pass
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}
__device__ __forceinline__ uint32_t i8x2_to_h2(uint32_t w, uint32_t sel) {
    const uint32_t h = prmt(w ^ 0x80808080u, 0x64646464u, sel);
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h),
                              __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
// Eight nibbles (bytes b0..b3 of w) -> four fp16 pairs (n - 8) * scale, each
// rounded once, in the activations' streaming order: (low b0, low b2),
// (high b0, high b2), (low b1, low b3), (high b1, high b3).  0x6400 | n is
// 1024 + n and 0x6400 | (n << 4) is 1024 + 16 n; 1024 + n - 1032 and
// (1024 + 16 n) / 16 - 72 are n - 8 exactly.
__device__ __forceinline__ void decode_q4_word_scaled(uint32_t w, __half2 sc, uint32_t* o) {
    const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    const __half2 k16th = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
    const __half2 km72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));
    const uint32_t w8 = w >> 8;
    const uint32_t l02 = (w & 0x000F000Fu) | 0x64006400u, h02 = (w & 0x00F000F0u) | 0x64006400u;
    const uint32_t l13 = (w8 & 0x000F000Fu) | 0x64006400u, h13 = (w8 & 0x00F000F0u) | 0x64006400u;
    const __half2 d0 = __hsub2(*reinterpret_cast<const __half2*>(&l02), k1032);
    const __half2 d1 = __hfma2(*reinterpret_cast<const __half2*>(&h02), k16th, km72);
    const __half2 d2 = __hsub2(*reinterpret_cast<const __half2*>(&l13), k1032);
    const __half2 d3 = __hfma2(*reinterpret_cast<const __half2*>(&h13), k16th, km72);
    const __half2 r0 = __hmul2(d0, sc), r1 = __hmul2(d1, sc), r2 = __hmul2(d2, sc), r3 = __hmul2(d3, sc);
    o[0] = *reinterpret_cast<const uint32_t*>(&r0);
    o[1] = *reinterpret_cast<const uint32_t*>(&r1);
    o[2] = *reinterpret_cast<const uint32_t*>(&r2);
    o[3] = *reinterpret_cast<const uint32_t*>(&r3);
}

template <int FMT>
struct Raw;
template <>
struct Raw<0> { static constexpr int ROW = 32; };   // Q4: 64 k = 32 bytes per row and stage
template <>
struct Raw<1> { static constexpr int ROW = 64; };   // Q8: 64 bytes per row and stage

// Loads come in super-stages of G stages (G x 64 k), two TMA boxes each: a TMA
// box costs about the same however few bytes it holds, so the weight rows are
// fetched G stages at a time (G * ROW bytes per row) and the activation tile as
// one 3-D box of G 64-k chunks.
// Shared memory per super-slot: X [G][BN rows][128 B] (each chunk one
// 128-byte-swizzled K-major operand tile), then W [128 rows][G * ROW B]
// (128- or 64-byte swizzle).  AM 0 adds AS decoded tiles [128][128 B] in
// front; AM 1 keeps the decoded tiles in tensor memory.
template <int FMT, int BN, int G, int LSS, int AS, int AM>
struct Layout {
    static constexpr int WROW = G * Raw<FMT>::ROW;            // 64 or 128 bytes
    static constexpr int X_CHUNK = BN * 128;
    static constexpr int X_BYTES = G * X_CHUNK;
    static constexpr int W_BYTES = BM * WROW;
    static constexpr int SLOT = X_BYTES + W_BYTES;             // multiple of 1024
    static constexpr int A_OFF = 0;
    static constexpr int S_OFF = AM == 0 ? AS * A_BYTES : 0;
    static constexpr int BAR_OFF = S_OFF + LSS * SLOT;
    // full[LSS], empty[LSS], afull[AS], aempty[AS / 2] (one per pair of decoded slots), accf;
    // then tmem slot, abort, never
    static constexpr int NBAR = 2 * LSS + AS + AS / 2 + 1;
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

constexpr int DEC_WARPS = 16;                // 4 groups (stages kb % 4) x 4 row quarters
constexpr int THREADS = (DEC_WARPS + 2) * 32;
constexpr int PRODUCER_WARP = DEC_WARPS;
constexpr int MMA_WARP = DEC_WARPS + 1;

// int8 pair (bytes sel of w) -> bf16x2 exactly: with 0x43 as the high byte, the
// low seven bits of v give 128 + (v & 127) and the sign bit gives 128 or 256
// (0x4300 / 0x4380); their difference is v, an integer bf16 holds exactly.
__device__ __forceinline__ uint32_t i8x2_to_bf2(uint32_t w, uint32_t sel) {
    const uint32_t t = prmt(w, 0x43434343u, sel);
    const uint32_t lo = t & 0xFF7FFF7Fu, hi = t & 0xFF80FF80u;
    const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&lo),
                                     *reinterpret_cast<const __nv_bfloat162*>(&hi));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// KS: K split over a cluster of KS CTAs along z (1 or 2); the two partial
// accumulators are exchanged through distributed shared memory and each CTA
// finishes half of the tile's columns.
template <int FMT, int BN, int XBF, int G, int LSS, int AS, int AM, int KS>
__global__ void __launch_bounds__(THREADS, 1)
k_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const Params p) {
    using L = Layout<FMT, BN, G, LSS, AS, AM>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM;          // first weight row
    const int t0 = blockIdx.y * BN;          // first activation row
    const int kz = KS > 1 ? (int)blockIdx.z : 0;
    const int nk = (int)(p.K / BK) / KS;     // stages of this CTA's k range
    const int k0 = kz * nk;                  // its first stage
    const int ns = nk / G;                   // super-stages
    const int j0 = k0 / G;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (LSS + s); };
    auto afull_bar = [&](int a) { return bar0 + 8u * (2 * LSS + a); };
    auto aempty_bar = [&](int pr) { return bar0 + 8u * (2 * LSS + AS + pr); };   // decoded slots 2pr, 2pr + 1
    const uint32_t accf_bar = bar0 + 8u * (2 * LSS + AS + AS / 2);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never_flag = abort_flag + 1;
    auto slot_base = [&](int s) { return sb + (uint32_t)(L::S_OFF + s * L::SLOT); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < LSS; ++s) {
            mbar_init(full_bar(s), 1);   // the weight lane's arrival + both boxes' bytes
            mbar_init(empty_bar(s), 1);  // the MMA's commit after the super-stage's last stage
        }
        for (int a = 0; a < AS; ++a) mbar_init(afull_bar(a), 4);       // one arrival per warp of the decoding group
        for (int pr = 0; pr < AS / 2; ++pr) mbar_init(aempty_bar(pr), 1);  // the MMA's commit of the stage pair
        mbar_init(accf_bar, 1);
        *abort_flag = 0;
        *never_flag = 0;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto give_up = [&]() {
        *abort_flag = 1;
        atomicCAS(&g_err_tc, 0, DEV_TIMEOUT);
    };

    if (warp == PRODUCER_WARP) {
        // ================= TMA producers =================
        // Lane s < LSS issues the weight box of super-slot s (and posts the bytes of
        // both boxes), lane LSS + s its activation box: a thread keeps only a few bulk
        // copies in flight, so the boxes come from 2 LSS threads.
        const int s = lane % LSS;
        const bool wl = lane < LSS, xl = lane >= LSS && lane < 2 * LSS;
        if (wl || xl) {
            if (lane == 0) {
                tma_prefetch_desc(&tmW);
                tma_prefetch_desc(&tmX);
            }
            const uint32_t base = slot_base(s);
            int issued = 0;        // super-stages issued by this lane
            auto issue = [&](int j) {
                if (wl) {
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)(L::X_BYTES + L::W_BYTES));
                    tma_load_2d(base + L::X_BYTES, &tmW, full_bar(s), (j0 + j) * L::WROW, m0);
                } else {
                    tma_load_3d(base, &tmX, full_bar(s), 0, t0, (j0 + j) * G);
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
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BM, BN, XBF);
            int a = 0, s = 0, u = 0;          // decoded slot, super-slot and chunk of stage kb
            uint32_t aph = 0;
            for (int kb = 0; kb < nk; kb += 2) {
                if (!mbar_wait(afull_bar(a), aph, p.wait_ns, abort_flag) ||
                    !mbar_wait(afull_bar(a + 1), aph, p.wait_ns, abort_flag)) {
                    give_up();
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint64_t bd = smem_desc_sw128(slot_base(s) + (uint32_t)(u * L::X_CHUNK));
                    const uint64_t ad = AM == 0 ? smem_desc_sw128(sb + L::A_OFF + (a + h) * A_BYTES) : 0;
                    const uint32_t at = tmem + (uint32_t)(L::A_COL + (a + h) * 32);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint32_t acc = (kb + h + kk) != 0 ? 1u : 0u;
                        // +32 bytes of K = +2 in the descriptor's 16-byte address units
                        if (AM == 0) tc_mma_f16(tmem, ad + 2u * kk, bd + 2u * kk, idesc, acc);
                        else tc_mma_f16_ts(tmem, at + 8u * kk, bd + 2u * kk, idesc, acc);
                    }
                    if (++u == G) {
                        u = 0;
                        tc_commit(empty_bar(s));                // super-slot free after its last stage
                        if (++s == LSS) s = 0;
                    }
                }
                tc_commit(aempty_bar(a >> 1));                  // decoded slots a, a + 1 free
                a += 2;
                if (a == AS) { a = 0; aph ^= 1u; }
            }
            tc_commit(accf_bar);   // also lets teardown know every MMA has finished
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
        const int64_t n = (int64_t)m0 + r;
        const bool row_ok = n < p.N;
        const uint32_t xr = (uint32_t)(r & 7);
        const uint32_t t_lane = (uint32_t)(32 * q4w) << 16;
        // weight rows of G * ROW bytes: 128-byte swizzle (chunk c at c ^ (r % 8)), 64-byte
        // swizzle (chunk c at c ^ ((r / 2) % 4)) or 32-byte swizzle (chunk c at c ^ ((r / 4) % 2))
        const uint32_t wsw = L::WROW == 128 ? (uint32_t)(r & 7)
                           : L::WROW == 64  ? (uint32_t)((r >> 1) & 3)
                                            : (uint32_t)((r >> 2) & 1);
        // Q4 scales of this row: the two fp16 of stage kb (blocks 2 kb, 2 kb + 1), loaded two
        // of this group's stages ahead
        const uint32_t* srow = reinterpret_cast<const uint32_t*>(p.ws + n * (p.K / 32)) + k0;
        uint32_t sc0 = 0, sc1 = 0;
        if (FMT == 0 && row_ok) {
            if (grp < nk) sc0 = __ldg(srow + grp);
            if (grp + 4 < nk) sc1 = __ldg(srow + grp + 4);
        }
        // Every group waits for every super-stage in order (decoding only its own stages
        // in it), so each round of each super-slot is waited for in order and a parity
        // wait never mistakes round r for round r - 2, whatever LSS is.
        int s = 0;
        uint32_t ph = 0;
        bool stop = false;
        for (int j = 0; j < ns && !stop; ++j) {
          if (!mbar_wait(full_bar(s), ph, p.wait_ns, abort_flag)) {
              give_up();
              break;
          }
#pragma unroll
          for (int u = 0; u < G; ++u) {
            const int kb = j * G + u;
            if ((kb & 3) != grp) continue;
            const int a = kb % AS;                             // decoded slot
            const uint32_t aph = (uint32_t)((kb / AS) & 1);
            uint32_t sc_next = 0;
            if (FMT == 0 && row_ok && kb + 8 < nk) sc_next = __ldg(srow + kb + 8);
            if (!mbar_wait(aempty_bar(a >> 1), aph ^ 1u, p.wait_ns, abort_flag)) {
                give_up();
                stop = true;
                break;
            }
            const uint32_t wrow = slot_base(s) + (uint32_t)(L::X_BYTES + r * L::WROW);
            // this thread's 64 decoded values (the whole stage for row r), two per word
            uint32_t o[32];
            if (FMT == 0) {
                // stage u = chunks 2u, 2u + 1 (one 32-k block each) of the row.  Each block is
                // decoded in the activations' streaming order (the guard pass wrote them in
                // that order): columns 16 b .. 16 b + 15 for block b.
                const uint4 v0 = ld_shared_v4(wrow + (((uint32_t)(2 * u) ^ wsw) << 4));
                const uint4 v1 = ld_shared_v4(wrow + (((uint32_t)(2 * u + 1) ^ wsw) << 4));
                const __half2 s0 = __halves2half2(__ushort_as_half((uint16_t)(sc0 & 0xFFFF)),
                                                  __ushort_as_half((uint16_t)(sc0 & 0xFFFF)));
                const __half2 s1 = __halves2half2(__ushort_as_half((uint16_t)(sc0 >> 16)),
                                                  __ushort_as_half((uint16_t)(sc0 >> 16)));
                decode_q4_word_scaled(v0.x, s0, o);
                decode_q4_word_scaled(v0.y, s0, o + 4);
                decode_q4_word_scaled(v0.z, s0, o + 8);
                decode_q4_word_scaled(v0.w, s0, o + 12);
                decode_q4_word_scaled(v1.x, s1, o + 16);
                decode_q4_word_scaled(v1.y, s1, o + 20);
                decode_q4_word_scaled(v1.z, s1, o + 24);
                decode_q4_word_scaled(v1.w, s1, o + 28);
            } else {
                // stage u = chunks 4u .. 4u + 3 of the row, in k order
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = ld_shared_v4(wrow + (((uint32_t)(4 * u + c) ^ wsw) << 4));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (XBF) {
                            o[8 * c + 2 * i] = i8x2_to_bf2(wv[i], 0x4140u);
                            o[8 * c + 2 * i + 1] = i8x2_to_bf2(wv[i], 0x4342u);
                        } else {
                            o[8 * c + 2 * i] = i8x2_to_h2(wv[i], 0x4140u);
                            o[8 * c + 2 * i + 1] = i8x2_to_h2(wv[i], 0x4342u);
                        }
                    }
                }
            }
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
            if (lane == 0) mbar_arrive(afull_bar(a));
            sc0 = sc1;
            sc1 = sc_next;
          }
          if (++s == LSS) {
              s = 0;
              ph ^= 1u;
          }
        }

        // ---- epilogue: TMEM -> registers -> scale -> Y[t][n] ----
        // warp w reads TMEM lanes 32 (w % 4).. and the accumulator columns
        // [g BN/4, (g + 1) BN/4) of its group g = w / 4, 16 at a time
        if (KS > 1) {
            // split K: wait for this CTA's MMAs; the exchange follows below
            if (!*abort_flag && !mbar_wait(accf_bar, 0, p.wait_ns, abort_flag)) give_up();
            tc_fence_after();
        } else if (!*abort_flag && mbar_wait(accf_bar, 0, p.wait_ns, abort_flag)) {
            tc_fence_after();
            pdl_wait();   // outputs and guard scales only after the previous kernel has finished
            const float rsn = (FMT == 1 && row_ok) ? p.rs[n] : 0.f;
            constexpr int CW = BN / 4;
#pragma unroll 1
            for (int cc = grp * CW; cc < (grp + 1) * CW; cc += 16) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem + t_lane + (uint32_t)cc, v);
                tmem_ld_wait();
                const int64_t tb = (int64_t)t0 + cc;
                float rsx_l = 0.f;
                if (FMT == 0 && lane < 16 && tb + lane < p.T) rsx_l = p.rsx[tb + lane];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const float sx = FMT == 0 ? __shfl_sync(0xffffffffu, rsx_l, jj) : rsn;
                    const int64_t t = tb + jj;
                    if (row_ok && t < p.T) {
                        const float val = __uint_as_float(v[jj]) * sx;
                        if (p.yt == CQ_F32) reinterpret_cast<float*>(p.y)[t * p.N + n] = val;
                        else reinterpret_cast<__nv_bfloat16*>(p.y)[t * p.N + n] = __float2bfloat16_rn(val);
                    }
                }
            }
        } else if (!*abort_flag) {
            give_up();
        }
    }

    if (KS > 1) {
        // ---- split-K exchange: every thread of both CTAs passes both cluster barriers ----
        // After the first, both CTAs' MMAs are done and their rings idle.  Rank r finishes
        // columns [r BN/2, (r + 1) BN/2): it sends the other half of its accumulator into
        // the partner's ring memory, then, after the second barrier, adds the partner's
        // half to its own (a + b, the same in both orders).  Buffer: [128 rows][BN/2] f32,
        // 16-byte chunk c of row r stored at chunk c ^ (r % CH) (CH chunks per row), so
        // both the remote 16-byte stores and the local 16-byte loads of a warp's 32 rows
        // spread over the banks.
        constexpr int HALF = BN / 2;
        const uint32_t rank = cluster_ctarank(), partner = rank ^ 1u;
        cluster_sync_all();
        const bool dec = warp < DEC_WARPS;
        const int q4w = warp & 3, grp = warp >> 2;
        const int r = 32 * q4w + lane;
        const uint32_t t_lane = (uint32_t)(32 * q4w) << 16;
        constexpr int CW = HALF / 4;              // columns per decoder group
        constexpr int CH = HALF / 4;              // 16-byte chunks per buffer row
        const uint32_t row_off = (uint32_t)(r * HALF * 4);
        const uint32_t csw = (uint32_t)(r % CH);
        if (dec && !*abort_flag) {
            const uint32_t dst = mapa_shared(sb, partner) + row_off;
            const int hb = (int)partner * HALF;
#pragma unroll 1
            for (int cc = grp * CW; cc < (grp + 1) * CW; cc += 16) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem + t_lane + (uint32_t)(hb + cc), v);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st_cluster_v4(dst + (((uint32_t)(cc / 4 + q) ^ csw) << 4), v[4 * q], v[4 * q + 1], v[4 * q + 2],
                                  v[4 * q + 3]);
            }
        }
        cluster_sync_all();
        if (dec && !*abort_flag) {
            pdl_wait();   // outputs and guard scales only after the previous kernel has finished
            const int64_t n = (int64_t)m0 + r;
            const bool row_ok = n < p.N;
            const float rsn = (FMT == 1 && row_ok) ? p.rs[n] : 0.f;
            const int hb = (int)rank * HALF;
#pragma unroll 1
            for (int cc = grp * CW; cc < (grp + 1) * CW; cc += 16) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem + t_lane + (uint32_t)(hb + cc), v);
                tmem_ld_wait();
                float pr[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = ld_shared_v4(sb + row_off + (((uint32_t)(cc / 4 + q) ^ csw) << 4));
                    pr[4 * q] = __uint_as_float(w.x);
                    pr[4 * q + 1] = __uint_as_float(w.y);
                    pr[4 * q + 2] = __uint_as_float(w.z);
                    pr[4 * q + 3] = __uint_as_float(w.w);
                }
                const int64_t tb = (int64_t)t0 + hb + cc;
                float rsx_l = 0.f;
                if (FMT == 0 && lane < 16 && tb + lane < p.T) rsx_l = p.rsx[tb + lane];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const float sx = FMT == 0 ? __shfl_sync(0xffffffffu, rsx_l, jj) : rsn;
                    const int64_t t = tb + jj;
                    if (row_ok && t < p.T) {
                        const float val = (__uint_as_float(v[jj]) + pr[jj]) * sx;
                        if (p.yt == CQ_F32) reinterpret_cast<float*>(p.y)[t * p.N + n] = val;
                        else reinterpret_cast<__nv_bfloat16*>(p.y)[t * p.N + n] = __float2bfloat16_rn(val);
                    }
                }
            }
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        if (*abort_flag && lane == 0) mbar_wait(accf_bar, 0, p.wait_ns, never_flag);  // MMAs done
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

template <int FMT, int BN, int XBF, int G, int LSS, int AS, int AM, int KS = 1>
cudaError_t launch_bn(const TcArgs& a, const Params& p, dim3 grid, cudaStream_t s) {
    using L = Layout<FMT, BN, G, LSS, AS, AM>;
    static_assert(L::TOTAL <= 232448, "shared memory budget");
    static_assert(KS == 1 || (KS == 2 && L::S_OFF + LSS * L::SLOT >= (BN / 2) * 128 * 4),
                  "the partner's half accumulator fits in the ring memory");
    static_assert(2 * LSS <= 32, "two producer lanes per super-slot");
    // Group g decodes the stages kb % 4 == g: with AS a multiple of 4 each decoded slot
    // (and pair of slots) belongs to fixed groups that wait for its rounds in order.
    static_assert(AS % 4 == 0 && (G == 1 || G == 2 || G == 4), "decoded slots owned by fixed decoder groups");
    // weights: rows of G stages (G * ROW bytes) per box
    CUtensorMap mw, mx;
    {
        const uint64_t kbytes = FMT == 0 ? (uint64_t)a.K / 2 : (uint64_t)a.K;
        uint64_t d[2] = {kbytes, (uint64_t)a.N};
        uint64_t st[1] = {kbytes};
        uint32_t box[2] = {(uint32_t)L::WROW, (uint32_t)BM};
        if (!encode_tiled(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.wq, d, st, box,
                          L::WROW == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : L::WROW == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B))
            return cudaErrorInvalidValue;
    }
    // activations seen as {64 elements, T rows, K/64 chunks} (strides K*2 B, 128 B): one
    // box of G chunks of BN rows lands as [chunk][row][128 B], G operand tiles
    {
        uint64_t d[3] = {64, (uint64_t)a.T, (uint64_t)a.K / 64};
        uint64_t st[2] = {(uint64_t)a.K * 2, 128};
        uint32_t box[3] = {64, (uint32_t)BN, (uint32_t)G};
        if (!encode_tiled(&mx, XBF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.x, d,
                          st, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    auto kern = k_tc<FMT, BN, XBF, G, LSS, AS, AM, KS>;
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
    if (KS > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
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
    return cudaLaunchKernelEx(&cfg, kern, mw, mx, p);
}

cudaError_t launch(int fmt, const TcArgs& a, cudaStream_t s) {
    const int xbf = fmt == 0 ? 0 : a.x_bf16;
    const int64_t mt = (a.N + BM - 1) / BM;
    const int64_t nk = a.K / BK;
    // One CTA per SM.  Time of a CTA ~ its stages x the measured cost of a 64-k stage
    // (about 800 / 830 / 940 cycles at BN = 64 / 128 / 256: the MMA issue path and the
    // loads, not the MMA itself, set it below BN = 256), plus about 6000 cycles for the
    // exchange when K is split over two CTAs; times the waves.  The cheapest candidate
    // wins (ties: the earlier, wider one).
    int bn = (int)options().tc_bn;
    int ks = (int)options().tc_ksplit;
    const bool ks2_ok = nk % 8 == 0;
    {
        struct Cand { int bn, ks; };
        const Cand cands[] = {{256, 1}, {256, 2}, {128, 1}, {128, 2}, {64, 1}};
        double best = -1.0;
        int bbn = 128, bks = 1;
        for (const Cand& c : cands) {
            if (bn != 0 && c.bn != bn) continue;
            if (ks != 0 && c.ks != ks) continue;
            // split only to fill the GPU: when the unsplit tiles leave a quarter of the SMs idle
            if (c.ks == 2 && (!ks2_ok || (ks == 0 && mt * ((a.T + c.bn - 1) / c.bn) * 4 > 3 * num_sms()))) continue;
            const double stage = c.bn == 256 ? 940.0 : c.bn == 128 ? 830.0 : 800.0;
            const int64_t ctas = mt * ((a.T + c.bn - 1) / c.bn) * c.ks;
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
        bn = bbn;
        ks = bks;
    }
    Params p = {};
    p.rsx = a.rsx;
    p.rs = a.rs;
    p.ws = a.ws;
    p.y = a.y;
    p.yt = a.yt;
    p.T = a.T;
    p.N = a.N;
    p.K = a.K;
    p.wait_ns = (uint64_t)options().wait_ns;
    p.stall = (int)options().test_stall;
    options().test_stall = 0;
    p.pdl = 1;   // the guard pass (Q4) or the previous kernel touches neither the weights nor anything before the wait
    dim3 grid((unsigned)mt, (unsigned)((a.T + bn - 1) / bn), (unsigned)ks);
    if (options().trace)
        fprintf(stderr, "cq: tcgen05 fmt=%d T=%lld N=%lld K=%lld BN=%d ksplit=%d grid=(%u,%u,%u)\n", fmt,
                (long long)a.T, (long long)a.N, (long long)a.K, bn, ks, grid.x, grid.y, grid.z);
    // decoded weight operand: 1 = shared memory, 2 = tensor memory (default)
    const int am = options().tc_amode == 1 ? 0 : 1;
    // <FMT, BN, XBF, G, LSS, AS, AM>: super-stages of G stages (weight rows of 64 or 128
    // bytes per box), as many super-slots as fit next to the decoded slots
    if (am == 0) {
        if (fmt == 0) {
            if (bn == 256) return ks == 2 ? launch_bn<0, 256, 0, 2, 2, 4, 0, 2>(a, p, grid, s) : launch_bn<0, 256, 0, 2, 2, 4, 0, 1>(a, p, grid, s);
            if (bn == 128) return ks == 2 ? launch_bn<0, 128, 0, 2, 4, 4, 0, 2>(a, p, grid, s) : launch_bn<0, 128, 0, 2, 4, 4, 0, 1>(a, p, grid, s);
            return launch_bn<0, 64, 0, 4, 3, 4, 0>(a, p, grid, s);
        }
        if (xbf) {
            if (bn == 256) return ks == 2 ? launch_bn<1, 256, 1, 2, 2, 4, 0, 2>(a, p, grid, s) : launch_bn<1, 256, 1, 2, 2, 4, 0, 1>(a, p, grid, s);
            if (bn == 128) return ks == 2 ? launch_bn<1, 128, 1, 2, 3, 4, 0, 2>(a, p, grid, s) : launch_bn<1, 128, 1, 2, 3, 4, 0, 1>(a, p, grid, s);
            return launch_bn<1, 64, 1, 2, 4, 4, 0>(a, p, grid, s);
        }
        if (bn == 256) return ks == 2 ? launch_bn<1, 256, 0, 2, 2, 4, 0, 2>(a, p, grid, s) : launch_bn<1, 256, 0, 2, 2, 4, 0, 1>(a, p, grid, s);
        if (bn == 128) return ks == 2 ? launch_bn<1, 128, 0, 2, 3, 4, 0, 2>(a, p, grid, s) : launch_bn<1, 128, 0, 2, 3, 4, 0, 1>(a, p, grid, s);
        return launch_bn<1, 64, 0, 2, 4, 4, 0>(a, p, grid, s);
    }
    if (fmt == 0) {
        if (bn == 256) return ks == 2 ? launch_bn<0, 256, 0, 2, 3, 8, 1, 2>(a, p, grid, s) : launch_bn<0, 256, 0, 2, 3, 8, 1, 1>(a, p, grid, s);
        if (bn == 128) return ks == 2 ? launch_bn<0, 128, 0, 2, 5, 8, 1, 2>(a, p, grid, s) : launch_bn<0, 128, 0, 2, 5, 8, 1, 1>(a, p, grid, s);
        return launch_bn<0, 64, 0, 4, 4, 8, 1>(a, p, grid, s);
    }
    if (xbf) {
        if (bn == 256) return ks == 2 ? launch_bn<1, 256, 1, 1, 5, 8, 1, 2>(a, p, grid, s) : launch_bn<1, 256, 1, 1, 5, 8, 1, 1>(a, p, grid, s);
        if (bn == 128) return ks == 2 ? launch_bn<1, 128, 1, 2, 4, 8, 1, 2>(a, p, grid, s) : launch_bn<1, 128, 1, 2, 4, 8, 1, 1>(a, p, grid, s);
        return launch_bn<1, 64, 1, 2, 6, 8, 1>(a, p, grid, s);
    }
    if (bn == 256) return ks == 2 ? launch_bn<1, 256, 0, 1, 5, 8, 1, 2>(a, p, grid, s) : launch_bn<1, 256, 0, 1, 5, 8, 1, 1>(a, p, grid, s);
    if (bn == 128) return ks == 2 ? launch_bn<1, 128, 0, 2, 4, 8, 1, 2>(a, p, grid, s) : launch_bn<1, 128, 0, 2, 4, 8, 1, 1>(a, p, grid, s);
    return launch_bn<1, 64, 0, 2, 6, 8, 1>(a, p, grid, s);
}

}  // namespace

cudaError_t launch_tc_q4(const TcArgs& a, cudaStream_t s) { return launch(0, a, s); }
cudaError_t launch_tc_q8(const TcArgs& a, cudaStream_t s) { return launch(1, a, s); }

}  // namespace cq
