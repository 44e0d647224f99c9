// Weight-streaming GEMM for few activation rows (T <= 32) and the routed
// MoE expert panels.
//
// Y^T = W . X^T with the weight rows in the MMA's M dimension and the
// activation rows (tokens or routed pairs) in N, so a small T only narrows
// N.  One CTA owns RB weight rows and a contiguous range of K:
//  - a producer warp streams the packed weights (and, for Q4, the fp16
//    block scales) and the matching slice of the activations into a
//    shared-memory ring with TMA, one stage per 256 k (Q4) or 128 k (Q8),
//    each stage tracked by full/empty mbarriers; producer lane s issues
//    every copy of ring slot s;
//  - dense Q4 takes the caller's activations as given (fp16 or bf16, k
//    order) and decodes the weights into pairs of adjacent k to match them;
//  - eight consumer warps take part in every stage.  With up to 16
//    activation columns each warp owns 16 weight rows and the whole stage
//    (RB = 128); with 32 columns each warp owns 16 rows and half of the
//    stage's k (RB = 64; the halves are summed in a fixed order at the
//    end), which halves each warp's activation reads from shared memory.
// Decoding goes straight from shared memory into mma.sync A fragments:
//  - Q4: lane c of a quad decodes word c (bytes 4c .. 4c + 3, that is
//    k = 4c .. 4c + 3 in the low nibbles and k = 4c + 16 .. 4c + 19 in the
//    high ones) of one 32-k block for its two rows.  Dense (the activations
//    as given, in the activation type): the nibbles of adjacent bytes are
//    paired, (b0, b1) and (b2, b3), so each pair is two adjacent k and the
//    MMA's activation operand is two 8-byte runs of the row in k order.
//    MoE (the guarded fp16 rows, written by the gather pass so that the
//    eight partners of one word are one 16-byte chunk): the nibbles of
//    bytes (b0, b2) and (b1, b3) are paired.  Either way a pair becomes
//    128 + n (bf16) or 1024 + n (fp16) by masking and byte moves, and one
//    subtraction (or a fused multiply-add by 1/16 for 1024 + 16 n) leaves
//    n - 8 exactly.  The two MMAs of one block take all 32 k of that block,
//    so their f32 result is multiplied by the block scale (exact in f32)
//    into the running sum: the scale is folded per 32-k block.
//  - Q8 (activations fp16 or bf16 as given): int8 pairs become fp16
//    exactly ((v ^ 0x80) | 0x6400 is 1024 + v + 128) or bf16 exactly (low
//    seven bits and the sign bit go to two bf16 numbers whose difference is
//    v); the row scale is applied in the epilogue.
// When K is split across a thread-block cluster, each rank pushes its
// partial values into the receive buffer of the rank that finishes them and
// the sums are taken in rank order, so results are deterministic.
// Launches overlap through programmatic dependent launch: every CTA lets
// the next kernel in the stream start as soon as it runs, and the
// producer requests the weights of its first ring fill before it waits for
// the previous kernel (weights are never written by this library); the
// activations, the expert layout and the outputs are touched only after
// that wait.
//
// Prior art on the pages: the 8-row expert panels ("cortiq-engine 0.8.41
// src/gpu_metal/clover.rs", q4tp_mul_mm_n8) and the 32-token MMA tiles for
// short inputs ("oxinfer 0.0.5 src/metal.rs", mma_tile with TM = 32).
#include <algorithm>
#include <cooperative_groups.h>
#include <cstring>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cq_internal.h"
#include "cq_ptx.cuh"

namespace cg = cooperative_groups;

namespace cq {

namespace {

constexpr int CONSUMERS = 8;     // consumer warps, all of them in every stage
constexpr int PRODUCER = CONSUMERS;
constexpr int THREADS = (CONSUMERS + 1) * 32;

enum Mode { DENSE = 0, GATEUP = 1, DOWN = 2 };

struct Params {
    int64_t K;
    int nst_total;        // stages over the whole K
    int ks;               // K split (cluster size)
    int64_t N;            // DENSE: output rows; MoE: rows of one expert matrix
    int64_t T;            // DENSE: activation rows
    const float* rsx;     // Q4 guard inverse scales per activation row (GATEUP; unused by dense Q4)
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
    int64_t I, H;
    uint64_t wait_ns;
    int pdl;              // launch with a programmatic dependency on the previous kernel
    const int32_t* act;   // MoE: active experts, ascending
    const int32_t* n_act; // MoE: number of active experts
    int rbs;              // MoE: row blocks per expert matrix
    int* err;             // the stream's device error word
    // DENSE, z-batched: job blockIdx.z writes yj[z] (rows of pitch ldy), Q8 row scales rsj[z]
    void* yj[ZMAX];
    const float* rsj[ZMAX];
    int64_t ldy;
    const float* add;     // DENSE: nullable f32 [T][N] added before the output rounding
    // DOWN: the weighted combine, folded in (Y [T][H] written by the last item of each row block)
    const int32_t* inv;   // grouped position of each pair id
    int32_t* cnt;         // [H / 128] items finished per row block (zero at the start of the call)
    int topk;
};

// Tensor maps of every job (MoE modes: job 0 only): weights, Q4 scales, activations.
struct SMaps {
    CUtensorMap w[ZMAX];
    CUtensorMap s[ZMAX];
    CUtensorMap x[ZMAX];
};

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128a(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

// Eight nibbles (bytes b0..b3 of w, one 32-bit word of a Q4 block) -> four
// fp16 pairs holding n - 8 exactly:
// d[0] = low nibbles of (b0, b2), d[1] = high nibbles of (b0, b2),
// d[2] = low nibbles of (b1, b3), d[3] = high nibbles of (b1, b3).
// 0x6400 | n is 1024 + n and 0x6400 | (n << 4) is 1024 + 16 n; 1024 + n - 1032
// and (1024 + 16 n) / 16 - 72 are both n - 8 with no rounding.
__device__ __forceinline__ void decode_q4_word(uint32_t w, uint32_t d[4]) {
    const uint32_t c6400 = 0x64006400u, k1032 = 0x64086408u, k16th = 0x2C002C00u, km72 = 0xD480D480u;
    const uint32_t w8 = w >> 8;
    d[0] = sub_f16x2(and_or<0x000F000Fu>(w, c6400), k1032);
    d[1] = fma_f16x2(and_or<0x00F000F0u>(w, c6400), k16th, km72);
    d[2] = sub_f16x2(and_or<0x000F000Fu>(w8, c6400), k1032);
    d[3] = fma_f16x2(and_or<0x00F000F0u>(w8, c6400), k16th, km72);
}

// The same nibbles paired by adjacent bytes (dense path, activations in k
// order): bytes b0..b3 of w hold k = j .. j + 3 (low nibbles) and j + 16 ..
// j + 19 (high nibbles), and
// d[0] = k (j, j + 1), d[1] = (j + 2, j + 3), d[2] = (j + 16, j + 17),
// d[3] = (j + 18, j + 19).  The masked nibbles are moved next to a constant
// high byte by one byte permutation per pair.  bf16 (seven stored mantissa
// bits): the high nibbles are shifted down first; 0x4300 | n is 128 + n, and
// 128 + n - 136 is n - 8 exactly.  fp16: 1024 + n and 1024 + 16 n as in the
// streaming-order decode above.
__device__ __forceinline__ void decode_q4_word_adj_bf16(uint32_t w, uint32_t d[4]) {
    const uint32_t c43 = 0x43434343u, k136 = 0x43084308u;
    const uint32_t lo = and_mask<0x0F0F0F0Fu>(w), hi = and_mask<0x0F0F0F0Fu>(w >> 4);
    d[0] = sub_bf16x2(prmt(lo, c43, 0x4140u), k136);
    d[1] = sub_bf16x2(prmt(lo, c43, 0x4342u), k136);
    d[2] = sub_bf16x2(prmt(hi, c43, 0x4140u), k136);
    d[3] = sub_bf16x2(prmt(hi, c43, 0x4342u), k136);
}
__device__ __forceinline__ void decode_q4_word_adj(uint32_t w, uint32_t d[4]) {
    const uint32_t c64 = 0x64646464u, k1032 = 0x64086408u, k16th = 0x2C002C00u, km72 = 0xD480D480u;
    const uint32_t lo = and_mask<0x0F0F0F0Fu>(w), hi = and_mask<0xF0F0F0F0u>(w);
    d[0] = sub_f16x2(prmt(lo, c64, 0x4140u), k1032);
    d[1] = sub_f16x2(prmt(lo, c64, 0x4342u), k1032);
    d[2] = fma_f16x2(prmt(hi, c64, 0x4140u), k16th, km72);
    d[3] = fma_f16x2(prmt(hi, c64, 0x4342u), k16th, km72);
}

// int8 pair (bytes sel of w) -> half2 exactly: (v ^ 0x80) | 0x6400 is
// 1024 + v + 128; subtracting 1152 leaves v.
__device__ __forceinline__ uint32_t i8x2_to_h2(uint32_t wx /* w ^ 0x80808080 */, uint32_t sel) {
    return sub_f16x2(prmt(wx, 0x64646464u, sel), 0x64806480u);
}
// int8 pair (bytes sel of w) -> bf16x2 exactly: with 0x43 as the high byte,
// the low seven bits of v give 128 + (v & 127) and the sign bit gives 128 or
// 256 (0x4300 / 0x4380); their difference is v, an integer bf16 holds exactly.
__device__ __forceinline__ uint32_t i8x2_to_bf2(uint32_t w, uint32_t sel) {
    const uint32_t t = prmt(w, 0x43434343u, sel);
    return sub_bf16x2(and_mask<0xFF7FFF7Fu>(t), and_mask<0xFF80FF80u>(t));
}

// One stage in shared memory, filled by three TMA copies (five for gate/up):
//  W  [RB rows][128 B], 128-byte swizzle: 16-byte chunk j of row r at j ^ (r % 8)
//     (Q4: 256 k = eight 32-k blocks; Q8: 128 k = eight 16-k runs)
//  S  [RB rows][8 fp16] block scales (Q4 only)
//  X  [NCOL rows][XSL slabs of 64 k][128 B], 128-byte swizzle over the 3-D
//     view {64 elements, K/64 slabs, rows} of the activations; a row's chunk
//     c of slab s sits at c ^ ((XSL row + s) % 8).
// Weight rows per stage for MT m16 tiles per warp and KW warp groups along k.
__host__ __device__ constexpr int rows_per_stage(int MT, int KW) { return CONSUMERS / KW * MT * 16; }

template <int FMT, int NCOL, int RB>
struct StageGeo {
    static constexpr int KSTAGE = FMT == 0 ? 256 : 128;   // FMT 1 Q8-row, 2 Q8 per 32-k block: 128 k
    static constexpr int W_BYTES = RB * 128;
    static constexpr int S_BYTES = FMT != 1 ? RB * 16 : 0;   // Q4: 8 fp16 per row, Q8/32: 4 f32
    static constexpr int XSL = KSTAGE / 64;            // 64-k slabs per stage
    static constexpr int X_OFF = W_BYTES + S_BYTES;    // 1024-aligned
    static constexpr int X_BYTES = NCOL * XSL * 128;
    static constexpr int BYTES = X_OFF + X_BYTES;
};

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// MT: m16 tiles per consumer warp; KW: warp groups along k (the stage's
// eight 32-k blocks, or 16-k runs, are split over them), so 8 / KW warps
// cover the stage's RB = 8 / KW * MT * 16 rows.
// RAW: the activations are the caller's rows as given (fp16 or bf16, k order),
// matched by the adjacent-k decode; no guard scale applies (Q4 dense only).
template <int FMT, int NT, int MT, int KW, int XBF, int MODE, int NSLOT, int RAW>
__global__ void __launch_bounds__(THREADS, 2)
k_skinny(const __grid_constant__ SMaps maps, const Params p) {
    constexpr int NCOL = 8 * NT;
    constexpr int RG = CONSUMERS / KW;        // warps along rows
    constexpr int RB = rows_per_stage(MT, KW);
    static_assert(KW == 1 || KW == 2, "k split over one or two warp groups");
    static_assert(FMT == 1 || (MT == 1 && (XBF == 0 || RAW)), "Q4 stages: one m16 tile per warp; bf16 activations as given");
    static_assert(RAW == 0 || (FMT != 1 && MODE == DENSE), "activations as given: dense Q4 or Q8/32");
    static_assert(FMT != 2 || (RAW == 1 && KW == 1), "Q8/32: activations as given, every warp on the whole stage");
    static_assert(MODE == DENSE || RB == 128, "expert panels use 128-row stages");
    using G = StageGeo<FMT, NCOL, RB>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    // dense, z-batched: job blockIdx.z (its own weights, activations and output)
    const int jz = MODE == DENSE ? (int)blockIdx.z : 0;
    const CUtensorMap* tmW = &maps.w[jz];
    const CUtensorMap* tmS = &maps.s[jz];
    const CUtensorMap* tmX = &maps.x[jz];
    pdl_launch_dependents();   // the next kernel in the stream may be scheduled now
    // dense Q8: the epilogue's row scale of this thread's row (tid % RB; weights-side data,
    // never written by this library, so read before waiting for the previous kernel)
    float rs_pre = 1.f;
    if (MODE == DENSE && FMT == 1 && warp < CONSUMERS) {
        const float* const RSj = jz == 0 ? p.rsj[0] : jz == 1 ? p.rsj[1] : jz == 2 ? p.rsj[2] : p.rsj[3];
        const int64_t n = (int64_t)blockIdx.y * RB + (threadIdx.x & (RB - 1));
        if (n < p.N) rs_pre = RSj[n];
    }
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
        if (MODE == GATEUP) {     // 64 gate rows, then the 64 matching up rows
            it.row_box[0] = it.rb * (RB / 2);
            it.row_box[1] = (int)p.I + it.rb * (RB / 2);
        } else {
            it.row_box[0] = it.rb * RB;
            it.row_box[1] = 0;
        }
        return it;
    };

    // ---- k range ----
    const int ks = MODE == DENSE ? (int)blockIdx.x : 0;
    const int st0 = (int)((int64_t)p.nst_total * ks / p.ks);
    const int st1 = (int)((int64_t)p.nst_total * (ks + 1) / p.ks);
    const int nst = st1 - st0;

    // ---- shared memory carve-up ----
    // part [RB][NCOL] f32: the CTA's partial tile (dense: aliases the ring, which
    // is idle once every stage has been consumed)
    constexpr int RING = NSLOT * G::BYTES;
    constexpr int PART_OFF = (MODE == DENSE) ? 0 : RING;
    constexpr int PART_BYTES = RB * NCOL * 4;
    // dense: recv [ks][slice] f32, the partial sums the cluster's ranks push to this rank
    // (a region of its own, so ranks still streaming are never written into)
    constexpr int RECV_OFF = (MODE == DENSE) ? (RING > PART_BYTES ? RING : PART_BYTES) : RING + PART_BYTES;
    // MoE: the group's per-column epilogue scales [2][NCOL] (guard inverse, routing weight)
    constexpr int RECV_BYTES = (MODE == DENSE) ? PART_BYTES : 2 * NCOL * 4;
    constexpr int BAR_OFF = RECV_OFF + RECV_BYTES;
    float* part = reinterpret_cast<float*>(smem + PART_OFF);
    float* recv = reinterpret_cast<float*>(smem + RECV_OFF);
    // full[NSLOT], empty[NSLOT]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * NSLOT);
    volatile int* never_flag = abort_flag + 1;  // stays 0: waits that must not be cut short
    volatile int* last_flag = abort_flag + 2;   // DOWN: this CTA finished a row block's last item

    const uint32_t smem_base = smem_u32(smem);
    const uint32_t bar_base = smem_u32(bars);
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (NSLOT + s); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), CONSUMERS);
        }
        *abort_flag = 0;
        *never_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == PRODUCER) {
        // ================= producers =================
        // Lane s owns ring slot s and issues every copy of the stages that land in it
        // (stage gi goes to slot gi % NSLOT): one thread keeps only a few bulk copies
        // outstanding, so the ring is filled from NSLOT threads.
        if (lane < NSLOT) {
            const int s = lane;
            if (lane == 0) {
                tma_prefetch_desc(tmW);
                if (FMT != 1) tma_prefetch_desc(tmS);
                tma_prefetch_desc(tmX);
            }
            int last_gi = -1;         // the last stage this lane issued
            uint32_t last_phase = 0;  // and the phase of its round
            bool ok = true;
            auto load_w = [&](const Item& it, int i) {
                const uint32_t sbase = smem_base + (uint32_t)(s * G::BYTES);
                const int st = st0 + i;
                if (MODE == GATEUP) {      // gate rows and up rows are two 64-row boxes
                    for (int bx = 0; bx < 2; ++bx) {
                        tma_load_3d(sbase + (uint32_t)(bx * (RB / 2) * 128), tmW, full_bar(s), st * 128,
                                    it.row_box[bx], it.expert);
                        tma_load_3d(sbase + (uint32_t)(G::W_BYTES + bx * (RB / 2) * 16), tmS, full_bar(s), st * 8,
                                    it.row_box[bx], it.expert);
                    }
                } else {
                    tma_load_3d(sbase, tmW, full_bar(s), st * 128, it.row_box[0], it.expert);
                    if (FMT != 1)   // block scales: 8 fp16 (Q4) or 4 f32 (Q8/32) per row and stage
                        tma_load_3d(sbase + (uint32_t)G::W_BYTES, tmS, full_bar(s), st * (FMT == 0 ? 8 : 4), it.row_box[0], it.expert);
                }
            };
            auto load_x = [&](const Item& it, int i, int grp) {
                const uint32_t sbase = smem_base + (uint32_t)(s * G::BYTES);
                const int st = st0 + i;
                // activation rows of this column group (dense: tokens; MoE: grouped pairs)
                const int xrow0 = (int)(it.col0 + (int64_t)grp * NCOL);
                tma_load_3d(sbase + (uint32_t)G::X_OFF, tmX, full_bar(s), 0, st * G::XSL, xrow0);
            };
            constexpr uint32_t FULL_BYTES = (uint32_t)G::BYTES;   // bytes of a stage
            // The weights of the first ring fill are requested before waiting for the
            // previous kernel in the stream; the activations follow the wait.
            const bool pre = MODE == DENSE && s < nst;
            if (MODE == DENSE) {
                if (pre) {                                   // fresh slot: no empty wait needed
                    mbar_arrive_expect_tx(full_bar(s), FULL_BYTES);
                    load_w(get_item(0), s);
                }
                pdl_wait();
                if (pre) {
                    load_x(get_item(0), s, 0);
                    last_gi = s;
                    last_phase = 0;   // round 0
                }
            }
            // walk every stage in order; this lane issues the ones that land in slot s
            int gi = 0, slot = 0;
            uint32_t phase = 0;
            Item nxt = get_item(first);
            for (int idx = first; idx < nitems && ok; idx += stride) {
                const Item it = nxt;
                if (MODE != DENSE && idx + stride < nitems) nxt = get_item(idx + stride);
                for (int grp = 0; grp < it.ngroups && ok; ++grp) {
                    for (int i = 0; i < nst; ++i, ++gi) {
                        const int my = slot == s && !(pre && gi == s);
                        const uint32_t ph = phase;
                        if (++slot == NSLOT) {
                            slot = 0;
                            phase ^= 1u;
                        }
                        if (!my) continue;
                        // round r of the slot waits for the consumers' release of round r - 1
                        if (!mbar_wait(empty_bar(s), ph ^ 1u, p.wait_ns, abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full_bar(s), FULL_BYTES);
                        load_w(it, i);
                        load_x(it, i, grp);
                        last_gi = gi;
                        last_phase = ph;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicCAS(p.err, 0, DEV_TIMEOUT);
            }
            if (*abort_flag && last_gi >= 0) {  // this lane's last copies must land before the CTA can exit
                mbar_wait(full_bar(s), last_phase, p.wait_ns, never_flag);
            }
        }
        __syncwarp();
    } else {
        // ================= consumers =================
        const int rg = warp % RG, kq = warp / RG;
        const int row0 = rg * (16 * MT) + g;      // this lane's first row in the stage (row0 % 8 == g)
        const uint32_t kqv = KW == 1 ? 0u : (uint32_t)kq;
        // Lane-constant parts of the shared-memory addresses.  Stage bases are
        // 1024-aligned and these offsets leave bits 4..6 to the swizzle terms, so
        // the per-block 16-byte chunk choice is one XOR with a compile-time value.
        //  W: row row0, chunk (j ^ g), word c; row row0 + 8 is 1024 bytes further.
        const uint32_t w_lane = ((uint32_t)(row0 * 128 + 4 * c) ^ ((uint32_t)g << 4)) ^ (kqv << 4);
        //  X (Q4): row 8 nt + g, slab j / 2, swizzled by the line (4 row + slab) % 8 =
        //  (4 (g % 2)) ^ (j / 2).  Streaming order (MoE): chunk 4 (j % 2) + c.  k order
        //  (dense): elements 4c .. 4c + 3 of block j, byte 8 (c % 2) of chunk
        //  4 (j % 2) + c / 2, and elements 4c + 16 .. 4c + 19 two chunks further.
        const uint32_t x_lane = RAW ? (uint32_t)(512 * g + 8 * (c & 1)) |
                                          (((((uint32_t)c >> 1)) ^ (4u * (uint32_t)(g & 1)) ^ (4u * kqv)) << 4)
                                    : (uint32_t)(512 * g) | ((((uint32_t)c) ^ (4u * (uint32_t)(g & 1)) ^ (4u * kqv)) << 4);
        uint32_t slot = 0, phase = 0;             // ring position of the next stage (same walk as the producers)
        // MoE: the next item's expert and columns are read while this one streams, and the
        // group's per-column epilogue scales (thread t < NCOL: column t) before its stages, so
        // their loads' latency hides behind the MMAs; they reach the epilogue through shared memory
        float* escol = reinterpret_cast<float*>(smem + RECV_OFF);
        Item nxt = get_item(first);
        for (int idx = first; idx < nitems; idx += stride) {
          const Item it = nxt;
          if (MODE != DENSE && idx + stride < nitems) nxt = get_item(idx + stride);
          const int64_t col0 = it.col0, ncols_total = it.ncols;
          const int rb = it.rb;
          for (int grp = 0; grp < it.ngroups; ++grp) {
            const int64_t cbase = (int64_t)grp * NCOL;
            float eca = 0.f, ecw = 0.f;   // DOWN: guard inverse and routing weight; GATEUP: guard inverse
            if (MODE != DENSE && threadIdx.x < NCOL && cbase + (int)threadIdx.x < ncols_total) {
                const int64_t pos = col0 + cbase + threadIdx.x;
                if (MODE == DOWN) {
                    eca = p.rsa[pos];
                    ecw = p.w[p.perm[pos]];
                } else {
                    eca = p.rsx[pos];
                }
            }
            float acc[MT][NT][4];
#pragma unroll
            for (int a = 0; a < MT; ++a)
#pragma unroll
                for (int b = 0; b < NT; ++b)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[a][b][q] = 0.f;

            bool ok = !*abort_flag;
            for (int i = 0; i < nst && ok; ++i) {
                if (!mbar_wait(full_bar((int)slot), phase, p.wait_ns, abort_flag)) {
                    ok = false;
                    *abort_flag = 1;
                    atomicCAS(p.err, 0, DEV_TIMEOUT);
                    break;
                }
                const uint32_t sW = smem_base + slot * (uint32_t)G::BYTES;
                const uint32_t sX = sW + (uint32_t)G::X_OFF;
                if (FMT == 0) {
                    // Block j = jf + kq: the two MMAs over its 32 k see one scale per row, so
                    // their f32 result is scaled once into the sum.
                    const uint32_t wS = sW + w_lane, xS = sX + x_lane;
                    const uint32_t sS = sW + (uint32_t)G::W_BYTES + (uint32_t)(row0 * 16) + 2u * kqv;
                    uint4 sc0 = make_uint4(0, 0, 0, 0), sc1 = make_uint4(0, 0, 0, 0);
                    if (KW == 1) {                      // all eight block scales of both rows
                        sc0 = lds128a(sS);
                        sc1 = lds128a(sS + 128);
                    }
#pragma unroll(KW == 1 ? 8 : 2)
                    for (int jj = 0; jj < 8 / KW; ++jj) {
                        const int jf = KW == 1 ? jj : 2 * jj;     // the block index without this warp's k half
                        const uint32_t wad = wS ^ ((uint32_t)jf << 4);
                        const uint32_t wa = lds32(wad), wb = lds32(wad + 1024);
                        const uint32_t jx = (4u * (uint32_t)(jf & 1)) ^ (uint32_t)(jf >> 1);
                        const uint32_t xad = (xS ^ (jx << 4)) + 128u * (uint32_t)(jf >> 1);
                        uint4 bx[NT];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            if (RAW) {   // the two 8-byte runs, k order
                                const uint2 lo = lds64(xad + 4096u * nt), hi = lds64((xad + 4096u * nt) ^ 32u);
                                bx[nt] = make_uint4(lo.x, lo.y, hi.x, hi.y);
                            } else {
                                bx[nt] = lds128a(xad + 4096u * nt);
                            }
                        }
                        float sa, sb;
                        if (KW == 1) {
                            const uint32_t wsa = (jf >> 1) == 0 ? sc0.x : (jf >> 1) == 1 ? sc0.y : (jf >> 1) == 2 ? sc0.z : sc0.w;
                            const uint32_t wsb = (jf >> 1) == 0 ? sc1.x : (jf >> 1) == 1 ? sc1.y : (jf >> 1) == 2 ? sc1.z : sc1.w;
                            sa = __half2float(__ushort_as_half((unsigned short)((jf & 1) ? (wsa >> 16) : (wsa & 0xFFFFu))));
                            sb = __half2float(__ushort_as_half((unsigned short)((jf & 1) ? (wsb >> 16) : (wsb & 0xFFFFu))));
                        } else {
                            sa = __half2float(__ushort_as_half((unsigned short)lds16(sS + 2u * jf)));
                            sb = __half2float(__ushort_as_half((unsigned short)lds16(sS + 128u + 2u * jf)));
                        }
                        uint32_t d[4], e[4];
                        if (RAW && XBF) {
                            decode_q4_word_adj_bf16(wa, d);
                            decode_q4_word_adj_bf16(wb, e);
                        } else if (RAW) {
                            decode_q4_word_adj(wa, d);
                            decode_q4_word_adj(wb, e);
                        } else {
                            decode_q4_word(wa, d);
                            decode_q4_word(wb, e);
                        }
                        const uint32_t a1[4] = {d[0], e[0], d[1], e[1]};
                        const uint32_t a2[4] = {d[2], e[2], d[3], e[3]};
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            float pb[4] = {0.f, 0.f, 0.f, 0.f};
                            if (XBF) {
                                mma_16816_bf16(pb, a1, bx[nt].x, bx[nt].y);
                                mma_16816_bf16(pb, a2, bx[nt].z, bx[nt].w);
                            } else {
                                mma_16816_f16(pb, a1, bx[nt].x, bx[nt].y);
                                mma_16816_f16(pb, a2, bx[nt].z, bx[nt].w);
                            }
                            acc[0][nt][0] = fmaf(sa, pb[0], acc[0][nt][0]);
                            acc[0][nt][1] = fmaf(sa, pb[1], acc[0][nt][1]);
                            acc[0][nt][2] = fmaf(sb, pb[2], acc[0][nt][2]);
                            acc[0][nt][3] = fmaf(sb, pb[3], acc[0][nt][3]);
                        }
                    }
                } else if (FMT == 2) {
                    // Q8 per 32-k block, activations as given (k order): four blocks per stage.
                    // Lane c of a quad takes words c (k = 4c .. 4c + 3) and c + 4 (k = 16 + 4c ..)
                    // of each block for its rows, the same k as the two 8-byte activation runs
                    // it reads, so each pair of bytes is an adjacent-k pair of both operands; the
                    // block's two MMAs see one f32 scale per row, applied to their f32 result.
                    const uint32_t wS = sW + w_lane;
                    const uint32_t sS = sW + (uint32_t)G::W_BYTES + (uint32_t)(row0 * 16);
                    const uint4 sc0 = lds128a(sS), sc1 = lds128a(sS + 128);   // rows row0, row0 + 8
#pragma unroll
                    for (int jf = 0; jf < 4; ++jf) {
                        const uint32_t wa = wS ^ ((uint32_t)(2 * jf) << 4), wb = wS ^ ((uint32_t)(2 * jf + 1) << 4);
                        uint32_t wa0 = lds32(wa), wa1 = lds32(wb), wb0 = lds32(wa + 1024), wb1 = lds32(wb + 1024);
                        uint4 bx[NT];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            // row r = 8 nt + g, slab jf / 2, chunks 4 (jf % 2) + c / 2 (+ 2 for the high run),
                            // 128-byte swizzle key (2 r + slab) % 8 over the [row][2 slabs][128 B] box
                            const uint32_t slab = (uint32_t)(jf >> 1), key = ((uint32_t)(2 * g) + slab) & 7u;
                            const uint32_t rowb = sX + (uint32_t)((8 * nt + g) * 256) + slab * 128u + 8u * (uint32_t)(c & 1);
                            const uint32_t clo = (uint32_t)(4 * (jf & 1) + (c >> 1));
                            const uint2 lo = lds64(rowb + ((clo ^ key) << 4)), hi = lds64(rowb + (((clo + 2u) ^ key) << 4));
                            bx[nt] = make_uint4(lo.x, lo.y, hi.x, hi.y);
                        }
                        uint32_t a1[4], a2[4];
                        if (XBF) {
                            a1[0] = i8x2_to_bf2(wa0, 0x4140u); a1[1] = i8x2_to_bf2(wb0, 0x4140u);
                            a1[2] = i8x2_to_bf2(wa0, 0x4342u); a1[3] = i8x2_to_bf2(wb0, 0x4342u);
                            a2[0] = i8x2_to_bf2(wa1, 0x4140u); a2[1] = i8x2_to_bf2(wb1, 0x4140u);
                            a2[2] = i8x2_to_bf2(wa1, 0x4342u); a2[3] = i8x2_to_bf2(wb1, 0x4342u);
                        } else {
                            wa0 ^= 0x80808080u; wb0 ^= 0x80808080u; wa1 ^= 0x80808080u; wb1 ^= 0x80808080u;
                            a1[0] = i8x2_to_h2(wa0, 0x4140u); a1[1] = i8x2_to_h2(wb0, 0x4140u);
                            a1[2] = i8x2_to_h2(wa0, 0x4342u); a1[3] = i8x2_to_h2(wb0, 0x4342u);
                            a2[0] = i8x2_to_h2(wa1, 0x4140u); a2[1] = i8x2_to_h2(wb1, 0x4140u);
                            a2[2] = i8x2_to_h2(wa1, 0x4342u); a2[3] = i8x2_to_h2(wb1, 0x4342u);
                        }
                        const float sa = __uint_as_float(jf == 0 ? sc0.x : jf == 1 ? sc0.y : jf == 2 ? sc0.z : sc0.w);
                        const float sb = __uint_as_float(jf == 0 ? sc1.x : jf == 1 ? sc1.y : jf == 2 ? sc1.z : sc1.w);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            float pb[4] = {0.f, 0.f, 0.f, 0.f};
                            if (XBF) {
                                mma_16816_bf16(pb, a1, bx[nt].x, bx[nt].y);
                                mma_16816_bf16(pb, a2, bx[nt].z, bx[nt].w);
                            } else {
                                mma_16816_f16(pb, a1, bx[nt].x, bx[nt].y);
                                mma_16816_f16(pb, a2, bx[nt].z, bx[nt].w);
                            }
                            acc[0][nt][0] = fmaf(sa, pb[0], acc[0][nt][0]);
                            acc[0][nt][1] = fmaf(sa, pb[1], acc[0][nt][1]);
                            acc[0][nt][2] = fmaf(sb, pb[2], acc[0][nt][2]);
                            acc[0][nt][3] = fmaf(sb, pb[3], acc[0][nt][3]);
                        }
                    }
                } else {
                    const uint8_t* pW = smem + slot * G::BYTES;
                    const uint8_t* pX = pW + G::X_OFF;
#pragma unroll
                    for (int kk = 0; kk < 2 / KW; ++kk) {
                        // this lane's 16-k run j = 2c + kh: chunk j of each of its rows, and
                        // activations k = 16 j .. 16 j + 15 = slab j / 4, 32 bytes at 32 (j % 4)
                        const int kh = KW == 1 ? kk : kq;
                        const int j = 2 * c + kh;
                        const int slab = j >> 2;
                        uint4 b0[NT], b1[NT];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const int xrow = 8 * nt + g;
                            const uint8_t* xr = pX + xrow * (G::XSL * 128) + slab * 128;
                            const int sw = (G::XSL * xrow + slab) & 7;
                            b0[nt] = lds128(xr + (((2 * (j & 3)) ^ sw) << 4));
                            b1[nt] = lds128(xr + (((2 * (j & 3) + 1) ^ sw) << 4));
                        }
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            const int r0 = row0 + 16 * mt;
                            const uint4 w0 = lds128(pW + r0 * 128 + ((j ^ g) << 4));
                            const uint4 w1 = lds128(pW + (r0 + 8) * 128 + ((j ^ g) << 4));
                            const uint32_t q0[4] = {w0.x, w0.y, w0.z, w0.w};
                            const uint32_t q1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                            for (int s4 = 0; s4 < 4; ++s4) {
                                uint32_t a[4];
                                if (XBF) {
                                    a[0] = i8x2_to_bf2(q0[s4], 0x4140u);
                                    a[1] = i8x2_to_bf2(q1[s4], 0x4140u);
                                    a[2] = i8x2_to_bf2(q0[s4], 0x4342u);
                                    a[3] = i8x2_to_bf2(q1[s4], 0x4342u);
                                } else {
                                    const uint32_t x0w = q0[s4] ^ 0x80808080u, x1w = q1[s4] ^ 0x80808080u;
                                    a[0] = i8x2_to_h2(x0w, 0x4140u);
                                    a[1] = i8x2_to_h2(x1w, 0x4140u);
                                    a[2] = i8x2_to_h2(x0w, 0x4342u);
                                    a[3] = i8x2_to_h2(x1w, 0x4342u);
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
                if (lane == 0) mbar_arrive(empty_bar((int)slot));
                if (++slot == (uint32_t)NSLOT) {
                    slot = 0;
                    phase ^= 1u;
                }
            }

            // ---- the CTA's partial tile ----
            // (dense: part aliases the ring, so every warp must be done with it; the k
            // halves of KW == 2 are added in a fixed order)
            if (MODE == DENSE) asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS * 32) : "memory");
            if (MODE != DENSE && threadIdx.x < NCOL) {   // read after the barrier below
                escol[threadIdx.x] = eca;
                escol[NCOL + threadIdx.x] = ecw;
            }
#pragma unroll
            for (int h = 0; h < KW; ++h) {
                if (kq == h) {
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const int r = row0 + 16 * mt, col = 8 * nt + 2 * c;
                            float2* p0 = reinterpret_cast<float2*>(part + r * NCOL + col);
                            float2* p1 = reinterpret_cast<float2*>(part + (r + 8) * NCOL + col);
                            if (h == 0) {
                                *p0 = make_float2(acc[mt][nt][0], acc[mt][nt][1]);
                                *p1 = make_float2(acc[mt][nt][2], acc[mt][nt][3]);
                            } else {
                                const float2 u0 = *p0, u1 = *p1;
                                *p0 = make_float2(u0.x + acc[mt][nt][0], u0.y + acc[mt][nt][1]);
                                *p1 = make_float2(u1.x + acc[mt][nt][2], u1.y + acc[mt][nt][3]);
                            }
                        }
                }
                asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS * 32) : "memory");
            }

            if (MODE != DENSE) {
              // MoE epilogues (single CTA per k range).  The barrier after them is taken by
              // every consumer warp whatever the abort flag says, so the counts always match.
              if (!*abort_flag) {
                if (MODE == GATEUP) {
                    // element (i, col): gate at local row i, up at local row 64 + i
                    for (int e = threadIdx.x; e < (RB / 2) * NCOL; e += CONSUMERS * 32) {
                        const int i = e & (RB / 2 - 1), col = e / (RB / 2);
                        const int64_t q = cbase + col;
                        if (q >= ncols_total) continue;
                        const int64_t pos = col0 + q;
                        const float sc = escol[col];
                        const float gv = part[i * NCOL + col] * sc;
                        const float uv = part[(RB / 2 + i) * NCOL + col] * sc;
                        p.out[pos * p.I + (int64_t)rb * (RB / 2) + i] = gv / (1.0f + expf(-gv)) * uv;
                    }
                } else {
                    for (int e = threadIdx.x; e < RB * NCOL; e += CONSUMERS * 32) {
                        const int r = e & (RB - 1), col = e / RB;
                        const int64_t q = cbase + col;
                        if (q >= ncols_total) continue;
                        const int64_t pos = col0 + q;
                        const float v = part[r * NCOL + col] * escol[col] * escol[NCOL + col];
                        p.out[pos * p.H + (int64_t)rb * RB + r] = v;
                    }
                }
              }
              asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS * 32) : "memory");
            }
          }
        }
        if (MODE == DOWN) {
            // The weighted combine, folded in.  Once this CTA's items are done (their eo
            // rows written by every consumer thread, then a CTA barrier), thread 0 makes
            // them visible with one device-scope fence and counts each item for its row
            // block with one atomic; the CTA whose count completes a row block (all active
            // experts in) fences again and sums, for every token, the eo rows of its slots
            // in slot order j = 0 .. topk - 1, so the result does not depend on which CTA
            // finishes last.  It also resets the counter.  The row blocks to finish go
            // through shared memory (the idle partial-tile buffer).
            int* done = reinterpret_cast<int*>(part);
            asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS * 32) : "memory");
            if (threadIdx.x == 0) {
                int nd = 0;
                if (!*abort_flag) {
                    __threadfence();
                    for (int idx = first; idx < nitems; idx += stride) {
                        const int rbi = idx % p.rbs;
                        if (atomicAdd(p.cnt + rbi, 1) == *p.n_act - 1) done[nd++] = rbi;
                    }
                    if (nd) __threadfence();
                }
                *last_flag = nd;
            }
            asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS * 32) : "memory");
            for (int di = 0; di < *last_flag; ++di) {
                const int rb = done[di];
                // one consumer warp per pair of tokens, lane l owning rows 4 l .. 4 l + 3 of the
                // block; the slots' grouped positions come in one coalesced load per token
                // (lane j holds slot j's), then the rows of eight slots of both tokens are
                // loaded together (independent loads in flight) and added in slot order
                const int64_t n0 = (int64_t)rb * RB + 4 * lane;
                for (int64_t t0 = 2 * warp; t0 < p.T; t0 += 2 * CONSUMERS) {
                    const bool two = t0 + 1 < p.T;
                    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
                    for (int j0 = 0; j0 < p.topk; j0 += 32) {
                        int qa = 0, qb = 0;
                        if (j0 + lane < p.topk) {
                            qa = __ldg(p.inv + t0 * p.topk + j0 + lane);
                            if (two) qb = __ldg(p.inv + (t0 + 1) * p.topk + j0 + lane);
                        }
                        const int nj = min(32, p.topk - j0);
                        for (int j1 = 0; j1 < nj; j1 += 8) {
                            float4 v[2][8];
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj) {
                                const int64_t q0 = __shfl_sync(0xffffffffu, qa, (j1 + jj) & 31);
                                const int64_t q1 = __shfl_sync(0xffffffffu, qb, (j1 + jj) & 31);
                                if (j1 + jj < nj) {
                                    v[0][jj] = __ldcg(reinterpret_cast<const float4*>(p.out + q0 * p.H + n0));
                                    if (two) v[1][jj] = __ldcg(reinterpret_cast<const float4*>(p.out + q1 * p.H + n0));
                                }
                            }
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
#pragma unroll
                                for (int jj = 0; jj < 8; ++jj) {
                                    if (j1 + jj < nj && (u == 0 || two)) {
                                        acc[u].x += v[u][jj].x;
                                        acc[u].y += v[u][jj].y;
                                        acc[u].z += v[u][jj].z;
                                        acc[u].w += v[u][jj].w;
                                    }
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        if (u == 1 && !two) break;
                        const int64_t t = t0 + u;
                        if (p.yt == CQ_F32) {
                            *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.y) + t * p.H + n0) = acc[u];
                        } else {
                            __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(p.y) + t * p.H + n0);
                            o[0] = __floats2bfloat162_rn(acc[u].x, acc[u].y);
                            o[1] = __floats2bfloat162_rn(acc[u].z, acc[u].w);
                        }
                    }
                }
                if (threadIdx.x == 0) p.cnt[rb] = 0;
            }
        }
    }

    if (MODE == DENSE) {
        const int rb = blockIdx.y;
        void* const Yj = jz == 0 ? p.yj[0] : jz == 1 ? p.yj[1] : jz == 2 ? p.yj[2] : p.yj[3];
        const float* const RSj = jz == 0 ? p.rsj[0] : jz == 1 ? p.rsj[1] : jz == 2 ? p.rsj[2] : p.rsj[3];
        pdl_wait();   // outputs only after the previous kernel has finished
        // ---- sum the cluster's partial tiles in rank order, epilogue ----
        // Rank q finishes slice q of the tile.  Every rank pushes its partial values of
        // slice q into rank q's recv[rank][.]; after one cluster barrier each rank adds
        // its slice locally in rank order.
        if (p.ks > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            const int rank = (int)cluster.block_rank();
            const int per = (RB * NCOL + p.ks - 1) / p.ks;
            if (warp < CONSUMERS && !*abort_flag) {
                // element e is (row e % RB, column e / RB), as in the sums below
                for (int e = threadIdx.x; e < RB * NCOL; e += CONSUMERS * 32) {
                    const int q = e / per;
                    cluster.map_shared_rank(recv, q)[rank * per + (e - q * per)] = part[(e & (RB - 1)) * NCOL + e / RB];
                }
            }
            cluster.sync();
            if (warp < CONSUMERS && !*abort_flag) {
                const int lo = rank * per, hi = min(RB * NCOL, lo + per);
                for (int e = lo + threadIdx.x; e < hi; e += CONSUMERS * 32) {
                    const int r = e & (RB - 1), col = e / RB;
                    float s = 0.f;
                    for (int q = 0; q < p.ks; ++q) s += recv[q * per + (e - lo)];
                    const int64_t n = (int64_t)rb * RB + r, t = col;
                    if (n < p.N && t < p.T) {
                        const float rsn = r == (int)(threadIdx.x & (RB - 1)) ? rs_pre : RSj[n];
                        float v = s * (FMT == 1 ? rsn * (p.rsx ? p.rsx[t] : 1.f) : (RAW ? 1.f : p.rsx[t]));
                        if (p.add) v += p.add[t * p.N + n];
                        if (p.yt == CQ_F32) reinterpret_cast<float*>(Yj)[t * p.ldy + n] = v;
                        else reinterpret_cast<__nv_bfloat16*>(Yj)[t * p.ldy + n] = __float2bfloat16_rn(v);
                    }
                }
            }
        } else if (warp < CONSUMERS && !*abort_flag) {
            for (int e = threadIdx.x; e < RB * NCOL; e += CONSUMERS * 32) {
                const int r = e & (RB - 1), col = e / RB;
                const int64_t n = (int64_t)rb * RB + r, t = col;
                if (n < p.N && t < p.T) {
                    const float rsn = r == (int)(threadIdx.x & (RB - 1)) ? rs_pre : RSj[n];
                    float v = part[r * NCOL + col] * (FMT == 1 ? rsn * (p.rsx ? p.rsx[t] : 1.f) : (RAW ? 1.f : p.rsx[t]));
                    if (p.add) v += p.add[t * p.N + n];
                    if (p.yt == CQ_F32) reinterpret_cast<float*>(Yj)[t * p.ldy + n] = v;
                    else reinterpret_cast<__nv_bfloat16*>(Yj)[t * p.ldy + n] = __float2bfloat16_rn(v);
                }
            }
        }
    }
}

template <int FMT, int NT, int RB, int MODE, int NSLOT>
constexpr size_t smem_bytes() {
    constexpr int NCOL = 8 * NT;
    using G = StageGeo<FMT, NCOL, RB>;
    constexpr int RING = NSLOT * G::BYTES;
    constexpr int PART_BYTES = RB * NCOL * 4;
    constexpr int RECV_OFF = (MODE == DENSE) ? (RING > PART_BYTES ? RING : PART_BYTES) : RING + PART_BYTES;
    constexpr int BAR_OFF = RECV_OFF + ((MODE == DENSE) ? PART_BYTES : 2 * NCOL * 4);
    return (size_t)BAR_OFF + 2 * NSLOT * 8 + 16 + 1024;   // + abort, never and last flags
}

// Weights [E][R][K bytes] and scales [E][R][K/32], boxes of rows_box rows.
bool make_maps(CUtensorMap* mw, CUtensorMap* ms, int fmt, const uint8_t* wq, const uint16_t* ws, int64_t R,
               int64_t K, int64_t E, int rows_box) {
    const uint64_t kbytes = fmt == 0 ? (uint64_t)K / 2 : (uint64_t)K;   // fmt 1, 2: int8
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
    } else if (fmt == 2) {   // f32 block scales [E][R][K/32], boxes of 4 per row (one 128-k stage)
        uint64_t ds[3] = {(uint64_t)K / 32, (uint64_t)R, (uint64_t)E};
        uint64_t ss[2] = {(uint64_t)K / 32 * 4, (uint64_t)K / 32 * 4 * (uint64_t)R};
        uint32_t bs[3] = {4, (uint32_t)rows_box, 1};
        if (!encode_tiled(ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ws, ds, ss, bs, CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
    } else {
        *ms = *mw;
    }
    return true;
}

// Activations [rows][K] 16-bit seen as {64 elements, K/64 slabs, rows}; one box
// is xsl slabs of ncol rows, stored [row][slab][128 B] with the 128-byte swizzle.
bool make_xmap(CUtensorMap* mx, const void* x, int64_t rows, int64_t K, int64_t ldx, int bf16, int ncol, int xsl) {
    uint64_t d[3] = {64, (uint64_t)K / 64, (uint64_t)rows};
    uint64_t st[2] = {128, (uint64_t)ldx * 2};
    uint32_t box[3] = {64, (uint32_t)xsl, (uint32_t)ncol};
    return encode_tiled(mx, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, x, d, st,
                        box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// maps: w and s filled for each of the nz jobs; xs[j] the activations of job j
// (xrows rows of pitch ldx).
template <int FMT, int NT, int MT, int KW, int XBF, int MODE, int NSLOT, int RAW = 0>
cudaError_t launch_t(SMaps maps, const void* const* xs, int nz, int64_t xrows, int64_t ldx, const Params& p,
                     dim3 grid, int cluster, cudaStream_t s) {
    constexpr int RB = rows_per_stage(MT, KW);
    for (int j = 0; j < nz; ++j)
        if (!make_xmap(&maps.x[j], xs[j], xrows, p.K, ldx, XBF, 8 * NT, StageGeo<FMT, 8 * NT, RB>::XSL))
            return cudaErrorInvalidValue;
    auto kern = k_skinny<FMT, NT, MT, KW, XBF, MODE, NSLOT, RAW>;
    constexpr size_t smem = smem_bytes<FMT, NT, RB, MODE, NSLOT>();
    static_assert(smem <= 113 * 1024, "two CTAs per SM");
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
    return counted(cudaLaunchKernelEx(&cfg, kern, maps, p));
}

// Layout and ring depth per column count (as many stages as fit two CTAs
// per SM): up to 16 columns, 128-row stages with every warp on the whole
// stage; 32 columns, 64-row stages with the k blocks split over two warp
// groups, so each warp reads half of the activations.
struct DenseCfg {
    int nt, mt, kw, rb;
};
DenseCfg dense_cfg(int64_t T) {
    if (T <= 8) return {1, 1, 1, rows_per_stage(1, 1)};
    if (T <= 16) return {2, 1, 1, rows_per_stage(1, 1)};
    return {4, 1, 2, rows_per_stage(1, 2)};
}

// Q4 takes the activations as given (RAW), in k order.
template <int FMT, int XBF>
cudaError_t launch_dense_nt(const SMaps& maps, const void* const* xs, int nz, int64_t ldx, const Params& p, dim3 grid,
                            int cluster, int64_t T, cudaStream_t s) {
    if constexpr (FMT == 2) {   // Q8/32: 128-row stages, every warp on the whole stage
        if (T <= 8) return launch_t<2, 1, 1, 1, XBF, DENSE, 5, 1>(maps, xs, nz, T, ldx, p, grid, cluster, s);
        if (T <= 16) return launch_t<2, 2, 1, 1, XBF, DENSE, 4, 1>(maps, xs, nz, T, ldx, p, grid, cluster, s);
        return launch_t<2, 4, 1, 1, XBF, DENSE, 3, 1>(maps, xs, nz, T, ldx, p, grid, cluster, s);
    } else {
        constexpr int RAW = FMT == 0 ? 1 : 0;
        if (T <= 8) return launch_t<FMT, 1, 1, 1, XBF, DENSE, FMT == 0 ? 4 : 5, RAW>(maps, xs, nz, T, ldx, p, grid, cluster, s);
        if (T <= 16) return launch_t<FMT, 2, 1, 1, XBF, DENSE, FMT == 0 ? 3 : 5, RAW>(maps, xs, nz, T, ldx, p, grid, cluster, s);
        return launch_t<FMT, 4, 1, 2, XBF, DENSE, FMT == 0 ? 4 : 6, RAW>(maps, xs, nz, T, ldx, p, grid, cluster, s);
    }
}

cudaError_t launch_dense(int fmt, const SkinnyDense& a, cudaStream_t s) {
    const DenseCfg cf = fmt == 2 ? DenseCfg{a.T <= 8 ? 1 : a.T <= 16 ? 2 : 4, 1, 1, rows_per_stage(1, 1)} : dense_cfg(a.T);
    const int nz = a.jobs();
    SMaps maps;
    memset(&maps, 0, sizeof maps);
    const void* xs[ZMAX] = {};
    Params p = {};
    for (int j = 0; j < nz; ++j) {
        const SkJob jb = a.job(j);
        const uint16_t* scales = fmt == 2 ? reinterpret_cast<const uint16_t*>(a.wsf) : jb.ws;
        if (!make_maps(&maps.w[j], &maps.s[j], fmt, jb.wq, scales, a.N, a.K, 1, cf.rb)) return cudaErrorInvalidValue;
        xs[j] = jb.x;
        p.yj[j] = jb.y;
        p.rsj[j] = jb.rs;
    }
    p.K = a.K;
    p.nst_total = (int)(a.K / (fmt == 0 ? 256 : 128));
    p.add = a.add;
    p.N = a.N;
    p.T = a.T;
    p.rsx = a.rsx;
    p.rs = a.rs;
    p.y = a.y;
    p.yt = a.yt;
    p.ldy = a.ldy > 0 ? a.ldy : a.N;
    p.wait_ns = (uint64_t)options().wait_ns;
    p.pdl = 1;
    p.err = a.err;
    // K split (cluster size): as many CTAs as fit two per SM (a CTA alone keeps too few
    // bytes in flight to draw its share of the bandwidth), at least two stages each.
    const int64_t rbs = (a.N + cf.rb - 1) / cf.rb;
    int ks = 1;
    const int64_t cap = 2 * (int64_t)num_sms();
    for (int cand : {2, 4, 8})
        if (rbs * cand * nz <= cap && p.nst_total / cand >= 2) ks = cand;
    p.ks = ks;
    dim3 grid((unsigned)ks, (unsigned)rbs, (unsigned)nz);
    if (options().trace)
        fprintf(stderr, "cq: skinny fmt=%d T=%lld N=%lld K=%lld rows/stage=%d grid=(%d,%lld,%d) cluster=%d\n", fmt,
                (long long)a.T, (long long)a.N, (long long)a.K, cf.rb, ks, (long long)rbs, nz, ks);
    const int64_t ldx = a.ldx > 0 ? a.ldx : a.K;
    if (fmt == 0)
        return a.x_bf16 ? launch_dense_nt<0, 1>(maps, xs, nz, ldx, p, grid, ks, a.T, s)
                        : launch_dense_nt<0, 0>(maps, xs, nz, ldx, p, grid, ks, a.T, s);
    if (fmt == 2)
        return a.x_bf16 ? launch_dense_nt<2, 1>(maps, xs, nz, ldx, p, grid, ks, a.T, s)
                        : launch_dense_nt<2, 0>(maps, xs, nz, ldx, p, grid, ks, a.T, s);
    return a.x_bf16 ? launch_dense_nt<1, 1>(maps, xs, nz, ldx, p, grid, ks, a.T, s)
                    : launch_dense_nt<1, 0>(maps, xs, nz, ldx, p, grid, ks, a.T, s);
}

}  // namespace

// Up to 16 activation rows, one job and a whole number of stages: the row-partitioned kernel
// (k_rows.cu), unless the K-split kernel here is asked for.
cudaError_t launch_small_t(int fmt, const SkinnyDense& a, cudaStream_t s) {
    const int64_t sk = options().stream_kernel;
    if (sk == 2 ? rows_path_serves(fmt, a.T, a.K, a.jobs()) : sk == 0 && rows_path_preferred(fmt, a.T, a.K, a.N, a.jobs()))
        return launch_rows(fmt, a, s);
    return launch_dense(fmt, a, s);
}
cudaError_t launch_skinny_q4(const SkinnyDense& a, cudaStream_t s) { return launch_small_t(0, a, s); }
cudaError_t launch_skinny_q8(const SkinnyDense& a, cudaStream_t s) { return launch_small_t(1, a, s); }
cudaError_t launch_skinny_q8b(const SkinnyDense& a, cudaStream_t s) { return launch_small_t(2, a, s); }

// Gate/up panels: activations are the guarded rows already gathered into
// grouped order ([P][H] fp16, inverse scales [P]).  One item is 64 gate rows
// and the 64 matching up rows of one expert.
cudaError_t launch_moe_gateup(const SkinnyMoe& m, cudaStream_t s) {
    SMaps maps;
    memset(&maps, 0, sizeof maps);
    constexpr int RB = rows_per_stage(1, 1);
    if (!make_maps(&maps.w[0], &maps.s[0], 0, m.gu_q, m.gu_s, 2 * m.I, m.H, m.E, RB / 2)) return cudaErrorInvalidValue;
    Params p = {};
    p.K = m.H;
    p.nst_total = (int)(m.H / 256);
    p.ks = 1;
    p.N = 2 * m.I;
    p.rsx = m.rsx;
    p.seg = m.seg;
    p.perm = m.perm;
    p.status = m.status;
    p.w = m.w;
    p.out = m.a;
    p.I = m.I;
    p.H = m.H;
    p.wait_ns = (uint64_t)options().wait_ns;
    p.act = m.act;
    p.n_act = m.n_act;
    p.pdl = 1;
    p.err = m.err;
    p.rbs = (int)(m.I / (RB / 2));
    // persistent: two CTAs per SM share the (active expert x row block) items
    const int64_t items_max = m.E * p.rbs;
    dim3 grid((unsigned)std::min<int64_t>(2 * (int64_t)num_sms(), items_max), 1, 1);
    const void* xs[1] = {m.xh};
    return launch_t<0, 1, 1, 1, 0, GATEUP, 4>(maps, xs, 1, m.T * m.topk, m.H, p, grid, 1, s);
}

cudaError_t launch_moe_down(const SkinnyMoe& m, cudaStream_t s) {
    SMaps maps;
    memset(&maps, 0, sizeof maps);
    constexpr int RB = rows_per_stage(1, 1);
    if (!make_maps(&maps.w[0], &maps.s[0], 0, m.d_q, m.d_s, m.H, m.I, m.E, RB)) return cudaErrorInvalidValue;
    Params p = {};
    p.K = m.I;
    p.nst_total = (int)(m.I / 256);
    p.ks = 1;
    p.N = m.H;
    p.rsa = m.rsa;
    p.seg = m.seg;
    p.perm = m.perm;
    p.status = m.status;
    p.w = m.w;
    p.out = m.eo;
    p.I = m.I;
    p.H = m.H;
    p.T = m.T;
    p.topk = (int)m.topk;
    p.inv = m.inv;
    p.cnt = m.cnt;
    p.y = m.y;
    p.yt = m.yt;
    p.wait_ns = (uint64_t)options().wait_ns;
    p.act = m.act;
    p.n_act = m.n_act;
    p.pdl = 1;
    p.err = m.err;
    p.rbs = (int)(m.H / RB);
    const int64_t items_max = m.E * p.rbs;
    dim3 grid((unsigned)std::min<int64_t>(2 * (int64_t)num_sms(), items_max), 1, 1);
    const void* xs[1] = {m.ah};
    return launch_t<0, 1, 1, 1, 0, DOWN, 4>(maps, xs, 1, m.T * m.topk, m.I, p, grid, 1, s);
}

}  // namespace cq
