// Large-T GEMM on the 5th-generation tensor cores (tcgen05, accumulator in
// tensor memory), weights dequantized on the fly in shared memory.
//
// Y^T tile = W tile (128 weight rows, M) x X tile^T (BN activation rows, N),
// K in stages of 64.  Warp roles in a CTA of 192 threads:
//   warp 4      TMA producer: raw weight tile (Q4 nibbles 128 x 32 B or Q8
//               bytes 128 x 64 B, swizzled so the decode reads are
//               bank-conflict free) and the activation tile (BN x 64 fp16 /
//               bf16, 128-byte swizzle = the MMA's K-major operand layout);
//   warps 0-3   decoders, one thread per weight row: raw row -> 64 fp16/bf16
//               values written into the A operand tile in the 128-byte
//               swizzled K-major layout, then the epilogue;
//   warp 5      allocates the tensor memory and issues tcgen05.mma
//               (M = 128, N = BN, K = 16) from one thread, committing each
//               stage back to the producer and the last to the epilogue.
// Q4 decode: (nibble - 8) * fp16 block scale, rounded once to fp16 (the
// scale folded into the half operand, as in mma_tile of "oxinfer 0.0.5
// src/metal.rs"); the activations arrive as fp16 behind a per-row
// power-of-two guard whose inverse the epilogue applies.  Q8-row decode:
// int8 -> the activation type exactly; the row scale is applied to the f32
// accumulator in the epilogue ("cortiq-engine 0.8.3 src/gpu_metal/qi21.rs",
// module header on q8_row).
// Every wait is time-bounded; on a timeout the CTA stops, lets copies in
// flight land, frees its tensor memory and reports CQ_ERR_TIMEOUT.
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
__device__ __forceinline__ uint32_t nib2_to_h2(uint32_t v) {
    const uint32_t h = (v & 0x000F000Fu) | 0x64006400u;
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h),
                              __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408)));
    return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, __half2 s) {
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), s);
    return *reinterpret_cast<const uint32_t*>(&r);
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

template <int FMT>
struct Raw;
template <>
struct Raw<0> { static constexpr int ROW = 32; };   // Q4: 64 k = 32 bytes per row
template <>
struct Raw<1> { static constexpr int ROW = 64; };   // Q8: 64 bytes per row

// Shared memory: a load ring of LS stages (raw weight tile + activation
// tile, filled by TMA) and (AM 0) a shorter ring of AS decoded weight tiles;
// with AM 1 the decoded tiles are AS == LS slots of tensor memory.
template <int FMT, int BN, int LS, int AS, int AM>
struct Layout {
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int R_BYTES = BM * Raw<FMT>::ROW;
    static constexpr int R_STRIDE = (R_BYTES + 1023) / 1024 * 1024;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = A_OFF + (AM == 0 ? AS * A_BYTES : 0);   // AM 1: decoded tiles in TMEM
    static constexpr int R_OFF = B_OFF + LS * B_BYTES;
    static constexpr int BAR_OFF = R_OFF + LS * R_STRIDE;
    // full[LS], empty[LS], afull[AS], aempty[AS], accf; then tmem slot, abort, never
    static constexpr int NBAR = 2 * LS + 2 * AS + 1;
    static constexpr int MISC = NBAR * 8 + 16;
    static constexpr int TOTAL = BAR_OFF + MISC + 1024;  // + alignment slack
    // tensor memory: accumulator in columns [0, BN); AM 1 adds AS decoded A tiles of 32 columns
    static constexpr int A_COL = BN;
    static constexpr int NEED = AM == 0 ? BN : BN + AS * 32;
    static constexpr int TMEM_COLS = NEED <= 32 ? 32 : NEED <= 64 ? 64 : NEED <= 128 ? 128 : NEED <= 256 ? 256 : 512;
    static_assert(NEED <= 512, "tensor memory budget");
};

constexpr int DEC_WARPS = 8;                 // two decoder threads per weight row
constexpr int THREADS = (DEC_WARPS + 2) * 32;
constexpr int PRODUCER_WARP = DEC_WARPS;
constexpr int MMA_WARP = DEC_WARPS + 1;

// int8 byte i of w -> f32 exactly: 0x4B0000uu is 2^23 + u with u = v + 128.
__device__ __forceinline__ float i8_to_f32(uint32_t wx /* w ^ 0x80808080 */, uint32_t sel) {
    return __uint_as_float(prmt(wx, 0x4B000000u, sel)) - 8388736.0f;
}
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&r);
}

template <int FMT, int BN, int XBF, int LS, int AS, int CL, int AM>
__global__ void __launch_bounds__(THREADS, 1)
k_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const Params p) {
    using L = Layout<FMT, BN, LS, AS, AM>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM;          // first weight row
    const int t0 = blockIdx.y * BN;          // first activation row
    const int nk = (int)(p.K / BK);

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (LS + s); };
    auto afull_bar = [&](int a) { return bar0 + 8u * (2 * LS + a); };
    auto aempty_bar = [&](int a) { return bar0 + 8u * (2 * LS + AS + a); };
    const uint32_t accf_bar = bar0 + 8u * (2 * LS + 2 * AS);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never_flag = abort_flag + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < LS; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), CL);   // a slot is free once every CTA of the cluster has consumed it
        }
        for (int a = 0; a < AS; ++a) {
            mbar_init(afull_bar(a), DEC_WARPS * 32);
            mbar_init(aempty_bar(a), 1);
        }
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
    // cluster of CL CTAs along the weight rows: CTA `rank` loads rows
    // [rank*BN/CL, (rank+1)*BN/CL) of each activation tile and multicasts them
    constexpr int XS = BN / CL;
    constexpr uint16_t CMASK = (uint16_t)((1u << CL) - 1u);
    const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
    if (CL > 1) cluster_sync_all();   // every CTA's barriers are initialised before any multicast

    auto give_up = [&]() {
        *abort_flag = 1;
        atomicCAS(&g_err_tc, 0, DEV_TIMEOUT);
    };

    if (warp == PRODUCER_WARP) {
        // ================= TMA producers =================
        // Lane s owns ring slot s and issues that slot's copies: one thread keeps only a
        // few bulk copies outstanding, so the ring is filled from LS threads.
        if (lane < LS) {
            if (lane == 0) {
                tma_prefetch_desc(&tmW);
                tma_prefetch_desc(&tmX);
            }
            const int s = lane;
            int issued = 0;        // stages issued by this lane
            auto load_x = [&](int kb) {
                const uint32_t dst = sb + L::B_OFF + s * L::B_BYTES + rank * (XS * 128);
                if (CL == 1) tma_load_2d(dst, &tmX, full_bar(s), kb * BK, t0);
                else tma_load_2d_mc(dst, &tmX, full_bar(s), kb * BK, t0 + (int)rank * XS, CMASK);
            };
            if (!p.stall) {
                // With a programmatic dependency, the raw weights of the first ring fill are
                // requested before waiting for the guarded activations.
                const bool pre = p.pdl && s < nk;
                if (pre) {
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)(L::R_BYTES + L::B_BYTES));
                    tma_load_2d(sb + L::R_OFF + s * L::R_STRIDE, &tmW, full_bar(s), s * Raw<FMT>::ROW, m0);
                }
                pdl_wait();
                if (pre) {
                    load_x(s);
                    ++issued;
                }
                for (int kb = s + (pre ? LS : 0); kb < nk; kb += LS) {
                    if (!mbar_wait(empty_bar(s), (uint32_t)(((kb / LS) & 1) ^ 1), p.wait_ns, abort_flag)) {
                        give_up();
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)(L::R_BYTES + L::B_BYTES));
                    tma_load_2d(sb + L::R_OFF + s * L::R_STRIDE, &tmW, full_bar(s), kb * Raw<FMT>::ROW, m0);
                    load_x(kb);
                    ++issued;
                }
            } else {
                pdl_wait();   // every path waits once, so kernels later in the stream stay ordered
            }
            if (*abort_flag && issued > 0) {
                // this lane's last copy must land before the CTA can exit
                const int kb_last = s + (issued - 1) * LS;
                mbar_wait(full_bar(s), (uint32_t)((kb_last / LS) & 1), p.wait_ns, never_flag);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ================= MMA issuer =================
        // The whole warp runs the loop (converged); one lane issues the tensor-core work.
        // With the decoded tiles in tensor memory (AM 1) there is one decoded slot per load
        // slot, so one commit frees both and the only wait is the decoders' hand-off.
        constexpr uint32_t idesc = idesc_f16(BM, BN, XBF);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % LS, a = kb % AS;
            bool ok = mbar_wait(afull_bar(a), (uint32_t)((kb / AS) & 1), p.wait_ns, abort_flag);
            if (AM == 0 && ok) ok = mbar_wait(full_bar(s), (uint32_t)((kb / LS) & 1), p.wait_ns, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) give_up();
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t a_base = sb + L::A_OFF + a * A_BYTES;
                const uint32_t b_base = sb + L::B_OFF + s * L::B_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    if (AM == 0)
                        tc_mma_f16(tmem, smem_desc_sw128(a_base + 32 * kk), smem_desc_sw128(b_base + 32 * kk),
                                   idesc, (kb | kk) != 0 ? 1u : 0u);
                    else   // A from tensor memory: 8 columns per K=16 step
                        tc_mma_f16_ts(tmem, tmem + (uint32_t)(L::A_COL + a * 32 + kk * 8),
                                      smem_desc_sw128(b_base + 32 * kk), idesc, (kb | kk) != 0 ? 1u : 0u);
                }
                // raw + activation slot (and, AM 1, its decoded tile) free once these MMAs are
                // done, in every CTA of the cluster, since the peers multicast into this slot too
                if (CL == 1) tc_commit(empty_bar(s));
                else tc_commit_mc(empty_bar(s), CMASK);
                if (AM == 0) tc_commit(aempty_bar(a));   // decoded slot free
            }
            __syncwarp();
        }
        if (lane == 0) tc_commit(accf_bar);   // also lets teardown know every MMA has finished
        __syncwarp();
    } else {
        // ================= decoders (two threads per weight row), then epilogue =================
        const int r = threadIdx.x & (BM - 1);      // weight row within the tile
        const int h = threadIdx.x >> 7;            // which 32-k half of the 64-k stage
        const int64_t n = (int64_t)m0 + r;
        const bool row_ok = n < p.N;
        const uint32_t a_row = (uint32_t)(r * 128);
        const uint32_t xr = (uint32_t)(r & 7);
        // Q4 scales: 8 fp16 (4 stages x 2 blocks) per 16-byte load, one group ahead
        uint4 sc_cur = make_uint4(0, 0, 0, 0), sc_next = make_uint4(0, 0, 0, 0);
        const uint16_t* srow = p.ws + n * (p.K / 32);
        if (FMT == 0 && row_ok) sc_next = __ldg(reinterpret_cast<const uint4*>(srow));
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % LS, a = kb % AS;
            if (FMT == 0 && (kb & 3) == 0) {
                sc_cur = sc_next;
                if (row_ok && kb + 4 < nk) sc_next = __ldg(reinterpret_cast<const uint4*>(srow + 2 * (kb + 4)));
            }
            // AM 1: decoded slot a == load slot s, free once the slot was refilled
            if (!mbar_wait(full_bar(s), (uint32_t)((kb / LS) & 1), p.wait_ns, abort_flag) ||
                (AM == 0 && !mbar_wait(aempty_bar(a), (uint32_t)(((kb / AS) & 1) ^ 1), p.wait_ns, abort_flag))) {
                give_up();
                break;
            }
            const uint32_t raw = sb + L::R_OFF + s * L::R_STRIDE;
            const uint32_t adst = sb + L::A_OFF + a * A_BYTES + a_row;
            // this thread's 32 decoded values (k = 32h .. 32h+31 of the stage), two per word, in k order
            uint32_t o[16];
            if (FMT == 0) {
                // 32-byte rows, 32-byte swizzle: chunk j of row r sits at j ^ ((r >> 2) & 1)
                const uint4 v = ld_shared_v4(raw + r * 32 + (((uint32_t)h ^ (uint32_t)((r >> 2) & 1)) << 4));
                const uint32_t kq = (uint32_t)(kb & 3);
                const uint32_t w2 = kq == 0 ? sc_cur.x : kq == 1 ? sc_cur.y : kq == 2 ? sc_cur.z : sc_cur.w;
                const uint16_t sbits = (uint16_t)(h ? (w2 >> 16) : (w2 & 0xFFFF));
                const __half2 sh = __halves2half2(__ushort_as_half(sbits), __ushort_as_half(sbits));
                const uint32_t px = prmt(v.x, 0u, 0x3120u), py = prmt(v.y, 0u, 0x3120u);
                const uint32_t pz = prmt(v.z, 0u, 0x3120u), pw = prmt(v.w, 0u, 0x3120u);
                // elements 0-7 of the block: low nibbles of bytes 0-7
                o[0] = hmul2_u32(nib2_to_h2(px), sh);
                o[1] = hmul2_u32(nib2_to_h2(px >> 8), sh);
                o[2] = hmul2_u32(nib2_to_h2(py), sh);
                o[3] = hmul2_u32(nib2_to_h2(py >> 8), sh);
                // elements 8-15: low nibbles of bytes 8-15
                o[4] = hmul2_u32(nib2_to_h2(pz), sh);
                o[5] = hmul2_u32(nib2_to_h2(pz >> 8), sh);
                o[6] = hmul2_u32(nib2_to_h2(pw), sh);
                o[7] = hmul2_u32(nib2_to_h2(pw >> 8), sh);
                // elements 16-23: high nibbles of bytes 0-7
                o[8] = hmul2_u32(nib2_to_h2(px >> 4), sh);
                o[9] = hmul2_u32(nib2_to_h2(px >> 12), sh);
                o[10] = hmul2_u32(nib2_to_h2(py >> 4), sh);
                o[11] = hmul2_u32(nib2_to_h2(py >> 12), sh);
                // elements 24-31: high nibbles of bytes 8-15
                o[12] = hmul2_u32(nib2_to_h2(pz >> 4), sh);
                o[13] = hmul2_u32(nib2_to_h2(pz >> 12), sh);
                o[14] = hmul2_u32(nib2_to_h2(pw >> 4), sh);
                o[15] = hmul2_u32(nib2_to_h2(pw >> 12), sh);
            } else {
                // 64-byte rows, 64-byte swizzle: chunk j of row r sits at j ^ ((r >> 1) & 3)
                const uint32_t sw = (uint32_t)((r >> 1) & 3);
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const uint32_t q = (uint32_t)(2 * h + qq);
                    const uint4 v = ld_shared_v4(raw + r * 64 + ((q ^ sw) << 4));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (XBF) {
                            const uint32_t wx = wv[i] ^ 0x80808080u;
                            o[8 * qq + 2 * i] = pack_bf2(i8_to_f32(wx, 0x7440u), i8_to_f32(wx, 0x7441u));
                            o[8 * qq + 2 * i + 1] = pack_bf2(i8_to_f32(wx, 0x7442u), i8_to_f32(wx, 0x7443u));
                        } else {
                            o[8 * qq + 2 * i] = i8x2_to_h2(wv[i], 0x4140u);
                            o[8 * qq + 2 * i + 1] = i8x2_to_h2(wv[i], 0x4342u);
                        }
                    }
                }
            }
            if (AM == 0) {
                // shared-memory A tile, 128-byte swizzled K-major: 16-byte chunk 4h+j of row r
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    st_shared_v4(adst + ((((uint32_t)(4 * h + j)) ^ xr) << 4), o[4 * j], o[4 * j + 1], o[4 * j + 2],
                                 o[4 * j + 3]);
                fence_proxy_async_smem();
                mbar_arrive(afull_bar(a));
            } else {
                // tensor-memory A tile: lane r, columns A_COL + 32a + 16h .. +15.  The store
                // of this stage is handed to the MMA one stage later, so its latency overlaps
                // the next stage's wait and decode.
                if (kb > 0) {
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(afull_bar((kb - 1) % AS));
                }
                tmem_st_32x32b_x16(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(L::A_COL + a * 32 + 16 * h), o);
                if (kb + 1 == nk) {
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(afull_bar(a));
                }
            }
        }

        // ---- epilogue: TMEM -> registers -> scale -> Y[t][n] ----
        // warp w reads TMEM lanes 32*(w % 4).. and the columns of half w / 4
        if (!*abort_flag && mbar_wait(accf_bar, 0, p.wait_ns, abort_flag)) {
            tc_fence_after();
            pdl_wait();   // outputs and guard scales only after the previous kernel has finished
            const float rsn = (FMT == 1 && row_ok) ? p.rs[n] : 0.f;
            const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll 1
            for (int cc = h * (BN / 64); cc < (h + 1) * (BN / 64); ++cc) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + lane_base + (uint32_t)(cc * 32), v);
                tmem_ld_wait();
                const int64_t tb = (int64_t)t0 + cc * 32;
                float rsx_l = 0.f;
                if (FMT == 0 && tb + lane < p.T) rsx_l = p.rsx[tb + lane];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float sx = FMT == 0 ? __shfl_sync(0xffffffffu, rsx_l, j) : rsn;
                    const int64_t t = tb + j;
                    if (row_ok && t < p.T) {
                        const float val = __uint_as_float(v[j]) * sx;
                        if (p.yt == CQ_F32) reinterpret_cast<float*>(p.y)[t * p.N + n] = val;
                        else reinterpret_cast<__nv_bfloat16*>(p.y)[t * p.N + n] = __float2bfloat16_rn(val);
                    }
                }
            }
        } else if (!*abort_flag) {
            give_up();
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
    // no CTA leaves while a peer may still multicast into it or signal its barriers
    if (CL > 1) cluster_sync_all();
}

template <int FMT, int BN, int XBF, int LS, int AS, int CL, int AM>
cudaError_t launch_bn(const CUtensorMap& mw, const CUtensorMap& mx, const Params& p, dim3 grid, cudaStream_t s) {
    using L = Layout<FMT, BN, LS, AS, AM>;
    static_assert(L::TOTAL <= 232448, "shared memory budget");
    static_assert(LS <= 32, "one producer lane per ring slot");
    static_assert(AM == 0 || AS == LS, "tensor-memory decoded slots pair with load slots");
    auto kern = k_tc<FMT, BN, XBF, LS, AS, CL, AM>;
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
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = CL;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
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
    int bn = (int)options().tc_bn;
    if (bn != 64 && bn != 128 && bn != 256) {
        bn = 256;
        if (mt * ((a.T + 255) / 256) < num_sms()) bn = 128;
        if (bn == 128 && mt * ((a.T + 127) / 128) < num_sms() && a.T <= 64) bn = 64;
    }
    // cluster size along the weight rows (the activation tile is multicast)
    int cl = (int)options().tc_cluster;
    if (cl != 1 && cl != 2 && cl != 4) {
        const int64_t ctas = mt * ((a.T + bn - 1) / bn);
        cl = (mt >= 4 && ctas <= 128) ? 4 : (mt >= 2 ? 2 : 1);
    }
    CUtensorMap mw, mx;
    {
        const uint64_t kbytes = fmt == 0 ? (uint64_t)a.K / 2 : (uint64_t)a.K;
        uint64_t d[2] = {kbytes, (uint64_t)a.N};
        uint64_t st[1] = {kbytes};
        uint32_t box[2] = {(uint32_t)(fmt == 0 ? 32 : 64), (uint32_t)BM};
        if (!encode_tiled(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.wq, d, st, box,
                          fmt == 0 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    }
    {
        uint64_t d[2] = {(uint64_t)a.K, (uint64_t)a.T};
        uint64_t st[1] = {(uint64_t)a.K * 2};
        uint32_t box[2] = {(uint32_t)BK, (uint32_t)(bn / cl)};
        if (!encode_tiled(&mx, xbf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.x, d,
                          st, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
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
    p.pdl = fmt == 0 ? 1 : 0;     // Q4: the guard pass just before touches neither weights nor Y
    // grid x padded to whole clusters: extra CTAs see only zero-filled weight rows and store nothing
    const int64_t gx = (mt + cl - 1) / cl * cl;
    dim3 grid((unsigned)gx, (unsigned)((a.T + bn - 1) / bn), 1);
    if (options().trace)
        fprintf(stderr, "cq: tcgen05 fmt=%d T=%lld N=%lld K=%lld BN=%d cluster=%d grid=(%u,%u)\n", fmt,
                (long long)a.T, (long long)a.N, (long long)a.K, bn, cl, grid.x, grid.y);
    // decoded weight operand: 1 = shared memory, 2 = tensor memory (default)
    const int am = options().tc_amode == 1 ? 0 : 1;
#define CQ_TC_CL(F, B, X, LSv, ASv, AMv)                                                  \
    do {                                                                                  \
        if (cl == 4) return launch_bn<F, B, X, LSv, ASv, 4, AMv>(mw, mx, p, grid, s);      \
        if (cl == 2) return launch_bn<F, B, X, LSv, ASv, 2, AMv>(mw, mx, p, grid, s);      \
        return launch_bn<F, B, X, LSv, ASv, 1, AMv>(mw, mx, p, grid, s);                  \
    } while (0)
    if (am == 0) {
        if (fmt == 0) {
            if (bn == 256) CQ_TC_CL(0, 256, 0, 5, 2, 0);
            if (bn == 128) CQ_TC_CL(0, 128, 0, 8, 3, 0);
            CQ_TC_CL(0, 64, 0, 12, 4, 0);
        }
        if (xbf) {
            if (bn == 256) CQ_TC_CL(1, 256, 1, 4, 3, 0);
            if (bn == 128) CQ_TC_CL(1, 128, 1, 7, 3, 0);
            CQ_TC_CL(1, 64, 1, 10, 4, 0);
        }
        if (bn == 256) CQ_TC_CL(1, 256, 0, 4, 3, 0);
        if (bn == 128) CQ_TC_CL(1, 128, 0, 7, 3, 0);
        CQ_TC_CL(1, 64, 0, 10, 4, 0);
    }
    // AM 1: one tensor-memory decoded slot per load slot (AS == LS)
    if (fmt == 0) {
        if (bn == 256) CQ_TC_CL(0, 256, 0, 6, 6, 1);
        if (bn == 128) CQ_TC_CL(0, 128, 0, 10, 10, 1);
        CQ_TC_CL(0, 64, 0, 14, 14, 1);
    }
    if (xbf) {
        if (bn == 256) CQ_TC_CL(1, 256, 1, 5, 5, 1);
        if (bn == 128) CQ_TC_CL(1, 128, 1, 9, 9, 1);
        CQ_TC_CL(1, 64, 1, 13, 13, 1);
    }
    if (bn == 256) CQ_TC_CL(1, 256, 0, 5, 5, 1);
    if (bn == 128) CQ_TC_CL(1, 128, 0, 9, 9, 1);
    CQ_TC_CL(1, 64, 0, 13, 13, 1);
#undef CQ_TC_CL
}

}  // namespace

cudaError_t launch_tc_q4(const TcArgs& a, cudaStream_t s) { return launch(0, a, s); }
cudaError_t launch_tc_q8(const TcArgs& a, cudaStream_t s) { return launch(1, a, s); }

}  // namespace cq
