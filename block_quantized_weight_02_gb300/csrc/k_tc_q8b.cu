// Large-T GEMM for Q8 per-32-k-block weights ("oxinfer 0.0.5 src/metal.rs",
// Dequantizers, struct Q8W: int8 weights, one f32 scale per 32 k) on the
// tcgen05 tensor cores: the FMT = 2 instantiations of the kernel in k_tc.cuh.
// The decoders turn each int8 pair into fp16 exactly and multiply it by its
// block's scale rounded to fp16 (one rounding of q * fp16(scale)); the
// activations arrive as fp16 in k order behind the per-row power-of-two guard,
// whose inverse the epilogue applies.
#include "k_tc.cuh"

namespace cq {

cudaError_t launch_tc_q8b(const TcArgs& a, cudaStream_t s) {
    const int64_t mt = (a.N + BM - 1) / BM;
    const Plan pl = plan_tiles(a, mt, true);
    const int bn = pl.bn, ks = pl.ks;
    Params p = make_params(a);
    p.tiles_y = (int)((a.T + bn - 1) / bn);
    dim3 grid((unsigned)mt, (unsigned)(p.tiles_y * a.jobs()), (unsigned)ks);
    const bool pair = (bn >= 128 || bn == 32) && pl.pair_ok;
    trace_plan("q8/32", 2, a, pl, pair, grid);
    // <FMT, BN, XBF, G, LSS, AS, AM, KS, CG>: the ring shapes of the Q8-row kernel with fp16 activations
    if (bn == 192) return launch_bn<2, 192, 0, 2, 5, 8, 1, 1, 2>(a, p, grid, s);
    if (bn == 32) {
        if (pair) return ks == 2 ? launch_bn<2, 32, 0, 2, 10, 12, 1, 2, 2>(a, p, grid, s) : launch_bn<2, 32, 0, 2, 10, 12, 1, 1, 2>(a, p, grid, s);
        return ks == 2 ? launch_bn<2, 32, 0, 2, 8, 12, 1, 2>(a, p, grid, s) : launch_bn<2, 32, 0, 2, 8, 12, 1, 1>(a, p, grid, s);
    }
    if (pair && bn == 128) return ks == 2 ? launch_bn<2, 128, 0, 2, 6, 12, 1, 2, 2>(a, p, grid, s) : launch_bn<2, 128, 0, 2, 6, 12, 1, 1, 2>(a, p, grid, s);
    if (pair) return ks == 2 ? launch_bn<2, 256, 0, 2, 4, 8, 1, 2, 2>(a, p, grid, s) : launch_bn<2, 256, 0, 2, 4, 8, 1, 1, 2>(a, p, grid, s);
    if (bn == 256) return ks == 2 ? launch_bn<2, 256, 0, 1, 5, 8, 1, 2>(a, p, grid, s) : launch_bn<2, 256, 0, 1, 5, 8, 1, 1>(a, p, grid, s);
    if (bn == 128) return ks == 2 ? launch_bn<2, 128, 0, 2, 4, 12, 1, 2>(a, p, grid, s) : launch_bn<2, 128, 0, 2, 4, 12, 1, 1>(a, p, grid, s);
    return launch_bn<2, 64, 0, 2, 6, 12, 1>(a, p, grid, s);
}

}  // namespace cq
