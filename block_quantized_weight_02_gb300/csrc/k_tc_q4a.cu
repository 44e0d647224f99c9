// Large-T GEMM for affine Q4 weights ("oxinfer 0.0.5 src/metal.rs",
// Dequantizers, struct Q4A: the Q4 split plane plus one bf16 offset per group
// of gk blocks of 32) on the tcgen05 tensor cores: the affine-mode
// instantiations of the kernel in k_tc.cuh.  The decoders form each weight as
// fp16((nibble - 8) * scale + fp16(offset)) with one rounding, so the
// contraction and the epilogue are those of the plain Q4 GEMM; the offsets
// cost two scalar loads per row and stage, prefetched with the block scales.
#include "k_tc.cuh"

namespace cq {

cudaError_t launch_tc_q4a(const TcArgs& a, cudaStream_t s) {
    if (!a.off || a.gk < 1 || a.jobs() != 1) return cudaErrorInvalidValue;
    const int64_t mt = (a.N + BM - 1) / BM;
    const Plan pl = plan_tiles(a, mt, false);
    Params p = make_params(a);
    p.tiles_y = (int)((a.T + pl.bn - 1) / pl.bn);
    dim3 grid((unsigned)mt, (unsigned)p.tiles_y, (unsigned)pl.ks);
    trace_plan("affine", 0, a, pl, (pl.bn >= 128 || pl.bn == 32) && pl.pair_ok, grid);
    return launch_q4_tmem<2>(a, p, pl, grid, s);
}

}  // namespace cq
