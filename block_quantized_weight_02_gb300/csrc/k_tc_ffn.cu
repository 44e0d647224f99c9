// The gate/up GEMM of the dense FFN chain on the tcgen05 tensor cores: the
// gate/up (SwiGLU epilogue) instantiations of the kernel in k_tc.cuh.  Each
// CTA owns 64 gate rows and the matching 64 up rows of the [2I][K] Q4 weight,
// so a = silu(g) * u is formed from its own accumulator and written in f32.
#include "k_tc.cuh"

namespace cq {

cudaError_t launch_tc_q4_gateup(const TcArgs& a, cudaStream_t s) {
    // a.N is I (gate rows); a row tile is 64 gate rows and their 64 up rows
    const int64_t mt = (a.N + BM / 2 - 1) / (BM / 2);
    const Plan pl = plan_tiles(a, mt, true);
    Params p = make_params(a);
    p.y_tma = 0;    // a[T][I] f32 leaves by direct stores after the SwiGLU
    p.tiles_y = (int)((a.T + pl.bn - 1) / pl.bn);
    dim3 grid((unsigned)mt, (unsigned)p.tiles_y, (unsigned)pl.ks);
    trace_plan("gate/up", 0, a, pl, (pl.bn >= 128 || pl.bn == 32) && pl.pair_ok, grid);
    return launch_q4_tmem<1>(a, p, pl, grid, s);
}

}  // namespace cq
