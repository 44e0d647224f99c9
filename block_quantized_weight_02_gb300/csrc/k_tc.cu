// Large-T Q4 / Q8-row GEMMs on the tcgen05 tensor cores: the dense
// instantiations of the kernel in k_tc.cuh (which describes the design).
#include "k_tc.cuh"

namespace cq {
namespace {

// One launch of the plan's tile shape over grid = (row tiles, token tiles x jobs, K split).
cudaError_t launch_one(int fmt, int xbf, int am, const Plan& pl, const TcArgs& a, const Params& p, dim3 grid,
                       cudaStream_t s) {
    const int bn = pl.bn, ks = pl.ks;
    const bool pair = am == 1 && (bn >= 128 || bn == 32) && pl.pair_ok;
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
    if (fmt == 0) return launch_q4_tmem_one<0>(a, p, pl, grid, s);
    if (xbf) {
        if (bn == 192) return launch_bn<1, 192, 1, 2, 5, 8, 1, 1, 2>(a, p, grid, s);
        if (bn == 32) {
            if (pair) return ks == 2 ? launch_bn<1, 32, 1, 2, 10, 12, 1, 2, 2>(a, p, grid, s) : launch_bn<1, 32, 1, 2, 10, 12, 1, 1, 2>(a, p, grid, s);
            return ks == 2 ? launch_bn<1, 32, 1, 2, 8, 12, 1, 2>(a, p, grid, s) : launch_bn<1, 32, 1, 2, 8, 12, 1, 1>(a, p, grid, s);
        }
        if (pair && bn == 128) return ks == 2 ? launch_bn<1, 128, 1, 2, 6, 12, 1, 2, 2>(a, p, grid, s) : launch_bn<1, 128, 1, 2, 6, 12, 1, 1, 2>(a, p, grid, s);
        if (pair) return ks == 2 ? launch_bn<1, 256, 1, 2, 4, 8, 1, 2, 2>(a, p, grid, s) : launch_bn<1, 256, 1, 2, 4, 8, 1, 1, 2>(a, p, grid, s);
        if (bn == 256) return ks == 2 ? launch_bn<1, 256, 1, 1, 5, 8, 1, 2>(a, p, grid, s) : launch_bn<1, 256, 1, 1, 5, 8, 1, 1>(a, p, grid, s);
        if (bn == 128) return ks == 2 ? launch_bn<1, 128, 1, 2, 4, 12, 1, 2>(a, p, grid, s) : launch_bn<1, 128, 1, 2, 4, 12, 1, 1>(a, p, grid, s);
        return launch_bn<1, 64, 1, 2, 6, 12, 1>(a, p, grid, s);
    }
    if (bn == 192) return launch_bn<1, 192, 0, 2, 5, 8, 1, 1, 2>(a, p, grid, s);
    if (bn == 32) {
        if (pair) return ks == 2 ? launch_bn<1, 32, 0, 2, 10, 12, 1, 2, 2>(a, p, grid, s) : launch_bn<1, 32, 0, 2, 10, 12, 1, 1, 2>(a, p, grid, s);
        return ks == 2 ? launch_bn<1, 32, 0, 2, 8, 12, 1, 2>(a, p, grid, s) : launch_bn<1, 32, 0, 2, 8, 12, 1, 1>(a, p, grid, s);
    }
    if (pair && bn == 128) return ks == 2 ? launch_bn<1, 128, 0, 2, 6, 12, 1, 2, 2>(a, p, grid, s) : launch_bn<1, 128, 0, 2, 6, 12, 1, 1, 2>(a, p, grid, s);
    if (pair) return ks == 2 ? launch_bn<1, 256, 0, 2, 4, 8, 1, 2, 2>(a, p, grid, s) : launch_bn<1, 256, 0, 2, 4, 8, 1, 1, 2>(a, p, grid, s);
    if (bn == 256) return ks == 2 ? launch_bn<1, 256, 0, 1, 5, 8, 1, 2>(a, p, grid, s) : launch_bn<1, 256, 0, 1, 5, 8, 1, 1>(a, p, grid, s);
    if (bn == 128) return ks == 2 ? launch_bn<1, 128, 0, 2, 4, 12, 1, 2>(a, p, grid, s) : launch_bn<1, 128, 0, 2, 4, 12, 1, 1>(a, p, grid, s);
    return launch_bn<1, 64, 0, 2, 6, 12, 1>(a, p, grid, s);
}

cudaError_t launch(int fmt, const TcArgs& a, cudaStream_t s) {
    const int xbf = fmt == 0 ? 0 : a.x_bf16;
    const int64_t mt = (a.N + BM - 1) / BM;
    const Plan pl = plan_tiles(a, mt, false);
    Params p = make_params(a);
    p.tiles_y = (int)((a.T + pl.bn - 1) / pl.bn);
    dim3 grid((unsigned)mt, (unsigned)(p.tiles_y * a.jobs()), (unsigned)pl.ks);
    // decoded weight operand: 1 = shared memory, 2 = tensor memory (default)
    const int am = options().tc_amode == 1 ? 0 : 1;
    const bool pair = am == 1 && (pl.bn >= 128 || pl.bn == 32) && pl.pair_ok;
    trace_plan("dense", fmt, a, pl, pair, grid);
    // a partial last wave of full-length tiles moves into a second, K-split launch
    const Tail tl = am == 1 ? tail_plan(pl, pair, mt, a.T, a.jobs(), a.K) : Tail{0, 0};
    if (tl.r == 0) return launch_one(fmt, xbf, am, pl, a, p, grid, s);
    cudaError_t e = launch_one(fmt, xbf, am, pl, a, p, dim3((unsigned)(mt - tl.r), grid.y, 1), s);
    if (e != cudaSuccess) return e;
    Params pt = p;
    pt.mt0 = (int)(mt - tl.r);
    pt.tiles_y = (int)((a.T + tl.bn - 1) / tl.bn);
    const Plan plt = {tl.bn, 2, pl.pair_ok};
    const dim3 gt((unsigned)tl.r, (unsigned)(pt.tiles_y * a.jobs()), 2);
    trace_plan("tail", fmt, a, plt, pair, gt);
    return launch_one(fmt, xbf, am, plt, a, pt, gt, s);
}

}  // namespace

cudaError_t launch_tc_q4(const TcArgs& a, cudaStream_t s) { return launch(0, a, s); }
cudaError_t launch_tc_q8(const TcArgs& a, cudaStream_t s) { return launch(1, a, s); }

}  // namespace cq
