// C entry to the GEMM planner header for the CPU tests (compiled by tests/test_gemm_plan.py).
#include "gemm_plan.h"

extern "C" void gemm_plan(int M, int N, int K, int bn, int weight, int splittable, int num_sms, int quads,
                          unsigned long long split_ws_bytes, long long* out)
{
    const mlp::GemmPlan p = mlp::plan_gemm(M, N, K, bn, weight, splittable != 0, num_sms, quads,
                                           static_cast<size_t>(split_ws_bytes));
    const long long v[11] = {p.bn, p.cg, p.cluster_pairs, p.tm, p.units, p.tiles, p.split_tiles, p.split_k,
                             p.grid, p.n_fastest, p.raster_group};
    for (int i = 0; i < 11; ++i) out[i] = v[i];
}
