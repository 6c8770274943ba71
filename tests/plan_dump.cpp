// Prints the single-token decode kernel's launch plan for the shapes given
// on standard input, one JSON object per line, for the host-side checks in
// test_plan_cpu.py.  Input lines: d d_out k elem_bytes ncta smem_budget grid.
#include <cstdio>

#include "gsi_plan.h"

int main() {
  long long d, d_out, k, budget;
  int es, ncta, grid;
  while (std::scanf("%lld %lld %lld %d %d %lld %d", &d, &d_out, &k, &es, &ncta, &budget, &grid) == 7) {
    const gsi::DecodePlan p = gsi::plan_decode(d, d_out, k, es, ncta, size_t(budget), grid != 0);
    const gsi::FusedLayout L = gsi::layout_fused(k, 1);  // the one-token call's workspace
    std::printf(
        "{\"d\": %lld, \"d_out\": %lld, \"k\": %lld, \"es\": %d, \"ncta\": %d, \"budget\": %lld, \"grid_req\": %d, "
        "\"ok\": %d, \"vr\": %d, \"rw\": %d, \"rpc\": %d, \"ks\": %d, \"seg_bytes\": %d, \"sw\": %d, "
        "\"red_stride\": %d, \"m_late\": %d, \"grid\": %d, \"off_g\": %d, \"off_y\": %d, \"off_in\": %d, "
        "\"off_gram\": %d, \"off_red\": %d, \"off_v\": %d, \"off_m\": %d, \"smem\": %zu, "
        "\"nw\": %d, \"cluster\": %d, \"max_stages\": %d, \"bars\": %d, \"max_clusters\": %d, "
        "\"ws_part_g\": %zu, \"ws_part_x\": %zu, \"ws_total\": %zu, \"words_off\": %d, \"words\": %d}\n",
        d, d_out, k, es, ncta, budget, grid, int(p.ok), p.vr, p.rw, p.rpc, p.ks, p.seg_bytes, p.sw, p.red_stride,
        p.m_late, p.grid, p.off_g, p.off_y, p.off_in, p.off_gram, p.off_red, p.off_v, p.off_m, p.smem,
        gsi::kApplyThreads / 32, gsi::kDecodeCluster, gsi::kDecodeMaxStages, gsi::kDecodeBars,
        gsi::kDecodeMaxClusters, L.part_x - L.part_g, L.total - L.part_x, L.total, gsi::kDecodeWordsOff,
        gsi::kDecodeCtaWords);
  }
  return 0;
}
