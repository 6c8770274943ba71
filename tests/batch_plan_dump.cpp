// Prints the small-batch decode kernel's launch plan for the shapes given on
// standard input, one JSON object per line, for the host-side checks in
// test_batch_plan_cpu.py.  Input lines: d d_out k T ncta smem_budget.
#include <cstdio>

#include "gsi_plan.h"

int main() {
  long long d, d_out, k, T, budget;
  int ncta;
  while (std::scanf("%lld %lld %lld %lld %d %lld", &d, &d_out, &k, &T, &ncta, &budget) == 6) {
    const gsi::BatchPlan p = gsi::plan_batch(d, d_out, k, T, ncta, size_t(budget));
    const gsi::BatchLayout L = gsi::layout_batch(k, T);
    std::printf(
        "{\"d\": %lld, \"d_out\": %lld, \"k\": %lld, \"T\": %lld, \"ncta\": %d, \"budget\": %lld, \"ok\": %d, "
        "\"vr\": %d, \"rpc\": %d, \"ks\": %d, \"kb\": %d, \"stages\": %d, \"stage_bytes\": %d, \"gbf_pitch\": %d, "
        "\"xs_pitch\": %d, \"off_gbf\": %d, \"off_dec\": %d, \"off_wsh\": %d, \"off_scr\": %d, \"off_v\": %d, "
        "\"off_xs\": %d, \"off_in\": %d, \"off_nin\": %d, \"off_g32\": %d, \"off_qin\": %d, \"off_gram\": %d, "
        "\"off_m\": %d, \"off_fs\": %d, \"off_nx\": %d, \"smem\": %zu, \"threads\": %d, \"warps\": %d, \"maxT\": %d, \"cluster\": %d, "
        "\"max_clusters\": %d, \"max_k\": %d, \"max_mt\": %d, \"kc\": %d, \"max_stages\": %d, \"slack\": %d, "
        "\"ws_part_g\": %zu, \"ws_part_x\": %zu, \"ws_total\": %zu}\n",
        d, d_out, k, T, ncta, budget, int(p.ok), p.vr, p.rpc, p.ks, p.kb, p.stages, p.stage_bytes, p.gbf_pitch,
        p.xs_pitch, p.off_gbf, p.off_dec, p.off_wsh, p.off_scr, p.off_v, p.off_xs, p.off_in, p.off_nin, p.off_g32,
        p.off_qin, p.off_gram, p.off_m, p.off_fs, p.off_nx, p.smem, gsi::kBatchThreads, gsi::kBatchWarps, gsi::kBatchMaxT,
        gsi::kBatchCluster, gsi::kBatchMaxClusters, gsi::kBatchMaxK, gsi::kBatchMaxMt, gsi::kBatchKC, gsi::kBatchMaxStages,
        gsi::kBatchSmemSlack, L.part_g, L.part_x, L.total);
  }
  return 0;
}
