// Prints the tensor-core path's workspace layout and finalize plan for the
// shapes given on standard input, one JSON object per line, for the host-side
// checks in test_tensor_plan_cpu.py.  Input lines: d k T.
#include <cstdio>

#include "gsi_plan.h"

int main() {
  long long d, k, T;
  while (std::scanf("%lld %lld %lld", &d, &k, &T) == 3) {
    const gsi::TensorLayout L = gsi::layout_tensor(d, k, T);
    std::printf(
        "{\"d\": %lld, \"k\": %lld, \"T\": %lld, \"nb\": %d, \"fin_smem\": %zu, \"gsplit\": %d, \"ctrl\": %zu, "
        "\"vt\": %zu, \"g\": %zu, \"gbf\": %zu, \"gfast\": %zu, \"xslow\": %zu, \"idx\": %zu, \"gt\": %zu, "
        "\"norms\": %zu, \"total\": %zu, \"fin_tok\": %d, \"norm_threads\": %d, \"fin_threads\": %d, "
        "\"fin_cols\": %d, \"fin_stages\": %d, \"fin_stage_bytes\": %lld, \"fin_max_blocks\": %d, "
        "\"gsplit_max\": %d}\n",
        d, k, T, gsi::fin_blocks(T, k), gsi::fin_smem(k), gsi::g_split(T), L.ctrl, L.vt, L.g, L.gbf, L.gfast,
        L.xslow, L.idx, L.gt, L.norms, L.total, gsi::kFinTok, gsi::kNormThreads, gsi::kFinThreads, gsi::kFinCols,
        gsi::kFinStages, (long long)gsi::kFinStageBytes, gsi::kFinMaxBlocks, gsi::kGSplitMax);
  }
  return 0;
}
