// Tensor-core (tcgen05) path of the draft heads.
#include "draft_tc.cuh"

namespace spec {
namespace tc {

bool draft_tc_supported(int, int) { return false; }

DraftTcPlan draft_tc_plan(int rows, int, int, int, int) {
    DraftTcPlan p;
    p.rows_pad = rows;
    return p;
}

spec_status draft_head_tc(const DraftTcPlan&, const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*,
                          const __nv_bfloat16*, const __nv_bfloat16*, int, int, __nv_bfloat16*, int, int, int, int, int,
                          int, int, float*, draft::Cand*, float2*, void*, cudaStream_t) {
    return fail(SPEC_EUNSUPPORTED, "tensor-core draft path not built");
}

}  // namespace tc
}  // namespace spec
