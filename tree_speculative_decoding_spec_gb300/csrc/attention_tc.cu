// Tensor-core (tcgen05) path of tree attention.
#include "attention_tc.cuh"

namespace spec {
namespace tc {

bool attn_tc_supported(int, int) { return false; }

AttnTcPlan attn_tc_plan(int, int, int, int, int, int, int) { return AttnTcPlan{}; }

spec_status attn_tc_run(const AttnTcPlan&, const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*,
                        const int32_t*, const __nv_bfloat16*, const __nv_bfloat16*, const spec_tree*, int, int, int,
                        int, int, float, float*, float*, void*, cudaStream_t) {
    return fail(SPEC_EUNSUPPORTED, "tensor-core attention path not built");
}

}  // namespace tc
}  // namespace spec
