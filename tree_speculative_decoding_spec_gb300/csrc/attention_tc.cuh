// Tensor-core (tcgen05) path of tree attention, bf16 inputs.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace spec {
namespace tc {

struct AttnTcPlan {
    size_t part_bytes = 0;
};

bool attn_tc_supported(int rows_per_kv_head, int D);
AttnTcPlan attn_tc_plan(int B, int Hq, int Hkv, int T, int Lmax, int D, int sm_count);
spec_status attn_tc_run(const AttnTcPlan& p, const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc,
                        const int32_t* prefix_len, const __nv_bfloat16* kt, const __nv_bfloat16* vt,
                        const spec_tree* tree, int B, int Hq, int Hkv, int Lmax, int D, float scale, float* out,
                        float* lse, void* ws, cudaStream_t s);

}  // namespace tc
}  // namespace spec
