// Tensor-core (tcgen05) path of the draft heads, bf16 weights.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace spec {
namespace draft {
// A top-k candidate (logit, token); "better" = larger logit, then lower token.
struct Cand {
    float v;
    int i;
};
}  // namespace draft
namespace tc {

struct DraftTcPlan {
    int rows_pad = 0;              // rows padded to the MMA N granule
    int nslices = 0;               // vocabulary slices (one per 128-row W2 tile)
};

bool draft_tc_supported(int d, int V);
DraftTcPlan draft_tc_plan(int rows, int d, int V);

// One head: the MLP (split over K; the last split of each weight tile applies
// bias, SiLU, residual and bf16 rounding) then the projection with per-slice
// top-k and (max, sum exp) partials.  X holds the head's input rows (row stride
// ldx: the gathered [h || E[tok]] rows, or h itself for an unconditioned head);
// z receives the bf16 MLP output.  Kernels are launched with programmatic
// dependent launch.
// One head layer on the tensor cores for R activation rows:
//   y[r, m] = act(W[m, :] . X[r, 0:d_in] + bias[m]) (+ residual[b(r), m]),  m < M
// (act 1: SiLU, 0: identity; b(r) = r / n_int when cond, else r), stored as
// bf16 in z [R, M] or, when zf is set, as fp32 in zf [R, M].  Input columns
// >= dep_k0 come from the previous kernel.  W's rows are ldw elements apart
// (0: d_in); bias, residual and ws (the status word) may be NULL.
spec_status mlp_tc(const __nv_bfloat16* W, const __nv_bfloat16* bias, int M, const __nv_bfloat16* X, int d_in, int ldx,
                   int R, int cond, int n_int, int dep_k0, int act, const __nv_bfloat16* residual, __nv_bfloat16* z,
                   float* zf, void* ws, cudaStream_t s, int ldw = 0);

// The vocabulary projection with the per-slice top-k / (max, sum exp) epilogue.
spec_status proj_tc(const DraftTcPlan& plan, const __nv_bfloat16* W2, const __nv_bfloat16* z, int R, int d, int V, int k,
                    int kmax, draft::Cand* pc, float2* pl, void* ws, cudaStream_t s);

spec_status draft_head_tc(const DraftTcPlan& p, const __nv_bfloat16* W1, const __nv_bfloat16* b1,
                          const __nv_bfloat16* W2, const __nv_bfloat16* h, const __nv_bfloat16* X, int d_in, int ldx,
                          __nv_bfloat16* z, int R, int d, int V, int cond, int n_int, int k, int kmax, int dep_k0,
                          draft::Cand* pc, float2* pl, void* ws, cudaStream_t s);

}  // namespace tc
}  // namespace spec
