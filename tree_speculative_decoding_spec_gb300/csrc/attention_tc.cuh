// Tensor-core (tcgen05) path of tree attention, bf16 inputs, head dim 128.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace spec {
namespace tc {

// Addressing of the cached prefix.  table == nullptr: contiguous caches
// [B, Hkv, Lmax, D].  Otherwise a paged pool [num_blocks, Hkv, bs, D]:
// position j of sequence b lives in pool block table[b * max_blocks + j / bs],
// row j % bs (bs a multiple of 64).
struct KvPages {
    const int32_t* table = nullptr;
    int max_blocks = 0;
    int bs = 0;
    int num_blocks = 0;
};

struct AttnTcPlan {
    int n_rb = 0;       // 128-row query blocks per KV head
    int chunk = 0;      // prefix keys per split (multiple of 128)
    int n_pre = 0;      // prefix splits; split n_pre holds the tree keys
    bool fused = false; // the splits of a (head, row block, sequence) form one cluster and merge on chip
    size_t part_bytes = 0;   // split partials in HBM (none with a single split or an on-chip merge)
};

// Used when there are at least 64 query rows per KV head (tree nodes x query
// heads per KV head) and the head dimension is 128.
bool attn_tc_supported(int rows_per_kv_head, int D);
AttnTcPlan attn_tc_plan(int B, int Hq, int Hkv, int T, int Lmax, int D, int sm_count);

// Queue the split-KV kernel.  With a single split (p.n_pre == 1) or p.fused it
// writes out [B*Hq*T][D] and lse (may be NULL) itself; otherwise per-(row,
// split) partials in the layout the combine kernel of attention.cu reads
// ([B*Hq*T][n_pre+1][D+4] floats).  kc, vc: the contiguous caches, or the
// pools when pg.table is set (Lmax = pg.max_blocks * pg.bs then).
spec_status attn_tc_run(const AttnTcPlan& p, const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc,
                        const int32_t* prefix_len, const __nv_bfloat16* kt, const __nv_bfloat16* vt,
                        const spec_tree* tree, int B, int Hq, int Hkv, int Lmax, float scale, float* part, float* out,
                        float* lse, void* ws, cudaStream_t s, const KvPages& pg = KvPages{});

}  // namespace tc
}  // namespace spec
