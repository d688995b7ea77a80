// Tensor-core (tcgen05) path of the draft heads, bf16 weights.
//
// Both GEMMs of a head are "skinny": a few to a few hundred activation rows
// against a weight matrix streamed once from HBM.  They run swap-AB: weight
// rows fill the MMA's M = 128 side, activation rows its N side (padded to 16),
// so one CTA owns a 128-row weight tile and TMEM holds its 128 x N fp32 result.
//
// Per CTA: thread 0 issues TMA loads of 128 x 64 weight and N x 64 activation
// tiles (128-byte swizzle) into a ring of shared-memory stages; thread 32
// issues tcgen05.mma (K = 16 per instruction) as stages land and releases each
// stage through tcgen05.commit; after the last stage all four warps read TMEM.
// Every wait is bounded (2 s); on expiry the kernel records SPEC_ETIMEOUT in the
// workspace status word, drains its own loads and frees TMEM.
//
// Epilogues:
//   MLP (W1, split over K): the splits of a weight tile form one thread-block
//       cluster; each keeps its fp32 partial tile in shared memory and the
//       cluster reduces it over distributed shared memory, applying bias,
//       SiLU, the residual h and bf16 rounding.
//   projection (W2): per activation row, the top-k (value desc, token asc)
//       and (max, sum exp) of the tile's 128 logits; logits never reach HBM.
#include <mutex>

#include "draft_tc.cuh"
#include "tc.cuh"

namespace spec {
namespace tc {

constexpr int kBM = 128;        // MMA M: weight rows per CTA
constexpr int kMaxSplits = 8;   // MLP split-K: one cluster (portable size) per weight tile
constexpr int kKB = 2;          // 64-column K blocks per pipeline stage
// Weight loads carry the L2 evict-first policy (streamed once per step) and 256-byte L2 promotion.
constexpr bool kWeightsEvictFirst = true;
// Each CTA starts its K loop at a different stage (by weight tile), so that the CTAs
// do not all read the same activation lines from L2 at the same moment.
constexpr bool kRotateK = true;
constexpr int kBK = 64;         // K per TMA box: one 128-byte swizzled row of bf16
constexpr int kBKS = kBK * kKB; // K per stage
constexpr int kThreads = 128;
constexpr int kStageA = kBM * kBKS * 2;
constexpr int kBoxA = kBM * kBK * 2;      // one K block of the weight tile

struct UmmaParams {
    int M;          // weight rows
    int k_iters;    // K stages per split
    int total_iters;
    int n_pad;      // MMA N
    int n_valid;    // valid activation rows in this launch
    int stages;
    uint32_t tmem_cols;
    // projection epilogue
    int topk;
    int V;
    int nslices;
    int row0;           // first activation row of this launch (output row offset)
    draft::Cand* part_c;
    float2* part_l;
    int kmax;
    void* ws;           // status word (NULL: a timeout goes unrecorded)
    // MLP finish (cluster of a weight tile's splits): y = act(sum + bias) (+ h_b when h is
    // set), written as bf16 to z or, when zf is set, as fp32 to zf
    const __nv_bfloat16* bias;
    const __nv_bfloat16* h;
    __nv_bfloat16* z;
    int cond;
    int n_int;
    // MLP: input columns >= dep_k0 come from the previous kernel; a CTA whose K range
    // lies below it (and is not CTA (0, 0), which always waits so that this kernel
    // completes after the previous one) starts without waiting for it
    int dep_k0;
    int act;            // MLP: 1 SiLU, 0 identity
    // MLP with more activation rows than one MMA N: grid z indexes groups of group_rows
    // rows (0: a single group of n_valid rows); rows_total bounds the last group
    int group_rows;
    int rows_total;
    float* zf;          // MLP: fp32 output instead of z
};

__device__ __forceinline__ bool cbetter(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

template <int EPI, int KMAX>
__global__ void __launch_bounds__(kThreads, 1) k_umma(const __grid_constant__ CUtensorMap tmA,
                                                      const __grid_constant__ CUtensorMap tmB, const UmmaParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stage_b = p.n_pad * kBKS * 2;
    const int box_b = p.n_pad * kBK * 2;
    uint8_t* sA = smem;
    uint8_t* sB = smem + p.stages * kStageA;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + p.stages * stage_b);
    uint64_t* empty = full + p.stages;
    uint64_t* accum = empty + p.stages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kBM;
    const int it0 = blockIdx.y * p.k_iters;
    const int grow0 = p.group_rows ? static_cast<int>(blockIdx.z) * p.group_rows : 0;   // first row of the group
    const int n_valid = p.group_rows ? min(p.group_rows, p.rows_total - grow0) : p.n_valid;
    const int row0 = p.row0 + grow0;
    // stage i of this CTA covers K stage it0 + (i + rot) mod n_it
    const int rot = kRotateK ? static_cast<int>(blockIdx.x % max(1, min(p.k_iters, p.total_iters - it0))) : 0;
    const int n_it = max(0, min(p.k_iters, p.total_iters - it0));

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 0) tmem_alloc(tmem_slot, p.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // The next kernel on the stream may start launching now: it only reads its
    // own weights until its griddep_wait().
    griddep_launch();

    int issued = 0;   // producer: stages loaded
    if (warp == 0) {
        if (lane == 0) {
            // Weight tiles do not depend on the previous kernel: fill the ring first,
            // then wait for the previous kernel's results before loading activations.
            // Weights are read once per call: evict-first in L2.
            const uint64_t wpol = kWeightsEvictFirst ? l2_policy_evict_first() : 0;
            auto load_w = [&](void* dst, uint64_t* bar, int x) {
                if constexpr (kWeightsEvictFirst) tma_load_2d_hint(dst, &tmA, bar, x, m0, wpol);
                else tma_load_2d(dst, &tmA, bar, x, m0);
            };
            const int pre = min(n_it, p.stages);
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full[i], kStageA + stage_b);
                for (int kb = 0; kb < kKB; ++kb)
                    load_w(sA + i * kStageA + kb * kBoxA, &full[i], (it0 + (i + rot) % n_it) * kBKS + kb * kBK);
            }
            const bool independent = EPI == 0 && (it0 + n_it) * kBKS <= p.dep_k0 && (blockIdx.x | blockIdx.y) != 0;
            if (!independent) griddep_wait();
            for (int i = 0; i < pre; ++i)
                for (int kb = 0; kb < kKB; ++kb)
                    tma_load_2d(sB + i * stage_b + kb * box_b, &tmB, &full[i], (it0 + (i + rot) % n_it) * kBKS + kb * kBK, grow0);
            issued = pre;
            for (int i = pre; i < n_it; ++i) {
                const int s = i % p.stages;
                if (!mbar_wait(&empty[s], ((i / p.stages) - 1) & 1)) {
                    if (p.ws) flag_status(p.ws, SPEC_ETIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&full[s], kStageA + stage_b);
                const int kx = (it0 + (i + rot) % n_it) * kBKS;
                for (int kb = 0; kb < kKB; ++kb) {
                    load_w(sA + s * kStageA + kb * kBoxA, &full[s], kx + kb * kBK);
                    tma_load_2d(sB + s * stage_b + kb * box_b, &tmB, &full[s], kx + kb * kBK, grow0);
                }
                issued = i + 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kBM, p.n_pad);
            for (int i = 0; i < n_it; ++i) {
                const int s = i % p.stages;
                if (!mbar_wait(&full[s], (i / p.stages) & 1)) {
                    if (p.ws) flag_status(p.ws, SPEC_ETIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(sA + s * kStageA), b0 = smem_u32(sB + s * stage_b);
#pragma unroll
                for (int kb = 0; kb < kKB; ++kb)
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16(tmem, sdesc_k128(a0 + kb * kBoxA + kk * 32), sdesc_k128(b0 + kb * box_b + kk * 32),
                                 idesc, (i > 0 || kb > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&empty[s]);
            }
            mma_commit(accum);
        }
        __syncwarp();
    }

    const bool have = mbar_wait(accum, 0);
    if (!have && p.ws) flag_status(p.ws, SPEC_ETIMEOUT);
    tc_fence_after();
    const int all_have = __syncthreads_and(have ? 1 : 0);   // one decision for the whole CTA
    const bool run_epi = all_have && !*abort_flag && n_it > 0;

    if (EPI == 0) {
        // Split-K reduction inside the cluster of this weight tile's splits (cluster rank
        // = split): each CTA puts its fp32 partial tile [n][128 weight rows] in its own
        // shared memory (the stage buffers are free), then CTA q reduces activation rows
        // n = q, q + splits, ... over the cluster's shared memory and writes
        // z = h + SiLU(sum + b1) in bf16.  Every CTA reaches both cluster barriers, also
        // after a timeout; a CTA whose accumulator is not valid clears its flag and no
        // row is written.
        float* red = reinterpret_cast<float*>(smem);
        int* ok_flag = reinterpret_cast<int*>(red + n_valid * kBM);
        if (run_epi) {
            for (int c0 = 0; c0 < p.n_pad; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c0 + j < n_valid) red[(c0 + j) * kBM + threadIdx.x] = __uint_as_float(r[j]);
            }
        }
        if (threadIdx.x == 0) *ok_flag = run_epi ? 1 : 0;
        cluster_sync();
        const int nsplit = static_cast<int>(gridDim.y);
        const uint32_t rank = cluster_ctarank();
        bool all_ok = true;
        for (int sp = 0; sp < nsplit; ++sp) all_ok &= dsmem_ld_s32(dsmem_map(smem_u32(ok_flag), sp)) != 0;
        const int m = m0 + threadIdx.x;
        if (all_ok && m < p.M) {
            const float bias = p.bias ? __bfloat162float(p.bias[m]) : 0.f;
            for (int n = static_cast<int>(rank); n < n_valid; n += nsplit) {
                const uint32_t a = smem_u32(red + n * kBM + threadIdx.x);
                float v[kMaxSplits];
#pragma unroll
                for (int sp = 0; sp < kMaxSplits; ++sp) v[sp] = sp < nsplit ? dsmem_ld_f32(dsmem_map(a, sp)) : 0.f;
                float x = bias;
#pragma unroll
                for (int sp = 0; sp < kMaxSplits; ++sp) x += v[sp];
                const int row = row0 + n;
                const int b = p.cond ? row / p.n_int : row;
                const float y = p.act ? x / (1.0f + expf(-x)) : x;
                const float zz = p.h ? __bfloat162float(p.h[static_cast<size_t>(b) * p.M + m]) + y : y;
                if (p.zf) p.zf[static_cast<size_t>(row) * p.M + m] = zz;
                else p.z[static_cast<size_t>(row) * p.M + m] = __float2bfloat16_rn(zz);
            }
        }
        cluster_sync();   // the peers have read this CTA's partials
    }
    if (run_epi && EPI == 1) {
        // stage buffers are free now: reuse them for the transposed tile
        float* tile = reinterpret_cast<float*>(smem);                      // [32 columns][4 quarters][33]
        const int j = threadIdx.x >> 2, q = threadIdx.x & 3;               // column j, rows 32q .. 32q+31
        const int k = p.topk;
        for (int c0 = 0; c0 < p.n_pad; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, r);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) tile[jj * 132 + warp * 33 + lane] = __uint_as_float(r[jj]);
            __syncthreads();
            const int n = c0 + j;
            const int v0 = m0 + 32 * q;   // first vocabulary row of this thread's quarter
            // the 4 threads of a column are adjacent lanes and take every branch below together:
            // their shuffles use the group's own mask
            const unsigned gmask = 0xFu << (lane & ~3);
            if (n < n_valid) {
                float xs[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) xs[i] = v0 + i < p.V ? tile[j * 132 + q * 33 + i] : -INFINITY;
                // quarter (max, sum of exp), merged over the column's 4 threads
                float mq[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mq[e] = fmaxf(fmaxf(xs[e], xs[e + 8]), fmaxf(xs[e + 16], xs[e + 24]));
                float mx = fmaxf(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])), fmaxf(fmaxf(mq[4], mq[5]), fmaxf(mq[6], mq[7])));
                const float mref = mx == -INFINITY ? 0.f : mx;
                float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 32; ++i) ps[i & 3] += expf(xs[i] - mref);
                float sm = (ps[0] + ps[1]) + (ps[2] + ps[3]);
#pragma unroll
                for (int o = 1; o <= 2; o <<= 1) {
                    const float m2 = __shfl_xor_sync(gmask, mx, o, 4);
                    const float s2 = __shfl_xor_sync(gmask, sm, o, 4);
                    const float M = fmaxf(mx, m2);
                    if (M != -INFINITY) sm = sm * expf(mx - M) + s2 * expf(m2 - M);
                    mx = M;
                }
                const size_t out = static_cast<size_t>(row0 + n) * p.nslices + blockIdx.x;
                if (q == 0) p.part_l[out] = make_float2(mx, mx == -INFINITY ? 0.f : sm);
                // top-k by tournament: k rounds of (tree argmax over the thread's 32 logits,
                // then over the 4 threads), the winner knocked out; lower index wins ties.
                // NaN never wins; a round whose best is -inf ends the list (the slots left
                // keep the (-inf, INT_MAX) placeholder).
#pragma unroll
                for (int i = 0; i < 32; ++i) xs[i] = xs[i] == xs[i] ? xs[i] : -INFINITY;
                int rr = 0;
#pragma unroll 1
                for (; rr < k; ++rr) {
                    float tv[16];
                    int ti[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const bool right = xs[2 * e + 1] > xs[2 * e];
                        tv[e] = right ? xs[2 * e + 1] : xs[2 * e];
                        ti[e] = right ? 2 * e + 1 : 2 * e;
                    }
#pragma unroll
                    for (int w2 = 8; w2 > 0; w2 >>= 1)
#pragma unroll
                        for (int e = 0; e < w2; ++e) {
                            const bool right = tv[2 * e + 1] > tv[2 * e];
                            tv[e] = right ? tv[2 * e + 1] : tv[2 * e];
                            ti[e] = right ? ti[2 * e + 1] : ti[2 * e];
                        }
                    float bv = tv[0];
                    int bi = bv == -INFINITY ? 0x7fffffff : v0 + ti[0];
#pragma unroll
                    for (int o = 1; o <= 2; o <<= 1) {
                        const float v2 = __shfl_xor_sync(gmask, bv, o, 4);
                        const int i2 = __shfl_xor_sync(gmask, bi, o, 4);
                        if (cbetter(v2, i2, bv, bi)) { bv = v2; bi = i2; }
                    }
                    if (bv == -INFINITY) break;   // uniform over the 4-lane group
                    if (q == 0) p.part_c[out * p.kmax + rr] = draft::Cand{bv, bi};
#pragma unroll
                    for (int i = 0; i < 32; ++i) xs[i] = v0 + i == bi ? -INFINITY : xs[i];
                }
                if (q == 0)
                    for (; rr < k; ++rr) p.part_c[out * p.kmax + rr] = draft::Cand{-INFINITY, 0x7fffffff};
            }
            __syncthreads();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        // a wait ran out: let this CTA's own loads land before the shared memory is released
        for (int i = max(0, issued - p.stages); i < issued; ++i)
            mbar_wait(&full[i % p.stages], (i / p.stages) & 1, 100000000ull);
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

// ---------------------------------------------------------------- host

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int n_pad_of(int rows) { return std::max(16, static_cast<int>(round_up(rows, 16))); }

uint32_t tmem_cols_of(int n_pad) {
    uint32_t c = 32;
    while (c < static_cast<uint32_t>(n_pad)) c <<= 1;
    return c;
}

int stages_of(int n_pad) {
    const int per = kStageA + n_pad * kBKS * 2;
    // as many stages as keep two CTAs per SM (228 KB per SM, 1 KB reserved per CTA; the
    // fixed part: alignment slack, barriers, flags)
    const int fixed = 1024 + 17 * 8 + 16;
    return std::max(2, std::min(8, (233472 / 2 - 1024 - fixed) / per));
}

size_t smem_of(int n_pad, int stages) {
    return 1024 + static_cast<size_t>(stages) * (kStageA + n_pad * kBKS * 2) + (2 * stages + 1) * 8 + 16;
}

constexpr int kMaxN = 256;

}  // namespace

cudaError_t make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                              uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The merge kernel keeps one list head per 128-token slice, at most 1024 slices.
bool draft_tc_supported(int d, int V) {
    return d >= 8 && d % 8 == 0 && V >= 1 && (V + kBM - 1) / kBM <= 1024 && encode_fn() != nullptr;
}

// Split-K factor of the MLP: as many splits as fit in one wave of resident
// CTAs (`resident` per SM), so no CTA waits for a second wave.
static int mlp_splits(int d, int d_in, int resident) {
    const int m_tiles = (d + kBM - 1) / kBM;
    const int total = (d_in + kBKS - 1) / kBKS;
    const int want = std::min(kMaxSplits, std::max(1, resident * device_sm_count() / m_tiles));
    const int per = (total + want - 1) / want;
    return (total + per - 1) / per;
}

DraftTcPlan draft_tc_plan(int rows, int d, int V) {
    DraftTcPlan p;
    p.rows_pad = n_pad_of(rows);
    p.nslices = (V + kBM - 1) / kBM;
    (void)d;
    return p;
}

template <int EPI, int KMAX>
static spec_status launch_umma(const CUtensorMap& ta, const CUtensorMap& tb, dim3 grid, const UmmaParams& p,
                               cudaStream_t s, const char* name) {
    const size_t smem = smem_of(p.n_pad, p.stages);
    SPEC_CUDA_TRY(cudaFuncSetAttribute(k_umma<EPI, KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    if (EPI == 0)   // the splits of one weight tile (grid.y of them) share a cluster
        SPEC_CUDA_TRY(launch_cluster(name, k_umma<EPI, KMAX>, grid, dim3(kThreads), smem, s, true, dim3(1, grid.y, 1),
                                     ta, tb, p));
    else
        SPEC_CUDA_TRY(launch_ex(name, k_umma<EPI, KMAX>, grid, dim3(kThreads), smem, s, true, ta, tb, p));
    return SPEC_OK;
}

spec_status mlp_tc(const __nv_bfloat16* W, const __nv_bfloat16* bias, int M, const __nv_bfloat16* X, int d_in, int ldx,
                   int R, int cond, int n_int, int dep_k0, int act, const __nv_bfloat16* residual, __nv_bfloat16* z,
                   float* zf, void* ws, cudaStream_t s, int ldw) {
    if (ldw == 0) ldw = d_in;
    const int total_mlp = (d_in + kBKS - 1) / kBKS;
    // activation rows in groups of at most 256 (the MMA's largest N): one launch with a
    // grid z of groups (at most 65535 per launch), the last group partial
    const int n_pad = n_pad_of(std::min(kMaxN, R));
    // CTAs per SM by shared memory (228 KB per SM, 1 KB reserved per CTA); at most 2
    const int resident = static_cast<int>(std::max<size_t>(
        1, std::min<size_t>(2, 233472 / (smem_of(n_pad, stages_of(n_pad)) + 1024))));
    // split K only while the weight tiles of one row group leave SMs idle: with many groups
    // (a table over the whole vocabulary) the groups fill the GPU, unsplit
    const int64_t tiles_groups = static_cast<int64_t>((M + kBM - 1) / kBM) * ((R + kMaxN - 1) / kMaxN);
    const int splits = tiles_groups >= static_cast<int64_t>(resident) * device_sm_count() ? 1 : mlp_splits(M, d_in, resident);
    const int per_split = (total_mlp + splits - 1) / splits;
    const int64_t rows_per_launch = static_cast<int64_t>(kMaxN) * 65535;
    for (int64_t g0 = 0; g0 < R; g0 += rows_per_launch) {
        const int rows = static_cast<int>(std::min<int64_t>(rows_per_launch, R - g0));
        const int groups = (rows + kMaxN - 1) / kMaxN;
        CUtensorMap ta, tb;
        SPEC_CUDA_TRY(make_tmap_bf16_2d(&ta, W, M, d_in, ldw, kBM));
        SPEC_CUDA_TRY(make_tmap_bf16_2d(&tb, X + static_cast<size_t>(g0) * ldx, rows, d_in, ldx, n_pad));
        UmmaParams p{};
        p.M = M;
        p.k_iters = per_split;
        p.total_iters = total_mlp;
        p.n_pad = n_pad;
        p.n_valid = std::min(kMaxN, rows);
        p.group_rows = groups > 1 ? kMaxN : 0;
        p.rows_total = rows;
        p.stages = stages_of(n_pad);
        p.tmem_cols = tmem_cols_of(n_pad);
        p.ws = ws;
        p.row0 = static_cast<int>(g0);
        p.bias = bias;
        p.h = residual;
        p.z = z;
        p.zf = zf;
        p.act = act;
        p.cond = cond;
        p.n_int = n_int;
        p.dep_k0 = dep_k0;
        spec_status st =
            launch_umma<0, 8>(ta, tb, dim3((M + kBM - 1) / kBM, splits, groups), p, s, "draft_mlp_tc");
        if (st != SPEC_OK) return st;
    }
    return SPEC_OK;
}

spec_status proj_tc(const DraftTcPlan& plan, const __nv_bfloat16* W2, const __nv_bfloat16* z, int R, int d, int V, int k,
                    int kmax, draft::Cand* pc, float2* pl, void* ws, cudaStream_t s) {
    for (int g0 = 0; g0 < R; g0 += kMaxN) {
        const int rows = std::min(kMaxN, R - g0);
        const int n_pad = n_pad_of(rows);
        CUtensorMap ta, tb;
        SPEC_CUDA_TRY(make_tmap_bf16_2d(&ta, W2, V, d, d, kBM));
        SPEC_CUDA_TRY(make_tmap_bf16_2d(&tb, z + static_cast<size_t>(g0) * d, rows, d, d, n_pad));
        UmmaParams p{};
        p.M = V;
        p.total_iters = (d + kBKS - 1) / kBKS;
        p.k_iters = p.total_iters;
        p.n_pad = n_pad;
        p.n_valid = rows;
        p.stages = stages_of(n_pad);
        p.tmem_cols = tmem_cols_of(n_pad);
        p.topk = k;
        p.V = V;
        p.nslices = plan.nslices;
        p.row0 = g0;
        p.part_c = pc;
        p.part_l = pl;
        p.kmax = kmax;
        p.ws = ws;
        const dim3 grid(plan.nslices, 1);
        spec_status st = kmax == 8 ? launch_umma<1, 8>(ta, tb, grid, p, s, "draft_proj_tc")
                                   : launch_umma<1, 16>(ta, tb, grid, p, s, "draft_proj_tc");
        if (st != SPEC_OK) return st;
    }
    return SPEC_OK;
}

spec_status draft_head_tc(const DraftTcPlan& plan, const __nv_bfloat16* W1, const __nv_bfloat16* b1,
                          const __nv_bfloat16* W2, const __nv_bfloat16* h, const __nv_bfloat16* X, int d_in, int ldx,
                          __nv_bfloat16* z, int R, int d, int V, int cond, int n_int, int k, int kmax, int dep_k0,
                          draft::Cand* pc, float2* pl, void* ws, cudaStream_t s) {
    spec_status st = mlp_tc(W1, b1, d, X, d_in, ldx, R, cond, n_int, dep_k0, 1, h, z, nullptr, ws, s);
    if (st != SPEC_OK) return st;
    return proj_tc(plan, W2, z, R, d, V, k, kmax, pc, pl, ws, s);
}

}  // namespace tc
}  // namespace spec
