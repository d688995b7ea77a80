// tree_attention: the T tree tokens attend over the cached prefix plus their
// own ancestors.
//
// Hydra Guide, "Tree Attention Matrix with Topology-Aware Causal Masking": the
// prefix is always visible; among the tree tokens node i sees exactly anc*(i)
// (itself and its ancestors).  The ancestor sets arrive as one bit row per node
// (spec_tree.anc) and are applied to the scores in registers.
//
// Split-KV layout: the key sequence of one (sequence, KV head) is cut into
// `n_pre` prefix chunks plus one tail chunk holding the T tree keys.  One CTA
// takes a block of query rows (all query heads of the KV group x tree nodes)
// against one chunk with an online softmax and writes (max, sum, unnormalised
// output) to the workspace; a combine kernel merges the chunks of each row.
#include <algorithm>
#include <cmath>

#include "attention_tc.cuh"
#include "common.cuh"

namespace spec {
namespace attn {

constexpr int BR = 64;   // query rows per CTA
constexpr int BC = 64;   // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- CUDA-core split-KV kernel

template <typename T, int D>
__global__ void __launch_bounds__(256) k_attn_fma(const T* __restrict__ q, const T* __restrict__ kc,
                                                  const T* __restrict__ vc, const int32_t* __restrict__ prefix_len,
                                                  const T* __restrict__ kt, const T* __restrict__ vt,
                                                  const uint64_t* __restrict__ anc, int Tn, int words, int Hq, int Hkv,
                                                  int Lmax, float scale_log2, int chunk, int n_pre, int n_rowblocks,
                                                  float* __restrict__ part, const tc::KvPages pg, void* ws) {
    griddep_launch();   // the combine may start launching: it waits for the partials
    constexpr int LD = D + 4;
    constexpr int LP = BC + 4;
    constexpr int DT = D / 16;   // output dims per thread
    extern __shared__ float4 smem4[];
    float* Qs = reinterpret_cast<float*>(smem4);
    float* Ks = Qs + BR * LD;
    float* Vs = Ks + BC * LD;
    float* Ps = Vs + BC * LD;

    const int g = Hq / Hkv;
    const int R = Tn * g;
    const int c = blockIdx.x;
    const int kvh = blockIdx.y / n_rowblocks, rb = blockIdx.y % n_rowblocks;
    const int b = blockIdx.z;
    const int L = min(max(prefix_len[b], 0), Lmax);
    const bool tail = (c == n_pre);
    const int k_begin = tail ? 0 : c * chunk;
    const int k_end = tail ? Tn : min(L, k_begin + chunk);
    if (k_begin >= k_end) return;
    const int t = threadIdx.x;
    const int rg = t >> 4, kg = t & 15;
    const int r0 = rb * BR;

    for (int idx = t; idx < BR * (D / 4); idx += 256) {
        const int rl = idx / (D / 4), c4 = idx % (D / 4);
        const int r = r0 + rl;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (r < R) {
            const int hl = r / Tn, i = r % Tn;
            const int h = kvh * g + hl;
            load4(q + ((static_cast<size_t>(b) * Hq + h) * Tn + i) * D + c4 * 4, v);
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] *= scale_log2;
        }
        *reinterpret_cast<float4*>(&Qs[rl * LD + c4 * 4]) = make_float4(v[0], v[1], v[2], v[3]);
    }
    int node[4];
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) node[ii] = (r0 + 4 * rg + ii) % Tn;

    float m_run[4], l_run[4], o[4][DT];
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
        m_run[ii] = -INFINITY;
        l_run[ii] = 0.f;
#pragma unroll
        for (int e = 0; e < DT; ++e) o[ii][e] = 0.f;
    }
    const size_t kv_off = tail ? (static_cast<size_t>(b) * Hkv + kvh) * Tn * D
                               : (static_cast<size_t>(b) * Hkv + kvh) * static_cast<size_t>(Lmax) * D;
    const T* Kb = (tail ? kt : kc) + kv_off;
    const T* Vb = (tail ? vt : vc) + kv_off;

    for (int j0 = k_begin; j0 < k_end; j0 += BC) {
        __syncthreads();
        for (int idx = t; idx < BC * (D / 4); idx += 256) {
            const int jl = idx / (D / 4), c4 = idx % (D / 4);
            const int j = j0 + jl;
            float kv[4] = {0.f, 0.f, 0.f, 0.f}, vv[4] = {0.f, 0.f, 0.f, 0.f};
            if (j < k_end) {
                if (!tail && pg.table) {   // paged prefix: the key's pool block and row
                    const int blk = pg.table[static_cast<size_t>(b) * pg.max_blocks + j / pg.bs];
                    if (blk >= 0 && blk < pg.num_blocks) {
                        const size_t row = (static_cast<size_t>(blk) * Hkv + kvh) * pg.bs + j % pg.bs;
                        load4(kc + row * D + c4 * 4, kv);
                        load4(vc + row * D + c4 * 4, vv);
                    } else {
                        flag_status(ws, SPEC_EINVAL);   // the key reads as zeros
                    }
                } else {
                    load4(Kb + static_cast<size_t>(j) * D + c4 * 4, kv);
                    load4(Vb + static_cast<size_t>(j) * D + c4 * 4, vv);
                }
            }
            *reinterpret_cast<float4*>(&Ks[jl * LD + c4 * 4]) = make_float4(kv[0], kv[1], kv[2], kv[3]);
            *reinterpret_cast<float4*>(&Vs[jl * LD + c4 * 4]) = make_float4(vv[0], vv[1], vv[2], vv[3]);
        }
        __syncthreads();

        float s[4][4];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) s[ii][jj] = 0.f;
#pragma unroll 4
        for (int dd = 0; dd < D; dd += 4) {
            float4 qa[4], kb[4];
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) qa[ii] = *reinterpret_cast<const float4*>(&Qs[(4 * rg + ii) * LD + dd]);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) kb[jj] = *reinterpret_cast<const float4*>(&Ks[(kg + 16 * jj) * LD + dd]);
#pragma unroll
            for (int ii = 0; ii < 4; ++ii)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    s[ii][jj] += qa[ii].x * kb[jj].x + qa[ii].y * kb[jj].y + qa[ii].z * kb[jj].z + qa[ii].w * kb[jj].w;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int key = j0 + kg + 16 * jj;
            const bool in = key < k_end;
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
                bool ok = in;
                if (tail && ok) ok = (anc[static_cast<size_t>(node[ii]) * words + (key >> 6)] >> (key & 63)) & 1ull;
                if (!ok) s[ii][jj] = -INFINITY;
            }
        }
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
            float mt = fmaxf(fmaxf(s[ii][0], s[ii][1]), fmaxf(s[ii][2], s[ii][3]));
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            const float m_new = fmaxf(m_run[ii], mt);
            float alpha = 1.f, lt = 0.f;
            float p[4];
            if (m_new == -INFINITY) {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) p[jj] = 0.f;
            } else {
                alpha = exp2f(m_run[ii] - m_new);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) { p[jj] = exp2f(s[ii][jj] - m_new); lt += p[jj]; }
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
            l_run[ii] = l_run[ii] * alpha + lt;
            m_run[ii] = m_new;
#pragma unroll
            for (int e = 0; e < DT; ++e) o[ii][e] *= alpha;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) Ps[(4 * rg + ii) * LP + kg + 16 * jj] = p[jj];
        }
        __syncwarp();
#pragma unroll 4
        for (int j = 0; j < BC; ++j) {
            float pj[4];
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) pj[ii] = Ps[(4 * rg + ii) * LP + j];
#pragma unroll
            for (int half = 0; half < DT / 4; ++half) {
                const float4 v = *reinterpret_cast<const float4*>(&Vs[j * LD + half * 64 + kg * 4]);
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    o[ii][half * 4 + 0] += pj[ii] * v.x;
                    o[ii][half * 4 + 1] += pj[ii] * v.y;
                    o[ii][half * 4 + 2] += pj[ii] * v.z;
                    o[ii][half * 4 + 3] += pj[ii] * v.w;
                }
            }
        }
    }
    const int n_chunks = n_pre + 1;
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
        const int r = r0 + 4 * rg + ii;
        if (r >= R) continue;
        const int hl = r / Tn, i = r % Tn;
        const int h = kvh * g + hl;
        const size_t row = (static_cast<size_t>(b) * Hq + h) * Tn + i;
        float* base = part + (row * n_chunks + c) * (D + 4);
        if (kg == 0) { base[0] = m_run[ii]; base[1] = l_run[ii]; }
#pragma unroll
        for (int half = 0; half < DT / 4; ++half)
            *reinterpret_cast<float4*>(&base[4 + half * 64 + kg * 4]) =
                make_float4(o[ii][half * 4 + 0], o[ii][half * 4 + 1], o[ii][half * 4 + 2], o[ii][half * 4 + 3]);
    }
}

// ---------------------------------------------------------------- combine

// One warp per (sequence, query head, node) row, 8 rows per CTA: merge the
// row's split partials (max m_c in base 2, sum l_c, unnormalised O_c):
// O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c, lse = (M + log2 l) ln 2.
// Slots read: the non-empty prefix splits, plus the tree slot n_pre unless the
// tree keys were folded into the last prefix split (tensor-core layout).  The
// partials are taken kCombineGroup at a time, every load of a group (m, l and
// the lane's 4 O values of each partial) issued together, with a running
// maximum across groups: one memory round trip per group.
constexpr int kCombineGroup = 4;

__global__ void __launch_bounds__(256) k_attn_combine(const float* __restrict__ part, const int32_t* __restrict__ prefix_len,
                                                      int Tn, int Hq, int D, int Lmax, int chunk, int n_pre, int folded,
                                                      int nrows, float* __restrict__ out, float* __restrict__ lse) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= nrows) return;
    const int lane = threadIdx.x & 31;
    const int b = row / (Hq * Tn);
    const int L = min(max(prefix_len[b], 0), Lmax);
    const int nvalid = (L + chunk - 1) / chunk;
    const int nread = folded ? max(nvalid, 1) : nvalid + 1;
    const float* base = part + static_cast<size_t>(row) * (n_pre + 1) * (D + 4);
    auto slot = [&](int i) { return (!folded && i == nvalid) ? n_pre : i; };
    griddep_wait();   // the attention kernel's partials (launched early: the launch overlaps it)
    const bool has = 4 * lane < D;
    float M = -INFINITY;
    float l = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < nread; i0 += kCombineGroup) {
        float pm[kCombineGroup], pl[kCombineGroup];
        float4 pv[kCombineGroup];
#pragma unroll
        for (int j = 0; j < kCombineGroup; ++j) {
            pm[j] = -INFINITY;
            pl[j] = 0.f;
            pv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i0 + j < nread) {
                const float* pc = base + static_cast<size_t>(slot(i0 + j)) * (D + 4);
                const float2 ml = *reinterpret_cast<const float2*>(pc);
                pm[j] = ml.x;
                pl[j] = ml.y;
                if (has) pv[j] = *reinterpret_cast<const float4*>(pc + 4 + 4 * lane);
            }
        }
        float gm = pm[0];
#pragma unroll
        for (int j = 1; j < kCombineGroup; ++j) gm = fmaxf(gm, pm[j]);
        const float Mn = fmaxf(M, gm);
        if (Mn == -INFINITY) continue;   // nothing but empty partials so far
        const float sc = M == -INFINITY ? 0.f : exp2f(M - Mn);
        l *= sc;
        o.x *= sc; o.y *= sc; o.z *= sc; o.w *= sc;
#pragma unroll
        for (int j = 0; j < kCombineGroup; ++j) {
            const float w = pm[j] == -INFINITY ? 0.f : exp2f(pm[j] - Mn);
            l += w * pl[j];
            o.x += w * pv[j].x; o.y += w * pv[j].y; o.z += w * pv[j].z; o.w += w * pv[j].w;
        }
        M = Mn;
    }
    if (has) {
        const float inv = 1.f / l;
        *reinterpret_cast<float4*>(out + static_cast<size_t>(row) * D + 4 * lane) =
            make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
    }
    if (lse && lane == 0) lse[row] = (M + log2f(l)) * kLn2;
}

// ---------------------------------------------------------------- planning

struct Plan {
    bool tc;
    int n_rowblocks, chunk, n_pre;
    size_t part_bytes, total;
    tc::AttnTcPlan tcp;
};

Plan make_plan(const spec_tree* t, int B, int Hq, int Hkv, int Lmax, int D, spec_dtype dt) {
    Plan p{};
    const int g = Hq / Hkv;
    const int R = t->T * g;
    p.tc = (dt == SPEC_BF16) && tc::attn_tc_supported(R, D);
    if (p.tc) {
        p.tcp = tc::attn_tc_plan(B, Hq, Hkv, t->T, Lmax, D, device_sm_count());
        p.part_bytes = p.tcp.part_bytes;
    } else {
        p.n_rowblocks = (R + BR - 1) / BR;
        const int64_t base = static_cast<int64_t>(B) * Hkv * p.n_rowblocks;
        const int64_t target = 2ll * device_sm_count();
        const int max_chunks = (Lmax + BC - 1) / BC;
        const int want = static_cast<int>(std::min<int64_t>(std::max<int64_t>((target + base - 1) / base, 1), max_chunks));
        p.chunk = static_cast<int>(round_up((Lmax + want - 1) / want, BC));
        p.n_pre = (Lmax + p.chunk - 1) / p.chunk;
        p.part_bytes = sizeof(float) * static_cast<size_t>(B) * Hq * t->T * (p.n_pre + 1) * (D + 4);
    }
    p.total = kWsHeader + round_up(p.part_bytes, 256);
    return p;
}

spec_status check_args(const spec_tree* t, int B, int Hq, int Hkv, int Lmax, int D, spec_dtype dt) {
    spec_status st = check_tree(t);
    if (st != SPEC_OK) return st;
    if (dt != SPEC_F32 && dt != SPEC_BF16) return fail(SPEC_EINVAL, "dtype %d unknown", (int)dt);
    if (B < 1 || B > 65535) return fail(SPEC_EINVAL, "B = %d out of 1..65535", B);
    if (Hkv < 1 || Hq < Hkv || Hq % Hkv || Hq > 1024) return fail(SPEC_EINVAL, "Hq = %d must be a multiple of Hkv = %d", Hq, Hkv);
    if (D != 64 && D != 128) return fail(SPEC_EUNSUPPORTED, "D = %d: only 64 and 128 are built", D);
    if (Lmax < 1 || Lmax > (1 << 22)) return fail(SPEC_EINVAL, "Lmax = %d out of 1..2^22", Lmax);
    if (static_cast<int64_t>(t->T) * (Hq / Hkv) > 65535ll * BR) return fail(SPEC_EINVAL, "too many query rows per KV head");
    return SPEC_OK;
}

template <typename T>
spec_status run_fma(const T* q, const T* kc, const T* vc, const int32_t* prefix_len, const T* kt, const T* vt,
                    const spec_tree* t, int B, int Hq, int Hkv, int Lmax, int D, float scale, float* out, float* lse,
                    void* ws, const Plan& p, cudaStream_t s, const tc::KvPages& pg) {
    float* part = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + kWsHeader);
    const dim3 grid(p.n_pre + 1, Hkv * p.n_rowblocks, B);
    const float sl2 = scale * kLog2e;
    if (D == 128) {
        const size_t smem = sizeof(float) * (BR * 132 + 2 * BC * 132 + BR * (BC + 4));
        SPEC_CUDA_TRY(cudaFuncSetAttribute(k_attn_fma<T, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        SPEC_CUDA_TRY(launch("attn_fma", k_attn_fma<T, 128>, grid, dim3(256), smem, s, q, kc, vc, prefix_len, kt, vt,
                             t->anc, t->T, t->words, Hq, Hkv, Lmax, sl2, p.chunk, p.n_pre, p.n_rowblocks, part, pg,
                             ws));
    } else {
        const size_t smem = sizeof(float) * (BR * 68 + 2 * BC * 68 + BR * (BC + 4));
        SPEC_CUDA_TRY(cudaFuncSetAttribute(k_attn_fma<T, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        SPEC_CUDA_TRY(launch("attn_fma", k_attn_fma<T, 64>, grid, dim3(256), smem, s, q, kc, vc, prefix_len, kt, vt,
                             t->anc, t->T, t->words, Hq, Hkv, Lmax, sl2, p.chunk, p.n_pre, p.n_rowblocks, part, pg,
                             ws));
    }
    const int nrows = B * Hq * t->T;
    SPEC_CUDA_TRY(launch_ex("attn_combine", k_attn_combine, dim3((nrows + 7) / 8), dim3(256), 0, s, true, part, prefix_len, t->T,
                         Hq, D, Lmax, p.chunk, p.n_pre, 0, nrows, out, lse));
    return SPEC_OK;
}

}  // namespace attn
}  // namespace spec

using namespace spec;

extern "C" size_t tree_attention_workspace_size(const spec_tree* tree, int32_t B, int32_t Hq, int32_t Hkv,
                                                int32_t Lmax, int32_t D, spec_dtype dt) {
    clear_error();
    if (attn::check_args(tree, B, Hq, Hkv, Lmax, D, dt) != SPEC_OK) return 0;
    return attn::make_plan(tree, B, Hq, Hkv, Lmax, D, dt).total;
}

namespace spec {
namespace attn {

// Both entry points: contiguous caches (pg.table == nullptr) or a paged pool.
static spec_status run_checked(const void* q, const void* k_cache, const void* v_cache, const int32_t* prefix_len,
                               const void* k_tree, const void* v_tree, const spec_tree* tree, int32_t B, int32_t Hq,
                               int32_t Hkv, int32_t Lmax, int32_t D, float scale, spec_dtype dt, float* out, float* lse,
                               void* ws, size_t ws_bytes, cudaStream_t s, const tc::KvPages& pg) {
    spec_status st = check_args(tree, B, Hq, Hkv, Lmax, D, dt);
    if (st != SPEC_OK) return st;
    if (!q || !k_cache || !v_cache || !prefix_len || !k_tree || !v_tree || !out)
        return fail(SPEC_EINVAL, "q, caches, prefix_len, tree K/V and out must not be NULL");
    if (scale == 0.f) scale = 1.f / sqrtf(static_cast<float>(D));   // the usual 1/sqrt(D)
    if (!(scale > 0.f) || !(scale < 1e30f)) return fail(SPEC_EINVAL, "scale must be positive and finite, or 0");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_tree) || !aligned16(v_tree) ||
        !aligned16(out) || !aligned4(prefix_len) || (lse && !aligned4(lse)))
        return fail(SPEC_EALIGN, "tensors must be 16-byte aligned (prefix_len and lse 4-byte)");
    const Plan p = make_plan(tree, B, Hq, Hkv, Lmax, D, dt);
    if (!ws || ws_bytes < p.total) return fail(SPEC_EWORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, p.total);
    if (!aligned16(ws)) return fail(SPEC_EALIGN, "workspace must be 16-byte aligned");
    if (dt == SPEC_BF16) {
        using T = __nv_bfloat16;
        SPEC_CUDA_TRY(reset_device_status(ws, s));
        if (p.tc) {
            float* part = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + kWsHeader);
            st = tc::attn_tc_run(p.tcp, static_cast<const T*>(q), static_cast<const T*>(k_cache),
                                 static_cast<const T*>(v_cache), prefix_len, static_cast<const T*>(k_tree),
                                 static_cast<const T*>(v_tree), tree, B, Hq, Hkv, Lmax, scale, part, out, lse, ws, s, pg);
            if (st != SPEC_OK || p.tcp.fused || p.tcp.n_pre == 1) return st;   // merged on chip, or one split
            const int nrows = B * Hq * tree->T;
            SPEC_CUDA_TRY(launch_ex("attn_combine", k_attn_combine, dim3((nrows + 7) / 8), dim3(256), 0, s, true, part,
                                 prefix_len, tree->T, Hq, D, Lmax, p.tcp.chunk, p.tcp.n_pre, 1, nrows, out, lse));
            return SPEC_OK;
        }
        return run_fma<T>(static_cast<const T*>(q), static_cast<const T*>(k_cache), static_cast<const T*>(v_cache),
                          prefix_len, static_cast<const T*>(k_tree), static_cast<const T*>(v_tree), tree, B, Hq, Hkv,
                          Lmax, D, scale, out, lse, ws, p, s, pg);
    }
    SPEC_CUDA_TRY(reset_device_status(ws, s));
    return run_fma<float>(static_cast<const float*>(q), static_cast<const float*>(k_cache),
                          static_cast<const float*>(v_cache), prefix_len, static_cast<const float*>(k_tree),
                          static_cast<const float*>(v_tree), tree, B, Hq, Hkv, Lmax, D, scale, out, lse, ws, p, s, pg);
}

// Paged arguments: block size a multiple of 64, table entries checked on the device.
static spec_status check_pages(int32_t num_blocks, const int32_t* block_table, int32_t max_blocks, int32_t block_size,
                               int32_t Hkv) {
    if (block_size < 64 || block_size % 64 != 0) return fail(SPEC_EINVAL, "block_size = %d: a positive multiple of 64", block_size);
    if (num_blocks < 1 || max_blocks < 1) return fail(SPEC_EINVAL, "num_blocks = %d, max_blocks = %d must be positive", num_blocks, max_blocks);
    if (static_cast<int64_t>(max_blocks) * block_size > (1 << 22))
        return fail(SPEC_EINVAL, "max_blocks * block_size = %lld > 2^22", static_cast<long long>(max_blocks) * block_size);
    if (static_cast<int64_t>(num_blocks) * (Hkv > 0 ? Hkv : 1) * block_size > INT32_MAX)
        return fail(SPEC_EINVAL, "pool of %d blocks too large (num_blocks * Hkv * block_size rows >= 2^31)", num_blocks);
    if (!block_table) return fail(SPEC_EINVAL, "block_table must not be NULL");
    if (!aligned4(block_table)) return fail(SPEC_EALIGN, "block_table must be 4-byte aligned");
    return SPEC_OK;
}

}  // namespace attn
}  // namespace spec

extern "C" spec_status tree_attention(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* prefix_len, const void* k_tree, const void* v_tree,
                                      const spec_tree* tree, int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax,
                                      int32_t D, float scale, spec_dtype dt, float* out, float* lse, void* ws,
                                      size_t ws_bytes, spec_stream_t s_) {
    clear_error();
    return attn::run_checked(q, k_cache, v_cache, prefix_len, k_tree, v_tree, tree, B, Hq, Hkv, Lmax, D, scale, dt, out,
                             lse, ws, ws_bytes, reinterpret_cast<cudaStream_t>(s_), tc::KvPages{});
}

extern "C" size_t tree_attention_paged_workspace_size(const spec_tree* tree, int32_t B, int32_t Hq, int32_t Hkv,
                                                      int32_t max_blocks, int32_t block_size, int32_t D, spec_dtype dt) {
    clear_error();
    if (block_size < 64 || block_size % 64 != 0 || max_blocks < 1 ||
        static_cast<int64_t>(max_blocks) * block_size > (1 << 22))
        return 0;
    return tree_attention_workspace_size(tree, B, Hq, Hkv, max_blocks * block_size, D, dt);
}

extern "C" spec_status tree_attention_paged(const void* q, const void* k_pool, const void* v_pool, int32_t num_blocks,
                                            const int32_t* block_table, int32_t max_blocks, int32_t block_size,
                                            const int32_t* prefix_len, const void* k_tree, const void* v_tree,
                                            const spec_tree* tree, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                            float scale, spec_dtype dt, float* out, float* lse, void* ws,
                                            size_t ws_bytes, spec_stream_t s_) {
    clear_error();
    spec_status st = attn::check_pages(num_blocks, block_table, max_blocks, block_size, Hkv);
    if (st != SPEC_OK) return st;
    tc::KvPages pg;
    pg.table = block_table;
    pg.max_blocks = max_blocks;
    pg.bs = block_size;
    pg.num_blocks = num_blocks;
    return attn::run_checked(q, k_pool, v_pool, prefix_len, k_tree, v_tree, tree, B, Hq, Hkv, max_blocks * block_size, D,
                             scale, dt, out, lse, ws, ws_bytes, reinterpret_cast<cudaStream_t>(s_), pg);
}

// ---------------------------------------------------------------- tree_attention without caller scratch
//
// Some callers cannot allocate device memory: a plugin running inside a host
// engine that has already handed out the device memory and forbids further
// cudaMalloc calls, or a caller whose own interface has no way to carry a
// workspace pointer through.  tree_attention_noalloc serves them with scratch
// held in the file-scope array below instead of a caller-provided workspace.
// The array is part of this library's device image, so every GPU that loads
// the library holds it until the process exits.

namespace spec {
namespace attn {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device (host code sees only a
// host-side stand-in under the array's name).  Looked up on every call rather than
// cached: after a context teardown (cudaDeviceReset) the module reloads and an old
// address would no longer be valid.  The first lookup on a device loads the module.
static spec_status noalloc_scratch(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
        return fail(SPEC_ECUDA, "cudaGetSymbolAddress of the built-in scratch failed: %s", cudaGetErrorString(e));
    *out = p;
    return SPEC_OK;
}

}  // namespace attn
}  // namespace spec

extern "C" spec_status tree_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* prefix_len, const void* k_tree, const void* v_tree,
                                              const spec_tree* tree, int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax,
                                              int32_t D, float scale, spec_dtype dt, float* out, float* lse,
                                              spec_stream_t s) {
    clear_error();
    spec_status st = attn::check_args(tree, B, Hq, Hkv, Lmax, D, dt);
    if (st != SPEC_OK) return st;
    const size_t need = attn::make_plan(tree, B, Hq, Hkv, Lmax, D, dt).total;
    if (need > attn::kNoAllocScratchBytes)
        return fail(SPEC_EWORKSPACE,
                    "tree_attention_noalloc: these shapes need %zu bytes of scratch, more than the %zu-byte built-in "
                    "buffer; call tree_attention with a workspace instead",
                    need, attn::kNoAllocScratchBytes);
    void* ws = nullptr;
    st = attn::noalloc_scratch(&ws);
    if (st != SPEC_OK) return st;
    return tree_attention(q, k_cache, v_cache, prefix_len, k_tree, v_tree, tree, B, Hq, Hkv, Lmax, D, scale, dt, out,
                          lse, ws, attn::kNoAllocScratchBytes, s);
}

// Status word of the built-in scratch: what spec_read_device_status returns for a
// caller workspace, for the calls that use the built-in array instead.
extern "C" spec_status tree_attention_noalloc_status(int32_t* status, spec_stream_t s) {
    clear_error();
    if (!status) return fail(SPEC_EINVAL, "status must not be NULL");
    void* ws = nullptr;
    spec_status st = attn::noalloc_scratch(&ws);
    if (st != SPEC_OK) return st;
    return spec_read_device_status(ws, status, s);
}
