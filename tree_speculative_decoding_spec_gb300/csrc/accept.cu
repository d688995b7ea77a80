// tree_accept: longest accepted path over the candidate tree, and the extra token.
//
// Greedy -- Hydra Guide, "Parallel Verification and Greedy Acceptance
// Algorithm": follow the target's argmax down the tree while a child carries
// it; emit the argmax at the node where the walk stops.
// Rejection -- Speculative Decoding (thegustafson.com), "The acceptance
// criterion", "The correctness guarantee", "A worked example": accept the edge
// into c with token x iff u_c < p(x)/q(x); at the deepest accepted node draw
// the extra token from norm(max(p - q, 0)) if the node has children (all of
// them rejected), else from p (the bonus token).
//
// Two launches per call:
//   rows   grid (vocab slices x B*T rows), one pass over each logits row slice:
//          greedy: the slice's best and second-best values (argmax, ties to the
//          lower id); rejection: (max, sum exp) of logits/temperature for p and,
//          on rows of nodes with children, for q.
//   walk   one CTA per sequence: merge the slices, decide every edge, resolve
//          accepted(c) = accepted(parent) && pass(c) depth by depth, pick the
//          deepest accepted node (lowest index on ties) and, for rejection,
//          draw the extra token by inverse CDF over the vocabulary.
#include <algorithm>

#include "common.cuh"
#include "philox.cuh"

namespace spec {
namespace accept {

constexpr int kRowThreads = 256;
constexpr int kWalkThreads = 1024;
constexpr int kLseIter = 16;   // 4-wide loads per thread and operand: a slice holds <= 256*4*16 tokens
constexpr int kWalkCacheMax = 40960;   // vocabularies up to this size keep the draw's weights in shared memory

struct Plan {
    int slices, slice;
    size_t off_part, total;
};

Plan make_plan(const spec_tree* t, int B, int V) {
    Plan p{};
    const int64_t rows = static_cast<int64_t>(B) * t->T;
    const int64_t target = 2ll * device_sm_count();
    const int max_slices = std::max(1, V / 2048);
    p.slices = static_cast<int>(std::min<int64_t>(std::max<int64_t>((target + rows - 1) / rows, 1), max_slices));
    // the rejection row kernel keeps a thread's values in registers: <= 16384 tokens per slice
    p.slices = std::max(p.slices, (V + kRowThreads * 4 * kLseIter - 1) / (kRowThreads * 4 * kLseIter));
    p.slice = static_cast<int>(round_up((V + p.slices - 1) / p.slices, 4));
    p.slices = (V + p.slice - 1) / p.slice;
    p.off_part = kWsHeader;
    p.total = kWsHeader + round_up(sizeof(float4) * static_cast<size_t>(rows) * p.slices, 256);
    return p;
}

// ---------------------------------------------------------------- rows (greedy)

// better = larger value, then lower index
__device__ __forceinline__ void top2_push(float& v1, int& i1, float& v2, float v, int i) {
    if (v > v1 || (v == v1 && i < i1)) { v2 = v1; v1 = v; i1 = i; }
    else if (v > v2) { v2 = v; }
}
__device__ __forceinline__ void top2_merge(float& v1, int& i1, float& v2, float w1, int j1, float w2) {
    if (w1 > v1 || (w1 == v1 && j1 < i1)) { v2 = fmaxf(v1, w2); v1 = w1; i1 = j1; }
    else { v2 = fmaxf(v2, w1); }
}

// Loads in batches of kGreedyBatch float4 per thread: with 16 in flight the kernel held
// 102 registers, two CTAs per SM, and the 320-CTA grid of the Vicuna-7B shape ran a
// second wave of 16 CTAs (a second HBM round trip).
constexpr int kGreedyBatch = 8;

__global__ void __launch_bounds__(kRowThreads, 3) k_rows_greedy(const float* __restrict__ logits, int V, int slice,
                                                             int slices, float4* __restrict__ part, void* ws) {
    griddep_wait();   // launched early behind the previous kernel: its outputs are complete from here
    clear_status_then_trigger(ws);   // the walk may start loading the tree while the rows are read
    const int sl = blockIdx.x;
    const size_t row = blockIdx.y;
    const float* x = logits + row * V;
    const int v0 = sl * slice, v1 = min(V, v0 + slice);
    float b1 = -INFINITY, b2 = -INFINITY;
    int i1 = 0x7fffffff;
    if ((V & 3) == 0) {
        // each batch of the thread's loads is issued before any compare of it
        for (int it0 = 0; v0 + 4 * kRowThreads * it0 < v1; it0 += kGreedyBatch) {
            float4 q[kGreedyBatch];
#pragma unroll
            for (int it = 0; it < kGreedyBatch; ++it) {
                const int e = v0 + 4 * (static_cast<int>(threadIdx.x) + kRowThreads * (it0 + it));
                q[it] = e < v1 ? __ldcs(reinterpret_cast<const float4*>(x + e))
                               : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
#pragma unroll
            for (int it = 0; it < kGreedyBatch; ++it) {
                const int e = v0 + 4 * (static_cast<int>(threadIdx.x) + kRowThreads * (it0 + it));
                if (e < v1) {
                    top2_push(b1, i1, b2, q[it].x, e);
                    top2_push(b1, i1, b2, q[it].y, e + 1);
                    top2_push(b1, i1, b2, q[it].z, e + 2);
                    top2_push(b1, i1, b2, q[it].w, e + 3);
                }
            }
        }
    } else {
        for (int e = v0 + threadIdx.x; e < v1; e += kRowThreads) top2_push(b1, i1, b2, x[e], e);
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float w1 = __shfl_xor_sync(0xffffffffu, b1, o);
        const int j1 = __shfl_xor_sync(0xffffffffu, i1, o);
        const float w2 = __shfl_xor_sync(0xffffffffu, b2, o);
        top2_merge(b1, i1, b2, w1, j1, w2);
    }
    __shared__ float4 red[kRowThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float4(b1, __int_as_float(i1), b2, 0.f);
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kRowThreads / 32; ++w) top2_merge(b1, i1, b2, red[w].x, __float_as_int(red[w].y), red[w].z);
        part[row * slices + sl] = make_float4(b1, __int_as_float(i1), b2, 0.f);
    }
}

// ---------------------------------------------------------------- rows (rejection)

// exp(y) for y <= 0 as 2^(y log2 e) on the special-function unit: each element of a row
// sum costs one FFMA and one ex2 (the scale and the shift folded into the FFMA); ex2 of
// -inf is 0.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// This thread's share of [v0, v1) of one logits row, raw, in registers (-inf past v1): one
// HBM pass, every load issued before any use.
__device__ __forceinline__ float thread_load(const float* __restrict__ row, int v0, int v1, bool vec4,
                                             float (&x)[4 * kLseIter]) {
    float m = -INFINITY;
    if (vec4) {
#pragma unroll
        for (int it = 0; it < kLseIter; ++it) {
            const int e = v0 + 4 * (static_cast<int>(threadIdx.x) + kRowThreads * it);
            float4 q = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (e < v1) q = __ldcs(reinterpret_cast<const float4*>(row + e));
            x[4 * it] = q.x; x[4 * it + 1] = q.y; x[4 * it + 2] = q.z; x[4 * it + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int it = 0; it < 4 * kLseIter; ++it) {
            const int e = v0 + static_cast<int>(threadIdx.x) + kRowThreads * it;
            x[it] = e < v1 ? row[e] : -INFINITY;
        }
    }
#pragma unroll
    for (int i = 0; i < 4 * kLseIter; i += 4) m = fmaxf(m, fmaxf(fmaxf(x[i], x[i + 1]), fmaxf(x[i + 2], x[i + 3])));
    return m;   // raw maximum (inv_temp > 0 keeps the order)
}

// (max, sum exp(x - max)) of x = logits * inv_temp over this thread's share of [v0, v1).
__device__ __forceinline__ float2 thread_lse(const float* __restrict__ row, int v0, int v1, float inv_temp, bool vec4) {
    float x[4 * kLseIter];
    const float mraw = thread_load(row, v0, v1, vec4, x);
    if (mraw == -INFINITY) return make_float2(-INFINITY, 0.f);
    const float m = mraw * inv_temp;
    const float c = inv_temp * kLog2e, off = -m * kLog2e;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4 * kLseIter; i += 2) {
        s0 += ex2_approx(fmaf(x[i], c, off));
        s1 += ex2_approx(fmaf(x[i + 1], c, off));
    }
    return make_float2(m, s0 + s1);
}

// (m, s, t) with m the max, s = sum exp(x - m) and t = sum exp(x - m) * x over
// this thread's share: (m + ln s) - t / s is the entropy of softmax(x).
__device__ __forceinline__ float3 thread_lse_ent(const float* __restrict__ row, int v0, int v1, float inv_temp, bool vec4) {
    float x[4 * kLseIter];
    const float mraw = thread_load(row, v0, v1, vec4, x);
    if (mraw == -INFINITY) return make_float3(-INFINITY, 0.f, 0.f);
    const float m = mraw * inv_temp;
    const float c = inv_temp * kLog2e, off = -m * kLog2e;
    float sum = 0.f, t = 0.f;   // t over the raw values, scaled by inv_temp at the end
#pragma unroll
    for (int i = 0; i < 4 * kLseIter; ++i) {
        const float e = ex2_approx(fmaf(x[i], c, off));
        sum += e;
        t = x[i] == -INFINITY ? t : fmaf(e, x[i], t);
    }
    return make_float3(m, sum, t * inv_temp);
}

// Merge (m2, s2, t2) into (m, s, t): s and t are both scaled to the larger maximum.
__device__ __forceinline__ void lse_ent_merge(float& m, float& s, float& t, float m2, float s2, float t2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) { m = m2; s = s2; t = t2; return; }
    if (m2 > m) {
        const float a = expf(m - m2);
        s = s * a + s2;
        t = t * a + t2;
        m = m2;
    } else {
        const float a = expf(m2 - m);
        s += s2 * a;
        t += t2 * a;
    }
}

// Typical acceptance: (m, s, t) of every row of logits_p (for entropy and log-sum-exp).
__global__ void __launch_bounds__(kRowThreads) k_rows_ent(const float* __restrict__ lp, int V, int slice, int slices,
                                                          float inv_temp, float4* __restrict__ part, void* ws) {
    griddep_wait();   // launched early behind the previous kernel: its outputs are complete from here
    clear_status_then_trigger(ws);   // the walk may start loading the tree while the rows are read
    const int sl = blockIdx.x;
    const size_t row = blockIdx.y;
    const int v0 = sl * slice, v1 = min(V, v0 + slice);
    const float3 P = thread_lse_ent(lp + row * V, v0, v1, inv_temp, (V & 3) == 0);
    float m = P.x, sm = P.y, t = P.z;
    for (int o = 16; o > 0; o >>= 1)
        lse_ent_merge(m, sm, t, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, sm, o),
                      __shfl_xor_sync(0xffffffffu, t, o));
    __shared__ float4 red[kRowThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float4(m, sm, t, 0.f);
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kRowThreads / 32; ++w) lse_ent_merge(m, sm, t, red[w].x, red[w].y, red[w].z);
        part[row * slices + sl] = make_float4(m, sm, t, 0.f);
    }
}

__global__ void __launch_bounds__(kRowThreads) k_rows_lse(const float* __restrict__ lp, const float* __restrict__ lq,
                                                          const int32_t* __restrict__ child_off, int Tn, int V,
                                                          int slice, int slices, float inv_temp,
                                                          float4* __restrict__ part, void* ws) {
    griddep_wait();   // launched early behind the previous kernel: its outputs are complete from here
    clear_status_then_trigger(ws);   // the walk may start loading the tree while the rows are read
    const int sl = blockIdx.x;
    const size_t row = blockIdx.y;
    const int u = static_cast<int>(row % Tn);
    const bool internal = child_off[u + 1] > child_off[u];
    const int v0 = sl * slice, v1 = min(V, v0 + slice);
    const bool vec4 = (V & 3) == 0;
    const float2 P = thread_lse(lp + row * V, v0, v1, inv_temp, vec4);
    float mp = P.x, sp = P.y, mq = -INFINITY, sq = 0.f;
    if (internal) {
        const float2 Q = thread_lse(lq + row * V, v0, v1, inv_temp, vec4);
        mq = Q.x;
        sq = Q.y;
    }
    for (int o = 16; o > 0; o >>= 1) {
        lse_merge(mp, sp, __shfl_xor_sync(0xffffffffu, mp, o), __shfl_xor_sync(0xffffffffu, sp, o));
        lse_merge(mq, sq, __shfl_xor_sync(0xffffffffu, mq, o), __shfl_xor_sync(0xffffffffu, sq, o));
    }
    __shared__ float4 red[kRowThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float4(mp, sp, mq, sq);
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kRowThreads / 32; ++w) {
            lse_merge(mp, sp, red[w].x, red[w].y);
            lse_merge(mq, sq, red[w].z, red[w].w);
        }
        part[row * slices + sl] = make_float4(mp, sp, mq, sq);
    }
}

// ---------------------------------------------------------------- walk helpers

// Block-wide reductions for 1024 threads (32 warps) through shared memory.
__device__ __forceinline__ int block_max_int(int v, int* scratch) {
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    int r = scratch[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = max(r, scratch[w]);
    return r;
}
__device__ __forceinline__ float block_min_f(float v, float* scratch) {
    v = warp_min(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = scratch[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = fminf(r, scratch[w]);
    return r;
}

// accepted(c) = accepted(parent(c)) && pass(c), resolved depth by depth; then the
// deepest accepted node (lowest index on equal depth) and the root-first path.
__device__ int resolve_path(const int32_t* __restrict__ parent, const int32_t* __restrict__ depth, int Tn, int max_depth,
                            unsigned char* acc, const unsigned char* pass, int* iscratch) {
    for (int u = threadIdx.x; u < Tn; u += blockDim.x) acc[u] = (u == 0);
    __syncthreads();
    for (int lev = 1; lev <= max_depth; ++lev) {
        for (int u = threadIdx.x; u < Tn; u += blockDim.x)
            if (depth[u] == lev) acc[u] = acc[parent[u]] && pass[u];
        __syncthreads();
    }
    int key = -1;
    for (int u = threadIdx.x; u < Tn; u += blockDim.x)
        if (acc[u]) key = max(key, depth[u] * 2048 + (2047 - u));
    key = block_max_int(key, iscratch);
    return 2047 - (key % 2048);
}

__device__ void write_path(const int32_t* __restrict__ parent, const int32_t* __restrict__ depth, int ustar, int b,
                           int max_depth, int32_t* __restrict__ accept_len, int32_t* __restrict__ accept_path) {
    if (threadIdx.x != 0) return;
    const int m = depth[ustar];
    accept_len[b] = m;
    int32_t* path = accept_path + static_cast<size_t>(b) * (max_depth + 1);
    for (int k = m + 1; k <= max_depth; ++k) path[k] = -1;
    int u = ustar;
    for (int k = m; k >= 0; --k) { path[k] = u; u = parent[u]; }
}

// ---------------------------------------------------------------- walk (greedy)

__global__ void __launch_bounds__(kWalkThreads) k_walk_greedy(const float4* __restrict__ part, int slices,
                                                              const int32_t* __restrict__ node_tok,
                                                              const int32_t* __restrict__ parent,
                                                              const int32_t* __restrict__ depth, int Tn, int max_depth,
                                                              int32_t* __restrict__ accept_len,
                                                              int32_t* __restrict__ accept_path,
                                                              int32_t* __restrict__ next_token, float* __restrict__ margin) {
    const int b = blockIdx.x;
    // The tree and the node tokens are inputs of the call, complete before the rows
    // kernel started: they are copied to shared memory while that kernel runs.
    __shared__ int32_t s_par[SPEC_MAX_T], s_dep[SPEC_MAX_T], s_tok[SPEC_MAX_T];
    for (int u = threadIdx.x; u < Tn; u += blockDim.x) {
        s_par[u] = parent[u];
        s_dep[u] = depth[u];
        s_tok[u] = node_tok[static_cast<size_t>(b) * Tn + u];
    }
    __syncthreads();
    griddep_wait();   // the rows kernel's partials
    __shared__ int amax[SPEC_MAX_T];
    __shared__ float gap[SPEC_MAX_T];
    __shared__ unsigned char pass[SPEC_MAX_T], acc[SPEC_MAX_T];
    __shared__ int iscr[32];
    __shared__ float fscr[32];
    for (int u = threadIdx.x; u < Tn; u += blockDim.x) {
        const float4* pr = part + (static_cast<size_t>(b) * Tn + u) * slices;
        float v1 = pr[0].x, v2 = pr[0].z;
        int i1 = __float_as_int(pr[0].y);
        for (int s = 1; s < slices; ++s) top2_merge(v1, i1, v2, pr[s].x, __float_as_int(pr[s].y), pr[s].z);
        amax[u] = i1;
        gap[u] = v1 - v2;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < Tn; c += blockDim.x)
        pass[c] = (c > 0) && s_tok[c] == amax[s_par[c]];
    __syncthreads();
    const int ustar = resolve_path(s_par, s_dep, Tn, max_depth, acc, pass, iscr);
    float mg = INFINITY;
    for (int u = threadIdx.x; u < Tn; u += blockDim.x)
        if (acc[u]) mg = fminf(mg, gap[u]);
    mg = block_min_f(mg, fscr);
    write_path(s_par, s_dep, ustar, b, max_depth, accept_len, accept_path);
    if (threadIdx.x == 0) {
        next_token[b] = amax[ustar];
        if (margin) margin[b] = mg;
    }
}

// ---------------------------------------------------------------- walk (rejection)

__global__ void __launch_bounds__(kWalkThreads, 1) k_walk_reject(const float4* __restrict__ part, int slices,
                                                              const float* __restrict__ lp, const float* __restrict__ lq,
                                                              const int32_t* __restrict__ node_tok,
                                                              const int32_t* __restrict__ parent,
                                                              const int32_t* __restrict__ depth,
                                                              const int32_t* __restrict__ child_off, int Tn,
                                                              int max_depth, int V, float inv_temp, uint64_t seed,
                                                              uint64_t offset, int32_t* __restrict__ accept_len,
                                                              int32_t* __restrict__ accept_path,
                                                              int32_t* __restrict__ next_token, float* __restrict__ margin,
                                                              void* ws, int typical, float eps, float alpha) {
    // typical == 0: min(1, p/q) rejection with residual resampling; typical == 1:
    // Medusa typical acceptance (threshold min(eps, alpha exp(-H(p_parent))), extra
    // token from p at the last accepted node).  lse_q holds that threshold then.
    const int b = blockIdx.x;
    // The tree and the node tokens are inputs of the call, complete before the rows kernel
    // started: they are copied to shared memory while that kernel runs.
    __shared__ int32_t s_par[SPEC_MAX_T], s_dep[SPEC_MAX_T], s_tok[SPEC_MAX_T];
    __shared__ unsigned char s_int[SPEC_MAX_T];
    for (int u = threadIdx.x; u < Tn; u += blockDim.x) {
        s_par[u] = parent[u];
        s_dep[u] = depth[u];
        s_tok[u] = node_tok[static_cast<size_t>(b) * Tn + u];
        s_int[u] = child_off[u + 1] > child_off[u];
    }
    griddep_wait();   // the rows kernel's partials (launched early: the launch overlaps it)
    __shared__ float lse_p[SPEC_MAX_T], lse_q[SPEC_MAX_T];
    __shared__ unsigned char pass[SPEC_MAX_T], acc[SPEC_MAX_T];
    __shared__ float dmar[SPEC_MAX_T];
    __shared__ int iscr[32];
    __shared__ float fscr[32];
    for (int u = threadIdx.x; u < Tn; u += blockDim.x) {
        const float4* pr = part + (static_cast<size_t>(b) * Tn + u) * slices;
        if (typical) {
            float m = -INFINITY, sm = 0.f, t = 0.f;
            for (int s = 0; s < slices; ++s) lse_ent_merge(m, sm, t, pr[s].x, pr[s].y, pr[s].z);
            lse_p[u] = m + logf(sm);
            const float H = lse_p[u] - t / sm;   // entropy of p_u (nats)
            lse_q[u] = fminf(eps, alpha * expf(-H));
            continue;
        }
        float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
        for (int s = 0; s < slices; ++s) { lse_merge(mp, sp, pr[s].x, pr[s].y); lse_merge(mq, sq, pr[s].z, pr[s].w); }
        lse_p[u] = mp + logf(sp);
        lse_q[u] = s_int[u] ? mq + logf(sq) : NAN;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < Tn; c += blockDim.x) {
        pass[c] = 0;
        dmar[c] = INFINITY;
        if (c == 0) continue;
        const int par = s_par[c];
        const int x = s_tok[c];
        if (x < 0 || x >= V) {   // a token outside the vocabulary is never accepted
            flag_status(ws, SPEC_EINVAL);
            continue;
        }
        const size_t prow = (static_cast<size_t>(b) * Tn + par) * V;
        const float logp = lp[prow + x] * inv_temp - lse_p[par];
        if (typical) {
            const float pv = expf(logp);
            pass[c] = pv > lse_q[par];
            if (lse_q[par] > 0.f) dmar[c] = fabsf(pv / lse_q[par] - 1.f);   // relative: thresholds can be tiny
            continue;
        }
        const float logq = lq[prow + x] * inv_temp - lse_q[par];
        const float ratio = expf(logp - logq);
        const float u = uniform24(spec_draw(seed, offset, static_cast<uint32_t>(c), static_cast<uint32_t>(b)).w[0]);
        pass[c] = u < ratio;
        if (ratio < 1.f) dmar[c] = fabsf(u - ratio);
    }
    __syncthreads();
    const int ustar = resolve_path(s_par, s_dep, Tn, max_depth, acc, pass, iscr);
    float mg = INFINITY;
    for (int c = threadIdx.x; c < Tn; c += blockDim.x)
        if (c > 0 && acc[s_par[c]]) mg = fminf(mg, dmar[c]);
    mg = block_min_f(mg, fscr);
    write_path(s_par, s_dep, ustar, b, max_depth, accept_len, accept_path);

    // ---- the extra token: inverse CDF over the vocabulary, ascending token order
    const bool leaf = !s_int[ustar];
    const size_t srow = (static_cast<size_t>(b) * Tn + ustar) * V;
    const float lsp = lse_p[ustar], lsq = lse_q[ustar];
    const float* rp = lp + srow;
    const float* rq = typical ? nullptr : lq + srow;
    // weight of token x: p (leaf, or residual all zero) or max(p - q, 0); exp(y) as
    // 2^(y log2 e), the scale and the shift in one FFMA
    const float wc = inv_temp * kLog2e, wop = -lsp * kLog2e, woq = -lsq * kLog2e;
    auto weight = [&](int x, bool resid) -> float {
        const float pv = ex2_approx(fmaf(rp[x], wc, wop));
        if (!resid) return pv;
        return fmaxf(pv - ex2_approx(fmaf(rq[x], wc, woq)), 0.f);
    };
    // The range sums below compute every token's weight once, 16 loads per lane in flight;
    // a vocabulary of at most kWalkCacheMax tokens keeps them in shared memory, where the
    // scans read them (one pass over the two rows instead of a dependent load per 32 tokens)
    extern __shared__ float wcache[];
    const bool cached = V <= kWalkCacheMax;
    auto wt = [&](int x, bool resid) -> float { return cached ? wcache[x] : weight(x, resid); };
    // Draw: warp w owns the contiguous token range [w*Rw, (w+1)*Rw); each warp sums its range
    // with coalesced loads, warp 0 scans the 32 range sums, the warp holding the target
    // scans its range 32 tokens at a time (ascending token order throughout).
    __shared__ float wsum[32], wexcl[32];
    __shared__ float s_total, s_target;
    __shared__ int s_wstar, pick;
    __shared__ float smar;
    const int wid = threadIdx.x >> 5, ln = threadIdx.x & 31;
    const int Rw = ((V + 31) / 32 + 31) / 32 * 32;
    const int w0 = min(V, wid * Rw), w1 = min(V, w0 + Rw);
    bool resid = !leaf && !typical;
    auto range_sum = [&](bool rs) {
        float acc = 0.f;
#pragma unroll 16
        for (int x = w0 + ln; x < w1; x += 32) {
            const float wv = weight(x, rs);
            if (cached) wcache[x] = wv;
            acc += wv;
        }
        return warp_sum(acc);
    };
    float my = range_sum(resid);
    if (ln == 0) wsum[wid] = my;
    __syncthreads();
    if (resid) {
        float tot = 0.f;
        for (int i = 0; i < 32; ++i) tot += wsum[i];
        if (tot == 0.f) {   // alpha = 1: no residual mass, fall back to p
            resid = false;
            __syncthreads();
            my = range_sum(false);
            if (ln == 0) wsum[wid] = my;
            __syncthreads();
        }
    }
    const float u1 = uniform24(spec_draw(seed, offset, 0u, static_cast<uint32_t>(b)).w[1]);
    if (wid == 0) {
        const float v = wsum[ln];
        float inc = v;
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, inc, o);
            if (ln >= o) inc += t;
        }
        wexcl[ln] = inc - v;
        const float total = __shfl_sync(0xffffffffu, inc, 31);
        const float target = u1 * total;
        const unsigned hit = __ballot_sync(0xffffffffu, v > 0.f && v > target - (inc - v));
        if (ln == 0) {
            s_total = total;
            s_target = target;
            s_wstar = hit ? __ffs(hit) - 1 : -1;
        }
    }
    __syncthreads();
    const int wstar = s_wstar;
    if (wstar < 0) {
        // target at or beyond the total (rounding): take the last token of positive weight
        int lastx = -1;
        for (int x = threadIdx.x; x < V; x += blockDim.x)
            if (wt(x, resid) > 0.f) lastx = x;
        lastx = block_max_int(lastx, iscr);
        if (threadIdx.x == 0) {
            pick = max(lastx, 0);
            smar = 0.f;
        }
    } else if (wid == wstar) {
        const float need = s_target - wexcl[wstar];
        float run = 0.f, lo = 0.f, hi = 0.f;
        int found = -1, lastpos = -1;
        for (int base = w0; base < w1; base += 32) {
            const int x = base + ln;
            const float wv = x < w1 ? wt(x, resid) : 0.f;
            float inc = wv;
            for (int o = 1; o < 32; o <<= 1) {
                const float t = __shfl_up_sync(0xffffffffu, inc, o);
                if (ln >= o) inc += t;
            }
            const float cum = run + inc;
            const unsigned hit = __ballot_sync(0xffffffffu, wv > 0.f && cum > need);
            const unsigned pos = __ballot_sync(0xffffffffu, wv > 0.f);
            if (pos) lastpos = base + 31 - __clz(pos);
            if (hit) {
                const int l = __ffs(hit) - 1;
                found = base + l;
                hi = __shfl_sync(0xffffffffu, cum, l);
                lo = hi - __shfl_sync(0xffffffffu, wv, l);
                break;
            }
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (ln == 0) {
            if (found < 0) {   // rounding left the target past this range's last positive token
                pick = lastpos;
                smar = 0.f;
            } else {
                pick = found;
                smar = fminf(hi - need, need - lo) / s_total;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        next_token[b] = pick;
        if (margin) margin[b] = fminf(mg, fabsf(smar));
    }
}

spec_status check_args(int mode, const spec_tree* t, int B, int V, float temperature) {
    spec_status st = check_tree(t);
    if (st != SPEC_OK) return st;
    if (mode < 0 || mode > 2) return fail(SPEC_EINVAL, "mode = %d must be 0 (greedy), 1 (rejection) or 2 (typical)", mode);
    if (B < 1 || B > 65535) return fail(SPEC_EINVAL, "B = %d out of 1..65535", B);
    if (V < 2 || V > (1 << 24)) return fail(SPEC_EINVAL, "V = %d out of 2..2^24", V);
    if (mode >= 1 && !(temperature > 0.f && temperature < 1e30f)) return fail(SPEC_EINVAL, "temperature must be positive");
    if (static_cast<int64_t>(B) * t->T > 65535) return fail(SPEC_EINVAL, "B * T = %lld rows exceed 65535", (long long)B * t->T);
    return SPEC_OK;
}

}  // namespace accept
}  // namespace spec

using namespace spec;

extern "C" size_t tree_accept_workspace_size(int32_t mode, const spec_tree* tree, int32_t B, int32_t V) {
    clear_error();
    if (accept::check_args(mode, tree, B, V, 1.0f) != SPEC_OK) return 0;
    return accept::make_plan(tree, B, V).total;
}

extern "C" spec_status tree_accept(int32_t mode, const float* logits_p, const float* logits_q, const int32_t* node_tok,
                                   const spec_tree* tree, int32_t B, int32_t V, float temperature, uint64_t seed,
                                   uint64_t offset, int32_t* accept_len, int32_t* accept_path, int32_t* next_token,
                                   float* margin, void* ws, size_t ws_bytes, spec_stream_t s_) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(s_);
    clear_error();
    if (mode == 2) return fail(SPEC_EINVAL, "mode 2 (typical acceptance) is tree_accept_typical");
    spec_status st = accept::check_args(mode, tree, B, V, temperature);
    if (st != SPEC_OK) return st;
    if (!logits_p || !node_tok || !accept_len || !accept_path || !next_token)
        return fail(SPEC_EINVAL, "logits_p, node_tok and the outputs must not be NULL");
    if (mode == 1 && !logits_q) return fail(SPEC_EINVAL, "rejection needs logits_q");
    if (!aligned16(logits_p) || (logits_q && !aligned16(logits_q))) return fail(SPEC_EALIGN, "logits must be 16-byte aligned");
    if (!aligned4(node_tok) || !aligned4(accept_len) || !aligned4(accept_path) || !aligned4(next_token) ||
        (margin && !aligned4(margin)))
        return fail(SPEC_EALIGN, "token buffers must be 4-byte aligned");
    const accept::Plan p = accept::make_plan(tree, B, V);
    if (!ws || ws_bytes < p.total) return fail(SPEC_EWORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, p.total);
    if (!aligned16(ws)) return fail(SPEC_EALIGN, "workspace must be 16-byte aligned");
    float4* part = reinterpret_cast<float4*>(static_cast<unsigned char*>(ws) + p.off_part);
    const dim3 grid(p.slices, B * tree->T);
    // the rows kernel clears the status word (it flags nothing itself; the walk flags after its wait)
    if (mode == 0) {
        SPEC_CUDA_TRY(launch_ex("accept_rows_greedy", accept::k_rows_greedy, grid, dim3(accept::kRowThreads), 0, s, true, logits_p, V,
                             p.slice, p.slices, part, ws));
        // one thread per node is enough here (no vocabulary scans): small trees get cheap barriers
        const int walk_threads = std::min(accept::kWalkThreads, std::max(32, (tree->T + 31) / 32 * 32));
        SPEC_CUDA_TRY(launch_ex("accept_walk_greedy", accept::k_walk_greedy, dim3(B), dim3(walk_threads), 0, s, true, part,
                             p.slices, node_tok, tree->parent, tree->depth, tree->T, tree->max_depth, accept_len,
                             accept_path, next_token, margin));
    } else {
        const float inv_temp = 1.0f / temperature;
        SPEC_CUDA_TRY(launch_ex("accept_rows_lse", accept::k_rows_lse, grid, dim3(accept::kRowThreads), 0, s, true, logits_p,
                                logits_q, tree->child_off, tree->T, V, p.slice, p.slices, inv_temp, part, ws));
        const size_t wsmem = V <= accept::kWalkCacheMax ? sizeof(float) * static_cast<size_t>(V) : 0;
        SPEC_CUDA_TRY(cudaFuncSetAttribute(accept::k_walk_reject, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(sizeof(float) * accept::kWalkCacheMax)));
        SPEC_CUDA_TRY(launch_ex("accept_walk_reject", accept::k_walk_reject, dim3(B), dim3(accept::kWalkThreads), wsmem, s, true, part,
                             p.slices, logits_p, logits_q, node_tok, tree->parent, tree->depth, tree->child_off,
                             tree->T, tree->max_depth, V, inv_temp, seed, offset, accept_len, accept_path, next_token,
                             margin, ws, 0, 0.f, 0.f));
    }
    return SPEC_OK;
}

extern "C" spec_status tree_accept_typical(const float* logits_p, const int32_t* node_tok, const spec_tree* tree,
                                           int32_t B, int32_t V, float temperature, float epsilon, float alpha,
                                           uint64_t seed, uint64_t offset, int32_t* accept_len, int32_t* accept_path,
                                           int32_t* next_token, float* margin, void* ws, size_t ws_bytes,
                                           spec_stream_t s_) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(s_);
    clear_error();
    spec_status st = accept::check_args(2, tree, B, V, temperature);
    if (st != SPEC_OK) return st;
    if (!(epsilon >= 0.f && epsilon < 1e30f) || !(alpha >= 0.f && alpha < 1e30f))
        return fail(SPEC_EINVAL, "epsilon and alpha must be finite and >= 0");
    if (!logits_p || !node_tok || !accept_len || !accept_path || !next_token)
        return fail(SPEC_EINVAL, "logits_p, node_tok and the outputs must not be NULL");
    if (!aligned16(logits_p)) return fail(SPEC_EALIGN, "logits must be 16-byte aligned");
    if (!aligned4(node_tok) || !aligned4(accept_len) || !aligned4(accept_path) || !aligned4(next_token) ||
        (margin && !aligned4(margin)))
        return fail(SPEC_EALIGN, "token buffers must be 4-byte aligned");
    const accept::Plan p = accept::make_plan(tree, B, V);
    if (!ws || ws_bytes < p.total) return fail(SPEC_EWORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, p.total);
    if (!aligned16(ws)) return fail(SPEC_EALIGN, "workspace must be 16-byte aligned");
    float4* part = reinterpret_cast<float4*>(static_cast<unsigned char*>(ws) + p.off_part);
    const dim3 grid(p.slices, B * tree->T);
    const float inv_temp = 1.0f / temperature;
    // the rows kernel clears the status word (it flags nothing itself; the walk flags after its wait)
    SPEC_CUDA_TRY(launch_ex("accept_rows_ent", accept::k_rows_ent, grid, dim3(accept::kRowThreads), 0, s, true, logits_p, V,
                         p.slice, p.slices, inv_temp, part, ws));
    const size_t wsmem = V <= accept::kWalkCacheMax ? sizeof(float) * static_cast<size_t>(V) : 0;
    SPEC_CUDA_TRY(cudaFuncSetAttribute(accept::k_walk_reject, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(float) * accept::kWalkCacheMax)));
    SPEC_CUDA_TRY(launch_ex("accept_walk_typical", accept::k_walk_reject, dim3(B), dim3(accept::kWalkThreads), wsmem, s, true, part,
                         p.slices, logits_p, static_cast<const float*>(nullptr), node_tok, tree->parent, tree->depth,
                         tree->child_off, tree->T, tree->max_depth, V, inv_temp, seed, offset, accept_len, accept_path,
                         next_token, margin, ws, 1, epsilon, alpha));
    return SPEC_OK;
}
