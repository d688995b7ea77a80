// hydra_draft: Medusa / Hydra draft heads filling the candidate tree.
//
// Medusa Heads (ultralytics glossary), "So sagen die Köpfe voraus": one
// feed-forward layer with SiLU and a residual, then a vocabulary projection.
// Hydra Guide, "1. Embedding Conditioning Mechanics" and "Candidate Tree
// Construction": later heads also read the base embedding of the parent's
// token, and every node's children are the top-k of the head run on it.
//
// One head (depth k+1):
//   gather   u_in rows = [h_b || E[tok(u)]] (or h_b) for every parent row
//   mlp      z = h_b + SiLU(W1 u_in + b1), rounded to the input dtype
//   proj     logits = W2 z and, per row and vocabulary slice, the slice's
//            top-k and (max, sum exp); the tensor-core path takes these
//            straight from its accumulators (logits never reach memory), the
//            CUDA-core path (fp32) stores the logits and scans them
//   select   merge the partials of each row, write the children's tokens,
//            logits and cumulative log-probabilities.
// Rows are (sequence, parent node) pairs; a Medusa head (cond = 0) has one row
// per sequence, shared by every parent of that depth.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "draft_tc.cuh"

namespace spec {
namespace draft {

// ---------------------------------------------------------------- gather

template <typename T>
__global__ void k_gather(const T* __restrict__ h, const T* __restrict__ emb, const int32_t* __restrict__ node_tok,
                         const int32_t* __restrict__ internal, int int_off, int n_int, int Tn, int d, int cond,
                         int R, int d_in_pad, T* __restrict__ xin) {
    const int r = blockIdx.x;
    if (r >= R) return;
    const int b = cond ? r / n_int : r;
    const int u = cond ? internal[int_off + r % n_int] : 0;
    const int vec = 16 / sizeof(T);
    const uint4* hs = reinterpret_cast<const uint4*>(h + static_cast<size_t>(b) * d);
    uint4* dst = reinterpret_cast<uint4*>(xin + static_cast<size_t>(r) * d_in_pad);
    for (int i = threadIdx.x; i < d / vec; i += blockDim.x) dst[i] = hs[i];
    if (cond) {
        const int tok = node_tok[static_cast<size_t>(b) * Tn + u];
        const uint4* es = reinterpret_cast<const uint4*>(emb + static_cast<size_t>(tok) * d);
        for (int i = threadIdx.x; i < d / vec; i += blockDim.x) dst[d / vec + i] = es[i];
    }
}

// ---------------------------------------------------------------- CUDA-core GEMM (fp32 path, small shapes)
//
// acc[n][m] = sum_k W[m][k] * X[n][k]; W [M, K], X [N, K] row-major.
// 64 (m) x 32 (n) tile per CTA, 256 threads, 4 x 2 outputs per thread.

constexpr int GBM = 64, GBN = 32, GBK = 32;

template <typename T, int EPI>
__global__ void __launch_bounds__(256) k_gemm_fma(const T* __restrict__ W, const T* __restrict__ X, int M, int N, int K,
                                                   int ldx, const T* __restrict__ bias, const T* __restrict__ h,
                                                   int cond, int n_int, T* __restrict__ z_out, float* __restrict__ logits) {
    __shared__ float Ws[GBK][GBM + 4];
    __shared__ float Xs[GBK][GBN + 4];
    const int t = threadIdx.x;
    const int m0 = blockIdx.x * GBM, n0 = blockIdx.y * GBN;
    const int tx = t % 16, ty = t / 16;
    float acc[4][2] = {};
    for (int k0 = 0; k0 < K; k0 += GBK) {
#pragma unroll
        for (int i = 0; i < (GBM * GBK) / 256; ++i) {
            const int idx = t + i * 256;
            const int ml = idx / GBK, kl = idx % GBK;
            const int m = m0 + ml, k = k0 + kl;
            Ws[kl][ml] = (m < M && k < K) ? to_f32(W[static_cast<size_t>(m) * K + k]) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < (GBN * GBK) / 256; ++i) {
            const int idx = t + i * 256;
            const int nl = idx / GBK, kl = idx % GBK;
            const int n = n0 + nl, k = k0 + kl;
            Xs[kl][nl] = (n < N && k < K) ? to_f32(X[static_cast<size_t>(n) * ldx + k]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < GBK; ++kk) {
            float a[4], b[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = Ws[kk][tx * 4 + i];
#pragma unroll
            for (int j = 0; j < 2; ++j) b[j] = Xs[kk][ty * 2 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int m = m0 + tx * 4 + i, n = n0 + ty * 2 + j;
            if (m >= M || n >= N) continue;
            if (EPI == 0) {
                const int b = cond ? n / n_int : n;
                const float a = acc[i][j] + (bias ? to_f32(bias[m]) : 0.f);
                const float zz = to_f32(h[static_cast<size_t>(b) * M + m]) + a / (1.0f + expf(-a));
                z_out[static_cast<size_t>(n) * M + m] = from_f32<T>(zz);
            } else {
                logits[static_cast<size_t>(n) * M + m] = acc[i][j];
            }
        }
    }
}

// ---------------------------------------------------------------- top-k over logits rows (fp32 path)

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) { return va > vb || (va == vb && ia < ib); }

// Insert (v, i) into a descending list of length k (registers, fully unrolled).
template <int KMAX>
__device__ __forceinline__ void insert_topk(float (&lv)[KMAX], int (&li)[KMAX], int k, float v, int i) {
    if (!better(v, i, lv[k - 1], li[k - 1])) return;
#pragma unroll
    for (int s = KMAX - 1; s > 0; --s) {
        if (s < k && better(v, i, lv[s - 1], li[s - 1])) { lv[s] = lv[s - 1]; li[s] = li[s - 1]; }
        else if (s < k && better(v, i, lv[s], li[s])) { lv[s] = v; li[s] = i; }
    }
    if (better(v, i, lv[0], li[0])) { lv[0] = v; li[0] = i; }
}

// Per (row, vocab slice): the slice's top-k and (max, sum exp) -> partials.
// Used by the fp32 path on stored logits; the tensor-core path produces the
// same partials from its accumulators.
template <int KMAX>
__global__ void __launch_bounds__(256) k_topk_slices(const float* __restrict__ logits, int V, int k, int slice,
                                                     Cand* __restrict__ part_c, float2* __restrict__ part_l, int nslices) {
    const int r = blockIdx.y, sl = blockIdx.x;
    const int v0 = sl * slice, v1 = min(V, v0 + slice);
    const float* row = logits + static_cast<size_t>(r) * V;
    float lv[KMAX];
    int li[KMAX];
#pragma unroll
    for (int s = 0; s < KMAX; ++s) { lv[s] = -INFINITY; li[s] = 0x7fffffff; }
    float m = -INFINITY, ssum = 0.f;
    for (int x = v0 + threadIdx.x; x < v1; x += blockDim.x) {
        const float v = row[x];
        insert_topk<KMAX>(lv, li, k, v, x);
        if (v > m) { ssum = ssum * expf(m - v) + 1.f; m = v; }
        else ssum += expf(v - m);
    }
    __shared__ Cand sc[256 * KMAX];
    __shared__ float2 sl2[256];
    for (int s = 0; s < k; ++s) sc[threadIdx.x * KMAX + s] = Cand{lv[s], li[s]};
    sl2[threadIdx.x] = make_float2(m, ssum);
    __syncthreads();
    if (threadIdx.x == 0) {
        float M = -INFINITY, S = 0.f;
        for (int t = 0; t < blockDim.x; ++t) lse_merge(M, S, sl2[t].x, sl2[t].y);
        part_l[static_cast<size_t>(r) * nslices + sl] = make_float2(M, S);
    }
    // k rounds of "best head of the per-thread sorted lists"
    __shared__ int head[256];
    head[threadIdx.x] = 0;
    __syncthreads();
    for (int s = 0; s < k; ++s) {
        __shared__ float bv[8];
        __shared__ int bi[8], bt[8];
        const int hd = head[threadIdx.x];
        float v = hd < k ? sc[threadIdx.x * KMAX + hd].v : -INFINITY;
        int i = hd < k ? sc[threadIdx.x * KMAX + hd].i : 0x7fffffff;
        int tt = threadIdx.x;
        for (int o = 16; o > 0; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
            const int t2 = __shfl_xor_sync(0xffffffffu, tt, o);
            if (better(v2, i2, v, i)) { v = v2; i = i2; tt = t2; }
        }
        if ((threadIdx.x & 31) == 0) { bv[threadIdx.x >> 5] = v; bi[threadIdx.x >> 5] = i; bt[threadIdx.x >> 5] = tt; }
        __syncthreads();
        if (threadIdx.x == 0) {
            float v0b = bv[0];
            int i0b = bi[0], t0b = bt[0];
            for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
                if (better(bv[w], bi[w], v0b, i0b)) { v0b = bv[w]; i0b = bi[w]; t0b = bt[w]; }
            part_c[(static_cast<size_t>(r) * nslices + sl) * KMAX + s] = Cand{v0b, i0b};
            head[t0b] += 1;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- select: merge slices, fill children

template <int KMAX>
__global__ void __launch_bounds__(256) k_select(const Cand* __restrict__ part_c, const float2* __restrict__ part_l,
                                                int nslices, int k, int cond, int n_int, int int_off,
                                                const int32_t* __restrict__ internal, const int32_t* __restrict__ child_off,
                                                const int32_t* __restrict__ child_idx, const int32_t* __restrict__ rank,
                                                int Tn, int V, int32_t* __restrict__ node_tok, float* __restrict__ node_logit,
                                                float* __restrict__ node_logprob, void* ws) {
    const int r = blockIdx.x;
    __shared__ float topv[KMAX];
    __shared__ int topi[KMAX];
    __shared__ float lse_s;
    // (max, sum) over slices
    {
        float M = -INFINITY, S = 0.f;
        for (int s = threadIdx.x; s < nslices; s += blockDim.x) {
            const float2 p = part_l[static_cast<size_t>(r) * nslices + s];
            lse_merge(M, S, p.x, p.y);
        }
        __shared__ float2 red[256];
        red[threadIdx.x] = make_float2(M, S);
        __syncthreads();
        if (threadIdx.x == 0) {
            float MM = -INFINITY, SS = 0.f;
            for (int t = 0; t < blockDim.x; ++t) lse_merge(MM, SS, red[t].x, red[t].y);
            lse_s = MM + logf(SS);
        }
    }
    // top-k over nslices sorted lists of length k: k rounds of a block arg-best over list heads
    __shared__ int head[1024];
    for (int s = threadIdx.x; s < nslices; s += blockDim.x) head[s] = 0;
    __syncthreads();
    for (int round = 0; round < k; ++round) {
        float v = -INFINITY;
        int i = 0x7fffffff, who = -1;
        for (int s = threadIdx.x; s < nslices; s += blockDim.x) {
            const int hd = head[s];
            if (hd >= k) continue;
            const Cand c = part_c[(static_cast<size_t>(r) * nslices + s) * KMAX + hd];
            if (who < 0 || better(c.v, c.i, v, i)) { v = c.v; i = c.i; who = s; }
        }
        for (int o = 16; o > 0; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
            const int w2 = __shfl_xor_sync(0xffffffffu, who, o);
            if (w2 >= 0 && (who < 0 || better(v2, i2, v, i))) { v = v2; i = i2; who = w2; }
        }
        __shared__ float bv[8];
        __shared__ int bi[8], bw[8];
        if ((threadIdx.x & 31) == 0) { bv[threadIdx.x >> 5] = v; bi[threadIdx.x >> 5] = i; bw[threadIdx.x >> 5] = who; }
        __syncthreads();
        if (threadIdx.x == 0) {
            float vb = bv[0];
            int ib = bi[0], wb = bw[0];
            for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
                if (bw[w] >= 0 && (wb < 0 || better(bv[w], bi[w], vb, ib))) { vb = bv[w]; ib = bi[w]; wb = bw[w]; }
            // fewer than k finite logits (NaN/inf weights) leave placeholders: keep tokens in range
            if (ib < 0 || ib >= V) { flag_status(ws, SPEC_EINVAL); ib = 0; }
            topv[round] = vb;
            topi[round] = ib;
            if (wb >= 0) head[wb] += 1;
        }
        __syncthreads();
    }
    // children of this row's parent node(s)
    const int b = cond ? r / n_int : r;
    const int j0 = cond ? r % n_int : 0, j1 = cond ? j0 + 1 : n_int;
    for (int j = j0; j < j1; ++j) {
        const int u = internal[int_off + j];
        const float base = node_logprob ? node_logprob[static_cast<size_t>(b) * Tn + u] : 0.f;
        for (int a = child_off[u] + threadIdx.x; a < child_off[u + 1]; a += blockDim.x) {
            const int c = child_idx[a];
            const int rr = rank[c];
            node_tok[static_cast<size_t>(b) * Tn + c] = topi[rr];
            node_logit[static_cast<size_t>(b) * Tn + c] = topv[rr];
            if (node_logprob) node_logprob[static_cast<size_t>(b) * Tn + c] = base + (topv[rr] - lse_s);
        }
    }
}

// Node 0 of every sequence: its token is the root token (clamped to the
// vocabulary, with SPEC_EINVAL in the status word, so later reads stay in bounds).
__global__ void k_init_root(const int32_t* __restrict__ root_tok, int B, int Tn, int V, int32_t* __restrict__ node_tok,
                            float* __restrict__ node_logit, float* __restrict__ node_logprob, void* ws) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int tok = root_tok[b];
    if (tok < 0 || tok >= V) {
        flag_status(ws, SPEC_EINVAL);
        tok = min(max(tok, 0), V - 1);
    }
    node_tok[static_cast<size_t>(b) * Tn] = tok;
    node_logit[static_cast<size_t>(b) * Tn] = 0.f;
    if (node_logprob) node_logprob[static_cast<size_t>(b) * Tn] = 0.f;
}

// ---------------------------------------------------------------- planning

struct Plan {
    int K;
    int max_rows;        // largest row count over heads
    int d_in_max;        // largest u_in width
    int kmax;            // largest top-k
    int nslices_fma;     // vocab slices for the fp32 path
    int slice_fma;
    size_t off_xin, off_z, off_logits, off_pc, off_pl, total;
    bool tc;             // bf16 tensor-core path
    tc::DraftTcPlan tcp;
};

inline int rows_of(const spec_tree* t, int k, int cond, int B) {
    return cond ? B * t->n_internal_at_depth[k] : B;
}

Plan make_plan(const spec_tree* t, int B, int d, int V, int K, const int32_t* cond, const int32_t* topk, spec_dtype dt) {
    Plan p{};
    p.K = K;
    for (int k = 0; k < K; ++k) {
        if (t->n_internal_at_depth[k] == 0) continue;
        p.max_rows = std::max(p.max_rows, rows_of(t, k, cond[k], B));
        p.d_in_max = std::max(p.d_in_max, d * (cond[k] ? 2 : 1));
        p.kmax = std::max(p.kmax, topk[k]);
    }
    p.kmax = p.kmax <= 8 ? 8 : 16;
    p.tc = (dt == SPEC_BF16) && tc::draft_tc_supported(d, V);
    size_t off = kWsHeader;
    auto take = [&](size_t bytes) { size_t at = off; off = round_up(off + bytes, 256); return at; };
    const size_t es = dt == SPEC_BF16 ? 2 : 4;
    if (p.tc) {
        p.tcp = tc::draft_tc_plan(p.max_rows, d, p.d_in_max, V, p.kmax);
        p.off_xin = take(es * static_cast<size_t>(p.tcp.rows_pad) * p.d_in_max);
        p.off_z = take(es * static_cast<size_t>(p.tcp.rows_pad) * d);
        p.off_logits = take(p.tcp.mlp_partial_bytes);
        p.off_pc = take(sizeof(Cand) * static_cast<size_t>(p.tcp.rows_pad) * p.tcp.nslices * p.kmax);
        p.off_pl = take(sizeof(float2) * static_cast<size_t>(p.tcp.rows_pad) * p.tcp.nslices);
    } else {
        // at most 1024 slices per row (the select kernel keeps one list head per slice)
        p.slice_fma = std::max(4096, static_cast<int>(round_up((V + 1023) / 1024, 256)));
        p.nslices_fma = (V + p.slice_fma - 1) / p.slice_fma;
        p.off_xin = take(es * static_cast<size_t>(p.max_rows) * p.d_in_max);
        p.off_z = take(es * static_cast<size_t>(p.max_rows) * d);
        p.off_logits = take(sizeof(float) * static_cast<size_t>(p.max_rows) * V);
        p.off_pc = take(sizeof(Cand) * static_cast<size_t>(p.max_rows) * p.nslices_fma * p.kmax);
        p.off_pl = take(sizeof(float2) * static_cast<size_t>(p.max_rows) * p.nslices_fma);
    }
    p.total = off;
    return p;
}

spec_status check_args(const spec_tree* t, int B, int d, int V, int K, const int32_t* cond, const int32_t* topk, spec_dtype dt) {
    spec_status st = check_tree(t);
    if (st != SPEC_OK) return st;
    if (dt != SPEC_F32 && dt != SPEC_BF16) return fail(SPEC_EINVAL, "dtype %d unknown", (int)dt);
    if (B < 1 || B > (1 << 16)) return fail(SPEC_EINVAL, "B = %d out of range", B);
    if (d < 8 || d > 16384 || d % 8) return fail(SPEC_EINVAL, "d = %d must be a multiple of 8 in 8..16384", d);
    if (V < 2 || V > (1 << 24)) return fail(SPEC_EINVAL, "V = %d out of 2..2^24", V);
    if (K < 1 || K > SPEC_MAX_DEPTH) return fail(SPEC_EINVAL, "K = %d out of 1..%d", K, SPEC_MAX_DEPTH);
    if (K < t->max_depth) return fail(SPEC_EINVAL, "K = %d heads for a tree of depth %d", K, t->max_depth);
    if (!cond || !topk) return fail(SPEC_EINVAL, "cond and topk must not be NULL");
    for (int k = 0; k < K; ++k) {
        if (cond[k] != 0 && cond[k] != 1) return fail(SPEC_EINVAL, "cond[%d] = %d must be 0 or 1", k, cond[k]);
        if (topk[k] < 1 || topk[k] > SPEC_MAX_TOPK || topk[k] > V)
            return fail(SPEC_EINVAL, "topk[%d] = %d out of 1..min(%d, V)", k, topk[k], SPEC_MAX_TOPK);
        if (k + 1 <= t->max_depth && t->max_rank_at_depth[k + 1] >= topk[k])
            return fail(SPEC_EINVAL, "a depth-%d node has rank %d >= topk[%d] = %d", k + 1, t->max_rank_at_depth[k + 1], k, topk[k]);
        if (static_cast<int64_t>(rows_of(t, k, cond[k], B)) > (1 << 20))
            return fail(SPEC_EINVAL, "head %d has too many rows", k);
    }
    return SPEC_OK;
}

template <typename T>
spec_status run(const T* h, const T* emb, int K, const void* const* W1, const void* const* b1, const void* const* W2,
                const int32_t* cond, const int32_t* topk, const int32_t* root_tok, const spec_tree* t, int B, int d,
                int V, int32_t* node_tok, float* node_logit, float* node_logprob, void* ws, const Plan& p,
                cudaStream_t s) {
    unsigned char* w = static_cast<unsigned char*>(ws);
    T* xin = reinterpret_cast<T*>(w + p.off_xin);
    T* z = reinterpret_cast<T*>(w + p.off_z);
    float* logits = reinterpret_cast<float*>(w + p.off_logits);
    Cand* pc = reinterpret_cast<Cand*>(w + p.off_pc);
    float2* pl = reinterpret_cast<float2*>(w + p.off_pl);
    SPEC_CUDA_TRY(reset_device_status(ws, s));
    SPEC_CUDA_TRY(launch("draft_init_root", k_init_root, dim3((B + 127) / 128), dim3(128), 0, s, root_tok, B, t->T, V,
                         node_tok, node_logit, node_logprob, ws));
    for (int k = 0; k < K; ++k) {
        const int n_int = t->n_internal_at_depth[k];
        if (n_int == 0) continue;   // no node of depth k has children: nothing to draft at depth k+1
        int int_off = 0;
        for (int j = 0; j < k; ++j) int_off += t->n_internal_at_depth[j];
        const int R = rows_of(t, k, cond[k], B);
        const int d_in = d * (cond[k] ? 2 : 1);
        const T* W1k = static_cast<const T*>(W1[k]);
        const T* b1k = b1 ? static_cast<const T*>(b1[k]) : nullptr;
        const T* W2k = static_cast<const T*>(W2[k]);
        const int d_in_pad = p.tc ? p.d_in_max : d_in;
        SPEC_CUDA_TRY(launch("draft_gather", k_gather<T>, dim3(R), dim3(128), 0, s, h, emb, node_tok, t->internal,
                             int_off, n_int, t->T, d, cond[k], R, d_in_pad, xin));
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            if (p.tc) {
                spec_status st = tc::draft_head_tc(p.tcp, W1k, b1k, W2k, h, xin, d_in, d_in_pad, z, R, d, V, cond[k],
                                                   n_int, topk[k], p.kmax, logits, pc, pl, ws, s);
                if (st != SPEC_OK) return st;
                if (p.kmax == 8)
                    SPEC_CUDA_TRY(launch("draft_select", k_select<8>, dim3(R), dim3(256), 0, s, pc, pl, p.tcp.nslices, topk[k],
                                         cond[k], n_int, int_off, t->internal, t->child_off, t->child_idx, t->rank,
                                         t->T, V, node_tok, node_logit, node_logprob, ws));
                else
                    SPEC_CUDA_TRY(launch("draft_select", k_select<16>, dim3(R), dim3(256), 0, s, pc, pl, p.tcp.nslices, topk[k],
                                         cond[k], n_int, int_off, t->internal, t->child_off, t->child_idx, t->rank,
                                         t->T, V, node_tok, node_logit, node_logprob, ws));
                continue;
            }
        }
        SPEC_CUDA_TRY(launch("draft_mlp_fma", k_gemm_fma<T, 0>, dim3((d + GBM - 1) / GBM, (R + GBN - 1) / GBN), dim3(256), 0, s,
                             W1k, xin, d, R, d_in, d_in_pad, b1k, h, cond[k], n_int, z, nullptr));
        SPEC_CUDA_TRY(launch("draft_proj_fma", k_gemm_fma<T, 1>, dim3((V + GBM - 1) / GBM, (R + GBN - 1) / GBN), dim3(256), 0, s,
                             W2k, z, V, R, d, d, nullptr, nullptr, 0, 1, nullptr, logits));
        if (p.kmax == 8) {
            SPEC_CUDA_TRY(launch("draft_topk_slices", k_topk_slices<8>, dim3(p.nslices_fma, R), dim3(256), 0, s, logits, V,
                                 topk[k], p.slice_fma, pc, pl, p.nslices_fma));
            SPEC_CUDA_TRY(launch("draft_select", k_select<8>, dim3(R), dim3(256), 0, s, pc, pl, p.nslices_fma, topk[k], cond[k],
                                 n_int, int_off, t->internal, t->child_off, t->child_idx, t->rank, t->T, V, node_tok,
                                 node_logit, node_logprob, ws));
        } else {
            SPEC_CUDA_TRY(launch("draft_topk_slices", k_topk_slices<16>, dim3(p.nslices_fma, R), dim3(256), 0, s, logits, V,
                                 topk[k], p.slice_fma, pc, pl, p.nslices_fma));
            SPEC_CUDA_TRY(launch("draft_select", k_select<16>, dim3(R), dim3(256), 0, s, pc, pl, p.nslices_fma, topk[k], cond[k],
                                 n_int, int_off, t->internal, t->child_off, t->child_idx, t->rank, t->T, V, node_tok,
                                 node_logit, node_logprob, ws));
        }
    }
    return SPEC_OK;
}

}  // namespace draft
}  // namespace spec

using namespace spec;

extern "C" size_t hydra_draft_workspace_size(const spec_tree* tree, int32_t B, int32_t d, int32_t V, int32_t K,
                                             const int32_t* cond, const int32_t* topk, spec_dtype dt) {
    clear_error();
    if (draft::check_args(tree, B, d, V, K, cond, topk, dt) != SPEC_OK) return 0;
    return draft::make_plan(tree, B, d, V, K, cond, topk, dt).total;
}

extern "C" spec_status hydra_draft(const void* h, const void* emb, int32_t K, const void* const* W1,
                                   const void* const* b1, const void* const* W2, const int32_t* cond,
                                   const int32_t* topk, const int32_t* root_tok, const spec_tree* tree, int32_t B,
                                   int32_t d, int32_t V, spec_dtype dt, int32_t* node_tok, float* node_logit,
                                   float* node_logprob, void* ws, size_t ws_bytes, spec_stream_t s_) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(s_);
    clear_error();
    spec_status st = draft::check_args(tree, B, d, V, K, cond, topk, dt);
    if (st != SPEC_OK) return st;
    if (!h || !emb || !W1 || !W2 || !root_tok || !node_tok || !node_logit)
        return fail(SPEC_EINVAL, "h, emb, W1, W2, root_tok, node_tok and node_logit must not be NULL");
    if (!aligned16(h) || !aligned16(emb)) return fail(SPEC_EALIGN, "h and emb must be 16-byte aligned");
    if (!aligned4(root_tok) || !aligned4(node_tok) || !aligned4(node_logit) || (node_logprob && !aligned4(node_logprob)))
        return fail(SPEC_EALIGN, "token and logit buffers must be 4-byte aligned");
    for (int k = 0; k < K; ++k) {
        if (!W1[k] || !W2[k]) return fail(SPEC_EINVAL, "W1[%d] and W2[%d] must not be NULL", k, k);
        if (!aligned16(W1[k]) || !aligned16(W2[k]) || (b1 && b1[k] && !aligned16(b1[k])))
            return fail(SPEC_EALIGN, "head %d weights must be 16-byte aligned", k);
    }
    const draft::Plan p = draft::make_plan(tree, B, d, V, K, cond, topk, dt);
    if (!ws || ws_bytes < p.total) return fail(SPEC_EWORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, p.total);
    if (!aligned16(ws)) return fail(SPEC_EALIGN, "workspace must be 16-byte aligned");
    if (dt == SPEC_BF16)
        return draft::run<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(h), static_cast<const __nv_bfloat16*>(emb), K,
                                         W1, b1, W2, cond, topk, root_tok, tree, B, d, V, node_tok, node_logit,
                                         node_logprob, ws, p, s);
    return draft::run<float>(static_cast<const float*>(h), static_cast<const float*>(emb), K, W1, b1, W2, cond, topk,
                             root_tok, tree, B, d, V, node_tok, node_logit, node_logprob, ws, p, s);
}
