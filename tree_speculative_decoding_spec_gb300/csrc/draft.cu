// hydra_draft: Medusa / Hydra draft heads filling the candidate tree.
//
// Medusa Heads (ultralytics glossary), "So sagen die Köpfe voraus": one
// feed-forward layer with SiLU and a residual, then a vocabulary projection.
// Hydra Guide, "1. Embedding Conditioning Mechanics" and "Candidate Tree
// Construction": later heads also read the base embedding of the parent's
// token, and every node's children are the top-k of the head run on it.
//
// Rows are (sequence, parent node) pairs of one depth; a Medusa head
// (cond = 0) has one row per sequence, shared by every parent of that depth.
// One head (filling depth k+1) on the bf16 path is three launches:
//   mlp      z = h + SiLU(W1 u_in + b1) (tcgen05, split over K; the last split
//            of each weight tile adds bias, SiLU and the residual, rounds to bf16)
//   proj     logits = W2 z (tcgen05); per row and 128-token slice, the slice's
//            top-k and (max, sum exp) straight from TMEM (logits never reach HBM)
//   select   merge the slices of each row, write the children's tokens, logits
//            and cumulative log-probabilities, and the next depth's input rows
//            u_in = [h_b || E[tok(child)]]
// and the launches are chained with programmatic dependent launch, so each
// kernel's weight loads start while the previous kernel drains.  The fp32 path
// (CUDA cores) stores logits and scans them per slice instead of `proj`.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "draft_tc.cuh"

namespace spec {
namespace draft {

// ---------------------------------------------------------------- CUDA-core GEMM (fp32 path, small shapes)
//
// acc[n][m] = sum_k W[m][k] * X[n][k]; W [M, K] (row stride ldw), X [N, K] (row stride ldx).
// 64 (m) x 32 (n) tile per CTA, 256 threads, 4 x 2 outputs per thread.

constexpr int GBM = 64, GBN = 32, GBK = 32;

template <typename T, int EPI>
__global__ void __launch_bounds__(256) k_gemm_fma(const T* __restrict__ W, int ldw, const T* __restrict__ X, int M, int N, int K,
                                                   int ldx, const T* __restrict__ bias, const T* __restrict__ h,
                                                   int cond, int n_int, T* __restrict__ z_out, float* __restrict__ logits,
                                                   int act, float* __restrict__ zf) {
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
            Ws[kl][ml] = (m < M && k < K) ? to_f32(W[static_cast<size_t>(m) * ldw + k]) : 0.f;
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
            if (EPI == 0) {   // act(W x + bias) (+ h_b when h is set), to z_out or, if set, fp32 zf
                const int b = cond ? n / n_int : n;
                const float a = acc[i][j] + (bias ? to_f32(bias[m]) : 0.f);
                const float y = act ? a / (1.0f + expf(-a)) : a;
                const float zz = h ? to_f32(h[static_cast<size_t>(b) * M + m]) + y : y;
                if (zf) zf[static_cast<size_t>(n) * M + m] = zz;
                else z_out[static_cast<size_t>(n) * M + m] = from_f32<T>(zz);
            } else {
                logits[static_cast<size_t>(n) * M + m] = acc[i][j];
            }
        }
    }
}

// The same product for a few activation rows (N <= kGemvRows, N * K floats in
// shared memory): one warp per weight row m, the CTA's rows staged once in
// shared memory as fp32, each lane taking every 32nd k of the row (coalesced
// loads, eight in flight) and a shuffle reduction per activation row.  A
// launch costs about one round trip of loads instead of the tiled kernel's
// K / 32 dependent ones.  Same epilogues and arguments as k_gemm_fma.
constexpr int kGemvRows = 16;
constexpr int kGemvWarps = 8;
constexpr size_t kGemvSmemMax = 48 * 1024;

inline bool gemv_fits(int N, int K) {
    return N >= 1 && N <= kGemvRows && static_cast<size_t>(N) * K * sizeof(float) <= kGemvSmemMax;
}

template <typename T, int EPI>
__global__ void __launch_bounds__(kGemvWarps * 32) k_gemv_rows(const T* __restrict__ W, int ldw, const T* __restrict__ X,
                                                               int M, int N, int K, int ldx, const T* __restrict__ bias,
                                                               const T* __restrict__ h, int cond, int n_int,
                                                               T* __restrict__ z_out, float* __restrict__ logits, int act,
                                                               float* __restrict__ zf) {
    extern __shared__ float xs[];   // [N][K]
    for (int idx = threadIdx.x; idx < N * K; idx += blockDim.x)
        xs[idx] = to_f32(X[static_cast<size_t>(idx / K) * ldx + idx % K]);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int m = blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
    if (m >= M) return;
    const T* wr = W + static_cast<size_t>(m) * ldw;
    float acc[kGemvRows];
#pragma unroll
    for (int n = 0; n < kGemvRows; ++n) acc[n] = 0.f;
#pragma unroll 8
    for (int k = lane; k < K; k += 32) {
        const float wv = to_f32(wr[k]);
#pragma unroll
        for (int n = 0; n < kGemvRows; ++n)
            if (n < N) acc[n] = fmaf(wv, xs[n * K + k], acc[n]);
    }
#pragma unroll
    for (int n = 0; n < kGemvRows; ++n) {
        if (n >= N) break;
        const float sum = warp_sum(acc[n]);
        if (lane != n) continue;
        if (EPI == 0) {   // act(W x + bias) (+ h_b when h is set), to z_out or, if set, fp32 zf
            const int b = cond ? n / n_int : n;
            const float a = sum + (bias ? to_f32(bias[m]) : 0.f);
            const float y = act ? a / (1.0f + expf(-a)) : a;
            const float zz = h ? to_f32(h[static_cast<size_t>(b) * M + m]) + y : y;
            if (zf) zf[static_cast<size_t>(n) * M + m] = zz;
            else z_out[static_cast<size_t>(n) * M + m] = from_f32<T>(zz);
        } else {
            logits[static_cast<size_t>(n) * M + m] = sum;
        }
    }
}

// acc[n][m] = W[m] . X[n] for the fp32 / CUDA-core path: the warp-per-row kernel for a few
// activation rows, the tiled kernel otherwise.
template <typename T, int EPI, typename... Args>
cudaError_t launch_gemm(const char* name, cudaStream_t s, const T* W, int ldw, const T* X, int M, int N, int K, int ldx,
                        Args... rest) {
    if (gemv_fits(N, K))
        return launch(name, k_gemv_rows<T, EPI>, dim3((M + kGemvWarps - 1) / kGemvWarps), dim3(kGemvWarps * 32),
                      static_cast<size_t>(N) * K * sizeof(float), s, W, ldw, X, M, N, K, ldx, rest...);
    return launch(name, k_gemm_fma<T, EPI>, dim3((M + GBM - 1) / GBM, (N + GBN - 1) / GBN), dim3(256), 0, s, W, ldw, X,
                  M, N, K, ldx, rest...);
}

// ---------------------------------------------------------------- LayerNorm (head form 1)

// z[r] = (y[r] - mean) / sqrt(var + eps) * gamma + beta over the d entries of
// row r (mean and biased variance in fp32, the variance from the deviations);
// gamma/beta NULL: 1/0.  One CTA of 256 threads per row: the row is read once
// into registers (kLnVec float4 per thread, d <= 4 * 256 * kLnVec), so the
// kernel costs one load round trip and two block reductions.  Launched as a
// programmatic dependent: y comes from the kernel before it.
constexpr int kLnThreads = 256;
constexpr int kLnVec = 16;
static_assert(4 * kLnThreads * kLnVec >= 16384, "a LayerNorm row of the largest d fits the registers");
template <typename T>
__global__ void __launch_bounds__(kLnThreads) k_layernorm(const float* __restrict__ y, int d, const T* __restrict__ gamma,
                                                          const T* __restrict__ beta, float eps, T* __restrict__ z) {
    __shared__ float red[2][kLnThreads / 32];
    griddep_wait();
    griddep_launch();
    const int n4 = d / 4;
    const float4* yr = reinterpret_cast<const float4*>(y + static_cast<size_t>(blockIdx.x) * d);
    float4 v[kLnVec];
#pragma unroll
    for (int j = 0; j < kLnVec; ++j) {
        const int i = threadIdx.x + j * kLnThreads;
        v[j] = i < n4 ? yr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    auto block_sum = [&](float t, int slot) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if ((threadIdx.x & 31) == 0) red[slot][threadIdx.x >> 5] = t;
        __syncthreads();
        float r = 0.f;
#pragma unroll
        for (int w = 0; w < kLnThreads / 32; ++w) r += red[slot][w];
        return r;
    };
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < kLnVec; ++j) sum += (v[j].x + v[j].y) + (v[j].z + v[j].w);
    const float mean = block_sum(sum, 0) / d;
    float sq = 0.f;
#pragma unroll
    for (int j = 0; j < kLnVec; ++j)
        if (threadIdx.x + j * kLnThreads < n4) {
            const float a = v[j].x - mean, b = v[j].y - mean, c = v[j].z - mean, e = v[j].w - mean;
            sq += (a * a + b * b) + (c * c + e * e);
        }
    const float inv = 1.0f / sqrtf(block_sum(sq, 1) / d + eps);
    T* zr = z + static_cast<size_t>(blockIdx.x) * d;
#pragma unroll
    for (int j = 0; j < kLnVec; ++j) {
        const int i = threadIdx.x + j * kLnThreads;
        if (i < n4) {
            const float x[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float g = gamma ? to_f32(gamma[4 * i + e]) : 1.f;
                const float bb = beta ? to_f32(beta[4 * i + e]) : 0.f;
                zr[4 * i + e] = from_f32<T>((x[e] - mean) * inv * g + bb);
            }
        }
    }
}

// ---------------------------------------------------------------- top-k over logits rows (fp32 path)

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) { return va > vb || (va == vb && ia < ib); }

// Insert (v, i) into a descending list of KMAX candidates (registers, every
// index static); callers keep KMAX >= k and use the first k.
template <int KMAX>
__device__ __forceinline__ void insert_topk(float (&lv)[KMAX], int (&li)[KMAX], float v, int i) {
    if (!better(v, i, lv[KMAX - 1], li[KMAX - 1])) return;
#pragma unroll
    for (int s = KMAX - 1; s > 0; --s) {
        if (better(v, i, lv[s - 1], li[s - 1])) { lv[s] = lv[s - 1]; li[s] = li[s - 1]; }
        else if (better(v, i, lv[s], li[s])) { lv[s] = v; li[s] = i; }
    }
    if (better(v, i, lv[0], li[0])) { lv[0] = v; li[0] = i; }
}

// a and b: best-first lists of N candidates (N a power of two).  Leaves in a
// the best N of both, best-first: the element-wise better of a[e] and
// b[N-1-e] is a bitonic sequence holding exactly those N, which log2(N)
// half-cleaner stages sort.  Every index is static (registers only).
template <int N>
__device__ __forceinline__ void merge_top(float (&av)[N], int (&ai)[N], const float (&bv)[N], const int (&bi)[N]) {
#pragma unroll
    for (int e = 0; e < N; ++e)
        if (better(bv[N - 1 - e], bi[N - 1 - e], av[e], ai[e])) {
            av[e] = bv[N - 1 - e];
            ai[e] = bi[N - 1 - e];
        }
#pragma unroll
    for (int j = N / 2; j > 0; j >>= 1)
#pragma unroll
        for (int e = 0; e < N; ++e)
            if ((e & j) == 0 && better(av[e + j], ai[e + j], av[e], ai[e])) {
                const float tv = av[e];
                const int ti = ai[e];
                av[e] = av[e + j];
                ai[e] = ai[e + j];
                av[e + j] = tv;
                ai[e + j] = ti;
            }
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
        insert_topk<KMAX>(lv, li, v, x);
        if (v > m) { ssum = ssum * expf(m - v) + 1.f; m = v; }
        else ssum += expf(v - m);
    }
    __shared__ Cand sc[256 * KMAX];
    __shared__ float2 sl2[8];
#pragma unroll
    for (int s = 0; s < KMAX; ++s) sc[threadIdx.x * KMAX + s] = Cand{lv[s], li[s]};
    // (max, sum exp) of the slice: a shuffle reduction per warp, then the warps' results
    for (int o = 16; o > 0; o >>= 1) lse_merge(m, ssum, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, ssum, o));
    if ((threadIdx.x & 31) == 0) sl2[threadIdx.x >> 5] = make_float2(m, ssum);
    __syncthreads();
    if (threadIdx.x == 0) {
        float M = -INFINITY, S = 0.f;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) lse_merge(M, S, sl2[w].x, sl2[w].y);
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


// ---------------------------------------------------------------- folded first layer (conditioned heads)
//
// Hydra Guide, "1. Embedding Conditioning Mechanics": a conditioned head's first
// layer reads u = [h_b || E[tok]], so W1 u = W1[:, :d] h_b + W1[:, d:] E[tok].  The
// second term depends on the token alone; hydra_fold_embedding tabulates it once
// per set of weights (tab[v, m] = W1[m, d:] . E[v] in fp32) and a step then streams
// only the h_b half of W1: k_fold_h forms a[b] = W1[:, :d] h_b, and the select that
// picks a child's token writes the child's head input z = h_b + SiLU(a[b] + tab[tok]
// + b1) itself, so the head's MLP leaves the chain between two projections.

// a[b, m] = W1[m, 0:d] . h[b] + b1[m] in fp32, on the warp-level tensor-core MMA
// (m16n8k16, bf16 inputs, fp32 accumulation): weight rows on M, sequences on N
// (eight per pass).  The work is bound by streaming W1, not by the MMA; the MMA
// keeps the instruction count flat in the number of sequences.  A dot product
// does not depend on the order of its k terms, so each lane feeds its fragment
// registers straight from its own 16-byte loads: in a 64-wide block of k, lane
// (g = lane / 4, t = lane % 4) loads k in [8t, 8t + 8) and [32 + 8t, 32 + 8t + 8)
// of weight rows g and g + 8 and of h[b0 + g], and its four MMAs take the 32-bit
// pairs in that order for both operands (the fragment's k slots {2t, 2t+1,
// 2t+8, 2t+9} of a thread always meet the same physical k in A and in B).  A CTA
// covers 16 weight rows; its 16 warps take every 16th 64-wide k block and
// reduce through shared memory.  With z set (the first head, conditioned on the
// root token): z[b, m] = h[b, m] + SiLU(a[b, m] + tab[root_b, m]) in bf16
// instead.  A programmatic dependent that reads nothing the kernels before it
// write; it waits for them only before exiting, so a later kernel's wait still
// covers everything queued ahead of this one.
constexpr int kFoldWarps = 16;
constexpr int kFoldRows = 16;    // weight rows per CTA (MMA M)
constexpr int kFoldSeq = 8;      // sequences per pass (MMA N)
constexpr int kFoldUnroll = 2;   // 64-wide k blocks per warp in flight

__device__ __forceinline__ void mma_16816_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

__global__ void __launch_bounds__(kFoldWarps * 32, 2) k_fold_h(const __nv_bfloat16* __restrict__ W1, int ldw,
                                                               const __nv_bfloat16* __restrict__ h, int B, int d,
                                                               float* __restrict__ a_out, const float* __restrict__ tab,
                                                               const __nv_bfloat16* __restrict__ b1,
                                                               const int32_t* __restrict__ root_tok, int V,
                                                               __nv_bfloat16* __restrict__ z, int32_t* __restrict__ node_tok,
                                                               float* __restrict__ node_logit,
                                                               float* __restrict__ node_logprob, int Tn, void* ws) {
    __shared__ float4 red[kFoldWarps][32];
    if (node_tok) {
        // the step's first kernel (no root kernel before it): block 0 clears the status word
        // before any dependent can start, then checks the root tokens and writes node 0
        clear_status_then_trigger(ws);
        if (blockIdx.x == 0)
            for (int b = threadIdx.x; b < B; b += blockDim.x) {
                const int t = root_tok[b];
                if (t < 0 || t >= V) flag_status(ws, SPEC_EINVAL);
                node_tok[static_cast<size_t>(b) * Tn] = min(max(t, 0), V - 1);
                node_logit[static_cast<size_t>(b) * Tn] = 0.f;
                if (node_logprob) node_logprob[static_cast<size_t>(b) * Tn] = 0.f;
            }
    } else {
        griddep_launch();
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int m0 = blockIdx.x * kFoldRows;
    const int r0 = m0 + g, r1 = m0 + g + 8;
    const bool v0 = r0 < d, v1 = r1 < d;
    const uint4* w0 = reinterpret_cast<const uint4*>(W1 + static_cast<size_t>(v0 ? r0 : 0) * ldw);
    const uint4* w1 = reinterpret_cast<const uint4*>(W1 + static_cast<size_t>(v1 ? r1 : 0) * ldw);
    const int nblk = (d + 63) / 64;
    const int nchunk = d / 8;                      // 16-byte chunks of a row's h_b half
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (int b0 = 0; b0 < B; b0 += kFoldSeq) {
        const int bq = b0 + g;                     // this lane's B column (sequence)
        const uint4* hq = reinterpret_cast<const uint4*>(h + static_cast<size_t>(bq < B ? bq : 0) * d);
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k0 = warp; k0 < nblk; k0 += kFoldWarps * kFoldUnroll) {
            uint4 a[kFoldUnroll][4], x[kFoldUnroll][2];
#pragma unroll
            for (int u = 0; u < kFoldUnroll; ++u) {
                const int blk = k0 + u * kFoldWarps;
                const int c0 = blk * 8 + t, c1 = blk * 8 + 4 + t;   // chunk indices (8 k each)
                const bool ok0 = blk < nblk && c0 < nchunk, ok1 = blk < nblk && c1 < nchunk;
                a[u][0] = ok0 && v0 ? __ldcs(w0 + c0) : zero;
                a[u][1] = ok1 && v0 ? __ldcs(w0 + c1) : zero;
                a[u][2] = ok0 && v1 ? __ldcs(w1 + c0) : zero;
                a[u][3] = ok1 && v1 ? __ldcs(w1 + c1) : zero;
                x[u][0] = ok0 && bq < B ? __ldg(hq + c0) : zero;
                x[u][1] = ok1 && bq < B ? __ldg(hq + c1) : zero;
            }
#pragma unroll
            for (int u = 0; u < kFoldUnroll; ++u) {
                // word j of this lane's 8-word k set: chunk j / 4, component j % 4
                const uint32_t ra[8] = {a[u][0].x, a[u][0].y, a[u][0].z, a[u][0].w, a[u][1].x, a[u][1].y, a[u][1].z, a[u][1].w};
                const uint32_t rb[8] = {a[u][2].x, a[u][2].y, a[u][2].z, a[u][2].w, a[u][3].x, a[u][3].y, a[u][3].z, a[u][3].w};
                const uint32_t rx[8] = {x[u][0].x, x[u][0].y, x[u][0].z, x[u][0].w, x[u][1].x, x[u][1].y, x[u][1].z, x[u][1].w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_16816_bf16(c, ra[2 * j], rb[2 * j], ra[2 * j + 1], rb[2 * j + 1], rx[2 * j], rx[2 * j + 1]);
            }
        }
        // c[0], c[1]: row g, sequences b0 + 2t, b0 + 2t + 1; c[2], c[3]: row g + 8, the same sequences
        red[warp][lane] = make_float4(c[0], c[1], c[2], c[3]);
        __syncthreads();
        if (warp == 0) {
            float4 s4 = red[0][lane];
#pragma unroll 1
            for (int w = 1; w < kFoldWarps; ++w) {
                const float4 o = red[w][lane];
                s4.x += o.x;
                s4.y += o.y;
                s4.z += o.z;
                s4.w += o.w;
            }
            const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = (e < 2) ? r0 : r1;
                const int b = b0 + 2 * t + (e & 1);
                if (m >= d || b >= B) continue;
                const float a = sv[e] + (b1 ? __bfloat162float(b1[m]) : 0.f);
                if (!z) {
                    a_out[static_cast<size_t>(b) * d + m] = a;
                } else {
                    const int tok = min(max(root_tok[b], 0), V - 1);   // k_init_root flags a bad token
                    const float xx = a + tab[static_cast<size_t>(tok) * d + m];
                    z[static_cast<size_t>(b) * d + m] =
                        __float2bfloat16_rn(__bfloat162float(h[static_cast<size_t>(b) * d + m]) + silu(xx));
                }
            }
        }
        __syncthreads();   // red is reused by the next pass
    }
    griddep_wait();
}

// ---------------------------------------------------------------- select: merge slices, fill children

// Eight consecutive elements m = 8c .. 8c+7 of a folded head's a[b] (fp32) and h_b
// (as stored), held raw; store() writes z[m] = h_b[m] + SiLU(a[m] + tab[m]) given
// the table's two float4 of the chunk.
constexpr int kZPre = 2;   // chunks per thread loaded before the top-k
template <typename T>
struct ZChunk {
    float4 a0, a1;
    uint4 hw[sizeof(T) / 2];
    __device__ __forceinline__ void load(const float* ab, const T* hb, int c) {
        a0 = reinterpret_cast<const float4*>(ab)[2 * c];
        a1 = reinterpret_cast<const float4*>(ab)[2 * c + 1];
#pragma unroll
        for (int i = 0; i < static_cast<int>(sizeof(T)) / 2; ++i)
            hw[i] = reinterpret_cast<const uint4*>(hb + 8 * c)[i];
    }
    __device__ __forceinline__ void store(T* zr, int c, const float4 t0, const float4 t1) const {
        const float x[8] = {a0.x + t0.x, a0.y + t0.y, a0.z + t0.z, a0.w + t0.w,
                            a1.x + t1.x, a1.y + t1.y, a1.z + t1.z, a1.w + t1.w};
        const T* hv = reinterpret_cast<const T*>(hw);
        T out[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = from_f32<T>(to_f32(hv[e]) + x[e] / (1.0f + expf(-x[e])));
#pragma unroll
        for (int i = 0; i < static_cast<int>(sizeof(T)) / 2; ++i)
            reinterpret_cast<uint4*>(zr + 8 * c)[i] = reinterpret_cast<const uint4*>(out)[i];
    }
};

// Copy the next depth's input row [h_b || E[tok]] (2d elements) with the whole CTA.
template <typename T>
__device__ __forceinline__ void write_next_row(T* __restrict__ dst, const T* __restrict__ hb, const T* __restrict__ er,
                                               int d) {
    const int vec = 16 / sizeof(T);
    const uint4* hs = reinterpret_cast<const uint4*>(hb);
    const uint4* es = reinterpret_cast<const uint4*>(er);
    uint4* o = reinterpret_cast<uint4*>(dst);
    for (int i = threadIdx.x; i < d / vec; i += blockDim.x) {
        o[i] = hs[i];
        o[d / vec + i] = es[i];
    }
}

// One CTA per row: top-k over the row's sorted per-slice candidate lists and
// the row's log-sum-exp, then the children of the row's parent node(s).
// Merging: each thread holds its slice's sorted list in registers (more
// slices than threads are folded in by bitonic merges); k rounds then take the
// best list head of the CTA -- warp reductions and one barrier per round --
// and pop it from its owner's list.
//
// The tree's structure (children, ranks, input rows, ancestors) is written once
// by spec_tree_build and by none of the kernels this one follows, so a CTA with
// one parent node (every conditioned head, and the root) reads it before
// griddep_wait(): the chain of dependent index loads then overlaps the
// projection still streaming instead of following it.  Tokens and log-probs of
// earlier depths are read only after the wait.
template <int KMAX, typename T>
__global__ void __launch_bounds__(256) k_select(const Cand* __restrict__ part_c, const float2* __restrict__ part_l,
                                                int nslices, int k, int cond, int n_int, int int_off,
                                                const int32_t* __restrict__ internal, const int32_t* __restrict__ child_off,
                                                const int32_t* __restrict__ child_idx, const int32_t* __restrict__ rank,
                                                const int32_t* __restrict__ parent,
                                                const int32_t* __restrict__ row_of, int Tn, int V,
                                                int32_t* __restrict__ node_tok, float* __restrict__ node_logit,
                                                float* __restrict__ node_logprob, void* ws, int next_n_int,
                                                int next_cond, int next_ld, int kdepth,
                                                const T* __restrict__ h, const T* __restrict__ emb, int d,
                                                T* __restrict__ xin, int cpr, const float* __restrict__ ftab,
                                                const float* __restrict__ fa, T* __restrict__ zf) {
    // cpr CTAs per row (one per child of a single parent that needs next-depth rows): each
    // computes the row's top-k (the same result) and copies its own child's rows, so the
    // embedding rows pass through cpr SMs instead of one; CTA 0 of the row writes the
    // node outputs.
    const int r = blockIdx.x / cpr, ci = blockIdx.x % cpr;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ float topv[KMAX];
    __shared__ int topi[KMAX];
    __shared__ float2 wlse[8];
    __shared__ float lse_s;
    // children of the current parent node: next-depth row, rank (at most k <= KMAX)
    __shared__ int c_row[KMAX], c_rank[KMAX];
    __shared__ int anc_node[SPEC_MAX_DEPTH + 1], anc_tok[SPEC_MAX_DEPTH + 1];

    const int b = cond ? r / n_int : r;
    const int j0 = cond ? r % n_int : 0, j1 = cond ? j0 + 1 : n_int;
    const bool one = j1 - j0 == 1;
    const bool rows = next_n_int > 0;
    const bool anc = rows && next_cond == 2;
    const size_t bT = static_cast<size_t>(b) * Tn;

    // 0. structure of a single parent node u: thread a < nc holds child a
    int u1 = 0, nc1 = 0, my_c = 0;
    if (one) {
        u1 = internal[int_off + j0];
        const int a0 = child_off[u1];
        nc1 = child_off[u1 + 1] - a0;
        if (tid < nc1) {
            my_c = child_idx[a0 + tid];
            c_rank[tid] = rank[my_c];
            c_row[tid] = rows ? row_of[my_c] : -1;
        }
        if (anc && tid == 0) {
            int a = u1;
            for (int i = kdepth; i >= 1; --i) {
                anc_node[i] = a;
                a = parent[a];
            }
        }
    }
    __syncthreads();   // anc_node is read by other threads after the wait

    // Once the projection before this kernel is complete, the next head's MLP may
    // launch: it streams its weights and waits for this kernel's outputs (tokens,
    // input rows) with its own griddep_wait().  Triggering only after the wait keeps
    // that MLP's CTAs off the SMs while the projection still streams.
    griddep_wait();
    griddep_launch();

    // a folded next head: a[b] (complete with the kernel before this one) and h_b do not
    // depend on this kernel's picks, so this thread's first kZPre chunks of them load now,
    // with the candidate lists; only the table rows wait for the top-k
    ZChunk<T> zpre[kZPre];
    if (ftab && rows) {
        const float* ab = fa + static_cast<size_t>(b) * d;
        const T* hb = h + static_cast<size_t>(b) * d;
#pragma unroll
        for (int j = 0; j < kZPre; ++j) {
            const int c = tid + j * static_cast<int>(blockDim.x);
            if (c < d / 8) zpre[j].load(ab, hb, c);
        }
    }

    // loads of earlier depths' outputs, issued with the candidate lists below
    float base1 = 0.f;
    if (one && node_logprob && tid < nc1) base1 = node_logprob[bT + u1];
    if (one && anc && tid >= 1 && tid <= kdepth) anc_tok[tid] = node_tok[bT + anc_node[tid]];

    // 1. each thread takes the list of slice tid (first k valid, placeholders after)
    // and its (max, sum exp); slices beyond blockDim are folded in by bitonic merges
    float lv[KMAX];
    int li[KMAX];
    float M = -INFINITY, S = 0.f;
    auto load_list = [&](int sl, float (&v)[KMAX], int (&ix)[KMAX]) {
        const Cand* src = part_c + (static_cast<size_t>(r) * nslices + sl) * KMAX;
#pragma unroll
        for (int e = 0; e < KMAX; ++e) {
            const Cand c = (sl < nslices && e < k) ? src[e] : Cand{-INFINITY, 0x7fffffff};
            v[e] = c.v;
            ix[e] = c.i;
        }
        if (sl < nslices) {
            const float2 p = part_l[static_cast<size_t>(r) * nslices + sl];
            lse_merge(M, S, p.x, p.y);
        }
    };
    load_list(tid, lv, li);
#pragma unroll 1
    for (int sl = tid + blockDim.x; sl < nslices; sl += blockDim.x) {
        float bv[KMAX];
        int bi[KMAX];
        load_list(sl, bv, bi);
        merge_top<KMAX>(lv, li, bv, bi);
    }
    for (int o = 16; o > 0; o >>= 1) lse_merge(M, S, __shfl_xor_sync(0xffffffffu, M, o), __shfl_xor_sync(0xffffffffu, S, o));
    if (lane == 0) wlse[warp] = make_float2(M, S);

    // 2. k rounds over the list heads.  A candidate is compared through a 32-bit key
    // that orders like its logit (NaN lowest, -0 as +0), so the warp's best head is one
    // max-reduction of keys and one min-reduction of the indices holding that key (lower
    // token wins ties); the CTA's best is the same two reductions over the warps'
    // (double-buffered shared slots, one barrier per round); the owner pops it.
    // Candidates are unique (the slices are disjoint), so the index identifies the owner.
    __shared__ uint2 slot[2][8];
    const int nw = blockDim.x >> 5;
#pragma unroll 1
    for (int rr = 0; rr < k; ++rr) {
        const unsigned key = order_key(lv[0]);
        const unsigned wk = __reduce_max_sync(0xffffffffu, key);
        const unsigned wi = __reduce_min_sync(0xffffffffu, key == wk ? static_cast<unsigned>(li[0]) : 0xffffffffu);
        if (lane == 0) slot[rr & 1][warp] = make_uint2(wk, wi);
        __syncthreads();
        const uint2 c = lane < nw ? slot[rr & 1][lane] : make_uint2(0u, 0xffffffffu);
        const unsigned bk = __reduce_max_sync(0xffffffffu, c.x);
        const unsigned bi = __reduce_min_sync(0xffffffffu, c.x == bk ? c.y : 0xffffffffu);
        if (static_cast<unsigned>(li[0]) == bi) {   // this thread's head won: pop it
#pragma unroll
            for (int e = 0; e + 1 < KMAX; ++e) { lv[e] = lv[e + 1]; li[e] = li[e + 1]; }
            lv[KMAX - 1] = -INFINITY;
            li[KMAX - 1] = 0x7fffffff;
        }
        if (tid == 0) {
            int ix = static_cast<int>(bi);
            // fewer than k finite logits (NaN/inf weights) leave placeholders: keep tokens in range
            if (ix < 0 || ix >= V) { flag_status(ws, SPEC_EINVAL); ix = 0; }
            topv[rr] = key_value(bk);
            topi[rr] = ix;
        }
    }
    if (tid == 0) {
        float MM = -INFINITY, SS = 0.f;
        for (int w = 0; w < nw; ++w) lse_merge(MM, SS, wlse[w].x, wlse[w].y);
        lse_s = MM + logf(SS);
    }
    __syncthreads();

    // 3. children of this row's parent node(s); next depth's input rows
    const int per = d / (16 / static_cast<int>(sizeof(T)));   // 16-byte chunks per d-wide block
    const size_t row0 = static_cast<size_t>(b) * next_n_int;
    for (int j = j0; j < j1; ++j) {
        int u = u1, nc = nc1;
        if (one) {
            if (tid < nc && ci == 0) {
                const int rr = c_rank[tid];
                node_tok[bT + my_c] = topi[rr];
                node_logit[bT + my_c] = topv[rr];
                if (node_logprob) node_logprob[bT + my_c] = base1 + (topv[rr] - lse_s);
            }
        } else {
            // several parent nodes share this row (an unconditioned head below the root)
            u = internal[int_off + j];
            const int a0 = child_off[u];
            nc = child_off[u + 1] - a0;
            const float base = node_logprob ? node_logprob[bT + u] : 0.f;
            __syncthreads();   // the previous parent's c_row / c_rank / anc_tok are consumed
            if (tid < nc) {
                const int c = child_idx[a0 + tid];
                const int rr = rank[c];
                node_tok[bT + c] = topi[rr];
                node_logit[bT + c] = topv[rr];
                if (node_logprob) node_logprob[bT + c] = base + (topv[rr] - lse_s);
                c_rank[tid] = rr;
                c_row[tid] = rows ? row_of[c] : -1;
            }
            if (anc && tid == 0) {
                int a = u;
                for (int i = kdepth; i >= 1; --i) {
                    anc_tok[i] = node_tok[bT + a];
                    a = parent[a];
                }
            }
            __syncthreads();
        }
        if (!rows) continue;
        if (ftab) {
            // the next head is folded (cond 1): its input row is z = h_b + SiLU(a[b] +
            // tab[tok]) itself (b1 is inside a), 8 elements per thread and chunk
            const float* ab = fa + static_cast<size_t>(b) * d;
            const T* hb = h + static_cast<size_t>(b) * d;
            for (int a = 0; a < nc; ++a) {
                if (c_row[a] < 0 || (cpr > 1 && a != ci)) continue;
                const float4* tr = reinterpret_cast<const float4*>(ftab + static_cast<size_t>(topi[c_rank[a]]) * d);
                T* zr = zf + (row0 + c_row[a]) * d;
                int j = 0;
                for (int c = tid; c < d / 8; c += blockDim.x, ++j) {
                    const float4 t0 = tr[2 * c], t1 = tr[2 * c + 1];
                    ZChunk<T> zc;
                    if (j < kZPre) {
#pragma unroll
                        for (int q = 0; q < kZPre; ++q)
                            if (q == j) zc = zpre[q];
                    } else {
                        zc.load(ab, hb, c);
                    }
                    zc.store(zr, c, t0, t1);
                }
            }
            continue;
        }
        if (anc) {
            // all-ancestor rows [h_b || E[tok(a_1)] || ... || E[tok(a_k)] || E[tok(c)]]: the
            // blocks of u's path (depths 1..k, shared by all children) then each child's own
            for (int i = 1; i <= kdepth; ++i) {
                const uint4* er = reinterpret_cast<const uint4*>(emb + static_cast<size_t>(anc_tok[i]) * d);
                for (int w = tid; w < per; w += blockDim.x) {
                    const uint4 v = er[w];
#pragma unroll
                    for (int a = 0; a < KMAX; ++a)
                        if (a < nc && c_row[a] >= 0 && (cpr == 1 || a == ci))
                            reinterpret_cast<uint4*>(xin + (row0 + c_row[a]) * next_ld)[i * per + w] = v;
                }
            }
        }
        // the children's own embedding blocks (block 1 for cond 1, block k + 1 for cond 2;
        // the h_b parts were written by the step's first kernel); every load of a chunk
        // column is issued before any store
        const int own = anc ? kdepth + 1 : 1;
        for (int w0 = tid; w0 < per; w0 += 2 * blockDim.x) {
            const int w1 = w0 + blockDim.x;   // second chunk column of this thread (if any)
            const bool two = w1 < per;
            uint4 ev0[KMAX], ev1[KMAX];
#pragma unroll
            for (int a = 0; a < KMAX; ++a)
                if (a < nc && (cpr == 1 || a == ci)) {
                    const uint4* er = reinterpret_cast<const uint4*>(emb + static_cast<size_t>(topi[c_rank[a]]) * d);
                    ev0[a] = er[w0];
                    if (two) ev1[a] = er[w1];
                }
#pragma unroll
            for (int a = 0; a < KMAX; ++a) {
                if (a < nc && c_row[a] >= 0 && (cpr == 1 || a == ci)) {
                    uint4* o = reinterpret_cast<uint4*>(xin + (row0 + c_row[a]) * next_ld) + own * per;
                    o[w0] = ev0[a];
                    if (two) o[w1] = ev1[a];
                }
            }
        }
    }
}

// The h_b parts of the conditioned heads' input rows ([h_b || E[...]]) at
// depths >= 1 depend on no drafted token, so the step's first kernel writes
// them all; each select then writes only the embedding parts of the next
// depth.  Depth slot i lists n_int[i] rows per sequence, starting at row
// first[i] of the per-sequence numbering and at element off[i] of the
// input-row region (rows of ld[i] elements, sequence-major).
struct HRows {
    int per_seq;
    int n;
    int first[SPEC_MAX_DEPTH];
    int n_int[SPEC_MAX_DEPTH];
    int ld[SPEC_MAX_DEPTH];
    size_t off[SPEC_MAX_DEPTH];
};

// CTA (b, 0): node 0 of sequence b -- its token is the root token (clamped to
// the vocabulary so later reads stay in bounds; CTA (0, 0) puts SPEC_EINVAL in
// the status word for any root token outside it) -- and head 0's whole input row when head 0 is conditioned (cond0 1:
// [h_b || E[root]], 2: h_b).  CTA (b, 1 + r): the h_b part of row r of
// sequence b in HRows.
template <typename T>
__global__ void k_init_root(const int32_t* __restrict__ root_tok, int B, int Tn, int V, int32_t* __restrict__ node_tok,
                            float* __restrict__ node_logit, float* __restrict__ node_logprob, void* ws, int cond0,
                            const T* __restrict__ h, const T* __restrict__ emb, int d, T* __restrict__ xin0,
                            T* __restrict__ xbase, const HRows hr) {
    const int b = blockIdx.x;
    // Block (0, 0) clears this call's status word before the kernel lets its dependents
    // (head 0's first kernel streams its weights meanwhile) start, then checks every root
    // token: the only flags this kernel raises come after the clear.  The other blocks
    // clamp their token silently.
    clear_status_then_trigger(ws);
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int bb = threadIdx.x; bb < B; bb += blockDim.x)
            if (root_tok[bb] < 0 || root_tok[bb] >= V) flag_status(ws, SPEC_EINVAL);
    if (blockIdx.y > 0) {
        const int r = static_cast<int>(blockIdx.y) - 1;
        int i = 0;
        while (i + 1 < hr.n && r >= hr.first[i + 1]) ++i;
        const size_t row = static_cast<size_t>(b) * hr.n_int[i] + (r - hr.first[i]);
        const uint4* hs = reinterpret_cast<const uint4*>(h + static_cast<size_t>(b) * d);
        uint4* o = reinterpret_cast<uint4*>(xbase + hr.off[i] + row * hr.ld[i]);
        for (int w = threadIdx.x; w < d / (16 / static_cast<int>(sizeof(T))); w += blockDim.x) o[w] = hs[w];
        return;
    }
    const int tok = min(max(root_tok[b], 0), V - 1);
    if (threadIdx.x == 0) {
        node_tok[static_cast<size_t>(b) * Tn] = tok;
        node_logit[static_cast<size_t>(b) * Tn] = 0.f;
        if (node_logprob) node_logprob[static_cast<size_t>(b) * Tn] = 0.f;
    }
    if (cond0 == 1) {
        write_next_row(xin0 + static_cast<size_t>(b) * 2 * d, h + static_cast<size_t>(b) * d,
                       emb + static_cast<size_t>(tok) * d, d);
    } else if (cond0 == 2) {   // all-ancestor conditioning at depth 0: h_b alone
        const uint4* hs = reinterpret_cast<const uint4*>(h + static_cast<size_t>(b) * d);
        uint4* o = reinterpret_cast<uint4*>(xin0 + static_cast<size_t>(b) * d);
        for (int w = threadIdx.x; w < d / (16 / static_cast<int>(sizeof(T))); w += blockDim.x) o[w] = hs[w];
    }
}

// ---------------------------------------------------------------- planning

struct Plan {
    int K;
    int max_rows;        // largest row count over heads
    int kmax;            // list length of the top-k partials (8 or 16)
    int nslices;         // vocabulary slices per row
    int slice_fma;       // fp32 path: tokens per slice
    size_t off_xin, off_z, off_scratch, off_pc, off_pl, off_hid, off_y, off_fa, total;
    size_t xin_at[SPEC_MAX_DEPTH + 1];   // element offset of depth k's input rows (conditioned heads)
    HRows hr;
    bool tc;             // bf16 tensor-core path
    tc::DraftTcPlan tcp;
};

inline int rows_of(const spec_tree* t, int k, int cond, int B) {
    return cond ? B * t->n_internal_at_depth[k] : B;
}

// Input width of head k: d (cond 0), 2d (cond 1), (k + 1) d (cond 2).
inline int d_in_of(int cond, int k, int d) { return d * (cond == 1 ? 2 : cond == 2 ? k + 1 : 1); }

// Lay out every conditioned depth's input rows (B x n_int rows of d_in elements
// each) one after the other; fills xin_at and the HRows table (depths >= 1).
// Returns the total element count (at least 1).
size_t xin_elems(Plan& p, const spec_tree* t, int K, const int32_t* cond, int B, int d, const bool* fold = nullptr) {
    size_t elems = 0;
    p.hr = HRows{};
    for (int k = 0; k < K && k <= SPEC_MAX_DEPTH; ++k) {
        p.xin_at[k] = 0;
        const int n_int = t->n_internal_at_depth[k];
        if (!cond[k] || n_int == 0 || (fold && fold[k])) continue;   // folded heads read z rows
        const int ld = d_in_of(cond[k], k, d);
        p.xin_at[k] = elems;
        if (k >= 1 && p.hr.n < SPEC_MAX_DEPTH) {
            p.hr.first[p.hr.n] = p.hr.per_seq;
            p.hr.n_int[p.hr.n] = n_int;
            p.hr.ld[p.hr.n] = ld;
            p.hr.off[p.hr.n] = elems;
            p.hr.per_seq += n_int;
            ++p.hr.n;
        }
        elems += static_cast<size_t>(B) * n_int * ld;
    }
    return std::max<size_t>(elems, 1);
}

// Per-head description (host).  Form 0: z = h + SiLU(W1 u + b1); form 1: the
// LayerNorm fusion head (see spec_head in the header).
struct Heads {
    int K = 0;
    int32_t cond[SPEC_MAX_DEPTH] = {}, topk[SPEC_MAX_DEPTH] = {}, form[SPEC_MAX_DEPTH] = {}, hidden[SPEC_MAX_DEPTH] = {};
    const void* W1[SPEC_MAX_DEPTH] = {};
    const void* b1[SPEC_MAX_DEPTH] = {};
    const void* W1b[SPEC_MAX_DEPTH] = {};
    const void* b1b[SPEC_MAX_DEPTH] = {};
    const void* gamma[SPEC_MAX_DEPTH] = {};
    const void* beta[SPEC_MAX_DEPTH] = {};
    const void* W2[SPEC_MAX_DEPTH] = {};
    const float* tab[SPEC_MAX_DEPTH] = {};   // folded embedding tables (cond-1 form-0 heads; NULL: none)
    int hid_width = 0;   // widest form-1 inner layer that feeds W1b (0: none)
    bool ln = false;     // some head has form 1
};

Heads heads_from_arrays(int K, const void* const* W1, const void* const* b1, const void* const* W2,
                        const int32_t* cond, const int32_t* topk, int d) {
    Heads hs;
    hs.K = K;
    for (int k = 0; k < K; ++k) {
        hs.cond[k] = cond[k];
        hs.topk[k] = topk[k];
        hs.hidden[k] = d;
        hs.W1[k] = W1[k];
        hs.b1[k] = b1 ? b1[k] : nullptr;
        hs.W2[k] = W2[k];
    }
    return hs;
}

Heads heads_from_desc(int K, const spec_head* h) {
    Heads hs;
    hs.K = K;
    for (int k = 0; k < K; ++k) {
        hs.cond[k] = h[k].cond;
        hs.topk[k] = h[k].topk;
        hs.form[k] = h[k].form;
        hs.hidden[k] = h[k].hidden;
        hs.W1[k] = h[k].W1;
        hs.b1[k] = h[k].b1;
        hs.W1b[k] = h[k].W1b;
        hs.b1b[k] = h[k].b1b;
        hs.gamma[k] = h[k].gamma;
        hs.beta[k] = h[k].beta;
        hs.W2[k] = h[k].W2;
        if (h[k].form == 1) {
            hs.ln = true;
            if (h[k].W1b) hs.hid_width = std::max(hs.hid_width, h[k].hidden);
        }
    }
    return hs;
}

spec_status check_heads(const Heads& hs, int d) {
    for (int k = 0; k < hs.K; ++k) {
        if (hs.form[k] != 0 && hs.form[k] != 1) return fail(SPEC_EINVAL, "head %d: form %d must be 0 or 1", k, hs.form[k]);
        if (!hs.W1[k] || !hs.W2[k]) return fail(SPEC_EINVAL, "head %d: W1 and W2 must not be NULL", k);
        if (hs.form[k] == 0 || !hs.W1b[k]) {
            if (hs.hidden[k] != d) return fail(SPEC_EINVAL, "head %d: hidden = %d must be d = %d here", k, hs.hidden[k], d);
        } else if (hs.hidden[k] < 8 || hs.hidden[k] > 65536 || hs.hidden[k] % 8) {
            return fail(SPEC_EINVAL, "head %d: hidden = %d must be a multiple of 8 in 8..65536", k, hs.hidden[k]);
        }
        if (hs.form[k] == 0 && (hs.W1b[k] || hs.b1b[k] || hs.gamma[k] || hs.beta[k]))
            return fail(SPEC_EINVAL, "head %d: form 0 takes no W1b, b1b, gamma or beta", k);
        const void* ptrs[] = {hs.W1[k], hs.b1[k], hs.W1b[k], hs.b1b[k], hs.gamma[k], hs.beta[k], hs.W2[k]};
        for (const void* q : ptrs)
            if (q && !aligned16(q)) return fail(SPEC_EALIGN, "head %d weights must be 16-byte aligned", k);
    }
    return SPEC_OK;
}

// Head k runs folded: the bf16 tensor-core path, a cond-1 form-0 head with a table.
inline bool folded(const Heads* hs, bool tc, int k) {
    return tc && hs && hs->tab[k] && hs->cond[k] == 1 && hs->form[k] == 0;
}

Plan make_plan(const spec_tree* t, int B, int d, int V, int K, const int32_t* cond, const int32_t* topk, spec_dtype dt,
               const Heads* hs = nullptr) {
    Plan p{};
    p.K = K;
    for (int k = 0; k < K; ++k) {
        if (t->n_internal_at_depth[k] == 0) continue;
        p.max_rows = std::max(p.max_rows, rows_of(t, k, cond[k], B));
        p.kmax = std::max(p.kmax, topk[k]);
    }
    p.kmax = p.kmax <= 8 ? 8 : 16;
    p.tc = (dt == SPEC_BF16) && tc::draft_tc_supported(d, V);
    size_t off = kWsHeader;
    auto take = [&](size_t bytes) { size_t at = off; off = round_up(off + bytes, 256); return at; };
    const size_t es = dt == SPEC_BF16 ? 2 : 4;
    if (p.tc) {
        p.tcp = tc::draft_tc_plan(p.max_rows, d, V);
        p.nslices = p.tcp.nslices;
        bool fold[SPEC_MAX_DEPTH] = {};
        for (int k = 0; k < K; ++k) fold[k] = folded(hs, true, k);
        p.off_xin = take(es * xin_elems(p, t, K, cond, B, d, fold));
        p.off_fa = take(sizeof(float) * static_cast<size_t>(K) * B * d);   // a[k][b] of folded heads
        p.off_z = take(es * static_cast<size_t>(p.tcp.rows_pad) * d);
        p.off_scratch = 0;   // unused: the MLP reduces its split-K partials on chip
        p.off_pc = take(sizeof(Cand) * static_cast<size_t>(p.max_rows) * p.nslices * p.kmax);
        p.off_pl = take(sizeof(float2) * static_cast<size_t>(p.max_rows) * p.nslices);
    } else {
        // at most 1024 slices per row
        p.slice_fma = std::max(4096, static_cast<int>(round_up((V + 1023) / 1024, 256)));
        p.nslices = (V + p.slice_fma - 1) / p.slice_fma;
        p.off_xin = take(es * xin_elems(p, t, K, cond, B, d));
        p.off_z = take(es * static_cast<size_t>(p.max_rows) * d);
        p.off_scratch = take(sizeof(float) * static_cast<size_t>(p.max_rows) * V);
        p.off_pc = take(sizeof(Cand) * static_cast<size_t>(p.max_rows) * p.nslices * p.kmax);
        p.off_pl = take(sizeof(float2) * static_cast<size_t>(p.max_rows) * p.nslices);
    }
    if (hs && hs->ln) {   // form-1 heads: the inner activations and the fp32 rows before LayerNorm
        const int rows_pad = p.tc ? p.tcp.rows_pad : p.max_rows;
        p.off_hid = take(es * static_cast<size_t>(rows_pad) * std::max(hs->hid_width, 8));
        p.off_y = take(sizeof(float) * static_cast<size_t>(rows_pad) * d);
    }
    p.total = off;
    return p;
}

spec_status check_args(const spec_tree* t, int B, int d, int V, int K, const int32_t* cond, const int32_t* topk, spec_dtype dt) {
    spec_status st = check_tree(t);
    if (st != SPEC_OK) return st;
    if (dt != SPEC_F32 && dt != SPEC_BF16) return fail(SPEC_EINVAL, "dtype %d unknown", (int)dt);
    if (B < 1 || B > 65535) return fail(SPEC_EINVAL, "B = %d out of 1..65535", B);
    if (d < 8 || d > 16384 || d % 8) return fail(SPEC_EINVAL, "d = %d must be a multiple of 8 in 8..16384", d);
    if (V < 2 || V > (1 << 24)) return fail(SPEC_EINVAL, "V = %d out of 2..2^24", V);
    if (K < 1 || K > SPEC_MAX_DEPTH) return fail(SPEC_EINVAL, "K = %d out of 1..%d", K, SPEC_MAX_DEPTH);
    if (K < t->max_depth) return fail(SPEC_EINVAL, "K = %d heads for a tree of depth %d", K, t->max_depth);
    if (!cond || !topk) return fail(SPEC_EINVAL, "cond and topk must not be NULL");
    for (int k = 0; k < K; ++k) {
        if (cond[k] < 0 || cond[k] > 2) return fail(SPEC_EINVAL, "cond[%d] = %d must be 0, 1 or 2", k, cond[k]);
        if (topk[k] < 1 || topk[k] > SPEC_MAX_TOPK || topk[k] > V)
            return fail(SPEC_EINVAL, "topk[%d] = %d out of 1..min(%d, V)", k, topk[k], SPEC_MAX_TOPK);
        if (k + 1 <= t->max_depth && t->max_rank_at_depth[k + 1] >= topk[k])
            return fail(SPEC_EINVAL, "a depth-%d node has rank %d >= topk[%d] = %d", k + 1, t->max_rank_at_depth[k + 1], k, topk[k]);
        if (static_cast<int64_t>(rows_of(t, k, cond[k], B)) > 65535)
            return fail(SPEC_EINVAL, "head %d has %lld rows, more than 65535", k, (long long)rows_of(t, k, cond[k], B));
    }
    return SPEC_OK;
}

template <int KMAX, typename T>
spec_status launch_select(bool pdl, const Plan& p, const spec_tree* t, int R, int k, int topk, int cond, int n_int,
                          int int_off, int next_n_int, int V, const Cand* pc, const float2* pl, int32_t* node_tok,
                          float* node_logit, float* node_logprob, void* ws, const T* h, const T* emb, int d, T* xin,
                          int next_cond, int next_ld, const float* ftab, const float* fa, T* zf, cudaStream_t s) {
    // one CTA per child where each CTA has a single parent node and children get next-depth rows
    const bool single_parent = cond != 0 || n_int == 1;
    const int cpr = (next_n_int > 0 && single_parent && k + 1 <= t->max_depth)
                        ? std::max(1, std::min(topk, t->max_rank_at_depth[k + 1] + 1)) : 1;
    SPEC_CUDA_TRY(launch_ex("draft_select", k_select<KMAX, T>, dim3(R * cpr), dim3(256), 0, s, pdl, pc, pl, p.nslices, topk,
                            cond, n_int, int_off, t->internal, t->child_off, t->child_idx, t->rank, t->parent,
                            t->row_of, t->T, V, node_tok, node_logit, node_logprob, ws, next_n_int, next_cond, next_ld, k,
                            h, emb, d, xin, cpr, ftab, fa, zf));
    return SPEC_OK;
}

template <typename T>
spec_status run(const T* h, const T* emb, const Heads& hs, float ln_eps, const int32_t* root_tok, const spec_tree* t,
                int B, int d, int V, int32_t* node_tok, float* node_logit, float* node_logprob, void* ws, const Plan& p,
                cudaStream_t s) {
    const int K = hs.K;
    const int32_t* cond = hs.cond;
    const int32_t* topk = hs.topk;
    unsigned char* w = static_cast<unsigned char*>(ws);
    T* xbase = reinterpret_cast<T*>(w + p.off_xin);
    T* z = reinterpret_cast<T*>(w + p.off_z);
    float* scratch = reinterpret_cast<float*>(w + p.off_scratch);
    Cand* pc = reinterpret_cast<Cand*>(w + p.off_pc);
    float2* pl = reinterpret_cast<float2*>(w + p.off_pl);
    T* hid = reinterpret_cast<T*>(w + p.off_hid);
    float* yln = reinterpret_cast<float*>(w + p.off_y);
    float* fa = reinterpret_cast<float*>(w + p.off_fa);
    bool fold[SPEC_MAX_DEPTH + 1] = {};
    for (int k = 0; k < K; ++k) fold[k] = folded(&hs, p.tc, k);
    const bool first_cond = t->n_internal_at_depth[0] > 0 && cond[0] && !fold[0];
    // k_init_root clears the status word (no memset: it would break the launch chain).  When
    // head 0 is folded and no depth needs h_b rows, the folded first layer of head 0 does the
    // root kernel's work itself and the chain starts one launch shorter.
    const bool root_in_fold = fold[0] && t->n_internal_at_depth[0] > 0 && p.hr.per_seq == 0;
    if (!root_in_fold)
        SPEC_CUDA_TRY(launch("draft_init_root", k_init_root<T>, dim3(B, 1 + p.hr.per_seq), dim3(128), 0, s, root_tok, B,
                             t->T, V, node_tok, node_logit, node_logprob, ws, first_cond ? cond[0] : 0, h, emb, d,
                             xbase + p.xin_at[0], xbase, p.hr));
    int int_off = 0;
    for (int k = 0; k < K; int_off += t->n_internal_at_depth[k], ++k) {
        const int n_int = t->n_internal_at_depth[k];
        if (n_int == 0) continue;   // no node of depth k has children: nothing to draft at depth k+1
        const int R = rows_of(t, k, cond[k], B);
        const int d_in = d_in_of(cond[k], k, d);
        // conditioned rows: h_b halves by the step's first kernel, embedding halves by the previous select
        const T* X = cond[k] ? xbase + p.xin_at[k] : h;
        T* xin = k + 1 <= SPEC_MAX_DEPTH ? xbase + p.xin_at[k + 1] : xbase;   // next depth's rows
        const int ldx = cond[k] ? d_in : d;
        const int next_n_int = (k + 1 < K && k + 1 <= SPEC_MAX_DEPTH && t->n_internal_at_depth[k + 1] > 0 && cond[k + 1])
                                   ? t->n_internal_at_depth[k + 1] : 0;
        const int next_cond = next_n_int > 0 ? cond[k + 1] : 0;
        const int next_ld = next_n_int > 0 ? d_in_of(next_cond, k + 1, d) : 0;
        const T* W1k = static_cast<const T*>(hs.W1[k]);
        const T* b1k = static_cast<const T*>(hs.b1[k]);
        const T* W2k = static_cast<const T*>(hs.W2[k]);
        // Input columns that come from the previous kernel: the embedding parts of a
        // conditioned head's rows (the previous select writes them, the step's first
        // kernel the h_b parts, long complete by then); every column of the first head's
        // rows, which that first kernel gathers while the head's MLP starts.
        const int dep_k0 = !cond[k] ? d_in : k == 0 ? 0 : d;
        // form 1: a = SiLU(W1 u + b1) into hid (W1b set) or yln; y = W1b a + b1b into yln;
        // z = LayerNorm(y) (queued between the MLP and the projection)
        const bool ln = hs.form[k] == 1;
        const T* W1bk = static_cast<const T*>(hs.W1b[k]);
        auto layernorm = [&]() -> spec_status {
            SPEC_CUDA_TRY(launch_ex("draft_layernorm", k_layernorm<T>, dim3(R), dim3(kLnThreads), 0, s, p.tc, yln, d,
                                    static_cast<const T*>(hs.gamma[k]), static_cast<const T*>(hs.beta[k]), ln_eps, z));
            return SPEC_OK;
        };
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            if (p.tc) {
                spec_status st;
                const bool fnext = next_n_int > 0 && fold[k + 1];
                const int fold_grid = (d + kFoldRows - 1) / kFoldRows;
                if (fold[k]) {
                    // the first head's z from its folded layer (later heads' z come from the select)
                    if (k == 0)
                        SPEC_CUDA_TRY(launch_ex("draft_fold_h", k_fold_h, dim3(fold_grid), dim3(kFoldWarps * 32), 0, s,
                                                !root_in_fold, W1k, 2 * d, h, B, d, static_cast<float*>(nullptr), hs.tab[0],
                                                b1k, root_tok, V, z, root_in_fold ? node_tok : nullptr, node_logit,
                                                node_logprob, t->T, ws));
                    st = tc::proj_tc(p.tcp, W2k, z, R, d, V, topk[k], p.kmax, pc, pl, ws, s);
                } else if (!ln) {
                    st = tc::draft_head_tc(p.tcp, W1k, b1k, W2k, h, X, d_in, ldx, z, R, d, V, cond[k], n_int, topk[k],
                                           p.kmax, dep_k0, pc, pl, ws, s);
                } else {
                    st = tc::mlp_tc(W1k, b1k, hs.hidden[k], X, d_in, ldx, R, cond[k], n_int, dep_k0, 1, nullptr,
                                    W1bk ? hid : nullptr, W1bk ? nullptr : yln, ws, s);
                    if (st == SPEC_OK && W1bk)
                        st = tc::mlp_tc(W1bk, static_cast<const T*>(hs.b1b[k]), d, hid, hs.hidden[k], hs.hidden[k], R,
                                        0, 1, 0, 0, nullptr, nullptr, yln, ws, s);
                    if (st == SPEC_OK) st = layernorm();
                    if (st == SPEC_OK) st = tc::proj_tc(p.tcp, W2k, z, R, d, V, topk[k], p.kmax, pc, pl, ws, s);
                }
                if (st != SPEC_OK) return st;
                // the next head's a = W1[:, :d] h_b streams behind this projection; the select then
                // writes that head's z rows
                float* fa_next = fa + static_cast<size_t>(k + 1) * B * d;
                if (fnext)
                    SPEC_CUDA_TRY(launch_ex("draft_fold_h", k_fold_h, dim3(fold_grid), dim3(kFoldWarps * 32), 0, s, true,
                                            static_cast<const T*>(hs.W1[k + 1]), 2 * d, h, B, d, fa_next,
                                            static_cast<const float*>(nullptr), static_cast<const T*>(hs.b1[k + 1]),
                                            static_cast<const int32_t*>(nullptr), V, static_cast<T*>(nullptr),
                                            static_cast<int32_t*>(nullptr), static_cast<float*>(nullptr),
                                            static_cast<float*>(nullptr), t->T, ws));
                const float* ftab = fnext ? hs.tab[k + 1] : nullptr;
                st = p.kmax == 8 ? launch_select<8, T>(true, p, t, R, k, topk[k], cond[k], n_int, int_off, next_n_int, V,
                                                       pc, pl, node_tok, node_logit, node_logprob, ws, h, emb, d, xin, next_cond,
                                                       next_ld, ftab, fa_next, z, s)
                                 : launch_select<16, T>(true, p, t, R, k, topk[k], cond[k], n_int, int_off, next_n_int, V,
                                                        pc, pl, node_tok, node_logit, node_logprob, ws, h, emb, d, xin, next_cond,
                                                        next_ld, ftab, fa_next, z, s);
                if (st != SPEC_OK) return st;
                continue;
            }
        }
        if (!ln) {
            SPEC_CUDA_TRY((launch_gemm<T, 0>("draft_mlp_fma", s, W1k, d_in, X, d, R, d_in, ldx, b1k, h, cond[k], n_int, z,
                                             static_cast<float*>(nullptr), 1, static_cast<float*>(nullptr))));
        } else {
            const int hd = hs.hidden[k];
            SPEC_CUDA_TRY((launch_gemm<T, 0>("draft_mlp_fma", s, W1k, d_in, X, hd, R, d_in, ldx, b1k,
                                             static_cast<const T*>(nullptr), cond[k], n_int, W1bk ? hid : nullptr,
                                             static_cast<float*>(nullptr), 1, W1bk ? static_cast<float*>(nullptr) : yln)));
            if (W1bk)
                SPEC_CUDA_TRY((launch_gemm<T, 0>("draft_mlp_fma", s, W1bk, hd, static_cast<const T*>(hid), d, R, hd, hd,
                                                 static_cast<const T*>(hs.b1b[k]), static_cast<const T*>(nullptr), 0, 1,
                                                 static_cast<T*>(nullptr), static_cast<float*>(nullptr), 0, yln)));
            spec_status st = layernorm();
            if (st != SPEC_OK) return st;
        }
        SPEC_CUDA_TRY((launch_gemm<T, 1>("draft_proj_fma", s, W2k, d, static_cast<const T*>(z), V, R, d, d,
                                         static_cast<const T*>(nullptr), static_cast<const T*>(nullptr), 0, 1,
                                         static_cast<T*>(nullptr), scratch, 0, static_cast<float*>(nullptr))));
        spec_status st;
        if (p.kmax == 8) {
            SPEC_CUDA_TRY(launch("draft_topk_slices", k_topk_slices<8>, dim3(p.nslices, R), dim3(256), 0, s, scratch, V,
                                 topk[k], p.slice_fma, pc, pl, p.nslices));
            st = launch_select<8, T>(false, p, t, R, k, topk[k], cond[k], n_int, int_off, next_n_int, V, pc, pl, node_tok,
                                     node_logit, node_logprob, ws, h, emb, d, xin, next_cond, next_ld, nullptr, nullptr,
                                     z, s);
        } else {
            SPEC_CUDA_TRY(launch("draft_topk_slices", k_topk_slices<16>, dim3(p.nslices, R), dim3(256), 0, s, scratch, V,
                                 topk[k], p.slice_fma, pc, pl, p.nslices));
            st = launch_select<16, T>(false, p, t, R, k, topk[k], cond[k], n_int, int_off, next_n_int, V, pc, pl, node_tok,
                                      node_logit, node_logprob, ws, h, emb, d, xin, next_cond, next_ld, nullptr, nullptr,
                                      z, s);
        }
        if (st != SPEC_OK) return st;
    }
    return SPEC_OK;
}

}  // namespace draft
}  // namespace spec

using namespace spec;

namespace spec {
namespace draft {

// Shared by both entry points once the heads are described.
static spec_status draft_call(const void* h, const void* emb, const Heads& hs, float ln_eps, const int32_t* root_tok,
                              const spec_tree* tree, int32_t B, int32_t d, int32_t V, spec_dtype dt, int32_t* node_tok,
                              float* node_logit, float* node_logprob, void* ws, size_t ws_bytes, cudaStream_t s) {
    spec_status st = check_args(tree, B, d, V, hs.K, hs.cond, hs.topk, dt);
    if (st != SPEC_OK) return st;
    st = check_heads(hs, d);
    if (st != SPEC_OK) return st;
    if (hs.ln && !(ln_eps > 0.f && ln_eps < 1e30f)) return fail(SPEC_EINVAL, "ln_eps must be positive and finite");
    if (!h || !emb || !root_tok || !node_tok || !node_logit)
        return fail(SPEC_EINVAL, "h, emb, root_tok, node_tok and node_logit must not be NULL");
    if (!aligned16(h) || !aligned16(emb)) return fail(SPEC_EALIGN, "h and emb must be 16-byte aligned");
    if (!aligned4(root_tok) || !aligned4(node_tok) || !aligned4(node_logit) || (node_logprob && !aligned4(node_logprob)))
        return fail(SPEC_EALIGN, "token and logit buffers must be 4-byte aligned");
    const Plan p = make_plan(tree, B, d, V, hs.K, hs.cond, hs.topk, dt, &hs);
    if (!ws || ws_bytes < p.total) return fail(SPEC_EWORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, p.total);
    if (!aligned16(ws)) return fail(SPEC_EALIGN, "workspace must be 16-byte aligned");
    for (int k = 0; k < hs.K; ++k)
        if (hs.tab[k] && !aligned16(hs.tab[k])) return fail(SPEC_EALIGN, "folded table %d must be 16-byte aligned", k);
    if (dt == SPEC_BF16)
        return run<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(h), static_cast<const __nv_bfloat16*>(emb), hs, ln_eps,
                                  root_tok, tree, B, d, V, node_tok, node_logit, node_logprob, ws, p, s);
    return run<float>(static_cast<const float*>(h), static_cast<const float*>(emb), hs, ln_eps, root_tok, tree, B, d, V,
                      node_tok, node_logit, node_logprob, ws, p, s);
}

}  // namespace draft
}  // namespace spec

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
    clear_error();
    if (K < 1 || K > SPEC_MAX_DEPTH) return fail(SPEC_EINVAL, "K = %d out of 1..%d", K, SPEC_MAX_DEPTH);
    if (!W1 || !W2 || !cond || !topk) return fail(SPEC_EINVAL, "W1, W2, cond and topk must not be NULL");
    const draft::Heads hs = draft::heads_from_arrays(K, W1, b1, W2, cond, topk, d);
    return draft::draft_call(h, emb, hs, 0.f, root_tok, tree, B, d, V, dt, node_tok, node_logit, node_logprob, ws,
                             ws_bytes, reinterpret_cast<cudaStream_t>(s_));
}

extern "C" spec_status hydra_draft_folded(const void* h, const void* emb, int32_t K, const void* const* W1,
                                          const void* const* b1, const void* const* W2, const float* const* tab,
                                          const int32_t* cond, const int32_t* topk, const int32_t* root_tok,
                                          const spec_tree* tree, int32_t B, int32_t d, int32_t V, spec_dtype dt,
                                          int32_t* node_tok, float* node_logit, float* node_logprob, void* ws,
                                          size_t ws_bytes, spec_stream_t s_) {
    clear_error();
    if (K < 1 || K > SPEC_MAX_DEPTH) return fail(SPEC_EINVAL, "K = %d out of 1..%d", K, SPEC_MAX_DEPTH);
    if (!W1 || !W2 || !cond || !topk) return fail(SPEC_EINVAL, "W1, W2, cond and topk must not be NULL");
    draft::Heads hs = draft::heads_from_arrays(K, W1, b1, W2, cond, topk, d);
    if (tab)
        for (int k = 0; k < K; ++k) hs.tab[k] = tab[k];
    return draft::draft_call(h, emb, hs, 0.f, root_tok, tree, B, d, V, dt, node_tok, node_logit, node_logprob, ws,
                             ws_bytes, reinterpret_cast<cudaStream_t>(s_));
}

extern "C" size_t hydra_fold_table_bytes(int32_t d, int32_t V) {
    clear_error();
    if (d < 8 || d > 16384 || d % 8 || V < 2 || V > (1 << 24)) return 0;
    return sizeof(float) * static_cast<size_t>(d) * V;
}

extern "C" spec_status hydra_fold_embedding(const void* W1, const void* emb, int32_t d, int32_t V, spec_dtype dt,
                                            float* tab, spec_stream_t s_) {
    clear_error();
    if (dt != SPEC_F32 && dt != SPEC_BF16) return fail(SPEC_EINVAL, "dtype %d unknown", (int)dt);
    if (d < 8 || d > 16384 || d % 8) return fail(SPEC_EINVAL, "d = %d must be a multiple of 8 in 8..16384", d);
    if (V < 2 || V > (1 << 24)) return fail(SPEC_EINVAL, "V = %d out of 2..2^24", V);
    if (!W1 || !emb || !tab) return fail(SPEC_EINVAL, "W1, emb and tab must not be NULL");
    if (!aligned16(W1) || !aligned16(emb) || !aligned16(tab)) return fail(SPEC_EALIGN, "W1, emb and tab must be 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(s_);
    if (dt == SPEC_BF16 && tc::draft_tc_supported(d, V)) {
        // tab[v, m] = W1[m, d:2d] . emb[v] on the tensor cores: the head-layer GEMM with the
        // embedding half of W1 (row stride 2d) as the weights, the vocabulary as the
        // activation rows (256 per launch) and an identity epilogue writing fp32 rows
        return tc::mlp_tc(static_cast<const __nv_bfloat16*>(W1) + d, nullptr, d, static_cast<const __nv_bfloat16*>(emb),
                          d, d, V, 0, 1, 0, 0, nullptr, nullptr, tab, nullptr, s, 2 * d);
    }
    // tab[v, m] = W1[m, d:2d] . emb[v]: the CUDA-core GEMM with the embedding half of W1
    // (row stride 2d) as the weights and the vocabulary as the rows, in chunks of grid rows
    const int chunk = 65535 * draft::GBN;
    for (int v0 = 0; v0 < V; v0 += chunk) {
        const int n = std::min(chunk, V - v0);
        const dim3 grid((d + draft::GBM - 1) / draft::GBM, (n + draft::GBN - 1) / draft::GBN);
        if (dt == SPEC_BF16) {
            using T = __nv_bfloat16;
            const T* W = static_cast<const T*>(W1) + d;
            SPEC_CUDA_TRY(launch("fold_embedding", draft::k_gemm_fma<T, 1>, grid, dim3(256), 0, s, W, 2 * d,
                                 static_cast<const T*>(emb) + static_cast<size_t>(v0) * d, d, n, d, d,
                                 static_cast<const T*>(nullptr), static_cast<const T*>(nullptr), 0, 1,
                                 static_cast<T*>(nullptr), tab + static_cast<size_t>(v0) * d, 0, static_cast<float*>(nullptr)));
        } else {
            const float* W = static_cast<const float*>(W1) + d;
            SPEC_CUDA_TRY(launch("fold_embedding", draft::k_gemm_fma<float, 1>, grid, dim3(256), 0, s, W, 2 * d,
                                 static_cast<const float*>(emb) + static_cast<size_t>(v0) * d, d, n, d, d,
                                 static_cast<const float*>(nullptr), static_cast<const float*>(nullptr), 0, 1,
                                 static_cast<float*>(nullptr), tab + static_cast<size_t>(v0) * d, 0,
                                 static_cast<float*>(nullptr)));
        }
    }
    return SPEC_OK;
}

extern "C" size_t hydra_draft_heads_workspace_size(const spec_tree* tree, int32_t B, int32_t d, int32_t V, int32_t K,
                                                   const spec_head* heads, spec_dtype dt) {
    clear_error();
    if (K < 1 || K > SPEC_MAX_DEPTH || !heads) return 0;
    const draft::Heads hs = draft::heads_from_desc(K, heads);
    if (draft::check_args(tree, B, d, V, K, hs.cond, hs.topk, dt) != SPEC_OK) return 0;
    if (draft::check_heads(hs, d) != SPEC_OK) return 0;
    return draft::make_plan(tree, B, d, V, K, hs.cond, hs.topk, dt, &hs).total;
}

extern "C" spec_status hydra_draft_heads(const void* h, const void* emb, int32_t K, const spec_head* heads,
                                         const int32_t* root_tok, const spec_tree* tree, int32_t B, int32_t d,
                                         int32_t V, float ln_eps, spec_dtype dt, int32_t* node_tok, float* node_logit,
                                         float* node_logprob, void* ws, size_t ws_bytes, spec_stream_t s_) {
    clear_error();
    if (K < 1 || K > SPEC_MAX_DEPTH) return fail(SPEC_EINVAL, "K = %d out of 1..%d", K, SPEC_MAX_DEPTH);
    if (!heads) return fail(SPEC_EINVAL, "heads must not be NULL");
    const draft::Heads hs = draft::heads_from_desc(K, heads);
    return draft::draft_call(h, emb, hs, ln_eps, root_tok, tree, B, d, V, dt, node_tok, node_logit, node_logprob, ws,
                             ws_bytes, reinterpret_cast<cudaStream_t>(s_));
}
